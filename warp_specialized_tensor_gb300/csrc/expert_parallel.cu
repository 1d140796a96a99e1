// expert_parallel.cu -- index plans and row movement for the expert-parallel
// grouped GEMM.
//
// "How We Built TLX: A Hardware-Native GPU Compiler for Production ML at
// Scale" (Meta Engineering), "Case Study 3: Distributed Grouped GEMM for LLM
// Pretraining" and "TLX in Production": the experts of a mixture-of-experts
// layer are spread over the GPUs of a node; each GPU sends every routed
// (token, expert) pair to the GPU that owns the expert, runs its own experts'
// grouped GEMM on what it received, and sends the products back.
//
// Layout used here: R ranks, G experts, G divisible by R; rank r owns the
// contiguous experts [r*G/R, (r+1)*G/R).  A token's k routed experts are its
// pairs p = t*k + s.
//   dispatch plan (host):  the pairs a rank sends, ordered by destination
//                          rank, then the destination's local expert, then
//                          pair id; per (destination, local expert) counts.
//   receive plan (host):   rows arrive grouped by source rank, each source's
//                          block ordered by local expert; the grouped GEMM
//                          wants them by expert: for local expert e and
//                          source s in order, the rows of (s, e).  The plan
//                          gives the expert-major order as indices into the
//                          received rows, plus the grouped GEMM's offsets.
//   wst_permute_rows:      one CUDA kernel that gathers and / or scatters
//                          whole rows by device index arrays (every data
//                          movement of the dispatch and the combine).
// The exchange itself (an all-to-all of rows with these counts) is the
// caller's collective.
#include <cstring>
#include <vector>

#include "wst.h"
#include "wst_common.cuh"
#include "wst_host.h"

namespace wst {

// Row permutation: dst[d ? d[i] : i] = src[s ? s[i] : i] for i < n, each row
// `vecs` 16-byte vectors.  One warp per row, rows strided over the grid;
// indices outside [0, n_src) / [0, n_dst) skip the row and latch
// WST_ERR_INVALID_ARG in the workspace header.
__global__ void __launch_bounds__(256) k_permute_rows(int n, int vecs, const uint4* __restrict__ src,
                                                      long long src_stride, const int* __restrict__ sidx,
                                                      int n_src, uint4* __restrict__ dst,
                                                      long long dst_stride, const int* __restrict__ didx,
                                                      int n_dst, WsHeader* ws) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long i = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < n; i += warps) {
    const int si = sidx ? __ldg(sidx + i) : (int)i;
    const int di = didx ? __ldg(didx + i) : (int)i;
    if (si < 0 || si >= n_src || di < 0 || di >= n_dst) {
      if (lane == 0) latch_error(ws, 1u /*WST_ERR_INVALID_ARG*/, 0x50000u);
      continue;
    }
    const uint4* s = src + (long long)si * src_stride;
    uint4* d = dst + (long long)di * dst_stride;
    for (int v = lane; v < vecs; v += 32) d[v] = __ldg(s + v);
  }
}

int run_permute_rows(int n, size_t row_bytes, const void* src, size_t src_stride_bytes,
                     const int* sidx, int n_src, void* dst, size_t dst_stride_bytes,
                     const int* didx, int n_dst, void* ws, cudaStream_t stream) {
  DeviceInfo dev;
  int st = current_device_info(&dev);
  if (st) return st;
  if (n == 0) return ST_OK;
  // 8 warps per CTA, 8 CTAs per SM, never more warps than rows.
  long long ctas = ((long long)n + 7) / 8;
  const long long cap = 8LL * dev.num_sms;
  if (ctas > cap) ctas = cap;
  k_permute_rows<<<(unsigned)ctas, 256, 0, stream>>>(
      n, (int)(row_bytes / 16), static_cast<const uint4*>(src), (long long)(src_stride_bytes / 16), sidx,
      n_src, static_cast<uint4*>(dst), (long long)(dst_stride_bytes / 16), didx, n_dst,
      static_cast<WsHeader*>(ws));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch k_permute_rows");
  return ST_OK;
}

}  // namespace wst

using namespace wst;

namespace {
wst_status ep_fail(wst_status s, const char* msg) {
  set_error("%s", msg);
  return s;
}
}  // namespace

extern "C" {

wst_status wst_ep_dispatch_plan(int num_tokens, int top_k, const int* routing, int num_experts,
                                int world_size, int* send_counts, int* send_group_counts,
                                int* send_pairs) {
  set_error("%s", "");
  if (num_tokens < 0 || top_k < 1 || num_experts < 1 || world_size < 1)
    return ep_fail(WST_ERR_INVALID_ARG, "ep dispatch plan: sizes out of range");
  if (num_experts % world_size)
    return ep_fail(WST_ERR_INVALID_ARG, "ep dispatch plan: num_experts must be a multiple of world_size");
  if ((num_tokens > 0 && (!routing || !send_pairs)) || !send_counts || !send_group_counts)
    return ep_fail(WST_ERR_INVALID_ARG, "ep dispatch plan: NULL array");
  const long long pairs = (long long)num_tokens * top_k;
  if (pairs > 0x7fffffffLL) return ep_fail(WST_ERR_INVALID_ARG, "ep dispatch plan: too many pairs");
  // Counting sort of the pairs by expert (stable: pair ids ascend within an
  // expert); expert-major order is destination-major, local-expert-minor
  // because each rank owns a contiguous block of experts.
  std::vector<long long> start((size_t)num_experts + 1, 0);
  for (long long p = 0; p < pairs; ++p) {
    const int e = routing[p];
    if (e < 0 || e >= num_experts) {
      set_error("ep dispatch plan: expert id %d of pair %lld outside [0, %d)", e, p, num_experts);
      return WST_ERR_INVALID_ARG;
    }
    ++start[(size_t)e + 1];
  }
  const int per_rank = num_experts / world_size;
  for (int e = 0; e < num_experts; ++e) send_group_counts[e] = (int)start[(size_t)e + 1];
  for (int r = 0; r < world_size; ++r) {
    long long c = 0;
    for (int j = 0; j < per_rank; ++j) c += start[(size_t)r * per_rank + j + 1];
    send_counts[r] = (int)c;
  }
  for (int e = 0; e < num_experts; ++e) start[(size_t)e + 1] += start[(size_t)e];
  for (long long p = 0; p < pairs; ++p) send_pairs[start[(size_t)routing[p]]++] = (int)p;
  return WST_OK;
}

wst_status wst_ep_receive_plan(int world_size, int experts_per_rank, const int* recv_group_counts,
                               int* group_offsets, int* expert_rows) {
  set_error("%s", "");
  if (world_size < 1 || experts_per_rank < 1)
    return ep_fail(WST_ERR_INVALID_ARG, "ep receive plan: sizes out of range");
  if (!recv_group_counts || !group_offsets)
    return ep_fail(WST_ERR_INVALID_ARG, "ep receive plan: NULL array");
  // First received row of each (source, expert) block.
  std::vector<long long> block((size_t)world_size * experts_per_rank);
  long long total = 0;
  for (int s = 0; s < world_size; ++s)
    for (int e = 0; e < experts_per_rank; ++e) {
      const int c = recv_group_counts[(size_t)s * experts_per_rank + e];
      if (c < 0) return ep_fail(WST_ERR_INVALID_ARG, "ep receive plan: negative count");
      block[(size_t)s * experts_per_rank + e] = total;
      total += c;
    }
  if (total > 0x7fffffffLL) return ep_fail(WST_ERR_INVALID_ARG, "ep receive plan: too many rows");
  if (total > 0 && !expert_rows) return ep_fail(WST_ERR_INVALID_ARG, "ep receive plan: NULL array");
  long long o = 0;
  for (int e = 0; e < experts_per_rank; ++e) {
    group_offsets[e] = (int)o;
    for (int s = 0; s < world_size; ++s) {
      const int c = recv_group_counts[(size_t)s * experts_per_rank + e];
      const long long b = block[(size_t)s * experts_per_rank + e];
      for (int i = 0; i < c; ++i) expert_rows[o++] = (int)(b + i);
    }
  }
  group_offsets[experts_per_rank] = (int)o;
  return WST_OK;
}

wst_status wst_permute_rows(int n_rows, size_t row_bytes, const void* src, size_t src_stride,
                            const int* d_src_index, int n_src_rows, void* dst, size_t dst_stride,
                            const int* d_dst_index, int n_dst_rows, void* workspace, void* stream) {
  set_error("%s", "");
  if (n_rows < 0 || n_src_rows < 0 || n_dst_rows < 0)
    return ep_fail(WST_ERR_INVALID_ARG, "permute rows: negative size");
  if (!workspace) return ep_fail(WST_ERR_INVALID_ARG, "permute rows: workspace is NULL");
  if (n_rows == 0) return WST_OK;
  if (!src || !dst) return ep_fail(WST_ERR_INVALID_ARG, "permute rows: NULL src or dst");
  if (row_bytes == 0 || row_bytes % 16 || src_stride % 16 || dst_stride % 16 ||
      src_stride < row_bytes || dst_stride < row_bytes)
    return ep_fail(WST_ERR_ALIGNMENT, "permute rows: row bytes and strides must be multiples of 16, strides >= row bytes");
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) |
       reinterpret_cast<uintptr_t>(workspace)) & 15u)
    return ep_fail(WST_ERR_ALIGNMENT, "permute rows: src, dst and workspace must be 16-byte aligned");
  if (row_bytes / 16 > 0x7fffffffULL) return ep_fail(WST_ERR_INVALID_ARG, "permute rows: row too long");
  if (!d_src_index && n_rows > n_src_rows)
    return ep_fail(WST_ERR_INVALID_ARG, "permute rows: more rows than the source holds");
  if (!d_dst_index && n_rows > n_dst_rows)
    return ep_fail(WST_ERR_INVALID_ARG, "permute rows: more rows than the destination holds");
  return (wst_status)run_permute_rows(n_rows, row_bytes, src, src_stride, d_src_index, n_src_rows,
                                      dst, dst_stride, d_dst_index, n_dst_rows, workspace,
                                      static_cast<cudaStream_t>(stream));
}

}  // extern "C"
