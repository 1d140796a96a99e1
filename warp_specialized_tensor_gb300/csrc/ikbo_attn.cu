// ikbo_attn.cu -- instantiations and launcher of the IKBO attention kernel:
// tensor maps over Q and the users' K/V, kernel arguments, grid size, launch.
#include <algorithm>

#include "ikbo_attn_ws.cuh"
#include "wst_host.h"

namespace wst {

namespace {

template <bool OUT_F32>
int launch_attn(const AttnProblem& pr, const DeviceInfo& dev, cudaStream_t stream) {
  auto kern = k_ikbo_attn_ws<OUT_F32>;
  int st;
  CUtensorMap tmQ, tmK, tmV, tmO;
  const uint64_t nq = (uint64_t)pr.num_cand * (uint64_t)pr.Lq;
  const uint64_t row_bytes = (uint64_t)pr.H * kAttnDh * 2;
  {
    // Q rows, one head at a time: {Dh, H, rows}, boxes of 64 d x 1 head x 128 rows
    uint64_t dims[3] = {(uint64_t)kAttnDh, (uint64_t)pr.H, nq};
    uint64_t str[2] = {(uint64_t)kAttnDh * 2, row_bytes};
    uint32_t box[3] = {64, 1, (uint32_t)kAttnBM};
    if ((st = encode_map(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, pr.Q, dims, str, box,
                         CU_TENSOR_MAP_SWIZZLE_128B)))
      return st;
  }
  {
    // K and V: {Dh, H, Lkv, users}, boxes of 64 d x 1 head x 64 keys x 1 user;
    // keys past Lkv read as zero (and are masked in the softmax)
    uint64_t dims[4] = {(uint64_t)kAttnDh, (uint64_t)pr.H, (uint64_t)pr.Lkv, (uint64_t)pr.num_users};
    uint64_t str[3] = {(uint64_t)kAttnDh * 2, row_bytes, row_bytes * (uint64_t)pr.Lkv};
    uint32_t box[4] = {64, 1, (uint32_t)kAttnBN, 1};
    if ((st = encode_map(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, pr.K, dims, str, box,
                         CU_TENSOR_MAP_SWIZZLE_128B)))
      return st;
    if ((st = encode_map(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, pr.V, dims, str, box,
                         CU_TENSOR_MAP_SWIZZLE_128B)))
      return st;
  }
  if (!OUT_F32) {
    // bf16 O rows: {Dh, H, rows}, boxes of 64 d x 1 head x 32 rows (one
    // softmax warp's rows of a tile)
    uint64_t dims[3] = {(uint64_t)kAttnDh, (uint64_t)pr.H, nq};
    uint64_t str[2] = {(uint64_t)kAttnDh * 2, row_bytes};
    uint32_t box[3] = {64, 1, 32};
    if ((st = encode_map(&tmO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, pr.O, dims, str, box,
                         CU_TENSOR_MAP_SWIZZLE_128B)))
      return st;
  } else {
    tmO = tmQ;  // unused
  }
  AttnArgs a{};
  a.num_users = pr.num_users;
  a.num_cand = pr.num_cand;
  a.Lq = pr.Lq;
  a.H = pr.H;
  a.Lkv = pr.Lkv;
  a.kv_blocks = (pr.Lkv + kAttnBN - 1) / kAttnBN;
  a.scale_log2 = (float)((double)pr.scale * 1.4426950408889634);  // scale * log2(e)
  a.uoff = pr.uoff;
  a.O = pr.O;
  a.ws = static_cast<WsHeader*>(pr.ws);
  a.timeout_ns = wait_timeout_ns();
  a.epoch = next_flag_epoch();

  // Persistent grid: one CTA per SM.  Without the key-block split, no more
  // CTAs than the items can use (the per-user item counts live on the
  // device: bound them by H * (query tiles + users)); with it, every SM
  // takes a share of the last wave.
  const bool split = pr.ws_bytes >= kAttnWorkspaceBytes && dev.num_sms <= kAttnMaxCtas;
  const long long items_max =
      (long long)pr.H * ((long long)((nq + kAttnBM - 1) / kAttnBM) + pr.num_users);
  const long long grid =
      split ? dev.num_sms : std::max(1LL, std::min<long long>(dev.num_sms, items_max));
  uint8_t* ws = static_cast<uint8_t*>(pr.ws);
  a.split = split ? 1 : 0;
  a.flags = split ? reinterpret_cast<uint32_t*>(ws + kAttnFlagsOffset) : nullptr;
  a.slots = split ? reinterpret_cast<float*>(ws + kAttnSlotsOffset) : nullptr;
  if ((st = ensure_smem_attr((const void*)kern, kAttnSmemBytes))) return st;
  // Cooperative: a CTA merging a split item waits for CTAs of higher index,
  // which must all be resident.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kAttnThreads, 1, 1);
  cfg.dynamicSmemBytes = kAttnSmemBytes;
  cfg.stream = stream;
  cfg.attrs = split ? attr : nullptr;
  cfg.numAttrs = split ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmQ, tmK, tmV, tmO, a);
  if (e != cudaSuccess) return cuda_fail(e, "launch k_ikbo_attn_ws");
  return ST_OK;
}

}  // namespace

int run_ikbo_attention(const AttnProblem& pr, cudaStream_t stream) {
  DeviceInfo dev;
  int st = current_device_info(&dev);
  if (st) return st;
  return pr.o_f32 ? launch_attn<true>(pr, dev, stream) : launch_attn<false>(pr, dev, stream);
}

size_t attention_workspace_bytes() { return kAttnWorkspaceBytes; }

}  // namespace wst
