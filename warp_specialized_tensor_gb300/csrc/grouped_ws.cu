// grouped_ws.cu -- instantiations and launcher of the grouped (MoE) GEMM.
#include "grouped_ws.cuh"
#include "wst_host.h"

namespace wst {

namespace {

// Tile schedule: the static persistent walk unless the process-wide option
// WST_OPT_GROUPED_SCHEDULE selects hardware cluster launch control (read on
// every call).
inline bool grouped_use_clc() { return option_value(OPT_GROUPED_SCHEDULE) == 1; }

template <bool OUT_F32, int EPI, bool CLC>
int launch_grouped(const GemmProblem& pr, const DeviceInfo& dev, cudaStream_t stream) {
  auto kern = k_grouped_ws<OUT_F32, EPI, CLC>;
  int st;
  CUtensorMap tmW, tmX, tmXt, tmC;
  GroupedArgs a{};
  a.w_shared = (pr.strideB == 0) ? 1 : 0;
  {
    // B[g] rows (expert output features), K contiguous: {K, N, G}
    uint64_t dims[3] = {(uint64_t)pr.K, (uint64_t)pr.N, (uint64_t)(a.w_shared ? 1 : pr.batch)};
    uint64_t str[2] = {(uint64_t)pr.ldb * 2,
                       (uint64_t)(a.w_shared ? (long long)pr.N * pr.ldb : pr.strideB) * 2};
    uint32_t box[3] = {64, 128, 1};
    if ((st = encode_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, pr.B, dims, str, box,
                         CU_TENSOR_MAP_SWIZZLE_128B)))
      return st;
  }
  {
    // token rows of A, K contiguous: {K, M_total}; 128-row boxes, and
    // 16-row boxes for thin tiles
    uint64_t dims[2] = {(uint64_t)pr.K, (uint64_t)pr.M};
    uint64_t str[1] = {(uint64_t)pr.lda * 2};
    uint32_t box[2] = {64, (uint32_t)kGrpXBoxRows};
    if ((st = encode_map(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pr.A, dims, str, box,
                         CU_TENSOR_MAP_SWIZZLE_128B)))
      return st;
    box[1] = (uint32_t)kGrpXThinRows;
    if ((st = encode_map(&tmXt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pr.A, dims, str, box,
                         CU_TENSOR_MAP_SWIZZLE_128B)))
      return st;
  }
  {
    // C rows (tokens) x features, row-major: {N, M_total}; box = one
    // epilogue warp's transposed block of 32 features x 32 tokens
    const uint64_t es = OUT_F32 ? 4 : 2;
    uint64_t dims[2] = {(uint64_t)pr.N, (uint64_t)pr.M};
    uint64_t str[1] = {(uint64_t)pr.ldc * es};
    uint32_t box[2] = {32, 32};
    if ((st = encode_map(&tmC, OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         2, pr.C, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE)))
      return st;
  }
  a.G = pr.batch;
  a.M_total = pr.M;
  a.N = pr.N;
  a.K = pr.K;
  a.n_tiles = (pr.N + kGrpTileN - 1) / kGrpTileN;
  a.k_blocks = (pr.K + kGrpBK - 1) / kGrpBK;
  a.offsets = pr.offsets;
  a.bias = static_cast<const __nv_bfloat16*>(pr.bias);
  a.bias_stride = pr.strideBias;
  a.C = pr.C;
  a.ldc = pr.ldc;
  a.ws = static_cast<WsHeader*>(pr.ws);
  a.timeout_ns = wait_timeout_ns();

  if ((st = ensure_smem_attr((const void*)kern, kGrpSmemBytes))) return st;
  cudaError_t e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(kGrpThreads, 1, 1);
  cfg.dynamicSmemBytes = kGrpSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  long long pairs;
  if (CLC) {
    // One pair per tile.  The group sizes are on the device, so bound the
    // tile count: sum_g ceil(M_g/256) <= floor(M_total/256) + min(G, M_total).
    pairs = (long long)a.n_tiles *
            ((long long)a.M_total / kGrpTileT + std::min<long long>(a.G, a.M_total));
    if (pairs < 1) pairs = 1;  // pair 0 still validates the offsets
    if (2 * pairs > 0x7fffffffLL) {
      set_error("grouped GEMM: %lld tiles exceed the grid limit of cluster launch control", pairs);
      return ST_UNSUPPORTED;
    }
  } else {
    // Persistent grid: every CTA pair that can be resident at once.
    static int max_clusters[64] = {0};
    int& mc = max_clusters[dev.device & 63];
    if (mc == 0) {
      cfg.gridDim = dim3((unsigned)(dev.num_sms & ~1), 1, 1);
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (e != cudaSuccess || n < 1) {
        cudaGetLastError();
        n = dev.num_sms / 2;
      }
      mc = n;
    }
    pairs = mc;
  }
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  e = cudaLaunchKernelEx(&cfg, kern, tmW, tmX, tmXt, tmC, a);
  if (e != cudaSuccess) return cuda_fail(e, "launch k_grouped_ws");
  return ST_OK;
}

}  // namespace

namespace {

template <bool CLC>
int dispatch_grouped(const GemmProblem& pr, const DeviceInfo& dev, cudaStream_t stream) {
  if (pr.c_f32) {
    switch (pr.epi) {
      case 0: return launch_grouped<true, 0, CLC>(pr, dev, stream);
      case 1: return launch_grouped<true, 1, CLC>(pr, dev, stream);
      case 2: return launch_grouped<true, 2, CLC>(pr, dev, stream);
      default: return launch_grouped<true, 3, CLC>(pr, dev, stream);
    }
  }
  switch (pr.epi) {
    case 0: return launch_grouped<false, 0, CLC>(pr, dev, stream);
    case 1: return launch_grouped<false, 1, CLC>(pr, dev, stream);
    case 2: return launch_grouped<false, 2, CLC>(pr, dev, stream);
    default: return launch_grouped<false, 3, CLC>(pr, dev, stream);
  }
}

}  // namespace

int run_gemm_grouped(const GemmProblem& pr, const DeviceInfo& dev, cudaStream_t stream) {
  return grouped_use_clc() ? dispatch_grouped<true>(pr, dev, stream)
                           : dispatch_grouped<false>(pr, dev, stream);
}

}  // namespace wst
