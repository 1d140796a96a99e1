// gemm_ws_launch.cuh -- host launcher template of the warp-specialized GEMM:
// tensor maps, kernel arguments, grid size, launch.  Included by the two
// translation units that instantiate the dense and the grouped variants.
#pragma once
#include "gemm_ws.cuh"
#include "wst_host.h"

namespace wst {

namespace {

constexpr int kBN = 256;
constexpr int kStages = 4;

template <bool OUT_F32, int EPI, bool GROUPED>
int launch_cfg(const GemmProblem& pr, const DeviceInfo& dev, cudaStream_t stream) {
  constexpr int EW = EPI == 2 ? 8 : 4;
  using Cfg = GemmCfg<kBN, kStages, EW, OUT_F32, EPI, GROUPED>;
  auto kern = k_gemm_ws<kBN, kStages, EW, OUT_F32, EPI, GROUPED>;

  // ---- tensor maps
  CUtensorMap tmA, tmB, tmC;
  GemmArgs a{};
  const CUtensorMapDataType out_dt =
      OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t es = OUT_F32 ? 4 : 2;
  const uint32_t cw = OUT_F32 ? 32 : 64;
  int st;
  if (!GROUPED) {
    a.a3d = (pr.batch > 1 && pr.strideA != 0);
    a.b3d = (pr.batch > 1 && pr.strideB != 0);
    a.c3d = (pr.batch > 1);
    {
      uint64_t dims[3] = {(uint64_t)pr.K, (uint64_t)pr.M, (uint64_t)pr.batch};
      uint64_t str[2] = {(uint64_t)pr.lda * 2, (uint64_t)pr.strideA * 2};
      uint32_t box[3] = {64, 128, 1};
      if ((st = encode_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.a3d ? 3 : 2, pr.A, dims, str,
                           box, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    }
    {
      uint64_t dims[3] = {(uint64_t)pr.K, (uint64_t)pr.N, (uint64_t)pr.batch};
      uint64_t str[2] = {(uint64_t)pr.ldb * 2, (uint64_t)pr.strideB * 2};
      uint32_t box[3] = {64, (uint32_t)kBN, 1};
      if ((st = encode_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.b3d ? 3 : 2, pr.B, dims, str,
                           box, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    }
    {
      uint64_t dims[3] = {(uint64_t)pr.N, (uint64_t)pr.M, (uint64_t)pr.batch};
      uint64_t str[2] = {(uint64_t)pr.ldc * es, (uint64_t)pr.strideC * es};
      uint32_t box[3] = {cw, 32, 1};
      if ((st = encode_map(&tmC, out_dt, a.c3d ? 3 : 2, pr.C, dims, str, box,
                           CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    }
  } else {
    a.a3d = 0;
    a.b3d = pr.strideB != 0;
    a.c3d = 0;
    {
      uint64_t dims[2] = {(uint64_t)pr.K, (uint64_t)(pr.M > 0 ? pr.M : 1)};
      uint64_t str[1] = {(uint64_t)pr.lda * 2};
      uint32_t box[2] = {64, 128};
      if ((st = encode_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pr.A, dims, str, box,
                           CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    }
    {
      uint64_t dims[3] = {(uint64_t)pr.K, (uint64_t)pr.N, (uint64_t)pr.batch};
      uint64_t str[2] = {(uint64_t)pr.ldb * 2, (uint64_t)pr.strideB * 2};
      uint32_t box[3] = {64, (uint32_t)kBN, 1};
      if ((st = encode_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.b3d ? 3 : 2, pr.B, dims, str,
                           box, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    }
    {
      uint64_t dims[2] = {(uint64_t)pr.N, (uint64_t)(pr.M > 0 ? pr.M : 1)};
      uint64_t str[1] = {(uint64_t)pr.ldc * es};
      uint32_t box[2] = {cw, 32};
      if ((st = encode_map(&tmC, out_dt, 2, pr.C, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    }
  }

  // ---- arguments
  a.batch = pr.batch;
  a.M = pr.M;
  a.N = pr.N;
  a.K = pr.K;
  a.m_tiles = (pr.M + kBM - 1) / kBM;
  a.n_tiles = (pr.N + kBN - 1) / kBN;
  a.k_blocks = (pr.K + kBK - 1) / kBK;
  a.tiles_total = GROUPED ? 0 : (long long)pr.batch * a.m_tiles * a.n_tiles;
  a.group_m = 16;
  a.bias = static_cast<const __nv_bfloat16*>(pr.bias);
  a.bias_stride = pr.strideBias;
  a.C = pr.C;
  a.ldc = pr.ldc;
  a.offsets = pr.offsets;
  a.G = GROUPED ? pr.batch : 0;
  a.M_total = pr.M;
  a.ws = static_cast<WsHeader*>(pr.ws);
  a.timeout_ns = wait_timeout_ns();

  long long grid = dev.num_sms;
  if (!GROUPED && a.tiles_total < grid) grid = a.tiles_total;
  if (grid < 1) grid = 1;

  // ---- launch
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Cfg::kSmemBytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(gemm)");
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, a);
  if (e != cudaSuccess) return cuda_fail(e, "launch k_gemm_ws");
  return ST_OK;
}

template <bool GROUPED>
int dispatch(const GemmProblem& pr, const DeviceInfo& dev, cudaStream_t s) {
  if (pr.c_f32) {
    switch (pr.epi) {
      case 0: return launch_cfg<true, 0, GROUPED>(pr, dev, s);
      case 1: return launch_cfg<true, 1, GROUPED>(pr, dev, s);
      default: return launch_cfg<true, 2, GROUPED>(pr, dev, s);
    }
  }
  switch (pr.epi) {
    case 0: return launch_cfg<false, 0, GROUPED>(pr, dev, s);
    case 1: return launch_cfg<false, 1, GROUPED>(pr, dev, s);
    default: return launch_cfg<false, 2, GROUPED>(pr, dev, s);
  }
}

}  // namespace

}  // namespace wst
