// gemm_dense.cu -- instantiations and launcher of the warp-specialized dense /
// strided-batched GEMM: tensor maps, kernel arguments, grid size, launch.
#include <cstdlib>

#include "gemm_ws.cuh"
#include "wst_host.h"

namespace wst {

namespace {

constexpr int kBN = 256;

// Ring depth: 4 x 48 KB (1-CTA tile) or 6 x 32 KB per CTA (2-CTA pair).
template <int CG>
constexpr int stages_for() { return CG == 2 ? 6 : 4; }

// CTA-pair tiles for dense problems with more than one 128-row block and
// more than 8 K-blocks, unless the process-wide option
// WST_OPT_DENSE_CTA_GROUP forces a choice.  With 8 K-blocks or fewer the
// pair's per-tile coupling (the leader's MMAs wait for both CTAs' loads,
// both epilogues release the accumulator) outweighs the halved B traffic:
// measured on GB300 with bias + SiLU, 512 x (1024 x 256 x 512) ran 0.148 ms
// on single CTAs against 0.178 ms on pairs, while from K = 1024 up pairs
// won (256 x (1024 x 256 x 1024): 0.129 vs 0.136 ms; 8192^3: 0.612 vs
// 0.691 ms).
inline int dense_cta_group(int M, int K) {
  const int forced = option_value(OPT_DENSE_CTA_GROUP);
  if (forced == 1 || forced == 2) return forced;
  return M > kBM && K > 8 * kBK ? 2 : 1;
}

template <bool OUT_F32, int EPI, int CG, int NORM>
int launch_cfg(const GemmProblem& pr, const DeviceInfo& dev, cudaStream_t stream) {
  // 8 epilogue warps for SiLU / GELU (special-function heavy), except with
  // the row-statistics warps, where 4 keep the block at 384 threads.
  constexpr int EW = (EPI >= 2 && NORM != 1 && NORM != 2) ? 8 : 4;
  constexpr int kStages = stages_for<CG>();
  using Cfg = GemmCfg<kBN, kStages, EW, OUT_F32, EPI, CG, NORM>;
  auto kern = k_gemm_ws<kBN, kStages, EW, OUT_F32, EPI, CG, NORM>;

  // ---- tensor maps
  CUtensorMap tmA, tmB, tmC;
  GemmArgs a{};
  const CUtensorMapDataType out_dt =
      OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t es = OUT_F32 ? 4 : 2;
  const uint32_t cw = OUT_F32 ? 32 : 64;
  int st;
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
    uint32_t box[3] = {64, (uint32_t)Cfg::kBRows, 1};
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

  // ---- arguments
  a.batch = pr.batch;
  a.M = pr.M;
  a.N = pr.N;
  a.K = pr.K;
  a.m_tiles = (pr.M + Cfg::kTileM - 1) / Cfg::kTileM;
  a.n_tiles = (pr.N + kBN - 1) / kBN;
  a.k_blocks = (pr.K + kBK - 1) / kBK;
  a.tiles_total = (long long)pr.batch * a.m_tiles * a.n_tiles;
  // Raster bands of 8 m-tiles: at 8192^3 on GB300 bands of 8 read 1.08 GB
  // from DRAM per launch against 1.26 GB for 16, 1.42 GB for 4 and 2.07 GB
  // for 32 (L2 hit 77 / 73 / 72 / 65 %), and over 100 back-to-back calls,
  // where the power cap sets the clock, ran 0.660 vs 0.672 / 0.682 / 0.698 ms.
  a.group_m = 8;
  a.bias = static_cast<const __nv_bfloat16*>(pr.bias);
  a.bias_stride = pr.strideBias;
  a.C = pr.C;
  a.ldc = pr.ldc;
  a.c_stride = pr.strideC;
  a.ws = static_cast<WsHeader*>(pr.ws);
  a.timeout_ns = wait_timeout_ns();
  a.inject_drop_load = take_fault_injection() ? 1 : 0;
  a.eps = pr.eps;
  a.inv_k = 1.0f / (float)pr.K;
  a.colsum = pr.colsum;
  a.colsum_stride = pr.colsum_stride;
  a.row_stats = pr.row_stats;
  a.row_stats_stride = pr.row_stats_stride;

  // Persistent grid: one CTA (pair) per SM (pair) that can be resident.
  long long grid = dev.num_sms;
  if (CG == 2) {
    static int max_clusters[64] = {0};
    int& mc = max_clusters[dev.device & 63];
    if (mc == 0) {
      cudaLaunchConfig_t q{};
      q.gridDim = dim3((unsigned)(dev.num_sms & ~1), 1, 1);
      q.blockDim = dim3(Cfg::kThreads, 1, 1);
      q.dynamicSmemBytes = Cfg::kSmemBytes;
      cudaLaunchAttribute ca[1];
      ca[0].id = cudaLaunchAttributeClusterDimension;
      ca[0].val.clusterDim.x = 2;
      ca[0].val.clusterDim.y = 1;
      ca[0].val.clusterDim.z = 1;
      q.attrs = ca;
      q.numAttrs = 1;
      if ((st = ensure_smem_attr((const void*)kern, Cfg::kSmemBytes))) return st;
      cudaError_t qe;
      int n = 0;
      qe = cudaOccupancyMaxActiveClusters(&n, kern, &q);
      if (qe != cudaSuccess || n < 1) {
        cudaGetLastError();
        n = dev.num_sms / 2;
      }
      mc = n;
    }
    grid = 2ll * mc;
  }
  if (a.tiles_total * CG < grid) grid = a.tiles_total * CG;
  if (grid < CG) grid = CG;

  // ---- launch
  if ((st = ensure_smem_attr((const void*)kern, Cfg::kSmemBytes))) return st;
  cudaError_t e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CG == 2 ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, a);
  if (e != cudaSuccess) return cuda_fail(e, "launch k_gemm_ws");
  return ST_OK;
}

template <int CG, int NORM>
int dispatch(const GemmProblem& pr, const DeviceInfo& dev, cudaStream_t s) {
  if (pr.c_f32) {
    switch (pr.epi) {
      case 0: return launch_cfg<true, 0, CG, NORM>(pr, dev, s);
      case 1: return launch_cfg<true, 1, CG, NORM>(pr, dev, s);
      case 2: return launch_cfg<true, 2, CG, NORM>(pr, dev, s);
      default: return launch_cfg<true, 3, CG, NORM>(pr, dev, s);
    }
  }
  switch (pr.epi) {
    case 0: return launch_cfg<false, 0, CG, NORM>(pr, dev, s);
    case 1: return launch_cfg<false, 1, CG, NORM>(pr, dev, s);
    case 2: return launch_cfg<false, 2, CG, NORM>(pr, dev, s);
    default: return launch_cfg<false, 3, CG, NORM>(pr, dev, s);
  }
}

}  // namespace

int run_gemm_grouped(const GemmProblem& pr, const DeviceInfo& dev, cudaStream_t stream);

namespace {

// The passes over rows of bf16 data ahead of the norm GEMMs, in one launch
// and one warp per row: the row statistics of A (the first ceil(rows_a / 8)
// blocks) and the column sums s[n] = sum_k B[n][k] of B (the rest).
// Statistics: RMSNorm r = 1/sqrt(mean a^2 + eps), shift 0; LayerNorm the
// sums of d = a - c and d^2 about the row's first element c, mu = c + E[d],
// var = E[d^2] - E[d]^2 (clamped at 0), r = 1/sqrt(var + eps), shift r*mu,
// the same formulas as the GEMM's statistics warps.  Rows start 16-byte
// aligned (the operands and their strides are); each lane keeps eight
// 16-byte loads in flight (a row of 8192 bf16 is four rounds), then a
// scalar tail and a warp reduction.
struct NormPassArgs {
  const __nv_bfloat16* A;
  long long lda, strideA;
  int M, K, rows_a;
  float eps;
  float2* stats;
  const __nv_bfloat16* B;
  long long ldb, strideB;
  int N, rows_b;
  long long colsum_stride;
  float* colsum;
};

// Calls f(w) for every 16-byte chunk of the row's first K & ~7 elements
// that falls to this lane, eight loads at a time, and returns where the
// scalar tail starts.
template <class F>
__device__ __forceinline__ int sweep_row(const __nv_bfloat16* row, int K, int lane, F&& f) {
  const int kv = K & ~7;
  int k = lane * 8;
  for (; k + 7 * 256 < kv; k += 8 * 256) {
    uint4 w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) w[u] = __ldg(reinterpret_cast<const uint4*>(row + k + u * 256));
#pragma unroll
    for (int u = 0; u < 8; ++u) f(w[u]);
  }
  for (; k < kv; k += 256) f(__ldg(reinterpret_cast<const uint4*>(row + k)));
  return kv;
}

template <bool LN>
__global__ void __launch_bounds__(256) k_norm_pass(const NormPassArgs a) {
  const int lane = (int)(threadIdx.x & 31);
  const int blocks_a = (a.rows_a + 7) / 8;
  if ((int)blockIdx.x < blocks_a) {
    const int gw = (int)blockIdx.x * 8 + (int)(threadIdx.x >> 5);
    if (gw >= a.rows_a) return;
    const int b = gw / a.M, m = gw - b * a.M;
    const __nv_bfloat16* row = a.A + (long long)b * a.strideA + (long long)m * a.lda;
    const float c = LN ? __bfloat162float(row[0]) : 0.0f;
    float s1[4] = {0.0f, 0.0f, 0.0f, 0.0f}, s2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const int kv = sweep_row(row, a.K, lane, [&](const uint4& w) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        const float dx = f.x - c, dy = f.y - c;
        s2[e] = fmaf(dx, dx, fmaf(dy, dy, s2[e]));
        if (LN) s1[e] += dx + dy;
      }
    });
    for (int t = kv + lane; t < a.K; t += 32) {
      const float d = __bfloat162float(row[t]) - c;
      s2[0] = fmaf(d, d, s2[0]);
      if (LN) s1[0] += d;
    }
    float ss = (s2[0] + s2[1]) + (s2[2] + s2[3]);
    float sm = (s1[0] + s1[1]) + (s1[2] + s1[3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (LN) sm += __shfl_xor_sync(0xffffffffu, sm, o);
    }
    if (lane == 0) {
      const float inv_k = 1.0f / (float)a.K;
      if (LN) {
        const float dm = sm * inv_k;
        const float r = rsqrtf(fmaxf(ss * inv_k - dm * dm, 0.0f) + a.eps);
        a.stats[gw] = make_float2(r, r * (c + dm));
      } else {
        a.stats[gw] = make_float2(rsqrtf(ss * inv_k + a.eps), 0.0f);
      }
    }
  } else {
    const int gw = ((int)blockIdx.x - blocks_a) * 8 + (int)(threadIdx.x >> 5);
    if (gw >= a.rows_b) return;
    const int b = gw / a.N, n = gw - b * a.N;
    const __nv_bfloat16* row = a.B + (long long)b * a.strideB + (long long)n * a.ldb;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const int kv = sweep_row(row, a.K, lane, [&](const uint4& w) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        acc[e] += f.x + f.y;
      }
    });
    for (int t = kv + lane; t < a.K; t += 32) acc[0] += __bfloat162float(row[t]);
    float sum = (acc[0] + acc[1]) + (acc[2] + acc[3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    // each batch entry's sums start on a padded row (the epilogue reads
    // them as float4)
    if (lane == 0) a.colsum[(long long)b * a.colsum_stride + n] = sum;
  }
}

}  // namespace

int run_norm_pass(const NormPass& np, cudaStream_t stream) {
  const long long rows_a = np.stats ? (long long)np.nb_a * np.M : 0;
  const long long rows_b = np.colsum ? (long long)np.nb_b * np.N : 0;
  if (rows_a > 0x7fffffffLL || rows_b > 0x7fffffffLL) {
    set_error("norm GEMM: %lld rows of A / %lld rows of B exceed the statistics kernel's range",
              rows_a, rows_b);
    return ST_UNSUPPORTED;
  }
  if (rows_a + rows_b == 0) return ST_OK;
  NormPassArgs a{};
  a.A = static_cast<const __nv_bfloat16*>(np.A);
  a.lda = np.lda;
  a.strideA = np.strideA;
  a.M = np.M;
  a.K = np.K;
  a.rows_a = (int)rows_a;
  a.eps = np.eps;
  a.stats = np.stats;
  a.B = static_cast<const __nv_bfloat16*>(np.B);
  a.ldb = np.ldb;
  a.strideB = np.strideB;
  a.N = np.N;
  a.rows_b = (int)rows_b;
  a.colsum_stride = np.colsum_stride;
  a.colsum = np.colsum;
  const unsigned grid = (unsigned)((rows_a + 7) / 8 + (rows_b + 7) / 8);
  if (np.layernorm)
    k_norm_pass<true><<<grid, 256, 0, stream>>>(a);
  else
    k_norm_pass<false><<<grid, 256, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch k_norm_pass");
  return ST_OK;
}

int run_gemm(const GemmProblem& pr, cudaStream_t stream) {
  DeviceInfo dev;
  int st = current_device_info(&dev);
  if (st) return st;
  if (pr.grouped) return run_gemm_grouped(pr, dev, stream);
  const bool pair = dense_cta_group(pr.M, pr.K) == 2;
  if (pr.norm == 1) return pair ? dispatch<2, 1>(pr, dev, stream) : dispatch<1, 1>(pr, dev, stream);
  if (pr.norm == 2) return pair ? dispatch<2, 2>(pr, dev, stream) : dispatch<1, 2>(pr, dev, stream);
  if (pr.norm == 3) return pair ? dispatch<2, 3>(pr, dev, stream) : dispatch<1, 3>(pr, dev, stream);
  if (pr.norm == 4) return pair ? dispatch<2, 4>(pr, dev, stream) : dispatch<1, 4>(pr, dev, stream);
  return pair ? dispatch<2, 0>(pr, dev, stream) : dispatch<1, 0>(pr, dev, stream);
}

}  // namespace wst
