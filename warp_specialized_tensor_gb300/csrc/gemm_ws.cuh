// gemm_ws.cuh -- persistent, warp-specialized bf16 GEMM for sm_103a.
//
// Dense / strided-batched GEMM.  Per CTA (one per SM, persistent; with
// CG = 2 a cluster of two CTAs shares one 256 x BN tile):
//
//   warp 0      TMA producer: one thread streams A and B K-blocks (64 bf16 =
//               128 B rows, 128-byte swizzle) into a STAGES-deep shared-memory
//               ring; full[s] carries the transaction bytes, empty[s] is
//               released by the MMA completion.
//   warp 1      MMA issuer: one thread issues tcgen05.mma (128 x BN x 16,
//               bf16 -> fp32) into one of two tensor-memory accumulators and
//               commits completion to empty[s] (ring slot free) and, after the
//               last K-block of a tile, to acc_full[a].
//   warp 2      allocates / frees the tensor memory (2 x BN columns).
//   warps 4..   epilogue: wait acc_full[a], tcgen05.ld 32 columns at a time,
//               optional bias / SiLU, fp32 -> bf16 (RNE) or fp32, stage in a
//               swizzled per-warp shared buffer and TMA-store it; then
//               release acc_empty[a].  Two accumulators let the epilogue of
//               tile i overlap the MMAs of tile i+1.
//
// This is the Blackwell matmul of "How We Built TLX: A Hardware-Native GPU
// Compiler for Production ML at Scale" (Meta Engineering), section
// "Introducing TLX" (producer / MMA / epilogue roles, NUM_STAGES ring with
// load and dot barriers, TMEM accumulator, use_acc = k > 0), made persistent
// ("TLX Provides a Building Block ...": one persistent kernel, ping-pong
// between consumers).
#pragma once

#include <type_traits>

#include "wst_common.cuh"

namespace wst {

constexpr int kBM = 128;     // tile rows (TMEM lanes)
constexpr int kBK = 64;      // K-block: 64 bf16 = one 128-byte swizzle row
constexpr int kUmmaK = 16;   // K per tcgen05.mma (kind::f16)

struct GemmArgs {
  int batch, M, N, K;
  int m_tiles, n_tiles, k_blocks;
  long long tiles_total;
  int group_m;            // raster: m-tiles per band
  int a3d, b3d, c3d;      // operand maps carry a batch / group coordinate
  const __nv_bfloat16* bias;
  long long bias_stride;
  void* C;                // for masked stores of partial tiles
  long long ldc;
  long long c_stride;     // batch stride of C in elements (dense batched)
  WsHeader* ws;
  unsigned long long timeout_ns;
  int inject_drop_load;   // test hook: CTA 0 skips its first K-block's loads
  float eps, inv_k;       // row normalisation (NORM kernels only)
  const float* colsum;    // LayerNorm: s[b][n] = sum_k B[b][n][k]
  long long colsum_stride;
  const float2* row_stats;   // NORM 3 / 4: (r, r*mu) of row m of batch b at [b * stride + m]
  long long row_stats_stride;
};

struct Tile {
  int b;        // batch entry
  int m0;       // first row
  int n0;       // first column
  int row_end;  // rows >= row_end are outside the problem
};

// --------------------------------------------------------------------------
// schedulers
// --------------------------------------------------------------------------
template <int BN, int TM>
__device__ __forceinline__ Tile dense_tile(const GemmArgs& p, long long t) {
  const long long per_batch = (long long)p.m_tiles * p.n_tiles;
  const int b = (int)(t / per_batch);
  const int r = (int)(t - (long long)b * per_batch);
  // Banded raster: group_m consecutive m-tiles sweep all n-tiles together,
  // so a wave of CTAs shares A rows and B columns in L2.
  const int band = p.group_m * p.n_tiles;
  const int bi = r / band;
  const int first_m = bi * p.group_m;
  const int rows = min(p.group_m, p.m_tiles - first_m);
  const int rr = r - bi * band;
  const int m = first_m + rr % rows;
  const int n = rr / rows;
  return Tile{b, m * TM, n * BN, p.M};
}

// --------------------------------------------------------------------------
// epilogue helpers
// --------------------------------------------------------------------------
// GELU(x) = x * Phi(x) (exact erf form; normcdff is the CUDA math library's
// standard normal distribution function).
__device__ __forceinline__ float gelu_f(float x) { return x * normcdff(x); }

__device__ __forceinline__ float silu_f(float x) {
  // x * sigmoid(x), sigmoid(x) = (1 + tanh(x / 2)) / 2: one special-function
  // instruction (tanh.approx) instead of two (exponential and reciprocal).
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * x));
  return x * fmaf(0.5f, t, 0.5f);
}

template <int EPI>
__device__ __forceinline__ void apply_bias_act(float (&v)[32], const __nv_bfloat16* bias_row,
                                               int col, int N) {
  if constexpr (EPI == 0) {
    return;
  } else {
    if (col + 32 <= N) {
      const uint4* bp = reinterpret_cast<const uint4*>(bias_row + col);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 w = __ldg(bp + q);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float2 f = __bfloat1622float2(h[e]);
          v[q * 8 + e * 2] += f.x;
          v[q * 8 + e * 2 + 1] += f.y;
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col + j < N) v[j] += __bfloat162float(bias_row[col + j]);
    }
    if constexpr (EPI == 2) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = silu_f(v[j]);
    }
    if constexpr (EPI == 3) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = gelu_f(v[j]);
    }
  }
}

// Packed fp32 pairs (one 64-bit register: low half = first element), for the
// row statistics: half the instructions of the scalar form, each lane rounded
// as its scalar operation.
__device__ __forceinline__ uint64_t f2_bf16x2(uint32_t w) {  // bf16 pair -> fp32 pair (exact)
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(w << 16), "r"(w & 0xffff0000u));
  return r;
}
__device__ __forceinline__ uint64_t f2_splat(float x) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ float f2_lo(uint64_t a) { return __uint_as_float((uint32_t)a); }
__device__ __forceinline__ float f2_hi(uint64_t a) { return __uint_as_float((uint32_t)(a >> 32)); }

// Row normalisation of 32 accumulator columns [col, col+32) of one row:
// RMSNorm v *= r; LayerNorm v = r*v - (r*mu)*s[n] (s the column sums of B, the
// same for every row: the warp's lanes read the same addresses).  The sums
// are read as float4: each batch's row of s is 16-byte aligned and padded to a
// multiple of 4 floats, and col is a multiple of 32.
template <int NORM>
__device__ __forceinline__ void apply_norm(float (&v)[32], float scale, float shift,
                                           const float* cs, int col, int N) {
  if constexpr (NORM == 1) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= scale;
  } else {
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
      const float4 s = col + j < N ? __ldg(reinterpret_cast<const float4*>(cs + col + j))
                                   : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      v[j] = fmaf(scale, v[j], -shift * s.x);
      v[j + 1] = fmaf(scale, v[j + 1], -shift * s.y);
      v[j + 2] = fmaf(scale, v[j + 2], -shift * s.z);
      v[j + 3] = fmaf(scale, v[j + 3], -shift * s.w);
    }
  }
}

// --------------------------------------------------------------------------
// the kernel
// --------------------------------------------------------------------------
// NORM: 0 none, 1 RMSNorm, 2 LayerNorm of the rows of A with the row
// statistics gathered in the kernel; 3 RMSNorm, 4 LayerNorm with them
// precomputed (GemmArgs::row_stats).
template <int BN, int STAGES, int EPI_WARPS, bool OUT_F32, int EPI, int CG, int NORM>
struct GemmCfg {
  static constexpr bool kInStats = NORM == 1 || NORM == 2;  // statistics from the ring
  static constexpr int kStatsWarps = kInStats ? 4 : 0;     // row sum-of-squares warps
  static constexpr int kThreads = 128 + 32 * EPI_WARPS + 32 * kStatsWarps;
  static constexpr int kTileM = kBM * CG;              // rows of one (cluster) tile
  static constexpr int kABytes = kBM * kBK * 2;        // 16 KB: this CTA's 128 rows
  static constexpr int kBRows = BN / CG;               // this CTA's share of the B tile
  static constexpr int kBBytes = kBRows * kBK * 2;     // 32 KB (1-CTA) / 16 KB (pair)
  static constexpr int kStageBytes = kABytes + kBBytes;  // per CTA
  static constexpr uint32_t kTxBytes = CG * kStageBytes;  // expected by the leader's full[s]
  // staging buffers per epilogue warp (one for LayerNorm: its row shifts take
  // the shared memory of the second)
  static constexpr int kStageBufs = EPI_WARPS == 4 && NORM != 2 ? 2 : 1;
  static constexpr int kStgBytes = 32 * 128;           // 32 rows x 128 B
  static constexpr int kColsPerChunk = OUT_F32 ? 32 : 64;
  static constexpr int kWarpCols = BN / (EPI_WARPS / 4);  // columns one epilogue warp drains
  static constexpr int kTmemCols = 2 * BN;
  // per-row scales (and LayerNorm shifts r*mu), 2 buffers each
  static constexpr int kScaleBytes = kInStats ? (NORM == 2 ? 4 : 2) * kBM * 4 : 0;
  static constexpr size_t kSmemBytes = (size_t)STAGES * kStageBytes +
                                       (size_t)EPI_WARPS * kStageBufs * kStgBytes + kScaleBytes +
                                       256 /*bars*/ + 1024 /*alignment slack*/;
  static_assert(kTmemCols <= 512, "tensor memory holds 512 columns");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(kWarpCols % kColsPerChunk == 0, "epilogue chunking");
  static_assert(CG == 1 || CG == 2, "CTA group of 1 or 2");
};

// NORM 1 / 2: C = epi(r[m] * (A.B^T)[m][n] (+ bias)), r[m] = 1/sqrt(mean_k
// A[m][k]^2 + eps) (LayerNorm: minus r[m] mu[m] s[n]).  Four extra "stats" warps read every A stage from the ring (each
// lane one row: eight 16-byte swizzled chunks per stage), accumulate the
// row's sum of squares in fp32, release the stage together with the MMA, and
// hand 1/sqrt(ss/K + eps) per row to the epilogue through a double-buffered
// shared array.  The norm costs no extra pass over A in HBM.  On a single
// CTA the stats warps read a stage as soon as it lands (full[s]), alongside
// the MMAs, and empty[s] needs both the MMA commit and the stats warps.  On
// a CTA pair they read it after the MMAs that use it: the MMA issuer's
// per-stage commit goes to consumed[s] (in both CTAs, by the commit's
// multicast) instead of empty[s], and the stats warps release empty[s] once
// they have read the stage.  (In a pair, both CTAs' loads complete on the
// leader's full[s], which the peer's warps cannot wait on; relaying full[s]
// to the peer with a thread's remote arrive per stage ran 2.6x slower on
// GB300.)  Every tile recomputes its rows' statistics, so across the N tiles
// of a row band the work repeats N / BN times; NORM 3 / 4 instead read r and
// r*mu per row from a buffer a separate pass over A filled (no stats warps,
// the plain GEMM's ring), which is faster once N spans several tiles.
//
// CG = 2: a cluster of two CTAs computes one 256 x BN tile with
// tcgen05.mma.cta_group::2 issued by the even CTA (the leader).  Each CTA
// loads its own 128 rows of A and its half of B's BN rows (no multicast);
// both CTAs' loads complete on the leader's full[s]; the leader's commits
// arrive on empty[s] / acc_full[a] in both CTAs; both epilogues arrive on the
// leader's acc_empty[a]; each CTA drains its own 128 accumulator rows.
template <int BN, int STAGES, int EPI_WARPS, bool OUT_F32, int EPI, int CG, int NORM>
__global__ void __launch_bounds__(128 + 32 * EPI_WARPS + ((NORM == 1 || NORM == 2) ? 128 : 0), 1)
    k_gemm_ws(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmC, const GemmArgs p) {
  using Cfg = GemmCfg<BN, STAGES, EPI_WARPS, OUT_F32, EPI, CG, NORM>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smem + STAGES * Cfg::kABytes;
  uint8_t* smStg = smB + STAGES * Cfg::kBBytes;
  float* row_scale = reinterpret_cast<float*>(smStg + EPI_WARPS * Cfg::kStageBufs * Cfg::kStgBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(row_scale) + Cfg::kScaleBytes);
  // bars: full[STAGES] | empty[STAGES] | acc_full[2] | acc_empty[2] | scale_full[2] | scale_empty[2]
  //       | consumed[STAGES] (NORM)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 8);
  static_assert((3 * STAGES + 8) * 8 + 8 <= 256, "barrier area");
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t bar_base = smem_addr(bars);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto accf_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + a); };
  auto acce_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 2 + a); };
  auto sclf_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 4 + a); };
  auto scle_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 6 + a); };
  auto cons_bar = [&](int s) { return bar_base + 8u * (2 * STAGES + 8 + s); };
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;   // CTA rank in the pair
  const long long cluster_id = blockIdx.x / CG;
  const long long num_clusters = gridDim.x / CG;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      // released by the MMA commit; with the row statistics, on CTA pairs
      // by the stats warps, which wait for the MMA commit on consumed[s],
      // and on single CTAs by both (the stats warps read the stage as soon
      // as it lands, alongside the MMAs)
      mbar_init(empty_bar(s), !Cfg::kInStats ? 1 : (CG == 1 ? 1 + Cfg::kStatsWarps : Cfg::kStatsWarps));
      mbar_init(cons_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), CG * EPI_WARPS);
      mbar_init(sclf_bar(a), 4);
      mbar_init(scle_bar(a), EPI_WARPS);
    }
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 2) {
    tmem_alloc<CG>(smem_addr(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish<CG>();
  }
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // peer barriers initialised before any remote arrive
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const Guard guard{p.ws, abort_flag, p.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (long long t = cluster_id; ok && t < p.tiles_total; t += num_clusters) {
        const Tile tl = dense_tile<BN, Cfg::kTileM>(p, t);
        const int a_row = tl.m0 + (int)rank * kBM;
        const int b_row = tl.n0 + (int)rank * Cfg::kBRows;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          const bool got = CG == 2
              ? wait_phase_cluster(guard, empty_bar(stage), phase ^ 1u, (kRoleProducer << 16) | stage)
              : wait_phase(guard, empty_bar(stage), phase ^ 1u, (kRoleProducer << 16) | stage);
          if (!got) {
            ok = false;
            break;
          }
          if (p.inject_drop_load && blockIdx.x == 0 && t == cluster_id && kb == 0) {
            // Fault-injection test hook: leave this slot's full barrier
            // unarmed and unfilled, so the MMA issuer's bounded wait runs out.
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            continue;
          }
          // The leader's full[s] expects both CTAs' bytes; the peer only
          // contributes its copies' completions.
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), Cfg::kTxBytes);
          const uint32_t dA = smem_addr(smA + stage * Cfg::kABytes);
          const uint32_t dB = smem_addr(smB + stage * Cfg::kBBytes);
          const int kx = kb * kBK;
          if constexpr (CG == 1) {
            if (p.a3d) tma_load_3d(dA, &tmA, full_bar(stage), kx, a_row, tl.b);
            else       tma_load_2d(dA, &tmA, full_bar(stage), kx, a_row);
            if (p.b3d) tma_load_3d(dB, &tmB, full_bar(stage), kx, b_row, tl.b);
            else       tma_load_2d(dB, &tmB, full_bar(stage), kx, b_row);
          } else {
            const uint32_t fb = map_to_cta(full_bar(stage), 0);
            if (p.a3d) tma_load_3d_pair(dA, &tmA, fb, kx, a_row, tl.b);
            else       tma_load_2d_pair(dA, &tmA, fb, kx, a_row);
            if (p.b3d) tma_load_3d_pair(dB, &tmB, fb, kx, b_row, tl.b);
            else       tma_load_2d_pair(dB, &tmB, fb, kx, b_row);
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // Drain: every slot released => every MMA that read the ring completed.
      for (int i = 0; i < STAGES && ok; ++i) {
        ok = CG == 2
            ? wait_phase_cluster(guard, empty_bar(stage), phase ^ 1u, (kRoleProducer << 16) | 0x100 | stage)
            : wait_phase(guard, empty_bar(stage), phase ^ 1u, (kRoleProducer << 16) | 0x100 | stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // Only the leader CTA of a pair issues MMAs (for both CTAs).
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(Cfg::kTileM, BN, false, false);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (long long t = cluster_id; ok && t < p.tiles_total; t += num_clusters) {
        const bool free_acc = CG == 2
            ? wait_phase_cluster(guard, acce_bar(acc), acc_phase ^ 1u, (kRoleMma << 16) | 0x100 | acc)
            : wait_phase(guard, acce_bar(acc), acc_phase ^ 1u, (kRoleMma << 16) | 0x100 | acc);
        if (!free_acc) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_phase(guard, full_bar(stage), phase, (kRoleMma << 16) | stage)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t aBase = smem_addr(smA + stage * Cfg::kABytes);
          const uint32_t bBase = smem_addr(smB + stage * Cfg::kBBytes);
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            const uint64_t ad = sdesc_sw128(aBase + k * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(bBase + k * 32, 16, 1024);
            umma_bf16<CG>(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          // slot free (in both CTAs) once these MMAs finish; with the row
          // statistics, once the stats warps have read it too (on a pair,
          // after these MMAs)
          const uint32_t rel = (Cfg::kInStats && CG == 2) ? cons_bar(stage) : empty_bar(stage);
          if constexpr (CG == 1) umma_commit(rel);
          else                   umma_commit_pair(rel, 0x3);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        // accumulator complete (in both CTAs)
        if constexpr (CG == 1) umma_commit(accf_bar(acc));
        else                   umma_commit_pair(accf_bar(acc), 0x3);
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
    }
  } else if (Cfg::kInStats && warp >= 4 + EPI_WARPS) {
    // ------------------------------------------------------------------ row statistics
    const int r = (warp - 4 - EPI_WARPS) * 32 + (int)lane;  // CTA-local row of A
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (long long t = cluster_id; ok && t < p.tiles_total; t += num_clusters) {
      // RMSNorm: ss = sum a^2.  LayerNorm: sums of d = a - c and d^2 about a
      // shift c, the row's first element (the "shifted data" one-pass
      // variance of Chan, Golub and LeVeque, "Algorithms for computing the
      // sample variance: analysis and recommendations", The American
      // Statistician 37(3), 1983): var = E[d^2] - E[d]^2 cancels only as
      // much as (c - mu)^2 / var, which is small because c is a value of the
      // row, where the unshifted E[a^2] - mu^2 cancels mu^2 / var.
      // The sums are kept as packed pairs (even and odd K positions); the
      // halves are added at the end.
      // four independent accumulator pairs (the e-th 4-byte word of each
      // 16-byte chunk), so the adds do not form one long dependency chain
      uint64_t ss2[4] = {0, 0, 0, 0}, sm2[4] = {0, 0, 0, 0};
      float c = 0.0f;
      uint64_t negc2 = 0;
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        // On a pair: the MMAs that read this stage completed (their commit,
        // multicast to both CTAs, arrives on consumed[s]; the peer cannot
        // wait on the leader's full[s]).  On a single CTA: the stage landed.
        const uint32_t ready = CG == 2 ? cons_bar(stage) : full_bar(stage);
        // Every lane waits (and so acquires the copies' data) itself: one
        // round of barrier latency per stage instead of lane 0's wait
        // followed by the other lanes' acquire.
        bool got = CG == 2 ? wait_phase_cluster(guard, ready, phase, (kRoleEpilogue << 16) | 0x400 | stage)
                           : wait_phase(guard, ready, phase, (kRoleEpilogue << 16) | 0x400 | stage);
        got = __all_sync(0xffffffffu, got);
        if (!got) {
          ok = false;
          break;
        }
        const uint32_t row_addr = smem_addr(smA + stage * Cfg::kABytes) + (uint32_t)r * 128u;
        if constexpr (NORM == 2) {
          if (kb == 0) {
            // element k = 0 of the row: the first two bytes of logical
            // 16-byte chunk 0, stored at chunk (0 ^ (r & 7)) by the swizzle
            uint32_t w;
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w) : "r"(row_addr + ((uint32_t)(r & 7) << 4)));
            c = __uint_as_float(w << 16);
            negc2 = f2_splat(-c);
          }
        }
        // K positions past K in the last block are zero-filled by the copy;
        // LayerNorm's shifted sums must skip them (they would add -c and c^2)
        const int kvalid = p.K - kb * kBK;
        auto accumulate = [&](auto masked) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint32_t w0, w1, w2, w3;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                         : "r"(row_addr + ((uint32_t)(j ^ (r & 7)) << 4)));
            const uint32_t w[4] = {w0, w1, w2, w3};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint64_t f2 = f2_bf16x2(w[e]);
              if constexpr (NORM == 1) {
                ss2[e] = f2_fma(f2, f2, ss2[e]);
              } else {
                uint64_t d2 = f2_add(f2, negc2);
                if constexpr (decltype(masked)::value) {
                  const float dx = 8 * j + 2 * e < kvalid ? f2_lo(d2) : 0.0f;
                  const float dy = 8 * j + 2 * e + 1 < kvalid ? f2_hi(d2) : 0.0f;
                  asm("mov.b64 %0, {%1, %2};" : "=l"(d2) : "f"(dx), "f"(dy));
                }
                ss2[e] = f2_fma(d2, d2, ss2[e]);
                sm2[e] = f2_add(sm2[e], d2);
              }
            }
          }
        };
        if (NORM == 2 && kvalid < kBK) accumulate(std::true_type{});
        else                           accumulate(std::false_type{});
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(stage));
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (!warp_wait_phase(guard, scle_bar(acc), acc_phase ^ 1u, (kRoleEpilogue << 16) | 0x500 | acc)) break;
      const uint64_t ss_a = f2_add(f2_add(ss2[0], ss2[1]), f2_add(ss2[2], ss2[3]));
      const float ss = f2_lo(ss_a) + f2_hi(ss_a);
      if constexpr (NORM == 1) {
        row_scale[acc * kBM + r] = rsqrtf(ss * p.inv_k + p.eps);
      } else {
        const uint64_t sm_a = f2_add(f2_add(sm2[0], sm2[1]), f2_add(sm2[2], sm2[3]));
        const float sm = f2_lo(sm_a) + f2_hi(sm_a);
        // LayerNorm: mean = c + E[d], biased variance = E[d^2] - E[d]^2
        // (fp32, clamped at 0)
        const float dm = sm * p.inv_k;
        const float mu = c + dm;
        const float rs = rsqrtf(fmaxf(ss * p.inv_k - dm * dm, 0.0f) + p.eps);
        row_scale[acc * kBM + r] = rs;
        row_scale[2 * kBM + acc * kBM + r] = rs * mu;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(sclf_bar(acc));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ epilogue
    const int ew = warp - 4;              // 0 .. EPI_WARPS-1
    const int q = warp & 3;               // TMEM lane quadrant this warp may access
    const int col_begin = (ew >> 2) * Cfg::kWarpCols;
    uint8_t* stg = smStg + ew * Cfg::kStageBufs * Cfg::kStgBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    int buf = 0;
    for (long long t = cluster_id; t < p.tiles_total; t += num_clusters) {
      const Tile tl = dense_tile<BN, Cfg::kTileM>(p, t);
      const bool got = CG == 2
          ? warp_wait_phase_cluster(guard, accf_bar(acc), acc_phase, (kRoleEpilogue << 16) | acc)
          : warp_wait_phase(guard, accf_bar(acc), acc_phase, (kRoleEpilogue << 16) | acc);
      if (!got) break;
      tc_fence_after_sync();

      // first row this warp drains (this CTA holds rows rank*128 .. +127 of the tile)
      const int row_base = tl.m0 + (int)rank * kBM + q * 32;
      const int row = row_base + (int)lane;
      const bool full_rows = row_base + 32 <= tl.row_end;
      const __nv_bfloat16* bias_row =
          EPI ? p.bias + (long long)tl.b * p.bias_stride : nullptr;
      const float* cs_row = (NORM == 2 || NORM == 4) ? p.colsum + (long long)tl.b * p.colsum_stride : nullptr;
      const uint32_t t_lane = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      float scale = 1.0f, shift = 0.0f;
      if constexpr (NORM >= 3) {
        // precomputed statistics of this lane's row
        if (row < tl.row_end) {
          const float2 rs = __ldg(p.row_stats + (long long)tl.b * p.row_stats_stride + row);
          scale = rs.x;
          shift = rs.y;
        }
      } else if constexpr (NORM) {
        if (!warp_wait_phase(guard, sclf_bar(acc), acc_phase, (kRoleEpilogue << 16) | 0x600 | acc)) break;
        (void)mbar_try_wait(sclf_bar(acc), acc_phase);
        scale = row_scale[acc * kBM + q * 32 + (int)lane];
        if constexpr (NORM == 2) shift = row_scale[2 * kBM + acc * kBM + q * 32 + (int)lane];
        __syncwarp();
        if (lane == 0) mbar_arrive(scle_bar(acc));
      }

#pragma unroll 1
      for (int c0 = col_begin; c0 < col_begin + Cfg::kWarpCols; c0 += Cfg::kColsPerChunk) {
        float v0[32];
        tmem_load32(t_lane + c0, v0);
        if constexpr (NORM) apply_norm<(NORM == 2 || NORM == 4) ? 2 : 1>(v0, scale, shift, cs_row, tl.n0 + c0, p.N);
        apply_bias_act<EPI>(v0, bias_row, tl.n0 + c0, p.N);
        uint32_t packed[16];
        float v1[32];
        if constexpr (!OUT_F32) {
          tmem_load32(t_lane + c0 + 32, v1);
          if constexpr (NORM) apply_norm<(NORM == 2 || NORM == 4) ? 2 : 1>(v1, scale, shift, cs_row, tl.n0 + c0 + 32, p.N);
          apply_bias_act<EPI>(v1, bias_row, tl.n0 + c0 + 32, p.N);
#pragma unroll
          for (int j = 0; j < 16; ++j) packed[j] = pack_bf16x2(v0[2 * j], v0[2 * j + 1]);
        }
        // Chunks that start past the last row / column store nothing (a TMA
        // store is never issued at an out-of-range start coordinate).
        // A TMA store clips the innermost dimension only at 16-byte
        // granularity, so chunks that cross the last column (or the last
        // row) use masked direct stores instead.
        const bool chunk_live = row_base < tl.row_end && tl.n0 + c0 < p.N;
        if (!chunk_live) {
          // nothing to store
        } else if (full_rows && tl.n0 + c0 + Cfg::kColsPerChunk <= p.N) {
          // Stage the 32 x 128 B block (128-byte swizzle) and TMA-store it.
          uint8_t* sb = stg + buf * Cfg::kStgBytes;
          if (Cfg::kStageBufs == 2) {
            if (lane == 0) bulk_wait_group_read<1>();
          } else {
            if (lane == 0) bulk_wait_group_read<0>();
          }
          __syncwarp();
          const uint32_t row_addr = smem_addr(sb) + lane * 128u;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t dst = row_addr + ((uint32_t)(j ^ (lane & 7)) << 4);
            if constexpr (OUT_F32) {
              st_shared_v4(dst, __float_as_uint(v0[4 * j]), __float_as_uint(v0[4 * j + 1]),
                           __float_as_uint(v0[4 * j + 2]), __float_as_uint(v0[4 * j + 3]));
            } else {
              uint32_t w0, w1, w2, w3;
              if (j < 4) {
                w0 = packed[4 * j]; w1 = packed[4 * j + 1]; w2 = packed[4 * j + 2]; w3 = packed[4 * j + 3];
              } else {
                const int jj = j - 4;
                w0 = pack_bf16x2(v1[8 * jj], v1[8 * jj + 1]);
                w1 = pack_bf16x2(v1[8 * jj + 2], v1[8 * jj + 3]);
                w2 = pack_bf16x2(v1[8 * jj + 4], v1[8 * jj + 5]);
                w3 = pack_bf16x2(v1[8 * jj + 6], v1[8 * jj + 7]);
              }
              st_shared_v4(dst, w0, w1, w2, w3);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (p.c3d) tma_store_3d(&tmC, smem_addr(sb), tl.n0 + c0, row_base, tl.b);
            else       tma_store_2d(&tmC, smem_addr(sb), tl.n0 + c0, row_base);
            bulk_commit_group();
          }
          if (Cfg::kStageBufs == 2) buf ^= 1;
        } else if (row < tl.row_end) {
          // Partial tile: rows past M and columns past N must not be
          // written.  Masked stores.
          const int colg = tl.n0 + c0;
          const long long row_off = (long long)tl.b * p.c_stride + (long long)row * p.ldc;
          if constexpr (OUT_F32) {
            float* crow = reinterpret_cast<float*>(p.C) + row_off;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int cc = colg + 4 * j;
              if (cc + 4 <= p.N) {
                *reinterpret_cast<float4*>(crow + cc) =
                    make_float4(v0[4 * j], v0[4 * j + 1], v0[4 * j + 2], v0[4 * j + 3]);
              } else {
                for (int e = 0; e < 4; ++e)
                  if (cc + e < p.N) crow[cc + e] = v0[4 * j + e];
              }
            }
          } else {
            __nv_bfloat16* crow = reinterpret_cast<__nv_bfloat16*>(p.C) + row_off;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int cc = colg + 8 * j;
              const float* src = j < 4 ? &v0[8 * j] : &v1[8 * (j - 4)];
              if (cc + 8 <= p.N) {
                uint4 w;
                w.x = pack_bf16x2(src[0], src[1]);
                w.y = pack_bf16x2(src[2], src[3]);
                w.z = pack_bf16x2(src[4], src[5]);
                w.w = pack_bf16x2(src[6], src[7]);
                *reinterpret_cast<uint4*>(crow + cc) = w;
              } else {
                for (int e = 0; e < 8; ++e)
                  if (cc + e < p.N) crow[cc + e] = __float2bfloat16_rn(src[e]);
              }
            }
          }
        }
      }
      // All TMEM reads of this accumulator are complete (waited in tmem_load32).
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 1) mbar_arrive(acce_bar(acc));
        else                   mbar_arrive_cluster(map_to_cta(acce_bar(acc), 0));
      }
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (*abort_flag) {
    // Give any copy or MMA still in flight time to land before the shared
    // memory and tensor memory are released (bounded: ~200 us).
    for (int i = 0; i < 200; ++i) __nanosleep(1000);
  }
  // No CTA of a pair leaves while its peer may still arrive on its barriers.
  if constexpr (CG == 2) cluster_sync();
  tc_fence_after_sync();
  if (warp == 2) tmem_dealloc<CG>(tmem_base, Cfg::kTmemCols);
}

}  // namespace wst
