// grouped_ws.cuh -- persistent, warp-specialized grouped GEMM (mixture-of-
// experts expert matmuls) for sm_103a, on CTA pairs.
//
// Group g owns token rows [off[g], off[g+1]) of A and C and the weight matrix
// B[g] (N x K, K contiguous):   C[t][n] = sum_k A[t][k] * B[g][n][k].
//
// The tensor core computes the transposed tile  D[n][t] = B[g][n][:] . A[t][:]
// ("swap AB"): the expert's output features n sit on the 256-row MMA side
// (two CTAs x 128 TMEM lanes), and the tokens of the group sit on the MMA's N
// side, whose size is a multiple of 16 up to 256.  A group of T tokens is cut
// into 256-token tiles and one remainder tile rounded up to 16, so a ragged
// group wastes at most 15 token columns instead of up to 127 rows of a
// 128-row tile.  (Measured on GB300 against equal-width token tiles and
// against fetching token rows in 32-row boxes: both were slower than this
// layout, which fetches each CTA's token rows as one 128-row box.)  Both
// operands are K-major in memory, as the hardware wants.
//
// Roles per CTA (persistent, one CTA per SM, pairs in clusters of 2):
//   warp 0     TMA producer: this CTA's 128 rows of B[g] and its half of the
//              token tile (rows t0 + rank*Ntile/2 ...) per 64-wide K-block;
//              both CTAs' copies complete on the leader's full[s].
//   warp 1     MMA issuer (leader CTA only): tcgen05.mma.cta_group::2,
//              M = 256, N = token-tile width, into one of two TMEM
//              accumulators; commits release ring slots / accumulators in
//              both CTAs.
//   warp 2     TMEM allocation (both CTAs, 512 columns).
//   warp 3     lane 1 of CTA 0 validates the offsets; with the
//              cluster-launch-control schedule, lane 0 is the tile scheduler.
//   warps 4-7  epilogue: each warp drains its 32 feature lanes, 32 tokens at a
//              time, adds bias / SiLU / GELU and transposes through a private
//              double-buffered shared block; blocks of 32 tokens inside the
//              group leave through TMA stores, the group's last partial block
//              through masked vector stores of whole 64-byte (bf16) /
//              128-byte (fp32) row segments, so rows past the group end (the
//              next expert's tokens) are never touched.
//
// "How We Built TLX: A Hardware-Native GPU Compiler for Production ML at
// Scale" (Meta Engineering): "TLX in Production" and "Case Study 3:
// Distributed Grouped GEMM for LLM Pretraining" (grouped expert GEMM),
// "Introducing TLX" (producer / MMA / epilogue roles over an mbarrier ring).
#pragma once

#include "wst_common.cuh"

namespace wst {

constexpr int kGrpTileN = 256;   // feature rows per CTA pair (MMA M)
constexpr int kGrpTileT = 256;   // tokens per tile (MMA N, last tile of a group narrower)
constexpr int kGrpBK = 64;
constexpr int kGrpStages = 6;
constexpr int kGrpEpiWarps = 4;
constexpr int kGrpThreads = 128 + 32 * kGrpEpiWarps;
constexpr int kGrpWBytes = 128 * kGrpBK * 2;   // this CTA's 128 rows of B[g]
constexpr int kGrpXBytes = 128 * kGrpBK * 2;   // up to 128 token rows per CTA
// Tile schedule (template parameter CLC):
//  * static: the grid is one CTA pair per pair of SMs and pair c takes
//    tiles c, c + #pairs, ... (every role walks the same sequence);
//  * cluster launch control: the grid holds one pair per tile (an upper
//    bound: the group sizes live on the device) and pair c starts on tile c.
//    Warp 3 of the leader asks the hardware to cancel a pair that has not
//    been launched yet (clusterlaunchcontrol.try_cancel, response multicast
//    to both CTAs) and takes over its tile, until no pair is left to cancel
//    or the cancelled pair's tile lies past the last tile.  Each CTA's
//    scheduler lane hands the tiles to its own roles through a 2-slot
//    shared-memory queue, so a pair claims at most one tile ahead of the one
//    its tensor core is working on.  Pairs launched past the last tile
//    count the tiles and exit at once.
constexpr int kGrpTQ = 2;  // tile-queue slots
constexpr int kGrpXBoxRows = 128;              // token rows per TMA box (one box per CTA)
constexpr int kGrpXBoxBytes = kGrpXBoxRows * kGrpBK * 2;
// Thin token tiles (a group's remainder, at most 128 tokens: at most 64 rows
// per CTA) load only the rows they use, in 16-row boxes: their K loop is
// bound by the bytes each K-block moves, and a full 128-row token box would
// double them (measured on GB300: a thin tile costs its pair ~10 us, about
// half of a full tile, almost all of it streaming bytes it does not use).
constexpr int kGrpXThinRows = 16;
constexpr int kGrpXThinBytes = kGrpXThinRows * kGrpBK * 2;
constexpr int kGrpThinMaxRows = 64;            // per CTA
constexpr int kGrpStageBytes = kGrpWBytes + kGrpXBytes;
constexpr int kGrpStgBytes = 32 * 32 * 4;      // per-warp transpose buffer (fp32 worst case)
constexpr int kGrpStgBufs = 2;                 // double-buffered for the TMA stores
// Group offsets copied to shared memory at the start (problems of up to
// kGrpTabMax - 1 groups): walking the groups there instead of through
// dependent global loads keeps the tile boundaries short.
constexpr int kGrpTabMax = 256;
constexpr size_t kGrpSmemBytes = (size_t)kGrpStages * kGrpStageBytes +
                                 (size_t)kGrpEpiWarps * kGrpStgBufs * kGrpStgBytes +
                                 512 /*barriers, queue*/ + kGrpTabMax * 4 + 1024;
static_assert(kGrpSmemBytes <= 232448, "shared memory per CTA");

struct GroupedArgs {
  int G, M_total, N, K;
  int n_tiles, k_blocks;
  const int* offsets;  // device int32[G+1]
  const __nv_bfloat16* bias;
  long long bias_stride;
  void* C;
  long long ldc;
  int w_shared;        // 1: every group uses the same weight matrix (group stride 0)
  WsHeader* ws;
  unsigned long long timeout_ns;
};

struct GrpTile {
  int g;      // group
  int t0;     // first token row (absolute)
  int nt;     // valid tokens in this tile (1..256)
  int nmma;   // MMA N: nt rounded up to 16
  int n0;     // first feature row of B[g] / column of C
};

// Walks groups in order; every role of a CTA runs its own walker over the
// same increasing tile indices.  Offsets are clamped into [0, M_total].
struct GrpWalker {
  int g;
  long long base, count;
  int r0, r1, tt, sz;  // rows, token tiles, token-tile width
  const int* tab;      // the offsets in shared memory, or nullptr

  __device__ __forceinline__ void load(const GroupedArgs& p) {
    if (g >= p.G) { count = 0; return; }
    int a = tab ? tab[g] : __ldg(p.offsets + g);
    int b = tab ? tab[g + 1] : __ldg(p.offsets + g + 1);
    a = min(max(a, 0), p.M_total);
    b = min(max(b, a), p.M_total);
    r0 = a;
    r1 = b;
    tt = (b - a + kGrpTileT - 1) / kGrpTileT;
    sz = kGrpTileT;
    count = (long long)tt * p.n_tiles;
  }
  __device__ __forceinline__ void init(const GroupedArgs& p, const int* table) {
    tab = table;
    g = 0;
    base = 0;
    load(p);
  }
  __device__ __forceinline__ void init(const GroupedArgs& p) { init(p, tab); }
  __device__ __forceinline__ bool seek(const GroupedArgs& p, long long t) {
    if (t < base) init(p);
    while (g < p.G && t >= base + count) {
      base += count;
      ++g;
      load(p);
    }
    return g < p.G;
  }
  // n-tile fastest: consecutive tiles share the token block (L2 reuse).
  __device__ __forceinline__ GrpTile tile(const GroupedArgs& p, long long t) const {
    const int r = (int)(t - base);
    const int tok = r / p.n_tiles;
    const int nt_i = r - tok * p.n_tiles;
    GrpTile x;
    x.g = g;
    x.t0 = r0 + tok * sz;
    x.nt = min(sz, r1 - x.t0);
    x.nmma = (x.nt + 15) & ~15;
    x.n0 = nt_i * kGrpTileN;
    return x;
  }
};

// Number of tiles of the problem, with the walker's clamping; computed by a
// whole warp (one group per lane and pass), every lane returns it.
__device__ __forceinline__ long long grp_total_tiles(const GroupedArgs& p) {
  const int lane = (int)(threadIdx.x & 31);
  long long cnt = 0;
  for (int g0 = 0; g0 < p.G; g0 += 32) {
    const int g = g0 + lane;
    if (g < p.G) {
      int a = __ldg(p.offsets + g);
      int b = __ldg(p.offsets + g + 1);
      a = min(max(a, 0), p.M_total);
      b = min(max(b, a), p.M_total);
      cnt += (b - a + kGrpTileT - 1) / kGrpTileT;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  return cnt * p.n_tiles;
}

static __device__ __noinline__ void grouped_check_offsets(const GroupedArgs& p) {
  bool bad = __ldg(p.offsets) != 0 || __ldg(p.offsets + p.G) != p.M_total;
  int prev = 0;
  for (int g = 0; g <= p.G && !bad; ++g) {
    const int v = __ldg(p.offsets + g);
    if (v < prev || v > p.M_total) bad = true;
    prev = v;
  }
  if (bad) latch_error(p.ws, kErrBadOffsets, 2);
}

// x * sigmoid(x) with sigmoid(x) = (1 + tanh(x / 2)) / 2 (one tanh.approx).
__device__ __forceinline__ float grp_silu(float x) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * x));
  return x * fmaf(0.5f, t, 0.5f);
}
// GELU(x) = x * Phi(x) (exact erf form, the CUDA math library's normcdff).
__device__ __forceinline__ float grp_gelu(float x) { return x * normcdff(x); }

template <bool OUT_F32, int EPI, bool CLC>
__global__ void __launch_bounds__(kGrpThreads, 1)
    k_grouped_ws(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                 const __grid_constant__ CUtensorMap tmXt, const __grid_constant__ CUtensorMap tmC,
                 const GroupedArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smW = smem;
  uint8_t* smX = smW + kGrpStages * kGrpWBytes;
  uint8_t* smStg = smX + kGrpStages * kGrpXBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smStg + kGrpEpiWarps * kGrpStgBufs * kGrpStgBytes);
  // bars: full[S] | empty[S] | acc_full[2] | acc_empty[2] | tq_full[TQ] | tq_empty[TQ]
  //       | clc_full | clc_empty; then the 16-byte cancel response
  constexpr int kNumBars = 2 * kGrpStages + 4 + 2 * kGrpTQ + 2;
  static_assert(kNumBars % 2 == 0, "16-byte aligned response");
  uint8_t* clc_resp = reinterpret_cast<uint8_t*>(bars + kNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(clc_resp + 16);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile int* tq_id = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [kGrpTQ]
  static_assert(kNumBars * 8 + 16 + (2 + kGrpTQ) * 4 <= 512, "barrier area");
  int* off_tab = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bars) + 512);
  const int* tab = p.G < kGrpTabMax ? off_tab : nullptr;

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t bar_base = smem_addr(bars);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (kGrpStages + s); };
  auto accf_bar = [&](int a) { return bar_base + 8u * (2 * kGrpStages + a); };
  auto acce_bar = [&](int a) { return bar_base + 8u * (2 * kGrpStages + 2 + a); };
  auto tqf_bar = [&](int i) { return bar_base + 8u * (2 * kGrpStages + 4 + i); };
  auto tqe_bar = [&](int i) { return bar_base + 8u * (2 * kGrpStages + 4 + kGrpTQ + i); };
  const uint32_t clcf_bar = bar_base + 8u * (kNumBars - 2);
  const uint32_t clce_bar = bar_base + 8u * (kNumBars - 1);
  const uint32_t rank = cluster_ctarank();
  const long long cluster_id = blockIdx.x / 2;
  const long long num_clusters = gridDim.x / 2;

  if constexpr (CLC) {
    // A pair launched past the last tile has nothing to do (both CTAs of the
    // pair reach the same verdict, before any cluster-wide step).
    if (cluster_id >= grp_total_tiles(p)) {
      if (blockIdx.x == 0 && threadIdx.x == 0) grouped_check_offsets(p);
      return;
    }
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGrpStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), 2 * kGrpEpiWarps);
    }
    // Tile queue (cluster launch control): filled by this CTA's scheduler
    // lane, emptied by this CTA's producer, epilogue warps and (leader) MMA
    // issuer.  The cancel response is released by both CTAs' schedulers.
    for (int i = 0; i < kGrpTQ; ++i) {
      mbar_init(tqf_bar(i), 1);
      mbar_init(tqe_bar(i), 1 + kGrpEpiWarps + (rank == 0 ? 1 : 0));
    }
    mbar_init(clcf_bar, 1);
    mbar_init(clce_bar, 2);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmXt);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 2) {
    tmem_alloc<2>(smem_addr(tmem_slot), 512);
    tmem_relinquish<2>();
  }
  if (warp == 3 && tab) {
    for (int i = (int)lane; i <= p.G; i += 32) off_tab[i] = min(max(__ldg(p.offsets + i), 0), p.M_total);
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const Guard guard{p.ws, abort_flag, p.timeout_ns};

  // Next tile index for one consuming thread.  Static: the pair's own
  // sequence.  Cluster launch control: the next entry of this CTA's tile
  // queue (false at the end marker or when the CTA is aborting; every
  // consumer reads every entry, including the end marker).
  auto next_tile = [&](long long& t, bool& first, int& slot, uint32_t& ph) -> bool {
    if constexpr (!CLC) {
      t = first ? cluster_id : t + num_clusters;
      first = false;
      return true;
    } else {
      if (!wait_phase(guard, tqf_bar(slot), ph, (kRoleProducer << 16) | 0x500 | slot)) return false;
      const int id = tq_id[slot];
      mbar_arrive(tqe_bar(slot));
      if (++slot == kGrpTQ) { slot = 0; ph ^= 1u; }
      t = id;
      return id >= 0;
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      GrpWalker gw;
      gw.init(p, tab);
      int tqs = 0;
      uint32_t tqph = 0;
      long long t = 0;
      bool first = true;
      while (ok && next_tile(t, first, tqs, tqph) && gw.seek(p, t)) {
        const GrpTile tl = gw.tile(p, t);
        const int w_row = tl.n0 + (int)rank * 128;
        const int x_row = tl.t0 + (int)rank * (tl.nmma >> 1);
        const int x_rows = tl.nmma >> 1;  // token rows this CTA holds
        const bool thin = x_rows <= kGrpThinMaxRows;
        const int x_boxes = thin ? (x_rows + kGrpXThinRows - 1) / kGrpXThinRows
                                 : (x_rows + kGrpXBoxRows - 1) / kGrpXBoxRows;
        const uint32_t tx = 2u * (uint32_t)(kGrpWBytes + x_boxes * (thin ? kGrpXThinBytes : kGrpXBoxBytes));
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_phase_cluster(guard, empty_bar(stage), phase ^ 1u, (kRoleProducer << 16) | stage)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), tx);
          const uint32_t fb = map_to_cta(full_bar(stage), 0);
          const int kx = kb * kGrpBK;
          tma_load_3d_pair(smem_addr(smW + stage * kGrpWBytes), &tmW, fb, kx, w_row,
                           p.w_shared ? 0 : tl.g);
          const uint32_t xdst = smem_addr(smX + stage * kGrpXBytes);
          if (thin) {
            for (int i = 0; i < x_boxes; ++i)
              tma_load_2d_pair(xdst + i * kGrpXThinBytes, &tmXt, fb, kx, x_row + i * kGrpXThinRows);
          } else {
            for (int i = 0; i < x_boxes; ++i)
              tma_load_2d_pair(xdst + i * kGrpXBoxBytes, &tmX, fb, kx, x_row + i * kGrpXBoxRows);
          }
          if (++stage == kGrpStages) { stage = 0; phase ^= 1u; }
        }
      }
      for (int i = 0; i < kGrpStages && ok; ++i) {
        ok = wait_phase_cluster(guard, empty_bar(stage), phase ^ 1u, (kRoleProducer << 16) | 0x100 | stage);
        if (++stage == kGrpStages) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (leader)
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      GrpWalker gw;
      gw.init(p, tab);
      int tqs = 0;
      uint32_t tqph = 0;
      long long t = 0;
      bool first = true;
      while (ok && next_tile(t, first, tqs, tqph) && gw.seek(p, t)) {
        const GrpTile tl = gw.tile(p, t);
        const uint32_t idesc = idesc_bf16_f32(kGrpTileN, tl.nmma, false, false);
        if (!wait_phase_cluster(guard, acce_bar(acc), acc_phase ^ 1u, (kRoleMma << 16) | 0x100 | acc)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kGrpTileT);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_phase(guard, full_bar(stage), phase, (kRoleMma << 16) | stage)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t wBase = smem_addr(smW + stage * kGrpWBytes);
          const uint32_t xBase = smem_addr(smX + stage * kGrpXBytes);
#pragma unroll
          for (int k = 0; k < kGrpBK / 16; ++k) {
            const uint64_t ad = sdesc_sw128(wBase + k * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(xBase + k * 32, 16, 1024);
            umma_bf16<2>(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          umma_commit_pair(empty_bar(stage), 0x3);
          if (++stage == kGrpStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit_pair(accf_bar(acc), 0x3);
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
    }
  } else if (warp == 3) {
    // Lane 1: validate the device offsets off the producers' critical path
    // (one pass, latches WST_ERR_BAD_OFFSETS).
    if (lane == 1 && blockIdx.x == 0) grouped_check_offsets(p);
    if constexpr (CLC) {
      // Lane 0 (both CTAs): the tile scheduler.  The leader issues the cancel
      // requests; both CTAs receive each response and queue the same tiles.
      if (lane == 0) {
        const uint32_t resp = smem_addr(clc_resp);
        int slot = 0;
        uint32_t ph = 0, cph = 0;
        auto push = [&](int id) -> bool {
          if (!wait_phase(guard, tqe_bar(slot), ph ^ 1u, (kRoleProducer << 16) | 0x600 | slot)) return false;
          tq_id[slot] = id;
          mbar_arrive(tqf_bar(slot));
          if (++slot == kGrpTQ) { slot = 0; ph ^= 1u; }
          return true;
        };
        GrpWalker sw;
        sw.init(p, tab);
        bool ok = push((int)cluster_id);
        while (ok) {
          if (rank == 0) {
            // Both schedulers have read the previous response.
            if (!wait_phase_cluster(guard, clce_bar, cph ^ 1u, (kRoleProducer << 16) | 0x700)) break;
            mbar_arrive_expect_tx(clcf_bar, 16);
            clc_try_cancel_all(resp, clcf_bar);
          } else {
            mbar_arrive_expect_tx(clcf_bar, 16);
          }
          if (!wait_phase(guard, clcf_bar, cph, (kRoleProducer << 16) | 0x701)) break;
          uint32_t first_x = 0;
          const bool got = clc_query(resp, first_x);
          if (rank == 0) mbar_arrive(clce_bar);
          else mbar_arrive_cluster(map_to_cta(clce_bar, 0));
          cph ^= 1u;
          const long long t = (long long)(first_x >> 1);
          if (!got || !sw.seek(p, t)) break;
          ok = push((int)t);
        }
        if (ok) push(-1);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const uint32_t stg_base = smem_addr(smStg + (warp - 4) * kGrpStgBufs * kGrpStgBytes);
    int sbuf = 0;
    bool last_tma = false;  // the previous chunk (other buffer) committed a TMA store
    int acc = 0;
    uint32_t acc_phase = 0;
    GrpWalker gw;
    gw.init(p, tab);
    int tqs = 0;
    uint32_t tqph = 0;
    long long t = 0;
    bool first = true;
    while (true) {
      uint32_t got = 0;
      if (lane == 0) got = next_tile(t, first, tqs, tqph) ? 1u : 0u;
      got = __shfl_sync(0xffffffffu, got, 0);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (!got || !gw.seek(p, t)) break;
      const GrpTile tl = gw.tile(p, t);
      if (!warp_wait_phase_cluster(guard, accf_bar(acc), acc_phase, (kRoleEpilogue << 16) | acc)) break;
      tc_fence_after_sync();
      const int n_base = tl.n0 + (int)rank * 128 + q * 32;  // this warp's 32 features
      const int n_lane = n_base + (int)lane;
      float bias_v = 0.0f;
      if constexpr (EPI != 0) {
        if (n_lane < p.N) bias_v = __bfloat162float(p.bias[(long long)tl.g * p.bias_stride + n_lane]);
      }
      const uint32_t t_lane = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kGrpTileT);
#pragma unroll 1
      for (int c0 = 0; c0 < tl.nmma; c0 += 32) {
        float v[32];
        tmem_load32(t_lane + c0, v);
        if constexpr (EPI != 0) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            v[j] += bias_v;
            if constexpr (EPI == 2) v[j] = grp_silu(v[j]);
            if constexpr (EPI == 3) v[j] = grp_gelu(v[j]);
          }
        }
        // A chunk of 32 tokens all inside the group and 32 features all
        // inside N leaves through a TMA store of the transposed block; a
        // chunk at the group's end (whose box would cover the next group's
        // rows) or at the last features uses masked stores.
        const bool whole = c0 + 32 <= tl.nt && n_base + 32 <= p.N;
        const uint32_t stg_addr = stg_base + (uint32_t)(sbuf * kGrpStgBytes);
        // Every TMA store that read this buffer has finished reading it: all
        // but the newest committed store when that one used the other
        // buffer, else all of them.
        if (lane == 0) {
          if (last_tma) bulk_wait_group_read<1>();
          else bulk_wait_group_read<0>();
        }
        __syncwarp();
        // Transpose: lane (feature) writes column `lane` of the [token][feature] block.
        if constexpr (OUT_F32) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(stg_addr + j * 128u + lane * 4u), "f"(v[j]) : "memory");
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const __nv_bfloat16 h = __float2bfloat16_rn(v[j]);
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(stg_addr + j * 64u + lane * 2u),
                         "h"(*reinterpret_cast<const unsigned short*>(&h)) : "memory");
          }
        }
        if (whole) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmC, stg_addr, n_base, tl.t0 + c0);
            bulk_commit_group();
          }
          sbuf ^= 1;
          last_tma = true;
          continue;
        }
        __syncwarp();
        // Row segments of C: 64 B (bf16) / 128 B (fp32) per token row.
        constexpr int kSegs = OUT_F32 ? 8 : 4;        // 16-byte segments per row
        constexpr int kRowsPerPass = 32 / kSegs;
        constexpr int kElems = OUT_F32 ? 4 : 8;       // elements per segment
        const int seg = (int)lane % kSegs;
        const int ncol = n_base + seg * kElems;
#pragma unroll
        for (int pass = 0; pass < kSegs; ++pass) {
          const int row = (int)lane / kSegs + pass * kRowsPerPass;  // token within the chunk
          const int tok = c0 + row;
          const uint32_t src = stg_addr + row * (OUT_F32 ? 128u : 64u) + seg * 16u;
          uint4 w;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                       : "r"(src));
          if (tok < tl.nt && ncol < p.N) {
            const long long off = (long long)(tl.t0 + tok) * p.ldc + ncol;
            if (ncol + kElems <= p.N) {
              if constexpr (OUT_F32) *reinterpret_cast<uint4*>(reinterpret_cast<float*>(p.C) + off) = w;
              else *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.C) + off) = w;
            } else {
              const uint32_t parts[4] = {w.x, w.y, w.z, w.w};
              for (int e = 0; e < kElems && ncol + e < p.N; ++e) {
                if constexpr (OUT_F32) {
                  reinterpret_cast<float*>(p.C)[off + e] = __uint_as_float(parts[e]);
                } else {
                  const unsigned short hv = (unsigned short)(parts[e >> 1] >> ((e & 1) * 16));
                  reinterpret_cast<unsigned short*>(p.C)[off + e] = hv;
                }
              }
            }
          }
        }
        __syncwarp();
        sbuf ^= 1;
        last_tma = false;
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_cta(acce_bar(acc), 0));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (lane == 0) bulk_wait_group<0>();  // this warp's TMA stores are complete
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (*abort_flag) {
    for (int i = 0; i < 200; ++i) __nanosleep(1000);
  }
  cluster_sync();
  tc_fence_after_sync();
  if (warp == 2) tmem_dealloc<2>(tmem_base, 512);
}

}  // namespace wst
