// ikbo_ws.cuh -- in-kernel-broadcast (IKBO) linear compression for sm_103a.
//
//   Y[c] = W . concat(U[user(c)], Cf[c])
//        = W_u . U[user(c)]  +  W_c . Cf[c]          (matmul decomposition)
//
// "How We Built TLX: A Hardware-Native GPU Compiler for Production ML at
// Scale" (Meta Engineering), "Case Study 2: In-Kernel Broadcast Optimization
// for RecSys" and "TLX Provides a Building Block for the Final Stage of This
// Optimization": the user features are never replicated per candidate; the
// user partial product P[u] = W_u . U[u] is computed once per user, and one
// persistent warp-specialized kernel runs the user GEMMs and the candidate
// GEMMs through the same shared-memory ring and mbarriers without draining
// it in between; tile-level release/acquire flags hand P[u] from the CTA
// that computed it to the CTAs whose candidates need it.
//
// GEMM orientation on the tensor core (D = 128 lanes):
//   user item u : P[u]^T [D x O] = U[u]^T [D x Du] . W_u^T [Du x O]
//   cand item c : Y[c]^T [D x O] = Cf[c]^T [D x Dc] . W_c^T [Dc x O]  (+ P[u]^T)
// A = U[u]^T / Cf[c]^T is read straight from the [f][d] layout as an
// MN-major operand (d contiguous); B = W^T is K-major (W rows are f-contiguous)
// and stays resident in shared memory for the whole kernel.  TMEM lane d of
// the accumulator holds the O outputs of embedding position d, so the
// epilogue writes Y[c][o][d] with d across the warp: fully coalesced.
//
// Work per CTA (cooperative launch, every CTA resident): first the user items
// u = blockIdx.x, blockIdx.x + gridDim.x, ...; then one contiguous range of
// candidates, sized so that every CTA moves about the same number of bytes.
// A CTA only ever waits for flags set by the FIRST items of other CTAs, which
// never wait themselves, so the schedule cannot deadlock; every wait is
// bounded regardless.
#pragma once

#include "wst_common.cuh"

namespace wst {

constexpr int kIkboMaxStages = 12;
constexpr int kIkboMaxSlots = 16;
// One epilogue warpgroup (measured on GB300: two warpgroups taking alternate
// items were slower, 72 vs 66 us on the 64 x 128 workload).
constexpr int kIkboEpiGroups = 1;
constexpr int kIkboThreads = 128 + 128 * kIkboEpiGroups;  // warps 0-3 roles, 4.. epilogue
constexpr int kIkboABytes = 128 * 64 * 2;  // one K-block of U^T / Cf^T: 64 f x 128 d
constexpr int kIkboMaxGrid = 256;          // CTAs (<= SMs) the candidate split covers
constexpr int kIkboClcChunk = 16;          // candidates per unit (cluster-launch-control schedule)
constexpr int kIkboStgBytes = 32 * 32 * 4; // per-warp output staging: 32 o x 32 d fp32
// Output staging buffers per epilogue warp (double-buffered when each warp
// handles every item) and in total; the launcher sizes shared memory with
// the same constant.
constexpr int kIkboStgPerWarp = kIkboEpiGroups == 1 ? 2 : 1;
constexpr int kIkboStgTotal = 4 * kIkboEpiGroups * kIkboStgPerWarp * kIkboStgBytes;

struct IkboArgs {
  int num_users, num_cand, Du, Dc, D, O;
  int kb_u, kb_c;      // K-blocks of the user and the candidate part
  int stages, slots;   // ring depth, TMEM accumulator slots
  const int* uoff;     // device int32[num_users+1]
  float* Y;
  uint32_t* flags;     // [num_users]
  float* P;            // [num_users][O][D]
  WsHeader* ws;
  unsigned long long timeout_ns;
  uint32_t epoch;      // this call's flag value (nonzero, distinct from earlier calls')
  // Static schedule: the candidate range of CTA i is [split[i], split[i+1]),
  // contiguous ranges sized on the host so every CTA moves about the same
  // number of bytes.  Cluster-launch-control schedule: unit w of the grid
  // is user item w for w < num_users, else the candidates
  // [(w - num_users) * chunk, ...) (chunk per unit).
  int chunk;
  int split[kIkboMaxGrid + 1];
};

// A unit of work: one user item, or a contiguous range of candidates.
struct IkboUnit {
  bool user;
  int idx;     // user (user item)
  int lo, hi;  // candidates [lo, hi) (candidate unit)
  __device__ __forceinline__ int items() const { return user ? 1 : hi - lo; }
};

// Unit w of the cluster-launch-control grid.
__device__ __forceinline__ IkboUnit ikbo_clc_unit(const IkboArgs& p, int w) {
  IkboUnit u;
  u.user = w < p.num_users;
  u.idx = w;
  const long long c0 = (long long)(w - p.num_users) * p.chunk;
  u.lo = u.user ? 0 : (int)c0;
  u.hi = u.user ? 0 : (int)min(c0 + p.chunk, (long long)p.num_cand);
  return u;
}

static __device__ __noinline__ void ikbo_check_offsets(const IkboArgs& p) {
  bool bad = __ldg(p.uoff) != 0 || __ldg(p.uoff + p.num_users) != p.num_cand;
  int prev = 0;
  for (int u = 0; u <= p.num_users && !bad; ++u) {
    int v = __ldg(p.uoff + u);
    if (v < prev || v > p.num_cand) bad = true;
    prev = v;
  }
  if (bad) latch_error(p.ws, kErrBadOffsets, 1);
}

// CLC = false: cooperative persistent grid, static schedule (each CTA's user
// items, then its host-balanced candidate range).  CLC = true: one CTA per
// unit launched; running CTAs take over units of CTAs not yet started by
// hardware cluster launch control (clusterlaunchcontrol.try_cancel), so
// faster CTAs take more candidate chunks.  The user units have the lowest
// indices and start first, and their items never wait, so a candidate unit
// only waits for partials that running CTAs are computing; every wait is
// bounded regardless.
template <bool CLC>
__global__ void __launch_bounds__(kIkboThreads, 1)
    k_ikbo_ws(const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmC,
              const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmY,
              const IkboArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int kb_w = p.kb_u + p.kb_c;
  const int w_kb_bytes = p.O * 128;  // one K-block of W^T: O rows x 128 B
  uint8_t* smW = smem;
  uint8_t* smA = smW + align_up((size_t)kb_w * w_kb_bytes, 1024);
  uint8_t* smY = smA + (size_t)p.stages * kIkboABytes;  // output staging (kIkboStgTotal bytes)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smY + kIkboStgTotal);
  // bars: full[stages] | empty[stages] | accf[slots] | acce[slots] | w | users_done
  //       | tq_full[2] | tq_empty[2] | clc ; then the 16-byte cancel response
  uint8_t* clc_resp = reinterpret_cast<uint8_t*>(bars + 2 * kIkboMaxStages + 2 * kIkboMaxSlots + 8);
  uint32_t* misc = reinterpret_cast<uint32_t*>(clc_resp + 16);
  uint32_t* tmem_slot = misc;                       // [0]
  volatile uint32_t* abort_flag = misc + 1;         // [1]
  volatile int* tq_id = reinterpret_cast<volatile int*>(misc + 2);  // [2..3]: unit queue (CLC)
  uint32_t* cnt = misc + 4;                         // [4 .. 4+slots): user-publish counters

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t bar_base = smem_addr(bars);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (kIkboMaxStages + s); };
  auto accf_bar = [&](int a) { return bar_base + 8u * (2 * kIkboMaxStages + a); };
  auto acce_bar = [&](int a) { return bar_base + 8u * (2 * kIkboMaxStages + kIkboMaxSlots + a); };
  const uint32_t w_bar = bar_base + 8u * (2 * kIkboMaxStages + 2 * kIkboMaxSlots);
  // users_done: this CTA's user partials are all published (see the producer)
  const uint32_t ud_bar = w_bar + 8u;
  auto tqf_bar = [&](int i) { return w_bar + 16u + 8u * i; };
  auto tqe_bar = [&](int i) { return w_bar + 32u + 8u * i; };
  const uint32_t clc_bar = w_bar + 48u;

  // This CTA's units.  Static: user items blockIdx.x + k * gridDim.x, then
  // one candidate range.  CLC: blockIdx.x's unit, then the units the
  // scheduler lane takes over, through a 2-slot queue that every role reads.
  const int n_user_units =
      !CLC && blockIdx.x < (unsigned)p.num_users ? (p.num_users - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int c_lo = CLC ? 0 : p.split[blockIdx.x];
  const int c_hi = CLC ? 0 : p.split[blockIdx.x + 1];
  const int n_static_units = n_user_units + (c_hi > c_lo ? 1 : 0);
  auto static_unit = [&](int k) -> IkboUnit {
    IkboUnit u;
    u.user = k < n_user_units;
    u.idx = (int)blockIdx.x + k * (int)gridDim.x;
    u.lo = c_lo;
    u.hi = c_hi;
    return u;
  };
  // Next unit for one consuming thread (k counts its units).
  auto next_unit = [&](int& k, int& slot, uint32_t& ph, IkboUnit& u) -> bool {
    if constexpr (!CLC) {
      if (k >= n_static_units) return false;
      u = static_unit(k++);
      return true;
    } else {
      Guard g{p.ws, abort_flag, p.timeout_ns};
      if (!wait_phase(g, tqf_bar(slot), ph, (kRoleProducer << 16) | 0x500 | slot)) return false;
      const int id = tq_id[slot];
      mbar_arrive(tqe_bar(slot));
      if (++slot == 2) { slot = 0; ph ^= 1u; }
      if (id < 0) return false;
      u = ikbo_clc_unit(p, id);
      ++k;
      return true;
    }
  };

  // The first unit's first K-blocks are loaded by thread 0 before the
  // CTA-wide barrier (they need only the barriers it has just initialised).
  const IkboUnit first = CLC ? ikbo_clc_unit(p, (int)blockIdx.x) : static_unit(0);
  const bool have_first = CLC ? first.items() > 0 : n_static_units > 0;
  const int first_nkb = !have_first ? 0 : (first.user ? p.kb_u : p.kb_c);
  const int pre_kb = first_nkb < p.stages ? first_nkb : p.stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < p.slots; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), 4);
      cnt[a] = 0;
    }
    mbar_init(w_bar, 1);
    mbar_init(ud_bar, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(tqf_bar(i), 1);
      mbar_init(tqe_bar(i), 6);  // producer, MMA issuer, 4 epilogue warps
    }
    mbar_init(clc_bar, 1);
    *abort_flag = 0u;
    fence_mbar_init();
    // Start W^T and the first item's K-blocks now rather than after the
    // CTA-wide barrier and the tensor-memory allocation.
    mbar_arrive_expect_tx(w_bar, (uint32_t)(kb_w * w_kb_bytes));
    for (int j = 0; j < kb_w; ++j) {
      const int x = j < p.kb_u ? j * 64 : p.Du + (j - p.kb_u) * 64;
      tma_load_2d(smem_addr(smW + j * w_kb_bytes), &tmW, w_bar, x, 0);
    }
    {
      const int idx0 = first.user ? first.idx : first.lo;
      for (int kb = 0; kb < pre_kb; ++kb) {
        mbar_arrive_expect_tx(full_bar(kb), kIkboABytes);
        const uint32_t dA = smem_addr(smA + kb * kIkboABytes);
        tma_load_3d(dA, first.user ? &tmU : &tmC, full_bar(kb), 0, kb * 64, idx0);
        tma_load_3d(dA + kIkboABytes / 2, first.user ? &tmU : &tmC, full_bar(kb), 64, kb * 64, idx0);
      }
    }
    tma_prefetch_desc(&tmU);
    tma_prefetch_desc(&tmC);
    tma_prefetch_desc(&tmY);
  }
  if (warp == 2) {
    tmem_alloc<1>(smem_addr(tmem_slot), 512);
    tmem_relinquish<1>();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t target = p.epoch;
  const Guard guard{p.ws, abort_flag, p.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      // W^T (resident for the whole kernel) and the first item's first
      // K-blocks were issued before the CTA-wide barrier.
      int stage = pre_kb == p.stages ? 0 : pre_kb;
      uint32_t phase = pre_kb == p.stages ? 1u : 0u;
      bool ok = true;
      int k = 0, tqs = 0;
      uint32_t tqph = 0;
      bool first_item = true;
      IkboUnit u;
      while (ok && next_unit(k, tqs, tqph, u)) {
        if (!CLC && !u.user && n_user_units > 0) {
          // Hold this CTA's candidate loads until its user partials are
          // published.  The publishing warps' GPU-scope fences wait for the
          // SM's outstanding memory traffic; with a ring of candidate loads
          // in flight behind them they took ~10 us (measured on GB300),
          // and every CTA's candidates wait for some user's partial.
          if (!wait_phase(guard, ud_bar, 0, (kRoleProducer << 16) | 0x300)) break;
        }
        const int nkb = u.user ? p.kb_u : p.kb_c;
        const CUtensorMap* m = u.user ? &tmU : &tmC;
        for (int i = 0; i < u.items() && ok; ++i) {
          const int idx = u.user ? u.idx : u.lo + i;
          for (int kb = (first_item ? pre_kb : 0); kb < nkb; ++kb) {
            if (!wait_phase(guard, empty_bar(stage), phase ^ 1u, (kRoleProducer << 16) | stage)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(full_bar(stage), kIkboABytes);
            const uint32_t dA = smem_addr(smA + stage * kIkboABytes);
            tma_load_3d(dA, m, full_bar(stage), 0, kb * 64, idx);
            tma_load_3d(dA + kIkboABytes / 2, m, full_bar(stage), 64, kb * 64, idx);
            if (++stage == p.stages) { stage = 0; phase ^= 1u; }
          }
          first_item = false;
        }
      }
      for (int i = 0; i < p.stages && ok; ++i) {
        ok = wait_phase(guard, empty_bar(stage), phase ^ 1u, (kRoleProducer << 16) | 0x100 | stage);
        if (++stage == p.stages) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, p.O, /*A MN-major*/ true, false);
      int stage = 0;
      uint32_t phase = 0;
      int slot = 0;
      uint32_t slot_phase = 0;
      bool ok = wait_phase(guard, w_bar, 0, (kRoleMma << 16) | 0x200);
      if (ok) tc_fence_after_sync();
      int k = 0, tqs = 0;
      uint32_t tqph = 0;
      IkboUnit u;
      while (ok && next_unit(k, tqs, tqph, u)) {
        const int nkb = u.user ? p.kb_u : p.kb_c;
        const int wkb0 = u.user ? 0 : p.kb_u;
        for (int i = 0; i < u.items() && ok; ++i) {
          if (!wait_phase(guard, acce_bar(slot), slot_phase ^ 1u, (kRoleMma << 16) | 0x100 | slot)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem_base + (uint32_t)(slot * p.O);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!wait_phase(guard, full_bar(stage), phase, (kRoleMma << 16) | stage)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t aBase = smem_addr(smA + stage * kIkboABytes);
            const uint32_t bBase = smem_addr(smW + (wkb0 + kb) * w_kb_bytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              // A (MN-major): 16 f-rows of 128 B per step; the two 64-d halves
              // are 8 KB apart (leading offset), 8-row f groups 1 KB apart.
              const uint64_t ad = sdesc_sw128(aBase + kk * 2048, kIkboABytes / 2, 1024);
              // B (K-major): 16 f = 32 B per step inside the 128-byte swizzle row.
              const uint64_t bd = sdesc_sw128(bBase + kk * 32, 16, 1024);
              umma_bf16<1>(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
            umma_commit(empty_bar(stage));
            if (++stage == p.stages) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          umma_commit(accf_bar(slot));
          if (++slot == p.slots) { slot = 0; slot_phase ^= 1u; }
        }
      }
    }
  } else if (warp == 3) {
    // Lane 0 of CTA 0 validates the device offsets off the producers'
    // critical path (one pass, latches WST_ERR_BAD_OFFSETS).  With the
    // cluster-launch-control schedule, lane 1 is the unit scheduler.
    if (lane == 0 && blockIdx.x == 0) ikbo_check_offsets(p);
    if constexpr (CLC) {
      if (lane == 1) {
        const uint32_t resp = smem_addr(clc_resp);
        int slot = 0;
        uint32_t ph = 0, cph = 0;
        auto push = [&](int id) -> bool {
          if (!wait_phase(guard, tqe_bar(slot), ph ^ 1u, (kRoleProducer << 16) | 0x600 | slot)) return false;
          tq_id[slot] = id;
          mbar_arrive(tqf_bar(slot));
          if (++slot == 2) { slot = 0; ph ^= 1u; }
          return true;
        };
        bool ok = push((int)blockIdx.x);
        while (ok) {
          mbar_arrive_expect_tx(clc_bar, 16);
          clc_try_cancel(resp, clc_bar);
          if (!wait_phase(guard, clc_bar, cph, (kRoleProducer << 16) | 0x701)) { ok = false; break; }
          cph ^= 1u;
          uint32_t first_x = 0;
          if (!clc_query(resp, first_x)) break;
          ok = push((int)first_x);
        }
        if (ok) push(-1);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int d = q * 32 + (int)lane;  // embedding position = TMEM lane
    const int nchunk = p.O / 32;
    int cached_user = -1;
    int ucur = 0;  // user cursor within a candidate unit
    float pc[2][32];
    int it = 0;    // items drained by this warp (slot sequence)
    int k = 0, tqs = 0;
    uint32_t tqph = 0;
    bool ok = true;
    IkboUnit u;
    while (ok) {
      uint32_t got = 0;
      if (lane == 0) got = next_unit(k, tqs, tqph, u) ? 1u : 0u;
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      u.user = __shfl_sync(0xffffffffu, (int)u.user, 0) != 0;
      u.idx = __shfl_sync(0xffffffffu, u.idx, 0);
      u.lo = __shfl_sync(0xffffffffu, u.lo, 0);
      u.hi = __shfl_sync(0xffffffffu, u.hi, 0);
      if (!u.user && u.hi > u.lo) {
        // first user whose range ends after u.lo
        int lo = 0, hi = p.num_users - 1;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (__ldg(p.uoff + mid + 1) <= u.lo) lo = mid + 1; else hi = mid;
        }
        ucur = lo;
      }
      for (int i = 0; i < u.items(); ++i, ++it) {
        const int slot = it % p.slots;
        const uint32_t slot_phase = (uint32_t)(it / p.slots) & 1u;
        const bool is_user = u.user;
        const int idx = is_user ? u.idx : u.lo + i;
        if (!is_user) {
          while (ucur < p.num_users - 1 && __ldg(p.uoff + ucur + 1) <= idx) ++ucur;
          if (ucur != cached_user) {
            uint32_t fok = 1;
            if (lane == 0) fok = wait_flag(guard, p.flags + ucur, target, (kRoleFlag << 16) | (ucur & 0xFFFF)) ? 1u : 0u;
            fok = __shfl_sync(0xffffffffu, fok, 0);
            if (!fok) { ok = false; break; }
            (void)ld_acquire_gpu(p.flags + ucur);
            cached_user = ucur;
            const float* pu = p.P + (size_t)ucur * p.O * p.D;
#pragma unroll
            for (int j = 0; j < 32; ++j) pc[0][j] = __ldcg(pu + (size_t)j * p.D + d);
            if (nchunk > 1) {
#pragma unroll
              for (int j = 0; j < 32; ++j) pc[1][j] = __ldcg(pu + (size_t)(32 + j) * p.D + d);
            }
          }
        }
        if (!warp_wait_phase(guard, accf_bar(slot), slot_phase, (kRoleEpilogue << 16) | slot)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t t_lane = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(slot * p.O);
        if (is_user) {
          float* pu = p.P + (size_t)idx * p.O * p.D;
          for (int j = 0; j < nchunk; ++j) {
            float v[32];
            tmem_load32(t_lane + j * 32, v);
#pragma unroll
            for (int e = 0; e < 32; ++e) __stcg(pu + (size_t)(j * 32 + e) * p.D + d, v[e]);
          }
          // Publish P[u]: __syncwarp orders the lanes' stores before lane 0's
          // GPU-scope release fence; the fence and the shared-memory counter
          // form a release pattern, so the last of the four warps to count in
          // (after its own fence) releases flag[u] = this call's epoch with
          // every warp's stores ordered before it.  One fence per warp, not
          // one per thread: 128 fences in a row under a full memory system
          // delayed the flag by ~10 us.
          __syncwarp();
          if (lane == 0) {
            fence_acq_rel_gpu();
            const uint32_t old = atomicAdd(cnt + slot, 1u);
            if ((old & 3u) == 3u) {
              fence_acq_rel_gpu();
              st_release_gpu(p.flags + idx, target);
              if (!CLC && k == n_user_units) mbar_arrive(ud_bar);
            }
          }
        } else {
          const float* pu = p.P + (size_t)ucur * p.O * p.D;
          for (int j = 0; j < nchunk; ++j) {
            float v[32];
            tmem_load32(t_lane + j * 32, v);
            if (j == 0) {
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] += pc[0][e];
            } else if (j == 1) {
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] += pc[1][e];
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] += __ldcg(pu + (size_t)(j * 32 + e) * p.D + d);
            }
            // Stage this warp's 32 o x 32 d block (row o = 128 B, lane = d) and
            // TMA-store it to Y[idx][32j .. 32j+31][32q .. 32q+31].
            const int sbuf = kIkboStgPerWarp == 2 ? (it * nchunk + j) & 1 : 0;
            uint8_t* sb = smY + ((warp - 4) * kIkboStgPerWarp + sbuf) * kIkboStgBytes;
            if (lane == 0) {
              if (kIkboStgPerWarp == 2) bulk_wait_group_read<1>();
              else bulk_wait_group_read<0>();
            }
            __syncwarp();
            const uint32_t base = smem_addr(sb) + lane * 4u;
#pragma unroll
            for (int e = 0; e < 32; ++e)
              asm volatile("st.shared.f32 [%0], %1;" ::"r"(base + e * 128u), "f"(v[e]) : "memory");
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmY, smem_addr(sb), q * 32, idx * p.O + j * 32);
              bulk_commit_group();
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar(slot));
      }
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (*abort_flag) {
    for (int i = 0; i < 200; ++i) __nanosleep(1000);
  }
  tc_fence_after_sync();
  if (warp == 2) tmem_dealloc<1>(tmem_base, 512);
}

}  // namespace wst
