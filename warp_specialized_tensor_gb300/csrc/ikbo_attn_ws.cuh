// ikbo_attn_ws.cuh -- IKBO attention for sm_103a: the candidates of one user
// share one read of that user's keys and values.
//
// "How We Built TLX: A Hardware-Native GPU Compiler for Production ML at
// Scale" (Meta Engineering), "Case Study 2: In-Kernel Broadcast Optimization
// for RecSys" names an IKBO form of FlashAttention: the candidates of a user
// share the K/V reads of the user's context, which moves the kernel from
// memory-bound toward compute-bound, and it runs as a persistent,
// warp-specialized kernel.  The pages give no formula; the reading built here:
//
//   query row r of candidate c (rows c*Lq .. c*Lq + Lq - 1), head h, attends
//   over the Lkv context rows of its user u, without a mask:
//     O[r][h] = sum_j softmax_j(scale * Q[r][h] . K[u][j][h]) * V[u][j][h]
//
// In-kernel broadcast: the query rows of ALL candidates of user u are stacked
// and cut into 128-row tiles; every tile streams K[u][:, h] and V[u][:, h]
// once, so the context is read once per 128 query rows instead of once per
// candidate.  Work item = (user u, head h, query tile t), with t fastest so
// the tiles that share a context run side by side and hit L2.  Persistent
// CTAs take items blockIdx.x, blockIdx.x + gridDim.x, ...
//
// Per item and 128-key block j (online softmax in base 2, cs = scale*log2(e)):
//   MMA      S_j = Q . K_j^T          A = Q from TMEM, B = K_j from shared
//                                     memory; M = 128 rows, N = 128 keys, K = Dh
//   softmax  x = cs * S_j;  if max(x) > m + 8 (any lane of the warp): wait
//            for the PV products so far, rescale O in TMEM and l by 2^(m - m'),
//            m = m'  (only when the running maximum grows by more than 2^8,
//            so P = 2^(x - m) <= 256 stays exact enough in bf16);
//            P_j = 2^(x - m) as bf16 pairs written back over S_j's TMEM
//            columns;  l += rowsum(P_j)
//   MMA      O += P_j . V_j           A = P_j from TMEM, B = V_j from shared
//                                     memory; M = 128, N = Dh, K = 128 keys
// and finally O / l.  Q and P live in TMEM: with MMAs this small, operand
// reads from shared memory rather than the tensor math set the pace
// (measured on GB300: Q and P read from shared memory cost about half of
// the kernel's time), so shared memory only feeds K and V.  TMEM holds Q
// (64 columns of bf16 pairs), two S/P buffers of 128 columns and O (128).
// (128-key blocks: with 64 keys the N = 64 products ran at about half the
// tensor rate and the per-block handshakes doubled.)
// The issuer queues PV_{j-2} and then S_j, which overwrites the buffer
// PV_{j-2} reads (the tensor core runs one thread's MMAs in issue order), so
// S runs two blocks ahead of PV and the softmax always finds S ready.
//
// Roles (256 threads): warp 0 TMA producer (Q once per item into a staging
// buffer; K_j and V_j per block through separate 3-deep rings, since K_j is
// consumed two blocks before V_j); warp 1 MMA issuer (one thread); warp 2
// TMEM allocation; warp 3 lane 1 of CTA 0 validates the offsets; warps 4-7
// copy Q into TMEM, run the softmax and write the output (thread = query
// row = TMEM lane).
#pragma once

#include "wst_common.cuh"

namespace wst {

constexpr int kAttnDh = 128;          // head dimension (the MMA K of S, N of PV)
constexpr int kAttnBM = 128;          // query rows per tile
constexpr int kAttnBN = 128;          // keys per block
constexpr int kAttnStages = 3;        // K ring and V ring depth (each)
constexpr int kAttnThreads = 256;
constexpr int kAttnQBytes = kAttnBM * kAttnDh * 2;        // 32 KB: two 64-wide d halves
constexpr int kAttnKBytes = kAttnBN * kAttnDh * 2;        // 32 KB: two 64-wide d halves
// barriers: q_full, q_empty, qt_full, k_full[S], k_empty[S], v_full[S],
// v_empty[S], s_full[2], p_full[2], pv_done[2], o_empty
constexpr int kAttnNumBars = 3 + 4 * kAttnStages + 7;
constexpr size_t kAttnSmemBytes = (size_t)kAttnQBytes + 2 * (size_t)kAttnStages * kAttnKBytes +
                                  512 /*barriers*/ + 1024 /*align*/;
static_assert(kAttnSmemBytes <= 232448, "shared memory per CTA");
static_assert(kAttnNumBars * 8 + 8 <= 512, "barrier area");
// TMEM columns: Q at 0 (64 columns of bf16 pairs), S/P buffers at 64 and
// 192 (P as bf16 pairs in the first 64 columns of its S buffer), O at 320.
constexpr int kAttnTmemQ = 0;
constexpr int kAttnTmemS = 64;
constexpr int kAttnTmemO = 320;
static_assert(kAttnTmemO + kAttnDh <= 512, "TMEM columns");
constexpr float kAttnRescaleLog2 = 8.0f;  // rescale O only when the max grows by > 2^8

struct AttnArgs {
  int num_users, num_cand, Lq, H, Lkv;
  int kv_blocks;         // ceil(Lkv / 64)
  float scale_log2;      // scale * log2(e)
  const int* uoff;       // device int32[num_users + 1]
  void* O;               // [num_cand * Lq][H][Dh], fp32 or bf16
  WsHeader* ws;
  unsigned long long timeout_ns;
};

// 4-D TMA tile load (K and V: {Dh, H, Lkv, users}).
__device__ __forceinline__ void attn_tma_load_4d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                                 int x, int y, int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}

// 2^x on the special-function unit (ex2.approx.ftz: 2^-inf = +0).
__device__ __forceinline__ float attn_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Store 32 consecutive fp32 columns of this thread's TMEM lane (warp-wide).
__device__ __forceinline__ void attn_tmem_store32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
      "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]),
      "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]),
      "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}

__device__ __forceinline__ void attn_tmem_store_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// tcgen05.mma (cta_group::1, kind::f16) with the A operand in TMEM: lane r
// holds row r, each 32-bit column two consecutive K elements (low half first).
__device__ __forceinline__ void attn_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct AttnItem {
  int u, h;
  int row0;   // first query row of the tile
  int rows;   // valid query rows (1..128)
};

// Walks users in order; each role runs its own walker over the same
// increasing item indices.  Offsets are clamped into [0, num_cand].
struct AttnWalker {
  int u;
  long long base, count;
  int q0, nq, tiles;

  __device__ __forceinline__ void load(const AttnArgs& p) {
    if (u >= p.num_users) { count = 0; return; }
    int a = __ldg(p.uoff + u);
    int b = __ldg(p.uoff + u + 1);
    a = min(max(a, 0), p.num_cand);
    b = min(max(b, a), p.num_cand);
    q0 = a * p.Lq;
    nq = (b - a) * p.Lq;
    tiles = (nq + kAttnBM - 1) / kAttnBM;
    count = (long long)tiles * p.H;
  }
  __device__ __forceinline__ void init(const AttnArgs& p) {
    u = 0;
    base = 0;
    load(p);
  }
  __device__ __forceinline__ bool seek(const AttnArgs& p, long long t) {
    while (u < p.num_users && t >= base + count) {
      base += count;
      ++u;
      load(p);
    }
    return u < p.num_users;
  }
  __device__ __forceinline__ AttnItem item(long long t) const {
    const int r = (int)(t - base);
    AttnItem it;
    it.u = u;
    it.h = r / tiles;
    const int qt = r - it.h * tiles;
    it.row0 = q0 + qt * kAttnBM;
    it.rows = min(kAttnBM, nq - qt * kAttnBM);
    return it;
  }
};

static __device__ __noinline__ void attn_check_offsets(const AttnArgs& p) {
  bool bad = __ldg(p.uoff) != 0 || __ldg(p.uoff + p.num_users) != p.num_cand;
  int prev = 0;
  for (int u = 0; u <= p.num_users && !bad; ++u) {
    const int v = __ldg(p.uoff + u);
    if (v < prev || v > p.num_cand) bad = true;
    prev = v;
  }
  if (bad) latch_error(p.ws, kErrBadOffsets, 3);
}

template <bool OUT_F32>
__global__ void __launch_bounds__(kAttnThreads, 1)
    k_ikbo_attn_ws(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                                    // [2 halves][128 rows][64 d] staging
  uint8_t* sK = sQ + kAttnQBytes;                        // [stage][2 halves][64 keys][64 d]
  uint8_t* sV = sK + kAttnStages * kAttnKBytes;          // [stage][2 halves][64 keys][64 d]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + kAttnStages * kAttnKBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kAttnNumBars);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t bar_base = smem_addr(bars);
  const uint32_t q_full = bar_base;          // Q tile landed in the staging buffer
  const uint32_t q_empty = bar_base + 8u;    // staging buffer copied into TMEM
  const uint32_t qt_full = bar_base + 16u;   // Q in TMEM (4 softmax warps)
  auto kf_bar = [&](int s) { return bar_base + 8u * (3 + s); };
  auto ke_bar = [&](int s) { return bar_base + 8u * (3 + kAttnStages + s); };
  auto vf_bar = [&](int s) { return bar_base + 8u * (3 + 2 * kAttnStages + s); };
  auto ve_bar = [&](int s) { return bar_base + 8u * (3 + 3 * kAttnStages + s); };
  auto sf_bar = [&](int b) { return bar_base + 8u * (3 + 4 * kAttnStages + b); };
  auto pf_bar = [&](int b) { return bar_base + 8u * (5 + 4 * kAttnStages + b); };
  auto pv_bar = [&](int b) { return bar_base + 8u * (7 + 4 * kAttnStages + b); };
  const uint32_t oe_bar = bar_base + 8u * (9 + 4 * kAttnStages);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 4);
    mbar_init(qt_full, 4);
    for (int s = 0; s < kAttnStages; ++s) {
      mbar_init(kf_bar(s), 1);
      mbar_init(ke_bar(s), 1);
      mbar_init(vf_bar(s), 1);
      mbar_init(ve_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sf_bar(b), 1);
      mbar_init(pf_bar(b), 4);   // the 4 softmax warps
      mbar_init(pv_bar(b), 1);
    }
    mbar_init(oe_bar, 4);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 2) {
    tmem_alloc<1>(smem_addr(tmem_slot), 512);
    tmem_relinquish<1>();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const Guard guard{p.ws, abort_flag, p.timeout_ns};
  const long long stride = gridDim.x;
  const int nblk = p.kv_blocks;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      AttnWalker w;
      w.init(p);
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0, it = 0;
      bool ok = true;
      for (long long t = blockIdx.x; ok && w.seek(p, t); t += stride, ++it) {
        const AttnItem x = w.item(t);
        if (!wait_phase(guard, q_empty, (it & 1u) ^ 1u, (kRoleProducer << 16) | 0x800)) break;
        mbar_arrive_expect_tx(q_full, kAttnQBytes);
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d(smem_addr(sQ + hf * (kAttnQBytes / 2)), &tmQ, q_full, hf * 64, x.h, x.row0);
        for (int j = 0; j < nblk; ++j) {
          if (!wait_phase(guard, ke_bar(ks), kph ^ 1u, (kRoleProducer << 16) | ks)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(kf_bar(ks), kAttnKBytes);
          for (int hf = 0; hf < 2; ++hf)
            attn_tma_load_4d(smem_addr(sK + ks * kAttnKBytes + hf * (kAttnKBytes / 2)), &tmK, kf_bar(ks),
                             hf * 64, x.h, j * kAttnBN, x.u);
          if (++ks == kAttnStages) { ks = 0; kph ^= 1u; }
          if (!wait_phase(guard, ve_bar(vs), vph ^ 1u, (kRoleProducer << 16) | 0x10 | vs)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(vf_bar(vs), kAttnKBytes);
          for (int hf = 0; hf < 2; ++hf)
            attn_tma_load_4d(smem_addr(sV + vs * kAttnKBytes + hf * (kAttnKBytes / 2)), &tmV, vf_bar(vs),
                             hf * 64, x.h, j * kAttnBN, x.u);
          if (++vs == kAttnStages) { vs = 0; vph ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // S = Q K^T: A = Q (TMEM), B = K_j (K-major over d: two 64-wide halves
      //            8 KB apart, 16 d = 32 B per step).
      // O += P V:  A = P (TMEM), B = V_j (MN-major: d contiguous, two 64-wide
      //            d halves 8 KB apart, 16 keys = 2 KB per step).
      constexpr uint32_t idesc_s = idesc_bf16_f32(kAttnBM, kAttnBN, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kAttnBM, kAttnDh, false, true);
      const uint32_t a_q = tmem_base + kAttnTmemQ;
      const uint32_t d_o = tmem_base + kAttnTmemO;
      AttnWalker w;
      w.init(p);
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0, it = 0;
      long long gb = 0;  // blocks before this item (buffer parity)
      bool ok = true;
      for (long long t = blockIdx.x; ok && w.seek(p, t); t += stride, ++it) {
        if (!wait_phase(guard, qt_full, it & 1u, (kRoleMma << 16) | 0x800)) break;
        tc_fence_after_sync();
        // Step j: PV_{j-2} (if j >= 2), then S_j (if j < nblk).  S_j
        // overwrites the TMEM buffer that holds P_{j-2}; the tensor core
        // performs this thread's MMAs in issue order, so PV_{j-2} reads P
        // before S_j writes there (and PV_{j-2} waited for the softmax to
        // finish block j-2, so S_{j-2} has been read as well).
        for (int j = 0; j < nblk + 2 && ok; ++j) {
          if (j >= 2) {
            const int jj = j - 2;
            const long long g = gb + jj;
            const int b = (int)(g & 1);
            if (!wait_phase(guard, vf_bar(vs), vph, (kRoleMma << 16) | 0x10 | vs) ||
                !wait_phase(guard, pf_bar(b), (uint32_t)((g >> 1) & 1), (kRoleMma << 16) | 0x200 | b) ||
                (jj == 0 && !wait_phase(guard, oe_bar, (it & 1u) ^ 1u, (kRoleMma << 16) | 0x300))) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint64_t vd0 = sdesc_sw128(smem_addr(sV + vs * kAttnKBytes), kAttnKBytes / 2, 1024);
            const uint32_t a_p = tmem_base + (uint32_t)(kAttnTmemS + kAttnBN * b);
#pragma unroll
            for (int kk = 0; kk < kAttnBN / 16; ++kk)  // 16 keys: 8 TMEM columns of P, 2 KB of V
              attn_mma_ts(d_o, a_p + (uint32_t)(kk * 8), vd0 + (uint32_t)(kk * 128), idesc_o,
                          (jj > 0 || kk != 0) ? 1u : 0u);
            umma_commit(pv_bar(b));
            umma_commit(ve_bar(vs));
            if (++vs == kAttnStages) { vs = 0; vph ^= 1u; }
          }
          if (j < nblk) {
            if (!wait_phase(guard, kf_bar(ks), kph, (kRoleMma << 16) | ks)) { ok = false; break; }
            tc_fence_after_sync();
            const int b = (int)((gb + j) & 1);
            const uint64_t kd0 = sdesc_sw128(smem_addr(sK + ks * kAttnKBytes), 16, 1024);
            const uint32_t d_s = tmem_base + (uint32_t)(kAttnTmemS + kAttnBN * b);
#pragma unroll
            for (int kk = 0; kk < kAttnDh / 16; ++kk) {
              // 16 d: 8 TMEM columns of Q; 32 B within a 64-wide half of K (16 KB apart)
              const uint32_t ko = (uint32_t)((kk >> 2) * (kAttnKBytes / 2) + (kk & 3) * 32);
              attn_mma_ts(d_s, a_q + (uint32_t)(kk * 8), kd0 + (ko >> 4), idesc_s, kk != 0 ? 1u : 0u);
            }
            umma_commit(sf_bar(b));
            umma_commit(ke_bar(ks));
            if (++ks == kAttnStages) { ks = 0; kph ^= 1u; }
          }
        }
        gb += nblk;
      }
    }
  } else if (warp == 3) {
    if (lane == 1 && blockIdx.x == 0) attn_check_offsets(p);
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ Q copy, softmax, output
    const int q = warp & 3;
    const int row = q * 32 + (int)lane;  // query row of the tile = TMEM lane
    const uint32_t t_lane = tmem_base + ((uint32_t)(q * 32) << 16);
    const uint32_t t_o = t_lane + kAttnTmemO;
    // Q row of item `it` -> TMEM (64 columns of bf16 pairs), then release
    // the staging buffer and tell the MMA issuer.
    auto copy_q = [&](uint32_t it) -> bool {
      if (!warp_wait_phase(guard, q_full, it & 1u, (kRoleEpilogue << 16) | 0x400)) return false;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float qv[32];
        const uint32_t qrow = smem_addr(sQ + hf * (kAttnQBytes / 2)) + (uint32_t)((row >> 3) * 1024 + (row & 7) * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // 16-byte chunk c of the row sits at chunk c ^ (row % 8)
          uint32_t a, b2, c2, d;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(a), "=r"(b2), "=r"(c2), "=r"(d)
                       : "r"(qrow + (uint32_t)(((c ^ (row & 7)) & 7) * 16)));
          qv[4 * c + 0] = __uint_as_float(a);
          qv[4 * c + 1] = __uint_as_float(b2);
          qv[4 * c + 2] = __uint_as_float(c2);
          qv[4 * c + 3] = __uint_as_float(d);
        }
        attn_tmem_store32(t_lane + kAttnTmemQ + hf * 32, qv);
      }
      attn_tmem_store_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(q_empty);
        mbar_arrive(qt_full);
      }
      return true;
    };
    AttnWalker w;
    w.init(p);
    long long gb = 0;
    uint32_t it = 0;
    long long t = blockIdx.x;
    bool ok = w.seek(p, t) && copy_q(0);
    while (ok) {
      const AttnItem x = w.item(t);
      float m = -INFINITY, l = 0.0f;
      for (int j = 0; j < nblk; ++j) {
        const long long g = gb + j;
        const int b = (int)(g & 1);
        const uint32_t ph = (uint32_t)((g >> 1) & 1);
        if (!warp_wait_phase(guard, sf_bar(b), ph, (kRoleEpilogue << 16) | b)) { ok = false; break; }
        tc_fence_after_sync();
        float s[kAttnBN];
#pragma unroll
        for (int c = 0; c < kAttnBN / 32; ++c)
          tmem_load32(t_lane + kAttnTmemS + kAttnBN * b + 32 * c, *reinterpret_cast<float(*)[32]>(s + 32 * c));
        // Row extremum of the raw scores (the maximum of cs * s is cs * max s
        // for cs >= 0 and cs * min s otherwise); keys past the end of the
        // context (last block only) take no part and get no weight.
        const int kvalid = p.Lkv - j * kAttnBN;
        const float cs = p.scale_log2;
        const bool pos = cs >= 0.0f;
        float e8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) e8[i] = pos ? -INFINITY : INFINITY;
        if (kvalid >= kAttnBN) {
#pragma unroll
          for (int i = 0; i < kAttnBN; ++i) e8[i & 7] = pos ? fmaxf(e8[i & 7], s[i]) : fminf(e8[i & 7], s[i]);
        } else {
#pragma unroll
          for (int i = 0; i < kAttnBN; ++i)
            if (i < kvalid) e8[i & 7] = pos ? fmaxf(e8[i & 7], s[i]) : fminf(e8[i & 7], s[i]);
        }
        float ext;
        if (pos)
          ext = fmaxf(fmaxf(fmaxf(e8[0], e8[1]), fmaxf(e8[2], e8[3])), fmaxf(fmaxf(e8[4], e8[5]), fmaxf(e8[6], e8[7])));
        else
          ext = fminf(fminf(fminf(e8[0], e8[1]), fminf(e8[2], e8[3])), fminf(fminf(e8[4], e8[5]), fminf(e8[6], e8[7])));
        const float mx = ext * cs;
        if (j == 0) {
          m = mx;  // the first PV product overwrites O: nothing to rescale
        } else {
          const bool grow = mx > m + kAttnRescaleLog2;
          if (__any_sync(0xffffffffu, grow)) {
            // O holds the PV products of blocks < j: wait for the last one,
            // then rescale O and l of the rows whose maximum grew.
            const long long gp = g - 1;
            if (!warp_wait_phase(guard, pv_bar((int)(gp & 1)), (uint32_t)((gp >> 1) & 1),
                                 (kRoleEpilogue << 16) | 0x100)) { ok = false; break; }
            tc_fence_after_sync();
            const float alpha = grow ? attn_ex2(m - mx) : 1.0f;
            if (grow) {
              l *= alpha;
              m = mx;
            }
#pragma unroll
            for (int c = 0; c < kAttnDh / 32; ++c) {
              float v[32];
              tmem_load32(t_o + c * 32, v);
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] *= alpha;
              attn_tmem_store32(t_o + c * 32, v);
            }
            attn_tmem_store_wait();
          }
        }
        // P = 2^(cs * s - m), one FFMA and one ex2 per score.
        float rs8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rs8[i] = 0.0f;
        if (kvalid >= kAttnBN) {
#pragma unroll
          for (int i = 0; i < kAttnBN; ++i) {
            s[i] = attn_ex2(fmaf(s[i], cs, -m));
            rs8[i & 7] += s[i];
          }
        } else {
#pragma unroll
          for (int i = 0; i < kAttnBN; ++i) {
            s[i] = i < kvalid ? attn_ex2(fmaf(s[i], cs, -m)) : 0.0f;
            rs8[i & 7] += s[i];
          }
        }
        l += ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
        // P_j -> TMEM as bf16 pairs over the first 64 columns of S_j's buffer
        // (the A operand of the PV product), then hand it to the MMA issuer.
#pragma unroll
        for (int h2 = 0; h2 < kAttnBN / 64; ++h2) {
          float pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c)
            pk[c] = __uint_as_float(pack_bf16x2(s[64 * h2 + 2 * c], s[64 * h2 + 2 * c + 1]));
          attn_tmem_store32(t_lane + kAttnTmemS + kAttnBN * b + 32 * h2, pk);
        }
        attn_tmem_store_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(pf_bar(b));
      }
      if (!ok) break;
      // Bring the next item's Q into TMEM before this item's output, so its
      // first S products overlap the epilogue.  Every S product of this item
      // (the readers of Q in TMEM) completed before the last s_full above.
      t += stride;
      ++it;
      const bool more = w.seek(p, t);
      if (more && !copy_q(it)) break;
      // Output: wait for the last PV product, read O, divide by l, store.
      const long long gl = gb + nblk - 1;
      if (!warp_wait_phase(guard, pv_bar((int)(gl & 1)), (uint32_t)((gl >> 1) & 1),
                           (kRoleEpilogue << 16) | 0x300)) { ok = false; break; }
      tc_fence_after_sync();
      gb += nblk;
      const float inv = 1.0f / l;
      const bool store = row < x.rows;
      const long long base = ((long long)(x.row0 + row) * p.H + x.h) * kAttnDh;
#pragma unroll
      for (int c = 0; c < kAttnDh / 32; ++c) {
        float v[32];
        tmem_load32(t_o + c * 32, v);
        if (store) {
          if constexpr (OUT_F32) {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.O) + base + c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.O) + base + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pack_bf16x2(v[8 * i] * inv, v[8 * i + 1] * inv),
                                  pack_bf16x2(v[8 * i + 2] * inv, v[8 * i + 3] * inv),
                                  pack_bf16x2(v[8 * i + 4] * inv, v[8 * i + 5] * inv),
                                  pack_bf16x2(v[8 * i + 6] * inv, v[8 * i + 7] * inv));
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(oe_bar);
      if (!more) break;
    }
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
