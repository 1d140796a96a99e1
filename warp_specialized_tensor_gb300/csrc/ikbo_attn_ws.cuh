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
// and finally O / l.  P lives in TMEM (the A operand of PV); Q stays in
// shared memory (the A operand of S), double-buffered over fragments.  TMEM
// holds three S/P buffers of 128 columns and O (128), so S runs three blocks
// ahead of PV.  Two threads issue the MMAs (S and PV), so that one
// thread's barrier waits (each ~160 cycles while MMAs are in flight,
// measured on GB300) overlap the other's products.
// (128-key blocks: with 64 keys the N = 64 products ran at about half the
// tensor rate and the per-block handshakes doubled.)
// S_j overwrites the buffer PV_{j-3} reads: the S issuer waits for PV_{j-3}
// to complete first.
// The softmax takes full blocks' scores in pairs (three-input max, packed
// fp32x2 FMA and add).  Full 128-row tiles with bf16 output leave through
// the fragment's Q buffer (free once its S products are done) and TMA
// stores; ragged tiles and fp32 output use direct stores.
//
// Schedule: items are dealt round-robin to the persistent CTAs for as many
// full waves as there are; the items of the last, partial wave (when it is
// at most half full) are split by key blocks over ALL CTAs: each tail item
// gets a contiguous group of 2 or more CTAs, which cut its key blocks into
// equal contiguous shares (one fragment per CTA).  A CTA that covers an
// item's later key blocks without its first publishes its un-normalised O,
// row maxima m and row sums l in the workspace and releases a per-warp
// flag; the CTA holding the item's first block merges them with its own:
// m* = max m_i,  l* = sum l_i 2^(m_i - m*),  O = sum O_i 2^(m_i - m*) / l*.
// Flags carry a per-call value from the host.  Waits go only from lower to
// higher CTA indices and the launch is cooperative, so every waited-for CTA
// is resident.  (With 512 items on 152 SMs the last wave holds 56 items:
// 84 % wave efficiency without the split.)
//
// Roles (256 threads): warp 0 TMA producer of Q (once per item, into one of
// two Q buffers) and K (3-deep ring); warp 3 lane 0 TMA producer of V (2-deep
// ring: V_j is consumed three blocks after K_j); warp 1 issues the S
// products and warp 2 the PV products (one thread each; warp 2 also
// allocates the tensor memory); warp 3 lane 1 of CTA 0 validates the
// offsets; warps 4-7 run the softmax and write the output (thread = query
// row = TMEM lane).
#pragma once

#include "wst_common.cuh"

namespace wst {

constexpr int kAttnDh = 128;          // head dimension (the MMA K of S, N of PV)
constexpr int kAttnBM = 128;          // query rows per tile
constexpr int kAttnBN = 128;          // keys per block
constexpr int kAttnKStages = 3;       // K ring depth
constexpr int kAttnVStages = 2;       // V ring depth (V_j is read three blocks after K_j)
constexpr int kAttnSBufs = 3;         // S/P buffers in TMEM: S runs three blocks ahead of PV
constexpr int kAttnThreads = 256;
constexpr int kAttnQBytes = kAttnBM * kAttnDh * 2;        // 32 KB: two 64-wide d halves
constexpr int kAttnKBytes = kAttnBN * kAttnDh * 2;        // 32 KB: two 64-wide d halves
// barriers: q_full[2], o_staged[2], k_full[KS], k_empty[KS], v_full[VS],
// v_empty[VS], s_full[3], p_full[3], pv_done[3], o_empty, merge_full[4]
// (one per softmax warp)
constexpr int kAttnNumBars = 4 + 2 * kAttnKStages + 2 * kAttnVStages + 3 * kAttnSBufs + 5;
// Users whose candidate offsets are copied into shared memory at the start
// (the item walkers then read them there instead of through dependent
// global loads); calls with more users read them from global memory.
constexpr int kAttnSmemUsers = 256;
constexpr size_t kAttnOffsBytes = (kAttnSmemUsers + 1) * 4 + 12;  // padded to 16 bytes
constexpr size_t kAttnSmemBytes = 2 * (size_t)kAttnQBytes +
                                  (size_t)(kAttnKStages + kAttnVStages) * kAttnKBytes +
                                  512 /*barriers*/ + kAttnOffsBytes + 1024 /*align*/;
static_assert(kAttnSmemBytes <= 232448, "shared memory per CTA");
static_assert(kAttnNumBars * 8 + 32 <= 512, "barrier area + TMEM slot, abort flag, item count");
// TMEM columns: S/P buffers at 0, 128 and 256 (P as bf16 pairs in the first
// 64 columns of its S buffer), O at 384.  Q stays in shared memory.
constexpr int kAttnTmemS = 0;
constexpr int kAttnTmemO = kAttnSBufs * kAttnBN;
static_assert(kAttnTmemO + kAttnDh <= 512, "TMEM columns");
constexpr float kAttnRescaleLog2 = 8.0f;  // rescale O only when the max grows by > 2^8
constexpr float kAttnRescaleBound = 256.0f;  // 2^kAttnRescaleLog2: the largest P kept
// Score pair of a full block at which the next S product is first tested
// (pairs 16, 32, 48 and 60 measured alike).
constexpr int kAttnEarlyTestPair = 40;

// Stream-K workspace after the 256-byte header: uint32 flags[kAttnMaxCtas][4]
// (one per softmax warp), then one partial slot per CTA: O as [4 warps][Dh/4
// column quads][32 rows][4] fp32 (one warp's share is 16 KB contiguous; a
// thread writes and reads its row's 4 columns as one 16-byte access, a warp
// 512 contiguous bytes), then m[128], l[128].
constexpr int kAttnMaxCtas = 256;
constexpr size_t kAttnFlagsOffset = 256;
constexpr size_t kAttnSlotsOffset = kAttnFlagsOffset + (size_t)kAttnMaxCtas * 4 * 4;
constexpr size_t kAttnSlotFloats = (size_t)kAttnDh * kAttnBM + 2 * kAttnBM;
constexpr size_t kAttnWorkspaceBytes = kAttnSlotsOffset + (size_t)kAttnMaxCtas * kAttnSlotFloats * 4;
constexpr int kAttnWarpPartBytes = kAttnDh * 32 * 4;        // 16 KB: one warp's O share
constexpr int kAttnMergeBatch = 2;                           // partials staged per warp at a time
static_assert(4 * kAttnMergeBatch * kAttnWarpPartBytes <= (kAttnKStages + kAttnVStages) * kAttnKBytes,
              "merge staging fits in the K/V rings");

// Bulk (TMA engine) copy of `bytes` contiguous bytes global -> shared,
// completing on an mbarrier (both addresses 16-byte aligned, size a
// multiple of 16).
__device__ __forceinline__ void attn_bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Order this thread's earlier generic-proxy accesses (the flag acquires)
// before its later async-proxy accesses to global memory.
__device__ __forceinline__ void attn_fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

struct AttnArgs {
  int num_users, num_cand, Lq, H, Lkv;
  int kv_blocks;         // ceil(Lkv / 64)
  float scale_log2;      // scale * log2(e)
  const int* uoff;       // device int32[num_users + 1]
  void* O;               // [num_cand * Lq][H][Dh], fp32 or bf16
  WsHeader* ws;
  unsigned long long timeout_ns;
  uint32_t epoch;        // this call's flag value (split only; nonzero, distinct from earlier calls')
  int split;             // 1: split the last partial wave by key blocks
  uint32_t* flags;       // [kAttnMaxCtas][4]   (split only)
  float* slots;          // [kAttnMaxCtas][kAttnSlotFloats]
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

// Three-input max / min (one instruction for two new scores).
__device__ __forceinline__ float attn_max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float attn_min3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Packed fp32 pairs: (x0, x1) = (x0 * a + c, x1 * a + c) and
// (r0, r1) += (y0, y1), each lane rounded as its scalar form.
__device__ __forceinline__ void attn_fma2(float& x0, float& x1, float a, float c) {
  uint64_t x, av, cv;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x0), "f"(x1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(av) : "f"(a));
  asm("mov.b64 %0, {%1, %1};" : "=l"(cv) : "f"(c));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(x) : "l"(x), "l"(av), "l"(cv));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x0), "=f"(x1) : "l"(x));
}
__device__ __forceinline__ void attn_add2(float& r0, float& r1, float y0, float y1) {
  uint64_t r, y;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(r0), "f"(r1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(y0), "f"(y1));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(r), "l"(y));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r0), "=f"(r1) : "l"(r));
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
  const int* offs;  // the user offsets: a shared-memory copy, or p.uoff

  __device__ __forceinline__ void load(const AttnArgs& p) {
    if (u >= p.num_users) { count = 0; return; }
    int a = offs[u];
    int b = offs[u + 1];
    a = min(max(a, 0), p.num_cand);
    b = min(max(b, a), p.num_cand);
    q0 = a * p.Lq;
    nq = (b - a) * p.Lq;
    tiles = (nq + kAttnBM - 1) / kAttnBM;
    count = (long long)tiles * p.H;
  }
  __device__ __forceinline__ void init(const AttnArgs& p, const int* offsets) {
    offs = offsets;
    u = 0;
    base = 0;
    load(p);
  }
  // Walk forward to the user holding item t (from the start again if t lies
  // before the current user: a CTA's tail fragment, which can come first,
  // has a higher item index than its whole items).
  __device__ __forceinline__ bool seek(const AttnArgs& p, long long t) {
    if (t < base) init(p, offs);
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

// One unit of work: key blocks [jb, je) of item `item`.
struct AttnFrag {
  long long item;
  int jb, je;
};

// The schedule every role walks in the same order: whole items round-robin
// (t = blockIdx.x, + gridDim.x, ... below n_full), then at most one tail
// fragment.  The R tail items (the last, partial wave) are spread over all
// CTAs: tail item r owns the contiguous CTAs [c0(r), c0(r+1)),
// c0(r) = floor(r G / R) (2 or more CTAs each, since R <= G / 2), and the
// k CTAs of an item split its key blocks evenly: the i-th takes blocks
// [floor(i nblk / k), floor((i + 1) nblk / k)).  Every tail CTA has one
// contiguous fragment of one item, so the tail costs one item boundary and
// at most ceil(nblk / 2) blocks; the CTA holding the item's first block
// merges the partials of the others, which all have higher indices.  CTAs
// whose fragment starts past the item's first block run it before their
// whole items (see next()).
struct AttnSched {
  long long n_full, t;
  int nblk;
  long long tail_item;   // this CTA's tail item (-1: none)
  int tail_jb, tail_je;  // its key blocks
  int tail_i, tail_k;    // its rank among the item's CTAs, and their count
  bool tail_left;

  __device__ __forceinline__ static int part(int i, int k, int nb) {
    return (int)((long long)i * nb / k);
  }

  __device__ __forceinline__ void init(long long n_items, int nblk_, bool split) {
    nblk = nblk_;
    const long long G = gridDim.x;
    // Split only a last wave that is at most half full: a fuller one gains
    // less than its merges cost.
    const long long tail = n_items % G;
    n_full = split && 2 * tail <= G ? n_items - tail : n_items;
    t = blockIdx.x;
    const long long R = n_items - n_full;
    tail_item = -1;
    tail_left = false;
    if (R > 0) {
      const long long c = blockIdx.x;
      const long long r = ((c + 1) * R - 1) / G;
      const long long c0 = r * G / R, c1 = (r + 1) * G / R;
      tail_i = (int)(c - c0);
      tail_k = (int)(c1 - c0);
      tail_jb = part(tail_i, tail_k, nblk);
      tail_je = part(tail_i + 1, tail_k, nblk);
      if (tail_je > tail_jb) {
        tail_item = n_full + r;
        tail_left = true;
      }
    }
  }
  __device__ __forceinline__ bool next(AttnFrag& f) {
    // A CTA that publishes a partial (its share starts past the item's first
    // block) runs its tail fragment FIRST: its partial is then ready long
    // before the merging CTA (which runs its fragment last) needs it, and
    // half of the CTAs reach their item boundaries about half an item out
    // of step with the other half, so the boundaries' bursts of new-context
    // loads from HBM do not all fall at once.
    if (tail_left && tail_jb > 0) {
      f.item = tail_item;
      f.jb = tail_jb;
      f.je = tail_je;
      tail_left = false;
      return true;
    }
    if (t < n_full) {
      f.item = t;
      f.jb = 0;
      f.je = nblk;
      t += gridDim.x;
      return true;
    }
    if (tail_left) {
      f.item = tail_item;
      f.jb = tail_jb;
      f.je = tail_je;
      tail_left = false;
      return true;
    }
    return false;
  }
};

// Items (user, head, 128-row query tile) of the whole call; offsets clamped
// as the walker clamps them.  One warp; when `soffs` is given (at most
// kAttnSmemUsers users) it also copies the offsets there.
__device__ __forceinline__ long long attn_count_items(const AttnArgs& p, uint32_t lane, int* soffs) {
  long long cnt = 0;
  if (soffs && lane == 0) soffs[p.num_users] = __ldg(p.uoff + p.num_users);
  for (int u = (int)lane; u < p.num_users; u += 32) {
    int a = __ldg(p.uoff + u);
    int b = __ldg(p.uoff + u + 1);
    if (soffs) soffs[u] = a;
    a = min(max(a, 0), p.num_cand);
    b = min(max(b, a), p.num_cand);
    cnt += ((long long)(b - a) * p.Lq + kAttnBM - 1) / kAttnBM;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  return cnt * p.H;
}

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

// tmO (bf16 output only): O as {Dh, H, rows}, boxes of 64 d x 1 head x 32
// rows; a softmax warp stores its 32 rows of a full tile through the Q
// staging buffer (free once the next Q is in TMEM).
template <bool OUT_F32>
__global__ void __launch_bounds__(kAttnThreads, 1)
    k_ikbo_attn_ws(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                   const AttnArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                                    // [2 bufs][2 halves][128 rows][64 d]
  uint8_t* sK = sQ + 2 * kAttnQBytes;                    // [stage][2 d-halves][128 keys][64 d]
  uint8_t* sV = sK + kAttnKStages * kAttnKBytes;         // [stage][2 d-halves][128 keys][64 d]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + kAttnVStages * kAttnKBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kAttnNumBars);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  long long* n_items_s = reinterpret_cast<long long*>(tmem_slot + 4);  // 8-byte aligned
  int* soffs = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bars) + 512);
  const int* offs = p.num_users <= kAttnSmemUsers ? soffs : p.uoff;

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t bar_base = smem_addr(bars);
  // q_full[qb]: fragment's Q tile landed in Q buffer qb (= fragment index & 1).
  // o_staged[qb]: the 4 softmax warps are done with Q buffer qb for a
  // fragment (its S products completed and its output's TMA stores, which
  // stage through it, have read it); the producer waits for fragment k
  // before loading the Q of fragment k + 2 there.
  auto qf_bar = [&](int b) { return bar_base + 8u * b; };
  auto os_bar = [&](int b) { return bar_base + 8u * (2 + b); };
  auto kf_bar = [&](int s) { return bar_base + 8u * (4 + s); };
  auto ke_bar = [&](int s) { return bar_base + 8u * (4 + kAttnKStages + s); };
  auto vf_bar = [&](int s) { return bar_base + 8u * (4 + 2 * kAttnKStages + s); };
  auto ve_bar = [&](int s) { return bar_base + 8u * (4 + 2 * kAttnKStages + kAttnVStages + s); };
  constexpr int kSB0 = 4 + 2 * kAttnKStages + 2 * kAttnVStages;
  auto sf_bar = [&](int b) { return bar_base + 8u * (kSB0 + b); };
  auto pf_bar = [&](int b) { return bar_base + 8u * (kSB0 + kAttnSBufs + b); };
  auto pv_bar = [&](int b) { return bar_base + 8u * (kSB0 + 2 * kAttnSBufs + b); };
  const uint32_t oe_bar = bar_base + 8u * (kSB0 + 3 * kAttnSBufs);
  auto mg_bar = [&](int w) { return bar_base + 8u * (kSB0 + 3 * kAttnSBufs + 1 + w); };

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(qf_bar(b), 1);
      mbar_init(os_bar(b), 4);
    }
    for (int st = 0; st < kAttnKStages; ++st) {
      mbar_init(kf_bar(st), 1);
      mbar_init(ke_bar(st), 1);
    }
    for (int st = 0; st < kAttnVStages; ++st) {
      mbar_init(vf_bar(st), 1);
      mbar_init(ve_bar(st), 1);
    }
    for (int b = 0; b < kAttnSBufs; ++b) {
      mbar_init(sf_bar(b), 1);
      mbar_init(pf_bar(b), 4);   // the 4 softmax warps
      mbar_init(pv_bar(b), 1);
    }
    mbar_init(oe_bar, 4);
    for (int w4 = 0; w4 < 4; ++w4) mbar_init(mg_bar(w4), 1);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    if (!OUT_F32) tma_prefetch_desc(&tmO);
  }
  if (warp == 2) {
    tmem_alloc<1>(smem_addr(tmem_slot), 512);
    tmem_relinquish<1>();
  }
  if (warp == 3) {
    const long long n = attn_count_items(p, lane, p.num_users <= kAttnSmemUsers ? soffs : nullptr);
    if (lane == 0) *n_items_s = n;
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const Guard guard{p.ws, abort_flag, p.timeout_ns};
  const int nblk = p.kv_blocks;
  const long long n_items = *n_items_s;
  const uint32_t target = p.epoch;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer (Q and K)
    // K_j is read by S_j, three blocks before PV_j reads V_j; with one
    // thread loading both in order, a V slot freed late would hold back the
    // next K load, so V has its own producer (warp 3).
    if (lane == 0) {
      AttnWalker w;
      w.init(p, offs);
      AttnSched sc;
      sc.init(n_items, nblk, p.split != 0);
      AttnFrag f;
      int ks = 0;
      uint32_t kph = 0, it = 0;
      bool ok = true;
      for (; ok && sc.next(f) && w.seek(p, f.item); ++it) {
        const AttnItem x = w.item(f.item);
        const int qb = (int)(it & 1u);
        // Q buffer qb is free once fragment it - 2 is done with it
        if (it >= 2 && !wait_phase(guard, os_bar(qb), ((it - 2u) >> 1) & 1u, (kRoleProducer << 16) | 0x900)) break;
        mbar_arrive_expect_tx(qf_bar(qb), kAttnQBytes);
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d(smem_addr(sQ + qb * kAttnQBytes + hf * (kAttnQBytes / 2)), &tmQ, qf_bar(qb), hf * 64,
                      x.h, x.row0);
        for (int j = f.jb; j < f.je; ++j) {
          if (!wait_phase(guard, ke_bar(ks), kph ^ 1u, (kRoleProducer << 16) | ks)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(kf_bar(ks), kAttnKBytes);
          for (int hf = 0; hf < 2; ++hf)
            attn_tma_load_4d(smem_addr(sK + ks * kAttnKBytes + hf * (kAttnKBytes / 2)), &tmK, kf_bar(ks),
                             hf * 64, x.h, j * kAttnBN, x.u);
          if (++ks == kAttnKStages) { ks = 0; kph ^= 1u; }
        }
      }
    }
  } else if (warp == 3 && lane == 0) {
    // ------------------------------------------------------------------ producer (V)
    AttnWalker w;
    w.init(p, offs);
    AttnSched sc;
    sc.init(n_items, nblk, p.split != 0);
    AttnFrag f;
    int vs = 0;
    uint32_t vph = 0;
    bool ok = true;
    while (ok && sc.next(f) && w.seek(p, f.item)) {
      const AttnItem x = w.item(f.item);
      for (int j = f.jb; j < f.je; ++j) {
        if (!wait_phase(guard, ve_bar(vs), vph ^ 1u, (kRoleProducer << 16) | 0x10 | vs)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(vf_bar(vs), kAttnKBytes);
        for (int hf = 0; hf < 2; ++hf)
          attn_tma_load_4d(smem_addr(sV + vs * kAttnKBytes + hf * (kAttnKBytes / 2)), &tmV, vf_bar(vs),
                           hf * 64, x.h, j * kAttnBN, x.u);
        if (++vs == kAttnVStages) { vs = 0; vph ^= 1u; }
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------------ MMA issuers
    // Warp 1 issues the S products, warp 2 the PV products (one thread
    // each).  An mbarrier wait issued while the SM's tensor core works on
    // MMAs takes ~160 cycles even when its phase completed long ago
    // (measured on GB300); with one issuer, the waits of every key block
    // left the tensor pipe idle, with two, one thread's MMAs run while the
    // other waits.  S_j overwrites the buffer of P_{j-3}, so the S issuer
    // first waits for PV_{j-3} to complete (three buffers: long done).
    //   S = Q K^T: A = Q (shared memory, K-major over d: two 64-wide halves
    //              16 KB apart, 16 d = 32 B per step), B = K_j (the same).
    //   O += P V:  A = P (TMEM), B = V_j (MN-major: d contiguous, two 64-wide
    //              d halves 16 KB apart, 16 keys = 2 KB per step).
    if (lane == 0) {
      const bool s_role = warp == 1;
      constexpr uint32_t idesc_s = idesc_bf16_f32(kAttnBM, kAttnBN, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kAttnBM, kAttnDh, false, true);
      const uint32_t d_o = tmem_base + kAttnTmemO;
      AttnSched sc;
      sc.init(n_items, nblk, p.split != 0);
      AttnFrag f;
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0, it = 0;
      int sb = 0;            // S buffer of the next product (global block mod 3)
      uint32_t sph = 0;      // ... and its use-count parity (global block / 3)
      long long nprod = 0;   // products issued by this thread so far
      bool ok = true;
      for (; ok && sc.next(f); ++it) {
        const int nb = f.je - f.jb;
        if (s_role) {
          const int qb = (int)(it & 1u);
          if (!wait_phase(guard, qf_bar(qb), (it >> 1) & 1u, (kRoleMma << 16) | 0x800)) break;
          const uint32_t q_addr = smem_addr(sQ + qb * kAttnQBytes);
          for (int j = 0; j < nb; ++j, ++nprod) {
            const int b = sb;
            // PV_{g-3} has read the P that S_g overwrites (use sph ^ 1 of
            // this buffer: the previous use completed)
            // both phases tested at once (their latencies overlap), then
            // waited for only if not yet complete
            const bool pv_ok = nprod < kAttnSBufs || mbar_test_wait(pv_bar(b), sph ^ 1u);
            const bool k_ok = mbar_test_wait(kf_bar(ks), kph);
            if (!pv_ok && !wait_phase(guard, pv_bar(b), sph ^ 1u, (kRoleMma << 16) | 0x400 | b)) {
              ok = false;
              break;
            }
            if (!k_ok && !wait_phase(guard, kf_bar(ks), kph, (kRoleMma << 16) | ks)) { ok = false; break; }
            tc_fence_after_sync();
            const uint32_t k_addr = smem_addr(sK + ks * kAttnKBytes);
            const uint32_t d_s = tmem_base + (uint32_t)(kAttnTmemS + kAttnBN * b);
#pragma unroll
            for (int kk = 0; kk < kAttnDh / 16; ++kk) {
              // 16 d: 32 B within a 64-wide half of Q and of K (16 KB apart)
              const uint32_t ko = (uint32_t)((kk >> 2) * (kAttnKBytes / 2) + (kk & 3) * 32);
              umma_bf16<1>(d_s, sdesc_sw128(q_addr + ko, 16, 1024), sdesc_sw128(k_addr + ko, 16, 1024),
                           idesc_s, kk != 0 ? 1u : 0u);
            }
            umma_commit(sf_bar(b));
            umma_commit(ke_bar(ks));
            if (++ks == kAttnKStages) { ks = 0; kph ^= 1u; }
            if (++sb == kAttnSBufs) { sb = 0; sph ^= 1u; }
          }
        } else {
          for (int jj = 0; jj < nb; ++jj, ++nprod) {
            const int b = sb;
            const bool v_ok = mbar_test_wait(vf_bar(vs), vph);
            const bool p_ok = mbar_test_wait(pf_bar(b), sph);
            if ((!v_ok && !wait_phase(guard, vf_bar(vs), vph, (kRoleMma << 16) | 0x10 | vs)) ||
                (!p_ok && !wait_phase(guard, pf_bar(b), sph, (kRoleMma << 16) | 0x200 | b)) ||
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
            if (++vs == kAttnVStages) { vs = 0; vph ^= 1u; }
            if (++sb == kAttnSBufs) { sb = 0; sph ^= 1u; }
          }
        }
      }
    }
  } else if (warp == 3) {
    if (lane == 1 && blockIdx.x == 0) attn_check_offsets(p);
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax, output
    const int q = warp & 3;
    const int row = q * 32 + (int)lane;  // query row of the tile = TMEM lane
    const uint32_t t_lane = tmem_base + ((uint32_t)(q * 32) << 16);
    const uint32_t t_o = t_lane + kAttnTmemO;
    AttnWalker w;
    w.init(p, offs);
    AttnSched sc;
    sc.init(n_items, nblk, p.split != 0);
    AttnFrag f;
    long long gb = 0;
    uint32_t it = 0;
    bool pending_release = false;  // published a partial, flag not yet released
    int pending_os = -1;           // Q buffer whose staged output a TMA store may still read
    uint32_t mg_phase = 0;         // merge batches this warp has staged
    auto release_partial = [&]() {
      if (lane == 0) {
        fence_acq_rel_gpu();
        st_release_gpu(p.flags + (size_t)blockIdx.x * 4 + q, target);
      }
      pending_release = false;
    };
    // S buffer and use-count parity of the next block (global block index
    // mod 3, and / 3), and of the previous block
    int sbuf = 0, pbuf = 0;
    uint32_t sphase = 0, pphase = 0;
    // The next block's S product was seen complete by an early test during
    // this block's exponentials (each lane's test acquires it), so its wait
    // can be skipped: a wait on a completed phase still costs ~160 cycles
    // while MMAs are in flight, on the softmax's critical path.
    bool s_ready = false;
    bool ok = sc.next(f) && w.seek(p, f.item);
    AttnItem x_next = ok ? w.item(f.item) : AttnItem{};
    while (ok) {
      const AttnItem x = x_next;
      const int nb = f.je - f.jb;
      const int qb = (int)(it & 1u);  // this fragment's Q buffer (also its output staging)
      float m = -INFINITY, l = 0.0f;
      for (int jr = 0; jr < nb; ++jr) {
        const int j = f.jb + jr;  // key block within the context
        const int b = sbuf;
        const uint32_t ph = sphase;
        if (!__all_sync(0xffffffffu, s_ready) &&
            !warp_wait_phase(guard, sf_bar(b), ph, (kRoleEpilogue << 16) | b)) { ok = false; break; }
        s_ready = false;
        tc_fence_after_sync();
        // the block after this one: its S buffer and use-count parity
        const int b_next = b + 1 == kAttnSBufs ? 0 : b + 1;
        const uint32_t ph_next = b + 1 == kAttnSBufs ? ph ^ 1u : ph;
        float s[kAttnBN];
#pragma unroll
        for (int c = 0; c < kAttnBN / 32; ++c)
          tmem_load32(t_lane + kAttnTmemS + kAttnBN * b + 32 * c, *reinterpret_cast<float(*)[32]>(s + 32 * c));
        const int kvalid = p.Lkv - j * kAttnBN;
        const float cs = p.scale_log2;
        const bool pos = cs >= 0.0f;
        // Row extremum of the raw scores (the maximum of cs * s is cs * max s
        // for cs >= 0 and cs * min s otherwise), scores 2i, 2i+1 going to
        // accumulator i % 8; keys past the end of the context (last block
        // only) take no part and get no weight.
        float e8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) e8[i] = pos ? -INFINITY : INFINITY;
        auto extremum = [&]() -> float {
          const float ext =
              pos ? fmaxf(fmaxf(fmaxf(e8[0], e8[1]), fmaxf(e8[2], e8[3])), fmaxf(fmaxf(e8[4], e8[5]), fmaxf(e8[6], e8[7])))
                  : fminf(fminf(fminf(e8[0], e8[1]), fminf(e8[2], e8[3])), fminf(fminf(e8[4], e8[5]), fminf(e8[6], e8[7])));
          return ext * cs;
        };
        // P = 2^(cs * s - m), one FFMA and one ex2 per score; for full
        // blocks in pairs (one packed FFMA and one packed add per two
        // scores; score e sums into rs8[e % 8]).
        float rs8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rs8[i] = 0.0f;
        bool p_done = false;  // s holds P_j and rs8 its row sums
        float mx;
        if (kvalid >= kAttnBN && jr > 0) {
          // After a fragment's first block the maximum rarely needs to grow
          // (only when some score exceeds m by more than 2^8), so the
          // exponentials run with the current m and no extremum is taken:
          // every P is >= 0, so a row sum of at most 2^8 proves that no P of
          // the row exceeds 2^8, i.e. that m need not grow, exactly the
          // test the extremum would make.  (The special-function, FMA and
          // comparison instructions share the sub-partition's dispatch, so
          // the comparisons saved are time saved.)  Only when some row's sum
          // is larger (or not finite) is S_j, still in TMEM, reloaded and the
          // general path taken.
#pragma unroll
          for (int i = 0; i < kAttnBN / 2; ++i) {
            if (i == kAttnEarlyTestPair) s_ready = mbar_test_wait(sf_bar(b_next), ph_next);
            attn_fma2(s[2 * i], s[2 * i + 1], cs, -m);
            s[2 * i] = attn_ex2(s[2 * i]);
            s[2 * i + 1] = attn_ex2(s[2 * i + 1]);
            attn_add2(rs8[2 * (i & 3)], rs8[2 * (i & 3) + 1], s[2 * i], s[2 * i + 1]);
          }
          const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
          if (__any_sync(0xffffffffu, !(rs <= kAttnRescaleBound))) {
#pragma unroll
            for (int c = 0; c < kAttnBN / 32; ++c)
              tmem_load32(t_lane + kAttnTmemS + kAttnBN * b + 32 * c, *reinterpret_cast<float(*)[32]>(s + 32 * c));
#pragma unroll
            for (int i = 0; i < 8; ++i) rs8[i] = 0.0f;
            if (pos) {
#pragma unroll
              for (int i = 0; i < kAttnBN / 2; ++i) e8[i & 7] = attn_max3(e8[i & 7], s[2 * i], s[2 * i + 1]);
            } else {
#pragma unroll
              for (int i = 0; i < kAttnBN / 2; ++i) e8[i & 7] = attn_min3(e8[i & 7], s[2 * i], s[2 * i + 1]);
            }
            mx = extremum();
          } else {
            p_done = true;
          }
        } else {
          if (kvalid >= kAttnBN) {
            if (pos) {
#pragma unroll
              for (int i = 0; i < kAttnBN / 2; ++i) e8[i & 7] = attn_max3(e8[i & 7], s[2 * i], s[2 * i + 1]);
            } else {
#pragma unroll
              for (int i = 0; i < kAttnBN / 2; ++i) e8[i & 7] = attn_min3(e8[i & 7], s[2 * i], s[2 * i + 1]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < kAttnBN; ++i)
              if (i < kvalid) e8[i & 7] = pos ? fmaxf(e8[i & 7], s[i]) : fminf(e8[i & 7], s[i]);
          }
          mx = extremum();
        }
        if (!p_done) {
          if (jr == 0) {
            m = mx;  // the first PV product overwrites O: nothing to rescale
          } else {
            const bool grow = mx > m + kAttnRescaleLog2;
            if (__any_sync(0xffffffffu, grow)) {
              // O holds the PV products of blocks < j: wait for the last one,
              // then rescale O and l of the rows whose maximum grew.
              if (!warp_wait_phase(guard, pv_bar(pbuf), pphase,
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
          if (kvalid >= kAttnBN) {
#pragma unroll
            for (int i = 0; i < kAttnBN / 2; ++i) {
              if (i == kAttnEarlyTestPair) s_ready = mbar_test_wait(sf_bar(b_next), ph_next);
              attn_fma2(s[2 * i], s[2 * i + 1], cs, -m);
              s[2 * i] = attn_ex2(s[2 * i]);
              s[2 * i + 1] = attn_ex2(s[2 * i + 1]);
              attn_add2(rs8[2 * (i & 3)], rs8[2 * (i & 3) + 1], s[2 * i], s[2 * i + 1]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < kAttnBN; ++i) {
              s[i] = i < kvalid ? attn_ex2(fmaf(s[i], cs, -m)) : 0.0f;
              rs8[i & 7] += s[i];
            }
          }
        }
        // a second early test (the first finds S_{j+1} complete in under half
        // of the blocks), its latency covered by the packing below
        if (!s_ready) s_ready = mbar_test_wait(sf_bar(b_next), ph_next);
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
        if (pending_release) release_partial();
        if (pending_os >= 0) {
          // The previous fragment's output stores have long read their
          // staging by now: release the Q buffer to the producer.
          if (lane == 0) {
            bulk_wait_group_read<0>();
            mbar_arrive(os_bar(pending_os));
          }
          pending_os = -1;
        }
        pbuf = b;
        pphase = ph;
        if (++sbuf == kAttnSBufs) { sbuf = 0; sphase ^= 1u; }
      }
      if (!ok) break;
      AttnFrag fn;
      const bool more = sc.next(fn) && w.seek(p, fn.item);
      if (more) x_next = w.item(fn.item);
      ++it;
      const float inv_l = 1.0f / l;  // of a whole item (a merged one computes its own)
      // Output: wait for the last PV product (the products of one thread
      // complete in order, so this fragment's S products, the readers of its
      // Q buffer, are done too), then one of three ends.
      if (!warp_wait_phase(guard, pv_bar(pbuf), pphase, (kRoleEpilogue << 16) | 0x300)) { ok = false; break; }
      tc_fence_after_sync();
      gb += nb;
      const bool store = row < x.rows;
      const long long base = ((long long)(x.row0 + row) * p.H + x.h) * kAttnDh;
      auto store_chunk = [&](int c, float (&v)[32], float inv) {
        if (!store) return;
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
      };
      // Full bf16 tiles leave through the fragment's Q buffer and TMA; the
      // rest (fp32 output, ragged tiles that must not touch the next
      // user's rows) through direct stores.
      const bool tma_out = !OUT_F32 && x.rows == kAttnBM;
      auto emit_chunk = [&](int c, float (&v)[32], float inv) {
        if (tma_out) {
          // 32 columns = 64 B of the row, in d-half c/2 at byte (c%2)*64:
          // 16-byte units (c%2)*4 .. +3, 128-byte swizzle as the Q tile.
          const uint32_t rb = smem_addr(sQ + qb * kAttnQBytes) + (uint32_t)((c >> 1) * (kAttnQBytes / 2) + row * 128);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const uint32_t unit = (uint32_t)((c & 1) * 4 + jj);
            st_shared_v4(rb + ((unit ^ (uint32_t)(row & 7)) << 4),
                         pack_bf16x2(v[8 * jj] * inv, v[8 * jj + 1] * inv),
                         pack_bf16x2(v[8 * jj + 2] * inv, v[8 * jj + 3] * inv),
                         pack_bf16x2(v[8 * jj + 4] * inv, v[8 * jj + 5] * inv),
                         pack_bf16x2(v[8 * jj + 6] * inv, v[8 * jj + 7] * inv));
          }
        } else {
          store_chunk(c, v, inv);
        }
      };
      bool staged = false;  // this warp's rows wait in the staging buffer
      if (f.jb != 0) {
        // Later key blocks of a split item: publish O, m, l for the CTA that
        // holds the item's first block.
        float* slot = p.slots + (size_t)blockIdx.x * kAttnSlotFloats;
        float4* part = reinterpret_cast<float4*>(slot + (size_t)q * (kAttnDh * 32));
#pragma unroll
        for (int c = 0; c < kAttnDh / 32; ++c) {
          float v[32];
          tmem_load32(t_o + c * 32, v);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            __stcg(part + (c * 8 + j) * 32 + lane, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
        }
        __stcg(slot + kAttnDh * kAttnBM + row, m);
        __stcg(slot + kAttnDh * kAttnBM + kAttnBM + row, l);
        // __syncwarp orders the lanes' stores before lane 0's GPU-scope
        // fence and release of the flag (one fence per warp: a fence in
        // every thread waits for each one's stores under a loaded memory
        // system).  The release waits until this warp has run the softmax
        // of the next fragment's first block, when the stores have drained
        // and the fence no longer stalls (the merging CTA needs the partial
        // only at the end of its own range).
        __syncwarp();
        pending_release = true;
      } else if (f.je != nblk) {
        // First key blocks of a split item (always this CTA's last fragment,
        // so the K/V rings are idle): merge the partials of the CTAs whose
        // ranges cover the rest of the item, up to kAttnMergeBatch at a time.
        // Their flags are awaited in parallel (one lane each), their 16 KB
        // shares copied into this warp's 48 KB of the rings, and the running
        // (m, l, O) rescaled in TMEM:  m' = max(m, m_k),
        // l' = l 2^(m - m') + sum l_k 2^(m_k - m'),  O' likewise.
        const uint32_t stg = smem_addr(sK) + (uint32_t)(q * kAttnMergeBatch * kAttnWarpPartBytes);
        // The item's CTAs after this one (ranks tail_i + 1 .. tail_k - 1,
        // at blockIdx.x + 1, ...), skipping those whose share of the key
        // blocks is empty.
        int pi = sc.tail_i + 1;
        auto next_partial = [&]() -> int {
          while (pi < sc.tail_k) {
            const int i = pi++;
            if (AttnSched::part(i + 1, sc.tail_k, nblk) > AttnSched::part(i, sc.tail_k, nblk))
              return (int)blockIdx.x + (i - sc.tail_i);
          }
          return -1;
        };
        static_assert(kAttnMergeBatch == 2 || kAttnMergeBatch == 3, "merge batch of 2 or 3");
        int cs0 = -1, cs1 = -1, cs2 = -1, nbat = 0;
        auto collect = [&]() {
          cs0 = next_partial();
          cs1 = cs0 >= 0 ? next_partial() : -1;
          cs2 = kAttnMergeBatch > 2 && cs1 >= 0 ? next_partial() : -1;
          nbat = (cs0 >= 0) + (cs1 >= 0) + (cs2 >= 0);
        };
        collect();
        bool emitted = false;
        while (nbat > 0) {
          const int b0 = cs0, b1 = cs1, b2 = cs2, nb0 = nbat;
          const int mine = lane == 0 ? b0 : (lane == 1 ? b1 : b2);
          uint32_t got = 1;
          if ((int)lane < nb0)
            got = wait_flag(guard, p.flags + (size_t)mine * 4 + q, target, (kRoleEpilogue << 16) | 0x700) ? 1u : 0u;
          // The waiting lanes' acquires and this warp barrier order the
          // copies below after the publishers' releases; the copies and the
          // m, l loads read L2, not this SM's L1.
          if (!__all_sync(0xffffffffu, got != 0)) { ok = false; break; }
          if (lane == 0) {
            // one 16 KB bulk copy per partial (this warp's rows)
            attn_fence_proxy_async_global();
            mbar_arrive_expect_tx(mg_bar(q), (uint32_t)(nb0 * kAttnWarpPartBytes));
#pragma unroll
            for (int k = 0; k < kAttnMergeBatch; ++k) {
              const int ck = k == 0 ? b0 : (k == 1 ? b1 : b2);
              if (k < nb0)
                attn_bulk_g2s(stg + (uint32_t)(k * kAttnWarpPartBytes),
                              p.slots + (size_t)ck * kAttnSlotFloats + (size_t)q * (kAttnDh * 32),
                              (uint32_t)kAttnWarpPartBytes, mg_bar(q));
            }
          }
          float mk[kAttnMergeBatch], lk[kAttnMergeBatch];
#pragma unroll
          for (int k = 0; k < kAttnMergeBatch; ++k) {
            const int ck = k == 0 ? b0 : (k == 1 ? b1 : b2);
            mk[k] = -INFINITY;
            lk[k] = 0.0f;
            if (k < nb0) {
              const float* sl = p.slots + (size_t)ck * kAttnSlotFloats;
              mk[k] = __ldcg(sl + kAttnDh * kAttnBM + row);
              lk[k] = __ldcg(sl + kAttnDh * kAttnBM + kAttnBM + row);
            }
          }
          collect();  // the next batch, while the copies fly
          const bool last = nbat == 0;
          if (!warp_wait_phase(guard, mg_bar(q), mg_phase & 1u, (kRoleEpilogue << 16) | 0xA00)) {
            ok = false;
            break;
          }
          (void)mbar_try_wait(mg_bar(q), mg_phase & 1u);  // each lane acquires the copies
          ++mg_phase;
          float mn = m;
#pragma unroll
          for (int k = 0; k < kAttnMergeBatch; ++k) mn = fmaxf(mn, mk[k]);
          const float a_self = attn_ex2(m - mn);
          float ak[kAttnMergeBatch];
          l *= a_self;
#pragma unroll
          for (int k = 0; k < kAttnMergeBatch; ++k) {
            ak[k] = k < nb0 ? attn_ex2(mk[k] - mn) : 0.0f;
            l = fmaf(lk[k], ak[k], l);
          }
          m = mn;
          const float inv = 1.0f / l;
#pragma unroll 1
          for (int c = 0; c < kAttnDh / 32; ++c) {
            float v[32];
            tmem_load32(t_o + c * 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= a_self;
#pragma unroll
            for (int k = 0; k < kAttnMergeBatch; ++k) {
              if (k < nb0) {
                const uint32_t src = stg + (uint32_t)(k * kAttnWarpPartBytes + ((c * 8) * 32 + (int)lane) * 16);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  float x0, x1, x2, x3;
                  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                               : "=f"(x0), "=f"(x1), "=f"(x2), "=f"(x3)
                               : "r"(src + (uint32_t)(j * 512)));
                  v[4 * j] = fmaf(ak[k], x0, v[4 * j]);
                  v[4 * j + 1] = fmaf(ak[k], x1, v[4 * j + 1]);
                  v[4 * j + 2] = fmaf(ak[k], x2, v[4 * j + 2]);
                  v[4 * j + 3] = fmaf(ak[k], x3, v[4 * j + 3]);
                }
              }
            }
            if (last) emit_chunk(c, v, inv);  // the merged, normalised rows
            else attn_tmem_store32(t_o + c * 32, v);
          }
          if (last) {
            emitted = true;
          } else {
            attn_tmem_store_wait();
            __syncwarp();  // the staging buffers are refilled by the next batch
          }
        }
        if (!ok) break;
        if (!emitted) {  // no partial had work (not reached: the item is split)
          const float inv = 1.0f / l;
#pragma unroll
          for (int c = 0; c < kAttnDh / 32; ++c) {
            float v[32];
            tmem_load32(t_o + c * 32, v);
            emit_chunk(c, v, inv);
          }
        }
        staged = tma_out;
      } else if (tma_out) {
        // The whole item: its rows, normalised, into the Q buffer's 128-byte
        // swizzle (written out directly: through the emit_chunk helper this
        // path took ~1400 cycles, GB300 clock stamps).
        const float inv = inv_l;
        const uint32_t rb0 = smem_addr(sQ + qb * kAttnQBytes) + (uint32_t)(row * 128);
#pragma unroll
        for (int c = 0; c < kAttnDh / 32; ++c) {
          float v[32];
          tmem_load32(t_o + c * 32, v);
          const uint32_t rb = rb0 + (uint32_t)((c >> 1) * (kAttnQBytes / 2));
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const uint32_t unit = (uint32_t)((c & 1) * 4 + jj);
            st_shared_v4(rb + ((unit ^ (uint32_t)(row & 7)) << 4),
                         pack_bf16x2(v[8 * jj] * inv, v[8 * jj + 1] * inv),
                         pack_bf16x2(v[8 * jj + 2] * inv, v[8 * jj + 3] * inv),
                         pack_bf16x2(v[8 * jj + 4] * inv, v[8 * jj + 5] * inv),
                         pack_bf16x2(v[8 * jj + 6] * inv, v[8 * jj + 7] * inv));
          }
        }
        staged = true;
      } else {
#pragma unroll
        for (int c = 0; c < kAttnDh / 32; ++c) {
          float v[32];
          tmem_load32(t_o + c * 32, v);
          store_chunk(c, v, inv_l);
        }
      }
      // O has been read: free it for the next fragment's PV products, then
      // store the staged rows (if any) and release the staging buffer.
      if (staged) fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(oe_bar);
        if (staged) {
          const uint32_t sb = smem_addr(sQ + qb * kAttnQBytes) + (uint32_t)(q * 32 * 128);
          tma_store_3d(&tmO, sb, 0, x.h, x.row0 + q * 32);
          tma_store_3d(&tmO, sb + kAttnQBytes / 2, 64, x.h, x.row0 + q * 32);
          bulk_commit_group();
        } else {
          mbar_arrive(os_bar(qb));
        }
      }
      // A staged buffer is released after the next fragment's first block
      // (waiting here for the stores to read it held the softmax at every
      // item boundary); the producer needs it only for the Q after next.
      if (staged) pending_os = qb;
      if (!more) break;
      f = fn;
    }
    if (pending_release) release_partial();
    if (lane == 0) bulk_wait_group<0>();  // this warp's output stores are complete
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
