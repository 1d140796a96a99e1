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
// into 128-row tiles, and every tile streams K[u][:, h] and V[u][:, h] once.
// The context is then read once per 128 query rows instead of once per
// candidate.  Work item = (user u, head h, query tile t), with t fastest so the
// tiles that share a context run side by side and hit L2.  Persistent CTAs
// take items blockIdx.x, blockIdx.x + gridDim.x, ...
//
// Per item and 64-key block j (FlashAttention-style online softmax, base 2,
// cs = scale * log2(e)):
//   MMA      S_j = Q . K_j^T            M = 128 rows, N = 64 keys, K = Dh    -> TMEM
//   softmax  m_j = max(m_{j-1}, rowmax(cs * S_j));  P_j = 2^(cs * S_j - m_j)
//            (bf16, shared memory);  l = l * 2^(m_{j-1} - m_j) + rowsum(P_j)
//   MMA      O_j = P_j . V_j            M = 128, N = Dh = 128, K = 64 keys   -> TMEM
//   softmax  O = O * 2^(m_{j-1} - m_j) + O_j            (fp32 registers)
// and finally O / l.  The MMA issuer runs S_{j+1} before PV_j, so the
// softmax of block j + 1 overlaps the PV product of block j.
//
// Roles: warp 0 TMA producer (Q once per item; K_j and V_j per block through
// a 4-stage ring); warp 1 MMA issuer (one thread); warp 2 TMEM allocation;
// warp 3 lane 1 of CTA 0 validates the offsets; warps 4-7 softmax and output
// (thread = query row = TMEM lane).
#pragma once

#include "wst_common.cuh"

namespace wst {

constexpr int kAttnDh = 128;          // head dimension (the MMA K of S, N of PV)
constexpr int kAttnBM = 128;          // query rows per tile
constexpr int kAttnBN = 64;           // keys per block
constexpr int kAttnStages = 4;
constexpr int kAttnThreads = 256;
constexpr int kAttnQBytes = kAttnBM * kAttnDh * 2;        // 32 KB: two 64-wide d halves
constexpr int kAttnKBytes = kAttnBN * kAttnDh * 2;        // 16 KB
constexpr int kAttnStageBytes = 2 * kAttnKBytes;          // K_j | V_j
constexpr int kAttnPBytes = kAttnBM * kAttnBN * 2;        // 16 KB
constexpr int kAttnNumBars = 2 + 2 * kAttnStages + 5 * 2;  // see the kernel's bar map
constexpr size_t kAttnSmemBytes = (size_t)kAttnQBytes + (size_t)kAttnStages * kAttnStageBytes +
                                  2 * (size_t)kAttnPBytes + 256 /*barriers*/ + 1024 /*align*/;
static_assert(kAttnSmemBytes <= 232448, "shared memory per CTA");
// TMEM columns: S buffers at 0 and 64, O buffers at 128 and 256.
constexpr int kAttnTmemS = 0;
constexpr int kAttnTmemO = 128;

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
  uint8_t* sQ = smem;                                    // [2 halves][128 rows][64 d]
  uint8_t* sKV = sQ + kAttnQBytes;                       // [stage]{K[2][64][64], V[2][64][64]}
  uint8_t* sP = sKV + kAttnStages * kAttnStageBytes;     // [2][128 rows][64 keys]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 2 * kAttnPBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kAttnNumBars);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  static_assert(kAttnNumBars * 8 + 8 <= 256, "barrier area");

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t bar_base = smem_addr(bars);
  // bars: q_full | q_empty | kv_full[S] | kv_empty[S] | s_full[2] | s_empty[2]
  //       | p_full[2] | pv_done[2] | o_empty[2]  (o_empty follows pv_done)
  const uint32_t q_full = bar_base;
  const uint32_t q_empty = bar_base + 8u;
  auto kvf_bar = [&](int s) { return bar_base + 8u * (2 + s); };
  auto kve_bar = [&](int s) { return bar_base + 8u * (2 + kAttnStages + s); };
  auto sf_bar = [&](int b) { return bar_base + 8u * (2 + 2 * kAttnStages + b); };
  auto se_bar = [&](int b) { return bar_base + 8u * (4 + 2 * kAttnStages + b); };
  auto pf_bar = [&](int b) { return bar_base + 8u * (6 + 2 * kAttnStages + b); };
  auto pv_bar = [&](int b) { return bar_base + 8u * (8 + 2 * kAttnStages + b); };
  auto oe_bar = [&](int b) { return bar_base + 8u * (10 + 2 * kAttnStages + b); };
  static_assert(kAttnNumBars == 12 + 2 * kAttnStages, "barrier count");

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kAttnStages; ++s) {
      mbar_init(kvf_bar(s), 1);
      mbar_init(kve_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sf_bar(b), 1);
      mbar_init(se_bar(b), 4);   // the 4 softmax warps
      mbar_init(pf_bar(b), 4);
      mbar_init(pv_bar(b), 1);
      mbar_init(oe_bar(b), 4);
    }
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
      int stage = 0;
      uint32_t phase = 0, it = 0;
      bool ok = true;
      for (long long t = blockIdx.x; ok && w.seek(p, t); t += stride, ++it) {
        const AttnItem x = w.item(t);
        if (!wait_phase(guard, q_empty, (it & 1u) ^ 1u, (kRoleProducer << 16) | 0x800)) break;
        mbar_arrive_expect_tx(q_full, kAttnQBytes);
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d(smem_addr(sQ + hf * (kAttnQBytes / 2)), &tmQ, q_full, hf * 64, x.h, x.row0);
        for (int j = 0; j < nblk; ++j) {
          if (!wait_phase(guard, kve_bar(stage), phase ^ 1u, (kRoleProducer << 16) | stage)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(kvf_bar(stage), kAttnStageBytes);
          uint8_t* st = sKV + stage * kAttnStageBytes;
          for (int hf = 0; hf < 2; ++hf) {
            attn_tma_load_4d(smem_addr(st + hf * (kAttnKBytes / 2)), &tmK, kvf_bar(stage), hf * 64,
                             x.h, j * kAttnBN, x.u);
            attn_tma_load_4d(smem_addr(st + kAttnKBytes + hf * (kAttnKBytes / 2)), &tmV,
                             kvf_bar(stage), hf * 64, x.h, j * kAttnBN, x.u);
          }
          if (++stage == kAttnStages) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // S = Q K^T: A = Q (K-major over d), B = K_j (K-major over d).
      // O = P V:   A = P (K-major over keys), B = V_j (MN-major: d contiguous,
      //            two 64-wide d halves 8 KB apart, 16 keys = 2 KB per step).
      constexpr uint32_t idesc_s = idesc_bf16_f32(kAttnBM, kAttnBN, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kAttnBM, kAttnDh, false, true);
      AttnWalker w;
      w.init(p);
      int stage = 0;
      uint32_t phase = 0, it = 0;
      long long gb = 0;  // blocks issued before this item (buffer parity)
      bool ok = true;
      for (long long t = blockIdx.x; ok && w.seek(p, t); t += stride, ++it) {
        if (!wait_phase(guard, q_full, it & 1u, (kRoleMma << 16) | 0x800)) break;
        tc_fence_after_sync();
        int prev_stage = 0;
        for (int j = 0; j <= nblk && ok; ++j) {
          const int cur_stage = stage;
          if (j < nblk) {
            const long long g = gb + j;
            const int b = (int)(g & 1);
            const uint32_t ph = (uint32_t)((g >> 1) & 1);
            if (!wait_phase(guard, kvf_bar(stage), phase, (kRoleMma << 16) | stage) ||
                !wait_phase(guard, se_bar(b), ph ^ 1u, (kRoleMma << 16) | 0x100 | b)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t qB = smem_addr(sQ);
            const uint32_t kB = smem_addr(sKV + stage * kAttnStageBytes);
            const uint32_t d_s = tmem_base + (uint32_t)(kAttnTmemS + b * kAttnBN);
#pragma unroll
            for (int kk = 0; kk < kAttnDh / 16; ++kk) {
              const uint32_t off = (uint32_t)((kk & 3) * 32);  // 16 d = 32 B
              const uint64_t ad = sdesc_sw128(qB + (kk >> 2) * (kAttnQBytes / 2) + off, 16, 1024);
              const uint64_t bd = sdesc_sw128(kB + (kk >> 2) * (kAttnKBytes / 2) + off, 16, 1024);
              umma_bf16<1>(d_s, ad, bd, idesc_s, kk != 0 ? 1u : 0u);
            }
            umma_commit(sf_bar(b));
            if (j == nblk - 1) umma_commit(q_empty);
            if (++stage == kAttnStages) { stage = 0; phase ^= 1u; }
          }
          if (j >= 1) {
            const long long g = gb + j - 1;
            const int b = (int)(g & 1);
            const uint32_t ph = (uint32_t)((g >> 1) & 1);
            if (!wait_phase(guard, pf_bar(b), ph, (kRoleMma << 16) | 0x200 | b) ||
                !wait_phase(guard, oe_bar(b), ph ^ 1u, (kRoleMma << 16) | 0x300 | b)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t pB = smem_addr(sP + b * kAttnPBytes);
            const uint32_t vB = smem_addr(sKV + prev_stage * kAttnStageBytes + kAttnKBytes);
            const uint32_t d_o = tmem_base + (uint32_t)(kAttnTmemO + b * kAttnDh);
#pragma unroll
            for (int kk = 0; kk < kAttnBN / 16; ++kk) {
              const uint64_t ad = sdesc_sw128(pB + kk * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(vB + kk * 2048, kAttnKBytes / 2, 1024);
              umma_bf16<1>(d_o, ad, bd, idesc_o, kk != 0 ? 1u : 0u);
            }
            umma_commit(pv_bar(b));
            umma_commit(kve_bar(prev_stage));
          }
          prev_stage = cur_stage;
        }
        gb += nblk;
      }
    }
  } else if (warp == 3) {
    if (lane == 1 && blockIdx.x == 0) attn_check_offsets(p);
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax + output
    const int q = warp & 3;
    const int row = q * 32 + (int)lane;  // query row of the tile = TMEM lane
    const uint32_t t_lane = tmem_base + ((uint32_t)(q * 32) << 16);
    AttnWalker w;
    w.init(p);
    long long gb = 0;
    bool ok = true;
    for (long long t = blockIdx.x; ok && w.seek(p, t); t += stride) {
      const AttnItem x = w.item(t);
      float o[kAttnDh];
#pragma unroll
      for (int i = 0; i < kAttnDh; ++i) o[i] = 0.0f;
      float m = -INFINITY, l = 0.0f, alpha_prev = 0.0f;
      for (int j = 0; j <= nblk; ++j) {
        float alpha = 0.0f;
        if (j < nblk) {
          const long long g = gb + j;
          const int b = (int)(g & 1);
          const uint32_t ph = (uint32_t)((g >> 1) & 1);
          if (!warp_wait_phase(guard, sf_bar(b), ph, (kRoleEpilogue << 16) | b)) { ok = false; break; }
          tc_fence_after_sync();
          float s[kAttnBN];
          tmem_load32(t_lane + kAttnTmemS + b * kAttnBN, *reinterpret_cast<float(*)[32]>(s));
          tmem_load32(t_lane + kAttnTmemS + b * kAttnBN + 32, *reinterpret_cast<float(*)[32]>(s + 32));
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(se_bar(b));
          // Keys past the end of the context (last block only) take no weight.
          const int kvalid = p.Lkv - j * kAttnBN;
          float mx = -INFINITY;
#pragma unroll
          for (int i = 0; i < kAttnBN; ++i) {
            s[i] = i < kvalid ? s[i] * p.scale_log2 : -INFINITY;
            mx = fmaxf(mx, s[i]);
          }
          const float m_new = fmaxf(m, mx);
          alpha = attn_ex2(m - m_new);
          float rs = 0.0f;
#pragma unroll
          for (int i = 0; i < kAttnBN; ++i) {
            s[i] = attn_ex2(s[i] - m_new);
            rs += s[i];
          }
          l = l * alpha + rs;
          m = m_new;
          // P_j row -> shared memory, 128-byte swizzled K-major layout:
          // 16-byte chunk c of row r sits at chunk position c ^ (r % 8).
          const uint32_t prow = smem_addr(sP + b * kAttnPBytes) + (uint32_t)((row >> 3) * 1024 + (row & 7) * 128);
#pragma unroll
          for (int c = 0; c < kAttnBN / 8; ++c) {
            st_shared_v4(prow + (uint32_t)(((c ^ (row & 7)) & 7) * 16),
                         pack_bf16x2(s[8 * c + 0], s[8 * c + 1]), pack_bf16x2(s[8 * c + 2], s[8 * c + 3]),
                         pack_bf16x2(s[8 * c + 4], s[8 * c + 5]), pack_bf16x2(s[8 * c + 6], s[8 * c + 7]));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(pf_bar(b));
        }
        if (j >= 1) {
          // O = O * alpha_{j-1} + P_{j-1} V_{j-1}
          const long long g = gb + j - 1;
          const int b = (int)(g & 1);
          const uint32_t ph = (uint32_t)((g >> 1) & 1);
          if (!warp_wait_phase(guard, pv_bar(b), ph, (kRoleEpilogue << 16) | 0x100 | b)) { ok = false; break; }
          tc_fence_after_sync();
#pragma unroll
          for (int c = 0; c < kAttnDh / 32; ++c) {
            float v[32];
            tmem_load32(t_lane + kAttnTmemO + b * kAttnDh + c * 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[c * 32 + i] = fmaf(o[c * 32 + i], alpha_prev, v[i]);
          }
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(oe_bar(b));
        }
        alpha_prev = alpha;
      }
      if (!ok) break;
      gb += nblk;
      if (row < x.rows) {
        const float inv = 1.0f / l;
        const long long base = ((long long)(x.row0 + row) * p.H + x.h) * kAttnDh;
        if constexpr (OUT_F32) {
          float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.O) + base);
#pragma unroll
          for (int i = 0; i < kAttnDh / 4; ++i)
            dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.O) + base);
#pragma unroll
          for (int i = 0; i < kAttnDh / 8; ++i)
            dst[i] = make_uint4(pack_bf16x2(o[8 * i] * inv, o[8 * i + 1] * inv),
                                pack_bf16x2(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                                pack_bf16x2(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                                pack_bf16x2(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
        }
      }
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
