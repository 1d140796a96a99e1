/*
 * wst.h -- C ABI of libwst: persistent, warp-specialized bf16 contractions
 * for NVIDIA GB300 (sm_103a).
 *
 * Three operations, each one hand-written CUDA kernel behind one call:
 *
 *   wst_gemm_bf16            dense (optionally strided-batched) GEMM with an
 *                            optional fused bias / bias+SiLU epilogue.
 *                            Source: "How We Built TLX: A Hardware-Native GPU
 *                            Compiler for Production ML at Scale" (Meta
 *                            Engineering), section "Introducing TLX": the
 *                            tiled matmul C = A.B with an fp32 accumulator,
 *                            restructured into a TMA producer, a single MMA
 *                            issuer accumulating in tensor memory, and an
 *                            epilogue that stores the tile; the fused
 *                            epilogue follows "Five key areas" (model-aware
 *                            kernel fusion).
 *   wst_grouped_gemm_bf16    one GEMM per group (mixture-of-experts expert
 *                            matmuls) over variable, device-resident row
 *                            offsets.  Source: same page, "TLX in
 *                            Production" and "Case Study 3: Distributed
 *                            Grouped GEMM for LLM Pretraining".
 *   wst_ikbo_linear_compress in-kernel-broadcast linear compression,
 *                            Y[c] = W . concat(U[user(c)], Cf[c]), with the
 *                            user part W_u.U[u] computed once per user and
 *                            broadcast inside the kernel.  Source: same page,
 *                            "Case Study 2: In-Kernel Broadcast Optimization
 *                            for RecSys" and "TLX Provides a Building Block
 *                            for the Final Stage of This Optimization"
 *                            (matmul decomposition, a persistent
 *                            warp-specialized kernel in which user and
 *                            candidate GEMMs share one buffer ring, and
 *                            tile-level release/acquire across CTAs).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All matrix pointers are DEVICE pointers to memory the caller owns and
 *    keeps alive until the work on `stream` has finished.  The library never
 *    allocates or frees device memory and never falls back to the CPU; the
 *    only device memory it keeps is the fixed scratch array of
 *    wst_ikbo_linear_compress_noalloc.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *    call is asynchronous: it validates its arguments on the host, enqueues
 *    one kernel on `stream`, and returns.
 *  - bf16 is IEEE-style bfloat16; accumulation is fp32; bf16 outputs are
 *    rounded to nearest even.
 *  - Alignment: every matrix pointer is 16-byte aligned and every leading
 *    dimension / batch stride, in bytes, is a multiple of 16 (the tensor
 *    memory accelerator's rule).  Otherwise WST_ERR_ALIGNMENT.
 *  - `workspace` is a caller-owned device buffer of at least
 *    wst_workspace_size(...) bytes, zero-filled once before first use (for
 *    example with wst_workspace_init).  It carries the device error word and,
 *    for IKBO, the per-user partial products and their ready flags.  One
 *    workspace must not be used by two calls that can run at the same time.
 *  - Errors found on the host are returned before anything is enqueued.
 *    Errors found on the device (a bounded wait that ran out, inconsistent
 *    device offsets, a row index out of range in wst_permute_rows) are
 *    latched in the workspace; wst_sync_status reads and clears them.  No
 *    call aborts, traps or throws.
 */
#ifndef WST_H_
#define WST_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  WST_OK = 0,
  WST_ERR_INVALID_ARG = 1,  /* a size, pointer, stride or enum is out of range   */
  WST_ERR_ALIGNMENT = 2,    /* pointer / stride breaks the 16-byte rule          */
  WST_ERR_UNSUPPORTED = 3,  /* valid request this build does not implement        */
  WST_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed (see message)    */
  WST_ERR_TIMEOUT = 5,      /* a device-side bounded wait ran out                 */
  WST_ERR_BAD_OFFSETS = 6   /* device offsets not non-decreasing from 0 to total  */
} wst_status;

typedef enum { WST_F32 = 0, WST_BF16 = 1 } wst_dtype;

typedef enum {
  WST_EPI_NONE = 0,      /* C = A.B^T                                   */
  WST_EPI_BIAS = 1,      /* C = A.B^T + bias[n]                         */
  WST_EPI_BIAS_SILU = 2, /* C = SiLU(A.B^T + bias[n]), SiLU(x)=x/(1+e^-x) */
  WST_EPI_BIAS_GELU = 3  /* C = GELU(A.B^T + bias[n]), GELU(x)=x*Phi(x), Phi the standard
                            normal distribution function (exact erf form) */
} wst_epilogue;

/*
 * Process-wide tuning options.  They choose between equivalent schedules of
 * the same computation (the results are bitwise equal); the pages have no
 * counterpart.  A value applies to every later call on every thread of the
 * process; set options between calls, not while another thread is calling.
 * (WST_OPT_NORM_STATS alone changes the order of a sum; see below.)
 *   WST_OPT_GROUPED_SCHEDULE  tile schedule of wst_grouped_gemm_bf16:
 *                             WST_SCHED_STATIC (default: persistent CTA pairs
 *                             walk the tiles in a fixed order) or
 *                             WST_SCHED_CLC (one CTA pair per tile launched,
 *                             running pairs take unstarted pairs' tiles by
 *                             hardware cluster launch control).
 *   WST_OPT_DENSE_CTA_GROUP   tile shape of the dense, batched and
 *                             norm-fused GEMMs: 0 automatic (default: CTA
 *                             pairs on 256-row tiles when M > 128 and
 *                             K > 512, else one CTA per 128-row tile), 1
 *                             always one CTA per 128-row tile, 2 always CTA
 *                             pairs.
 *   WST_OPT_IKBO_SCHEDULE     candidate schedule of the IKBO linear
 *                             compression (both entry points):
 *                             WST_SCHED_STATIC (default: a persistent grid,
 *                             each CTA's user items, then one contiguous
 *                             candidate range balanced on the host) or
 *                             WST_SCHED_CLC (one CTA per user item and per
 *                             16-candidate chunk launched; running CTAs take
 *                             over unstarted ones by hardware cluster launch
 *                             control).
 *   WST_OPT_NORM_STATS        where wst_gemm_rmsnorm_bf16 and
 *                             wst_gemm_layernorm_bf16 take the row
 *                             statistics: WST_NORM_STATS_AUTO (default: a
 *                             separate pass over A when N > 2048 (RMSNorm)
 *                             or N > 512 (LayerNorm) and the workspace
 *                             holds the statistics, else in the GEMM), WST_NORM_STATS_FUSED (always gathered
 *                             in the GEMM from the A tiles in shared memory)
 *                             or WST_NORM_STATS_PASS (always the separate
 *                             pass; a workspace smaller than
 *                             wst_gemm_norm_workspace_size() is then
 *                             WST_ERR_INVALID_ARG).  The two forms sum in a
 *                             different order: results agree to rounding,
 *                             not bitwise.
 * wst_set_option returns WST_ERR_INVALID_ARG for an unknown option or value.
 */
typedef enum {
  WST_OPT_GROUPED_SCHEDULE = 0,
  WST_OPT_DENSE_CTA_GROUP = 1,
  WST_OPT_IKBO_SCHEDULE = 2,
  WST_OPT_NORM_STATS = 3
} wst_option;

typedef enum { WST_SCHED_STATIC = 0, WST_SCHED_CLC = 1 } wst_schedule;
typedef enum {
  WST_NORM_STATS_AUTO = 0,
  WST_NORM_STATS_FUSED = 1,
  WST_NORM_STATS_PASS = 2
} wst_norm_stats;

wst_status wst_set_option(wst_option opt, int value);
/* Current value of an option in *value (WST_ERR_INVALID_ARG if unknown). */
wst_status wst_get_option(wst_option opt, int* value);

/* Bytes of workspace a call needs.  GEMM and grouped GEMM need
 * wst_workspace_size(0, 0, 0); IKBO needs wst_workspace_size(num_users, O, D). */
size_t wst_workspace_size(int num_users, int O, int D);

/* Zero-fill `bytes` of `workspace` on `stream` (asynchronous). */
wst_status wst_workspace_init(void* workspace, size_t bytes, void* stream);

/*
 * Dense / strided-batched GEMM.  For b in [0,batch), m in [0,M), n in [0,N):
 *   C[b][m][n] = epi( sum_k A[b][m][k] * B[b][n][k] (+ bias[b][n]) )
 *   A     bf16, element (b,m,k) at A + b*strideA + m*lda + k   (row-major M x K)
 *   B     bf16, element (b,n,k) at B + b*strideB + n*ldb + k   (N x K, K
 *         contiguous: the column-major K x N operand)
 *   bias  bf16, element (b,n) at bias + b*strideBias + n; NULL unless epi>0;
 *         strideBias 0 shares one bias row across the batch
 *   C     c_type, element (b,m,n) at C + b*strideC + m*ldc + n
 *   Strides are in ELEMENTS.  strideA / strideB may be 0 (operand shared by
 *   the whole batch); strideC must be 0 only when batch == 1.
 * Requires batch >= 1, M, N, K >= 1, lda >= K, ldb >= K, ldc >= N.
 */
wst_status wst_gemm_bf16(int batch, int M, int N, int K,
                         const void* A, long lda, long strideA,
                         const void* B, long ldb, long strideB,
                         const void* bias, long strideBias,
                         void* C, long ldc, long strideC, wst_dtype c_type,
                         wst_epilogue epi, void* workspace, void* stream);

/*
 * GEMM on RMS-normalised rows of A (normalisation fused into the GEMM).  Same
 * arguments, layouts and rules as wst_gemm_bf16, plus eps >= 0:
 *   r[b][m]    = 1 / sqrt( (1/K) sum_k A[b][m][k]^2 + eps )
 *   C[b][m][n] = epi( r[b][m] * sum_k A[b][m][k] * B[b][n][k] (+ bias[b][n]) )
 * i.e. y = RMSNorm(x) W^T (+ b) with the norm's learned per-feature scale
 * folded into B by the caller.  The normalised A is never formed: r is
 * applied to the fp32 accumulators in the GEMM's epilogue.  The row
 * statistics come either from the A tiles as they stream through shared
 * memory (A read from HBM once; every 256-column tile of N recomputes them)
 * or from a separate pass over A into the workspace (one more read of A,
 * the GEMM then runs without the statistics warps); WST_OPT_NORM_STATS
 * chooses, by default the pass when N > 2048 and workspace_bytes >=
 * wst_gemm_norm_workspace_size(batch, M, N, strideA, strideB, 0).
 * workspace: 16-byte aligned, at least 256 bytes (the status header).
 * Source: the TLX write-up ("How We Built TLX: A Hardware-Native GPU Compiler
 * for Production ML at Scale", companion work on norm fusion into GEMMs, and
 * "Five key areas": model-aware fusion); the pages give no formula, this is
 * the plainest RMSNorm reading.  Runs on 256 x 256 CTA-pair tiles when
 * M > 128 and K > 512, else on single-CTA 128 x 256 tiles.
 */
wst_status wst_gemm_rmsnorm_bf16(int batch, int M, int N, int K,
                                 const void* A, long lda, long strideA,
                                 const void* B, long ldb, long strideB, float eps,
                                 const void* bias, long strideBias,
                                 void* C, long ldc, long strideC, wst_dtype c_type,
                                 wst_epilogue epi, void* workspace, size_t workspace_bytes,
                                 void* stream);

/*
 * GEMM on LayerNorm-normalised rows of A.  Same arguments, layouts and rules
 * as wst_gemm_rmsnorm_bf16, with
 *   mu[b][m]   = (1/K) sum_k A[b][m][k]
 *   var[b][m]  = (1/K) sum_k (A[b][m][k] - mu[b][m])^2      (biased)
 *   C[b][m][n] = epi( sum_k (A[b][m][k] - mu) / sqrt(var + eps) * B[b][n][k]
 *                     (+ bias[b][n]) )
 * i.e. y = LayerNorm(x) W^T (+ b), the norm's per-feature scale folded into B
 * and its shift into bias by the caller.  Computed as
 *   r (A.B^T)[m][n] - r mu s[n],   r = 1/sqrt(var + eps),  s[n] = sum_k B[n][k],
 * a first kernel writing the column sums s (fp32) into the workspace.  The
 * statistics are shifted-data sums in fp32 about the row's first element c
 * (mu = c + E[d], var = E[d^2] - E[d]^2 with d = A - c, clamped at 0), taken
 * from the A tiles in the GEMM or by a separate pass over A, as for
 * wst_gemm_rmsnorm_bf16 (WST_OPT_NORM_STATS; by default the pass when N >
 * 512 and workspace_bytes >= wst_gemm_norm_workspace_size(batch, M, N,
 * strideA, strideB, 1)).
 * workspace: 16-byte aligned, at least wst_gemm_layernorm_workspace_size(
 * batch, N, strideB) bytes (workspace_bytes says how many were given;
 * smaller returns WST_ERR_INVALID_ARG).  Two or three kernel launches on
 * `stream`.
 * Source: the same TLX norm-fusion item as wst_gemm_rmsnorm_bf16 (the pages
 * name LayerNorm and RMSNorm without formulas); standard LayerNorm reading.
 */
wst_status wst_gemm_layernorm_bf16(int batch, int M, int N, int K,
                                   const void* A, long lda, long strideA,
                                   const void* B, long ldb, long strideB, float eps,
                                   const void* bias, long strideBias,
                                   void* C, long ldc, long strideC, wst_dtype c_type,
                                   wst_epilogue epi, void* workspace, size_t workspace_bytes,
                                   void* stream);

/* Workspace bytes wst_gemm_layernorm_bf16 needs: the status header plus
 * batch (1 when strideB == 0) rows of N fp32 column sums, each padded to a
 * multiple of 4 floats. */
size_t wst_gemm_layernorm_workspace_size(int batch, int N, long strideB);

/* Workspace bytes with which the norm GEMMs (layernorm != 0: LayerNorm) can
 * take the row statistics from a separate pass: the header, the LayerNorm
 * column sums, then 8 bytes (r, r*mu as two fp32) per row of A (batch * M
 * rows; M when batch == 1 or strideA == 0), 16-byte aligned.  0 for
 * invalid sizes. */
size_t wst_gemm_norm_workspace_size(int batch, int M, int N, long strideA, long strideB,
                                    int layernorm);

/*
 * Grouped GEMM over G groups sharing N and K.  d_offsets is a DEVICE int32
 * array of G+1 entries, non-decreasing, d_offsets[0] = 0, d_offsets[G] =
 * M_total; group g owns rows [d_offsets[g], d_offsets[g+1]) of A and C
 * (empty groups allowed):
 *   C[m][n] = epi( sum_k A[m][k] * B[g][n][k] (+ bias[g][n]) ),  m in group g
 *   A     bf16 [M_total][K] row-major, leading dimension lda
 *   B     bf16, element (g,n,k) at B + g*strideB_group + n*ldb + k
 *   bias  bf16, element (g,n) at bias + g*strideBias + n, or NULL (epi == 0)
 *   C     c_type [M_total][N], leading dimension ldc.  Rows outside every
 *         group are never written.
 * Offsets that break the rule are detected on the device: the kernel clamps
 * them into [0, M_total] (so no access leaves the buffers) and latches
 * WST_ERR_BAD_OFFSETS for wst_sync_status.
 */
wst_status wst_grouped_gemm_bf16(int G, int M_total, int N, int K,
                                 const void* A, long lda,
                                 const void* B, long ldb, long strideB_group,
                                 const int* d_offsets,
                                 const void* bias, long strideBias,
                                 void* C, long ldc, wst_dtype c_type,
                                 wst_epilogue epi, void* workspace, void* stream);

/*
 * Expert parallelism: the grouped GEMM's experts spread over the R ranks
 * (GPUs) of a node ("How We Built TLX: A Hardware-Native GPU Compiler for
 * Production ML at Scale", "Case Study 3: Distributed Grouped GEMM for LLM
 * Pretraining" and "TLX in Production": the distributed grouped GEMM of
 * mixture-of-experts pretraining).  G experts, G divisible by R; rank r owns
 * experts [r*G/R, (r+1)*G/R).  A token t routed to k experts forms the pairs
 * p = t*k + s (s < k).  One layer on a rank:
 *   1. wst_ep_dispatch_plan on the rank's routing table (host);
 *   2. exchange the per-(rank, local expert) counts (an all-to-all);
 *   3. wst_permute_rows gathers the token rows of the pairs in send order;
 *   4. all-to-all of the rows (send_counts out, the received counts in);
 *   5. wst_ep_receive_plan orders the received rows by local expert;
 *      wst_permute_rows gathers them, wst_grouped_gemm_bf16 multiplies them
 *      by the rank's experts (group offsets from the plan);
 *   6. wst_permute_rows scatters the products back to received order, the
 *      reverse all-to-all returns them, and wst_permute_rows scatters them
 *      to their pairs.
 * The exchanges are the caller's collectives (for example NCCL); the plans
 * are host functions and need no GPU.
 *
 * wst_ep_dispatch_plan: HOST arrays.
 *   routing            int32 [num_tokens][top_k], expert ids in [0, num_experts)
 *   send_counts        out int32 [world_size]: pairs sent to each rank
 *   send_group_counts  out int32 [num_experts]: pairs per expert (entry
 *                      r*G/R + j: rank r's local expert j)
 *   send_pairs         out int32 [num_tokens*top_k]: the pair carried by each
 *                      send row, ordered by destination rank, then local
 *                      expert, then pair id
 * Returns WST_ERR_INVALID_ARG for a bad size, an expert id out of range or
 * num_experts not divisible by world_size.
 */
wst_status wst_ep_dispatch_plan(int num_tokens, int top_k, const int* routing, int num_experts,
                                int world_size, int* send_counts, int* send_group_counts,
                                int* send_pairs);

/*
 * wst_ep_receive_plan: HOST arrays.  Rows arrive from the world_size ranks
 * in source order, each source's block ordered by local expert, with
 * recv_group_counts[s][e] rows from source s for local expert e.
 *   group_offsets  out int32 [experts_per_rank+1]: the grouped GEMM's offsets
 *                  of the expert-major order
 *   expert_rows    out int32 [total received rows]: expert-major row i is
 *                  received row expert_rows[i] (local expert e, then source s)
 */
wst_status wst_ep_receive_plan(int world_size, int experts_per_rank, const int* recv_group_counts,
                               int* group_offsets, int* expert_rows);

/*
 * Row permutation on the GPU: for i < n_rows,
 *   dst row (d_dst_index ? d_dst_index[i] : i) = src row (d_src_index ? d_src_index[i] : i).
 * src, dst: DEVICE pointers, rows of row_bytes bytes at src_stride /
 * dst_stride bytes apart (row_bytes and strides multiples of 16, pointers
 * 16-byte aligned); the index arrays are DEVICE int32 (or NULL), and the
 * source / destination hold n_src_rows / n_dst_rows rows.  An index outside
 * them skips the row and latches WST_ERR_INVALID_ARG in `workspace` (a
 * zero-filled workspace of at least wst_workspace_size(0, 0, 0) bytes) for
 * wst_sync_status.  Asynchronous on `stream`.
 */
wst_status wst_permute_rows(int n_rows, size_t row_bytes, const void* src, size_t src_stride,
                            const int* d_src_index, int n_src_rows, void* dst, size_t dst_stride,
                            const int* d_dst_index, int n_dst_rows, void* workspace, void* stream);

/*
 * IKBO linear compression.  Candidates of user u are [off[u], off[u+1]) of
 * the DEVICE int32 array d_user_offsets (num_users+1 entries, non-decreasing,
 * from 0 to num_cand).  For every candidate c of user u:
 *   Y[c][o][d] = sum_{f<Du} W[o][f] U[u][f][d] + sum_{f<Dc} W[o][Du+f] Cf[c][f][d]
 *   U   bf16 [num_users][Du][D]   (d contiguous)
 *   Cf  bf16 [num_cand][Dc][D]    (d contiguous)
 *   W   bf16 [O][Du+Dc]           (user columns first)
 *   Y   fp32 [num_cand][O][D]     (d contiguous)
 * The user part P[u] = W[:, :Du].U[u] is computed once per user per call
 * into the workspace and added to each of that user's candidates inside the
 * kernel; the broadcast user features are never materialised.
 * This build supports D == 128, O a multiple of 32 up to 256, Du and Dc
 * multiples of 8 with Du + Dc <= 512 (else WST_ERR_UNSUPPORTED).  The
 * kernel is a cooperative launch: all of its CTAs are resident at once.
 */
wst_status wst_ikbo_linear_compress(int num_users, int num_cand, int Du, int Dc,
                                    int D, int O,
                                    const void* U, const void* Cf, const void* W,
                                    const int* d_user_offsets,
                                    void* Y, void* workspace, void* stream);

/*
 * Allocation-free form of wst_ikbo_linear_compress (the pages have no
 * counterpart; this is a library convenience).  For callers that cannot
 * allocate device memory when they call -- code under a fixed memory budget,
 * behind an allocator it must not bypass, or inside a host framework that
 * owns every allocation -- the per-user partial products, ready flags and
 * error word live in a device array inside the library instead of a
 * caller-owned workspace.  Same arguments and results as
 * wst_ikbo_linear_compress, minus the workspace, plus:
 *   d_status  optional DEVICE int32 (NULL to skip) that receives this call's
 *             device-side status (0, WST_ERR_TIMEOUT or WST_ERR_BAD_OFFSETS)
 *             once the call's work on `stream` has run.
 * Limits and behaviour:
 *  - The array holds 4 MiB on every GPU that loads the library, until the
 *    process exits; wst_workspace_size(num_users, O, D) must not exceed it
 *    (64 users at O = 32, D = 128 need about 1 MiB).  Larger requests return
 *    WST_ERR_INVALID_ARG before anything is enqueued.
 *  - The call allocates and frees nothing.  Its first call on a device (and
 *    the first after a cudaDeviceReset, which gives the device a new
 *    context) looks up the array's device address with cudaGetSymbolAddress
 *    and caches it for that context; make that first call before any stream
 *    capture.  If it comes while `stream` is being captured, the call returns
 *    WST_ERR_UNSUPPORTED and enqueues nothing.
 *  - Every call on a device shares the one array and clears its header and
 *    flags at the start: calls that can overlap on the GPU (other streams,
 *    other host threads) race and must be serialised by the caller.
 */
wst_status wst_ikbo_linear_compress_noalloc(int num_users, int num_cand, int Du, int Dc,
                                            int D, int O,
                                            const void* U, const void* Cf, const void* W,
                                            const int* d_user_offsets, void* Y,
                                            int* d_status, void* stream);

/*
 * IKBO attention ("How We Built TLX: A Hardware-Native GPU Compiler for
 * Production ML at Scale", Case Study 2, which names an IKBO form of
 * FlashAttention whose key/value reads are shared by the candidates of one
 * user; the pages give no formula, and the reading implemented is below).
 * Candidates of user u are [off[u], off[u+1]) of the DEVICE int32 array
 * d_user_offsets (num_users+1 entries, non-decreasing, from 0 to num_cand);
 * candidate c owns the Lq query rows [c*Lq, (c+1)*Lq).  For every query row r
 * of a candidate of user u and every head h:
 *   O[r][h][:] = sum_j softmax_j(scale * Q[r][h][:] . K[u][j][h][:]) V[u][j][h][:]
 * over all Lkv context rows j of user u (no mask).
 *   Q   bf16 [num_cand*Lq][H][Dh]    (Dh contiguous)
 *   K   bf16 [num_users][Lkv][H][Dh]
 *   V   bf16 [num_users][Lkv][H][Dh]
 *   O   o_type [num_cand*Lq][H][Dh]  (fp32 or bf16)
 *   scale  any finite float (1/sqrt(Dh) is the usual choice)
 * The query rows of all candidates of a user are processed together in
 * 128-row tiles, so each user's K/V is read once per tile and per head, not
 * once per candidate.  The probabilities are rounded to bf16 before the
 * product with V; row maxima, sums and the output accumulate in fp32.
 * This build supports Dh == 128 (else WST_ERR_UNSUPPORTED) and needs
 * num_cand*Lq < 2^31.  Offsets that break the rule are clamped into range on
 * the device and latched as WST_ERR_BAD_OFFSETS.
 * workspace: 16-byte aligned, zero-filled once (wst_workspace_init) and
 * then reused; `workspace_bytes` says how large it is.  With at least
 * wst_ikbo_attention_workspace_size() bytes the items (user, head, 128-row
 * query tile) of the last partial wave of the persistent grid are split by
 * key blocks over all CTAs and their partial results merged through the
 * workspace (so the result of a split item is summed in another order);
 * with less (at least the 256-byte error-word header) whole items only.
 * One call at a time per workspace.
 */
wst_status wst_ikbo_attention_bf16(int num_users, int num_cand, int Lq, int H, int Dh, int Lkv,
                                   const void* Q, const void* K, const void* V,
                                   const int* d_user_offsets, float scale,
                                   void* O, wst_dtype o_type, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* Workspace bytes for wst_ikbo_attention_bf16's split schedule (header,
 * per-CTA flags and one partial O/m/l slot per CTA, for up to 256 CTAs). */
size_t wst_ikbo_attention_workspace_size(void);

/* Synchronize `stream`, then return and clear the first device-side error
 * latched in `workspace` (WST_OK if none). */
wst_status wst_sync_status(void* workspace, void* stream);

/* Static description of a status code. */
const char* wst_status_string(wst_status s);

/* Text of the last host-side error on the calling thread ("" if none). */
const char* wst_last_error(void);

/* Library version string. */
const char* wst_version(void);

#ifdef __cplusplus
}
#endif

#endif /* WST_H_ */
