// wst_host.h -- host-side helpers shared by the launchers and the C ABI:
// tensor-map encoding (driver entry point fetched through the runtime, so
// the library loads on machines without a driver), device properties, the
// thread-local error message, and the problem descriptions handed from the
// validating ABI layer to the per-kernel launchers.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace wst {

// Status codes, identical to wst_status in include/wst.h.
enum Status : int {
  ST_OK = 0,
  ST_INVALID_ARG = 1,
  ST_ALIGNMENT = 2,
  ST_UNSUPPORTED = 3,
  ST_CUDA = 4,
  ST_TIMEOUT = 5,
  ST_BAD_OFFSETS = 6,
};

void set_error(const char* fmt, ...);
int cuda_fail(cudaError_t e, const char* what);  // records the message, returns ST_CUDA

struct DeviceInfo {
  int device;
  int num_sms;
  int max_smem_optin;
};
int current_device_info(DeviceInfo* out);  // Status

// Process-wide tuning options (wst_option in include/wst.h).
enum Option : int {
  OPT_GROUPED_SCHEDULE = 0,
  OPT_DENSE_CTA_GROUP = 1,
  OPT_IKBO_SCHEDULE = 2,
  OPT_NORM_STATS = 3,
  OPT_COUNT = 4
};
int option_value(int opt);

unsigned long long wait_timeout_ns();
// A fresh nonzero value for the cross-CTA ready flags of one call (IKBO
// partials, split attention items): a process-wide counter, so flags left in
// a workspace by earlier calls never equal it (zeroed workspaces hold 0).
uint32_t next_flag_epoch();

// Test hook for the bounded-wait error path: when the environment variable
// WST_FAULT_INJECT=drop_load is set, the first dense GEMM launch of the
// process (only that one) leaves one K-block unloaded, so its MMA issuer's
// bounded wait runs out and the call latches WST_ERR_TIMEOUT.  No fault,
// trap or hang: the kernel exits cleanly and later calls are normal.
bool take_fault_injection();

// Raise a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device (cached: the attribute call is made once per kernel,
// device and size).  Returns Status.
int ensure_smem_attr(const void* kernel, size_t bytes);

// Encode a tiled tensor map (rank 2 or 3).  dims / box innermost first,
// strides_bytes has rank-1 entries.  Returns Status.
int encode_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr,
               const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
               CUtensorMapSwizzle sw);

struct GemmProblem {
  int grouped;     // 0 dense / batched, 1 grouped
  int batch;       // dense: batch count; grouped: G
  int M, N, K;     // grouped: M = M_total
  const void* A;
  long long lda, strideA;
  const void* B;
  long long ldb, strideB;  // grouped: strideB = per-group stride
  const void* bias;
  long long strideBias;
  void* C;
  long long ldc, strideC;
  int c_f32;
  int epi;
  const int* offsets;
  void* ws;
  int norm;    // dense only: 1 RMSNorm, 2 LayerNorm of the rows of A
  float eps;
  const float* colsum;        // LayerNorm: column sums of B, [batch][N] (stride 0: shared)
  long long colsum_stride;
  const float2* row_stats;    // norm 3 / 4: precomputed (r, r*mu) per row of A
  long long row_stats_stride;
};

struct IkboProblem {
  int num_users, num_cand, Du, Dc, D, O;
  const void* U;
  const void* Cf;
  const void* W;
  const int* uoff;
  void* Y;
  void* ws;
};

// IKBO attention: Q [num_cand*Lq][H][Dh], K/V [num_users][Lkv][H][Dh] (bf16),
// O [num_cand*Lq][H][Dh] (fp32 or bf16).
struct AttnProblem {
  int num_users, num_cand, Lq, H, Dh, Lkv;
  const void* Q;
  const void* K;
  const void* V;
  const int* uoff;
  float scale;
  void* O;
  bool o_f32;
  void* ws;
  size_t ws_bytes;
};

int run_gemm(const GemmProblem& p, cudaStream_t stream);
// s[b][n] = sum_k B[b][n][k] in fp32 for b < nb (LayerNorm fusion).
// Passes over rows of bf16 data ahead of the norm GEMMs, one launch: the
// row statistics (r, r*mu) of nb_a x M rows of A into stats (none when stats
// is NULL) and the column sums of nb_b x N rows of B into colsum, batch entry
// b's row starting at b * colsum_stride floats (none when colsum is NULL).
struct NormPass {
  const void* A;
  long long lda, strideA;
  int nb_a, M, K;
  float eps;
  bool layernorm;
  float2* stats;
  const void* B;
  long long ldb, strideB;
  int nb_b, N;
  long long colsum_stride;
  float* colsum;
};
int run_norm_pass(const NormPass& np, cudaStream_t stream);
int run_ikbo_attention(const AttnProblem& p, cudaStream_t stream);
size_t attention_workspace_bytes();
int run_ikbo(const IkboProblem& p, cudaStream_t stream);
int run_ikbo_noalloc(IkboProblem p, int* d_status, cudaStream_t stream);
size_t ikbo_noalloc_capacity();

}  // namespace wst
