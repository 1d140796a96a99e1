// wst_api.cu -- the C ABI (include/wst.h): argument validation, status
// handling, and the host helpers declared in wst_host.h.
//
// Every entry point validates on the host and returns a status before
// anything is enqueued; nothing here throws, aborts, allocates device memory
// or runs any part of the computation on the CPU.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "wst.h"
#include "wst_common.cuh"
#include "wst_host.h"

namespace wst {

namespace {
thread_local char g_err[512];

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeFn g_encode = nullptr;

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ok[kMaxDevices];
std::mutex g_dev_mu;
}  // namespace

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
}

int cuda_fail(cudaError_t e, const char* what) {
  set_error("%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
  return ST_CUDA;
}

uint32_t next_flag_epoch() {
  static std::atomic<uint32_t> counter{0};
  uint32_t e = counter.fetch_add(1u, std::memory_order_relaxed) + 1u;
  if (e == 0u) e = counter.fetch_add(1u, std::memory_order_relaxed) + 1u;  // skip 0 on wrap
  return e;
}

int current_device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("device ordinal %d out of range", dev);
    return ST_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_dev_ok[dev]) {
    int major = 0, minor = 0, sms = 0, smem = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) ||
        (e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)))
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3) {
      set_error("libwst is built for sm_103a (GB300); device %d is sm_%d%d", dev, major, minor);
      return ST_UNSUPPORTED;
    }
    g_dev[dev] = DeviceInfo{dev, sms, smem};
    g_dev_ok[dev] = true;
  }
  *out = g_dev[dev];
  return ST_OK;
}

namespace {
std::atomic<int> g_options[OPT_COUNT];  // zero-initialised: every option's default is 0
}  // namespace

int option_value(int opt) {
  return (opt >= 0 && opt < OPT_COUNT) ? g_options[opt].load(std::memory_order_relaxed) : 0;
}

unsigned long long wait_timeout_ns() {
  static unsigned long long v = [] {
    const char* s = std::getenv("WST_TIMEOUT_MS");
    long long ms = s ? std::atoll(s) : 0;
    if (ms <= 0) ms = 2000;
    return (unsigned long long)ms * 1000000ull;
  }();
  return v;
}

bool take_fault_injection() {
  static const bool armed = [] {
    const char* s = std::getenv("WST_FAULT_INJECT");
    return s && std::strcmp(s, "drop_load") == 0;
  }();
  static std::atomic<int> used{0};
  return armed && used.fetch_add(1) == 0;
}

int ensure_smem_attr(const void* kernel, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> done;
  std::lock_guard<std::mutex> lk(mu);
  size_t& have = done[std::make_pair(kernel, dev)];
  if (have >= bytes) return ST_OK;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  have = bytes;
  return ST_OK;
}

int encode_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr,
               const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
               CUtensorMapSwizzle sw) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeFn>(fn);
  });
  if (!g_encode) {
    set_error("cuTensorMapEncodeTiled is not available from the CUDA driver");
    return ST_CUDA;
  }
  cuuint64_t d[5];
  cuuint64_t s[4];
  cuuint32_t b[5];
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) s[i] = strides_bytes[i];
  CUresult r = g_encode(m, dt, (cuuint32_t)rank, const_cast<void*>(ptr), d, s, b, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (CUresult %d, rank %d)", (int)r, rank);
    return ST_CUDA;
  }
  return ST_OK;
}

}  // namespace wst

using namespace wst;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The pointer must be memory the GPU addresses as device memory.
int check_device_ptr(const void* p, const char* name) {
  if (!p) {
    set_error("%s is NULL", name);
    return ST_INVALID_ARG;
  }
  cudaPointerAttributes at{};
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    set_error("%s: not a CUDA pointer (%s)", name, cudaGetErrorString(e));
    return ST_INVALID_ARG;
  }
  if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) {
    set_error("%s must be device (or managed) memory", name);
    return ST_INVALID_ARG;
  }
  return ST_OK;
}

#define WST_TRY(expr)            \
  do {                           \
    int st__ = (expr);           \
    if (st__) return (wst_status)st__; \
  } while (0)

wst_status fail(wst_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  char buf[512];
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  set_error("%s", buf);
  return s;
}

}  // namespace

extern "C" {

size_t wst_workspace_size(int num_users, int O, int D) {
  if (num_users < 0 || O < 0 || D < 0) return 0;
  return workspace_bytes(num_users, O, D);
}

wst_status wst_workspace_init(void* workspace, size_t bytes, void* stream) {
  g_err[0] = 0;
  if (bytes < kWsHeaderBytes) return fail(WST_ERR_INVALID_ARG, "workspace smaller than %zu bytes", kWsHeaderBytes);
  WST_TRY(check_device_ptr(workspace, "workspace"));
  cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return (wst_status)cuda_fail(e, "cudaMemsetAsync(workspace)");
  return WST_OK;
}

static wst_status validate_common(int epi, int c_type, const void* ws) {
  if (epi < 0 || epi > 3) return fail(WST_ERR_INVALID_ARG, "unknown epilogue %d", epi);
  if (c_type != WST_F32 && c_type != WST_BF16) return fail(WST_ERR_INVALID_ARG, "unknown c_type %d", c_type);
  if (!ws) return fail(WST_ERR_INVALID_ARG, "workspace is NULL");
  if (!aligned16(ws)) return fail(WST_ERR_ALIGNMENT, "workspace not 16-byte aligned");
  return WST_OK;
}

wst_status wst_gemm_bf16(int batch, int M, int N, int K, const void* A, long lda, long strideA,
                         const void* B, long ldb, long strideB, const void* bias, long strideBias,
                         void* C, long ldc, long strideC, wst_dtype c_type, wst_epilogue epi,
                         void* workspace, void* stream) {
  g_err[0] = 0;
  wst_status s = validate_common((int)epi, (int)c_type, workspace);
  if (s) return s;
  if (batch < 1 || M < 1 || N < 1 || K < 1)
    return fail(WST_ERR_INVALID_ARG, "sizes must be >= 1 (batch=%d M=%d N=%d K=%d)", batch, M, N, K);
  if (!A || !B || !C) return fail(WST_ERR_INVALID_ARG, "A, B and C must be non-NULL");
  if (lda < K || ldb < K || ldc < N)
    return fail(WST_ERR_INVALID_ARG, "leading dimensions too small (lda=%ld ldb=%ld ldc=%ld)", lda, ldb, ldc);
  if (strideA < 0 || strideB < 0 || strideC < 0 || strideBias < 0)
    return fail(WST_ERR_INVALID_ARG, "negative batch stride");
  const long es = c_type == WST_F32 ? 4 : 2;
  if (batch > 1 && strideC < (long)(M - 1) * ldc + N)
    return fail(WST_ERR_INVALID_ARG, "strideC=%ld makes batch outputs overlap", strideC);
  if (epi != WST_EPI_NONE && !bias) return fail(WST_ERR_INVALID_ARG, "epilogue needs a bias");
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || (epi && !aligned16(bias)))
    return fail(WST_ERR_ALIGNMENT, "A, B, C and bias must be 16-byte aligned");
  if ((lda * 2) % 16 || (ldb * 2) % 16 || (ldc * es) % 16 || (strideA * 2) % 16 ||
      (strideB * 2) % 16 || (strideC * es) % 16 || (epi && (strideBias * 2) % 16))
    return fail(WST_ERR_ALIGNMENT, "leading dimensions and batch strides must be multiples of 16 bytes");
  WST_TRY(check_device_ptr(A, "A"));
  WST_TRY(check_device_ptr(B, "B"));
  WST_TRY(check_device_ptr(C, "C"));
  if (epi) WST_TRY(check_device_ptr(bias, "bias"));
  WST_TRY(check_device_ptr(workspace, "workspace"));

  GemmProblem p{};
  p.grouped = 0;
  p.batch = batch;
  p.M = M;
  p.N = N;
  p.K = K;
  p.A = A;
  p.lda = lda;
  p.strideA = batch > 1 ? strideA : 0;
  p.B = B;
  p.ldb = ldb;
  p.strideB = batch > 1 ? strideB : 0;
  p.bias = epi ? bias : nullptr;
  p.strideBias = strideBias;
  p.C = C;
  p.ldc = ldc;
  p.strideC = batch > 1 ? strideC : 0;
  p.c_f32 = c_type == WST_F32;
  p.epi = (int)epi;
  p.offsets = nullptr;
  p.ws = workspace;
  return (wst_status)run_gemm(p, static_cast<cudaStream_t>(stream));
}

namespace {

// Validation and problem set-up shared by the normalised-row GEMMs.
wst_status norm_gemm_problem(const char* what, int batch, int M, int N, int K, const void* A,
                             long lda, long strideA, const void* B, long ldb, long strideB,
                             float eps, const void* bias, long strideBias, void* C, long ldc,
                             long strideC, wst_dtype c_type, wst_epilogue epi, void* workspace,
                             GemmProblem& p) {
  if (!(eps >= 0.0f) || eps > 3.0e38f) return fail(WST_ERR_INVALID_ARG, "%s: eps must be finite and >= 0", what);
  wst_status s = validate_common((int)epi, (int)c_type, workspace);
  if (s) return s;
  if (batch < 1 || M < 1 || N < 1 || K < 1)
    return fail(WST_ERR_INVALID_ARG, "sizes must be >= 1 (batch=%d M=%d N=%d K=%d)", batch, M, N, K);
  if (!A || !B || !C) return fail(WST_ERR_INVALID_ARG, "A, B and C must be non-NULL");
  if (lda < K || ldb < K || ldc < N)
    return fail(WST_ERR_INVALID_ARG, "leading dimensions too small (lda=%ld ldb=%ld ldc=%ld)", lda, ldb, ldc);
  if (strideA < 0 || strideB < 0 || strideC < 0 || strideBias < 0)
    return fail(WST_ERR_INVALID_ARG, "negative batch stride");
  const long es = c_type == WST_F32 ? 4 : 2;
  if (batch > 1 && strideC < (long)(M - 1) * ldc + N)
    return fail(WST_ERR_INVALID_ARG, "strideC=%ld makes batch outputs overlap", strideC);
  if (epi != WST_EPI_NONE && !bias) return fail(WST_ERR_INVALID_ARG, "epilogue needs a bias");
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || (epi && !aligned16(bias)))
    return fail(WST_ERR_ALIGNMENT, "A, B, C and bias must be 16-byte aligned");
  if ((lda * 2) % 16 || (ldb * 2) % 16 || (ldc * es) % 16 || (strideA * 2) % 16 ||
      (strideB * 2) % 16 || (strideC * es) % 16 || (epi && (strideBias * 2) % 16))
    return fail(WST_ERR_ALIGNMENT, "leading dimensions and batch strides must be multiples of 16 bytes");
  WST_TRY(check_device_ptr(A, "A"));
  WST_TRY(check_device_ptr(B, "B"));
  WST_TRY(check_device_ptr(C, "C"));
  if (epi) WST_TRY(check_device_ptr(bias, "bias"));
  WST_TRY(check_device_ptr(workspace, "workspace"));

  p = GemmProblem{};
  p.grouped = 0;
  p.batch = batch;
  p.M = M;
  p.N = N;
  p.K = K;
  p.A = A;
  p.lda = lda;
  p.strideA = batch > 1 ? strideA : 0;
  p.B = B;
  p.ldb = ldb;
  p.strideB = batch > 1 ? strideB : 0;
  p.bias = epi ? bias : nullptr;
  p.strideBias = strideBias;
  p.C = C;
  p.ldc = ldc;
  p.strideC = batch > 1 ? strideC : 0;
  p.c_f32 = c_type == WST_F32;
  p.epi = (int)epi;
  p.offsets = nullptr;
  p.ws = workspace;
  p.eps = eps;
  return WST_OK;
}

// fp32 column sums of B per batch row, padded to a multiple of 4 floats.
inline long long colsum_stride(int N) { return ((long long)N + 3) & ~3LL; }

// Bytes of the LayerNorm column sums after the header (0 for RMSNorm).
long long colsum_bytes(int batch, int N, long strideB) {
  const long long rows = (batch > 1 && strideB != 0) ? batch : 1;
  return rows * colsum_stride(N) * 4;
}

// Rows of precomputed statistics: one per row of A (one batch's worth when
// A is shared by the batch), 8 bytes each (r, r*mu), 16-byte aligned after
// the header and the column sums.
long long stats_rows(int batch, int M, long strideA) {
  return (batch > 1 && strideA != 0) ? (long long)batch * M : (long long)M;
}
long long stats_offset(int batch, int N, long strideB, bool layernorm) {
  const long long off = (long long)kWsHeaderBytes + (layernorm ? colsum_bytes(batch, N, strideB) : 0);
  return (off + 15) & ~15LL;
}

// Statistics precomputed by a pass over A (NORM 3 / 4) or gathered in the
// GEMM from the A tiles (NORM 1 / 2).  In the GEMM every tile recomputes its
// rows' statistics, once per 256 columns of N; the pass reads A once more,
// whose cost relative to the GEMM falls as 1/N.  Measured on GB300 (M 8192,
// K 4096): LayerNorm's in-GEMM statistics (three operations per pair of
// elements) lose from N = 1024 (0.0640 vs 0.0598 ms) and RMSNorm's (one)
// only above N = 2048 (N = 2048: 0.0962 vs 0.0997 ms; 4096: 0.1640 vs
// 0.1618 ms; 8192^3: 0.655 vs 0.617 ms).  So the automatic choice takes the
// pass for N > 512 (LayerNorm) or N > 2048 (RMSNorm) when the workspace
// holds the statistics.
int choose_prestats(const GemmProblem& p, bool layernorm, size_t workspace_bytes, bool& pre) {
  const int opt = option_value(OPT_NORM_STATS);
  const long long need = stats_offset(p.batch, p.N, p.strideB, layernorm) +
                         8 * stats_rows(p.batch, p.M, p.strideA);
  const bool fits = workspace_bytes >= (size_t)need;
  if (opt == 2 && !fits)
    return fail(WST_ERR_INVALID_ARG, "%s: precomputed statistics need a workspace of %lld bytes, %zu given",
                layernorm ? "layernorm" : "rmsnorm", need, workspace_bytes);
  pre = fits && (opt == 2 || (opt == 0 && p.N > (layernorm ? 512 : 2048)));
  return WST_OK;
}

// Adds the statistics of A to the pass and points the GEMM (NORM 3 / 4) at
// them: one batch's rows when A is shared by the batch.
void plan_prestats(GemmProblem& p, bool layernorm, NormPass& np) {
  const bool shared_a = !(p.batch > 1 && p.strideA != 0);
  float2* out = reinterpret_cast<float2*>(static_cast<uint8_t*>(p.ws) +
                                          stats_offset(p.batch, p.N, p.strideB, layernorm));
  np.A = p.A;
  np.lda = p.lda;
  np.strideA = shared_a ? 0 : p.strideA;
  np.nb_a = shared_a ? 1 : p.batch;
  np.M = p.M;
  np.K = p.K;
  np.eps = p.eps;
  np.layernorm = layernorm;
  np.stats = out;
  p.row_stats = out;
  p.row_stats_stride = shared_a ? 0 : p.M;
  p.norm = layernorm ? 4 : 3;
}

}  // namespace

size_t wst_gemm_norm_workspace_size(int batch, int M, int N, long strideA, long strideB,
                                    int layernorm) {
  if (batch < 1 || M < 1 || N < 1 || strideA < 0 || strideB < 0) return 0;
  return (size_t)(stats_offset(batch, N, strideB, layernorm != 0) + 8 * stats_rows(batch, M, strideA));
}

wst_status wst_gemm_rmsnorm_bf16(int batch, int M, int N, int K, const void* A, long lda,
                                 long strideA, const void* B, long ldb, long strideB, float eps,
                                 const void* bias, long strideBias, void* C, long ldc,
                                 long strideC, wst_dtype c_type, wst_epilogue epi,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  g_err[0] = 0;
  if (workspace_bytes < kWsHeaderBytes)
    return fail(WST_ERR_INVALID_ARG, "rmsnorm: workspace of %zu bytes, %zu needed", workspace_bytes,
                kWsHeaderBytes);
  GemmProblem p;
  WST_TRY(norm_gemm_problem("rmsnorm", batch, M, N, K, A, lda, strideA, B, ldb, strideB, eps,
                            bias, strideBias, C, ldc, strideC, c_type, epi, workspace, p));
  bool pre = false;
  WST_TRY((wst_status)choose_prestats(p, false, workspace_bytes, pre));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  p.norm = 1;
  if (pre) {
    NormPass np{};
    plan_prestats(p, false, np);
    WST_TRY((wst_status)run_norm_pass(np, st));
  }
  return (wst_status)run_gemm(p, st);
}

size_t wst_gemm_layernorm_workspace_size(int batch, int N, long strideB) {
  if (batch < 1 || N < 1 || strideB < 0) return 0;
  return kWsHeaderBytes + (size_t)colsum_bytes(batch, N, strideB);
}

wst_status wst_gemm_layernorm_bf16(int batch, int M, int N, int K, const void* A, long lda,
                                   long strideA, const void* B, long ldb, long strideB, float eps,
                                   const void* bias, long strideBias, void* C, long ldc,
                                   long strideC, wst_dtype c_type, wst_epilogue epi,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  g_err[0] = 0;
  const size_t need = wst_gemm_layernorm_workspace_size(batch, N, strideB);
  if (need && workspace_bytes < need)
    return fail(WST_ERR_INVALID_ARG, "layernorm: workspace of %zu bytes, %zu needed", workspace_bytes, need);
  GemmProblem p;
  WST_TRY(norm_gemm_problem("layernorm", batch, M, N, K, A, lda, strideA, B, ldb, strideB, eps,
                            bias, strideBias, C, ldc, strideC, c_type, epi, workspace, p));
  const int nb = (batch > 1 && strideB != 0) ? batch : 1;
  float* s = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kWsHeaderBytes);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  bool pre = false;
  WST_TRY((wst_status)choose_prestats(p, true, workspace_bytes, pre));
  // the column sums of B, and with the separate pass the statistics of A,
  // in one launch
  NormPass np{};
  np.B = B;
  np.ldb = ldb;
  np.strideB = nb > 1 ? strideB : 0;
  np.nb_b = nb;
  np.N = N;
  np.K = K;
  np.layernorm = true;
  np.colsum_stride = colsum_stride(N);
  np.colsum = s;
  p.norm = 2;
  if (pre) plan_prestats(p, true, np);
  WST_TRY((wst_status)run_norm_pass(np, st));
  p.colsum = s;
  p.colsum_stride = nb > 1 ? colsum_stride(N) : 0;
  return (wst_status)run_gemm(p, st);
}

wst_status wst_grouped_gemm_bf16(int G, int M_total, int N, int K, const void* A, long lda,
                                 const void* B, long ldb, long strideB_group, const int* d_offsets,
                                 const void* bias, long strideBias, void* C, long ldc,
                                 wst_dtype c_type, wst_epilogue epi, void* workspace,
                                 void* stream) {
  g_err[0] = 0;
  wst_status s = validate_common((int)epi, (int)c_type, workspace);
  if (s) return s;
  if (G < 1 || M_total < 0 || N < 1 || K < 1)
    return fail(WST_ERR_INVALID_ARG, "sizes out of range (G=%d M_total=%d N=%d K=%d)", G, M_total, N, K);
  if (!A || !B || !C || !d_offsets) return fail(WST_ERR_INVALID_ARG, "A, B, C and offsets must be non-NULL");
  if (lda < K || ldb < K || ldc < N)
    return fail(WST_ERR_INVALID_ARG, "leading dimensions too small (lda=%ld ldb=%ld ldc=%ld)", lda, ldb, ldc);
  if (strideB_group < 0 || strideBias < 0) return fail(WST_ERR_INVALID_ARG, "negative group stride");
  if (epi != WST_EPI_NONE && !bias) return fail(WST_ERR_INVALID_ARG, "epilogue needs a bias");
  const long es = c_type == WST_F32 ? 4 : 2;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || (epi && !aligned16(bias)) ||
      (reinterpret_cast<uintptr_t>(d_offsets) & 3u))
    return fail(WST_ERR_ALIGNMENT, "A, B, C, bias must be 16-byte aligned and offsets 4-byte aligned");
  if ((lda * 2) % 16 || (ldb * 2) % 16 || (ldc * es) % 16 || (strideB_group * 2) % 16 ||
      (epi && (strideBias * 2) % 16))
    return fail(WST_ERR_ALIGNMENT, "leading dimensions and strides must be multiples of 16 bytes");
  WST_TRY(check_device_ptr(A, "A"));
  WST_TRY(check_device_ptr(B, "B"));
  WST_TRY(check_device_ptr(C, "C"));
  WST_TRY(check_device_ptr(d_offsets, "d_offsets"));
  if (epi) WST_TRY(check_device_ptr(bias, "bias"));
  WST_TRY(check_device_ptr(workspace, "workspace"));
  if (M_total == 0) return WST_OK;  // no rows: nothing to compute or store

  GemmProblem p{};
  p.grouped = 1;
  p.batch = G;
  p.M = M_total;
  p.N = N;
  p.K = K;
  p.A = A;
  p.lda = lda;
  p.strideA = 0;
  p.B = B;
  p.ldb = ldb;
  p.strideB = G > 1 ? strideB_group : 0;
  p.bias = epi ? bias : nullptr;
  p.strideBias = strideBias;
  p.C = C;
  p.ldc = ldc;
  p.strideC = 0;
  p.c_f32 = c_type == WST_F32;
  p.epi = (int)epi;
  p.offsets = d_offsets;
  p.ws = workspace;
  return (wst_status)run_gemm(p, static_cast<cudaStream_t>(stream));
}

wst_status wst_ikbo_attention_bf16(int num_users, int num_cand, int Lq, int H, int Dh, int Lkv,
                                   const void* Q, const void* K, const void* V,
                                   const int* d_user_offsets, float scale, void* O,
                                   wst_dtype o_type, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  g_err[0] = 0;
  if (workspace_bytes < kWsHeaderBytes)
    return fail(WST_ERR_INVALID_ARG, "attention: workspace of %zu bytes (at least %zu)",
                workspace_bytes, kWsHeaderBytes);
  if (num_users < 1 || num_cand < 0 || Lq < 1 || H < 1 || Dh < 1 || Lkv < 1)
    return fail(WST_ERR_INVALID_ARG, "sizes out of range (users=%d cand=%d Lq=%d H=%d Dh=%d Lkv=%d)",
                num_users, num_cand, Lq, H, Dh, Lkv);
  if (o_type != WST_F32 && o_type != WST_BF16) return fail(WST_ERR_INVALID_ARG, "unknown o_type %d", (int)o_type);
  if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f)
    return fail(WST_ERR_INVALID_ARG, "scale must be finite");
  if (!Q || !K || !V || !d_user_offsets || !O || !workspace)
    return fail(WST_ERR_INVALID_ARG, "Q, K, V, offsets, O and workspace must be non-NULL");
  if (Dh != 128) return fail(WST_ERR_UNSUPPORTED, "Dh=%d: this build supports Dh == 128", Dh);
  if ((long long)num_cand * Lq > 0x7fffffffLL)
    return fail(WST_ERR_UNSUPPORTED, "num_cand*Lq = %lld query rows: needs < 2^31", (long long)num_cand * Lq);
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(d_user_offsets) & 3u))
    return fail(WST_ERR_ALIGNMENT, "Q, K, V, O, workspace must be 16-byte aligned, offsets 4-byte");
  WST_TRY(check_device_ptr(Q, "Q"));
  WST_TRY(check_device_ptr(K, "K"));
  WST_TRY(check_device_ptr(V, "V"));
  WST_TRY(check_device_ptr(O, "O"));
  WST_TRY(check_device_ptr(d_user_offsets, "d_user_offsets"));
  WST_TRY(check_device_ptr(workspace, "workspace"));
  if (num_cand == 0) return WST_OK;  // no query rows: nothing to output

  AttnProblem p{};
  p.num_users = num_users;
  p.num_cand = num_cand;
  p.Lq = Lq;
  p.H = H;
  p.Dh = Dh;
  p.Lkv = Lkv;
  p.Q = Q;
  p.K = K;
  p.V = V;
  p.uoff = d_user_offsets;
  p.scale = scale;
  p.O = O;
  p.o_f32 = o_type == WST_F32;
  p.ws = workspace;
  p.ws_bytes = workspace_bytes;
  return (wst_status)run_ikbo_attention(p, static_cast<cudaStream_t>(stream));
}

size_t wst_ikbo_attention_workspace_size(void) { return attention_workspace_bytes(); }

wst_status wst_ikbo_linear_compress(int num_users, int num_cand, int Du, int Dc, int D, int O,
                                    const void* U, const void* Cf, const void* W,
                                    const int* d_user_offsets, void* Y, void* workspace,
                                    void* stream) {
  g_err[0] = 0;
  if (num_users < 1 || num_cand < 0 || Du < 1 || Dc < 1 || D < 1 || O < 1)
    return fail(WST_ERR_INVALID_ARG, "sizes out of range (users=%d cand=%d Du=%d Dc=%d D=%d O=%d)",
                num_users, num_cand, Du, Dc, D, O);
  if (!U || !Cf || !W || !d_user_offsets || !Y || !workspace)
    return fail(WST_ERR_INVALID_ARG, "U, Cf, W, offsets, Y and workspace must be non-NULL");
  if (D != 128) return fail(WST_ERR_UNSUPPORTED, "D=%d: this build supports D == 128", D);
  if (O % 32 || O > 256) return fail(WST_ERR_UNSUPPORTED, "O=%d: needs a multiple of 32 up to 256", O);
  if (Du % 8 || Dc % 8) return fail(WST_ERR_UNSUPPORTED, "Du=%d, Dc=%d: need multiples of 8", Du, Dc);
  if (Du + Dc > 512) return fail(WST_ERR_UNSUPPORTED, "Du + Dc = %d > 512", Du + Dc);
  if (!aligned16(U) || !aligned16(Cf) || !aligned16(W) || !aligned16(Y) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(d_user_offsets) & 3u))
    return fail(WST_ERR_ALIGNMENT, "U, Cf, W, Y, workspace must be 16-byte aligned, offsets 4-byte");
  WST_TRY(check_device_ptr(U, "U"));
  WST_TRY(check_device_ptr(Cf, "Cf"));
  WST_TRY(check_device_ptr(W, "W"));
  WST_TRY(check_device_ptr(Y, "Y"));
  WST_TRY(check_device_ptr(d_user_offsets, "d_user_offsets"));
  WST_TRY(check_device_ptr(workspace, "workspace"));
  if (num_cand == 0) return WST_OK;  // no candidates: nothing to output

  IkboProblem p{};
  p.num_users = num_users;
  p.num_cand = num_cand;
  p.Du = Du;
  p.Dc = Dc;
  p.D = D;
  p.O = O;
  p.U = U;
  p.Cf = Cf;
  p.W = W;
  p.uoff = d_user_offsets;
  p.Y = Y;
  p.ws = workspace;
  return (wst_status)run_ikbo(p, static_cast<cudaStream_t>(stream));
}

wst_status wst_ikbo_linear_compress_noalloc(int num_users, int num_cand, int Du, int Dc, int D,
                                            int O, const void* U, const void* Cf, const void* W,
                                            const int* d_user_offsets, void* Y, int* d_status,
                                            void* stream) {
  g_err[0] = 0;
  if (num_users < 1 || num_cand < 0 || Du < 1 || Dc < 1 || D < 1 || O < 1)
    return fail(WST_ERR_INVALID_ARG, "sizes out of range (users=%d cand=%d Du=%d Dc=%d D=%d O=%d)",
                num_users, num_cand, Du, Dc, D, O);
  if (!U || !Cf || !W || !d_user_offsets || !Y)
    return fail(WST_ERR_INVALID_ARG, "U, Cf, W, offsets and Y must be non-NULL");
  if (D != 128) return fail(WST_ERR_UNSUPPORTED, "D=%d: this build supports D == 128", D);
  if (O % 32 || O > 256) return fail(WST_ERR_UNSUPPORTED, "O=%d: needs a multiple of 32 up to 256", O);
  if (Du % 8 || Dc % 8) return fail(WST_ERR_UNSUPPORTED, "Du=%d, Dc=%d: need multiples of 8", Du, Dc);
  if (Du + Dc > 512) return fail(WST_ERR_UNSUPPORTED, "Du + Dc = %d > 512", Du + Dc);
  if (workspace_bytes(num_users, O, D) > ikbo_noalloc_capacity())
    return fail(WST_ERR_INVALID_ARG,
                "%d users x O=%d x D=%d need %zu bytes of scratch; the allocation-free entry point "
                "holds %zu bytes (use wst_ikbo_linear_compress with a workspace)",
                num_users, O, D, workspace_bytes(num_users, O, D), ikbo_noalloc_capacity());
  if (!aligned16(U) || !aligned16(Cf) || !aligned16(W) || !aligned16(Y) ||
      (reinterpret_cast<uintptr_t>(d_user_offsets) & 3u) ||
      (reinterpret_cast<uintptr_t>(d_status) & 3u))
    return fail(WST_ERR_ALIGNMENT, "U, Cf, W, Y must be 16-byte aligned, offsets and status 4-byte");
  WST_TRY(check_device_ptr(U, "U"));
  WST_TRY(check_device_ptr(Cf, "Cf"));
  WST_TRY(check_device_ptr(W, "W"));
  WST_TRY(check_device_ptr(Y, "Y"));
  WST_TRY(check_device_ptr(d_user_offsets, "d_user_offsets"));
  if (d_status) WST_TRY(check_device_ptr(d_status, "d_status"));
  if (num_cand == 0) {
    if (d_status) {
      cudaError_t e = cudaMemsetAsync(d_status, 0, sizeof(int), static_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) return (wst_status)cuda_fail(e, "cudaMemsetAsync(status)");
    }
    return WST_OK;
  }
  IkboProblem p{};
  p.num_users = num_users;
  p.num_cand = num_cand;
  p.Du = Du;
  p.Dc = Dc;
  p.D = D;
  p.O = O;
  p.U = U;
  p.Cf = Cf;
  p.W = W;
  p.uoff = d_user_offsets;
  p.Y = Y;
  p.ws = nullptr;
  return (wst_status)run_ikbo_noalloc(p, d_status, static_cast<cudaStream_t>(stream));
}

wst_status wst_sync_status(void* workspace, void* stream) {
  g_err[0] = 0;
  if (!workspace) return fail(WST_ERR_INVALID_ARG, "workspace is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return (wst_status)cuda_fail(e, "cudaStreamSynchronize");
  uint32_t hdr[2] = {0, 0};
  e = cudaMemcpyAsync(hdr, workspace, sizeof hdr, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return (wst_status)cuda_fail(e, "reading the workspace error word");
  if (hdr[0] == 0) return WST_OK;
  e = cudaMemsetAsync(workspace, 0, sizeof hdr, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return (wst_status)cuda_fail(e, "clearing the workspace error word");
  set_error("device error %u (info 0x%08x)", hdr[0], hdr[1]);
  if (hdr[0] == WST_ERR_TIMEOUT || hdr[0] == WST_ERR_BAD_OFFSETS || hdr[0] == WST_ERR_INVALID_ARG)
    return (wst_status)hdr[0];
  return WST_ERR_CUDA;
}

const char* wst_status_string(wst_status s) {
  switch (s) {
    case WST_OK: return "WST_OK";
    case WST_ERR_INVALID_ARG: return "WST_ERR_INVALID_ARG: an argument is out of range";
    case WST_ERR_ALIGNMENT: return "WST_ERR_ALIGNMENT: pointer or stride breaks the 16-byte rule";
    case WST_ERR_UNSUPPORTED: return "WST_ERR_UNSUPPORTED: valid request this build does not implement";
    case WST_ERR_CUDA: return "WST_ERR_CUDA: a CUDA call failed";
    case WST_ERR_TIMEOUT: return "WST_ERR_TIMEOUT: a device-side bounded wait ran out";
    case WST_ERR_BAD_OFFSETS: return "WST_ERR_BAD_OFFSETS: device offsets are inconsistent";
  }
  return "unknown wst_status";
}

wst_status wst_set_option(wst_option opt, int value) {
  g_err[0] = 0;
  int hi;
  switch ((int)opt) {
    case OPT_GROUPED_SCHEDULE: hi = 1; break;
    case OPT_DENSE_CTA_GROUP: hi = 2; break;
    case OPT_IKBO_SCHEDULE: hi = 1; break;
    case OPT_NORM_STATS: hi = 2; break;
    default: return fail(WST_ERR_INVALID_ARG, "unknown option %d", (int)opt);
  }
  if (value < 0 || value > hi)
    return fail(WST_ERR_INVALID_ARG, "option %d: value %d outside [0, %d]", (int)opt, value, hi);
  g_options[(int)opt].store(value, std::memory_order_relaxed);
  return WST_OK;
}

wst_status wst_get_option(wst_option opt, int* value) {
  g_err[0] = 0;
  if (!value) return fail(WST_ERR_INVALID_ARG, "value is NULL");
  if ((int)opt < 0 || (int)opt >= OPT_COUNT) return fail(WST_ERR_INVALID_ARG, "unknown option %d", (int)opt);
  *value = g_options[(int)opt].load(std::memory_order_relaxed);
  return WST_OK;
}

const char* wst_last_error(void) { return g_err; }

const char* wst_version(void) { return "wst 0.1.0 (sm_103a)"; }

}  // extern "C"
