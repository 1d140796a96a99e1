// ikbo_ws.cu -- launcher of the IKBO linear-compression kernel.
#include <mutex>

#include "ikbo_ws.cuh"
#include "wst_host.h"

namespace wst {

int run_ikbo(const IkboProblem& pr, cudaStream_t stream) {
  DeviceInfo dev;
  int st = current_device_info(&dev);
  if (st) return st;

  const int F = pr.Du + pr.Dc;
  IkboArgs a{};
  a.num_users = pr.num_users;
  a.num_cand = pr.num_cand;
  a.Du = pr.Du;
  a.Dc = pr.Dc;
  a.D = pr.D;
  a.O = pr.O;
  a.kb_u = (pr.Du + 63) / 64;
  a.kb_c = (pr.Dc + 63) / 64;
  const size_t w_bytes = align_up((size_t)(a.kb_u + a.kb_c) * pr.O * 128, 1024);
  const size_t fixed = w_bytes + kIkboStgTotal /*output staging*/ +
                       1024 /*barriers, flags*/ + 1024 /*alignment slack*/;
  const size_t smem_cap = dev.max_smem_optin > 0 ? (size_t)dev.max_smem_optin : 232448;
  if (fixed + 4 * (size_t)kIkboABytes > smem_cap) {
    set_error("ikbo: W tile of %zu bytes leaves too little shared memory for the ring", w_bytes);
    return ST_UNSUPPORTED;
  }
  // Ring depth: 4 stages of 16 KB.  With one CTA per SM, 4 x 16 KB in
  // flight per SM already covers HBM's bandwidth-latency product (about
  // 6.8 MB at 6.8 TB/s and ~1 us, against 152 x 64 KB); a deeper ring only
  // lengthens every request's queue, including the user partials' stores,
  // their release fences and the candidates' flag polls, which gate each
  // CTA's first epilogue.  Measured on GB300 (64 users x 128 candidates,
  // one box, interleaved): 3 or 4 stages 0.0546 ms, 6 stages 0.0575 ms,
  // 12 stages (shared memory permitting) 0.0598 ms.
  constexpr int kIkboRingStages = 4;
  int stages = (int)((smem_cap - fixed) / kIkboABytes);
  if (stages > kIkboRingStages) stages = kIkboRingStages;
  a.stages = stages;
  a.slots = 512 / pr.O < kIkboMaxSlots ? 512 / pr.O : kIkboMaxSlots;
  a.uoff = pr.uoff;
  a.Y = static_cast<float*>(pr.Y);
  uint8_t* ws = static_cast<uint8_t*>(pr.ws);
  a.flags = reinterpret_cast<uint32_t*>(ws + ikbo_flags_offset());
  a.P = reinterpret_cast<float*>(ws + ikbo_partials_offset(pr.num_users));
  a.ws = reinterpret_cast<WsHeader*>(ws);
  a.timeout_ns = wait_timeout_ns();
  a.epoch = next_flag_epoch();

  CUtensorMap tmU, tmC, tmW, tmY;
  {
    uint64_t dims[3] = {(uint64_t)pr.D, (uint64_t)pr.Du, (uint64_t)pr.num_users};
    uint64_t str[2] = {(uint64_t)pr.D * 2, (uint64_t)pr.Du * pr.D * 2};
    uint32_t box[3] = {64, 64, 1};
    if ((st = encode_map(&tmU, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, pr.U, dims, str, box,
                         CU_TENSOR_MAP_SWIZZLE_128B)))
      return st;
  }
  {
    uint64_t dims[3] = {(uint64_t)pr.D, (uint64_t)pr.Dc, (uint64_t)pr.num_cand};
    uint64_t str[2] = {(uint64_t)pr.D * 2, (uint64_t)pr.Dc * pr.D * 2};
    uint32_t box[3] = {64, 64, 1};
    if ((st = encode_map(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, pr.Cf, dims, str, box,
                         CU_TENSOR_MAP_SWIZZLE_128B)))
      return st;
  }
  {
    uint64_t dims[2] = {(uint64_t)F, (uint64_t)pr.O};
    uint64_t str[1] = {(uint64_t)F * 2};
    uint32_t box[2] = {64, (uint32_t)pr.O};
    if ((st = encode_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pr.W, dims, str, box,
                         CU_TENSOR_MAP_SWIZZLE_128B)))
      return st;
  }

  {
    // Y viewed as [num_cand * O rows][D] fp32; box = one warp's 32 o x 32 d block.
    uint64_t dims[2] = {(uint64_t)pr.D, (uint64_t)pr.num_cand * pr.O};
    uint64_t str[1] = {(uint64_t)pr.D * 4};
    uint32_t box[2] = {32, 32};
    if ((st = encode_map(&tmY, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, pr.Y, dims, str, box,
                         CU_TENSOR_MAP_SWIZZLE_NONE)))
      return st;
  }

  const size_t smem = fixed + (size_t)stages * kIkboABytes;
  cudaError_t e;
  if (option_value(OPT_IKBO_SCHEDULE) == 1) {
    // Cluster launch control: one CTA per unit (each user item, then chunks
    // of kIkboClcChunk candidates); running CTAs take over unstarted ones.
    a.chunk = kIkboClcChunk;
    const long long units = (long long)pr.num_users + ((long long)pr.num_cand + kIkboClcChunk - 1) / kIkboClcChunk;
    if (units > 0x7fffffffLL) {
      set_error("ikbo: %lld units exceed the grid limit", units);
      return ST_UNSUPPORTED;
    }
    if ((st = ensure_smem_attr((const void*)k_ikbo_ws<true>, smem))) return st;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)units, 1, 1);
    cfg.blockDim = dim3(kIkboThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    e = cudaLaunchKernelEx(&cfg, k_ikbo_ws<true>, tmU, tmC, tmW, tmY, a);
    if (e != cudaSuccess) return cuda_fail(e, "launch k_ikbo_ws (cluster launch control)");
    return ST_OK;
  }
  if ((st = ensure_smem_attr((const void*)k_ikbo_ws<false>, smem))) return st;
  int grid = dev.num_sms < kIkboMaxGrid ? dev.num_sms : kIkboMaxGrid;
  const long long items = (long long)pr.num_users + pr.num_cand;
  if (items < grid) grid = (int)items;
  if (grid < 1) grid = 1;

  // Candidate split: CTA i first runs users i, i+grid, ...; then candidates
  // [split[i], split[i+1]).  Each item costs the bytes it moves (its feature
  // K-blocks plus its fp32 output tile); ranges are contiguous and balance
  // the cumulative cost (a running maximum keeps them non-decreasing).
  {
    const long long cu = (long long)a.kb_u * kIkboABytes + (long long)pr.O * pr.D * 4;
    const long long cc = (long long)a.kb_c * kIkboABytes + (long long)pr.O * pr.D * 4;
    const long long total = (long long)pr.num_users * cu + (long long)pr.num_cand * cc;
    int best = 0;
    a.split[0] = 0;
    for (int j = 1; j < grid; ++j) {
      const long long users_before =
          (long long)(pr.num_users / grid) * j + (j < pr.num_users % grid ? j : pr.num_users % grid);
      const long long budget = total * j / grid - users_before * cu;
      long long b = budget > 0 ? budget / cc : 0;
      if (b > pr.num_cand) b = pr.num_cand;
      if ((int)b > best) best = (int)b;
      a.split[j] = best;
    }
    a.split[grid] = pr.num_cand;
  }

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kIkboThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_ikbo_ws<false>, tmU, tmC, tmW, tmY, a);
  if (e != cudaSuccess) return cuda_fail(e, "launch k_ikbo_ws");
  return ST_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant (wst_ikbo_linear_compress_noalloc).
//
// Some callers cannot allocate device memory at call time: code that runs
// under a strict memory budget or a custom allocator it must not bypass, or a
// plugin whose host framework owns every allocation.  For them the same
// kernel runs with its scratch (header, ready flags, per-user partial
// products) in this file-scope device array instead of a caller workspace.
// Every GPU that loads the library holds the array until the process exits.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) uint8_t g_ikbo_scratch[kNoAllocScratchBytes];

size_t ikbo_noalloc_capacity() { return kNoAllocScratchBytes; }

// Device address of g_ikbo_scratch in the calling thread's current CUDA
// context.  The host-side symbol is only a stand-in, so the address is looked
// up with cudaGetSymbolAddress, with the device current, and cached per
// device together with the context's unique id (cuCtxGetId): after a
// cudaDeviceReset the runtime makes a new context with a new id, the module is
// loaded again, and the stale address is replaced instead of being reused.
// A lookup may load the module, which is not a stream operation: if it is
// needed while `stream` is being captured into a graph, the call is refused.
namespace {
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct ScratchCache {
  unsigned long long ctx_id;
  void* addr;
};

int current_context_id(unsigned long long* id) {
  static std::once_flag once;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(fn);
  });
  if (!get_current || !get_id) {
    set_error("cuCtxGetCurrent / cuCtxGetId are not available from the CUDA driver");
    return ST_CUDA;
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) {
    *id = 0;  // no context yet: the lookup below creates the primary context
    return ST_OK;
  }
  if (get_id(ctx, id) != CUDA_SUCCESS) {
    set_error("cuCtxGetId failed");
    return ST_CUDA;
  }
  return ST_OK;
}
}  // namespace

static int ikbo_noalloc_scratch(cudaStream_t stream, void** out) {
  static std::mutex mu;
  static ScratchCache cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) {
    set_error("device ordinal %d out of range", dev);
    return ST_UNSUPPORTED;
  }
  unsigned long long id = 0;
  int st = current_context_id(&id);
  if (st) return st;
  std::lock_guard<std::mutex> lk(mu);
  if (id != 0 && cache[dev].addr && cache[dev].ctx_id == id) {
    *out = cache[dev].addr;
    return ST_OK;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  if (cap != cudaStreamCaptureStatusNone) {
    set_error("ikbo (allocation-free): the first call in a CUDA context looks up the scratch "
              "array's device address and must not run while the stream is being captured; "
              "make one call before capturing");
    return ST_UNSUPPORTED;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_ikbo_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(ikbo scratch)");
  if (id == 0 && (st = current_context_id(&id))) return st;
  cache[dev] = ScratchCache{id, p};
  *out = p;
  return ST_OK;
}

int run_ikbo_noalloc(IkboProblem pr, int* d_status, cudaStream_t stream) {
  const size_t need = workspace_bytes(pr.num_users, pr.O, pr.D);
  if (need > kNoAllocScratchBytes) {
    set_error("ikbo (allocation-free): %d users x O=%d x D=%d need %zu bytes of scratch; "
              "this entry point holds %zu bytes (use wst_ikbo_linear_compress with a workspace)",
              pr.num_users, pr.O, pr.D, need, kNoAllocScratchBytes);
    return ST_INVALID_ARG;
  }
  void* scratch = nullptr;
  int st = ikbo_noalloc_scratch(stream, &scratch);
  if (st) return st;
  // The array keeps the previous call's contents: clear the header (error
  // word) and the ready flags so this call starts from zero (the flags'
  // per-call value alone would already tell old flags apart).
  cudaError_t e = cudaMemsetAsync(scratch, 0, ikbo_partials_offset(pr.num_users), stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(ikbo scratch)");
  pr.ws = scratch;
  st = run_ikbo(pr, stream);
  if (st) return st;
  if (d_status) {
    e = cudaMemcpyAsync(d_status, scratch, sizeof(int), cudaMemcpyDeviceToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(status)");
  }
  return ST_OK;
}

}  // namespace wst
