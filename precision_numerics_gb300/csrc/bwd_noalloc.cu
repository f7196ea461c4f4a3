// attn_bwd_noalloc: the BF16 backward with its scratch in a fixed, library-owned
// device array instead of a caller-provided workspace.
//
// Why it exists: some callers are not allowed to allocate device memory --
// for example a component running under a host framework that owns the
// whole device-memory budget and hands out only the tensors it manages, or a
// latency-critical loop where cudaMalloc/cudaFree (and the implicit
// synchronization they can bring) is not acceptable.  Such callers still
// pass their inputs and outputs; the backward's scratch (-LSE*log2(e), delta
// and the FP32 dQ accumulator) comes from g_bwd_scratch below.
//
// Costs and rules of use:
//  * g_bwd_scratch is kBwdScratchBytes (32 MiB) of device memory on every GPU
//    on which this file's module is loaded (at the latest by the first call
//    of attn_bwd_noalloc on that GPU); it stays allocated until the process
//    exits.
//  * Every call shares the one array.  Calls whose kernels can overlap on
//    the GPU (different streams, or different host threads without ordering)
//    race on it and produce wrong results; serialise them.
//  * The array keeps the previous call's contents.  Every call rewrites all
//    of the part it uses before reading it: the preprocess kernel writes
//    -LSE*log2(e) and delta for every padded row and zeroes the dQ
//    accumulator.
//  * The first call on a device looks up the array's device address with
//    cudaGetSymbolAddress while that device is current; make that first call
//    before any stream capture.  The address is cached together with the
//    unique id of the CUDA context it belongs to: after cudaDeviceReset (a new
//    primary context, in which the module and the array are loaded afresh) the
//    next call looks the address up again, so that first call after a reset
//    should also come before any stream capture.  No call allocates memory.
#include <mutex>
#include <stdio.h>

#include "attn_internal.h"

namespace attn {

namespace {

constexpr size_t kBwdScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_bwd_scratch[kBwdScratchBytes];

std::mutex g_setup_mutex;
// Per device: the array's device address and the id of the context it is valid in.
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

attn_status noalloc_fail(attn_status s, const char* msg) {
  set_last_error(msg);
  return s;
}

// Unique id of the calling thread's current CUDA context (driver entry
// points resolved once, no -lcuda); false when there is none or the driver
// lacks the calls.
bool current_context_id(unsigned long long* id) {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

}  // namespace

}  // namespace attn

using namespace attn;

extern "C" {

attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* dout, void* dq, void* dk, void* dv,
                             int B, int H, int N, int d, float scale, int causal,
                             cudaStream_t stream) {
  // Shape and size checks first: nothing is launched for a rejected call.  The
  // shape check is attn_bwd's own, so both entry points report the same status
  // (ATTN_ERR_UNSUPPORTED for a head size outside {64, 128}, for instance).
  Problem p;
  const attn_status shape = check_problem(B, H, N, d, ATTN_DTYPE_BF16, scale, true, &p);
  if (shape != ATTN_OK) return shape;
  const size_t need = bwd_workspace_bytes(p);
  if (need > kBwdScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "attn_bwd_noalloc: this problem needs %zu bytes of scratch, more than the fixed "
             "%zu-byte array; use attn_bwd with a caller workspace",
             need, kBwdScratchBytes);
    return noalloc_fail(ATTN_ERR_INVALID_ARG, msg);
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return noalloc_fail(ATTN_ERR_CUDA, "attn_bwd_noalloc: no usable current device");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    unsigned long long ctx = 0;
    const bool have_ctx = current_context_id(&ctx);
    if (g_scratch_ptr[dev] == nullptr || !have_ctx || g_scratch_ctx[dev] != ctx) {
      // Host code must not use g_bwd_scratch directly (that is a host-side
      // stand-in); ask the runtime for the device address in the current
      // context (this also sets the context up if no call has yet).
      void* addr = nullptr;
      cudaError_t err = cudaGetSymbolAddress(&addr, g_bwd_scratch);
      if (err != cudaSuccess || addr == nullptr) {
        char msg[256];
        snprintf(msg, sizeof(msg), "attn_bwd_noalloc: cudaGetSymbolAddress failed: %s",
                 cudaGetErrorString(err));
        return noalloc_fail(ATTN_ERR_CUDA, msg);
      }
      g_scratch_ptr[dev] = addr;
      g_scratch_ctx[dev] = current_context_id(&ctx) ? ctx : 0;
    }
    scratch = g_scratch_ptr[dev];
  }
  // The regular entry point validates every pointer and runs the three
  // backward kernels with the fixed array as its workspace.
  return attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal,
                  ATTN_DTYPE_BF16, scratch, kBwdScratchBytes, stream);
}

}  // extern "C"
