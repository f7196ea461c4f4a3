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
//    before any stream capture.  No call allocates memory.
#include <mutex>
#include <stdio.h>

#include "attn_internal.h"

namespace attn {

namespace {

constexpr size_t kBwdScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_bwd_scratch[kBwdScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

attn_status noalloc_fail(attn_status s, const char* msg) {
  set_last_error(msg);
  return s;
}

}  // namespace

}  // namespace attn

using namespace attn;

extern "C" {

attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* dout, void* dq, void* dk, void* dv,
                             int B, int H, int N, int d, float scale, int causal,
                             cudaStream_t stream) {
  // Shape and size checks first: nothing is launched for a rejected call.
  const size_t need = attn_bwd_workspace_bytes(B, H, N, d, ATTN_DTYPE_BF16);
  if (need == 0)
    return noalloc_fail(ATTN_ERR_INVALID_ARG,
                        "attn_bwd_noalloc: invalid shape (see attn_bwd_workspace_bytes)");
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
    if (g_scratch_ptr[dev] == nullptr) {
      // Host code must not use g_bwd_scratch directly (that is a host-side
      // stand-in); ask the runtime for the device address on this device.
      void* p = nullptr;
      cudaError_t err = cudaGetSymbolAddress(&p, g_bwd_scratch);
      if (err != cudaSuccess || p == nullptr) {
        char msg[256];
        snprintf(msg, sizeof(msg), "attn_bwd_noalloc: cudaGetSymbolAddress failed: %s",
                 cudaGetErrorString(err));
        return noalloc_fail(ATTN_ERR_CUDA, msg);
      }
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  // The regular entry point validates every pointer and runs the three
  // backward kernels with the fixed array as its workspace.
  return attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal,
                  ATTN_DTYPE_BF16, scratch, kBwdScratchBytes, stream);
}

}  // extern "C"
