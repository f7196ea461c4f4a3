// C-ABI entry points: argument validation, tensor-map encoding, dispatch to
// the BF16 tensor-core kernels or the FP32 reference-mode kernels, and the
// device status words behind attn_check_status().
#include <math.h>
#include <atomic>
#include <mutex>
#include <stdarg.h>
#include <stdio.h>
#include <string>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {

static __device__ unsigned int g_status_misc;

namespace {

thread_local std::string t_last_error;

attn_status fail(attn_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return s;
}

attn_status cuda_fail(cudaError_t err, const char* what) {
  return fail(ATTN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

// Shape and scalar checks shared by every entry point.
attn_status check_problem(int B, int H, int N, int d, attn_dtype dt, float scale, bool need_scale,
                          Problem* out) {
  if (dt != ATTN_DTYPE_BF16 && dt != ATTN_DTYPE_FP32)
    return fail(ATTN_ERR_INVALID_ARG, "dt must be ATTN_DTYPE_BF16 or ATTN_DTYPE_FP32 (got %d)",
                (int)dt);
  if (B < 1 || H < 1 || N < 1)
    return fail(ATTN_ERR_INVALID_ARG, "B, H, N must be >= 1 (got B=%d H=%d N=%d)", B, H, N);
  if (d != 64 && d != 128)
    return fail(ATTN_ERR_UNSUPPORTED, "head dim d=%d is not supported (64 or 128)", d);
  const long long elems = (long long)B * H * N * d;
  if (elems >= (1ll << 31))
    return fail(ATTN_ERR_INVALID_ARG, "B*H*N*d = %lld exceeds 2^31 - 1", elems);
  if (dt == ATTN_DTYPE_FP32 && (long long)B * H > 65535)
    return fail(ATTN_ERR_UNSUPPORTED, "FP32 reference mode supports B*H <= 65535");
  if (need_scale && !(isfinite(scale) && scale > 0.f))
    return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0 (got %g)", (double)scale);
  out->B = B;
  out->H = H;
  out->N = N;
  out->d = d;
  out->scale = scale;
  out->causal = 0;
  return ATTN_OK;
}

namespace {

// Pointer must be non-null, 16-byte aligned and reachable from the current
// device (device memory of this device, or managed memory).
attn_status check_ptr(const void* p, const char* name) {
  if (p == nullptr) return fail(ATTN_ERR_INVALID_ARG, "%s is NULL", name);
  if (reinterpret_cast<uintptr_t>(p) & 15u)
    return fail(ATTN_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  cudaPointerAttributes attr;
  cudaError_t err = cudaPointerGetAttributes(&attr, p);
  if (err != cudaSuccess) {
    cudaGetLastError();
    return fail(ATTN_ERR_INVALID_ARG, "%s: cannot query pointer (%s)", name,
                cudaGetErrorName(err));
  }
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return fail(ATTN_ERR_INVALID_ARG, "%s is not device memory", name);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaGetDevice failed");
  if (attr.type == cudaMemoryTypeDevice && attr.device != dev)
    return fail(ATTN_ERR_INVALID_ARG, "%s lives on device %d, current device is %d", name,
                attr.device, dev);
  return ATTN_OK;
}

#define ATTN_CHECK(expr)          \
  do {                            \
    attn_status _s = (expr);      \
    if (_s != ATTN_OK) return _s; \
  } while (0)

// One-block kernel that waits on a barrier nobody arrives at, with a limit.
__global__ void wait_selftest_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait_ns(&bar, 0, limit_ns))
    atomicOr(&g_status_misc, (unsigned int)ATTN_ERR_TIMEOUT);
  __syncthreads();
}

}  // namespace

void set_last_error(const char* msg) { t_last_error = msg; }

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int device_sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < kMaxDevices) {
    const int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 0;
  if (dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

bool make_tmap_bhnd(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

size_t bwd_workspace_bytes(const Problem& p) {
  const size_t rows = (size_t)p.B * p.H * n_pad(p.N);
  return align256(rows * 4) * 2 + align256(rows * p.d * 4);
}

BwdWorkspace bwd_workspace_carve(void* base, const Problem& p) {
  const size_t rows = (size_t)p.B * p.H * n_pad(p.N);
  char* b = static_cast<char*>(base);
  BwdWorkspace ws;
  ws.neg_lse2 = reinterpret_cast<float*>(b);
  ws.delta = reinterpret_cast<float*>(b + align256(rows * 4));
  ws.dqacc = reinterpret_cast<float*>(b + 2 * align256(rows * 4));
  return ws;
}

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t read_and_clear_status_misc(unsigned int* out, cudaStream_t stream) {
  static const unsigned int zero = 0;
  cudaError_t err = cudaMemcpyFromSymbolAsync(out, g_status_misc, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
  if (err != cudaSuccess) return err;
  err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return err;
  err = cudaMemcpyToSymbolAsync(g_status_misc, &zero, sizeof(unsigned int), 0,
                                cudaMemcpyHostToDevice, stream);
  if (err != cudaSuccess) return err;
  return cudaStreamSynchronize(stream);
}

namespace {

attn_status check_workspace(const Problem& p, void* workspace, size_t bytes) {
  if (workspace == nullptr) return fail(ATTN_ERR_INVALID_ARG, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(ATTN_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  const size_t need = bwd_workspace_bytes(p);
  if (bytes < need)
    return fail(ATTN_ERR_INVALID_ARG, "workspace has %zu bytes, %zu needed", bytes, need);
  return check_ptr(workspace, "workspace");
}

attn_status launched(cudaError_t err, const char* what) {
  if (err != cudaSuccess) return cuda_fail(err, what);
  t_last_error.clear();
  return ATTN_OK;
}

}  // namespace

}  // namespace attn

using namespace attn;

extern "C" {

int attn_version(void) { return 100; }

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG: invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED: request outside the supported set";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA: a CUDA call failed";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT: a bounded in-kernel wait gave up";
  }
  return "unknown attn_status";
}

const char* attn_last_error(void) { return t_last_error.c_str(); }

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int N, int d, float scale, int causal, attn_dtype dt,
                     cudaStream_t stream) {
  Problem p;
  ATTN_CHECK(check_problem(B, H, N, d, dt, scale, true, &p));
  p.causal = causal != 0;
  ATTN_CHECK(check_ptr(q, "q"));
  ATTN_CHECK(check_ptr(k, "k"));
  ATTN_CHECK(check_ptr(v, "v"));
  ATTN_CHECK(check_ptr(o, "o"));
  ATTN_CHECK(check_ptr(lse, "lse"));
  if (dt == ATTN_DTYPE_FP32)
    return launched(launch_fwd_fp32(p, static_cast<const float*>(q), static_cast<const float*>(k),
                                    static_cast<const float*>(v), static_cast<float*>(o), lse,
                                    stream),
                    "attn_fwd (fp32)");
  if (encode_tiled_fn() == nullptr)
    return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
  return launched(launch_fwd_bf16(p, q, k, v, o, lse, stream), "attn_fwd (bf16)");
}

attn_status attn_fwd_stable(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int H, int N, int d, float scale, int causal, float beta,
                            attn_dtype dt, cudaStream_t stream) {
  Problem p;
  ATTN_CHECK(check_problem(B, H, N, d, dt, scale, true, &p));
  p.causal = causal != 0;
  if (dt != ATTN_DTYPE_BF16)
    return fail(ATTN_ERR_UNSUPPORTED, "attn_fwd_stable is implemented for BF16 only");
  if (!(isfinite(beta) && beta > 1.f))
    return fail(ATTN_ERR_INVALID_ARG, "beta must be finite and > 1 (got %g)", (double)beta);
  ATTN_CHECK(check_ptr(q, "q"));
  ATTN_CHECK(check_ptr(k, "k"));
  ATTN_CHECK(check_ptr(v, "v"));
  ATTN_CHECK(check_ptr(o, "o"));
  ATTN_CHECK(check_ptr(lse, "lse"));
  if (encode_tiled_fn() == nullptr)
    return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
  return launched(launch_fwd_bf16(p, q, k, v, o, lse, stream, beta), "attn_fwd_stable");
}

attn_status attn_quantize_int8(const void* x, void* codes, float* scales, int B, int H, int N,
                               int d, cudaStream_t stream) {
  Problem p;
  ATTN_CHECK(check_problem(B, H, N, d, ATTN_DTYPE_BF16, 1.f, false, &p));
  ATTN_CHECK(check_ptr(x, "x"));
  ATTN_CHECK(check_ptr(codes, "codes"));
  ATTN_CHECK(check_ptr(scales, "scales"));
  return launched(launch_quantize_int8(p, x, codes, scales, stream), "attn_quantize_int8");
}

attn_status attn_fwd_int8(const void* q8, const float* q_scale, const void* k8,
                          const float* k_scale, const void* v, void* o, float* lse, int B, int H,
                          int N, int d, float scale, int causal, cudaStream_t stream) {
  Problem p;
  ATTN_CHECK(check_problem(B, H, N, d, ATTN_DTYPE_BF16, scale, true, &p));
  p.causal = causal != 0;
  const void* ptrs[7] = {q8, q_scale, k8, k_scale, v, o, lse};
  const char* names[7] = {"q8", "q_scale", "k8", "k_scale", "v", "o", "lse"};
  for (int i = 0; i < 7; ++i) ATTN_CHECK(check_ptr(ptrs[i], names[i]));
  return launched(launch_fwd_int8(p, q8, q_scale, k8, k_scale, v, o, lse, stream),
                  "attn_fwd_int8");
}

attn_status attn_quantize_int8_as_bf16(const void* x, void* codes, float* scales, int B, int H,
                                       int N, int d, cudaStream_t stream) {
  Problem p;
  ATTN_CHECK(check_problem(B, H, N, d, ATTN_DTYPE_BF16, 1.f, false, &p));
  ATTN_CHECK(check_ptr(x, "x"));
  ATTN_CHECK(check_ptr(codes, "codes"));
  ATTN_CHECK(check_ptr(scales, "scales"));
  return launched(launch_quantize_int8_as_bf16(p, x, codes, scales, stream),
                  "attn_quantize_int8_as_bf16");
}

attn_status attn_fwd_int8_as_bf16(const void* q_codes, const float* q_scale, const void* k_codes,
                                  const float* k_scale, const void* v, void* o, float* lse, int B,
                                  int H, int N, int d, float scale, int causal,
                                  cudaStream_t stream) {
  Problem p;
  ATTN_CHECK(check_problem(B, H, N, d, ATTN_DTYPE_BF16, scale, true, &p));
  p.causal = causal != 0;
  const void* ptrs[7] = {q_codes, q_scale, k_codes, k_scale, v, o, lse};
  const char* names[7] = {"q_codes", "q_scale", "k_codes", "k_scale", "v", "o", "lse"};
  for (int i = 0; i < 7; ++i) ATTN_CHECK(check_ptr(ptrs[i], names[i]));
  if (encode_tiled_fn() == nullptr)
    return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
  return launched(launch_fwd_int8_as_bf16(p, q_codes, q_scale, k_codes, k_scale, v, o, lse, stream),
                  "attn_fwd_int8_as_bf16");
}

size_t attn_bwd_workspace_bytes(int B, int H, int N, int d, attn_dtype dt) {
  Problem p;
  if (check_problem(B, H, N, d, dt, 1.f, false, &p) != ATTN_OK) return 0;
  return bwd_workspace_bytes(p);
}

attn_status attn_bwd_preprocess(const void* o, const float* lse, const void* dout, int B, int H,
                                int N, int d, attn_dtype dt, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  Problem p;
  ATTN_CHECK(check_problem(B, H, N, d, dt, 1.f, false, &p));
  if (dt != ATTN_DTYPE_BF16)
    return fail(ATTN_ERR_UNSUPPORTED, "the backward phases are exported for BF16 only");
  ATTN_CHECK(check_ptr(o, "o"));
  ATTN_CHECK(check_ptr(lse, "lse"));
  ATTN_CHECK(check_ptr(dout, "dout"));
  ATTN_CHECK(check_workspace(p, workspace, workspace_bytes));
  return launched(
      launch_bwd_preprocess_bf16(p, o, dout, lse, bwd_workspace_carve(workspace, p), stream),
      "attn_bwd_preprocess");
}

attn_status attn_bwd_main(const void* q, const void* k, const void* v, const void* dout,
                          void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                          attn_dtype dt, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
  Problem p;
  ATTN_CHECK(check_problem(B, H, N, d, dt, scale, true, &p));
  p.causal = causal != 0;
  if (dt != ATTN_DTYPE_BF16)
    return fail(ATTN_ERR_UNSUPPORTED, "the backward phases are exported for BF16 only");
  ATTN_CHECK(check_ptr(q, "q"));
  ATTN_CHECK(check_ptr(k, "k"));
  ATTN_CHECK(check_ptr(v, "v"));
  ATTN_CHECK(check_ptr(dout, "dout"));
  ATTN_CHECK(check_ptr(dk, "dk"));
  ATTN_CHECK(check_ptr(dv, "dv"));
  ATTN_CHECK(check_workspace(p, workspace, workspace_bytes));
  if (encode_tiled_fn() == nullptr)
    return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
  return launched(
      launch_bwd_main_bf16(p, q, k, v, dout, dk, dv, bwd_workspace_carve(workspace, p), stream),
      "attn_bwd_main");
}

attn_status attn_bwd_dq_convert(void* dq, int B, int H, int N, int d, float scale, attn_dtype dt,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Problem p;
  ATTN_CHECK(check_problem(B, H, N, d, dt, scale, true, &p));
  if (dt != ATTN_DTYPE_BF16)
    return fail(ATTN_ERR_UNSUPPORTED, "the backward phases are exported for BF16 only");
  ATTN_CHECK(check_ptr(dq, "dq"));
  ATTN_CHECK(check_workspace(p, workspace, workspace_bytes));
  return launched(launch_bwd_dq_convert_bf16(p, bwd_workspace_carve(workspace, p), dq, stream),
                  "attn_bwd_dq_convert");
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                     int H, int N, int d, float scale, int causal, attn_dtype dt,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Problem p;
  ATTN_CHECK(check_problem(B, H, N, d, dt, scale, true, &p));
  p.causal = causal != 0;
  const void* ins[6] = {q, k, v, o, lse, dout};
  const char* in_names[6] = {"q", "k", "v", "o", "lse", "dout"};
  for (int i = 0; i < 6; ++i) ATTN_CHECK(check_ptr(ins[i], in_names[i]));
  ATTN_CHECK(check_ptr(dq, "dq"));
  ATTN_CHECK(check_ptr(dk, "dk"));
  ATTN_CHECK(check_ptr(dv, "dv"));
  ATTN_CHECK(check_workspace(p, workspace, workspace_bytes));
  const BwdWorkspace ws = bwd_workspace_carve(workspace, p);
  if (dt == ATTN_DTYPE_FP32)
    return launched(
        launch_bwd_fp32(p, static_cast<const float*>(q), static_cast<const float*>(k),
                        static_cast<const float*>(v), static_cast<const float*>(o), lse,
                        static_cast<const float*>(dout), static_cast<float*>(dq),
                        static_cast<float*>(dk), static_cast<float*>(dv), ws, stream),
        "attn_bwd (fp32)");
  if (encode_tiled_fn() == nullptr)
    return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
  cudaError_t err = launch_bwd_preprocess_bf16(p, o, dout, lse, ws, stream);
  if (err != cudaSuccess) return cuda_fail(err, "attn_bwd preprocess");
  err = launch_bwd_main_bf16(p, q, k, v, dout, dk, dv, ws, stream);
  if (err != cudaSuccess) return cuda_fail(err, "attn_bwd main");
  return launched(launch_bwd_dq_convert_bf16(p, ws, dq, stream), "attn_bwd dq_convert");
}

attn_status attn_check_status(cudaStream_t stream) {
  cudaError_t err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return cuda_fail(err, "attn_check_status: stream");
  unsigned int a = 0, b = 0, c = 0;
  if ((err = read_and_clear_status_fwd(&a, stream)) != cudaSuccess ||
      (err = read_and_clear_status_bwd(&b, stream)) != cudaSuccess ||
      (err = read_and_clear_status_misc(&c, stream)) != cudaSuccess)
    return cuda_fail(err, "attn_check_status: status read");
  const unsigned int any = a | b | c;
  if (any & ATTN_ERR_TIMEOUT)
    return fail(ATTN_ERR_TIMEOUT, "a kernel gave up on a bounded wait (status %u/%u/%u)", a, b, c);
  if (any != 0)
    return fail(ATTN_ERR_INVALID_ARG, "a kernel reported a bad launch setup (status %u/%u/%u)", a,
                b, c);
  t_last_error.clear();
  return ATTN_OK;
}

attn_status attn_selftest_wait_timeout(unsigned long long limit_ns, cudaStream_t stream) {
  if (limit_ns < 1 || limit_ns > 1000000000ull)
    return fail(ATTN_ERR_INVALID_ARG, "limit_ns must be in [1, 1e9] (got %llu)", limit_ns);
  return launched(launch_wait_selftest(limit_ns, stream), "attn_selftest_wait_timeout");
}

}  // extern "C"
