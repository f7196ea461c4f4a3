// Internal launch interface shared by the C-ABI layer and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "attn.h"

namespace attn {

// Problem description after validation.  Tensors are [B, H, N, d],
// contiguous, d fastest; LSE is [B, H, N].
struct Problem {
  int B, H, N, d;
  float scale;
  int causal;
};

// Tile geometry of the BF16 tensor-core path.
constexpr int kBlockM = 128;  // query rows per tile (one TMEM lane per row)
constexpr int kBlockN = 128;  // key rows per tile

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
inline int n_pad(int N) { return ceil_div(N, kBlockN) * kBlockN; }

// Launch with programmatic stream serialization: the kernel may be scheduled
// before the previous kernel in the stream has completed (its set-up then
// overlaps that kernel's tail), so it must call griddep_wait() before its
// first global-memory access, in every thread that makes one.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Backward workspace layout (all offsets 256-byte aligned):
//   neg_lse2 FP32 [B*H][Npad] -(LSE * log2(e)); -inf for padded rows
//   delta FP32 [B*H][Npad]    rowsum(dO o O); 0 for padded rows
//   dqacc FP32 [B*H][Npad][d] unscaled dQ accumulator
struct BwdWorkspace {
  float* neg_lse2;
  float* delta;
  float* dqacc;
};
size_t bwd_workspace_bytes(const Problem& p);
BwdWorkspace bwd_workspace_carve(void* base, const Problem& p);

// Kernel launchers.  Return cudaSuccess or the launch error.
// beta > 0 selects the stabilised normaliser (beta * repeated row max).
cudaError_t launch_fwd_bf16(const Problem& p, const void* q, const void* k, const void* v, void* o,
                            float* lse, cudaStream_t stream, float beta = 0.f);
cudaError_t launch_bwd_preprocess_bf16(const Problem& p, const void* o, const void* dout,
                                       const float* lse, const BwdWorkspace& ws,
                                       cudaStream_t stream);
cudaError_t launch_bwd_main_bf16(const Problem& p, const void* q, const void* k, const void* v,
                                 const void* dout, void* dk, void* dv, const BwdWorkspace& ws,
                                 cudaStream_t stream);
cudaError_t launch_bwd_dq_convert_bf16(const Problem& p, const BwdWorkspace& ws, void* dq,
                                       cudaStream_t stream);

cudaError_t launch_fwd_fp32(const Problem& p, const float* q, const float* k, const float* v,
                            float* o, float* lse, cudaStream_t stream);
cudaError_t launch_bwd_fp32(const Problem& p, const float* q, const float* k, const float* v,
                            const float* o, const float* lse, const float* dout, float* dq,
                            float* dk, float* dv, const BwdWorkspace& ws, cudaStream_t stream);

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream);

// INT8-input forward: per-token quantization of a BF16 [B,H,N,d] tensor, and
// the forward on INT8 Q, K (with their per-row scales) and BF16 V.
cudaError_t launch_quantize_int8(const Problem& p, const void* x, void* codes, float* scales,
                                 cudaStream_t stream);
cudaError_t launch_fwd_int8(const Problem& p, const void* q8, const float* qs, const void* k8,
                            const float* ks, const void* v, void* o, float* lse,
                            cudaStream_t stream);
// The same on INT8 codes held in BF16, with scales in the padded per-head
// layout [B*H][n_pad(N)], on the tcgen05 forward kernel.
cudaError_t launch_quantize_int8_as_bf16(const Problem& p, const void* x, void* codes,
                                         float* scales, cudaStream_t stream);
cudaError_t launch_fwd_int8_as_bf16(const Problem& p, const void* qc, const float* qs,
                                    const void* kc, const float* ks, const void* v, void* o,
                                    float* lse, cudaStream_t stream);

// Device status words (one per kernel translation unit): read and clear.
cudaError_t read_and_clear_status_fwd(unsigned int* out, cudaStream_t stream);
cudaError_t read_and_clear_status_bwd(unsigned int* out, cudaStream_t stream);
cudaError_t read_and_clear_status_misc(unsigned int* out, cudaStream_t stream);

// Shape and scalar checks shared by every entry point (d, N, B*H*N*d, dtype,
// and the scale when need_scale); fills *out and records the error detail.
attn_status check_problem(int B, int H, int N, int d, attn_dtype dt, float scale, bool need_scale,
                          Problem* out);

// Record the detail text returned by attn_last_error() on this thread.
void set_last_error(const char* msg);

// Number of SMs of the current device (cached per device); 0 if the query fails.
int device_sm_count();

// Driver entry point for cuTensorMapEncodeTiled (resolved once, no -lcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// 3-D BF16 tensor map over a [B*H, N, d] tensor with a (64 x box_rows x 1) box
// and 128-byte swizzle.  Returns false when the driver rejects it.
bool make_tmap_bhnd(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows = 128);

}  // namespace attn
