/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact tiled attention library.
 *
 * The library computes exact scaled-dot-product attention in the
 * FlashAttention style: blockwise Q K^T, an FP32 online softmax (running
 * row max and row sum, rescaling of the partial output) and blockwise P V,
 * forward and backward.  The operation is the "Baseline Attention" of
 * "Is Flash Attention Stable?" (abstract): O = softmax(scale * Q K^T) V, with
 * an optional causal mask; its tiled evaluation follows the block division
 * of "Why Low-Precision Transformer Training Fails", Algorithm 1 (Q split
 * into row blocks, K and V into column blocks).  The backward pass uses
 * delta = rowsum(dO o O) as defined in that paper (Figures 3 and 5).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors Q, K, V, O, dO, dQ, dK, dV are [B, H, N, d], contiguous,
 *    d fastest, in DEVICE memory (device or managed allocations), 16-byte
 *    aligned.  LSE is FP32 [B, H, N] (natural log): LSE_i = ln sum_j
 *    exp(scale * q_i . k_j) over the visible keys.
 *  - causal != 0 hides key j from query i when j > i (square, top-left).
 *  - dt selects the element type of Q, K, V, O, dO, dQ, dK, dV:
 *      ATTN_DTYPE_BF16 -- tensor-core path (TMA + tcgen05/TMEM), FP32
 *                         softmax and accumulation, BF16 results;
 *      ATTN_DTYPE_FP32 -- reference mode: the same tiled online softmax in
 *                         FP32 CUDA-core arithmetic (no tensor cores).
 *  - Supported: d in {64, 128}; N >= 1; B*H*N*d < 2^31; scale finite > 0.
 *  - Ownership: the caller allocates every buffer and owns the stream; the
 *    library makes no allocation calls and keeps no per-call state (its one
 *    fixed device array is described at attn_bwd_noalloc).
 *  - Asynchrony: kernels are enqueued on `stream` and the call returns
 *    without synchronizing.  Argument errors are reported synchronously,
 *    before anything is enqueued; launch failures map to ATTN_ERR_CUDA.
 *  - Every wait inside a kernel is bounded (about 2 s).  A wait that gives
 *    up records ATTN_ERR_TIMEOUT on the device and the kernel returns;
 *    attn_check_status() reports it.
 *  - The device is the one current on the calling thread; all pointers
 *    must belong to it.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* bad pointer, shape, scale or workspace size */
  ATTN_ERR_UNSUPPORTED = 2, /* valid request outside the supported set     */
  ATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed           */
  ATTN_ERR_TIMEOUT = 4      /* a bounded in-kernel wait gave up            */
} attn_status;

typedef enum { ATTN_DTYPE_BF16 = 0, ATTN_DTYPE_FP32 = 1 } attn_dtype;

/* Library version, major * 10000 + minor * 100 + patch. */
ATTN_API int attn_version(void);

/* Static description of a status code. */
ATTN_API const char* attn_status_string(attn_status s);

/* Human-readable detail of the last error returned on the calling thread
 * (empty string when none).  The pointer stays valid until the next call on
 * the same thread. */
ATTN_API const char* attn_last_error(void);

/*
 * Forward pass ("Is Flash Attention Stable?", abstract: Baseline Attention;
 * tiled as in "Why Low-Precision Transformer Training Fails", Algorithm 1).
 *   q, k, v : [B,H,N,d] inputs (dt).
 *   o       : [B,H,N,d] output (dt), O = softmax(scale Q K^T [+mask]) V.
 *   lse     : [B,H,N] FP32 output, natural-log log-sum-exp of each row of
 *             scale Q K^T over the visible keys.
 * Returns ATTN_OK once the kernel is enqueued.
 */
ATTN_API attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int N, int d, float scale, int causal, attn_dtype dt,
                              cudaStream_t stream);

/*
 * Forward pass with the stabilised normaliser of "Why Low-Precision Transformer
 * Training Fails" (Figure 7 and Algorithm 1): while a row's running maximum
 * r_m of scale * q.k is attained by two or more keys, the exponentials are
 * taken relative to m = beta * r_m if r_m > 0 and m = 0 if r_m <= 0, so that
 * no unnormalised probability exp(S - m) is exactly 1.  Mathematically O and
 * LSE are those of attn_fwd (LSE is formed with the normaliser actually
 * used); only the rounding differs.  attn_bwd accepts its outputs unchanged.
 * BF16 only; beta must be finite and > 1.  With c = scale * log2(e), m is
 * then kept within [r_m + 2^-8 / c, r_m + 64 / c]:
 *   - the floor makes the row's largest exponent "sufficiently negative" (the
 *     paper's words) once rounded: 2^(c (r_m - m)) <= 2^(-2^-8) rounds to at
 *     most 1 - 2^-8 in BF16, also for repeated maxima that are 0, tiny, or
 *     tiny and negative, where beta * r_m or 0 alone would leave the BF16
 *     operand of the P V product at exactly 1;
 *   - the cap keeps the largest exponential at or above 2^-64, so a very
 *     large repeated maximum cannot underflow the whole row.
 */
ATTN_API attn_status attn_fwd_stable(const void* q, const void* k, const void* v, void* o,
                                     float* lse, int B, int H, int N, int d, float scale,
                                     int causal, float beta, attn_dtype dt, cudaStream_t stream);

/*
 * Per-token symmetric INT8 quantization ("INT-FlashAttention: Enabling Flash
 * Attention for INT8 Quantization", abstract; the page fixes no scheme, the
 * one here is a reading): for every row r of every head of the BF16 tensor
 * x [B,H,N,d], scales[r] = max_j |x_rj| / 127 (FP32) and codes[r][j] =
 * rint(x_rj / scales[r]) clamped to [-127, 127], rint rounding half to even;
 * a row of zeros gets scale 0 and codes 0.
 *   x      : [B,H,N,d] BF16, device.
 *   codes  : [B,H,N,d] int8, device, written.
 *   scales : [B,H,N] FP32, device, written.
 * d in {64, 128}; all pointers 16-byte aligned.
 */
ATTN_API attn_status attn_quantize_int8(const void* x, void* codes, float* scales, int B, int H,
                                        int N, int d, cudaStream_t stream);

/*
 * Forward on per-token INT8 Q and K (as written by attn_quantize_int8) and
 * BF16 V: S_ij = scale * q_scale[i] * k_scale[j] * (q8_i . k8_j) with the
 * integer dot product exact, then the FP32 online softmax and P V (P rounded
 * to BF16), O = softmax(S [+mask]) V and LSE = ln sum_j exp(S_ij) as in
 * attn_fwd.  sm_103a has no INT8 tcgen05 MMA, so this path runs on the
 * warp-level mma.sync tensor-core instructions and is several times slower
 * than attn_fwd; attn_fwd_int8_as_bf16 computes the same scores on the
 * tcgen05 path from codes held in BF16.
 *   q8, k8  : [B,H,N,d] int8, device.   q_scale, k_scale : [B,H,N] FP32.
 *   v       : [B,H,N,d] BF16.           o : [B,H,N,d] BF16.   lse : [B,H,N] FP32.
 * d in {64, 128}; all pointers 16-byte aligned, device memory.
 */
ATTN_API attn_status attn_fwd_int8(const void* q8, const float* q_scale, const void* k8,
                                   const float* k_scale, const void* v, void* o, float* lse,
                                   int B, int H, int N, int d, float scale, int causal,
                                   cudaStream_t stream);

/*
 * The quantization of attn_quantize_int8 with the codes held in BF16: every
 * code is an integer in [-127, 127], which BF16 represents exactly, so these
 * are the same codes in a 2-byte type.  The scales are laid out per head with
 * the row count padded: scales[(b*H + h) * N_pad + n], N_pad = N rounded up
 * to a multiple of 128; the padded entries are written as 0.
 *   x      : [B,H,N,d] BF16, device.
 *   codes  : [B,H,N,d] BF16, device, written.
 *   scales : B*H*N_pad FP32, device, written.
 * d in {64, 128}; all pointers 16-byte aligned.
 */
ATTN_API attn_status attn_quantize_int8_as_bf16(const void* x, void* codes, float* scales, int B,
                                                int H, int N, int d, cudaStream_t stream);

/*
 * attn_fwd_int8 on codes held in BF16 (attn_quantize_int8_as_bf16): the same
 * scores S_ij = scale * q_scale[i] * k_scale[j] * (q8_i . k8_j), the integer
 * dot product exact, evaluated on the BF16 tcgen05 path of attn_fwd -- every
 * product of two codes (|c| <= 127) and every partial sum over d <= 128
 * terms (< 2^24) is exact in the FP32 accumulator, whatever the order.  The
 * row scale is clamped below at 1e-20 (a row of zero codes has zero scores
 * either way).  Compared with attn_fwd_int8, Q and K take two bytes per code
 * and the path runs at the speed of the BF16 forward.
 *   q_codes, k_codes : [B,H,N,d] BF16 holding integer codes, device.
 *   q_scale, k_scale : B*H*N_pad FP32 (layout of attn_quantize_int8_as_bf16).
 *   v : [B,H,N,d] BF16.   o : [B,H,N,d] BF16.   lse : [B,H,N] FP32.
 * d in {64, 128}; all pointers 16-byte aligned, device memory.
 */
ATTN_API attn_status attn_fwd_int8_as_bf16(const void* q_codes, const float* q_scale,
                                           const void* k_codes, const float* k_scale,
                                           const void* v, void* o, float* lse, int B, int H,
                                           int N, int d, float scale, int causal,
                                           cudaStream_t stream);

/*
 * Bytes of device workspace attn_bwd needs for this problem (0 on invalid
 * arguments).  Layout (internal): -LSE*log2(e) and delta, FP32 [B*H][Npad]
 * each, and the FP32 dQ accumulator [B*H][Npad][d], Npad = N rounded up to
 * 128.  The workspace needs no initialisation; attn_bwd overwrites it.
 */
ATTN_API size_t attn_bwd_workspace_bytes(int B, int H, int N, int d, attn_dtype dt);

/*
 * Backward pass from the saved LSE: dQ, dK, dV of L = sum(dO o O).
 * The gradient of the attention definition, with delta = rowsum(dO o O)
 * ("Why Low-Precision Transformer Training Fails", Figures 3 and 5),
 * dS = P o (dO V^T - delta), dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO.
 *   q, k, v, o, dout : [B,H,N,d] inputs (dt); o is the forward output.
 *   lse              : [B,H,N] FP32, the forward's LSE.
 *   dq, dk, dv       : [B,H,N,d] outputs (dt).
 *   workspace        : device buffer of at least
 *                      attn_bwd_workspace_bytes(...) bytes, 256-byte aligned,
 *                      not shared with a concurrently running call.
 * Enqueues three kernels on `stream`: preprocess (delta, -LSE*log2(e), zero
 * the dQ accumulator), the main kernel (dK, dV, dQ accumulation), and the
 * dQ conversion (scale and round).  The three phases are also exported
 * below so that each can be timed on its own.
 */
ATTN_API attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, float scale, int causal, attn_dtype dt,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Phase 1 of attn_bwd (BF16 only): delta_i = rowsum(dO o O)_i in FP32 from
 * the stored O, -LSE*log2(e), and a zeroed dQ accumulator, into `workspace`. */
ATTN_API attn_status attn_bwd_preprocess(const void* o, const float* lse, const void* dout, int B,
                                         int H, int N, int d, attn_dtype dt, void* workspace,
                                         size_t workspace_bytes, cudaStream_t stream);

/* Phase 2 of attn_bwd (BF16 only): dK and dV (written to dk, dv) and the FP32
 * dQ accumulation into `workspace`; needs phase 1 to have run on it. */
ATTN_API attn_status attn_bwd_main(const void* q, const void* k, const void* v, const void* dout,
                                   void* dk, void* dv, int B, int H, int N, int d, float scale,
                                   int causal, attn_dtype dt, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream);

/* Phase 3 of attn_bwd (BF16 only): dQ = bf16(scale * accumulator). */
ATTN_API attn_status attn_bwd_dq_convert(void* dq, int B, int H, int N, int d, float scale,
                                         attn_dtype dt, void* workspace, size_t workspace_bytes,
                                         cudaStream_t stream);

/*
 * Synchronizes `stream`, then reads and clears the device-side status words
 * of the library on the current device.  Returns ATTN_ERR_TIMEOUT if any
 * kernel gave up on a bounded wait since the last check, ATTN_ERR_CUDA if
 * the stream reports an error, else ATTN_OK.
 *
 * The status words are per device and per process, not per stream or per
 * call: a timeout recorded by any of this library's kernels on the current
 * device, launched from any stream or host thread, is reported by the next
 * attn_check_status on that device, whatever stream it is given, and that
 * check clears it.  `stream` only selects what is synchronized first; a
 * caller that needs to attribute a timeout to one call must check after that
 * call with no other call of the library in flight on the device.
 */
ATTN_API attn_status attn_check_status(cudaStream_t stream);

/*
 * Self-test of the bounded-wait path: enqueues a one-block kernel that waits
 * on a shared-memory barrier nothing ever arrives at, for at most limit_ns
 * nanoseconds (1 <= limit_ns <= 10^9), then records ATTN_ERR_TIMEOUT and
 * returns.  attn_check_status() afterwards must report ATTN_ERR_TIMEOUT.
 */
ATTN_API attn_status attn_selftest_wait_timeout(unsigned long long limit_ns, cudaStream_t stream);

/*
 * attn_bwd without a caller workspace, for callers that must not allocate
 * device memory (no counterpart in the pages: this is a library-usage entry
 * point, not part of the method).  Typical such callers run inside a host
 * framework that owns the whole device-memory budget, or in latency-critical
 * loops where cudaMalloc/cudaFree and their implicit synchronization are not
 * acceptable.  Same arguments and results as attn_bwd with dt = BF16; the
 * scratch (-LSE*log2(e), delta, FP32 dQ accumulator) lives in a fixed 32 MiB
 * device array inside the library instead of `workspace`.
 *   - Limit: attn_bwd_workspace_bytes(B, H, N, d, BF16) must be at most
 *     33554432 bytes (e.g. B8 H12 N1024 d64 fits); larger problems return
 *     ATTN_ERR_INVALID_ARG before anything is launched.
 *   - The array occupies 32 MiB on each GPU where the library's module is
 *     loaded (at the latest from this entry point's first call there) until
 *     the process exits.  No call allocates memory.
 *   - All calls share the array: calls that can overlap on the GPU (other
 *     streams, unordered host threads) race and give wrong results.  Each call
 *     rewrites what it reads (the dQ accumulator is zeroed every call).
 *   - The first call on a device looks up the array's device address; make
 *     that first call before any stream capture.  The address is kept with
 *     the id of the CUDA context it belongs to; after cudaDeviceReset the next
 *     call looks it up again, so that call too belongs before any capture.
 *   - Shape errors are those of attn_bwd (ATTN_ERR_UNSUPPORTED for a head size
 *     outside {64, 128}, ATTN_ERR_INVALID_ARG for a bad N, B*H or scale).
 */
ATTN_API attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                      const float* lse, const void* dout, void* dq, void* dk,
                                      void* dv, int B, int H, int N, int d, float scale,
                                      int causal, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
