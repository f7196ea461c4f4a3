// FP32 reference mode: the same tiled online-softmax forward in plain FP32
// CUDA-core arithmetic (no tensor cores, no BF16 rounding of P), and the
// backward from the saved LSE.  Small shapes only; it pins the tiled
// algorithm (running max, running sum, rescaled partial output -- "Why
// Low-Precision Transformer Training Fails", Algorithm 1 and Figure 7) to
// the FP64 definition at FP32 accuracy.
//
// Forward: one warp per query row; K/V are visited in blocks of 32 keys,
// lane j scoring key j of the block.  Backward: delta = rowsum(dO o O)
// (that paper's Figures 3 and 5), then one warp per query row for dQ and one
// warp per key row for dK and dV, each recomputing P from the LSE.
#include <math.h>

#include "attn_internal.h"

namespace attn {

namespace {

constexpr int kRowsPerBlock = 4;  // warps per block, one row each
constexpr int kKeyBlock = 32;     // keys per online-softmax step

template <int D>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
    fwd_fp32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                    const float* __restrict__ v, float* __restrict__ o, float* __restrict__ lse,
                    int N, float scale, int causal) {
  constexpr int kPer = D / 32;  // output columns per lane: lane + 32 * c
  __shared__ float s_q[kRowsPerBlock][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + warp;
  const size_t head = (size_t)blockIdx.y * N * D;
  if (row >= N) return;
  for (int c = lane; c < D; c += 32) s_q[warp][c] = q[head + (size_t)row * D + c];
  __syncwarp();

  float m = -INFINITY, l = 0.f, acc[kPer];
#pragma unroll
  for (int c = 0; c < kPer; ++c) acc[c] = 0.f;
  const int n_keys = causal ? row + 1 : N;
  for (int kv0 = 0; kv0 < n_keys; kv0 += kKeyBlock) {
    const int key = kv0 + lane;
    float s = -INFINITY;
    if (key < n_keys) {
      const float* kr = k + head + (size_t)key * D;
      float dot = 0.f;
      for (int t = 0; t < D; ++t) dot = fmaf(s_q[warp][t], kr[t], dot);
      s = dot * scale;
    }
    float mx = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float m_new = fmaxf(m, mx);
    const float alpha = expf(m - m_new);
    const float p = (key < n_keys) ? expf(s - m_new) : 0.f;
    float ps = p;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l = l * alpha + ps;
#pragma unroll
    for (int c = 0; c < kPer; ++c) acc[c] *= alpha;
    const int nk = min(kKeyBlock, n_keys - kv0);
    for (int j = 0; j < nk; ++j) {
      const float pj = __shfl_sync(0xffffffffu, p, j);
      const float* vr = v + head + (size_t)(kv0 + j) * D;
#pragma unroll
      for (int c = 0; c < kPer; ++c) acc[c] = fmaf(pj, vr[lane + 32 * c], acc[c]);
    }
    m = m_new;
  }
  const float inv_l = 1.f / l;
#pragma unroll
  for (int c = 0; c < kPer; ++c) o[head + (size_t)row * D + lane + 32 * c] = acc[c] * inv_l;
  if (lane == 0) lse[(size_t)blockIdx.y * N + row] = m + logf(l);
}

// delta_i = sum_c dO_ic O_ic
template <int D>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
    delta_fp32_kernel(const float* __restrict__ o, const float* __restrict__ dout,
                      float* __restrict__ delta, int N, int Npad) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + warp;
  if (row >= N) return;
  const size_t base = ((size_t)blockIdx.y * N + row) * D;
  float s = 0.f;
  for (int c = lane; c < D; c += 32) s = fmaf(dout[base + c], o[base + c], s);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) delta[(size_t)blockIdx.y * Npad + row] = s;
}

// dQ_i = scale * sum_j P_ij (dP_ij - delta_i) K_j, one warp per query row i.
template <int D>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
    dq_fp32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                   const float* __restrict__ v, const float* __restrict__ lse,
                   const float* __restrict__ dout, const float* __restrict__ delta,
                   float* __restrict__ dq, int N, int Npad, float scale, int causal) {
  constexpr int kPer = D / 32;
  __shared__ float s_q[kRowsPerBlock][D];
  __shared__ float s_do[kRowsPerBlock][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + warp;
  const size_t head = (size_t)blockIdx.y * N * D;
  if (row >= N) return;
  for (int c = lane; c < D; c += 32) {
    s_q[warp][c] = q[head + (size_t)row * D + c];
    s_do[warp][c] = dout[head + (size_t)row * D + c];
  }
  __syncwarp();
  const float lse_i = lse[(size_t)blockIdx.y * N + row];
  const float d_i = delta[(size_t)blockIdx.y * Npad + row];
  float acc[kPer];
#pragma unroll
  for (int c = 0; c < kPer; ++c) acc[c] = 0.f;
  const int n_keys = causal ? row + 1 : N;
  for (int kv0 = 0; kv0 < n_keys; kv0 += 32) {
    const int key = kv0 + lane;
    float ds = 0.f;
    if (key < n_keys) {
      const float* kr = k + head + (size_t)key * D;
      const float* vr = v + head + (size_t)key * D;
      float s = 0.f, dp = 0.f;
      for (int t = 0; t < D; ++t) {
        s = fmaf(s_q[warp][t], kr[t], s);
        dp = fmaf(s_do[warp][t], vr[t], dp);
      }
      const float p = expf(s * scale - lse_i);
      ds = p * (dp - d_i);
    }
    const int nk = min(32, n_keys - kv0);
    for (int j = 0; j < nk; ++j) {
      const float dsj = __shfl_sync(0xffffffffu, ds, j);
      const float* kr = k + head + (size_t)(kv0 + j) * D;
#pragma unroll
      for (int c = 0; c < kPer; ++c) acc[c] = fmaf(dsj, kr[lane + 32 * c], acc[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < kPer; ++c) dq[head + (size_t)row * D + lane + 32 * c] = acc[c] * scale;
}

// dV_j = sum_i P_ij dO_i ; dK_j = scale * sum_i P_ij (dP_ij - delta_i) Q_i,
// one warp per key row j.
template <int D>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
    dkdv_fp32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                     const float* __restrict__ v, const float* __restrict__ lse,
                     const float* __restrict__ dout, const float* __restrict__ delta,
                     float* __restrict__ dk, float* __restrict__ dv, int N, int Npad, float scale,
                     int causal) {
  constexpr int kPer = D / 32;
  __shared__ float s_k[kRowsPerBlock][D];
  __shared__ float s_v[kRowsPerBlock][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int key = blockIdx.x * kRowsPerBlock + warp;
  const size_t head = (size_t)blockIdx.y * N * D;
  if (key >= N) return;
  for (int c = lane; c < D; c += 32) {
    s_k[warp][c] = k[head + (size_t)key * D + c];
    s_v[warp][c] = v[head + (size_t)key * D + c];
  }
  __syncwarp();
  float acc_k[kPer], acc_v[kPer];
#pragma unroll
  for (int c = 0; c < kPer; ++c) acc_k[c] = acc_v[c] = 0.f;
  const int i_begin = causal ? key : 0;
  for (int i0 = i_begin; i0 < N; i0 += 32) {
    const int qi = i0 + lane;
    float p = 0.f, ds = 0.f;
    if (qi < N) {
      const float* qr = q + head + (size_t)qi * D;
      const float* dor = dout + head + (size_t)qi * D;
      float s = 0.f, dp = 0.f;
      for (int t = 0; t < D; ++t) {
        s = fmaf(qr[t], s_k[warp][t], s);
        dp = fmaf(dor[t], s_v[warp][t], dp);
      }
      p = expf(s * scale - lse[(size_t)blockIdx.y * N + qi]);
      ds = p * (dp - delta[(size_t)blockIdx.y * Npad + qi]);
    }
    const int nq = min(32, N - i0);
    for (int j = 0; j < nq; ++j) {
      const float pj = __shfl_sync(0xffffffffu, p, j);
      const float dsj = __shfl_sync(0xffffffffu, ds, j);
      const float* qr = q + head + (size_t)(i0 + j) * D;
      const float* dor = dout + head + (size_t)(i0 + j) * D;
#pragma unroll
      for (int c = 0; c < kPer; ++c) {
        acc_v[c] = fmaf(pj, dor[lane + 32 * c], acc_v[c]);
        acc_k[c] = fmaf(dsj, qr[lane + 32 * c], acc_k[c]);
      }
    }
  }
#pragma unroll
  for (int c = 0; c < kPer; ++c) {
    dv[head + (size_t)key * D + lane + 32 * c] = acc_v[c];
    dk[head + (size_t)key * D + lane + 32 * c] = acc_k[c] * scale;
  }
}

template <int D>
cudaError_t fwd_fp32_impl(const Problem& p, const float* q, const float* k, const float* v,
                          float* o, float* lse, cudaStream_t stream) {
  dim3 grid(ceil_div(p.N, kRowsPerBlock), p.B * p.H);
  fwd_fp32_kernel<D><<<grid, 32 * kRowsPerBlock, 0, stream>>>(q, k, v, o, lse, p.N, p.scale,
                                                               p.causal);
  return cudaGetLastError();
}

template <int D>
cudaError_t bwd_fp32_impl(const Problem& p, const float* q, const float* k, const float* v,
                          const float* o, const float* lse, const float* dout, float* dq,
                          float* dk, float* dv, const BwdWorkspace& ws, cudaStream_t stream) {
  dim3 grid(ceil_div(p.N, kRowsPerBlock), p.B * p.H);
  const int Npad = n_pad(p.N);
  delta_fp32_kernel<D><<<grid, 32 * kRowsPerBlock, 0, stream>>>(o, dout, ws.delta, p.N, Npad);
  dq_fp32_kernel<D><<<grid, 32 * kRowsPerBlock, 0, stream>>>(q, k, v, lse, dout, ws.delta, dq, p.N,
                                                             Npad, p.scale, p.causal);
  dkdv_fp32_kernel<D><<<grid, 32 * kRowsPerBlock, 0, stream>>>(q, k, v, lse, dout, ws.delta, dk,
                                                               dv, p.N, Npad, p.scale, p.causal);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_fp32(const Problem& p, const float* q, const float* k, const float* v,
                            float* o, float* lse, cudaStream_t stream) {
  return p.d == 128 ? fwd_fp32_impl<128>(p, q, k, v, o, lse, stream)
                    : fwd_fp32_impl<64>(p, q, k, v, o, lse, stream);
}

cudaError_t launch_bwd_fp32(const Problem& p, const float* q, const float* k, const float* v,
                            const float* o, const float* lse, const float* dout, float* dq,
                            float* dk, float* dv, const BwdWorkspace& ws, cudaStream_t stream) {
  return p.d == 128 ? bwd_fp32_impl<128>(p, q, k, v, o, lse, dout, dq, dk, dv, ws, stream)
                    : bwd_fp32_impl<64>(p, q, k, v, o, lse, dout, dq, dk, dv, ws, stream);
}

}  // namespace attn
