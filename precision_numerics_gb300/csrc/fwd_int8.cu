// INT8-input attention forward for sm_103a.
//
// What is computed ("INT-FlashAttention: Enabling Flash Attention for INT8
// Quantization", abstract: INT8 quantization inside the FlashAttention
// forward; the page gives no more detail, so the scheme is a reading):
//   Q and K are quantized per token -- one symmetric FP32 scale per row of
//   each head, s = max|x| / 127, code = rint(x / s) clamped to [-127, 127]
//   (attn_quantize_int8 below); V stays BF16.  The scores are
//   S_ij = scale * s_q[i] * s_k[j] * (q8_i . k8_j), the integer dot product
//   exact in INT32; then the FP32 online softmax and P V (P rounded to BF16)
//   as in the BF16 forward, O = P V / l and LSE = m + ln l.
//
// sm_103a has no INT8 form of tcgen05.mma (ptxas rejects kind::i8 for this
// target).  The fast path is attn_fwd_int8_as_bf16: the same codes held in
// BF16 run through the tcgen05 forward of fwd_bf16.cu, where every product
// and partial sum of the integer dot product is exact in FP32.  For int8
// codes, this file's kernel uses the warp-level tensor-core path:
// mma.sync m16n8k32 s8 for Q K^T and m16n8k16 bf16 for P V.  CTA = 64 query
// rows of one (b, h), 4 warps x 16 rows; key tiles of 64 rows stream through
// a two-stage cp.async ring.  Each thread holds rows g and g+8 of its warp's
// 16 (g = lane / 4) and, of every 8-column tile, columns 2t and 2t+1
// (t = lane % 4), the mma accumulator layout; a row's max and sum are
// reduced over its four threads with shuffles.  Control flow is uniform, and
// the only waits are __syncthreads and cp.async groups.
#include <math.h>
#include <stdint.h>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kI8Rows = 64;     // query rows per CTA
constexpr int kI8Keys = 64;     // key rows per tile
constexpr int kI8Threads = 128;

template <int D>
struct I8Cfg {
  static constexpr int kRowI8 = D + 16;       // padded INT8 row (bytes): conflict-free 32-bit loads
  static constexpr int kRowV = 2 * D + 16;    // padded BF16 V row (bytes): conflict-free ldmatrix
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kI8Rows * kRowI8;
  static constexpr int kOffV = kOffK + 2 * kI8Keys * kRowI8;
  static constexpr int kOffKs = kOffV + 2 * kI8Keys * kRowV;
  static constexpr int kSmemBytes = kOffKs + 2 * kI8Keys * 4;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  // src-size 0 zero-fills the 16 bytes (rows past N); src stays a valid address.
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// C[16x8] (int32) += A[16x32] (s8, row) * B[32x8] (s8, col).
__device__ __forceinline__ void mma_s8(int (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// C[16x8] (f32) += A[16x16] (bf16, row) * B[16x8] (bf16, col).
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Two transposed 8x8 BF16 matrices: the B fragment of m16n8k16 from a
// row-major [key][d] tile (lanes 0-15 give the 16 key rows' addresses).
__device__ __forceinline__ void ldmatrix_x2_trans(uint32_t& r0, uint32_t& r1, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}

// ----------------------------------------------------------------- quantize
// Each lane handles 16-byte units (8 values): a row of d values is D/8 lanes
// (16 at d = 128, 8 at d = 64), so one warp load covers 32 / (D/8) rows, and
// a warp keeps kQuantGroups such row groups in flight.  FP32 max|x| by
// shuffles inside the row's lane group, s = max / 127, codes rint(x / s)
// clamped to +-127 (rint: half to even), zero row -> 0.
//
// BF16_CODES: codes written as BF16 values (exact integers) and scales in the
// padded per-head layout [B*H][n_pad] (n_pad = N rounded up to 128), whose
// padding the lanes of each head's last row zero; otherwise int8 codes and
// scales [B*H*N].
constexpr int kQuantGroups = 4;
template <int D>
constexpr long long quant_rows_per_block() {
  return 8LL * kQuantGroups * (32 / (D / 8));
}
template <int D, bool BF16_CODES>
__global__ void __launch_bounds__(256) quantize_int8_kernel(const uint16_t* __restrict__ x,
                                                            void* __restrict__ codes_out,
                                                            float* __restrict__ scales,
                                                            long long rows, int N, int n_pad) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerLoad = 32 / kLanesPerRow;
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerRow, part = lane % kLanesPerRow;
  const long long warp_global = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const long long row_base = warp_global * (kQuantGroups * kRowsPerLoad);
  uint4 w[kQuantGroups];
#pragma unroll
  for (int q = 0; q < kQuantGroups; ++q) {
    const long long row = row_base + q * kRowsPerLoad + sub;
    w[q] = row < rows ? *reinterpret_cast<const uint4*>(x + row * D + part * 8)
                      : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int q = 0; q < kQuantGroups; ++q) {
    const long long row = row_base + q * kRowsPerLoad + sub;
    const uint32_t u[4] = {w[q].x, w[q].y, w[q].z, w[q].w};
    float v[8];
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      v[e] = __uint_as_float(e & 1 ? (u[e >> 1] & 0xFFFF0000u) : (u[e >> 1] << 16));
      amax = fmaxf(amax, fabsf(v[e]));
    }
    // All lanes take part (rows past the end hold zeros); the xor offsets stay
    // inside the row's aligned group of kLanesPerRow lanes.
#pragma unroll
    for (int off = kLanesPerRow / 2; off > 0; off >>= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (row >= rows) continue;
    const float s = amax / 127.f;
    uint32_t packed[2] = {0u, 0u};
    uint32_t bf[4];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float r = s > 0.f ? rintf(v[e] / s) : 0.f;
      const float cf = fminf(fmaxf(r, -127.f), 127.f);
      packed[e >> 2] |= (static_cast<uint32_t>(static_cast<int>(cf)) & 0xFFu) << (8 * (e & 3));
      if (e & 1) bf[e >> 1] = pack_bf16x2(__uint_as_float(bf[e >> 1]), cf);
      else bf[e >> 1] = __float_as_uint(cf);
    }
    if constexpr (BF16_CODES) {
      uint16_t* codes = static_cast<uint16_t*>(codes_out);
      *reinterpret_cast<uint4*>(codes + row * D + part * 8) = make_uint4(bf[0], bf[1], bf[2], bf[3]);
      const long long bh = row / N, n = row - bh * N;
      if (part == 0) scales[bh * n_pad + n] = s;
      if (n == N - 1)  // this head's padded scale entries
        for (int z = N + part; z < n_pad; z += kLanesPerRow) scales[bh * n_pad + z] = 0.f;
    } else {
      int8_t* codes = static_cast<int8_t*>(codes_out);
      *reinterpret_cast<uint2*>(codes + row * D + part * 8) = make_uint2(packed[0], packed[1]);
      if (part == 0) scales[row] = s;
    }
  }
}

// ---------------------------------------------------------------- attention
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kI8Threads, 3)  // 3 CTAs per SM: 168 registers
    fwd_int8_kernel(const int8_t* __restrict__ q8, const float* __restrict__ qs,
                    const int8_t* __restrict__ k8, const float* __restrict__ ks,
                    const uint16_t* __restrict__ v, uint16_t* __restrict__ o,
                    float* __restrict__ lse, int BH, int N, int num_qt, float scale) {
  using C = I8Cfg<D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int qt = num_qt - 1 - (int)(blockIdx.x / BH);  // heaviest query tiles first
  const int bh = (int)(blockIdx.x % BH);
  const int q0 = qt * kI8Rows;
  const size_t head = (size_t)bh * N;
  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sK = smem_u32(smem + C::kOffK);
  const uint32_t sV = smem_u32(smem + C::kOffV);
  const float* sKs = reinterpret_cast<const float*>(smem + C::kOffKs);

  const int last_q = min(q0 + kI8Rows, N) - 1;
  const int n_kt = CAUSAL ? last_q / kI8Keys + 1 : (N + kI8Keys - 1) / kI8Keys;

  // Loads of one key tile (INT8 K, BF16 V, K scales) into ring stage st.
  auto load_kv = [&](int j, int st) {
    constexpr int kI8Units = D / 16, kVUnits = D / 8;  // 16-byte units per row
    for (int u = threadIdx.x; u < kI8Keys * kI8Units; u += kI8Threads) {
      const int rr = u / kI8Units, cc = u % kI8Units;
      const int key = j * kI8Keys + rr;
      const bool ok = key < N;
      cp_async16(sK + st * kI8Keys * C::kRowI8 + rr * C::kRowI8 + cc * 16,
                 k8 + (head + (ok ? key : 0)) * D + cc * 16, ok);
    }
    for (int u = threadIdx.x; u < kI8Keys * kVUnits; u += kI8Threads) {
      const int rr = u / kVUnits, cc = u % kVUnits;
      const int key = j * kI8Keys + rr;
      const bool ok = key < N;
      cp_async16(sV + st * kI8Keys * C::kRowV + rr * C::kRowV + cc * 16,
                 v + (head + (ok ? key : 0)) * D + cc * 8, ok);
    }
    // K scales with plain loads: a head's scales need not start on 16 bytes.
    // Stage st was last read before the previous iteration's closing barrier.
    if (threadIdx.x < kI8Keys) {
      const int key = j * kI8Keys + threadIdx.x;
      reinterpret_cast<float*>(smem + C::kOffKs)[st * kI8Keys + threadIdx.x] =
          key < N ? ks[head + key] : 0.f;
    }
  };

  // Q tile (INT8) once, then the first key tile.
  {
    constexpr int kUnits = D / 16;
    for (int u = threadIdx.x; u < kI8Rows * kUnits; u += kI8Threads) {
      const int rr = u / kUnits, cc = u % kUnits;
      const int row = q0 + rr;
      const bool ok = row < N;
      cp_async16(sQ + rr * C::kRowI8 + cc * 16, q8 + (head + (ok ? row : 0)) * D + cc * 16, ok);
    }
  }
  load_kv(0, 0);
  cp_async_commit();

  const int r_lo = q0 + warp * 16 + g, r_hi = r_lo + 8;  // this thread's two query rows
  const float rs_lo = r_lo < N ? qs[head + r_lo] * scale : 0.f;
  const float rs_hi = r_hi < N ? qs[head + r_hi] * scale : 0.f;
  constexpr float kLog2e = 1.4426950408889634f;

  uint32_t aq[D / 32][4];  // Q fragments, reused for every key tile
  float acc[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

  for (int j = 0; j < n_kt; ++j) {
    const int st = j & 1;
    if (j + 1 < n_kt) load_kv(j + 1, st ^ 1);
    cp_async_commit();
    cp_async_wait<1>();  // tile j (and Q) landed
    __syncthreads();
    if (j == 0) {
#pragma unroll
      for (int kk = 0; kk < D / 32; ++kk) {
        const uint32_t base = sQ + (warp * 16 + g) * C::kRowI8 + kk * 32 + 4 * t;
        aq[kk][0] = lds32(base);
        aq[kk][1] = lds32(base + 8 * C::kRowI8);
        aq[kk][2] = lds32(base + 16);
        aq[kk][3] = lds32(base + 8 * C::kRowI8 + 16);
      }
    }
    // S = Q8 K8^T (exact INT32), 8 column tiles of 8 keys.
    int sc[kI8Keys / 8][4];
#pragma unroll
    for (int n = 0; n < kI8Keys / 8; ++n) {
      sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0;
      const uint32_t kb = sK + st * kI8Keys * C::kRowI8 + (n * 8 + g) * C::kRowI8 + 4 * t;
#pragma unroll
      for (int kk = 0; kk < D / 32; ++kk)
        mma_s8(sc[n], aq[kk], lds32(kb + kk * 32), lds32(kb + kk * 32 + 16));
    }
    // Dequantize, mask, online softmax (rows r_lo, r_hi; 16 columns each).
    const float* ksc = sKs + st * kI8Keys;
    const int kv0 = j * kI8Keys;
    const bool edge = kv0 + kI8Keys > N || (CAUSAL && kv0 + kI8Keys - 1 > q0);
    float s_lo[kI8Keys / 8][2], s_hi[kI8Keys / 8][2];
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int n = 0; n < kI8Keys / 8; ++n) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int col = n * 8 + 2 * t + e;
        const float kscale = ksc[col];
        float a = static_cast<float>(sc[n][e]) * rs_lo * kscale;
        float b = static_cast<float>(sc[n][2 + e]) * rs_hi * kscale;
        if (edge) {
          const int key = kv0 + col;
          if (key >= N || (CAUSAL && key > r_lo)) a = -INFINITY;
          if (key >= N || (CAUSAL && key > r_hi)) b = -INFINITY;
        }
        s_lo[n][e] = a;
        s_hi[n][e] = b;
        mx_lo = fmaxf(mx_lo, a);
        mx_hi = fmaxf(mx_hi, b);
      }
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, off));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, off));
    }
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float mu_lo = mn_lo == -INFINITY ? 0.f : mn_lo, mu_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
    const float al_lo = ex2((m_lo - mu_lo) * kLog2e), al_hi = ex2((m_hi - mu_hi) * kLog2e);
    m_lo = mn_lo;
    m_hi = mn_hi;
    l_lo *= al_lo;
    l_hi *= al_hi;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      acc[n][0] *= al_lo;
      acc[n][1] *= al_lo;
      acc[n][2] *= al_hi;
      acc[n][3] *= al_hi;
    }
    uint32_t pa[kI8Keys / 16][4];  // P as A fragments of m16n8k16 (16 keys each)
    const float nm_lo = -mu_lo * kLog2e, nm_hi = -mu_hi * kLog2e;
#pragma unroll
    for (int n = 0; n < kI8Keys / 8; ++n) {
      const float p0 = ex2(fmaf(s_lo[n][0], kLog2e, nm_lo)), p1 = ex2(fmaf(s_lo[n][1], kLog2e, nm_lo));
      const float p2 = ex2(fmaf(s_hi[n][0], kLog2e, nm_hi)), p3 = ex2(fmaf(s_hi[n][1], kLog2e, nm_hi));
      l_lo += p0 + p1;
      l_hi += p2 + p3;
      pa[n >> 1][(n & 1) * 2 + 0] = pack_bf16x2(p0, p1);  // row g,   keys 16kb + 8(n&1) + 2t
      pa[n >> 1][(n & 1) * 2 + 1] = pack_bf16x2(p2, p3);  // row g+8
    }
    // O += P V: 16-key blocks kb, 8-column tiles of d.
    const uint32_t vb = sV + st * kI8Keys * C::kRowV + (lane & 15) * C::kRowV;
#pragma unroll
    for (int kb = 0; kb < kI8Keys / 16; ++kb) {
      // m16n8k16 A: {row g k 0-7, row g+8 k 0-7, row g k 8-15, row g+8 k 8-15}
      const uint32_t a[4] = {pa[kb][0], pa[kb][1], pa[kb][2], pa[kb][3]};
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        uint32_t b0, b1;
        ldmatrix_x2_trans(b0, b1, vb + kb * 16 * C::kRowV + n * 16);
        mma_bf16(acc[n], a, b0, b1);
      }
    }
    __syncthreads();  // stage st is refilled by the next iteration's loads
  }
  cp_async_wait<0>();

  // Row sums over the four threads of each row, then O / l and LSE.
#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, off);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, off);
  }
  const float il_lo = l_lo > 0.f ? 1.f / l_lo : 0.f, il_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    const int col = n * 8 + 2 * t;
    if (r_lo < N)
      *reinterpret_cast<uint32_t*>(o + (head + r_lo) * D + col) =
          pack_bf16x2(acc[n][0] * il_lo, acc[n][1] * il_lo);
    if (r_hi < N)
      *reinterpret_cast<uint32_t*>(o + (head + r_hi) * D + col) =
          pack_bf16x2(acc[n][2] * il_hi, acc[n][3] * il_hi);
  }
  if (t == 0) {
    if (r_lo < N) lse[head + r_lo] = m_lo + logf(l_lo);
    if (r_hi < N) lse[head + r_hi] = m_hi + logf(l_hi);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_int8_impl(const Problem& p, const int8_t* q8, const float* qs, const int8_t* k8,
                             const float* ks, const uint16_t* v, uint16_t* o, float* lse,
                             cudaStream_t stream) {
  using C = I8Cfg<D>;
  auto kernel = fwd_int8_kernel<D, CAUSAL>;
  cudaError_t err =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (err != cudaSuccess) return err;
  const int BH = p.B * p.H;
  const int num_qt = ceil_div(p.N, kI8Rows);
  kernel<<<dim3((unsigned)BH * num_qt), dim3(kI8Threads), C::kSmemBytes, stream>>>(
      q8, qs, k8, ks, v, o, lse, BH, p.N, num_qt, p.scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_int8(const Problem& p, const void* x, void* codes, float* scales,
                                 cudaStream_t stream) {
  const long long rows = (long long)p.B * p.H * p.N;
  const auto* xx = static_cast<const uint16_t*>(x);
  if (p.d == 128) {
    constexpr long long per = quant_rows_per_block<128>();
    quantize_int8_kernel<128, false><<<(unsigned)((rows + per - 1) / per), 256, 0, stream>>>(
        xx, codes, scales, rows, p.N, p.N);
  } else {
    constexpr long long per = quant_rows_per_block<64>();
    quantize_int8_kernel<64, false><<<(unsigned)((rows + per - 1) / per), 256, 0, stream>>>(
        xx, codes, scales, rows, p.N, p.N);
  }
  return cudaGetLastError();
}

cudaError_t launch_quantize_int8_as_bf16(const Problem& p, const void* x, void* codes,
                                         float* scales, cudaStream_t stream) {
  const long long rows = (long long)p.B * p.H * p.N;
  const auto* xx = static_cast<const uint16_t*>(x);
  const int np = n_pad(p.N);
  if (p.d == 128) {
    constexpr long long per = quant_rows_per_block<128>();
    quantize_int8_kernel<128, true><<<(unsigned)((rows + per - 1) / per), 256, 0, stream>>>(
        xx, codes, scales, rows, p.N, np);
  } else {
    constexpr long long per = quant_rows_per_block<64>();
    quantize_int8_kernel<64, true><<<(unsigned)((rows + per - 1) / per), 256, 0, stream>>>(
        xx, codes, scales, rows, p.N, np);
  }
  return cudaGetLastError();
}

cudaError_t launch_fwd_int8(const Problem& p, const void* q8, const float* qs, const void* k8,
                            const float* ks, const void* v, void* o, float* lse,
                            cudaStream_t stream) {
  const auto* q = static_cast<const int8_t*>(q8);
  const auto* k = static_cast<const int8_t*>(k8);
  const auto* vv = static_cast<const uint16_t*>(v);
  auto* oo = static_cast<uint16_t*>(o);
  if (p.d == 128)
    return p.causal ? launch_int8_impl<128, true>(p, q, qs, k, ks, vv, oo, lse, stream)
                    : launch_int8_impl<128, false>(p, q, qs, k, ks, vv, oo, lse, stream);
  return p.causal ? launch_int8_impl<64, true>(p, q, qs, k, ks, vv, oo, lse, stream)
                  : launch_int8_impl<64, false>(p, q, qs, k, ks, vv, oo, lse, stream);
}

}  // namespace attn
