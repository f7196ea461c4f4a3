// BF16 attention backward for sm_103a from the saved LSE.
//
// What is computed (the gradient of softmax attention for L = sum(dO o O)):
//   delta_i = rowsum(dO o O)_i      ("Why Low-Precision Transformer Training
//                                     Fails", Figures 3 and 5), from the
//                                     stored BF16 O, in FP32
//   P_ij    = exp(scale q_i.k_j - LSE_i)          (recomputed, causal mask)
//   dV      = P^T dO
//   dP      = dO V^T
//   dS      = P o (dP - delta)
//   dK      = scale dS^T Q,   dQ = scale dS K
//
// Three kernels, in stream order:
//   1. preprocess   delta, -LSE * log2(e) (-inf on padded rows, so the
//                   recomputed P of a padded query row is exactly 0), and a
//                   zeroed FP32 dQ accumulator.  Memory-bound.
//   2. main         one CTA per (b, h, 128-key tile j), K_j and V_j resident in
//                   shared memory; the CTA walks the query tiles i (causal:
//                   i >= j) with Q_i, dO_i, LSE_i, delta_i streamed by TMA.
//                   Per tile, five tcgen05 MMAs (128 x 128 x 128 each):
//                     S^T  = K_j Q_i^T            (SS)  -> TMEM
//                     dP^T = V_j dO_i^T           (SS)  -> TMEM
//                     dV  += P^T dO_i             (TS, P^T in TMEM)
//                     dK  += dS^T Q_i             (TS, dS^T in TMEM)
//                     dQ_i = dS K_j               (SS, dS from shared memory)
//                   and dQ_i is added into the FP32 accumulator with
//                   red.global.add.f32 (a warp's 32 reductions cover 128
//                   contiguous bytes).  Warp roles (d = 64 variant; the d = 128
//                   one is described at r64): 0 TMA producer, 1 MMA issuer,
//                   2 TMEM owner, 4-7 P / dS compute (one key row per thread),
//                   8-11 dQ drain; the epilogue writes dV (warps 4-7) and
//                   scale * dK (warps 8-11) with TMA stores.
//   3. dq_convert   dQ = bf16(scale * accumulator).  Memory-bound.
//
// Two variants of the main kernel: d = 64 uses 128-row query tiles
// (bwd_main_kernel below; TMEM dV [0,64), dK [64,128), S^T [128,256), dP^T
// [256,384), dQ [384,448)); d = 128 uses 64-row query tiles with an
// overlapped MMA order (r64::bwd_main_d128_kernel, described there).
// bwd_main_kernel also supports d = 128 (dQ then reuses the S^T columns: the
// MMA that reads P^T from there is issued first, and tcgen05 MMAs of one
// thread execute in order).
#include <math.h>

#include <type_traits>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {

static __device__ unsigned int g_status_bwd;

namespace {

__device__ __forceinline__ void set_fail(unsigned int code) { atomicOr(&g_status_bwd, code); }

// ---------------------------------------------------------------------------
// 1. preprocess
// ---------------------------------------------------------------------------
// Each group of d/8 threads handles one padded row; each thread owns 8
// consecutive columns (16 bytes of O and of dO, 32 bytes of the accumulator).
template <int D>
__global__ void __launch_bounds__(256)
    bwd_preprocess_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout,
                          const float* __restrict__ lse, float* __restrict__ neg_lse2,
                          float* __restrict__ delta, float4* __restrict__ dqacc, int N, int Npad,
                          int blocks_per_head) {
  constexpr int kGroup = D / 8;
  constexpr int kRows = 256 / kGroup;
  // One-dimensional grid (B*H may exceed the 65535 limit of gridDim.y).
  const int bh = (int)(blockIdx.x / (unsigned)blocks_per_head);
  const int row = (int)(blockIdx.x % (unsigned)blocks_per_head) * kRows + threadIdx.x / kGroup;
  const int part = threadIdx.x % kGroup;
  const bool active = row < Npad;
  float s = 0.f;
  if (active && row < N) {
    const size_t idx = ((size_t)bh * N + row) * kGroup + part;
    const uint4 a = o[idx], b = dout[idx];
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s = fmaf(__uint_as_float(av[i] << 16), __uint_as_float(bv[i] << 16), s);
      s = fmaf(__uint_as_float(av[i] & 0xFFFF0000u), __uint_as_float(bv[i] & 0xFFFF0000u), s);
    }
  }
#pragma unroll
  for (int off = kGroup / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (!active) return;
  const size_t prow = (size_t)bh * Npad + row;
  if (part == 0) {
    delta[prow] = s;
    neg_lse2[prow] = row < N ? -(lse[(size_t)bh * N + row] * 1.4426950408889634f) : -INFINITY;
  }
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  dqacc[prow * (D / 4) + 2 * part] = z;
  dqacc[prow * (D / 4) + 2 * part + 1] = z;
}

// ---------------------------------------------------------------------------
// 3. dq_convert
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256)
    bwd_dq_convert_kernel(const float4* __restrict__ dqacc, uint4* __restrict__ dq, int N,
                          int Npad, float scale, int total_units) {
  const int u = blockIdx.x * blockDim.x + threadIdx.x;  // one unit = 8 columns of one row
  if (u >= total_units) return;
  constexpr int kUnitsPerRow = D / 8;
  const int col8 = u % kUnitsPerRow;
  const int row = (u / kUnitsPerRow) % N;
  const int bh = u / (kUnitsPerRow * N);
  const size_t src = ((size_t)bh * Npad + row) * (D / 4) + 2 * col8;
  const float4 a = dqacc[src], b = dqacc[src + 1];
  uint4 out;
  out.x = pack_bf16x2(a.x * scale, a.y * scale);
  out.y = pack_bf16x2(a.z * scale, a.w * scale);
  out.z = pack_bf16x2(b.x * scale, b.y * scale);
  out.w = pack_bf16x2(b.z * scale, b.w * scale);
  dq[u] = out;
}

// ---------------------------------------------------------------------------
// 2. main kernel
// ---------------------------------------------------------------------------
constexpr int kThreads = 384;

template <int D>
struct BwdCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunkBytes = 128 * 128;   // 128 rows x 128 bytes
  static constexpr int kTileBytes = 128 * D * 2;  // 128 rows x d BF16
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;        // 2 stages
  static constexpr int kOffDO = kOffQ + 2 * kTileBytes;   // 2 stages
  static constexpr int kOffDS = kOffDO + 2 * kTileBytes;  // 128 key rows x 128 query cols BF16
  static constexpr int kDSBytes = 128 * 128 * 2;
  static constexpr int kOffLse = kOffDS + kDSBytes;    // 2 stages x 128 FP32
  static constexpr int kOffDelta = kOffLse + 2 * 512;  // 2 stages x 128 FP32
  static constexpr int kOffBar = kOffDelta + 2 * 512;
  // kv_full, qdo_full[2], qdo_empty[2], s_full, dp_full, p_ready, ds_ready,
  // dq_full, dq_free, dkv_done, mma_final, epi_dv, epi_dk
  static constexpr int kNumBars = 15;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;
  static constexpr uint32_t kColDV = 0;
  static constexpr uint32_t kColDK = D;
  static constexpr uint32_t kColS = 2 * D;
  static constexpr uint32_t kColDP = 2 * D + 128;
  static constexpr uint32_t kColDQ = (D == 128) ? kColS : 384u;
  static constexpr bool kDqAliasesS = (D == 128);
  static constexpr uint32_t kTmemCols = 512;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV,
                    const float* __restrict__ neg_lse2, const float* __restrict__ delta,
                    float* __restrict__ dqacc, int BH, int N, int Npad, float scale,
                    float scale_log2) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_qt = Npad / kBlockM;

  // Key tiles with the most query tiles (causal: small j) first.
  const int j = blockIdx.x / BH;
  const int bh = blockIdx.x % BH;
  const int i_first = CAUSAL ? j : 0;
  const int nq = n_qt - i_first;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* bar_kv = bars + 0;
  uint64_t* bar_qfull = bars + 1;   // [2]
  uint64_t* bar_qempty = bars + 3;  // [2]
  uint64_t* bar_sfull = bars + 5;
  uint64_t* bar_dpfull = bars + 6;
  uint64_t* bar_pready = bars + 7;
  uint64_t* bar_dsready = bars + 8;
  uint64_t* bar_dqfull = bars + 9;
  uint64_t* bar_dqfree = bars + 10;
  uint64_t* bar_dkvdone = bars + 11;
  uint64_t* bar_final = bars + 12;
  uint64_t* bar_epi_dv = bars + 13;
  uint64_t* bar_epi_dk = bars + 14;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    *s_abort = (smem_u32(smem) & 1023u) != 0;
    if (*s_abort) set_fail(ATTN_ERR_INVALID_ARG);
    mbar_init(bar_kv, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_qfull[s], 1);
      mbar_init(&bar_qempty[s], 1 + 4);  // MMA commit + one arrive per compute warp
    }
    mbar_init(bar_sfull, 1);
    mbar_init(bar_dpfull, 1);
    mbar_init(bar_pready, 128);
    mbar_init(bar_dsready, 128);
    mbar_init(bar_dqfull, 1);
    mbar_init(bar_dqfree, 128);
    mbar_init(bar_dkvdone, 1);
    mbar_init(bar_final, 1);
    mbar_init(bar_epi_dv, 128);
    mbar_init(bar_epi_dk, 128);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool abort_all = *s_abort != 0;

  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sDO = smem + C::kOffDO;
  uint8_t* sDS = smem + C::kOffDS;
  float* sLse = reinterpret_cast<float*>(smem + C::kOffLse);
  float* sDelta = reinterpret_cast<float*>(smem + C::kOffDelta);

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 72;");
    if (warp == 0 && lane == 0 && !abort_all) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      mbar_arrive_expect_tx(bar_kv, 2 * C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_3d(sK + c * C::kChunkBytes, &tmK, bar_kv, c * 64, j * kBlockN, bh);
        tma_load_3d(sV + c * C::kChunkBytes, &tmV, bar_kv, c * 64, j * kBlockN, bh);
      }
      bool ok = true;
      int issued = 0;
      for (int it = 0; it < nq; ++it) {
        const int st = it & 1, use = it >> 1;
        const int i = i_first + it;
        if (use > 0 && !mbar_wait(&bar_qempty[st], (use - 1) & 1)) { ok = false; break; }
        mbar_arrive_expect_tx(&bar_qfull[st], 2 * C::kTileBytes + 2 * 512);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(sQ + st * C::kTileBytes + c * C::kChunkBytes, &tmQ, &bar_qfull[st], c * 64,
                      i * kBlockM, bh);
          tma_load_3d(sDO + st * C::kTileBytes + c * C::kChunkBytes, &tmDO, &bar_qfull[st], c * 64,
                      i * kBlockM, bh);
        }
        const size_t prow = (size_t)bh * Npad + (size_t)i * kBlockM;
        bulk_load(sLse + st * 128, neg_lse2 + prow, 512, &bar_qfull[st]);
        bulk_load(sDelta + st * 128, delta + prow, 512, &bar_qfull[st]);
        issued = it + 1;
      }
      if (!ok) set_fail(ATTN_ERR_TIMEOUT);
      // Do not leave while copies into this CTA's shared memory are in flight.
      mbar_wait(bar_kv, 0);
      for (int it = max(0, issued - 2); it < issued; ++it)
        mbar_wait(&bar_qfull[it & 1], (it >> 1) & 1);
    } else if (warp == 1 && !abort_all) {
      // ------------------------------------------------------------ MMA issuer
      // Whole warp, warp-uniform operands; elect.sync picks the issuing lane.
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);  // K-major A and B
      constexpr uint32_t idesc_acc = idesc_bf16(128, D, false, true);   // TMEM A, MN-major B
      constexpr uint32_t idesc_dq = idesc_bf16(128, D, true, true);     // MN-major A and B
      const uint64_t kK = sdesc_sw128(smem_u32(sK), 16, 1024);          // K-major views
      const uint64_t kV = sdesc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t kQ = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t kDO = sdesc_sw128(smem_u32(sDO), 16, 1024);
      const uint64_t mQ = sdesc_sw128(smem_u32(sQ), C::kChunkBytes, 1024);  // MN-major views
      const uint64_t mDO = sdesc_sw128(smem_u32(sDO), C::kChunkBytes, 1024);
      const uint64_t mDS = sdesc_sw128(smem_u32(sDS), C::kChunkBytes, 1024);
      const uint64_t mK = sdesc_sw128(smem_u32(sK), C::kChunkBytes, 1024);
      bool ok = warp_wait(bar_kv, 0);
      for (int it = 0; it < nq && ok; ++it) {
        const int st = it & 1, use = it >> 1;
        if (!warp_wait(&bar_qfull[st], use & 1)) { ok = false; break; }
        if (C::kDqAliasesS && it > 0 && !warp_wait(bar_dqfree, (it - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t so = st * C::kTileBytes;
        // S^T = K_j Q_i^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          mma_ss_elect(tmem + C::kColS, sdesc_add(kK, off), sdesc_add(kQ, so + off), idesc_s,
                       kk > 0 ? 1u : 0u);
        }
        mma_commit_elect(bar_sfull);
        // dP^T = V_j dO_i^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          mma_ss_elect(tmem + C::kColDP, sdesc_add(kV, off), sdesc_add(kDO, so + off), idesc_s,
                       kk > 0 ? 1u : 0u);
        }
        mma_commit_elect(bar_dpfull);
        // dV += P^T dO_i
        if (!warp_wait(bar_pready, it & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBlockM / 16; ++kk)
          mma_ts_elect(tmem + C::kColDV, tmem + C::kColS + kk * 8, sdesc_add(mDO, so + kk * 2048),
                       idesc_acc, (it > 0 || kk > 0) ? 1u : 0u);
        // dK += dS^T Q_i
        if (!warp_wait(bar_dsready, it & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBlockM / 16; ++kk)
          mma_ts_elect(tmem + C::kColDK, tmem + C::kColDP + kk * 8, sdesc_add(mQ, so + kk * 2048),
                       idesc_acc, (it > 0 || kk > 0) ? 1u : 0u);
        mma_commit_elect(&bar_qempty[st]);
        // dQ_i = dS K_j
        if (!C::kDqAliasesS && it > 0 && !warp_wait(bar_dqfree, (it - 1) & 1)) { ok = false; break; }
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          mma_ss_elect(tmem + C::kColDQ, sdesc_add(mDS, kk * 2048), sdesc_add(mK, kk * 2048),
                       idesc_dq, kk > 0 ? 1u : 0u);
        mma_commit_elect(bar_dqfull);
      }
      if (ok) mma_commit_elect(bar_dkvdone);
      else if (lane == 0) set_fail(ATTN_ERR_TIMEOUT);
      mma_commit_elect(bar_final);
      mbar_wait(bar_final, 0);
    }
    __syncwarp();
  } else if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 216;");
    // -------------------------------------------------- P and dS (key rows)
    const int r = (warp & 3) * 32 + lane;  // key row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::kColS;
    const uint32_t tDP = tmem + lane_off + C::kColDP;
    const bool key_valid = j * kBlockN + r < N;
    const uint32_t aDS = smem_u32(sDS);
    bool ok = !abort_all;
    for (int it = 0; it < nq && ok; ++it) {
      const int st = it & 1, use = it >> 1;
      const int i = i_first + it;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_qfull[st], use & 1));
      if (!ok) break;
      ok = __all_sync(0xffffffffu, mbar_wait(bar_sfull, it & 1));
      if (!ok) break;
      tc_fence_after();
      uint32_t p[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, p[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) reg_fence(p[c]);
      const float* L2 = sLse + st * 128;
      // Keys after the query (diagonal tile only) and padded keys get P = 0;
      // padded queries have -LSE*log2(e) = -inf, so their P is 0 already.
      const int vis_from = (CAUSAL && i == j) ? r : 0;  // query columns c >= vis_from visible
      // Packed FP32 pair fma for the argument (bit-identical to scalar fmas);
      // only the diagonal tile and a tile with padded keys take the masked loop.
      const bool need_mask = (CAUSAL && i == j) || (j + 1) * kBlockN > N;
      const uint64_t c2 = f2_pack(scale_log2, scale_log2);
      auto p_block = [&](auto masked) {
#pragma unroll
        for (int c = 0; c < 128; c += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(L2 + c);
          const uint64_t l2[2] = {f2_pack(l4.x, l4.y), f2_pack(l4.z, l4.w)};
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int cc = c + e;
            float x0, x1;
            f2_unpack(fma2(f2_pack(__uint_as_float(p[cc >> 5][cc & 31]),
                                   __uint_as_float(p[cc >> 5][(cc & 31) + 1])),
                           c2, l2[e >> 1]),
                      x0, x1);
            float p0 = ex2(x0), p1 = ex2(x1);
            if (decltype(masked)::value) {
              if (!key_valid || cc < vis_from) p0 = 0.f;
              if (!key_valid || cc + 1 < vis_from) p1 = 0.f;
            }
            p[cc >> 5][cc & 31] = __float_as_uint(p0);
            p[cc >> 5][(cc & 31) + 1] = __float_as_uint(p1);
          }
        }
      };
      if (need_mask) {
        p_block(std::true_type{});
      } else {
        p_block(std::false_type{});
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(p[c][2 * e]), __uint_as_float(p[c][2 * e + 1]));
        tmem_st16(tS + c * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_pready);

      ok = __all_sync(0xffffffffu, mbar_wait(bar_dpfull, it & 1));
      if (!ok) break;
      // The dS buffer in shared memory is free once the previous dQ MMA is done.
      if (it > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar_dqfull, (it - 1) & 1));
        if (!ok) break;
      }
      tc_fence_after();
      const float* Dl = sDelta + st * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t dp[32];
        tmem_ld32(tDP + c * 32, dp);
        tmem_wait_ld();
        reg_fence(dp);
        uint32_t pk[16];
        // dS = P o (dP - delta), packed: the difference as fma(delta, -1, dP).
        const uint64_t m1 = f2_pack(-1.f, -1.f);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c0 = c * 32 + 2 * e;
          const float2 d2 = *reinterpret_cast<const float2*>(Dl + c0);
          const uint64_t diff = fma2(f2_pack(d2.x, d2.y), m1,
                                     f2_pack(__uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1])));
          float ds0, ds1;
          f2_unpack(mul2(f2_pack(__uint_as_float(p[c][2 * e]), __uint_as_float(p[c][2 * e + 1])), diff),
                    ds0, ds1);
          pk[e] = pack_bf16x2(ds0, ds1);
        }
        tmem_st16(tDP + c * 16, pk);
        // dS^T row r, query columns 32c .. 32c+31 -> MN-major (query-contiguous)
        // 128-byte swizzled layout: chunk (c / 2) of 64 queries, units 4(c%2)..+3.
        const uint32_t base = aDS + (c >> 1) * C::kChunkBytes;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          st_shared_v4(base + sw128_offset(r, (c & 1) * 4 + u), pk[4 * u], pk[4 * u + 1],
                       pk[4 * u + 2], pk[4 * u + 3]);
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_dsready);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_qempty[st]);
    }
    if (!ok) set_fail(ATTN_ERR_TIMEOUT);
    // ---------------------------------------------------------- dV epilogue
    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_dkvdone, 0));
      if (ok) {
        tc_fence_after();
        const uint32_t tDV = tmem + lane_off + C::kColDV;
        const uint32_t aStage = smem_u32(sQ);  // free after the loop
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tDV + c * 32, o);
          tmem_wait_ld();
          reg_fence(o);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1]));
          const uint32_t base = aStage + (c >> 1) * C::kChunkBytes;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            st_shared_v4(base + sw128_offset(r, (c & 1) * 4 + u), pk[4 * u], pk[4 * u + 1],
                         pk[4 * u + 2], pk[4 * u + 3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar_epi_dv);
        if (r == 0) {
          if (mbar_wait(bar_epi_dv, 0)) {
            for (int c = 0; c < C::kChunks; ++c)
              tma_store_3d(&tmDV, sQ + c * C::kChunkBytes, c * 64, j * kBlockN, bh);
            bulk_commit_group();
            bulk_wait_group0();
          } else {
            set_fail(ATTN_ERR_TIMEOUT);
          }
        }
      } else {
        set_fail(ATTN_ERR_TIMEOUT);
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 216;");
    // ------------------------------------------------------------ dQ drain
    const int r = (warp & 3) * 32 + lane;  // query row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tDQ = tmem + lane_off + C::kColDQ;
    bool ok = !abort_all;
    for (int it = 0; it < nq && ok; ++it) {
      const int i = i_first + it;
      ok = __all_sync(0xffffffffu, mbar_wait(bar_dqfull, it & 1));
      if (!ok) break;
      tc_fence_after();
      uint32_t acc[D / 32][32];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(tDQ + c * 32, acc[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) reg_fence(acc[c]);
      tc_fence_before();
      mbar_arrive(bar_dqfree);
      float* dst = dqacc + ((size_t)bh * Npad + (size_t)i * kBlockM + r) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          red_add_v4(dst + c * 32 + e, __uint_as_float(acc[c][e]), __uint_as_float(acc[c][e + 1]),
                     __uint_as_float(acc[c][e + 2]), __uint_as_float(acc[c][e + 3]));
    }
    if (!ok) set_fail(ATTN_ERR_TIMEOUT);
    // ---------------------------------------------------------- dK epilogue
    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_dkvdone, 0));
      if (ok) {
        tc_fence_after();
        const uint32_t tDK = tmem + lane_off + C::kColDK;
        const uint32_t aStage = smem_u32(sDO);  // free after the loop
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tDK + c * 32, o);
          tmem_wait_ld();
          reg_fence(o);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * scale,
                                __uint_as_float(o[2 * e + 1]) * scale);
          const uint32_t base = aStage + (c >> 1) * C::kChunkBytes;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            st_shared_v4(base + sw128_offset(r, (c & 1) * 4 + u), pk[4 * u], pk[4 * u + 1],
                         pk[4 * u + 2], pk[4 * u + 3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar_epi_dk);
        if (r == 0) {
          if (mbar_wait(bar_epi_dk, 0)) {
            for (int c = 0; c < C::kChunks; ++c)
              tma_store_3d(&tmDK, sDO + c * C::kChunkBytes, c * 64, j * kBlockN, bh);
            bulk_commit_group();
            bulk_wait_group0();
          } else {
            set_fail(ATTN_ERR_TIMEOUT);
          }
        }
      } else {
        set_fail(ATTN_ERR_TIMEOUT);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// 2'. main kernel, d = 128: 64-row query tiles, overlapped pipeline
// ---------------------------------------------------------------------------
// Same mathematics as bwd_main_kernel, arranged so that the tensor pipe is
// not left waiting on the P / dS computation or on the dQ drain.  Per
// 64-row query tile i (index it) the MMAs are
//   S^T(it)  = K_j Q_i^T     M=128 N=64 K=128   SS  -> S buffer it%2
//   dP^T(it) = V_j dO_i^T    M=128 N=64 K=128   SS  -> dP region
//   dV      += P^T dO_i      M=128 N=128 K=64   TS  (P^T in the S buffer)
//   dK      += dS^T Q_i      M=128 N=128 K=64   TS  (dS^T in the dP region)
//   dQ^T(it) = K_j^T dS^T    M=128 N=64 K=128   SS  (dS^T from shared memory)
// issued in the order dV(it), dK(it), dP^T(it+1), dQ^T(it), S^T(it+2), so the
// P and dS work of tile it+1 runs while the tensor pipe finishes tile it.
// dQ^T puts head-dim index d on the TMEM lanes: each drain thread owns one d,
// and a warp's 32 reductions into the FP32 accumulator cover 128 contiguous
// bytes of one query row.  Warps 4-11 form two warpgroups that split every
// tile's 64 query columns (P and dS) between them, so each SM sub-partition
// has two warps to overlap the exp and TMEM latency; warps 12-15 drain dQ^T
// into the accumulator, so the reductions' issue stalls stay off the P / dS
// path.
// TMEM (512 columns): dV [0,128), dK [128,256), S buffers [256,320) and
// [320,384), dP [384,448), dQ^T [448,512).  Shared memory: K_j, V_j (32 KB
// each), a 3-stage ring of Q_i / dO_i (16 KB each) with -LSE*log2(e) and delta,
// and two dS^T buffers (16 KB each).  Each barrier that a role waits on is
// either completed once per tile or split per buffer, so no waiter can fall
// two phases behind the barrier it polls.
namespace r64 {

constexpr int kBM = 64;                    // query rows per tile
constexpr int kThreadsR = 512;             // + warps 12-15: dQ drain
constexpr int kRegsWG0 = 96, kRegsCompute = 168, kRegsDrain = 80;  // setmaxnreg split
static_assert(kRegsWG0 + 2 * kRegsCompute + kRegsDrain <= 512, "split exceeds the launch pool");
constexpr int kStages = 3;                 // Q / dO ring depth
constexpr int kKVBytes = 128 * 128 * 2;    // K_j or V_j (128 rows x 128 d)
constexpr int kKVChunk = 128 * 128;        // one 64-column chunk of K_j / V_j
constexpr int kQBytes = kBM * 128 * 2;     // Q_i or dO_i (64 rows x 128 d)
constexpr int kQChunk = kBM * 128;         // one 64-column chunk of Q_i / dO_i
constexpr int kDSBytes = 128 * kBM * 2;    // dS^T: 128 key rows x 64 query cols
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kKVBytes;
constexpr int kOffQ = kOffV + kKVBytes;
constexpr int kOffDO = kOffQ + kStages * kQBytes;
constexpr int kOffDS = kOffDO + kStages * kQBytes;
constexpr int kOffLse = kOffDS + 2 * kDSBytes;
constexpr int kOffDelta = kOffLse + kStages * kBM * 4;
constexpr int kOffBar = kOffDelta + kStages * kBM * 4;
// kv_full, q_full[3], q_empty[3], s_full[2], p_ready[2], dp_full, ds_ready,
// dq_full, dq_free, dq_done[2], dkv_done, mma_final, epi_dv, epi_dk
constexpr int kNumBars = 1 + 3 + 3 + 2 + 2 + 1 + 1 + 1 + 1 + 2 + 1 + 1 + 1 + 1;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;
constexpr uint32_t kColDV = 0, kColDK = 128, kColS = 256, kColDP = 384, kColDQ = 448;
// P^T and dS^T (BF16 pairs) are written by warpgroup h into the first 16 of
// its own 32 FP32 columns [32h, 32h+32), so neither warpgroup overwrites
// values the other has not read yet.  K step kk of the dV / dK products
// (query columns 16kk .. 16kk+15) is then at packed column:
__host__ __device__ constexpr uint32_t packed_col(int kk) { return (kk >> 1) * 32 + (kk & 1) * 8; }

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreadsR, 1)
    bwd_main_d128_kernel(const __grid_constant__ CUtensorMap tmQ,   // box 64 rows
                         const __grid_constant__ CUtensorMap tmK,   // box 128 rows
                         const __grid_constant__ CUtensorMap tmV,   // box 128 rows
                         const __grid_constant__ CUtensorMap tmDO,  // box 64 rows
                         const __grid_constant__ CUtensorMap tmDK,  // box 128 rows
                         const __grid_constant__ CUtensorMap tmDV,  // box 128 rows
                         const float* __restrict__ neg_lse2, const float* __restrict__ delta,
                         float* __restrict__ dqacc, int BH, int N, int Npad, float scale,
                         float scale_log2) {
  constexpr int D = 128;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Key tiles with the most query tiles (causal: small j) first.
  const int j = blockIdx.x / BH;
  const int bh = blockIdx.x % BH;
  const int n_qt = (N + kBM - 1) / kBM;
  const int i_first = CAUSAL ? 2 * j : 0;
  const int nq = max(0, n_qt - i_first);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* bar_kv = bars + 0;
  uint64_t* bar_qfull = bars + 1;    // [3]
  uint64_t* bar_qempty = bars + 4;   // [3]
  uint64_t* bar_sfull = bars + 7;    // [2]
  uint64_t* bar_pready = bars + 9;   // [2]
  uint64_t* bar_dpfull = bars + 11;
  uint64_t* bar_dsready = bars + 12;
  uint64_t* bar_dqfull = bars + 13;
  uint64_t* bar_dqfree = bars + 14;
  uint64_t* bar_dqdone = bars + 15;  // [2]
  uint64_t* bar_dkvdone = bars + 17;
  uint64_t* bar_final = bars + 18;
  uint64_t* bar_epi_dv = bars + 19;
  uint64_t* bar_epi_dk = bars + 20;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    *s_abort = (smem_u32(smem) & 1023u) != 0;
    if (*s_abort) set_fail(ATTN_ERR_INVALID_ARG);
    mbar_init(bar_kv, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_qfull[s], 1);
      mbar_init(&bar_qempty[s], 1 + 8);  // MMA commit + one arrive per compute warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_sfull[b], 1);
      mbar_init(&bar_pready[b], 256);
      mbar_init(&bar_dqdone[b], 1);
    }
    mbar_init(bar_dpfull, 1);
    mbar_init(bar_dsready, 256);
    mbar_init(bar_dqfull, 1);
    mbar_init(bar_dqfree, 128);
    mbar_init(bar_dkvdone, 1);
    mbar_init(bar_final, 1);
    mbar_init(bar_epi_dv, 128);
    mbar_init(bar_epi_dk, 128);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool abort_all = *s_abort != 0 || nq == 0;

  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sDO = smem + kOffDO;
  uint8_t* sDS = smem + kOffDS;
  float* sLse = reinterpret_cast<float*>(smem + kOffLse);
  float* sDelta = reinterpret_cast<float*>(smem + kOffDelta);

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsWG0));
    if (warp == 0 && lane == 0 && !abort_all) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      mbar_arrive_expect_tx(bar_kv, 2 * kKVBytes);
      for (int c = 0; c < 2; ++c) {
        tma_load_3d(sK + c * kKVChunk, &tmK, bar_kv, c * 64, j * kBlockN, bh);
        tma_load_3d(sV + c * kKVChunk, &tmV, bar_kv, c * 64, j * kBlockN, bh);
      }
      bool ok = true;
      int issued = 0;
      for (int it = 0; it < nq; ++it) {
        const int st = it % kStages, use = it / kStages;
        const int i = i_first + it;
        if (use > 0 && !mbar_wait(&bar_qempty[st], (use - 1) & 1)) { ok = false; break; }
        mbar_arrive_expect_tx(&bar_qfull[st], 2 * kQBytes + 2 * kBM * 4);
        for (int c = 0; c < 2; ++c) {
          tma_load_3d(sQ + st * kQBytes + c * kQChunk, &tmQ, &bar_qfull[st], c * 64, i * kBM, bh);
          tma_load_3d(sDO + st * kQBytes + c * kQChunk, &tmDO, &bar_qfull[st], c * 64, i * kBM,
                      bh);
        }
        const size_t prow = (size_t)bh * Npad + (size_t)i * kBM;
        bulk_load(sLse + st * kBM, neg_lse2 + prow, kBM * 4, &bar_qfull[st]);
        bulk_load(sDelta + st * kBM, delta + prow, kBM * 4, &bar_qfull[st]);
        issued = it + 1;
      }
      if (!ok) set_fail(ATTN_ERR_TIMEOUT);
      // Do not leave while copies into this CTA's shared memory are in flight.
      mbar_wait(bar_kv, 0);
      for (int it = max(0, issued - kStages); it < issued; ++it)
        mbar_wait(&bar_qfull[it % kStages], (it / kStages) & 1);
    } else if (warp == 1 && !abort_all) {
      // ------------------------------------------------------------ MMA issuer
      // Whole warp, warp-uniform operands; elect.sync picks the issuing lane.
      constexpr uint32_t idesc_s = idesc_bf16(128, kBM, false, false);  // K-major A and B
      constexpr uint32_t idesc_acc = idesc_bf16(128, D, false, true);   // TMEM A, MN-major B
      constexpr uint32_t idesc_dq = idesc_bf16(128, kBM, true, true);   // MN-major A and B
      const uint64_t kK = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t kV = sdesc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t kQ = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t kDO = sdesc_sw128(smem_u32(sDO), 16, 1024);
      const uint64_t mQ = sdesc_sw128(smem_u32(sQ), kQChunk, 1024);
      const uint64_t mDO = sdesc_sw128(smem_u32(sDO), kQChunk, 1024);
      const uint64_t mK = sdesc_sw128(smem_u32(sK), kKVChunk, 1024);
      const uint64_t mDS = sdesc_sw128(smem_u32(sDS), kDSBytes, 1024);
      // S^T or dP^T (into column d_col) = X_j Y_i^T over the 128 head dims.
      auto issue_xy = [&](uint32_t d_col, uint64_t dX, uint64_t dY, uint32_t y_off) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t cx = (kk >> 2) * kKVChunk + (kk & 3) * 32;
          const uint32_t cy = (kk >> 2) * kQChunk + (kk & 3) * 32;
          mma_ss_elect(tmem + d_col, sdesc_add(dX, cx), sdesc_add(dY, y_off + cy), idesc_s,
                       kk > 0 ? 1u : 0u);
        }
      };
      bool ok = warp_wait(bar_kv, 0);
      // Prologue: S^T(0), dP^T(0), S^T(1).
      if (ok) ok = warp_wait(&bar_qfull[0], 0);
      if (ok) {
        tc_fence_after();
        issue_xy(kColS, kK, kQ, 0);
        mma_commit_elect(&bar_sfull[0]);
        issue_xy(kColDP, kV, kDO, 0);
        mma_commit_elect(bar_dpfull);
      }
      if (ok && nq > 1) {
        ok = warp_wait(&bar_qfull[1], 0);
        if (ok) {
          tc_fence_after();
          issue_xy(kColS + kBM, kK, kQ, kQBytes);
          mma_commit_elect(&bar_sfull[1]);
        }
      }
      for (int it = 0; it < nq && ok; ++it) {
        const int st = it % kStages, b = it & 1;
        const uint32_t so = st * kQBytes;
        // dV += P^T dO_i
        if (!warp_wait(&bar_pready[b], (it >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk)
          mma_ts_elect(tmem + kColDV, tmem + kColS + b * kBM + packed_col(kk),
                       sdesc_add(mDO, so + kk * 2048), idesc_acc, (it > 0 || kk > 0) ? 1u : 0u);
        // dK += dS^T Q_i
        if (!warp_wait(bar_dsready, it & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk)
          mma_ts_elect(tmem + kColDK, tmem + kColDP + packed_col(kk), sdesc_add(mQ, so + kk * 2048),
                       idesc_acc, (it > 0 || kk > 0) ? 1u : 0u);
        mma_commit_elect(&bar_qempty[st]);
        // dP^T(it+1): the dP region is free (dK(it) above read dS^T from it).
        if (it + 1 < nq) {
          issue_xy(kColDP, kV, kDO, ((it + 1) % kStages) * kQBytes);
          mma_commit_elect(bar_dpfull);
        }
        // dQ^T(it) = K_j^T dS^T(it)
        if (it > 0 && !warp_wait(bar_dqfree, (it - 1) & 1)) { ok = false; break; }
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          mma_ss_elect(tmem + kColDQ, sdesc_add(mK, kk * 2048),
                       sdesc_add(mDS, b * kDSBytes + kk * 2048), idesc_dq, kk > 0 ? 1u : 0u);
        mma_commit_elect(bar_dqfull);
        mma_commit_elect(&bar_dqdone[b]);
        // S^T(it+2) into buffer b (P^T(it) was read by dV(it) above).
        if (it + 2 < nq) {
          const int st2 = (it + 2) % kStages;
          if (!warp_wait(&bar_qfull[st2], ((it + 2) / kStages) & 1)) { ok = false; break; }
          tc_fence_after();
          issue_xy(kColS + b * kBM, kK, kQ, st2 * kQBytes);
          mma_commit_elect(&bar_sfull[b]);
        }
      }
      if (ok) mma_commit_elect(bar_dkvdone);
      else if (lane == 0) set_fail(ATTN_ERR_TIMEOUT);
      mma_commit_elect(bar_final);
      mbar_wait(bar_final, 0);
    }
    __syncwarp();
  } else if (warp >= 12) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsDrain));
    // ------------------------------------------------------------ dQ drain
    // dQ^T(it), all 64 query columns: lane r adds head dim r of each query row;
    // a warp's 32 reductions of one column cover 128 contiguous bytes.
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tDQ = tmem + lane_off + kColDQ;
    bool ok = !abort_all;
    for (int itd = 0; itd < nq && ok; ++itd) {
      ok = warp_wait(bar_dqfull, itd & 1);
      if (!ok) break;
      tc_fence_after();
      uint32_t acc[2][32];
      tmem_ld32(tDQ, acc[0]);
      tmem_ld32(tDQ + 32, acc[1]);
      tmem_wait_ld();
      reg_fence(acc[0]);
      reg_fence(acc[1]);
      tc_fence_before();
      mbar_arrive(bar_dqfree);
      float* dst = dqacc + ((size_t)bh * Npad + (size_t)(i_first + itd) * kBM) * D + r;
#pragma unroll
      for (int c = 0; c < 64; ++c)
        asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dst + (size_t)c * D),
                     "f"(__uint_as_float(acc[c >> 5][c & 31]))
                     : "memory");
    }
    if (!ok) set_fail(ATTN_ERR_TIMEOUT);
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsCompute));
    // ------------------------------------------- P and dS (two warpgroups)
    // Warpgroup h (warps 4-7: h = 0, warps 8-11: h = 1) owns query columns
    // [32h, 32h+32) of every 64-row tile: it computes those columns of P^T
    // and dS^T (thread = key row = TMEM lane).
    const int h = (warp - 4) >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tDP = tmem + lane_off + kColDP;
    const int kv = j * kBlockN + r;
    const bool key_valid = kv < N;
    const uint32_t dsBase0 = smem_u32(sDS);
    const uint64_t c2 = f2_pack(scale_log2, scale_log2);
    bool ok = !abort_all;
    for (int it = 0; it < nq && ok; ++it) {
      const int st = it % kStages, b = it & 1;
      const int i = i_first + it;
      const uint32_t tS = tmem + lane_off + kColS + b * kBM;
      ok = warp_wait(&bar_qfull[st], (it / kStages) & 1);
      if (!ok) break;
      ok = warp_wait(&bar_sfull[b], (it >> 1) & 1);
      if (!ok) break;
      tc_fence_after();
      uint32_t p[32];
      tmem_ld32(tS + h * 32, p);
      tmem_wait_ld();
      reg_fence(p);
      const float* L2 = sLse + st * kBM + h * 32;
      // P = exp2(c s - LSE log2 e), the argument of each column pair in one
      // packed FP32 fma (bit-identical to two scalar fmas).  Local column c is
      // query i*64 + 32h + c.  Causal: it sees this key only when c >= vis_to;
      // padded keys see nothing.  Only tiles that cross the diagonal or hold
      // padded keys take the masked loop.  Padded queries have
      // -LSE log2(e) = -inf, so their P is 0 already.
      const int vis_to = CAUSAL ? kv - i * kBM - h * 32 : 0;
      const bool need_mask =
          (CAUSAL && i * kBM < (j + 1) * kBlockN) || (j + 1) * kBlockN > N;
      auto p_block = [&](auto masked) {
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(L2 + c);
          const uint64_t l2[2] = {f2_pack(l4.x, l4.y), f2_pack(l4.z, l4.w)};
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int cc = c + e;
            float x0, x1;
            f2_unpack(fma2(f2_pack(__uint_as_float(p[cc]), __uint_as_float(p[cc + 1])), c2,
                           l2[e >> 1]),
                      x0, x1);
            float p0 = ex2(x0), p1 = ex2(x1);
            if (decltype(masked)::value) {
              if (!key_valid || cc < vis_to) p0 = 0.f;
              if (!key_valid || cc + 1 < vis_to) p1 = 0.f;
            }
            p[cc] = __float_as_uint(p0);
            p[cc + 1] = __float_as_uint(p1);
          }
        }
      };
      if (need_mask) {
        p_block(std::true_type{});
      } else {
        p_block(std::false_type{});
      }
      {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(p[2 * e]), __uint_as_float(p[2 * e + 1]));
        tmem_st16(tS + h * 32, pk);  // inside this warpgroup's own S columns
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar_pready[b]);

      ok = warp_wait(bar_dpfull, it & 1);
      if (!ok) break;
      // dS^T buffer b is free once dQ^T(it-2), which read it, has completed.
      if (it >= 2) {
        ok = warp_wait(&bar_dqdone[b], ((it >> 1) - 1) & 1);
        if (!ok) break;
      }
      tc_fence_after();
      const float* Dl = sDelta + st * kBM + h * 32;
      {
        uint32_t dp[32];
        tmem_ld32(tDP + h * 32, dp);
        tmem_wait_ld();
        reg_fence(dp);
        uint32_t pk[16];
        // dS = P o (dP - delta): dP - delta as fma(delta, -1, dP) (exact
        // negation, one rounding: the subtraction), then the product, both packed.
        const uint64_t m1 = f2_pack(-1.f, -1.f);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 d2 = *reinterpret_cast<const float2*>(Dl + 2 * e);
          const uint64_t diff = fma2(f2_pack(d2.x, d2.y), m1,
                                     f2_pack(__uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1])));
          float ds0, ds1;
          f2_unpack(mul2(f2_pack(__uint_as_float(p[2 * e]), __uint_as_float(p[2 * e + 1])), diff),
                    ds0, ds1);
          pk[e] = pack_bf16x2(ds0, ds1);
        }
        tmem_st16(tDP + h * 32, pk);  // inside this warpgroup's own dP columns
        // dS^T row r, query columns 32h .. 32h+31: 16-byte units 4h .. 4h+3 of
        // the row's 128-byte swizzled line (MN-major B operand of dQ^T).
        const uint32_t dsBase = dsBase0 + b * kDSBytes;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          st_shared_v4(dsBase + sw128_offset(r, h * 4 + u), pk[4 * u], pk[4 * u + 1],
                       pk[4 * u + 2], pk[4 * u + 3]);
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_dsready);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_qempty[st]);
    }
    if (!ok) set_fail(ATTN_ERR_TIMEOUT);
    // ------------------------- epilogue: h = 0 stores dV, h = 1 stores scale*dK
    if (ok && !abort_all) {
      ok = warp_wait(bar_dkvdone, 0);
      if (ok) {
        tc_fence_after();
        const uint32_t tAcc = tmem + lane_off + (h == 0 ? kColDV : kColDK);
        const float mul = h == 0 ? 1.f : scale;
        uint8_t* stage = h == 0 ? sQ : sDO;  // the Q / dO rings are free after the loop
        const uint32_t aStage = smem_u32(stage);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tAcc + c * 32, o);
          tmem_wait_ld();
          reg_fence(o);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * mul, __uint_as_float(o[2 * e + 1]) * mul);
          const uint32_t base = aStage + (c >> 1) * kKVChunk;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            st_shared_v4(base + sw128_offset(r, (c & 1) * 4 + u), pk[4 * u], pk[4 * u + 1],
                         pk[4 * u + 2], pk[4 * u + 3]);
        }
        fence_proxy_async_smem();
        uint64_t* bar_epi = h == 0 ? bar_epi_dv : bar_epi_dk;
        mbar_arrive(bar_epi);
        if (r == 0) {
          if (mbar_wait(bar_epi, 0)) {
            const CUtensorMap* map = h == 0 ? &tmDV : &tmDK;
            for (int c = 0; c < 2; ++c)
              tma_store_3d(map, stage + c * kKVChunk, c * 64, j * kBlockN, bh);
            bulk_commit_group();
            bulk_wait_group0();
          } else {
            set_fail(ATTN_ERR_TIMEOUT);
          }
        }
      } else {
        set_fail(ATTN_ERR_TIMEOUT);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace r64

template <int D>
cudaError_t preprocess_impl(const Problem& p, const void* o, const void* dout, const float* lse,
                            const BwdWorkspace& ws, cudaStream_t stream) {
  constexpr int kRows = 256 / (D / 8);
  const int Npad = n_pad(p.N);
  const int per_head = ceil_div(Npad, kRows);
  const unsigned blocks = (unsigned)per_head * (unsigned)(p.B * p.H);
  bwd_preprocess_kernel<D><<<blocks, 256, 0, stream>>>(
      static_cast<const uint4*>(o), static_cast<const uint4*>(dout), lse, ws.neg_lse2, ws.delta,
      reinterpret_cast<float4*>(ws.dqacc), p.N, Npad, per_head);
  return cudaGetLastError();
}

template <int D>
cudaError_t dq_convert_impl(const Problem& p, const BwdWorkspace& ws, void* dq,
                            cudaStream_t stream) {
  const long long units = (long long)p.B * p.H * p.N * (D / 8);
  const int blocks = (int)((units + 255) / 256);
  bwd_dq_convert_kernel<D><<<blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(ws.dqacc),
                                                       static_cast<uint4*>(dq), p.N, n_pad(p.N),
                                                       p.scale, (int)units);
  return cudaGetLastError();
}

template <int D, bool CAUSAL>
cudaError_t main_impl(const Problem& p, const CUtensorMap* maps, const BwdWorkspace& ws,
                      cudaStream_t stream) {
  using C = BwdCfg<D>;
  auto kernel = bwd_main_kernel<D, CAUSAL>;
  cudaError_t err =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (err != cudaSuccess) return err;
  const int BH = p.B * p.H;
  const int Npad = n_pad(p.N);
  const int n_kt = Npad / kBlockN;
  kernel<<<dim3(BH * n_kt), dim3(kThreads), C::kSmemBytes, stream>>>(
      maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], ws.neg_lse2, ws.delta, ws.dqacc, BH, p.N,
      Npad, p.scale, p.scale * 1.4426950408889634f);
  return cudaGetLastError();
}

template <bool CAUSAL>
cudaError_t main_d128_impl(const Problem& p, const CUtensorMap* maps, const BwdWorkspace& ws,
                           cudaStream_t stream) {
  auto kernel = r64::bwd_main_d128_kernel<CAUSAL>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         r64::kSmemBytes);
  if (err != cudaSuccess) return err;
  const int BH = p.B * p.H;
  const int Npad = n_pad(p.N);
  const int n_kt = Npad / kBlockN;
  kernel<<<dim3(BH * n_kt), dim3(r64::kThreadsR), r64::kSmemBytes, stream>>>(
      maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], ws.neg_lse2, ws.delta, ws.dqacc, BH, p.N,
      Npad, p.scale, p.scale * 1.4426950408889634f);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_preprocess_bf16(const Problem& p, const void* o, const void* dout,
                                       const float* lse, const BwdWorkspace& ws,
                                       cudaStream_t stream) {
  return p.d == 128 ? preprocess_impl<128>(p, o, dout, lse, ws, stream)
                    : preprocess_impl<64>(p, o, dout, lse, ws, stream);
}

cudaError_t launch_bwd_dq_convert_bf16(const Problem& p, const BwdWorkspace& ws, void* dq,
                                       cudaStream_t stream) {
  return p.d == 128 ? dq_convert_impl<128>(p, ws, dq, stream)
                    : dq_convert_impl<64>(p, ws, dq, stream);
}

cudaError_t launch_bwd_main_bf16(const Problem& p, const void* q, const void* k, const void* v,
                                 const void* dout, void* dk, void* dv, const BwdWorkspace& ws,
                                 cudaStream_t stream) {
  const int BH = p.B * p.H;
  CUtensorMap maps[6];
  const void* ptrs[6] = {q, k, v, dout, dk, dv};
  // d = 128 streams 64-row query tiles (Q and dO maps with 64-row boxes).
  const int q_rows = p.d == 128 ? r64::kBM : kBlockM;
  const int box_rows[6] = {q_rows, kBlockN, kBlockN, q_rows, kBlockN, kBlockN};
  for (int i = 0; i < 6; ++i)
    if (!make_tmap_bhnd(&maps[i], ptrs[i], BH, p.N, p.d, box_rows[i]))
      return cudaErrorInvalidValue;
  if (p.d == 128)
    return p.causal ? main_d128_impl<true>(p, maps, ws, stream)
                    : main_d128_impl<false>(p, maps, ws, stream);
  return p.causal ? main_impl<64, true>(p, maps, ws, stream)
                  : main_impl<64, false>(p, maps, ws, stream);
}

cudaError_t read_and_clear_status_bwd(unsigned int* out, cudaStream_t stream) {
  static const unsigned int zero = 0;
  cudaError_t err = cudaMemcpyFromSymbolAsync(out, g_status_bwd, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
  if (err != cudaSuccess) return err;
  err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return err;
  err = cudaMemcpyToSymbolAsync(g_status_bwd, &zero, sizeof(unsigned int), 0,
                                cudaMemcpyHostToDevice, stream);
  if (err != cudaSuccess) return err;
  return cudaStreamSynchronize(stream);
}

}  // namespace attn
