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
//                   shared memory; the CTA walks 64-row query tiles i (causal:
//                   from the tile holding query j * 128 on) with Q_i, dO_i,
//                   LSE_i, delta_i streamed by TMA.  Five tcgen05 MMAs per
//                   tile (described at r64 below); dQ_i is added into the FP32
//                   accumulator with red.global.add.f32.  d = 128 launches
//                   one CTA per (b, h, j); d = 64 runs the same pipeline in
//                   persistent CTAs (bwd_main_persistent_kernel), one per SM,
//                   each walking a list of (b, h, j) items.
//   3. dq_convert   dQ = bf16(scale * accumulator).  Memory-bound.
#include <math.h>

#include <algorithm>

#include <type_traits>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {

static __device__ unsigned int g_status_bwd;

#ifdef ATTN_TEST_HOOKS
// Test instrumentation, compiled only into the separate test build of the
// library (ATTN_TEST_HOOKS), never into libattn.so: when g_hook_stall_bwd is
// set, the first P/dS warpgroup of CTA 0 of the backward main kernel first
// waits on a barrier that nothing ever arrives at, so the wait runs out
// (after the test build's short limit) and the kernel takes its failure path.
static __device__ int g_hook_stall_bwd;
#endif

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
  griddep_launch_dependents();
  griddep_wait();  // O and LSE come from the forward just before
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
  griddep_launch_dependents();
  griddep_wait();  // the accumulator is complete once the main kernel is
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
// 2. main kernel: 64-row query tiles, overlapped pipeline
// ---------------------------------------------------------------------------
// Arranged so that the tensor pipe is not left waiting on the P / dS
// computation or on the dQ drain.  Per 64-row query tile i (index it) the
// MMAs are
//   S^T(it)  = K_j Q_i^T     M=128 N=64 K=d     SS  -> S buffer it%2
//   dP^T(it) = V_j dO_i^T    M=128 N=64 K=d     SS  -> dP region
//   dV      += P^T dO_i      M=128 N=d  K=64    TS  (P^T in the S buffer)
//   dK      += dS^T Q_i      M=128 N=d  K=64    TS  (dS^T in the dP region)
//   dQ^T(it) = K_j^T dS^T    M=d   N=64 K=128   SS  (dS^T from shared memory)
// issued in the order dV(it), dK(it), dP^T(it+1), S^T(it+2), dQ^T(it), so the
// P and dS work of tile it+1 runs while the tensor pipe finishes tile it.
// dQ^T puts head-dim index d on the TMEM lanes: each drain thread owns one d,
// and a warp's reductions into the FP32 accumulator cover contiguous bytes of
// one query row (at d = 64 the M = 64 accumulator fills lanes 0-15 of each
// warp's quarter of TMEM).  Warps 4-11 form two warpgroups that split every
// tile's 64 query columns (P and dS) between them, so each SM sub-partition
// has two warps to overlap the exp and TMEM latency; warps 12-15 drain dQ^T
// into the accumulator, so the reductions' issue stalls stay off the P / dS
// path.
// TMEM (512 columns allocated): dV [0,d), dK [d,2d), S buffers [2d,2d+64) and
// [2d+64,2d+128), dP [2d+128,2d+192), dQ^T [2d+192,2d+256).  Shared memory:
// K_j, V_j (128 x d each), a 3-stage ring of Q_i / dO_i (64 x d each) with
// -LSE*log2(e) and delta, and two dS^T buffers (16 KB each).  Each barrier
// that a role waits on is either completed once per tile or split per buffer,
// so no waiter can fall two phases behind the barrier it polls.
namespace r64 {

constexpr int kBM = 64;                    // query rows per tile
constexpr int kThreadsR = 512;             // + warps 12-15: dQ drain
constexpr int kRegsWG0 = 96, kRegsCompute = 168, kRegsDrain = 80;  // setmaxnreg split
static_assert(kRegsWG0 + 2 * kRegsCompute + kRegsDrain <= 512, "split exceeds the launch pool");
// A 512-thread launch gives 128 registers per thread: setmaxnreg.dec must ask
// for fewer, setmaxnreg.inc for more.
static_assert(kRegsWG0 <= 128 && kRegsDrain <= 128 && kRegsCompute >= 128, "setmaxnreg directions");
constexpr int kStages = 3;                 // Q / dO ring depth
constexpr int kKVChunk = 128 * 128;        // one 64-column chunk of K_j / V_j (128 rows)
constexpr int kQChunk = kBM * 128;         // one 64-column chunk of Q_i / dO_i (64 rows)
constexpr int kDSBytes = 128 * kBM * 2;    // dS^T: 128 key rows x 64 query cols
// kv_full, q_full[3], q_empty[3], s_full[2], p_ready[2], dp_full, ds_ready,
// dq_full, dq_free, dq_done[2], dkv_done, mma_final, epi_dv, epi_dk
constexpr int kNumBars = 1 + 3 + 3 + 2 + 2 + 1 + 1 + 1 + 1 + 2 + 1 + 1 + 1 + 1;

template <int D>
struct Cfg {
  static constexpr int kChunks = D / 64;          // 64-column (128-byte) chunks per row
  static constexpr int kKVBytes = 128 * D * 2;    // K_j or V_j (128 rows x d)
  static constexpr int kQBytes = kBM * D * 2;     // Q_i or dO_i (64 rows x d)
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKVBytes;
  static constexpr int kOffQ = kOffV + kKVBytes;
  static constexpr int kOffDO = kOffQ + kStages * kQBytes;
  static constexpr int kOffDS = kOffDO + kStages * kQBytes;
  static constexpr int kOffLse = kOffDS + 2 * kDSBytes;
  static constexpr int kOffDelta = kOffLse + kStages * kBM * 4;
  static constexpr int kOffBar = kOffDelta + kStages * kBM * 4;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;
  // TMEM columns: dV, dK (d each), two S^T buffers (64 each), dP^T (64), dQ^T (64).
  static constexpr uint32_t kColDV = 0, kColDK = D, kColS = 2 * D, kColDP = 2 * D + 128,
                            kColDQ = 2 * D + 192;
  static_assert(kColDQ + kBM <= 512, "TMEM columns");
  // The epilogue stages dV in the Q ring and scale * dK in the dO ring.
  static_assert(kStages * kQBytes >= kKVBytes, "epilogue staging");
};
// P^T and dS^T (BF16 pairs) are written by warpgroup h into the first 16 of
// its own 32 FP32 columns [32h, 32h+32), so neither warpgroup overwrites
// values the other has not read yet.  K step kk of the dV / dK products
// (query columns 16kk .. 16kk+15) is then at packed column:
__host__ __device__ constexpr uint32_t packed_col(int kk) { return (kk >> 1) * 32 + (kk & 1) * 8; }

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreadsR, 1)
    bwd_main_r64_kernel(const __grid_constant__ CUtensorMap tmQ,   // box 64 rows
                         const __grid_constant__ CUtensorMap tmK,   // box 128 rows
                         const __grid_constant__ CUtensorMap tmV,   // box 128 rows
                         const __grid_constant__ CUtensorMap tmDO,  // box 64 rows
                         const __grid_constant__ CUtensorMap tmDK,  // box 128 rows
                         const __grid_constant__ CUtensorMap tmDV,  // box 128 rows
                         const float* __restrict__ neg_lse2, const float* __restrict__ delta,
                         float* __restrict__ dqacc, int BH, int N, int Npad, int heads_per_group,
                         float scale, float scale_log2) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // CTA order: groups of heads_per_group heads; within a group, key tiles
  // with the most query tiles (causal: small j) first, then heads.
  const int n_kt = Npad / kBlockN;
  const int group = blockIdx.x / (heads_per_group * n_kt);
  const int in_group = blockIdx.x - group * heads_per_group * n_kt;
  const int g0 = group * heads_per_group;
  const int g_size = min(heads_per_group, BH - g0);
  const int j = in_group / g_size;
  const int bh = g0 + in_group % g_size;
  const int n_qt = (N + kBM - 1) / kBM;
  const int i_first = CAUSAL ? 2 * j : 0;
  const int nq = max(0, n_qt - i_first);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
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

  // The next kernel in the stream may be scheduled once every CTA is running.
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    *s_abort = (smem_u32(smem) & 1023u) != 0;
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
#ifdef ATTN_TEST_HOOKS
    mbar_init(reinterpret_cast<uint64_t*>(tmem_slot + 2), 1);  // nothing arrives here
#endif
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
  // Set-up above touches no global memory; from here on the preprocess
  // kernel's results must be complete and visible.
  griddep_wait();
  if (threadIdx.x == 0 && *s_abort != 0) set_fail(ATTN_ERR_INVALID_ARG);

  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sDO = smem + C::kOffDO;
  uint8_t* sDS = smem + C::kOffDS;
  float* sLse = reinterpret_cast<float*>(smem + C::kOffLse);
  float* sDelta = reinterpret_cast<float*>(smem + C::kOffDelta);

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsWG0));
    if (warp == 0 && lane == 0 && !abort_all) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      mbar_arrive_expect_tx(bar_kv, 2 * C::kKVBytes);
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_3d(sK + c * kKVChunk, &tmK, bar_kv, c * 64, j * kBlockN, bh);
        tma_load_3d(sV + c * kKVChunk, &tmV, bar_kv, c * 64, j * kBlockN, bh);
      }
      bool ok = true;
      int issued = 0;
      for (int it = 0; it < nq; ++it) {
        const int st = it % kStages, use = it / kStages;
        const int i = i_first + it;
        if (use > 0 && !mbar_wait(&bar_qempty[st], (use - 1) & 1)) { ok = false; break; }
        mbar_arrive_expect_tx(&bar_qfull[st], 2 * C::kQBytes + 2 * kBM * 4);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(sQ + st * C::kQBytes + c * kQChunk, &tmQ, &bar_qfull[st], c * 64, i * kBM,
                      bh);
          tma_load_3d(sDO + st * C::kQBytes + c * kQChunk, &tmDO, &bar_qfull[st], c * 64, i * kBM,
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
      constexpr uint32_t idesc_dq = idesc_bf16(D, kBM, true, true);     // MN-major A and B
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
        issue_xy(C::kColS, kK, kQ, 0);
        mma_commit_elect(&bar_sfull[0]);
        issue_xy(C::kColDP, kV, kDO, 0);
        mma_commit_elect(bar_dpfull);
      }
      if (ok && nq > 1) {
        ok = warp_wait(&bar_qfull[1], 0);
        if (ok) {
          tc_fence_after();
          issue_xy(C::kColS + kBM, kK, kQ, C::kQBytes);
          mma_commit_elect(&bar_sfull[1]);
        }
      }
      for (int it = 0; it < nq && ok; ++it) {
        const int st = it % kStages, b = it & 1;
        const uint32_t so = st * C::kQBytes;
        // dV += P^T dO_i
        if (!warp_wait(&bar_pready[b], (it >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk)
          mma_ts_elect(tmem + C::kColDV, tmem + C::kColS + b * kBM + packed_col(kk),
                       sdesc_add(mDO, so + kk * 2048), idesc_acc, (it > 0 || kk > 0) ? 1u : 0u);
        // dK += dS^T Q_i
        if (!warp_wait(bar_dsready, it & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk)
          mma_ts_elect(tmem + C::kColDK, tmem + C::kColDP + packed_col(kk), sdesc_add(mQ, so + kk * 2048),
                       idesc_acc, (it > 0 || kk > 0) ? 1u : 0u);
        mma_commit_elect(&bar_qempty[st]);
        // dP^T(it+1): the dP region is free (dK(it) above read dS^T from it).
        if (it + 1 < nq) {
          issue_xy(C::kColDP, kV, kDO, ((it + 1) % kStages) * C::kQBytes);
          mma_commit_elect(bar_dpfull);
        }
        // S^T(it+2) into buffer b (P^T(it) was read by dV(it) above), ahead of
        // dQ^T(it), which no compute warp waits for.
        if (it + 2 < nq) {
          const int st2 = (it + 2) % kStages;
          if (!warp_wait(&bar_qfull[st2], ((it + 2) / kStages) & 1)) { ok = false; break; }
          tc_fence_after();
          issue_xy(C::kColS + b * kBM, kK, kQ, st2 * C::kQBytes);
          mma_commit_elect(&bar_sfull[b]);
        }
        // dQ^T(it) = K_j^T dS^T(it)
        if (it > 0 && !warp_wait(bar_dqfree, (it - 1) & 1)) { ok = false; break; }
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          mma_ss_elect(tmem + C::kColDQ, sdesc_add(mK, kk * 2048),
                       sdesc_add(mDS, b * kDSBytes + kk * 2048), idesc_dq, kk > 0 ? 1u : 0u);
        mma_commit_elect(bar_dqfull);
        mma_commit_elect(&bar_dqdone[b]);
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
    // dQ^T(it), all 64 query columns: each thread adds one head dim of every
    // query row; a warp's reductions of one column cover contiguous bytes.
    // d = 128 (M = 128): head dim m is TMEM lane m, 32 per warp.  d = 64
    // (M = 64): head dim m is lane (m / 16) * 32 + m % 16, so lanes 0-15 of
    // each warp hold 16 head dims and lanes 16-31 hold nothing of dQ^T.
    const int dim = D == 128 ? (warp & 3) * 32 + lane : (warp & 3) * 16 + (lane & 15);
    const bool holds_dim = D == 128 || lane < 16;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tDQ = tmem + lane_off + C::kColDQ;
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
      float* dst = dqacc + ((size_t)bh * Npad + (size_t)(i_first + itd) * kBM) * D + dim;
      if (holds_dim) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dst + (size_t)c * D),
                       "f"(__uint_as_float(acc[c >> 5][c & 31]))
                       : "memory");
      }
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
    const uint32_t tDP = tmem + lane_off + C::kColDP;
    const int kv = j * kBlockN + r;
    const bool key_valid = kv < N;
    const uint32_t dsBase0 = smem_u32(sDS);
    const uint64_t c2 = f2_pack(scale_log2, scale_log2);
    bool ok = !abort_all;
#ifdef ATTN_TEST_HOOKS
    if (ok && g_hook_stall_bwd && blockIdx.x == 0 && h == 0)
      ok = warp_wait(reinterpret_cast<uint64_t*>(tmem_slot + 2), 0);
#endif
    for (int it = 0; it < nq && ok; ++it) {
      const int st = it % kStages, b = it & 1;
      const int i = i_first + it;
      const uint32_t tS = tmem + lane_off + C::kColS + b * kBM;
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
        const uint32_t tAcc = tmem + lane_off + (h == 0 ? C::kColDV : C::kColDK);
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
            for (int c = 0; c < C::kChunks; ++c)
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


// ---------------------------------------------------------------------------
// 2'. main kernel, persistent variant (used for d = 64)
// ---------------------------------------------------------------------------
// The five products of the kernel above, in CTAs that stay resident: each CTA
// walks a static list of (b, h, j) items (heaviest first, dealt in snake
// order), with the barrier phases counted across items.  At d = 64 the
// products of a 64-row tile take ~900 cycles while the P and dS work of the
// compute warps takes longer, so this variant spends the TMEM and shared
// memory that d = 64 leaves free on taking waits off the compute warps' chain:
//   - dP^T is double-buffered and issued two tiles ahead (with S^T), so the
//     dS of a tile never waits for the dK product of the previous tile;
//   - dQ^T is double-buffered, so the dQ^T product never waits for the drain
//     warps to have read the previous one;
//   - K_j and V_j are double-buffered, so the next item's K and V load while
//     the current item runs, and its first products follow the current
//     item's last ones without a load in between.
// Per 64-row tile T (b = T % 2) the MMA warp issues dV(T), dK(T), S^T(T+2) and
// dP^T(T+2) into S and dP buffers b, then dQ^T(T) into dQ buffer b.  After an
// item the drain warps stage dV and scale * dK, and warp 3 stores them with TMA.
// dV and dK are read out of TMEM by the drain warps, so the compute warps go
// straight on to the next item's first P.  Measured on the gpt2 workload and
// not kept: a five-tile Q / dO ring (2.5% slower), issuing dV(T) together with
// dK(T) (K steps alternating between the two accumulators: 5% slower, as dV
// then waits for dS), and dQ^T(T) interleaved with S^T(T+2) and dP^T(T+2) (13%
// slower: the compute warps, not the tensor pipe, set the pace, and S^T(T+2)
// then completes later).
// ds_ready is split per buffer like p_ready: with dP^T issued two tiles ahead,
// the compute warps can finish dS(T+1) before the MMA warp has seen dS(T), so
// a single barrier could complete twice under a waiter.
// kv_full[2], kv_free[2], q_full[5], q_empty[5], s_full[2], p_ready[2],
// dp_full[2], ds_ready[2], dq_full[2], dq_free[2], dq_done[2], item_done,
// acc_free, mma_final, epi_full[2], epi_free[2]
constexpr int kStagesP = 3;
constexpr int kNumBarsP = 2 + 2 + 3 + 3 + 2 + 2 + 2 + 2 + 2 + 2 + 2 + 1 + 1 + 1 + 2 + 2;
template <int D>
struct PCfg {
  static_assert(D == 64, "the persistent variant is laid out for d = 64");
  static constexpr int kKVBytes = 128 * D * 2;    // K_j or V_j (128 rows x d), one chunk
  static constexpr int kQBytes = kBM * D * 2;     // Q_i or dO_i (64 rows x d)
  static constexpr int kOffK = 0;                 // two K slots
  static constexpr int kOffV = kOffK + 2 * kKVBytes;  // two V slots
  static constexpr int kOffQ = kOffV + 2 * kKVBytes;
  static constexpr int kOffDO = kOffQ + kStagesP * kQBytes;
  static constexpr int kOffDS = kOffDO + kStagesP * kQBytes;
  static constexpr int kOffStage = kOffDS + 2 * kDSBytes;
  static constexpr int kOffLse = kOffStage + 2 * kKVChunk;
  static constexpr int kOffDelta = kOffLse + kStagesP * kBM * 4;
  static constexpr int kOffBar = kOffDelta + kStagesP * kBM * 4;
  static constexpr int kSmemBytes = kOffBar + kNumBarsP * 8 + 16;
  // TMEM: dV, dK (64 each), S^T, dP^T and dQ^T double-buffered (64 each).
  static constexpr uint32_t kColDV = 0, kColDK = 64, kColS = 128, kColDP = 256, kColDQ = 384;
  static_assert(kColDQ + 2 * kBM <= 512, "TMEM columns");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

// Work item L of the main kernel: head bh, key tile j, and its query tiles.
// Items are numbered by groups of hpg heads; within a group, key tiles with
// the most query tiles (causal: small j) first, then heads.
struct BwdItem {
  int bh, j, i_first, nq;
};
__device__ __forceinline__ BwdItem bwd_item(int L, int BH, int n_kt, int n_qt, int hpg,
                                            bool causal) {
  const int group = L / (hpg * n_kt);
  const int in_group = L - group * hpg * n_kt;
  const int g0 = group * hpg;
  const int g_size = min(hpg, BH - g0);
  BwdItem it;
  it.j = in_group / g_size;
  it.bh = g0 + in_group % g_size;
  it.i_first = causal ? 2 * it.j : 0;
  it.nq = max(0, n_qt - it.i_first);
  return it;
}

// Item of round r for this CTA in snake order, or -1 once the list is done
// (every later round is past the end as well).
__device__ __forceinline__ int item_of(int r, int total) {
  const long long G = gridDim.x;
  const long long c = (r & 1) ? (G - 1 - (long long)blockIdx.x) : (long long)blockIdx.x;
  const long long idx = (long long)r * G + c;
  return idx < total ? (int)idx : -1;
}
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreadsR, 1)
    bwd_main_persistent_kernel(const __grid_constant__ CUtensorMap tmQ,   // box 64 rows
                         const __grid_constant__ CUtensorMap tmK,   // box 128 rows
                         const __grid_constant__ CUtensorMap tmV,   // box 128 rows
                         const __grid_constant__ CUtensorMap tmDO,  // box 64 rows
                         const __grid_constant__ CUtensorMap tmDK,  // box 128 rows
                         const __grid_constant__ CUtensorMap tmDV,  // box 128 rows
                         const float* __restrict__ neg_lse2, const float* __restrict__ delta,
                         float* __restrict__ dqacc, int BH, int N, int Npad, int heads_per_group,
                         float scale, float scale_log2) {
  using C = PCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_kt = Npad / kBlockN;
  const int n_qt = (N + kBM - 1) / kBM;
  const int total = BH * n_kt;
  auto item = [&](int L) { return bwd_item(L, BH, n_kt, n_qt, heads_per_group, CAUSAL); };

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* bar_kvfull = bars + 0;     // [2] K_j / V_j slot loaded
  uint64_t* bar_kvfree = bars + 2;     // [2] every product reading the slot has completed
  uint64_t* bar_qfull = bars + 4;      // [5]
  uint64_t* bar_qempty = bars + 7;     // [5]
  uint64_t* bar_sfull = bars + 10;     // [2]
  uint64_t* bar_pready = bars + 12;    // [2]
  uint64_t* bar_dpfull = bars + 14;    // [2]
  uint64_t* bar_dsready = bars + 16;   // [2]
  uint64_t* bar_dqfull = bars + 18;    // [2]
  uint64_t* bar_dqfree = bars + 20;    // [2]
  uint64_t* bar_dqdone = bars + 22;    // [2]
  uint64_t* bar_itemdone = bars + 24;  // every product of an item has completed
  uint64_t* bar_accfree = bars + 25;   // the drain warps have read dV and dK out of TMEM
  uint64_t* bar_final = bars + 26;
  uint64_t* bar_epifull = bars + 27;   // [2] a staged dV / dK chunk is complete
  uint64_t* bar_epifree = bars + 29;   // [2] its TMA store has read the staging slot
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBarsP);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  // The next kernel in the stream may be scheduled once every CTA is running.
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    *s_abort = (smem_u32(smem) & 1023u) != 0;
    for (int s = 0; s < kStagesP; ++s) {
      mbar_init(&bar_qfull[s], 1);
      mbar_init(&bar_qempty[s], 1 + 8);  // MMA commit + one arrive per compute warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_kvfull[b], 1);
      mbar_init(&bar_kvfree[b], 1);
      mbar_init(&bar_sfull[b], 1);
      mbar_init(&bar_pready[b], 256);
      mbar_init(&bar_dpfull[b], 1);
      mbar_init(&bar_dsready[b], 256);
      mbar_init(&bar_dqfull[b], 1);
      mbar_init(&bar_dqfree[b], 128);
      mbar_init(&bar_dqdone[b], 1);
      mbar_init(&bar_epifull[b], 128);
      mbar_init(&bar_epifree[b], 1);
    }
    mbar_init(bar_itemdone, 1);
    mbar_init(bar_accfree, 128);
    mbar_init(bar_final, 1);
#ifdef ATTN_TEST_HOOKS
    mbar_init(reinterpret_cast<uint64_t*>(tmem_slot + 2), 1);  // nothing arrives here
#endif
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
  const bool abort_all = *s_abort != 0;
  // Set-up above touches no global memory; from here on the preprocess
  // kernel's results must be complete and visible.
  griddep_wait();
  if (threadIdx.x == 0 && abort_all) set_fail(ATTN_ERR_INVALID_ARG);

  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sDO = smem + C::kOffDO;
  uint8_t* sDS = smem + C::kOffDS;
  float* sLse = reinterpret_cast<float*>(smem + C::kOffLse);
  float* sDelta = reinterpret_cast<float*>(smem + C::kOffDelta);

  // Barrier phases run on across items.  Every role numbers the 64-row query
  // tiles it has handled in this CTA (T) and the items (n); the Q / dO ring
  // slot is T % 3, the S^T, dP^T and dQ^T buffers T % 2, the K / V slot n % 2.
  // A barrier of a double buffer completes once per use of its buffer, and
  // each use is consumed before the next one can start, so no waiter falls
  // two phases behind.  Items with no query tile (none occur for the shapes
  // accepted) are skipped by every role alike.
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsWG0));
    if (warp == 0 && lane == 0 && !abort_all) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      bool ok = true;
      int T = 0, items = 0;
      auto load_q = [&](int tile, int bh) -> bool {
        const int st = T % kStagesP, use = T / kStagesP;
        if (use > 0 && !mbar_wait(&bar_qempty[st], (use - 1) & 1)) return false;
        mbar_arrive_expect_tx(&bar_qfull[st], 2 * C::kQBytes + 2 * kBM * 4);
        tma_load_3d(sQ + st * C::kQBytes, &tmQ, &bar_qfull[st], 0, tile * kBM, bh);
        tma_load_3d(sDO + st * C::kQBytes, &tmDO, &bar_qfull[st], 0, tile * kBM, bh);
        const size_t prow = (size_t)bh * Npad + (size_t)tile * kBM;
        bulk_load(sLse + st * kBM, neg_lse2 + prow, kBM * 4, &bar_qfull[st]);
        bulk_load(sDelta + st * kBM, delta + prow, kBM * 4, &bar_qfull[st]);
        ++T;
        return true;
      };
      for (int rr = 0; ok; ++rr) {
        const int L = item_of(rr, total);
        if (L < 0) break;
        const BwdItem it = item(L);
        if (it.nq == 0) continue;
        // The item's first Q / dO tile, then K_j and V_j into slot n % 2 once
        // the item two back, which used that slot, has completed its products.
        if (!load_q(it.i_first, it.bh)) { ok = false; break; }
        const int slot = items & 1;
        if (items >= 2 && !mbar_wait(&bar_kvfree[slot], ((items >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bar_kvfull[slot], 2 * C::kKVBytes);
        tma_load_3d(sK + slot * C::kKVBytes, &tmK, &bar_kvfull[slot], 0, it.j * kBlockN, it.bh);
        tma_load_3d(sV + slot * C::kKVBytes, &tmV, &bar_kvfull[slot], 0, it.j * kBlockN, it.bh);
        ++items;
        for (int q = 1; q < it.nq; ++q)
          if (!load_q(it.i_first + q, it.bh)) { ok = false; break; }
      }
      if (!ok) set_fail(ATTN_ERR_TIMEOUT);
      // Do not leave while copies into this CTA's shared memory are in flight.
      for (int x = max(0, items - 2); x < items; ++x)
        mbar_wait(&bar_kvfull[x & 1], (x >> 1) & 1);
      for (int x = max(0, T - kStagesP); x < T; ++x)
        mbar_wait(&bar_qfull[x % kStagesP], (x / kStagesP) & 1);
    } else if (warp == 1 && !abort_all) {
      // ------------------------------------------------------------ MMA issuer
      // Whole warp, warp-uniform operands; elect.sync picks the issuing lane.
      constexpr uint32_t idesc_s = idesc_bf16(128, kBM, false, false);  // K-major A and B
      constexpr uint32_t idesc_acc = idesc_bf16(128, D, false, true);   // TMEM A, MN-major B
      constexpr uint32_t idesc_dq = idesc_bf16(D, kBM, true, true);     // MN-major A and B
      const uint64_t kQ = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t kDO = sdesc_sw128(smem_u32(sDO), 16, 1024);
      const uint64_t mQ = sdesc_sw128(smem_u32(sQ), kQChunk, 1024);
      const uint64_t mDO = sdesc_sw128(smem_u32(sDO), kQChunk, 1024);
      const uint64_t mDS = sdesc_sw128(smem_u32(sDS), kDSBytes, 1024);
      // S^T or dP^T (into column d_col) = X_j Y_i^T over the d = 64 head dims.
      auto issue_xy = [&](uint32_t d_col, uint64_t dX, uint64_t dY, uint32_t y_off) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_elect(tmem + d_col, sdesc_add(dX, kk * 32), sdesc_add(dY, y_off + kk * 32),
                       idesc_s, kk > 0 ? 1u : 0u);
      };
      bool ok = true;
      int T0 = 0, items = 0;
      for (int rr = 0; ok; ++rr) {
        const int L = item_of(rr, total);
        if (L < 0) break;
        const BwdItem it = item(L);
        if (it.nq == 0) continue;
        const int slot = items & 1;
        const uint64_t kK = sdesc_sw128(smem_u32(sK + slot * C::kKVBytes), 16, 1024);
        const uint64_t kV = sdesc_sw128(smem_u32(sV + slot * C::kKVBytes), 16, 1024);
        const uint64_t mK = sdesc_sw128(smem_u32(sK + slot * C::kKVBytes), kKVChunk, 1024);
        // S^T(T) and dP^T(T) into buffers T % 2, once Q_i / dO_i have landed.
        auto issue_sdp = [&](int T) -> bool {
          const int stT = T % kStagesP;
          if (!warp_wait(&bar_qfull[stT], (T / kStagesP) & 1)) return false;
          tc_fence_after();
          issue_xy(C::kColS + (T & 1) * kBM, kK, kQ, stT * C::kQBytes);
          mma_commit_elect(&bar_sfull[T & 1]);
          issue_xy(C::kColDP + (T & 1) * kBM, kV, kDO, stT * C::kQBytes);
          mma_commit_elect(&bar_dpfull[T & 1]);
          return true;
        };
        // Prologue: S^T and dP^T of the item's first two tiles.  Their buffers
        // are free: the products of the previous item that read them (dV and
        // dK of its last two tiles) were issued earlier on this thread.
        ok = warp_wait(&bar_kvfull[slot], (items >> 1) & 1);
        if (!ok) break;
        if (!issue_sdp(T0)) { ok = false; break; }
        if (it.nq > 1 && !issue_sdp(T0 + 1)) { ok = false; break; }
        for (int q = 0; q < it.nq && ok; ++q) {
          const int T = T0 + q;
          const int st = T % kStagesP, b = T & 1;
          const uint32_t so = st * C::kQBytes;
          // dV += P^T dO_i.  The first dV / dK products of an item overwrite the
          // accumulators, so they wait until the drain warps have read the
          // previous item's dV and dK out of TMEM.
          if (!warp_wait(&bar_pready[b], (T >> 1) & 1)) { ok = false; break; }
          if (q == 0 && items > 0 && !warp_wait(bar_accfree, (items - 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBM / 16; ++kk)
            mma_ts_elect(tmem + C::kColDV, tmem + C::kColS + b * kBM + packed_col(kk),
                         sdesc_add(mDO, so + kk * 2048), idesc_acc, (q > 0 || kk > 0) ? 1u : 0u);
          // dK += dS^T Q_i
          if (!warp_wait(&bar_dsready[b], (T >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBM / 16; ++kk)
            mma_ts_elect(tmem + C::kColDK, tmem + C::kColDP + b * kBM + packed_col(kk),
                         sdesc_add(mQ, so + kk * 2048), idesc_acc, (q > 0 || kk > 0) ? 1u : 0u);
          mma_commit_elect(&bar_qempty[st]);
          // S^T(T+2) and dP^T(T+2) into buffers b: dV(T) and dK(T) above have
          // read P^T(T) and dS^T(T) from them.  Issued ahead of dQ^T(T), which
          // no compute warp waits for (61.4 -> 61.1 us on the gpt2 workload).
          if (q + 2 < it.nq && !issue_sdp(T + 2)) { ok = false; break; }
          // dQ^T(T) = K_j^T dS^T(T) into dQ buffer b, once the drain warps have
          // read dQ^T(T-2) from it.
          if (T >= 2 && !warp_wait(&bar_dqfree[b], ((T >> 1) - 1) & 1)) { ok = false; break; }
#pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk)
            mma_ss_elect(tmem + C::kColDQ + b * kBM, sdesc_add(mK, kk * 2048),
                         sdesc_add(mDS, b * kDSBytes + kk * 2048), idesc_dq, kk > 0 ? 1u : 0u);
          mma_commit_elect(&bar_dqfull[b]);
          mma_commit_elect(&bar_dqdone[b]);
        }
        if (!ok) break;
        // dV, dK complete; the K / V slot may be refilled.
        mma_commit_elect(bar_itemdone);
        mma_commit_elect(&bar_kvfree[slot]);
        T0 += it.nq;
        ++items;
      }
      if (!ok && lane == 0) set_fail(ATTN_ERR_TIMEOUT);
      mma_commit_elect(bar_final);
      mbar_wait(bar_final, 0);
    } else if (warp == 3 && lane == 0 && !abort_all) {
      // ---------------------------------------------------- dV / dK stores
      // One TMA store per staged 64-column chunk; the staging slot is handed
      // back once the store has read it.
      bool ok = true;
      int es[2] = {0, 0};
      for (int rr = 0; ok; ++rr) {
        const int L = item_of(rr, total);
        if (L < 0) break;
        const BwdItem it = item(L);
        if (it.nq == 0) continue;
        for (int h = 0; h < 2; ++h) {
          if (!mbar_wait(&bar_epifull[h], es[h] & 1)) { ok = false; break; }
          tma_store_3d(h == 0 ? &tmDV : &tmDK, smem + C::kOffStage + h * kKVChunk, 0,
                       it.j * kBlockN, it.bh);
          bulk_commit_group();
          bulk_wait_group_read0();
          mbar_arrive(&bar_epifree[h]);
          ++es[h];
        }
      }
      if (!ok) set_fail(ATTN_ERR_TIMEOUT);
      // The output stores complete before this CTA ends.
      bulk_wait_group0();
    }
    __syncwarp();
  } else if (warp >= 12) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsDrain));
    // ------------------------------------------------------------ dQ drain
    // dQ^T(T) (M = 64) from dQ buffer T % 2: head dim m is TMEM lane
    // (m / 16) * 32 + m % 16, so lanes 0-15 of each warp hold 16 head dims
    // and add them, one query row per reduction (64 contiguous bytes).
    const int dim = (warp & 3) * 16 + (lane & 15);
    const bool holds_dim = lane < 16;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tDQ = tmem + lane_off + C::kColDQ;
    const int r = (warp & 3) * 32 + lane;  // key row = TMEM lane, for the dV / dK epilogue
    bool ok = !abort_all;
    int T = 0, items = 0, es = 0;
    for (int rr = 0; ok; ++rr) {
      const int L = item_of(rr, total);
      if (L < 0) break;
      const BwdItem it = item(L);
      if (it.nq == 0) continue;
      for (int q = 0; q < it.nq && ok; ++q, ++T) {
        const int b = T & 1;
        ok = warp_wait(&bar_dqfull[b], (T >> 1) & 1);
        if (!ok) break;
        tc_fence_after();
        uint32_t acc[2][32];
        tmem_ld32(tDQ + b * kBM, acc[0]);
        tmem_ld32(tDQ + b * kBM + 32, acc[1]);
        tmem_wait_ld();
        reg_fence(acc[0]);
        reg_fence(acc[1]);
        tc_fence_before();
        mbar_arrive(&bar_dqfree[b]);
        float* dst = dqacc + ((size_t)it.bh * Npad + (size_t)(it.i_first + q) * kBM) * D + dim;
        if (holds_dim) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dst + (size_t)c * D),
                         "f"(__uint_as_float(acc[c >> 5][c & 31]))
                         : "memory");
        }
      }
      if (!ok) break;
      // ------------------------ epilogue: dV and scale * dK of the item
      // Once every product of the item has completed, read dV and dK out of
      // TMEM (32 columns at a time), release the accumulators to the next
      // item's products, and stage them as BF16 for warp 3's TMA stores.
      ok = warp_wait(bar_itemdone, items & 1);
      if (!ok) break;
      ++items;
      tc_fence_after();
      if (es > 0) {
        ok = warp_wait(&bar_epifree[0], (es - 1) & 1) && warp_wait(&bar_epifree[1], (es - 1) & 1);
        if (!ok) break;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t tAcc = tmem + lane_off + (h == 0 ? C::kColDV : C::kColDK);
        const uint32_t aStage = smem_u32(smem + C::kOffStage + h * kKVChunk);
        const float mul = h == 0 ? 1.f : scale;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t o[32];
          tmem_ld32(tAcc + hh * 32, o);
          tmem_wait_ld();
          reg_fence(o);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * mul, __uint_as_float(o[2 * e + 1]) * mul);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            st_shared_v4(aStage + sw128_offset(r, hh * 4 + u), pk[4 * u], pk[4 * u + 1],
                         pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar_accfree);  // the next item's dV / dK products may overwrite them
      fence_proxy_async_smem();
      mbar_arrive(&bar_epifull[0]);  // warp 3 stores dV
      mbar_arrive(&bar_epifull[1]);  // and dK
      ++es;
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
    const uint32_t dsBase0 = smem_u32(sDS);
    const uint64_t c2 = f2_pack(scale_log2, scale_log2);
    bool ok = !abort_all;
#ifdef ATTN_TEST_HOOKS
    if (ok && g_hook_stall_bwd && blockIdx.x == 0 && h == 0)
      ok = warp_wait(reinterpret_cast<uint64_t*>(tmem_slot + 2), 0);
#endif
    int T = 0;
    for (int rr = 0; ok; ++rr) {
      const int L = item_of(rr, total);
      if (L < 0) break;
      const BwdItem itm = item(L);
      if (itm.nq == 0) continue;
      const int j = itm.j;
      const int kv = j * kBlockN + r;
      const bool key_valid = kv < N;
      for (int q = 0; q < itm.nq && ok; ++q, ++T) {
        const int st = T % kStagesP, b = T & 1;
        const int i = itm.i_first + q;
        const uint32_t tS = tmem + lane_off + C::kColS + b * kBM;
        const uint32_t tDP = tmem + lane_off + C::kColDP + b * kBM;
        ok = warp_wait(&bar_qfull[st], (T / kStagesP) & 1);
        if (!ok) break;
        ok = warp_wait(&bar_sfull[b], (T >> 1) & 1);
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

        ok = warp_wait(&bar_dpfull[b], (T >> 1) & 1);
        if (!ok) break;
        // dS^T buffer b is free once dQ^T(T-2), which read it, has completed.
        if (T >= 2) {
          ok = warp_wait(&bar_dqdone[b], ((T >> 1) - 1) & 1);
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
        mbar_arrive(&bar_dsready[b]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_qempty[st]);
      }
    }
    if (!ok) set_fail(ATTN_ERR_TIMEOUT);
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
  return launch_pdl(bwd_preprocess_kernel<D>, dim3(blocks), dim3(256), 0, stream,
                    static_cast<const uint4*>(o), static_cast<const uint4*>(dout), lse, ws.neg_lse2,
                    ws.delta, reinterpret_cast<float4*>(ws.dqacc), p.N, Npad, per_head);
}

template <int D>
cudaError_t dq_convert_impl(const Problem& p, const BwdWorkspace& ws, void* dq,
                            cudaStream_t stream) {
  const long long units = (long long)p.B * p.H * p.N * (D / 8);
  const int blocks = (int)((units + 255) / 256);
  return launch_pdl(bwd_dq_convert_kernel<D>, dim3(blocks), dim3(256), 0, stream,
                    reinterpret_cast<const float4*>(ws.dqacc), static_cast<uint4*>(dq), p.N,
                    n_pad(p.N), p.scale, (int)units);
}

// Heads per CTA group of the main kernel.  Ordering CTAs by head group keeps
// the Q / dO tiles, LSE / delta rows and dQ accumulator rows of the heads in
// flight (about 8 N d bytes per head) inside a 48 MiB share of the L2, so that
// the key-tile CTAs of a head re-read them from L2 rather than HBM.  Within a
// group the heaviest key tiles come first; the last group is dispatched last,
// so it must hold enough work per SM (1.2 x the heaviest CTA) that its
// heaviest CTAs do not outlast the rest of the launch.  Fewer groups win when
// the two limits disagree.
int bwd_heads_per_group(int BH, int N, int d, bool causal) {
  const int num_sms = device_sm_count();
  if (num_sms <= 0) return BH;  // one group: the plain heaviest-first order
  const double per_head_bytes = 8.0 * N * d;
  const int g_l2 = max(1, (int)(48.0 * 1048576.0 / per_head_bytes));
  const int n_qt = ceil_div(N, r64::kBM), n_kt = n_pad(N) / kBlockN;
  double tiles_per_head = 0.0;
  for (int j = 0; j < n_kt; ++j) tiles_per_head += max(0, n_qt - (causal ? 2 * j : 0));
  const double g_tail = 1.2 * n_qt * num_sms / tiles_per_head;
  int groups = ceil_div(BH, g_l2);
  groups = min(groups, max(1, (int)(BH / g_tail)));
  return ceil_div(BH, groups);
}

template <int D, bool CAUSAL>
cudaError_t main_r64_impl(const Problem& p, const CUtensorMap* maps, const BwdWorkspace& ws,
                          cudaStream_t stream) {
  auto kernel = r64::bwd_main_r64_kernel<D, CAUSAL>;
  constexpr int kSmem = r64::Cfg<D>::kSmemBytes;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (err != cudaSuccess) return err;
  const int BH = p.B * p.H;
  const int Npad = n_pad(p.N);
  const int n_kt = Npad / kBlockN;
  const int hpg = bwd_heads_per_group(BH, p.N, D, CAUSAL);
  return launch_pdl(kernel, dim3(BH * n_kt), dim3(r64::kThreadsR), kSmem, stream, maps[0], maps[1],
                    maps[2], maps[3], maps[4], maps[5], static_cast<const float*>(ws.neg_lse2),
                    static_cast<const float*>(ws.delta), ws.dqacc, BH, p.N, Npad, hpg, p.scale,
                    p.scale * 1.4426950408889634f);
}

// d = 64: persistent CTAs, one per SM, walking the (head, key tile) items in
// snake order.  The list is ordered heaviest first across all heads (one
// group): a static schedule over head groups left late heavy items.  When it
// was introduced it ran the gpt2 workload's backward main phase in 66 us
// against 74 for one CTA per item (61 us with the double-buffered products
// it has now); at d = 128 persistence measured slower (311 against 295 us on
// the llama7b workload), so d = 128 keeps one CTA per item.
template <int D, bool CAUSAL>
cudaError_t main_persistent_impl(const Problem& p, const CUtensorMap* maps, const BwdWorkspace& ws,
                                 cudaStream_t stream) {
  auto kernel = r64::bwd_main_persistent_kernel<D, CAUSAL>;
  constexpr int kSmem = r64::PCfg<D>::kSmemBytes;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (err != cudaSuccess) return err;
  const int BH = p.B * p.H;
  const int Npad = n_pad(p.N);
  const int n_kt = Npad / kBlockN;
  const int total = BH * n_kt;
  const int sms = device_sm_count();
  const int grid = sms > 0 ? std::min(total, sms) : total;
  return launch_pdl(kernel, dim3(grid), dim3(r64::kThreadsR), kSmem, stream, maps[0], maps[1],
                    maps[2], maps[3], maps[4], maps[5], static_cast<const float*>(ws.neg_lse2),
                    static_cast<const float*>(ws.delta), ws.dqacc, BH, p.N, Npad, BH, p.scale,
                    p.scale * 1.4426950408889634f);
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
  // 64-row query tiles (Q and dO maps with 64-row boxes).
  const int q_rows = r64::kBM;
  const int box_rows[6] = {q_rows, kBlockN, kBlockN, q_rows, kBlockN, kBlockN};
  for (int i = 0; i < 6; ++i)
    if (!make_tmap_bhnd(&maps[i], ptrs[i], BH, p.N, p.d, box_rows[i]))
      return cudaErrorInvalidValue;
  if (p.d == 128)
    return p.causal ? main_r64_impl<128, true>(p, maps, ws, stream)
                    : main_r64_impl<128, false>(p, maps, ws, stream);
  return p.causal ? main_persistent_impl<64, true>(p, maps, ws, stream)
                  : main_persistent_impl<64, false>(p, maps, ws, stream);
}

#ifdef ATTN_TEST_HOOKS
extern "C" ATTN_API int attn_testhook_stall_bwd(int on) {
  return (int)cudaMemcpyToSymbol(g_hook_stall_bwd, &on, sizeof(on));
}
#endif

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
