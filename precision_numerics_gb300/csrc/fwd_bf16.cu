// BF16 attention forward for sm_103a: TMA + tcgen05 (TMEM accumulators),
// warp-specialised producer / MMA / softmax roles, FP32 online softmax.
//
// What is computed: O = softmax(scale Q K^T [+ causal mask]) V and the
// natural-log LSE of each row ("Is Flash Attention Stable?", abstract:
// Baseline Attention), evaluated blockwise as in "Why Low-Precision
// Transformer Training Fails", Algorithm 1: Q is cut into 128-row blocks,
// K and V into 128-row blocks; for each K/V block the row max m is updated,
// P = exp(S - m) (P-bar in that paper's Figures 5 and 7), the row sum and
// the partial output are rescaled by exp(m_old - m_new), and P V is
// accumulated.  The softmax runs in FP32; P is rounded to BF16 (nearest
// even) only as the operand of the P V product; the row sum accumulates the
// FP32 values.
//
// Persistent CTAs: the grid has at most one CTA per SM, and each CTA walks a
// fixed list of work items (an item = 2 query tiles of 128 rows, 256 rows of
// one (b, h)).  Items are numbered heaviest first (causal: the last query
// rows of every head first) and dealt to the CTAs in snake order (CTA c
// takes item c of round 0, item G-1-c of round 1, ...), so the rounds'
// heavy and light items even out.  Barriers and TMEM are set up once per
// CTA; the next item's Q tiles load as soon as the current item's last S
// products have read Q, and its first S products are issued while the
// softmax warps still write the current item's output, so an item's start
// overlaps the previous item's end.
//
// 16 warps:
//   warp 0      TMA producer (Q once per item; K_j, V_j through a ring)
//   warp 1      MMA issuer: S_t = Q_t K_j^T, O_t += P_t V_j
//   warp 2      TMEM allocation owner
//   warp 3      TMA stores of the staged output (d = 128)
//   warps 4-7   softmax of tile 0, warps 8-11 softmax of tile 1; each
//               thread owns one query row (one TMEM lane), so row max and
//               row sum need no cross-thread reduction.  They also stage
//               the item's O for TMA stores and write its LSE.
//   warps 12-15 correction: rescale O_t by exp(m_old - m_new) for both tiles
//               while the softmax warps compute the exponentials, so the
//               rescale is off the softmax's critical path.
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+d),
// O_1 [256+d,256+2d).  P_t (BF16, two per 32-bit column) overwrites the
// first 64 columns of S_t and is the A operand of the P V MMA.  The MMA
// issue order PV_0(j), S_0(j+1), PV_1(j), S_1(j+1) lets the tensor pipe
// work on one tile while the other tile's softmax runs.
#include <math.h>

#include <algorithm>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {

static __device__ unsigned int g_status_fwd;

namespace {

constexpr int kThreads = 512;
// Correction warps: 32-column O chunks loaded per TMEM round trip, and the
// register split (setmaxnreg) that goes with it.
constexpr int kCorrChunks = 1;
constexpr int kRegsWG0 = 80, kRegsCorr = 80, kRegsSoftmax = 176;  // 80 + 80 + 2 * 176 <= 512
// A 512-thread launch gives 128 registers per thread: setmaxnreg.dec must ask
// for fewer, setmaxnreg.inc for more.
static_assert(kRegsWG0 <= 128 && kRegsCorr <= 128 && kRegsSoftmax >= 128, "setmaxnreg directions");

template <int D>
struct FwdCfg {
  static constexpr int kStages = (D == 128) ? 2 : 3;
  static constexpr int kChunks = D / 64;          // 64-column (128-byte) chunks per row
  static constexpr int kChunkBytes = 128 * 128;   // 128 rows x 128 bytes
  static constexpr int kTileBytes = 128 * D * 2;  // 128 rows x d BF16
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  // Output: at d = 128 staged one 64-column chunk (128 rows x 128 bytes) per
  // query tile and written by TMA; at d = 64 each thread's row is one 128-byte
  // line, written straight from registers (measured ~5% faster there; at
  // d = 128 the direct stores were ~1.5% slower).
  static constexpr bool kStagedOut = (D == 128);
  static constexpr int kOffStage = kOffV + kStages * kTileBytes;
  // INT8 variant: the key scales of each K tile (128 FP32) in a ring of their
  // own, with a full barrier per slot.  Slot g % kKsSlots is refilled for key
  // tile g + kKsSlots when K of that tile loads, which waits until the S
  // products of tile g + 1 have completed; those were issued only once both
  // softmax warpgroups had finished tile g.  So the slot's previous scales
  // have been read, and no softmax warp falls two phases behind its barrier.
  static constexpr int kKsSlots = kStages + 1;
  static constexpr int kOffKs = kOffStage + (kStagedOut ? 2 * kChunkBytes : 0);
  static constexpr int kOffBar = kOffKs + kKsSlots * 128 * 4;
  // q_full, q_empty, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2],
  // p_full[2], o_done[2], mma_final, alpha[2][4] (one per tile and softmax
  // warp), epi_full[2], epi_free[2], ks_full[kKsSlots]
  static constexpr int kNumBars = 2 + 4 * kStages + 19 + kKsSlots;
  static constexpr int kOffAlpha = kOffBar + kNumBars * 8 + 16;  // FP32 [2][128]
  static constexpr int kSmemBytes = kOffAlpha + 2 * 128 * 4;
  static constexpr uint32_t kTmemCols = 512;
  // TMEM column of S_t and O_t.
  static __device__ __forceinline__ uint32_t col_s(int t) { return 128u * t; }
  static __device__ __forceinline__ uint32_t col_o(int t) { return 256u + D * t; }
};

__device__ __forceinline__ void set_fail(unsigned int code) { atomicOr(&g_status_fwd, code); }

#ifdef ATTN_TEST_HOOKS
// Test instrumentation, compiled only into the separate test build of the
// library (ATTN_TEST_HOOKS), never into libattn.so:
//  - g_hook_pbar_ones: when set, every query row adds the number of its BF16
//    P-bar operands (the P V inputs) equal to exactly 1.0 into
//    g_hook_pbar_ones[b*H*N + h*N + row] (rows below g_hook_rows only);
//  - g_hook_stall: when set, the first softmax warpgroup of CTA 0 first waits
//    on a barrier that nothing ever arrives at, so the wait runs out (after the
//    test build's short limit) and the kernel takes its failure path.
static __device__ unsigned int* g_hook_pbar_ones;
static __device__ unsigned long long g_hook_rows;
static __device__ int g_hook_stall;
#endif

// Number of K/V tiles the query tile starting at row q_first visits.
__device__ __forceinline__ int kv_tiles_for(int q_first, int N, bool causal) {
  if (q_first >= N) return 0;
  if (!causal) return (N + kBlockN - 1) / kBlockN;
  const int q_last = min(q_first + kBlockM - 1, N - 1);
  return q_last / kBlockN + 1;
}

// Item of round r for this CTA in snake order, or -1 once the list is done
// (every later round is past the end as well).
__device__ __forceinline__ int item_of(int r, int total) {
  const long long G = gridDim.x;
  const long long c = (r & 1) ? (G - 1 - (long long)blockIdx.x) : (long long)blockIdx.x;
  const long long idx = (long long)r * G + c;
  return idx < total ? (int)idx : -1;
}

// Item L (heaviest first): head bh, first query row q0, K/V tiles of its two
// query tiles.
struct Item {
  int bh, q0, n[2], nmax;
};
__device__ __forceinline__ Item item_coords(int L, int BH, int N, int num_qt, bool causal) {
  Item it;
  const int qt = num_qt - 1 - L / BH;
  it.bh = L % BH;
  it.q0 = qt * (2 * kBlockM);
  it.n[0] = kv_tiles_for(it.q0, N, causal);
  it.n[1] = kv_tiles_for(it.q0 + kBlockM, N, causal);
  it.nmax = max(it.n[0], it.n[1]);
  return it;
}

// I8: Q and K hold per-token INT8 codes as BF16 values (exact integers), with
// FP32 row scales qs / ks in the padded layout [B*H][Npad]; the S products
// are then exact integer dot products (every product |c_q c_k| <= 127^2 and
// every partial sum over d <= 128 terms stays below 2^24, exact in the FP32
// accumulator in any order), and the logits are scale * qs_i * ks_j * S_ij.
template <int D, bool CAUSAL, bool STABLE, bool I8>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    uint16_t* __restrict__ out, float* __restrict__ lse, int BH, int N, int num_qt, float scale,
                    float scale_log2, float beta, const float* __restrict__ qs,
                    const float* __restrict__ ks, int Npad) {
  using C = FwdCfg<D>;
  static_assert(kRegsWG0 + kRegsCorr + 2 * kRegsSoftmax <= 512, "setmaxnreg split exceeds the launch pool");
  extern __shared__ __align__(1024) uint8_t smem[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int total = BH * num_qt;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* bar_q = bars;
  uint64_t* bar_qempty = bars + 1;
  uint64_t* bar_kfull = bars + 2;
  uint64_t* bar_kempty = bar_kfull + C::kStages;
  uint64_t* bar_vfull = bar_kempty + C::kStages;
  uint64_t* bar_vempty = bar_vfull + C::kStages;
  uint64_t* bar_sfull = bar_vempty + C::kStages;
  uint64_t* bar_pfull = bar_sfull + 2;
  uint64_t* bar_odone = bar_pfull + 2;
  uint64_t* bar_final = bar_odone + 2;
  uint64_t* bar_alpha = bar_final + 1;
  uint64_t* bar_epifull = bar_alpha + 8;  // a staged O chunk is complete
  uint64_t* bar_epifree = bar_epifull + 2;  // its TMA store has read the staging slot
  uint64_t* bar_ksfull = bar_epifree + 2;  // INT8: a key-scale slot has landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  float* s_alpha = reinterpret_cast<float*>(smem + C::kOffAlpha);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  // The next kernel in the stream may be scheduled once every CTA is running.
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    *s_abort = (smem_u32(smem) & 1023u) != 0;
    mbar_init(bar_q, 1);
    mbar_init(bar_qempty, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bar_kfull[s], 1);
      mbar_init(&bar_kempty[s], 1);
      mbar_init(&bar_vfull[s], 1);
      mbar_init(&bar_vempty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar_sfull[t], 1);
      mbar_init(&bar_pfull[t], 256);  // softmax (P stored) + correction (O rescaled)
      for (int q = 0; q < 4; ++q) mbar_init(&bar_alpha[t * 4 + q], 32);
      mbar_init(&bar_odone[t], 1);
      mbar_init(&bar_epifull[t], 128);
      mbar_init(&bar_epifree[t], 1);
    }
    for (int k = 0; k < C::kKsSlots; ++k) mbar_init(&bar_ksfull[k], 1);
    mbar_init(bar_final, 1);
#ifdef ATTN_TEST_HOOKS
    mbar_init(reinterpret_cast<uint64_t*>(tmem_slot + 2), 1);  // nothing arrives here
#endif
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
  // Set-up above touches no global memory; from here on the previous kernel's
  // results must be complete and visible.
  griddep_wait();
  if (threadIdx.x == 0 && abort_all) set_fail(ATTN_ERR_INVALID_ARG);

  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;

  // Barrier phases run on across items: every role counts the completions it
  // has consumed (K/V ring position g, items, S and P tiles per query tile).
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsWG0));
    if (warp == 0 && lane == 0 && !abort_all) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      bool ok = true;
      int g = 0, items = 0, issued_k = 0, issued_v = 0, issued_ks = 0;
      for (int r = 0; ok; ++r) {
        const int L = item_of(r, total);
        if (L < 0) break;
        const Item it = item_coords(L, BH, N, num_qt, CAUSAL);
        // The Q slots are free once the previous item's last S products have run.
        if (items > 0 && !mbar_wait(bar_qempty, (items - 1) & 1)) { ok = false; break; }
        mbar_arrive_expect_tx(bar_q, 2 * C::kTileBytes);
        for (int t = 0; t < 2; ++t)
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(sQ + t * C::kTileBytes + c * C::kChunkBytes, &tmQ, bar_q, c * 64,
                        it.q0 + t * kBlockM, it.bh);
        ++items;
        for (int j = 0; j < it.nmax; ++j, ++g) {
          const int st = g % C::kStages;
          const int use = g / C::kStages;
          if (use > 0 && !mbar_wait(&bar_kempty[st], (use - 1) & 1)) { ok = false; break; }
          mbar_arrive_expect_tx(&bar_kfull[st], C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(sK + st * C::kTileBytes + c * C::kChunkBytes, &tmK, &bar_kfull[st], c * 64,
                        j * kBlockN, it.bh);
          if constexpr (I8) {
            uint64_t* kb = &bar_ksfull[g % C::kKsSlots];
            mbar_arrive_expect_tx(kb, 128 * 4);
            bulk_load(smem + C::kOffKs + (g % C::kKsSlots) * 128 * 4,
                      ks + (size_t)it.bh * Npad + j * kBlockN, 128 * 4, kb);
            issued_ks = g + 1;
          }
          issued_k = g + 1;
          if (use > 0 && !mbar_wait(&bar_vempty[st], (use - 1) & 1)) { ok = false; break; }
          mbar_arrive_expect_tx(&bar_vfull[st], C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(sV + st * C::kTileBytes + c * C::kChunkBytes, &tmV, &bar_vfull[st], c * 64,
                        j * kBlockN, it.bh);
          issued_v = g + 1;
        }
      }
      if (!ok) set_fail(ATTN_ERR_TIMEOUT);
      // Do not leave while copies into this CTA's shared memory are in flight.
      if (items > 0) mbar_wait(bar_q, (items - 1) & 1);
      for (int x = max(0, issued_k - C::kStages); x < issued_k; ++x)
        mbar_wait(&bar_kfull[x % C::kStages], (x / C::kStages) & 1);
      for (int x = max(0, issued_v - C::kStages); x < issued_v; ++x)
        mbar_wait(&bar_vfull[x % C::kStages], (x / C::kStages) & 1);
      for (int x = max(0, issued_ks - C::kKsSlots); x < issued_ks; ++x)
        mbar_wait(&bar_ksfull[x % C::kKsSlots], (x / C::kKsSlots) & 1);
    } else if (warp == 1 && !abort_all) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs this role with warp-uniform operands; elect.sync
      // inside each MMA / commit picks the one lane that issues it.
      constexpr uint32_t idesc_qk = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(128, D, false, true);
      const uint64_t descQ = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t descK = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t descV = sdesc_sw128(smem_u32(sV), C::kChunkBytes, 1024);
      auto issue_s = [&](int t, int st) {
        const uint64_t a0 = sdesc_add(descQ, t * C::kTileBytes);
        const uint64_t b0 = sdesc_add(descK, st * C::kTileBytes);
        const uint32_t d = tmem + C::col_s(t);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          mma_ss_elect(d, sdesc_add(a0, off), sdesc_add(b0, off), idesc_qk, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, int st, bool acc) {
        const uint64_t b0 = sdesc_add(descV, st * C::kTileBytes);
        const uint32_t d = tmem + C::col_o(t), a = tmem + C::col_s(t);
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          mma_ts_elect(d, a + kk * 8, sdesc_add(b0, kk * 2048), idesc_pv,
                       (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = true;
      int g = 0, items = 0;
      int pc[2] = {0, 0};  // P tiles consumed per query tile (p_full phases)
      for (int r = 0; ok; ++r) {
        const int L = item_of(r, total);
        if (L < 0) break;
        const Item it = item_coords(L, BH, N, num_qt, CAUSAL);
        // S_t(0).  S_t's columns are free: the previous item's P_t V, issued
        // earlier on this thread, reads P_t before these products run.
        ok = warp_wait(bar_q, items & 1);
        if (ok) ok = warp_wait(&bar_kfull[g % C::kStages], (g / C::kStages) & 1);
        if (!ok) break;
        tc_fence_after();
        for (int t = 0; t < 2; ++t) {
          if (it.n[t] == 0) continue;
          issue_s(t, g % C::kStages);
          mma_commit_elect(&bar_sfull[t]);
        }
        mma_commit_elect(&bar_kempty[g % C::kStages]);  // K is free once S(0) has completed
        if (it.nmax == 1) mma_commit_elect(bar_qempty);  // every S product of the item issued
        ++items;
        for (int j = 0; j < it.nmax && ok; ++j) {
          const int gj = g + j;
          const int st = gj % C::kStages;
          const int st1 = (gj + 1) % C::kStages;
          const bool has_next = j + 1 < it.nmax;
          if (!warp_wait(&bar_vfull[st], (gj / C::kStages) & 1)) { ok = false; break; }
          if (has_next && !warp_wait(&bar_kfull[st1], ((gj + 1) / C::kStages) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int t = 0; t < 2 && ok; ++t) {
            if (j >= it.n[t]) continue;
            if (!warp_wait(&bar_pfull[t], (pc[t] + j) & 1)) { ok = false; break; }
            tc_fence_after();
            issue_pv(t, st, j > 0);
            if (j + 1 < it.n[t]) {
              issue_s(t, st1);
              mma_commit_elect(&bar_sfull[t]);
            } else {
              mma_commit_elect(&bar_odone[t]);
            }
          }
          if (!ok) break;
          mma_commit_elect(&bar_vempty[st]);
          // Release K_{j+1} as soon as the S(j+1) products above have read it, so
          // the producer can start loading K_{j+1+S} a full iteration ahead.
          if (has_next) mma_commit_elect(&bar_kempty[st1]);
          // The item's last S products were issued above: Q may be replaced.
          if (j + 2 == it.nmax) mma_commit_elect(bar_qempty);
        }
        g += it.nmax;
        pc[0] += it.n[0];
        pc[1] += it.n[1];
      }
      if (!ok && lane == 0) set_fail(ATTN_ERR_TIMEOUT);
      // Every MMA this warp issued completes before TMEM is released.
      mma_commit_elect(bar_final);
      mbar_wait(bar_final, 0);
    } else if (C::kStagedOut && warp == 3 && lane == 0 && !abort_all) {
      // ------------------------------------------------------------ O stores
      // One TMA store per staged 64-column chunk of O, in the order the
      // softmax warpgroups stage them (tile 0 finishes an item no later than
      // tile 1); the staging slot is handed back once the store has read it,
      // so no softmax warp waits for a store.
      bool ok = true;
      int es[2] = {0, 0};
      for (int rr = 0; ok; ++rr) {
        const int L = item_of(rr, total);
        if (L < 0) break;
        const Item it = item_coords(L, BH, N, num_qt, CAUSAL);
        for (int t = 0; t < 2 && ok; ++t) {
          if (it.n[t] == 0) continue;
          for (int c = 0; c < C::kChunks; ++c) {
            if (!mbar_wait(&bar_epifull[t], es[t] & 1)) { ok = false; break; }
            tma_store_3d(&tmO, smem + C::kOffStage + t * C::kChunkBytes, c * 64,
                         it.q0 + t * kBlockM, it.bh);
            bulk_commit_group();
            bulk_wait_group_read0();
            mbar_arrive(&bar_epifree[t]);
            ++es[t];
          }
        }
      }
      if (!ok) set_fail(ATTN_ERR_TIMEOUT);
      // The output stores complete before this CTA ends.
      bulk_wait_group0();
    }
    __syncwarp();
  } else if (warp >= 12) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCorr));
    // -------------------------------------------------------------- correction
    // O_t(j-1) has completed when the softmax of tile t publishes alpha(j):
    // that happens after S_t(j) completed, and the commit that signalled S_t(j)
    // covers every earlier MMA, PV_t(j-1) included.
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok = !abort_all;
    int ac[2] = {0, 0};  // alpha phases consumed per query tile
    for (int rr = 0; ok; ++rr) {
      const int L = item_of(rr, total);
      if (L < 0) break;
      const Item it = item_coords(L, BH, N, num_qt, CAUSAL);
      for (int j = 0; j < it.nmax && ok; ++j) {
        for (int t = 0; t < 2; ++t) {
          if (j >= it.n[t]) continue;
          // Only the softmax warp that owns the same 32 TMEM lanes is waited for.
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_alpha[t * 4 + (warp & 3)], (ac[t] + j) & 1));
          if (!ok) break;
          const float alpha = s_alpha[t * 128 + r];
          if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
            tc_fence_after();
            const uint32_t tO = tmem + lane_off + C::col_o(t);
            const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
            for (int c = 0; c < D / 32; c += kCorrChunks) {  // 32-column chunks per TMEM round trip
              uint32_t o[kCorrChunks][32];
#pragma unroll
              for (int h = 0; h < kCorrChunks; ++h) tmem_ld32(tO + (c + h) * 32, o[h]);
              tmem_wait_ld();
#pragma unroll
              for (int h = 0; h < kCorrChunks; ++h) {
                reg_fence(o[h]);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  float lo, hi;
                  f2_unpack(mul2(f2_pack(__uint_as_float(o[h][2 * i]), __uint_as_float(o[h][2 * i + 1])),
                                 a2),
                            lo, hi);
                  o[h][2 * i] = __float_as_uint(lo);
                  o[h][2 * i + 1] = __float_as_uint(hi);
                }
                tmem_st32(tO + (c + h) * 32, o[h]);
              }
            }
            tmem_wait_st();
          }
          tc_fence_before();
          mbar_arrive(&bar_pfull[t]);
        }
      }
      ac[0] += it.n[0];
      ac[1] += it.n[1];
    }
    if (!ok) set_fail(ATTN_ERR_TIMEOUT);
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // -------------------------------------------------------------- softmax
    const int t = (warp - 4) >> 2;
    const int r = (warp & 3) * 32 + lane;  // query row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::col_s(t);
    const uint32_t tO = tmem + lane_off + C::col_o(t);
    const uint32_t aStage = smem_u32(smem + C::kOffStage + t * C::kChunkBytes);
    bool ok = !abort_all;
    int sc = 0;  // S_t tiles consumed so far (s_full phases)
    int oc = 0;  // items whose O_t was completed so far (o_done phases)
    int gbase = 0;  // K/V ring position of the item's first key tile
    int es = 0;  // O chunks stored so far (epi_full / epi_free phases)
    for (int rr = 0; ok; ++rr) {
      const int L = item_of(rr, total);
      if (L < 0) break;
      const Item it = item_coords(L, BH, N, num_qt, CAUSAL);
      const int n = it.n[t];
      const int q_first = it.q0 + t * kBlockM;
      const int qi = q_first + r;
      // I8: the row's INT8 scale enters through the exponent factor c_row (a
      // row of zero codes has zero scores whatever its scale, so the scale is
      // kept above 1e-20 to keep c_row * -inf at -inf).
      const float sq = I8 ? fmaxf(qi < N ? qs[(size_t)it.bh * Npad + qi] : 0.f, 1e-20f) : 1.f;
      const float c_row = I8 ? scale_log2 * sq : scale_log2;
      // m_run: running row max; m_norm: the normaliser the exponentials of the
      // previous tiles used (equal to m_run except in the stabilised variant).
      float m_run = -INFINITY, m_norm = -INFINITY, l_run = 0.f;
      int n_at_max = 0;  // stabilised variant: elements equal to m_run so far (saturates at 2)
#ifdef ATTN_TEST_HOOKS
      unsigned int n_ones = 0;  // BF16 P-bar operands equal to 1.0 in this row
      if (g_hook_stall && blockIdx.x == 0 && t == 0 && rr == 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(reinterpret_cast<uint64_t*>(tmem_slot + 2), 0));
        if (!ok) break;
      }
#endif
      for (int j = 0; j < n; ++j) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_sfull[t], (sc + j) & 1));
        if (!ok) break;
        tc_fence_after();
        uint32_t s[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, s[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_fence(s[c]);
        if constexpr (I8) {
          // S_ij * ks_j: the key scales of this tile from the scale ring (entries
          // past N belong to masked keys).
          const int gk = gbase + j;
          ok = __all_sync(0xffffffffu,
                          mbar_wait(&bar_ksfull[gk % C::kKsSlots], (gk / C::kKsSlots) & 1));
          if (!ok) break;
          const float4* kr =
              reinterpret_cast<const float4*>(smem + C::kOffKs + (gk % C::kKsSlots) * 128 * 4);
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float4 k4 = kr[c * 8 + u];
              float a0, a1, a2, a3;
              f2_unpack(mul2(f2_pack(__uint_as_float(s[c][4 * u]), __uint_as_float(s[c][4 * u + 1])),
                             f2_pack(k4.x, k4.y)),
                        a0, a1);
              f2_unpack(mul2(f2_pack(__uint_as_float(s[c][4 * u + 2]), __uint_as_float(s[c][4 * u + 3])),
                             f2_pack(k4.z, k4.w)),
                        a2, a3);
              s[c][4 * u] = __float_as_uint(a0);
              s[c][4 * u + 1] = __float_as_uint(a1);
              s[c][4 * u + 2] = __float_as_uint(a2);
              s[c][4 * u + 3] = __float_as_uint(a3);
            }
        }

        const int kv0 = j * kBlockN;
        if (kv0 + kBlockN > N || (CAUSAL && kv0 + kBlockN - 1 > q_first)) {
          const int lim = (CAUSAL ? min(qi + 1, N) : N) - kv0;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= lim) s[c >> 5][c & 31] = __float_as_uint(-INFINITY);
        }
        // Row max as four independent chains of three-input maxima (short
        // dependency chains: few warps share an SM sub-partition to hide them).
        float mx4[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float m = fmaxf(__uint_as_float(s[c][0]), __uint_as_float(s[c][1]));
#pragma unroll
          for (int e = 2; e < 32; e += 2)
            m = fmax3(m, __uint_as_float(s[c][e]), __uint_as_float(s[c][e + 1]));
          mx4[c] = m;
        }
        const float m_tile = fmax3(mx4[0], mx4[1], mx4[2]);
        const float tile_max = fmaxf(m_tile, mx4[3]);
        const float m_new = fmaxf(tile_max, m_run);
        float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        if (STABLE) {
          // "Why Low-Precision Transformer Training Fails", Figure 7 / Algorithm 1:
          // when the row max r_m is attained more than once, normalise by beta * r_m
          // (r_m > 0) or by 0 (r_m < 0), so that no exp(S - m) equals exactly 1.
          // The count of elements equal to the running max is kept across tiles.
          if (tile_max >= m_run) {
            int cnt = 0;
#pragma unroll
            for (int c = 0; c < 128; ++c) cnt += __uint_as_float(s[c >> 5][c & 31]) == tile_max;
            n_at_max = min(2, (tile_max > m_run ? 0 : n_at_max) + cnt);
          }
          if (n_at_max >= 2 && m_new != -INFINITY) {
            m_use = m_new > 0.f ? beta * m_new : 0.f;
            // "Sufficiently negative": the row's largest exponent c * (r_m - m)
            // (base 2) is at most -2^-8, so its P-bar = 2^(c (r_m - m)) <= 0.99730
            // rounds to at most 1 - 2^-8 in BF16.  Without this floor a small
            // repeated maximum (0 <= c (beta - 1) r_m < 2.8e-3, r_m = 0, or
            // -2.8e-3 < c r_m < 0) still gives P-bar operands equal to 1.
            m_use = fmaxf(m_use, m_new + 0.00390625f / scale_log2);
            // Keep the row's largest exponent c * (r_m - m) at or above -64 (base 2),
            // so a very large repeated maximum cannot underflow every exponential
            // of the row (the pages do not discuss that range).
            m_use = fminf(m_use, m_new + 64.f / scale_log2);
          }
        }
        const float neg_ms = -m_use * c_row;
        const float alpha = ex2((m_norm - m_use) * c_row);
        s_alpha[t * 128 + r] = alpha;
        mbar_arrive(&bar_alpha[t * 4 + (warp & 3)]);  // the correction warp rescales O_t meanwhile
        // Eight partial row sums held as four packed pairs: element e of the
        // row goes to partial sum e mod 8.  Packed FP32 pair instructions halve
        // the FMA-pipe instruction count of the argument and sum updates.
        uint64_t sums2[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) sums2[u] = 0ull;
        const uint64_t c2 = f2_pack(c_row, c_row);
        const uint64_t nm2 = f2_pack(neg_ms, neg_ms);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1;
            f2_unpack(fma2(f2_pack(__uint_as_float(s[c][2 * i]), __uint_as_float(s[c][2 * i + 1])),
                           c2, nm2),
                      x0, x1);
            const float p0 = ex2(x0);
            const float p1 = ex2(x1);
            sums2[i & 3] = add2(sums2[i & 3], f2_pack(p0, p1));
            pk[i] = pack_bf16x2(p0, p1);
#ifdef ATTN_TEST_HOOKS
            n_ones += ((pk[i] & 0xFFFFu) == 0x3F80u) + ((pk[i] >> 16) == 0x3F80u);
#endif
          }
          tmem_st16(tS + c * 16, pk);
        }
        float sums[8];
#pragma unroll
        for (int u = 0; u < 4; ++u) f2_unpack(sums2[u], sums[2 * u], sums[2 * u + 1]);
        const float tile_sum = ((sums[0] + sums[1]) + (sums[2] + sums[3])) +
                               ((sums[4] + sums[5]) + (sums[6] + sums[7]));
        l_run = l_run * alpha + tile_sum;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar_pfull[t]);
        m_run = m_new;
        m_norm = m_use;
      }
      sc += n;
      gbase += it.nmax;
      if (!ok || n == 0) continue;
      // ------------------------------------------------------------ epilogue
      // O = O_acc / l, rounded to BF16, staged one 64-column chunk at a time in
      // this tile's slot; warp 3 writes it with a TMA store (rows past N are
      // clipped);
      // LSE = m * scale + ln(l).  The next item's first P V product, which
      // overwrites O_t, waits for this warpgroup's next P, so it cannot run
      // before O_t has been read here.
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_odone[t], oc & 1));
      if (!ok) break;
      ++oc;
      tc_fence_after();
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      const uint64_t il2 = f2_pack(inv_l, inv_l);
      if constexpr (C::kStagedOut) {
        for (int c = 0; c < C::kChunks && ok; ++c) {
          // The slot is free once the previous chunk's store has read it.
          if (es > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bar_epifree[t], (es - 1) & 1));
            if (!ok) break;
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t o[32];
            tmem_ld32(tO + c * 64 + h * 32, o);
            tmem_wait_ld();
            reg_fence(o);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float lo, hi;
              f2_unpack(mul2(f2_pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), il2),
                        lo, hi);
              pk[i] = pack_bf16x2(lo, hi);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
              st_shared_v4(aStage + sw128_offset(r, h * 4 + u), pk[4 * u], pk[4 * u + 1],
                           pk[4 * u + 2], pk[4 * u + 3]);
          }
          fence_proxy_async_smem();
          mbar_arrive(&bar_epifull[t]);  // warp 3 stores the chunk
          ++es;
        }
      } else {
        uint4* row = reinterpret_cast<uint4*>(out + ((size_t)it.bh * N + qi) * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_wait_ld();
          reg_fence(o);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float lo, hi;
            f2_unpack(mul2(f2_pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), il2),
                      lo, hi);
            pk[i] = pack_bf16x2(lo, hi);
          }
          if (qi < N) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              row[c * 4 + u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          }
        }
      }
      if (!ok) break;
      if (qi < N) lse[(size_t)it.bh * N + qi] = m_norm * (I8 ? scale * sq : scale) + logf(l_run);
#ifdef ATTN_TEST_HOOKS
      if (qi < N && g_hook_pbar_ones != nullptr && (size_t)it.bh * N + qi < g_hook_rows)
        atomicAdd(g_hook_pbar_ones + (size_t)it.bh * N + qi, n_ones);
#endif
    }
    if (!ok) set_fail(ATTN_ERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool CAUSAL, bool STABLE, bool I8 = false>
cudaError_t launch_fwd_impl(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& mv, const CUtensorMap& mo, void* o, float* lse,
                            float beta, cudaStream_t stream, const float* qs = nullptr,
                            const float* ks = nullptr) {
  using C = FwdCfg<D>;
  auto kernel = fwd_bf16_kernel<D, CAUSAL, STABLE, I8>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
  if (err != cudaSuccess) return err;
  const int BH = p.B * p.H;
  const int num_qt = ceil_div(p.N, 2 * kBlockM);
  const int total = BH * num_qt;
  // One CTA per SM (one fits: 512 TMEM columns, ~200 KB of shared memory);
  // without an SM count, one CTA per item.
  const int sms = device_sm_count();
  const int grid = sms > 0 ? std::min(total, sms) : total;
  const float scale_log2 = p.scale * 1.4426950408889634f;
  return launch_pdl(kernel, dim3(grid), dim3(kThreads), C::kSmemBytes, stream, mq, mk, mv, mo,
                    static_cast<uint16_t*>(o), lse, BH, p.N, num_qt, p.scale, scale_log2, beta, qs,
                    ks, n_pad(p.N));
}

}  // namespace

cudaError_t launch_fwd_bf16(const Problem& p, const void* q, const void* k, const void* v, void* o,
                            float* lse, cudaStream_t stream, float beta) {
  const int BH = p.B * p.H;
  CUtensorMap mq, mk, mv, mo;
  if (!make_tmap_bhnd(&mq, q, BH, p.N, p.d) || !make_tmap_bhnd(&mk, k, BH, p.N, p.d) ||
      !make_tmap_bhnd(&mv, v, BH, p.N, p.d) || !make_tmap_bhnd(&mo, o, BH, p.N, p.d))
    return cudaErrorInvalidValue;
  const bool st = beta > 0.f;  // beta <= 0: the plain kernel
#define ATTN_FWD_CASE(DD, CC, SS) \
  if (p.d == DD && (p.causal != 0) == CC && st == SS) \
    return launch_fwd_impl<DD, CC, SS>(p, mq, mk, mv, mo, o, lse, beta, stream);
  ATTN_FWD_CASE(128, true, false)
  ATTN_FWD_CASE(128, false, false)
  ATTN_FWD_CASE(64, true, false)
  ATTN_FWD_CASE(64, false, false)
  ATTN_FWD_CASE(128, true, true)
  ATTN_FWD_CASE(128, false, true)
  ATTN_FWD_CASE(64, true, true)
  ATTN_FWD_CASE(64, false, true)
#undef ATTN_FWD_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_int8_as_bf16(const Problem& p, const void* qc, const float* qs,
                                    const void* kc, const float* ks, const void* v, void* o,
                                    float* lse, cudaStream_t stream) {
  const int BH = p.B * p.H;
  CUtensorMap mq, mk, mv, mo;
  if (!make_tmap_bhnd(&mq, qc, BH, p.N, p.d) || !make_tmap_bhnd(&mk, kc, BH, p.N, p.d) ||
      !make_tmap_bhnd(&mv, v, BH, p.N, p.d) || !make_tmap_bhnd(&mo, o, BH, p.N, p.d))
    return cudaErrorInvalidValue;
  if (p.d == 128)
    return p.causal ? launch_fwd_impl<128, true, false, true>(p, mq, mk, mv, mo, o, lse, 0.f, stream, qs, ks)
                    : launch_fwd_impl<128, false, false, true>(p, mq, mk, mv, mo, o, lse, 0.f, stream, qs, ks);
  return p.causal ? launch_fwd_impl<64, true, false, true>(p, mq, mk, mv, mo, o, lse, 0.f, stream, qs, ks)
                  : launch_fwd_impl<64, false, false, true>(p, mq, mk, mv, mo, o, lse, 0.f, stream, qs, ks);
}

#ifdef ATTN_TEST_HOOKS
extern "C" ATTN_API int attn_testhook_pbar_counter(unsigned int* counts, unsigned long long rows) {
  cudaError_t e = cudaMemcpyToSymbol(g_hook_pbar_ones, &counts, sizeof(counts));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_hook_rows, &rows, sizeof(rows));
  return (int)e;
}

extern "C" ATTN_API int attn_testhook_stall(int on) {
  return (int)cudaMemcpyToSymbol(g_hook_stall, &on, sizeof(on));
}
#endif

cudaError_t read_and_clear_status_fwd(unsigned int* out, cudaStream_t stream) {
  static const unsigned int zero = 0;
  cudaError_t err = cudaMemcpyFromSymbolAsync(out, g_status_fwd, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
  if (err != cudaSuccess) return err;
  err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return err;
  err = cudaMemcpyToSymbolAsync(g_status_fwd, &zero, sizeof(unsigned int), 0,
                                cudaMemcpyHostToDevice, stream);
  if (err != cudaSuccess) return err;
  return cudaStreamSynchronize(stream);
}

}  // namespace attn
