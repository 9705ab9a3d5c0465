// tcgen05 tensor-core chunkwise Gated DeltaNet forward: bf16 q/k/v/out, fp32
// gates and state, dk = dv = 128, chunk C = 64.
//
// One cluster of two CTAs owns one (sequence, head) and walks its chunks in
// order (Nyysyyan, "Chunk Computation": chunks serial, tokens of a chunk
// parallel).  The work of a chunk splits into the part that does not depend on
// the running state and the part that does (myhz0606, "DeltaNet的Chunkwise
// Form推导", section 4.5: W and U depend only on the chunk's own k, v, beta):
//
// CTA 0, "WY" (three warpgroups on chunks j = w mod 3, one TMA producer warp):
//   K K^T                    tcgen05, M=128 (rows 64..127 unused)
//   A = strictly-lower(beta_i e^{g_i-g_j} k_i.k_j)          fp32 epilogue
//   T = (I + A)^{-1}         16x16 diagonal blocks, then block rows, fp32
//   W~^T = K^T (T diag(beta e^g))^T                        tcgen05
//   -W~^T (bf16) and T diag(beta) (hi/lo bf16) go to CTA 1 by DSMEM bulk copies,
//   in chunk order, into two hand-off slots.
// CTA 1, "state" (three warpgroups, a TMA producer warp and an MMA warp):
//   chain (serial):  SW = U^T + S (-W~^T) = delta^T;  S <- e^{g_last} S + delta~^T K
//                    (S accumulates in TMEM; delta feeds the MMAs from TMEM)
//   MMA warp:        U^T = V^T (T diag(beta))^T into SW ahead of the chain;
//                    O += delta^T P^T onto the output accumulator
//   aux P (ahead):   Q K^T (M=64) -> P' = lower(q_t.k_j e^{-g_j}) (factored decay),
//                    or P = lower(q_t.k_j e^{g_t-g_j}) and Q <- diag(e^g) Q in place
//   aux O (behind):  o_t = e^{g_t} O_t (factored) or O_t -> out for chunk j - 1, then
//                    O = S Q^T (j) (S as hi + lo) into the emptied accumulator once the
//                    chain has queued its S W~^T
// The factored form keeps the output accumulator in the frame of e^{-g_t}: the
// state part S q_t and every in-chunk term e^{-g_j} (q_t.k_j) delta_j share that
// factor, which aux O multiplies back.  It is used when the chunk's total decay
// e^{g_last} is above 2^-80, so that e^{-g_j} stays inside the fp32 range.
//
// Linear mode (beta == NULL; Nyysyyan, "Mamba2" and "Linear attention"): the
// erase strength is 0 and the write strength 1, so A = 0, T = I, W~ = 0 and
// delta = U = V exactly, independent of the state: S_t = alpha_t S_{t-1} + v_t k_t^T.
// gdn_tc_linear_kernel runs the state CTA alone (one CTA per (sequence, head)); its
// chain is the state update and the S epilogue, and between them it makes the next
// chunk's delta = V and delta~ = V diag(e^{g_last-g}) from the V tile into one of two
// TMEM buffers while the state update runs; the MMA warp's delta^T P^T reads delta from
// there.  The results are those of the delta-rule pipeline with these factors, bit for
// bit (its extra products are exact zeros).
//
// W~ uses the decayed triangular factor (W~_i = gamma_i w_i with the WY
// recursion of Nyysyyan's "Gated-DeltaNet" section); then
// delta = U - W~ S^T and the chunk's states and outputs follow from the unrolled
// recurrence.
//
// Precision: operands are bf16, accumulators fp32.  T, delta, the decayed delta
// (delta~ = delta diag(e^{g_last-g})) and P are carried as two bf16 terms
// (hi = bf16(x), lo = bf16(x - hi)) and multiplied as hi*hi + hi*lo + lo*hi, or
// hi + lo against an exact bf16 operand (K, V, Q).  The state enters S Q^T (the
// outputs' read of the carried state) as hi + lo as well, so that outputs dominated by
// a decaying carried state keep the rounding of a 16-bit mantissa; it enters S W~^T,
// and W~ enters, as single bf16 terms (and Q scaled by e^{g} in the strong-decay form).
// The running state itself stays fp32 (in TMEM).
//
// Synchronisation (mbarriers; "phase j" completes once per chunk j):
//   WY:    kv_full[s]  (TMA bytes + producer arrive)   kv_empty[s] (WG after its MMAs)
//          wg_mma[w]   (MMA commits of warpgroup w)
//          hand_empty[b] (arrived by CTA 1 once chunk j's slot has been read)
//   state: qk_full[s]; qk_empty[s] (chain after its state update + aux P after its
//          Q K^T); hand_full[b] (bulk-copy bytes); bar_u[b], bar_dp[b] (MMA warp
//          commits); bar_sq[b] (aux O's commit); bar_c, bar_ds (chain commits);
//          sw_issued, delta_ready[b] (chain arrives); p_full[b] (aux P);
//          o_empty[b] (aux O); bar_qk (aux P's commit).  Per-parity pairs [b] advance
//          once per two chunks, so no waiter can find its barrier two phases ahead.
// "Empty" barriers are waited with parity ^ 1 so that their first wait passes.
// Every wait is bounded; a wait that gives up records a code in a device status
// word, every role of both CTAs leaves its loop, and both CTAs still meet at the
// final cluster barrier.
//
// Instruction footprint matters here: with every SM of a GPC running this
// kernel, instruction-cache misses queue at the GPC level, so the per-chunk
// loops favour rolled loops and one out-of-line polling routine over unrolled
// code.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "gdn_internal.h"
#include "tc_common.cuh"

namespace gdn {

__device__ int g_tc_status = 0;

namespace {

using namespace ptx;

constexpr int kThreads = 448;  // 3 warpgroups, a TMA producer warp and (state CTA) an MMA warp
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;

// ---- CTA 0 ("WY") shared memory ----
constexpr int WY_KV = 0;                 // 3 stages x 16 KB: K p0 | K p1 (8 KB each)
constexpr int WY_STAGE = 16384;
constexpr int WY_NST = 3;
constexpr int WY_SCR = WY_NST * WY_STAGE;  // 49152: per-warpgroup scratch
constexpr int WY_SCR_BYTES = 53248;
constexpr int WY_NWG = 3;                  // warpgroup w takes chunks j = w (mod 3), stage w
//   A/T fp32 [64][68] @0 | X fp32 [3][256] @17408 | Tw hi @20480 | Tw lo @28672
//   | Tu hi @36864 | Tu lo @45056
constexpr int LDA = 68;
constexpr int SC_X = 17408, SC_TWH = 20480, SC_TWL = 28672, SC_TUH = 36864, SC_TUL = 45056;
constexpr int WY_DER = WY_SCR + WY_NWG * WY_SCR_BYTES;  // [3 stages][G, EG, BG, BE, EN][64] fp32
constexpr int WY_DER_STAGE = 5 * 64;                // floats per stage
constexpr int WY_FLAG = WY_DER + WY_NST * WY_DER_STAGE * 4;  // [3] int: factored decay allowed
constexpr int WY_BAR = WY_FLAG + 64;
constexpr int WY_MISC = WY_BAR + 128;
constexpr int WY_USED = WY_MISC + 64;

// ---- CTA 1 ("state") shared memory ----
constexpr int ST_QK = 0;                 // 2 stages x 48 KB: per dk panel p (16 KB): Q rows, K rows
constexpr int ST_STAGE = 49152;          //   (8 KB each); then V p0 @32 KB, V p1 @40 KB
constexpr int ST_V = 32768;
constexpr int ST_NST = 2;
constexpr int ST_HS = ST_NST * ST_STAGE;  // 98304: 2 handoff slots of 32 KB each:
constexpr int HS_BYTES = 32768;          //   -W~^T bf16 [128 dk][64 tok] (MN-major B) @0,
constexpr int HS_TUH = 16384, HS_TUL = 24576;  // T diag(beta) hi, lo bf16 [64][64] (K-major B)
constexpr int ST_PS = ST_HS + 2 * HS_BYTES;  // 163840: 2 P slots of 16 KB: hi @0, lo @8 KB,
constexpr int PS_BYTES = 16384;          //   bf16 [64 t][64 j], K-major B operand
constexpr int ST_SB = ST_PS + 2 * PS_BYTES;  // 196608: S bf16 [128 dv][128 dk], 2 K panels
constexpr int ST_DER = ST_SB + 32768;    // [2 stages][GN, EG, ED][64] fp32 (GN: e^{-g}, or g)
constexpr int ST_DER_STAGE = 3 * 64;
constexpr int ST_FLAG = ST_DER + ST_NST * ST_DER_STAGE * 4;  // [2] int
constexpr int ST_BAR = ST_FLAG + 64;
constexpr int ST_MISC = ST_BAR + 192;
constexpr int ST_USED = ST_MISC + 64;
// The output tile of a chunk is staged in the chunk's P slot once delta^T P^T has
// read it (token t at t * 256 bytes), then copied out with 16-byte stores.

constexpr int SMEM_USED = WY_USED > ST_USED ? WY_USED : ST_USED;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack for aligning the base
static_assert(SC_TUL + 8192 <= WY_SCR_BYTES, "WY scratch");
static_assert(WY_NWG == WY_NST, "one K stage per WY warpgroup");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// barrier slots (8 bytes each)
enum WyBar { WB_KV_FULL = 0, WB_KV_EMPTY = 3, WB_MMA = 6, WB_HE = 9, WB_COUNT = 11 };
static_assert(WB_COUNT * 8 <= WY_MISC - WY_BAR, "WY barriers");
enum StBar {
  SB_QK_FULL = 0, SB_QK_EMPTY = 2, SB_HF = 4, SB_C = 6, SB_DS = 7, SB_QKM = 8, SB_DP = 9,
  SB_PF = 11, SB_U = 13, SB_DR = 15, SB_SWI = 17, SB_SQ = 18, SB_PE = 20,
  SB_COUNT = 22
};
static_assert(SB_COUNT * 8 <= ST_MISC - ST_BAR, "state barriers");

// TMEM columns.  WY: per warpgroup w at 128*w: K K^T 0, W~^T 64.
constexpr uint32_t WT_KK = 0, WT_W = 64, WT_WG = 128;
// state: S 0..127, U^T + S(-W~^T) 128 (one accumulator: U^T(j + 1) is issued only after
// the delta epilogue of chunk j has read it), outputs of chunk j at 192 + 64 (j % 2),
// QK 320, delta hi 384, delta lo 416, delta~ hi 448, delta~ lo 480 (packed bf16 pairs,
// A operands).  The delta rule puts the lo term of the state operand of S Q^T (packed
// bf16 pairs, an A operand) at 320 and accumulates Q K^T (j) in output accumulator j % 2
// instead, which is free from the drain of chunk j - 2 until S Q^T (j).
constexpr uint32_t TT_S = 0, TT_SW = 128, TT_O = 192, TT_QK = 320, TT_SLO = 320, TT_DH = 384,
                   TT_DL = 416, TT_DSH = 448, TT_DSL = 480;
constexpr uint32_t TM_COLS = 512;
// Linear mode: delta (= V, exact bf16 pairs) and delta~ (hi / lo) of chunk j in buffer
// j % 2.  Buffer 0 is the delta-rule columns; buffer 1 takes the U/SW accumulator (this
// mode has no U and no S W~^T) and the delta lo columns (delta = V needs no lo term).
__device__ __forceinline__ uint32_t tl_dh(int b) { return b ? TT_SW : TT_DH; }
__device__ __forceinline__ uint32_t tl_dsh(int b) { return b ? TT_SW + 32 : TT_DSH; }
__device__ __forceinline__ uint32_t tl_dsl(int b) { return b ? TT_DL : TT_DSL; }


// The lo term of 32 state columns (32p .. 32p + 31 of row `row`), bf16(x - bf16(x)), as
// packed pairs into the state-lo columns of TMEM: the K = 128 A operand of S lo Q^T.
__device__ __forceinline__ void state_lo_to_tmem(uint32_t tq, int p, const float* v) {
  uint32_t lo[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    uint32_t hi;
    split2(v[2 * e], v[2 * e + 1], hi, lo[e]);
  }
  tmem_st16(tq + TT_SLO + 16 * p, lo);
}
// S Q^T with the state as two bf16 terms: S hi (shared memory, K-major, two 64-column
// panels) and S lo (TMEM, packed pairs), against Q (K-major, two panels), then commit.
__device__ __noinline__ void sq_hilo_commit(uint32_t d, uint64_t a_hi, uint32_t a_lo_tmem,
                                            uint64_t b, uint32_t id, uint64_t* bar) {
  tc_fence_after();
  mma_k128<false>(d, a_hi, 16384 >> 4, b, 16384 >> 4, id, 0);
#pragma unroll 1
  for (int p = 0; p < 2; ++p) {
    const uint64_t bp = b + (uint64_t)(p * (16384 >> 4));
#pragma unroll
    for (int k = 0; k < 4; ++k)
      mma_bf16_ta(d, a_lo_tmem + 32 * p + 8 * k, bp + kStepK * k, id, 1u);
  }
  mma_commit(bar);
}

// ============================================================ CTA 0: WY ======
__device__ __forceinline__ void run_wy(uint8_t* sm, uint32_t tmem, const CUtensorMap* tm_k,
                       const float* __restrict__ log_alpha, const float* __restrict__ beta,
                       const Unit& u, int H, volatile int* abort_flag) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + WY_BAR);
  float* der_all = reinterpret_cast<float*>(sm + WY_DER);
  int* flags = reinterpret_cast<int*>(sm + WY_FLAG);

  if (warp == kProducerWarp) {
    // ---------------- producer: K tiles by TMA, gate factors ----------------
    int issued = 0;
    GateLoad next = load_gates(log_alpha, beta, u, H, 0, lane);
    #pragma unroll 1
    for (int j = 0; j < u.nc; ++j) {
      const int s = j % WY_NST;
      const uint32_t use = j / WY_NST;
      const GateLoad cur = next;
      next = load_gates(log_alpha, beta, u, H, j + 1, lane);  // in flight during the wait
      if (warp_wait_fails(&bars[WB_KV_EMPTY + s], (use & 1) ^ 1, abort_flag, false))
        break;
      uint8_t* st = sm + WY_KV + s * WY_STAGE;
      const int r = (int)(u.row0 + (long long)j * kC);
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[WB_KV_FULL + s], 2 * 8192);
        tma_load_3d(st, tm_k, &bars[WB_KV_FULL + s], 0, u.h, r);
        tma_load_3d(st + 8192, tm_k, &bars[WB_KV_FULL + s], 64, u.h, r);
      }
      issued = j + 1;
      float g0, g1, tot;
      scan_gates(cur, lane, g0, g1, tot);
      // write strengths b (beta, or 1 in the linear mode) and erase strengths
      // (beta, or 0 in the linear mode, which makes A = 0, T = I and W~ = 0)
      const float b0 = cur.b0, b1 = cur.b1;
      const float er0 = beta ? b0 : 0.f, er1 = beta ? b1 : 0.f;
      float* der = der_all + s * WY_DER_STAGE;  // G, EG, BG, BE, EN
      const float e0 = ex2(g0), e1 = ex2(g1);
      der[lane] = g0;                 der[lane + 32] = g1;
      der[64 + lane] = e0;            der[64 + lane + 32] = e1;
      der[128 + lane] = er0 * e0;     der[128 + lane + 32] = er1 * e1;
      der[192 + lane] = b0;           der[192 + lane + 32] = b1;
      der[256 + lane] = ex2(-g0);     der[256 + lane + 32] = ex2(-g1);
      if (lane == 0) flags[s] = (-tot < kMaxFactoredDecayLog2) ? 1 : 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[WB_KV_FULL + s]);
    }
    // copies still in flight must land before the CTA can leave
    #pragma unroll 1
    for (int j = issued - WY_NST; j < issued; ++j)
      if (j >= 0) (void)mbar_wait(&bars[WB_KV_FULL + j % WY_NST], (j / WY_NST) & 1, 100000000ull);
    return;
  }
  if (warp >= 4 * WY_NWG) return;

  // ---------------- warpgroups: w takes chunks j = w (mod 3) ----------------
  const int w = warp >> 2;
  const int wtid = tid & 127;
  const int q4 = warp & 3;
  const int row = q4 * 32 + lane;
  const uint32_t nb = 1 + w;  // named barrier of this warpgroup (1..3); 4 + w: half of it
  volatile int* ticket = reinterpret_cast<volatile int*>(sm + WY_MISC + 8);
  uint8_t* scr = sm + WY_SCR + w * WY_SCR_BYTES;
  float* Am = reinterpret_cast<float*>(scr);
  float* Xs = reinterpret_cast<float*>(scr + SC_X);
  const uint32_t tw = tmem + w * WT_WG;
  const uint32_t tq = tw + ((uint32_t)(q4 * 32) << 16);
  uint32_t mph = 0;

#define WY_WAIT(bar, par, cl) \
  if (group_waits_fail(abort_flag, nb, 128, (bar), (par), (cl))) break;

  #pragma unroll 1
  for (int j = w; j < u.nc; j += WY_NWG) {
    const int s = j % WY_NST;
    uint8_t* st = sm + WY_KV + s * WY_STAGE;
    const float* G = der_all + s * WY_DER_STAGE;
    const float* BG = G + 128;
    const float* BE = G + 192;
    const float* EN = G + 256;
    WY_WAIT(&bars[WB_KV_FULL + s], (j / WY_NST) & 1, false);
    const bool factored = flags[s] != 0;

    // ---- K K^T (rows 0..63 of the M=128 accumulator) ----
    if (wtid == 0) {
      tc_fence_after();
      const uint32_t id = idesc_bf16(128, 64, 0, 0);
      const uint64_t dkk = desc_k(st, 0, 8192);
      mma_k128<false>(tw + WT_KK, dkk, 8192 >> 4, dkk, 8192 >> 4, id, 0);
      mma_commit(&bars[WB_MMA + w]);
    }
    // the bulk copy of this warpgroup's previous chunk reads the scratch that A is
    // about to overwrite; it has had the K K^T round trip to finish
    if (wtid == 0) bulk_wait_read_all();
    WY_WAIT(&bars[WB_MMA + w], mph, false);
    mph ^= 1;
    tc_fence_after();

    // ---- A = strictly-lower(beta_i e^{g_i - g_j} k_i.k_j), fp32 ----
    if (q4 < 2) {
      if (factored)
        wy_epi_a<true>(tq + WT_KK, Am + row * LDA, row, BG[row], 0.f, EN);
      else
        wy_epi_a<false>(tq + WT_KK, Am + row * LDA, row, beta ? BE[row] : 0.f, G[row], G);
    }
    named_sync(nb, 128);

    // ---- T = (I + A)^{-1} in place: diagonal 16x16 blocks ----
    if (wtid < 64) {
      const int b = wtid >> 4, c = wtid & 15;
      const float* Ab = Am + (16 * b) * LDA + 16 * b;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float acc = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int m = 0; m < r; ++m) acc = fmaf(-Ab[r * LDA + m], x[m], acc);
        x[r] = acc;
      }
      named_sync(4 + w, 64);
      float* Tb = Am + (16 * b) * LDA + 16 * b + c;
#pragma unroll
      for (int r = 0; r < 16; ++r) Tb[r * LDA] = x[r];
    }
    named_sync(nb, 128);
    // ---- block rows: X = sum_k A_{ib,k} T_{k,jb}; T_{ib,jb} = -T_{ib,ib} X ----
    // each thread owns 1 x 4 strips of the 16 x 16 blocks
#pragma unroll 1
    for (int ib = 1; ib < 4; ++ib) {
      // strip e covers block jb = e / 64 (1 x 4 of its 16 x 16).  Thread t takes strip
      // t, and in block row 3 threads t >= 64 also take strip t + 64, so every thread
      // of row 3 does three block products (jb 0: 3; jb 1 + jb 2: 2 + 1).
      for (int e = wtid; e < ib * 64; e += (ib == 3) ? (wtid >= 64 ? 64 : 192) : 128) {
        const int jb = e >> 6, r = (e >> 2) & 15, cq = e & 3;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        const float* arow = Am + (16 * ib + r) * LDA;
#pragma unroll 1
        for (int kb = jb; kb < ib; ++kb) {
#pragma unroll
          for (int m4 = 0; m4 < 4; ++m4) {
            const float4 a = ld4(arow + 16 * kb + 4 * m4);
            const float* tr = Am + (16 * kb + 4 * m4) * LDA + 16 * jb + 4 * cq;
            const float4 t0 = ld4(tr), t1 = ld4(tr + LDA), t2 = ld4(tr + 2 * LDA),
                         t3 = ld4(tr + 3 * LDA);
            a0 = fmaf(a.x, t0.x, a0); a1 = fmaf(a.x, t0.y, a1); a2 = fmaf(a.x, t0.z, a2); a3 = fmaf(a.x, t0.w, a3);
            a0 = fmaf(a.y, t1.x, a0); a1 = fmaf(a.y, t1.y, a1); a2 = fmaf(a.y, t1.z, a2); a3 = fmaf(a.y, t1.w, a3);
            a0 = fmaf(a.z, t2.x, a0); a1 = fmaf(a.z, t2.y, a1); a2 = fmaf(a.z, t2.z, a2); a3 = fmaf(a.z, t2.w, a3);
            a0 = fmaf(a.w, t3.x, a0); a1 = fmaf(a.w, t3.y, a1); a2 = fmaf(a.w, t3.z, a2); a3 = fmaf(a.w, t3.w, a3);
          }
        }
        st4(Xs + jb * 256 + r * 16 + 4 * cq, a0, a1, a2, a3);
      }
      named_sync(nb, 128);
      for (int e = wtid; e < ib * 64; e += (ib == 3) ? (wtid >= 64 ? 64 : 192) : 128) {
        const int jb = e >> 6, r = (e >> 2) & 15, cq = e & 3;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        const float* trow = Am + (16 * ib + r) * LDA + 16 * ib;
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4) {
          const float4 a = ld4(trow + 4 * m4);
          const float* xr = Xs + jb * 256 + (4 * m4) * 16 + 4 * cq;
          const float4 t0 = ld4(xr), t1 = ld4(xr + 16), t2 = ld4(xr + 32), t3 = ld4(xr + 48);
          a0 = fmaf(a.x, t0.x, a0); a1 = fmaf(a.x, t0.y, a1); a2 = fmaf(a.x, t0.z, a2); a3 = fmaf(a.x, t0.w, a3);
          a0 = fmaf(a.y, t1.x, a0); a1 = fmaf(a.y, t1.y, a1); a2 = fmaf(a.y, t1.z, a2); a3 = fmaf(a.y, t1.w, a3);
          a0 = fmaf(a.z, t2.x, a0); a1 = fmaf(a.z, t2.y, a1); a2 = fmaf(a.z, t2.z, a2); a3 = fmaf(a.z, t2.w, a3);
          a0 = fmaf(a.w, t3.x, a0); a1 = fmaf(a.w, t3.y, a1); a2 = fmaf(a.w, t3.z, a2); a3 = fmaf(a.w, t3.w, a3);
        }
        st4(Am + (16 * ib + r) * LDA + 16 * jb + 4 * cq, -a0, -a1, -a2, -a3);
      }
      named_sync(nb, 128);
    }

    // ---- T diag(beta e^g), T diag(beta) as bf16 hi/lo B operands ----
#pragma unroll 1
    for (int it0 = 0; it0 < 512; it0 += 128) {
      const int it = it0 + wtid;
      const int i = it >> 3, jc = (it & 7) * 8;
      const float4 ta = ld4(Am + i * LDA + jc), tb = ld4(Am + i * LDA + jc + 4);
      const float tv[8] = {ta.x, ta.y, ta.z, ta.w, tb.x, tb.y, tb.z, tb.w};
      const float4 bg0 = ld4(BG + jc), bg1 = ld4(BG + jc + 4);
      const float4 be0 = ld4(BE + jc), be1 = ld4(BE + jc + 4);
      const float bgv[8] = {bg0.x, bg0.y, bg0.z, bg0.w, bg1.x, bg1.y, bg1.z, bg1.w};
      const float bev[8] = {be0.x, be0.y, be0.z, be0.w, be1.x, be1.y, be1.z, be1.w};
      float twv[8], tuv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float t = (jc + e <= i) ? tv[e] : 0.f;
        twv[e] = t * bgv[e];
        tuv[e] = t * bev[e];
      }
      st_sw128_8_split(scr + SC_TWH, scr + SC_TWL, i, jc, 64, twv);
      st_sw128_8_split(scr + SC_TUH, scr + SC_TUL, i, jc, 64, tuv);
    }
    fence_async_smem();
    tc_fence_before();
    named_sync(nb, 128);

    // ---- W~^T = K^T Tw^T (hi + lo); U is formed by the state CTA from Tu ----
    if (wtid == 0) {
      tc_fence_after();
      const uint32_t id = idesc_bf16(128, 64, 1, 0);
      const uint64_t da = desc_mn(st, 0, 8192);
      const uint64_t dh = desc_k(scr + SC_TWH, 0, 8192), dl = desc_k(scr + SC_TWL, 0, 8192);
      mma_k64<false, false, false>(tw + WT_W, da, 0, dh, id, 0);
      mma_k64<false, false, false>(tw + WT_W, da, 0, dl, id, 1);
      mma_commit(&bars[WB_MMA + w]);
    }
    WY_WAIT(&bars[WB_MMA + w], mph, false);
    mph ^= 1;
    tc_fence_after();
    if (wtid == 0) mbar_arrive(&bars[WB_KV_EMPTY + s]);  // K of this stage is consumed

    // ---- hand chunk j to the state CTA (slot j % 2): -W~^T staged at scratch 0, and
    //      Tu hi / lo straight from scratch (they already have the slot's layout) ----
    const int slot = j & 1;
    const uint32_t huse = (uint32_t)(j >> 1);
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
      uint32_t rw[32];
      tmem_ld32(tq + WT_W + 32 * hh, rw);
      tmem_wait_ld();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t wv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          wv[e] = pack_bf16(-__uint_as_float(rw[8 * q + 2 * e]),
                            -__uint_as_float(rw[8 * q + 2 * e + 1]));
        st_shared_v4(smem_u32(scr + sw128_offset(row, 32 * hh + 8 * q, 128)), wv[0], wv[1], wv[2],
                     wv[3]);
      }
    }
    fence_async_smem();
    tc_fence_before();
    // Hand-offs leave in chunk order: when chunk j waits for its slot, chunk j - 4 has
    // been consumed, so the slot's barrier is at most one phase behind and its parity
    // is unambiguous.
    {
      const bool ok_ = (wtid != 0) || wait_ticket(ticket, j, abort_flag);
      if (named_sync_or(nb, 128, !ok_ || *abort_flag != 0)) break;
    }
    WY_WAIT(&bars[WB_HE + slot], (huse & 1) ^ 1, true);
    if (wtid == 0) {
      const uint32_t rb = map_shared(smem_u32(sm + ST_BAR + 8 * (SB_HF + slot)), 1);
      const uint32_t rs = map_shared(smem_u32(sm + ST_HS + slot * HS_BYTES), 1);
      mbar_arrive_expect_tx_remote(rb, HS_BYTES);
      bulk_copy_to_cluster(rs, scr, 16384, rb);
      bulk_copy_to_cluster(rs + HS_TUH, scr + SC_TUH, 16384, rb);
      bulk_commit();
      *ticket = j + 1;
    }
  }
#undef WY_WAIT
  if (wtid == 0) bulk_wait_all();  // every copy this warpgroup issued has landed
}

// One quarter (tokens 16*qq .. 16*qq + 15) of the delta epilogue of the state CTA:
// the accumulator t_sw already holds delta^T = U^T + S(-W~^T); write delta and
// delta~ = delta e^{g_last - g} to TMEM as hi / lo bf16 pairs (the A operands of
// the next MMAs).
__device__ __forceinline__ void delta_quarter(uint32_t tq, uint32_t t_sw, const float* ED, int qq) {
  uint32_t r[16];
  tmem_ld16(tq + t_sw + 16 * qq, r);
  tmem_wait_ld();
  uint32_t dh[8], dl[8], sh[8], sl[8];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float4 ea = ld4(ED + 16 * qq + 8 * q), eb = ld4(ED + 16 * qq + 8 * q + 4);
    const float ev[8] = {ea.x, ea.y, ea.z, ea.w, eb.x, eb.y, eb.z, eb.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float d0 = __uint_as_float(r[8 * q + 2 * e]);
      const float d1 = __uint_as_float(r[8 * q + 2 * e + 1]);
      split2(d0, d1, dh[4 * q + e], dl[4 * q + e]);
      split2(d0 * ev[2 * e], d1 * ev[2 * e + 1], sh[4 * q + e], sl[4 * q + e]);
    }
  }
  tmem_st8(tq + TT_DH + 8 * qq, dh);
  tmem_st8(tq + TT_DL + 8 * qq, dl);
  tmem_st8(tq + TT_DSH + 8 * qq, sh);
  tmem_st8(tq + TT_DSL + 8 * qq, sl);
}

// Linear mode: row `row` (a dv index) of delta^T = V^T as exact bf16 pairs and of
// delta~^T = V^T diag(e^{g_last - g}) as hi / lo pairs, for the chunk's tokens, read
// from the V tile (two 64-column panels, 128-byte swizzle) into TMEM buffer b.  Tokens
// from lc on belong to no sequence of this unit and write nothing (zeros).
__device__ __forceinline__ void lin_delta(uint32_t tq, const uint8_t* vt, const float* ED,
                                          int row, int b, int lc) {
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {  // tokens 32h .. 32h + 31, two per TMEM column
    uint32_t dh[16], sh[16], sl[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int t = 32 * h + 2 * c;
      const uint32_t v0 = t < lc ? *reinterpret_cast<const uint16_t*>(vt + sw128_offset(t, row, 64)) : 0u;
      const uint32_t v1 =
          t + 1 < lc ? *reinterpret_cast<const uint16_t*>(vt + sw128_offset(t + 1, row, 64)) : 0u;
      dh[c] = v0 | (v1 << 16);
      split2(__uint_as_float(v0 << 16) * ED[t], __uint_as_float(v1 << 16) * ED[t + 1], sh[c], sl[c]);
    }
    tmem_st16(tq + tl_dh(b) + 16 * h, dh);
    tmem_st16(tq + tl_dsh(b) + 16 * h, sh);
    tmem_st16(tq + tl_dsl(b) + 16 * h, sl);
  }
}

// ========================================================= CTA 1: state ======
template <bool LINEAR>
__device__ __forceinline__ void run_state(uint8_t* sm, uint32_t tmem, const CUtensorMap* tm_q,
                          const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                          const float* __restrict__ log_alpha,
                          const float* __restrict__ beta, const float* __restrict__ S0,
                          __nv_bfloat16* __restrict__ out, float* __restrict__ S_final,
                          const Unit& u, int H, volatile int* abort_flag) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + ST_BAR);
  float* der_all = reinterpret_cast<float*>(sm + ST_DER);
  int* flags = reinterpret_cast<int*>(sm + ST_FLAG);

  if (warp == kProducerWarp) {
    // ---------------- producer: Q, K, V tiles by TMA, gate factors ----------------
    int issued = 0;
    GateLoad next = load_gates(log_alpha, beta, u, H, 0, lane);
    #pragma unroll 1
    for (int j = 0; j < u.nc; ++j) {
      const int s = j % ST_NST;
      const uint32_t use = j / ST_NST;
      const GateLoad cur = next;
      next = load_gates(log_alpha, beta, u, H, j + 1, lane);  // in flight during the wait
      if (warp_wait_fails(&bars[SB_QK_EMPTY + s], (use & 1) ^ 1, abort_flag, false))
        break;
      uint8_t* st = sm + ST_QK + s * ST_STAGE;
      const int r = (int)(u.row0 + (long long)j * kC);
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[SB_QK_FULL + s], 6 * 8192);
        tma_load_3d(st, tm_q, &bars[SB_QK_FULL + s], 0, u.h, r);
        tma_load_3d(st + 8192, tm_k, &bars[SB_QK_FULL + s], 0, u.h, r);
        tma_load_3d(st + 16384, tm_q, &bars[SB_QK_FULL + s], 64, u.h, r);
        tma_load_3d(st + 24576, tm_k, &bars[SB_QK_FULL + s], 64, u.h, r);
        tma_load_3d(st + ST_V, tm_v, &bars[SB_QK_FULL + s], 0, u.h, r);
        tma_load_3d(st + ST_V + 8192, tm_v, &bars[SB_QK_FULL + s], 64, u.h, r);
      }
      issued = j + 1;
      float g0, g1, tot;
      scan_gates(cur, lane, g0, g1, tot);
      const bool factored = -tot < kMaxFactoredDecayLog2;
      float* der = der_all + s * ST_DER_STAGE;  // GN (e^{-g} or g), EG, ED
      der[lane] = factored ? ex2(-g0) : g0;
      der[lane + 32] = factored ? ex2(-g1) : g1;
      der[64 + lane] = ex2(g0);         der[64 + lane + 32] = ex2(g1);
      der[128 + lane] = ex2(tot - g0);  der[128 + lane + 32] = ex2(tot - g1);
      if (lane == 0) flags[s] = factored ? 1 : 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[SB_QK_FULL + s]);
    }
    #pragma unroll 1
    for (int j = issued - ST_NST; j < issued; ++j)
      if (j >= 0) (void)mbar_wait(&bars[SB_QK_FULL + j % ST_NST], (j / ST_NST) & 1, 100000000ull);
    return;
  }
  if (LINEAR && warp == kMmaWarp) {
    // ------------- MMA warp, linear mode: delta^T P^T (j) = V^T (P hi + P lo) -------------
    // once the chain has made delta (j), aux P has published P (j) and S Q^T (j) has
    // completed
    int nd = 0;
    uint64_t t_idle = globaltimer_ns();
    #pragma unroll 1
    while (nd < u.nc) {
      const int j = nd;
      if (mbar_test(&bars[SB_DR + (j & 1)], (j >> 1) & 1, false) &&
          mbar_test(&bars[SB_PF + (j & 1)], (j >> 1) & 1, false) &&
          mbar_test(&bars[SB_SQ + (j & 1)], (j >> 1) & 1, false)) {
        ++nd;
        if (lane == 0) {
          tc_fence_after();
          const uint8_t* ps = sm + ST_PS + (j & 1) * PS_BYTES;
          const uint32_t id = idesc_bf16(128, 64, 0, 0);
          const uint64_t ph = desc_k(ps, 0, 8192), pl = desc_k(ps + 8192, 0, 8192);
          const uint32_t d = tmem + TT_O + 64 * (j & 1), a = tmem + tl_dh(j & 1);
          mma_k64<true, false, false>(d, 0, a, ph, id, 1);
          mma_k64<true, false, false>(d, 0, a, pl, id, 1);
          mma_commit(&bars[SB_DP + (j & 1)]);
        }
        __syncwarp();
        t_idle = globaltimer_ns();
      } else if (*abort_flag != 0) {
        break;
      } else if (globaltimer_ns() - t_idle > kWaitNs) {
        atomicOr((int*)abort_flag, ST_WAIT);
        break;
      }
    }
    return;
  }
  if (warp == kMmaWarp) {
    // ------------- MMA warp: the tensor-core work that is not on the chain's path -------------
    // U^T = V^T Tu^T (j + 1) goes in behind the chain's state update (j), into the U/SW
    // accumulator (which the chain's delta epilogue of j has read by then), ahead of
    // delta^T P^T (j); S Q^T is issued by aux O and Q K^T by
    // aux P, so that the issue work is spread over three warp schedulers.  Each kind is
    // issued in chunk order; the warp polls (non-blocking tests), U first.
    int nu = 0, ns = 0, nd = 0;  // next U, S Q^T, delta^T P^T
    uint64_t t_idle = globaltimer_ns();
    #pragma unroll 1
    while (nd < u.nc) {
      int kind = -1;
      if (nu < u.nc) {  // U(i) goes in behind the state update of i - 1
        const int i = nu;
        if ((i == 0 || mbar_test(&bars[SB_DR + ((i - 1) & 1)], ((i - 1) >> 1) & 1, false)) &&
            mbar_test(&bars[SB_QK_FULL + i % ST_NST], (i / ST_NST) & 1, false) &&
            mbar_test(&bars[SB_HF + (i & 1)], (i >> 1) & 1, true))
          kind = 0;
      }
      if (kind < 0 && ns < u.nc) {
        // S Q^T (i) starts output accumulator i % 2 once the chain has queued S W~^T (i),
        // which reads the same bf16 S (and waited for the chunk's stage), and aux P has
        // published P (i): it read its Q K^T out of that accumulator (and, in the
        // strong-decay form, scaled Q)
        const int i = ns;
        if (mbar_test(&bars[SB_SWI], i & 1, false) &&
            mbar_test(&bars[SB_PF + (i & 1)], (i >> 1) & 1, false))
          kind = 1;
      }
      if (kind < 0 && nd < ns && (nu > nd + 1 || nu == u.nc)) {
        // delta of chunk j in TMEM; S Q^T (j), issued before by this thread into the same
        // accumulator, runs first; U^T (j + 1) goes into the tensor pipe first
        const int j = nd;
        if (mbar_test(&bars[SB_DR + (j & 1)], (j >> 1) & 1, false)) kind = 2;
      }
      const bool did = kind >= 0;
      if (did) {
        if (kind == 0) {
          const int i = nu++;
          if (lane == 0) {  // U^T(i) = V^T Tu^T (hi + lo) into the U/SW accumulator
            tc_fence_after();
            uint8_t* stg = sm + ST_QK + (i % ST_NST) * ST_STAGE;
            uint8_t* hs = sm + ST_HS + (i & 1) * HS_BYTES;
            const uint32_t id_u = idesc_bf16(128, 64, 1, 0);
            const uint32_t d = tmem + TT_SW;
            const uint64_t dv = desc_mn(stg + ST_V, 0, 8192);
            mma_k64<false, false, false>(d, dv, 0, desc_k(hs + HS_TUH, 0, 8192), id_u, 0);
            mma_k64<false, false, false>(d, dv, 0, desc_k(hs + HS_TUL, 0, 8192), id_u, 1);
            mma_commit(&bars[SB_U + (i & 1)]);
          }
        } else if (kind == 1) {
          const int i = ns++;
          if (lane == 0)  // O = S Q^T (i), S as hi (shared memory) + lo (TMEM)
            sq_hilo_commit(tmem + TT_O + 64 * (i & 1), desc_k(sm + ST_SB, 0, 16384),
                           tmem + TT_SLO, desc_k(sm + ST_QK + (i % ST_NST) * ST_STAGE, 0, 16384),
                           idesc_bf16(128, 64, 0, 0), &bars[SB_SQ + (i & 1)]);
        } else {
          const int j = nd++;
          if (lane == 0) {  // += delta^T P^T (j): hi*hi + hi*lo + lo*hi
            tc_fence_after();
            const uint8_t* ps = sm + ST_PS + (j & 1) * PS_BYTES;
            const uint32_t id = idesc_bf16(128, 64, 0, 0);
            const uint64_t ph = desc_k(ps, 0, 8192), pl = desc_k(ps + 8192, 0, 8192);
            const uint32_t d = tmem + TT_O + 64 * (j & 1);
            mma_k64<true, false, false>(d, 0, tmem + TT_DH, ph, id, 1);
            mma_k64<true, false, false>(d, 0, tmem + TT_DH, pl, id, 1);
            mma_k64<true, false, false>(d, 0, tmem + TT_DL, ph, id, 1);
            mma_commit(&bars[SB_DP + (j & 1)]);
          }
        }
        __syncwarp();
      }
      if (did) {
        t_idle = globaltimer_ns();
      } else if (*abort_flag != 0) {
        break;
      } else if (globaltimer_ns() - t_idle > kWaitNs) {
        atomicOr((int*)abort_flag, ST_WAIT);
        break;
      }
    }
    return;
  }
  if (warp > kMmaWarp) return;

  const int q4 = warp & 3;
  const int row = q4 * 32 + lane;
  const uint32_t tq = tmem + ((uint32_t)(q4 * 32) << 16);

  if (warp < 4) {
    // ======================= chain: the serial state pass =======================
    bool alive = true;
#define CH_WAIT(bar, par, cl)                                   \
  if (group_waits_fail(abort_flag, 1, 128, (bar), (par), (cl))) { \
    alive = false;                                              \
    break;                                                      \
  }
#define CH_WAIT3(b1, p1, c1, b2, p2, b3, p3)                                   \
  if (group_waits_fail(abort_flag, 1, 128, (b1), (p1), (c1), (b2), (p2), (b3), (p3))) { \
    alive = false;                                                             \
    break;                                                                     \
  }
    // initial state: bf16 copy for the first MMAs, gamma_0 * S0 into TMEM
    do {
      float gam = 1.f;
      if (u.nc > 0) {
        CH_WAIT(&bars[SB_QK_FULL + 0], 0, false);
        gam = der_all[64 + 63];  // e^{g_last} of chunk 0
      }
#pragma unroll 1
      for (int p = 0; p < 4; ++p) {
        float v[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 t4 = make_float4(0.f, 0.f, 0.f, 0.f);
          if (S0) t4 = *reinterpret_cast<const float4*>(S0 + u.s0idx + (size_t)row * kD + 32 * p + 4 * q);
          v[4 * q] = t4.x; v[4 * q + 1] = t4.y; v[4 * q + 2] = t4.z; v[4 * q + 3] = t4.w;
        }
        if (u.nc == 0) {
          if (S_final)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              st4(S_final + u.sidx + (size_t)row * kD + 32 * p + 4 * q, v[4 * q], v[4 * q + 1],
                  v[4 * q + 2], v[4 * q + 3]);
          continue;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) st_sw128_8(sm + ST_SB, row, 32 * p + 8 * q, 128, v + 8 * q);
        if constexpr (!LINEAR) state_lo_to_tmem(tq, p, v);
        uint32_t sv[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) sv[e] = __float_as_uint(gam * v[e]);
        tmem_st32(tq + TT_S + 32 * p, sv);
      }
      if constexpr (LINEAR) {
        if (u.nc > 0)
          lin_delta(tq, sm + ST_QK + ST_V, der_all + 128, row, 0, (int)min((long long)kC, u.len));
      }
      tmem_wait_st();
      fence_async_smem();
      tc_fence_before();
      named_sync(1, 128);
      if (LINEAR && tid == 0 && u.nc > 0) mbar_arrive(&bars[SB_DR + 0]);  // delta (0) made
    } while (0);

    #pragma unroll 1
    for (int j = 0; alive && j < u.nc; ++j) {
      const int s = j % ST_NST;
      const float* ED = der_all + s * ST_DER_STAGE + 128;
      uint8_t* stg = sm + ST_QK + s * ST_STAGE;
      const int b = j & 1;  // handoff slot, P slot and output accumulator of chunk j
      const uint32_t buse = (uint32_t)(j >> 1);
      uint8_t* hs = sm + ST_HS + b * HS_BYTES;

      if constexpr (LINEAR) {
        // delta~ (j) was made in the previous iteration; the bf16 S of chunk j is final
        if (tid == 0) {
          mbar_arrive(&bars[SB_SWI]);  // S Q^T (j) may be queued
          tc_fence_after();
          const uint32_t id = idesc_bf16(128, 128, 0, 1);
          const uint64_t dkb = desc_mn(stg + 8192, 0, 16384);
          mma_k64<true, true, true>(tmem + TT_S, 0, tmem + tl_dsh(b), dkb, id, 1);
          mma_k64<true, true, true>(tmem + TT_S, 0, tmem + tl_dsl(b), dkb, id, 1);
          mma_commit(&bars[SB_DS]);
        }
        // delta (j + 1), delta~ (j + 1) into buffer b ^ 1 while the state update runs:
        // chunk j + 1 is loaded, and delta^T P^T (j - 1) has read that buffer's delta
        // (the state update of j - 1, its delta~, completed in the last iteration)
        if (j + 1 < u.nc) {
          CH_WAIT3(&bars[SB_QK_FULL + (j + 1) % ST_NST], ((j + 1) / ST_NST) & 1, false,
                   j > 0 ? &bars[SB_DP + (b ^ 1)] : nullptr, ((j - 1) >> 1) & 1, nullptr, 0);
          tc_fence_after();
          const int s1 = (j + 1) % ST_NST;
          lin_delta(tq, sm + ST_QK + s1 * ST_STAGE + ST_V, der_all + s1 * ST_DER_STAGE + 128, row,
                    b ^ 1, (int)min((long long)kC, u.len - (long long)(j + 1) * kC));
          tmem_wait_st();
          tc_fence_before();
        }
      } else {
        // ---- delta^T = U^T + S (-W~^T): U^T = V^T Tu^T is already in the accumulator
        //      (issued by the MMA warp) ----
        CH_WAIT3(&bars[SB_HF + b], buse & 1, true, &bars[SB_U + b], buse & 1, nullptr, 0);
        if (tid == 0) {
          tc_fence_after();
          const uint32_t id = idesc_bf16(128, 64, 0, 1);
          const uint64_t ds = desc_k(sm + ST_SB, 0, 16384), dw = desc_mn(hs, 0, 16384);
          mma_k128<true>(tmem + TT_SW, ds, 16384 >> 4, dw, 0, id, 1);
          mma_commit(&bars[SB_C]);
          mbar_arrive(&bars[SB_SWI]);  // S Q^T may now be queued behind S W~^T
        }
        // S W~^T done; delta of chunk j - 1 read by its delta^T P^T
        CH_WAIT3(&bars[SB_C], j & 1, false, j > 0 ? &bars[SB_DP + ((j - 1) & 1)] : nullptr,
                 ((j - 1) >> 1) & 1, nullptr, 0);
        tc_fence_after();
        // the slot's only readers were the MMAs whose completion was just observed
        if (tid == 0) mbar_arrive_remote_relaxed(map_shared(smem_u32(sm + WY_BAR + 8 * (WB_HE + b)), 0));

        // ---- delta and its decayed copy as hi/lo bf16 A operands in TMEM ----
#pragma unroll 1
        for (int qq = 0; qq < 4; ++qq) delta_quarter(tq, TT_SW, ED, qq);
        tmem_wait_st();
        tc_fence_before();
        named_sync(1, 128);

        // ---- S <- e^{g_last} S + delta~^T K (accumulated onto the pre-scaled S) ----
        if (tid == 0) {
          tc_fence_after();
          const uint32_t id = idesc_bf16(128, 128, 0, 1);
          const uint64_t dkb = desc_mn(stg + 8192, 0, 16384);
          mma_k64<true, true, true>(tmem + TT_S, 0, tmem + TT_DSH, dkb, id, 1);
          mma_k64<true, true, true>(tmem + TT_S, 0, tmem + TT_DSL, dkb, id, 1);
          mma_commit(&bars[SB_DS]);
          // delta of chunk j is in TMEM and the accumulator of U^T + S(-W~^T) is free
          mbar_arrive(&bars[SB_DR + b]);
        }
      }
      // the state update is done, S Q^T of chunk j has read S, chunk j + 1 is loaded
      const bool last = (j + 1 == u.nc);
      CH_WAIT3(&bars[SB_DS], j & 1, false, &bars[SB_SQ + b], (j >> 1) & 1,
               last ? nullptr : &bars[SB_QK_FULL + (j + 1) % ST_NST], ((j + 1) / ST_NST) & 1);
      tc_fence_after();
      if (tid == 0) mbar_arrive(&bars[SB_QK_EMPTY + s]);  // the chain's last read of stage s
      if (LINEAR && tid == 0 && !last) mbar_arrive(&bars[SB_DR + (b ^ 1)]);  // delta (j + 1) made
      const float gam = last ? 1.f : der_all[((j + 1) % ST_NST) * ST_DER_STAGE + 64 + 63];

      // ---- new state: bf16 copy for the next chunk, pre-scaled fp32 back to TMEM ----
#pragma unroll 1
      for (int p = 0; p < 4; ++p) {
        uint32_t r[32];
        tmem_ld32(tq + TT_S + 32 * p, r);
        tmem_wait_ld();
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
        if (last) {
          if (S_final)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              st4(S_final + u.sidx + (size_t)row * kD + 32 * p + 4 * q, v[4 * q], v[4 * q + 1],
                  v[4 * q + 2], v[4 * q + 3]);
        } else {
          // bf16 S (the hi term) into shared memory and, in the delta rule, the lo term
          // bf16(S - hi) into TMEM (S Q^T (j), the last reader of both, completed)
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            hi[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
            if constexpr (!LINEAR)
              lo[e] = pack_bf16(v[2 * e] - __uint_as_float(hi[e] << 16),
                                v[2 * e + 1] - __uint_as_float(hi[e] & 0xffff0000u));
          }
#pragma unroll
          for (int q = 0; q < 4; ++q)
            st_shared_v4(smem_u32(sm + ST_SB + sw128_offset(row, 32 * p + 8 * q, 128)), hi[4 * q],
                         hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]);
          if constexpr (!LINEAR) tmem_st16(tq + TT_SLO + 16 * p, lo);
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(gam * v[e]);
          tmem_st32(tq + TT_S + 32 * p, r);
        }
      }
      tmem_wait_st();
      fence_async_smem();
      tc_fence_before();
      named_sync(1, 128);
    }
#undef CH_WAIT
    return;
  }

  if (warp < 8) {
    // ============ aux P: Q K^T -> P (or P' = P e^{-g_t}), ahead of the chain ============
    const int atid = tid - 128;
#define AP_WAIT(bar, par) \
  if (group_wait_fails((bar), (par), abort_flag, false, 2, 128)) break;
    #pragma unroll 1
    for (int j = 0; j < u.nc; ++j) {
      const int s = j % ST_NST;
      const int b = j & 1;
      uint8_t* stg = sm + ST_QK + s * ST_STAGE;
      uint8_t* ps = sm + ST_PS + b * PS_BYTES;
      const float* GN = der_all + s * ST_DER_STAGE;
      const float* EG = GN + 64;
      AP_WAIT(&bars[SB_QK_FULL + s], (j / ST_NST) & 1);
      const bool factored = flags[s] != 0;
      // the delta rule accumulates Q K^T in output accumulator b, free once the outputs of
      // chunk j - 2 (which also leave P slot b) were drained
      const uint32_t t_qk = LINEAR ? TT_QK : TT_O + 64 * b;
      if constexpr (!LINEAR) AP_WAIT(&bars[SB_PE + b], ((j >> 1) & 1) ^ 1);

      // ---- Q K^T as an M=64 accumulator (row m in TMEM lane 32 (m / 16) + m % 16, so
      //      every warp of this group holds 16 rows), issued from warp 6 ----
      if (atid == 64) {
        tc_fence_after();
        mma_k128_commit(tmem + t_qk, desc_k(stg, 0, 16384), desc_k(stg + 8192, 0, 16384),
                        idesc_bf16(64, 64, 0, 0), &bars[SB_QKM]);
      }
      AP_WAIT(&bars[SB_QKM], j & 1);
      if constexpr (LINEAR) AP_WAIT(&bars[SB_PE + b], ((j >> 1) & 1) ^ 1);  // slot b is free
      tc_fence_after();
      // factored:  P'_{t,j} = q_t.k_j e^{-g_j}      (the e^{g_t} is applied to the outputs)
      // otherwise: P_{t,j}  = q_t.k_j e^{g_t - g_j} (and Q is scaled by e^{g_t} below)
      {
        // the TMEM loads are warp-wide; lanes 16..31 of each warp hold no row
        const int prow = 16 * q4 + (lane & 15);
        if (factored)
          aux_epi_p<true>(tq + t_qk, ps, prow, 0.f, GN, lane < 16);
        else
          aux_epi_p<false>(tq + t_qk, ps, prow, GN[prow], GN, lane < 16);
      }
      if (!factored) {
        // Q <- diag(e^{g}) Q in place (bf16), after Q K^T has read it: 16-byte pieces,
        // each inside one row (row = offset / 128 in either 64-column panel)
#pragma unroll 1
        for (int it0 = 0; it0 < 1024; it0 += 128) {
          const int it = it0 + atid;
          const int pnl = it >> 9, off = (it & 511) * 16;
          uint4* pq = reinterpret_cast<uint4*>(stg + pnl * 16384 + off);
          const float e = EG[off >> 7];
          uint4 x = *pq;
          uint32_t* w = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float lo = __uint_as_float(w[c] << 16), hi = __uint_as_float(w[c] & 0xffff0000u);
            w[c] = pack_bf16(lo * e, hi * e);
          }
          *pq = x;
        }
      }
      fence_async_smem();
      tc_fence_before();
      named_sync(2, 128);
      if (atid == 0) {
        mbar_arrive(&bars[SB_PF + b]);
        mbar_arrive(&bars[SB_QK_EMPTY + s]);  // aux P reads nothing more of stage s
      }
    }
#undef AP_WAIT
    return;
  }

  // ============ aux O: o_t = e^{g_t} O'_t (or O_t) -> out ============
  // aux O holds no stage: each of its warps recomputes the chunk's gate factors from
  // the gates in global memory (the same scan as the producer, so the same values and
  // the same choice of form), and the bf16 outputs are staged in the chunk's P slot,
  // which delta^T P^T no longer reads.  In the linear mode it also issues S Q^T (i) into
  // output accumulator i % 2 before it drains the outputs of chunk i - 1 out of the other
  // one (one issue site); in the delta rule the MMA warp issues S Q^T.
  const int atid = tid - 256;
#define AO_WAIT(bar, par) \
  if (group_wait_fails((bar), (par), abort_flag, false, 3, 128)) break;
  // Linear mode, S Q^T (i): issued (from warp 11) once the chain has queued S W~^T (i),
  // which reads the same bf16 S, and, in the strong-decay form, once aux P has scaled Q.
  // The chunk's form is read from its stage, which the chain waited for before signalling.
#define AO_ISSUE_SQ(i)                                                                          \
  {                                                                                           \
    AO_WAIT(&bars[SB_SWI], (i) & 1);                                                          \
    const int si = (i) % ST_NST;                                                              \
    if (flags[si] == 0) AO_WAIT(&bars[SB_PF + ((i) & 1)], ((i) >> 1) & 1);                    \
    if (atid == 96)                                                                           \
      mma_k128_commit(tmem + TT_O + 64 * ((i) & 1), desc_k(sm + ST_SB, 0, 16384),              \
                      desc_k(sm + ST_QK + si * ST_STAGE, 0, 16384), idesc_bf16(128, 64, 0, 0),   \
                      &bars[SB_SQ + ((i) & 1)]);                                              \
  }
  GateLoad gnext = load_gates(log_alpha, beta, u, H, 0, lane);
  #pragma unroll 1
  for (int i = 0; i <= u.nc; ++i) {
    const int j = i - 1, b = j & 1;
    if (LINEAR && i < u.nc) AO_ISSUE_SQ(i)
    if (i > 0) {
      __nv_bfloat16* ost0 = reinterpret_cast<__nv_bfloat16*>(sm + ST_PS + b * PS_BYTES);
      const GateLoad gcur = gnext;
      gnext = load_gates(log_alpha, beta, u, H, i, lane);  // in flight during the wait
      float g0, g1, tot;
      scan_gates(gcur, lane, g0, g1, tot);
      const bool factored = -tot < kMaxFactoredDecayLog2;
      const float e0 = factored ? ex2(g0) : 1.f, e1 = factored ? ex2(g1) : 1.f;
      // S Q^T and delta^T P^T of chunk j (the MMA warp commits delta^T P^T last)
      AO_WAIT(&bars[SB_DP + b], (j >> 1) & 1);
      tc_fence_after();
      // ---- bf16 outputs staged in P slot b (row t at t * 256 bytes), 8 tokens a step ----
      const uint32_t to = tq + TT_O + 64 * b;
#pragma unroll 1
      for (int q = 0; q < 8; ++q) {
        uint32_t a[8];
        tmem_ld8(to + 8 * q, a);
        tmem_wait_ld();
        const float ev = q < 4 ? e0 : e1;  // e^{g_t} of tokens 8q .. 8q + 7 (lanes t % 32)
#pragma unroll
        for (int e = 0; e < 8; ++e)
          ost0[(8 * q + e) * kD + row] = __float2bfloat16_rn(
              __shfl_sync(0xffffffffu, ev, (8 * q + e) & 31) * __uint_as_float(a[e]));
      }
      tc_fence_before();
      named_sync(3, 128);  // outputs staged; the accumulator is free for its next S Q^T
      const long long c0 = (long long)j * kC;
      const int lc = (int)min((long long)kC, u.len - c0);
      const size_t obase = (size_t)(u.row0 + c0) * H + u.h;
#pragma unroll 1
      for (int it0 = 0; it0 < 1024; it0 += 128) {
        const int it = it0 + atid;
        const int t = it >> 4, ch = it & 15;
        if (t < lc) {
          const uint4 v = *reinterpret_cast<const uint4*>(ost0 + t * kD + 8 * ch);
          *reinterpret_cast<uint4*>(out + (obase + (size_t)t * H) * kD + 8 * ch) = v;
        }
      }
      named_sync(3, 128);
      if (atid == 0) mbar_arrive(&bars[SB_PE + b]);  // P slot b may be refilled
    }
  }
#undef AO_ISSUE_SQ
#undef AO_WAIT
}


__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
gdn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const float* __restrict__ log_alpha,
              const float* __restrict__ beta, const float* __restrict__ S0,
              __nv_bfloat16* __restrict__ out, float* __restrict__ S_final,
              const int32_t* __restrict__ cu_seqlens, int H, int T) {
  extern __shared__ uint8_t smem_raw[];
  // Align to 1024 bytes by pointer arithmetic on the shared array itself (accesses
  // stay shared-memory accesses); the offset is the same in both CTAs.
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const Unit u = make_unit(blockIdx.x >> 1, cu_seqlens, H, T);

  uint8_t* misc = sm + (rank == 0 ? WY_MISC : ST_MISC);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  if (warp == 0) tmem_alloc(tslot, TM_COLS);
  if (tid == 32) {
    *abort_flag = 0;
    if (rank == 0) {
      uint64_t* b = reinterpret_cast<uint64_t*>(sm + WY_BAR);
      for (int s = 0; s < WY_NST; ++s) {
        mbar_init(&b[WB_KV_FULL + s], 2);
        mbar_init(&b[WB_KV_EMPTY + s], 1);
      }
      for (int k = 0; k < WY_NWG; ++k) mbar_init(&b[WB_MMA + k], 1);
      for (int k = 0; k < 2; ++k) mbar_init(&b[WB_HE + k], 1);
      *reinterpret_cast<volatile int*>(sm + WY_MISC + 8) = 0;  // hand-off ticket
      prefetch_tensormap(&tm_k);
    } else {
      uint64_t* b = reinterpret_cast<uint64_t*>(sm + ST_BAR);
      for (int s = 0; s < ST_NST; ++s) {
        mbar_init(&b[SB_QK_FULL + s], 2);
        mbar_init(&b[SB_QK_EMPTY + s], 2);  // the chain (after its state update) and aux P
      }
      for (int k = SB_HF; k < SB_COUNT; ++k) mbar_init(&b[k], 1);
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
    }
    fence_mbarrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  cluster_sync();  // both CTAs' barriers exist before any remote arrive or copy

  if (rank == 0)
    run_wy(sm, tmem, &tm_k, log_alpha, beta, u, H, abort_flag);
  else
    run_state<false>(sm, tmem, &tm_q, &tm_k, &tm_v, log_alpha, beta, S0, out, S_final, u, H,
                     abort_flag);

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // after a wait gave up, let any remote stores or copies still in flight land
    // before either CTA can pass the final cluster barrier
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000ull) {
    }
    if (tid == 0) atomicOr(&g_tc_status, *abort_flag);
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
  cluster_sync();  // neither CTA leaves while the other may still touch its memory
}

// ---------------------------------------------------------------------------------
// The linear mode over more SMs.  In the linear mode a segment of tokens maps the state
// affinely with a scalar gain: S_end = Gamma S_start + L, Gamma = e^{sum of log alpha}
// over the segment ([N] "Mamba2": the state is a decayed sum of the writes).  When the
// (sequence, head) units fill at most half of the SMs, every sequence of a fixed-length
// batch is cut into R chunk-aligned, non-empty segments that run as units of their own:
//   1. the linear kernel on the N R segments, the first of each sequence from S0, the
//      others from zero: outputs o(0) and end states L_r;
//   2. the correction of segments r >= 1, o_t += e^{G_t} S_start q_t (G_t the sum of log
//      alpha from the segment's first token through t: what the start state adds to the
//      output, which is linear in it), each CTA folding the start state it needs,
//      S_start_1 = L_0 and S_start_r = Gamma_{r-1} S_start_{r-1} + L_{r-1}, and one CTA
//      per (sequence, head) writing S_final = Gamma_{R-1} S_start_{R-1} + L_{R-1}.
constexpr int kLsMaxSeg = 4;

// Token bounds [a, b) of segment r of a length-T sequence: whole chunks, as even as the
// chunk count allows (R from linear_split_segments leaves none empty).
__host__ __device__ __forceinline__ void seg_bounds(int T, int R, int r, int& a, int& b) {
  const int nch = (T + kC - 1) / kC, per = (nch + R - 1) / R;
  a = min(r * per * kC, T);
  b = min((r + 1) * per * kC, T);
}
__host__ __device__ __forceinline__ int seg_tiles(int T, int R, int r) {
  int a, b;
  seg_bounds(T, R, r, a, b);
  return a < b ? (b - a + 63) / 64 : 0;
}
// The correction's segment r >= 1: segment r of the split, or, when the start states are
// given (`whole`), the whole sequence as its one segment.
__host__ __device__ __forceinline__ void corr_bounds(int T, int R, int r, bool whole, int& a,
                                                     int& b) {
  if (whole) {
    a = 0;
    b = T;
  } else {
    seg_bounds(T, R, r, a, b);
  }
}
__host__ __device__ __forceinline__ int corr_tiles(int T, int R, int r, bool whole) {
  int a, b;
  corr_bounds(T, R, r, whole, a, b);
  return a < b ? (b - a + 63) / 64 : 0;
}

// Linear mode (no erase, write strength 1): the WY factors are T = I, W~ = 0, U = V, so
// the state CTA runs alone, one CTA per (sequence, head): its chain is the state update
// and the S epilogue, with delta and delta~ made from the V tile by aux P.  With R > 1
// (fixed-length batch, no cu_seqlens) CTA (n R + r) H + h runs segment r of sequence n,
// from S0[n][h] when r = 0 and from zero otherwise, and writes its end state to
// S_final[(n R + r) H + h].
__global__ void __launch_bounds__(kThreads, 1)
gdn_tc_linear_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const float* __restrict__ log_alpha,
                     const float* __restrict__ S0, __nv_bfloat16* __restrict__ out,
                     float* __restrict__ S_final, const int32_t* __restrict__ cu_seqlens, int H,
                     int T, int R) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5;
  Unit u = make_unit(blockIdx.x, cu_seqlens, H, T);
  if (R > 1) {
    const int nr = blockIdx.x / H, n = nr / R, r = nr % R;
    int a, b;
    seg_bounds(T, R, r, a, b);
    u.row0 = (long long)n * T + a;
    u.len = b - a;
    u.nc = (int)((u.len + kC - 1) / kC);
    u.s0idx = ((size_t)n * H + u.h) * kD * kD;
    if (r > 0) S0 = nullptr;
  }
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + ST_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + ST_MISC + 4);
  if (warp == 0) tmem_alloc(tslot, TM_COLS);
  if (tid == 32) {
    *abort_flag = 0;
    uint64_t* b = reinterpret_cast<uint64_t*>(sm + ST_BAR);
    for (int s = 0; s < ST_NST; ++s) {
      mbar_init(&b[SB_QK_FULL + s], 2);
      mbar_init(&b[SB_QK_EMPTY + s], 2);  // the chain (after its state update) and aux P
    }
    for (int k = SB_HF; k < SB_COUNT; ++k) mbar_init(&b[k], 1);
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    fence_mbarrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  run_state<true>(sm, tmem, &tm_q, &tm_k, &tm_v, log_alpha, nullptr, S0, out, S_final, u, H,
                  abort_flag);
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) atomicOr(&g_tc_status, *abort_flag);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}


// The correction's epilogue warps (0-3) synchronise among themselves on named barrier 1.
constexpr uint32_t kLsEpiBar = 1;
// Sum over the 128 epilogue threads (all of them call it).
__device__ __forceinline__ float ls_block_sum(float x, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  named_sync(kLsEpiBar, 128);  // red free from its last use
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
  named_sync(kLsEpiBar, 128);
  return (red[0] + red[1]) + (red[2] + red[3]);
}
// Sum of log alpha over tokens [t0, t1) of sequence n, head h (0 without a gate): the 128
// epilogue threads, sixteen strided loads each in flight per round of 2048 tokens.
__device__ __forceinline__ float ls_la_sum(const float* __restrict__ log_alpha, int n, int T,
                                           int H, int h, int t0, int t1, float* red) {
  float s = 0.f;
  if (log_alpha) {
    const float* la = log_alpha + (size_t)n * T * H + h;
    for (int base = t0; base < t1; base += 2048) {
      float v[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = base + (int)threadIdx.x + 128 * e;
        v[e] = t < t1 ? la[(size_t)t * H] : 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] += v[e + 8];
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] += v[e + 4];
      s += (v[0] + v[1]) + (v[2] + v[3]);
    }
  }
  return ls_block_sum(s, red);
}
// Sums of log alpha over [t0, tm) and [tm, t1) of sequence n, head h in one pass.
__device__ __forceinline__ float2 ls_la_sum2(const float* __restrict__ log_alpha, int n, int T,
                                             int H, int h, int t0, int tm, int t1, float* red) {
  float s0 = 0.f, s1 = 0.f;
  if (log_alpha) {
    const float* la = log_alpha + (size_t)n * T * H + h;
    for (int base = t0; base < t1; base += 2048) {
      float v[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = base + (int)threadIdx.x + 128 * e;
        v[e] = t < t1 ? la[(size_t)t * H] : 0.f;
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int t = base + (int)threadIdx.x + 128 * e;
        if (t < tm) s0 += v[e]; else s1 += v[e];
      }
    }
  }
  const float a = ls_block_sum(s0, red);
  return make_float2(a, ls_block_sum(s1, red));
}

// The correction.  Its work is the (sequence, head, segment r >= 1, 64-token tile) list in
// that order; with cps > 0 each segment is split into cps contiguous shares, one per CTA
// (grid = segments x cps), else each CTA takes a contiguous run of whole segments.  The
// CTAs of the last segment of a (sequence, head) also write its S_final.  With Sst given
// (R = 2), each whole sequence is the one corrected segment: its start state is
// Sst[n][h], and S_final holds its end state from zero on entry (updated in place).
// Warp 4 (one thread) loads q and out tiles by TMA into a three-stage ring, issues
// D^T (dv x 64 tokens) = S_hi Q^T + S_lo Q^T into one of two TMEM accumulators a tile
// ahead of the epilogue, and stores each corrected out tile back by TMA.  Warps 0-3, a
// thread per state row / output column d: on reaching a segment they fold its start
// state from the segments' end states L (fp32) into tensor memory as bf16 hi and lo
// pairs (the A operand); per tile they scan the gates and add e^{G_t} times their TMEM
// lane into the out tile in shared memory.  Two CTAs fit an SM.
constexpr int kLsStages = 3, kLsStageBytes = 32768;  // per stage: q 16 KB, out 16 KB
constexpr int kLsSmem = kLsStages * kLsStageBytes + 1024;
constexpr int kLsThreads = 160;
constexpr uint32_t kLsTmHi = 0, kLsTmLo = 64, kLsTmAcc = 128;  // TMEM columns

__global__ void __launch_bounds__(kLsThreads, 2)
ls_corr_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
               int N, int H, int T, int R, int cps, const float* __restrict__ log_alpha,
               const float* __restrict__ L, float* __restrict__ S_final,
               const float* __restrict__ Sst, __nv_bfloat16* __restrict__ out) {
  const bool whole = Sst != nullptr;
  extern __shared__ uint8_t ls_smem_raw[];
  uint8_t* sm = ls_smem_raw + ((1024u - (smem_u32(ls_smem_raw) & 1023u)) & 1023u);
  // full[s], out_ready[s] (the epilogue has written stage s's out tile), acc_full[a],
  // acc_empty[a], s_ready (a segment's start state is in TMEM)
  __shared__ __align__(8) uint64_t bars[2 * kLsStages + 5];
  uint64_t* full = bars;
  uint64_t* out_ready = bars + kLsStages;
  uint64_t* acc_full = bars + 2 * kLsStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* s_ready = acc_full + 4;
  __shared__ uint32_t tslot;
  __shared__ int abort_s;
  __shared__ __align__(16) float sc[64], eg[64], red[4];
  volatile int* abort_flag = &abort_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int tpu = 0;  // tiles per (sequence, head)
  for (int r = 1; r < R; ++r) tpu += corr_tiles(T, R, r, whole);
  const long long tot = (long long)N * H * tpu, nseg = (long long)N * H * (R - 1);
  auto seg_first = [&](long long sg) {  // list index of segment sg's first tile
    if (sg >= nseg) return tot;
    long long i = sg / (R - 1) * tpu;
    for (int q = 1; q < 1 + (int)(sg % (R - 1)); ++q) i += corr_tiles(T, R, q, whole);
    return i;
  };
  long long i0, i1;
  if (cps > 0) {
    const long long sg = blockIdx.x / cps, base = seg_first(sg);
    const int j = blockIdx.x % cps, nt = corr_tiles(T, R, 1 + (int)(sg % (R - 1)), whole);
    i0 = base + (long long)nt * j / cps;
    i1 = base + (long long)nt * (j + 1) / cps;
  } else {
    i0 = seg_first(nseg * blockIdx.x / gridDim.x);
    i1 = seg_first(nseg * (blockIdx.x + 1) / gridDim.x);
  }
  if (i0 >= i1) return;
  const int n_t = (int)(i1 - i0);
  // tile i of the list: (sequence, head) unit, segment r, tile k of the segment
  auto decode = [&](long long i, int& unit, int& r, int& k) {
    unit = (int)(i / tpu);
    k = (int)(i % tpu);
    r = 1;
    while (r + 1 < R && k >= corr_tiles(T, R, r, whole)) k -= corr_tiles(T, R, r++, whole);
  };
  if (tid == 0) {
    for (int s = 0; s < kLsStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&out_ready[s], 4);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);
    }
    mbar_init(s_ready, 4);
    abort_s = 0;
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_o);
    fence_mbarrier_init();
  }
  if (warp == 0) tmem_alloc(&tslot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tslot;

  if (warp == 4) {
    if (lane == 0) {  // loads, products and stores
      auto load = [&](int it) {
        int unit, r, k, a, b;
        decode(i0 + it, unit, r, k);
        corr_bounds(T, R, r, whole, a, b);
        const int s = it % kLsStages, h = unit % H, row = (unit / H) * T + a + 64 * k;
        uint8_t* qb = sm + s * kLsStageBytes;
        mbar_arrive_expect_tx(&full[s], 32768);
        for (int c = 0; c < 2; ++c) {
          tma_load_3d(qb + c * 8192, &tm_q, &full[s], 64 * c, h, row);
          tma_load_3d(qb + 16384 + c * 8192, &tm_o, &full[s], 64 * c, h, row);
        }
      };
      const uint32_t id = idesc_bf16(128, 64, 0, 0);
      long long seg = -1;
      int nseg = 0;
      auto product = [&](int it) {  // false: a wait gave up
        int unit, r, k;
        decode(i0 + it, unit, r, k);
        const int s = it % kLsStages, a = it & 1;
        if ((long long)unit * R + r != seg) {  // its start state is in TMEM once s_ready flips
          seg = (long long)unit * R + r;
          if (!wait_bar(s_ready, nseg++ & 1, abort_flag, false)) return false;
        }
        if (!wait_bar(&full[s], (it / kLsStages) & 1, abort_flag, false)) return false;
        if (it >= 2 && !wait_bar(&acc_empty[a], ((it >> 1) - 1) & 1, abort_flag, false))
          return false;
        tc_fence_after();
        const uint8_t* qb = sm + s * kLsStageBytes;
        const uint32_t d = tmem + kLsTmAcc + 64u * a;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t dq = desc_k(qb, ks, 8192);
          mma_bf16_ta(d, tmem + kLsTmHi + 8 * ks, dq, id, ks != 0);
          mma_bf16_ta(d, tmem + kLsTmLo + 8 * ks, dq, id, 1u);
        }
        mma_commit(&acc_full[a]);
        return true;
      };
      for (int it = 0; it < min(kLsStages, n_t); ++it) load(it);
      bool ok = product(0);
      for (int it = 0; ok && it < n_t; ++it) {
        if (it + 1 < n_t && !(ok = product(it + 1))) break;  // one tile ahead
        // tile it back to HBM once the epilogue has written it
        const int s = it % kLsStages;
        if (!(ok = wait_bar(&out_ready[s], (it / kLsStages) & 1, abort_flag, false))) break;
        int unit, r, k, a, b;
        decode(i0 + it, unit, r, k);
        corr_bounds(T, R, r, whole, a, b);
        // a whole tile goes back by TMA store; a sequence's ragged last tile was written
        // to its rows by the epilogue (past them are another sequence's), so its group is
        // empty
        const uint8_t* ob = sm + s * kLsStageBytes + 16384;
        if (a + 64 * k + 64 <= b)
          for (int c = 0; c < 2; ++c)
            tma_store_3d(&tm_o, ob + c * 8192, 64 * c, unit % H, (unit / H) * T + a + 64 * k);
        bulk_commit();
        // the stage of tile it - 1 takes tile it + 2 once that tile's store has read it
        if (it >= 1 && it + 2 < n_t) {
          bulk_wait_read_1();
          load(it + 2);
        }
      }
      bulk_wait_all();
    }
  } else {  // warps 0-3
    const uint32_t tl_row = tmem + ((uint32_t)(32 * warp) << 16);  // this warp's TMEM lanes
    long long seg = -1;  // the segment whose start state is in TMEM
    float pcur = 0.f;    // sum of log alpha from the segment's first token to the tile's
    float gam[kLsMaxSeg - 1] = {1.f, 1.f, 1.f};  // Gamma_j of the segment's earlier ones
    const size_t DD = (size_t)kD * kD, row = (size_t)tid * kD;
    // Columns 64 hv .. 64 hv + 63 of row `tid` of S_start_r from the end states, given in
    // x the same columns of L_0: S_start_{j+1} = Gamma_j S_start_j + L_j.
    auto fold_start = [&](const float* Lu, int r, int hv, float4 (&x)[16]) {
#pragma unroll 1
      for (int j = 1; j < r; ++j) {
        const float gj = j == 1 ? gam[0] : (j == 2 ? gam[1] : gam[2]);
        const float* Lj = Lu + (size_t)j * H * DD + 64 * hv;
        float4 y[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) y[e] = ld4(Lj + 4 * e);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          x[e].x = fmaf(gj, x[e].x, y[e].x);
          x[e].y = fmaf(gj, x[e].y, y[e].y);
          x[e].z = fmaf(gj, x[e].z, y[e].z);
          x[e].w = fmaf(gj, x[e].w, y[e].w);
        }
      }
    };
    // warps 0-1: log alpha of token 32 warp + lane of a tile, loaded a tile ahead
    auto gate_of = [&](int it) {
      int unit, r, k, a, b;
      decode(i0 + it, unit, r, k);
      corr_bounds(T, R, r, whole, a, b);
      const int t = 32 * warp + lane, t0 = a + 64 * k;
      return (log_alpha && t0 + t < b)
                 ? log_alpha[((size_t)(unit / H) * T + t0 + t) * H + unit % H]
                 : 0.f;
    };
    float la_next = warp < 2 ? gate_of(0) : 0.f;
    // this thread's output column d = tid in the out tile: panel, 16-byte chunk, byte
    const uint32_t col_off = (uint32_t)((tid >> 6) * 8192 + (tid & 7) * 2);
    const int col_chunk = (tid & 63) >> 3;
    for (int it = 0; it < n_t; ++it) {
      const int s = it % kLsStages, a_ = it & 1;
      int unit, r, k, a, b;
      decode(i0 + it, unit, r, k);
      corr_bounds(T, R, r, whole, a, b);
      const int n = unit / H, h = unit % H, t0 = a + 64 * k, len = min(64, b - t0);
      // this thread's row of L_j (Lu + j H DD), or of the given start state
      const float* Lu = whole ? Sst + ((size_t)n * H + h) * DD + row
                              : L + ((size_t)n * R * H + h) * DD + row;
      if ((long long)unit * R + r != seg) {  // the same for all four warps
        // the previous segment's products are complete: its last tile's were waited for
        seg = (long long)unit * R + r;
        float4 x[16];  // L_0 row, columns 0 .. 63: in flight while the gate sums run
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] = ld4(Lu + 4 * e);
        // the CTAs of a sequence's last segment also write S_final, each a share of its
        // elements: they need the segment's whole gate sum besides their prefix
        const bool fin = S_final != nullptr && r == R - 1;
        float gfin = 0.f;
        if (fin) {
          const float2 ps = ls_la_sum2(log_alpha, n, T, H, h, a, t0, b, red);
          pcur = ps.x;
          gfin = expf(ps.x + ps.y);
        } else {  // a CTA that starts at its segment's first tile has no prefix to sum
          pcur = k > 0 ? ls_la_sum(log_alpha, n, T, H, h, a, t0, red) : 0.f;
        }
        for (int j = 1; j < r; ++j) {
          int ja, jb;
          seg_bounds(T, R, j, ja, jb);
          const float g = expf(ls_la_sum(log_alpha, n, T, H, h, ja, jb, red));
          gam[0] = j == 1 ? g : gam[0];
          gam[1] = j == 2 ? g : gam[1];
          gam[2] = j == 3 ? g : gam[2];
        }
#pragma unroll 1
        for (int hv = 0; hv < 2; ++hv) {  // columns 64 hv .. 64 hv + 63
          if (hv == 1)
#pragma unroll
            for (int e = 0; e < 16; ++e) x[e] = ld4(Lu + 64 + 4 * e);
          fold_start(Lu, r, hv, x);
          uint32_t hi[32], lo[32];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            split2(x[e].x, x[e].y, hi[2 * e], lo[2 * e]);
            split2(x[e].z, x[e].w, hi[2 * e + 1], lo[2 * e + 1]);
          }
          tmem_st32(tl_row + kLsTmHi + 32 * hv, hi);
          tmem_st32(tl_row + kLsTmLo + 32 * hv, lo);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_ready);
        if (fin) {  // S_final = Gamma_r S_start_r + L_r over this CTA's share, coalesced
          // the shares of this CTA's tiles k .. kend - 1 of the segment's nt, so the CTAs of
          // the segment cover the whole state between them
          const int nt = corr_tiles(T, R, r, whole);
          const long long sf = i0 + it - k;  // list index of the segment's first tile
          const int kend = (int)(min(i1, sf + nt) - sf);
          const int f0 = (int)(DD / 4) * k / nt, f1 = (int)(DD / 4) * kend / nt;
          // L_0 (or the given start state), L_j for the fold, L_r (or, given start states,
          // the end state from zero, updated in place)
          float4* S4 = reinterpret_cast<float4*>(S_final + ((size_t)n * H + h) * DD);
          const float4* L4 = reinterpret_cast<const float4*>(
              whole ? Sst + ((size_t)n * H + h) * DD : L + ((size_t)n * R * H + h) * DD);
          const size_t js = (size_t)H * DD / 4;  // L_j to L_{j+1}, in float4
          const float4* E4 = whole ? S4 : L4 + r * js;
          for (int f = f0 + tid; f < f1; f += 8 * 128) {  // eight float4 a thread in flight
            float4 v[8], y[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int ff = min(f + 128 * u, f1 - 1);  // past the share: a repeat, not stored
              v[u] = L4[ff];
              y[u] = E4[ff];
            }
            for (int j = 1; j < r; ++j) {
              const float gj = j == 1 ? gam[0] : (j == 2 ? gam[1] : gam[2]);
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const float4 z = L4[min(f + 128 * u, f1 - 1) + j * js];
                v[u] = make_float4(fmaf(gj, v[u].x, z.x), fmaf(gj, v[u].y, z.y),
                                   fmaf(gj, v[u].z, z.z), fmaf(gj, v[u].w, z.w));
              }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
              if (f + 128 * u < f1)
                S4[f + 128 * u] = make_float4(fmaf(gfin, v[u].x, y[u].x), fmaf(gfin, v[u].y, y[u].y),
                                              fmaf(gfin, v[u].z, y[u].z), fmaf(gfin, v[u].w, y[u].w));
          }
        }
      }
      if (warp < 2) {  // inclusive scan of the tile's 64 log alpha, 32 per warp
        const int t = 32 * warp + lane;
        float x = la_next;
        if (it + 1 < n_t) la_next = gate_of(it + 1);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        sc[t] = x;
      }
      named_sync(kLsEpiBar, 128);
      if (tid < 64) eg[tid] = expf(pcur + sc[tid] + (tid >= 32 ? sc[31] : 0.f));
      pcur += sc[31] + sc[63];
      // the out tile has landed and the product is done
      if (group_waits_fail(abort_flag, kLsEpiBar, 128, &full[s], (it / kLsStages) & 1, false,
                           &acc_full[a_], (it >> 1) & 1))
        break;
      tc_fence_after();
      uint8_t* ob = sm + s * kLsStageBytes + 16384 + col_off;
      const uint32_t tl = tl_row + kLsTmAcc + 64u * a_;
#pragma unroll 1
      for (int cb = 0; cb < 2; ++cb) {  // tokens 32 cb .. 32 cb + 31 of column d
        uint32_t u[32];
        tmem_ld32(tl + 32 * cb, u);
        // all 32 out values and gate factors first, so that the loads overlap
        unsigned short ov[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
          ov[j] = *reinterpret_cast<const unsigned short*>(
              ob + (32 * cb + j) * 128 + ((col_chunk ^ (j & 7)) << 4));
        float e[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 v = *reinterpret_cast<const float4*>(eg + 32 * cb + 4 * q);
          e[4 * q] = v.x;
          e[4 * q + 1] = v.y;
          e[4 * q + 2] = v.z;
          e[4 * q + 3] = v.w;
        }
        tmem_wait_ld();
        if (len == 64) {  // back into the tile, for the TMA store
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float o = __uint_as_float((uint32_t)ov[j] << 16) + e[j] * __uint_as_float(u[j]);
            *reinterpret_cast<__nv_bfloat16*>(ob + (32 * cb + j) * 128 +
                                              ((col_chunk ^ (j & 7)) << 4)) = __float2bfloat16_rn(o);
          }
        } else {  // a ragged last tile: straight to its own rows
          __nv_bfloat16* og = out + ((size_t)n * T + t0) * H * kD + (size_t)h * kD + tid;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (32 * cb + j < len) {
              const float o =
                  __uint_as_float((uint32_t)ov[j] << 16) + e[j] * __uint_as_float(u[j]);
              og[(size_t)(32 * cb + j) * H * kD] = __float2bfloat16_rn(o);
            }
        }
      }
      tc_fence_before();
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&acc_empty[a_]);
        mbar_arrive(&out_ready[s]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {  // let copies and products still in flight land before TMEM goes
    const uint64_t tw = globaltimer_ns();
    while (globaltimer_ns() - tw < 50000ull) {
    }
    if (tid == 0) atomicOr(&g_tc_status, *abort_flag);
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// S_end += S_start, element by element (the correction of an empty segment: Gamma = 1).
__global__ void __launch_bounds__(256)
ls_add_kernel(float* __restrict__ S_end, const float* __restrict__ S_start, long long n) {
  for (long long i = (long long)blockIdx.x * 256 + threadIdx.x; i < n; i += (long long)gridDim.x * 256)
    S_end[i] += S_start[i];
}

}  // namespace

bool tc_supported(int dk, int dv, int C, int bf16) {
  return bf16 && dk == kD && dv == kD && C == kC;
}

int tc_launches(const FwdArgs&) { return 1; }

bool linear_correct_supported(int dk, int dv, int bf16) { return tc_supported(dk, dv, kC, bf16); }

cudaError_t launch_linear_correct(const void* q, const float* log_alpha, const float* S_start,
                                  void* out, float* S_end, int B, int H, int T,
                                  cudaStream_t stream) {
  const long long units = (long long)B * H, rows = (long long)B * T;
  if (units <= 0) return cudaSuccess;
  if (rows > 0x7fffffffLL || units > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (T == 0) {  // an empty segment: Gamma = 1 and no outputs
    if (!S_end) return cudaSuccess;
    const long long n = units * kD * kD;
    ls_add_kernel<<<(unsigned)std::min<long long>((n + 255) / 256, 4096), 256, 0, stream>>>(
        S_end, S_start, n);
    return cudaGetLastError();
  }
  static std::atomic<unsigned long long> smem_corr{0};
  cudaError_t e = ensure_smem_cap(ls_corr_kernel, kLsSmem, smem_corr, true);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  CUtensorMap mq, mo;
  if (!make_map(&mq, q, rows, H) || !make_map(&mo, out, rows, H)) return cudaErrorInvalidValue;
  // the split's grid rule with each whole sequence as the one corrected segment
  const long long slots = 2LL * sms;
  const int cps = units <= slots ? (int)std::min<long long>(slots / units, (T + 63) / 64) : 0;
  const unsigned grid = (unsigned)(cps > 0 ? units * cps : slots);
  ls_corr_kernel<<<grid, kLsThreads, kLsSmem, stream>>>(mq, mo, B, H, T, 2, cps, log_alpha,
                                                        nullptr, S_end, S_start,
                                                        (__nv_bfloat16*)out);
  return cudaGetLastError();
}


// Segments per sequence of the linear mode's split (1: no split): as many as the SMs
// hold beside the N H units (at most kLsMaxSeg), each with at least two chunks.
int linear_split_segments(long long N, int H, int T) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 1;
  const long long units = N * H;
  if (units <= 0 || 2 * units > sms) return 1;
  int R = (int)std::min<long long>(kLsMaxSeg, sms / units);
  const int nch = (T + kC - 1) / kC;
  while (R > 1 && nch < 2 * R) --R;
  if (R > 1) R = (nch + (nch + R - 1) / R - 1) / ((nch + R - 1) / R);  // none left empty
  return R;
}

cudaError_t launch_tc(const FwdArgs& a, cudaStream_t stream) {
  const long long rows = (long long)a.B * a.T;
  if (rows == 0) return launch_rec(a, stream);  // nothing to load: state copy only
  if (rows > 0x7fffffffLL) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, rows, a.H) || !make_map(&mk, a.k, rows, a.H) ||
      !make_map(&mv, a.v, rows, a.H))
    return cudaErrorInvalidValue;
  if (a.beta == nullptr) {  // linear mode: the state CTA alone, one per unit
    const long long units = (long long)a.N * a.H;
    if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    static std::atomic<unsigned long long> smem_lin{0}, smem_corr{0};
    cudaError_t e = ensure_smem_cap(gdn_tc_linear_kernel, SMEM_BYTES, smem_lin);
    if (e != cudaSuccess) return e;
    const int R = a.cu_seqlens ? 1 : linear_split_segments(a.N, a.H, a.T);
    if (R <= 1) {
      gdn_tc_linear_kernel<<<(unsigned)units, kThreads, SMEM_BYTES, stream>>>(
          mq, mk, mv, a.log_alpha, a.S0, (__nv_bfloat16*)a.out, a.S_final, a.cu_seqlens, a.H,
          a.T, 1);
      return cudaGetLastError();
    }
    // R whole-chunk segments per sequence on more SMs, then the correction (which folds
    // the start states and writes S_final); the segments' end states L in pool scratch
    if ((e = ensure_smem_cap(ls_corr_kernel, kLsSmem, smem_corr, true)) != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    void* Lv = nullptr;
    if ((e = scratch_alloc(&Lv, (size_t)units * R * kD * kD * sizeof(float), stream)) != cudaSuccess)
      return e;
    float* L = static_cast<float*>(Lv);
    // two correction CTAs an SM: a share of one segment each when there are enough, else
    // runs of whole segments
    const long long nseg = units * (R - 1), slots = 2LL * sms;
    const int cps = nseg <= slots ? (int)std::min<long long>(slots / nseg, seg_tiles(a.T, R, 1)) : 0;
    const unsigned grid = (unsigned)(cps > 0 ? nseg * cps : slots);
    CUtensorMap mo;
    e = make_map(&mo, a.out, rows, a.H) ? cudaSuccess : cudaErrorInvalidValue;
    if (e == cudaSuccess) {
      gdn_tc_linear_kernel<<<(unsigned)(units * R), kThreads, SMEM_BYTES, stream>>>(
          mq, mk, mv, a.log_alpha, a.S0, (__nv_bfloat16*)a.out, L, nullptr, a.H, a.T, R);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) {
      ls_corr_kernel<<<grid, kLsThreads, kLsSmem, stream>>>(
          mq, mo, a.N, a.H, a.T, R, cps, a.log_alpha, L, a.S_final, nullptr,
          (__nv_bfloat16*)a.out);
      e = cudaGetLastError();
    }
    const cudaError_t ef = cudaFreeAsync(Lv, stream);
    return e != cudaSuccess ? e : ef;
  }
  const long long blocks = 2LL * a.N * a.H;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  static std::atomic<unsigned long long> smem_set{0};
  const cudaError_t e = ensure_smem_cap(gdn_tc_kernel, SMEM_BYTES, smem_set);
  if (e != cudaSuccess) return e;
  gdn_tc_kernel<<<(unsigned)blocks, kThreads, SMEM_BYTES, stream>>>(
      mq, mk, mv, a.log_alpha, a.beta, a.S0, (__nv_bfloat16*)a.out, a.S_final, a.cu_seqlens, a.H,
      a.T);
  return cudaGetLastError();
}

// Self-test of the failure-detection path: one thread waits, through the same
// bounded wait the kernels use, on an mbarrier that nothing arrives on.  The wait
// gives up after its limit (kWaitNs), records ST_WAIT, and the kernel publishes it in
// the status word as the forward kernel does on a failed wait, then returns.
__global__ void gdn_wait_selftest_kernel() {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int flag;
  volatile int* abort_flag = &flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    *abort_flag = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0 && !wait_bar(&bar, 0, abort_flag, false))
    atomicOr(&g_tc_status, *abort_flag);
}

cudaError_t launch_wait_selftest(cudaStream_t stream) {
  gdn_wait_selftest_kernel<<<1, 32, 0, stream>>>();
  return cudaGetLastError();
}

cudaError_t tc_status_address(int** ptr) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static int* addr[kMaxDev] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_tc_status)) != cudaSuccess) return e;
    addr[dev] = static_cast<int*>(p);
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

int tc_read_and_clear_status(cudaStream_t stream, cudaError_t* err) {
  int v = 0;
  *err = cudaMemcpyFromSymbolAsync(&v, g_tc_status, sizeof(int), 0, cudaMemcpyDeviceToHost, stream);
  if (*err == cudaSuccess) *err = cudaStreamSynchronize(stream);
  if (*err != cudaSuccess || v == 0) return v;
  const int zero = 0;
  *err = cudaMemcpyToSymbolAsync(g_tc_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream);
  if (*err == cudaSuccess) *err = cudaStreamSynchronize(stream);
  return v;
}

}  // namespace gdn
