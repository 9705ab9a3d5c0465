// tcgen05 tensor-core chunkwise Gated DeltaNet forward: bf16 q/k/v/out, fp32
// gates and state, dk = dv = 128, chunk C = 64.
//
// One CTA owns one (sequence, head) and its whole 128 x 128 fp32 state, and walks
// the sequence's chunks in order (Nyysyyan, "Chunk Computation").  Every
// contraction runs on the tensor cores with M = 128 (dk or dv as M):
//
//   [K;Q] K^T         -> K K^T (rows 0..63) and Q K^T (rows 64..127)      MMA-A
//   A = strictly-lower(beta_i e^{g_i-g_j} k_i.k_j), P = lower(e^{g_t-g_j} q_t.k_j)
//   T = (I + A)^{-1}  (blocked forward substitution, fp32, shared memory)
//   W~^T = K^T (T diag(beta e^g))^T,  U^T = V^T (T diag(beta))^T,  S Q^T    MMA-B
//   delta^T = U^T - S W~^T           (accumulated onto U^T in TMEM)     MMA-C
//   delta^T P^T,  dS = (delta diag(e^{g_last-g}))^T K                    MMA-D
//   o_t = e^{g_t} (S Q^T)_t + (delta^T P^T)_t,  S <- e^{g_last} S + dS
//
// The WY factors use the decayed triangular factor (myhz0606, "DeltaNet的
// Chunkwise Form推导", section 4.5; Nyysyyan, "Gated-DeltaNet": the U
// recursion with gamma_i / gamma_s, and W~ = gamma_i w_i).
//
// Precision: operands are bf16 in 128-byte-swizzled shared memory and
// accumulators fp32 in tensor memory.  T, delta, the decayed delta and P are
// carried as two bf16 terms (hi = bf16(x), lo = bf16(x - hi)) and multiplied as
// hi*hi + hi*lo + lo*hi (or hi + lo against an exact bf16 operand), which keeps
// their rounding near 2^-16; the state S and W~ are single bf16 operands.  The
// running state stays fp32 in registers.
//
// Every wait is bounded; a wait that gives up records a code in a device status
// word and the CTA leaves the chunk loop after its copies in flight have landed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_internal.h"
#include "tc_ptx.cuh"

namespace gdn {

__device__ int g_tc_status = 0;

namespace {

using namespace ptx;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kThreads = 256;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait

// Shared memory map (bytes from a 1024-aligned base).
constexpr int OFF_KQ = 0;          // 2 stages x 32 KB; per dk panel p: K rows (8 KB), Q rows (8 KB)
constexpr int KQ_STAGE = 32768;
constexpr int OFF_V = 65536;       // 16 KB: 2 dv panels of 64 token rows
constexpr int OFF_SB = 81920;      // S bf16 [128 dv][128 dk], 2 K panels of 16 KB
constexpr int OFF_WT = 114688;     // -W~^T bf16 [128 dk][64 tok] (MN-major B); later output staging
constexpr int OFF_PH = 131072;     // P hi bf16 [64 t][64 j] (K-major B)
constexpr int OFF_PL = 139264;     // P lo
constexpr int OFF_AR = 147456;     // 64 KB arena
//   prep phase:  A/T fp32 [64][68] | X fp32 [3][16][16] | Tw hi, Tw lo, Tu hi, Tu lo bf16 [64][64]
constexpr int LDA = 68;
constexpr int AR_A = 0;
constexpr int AR_X = 64 * LDA * 4;           // 17408
constexpr int AR_TWH = 20480;
constexpr int AR_TWL = AR_TWH + 8192;
constexpr int AR_TUH = AR_TWL + 8192;
constexpr int AR_TUL = AR_TUH + 8192;        // ends at 53248
//   state phase: delta hi, delta lo, decayed delta hi, lo, bf16 [128 dv][64 tok] (K-major A)
constexpr int AR_DH = 0;
constexpr int AR_DL = 16384;
constexpr int AR_DSH = 32768;
constexpr int AR_DSL = 49152;
constexpr int OFF_RAW = OFF_AR + 65536;      // raw gates [2 stages][la 64 | beta 64]
constexpr int OFF_DER = OFF_RAW + 1024;      // G, EG, ED, BG, BE, SCAN [6][64] fp32
constexpr int OFF_BAR = OFF_DER + 1536;
constexpr int OFF_MISC = OFF_BAR + 64;
constexpr int SMEM_USED = OFF_MISC + 64;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack for aligning the base
static_assert(AR_TUL + 8192 <= 65536, "arena");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// TMEM columns (fp32 accumulators, 128 lanes each).
constexpr uint32_t TM_KQ = 0;      // [K K^T ; Q K^T]   64 cols
constexpr uint32_t TM_W = 64;      // W~^T               64
constexpr uint32_t TM_U = 128;     // U^T, then delta^T  64
constexpr uint32_t TM_SQ = 192;    // S Q^T              64
constexpr uint32_t TM_DP = 256;    // delta^T P^T        64
constexpr uint32_t TM_DS = 320;    // dS                 128
constexpr uint32_t TM_COLS = 512;

constexpr int ST_WAIT_KQ = 1, ST_WAIT_V = 2, ST_WAIT_MMA = 4;

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
// Store 8 consecutive columns (col % 8 == 0) of `row` into a 128B-swizzled bf16 tile.
__device__ __forceinline__ void st_sw128_8(uint8_t* tile, int row, int col, int rows,
                                           const float* v) {
  st_shared_v4(smem_u32(tile + sw128_offset(row, col, rows)), pack_bf16(v[0], v[1]),
               pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
}
// Same, as two bf16 terms: hi = bf16(v), lo = bf16(v - hi).
__device__ __forceinline__ void st_sw128_8_split(uint8_t* hi_tile, uint8_t* lo_tile, int row,
                                                 int col, int rows, const float* v) {
  float hi[8], lo[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    hi[u] = __bfloat162float(__float2bfloat16_rn(v[u]));
    lo[u] = v[u] - hi[u];
  }
  st_sw128_8(hi_tile, row, col, rows, hi);
  st_sw128_8(lo_tile, row, col, rows, lo);
}

// K-major operand, 128B swizzle, K advanced by 16 elements per step.
__device__ __forceinline__ uint64_t desc_k(const uint8_t* tile, int kstep, int panel_bytes) {
  return smem_desc(smem_u32(tile) + (kstep >> 2) * panel_bytes + (kstep & 3) * 32, 16, 1024);
}
// MN-major operand stored as [K rows][MN cols] in 64-column panels, K advanced by 16 rows.
__device__ __forceinline__ uint64_t desc_mn(const uint8_t* tile, int kstep, int panel_bytes) {
  return smem_desc(smem_u32(tile) + kstep * 2048, panel_bytes, 1024);
}

constexpr float kLog2e = 1.4426950408889634f;
// 2^x by the PTX ex2.approx instruction (flushes subnormal results to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}

__global__ void __launch_bounds__(kThreads, 1)
gdn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const float* __restrict__ log_alpha,
              const float* __restrict__ beta, const float* __restrict__ S0,
              __nv_bfloat16* __restrict__ out, float* __restrict__ S_final,
              const int32_t* __restrict__ cu_seqlens, int H, int T) {
  extern __shared__ uint8_t smem_raw[];
  // Align to 1024 bytes by pointer arithmetic on the shared array itself, so that
  // every access below stays a shared-memory (not generic) access.
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* AR = sm + OFF_AR;
  float* Am = reinterpret_cast<float*>(AR + AR_A);   // A, then T in place
  float* Xs = reinterpret_cast<float*>(AR + AR_X);
  float* raw = reinterpret_cast<float*>(sm + OFF_RAW);
  float* G = reinterpret_cast<float*>(sm + OFF_DER);
  float* EG = G + 64;
  float* ED = G + 128;
  float* BG = G + 192;
  float* BE = G + 256;
  float* SCAN = G + 320;
  uint64_t* bar_kq = reinterpret_cast<uint64_t*>(sm + OFF_BAR);  // [2]
  uint64_t* bar_v = bar_kq + 2;
  uint64_t* bar_mma = bar_kq + 3;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + OFF_MISC + 4);
  __nv_bfloat16* ost = reinterpret_cast<__nv_bfloat16*>(sm + OFF_WT);  // output staging [64][128]

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3;          // TMEM lane quarter this warp may access
  const int half = warp >> 2;         // column half this warp handles
  const int row = quad * 32 + lane;   // TMEM lane = accumulator row
  const int h = blockIdx.x % H;
  const int n = blockIdx.x / H;

  long long row0, len;
  if (cu_seqlens) {
    int a = cu_seqlens[n], b = cu_seqlens[n + 1];
    a = min(max(a, 0), T);
    b = min(max(b, a), T);
    row0 = a;
    len = b - a;
  } else {
    row0 = (long long)n * T;
    len = T;
  }
  const int nc = (int)((len + kC - 1) / kC);

  if (warp == 0) tmem_alloc(tslot, TM_COLS);
  if (tid == 0) {
    mbar_init(&bar_kq[0], 1);
    mbar_init(&bar_kq[1], 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_mma, 1);
    *s_abort = 0;
    fence_mbarrier_init();
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
  }

  // Running state: this thread holds S[row][64*half .. 64*half + 63] in fp32.
  float S[64];
  const size_t sidx = (((size_t)n * H + h) * kD + row) * kD + 64 * half;
  if (S0) {
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const float4 t4 = *reinterpret_cast<const float4*>(S0 + sidx + 4 * q);
      S[4 * q] = t4.x; S[4 * q + 1] = t4.y; S[4 * q + 2] = t4.z; S[4 * q + 3] = t4.w;
    }
  } else {
#pragma unroll
    for (int q = 0; q < 64; ++q) S[q] = 0.f;
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) st_sw128_8(sm + OFF_SB, row, 64 * half + 8 * q, 128, S + 8 * q);

  // Gate values of one chunk: thread t in [0, 64) of a 64-thread group loads token t.
  auto fetch_gates = [&](int chunk, float& la, float& be) {
    const int t = tid & 63;
    const long long c0 = (long long)chunk * kC;
    la = 0.f;
    be = 0.f;
    if (c0 + t < len) {
      const size_t gi = (size_t)(row0 + c0 + t) * H + h;
      la = __ldg(log_alpha + gi);
      be = __ldg(beta + gi);
    }
  };
  auto issue_kq = [&](int chunk, int stage) {
    const int r = (int)(row0 + (long long)chunk * kC);
    uint8_t* base = sm + OFF_KQ + stage * KQ_STAGE;
    mbar_arrive_expect_tx(&bar_kq[stage], 4 * 8192);
    tma_load_3d(base, &tm_k, &bar_kq[stage], 0, h, r);
    tma_load_3d(base + 8192, &tm_q, &bar_kq[stage], 0, h, r);
    tma_load_3d(base + 16384, &tm_k, &bar_kq[stage], 64, h, r);
    tma_load_3d(base + 16384 + 8192, &tm_q, &bar_kq[stage], 64, h, r);
  };
  auto issue_v = [&](int chunk) {
    const int r = (int)(row0 + (long long)chunk * kC);
    mbar_arrive_expect_tx(bar_v, 2 * 8192);
    tma_load_3d(sm + OFF_V, &tm_v, bar_v, 0, h, r);
    tma_load_3d(sm + OFF_V + 8192, &tm_v, bar_v, 64, h, r);
  };

  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16);  // this warp's lane quarter

  // Copies in flight and the mbarrier parity each will complete (for a clean abort).
  int kq_pending[2] = {0, 0}, kq_par[2] = {0, 0};
  int v_pending = 0, v_par = 0;
  if (nc > 0) {
    if (tid == 0) { issue_kq(0, 0); issue_v(0); }
    kq_pending[0] = 1;
    v_pending = 1;
    if (tid < 64) {
      float la, be;
      fetch_gates(0, la, be);
      raw[tid] = la;
      raw[64 + tid] = be;
    }
  }
  uint32_t mma_phase = 0;
  bool aborted = false;

  // Wait for the MMA batch just committed; every thread leaves together.
  auto wait_mma = [&]() -> bool {
    const bool ok = mbar_wait(bar_mma, mma_phase, kWaitNs);
    mma_phase ^= 1;
    if (!ok) atomicOr((int*)s_abort, ST_WAIT_MMA);
    tc_fence_after();
    __syncthreads();
    return *s_abort == 0;
  };

  for (int j = 0; j < nc; ++j) {
    const int s = j & 1;
    const long long c0 = (long long)j * kC;
    const int lc = (int)min((long long)kC, len - c0);
    uint8_t* KQ = sm + OFF_KQ + s * KQ_STAGE;

    // ---- prefetch chunk j+1: K, Q by TMA; gates into registers (stored at chunk end) ----
    float nla = 0.f, nbe = 0.f;
    if (j + 1 < nc) {
      if (tid == 0) issue_kq(j + 1, s ^ 1);
      kq_pending[s ^ 1] = 1;
      kq_par[s ^ 1] = ((j + 1) >> 1) & 1;
      if (tid >= 64 && tid < 128) fetch_gates(j + 1, nla, nbe);
    }

    // ---- gates: in-chunk cumsum of log alpha and the derived factors ----
    {
      const bool ok = mbar_wait(&bar_kq[s], (j >> 1) & 1, kWaitNs);
      if (ok) kq_pending[s] = 0;
      if (!ok) atomicOr((int*)s_abort, ST_WAIT_KQ);
      if (tid < 64) {
        float x = raw[s * 128 + tid];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        SCAN[tid] = x;
      }
      __syncthreads();
      if (*s_abort) { aborted = true; break; }
      if (tid < 64) {
        // gate sums in log2 units, so every decay factor is one ex2
        const float total = (SCAN[31] + SCAN[63]) * kLog2e;
        const float g = (SCAN[tid] + (tid >= 32 ? SCAN[31] : 0.f)) * kLog2e;
        const float b = raw[s * 128 + 64 + tid];
        const float eg = ex2(g);
        G[tid] = g;
        EG[tid] = eg;
        ED[tid] = ex2(total - g);
        BG[tid] = b * eg;
        BE[tid] = b;
      }
      __syncthreads();
    }

    // ---- MMA-A: [K;Q] K^T ----
    if (tid == 0) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, 64, 0, 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_bf16(tmem + TM_KQ, desc_k(KQ, kk, 16384), desc_k(KQ, kk, 16384), idesc, kk > 0);
      mma_commit(bar_mma);
    }
    if (!wait_mma()) { aborted = true; break; }

    // ---- epilogue A: decayed, beta-scaled, masked A (fp32) and P (bf16 hi/lo) ----
    {
      uint32_t r[32];
      tmem_ld32(tq + TM_KQ + 32 * half, r);
      float gc[32];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 g4 = ld4(G + 32 * half + 4 * q);
        gc[4 * q] = g4.x; gc[4 * q + 1] = g4.y; gc[4 * q + 2] = g4.z; gc[4 * q + 3] = g4.w;
      }
      tmem_wait_ld();
      if (quad < 2) {
        const int i = row;
        const float gi = G[i], bi = BE[i];
        float* arow = Am + i * LDA + 32 * half;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int jc = 32 * half + 4 * q + u;
            v[u] = (jc < i) ? bi * ex2(gi - gc[4 * q + u]) * __uint_as_float(r[4 * q + u]) : 0.f;
          }
          st4(arow + 4 * q, v[0], v[1], v[2], v[3]);
        }
      } else {
        const int t = row - 64;
        const float gt = G[t];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int jc = 32 * half + 8 * q + u;
            v[u] = (jc <= t) ? ex2(gt - gc[8 * q + u]) * __uint_as_float(r[8 * q + u]) : 0.f;
          }
          st_sw128_8_split(sm + OFF_PH, sm + OFF_PL, t, 32 * half + 8 * q, 64, v);
        }
      }
    }
    __syncthreads();

    // ---- T = (I + A)^{-1}, in place over A ----
    // 16 x 16 diagonal blocks: one thread per column, then written back together.
    if (tid < 64) {
      const int b = tid >> 4, c = tid & 15;
      const float* Ab = Am + (16 * b) * LDA + 16 * b;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float acc = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int m = 0; m < r; ++m) acc = fmaf(-Ab[r * LDA + m], x[m], acc);
        x[r] = acc;
      }
      asm volatile("bar.sync 1, 64;" ::: "memory");
      float* Tb = Am + (16 * b) * LDA + 16 * b + c;
#pragma unroll
      for (int r = 0; r < 16; ++r) Tb[r * LDA] = x[r];
    }
    __syncthreads();
    // Block rows ib = 1..3: X_{ib,jb} = sum_{kb=jb}^{ib-1} A_{ib,kb} T_{kb,jb}, then
    // T_{ib,jb} = -T_{ib,ib} X_{ib,jb}; each thread owns a 1 x 4 strip.
#pragma unroll 1
    for (int ib = 1; ib < 4; ++ib) {
      const bool active = tid < ib * 64;
      const int jb = tid >> 6, r = (tid >> 2) & 15, cq = tid & 3;
      if (active) {
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
      __syncthreads();
      if (active) {
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
      __syncthreads();
    }

    // ---- T diag(beta e^g) and T diag(beta) as bf16 hi/lo B operands ----
#pragma unroll
    for (int it0 = 0; it0 < 512; it0 += kThreads) {
      const int it = it0 + tid;
      const int i = it >> 3, jc = (it & 7) * 8;
      const float4 ta = ld4(Am + i * LDA + jc), tb = ld4(Am + i * LDA + jc + 4);
      const float tv[8] = {ta.x, ta.y, ta.z, ta.w, tb.x, tb.y, tb.z, tb.w};
      const float4 bg0 = ld4(BG + jc), bg1 = ld4(BG + jc + 4);
      const float4 be0 = ld4(BE + jc), be1 = ld4(BE + jc + 4);
      const float bgv[8] = {bg0.x, bg0.y, bg0.z, bg0.w, bg1.x, bg1.y, bg1.z, bg1.w};
      const float bev[8] = {be0.x, be0.y, be0.z, be0.w, be1.x, be1.y, be1.z, be1.w};
      float tw[8], tu[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float t = (jc + u <= i) ? tv[u] : 0.f;
        tw[u] = t * bgv[u];
        tu[u] = t * bev[u];
      }
      st_sw128_8_split(AR + AR_TWH, AR + AR_TWL, i, jc, 64, tw);
      st_sw128_8_split(AR + AR_TUH, AR + AR_TUL, i, jc, 64, tu);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA-B: W~^T = K^T Tw^T, U^T = V^T Tu^T (hi + lo), S Q^T ----
    {
      const bool ok = mbar_wait(bar_v, j & 1, kWaitNs);
      if (ok) v_pending = 0;
      if (!ok) atomicOr((int*)s_abort, ST_WAIT_V);
      __syncthreads();
      if (*s_abort) { aborted = true; break; }
    }
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id_t = idesc_bf16(128, 64, 1, 0);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ak = desc_mn(KQ, kk, 16384);
        const uint64_t av = desc_mn(sm + OFF_V, kk, 8192);
        mma_bf16(tmem + TM_W, ak, desc_k(AR + AR_TWH, kk, 8192), id_t, kk > 0);
        mma_bf16(tmem + TM_W, ak, desc_k(AR + AR_TWL, kk, 8192), id_t, 1);
        mma_bf16(tmem + TM_U, av, desc_k(AR + AR_TUH, kk, 8192), id_t, kk > 0);
        mma_bf16(tmem + TM_U, av, desc_k(AR + AR_TUL, kk, 8192), id_t, 1);
      }
      const uint32_t id_sq = idesc_bf16(128, 64, 0, 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_bf16(tmem + TM_SQ, desc_k(sm + OFF_SB, kk, 16384), desc_k(KQ + 8192, kk, 16384), id_sq,
                 kk > 0);
      mma_commit(bar_mma);
    }
    if (!wait_mma()) { aborted = true; break; }
    if (j + 1 < nc) {
      if (tid == 0) issue_v(j + 1);  // the V buffer is free: MMA-B has completed
      v_pending = 1;
      v_par = (j + 1) & 1;
    }

    // ---- epilogue B: -W~^T as the bf16 MN-major B operand [dk][tok] ----
    {
      uint32_t r[32];
      tmem_ld32(tq + TM_W + 32 * half, r);
      tmem_wait_ld();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = -__uint_as_float(r[8 * q + u]);
        st_sw128_8(sm + OFF_WT, row, 32 * half + 8 * q, 128, v);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA-C: delta^T = U^T + S (-W~^T) ----
    if (tid == 0) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, 64, 0, 1);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_bf16(tmem + TM_U, desc_k(sm + OFF_SB, kk, 16384), desc_mn(sm + OFF_WT, kk, 16384),
                 idesc, 1);
      mma_commit(bar_mma);
    }
    if (!wait_mma()) { aborted = true; break; }

    // ---- epilogue C: delta^T and its decayed copy as bf16 hi/lo A operands ----
    {
      uint32_t r[32];
      tmem_ld32(tq + TM_U + 32 * half, r);
      float ed[32];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 e4 = ld4(ED + 32 * half + 4 * q);
        ed[4 * q] = e4.x; ed[4 * q + 1] = e4.y; ed[4 * q + 2] = e4.z; ed[4 * q + 3] = e4.w;
      }
      tmem_wait_ld();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float v[8], w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          v[u] = __uint_as_float(r[8 * q + u]);
          w[u] = v[u] * ed[8 * q + u];
        }
        st_sw128_8_split(AR + AR_DH, AR + AR_DL, row, 32 * half + 8 * q, 128, v);
        st_sw128_8_split(AR + AR_DSH, AR + AR_DSL, row, 32 * half + 8 * q, 128, w);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA-D: delta^T P^T and dS = delta~^T K (hi/lo terms) ----
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id_dp = idesc_bf16(128, 64, 0, 0);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t dh = desc_k(AR + AR_DH, kk, 16384), dl = desc_k(AR + AR_DL, kk, 16384);
        const uint64_t ph = desc_k(sm + OFF_PH, kk, 8192), pl = desc_k(sm + OFF_PL, kk, 8192);
        mma_bf16(tmem + TM_DP, dh, ph, id_dp, kk > 0);
        mma_bf16(tmem + TM_DP, dh, pl, id_dp, 1);
        mma_bf16(tmem + TM_DP, dl, ph, id_dp, 1);
      }
      const uint32_t id_ds = idesc_bf16(128, 128, 0, 1);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t kb = desc_mn(KQ, kk, 16384);
        mma_bf16(tmem + TM_DS, desc_k(AR + AR_DSH, kk, 16384), kb, id_ds, kk > 0);
        mma_bf16(tmem + TM_DS, desc_k(AR + AR_DSL, kk, 16384), kb, id_ds, 1);
      }
      mma_commit(bar_mma);
    }
    if (!wait_mma()) { aborted = true; break; }

    // ---- epilogue D: outputs (staged in shared memory) and the state update ----
    {
      uint32_t a[32], b[32];
      tmem_ld32(tq + TM_SQ + 32 * half, a);
      tmem_ld32(tq + TM_DP + 32 * half, b);
      float eg[32];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 e4 = ld4(EG + 32 * half + 4 * q);
        eg[4 * q] = e4.x; eg[4 * q + 1] = e4.y; eg[4 * q + 2] = e4.z; eg[4 * q + 3] = e4.w;
      }
      tmem_wait_ld();
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        const int t = 32 * half + jj;
        ost[t * kD + row] =
            __float2bfloat16_rn(fmaf(eg[jj], __uint_as_float(a[jj]), __uint_as_float(b[jj])));
      }
      const float gam = EG[63];
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        uint32_t d[32];
        tmem_ld32(tq + TM_DS + 64 * half + 32 * p, d);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 32; ++u) S[32 * p + u] = fmaf(gam, S[32 * p + u], __uint_as_float(d[u]));
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) st_sw128_8(sm + OFF_SB, row, 64 * half + 8 * q, 128, S + 8 * q);
      if (j + 1 < nc && tid >= 64 && tid < 128) {
        raw[(s ^ 1) * 128 + (tid - 64)] = nla;
        raw[(s ^ 1) * 128 + 64 + (tid - 64)] = nbe;
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    // coalesced copy of the valid output rows: 16 bytes per thread per step
    {
      const size_t obase = (size_t)(row0 + c0) * H + h;
#pragma unroll
      for (int it0 = 0; it0 < 1024; it0 += kThreads) {
        const int it = it0 + tid;
        const int t = it >> 4, ch = it & 15;
        if (t < lc) {
          const uint4 v = *reinterpret_cast<const uint4*>(ost + t * kD + 8 * ch);
          *reinterpret_cast<uint4*>(out + (obase + (size_t)t * H) * kD + 8 * ch) = v;
        }
      }
    }
  }

  if (aborted) {
    // Let copies still in flight land before the CTA's shared memory goes away.
    if (tid == 0) {
      for (int st = 0; st < 2; ++st)
        if (kq_pending[st]) (void)mbar_wait(&bar_kq[st], kq_par[st], 100000000ull);
      if (v_pending) (void)mbar_wait(bar_v, v_par, 100000000ull);
      atomicOr(&g_tc_status, *s_abort);
    }
  } else if (S_final) {
#pragma unroll
    for (int q = 0; q < 16; ++q)
      *reinterpret_cast<float4*>(S_final + sidx + 4 * q) =
          make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [rows][H][128] bf16, box of 64 columns x 1 head x 64 rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, long long rows, int H) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace

bool tc_supported(int dk, int dv, int C, int bf16) {
  return bf16 && dk == kD && dv == kD && C == kC;
}

int tc_launches(const FwdArgs&) { return 1; }

cudaError_t launch_tc(const FwdArgs& a, cudaStream_t stream) {
  const long long rows = (long long)a.B * a.T;
  if (rows == 0) return launch_simt(a, stream);  // nothing to load: state copy only
  if (rows > 0x7fffffffLL) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, rows, a.H) || !make_map(&mk, a.k, rows, a.H) ||
      !make_map(&mv, a.v, rows, a.H))
    return cudaErrorInvalidValue;
  const long long blocks = (long long)a.N * a.H;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(gdn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES);
  if (e != cudaSuccess) return e;
  gdn_tc_kernel<<<(unsigned)blocks, kThreads, SMEM_BYTES, stream>>>(
      mq, mk, mv, a.log_alpha, a.beta, a.S0, (__nv_bfloat16*)a.out, a.S_final, a.cu_seqlens, a.H,
      a.T);
  return cudaGetLastError();
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
