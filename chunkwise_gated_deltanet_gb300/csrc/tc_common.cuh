// Device and host helpers shared by the tcgen05 chunk kernels (gdn_tc.cu: the linear
// mode; gdn_fwd.cu: the delta rule): gate scans, operand packing and shared-memory
// descriptors, bounded mbarrier waits, MMA issue loops, the (sequence, head) unit of a
// launch, and the TMA tensor maps of q, k, v.  Every translation unit that includes it
// gets its own private copies (unnamed namespace).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tc_ptx.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait


// The factored decay e^{g_i} e^{-g_j} replaces e^{g_i - g_j} when the chunk's
// total decay (in log2 units) is below this bound, so that neither factor
// overflows or underflows fp32.
constexpr float kMaxFactoredDecayLog2 = 80.f;

constexpr int ST_WAIT = 1;

constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float ex2(float x) {  // 2^x by the PTX ex2.approx instruction
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
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
// 8 consecutive columns (col % 8 == 0) of `row` into a 128B-swizzled bf16 tile.
__device__ __forceinline__ void st_sw128_8(uint8_t* tile, int row, int col, int rows,
                                           const float* v) {
  st_shared_v4(smem_u32(tile + sw128_offset(row, col, rows)), pack_bf16(v[0], v[1]),
               pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
}
// Two floats as a pair of packed bf16 terms: hi = bf16(x), lo = bf16(x - hi).
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(x0, x1);
  const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xffff0000u);
  lo = pack_bf16(x0 - h0, x1 - h1);
}
__device__ __forceinline__ void st_sw128_8_split(uint8_t* hi_tile, uint8_t* lo_tile, int row,
                                                 int col, int rows, const float* v) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) split2(v[2 * u], v[2 * u + 1], h[u], l[u]);
  const uint32_t off = sw128_offset(row, col, rows);
  st_shared_v4(smem_u32(hi_tile + off), h[0], h[1], h[2], h[3]);
  st_shared_v4(smem_u32(lo_tile + off), l[0], l[1], l[2], l[3]);
}
// K-major operand, 128B swizzle, K advanced by 16 elements per step.
__device__ __forceinline__ uint64_t desc_k(const uint8_t* tile, int kstep, int panel_bytes) {
  return smem_desc(smem_u32(tile) + (kstep >> 2) * panel_bytes + (kstep & 3) * 32, 16, 1024);
}
// MN-major operand stored as [K rows][MN cols] in 64-column panels, K advanced by 16 rows.
__device__ __forceinline__ uint64_t desc_mn(const uint8_t* tile, int kstep, int panel_bytes) {
  return smem_desc(smem_u32(tile) + kstep * 2048, panel_bytes, 1024);
}
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}

// Bounded parity wait that also gives up when another role of this CTA already
// gave up.  Returns false on timeout (recording `code`) or on abort.  The polling
// loop is one shared out-of-line function; only the first test is inlined at
// each call site, which keeps the hot code of every role small.
__device__ __noinline__ bool wait_bar_poll(uint64_t* bar, uint32_t parity,
                                           volatile int* abort_flag, bool cluster_scope) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    const bool ok = cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    if (ok) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitNs) {
      atomicOr((int*)abort_flag, ST_WAIT);
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         bool cluster_scope) {
  const bool ok = cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  return ok || wait_bar_poll(bar, parity, abort_flag, cluster_scope);
}

// A bounded wait taken by every thread of a named-barrier group (`nb`, `nthreads`),
// followed by one vote: true when the group must leave its loop because its own wait
// gave up or another role already did.  Out of line, shared by all call sites.
__device__ __noinline__ bool group_wait_fails(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag, bool cluster_scope,
                                              uint32_t nb, uint32_t nthreads) {
  const bool ok = wait_bar(bar, parity, abort_flag, cluster_scope);
  return named_sync_or(nb, nthreads, !ok || *abort_flag != 0);
}
// Inline form for the latency-critical roles, over up to three barriers (a null
// barrier is skipped) with a single vote: every wait point that is not already
// satisfied costs a full round of the named barrier, so the chain merges the
// barriers it needs at the same point.
__device__ __forceinline__ bool group_waits_fail(volatile int* abort_flag, uint32_t nb,
                                                 uint32_t nthreads, uint64_t* b1, uint32_t p1,
                                                 bool c1, uint64_t* b2 = nullptr, uint32_t p2 = 0,
                                                 uint64_t* b3 = nullptr, uint32_t p3 = 0) {
  bool ok = wait_bar(b1, p1, abort_flag, c1);
  if (ok && b2) ok = wait_bar(b2, p2, abort_flag, false);
  if (ok && b3) ok = wait_bar(b3, p3, abort_flag, false);
  return named_sync_or(nb, nthreads, !ok || *abort_flag != 0);
}
// The same for a single warp.
__device__ __noinline__ bool warp_wait_fails(uint64_t* bar, uint32_t parity,
                                             volatile int* abort_flag, bool cluster_scope) {
  return !__all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, cluster_scope));
}

// MMA issue from one thread.  Descriptors are built once per operand and advanced
// by constants (16-byte units: 2 per k-step for a K-major operand, 128 for an
// MN-major one, whose k-step is 16 rows of 128 bytes); a tcgen05.mma then costs the
// issuing thread little beyond the tensor core's own rate.
constexpr uint32_t kStepK = 2;
constexpr uint32_t kStepMN = 128;
// K = 128 (8 k-steps): A K-major in two 64-column panels pa16 apart; B K-major in
// panels pb16 apart, or MN-major.  Rolled over the panels, 4 constant steps inside.
template <bool B_MN>
__device__ __forceinline__ void mma_k128(uint32_t d, uint64_t a, uint32_t pa16, uint64_t b,
                                         uint32_t pb16, uint32_t id, uint32_t acc_first) {
#pragma unroll 1
  for (int p = 0; p < 2; ++p) {
    const uint64_t ap = a + (uint64_t)(p * pa16);
    const uint64_t bp = b + (uint64_t)(B_MN ? p * 4 * kStepMN : p * pb16);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      mma_bf16(d, ap + kStepK * k, bp + (B_MN ? kStepMN : kStepK) * k, id, (p | k) ? 1u : acc_first);
  }
}
// Out-of-line form of mma_k128<false> followed by a commit, shared by the roles that
// are not on the serial path (one copy of the issue code in the instruction cache).
__device__ __noinline__ void mma_k128_commit(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                             uint64_t* bar) {
  tc_fence_after();
  mma_k128<false>(d, a, 16384 >> 4, b, 16384 >> 4, id, 0);
  mma_commit(bar);
}
// K = 64 (4 k-steps): A from TMEM (8 columns per step) or MN-major smem; B K-major
// or MN-major.  UNROLL for the chain's own MMAs, rolled elsewhere.
template <bool A_TMEM, bool B_MN, bool UNROLL>
__device__ __forceinline__ void mma_k64(uint32_t d, uint64_t a, uint32_t a_tmem, uint64_t b,
                                        uint32_t id, uint32_t acc_first) {
  if (UNROLL) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint64_t bk = b + (B_MN ? kStepMN : kStepK) * k;
      if (A_TMEM)
        mma_bf16_ta(d, a_tmem + 8 * k, bk, id, k ? 1u : acc_first);
      else
        mma_bf16(d, a + kStepMN * k, bk, id, k ? 1u : acc_first);
    }
  } else {
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
      if (A_TMEM)
        mma_bf16_ta(d, a_tmem, b, id, k ? 1u : acc_first);
      else
        mma_bf16(d, a, b, id, k ? 1u : acc_first);
      a += kStepMN;
      a_tmem += 8;
      b += B_MN ? kStepMN : kStepK;
    }
  }
}

// Bounded wait until the hand-off ticket reaches `want`; false on timeout or abort.
__device__ __forceinline__ bool wait_ticket(volatile int* ticket, int want,
                                            volatile int* abort_flag) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (*ticket == want) return true;
    if (*abort_flag) return false;
    if (it == 0) {
      t0 = globaltimer_ns();
    } else if (globaltimer_ns() - t0 > kWaitNs) {
      atomicOr((int*)abort_flag, ST_WAIT);
      return false;
    }
  }
}

struct Unit {
  long long row0, len;
  int nc, h;
  size_t sidx;   // offset of S[n][h] in S_final
  size_t s0idx;  // and in S0
};

// Gate inputs of one chunk for a whole warp: thread `lane` owns tokens lane and
// lane + 32 (zeros past the sequence end).  Split from the scan so the loads of
// the next chunk can be in flight while the current one is processed.  A NULL
// log_alpha reads as alpha = 1; a NULL beta (the linear mode, erase 0) as a write
// strength of 1.
struct GateLoad {
  float la0, la1, b0, b1;
};
// A gate of alpha = 0 (log alpha = -inf, the whole state forgotten) enters as log alpha =
// -80: alpha = e^-80 ~ 1.8e-35 leaves nothing measurable of the earlier state, and the
// in-chunk gate sums and their differences stay finite (-inf - -inf would be NaN) and
// accurate (|sum| <= 80 * 64).
constexpr float kMinLogAlpha = -80.f;
__device__ __forceinline__ GateLoad load_gates(const float* __restrict__ log_alpha,
                                               const float* __restrict__ beta, const Unit& u, int H,
                                               int chunk, int lane) {
  GateLoad g{0.f, 0.f, 0.f, 0.f};
  const long long c0 = (long long)chunk * kC;
  if (chunk < u.nc && c0 + lane < u.len) {
    const size_t gi = (size_t)(u.row0 + c0 + lane) * H + u.h;
    g.la0 = log_alpha ? __ldg(log_alpha + gi) : 0.f;
    g.b0 = beta ? __ldg(beta + gi) : 1.f;
  }
  if (chunk < u.nc && c0 + lane + 32 < u.len) {
    const size_t gi = (size_t)(u.row0 + c0 + lane + 32) * H + u.h;
    g.la1 = log_alpha ? __ldg(log_alpha + gi) : 0.f;
    g.b1 = beta ? __ldg(beta + gi) : 1.f;
  }
  return g;
}
// In-chunk cumulative gate sums in log2 units (g0 for token lane, g1 for token
// lane + 32) and their total, each log alpha taken at least kMinLogAlpha.
__device__ __forceinline__ void scan_gates(const GateLoad& in, int lane, float& g0, float& g1,
                                           float& tot) {
  float x0 = fmaxf(in.la0, kMinLogAlpha), x1 = fmaxf(in.la1, kMinLogAlpha);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y0 = __shfl_up_sync(0xffffffffu, x0, o);
    const float y1 = __shfl_up_sync(0xffffffffu, x1, o);
    if (lane >= o) {
      x0 += y0;
      x1 += y1;
    }
  }
  const float t0 = __shfl_sync(0xffffffffu, x0, 31);
  const float t1 = __shfl_sync(0xffffffffu, x1, 31);
  g0 = x0 * kLog2e;
  g1 = (x1 + t0) * kLog2e;
  tot = (t0 + t1) * kLog2e;
}

// Row i of A = strictly-lower(beta_i e^{g_i - g_j} k_i.k_j) from the K K^T
// accumulator (two halves of 32 columns) into fp32 scratch.  FACTORED: ci =
// beta_i e^{g_i} and colv = e^{-g_j}; otherwise ci = beta_i, gi = g_i, colv = g_j.
// One instantiation per form keeps the hot form's code contiguous.
template <bool FACTORED>
__device__ __forceinline__ void wy_epi_a(uint32_t t_kk, float* arow, int i, float ci, float gi,
                                         const float* colv) {
#pragma unroll 1
  for (int hh = 0; hh < 2; ++hh) {
    uint32_t r[32];
    tmem_ld32(t_kk + 32 * hh, r);
    tmem_wait_ld();
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int jc0 = 32 * hh + 4 * q;
      const float4 c4 = ld4(colv + jc0);
      const float c[4] = {c4.x, c4.y, c4.z, c4.w};
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x = __uint_as_float(r[4 * q + e]);
        const float f = FACTORED ? ci * c[e] : ci * ex2(gi - c[e]);
        v[e] = (jc0 + e < i) ? f * x : 0.f;
      }
      st4(arow + jc0, v[0], v[1], v[2], v[3]);
    }
  }
}

// Row t of P (or P') from the Q K^T accumulator as hi/lo bf16 into a P slot.
// FACTORED: P'_{t,j} = q_t.k_j e^{-g_j} with colv = e^{-g_j}; otherwise
// P_{t,j} = q_t.k_j e^{g_t - g_j} with gt = g_t and colv = g_j.
template <bool FACTORED>
__device__ __forceinline__ void aux_epi_p(uint32_t t_qk, uint8_t* ps, int t, float gt,
                                          const float* colv, bool store) {
#pragma unroll 1
  for (int c = 0; c < 8; ++c) {  // columns 8c .. 8c + 7
    uint32_t r[8];
    tmem_ld8(t_qk + 8 * c, r);
    tmem_wait_ld();
    const int jc0 = 8 * c;
    const float4 ca = ld4(colv + jc0), cb = ld4(colv + jc0 + 4);
    const float cv[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float x = __uint_as_float(r[e]);
      v[e] = (jc0 + e <= t) ? (FACTORED ? x * cv[e] : ex2(gt - cv[e]) * x) : 0.f;
    }
    if (store) st_sw128_8_split(ps, ps + 8192, t, jc0, 64, v);
  }
}

// (sequence, head) unit `unit` = n * H + h: its rows (cu_seqlens clamped to [0, T]),
// chunk count and state offset.
__device__ __forceinline__ Unit make_unit(int unit, const int32_t* __restrict__ cu_seqlens, int H,
                                          int T) {
  Unit u;
  u.h = unit % H;
  const int n = unit / H;
  if (cu_seqlens) {
    int a = cu_seqlens[n], b = cu_seqlens[n + 1];
    a = min(max(a, 0), T);
    b = min(max(b, a), T);
    u.row0 = a;
    u.len = b - a;
  } else {
    u.row0 = (long long)n * T;
    u.len = T;
  }
  u.nc = (int)((u.len + kC - 1) / kC);
  u.sidx = ((size_t)n * H + u.h) * kD * kD;
  u.s0idx = u.sidx;
  return u;
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

// [rows][H][128] bf16, box of 64 columns x 1 head x 64 rows, 128-byte swizzle (or none:
// the box is then 64 rows of 128 plain bytes).
bool make_map(CUtensorMap* m, const void* base, long long rows, int H, bool swizzle = true) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}


}  // namespace
}  // namespace gdn
