// Chunked backward of the Gated DeltaNet recurrence (gradients of q, k, v, log alpha,
// beta and S0), the reverse-mode derivative of the chunk form (Nyysyyan,
// "Gated-DeltaNet", the WY representation and the chunkwise algorithm).  The pages derive
// no backward; this follows the derivative written per chunk as matrix products.  In a
// chunk of C tokens with chunk-start state S, gradient dS' of the chunk-end state,
// g the in-chunk cumulative log gate, D_ij = e^{g_i - g_j} (j <= i), E = e^{g_last - g},
// A = strictly-lower(beta_i K K^T o D), T = (I + A)^{-1}, W~ = T diag(beta e^g) K,
// U = T diag(beta) V, delta = U - W~ S^T, P = lower(Q K^T o D):
//
//   d delta = P^T dO + E K dS'^T
//   dS      = dO^T diag(e^g) Q + e^{g_last} dS' - d delta^T W~     (handed to chunk j-1)
//   dP      = lower(dO delta^T)
//   dQ      = e^g o (dO S) + (dP o D) K
//   dW      = -d delta S,  dT = d delta (beta o V)^T + dW (beta e^g o K)^T
//   dA      = strictly-lower(-T^T dT T^T),  X = dA o D o beta_i
//   dK      = (dP o D)^T Q + E o (delta dS') + beta e^g o T^T dW + X K + X^T K
//   dV      = beta o T^T d delta
//   dbeta   = (T^T d delta . v) + e^g (T^T dW . k) + rowsum(dA o KK^T o D)
//   dg      = rowsum(dD o D) - colsum(dD o D) + e^g (beta (T^T dW . k) + dO S . q)
//             - E (delta dS' . k), plus sum(E (delta dS' . k)) + e^{g_last} <dS', S>
//             at the last token;  dD = dA beta_i K K^T + dP o Q K^T
//   d log alpha = the reverse cumulative sum of dg inside the chunk.
//
// Layout of the work.  Every (chunk, head) pair is one batch entry b of padded fp32
// buffers in the workspace (a ragged last chunk is zero-filled with beta = 0 and
// log alpha = 0, which adds nothing to any sum).  The two serial parts, the chunk-start
// states S_j (forward) and the chunk-end state gradients dS'_j (reverse), run in one
// chain kernel with the state of a (sequence, head) in tensor memory.  Everything else is
// chunk-parallel: a persistent batched product kernel (a whole entry's product per work
// item) and small per-chunk kernels for the triangular solve, the gate terms and the final
// per-token sums.
//
// Accuracy is fp32's: the products (batched and in both chains) run on the tcgen05 tensor
// cores in three TF32 passes (hi*hi + hi*lo + lo*hi of a two-part TF32 split of each fp32
// operand, accumulated in fp32: ~2^-22 relative error per product); the rest is fp32 on
// the CUDA cores.  Head sizes dk = dv = 64 or 128.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "gdn_internal.h"
#include "tc_common.cuh"

namespace gdn {
namespace {

constexpr int kCk = 64;             // chunk length
constexpr float kLogAlphaMin = -80.f;  // alpha = 0 (log alpha = -inf) is taken as e^-80

// Per-batch-entry gate vectors, each kCk long.
enum { G_BETA = 0, G_G = 1, G_EG = 2, G_E = 3, G_BEG = 4, kGates = 5 };

// Four consecutive elements (8- or 16-byte aligned) as fp32, and back.
template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                     __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}
template <typename T>
__device__ __forceinline__ void store4(T* p, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 w;
  w.x = *reinterpret_cast<const unsigned*>(&a);
  w.y = *reinterpret_cast<const unsigned*>(&b);
  *reinterpret_cast<uint2*>(p) = w;
}

// ---------------------------------------------------------------------------------
// Chunk table: for every chunk of cl tokens (cl <= kCk; the batch entry of a shorter
// chunk is zero-padded to kCk rows) its first token row and length, for every sequence
// the index of its first chunk, and the count of live batch entries (chunks x H).
// One CTA; sequences in tiles of 1024 with a block scan.  Entries past nc_max (only
// reachable with offsets that overrun the token count) are dropped.
__global__ void __launch_bounds__(1024)
ck_table_kernel(const int32_t* __restrict__ cu, int N, int T, int H, int cl, long long nc_max,
                long long* __restrict__ crow0, int* __restrict__ clen, int* __restrict__ cbase,
                long long* __restrict__ nlive) {
  __shared__ int wsum[32];
  __shared__ long long carry;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int n0 = 0; n0 < N; n0 += 1024) {
    const int n = n0 + threadIdx.x;
    long long start = 0;
    int len = 0;
    if (n < N) {
      if (cu) {
        // offsets clamped to [0, T] (T is the packed token count), as the forward does,
        // so that no chunk of a malformed offset table reaches outside the tensors
        const long long a = min(max((long long)cu[n], 0LL), (long long)T);
        const long long b = min(max((long long)cu[n + 1], a), (long long)T);
        start = a;
        len = (int)(b - a);
      } else {
        start = (long long)n * T;
        len = T;
      }
    }
    const int nc = len > 0 ? (len + cl - 1) / cl : 0;
    int x = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[w] = x;
    __syncthreads();
    if (w == 0) {
      int s = wsum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      wsum[lane] = s;
    }
    __syncthreads();
    const long long incl = carry + x + (w > 0 ? wsum[w - 1] : 0);
    const long long base = incl - nc;
    if (n < N) {
      cbase[n] = (int)(base < nc_max ? base : nc_max);
      for (int j = 0; j < nc && base + j < nc_max; ++j) {
        crow0[base + j] = start + (long long)j * cl;
        clen[base + j] = min(cl, len - j * cl);
      }
    }
    __syncthreads();
    if (threadIdx.x == 1023) carry = incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const long long total = carry < nc_max ? carry : nc_max;
    cbase[N] = (int)total;
    nlive[0] = total * H;
  }
}

// ---------------------------------------------------------------------------------
// Gather one (chunk, head): q, k, v, dO as padded fp32 [kCk][D] tiles, and the gate
// vectors: beta, g (in-chunk inclusive cumulative log alpha), e^g, E = e^{g_last - g},
// beta e^g, and Gamma = e^{g_last}.
struct GatherArgs {
  const void *q, *k, *v, *dout;
  const float *log_alpha, *beta;
  const long long* crow0;
  const int* clen;
  const long long* nlive;
  float *Qc, *Kc, *Vc, *dOc, *gates, *gam;
  int H;
};

template <int D, typename TIn>
__global__ void __launch_bounds__(256) ck_gather_kernel(GatherArgs p) {
  const long long b = blockIdx.x;
  if (b >= *p.nlive) return;
  const long long cid = b / p.H;
  const int h = (int)(b - cid * p.H);
  const long long row0 = p.crow0[cid];
  const int len = p.clen[cid];
  const TIn* q = reinterpret_cast<const TIn*>(p.q);
  const TIn* k = reinterpret_cast<const TIn*>(p.k);
  const TIn* v = reinterpret_cast<const TIn*>(p.v);
  const TIn* dO = reinterpret_cast<const TIn*>(p.dout);
  const size_t ob = (size_t)b * kCk * D;
  for (int i = threadIdx.x; i < kCk * D / 4; i += 256) {
    const int c = i / (D / 4), x = 4 * (i % (D / 4));
    float4 qv = make_float4(0.f, 0.f, 0.f, 0.f), kv = qv, vv = qv, ov = qv;
    if (c < len) {
      const size_t o = ((size_t)(row0 + c) * p.H + h) * D + x;
      qv = load4(q + o);
      kv = load4(k + o);
      vv = load4(v + o);
      if (dO) ov = load4(dO + o);
    }
    const size_t d = ob + (size_t)c * D + x;
    store4(p.Qc + d, qv);
    store4(p.Kc + d, kv);
    store4(p.Vc + d, vv);
    if (dO) store4(p.dOc + d, ov);  // the forward gathers no dO
  }
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x, c0 = 2 * lane, c1 = c0 + 1;
    float la0 = 0.f, la1 = 0.f, b0 = 0.f, b1 = 0.f;
    // a NULL log_alpha is alpha = 1; a NULL beta (the forward's linear mode) an erase
    // strength of 0, so A = 0, T = I and W~ = 0
    if (c0 < len) {
      if (p.log_alpha) la0 = fmaxf(p.log_alpha[(size_t)(row0 + c0) * p.H + h], kLogAlphaMin);
      if (p.beta) b0 = p.beta[(size_t)(row0 + c0) * p.H + h];
    }
    if (c1 < len) {
      if (p.log_alpha) la1 = fmaxf(p.log_alpha[(size_t)(row0 + c1) * p.H + h], kLogAlphaMin);
      if (p.beta) b1 = p.beta[(size_t)(row0 + c1) * p.H + h];
    }
    float s = la0 + la1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    const float g1 = s, g0 = s - la1;
    const float glast = __shfl_sync(0xffffffffu, s, 31);
    float* G = p.gates + (size_t)b * kGates * kCk;
    const float e0 = expf(g0), e1 = expf(g1);
    G[G_BETA * kCk + c0] = b0;
    G[G_BETA * kCk + c1] = b1;
    G[G_G * kCk + c0] = g0;
    G[G_G * kCk + c1] = g1;
    G[G_EG * kCk + c0] = e0;
    G[G_EG * kCk + c1] = e1;
    G[G_E * kCk + c0] = expf(glast - g0);
    G[G_E * kCk + c1] = expf(glast - g1);
    G[G_BEG * kCk + c0] = b0 * e0;
    G[G_BEG * kCk + c1] = b1 * e1;
    if (lane == 0) p.gam[b] = expf(glast);
  }
}

// ---------------------------------------------------------------------------------
// Batched GEMM with fp32 accuracy: for every live batch entry b, the sum of one or two
// products (terms t)
//   C(m, n) = alpha * sum_t sum_k as_t[m] * A_t(m, k) * ks_t[k] * B_t(k, n) * bs_t[n]
// A_t(m, k) = A_t[b*ab + m*am + k*ak] (likewise B_t and C), so either operand may be read
// transposed; one of each operand's two strides is 1, and C's column stride is 1.  ks_t,
// bs_t, as_t: optional per-entry vectors (stride vb).  mask 1 keeps n <= m, mask 2 n < m.  With
// C2, the product is also written there times Dg(m, n) = e^{g_m - g_n} for n <= m (0
// above), g = gv.  M and N are 64 or 128, each term's K 64 or 128: every entry's whole
// product is one tile.
//
// On the tcgen05 tensor cores in three TF32 passes: each fp32 operand is split into two
// TF32 parts and lo*hi + hi*lo + hi*hi is accumulated in fp32 in tensor memory (~2^-22
// relative error per product, the fp32 level).  A persistent CTA walks the live entries
// (b = blockIdx.x, + gridDim.x, ...) with four roles joined by mbarriers:
//   warp 0     TMA: 32-deep k panels of both operands, as stored, into a raw ring of 3 to 8
//              slots (as many as fit: the loads in flight are what the CTA's bandwidth
//              rests on), with the panel's scale vectors by bulk copy; a panel contiguous in
//              k lands in the MMA's K-major
//              128-byte-swizzled layout already, one contiguous in m or n as [32 k][rows];
//   warps 2-9  split: each raw panel into TF32 hi and lo panels, K-major and swizzled,
//              scaled on the way (a ring of 2 slots); the transposing reads of a plain
//              panel go down its columns, one row per lane, free of bank conflicts;
//   warps 1,14 MMA: 12 tcgen05.mma (kind::tf32) per panel, as C^T = B^T A^T (the columns n
//              of C are the TMEM lanes); one warp per accumulator, even and odd entries;
//   warps 10-13 epilogue: tcgen05.ld of the accumulator (a thread per column n, 32 rows m
//              per load), alpha, mask, C2, and the stores (a warp writes 32
//              consecutive n of a row m per instruction).
// Every wait is bounded; one that gives up stops the CTA and records a code in the
// library's status word (read by gdn_check_status).
struct MmTerm {
  const float* A;
  long long ab;
  int am, ak;
  const float* B;
  long long bb;
  int bk, bn;
  const float *ks, *bs, *as;  // scales per k, per column n of B, per row m of A
  int K;
};

struct Mm {
  MmTerm t[2];
  int nt;  // 1 or 2 terms
  float* C;
  long long cb;
  int cm, cn;
  float* C2;
  const float* gv;
  long long vb;
  float alpha;
  int mask, M, N;
  const long long* nlive;
};

struct MmArgs {
  Mm m;
  int akc[2], bkc[2];  // 1: the operand is contiguous in k
  int np0, np;         // k panels of the first term, of both
  int* status;
};

constexpr int kMmSplitThreads = 256;  // 8 split warps
constexpr int kMmThreads = 64 + kMmSplitThreads + 128;
constexpr int kMmRing = 214784;       // both rings: 2 split slots, 2 to 8 raw slots
constexpr int kMmXch = 16384;         // epilogue exchange buffer: 2 x [32][64] fp32
constexpr int kMmMaxRaw = 8, kMmMaxSplit = 2;
constexpr int kMmAux = 640;           // per raw slot: 32 ks + kCk bs + kCk as values
constexpr int kMmSmem = kMmRing + kMmXch + 1024;
constexpr int kMmTmemCols = 512;      // two accumulators of up to 256 columns

// Instruction descriptor, kind::tf32: fp32 accumulator, TF32 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
// One thread: D(tmem) (+)= A(smem) B(smem)^T, kind::tf32.
__device__ __forceinline__ void umma_tf32(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                          uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}

// fp32 -> TF32 hi + lo, each rounded to nearest with ties away from zero (the format's
// conversion) by adding half a TF32 unit to the magnitude bits and clearing the 13 low
// bits; x - hi is exact in fp32.  Integer and one fp32 operation only.
__device__ __forceinline__ void tf32_split_rn(float x, uint32_t& hi, uint32_t& lo) {
  hi = (__float_as_uint(x) + 0x1000u) & 0xffffe000u;
  lo = (__float_as_uint(x - __uint_as_float(hi)) + 0x1000u) & 0xffffe000u;
}

// One raw k panel of an operand (R rows) into TF32 hi and lo panels, K-major with the
// 128-byte swizzle (row r at r * 128 bytes, 16-byte chunk c of it at (c ^ r % 8) * 16).
// KC: the raw panel has that layout already (TMA with the swizzle); else it is [32 k][R]
// plain fp32, read down its columns (one row per lane).  ks, rs: optional scales per k of
// the panel and per row, in shared memory.  Thread ts = 0 .. NT - 1 of NT; each
// takes R * 8 / NT 16-byte chunks (NT threads), loaded together before any is converted.
template <int R, bool KC, int NT = kMmSplitThreads>
__device__ __forceinline__ void mm_split(const uint8_t* raw, uint8_t* hi, uint8_t* lo,
                                         const float* ks, const float* rs, int ts) {
  constexpr int kPer = R * 8 / NT;
  float4 x[kPer];
  int off[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int t = ts + NT * i;
    int c, r;  // logical 16-byte chunk (4 consecutive k) of row r
    if (KC) {
      off[i] = 16 * t;
      r = t >> 3;
      c = (t & 7) ^ (r & 7);
      x[i] = *reinterpret_cast<const float4*>(raw + off[i]);
    } else {
      r = t & (R - 1);
      c = t / R;
      off[i] = r * 128 + ((c ^ (r & 7)) << 4);
      const float* rf = reinterpret_cast<const float*>(raw) + 4 * c * R + r;
      x[i] = make_float4(rf[0], rf[R], rf[2 * R], rf[3 * R]);
    }
    if (ks) {
      const float4 f = *reinterpret_cast<const float4*>(ks + 4 * c);
      x[i].x *= f.x; x[i].y *= f.y; x[i].z *= f.z; x[i].w *= f.w;
    }
    if (rs) {
      const float f = rs[r];
      x[i].x *= f; x[i].y *= f; x[i].z *= f; x[i].w *= f;
    }
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    uint4 h, l;
    tf32_split_rn(x[i].x, h.x, l.x);
    tf32_split_rn(x[i].y, h.y, l.y);
    tf32_split_rn(x[i].z, h.z, l.z);
    tf32_split_rn(x[i].w, h.w, l.w);
    *reinterpret_cast<uint4*>(hi + off[i]) = h;
    *reinterpret_cast<uint4*>(lo + off[i]) = l;
  }
}

__device__ __forceinline__ void mm_split_any(const uint8_t* raw, uint8_t* hi, uint8_t* lo, int R,
                                             bool kc, const float* ks, const float* rs, int ts) {
  if (R == 128) {
    if (kc) mm_split<128, true>(raw, hi, lo, ks, rs, ts);
    else mm_split<128, false>(raw, hi, lo, ks, rs, ts);
  } else {
    if (kc) mm_split<64, true>(raw, hi, lo, ks, rs, ts);
    else mm_split<64, false>(raw, hi, lo, ks, rs, ts);
  }
}

__global__ void __launch_bounds__(kMmThreads, 1)
    ck_mm_kernel(const __grid_constant__ CUtensorMap mapA0, const __grid_constant__ CUtensorMap mapB0,
                 const __grid_constant__ CUtensorMap mapA1, const __grid_constant__ CUtensorMap mapB1,
                 const MmArgs p) {
  extern __shared__ uint8_t mm_smem_raw[];
  uint8_t* sm = mm_smem_raw + ((1024u - (smem_u32(mm_smem_raw) & 1023u)) & 1023u);
  enum { RF = 0, RE = 8, SF = 16, SE = 20, AF = 24, AE = 26, DONE = 28, NBAR = 29 };
  __shared__ __align__(8) uint64_t bars[NBAR];
  __shared__ uint32_t tslot;
  __shared__ int abort_s;
  volatile int* abort_flag = &abort_s;
  const Mm& m = p.m;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int M = m.M, N = m.N, np = p.np, np0 = p.np0;
  const long long nlive = *m.nlive;
  // one raw slot: a k panel of A and B, (M + N) x 128 bytes, with an aux slot for the
  // panel's 32 ks values and the kCk bs values (the scale vectors ride with the panel's
  // copies); one split slot: the hi and lo panels.  Ring depths: two split slots (the split
  // keeps ahead of the MMAs), and as many raw slots as fit, up to 8: the copies in flight
  // carry the CTA's share of the memory bandwidth.
  const int pan_bytes = (M + N) * 128, split_bytes = 2 * pan_bytes;
  const int ns = 2;
  const int ring = kMmRing + (N == 64 ? 0 : kMmXch);  // the exchange buffer only for N = 64
  const int nr = min(kMmMaxRaw, (ring - ns * split_bytes) / (pan_bytes + kMmAux));
  constexpr int kSplitWarps = kMmSplitThreads / 32;
  if (tid == 0) {
    for (int i = 0; i < kMmMaxRaw; ++i) {
      mbar_init(&bars[RF + i], 1);
      mbar_init(&bars[RE + i], kSplitWarps);
    }
    for (int i = 0; i < kMmMaxSplit; ++i) {
      mbar_init(&bars[SF + i], kSplitWarps);
      mbar_init(&bars[SE + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[AF + i], 1);
      mbar_init(&bars[AE + i], 4);
    }
    mbar_init(&bars[DONE], 1);
    abort_s = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) tmem_alloc(&tslot, kMmTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tslot;
  uint8_t* const spl0 = sm;
  uint8_t* const raw0 = sm + ns * split_bytes;
  uint8_t* const aux0 = raw0 + nr * pan_bytes;
  uint8_t* const xch0 = sm + kMmRing;  // the epilogue's exchange buffer (N = 64)

  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      prefetch_tensormap(&mapA0);
      prefetch_tensormap(&mapB0);
      if (m.nt > 1) {
        prefetch_tensormap(&mapA1);
        prefetch_tensormap(&mapB1);
      }
      uint32_t bytes[2];
      for (int t = 0; t < 2; ++t)
        bytes[t] = pan_bytes + (m.t[t].ks ? 128 : 0) + (m.t[t].bs ? 4 * kCk : 0) +
                   (m.t[t].as ? 4 * kCk : 0);
      int q = 0, s = 0, ph = 0;  // panel count, its raw slot and that slot's phase
      for (long long b = blockIdx.x; b < nlive; b += gridDim.x) {
        bool ok = true;
        for (int pn = 0; pn < np; ++pn, ++q) {
          if (!(ok = wait_bar(&bars[RE + s], ph ^ 1, abort_flag, false))) break;
          uint8_t* raw = raw0 + s * pan_bytes;
          uint8_t* aux = aux0 + s * kMmAux;
          const int t = pn >= np0, k0 = 32 * (pn - (t ? np0 : 0));
          mbar_arrive_expect_tx(&bars[RF + s], bytes[t]);
          if (m.t[t].ks) bulk_load(aux, m.t[t].ks + b * m.vb + k0, 128, &bars[RF + s]);
          if (m.t[t].bs) bulk_load(aux + 128, m.t[t].bs + b * m.vb, 4 * kCk, &bars[RF + s]);
          if (m.t[t].as) bulk_load(aux + 384, m.t[t].as + b * m.vb, 4 * kCk, &bars[RF + s]);
          const CUtensorMap* ma = t ? &mapA1 : &mapA0;
          const CUtensorMap* mb = t ? &mapB1 : &mapB0;
          if (p.akc[t]) tma_load_3d(raw, ma, &bars[RF + s], k0, 0, (int)b);
          else tma_load_3d(raw, ma, &bars[RF + s], 0, k0, (int)b);
          if (p.bkc[t]) tma_load_3d(raw + M * 128, mb, &bars[RF + s], k0, 0, (int)b);
          else tma_load_3d(raw + M * 128, mb, &bars[RF + s], 0, k0, (int)b);
          if (++s == nr) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
      }
      // Copies still in flight land before the CTA's shared memory is released: the last
      // min(q, nr) panels, each in its own slot.
      for (int u = 0; u < min(q, nr); ++u) {
        if (--s < 0) { s = nr - 1; ph ^= 1; }
        (void)mbar_wait(&bars[RF + s], ph, kWaitNs);
      }
    }
  } else if (warp == 1) {
    // MMA issuer: C^T = B^T A^T, so that C's columns are TMEM lanes.  The hi and lo panels
    // of an operand lie back to back, so that one descriptor spans both: with N = 64, one
    // MMA per 8-deep k step multiplies [B_hi; B_lo] (128 rows) by [A_hi; A_lo] (2M rows)
    // and the four quadrants of the accumulator sum to C; with N = 128, B_hi times
    // [A_hi; A_lo] and B_lo times A_hi (two MMAs) leave C as the sum of two column halves.
    if (lane == 0) {
      const bool stacked = N == 64;
      const uint32_t id2 = idesc_tf32(128, 2 * M), id1 = idesc_tf32(128, M);
      int i = 0, s = 0, sph = 0;  // item count; split slot and its phase
      for (long long b = blockIdx.x; b < nlive; b += gridDim.x, ++i) {
        const int a = i & 1;
        if (!wait_bar(&bars[AE + a], ((i >> 1) & 1) ^ 1, abort_flag, false)) break;
        tc_fence_after();
        const uint32_t d = tmem + 256u * a;
        bool ok = true;
        for (int pn = 0; pn < np; ++pn) {
          if (!(ok = wait_bar(&bars[SF + s], sph, abort_flag, false))) break;
          tc_fence_after();
          // descriptors once per panel, advanced 32 bytes (2 units) per 8-deep k step
          const uint32_t ahi = smem_u32(spl0 + s * split_bytes);
          const uint32_t bhi = ahi + 2 * M * 128, blo = bhi + N * 128;
          const uint64_t dah = smem_desc(ahi, 16, 1024);
          const uint64_t dbh = smem_desc(bhi, 16, 1024), dbl = smem_desc(blo, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t o = 2u * kk;
            umma_tf32(d, dbh + o, dah + o, id2, (pn | kk) != 0);
            if (!stacked) umma_tf32(d, dbl + o, dah + o, id1, 1u);
          }
          mma_commit(&bars[SE + s]);
          if (++s == ns) { s = 0; sph ^= 1; }
        }
        if (!ok) break;
        mma_commit(&bars[AF + a]);
      }
      // Every MMA issued is complete before tensor memory is freed.
      mma_commit(&bars[DONE]);
      (void)mbar_wait(&bars[DONE], 0, kWaitNs);
    }
  } else if (warp < 2 + kSplitWarps) {  // split
    const int ts = tid - 64;
    int r = 0, rph = 0, s = 0, sph = 0;  // raw and split slots and their phases
    for (long long b = blockIdx.x; b < nlive; b += gridDim.x) {
      bool ok = true;
      for (int pn = 0; pn < np; ++pn) {
        ok = wait_bar(&bars[RF + r], rph, abort_flag, false) &&
             wait_bar(&bars[SE + s], sph ^ 1, abort_flag, false);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        const uint8_t* raw = raw0 + r * pan_bytes;
        const uint8_t* aux = aux0 + r * kMmAux;
        uint8_t* spl = spl0 + s * split_bytes;
        const int t = pn >= np0;
        const float* ks = m.t[t].ks ? reinterpret_cast<const float*>(aux) : nullptr;
        const float* bs = m.t[t].bs ? reinterpret_cast<const float*>(aux + 128) : nullptr;
        const float* as = m.t[t].as ? reinterpret_cast<const float*>(aux + 384) : nullptr;
        mm_split_any(raw, spl, spl + M * 128, M, p.akc[t], nullptr, as, ts);
        mm_split_any(raw + M * 128, spl + 2 * M * 128, spl + 2 * M * 128 + N * 128, N, p.bkc[t],
                     ks, bs, ts);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars[SF + s]);
          mbar_arrive(&bars[RE + r]);
        }
        if (++r == nr) { r = 0; rph ^= 1; }
        if (++s == ns) { s = 0; sph ^= 1; }
      }
      if (!ok) break;
    }
  } else {
    // Epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31, i.e. one column n of C (or, with
    // N = 64, the hi half of column n in lanes 0..63 and its lo half in lanes 64..127;
    // the lo warps hand their sums to the hi warps through shared memory).
    const int qd = warp & 3, tl_row = 32 * qd + lane;
    const bool stacked = N == 64;
    const int n = stacked ? (tl_row & 63) : tl_row;
    const bool top = !stacked || tl_row < 64;
    float* xch = reinterpret_cast<float*>(xch0);
    const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
    int i = 0;
    for (long long b = blockIdx.x; b < nlive; b += gridDim.x, ++i) {
      const int a = i & 1;
      if (group_wait_fails(&bars[AF + a], (i >> 1) & 1, abort_flag, false, 2, 128)) break;
      tc_fence_after();
      const float* gv = m.gv ? m.gv + b * m.vb : nullptr;
      // Dg(m, n) = 2^{(g_m - g_n) log2 e} by ex2.approx (relative error ~2^-22)
      const float gn = gv ? gv[n] * kLog2e : 0.f;
      float* C = m.C + b * m.cb + n;
      float* C2 = m.C2 ? m.C2 + b * m.cb + n : nullptr;
      for (int mb = 0; mb < M / 32; ++mb) {
        uint32_t r[32], r2[32];
        tmem_ld32(tl + 256u * a + 32u * mb, r);
        tmem_ld32(tl + 256u * a + M + 32u * mb, r2);
        const float gml = gv ? gv[32 * mb + lane] * kLog2e : 0.f;
        tmem_wait_ld();
        if (mb == M / 32 - 1) {  // the accumulator is free for the MMA warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[AE + a]);
        }
        float x[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]) + __uint_as_float(r2[j]);
        if (stacked) {  // [32 m][64 n], two halves used in turn
          float* xs = xch + (mb & 1) * 32 * 64;
          if (!top) {
#pragma unroll
            for (int j = 0; j < 32; ++j) xs[j * 64 + n] = x[j];
          }
          named_sync(3, 128);
          if (!top) continue;
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] += xs[j * 64 + n];
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] *= m.alpha;
        if (C2) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int mm = 32 * mb + j;
            const float gm = __shfl_sync(0xffffffffu, gml, j);
            C2[(long long)mm * m.cm] = n <= mm ? x[j] * ex2(gm - gn) : 0.f;
          }
        }
        if (m.mask) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int mm = 32 * mb + j;
            if ((m.mask == 1 && n > mm) || (m.mask == 2 && n >= mm)) x[j] = 0.f;
          }
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) C[(long long)(32 * mb + j) * m.cm] = x[j];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kMmTmemCols);
  }
  if (tid == 0 && *abort_flag) atomicOr(p.status, *abort_flag);
}

// ---------------------------------------------------------------------------------
// Per (chunk, head): A = strictly-lower(beta_i KK^T_ij D_ij), T = (I + A)^{-1}, and
// P = lower(QK^T o D).  T in 16 x 16 blocks: the diagonal blocks by forward substitution
// (one thread per column), then block rows in order from (I + A) T = I:
// T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj.
struct TsolveArgs {
  const float *KK, *QK, *gates;
  float *T, *P;
  const long long* nlive;
};

__global__ void __launch_bounds__(128) ck_tsolve_kernel(TsolveArgs p) {
  const long long b = blockIdx.x;
  if (b >= *p.nlive) return;
  __shared__ float As[kCk][kCk + 1], Ts[kCk][kCk + 1], Wb[3 * 256], g[kCk], be[kCk];
  const int tid = threadIdx.x;
  const float* G = p.gates + (size_t)b * kGates * kCk;
  const size_t ob = (size_t)b * kCk * kCk;
  // both 64 x 64 inputs as 8 float4 per thread, all loads in flight together
  float4 kk[8], qk[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    kk[i] = ld4(p.KK + ob + 4 * tid + 512 * i);
    qk[i] = ld4(p.QK + ob + 4 * tid + 512 * i);
  }
  if (tid < kCk) {
    g[tid] = G[G_G * kCk + tid];
    be[tid] = G[G_BETA * kCk + tid];
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int idx = 4 * tid + 512 * i, r = idx >> 6, j0 = idx & 63;
    const float x[4] = {kk[i].x, kk[i].y, kk[i].z, kk[i].w};
    const float y[4] = {qk[i].x, qk[i].y, qk[i].z, qk[i].w};
    float pd[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = j0 + e;
      const float Dij = j <= r ? expf(g[r] - g[j]) : 0.f;
      As[r][j] = j < r ? be[r] * x[e] * Dij : 0.f;
      pd[e] = y[e] * Dij;
      Ts[r][j] = 0.f;
    }
    st4(p.P + ob + idx, pd[0], pd[1], pd[2], pd[3]);
  }
  __syncthreads();
  // Diagonal 16 x 16 blocks: T_ii = (I + A_ii)^{-1}, one thread per column of a block.
  if (tid < kCk) {
    const int o = tid & ~15, c = tid & 15;
    Ts[o + c][o + c] = 1.f;
    for (int r = c + 1; r < 16; ++r) {
      float s0 = 0.f, s1 = 0.f;
      int j = c;
      for (; j + 1 < r; j += 2) {
        s0 = fmaf(As[o + r][o + j], Ts[o + j][o + c], s0);
        s1 = fmaf(As[o + r][o + j + 1], Ts[o + j + 1][o + c], s1);
      }
      if (j < r) s0 = fmaf(As[o + r][o + j], Ts[o + j][o + c], s0);
      Ts[o + r][o + c] = -(s0 + s1);
    }
  }
  __syncthreads();
  // Block rows below, in order: T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj  (j < i).  Thread
  // tid takes elements e = tid + 128 i of the block row (block j = i / 2, row r, column c);
  // with the block row unrolled every trip count is a constant, so the thread's dot
  // products are independent chains the compiler interleaves.
  const int r0 = tid >> 4, c = tid & 15;
#pragma unroll
  for (int bi = 1; bi < kCk / 16; ++bi) {
    float acc[6];
#pragma unroll
    for (int i = 0; i < 2 * bi; ++i) {
      const int j = i >> 1, r = r0 + 8 * (i & 1);
      float x = 0.f;
#pragma unroll
      for (int k = 16 * j; k < 16 * bi; ++k) x = fmaf(As[16 * bi + r][k], Ts[k][16 * j + c], x);
      acc[i] = x;
    }
#pragma unroll
    for (int i = 0; i < 2 * bi; ++i) Wb[tid + 128 * i] = acc[i];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2 * bi; ++i) {
      const int j = i >> 1, r = r0 + 8 * (i & 1);
      float x = 0.f;
      for (int m = 0; m <= r; ++m)
        x = fmaf(Ts[16 * bi + r][16 * bi + m], Wb[(j << 8) + (m << 4) + c], x);
      acc[i] = x;
    }
#pragma unroll
    for (int i = 0; i < 2 * bi; ++i) {
      const int j = i >> 1, r = r0 + 8 * (i & 1);
      Ts[16 * bi + r][16 * j + c] = -acc[i];
    }
    __syncthreads();
  }
  for (int idx = tid; idx < kCk * kCk; idx += 128) p.T[ob + idx] = Ts[idx >> 6][idx & 63];
}

// ---------------------------------------------------------------------------------
// The state chain of one (sequence, head), chunk by chunk (forward, or in reverse for the
// gradient).  Per chunk, with the state St (D x D):
//   X1(c, r) = Add1(c, r) + s1_c * sum_k A1(c, k) St(r, k)       -> out1
//   St(r, k) = Add2(r, k) + Gamma St(r, k) + sum_c s2_c X1(c, r) A2(c, k)
// forward:  Add1 = U, s1 = -1, A1 = W~, s2 = E, A2 = K, no Add2 (X1 = delta, St = S)
// reverse:  Add1 = P^T dO, s1 = E, A1 = K, s2 = -1, A2 = W~, Add2 = dO^T diag(e^g) Q
//           (X1 = d delta, St = dS')
// St is stored for every chunk before its update; the last update goes to fin.
struct ChainArgs {
  const int* cbase;
  const float* init;  // [N][H][D][D] or null (zeros)
  float* fin;         // [N][H][D][D] or null
  float* st;
  const float *add1, *a1, *a2, *add2;
  float* out1;
  const float *gates, *gam;
  int H;
};

// ---------------------------------------------------------------------------------
// The chain on the tcgen05 tensor cores (dk = dv = 128 or 64): one CTA per (sequence,
// head) holds the whole state St (D x D fp32) in tensor memory, as the accumulator of its
// update, and runs both products of a chunk in three TF32 passes:
//   X1^T(r, c) = sum_k St(r, k) A1(c, k):  A = the hi and lo parts of St, copied to tensor
//                memory; B = [A1_hi; A1_lo] (128 rows) for St_hi and A1_hi for St_lo;
//   St(r, k)  += sum_c (s2 o X1)(c, r) A2(c, k):  A = the hi and lo parts of s2 o X1 in
//                tensor memory; B = A2^T, hi and lo (A2 transposed on chip).
// Roles: warp 0 TMA (A1 as four [64 c][32 k] swizzled panels straight into the lo halves
// of its split panels, split there in place; A2 as two [32 c][128 d] plain panels into a
// raw slot); warps 2-5 split them into TF32 hi and lo K-major panels; warp 1 issues the
// MMAs; warps 6-13 (two per TMEM lane quarter, one state row per thread, each warp one
// half of the columns) run the two passes of a chunk:
//   state pass: St's hi and lo parts -> tensor memory, Gamma St + Add2 -> the accumulator,
//               and St -> st (the chunk-start state) by TMA store from a swizzled 32 x 32
//               tile per warp and column quarter; Add2 comes in by TMA into the same tiles
//               one chunk ahead;
//   X pass:     the product -> X1 = Add1 + s1 o (St A1^T)^T -> out1, and the hi and lo parts
//               of s2 o X1 -> tensor memory.
// Every wait is bounded and reports through the status word.
struct ChainTcArgs {
  ChainArgs c;
  int* status;
};

constexpr int kCtThreads = 448;  // 14 warps
// shared memory: A1 hi/lo 64 KB (4 panels of [hi 8 KB | lo 8 KB]), A2 raw 32 KB, A2 hi/lo
// 64 KB, and two 4 KB tiles ([32 rows][32 fp32], 128-byte swizzle) per pass warp
constexpr int kCtS1 = 0, kCtRaw2 = 65536, kCtS2 = 98304, kCtTile = 163840;
constexpr int kCtSmem = kCtTile + 8 * 2 * 4096 + 1024;
// tensor memory columns: St, St_hi, St_lo, the X1 product (its lo part at +64), whose
// columns then take s2 o X1's hi and lo parts
constexpr uint32_t kTcSt = 0, kTcShi = 128, kTcSlo = 256, kTcX = 384, kTcXhi = 384,
                   kTcXlo = 448;

// One thread: D(tmem) (+)= A(tmem) B(smem)^T, kind::tf32.
__device__ __forceinline__ void umma_tf32_ta(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id,
                                             uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(id), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void split32_to_tmem(uint32_t t_hi, uint32_t t_lo, const float* v) {
  uint32_t h[32], l[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) tf32_split_rn(v[e], h[e], l[e]);
  tmem_st32(t_hi, h);
  tmem_st32(t_lo, l);
}

template <bool REV, int D>
__global__ void __launch_bounds__(kCtThreads, 1)
    ck_chain_tc_kernel(const __grid_constant__ CUtensorMap mapA1,
                       const __grid_constant__ CUtensorMap mapA2,
                       const __grid_constant__ CUtensorMap mapSt,
                       const __grid_constant__ CUtensorMap mapAdd2, const ChainTcArgs args) {
  // D = 128 or 64: the state's rows are TMEM lanes 0 .. D-1 (with D = 64 the upper lanes
  // hold zeros in the A operands, so they add nothing); the A1 panels number D / 32, an A2
  // panel is [32 c][D] (A2P bytes), its transposed hi or lo panel [D rows][32 c] (S2P bytes)
  constexpr int NP1 = D / 32, A2P = 32 * D * 4, S2P = D * 128, NQ = D / 64;
  extern __shared__ uint8_t ct_smem_raw[];
  uint8_t* sm = ct_smem_raw + ((1024u - (smem_u32(ct_smem_raw) & 1023u)) & 1023u);
  enum { R1F, R2F, R2E, S1F, S1E, S2F, S2E, SPD, G1D, XED, G2D, DONE, AD0, NBAR = AD0 + 8 };
  __shared__ __align__(8) uint64_t bars[NBAR];
  __shared__ uint32_t tslot;
  __shared__ int abort_s;
  volatile int* abort_flag = &abort_s;
  const ChainArgs& p = args.c;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int unit = blockIdx.x, n = unit / p.H, h = unit % p.H;
  const int base = p.cbase[n], nc = p.cbase[n + 1] - base;
  const size_t sidx = ((size_t)n * p.H + h) * D * D;
  auto entry = [&](int jj) { return (long long)(base + (REV ? nc - 1 - jj : jj)) * p.H + h; };
  if (tid == 0) {
    mbar_init(&bars[R1F], 1);
    mbar_init(&bars[R2F], 1);
    mbar_init(&bars[R2E], 4);
    mbar_init(&bars[S1F], 4);
    mbar_init(&bars[S1E], 1);
    mbar_init(&bars[S2F], 4);
    mbar_init(&bars[S2E], 1);
    mbar_init(&bars[SPD], 8);
    mbar_init(&bars[G1D], 1);
    mbar_init(&bars[XED], 8);
    mbar_init(&bars[G2D], 1);
    mbar_init(&bars[DONE], 1);
    for (int w = 0; w < 8; ++w) mbar_init(&bars[AD0 + w], 1);
    abort_s = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) tmem_alloc(&tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tslot;

  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      prefetch_tensormap(&mapA1);
      prefetch_tensormap(&mapA2);
      int issued1 = 0, issued2 = 0;
      for (int jj = 0; jj < nc; ++jj) {
        const int b = (int)entry(jj);
        const uint32_t ph = (jj & 1) ^ 1;
        // A1 lands in the lo halves of the split panels, free once the previous X1 product
        // is complete
        if (!wait_bar(&bars[S1E], ph, abort_flag, false)) break;
        // the chunk's Add1 block, read by the X pass with plain loads, into L2
        bulk_prefetch_l2(p.add1 + (size_t)b * kCk * D, kCk * D * 4);
        mbar_arrive_expect_tx(&bars[R1F], NP1 * 8192);
        for (int q = 0; q < NP1; ++q)
          tma_load_3d(sm + kCtS1 + q * 16384 + 8192, &mapA1, &bars[R1F], 32 * q, 0, b);
        issued1 = jj + 1;
        if (!wait_bar(&bars[R2E], ph, abort_flag, false)) break;
        mbar_arrive_expect_tx(&bars[R2F], 2 * A2P);
        for (int q = 0; q < 2; ++q)
          tma_load_3d(sm + kCtRaw2 + q * A2P, &mapA2, &bars[R2F], 0, 32 * q, b);
        issued2 = jj + 1;
      }
      // copies still in flight land before shared memory is released
      if (issued1) (void)mbar_wait(&bars[R1F], (issued1 - 1) & 1, kWaitNs);
      if (issued2) (void)mbar_wait(&bars[R2F], (issued2 - 1) & 1, kWaitNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      const uint32_t id128 = idesc_tf32(128, 128), id64 = idesc_tf32(128, 64);
      const uint32_t idD = idesc_tf32(128, D);
      const uint64_t d1 = smem_desc(smem_u32(sm + kCtS1), 16, 1024);
      const uint64_t d2h = smem_desc(smem_u32(sm + kCtS2), 16, 1024);
      const uint64_t d2l = smem_desc(smem_u32(sm + kCtS2 + 2 * S2P), 16, 1024);
      for (int jj = 0; jj < nc; ++jj) {
        const uint32_t ph = jj & 1;
        if (!wait_bar(&bars[SPD], ph, abort_flag, false) ||
            !wait_bar(&bars[S1F], ph, abort_flag, false))
          break;
        tc_fence_after();
        // X1^T = St_hi [A1_hi; A1_lo]^T + St_lo A1_hi^T: 4 panels of 16 KB (hi | lo)
#pragma unroll
        for (int ks = 0; ks < D / 8; ++ks) {
          const uint64_t o = (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2);  // 16-byte units
          umma_tf32_ta(tmem + kTcX, tmem + kTcShi + 8 * ks, d1 + o, id128, ks != 0);
          umma_tf32_ta(tmem + kTcX, tmem + kTcSlo + 8 * ks, d1 + o, id64, 1u);
        }
        mma_commit(&bars[G1D]);
        mma_commit(&bars[S1E]);
        if (!wait_bar(&bars[XED], ph, abort_flag, false) ||
            !wait_bar(&bars[S2F], ph, abort_flag, false))
          break;
        tc_fence_after();
        // St += Xs_hi A2T_hi^T + Xs_hi A2T_lo^T + Xs_lo A2T_hi^T: 2 panels of 16 KB each
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t o = (uint64_t)((ks >> 2) * (S2P / 16) + (ks & 3) * 2);
          umma_tf32_ta(tmem + kTcSt, tmem + kTcXhi + 8 * ks, d2h + o, idD, 1u);
          umma_tf32_ta(tmem + kTcSt, tmem + kTcXhi + 8 * ks, d2l + o, idD, 1u);
          umma_tf32_ta(tmem + kTcSt, tmem + kTcXlo + 8 * ks, d2h + o, idD, 1u);
        }
        mma_commit(&bars[G2D]);
        mma_commit(&bars[S2E]);
      }
      mma_commit(&bars[DONE]);
      (void)mbar_wait(&bars[DONE], 0, kWaitNs);
    }
  } else if (warp < 6) {  // split: A1 in place (K-major already), A2 transposed
    const int ts = tid - 64;
    for (int jj = 0; jj < nc; ++jj) {
      const uint32_t ph = jj & 1;
      bool ok = wait_bar(&bars[R1F], ph, abort_flag, false);
      if (!__all_sync(0xffffffffu, ok)) break;
#pragma unroll 1
      for (int q = 0; q < NP1; ++q)
        mm_split<64, true, 128>(sm + kCtS1 + q * 16384 + 8192, sm + kCtS1 + q * 16384,
                                sm + kCtS1 + q * 16384 + 8192, nullptr, nullptr, ts);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[S1F]);
      ok = wait_bar(&bars[R2F], ph, abort_flag, false) &&
           wait_bar(&bars[S2E], ph ^ 1, abort_flag, false);
      if (!__all_sync(0xffffffffu, ok)) break;
#pragma unroll 1
      for (int q = 0; q < 2; ++q)
        mm_split<D, false, 128>(sm + kCtRaw2 + q * A2P, sm + kCtS2 + q * S2P,
                                sm + kCtS2 + 2 * S2P + q * S2P, nullptr, nullptr, ts);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[S2F]);
        mbar_arrive(&bars[R2E]);
      }
    }
  } else {  // the state and X passes: row r of the state, column half hf
    const int pw = warp - 6, qd = warp & 3, hf = pw >> 2, r = 32 * qd + lane;
    // a warp's rows are all state rows (r < D) or none (D = 64, lanes 64..127)
    const bool rows = 32 * qd < D;
    const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
    uint8_t* const tiles = sm + kCtTile + pw * 8192;  // two [32][32] fp32 tiles, swizzled
    uint64_t* const abar = &bars[AD0 + pw];
    // Add2 of a chunk into this warp's tiles: rows 32 qd.., columns D/2 hf + 32 hq..
    int add2_loads = 0;  // issued by lane 0
    auto load_add2 = [&](int jj) {
      const int b = (int)entry(jj);
      ++add2_loads;
      mbar_arrive_expect_tx(abar, 4096 * NQ);
      for (int hq = 0; hq < NQ; ++hq)
        tma_load_3d(tiles + hq * 4096, &mapAdd2, abar, (D / 2) * hf + 32 * hq, 32 * qd, b);
    };
    if (REV && rows && lane == 0 && nc > 0) load_add2(0);
    const float* G = p.gates;
    for (int jj = 0; jj < nc; ++jj) {
      const long long b = entry(jj);
      const float* gb = G + (size_t)b * kGates * kCk;
      const float gam = p.gam[b];
      // ---- state pass (the state after chunk jj - 1, or the initial state)
      {
        uint64_t* b1 = REV && rows ? abar : nullptr;
        bool fail;
        if (jj > 0) {
          fail = group_waits_fail(abort_flag, 2, 256, &bars[G2D], (jj - 1) & 1, false, b1, jj & 1);
        } else if (REV) {  // every pass warp takes part in the vote
          const bool ok = !b1 || wait_bar(b1, 0, abort_flag, false);
          fail = named_sync_or(2, 256, !ok || *abort_flag != 0);
        } else {
          fail = false;
        }
        if (fail) break;
        tc_fence_after();
      }
      if (!rows) {  // lanes beyond the state: zero A operands, nothing else
        uint32_t z[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) z[e] = 0u;
#pragma unroll
        for (int hq = 0; hq < NQ; ++hq) {
          tmem_st32(tl + kTcShi + (D / 2) * hf + 32 * hq, z);
          tmem_st32(tl + kTcSlo + (D / 2) * hf + 32 * hq, z);
        }
      }
#pragma unroll 1
      for (int hq = 0; hq < (rows ? NQ : 0); ++hq) {
        const int c0 = (D / 2) * hf + 32 * hq;  // 32 state columns
        uint8_t* const tile = tiles + hq * 4096;
        const uint32_t trow = smem_u32(tile) + lane * 128;  // this thread's row of the tile
        float v[32];
        if (jj > 0) {
          uint32_t u[32];
          tmem_ld32(tl + kTcSt + c0, u);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(u[e]);
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 x = p.init ? ld4(p.init + sidx + (size_t)r * D + c0 + e)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            v[e] = x.x; v[e + 1] = x.y; v[e + 2] = x.z; v[e + 3] = x.w;
          }
        }
        uint32_t w[32];
        if (REV) {  // Add2(r, c0 + 4c ..) from the tile's 16-byte chunk c ^ (r % 8)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            float4 x;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w)
                         : "r"(trow + ((c ^ (lane & 7)) << 4)));
            w[4 * c] = __float_as_uint(fmaf(gam, v[4 * c], x.x));
            w[4 * c + 1] = __float_as_uint(fmaf(gam, v[4 * c + 1], x.y));
            w[4 * c + 2] = __float_as_uint(fmaf(gam, v[4 * c + 2], x.z));
            w[4 * c + 3] = __float_as_uint(fmaf(gam, v[4 * c + 3], x.w));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(gam * v[e]);
        }
        tmem_st32(tl + kTcSt + c0, w);
        split32_to_tmem(tl + kTcShi + c0, tl + kTcSlo + c0, v);
        // the chunk-start state: the tile, then one TMA store per warp and quarter
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_shared_v4(trow + ((c ^ (lane & 7)) << 4), __float_as_uint(v[4 * c]),
                       __float_as_uint(v[4 * c + 1]), __float_as_uint(v[4 * c + 2]),
                       __float_as_uint(v[4 * c + 3]));
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&mapSt, tile, c0, 32 * qd, (int)b);
          bulk_commit();
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[SPD]);
      // the tiles take the next chunk's Add2 once the stores have read them
      if (lane == 0 && rows) {
        bulk_wait_read_all();
        if (REV && jj + 1 < nc) load_add2(jj + 1);
      }
      __syncwarp();
      // ---- X pass; Add1(c, r) for the 32 c of this half is loaded while the product runs
      float add1[32];
      if (rows) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          add1[e] = p.add1[(size_t)b * kCk * D + (size_t)(32 * hf + e) * D + r];
      }
      if (group_wait_fails(&bars[G1D], jj & 1, abort_flag, false, 2, 256)) break;
      tc_fence_after();
      // lanes beyond the state: their product rows are zero, and so stay the hi and lo
      // parts written over them
      if (rows) {
        const int c0 = 32 * hf;  // 32 chunk positions c
        uint32_t u[32], u2[32];
        tmem_ld32(tl + kTcX + c0, u);
        tmem_ld32(tl + kTcX + 64 + c0, u2);
        tmem_wait_ld();
        float xs[32];
        float* o1 = p.out1 + (size_t)b * kCk * D + r;
        const float ecl = gb[G_E * kCk + c0 + lane];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float pr = __uint_as_float(u[e]) + __uint_as_float(u2[e]);
          const float ec = __shfl_sync(0xffffffffu, ecl, e);
          const float x = REV ? fmaf(ec, pr, add1[e]) : add1[e] - pr;
          o1[(size_t)(c0 + e) * D] = x;
          xs[e] = REV ? -x : ec * x;
        }
        split32_to_tmem(tl + kTcXhi + c0, tl + kTcXlo + c0, xs);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[XED]);
    }
    // the final state (the vote keeps the eight warps together after a failed wait)
    if (p.fin) {
      bool ok = true;
      if (nc > 0) {
        ok = !group_wait_fails(&bars[G2D], (nc - 1) & 1, abort_flag, false, 2, 256);
        tc_fence_after();
      }
      if (ok && rows) {
#pragma unroll 1
        for (int hq = 0; hq < NQ; ++hq) {
          const int c0 = (D / 2) * hf + 32 * hq;
          float* f = p.fin + sidx + (size_t)r * D + c0;
          if (nc > 0) {
            uint32_t u[32];
            tmem_ld32(tl + kTcSt + c0, u);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              st4(f + e, __uint_as_float(u[e]), __uint_as_float(u[e + 1]),
                  __uint_as_float(u[e + 2]), __uint_as_float(u[e + 3]));
          } else {
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 x = p.init ? ld4(p.init + sidx + (size_t)r * D + c0 + e)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
              st4(f + e, x.x, x.y, x.z, x.w);
            }
          }
        }
      }
    }
    // the TMA stores are complete before the CTA ends; an Add2 load still in flight (after a
    // failed wait) lands first
    if (lane == 0) {
      bulk_wait_all();
      if (REV && add2_loads > 0) (void)mbar_wait(abar, (add2_loads - 1) & 1, kWaitNs);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (tid == 0 && *abort_flag) atomicOr(args.status, *abort_flag);
}

// ---------------------------------------------------------------------------------
// Per (chunk, head), from dA = strictly-lower(-T^T dT T^T): X + X^T with X = dA o D o beta_i
// (the operand of dK's X K + X^T K), the row sums of dA o KK^T o D (the triangular solve's part of dbeta) and
// dg1 = rowsum(dD o D) - colsum(dD o D) with dD = dA beta_i KK^T + dP o QK^T.
struct DaArgs {
  const float *dA, *KK, *QK, *dPm, *gates;
  float *X, *db3, *dg1;
  const long long* nlive;
};

__global__ void __launch_bounds__(256) ck_da_kernel(DaArgs p) {
  const long long b = blockIdx.x;
  if (b >= *p.nlive) return;
  __shared__ float Ad[kCk][kCk + 1], E2[kCk][kCk + 1], g[kCk], be[kCk];
  const int tid = threadIdx.x;
  const float* G = p.gates + (size_t)b * kGates * kCk;
  const size_t ob = (size_t)b * kCk * kCk;
  // the four 64 x 64 inputs as 4 float4 each per thread, all loads in flight together;
  // a thread's float4 i covers row tid / 16 + 16 i, columns 4 (tid % 16) ..
  float4 da[4], kk[4], dp[4], qk[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const size_t o = ob + 4 * tid + 1024 * i;
    da[i] = ld4(p.dA + o);
    kk[i] = ld4(p.KK + o);
    dp[i] = ld4(p.dPm + o);
    qk[i] = ld4(p.QK + o);
  }
  if (tid < kCk) {
    g[tid] = G[G_G * kCk + tid];
    be[tid] = G[G_BETA * kCk + tid];
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = tid / 16 + 16 * i, j0 = 4 * (tid % 16);
    Ad[r][j0] = da[i].x; Ad[r][j0 + 1] = da[i].y; Ad[r][j0 + 2] = da[i].z; Ad[r][j0 + 3] = da[i].w;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = tid / 16 + 16 * i, j0 = 4 * (tid % 16);
    const float a4[4] = {da[i].x, da[i].y, da[i].z, da[i].w};
    const float k4[4] = {kk[i].x, kk[i].y, kk[i].z, kk[i].w};
    const float d4[4] = {dp[i].x, dp[i].y, dp[i].z, dp[i].w};
    const float q4[4] = {qk[i].x, qk[i].y, qk[i].z, qk[i].w};
    float xs[4], e1 = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = j0 + e;
      const float Dij = j <= r ? expf(g[r] - g[j]) : 0.f;
      // X + X^T: dA is strictly lower, so each element takes the one of X(r, j), X(j, r)
      // that can be nonzero
      const int hi = r > j ? r : j, lo = r > j ? j : r;
      xs[e] = r == j ? 0.f : Ad[hi][lo] * expf(g[hi] - g[lo]) * be[hi];
      e1 += a4[e] * k4[e] * Dij;
      E2[r][j] = (a4[e] * be[r] * k4[e] + d4[e] * q4[e]) * Dij;
    }
    st4(p.X + ob + 4 * tid + 1024 * i, xs[0], xs[1], xs[2], xs[3]);
    // row sum of dA o KK^T o D over the row's 16 threads (a half warp)
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) e1 += __shfl_xor_sync(0xffffffffu, e1, o);
    if ((tid & 15) == 0) p.db3[(size_t)b * kCk + r] = e1;
  }
  __syncthreads();
  if (tid < kCk) {
    float r2 = 0.f, c2 = 0.f;
    for (int j = 0; j < kCk; ++j) {
      r2 += E2[tid][j];
      c2 += E2[j][tid];
    }
    p.dg1[(size_t)b * kCk + tid] = r2 - c2;
  }
}

// <dS', S> per (chunk, head).
__global__ void __launch_bounds__(256)
ck_sdot_kernel(const float* __restrict__ dSn, const float* __restrict__ S, float* __restrict__ sdot,
               int DD, const long long* __restrict__ nlive) {
  const long long b = blockIdx.x;
  if (b >= *nlive) return;
  __shared__ float red[8];
  const float4* x = reinterpret_cast<const float4*>(dSn + (size_t)b * DD);
  const float4* y = reinterpret_cast<const float4*>(S + (size_t)b * DD);
  float s = 0.f;
  for (int i = threadIdx.x; i < DD / 4; i += 256) {
    const float4 a = x[i], c = y[i];
    s += a.x * c.x + a.y * c.y + a.z * c.z + a.w * c.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += red[w];
    sdot[b] = t;
  }
}

// ---------------------------------------------------------------------------------
// Per (chunk, head): the per-token sums and the stores.  dq, dk, dv go to the token rows
// of the chunk; dg is completed at the last token and summed in reverse into d log alpha.
struct ScatterArgs {
  const float *Qc, *Kc, *Vc, *dQa, *dKa, *dOS, *Rd, *TdW, *TdU, *gates, *gam, *db3, *dg1, *sdot;
  const long long* crow0;
  const int* clen;
  const long long* nlive;
  void *dq, *dk, *dv;
  float *dlog_alpha, *dbeta;
  int H;
};

template <int D, typename TIn>
__global__ void __launch_bounds__(256) ck_scatter_kernel(ScatterArgs p) {
  const long long b = blockIdx.x;
  if (b >= *p.nlive) return;
  __shared__ float sdg[kCk], sdE[kCk];
  const long long cid = b / p.H;
  const int h = (int)(b - cid * p.H);
  const long long row0 = p.crow0[cid];
  const int len = p.clen[cid];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const float* G = p.gates + (size_t)b * kGates * kCk;
  TIn* dq = reinterpret_cast<TIn*>(p.dq);
  TIn* dk = reinterpret_cast<TIn*>(p.dk);
  TIn* dv = reinterpret_cast<TIn*>(p.dv);
  for (int c = w; c < kCk; c += 8) {
    const float eg = G[G_EG * kCk + c], E = G[G_E * kCk + c];
    const float be = G[G_BETA * kCk + c], beg = G[G_BEG * kCk + c];
    const size_t o = ((size_t)b * kCk + c) * D + 4 * lane;  // lane: columns 4 lane .. + 3
    const size_t ot = ((size_t)(row0 + c) * p.H + h) * D + 4 * lane;
    float d1 = 0.f, d2 = 0.f, d3 = 0.f, d4 = 0.f;
    if (4 * lane < D) {
      const float4 dos = load4(p.dOS + o), qv = load4(p.Qc + o), kv = load4(p.Kc + o);
      const float4 rd = load4(p.Rd + o), tdw = load4(p.TdW + o), tdu = load4(p.TdU + o);
      const float4 vv = load4(p.Vc + o);
      d1 = tdu.x * vv.x + tdu.y * vv.y + tdu.z * vv.z + tdu.w * vv.w;
      d2 = tdw.x * kv.x + tdw.y * kv.y + tdw.z * kv.z + tdw.w * kv.w;
      d3 = dos.x * qv.x + dos.y * qv.y + dos.z * qv.z + dos.w * qv.w;
      d4 = rd.x * kv.x + rd.y * kv.y + rd.z * kv.z + rd.w * kv.w;
      if (c < len) {
        const float4 qa = load4(p.dQa + o), ka = load4(p.dKa + o);
        store4(dq + ot, make_float4(fmaf(eg, dos.x, qa.x), fmaf(eg, dos.y, qa.y),
                                    fmaf(eg, dos.z, qa.z), fmaf(eg, dos.w, qa.w)));
        store4(dk + ot, make_float4(fmaf(beg, tdw.x, fmaf(E, rd.x, ka.x)),
                                    fmaf(beg, tdw.y, fmaf(E, rd.y, ka.y)),
                                    fmaf(beg, tdw.z, fmaf(E, rd.z, ka.z)),
                                    fmaf(beg, tdw.w, fmaf(E, rd.w, ka.w))));
        store4(dv + ot, make_float4(be * tdu.x, be * tdu.y, be * tdu.z, be * tdu.w));
      }
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) {
      d1 += __shfl_xor_sync(0xffffffffu, d1, s);
      d2 += __shfl_xor_sync(0xffffffffu, d2, s);
      d3 += __shfl_xor_sync(0xffffffffu, d3, s);
      d4 += __shfl_xor_sync(0xffffffffu, d4, s);
    }
    if (lane == 0) {
      if (c < len) p.dbeta[(size_t)(row0 + c) * p.H + h] = d1 + eg * d2 + p.db3[(size_t)b * kCk + c];
      sdg[c] = p.dg1[(size_t)b * kCk + c] + (be * d2 + d3) * eg - d4 * E;
      sdE[c] = d4 * E;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && len > 0) {
    float tot = p.sdot[b] * p.gam[b];
    for (int c = 0; c < len; ++c) tot += sdE[c];
    sdg[len - 1] += tot;
    float run = 0.f;
    for (int c = len - 1; c >= 0; --c) {
      run += sdg[c];
      p.dlog_alpha[(size_t)(row0 + c) * p.H + h] = run;
    }
  }
}

// ---------------------------------------------------------------------------------
// Workspace: chunk tables, gate vectors, and the per-entry fp32 buffers.
enum { QC, KC, WT, DOS, DW, RD, TDW, DQA, DKA, NCD };           // [kCk][D]
enum { VC, DOC, UB, DL, YB, DDL, TDU, NCV };                     // [kCk][D]
enum { KKB, QKB, TB, PB, DPM, DPD, DTB, M1B, DAB, XB, NCC };     // [kCk][kCk]
enum { SB, ZB, DSN, NDD };                                        // [D][D]

struct CkLayout {
  long long nc, nb;
  size_t crow0, clen, cbase, nlive, gates, gam, db3, dg1, sdot;
  size_t cd[NCD], cv[NCV], cc[NCC], dd[NDD], total;
};

size_t al256(size_t x) { return (x + 255) / 256 * 256; }

CkLayout ck_layout(long long rows, int H, int D, int N) {
  CkLayout L;
  L.nc = rows / kCk + N;  // bounds the chunk count of any split of rows tokens into N
  L.nb = L.nc * H;
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o += al256(bytes); return at; };
  L.crow0 = take((size_t)L.nc * 8);
  L.clen = take((size_t)L.nc * 4);
  L.cbase = take((size_t)(N + 1) * 4);
  L.nlive = take(8);
  L.gates = take((size_t)L.nb * kGates * kCk * 4);
  L.gam = take((size_t)L.nb * 4);
  L.db3 = take((size_t)L.nb * kCk * 4);
  L.dg1 = take((size_t)L.nb * kCk * 4);
  L.sdot = take((size_t)L.nb * 4);
  for (int i = 0; i < NCD; ++i) L.cd[i] = take((size_t)L.nb * kCk * D * 4);
  for (int i = 0; i < NCV; ++i) L.cv[i] = take((size_t)L.nb * kCk * D * 4);
  for (int i = 0; i < NCC; ++i) L.cc[i] = take((size_t)L.nb * kCk * kCk * 4);
  for (int i = 0; i < NDD; ++i) L.dd[i] = take((size_t)L.nb * D * D * 4);
  L.total = o;
  return L;
}

// Tensor map of one operand over all entries: a [32 k] x [rows] box per k panel, with the
// 128-byte swizzle when the operand is contiguous in k (the MMA's K-major layout), plain
// when it is contiguous in its rows (then split and transposed on chip).
bool mm_map(CUtensorMap* map, const float* base, long long nb, long long bstride, int rows,
            int K, int row_stride, int k_stride) {
  auto enc = get_encoder();
  if (!enc) return false;
  const bool kc = k_stride == 1;
  cuuint64_t dims[3] = {(cuuint64_t)(kc ? K : rows), (cuuint64_t)(kc ? rows : K), (cuuint64_t)nb};
  cuuint64_t strides[2] = {(cuuint64_t)(kc ? row_stride : k_stride) * 4, (cuuint64_t)bstride * 4};
  cuuint32_t box[3] = {(cuuint32_t)(kc ? 32 : rows), (cuuint32_t)(kc ? rows : 32), 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             kc ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [nb][rows][D] fp32 as boxes of 32 rows x D columns, plain (the chain's A2 panels).
bool tile_map_plain(CUtensorMap* map, const float* base, long long nb, int rows, int D) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)nb};
  cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)rows * D * 4};
  cuuint32_t box[3] = {(cuuint32_t)D, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [nb][D][D] fp32 as 32 x 32 boxes with the 128-byte swizzle (the chain's state tiles).
bool state_tile_map(CUtensorMap* map, const float* base, long long nb, int D) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)D, (cuuint64_t)nb};
  cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)D * D * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct MmLauncher {
  long long nb;
  const long long* nlive;
  cudaStream_t s;
  int* status;
  int grid;
  cudaError_t err = cudaSuccess;
  // C = alpha * op(A) op(B), operands given by (pointer, batch stride, row stride,
  // inner stride); see ck_mm_kernel.
  Mm make(const float* A, long long ab, int am, int ak, const float* B, long long bb, int bk,
          int bn, float* C, long long cb, int cm, int cn, int M, int N, int K) const {
    Mm m;
    m.nt = 1;
    m.t[0] = MmTerm{A, ab, am, ak, B, bb, bk, bn, nullptr, nullptr, nullptr, K};
    m.t[1] = m.t[0];
    m.C = C; m.cb = cb; m.cm = cm; m.cn = cn;
    m.C2 = nullptr;
    m.gv = nullptr;
    m.vb = (long long)kGates * kCk;
    m.alpha = 1.f; m.mask = 0;
    m.M = M; m.N = N;
    m.nlive = nlive;
    return m;
  }
  // A second term, + op(A) op(B) (same M and N), summed on the tensor cores.
  static void add(Mm& m, const float* A, long long ab, int am, int ak, const float* B, long long bb,
                  int bk, int bn, int K) {
    m.t[1] = MmTerm{A, ab, am, ak, B, bb, bk, bn, nullptr, nullptr, nullptr, K};
    m.nt = 2;
  }
  void run(const Mm& m) {
    if (err != cudaSuccess) return;
    auto dim_ok = [](int x) { return x == 64 || x == 128; };
    bool ok = dim_ok(m.M) && dim_ok(m.N) && m.cn == 1 && (m.nt == 1 || m.nt == 2) && nb > 0 &&
              nb <= 0x7fffffffLL;
    for (int t = 0; ok && t < m.nt; ++t) {
      const MmTerm& x = m.t[t];
      // the scale vectors are kCk long: ks needs K <= kCk, bs N <= kCk, as M <= kCk
      ok = dim_ok(x.K) && (x.am == 1 || x.ak == 1) && (x.bk == 1 || x.bn == 1) &&
           (!x.ks || x.K <= kCk) && (!x.bs || m.N <= kCk) && (!x.as || m.M <= kCk);
    }
    if (!ok) {
      err = cudaErrorInvalidValue;
      return;
    }
    MmArgs a;
    a.m = m;
    CUtensorMap map[2][2];
    for (int t = 0; t < 2; ++t) {
      const MmTerm& x = m.t[t < m.nt ? t : 0];
      a.akc[t] = x.ak == 1;
      a.bkc[t] = x.bk == 1;
      if (!mm_map(&map[t][0], x.A, nb, x.ab, m.M, x.K, x.am, x.ak) ||
          !mm_map(&map[t][1], x.B, nb, x.bb, m.N, x.K, x.bn, x.bk)) {
        err = cudaErrorInvalidValue;
        return;
      }
    }
    a.np0 = m.t[0].K / 32;
    a.np = a.np0 + (m.nt > 1 ? m.t[1].K / 32 : 0);
    a.status = status;
    ck_mm_kernel<<<(unsigned)grid, kMmThreads, kMmSmem, s>>>(map[0][0], map[0][1], map[1][0],
                                                             map[1][1], a);
    err = cudaGetLastError();
  }
};

// A second stream per device for the products that do not depend on a chain, with the
// events of the fork and the joins.  Created on first use; the launch sequence that uses
// them runs under g_side_mu.
struct SideStream {
  cudaStream_t st = nullptr;
  cudaEvent_t fork = nullptr, yz = nullptr, fwd = nullptr, side = nullptr;
};
constexpr int kMaxDevices = 64;
std::mutex g_side_mu;
SideStream g_side[kMaxDevices];

cudaError_t side_stream(SideStream*& out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  SideStream& x = g_side[dev];
  if (!x.st) {
    if ((e = cudaStreamCreateWithFlags(&x.st, cudaStreamNonBlocking)) != cudaSuccess) return e;
    for (cudaEvent_t* ev : {&x.fork, &x.yz, &x.fwd, &x.side})
      if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
  }
  out = &x;
  return cudaSuccess;
}

// Orders the caller's stream after everything queued on the side stream when a launch
// sequence leaves early (an error after the fork); the normal path joins explicitly and
// sets `done`.
struct SideJoin {
  SideStream* side;
  cudaStream_t s2, s;
  bool done = false;
  ~SideJoin() {
    if (done) return;
    if (cudaEventRecord(side->side, s2) == cudaSuccess) (void)cudaStreamWaitEvent(s, side->side, 0);
  }
};

// One chain on the tcgen05 kernel: one CTA per (sequence, head).
template <int D, bool REV>
cudaError_t launch_chain(const ChainArgs& c, long long nb, int N, int H, int* status,
                         cudaStream_t s) {
  const unsigned units = (unsigned)((long long)N * H);
  CUtensorMap m1, m2, mst, madd2;
  if (!mm_map(&m1, c.a1, nb, (long long)kCk * D, kCk, D, D, 1) ||
      !tile_map_plain(&m2, c.a2, nb, kCk, D) || !state_tile_map(&mst, c.st, nb, D))
    return cudaErrorInvalidValue;
  // Add2 is read only by the reverse chain; the forward one gets a copy of the st map
  madd2 = mst;
  if (REV && !state_tile_map(&madd2, c.add2, nb, D)) return cudaErrorInvalidValue;
  ChainTcArgs t{c, status};
  ck_chain_tc_kernel<REV, D><<<units, kCtThreads, kCtSmem, s>>>(m1, m2, mst, madd2, t);
  return cudaGetLastError();
}

template <int D, typename TIn>
cudaError_t launch_ck_t(const BwdArgs& a, cudaStream_t s) {
  const long long rows = (long long)a.B * a.T;
  const CkLayout L = ck_layout(rows, a.H, D, a.N);
  unsigned char* ws = reinterpret_cast<unsigned char*>(a.workspace);
  auto F = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
  long long* crow0 = reinterpret_cast<long long*>(ws + L.crow0);
  int* clen = reinterpret_cast<int*>(ws + L.clen);
  int* cbase = reinterpret_cast<int*>(ws + L.cbase);
  long long* nlive = reinterpret_cast<long long*>(ws + L.nlive);
  float* gates = F(L.gates);
  float* gam = F(L.gam);
  float *Qc = F(L.cd[QC]), *Kc = F(L.cd[KC]), *Wt = F(L.cd[WT]), *dOS = F(L.cd[DOS]);
  float *dW = F(L.cd[DW]), *Rd = F(L.cd[RD]), *TdW = F(L.cd[TDW]), *dQa = F(L.cd[DQA]);
  float* dKa = F(L.cd[DKA]);
  float *Vc = F(L.cv[VC]), *dOc = F(L.cv[DOC]), *U = F(L.cv[UB]), *Dl = F(L.cv[DL]);
  float *Y = F(L.cv[YB]), *dDl = F(L.cv[DDL]), *TdU = F(L.cv[TDU]);
  float *KK = F(L.cc[KKB]), *QK = F(L.cc[QKB]), *Tm = F(L.cc[TB]), *P = F(L.cc[PB]);
  float *dPm = F(L.cc[DPM]), *dPD = F(L.cc[DPD]), *dT = F(L.cc[DTB]), *M1 = F(L.cc[M1B]);
  float *dA = F(L.cc[DAB]), *X = F(L.cc[XB]);
  float *S = F(L.dd[SB]), *Z = F(L.dd[ZB]), *dSn = F(L.dd[DSN]);

  ck_table_kernel<<<1, 1024, 0, s>>>(a.cu_seqlens, a.N, a.T, a.H, kCk, L.nc, crow0, clen, cbase,
                                     nlive);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned nb = (unsigned)L.nb;

  GatherArgs ga;
  ga.q = a.q; ga.k = a.k; ga.v = a.v; ga.dout = a.dout;
  ga.log_alpha = a.log_alpha; ga.beta = a.beta;
  ga.crow0 = crow0; ga.clen = clen; ga.nlive = nlive;
  ga.Qc = Qc; ga.Kc = Kc; ga.Vc = Vc; ga.dOc = dOc; ga.gates = gates; ga.gam = gam; ga.H = a.H;
  ck_gather_kernel<D, TIn><<<nb, 256, 0, s>>>(ga);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  // The product kernel: persistent, one CTA per SM at most; its shared-memory cap is
  // raised here, before any side-stream work exists.
  static std::atomic<unsigned long long> set_mm{0};
  if ((e = ensure_smem_cap(ck_mm_kernel, kMmSmem, set_mm)) != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  int* status = nullptr;
  if ((e = tc_status_address(&status)) != cudaSuccess) return e;
  const int mm_grid = (int)std::min<long long>(L.nb, std::max(sms, 1));
  // The side stream's products run beside a chain, which holds one SM per (sequence,
  // head) for its whole length: they take the SMs it leaves (a CTA of either kernel fills
  // an SM's shared memory), so that none of their CTAs waits for the chain to end.
  const long long units = (long long)a.N * a.H;
  const int side_grid =
      units < sms ? (int)std::min<long long>(L.nb, std::max<long long>(sms - units, 1)) : mm_grid;
  const long long CD = (long long)kCk * D, CC = (long long)kCk * kCk, DD = (long long)D * D;
  MmLauncher mm{L.nb, nlive, s, status, mm_grid};
  // KK^T = K K^T, QK^T = Q K^T
  mm.run(mm.make(Kc, CD, D, 1, Kc, CD, 1, D, KK, CC, kCk, 1, kCk, kCk, D));
  mm.run(mm.make(Qc, CD, D, 1, Kc, CD, 1, D, QK, CC, kCk, 1, kCk, kCk, D));
  if (mm.err != cudaSuccess) return mm.err;
  TsolveArgs ta{KK, QK, gates, Tm, P, nlive};
  ck_tsolve_kernel<<<nb, 128, 0, s>>>(ta);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // The chain kernels' shared-memory caps are raised before the fork, so that this
  // per-device first-call step cannot fail while side-stream work is in flight.
  static std::atomic<unsigned long long> set_f{0}, set_r{0};
  if ((e = ensure_smem_cap(ck_chain_tc_kernel<false, D>, kCtSmem, set_f)) != cudaSuccess) return e;
  if ((e = ensure_smem_cap(ck_chain_tc_kernel<true, D>, kCtSmem, set_r)) != cudaSuccess) return e;
  {  // W~ = T diag(beta e^g) K,  U = T diag(beta) V
    Mm m = mm.make(Tm, CC, kCk, 1, Kc, CD, D, 1, Wt, CD, D, 1, kCk, D, kCk);
    m.t[0].ks = gates + G_BEG * kCk;
    mm.run(m);
    m = mm.make(Tm, CC, kCk, 1, Vc, CD, D, 1, U, CD, D, 1, kCk, D, kCk);
    m.t[0].ks = gates + G_BETA * kCk;
    mm.run(m);
  }
  if (mm.err != cudaSuccess) return mm.err;
  // Fork: the side stream takes P^T dO and dO^T diag(e^g) Q (they need the solve's P and
  // the gathered tiles only) on the SMs the forward chain leaves, while this stream runs
  // the chain.
  std::lock_guard<std::mutex> lock(g_side_mu);
  SideStream* side = nullptr;
  if ((e = side_stream(side)) != cudaSuccess) return e;
  cudaStream_t s2 = side->st;
  if ((e = cudaEventRecord(side->fork, s)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(s2, side->fork, 0)) != cudaSuccess) return e;
  // Every exit from here on, the error returns included, leaves the caller's stream
  // ordered after all side-stream work: the caller may free the workspace as soon as
  // its own stream has passed this call.
  SideJoin join{side, s2, s};
  MmLauncher mm2{L.nb, nlive, s2, status, side_grid};
  {  // Y = P^T dO,  Z = dO^T diag(e^g) Q
    mm2.run(mm2.make(P, CC, 1, kCk, dOc, CD, D, 1, Y, CD, D, 1, kCk, D, kCk));
    Mm m = mm2.make(dOc, CD, 1, D, Qc, CD, D, 1, Z, DD, D, 1, D, D, kCk);
    m.t[0].ks = gates + G_EG * kCk;
    mm2.run(m);
  }
  if (mm2.err != cudaSuccess) return mm2.err;
  if ((e = cudaEventRecord(side->yz, s2)) != cudaSuccess) return e;

  ChainArgs cf;
  cf.cbase = cbase; cf.init = a.S0; cf.fin = nullptr; cf.st = S;
  cf.add1 = U; cf.a1 = Wt; cf.a2 = Kc; cf.add2 = nullptr; cf.out1 = Dl;
  cf.gates = gates; cf.gam = gam; cf.H = a.H;
  if ((e = launch_chain<D, false>(cf, L.nb, a.N, a.H, status, s)) != cudaSuccess) return e;

  // The side stream continues with the products of delta and S (dO delta^T, (dP o D) K,
  // dO S) while this stream runs the reverse chain.
  if ((e = cudaEventRecord(side->fwd, s)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(s2, side->fwd, 0)) != cudaSuccess) return e;
  {
    // dP = lower(dO delta^T), and dP o D
    Mm m = mm2.make(dOc, CD, D, 1, Dl, CD, 1, D, dPm, CC, kCk, 1, kCk, kCk, D);
    m.mask = 1;
    m.C2 = dPD;
    m.gv = gates + G_G * kCk;
    mm2.run(m);
    // (dP o D) K, dO S
    mm2.run(mm2.make(dPD, CC, kCk, 1, Kc, CD, D, 1, dQa, CD, D, 1, kCk, D, kCk));
    mm2.run(mm2.make(dOc, CD, D, 1, S, DD, D, 1, dOS, CD, D, 1, kCk, D, D));
  }
  if (mm2.err != cudaSuccess) return mm2.err;
  if ((e = cudaEventRecord(side->side, s2)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(s, side->yz, 0)) != cudaSuccess) return e;
  ChainArgs cr;
  cr.cbase = cbase; cr.init = a.dS_final; cr.fin = a.dS0; cr.st = dSn;
  cr.add1 = Y; cr.a1 = Kc; cr.a2 = Wt; cr.add2 = Z; cr.out1 = dDl;
  cr.gates = gates; cr.gam = gam; cr.H = a.H;
  if ((e = launch_chain<D, true>(cr, L.nb, a.N, a.H, status, s)) != cudaSuccess) return e;

  {
    // dW = -d delta S, delta dS'
    Mm m = mm.make(dDl, CD, D, 1, S, DD, D, 1, dW, CD, D, 1, kCk, D, D);
    m.alpha = -1.f;
    mm.run(m);
    mm.run(mm.make(Dl, CD, D, 1, dSn, DD, D, 1, Rd, CD, D, 1, kCk, D, D));
    // T^T d delta, T^T dW
    mm.run(mm.make(Tm, CC, 1, kCk, dDl, CD, D, 1, TdU, CD, D, 1, kCk, D, kCk));
    mm.run(mm.make(Tm, CC, 1, kCk, dW, CD, D, 1, TdW, CD, D, 1, kCk, D, kCk));
    // dT = d delta (beta o V)^T + dW (beta e^g o K)^T
    m = mm.make(dDl, CD, D, 1, Vc, CD, 1, D, dT, CC, kCk, 1, kCk, kCk, D);
    m.t[0].bs = gates + G_BETA * kCk;
    MmLauncher::add(m, dW, CD, D, 1, Kc, CD, 1, D, D);
    m.t[1].bs = gates + G_BEG * kCk;
    mm.run(m);
    // dA = strictly-lower(-T^T dT T^T)
    m = mm.make(Tm, CC, 1, kCk, dT, CC, kCk, 1, M1, CC, kCk, 1, kCk, kCk, kCk);
    m.alpha = -1.f;
    mm.run(m);
    m = mm.make(M1, CC, kCk, 1, Tm, CC, 1, kCk, dA, CC, kCk, 1, kCk, kCk, kCk);
    m.mask = 2;
    mm.run(m);
  }
  if (mm.err != cudaSuccess) return mm.err;
  float* db3 = F(L.db3);
  float* dg1 = F(L.dg1);
  float* sdot = F(L.sdot);
  // Join: the dA terms need dP, and dK needs dP o D.
  if ((e = cudaStreamWaitEvent(s, side->side, 0)) != cudaSuccess) return e;
  join.done = true;
  DaArgs da{dA, KK, QK, dPm, gates, X, db3, dg1, nlive};
  ck_da_kernel<<<nb, 256, 0, s>>>(da);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  {  // dK's products: (dP o D)^T Q + X K + X^T K, with X + X^T made by the dA kernel
    Mm m = mm.make(dPD, CC, 1, kCk, Qc, CD, D, 1, dKa, CD, D, 1, kCk, D, kCk);
    MmLauncher::add(m, X, CC, kCk, 1, Kc, CD, D, 1, kCk);
    mm.run(m);
  }
  if (mm.err != cudaSuccess) return mm.err;
  ck_sdot_kernel<<<nb, 256, 0, s>>>(dSn, S, sdot, (int)DD, nlive);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ScatterArgs sa;
  sa.Qc = Qc; sa.Kc = Kc; sa.Vc = Vc; sa.dQa = dQa; sa.dKa = dKa; sa.dOS = dOS; sa.Rd = Rd;
  sa.TdW = TdW; sa.TdU = TdU; sa.gates = gates; sa.gam = gam; sa.db3 = db3; sa.dg1 = dg1;
  sa.sdot = sdot; sa.crow0 = crow0; sa.clen = clen; sa.nlive = nlive;
  sa.dq = a.dq; sa.dk = a.dk_out; sa.dv = a.dv_out; sa.dlog_alpha = a.dlog_alpha;
  sa.dbeta = a.dbeta; sa.H = a.H;
  ck_scatter_kernel<D, TIn><<<nb, 256, 0, s>>>(sa);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// The chunk-form forward on the same kernels, for q/k/v in fp32 (or bf16 off the bf16
// headline kernel's shape), dk = dv = 64 or 128, chunks of C = 16, 32 or 64 tokens (a
// shorter chunk's entry is zero-padded to 64 rows, where beta = 0 and log alpha = 0 make
// the padding add nothing) (Nyysyyan, "Chunk Computation"; myhz0606 section 4.5): per
// (chunk, head) entry, A = strictly-lower(beta_i K K^T o D), T = (I + A)^{-1}, W~ =
// T diag(beta e^g) K, U = T diag(beta) V, P = lower(Q K^T o D); the forward chain gives the
// chunk-start states S_j, delta = U - W~ S_j^T and the final state; then
//   O = diag(e^g) Q S_j^T + P delta
// is one two-term product, and a last kernel writes O's real rows to out.  All products
// and the chain run in three TF32 passes (fp32 accuracy).
enum { FQ, FK, FV, FW, FU, FDL, FO, NFCD };  // [kCk][D]
enum { FKK, FQK, FT, FP, NFCC };             // [kCk][kCk]

struct FwdLayout {
  long long nc, nb;
  size_t crow0, clen, cbase, nlive, gates, gam, s, cd[NFCD], cc[NFCC], total;
};

FwdLayout fwd_layout(long long rows, int H, int D, int N, int C) {
  FwdLayout L;
  L.nc = rows / C + N;  // bounds the chunk count of any split of rows tokens into N
  L.nb = L.nc * H;
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o += al256(bytes); return at; };
  L.crow0 = take((size_t)L.nc * 8);
  L.clen = take((size_t)L.nc * 4);
  L.cbase = take((size_t)(N + 1) * 4);
  L.nlive = take(8);
  L.gates = take((size_t)L.nb * kGates * kCk * 4);
  L.gam = take((size_t)L.nb * 4);
  L.s = take((size_t)L.nb * D * D * 4);
  for (int i = 0; i < NFCD; ++i) L.cd[i] = take((size_t)L.nb * kCk * D * 4);
  for (int i = 0; i < NFCC; ++i) L.cc[i] = take((size_t)L.nb * kCk * kCk * 4);
  L.total = o;
  return L;
}

// O's real rows of every entry to out [rows][H][D] (the input dtype).
template <int D, typename TOut>
__global__ void __launch_bounds__(256)
ck_out_kernel(const float* __restrict__ O, const long long* __restrict__ crow0,
              const int* __restrict__ clen, const long long* __restrict__ nlive, void* out, int H) {
  const long long b = blockIdx.x;
  if (b >= *nlive) return;
  const long long cid = b / H;
  const int h = (int)(b - cid * H);
  const long long row0 = crow0[cid];
  const int len = clen[cid];
  TOut* o = reinterpret_cast<TOut*>(out);
  for (int i = threadIdx.x; i < len * (D / 4); i += 256) {
    const int c = i / (D / 4), x = 4 * (i % (D / 4));
    store4(o + ((size_t)(row0 + c) * H + h) * D + x, load4(O + ((size_t)b * kCk + c) * D + x));
  }
}

// The forward's scratch comes from a stream-ordered pool of the library's own per device
// (memory kept for reuse, so that repeated calls do not return to the driver).
std::mutex g_pool_mu;
cudaMemPool_t g_pool[kMaxDevices] = {};

cudaError_t pool_alloc(void** ptr, size_t bytes, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaMemPool_t pool;
  {
    std::lock_guard<std::mutex> lock(g_pool_mu);
    if (!g_pool[dev]) {
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      if ((e = cudaMemPoolCreate(&g_pool[dev], &props)) != cudaSuccess) return e;
      uint64_t keep = ~0ull;
      if ((e = cudaMemPoolSetAttribute(g_pool[dev], cudaMemPoolAttrReleaseThreshold, &keep)) !=
          cudaSuccess)
        return e;
    }
    pool = g_pool[dev];
  }
  return cudaMallocFromPoolAsync(ptr, bytes, pool, s);
}

template <int D, typename TIn>
cudaError_t launch_fwd_ck_t(const FwdArgs& a, cudaStream_t s) {
  const long long rows = (long long)a.B * a.T;
  // the linear mode (beta NULL): erase 0 (the gather's gates), write 1 (delta = V)
  const bool linear = a.beta == nullptr;
  const FwdLayout L = fwd_layout(rows, a.H, D, a.N, a.C);
  cudaError_t e;
  static std::atomic<unsigned long long> set_mm{0}, set_c{0};
  if ((e = ensure_smem_cap(ck_mm_kernel, kMmSmem, set_mm)) != cudaSuccess) return e;
  if ((e = ensure_smem_cap(ck_chain_tc_kernel<false, D>, kCtSmem, set_c)) != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  int* status = nullptr;
  if ((e = tc_status_address(&status)) != cudaSuccess) return e;
  void* wsv = nullptr;
  if ((e = pool_alloc(&wsv, L.total, s)) != cudaSuccess) return e;
  unsigned char* ws = reinterpret_cast<unsigned char*>(wsv);
  auto F = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
  long long* crow0 = reinterpret_cast<long long*>(ws + L.crow0);
  int* clen = reinterpret_cast<int*>(ws + L.clen);
  int* cbase = reinterpret_cast<int*>(ws + L.cbase);
  long long* nlive = reinterpret_cast<long long*>(ws + L.nlive);
  float *gates = F(L.gates), *gam = F(L.gam), *S = F(L.s);
  float *Qc = F(L.cd[FQ]), *Kc = F(L.cd[FK]), *Vc = F(L.cd[FV]), *Wt = F(L.cd[FW]);
  float *U = F(L.cd[FU]), *Dl = F(L.cd[FDL]), *O = F(L.cd[FO]);
  float *KK = F(L.cc[FKK]), *QK = F(L.cc[FQK]), *Tm = F(L.cc[FT]), *P = F(L.cc[FP]);
  const unsigned nb = (unsigned)L.nb;
  const long long CD = (long long)kCk * D, CC = (long long)kCk * kCk, DD = (long long)D * D;
  auto run = [&]() -> cudaError_t {
    cudaError_t e2;
    ck_table_kernel<<<1, 1024, 0, s>>>(a.cu_seqlens, a.N, a.T, a.H, a.C, L.nc, crow0, clen,
                                       cbase, nlive);
    if ((e2 = cudaGetLastError()) != cudaSuccess) return e2;
    GatherArgs ga;
    ga.q = a.q; ga.k = a.k; ga.v = a.v; ga.dout = nullptr;
    ga.log_alpha = a.log_alpha; ga.beta = a.beta;
    ga.crow0 = crow0; ga.clen = clen; ga.nlive = nlive;
    ga.Qc = Qc; ga.Kc = Kc; ga.Vc = Vc; ga.dOc = nullptr; ga.gates = gates; ga.gam = gam;
    ga.H = a.H;
    ck_gather_kernel<D, TIn><<<nb, 256, 0, s>>>(ga);
    if ((e2 = cudaGetLastError()) != cudaSuccess) return e2;
    MmLauncher mm{L.nb, nlive, s, status, (int)std::min<long long>(L.nb, std::max(sms, 1))};
    mm.run(mm.make(Kc, CD, D, 1, Kc, CD, 1, D, KK, CC, kCk, 1, kCk, kCk, D));
    mm.run(mm.make(Qc, CD, D, 1, Kc, CD, 1, D, QK, CC, kCk, 1, kCk, kCk, D));
    if (mm.err != cudaSuccess) return mm.err;
    TsolveArgs ta{KK, QK, gates, Tm, P, nlive};
    ck_tsolve_kernel<<<nb, 128, 0, s>>>(ta);
    if ((e2 = cudaGetLastError()) != cudaSuccess) return e2;
    {  // W~ = T diag(beta e^g) K,  U = T diag(beta) V
      Mm m = mm.make(Tm, CC, kCk, 1, Kc, CD, D, 1, Wt, CD, D, 1, kCk, D, kCk);
      m.t[0].ks = gates + G_BEG * kCk;
      mm.run(m);
      if (!linear) {  // the linear mode writes with strength 1: U = V
        m = mm.make(Tm, CC, kCk, 1, Vc, CD, D, 1, U, CD, D, 1, kCk, D, kCk);
        m.t[0].ks = gates + G_BETA * kCk;
        mm.run(m);
      }
    }
    if (mm.err != cudaSuccess) return mm.err;
    ChainArgs cf;
    cf.cbase = cbase; cf.init = a.S0; cf.fin = a.S_final; cf.st = S;
    cf.add1 = linear ? Vc : U; cf.a1 = Wt; cf.a2 = Kc; cf.add2 = nullptr; cf.out1 = Dl;
    cf.gates = gates; cf.gam = gam; cf.H = a.H;
    if ((e2 = launch_chain<D, false>(cf, L.nb, a.N, a.H, status, s)) != cudaSuccess) return e2;
    {  // O = diag(e^g) Q S_j^T + P delta
      Mm m = mm.make(Qc, CD, D, 1, S, DD, 1, D, O, CD, D, 1, kCk, D, D);
      m.t[0].as = gates + G_EG * kCk;
      MmLauncher::add(m, P, CC, kCk, 1, Dl, CD, D, 1, kCk);
      mm.run(m);
    }
    if (mm.err != cudaSuccess) return mm.err;
    ck_out_kernel<D, TIn><<<nb, 256, 0, s>>>(O, crow0, clen, nlive, a.out, a.H);
    return cudaGetLastError();
  };
  e = run();
  // the scratch returns to the pool behind the launches (also after a failed launch)
  const cudaError_t ef = cudaFreeAsync(wsv, s);
  return e != cudaSuccess ? e : ef;
}

}  // namespace

bool bwd_chunked_supported(int dk, int dv) { return dk == dv && (dk == 64 || dk == 128); }

size_t bwd_chunked_workspace_bytes(long long rows, int H, int dk, int dv, int N) {
  if (rows == 0 || !bwd_chunked_supported(dk, dv)) return 0;
  return ck_layout(rows, H, dk, N).total;
}

cudaError_t launch_bwd_chunked(const BwdArgs& a, cudaStream_t stream) {
  if (!bwd_chunked_supported(a.dk, a.dv)) return cudaErrorInvalidValue;
  if ((long long)a.N * a.H > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (a.dk == 64) return a.bf16 ? launch_ck_t<64, __nv_bfloat16>(a, stream) : launch_ck_t<64, float>(a, stream);
  return a.bf16 ? launch_ck_t<128, __nv_bfloat16>(a, stream) : launch_ck_t<128, float>(a, stream);
}

cudaError_t scratch_alloc(void** ptr, size_t bytes, cudaStream_t stream) {
  return pool_alloc(ptr, bytes, stream);
}

bool fwd_chunked_supported(int dk, int dv, int C) {
  return dk == dv && (dk == 64 || dk == 128) && (C == 16 || C == 32 || C == kCk);
}

int fwd_chunked_launches() { return 10; }

cudaError_t launch_fwd_chunked(const FwdArgs& a, cudaStream_t stream) {
  if (!fwd_chunked_supported(a.dk, a.dv, a.C)) return cudaErrorInvalidValue;
  if ((long long)a.N * a.H > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (a.dk == 64) return a.bf16 ? launch_fwd_ck_t<64, __nv_bfloat16>(a, stream) : launch_fwd_ck_t<64, float>(a, stream);
  return a.bf16 ? launch_fwd_ck_t<128, __nv_bfloat16>(a, stream) : launch_fwd_ck_t<128, float>(a, stream);
}

}  // namespace gdn
