// Backward of the Gated DeltaNet recurrence: gradients of q, k, v, log alpha, beta
// and S0 for given gradients of the outputs and of the final state.
//
// The pages derive no backward pass; this is the reverse-mode derivative of the
// recurrence (Nyysyyan, "Gated-DeltaNet", first equation block) in its
// gate -> predict -> write order:
//
//   a = e^{log alpha},  p = S_{t-1} k,  u = beta (v - a p),  S_t = a S_{t-1} + u k^T,
//   o_t = S_t q_t
//
// walked backwards with G = dL/dS_t:
//
//   G += dO q^T;  dq = S_t^T dO = a S_{t-1}^T dO + k (u . dO);  du = G k;
//   dv = beta du;  dbeta = du . (v - a p);  da = <G, S_{t-1}> - beta du . p;
//   dp = -beta a du;  dk = G^T u + S_{t-1}^T dp;  G <- a G + dp k^T;
//   dlog_alpha = a da,  dS0 = G at the start.
//
// Rows of S and of G evolve independently given the token's k, q, a and beta, so
// one CTA owns a block of RB rows of one (sequence, head) and runs two passes:
//   pass 1  the forward over the whole sequence for its rows, storing the rows'
//           state every kSub tokens (a checkpoint) in the workspace;
//   pass 2  the blocks of kSub tokens in reverse: the block's states are recomputed
//           from its checkpoint into registers, then its tokens are walked backwards.
// dv is complete per row and written directly; dq, dk, dbeta and dalpha sum over
// all rows, so each CTA writes its rows' sums per token to the workspace and a
// second kernel adds the row blocks (a fixed order: the result is deterministic).
// Token inputs are staged in shared memory by cp.async, one block ahead.
//
// fp32 CUDA cores throughout.  This is the recurrent form of the backward; the
// chunked tensor-core form is the next step for it.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gdn_internal.h"

// Scratch of the allocation-free backward (gdn_chunk_bwd_noalloc): a fixed array in
// the library's own device memory, so that a caller that cannot allocate device memory
// still gets the per-token backward's checkpoints and per-row partial sums.  Every
// device that loads the library holds it until the process exits.  In host code this
// name is only a stand-in for the device array: kernels get its device address from
// bwd_noalloc_scratch() below, never the name itself.
static __device__ __align__(256) unsigned char g_bwd_noalloc_scratch[gdn::kBwdNoAllocScratchBytes];

namespace gdn {
namespace {

constexpr int kBwdThreads = 256;  // 8 warps
constexpr int kSub = 8;           // tokens per checkpoint interval / register block

// rows of S per CTA: each warp holds 2 accesses of 32 / (DK / 4) rows
template <int DK>
__host__ __device__ constexpr int bwd_rows() { return 16 * (32 / (DK / 4)); }

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ float4 ld4s(const T* p);  // 4 consecutive elements from smem
template <>
__device__ __forceinline__ float4 ld4s<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 ld4s<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                     __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}
__device__ __forceinline__ float4 axpy4(float a, float4 x, float4 y) {  // a x + y
  return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}
__device__ __forceinline__ float4 scale4(float a, float4 x) {
  return make_float4(a * x.x, a * x.y, a * x.z, a * x.w);
}
__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}
// sum over the LPR lanes of a row group (lanes differ in their low bits)
template <int LPR>
__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Shared-memory layout of one CTA (element type TIn for the staged token inputs).
template <int DK, typename TIn>
struct BwdSmem {
  static constexpr int RB = bwd_rows<DK>();
  // per token: dq[DK], dk[DK], dbeta, dalpha, padded to keep float4 stores aligned
  static constexpr int RED = 2 * DK + 4;
  // one staging buffer: k, q [kSub][DK], v, dO [kSub][RB] (TIn), log alpha, beta [kSub]
  static constexpr size_t kOff = 0;
  static constexpr size_t qOff = kOff + (size_t)kSub * DK * sizeof(TIn);
  static constexpr size_t vOff = qOff + (size_t)kSub * DK * sizeof(TIn);
  static constexpr size_t oOff = vOff + (size_t)kSub * RB * sizeof(TIn);
  static constexpr size_t laOff = oOff + (size_t)kSub * RB * sizeof(TIn);
  static constexpr size_t beOff = laOff + kSub * sizeof(float);
  static constexpr size_t stage = (beOff + kSub * sizeof(float) + 127) / 128 * 128;
  static constexpr size_t redOff = 2 * stage;
  static constexpr size_t bytes = redOff + (size_t)8 * kSub * RED * sizeof(float);
};

struct BwdArgsDev {
  const void *q, *k, *v, *dout;
  const float *log_alpha, *beta, *S0, *dS_final;
  void *dv;
  float* dS0;
  float* ckpt;     // [slots][H][dv][DK]
  float* part_q;   // [NRB][rows * H][DK]
  float* part_k;   // [NRB][rows * H][DK]
  float* part_b;   // [NRB][rows * H]
  float* part_a;   // [NRB][rows * H]
  const int32_t* cu_seqlens;
  long long rows;  // B * T
  int H, T, dv_, N;
};

template <int DK, typename TIn>
__global__ void __launch_bounds__(kBwdThreads, 2) gdn_bwd_rows_kernel(const BwdArgsDev A) {
  using SM = BwdSmem<DK, TIn>;
  constexpr int LPR = DK / 4;       // lanes per row, 4 columns each
  constexpr int RPW = 32 / LPR;     // rows per warp access
  constexpr int RB = SM::RB;
  constexpr int RED = SM::RED;
  extern __shared__ __align__(128) unsigned char smem[];
  float* red = reinterpret_cast<float*>(smem + SM::redOff);

  const int H = A.H, dv = A.dv_;
  const int unit = blockIdx.x, rb = blockIdx.y;
  const int n = unit / H, h = unit % H;
  const int rb0 = rb * RB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c4 = lane % LPR, rsub = lane / LPR;
  const int rl0 = warp * RPW + rsub, rl1 = rl0 + 8 * RPW;  // this thread's rows in the block
  const int r0 = rb0 + rl0, r1 = rb0 + rl1;
  const bool ok0 = r0 < dv, ok1 = r1 < dv;
  const int nrows = min(RB, dv - rb0);  // rows of the block inside dv (a multiple of 16)

  long long row0, len;
  if (A.cu_seqlens) {
    int a = A.cu_seqlens[n], b = A.cu_seqlens[n + 1];
    a = min(max(a, 0), A.T);
    b = min(max(b, a), A.T);
    row0 = a;
    len = b - a;
  } else {
    row0 = (long long)n * A.T;
    len = A.T;
  }
  const int nsb = (int)((len + kSub - 1) / kSub);
  const long long slot0 = row0 / kSub + n;  // this sequence's first checkpoint slot
  const size_t sidx = ((size_t)n * H + h) * dv * DK;  // S0 / dS_final / dS0 of this unit
  const TIn* kin = reinterpret_cast<const TIn*>(A.k);
  const TIn* qin = reinterpret_cast<const TIn*>(A.q);
  const TIn* vin = reinterpret_cast<const TIn*>(A.v);
  const TIn* oin = reinterpret_cast<const TIn*>(A.dout);

  // issue the cp.async copies of block sb (its first kSub tokens) into buffer sb & 1
  auto stage_load = [&](int sb, bool backward) {
    unsigned char* st = smem + (size_t)(sb & 1) * SM::stage;
    const long long t0 = (long long)sb * kSub;
    const int nt = (int)min((long long)kSub, len - t0);
    constexpr int KCH = DK * (int)sizeof(TIn) / 16;  // 16-byte pieces of a k or q row
    for (int idx = tid; idx < nt * KCH; idx += kBwdThreads) {
      const int i = idx / KCH, c = idx % KCH;
      const size_t g = ((size_t)(row0 + t0 + i) * H + h) * DK;
      cp_async16(st + SM::kOff + (size_t)i * DK * sizeof(TIn) + 16 * c,
                 reinterpret_cast<const unsigned char*>(kin + g) + 16 * c);
      if (backward)
        cp_async16(st + SM::qOff + (size_t)i * DK * sizeof(TIn) + 16 * c,
                   reinterpret_cast<const unsigned char*>(qin + g) + 16 * c);
    }
    const int VCH = nrows * (int)sizeof(TIn) / 16;  // 16-byte pieces of the block's rows
    for (int idx = tid; idx < nt * VCH; idx += kBwdThreads) {
      const int i = idx / VCH, c = idx % VCH;
      const size_t g = ((size_t)(row0 + t0 + i) * H + h) * dv + rb0;
      cp_async16(st + SM::vOff + (size_t)i * RB * sizeof(TIn) + 16 * c,
                 reinterpret_cast<const unsigned char*>(vin + g) + 16 * c);
      if (backward)
        cp_async16(st + SM::oOff + (size_t)i * RB * sizeof(TIn) + 16 * c,
                   reinterpret_cast<const unsigned char*>(oin + g) + 16 * c);
    }
    if (tid < nt) {
      const size_t g = (size_t)(row0 + t0 + tid) * H + h;
      cp_async4(st + SM::laOff + 4 * tid, A.log_alpha + g);
      cp_async4(st + SM::beOff + 4 * tid, A.beta + g);
    }
    cp_async_commit();
  };
  // the inputs of token i of the staged block in buffer b
  struct Tok {
    float4 k, q;
    float a, b, v0, v1, o0, o1;
  };
  auto token = [&](int b, int i, bool backward) {
    const unsigned char* st = smem + (size_t)b * SM::stage;
    Tok x;
    x.k = ld4s<TIn>(reinterpret_cast<const TIn*>(st + SM::kOff) + i * DK + 4 * c4);
    x.q = backward ? ld4s<TIn>(reinterpret_cast<const TIn*>(st + SM::qOff) + i * DK + 4 * c4)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    x.a = __expf(reinterpret_cast<const float*>(st + SM::laOff)[i]);
    x.b = reinterpret_cast<const float*>(st + SM::beOff)[i];
    const TIn* vs = reinterpret_cast<const TIn*>(st + SM::vOff) + i * RB;
    const TIn* os = reinterpret_cast<const TIn*>(st + SM::oOff) + i * RB;
    x.v0 = ok0 ? to_f<TIn>(vs[rl0]) : 0.f;
    x.v1 = ok1 ? to_f<TIn>(vs[rl1]) : 0.f;
    x.o0 = (backward && ok0) ? to_f<TIn>(os[rl0]) : 0.f;
    x.o1 = (backward && ok1) ? to_f<TIn>(os[rl1]) : 0.f;
    return x;
  };

  // ---------------- pass 1: forward, checkpoint every kSub tokens ----------------
  float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0;
  if (A.S0) {
    if (ok0) s0 = *reinterpret_cast<const float4*>(A.S0 + sidx + (size_t)r0 * DK + 4 * c4);
    if (ok1) s1 = *reinterpret_cast<const float4*>(A.S0 + sidx + (size_t)r1 * DK + 4 * c4);
  }
  if (nsb > 0) stage_load(0, false);
  for (int sb = 0; sb < nsb; ++sb) {
    if (sb + 1 < nsb) {
      stage_load(sb + 1, false);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    float* ck = A.ckpt + ((size_t)(slot0 + sb) * H + h) * dv * DK;
    if (ok0) *reinterpret_cast<float4*>(ck + (size_t)r0 * DK + 4 * c4) = s0;
    if (ok1) *reinterpret_cast<float4*>(ck + (size_t)r1 * DK + 4 * c4) = s1;
    const int nt = (int)min((long long)kSub, len - (long long)sb * kSub);
#pragma unroll
    for (int i = 0; i < kSub; ++i) {
      if (i < nt) {
        const Tok x = token(sb & 1, i, false);
        const float p0 = row_sum<LPR>(dot4(s0, x.k)), p1 = row_sum<LPR>(dot4(s1, x.k));
        const float u0 = x.b * (x.v0 - x.a * p0), u1 = x.b * (x.v1 - x.a * p1);
        s0 = axpy4(u0, x.k, scale4(x.a, s0));
        s1 = axpy4(u1, x.k, scale4(x.a, s1));
      }
    }
    __syncthreads();  // buffer sb & 1 is read; the next prefetch may refill it
  }

  // ---------------- pass 2: blocks in reverse, tokens in reverse ----------------
  float4 g0 = make_float4(0.f, 0.f, 0.f, 0.f), g1 = g0;
  if (A.dS_final) {
    if (ok0) g0 = *reinterpret_cast<const float4*>(A.dS_final + sidx + (size_t)r0 * DK + 4 * c4);
    if (ok1) g1 = *reinterpret_cast<const float4*>(A.dS_final + sidx + (size_t)r1 * DK + 4 * c4);
  }
  const size_t uh = (size_t)A.rows * H;  // stride of one row block in the partial buffers
  if (nsb > 0) stage_load(nsb - 1, true);
  for (int sb = nsb - 1; sb >= 0; --sb) {
    float4 st0[kSub], st1[kSub];  // the rows' state before each token of the block
    float pv0[kSub], pv1[kSub];   // the rows' predictions S_{t-1} k_t
    {
      const float* ck = A.ckpt + ((size_t)(slot0 + sb) * H + h) * dv * DK;
      st0[0] = ok0 ? *reinterpret_cast<const float4*>(ck + (size_t)r0 * DK + 4 * c4)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      st1[0] = ok1 ? *reinterpret_cast<const float4*>(ck + (size_t)r1 * DK + 4 * c4)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (sb > 0) {
      stage_load(sb - 1, true);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const int b = sb & 1;
    const int nt = (int)min((long long)kSub, len - (long long)sb * kSub);
#pragma unroll
    for (int i = 0; i < kSub; ++i) {
      if (i < nt) {
        const Tok x = token(b, i, false);
        pv0[i] = row_sum<LPR>(dot4(st0[i], x.k));
        pv1[i] = row_sum<LPR>(dot4(st1[i], x.k));
        if (i + 1 < kSub) {
          const float u0 = x.b * (x.v0 - x.a * pv0[i]), u1 = x.b * (x.v1 - x.a * pv1[i]);
          st0[i + 1] = axpy4(u0, x.k, scale4(x.a, st0[i]));
          st1[i + 1] = axpy4(u1, x.k, scale4(x.a, st1[i]));
        }
      }
    }
#pragma unroll
    for (int i = kSub - 1; i >= 0; --i) {
      if (i < nt) {
        const Tok x = token(b, i, true);
        const float p0 = pv0[i], p1 = pv1[i];
        const float e0 = x.v0 - x.a * p0, e1 = x.v1 - x.a * p1;  // prediction errors
        const float u0 = x.b * e0, u1 = x.b * e1;
        g0 = axpy4(x.o0, x.q, g0);  // G += dO q^T
        g1 = axpy4(x.o1, x.q, g1);
        const float du0 = row_sum<LPR>(dot4(g0, x.k)), du1 = row_sum<LPR>(dot4(g1, x.k));
        const long long t = (long long)sb * kSub + i;
        const size_t grow = (size_t)(row0 + t) * H + h;
        if (c4 == 0) {
          if (ok0) reinterpret_cast<TIn*>(A.dv)[grow * dv + r0] = from_f<TIn>(x.b * du0);
          if (ok1) reinterpret_cast<TIn*>(A.dv)[grow * dv + r1] = from_f<TIn>(x.b * du1);
        }
        // <G, S_{t-1}> enters dalpha as this lane's partial sum (the warp and block
        // sums below finish it); per-row scalars count once per row (lane c4 == 0)
        float db = 0.f, da = dot4(g0, st0[i]) + dot4(g1, st1[i]);
        if (c4 == 0) {
          db = du0 * e0 + du1 * e1;
          da -= x.b * (du0 * p0 + du1 * p1);
        }
        const float dp0 = -x.b * x.a * du0, dp1 = -x.b * x.a * du1;
        // dq = a S_{t-1}^T dO + k (u . dO);  dk = G^T u + S_{t-1}^T dp (this warp's rows)
        float4 dq = add4(scale4(x.a * x.o0, st0[i]), scale4(x.a * x.o1, st1[i]));
        dq = axpy4(u0 * x.o0 + u1 * x.o1, x.k, dq);
        float4 dk = add4(scale4(u0, g0), scale4(u1, g1));
        dk = axpy4(dp0, st0[i], dk);
        dk = axpy4(dp1, st1[i], dk);
        g0 = axpy4(dp0, x.k, scale4(x.a, g0));  // G <- a G + dp k^T
        g1 = axpy4(dp1, x.k, scale4(x.a, g1));
        // sum over the row groups of the warp, then over the whole warp for scalars
#pragma unroll
        for (int o = LPR; o < 32; o <<= 1) {
          dq.x += __shfl_xor_sync(0xffffffffu, dq.x, o);
          dq.y += __shfl_xor_sync(0xffffffffu, dq.y, o);
          dq.z += __shfl_xor_sync(0xffffffffu, dq.z, o);
          dq.w += __shfl_xor_sync(0xffffffffu, dq.w, o);
          dk.x += __shfl_xor_sync(0xffffffffu, dk.x, o);
          dk.y += __shfl_xor_sync(0xffffffffu, dk.y, o);
          dk.z += __shfl_xor_sync(0xffffffffu, dk.z, o);
          dk.w += __shfl_xor_sync(0xffffffffu, dk.w, o);
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          db += __shfl_xor_sync(0xffffffffu, db, o);
          da += __shfl_xor_sync(0xffffffffu, da, o);
        }
        float* rw = red + ((size_t)warp * kSub + i) * RED;
        if (rsub == 0) {
          *reinterpret_cast<float4*>(rw + 4 * c4) = dq;
          *reinterpret_cast<float4*>(rw + DK + 4 * c4) = dk;
        }
        if (lane == 0) {
          rw[2 * DK] = db;
          rw[2 * DK + 1] = da;
        }
      }
    }
    __syncthreads();
    // add the 8 warps' sums of every token of the block, in warp order
    for (int idx = tid; idx < nt * RED; idx += kBwdThreads) {
      const int i = idx / RED, c = idx % RED;
      if (c >= 2 * DK + 2) continue;  // padding
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) acc += red[((size_t)w * kSub + i) * RED + c];
      const size_t grow = (size_t)(row0 + (long long)sb * kSub + i) * H + h;
      const size_t pb = (size_t)rb * uh + grow;
      if (c < DK)
        A.part_q[pb * DK + c] = acc;
      else if (c < 2 * DK)
        A.part_k[pb * DK + (c - DK)] = acc;
      else if (c == 2 * DK)
        A.part_b[pb] = acc;
      else
        A.part_a[pb] = acc;
    }
    __syncthreads();  // red and staging buffer b are free again
  }
  if (A.dS0) {
    if (ok0) *reinterpret_cast<float4*>(A.dS0 + sidx + (size_t)r0 * DK + 4 * c4) = g0;
    if (ok1) *reinterpret_cast<float4*>(A.dS0 + sidx + (size_t)r1 * DK + 4 * c4) = g1;
  }
}

// dq, dk: the row blocks' sums, added in block order and stored in the input dtype;
// dbeta and dlog_alpha = a * dalpha likewise.  One thread per 4 columns of a
// (token, head).
template <int DK, typename TIn>
__global__ void __launch_bounds__(256)
gdn_bwd_reduce_kernel(const float* __restrict__ part_q, const float* __restrict__ part_k,
                      const float* __restrict__ part_b, const float* __restrict__ part_a,
                      const float* __restrict__ log_alpha, void* dq, void* dk,
                      float* dlog_alpha, float* dbeta, long long uh, int nrb) {
  constexpr int G4 = DK / 4;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= uh * G4) return;
  const long long u = idx / G4;
  const int c = (int)(idx % G4);
  float4 aq = make_float4(0.f, 0.f, 0.f, 0.f), ak = aq;
  for (int r = 0; r < nrb; ++r) {
    const size_t pb = (size_t)r * uh + u;
    aq = add4(aq, *reinterpret_cast<const float4*>(part_q + pb * DK + 4 * c));
    ak = add4(ak, *reinterpret_cast<const float4*>(part_k + pb * DK + 4 * c));
  }
  TIn* q = reinterpret_cast<TIn*>(dq) + (size_t)u * DK + 4 * c;
  TIn* k = reinterpret_cast<TIn*>(dk) + (size_t)u * DK + 4 * c;
  q[0] = from_f<TIn>(aq.x); q[1] = from_f<TIn>(aq.y); q[2] = from_f<TIn>(aq.z); q[3] = from_f<TIn>(aq.w);
  k[0] = from_f<TIn>(ak.x); k[1] = from_f<TIn>(ak.y); k[2] = from_f<TIn>(ak.z); k[3] = from_f<TIn>(ak.w);
  if (c == 0) {
    float b = 0.f, a = 0.f;
    for (int r = 0; r < nrb; ++r) {
      b += part_b[(size_t)r * uh + u];
      a += part_a[(size_t)r * uh + u];
    }
    dbeta[u] = b;
    dlog_alpha[u] = __expf(log_alpha[u]) * a;
  }
}

// Workspace carve-up (all fp32, each part 256-byte aligned).
struct BwdWorkspace {
  size_t ckpt, part_q, part_k, part_b, part_a, total;
};
size_t align256(size_t x) { return (x + 255) / 256 * 256; }
BwdWorkspace bwd_layout(long long rows, int H, int dk, int dv, int N) {
  const int RB = dk == 16 ? bwd_rows<16>() : dk == 32 ? bwd_rows<32>()
               : dk == 64 ? bwd_rows<64>() : bwd_rows<128>();
  const long long nrb = (dv + RB - 1) / RB;
  const long long slots = rows / kSub + N + 1;
  BwdWorkspace w;
  w.ckpt = 0;
  w.part_q = w.ckpt + align256((size_t)slots * H * dv * dk * 4);
  w.part_k = w.part_q + align256((size_t)nrb * rows * H * dk * 4);
  w.part_b = w.part_k + align256((size_t)nrb * rows * H * dk * 4);
  w.part_a = w.part_b + align256((size_t)nrb * rows * H * 4);
  w.total = w.part_a + align256((size_t)nrb * rows * H * 4);
  return w;
}

template <int DK, typename TIn>
cudaError_t launch_bwd_t(const BwdArgs& a, cudaStream_t stream) {
  using SM = BwdSmem<DK, TIn>;
  const long long rows = (long long)a.B * a.T;
  const BwdWorkspace w = bwd_layout(rows, a.H, DK, a.dv, a.N);
  unsigned char* ws = reinterpret_cast<unsigned char*>(a.workspace);
  BwdArgsDev d;
  d.q = a.q; d.k = a.k; d.v = a.v; d.dout = a.dout;
  d.log_alpha = a.log_alpha; d.beta = a.beta; d.S0 = a.S0; d.dS_final = a.dS_final;
  d.dv = a.dv_out; d.dS0 = a.dS0;
  d.ckpt = reinterpret_cast<float*>(ws + w.ckpt);
  d.part_q = reinterpret_cast<float*>(ws + w.part_q);
  d.part_k = reinterpret_cast<float*>(ws + w.part_k);
  d.part_b = reinterpret_cast<float*>(ws + w.part_b);
  d.part_a = reinterpret_cast<float*>(ws + w.part_a);
  d.cu_seqlens = a.cu_seqlens;
  d.rows = rows; d.H = a.H; d.T = a.T; d.dv_ = a.dv; d.N = a.N;
  const int nrb = (a.dv + SM::RB - 1) / SM::RB;
  const long long units = (long long)a.N * a.H;
  if (units == 0) return cudaSuccess;
  if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
  static std::atomic<unsigned long long> smem_set{0};
  cudaError_t e = ensure_smem_cap(gdn_bwd_rows_kernel<DK, TIn>, (int)SM::bytes, smem_set);
  if (e != cudaSuccess) return e;
  gdn_bwd_rows_kernel<DK, TIn><<<dim3((unsigned)units, nrb), kBwdThreads, SM::bytes, stream>>>(d);
  e = cudaGetLastError();
  if (e != cudaSuccess || rows == 0) return e;
  const long long uh = rows * a.H;
  const long long threads = uh * (DK / 4);
  gdn_bwd_reduce_kernel<DK, TIn><<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(
      d.part_q, d.part_k, d.part_b, d.part_a, a.log_alpha, a.dq, a.dk_out, a.dlog_alpha,
      a.dbeta, uh, nrb);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_workspace_bytes(long long rows, int H, int dk, int dv, int N) {
  if (rows == 0) return 0;
  return bwd_layout(rows, H, dk, dv, N).total;
}

// Device address of the fixed scratch array on the current device, looked up once per
// device (with that device current) and kept.  The first lookup may load the library's
// device code on that device, so a first call should not happen during stream capture.
cudaError_t bwd_noalloc_scratch(void** ptr) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static void* addr[kMaxDev] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream) {
  switch (a.dk) {
    case 16: return a.bf16 ? launch_bwd_t<16, __nv_bfloat16>(a, stream) : launch_bwd_t<16, float>(a, stream);
    case 32: return a.bf16 ? launch_bwd_t<32, __nv_bfloat16>(a, stream) : launch_bwd_t<32, float>(a, stream);
    case 64: return a.bf16 ? launch_bwd_t<64, __nv_bfloat16>(a, stream) : launch_bwd_t<64, float>(a, stream);
    case 128: return a.bf16 ? launch_bwd_t<128, __nv_bfloat16>(a, stream) : launch_bwd_t<128, float>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
