// The forward by the per-token recurrence on CUDA cores, fp32 arithmetic: the path for
// fp32 inputs and for the shapes the tcgen05 kernel does not cover.
//
//   a = e^{log alpha},  p = S_{t-1} k,  u = beta (v - a p),  S_t = a S_{t-1} + u k^T,
//   o_t = S_t q_t
//
// (Nyysyyan, "Gated-DeltaNet", first equation block, in its gate -> predict -> write
// order; in the linear mode of the "Mamba2" section the erase strength is 0 and the
// write strength 1, so u = v.)  On CUDA cores the chunk form buys nothing over the
// recurrence it equals, and the recurrence is exact in fp32 and parallel over the rows
// of S: row r of S_t, and o_t[r], depend only on row r of S_{t-1} and on the token.  So
// one CTA owns RB rows of one (sequence, head) and walks the sequence; each thread holds
// 4 columns of 2 rows in registers, a row's dot products are warp-shuffle sums over the
// dk / 4 lanes that hold it, and no CTA needs another's results.  Token inputs are
// staged in shared memory by cp.async, one block of kRecSub tokens ahead.  CTAs have 8
// warps; when that leaves most SMs idle (few (sequence, head) pairs), CTAs of 8 rows
// (16 at dk = 16) spread the same rows over more SMs, so that each per-token chain runs
// with its scheduler nearly to itself.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kRecSub = 16;  // tokens per staged block

// rows one warp access covers, and the warps of the small-CTA shape (8 rows per CTA,
// 16 at dk = 16): at least 16 bytes of each staged v row for either input type
template <int DK>
__host__ __device__ constexpr int rec_rpw() { return 32 / (DK / 4); }
template <int DK>
__host__ __device__ constexpr int rec_small_warps() { return rec_rpw<DK>() >= 4 ? 1 : 4 / rec_rpw<DK>(); }
// rows per CTA of NW warps: each warp holds 2 accesses
template <int DK, int NW>
__host__ __device__ constexpr int rec_rows() { return 2 * NW * rec_rpw<DK>(); }

template <typename T>
__device__ __forceinline__ float rec_f(T x);
template <>
__device__ __forceinline__ float rec_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float rec_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ float4 rec_ld4(const T* p);
template <>
__device__ __forceinline__ float4 rec_ld4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 rec_ld4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                     __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}
template <typename T>
__device__ __forceinline__ T rec_out(float x);
template <>
__device__ __forceinline__ float rec_out<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 rec_out<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ void rec_cp16(void* dst, const void* src) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void rec_cp4(void* dst, const void* src) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void rec_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void rec_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float rec_dot(float4 a, float4 b) {
  return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}
template <int LPR>
__device__ __forceinline__ float rec_rowsum(float x) {
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
// a s + u k
__device__ __forceinline__ float4 rec_update(float a, float4 s, float u, float4 k) {
  return make_float4(fmaf(u, k.x, a * s.x), fmaf(u, k.y, a * s.y), fmaf(u, k.z, a * s.z),
                     fmaf(u, k.w, a * s.w));
}

// one staging buffer: k, q [kRecSub][DK], v [kRecSub][RB] (TIn), log alpha, beta [kRecSub]
template <int DK, typename TIn, int NW>
struct RecSmem {
  static constexpr int RB = rec_rows<DK, NW>();
  static constexpr size_t kOff = 0;
  static constexpr size_t qOff = kOff + (size_t)kRecSub * DK * sizeof(TIn);
  static constexpr size_t vOff = qOff + (size_t)kRecSub * DK * sizeof(TIn);
  static constexpr size_t laOff = vOff + (size_t)kRecSub * RB * sizeof(TIn);
  static constexpr size_t beOff = laOff + kRecSub * sizeof(float);
  static constexpr size_t stage = (beOff + kRecSub * sizeof(float) + 127) / 128 * 128;
  static constexpr size_t bytes = 2 * stage;
};

template <int DK, typename TIn, int NW>
__global__ void __launch_bounds__(32 * NW)
gdn_rec_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k, const TIn* __restrict__ v,
               const float* __restrict__ log_alpha, const float* __restrict__ beta,
               const float* __restrict__ S0, TIn* __restrict__ out, float* __restrict__ S_final,
               const int32_t* __restrict__ cu_seqlens, int H, int T, int dv) {
  using SM = RecSmem<DK, TIn, NW>;
  constexpr int kRecThreads = 32 * NW;
  constexpr int LPR = DK / 4;    // lanes per row, 4 columns each
  constexpr int RPW = 32 / LPR;  // rows per warp access
  constexpr int RB = SM::RB;
  extern __shared__ __align__(128) unsigned char rec_smem[];
  const int unit = blockIdx.x, rb = blockIdx.y;
  const int n = unit / H, h = unit % H;
  const int rb0 = rb * RB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c4 = lane % LPR, rsub = lane / LPR;
  const int rl0 = warp * RPW + rsub, rl1 = rl0 + NW * RPW;  // this thread's rows in the block
  const int r0 = rb0 + rl0, r1 = rb0 + rl1;
  const bool ok0 = r0 < dv, ok1 = r1 < dv;
  const int nrows = min(RB, dv - rb0);  // a multiple of 8
  const bool linear = beta == nullptr;  // erase 0, write 1

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
  const size_t sidx = ((size_t)n * H + h) * dv * DK;

  auto stage_load = [&](int sb) {
    unsigned char* st = rec_smem + (size_t)(sb & 1) * SM::stage;
    const long long t0 = (long long)sb * kRecSub;
    const int nt = (int)min((long long)kRecSub, len - t0);
    constexpr int KCH = DK * (int)sizeof(TIn) / 16;
    for (int idx = tid; idx < nt * KCH; idx += kRecThreads) {
      const int i = idx / KCH, c = idx % KCH;
      const size_t g = ((size_t)(row0 + t0 + i) * H + h) * DK;
      rec_cp16(st + SM::kOff + (size_t)i * DK * sizeof(TIn) + 16 * c,
               reinterpret_cast<const unsigned char*>(k + g) + 16 * c);
      rec_cp16(st + SM::qOff + (size_t)i * DK * sizeof(TIn) + 16 * c,
               reinterpret_cast<const unsigned char*>(q + g) + 16 * c);
    }
    const int VCH = nrows * (int)sizeof(TIn) / 16;
    for (int idx = tid; idx < nt * VCH; idx += kRecThreads) {
      const int i = idx / VCH, c = idx % VCH;
      const size_t g = ((size_t)(row0 + t0 + i) * H + h) * dv + rb0;
      rec_cp16(st + SM::vOff + (size_t)i * RB * sizeof(TIn) + 16 * c,
               reinterpret_cast<const unsigned char*>(v + g) + 16 * c);
    }
    if (tid < nt) {
      const size_t g = (size_t)(row0 + t0 + tid) * H + h;
      float* la = reinterpret_cast<float*>(st + SM::laOff);
      float* be = reinterpret_cast<float*>(st + SM::beOff);
      if (log_alpha) rec_cp4(la + tid, log_alpha + g); else la[tid] = 0.f;
      if (beta) rec_cp4(be + tid, beta + g); else be[tid] = 1.f;
    }
    rec_commit();
  };

  float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0;
  if (S0) {
    if (ok0) s0 = *reinterpret_cast<const float4*>(S0 + sidx + (size_t)r0 * DK + 4 * c4);
    if (ok1) s1 = *reinterpret_cast<const float4*>(S0 + sidx + (size_t)r1 * DK + 4 * c4);
  }
  const int nsb = (int)((len + kRecSub - 1) / kRecSub);
  if (nsb > 0) stage_load(0);
  for (int sb = 0; sb < nsb; ++sb) {
    if (sb + 1 < nsb) {
      stage_load(sb + 1);
      rec_wait<1>();
    } else {
      rec_wait<0>();
    }
    __syncthreads();
    const unsigned char* st = rec_smem + (size_t)(sb & 1) * SM::stage;
    const long long t0 = (long long)sb * kRecSub;
    const int nt = (int)min((long long)kRecSub, len - t0);
#pragma unroll 4
    for (int i = 0; i < nt; ++i) {
      const float4 kk = rec_ld4<TIn>(reinterpret_cast<const TIn*>(st + SM::kOff) + i * DK + 4 * c4);
      const float4 qq = rec_ld4<TIn>(reinterpret_cast<const TIn*>(st + SM::qOff) + i * DK + 4 * c4);
      const float a = __expf(reinterpret_cast<const float*>(st + SM::laOff)[i]);
      const float b = reinterpret_cast<const float*>(st + SM::beOff)[i];
      const TIn* vs = reinterpret_cast<const TIn*>(st + SM::vOff) + i * RB;
      const float v0 = ok0 ? rec_f<TIn>(vs[rl0]) : 0.f, v1 = ok1 ? rec_f<TIn>(vs[rl1]) : 0.f;
      float u0 = b * v0, u1 = b * v1;
      if (!linear) {  // the correction subtracts the gated state's prediction along k
        const float p0 = rec_rowsum<LPR>(rec_dot(s0, kk)), p1 = rec_rowsum<LPR>(rec_dot(s1, kk));
        u0 -= b * a * p0;
        u1 -= b * a * p1;
      }
      s0 = rec_update(a, s0, u0, kk);
      s1 = rec_update(a, s1, u1, kk);
      const float o0 = rec_rowsum<LPR>(rec_dot(s0, qq)), o1 = rec_rowsum<LPR>(rec_dot(s1, qq));
      if (c4 == 0) {
        const size_t g = ((size_t)(row0 + t0 + i) * H + h) * dv;
        if (ok0) out[g + r0] = rec_out<TIn>(o0);
        if (ok1) out[g + r1] = rec_out<TIn>(o1);
      }
    }
    __syncthreads();  // buffer sb & 1 is read; the next prefetch may refill it
  }
  if (S_final) {
    if (ok0) *reinterpret_cast<float4*>(S_final + sidx + (size_t)r0 * DK + 4 * c4) = s0;
    if (ok1) *reinterpret_cast<float4*>(S_final + sidx + (size_t)r1 * DK + 4 * c4) = s1;
  }
}

template <int DK, typename TIn, int NW>
cudaError_t launch_rec_nw(const FwdArgs& a, long long units, cudaStream_t stream) {
  using SM = RecSmem<DK, TIn, NW>;
  const int nrb = (a.dv + SM::RB - 1) / SM::RB;
  gdn_rec_kernel<DK, TIn, NW><<<dim3((unsigned)units, nrb), 32 * NW, SM::bytes, stream>>>(
      (const TIn*)a.q, (const TIn*)a.k, (const TIn*)a.v, a.log_alpha, a.beta, a.S0, (TIn*)a.out,
      a.S_final, a.cu_seqlens, a.H, a.T, a.dv);
  return cudaGetLastError();
}

int rec_sm_count() {
  static std::atomic<int> sms{0};
  int n = sms.load();
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    sms.store(n);
  }
  return n;
}

template <int DK, typename TIn>
cudaError_t launch_rec_t(const FwdArgs& a, cudaStream_t stream) {
  const long long units = (long long)a.N * a.H;
  if (units == 0) return cudaSuccess;
  if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
  // 8-warp CTAs unless they would leave more than half of the SMs idle
  const long long big = units * ((a.dv + rec_rows<DK, 8>() - 1) / rec_rows<DK, 8>());
  if (2 * big >= rec_sm_count()) return launch_rec_nw<DK, TIn, 8>(a, units, stream);
  return launch_rec_nw<DK, TIn, rec_small_warps<DK>()>(a, units, stream);
}

}  // namespace

cudaError_t launch_rec(const FwdArgs& a, cudaStream_t stream) {
  switch (a.dk) {
    case 16: return a.bf16 ? launch_rec_t<16, __nv_bfloat16>(a, stream) : launch_rec_t<16, float>(a, stream);
    case 32: return a.bf16 ? launch_rec_t<32, __nv_bfloat16>(a, stream) : launch_rec_t<32, float>(a, stream);
    case 64: return a.bf16 ? launch_rec_t<64, __nv_bfloat16>(a, stream) : launch_rec_t<64, float>(a, stream);
    case 128: return a.bf16 ? launch_rec_t<128, __nv_bfloat16>(a, stream) : launch_rec_t<128, float>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
