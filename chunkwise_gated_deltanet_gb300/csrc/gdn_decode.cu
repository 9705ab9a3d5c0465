// Single-token decode step of the Gated DeltaNet recurrence, the recurrent form
// (Nyysyyan, "Gated-DeltaNet" section, first equation block; kkkzoz, "Gated
// DeltaNet" section: gate, predict, delta, write, then read):
//
//     S <- alpha S (I - beta k k^T) + beta v k^T,   o = S q
//
// rewritten so that the state is read once and written once:
//
//     p = S k,  u = beta (v - alpha p),  S <- alpha S + u k^T,
//     o = S_new q = alpha (S q) + u (k . q).
//
// The step is bound by HBM: 2 dk dv 4 bytes of state move per (sequence, head),
// against about 7 dk dv FLOPs.  Rows of S are independent once k, q, alpha and
// beta are known, so the work is cut by rows: one warp per CTA takes kDecRows4
// float4 accesses per lane over a block of rows.  A row is covered by
// LPR = dk / 4 lanes holding 4 consecutive columns each, so one warp access covers
// RPW = 32 / LPR whole rows (one 512-byte contiguous run for dk = 128); a CTA
// covers RPW * kDecRows4 rows (8 for dk = 128), and a (sequence, head) takes
// ceil(dv / that) CTAs.  Small single-warp CTAs keep 32 of them resident per SM,
// each with all of its loads in flight before its first use, which keeps HBM
// busy through the read-then-write shape of the step; each lane holds its part of
// S in registers between the read and the write, with no synchronisation.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kDecThreads = 32;  // one warp
constexpr int kDecRows4 = 8;     // float4 accesses of S per lane

__device__ __forceinline__ float4 load4(const void* p, size_t idx, bool bf16) {
  if (bf16) {
    const uint2 w = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(p) + idx);
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                       __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
  }
  return *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + idx);
}
__device__ __forceinline__ float load1(const void* p, size_t idx, bool bf16) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[idx]);
  return reinterpret_cast<const float*>(p)[idx];
}

template <int DK>
__device__ __forceinline__ constexpr int rows_per_cta() { return (32 / (DK / 4)) * kDecRows4; }

template <int DK, bool BF16>
__global__ void __launch_bounds__(kDecThreads)
gdn_decode_kernel(const void* __restrict__ q, const void* __restrict__ k,
                  const void* __restrict__ v, const float* __restrict__ log_alpha,
                  const float* __restrict__ beta, float* __restrict__ S, void* __restrict__ out,
                  int dv, int splits) {
  constexpr int LPR = DK / 4;        // lanes per row
  constexpr int RPW = 32 / LPR;      // rows per warp access
  const int nh = blockIdx.x / splits;
  const int row0 = (blockIdx.x - nh * splits) * rows_per_cta<DK>();
  const int lane = threadIdx.x;
  const int c4 = lane % LPR;         // this lane's columns 4 c4 .. 4 c4 + 3
  const int rsub = lane / LPR;       // row within the warp access
  constexpr bool isbf = BF16;

  const float alpha = expf(log_alpha[nh]);
  const float b = beta[nh];
  const float4 kk = load4(k, (size_t)nh * DK + 4 * c4, isbf);
  const float4 qq = load4(q, (size_t)nh * DK + 4 * c4, isbf);
  // k . q over the row's DK columns (the LPR lanes of a row group hold all of them)
  float kq = kk.x * qq.x + kk.y * qq.y + kk.z * qq.z + kk.w * qq.w;
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);

  float4* Sv = reinterpret_cast<float4*>(S + (size_t)nh * dv * DK);
  float4 s[kDecRows4];
  // issue every load of this lane's part of S before using any
#pragma unroll
  for (int it = 0; it < kDecRows4; ++it) {
    const int r = row0 + it * RPW + rsub;
    if (r < dv) s[it] = Sv[(size_t)r * LPR + c4];
  }
#pragma unroll
  for (int it = 0; it < kDecRows4; ++it) {
    const int r = row0 + it * RPW + rsub;
    float p = 0.f, sq = 0.f;
    if (r < dv) {
      p = s[it].x * kk.x + s[it].y * kk.y + s[it].z * kk.z + s[it].w * kk.w;
      sq = s[it].x * qq.x + s[it].y * qq.y + s[it].z * qq.z + s[it].w * qq.w;
    }
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) {
      p += __shfl_xor_sync(0xffffffffu, p, o);
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
    }
    if (r < dv) {
      const float vr = load1(v, (size_t)nh * dv + r, isbf);
      const float u = b * (vr - alpha * p);       // beta (v - alpha S k)
      const float4 sn = make_float4(fmaf(alpha, s[it].x, u * kk.x), fmaf(alpha, s[it].y, u * kk.y),
                                    fmaf(alpha, s[it].z, u * kk.z), fmaf(alpha, s[it].w, u * kk.w));
      Sv[(size_t)r * LPR + c4] = sn;
      if (c4 == 0) {
        const float o = fmaf(alpha, sq, u * kq);  // (alpha S + u k^T) q
        if (isbf)
          reinterpret_cast<__nv_bfloat16*>(out)[(size_t)nh * dv + r] = __float2bfloat16_rn(o);
        else
          reinterpret_cast<float*>(out)[(size_t)nh * dv + r] = o;
      }
    }
  }
}

template <int DK>
cudaError_t launch_decode_dk(const DecodeArgs& a, cudaStream_t stream) {
  const int splits = (a.dv + rows_per_cta<DK>() - 1) / rows_per_cta<DK>();
  const long long ctas = (long long)a.N * a.H * splits;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (a.bf16)
    gdn_decode_kernel<DK, true><<<(unsigned)ctas, kDecThreads, 0, stream>>>(
        a.q, a.k, a.v, a.log_alpha, a.beta, a.S, a.out, a.dv, splits);
  else
    gdn_decode_kernel<DK, false><<<(unsigned)ctas, kDecThreads, 0, stream>>>(
        a.q, a.k, a.v, a.log_alpha, a.beta, a.S, a.out, a.dv, splits);
  return cudaGetLastError();
}

}  // namespace

long long decode_ctas(long long N, long long H, int dk, int dv) {
  const int rows = (32 / (dk / 4)) * kDecRows4;  // rows_per_cta<dk>()
  return N * H * ((dv + rows - 1) / rows);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if ((long long)a.N * a.H == 0) return cudaSuccess;
  switch (a.dk) {
    case 16: return launch_decode_dk<16>(a, stream);
    case 32: return launch_decode_dk<32>(a, stream);
    case 64: return launch_decode_dk<64>(a, stream);
    case 128: return launch_decode_dk<128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
