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
// One CTA of 8 warps per (sequence, head).  S is dv x dk fp32 (row-major, dk
// inner).  A row is covered by LPR = dk / 4 lanes holding 4 consecutive columns
// each, so one warp-wide float4 access covers 32 / LPR whole rows (one 512-byte
// contiguous run for dk = 128).  Warp w takes rows w * RPW, (w + 8) * RPW, ...
// Each lane keeps its part of S in registers between the read and the write; no
// CTA-wide synchronisation is needed.  The step is bound by HBM: 2 dk dv 4 bytes of
// state per (sequence, head) against a few hundred FLOPs per byte-pair.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kDecThreads = 256;  // 8 warps

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
__global__ void __launch_bounds__(kDecThreads)
gdn_decode_kernel(const void* __restrict__ q, const void* __restrict__ k,
                  const void* __restrict__ v, const float* __restrict__ log_alpha,
                  const float* __restrict__ beta, float* __restrict__ S, void* __restrict__ out,
                  int dv, int bf16) {
  constexpr int LPR = DK / 4;        // lanes per row
  constexpr int RPW = 32 / LPR;      // rows per warp access
  constexpr int MAXIT = 128 / (8 * RPW);  // accesses per lane for dv = 128
  const int nh = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c4 = lane % LPR;         // this lane's columns 4 c4 .. 4 c4 + 3
  const int rsub = lane / LPR;       // row within the warp access
  const bool isbf = bf16 != 0;

  const float alpha = expf(log_alpha[nh]);
  const float b = beta[nh];
  const float4 kk = load4(k, (size_t)nh * DK + 4 * c4, isbf);
  const float4 qq = load4(q, (size_t)nh * DK + 4 * c4, isbf);
  // k . q over the row's DK columns (the LPR lanes of a row group hold all of them)
  float kq = kk.x * qq.x + kk.y * qq.y + kk.z * qq.z + kk.w * qq.w;
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);

  float4* Sv = reinterpret_cast<float4*>(S + (size_t)nh * dv * DK);
  float4 s[MAXIT];
  // issue every load of this lane's part of S before using any
#pragma unroll
  for (int it = 0; it < MAXIT; ++it) {
    const int r = (it * 8 + warp) * RPW + rsub;
    if (r < dv) s[it] = Sv[(size_t)r * LPR + c4];
  }
#pragma unroll
  for (int it = 0; it < MAXIT; ++it) {
    const int r = (it * 8 + warp) * RPW + rsub;
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

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  const long long ctas = (long long)a.N * a.H;
  if (ctas == 0) return cudaSuccess;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)ctas);
  switch (a.dk) {
    case 16:
      gdn_decode_kernel<16><<<grid, kDecThreads, 0, stream>>>(a.q, a.k, a.v, a.log_alpha, a.beta,
                                                              a.S, a.out, a.dv, a.bf16);
      break;
    case 32:
      gdn_decode_kernel<32><<<grid, kDecThreads, 0, stream>>>(a.q, a.k, a.v, a.log_alpha, a.beta,
                                                              a.S, a.out, a.dv, a.bf16);
      break;
    case 64:
      gdn_decode_kernel<64><<<grid, kDecThreads, 0, stream>>>(a.q, a.k, a.v, a.log_alpha, a.beta,
                                                              a.S, a.out, a.dv, a.bf16);
      break;
    case 128:
      gdn_decode_kernel<128><<<grid, kDecThreads, 0, stream>>>(a.q, a.k, a.v, a.log_alpha, a.beta,
                                                               a.S, a.out, a.dv, a.bf16);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace gdn
