// Folding affine state maps: S <- S M_i + L_i for i = 0 .. count-1, for a batch of
// (sequence, head) states.
//
// Over a segment of tokens the recurrence maps each row s of the state (1 x dk) as
// s <- s M + l, with M the ordered product of the per-token factors
// alpha_t (I - beta_t k_t k_t^T) and l the row the segment produces from a zero
// state (Nyysyyan, "Gated-DeltaNet": the WY identity for the product of the
// A_t = I - beta_t k_t k_t^T and the unrolled state S_i = gamma_i S_0 A_1..A_i +
// G_i).  Chaining the maps of consecutive segments is this fold; it is what a
// sequence-parallel forward needs between its segments.
//
// Rows of S are independent under s <- s M + l, so one CTA owns a block of rows of
// one state and keeps them in shared memory through every step of the fold.  Each
// step streams M_i through shared memory in slices of up to 32 rows (every thread
// loads a few float4 of the slice, coalesced), and each thread accumulates a
// 4-row x 4-column tile of the new rows; then the block's rows of L_i are added.
// fp32 CUDA cores: 2 dv dk^2 FLOPs per state and step.  (Measured design choice:
// streaming M from L2 per thread, or one tiled launch per step, ran 1.6x and 2.7x
// slower per step at dk = dv = 128.)
#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kFoldThreads = 256;

template <int DK>
__host__ __device__ constexpr int fold_rows() { return kFoldThreads / (DK / 4) * 4; }

// M is [count, units, DK, DK] and L [count, units, dv, DK]; `units` is their full
// state count (the step stride), u0 the first state of this launch.
template <int DK>
__global__ void __launch_bounds__(kFoldThreads)
gdn_state_fold_kernel(const float* __restrict__ S_in, const float* __restrict__ M,
                      const float* __restrict__ L, int count, float* __restrict__ S_out,
                      int units, int u0, int dv) {
  constexpr int LPC = DK / 4;              // threads per row (4 columns each)
  constexpr int RB = fold_rows<DK>();      // rows per CTA, 4 per thread
  constexpr int KS = DK < 32 ? DK : 32;    // rows of M per staged slice
  constexpr int SLICE4 = KS * DK / 4;      // float4 per slice
  __shared__ __align__(16) float Ss[RB][DK + 4];
  __shared__ __align__(16) float Ms[KS][DK];
  const int tid = threadIdx.x;
  const int u = u0 + blockIdx.y, rb0 = blockIdx.x * RB;
  const int cq = tid % LPC, r0 = (tid / LPC) * 4;  // columns 4cq .. 4cq+3, rows r0 .. r0+3
  const size_t so = (size_t)u * dv * DK;
  const size_t mstep = (size_t)units * DK * DK, lstep = (size_t)units * dv * DK;

#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = rb0 + r0 + r;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (S_in && row < dv)
      x = *reinterpret_cast<const float4*>(S_in + so + (size_t)row * DK + 4 * cq);
    *reinterpret_cast<float4*>(&Ss[r0 + r][4 * cq]) = x;
  }
  __syncthreads();
  for (int i = 0; i < count; ++i) {
    float4 acc[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (S_in || i > 0) {  // a zero state times M_i is zero: the first step is L_0 alone
      const float* Mi = M + i * mstep + (size_t)u * DK * DK;
      for (int k0 = 0; k0 < DK; k0 += KS) {
        for (int idx = tid; idx < SLICE4; idx += kFoldThreads) {
          const int row = idx / LPC, c = idx % LPC;
          *reinterpret_cast<float4*>(&Ms[row][4 * c]) =
              __ldg(reinterpret_cast<const float4*>(Mi + (size_t)(k0 + row) * DK + 4 * c));
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < KS; ++kk) {
          const float4 m = *reinterpret_cast<const float4*>(&Ms[kk][4 * cq]);
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const float x = Ss[r0 + r][k0 + kk];
            acc[r].x = fmaf(x, m.x, acc[r].x);
            acc[r].y = fmaf(x, m.y, acc[r].y);
            acc[r].z = fmaf(x, m.z, acc[r].z);
            acc[r].w = fmaf(x, m.w, acc[r].w);
          }
        }
        __syncthreads();  // the slice (and, after the last one, the old rows) are read
      }
    }
    const float* Li = L + i * lstep + so + 4 * cq;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int row = rb0 + r0 + r;
      if (row < dv) {
        const float4 l = __ldg(reinterpret_cast<const float4*>(Li + (size_t)row * DK));
        acc[r].x += l.x; acc[r].y += l.y; acc[r].z += l.z; acc[r].w += l.w;
      }
      // each thread rewrites only its own rows and columns, which no other thread
      // reads before the barrier below
      *reinterpret_cast<float4*>(&Ss[r0 + r][4 * cq]) = acc[r];
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = rb0 + r0 + r;
    if (row < dv)
      *reinterpret_cast<float4*>(S_out + so + (size_t)row * DK + 4 * cq) =
          *reinterpret_cast<const float4*>(&Ss[r0 + r][4 * cq]);
  }
}

template <int DK>
cudaError_t launch_fold_dk(const float* S_in, const float* M, const float* L, int count,
                           float* S_out, int units, int dv, cudaStream_t stream) {
  const int blocks = (dv + fold_rows<DK>() - 1) / fold_rows<DK>();
  for (int u0 = 0; u0 < units; u0 += 65535) {  // the grid's y limit
    const int n = units - u0 < 65535 ? units - u0 : 65535;
    gdn_state_fold_kernel<DK><<<dim3(blocks, n), kFoldThreads, 0, stream>>>(
        S_in, M, L, count, S_out, units, u0, dv);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// The linear mode's map over each sequence (Nyysyyan, "Mamba2": the state is the decayed
// sum of the writes, so M = (product of alpha_t) I): one block per (sequence, head) sums
// its log alpha (fp32, strided loads eight in flight), then writes the dk x dk M.
__global__ void __launch_bounds__(256)
gain_map_kernel(const float* __restrict__ log_alpha, float* __restrict__ M, int H, int T, int dk,
                const int32_t* __restrict__ cu_seqlens) {
  const int unit = blockIdx.x, n = unit / H, h = unit % H;
  long long a = (long long)n * T, b = a + T;
  if (cu_seqlens) {  // a packed member, clamped to the token range like the forward
    const long long lo = min(max((long long)cu_seqlens[n], 0LL), (long long)T);
    a = lo;
    b = min(max((long long)cu_seqlens[n + 1], lo), (long long)T);
  }
  __shared__ float red[8];
  float s = 0.f;
  if (log_alpha)
    for (long long t0 = a + threadIdx.x; t0 < b; t0 += 8 * 256) {
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const long long t = t0 + 256LL * e;
        v[e] = t < b ? log_alpha[t * H + h] : 0.f;
      }
      s += ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  const float g = expf(((red[0] + red[1]) + (red[2] + red[3])) + ((red[4] + red[5]) + (red[6] + red[7])));
  float* m = M + (size_t)unit * dk * dk;
  for (int i = threadIdx.x; i < dk * dk; i += 256) m[i] = (i / dk == i % dk) ? g : 0.f;
}

}  // namespace

cudaError_t launch_gain_map(const float* log_alpha, float* M, int units, int H, int T, int dk,
                            const int32_t* cu_seqlens, cudaStream_t stream) {
  if (units == 0) return cudaSuccess;
  gain_map_kernel<<<units, 256, 0, stream>>>(log_alpha, M, H, T, dk, cu_seqlens);
  return cudaGetLastError();
}

cudaError_t launch_state_fold(const float* S_in, const float* M, const float* L, int count,
                              float* S_out, int units, int dv, int dk, cudaStream_t stream) {
  if (units == 0) return cudaSuccess;
  switch (dk) {
    case 16: return launch_fold_dk<16>(S_in, M, L, count, S_out, units, dv, stream);
    case 32: return launch_fold_dk<32>(S_in, M, L, count, S_out, units, dv, stream);
    case 64: return launch_fold_dk<64>(S_in, M, L, count, S_out, units, dv, stream);
    case 128: return launch_fold_dk<128>(S_in, M, L, count, S_out, units, dv, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
