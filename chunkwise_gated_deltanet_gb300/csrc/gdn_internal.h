// Internal declarations shared by the host-side translation units of libgdn.
// Not part of the public ABI (that is include/gdn.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace gdn {

// Raise a kernel's dynamic shared-memory cap to `bytes`, once per device.  The
// attribute belongs to the function in the current context; it is not set per
// launch, because changing a kernel's attributes while launches of it are in
// flight on other streams can serialise them.  `done` holds one bit per device.  With
// `max_carveout` the kernel also asks for the largest shared-memory carveout, so that
// as many CTAs as its shared memory allows fit an SM.
template <typename Kernel>
cudaError_t ensure_smem_cap(Kernel* kernel, int bytes, std::atomic<unsigned long long>& done,
                            bool max_carveout = false) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && max_carveout)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Everything a forward launch needs, already validated by the API layer.
struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* log_alpha;
  const float* beta;
  const float* S0;        // may be null (zeros)
  void* out;
  float* S_final;         // may be null (not written)
  const int32_t* cu_seqlens;  // may be null (fixed-length sequences)
  int B, H, T, dk, dv, C;
  int N;                  // number of sequences (B, or N_seqs when packed)
  int bf16;               // 1: q/k/v/out are bf16, 0: fp32
};

// Per-token recurrence on CUDA cores, fp32 arithmetic, any supported shape (C unused).
cudaError_t launch_rec(const FwdArgs& a, cudaStream_t stream);

// The chunk form on the backward's tcgen05 kernels (three TF32 passes): dk = dv = 64 or
// 128, C = 16, 32 or 64, fp32 or bf16 q/k/v; scratch from a stream-ordered pool of the
// library's.
bool fwd_chunked_supported(int dk, int dv, int C);
int fwd_chunked_launches();
cudaError_t launch_fwd_chunked(const FwdArgs& a, cudaStream_t stream);

// tcgen05 kernel: bf16, dk = dv = 128, C = 64.
bool tc_supported(int dk, int dv, int C, int bf16);
cudaError_t launch_tc(const FwdArgs& a, cudaStream_t stream);
int tc_launches(const FwdArgs& a);
// Segments per sequence the linear mode's split runs with for these sizes (1: no split).
int linear_split_segments(long long N, int H, int T);
// The linear mode's start-state correction of whole fixed-length sequences (bf16,
// dk = dv = 128): out += e^{G_t} S_start q_t, S_end <- Gamma S_start + S_end.
bool linear_correct_supported(int dk, int dv, int bf16);
cudaError_t launch_linear_correct(const void* q, const float* log_alpha, const float* S_start,
                                  void* out, float* S_end, int B, int H, int T,
                                  cudaStream_t stream);
// Stream-ordered scratch from the library's per-device memory pool (cudaFreeAsync frees).
cudaError_t scratch_alloc(void** ptr, size_t bytes, cudaStream_t stream);
// Single-token decode step (recurrent form), already validated by the API layer.
struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* log_alpha;
  const float* beta;
  float* S;               // updated in place
  void* out;
  int N, H, dk, dv;
  int bf16;
};
// The forward on host buffers, pipelined over token ranges (fixed-length batches).
struct HostFwdArgs {
  const void* q;          // host [B, T, H, dk]
  const void* k;
  const void* v;          // host [B, T, H, dv]
  const float* log_alpha; // host [B, T, H] or null (alpha = 1, linear mode only)
  const float* beta;      // host [B, T, H] or null (the linear mode)
  const float* S0;        // host [B, H, dv, dk] or null
  void* out;              // host [B, T, H, dv]
  float* S_final;         // host [B, H, dv, dk] or null
  void* workspace;        // device, host_fwd_workspace_bytes(...)
  int B, H, T, dk, dv, C, pieces;
  int bf16;
  int tc;                 // 1: the tcgen05 kernel, 2: the chunk form on the TF32 kernels,
                          // 0: the SIMT kernel
};
size_t host_fwd_workspace_bytes(int B, int H, int T, int dk, int dv, int C, int esz, int pieces,
                                bool has_beta);
cudaError_t launch_host_fwd(const HostFwdArgs& a, cudaStream_t stream);

// The decode step on host buffers, pipelined over slices of sequences.
struct HostDecodeArgs {
  const void* q;          // host [N, H, dk]
  const void* k;
  const void* v;          // host [N, H, dv]
  const float* log_alpha; // host [N, H]
  const float* beta;      // host [N, H]
  float* S;               // host [N, H, dv, dk], updated in place
  void* out;              // host [N, H, dv]
  void* workspace;        // device, host_decode_workspace_bytes(...)
  int N, H, dk, dv, pieces;
  int bf16;
};
size_t host_decode_workspace_bytes(int N, int H, int dk, int dv, int esz);
cudaError_t launch_host_decode(const HostDecodeArgs& a, cudaStream_t stream);

// One CTA whose bounded wait can never be satisfied (failure-detection self-test).
cudaError_t launch_wait_selftest(cudaStream_t stream);

// Backward (gradients of q, k, v, log alpha, beta, S0), already validated.
struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* log_alpha;
  const float* beta;
  const float* S0;        // may be null (zeros)
  const void* dout;
  const float* dS_final;  // may be null (zeros)
  void* dq;
  void* dk_out;
  void* dv_out;
  float* dlog_alpha;
  float* dbeta;
  float* dS0;             // may be null (not written)
  void* workspace;        // bwd_workspace_bytes(...) bytes, 256-byte aligned
  const int32_t* cu_seqlens;
  int B, H, T, dk, dv, N;
  int bf16;
};
size_t bwd_workspace_bytes(long long rows, int H, int dk, int dv, int N);
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream);
// Size of the per-token backward's fixed scratch array (gdn_chunk_bwd_noalloc), and its
// device address on the current device (looked up once per device).
constexpr size_t kBwdNoAllocScratchBytes = size_t(64) << 20;
cudaError_t bwd_noalloc_scratch(void** ptr);
// The chunk-form backward (dk = dv = 64 or 128, rows > 0).
bool bwd_chunked_supported(int dk, int dv);
size_t bwd_chunked_workspace_bytes(long long rows, int H, int dk, int dv, int N);
cudaError_t launch_bwd_chunked(const BwdArgs& a, cudaStream_t stream);
// M[n][h] = e^{sum of log alpha over sequence n} I (dk x dk), already validated; packed
// members from cu_seqlens (T is then the packed token count).
cudaError_t launch_gain_map(const float* log_alpha, float* M, int units, int H, int T, int dk,
                            const int32_t* cu_seqlens, cudaStream_t stream);
// S <- S M_i + L_i for i < count per state (S_in NULL: zeros), already validated.
cudaError_t launch_state_fold(const float* S_in, const float* M, const float* L, int count,
                              float* S_out, int units, int dv, int dk, cudaStream_t stream);
// CTAs the decode step launches for these sizes (dk one of 16, 32, 64, 128).
long long decode_ctas(long long N, long long H, int dk, int dv);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

// Reads and clears the tcgen05 kernel's device status word (synchronous copy).
// Returns 0 if clear, else the code a bounded wait recorded.
int tc_read_and_clear_status(cudaStream_t stream, cudaError_t* err);
// Device address of that status word on the current device (looked up once per device),
// for other kernels' bounded waits to record their codes in.
cudaError_t tc_status_address(int** ptr);

}  // namespace gdn
