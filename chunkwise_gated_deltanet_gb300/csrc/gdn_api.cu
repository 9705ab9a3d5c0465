// C ABI of libgdn: argument checks, kernel selection, error reporting.
// The operation and the meaning of every argument are documented in include/gdn.h.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

bool head_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool chunk_ok(int c) { return c == 16 || c == 32 || c == 64; }
bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" {

int gdn_version(void) { return 1 * 10000 + 0 * 100 + 0; }

const char* gdn_last_error(void) { return g_err; }

int gdn_select_path(int dk, int dv, int C, int qkv_dtype) {
  if (!head_ok(dk) || !head_ok(dv) || !chunk_ok(C)) return GDN_PATH_NONE;
  if (qkv_dtype != GDN_F32 && qkv_dtype != GDN_BF16) return GDN_PATH_NONE;
  if (gdn::tc_supported(dk, dv, C, qkv_dtype == GDN_BF16)) return GDN_PATH_TCGEN05;
  if (gdn::fwd_chunked_supported(dk, dv, C)) return GDN_PATH_TF32;
  return GDN_PATH_SIMT;
}

int gdn_linear_split_segments(int N, int H, int T, int dk, int dv, int C, int qkv_dtype) {
  if (N <= 0 || H <= 0 || T < 0) return 0;
  if (gdn_select_path(dk, dv, C, qkv_dtype) != GDN_PATH_TCGEN05) return 1;
  return gdn::linear_split_segments(N, H, T);
}

int gdn_launches_per_call(int dk, int dv, int C, int qkv_dtype) {
  gdn::FwdArgs a{};
  a.dk = dk; a.dv = dv; a.C = C; a.bf16 = qkv_dtype == GDN_BF16;
  switch (gdn_select_path(dk, dv, C, qkv_dtype)) {
    case GDN_PATH_TCGEN05: return gdn::tc_launches(a);
    case GDN_PATH_TF32: return gdn::fwd_chunked_launches();
    case GDN_PATH_SIMT: return 1;  // the recurrence kernel
    default: return 0;
  }
}

}  // extern "C"

namespace {

// The checks and launch shared by gdn_chunk_fwd and gdn_linear_chunk_fwd.  With
// linear set, beta is NULL (erase 0, write 1) and log_alpha may be NULL (alpha = 1).
int chunk_fwd_impl(const char* fn, bool linear, const void* q, const void* k, const void* v,
                   const float* log_alpha, const float* beta, const float* S0, void* out,
                   float* S_final, int B, int H, int T, int dk, int dv, int C,
                   const int32_t* cu_seqlens, int N_seqs, int qkv_dtype, void* stream) {
  if (qkv_dtype != GDN_F32 && qkv_dtype != GDN_BF16)
    return fail(GDN_EDTYPE, "%s: qkv_dtype %d is neither GDN_F32 nor GDN_BF16", fn, qkv_dtype);
  if (T > 0 && (!q || !k || !v || !out))
    return fail(GDN_EINVAL, "%s: q, k, v and out must be non-NULL", fn);
  if (T > 0 && !linear && (!log_alpha || !beta))
    return fail(GDN_EINVAL, "%s: log_alpha and beta must be non-NULL", fn);
  if (B <= 0 || H <= 0 || T < 0)
    return fail(GDN_EINVAL, "%s: need B > 0, H > 0, T >= 0 (got B=%d H=%d T=%d)", fn, B, H, T);
  if (!head_ok(dk) || !head_ok(dv))
    return fail(GDN_EINVAL, "%s: dk and dv must be 16, 32, 64 or 128 (got %d, %d)", fn, dk, dv);
  if (!chunk_ok(C)) return fail(GDN_EINVAL, "%s: C must be 16, 32 or 64 (got %d)", fn, C);
  int N = B;
  if (cu_seqlens) {
    if (B != 1) return fail(GDN_EINVAL, "%s: packed sequences need B == 1 (got %d)", fn, B);
    if (N_seqs <= 0)
      return fail(GDN_EINVAL, "%s: N_seqs must be > 0 with cu_seqlens (got %d)", fn, N_seqs);
    N = N_seqs;
  }
  const void* ptrs[] = {q, k, v, log_alpha, beta, S0, out, S_final, cu_seqlens};
  const char* names[] = {"q", "k", "v", "log_alpha", "beta", "S0", "out", "S_final",
                         "cu_seqlens"};
  for (int i = 0; i < 9; ++i)
    if (ptrs[i] && !aligned16(ptrs[i]))
      return fail(GDN_EINVAL, "%s: %s is not 16-byte aligned", fn, names[i]);
  const long long rows = (long long)B * T;
  if (rows * H * (dk > dv ? dk : dv) > (1LL << 40))
    return fail(GDN_EINVAL, "%s: problem too large", fn);

  gdn::FwdArgs a;
  a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = linear ? nullptr : beta;
  a.S0 = S0; a.out = out; a.S_final = S_final; a.cu_seqlens = cu_seqlens;
  a.B = B; a.H = H; a.T = T; a.dk = dk; a.dv = dv; a.C = C; a.N = N;
  a.bf16 = qkv_dtype == GDN_BF16;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  const int path = gdn_select_path(dk, dv, C, qkv_dtype);
  if (path == GDN_PATH_TCGEN05)
    e = gdn::launch_tc(a, s);
  else if (path == GDN_PATH_TF32)
    e = gdn::launch_fwd_chunked(a, s);
  else
    e = gdn::launch_rec(a, s);
  if (e != cudaSuccess)
    return fail(GDN_ELAUNCH, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return GDN_OK;
}

}  // namespace

extern "C" {

int gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* log_alpha,
                  const float* beta, const float* S0, void* out, float* S_final, int B, int H,
                  int T, int dk, int dv, int C, const int32_t* cu_seqlens, int N_seqs,
                  int qkv_dtype, void* stream) {
  return chunk_fwd_impl("gdn_chunk_fwd", false, q, k, v, log_alpha, beta, S0, out, S_final, B,
                        H, T, dk, dv, C, cu_seqlens, N_seqs, qkv_dtype, stream);
}

int gdn_linear_chunk_fwd(const void* q, const void* k, const void* v, const float* log_alpha,
                         const float* S0, void* out, float* S_final, int B, int H, int T, int dk,
                         int dv, int C, const int32_t* cu_seqlens, int N_seqs, int qkv_dtype,
                         void* stream) {
  return chunk_fwd_impl("gdn_linear_chunk_fwd", true, q, k, v, log_alpha, nullptr, S0, out,
                        S_final, B, H, T, dk, dv, C, cu_seqlens, N_seqs, qkv_dtype, stream);
}

int gdn_linear_state_correct_supported(int dk, int dv, int qkv_dtype) {
  return gdn::linear_correct_supported(dk, dv, qkv_dtype == GDN_BF16) ? 1 : 0;
}

int gdn_linear_state_correct(const void* q, const float* log_alpha, const float* S_start,
                             void* out, float* S_end, int B, int H, int T, int dk, int dv,
                             int qkv_dtype, void* stream) {
  const char* fn = "gdn_linear_state_correct";
  if (qkv_dtype != GDN_F32 && qkv_dtype != GDN_BF16)
    return fail(GDN_EDTYPE, "%s: qkv_dtype must be GDN_F32 or GDN_BF16", fn);
  if (!gdn::linear_correct_supported(dk, dv, qkv_dtype == GDN_BF16))
    return fail(GDN_EINVAL, "%s: needs bf16 with dk = dv = 128 (got dk %d, dv %d)", fn, dk, dv);
  if (B <= 0 || H <= 0 || T < 0)
    return fail(GDN_EINVAL, "%s: need B, H > 0 and T >= 0", fn);
  if (!S_start || (T > 0 && (!q || !out)))
    return fail(GDN_EINVAL, "%s: S_start (and q, out when T > 0) must be non-NULL", fn);
  if ((long long)B * T > 0x7fffffffLL)
    return fail(GDN_EINVAL, "%s: problem too large", fn);
  const void* ptrs[] = {q, log_alpha, S_start, out, S_end};
  const char* names[] = {"q", "log_alpha", "S_start", "out", "S_end"};
  for (int i = 0; i < 5; ++i)
    if (ptrs[i] && !aligned16(ptrs[i]))
      return fail(GDN_EINVAL, "%s: %s is not 16-byte aligned", fn, names[i]);
  const cudaError_t e = gdn::launch_linear_correct(q, log_alpha, S_start, out, S_end, B, H, T,
                                                   (cudaStream_t)stream);
  if (e != cudaSuccess)
    return fail(GDN_ELAUNCH, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return GDN_OK;
}

int gdn_decode_step(const void* q, const void* k, const void* v, const float* log_alpha,
                    const float* beta, float* S, void* out, int N, int H, int dk, int dv,
                    int qkv_dtype, void* stream) {
  if (qkv_dtype != GDN_F32 && qkv_dtype != GDN_BF16)
    return fail(GDN_EDTYPE, "gdn_decode_step: qkv_dtype %d is neither GDN_F32 nor GDN_BF16",
                qkv_dtype);
  if (N < 0 || H < 0)
    return fail(GDN_EINVAL, "gdn_decode_step: need N >= 0, H >= 0 (got N=%d H=%d)", N, H);
  if (!head_ok(dk) || !head_ok(dv))
    return fail(GDN_EINVAL, "gdn_decode_step: dk and dv must be 16, 32, 64 or 128 (got %d, %d)",
                dk, dv);
  if ((long long)N * H == 0) return GDN_OK;
  if (!q || !k || !v || !log_alpha || !beta || !S || !out)
    return fail(GDN_EINVAL, "gdn_decode_step: q, k, v, log_alpha, beta, S and out must be non-NULL");
  const void* ptrs[] = {q, k, v, log_alpha, beta, S, out};
  const char* names[] = {"q", "k", "v", "log_alpha", "beta", "S", "out"};
  for (int i = 0; i < 7; ++i)
    if (!aligned16(ptrs[i]))
      return fail(GDN_EINVAL, "gdn_decode_step: %s is not 16-byte aligned", names[i]);
  if (gdn::decode_ctas(N, H, dk, dv) > 0x7fffffffLL)
    return fail(GDN_EINVAL, "gdn_decode_step: problem too large");
  gdn::DecodeArgs a;
  a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.S = S; a.out = out;
  a.N = N; a.H = H; a.dk = dk; a.dv = dv; a.bf16 = qkv_dtype == GDN_BF16;
  const cudaError_t e = gdn::launch_decode(a, (cudaStream_t)stream);
  if (e != cudaSuccess)
    return fail(GDN_ELAUNCH, "gdn_decode_step: launch failed: %s", cudaGetErrorString(e));
  return GDN_OK;
}

size_t gdn_chunk_bwd_workspace_bytes(int B, int H, int T, int dk, int dv, int N_seqs) {
  if (B <= 0 || H <= 0 || T <= 0 || N_seqs <= 0 || !head_ok(dk) || !head_ok(dv)) return 0;
  const size_t a = gdn::bwd_workspace_bytes((long long)B * T, H, dk, dv, N_seqs);
  const size_t b = gdn::bwd_chunked_workspace_bytes((long long)B * T, H, dk, dv, N_seqs);
  return a > b ? a : b;
}

int gdn_bwd_select_path(int dk, int dv, int qkv_dtype) {
  if (!head_ok(dk) || !head_ok(dv)) return 0;
  if (qkv_dtype != GDN_F32 && qkv_dtype != GDN_BF16) return 0;
  return gdn::bwd_chunked_supported(dk, dv) ? GDN_BWD_CHUNKED : GDN_BWD_TOKENS;
}

int gdn_chunk_bwd(const void* q, const void* k, const void* v, const float* log_alpha,
                  const float* beta, const float* S0, const void* d_out, const float* dS_final,
                  void* d_q, void* d_k, void* d_v, float* d_log_alpha, float* d_beta,
                  float* d_S0, void* workspace, size_t workspace_bytes, int B, int H, int T,
                  int dk, int dv, const int32_t* cu_seqlens, int N_seqs, int qkv_dtype,
                  void* stream) {
  return gdn_chunk_bwd_ex(q, k, v, log_alpha, beta, S0, d_out, dS_final, d_q, d_k, d_v,
                          d_log_alpha, d_beta, d_S0, workspace, workspace_bytes, B, H, T, dk,
                          dv, cu_seqlens, N_seqs, qkv_dtype, GDN_BWD_AUTO, stream);
}

int gdn_chunk_bwd_ex(const void* q, const void* k, const void* v, const float* log_alpha,
                     const float* beta, const float* S0, const void* d_out,
                     const float* dS_final, void* d_q, void* d_k, void* d_v,
                     float* d_log_alpha, float* d_beta, float* d_S0, void* workspace,
                     size_t workspace_bytes, int B, int H, int T, int dk, int dv,
                     const int32_t* cu_seqlens, int N_seqs, int qkv_dtype, int bwd_path,
                     void* stream) {
  const char* fn = "gdn_chunk_bwd";
  if (bwd_path != GDN_BWD_AUTO && bwd_path != GDN_BWD_TOKENS && bwd_path != GDN_BWD_CHUNKED)
    return fail(GDN_EINVAL, "%s: unknown backward path %d", fn, bwd_path);
  if (bwd_path == GDN_BWD_CHUNKED && !gdn::bwd_chunked_supported(dk, dv))
    return fail(GDN_EINVAL, "%s: the chunked path needs dk = dv = 64 or 128 (got %d, %d)", fn,
                dk, dv);
  if (qkv_dtype != GDN_F32 && qkv_dtype != GDN_BF16)
    return fail(GDN_EDTYPE, "%s: qkv_dtype %d is neither GDN_F32 nor GDN_BF16", fn, qkv_dtype);
  if (T > 0 && (!q || !k || !v || !log_alpha || !beta || !d_out || !d_q || !d_k || !d_v ||
                !d_log_alpha || !d_beta))
    return fail(GDN_EINVAL, "%s: the inputs, d_out and the gradient outputs must be non-NULL",
                fn);
  if (B <= 0 || H <= 0 || T < 0)
    return fail(GDN_EINVAL, "%s: need B > 0, H > 0, T >= 0 (got B=%d H=%d T=%d)", fn, B, H, T);
  if (!head_ok(dk) || !head_ok(dv))
    return fail(GDN_EINVAL, "%s: dk and dv must be 16, 32, 64 or 128 (got %d, %d)", fn, dk, dv);
  int N = B;
  if (cu_seqlens) {
    if (B != 1) return fail(GDN_EINVAL, "%s: packed sequences need B == 1 (got %d)", fn, B);
    if (N_seqs <= 0)
      return fail(GDN_EINVAL, "%s: N_seqs must be > 0 with cu_seqlens (got %d)", fn, N_seqs);
    N = N_seqs;
  }
  const void* ptrs[] = {q, k, v, log_alpha, beta, S0, d_out, dS_final, d_q, d_k, d_v,
                        d_log_alpha, d_beta, d_S0, workspace, cu_seqlens};
  const char* names[] = {"q", "k", "v", "log_alpha", "beta", "S0", "d_out", "dS_final", "d_q",
                         "d_k", "d_v", "d_log_alpha", "d_beta", "d_S0", "workspace",
                         "cu_seqlens"};
  for (int i = 0; i < 16; ++i)
    if (ptrs[i] && !aligned16(ptrs[i]))
      return fail(GDN_EINVAL, "%s: %s is not 16-byte aligned", fn, names[i]);
  const long long rows = (long long)B * T;
  if (rows * H * (dk > dv ? dk : dv) > (1LL << 40))
    return fail(GDN_EINVAL, "%s: problem too large", fn);
  if (bwd_path == GDN_BWD_AUTO) bwd_path = gdn_bwd_select_path(dk, dv, qkv_dtype);
  const bool chunked = bwd_path == GDN_BWD_CHUNKED && rows > 0;
  const size_t need = chunked ? gdn::bwd_chunked_workspace_bytes(rows, H, dk, dv, N)
                              : gdn::bwd_workspace_bytes(rows, H, dk, dv, N);
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(GDN_EINVAL, "%s: workspace of %zu bytes needed (got %zu%s)", fn, need,
                workspace_bytes, workspace ? "" : ", NULL");
  gdn::BwdArgs a;
  a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.S0 = S0;
  a.dout = d_out; a.dS_final = dS_final;
  a.dq = d_q; a.dk_out = d_k; a.dv_out = d_v; a.dlog_alpha = d_log_alpha; a.dbeta = d_beta;
  a.dS0 = d_S0; a.workspace = workspace; a.cu_seqlens = cu_seqlens;
  a.B = B; a.H = H; a.T = T; a.dk = dk; a.dv = dv; a.N = N; a.bf16 = qkv_dtype == GDN_BF16;
  const cudaError_t e = chunked ? gdn::launch_bwd_chunked(a, (cudaStream_t)stream)
                                : gdn::launch_bwd(a, (cudaStream_t)stream);
  if (e != cudaSuccess)
    return fail(GDN_ELAUNCH, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return GDN_OK;
}

size_t gdn_chunk_bwd_noalloc_max_scratch_bytes(void) { return gdn::kBwdNoAllocScratchBytes; }

int gdn_chunk_bwd_noalloc(const void* q, const void* k, const void* v, const float* log_alpha,
                          const float* beta, const float* S0, const void* d_out,
                          const float* dS_final, void* d_q, void* d_k, void* d_v,
                          float* d_log_alpha, float* d_beta, float* d_S0, int B, int H, int T,
                          int dk, int dv, const int32_t* cu_seqlens, int N_seqs, int qkv_dtype,
                          void* stream) {
  const char* fn = "gdn_chunk_bwd_noalloc";
  // The per-token path with the library's fixed scratch array as its workspace: the
  // size it needs is checked against the array first, then gdn_chunk_bwd_ex validates
  // everything else and launches exactly as for a caller-supplied workspace.
  void* scratch = nullptr;
  if (B > 0 && H > 0 && T > 0 && head_ok(dk) && head_ok(dv) && (!cu_seqlens || N_seqs > 0)) {
    const int N = cu_seqlens ? N_seqs : B;
    const size_t need = gdn::bwd_workspace_bytes((long long)B * T, H, dk, dv, N);
    if (need > gdn::kBwdNoAllocScratchBytes)
      return fail(GDN_EINVAL, "%s: these sizes need %zu bytes of scratch, more than the "
                  "library's fixed %zu-byte array; use gdn_chunk_bwd with a workspace", fn,
                  need, (size_t)gdn::kBwdNoAllocScratchBytes);
    const cudaError_t e = gdn::bwd_noalloc_scratch(&scratch);
    if (e != cudaSuccess)
      return fail(GDN_ECUDA, "%s: looking up the scratch array failed: %s", fn,
                  cudaGetErrorString(e));
  }
  return gdn_chunk_bwd_ex(q, k, v, log_alpha, beta, S0, d_out, dS_final, d_q, d_k, d_v,
                          d_log_alpha, d_beta, d_S0, scratch,
                          scratch ? gdn::kBwdNoAllocScratchBytes : 0, B, H, T, dk, dv,
                          cu_seqlens, N_seqs, qkv_dtype, GDN_BWD_TOKENS, stream);
}

int gdn_linear_segment_map(const float* log_alpha, float* M, int B, int H, int T, int dk,
                           const int32_t* cu_seqlens, int N_seqs, void* stream) {
  const char* fn = "gdn_linear_segment_map";
  if (B <= 0 || H <= 0 || T < 0 || !head_ok(dk))
    return fail(GDN_EINVAL, "%s: need B, H > 0, T >= 0 and dk in {16, 32, 64, 128}", fn);
  if (cu_seqlens && (B != 1 || N_seqs <= 0))
    return fail(GDN_EINVAL, "%s: a packed batch needs B = 1 and N_seqs > 0", fn);
  if (!M) return fail(GDN_EINVAL, "%s: M must be non-NULL", fn);
  if ((log_alpha && !aligned16(log_alpha)) || !aligned16(M))
    return fail(GDN_EINVAL, "%s: log_alpha and M must be 16-byte aligned", fn);
  const long long units = (long long)(cu_seqlens ? N_seqs : B) * H;
  if (units > 0x7fffffffLL || (long long)B * T > 0x7fffffffLL)
    return fail(GDN_EINVAL, "%s: problem too large", fn);
  const cudaError_t e = gdn::launch_gain_map(log_alpha, M, (int)units, H, T, dk,
                                             cu_seqlens, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(GDN_ELAUNCH, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return GDN_OK;
}

int gdn_state_fold(const float* S_in, const float* M, const float* L, int count, float* S_out,
                   int units, int dv, int dk, void* stream) {
  if (units < 0 || count < 1)
    return fail(GDN_EINVAL, "gdn_state_fold: need units >= 0 and count >= 1 (got %d, %d)", units,
                count);
  if (!head_ok(dk) || !head_ok(dv))
    return fail(GDN_EINVAL, "gdn_state_fold: dk and dv must be 16, 32, 64 or 128 (got %d, %d)",
                dk, dv);
  if (units == 0) return GDN_OK;
  const bool needs_m = S_in || count > 1;
  if ((needs_m && !M) || !L || !S_out)
    return fail(GDN_EINVAL, "gdn_state_fold: L and S_out (and M when it is read) must be "
                "non-NULL");
  const void* ptrs[] = {S_in, M, L, S_out};
  const char* names[] = {"S_in", "M", "L", "S_out"};
  for (int i = 0; i < 4; ++i)
    if (ptrs[i] && !aligned16(ptrs[i]))
      return fail(GDN_EINVAL, "gdn_state_fold: %s is not 16-byte aligned", names[i]);
  const size_t sbytes = (size_t)units * dv * dk * sizeof(float);
  const size_t mbytes = (size_t)count * units * dk * dk * sizeof(float);
  const size_t lbytes = (size_t)count * sbytes;
  auto overlap = [](const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return a && b && x < y + nb && y < x + na;
  };
  if (needs_m && overlap(S_out, sbytes, M, mbytes))
    return fail(GDN_EINVAL, "gdn_state_fold: S_out overlaps M");
  if ((S_out != S_in && overlap(S_out, sbytes, S_in, sbytes)) ||
      (S_out != L && overlap(S_out, sbytes, L, lbytes)))
    return fail(GDN_EINVAL, "gdn_state_fold: S_out overlaps S_in or L without being either");
  const cudaError_t e = gdn::launch_state_fold(S_in, M, L, count, S_out, units, dv, dk,
                                               (cudaStream_t)stream);
  if (e != cudaSuccess)
    return fail(GDN_ELAUNCH, "gdn_state_fold: launch failed: %s", cudaGetErrorString(e));
  return GDN_OK;
}

size_t gdn_chunk_fwd_host_workspace_bytes(int B, int H, int T, int dk, int dv, int C,
                                          int qkv_dtype, int pieces, int linear) {
  if (B <= 0 || H <= 0 || T < 0 || !head_ok(dk) || !head_ok(dv) || !chunk_ok(C) ||
      pieces < 1 || pieces > 64 || (qkv_dtype != GDN_F32 && qkv_dtype != GDN_BF16))
    return 0;
  return gdn::host_fwd_workspace_bytes(B, H, T, dk, dv, C, qkv_dtype == GDN_BF16 ? 2 : 4,
                                       pieces, !linear);
}

int gdn_chunk_fwd_host(const void* q, const void* k, const void* v, const float* log_alpha,
                       const float* beta, const float* S0, void* out, float* S_final, int B,
                       int H, int T, int dk, int dv, int C, int qkv_dtype, int pieces,
                       void* workspace, size_t workspace_bytes, void* stream) {
  const char* fn = "gdn_chunk_fwd_host";
  if (qkv_dtype != GDN_F32 && qkv_dtype != GDN_BF16)
    return fail(GDN_EDTYPE, "%s: qkv_dtype %d is neither GDN_F32 nor GDN_BF16", fn, qkv_dtype);
  if (B <= 0 || H <= 0 || T < 0)
    return fail(GDN_EINVAL, "%s: need B > 0, H > 0, T >= 0 (got B=%d H=%d T=%d)", fn, B, H, T);
  if (!head_ok(dk) || !head_ok(dv))
    return fail(GDN_EINVAL, "%s: dk and dv must be 16, 32, 64 or 128 (got %d, %d)", fn, dk, dv);
  if (!chunk_ok(C)) return fail(GDN_EINVAL, "%s: C must be 16, 32 or 64 (got %d)", fn, C);
  if (pieces < 1 || pieces > 64)
    return fail(GDN_EINVAL, "%s: pieces must be in [1, 64] (got %d)", fn, pieces);
  const bool linear = beta == nullptr;
  if (T > 0 && (!q || !k || !v || !out || (!linear && !log_alpha)))
    return fail(GDN_EINVAL, "%s: q, k, v, out (and log_alpha with beta) must be non-NULL", fn);
  if ((long long)B * T * H * (dk > dv ? dk : dv) > (1LL << 40))
    return fail(GDN_EINVAL, "%s: problem too large", fn);
  const size_t need = gdn::host_fwd_workspace_bytes(B, H, T, dk, dv, C,
                                                    qkv_dtype == GDN_BF16 ? 2 : 4, pieces,
                                                    !linear);
  if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u))
    return fail(GDN_EINVAL, "%s: a 256-byte aligned device workspace of %zu bytes is needed "
                "(got %zu)", fn, need, workspace_bytes);
  gdn::HostFwdArgs a;
  a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.S0 = S0;
  a.out = out; a.S_final = S_final; a.workspace = workspace;
  a.B = B; a.H = H; a.T = T; a.dk = dk; a.dv = dv; a.C = C; a.pieces = pieces;
  a.bf16 = qkv_dtype == GDN_BF16;
  const int path = gdn_select_path(dk, dv, C, qkv_dtype);
  a.tc = path == GDN_PATH_TCGEN05 ? 1 : (path == GDN_PATH_TF32 ? 2 : 0);
  const cudaError_t e = gdn::launch_host_fwd(a, (cudaStream_t)stream);
  if (e != cudaSuccess)
    return fail(GDN_ECUDA, "%s: %s", fn, cudaGetErrorString(e));
  return GDN_OK;
}

size_t gdn_decode_step_host_workspace_bytes(int N, int H, int dk, int dv, int qkv_dtype) {
  if (N < 0 || H < 0 || !head_ok(dk) || !head_ok(dv) ||
      (qkv_dtype != GDN_F32 && qkv_dtype != GDN_BF16))
    return 0;
  return gdn::host_decode_workspace_bytes(N, H, dk, dv, qkv_dtype == GDN_BF16 ? 2 : 4);
}

int gdn_decode_step_host(const void* q, const void* k, const void* v, const float* log_alpha,
                         const float* beta, float* S, void* out, int N, int H, int dk, int dv,
                         int qkv_dtype, int pieces, void* workspace, size_t workspace_bytes,
                         void* stream) {
  const char* fn = "gdn_decode_step_host";
  if (qkv_dtype != GDN_F32 && qkv_dtype != GDN_BF16)
    return fail(GDN_EDTYPE, "%s: qkv_dtype %d is neither GDN_F32 nor GDN_BF16", fn, qkv_dtype);
  if (N < 0 || H < 0)
    return fail(GDN_EINVAL, "%s: need N >= 0, H >= 0 (got N=%d H=%d)", fn, N, H);
  if (!head_ok(dk) || !head_ok(dv))
    return fail(GDN_EINVAL, "%s: dk and dv must be 16, 32, 64 or 128 (got %d, %d)", fn, dk, dv);
  if (pieces < 1 || pieces > 64)
    return fail(GDN_EINVAL, "%s: pieces must be in [1, 64] (got %d)", fn, pieces);
  if ((long long)N * H == 0) return GDN_OK;
  if (!q || !k || !v || !log_alpha || !beta || !S || !out)
    return fail(GDN_EINVAL, "%s: q, k, v, log_alpha, beta, S and out must be non-NULL", fn);
  if (gdn::decode_ctas(N, H, dk, dv) > 0x7fffffffLL)
    return fail(GDN_EINVAL, "%s: problem too large", fn);
  const size_t need = gdn::host_decode_workspace_bytes(N, H, dk, dv, qkv_dtype == GDN_BF16 ? 2 : 4);
  if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u))
    return fail(GDN_EINVAL, "%s: a 256-byte aligned device workspace of %zu bytes is needed "
                "(got %zu)", fn, need, workspace_bytes);
  gdn::HostDecodeArgs a;
  a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.S = S; a.out = out;
  a.workspace = workspace; a.N = N; a.H = H; a.dk = dk; a.dv = dv; a.pieces = pieces;
  a.bf16 = qkv_dtype == GDN_BF16;
  const cudaError_t e = gdn::launch_host_decode(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(GDN_ECUDA, "%s: %s", fn, cudaGetErrorString(e));
  return GDN_OK;
}

int gdn_selftest_wait_timeout(void* stream) {
  const cudaError_t e = gdn::launch_wait_selftest((cudaStream_t)stream);
  if (e != cudaSuccess)
    return fail(GDN_ELAUNCH, "gdn_selftest_wait_timeout: launch failed: %s", cudaGetErrorString(e));
  return GDN_OK;
}

int gdn_check_status(void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess)
    return fail(GDN_ECUDA, "gdn_check_status: stream failed: %s", cudaGetErrorString(e));
  int code = gdn::tc_read_and_clear_status(s, &e);
  if (e != cudaSuccess)
    return fail(GDN_ECUDA, "gdn_check_status: reading the status word failed: %s",
                cudaGetErrorString(e));
  if (code != 0)
    return fail(GDN_ETIMEOUT,
                "gdn_check_status: a tcgen05 kernel gave up a bounded wait (code 0x%x)", code);
  return GDN_OK;
}

}  // extern "C"
