/*
 * gdn.h -- C ABI of the GB300 chunkwise Gated DeltaNet forward.
 *
 * The operation (qiita Nyysyyan, "Gated-DeltaNet" section, first equation block;
 * the same layer as kkkzoz "linear-attention", "Gated DeltaNet" section):
 *
 *     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = S_t q_t                          (read after token t is written)
 *
 * for every (sequence, head) pair independently, with S a dv x dk fp32 matrix
 * that starts at S0 and ends at S_final.  It is computed chunk by chunk
 * (Nyysyyan, "Chunk Computation"): inside a chunk of C tokens every token is
 * handled at once through the WY representation (myhz0606, "DeltaNet的Chunkwise
 * Form推导", section 4.5; Nyysyyan, "Gated-DeltaNet", W and U matrix forms);
 * chunks of one sequence run in order, each handing its final state to the next.
 *
 * All pointers except `cu_seqlens`'s host copy are DEVICE pointers owned by the
 * caller, contiguous, 16-byte aligned.  No call allocates, frees or
 * synchronises unless stated.  Every function returns a gdn_status; on a non-OK
 * status `gdn_last_error()` gives a message for the calling host thread.
 *
 * Current device: every call works on the calling thread's current CUDA device
 * (cudaSetDevice).  The device pointers and the stream passed to a call must belong
 * to that device: tensor maps, kernel attributes and the library's internal streams
 * are resolved on it, so a mismatch fails with a CUDA error (GDN_ELAUNCH or GDN_ECUDA).
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_EINVAL = 1,    /* bad size, NULL required pointer, misalignment: nothing launched */
  GDN_EDTYPE = 2,    /* unknown qkv dtype code: nothing launched */
  GDN_ELAUNCH = 3,   /* a kernel launch failed (message from the CUDA runtime) */
  GDN_ETIMEOUT = 4,  /* a kernel gave up a bounded wait (see gdn_check_status) */
  GDN_ECUDA = 5      /* another CUDA runtime error */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* Which kernel family a call with these sizes runs (for callers and tests). */
typedef enum {
  GDN_PATH_NONE = 0,      /* sizes not supported */
  GDN_PATH_SIMT = 1,      /* CUDA-core kernel, fp32 arithmetic, the per-token recurrence
                             (exact; C is not used): head sizes 16 and 32, dk != dv */
  GDN_PATH_TCGEN05 = 2,   /* bf16 tcgen05 tensor-core kernel: dk = dv = 128, C = 64 */
  GDN_PATH_TF32 = 3       /* the chunk form on tcgen05 tensor cores in three TF32 passes
                             (fp32 accuracy), as a sequence of batched per-chunk kernels:
                             dk = dv = 64 or 128, C = 16, 32 or 64, every shape and dtype
                             the bf16 kernel does not take; scratch from a stream-ordered
                             memory pool the library keeps per device.  The linear mode
                             runs here too, with erase 0 (T = I, W~ = 0) and U = V. */
} gdn_path;

/*
 * gdn_chunk_fwd -- chunkwise forward of the Gated DeltaNet recurrence.
 *
 * q, k       [B, T, H, dk]   qkv_dtype (fp32 or bf16), token-major, heads inner
 * v          [B, T, H, dv]   qkv_dtype
 * log_alpha  [B, T, H]       fp32, natural log of the gate alpha_t in (0, 1], so <= 0
 * beta       [B, T, H]       fp32, writing strength beta_t (normally in (0, 1))
 * S0         [N, H, dv, dk]  fp32 initial state per (sequence, head), or NULL = zeros
 * out        [B, T, H, dv]   qkv_dtype, written for every token (bf16 rounded to
 *                            nearest even from fp32)
 * S_final    [N, H, dv, dk]  fp32 final state per (sequence, head), or NULL = not written
 * B, H, T    batch, heads, tokens per sequence; with cu_seqlens, B must be 1 and T is
 *            the total packed token count
 * dk, dv     head sizes, each one of 16, 32, 64, 128
 * C          chunk length, one of 16, 32, 64; a sequence's last chunk may be shorter (the
 *            CUDA-core path computes the recurrence token by token, which the chunk form
 *            equals, and does not use it)
 * cu_seqlens int32 [N_seqs + 1] DEVICE array of packed sequence offsets
 *            (cu_seqlens[0] = 0, non-decreasing, cu_seqlens[N_seqs] = T), or NULL for
 *            N = B fixed-length sequences.  The state restarts at every offset.
 * N_seqs     number of packed sequences (ignored when cu_seqlens is NULL)
 * qkv_dtype  a gdn_dtype code
 * stream     cudaStream_t to launch on (NULL = legacy default stream)
 *
 * With T == 0 the token arrays may be NULL; S_final then receives S0 (or zeros).
 *
 * Asynchronous: GDN_OK means every launch was queued.  Values of log_alpha > 0
 * are not checked (exp of in-chunk gate sums could overflow).  The contents of
 * cu_seqlens are not read on the host: offsets out of [0, T] are clamped on the
 * device, so bad offsets give wrong results, never out-of-bounds accesses.
 * `out` and `S_final` must not overlap the inputs.
 */
int gdn_chunk_fwd(const void* q, const void* k, const void* v,
                  const float* log_alpha, const float* beta, const float* S0,
                  void* out, float* S_final,
                  int B, int H, int T, int dk, int dv, int C,
                  const int32_t* cu_seqlens, int N_seqs, int qkv_dtype,
                  void* stream);

/*
 * gdn_chunk_bwd -- gradients of gdn_chunk_fwd's recurrence: for a loss whose gradients
 * with respect to `out` and `S_final` are d_out and dS_final, compute the gradients of
 * q, k, v, log_alpha, beta and S0.
 *
 * The pages derive no backward pass; this is the reverse-mode derivative of the
 * recurrence (Nyysyyan, "Gated-DeltaNet", first equation block), walked backwards in
 * time with the state gradient G = dL/dS_t:
 *   G += dO_t q_t^T;  dq_t = S_t^T dO_t;  du = G k_t;  dv_t = beta_t du;
 *   dbeta_t = du . (v_t - a_t S_{t-1} k_t);
 *   dlog_alpha_t = a_t (<G, S_{t-1}> - beta_t du . S_{t-1} k_t);
 *   dk_t = G^T u_t - beta_t a_t S_{t-1}^T du   (u_t = beta_t (v_t - a_t S_{t-1} k_t));
 *   G <- a_t G (I - beta_t k_t k_t^T);   dS0 = G at the start
 * (a_t = exp(log_alpha_t)).  The kernels are those gdn_bwd_select_path names: for
 * dk = dv = 64 or 128 the chunked path (the same derivative in the chunk form, see
 * gdn_chunk_bwd_ex), otherwise the per-token path, which walks this recurrence with the
 * states recomputed from checkpoints every 8 tokens kept in `workspace`, in fp32 on the
 * CUDA cores.  Both are deterministic.
 *
 * q, k, v, log_alpha, beta, S0, B, H, T, dk, dv, cu_seqlens, N_seqs, qkv_dtype: as
 *            passed to gdn_chunk_fwd (S0 NULL = zeros)
 * d_out      [B, T, H, dv]   qkv_dtype, gradient of `out`
 * dS_final   [N, H, dv, dk]  fp32 gradient of S_final, or NULL = zeros
 * d_q, d_k   [B, T, H, dk]   qkv_dtype outputs (rounded to nearest even for bf16)
 * d_v        [B, T, H, dv]   qkv_dtype output
 * d_log_alpha, d_beta [B, T, H] fp32 outputs
 * d_S0       [N, H, dv, dk]  fp32 output, or NULL = not written
 * workspace  device scratch of at least gdn_chunk_bwd_workspace_bytes(...) bytes
 *            (may be NULL when that is 0); its contents need no initialisation
 *
 * Device pointers, caller-owned, 16-byte aligned; outputs must not overlap inputs.
 * Asynchronous; the path gdn_bwd_select_path names (2 kernel launches on the per-token
 * path, 28 on the chunked one).  Errors: GDN_EINVAL / GDN_EDTYPE before any launch
 * (including a missing or short workspace, with the size needed in the message),
 * GDN_ELAUNCH.  With packed sequences, token rows outside every sequence get
 * unspecified gradients.
 */
int gdn_chunk_bwd(const void* q, const void* k, const void* v,
                  const float* log_alpha, const float* beta, const float* S0,
                  const void* d_out, const float* dS_final,
                  void* d_q, void* d_k, void* d_v, float* d_log_alpha, float* d_beta,
                  float* d_S0, void* workspace, size_t workspace_bytes,
                  int B, int H, int T, int dk, int dv,
                  const int32_t* cu_seqlens, int N_seqs, int qkv_dtype, void* stream);

/* Workspace bytes gdn_chunk_bwd and gdn_chunk_bwd_ex (either path) need (N_seqs = number
 * of sequences: B, or the packed count); 0 for T == 0 or unsupported sizes. */
size_t gdn_chunk_bwd_workspace_bytes(int B, int H, int T, int dk, int dv, int N_seqs);

/* Backward kernel families. */
typedef enum {
  GDN_BWD_AUTO = 0,     /* the one gdn_bwd_select_path names */
  GDN_BWD_TOKENS = 1,   /* per-token recurrence over row blocks of the state, from
                           checkpoints every 8 tokens: every head size */
  GDN_BWD_CHUNKED = 2   /* the chunk form: per chunk of 64 tokens the derivative as dense
                           products, with the chunk-start states and the chunk-end state
                           gradients from two chains over the chunks; dk = dv = 64 or 128 */
} gdn_bwd_path;

/* The backward path gdn_chunk_bwd takes for these sizes (GDN_BWD_TOKENS or
 * GDN_BWD_CHUNKED), 0 if unsupported. */
int gdn_bwd_select_path(int dk, int dv, int qkv_dtype);

/*
 * gdn_chunk_bwd_ex -- gdn_chunk_bwd on a chosen path (gdn_bwd_path).  Both paths compute
 * the same derivative to fp32 accuracy and are deterministic: the per-token path in fp32
 * on the CUDA cores, the chunked path with its products on the tensor cores in three TF32
 * passes (a two-part TF32 split of each fp32 operand, hi*hi + hi*lo + lo*hi accumulated in
 * fp32, ~2^-22 relative error per product).  The chunked path is the derivative of the chunk form (Nyysyyan,
 * "Gated-DeltaNet", WY representation and chunkwise algorithm): per chunk, with T the
 * inverse of the chunk's unit lower-triangular WY matrix, W~ = T diag(beta e^g) K and
 * U = T diag(beta) V,
 *   d delta = P^T dO + E K dS'^T,   dS = dO^T diag(e^g) Q + e^{g_last} dS' - d delta^T W~,
 * and dQ, dK, dV, dbeta, dlog_alpha through P = lower(Q K^T o D), the state write and
 * the WY factors (dA = -T^T dT T^T for the triangular solve); T == 0 and unsupported head
 * sizes run the per-token path.  Errors as gdn_chunk_bwd, plus GDN_EINVAL for an unknown
 * path or GDN_BWD_CHUNKED with head sizes it does not support.
 */
int gdn_chunk_bwd_ex(const void* q, const void* k, const void* v,
                     const float* log_alpha, const float* beta, const float* S0,
                     const void* d_out, const float* dS_final,
                     void* d_q, void* d_k, void* d_v, float* d_log_alpha, float* d_beta,
                     float* d_S0, void* workspace, size_t workspace_bytes,
                     int B, int H, int T, int dk, int dv,
                     const int32_t* cu_seqlens, int N_seqs, int qkv_dtype, int bwd_path,
                     void* stream);

/*
 * gdn_chunk_bwd_noalloc -- gdn_chunk_bwd on the per-token path (GDN_BWD_TOKENS) for
 * callers that cannot allocate device memory: code running where cudaMalloc is not
 * allowed or not wanted (inside a caller's own memory pool, a plugin that receives only
 * its input and output buffers, a path that must not synchronise the device the way an
 * allocation can), or with no allocator at hand at all.  It takes no workspace; the
 * per-token backward's scratch (checkpoints and per-row partial sums) lives in one
 * fixed array of gdn_chunk_bwd_noalloc_max_scratch_bytes() bytes (64 MiB) inside the
 * library's device memory, which every device that loads the library holds until the
 * process exits.  The pages have no counterpart of this entry point: it is a packaging
 * of the same backward, with the same results as gdn_chunk_bwd_ex(..., GDN_BWD_TOKENS).
 *
 * Arguments as for gdn_chunk_bwd without `workspace` / `workspace_bytes`; the caller
 * still owns and passes every input and output.
 *
 * Sizes whose scratch (gdn_chunk_bwd_workspace_bytes for the per-token path) exceeds the
 * fixed array are rejected with GDN_EINVAL before any launch; at dk = dv = 128 that is
 * about 16 KB per token and head.  Nothing is allocated or freed: no cudaMalloc, cudaFree
 * or allocating library routine.  The first call on a device looks up the array's device
 * address with that device current (this may load the library's device code there), so
 * make that first call before any stream capture.  Every call shares the one array and
 * it keeps the last call's contents; the kernels write every scratch word they read, so
 * nothing needs clearing, but calls that overlap on the GPU (on different streams, or
 * from different host threads without ordering) race on it and must not run at once.
 */
size_t gdn_chunk_bwd_noalloc_max_scratch_bytes(void);
int gdn_chunk_bwd_noalloc(const void* q, const void* k, const void* v,
                          const float* log_alpha, const float* beta, const float* S0,
                          const void* d_out, const float* dS_final,
                          void* d_q, void* d_k, void* d_v, float* d_log_alpha, float* d_beta,
                          float* d_S0, int B, int H, int T, int dk, int dv,
                          const int32_t* cu_seqlens, int N_seqs, int qkv_dtype, void* stream);

/*
 * gdn_chunk_fwd_host -- gdn_chunk_fwd (or, with beta == NULL, gdn_linear_chunk_fwd) on
 * HOST buffers, end to end: copies the inputs in, runs the forward, copies the outputs
 * back, and returns once they are in host memory.  Fixed-length batches only.
 *
 * The batch is cut into at most `pieces` consecutive ranges of whole chunks (1..64),
 * each about half as long as the one before, so that little work follows the last input
 * copy.  Inputs go in on one internal copy stream, range r is computed on `stream` from range
 * r-1's fp32 final state (so the results equal the unsplit forward's bit for bit), and
 * outputs come back on a second internal copy stream; the copies of one range overlap
 * the computation of the next, and the two copy directions overlap each other.  Each
 * range of a [B, T, H, d] tensor moves as one strided 2-D copy.
 *
 * q, k, v, log_alpha, beta, S0, out, S_final: as for gdn_chunk_fwd, but HOST pointers
 *            (page-locked memory is needed for the copies to overlap); beta NULL selects
 *            the linear mode, where log_alpha may also be NULL (alpha = 1)
 * workspace  DEVICE scratch, 256-byte aligned, of at least
 *            gdn_chunk_fwd_host_workspace_bytes(B, H, T, dk, dv, C, qkv_dtype, pieces,
 *            beta == NULL) bytes (device copies of the inputs and outputs and three
 *            states); contents need no initialisation
 * stream     cudaStream_t the forward runs on (NULL = legacy default stream)
 *
 * Synchronous (returns with the outputs in host memory).  Errors: GDN_EINVAL /
 * GDN_EDTYPE before any copy or launch; GDN_ECUDA for a failed copy, launch or
 * synchronisation (message from the CUDA runtime).
 */
int gdn_chunk_fwd_host(const void* q, const void* k, const void* v,
                       const float* log_alpha, const float* beta, const float* S0,
                       void* out, float* S_final,
                       int B, int H, int T, int dk, int dv, int C, int qkv_dtype, int pieces,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Device workspace bytes gdn_chunk_fwd_host needs (linear: 1 when beta is NULL); 0 for
 * invalid sizes. */
size_t gdn_chunk_fwd_host_workspace_bytes(int B, int H, int T, int dk, int dv, int C,
                                          int qkv_dtype, int pieces, int linear);

/*
 * gdn_linear_chunk_fwd -- the same chunkwise forward in the linear mode: no delta-rule
 * erase, a plain write (Nyysyyan, "Mamba2" section, its recurrence and chunk form;
 * "Linear attention" section when alpha = 1):
 *
 *     S_t = alpha_t S_{t-1} + v_t k_t^T,   o_t = S_t q_t
 *
 * which is gdn_chunk_fwd's recurrence with the erase strength set to 0 and the
 * write strength to 1.  Arguments, layouts, ownership, paths and errors are those of
 * gdn_chunk_fwd, without beta; log_alpha may be NULL, meaning alpha_t = 1 (plain
 * linear attention).  On the tensor-core path (GDN_PATH_TCGEN05) this mode has a kernel
 * of its own: with no erase the pseudo-values are V itself, so one CTA per (sequence,
 * head) runs without the WY factors; the results equal gdn_chunk_fwd's pipeline run with
 * these factors, bit for bit, except where gdn_linear_split_segments splits the sequences
 * (few (sequence, head) units; see there), which changes the order of the sums.  On
 * GDN_PATH_TF32 it runs the same batched chunk-form kernels as gdn_chunk_fwd with the
 * erase gates 0 (so T = I and W~ = 0) and U = V.
 */
int gdn_linear_chunk_fwd(const void* q, const void* k, const void* v,
                         const float* log_alpha, const float* S0,
                         void* out, float* S_final,
                         int B, int H, int T, int dk, int dv, int C,
                         const int32_t* cu_seqlens, int N_seqs, int qkv_dtype,
                         void* stream);

/*
 * gdn_decode_step -- one token of the same recurrence for a batch of sequences,
 * the recurrent form (Nyysyyan, "Gated-DeltaNet" section, first equation block;
 * kkkzoz, "Gated DeltaNet" section: gate, predict, delta, write, then read):
 *
 *     S <- alpha S (I - beta k k^T) + beta v k^T,   o = S q
 *
 * computed as p = S k, u = beta (v - alpha p), S <- alpha S + u k^T and
 * o = alpha (S q) + u (k . q), with the state read once and written once.
 *
 * q, k       [N, H, dk]      qkv_dtype, the token of each (sequence, head)
 * v          [N, H, dv]      qkv_dtype
 * log_alpha  [N, H]          fp32, natural log of alpha in (0, 1], so <= 0
 * beta       [N, H]          fp32 writing strength
 * S          [N, H, dv, dk]  fp32 state per (sequence, head), updated IN PLACE (required)
 * out        [N, H, dv]      qkv_dtype, o for every (sequence, head)
 * N, H       sequences and heads (N * H >= 0; 0 launches nothing)
 * dk, dv     head sizes, each one of 16, 32, 64, 128
 * qkv_dtype  a gdn_dtype code
 * stream     cudaStream_t (NULL = legacy default stream)
 *
 * Asynchronous.  Arithmetic is fp32 (bf16 inputs are widened exactly); `out` is
 * rounded to nearest even for bf16.  `out` must not overlap the inputs or S.
 */
int gdn_decode_step(const void* q, const void* k, const void* v,
                    const float* log_alpha, const float* beta, float* S, void* out,
                    int N, int H, int dk, int dv, int qkv_dtype, void* stream);
/*
 * gdn_state_fold -- fold affine state maps: S <- S M_i + L_i for i = 0 .. count-1,
 * starting from S_in, for each of `units` (sequence, head) states.
 *
 * Over a segment of tokens the recurrence maps each row s of a state as s <- s M + l
 * (Nyysyyan, "Gated-DeltaNet": the WY identity for the product of the per-token
 * factors and the unrolled state S_i = gamma_i S_0 A_1..A_i + G_i), where
 *   M = the ordered product of alpha_t (I - beta_t k_t k_t^T) over the segment: the
 *       S_final of gdn_chunk_fwd run on the segment with v = 0 (dv = dk) and S0 = I;
 *   L = the S_final of gdn_chunk_fwd run on the segment from a zero state.
 * (In the linear mode M = (product of alpha_t) I, obtained the same way.)  Folding
 * the maps of segments 0 .. r-1 gives the state at the start of segment r: this is
 * the step between the segments of a sequence-parallel forward.
 *
 * S_in   [units, dv, dk] fp32, or NULL = zeros (then M_0 is not read)
 * M      [count, units, dk, dk] fp32 (may be NULL when count == 1 and S_in is NULL)
 * L      [count, units, dv, dk] fp32
 * S_out  [units, dv, dk] fp32; may be S_in itself or L itself (the same pointer),
 *        must not otherwise overlap S_in, M or L
 * count >= 1; dv, dk one of 16, 32, 64, 128; units >= 0 (0 launches nothing)
 *
 * Device pointers, 16-byte aligned, caller-owned; fp32 arithmetic; asynchronous on
 * `stream`.  Errors: GDN_EINVAL before any launch, GDN_ELAUNCH.
 */
int gdn_state_fold(const float* S_in, const float* M, const float* L, int count,
                   float* S_out, int units, int dv, int dk, void* stream);

/*
 * gdn_decode_step_host -- gdn_decode_step on HOST buffers, end to end and synchronous:
 * the batch is cut into at most `pieces` (1..64) slices of whole sequences; a slice's
 * inputs and state go in on one internal copy stream, its step runs on `stream`, and
 * its output and new state come back on a second copy stream while later slices still
 * come in (page-locked host memory is needed for the copies to overlap).
 *
 * q, k, v, log_alpha, beta, S, out: as for gdn_decode_step, but HOST pointers; S is
 *            updated in place
 * workspace  DEVICE scratch, 256-byte aligned, of at least
 *            gdn_decode_step_host_workspace_bytes(N, H, dk, dv, qkv_dtype) bytes
 *
 * Returns with out and S written.  Errors: GDN_EINVAL / GDN_EDTYPE before any copy or
 * launch; GDN_ECUDA for a failed copy, launch or synchronisation.
 */
int gdn_decode_step_host(const void* q, const void* k, const void* v,
                         const float* log_alpha, const float* beta, float* S, void* out,
                         int N, int H, int dk, int dv, int qkv_dtype, int pieces,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Device workspace bytes gdn_decode_step_host needs; 0 for invalid sizes. */
size_t gdn_decode_step_host_workspace_bytes(int N, int H, int dk, int dv, int qkv_dtype);

/* The path gdn_chunk_fwd takes for these sizes, GDN_PATH_NONE if unsupported. */
int gdn_select_path(int dk, int dv, int C, int qkv_dtype);

/* Kernels gdn_chunk_fwd launches per call for these sizes (0 if unsupported). */
int gdn_launches_per_call(int dk, int dv, int C, int qkv_dtype);

/*
 * Segments per sequence that gdn_linear_chunk_fwd cuts a fixed-length batch of N
 * sequences into on the tensor-core path (1: none; 0: invalid sizes).  When the N x H
 * (sequence, head) units fill at most half of the device's SMs, each sequence runs as R
 * whole-chunk segments on separate SMs (R <= 4, at least two chunks each, none empty),
 * and one more kernel folds the segments' end states into the start states and S_final
 * (the linear mode's segment map is S_end = Gamma S_start + L with a scalar Gamma) and
 * adds e^{G_t} S_start q_t to the later segments' outputs: 2 launches in place of 1.
 * Packed batches are not split.
 * Scratch comes from the library's stream-ordered memory pool.  Uses the current device.
 */
int gdn_linear_split_segments(int N, int H, int T, int dk, int dv, int C, int qkv_dtype);

/*
 * gdn_linear_state_correct -- the linear mode's start-state correction.  In the linear
 * mode (gdn_linear_chunk_fwd) the outputs and the end state of a run are affine in its
 * start state with a scalar gain (Nyysyyan, "Mamba2": the state is the decayed sum of the
 * writes):
 *
 *     o_t   = o_t(from zero) + e^{G_t} S_start q_t,   G_t = sum of log alpha over 0..t
 *     S_end = Gamma S_start + S_end(from zero),       Gamma = e^{G_{T-1}}
 *
 * Given out and S_end of a gdn_linear_chunk_fwd run of B fixed-length sequences from a
 * zero start state (S0 NULL), this call adds the contribution of S_start in place, so
 * that they become the run's results from S_start.  A sequence-parallel rank uses it to
 * finish its segment once the exchange has given it the start state.
 *   q [B, T, H, dk] bf16, log_alpha [B, T, H] fp32 or NULL (alpha = 1): as passed to the
 *   run; S_start [B, H, dv, dk] fp32; out [B, T, H, dv] bf16, read and written;
 *   S_end [B, H, dv, dk] fp32, read and written, or NULL (not updated).  T = 0 gives
 *   S_end += S_start.  Device pointers, 16-byte aligned, asynchronous on `stream`.
 * Only bf16 with dk = dv = 128 (gdn_linear_state_correct_supported), fixed-length
 * batches; anything else returns GDN_EINVAL before any launch.  The product with
 * S_start runs on the tensor cores with S_start as two bf16 terms; the sums are fp32; out
 * is rounded to bf16 once more.
 */
int gdn_linear_state_correct(const void* q, const float* log_alpha, const float* S_start,
                             void* out, float* S_end, int B, int H, int T, int dk, int dv,
                             int qkv_dtype, void* stream);
/* 1 when gdn_linear_state_correct takes these sizes and dtype, else 0. */
int gdn_linear_state_correct_supported(int dk, int dv, int qkv_dtype);

/*
 * gdn_linear_segment_map -- the linear mode's state map over each sequence: with no erase
 * the state is the decayed sum of the writes (Nyysyyan, "Mamba2"), so the M of
 * S_end = S_start M + L is (product of alpha_t) I.  Writes M[n][h] = e^{sum of log alpha
 * over sequence n} I for every sequence and head, the M that gdn_state_fold takes.
 *   log_alpha [B, T, H] fp32 or NULL (alpha = 1: M = I); M [N, H, dk, dk] fp32, written;
 *   cu_seqlens as for gdn_chunk_fwd (B = 1, N = N_seqs members, clamped to [0, T]) or
 *   NULL (N = B).  Device pointers, 16-byte aligned, asynchronous on `stream`; one
 *   launch.  Errors: GDN_EINVAL for bad sizes or pointers, before any launch.
 */
int gdn_linear_segment_map(const float* log_alpha, float* M, int B, int H, int T, int dk,
                           const int32_t* cu_seqlens, int N_seqs, void* stream);

/*
 * Synchronise `stream`, then read and clear the device status word that kernels
 * set when a bounded wait (mbarrier, async copy) gives up.  Returns GDN_OK or
 * GDN_ETIMEOUT (message names the wait), or GDN_ECUDA if the stream failed.
 */
int gdn_check_status(void* stream);

/*
 * Self-test of the failure detection: launch one CTA whose bounded wait (the same
 * wait routine and limit, 2 s, that the kernels use) waits on an mbarrier that
 * nothing arrives on.  The wait gives up, the kernel records it in the status word
 * and returns, so the next gdn_check_status(stream) returns GDN_ETIMEOUT; the context
 * stays usable.  Returns GDN_OK once launched, GDN_ELAUNCH otherwise.
 */
int gdn_selftest_wait_timeout(void* stream);

/* Message for the last non-OK status returned on this host thread. */
const char* gdn_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
