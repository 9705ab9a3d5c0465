// The forward on host buffers: copies in, the chunkwise forward, copies out, pipelined
// over consecutive token ranges.
//
// A fixed-length batch [B, T, H, d] is cut into `pieces` ranges of whole chunks, each
// about half as long as the one before.  Range r of every tensor is one strided block
// (B rows of L*H*d elements, pitch T*H*d), so it moves with a single cudaMemcpy2DAsync.  Inputs go in on one copy stream, ranges are
// computed in order on the caller's stream (range r starts from range r-1's fp32 final
// state, so the result is the unsplit forward's), outputs come back on a second copy
// stream; events order the three.  The copy of range r+1 and the write-back of range
// r-1 then overlap the computation of range r, and the two copy directions overlap
// each other.  Only the last range's computation and write-back follow the last input
// copy, hence the decreasing lengths: the input copies take about four times as long per
// chunk as the computation, so each range's computation still hides behind the next
// range's copy while the tail shrinks.  (A write-back that overlaps the input copies
// slows them by about half its own time, so the tail is the part worth shrinking.)
#include <cuda_runtime.h>

#include <mutex>

#include "gdn_internal.h"

namespace gdn {
namespace {

size_t al256(size_t x) { return (x + 255) / 256 * 256; }

struct HostLayout {
  int pieces;
  long long bound[65];  // range r is tokens [bound[r], bound[r + 1]), whole chunks
  size_t q, k, v, la, be, out, s0, st, total;  // byte offsets of the device buffers
};

// Weight of range r is kRangeRatio^r; boundaries are rounded to whole chunks with at
// least one chunk per range.
constexpr double kRangeRatio = 0.5;

HostLayout host_layout(int B, int H, int T, int dk, int dv, int C, int esz, int pieces,
                       bool has_beta) {
  HostLayout L;
  const long long nc = (T + C - 1) / C;
  int P = (int)(nc < pieces ? nc : pieces);
  if (P < 1) P = 1;
  double wsum = 0.0, w = 1.0;
  for (int r = 0; r < P; ++r, w *= kRangeRatio) wsum += w;
  L.bound[0] = 0;
  double acc = 0.0;
  long long prev = 0;
  w = 1.0;
  for (int r = 0; r < P; ++r, w *= kRangeRatio) {
    acc += w / wsum;
    long long c = (r == P - 1) ? nc : (long long)(acc * (double)nc + 0.5);
    if (c < prev + 1) c = prev + 1;
    if (c > nc - (P - 1 - r)) c = nc - (P - 1 - r);
    L.bound[r + 1] = c * C < T ? c * C : T;
    prev = c;
  }
  L.pieces = P;
  const size_t rows = (size_t)B * T * H;
  L.q = 0;
  L.k = L.q + al256(rows * dk * esz);
  L.v = L.k + al256(rows * dk * esz);
  L.la = L.v + al256(rows * dv * esz);
  L.be = L.la + al256(rows * 4);
  L.out = L.be + (has_beta ? al256(rows * 4) : 0);
  L.s0 = L.out + al256(rows * dv * esz);
  const size_t state = al256((size_t)B * H * dv * dk * 4);
  L.st = L.s0 + state;
  L.total = L.st + 2 * state;  // two final-state buffers, used in turn by the ranges
  return L;
}

// Two copy streams per device, made once.
struct CopyStreams {
  cudaStream_t in = nullptr, out = nullptr;
};
CopyStreams g_streams[64];
std::mutex g_streams_mu;

cudaError_t copy_streams(CopyStreams* cs) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_streams_mu);
  CopyStreams& s = g_streams[dev & 63];
  if (!s.in) {
    e = cudaStreamCreateWithFlags(&s.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&s.out, cudaStreamNonBlocking);
    if (e != cudaSuccess) return e;
  }
  *cs = s;
  return cudaSuccess;
}

// block of tokens [a, a + len) of a [B, T, H, width] host tensor <-> the contiguous
// [B, len, H, width] device block
cudaError_t copy_range(void* dst, const void* src, bool to_device, int B, int T, int H,
                       long long a, long long len, int width, int esz, cudaStream_t s) {
  const size_t row = (size_t)len * H * width * esz;       // one sequence's part
  const size_t pitch = (size_t)T * H * width * esz;        // one sequence on the host
  const size_t off = (size_t)a * H * width * esz;
  if (row == 0) return cudaSuccess;
  if (to_device)
    return cudaMemcpy2DAsync(dst, row, static_cast<const char*>(src) + off, pitch, row, B,
                             cudaMemcpyHostToDevice, s);
  return cudaMemcpy2DAsync(static_cast<char*>(dst) + off, pitch, src, row, row, B,
                           cudaMemcpyDeviceToHost, s);
}

}  // namespace

size_t host_fwd_workspace_bytes(int B, int H, int T, int dk, int dv, int C, int esz, int pieces,
                                bool has_beta) {
  return host_layout(B, H, T, dk, dv, C, esz, pieces, has_beta).total;
}

cudaError_t launch_host_fwd(const HostFwdArgs& a, cudaStream_t stream) {
  const int esz = a.bf16 ? 2 : 4;
  const bool linear = a.beta == nullptr;
  const HostLayout L = host_layout(a.B, a.H, a.T, a.dk, a.dv, a.C, esz, a.pieces, !linear);
  char* ws = static_cast<char*>(a.workspace);
  CopyStreams cs;
  cudaError_t e = copy_streams(&cs);
  if (e != cudaSuccess) return e;
  const size_t state_bytes = (size_t)a.B * a.H * a.dv * a.dk * 4;
  const int n = L.pieces;
  cudaEvent_t ev[3 * 64];
  const int n_ev = 2 * n + 1;
  if (n > 64) return cudaErrorInvalidValue;
  for (int i = 0; i < n_ev; ++i) {
    e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
    if (e != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
      return e;
    }
  }
  cudaEvent_t* loaded = ev;          // range r is on the device
  cudaEvent_t* computed = ev + n;    // range r's outputs are ready
  cudaEvent_t start = ev[2 * n];     // the caller's earlier work is ordered first
  e = cudaEventRecord(start, stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.in, start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.out, start, 0);
  float* s0_dev = a.S0 ? reinterpret_cast<float*>(ws + L.s0) : nullptr;
  if (e == cudaSuccess && a.S0)
    e = cudaMemcpyAsync(s0_dev, a.S0, state_bytes, cudaMemcpyHostToDevice, cs.in);
  // every input range goes in first, in order, so the copy engine never waits
  for (int r = 0; r < n && e == cudaSuccess; ++r) {
    const long long t0 = L.bound[r], len = L.bound[r + 1] - t0;
    const size_t tok = (size_t)a.B * t0 * a.H;  // token-heads before this range
    e = copy_range(ws + L.q + tok * a.dk * esz, a.q, true, a.B, a.T, a.H, t0, len, a.dk, esz, cs.in);
    if (e == cudaSuccess)
      e = copy_range(ws + L.k + tok * a.dk * esz, a.k, true, a.B, a.T, a.H, t0, len, a.dk, esz, cs.in);
    if (e == cudaSuccess)
      e = copy_range(ws + L.v + tok * a.dv * esz, a.v, true, a.B, a.T, a.H, t0, len, a.dv, esz, cs.in);
    if (e == cudaSuccess && a.log_alpha)
      e = copy_range(ws + L.la + tok * 4, a.log_alpha, true, a.B, a.T, a.H, t0, len, 1, 4, cs.in);
    if (e == cudaSuccess && !linear)
      e = copy_range(ws + L.be + tok * 4, a.beta, true, a.B, a.T, a.H, t0, len, 1, 4, cs.in);
    if (e == cudaSuccess) e = cudaEventRecord(loaded[r], cs.in);
  }
  // ranges in order on the caller's stream, each from the previous final state
  const float* prev = s0_dev;
  for (int r = 0; r < n && e == cudaSuccess; ++r) {
    const long long t0 = L.bound[r], len = L.bound[r + 1] - t0;
    const size_t tok = (size_t)a.B * t0 * a.H;
    float* st = reinterpret_cast<float*>(ws + L.st + (size_t)(r & 1) * al256(state_bytes));
    e = cudaStreamWaitEvent(stream, loaded[r], 0);
    if (e != cudaSuccess) break;
    FwdArgs f{};
    f.q = ws + L.q + tok * a.dk * esz;
    f.k = ws + L.k + tok * a.dk * esz;
    f.v = ws + L.v + tok * a.dv * esz;
    f.log_alpha = a.log_alpha ? reinterpret_cast<const float*>(ws + L.la + tok * 4) : nullptr;
    f.beta = linear ? nullptr : reinterpret_cast<const float*>(ws + L.be + tok * 4);
    f.S0 = prev;
    f.out = ws + L.out + tok * a.dv * esz;
    f.S_final = st;
    f.cu_seqlens = nullptr;
    f.B = a.B; f.H = a.H; f.T = (int)len; f.dk = a.dk; f.dv = a.dv; f.C = a.C; f.N = a.B;
    f.bf16 = a.bf16;
    e = a.tc == 1 ? launch_tc(f, stream)
                  : (a.tc == 2 ? launch_fwd_chunked(f, stream) : launch_rec(f, stream));
    if (e == cudaSuccess) e = cudaEventRecord(computed[r], stream);
    prev = st;
    if (e != cudaSuccess) break;
    // range r's outputs come back while range r + 1 is computed
    e = cudaStreamWaitEvent(cs.out, computed[r], 0);
    if (e == cudaSuccess)
      e = copy_range(a.out, ws + L.out + tok * a.dv * esz, false, a.B, a.T, a.H, t0, len, a.dv,
                     esz, cs.out);
  }
  if (e == cudaSuccess && a.S_final)
    e = cudaMemcpyAsync(a.S_final, prev ? prev : s0_dev, state_bytes, cudaMemcpyDeviceToHost,
                        cs.out);
  // the call returns with the outputs in host memory
  cudaError_t e2 = cudaStreamSynchronize(cs.out);
  if (e == cudaSuccess) e = e2;
  e2 = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = e2;
  e2 = cudaStreamSynchronize(cs.in);
  if (e == cudaSuccess) e = e2;
  for (int i = 0; i < n_ev; ++i) cudaEventDestroy(ev[i]);
  return e;
}


// ---- the decode step on host buffers: slices of sequences, pipelined ----
// Sequences are independent, so a slice of n sequences of every tensor (q, k, v,
// gates, the state, the output) is one contiguous block: slice r goes in on one copy
// stream, its step runs on the caller's stream, its state and output come back on the
// other copy stream while later slices are still coming in.

namespace {

struct DecodeLayout {
  size_t q, k, v, la, be, s, out, total;
};

DecodeLayout decode_layout(int N, int H, int dk, int dv, int esz) {
  const size_t nh = (size_t)N * H;
  DecodeLayout L;
  L.q = 0;
  L.k = L.q + al256(nh * dk * esz);
  L.v = L.k + al256(nh * dk * esz);
  L.la = L.v + al256(nh * dv * esz);
  L.be = L.la + al256(nh * 4);
  L.s = L.be + al256(nh * 4);
  L.out = L.s + al256(nh * dv * dk * 4);
  L.total = L.out + al256(nh * dv * esz);
  return L;
}

}  // namespace

size_t host_decode_workspace_bytes(int N, int H, int dk, int dv, int esz) {
  return decode_layout(N, H, dk, dv, esz).total;
}

cudaError_t launch_host_decode(const HostDecodeArgs& a, cudaStream_t stream) {
  const int esz = a.bf16 ? 2 : 4;
  const DecodeLayout L = decode_layout(a.N, a.H, a.dk, a.dv, esz);
  char* ws = static_cast<char*>(a.workspace);
  if (a.pieces < 1 || a.pieces > 64) return cudaErrorInvalidValue;
  const int per = (a.N + a.pieces - 1) / a.pieces;
  const int n = per > 0 ? (a.N + per - 1) / per : 0;
  if (n == 0) return cudaSuccess;
  CopyStreams cs;
  cudaError_t e = copy_streams(&cs);
  if (e != cudaSuccess) return e;
  cudaEvent_t ev[2 * 64 + 1];
  const int n_ev = 2 * n + 1;
  for (int i = 0; i < n_ev; ++i) {
    e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
    if (e != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
      return e;
    }
  }
  cudaEvent_t* loaded = ev;
  cudaEvent_t* computed = ev + n;
  e = cudaEventRecord(ev[2 * n], stream);  // the caller's earlier work comes first
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.in, ev[2 * n], 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.out, ev[2 * n], 0);
  const size_t H = (size_t)a.H;
  // byte offset of sequence n0 in a [N, H, width] array of `bytes`-sized elements
  auto at = [&](int n0, size_t width, size_t bytes) { return (size_t)n0 * H * width * bytes; };
  const char* src_q = static_cast<const char*>(a.q);
  const char* src_k = static_cast<const char*>(a.k);
  const char* src_v = static_cast<const char*>(a.v);
  const char* src_la = reinterpret_cast<const char*>(a.log_alpha);
  const char* src_be = reinterpret_cast<const char*>(a.beta);
  char* host_s = reinterpret_cast<char*>(a.S);
  char* host_o = static_cast<char*>(a.out);
  const size_t sw = (size_t)a.dv * a.dk;  // state elements per (sequence, head)
  for (int r = 0; r < n && e == cudaSuccess; ++r) {
    const int n0 = r * per, nn = (n0 + per < a.N ? per : a.N - n0);
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice;
    e = cudaMemcpyAsync(ws + L.q + at(n0, a.dk, esz), src_q + at(n0, a.dk, esz),
                        at(nn, a.dk, esz), h2d, cs.in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ws + L.k + at(n0, a.dk, esz), src_k + at(n0, a.dk, esz),
                          at(nn, a.dk, esz), h2d, cs.in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ws + L.v + at(n0, a.dv, esz), src_v + at(n0, a.dv, esz),
                          at(nn, a.dv, esz), h2d, cs.in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ws + L.la + at(n0, 1, 4), src_la + at(n0, 1, 4), at(nn, 1, 4), h2d,
                          cs.in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ws + L.be + at(n0, 1, 4), src_be + at(n0, 1, 4), at(nn, 1, 4), h2d,
                          cs.in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ws + L.s + at(n0, sw, 4), host_s + at(n0, sw, 4), at(nn, sw, 4), h2d,
                          cs.in);
    if (e == cudaSuccess) e = cudaEventRecord(loaded[r], cs.in);
  }
  for (int r = 0; r < n && e == cudaSuccess; ++r) {
    const int n0 = r * per, nn = (n0 + per < a.N ? per : a.N - n0);
    e = cudaStreamWaitEvent(stream, loaded[r], 0);
    if (e != cudaSuccess) break;
    DecodeArgs d;
    d.q = ws + L.q + at(n0, a.dk, esz);
    d.k = ws + L.k + at(n0, a.dk, esz);
    d.v = ws + L.v + at(n0, a.dv, esz);
    d.log_alpha = reinterpret_cast<const float*>(ws + L.la + at(n0, 1, 4));
    d.beta = reinterpret_cast<const float*>(ws + L.be + at(n0, 1, 4));
    d.S = reinterpret_cast<float*>(ws + L.s + at(n0, sw, 4));
    d.out = ws + L.out + at(n0, a.dv, esz);
    d.N = nn; d.H = a.H; d.dk = a.dk; d.dv = a.dv; d.bf16 = a.bf16;
    e = launch_decode(d, stream);
    if (e == cudaSuccess) e = cudaEventRecord(computed[r], stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.out, computed[r], 0);
    const cudaMemcpyKind d2h = cudaMemcpyDeviceToHost;
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(host_o + at(n0, a.dv, esz), ws + L.out + at(n0, a.dv, esz),
                          at(nn, a.dv, esz), d2h, cs.out);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(host_s + at(n0, sw, 4), ws + L.s + at(n0, sw, 4), at(nn, sw, 4), d2h,
                          cs.out);
  }
  cudaError_t e2 = cudaStreamSynchronize(cs.out);
  if (e == cudaSuccess) e = e2;
  e2 = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = e2;
  e2 = cudaStreamSynchronize(cs.in);
  if (e == cudaSuccess) e = e2;
  for (int i = 0; i < n_ev; ++i) cudaEventDestroy(ev[i]);
  return e;
}

}  // namespace gdn
