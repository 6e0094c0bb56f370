// host_pipeline.cu -- gdr_prefill_host: the prefill on arrays in host memory, pipelined over
// pieces of the packed token axis so that the host<->device copies of one piece overlap the
// kernels of its neighbours.
//
// The packed token range [0, T) is cut into pieces of about `piece_tokens` tokens.  A cut inside
// a sequence falls on a chunk boundary of that sequence (a multiple of 64 tokens from its start),
// so each sequence is split into the same chunks as in one gdr_prefill call.  Piece i runs as an
// ordinary prefill over the sequences it touches, clipped to the piece; the states of all
// sequences live in one device array and are handed over in place (S0 = S_final) from piece to
// piece, so a sequence that continues into the next piece resumes from the state the previous
// piece left.
//
// Three streams: the inputs of piece i go to staging buffer i % 2 on an internal copy-in stream,
// the prefill runs on the caller's stream, and its outputs go back on an internal copy-out
// stream.  Events order the three; staging buffer i % 2 is refilled for piece i + 2 only after
// piece i's prefill (inputs) and copy-out (outputs) are done.  The caller's stream waits for the
// last copy, so the call behaves like any other call enqueued on it.
#include <algorithm>
#include <mutex>
#include <vector>

#include "gdr_internal.cuh"

namespace gdr {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kRing = 4;  // events per kind in flight (reuse distance 2 pieces)
constexpr int64_t kChunkTokens = 64;  // the chunk length of the tensor-core prefill

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Offsets of the regions of the caller's device buffer.
struct HostPlan {
  int64_t piece;        // target tokens per piece (multiple of 64)
  int64_t cap;          // staging capacity in tokens (a piece may run up to 63 tokens long)
  size_t states, cu, pcu[2], ws, ws_bytes, in[2], out[2], total;
  size_t q_tok, v_tok, a_tok, b_tok, in_bytes;  // bytes per token (all heads) of each input
  size_t o_tok;                                  // bytes per token of the output
};

bool make_plan(const gdr_shape& sh, int64_t piece_tokens, HostPlan* p) {
  if (sh.n_seqs < 1 || sh.H < 1 || sh.d_k < 1 || sh.d_v < 1 || sh.total_tokens < 0) return false;
  const size_t e = sh.dtype == GDR_BF16 ? 2 : 4;
  const int64_t T = sh.total_tokens;
  int64_t P = piece_tokens > 0 ? piece_tokens : std::max<int64_t>(4096, (T + 7) / 8);
  P = (std::max<int64_t>(P, 64) + 63) / 64 * 64;
  p->piece = P;
  p->cap = std::min<int64_t>(P + 64, std::max<int64_t>(T, 1));
  p->q_tok = (size_t)sh.H * sh.d_k * e;
  p->v_tok = (size_t)sh.H * sh.d_v * e;
  p->a_tok = (size_t)sh.H * (sh.gate == GDR_GATE_CHANNEL ? sh.d_k : 1) * 4;
  p->b_tok = (size_t)sh.H * 4;
  p->o_tok = p->v_tok;
  const size_t cap = (size_t)p->cap;
  p->in_bytes = 2 * up256(cap * p->q_tok) + up256(cap * p->v_tok) + up256(cap * p->a_tok) +
                up256(cap * p->b_tok);
  // a piece touches at most n_seqs sequences: its workspace is that of n_seqs sequences, with
  // the work-queue rings of the largest piece that can still use them
  gdr_shape ring_shape = sh;
  ring_shape.n_seqs = (int)std::min<long>((long)sh.n_seqs, WorkspaceLayout::kRingMaxPairs / sh.H);
  const size_t ring = ring_shape.n_seqs >= 1 ? WorkspaceLayout::ring_bytes(ring_shape) : 0;
  size_t off = 0;
  p->states = off;
  off += up256((size_t)sh.n_seqs * sh.H * sh.d_k * sh.d_v * 4);
  p->cu = off;
  off += up256((size_t)(sh.n_seqs + 1) * 4);
  for (int b = 0; b < 2; ++b) {
    p->pcu[b] = off;
    off += up256((size_t)(sh.n_seqs + 1) * 4);
  }
  p->ws = off;
  p->ws_bytes = WorkspaceLayout::total(sh.n_seqs) + ring;
  off += up256(p->ws_bytes);
  for (int b = 0; b < 2; ++b) {
    p->in[b] = off;
    off += p->in_bytes;
    p->out[b] = off;
    off += up256(cap * p->o_tok);
  }
  p->total = off;
  return true;
}

__global__ void piece_offsets_kernel(const int32_t* __restrict__ cu, int s_lo, int n, int32_t a,
                                     int32_t len, int32_t* __restrict__ pcu) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i <= n; i += gridDim.x * blockDim.x) {
    const int32_t v = cu[s_lo + i] - a;
    pcu[i] = v < 0 ? 0 : (v > len ? len : v);
  }
}

// The internal streams and events of one device (created on first use, kept for the process).
struct DeviceRes {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, in_done = nullptr, last = nullptr, end = nullptr;
  cudaEvent_t h2d[kRing], comp[kRing], d2h[kRing];
};
std::mutex g_mutex[kMaxDevices];
DeviceRes g_res[kMaxDevices];

cudaError_t init_res(DeviceRes& r) {
  if (r.ready) return cudaSuccess;
  cudaError_t e = cudaStreamCreateWithFlags(&r.in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&r.out, cudaStreamNonBlocking);
  cudaEvent_t* evs[] = {&r.start, &r.in_done, &r.last, &r.end};
  for (cudaEvent_t* ev : evs)
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  for (int i = 0; i < kRing && e == cudaSuccess; ++i) {
    e = cudaEventCreateWithFlags(&r.h2d[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r.comp[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r.d2h[i], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) r.ready = true;
  return e;
}

// Piece boundaries of [0, T): about `P` tokens each, a cut inside a sequence moved forward to
// that sequence's next chunk boundary (or its end).
std::vector<int64_t> piece_cuts(const std::vector<int64_t>& cu, int64_t T, int64_t P) {
  std::vector<int64_t> cuts{0};
  int64_t pos = 0;
  while (pos < T) {
    int64_t b = std::min(T, pos + P);
    if (b < T) {
      const int s = (int)(std::upper_bound(cu.begin(), cu.end(), b) - cu.begin()) - 1;
      const int64_t aligned = cu[s] + (b - cu[s] + kChunkTokens - 1) / kChunkTokens * kChunkTokens;
      b = std::min(aligned, cu[s + 1]);
    }
    cuts.push_back(b);
    pos = b;
  }
  return cuts;
}

}  // namespace
}  // namespace gdr

extern "C" size_t gdr_prefill_host_buffer_size(const gdr_shape* shape, int64_t piece_tokens) {
  gdr::HostPlan p;
  if (!shape || !gdr::make_plan(*shape, piece_tokens, &p)) return 0;
  return p.total;
}

extern "C" gdr_status gdr_prefill_host(const gdr_shape* shape, const void* q, const void* k,
                                       const void* v, const float* alpha, const float* beta,
                                       const float* S0, const int32_t* cu_seqlens, void* out,
                                       float* S_final, int64_t piece_tokens, void* buffer,
                                       size_t buffer_bytes, void* stream) {
  using namespace gdr;
  gdr_status st = validate_shape(shape, true);
  if (st != GDR_OK) return st;
  const gdr_shape sh = *shape;
  const int64_t T = sh.total_tokens;
  if (T > INT32_MAX) return GDR_ERR_UNSUPPORTED;
  if (T > 0 && (!q || !k || !v || !alpha || !beta || !out)) return GDR_ERR_INVALID_ARG;
  if (!cu_seqlens && sh.n_seqs != 1) return GDR_ERR_INVALID_ARG;
  // the offsets must tile [0, T) exactly: cu[0] = 0, non-decreasing, cu[n] = T
  std::vector<int64_t> cu(sh.n_seqs + 1);
  std::vector<int32_t> cu32(sh.n_seqs + 1);
  for (int i = 0; i <= sh.n_seqs; ++i) {
    cu32[i] = cu_seqlens ? cu_seqlens[i] : (i == 0 ? 0 : (int32_t)T);
    cu[i] = cu32[i];
    if (i > 0 && cu[i] < cu[i - 1]) return GDR_ERR_INVALID_ARG;
  }
  if (cu[0] != 0 || cu[sh.n_seqs] != T) return GDR_ERR_INVALID_ARG;
  HostPlan p;
  if (!make_plan(sh, piece_tokens, &p)) return GDR_ERR_INVALID_ARG;
  if (!buffer || ((uintptr_t)buffer & 255u) || buffer_bytes < p.total) return GDR_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDR_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex[dev]);
  DeviceRes& r = g_res[dev];
  if (init_res(r) != cudaSuccess) return GDR_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  unsigned char* base = static_cast<unsigned char*>(buffer);
  float* d_states = reinterpret_cast<float*>(base + p.states);
  int32_t* d_cu = reinterpret_cast<int32_t*>(base + p.cu);
  const size_t state_elems = (size_t)sh.H * sh.d_k * sh.d_v;
  const size_t states_bytes = (size_t)sh.n_seqs * state_elems * 4;
  const unsigned char* src[5] = {static_cast<const unsigned char*>(q),
                                 static_cast<const unsigned char*>(k),
                                 static_cast<const unsigned char*>(v),
                                 reinterpret_cast<const unsigned char*>(alpha),
                                 reinterpret_cast<const unsigned char*>(beta)};
  const size_t tok[5] = {p.q_tok, p.q_tok, p.v_tok, p.a_tok, p.b_tok};
  cudaError_t e = cudaSuccess;
  auto ok = [&](cudaError_t x) {
    if (e == cudaSuccess) e = x;
    return e == cudaSuccess;
  };
  // work already on the caller's stream comes first
  ok(cudaEventRecord(r.start, s));
  ok(cudaStreamWaitEvent(r.in, r.start, 0));
  ok(cudaStreamWaitEvent(r.out, r.start, 0));
  ok(cudaMemcpyAsync(d_cu, cu32.data(), cu32.size() * 4, cudaMemcpyHostToDevice, r.in));
  if (S0) {
    ok(cudaMemcpyAsync(d_states, S0, states_bytes, cudaMemcpyHostToDevice, r.in));
  } else {
    ok(cudaMemsetAsync(d_states, 0, states_bytes, r.in));
  }
  const std::vector<int64_t> cuts = piece_cuts(cu, T, p.piece);
  const int npieces = (int)cuts.size() - 1;
  gdr_status launch_st = GDR_OK;  // the first failed piece launch, if any
  for (int i = 0; i < npieces && e == cudaSuccess; ++i) {
    const int b = i & 1;
    const int64_t a0 = cuts[i], a1 = cuts[i + 1], len = a1 - a0;
    const int s_lo = (int)(std::upper_bound(cu.begin(), cu.end(), a0) - cu.begin()) - 1;
    const int s_hi = (int)(std::lower_bound(cu.begin() + 1, cu.end(), a1) - (cu.begin() + 1));
    const int n = s_hi - s_lo + 1;
    // inputs of piece i (staging b is free once piece i - 2's prefill is done)
    if (i >= 2) ok(cudaStreamWaitEvent(r.in, r.comp[(i - 2) % kRing], 0));
    int32_t* d_pcu = reinterpret_cast<int32_t*>(base + p.pcu[b]);
    piece_offsets_kernel<<<(n + 1 + 255) / 256, 256, 0, r.in>>>(d_cu, s_lo, n, (int32_t)a0,
                                                                  (int32_t)len, d_pcu);
    ok(cudaGetLastError());
    unsigned char* dst[5];
    size_t off = p.in[b];
    for (int j = 0; j < 5; ++j) {
      dst[j] = base + off;
      off += up256((size_t)p.cap * tok[j]);
      ok(cudaMemcpyAsync(dst[j], src[j] + (size_t)a0 * tok[j], (size_t)len * tok[j],
                         cudaMemcpyHostToDevice, r.in));
    }
    ok(cudaEventRecord(r.h2d[i % kRing], r.in));
    // the prefill of piece i on the caller's stream (output staging b is free once piece
    // i - 2's copy-out is done)
    ok(cudaStreamWaitEvent(s, r.h2d[i % kRing], 0));
    if (i >= 2) ok(cudaStreamWaitEvent(s, r.d2h[(i - 2) % kRing], 0));
    if (e != cudaSuccess) break;
    gdr_shape ps = sh;
    ps.n_seqs = n;
    ps.total_tokens = len;
    float* st_p = d_states + (size_t)s_lo * state_elems;
    st = prefill_launch(&ps, dst[0], dst[1], dst[2], reinterpret_cast<const float*>(dst[3]),
                        reinterpret_cast<const float*>(dst[4]), st_p, d_pcu, base + p.out[b],
                        st_p, base + p.ws, p.ws_bytes, s);
    if (st != GDR_OK) {
      launch_st = st;
      break;
    }
    ok(cudaEventRecord(r.comp[i % kRing], s));
    // outputs of piece i back to the host
    ok(cudaStreamWaitEvent(r.out, r.comp[i % kRing], 0));
    ok(cudaMemcpyAsync(static_cast<unsigned char*>(out) + (size_t)a0 * p.o_tok, base + p.out[b],
                       (size_t)len * p.o_tok, cudaMemcpyDeviceToHost, r.out));
    ok(cudaEventRecord(r.d2h[i % kRing], r.out));
  }
  // The final states once every piece (and the copy-in of the entering states) is done.  This
  // join also runs after a failed piece: copies of earlier pieces into the caller's host arrays
  // may still be queued on the internal streams, and the caller's stream must not pass the
  // call before they have finished.  (The `ok` calls still execute after an error; they only
  // stop recording it.)
  ok(cudaEventRecord(r.in_done, r.in));
  ok(cudaEventRecord(r.last, s));
  ok(cudaStreamWaitEvent(r.out, r.in_done, 0));
  ok(cudaStreamWaitEvent(r.out, r.last, 0));
  if (S_final && launch_st == GDR_OK)
    ok(cudaMemcpyAsync(S_final, d_states, states_bytes, cudaMemcpyDeviceToHost, r.out));
  ok(cudaEventRecord(r.end, r.out));
  ok(cudaStreamWaitEvent(s, r.end, 0));
  if (launch_st != GDR_OK) return launch_st;
  return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}
