// decode.cu -- one-token decode step of the gated delta rule, fused in one pass over the state.
//
// Per (sequence, head), from engineermaxxing "From GPT-2 to Kimi K3: one memory, seven eviction
// policies" §06b (decay per row of S, read, correct) and dev.to "From GPT-2 to Kimi K3: How
// Language Models Learned to Manage Memory" §4-§5 (fade, then read the faded state, then
// correct):
//     S_a   = Diag(alpha) S                    (the faded state, never written to memory)
//     y_k   = S_a^T k          y_q = S_a^T q   (one read pass computes both)
//     delta = beta (v - y_k)
//     o     = S'^T q = y_q + (q . k) delta     (S' = S_a + k delta^T)
//     S'    = S_a + k delta^T                  (written back in place)
// Each element of S is read once and written once: the kernel is bound by HBM bandwidth
// (2 * d_k * d_v * 4 bytes per head per step).
//
// The same pass serves two more rules (KIND): gated linear attention (engineermaxxing §05b:
// S' = S_a + k v^T, no erase, no beta: delta = v) and normalised phi-linear attention
// (heqinghuang §07, engineermaxxing §02g: phi = elu + 1 on q and k, no decay, delta = v, the
// normaliser z <- z + phi(k) kept beside the state and o divided by phi(q) . z + eps).
//
// Mapping: one CTA (8 warps) per (sequence, head).  Lane l owns d_v columns [l*CPL, l*CPL+CPL)
// (CPL = d_v / 32, one 16-byte load for d = 128); warp w owns d_k rows [w*RPW, w*RPW+RPW).  The
// whole d_k x d_v slab is held in registers between the read and the write, so the state is
// streamed exactly once in each direction.  Column sums over rows are per-thread FMAs, then one
// cross-warp reduction through shared memory; q . k is a warp-shuffle reduction.
#include "gdr_internal.cuh"

namespace gdr {
namespace {

__device__ __forceinline__ void vload(float (&x)[4], const float* p) {
  float4 t = __ldcs(reinterpret_cast<const float4*>(p));
  x[0] = t.x, x[1] = t.y, x[2] = t.z, x[3] = t.w;
}
__device__ __forceinline__ void vload(float (&x)[2], const float* p) {
  float2 t = __ldcs(reinterpret_cast<const float2*>(p));
  x[0] = t.x, x[1] = t.y;
}
__device__ __forceinline__ void vstore(float* p, const float (&x)[4]) {
  __stcs(reinterpret_cast<float4*>(p), make_float4(x[0], x[1], x[2], x[3]));
}
__device__ __forceinline__ void vstore(float* p, const float (&x)[2]) {
  __stcs(reinterpret_cast<float2*>(p), make_float2(x[0], x[1]));
}

constexpr int kDecodeWarps = 8;

template <int D, typename T, bool CHANNEL, int KIND, bool PRO>
__global__ void __launch_bounds__(kDecodeWarps * 32, 2)
    decode_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                  const float* __restrict__ alpha, const float* __restrict__ beta,
                  float* __restrict__ S, T* __restrict__ out, float* __restrict__ z, float eps) {
  constexpr bool prologue = PRO;  // the layer prologue on load (raw projections)
  constexpr bool ERASE = KIND == kKindDelta;      // the delta rule's correction
  constexpr bool NORM = KIND == kKindNormLinear;  // phi features, normaliser, no decay
  constexpr int CPL = D / 32;           // columns per lane
  constexpr int RPW = D / kDecodeWarps;  // rows per warp
  __shared__ float s_q[D], s_k[D], s_a[D], s_v[D], s_delta[D];
  __shared__ float s_red_k[kDecodeWarps][D], s_red_q[kDecodeWarps][D];
  __shared__ float s_ss[2][D / 32];
  __shared__ float s_qz[D / 32];

  const int pair = blockIdx.x;  // n * H + h
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float* Sp = S + (size_t)pair * D * D;
  const int col0 = lane * CPL;

  // 1. issue the whole slab of state loads first (the only large stream)
  float x[RPW][CPL];
#pragma unroll
  for (int r = 0; r < RPW; ++r) vload(x[r], Sp + (size_t)(warp * RPW + r) * D + col0);

  // 2. the token's vectors; with the layer prologue (heqinghuang "gpt2-to-kimi" §09,
  // engineermaxxing §05c/§06b) q, k are the silu of their projections, to be scaled to unit
  // length by iq, ik below, and alpha the sigmoid of its projection
  if (tid < D) {
    const size_t o = (size_t)pair * D + tid;
    float qv = to_f32(q[o]), kv = to_f32(k[o]);
    float av = NORM ? 1.f : CHANNEL ? alpha[o] : alpha[pair];
    if (NORM) {  // z <- z + phi(k); this warp's share of phi(q) . z
      qv = phi_f(qv), kv = phi_f(kv);
      const float zn = z[o] + kv;
      z[o] = zn;
      float qz = qv * zn;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) qz += __shfl_xor_sync(0xffffffffu, qz, off);
      if (lane == 0) s_qz[warp] = qz;
    }
    if (prologue) {
      qv = silu_f(qv), kv = silu_f(kv), av = sigmoid_f(av);
      float sq = qv * qv, sk = kv * kv;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, off);
        sk += __shfl_xor_sync(0xffffffffu, sk, off);
      }
      if (lane == 0) s_ss[0][warp] = sq, s_ss[1][warp] = sk;
    }
    s_q[tid] = qv;
    s_k[tid] = kv;
    s_v[tid] = to_f32(v[o]);
    s_a[tid] = av;
  }
  __syncthreads();
  float iq = 1.f, ik = 1.f;
  if (prologue) {
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int w = 0; w < D / 32; ++w) sq += s_ss[0][w], sk += s_ss[1][w];
    iq = inv_norm(sq), ik = inv_norm(sk);
  }

  // 3. fade the rows and accumulate the two column reads
  float yk[CPL], yq[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) yk[c] = yq[c] = 0.f;
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const int row = warp * RPW + r;
    const float a = s_a[row], kr = s_k[row] * ik, qr = s_q[row] * iq;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      x[r][c] *= a;
      if (ERASE) yk[c] = fmaf(kr, x[r][c], yk[c]);
      yq[c] = fmaf(qr, x[r][c], yq[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    s_red_k[warp][col0 + c] = yk[c];
    s_red_q[warp][col0 + c] = yq[c];
  }
  // q . k (every warp computes it; it is needed by the threads that finish the columns)
  float qk = 0.f;
#pragma unroll
  for (int c = lane; c < D; c += 32) qk = fmaf(s_q[c], s_k[c], qk);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) qk += __shfl_xor_sync(0xffffffffu, qk, off);
  qk *= iq * ik;
  __syncthreads();

  // 4. finish the columns: delta and the read-out
  if (tid < D) {
    float tk = 0.f, tq = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) {
      tk += s_red_k[w][tid];
      tq += s_red_q[w][tid];
    }
    float d = s_v[tid];  // gated linear and normalised linear attention write v itself
    if (ERASE) d = (prologue ? sigmoid_f(beta[pair]) : beta[pair]) * (d - tk);
    s_delta[tid] = d;
    float o = fmaf(qk, d, tq);
    if (NORM) {
      float den = eps;
#pragma unroll
      for (int w = 0; w < D / 32; ++w) den += s_qz[w];
      o /= den;
    }
    out[(size_t)pair * D + tid] = from_f32<T>(o);
  }
  __syncthreads();

  // 5. write back S' = S_a + k delta^T
  float dl[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) dl[c] = s_delta[col0 + c];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const float kr = s_k[warp * RPW + r] * ik;
#pragma unroll
    for (int c = 0; c < CPL; ++c) x[r][c] = fmaf(kr, dl[c], x[r][c]);
    vstore(Sp + (size_t)(warp * RPW + r) * D + col0, x[r]);
  }
}

template <int D, typename T, int KIND>
void launch_kind(const gdr_shape& sh, const void* q, const void* k, const void* v,
                 const float* alpha, const float* beta, float* S, float* z, float eps,
                 void* out, cudaStream_t s) {
  const unsigned grid = (unsigned)sh.n_seqs * (unsigned)sh.H;
  const bool pro = KIND != kKindNormLinear && (sh.flags & GDR_FLAG_LAYER_PROLOGUE) != 0;
  const bool ch = KIND == kKindNormLinear || sh.gate == GDR_GATE_CHANNEL;
  auto kern = ch ? (pro ? decode_kernel<D, T, true, KIND, true>
                         : decode_kernel<D, T, true, KIND, false>)
                 : (pro ? decode_kernel<D, T, false, KIND, true>
                         : decode_kernel<D, T, false, KIND, false>);
  kern<<<grid, kDecodeWarps * 32, 0, s>>>((const T*)q, (const T*)k, (const T*)v, alpha, beta, S,
                                          (T*)out, z, eps);
}

template <int D, typename T>
cudaError_t launch_typed(const gdr_shape& sh, int kind, const void* q, const void* k,
                         const void* v, const float* alpha, const float* beta, float* S,
                         float* z, float eps, void* out, cudaStream_t s) {
  if (kind == kKindNormLinear)
    launch_kind<D, T, kKindNormLinear>(sh, q, k, v, alpha, beta, S, z, eps, out, s);
  else if (kind == kKindGatedLinear)
    launch_kind<D, T, kKindGatedLinear>(sh, q, k, v, alpha, beta, S, z, eps, out, s);
  else
    launch_kind<D, T, kKindDelta>(sh, q, k, v, alpha, beta, S, z, eps, out, s);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const gdr_shape& sh, int kind, const void* q, const void* k,
                          const void* v, const float* alpha, const float* beta, float* S,
                          float* z, float eps, void* out, cudaStream_t s) {
  if (sh.d_k == 128)
    return sh.dtype == GDR_BF16
               ? launch_typed<128, __nv_bfloat16>(sh, kind, q, k, v, alpha, beta, S, z, eps, out, s)
               : launch_typed<128, float>(sh, kind, q, k, v, alpha, beta, S, z, eps, out, s);
  return sh.dtype == GDR_BF16
             ? launch_typed<64, __nv_bfloat16>(sh, kind, q, k, v, alpha, beta, S, z, eps, out, s)
             : launch_typed<64, float>(sh, kind, q, k, v, alpha, beta, S, z, eps, out, s);
}

}  // namespace gdr
