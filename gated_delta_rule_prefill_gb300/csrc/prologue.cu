// prologue.cu -- the layer prologue as a pass of its own over HBM: raw projections in, the rule's
// inputs out (heqinghuang "gpt2-to-kimi" §09: unit-length silu queries and keys, beta a sigmoid
// of its projection; engineermaxxing "From GPT-2 to Kimi K3" §05c / §06b: the decay a sigmoid of
// its projection, per head or per key channel):
//     q = silu(xq) / max(||silu(xq)||_2, 1e-12)   (over the d_k channels of a (token, head))
//     k likewise,  alpha = sigmoid(a),  beta = sigmoid(b)
// The prefill and decode kernels apply the same maps on load (GDR_FLAG_LAYER_PROLOGUE); this pass
// serves callers that keep the mapped tensors, and is the unfused baseline of that fusion.
//
// Bound by HBM bandwidth: every element is read once and written once.  Mapping: one warp per
// (token, head) row of q and of k (lane l holds channels [l*CPL, l*CPL + CPL), one 8- or 16-byte
// access); alpha and beta are flat elementwise streams of float4.  A grid-stride loop over a grid
// of a few CTAs per SM keeps every SM busy for any T.  The math is fp32 with accurate silu and
// sigmoid (the pass is memory bound, so the exact forms cost nothing).
#include "gdr_internal.cuh"

namespace gdr {
namespace {

constexpr int kProThreads = 256;

template <typename T, int CPL>
struct RowIO;
template <>
struct RowIO<__nv_bfloat16, 4> {  // d = 128 bf16: 8 bytes a lane
  static __device__ void load(const __nv_bfloat16* p, float* x) {
    const uint2 u = __ldcs(reinterpret_cast<const uint2*>(p));
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    x[0] = a.x, x[1] = a.y, x[2] = b.x, x[3] = b.y;
  }
  static __device__ void store(__nv_bfloat16* p, const float* x) {
    uint2 u;
    *reinterpret_cast<__nv_bfloat162*>(&u.x) = __floats2bfloat162_rn(x[0], x[1]);
    *reinterpret_cast<__nv_bfloat162*>(&u.y) = __floats2bfloat162_rn(x[2], x[3]);
    __stcs(reinterpret_cast<uint2*>(p), u);
  }
};
template <>
struct RowIO<__nv_bfloat16, 2> {  // d = 64 bf16: 4 bytes a lane
  static __device__ void load(const __nv_bfloat16* p, float* x) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
    x[0] = a.x, x[1] = a.y;
  }
  static __device__ void store(__nv_bfloat16* p, const float* x) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(x[0], x[1]);
  }
};
template <>
struct RowIO<float, 4> {  // d = 128 fp32: 16 bytes a lane
  static __device__ void load(const float* p, float* x) {
    const float4 u = __ldcs(reinterpret_cast<const float4*>(p));
    x[0] = u.x, x[1] = u.y, x[2] = u.z, x[3] = u.w;
  }
  static __device__ void store(float* p, const float* x) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(x[0], x[1], x[2], x[3]));
  }
};
template <>
struct RowIO<float, 2> {  // d = 64 fp32: 8 bytes a lane
  static __device__ void load(const float* p, float* x) {
    const float2 u = __ldcs(reinterpret_cast<const float2*>(p));
    x[0] = u.x, x[1] = u.y;
  }
  static __device__ void store(float* p, const float* x) {
    __stcs(reinterpret_cast<float2*>(p), make_float2(x[0], x[1]));
  }
};

// rows: 2 * T * H rows of D channels (the q rows, then the k rows); gates: n_a + n_b values.
// A warp takes kRows consecutive rows at a time and a thread kVec float4 of a gate stream at a
// time, every load issued before any result is used, so that enough bytes are in flight per SM
// to cover the HBM latency.
constexpr int kRows = 8, kVec = 4;
template <int D, typename T>
__global__ void __launch_bounds__(kProThreads)
    prologue_kernel(const T* xq, const T* xk, T* q, T* k, int64_t rows, const float* a,
                    float* alpha, int64_t n_a, const float* b, float* beta, int64_t n_b) {
  constexpr int CPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (kProThreads / 32);
  const int64_t w0 = (int64_t)blockIdx.x * (kProThreads / 32) + (threadIdx.x >> 5);
  for (int64_t g = w0 * kRows; g < 2 * rows; g += warps * kRows) {
    float x[kRows][CPL];
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const int64_t row = g + i;
      if (row < 2 * rows) {
        const bool isk = row >= rows;
        RowIO<T, CPL>::load((isk ? xk : xq) + (isk ? row - rows : row) * D + lane * CPL, x[i]);
      } else {
#pragma unroll
        for (int c = 0; c < CPL; ++c) x[i][c] = 0.f;
      }
    }
    float ss[kRows];
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      ss[i] = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        x[i][c] = silu_f(x[i][c]);
        ss[i] = fmaf(x[i][c], x[i][c], ss[i]);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int i = 0; i < kRows; ++i) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], off);
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const int64_t row = g + i;
      if (row < 2 * rows) {
        const float inv = inv_norm(ss[i]);
#pragma unroll
        for (int c = 0; c < CPL; ++c) x[i][c] *= inv;
        const bool isk = row >= rows;
        RowIO<T, CPL>::store((isk ? k : q) + (isk ? row - rows : row) * D + lane * CPL, x[i]);
      }
    }
  }
  // the gates: float4 streams, then the scalar tail of a stream whose length is not a multiple of 4
  const int64_t threads = (int64_t)gridDim.x * kProThreads;
  const int64_t t0 = (int64_t)blockIdx.x * kProThreads + threadIdx.x;
  for (int s = 0; s < 2; ++s) {
    const float* in = s ? b : a;
    float* out = s ? beta : alpha;
    const int64_t n = s ? n_b : n_a;
    if (!in) continue;
    const int64_t n4 = n / 4;
    for (int64_t i = t0; i < n4; i += threads * kVec) {
      float4 u[kVec];
#pragma unroll
      for (int j = 0; j < kVec; ++j)
        if (i + j * threads < n4) u[j] = __ldcs(reinterpret_cast<const float4*>(in) + i + j * threads);
#pragma unroll
      for (int j = 0; j < kVec; ++j) {
        if (i + j * threads < n4) {
          u[j].x = sigmoid_f(u[j].x), u[j].y = sigmoid_f(u[j].y);
          u[j].z = sigmoid_f(u[j].z), u[j].w = sigmoid_f(u[j].w);
          __stcs(reinterpret_cast<float4*>(out) + i + j * threads, u[j]);
        }
      }
    }
    for (int64_t i = 4 * n4 + t0; i < n; i += threads) out[i] = sigmoid_f(in[i]);
  }
}

template <int D, typename T>
cudaError_t launch_typed(const gdr_shape& sh, const void* xq, const void* xk, const float* a,
                         const float* b, void* q, void* k, float* alpha, float* beta,
                         cudaStream_t s) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorUnknown;
  const int64_t rows = sh.total_tokens * sh.H;
  const int64_t n_a = sh.gate == GDR_GATE_CHANNEL ? rows * D : rows;
  // up to 4 CTAs of 8 warps per SM, each warp kRows rows at a time
  const int64_t per_cta = (int64_t)(kProThreads / 32) * kRows;
  const int64_t need = (2 * rows + per_cta - 1) / per_cta;
  const unsigned grid = (unsigned)(need < 4LL * sms ? (need > 0 ? need : 1) : 4LL * sms);
  prologue_kernel<D, T><<<grid, kProThreads, 0, s>>>(
      (const T*)xq, (const T*)xk, (T*)q, (T*)k, rows, a, alpha, a ? n_a : 0, b, beta,
      b ? rows : 0);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_layer_prologue(const gdr_shape& sh, const void* xq, const void* xk,
                                  const float* a, const float* b, void* q, void* k, float* alpha,
                                  float* beta, cudaStream_t s) {
  if (sh.dtype == GDR_BF16)
    return sh.d_k == 128
               ? launch_typed<128, __nv_bfloat16>(sh, xq, xk, a, b, q, k, alpha, beta, s)
               : launch_typed<64, __nv_bfloat16>(sh, xq, xk, a, b, q, k, alpha, beta, s);
  return sh.d_k == 128 ? launch_typed<128, float>(sh, xq, xk, a, b, q, k, alpha, beta, s)
                       : launch_typed<64, float>(sh, xq, xk, a, b, q, k, alpha, beta, s);
}

}  // namespace gdr
