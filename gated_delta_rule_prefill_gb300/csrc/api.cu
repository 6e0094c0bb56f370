// api.cu -- the C ABI of libgdr (declared in include/gdr.h): argument validation, the sequence
// pre-pass, kernel selection and launch on the caller's stream.
#include <string.h>

#include "gdr_internal.cuh"
#include "umma.cuh"

namespace gdr {
namespace {

constexpr int kPrepThreads = 1024;
constexpr int kSortMax = 8192;  // longest-first ordering up to this many sequences

// The library's error word on each device: every device-check failure of a prefill-like call
// is also recorded here (the first code since the last gdr_query_device_status, which takes it
// with an atomic exchange into g_device_status_taken and reads that back).
__device__ int32_t g_device_status;
__device__ int32_t g_device_status_taken;

__global__ void take_device_status_kernel() {
  g_device_status_taken = atomicExch(&g_device_status, 0);
}

// One warp waits on an mbarrier that nothing arrives on, with the kernels' bounded wait; each
// lane gives up after limit_ns, and lane 0 records the timeout as a kernel would.
__global__ void __launch_bounds__(32) wait_timeout_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    umma::mbar_init(&bar, 1);
    umma::fence_mbar_init();
  }
  __syncwarp();
  const bool done = umma::mbar_wait(&bar, 0, limit_ns);
  __syncwarp();
  if (threadIdx.x == 0 && !done) {
    report(status, GDR_DEVCHECK_TIMEOUT);
    report(&g_device_status, GDR_DEVCHECK_TIMEOUT);
  }
}

// One CTA: clears the status word, checks cu_seqlens, and writes the visiting order of the
// sequences (longest first, ties by index) so that long sequences start first.
__global__ void __launch_bounds__(kPrepThreads)
    prep_kernel(const int32_t* __restrict__ cu, int n_seqs, int64_t total, int32_t* order,
                int32_t* status, int32_t* dev_status) {
  __shared__ int32_t s_len[kSortMax];
  __shared__ int s_bad;
  if (threadIdx.x == 0) {
    *status = 0;
    s_bad = 0;
  }
  __syncthreads();
  const bool sort = n_seqs <= kSortMax;
  for (int i = threadIdx.x; i < n_seqs; i += blockDim.x) {
    int64_t a = cu ? cu[i] : 0, b = cu ? cu[i + 1] : total;
    int32_t len = (int32_t)(b - a);
    if (a < 0 || b < a || b > total) {
      s_bad = 1;
      len = 0;
    }
    if (sort) s_len[i] = len;
  }
  __syncthreads();
  if (s_bad && threadIdx.x == 0) {
    atomicCAS(status, 0, GDR_DEVCHECK_SEQLENS);
    atomicCAS(dev_status, 0, GDR_DEVCHECK_SEQLENS);
  }
  for (int i = threadIdx.x; i < n_seqs; i += blockDim.x) {
    if (!sort) {
      order[i] = i;
      continue;
    }
    const int32_t li = s_len[i];
    int rank = 0;
    for (int j = 0; j < n_seqs; ++j) {
      const int32_t lj = s_len[j];
      rank += (lj > li) || (lj == li && j < i);
    }
    order[rank] = i;
  }
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

gdr_status check_shape(const gdr_shape* sh, bool need_gate) {
  if (!sh) return GDR_ERR_INVALID_ARG;
  if (sh->n_seqs < 1 || sh->H < 1 || sh->total_tokens < 0 || sh->d_k < 1 || sh->d_v < 1)
    return GDR_ERR_INVALID_ARG;
  if (sh->dtype != GDR_F32 && sh->dtype != GDR_BF16) return GDR_ERR_INVALID_ARG;
  if (need_gate && sh->gate != GDR_GATE_SCALAR && sh->gate != GDR_GATE_CHANNEL)
    return GDR_ERR_INVALID_ARG;
  if (sh->chunk_size < 0 || (sh->flags & ~(GDR_FLAG_FORCE_SIMT | GDR_FLAG_NO_CLUSTER | GDR_FLAG_PREFER_QUEUE |
                                                GDR_FLAG_LAYER_PROLOGUE))) return GDR_ERR_INVALID_ARG;
  if (sh->d_k != sh->d_v || (sh->d_k != 64 && sh->d_k != 128)) return GDR_ERR_UNSUPPORTED;
  // grid sizes stay within 32-bit block counts
  if ((int64_t)sh->n_seqs * sh->H * 4 > (int64_t)INT32_MAX) return GDR_ERR_UNSUPPORTED;
  return GDR_OK;
}

gdr_status prefill_common(const gdr_shape* sh, const void* q, const void* k, const void* v,
                          const float* alpha, const float* beta, const float* S0,
                          const int32_t* cu, void* out, float* S_final, void* ws,
                          size_t ws_bytes, void* stream, int kind, const void* og = nullptr,
                          const float* z0 = nullptr, float* z_final = nullptr, float eps = 0.f) {
  const bool linear = kind == kKindLinear || kind == kKindNormLinear;
  gdr_status st = check_shape(sh, !linear);
  if (st != GDR_OK) return st;
  const bool prologue = (sh->flags & GDR_FLAG_LAYER_PROLOGUE) != 0;
  if (linear && prologue) return GDR_ERR_UNSUPPORTED;
  if (!cu && sh->n_seqs != 1) return GDR_ERR_INVALID_ARG;
  if (sh->total_tokens > 0) {
    if (!q || !k || !v || !out) return GDR_ERR_INVALID_ARG;
    if (!linear && !alpha) return GDR_ERR_INVALID_ARG;
    if (kind == kKindDelta && !beta) return GDR_ERR_INVALID_ARG;
  }
  const void* ptrs[] = {q, k, v, alpha, beta, S0, cu, out, S_final, og, z0, z_final};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return GDR_ERR_INVALID_ARG;
  if (og && og == out) return GDR_ERR_INVALID_ARG;
  if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < WorkspaceLayout::total(sh->n_seqs))
    return GDR_ERR_INVALID_ARG;
  if (out && (out == q || out == k || out == v)) return GDR_ERR_INVALID_ARG;
  if (sh->chunk_size != 0 && sh->chunk_size != 64) return GDR_ERR_UNSUPPORTED;

  cudaStream_t s = (cudaStream_t)stream;
  int32_t* status = (int32_t*)ws;
  int32_t* order = (int32_t*)((char*)ws + WorkspaceLayout::kHeaderBytes);
  uint32_t* ring_flags = nullptr;
  unsigned char* ring = nullptr;
  if (WorkspaceLayout::ring_bytes(*sh) > 0 && ws_bytes >= WorkspaceLayout::full(*sh)) {
    ring_flags = (uint32_t*)((char*)ws + WorkspaceLayout::total(sh->n_seqs));
    ring = (unsigned char*)ring_flags +
           WorkspaceLayout::flag_bytes(WorkspaceLayout::ring_pairs(*sh));
  }
  int32_t* dev_status = nullptr;
  if (cudaGetSymbolAddress((void**)&dev_status, g_device_status) != cudaSuccess) return GDR_ERR_CUDA;
  PrefillArgs a{sh->n_seqs, sh->H, sh->total_tokens, q, k, v, alpha, beta, S0, cu,
                out, S_final, order, status, ring_flags, ring, og, prologue, z0, z_final, eps,
                dev_status};
  prep_kernel<<<1, kPrepThreads, 0, s>>>(cu, sh->n_seqs, sh->total_tokens, order, status,
                                         dev_status);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess)
    e = prefill_tc_supported(*sh) ? launch_prefill_tc(*sh, a, kind, s)
                                  : launch_prefill_simt(*sh, a, kind, s);
  return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

}  // namespace

gdr_status validate_shape(const gdr_shape* sh, bool need_gate) { return check_shape(sh, need_gate); }

// One decode step of the delta rule, gated linear or normalised linear attention.
gdr_status decode_common(const gdr_shape* shape, int kind, const void* q, const void* k,
                         const void* v, const float* alpha, const float* beta, float* S_inout,
                         float* z_inout, float eps, void* out, void* stream) {
  const bool norm = kind == kKindNormLinear;
  gdr_status st = check_shape(shape, !norm);
  if (st != GDR_OK) return st;
  if (norm && (shape->flags & GDR_FLAG_LAYER_PROLOGUE)) return GDR_ERR_UNSUPPORTED;
  if (shape->total_tokens != shape->n_seqs) return GDR_ERR_INVALID_ARG;
  if (!q || !k || !v || !S_inout || !out) return GDR_ERR_INVALID_ARG;
  if ((!norm && !alpha) || (kind == kKindDelta && !beta) || (norm && !z_inout))
    return GDR_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, alpha, beta, S_inout, z_inout, out};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return GDR_ERR_INVALID_ARG;
  if (out == q || out == k || out == v || (const void*)S_inout == out ||
      (z_inout && ((const void*)z_inout == out || z_inout == S_inout)))
    return GDR_ERR_INVALID_ARG;
  cudaError_t e = launch_decode(*shape, kind, q, k, v, alpha, beta, S_inout, z_inout, eps, out,
                                (cudaStream_t)stream);
  return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

gdr_status prefill_launch(const gdr_shape* sh, const void* q, const void* k, const void* v,
                          const float* alpha, const float* beta, const float* S0,
                          const int32_t* cu, void* out, float* S_final, void* ws,
                          size_t ws_bytes, void* stream) {
  return prefill_common(sh, q, k, v, alpha, beta, S0, cu, out, S_final, ws, ws_bytes, stream,
                        kKindDelta);
}

}  // namespace gdr

extern "C" {

size_t gdr_prefill_workspace_size(const gdr_shape* shape) {
  if (!shape || shape->n_seqs < 1 || shape->H < 1) return 0;
  return gdr::WorkspaceLayout::full(*shape);
}

gdr_status gdr_prefill(const gdr_shape* shape, const void* q, const void* k, const void* v,
                       const float* alpha, const float* beta, const float* S0,
                       const int32_t* cu_seqlens, void* out, float* S_final, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return gdr::prefill_common(shape, q, k, v, alpha, beta, S0, cu_seqlens, out, S_final,
                             workspace, workspace_bytes, stream, gdr::kKindDelta);
}

gdr_status gdr_linear_attn(const gdr_shape* shape, const void* q, const void* k, const void* v,
                           const float* S0, const int32_t* cu_seqlens, void* out, float* S_final,
                           void* workspace, size_t workspace_bytes, void* stream) {
  return gdr::prefill_common(shape, q, k, v, nullptr, nullptr, S0, cu_seqlens, out, S_final,
                             workspace, workspace_bytes, stream, gdr::kKindLinear);
}

gdr_status gdr_prefill_output_gate(const gdr_shape* shape, const void* q, const void* k,
                                   const void* v, const float* alpha, const float* beta,
                                   const void* g, const float* S0, const int32_t* cu_seqlens,
                                   void* out, float* S_final, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  if (!g && shape && shape->total_tokens > 0) return GDR_ERR_INVALID_ARG;
  return gdr::prefill_common(shape, q, k, v, alpha, beta, S0, cu_seqlens, out, S_final,
                             workspace, workspace_bytes, stream, gdr::kKindDelta, g);
}

gdr_status gdr_gated_linear_attn(const gdr_shape* shape, const void* q, const void* k,
                                 const void* v, const float* alpha, const float* S0,
                                 const int32_t* cu_seqlens, void* out, float* S_final,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  return gdr::prefill_common(shape, q, k, v, alpha, nullptr, S0, cu_seqlens, out, S_final,
                             workspace, workspace_bytes, stream, gdr::kKindGatedLinear);
}

gdr_status gdr_normalized_linear_attn(const gdr_shape* shape, const void* q, const void* k,
                                      const void* v, float eps, const float* S0, const float* z0,
                                      const int32_t* cu_seqlens, void* out, float* S_final,
                                      float* z_final, void* workspace, size_t workspace_bytes,
                                      void* stream) {
  if (!(eps >= 0.f) || eps > 3.0e38f) return GDR_ERR_INVALID_ARG;  // also rejects NaN
  // every value block of a (sequence, head) reads z0 at its start; one of them writes z_final
  if (z0 && z0 == z_final) return GDR_ERR_INVALID_ARG;
  return gdr::prefill_common(shape, q, k, v, nullptr, nullptr, S0, cu_seqlens, out, S_final,
                             workspace, workspace_bytes, stream, gdr::kKindNormLinear, nullptr,
                             z0, z_final, eps);
}

gdr_status gdr_decode_step(const gdr_shape* shape, const void* q, const void* k, const void* v,
                           const float* alpha, const float* beta, float* S_inout, void* out,
                           void* stream) {
  return gdr::decode_common(shape, gdr::kKindDelta, q, k, v, alpha, beta, S_inout, nullptr, 0.f,
                            out, stream);
}

gdr_status gdr_gated_linear_decode_step(const gdr_shape* shape, const void* q, const void* k,
                                        const void* v, const float* alpha, float* S_inout,
                                        void* out, void* stream) {
  return gdr::decode_common(shape, gdr::kKindGatedLinear, q, k, v, alpha, nullptr, S_inout,
                            nullptr, 0.f, out, stream);
}

gdr_status gdr_normalized_linear_decode_step(const gdr_shape* shape, const void* q, const void* k,
                                             const void* v, float eps, float* S_inout,
                                             float* z_inout, void* out, void* stream) {
  if (!(eps >= 0.f) || eps > 3.0e38f) return GDR_ERR_INVALID_ARG;
  return gdr::decode_common(shape, gdr::kKindNormLinear, q, k, v, nullptr, nullptr, S_inout,
                            z_inout, eps, out, stream);
}

gdr_status gdr_layer_prologue(const gdr_shape* shape, const void* xq, const void* xk,
                              const float* a, const float* b, void* q, void* k, float* alpha,
                              float* beta, void* stream) {
  gdr_status st = gdr::check_shape(shape, a != nullptr);
  if (st != GDR_OK) return st;
  if (shape->total_tokens == 0) return GDR_OK;
  if (!xq || !xk || !q || !k) return GDR_ERR_INVALID_ARG;
  if (!a != !alpha || !b != !beta) return GDR_ERR_INVALID_ARG;
  const void* ptrs[] = {xq, xk, a, b, q, k, alpha, beta};
  for (const void* p : ptrs)
    if (p && !gdr::aligned16(p)) return GDR_ERR_INVALID_ARG;
  // outputs either are their own input (in place) or do not meet another operand's start
  if ((q != xq && (q == xk || q == k)) || (k != xk && k == xq)) return GDR_ERR_INVALID_ARG;
  cudaError_t e = gdr::launch_layer_prologue(*shape, xq, xk, a, b, q, k, alpha, beta,
                                             (cudaStream_t)stream);
  return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

gdr_status gdr_workspace_status(void* workspace, void* stream, int32_t* code) {
  if (!workspace || !code) return GDR_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return GDR_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDR_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), s) != cudaSuccess) return GDR_ERR_CUDA;
  *code = h;
  return GDR_OK;
}

gdr_status gdr_query_device_status(void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDR_ERR_CUDA;
  gdr::take_device_status_kernel<<<1, 1, 0, s>>>();
  if (cudaGetLastError() != cudaSuccess) return GDR_ERR_CUDA;
  int32_t h = 0;
  if (cudaMemcpyFromSymbolAsync(&h, gdr::g_device_status_taken, sizeof(h), 0,
                                cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return GDR_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDR_ERR_CUDA;
  return h == GDR_DEVCHECK_OK ? GDR_OK : GDR_ERR_DEVICE_CHECK;
}

gdr_status gdr_check_wait_timeout(void* workspace, uint64_t limit_ns, void* stream) {
  if (!workspace || ((uintptr_t)workspace & 255u)) return GDR_ERR_INVALID_ARG;
  if (limit_ns == 0 || limit_ns > 10000000000ull) return GDR_ERR_INVALID_ARG;
  gdr::wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((int32_t*)workspace, limit_ns);
  return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

const char* gdr_status_string(gdr_status status) {
  switch (status) {
    case GDR_OK:
      return "GDR_OK";
    case GDR_ERR_INVALID_ARG:
      return "GDR_ERR_INVALID_ARG";
    case GDR_ERR_UNSUPPORTED:
      return "GDR_ERR_UNSUPPORTED";
    case GDR_ERR_CUDA:
      return "GDR_ERR_CUDA";
    case GDR_ERR_DEVICE_CHECK:
      return "GDR_ERR_DEVICE_CHECK";
  }
  return "GDR_ERR_UNKNOWN";
}

}  // extern "C"
