// gdr_internal.cuh -- shared declarations of the GPU library (never included by the oracle).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdr.h"

namespace gdr {

// Per-token lower clamp of log(alpha).  e^-60 ~ 9e-27, so alpha = 0 (a full reset) is exact to
// within fp32 while cumulative sums of log-gates stay finite.
constexpr float kLogAlphaMin = -60.0f;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float log_gate(float a) { return fmaxf(__logf(a), kLogAlphaMin); }

// Workspace layout used by the prefill / linear-attention calls: the status word, the visiting
// order, then (for shapes the work-queue tensor-core prefill may run) its flags and a ring of
// operand slots per (sequence, head) chain, through which helper CTAs hand prepared chunks to
// the chain's CTA.
struct WorkspaceLayout {
  static constexpr size_t kHeaderBytes = 256;      // int32 status word + reserved
  static constexpr size_t kRingSlotBytes = 74752;  // one chunk's operand slot image
  static constexpr int kRingSlots = 6;             // chunks in flight per chain
  static constexpr long kRingMaxPairs = 76;        // chains of the largest work-queue launch
  static size_t order_bytes(int n_seqs) { return ((size_t)n_seqs * 4 + 255) / 256 * 256; }
  // the minimum: enough for every path except the work-queue prefill
  static size_t total(int n_seqs) { return kHeaderBytes + order_bytes(n_seqs); }
  static long ring_pairs(const gdr_shape& sh) {
    const long pairs = (long)sh.n_seqs * sh.H;
    return (sh.dtype == GDR_BF16 && sh.d_k == 128 && sh.d_v == 128 && pairs <= kRingMaxPairs)
               ? pairs : 0;
  }
  // work-item counter, ready[pairs][slots], loaded[pairs] (uint32)
  static size_t flag_bytes(long pairs) {
    return ((size_t)(1 + pairs * kRingSlots + pairs) * 4 + 255) / 256 * 256;
  }
  static size_t ring_bytes(const gdr_shape& sh) {
    const long p = ring_pairs(sh);
    return p ? flag_bytes(p) + (size_t)p * kRingSlots * kRingSlotBytes : 0;
  }
  // the full size (gdr_prefill_workspace_size): also enables the work-queue prefill
  static size_t full(const gdr_shape& sh) { return total(sh.n_seqs) + ring_bytes(sh); }
};

// Arguments of the chunked prefill kernels (device pointers; see gdr.h for layouts).
struct PrefillArgs {
  int n_seqs, H;
  int64_t total_tokens;
  const void* q;
  const void* k;
  const void* v;
  const float* alpha;
  const float* beta;
  const float* S0;
  const int32_t* cu_seqlens;  // may be null: one sequence
  void* out;
  float* S_final;
  const int32_t* order;  // sequence visiting order (longest first)
  int32_t* status;       // device-check word
  uint32_t* ring_flags;  // work-queue prefill: counter, ready, loaded (null: not available)
  unsigned char* ring;   // work-queue prefill: operand slots
  const void* og = nullptr;  // output gate g [T, H, d_v] (dtype of out): out = o * sigmoid(g)
  // q, k, alpha, beta hold the layer's raw projections: the kernels apply the layer prologue
  // (q, k = normalize(silu(.)), alpha, beta = sigmoid(.)) as they load them.
  bool prologue = false;
  // normalised phi-linear attention: entering / final normaliser z [N, H, d_k] (null: zeros /
  // not written) and the eps added to phi(q) . z
  const float* z0 = nullptr;
  float* z_final = nullptr;
  float eps = 0.f;
  // the library's per-device error word (gdr_query_device_status), written beside `status`
  int32_t* dev_status = nullptr;
};

// Records the first device-check failure (0 -> code).
__device__ __forceinline__ void report(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

// Records a device-check failure of a prefill-like call in its workspace word and in the
// library's per-device error word.
__device__ __forceinline__ void report(const PrefillArgs& a, int32_t code) {
  report(a.status, code);
  report(a.dev_status, code);
}

// phi(x) = elu(x) + 1: x + 1 above zero, e^x at and below it.
__device__ __forceinline__ float phi_f(float x) { return x > 0.f ? x + 1.f : __expf(x); }

// The layer prologue's maps in fp32: sigmoid(x) = 1 / (1 + e^-x) (the exponent capped at 80 so
// the fast division never meets an infinite divisor), silu(x) = x sigmoid(x), and the scale
// 1 / max(||x||, 1e-12) of the L2 normalisation from the squared norm ss.
__device__ __forceinline__ float sigmoid_f(float x) {
  return __fdividef(1.f, 1.f + __expf(fminf(-x, 80.f)));
}
__device__ __forceinline__ float silu_f(float x) { return x * sigmoid_f(x); }
__device__ __forceinline__ float inv_norm(float ss) { return ss >= 1e-24f ? rsqrtf(ss) : 1e12f; }

// The output gate of one element: o * sigmoid(g).
__device__ __forceinline__ float gate_out(float o, float g) { return o / (1.f + __expf(-g)); }

// Resolves (seq -> token range) with the bounds check every kernel performs before touching
// memory.  Returns false (after recording the failure) if the range is invalid.
__device__ __forceinline__ bool seq_range(const PrefillArgs& a, int seq, int64_t& t0,
                                          int64_t& t1) {
  if (a.cu_seqlens) {
    t0 = a.cu_seqlens[seq];
    t1 = a.cu_seqlens[seq + 1];
  } else {
    t0 = 0;
    t1 = a.total_tokens;
  }
  if (t0 < 0 || t1 < t0 || t1 > a.total_tokens) {
    report(a, GDR_DEVCHECK_SEQLENS);
    return false;
  }
  return true;
}

// What a prefill-like call computes: the gated delta rule, plain linear attention (alpha = 1,
// no erase), or gated linear attention (S <- Diag(alpha) S + k v^T: no erase, no beta).
enum PrefillKind : int {
  kKindDelta = 0,        // the gated delta rule
  kKindLinear = 1,       // plain linear attention
  kKindGatedLinear = 2,  // gated linear attention (no erase)
  kKindNormLinear = 3    // normalised phi-linear attention (phi = elu + 1, normaliser z)
};

// The shape checks every prefill-like call makes (GDR_OK or the error to return).
gdr_status validate_shape(const gdr_shape* sh, bool need_gate);

// gdr_prefill with an explicit workspace (validation, pre-pass and launch).
gdr_status prefill_launch(const gdr_shape* sh, const void* q, const void* k, const void* v,
                          const float* alpha, const float* beta, const float* S0,
                          const int32_t* cu, void* out, float* S_final, void* ws,
                          size_t ws_bytes, void* stream);

// Host-side launchers (each returns cudaSuccess or the launch error).
cudaError_t launch_prep(const PrefillArgs& a, int32_t* order, cudaStream_t s);
cudaError_t launch_prefill_simt(const gdr_shape& sh, const PrefillArgs& a, int kind,
                                cudaStream_t s);
bool prefill_tc_supported(const gdr_shape& sh);
cudaError_t launch_prefill_tc(const gdr_shape& sh, const PrefillArgs& a, int kind,
                              cudaStream_t s);
cudaError_t launch_layer_prologue(const gdr_shape& sh, const void* xq, const void* xk,
                                  const float* a, const float* b, void* q, void* k, float* alpha,
                                  float* beta, cudaStream_t s);
cudaError_t launch_decode(const gdr_shape& sh, int kind, const void* q, const void* k,
                          const void* v, const float* alpha, const float* beta, float* S,
                          float* z, float eps, void* out, cudaStream_t s);

}  // namespace gdr
