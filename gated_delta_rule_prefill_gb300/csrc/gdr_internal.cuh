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

// Workspace layout used by the prefill / linear-attention calls.
struct WorkspaceLayout {
  static constexpr size_t kHeaderBytes = 256;  // int32 status word + reserved
  static size_t order_bytes(int n_seqs) { return ((size_t)n_seqs * 4 + 255) / 256 * 256; }
  static size_t total(int n_seqs) { return kHeaderBytes + order_bytes(n_seqs); }
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
};

// Records the first device-check failure (0 -> code).
__device__ __forceinline__ void report(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

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
    report(a.status, GDR_DEVCHECK_SEQLENS);
    return false;
  }
  return true;
}

// gdr_prefill with an explicit workspace (validation, pre-pass and launch).
gdr_status prefill_launch(const gdr_shape* sh, const void* q, const void* k, const void* v,
                          const float* alpha, const float* beta, const float* S0,
                          const int32_t* cu, void* out, float* S_final, void* ws,
                          size_t ws_bytes, void* stream);

// Host-side launchers (each returns cudaSuccess or the launch error).
cudaError_t launch_prep(const PrefillArgs& a, int32_t* order, cudaStream_t s);
cudaError_t launch_prefill_simt(const gdr_shape& sh, const PrefillArgs& a, bool linear,
                                cudaStream_t s);
bool prefill_tc_supported(const gdr_shape& sh);
cudaError_t launch_prefill_tc(const gdr_shape& sh, const PrefillArgs& a, bool linear,
                              cudaStream_t s);
cudaError_t launch_decode(const gdr_shape& sh, const void* q, const void* k, const void* v,
                          const float* alpha, const float* beta, float* S, void* out,
                          cudaStream_t s);

}  // namespace gdr
