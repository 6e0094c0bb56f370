// noalloc.cu -- gdr_prefill_noalloc: the chunked prefill without a caller-provided workspace.
//
// Some callers cannot hand the library a scratch buffer: their device memory is fully
// budgeted by a host framework or by a static memory plan, so they have no spare allocation to
// give, and they must not call cudaMalloc themselves (an allocation can also synchronise the
// device, which a latency-critical caller has to avoid).  This entry point serves them: the
// prefill's scratch (the device-check word and the sequence visiting order) lives in a fixed
// array in this library's device memory instead of a workspace.
//
// The array is statically sized for at most GDR_NOALLOC_MAX_SEQS sequences; every GPU that
// loads the library keeps it until the process exits.  All calls share it and it keeps the
// contents of the last call: each call's pre-pass rewrites the whole part it uses (the check
// word is cleared first, the order array fully written), so nothing carries over, but two calls
// whose work overlaps on the GPU (different streams, or different host threads) race on it and
// must be serialised by the caller.
#include "gdr_internal.cuh"

namespace gdr {
namespace {

constexpr size_t kNoAllocScratchBytes = WorkspaceLayout::kHeaderBytes +
                                        ((size_t)GDR_NOALLOC_MAX_SEQS * 4 + 255) / 256 * 256;

// The shared scratch: a device-side symbol, so host code never uses its address directly; the
// device address is looked up with cudaGetSymbolAddress on every call, with the caller's device
// current (a cached address would go stale if the caller reset the device and the module were
// loaded again into a new context).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

}  // namespace
}  // namespace gdr

extern "C" gdr_status gdr_prefill_noalloc(const gdr_shape* shape, const void* q, const void* k,
                                          const void* v, const float* alpha, const float* beta,
                                          const float* S0, const int32_t* cu_seqlens, void* out,
                                          float* S_final, void* stream) {
  if (!shape) return GDR_ERR_INVALID_ARG;
  if (shape->n_seqs > GDR_NOALLOC_MAX_SEQS) return GDR_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (cudaGetSymbolAddress(&scratch, gdr::g_noalloc_scratch) != cudaSuccess) return GDR_ERR_CUDA;
  return gdr::prefill_launch(shape, q, k, v, alpha, beta, S0, cu_seqlens, out, S_final, scratch,
                             gdr::kNoAllocScratchBytes, stream);
}
