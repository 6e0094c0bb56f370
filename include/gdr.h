/*
 * gdr.h -- C ABI of libgdr: the gated delta rule (Kimi Delta Attention / Gated DeltaNet /
 * DeltaNet / linear attention) on one GB300 GPU (sm_103a).
 *
 * The update, per (sequence, head), token t, with state S (d_k x d_v, fp32, row i = key
 * channel i; read of a key is S^T k):
 *
 *     S_t = Diag(alpha_t) S_{t-1} + beta_t k_t (v_t - (Diag(alpha_t) S_{t-1})^T k_t)^T
 *     o_t = S_t^T q_t
 *
 * Sources (web pages; sections as numbered on each page):
 *   dev.to "From GPT-2 to Kimi K3: How Language Models Learned to Manage Memory", §3 (delta
 *     rule), §4 (Gated DeltaNet: fade, then read, then correct), §5 (one retention factor per
 *     key channel, i.e. per row of S);
 *   engineermaxxing "From GPT-2 to Kimi K3: one memory, seven eviction policies", §03b
 *     (read / subtract / write; state convention), §04b-§04f (chunked form and the triangular
 *     solve), §05c-§05d (gate, survival products), §06b (per-channel gate);
 *   heqinghuang "gpt2-to-kimi", §09-§11 (recurrent form, chunked DeltaNet, Gated DeltaNet);
 *   kylehh "Kimi K3: From KV Cache to Selective Memory", §5-§8.
 * The decay is applied before the read (the per-channel code of engineermaxxing §06b, dev.to
 * §4-§5); with a scalar gate the two orders coincide.
 *
 * Conventions shared by every call
 *   - Pointers are DEVICE pointers unless stated otherwise; the caller owns every buffer.  The
 *     library allocates nothing, keeps no state between calls and never frees caller memory
 *     (three stated exceptions: the per-device error word of gdr_query_device_status,
 *     gdr_prefill_noalloc's fixed scratch array and gdr_prefill_host's internal copy streams).
 *   - Layouts are packed and token-major, row-major, no padding:
 *       q, k            [T_total, H, d_k]   dtype = shape->dtype
 *       v, out          [T_total, H, d_v]   dtype = shape->dtype
 *       alpha           [T_total, H, d_k] fp32 (GDR_GATE_CHANNEL) or [T_total, H] fp32 (SCALAR)
 *       beta            [T_total, H] fp32
 *       S0, S_final     [n_seqs, H, d_k, d_v] fp32 (row = key channel)
 *       cu_seqlens      [n_seqs + 1] int32 offsets into the token axis (device memory)
 *   - alpha is the retention factor in [0, 1] (0 = reset); the kernels clamp log(alpha) at -60
 *     per token, which is a reset to within fp32.  beta is the write strength (any real value;
 *     (0, 1) in the method).  q and k are used as given (no normalisation, no 1/sqrt(d) scale).
 *   - Supported: d_k = d_v in {64, 128}; dtype GDR_F32 (fp32 FFMA path) or GDR_BF16 (tensor-core
 *     path for d = 128, fp32 FFMA otherwise).  Other shapes return GDR_ERR_UNSUPPORTED.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL = the legacy
 *     default stream).  Argument errors are returned synchronously, before any launch.  Launch
 *     failures return GDR_ERR_CUDA.  Checks that need device data (cu_seqlens monotone and within
 *     total_tokens) run on the device and record the first failure in the workspace status word,
 *     read with gdr_workspace_status(), and in the library's error word on that device, read
 *     with gdr_query_device_status(); sequences that fail the check are skipped.
 *   - 16-byte alignment is required for every pointer (GDR_ERR_INVALID_ARG otherwise).
 */
#ifndef GDR_H_
#define GDR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDR_OK = 0,
  GDR_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, bad size, bad enum, workspace too small */
  GDR_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. d_k != d_v, d not 64/128) */
  GDR_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
  GDR_ERR_DEVICE_CHECK = 4  /* a device-side check failed (gdr_query_device_status) */
} gdr_status;

typedef enum { GDR_F32 = 0, GDR_BF16 = 1 } gdr_dtype; /* dtype of q, k, v and out */
typedef enum { GDR_GATE_SCALAR = 0, GDR_GATE_CHANNEL = 1 } gdr_gate;

/* Device-side check codes written to the workspace status word (0 = no failure). */
enum {
  GDR_DEVCHECK_OK = 0,
  GDR_DEVCHECK_SEQLENS = 1, /* cu_seqlens not monotone, negative, or beyond total_tokens */
  GDR_DEVCHECK_TIMEOUT = 2  /* a tensor-core wait gave up (the kernel unwound; results invalid) */
};

typedef struct {
  int32_t n_seqs;       /* number of sequences (>= 1) */
  int32_t H;            /* heads (>= 1) */
  int64_t total_tokens; /* T_total = length of the packed token axis (>= 0) */
  int32_t d_k;          /* key / query channels = rows of S */
  int32_t d_v;          /* value channels = columns of S */
  int32_t dtype;        /* gdr_dtype of q, k, v, out */
  int32_t gate;         /* gdr_gate layout of alpha (ignored by gdr_linear_attn) */
  int32_t chunk_size;   /* 0 = the kernel's choice; otherwise must equal a supported size */
  int32_t flags;        /* GDR_FLAG_* (0 = default) */
} gdr_shape;

/* Force the fp32 FFMA chunked path even where a tensor-core path exists (for cross-checks). */
#define GDR_FLAG_FORCE_SIMT 1
/* On the tensor-core path, run the one-CTA-per-chain kernel even where a kernel with helper CTAs
 * that prepare each chain's chunks (work queue or clusters) would be chosen (for cross-checks). */
#define GDR_FLAG_NO_CLUSTER 2
/* Run the work-queue kernel wherever the workspace holds its operand rings, also where the
 * clustered kernel would be chosen (for cross-checks). */
#define GDR_FLAG_PREFER_QUEUE 4
/* The layer prologue on load (heqinghuang "gpt2-to-kimi" §09: unit-length silu queries and keys,
 * beta a sigmoid of its projection; engineermaxxing "From GPT-2 to Kimi K3" §05c and §06b: the
 * decay a sigmoid of its projection, per head or per channel).  q, k, alpha and beta then hold
 * the layer's raw projections xq, xk, a, b (same dtypes and layouts as the rule's inputs), and
 * every kernel forms q = xq * sigmoid(xq) / max(||.||_2, 1e-12) over the d_k channels of each
 * (token, head) (likewise k), alpha = sigmoid(a) and beta = sigmoid(b) as it loads them; the
 * inputs are not written.  Accepted by gdr_prefill, gdr_prefill_output_gate,
 * gdr_gated_linear_attn (no beta), gdr_decode_step and gdr_prefill_host; gdr_linear_attn returns
 * GDR_ERR_UNSUPPORTED.  On the tensor-core paths the normalised q and k are rounded to bf16 (the
 * operand type) before use; the fp32 paths keep them in fp32. */
#define GDR_FLAG_LAYER_PROLOGUE 8

/*
 * gdr_prefill -- chunked, packed variable-length prefill of the gated delta rule.
 * engineermaxxing §04e-§04f (per-chunk triangular solve), heqinghuang §10-§11 (chunked DeltaNet
 * with the running decay products folded in), dev.to §5 (per-channel gate).
 *   q, k, v, alpha, beta, out: as above (out must not alias an input).
 *   S0:         initial states, or NULL for zeros.
 *   cu_seqlens: NULL means one sequence of total_tokens tokens (then n_seqs must be 1).
 *   S_final:    final states, or NULL.  S_final may equal S0 (in-place hand-off).
 *   workspace:  device scratch of gdr_prefill_workspace_size(shape) bytes, 256-byte aligned;
 *               its contents need not be initialised; calls that overlap on the GPU must use
 *               different workspaces.  A smaller workspace is accepted down to 256 bytes plus
 *               4 * n_seqs rounded up to 256; it disables the work-queue tensor-core prefill
 *               (at most 76 (sequence, head) chains, bf16, d = 128), and a slower kernel runs
 *               instead with the same results.
 * Empty sequences (length 0) produce no output and S_final = S0 (or zeros).
 */
gdr_status gdr_prefill(const gdr_shape* shape, const void* q, const void* k, const void* v,
                       const float* alpha, const float* beta, const float* S0,
                       const int32_t* cu_seqlens, void* out, float* S_final, void* workspace,
                       size_t workspace_bytes, void* stream);

/* Workspace bytes gdr_prefill / gdr_linear_attn use for this shape (0 if n_seqs or H < 1): the
 * status word, the visiting order and, for bf16 d = 128 shapes of at most 76 (sequence, head)
 * chains, the work-queue prefill's flags and 6 operand slots of 74752 bytes per chain. */
size_t gdr_prefill_workspace_size(const gdr_shape* shape);

/*
 * gdr_normalized_linear_attn -- normalised phi-linear attention, chunked, packed varlen
 * (heqinghuang "gpt2-to-kimi" §07; engineermaxxing "From GPT-2 to Kimi K3" §02g):
 *   phi(x) = elu(x) + 1   (x + 1 for x > 0, e^x otherwise; applied to q and k by the kernel)
 *   S <- S + phi(k_t) v_t^T,   z <- z + phi(k_t),   o_t = S^T phi(q_t) / (phi(q_t) . z + eps)
 * per (sequence, head), the read after the write.  q, k, v, out, S0, S_final, cu_seqlens,
 * workspace: as gdr_prefill (no alpha, no beta; shape->gate ignored).  z0: entering
 * normalisers [n_seqs, H, d_k] fp32 or NULL for zeros; z_final: final normalisers or NULL; z_final
 * must not be z0.  eps: a finite value >= 0 (0 divides by phi(q) . z, which is > 0 from the
 * first token on unless phi underflows).  GDR_FLAG_LAYER_PROLOGUE is unsupported here.
 */
gdr_status gdr_normalized_linear_attn(const gdr_shape* shape, const void* q, const void* k,
                                      const void* v, float eps, const float* S0, const float* z0,
                                      const int32_t* cu_seqlens, void* out, float* S_final,
                                      float* z_final, void* workspace, size_t workspace_bytes,
                                      void* stream);

/*
 * gdr_gated_linear_decode_step -- one token per sequence of gated linear attention, state
 * updated in place (engineermaxxing "From GPT-2 to Kimi K3" §05b; per key channel as dev.to §5):
 *   S <- Diag(alpha) S + k v^T,   o = S^T q.
 * Arguments as gdr_decode_step without beta.  GDR_FLAG_LAYER_PROLOGUE is accepted (q, k, alpha
 * raw projections).
 */
gdr_status gdr_gated_linear_decode_step(const gdr_shape* shape, const void* q, const void* k,
                                        const void* v, const float* alpha, float* S_inout,
                                        void* out, void* stream);

/*
 * gdr_normalized_linear_decode_step -- one token per sequence of normalised phi-linear attention
 * (heqinghuang "gpt2-to-kimi" §07; engineermaxxing §02g's decode step), state and normaliser
 * updated in place:
 *   S <- S + phi(k) v^T,   z <- z + phi(k),   o = S^T phi(q) / (phi(q) . z + eps).
 * q, k, v, out: [n_seqs, H, d] in shape->dtype; S_inout [n_seqs, H, d_k, d_v] fp32; z_inout
 * [n_seqs, H, d_k] fp32 (device, 16-byte aligned, caller-owned, not aliasing each other or out);
 * shape->total_tokens must equal shape->n_seqs; eps finite and >= 0.  One HBM-bound kernel.
 */
gdr_status gdr_normalized_linear_decode_step(const gdr_shape* shape, const void* q, const void* k,
                                             const void* v, float eps, float* S_inout,
                                             float* z_inout, void* out, void* stream);

/*
 * gdr_layer_prologue -- the layer prologue as a pass of its own (the maps that
 * GDR_FLAG_LAYER_PROLOGUE applies inside the kernels; heqinghuang "gpt2-to-kimi" §09,
 * engineermaxxing "From GPT-2 to Kimi K3" §05c and §06b):
 *   q = silu(xq) / max(||silu(xq)||_2, 1e-12) over the d_k channels of each (token, head),
 *   k likewise, alpha = sigmoid(a), beta = sigmoid(b);   silu(x) = x sigmoid(x).
 *   xq, xk -> q, k: [T, H, d_k] in shape->dtype (fp32 math, one rounding to the dtype).
 *   a -> alpha: [T, H, d_k] (shape->gate = GDR_GATE_CHANNEL) or [T, H] fp32; both NULL to skip.
 *   b -> beta:  [T, H] fp32; both NULL to skip.
 * Uses shape->H, total_tokens, d_k (= d_v, 64 or 128), dtype and gate.  Outputs may be their
 * own inputs (in place); otherwise they must not overlap an input.  All pointers device, 16-byte
 * aligned, caller-owned.  One kernel, bound by HBM bandwidth; asynchronous on `stream`.
 */
gdr_status gdr_layer_prologue(const gdr_shape* shape, const void* xq, const void* xk,
                              const float* a, const float* b, void* q, void* k, float* alpha,
                              float* beta, void* stream);

/*
 * gdr_decode_step -- one token per sequence, state updated in place.
 * engineermaxxing §06b (the per-channel code: decay per row, read, correct), heqinghuang §09.
 * shape->total_tokens must equal shape->n_seqs; cu_seqlens is implied (token n = sequence n).
 *   q, k [N, H, d_k]; v, out [N, H, d_v]; alpha [N, H, d_k] or [N, H]; beta [N, H];
 *   S_inout [N, H, d_k, d_v] fp32, read and overwritten with the new state.
 * One fused pass per state: the read of the faded state, the correction, the read-out and the
 * write-back use each element of S once.  No workspace is needed.
 */
gdr_status gdr_decode_step(const gdr_shape* shape, const void* q, const void* k, const void* v,
                           const float* alpha, const float* beta, float* S_inout, void* out,
                           void* stream);

/*
 * gdr_linear_attn -- plain (unnormalised) linear attention, the alpha = 1, no-erase case:
 * S_t = S_{t-1} + k_t v_t^T, o_t = S_t^T q_t; chunked as O = Q S + tril(Q K^T) V, S += K^T V.
 * engineermaxxing §03b (identity transition) and §04b (chunked form); heqinghuang §10.
 * No feature map, no normaliser, no beta.  Arguments as gdr_prefill (shape->gate ignored).
 */
gdr_status gdr_linear_attn(const gdr_shape* shape, const void* q, const void* k, const void* v,
                           const float* S0, const int32_t* cu_seqlens, void* out, float* S_final,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * gdr_prefill_output_gate -- gdr_prefill with the KDA layer's output gate applied as the outputs
 * are written: out = o * sigmoid(g), element by element.  dev.to §5 (Kimi K3 replaces the
 * low-rank output gate by a full-rank, input-dependent one); the sigmoid multiplied into the
 * output feature by feature follows heqinghuang §15's description of the attention layers' gate.
 *   g: gate pre-activations [T_total, H, d_v], dtype = shape->dtype, 16-byte aligned, not `out`.
 * Every other argument as gdr_prefill (bf16 outputs are gated after their rounding to bf16 on
 * the tensor-core path: one more bf16 rounding).
 */
gdr_status gdr_prefill_output_gate(const gdr_shape* shape, const void* q, const void* k,
                                   const void* v, const float* alpha, const float* beta,
                                   const void* g, const float* S0, const int32_t* cu_seqlens,
                                   void* out, float* S_final, void* workspace,
                                   size_t workspace_bytes, void* stream);

/*
 * gdr_gated_linear_attn -- gated linear attention, the decayed additive update without the
 * delta rule's erase term: S_t = Diag(alpha_t) S_{t-1} + k_t v_t^T, o_t = S_t^T q_t.
 * engineermaxxing §05b (the scalar-gated additive update, RetNet / Mamba-2 / GLA lineage),
 * heqinghuang §11 (decay applied to the state before the write); one gate per key channel
 * (row of S) as in dev.to §5.  Chunked with the gated rule's decay products and no triangular
 * solve: O = (Q * Gamma) S + M V, S <- Diag(Gamma_n) S + (K * Gamma_n / Gamma)^T V.
 * Arguments as gdr_prefill without beta; alpha per channel [T, H, d_k] or scalar [T, H]
 * (shape->gate).
 */
gdr_status gdr_gated_linear_attn(const gdr_shape* shape, const void* q, const void* k,
                                 const void* v, const float* alpha, const float* S0,
                                 const int32_t* cu_seqlens, void* out, float* S_final,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * gdr_workspace_status -- synchronise `stream`, read the device-check word of a workspace used
 * by gdr_prefill / gdr_linear_attn into *code (a GDR_DEVCHECK_* value) and clear it.
 * Returns GDR_OK, or GDR_ERR_CUDA if the copy or the synchronisation failed.
 */
gdr_status gdr_workspace_status(void* workspace, void* stream, int32_t* code);

/*
 * gdr_query_device_status -- synchronise `stream`, then take (read and clear, atomically) the
 * library's error word on the current device: the first device-side check failure recorded by
 * any prefill-like call on this device since the previous query (GDR_DEVCHECK_SEQLENS from the
 * cu_seqlens check, GDR_DEVCHECK_TIMEOUT from a bounded wait that gave up).  The pages define no
 * interface; this is the error path of the library.  The word is per device and shared by all
 * calls on it (the one piece of state the library keeps besides the two listed above); the
 * failing call's own code is also in its workspace word (gdr_workspace_status).
 * Returns GDR_OK (no failure recorded), GDR_ERR_DEVICE_CHECK (a failure was recorded and is now
 * cleared) or GDR_ERR_CUDA (the synchronisation, the exchange or the copy failed).
 */
gdr_status gdr_query_device_status(void* stream);

/*
 * gdr_check_wait_timeout -- exercises the library's failure detection without a GPU fault.  (The
 * pages have no counterpart: this belongs to the library's error path.)  Launches one warp that
 * waits on an mbarrier which nothing completes, with the bounded wait every tensor-core kernel
 * uses for its MMA, copy and hand-over barriers, given up after `limit_ns` nanoseconds.  The
 * timeout is recorded as a kernel's would be: GDR_DEVCHECK_TIMEOUT in the workspace word (if it
 * was 0) and in the library's per-device error word, so gdr_workspace_status and
 * gdr_query_device_status then report it; the kernel returns normally and the context stays
 * usable.  Asynchronous on `stream`.
 *   workspace  device, >= 256 bytes, 256-byte aligned (only its status word is written)
 *   limit_ns   1 .. 10,000,000,000 (10 s)
 * Returns GDR_OK, GDR_ERR_INVALID_ARG (null or unaligned workspace, limit out of range) or
 * GDR_ERR_CUDA (the launch failed).
 */
gdr_status gdr_check_wait_timeout(void* workspace, uint64_t limit_ns, void* stream);

/*
 * gdr_prefill_noalloc -- gdr_prefill for callers that cannot provide a workspace.  (The pages
 * have no counterpart: this is a property of the library interface, not of the method.)
 *
 * For callers whose device memory is fully budgeted (by a host framework's allocator or a
 * static memory plan), so that they have no scratch buffer to pass and may not call cudaMalloc
 * (which can also synchronise the device).  Arguments and results are those of gdr_prefill
 * without the workspace; the call allocates and frees nothing.  Its scratch is a fixed array in
 * the library's device memory, sized for at most GDR_NOALLOC_MAX_SEQS sequences (larger n_seqs
 * returns GDR_ERR_UNSUPPORTED), held on every GPU that loads the library until the process
 * exits.
 *   - Every call looks up the array's device address on the current device
 *     (cudaGetSymbolAddress); the first call on a device may also load the library's device
 *     code there, so make that first call before any stream capture.
 *   - Every call shares the array and leaves its contents behind; each call rewrites what it
 *     uses, but calls that overlap on the GPU (other streams, other host threads) race on it:
 *     serialise them.
 *   - The device-check word of this entry point is internal: cu_seqlens failures skip the
 *     offending sequences but cannot be read back; validate cu_seqlens before the call.
 */
#define GDR_NOALLOC_MAX_SEQS 4096
gdr_status gdr_prefill_noalloc(const gdr_shape* shape, const void* q, const void* k,
                               const void* v, const float* alpha, const float* beta,
                               const float* S0, const int32_t* cu_seqlens, void* out,
                               float* S_final, void* stream);

/*
 * gdr_prefill_host -- gdr_prefill on arrays in HOST memory, with the host<->device copies inside
 * the call and overlapped with the kernels.  The result is that of gdr_prefill (same chunking,
 * same kernels): the pages define the operation (see gdr_prefill); how its inputs reach the GPU
 * is a property of this library, which the pages do not discuss.
 *
 * The packed token axis is cut into pieces of about piece_tokens tokens (0: max(4096, T / 8));
 * a cut inside a sequence is moved forward to that sequence's next 64-token chunk boundary.
 * Each piece's inputs are copied in on an internal stream while the previous piece runs on
 * `stream`, and its outputs are copied out on a second internal stream while the next piece
 * runs; the states of all sequences stay on the device between pieces (in place).  With a
 * 1.35 GB KDA input the call is bound by the host link, not by the kernels.
 *   q, k, v, alpha, beta, S0, out, S_final: HOST pointers, layouts as gdr_prefill.  Page-locked
 *               (pinned) memory is needed for the copies to overlap; pageable memory works but the
 *               copies then serialise with the host.  S0 NULL = zeros; S_final may be NULL.
 *   cu_seqlens: HOST int32 offsets, or NULL for one sequence.  Checked on the host: cu[0] = 0,
 *               non-decreasing, cu[n_seqs] = total_tokens (GDR_ERR_INVALID_ARG otherwise).
 *   buffer:     DEVICE scratch of gdr_prefill_host_buffer_size(shape, piece_tokens) bytes,
 *               256-byte aligned (states, offsets, the prefill workspace, two staging sets).
 *   stream:     the prefill kernels run on it; the copies wait for the work already enqueued on
 *               it, and it waits for the last copy, so the call is ordered on `stream` like any
 *               other.  Host arrays must stay valid and unmodified until `stream` has passed the
 *               call.
 * Returns after enqueueing (asynchronous, like gdr_prefill).  The first call on a device creates
 * two non-blocking streams and a few events on it, kept until the process exits; calls from
 * several host threads on one device are serialised by a lock while they enqueue.  The
 * device-check word is internal (cu_seqlens is checked on the host instead).
 */
gdr_status gdr_prefill_host(const gdr_shape* shape, const void* q, const void* k, const void* v,
                            const float* alpha, const float* beta, const float* S0,
                            const int32_t* cu_seqlens, void* out, float* S_final,
                            int64_t piece_tokens, void* buffer, size_t buffer_bytes,
                            void* stream);

/* Device buffer bytes gdr_prefill_host needs for this shape and piece size (0 if the shape is
 * malformed). */
size_t gdr_prefill_host_buffer_size(const gdr_shape* shape, int64_t piece_tokens);

/* Static, human-readable name of a status. */
const char* gdr_status_string(gdr_status status);

#ifdef __cplusplus
}
#endif

#endif /* GDR_H_ */
