// prefill_tc.cu -- chunked prefill of the gated delta rule on the 5th-generation tensor cores
// (tcgen05.mma, bf16 operands in shared memory, fp32 accumulators in TMEM, inputs staged by
// TMA), d_k = d_v = 128, chunks of C = 64 tokens, one CTA per chain (the kernels with helper CTAs
// for few chains are in prefill_cluster.cu and prefill_queue.cu; linear attention, which needs
// none of the per-chunk preparation, in linear_tc.cu).  This file also holds the tensor-map
// set-up and the dispatch between those kernels.
//
// Chunk algebra (derived from the recurrence; the alpha = 1 case is the per-chunk triangular
// solve of engineermaxxing "From GPT-2 to Kimi K3: one memory, seven eviction policies" §04e-§04f
// and heqinghuang "gpt2-to-kimi" §10; the decay folded through it is the running product of the
// gates, engineermaxxing §05d and heqinghuang §11, one factor per key channel as in dev.to "From
// GPT-2 to Kimi K3: How Language Models Learned to Manage Memory" §5).  Chunk of n <= 64 tokens,
// local index r, entering state S (d_k x d_v fp32), Gam_r = prod_{m<=r} alpha_m per key channel:
//   K~ = K * Gam,  Q~ = Q * Gam,  Kr = K / Gam,  K^ = K * Gam_n / Gam,  gamma = Gam_n
//   [A'; M] = [K~; Q~] Kr^T                  one M = 128 MMA (decay-weighted Gram matrices)
//   A = diag(beta) strict_lower(A'),  M <- lower(M)
//   T' = (I + A)^-1 diag(beta)               blockwise forward substitution (fp32, SIMT)
//   W = T' K~,  U = T' V - W S               MMAs; the - W S term accumulates onto T' V in TMEM
//   O = Q~ S + M U                           MMAs accumulating in one TMEM region
//   S <- Diag(gamma) S + K^^T U              fp32 state kept in TMEM, faded in place
// The split Gam_r / Gam_j of the pair decay is exact; it is used while the chunk's decay keeps
// min_c Gam_n[c] above e^-40, so every factor and product stays far inside the bf16 / fp32
// range.  Chunks with stronger decay (an alpha = 0 reset, say) take log-gate prefix sums
// G = sum max(log alpha, -60) and form A' and M from direct pairwise exponentials (exact,
// slower).
//
// Mapping: one CTA (8 warps) per (sequence, head, block of DV value columns); columns of S are
// independent, so the value dimension splits across CTAs.  Warp w reads TMEM lane quarter w & 3
// and the column half w >> 2 of every accumulator: thread t owns lane t & 127, i.e. key channel
// t & 127 of the state or token row t & 127 of the M = 128 Gram accumulator; M = 64
// accumulators (token rows) occupy lanes 32q + [0, 16) for rows 16q + [0, 16).  q, k, alpha and
// v tiles of the next chunk are fetched by TMA while the current chunk computes.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "tc_common.cuh"

namespace gdr {
namespace {

using namespace umma;
using namespace tc;

template <int DV>
struct TcSmem {
  // TMA staging of the chunk's inputs
  static constexpr uint32_t QIN = 0;                // [64][128] bf16 row-major     16 KB
  static constexpr uint32_t KIN = QIN + 16384;      // [64][128] bf16 row-major     16 KB
  static constexpr uint32_t AIN = KIN + 16384;      // [64][128] fp32 row-major     32 KB
  static constexpr uint32_t VIN = AIN + 32768;      // [64 tok][DV] SW128 (MN-major B)
  // bf16 operand tiles (128B swizzle)
  static constexpr uint32_t KQ = VIN + DV * 128;    // [K~ ; Q~] 128 x 128, K-major  32 KB
  static constexpr uint32_t KR = KQ + 32768;        // Kr 64 x 128, K-major          16 KB
  static constexpr uint32_t KH = KR + 16384;        // K^ [tok][ch] (MN-major A)     16 KB
  static constexpr uint32_t TT = KH + 16384;        // T' 64 x 64, K-major            8 KB
  static constexpr uint32_t MM = TT + 8192;         // M  64 x 64, K-major            8 KB
  static constexpr uint32_t WW = MM + 8192;         // W  64 x 128, K-major          16 KB
  static constexpr uint32_t UU = WW + 16384;        // U  [tok][DV] (MN-major B)
  static constexpr uint32_t SS = UU + DV * 128;     // S  [d_k][DV] (MN-major B)
  static constexpr uint32_t BETA = SS + DV * 256;   // beta [64]
  static constexpr uint32_t ALPHA = BETA + 256;     // scalar gates [64]
  static constexpr uint32_t GAM = ALPHA + 256;      // gamma [128]
  static constexpr uint32_t RED = GAM + 512;        // reductions [8]
  static constexpr uint32_t GS = RED + 64;          // scalar gates: log prefix sums [64]
  static constexpr uint32_t BARS = GS + 256;        // 4 mbarriers + TMEM slot
  static constexpr uint32_t END = BARS + 64;
  static constexpr size_t bytes = END + 1024;       // + alignment slack
  // fp32 scratch of the solve, in tiles that are dead while it runs
  static constexpr uint32_t SA = KR;                // A [64][64]  (Kr is consumed by then)
  static constexpr uint32_t ST32 = WW;              // T [64][64]  (W is written later)
  static constexpr uint32_t SX = UU;                // [32][32] (U is written later)
  static constexpr uint32_t TOT = WW;               // gate carries [32][128] (W later)
  static constexpr uint32_t DIAGP = UU;             // q_r . k_r partials [64][16] (U later)
  static_assert(bytes <= 232448, "shared memory per CTA");
  static_assert(DV * 128 >= 32 * 32 * 4, "block scratch fits in U");
};

// ERASE = false: gated linear attention (no correction, no beta): stages 3-4 are skipped and V
// itself is the U of the state pass.
template <int DV, bool CHANNEL, bool ERASE = true>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ TcMaps maps, const PrefillArgs a) {
  using L = TcSmem<DV>;
  constexpr int NB = kD / DV;
  constexpr int DH = DV / 2;  // accumulator columns per warp half
  constexpr bool kAlphaTile = CHANNEL;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~(uintptr_t)1023);
  float* sBeta = reinterpret_cast<float*>(sm + L::BETA);
  float* sAlpha = reinterpret_cast<float*>(sm + L::ALPHA);
  float* sGam = reinterpret_cast<float*>(sm + L::GAM);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
  uint64_t* bar_qk = bars + 1;
  uint64_t* bar_a = bars + 2;
  uint64_t* bar_v = bars + 3;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 4);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int H = a.H;
  const int rank = blockIdx.x / (H * NB);
  const int rem = blockIdx.x % (H * NB);
  const int h = rem / NB, vb = rem % NB;
  const int seq = a.order ? a.order[rank] : rank;
  int64_t t0, t1;
  if (!seq_range(a, seq, t0, t1)) return;
  __nv_bfloat16* __restrict__ out = static_cast<__nv_bfloat16*>(a.out);
  const int vc0 = vb * DV;
  const size_t sidx = ((size_t)seq * H + h) * kD * kD;

  if (warp == 0) tmem_alloc(tslot, kTmemCols);
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(bars + i, 1);
    fence_mbar_init();
    prefetch_tmap(&maps.q);
    prefetch_tmap(&maps.k);
    prefetch_tmap(&maps.v);
    if (kAlphaTile) prefetch_tmap(&maps.alpha);
  }
  cta_sync_tc();
  TcCtx x = make_ctx(sm, *tslot, bars + 0);
  x.prologue = a.prologue;
  uint32_t ph_qk = 0, ph_a = 0, ph_v = 0;
  bool failed = false;

  auto issue_qk = [&](int64_t tc) {
    if (tid == 0) {
      mbar_expect_tx(bar_qk, 2 * 16384);
      tma_load_3d(sm + L::QIN, &maps.q, 0, h, (int)tc, bar_qk);
      tma_load_3d(sm + L::KIN, &maps.k, 0, h, (int)tc, bar_qk);
    }
  };
  auto issue_a = [&](int64_t tc) {
    if (kAlphaTile && tid == 0) {
      mbar_expect_tx(bar_a, 32768);
      tma_load_3d(sm + L::AIN, &maps.alpha, 0, h, (int)tc, bar_a);
    }
  };
  auto issue_v = [&](int64_t tc) {
    if (tid == 0) {
      mbar_expect_tx(bar_v, DV * 128);
#pragma unroll
      for (int s = 0; s < DV / 64; ++s)
        tma_load_3d(sm + L::VIN + s * 8192, &maps.v, vc0 + 64 * s, h, (int)tc, bar_v);
    }
  };
  // per-token scalars of a chunk (beta, scalar alpha), read one chunk ahead into registers
  auto load_scalars = [&](int64_t tc, float& b, float& al) {
    b = 0.f;
    al = 1.f;
    if (tid < kC && tc + tid < t1) {
      const size_t o = (size_t)(tc + tid) * H + h;
      if (ERASE) b = a.beta[o];
      if (!CHANNEL) al = a.alpha[o];
    }
  };

  if (t0 < t1) {
    issue_qk(t0);
    issue_a(t0);
    issue_v(t0);
  }
  s_init<DH>(x, a.S0 ? a.S0 + sidx + (size_t)x.lrow * kD + vc0 : nullptr, sm + L::SS);
  zero_upper_tp(sm + L::TT, tid);
  float nb_beta, nb_alpha;
  load_scalars(t0, nb_beta, nb_alpha);

  // operand views of the state pass
  const Opnd opQ{x.sb + L::KQ + 8192, 16384, false};  // Q~ rows as K-major A (M = 64)
  const Opnd opKH{x.sb + L::KH, 8192, true};          // K^ as MN-major A (M = 128 channels)
  const Opnd opM{x.sb + L::MM, 8192, false};
  const Opnd opW{x.sb + L::WW, 8192, false};
  const Opnd opV{x.sb + L::VIN, 8192, true};          // V as MN-major B (K = tokens)
  const Opnd opU{x.sb + L::UU, 8192, true};           // U as MN-major B (K = tokens)
  const Opnd opS{x.sb + L::SS, 16384, true};          // S as MN-major B (K = key channels)
  const uint32_t id_v = idesc_bf16(64, DV, false, false, true);
  const uint32_t id_negw = idesc_bf16(64, DV, true, false, true);
  const uint32_t id_s = idesc_bf16(128, DV, false, true, true);

#pragma unroll 1
  for (int64_t tc = t0; tc < t1 && !failed; tc += kC) {
    const int n = (int)((t1 - tc) < (int64_t)kC ? (t1 - tc) : (int64_t)kC);
    const int64_t tn = tc + kC;  // next chunk

    if (tid < kC) {  // (the layer prologue maps the live tokens' raw gates here, not at the load)
      const bool pro = a.prologue && tid < n;
      sBeta[tid] = pro && ERASE ? sigmoid_ftz(nb_beta) : nb_beta;
      sAlpha[tid] = pro && !CHANNEL ? sigmoid_ftz(nb_alpha) : nb_alpha;
    }
    if (tn < t1) load_scalars(tn, nb_beta, nb_alpha);
    if (!wait_bar(bar_qk, ph_qk)) { failed = true; break; }
    if (kAlphaTile && !wait_bar(bar_a, ph_a)) { failed = true; break; }

    // 1. gates and operand tiles
    const bool safe = gate_stage<L, CHANNEL>(x, n);
    fence_async_smem();
    cta_sync_tc();
    if (safe && tn < t1) {  // q, k and alpha tiles are consumed: fetch the next chunk's
      issue_qk(tn);
      issue_a(tn);
    }
    // 2. decay-weighted Gram matrices [A'; M]
    if (!gram_stage<L, CHANNEL>(x, n, safe)) { failed = true; break; }
    if (!safe && tn < t1) {
      issue_qk(tn);
      issue_a(tn);
    }
    // the chunk's V tile (rows past the end of the sequence zeroed)
    if (!wait_bar(bar_v, ph_v)) { failed = true; break; }
    zero_v_tail<DV>(x, sm + L::VIN, n);

    if constexpr (ERASE) {
      // 3. T' = (I + A)^-1 diag(beta);  4. W = T' K~ and U~ = T' V
      solve_stage<L>(x);
      if (!w_stage<L>(x, true, opV, id_v)) { failed = true; break; }
      if (tn < t1) issue_v(tn);  // V is consumed
      w_epilogue<L>(x);
    } else {
      fence_async_smem();  // the zeroed V tail, before the MMAs read V
    }
    cta_sync_tc();

    // 5. U = U~ - W S and O = Q~ S; the state master is faded meanwhile
    if (warp == 0) {
      if (ERASE) mma_run<kD>(x.tm + kColU, opW, opS, id_negw, true);
      mma_run<kD>(x.tm + kColWO, opQ, opS, id_v, false);
      mma_commit_elect(x.bar_mma);
    }
    gamma_fade<DH>(x, sGam);
    // the MMA waits of stages 5-6 are per thread; one that gave up is remembered and the CTA
    // agrees on it at the chunk's closing barrier
    bool bad = !mbar_wait(x.bar_mma, x.ph_mma, kWaitNs);
    x.ph_mma ^= 1u;
    fence_after_sync();
    if (ERASE) u_epilogue<DH>(x, sm + L::UU);
    cta_sync_tc();

    // 6. O += M U and S += K^^T U (U = V without the correction)
    const Opnd& opUse = ERASE ? opU : opV;
    if (warp == 0) {
      mma_run<kC>(x.tm + kColWO, opM, opUse, id_v, true);
      mma_run<kC>(x.tm + kColS, opKH, opUse, id_s, true);
      mma_commit_elect(x.bar_mma);
    }
    bad |= !mbar_wait(x.bar_mma, x.ph_mma, kWaitNs);
    x.ph_mma ^= 1u;
    fence_after_sync();
    if (!ERASE && tn < t1) issue_v(tn);  // V is consumed
    o_epilogue<DH>(x, out, tc, n, H, h, vc0, kColWO, static_cast<const __nv_bfloat16*>(a.og));
    s_epilogue<DH>(x, sm + L::SS);
    fence_before_sync();
    if (__syncthreads_or(bad)) { failed = true; break; }
    fence_after_sync();
  }

  if (failed) {
    if (tid == 0) report(a, GDR_DEVCHECK_TIMEOUT);
    // let copies already in flight land before the shared memory is released
    mbar_wait(bar_qk, ph_qk, kWaitNs);
    if (kAlphaTile) mbar_wait(bar_a, ph_a, kWaitNs);
    mbar_wait(bar_v, ph_v, kWaitNs);
  } else if (a.S_final) {
    s_final<DH>(x, a.S_final + sidx + (size_t)x.lrow * kD + vc0);
  }
  cta_sync_tc();
  if (warp == 0) tmem_dealloc(x.tm, kTmemCols);
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [T][H][128] tensor, box of `box_x` channels x 1 head x 64 tokens.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elt, int H,
              int64_t T, int box_x, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * elt, (cuuint64_t)H * kD * elt};
  const cuuint32_t box[3] = {(cuuint32_t)box_x, 1, (cuuint32_t)kC};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace tc {
bool make_tc_maps(const gdr_shape& sh, const PrefillArgs& a, bool linear, TcMaps* maps) {
  memset(maps, 0, sizeof(*maps));
  const int H = sh.H;
  const int64_t T = sh.total_tokens;
  bool ok = make_map(&maps->q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, kD,
                     CU_TENSOR_MAP_SWIZZLE_NONE) &&
            make_map(&maps->k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, kD,
                     CU_TENSOR_MAP_SWIZZLE_NONE) &&
            make_map(&maps->v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  if (ok && linear)
    ok = make_map(&maps->k_sw, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, 64,
                  CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map(&maps->q_sw, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, 64,
                  CU_TENSOR_MAP_SWIZZLE_128B);
  if (ok && a.og)
    ok = make_map(&maps->og, a.og, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, kD,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
  if (ok && !linear && sh.gate == GDR_GATE_CHANNEL)
    ok = make_map(&maps->alpha, a.alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H, T, kD,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
  return ok;
}
}  // namespace tc

namespace {

template <int DV, bool CHANNEL, bool ERASE>
cudaError_t launch_one(const gdr_shape& sh, const PrefillArgs& a, const TcMaps& maps,
                       cudaStream_t s) {
  auto kern = prefill_tc_kernel<DV, CHANNEL, ERASE>;
  const size_t smem = TcSmem<DV>::bytes;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)sh.n_seqs * (unsigned)sh.H * (unsigned)(kD / DV);
  kern<<<grid, kThreads, smem, s>>>(maps, a);
  return cudaGetLastError();
}

template <int DV>
cudaError_t launch_dv(const gdr_shape& sh, const PrefillArgs& a, const TcMaps& maps, bool erase,
                      cudaStream_t s) {
  const bool ch = sh.gate == GDR_GATE_CHANNEL;
  if (!erase)
    return ch ? launch_one<DV, true, false>(sh, a, maps, s)
              : launch_one<DV, false, false>(sh, a, maps, s);
  return ch ? launch_one<DV, true, true>(sh, a, maps, s) : launch_one<DV, false, true>(sh, a, maps, s);
}

}  // namespace

bool prefill_tc_supported(const gdr_shape& sh) {
  return sh.dtype == GDR_BF16 && sh.d_k == kD && sh.d_v == kD &&
         !(sh.flags & GDR_FLAG_FORCE_SIMT) && sh.total_tokens > 0 &&
         sh.total_tokens < ((int64_t)1 << 31) && encode_fn() != nullptr;
}

cudaError_t launch_prefill_tc(const gdr_shape& sh, const PrefillArgs& a, int kind,
                              cudaStream_t s) {
  const bool linear = kind == kKindLinear || kind == kKindNormLinear;
  TcMaps maps;
  if (!tc::make_tc_maps(sh, a, linear, &maps)) return cudaErrorInvalidValue;
  if (linear) return tc::launch_linear_tc(sh, a, maps, kind == kKindNormLinear, s);  // linear_tc.cu
  const long pairs = (long)sh.n_seqs * sh.H;
  // gated linear attention: without stages 3-4; helper CTAs in clusters where they fit, else
  // the one-CTA kernel
  if (kind == kKindGatedLinear) {
    const int ncl = (sh.flags & GDR_FLAG_NO_CLUSTER) ? 1 : tc::cluster_size_for(sh);
    if (ncl > 1) return tc::launch_prefill_cluster(sh, a, maps, ncl, false, s);
    return pairs >= 120 ? launch_dv<128>(sh, a, maps, false, s) : launch_dv<64>(sh, a, maps, false, s);
  }
  // few (sequence, head) chains: helper CTAs prepare the chunks of each chain, in clusters (the
  // operands cross over DSMEM) or, when clusters would give a chain a single helper, from a
  // work queue over every SM (the operands cross through L2 rings in the workspace)
  if (!(sh.flags & GDR_FLAG_NO_CLUSTER)) {
    const int ncl = tc::cluster_size_for(sh);
    const int G = tc::queue_grid_for(sh, a);
    if (G > 0 && (ncl <= 2 || (sh.flags & GDR_FLAG_PREFER_QUEUE)))
      return tc::launch_prefill_queue(sh, a, maps, G, s);
    if (ncl > 1) return tc::launch_prefill_cluster(sh, a, maps, ncl, true, s);
  }
  // value-column split: enough CTAs to cover the SMs when there are few (sequence, head) pairs
  if (pairs >= 120) return launch_dv<128>(sh, a, maps, true, s);
  return launch_dv<64>(sh, a, maps, true, s);
}

}  // namespace gdr
