// prefill_tc.cu -- chunked prefill of the gated delta rule on the 5th-generation tensor cores
// (tcgen05.mma, bf16 operands in shared memory, fp32 accumulators in TMEM, inputs staged by
// TMA), d_k = d_v = 128, chunks of C = 64 tokens.  Also the plain linear-attention pass
// (alpha = 1, no erase).
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
// slower).  Linear attention: no gates (K~ = Kr = K^ = K, Q~ = Q), U = V, no solve.
//
// Mapping: one CTA (4 warps) per (sequence, head, block of DV value columns); columns of S are
// independent, so the value dimension splits across CTAs.  Thread t owns TMEM lane t: key
// channel t of the state, or token row t of the M = 128 Gram accumulator; M = 64 accumulators
// (token rows) occupy lanes 32w + [0, 16) for rows 16w + [0, 16).  q, k, alpha and v tiles of
// the next chunk are fetched by TMA while the current chunk computes.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "gdr_internal.cuh"
#include "umma.cuh"

namespace gdr {
namespace {

using namespace umma;

constexpr int kD = 128;          // d_k = d_v
constexpr int kC = 64;           // chunk
constexpr int kThreads = 128;    // 4 warps, one per TMEM lane quarter
constexpr float kSafeGamma = 4.2483543e-18f;  // e^-40
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s: a copy or MMA not done by then is a fault

// TMEM columns
constexpr uint32_t kColS = 0;     // fp32 state master, lanes = key channels
constexpr uint32_t kColU = 128;   // U accumulator (M = 64 layout)
constexpr uint32_t kColWO = 256;  // W accumulator, then O accumulator (M = 64 layout)
constexpr uint32_t kColAM = 384;  // [A'; M] accumulator (M = 128), 64 columns
constexpr uint32_t kTmemCols = 512;

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
  static constexpr uint32_t RED = GAM + 512;        // reductions
  static constexpr uint32_t BARS = RED + 64;        // 4 mbarriers + TMEM slot
  static constexpr uint32_t END = BARS + 64;
  static constexpr size_t bytes = END + 1024;       // + alignment slack
  // fp32 scratch of the solve, in tiles that are dead while it runs
  static constexpr uint32_t SA = KR;                // A [64][64]  (Kr is consumed by then)
  static constexpr uint32_t ST32 = WW;              // T [64][64]  (W is written later)
  static constexpr uint32_t SX = UU;                // 3 x [16][16] (U is written later)
  static_assert(bytes <= 232448, "shared memory per CTA");
  static_assert(DV * 128 >= 3 * 256 * 4, "block scratch fits in U");
};

// 8 consecutive bf16 elements (one 16-byte chunk) at (row, k0) of a 128B-swizzled tile.
__device__ __forceinline__ void st_chunk8(unsigned char* base, uint32_t slab_bytes, int row,
                                          int k0, const float* x) {
  __align__(16) __nv_bfloat162 h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
  *reinterpret_cast<uint4*>(base + sw128_offset(row, k0, slab_bytes)) =
      *reinterpret_cast<const uint4*>(h);
}

__device__ __forceinline__ void st_bf16(unsigned char* base, uint32_t off, float x) {
  *reinterpret_cast<__nv_bfloat16*>(base + off) = __float2bfloat16_rn(x);
}

// D (+)= A * B over K (multiple of 16).
__device__ __forceinline__ void mma_run(uint32_t d, Opnd A, Opnd B, int K, uint32_t idesc,
                                        bool acc) {
#pragma unroll 1
  for (int k = 0; k < K; k += 16) mma_bf16(d, A.at(k), B.at(k), idesc, (acc || k > 0) ? 1u : 0u);
}

// CTA-wide barrier that also orders tcgen05 operations around it.
__device__ __forceinline__ void cta_sync_tc() {
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
}

// Blockwise inverse of the unit lower-triangular I + A (A strictly lower, 64 x 64 fp32, row
// stride 64) into sT: 16 x 16 diagonal blocks by forward substitution, then the off-diagonal
// blocks by block diagonals, T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj.
__device__ void unit_lower_inverse(const float* sA, float* sT, float* sX, int tid) {
  constexpr int LD = kC;
  for (int i = tid; i < kC * kC; i += kThreads) {
    const int r = i / kC, c = i % kC;
    if ((c >> 4) > (r >> 4)) sT[r * LD + c] = 0.f;
  }
  if (tid < 64) {
    const int b = tid >> 4, c = tid & 15, o = 16 * b;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = (i == c) ? 1.f : 0.f;
#pragma unroll
      for (int j = 0; j < i; ++j) acc = fmaf(-sA[(o + i) * LD + o + j], x[j], acc);
      x[i] = (i < c) ? 0.f : acc;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) sT[(o + i) * LD + o + c] = x[i];
  }
  __syncthreads();
#pragma unroll 1
  for (int dist = 1; dist < 4; ++dist) {
    const int nblk = 4 - dist;  // blocks (i, j = i - dist), i = dist..3
    for (int e = tid; e < nblk * 256; e += kThreads) {
      const int bi = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
      const int i = bi + dist, j = bi;
      float acc = 0.f;
      for (int kb = j; kb < i; ++kb) {
        const float* arow = sA + (16 * i + rr) * LD + 16 * kb;
#pragma unroll
        for (int m = 0; m < 16; ++m) acc = fmaf(arow[m], sT[(16 * kb + m) * LD + 16 * j + cc], acc);
      }
      sX[bi * 256 + rr * 16 + cc] = acc;
    }
    __syncthreads();
    for (int e = tid; e < nblk * 256; e += kThreads) {
      const int bi = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
      const int i = bi + dist, j = bi;
      const float* trow = sT + (16 * i + rr) * LD + 16 * i;
      float acc = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) acc = fmaf(trow[m], sX[bi * 256 + m * 16 + cc], acc);
      sT[(16 * i + rr) * LD + 16 * j + cc] = -acc;
    }
    __syncthreads();
  }
}

struct TcMaps {
  CUtensorMap q, k, v, alpha;
};

template <int DV, bool CHANNEL, bool LINEAR>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ TcMaps maps, const PrefillArgs a) {
  using L = TcSmem<DV>;
  constexpr int NB = kD / DV;
  constexpr bool kAlphaTile = CHANNEL && !LINEAR;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(sm);
  const __nv_bfloat16* sQin = reinterpret_cast<const __nv_bfloat16*>(sm + L::QIN);
  const __nv_bfloat16* sKin = reinterpret_cast<const __nv_bfloat16*>(sm + L::KIN);
  float* sAin = reinterpret_cast<float*>(sm + L::AIN);
  float* sA = reinterpret_cast<float*>(sm + L::SA);
  float* sT32 = reinterpret_cast<float*>(sm + L::ST32);
  float* sX = reinterpret_cast<float*>(sm + L::SX);
  float* sBeta = reinterpret_cast<float*>(sm + L::BETA);
  float* sAlpha = reinterpret_cast<float*>(sm + L::ALPHA);
  float* sGam = reinterpret_cast<float*>(sm + L::GAM);
  float* sRed = reinterpret_cast<float*>(sm + L::RED);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
  uint64_t* bar_mma = bars + 0;
  uint64_t* bar_qk = bars + 1;
  uint64_t* bar_a = bars + 2;
  uint64_t* bar_v = bars + 3;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
  const uint32_t tm = *tslot;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;  // this warp's TMEM lane quarter
  uint32_t ph_mma = 0, ph_qk = 0, ph_a = 0, ph_v = 0;
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
  // waits on an mbarrier phase; every thread sees the same verdict
  auto wait_bar = [&](uint64_t* bar, uint32_t& ph) -> bool {
    const bool ok = mbar_wait(bar, ph, kWaitNs);
    ph ^= 1u;
    const bool all_ok = !__syncthreads_or(!ok);
    fence_after_sync();
    return all_ok;
  };
  // per-token scalars of a chunk (beta, scalar alpha), read one chunk ahead into registers
  auto load_scalars = [&](int64_t tc, float& b, float& al) {
    b = 0.f;
    al = 1.f;
    if (tid < kC && tc + tid < t1) {
      const size_t o = (size_t)(tc + tid) * H + h;
      if (!LINEAR) b = a.beta[o];
      if (!CHANNEL && !LINEAR) al = a.alpha[o];
    }
  };

  if (t0 < t1) {
    issue_qk(t0);
    issue_a(t0);
    issue_v(t0);
  }
  float nb_beta, nb_alpha;
  load_scalars(t0, nb_beta, nb_alpha);

  // ---- entering state: fp32 master in TMEM (lane = key channel), bf16 S operand row-wise
  {
    const float* s0 = a.S0 ? a.S0 + sidx + (size_t)tid * kD + vc0 : nullptr;
#pragma unroll
    for (int c0 = 0; c0 < DV; c0 += 32) {
      float x[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = s0 ? s0[c0 + j] : 0.f;
      tmem_st32(tm + lane_base + kColS + c0, x);
#pragma unroll
      for (int j = 0; j < 32; j += 8) st_chunk8(sm + L::SS, 16384, tid, c0 + j, x + j);
    }
    tmem_wait_st();
  }

  // operand views
  const Opnd opKQ{sb + L::KQ, 16384, false};          // [K~;Q~] as K-major A (M = 128)
  const Opnd opQ{sb + L::KQ + 8192, 16384, false};    // Q~ rows as K-major A (M = 64)
  const Opnd opKt{sb + L::KQ, 16384, true};           // K~ rows as MN-major B (K = tokens)
  const Opnd opKR{sb + L::KR, 8192, false};           // Kr as K-major B (N = 64 tokens)
  const Opnd opKH{sb + L::KH, 8192, true};            // K^ as MN-major A (M = 128 channels)
  const Opnd opT{sb + L::TT, 8192, false};
  const Opnd opM{sb + L::MM, 8192, false};
  const Opnd opW{sb + L::WW, 8192, false};
  const Opnd opV{sb + L::VIN, 8192, true};            // V as MN-major B (K = tokens)
  const Opnd opU{sb + L::UU, 8192, true};             // U as MN-major B (K = tokens)
  const Opnd opS{sb + L::SS, 16384, true};            // S as MN-major B (K = key channels)
  const uint32_t id_am = idesc_bf16(128, kC);
  const uint32_t id_w = idesc_bf16(64, kD, false, false, true);
  const uint32_t id_v = idesc_bf16(64, DV, false, false, true);
  const uint32_t id_negw = idesc_bf16(64, DV, true, false, true);
  const uint32_t id_s = idesc_bf16(128, DV, false, true, true);

#pragma unroll 1
  for (int64_t tc = t0; tc < t1 && !failed; tc += kC) {
    const int n = (int)((t1 - tc) < (int64_t)kC ? (t1 - tc) : (int64_t)kC);
    const int64_t tn = tc + kC;  // next chunk
    const int c = tid;           // key channel owned in the gate pass

    if (tid < kC) {
      sBeta[tid] = nb_beta;
      sAlpha[tid] = nb_alpha;
    }
    if (tn < t1) load_scalars(tn, nb_beta, nb_alpha);
    if (!wait_bar(bar_qk, ph_qk)) { failed = true; break; }
    if (kAlphaTile && !wait_bar(bar_a, ph_a)) { failed = true; break; }

    // ================= 1. gates and operand tiles (thread = key channel)
    float gam = 1.f;
    if (!LINEAR) {
#pragma unroll 8
      for (int r = 0; r < kC; ++r)
        if (r < n) gam *= kAlphaTile ? sAin[r * kD + c] : sAlpha[r];
      sGam[c] = gam;
    }
    float mn = gam;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    if (lane == 0) sRed[warp] = mn;
    __syncthreads();
    const bool safe =
        LINEAR || fminf(fminf(sRed[0], sRed[1]), fminf(sRed[2], sRed[3])) > kSafeGamma;

    if (safe) {
      float G = 1.f;  // running product of the gates
#pragma unroll 4
      for (int r = 0; r < kC; ++r) {
        const bool ok = r < n;
        const float kv = ok ? __bfloat162float(sKin[r * kD + c]) : 0.f;
        const float qv = ok ? __bfloat162float(sQin[r * kD + c]) : 0.f;
        float e = 1.f, ei = 1.f;
        if (!LINEAR && ok) {
          G *= kAlphaTile ? sAin[r * kD + c] : sAlpha[r];
          e = G;
          ei = __frcp_rn(G);
        }
        const float ke = kv * e, ki = kv * ei;
        st_bf16(sm + L::KQ, sw128_offset(r, c, 16384), ke);              // K~
        st_bf16(sm + L::KQ, sw128_offset(64 + r, c, 16384), qv * e);     // Q~
        st_bf16(sm + L::KR, sw128_offset(r, c, 8192), ki);               // Kr
        st_bf16(sm + L::KH, sw128_offset(r, c, 8192), ki * gam);         // K^
      }
    } else {
      // strong decay: log-gate prefix sums, in place of the staged gates
      float G = 0.f;
#pragma unroll 4
      for (int r = 0; r < kC; ++r) {
        if (r < n) G += log_gate(kAlphaTile ? sAin[r * kD + c] : sAlpha[r]);
        if (kAlphaTile) sAin[r * kD + c] = G;
      }
      const float Gn = G;
      G = 0.f;
#pragma unroll 4
      for (int r = 0; r < kC; ++r) {
        const bool ok = r < n;
        const float kv = ok ? __bfloat162float(sKin[r * kD + c]) : 0.f;
        const float qv = ok ? __bfloat162float(sQin[r * kD + c]) : 0.f;
        if (kAlphaTile) G = sAin[r * kD + c];
        else if (ok) G += log_gate(sAlpha[r]);
        const float e = __expf(G);
        st_bf16(sm + L::KQ, sw128_offset(r, c, 16384), kv * e);
        st_bf16(sm + L::KQ, sw128_offset(64 + r, c, 16384), qv * e);
        st_bf16(sm + L::KH, sw128_offset(r, c, 8192), kv * __expf(Gn - G));
      }
      if (!kAlphaTile) {  // scalar gates: keep the per-token prefix sums for the pair decays
        __syncthreads();
        if (tid == 0) {
          float g = 0.f;
          for (int r = 0; r < kC; ++r) {
            if (r < n) g += log_gate(sAlpha[r]);
            sAlpha[r] = g;
          }
        }
      }
    }
    fence_async_smem();
    cta_sync_tc();
    if (safe && tn < t1) {  // q, k and alpha tiles are consumed: fetch the next chunk's
      issue_qk(tn);
      issue_a(tn);
    }

    // ================= 2. decay-weighted Gram matrices [A'; M]
    if (safe) {
      if (tid == 0) {
        mma_run(tm + kColAM, opKQ, opKR, kD, id_am, false);
        mma_commit(bar_mma);
      }
      if (!wait_bar(bar_mma, ph_mma)) { failed = true; break; }
      const int r = tid & 63;
#pragma unroll
      for (int c0 = 0; c0 < kC; c0 += 32) {
        float x[32];
        tmem_ld32(tm + lane_base + kColAM + c0, x);
        if (tid < 64) {
          if (!LINEAR) {
            const float b = sBeta[r];
#pragma unroll
            for (int j = 0; j < 32; ++j) sA[r * kC + c0 + j] = (c0 + j < r) ? b * x[j] : 0.f;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = (c0 + j <= r) ? x[j] : 0.f;
#pragma unroll
          for (int j = 0; j < 32; j += 8) st_chunk8(sm + L::MM, 8192, r, c0 + j, x + j);
        }
      }
    } else {
      // direct pairwise decays over the lower triangle
      for (int p = tid; p < kC * (kC + 1) / 2; p += kThreads) {
        int r = (int)((sqrtf(8.f * p + 1.f) - 1.f) * 0.5f);
        while (r * (r + 1) / 2 > p) --r;
        while ((r + 1) * (r + 2) / 2 <= p) ++r;
        const int j = p - r * (r + 1) / 2;
        float acc_a = 0.f, acc_m = 0.f;
        if (r < n) {
          for (int cc = 0; cc < kD; ++cc) {
            const float dg = kAlphaTile ? sAin[r * kD + cc] - sAin[j * kD + cc]
                                        : sAlpha[r] - sAlpha[j];
            const float w = __bfloat162float(sKin[j * kD + cc]) * __expf(dg);
            acc_a = fmaf(__bfloat162float(sKin[r * kD + cc]), w, acc_a);
            acc_m = fmaf(__bfloat162float(sQin[r * kD + cc]), w, acc_m);
          }
        }
        sA[r * kC + j] = (j < r) ? sBeta[r] * acc_a : 0.f;
        st_bf16(sm + L::MM, sw128_offset(r, j, 8192), acc_m);
      }
      for (int p = tid; p < kC * kC; p += kThreads) {
        const int r = p / kC, j = p % kC;
        if (j > r) {
          sA[r * kC + j] = 0.f;
          st_bf16(sm + L::MM, sw128_offset(r, j, 8192), 0.f);
        }
      }
      __syncthreads();
      if (tn < t1) {
        issue_qk(tn);
        issue_a(tn);
      }
    }
    __syncthreads();

    // the chunk's V tile (zero the rows past the end of the sequence)
    if (!wait_bar(bar_v, ph_v)) { failed = true; break; }
    if (n < kC) {
      for (int i = tid; i < (kC - n) * (DV / 8); i += kThreads) {
        const int r = n + i / (DV / 8), ch = i % (DV / 8);
        *reinterpret_cast<uint4*>(sm + L::VIN + (ch >> 3) * 8192 + r * 128 + (ch & 7) * 16) =
            make_uint4(0, 0, 0, 0);
      }
      fence_async_smem();
    }

    if (!LINEAR) {
      // ================= 3. T' = (I + A)^-1 diag(beta)  (bf16 A operand)
      unit_lower_inverse(sA, sT32, sX, tid);
      for (int e = tid; e < kC * kC / 8; e += kThreads) {
        const int r = e >> 3, j0 = (e & 7) * 8;
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = sT32[r * kC + j0 + i] * sBeta[j0 + i];
        st_chunk8(sm + L::TT, 8192, r, j0, x);
      }
      fence_async_smem();
      cta_sync_tc();

      // ================= 4. W = T' K~  and  U~ = T' V
      if (tid == 0) {
        mma_run(tm + kColWO, opT, opKt, kC, id_w, false);
        mma_run(tm + kColU, opT, opV, kC, id_v, false);
        mma_commit(bar_mma);
      }
      if (!wait_bar(bar_mma, ph_mma)) { failed = true; break; }
      if (tn < t1) issue_v(tn);  // V is consumed
      {
        float x[32];
        const int r = warp * 16 + (lane & 15);
#pragma unroll
        for (int c0 = 0; c0 < kD; c0 += 32) {
          tmem_ld32(tm + lane_base + kColWO + c0, x);
          if (lane < 16) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) st_chunk8(sm + L::WW, 8192, r, c0 + j, x + j);
          }
        }
      }
      fence_async_smem();
    }
    cta_sync_tc();

    // ================= 5. U = U~ - W S  and  O = Q~ S
    if (tid == 0) {
      if (!LINEAR) mma_run(tm + kColU, opW, opS, kD, id_negw, true);
      mma_run(tm + kColWO, opQ, opS, kD, id_v, false);
      mma_commit(bar_mma);
    }
    if (!LINEAR) {
      // meanwhile: fade the state master, S <- Diag(gamma) S (lane = key channel)
      const float gm = sGam[tid];
#pragma unroll
      for (int c0 = 0; c0 < DV; c0 += 32) {
        float x[32];
        tmem_ld32(tm + lane_base + kColS + c0, x);
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] *= gm;
        tmem_st32(tm + lane_base + kColS + c0, x);
      }
      tmem_wait_st();
    }
    if (!wait_bar(bar_mma, ph_mma)) { failed = true; break; }
    if (!LINEAR) {
      float x[32];
      const int r = warp * 16 + (lane & 15);
#pragma unroll
      for (int c0 = 0; c0 < DV; c0 += 32) {
        tmem_ld32(tm + lane_base + kColU + c0, x);
        if (lane < 16) {
#pragma unroll
          for (int j = 0; j < 32; j += 8) st_chunk8(sm + L::UU, 8192, r, c0 + j, x + j);
        }
      }
      fence_async_smem();
    }
    cta_sync_tc();

    // ================= 6. O += M U  and  S += K^^T U
    if (tid == 0) {
      const Opnd opUse = LINEAR ? opV : opU;
      mma_run(tm + kColWO, opM, opUse, kC, id_v, true);
      mma_run(tm + kColS, opKH, opUse, kC, id_s, true);
      mma_commit(bar_mma);
    }
    if (!wait_bar(bar_mma, ph_mma)) { failed = true; break; }
    if (LINEAR && tn < t1) issue_v(tn);
    // O (M = 64 layout) -> out, rows < n
    {
      float x[32];
      const int r = warp * 16 + (lane & 15);
#pragma unroll
      for (int c0 = 0; c0 < DV; c0 += 32) {
        tmem_ld32(tm + lane_base + kColWO + c0, x);
        if (lane < 16 && r < n) {
          __nv_bfloat16* dst = out + ((size_t)(tc + r) * H + h) * kD + vc0 + c0;
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            __align__(16) __nv_bfloat162 hv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) hv[i] = __floats2bfloat162_rn(x[j + 2 * i], x[j + 2 * i + 1]);
            *reinterpret_cast<uint4*>(dst + j) = *reinterpret_cast<const uint4*>(hv);
          }
        }
      }
    }
    // new state -> bf16 S operand for the next chunk (lane = key channel)
#pragma unroll
    for (int c0 = 0; c0 < DV; c0 += 32) {
      float x[32];
      tmem_ld32(tm + lane_base + kColS + c0, x);
#pragma unroll
      for (int j = 0; j < 32; j += 8) st_chunk8(sm + L::SS, 16384, tid, c0 + j, x + j);
    }
    fence_async_smem();
    cta_sync_tc();
  }

  if (failed) {
    if (tid == 0) report(a.status, GDR_DEVCHECK_TIMEOUT);
    // let copies already in flight land before the shared memory is released
    mbar_wait(bar_qk, ph_qk, kWaitNs);
    if (kAlphaTile) mbar_wait(bar_a, ph_a, kWaitNs);
    mbar_wait(bar_v, ph_v, kWaitNs);
  } else if (a.S_final) {
    float* sf = a.S_final + sidx + (size_t)tid * kD + vc0;
#pragma unroll
    for (int c0 = 0; c0 < DV; c0 += 32) {
      float x[32];
      tmem_ld32(tm + lane_base + kColS + c0, x);
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4*>(sf + c0 + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
    }
  }
  cta_sync_tc();
  if (warp == 0) tmem_dealloc(tm, kTmemCols);
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

template <int DV, bool CHANNEL, bool LINEAR>
cudaError_t launch_one(const gdr_shape& sh, const PrefillArgs& a, const TcMaps& maps,
                       cudaStream_t s) {
  auto kern = prefill_tc_kernel<DV, CHANNEL, LINEAR>;
  const size_t smem = TcSmem<DV>::bytes;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)sh.n_seqs * (unsigned)sh.H * (unsigned)(kD / DV);
  kern<<<grid, kThreads, smem, s>>>(maps, a);
  return cudaGetLastError();
}

template <int DV>
cudaError_t launch_dv(const gdr_shape& sh, const PrefillArgs& a, const TcMaps& maps, bool linear,
                      cudaStream_t s) {
  if (linear) return launch_one<DV, true, true>(sh, a, maps, s);
  if (sh.gate == GDR_GATE_CHANNEL) return launch_one<DV, true, false>(sh, a, maps, s);
  return launch_one<DV, false, false>(sh, a, maps, s);
}

}  // namespace

bool prefill_tc_supported(const gdr_shape& sh) {
  return sh.dtype == GDR_BF16 && sh.d_k == kD && sh.d_v == kD &&
         !(sh.flags & GDR_FLAG_FORCE_SIMT) && sh.total_tokens > 0 &&
         sh.total_tokens < ((int64_t)1 << 31) && encode_fn() != nullptr;
}

cudaError_t launch_prefill_tc(const gdr_shape& sh, const PrefillArgs& a, bool linear,
                              cudaStream_t s) {
  TcMaps maps;
  memset(&maps, 0, sizeof(maps));
  const int H = sh.H;
  const int64_t T = sh.total_tokens;
  bool ok = make_map(&maps.q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, kD,
                     CU_TENSOR_MAP_SWIZZLE_NONE) &&
            make_map(&maps.k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, kD,
                     CU_TENSOR_MAP_SWIZZLE_NONE) &&
            make_map(&maps.v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  if (ok && !linear && sh.gate == GDR_GATE_CHANNEL)
    ok = make_map(&maps.alpha, a.alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H, T, kD,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!ok) return cudaErrorInvalidValue;
  // value-column split: enough CTAs to cover the SMs when there are few (sequence, head) pairs
  const long pairs = (long)sh.n_seqs * sh.H;
  if (pairs >= 120) return launch_dv<128>(sh, a, maps, linear, s);
  return launch_dv<64>(sh, a, maps, linear, s);
}

}  // namespace gdr
