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
// Mapping: one CTA (8 warps) per (sequence, head, block of DV value columns); columns of S are
// independent, so the value dimension splits across CTAs.  Warp w reads TMEM lane quarter w & 3
// and the column half w >> 2 of every accumulator: thread t owns lane t & 127, i.e. key channel
// t & 127 of the state or token row t & 127 of the M = 128 Gram accumulator; M = 64
// accumulators (token rows) occupy lanes 32q + [0, 16) for rows 16q + [0, 16).  q, k, alpha and
// v tiles of the next chunk are fetched by TMA while the current chunk computes.
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
constexpr int kThreads = 256;    // 8 warps: two per TMEM lane quarter
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
  static constexpr uint32_t RED = GAM + 512;        // reductions [8]
  static constexpr uint32_t DIAG = RED + 64;        // q_r . k_r [64]
  static constexpr uint32_t GS = DIAG + 256;        // scalar gates: log prefix sums [64]
  static constexpr uint32_t BARS = GS + 256;        // 4 mbarriers + TMEM slot
  static constexpr uint32_t END = BARS + 64;
  static constexpr size_t bytes = END + 1024;       // + alignment slack
  // fp32 scratch of the solve, in tiles that are dead while it runs
  static constexpr uint32_t SA = KR;                // A [64][64]  (Kr is consumed by then)
  static constexpr uint32_t ST32 = WW;              // T [64][64]  (W is written later)
  static constexpr uint32_t SX = UU;                // [32][32] (U is written later)
  static_assert(bytes <= 232448, "shared memory per CTA");
  static_assert(DV * 128 >= 32 * 32 * 4, "block scratch fits in U");
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

// fp32 64 x 64 scratch matrices (A, T) keep their 16-byte column groups XOR-swizzled by the
// row (group g of row r stored at position g ^ (r & 7)), so eight consecutive rows touching the
// same column group hit eight different bank groups.
__device__ __forceinline__ int f32x(int r, int j) {
  return r * kC + ((((j >> 2) ^ (r & 7))) << 2) + (j & 3);
}
__device__ __forceinline__ float4 ld4x(const float* m, int r, int grp) {
  return *reinterpret_cast<const float4*>(m + r * kC + ((grp ^ (r & 7)) << 2));
}
__device__ __forceinline__ void st4x(float* m, int r, int grp, float4 v) {
  *reinterpret_cast<float4*>(m + r * kC + ((grp ^ (r & 7)) << 2)) = v;
}
__device__ __forceinline__ void fma4(float4& acc, float a, float4 b) {
  acc.x = fmaf(a, b.x, acc.x);
  acc.y = fmaf(a, b.y, acc.y);
  acc.z = fmaf(a, b.z, acc.z);
  acc.w = fmaf(a, b.w, acc.w);
}

// T = (I + A)^-1 for A strictly lower (64 x 64, fp32, swizzled layout above), by doubling the
// inverted block size: the four 16 x 16 diagonal blocks by right-looking forward substitution
// (one column per thread, held in registers); then both 32 x 32 diagonal blocks at once,
// T_ba = -T_bb (A_ba T_aa) for (a, b) = (0, 1) and (2, 3); then the 64 x 64 inverse,
// T_[23][01] = -T_[23][23] (A_[23][01] T_[01][01]).  sX holds the 32 x 32 intermediate.
__device__ void unit_lower_inverse(const float* sA, float* sT, float* sX, int tid) {
  if (tid < 64) {
    const int b = tid >> 4, c = tid & 15, o = 16 * b;
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = (i == c) ? 1.f : 0.f;
#pragma unroll
    for (int j = 0; j < 15; ++j) {
      const float xj = acc[j];
#pragma unroll
      for (int i = j + 1; i < 16; ++i) acc[i] = fmaf(-sA[f32x(o + i, o + j)], xj, acc[i]);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) sT[f32x(o + i, o + c)] = acc[i];
  } else {
    // strictly-upper blocks of T are zero: rows 0-31 from column 32, and the 16 x 16 blocks
    // (0, 1) and (2, 3)
    for (int e = tid - 64; e < kC * 16; e += kThreads - 64) {
      const int r = e >> 4, grp = e & 15;
      if (grp >= 4 * ((r >> 4) + 1)) st4x(sT, r, grp, make_float4(0.f, 0.f, 0.f, 0.f));
    }
  }
  __syncthreads();
  // ---- level 32: blocks (1, 0) and (3, 2); 2 x 256 outputs, 2 per thread
  {
    const int blk = tid >> 7, e = tid & 127;       // blk 0: (1,0); blk 1: (3,2)
    const int rr = e >> 3, c2 = (e & 7) * 2;       // row in the block, column pair
    const int ra = 32 * blk, rb = ra + 16;         // first rows of block rows a and b
    float x0 = 0.f, x1 = 0.f;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float am = sA[f32x(rb + rr, ra + m)];
      x0 = fmaf(am, sT[f32x(ra + m, ra + c2)], x0);
      x1 = fmaf(am, sT[f32x(ra + m, ra + c2 + 1)], x1);
    }
    sX[blk * 256 + rr * 16 + c2] = x0;
    sX[blk * 256 + rr * 16 + c2 + 1] = x1;
    __syncthreads();
    float y0 = 0.f, y1 = 0.f;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float tm = m <= rr ? sT[f32x(rb + rr, rb + m)] : 0.f;
      y0 = fmaf(tm, sX[blk * 256 + m * 16 + c2], y0);
      y1 = fmaf(tm, sX[blk * 256 + m * 16 + c2 + 1], y1);
    }
    sT[f32x(rb + rr, ra + c2)] = -y0;
    sT[f32x(rb + rr, ra + c2 + 1)] = -y1;
    __syncthreads();
  }
  // ---- level 64: block [23][01] (32 x 32); 1024 outputs, 4 per thread (one float4 group)
  {
    const int rr = tid >> 3, grp = tid & 7;  // row 0..31 of the block, float4 group 0..7
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int m = 0; m < 32; ++m) fma4(x, sA[f32x(32 + rr, m)], ld4x(sT, m, grp));
    *reinterpret_cast<float4*>(sX + rr * 32 + 4 * grp) = x;
    __syncthreads();
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int m = 0; m < 32; ++m) {
      const float tm = m <= rr ? sT[f32x(32 + rr, 32 + m)] : 0.f;
      fma4(y, tm, *reinterpret_cast<const float4*>(sX + m * 32 + 4 * grp));
    }
    st4x(sT, 32 + rr, grp, make_float4(-y.x, -y.y, -y.z, -y.w));
    __syncthreads();
  }
}

// 8 bf16 values (one 16-byte chunk) -> fp32
__device__ __forceinline__ void ld_bf16x8(const __nv_bfloat16* p, float* x) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
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
  constexpr int DH = DV / 2;  // accumulator columns per warp half
  constexpr bool kAlphaTile = CHANNEL && !LINEAR;
  constexpr bool kScalar = !CHANNEL && !LINEAR;
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
  float* sDiag = reinterpret_cast<float*>(sm + L::DIAG);
  float* sGs = reinterpret_cast<float*>(sm + L::GS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
  uint64_t* bar_mma = bars + 0;
  uint64_t* bar_qk = bars + 1;
  uint64_t* bar_a = bars + 2;
  uint64_t* bar_v = bars + 3;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lrow = tid & 127;      // TMEM lane of this thread
  const int wh = warp >> 2;        // column half of the accumulators
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
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;  // TMEM lane quarter
  const int m64row = 16 * (warp & 3) + (lane & 15);  // token row of M = 64 accumulators
  const bool m64ok = lane < 16;
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
    const float* s0 = a.S0 ? a.S0 + sidx + (size_t)lrow * kD + vc0 : nullptr;
#pragma unroll
    for (int c0 = wh * DH; c0 < wh * DH + DH; c0 += 32) {
      float x[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = s0 ? s0[c0 + j] : 0.f;
      tmem_st32(tm + lane_base + kColS + c0, x);
#pragma unroll
      for (int j = 0; j < 32; j += 8) st_chunk8(sm + L::SS, 16384, lrow, c0 + j, x + j);
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

    if (tid < kC) {
      sBeta[tid] = nb_beta;
      sAlpha[tid] = nb_alpha;
    }
    if (tn < t1) load_scalars(tn, nb_beta, nb_alpha);
    if (!wait_bar(bar_qk, ph_qk)) { failed = true; break; }
    if (kAlphaTile && !wait_bar(bar_a, ph_a)) { failed = true; break; }

    // ================= 1. gates and operand tiles
    // thread = 8 key channels (group g8) x 4 tokens (row block rb)
    const int g8 = tid & 15, rb = tid >> 4;
    bool safe = true;
    if constexpr (kScalar) {
      // Scalar gates: the pair decay e^(G_r - G_j) is a per-token factor, applied in fp32 after
      // the Gram products of the raw (exact bf16) q and k; G = prefix sums of the clamped log
      // gates, two tokens per lane of warp 0.
      if (warp == 0) {
        const int r0 = 2 * lane;
        const float g0 = r0 < n ? log_gate(sAlpha[r0]) : 0.f;
        const float g1 = r0 + 1 < n ? log_gate(sAlpha[r0 + 1]) : 0.f;
        float sc = g0 + g1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float t = __shfl_up_sync(0xffffffffu, sc, off);
          if (lane >= off) sc += t;
        }
        sGs[r0] = sc - g1;
        sGs[r0 + 1] = sc;
      }
      __syncthreads();
      const float Gn = sGs[kC - 1];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int r = 4 * rb + rr;
        float k8[8], q8[8], kh[8];
        if (r < n) {
          ld_bf16x8(sKin + r * kD + 8 * g8, k8);
          ld_bf16x8(sQin + r * kD + 8 * g8, q8);
        } else {
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) k8[cc] = q8[cc] = 0.f;
        }
        const float eh = __expf(Gn - sGs[r]);
        float dq = 0.f;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          kh[cc] = k8[cc] * eh;
          dq = fmaf(q8[cc], k8[cc], dq);
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) dq += __shfl_xor_sync(0xffffffffu, dq, off);
        if (g8 == 0) sDiag[r] = dq;
        st_chunk8(sm + L::KQ, 16384, r, 8 * g8, k8);       // K (scaled to K~ after the Gram MMA)
        st_chunk8(sm + L::KQ, 16384, 64 + r, 8 * g8, q8);  // Q (scaled to Q~ likewise)
        st_chunk8(sm + L::KR, 8192, r, 8 * g8, k8);        // K
        st_chunk8(sm + L::KH, 8192, r, 8 * g8, kh);        // K^
      }
      if (rb == 0) {
        const float gm = __expf(Gn);
        *reinterpret_cast<float4*>(sGam + 8 * g8) = make_float4(gm, gm, gm, gm);
        *reinterpret_cast<float4*>(sGam + 8 * g8 + 4) = make_float4(gm, gm, gm, gm);
      }
    } else {
      // Per-channel gates (and linear attention): running products of the gates down the
      // thread's rows, then the carry of the earlier row blocks through shared memory.
      float p[4][8];  // prefix products Gam[4 rb + rr][8 g8 + cc]
      float gn[8];    // Gam_n (= gamma) of the 8 channels
      {
        float run[8];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) run[cc] = 1.f;
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          const int r = 4 * rb + rr;
          float a8[8];
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) a8[cc] = 1.f;
          if (!LINEAR && r < n) {
            const float4 u0 = *reinterpret_cast<const float4*>(sAin + r * kD + 8 * g8);
            const float4 u1 = *reinterpret_cast<const float4*>(sAin + r * kD + 8 * g8 + 4);
            a8[0] = u0.x, a8[1] = u0.y, a8[2] = u0.z, a8[3] = u0.w;
            a8[4] = u1.x, a8[5] = u1.y, a8[6] = u1.z, a8[7] = u1.w;
          }
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            run[cc] *= a8[cc];
            p[rr][cc] = run[cc];
          }
        }
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) gn[cc] = 1.f;
        if (!LINEAR) {
          float* sTot = reinterpret_cast<float*>(sm + L::WW);  // [16 row blocks][128 channels]
          *reinterpret_cast<float4*>(sTot + rb * kD + 8 * g8) = make_float4(run[0], run[1], run[2], run[3]);
          *reinterpret_cast<float4*>(sTot + rb * kD + 8 * g8 + 4) = make_float4(run[4], run[5], run[6], run[7]);
          __syncthreads();
          float carry[8];
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) carry[cc] = 1.f;
#pragma unroll
          for (int b2 = 0; b2 < 16; ++b2) {
            const float4 u0 = *reinterpret_cast<const float4*>(sTot + b2 * kD + 8 * g8);
            const float4 u1 = *reinterpret_cast<const float4*>(sTot + b2 * kD + 8 * g8 + 4);
            const float t8[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
              if (b2 < rb) carry[cc] *= t8[cc];
              gn[cc] *= t8[cc];
            }
          }
#pragma unroll
          for (int rr = 0; rr < 4; ++rr)
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) p[rr][cc] *= carry[cc];
        }
      }
      if (!LINEAR) {
        float mn = gn[0];
#pragma unroll
        for (int cc = 1; cc < 8; ++cc) mn = fminf(mn, gn[cc]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
        if (lane == 0) sRed[warp] = mn;
        if (rb == 0) {
          *reinterpret_cast<float4*>(sGam + 8 * g8) = make_float4(gn[0], gn[1], gn[2], gn[3]);
          *reinterpret_cast<float4*>(sGam + 8 * g8 + 4) = make_float4(gn[4], gn[5], gn[6], gn[7]);
        }
        __syncthreads();
        float mall = sRed[0];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) mall = fminf(mall, sRed[w]);
        safe = mall > kSafeGamma;
      }

      if (safe) {
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          const int r = 4 * rb + rr;
          float k8[8], q8[8];
          if (r < n) {
            ld_bf16x8(sKin + r * kD + 8 * g8, k8);
            ld_bf16x8(sQin + r * kD + 8 * g8, q8);
          } else {
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) k8[cc] = q8[cc] = 0.f;
          }
          float ke[8], qe[8], ki[8], kh[8], dq = 0.f;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            const float G = p[rr][cc];
            const float inv = LINEAR ? 1.f : __fdividef(1.f, G);
            ke[cc] = k8[cc] * G;
            qe[cc] = q8[cc] * G;
            ki[cc] = k8[cc] * inv;
            kh[cc] = ki[cc] * gn[cc];
            dq = fmaf(q8[cc], k8[cc], dq);
          }
          if (!LINEAR) {  // the diagonal of M carries no decay: q_r . k_r in fp32
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) dq += __shfl_xor_sync(0xffffffffu, dq, off);
            if (g8 == 0) sDiag[r] = dq;
          }
          st_chunk8(sm + L::KQ, 16384, r, 8 * g8, ke);       // K~
          st_chunk8(sm + L::KQ, 16384, 64 + r, 8 * g8, qe);  // Q~
          st_chunk8(sm + L::KR, 8192, r, 8 * g8, ki);        // Kr
          st_chunk8(sm + L::KH, 8192, r, 8 * g8, kh);        // K^
        }
      } else if (tid < kD) {
        // strong decay: log-gate prefix sums in place of the staged gates (thread = channel)
        const int c = tid;
        float G = 0.f;
#pragma unroll 4
        for (int r = 0; r < kC; ++r) {
          if (r < n) G += log_gate(sAin[r * kD + c]);
          sAin[r * kD + c] = G;
        }
        const float Gn = G;
#pragma unroll 4
        for (int r = 0; r < kC; ++r) {
          const bool ok = r < n;
          const float kv = ok ? __bfloat162float(sKin[r * kD + c]) : 0.f;
          const float qv = ok ? __bfloat162float(sQin[r * kD + c]) : 0.f;
          G = sAin[r * kD + c];
          const float e = __expf(G);
          st_bf16(sm + L::KQ, sw128_offset(r, c, 16384), kv * e);
          st_bf16(sm + L::KQ, sw128_offset(64 + r, c, 16384), qv * e);
          st_bf16(sm + L::KH, sw128_offset(r, c, 8192), kv * __expf(Gn - G));
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
      const int r = lrow & 63;
      const int c0 = 32 * wh;
      float x[32];
      tmem_ld32(tm + lane_base + kColAM + c0, x);
      if constexpr (kScalar) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          x[j] = (c0 + j <= r) ? x[j] * __expf(sGs[r] - sGs[c0 + j]) : 0.f;
      }
      if (lrow < 64) {
        if (!LINEAR) {
          const float b = sBeta[r];
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            st4x(sA, r, (c0 + j) >> 2,
                 make_float4((c0 + j < r) ? b * x[j] : 0.f, (c0 + j + 1 < r) ? b * x[j + 1] : 0.f,
                             (c0 + j + 2 < r) ? b * x[j + 2] : 0.f,
                             (c0 + j + 3 < r) ? b * x[j + 3] : 0.f));
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          x[j] = (c0 + j <= r) ? x[j] : 0.f;
          if (!LINEAR && c0 + j == r) x[j] = sDiag[r];
        }
#pragma unroll
        for (int j = 0; j < 32; j += 8) st_chunk8(sm + L::MM, 8192, r, c0 + j, x + j);
      }
      if constexpr (kScalar) {
        // the raw K and Q rows of the Gram operand become K~ = K e^G and Q~ = Q e^G in place
        __syncthreads();
        for (int e = tid; e < 2 * 128 * 8; e += kThreads) {
          const int slab = e >> 10, row = (e >> 3) & 127, ch = e & 7;
          uint4* pch = reinterpret_cast<uint4*>(sm + L::KQ + slab * 16384 + row * 128 + ch * 16);
          const float f = __expf(sGs[row & 63]);
          uint4 u = *pch;
          __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 v2 = __bfloat1622float2(hv[i]);
            hv[i] = __floats2bfloat162_rn(v2.x * f, v2.y * f);
          }
          *pch = u;
        }
        fence_async_smem();
      }
    } else {
      // direct pairwise decays over the lower triangle (per-channel gates only)
      for (int p2 = tid; p2 < kC * (kC + 1) / 2; p2 += kThreads) {
        int r = (int)((sqrtf(8.f * p2 + 1.f) - 1.f) * 0.5f);
        while (r * (r + 1) / 2 > p2) --r;
        while ((r + 1) * (r + 2) / 2 <= p2) ++r;
        const int j = p2 - r * (r + 1) / 2;
        float acc_a = 0.f, acc_m = 0.f;
        if (r < n) {
          for (int cc = 0; cc < kD; ++cc) {
            const float w = __bfloat162float(sKin[j * kD + cc]) *
                            __expf(sAin[r * kD + cc] - sAin[j * kD + cc]);
            acc_a = fmaf(__bfloat162float(sKin[r * kD + cc]), w, acc_a);
            acc_m = fmaf(__bfloat162float(sQin[r * kD + cc]), w, acc_m);
          }
        }
        sA[f32x(r, j)] = (j < r) ? sBeta[r] * acc_a : 0.f;
        st_bf16(sm + L::MM, sw128_offset(r, j, 8192), acc_m);
      }
      for (int p2 = tid; p2 < kC * kC; p2 += kThreads) {
        const int r = p2 / kC, j = p2 % kC;
        if (j > r) {
          sA[f32x(r, j)] = 0.f;
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
        for (int i = 0; i < 8; ++i) x[i] = sT32[f32x(r, j0 + i)] * sBeta[j0 + i];
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
#pragma unroll
      for (int c0 = wh * 64; c0 < wh * 64 + 64; c0 += 32) {
        float x[32];
        tmem_ld32(tm + lane_base + kColWO + c0, x);
        if (m64ok) {
#pragma unroll
          for (int j = 0; j < 32; j += 8) st_chunk8(sm + L::WW, 8192, m64row, c0 + j, x + j);
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
      const float gm = sGam[lrow];
#pragma unroll
      for (int c0 = wh * DH; c0 < wh * DH + DH; c0 += 32) {
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
#pragma unroll
      for (int c0 = wh * DH; c0 < wh * DH + DH; c0 += 32) {
        float x[32];
        tmem_ld32(tm + lane_base + kColU + c0, x);
        if (m64ok) {
#pragma unroll
          for (int j = 0; j < 32; j += 8) st_chunk8(sm + L::UU, 8192, m64row, c0 + j, x + j);
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
#pragma unroll
    for (int c0 = wh * DH; c0 < wh * DH + DH; c0 += 32) {
      float x[32];
      tmem_ld32(tm + lane_base + kColWO + c0, x);
      if (m64ok && m64row < n) {
        __nv_bfloat16* dst = out + ((size_t)(tc + m64row) * H + h) * kD + vc0 + c0;
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          __align__(16) __nv_bfloat162 hv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) hv[i] = __floats2bfloat162_rn(x[j + 2 * i], x[j + 2 * i + 1]);
          *reinterpret_cast<uint4*>(dst + j) = *reinterpret_cast<const uint4*>(hv);
        }
      }
    }
    // new state -> bf16 S operand for the next chunk (lane = key channel)
#pragma unroll
    for (int c0 = wh * DH; c0 < wh * DH + DH; c0 += 32) {
      float x[32];
      tmem_ld32(tm + lane_base + kColS + c0, x);
#pragma unroll
      for (int j = 0; j < 32; j += 8) st_chunk8(sm + L::SS, 16384, lrow, c0 + j, x + j);
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
    float* sf = a.S_final + sidx + (size_t)lrow * kD + vc0;
#pragma unroll
    for (int c0 = wh * DH; c0 < wh * DH + DH; c0 += 32) {
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
