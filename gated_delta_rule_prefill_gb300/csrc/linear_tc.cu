// linear_tc.cu -- chunked linear attention (alpha = 1, no erase term) on the tensor cores,
// d_k = d_v = 128, bf16 q/k/v, fp32 state.  Per chunk of C = 64 tokens entering with state S:
//   O = Q S + lower(Q K^T) V,   S <- S + K^T V
// (engineermaxxing "From GPT-2 to Kimi K3: one memory, seven eviction policies" §03b and §04b;
// heqinghuang "gpt2-to-kimi" §10).  With no gates there is nothing to prepare per chunk: q and k
// arrive by TMA directly as the 128B-swizzled [K; Q] operand tile (K rows 0-63, Q rows 64-127 of
// each 64-channel slab), v as the MN-major B tile.  Per chunk (one CTA, 8 warps):
//   S += K^T V                      (M = 128: K as MN-major A; fp32 state master in TMEM)
//   D = [K; Q] S,  A = [K; Q] K^T   (M = 128 each; rows 64-127 are Q S and Q K^T)
//   S master -> bf16 operand for the next chunk (double-buffered, so this waits only for the
//   state MMA), lower(Q K^T) -> bf16 M,  then  D += [Z; M] V  (rows 64-127: O)
// and the O rows leave TMEM while the next chunk's MMAs run.  q, k, v of the next chunk are
// fetched one chunk ahead.  That is the normalised form's loop; the plain form runs the same
// products transposed (S^T in TMEM as the A operand of S^T Q^T, its fp32 master in registers,
// no state tile in shared memory, whose room then holds a third q, k, v buffer: tiles two
// chunks ahead; described at that loop).  With few (sequence, head) pairs each sequence is
// split into runs of whole chunks, one CTA each, run g starting from S0 + sum of K^T V over the
// chunks before it.  Where the workspace has room (it holds the work-queue rings for such
// shapes), that sum comes from a first launch (MODE 1: every run but the last computes its own
// sum_c K_c^T V_c, once) and the second launch (MODE 2) adds the sums of the runs before it to
// S0; without the room, each run rebuilds it from the chunks before it (MODE 0).
//
// NORM: normalised phi-linear attention (heqinghuang "gpt2-to-kimi" §07, engineermaxxing §02g):
// phi = elu + 1 is applied in place to the staged [K; Q] tile (elementwise, so the swizzle does
// not matter; the result is rounded to bf16, the operand type; key rows past the chunk's end
// are zeroed), and each output row is divided by
//   phi(q_r) . z_r + eps = phi(q_r) . z_entry + sum_{j <= r} (Q K^T)[r][j] + eps,
// the second term being the row sums of the masked score tile the kernel forms anyway (fp32,
// before its bf16 rounding) and the first a 128-term dot product per row.  The normaliser is
// the state's extra column: z - z0 = phi(K)^T 1 accumulates in TMEM by one more M = 128, N = 16
// MMA per chunk against a tile of ones (the same A operand as the state update), including over
// a run's prefix chunks.
#include <cuda.h>

#include "tc_common.cuh"

namespace gdr {
namespace tc {
namespace {

using namespace umma;

struct LinSmem {
  static constexpr uint32_t KQ = 0;            // [K; Q] x 2 buffers, 32 KB each
  static constexpr uint32_t VIN = 65536;       // V [64 tok][128] SW128 x 2 buffers, 16 KB each
  static constexpr uint32_t ZM = VIN + 32768;  // [Z; M]: zeros 8 KB, then M [64][64] K-major
  static constexpr uint32_t SS = ZM + 16384;   // S [d_k][128] (MN-major B) x 2 buffers, 32 KB each
                                                // (plain form: the third q, k, v buffer)
  static constexpr uint32_t ONES = SS + 65536;  // NORM: 16 x 64 bf16 ones (K-major B, N = 16)
  static constexpr uint32_t BARS = ONES + 2048;  // ld[2], s, q, m2, pf_full[4], pf_mma[4], TMEM,
                                                 // ld (third buffer)
  static constexpr uint32_t ZB = BARS + 128;    // NORM: z entering chunk i at [i & 1] (2 x 128 fp32)
  static constexpr uint32_t DP = ZB + 1024;     // NORM: denominator halves [i & 1][half][64 rows]
  static constexpr uint32_t END = DP + 1024;
  static constexpr size_t bytes = END + 1024;
  // prefix stages (32 KB each, K at +0 / +16K, V at +8K / +24K): dead before the chunk loop
  __host__ __device__ static constexpr uint32_t pf(int st) {
    return st == 0 ? KQ : st == 1 ? KQ + 32768 : st == 2 ? VIN : SS;
  }
  static_assert(bytes <= 232448, "shared memory per CTA");
};

constexpr uint32_t kColD0 = 128, kColD1 = 256, kColA = 384;  // TMEM columns (S at 0)
constexpr uint32_t kColZ = 448;  // NORM: phi(K)^T 1, 16 equal columns

// phi = elu + 1 for the bf16 operand tiles: x + 1 above zero, else e^x = 2^(x log2 e) on the
// hardware ex2 (flush-to-zero form), its argument held at -126 or above so phi stays a normal
// positive number (>= 2^-126; e^x itself for x >= -87.3)
__device__ __forceinline__ float phi_tc(float x) {
  float e;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(fmaxf(x * 1.44269504f, -126.f)));
  return x > 0.f ? x + 1.f : e;
}
__device__ __forceinline__ uint4 phi8(uint4 u) {
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(h[e]);
    h[e] = __floats2bfloat162_rn(phi_tc(f.x), phi_tc(f.y));
  }
  return u;
}

// phi on `chunks` 16-byte chunks of bf16 at p, in place (thread-strided, all loads first)
__device__ __forceinline__ void phi_tile(unsigned char* p, int chunks, int tid) {
  for (int i = tid; i < chunks; i += 4 * kThreads) {
    uint4 u[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (i + k * kThreads < chunks) u[k] = reinterpret_cast<uint4*>(p)[i + k * kThreads];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (i + k * kThreads < chunks) reinterpret_cast<uint4*>(p)[i + k * kThreads] = phi8(u[k]);
  }
}

// phi on a [K; Q] tile pair (2 slabs of 128 rows x 128 B), key rows >= n set to 0 instead;
// a thread's 8 chunks are loaded before any is converted
__device__ __forceinline__ void phi_kq(unsigned char* p, int n, int tid) {
  uint4 u[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) u[k] = reinterpret_cast<uint4*>(p)[tid + k * kThreads];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = tid + k * kThreads;
    const int row = (i & 1023) >> 3;
    reinterpret_cast<uint4*>(p)[i] =
        (row >= 64 || row < n) ? phi8(u[k]) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// run sums in the workspace: per (sequence, head, run < nseg - 1) the d_k x d_v fp32 sum of
// phi(K)^T V (or K^T V) over the run's chunks, then its d_k key sums (NORM)
constexpr int kDeltaFloats = kD * kD + kD;

template <bool NORM, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    linear_tc_kernel(const __grid_constant__ TcMaps maps, const PrefillArgs a, int nseg,
                     float* delta) {
  using L = LinSmem;
  constexpr int DH = kD / 2;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
  uint64_t* bar_ld = bars;        // [2] q, k, v of a chunk
  uint64_t* bar_s = bars + 2;     // the state MMA
  uint64_t* bar_q = bars + 3;     // the Q S and Q K^T MMAs
  uint64_t* bar_m2 = bars + 4;    // the M V MMA
  uint64_t* pf_full = bars + 5;   // [4] prefix stage loaded
  uint64_t* pf_mma = bars + 9;    // [4] prefix stage consumed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 13);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int H = a.H;
  const int nrun = MODE == 1 ? nseg - 1 : nseg;  // CTAs per (sequence, head)
  const int per_seq = H * nrun;
  const int rank = blockIdx.x / per_seq;
  const int h = (blockIdx.x % per_seq) / nrun, g = blockIdx.x % nrun;
  const int seq = a.order ? a.order[rank] : rank;
  int64_t t0, t1;
  if (!seq_range(a, seq, t0, t1)) return;
  const int nch = (int)((t1 - t0 + kC - 1) / kC);
  const int lseg = (nch + nseg - 1) / nseg;
  const int c_begin = g * lseg, c_end = min(nch, c_begin + lseg);
  if (g > 0 && c_begin >= c_end) return;
  // MODE 1: only a run followed by a non-empty run has a sum to hand on (all its chunks full)
  if (MODE == 1 && (c_begin >= c_end || c_end >= nch)) return;
  // the chunks summed into the state before the chunk loop: the run's own (MODE 1), the ones
  // before the run (MODE 0), none (MODE 2: the sums come from the workspace)
  const int p_lo = MODE == 1 ? c_begin : 0;
  const int p_hi = MODE == 1 ? c_end : MODE == 0 ? c_begin : 0;
  float* drun = MODE == 1 ? delta + (((size_t)seq * H + h) * (nseg - 1) + g) * kDeltaFloats
                          : nullptr;
  const size_t sidx = ((size_t)seq * H + h) * kD * kD;
  __nv_bfloat16* __restrict__ out = static_cast<__nv_bfloat16*>(a.out);

  if (warp == 0) tmem_alloc(tslot, kTmemCols);
  for (int i = tid; i < 8192 / 16; i += kThreads)  // the zero half of [Z; M]
    reinterpret_cast<uint4*>(sm + L::ZM)[i] = make_uint4(0, 0, 0, 0);
  if (NORM)
    for (int i = tid; i < 2048 / 16; i += kThreads)  // bf16 ones
      reinterpret_cast<uint4*>(sm + L::ONES)[i] =
          make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  fence_async_smem();
  if (tid == 0) {
    for (int i = 0; i < 15; ++i)
      if (i != 13) mbar_init(bars + i, 1);
    fence_mbar_init();
    prefetch_tmap(&maps.q_sw);
    prefetch_tmap(&maps.k_sw);
    prefetch_tmap(&maps.v);
  }
  cta_sync_tc();
  TcCtx x = make_ctx(sm, *tslot, bar_s);
  bool failed = false;
  if (MODE == 2 && g > 0) {  // S0 + the sums of the runs before this one
    float v[DH];
    const float* s0r = a.S0 ? a.S0 + sidx + (size_t)x.lrow * kD + x.wh * DH : nullptr;
#pragma unroll
    for (int j = 0; j < DH; ++j) v[j] = s0r ? s0r[j] : 0.f;
    for (int gp = 0; gp < g; ++gp) {
      const float* dr = delta + (((size_t)seq * H + h) * (nseg - 1) + gp) * kDeltaFloats +
                        (size_t)x.lrow * kD + x.wh * DH;
#pragma unroll
      for (int j = 0; j < DH; j += 4) {
        const float4 u = *reinterpret_cast<const float4*>(dr + j);
        v[j] += u.x, v[j + 1] += u.y, v[j + 2] += u.z, v[j + 3] += u.w;
      }
    }
    tmem_st_half<DH>(x.tm + x.lane_base + kColS + x.wh * DH, v);
#pragma unroll
    for (int j = 0; j < DH; j += 8) st_chunk8(sm + L::SS, 16384, x.lrow, x.wh * DH + j, v + j);
    tmem_wait_st();
    fence_async_smem();
  } else {
    s_init<DH>(x, MODE != 1 && a.S0 ? a.S0 + sidx + (size_t)x.lrow * kD : nullptr, sm + L::SS);
  }
  float* sZ = reinterpret_cast<float*>(sm + L::ZB);   // NORM: [2][128] z entering a chunk
  float* sDp = reinterpret_cast<float*>(sm + L::DP);  // NORM: [2][2 halves][64 rows]
  const size_t zidx = ((size_t)seq * H + h) * kD;
  float z0v = (NORM && MODE != 1 && tid < kD && a.z0) ? a.z0[zidx + tid] : 0.f;  // channel tid
  if (NORM && MODE == 2 && tid < kD)
    for (int gp = 0; gp < g; ++gp)
      z0v += delta[(((size_t)seq * H + h) * (nseg - 1) + gp) * kDeltaFloats + kD * kD + tid];
  bool zinit = false;  // kColZ holds a sum (an MMA has written it)
  const Opnd opOnes{x.sb + L::ONES, 2048, false};
  const uint32_t id_z = idesc_bf16(128, 16, false, true, false);  // phi(K)^T (MN-major A) x ones
  cta_sync_tc();  // every row of the bf16 state tile is written before the first MMA
  const uint32_t id_s = idesc_bf16(128, kD, false, true, true);   // K as MN-major A, V MN-major B
  const uint32_t id_d = idesc_bf16(128, kD, false, false, true);  // K-major A, MN-major B
  const uint32_t id_a = idesc_bf16(128, kC, false, false, false);  // [K; Q] K^T (K-major B)

  if (NORM && p_hi > p_lo) {
    // run prefix with the feature map: every thread waits for each stage and applies phi to its
    // K tile; warp 0 then issues S += phi(K)^T V and z += phi(K)^T 1
    cta_sync_tc();  // S0 is in TMEM
    bool pf_ok = true, mma_ok = true;
    uint32_t ph_f = 0, ph_m = 0;
    auto pf_issue = [&](int cp) {
      const int st = cp & 3;
      const int tc = (int)(t0 + (int64_t)(p_lo + cp) * kC);
      unsigned char* b = sm + L::pf(st);
      mbar_expect_tx(pf_full + st, 32768);
      tma_load_3d(b, &maps.k_sw, 0, h, tc, pf_full + st);
      tma_load_3d(b + 16384, &maps.k_sw, 64, h, tc, pf_full + st);
      tma_load_3d(b + 8192, &maps.v, 0, h, tc, pf_full + st);
      tma_load_3d(b + 24576, &maps.v, 64, h, tc, pf_full + st);
    };
    // a stage is made ready (loaded, phi on its K) while the previous stage's MMAs run
    auto stage_ready = [&](int cp) {
      const int st = cp & 3;
      const bool ok = mbar_wait(pf_full + st, (ph_f >> st) & 1u, kWaitNs);
      ph_f ^= 1u << st;
      if (ok) {
        phi_tile(sm + L::pf(st), 512, tid);          // K, channels 0-63
        phi_tile(sm + L::pf(st) + 16384, 512, tid);  // K, channels 64-127
        fence_async_smem();
      }
      return ok;
    };
    if (tid == 0)
      for (int cp = 0; cp < 3 && cp < p_hi - p_lo; ++cp) pf_issue(cp);
    bool ok = stage_ready(0);
#pragma unroll 1
    for (int cp = 0; cp < p_hi - p_lo; ++cp) {
      const int st = cp & 3;
      __syncwarp();
      // stage cp is ready on every thread; this barrier also orders every read of chunk
      // cp - 1's stage before its refill below
      if (__syncthreads_or(!ok || !mma_ok)) { pf_ok = false; break; }
      if (warp == 0) {
        const Opnd opK{x.sb + L::pf(st), 16384, true};
        const Opnd opV{x.sb + L::pf(st) + 8192, 16384, true};
        mma_run<kC>(x.tm + kColS, opK, opV, id_s, true);
        mma_run<kC>(x.tm + kColZ, opK, opOnes, id_z, cp > 0);  // z += phi(K)^T 1
        mma_commit_elect(pf_mma + st);
      }
      if (cp + 3 < p_hi - p_lo && tid == 0) {  // stage (cp + 3) & 3 held chunk cp - 1
        if (cp >= 1) {
          const int sp = (cp - 1) & 3;
          mma_ok = mbar_wait(pf_mma + sp, (ph_m >> sp) & 1u, kWaitNs);
          ph_m ^= 1u << sp;
        }
        if (mma_ok) pf_issue(cp + 3);
      }
      if (cp + 1 < p_hi - p_lo) ok = stage_ready(cp + 1);
    }
    if (warp == 0) mma_commit_elect(bar_s);  // every prefix MMA complete
    zinit = true;
    if (__syncthreads_or(!pf_ok) || !wait_bar(bar_s, x.ph_mma)) {
      failed = true;
    } else {
      s_epilogue<DH>(x, sm + L::SS);
      cta_sync_tc();
    }
  } else if (p_hi > p_lo) {
    // run prefix: S += K_c^T V_c over chunks [p_lo, p_hi) (all full), 4 TMA stages, one chunk's
    // MMA per step; warp 0 drives it, the other warps wait at the barrier below
    cta_sync_tc();  // S0 is in TMEM
    bool pf_ok = true;
    if (warp == 0) {
      auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
        bool ok = true;
        if ((tid & 31) == 0) ok = mbar_wait(bar, parity, kWaitNs);
        return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      };
      uint32_t ph_f = 0, ph_m = 0;
      auto pf_issue = [&](int cp) {
        if (tid == 0) {
          const int st = cp & 3;
          const int tc = (int)(t0 + (int64_t)(p_lo + cp) * kC);
          unsigned char* b = sm + L::pf(st);
          mbar_expect_tx(pf_full + st, 32768);
          tma_load_3d(b, &maps.k_sw, 0, h, tc, pf_full + st);
          tma_load_3d(b + 16384, &maps.k_sw, 64, h, tc, pf_full + st);
          tma_load_3d(b + 8192, &maps.v, 0, h, tc, pf_full + st);
          tma_load_3d(b + 24576, &maps.v, 64, h, tc, pf_full + st);
        }
      };
      for (int cp = 0; cp < 3 && cp < p_hi - p_lo; ++cp) pf_issue(cp);
#pragma unroll 1
      for (int cp = 0; cp < p_hi - p_lo; ++cp) {
        const int st = cp & 3;
        if (!warp_wait(pf_full + st, (ph_f >> st) & 1u)) { pf_ok = false; break; }
        ph_f ^= 1u << st;
        const Opnd opK{x.sb + L::pf(st), 16384, true};
        const Opnd opV{x.sb + L::pf(st) + 8192, 16384, true};
        mma_run<kC>(x.tm + kColS, opK, opV, id_s, true);
        mma_commit_elect(pf_mma + st);
        if (cp + 3 < p_hi - p_lo) {  // stage (cp + 3) & 3 held chunk cp - 1: its MMA must be done
          if (cp >= 1) {
            const int sp = (cp - 1) & 3;
            if (!warp_wait(pf_mma + sp, (ph_m >> sp) & 1u)) { pf_ok = false; break; }
            ph_m ^= 1u << sp;
          }
          pf_issue(cp + 3);
        }
      }
      mma_commit_elect(bar_s);  // every prefix MMA complete
    }
    if (__syncthreads_or(!pf_ok) || !wait_bar(bar_s, x.ph_mma)) {
      failed = true;
    } else {
      s_epilogue<DH>(x, sm + L::SS);  // the bf16 operand copy of the run's entering state
      cta_sync_tc();
    }
  }

  if (MODE == 1) {  // hand the run's sums on through the workspace
    if (failed) {
      if (tid == 0) report(a, GDR_DEVCHECK_TIMEOUT);
    } else {
      s_final<DH>(x, drun + (size_t)x.lrow * kD);
      if (NORM && warp < 4) drun[kD * kD + tid] = tmem_ld1(x.tm + x.lane_base + kColZ);
    }
    cta_sync_tc();
    if (warp == 0) tmem_dealloc(x.tm, kTmemCols);
    return;
  }
  const int64_t ts = t0 + (int64_t)c_begin * kC;
  const int64_t te = t0 + (int64_t)c_end * kC < t1 ? t0 + (int64_t)c_end * kC : t1;
  const int nloc = c_end - c_begin;
  auto issue_ld = [&](int i) {  // chunk c_begin + i into buffer i & 1
    if (tid == 0) {
      const int b = i & 1;
      const int tc = (int)(ts + (int64_t)i * kC);
      unsigned char* kq = sm + L::KQ + b * 32768;
      unsigned char* vv = sm + L::VIN + b * 16384;
      mbar_expect_tx(bar_ld + b, 32768 + 16384);
      tma_load_3d(kq, &maps.k_sw, 0, h, tc, bar_ld + b);
      tma_load_3d(kq + 8192, &maps.q_sw, 0, h, tc, bar_ld + b);
      tma_load_3d(kq + 16384, &maps.k_sw, 64, h, tc, bar_ld + b);
      tma_load_3d(kq + 24576, &maps.q_sw, 64, h, tc, bar_ld + b);
      tma_load_3d(vv, &maps.v, 0, h, tc, bar_ld + b);
      tma_load_3d(vv + 8192, &maps.v, 64, h, tc, bar_ld + b);
    }
  };
  const bool o_rows = (warp & 3) >= 2;  // TMEM lanes 64-127 (Q rows) of this warp
  const int qrow = (warp & 3) * 32 + (tid & 31) - 64;
  auto d_col = [](int i) { return (i & 1) ? kColD1 : kColD0; };

  if constexpr (!NORM) {
    // ---- The runs without the normaliser, transposed: the state is kept as S^T (the thread of
    // TMEM lane v holds value column v; its fp32 master in registers, 64 key channels per thread,
    // two threads per lane) so that its bf16 copy in TMEM is the A operand of O^T = S^T Q^T, and
    // no state tile goes through shared memory.  Per chunk (one CTA, every product M = 128):
    //   [K; Q] K^T (its rows 64-127: Q K^T) -> M = lower(Q K^T) in shared memory,
    //   X = V^T K,   O^T = S^T Q^T,   then   O^T += V^T M^T,   S^T <- S^T + X (registers).
    // The previous chunk's O^T columns are stored by warps 4-7 (one bf16 value per lane and
    // token) while this chunk's tiles are awaited and its products run.  With no state tile in
    // shared memory its room holds a third q, k, v buffer, so tiles are requested two chunks
    // ahead.
    constexpr uint32_t cSB = 0, cD0 = 64, cD1 = 192, cX = 320, cA = 448;
    const int lane = tid & 31;
    const int vv = (warp & 3) * 32 + lane;  // the value column of this thread's TMEM lane
    float ms[64];                            // S^T[vv][64 wh + j]
    {  // the entering state (TMEM [k][v] fp32) -> shared memory -> this thread's registers
      float* sS = reinterpret_cast<float*>(sm + L::SS);  // [128][128] fp32, columns XOR-swizzled
      if (!failed) {
        float v[64];
        tmem_ld64(x.tm + x.lane_base + kColS + x.wh * 64, v);
#pragma unroll
        for (int j = 0; j < 64; ++j) sS[x.lrow * kD + ((x.wh * 64 + j) ^ (x.lrow & 31))] = v[j];
      }
      cta_sync_tc();
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const int k = x.wh * 64 + j;
        ms[j] = sS[k * kD + (vv ^ (k & 31))];
      }
      float pv[32];
#pragma unroll
      for (int i2 = 0; i2 < 32; ++i2) {
        const __nv_bfloat162 hv = __floats2bfloat162_rn(ms[2 * i2], ms[2 * i2 + 1]);
        pv[i2] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&hv));
      }
      tmem_st32(x.tm + x.lane_base + cSB + 32 * x.wh, pv);
      tmem_wait_st();
      cta_sync_tc();
    }
    const uint32_t id_vk = idesc_bf16(128, kD, false, true, true);     // V^T (smem) K (MN-major)
    const uint32_t id_t64 = idesc_bf16(128, kC, false, false, false);  // TMEM A, K-major B
    const uint32_t id_vm = idesc_bf16(128, kC, false, true, false);    // V^T (smem) M^T
    auto dcol = [](int i) { return (i & 1) ? cD1 : cD0; };
    // warps 4-7: O^T of local chunk i (columns 64-127 of its D^T) -> out rows [tc, tc + n)
    auto o_drain = [&](int i, int64_t tc, int n) {
      float o[64];
      tmem_ld64(x.tm + x.lane_base + dcol(i) + 64, o);
      __nv_bfloat16* dst = out + ((size_t)tc * H + h) * kD + vv;
#pragma unroll
      for (int j = 0; j < 64; ++j)
        if (j < n) dst[(size_t)j * H * kD] = __float2bfloat16_rn(o[j]);
    };
    // (bar_s continues from the run prefix's phase; the others are fresh)
    uint32_t ph_ld3 = 0, ph_x = x.ph_mma, ph_a = 0, ph_o = 0;  // ph_ld3: bit b for buffer b
    uint32_t ld_pending = 0;  // bit b: buffer b's tiles requested and not yet waited for
    auto kq_of = [](int bb) -> uint32_t { return bb == 0 ? L::KQ : bb == 1 ? L::KQ + 32768 : L::SS; };
    auto v_of = [](int bb) -> uint32_t {
      return bb == 0 ? L::VIN : bb == 1 ? L::VIN + 16384 : L::SS + 32768;
    };
    auto ldbar = [&](int bb) { return bb == 2 ? bars + 14 : bar_ld + bb; };
    auto issue_ld3 = [&](int i) {  // chunk c_begin + i into buffer i % 3
      const int bb = i % 3;
      if (tid == 0) {
        const int tc = (int)(ts + (int64_t)i * kC);
        unsigned char* kq = sm + kq_of(bb);
        unsigned char* vt = sm + v_of(bb);
        mbar_expect_tx(ldbar(bb), 32768 + 16384);
        tma_load_3d(kq, &maps.k_sw, 0, h, tc, ldbar(bb));
        tma_load_3d(kq + 8192, &maps.q_sw, 0, h, tc, ldbar(bb));
        tma_load_3d(kq + 16384, &maps.k_sw, 64, h, tc, ldbar(bb));
        tma_load_3d(kq + 24576, &maps.q_sw, 64, h, tc, ldbar(bb));
        tma_load_3d(vt, &maps.v, 0, h, tc, ldbar(bb));
        tma_load_3d(vt + 8192, &maps.v, 64, h, tc, ldbar(bb));
      }
      ld_pending |= 1u << bb;
    };
    if (!failed) {
      for (int i = 0; i < 2 && i < nloc; ++i) issue_ld3(i);
    }
#pragma unroll 1
    for (int i = 0; i < nloc && !failed; ++i) {
      const int b = i % 3;
      const int64_t tc = ts + (int64_t)i * kC;
      const int n = (int)((te - tc) < (int64_t)kC ? (te - tc) : (int64_t)kC);
      {
        const bool ok = mbar_wait(ldbar(b), (ph_ld3 >> b) & 1u, kWaitNs);
        ph_ld3 ^= 1u << b;
        ld_pending &= ~(1u << b);
        if (ok && n < kC) zero_v_tail<kD>(x, sm + v_of(b), n);  // padded rows: no V^T K
        if (__syncthreads_or(!ok)) { failed = true; break; }
        fence_after_sync();
      }
      // buffer (i + 2) % 3 held chunk i - 1, whose products are complete
      if (i + 2 < nloc) issue_ld3(i + 2);
      const uint32_t kqa = x.sb + kq_of(b);
      const Opnd opKQ{kqa, 16384, false};         // [K; Q], K-major A
      const Opnd opKb{kqa, 16384, false};         // K rows, K-major B
      const Opnd opKm{kqa, 16384, true};          // K, MN-major B (N = d_k)
      const Opnd opQ{kqa + 8192, 16384, false};   // Q rows, K-major B
      const Opnd opVa{x.sb + v_of(b), 8192, true};  // V^T, MN-major A
      const Opnd opM{x.sb + L::ZM + 8192, 8192, false};                // M rows, K-major B
      bool bad = false;
      if (warp == 0) {
        mma_run<kD>(x.tm + cA, opKQ, opKb, id_a, false);  // [K; Q] K^T
        mma_commit_elect(bar_q);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // X = V^T K
          mma_bf16_elect(x.tm + cX, opVa.at(16 * ks), opKm.at(16 * ks), id_vk, ks > 0 ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)  // O^T = S^T Q^T
          mma_bf16_tmem_a_elect(x.tm + dcol(i) + 64, x.tm + cSB + 8 * ks, opQ.at(16 * ks), id_t64,
                                ks > 0 ? 1u : 0u);
        mma_commit_elect(bar_s);  // X and S^T Q^T: the state copy may be rewritten after it
      }
      // while those products run: warps 4-7 store the previous chunk's O^T columns; M =
      // lower(Q K^T) (Q rows: TMEM lanes 64-127) becomes bf16 K-major rows, key columns 0-31 by
      // warps 2-3 at once and 32-63 by warps 6-7 after their stores
      if (i > 0 && x.wh == 1) o_drain(i - 1, tc - kC, kC);
      if (o_rows) {
        bad |= !mbar_wait(bar_q, ph_a, kWaitNs);
        __syncwarp();
        fence_after_sync();
        float v[32];
        tmem_ld32(x.tm + x.lane_base + cA + 32 * x.wh, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = (32 * x.wh + j <= qrow) ? v[j] : 0.f;
#pragma unroll
        for (int j = 0; j < 32; j += 8) st_chunk8(sm + L::ZM + 8192, 8192, qrow, 32 * x.wh + j, v + j);
        fence_async_smem();
      }
      ph_a ^= 1u;
      bad |= !mbar_wait(bar_s, ph_x, kWaitNs);
      ph_x ^= 1u;
      __syncwarp();
      fence_after_sync();
      {  // S^T <- S^T + X on this thread's 64 key channels, and its bf16 copy
        float xv[64];
        tmem_ld64(x.tm + x.lane_base + cX + x.wh * 64, xv);
        float pv[32];
#pragma unroll
        for (int j = 0; j < 64; ++j) ms[j] += xv[j];
#pragma unroll
        for (int i2 = 0; i2 < 32; ++i2) {
          const __nv_bfloat162 hv = __floats2bfloat162_rn(ms[2 * i2], ms[2 * i2 + 1]);
          pv[i2] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&hv));
        }
        tmem_st32(x.tm + x.lane_base + cSB + 32 * x.wh, pv);
        tmem_wait_st();
      }
      fence_before_sync();
      __syncthreads();  // M and the state copy are written
      fence_after_sync();
      if (warp == 0) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // O^T += V^T M^T
          mma_bf16_elect(x.tm + dcol(i) + 64, opVa.at(16 * ks), opM.at(16 * ks), id_vm, 1u);
        mma_commit_elect(bar_m2);
      }
      // buffer b and M are reused only after that product completes
      if (tid == 0) bad |= !mbar_wait(bar_m2, ph_o, kWaitNs);
      __syncwarp();
      ph_o ^= 1u;
      fence_before_sync();
      if (__syncthreads_or(bad)) { failed = true; break; }
      fence_after_sync();
    }
    if (!failed && nloc > 0 && x.wh == 1) {
      const int64_t tl = ts + (int64_t)(nloc - 1) * kC;
      o_drain(nloc - 1, tl, (int)(te - tl));
    }
    if (failed) {
      if (tid == 0) report(a, GDR_DEVCHECK_TIMEOUT);
      // let copies already in flight land before the shared memory is released
      for (int bb = 0; bb < 3; ++bb)
        if ((ld_pending >> bb) & 1u) mbar_wait(ldbar(bb), (ph_ld3 >> bb) & 1u, kWaitNs);
    } else if (a.S_final && c_end == nch) {  // the last run of the sequence hands the state on
#pragma unroll
      for (int j = 0; j < 64; ++j) a.S_final[sidx + (size_t)(x.wh * 64 + j) * kD + vv] = ms[j];
    }
    cta_sync_tc();
    if (warp == 0) tmem_dealloc(x.tm, kTmemCols);
    return;
  }
  // O rows of local chunk i (lanes 64-127 of its D) -> out rows [tc, tc + n) of head h
  auto o_store = [&](int i, int64_t tc, int n) {
    float v[64];
    tmem_ld64(x.tm + x.lane_base + d_col(i) + x.wh * 64, v);
    if (NORM && qrow < n) {  // divide by phi(q_r) . z_r + eps
      const float* dp = sDp + (i & 1) * 128;
      const float inv = 1.f / (dp[qrow] + dp[64 + qrow] + a.eps);
#pragma unroll
      for (int j = 0; j < 64; ++j) v[j] *= inv;
    }
    if (qrow < n) {
      __nv_bfloat16* dst = out + ((size_t)(tc + qrow) * H + h) * kD + x.wh * 64;
#pragma unroll
      for (int j = 0; j < 64; j += 8) {
        __align__(16) __nv_bfloat162 hv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) hv[k] = __floats2bfloat162_rn(v[j + 2 * k], v[j + 2 * k + 1]);
        *reinterpret_cast<uint4*>(dst + j) = *reinterpret_cast<const uint4*>(hv);
      }
    }
  };
  uint32_t ph_ld[2] = {0, 0}, ph_q = 0, ph_m2 = 0;
  // NORM: wait for chunk j's tiles, zero its V tail, apply phi to its [K; Q] tile (all threads)
  bool next_ok = true;
  auto make_ready = [&](int j) {
    const int bj = j & 1;
    const int64_t tcj = ts + (int64_t)j * kC;
    const int nj = (int)((te - tcj) < (int64_t)kC ? (te - tcj) : (int64_t)kC);
    const bool ok = mbar_wait(bar_ld + bj, ph_ld[bj], kWaitNs);
    ph_ld[bj] ^= 1u;
    if (ok) {
      if (nj < kC) zero_v_tail<kD>(x, sm + L::VIN + bj * 16384, nj);
      phi_kq(sm + L::KQ + bj * 32768, nj, tid);
      fence_async_smem();
    }
    return ok;
  };
  if (!failed && nloc > 0) issue_ld(0);
#pragma unroll 1
  for (int i = 0; i < nloc && !failed; ++i) {
    const int b = i & 1;
    const int64_t tc = ts + (int64_t)i * kC;
    const int n = (int)((te - tc) < (int64_t)kC ? (te - tc) : (int64_t)kC);
    if (NORM) {
      // the chunk's tiles were made ready (loaded, tail zeroed, phi applied) while the previous
      // chunk's last MMA ran; z entering the chunk = z0 + the ones-column sum (final since the
      // previous chunk's m2 wait, or the prefix's bar_s wait)
      if (i == 0) next_ok = make_ready(0);
      if (warp < 4)
        sZ[(i & 1) * kD + tid] = z0v + (zinit ? tmem_ld1(x.tm + x.lane_base + kColZ) : 0.f);
      fence_before_sync();
      if (__syncthreads_or(!next_ok)) { failed = true; break; }
      fence_after_sync();
    } else {
      const bool ok = mbar_wait(bar_ld + b, ph_ld[b], kWaitNs);
      ph_ld[b] ^= 1u;
      if (ok && n < kC) zero_v_tail<kD>(x, sm + L::VIN + b * 16384, n);  // padded rows: no K^T V
      if (__syncthreads_or(!ok)) { failed = true; break; }
      fence_after_sync();
    }
    if (i + 1 < nloc) issue_ld(i + 1);  // buffer b ^ 1: chunk i - 1's MMAs are complete
    const Opnd opKQ{x.sb + L::KQ + b * 32768, 16384, false};  // [K; Q], K-major A (M = 128)
    const Opnd opKa{x.sb + L::KQ + b * 32768, 16384, true};   // K as MN-major A (M = d_k)
    const Opnd opKb{x.sb + L::KQ + b * 32768, 16384, false};  // K rows as K-major B (N = 64)
    const Opnd opV{x.sb + L::VIN + b * 16384, 8192, true};
    const Opnd opS{x.sb + L::SS + b * 32768, 16384, true};    // this chunk's entering S
    const Opnd opZM{x.sb + L::ZM, 16384, false};
    if (warp == 0) {
      mma_run<kC>(x.tm + kColS, opKa, opV, id_s, true);  // S += K^T V
      mma_commit_elect(bar_s);
      mma_run<kD>(x.tm + d_col(i), opKQ, opS, id_d, false);  // [K; Q] S
      mma_run<kD>(x.tm + kColA, opKQ, opKb, id_a, false);    // [K; Q] K^T
      mma_commit_elect(bar_q);
    }
    if (i > 0 && o_rows) o_store(i - 1, tc - kC, kC);
    float qz = 0.f;  // NORM: this thread's half of phi(q_r) . z_entry, off the M-step path
    if (NORM && o_rows) {
      const unsigned char* qp = sm + L::KQ + b * 32768 + x.wh * 16384 + (64 + qrow) * 128;
      const float* z = sZ + (i & 1) * kD + 64 * x.wh;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        float q8[8];
        ld_bf16x8(reinterpret_cast<const __nv_bfloat16*>(qp + ((ch ^ (qrow & 7)) << 4)), q8);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e & 3] = fmaf(q8[e], z[8 * ch + e], acc[e & 3]);
      }
      qz = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
    // the state's bf16 operand for the next chunk (the other buffer: this chunk's Q S reads this)
    if (!wait_bar(bar_s, x.ph_mma)) { failed = true; break; }
    s_epilogue<DH>(x, sm + L::SS + (b ^ 1) * 32768);
    if (!wait_bar(bar_q, ph_q)) { failed = true; break; }
    if (o_rows) {  // M = lower(Q K^T) -> bf16 K-major A rows 64-127 of [Z; M]
      float v[32];
      tmem_ld32(x.tm + x.lane_base + kColA + 32 * x.wh, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = (32 * x.wh + j <= qrow) ? v[j] : 0.f;
      if (NORM) {  // this half's share of phi(q_r) . z_r: masked score sum + phi(q_r) . z_entry
        float rs[4] = {qz, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 32; ++j) rs[j & 3] += v[j];
        sDp[(i & 1) * 128 + x.wh * 64 + qrow] = (rs[0] + rs[1]) + (rs[2] + rs[3]);
      }
#pragma unroll
      for (int j = 0; j < 32; j += 8) st_chunk8(sm + L::ZM + 8192, 8192, qrow, 32 * x.wh + j, v + j);
      fence_async_smem();
    }
    cta_sync_tc();
    if (warp == 0) {
      mma_run<kC>(x.tm + d_col(i), opZM, opV, id_d, true);  // rows 64-127 += M V
      // NORM: z += phi(K)^T 1 here, off the chain of the chunk's other MMAs (read at the next
      // chunk's top, after the m2 wait)
      if (NORM) mma_run<kC>(x.tm + kColZ, opKa, opOnes, id_z, zinit);
      mma_commit_elect(bar_m2);
    }
    zinit = true;
    // NORM: the next chunk's tiles (buffer b ^ 1, loaded since this chunk began) made ready
    // while that MMA runs
    if (NORM && i + 1 < nloc) next_ok = make_ready(i + 1);
    // buffer b (q, k, v) and M are reused only after this MMA completes
    if (!wait_bar(bar_m2, ph_m2)) { failed = true; break; }
  }
  if (!failed && nloc > 0 && o_rows) {
    const int64_t tl = ts + (int64_t)(nloc - 1) * kC;
    o_store(nloc - 1, tl, (int)(te - tl));
  }
  if (failed) {
    if (tid == 0) report(a, GDR_DEVCHECK_TIMEOUT);
    // let copies already in flight land before the shared memory is released
    mbar_wait(bar_ld, ph_ld[0], kWaitNs);
    mbar_wait(bar_ld + 1, ph_ld[1], kWaitNs);
  } else {
    if (a.S_final && c_end == nch)  // the last run of the sequence hands the state on
      s_final<DH>(x, a.S_final + sidx + (size_t)x.lrow * kD);
    if (NORM && a.z_final && c_end == nch && warp < 4) {
      const float zt = zinit ? tmem_ld1(x.tm + x.lane_base + kColZ) : 0.f;
      a.z_final[zidx + tid] = z0v + zt;
    }
  }
  cta_sync_tc();
  if (warp == 0) tmem_dealloc(x.tm, kTmemCols);
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

}  // namespace

cudaError_t launch_linear_tc(const gdr_shape& sh, const PrefillArgs& a, const TcMaps& maps,
                             bool norm, cudaStream_t s) {
  // few (sequence, head) pairs: runs of at least 16 chunks per CTA, as many as fill the SMs once
  const long pairs = (long)sh.n_seqs * sh.H;
  const long avg_chunks = sh.total_tokens / ((long)sh.n_seqs * kC);
  long nseg = pairs > 0 ? sm_count() / pairs : 1;
  if (nseg > avg_chunks / 16) nseg = avg_chunks / 16;
  if (nseg > 8) nseg = 8;
  // an in-place hand-off (S_final = S0) keeps one run per sequence: a later run reads S0 while
  // the last run of the same sequence writes S_final
  if (nseg < 1 || (a.S0 && a.S0 == a.S_final)) nseg = 1;
  // the runs' sums through the workspace where its work-queue area holds them
  const size_t need = (size_t)pairs * (size_t)(nseg - 1) * kDeltaFloats * sizeof(float);
  const size_t room = a.ring ? (size_t)WorkspaceLayout::ring_pairs(sh) *
                                   WorkspaceLayout::kRingSlots * WorkspaceLayout::kRingSlotBytes
                             : 0;
  const bool two = nseg > 1 && need <= room;
  float* delta = two ? reinterpret_cast<float*>(a.ring) : nullptr;
  auto k0 = norm ? linear_tc_kernel<true, 0> : linear_tc_kernel<false, 0>;
  auto k1 = norm ? linear_tc_kernel<true, 1> : linear_tc_kernel<false, 1>;
  auto k2 = norm ? linear_tc_kernel<true, 2> : linear_tc_kernel<false, 2>;
  for (auto kern : {k0, k1, k2}) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)LinSmem::bytes);
    if (e != cudaSuccess) return e;
  }
  const unsigned grid = (unsigned)sh.n_seqs * (unsigned)sh.H * (unsigned)nseg;
  if (two) {
    const unsigned grid1 = (unsigned)sh.n_seqs * (unsigned)sh.H * (unsigned)(nseg - 1);
    k1<<<grid1, kThreads, LinSmem::bytes, s>>>(maps, a, (int)nseg, delta);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k2<<<grid, kThreads, LinSmem::bytes, s>>>(maps, a, (int)nseg, delta);
  } else {
    k0<<<grid, kThreads, LinSmem::bytes, s>>>(maps, a, (int)nseg, nullptr);
  }
  return cudaGetLastError();
}

}  // namespace tc
}  // namespace gdr
