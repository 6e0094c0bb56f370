// prefill_simt.cu -- chunked prefill of the gated delta rule (and of plain linear attention) in
// fp32 FFMA.  This is the exact-arithmetic path: fp32 inputs, d = 64, and the cross-check of the
// tensor-core path.
//
// Chunk algebra (derived from the recurrence; the alpha = 1 case is the per-chunk triangular
// solve of engineermaxxing "From GPT-2 to Kimi K3: one memory, seven eviction policies" §04e-§04f
// and heqinghuang "gpt2-to-kimi" §10; the decay products folded through it are the survival
// products of engineermaxxing §05d / heqinghuang §11, one per key channel as in dev.to "From
// GPT-2 to Kimi K3: How Language Models Learned to Manage Memory" §5).  For a chunk of n <= C
// tokens, local index r, entering state S (d_k x d_v), with G_r = sum_{m <= r} log(alpha_m)
// (per key channel, clamped at -60 per token):
//   A[r][j] = beta_r sum_c k_r[c] k_j[c] e^{G_r[c] - G_j[c]}   (j < r)
//   M[r][j] =        sum_c q_r[c] k_j[c] e^{G_r[c] - G_j[c]}   (j <= r)
//   (I + A) [W | U~] = diag(beta) [K * e^G | V]                (forward substitution)
//   U = U~ - W S;   O = (Q * e^G) S + M U;   S <- Diag(e^{G_n}) S + (K * e^{G_n - G})^T U
// Plain linear attention: O = Q S + tril(Q K^T) V;  S <- S + K^T V.
// Gated linear attention (no erase, no beta): U = V, the rest as the gated rule:
//   O = (Q * e^G) S + M V;  S <- Diag(e^{G_n}) S + (K * e^{G_n - G})^T V.
//
// Mapping: one CTA (256 threads) per (sequence, head, block of DVB value columns); the columns
// of S are independent (v and U enter column-wise), so the value dimension splits across CTAs
// with no communication.  Each CTA walks its sequence's chunks in order; the state block lives
// in shared memory for the whole walk.  All pair decays e^{G_r - G_j} are formed directly (no
// factorisation) when the chunk's decay is strong; otherwise as the products of e^{G_r} and
// e^{-G_j}, which are then far inside the fp32 range.  G is kept as an unevaluated sum hi + lo
// (the error of every addition carried in lo), so a difference G_r - G_j is as accurate as its
// own size allows, whatever the size of G after a reset; with the accurate logf and expf this
// makes any alpha in [0, 1] exact to fp32 rounding.
#include "gdr_internal.cuh"

namespace gdr {
namespace {

constexpr int kSimtThreads = 256;
constexpr int kDVB = 32;  // value columns per CTA

template <int D, int C>
struct SimtSmem {
  static constexpr int LD = D + 1;      // row stride of [C][D] tiles (conflict-free columns)
  static constexpr int LX = D + kDVB + 1;
  static constexpr int LC = C + 1;
  static constexpr int LV = kDVB + 1;
  static constexpr int off_Q = 0;
  static constexpr int off_K = off_Q + C * LD;
  static constexpr int off_Kh = off_K + C * LD;
  static constexpr int off_G = off_Kh + C * LD;   // G, rounded part (hi)
  static constexpr int off_Gl = off_G + C * LD;   // G, rounding error of hi (lo)
  static constexpr int off_X = off_Gl + C * LD;
  static constexpr int off_A = off_X + C * LX;
  static constexpr int off_M = off_A + C * LC;
  static constexpr int off_S = off_M + C * LC;
  static constexpr int off_V = off_S + D * LV;
  static constexpr int off_U = off_V + C * LV;
  static constexpr int off_B = off_U + C * LV;
  static constexpr int off_Gam = off_B + C;
  static constexpr int off_Z = off_Gam + D;    // the normaliser z (normalised linear attention)
  static constexpr int off_Flag = off_Z + D;   // the chunk's decay is weak enough to factorise
  static constexpr int total_floats = off_Flag + 4;
  static constexpr size_t bytes = (size_t)total_floats * 4;
};

template <int D, int C, typename T, bool CHANNEL, int KIND>
__global__ void __launch_bounds__(kSimtThreads) prefill_simt_kernel(PrefillArgs a) {
  using L = SimtSmem<D, C>;
  constexpr int NB = D / kDVB;
  constexpr bool NORM = KIND == kKindNormLinear;        // phi features, normaliser z
  constexpr bool LINEAR = KIND == kKindLinear || NORM;  // no gates
  constexpr bool ERASE = KIND == kKindDelta;    // the delta rule's correction (solve, beta)
  extern __shared__ float sm[];
  float* sQ = sm + L::off_Q;
  float* sK = sm + L::off_K;
  float* sKh = sm + L::off_Kh;
  float* sG = sm + L::off_G;
  float* sGl = sm + L::off_Gl;
  int* sFlag = reinterpret_cast<int*>(sm + L::off_Flag);
  float* sX = sm + L::off_X;
  float* sA = sm + L::off_A;
  float* sM = sm + L::off_M;
  float* sS = sm + L::off_S;
  float* sV = sm + L::off_V;
  float* sU = sm + L::off_U;
  float* sB = sm + L::off_B;
  float* sGam = sm + L::off_Gam;
  float* sZ = sm + L::off_Z;
  float* sDen = sB;  // normalised linear attention: the chunk's denominators (no beta there)

  const int tid = threadIdx.x;
  const int H = a.H;
  const int rank = blockIdx.x / (H * NB);
  const int rem = blockIdx.x % (H * NB);
  const int h = rem / NB, vb = rem % NB;
  const int seq = a.order ? a.order[rank] : rank;
  int64_t t0, t1;
  if (!seq_range(a, seq, t0, t1)) return;

  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  T* out = static_cast<T*>(a.out);
  const int vc0 = vb * kDVB;
  const size_t sidx = ((size_t)seq * H + h) * D * D;

  // entering state block [D][DVB] (and the whole normaliser z: every value block keeps a copy)
  if (NORM)
    for (int c = tid; c < D; c += kSimtThreads)
      sZ[c] = a.z0 ? a.z0[((size_t)seq * H + h) * D + c] : 0.f;
  for (int i = tid; i < D * kDVB; i += kSimtThreads) {
    const int r = i / kDVB, c = i % kDVB;
    sS[r * L::LV + c] = a.S0 ? a.S0[sidx + (size_t)r * D + vc0 + c] : 0.f;
  }

  for (int64_t tc = t0; tc < t1; tc += C) {
    const int n = (int)(t1 - tc < (int64_t)C ? t1 - tc : (int64_t)C);
    __syncthreads();  // previous chunk fully consumed
    // ---- 1. load the chunk (rows >= n: q = k = v = 0, alpha = 1, beta = 0)
    for (int i = tid; i < C * D; i += kSimtThreads) {
      const int r = i / D, c = i % D;
      const bool ok = r < n;
      const size_t o = ((size_t)(tc + r) * H + h) * D + c;
      float qv = ok ? to_f32(q[o]) : 0.f, kv = ok ? to_f32(k[o]) : 0.f;
      if (a.prologue) qv = silu_f(qv), kv = silu_f(kv);  // normalised below
      if (NORM && ok) qv = phi_f(qv), kv = phi_f(kv);    // rows >= n stay 0: no write, no z
      sQ[r * L::LD + c] = qv;
      sK[r * L::LD + c] = kv;
      if (!LINEAR) {
        float g = 0.f;
        if (ok) {
          const float al = CHANNEL ? a.alpha[o] : a.alpha[(size_t)(tc + r) * H + h];
          g = fmaxf(logf(a.prologue ? sigmoid_f(al) : al), kLogAlphaMin);
        }
        sG[r * L::LD + c] = g;
      }
    }
    for (int i = tid; i < C * kDVB; i += kSimtThreads) {
      const int r = i / kDVB, c = i % kDVB;
      sV[r * L::LV + c] = r < n ? to_f32(v[((size_t)(tc + r) * H + h) * D + vc0 + c]) : 0.f;
    }
    if (ERASE && tid < C) {
      const float b = tid < n ? a.beta[(size_t)(tc + tid) * H + h] : 0.f;
      sB[tid] = a.prologue && tid < n ? sigmoid_f(b) : b;
    }
    __syncthreads();
    if (a.prologue) {
      // the layer prologue's L2 normalisation of the silu rows of q and k: one warp per row
      // (heqinghuang "gpt2-to-kimi" §09); zero rows stay zero
      const int warp = tid >> 5, lane = tid & 31;
      for (int rw = warp; rw < 2 * C; rw += kSimtThreads / 32) {
        float* row = (rw < C ? sQ : sK) + (rw % C) * L::LD;
        float ss = 0.f;
        for (int c = lane; c < D; c += 32) ss = fmaf(row[c], row[c], ss);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float inv = inv_norm(ss);
        for (int c = lane; c < D; c += 32) row[c] *= inv;
      }
      __syncthreads();
    }

    bool factor = false;  // pair decays as e^{G_r} e^{-G_j} (weak decay) or directly
    if (!LINEAR) {
      // ---- 2. in-chunk inclusive prefix sums of the log-gates, per key channel, as hi + lo
      // (two-sum: lo collects the rounding error of every addition)
      if (tid == 0) *sFlag = 1;
      __syncthreads();
      for (int c = tid; c < D; c += kSimtThreads) {
        float hi = 0.f, lo = 0.f;
        for (int r = 0; r < C; ++r) {
          const float g = sG[r * L::LD + c];
          const float s2 = hi + g;
          const float bb = s2 - hi;
          lo += (hi - (s2 - bb)) + (g - bb);
          hi = s2;
          sG[r * L::LD + c] = hi;
          sGl[r * L::LD + c] = lo;
        }
        if (hi + lo < -80.f) *sFlag = 0;  // e^{-G} would leave the comfortable fp32 range
      }
      __syncthreads();
      factor = *sFlag != 0;
    }
    // e^{G_r} from its two parts: expf of the exact hi, times (1 + lo)
    auto eG = [&](int r, int c, float sign) {
      const float e = expf(sign * sG[r * L::LD + c]);
      return fmaf(e, sign * sGl[r * L::LD + c], e);
    };

    if (factor) {
      // ---- 3a. weak decay: the gate-scaled operands first (beta K~ into the solve's right-hand
      // side, Q~ in place, Kr = K e^{-G} into the K^ tile), then plain products below
      for (int i = tid; i < C * D; i += kSimtThreads) {
        const int r = i / D, c = i % D;
        const float e = eG(r, c, 1.f);
        const float kv = sK[r * L::LD + c];
        if (ERASE) sX[r * L::LX + c] = sB[r] * kv * e;  // beta K~
        sKh[r * L::LD + c] = kv * eG(r, c, -1.f);
        sQ[r * L::LD + c] *= e;
      }
      __syncthreads();
    }

    // ---- 3. pair matrices over the lower triangle (decay-weighted for the gated rule)
    for (int p = tid; p < C * (C + 1) / 2; p += kSimtThreads) {
      int r = (int)((sqrtf(8.f * p + 1.f) - 1.f) * 0.5f);
      while (r * (r + 1) / 2 > p) --r;
      while ((r + 1) * (r + 2) / 2 <= p) ++r;
      const int j = p - r * (r + 1) / 2;
      float acc_a = 0.f, acc_m = 0.f;
      const float* kr = sK + r * L::LD;
      const float* kj = sK + j * L::LD;
      const float* qr = sQ + r * L::LD;
      if (LINEAR) {
        for (int c = 0; c < D; ++c) acc_m = fmaf(qr[c], kj[c], acc_m);
      } else if (factor) {
        const float* xr = sX + r * L::LX;   // beta_r K~_r
        const float* krj = sKh + j * L::LD;  // Kr_j
        for (int c = 0; c < D; ++c) {
          if (ERASE) acc_a = fmaf(xr[c], krj[c], acc_a);
          acc_m = fmaf(qr[c], krj[c], acc_m);  // qr is Q~_r here
        }
        if (ERASE) sA[r * L::LC + j] = (j < r) ? acc_a : 0.f;
      } else {
        const float* gr = sG + r * L::LD;
        const float* gj = sG + j * L::LD;
        const float* glr = sGl + r * L::LD;
        const float* glj = sGl + j * L::LD;
        for (int c = 0; c < D; ++c) {
          const float w = kj[c] * expf((gr[c] - gj[c]) + (glr[c] - glj[c]));
          acc_a = fmaf(kr[c], w, acc_a);
          acc_m = fmaf(qr[c], w, acc_m);
        }
        if (ERASE) sA[r * L::LC + j] = (j < r) ? sB[r] * acc_a : 0.f;
      }
      sM[r * L::LC + j] = acc_m;
    }
    __syncthreads();
    if (NORM) {
      // ---- 3b. denominators phi(q_r) . z_r = phi(q_r) . z_entry + sum_{j <= r} M[r][j]
      for (int r = tid; r < C; r += kSimtThreads) {
        const float* qr = sQ + r * L::LD;
        float acc0 = 0.f, acc1 = 0.f;
        for (int c = 0; c < D; c += 2) {
          acc0 = fmaf(qr[c], sZ[c], acc0);
          acc1 = fmaf(qr[c + 1], sZ[c + 1], acc1);
        }
        const float* mr = sM + r * L::LC;
        for (int j = 0; j <= r; ++j) acc0 += mr[j];
        sDen[r] = acc0 + acc1 + a.eps;
      }
      __syncthreads();
    }

    if (!LINEAR) {
      // ---- 4. gate-scaled operands and the right-hand sides of the solve (strong decay: here;
      // weak decay: K^ = Kr gamma)
      for (int c = tid; c < D; c += kSimtThreads) sGam[c] = eG(C - 1, c, 1.f);
      if (factor) __syncthreads();
      for (int i = tid; i < C * D; i += kSimtThreads) {
        const int r = i / D, c = i % D;
        if (factor) {
          sKh[r * L::LD + c] *= sGam[c];
          continue;
        }
        const float kv = sK[r * L::LD + c];
        const float e = eG(r, c, 1.f);
        if (ERASE) sX[r * L::LX + c] = sB[r] * kv * e;  // beta K~
        sKh[r * L::LD + c] =
            kv * expf((sG[(C - 1) * L::LD + c] - sG[r * L::LD + c]) +
                      (sGl[(C - 1) * L::LD + c] - sGl[r * L::LD + c]));  // K^
        sQ[r * L::LD + c] *= e;                                            // Q~
      }
      if (ERASE) {
        for (int i = tid; i < C * kDVB; i += kSimtThreads) {
          const int r = i / kDVB, c = i % kDVB;
          sX[r * L::LX + D + c] = sB[r] * sV[r * L::LV + c];  // beta V
        }
      }
      __syncthreads();
    }
    if (ERASE) {
      // ---- 5. forward substitution (I + A) X = rhs; each thread owns whole columns of X
      for (int col = tid; col < D + kDVB; col += kSimtThreads) {
        for (int r = 1; r < n; ++r) {
          float acc0 = sX[r * L::LX + col], acc1 = 0.f;
          const float* ar = sA + r * L::LC;
          int j = 0;
          for (; j + 1 < r; j += 2) {
            acc0 = fmaf(-ar[j], sX[j * L::LX + col], acc0);
            acc1 = fmaf(-ar[j + 1], sX[(j + 1) * L::LX + col], acc1);
          }
          if (j < r) acc0 = fmaf(-ar[j], sX[j * L::LX + col], acc0);
          sX[r * L::LX + col] = acc0 + acc1;
        }
      }
      __syncthreads();

      // ---- 6. U = U~ - W S
      for (int i = tid; i < C * kDVB; i += kSimtThreads) {
        const int r = i / kDVB, c = i % kDVB;
        const float* wr = sX + r * L::LX;
        float acc0 = wr[D + c], acc1 = 0.f;
        for (int m = 0; m < D; m += 2) {
          acc0 = fmaf(-wr[m], sS[m * L::LV + c], acc0);
          acc1 = fmaf(-wr[m + 1], sS[(m + 1) * L::LV + c], acc1);
        }
        sU[r * L::LV + c] = acc0 + acc1;
      }
      __syncthreads();
    }
    const float* sUse = ERASE ? sU : sV;  // the values the chunk writes

    // ---- 7. O = Q~ S + M U
    for (int i = tid; i < C * kDVB; i += kSimtThreads) {
      const int r = i / kDVB, c = i % kDVB;
      if (r >= n) continue;
      const float* qr = sQ + r * L::LD;
      float acc0 = 0.f, acc1 = 0.f;
      for (int m = 0; m < D; m += 2) {
        acc0 = fmaf(qr[m], sS[m * L::LV + c], acc0);
        acc1 = fmaf(qr[m + 1], sS[(m + 1) * L::LV + c], acc1);
      }
      const float* mr = sM + r * L::LC;
      for (int j = 0; j <= r; ++j) acc0 = fmaf(mr[j], sUse[j * L::LV + c], acc0);
      const size_t oi = ((size_t)(tc + r) * H + h) * D + vc0 + c;
      float o = acc0 + acc1;
      if (NORM) o /= sDen[r];
      if (a.og) o = gate_out(o, to_f32(static_cast<const T*>(a.og)[oi]));
      out[oi] = from_f32<T>(o);
    }
    __syncthreads();

    // ---- 8. S <- Diag(e^{G_n}) S + K^T U
    const float* kh = LINEAR ? sK : sKh;
    for (int i = tid; i < D * kDVB; i += kSimtThreads) {
      const int m = i / kDVB, c = i % kDVB;
      float acc = LINEAR ? sS[m * L::LV + c] : sGam[m] * sS[m * L::LV + c];
      for (int j = 0; j < n; ++j) acc = fmaf(kh[j * L::LD + m], sUse[j * L::LV + c], acc);
      sS[m * L::LV + c] = acc;
    }
    if (NORM) {  // z <- z + sum of the chunk's phi(k) rows (rows >= n are 0)
      for (int c = tid; c < D; c += kSimtThreads) {
        float acc = sZ[c];
        for (int j = 0; j < n; ++j) acc += sK[j * L::LD + c];
        sZ[c] = acc;
      }
    }
  }
  __syncthreads();
  if (NORM && a.z_final && vb == 0)
    for (int c = tid; c < D; c += kSimtThreads) a.z_final[((size_t)seq * H + h) * D + c] = sZ[c];
  if (a.S_final) {
    for (int i = tid; i < D * kDVB; i += kSimtThreads) {
      const int r = i / kDVB, c = i % kDVB;
      a.S_final[sidx + (size_t)r * D + vc0 + c] = sS[r * L::LV + c];
    }
  }
}

template <int D, int C, typename T, bool CHANNEL, int KIND>
cudaError_t launch_one(const gdr_shape& sh, const PrefillArgs& a, cudaStream_t s) {
  auto kern = prefill_simt_kernel<D, C, T, CHANNEL, KIND>;
  const size_t smem = SimtSmem<D, C>::bytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)sh.n_seqs * (unsigned)sh.H * (unsigned)(D / kDVB);
  kern<<<grid, kSimtThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <int D, int C, typename T>
cudaError_t launch_t(const gdr_shape& sh, const PrefillArgs& a, int kind, cudaStream_t s) {
  if (kind == kKindLinear) return launch_one<D, C, T, true, kKindLinear>(sh, a, s);
  if (kind == kKindNormLinear) return launch_one<D, C, T, true, kKindNormLinear>(sh, a, s);
  const bool ch = sh.gate == GDR_GATE_CHANNEL;
  if (kind == kKindGatedLinear)
    return ch ? launch_one<D, C, T, true, kKindGatedLinear>(sh, a, s)
              : launch_one<D, C, T, false, kKindGatedLinear>(sh, a, s);
  return ch ? launch_one<D, C, T, true, kKindDelta>(sh, a, s)
            : launch_one<D, C, T, false, kKindDelta>(sh, a, s);
}

}  // namespace

cudaError_t launch_prefill_simt(const gdr_shape& sh, const PrefillArgs& a, int kind,
                                cudaStream_t s) {
  if (sh.d_k == 128)
    return sh.dtype == GDR_BF16 ? launch_t<128, 32, __nv_bfloat16>(sh, a, kind, s)
                                : launch_t<128, 32, float>(sh, a, kind, s);
  return sh.dtype == GDR_BF16 ? launch_t<64, 64, __nv_bfloat16>(sh, a, kind, s)
                              : launch_t<64, 64, float>(sh, a, kind, s);
}

}  // namespace gdr
