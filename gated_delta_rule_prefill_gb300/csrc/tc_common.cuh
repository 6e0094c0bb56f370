// tc_common.cuh -- the pieces shared by the tensor-core prefill kernels (prefill_tc.cu: one CTA
// per sequence-head chain; prefill_cluster.cu: a chain CTA fed by helper CTAs of its cluster):
// constants, tile helpers, the triangular solve and the per-chunk stages.  The chunk algebra is
// stated in prefill_tc.cu.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "gdr_internal.cuh"
#include "umma.cuh"

namespace gdr {
namespace tc {

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

// Operand slot of one chunk as a chain CTA consumes it (bytes from the slot base; K-major tiles
// of 128 rows have 16 KB slabs).  With a zero tile Z between T' and M, [T'; Z] and [Z; M] are
// 128 x 64 K-major tiles; [-W; Q~] is one 128 x 128 tile.
constexpr uint32_t kSlotWQ = 0;       // [-W; Q~]: -W rows at +0 / +16K, Q~ rows at +8K / +24K
constexpr uint32_t kSlotKH = 32768;   // K^  [tok][ch] (MN-major A), slabs 8 KB apart
constexpr uint32_t kSlotT = 49152;    // T'  [64][64]
constexpr uint32_t kSlotZ = 57344;    // zeros [64][64]
constexpr uint32_t kSlotM = 65536;    // M   [64][64]
constexpr uint32_t kSlotGam = 73728;  // gamma [128] fp32
constexpr uint32_t kSlotPayload = 65536 + 512;  // everything but Z
constexpr uint32_t kSlotBytes = 74752;          // 1024-aligned

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
// K/16 MMA steps; called by all 32 lanes of one warp (one elected lane issues).
template <int K>
__device__ __forceinline__ void mma_run(uint32_t d, const Opnd& A, const Opnd& B, uint32_t idesc,
                                        bool acc) {
#pragma unroll
  for (int k = 0; k < K; k += 16)
    mma_bf16_elect(d, A.at(k), B.at(k), idesc, (acc || k > 0) ? 1u : 0u);
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

// ---- warp-level tf32 products for the off-diagonal blocks of the triangular inverse.
// mma.sync m16n8k8 (row.col) fragments, g = lane / 4, t = lane % 4:
//   A (16 x 8): a0 (g, t), a1 (g + 8, t), a2 (g, t + 4), a3 (g + 8, t + 4)
//   B (8 x 8):  b0 (t, g), b1 (t + 4, g)
//   C (16 x 8): c0 (g, 2t), c1 (g, 2t + 1), c2 (g + 8, 2t), c3 (g + 8, 2t + 1)
__device__ __forceinline__ uint32_t tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void mma_tf32(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// A fragment of the 16 x 8 tile at (r0, k0) of a swizzled fp32 64 x 64 matrix
__device__ __forceinline__ void frag_a(const float* m, int r0, int k0, int g, int t,
                                       uint32_t (&a)[4]) {
  a[0] = tf32(m[f32x(r0 + g, k0 + t)]);
  a[1] = tf32(m[f32x(r0 + g + 8, k0 + t)]);
  a[2] = tf32(m[f32x(r0 + g, k0 + t + 4)]);
  a[3] = tf32(m[f32x(r0 + g + 8, k0 + t + 4)]);
}
// two bf16 entries (r, c), (r, c + 1) of T' = T diag(beta) in the 64 x 64 K-major operand tile
__device__ __forceinline__ void st_tp2(unsigned char* tt, const float* beta, int r, int c,
                                       float t0, float t1) {
  *reinterpret_cast<__nv_bfloat162*>(tt + sw128_offset(r, c, 8192)) =
      __floats2bfloat162_rn(t0 * beta[c], t1 * beta[c + 1]);
}
// 32 x 32 fp32 scratch, columns XOR-swizzled by 8 * (row % 4) against bank conflicts
__device__ __forceinline__ int x32(int r, int c) { return r * 32 + (c ^ ((r & 3) << 3)); }

// Zeroes the bf16 T' tile (64 x 64, 8 KB); the solve never writes its part right of the 8 x 8
// diagonal blocks, so a CTA does this once before its first chunk.
__device__ __forceinline__ void zero_upper_tp(unsigned char* tt, int tid) {
  for (int i = tid; i < 8192 / 16; i += kThreads)
    reinterpret_cast<uint4*>(tt)[i] = make_uint4(0u, 0u, 0u, 0u);
}

// T = (I + A)^-1 for A strictly lower (64 x 64, fp32, swizzled layout above), by doubling the
// inverted block size: the eight 8 x 8 diagonal blocks by right-looking forward substitution (one
// column per thread, held in registers); then the 16, 32 and 64 levels, each
// T_ba = -T_bb (A_ba T_aa) over the pairs of diagonal blocks (a, b) of the level below (level 64:
// T_[23][01] = -T_[23][23] (A_[23][01] T_[01][01])).  The two products of each doubling step run
// on the tensor cores as warp-level tf32 MMAs with fp32 accumulation (T' is rounded to bf16
// afterwards, 4x coarser than tf32).  sX holds the intermediates (up to 32 x 32 fp32).  Every
// entry of T is also written as the bf16 operand T' = T diag(beta) into tt where it is produced.
__device__ inline void unit_lower_inverse(const float* sA, float* sT, float* sX, int tid,
                                          unsigned char* tt, const float* beta) {
  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  if (tid < 64) {
    const int b = tid >> 3, c = tid & 7, o = 8 * b;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = (i == c) ? 1.f : 0.f;
#pragma unroll
    for (int j = 0; j < 7; ++j) {
      const float xj = acc[j];
#pragma unroll
      for (int i = j + 1; i < 8; ++i) acc[i] = fmaf(-sA[f32x(o + i, o + j)], xj, acc[i]);
    }
    const float bc = beta[o + c];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      sT[f32x(o + i, o + c)] = acc[i];
      st_bf16(tt, sw128_offset(o + i, o + c, 8192), acc[i] * bc);
    }
  }
  // Nothing right of the 8 x 8 diagonal blocks is stored: the fp32 products below take those
  // zeros as constant fragments, and the bf16 tile's upper part is zeroed once per CTA
  // (zero_upper_tp), before its first chunk.
  __syncthreads();
  // ---- level 16: warp p of warps 0-3 takes the 16 x 16 block p (8-blocks a = 2p, b = 2p + 1);
  // the MMAs are 16 rows high, the 8 rows of the block padded with zeros
  if (warp < 4) {
    const int ra = 16 * warp, rb = ra + 8;
    float* sXw = sX + warp * 64;  // X = A_ba T_aa, 8 x 8 row-major
    uint32_t a[4];
    a[0] = tf32(sA[f32x(rb + g, ra + t)]);
    a[2] = tf32(sA[f32x(rb + g, ra + t + 4)]);
    a[1] = a[3] = 0u;
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    mma_tf32(c, a, tf32(sT[f32x(ra + t, ra + g)]), tf32(sT[f32x(ra + t + 4, ra + g)]));
    *reinterpret_cast<float2*>(sXw + g * 8 + 2 * t) = make_float2(c[0], c[1]);
    __syncwarp();
    a[0] = tf32(sT[f32x(rb + g, rb + t)]);
    a[2] = tf32(sT[f32x(rb + g, rb + t + 4)]);
    float y[4] = {0.f, 0.f, 0.f, 0.f};
    mma_tf32(y, a, tf32(sXw[t * 8 + g]), tf32(sXw[(t + 4) * 8 + g]));
    *reinterpret_cast<float2*>(sT + f32x(rb + g, ra + 2 * t)) = make_float2(-y[0], -y[1]);
    st_tp2(tt, beta, rb + g, ra + 2 * t, -y[0], -y[1]);
  }
  __syncthreads();
  // ---- level 32: warp (p, j) of warps 0-3 computes the 8 columns 8j.. of pair p's blocks
  if (warp < 4) {
    const int p = warp >> 1, j = warp & 1;
    const int ra = 32 * p, rb = ra + 16;
    float* sXp = sX + p * 512;  // X_p as 16 x 32 rows of the x32 layout (columns 0-15 used)
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      if (ks < j) continue;  // T_aa rows above the column tile are zero
      uint32_t a[4];
      frag_a(sA, rb, ra + 8 * ks, g, t, a);
      mma_tf32(c, a, tf32(sT[f32x(ra + 8 * ks + t, ra + 8 * j + g)]),
               tf32(sT[f32x(ra + 8 * ks + t + 4, ra + 8 * j + g)]));
    }
    *reinterpret_cast<float2*>(sXp + x32(g, 8 * j + 2 * t)) = make_float2(c[0], c[1]);
    *reinterpret_cast<float2*>(sXp + x32(g + 8, 8 * j + 2 * t)) = make_float2(c[2], c[3]);
    __syncwarp();
    asm volatile("bar.sync 1, 128;" ::: "memory");  // warps 0-3 only
    float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      uint32_t a[4];
      frag_a(sT, rb, rb + 8 * ks, g, t, a);
      if (ks == 1) a[0] = a[2] = 0u;  // T_bb's upper-right 8 x 8 block is zero
      mma_tf32(y, a, tf32(sXp[x32(8 * ks + t, 8 * j + g)]),
               tf32(sXp[x32(8 * ks + t + 4, 8 * j + g)]));
    }
    *reinterpret_cast<float2*>(sT + f32x(rb + g, ra + 8 * j + 2 * t)) = make_float2(-y[0], -y[1]);
    *reinterpret_cast<float2*>(sT + f32x(rb + g + 8, ra + 8 * j + 2 * t)) =
        make_float2(-y[2], -y[3]);
    st_tp2(tt, beta, rb + g, ra + 8 * j + 2 * t, -y[0], -y[1]);
    st_tp2(tt, beta, rb + g + 8, ra + 8 * j + 2 * t, -y[2], -y[3]);
  }
  __syncthreads();
  // ---- level 64: warp (mi, ni) computes the 16 x 8 tile (rows 16 mi.., columns 8 ni..)
  {
    const int mi = warp >> 2, ni = warp & 3;
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      if (ks < ni) continue;  // rows of T_[01][01] above the column tile are zero
      uint32_t a[4];
      frag_a(sA, 32 + 16 * mi, 8 * ks, g, t, a);
      mma_tf32(c, a, tf32(sT[f32x(8 * ks + t, 8 * ni + g)]),
               tf32(sT[f32x(8 * ks + t + 4, 8 * ni + g)]));
    }
    *reinterpret_cast<float2*>(sX + x32(16 * mi + g, 8 * ni + 2 * t)) = make_float2(c[0], c[1]);
    *reinterpret_cast<float2*>(sX + x32(16 * mi + g + 8, 8 * ni + 2 * t)) = make_float2(c[2], c[3]);
    __syncthreads();
    float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      if (ks > 2 * mi + 1) continue;  // T_[23][23] is zero right of the row tile's diagonal
      uint32_t a[4];
      frag_a(sT, 32 + 16 * mi, 32 + 8 * ks, g, t, a);
      if (ks == 2 * mi + 1) a[0] = a[2] = 0u;  // upper-right 8 x 8 of the diagonal 16 x 16 block
      mma_tf32(y, a, tf32(sX[x32(8 * ks + t, 8 * ni + g)]),
               tf32(sX[x32(8 * ks + t + 4, 8 * ni + g)]));
    }
    *reinterpret_cast<float2*>(sT + f32x(32 + 16 * mi + g, 8 * ni + 2 * t)) =
        make_float2(-y[0], -y[1]);
    *reinterpret_cast<float2*>(sT + f32x(32 + 16 * mi + g + 8, 8 * ni + 2 * t)) =
        make_float2(-y[2], -y[3]);
    st_tp2(tt, beta, 32 + 16 * mi + g, 8 * ni + 2 * t, -y[0], -y[1]);
    st_tp2(tt, beta, 32 + 16 * mi + g + 8, 8 * ni + 2 * t, -y[2], -y[3]);
    __syncthreads();
  }
}

// The output gate for bf16 outputs: o * sigmoid(g) with sigmoid(g) = (1 + tanh(g / 2)) / 2 on
// the hardware tanh approximation (absolute error ~2^-11, below bf16's 2^-8 relative rounding),
// without the IEEE division of gate_out.
__device__ __forceinline__ float gate_out_bf16(float o, float g) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * g));
  return o * fmaf(0.5f, t, 0.5f);
}

// The output gate on two bf16 outputs in packed bf16 arithmetic: o * (1/2 + tanh(g/2) / 2) with
// the hardware tanh approximation on both halves at once.  The bf16 sigmoid carries a relative
// error of ~2^-9, the size of the output's own bf16 rounding.
__device__ __forceinline__ __nv_bfloat162 gate2_bf16(__nv_bfloat162 o, __nv_bfloat162 g) {
  const __nv_bfloat162 half = __float2bfloat162_rn(0.5f);
  const __nv_bfloat162 hg = __hmul2(g, half);
  uint32_t t;
  asm("tanh.approx.bf16x2 %0, %1;" : "=r"(t) : "r"(*reinterpret_cast<const uint32_t*>(&hg)));
  const __nv_bfloat162 sg = __hfma2(*reinterpret_cast<const __nv_bfloat162*>(&t), half, half);
  return __hmul2(o, sg);
}

// The output gate on 8 consecutive outputs: v[i] <- v[i] * sigmoid(g[i]) (g: 16-byte aligned bf16).
__device__ __forceinline__ void gate8(float* v, const __nv_bfloat16* g) {
  const uint4 u = *reinterpret_cast<const uint4*>(g);
  const __nv_bfloat162* hg = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(hg[i]);
    v[2 * i] = gate_out_bf16(v[2 * i], f.x);
    v[2 * i + 1] = gate_out_bf16(v[2 * i + 1], f.y);
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
  CUtensorMap k_sw, q_sw;  // k, q in 64-channel SW128 boxes (linear attention)
  CUtensorMap og;          // output gate g, 128-channel boxes (prefetched into L2)
};


// Per-CTA context of the stage functions.
struct TcCtx {
  unsigned char* sm;   // 1024-aligned dynamic shared memory
  uint32_t sb;         // its shared-window address
  uint32_t tm;         // TMEM base
  uint32_t lane_base;  // this warp's TMEM lane quarter
  int tid, warp, lane, lrow, wh, m64row;
  bool m64ok;
  uint64_t* bar_mma;
  uint32_t ph_mma;
  // If set, the stages also write the chunk's hand-over operands (Q~, K^, gamma, M, T', -W) into
  // this operand slot image in global memory, and skip the shared-memory copies only a chain
  // CTA would read (K^, M, W).
  unsigned char* gslot;
  bool prologue;  // the staged q, k, alpha are raw projections (the layer prologue runs first)
};

__device__ __forceinline__ TcCtx make_ctx(unsigned char* sm, uint32_t tm, uint64_t* bar_mma) {
  TcCtx x;
  x.sm = sm;
  x.sb = smem_u32(sm);
  x.tm = tm;
  x.tid = threadIdx.x;
  x.warp = x.tid >> 5;
  x.lane = x.tid & 31;
  x.lrow = x.tid & 127;
  x.wh = x.warp >> 2;
  x.lane_base = (uint32_t)((x.warp & 3) * 32) << 16;
  x.m64row = 16 * (x.warp & 3) + (x.lane & 15);
  x.m64ok = x.lane < 16;
  x.bar_mma = bar_mma;
  x.ph_mma = 0;
  x.gslot = nullptr;
  x.prologue = false;
  return x;
}

// Waits on an mbarrier phase; every thread sees the same verdict (false: it gave up).
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t& ph) {
  const bool ok = mbar_wait(bar, ph, kWaitNs);
  ph ^= 1u;
  __syncwarp();  // lanes leave the polling loop at different times; reconverge before the barrier
  const bool all_ok = !__syncthreads_or(!ok);
  fence_after_sync();
  return all_ok;
}

// 8 fp32 values -> one 16-byte chunk of bf16 (row-major tiles)
__device__ __forceinline__ void st_bf16x8(__nv_bfloat16* p, const float* x) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = u;
}

// The layer prologue's maps on the tensor-core paths.  sigmoid(x) = 1 / (1 + 2^(-x log2 e)) on
// the hardware ex2 and rcp approximations (flush-to-zero forms; the exponent capped at 80 so the
// divisor stays finite): relative error a few fp32 ulps, the precision the decay products need.
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_ftz(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sigmoid_ftz(float x) {
  return rcp_ftz(1.f + ex2_ftz(fminf(-x, 80.f) * 1.44269504f));
}
// silu of two bf16 values: silu(x) = x sigmoid(x) = h + h tanh(h) with h = x / 2, tanh on the
// packed-half unit (one instruction for both; error ~2^-11 of h, below the bf16 rounding of the
// normalised result).  |h| beyond the half range becomes +-inf, where tanh = +-1 gives the exact
// limits silu = x and 0.
__device__ __forceinline__ float2 silu2(__nv_bfloat162 v) {
  const float2 f = __bfloat1622float2(v);
  const float hx = 0.5f * f.x, hy = 0.5f * f.y;
  const __half2 hh = __floats2half2_rn(hx, hy);
  uint32_t t;
  asm("tanh.approx.f16x2 %0, %1;" : "=r"(t) : "r"(*reinterpret_cast<const uint32_t*>(&hh)));
  const float2 tf = __half22float2(*reinterpret_cast<const __half2*>(&t));
  return make_float2(fmaf(hx, tf.x, hx), fmaf(hy, tf.y, hy));
}

// ---- Stage 0: the layer prologue on the staged tiles, in place (heqinghuang "gpt2-to-kimi"
// §09: unit-length silu queries and keys; engineermaxxing "From GPT-2 to Kimi K3" §05c/§06b:
// the decay is a sigmoid of its projection).  q, k <- normalize(silu(.)) over the 128 channels
// of each token row, rounded to bf16 (the operand type of the tensor-core products); per-channel
// alpha <- sigmoid(alpha).  Rows >= n are left alone.  The thread map is gate_stage's (8 channels
// x 4 rows, a row's 16 threads one half-warp): each thread rewrites what it reads back itself
// before the gate stage's first barrier, and the norms are half-warp shuffles.  The eight rows
// of a thread (4 of q, 4 of k) go through each step together, so their latencies overlap.
template <class L, bool CHANNEL>
__device__ void prologue_stage(const TcCtx& x, int n) {
  const int g8 = x.tid & 15, rb = x.tid >> 4;
  __nv_bfloat16* sQin = reinterpret_cast<__nv_bfloat16*>(x.sm + L::QIN);
  __nv_bfloat16* sKin = reinterpret_cast<__nv_bfloat16*>(x.sm + L::KIN);
  float* sAin = reinterpret_cast<float*>(x.sm + L::AIN);
  float v[8][8], ss[8];  // row j = 2 rr + (0: q, 1: k)
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = 4 * rb + (j >> 1);
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (r < n) u = *reinterpret_cast<const uint4*>(((j & 1) ? sKin : sQin) + r * kD + 8 * g8);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
    ss[j] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 sl = silu2(h[i]);
      v[j][2 * i] = sl.x;
      v[j][2 * i + 1] = sl.y;
      ss[j] = fmaf(sl.x, sl.x, fmaf(sl.y, sl.y, ss[j]));
    }
  }
  if (CHANNEL) {
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = 4 * rb + rr;
      if (r < n) {
        float4* pa = reinterpret_cast<float4*>(sAin + r * kD + 8 * g8);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          float4 u = pa[i];
          u.x = sigmoid_ftz(u.x), u.y = sigmoid_ftz(u.y);
          u.z = sigmoid_ftz(u.z), u.w = sigmoid_ftz(u.w);
          pa[i] = u;
        }
      }
    }
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1)
#pragma unroll
    for (int j = 0; j < 8; ++j) ss[j] += __shfl_xor_sync(0xffffffffu, ss[j], off);
  // Rows whose silu norm is below 2 (squared 4), e.g. rows of only strongly negative values, take
  // silu again in fp32 (ex2 and rcp): there the packed-half tanh's absolute error (~2e-3 per
  // value at most) is no longer small against the norm that the row is divided by.  The test is
  // per row (half-warp uniform); the redo runs on the whole warp when either half needs it.
  unsigned redo = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) redo |= (ss[j] < 4.f ? 1u : 0u) << j;
  redo = __reduce_or_sync(0xffffffffu, redo);
  if (redo) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (!((redo >> j) & 1u)) continue;
      const int r = 4 * rb + (j >> 1);
      float e8[8];
      if (r < n) {
        ld_bf16x8(((j & 1) ? sKin : sQin) + r * kD + 8 * g8, e8);
      } else {
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) e8[cc] = 0.f;
      }
      float s2 = 0.f;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        e8[cc] *= sigmoid_ftz(e8[cc]);
        s2 = fmaf(e8[cc], e8[cc], s2);
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, off);
      if (ss[j] < 4.f) {
        ss[j] = s2;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) v[j][cc] = e8[cc];
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = 4 * rb + (j >> 1);
    if (r < n) {
      const float inv = inv_norm(ss[j]);
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) v[j][cc] *= inv;
      st_bf16x8(((j & 1) ? sKin : sQin) + r * kD + 8 * g8, v[j]);
    }
  }
}

// ---- Stage 1: gate prologue.  Reads the staged q, k (row-major bf16) and alpha (row-major
// fp32) tiles and the chunk's beta / scalar gates; writes the bf16 operand tiles KQ ([K~; Q~],
// or raw K and Q for scalar gates), KR (Kr) and KH (K^), gamma, the exact diagonal q_r . k_r and,
// for scalar gates, the per-token log prefix sums.  Returns whether the chunk's decay allows the
// factorised Gram products (otherwise the log prefix sums are left in the alpha tile).
// `before_writes` runs on every thread just before the stage's first CTA barrier, after which the
// stage writes the operand tiles and gamma (until then it writes only its own scratch); a caller
// that still reads those tiles asynchronously waits for the reads there.
struct NoHook {
  __device__ void operator()() const {}
};
template <class L, bool CHANNEL, class Hook = NoHook>
__device__ bool gate_stage(const TcCtx& x, int n, Hook before_writes = Hook()) {
  constexpr bool kScalar = !CHANNEL;
  unsigned char* sm = x.sm;
  const int tid = x.tid, warp = x.warp, lane = x.lane;
  const __nv_bfloat16* sQin = reinterpret_cast<const __nv_bfloat16*>(sm + L::QIN);
  const __nv_bfloat16* sKin = reinterpret_cast<const __nv_bfloat16*>(sm + L::KIN);
  float* sAin = reinterpret_cast<float*>(sm + L::AIN);
  float* sAlpha = reinterpret_cast<float*>(sm + L::ALPHA);
  float* sGam = reinterpret_cast<float*>(sm + L::GAM);
  float* sRed = reinterpret_cast<float*>(sm + L::RED);
  float* sDiagP = reinterpret_cast<float*>(sm + L::DIAGP);  // [64 rows][16] partial q_r . k_r
  float* sGs = reinterpret_cast<float*>(sm + L::GS);
  if (x.prologue) prologue_stage<L, CHANNEL>(x, n);
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
      before_writes();
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
        sDiagP[r * 16 + g8] = dq;
        st_chunk8(sm + L::KQ, 16384, r, 8 * g8, k8);       // K (scaled to K~ after the Gram MMA)
        st_chunk8(sm + L::KQ, 16384, 64 + r, 8 * g8, q8);  // Q (scaled to Q~ likewise)
        st_chunk8(sm + L::KR, 8192, r, 8 * g8, k8);        // K
        if (x.gslot) {
          st_chunk8(x.gslot + kSlotKH, 8192, r, 8 * g8, kh);  // K^ (hand-over only)
        } else {
          st_chunk8(sm + L::KH, 8192, r, 8 * g8, kh);        // K^
        }
      }
      if (rb == 0) {
        const float gm = __expf(Gn);
        *reinterpret_cast<float4*>(sGam + 8 * g8) = make_float4(gm, gm, gm, gm);
        *reinterpret_cast<float4*>(sGam + 8 * g8 + 4) = make_float4(gm, gm, gm, gm);
        if (x.gslot) {
          float* gg = reinterpret_cast<float*>(x.gslot + kSlotGam);
          *reinterpret_cast<float4*>(gg + 8 * g8) = make_float4(gm, gm, gm, gm);
          *reinterpret_cast<float4*>(gg + 8 * g8 + 4) = make_float4(gm, gm, gm, gm);
        }
      }
    } else {
      // Per-channel gates: running products of the gates down the
      // thread's rows, then the carry of the earlier row blocks through shared memory.
      float p[4][8];  // prefix products Gam[4 rb + rr][8 g8 + cc]
      float gn[8];    // Gam_n (= gamma) of the 8 channels
      float sufc[8];  // product of the gates of the later row blocks, per channel
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
          if (r < n) {
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
        {
          // row-block totals -> exclusive prefix and suffix products over the 16 row blocks
          // (one thread per channel) -> each thread's carries; gamma = the full product
          float* sTot = reinterpret_cast<float*>(sm + L::TOT);  // [32][128 channels]
          *reinterpret_cast<float4*>(sTot + rb * kD + 8 * g8) = make_float4(run[0], run[1], run[2], run[3]);
          *reinterpret_cast<float4*>(sTot + rb * kD + 8 * g8 + 4) = make_float4(run[4], run[5], run[6], run[7]);
          before_writes();
          __syncthreads();
          if (tid < kD) {
            float t16[16];
#pragma unroll
            for (int b2 = 0; b2 < 16; ++b2) t16[b2] = sTot[b2 * kD + tid];
            float acc = 1.f;
#pragma unroll
            for (int b2 = 0; b2 < 16; ++b2) {
              sTot[b2 * kD + tid] = acc;
              acc *= t16[b2];
            }
            float suf = 1.f;
#pragma unroll
            for (int b2 = 15; b2 >= 0; --b2) {
              sTot[(16 + b2) * kD + tid] = suf;
              suf *= t16[b2];
            }
            sGam[tid] = acc;
            if (x.gslot) reinterpret_cast<float*>(x.gslot + kSlotGam)[tid] = acc;
            float mn = acc;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
            if (lane == 0) sRed[warp] = mn;
          }
          __syncthreads();
          const float4 c0 = *reinterpret_cast<const float4*>(sTot + rb * kD + 8 * g8);
          const float4 c1 = *reinterpret_cast<const float4*>(sTot + rb * kD + 8 * g8 + 4);
          const float4 s0 = *reinterpret_cast<const float4*>(sTot + (16 + rb) * kD + 8 * g8);
          const float4 s1 = *reinterpret_cast<const float4*>(sTot + (16 + rb) * kD + 8 * g8 + 4);
          const float4 n0 = *reinterpret_cast<const float4*>(sGam + 8 * g8);
          const float4 n1 = *reinterpret_cast<const float4*>(sGam + 8 * g8 + 4);
          const float carry[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          sufc[0] = s0.x, sufc[1] = s0.y, sufc[2] = s0.z, sufc[3] = s0.w;
          sufc[4] = s1.x, sufc[5] = s1.y, sufc[6] = s1.z, sufc[7] = s1.w;
          gn[0] = n0.x, gn[1] = n0.y, gn[2] = n0.z, gn[3] = n0.w;
          gn[4] = n1.x, gn[5] = n1.y, gn[6] = n1.z, gn[7] = n1.w;
#pragma unroll
          for (int rr = 0; rr < 4; ++rr)
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) p[rr][cc] *= carry[cc];
          safe = fminf(fminf(sRed[0], sRed[1]), fminf(sRed[2], sRed[3])) > kSafeGamma;
        }
      }

      if (safe) {
        // K^ = K * Gam_n / Gam = K * (product of the later gates): a suffix product, no division;
        // Kr = K / Gam = K^ / Gam_n with one reciprocal per channel.  Rows go last to first so
        // the within-block suffix grows by one gate per row.
        float rgn[8], suf[8];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          rgn[cc] = __fdividef(1.f, gn[cc]);
          suf[cc] = sufc[cc];
        }
#pragma unroll
        for (int rr = 3; rr >= 0; --rr) {
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
            ke[cc] = k8[cc] * G;
            qe[cc] = q8[cc] * G;
            kh[cc] = k8[cc] * suf[cc];
            ki[cc] = kh[cc] * rgn[cc];
            dq = fmaf(q8[cc], k8[cc], dq);
          }
          if (rr > 0 && r < n) {  // the suffix of row r - 1 gains this row's gates
            const float4 u0 = *reinterpret_cast<const float4*>(sAin + r * kD + 8 * g8);
            const float4 u1 = *reinterpret_cast<const float4*>(sAin + r * kD + 8 * g8 + 4);
            suf[0] *= u0.x, suf[1] *= u0.y, suf[2] *= u0.z, suf[3] *= u0.w;
            suf[4] *= u1.x, suf[5] *= u1.y, suf[6] *= u1.z, suf[7] *= u1.w;
          }
          sDiagP[r * 16 + g8] = dq;  // M's diagonal carries no decay: q_r . k_r
          st_chunk8(sm + L::KQ, 16384, r, 8 * g8, ke);       // K~
          st_chunk8(sm + L::KQ, 16384, 64 + r, 8 * g8, qe);  // Q~
          st_chunk8(sm + L::KR, 8192, r, 8 * g8, ki);        // Kr
          if (x.gslot) {  // Q~ and K^ of the hand-over (K^ only there)
            st_chunk8(x.gslot + kSlotWQ, 16384, 64 + r, 8 * g8, qe);
            st_chunk8(x.gslot + kSlotKH, 8192, r, 8 * g8, kh);
          } else {
            st_chunk8(sm + L::KH, 8192, r, 8 * g8, kh);      // K^
          }
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
          if (x.gslot) {
            st_bf16(x.gslot + kSlotWQ, sw128_offset(64 + r, c, 16384), qv * e);
            st_bf16(x.gslot + kSlotKH, sw128_offset(r, c, 8192), kv * __expf(Gn - G));
          } else {
            st_bf16(sm + L::KH, sw128_offset(r, c, 8192), kv * __expf(Gn - G));
          }
        }
      }
    }
  return safe;
}

// ---- Stage 2: the decay-weighted Gram matrices.  One M = 128 tcgen05 MMA [K~; Q~] Kr^T into
// TMEM, then the epilogue: A = diag(beta) strict_lower(A') as fp32 (swizzled) and M as the bf16
// operand MM; strong-decay chunks form both from direct pairwise exponentials instead.
// Returns false if the MMA wait gave up.
template <class L, bool CHANNEL>
__device__ bool gram_stage(TcCtx& x, int n, bool safe) {
  constexpr bool kScalar = !CHANNEL;
  unsigned char* sm = x.sm;
  const int tid = x.tid, lrow = x.lrow, wh = x.wh;
  const uint32_t tm = x.tm, lane_base = x.lane_base;
  const __nv_bfloat16* sQin = reinterpret_cast<const __nv_bfloat16*>(sm + L::QIN);
  const __nv_bfloat16* sKin = reinterpret_cast<const __nv_bfloat16*>(sm + L::KIN);
  float* sAin = reinterpret_cast<float*>(sm + L::AIN);
  float* sA = reinterpret_cast<float*>(sm + L::SA);
  float* sBeta = reinterpret_cast<float*>(sm + L::BETA);
  const float* sDiagP = reinterpret_cast<const float*>(sm + L::DIAGP);
  float* sGs = reinterpret_cast<float*>(sm + L::GS);
  const Opnd opKQ{x.sb + L::KQ, 16384, false};  // [K~;Q~] as K-major A (M = 128)
  const Opnd opKR{x.sb + L::KR, 8192, false};   // Kr as K-major B (N = 64 tokens)
  const uint32_t id_am = idesc_bf16(128, kC);
    // ================= 2. decay-weighted Gram matrices [A'; M]
    if (safe) {
      if (x.warp == 0) {
        mma_run<kD>(tm + kColAM, opKQ, opKR, id_am, false);
        mma_commit_elect(x.bar_mma);
      }
      if (!wait_bar(x.bar_mma, x.ph_mma)) return false;
      const int r = lrow & 63;
      const int c0 = 32 * wh;
      float xv[32];
      tmem_ld32(tm + lane_base + kColAM + c0, xv);
      if constexpr (kScalar) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          xv[j] = (c0 + j <= r) ? xv[j] * __expf(sGs[r] - sGs[c0 + j]) : 0.f;
      }
      if (lrow < 64) {
        {
          const float b = sBeta[r];
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            st4x(sA, r, (c0 + j) >> 2,
                 make_float4((c0 + j < r) ? b * xv[j] : 0.f, (c0 + j + 1 < r) ? b * xv[j + 1] : 0.f,
                             (c0 + j + 2 < r) ? b * xv[j + 2] : 0.f,
                             (c0 + j + 3 < r) ? b * xv[j + 3] : 0.f));
        }
      } else {
        float dg = 0.f;  // q_r . k_r, summed from the gate stage's 16 partials
        if (r >= c0 && r < c0 + 32) {
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            const float4 p4 = *reinterpret_cast<const float4*>(sDiagP + r * 16 + i);
            dg += (p4.x + p4.y) + (p4.z + p4.w);
          }
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          xv[j] = (c0 + j <= r) ? xv[j] : 0.f;
          if (c0 + j == r) xv[j] = dg;
        }
        unsigned char* mm = x.gslot ? x.gslot + kSlotM : sm + L::MM;  // M: hand-over only
#pragma unroll
        for (int j = 0; j < 32; j += 8) st_chunk8(mm, 8192, r, c0 + j, xv + j);
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
          if (x.gslot && row >= 64)  // Q~ rows of the hand-over
            *reinterpret_cast<uint4*>(x.gslot + kSlotWQ + slab * 16384 + row * 128 + ch * 16) = u;
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
        st_bf16(x.gslot ? x.gslot + kSlotM : sm + L::MM, sw128_offset(r, j, 8192), acc_m);
      }
      for (int p2 = tid; p2 < kC * kC; p2 += kThreads) {
        const int r = p2 / kC, j = p2 % kC;
        if (j > r) {
          sA[f32x(r, j)] = 0.f;
          st_bf16(x.gslot ? x.gslot + kSlotM : sm + L::MM, sw128_offset(r, j, 8192), 0.f);
        }
      }
    }
    __syncthreads();

  return true;
}

// ---- Stage 3: T' = (I + A)^-1 diag(beta) as the bf16 A operand TT.
template <class L>
__device__ void solve_stage(const TcCtx& x) {
  unsigned char* sm = x.sm;
  const float* sA = reinterpret_cast<const float*>(sm + L::SA);
  float* sT32 = reinterpret_cast<float*>(sm + L::ST32);
  float* sX = reinterpret_cast<float*>(sm + L::SX);
  const float* sBeta = reinterpret_cast<const float*>(sm + L::BETA);
  unit_lower_inverse(sA, sT32, sX, x.tid, sm + L::TT, sBeta);
  if (x.gslot) {  // T' of the hand-over (the tile image, 16 bytes at a time)
    for (int e = x.tid; e < 8192 / 16; e += kThreads)
      reinterpret_cast<uint4*>(x.gslot + kSlotT)[e] = reinterpret_cast<const uint4*>(sm + L::TT)[e];
  }
  fence_async_smem();
  cta_sync_tc();
}

// ---- Stage 4: W = T' K~ (and, with a V operand, U~ = T' V into the U accumulator), then W (or
// -W) as the bf16 K-major A operand WW.  Returns false if the MMA wait gave up.
template <class L>
__device__ void w_issue(TcCtx& x, bool with_v, Opnd opV, uint32_t id_v) {
  const Opnd opT{x.sb + L::TT, 8192, false};
  const Opnd opKt{x.sb + L::KQ, 16384, true};  // K~ rows as MN-major B (K = tokens)
  if (x.warp == 0) {
    mma_run<kC>(x.tm + kColWO, opT, opKt, idesc_bf16(64, kD, false, false, true), false);
    if (with_v) mma_run<kC>(x.tm + kColU, opT, opV, id_v, false);
    mma_commit_elect(x.bar_mma);
  }
}
template <class L>
__device__ bool w_stage(TcCtx& x, bool with_v, Opnd opV, uint32_t id_v) {
  w_issue<L>(x, with_v, opV, id_v);
  return wait_bar(x.bar_mma, x.ph_mma);
}
template <class L, bool NEG = false>
__device__ void w_epilogue(const TcCtx& x) {
  float v[64];
  tmem_ld64(x.tm + x.lane_base + kColWO + x.wh * 64, v);
  if constexpr (NEG) {
#pragma unroll
    for (int j = 0; j < 64; ++j) v[j] = -v[j];
  }
  if (x.m64ok) {
#pragma unroll
    for (int j = 0; j < 64; j += 8) {
      if (x.gslot) {  // -W rows 0-63 of the hand-over's [-W; Q~] tile
        st_chunk8(x.gslot + kSlotWQ, 16384, x.m64row, x.wh * 64 + j, v + j);
      } else {
        st_chunk8(x.sm + L::WW, 8192, x.m64row, x.wh * 64 + j, v + j);
      }
    }
  }
  fence_async_smem();
}

// ---- chain pieces (value-column width DV; DH = DV / 2 columns per warp half)
// this warp half's DH columns of a TMEM region, one wait
template <int DH>
__device__ __forceinline__ void tmem_ld_half(uint32_t taddr, float (&v)[DH]) {
  static_assert(DH == 32 || DH == 64, "warp-half width");
  if constexpr (DH == 64) {
    tmem_ld64(taddr, v);
  } else {
    tmem_ld32(taddr, v);
  }
}
template <int DH>
__device__ __forceinline__ void tmem_st_half(uint32_t taddr, const float (&v)[DH]) {
#pragma unroll
  for (int c = 0; c < DH; c += 32) tmem_st32(taddr + c, *reinterpret_cast<const float(*)[32]>(v + c));
}
// fade the fp32 state master: S <- Diag(gamma) S (lane = key channel)
template <int DH>
__device__ void gamma_fade(const TcCtx& x, const float* gam) {
  const float gm = gam[x.lrow];
  const uint32_t t = x.tm + x.lane_base + kColS + x.wh * DH;
  float v[DH];
  tmem_ld_half<DH>(t, v);
#pragma unroll
  for (int j = 0; j < DH; ++j) v[j] *= gm;
  tmem_st_half<DH>(t, v);
  tmem_wait_st();
}
// U (M = 64 layout) -> bf16 [tok][DV] tile (MN-major B operand)
template <int DH>
__device__ void u_epilogue(const TcCtx& x, unsigned char* uu) {
  float v[DH];
  tmem_ld_half<DH>(x.tm + x.lane_base + kColU + x.wh * DH, v);
  if (x.m64ok) {
#pragma unroll
    for (int j = 0; j < DH; j += 8) st_chunk8(uu, 8192, x.m64row, x.wh * DH + j, v + j);
  }
  fence_async_smem();
}
// O (M = 64 layout, accumulator columns from `col`) -> out rows [tc, tc + n) of head h, value
// columns [vc0, vc0 + DV)
template <int DH>
__device__ void o_epilogue(const TcCtx& x, __nv_bfloat16* out, int64_t tc, int n, int H, int h,
                           int vc0, uint32_t col = kColWO, const __nv_bfloat16* og = nullptr) {
  float v[DH];
  tmem_ld_half<DH>(x.tm + x.lane_base + col + x.wh * DH, v);
  if (x.m64ok && x.m64row < n) {
    const size_t o0 = ((size_t)(tc + x.m64row) * H + h) * kD + vc0 + x.wh * DH;
    __nv_bfloat16* dst = out + o0;
#pragma unroll
    for (int j = 0; j < DH; j += 8) {
      if (og) gate8(v + j, og + o0 + j);
      __align__(16) __nv_bfloat162 hv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) hv[i] = __floats2bfloat162_rn(v[j + 2 * i], v[j + 2 * i + 1]);
      *reinterpret_cast<uint4*>(dst + j) = *reinterpret_cast<const uint4*>(hv);
    }
  }
}
// state master -> bf16 [d_k][DV] tile (MN-major B operand of the next chunk)
template <int DH>
__device__ void s_epilogue(const TcCtx& x, unsigned char* ss) {
  float v[DH];
  tmem_ld_half<DH>(x.tm + x.lane_base + kColS + x.wh * DH, v);
#pragma unroll
  for (int j = 0; j < DH; j += 8) st_chunk8(ss, 16384, x.lrow, x.wh * DH + j, v + j);
  fence_async_smem();
}
// entering state S0 (or zeros) -> fp32 master in TMEM and the bf16 operand tile
template <int DH>
__device__ void s_init(const TcCtx& x, const float* s0_row, unsigned char* ss) {
  float v[DH];
#pragma unroll
  for (int j = 0; j < DH; ++j) v[j] = s0_row ? s0_row[x.wh * DH + j] : 0.f;
  tmem_st_half<DH>(x.tm + x.lane_base + kColS + x.wh * DH, v);
#pragma unroll
  for (int j = 0; j < DH; j += 8) st_chunk8(ss, 16384, x.lrow, x.wh * DH + j, v + j);
  tmem_wait_st();
  fence_async_smem();  // the caller's next CTA barrier then orders the tile before any MMA
}
// state master -> S_final row (fp32)
template <int DH>
__device__ void s_final(const TcCtx& x, float* sf_row) {
  float v[DH];
  tmem_ld_half<DH>(x.tm + x.lane_base + kColS + x.wh * DH, v);
#pragma unroll
  for (int j = 0; j < DH; j += 4)
    *reinterpret_cast<float4*>(sf_row + x.wh * DH + j) =
        make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
}
// zero the V tile rows [n, 64) (SW128 [tok][DV] layout; a whole 128-byte row per slab)
template <int DV>
__device__ void zero_v_tail(const TcCtx& x, unsigned char* vin, int n) {
  if (n >= kC) return;
  for (int i = x.tid; i < (kC - n) * (DV / 8); i += kThreads) {
    const int r = n + i / (DV / 8), ch = i % (DV / 8);
    *reinterpret_cast<uint4*>(vin + (ch >> 3) * 8192 + r * 128 + (ch & 7) * 16) =
        make_uint4(0, 0, 0, 0);
  }
  fence_async_smem();
}

// host side: tensor maps of q, k, v and (per-channel gates) alpha; false if encoding failed
bool make_tc_maps(const gdr_shape& sh, const PrefillArgs& a, bool linear, TcMaps* maps);
// host side: the linear-attention kernel (bf16, d = 128)
cudaError_t launch_linear_tc(const gdr_shape& sh, const PrefillArgs& a, const TcMaps& maps,
                             bool norm, cudaStream_t s);
// host side: CTAs of the work-queue prefill for this shape and workspace (0: use another kernel)
int queue_grid_for(const gdr_shape& sh, const PrefillArgs& a);
cudaError_t launch_prefill_queue(const gdr_shape& sh, const PrefillArgs& a, const TcMaps& maps,
                                 int G, cudaStream_t s);
// host side: CTAs per cluster of the clustered prefill for this shape (1: use the one-CTA kernel)
int cluster_size_for(const gdr_shape& sh);
cudaError_t launch_prefill_cluster(const gdr_shape& sh, const PrefillArgs& a, const TcMaps& maps,
                                   int ncl, bool erase, cudaStream_t s);

}  // namespace tc
}  // namespace gdr
