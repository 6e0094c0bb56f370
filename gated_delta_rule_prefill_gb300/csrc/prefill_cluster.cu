// prefill_cluster.cu -- the tensor-core prefill for workloads with few (sequence, head) chains,
// as thread-block clusters of 1 + NH CTAs per chain.
//
// The chunk recurrence of a chain is sequential, but most of a chunk's work does not depend on
// the state: the gate prologue, the decay-weighted Gram matrices, the triangular solve and
// W = T' K~ (stages 1-4 of prefill_tc.cu).  In a cluster, CTA 0 (the chain CTA) runs only the
// state pass of every chunk (U = T' V - W S, O = Q~ S + M U, S <- gamma S + K^^T U), while the NH
// helper CTAs prepare the chunks round-robin (helper h takes chunks c with c mod NH = h) and copy
// the operands the state pass needs -- Q~, K^, -W, M, T' (bf16) and gamma -- into one of two slots
// in the chain CTA's shared memory with bulk copies over distributed shared memory.  The copies
// complete on the slot's mbarrier in the chain CTA; after consuming a slot the chain CTA re-arms
// it and publishes its count of consumed chunks into every helper's shared memory, which a
// helper waits on before it overwrites a slot.  Every wait is bounded; a timeout records
// GDR_DEVCHECK_TIMEOUT and the CTA unwinds to the closing cluster barrier.
//
// The slot stacks the operands so that the chain's products are M = 128 MMAs (an M = 64 MMA takes
// as long as an M = 128 one): with a zero tile Z between T' and M,
//   D = [T'; Z] V + [-W; Q~] S   gives U in rows 0-63 and Q~ S in rows 64-127,
//   D += [Z; M] U                completes O in rows 64-127 (rows 0-63 unchanged),
// so U and O leave TMEM from different lane quarters at the same time.
#include <cuda.h>

#include <atomic>
#include <mutex>

#include "tc_common.cuh"

namespace gdr {
namespace tc {
namespace {

using namespace umma;

struct ChainSmem {
  static constexpr uint32_t SLOT = 0;                      // 2 slots
  static constexpr uint32_t VIN = 2 * kSlotBytes;          // V [64 tok][128] SW128, 2 slabs
  static constexpr uint32_t UU = VIN + 16384;              // U [tok][128] (MN-major B)
  static constexpr uint32_t SS = UU + 16384;               // S [d_k][128] (MN-major B)
  static constexpr uint32_t OST = SS + 32768;              // output gate: O rows [64][256 B]
  static constexpr uint32_t END = OST + 16384;
  // full[2], v, mma, o, TMEM slot: in the second slot's tail, which no copy writes
  static constexpr uint32_t BARS = kSlotBytes + kSlotGam + 512;
};
static_assert(ChainSmem::BARS + 64 <= 2 * kSlotBytes, "barriers inside the second slot's tail");

// The chain CTA of the transposed state pass (no output gate): three operand slots without the
// zero tile (M where Z was), their gammas apart, and two V buffers.
struct ChainSmemT {
  static constexpr uint32_t kSlots = 3;
  static constexpr uint32_t SLOT_BYTES = 65536;    // -W / Q~ [WQ], K^ [KH], T' [T], M [Z]
  static constexpr uint32_t VIN = kSlots * SLOT_BYTES;  // V [64 tok][128] SW128 x 2 buffers
  static constexpr uint32_t GAM = VIN + 2 * 16384;  // gamma [128] fp32 per slot
  static constexpr uint32_t BARS = GAM + kSlots * 512;  // full[3], v[2], x, o; TMEM slot
  static constexpr uint32_t END = BARS + 128;
  static constexpr uint32_t kM = kSlotZ;  // M's offset in a slot
};
static_assert(ChainSmemT::END <= ChainSmem::END, "the transposed chain fits the cluster's CTAs");
static_assert(kSlotWQ + 32768 <= kSlotKH && kSlotKH + 16384 <= kSlotT &&
                  kSlotT + 8192 <= ChainSmemT::kM && ChainSmemT::kM + 8192 <= ChainSmemT::SLOT_BYTES,
              "slot tiles of the transposed chain");

struct HelperSmem {
  static constexpr uint32_t QIN = 0;              // [64][128] bf16 row-major
  static constexpr uint32_t KIN = QIN + 16384;
  static constexpr uint32_t AIN = KIN + 16384;    // [64][128] fp32 row-major
  static constexpr uint32_t KQ = AIN + 32768;     // [K~ ; Q~] 128 x 128 K-major
  static constexpr uint32_t KR = KQ + 32768;      // Kr 64 x 128
  static constexpr uint32_t KH = KR + 16384;      // K^ [tok][ch]
  static constexpr uint32_t TT = KH + 16384;      // T' 64 x 64
  static constexpr uint32_t MM = TT + 8192;       // M 64 x 64
  static constexpr uint32_t WW = MM + 8192;       // W 64 x 128
  static constexpr uint32_t SX = WW + 16384;      // solve scratch [32][32] fp32
  static constexpr uint32_t BETA = SX + 4096;
  static constexpr uint32_t ALPHA = BETA + 256;
  static constexpr uint32_t GAM = ALPHA + 256;
  static constexpr uint32_t RED = GAM + 512;
  static constexpr uint32_t GS = RED + 64;
  static constexpr uint32_t TOT = GS + 256;       // gate carries [32][128] fp32
  static constexpr uint32_t CONS = TOT + 16384;   // chunks consumed by the chain CTA (u32)
  static constexpr uint32_t BARS = CONS + 64;     // qk, alpha, mma, TMEM slot
  static constexpr uint32_t END = BARS + 64;
  static constexpr uint32_t SA = KR;              // A [64][64] fp32 (Kr is consumed by then)
  static constexpr uint32_t ST32 = WW;            // T [64][64] fp32 (W is written later)
  static constexpr uint32_t DIAGP = SX;           // q_r . k_r partials [64][16] (solve later)
};

constexpr size_t kClusterSmem =
    (ChainSmem::END > HelperSmem::END ? ChainSmem::END : HelperSmem::END) + 1024;
static_assert(kClusterSmem <= 232448, "shared memory per CTA");

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_to(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
// bulk copy from this CTA's shared memory into another CTA's, completing on its mbarrier
__device__ __forceinline__ void bulk_copy_to(uint32_t dst_cluster, uint32_t src_local,
                                             uint32_t bytes, uint32_t mbar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(dst_cluster),
      "r"(src_local), "r"(bytes), "r"(mbar_cluster)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// A plain (relaxed) store suffices for the consumed-chunk counter: the chain CTA's reads of
// the slot have completed before it is written (MMA completion observed on an mbarrier, and the
// generic reads of gamma precede a CTA barrier), and a release would also wait for the chain
// CTA's earlier output stores to global memory.
__device__ __forceinline__ void st_relaxed_remote(uint32_t addr_cluster, uint32_t v) {
  asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], %1;" ::"r"(addr_cluster), "r"(v)
               : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_local(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.cluster.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p))
               : "memory");
  return v;
}

// Waits until the chain CTA has consumed at least `need` chunks (bounded).
__device__ bool wait_consumed(const uint32_t* cons, uint32_t need) {
  bool ok = true;
  if (threadIdx.x == 0) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
      if (ld_acquire_local(cons) >= need) break;
      if (i == 0) {
        t0 = globaltimer_ns();
      } else if ((i & 63u) == 0 && globaltimer_ns() - t0 > kWaitNs) {
        ok = false;
        break;
      }
      __nanosleep(64);
    }
  }
  __syncwarp();  // lane 0 rejoins its warp before the aligned CTA barrier
  return !__syncthreads_or(!ok);
}

// The chain CTA of gated linear attention, with its state pass transposed.  The state is kept as
// S^T: the thread of TMEM lane v holds value column v, so S enters the products as an A operand
// read from tensor memory (a bf16 copy in TMEM: row m of A in lane m, two K values per 32-bit
// column, the lower K index in the low half), and the fp32 master stays in the registers of the
// thread that owns the lane (64 key channels each, two threads per lane).  Nothing of the state
// pass goes through shared memory; the helpers' slot tiles and V serve as B operands (U = V: no
// erase term).  Per chunk:
//   D^T = S^T Q~^T,  X = V^T K^,  D^T += V^T M^T   (O^T = D^T)
//   S^T <- S^T Diag(gamma) + X  in registers, and its bf16 copy.
// X has an accumulator of its own, so the previous chunk's O^T columns are stored by warps 4-7
// (one bf16 value per lane and token: 64 contiguous bytes per warp store) while this chunk's
// products run.  The freed shared memory holds three operand slots, so a slot is refilled while
// the two after it are consumed, and V is double-buffered, requested a chunk ahead.
// (The gated rule in the same arrangement -- U^T = V^T T'^T + S^T (-W)^T first, its bf16 copy in
// TMEM as the A operand of X and O^T -- was parity-green but slower than its untransposed chain,
// 1.12 against 1.08 ms on 32 heads x 32K tokens: its 66 KB hand-over per chunk, not the chain's
// own work, sets that pace.)
__device__ void chain_transposed(unsigned char* sm, const TcMaps& maps, const PrefillArgs& a,
                                 int h, int64_t t0, int64_t t1, int nch, size_t sidx,
                                 bool valid, int ncl) {
  using L = ChainSmemT;
  constexpr uint32_t kPayload = kSlotPayload - 16384 - 8192;  // no -W, no T'
  // TMEM columns: the state's bf16 copy, D^T (O^T in 64-127; two), X
  constexpr uint32_t cSB = 0, cD0 = 64, cD1 = 192, cX = 320;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, wh = warp >> 2;
  const int vv = q4 * 32 + lane;  // the value column held in this thread's TMEM lane
  const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
  const int H = a.H;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
  uint64_t* full = bars;       // [3]
  uint64_t* bar_v = bars + 3;  // [2]
  uint64_t* bar_x = bars + 5;  // X
  uint64_t* bar_o = bars + 6;  // O^T
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::BARS + 64);
  if (warp == 0) tmem_alloc(tslot, kTmemCols);
  if (tid == 0) {
    for (int i = 0; i < 7; ++i) mbar_init(bars + i, 1);
    fence_mbar_init();
    prefetch_tmap(&maps.v);
    for (int s = 0; s < (int)L::kSlots && s < nch; ++s) mbar_expect_tx(full + s, kPayload);
  }
  cta_sync_tc();
  cluster_sync();  // every CTA's barriers and counters are initialised
  const uint32_t tm = *tslot;
  auto dcol = [](int c) { return (c & 1) ? cD1 : cD0; };
  auto pack2 = [](float x, float y) {
    const __nv_bfloat162 hv = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<const uint32_t*>(&hv);
  };
  __nv_bfloat16* __restrict__ out = static_cast<__nv_bfloat16*>(a.out);
  // phases: bit s of ph_full for slot s, bit b of ph_v for V buffer b
  uint32_t ph_full = 0, ph_v = 0, ph_x = 0, ph_o = 0;
  auto issue_v = [&](int c) {  // one thread: chunk c's V tile into buffer c & 1
    unsigned char* dst = sm + L::VIN + (c & 1) * 16384;
    const int tc = (int)(t0 + (int64_t)c * kC);
    mbar_expect_tx(bar_v + (c & 1), 16384);
    tma_load_3d(dst, &maps.v, 0, h, tc, bar_v + (c & 1));
    tma_load_3d(dst + 8192, &maps.v, 64, h, tc, bar_v + (c & 1));
  };
  if (tid == 0 && nch > 0) issue_v(0);
  // the fp32 master: S^T[vv][64 wh + j] (S0, or zeros), and its bf16 copy in TMEM
  float ms[64];
  {
    const float* s0 = a.S0 ? a.S0 + sidx : nullptr;
#pragma unroll
    for (int j = 0; j < 64; ++j) ms[j] = s0 ? s0[(size_t)(64 * wh + j) * kD + vv] : 0.f;
    float pv[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) pv[i] = __uint_as_float(pack2(ms[2 * i], ms[2 * i + 1]));
    tmem_st32(tm + lane_base + cSB + 32 * wh, pv);
    tmem_wait_st();
  }
  cta_sync_tc();
  const uint32_t id_t64 = idesc_bf16(128, 64, false, false, false);  // TMEM A, K-major B, N = 64
  const uint32_t id_vk = idesc_bf16(128, 128, false, true, true);    // V^T (smem) K^
  const uint32_t id_vm = idesc_bf16(128, 64, false, true, false);    // V^T (smem) M^T
  const uint32_t cons_local = smem_u32(sm + HelperSmem::CONS);
  bool failed = false;
  int c_fail = 0;
  // warps 4-7: O^T of chunk c (columns 64-127 of its D^T) -> out rows [tc, tc + n) of head h
  auto o_drain = [&](int c, int64_t tc, int n) {
    float o[64];
    tmem_ld64(tm + lane_base + dcol(c) + 64, o);
    __nv_bfloat16* dst = out + ((size_t)tc * H + h) * kD + vv;
#pragma unroll
    for (int j = 0; j < 64; ++j)
      if (j < n) dst[(size_t)j * H * kD] = __float2bfloat16_rn(o[j]);
  };
#pragma unroll 1
  for (int c = 0; c < nch && !failed; ++c) {
    const int s = c % (int)L::kSlots, vb = c & 1;
    const int64_t tc = t0 + (int64_t)c * kC;
    const int n = (int)((t1 - tc) < (int64_t)kC ? (t1 - tc) : (int64_t)kC);
    const uint32_t slot = smem_u32(sm) + (uint32_t)s * L::SLOT_BYTES;
    const Opnd opQ{slot + kSlotWQ + 8192, 16384, false};  // Q~ rows: K-major B, N = 64
    const Opnd opKH{slot + kSlotKH, 8192, true};          // K^ [tok][ch]: MN-major B, N = 128
    const Opnd opM{slot + L::kM, 8192, false};            // M rows: K-major B, N = 64
    const Opnd opVa{smem_u32(sm + L::VIN) + (uint32_t)vb * 16384, 8192, true};  // V^T: A
    const float* gam = reinterpret_cast<const float*>(sm + L::GAM + s * 512);
    // the next V tile: its buffer's last readers, chunk c - 1's products, completed before that
    // chunk's closing barrier, which every thread passed after its wait for the buffer
    if (tid == 128 && c + 1 < nch) issue_v(c + 1);
    if (c > 0 && wh == 1) o_drain(c - 1, tc - kC, kC);
    // Waits are per thread; one that gave up is agreed on at the chunk's closing barrier.  Each
    // product barrier completes once per chunk, so no wait can see two of its phases pass.
    bool bad = false;
    bad |= !mbar_wait(full + s, (ph_full >> s) & 1u, kWaitNs);
    bad |= !mbar_wait(bar_v + vb, (ph_v >> vb) & 1u, kWaitNs);
    ph_full ^= 1u << s;
    ph_v ^= 1u << vb;
    __syncwarp();  // lanes leave their polling loops at different times
    if (n < kC) {  // the last chunk: every thread zeroes part of the V tail
      zero_v_tail<kD>(make_ctx(sm, tm, bar_x), sm + L::VIN + vb * 16384, n);
      __syncthreads();
    }
    fence_after_sync();
    if (warp == 0) {  // S^T Q~^T, X = V^T K^, then O^T += V^T M^T
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16_tmem_a_elect(tm + dcol(c) + 64, tm + cSB + 8 * ks, opQ.at(16 * ks), id_t64,
                              ks > 0 ? 1u : 0u);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16_elect(tm + cX, opVa.at(16 * ks), opKH.at(16 * ks), id_vk, ks > 0 ? 1u : 0u);
      mma_commit_elect(bar_x);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16_elect(tm + dcol(c) + 64, opVa.at(16 * ks), opM.at(16 * ks), id_vm, 1u);
      mma_commit_elect(bar_o);
    }
    bad |= !mbar_wait(bar_x, ph_x, kWaitNs);
    ph_x ^= 1u;
    __syncwarp();
    fence_after_sync();
    {  // S^T <- S^T Diag(gamma) + X on this thread's 64 key channels, and its bf16 copy
      const uint32_t k0 = (uint32_t)(64 * wh);
      float xv[64];
      tmem_ld64(tm + lane_base + cX + k0, xv);
#pragma unroll
      for (int j = 0; j < 64; j += 4) {
        const float4 g4 = *reinterpret_cast<const float4*>(gam + k0 + j);
        ms[j] = fmaf(g4.x, ms[j], xv[j]);
        ms[j + 1] = fmaf(g4.y, ms[j + 1], xv[j + 1]);
        ms[j + 2] = fmaf(g4.z, ms[j + 2], xv[j + 2]);
        ms[j + 3] = fmaf(g4.w, ms[j + 3], xv[j + 3]);
      }
      float pv[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) pv[i] = __uint_as_float(pack2(ms[2 * i], ms[2 * i + 1]));
      tmem_st32(tm + lane_base + cSB + 32 * wh, pv);
    }
    tmem_wait_st();
    // the slot is consumed once O's products are complete (gamma was read above, before the
    // barrier below): re-arm it for chunk c + 3 and tell the helpers, one warp per helper
    if (tid == 0) bad |= !mbar_wait(bar_o, ph_o, kWaitNs);
    __syncwarp();
    ph_o ^= 1u;
    fence_before_sync();
    if (__syncthreads_or(bad)) { failed = true; c_fail = c; break; }
    fence_after_sync();
    if (tid == 0 && c + (int)L::kSlots < nch) mbar_expect_tx(full + s, kPayload);
    if (lane == 0 && warp >= 1 && warp < ncl)
      st_relaxed_remote(map_to(cons_local, (uint32_t)warp), (uint32_t)(c + 1));
  }
  if (!failed && nch > 0 && wh == 1) {  // the last chunk's O rows
    const int64_t tl = t0 + (int64_t)(nch - 1) * kC;
    o_drain(nch - 1, tl, (int)(t1 - tl));
  }
  if (failed) {
    if (tid == 0) report(a, GDR_DEVCHECK_TIMEOUT);
    // the next chunk's V tile, requested at the top of the failed chunk, lands before the CTA
    // exits
    if (c_fail + 1 < nch)
      mbar_wait(bar_v + ((c_fail + 1) & 1), (ph_v >> ((c_fail + 1) & 1)) & 1u, kWaitNs);
  } else if (valid && a.S_final) {
#pragma unroll
    for (int j = 0; j < 64; ++j) a.S_final[sidx + (size_t)(64 * wh + j) * kD + vv] = ms[j];
  }
  cta_sync_tc();
  if (warp == 0) tmem_dealloc(tm, kTmemCols);
}

// ERASE = false: gated linear attention.  The helpers skip the triangular solve and W (a chunk's
// hand-over shrinks from 66 KB to 41 KB), and the chain CTA runs chain_transposed.
// OGATE: the output gate out = o * sigmoid(g) on the stored output rows (a.og).
// PRO: the layer prologue on load (a.prologue): the helpers map the staged raw q, k, alpha tiles
// and the scalar gates before the gate stage.
template <bool CHANNEL, bool ERASE = true, bool OGATE = false, bool PRO = false>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_cluster_kernel(const __grid_constant__ TcMaps maps, const PrefillArgs a, int ncl) {
  constexpr bool kAlphaTile = CHANNEL;
  constexpr int DV = kD, DH = DV / 2;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t crank = cluster_rank();
  const int nh = ncl - 1;
  const int H = a.H;
  const int pair = blockIdx.x / ncl;
  const int h = pair % H;
  const int seq = a.order ? a.order[pair / H] : pair / H;
  int64_t t0 = 0, t1 = 0;
  const bool valid = seq_range(a, seq, t0, t1);
  if (!valid) t1 = t0;  // skip the work but keep the cluster barriers
  const int nch = (int)((t1 - t0 + kC - 1) / kC);
  const size_t sidx = ((size_t)seq * H + h) * kD * kD;
  bool failed = false;

  // bytes a helper copies into a slot per chunk (gated linear attention: T' = I and W = 0 stay
  // in the slots from the start instead)
  constexpr uint32_t kPayload = ERASE ? kSlotPayload : kSlotPayload - 16384 - 8192;
  if (crank == 0 && !ERASE) {
    chain_transposed(sm, maps, a, h, t0, t1, nch, sidx, valid, ncl);
  } else if (crank == 0) {
    // ===================================================================== chain CTA
    // (the gated rule: S itself in TMEM, S and U as B operands in shared memory)
    using L = ChainSmem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* full = bars;  // [2]
    uint64_t* bar_v = bars + 2;
    uint64_t* bar_o = bars + 4;  // [Z; M] U of the chunk
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 5);
    if (warp == 0) tmem_alloc(tslot, kTmemCols);
    for (int i = tid; i < 2 * 8192 / 16; i += kThreads) {  // the Z tiles of both slots
      *reinterpret_cast<uint4*>(sm + L::SLOT + (i >> 9) * kSlotBytes + kSlotZ + (i & 511) * 16) =
          make_uint4(0, 0, 0, 0);
    }
    fence_async_smem();
    if (tid == 0) {
      for (int i = 0; i < 5; ++i) mbar_init(bars + i, 1);
      fence_mbar_init();
      prefetch_tmap(&maps.v);
      for (int s = 0; s < 2 && s < nch; ++s) mbar_expect_tx(full + s, kPayload);
    }
    cta_sync_tc();
    cluster_sync();  // every CTA's barriers and counters are initialised
    TcCtx x = make_ctx(sm, *tslot, bars + 3);
    x.prologue = PRO;
    uint32_t ph_v = 0, ph_full[2] = {0, 0};
    __nv_bfloat16* __restrict__ out = static_cast<__nv_bfloat16*>(a.out);
    auto issue_v = [&](int64_t tc) {  // one thread
      mbar_expect_tx(bar_v, 16384);
      tma_load_3d(sm + L::VIN, &maps.v, 0, h, (int)tc, bar_v);
      tma_load_3d(sm + L::VIN + 8192, &maps.v, 64, h, (int)tc, bar_v);
    };
    if (tid == 0 && nch > 0) issue_v(t0);
    s_init<DH>(x, a.S0 ? a.S0 + sidx + (size_t)x.lrow * kD : nullptr, sm + L::SS);
    cta_sync_tc();  // every row of the bf16 state tile is written before the first MMA
    const Opnd opV{x.sb + L::VIN, 8192, true};
    const Opnd opU{x.sb + L::UU, 8192, true};
    const Opnd opS{x.sb + L::SS, 16384, true};
    const uint32_t id_d = idesc_bf16(128, DV, false, false, true);  // K-major A, MN-major B
    const uint32_t id_s = idesc_bf16(128, DV, false, true, true);   // K^ as MN-major A
    const uint32_t cons_local = smem_u32(sm + HelperSmem::CONS);
    const bool u_rows = (warp & 3) < 2;  // TMEM lanes 0-63 (U) or 64-127 (O) of this warp
    const int drow = (warp & 3) * 32 + (tid & 31) - (u_rows ? 0 : 64);
    uint32_t ph_o = 0;

    // D alternates between two accumulators, so a chunk's output rows are written out during the
    // next chunk.  The state update K^^T U goes to a third accumulator (kColU) and is folded into
    // the fp32 master as S <- gamma S + K^^T U when the bf16 operand copy is made, so no TMEM
    // load or store of the master runs while the chunk's first products are on the tensor pipe.
    auto d_col = [](int c) { return (c & 1) ? kColAM : kColWO; };
    // O rows (TMEM lanes 64-127 of D) -> out rows [tc, tc + n) of head h.  A warp's 32 rows x 64
    // columns go through its own 4 KB of the bf16 state tile (the rows it rewrites itself in
    // s_update, free between the chunk's first MMA and that update), so that each global store
    // instruction writes four whole 128-byte row segments instead of 32 scattered pieces.
    // Output gate: the O rows of chunk c - 1 leave TMEM in chunk c's U window into the staging
    // tile OST (the O warps, 8 KB-swizzled rows of 256 bytes); all eight warps then gate and store
    // them during chunk c + 1's first MMAs, when every warp is idle, with the gate values each
    // thread loaded a chunk earlier (the rows were prefetched into L2 a chunk before that).
    uint4 gq[4];
    auto stage_o = [&](int c) {  // O warps: rows 0-63 of the staged tile
      float v[64];
      tmem_ld64(x.tm + x.lane_base + d_col(c) + x.wh * 64, v);
      const int r = (warp & 3) * 32 + (tid & 31) - 64;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        __align__(16) __nv_bfloat162 hv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          hv[i] = __floats2bfloat162_rn(v[8 * j + 2 * i], v[8 * j + 2 * i + 1]);
        *reinterpret_cast<uint4*>(sm + L::OST + r * 256 + (((8 * x.wh + j) ^ (r & 15)) << 4)) =
            *reinterpret_cast<const uint4*>(hv);
      }
    };
    auto load_og = [&](int64_t tc, int n) {  // every thread: 4 of the tile's 16-byte chunks
      const __nv_bfloat16* og = static_cast<const __nv_bfloat16*>(a.og);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = tid + kThreads * j, r = e >> 4, ch = e & 15;
        gq[j] = r < n ? *reinterpret_cast<const uint4*>(og + ((size_t)(tc + r) * H + h) * kD + ch * 8)
                      : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    auto store_gated = [&](int64_t tc, int n) {  // every thread: the same 4 chunks, gated
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = tid + kThreads * j, r = e >> 4, ch = e & 15;
        if (r < n) {
          uint4 w = *reinterpret_cast<const uint4*>(sm + L::OST + r * 256 + ((ch ^ (r & 15)) << 4));
          __nv_bfloat162* hw = reinterpret_cast<__nv_bfloat162*>(&w);
          const __nv_bfloat162* hg = reinterpret_cast<const __nv_bfloat162*>(&gq[j]);
#pragma unroll
          for (int i = 0; i < 4; ++i) hw[i] = gate2_bf16(hw[i], hg[i]);
          *reinterpret_cast<uint4*>(out + ((size_t)(tc + r) * H + h) * kD + ch * 8) = w;
        }
      }
    };
    auto o_store = [&](int c, int64_t tc, int n) {
      float v[64];
      tmem_ld64(x.tm + x.lane_base + d_col(c) + x.wh * 64, v);
      unsigned char* stage = sm + L::SS + x.wh * 16384 + (warp & 3) * 4096;
      const int lane = tid & 31;
#pragma unroll
      for (int j = 0; j < 64; j += 8) {
        __align__(16) __nv_bfloat162 hv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) hv[i] = __floats2bfloat162_rn(v[j + 2 * i], v[j + 2 * i + 1]);
        *reinterpret_cast<uint4*>(stage + lane * 128 + (((j >> 3) ^ (lane & 7)) << 4)) =
            *reinterpret_cast<const uint4*>(hv);
      }
      __syncwarp();
      const int row0 = (warp & 3) * 32 - 64;  // this warp's first O row
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int r = 4 * j + (lane >> 3), ch = lane & 7;
        const uint4 w = *reinterpret_cast<const uint4*>(stage + r * 128 + ((ch ^ (r & 7)) << 4));
        if (row0 + r < n)
          *reinterpret_cast<uint4*>(out + ((size_t)(tc + row0 + r) * H + h) * kD + x.wh * 64 +
                                    ch * 8) = w;
      }
      __syncwarp();
    };
    // S <- gamma S + K^^T U on this thread's row (key channel) and column half; the bf16 copy of
    // the new state is the next chunk's B operand
    auto s_update = [&](float gm) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t c0 = (uint32_t)(x.wh * 64 + hh * 32);
        float v[64];
        tmem_ld32x2(x.tm + x.lane_base + kColS + c0, x.tm + x.lane_base + kColU + c0, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = fmaf(gm, v[j], v[32 + j]);
        tmem_st32(x.tm + x.lane_base + kColS + c0, *reinterpret_cast<const float(*)[32]>(v));
#pragma unroll
        for (int j = 0; j < 32; j += 8) st_chunk8(sm + L::SS, 16384, x.lrow, (int)c0 + j, v + j);
      }
      tmem_wait_st();
      fence_async_smem();
    };
#pragma unroll 1
    for (int c = 0; c < nch && !failed; ++c) {
      const int s = c & 1;
      const int64_t tc = t0 + (int64_t)c * kC;
      const int n = (int)((t1 - tc) < (int64_t)kC ? (t1 - tc) : (int64_t)kC);
      const uint32_t slot = L::SLOT + s * kSlotBytes;
      const Opnd opTZ{x.sb + slot + kSlotT, 16384, false};
      const Opnd opZM{x.sb + slot + kSlotZ, 16384, false};
      const Opnd opWQ{x.sb + slot + kSlotWQ, 16384, false};
      const Opnd opKH{x.sb + slot + kSlotKH, 8192, true};
      // Waits inside a chunk are per thread (no CTA barrier where the mbarrier already orders
      // what a thread reads); a wait that gave up is remembered in `bad`, and the CTA agrees on
      // it at the chunk's closing barrier and unwinds.
      bool bad = false;
      float gm;
      if (OGATE && tid == 96)  // this chunk's gate rows into L2, read back in the next chunk
        tma_prefetch_l2_3d(&maps.og, 0, h, (int)tc);
      {  // the chunk's operands (every thread reads gamma of its row now) and V tile
        bad |= !mbar_wait(full + s, ph_full[s], kWaitNs);
        bad |= !mbar_wait(bar_v, ph_v, kWaitNs);
        ph_full[s] ^= 1u;
        ph_v ^= 1u;
        gm = reinterpret_cast<const float*>(sm + slot + kSlotGam)[x.lrow];
        __syncwarp();  // lanes leave their polling loops at different times
        if (n < kC) {  // the last chunk: every thread zeroes part of the V tail
          zero_v_tail<DV>(x, sm + L::VIN, n);
          __syncthreads();
        }
        fence_after_sync();
      }
      // D = [T'; Z] V + [-W; Q~] S, alone on the tensor pipe
      if (warp == 0) {
        mma_run<kC>(x.tm + d_col(c), opTZ, opV, id_d, false);
        mma_run<kD>(x.tm + d_col(c), opWQ, opS, id_d, true);
        mma_commit_elect(x.bar_mma);
      }
      if constexpr (OGATE) {  // chunk c - 2's gated rows leave the staging tile
        if (c >= 2) store_gated(tc - 2 * kC, kC);
        if (c >= 1) load_og(tc - kC, kC);
        __syncthreads();  // the staging tile is free for chunk c - 1's rows below
      }
      bad |= !mbar_wait(x.bar_mma, x.ph_mma, kWaitNs);
      x.ph_mma ^= 1u;
      fence_after_sync();
      // (with the output gate every thread has passed its V wait at the barrier above)
      if (OGATE && tid == 0 && c + 1 < nch) issue_v(tc + kC);  // V is consumed
      __syncwarp();
      // Named barrier 1: the U warps wait at it, the O warps only arrive, each after its own
      // waits for this chunk's V tile and first products.  So neither barrier can complete a
      // phase again (V of the next chunk, the second products) while a thread is still polling
      // the previous one -- a parity wait that slept through two phases would sleep on.
      if (u_rows) {
        // U rows -> bf16 [tok][DV] tile (MN-major B operand); then K^^T U (on the chain's
        // critical path) and O += M U are issued
        float v[64];
        tmem_ld64(x.tm + x.lane_base + d_col(c) + x.wh * 64, v);
#pragma unroll
        for (int j = 0; j < 64; j += 8) st_chunk8(sm + L::UU, 8192, drow, x.wh * 64 + j, v + j);
        fence_async_smem();
        fence_before_sync();
        asm volatile("bar.sync 1, 256;" ::: "memory");
        fence_after_sync();
        if (warp == 0) {
          mma_run<kC>(x.tm + kColU, opKH, opU, id_s, false);
          mma_commit_elect(x.bar_mma);
          mma_run<kC>(x.tm + d_col(c), opZM, opU, id_d, true);
          mma_commit_elect(bar_o);
        }
        if (!OGATE && tid == 32 && c + 1 < nch) issue_v(tc + kC);  // V is consumed, on every thread
      } else {
        asm volatile("bar.arrive 1, 256;" ::: "memory");
        if (c > 0) {
          if constexpr (OGATE) {
            stage_o(c - 1);
          } else {
            o_store(c - 1, tc - kC, kC);  // the previous chunk's output rows, off the tensor pipe
          }
        }
      }
      bad |= !mbar_wait(x.bar_mma, x.ph_mma, kWaitNs);
      x.ph_mma ^= 1u;
      __syncwarp();
      fence_after_sync();
      s_update(gm);
      // the slot is consumed once O's MMA is complete (gamma was read before the barrier below):
      // re-arm it for chunk c + 2 and tell the helpers
      if (tid == 0) bad |= !mbar_wait(bar_o, ph_o, kWaitNs);
      __syncwarp();  // warp 0 reconverges before the aligned CTA barrier below
      ph_o ^= 1u;
      fence_before_sync();
      if (__syncthreads_or(bad)) { failed = true; break; }
      fence_after_sync();
      if (tid == 0) {
        if (c + 2 < nch) mbar_expect_tx(full + s, kPayload);
        for (int r = 1; r < ncl; ++r) st_relaxed_remote(map_to(cons_local, r), (uint32_t)(c + 1));
      }
    }
    if constexpr (OGATE) {  // the last two chunks' rows
      if (!failed && nch > 0) {
        const int64_t tl = t0 + (int64_t)(nch - 1) * kC;
        if (nch >= 2) store_gated(tl - kC, kC);
        __syncthreads();
        if (!u_rows) stage_o(nch - 1);
        load_og(tl, (int)(t1 - tl));
        __syncthreads();
        store_gated(tl, (int)(t1 - tl));
      }
    } else if (!failed && nch > 0 && !u_rows) {
      const int64_t tl = t0 + (int64_t)(nch - 1) * kC;
      o_store(nch - 1, tl, (int)(t1 - tl));
    }
    if (failed) {
      if (tid == 0) report(a, GDR_DEVCHECK_TIMEOUT);
      mbar_wait(bar_v, ph_v, kWaitNs);
    } else if (valid && a.S_final) {
      s_final<DH>(x, a.S_final + sidx + (size_t)x.lrow * kD);
    }
    cta_sync_tc();
    if (warp == 0) tmem_dealloc(x.tm, kTmemCols);
  } else {
    // ===================================================================== helper CTA
    using L = HelperSmem;
    const int hid = (int)crank - 1;
    float* sBeta = reinterpret_cast<float*>(sm + L::BETA);
    float* sAlpha = reinterpret_cast<float*>(sm + L::ALPHA);
    uint32_t* cons = reinterpret_cast<uint32_t*>(sm + L::CONS);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* bar_qk = bars + 0;
    uint64_t* bar_a = bars + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3);
    if (warp == 0) tmem_alloc(tslot, kTmemCols);
    if (tid == 0) {
      *cons = 0;
      for (int i = 0; i < 3; ++i) mbar_init(bars + i, 1);
      fence_mbar_init();
      prefetch_tmap(&maps.q);
      prefetch_tmap(&maps.k);
      if (kAlphaTile) prefetch_tmap(&maps.alpha);
    }
    cta_sync_tc();
    cluster_sync();
    TcCtx x = make_ctx(sm, *tslot, bars + 2);
    x.prologue = PRO;
    zero_upper_tp(sm + L::TT, tid);
    uint32_t ph_qk = 0, ph_a = 0;
    // the chain CTA's layout: three slots (gated linear attention's transposed state pass) or
    // two (the gated rule)
    constexpr bool kT = !ERASE;
    constexpr int kNSlot = kT ? (int)ChainSmemT::kSlots : 2;
    constexpr uint32_t kSlotStride = kT ? ChainSmemT::SLOT_BYTES : kSlotBytes;
    const uint32_t chain_full = map_to(smem_u32(sm + (kT ? ChainSmemT::BARS : ChainSmem::BARS)), 0);
    const uint32_t chain_slots = map_to(smem_u32(sm + ChainSmem::SLOT), 0);
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
    auto load_scalars = [&](int64_t tc, float& b, float& al) {
      b = 0.f;
      al = 1.f;
      if (tid < kC && tc + tid < t1) {
        const size_t o = (size_t)(tc + tid) * H + h;
        if (ERASE) b = a.beta[o];
        if (!CHANNEL) al = a.alpha[o];
      }
    };
    float nb_beta = 0.f, nb_alpha = 1.f;
    if (hid < nch) {
      issue_qk(t0 + (int64_t)hid * kC);
      issue_a(t0 + (int64_t)hid * kC);
      load_scalars(t0 + (int64_t)hid * kC, nb_beta, nb_alpha);
    }
#pragma unroll 1
    for (int c = hid; c < nch && !failed; c += nh) {
      const int64_t tc = t0 + (int64_t)c * kC;
      const int n = (int)((t1 - tc) < (int64_t)kC ? (t1 - tc) : (int64_t)kC);
      const int cn = c + nh;  // this helper's next chunk
      const int64_t tn = t0 + (int64_t)cn * kC;
      if (tid < kC) {  // (the layer prologue maps the live tokens' raw gates here, not at the load)
        const bool pro = PRO && tid < n;
        sBeta[tid] = pro && ERASE ? sigmoid_ftz(nb_beta) : nb_beta;
        sAlpha[tid] = pro && !CHANNEL ? sigmoid_ftz(nb_alpha) : nb_alpha;
      }
      if (cn < nch) load_scalars(tn, nb_beta, nb_alpha);
      {  // the chunk's q, k (and alpha) tiles: per-thread waits, one barrier
        bool ok = mbar_wait(bar_qk, ph_qk, kWaitNs);
        ph_qk ^= 1u;
        if (kAlphaTile) {
          ok &= mbar_wait(bar_a, ph_a, kWaitNs);
          ph_a ^= 1u;
        }
        if (__syncthreads_or(!ok)) { failed = true; break; }
      }
      // the previous chunk's first copy group (Q~, K^, gamma) reads its tiles while the gate
      // prefix runs; the gate waits for it before it rewrites them
      const bool safe = gate_stage<L, CHANNEL>(x, n, [&] {
        if (tid == 0) bulk_wait_read<1>();
        __syncwarp();
      });
      // ... and the second (-W, T', M), before the Gram epilogue rewrites M
      if (tid == 0) bulk_wait_read<0>();
      __syncwarp();
      fence_async_smem();
      cta_sync_tc();
      if (safe && cn < nch) {
        issue_qk(tn);
        issue_a(tn);
      }
      if (!gram_stage<L, CHANNEL>(x, n, safe)) { failed = true; break; }
      if (!safe && cn < nch) {
        issue_qk(tn);
        issue_a(tn);
      }
      if (ERASE) {
        solve_stage<L>(x);
        if (!w_stage<L>(x, false, Opnd{0, 0, false}, 0)) { failed = true; break; }
        w_epilogue<L, true>(x);  // -W
      }
      fence_async_smem();
      cta_sync_tc();
      // hand the operands over: slot c mod kNSlot is free once chunk c - kNSlot has been consumed
      if (c >= kNSlot && !wait_consumed(cons, (uint32_t)(c - kNSlot + 1))) { failed = true; break; }
      if (tid == 0) {
        const int sl = c % kNSlot;
        const uint32_t dst = chain_slots + (uint32_t)sl * kSlotStride;
        const uint32_t mbar = chain_full + (uint32_t)sl * 8u;
        const uint32_t gam = kT ? chain_slots + ChainSmemT::GAM + (uint32_t)sl * 512u : dst + kSlotGam;
        const uint32_t src = x.sb;
        bulk_copy_to(dst + kSlotWQ + 8192, src + L::KQ + 8192, 8192, mbar);    // Q~, channels 0-63
        bulk_copy_to(dst + kSlotWQ + 24576, src + L::KQ + 24576, 8192, mbar);  // Q~, 64-127
        bulk_copy_to(dst + kSlotKH, src + L::KH, 16384, mbar);
        bulk_copy_to(gam, src + L::GAM, 512, mbar);
        bulk_commit();
        if (ERASE) {
          bulk_copy_to(dst + kSlotWQ, src + L::WW, 8192, mbar);           // -W, channels 0-63
          bulk_copy_to(dst + kSlotWQ + 16384, src + L::WW + 8192, 8192, mbar);  // -W, 64-127
          bulk_copy_to(dst + kSlotT, src + L::TT, 8192, mbar);
        }
        bulk_copy_to(dst + (kT ? ChainSmemT::kM : kSlotM), src + L::MM, 8192, mbar);
        bulk_commit();
      }
    }
    if (tid == 0) bulk_wait_all();  // every copy into the chain CTA has landed
    if (failed) {
      if (tid == 0) report(a, GDR_DEVCHECK_TIMEOUT);
      mbar_wait(bar_qk, ph_qk, kWaitNs);
      if (kAlphaTile) mbar_wait(bar_a, ph_a, kWaitNs);
    }
    cta_sync_tc();
    if (warp == 0) tmem_dealloc(x.tm, kTmemCols);
  }
  cluster_sync();  // no CTA leaves while the cluster may still address its shared memory
}

template <bool CHANNEL, bool ERASE, bool OGATE = false>
cudaError_t launch_typed(const gdr_shape& sh, const PrefillArgs& a, const TcMaps& maps, int ncl,
                         cudaStream_t s) {
  auto kern = a.prologue ? prefill_cluster_kernel<CHANNEL, ERASE, OGATE, true>
                         : prefill_cluster_kernel<CHANNEL, ERASE, OGATE, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kClusterSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sh.n_seqs * (unsigned)sh.H * (unsigned)ncl, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kClusterSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ncl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps, a, ncl);
}

// co-resident clusters of `ncl` CTAs of this kernel on the current device (0 if unknown)
constexpr int kMaxDevices = 64;
int max_active_clusters(int ncl) {
  static std::atomic<int> cache[kMaxDevices][9];
  static std::once_flag once;
  std::call_once(once, [] {
    for (auto& row : cache)
      for (auto& v : row) v.store(-1);
  });
  int dev = 0;
  if (ncl < 2 || ncl > 8 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return 0;
  const int known = cache[dev][ncl].load();
  if (known >= 0) return known;
  auto kern = prefill_cluster_kernel<true>;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kClusterSmem) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ncl, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kClusterSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ncl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  cache[dev][ncl].store(n);
  return n;
}

}  // namespace

// The largest cluster (1 chain CTA + up to 7 helpers) of which one per (sequence, head) chain
// fits on the device at once; 1 (the one-CTA kernel) when even pairs of CTAs do not fit.
int cluster_size_for(const gdr_shape& sh) {
  const long pairs = (long)sh.n_seqs * sh.H;
  for (int ncl = 8; ncl >= 2; --ncl)
    if (pairs <= max_active_clusters(ncl)) return ncl;
  return 1;
}

cudaError_t launch_prefill_cluster(const gdr_shape& sh, const PrefillArgs& a, const TcMaps& maps,
                                   int ncl, bool erase, cudaStream_t s) {
  const bool ch = sh.gate == GDR_GATE_CHANNEL;
  if (!erase)
    return ch ? launch_typed<true, false>(sh, a, maps, ncl, s)
              : launch_typed<false, false>(sh, a, maps, ncl, s);
  if (a.og)
    return ch ? launch_typed<true, true, true>(sh, a, maps, ncl, s)
              : launch_typed<false, true, true>(sh, a, maps, ncl, s);
  return ch ? launch_typed<true, true>(sh, a, maps, ncl, s)
            : launch_typed<false, true>(sh, a, maps, ncl, s);
}

}  // namespace tc
}  // namespace gdr
