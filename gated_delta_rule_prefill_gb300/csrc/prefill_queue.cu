// prefill_queue.cu -- the tensor-core prefill for workloads with few (sequence, head) chains, as one
// cooperative launch that fills every SM: P chain CTAs and G - P helper CTAs sharing a work queue.
//
// The chunk recurrence of a chain is sequential, but most of a chunk's work does not depend on
// the state: the gate prologue, the decay-weighted Gram matrices, the triangular solve and
// W = T' K~ (stages 1-4 of prefill_tc.cu).  Here CTA p < P runs only the state pass of chain p
// (U = T' V - W S, O = Q~ S + M U, S <- gamma S + K^^T U), and the helper CTAs take work items --
// (chain, chunk) pairs in chunk-major order, from an atomic counter -- run stages 1-4 for them and
// write the operands the state pass needs (Q~, K^, -W, M, T' in bf16 and gamma: 66 KB) straight
// from their epilogues into slot c mod R of the chain's ring in the workspace (global memory,
// resident in L2).  Once a chunk's stores are fenced, the helper sets ready[p][c mod R] = c + 1;
// the chain CTA bulk-loads the slot into one of two local shared-memory slots one chunk ahead and,
// as soon as the load has landed, sets loaded[p] = c + 1, which a helper waits for before it
// writes chunk c + R into the same ring slot.  Items are handed out in increasing chunk order and
// a helper hands its previous chunk over before it waits for a ring slot, so every chunk a helper
// waits on was taken earlier by a helper that waits only on earlier chunks: no cycle.  The cooperative launch guarantees that all CTAs are resident.  Every wait is bounded;
// a timeout records GDR_DEVCHECK_TIMEOUT and the CTA returns.
//
// The chain's products are M = 128 MMAs over stacked operands (an M = 64 tcgen05.mma takes as
// long as an M = 128 one): with a zero tile Z between T' and M in the slot,
//   D = [T'; Z] V + [-W; Q~] S   gives U in rows 0-63 and Q~ S in rows 64-127,
//   D += [Z; M] U                completes O in rows 64-127 (rows 0-63 unchanged).
#include <cuda.h>

#include "tc_common.cuh"

namespace gdr {
namespace tc {
namespace {

using namespace umma;

constexpr int kR = WorkspaceLayout::kRingSlots;
static_assert(WorkspaceLayout::kRingSlotBytes == kSlotBytes, "ring slot = local slot image");

struct QChainSmem {
  static constexpr uint32_t SLOT = 0;              // 2 local operand slots
  static constexpr uint32_t VIN = 2 * kSlotBytes;  // V [64 tok][128] SW128, 2 slabs
  static constexpr uint32_t UU = VIN + 16384;      // U [tok][128] (MN-major B)
  static constexpr uint32_t SS = UU + 16384;       // S [d_k][128] (MN-major B)
  static constexpr uint32_t BARS = SS + 32768;     // full[2], v, mma, o, TMEM slot
  static constexpr uint32_t END = BARS + 64;
};

struct QHelperSmem {
  static constexpr uint32_t QIN = 0;              // [64][128] bf16 row-major
  static constexpr uint32_t KIN = QIN + 16384;
  static constexpr uint32_t AIN = KIN + 16384;    // [64][128] fp32 row-major
  static constexpr uint32_t KQ = AIN + 32768;     // [K~ ; Q~] 128 x 128 K-major
  static constexpr uint32_t KR = KQ + 32768;      // Kr 64 x 128
  static constexpr uint32_t KH = KR + 16384;      // (unused: K^ goes to the ring only)
  static constexpr uint32_t TT = KH;              // T' 64 x 64
  static constexpr uint32_t MM = TT + 8192;       // (unused: M goes to the ring only)
  static constexpr uint32_t WW = MM;              // (unused: -W goes to the ring only)
  static constexpr uint32_t ST32 = TT + 8192;     // T [64][64] fp32
  static constexpr uint32_t SX = ST32 + 16384;    // solve scratch [32][32] fp32
  static constexpr uint32_t BETA = SX + 4096;
  static constexpr uint32_t ALPHA = BETA + 256;
  static constexpr uint32_t GAM = ALPHA + 256;
  static constexpr uint32_t RED = GAM + 512;
  static constexpr uint32_t GS = RED + 64;
  static constexpr uint32_t TOT = GS + 256;       // gate carries [32][128] fp32
  static constexpr uint32_t ITEM = TOT + 16384;   // the next work item (int32 x 2, x 2 buffers)
  static constexpr uint32_t CHAINS = ITEM + 64;   // per chain: first token, tokens, head [76]
  static constexpr uint32_t BARS = CHAINS + 76 * 16;  // qk, alpha, mma, TMEM slot
  static constexpr uint32_t END = BARS + 64;
  static constexpr uint32_t SA = KR;              // A [64][64] fp32 (Kr is consumed by then)
  static constexpr uint32_t DIAGP = SX;           // q_r . k_r partials [64][16] (solve later)
};

constexpr size_t kQueueSmem =
    (QChainSmem::END > QHelperSmem::END ? QChainSmem::END : QHelperSmem::END) + 1024;
static_assert(kQueueSmem <= 232448, "shared memory per CTA");

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// A plain (relaxed) store suffices for the loaded counter: it is written after the bulk load of
// the ring slot has completed (observed on an mbarrier), and a release would also wait for the
// chain CTA's earlier output stores.
__device__ __forceinline__ void st_relaxed_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// bulk copy from global memory into this CTA's shared memory, completing on its mbarrier
__device__ __forceinline__ void bulk_load(uint32_t dst_local, const void* src, uint32_t bytes,
                                          uint32_t mbar_local) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst_local), "l"(src), "r"(bytes), "r"(mbar_local)
      : "memory");
}
// Polls *p >= want (one thread; bounded).  Returns false if it gave up.
__device__ bool poll_ge(const uint32_t* p, uint32_t want) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (ld_acquire_gpu(p) >= want) return true;
    if (i == 0) {
      t0 = globaltimer_ns();
    } else if ((i & 63u) == 0 && globaltimer_ns() - t0 > kWaitNs) {
      return false;
    }
    __nanosleep(64);
  }
}

// chain p -> (sequence, head, token range); false if the sequence failed its check
__device__ __forceinline__ bool chain_range(const PrefillArgs& a, int p, int& h, int& seq,
                                            int64_t& t0, int64_t& t1) {
  h = p % a.H;
  seq = a.order ? a.order[p / a.H] : p / a.H;
  return seq_range(a, seq, t0, t1);
}

template <bool CHANNEL>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_queue_kernel(const __grid_constant__ TcMaps maps, const PrefillArgs a, int P) {
  constexpr bool kAlphaTile = CHANNEL;
  constexpr int DV = kD, DH = DV / 2;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int H = a.H;
  uint32_t* q_next = a.ring_flags;          // work-item counter
  uint32_t* q_ready = a.ring_flags + 1;     // [P][R]
  uint32_t* q_loaded = q_ready + P * kR;    // [P]

  if ((int)blockIdx.x < P) {
    // ===================================================================== chain CTA
    using L = QChainSmem;
    const int p = blockIdx.x;
    int h, seq;
    int64_t t0 = 0, t1 = 0;
    if (!chain_range(a, p, h, seq, t0, t1)) return;
    const int nch = (int)((t1 - t0 + kC - 1) / kC);
    const size_t sidx = ((size_t)seq * H + h) * kD * kD;
    const unsigned char* ring = a.ring + (size_t)p * kR * kSlotBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* full = bars;  // [2]
    uint64_t* bar_v = bars + 2;
    uint64_t* bar_o = bars + 4;  // [Z; M] U of the chunk
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 5);
    if (warp == 0) tmem_alloc(tslot, kTmemCols);
    for (int i = tid; i < 2 * 8192 / 16; i += kThreads) {  // the Z tiles of both local slots
      *reinterpret_cast<uint4*>(sm + L::SLOT + (i >> 9) * kSlotBytes + kSlotZ + (i & 511) * 16) =
          make_uint4(0, 0, 0, 0);
    }
    fence_async_smem();
    if (tid == 0) {
      for (int i = 0; i < 5; ++i) mbar_init(bars + i, 1);
      fence_mbar_init();
      prefetch_tmap(&maps.v);
    }
    cta_sync_tc();
    TcCtx x = make_ctx(sm, *tslot, bars + 3);
    x.prologue = a.prologue;
    // The loader thread (warp 2, lane 0) loads chunk cc's ring slot into local slot cc & 1 once a
    // helper has marked it ready.  Warp 0 issues the MMAs and warp 2 stores O rows while they run,
    // so a look at a ring flag (a global-memory round trip) is started at the top of a chunk and
    // its value used after the O rows: the latency hides behind them.  load_chunk blocks (bounded)
    // for the flag; 1 = issued, -1 = timed out.
    const bool loader = tid == 64;
    auto issue_load = [&](int cc) {
      fence_proxy_async_global();
      const unsigned char* src = ring + (size_t)(cc % kR) * kSlotBytes;
      const uint32_t dst = x.sb + L::SLOT + (uint32_t)(cc & 1) * kSlotBytes;
      const uint32_t mb = smem_u32(full + (cc & 1));
      mbar_expect_tx(full + (cc & 1), kSlotPayload);
      bulk_load(dst, src, kSlotZ, mb);                                       // -W, Q~, K^, T'
      bulk_load(dst + kSlotM, src + kSlotM, kSlotBytes - kSlotM - 512, mb);  // M, gamma
    };
    auto load_chunk = [&](int cc) -> int {
      if (!poll_ge(q_ready + p * kR + (cc % kR), (uint32_t)(cc + 1))) return -1;
      issue_load(cc);
      return 1;
    };
    int issued = 0, landed = 0;  // chunks whose ring load the loader has issued / seen complete
    uint32_t ph_v = 0, ph_full[2] = {0, 0}, ph_o = 0;
    bool failed = false;
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
    const bool u_rows = (warp & 3) < 2;  // TMEM lanes 0-63 (U) or 64-127 (O) of this warp
    const int drow = (warp & 3) * 32 + (tid & 31) - (u_rows ? 0 : 64);
    // D alternates between two accumulators, so a chunk's output rows are written out while
    // the next chunk's first MMAs run.
    auto d_col = [](int c) { return (c & 1) ? kColWO : kColU; };
    // O rows (TMEM lanes 64-127 of D) -> out rows [tc, tc + n) of head h
    auto o_store = [&](int c, int64_t tc, int n) {
      float v[64];
      tmem_ld64(x.tm + x.lane_base + d_col(c) + x.wh * 64, v);
      if (drow < n) {
        const size_t o0 = ((size_t)(tc + drow) * H + h) * kD + x.wh * 64;
        __nv_bfloat16* dst = out + o0;
        const __nv_bfloat16* og = static_cast<const __nv_bfloat16*>(a.og);
#pragma unroll
        for (int j = 0; j < 64; j += 8) {
          if (og) gate8(v + j, og + o0 + j);
          __align__(16) __nv_bfloat162 hv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) hv[i] = __floats2bfloat162_rn(v[j + 2 * i], v[j + 2 * i + 1]);
          *reinterpret_cast<uint4*>(dst + j) = *reinterpret_cast<const uint4*>(hv);
        }
      }
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
      {  // the chunk's operands (every thread reads gamma) and V tile
        if (loader && issued == c) {
          bad |= load_chunk(c) != 1;
          issued = c + 1;
        }
        bad |= !mbar_wait(full + s, ph_full[s], kWaitNs);
        bad |= !mbar_wait(bar_v, ph_v, kWaitNs);
        ph_full[s] ^= 1u;
        ph_v ^= 1u;
        __syncwarp();  // lanes leave their polling loops (and the loader its poll) at different times
        if (n < kC) {  // the last chunk: every thread zeroes part of the V tail
          zero_v_tail<DV>(x, sm + L::VIN, n);
          __syncthreads();
        }
        fence_after_sync();
        landed = c + 1;
      }
      // ring slot c mod R may be rewritten; chunk c + 1 goes to the local slot chunk c - 1 used
      uint32_t next_ready = 0;
      if (loader) {
        st_relaxed_gpu(q_loaded + p, (uint32_t)(c + 1));
        if (c + 1 < nch) next_ready = ld_acquire_gpu(q_ready + p * kR + ((c + 1) % kR));
      }
      // the loader lane rejoins its warp before the warp-collective TMEM instructions below
      // (tcgen05.ld / st and bar.sync are .aligned: the whole warp must execute them together)
      __syncwarp();
      // D = [T'; Z] V + [-W; Q~] S; meanwhile the state master is faded and the previous
      // chunk's output rows are stored
      if (warp == 0) {
        mma_run<kC>(x.tm + d_col(c), opTZ, opV, id_d, false);
        mma_run<kD>(x.tm + d_col(c), opWQ, opS, id_d, true);
        mma_commit_elect(x.bar_mma);
      }
      gamma_fade<DH>(x, reinterpret_cast<const float*>(sm + slot + kSlotGam));
      if (c > 0 && !u_rows) o_store(c - 1, tc - kC, kC);
      if (loader && c + 1 < nch && next_ready >= (uint32_t)(c + 2)) {
        issue_load(c + 1);
        issued = c + 2;
      }
      bad |= !mbar_wait(x.bar_mma, x.ph_mma, kWaitNs);
      x.ph_mma ^= 1u;
      fence_after_sync();
      if (loader && issued == c + 1 && c + 1 < nch &&  // a second look (warp 2 is idle here)
          ld_acquire_gpu(q_ready + p * kR + ((c + 1) % kR)) >= (uint32_t)(c + 2)) {
        issue_load(c + 1);
        issued = c + 2;
      }
      __syncwarp();
      if (u_rows) {  // U rows -> bf16 [tok][DV] tile (MN-major B operand)
        float v[64];
        tmem_ld64(x.tm + x.lane_base + d_col(c) + x.wh * 64, v);
#pragma unroll
        for (int j = 0; j < 64; j += 8) st_chunk8(sm + L::UU, 8192, drow, x.wh * 64 + j, v + j);
        fence_async_smem();
      }
      cta_sync_tc();  // U is written and every warp's fade of the state master is complete
      // S += K^^T U (on the chain's critical path), then O += M U
      if (warp == 0) {
        mma_run<kC>(x.tm + kColS, opKH, opU, id_s, true);
        mma_commit_elect(x.bar_mma);
        mma_run<kC>(x.tm + d_col(c), opZM, opU, id_d, true);
        mma_commit_elect(bar_o);
      }
      // V is consumed, and every thread has passed its wait for this chunk's tile: requested
      // only now, the next tile cannot complete the V barrier's next phase while a thread still
      // polls this one (a parity wait that slept through two phases would sleep on)
      if (tid == 32 && c + 1 < nch) issue_v(tc + kC);
      bad |= !mbar_wait(x.bar_mma, x.ph_mma, kWaitNs);
      x.ph_mma ^= 1u;
      __syncwarp();
      fence_after_sync();
      s_epilogue<DH>(x, sm + L::SS);
      // the local slot is free for chunk c + 2 once O's MMA is complete (gamma was read before
      // a barrier)
      if (tid == 0) bad |= !mbar_wait(bar_o, ph_o, kWaitNs);
      __syncwarp();  // warp 0 reconverges before the aligned CTA barrier below
      ph_o ^= 1u;
      fence_before_sync();
      if (__syncthreads_or(bad)) { failed = true; break; }
      fence_after_sync();
    }
    if (!failed && nch > 0 && !u_rows) {
      const int64_t tl = t0 + (int64_t)(nch - 1) * kC;
      o_store(nch - 1, tl, (int)(t1 - tl));
    }
    if (failed) {
      if (tid == 0) report(a, GDR_DEVCHECK_TIMEOUT);
      if (loader && issued > landed) {  // a ring load still in flight into shared memory
        const int cc = issued - 1;
        mbar_wait(full + (cc & 1), ph_full[cc & 1], kWaitNs);
      }
      mbar_wait(bar_v, ph_v, kWaitNs);
    } else if (a.S_final) {
      s_final<DH>(x, a.S_final + sidx + (size_t)x.lrow * kD);
    }
    cta_sync_tc();
    if (warp == 0) tmem_dealloc(x.tm, kTmemCols);
  } else {
    // ===================================================================== helper CTA
    using L = QHelperSmem;
    float* sBeta = reinterpret_cast<float*>(sm + L::BETA);
    float* sAlpha = reinterpret_cast<float*>(sm + L::ALPHA);
    int* sItem = reinterpret_cast<int*>(sm + L::ITEM);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* bar_qk = bars + 0;
    uint64_t* bar_a = bars + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3);
    if (warp == 0) tmem_alloc(tslot, kTmemCols);
    if (tid == 0) {
      for (int i = 0; i < 3; ++i) mbar_init(bars + i, 1);
      fence_mbar_init();
      prefetch_tmap(&maps.q);
      prefetch_tmap(&maps.k);
      if (kAlphaTile) prefetch_tmap(&maps.alpha);
    }
    cta_sync_tc();
    TcCtx x = make_ctx(sm, *tslot, bars + 2);
    x.prologue = a.prologue;
    zero_upper_tp(sm + L::TT, tid);
    uint32_t ph_qk = 0, ph_a = 0;
    bool failed = false;
    // the chains' (first token, tokens, head), once: a work item then needs no global reads
    struct ChainInfo {
      int64_t t0;
      int32_t ntok, h;
    };
    ChainInfo* sChains = reinterpret_cast<ChainInfo*>(sm + L::CHAINS);
    if (tid < P) {
      int hh, sq;
      int64_t u0 = 0, u1 = 0;
      const bool okc = chain_range(a, tid, hh, sq, u0, u1);
      sChains[tid] = ChainInfo{u0, okc ? (int32_t)(u1 - u0) : 0, hh};
    }
    __syncthreads();
    // chunks of the longest sequence (the first in the visiting order): items past it are void
    const int maxn = (sChains[0].ntok + kC - 1) / kC;
    // tid 0 takes the next item with a chunk to do and sends its TMA loads; every thread gets
    // (chain, chunk, head, first token, tokens) -- chain -1 when the queue is exhausted.  The
    // counter's next value is fetched one take ahead, so the atomic's latency stays hidden.
    struct Item {
      int p, c, h, n;
      int64_t tc;
    };
    uint32_t ahead = 0;
    if (tid == 0) ahead = atomicAdd(q_next, 1u);
    int takes = 0;
    auto take = [&]() -> Item {
      int* slot = sItem + 2 * (takes & 1);  // alternate buffers: no second barrier needed
      ++takes;
      if (tid == 0) {
        int p = -1, c = 0;
        for (;;) {
          const uint32_t i = ahead;
          c = (int)(i / (uint32_t)P);
          if (c >= maxn) { p = -1; break; }
          ahead = atomicAdd(q_next, 1u);
          p = (int)(i % (uint32_t)P);
          if (c * kC < sChains[p].ntok) break;
        }
        slot[0] = p;
        slot[1] = c;
      }
      __syncthreads();
      Item it{slot[0], slot[1], 0, 0, 0};
      if (it.p >= 0) {
        const ChainInfo ci = sChains[it.p];
        it.h = ci.h;
        it.tc = ci.t0 + (int64_t)it.c * kC;
        it.n = ci.ntok - it.c * kC < kC ? ci.ntok - it.c * kC : kC;
        if (tid == 0) {
          mbar_expect_tx(bar_qk, 2 * 16384);
          tma_load_3d(sm + L::QIN, &maps.q, 0, it.h, (int)it.tc, bar_qk);
          tma_load_3d(sm + L::KIN, &maps.k, 0, it.h, (int)it.tc, bar_qk);
          if (kAlphaTile) {
            mbar_expect_tx(bar_a, 32768);
            tma_load_3d(sm + L::AIN, &maps.alpha, 0, it.h, (int)it.tc, bar_a);
          }
        }
      }
      return it;
    };
    auto load_scalars = [&](const Item& it, float& b, float& al) {
      b = 0.f;
      al = 1.f;
      if (it.p >= 0 && tid < it.n) {
        const size_t o = (size_t)(it.tc + tid) * H + it.h;
        b = a.beta[o];
        if (!CHANNEL) al = a.alpha[o];
      }
    };
    Item cur = take();
    float nb_beta, nb_alpha;
    load_scalars(cur, nb_beta, nb_alpha);
    // The chunk handed over last: every thread fences its ring stores at the top of the next item,
    // and the flag is set after the barrier that follows -- before the item waits for a ring slot.
    int pub_p = -1, pub_c = 0;
    auto publish = [&]() {
      if (tid == 0 && pub_p >= 0)
        st_release_gpu(q_ready + pub_p * kR + (pub_c % kR), (uint32_t)(pub_c + 1));
      pub_p = -1;
    };
#pragma unroll 1
    while (cur.p >= 0) {
      if (tid < kC) {  // (the layer prologue maps the live tokens' raw gates here, not at the load)
        const bool pro = a.prologue && tid < cur.n;
        sBeta[tid] = pro ? sigmoid_ftz(nb_beta) : nb_beta;
        sAlpha[tid] = pro && !CHANNEL ? sigmoid_ftz(nb_alpha) : nb_alpha;
      }
      // hand the previous chunk over before waiting on any chain (a chain may need exactly that
      // chunk to move on): its ring stores are visible before its flag is set
      __threadfence();
      __syncthreads();
      publish();
      // ring slot c mod R must be free: the chain CTA has loaded chunk c - R from it
      bool ok = true;
      if (tid == 0 && cur.c >= kR) ok = poll_ge(q_loaded + cur.p, (uint32_t)(cur.c - kR + 1));
      __syncwarp();  // lane 0 rejoins its warp before the aligned CTA barrier
      if (__syncthreads_or(!ok)) { failed = true; break; }
      x.gslot = a.ring + ((size_t)cur.p * kR + (size_t)(cur.c % kR)) * kSlotBytes;
      if (!wait_bar(bar_qk, ph_qk)) { failed = true; break; }
      if (kAlphaTile && !wait_bar(bar_a, ph_a)) { failed = true; break; }

      const bool safe = gate_stage<L, CHANNEL>(x, cur.n);
      fence_async_smem();
      cta_sync_tc();
      Item nxt{-1, 0, 0, 0, 0};
      if (safe) nxt = take();  // q, k and alpha tiles are consumed: fetch the next item's
      if (!gram_stage<L, CHANNEL>(x, cur.n, safe)) { failed = true; break; }
      if (!safe) nxt = take();
      load_scalars(nxt, nb_beta, nb_alpha);
      solve_stage<L>(x);
      if (!w_stage<L>(x, false, Opnd{0, 0, false}, 0)) { failed = true; break; }
      w_epilogue<L, true>(x);  // -W
      pub_p = cur.p;
      pub_c = cur.c;
      cur = nxt;
    }
    if (failed) {
      if (tid == 0) report(a, GDR_DEVCHECK_TIMEOUT);
      mbar_wait(bar_qk, ph_qk, kWaitNs);
      if (kAlphaTile) mbar_wait(bar_a, ph_a, kWaitNs);
    } else {  // hand over the last chunk
      __threadfence();
      __syncthreads();
      publish();
    }
    cta_sync_tc();
    if (warp == 0) tmem_dealloc(x.tm, kTmemCols);
  }
}

template <bool CHANNEL>
cudaError_t launch_typed(const PrefillArgs& a, const TcMaps& maps, int P, int G,
                         cudaStream_t s) {
  auto kern = prefill_queue_kernel<CHANNEL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kQueueSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kQueueSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps, a, P);
}

// CTAs of this kernel that are resident at once on the current device (0 if unknown)
int max_resident() {
  static int cache[64] = {0};
  static bool known[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (known[dev]) return cache[dev];
  int per_sm = 0, sms = 0;
  auto kern = prefill_queue_kernel<true>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kQueueSmem) == cudaSuccess &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, kQueueSmem) ==
          cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) {
    cache[dev] = per_sm * sms;
  }
  cudaGetLastError();
  known[dev] = true;
  return cache[dev];
}

}  // namespace

// CTAs of the work-queue launch for this shape (0: use another kernel).  It needs the ring in
// the workspace and at least one helper CTA per two chains.
int queue_grid_for(const gdr_shape& sh, const PrefillArgs& a) {
  if (!a.ring || !a.ring_flags) return 0;
  const long pairs = (long)sh.n_seqs * sh.H;
  const int g = max_resident();
  if (pairs < 1 || pairs > WorkspaceLayout::kRingMaxPairs || g < 3 * pairs / 2 + 1) return 0;
  return g;
}

cudaError_t launch_prefill_queue(const gdr_shape& sh, const PrefillArgs& a, const TcMaps& maps,
                                 int G, cudaStream_t s) {
  const int P = (int)((long)sh.n_seqs * sh.H);
  cudaError_t e = cudaMemsetAsync(a.ring_flags, 0, WorkspaceLayout::flag_bytes(P), s);
  if (e != cudaSuccess) return e;
  if (sh.gate == GDR_GATE_CHANNEL) return launch_typed<true>(a, maps, P, G, s);
  return launch_typed<false>(a, maps, P, G, s);
}

}  // namespace tc
}  // namespace gdr
