// attn_fwd.cu -- causal context-parallel attention forward on sm_103a.
//
// One CTA computes a block of up to 256 query rows (two 128-row tiles, Q0
// and Q1, of the same head and the same contiguous-position chunk) of one
// attention rank.  It visits the KV chunks of the ring -- at step s the
// chunk of ring rank (r - s) mod R ([MTX] nougat.kr "MaxText long-context
// training and KV parallelism", section "Split heads or rotate KV": P2P
// keeps token sharding and computes a partial with each visiting KV chunk),
// in position order when one launch covers every step (for_each_kv_tile) --
// and, per 128-key tile visible from either query tile:
//
//   S_t = Q_t K^T          tcgen05.mma, Q and K in shared memory (TMA,
//                          128-byte swizzle), fp32 accumulator in TMEM
//   mask, online softmax   one thread per query row (TMEM lane = row);
//                          P_t = exp2(...) written back over S_t in TMEM
//                          as packed bf16
//   O_t += P_t V           tcgen05.mma with A read from TMEM, V in shared
//                          memory
//
// The two query tiles ping-pong: while one softmax warpgroup works on S_0,
// the tensor core runs the other tile's PV and QK^T, so neither waits for
// the other.  Tiles with no visible pair are never visited; tiles wholly
// inside the causal and document window skip the mask.  The merge of the
// ring partials is fused: the online softmax continues across ring steps,
// which is the exact merge evaluated incrementally.  In emit-partials mode
// a CTA covers one ring step and writes that step's normalised partial
// (O, LSE) in fp32 for the separate merge kernel.
//
// Warp roles (320 threads): warp 0 = TMA producer; warp 1 = TMEM allocator
// and MMA issuer; warps 2..5 = softmax / correction / epilogue of Q0 and
// warps 6..9 of Q1 (thread t of warp w owns row 32*(w%4)+t, the TMEM lanes
// that warp may access).
//
// K and V tiles stream through one ring of five shared-memory slots in load
// order K_0, V_0, K_1, V_1, ... (load n of the sequence uses slot n mod 5), so
// a tile's loads are issued about two tiles ahead of their use: a TMA load
// from L2 takes a few microseconds under load, more than one tile's work.
//
// The running max is only raised when it grows by more than 2^8 (log2
// units), so O is rescaled in TMEM rarely; the final normalisation uses the
// same max, which keeps the result exact.  Issue order on the tensor core
// per key tile j: QK0_j, PV1_{j-1}, QK1_j, PV0_j.  PV_t of one tile is
// always issued before QK_t of the next, and tcgen05.mma ops from one thread
// execute in issue order, so the next S_t never overwrites a P_t still
// being read.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>

#define CP_TU_ID ::cpattn::kTuAttnFwd
#include "debug.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace cpattn {
namespace {

constexpr int BM = 128;                      // query rows per tile
constexpr int BN = 128;                      // keys per tile
constexpr uint32_t HALF_BYTES = 128 * 128;   // one 64-column (128-byte) swizzled half of a 128-row tile
constexpr float kRescaleThreshold = 8.0f;    // log2 units
constexpr int kThreads = 320;

constexpr int kSlots = 5;                    // K/V ring slots (K of key tile j is load 2j, V load 2j+1)
constexpr int kTileBars = 3;                 // key tiles in flight at most: 5 slots, 2 per tile

enum Bar {
  BAR_Q = 0,
  BAR_T_FULL = 1,                          // +key tile % kTileBars: its K and V landed
  BAR_KV_EMPTY = 1 + kTileBars,            // +slot
  BAR_S_FULL = 1 + kTileBars + kSlots,     // +query tile
  BAR_P_FULL = 3 + kTileBars + kSlots,     // +query tile
  BAR_DRAIN = 5 + kTileBars + kSlots,      // every MMA of the CTA completed
  BAR_P_HALF = 6 + kTileBars + kSlots,     // +query tile: P of keys 0-63 written
  BAR_O0 = 8 + kTileBars + kSlots,         // every MMA of query tile 0 completed
  NUM_BARS = 9 + kTileBars + kSlots
};

template <int D>
struct FwdSmem {
  static constexpr uint32_t kQ = BM * D * 2;
  static constexpr uint32_t kKV = BN * D * 2;
  static constexpr uint32_t offQ = 0;                 // two query tiles
  static constexpr uint32_t offKV = offQ + 2 * kQ;    // kSlots K/V slots
  static constexpr uint32_t offBar = offKV + kSlots * kKV;
  static constexpr uint32_t offMisc = offBar + NUM_BARS * 8;
  static constexpr uint32_t kUsed = offMisc + 16;
  // 1 KB alignment slack; D=64 is padded so that one CTA (and one 512-column
  // TMEM allocation) is resident per SM.
  static constexpr uint32_t kBytes = (kUsed + 1024 < 120 * 1024) ? 120 * 1024 : kUsed + 1024;
};

// Visit every 128-key tile that may hold a visible key for query positions
// <= qpos_last whose documents start at or after lo_min.
// f(kv_row, kpos0, klen): first row of the tile in the [R*U*T] row space,
// the tile's first position, and its number of valid keys.
//
// One ring step (emit-partials, rank-local): the chunk of rank (r - s) mod R.
// All ring steps in one launch: the visiting chunks are walked in position
// order rather than ring order.  Every chunk is resident, so the order is
// free; the merge is exact, so it changes only the fp32 rounding order.  In
// position order all the long query blocks running at once sweep the same
// key tiles together and share them in L2; in ring order each starts from
// its own rank's chunk, and a tile's many readers come too far apart in time
// for L2 to keep it (at 256K tokens, 180x the compulsory DRAM reads).
template <typename F>
__device__ __forceinline__ void for_each_kv_tile(const AttnGeom& g, int r, int u, int s_begin, int s_end,
                                                 int lo_min, int qpos_last, F&& f) {
  if (g.kv_global) {
    // All-gathered K/V: row = position; one pass in position order.
    const int t1 = qpos_last / BN;
    for (int t = lo_min / BN; t <= t1; ++t) f(t * BN, t * BN, min(BN, g.L - t * BN));
    return;
  }
  if (s_begin == 0 && s_end == g.R && g.R > 1) {
    const int c = g.chunk;
    const int j1 = qpos_last / c;
    for (int j = lo_min / c; j <= j1; ++j) {
      int src, cslot0;
      chunk_owner(g, j, src, cslot0);
      const int cpos0 = j * c;
      const int lo = max(cpos0, lo_min);
      const int hi = min(cpos0 + c - 1, qpos_last);
      const int t1 = (hi - cpos0) / BN;
      for (int t = (lo - cpos0) / BN; t <= t1; ++t)
        f((src * g.U + u) * g.T + cslot0 + t * BN, cpos0 + t * BN, min(BN, c - t * BN));
    }
    return;
  }
  const int nchunks = g.nchunks;
  for (int s = s_begin; s < s_end; ++s) {
    const int src = (r - s + g.R) % g.R;
    const int a_src = src * g.U + u;
    for (int ch = 0; ch < nchunks; ++ch) {
      const int cslot0 = ch * g.chunk;
      const int cpos0 = slot_pos(g, src, cslot0);
      const int lo = max(cpos0, lo_min);
      const int hi = min(cpos0 + g.chunk - 1, qpos_last);
      if (lo > hi) continue;
      const int t1 = (hi - cpos0) / BN;
      for (int t = (lo - cpos0) / BN; t <= t1; ++t)
        f(a_src * g.T + cslot0 + t * BN, cpos0 + t * BN, min(BN, g.chunk - t * BN));
    }
  }
}

// One query tile's window: positions [qp0, qp_last], document starts in
// [lo_min, lo_max]; len == 0 marks an absent tile.
struct QWin {
  int qp0, qp_last, lo_min, lo_max, len;
  __device__ __forceinline__ bool sees(int kpos0, int klen) const {
    return len > 0 && kpos0 <= qp_last && kpos0 + klen - 1 >= lo_min;
  }
  __device__ __forceinline__ bool full(int kpos0, int klen) const {
    return klen == BN && kpos0 + BN - 1 <= qp0 && lo_max <= kpos0;
  }
};

// Window of query tile t (0 or 1) of work item `it` of ring rank r; the
// block's positions are contiguous.
__device__ __forceinline__ QWin make_qwin(const AttnGeom& g, const WorkItem& it, int r, int t, int32_t* status) {
  QWin w;
  w.len = max(0, min(BM, it.len - t * BM));
  w.qp0 = slot_pos(g, r, it.q0) + t * BM;
  w.qp_last = w.qp0 + w.len - 1;
  if (w.len > 0 && !CP_IN_BOUNDS(w.qp0 >= 0 && w.qp_last < g.L, status)) w.len = 0;
  w.lo_min = (w.len > 0 && g.doc_start) ? g.doc_start[w.qp0] : 0;
  w.lo_max = (w.len > 0 && g.doc_start) ? g.doc_start[w.qp_last] : 0;
  return w;
}

// Class of a key tile for one query tile: 0 = not seen (no MMA, no softmax
// pass), 1 = seen through the mask, 2 = wholly visible (the mask is skipped).
__device__ __forceinline__ int tile_class(const QWin& w, int kpos0, int klen) {
  return w.sees(kpos0, klen) ? (w.full(kpos0, klen) ? 2 : 1) : 0;
}

__device__ __forceinline__ bool warp_all(bool x) { return __all_sync(0xffffffffu, x); }

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const FwdArgs args) {
  using SM = FwdSmem<D>;
  constexpr int NH = D / 64;  // 64-column halves of a head row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sQ = s_base + SM::offQ, sKV = s_base + SM::offKV;
  // Load n of the K/V sequence (K of tile j is load 2j, V of tile j is 2j+1).
  auto slot_of = [](int n) { return n % kSlots; };
  auto parity_of = [](int n) { return static_cast<uint32_t>((n / kSlots) & 1); };
  auto bar = [&](int i) { return s_base + SM::offBar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::offMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM::offMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttnGeom& g = args.g;
  int32_t* status = args.status;
  int item_idx, h;
  if (args.stream_major) {
    const int per_stream = args.n_items_u * g.G;
    const int sidx = blockIdx.x / per_stream;  // K/V stream (u, KV head)
    const int rem = blockIdx.x - sidx * per_stream;
    const int su = sidx / g.Hkv_loc;
    item_idx = su * args.n_items_u + rem / g.G;
    h = (sidx - su * g.Hkv_loc) * g.G + rem % g.G;
  } else {
    item_idx = blockIdx.x / g.Hq_loc;
    h = blockIdx.x % g.Hq_loc;
  }
  if (!CP_IN_BOUNDS(item_idx < args.n_items, status)) return;
  WorkItem it = args.items[item_idx];
  const bool rank_local = args.rank_local != 0;  // one ring step; Q and K/V are local buffers
  if (rank_local) it.step = args.step;
  // A work item lies inside its attention rank's slots.
  if (!CP_IN_BOUNDS(it.a >= 0 && it.a < g.R * g.U && it.q0 >= 0 && it.len > 0 && it.len <= 2 * BM &&
                        it.q0 + it.len <= g.T && it.step < g.R, status))
    return;
  const int a = it.a, r = a / g.U, u = a % g.U;
  const int s_begin = it.step < 0 ? 0 : it.step;
  const int s_end = it.step < 0 ? g.R : it.step + 1;
  // Rank-local mode: Q row a*T + t is row t of the rank's buffer, and K/V
  // row a_src*T + t of the visiting chunk (a_src = ((r - step) mod R)*U + u)
  // is row t of the chunk buffer.
  // Sequence-sharded tensors (seq_io): ring rank r's slots are rows r*T ..
  // r*T + T-1 and member u's heads a column range of the full head count.
  const bool seq_io = args.seq_io != 0;
  const int q_row0 = rank_local ? 0 : (seq_io ? r : a) * g.T;
  const int kv_sub = rank_local ? (((r - s_begin + g.R) % g.R) * g.U + u) * g.T : 0;
  [[maybe_unused]] const int q_rows = rank_local ? g.T : (seq_io ? g.R : g.R * g.U) * g.T;  // rows of Q
  [[maybe_unused]] const int kv_rows =
      rank_local ? g.T : g.kv_global ? g.L : (seq_io ? g.R : g.R * g.U) * g.T;             // rows of K/V
  // First column of this head in Q and O, and of its KV head in K and V.
  auto qcol0 = [&]() { return (seq_io ? u * g.Hq_loc + h : h) * D; };
  auto kvcol0 = [&]() { return (seq_io ? u * g.Hkv_loc + h / g.G : h / g.G) * D; };
  const int hkv = h / g.G;

  // The two query tiles' windows; the block walks the keys in [lo_min of
  // tile 0, last position of the block].
  const QWin win0 = make_qwin(g, it, r, 0, status), win1 = make_qwin(g, it, r, 1, status);
  const int blk_lo_min = win0.lo_min;
  const int blk_qp_last = win0.qp0 + it.len - 1;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    mbar_init(bar(BAR_Q), 1);
    for (int i = 0; i < kTileBars; ++i) mbar_init(bar(BAR_T_FULL + i), 1);
    for (int i = 0; i < kSlots; ++i) mbar_init(bar(BAR_KV_EMPTY + i), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(BAR_S_FULL + i), 1);
      mbar_init(bar(BAR_P_FULL + i), 4);
      mbar_init(bar(BAR_P_HALF + i), 4);
    }
    mbar_init(bar(BAR_DRAIN), 1);
    mbar_init(bar(BAR_O0), 1);
    *abort_flag = 0;
    fence_mbar_init();
    // The query tiles' loads go out before the TMEM allocation and the
    // block-wide barrier, whose latency they then overlap.
    mbar_arrive_expect_tx(bar(BAR_Q), 2 * SM::kQ);
    const int qrow = q_row0 + it.q0;
    for (int t = 0; t < 2; ++t) {
      (void)CP_IN_BOUNDS(t * BM >= it.len || (qrow + t * BM >= 0 && qrow + t * BM < q_rows), status);
      for (int hh = 0; hh < NH; ++hh)
        tma_load_2d(sQ + t * SM::kQ + hh * HALF_BYTES, &tm_q, bar(BAR_Q), qcol0() + hh * 64, qrow + t * BM);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // S_t = tmem + 128 t (128 fp32 columns; P_t as packed bf16 in its first
  // 64) and O_t = tmem + 256 + D t.

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // Key tile nt: K into slot of load 2nt, V into slot of load 2nt+1, both
      // completing one tile barrier, so the issuer waits once per tile.  The
      // two slots were last used by V of tile nt-3 and K of tile nt-2, so the
      // tile barrier nt % 3 was last used by tile nt-3, whose wait is done.
      int n = 0;   // loads issued
      int nt = 0;  // key tiles issued
      for_each_kv_tile(g, r, u, s_begin, s_end, blk_lo_min, blk_qp_last, [&](int kv_row_all, int, int) {
        if (*abort_flag) return;
        // kv_row_all = (src*U + u)*T + slot in the head-sharded row space.
        const int kv_row = seq_io ? (kv_row_all / (g.T * g.U)) * g.T + kv_row_all % g.T : kv_row_all - kv_sub;
        const int slk = slot_of(n), slv = slot_of(n + 1);
        if (!mbar_wait(bar(BAR_KV_EMPTY + slk), parity_of(n) ^ 1, abort_flag, status)) return;
        if (!mbar_wait(bar(BAR_KV_EMPTY + slv), parity_of(n + 1) ^ 1, abort_flag, status)) return;
        const uint32_t tb = bar(BAR_T_FULL + nt % kTileBars);
        mbar_arrive_expect_tx(tb, 2 * SM::kKV);
        (void)CP_IN_BOUNDS(kv_row >= 0 && kv_row < kv_rows && hkv < g.Hkv_loc, status);
        for (int hh = 0; hh < NH; ++hh)
          tma_load_2d(sKV + slk * SM::kKV + hh * HALF_BYTES, &tm_k, tb, kvcol0() + hh * 64, kv_row);
        for (int hh = 0; hh < NH; ++hh)
          tma_load_2d(sKV + slv * SM::kKV + hh * HALF_BYTES, &tm_v, tb, kvcol0() + hh * 64, kv_row);
        n += 2;
        ++nt;
      });
      if (*abort_flag) {
        // Let every copy still in flight land before the CTA exits.
        mbar_wait(bar(BAR_Q), 0, nullptr, status);
        for (int i = max(0, nt - kTileBars); i < nt; ++i)
          mbar_wait(bar(BAR_T_FULL + i % kTileBars), (i / kTileBars) & 1, nullptr, status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop (warp-uniform operands); one
    // elected lane executes each tcgen05 instruction.
    {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, 1);
      int npv[2] = {0, 0};      // PVs issued per query tile
      int pend_sl = -1;         // V slot of a PV1 still to issue
      // Descriptors are built once; each MMA only adds a compile-time offset
      // to the start-address field (addresses stay below 256 KB, so the
      // 14-bit field never carries).  The issuing warp shares its scheduler
      // with softmax warps, so every instruction it saves shortens the
      // critical path of the tensor core.
      const uint64_t dq0 = smem_desc_sw128(sQ, 16, 1024);
      const uint64_t dq1 = smem_desc_sw128(sQ + SM::kQ, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(sKV, 16, 1024);          // slot 0 read as K (K-major)
      const uint64_t dv0 = smem_desc_sw128(sKV, HALF_BYTES, 1024);  // slot 0 read as V (MN-major)
      constexpr uint64_t kSlotStep = SM::kKV >> 4;
      auto issue_qk = [&](int t, int slot) {
        const uint64_t a0 = t ? dq1 : dq0;
        const uint64_t b0 = dk0 + static_cast<uint64_t>(slot) * kSlotStep;
        if constexpr (D == 128)
          mma_bf16_ss_k128_warp<HALF_BYTES>(tmem + 128 * t, a0, b0, idesc_qk, 0u);
        else
          mma_bf16_ss_k64_warp(tmem + 128 * t, a0, b0, idesc_qk, 0u);
        mma_commit_warp(bar(BAR_S_FULL + t));
      };
      // O_t += P_t V: A = P_t in TMEM (8 columns per 16 keys), B = V [keys x d]
      // read as N=d x K=keys, MN-major (16 keys = 16 rows of 128 bytes; the two
      // 64-column halves of d are HALF_BYTES apart), from V slot `sl`.  The
      // softmax signals P of keys 0-63 before it computes keys 64-127, so the
      // first four MMAs start while it finishes.  No per-PV completion
      // signal: the softmax learns that O_t is stable from the next S_t
      // commit (issued after this PV) or, at the end, from the drain commit.
      auto issue_pv = [&](int t, int sl, bool release_v) -> bool {
        if (!warp_all(mbar_wait(bar(BAR_P_HALF + t), npv[t] & 1, abort_flag, status))) return false;
        tc_fence_after();
        const uint64_t b0 = dv0 + static_cast<uint64_t>(sl) * kSlotStep;
        mma_bf16_ts_k64_warp(tmem + 256 + D * t, tmem + 128 * t, b0, idesc_pv, npv[t] > 0 ? 1u : 0u);
        if (!warp_all(mbar_wait(bar(BAR_P_FULL + t), npv[t] & 1, abort_flag, status))) return false;
        tc_fence_after();
        mma_bf16_ts_k64_warp(tmem + 256 + D * t, tmem + 128 * t + 32, b0 + 512, idesc_pv, 1u);
        if (release_v) mma_commit_warp(bar(BAR_KV_EMPTY + sl));
        ++npv[t];
        return true;
      };
      int j = 0;                // key tiles walked
      int ring_slot = 0;        // slot of the next K load
      bool ok = warp_all(mbar_wait(bar(BAR_Q), 0, abort_flag, status));
      if (ok) {
        // No abort-flag read per tile: every wait below leaves on the flag.
        for_each_kv_tile(g, r, u, s_begin, s_end, blk_lo_min, blk_qp_last, [&](int, int kpos0, int klen) {
          if (!ok) return;
          const bool v0 = win0.sees(kpos0, klen), v1 = win1.sees(kpos0, klen);
          const int kslot = ring_slot, vslot = ring_slot + 1 == kSlots ? 0 : ring_slot + 1;
          ring_slot = vslot + 1 == kSlots ? 0 : vslot + 1;
          // One wait per key tile: its K and V complete the same barrier.
          if (!(ok = warp_all(mbar_wait(bar(BAR_T_FULL + j % kTileBars), (j / kTileBars) & 1, abort_flag, status))))
            return;
          tc_fence_after();
          if (v0) issue_qk(0, kslot);
          if (pend_sl >= 0) {
            if (!(ok = issue_pv(1, pend_sl, true))) return;
            pend_sl = -1;
          }
          if (v1) issue_qk(1, kslot);
          mma_commit_warp(bar(BAR_KV_EMPTY + kslot));
          if (v0 && !(ok = issue_pv(0, vslot, !v1))) return;
          if (v1) pend_sl = vslot;
          ++j;
        });
      }
      // Query tile 0 has no MMA left: its epilogue overlaps the last softmax
      // and PV of tile 1.
      mma_commit_warp(bar(BAR_O0));
      if (ok && pend_sl >= 0 && !warp_all(*abort_flag != 0)) issue_pv(1, pend_sl, true);
      // Every MMA issued so far completes before TMEM and shared memory are released.
      mma_commit_warp(bar(BAR_DRAIN));
      mbar_wait(bar(BAR_DRAIN), 0, nullptr, status);
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int t = (warp - 2) >> 2;  // query tile of this warpgroup
    const QWin w = t ? win1 : win0;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tSt = tmem + 128 * t + lane_off, tOt = tmem + 256 + D * t + lane_off;
    const bool row_valid = row < w.len;
    const int my_pos = row_valid ? w.qp0 + row : -1;
    const int my_lo = (row_valid && g.doc_start) ? g.doc_start[my_pos] : 0;
    const float sl2 = g.scale * 1.4426950408889634f;
    float m = -INFINITY, l = 0.f;
    int k = 0;
    bool ok = true;
    for_each_kv_tile(g, r, u, s_begin, s_end, blk_lo_min, blk_qp_last, [&](int, int kpos0, int klen) {
      if (!ok || !w.sees(kpos0, klen)) return;
      ok = warp_all(mbar_wait(bar(BAR_S_FULL + t), k & 1, abort_flag, status));
      if (!ok) return;
      tc_fence_after();
      const bool full = w.full(kpos0, klen);
      uint32_t sr[BN];
      float* x = reinterpret_cast<float*>(sr);
      auto col32 = [&](int c) -> uint32_t(&)[32] { return *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]); };
      // P = exp2(S*scale*log2e - mb) of 32 columns -> 16 packed bf16 pairs,
      // row sum into rs2.  Pairs of columns go through packed fp32x2 fma/add
      // (half the issue slots of scalar code); exp2 stays per element on the
      // MUFU pipe.
      const f32x2 sl2x2 = make_f32x2(sl2, sl2);
      auto exp32 = [&](int c, float mb, f32x2 (&rs2)[4], uint32_t (&pk)[16]) {
        const f32x2 nmbx2 = make_f32x2(-mb, -mb);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float a0, a1;
          split_f32x2(fma_f32x2(make_f32x2(x[c * 32 + e], x[c * 32 + e + 1]), sl2x2, nmbx2), a0, a1);
          const float p0 = ex2_approx(a0);
          const float p1 = ex2_approx(a1);
          rs2[(e >> 1) & 3] = add_f32x2(rs2[(e >> 1) & 3], make_f32x2(p0, p1));
          pk[e >> 1] = pack_bf16x2(p0, p1);
        }
      };
      auto sum4 = [](const f32x2 (&rs2)[4]) {
        float lo[4], hi[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) split_f32x2(rs2[i], lo[i], hi[i]);
        return ((lo[0] + hi[0]) + (lo[1] + hi[1])) + ((lo[2] + hi[2]) + (lo[3] + hi[3]));
      };
      auto signal = [&](int b) {
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(b + t));
      };
      // Wholly visible tile, running max already set: keys 0-63 are
      // exponentiated against the running max m without first taking their
      // max; their row sum bounds every one of them, and the max of keys
      // 64-127 (computed while those exponentials run) bounds the rest.  If
      // every P stays below 2^16 the tile keeps m, and no max stands between
      // the scores and the first exponential.  Otherwise the warp reloads S
      // and takes the exact path below.  O and l grow by at most 2^16 per
      // key relative to m, far inside fp32 range, and the final
      // normalisation uses the same m, so the result is exact.
      if (full && warp_all(m != -INFINITY)) {
        tmem_ld32(tSt, col32(0));
        tmem_ld32(tSt + 32, col32(1));
        tmem_wait_ld();
        reg_fence(col32(0));
        reg_fence(col32(1));
        tmem_ld32(tSt + 64, col32(2));   // in flight while keys 0-63 are exponentiated
        tmem_ld32(tSt + 96, col32(3));
        f32x2 rs2[4] = {make_f32x2(0.f, 0.f), make_f32x2(0.f, 0.f), make_f32x2(0.f, 0.f), make_f32x2(0.f, 0.f)};
        uint32_t pk0[16], pk1[16];
        exp32(0, m, rs2, pk0);
        exp32(1, m, rs2, pk1);
        tmem_wait_ld();
        reg_fence(col32(2));
        reg_fence(col32(3));
        float m4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) m4[i] = fmaxf(x[64 + i], x[68 + i]);
#pragma unroll
        for (int e = 72; e < BN; e += 8)
#pragma unroll
          for (int i = 0; i < 4; ++i) m4[i] = fmax3(m4[i], x[e + i], x[e + 4 + i]);
        const float mx_hi = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        const float s_lo = sum4(rs2);
        if (warp_all(s_lo < 65536.f && mx_hi * sl2 < m + 16.f)) {
          tmem_st16(tSt, pk0);
          tmem_st16(tSt + 16, pk1);
          signal(BAR_P_HALF);
          f32x2 rh[4] = {make_f32x2(0.f, 0.f), make_f32x2(0.f, 0.f), make_f32x2(0.f, 0.f), make_f32x2(0.f, 0.f)};
          exp32(2, m, rh, pk0);
          tmem_st16(tSt + 32, pk0);
          exp32(3, m, rh, pk1);
          tmem_st16(tSt + 48, pk1);
          signal(BAR_P_FULL);
          l += s_lo + sum4(rh);
          ++k;
          return;
        }
      }
      // Exact path: masked tiles, the first tile of a row, and wholly visible
      // tiles whose scores outgrew the running max.
      const int c_lo = my_lo - kpos0;
      const int c_hi = min(my_pos - kpos0, klen - 1);
      // S row -> registers: four 32-column loads in flight, one wait.
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(tSt + c * 32, col32(c));
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) reg_fence(col32(c));
      if (!full) {
#pragma unroll
        for (int e = 0; e < BN; ++e)
          if (e < c_lo || e > c_hi) x[e] = -INFINITY;
      }
      // Row max: 3-input max in 8 independent chains.
      float m8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) m8[i] = fmaxf(x[i], x[8 + i]);
#pragma unroll
      for (int e = 16; e < BN; e += 16)  // covers x[16 .. 127]
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = fmax3(m8[i], x[e + i], x[e + 8 + i]);
      const float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
      const float m_new = fmaxf(m, mx * sl2);
      float alpha = 1.f;
      if (m_new > m + kRescaleThreshold) {
        alpha = ex2_approx(m - m_new);
        m = m_new;
      }
      const float mb = (m == -INFINITY) ? 0.f : m;
      // P is written packed into the first 64 columns of S (already read
      // into registers).
      f32x2 rs2[4] = {make_f32x2(0.f, 0.f), make_f32x2(0.f, 0.f), make_f32x2(0.f, 0.f), make_f32x2(0.f, 0.f)};
      auto exp_chunk = [&](int c) {
        uint32_t pk[16];
        exp32(c, mb, rs2, pk);
        tmem_st16(tSt + c * 16, pk);
      };
      exp_chunk(0);
      exp_chunk(1);
      // O is stable here: this tile's S_FULL commit came after the previous
      // PV_t; its rescale lands before the first half of this tile's PV.
      if (k > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(tOt + c * 32, ov);
          tmem_wait_ld();
          reg_fence(ov);
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st32(tOt + c * 32, ov);
        }
      }
      signal(BAR_P_HALF);
      exp_chunk(2);
      exp_chunk(3);
      signal(BAR_P_FULL);
      l = l * alpha + sum4(rs2);
      ++k;
    });
    if (ok && k > 0) {
      // Every MMA of this query tile, its last PV_t among them, has completed.
      ok = warp_all(mbar_wait(bar(t ? BAR_DRAIN : BAR_O0), 0, abort_flag, status));
      if (ok) tc_fence_after();
    }
    if (ok) {
      const bool has = l > 0.f;
      const float inv_l = has ? 1.f / l : 0.f;
      const float lse = has ? (m + lg2_approx(l)) * 0.69314718055994531f : -INFINITY;
      const bool partial = args.o_part != nullptr;
      const int q_slot = it.q0 + t * BM + row;
      // This row's O (element offset) and LSE index in the output layout.
      const int Hq_all = g.Hq_loc * g.U;
      const size_t o_row_off =
          seq_io ? (static_cast<size_t>(q_row0 + q_slot) * Hq_all + u * g.Hq_loc + h) * D
                 : (static_cast<size_t>(a * g.T + q_slot) * g.Hq_loc + h) * D;
      const int n_mem = g.T / g.U;  // slots per attention rank (sequence-sharded LSE rows)
      const size_t lse_idx =
          seq_io ? (static_cast<size_t>(r * g.U + q_slot / n_mem) * Hq_all + u * g.Hq_loc + h) * n_mem + q_slot % n_mem
                 : (static_cast<size_t>(a) * g.Hq_loc + h) * g.T + q_slot;
      // bf16 O of a warp whose 32 rows are all valid goes through shared
      // memory (this query tile's Q buffer, free once every MMA completed)
      // in the 128-byte-swizzled layout of the O map, then out with two TMA
      // stores of 32 rows x 64 columns: whole 128-byte lines instead of one
      // 16-byte piece of 32 different rows per store instruction.
      const bool o_tma = !partial && !args.o_fp32 && warp_all(row_valid);
      const uint32_t o_sm = sQ + t * SM::kQ + row * 128;
      uint32_t oall[D];  // the row of O: every 32-column load in flight, one wait
      if (k > 0) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32(tOt + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&oall[c * 32]));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&oall[c * 32]));
      }
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        const uint32_t* ov = &oall[c * 32];
        if (!row_valid) continue;
        if (!CP_IN_BOUNDS(q_slot < g.T && (!partial || r * g.R + s_begin < g.R * g.R), status)) continue;
        float o[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = (k > 0) ? __uint_as_float(ov[e]) * inv_l : 0.f;
        if (partial) {
          const size_t part_row = rank_local ? static_cast<size_t>(q_slot)
                                             : static_cast<size_t>(r * g.R + s_begin) * g.T + q_slot;
          float* dst = args.o_part + (part_row * g.Hq_loc + h) * D + c * 32;
#pragma unroll
          for (int e = 0; e < 32; e += 4) *reinterpret_cast<float4*>(dst + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
        } else if (o_tma) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            const int cc = c * 32 + e;                    // first column of this 16-byte piece
            const int piece = (cc & 63) >> 3;              // 16-byte piece within the 128-byte line
            st_shared_v4(o_sm + (cc >> 6) * HALF_BYTES + ((piece ^ (row & 7)) << 4), pack_bf16x2(o[e], o[e + 1]),
                         pack_bf16x2(o[e + 2], o[e + 3]), pack_bf16x2(o[e + 4], o[e + 5]),
                         pack_bf16x2(o[e + 6], o[e + 7]));
          }
        } else if (args.o_fp32) {
          float* dst = reinterpret_cast<float*>(args.o) + o_row_off + c * 32;
#pragma unroll
          for (int e = 0; e < 32; e += 4) *reinterpret_cast<float4*>(dst + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
        } else {
          __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(args.o) + o_row_off + c * 32;
#pragma unroll
          for (int e = 0; e < 32; e += 8)
            *reinterpret_cast<uint4*>(dst + e) =
                make_uint4(pack_bf16x2(o[e], o[e + 1]), pack_bf16x2(o[e + 2], o[e + 3]),
                           pack_bf16x2(o[e + 4], o[e + 5]), pack_bf16x2(o[e + 6], o[e + 7]));
        }
      }
      if (o_tma) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int y = q_row0 + it.q0 + t * BM + wq * 32;
          if (CP_IN_BOUNDS(y >= 0 && y + 32 <= q_rows, status)) {
            for (int hh = 0; hh < NH; ++hh)
              tma_store_2d(&tm_o, sQ + t * SM::kQ + hh * HALF_BYTES + wq * 32 * 128, qcol0() + hh * 64, y);
            bulk_commit();
            bulk_wait_read_all();
          }
        }
        __syncwarp();
      }
      if (row_valid && CP_IN_BOUNDS(q_slot < g.T, status)) {
        if (partial && rank_local)
          args.lse_part[static_cast<size_t>(h) * g.T + q_slot] = lse;
        else if (partial)
          args.lse_part[(static_cast<size_t>(r * g.R + s_begin) * g.Hq_loc + h) * g.T + q_slot] = lse;
        else
          args.lse[lse_idx] = lse;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
int launch_d(const FwdArgs& a, cudaStream_t stream) {
  const AttnGeom& g = a.g;
  // Rows of Q and of K/V: every rank's slots, or (one ring step of one rank)
  // that rank's T rows and the visiting chunk's T rows.
  // With seq_io the maps span the sequence-sharded tensors: R*T rows of all
  // heads.
  const uint64_t rows = a.rank_local ? static_cast<uint64_t>(g.T)
                                     : static_cast<uint64_t>(g.R) * (a.seq_io ? 1 : g.U) * g.T;
  const uint64_t kv_rows = a.rank_local ? rows : g.kv_global ? static_cast<uint64_t>(g.L) : rows;
  const uint64_t hq_cols = static_cast<uint64_t>(g.Hq_loc) * (a.seq_io ? g.U : 1) * D;
  const uint64_t hkv_cols = static_cast<uint64_t>(g.Hkv_loc) * (a.seq_io ? g.U : 1) * D;
  CUtensorMap mq, mk, mv, mo;
  if (!make_tile_map(&mq, a.q, hq_cols, rows) || !make_tile_map(&mk, a.k, hkv_cols, kv_rows) ||
      !make_tile_map(&mv, a.v, hkv_cols, kv_rows))
    return CP_ERR_CUDA;
  // bf16 O: the map of the TMA stores (32-row boxes), same shape as Q's.
  // Partial and fp32 outputs are written with plain stores; the map then
  // just repeats Q's.
  if (!a.o_part && !a.o_fp32) {
    if (!make_tile_map(&mo, a.o, hq_cols, rows, 32)) return CP_ERR_CUDA;
  } else {
    mo = mq;
  }
  const uint32_t smem = FwdSmem<D>::kBytes;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return CP_ERR_CUDA;
    attr_set = true;
  }
  const long long grid = static_cast<long long>(a.n_items) * g.Hq_loc;
  if (grid <= 0) return CP_OK;
  if (grid > 0x7fffffffLL) return CP_ERR_UNSUPPORTED;
  attn_fwd_kernel<D><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(mq, mk, mv, mo, a);
  return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

// Debug table of the tile classes (cp_tile_classes): one thread per work
// item walks the item's key tiles exactly as attn_fwd_kernel does and writes,
// per walked tile, {a, q0, len, step, kpos0, klen, class of query tile 0,
// class of query tile 1} (tile_class above).  At most `stride` rows per
// item; counts[i] = the number of tiles item i walks.
__global__ void tile_class_kernel(const FwdArgs args, int32_t* rows, int32_t* counts, int stride) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= args.n_items) return;
  const AttnGeom& g = args.g;
  const WorkItem it = args.items[i];
  const int r = it.a / g.U, u = it.a % g.U;
  const int s_begin = it.step < 0 ? 0 : it.step;
  const int s_end = it.step < 0 ? g.R : it.step + 1;
  const QWin win0 = make_qwin(g, it, r, 0, args.status), win1 = make_qwin(g, it, r, 1, args.status);
  int32_t* out = rows + static_cast<size_t>(i) * stride * 8;
  int n = 0;
  for_each_kv_tile(g, r, u, s_begin, s_end, win0.lo_min, win0.qp0 + it.len - 1, [&](int, int kpos0, int klen) {
    if (n < stride) {
      int32_t* o = out + static_cast<size_t>(n) * 8;
      o[0] = it.a;
      o[1] = it.q0;
      o[2] = it.len;
      o[3] = it.step;
      o[4] = kpos0;
      o[5] = klen;
      o[6] = tile_class(win0, kpos0, klen);
      o[7] = tile_class(win1, kpos0, klen);
    }
    ++n;
  });
  counts[i] = n;
}

}  // namespace

int launch_tile_classes(const FwdArgs& a, int32_t* rows, int32_t* counts, int stride, cudaStream_t stream) {
  if (a.n_items <= 0) return CP_OK;
  tile_class_kernel<<<(a.n_items + 127) / 128, 128, 0, stream>>>(a, rows, counts, stride);
  return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

int launch_attn_fwd(const FwdArgs& a, cudaStream_t stream) {
  if (a.d == 128) return launch_d<128>(a, stream);
  if (a.d == 64) return launch_d<64>(a, stream);
  return CP_ERR_UNSUPPORTED;
}

}  // namespace cpattn
