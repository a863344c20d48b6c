// attn_bwd.cu -- causal context-parallel attention backward on sm_103a.
//
// Gradients of O = softmax(scale Q K^T + mask) V from the forward's O and
// LSE, recomputing the probabilities instead of storing them (activation
// recompute: [L3P] siliconandsystems.com "Llama 3 parallelism", section
// "Long context changes more than attention cost").  With
// P = exp(scale S - LSE), D = rowsum(dO * O), dS = P * (dO V^T - D):
//
//   dV = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K,
//
// query heads of a GQA group summed into their KV head.  Three kernels,
// no atomics, deterministic:
//   delta    D per (query, head)                           bandwidth-bound
//   dkv      one CTA per 128-key tile and KV head: walks every visible
//            query tile (one ring step: of the ranks the chunk visits; all
//            steps in one launch: in position order) and every query head
//            of the group; S^T = K Q^T and dP^T = V dO^T in TMEM, P^T and
//            dS^T written back over them as packed bf16 and read from TMEM
//            as the A operands of dV += P^T dO and dK += dS^T Q; dV and dK
//            accumulated in TMEM; three Q and two dO tiles in flight, one
//            barrier for a query tile's Q and dO
//   dq       one CTA per 128-query tile and head: walks the visible key
//            tiles like the forward; Q in TMEM (S = Q K^T from TMEM), dO in
//            shared memory (dP = dO V^T), S, dP, dS and dQ each in a TMEM
//            buffer of its own, issued S_n, dP_n, dQ_{n-1}; four K and two
//            V tiles in flight, one barrier for a key tile's K and V
// Gradients of a KV chunk land on the rank that owns the chunk ([MTX]
// nougat.kr "MaxText long-context training and KV parallelism", "Split heads
// or rotate KV": the chunk's partial results travel with it).
//
// Attention rank a = r*U + u works on ring rank r's slots for head group u
// (U == 1 is plain sequence sharding); the ring runs over r within each
// head group.  The kernels read either the head-sharded layout of the
// Ulysses exchange or, with seq_io, the sequence-sharded tensors themselves
// (slot t of ring rank r is row r*T + t, group u a range of heads).
//
// Warp roles: warp 0 TMA producer, warp 1 TMEM allocator and MMA issuer,
// warps 2..9 element-wise: one TMEM lane = one row, warps 2-5 take the
// first 64 columns of their rows and warps 6-9 the last 64, so two
// element-wise warps share each SM sub-partition.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <type_traits>

#define CP_TU_ID ::cpattn::kTuAttnBwd
#include "debug.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace cpattn {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr uint32_t HALF_BYTES = 128 * 128;
constexpr int kThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 element-wise
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ bool warp_all(bool x) { return __all_sync(0xffffffffu, x); }



// Q K^T-type product over d: A and B both K-major, 128-byte swizzled.
// Issued warp-wide (see mma_bf16_ss_k128_warp).
template <int D>
__device__ __forceinline__ void mma_qk(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc) {
  if constexpr (D == 128)
    mma_bf16_ss_k128_warp<HALF_BYTES>(d_tmem, a, b, idesc, 0u);
  else
    mma_bf16_ss_k64_warp(d_tmem, a, b, idesc, 0u);
}

// ---------------------------------------------------------------- D = rowsum(dO * O)

// One warp per (attention rank, query head, 32 consecutive slots); lane i
// takes slot t0 + i: D = rowsum(dO * O) over its row with 16-byte loads,
// then -D and -LSE * log2(e) into the chunk-padded statistics layout
// (ld_index).  Consecutive slots make the warp's LSE loads and statistics
// stores whole 128-byte lines.  Then the padding slots get 0 and -inf.
// rows = attention ranks x T (T in rank-local mode).
template <int D, typename OT>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const OT* __restrict__ o,
                                                        const __nv_bfloat16* __restrict__ dO,
                                                        const float* __restrict__ lse, float* __restrict__ nlse,
                                                        float* __restrict__ nd, const AttnGeom g, int chunk_pad,
                                                        long long rows, int seq_io, int32_t* status) {
  const int H = g.Hq_loc, T = g.T;
  const int lane = threadIdx.x & 31;
  const long long ranks = rows / T;
  const int tblocks = (T + 31) / 32;
  const long long total = ranks * H * tblocks;
  [[maybe_unused]] const long long tp = static_cast<long long>(g.nchunks) * chunk_pad;
  const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long nwarps = nthreads >> 5;
  const long long gtid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long n_m = T / g.U;  // slots per attention rank (sequence-sharded LSE rows)
  for (long long wi = gtid >> 5; wi < total; wi += nwarps) {
    const long long ah = wi / tblocks;
    const int t = static_cast<int>(wi - ah * tblocks) * 32 + lane;
    const long long a_r = ah / H;
    const int h = static_cast<int>(ah - a_r * H);
    if (t >= T) continue;
    // Slot t of attention rank a_r, head h: head-sharded row a_r*T + t, or
    // with seq_io row (a_r/U)*T + t at head (a_r%U)*H + h of all H*U heads.
    const long long io = seq_io ? ((a_r / g.U) * T + t) * (static_cast<long long>(H) * g.U) + (a_r % g.U) * H + h
                                : (a_r * T + t) * H + h;
    const uint4* pd = reinterpret_cast<const uint4*>(dO + io * D);
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const uint4 dv = pd[c];
      const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
      float ov[8];
      if constexpr (sizeof(OT) == 2) {
        const uint4 x = reinterpret_cast<const uint4*>(o + io * D)[c];
        const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(o2[i]);
          ov[2 * i] = f.x;
          ov[2 * i + 1] = f.y;
        }
      } else {
        const float4 x0 = reinterpret_cast<const float4*>(o + io * D)[2 * c];
        const float4 x1 = reinterpret_cast<const float4*>(o + io * D)[2 * c + 1];
        ov[0] = x0.x, ov[1] = x0.y, ov[2] = x0.z, ov[3] = x0.w;
        ov[4] = x1.x, ov[5] = x1.y, ov[6] = x1.z, ov[7] = x1.w;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(d2[i]);
        acc0 = fmaf(ov[2 * i], f.x, acc0);
        acc1 = fmaf(ov[2 * i + 1], f.y, acc1);
      }
    }
    const float acc = acc0 + acc1;
    const long long li = seq_io ? (((a_r / g.U) * g.U + t / n_m) * (static_cast<long long>(H) * g.U) +
                                   (a_r % g.U) * H + h) * n_m + t % n_m
                                : (a_r * H + h) * T + t;
    const size_t di = ld_index(g, chunk_pad, static_cast<int>(a_r), h, t);
    if (CP_IN_BOUNDS(li >= 0 && li < ranks * H * T && di < static_cast<size_t>(ranks * H * tp), status)) {
      const float l = lse[li];
      nlse[di] = l == -INFINITY ? -INFINITY : -l * kLog2e;
      nd[di] = -acc;
    }
  }
  // Padding: slots [chunk, chunk_pad) of every chunk.
  const int padw = chunk_pad - g.chunk;
  const long long npad = ranks * H * g.nchunks * padw;
  for (long long i = gtid; i < npad; i += nthreads) {
    const long long c = i / padw;  // (rank, head, chunk)
    const long long idx = c * chunk_pad + g.chunk + (i - c * padw);
    if (CP_IN_BOUNDS(idx < ranks * H * tp, status)) {
      nlse[idx] = -INFINITY;
      nd[idx] = 0.f;
    }
  }
}

// ---------------------------------------------------------------- dQ (query-tile outer)

constexpr int kKStages = 4;  // K tiles in flight (K is last read by dQ, issued a tile later)
constexpr int kVStages = 2;  // V tiles in flight (V is read by dP only)

// One "full" barrier per key tile covers its K and V (indexed like K).
enum DqBar { DQ_Q_FULL = 0, DQ_DO_FULL, DQ_KV_FULL, DQ_K_EMPTY = DQ_KV_FULL + kKStages,
             DQ_V_EMPTY = DQ_K_EMPTY + kKStages, DQ_S_FULL = DQ_V_EMPTY + kVStages, DQ_DP_FULL, DQ_S_FREE,
             DQ_DP_FREE, DQ_DS_FULL, DQ_DS_EMPTY, DQ_DONE, DQ_DRAIN, DQ_NUM_BARS };

// Q lives in tensor memory (the A operand of S = Q K^T); dO sits in shared
// memory beside the streamed K and V tiles (the A operand of dP = dO V^T),
// which leaves tensor memory room for a dS buffer of its own.
template <int D>
struct DqSmem {
  static constexpr uint32_t kT = 128 * D * 2;
  static constexpr uint32_t offK = 0, offV = offK + kKStages * kT, offDO = offV + kVStages * kT;
  static constexpr uint32_t offBar = offDO + kT;
  static constexpr uint32_t offMisc = offBar + 24 * 8;
  static constexpr uint32_t kUsed = offMisc + 16;
  static constexpr uint32_t kBytes = (kUsed + 1024 < 120 * 1024) ? 120 * 1024 : kUsed + 1024;
  static_assert(DQ_NUM_BARS <= 24, "barrier slots");
};

// S = A B^T over K = D with A in TMEM (contiguous packed columns) and B K-major
// in shared memory.  Issued warp-wide.
template <int D>
__device__ __forceinline__ void mma_tk(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc) {
  if constexpr (D == 128)
    mma_bf16_ts_kmaj_k128_warp<HALF_BYTES>(d_tmem, a_tmem, b, idesc, 0u);
  else
    mma_bf16_ts_kmaj_k64_warp(d_tmem, a_tmem, b, idesc, 0u);
}

// Key tiles a query tile of ring rank r walks: one ring step (the chunk of
// rank (r - s) mod R), or, for every ring step in one launch, the chunks in
// position order (the order is free and the fp32 sums are exact up to
// rounding; in position order the CTAs resident at once read the same key
// tiles and share them in L2, as in the forward kernel).
template <typename F>
__device__ __forceinline__ void for_each_kv_tile(const AttnGeom& g, int r, int u, int s_begin, int s_end, int lo_min,
                                                 int qpos_last, F&& f) {
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
    for (int ch = 0; ch < nchunks; ++ch) {
      const int cslot0 = ch * g.chunk;
      const int cpos0 = slot_pos(g, src, cslot0);
      const int lo = max(cpos0, lo_min);
      const int hi = min(cpos0 + g.chunk - 1, qpos_last);
      if (lo > hi) continue;
      const int t1 = (hi - cpos0) / BN;
      for (int t = (lo - cpos0) / BN; t <= t1; ++t)
        f((src * g.U + u) * g.T + cslot0 + t * BN, cpos0 + t * BN, min(BN, g.chunk - t * BN));
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const BwdArgs args) {
  using SM = DqSmem<D>;
  constexpr int NH = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sK = s_base + SM::offK, sV = s_base + SM::offV, sDO = s_base + SM::offDO;
  auto bar = [&](int i) { return s_base + SM::offBar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::offMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM::offMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttnGeom& g = args.g;
  int32_t* status = args.status;
  const int Hq = g.Hq_loc;
  // Launch order: item-major (heads fastest), or stream-major (one K/V
  // stream (u, KV head) after another, the G query heads of the KV head
  // adjacent, so the CTAs resident at once read the same K/V tiles).
  int item_idx, h;
  if (args.stream_major) {
    const int per_stream = args.n_items_q_u * g.G;
    const int sidx = blockIdx.x / per_stream;
    const int rem = blockIdx.x - sidx * per_stream;
    const int su = sidx / g.Hkv_loc;
    item_idx = su * args.n_items_q_u + rem / g.G;
    h = (sidx - su * g.Hkv_loc) * g.G + rem % g.G;
  } else {
    item_idx = blockIdx.x / Hq;
    h = blockIdx.x % Hq;
  }
  if (!CP_IN_BOUNDS(item_idx < args.n_items_q, status)) return;
  const WorkItem it = args.items_q[item_idx];
  // A query tile lies inside its attention rank's slots.
  if (!CP_IN_BOUNDS(it.a >= 0 && it.a < g.R * g.U && it.q0 >= 0 && it.len > 0 && it.len <= BM &&
                        it.q0 + it.len <= g.T, status))
    return;
  const bool rank_local = args.rank_local != 0;
  const bool seq_io = args.seq_io != 0;
  // rows of Q, dO, K, V, dQ (sequence-sharded: ring rank r's slots are rows r*T..)
  [[maybe_unused]] const int rows = rank_local ? g.T : (seq_io ? g.R : g.R * g.U) * g.T;
  const int a = it.a, r = a / g.U, u = a % g.U;  // rank a = ring rank r, Ulysses member u
  const int s_begin = rank_local ? args.step : 0, s_end = rank_local ? args.step + 1 : g.R;
  // Rank-local mode: the rank's rows start at 0, and so do the visiting chunk's.
  const int q_row0 = rank_local ? 0 : (seq_io ? r : a) * g.T;
  const int kv_sub = rank_local ? (((r - s_begin + g.R) % g.R) * g.U + u) * g.T : 0;
  const int qpos0 = slot_pos(g, r, it.q0);
  const int qpos_last = qpos0 + it.len - 1;
  if (!CP_IN_BOUNDS(qpos0 >= 0 && qpos_last < g.L, status)) return;
  const int lo_min = g.doc_start ? g.doc_start[qpos0] : 0;
  const int lo_max = g.doc_start ? g.doc_start[qpos_last] : 0;
  const int hkv = h / g.G;

  if (threadIdx.x == 0) {
    mbar_init(bar(DQ_Q_FULL), 8);  // the element-wise warps, once Q sits in TMEM
    mbar_init(bar(DQ_DO_FULL), 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(bar(DQ_KV_FULL + i), 1);
      mbar_init(bar(DQ_K_EMPTY + i), 1);
    }
    for (int i = 0; i < kVStages; ++i) mbar_init(bar(DQ_V_EMPTY + i), 1);
    mbar_init(bar(DQ_S_FULL), 1);
    mbar_init(bar(DQ_DP_FULL), 1);
    mbar_init(bar(DQ_S_FREE), 8);
    mbar_init(bar(DQ_DP_FREE), 8);
    mbar_init(bar(DQ_DS_FULL), 8);
    mbar_init(bar(DQ_DS_EMPTY), 1);
    mbar_init(bar(DQ_DONE), 1);
    mbar_init(bar(DQ_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM: S at 0, dP at 128, dQ at 256, the A operand Q at 384 (D/2 packed
  // columns) and dS (packed bf16, 64 columns) at 448.
  const uint32_t tS = tmem, tdP = tmem + 128, tdQ = tmem + 256, tQ = tmem + 384, tdS = tmem + 448;

  if (warp == 0) {
    if (lane == 0) {
      // The tile's dO rows (rows past a ragged tile's end are other rows of
      // the tensor or the map's zero fill: their P is 0, and so is their dS).
      {
        const int qrow = q_row0 + it.q0;
        const int q_col = (seq_io ? u * Hq + h : h) * D;
        mbar_arrive_expect_tx(bar(DQ_DO_FULL), SM::kT);
        (void)CP_IN_BOUNDS(qrow >= 0 && qrow < rows, status);
        for (int hh = 0; hh < NH; ++hh)
          tma_load_2d(sDO + hh * HALF_BYTES, &tm_do, bar(DQ_DO_FULL), q_col + hh * 64, qrow);
      }
      int nk = 0;  // key tiles loaded
      for_each_kv_tile(g, r, u, s_begin, s_end, lo_min, qpos_last, [&](int kv_row_all, int, int) {
        if (*abort_flag) return;
        // kv_row_all = (src*U + u)*T + slot in the head-sharded row space.
        const int kv_row = seq_io ? (kv_row_all / (g.T * g.U)) * g.T + kv_row_all % g.T : kv_row_all - kv_sub;
        const int kv_col = (seq_io ? u * g.Hkv_loc + hkv : hkv) * D;
        const int ks = nk % kKStages, vs = nk % kVStages;
        if (!mbar_wait(bar(DQ_K_EMPTY + ks), ((nk / kKStages) & 1) ^ 1, abort_flag, status)) return;
        if (!mbar_wait(bar(DQ_V_EMPTY + vs), ((nk / kVStages) & 1) ^ 1, abort_flag, status)) return;
        mbar_arrive_expect_tx(bar(DQ_KV_FULL + ks), 2 * SM::kT);
        (void)CP_IN_BOUNDS(kv_row >= 0 && kv_row < rows && hkv < g.Hkv_loc, status);
        for (int hh = 0; hh < NH; ++hh) {
          tma_load_2d(sK + ks * SM::kT + hh * HALF_BYTES, &tm_k, bar(DQ_KV_FULL + ks), kv_col + hh * 64, kv_row);
          tma_load_2d(sV + vs * SM::kT + hh * HALF_BYTES, &tm_v, bar(DQ_KV_FULL + ks), kv_col + hh * 64, kv_row);
        }
        ++nk;
      });
      if (*abort_flag) {
        // Wait for this CTA's own copies: the last loads of each stage.
        mbar_wait(bar(DQ_DO_FULL), 0, nullptr, status);
        for (int i = max(0, nk - kKStages); i < nk; ++i)
          mbar_wait(bar(DQ_KV_FULL + i % kKStages), (i / kKStages) & 1, nullptr, status);
      }
    }
  } else if (warp == 1) {
    // The whole warp runs the issue loop (warp-uniform operands); one
    // elected lane executes each tcgen05 instruction.
    {
      constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, 0);
      constexpr uint32_t idesc_dq = idesc_bf16_f32(BM, D, 1);
      const uint64_t dK0 = smem_desc_sw128(sK, 16, 1024), dV0 = smem_desc_sw128(sV, 16, 1024);
      const uint64_t dDO = smem_desc_sw128(sDO, 16, 1024);
      const uint64_t dKmn0 = smem_desc_sw128(sK, HALF_BYTES, 1024);
      constexpr uint64_t kStep = SM::kT >> 4;  // one stage in descriptor units
      // Issue order for key tile n: S_n, dP_n, dQ_{n-1}.  S and dP have one
      // TMEM buffer each, free once the element-wise warps have loaded S_{n-1}
      // (resp. dP_{n-1}) into registers.  dS_{n-1} has a buffer of its own,
      // written once dQ_{n-2} has read it, so the element-wise warps form
      // dS_{n-1} while S_n and dP_n run.  The tensor pipe's queue holds only
      // a couple of MMAs, so anything the issuer does between two MMA groups
      // (a barrier check costs about 80 cycles even when the phase has
      // completed) idles the pipe once it is longer than that: one check per
      // group, two barriers checked at once before S_n, and a plain counted
      // loop.
      auto issue_dq = [&](int m) {  // dQ += dS_m K_m
        mma_bf16_ts_k128_warp(tdQ, tdS, dKmn0 + static_cast<uint64_t>(m % kKStages) * kStep, idesc_dq,
                              m > 0 ? 1u : 0u);
        mma_commit_warp(bar(DQ_K_EMPTY + m % kKStages));
        mma_commit_warp(bar(DQ_DS_EMPTY));
      };
      int ntiles = 0;
      for_each_kv_tile(g, r, u, s_begin, s_end, lo_min, qpos_last, [&](int, int, int) { ++ntiles; });
      bool ok = warp_all(mbar_wait(bar(DQ_Q_FULL), 0, abort_flag, status)) &&
                warp_all(mbar_wait(bar(DQ_DO_FULL), 0, abort_flag, status));
      for (int n = 0; ok && n < ntiles; ++n) {
        const int ks = n % kKStages, vs = n % kVStages;
        const uint32_t kv_par = (n / kKStages) & 1, prev = (n - 1) & 1;
        // K_n and V_n landed; S_{n-1} is in registers.
        if (!warp_all(n >= 1 ? mbar_try_wait2(bar(DQ_KV_FULL + ks), kv_par, bar(DQ_S_FREE), prev)
                             : mbar_try_wait(bar(DQ_KV_FULL + ks), kv_par)))
          ok = warp_all(mbar_wait(bar(DQ_KV_FULL + ks), kv_par, abort_flag, status)) &&
               (n < 1 || warp_all(mbar_wait(bar(DQ_S_FREE), prev, abort_flag, status)));
        if (!ok) break;
        tc_fence_after();
        mma_tk<D>(tS, tQ, dK0 + static_cast<uint64_t>(ks) * kStep, idesc_s);
        mma_commit_warp(bar(DQ_S_FULL));
        // dP_{n-1} is in registers.
        if (n >= 1 && !(ok = warp_all(mbar_wait(bar(DQ_DP_FREE), prev, abort_flag, status)))) break;
        tc_fence_after();
        if constexpr (D == 128)
          mma_bf16_ss_k128_warp<HALF_BYTES>(tdP, dDO, dV0 + static_cast<uint64_t>(vs) * kStep, idesc_s, 0u);
        else
          mma_bf16_ss_k64_warp(tdP, dDO, dV0 + static_cast<uint64_t>(vs) * kStep, idesc_s, 0u);
        mma_commit_warp(bar(DQ_DP_FULL));
        mma_commit_warp(bar(DQ_V_EMPTY + vs));
        if (n >= 1) {
          if (!(ok = warp_all(mbar_wait(bar(DQ_DS_FULL), prev, abort_flag, status)))) break;
          tc_fence_after();
          issue_dq(n - 1);
        }
      }
      if (ok && ntiles > 0 && warp_all(mbar_wait(bar(DQ_DS_FULL), (ntiles - 1) & 1, abort_flag, status))) {
        tc_fence_after();
        issue_dq(ntiles - 1);
        mma_commit_warp(bar(DQ_DONE));
      }
      mma_commit_warp(bar(DQ_DRAIN));
      mbar_wait(bar(DQ_DRAIN), 0, nullptr, status);
    }
  } else {
    const int wq = warp & 3;
    const int half = (warp - 2) >> 2;  // warps 2-5: key columns 0-63; warps 6-9: 64-127
    const int row = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const bool row_valid = row < it.len;
    const int my_pos = row_valid ? qpos0 + row : -1;
    const int my_lo = (row_valid && g.doc_start) ? g.doc_start[my_pos] : 0;
    // -LSE*log2(e) and -D of this row, prepared by the delta pass.
    const size_t lrow = ld_index(g, args.chunk_pad, rank_local ? 0 : a, h, row_valid ? it.q0 + row : 0);
    const bool ld_ok = !row_valid || CP_IN_BOUNDS(lrow < static_cast<size_t>(rank_local ? 1 : g.R * g.U) * Hq *
                                                             g.nchunks * args.chunk_pad,
                                                  status);
    const float nl2 = (row_valid && ld_ok) ? args.nlse[lrow] : -INFINITY;
    const float ndl = (row_valid && ld_ok) ? args.nd[lrow] : 0.f;
    const float sl2 = g.scale * kLog2e;
    {
      // This thread's half of its Q row into TMEM (lane = row; the bf16
      // pairs of a row in memory order are the packed columns).  Rows past
      // the tile's end are zero.
      constexpr int W = D / 4;  // 32-bit words per half row
      const size_t grow = static_cast<size_t>(q_row0 + it.q0 + row) * (seq_io ? Hq * g.U : Hq) + (seq_io ? u * Hq + h : h);
      const bool in = row_valid && CP_IN_BOUNDS(q_row0 + it.q0 + row < rows, status);
      const uint4* qsrc = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(args.q) + grow * D) + half * (W / 4);
      uint32_t qw[W];
#pragma unroll
      for (int i = 0; i < W / 4; ++i) {
        const uint4 x = in ? qsrc[i] : make_uint4(0u, 0u, 0u, 0u);
        qw[4 * i] = x.x, qw[4 * i + 1] = x.y, qw[4 * i + 2] = x.z, qw[4 * i + 3] = x.w;
      }
      if constexpr (D == 128)
        tmem_st32(tQ + lane_off + half * W, qw);
      else
        tmem_st16(tQ + lane_off + half * W, qw);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(DQ_Q_FULL));
    }
    int n = 0;
    bool ok = true;
    for_each_kv_tile(g, r, u, s_begin, s_end, lo_min, qpos_last, [&](int, int kpos0, int klen) {
      if (!ok) return;
      ok = warp_all(mbar_wait(bar(DQ_S_FULL), n & 1, abort_flag, status));
      if (!ok) return;
      tc_fence_after();
      const bool full = (klen == BN) && (kpos0 + BN - 1 <= qpos0) && (lo_max <= kpos0);
      const int c_lo = my_lo - kpos0;
      const int c_hi = min(my_pos - kpos0, klen - 1);
      // Phase A: P = exp2(S * scale*log2e - LSE*log2e), masked, as packed bf16
      // (this warp's half of the row: 32-column chunks c4 = 2*half, 2*half+1).
      float pf[BN / 2];  // P of this half of the row, fp32 (dS is formed from it)
      const f32x2 nsl2 = make_f32x2(sl2, sl2), nlse2 = make_f32x2(nl2, nl2);
      uint32_t sr2[2][32];  // both chunks of this half: one TMEM round trip
      tmem_ld32(tS + lane_off + 64 * half, sr2[0]);
      tmem_ld32(tS + lane_off + 64 * half + 32, sr2[1]);
      tmem_wait_ld();
      reg_fence(sr2[0]);
      reg_fence(sr2[1]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(DQ_S_FREE));
      // Two instantiations: tiles wholly inside the window take the loop with
      // no mask at all (a mask test folded into every element costs more
      // than the rest of the loop).
      auto phase_a = [&](auto masked) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c4 = 2 * half + cc;
          const uint32_t* sr = sr2[cc];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int col = c4 * 32 + e;
            const f32x2 y = fma_f32x2(make_f32x2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), nsl2, nlse2);
            float y0, y1;
            split_f32x2(y, y0, y1);
            float x0 = ex2_approx(y0), x1 = ex2_approx(y1);
            if constexpr (decltype(masked)::value) {
              if (col < c_lo || col > c_hi) x0 = 0.f;
              if (col + 1 < c_lo || col + 1 > c_hi) x1 = 0.f;
            }
            pf[cc * 32 + e] = x0;
            pf[cc * 32 + e + 1] = x1;
          }
        }
      };
      if (full)
        phase_a(std::false_type{});
      else
        phase_a(std::true_type{});
      // Phase B: dS = P * (dP - D), packed to bf16 pairs in the dS buffer
      // (keys 64*half + 32*cc.. -> columns 32*half + 16*cc..): the A operand
      // of dQ.  The dP columns are released as soon as they are in
      // registers; dS is stored once dQ_{n-1} has read the buffer.
      ok = warp_all(mbar_wait(bar(DQ_DP_FULL), n & 1, abort_flag, status));
      if (!ok) return;
      tc_fence_after();
      uint32_t pr2[2][32];
      tmem_ld32(tdP + lane_off + 64 * half, pr2[0]);
      tmem_ld32(tdP + lane_off + 64 * half + 32, pr2[1]);
      tmem_wait_ld();
      reg_fence(pr2[0]);
      reg_fence(pr2[1]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(DQ_DP_FREE));
      uint32_t dsp[2][16];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const uint32_t* pr = pr2[cc];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const f32x2 dd = add_f32x2(make_f32x2(__uint_as_float(pr[e]), __uint_as_float(pr[e + 1])),
                                     make_f32x2(ndl, ndl));
          float s0, s1;
          split_f32x2(mul_f32x2(make_f32x2(pf[cc * 32 + e], pf[cc * 32 + e + 1]), dd), s0, s1);
          dsp[cc][e / 2] = pack_bf16x2(s0, s1);
        }
      }
      if (n >= 1) {
        ok = warp_all(mbar_wait(bar(DQ_DS_EMPTY), (n - 1) & 1, abort_flag, status));
        if (!ok) return;
        tc_fence_after();
      }
      tmem_st16(tdS + lane_off + 32 * half, dsp[0]);
      tmem_st16(tdS + lane_off + 32 * half + 16, dsp[1]);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(DQ_DS_FULL));
      ++n;
    });
    if (ok && n > 0) {
      ok = warp_all(mbar_wait(bar(DQ_DONE), 0, abort_flag, status));
      if (ok) tc_fence_after();
    }
    // Accumulate mode adds to dQ (nothing to add when no key tile was seen).
    if (ok && !(args.accumulate && n == 0)) {
      float* dst = args.dq + (static_cast<size_t>(q_row0 + it.q0 + row) * (seq_io ? Hq * g.U : Hq) +
                              (seq_io ? u * Hq + h : h)) * D;
      const bool store_ok = !row_valid || CP_IN_BOUNDS(q_row0 + it.q0 + row < rows, status);
      for (int c4 = half * (D / 64); c4 < (half + 1) * (D / 64); ++c4) {
        uint32_t v[32];
        if (n > 0) {
          tmem_ld32(tdQ + lane_off + c4 * 32, v);
          tmem_wait_ld();
          reg_fence(v);
        }
        if (!row_valid || !store_ok) continue;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          float4 x = n > 0 ? make_float4(__uint_as_float(v[e]) * g.scale, __uint_as_float(v[e + 1]) * g.scale,
                                         __uint_as_float(v[e + 2]) * g.scale, __uint_as_float(v[e + 3]) * g.scale)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
          float4* p4 = reinterpret_cast<float4*>(dst + c4 * 32 + e);
          if (args.accumulate) {
            const float4 y = *p4;
            x.x += y.x;
            x.y += y.y;
            x.z += y.z;
            x.w += y.w;
          }
          *p4 = x;
        }
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

// ---------------------------------------------------------------- dK, dV (key-tile outer)

// One "full" barrier per query tile covers its Q and dO (indexed like Q).
enum DkvBar { KV_FULL = 0, KV_QD_FULL = 1, KV_Q_EMPTY = 4, KV_DO_EMPTY = 7, KV_S_FULL = 9,
              KV_DP_FULL = 10, KV_P_FULL = 11, KV_DS_FULL = 12, KV_ACC_DONE = 13, KV_DRAIN = 14,
              KV_LD_FULL = 15,   // +buffer: the LSE/D of a query tile are staged (4 writer warps)
              KV_LD_EMPTY = 17,  // +buffer: every element-wise warp has read them (8 warps)
              KV_NUM_BARS = 19 };

constexpr int kQStages = 3;   // Q tiles in flight (Q is last read by dK, the last product of a tile)
constexpr int kDOStages = 2;  // dO tiles in flight (dO is last read by dV)

template <int D>
struct DkvSmem {
  static constexpr uint32_t kT = 128 * D * 2;
  static constexpr uint32_t offK = 0, offV = kT, offQ = 2 * kT, offDO = offQ + kQStages * kT;
  static constexpr uint32_t offBar = offDO + kDOStages * kT;
  static constexpr uint32_t offLD = offBar + 24 * 8;   // 2 buffers x (128 -LSE*log2(e) + 128 -D floats)
  static constexpr uint32_t offMeta = offLD + 2 * 2 * 128 * 4;  // 2 x {first position, length} of the query tile
  static constexpr uint32_t offMisc = offMeta + 2 * 8;
  static constexpr uint32_t kUsed = offMisc + 16;
  // Up to 1 KB of slack aligns the tiles to the 128-byte swizzle's 1 KB
  // atoms, but no more than the per-CTA limit is requested: the dynamic base
  // is 1 KB-aligned in practice, and the kernel checks that the aligned
  // layout fits (an error status otherwise, before anything is touched).
  static constexpr uint32_t kMaxDyn = 227 * 1024;
  static constexpr uint32_t kBytes = (kUsed + 1024 < 120 * 1024) ? 120 * 1024
                                     : (kUsed + 1024 < kMaxDyn ? kUsed + 1024 : kMaxDyn);
  static_assert(kUsed <= kMaxDyn, "dkv shared-memory layout");
};

// Every query tile (of every ring rank, in ring order from the owner) and
// every query head of KV head jh that may see the key tile [kpos0, hi_max].
template <typename F>
__device__ __forceinline__ void for_each_q_tile(const AttnGeom& g, int src, int s_begin, int s_end, int kpos0,
                                                int hi_max, int jh, F&& f) {
  if (s_begin == 0 && s_end == g.R && g.R > 1) {
    // Every ring step in one launch: query chunks in position order (see
    // for_each_kv_tile).
    const int c = g.chunk;
    const int j1 = hi_max / c;
    for (int j = kpos0 / c; j <= j1; ++j) {
      int rr, cslot0;
      chunk_owner(g, j, rr, cslot0);
      const int cpos0 = j * c;
      const int lo = max(cpos0, kpos0);
      const int hi = min(cpos0 + c - 1, hi_max);
      const int t1 = (hi - cpos0) / BM;
      for (int t = (lo - cpos0) / BM; t <= t1; ++t)
        for (int hh = 0; hh < g.G; ++hh)
          f(rr, cslot0 + t * BM, cpos0 + t * BM, min(BM, c - t * BM), jh * g.G + hh);
    }
    return;
  }
  const int nchunks = g.nchunks;
  for (int s = s_begin; s < s_end; ++s) {
    const int rr = (src + s) % g.R;
    for (int ch = 0; ch < nchunks; ++ch) {
      const int cslot0 = ch * g.chunk;
      const int cpos0 = slot_pos(g, rr, cslot0);
      const int lo = max(cpos0, kpos0);
      const int hi = min(cpos0 + g.chunk - 1, hi_max);
      if (lo > hi) continue;
      const int t1 = (hi - cpos0) / BM;
      for (int t = (lo - cpos0) / BM; t <= t1; ++t)
        for (int hh = 0; hh < g.G; ++hh)
          f(rr, cslot0 + t * BM, cpos0 + t * BM, min(BM, g.chunk - t * BM), jh * g.G + hh);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                        const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const BwdArgs args) {
  using SM = DkvSmem<D>;
  constexpr int NH = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (static_cast<uint32_t>(smem - smem_raw) + SM::kUsed > SM::kBytes) {
    if (threadIdx.x == 0) record_status(args.status, CP_ERR_DEVICE_BOUNDS);
    return;
  }
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sK = s_base + SM::offK, sV = s_base + SM::offV, sQ = s_base + SM::offQ, sDO = s_base + SM::offDO;
  auto bar = [&](int i) { return s_base + SM::offBar + 8u * i; };
  // Two buffers b of [128 -LSE * log2(e)][128 -D] per query column, and the
  // first position and length of the query tile each holds.
  const uint32_t aLD = s_base + SM::offLD;
  volatile int* sMeta = reinterpret_cast<volatile int*>(smem + SM::offMeta);  // [2][2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::offMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM::offMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttnGeom& g = args.g;
  int32_t* status = args.status;
  const int Hkv = g.Hkv_loc, Hq = g.Hq_loc;
  // Launch order: item-major (KV heads fastest), or stream-major (one
  // (u, KV head) after another, so the CTAs resident at once read the same
  // query tiles of that KV head's query heads).
  int item_idx, jh;
  if (args.stream_major) {
    const int sidx = blockIdx.x / args.n_items_kv_u;
    const int su = sidx / Hkv;
    item_idx = su * args.n_items_kv_u + (blockIdx.x - sidx * args.n_items_kv_u);
    jh = sidx - su * Hkv;
  } else {
    item_idx = blockIdx.x / Hkv;
    jh = blockIdx.x % Hkv;
  }
  if (!CP_IN_BOUNDS(item_idx < args.n_items_kv, status)) return;
  const WorkItem it = args.items_kv[item_idx];
  // A key tile lies inside its attention rank's slots.
  if (!CP_IN_BOUNDS(it.a >= 0 && it.a < g.R * g.U && it.q0 >= 0 && it.len > 0 && it.len <= BM &&
                        it.q0 + it.len <= g.T, status))
    return;
  const bool rank_local = args.rank_local != 0;
  const bool seq_io = args.seq_io != 0;
  // rows of Q, dO, K, V, dK, dV (sequence-sharded: ring rank r's slots are rows r*T..)
  [[maybe_unused]] const int rows = rank_local ? g.T : (seq_io ? g.R : g.R * g.U) * g.T;
  const int a = it.a, src = a / g.U, u = a % g.U;  // key tile of rank a = ring rank src, member u
  const int s_begin = rank_local ? args.step : 0, s_end = rank_local ? args.step + 1 : g.R;
  // Rank-local mode: the chunk's rows start at 0, and so do the holder's.
  const int k_row0 = rank_local ? 0 : (seq_io ? src : a) * g.T;
  const int kpos0 = slot_pos(g, src, it.q0);
  const int kpos_last = kpos0 + it.len - 1;
  if (!CP_IN_BOUNDS(kpos0 >= 0 && kpos_last < g.L, status)) return;
  const int hi_max = g.doc_end ? g.doc_end[kpos_last] - 1 : g.L - 1;
  const int hi_min = g.doc_end ? g.doc_end[kpos0] - 1 : g.L - 1;

  if (threadIdx.x == 0) {
    mbar_init(bar(KV_FULL), 1);
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(bar(KV_QD_FULL + i), 1);
      mbar_init(bar(KV_Q_EMPTY + i), 1);
    }
    for (int i = 0; i < kDOStages; ++i) mbar_init(bar(KV_DO_EMPTY + i), 1);
    mbar_init(bar(KV_S_FULL), 1);
    mbar_init(bar(KV_DP_FULL), 1);
    mbar_init(bar(KV_P_FULL), 8);
    mbar_init(bar(KV_DS_FULL), 8);
    mbar_init(bar(KV_ACC_DONE), 1);
    mbar_init(bar(KV_DRAIN), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(KV_LD_FULL + i), 1);
      mbar_init(bar(KV_LD_EMPTY + i), 8);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM: S^T (then P^T, packed bf16) at 0, dP^T (then dS^T) at 128, dV at 256, dK at 256 + D.
  const uint32_t tSt = tmem, tdPt = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(KV_FULL), 2 * SM::kT);
      const int krow = k_row0 + it.q0;
      (void)CP_IN_BOUNDS(krow >= 0 && krow < rows, status);
      for (int hh = 0; hh < NH; ++hh) {
        const int kv_col = (seq_io ? u * Hkv + jh : jh) * D;
        tma_load_2d(sK + hh * HALF_BYTES, &tm_k, bar(KV_FULL), kv_col + hh * 64, krow);
        tma_load_2d(sV + hh * HALF_BYTES, &tm_v, bar(KV_FULL), kv_col + hh * 64, krow);
      }
      int nq = 0, nld = 0;  // query tiles (Q and dO) and statistics loads issued
      // statistics of every attention rank (one in rank-local mode)
      [[maybe_unused]] const size_t ld_total =
          static_cast<size_t>(rank_local ? 1 : g.R * g.U) * Hq * g.nchunks * args.chunk_pad;
      for_each_q_tile(g, src, s_begin, s_end, kpos0, hi_max, jh, [&](int rr, int qslot0, int qpos0, int qlen, int h) {
        if (*abort_flag) return;
        const int qs = nq % kQStages, ds = nq % kDOStages;
        const int qrow = (rank_local ? 0 : (seq_io ? rr : rr * g.U + u) * g.T) + qslot0;
        const int q_col = (seq_io ? u * Hq + h : h) * D;
        if (!mbar_wait(bar(KV_Q_EMPTY + qs), ((nq / kQStages) & 1) ^ 1, abort_flag, status)) return;
        if (!mbar_wait(bar(KV_DO_EMPTY + ds), ((nq / kDOStages) & 1) ^ 1, abort_flag, status)) return;
        mbar_arrive_expect_tx(bar(KV_QD_FULL + qs), 2 * SM::kT);
        (void)CP_IN_BOUNDS(qrow >= 0 && qrow < rows && h < Hq, status);
        for (int hh = 0; hh < NH; ++hh) {
          tma_load_2d(sQ + qs * SM::kT + hh * HALF_BYTES, &tm_q, bar(KV_QD_FULL + qs), q_col + hh * 64, qrow);
          tma_load_2d(sDO + ds * SM::kT + hh * HALF_BYTES, &tm_do, bar(KV_QD_FULL + qs), q_col + hh * 64, qrow);
        }
        ++nq;
        // The tile's -LSE*log2(e) and -D (128 each, chunk-padded so the copy
        // starts on a 512-byte boundary) and its position and length, for
        // the element-wise warps; the stage is reused once all 8 of them
        // have finished the tile two before.
        const int ls = nld & 1;
        if (nld >= 2 && !mbar_wait(bar(KV_LD_EMPTY + ls), ((nld >> 1) - 1) & 1, abort_flag, status)) return;
        const size_t li = ld_index(g, args.chunk_pad, rank_local ? 0 : rr * g.U + u, h, qslot0);
        (void)CP_IN_BOUNDS(li + 128 <= ld_total, status);
        sMeta[2 * ls] = qpos0;
        sMeta[2 * ls + 1] = qlen;
        mbar_arrive_expect_tx(bar(KV_LD_FULL + ls), 1024);
        bulk_load(aLD + ls * 1024, args.nlse + li, 512, bar(KV_LD_FULL + ls));
        bulk_load(aLD + ls * 1024 + 512, args.nd + li, 512, bar(KV_LD_FULL + ls));
        ++nld;
      });
      if (!*abort_flag) {
        // End of the walk: a stage with length 0 tells the element-wise warps.
        const int ls = nld & 1;
        if (nld < 2 || mbar_wait(bar(KV_LD_EMPTY + ls), ((nld >> 1) - 1) & 1, abort_flag, status)) {
          sMeta[2 * ls + 1] = 0;
          mbar_arrive(bar(KV_LD_FULL + ls));
        }
      }
      if (*abort_flag) {
        for (int i = max(0, nld - 2); i < nld; ++i)
          mbar_wait(bar(KV_LD_FULL + (i & 1)), (i >> 1) & 1, nullptr, status);
        // Wait for this CTA's own copies before it exits (a stage is reused
        // only after its previous load landed, so the last loads of each
        // stage are the only ones that can still be in flight).
        mbar_wait(bar(KV_FULL), 0, nullptr, status);
        for (int i = max(0, nq - kQStages); i < nq; ++i)
          mbar_wait(bar(KV_QD_FULL + i % kQStages), (i / kQStages) & 1, nullptr, status);
      }
    }
  } else if (warp == 1) {
    // The whole warp runs the issue loop (warp-uniform operands); one
    // elected lane executes each tcgen05 instruction.
    {
      constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, 0);
      constexpr uint32_t idesc_acc = idesc_bf16_f32(BM, D, 1);
      const uint64_t dK0 = smem_desc_sw128(sK, 16, 1024), dV0 = smem_desc_sw128(sV, 16, 1024);
      const uint64_t dQ0 = smem_desc_sw128(sQ, 16, 1024), dDO0 = smem_desc_sw128(sDO, 16, 1024);
      const uint64_t dQmn0 = smem_desc_sw128(sQ, HALF_BYTES, 1024), dDOmn0 = smem_desc_sw128(sDO, HALF_BYTES, 1024);
      constexpr uint64_t kStep = SM::kT >> 4;  // one stage in descriptor units
      // Issue order for query tile n: dV_{n-1}, S_n, dK_{n-1}, dP_n.  P^T and
      // dS^T stay in TMEM, where the element-wise warps wrote them over the
      // S^T and dP^T they came from, and are the A operands of dV and dK;
      // S_n (dP_n) overwrites those columns only after dV_{n-1} (dK_{n-1}),
      // issued before it by this thread, has read them.  Two checks per tile
      // (P_{n-1} written with Q_n and dO_n landed; dS_{n-1} written) and a
      // plain counted loop: each check between two MMA groups idles the
      // tensor pipe for about as long as it takes.
      auto issue_dv = [&](int m) {  // dV += P^T_m dO_m
        mma_bf16_ts_k128_halves_warp(tdV, tSt, dDOmn0 + static_cast<uint64_t>(m % kDOStages) * kStep, idesc_acc,
                                m > 0 ? 1u : 0u);
        mma_commit_warp(bar(KV_DO_EMPTY + m % kDOStages));
      };
      auto issue_dk = [&](int m) {  // dK += dS^T_m Q_m
        mma_bf16_ts_k128_halves_warp(tdK, tdPt, dQmn0 + static_cast<uint64_t>(m % kQStages) * kStep, idesc_acc,
                                m > 0 ? 1u : 0u);
        mma_commit_warp(bar(KV_Q_EMPTY + m % kQStages));
      };
      int ntiles = 0;
      for_each_q_tile(g, src, s_begin, s_end, kpos0, hi_max, jh, [&](int, int, int, int, int) { ++ntiles; });
      bool ok = warp_all(mbar_wait(bar(KV_FULL), 0, abort_flag, status));
      for (int n = 0; ok && n < ntiles; ++n) {
        const int qs = n % kQStages, ds = n % kDOStages;
        const uint32_t q_par = (n / kQStages) & 1, prev = (n - 1) & 1;
        if (!warp_all(n >= 1 ? mbar_try_wait2(bar(KV_P_FULL), prev, bar(KV_QD_FULL + qs), q_par)
                             : mbar_try_wait(bar(KV_QD_FULL + qs), q_par)))
          ok = (n < 1 || warp_all(mbar_wait(bar(KV_P_FULL), prev, abort_flag, status))) &&
               warp_all(mbar_wait(bar(KV_QD_FULL + qs), q_par, abort_flag, status));
        if (!ok) break;
        tc_fence_after();
        if (n > 0) issue_dv(n - 1);
        mma_qk<D>(tSt, dK0, dQ0 + static_cast<uint64_t>(qs) * kStep, idesc_s);
        mma_commit_warp(bar(KV_S_FULL));
        if (n > 0) {
          if (!(ok = warp_all(mbar_wait(bar(KV_DS_FULL), prev, abort_flag, status)))) break;
          tc_fence_after();
          issue_dk(n - 1);
        }
        mma_qk<D>(tdPt, dV0, dDO0 + static_cast<uint64_t>(ds) * kStep, idesc_s);
        mma_commit_warp(bar(KV_DP_FULL));
      }
      // dV and dK of the last query tile.
      if (ok && ntiles > 0 && warp_all(mbar_wait(bar(KV_P_FULL), (ntiles - 1) & 1, abort_flag, status))) {
        tc_fence_after();
        issue_dv(ntiles - 1);
        if (warp_all(mbar_wait(bar(KV_DS_FULL), (ntiles - 1) & 1, abort_flag, status))) {
          tc_fence_after();
          issue_dk(ntiles - 1);
          mma_commit_warp(bar(KV_ACC_DONE));
        }
      }
      mma_commit_warp(bar(KV_DRAIN));
      mbar_wait(bar(KV_DRAIN), 0, nullptr, status);
    }
  } else {
    const int wq = warp & 3;
    const int half = (warp - 2) >> 2;  // warps 2-5: query columns 0-63; warps 6-9: 64-127
    const int row = wq * 32 + lane;     // key row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const bool key_valid = row < it.len;
    const int kpos = kpos0 + row;
    const int hi_k = key_valid ? (g.doc_end ? g.doc_end[kpos] - 1 : g.L - 1) : -1;
    const float sl2 = g.scale * kLog2e;
    int n = 0;
    bool ok = true;
    auto process = [&](int qpos0, int qlen, uint32_t aLse, uint32_t aDel) {
      if (!ok) return;
      ok = warp_all(mbar_wait(bar(KV_S_FULL), n & 1, abort_flag, status));
      if (!ok) return;
      tc_fence_after();
      const bool full = (it.len == BN) && (qlen == BM) && (kpos_last <= qpos0) && (qpos0 + BM - 1 <= hi_min);
      const int c_lo = key_valid ? kpos - qpos0 : BM;
      const int c_hi = min(hi_k - qpos0, qlen - 1);
      // Phase A: P^T = exp2(S^T * scale*log2e - LSE*log2e), masked, packed to
      // bf16 pairs and written back over the S^T columns this warp has read
      // (32-column chunk cc of this half -> columns 64*half + 16*cc ..).
      float pf[BM / 2];  // P^T of this half of the row, fp32 (dS^T is formed from it)
      const f32x2 nsl2 = make_f32x2(sl2, sl2);
      uint32_t sr2[2][32];  // both chunks of this half: one TMEM round trip
      tmem_ld32(tSt + lane_off + 64 * half, sr2[0]);
      tmem_ld32(tSt + lane_off + 64 * half + 32, sr2[1]);
      tmem_wait_ld();
      reg_fence(sr2[0]);
      reg_fence(sr2[1]);
      // Two instantiations, as in the dQ kernel: no mask code on whole tiles.
      auto phase_a = [&](auto masked) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c4 = 2 * half + cc;
          const uint32_t* sr = sr2[cc];
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int col = c4 * 32 + e;
            const float2 nl = ld_shared_f32x2(aLse + 4 * col);  // -LSE * log2(e) of query columns col, col+1
            const f32x2 y = fma_f32x2(make_f32x2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), nsl2,
                                      make_f32x2(nl.x, nl.y));
            float y0, y1;
            split_f32x2(y, y0, y1);
            float x0 = ex2_approx(y0), x1 = ex2_approx(y1);
            if constexpr (decltype(masked)::value) {
              if (col < c_lo || col > c_hi) x0 = 0.f;
              if (col + 1 < c_lo || col + 1 > c_hi) x1 = 0.f;
            }
            pk[e / 2] = pack_bf16x2(x0, x1);
            pf[cc * 32 + e] = x0;
            pf[cc * 32 + e + 1] = x1;
          }
          tmem_st16(tSt + lane_off + 64 * half + 16 * cc, pk);
        }
      };
      if (full)
        phase_a(std::false_type{});
      else
        phase_a(std::true_type{});
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(KV_P_FULL));
      // Phase B: dS^T = P^T * (dP^T - D), packed to bf16 pairs over the dP^T
      // columns this warp has read (same column map as P^T).
      ok = warp_all(mbar_wait(bar(KV_DP_FULL), n & 1, abort_flag, status));
      if (!ok) return;
      tc_fence_after();
      uint32_t pr2[2][32];
      tmem_ld32(tdPt + lane_off + 64 * half, pr2[0]);
      tmem_ld32(tdPt + lane_off + 64 * half + 32, pr2[1]);
      tmem_wait_ld();
      reg_fence(pr2[0]);
      reg_fence(pr2[1]);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c4 = 2 * half + cc;
        const uint32_t* pr = pr2[cc];
        uint32_t dsp[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int col = c4 * 32 + e;
          const float2 nd = ld_shared_f32x2(aDel + 4 * col);  // -D of query columns col, col+1
          const f32x2 dd = add_f32x2(make_f32x2(__uint_as_float(pr[e]), __uint_as_float(pr[e + 1])),
                                     make_f32x2(nd.x, nd.y));
          float s0, s1;
          split_f32x2(mul_f32x2(make_f32x2(pf[cc * 32 + e], pf[cc * 32 + e + 1]), dd), s0, s1);
          dsp[e / 2] = pack_bf16x2(s0, s1);
        }
        tmem_st16(tdPt + lane_off + 64 * half + 16 * cc, dsp);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(KV_DS_FULL));
      ++n;
    };
    // Query tiles arrive from the producer warp: buffer n & 1 holds the
    // tile's -LSE*log2(e), -D, first position and length (length 0 ends the
    // walk).  Each warp hands the buffer back once it has finished the tile.
    while (ok) {
      const int ls = n & 1;
      if (!(ok = warp_all(mbar_wait(bar(KV_LD_FULL + ls), (n >> 1) & 1, abort_flag, status)))) break;
      const int qpos0 = sMeta[2 * ls], qlen = sMeta[2 * ls + 1];
      if (qlen == 0) break;
      const uint32_t aL = aLD + ls * 1024;
      process(qpos0, qlen, aL, aL + 512);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(KV_LD_EMPTY + ls));
    }
    if (ok && n > 0) {
      ok = warp_all(mbar_wait(bar(KV_ACC_DONE), 0, abort_flag, status));
      if (ok) tc_fence_after();
    }
    // Accumulate mode adds to dK and dV (nothing to add when no query tile was seen).
    if (ok && !(args.accumulate && n == 0)) {
      const size_t orow = (static_cast<size_t>(k_row0 + it.q0 + row) * (seq_io ? Hkv * g.U : Hkv) +
                           (seq_io ? u * Hkv + jh : jh)) * D;
      const bool store_ok = !key_valid || CP_IN_BOUNDS(k_row0 + it.q0 + row < rows, status);
      for (int c4 = half * (D / 64); c4 < (half + 1) * (D / 64); ++c4) {
        uint32_t v[32], k[32];
        if (n > 0) {
          tmem_ld32(tdV + lane_off + c4 * 32, v);
          tmem_ld32(tdK + lane_off + c4 * 32, k);
          tmem_wait_ld();
          reg_fence(v);
          reg_fence(k);
        }
        if (!key_valid || !store_ok) continue;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          float4 fv = make_float4(0.f, 0.f, 0.f, 0.f), fk = fv;
          if (n > 0) {
            fv = make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]),
                             __uint_as_float(v[e + 3]));
            fk = make_float4(__uint_as_float(k[e]) * g.scale, __uint_as_float(k[e + 1]) * g.scale,
                             __uint_as_float(k[e + 2]) * g.scale, __uint_as_float(k[e + 3]) * g.scale);
          }
          float4* pv = reinterpret_cast<float4*>(args.dv + orow + c4 * 32 + e);
          float4* pk = reinterpret_cast<float4*>(args.dk + orow + c4 * 32 + e);
          if (args.accumulate) {
            const float4 ov = *pv, ok4 = *pk;
            fv.x += ov.x;
            fv.y += ov.y;
            fv.z += ov.z;
            fv.w += ov.w;
            fk.x += ok4.x;
            fk.y += ok4.y;
            fk.z += ok4.z;
            fk.w += ok4.w;
          }
          *pv = fv;
          *pk = fk;
        }
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
int launch_bwd_d(const BwdArgs& a, cudaStream_t stream) {
  const AttnGeom& g = a.g;
  // Rows of every tensor: all ranks' slots, or (one ring step) one rank's
  // and one chunk's T rows.
  const uint64_t rows = a.rank_local ? static_cast<uint64_t>(g.T) : static_cast<uint64_t>(g.R) * g.U * g.T;
  const int phases = a.phases ? a.phases : 7;
  // With seq_io the maps span the sequence-sharded tensors: R*T rows of all heads.
  const uint64_t map_rows = a.seq_io ? static_cast<uint64_t>(g.R) * g.T : rows;
  const uint64_t wq = static_cast<uint64_t>(g.Hq_loc) * (a.seq_io ? g.U : 1) * D;
  const uint64_t wkv = static_cast<uint64_t>(g.Hkv_loc) * (a.seq_io ? g.U : 1) * D;
  CUtensorMap mq, mdo, mk, mv;
  if (!make_tile_map(&mq, a.q, wq, map_rows) || !make_tile_map(&mdo, a.dO, wq, map_rows) ||
      !make_tile_map(&mk, a.k, wkv, map_rows) || !make_tile_map(&mv, a.v, wkv, map_rows))
    return CP_ERR_CUDA;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(attn_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DqSmem<D>::kBytes) != cudaSuccess ||
        cudaFuncSetAttribute(attn_bwd_dkv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DkvSmem<D>::kBytes) != cudaSuccess)
      return CP_ERR_CUDA;
    attr_set = true;
  }
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (phases & 1) {
    const long long warps = static_cast<long long>(rows / g.T) * g.Hq_loc * ((g.T + 31) / 32);
    long long grid = (warps * 32 + 255) / 256;
    if (grid > sms * 16LL) grid = sms * 16LL;
    if (grid > 0 && a.o_fp32)
      bwd_delta_kernel<D, float><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
          static_cast<const float*>(a.o), static_cast<const __nv_bfloat16*>(a.dO), a.lse, a.nlse, a.nd, g,
          a.chunk_pad, static_cast<long long>(rows), a.seq_io, a.status);
    else if (grid > 0)
      bwd_delta_kernel<D, __nv_bfloat16><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dO), a.lse, a.nlse, a.nd, g,
          a.chunk_pad, static_cast<long long>(rows), a.seq_io, a.status);
  }
  const long long grid_kv = static_cast<long long>(a.n_items_kv) * g.Hkv_loc;
  const long long grid_q = static_cast<long long>(a.n_items_q) * g.Hq_loc;
  if (grid_kv > 0x7fffffffLL || grid_q > 0x7fffffffLL) return CP_ERR_UNSUPPORTED;
  if ((phases & 2) && grid_kv > 0)
    attn_bwd_dkv_kernel<D><<<static_cast<unsigned>(grid_kv), kThreads, DkvSmem<D>::kBytes, stream>>>(mq, mdo, mk,
                                                                                                      mv, a);
  if ((phases & 4) && grid_q > 0)
    attn_bwd_dq_kernel<D><<<static_cast<unsigned>(grid_q), kThreads, DqSmem<D>::kBytes, stream>>>(mq, mdo, mk, mv,
                                                                                                 a);
  return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

}  // namespace

int launch_attn_bwd(const BwdArgs& a, cudaStream_t stream) {
  if (a.d == 128) return launch_bwd_d<128>(a, stream);
  if (a.d == 64) return launch_bwd_d<64>(a, stream);
  return CP_ERR_UNSUPPORTED;
}

}  // namespace cpattn
