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
//            query tile of every ring rank (ring order: the chunk of rank
//            src visits ranks src, src+1, ...) and every query head of the
//            group; S^T = K Q^T and dP^T = V dO^T in TMEM, P^T and dS^T
//            through shared memory, dV and dK accumulated in TMEM
//   dq       one CTA per 128-query tile and head: walks the visible key
//            tiles in ring order like the forward; S = Q K^T and
//            dP = dO V^T in TMEM, dS through shared memory, dQ in TMEM
// Gradients of a KV chunk land on the rank that owns the chunk ([MTX]
// nougat.kr "MaxText long-context training and KV parallelism", "Split heads
// or rotate KV": the chunk's partial results travel with it).
//
// The kernels read the head-sharded layout of the Ulysses exchange (rank
// a = r*U + u holds ring rank r's slots for head group u; U == 1 is plain
// sequence sharding); the ring runs over r within each head group.
//
// Warp roles as in the forward: warp 0 TMA producer, warp 1 TMEM allocator
// and MMA issuer, warps 2..5 element-wise (one TMEM lane = one row each).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace cpattn {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr uint32_t HALF_BYTES = 128 * 128;
constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ bool warp_all(bool x) { return __all_sync(0xffffffffu, x); }

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Store 32 fp32 values as bf16 into a 128-row, K-major, 128-byte-swizzled
// tile (two 64-column halves of HALF_BYTES), row `row`, columns
// [32*c4, 32*c4+32).
__device__ __forceinline__ void store_row32_bf16(uint32_t tile, int row, int c4, const float* x) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int ch = c4 * 4 + q;  // 16-byte chunk: 8 columns
    const uint32_t addr = tile + row * 128 + (ch >> 3) * HALF_BYTES + (((ch & 7) ^ (row & 7)) << 4);
    st_shared_v4(addr, pack_bf16x2(x[8 * q + 0], x[8 * q + 1]), pack_bf16x2(x[8 * q + 2], x[8 * q + 3]),
                 pack_bf16x2(x[8 * q + 4], x[8 * q + 5]), pack_bf16x2(x[8 * q + 6], x[8 * q + 7]));
  }
}

__device__ __forceinline__ void store_row32_packed(uint32_t tile, int row, int c4, const uint32_t* p) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int ch = c4 * 4 + q;
    const uint32_t addr = tile + row * 128 + (ch >> 3) * HALF_BYTES + (((ch & 7) ^ (row & 7)) << 4);
    st_shared_v4(addr, p[4 * q + 0], p[4 * q + 1], p[4 * q + 2], p[4 * q + 3]);
  }
}

// Q K^T-type product over d: A and B both K-major, 128-byte swizzled.
template <int D>
__device__ __forceinline__ void mma_qk(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc) {
  if constexpr (D == 128)
    mma_bf16_ss_k128<HALF_BYTES>(d_tmem, a, b, idesc, 0u);
  else
    mma_bf16_ss_k64(d_tmem, a, b, idesc, 0u);
}

// ---------------------------------------------------------------- D = rowsum(dO * O)

__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(float x) { return x; }

template <int D, typename OT>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const OT* __restrict__ o,
                                                        const __nv_bfloat16* __restrict__ dO,
                                                        float* __restrict__ delta, long long rows, int H, int T) {
  constexpr int E = D / 32;  // elements per lane
  const int lane = threadIdx.x & 31;
  const long long total = rows * H;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long wi = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; wi < total; wi += nwarps) {
    const long long row = wi / H;
    const int h = static_cast<int>(wi - row * H);
    const OT* po = o + wi * D + lane * E;
    const __nv_bfloat16* pd = dO + wi * D + lane * E;
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc = fmaf(to_f32(po[e]), __bfloat162float(pd[e]), acc);
#pragma unroll
    for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      const long long r = row / T, t = row - r * T;
      delta[(r * H + h) * T + t] = acc;
    }
  }
}

// ---------------------------------------------------------------- dQ (query-tile outer)

enum DqBar { DQ_QD_FULL = 0, DQ_K_FULL = 1, DQ_K_EMPTY = 3, DQ_V_FULL = 5, DQ_V_EMPTY = 7, DQ_S_FULL = 9,
             DQ_S_EMPTY = 11, DQ_DP_FULL = 13, DQ_DS_FREE = 14, DQ_DS_FULL = 15, DQ_DONE = 16, DQ_DRAIN = 17,
             DQ_NUM_BARS = 18 };

template <int D>
struct DqSmem {
  static constexpr uint32_t kT = 128 * D * 2;
  static constexpr uint32_t kP = 128 * 128 * 2;
  static constexpr uint32_t offQ = 0, offDO = kT, offK = 2 * kT, offV = 4 * kT, offDS = 6 * kT;
  static constexpr uint32_t offBar = offDS + kP;
  static constexpr uint32_t offMisc = offBar + DQ_NUM_BARS * 8;
  static constexpr uint32_t kUsed = offMisc + 16;
  static constexpr uint32_t kBytes = (kUsed + 1024 < 120 * 1024) ? 120 * 1024 : kUsed + 1024;
};

template <typename F>
__device__ __forceinline__ void for_each_kv_tile(const AttnGeom& g, int r, int u, int lo_min, int qpos_last, F&& f) {
  const int nchunks = g.nchunks;
  for (int s = 0; s < g.R; ++s) {
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
  const uint32_t sQ = s_base + SM::offQ, sDO = s_base + SM::offDO, sK = s_base + SM::offK, sV = s_base + SM::offV,
                 sDS = s_base + SM::offDS;
  auto bar = [&](int i) { return s_base + SM::offBar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::offMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM::offMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttnGeom& g = args.g;
  int32_t* status = args.status;
  const int Hq = g.Hq_loc;
  const WorkItem it = args.items_q[blockIdx.x / Hq];
  const int h = blockIdx.x % Hq;
  const int a = it.a, r = a / g.U, u = a % g.U;  // rank a = ring rank r, Ulysses member u
  const int qpos0 = slot_pos(g, r, it.q0);
  const int qpos_last = qpos0 + it.len - 1;
  const int lo_min = g.doc_start ? g.doc_start[qpos0] : 0;
  const int lo_max = g.doc_start ? g.doc_start[qpos_last] : 0;
  const int hkv = h / g.G;

  if (threadIdx.x == 0) {
    mbar_init(bar(DQ_QD_FULL), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(DQ_K_FULL + i), 1);
      mbar_init(bar(DQ_K_EMPTY + i), 1);
      mbar_init(bar(DQ_V_FULL + i), 1);
      mbar_init(bar(DQ_V_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(DQ_S_FULL + i), 1);
      mbar_init(bar(DQ_S_EMPTY + i), 4);
    }
    mbar_init(bar(DQ_DP_FULL), 1);
    mbar_init(bar(DQ_DS_FREE), 1);
    mbar_init(bar(DQ_DS_FULL), 4);
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
  // TMEM: S double-buffered (columns 0 and 384), dP at 128, dQ at 256.
  const uint32_t tdP = tmem + 128, tdQ = tmem + 256;
  auto tS = [&](int b) { return tmem + (b ? 384u : 0u); };

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(DQ_QD_FULL), 2 * SM::kT);
      const int qrow = a * g.T + it.q0;
      for (int hh = 0; hh < NH; ++hh) {
        tma_load_2d(sQ + hh * HALF_BYTES, &tm_q, bar(DQ_QD_FULL), h * D + hh * 64, qrow);
        tma_load_2d(sDO + hh * HALF_BYTES, &tm_do, bar(DQ_QD_FULL), h * D + hh * 64, qrow);
      }
      int nk = 0, nv = 0;
      for_each_kv_tile(g, r, u, lo_min, qpos_last, [&](int kv_row, int, int) {
        if (*abort_flag) return;
        const int st = nk & 1;
        const uint32_t ph = ((nk >> 1) & 1) ^ 1;
        if (!mbar_wait(bar(DQ_K_EMPTY + st), ph, abort_flag, status)) return;
        mbar_arrive_expect_tx(bar(DQ_K_FULL + st), SM::kT);
        for (int hh = 0; hh < NH; ++hh)
          tma_load_2d(sK + st * SM::kT + hh * HALF_BYTES, &tm_k, bar(DQ_K_FULL + st), hkv * D + hh * 64, kv_row);
        ++nk;
        if (!mbar_wait(bar(DQ_V_EMPTY + st), ph, abort_flag, status)) return;
        mbar_arrive_expect_tx(bar(DQ_V_FULL + st), SM::kT);
        for (int hh = 0; hh < NH; ++hh)
          tma_load_2d(sV + st * SM::kT + hh * HALF_BYTES, &tm_v, bar(DQ_V_FULL + st), hkv * D + hh * 64, kv_row);
        ++nv;
      });
      if (*abort_flag) {
        mbar_wait(bar(DQ_QD_FULL), 0, nullptr, status);
        for (int i = max(0, nk - 2); i < nk; ++i) mbar_wait(bar(DQ_K_FULL + (i & 1)), (i >> 1) & 1, nullptr, status);
        for (int i = max(0, nv - 2); i < nv; ++i) mbar_wait(bar(DQ_V_FULL + (i & 1)), (i >> 1) & 1, nullptr, status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, 0);
      constexpr uint32_t idesc_dq = idesc_bf16_f32(BM, D, 1);
      // Descriptors built once; stage st adds st * tile bytes (>> 4).
      const uint64_t dQ0 = smem_desc_sw128(sQ, 16, 1024), dDO0 = smem_desc_sw128(sDO, 16, 1024);
      const uint64_t dK0 = smem_desc_sw128(sK, 16, 1024), dV0 = smem_desc_sw128(sV, 16, 1024);
      const uint64_t dKmn0 = smem_desc_sw128(sK, HALF_BYTES, 1024), dDS = smem_desc_sw128(sDS, 16, 1024);
      constexpr uint64_t kStep = SM::kT >> 4;  // one K/V stage in descriptor units
      // Issue order for key tile n: S_n (into S buffer n & 1), dP_n, dQ_{n-1}.
      // S_n only needs the element-wise warps to have read S_{n-2}, so it is
      // queued while they still work on tile n-1.
      int n = 0;
      if (mbar_wait(bar(DQ_QD_FULL), 0, abort_flag, status)) {
        for_each_kv_tile(g, r, u, lo_min, qpos_last, [&](int, int, int) {
          if (*abort_flag) return;
          const int st = n & 1;
          const uint32_t ph = (n >> 1) & 1;
          const uint64_t step = static_cast<uint64_t>(st) * kStep, pstep = static_cast<uint64_t>(st ^ 1) * kStep;
          if (!mbar_wait(bar(DQ_K_FULL + st), ph, abort_flag, status)) return;
          if (n >= 2 && !mbar_wait(bar(DQ_S_EMPTY + st), ph ^ 1, abort_flag, status)) return;
          tc_fence_after();
          mma_qk<D>(tS(st), dQ0, dK0 + step, idesc_s);
          mma_commit(bar(DQ_S_FULL + st));
          if (!mbar_wait(bar(DQ_V_FULL + st), ph, abort_flag, status)) return;
          // DS_FULL: dS_{n-1} is in shared memory and the dP columns are free.
          if (n > 0 && !mbar_wait(bar(DQ_DS_FULL), (n - 1) & 1, abort_flag, status)) return;
          tc_fence_after();
          mma_qk<D>(tdP, dDO0, dV0 + step, idesc_s);
          mma_commit(bar(DQ_DP_FULL));
          mma_commit(bar(DQ_V_EMPTY + st));
          if (n > 0) {
            // A = dS [queries x keys] K-major; B = K [keys x d] read as N=d x K=keys (MN-major).
            mma_bf16_ss_k128_bmn<HALF_BYTES>(tdQ, dDS, dKmn0 + pstep, idesc_dq, n > 1 ? 1u : 0u);
            mma_commit(bar(DQ_DS_FREE));
            mma_commit(bar(DQ_K_EMPTY + (st ^ 1)));
          }
          ++n;
        });
        if (n > 0 && !*abort_flag) {
          if (mbar_wait(bar(DQ_DS_FULL), (n - 1) & 1, abort_flag, status)) {
            tc_fence_after();
            const uint64_t pstep = static_cast<uint64_t>((n - 1) & 1) * kStep;
            mma_bf16_ss_k128_bmn<HALF_BYTES>(tdQ, dDS, dKmn0 + pstep, idesc_dq, n > 1 ? 1u : 0u);
            mma_commit(bar(DQ_DS_FREE));
            mma_commit(bar(DQ_K_EMPTY + ((n - 1) & 1)));
            mma_commit(bar(DQ_DONE));
          }
        }
      }
      mma_commit(bar(DQ_DRAIN));
      mbar_wait(bar(DQ_DRAIN), 0, nullptr, status);
    }
  } else {
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const bool row_valid = row < it.len;
    const int my_pos = row_valid ? qpos0 + row : -1;
    const int my_lo = (row_valid && g.doc_start) ? g.doc_start[my_pos] : 0;
    const size_t lrow = (static_cast<size_t>(a) * Hq + h) * g.T + it.q0 + row;
    const float lse2 = row_valid ? args.lse[lrow] * kLog2e : INFINITY;
    const float dlt = row_valid ? args.delta[lrow] : 0.f;
    const float sl2 = g.scale * kLog2e;
    int n = 0;
    bool ok = true;
    for_each_kv_tile(g, r, u, lo_min, qpos_last, [&](int, int kpos0, int klen) {
      if (!ok) return;
      const int sb = n & 1;
      ok = warp_all(mbar_wait(bar(DQ_S_FULL + sb), (n >> 1) & 1, abort_flag, status));
      if (!ok) return;
      tc_fence_after();
      const bool full = (klen == BN) && (kpos0 + BN - 1 <= qpos0) && (lo_max <= kpos0);
      const int c_lo = my_lo - kpos0;
      const int c_hi = min(my_pos - kpos0, klen - 1);
      // Phase A: P = exp2(S * scale*log2e - LSE*log2e), masked, as packed bf16.
      uint32_t pp[BN / 2];
      const f32x2 nsl2 = make_f32x2(sl2, sl2), nlse2 = make_f32x2(-lse2, -lse2);
#pragma unroll
      for (int c4 = 0; c4 < BN / 32; ++c4) {
        uint32_t sr[32];
        tmem_ld32(tS(sb) + lane_off + c4 * 32, sr);
        tmem_wait_ld();
        reg_fence(sr);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int col = c4 * 32 + e;
          const f32x2 y = fma_f32x2(make_f32x2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), nsl2, nlse2);
          float y0, y1;
          split_f32x2(y, y0, y1);
          float x0 = ex2_approx(y0), x1 = ex2_approx(y1);
          if (!full) {
            if (col < c_lo || col > c_hi) x0 = 0.f;
            if (col + 1 < c_lo || col + 1 > c_hi) x1 = 0.f;
          }
          pp[c4 * 16 + e / 2] = pack_bf16x2(x0, x1);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(DQ_S_EMPTY + sb));
      // Phase B: dS = P * (dP - D) as packed bf16, parked in the dP columns
      // already read (32-column chunk c4 lands in columns 16c4..).
      ok = warp_all(mbar_wait(bar(DQ_DP_FULL), n & 1, abort_flag, status));
      if (!ok) return;
      tc_fence_after();
#pragma unroll
      for (int c4 = 0; c4 < BN / 32; ++c4) {
        uint32_t pr[32], dsp[16];
        tmem_ld32(tdP + lane_off + c4 * 32, pr);
        tmem_wait_ld();
        reg_fence(pr);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const uint32_t pk = pp[c4 * 16 + e / 2];
          const f32x2 dd = add_f32x2(make_f32x2(__uint_as_float(pr[e]), __uint_as_float(pr[e + 1])),
                                     make_f32x2(-dlt, -dlt));
          float d0, d1;
          split_f32x2(dd, d0, d1);
          dsp[e / 2] = pack_bf16x2(__uint_as_float(pk << 16) * d0, __uint_as_float(pk & 0xffff0000u) * d1);
        }
        tmem_st16(tdP + lane_off + c4 * 16, dsp);
      }
      tmem_wait_st();
      // dS into shared memory once dQ of the previous key tile has read it.
      if (n > 0) {
        ok = warp_all(mbar_wait(bar(DQ_DS_FREE), (n - 1) & 1, abort_flag, status));
        if (!ok) return;
      }
#pragma unroll
      for (int c4 = 0; c4 < BN / 32; ++c4) {
        uint32_t dsp[16];
        tmem_ld16(tdP + lane_off + c4 * 16, dsp);
        tmem_wait_ld();
        reg_fence16(dsp);
        store_row32_packed(sDS, row, c4, dsp);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(DQ_DS_FULL));
      ++n;
    });
    if (ok && n > 0) {
      ok = warp_all(mbar_wait(bar(DQ_DONE), 0, abort_flag, status));
      if (ok) tc_fence_after();
    }
    if (ok) {
      float* dst = args.dq + (static_cast<size_t>(a * g.T + it.q0 + row) * Hq + h) * D;
      for (int c4 = 0; c4 < D / 32; ++c4) {
        uint32_t v[32];
        if (n > 0) {
          tmem_ld32(tdQ + lane_off + c4 * 32, v);
          tmem_wait_ld();
          reg_fence(v);
        }
        if (!row_valid) continue;
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(dst + c4 * 32 + e) =
              n > 0 ? make_float4(__uint_as_float(v[e]) * g.scale, __uint_as_float(v[e + 1]) * g.scale,
                                  __uint_as_float(v[e + 2]) * g.scale, __uint_as_float(v[e + 3]) * g.scale)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
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

enum DkvBar { KV_FULL = 0, KV_QD_FULL = 1, KV_QD_EMPTY = 3, KV_S_FULL = 5, KV_DP_FULL = 6, KV_ST_EMPTY = 7,
              KV_P_FULL = 8, KV_PB_FREE = 9, KV_DS_FULL = 10, KV_SPB_FREE = 11, KV_ACC_DONE = 12, KV_DRAIN = 13,
              KV_NUM_BARS = 14 };

template <int D>
struct DkvSmem {
  static constexpr uint32_t kT = 128 * D * 2;
  static constexpr uint32_t kP = 128 * 128 * 2;
  static constexpr uint32_t offK = 0, offV = kT, offQ = 2 * kT, offDO = 4 * kT, offPB = 6 * kT;
  static constexpr uint32_t offBar = offPB + kP;
  static constexpr uint32_t offLD = offBar + KV_NUM_BARS * 8;   // 128 lse2 + 128 delta floats
  static constexpr uint32_t offMisc = offLD + 2 * 128 * 4;
  static constexpr uint32_t kUsed = offMisc + 16;
  static constexpr uint32_t kBytes = (kUsed + 1024 < 120 * 1024) ? 120 * 1024 : kUsed + 1024;
};

// Every query tile (of every ring rank, in ring order from the owner) and
// every query head of KV head jh that may see the key tile [kpos0, hi_max].
template <typename F>
__device__ __forceinline__ void for_each_q_tile(const AttnGeom& g, int src, int kpos0, int hi_max, int jh, F&& f) {
  const int nchunks = g.nchunks;
  for (int s = 0; s < g.R; ++s) {
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
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sK = s_base + SM::offK, sV = s_base + SM::offV, sQ = s_base + SM::offQ, sDO = s_base + SM::offDO,
                 sPB = s_base + SM::offPB;
  auto bar = [&](int i) { return s_base + SM::offBar + 8u * i; };
  float* sLse = reinterpret_cast<float*>(smem + SM::offLD);
  float* sDel = sLse + 128;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::offMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM::offMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttnGeom& g = args.g;
  int32_t* status = args.status;
  const int Hkv = g.Hkv_loc, Hq = g.Hq_loc;
  const WorkItem it = args.items_kv[blockIdx.x / Hkv];
  const int jh = blockIdx.x % Hkv;
  const int a = it.a, src = a / g.U, u = a % g.U;  // key tile of rank a = ring rank src, member u
  const int kpos0 = slot_pos(g, src, it.q0);
  const int kpos_last = kpos0 + it.len - 1;
  const int hi_max = g.doc_end ? g.doc_end[kpos_last] - 1 : g.L - 1;
  const int hi_min = g.doc_end ? g.doc_end[kpos0] - 1 : g.L - 1;

  if (threadIdx.x == 0) {
    mbar_init(bar(KV_FULL), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(KV_QD_FULL + i), 1);
      mbar_init(bar(KV_QD_EMPTY + i), 1);
    }
    mbar_init(bar(KV_S_FULL), 1);
    mbar_init(bar(KV_DP_FULL), 1);
    mbar_init(bar(KV_ST_EMPTY), 4);
    mbar_init(bar(KV_P_FULL), 4);
    mbar_init(bar(KV_PB_FREE), 1);
    mbar_init(bar(KV_DS_FULL), 4);
    mbar_init(bar(KV_SPB_FREE), 1);
    mbar_init(bar(KV_ACC_DONE), 1);
    mbar_init(bar(KV_DRAIN), 1);
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
  const uint32_t tSt = tmem, tdPt = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(KV_FULL), 2 * SM::kT);
      const int krow = a * g.T + it.q0;
      for (int hh = 0; hh < NH; ++hh) {
        tma_load_2d(sK + hh * HALF_BYTES, &tm_k, bar(KV_FULL), jh * D + hh * 64, krow);
        tma_load_2d(sV + hh * HALF_BYTES, &tm_v, bar(KV_FULL), jh * D + hh * 64, krow);
      }
      int nq = 0;
      for_each_q_tile(g, src, kpos0, hi_max, jh, [&](int rr, int qslot0, int, int, int h) {
        if (*abort_flag) return;
        const int st = nq & 1;
        const uint32_t ph = ((nq >> 1) & 1) ^ 1;
        if (!mbar_wait(bar(KV_QD_EMPTY + st), ph, abort_flag, status)) return;
        mbar_arrive_expect_tx(bar(KV_QD_FULL + st), 2 * SM::kT);
        const int qrow = (rr * g.U + u) * g.T + qslot0;
        for (int hh = 0; hh < NH; ++hh) {
          tma_load_2d(sQ + st * SM::kT + hh * HALF_BYTES, &tm_q, bar(KV_QD_FULL + st), h * D + hh * 64, qrow);
          tma_load_2d(sDO + st * SM::kT + hh * HALF_BYTES, &tm_do, bar(KV_QD_FULL + st), h * D + hh * 64, qrow);
        }
        ++nq;
      });
      if (*abort_flag) {
        mbar_wait(bar(KV_FULL), 0, nullptr, status);
        for (int i = max(0, nq - 2); i < nq; ++i) mbar_wait(bar(KV_QD_FULL + (i & 1)), (i >> 1) & 1, nullptr, status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, 0);
      constexpr uint32_t idesc_acc = idesc_bf16_f32(BM, D, 1);
      const uint64_t dK0 = smem_desc_sw128(sK, 16, 1024), dV0 = smem_desc_sw128(sV, 16, 1024);
      const uint64_t dQ0 = smem_desc_sw128(sQ, 16, 1024), dDO0 = smem_desc_sw128(sDO, 16, 1024);
      const uint64_t dQmn0 = smem_desc_sw128(sQ, HALF_BYTES, 1024), dDOmn0 = smem_desc_sw128(sDO, HALF_BYTES, 1024);
      const uint64_t dPB = smem_desc_sw128(sPB, 16, 1024);
      constexpr uint64_t kStep = SM::kT >> 4;  // one Q/dO stage in descriptor units
      // Issue order for query tile n: S_n, dV_{n-1}, dP_n, dK_{n-1}.  S_n only
      // waits for the element-wise warps to have read S_{n-1} (phase A), so
      // it runs while they compute dS_{n-1}; dP_n, dV_{n-1} and dK_{n-1} run
      // while they compute P_n.
      int n = 0;
      if (mbar_wait(bar(KV_FULL), 0, abort_flag, status)) {
        for_each_q_tile(g, src, kpos0, hi_max, jh, [&](int, int, int, int, int) {
          if (*abort_flag) return;
          const int st = n & 1;
          const uint64_t step = static_cast<uint64_t>(st) * kStep, pstep = static_cast<uint64_t>(st ^ 1) * kStep;
          if (!mbar_wait(bar(KV_QD_FULL + st), (n >> 1) & 1, abort_flag, status)) return;
          if (n > 0 && !mbar_wait(bar(KV_ST_EMPTY), (n - 1) & 1, abort_flag, status)) return;
          tc_fence_after();
          mma_qk<D>(tSt, dK0, dQ0 + step, idesc_s);
          mma_commit(bar(KV_S_FULL));
          if (n > 0) {
            // A = P^T [keys x queries] K-major; B = dO [queries x d] as N=d x K=queries (MN-major).
            if (!mbar_wait(bar(KV_P_FULL), (n - 1) & 1, abort_flag, status)) return;
            tc_fence_after();
            mma_bf16_ss_k128_bmn<HALF_BYTES>(tdV, dPB, dDOmn0 + pstep, idesc_acc, n > 1 ? 1u : 0u);
            mma_commit(bar(KV_PB_FREE));
          }
          // DS_FULL: dS^T_{n-1} is in shared memory and the dP^T columns are free.
          if (n > 0 && !mbar_wait(bar(KV_DS_FULL), (n - 1) & 1, abort_flag, status)) return;
          tc_fence_after();
          mma_qk<D>(tdPt, dV0, dDO0 + step, idesc_s);
          mma_commit(bar(KV_DP_FULL));
          if (n > 0) {
            mma_bf16_ss_k128_bmn<HALF_BYTES>(tdK, dPB, dQmn0 + pstep, idesc_acc, n > 1 ? 1u : 0u);
            mma_commit(bar(KV_SPB_FREE));
            mma_commit(bar(KV_QD_EMPTY + (st ^ 1)));
          }
          ++n;
        });
        // dV and dK of the last query tile.
        if (n > 0 && !*abort_flag) {
          const uint64_t pstep = static_cast<uint64_t>((n - 1) & 1) * kStep;
          if (mbar_wait(bar(KV_P_FULL), (n - 1) & 1, abort_flag, status)) {
            tc_fence_after();
            mma_bf16_ss_k128_bmn<HALF_BYTES>(tdV, dPB, dDOmn0 + pstep, idesc_acc, n > 1 ? 1u : 0u);
            mma_commit(bar(KV_PB_FREE));
            if (mbar_wait(bar(KV_DS_FULL), (n - 1) & 1, abort_flag, status)) {
              tc_fence_after();
              mma_bf16_ss_k128_bmn<HALF_BYTES>(tdK, dPB, dQmn0 + pstep, idesc_acc, n > 1 ? 1u : 0u);
              mma_commit(bar(KV_SPB_FREE));
              mma_commit(bar(KV_QD_EMPTY + ((n - 1) & 1)));
              mma_commit(bar(KV_ACC_DONE));
            }
          }
        }
      }
      mma_commit(bar(KV_DRAIN));
      mbar_wait(bar(KV_DRAIN), 0, nullptr, status);
    }
  } else {
    const int wq = warp & 3;
    const int row = wq * 32 + lane;  // key row of the tile
    const int etid = threadIdx.x - 64;  // 0..127 across the element-wise warps
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const bool key_valid = row < it.len;
    const int kpos = kpos0 + row;
    const int hi_k = key_valid ? (g.doc_end ? g.doc_end[kpos] - 1 : g.L - 1) : -1;
    const float sl2 = g.scale * kLog2e;
    int n = 0;
    bool ok = true;
    for_each_q_tile(g, src, kpos0, hi_max, jh, [&](int rr, int qslot0, int qpos0, int qlen, int h) {
      // Stage this query tile's LSE (log2 units) and D for all 128 columns.
      // Every element-wise warp walks the same tiles and reaches both
      // barriers on every tile, also after an abort, so they stay balanced.
      named_bar_sync(1, 128);  // everyone finished reading the previous tile's values
      {
        const size_t li = (static_cast<size_t>(rr * g.U + u) * Hq + h) * g.T + qslot0 + etid;
        sLse[etid] = etid < qlen ? args.lse[li] * kLog2e : INFINITY;
        sDel[etid] = etid < qlen ? args.delta[li] : 0.f;
      }
      named_bar_sync(1, 128);
      if (!ok) return;
      ok = warp_all(mbar_wait(bar(KV_S_FULL), n & 1, abort_flag, status));
      if (!ok) return;
      tc_fence_after();
      const bool full = (it.len == BN) && (qlen == BM) && (kpos_last <= qpos0) && (qpos0 + BM - 1 <= hi_min);
      const int c_lo = key_valid ? kpos - qpos0 : BM;
      const int c_hi = min(hi_k - qpos0, qlen - 1);
      // Phase A: P^T row = exp2(S^T * scale*log2e - LSE*log2e), masked,
      // kept as packed bf16 pairs (the operand dV reads, and the P of dS).
      uint32_t pp[BM / 2];
#pragma unroll
      for (int c4 = 0; c4 < BM / 32; ++c4) {
        uint32_t sr[32];
        tmem_ld32(tSt + lane_off + c4 * 32, sr);
        tmem_wait_ld();
        reg_fence(sr);
        const f32x2 nsl2 = make_f32x2(sl2, sl2);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int col = c4 * 32 + e;
          const f32x2 y = fma_f32x2(make_f32x2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), nsl2,
                                    make_f32x2(-sLse[col], -sLse[col + 1]));
          float y0, y1;
          split_f32x2(y, y0, y1);
          float x0 = ex2_approx(y0), x1 = ex2_approx(y1);
          if (!full) {
            if (col < c_lo || col > c_hi) x0 = 0.f;
            if (col + 1 < c_lo || col + 1 > c_hi) x1 = 0.f;
          }
          pp[c4 * 16 + e / 2] = pack_bf16x2(x0, x1);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(KV_ST_EMPTY));
      // P^T into shared memory once dK of the previous tile has read dS^T there.
      if (n > 0) {
        ok = warp_all(mbar_wait(bar(KV_SPB_FREE), (n - 1) & 1, abort_flag, status));
        if (!ok) return;
      }
#pragma unroll
      for (int c4 = 0; c4 < BM / 32; ++c4) store_row32_packed(sPB, row, c4, pp + c4 * 16);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(KV_P_FULL));
      // Phase B: dS^T = P^T * (dP^T - D) as packed bf16, parked in the dP^T
      // columns already read (32-column chunk c4 lands in columns 16c4..).
      ok = warp_all(mbar_wait(bar(KV_DP_FULL), n & 1, abort_flag, status));
      if (!ok) return;
      tc_fence_after();
#pragma unroll
      for (int c4 = 0; c4 < BM / 32; ++c4) {
        uint32_t pr[32], dsp[16];
        tmem_ld32(tdPt + lane_off + c4 * 32, pr);
        tmem_wait_ld();
        reg_fence(pr);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int col = c4 * 32 + e;
          const uint32_t pk = pp[c4 * 16 + e / 2];
          const f32x2 dd = add_f32x2(make_f32x2(__uint_as_float(pr[e]), __uint_as_float(pr[e + 1])),
                                     make_f32x2(-sDel[col], -sDel[col + 1]));
          float d0, d1;
          split_f32x2(dd, d0, d1);
          dsp[e / 2] = pack_bf16x2(__uint_as_float(pk << 16) * d0, __uint_as_float(pk & 0xffff0000u) * d1);
        }
        tmem_st16(tdPt + lane_off + c4 * 16, dsp);
      }
      tmem_wait_st();
      // dS^T over P^T once dV has read P^T.
      ok = warp_all(mbar_wait(bar(KV_PB_FREE), n & 1, abort_flag, status));
      if (!ok) return;
      tc_fence_after();
#pragma unroll
      for (int c4 = 0; c4 < BM / 32; ++c4) {
        uint32_t dsp[16];
        tmem_ld16(tdPt + lane_off + c4 * 16, dsp);
        tmem_wait_ld();
        reg_fence16(dsp);
        store_row32_packed(sPB, row, c4, dsp);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(KV_DS_FULL));
      ++n;
    });
    if (ok && n > 0) {
      ok = warp_all(mbar_wait(bar(KV_ACC_DONE), 0, abort_flag, status));
      if (ok) tc_fence_after();
    }
    if (ok) {
      const size_t orow = (static_cast<size_t>(a * g.T + it.q0 + row) * Hkv + jh) * D;
      for (int c4 = 0; c4 < D / 32; ++c4) {
        uint32_t v[32], k[32];
        if (n > 0) {
          tmem_ld32(tdV + lane_off + c4 * 32, v);
          tmem_ld32(tdK + lane_off + c4 * 32, k);
          tmem_wait_ld();
          reg_fence(v);
          reg_fence(k);
        }
        if (!key_valid) continue;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          float4 fv = make_float4(0.f, 0.f, 0.f, 0.f), fk = fv;
          if (n > 0) {
            fv = make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]),
                             __uint_as_float(v[e + 3]));
            fk = make_float4(__uint_as_float(k[e]) * g.scale, __uint_as_float(k[e + 1]) * g.scale,
                             __uint_as_float(k[e + 2]) * g.scale, __uint_as_float(k[e + 3]) * g.scale);
          }
          *reinterpret_cast<float4*>(args.dv + orow + c4 * 32 + e) = fv;
          *reinterpret_cast<float4*>(args.dk + orow + c4 * 32 + e) = fk;
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
  const uint64_t rows = static_cast<uint64_t>(g.R) * g.U * g.T;
  CUtensorMap mq, mdo, mk, mv;
  if (!make_tile_map(&mq, a.q, static_cast<uint64_t>(g.Hq_loc) * D, rows) ||
      !make_tile_map(&mdo, a.dO, static_cast<uint64_t>(g.Hq_loc) * D, rows) ||
      !make_tile_map(&mk, a.k, static_cast<uint64_t>(g.Hkv_loc) * D, rows) ||
      !make_tile_map(&mv, a.v, static_cast<uint64_t>(g.Hkv_loc) * D, rows))
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
  {
    const long long warps = rows * g.Hq_loc;
    long long grid = (warps * 32 + 255) / 256;
    if (grid > sms * 16LL) grid = sms * 16LL;
    if (grid > 0 && a.o_fp32)
      bwd_delta_kernel<D, float><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
          static_cast<const float*>(a.o), static_cast<const __nv_bfloat16*>(a.dO), a.delta,
          static_cast<long long>(rows), g.Hq_loc, g.T);
    else if (grid > 0)
      bwd_delta_kernel<D, __nv_bfloat16><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dO), a.delta,
          static_cast<long long>(rows), g.Hq_loc, g.T);
  }
  const long long grid_kv = static_cast<long long>(a.n_items_kv) * g.Hkv_loc;
  const long long grid_q = static_cast<long long>(a.n_items_q) * g.Hq_loc;
  if (grid_kv > 0x7fffffffLL || grid_q > 0x7fffffffLL) return CP_ERR_UNSUPPORTED;
  if (grid_kv > 0)
    attn_bwd_dkv_kernel<D><<<static_cast<unsigned>(grid_kv), kThreads, DkvSmem<D>::kBytes, stream>>>(mq, mdo, mk,
                                                                                                      mv, a);
  if (grid_q > 0)
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
