// merge.cu -- exact merge of normalised attention partials by their
// log-sum-exp ([MTX] nougat.kr "MaxText long-context training and KV
// parallelism", section "Split heads or rotate KV": ring attention computes
// a partial with each visiting KV chunk and merges the results).
//
// For one (row, head): m = max_p lse_p, lse = m + ln sum_p e^(lse_p - m),
// o = sum_p e^(lse_p - lse) o_p; all parts empty (-inf) => o = 0, lse = -inf.
// Parts are folded in index order (ring order).
//
// HBM-bound: each (row, head) reads n_parts * (4d + 4) bytes and writes
// 2d + 4 (bf16 O) or 4d + 4 (fp32 O).  One warp owns 32 consecutive rows of
// one head:
//   1. lane i takes row i: the LSE partials [p][h][row] are read 128 bytes
//      at a time, and lane i computes the merged LSE and the weights
//      e^(lse_p - lse) of its row for every part, parked in shared memory;
//   2. the warp then walks its rows: a row's d floats of one part are 4d
//      contiguous bytes (d/4 lanes, one float4 each; two rows per warp step
//      for d = 64), and each lane issues the loads of up to eight parts of
//      two such steps before it folds them.
// Consecutive warps take consecutive heads of the same rows, so together
// they sweep contiguous (row, head, d) ranges of every part.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#define CP_TU_ID ::cpattn::kTuMerge
#include "cp_attn.h"
#include "debug.cuh"
#include "kernels.h"

namespace cpattn {
namespace {

constexpr int kRows = 32;     // rows per warp unit
constexpr int kBatch = 8;     // parts whose loads are in flight together
constexpr int kMaxSmem = 96 * 1024;

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <int D>
__global__ void __launch_bounds__(256) merge_kernel(int n_parts, int rows, int H, const float* __restrict__ o_parts,
                                                    const float* __restrict__ lse_parts, void* __restrict__ o_out,
                                                    float* __restrict__ lse_out, int batch, int out_fp32,
                                                    int32_t* status) {
  constexpr int TPR = D / 4;         // lanes per row (one float4 each)
  constexpr int RPI = 32 / TPR;      // rows per warp iteration
  extern __shared__ float s_w[];     // [warps][n_parts][kRows] weights
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* w = s_w + static_cast<size_t>(warp) * n_parts * kRows;
  const long long per_batch = static_cast<long long>(rows) * H;
  const int row_blocks = (rows + kRows - 1) / kRows;
  const long long units = static_cast<long long>(batch) * row_blocks * H;
  const long long warps_total = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const int sub = lane / TPR, c4 = lane % TPR;
  for (long long un = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + warp; un < units; un += warps_total) {
    const int h = static_cast<int>(un % H);
    const long long x = un / H;
    const int rb = static_cast<int>(x % row_blocks);
    const int b = static_cast<int>(x / row_blocks);
    const int row0 = rb * kRows;
    const int nrow = min(kRows, rows - row0);
    if (!CP_IN_BOUNDS(b < batch && h < H && row0 < rows, status)) continue;
    // 1. merged LSE and per-part weights of row row0 + lane.
    {
      const int row = row0 + lane;
      const bool valid = lane < nrow;
      const float* lp =
          lse_parts + static_cast<long long>(b) * n_parts * per_batch + static_cast<long long>(h) * rows + row;
      float m = -INFINITY;
      if (valid)
        for (int p = 0; p < n_parts; ++p) m = fmaxf(m, __ldg(lp + p * per_batch));
      float lse = -INFINITY;
      if (m != -INFINITY) {
        float sum = 0.f;
        for (int p = 0; p < n_parts; ++p) sum += __expf(__ldg(lp + p * per_batch) - m);
        lse = m + __logf(sum);
      }
      for (int p = 0; p < n_parts; ++p)
        w[p * kRows + lane] = (m != -INFINITY) ? __expf(__ldg(lp + p * per_batch) - lse) : 0.f;
      if (valid) lse_out[static_cast<long long>(b) * per_batch + static_cast<long long>(h) * rows + row] = lse;
    }
    __syncwarp();
    // 2. O rows, 2 * RPI at a time (two row groups' loads in flight).
    const float* ob = o_parts + static_cast<long long>(b) * n_parts * per_batch * D;
    for (int j0 = 0; j0 < nrow; j0 += 2 * RPI) {
      int jj[2];
      bool in[2];
      long long off[2];
      float4 acc[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        jj[q] = j0 + q * RPI + sub;
        in[q] = jj[q] < nrow;
        off[q] = (static_cast<long long>(row0 + (in[q] ? jj[q] : 0)) * H + h) * D + c4 * 4;
        acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int p0 = 0; p0 < n_parts; p0 += kBatch) {
        float4 v[2][kBatch];
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int i = 0; i < kBatch; ++i)
            if (in[q] && p0 + i < n_parts)
              v[q][i] = __ldg(reinterpret_cast<const float4*>(ob + (p0 + i) * per_batch * D + off[q]));
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int i = 0; i < kBatch; ++i) {
            if (in[q] && p0 + i < n_parts) {
              const float wt = w[(p0 + i) * kRows + jj[q]];
              acc[q].x = fmaf(wt, v[q][i].x, acc[q].x);
              acc[q].y = fmaf(wt, v[q][i].y, acc[q].y);
              acc[q].z = fmaf(wt, v[q][i].z, acc[q].z);
              acc[q].w = fmaf(wt, v[q][i].w, acc[q].w);
            }
          }
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if (!in[q]) continue;
        const long long oi = static_cast<long long>(b) * per_batch * D + off[q];
        if (!CP_IN_BOUNDS(oi + 4 <= static_cast<long long>(batch) * per_batch * D, status)) continue;
        if (out_fp32)
          *reinterpret_cast<float4*>(static_cast<float*>(o_out) + oi) = acc[q];
        else
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o_out) + oi) =
              make_uint2(pack2(acc[q].x, acc[q].y), pack2(acc[q].z, acc[q].w));
      }
    }
    __syncwarp();  // the next unit rewrites the weights
  }
}

}  // namespace

int launch_merge(int batch, int n_parts, int rows, int H, int d, const float* o_parts, const float* lse_parts,
                 void* o_out, float* lse_out, int out_fp32, cudaStream_t stream, int32_t* status) {
  if (static_cast<long long>(batch) * rows * H == 0) return CP_OK;
  if (n_parts <= 0) return CP_ERR_INVALID_ARG;
  // Shared memory: n_parts * 32 weights per warp; fewer warps per CTA when
  // there are many parts.
  const long long per_warp = static_cast<long long>(n_parts) * kRows * sizeof(float);
  int warps = 8;
  while (warps > 1 && per_warp * warps > kMaxSmem) warps >>= 1;
  if (per_warp * warps > kMaxSmem) return CP_ERR_UNSUPPORTED;  // more than 768 parts
  const int smem = static_cast<int>(per_warp * warps);
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long units = static_cast<long long>(batch) * ((rows + kRows - 1) / kRows) * H;
  long long grid = (units + warps - 1) / warps;
  const long long cap = static_cast<long long>(sms) * (64 / warps);
  if (grid > cap) grid = cap;
  const int threads = warps * 32;
  if (d == 128) {
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(merge_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return CP_ERR_CUDA;
    merge_kernel<128><<<static_cast<int>(grid), threads, smem, stream>>>(n_parts, rows, H, o_parts, lse_parts, o_out,
                                                                        lse_out, batch, out_fp32, status);
  } else if (d == 64) {
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(merge_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return CP_ERR_CUDA;
    merge_kernel<64><<<static_cast<int>(grid), threads, smem, stream>>>(n_parts, rows, H, o_parts, lse_parts, o_out,
                                                                       lse_out, batch, out_fp32, status);
  } else {
    return CP_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

}  // namespace cpattn
