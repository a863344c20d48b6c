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
// 2d + 4.  d/4 threads own one (row, head), one float4 of every part each;
// consecutive threads cover consecutive addresses, so all loads and stores
// are coalesced.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "cp_attn.h"
#include "kernels.h"

namespace cpattn {
namespace {

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <int D>
__global__ void __launch_bounds__(256) merge_kernel(int n_parts, long long rows, int H, const float* __restrict__ o_parts,
                                                    const float* __restrict__ lse_parts, void* __restrict__ o_out,
                                                    float* __restrict__ lse_out, long long batch, int out_fp32) {
  constexpr int TPR = D / 4;  // threads per (row, head)
  const long long per_batch = rows * H;
  const long long total = batch * per_batch * TPR;
  for (long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; tid < total;
       tid += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c4 = static_cast<int>(tid % TPR);
    const long long rh = tid / TPR;              // (batch, row, head) flat
    const long long b = rh / per_batch;
    const long long w = rh - b * per_batch;      // row * H + head
    const long long row = w / H;
    const int h = static_cast<int>(w - row * H);
    const float* lp = lse_parts + b * n_parts * per_batch + static_cast<long long>(h) * rows + row;
    float m = -INFINITY;
    for (int p = 0; p < n_parts; ++p) m = fmaxf(m, __ldg(lp + p * per_batch));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lse = -INFINITY;
    if (m != -INFINITY) {
      float sum = 0.f;
      for (int p = 0; p < n_parts; ++p) sum += __expf(__ldg(lp + p * per_batch) - m);
      lse = m + __logf(sum);
      const float* op = o_parts + b * n_parts * per_batch * D + w * D + c4 * 4;
      for (int p = 0; p < n_parts; ++p) {
        const float wgt = __expf(__ldg(lp + p * per_batch) - lse);
        const float4 x = __ldg(reinterpret_cast<const float4*>(op + p * per_batch * D));
        acc.x = fmaf(wgt, x.x, acc.x);
        acc.y = fmaf(wgt, x.y, acc.y);
        acc.z = fmaf(wgt, x.z, acc.z);
        acc.w = fmaf(wgt, x.w, acc.w);
      }
    }
    const long long oi = (b * per_batch + w) * D + c4 * 4;
    if (out_fp32)
      *reinterpret_cast<float4*>(static_cast<float*>(o_out) + oi) = acc;
    else
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o_out) + oi) = make_uint2(pack2(acc.x, acc.y), pack2(acc.z, acc.w));
    if (c4 == 0) lse_out[b * per_batch + static_cast<long long>(h) * rows + row] = lse;
  }
}

}  // namespace

int launch_merge(int batch, int n_parts, int rows, int H, int d, const float* o_parts, const float* lse_parts,
                 void* o_out, float* lse_out, int out_fp32, cudaStream_t stream) {
  const long long work = static_cast<long long>(batch) * rows * H * (d / 4);
  if (work == 0) return CP_OK;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int threads = 256;
  long long grid = (work + threads - 1) / threads;
  const long long cap = static_cast<long long>(sms) * 8;
  if (grid > cap) grid = cap;
  if (d == 128)
    merge_kernel<128><<<static_cast<int>(grid), threads, 0, stream>>>(n_parts, rows, H, o_parts, lse_parts, o_out,
                                                                      lse_out, batch, out_fp32);
  else if (d == 64)
    merge_kernel<64><<<static_cast<int>(grid), threads, 0, stream>>>(n_parts, rows, H, o_parts, lse_parts, o_out,
                                                                     lse_out, batch, out_fp32);
  else
    return CP_ERR_UNSUPPORTED;
  return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

}  // namespace cpattn
