// reshard.cu -- the Ulysses all-to-all of all ring groups as one in-memory
// permutation copy ([MTX] nougat.kr "MaxText long-context training and KV
// parallelism", section "Split heads or rotate KV": before attention each
// chip trades its token shard of all heads for the whole group sequence of a
// subset of heads, and a second exchange restores token sharding after it;
// [ULY] aionda.blog "Ulysses sequence parallelism", "Current state").
//
// Both layouts are sequences of contiguous blocks:
//   token-major: a block is one token's H/U heads (H/U * E elements),
//   head-major (LSE): a block is one head's n tokens.
// The kernel walks the OUTPUT in order, one 16-byte (or 4-byte) vector per
// thread and several vectors in flight per thread, so every write is fully
// coalesced and every read is a contiguous run of at least one block.  It is
// bandwidth-bound; the grid is a multiple of the SM count.
#include <cuda_runtime.h>

#include <cstdint>

#include "cp_attn.h"
#include "kernels.h"

namespace cpattn {
namespace {

struct ReshardGeom {
  long long R, U, n, H, Hl;  // Hl = H / U
  long long blk;             // block size in vectors
  int dir, kind;
};

// Input vector offset of output block `ob` (in units of vectors).
__device__ __forceinline__ long long in_block(const ReshardGeom& g, long long ob) {
  const long long U = g.U, n = g.n, H = g.H, Hl = g.Hl;
  if (g.kind == CP_TOKEN_MAJOR) {
    if (g.dir == CP_SEQ_TO_HEAD) {
      // out [r][u][s*n+t] (block = Hl heads)  <-  in [r][s][t][u*Hl ..]
      const long long t = ob % n;
      long long x = ob / n;
      const long long s = x % U;
      x /= U;
      const long long u = x % U;
      const long long r = x / U;
      return (((r * U + s) * n + t) * U + u) * g.blk;  // in row has H = U*Hl heads = U blocks
    } else {
      // out [r][s][t][u*Hl ..] (block index (r,s,t,u))  <-  in [r][u][s*n+t]
      const long long u = ob % U;
      long long x = ob / U;
      const long long t = x % n;
      x /= n;
      const long long s = x % U;
      const long long r = x / U;
      return ((r * U + u) * U * n + s * n + t) * g.blk;
    }
  } else {
    if (g.dir == CP_SEQ_TO_HEAD) {
      // out [r][u][h'][s*n .. +n]  (block index (r,u,h',s))  <-  in [r][s][u*Hl+h'][0..n)
      const long long s = ob % U;
      long long x = ob / U;
      const long long hl = x % Hl;
      x /= Hl;
      const long long u = x % U;
      const long long r = x / U;
      return ((r * U + s) * H + u * Hl + hl) * g.blk;
    } else {
      // out [r][s][h = u*Hl+h'][0..n)  (block index (r,s,h))  <-  in [r][u][h'][s*n ..]
      const long long h = ob % H;
      long long x = ob / H;
      const long long s = x % U;
      const long long r = x / U;
      const long long u = h / Hl, hl = h % Hl;
      return (((r * U + u) * Hl + hl) * U + s) * g.blk;
    }
  }
}

template <typename V, int ILP>
__global__ void __launch_bounds__(256) reshard_kernel(const V* __restrict__ in, V* __restrict__ out,
                                                      ReshardGeom g, long long total) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x * ILP;
  for (long long base = (static_cast<long long>(blockIdx.x) * blockDim.x * ILP) + threadIdx.x; base < total;
       base += stride) {
    V v[ILP];
    long long dst[ILP];
#pragma unroll
    for (int i = 0; i < ILP; ++i) {
      const long long o = base + static_cast<long long>(i) * blockDim.x;
      dst[i] = o;
      if (o < total) {
        const long long ob = o / g.blk, w = o - ob * g.blk;
        v[i] = __ldg(in + in_block(g, ob) + w);
      }
    }
#pragma unroll
    for (int i = 0; i < ILP; ++i)
      if (dst[i] < total) out[dst[i]] = v[i];
  }
}

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n = 148;
  }
  return n;
}

}  // namespace

int launch_reshard(int R, int U, int n, int H, int row_elems, int direction, int kind, int elem_bytes,
                   const void* in, void* out, cudaStream_t stream) {
  ReshardGeom g;
  g.R = R;
  g.U = U;
  g.n = n;
  g.H = H;
  g.Hl = H / U;
  g.dir = direction;
  g.kind = kind;
  const long long block_bytes = (kind == CP_TOKEN_MAJOR) ? g.Hl * row_elems * elem_bytes
                                                         : static_cast<long long>(n) * elem_bytes;
  const long long total_bytes = static_cast<long long>(R) * U * n * H * row_elems * elem_bytes;
  if (total_bytes == 0) return CP_OK;
  const int blocks_per_sm = 8, threads = 256;
  const long long grid_cap = static_cast<long long>(sm_count()) * blocks_per_sm;
  if (block_bytes % 16 == 0) {
    g.blk = block_bytes / 16;
    const long long total = total_bytes / 16;
    const long long need = (total + threads * 4 - 1) / (threads * 4);
    const int grid = static_cast<int>(need < grid_cap ? need : grid_cap);
    reshard_kernel<uint4, 4><<<grid, threads, 0, stream>>>(static_cast<const uint4*>(in), static_cast<uint4*>(out), g,
                                                           total);
  } else if (block_bytes % 4 == 0) {
    g.blk = block_bytes / 4;
    const long long total = total_bytes / 4;
    const long long need = (total + threads * 4 - 1) / (threads * 4);
    const int grid = static_cast<int>(need < grid_cap ? need : grid_cap);
    reshard_kernel<uint32_t, 4><<<grid, threads, 0, stream>>>(static_cast<const uint32_t*>(in),
                                                              static_cast<uint32_t*>(out), g, total);
  } else {
    return CP_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

}  // namespace cpattn
