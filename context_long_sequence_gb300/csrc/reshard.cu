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
// The kernel walks the OUTPUT in order.  Blocks longer than 4 KB are cut into
// 4 KB segments (LSE blocks are a whole rank's tokens of one head), and one
// warp copies one segment at a time (lanes take consecutive 16-byte vectors,
// or 4-byte words when a block is not a multiple of 16 bytes), so reads and
// writes are both contiguous and fully coalesced; the source offset is
// computed once per segment, not per vector.  Each warp keeps four segments
// in flight.  HBM-bound; the grid is a multiple of the SM count.
//
// gather_rows_kernel is the all-gather of K/V in the one-GPU emulation
// ([MTX] "Why KV comes back together": every chip collects the whole K/V):
// slot rows of every rank are written to their global positions.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#define CP_TU_ID ::cpattn::kTuReshard
#include "cp_attn.h"
#include "debug.cuh"
#include "kernels.h"

namespace cpattn {
namespace {

// Division by a runtime divisor d >= 1 for x < 2^31, by multiply and shift
// (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994: with 2^(l-1) < d <= 2^l and m = floor(2^(31+l)/d) + 1,
// floor(x/d) = floor(m*x / 2^(31+l)) for every 31-bit x; m < 2^32).
struct FastDiv {
  uint32_t d, m, sh;
  __host__ __device__ __forceinline__ uint32_t div(uint32_t x) const {
    return static_cast<uint32_t>((static_cast<uint64_t>(x) * m) >> sh);
  }
};

FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  FastDiv f;
  f.d = d;
  f.m = static_cast<uint32_t>((1ull << (31 + l)) / d + 1);
  f.sh = 31 + l;
  return f;
}

struct ReshardGeom {
  uint32_t U, n, H, Hl;  // Hl = H / U
  FastDiv fU, fn, fH, fHl;
  uint32_t blk;          // block size in vectors
  uint32_t nblocks;      // output blocks
  uint32_t seg, nseg;    // segment size in vectors, segments per block
  uint32_t nunits;       // nblocks * nseg
  int dir, kind;
  int32_t* status;       // device status words (bounds records of debug builds)
};

// Source block index of output block `ob`.
__device__ __forceinline__ uint32_t in_block(const ReshardGeom& g, uint32_t ob) {
  const uint32_t U = g.U, n = g.n, H = g.H, Hl = g.Hl;
  if (g.kind == CP_TOKEN_MAJOR) {
    if (g.dir == CP_SEQ_TO_HEAD) {
      // out [r][u][s*n+t] (block = Hl heads)  <-  in [r][s][t][u*Hl ..]
      uint32_t x = g.fn.div(ob);
      const uint32_t t = ob - x * n;
      uint32_t y = g.fU.div(x);
      const uint32_t s = x - y * U;
      const uint32_t r = g.fU.div(y);
      const uint32_t u = y - r * U;
      return ((r * U + s) * n + t) * U + u;  // an input row holds U blocks
    }
    // out [r][s][t][u*Hl ..] (block (r,s,t,u))  <-  in [r][u][s*n+t]
    uint32_t x = g.fU.div(ob);
    const uint32_t u = ob - x * U;
    uint32_t y = g.fn.div(x);
    const uint32_t t = x - y * n;
    const uint32_t r = g.fU.div(y);
    const uint32_t s = y - r * U;
    return (r * U + u) * U * n + s * n + t;
  }
  if (g.dir == CP_SEQ_TO_HEAD) {
    // out [r][u][h'][s*n .. +n]  (block (r,u,h',s))  <-  in [r][s][u*Hl+h'][0..n)
    uint32_t x = g.fU.div(ob);
    const uint32_t s = ob - x * U;
    uint32_t y = g.fHl.div(x);
    const uint32_t hl = x - y * Hl;
    const uint32_t r = g.fU.div(y);
    const uint32_t u = y - r * U;
    return (r * U + s) * H + u * Hl + hl;
  }
  // out [r][s][h = u*Hl+h'][0..n)  (block (r,s,h))  <-  in [r][u][h'][s*n ..]
  uint32_t x = g.fH.div(ob);
  const uint32_t h = ob - x * H;
  const uint32_t r = g.fU.div(x);
  const uint32_t s = x - r * U;
  const uint32_t u = g.fHl.div(h), hl = h - u * Hl;
  return ((r * U + u) * Hl + hl) * U + s;
}

constexpr int kBlocksInFlight = 4;
constexpr int kMaxJobs = 8;

// Several reshards in one launch: job j owns the global units
// [unit0[j], unit0[j+1]); all jobs use the same vector type.
struct ReshardBatch {
  ReshardGeom g[kMaxJobs];
  const void* in[kMaxJobs];
  void* out[kMaxJobs];
  uint32_t unit0[kMaxJobs + 1];
  int n;
};

template <typename V>
__global__ void __launch_bounds__(256) reshard_kernel(const __grid_constant__ ReshardBatch b) {
  const int lane = threadIdx.x & 31;
  const uint32_t warps = (gridDim.x * blockDim.x) >> 5;
  const uint32_t w0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t total = b.unit0[b.n];
  for (uint32_t base = w0 * kBlocksInFlight; base < total; base += warps * kBlocksInFlight) {
    const V* src[kBlocksInFlight];
    V* dst[kBlocksInFlight];
    uint32_t len[kBlocksInFlight];
#pragma unroll
    for (int i = 0; i < kBlocksInFlight; ++i) {
      const uint32_t gu = base + i;
      len[i] = 0;
      src[i] = nullptr;
      dst[i] = nullptr;
      if (gu < total) {
        int j = 0;
        while (j + 1 < b.n && gu >= b.unit0[j + 1]) ++j;
        const ReshardGeom& g = b.g[j];
        const uint32_t un = gu - b.unit0[j];
        const uint32_t ob = un / g.nseg;
        const uint32_t v0 = (un - ob * g.nseg) * g.seg;
        const uint32_t ib = in_block(g, ob);
        if (!CP_IN_BOUNDS(ib < g.nblocks && ob < g.nblocks && v0 < g.blk, g.status)) continue;
        len[i] = min(g.seg, g.blk - v0);
        src[i] = static_cast<const V*>(b.in[j]) + (static_cast<uint64_t>(ib) * g.blk + v0);
        dst[i] = static_cast<V*>(b.out[j]) + (static_cast<uint64_t>(ob) * g.blk + v0);
      }
    }
    // A warp's segments are at most 4 KB, so lane strides cover them in a few steps.
    uint32_t seg_max = 0;
#pragma unroll
    for (int i = 0; i < kBlocksInFlight; ++i) seg_max = max(seg_max, len[i]);
    for (uint32_t v = lane; v < seg_max; v += 32) {
      V val[kBlocksInFlight];
#pragma unroll
      for (int i = 0; i < kBlocksInFlight; ++i)
        if (v < len[i]) val[i] = __ldg(src[i] + v);
#pragma unroll
      for (int i = 0; i < kBlocksInFlight; ++i)
        if (v < len[i]) dst[i][v] = val[i];
    }
  }
}

// All-gather in the emulation: each warp moves one slot row to its position.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                                                          AttnGeom g, uint32_t vecs, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const uint32_t warps = (gridDim.x * blockDim.x) >> 5;
  const uint32_t rows = static_cast<uint32_t>(g.R) * g.T;
  for (uint32_t slot = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; slot < rows; slot += warps) {
    const int r = static_cast<int>(slot / g.T), t = static_cast<int>(slot % g.T);
    const int pos = slot_pos(g, r, t);
    if (!CP_IN_BOUNDS(pos >= 0 && pos < g.L, status)) continue;
    const uint64_t src = static_cast<uint64_t>(slot) * vecs;
    const uint64_t dst = static_cast<uint64_t>(pos) * vecs;
    for (uint32_t v = lane; v < vecs; v += 32) out[dst + v] = __ldg(in + src + v);
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

int launch_gather_rows(const AttnGeom& g, long long row_bytes, const void* in, void* out, cudaStream_t stream,
                       int32_t* status) {
  if (g.U != 1 || row_bytes <= 0 || row_bytes % 16 || row_bytes / 16 >= (1LL << 32)) return CP_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(g.R) * g.T;
  if (rows == 0) return CP_OK;
  const int threads = 256;
  long long grid = (rows * 32 + threads - 1) / threads;
  const long long cap = static_cast<long long>(sm_count()) * 8;
  if (grid > cap) grid = cap;
  gather_rows_kernel<<<static_cast<int>(grid), threads, 0, stream>>>(static_cast<const uint4*>(in),
                                                                     static_cast<uint4*>(out), g,
                                                                     static_cast<uint32_t>(row_bytes / 16), status);
  return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

namespace {

// Geometry of one reshard; vec_bytes = 16 or 4 (the vector type it needs).
// Returns CP_OK with g.nunits == 0 for an empty job.
int reshard_geom(int R, int U, int n, const ReshardSpec& j, int32_t* status, ReshardGeom* out_g, int* vec_bytes) {
  ReshardGeom g;
  g.status = status;
  g.U = U;
  g.n = n;
  g.H = j.H;
  g.Hl = j.H / U;
  g.dir = j.direction;
  g.kind = j.kind;
  g.fU = make_fastdiv(g.U);
  g.fn = make_fastdiv(g.n);
  g.fH = make_fastdiv(g.H);
  g.fHl = make_fastdiv(g.Hl);
  g.nunits = 0;
  const long long block_bytes = (j.kind == CP_TOKEN_MAJOR)
                                    ? static_cast<long long>(g.Hl) * j.row_elems * j.elem_bytes
                                    : static_cast<long long>(n) * j.elem_bytes;
  const long long nblocks = (j.kind == CP_TOKEN_MAJOR) ? static_cast<long long>(R) * U * n * U
                                                       : static_cast<long long>(R) * U * j.H;
  *vec_bytes = (block_bytes % 16 == 0) ? 16 : 4;
  *out_g = g;
  if (nblocks == 0 || block_bytes == 0) return CP_OK;
  if (nblocks >= (1LL << 31)) return CP_ERR_UNSUPPORTED;  // the block index math is 31-bit
  if (block_bytes % 4 != 0) return CP_ERR_UNSUPPORTED;
  const long long blk = block_bytes / *vec_bytes;
  if (blk >= (1LL << 32)) return CP_ERR_UNSUPPORTED;
  // Segments: 4 KB of a token-major block; 512 bytes of a head-major (LSE)
  // block, whose blocks are few and long.
  const long long seg = std::min<long long>(blk, (j.kind == CP_HEAD_MAJOR ? 512 : 4096) / *vec_bytes);
  const long long nseg = (blk + seg - 1) / seg;
  const long long nunits = nblocks * nseg;
  if (nunits >= (1LL << 32)) return CP_ERR_UNSUPPORTED;
  g.nblocks = static_cast<uint32_t>(nblocks);
  g.blk = static_cast<uint32_t>(blk);
  g.seg = static_cast<uint32_t>(seg);
  g.nseg = static_cast<uint32_t>(nseg);
  g.nunits = static_cast<uint32_t>(nunits);
  *out_g = g;
  return CP_OK;
}

template <typename V>
int launch_batch(const ReshardBatch& b, cudaStream_t stream) {
  const uint32_t total = b.unit0[b.n];
  if (total == 0) return CP_OK;
  const int threads = 256, warps_per_cta = threads / 32;
  const long long need = (static_cast<long long>(total) + warps_per_cta * kBlocksInFlight - 1) /
                         (warps_per_cta * kBlocksInFlight);
  const long long cap = static_cast<long long>(sm_count()) * 8;
  const int grid = static_cast<int>(need < cap ? need : cap);
  reshard_kernel<V><<<grid, threads, 0, stream>>>(b);
  return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

}  // namespace

int launch_reshard_batch(int R, int U, int n, const ReshardSpec* jobs, int count, cudaStream_t stream,
                         int32_t* status) {
  if (count < 0 || count > kMaxJobs) return CP_ERR_INVALID_ARG;
  // Jobs that need 16-byte vectors go in one launch, the others in a second.
  ReshardBatch b16{}, b4{};
  long long u16 = 0, u4 = 0;
  for (int i = 0; i < count; ++i) {
    ReshardGeom g;
    int vb = 16;
    const int rc = reshard_geom(R, U, n, jobs[i], status, &g, &vb);
    if (rc != CP_OK) return rc;
    if (g.nunits == 0) continue;
    ReshardBatch& b = vb == 16 ? b16 : b4;
    long long& u = vb == 16 ? u16 : u4;
    b.g[b.n] = g;
    b.in[b.n] = jobs[i].in;
    b.out[b.n] = jobs[i].out;
    b.unit0[b.n] = static_cast<uint32_t>(u);
    u += g.nunits;
    if (u >= (1LL << 32)) return CP_ERR_UNSUPPORTED;
    ++b.n;
    b.unit0[b.n] = static_cast<uint32_t>(u);
  }
  int rc = CP_OK;
  if (b16.n > 0) rc = launch_batch<uint4>(b16, stream);
  if (rc == CP_OK && b4.n > 0) rc = launch_batch<uint32_t>(b4, stream);
  return rc;
}

int launch_reshard(int R, int U, int n, int H, int row_elems, int direction, int kind, int elem_bytes,
                   const void* in, void* out, cudaStream_t stream, int32_t* status) {
  const ReshardSpec j{H, row_elems, direction, kind, elem_bytes, in, out};
  return launch_reshard_batch(R, U, n, &j, 1, stream, status);
}

}  // namespace cpattn
