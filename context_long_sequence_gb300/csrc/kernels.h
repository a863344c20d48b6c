// kernels.h -- internal launch interface between the C-ABI layer (cp_attn.cu)
// and the kernels.  Not part of the public ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime_api.h>

namespace cpattn {

// Query tile of one attention rank: slots [q0, q0+len) of attention rank
// a = r*U + u, lying inside one contiguous-position chunk; `step` is the ring
// step this item covers (emit-partials mode) or -1 for all steps.
struct WorkItem {
  int32_t a, q0, len, step;
};

// Geometry shared by the forward and backward kernels.  "Attention rank"
// (r, u): member u of ring rank r after the Ulysses reshard, holding the T
// slots of ring rank r's shard for Hq_loc query and Hkv_loc KV heads.
struct AttnGeom {
  int L, R, U, T;          // T = L / R slots per attention rank
  int Hq_loc, Hkv_loc, G;  // G = Hq_loc / Hkv_loc
  int layout;              // CP_LAYOUT_*
  int chunk;               // contiguous-position chunk length: T / nchunks
  int nchunks;             // chunks per ring rank: 1 (contiguous), 2 (zigzag), m (balanced)
  const int32_t* chunk_pos;  // balanced: [R][nchunks] first position of each chunk (host or
                             // device copy, matching where slot_pos runs); else null
  const int32_t* chunk_owner;  // balanced: [R*nchunks] position chunk j -> r*nchunks + k, the
                               // rank r and local chunk k holding it (inverse of chunk_pos); else null
  int kv_global;           // 1: K/V rows are in global position order (all-gathered), U == 1
  float scale;             // softmax scale
  const int32_t* doc_start;  // [L] start of the document holding each position, or null
  const int32_t* doc_end;    // [L] one past the end of that document, or null
};

// Global position of slot t of ring rank r.
__host__ __device__ inline int slot_pos(const AttnGeom& g, int r, int t) {
  if (g.layout == 0) return r * g.T + t;
  const int c = g.chunk;
  if (g.layout == 1) return t < c ? r * c + t : (2 * g.R - 1 - r) * c + (t - c);
  const int j = t / c;
  return g.chunk_pos[r * g.nchunks + j] + (t - j * c);
}

// Ring rank and first slot of the position chunk j (positions [j*chunk,
// (j+1)*chunk)): every layout cuts the sequence into chunks of g.chunk.
__host__ __device__ inline void chunk_owner(const AttnGeom& g, int j, int& src, int& cslot0) {
  if (g.layout == 0) {
    src = j;
    cslot0 = 0;
  } else if (g.layout == 1) {
    const bool first = j < g.R;
    src = first ? j : 2 * g.R - 1 - j;
    cslot0 = first ? 0 : g.chunk;
  } else {
    const int e = g.chunk_owner[j];
    src = e / g.nchunks;
    cslot0 = (e - src * g.nchunks) * g.chunk;
  }
}

struct FwdArgs {
  AttnGeom g;
  const void* q;  // [R*U*T][Hq_loc][d] bf16
  const void* k;  // [R*U*T][Hkv_loc][d] bf16
  const void* v;
  void* o;        // [R*U*T][Hq_loc][d] bf16 or fp32 (o_fp32)  (fused mode)
  int o_fp32;
  float* lse;     // [R*U][Hq_loc][T]            (fused mode)
  float* o_part;  // [R][R][T][Hq][d] fp32       (emit-partials mode, U == 1)
  float* lse_part;// [R][R][Hq][T]
  const WorkItem* items;
  int n_items;
  int d;
  int32_t* status;
  // rank_local = 1: one ring step of one attention rank (the transport
  // path).  Every item covers ring step `step` (its own step field is
  // ignored); Q holds only that rank's T rows, K and V only the visiting
  // chunk's T rows (the slots of rank (r - step) mod R); o_part
  // [T][Hq_loc][d] and lse_part [Hq_loc][T] receive that step's normalised
  // partial.  0 (the zero-initialised default): all ranks, as above.
  int rank_local;
  int step;
  // Launch order.  0: block b = item b / Hq_loc, head b % Hq_loc.  1 (with
  // `items` grouped by Ulysses member u, n_items_u each): blocks run one K/V
  // stream (u, KV head) after another, and within a stream the items in
  // list order with the G query heads of the KV head adjacent, so the CTAs
  // resident at once read the same K/V tiles.
  int stream_major;
  int n_items_u;
  // seq_io = 1 (fused mode, U > 1): q, k, v, o and lse are the
  // sequence-sharded API tensors, [R*T][Hq][d], [R*T][Hkv][d] and
  // [R*U][Hq][n] (n = T/U), instead of head-sharded copies.  Ring rank r's
  // U members hold its T ring-local slots in order, so slot t of ring rank r
  // is row r*T + t, and member u's heads are the column range [u*Hq_loc,
  // (u+1)*Hq_loc): the Ulysses exchange becomes the kernel's addressing.
  int seq_io;
};

int launch_attn_fwd(const FwdArgs& a, cudaStream_t stream);

// Debug table of the forward's tile classes for the work items of `a`:
// rows [n_items][stride][8] {a, q0, len, step, kpos0, klen, class0, class1},
// counts [n_items] (tiles walked per item; rows beyond `stride` are dropped).
int launch_tile_classes(const FwdArgs& a, int32_t* rows, int32_t* counts, int stride, cudaStream_t stream);

// Backward on the head-sharded layout of cp_attn_fwd_local (rank a = r*U+u;
// with U == 1 that is the sequence-sharded layout).  items_q: 128-row query
// tiles (all ring steps); items_kv: key tiles {a = owner rank, q0 = first
// slot, len, -1}.
struct BwdArgs {
  AttnGeom g;
  const void* q;  const void* k;  const void* v;
  const void* o;  const float* lse;  const void* dO;
  int o_fp32;     // o is fp32 instead of bf16
  float* dq;  float* dk;  float* dv;
  // Row statistics the delta pass prepares for the gradient kernels, per
  // (attention rank, query head, slot) in the chunk-padded layout
  // [R*U][Hq_loc][nchunks][chunk_pad] (ld_index below): every 128-slot query
  // tile starts on a 512-byte boundary, so it can be fetched with one bulk
  // copy; padding slots hold -inf and 0.
  float* nlse;    // -LSE * log2(e)   (-inf for a row with no visible key)
  float* nd;      // -D = -rowsum(dO * O)
  int chunk_pad;  // chunk rounded up to a multiple of 128
  const WorkItem* items_q;
  int n_items_q;
  const WorkItem* items_kv;
  int n_items_kv;
  int d;
  int32_t* status;
  // rank_local = 1: one ring step `step` (the transport path).  dq: items_q
  // are query tiles of one attention rank a = r*U + u, whose Q, dO, LSE,
  // delta and dq are that rank's own T-row buffers, against the visiting
  // chunk of rank ((r - step) mod R)*U + u held in k, v (T rows).  dkv:
  // items_kv are key tiles of the visiting chunk (its owner rank a), whose
  // k, v, dk, dv are the chunk's T-row buffers, against the queries of the
  // holder rank ((a/U + step) mod R)*U + u held in q, dO, lse, delta.
  // 0 (the zero-initialised default): every rank and ring step.
  int rank_local;
  int step;
  int accumulate;  // 1: dq, dk, dv += this call's contribution (else overwritten)
  int phases;      // bit 0: delta, bit 1: dkv, bit 2: dq; 0 means all three
  // Launch order as FwdArgs::stream_major, with items_q and items_kv grouped
  // by Ulysses member (n_items_q_u and n_items_kv_u each).
  int stream_major;
  int n_items_q_u, n_items_kv_u;
  // seq_io = 1 (all ranks, U > 1): q, k, v, o, dO, lse, dq, dk and dv are
  // the sequence-sharded API tensors, addressed as FwdArgs::seq_io describes
  // (slot t of ring rank r is row r*T + t; member u's heads a column range).
  int seq_io;
};

int launch_attn_bwd(const BwdArgs& a, cudaStream_t stream);

// Index of slot t of attention rank a (0 in rank-local buffers), query head h
// in the chunk-padded statistics layout of BwdArgs::nlse / nd.
__host__ __device__ inline size_t ld_index(const AttnGeom& g, int chunk_pad, int a, int h, int t) {
  const int ch = t / g.chunk;
  return (static_cast<size_t>(a) * g.Hq_loc + h) * (static_cast<size_t>(g.nchunks) * chunk_pad) +
         static_cast<size_t>(ch) * chunk_pad + (t - ch * g.chunk);
}

// All-gather of K or V in the emulation: out[slot_pos(r, t)] = in[r*T + t],
// rows of row_bytes (a multiple of 16).
int launch_gather_rows(const AttnGeom& g, long long row_bytes, const void* in, void* out, cudaStream_t stream,
                       int32_t* status);

// Block-permutation copy behind ulysses_reshard.  `status` (the device
// status words) receives the bounds records of debug builds.
int launch_reshard(int R, int U, int n, int H, int row_elems, int direction, int kind,
                   int elem_bytes, const void* in, void* out, cudaStream_t stream, int32_t* status);

// One reshard of a batch (the arguments of launch_reshard).
struct ReshardSpec {
  int H, row_elems, direction, kind, elem_bytes;
  const void* in;
  void* out;
};

// Up to 8 reshards of one plan geometry in one launch (two when some need
// 4-byte vectors and others 16-byte ones).
int launch_reshard_batch(int R, int U, int n, const ReshardSpec* jobs, int count, cudaStream_t stream,
                         int32_t* status);

// Merge of `n_parts` partials, `batch` independent groups laid out back to back.
int launch_merge(int batch, int n_parts, int rows, int H, int d, const float* o_parts,
                 const float* lse_parts, void* o_out, float* lse_out, int out_fp32, cudaStream_t stream,
                 int32_t* status);

}  // namespace cpattn
