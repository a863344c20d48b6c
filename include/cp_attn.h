/*
 * cp_attn.h -- C ABI of libcpattn: context-parallel causal attention for one
 * sm_103a GPU, with all P context-parallel ranks emulated side by side in the
 * GPU's memory.
 *
 * What the operations are (the web pages these follow; each citation names a
 * page and its section):
 *
 *  [MTX] nougat.kr, "MaxText long-context training and KV parallelism":
 *        "Why KV comes back together even after splitting the input" -- a
 *        long sequence is split over chips by token, and causal attention
 *        makes every query need the K/V of all earlier tokens;
 *        "Split heads or rotate KV" -- A2A (Ulysses) swaps token sharding for
 *        head sharding before attention and swaps back after it, the KV-head
 *        count capping the degree under GQA; P2P (ring) keeps token sharding,
 *        computes a partial with each visiting KV chunk and merges the
 *        partial results; later tokens carry more causal work, so the load
 *        must be balanced; USP combines A2A groups with a ring.
 *  [ULY] aionda.blog, "Ulysses sequence parallelism for long-context
 *        training", "Current state" -- all-to-all along the sequence axis so
 *        each GPU computes a subset of heads.
 *  [L3P] siliconandsystems.com, "Llama 3 parallelism", "Four parallelisms
 *        secure different resources" -- CP must keep the mask between packed
 *        documents; "Long context changes more than attention cost" --
 *        balance by actual attention work; activation recompute trades
 *        memory for compute.
 *
 * The pages give no formula.  The attention computed is textbook scaled
 * dot-product softmax attention, visibility M(i,k) = [pos_k <= pos_i] and
 * [same packed document], scale 1/sqrt(d) unless set, LSE in natural log,
 * query head h reading KV head floor(h / (Hq/Hkv)).
 *
 * Conventions common to every call
 *  - Device pointers are plain CUDA device addresses on the current device;
 *    host pointers are marked "host".  Nothing here takes ownership of a
 *    caller's buffer.  Calls are asynchronous on `stream` and return 0 on
 *    success or a negative CP_ERR_* code; on an error return nothing was
 *    enqueued.  Errors found on the device while a kernel runs (a bounded
 *    wait that ran out; in debug builds, an index out of range) are recorded
 *    in device status words read by cp_get_status() and
 *    cp_get_status_detail().
 *  - bf16 = bfloat16 (round-to-nearest-even on every conversion).
 *  - Token-major tensors are [tokens][heads][d] row-major.  "Sequence-sharded"
 *    tensors hold the P = U*R ranks' shards back to back, rank-major, rank
 *    g = r*U + u (Ulysses index innermost), each shard n = L/P tokens in slot
 *    order; cp_index_map() gives the global position of every slot.
 *  - LSE tensors are [rank][heads][tokens] fp32.
 *  - Every device pointer must be 16-byte aligned (CP_ERR_ALIGNMENT).
 */
#ifndef CP_ATTN_H
#define CP_ATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CP_ATTN_PLAN_VERSION 1

/* Return codes. */
#define CP_OK                  0
#define CP_ERR_INVALID_ARG    -1  /* a size, pointer or enum is out of range */
#define CP_ERR_UNSUPPORTED    -2  /* valid but not built: d not in {64,128}, U not dividing Hkv, ... */
#define CP_ERR_ALIGNMENT      -3  /* a device pointer is not 16-byte aligned */
#define CP_ERR_CUDA           -4  /* a CUDA runtime/driver call failed */
#define CP_ERR_DEVICE_TIMEOUT -5  /* a bounded device-side wait ran out (from cp_get_status) */
#define CP_ERR_DEVICE_BOUNDS  -6  /* a device-side index check failed (from cp_get_status) */
#define CP_ERR_WORKSPACE      -7  /* workspace pointer null or smaller than cp_workspace_size() */
#define CP_ERR_ARCH           -8  /* the current device is not sm_103 */

/* Token layouts of a ring rank's shard ([MTX] "Split heads or rotate KV",
 * [L3P] "Long context changes more than attention cost"). */
#define CP_LAYOUT_CONTIGUOUS 0    /* ring rank r holds positions [r*L/R, (r+1)*L/R) */
#define CP_LAYOUT_ZIGZAG     1    /* 2R chunks of c = L/(2R); rank r holds chunk r then chunk 2R-1-r */
#define CP_LAYOUT_BALANCED   2    /* m*R chunks of c = L/(m*R), m = chunks_per_rank, dealt out by
                                     attention work: a query at position i does i - doc_start(i) + 1
                                     units; chunks are taken from most to least work (equal work:
                                     lower chunk first) and each goes to the least-loaded rank that
                                     holds fewer than m chunks (equal load: lower rank first); a
                                     rank keeps its chunks in position order.  With m = 2 and one
                                     document this is exactly the zigzag layout. */

/* How a rank obtains the other ranks' K/V ([MTX] "Why KV comes back together",
 * "Split heads or rotate KV"; [L3P] "Four parallelisms secure different resources"). */
#define CP_KV_RING      0         /* ring (P2P): KV chunks visit the ranks in ring order */
#define CP_KV_ALLGATHER 1         /* all-gather: every rank first gathers the whole K/V, then
                                     attends over it in position order (U == 1, fused merge) */

/* Reshard directions and tensor kinds for ulysses_reshard(). */
#define CP_SEQ_TO_HEAD 0
#define CP_HEAD_TO_SEQ 1
#define CP_TOKEN_MAJOR 0          /* [tokens][H][row_elems]       (Q, K, V, O) */
#define CP_HEAD_MAJOR  1          /* [H][tokens], row_elems == 1  (LSE)        */

/* Operations for cp_workspace_size(). */
#define CP_OP_FWD 0
#define CP_OP_BWD 1
#define CP_OP_BWD_RANK_STATS 2  /* one attention rank's stats_rank buffer (cp_attn_bwd_delta) */

/* Plan description (host struct; copied by cp_plan_create). */
typedef struct {
  int32_t version;            /* CP_ATTN_PLAN_VERSION (a versioned plan: [L3P] "The parallel plan is a per-job contract") */
  int32_t L;                  /* global tokens (batch 1) */
  int32_t Hq, Hkv;            /* query heads, KV heads; Hkv divides Hq (GQA) */
  int32_t d;                  /* head dimension: 64 or 128 */
  int32_t ulysses_degree;     /* U >= 1; U divides Hkv ([MTX] "Split heads or rotate KV": KV heads cap A2A) */
  int32_t ring_degree;        /* R >= 1; P = U*R emulated ranks */
  int32_t layout;             /* CP_LAYOUT_*; R divides L (contiguous), 2R divides L (zigzag) or
                                 m*R divides L (balanced); U divides L/R */
  int32_t causal;             /* must be 1 (causal attention; [MTX] "Why KV comes back together") */
  int32_t num_docs;           /* 0 or 1: one document; >1: packed documents */
  const int32_t *doc_offsets; /* host; num_docs+1 entries, [0]=0, strictly increasing, [num_docs]=L; copied */
  float softmax_scale;        /* 0 => 1/sqrt(d) */
  int32_t emit_partials;      /* 1 => the forward writes one normalised (O, LSE) partial per ring step
                                 into the workspace and merges them in ring order with the same
                                 kernel as cp_merge_lse(); 0 => the merge is fused (online softmax
                                 continued across ring steps).  Requires U == 1. */
  int32_t out_fp32;           /* 0 => O is bf16 (round to nearest even); 1 => O is fp32 (the
                                 normalised accumulator, unrounded).  Applies to the o output of
                                 cp_attn_fwd, cp_attn_fwd_local and cp_attn_fwd_noalloc and to the
                                 o input of cp_attn_bwd; cp_merge_lse always writes bf16. */
  int32_t chunks_per_rank;    /* CP_LAYOUT_BALANCED: m >= 1 chunks per ring rank; ignored otherwise */
  int32_t kv_exchange;        /* CP_KV_RING (0) or CP_KV_ALLGATHER (1; requires U == 1 and
                                 emit_partials == 0).  The backward is the same computation either
                                 way: dK, dV land in the owner's slots (the reduce-scatter that
                                 mirrors the all-gather). */
} cp_plan_desc_t;

typedef struct cp_plan cp_plan_t;   /* opaque; immutable after creation; usable from any stream */

/* Validate `desc` and build the plan on the current device: the work list
 * (query tiles ordered by descending visible-tile count, [L3P] "balance by
 * actual attention work") and, with documents, a per-position document-start
 * table.  Allocates those device tables with cudaMalloc; they are freed by
 * cp_plan_destroy().  *out is set only on success. */
int cp_plan_create(const cp_plan_desc_t *desc, cp_plan_t **out);
void cp_plan_destroy(cp_plan_t *plan);

/* host_out[L]: global position of every slot of the sequence-sharded layout,
 * rank-major (rank g = r*U + u; member u of ring rank r holds ring-local slots
 * [u*n, (u+1)*n) of ring rank r's shard).  Host memory, caller-owned. */
int cp_index_map(const cp_plan_t *plan, int32_t *host_out);

/* Bytes of device workspace cp_attn_fwd (op CP_OP_FWD) or cp_attn_bwd
 * (CP_OP_BWD) needs for this plan. */
int cp_workspace_size(const cp_plan_t *plan, int op, size_t *bytes);

/* Ulysses all-to-all of all R groups at once ([MTX] "Split heads or rotate
 * KV", [ULY] "Current state"), as an in-memory permutation copy:
 *   CP_TOKEN_MAJOR, CP_SEQ_TO_HEAD:
 *     in  [R][U][n][H][E]  ->  out [R][U][U*n][H/U][E],
 *     out[r][u][s*n+t][h'] = in[r][s][t][u*H/U + h']
 *   CP_HEAD_MAJOR, CP_SEQ_TO_HEAD (E == 1):
 *     in  [R][U][H][n]     ->  out [R][U][H/U][U*n]
 *   CP_HEAD_TO_SEQ: the inverse maps.
 * n = L/(R*U) from the plan; H is the tensor's head count (U divides H);
 * E = row_elems elements of elem_bytes each.  in and out must not overlap.
 * Bit-exact (a copy).  16-byte vectors when H/U*E*elem_bytes (token-major)
 * or n*elem_bytes (head-major) is a multiple of 16, 4-byte words otherwise
 * (elem_bytes*E must then be a multiple of 4). */
int ulysses_reshard(const cp_plan_t *plan, int direction, int tensor_kind, int H,
                    int row_elems, int elem_bytes, const void *in, void *out,
                    cudaStream_t stream);

/* Several Ulysses reshards of one plan in one kernel launch, e.g. the Q, K,
 * V exchange before attention or the O and LSE exchange after it (the same
 * permutations as ulysses_reshard, one launch instead of one per tensor;
 * jobs whose blocks need 4-byte words go in a second launch).  jobs (host,
 * n_jobs entries, 1 .. CP_RESHARD_MAX_JOBS) hold ulysses_reshard's
 * arguments; the same rules apply to each, and in addition no job's output
 * may overlap any job's input or another job's output (CP_ERR_INVALID_ARG).
 * Bit-exact. */
#define CP_RESHARD_MAX_JOBS 8
typedef struct {
  int direction;   /* CP_SEQ_TO_HEAD | CP_HEAD_TO_SEQ */
  int tensor_kind; /* CP_TOKEN_MAJOR | CP_HEAD_MAJOR */
  int H;           /* heads of the tensor (U divides H) */
  int row_elems;   /* E: elements per (token, head) row; 1 for CP_HEAD_MAJOR */
  int elem_bytes;
  const void *in;  /* device */
  void *out;       /* device */
} cp_reshard_job_t;
int ulysses_reshard_batch(const cp_plan_t *plan, int n_jobs, const cp_reshard_job_t *jobs,
                          cudaStream_t stream);

/* Causal CP attention forward for all P emulated ranks.
 *   q  [P][n][Hq][d]  bf16, sequence-sharded (slot order of cp_index_map)
 *   k,v[P][n][Hkv][d] bf16
 *   o  [P][n][Hq][d]  bf16 out (fp32 if the plan's out_fp32 is set)
 *   lse[P][Hq][n]     fp32 out (natural log; -inf for a row with no visible key)
 * With U > 1 each Ulysses member u attends with its heads over the whole
 * ring group's sequence ([MTX] "Split heads or rotate KV": the two
 * exchanges around attention).  Every rank is in this GPU's memory, so the
 * exchanges are the kernel's addressing: member u of ring rank r reads rows
 * r*T .. r*T+T-1 of q, k, v (its group's slots, T = L/R) at its own heads
 * and writes o and lse in place; no head-sharded copy is made (the copy is
 * ulysses_reshard, for cp_attn_fwd_local and the per-step entries).
 * Per ring rank r and step s the visiting chunk comes from rank (r-s) mod R;
 * with CP_KV_ALLGATHER the call first gathers K and V of all ranks into
 * position order in the workspace, and every rank's queries then walk the
 * gathered keys in position order.  Tiles with no visible pair are skipped,
 * partially visible tiles are masked.
 * workspace: cp_workspace_size(plan, CP_OP_FWD) bytes (may be NULL when 0). */
int cp_attn_fwd(const cp_plan_t *plan, const void *q, const void *k, const void *v,
                void *o, float *lse, void *workspace, size_t workspace_bytes,
                cudaStream_t stream);

/* The attention between the two Ulysses exchanges: ring attention of every
 * attention rank (ring rank r, Ulysses member u) on head-sharded inputs, the
 * layout ulysses_reshard(CP_SEQ_TO_HEAD) produces ([MTX] "Split heads or
 * rotate KV": each chip computes its heads over the whole group sequence;
 * the ring runs over r for each head group u).
 *   q  [R][U][T][Hq/U][d] bf16,  k, v [R][U][T][Hkv/U][d] bf16, T = L/R
 *   o  [R][U][T][Hq/U][d] bf16 (fp32 if out_fp32) out,  lse [R][U][Hq/U][T] fp32 out
 * With U == 1 this is cp_attn_fwd with the fused merge; for a CP_KV_ALLGATHER
 * plan k and v are the gathered copies, [L][Hkv][d] in position order.
 * No workspace. */
int cp_attn_fwd_local(const cp_plan_t *plan, const void *q, const void *k, const void *v,
                      void *o, float *lse, cudaStream_t stream);

/* One attention rank's share of cp_attn_fwd_local: the outputs of rank
 * `rank` (= r*U + u; the ring rank r when U == 1), reading every rank's K/V
 * chunks from the same buffers, i.e. the work one GPU does when each rank
 * has its own GPU ([MTX] "Split heads or rotate KV": each chip keeps its
 * queries and visits every KV chunk).  Same layouts and results as
 * cp_attn_fwd_local (bit for bit on this rank's rows; for a CP_KV_ALLGATHER
 * plan k and v are the gathered copies in position order); other ranks'
 * rows of o and lse are not touched.  rank outside [0, P) => CP_ERR_INVALID_ARG.
 * No workspace. */
int cp_attn_fwd_rank(const cp_plan_t *plan, int rank, const void *q, const void *k, const void *v,
                     void *o, float *lse, cudaStream_t stream);

/* Causal CP attention backward from the forward's O and LSE (activation
 * recompute, [L3P] "Long context changes more than attention cost"): with
 * P = exp(scale*QK^T - LSE),
 *   D = rowsum(dO * O); dV = P^T dO; dS = P * (dO V^T - D);
 *   dQ = scale dS K;  dK = scale dS^T Q;  query heads sum into their KV head.
 * q, dO [P][n][Hq][d] bf16; o the same (fp32 if out_fp32); k, v [P][n][Hkv][d] bf16;
 * lse [P][Hq][n] fp32;
 * dq [P][n][Hq][d], dk, dv [P][n][Hkv][d] fp32 out (overwritten).
 * Gradients of a KV chunk land on the rank that owns the chunk.  With U > 1
 * (Ulysses, USP) the forward's exchanges run in reverse ([MTX] "Split heads
 * or rotate KV"): each member runs the ring backward of its heads over the
 * group's sequence.  As in cp_attn_fwd the exchanges are the kernels'
 * addressing (rows r*T.. of ring rank r, the member's heads), so no
 * head-sharded copy is made.  Deterministic: no atomics, fixed summation
 * order.
 * workspace: cp_workspace_size(plan, CP_OP_BWD) bytes: the per-row
 * statistics (-LSE*log2e and -D), 8 bytes per row and query head. */
int cp_attn_bwd(const cp_plan_t *plan, const void *q, const void *k, const void *v,
                const void *o, const float *lse, const void *dO,
                float *dq, float *dk, float *dv, void *workspace, size_t workspace_bytes,
                cudaStream_t stream);

/* ---- Ring steps for a transport that moves K/V chunks between processes
 * ([MTX] "Split heads or rotate KV": each chip keeps its queries, receives
 * the next KV chunk while it computes with the current one, and merges the
 * partial results; in the backward the chunk's gradients travel with it).
 * One call = one ring step s of one attention rank a = r*U + u, reading the
 * rank's own buffers and a visiting chunk held in separate buffers (the
 * layout each process keeps per rank):
 *   q_rank, do_rank [T][Hq/U][d] bf16; o_rank the same (fp32 if out_fp32);
 *   lse_rank [Hq/U][T] fp32;  T = L/R slots of ring rank r
 *   k_chunk, v_chunk [T][Hkv/U][d] bf16: the slots of attention rank
 *   a_src = ((r - s) mod R)*U + u, the chunk that visits rank a at step s.
 * With U == 1 these are plain sequence shards; with U > 1 they are the
 * head-sharded layout of ulysses_reshard (rows of rank a in its [T] block).
 * Plans with CP_KV_ALLGATHER return CP_ERR_UNSUPPORTED; rank outside [0, P)
 * or s outside [0, R) returns CP_ERR_INVALID_ARG.  No workspace. */

/* Forward partial of ring step s: the normalised attention of rank a's
 * queries over the keys of the visiting chunk that they see:
 *   o_part [T][Hq/U][d] fp32 out, lse_part [Hq/U][T] fp32 out
 * ((0, -inf) for rows that see none of the chunk).  Merging the R partials
 * with cp_merge_lse in step order gives rank a's rows of cp_attn_fwd_local. */
int cp_attn_fwd_step(const cp_plan_t *plan, int rank, int step, const void *q_rank,
                     const void *k_chunk, const void *v_chunk, float *o_part, float *lse_part,
                     cudaStream_t stream);

/* The backward's first pass over one rank's rows: D = rowsum(dO * O), and
 * the row statistics the gradient steps read, written to stats_rank
 * (cp_workspace_size(plan, CP_OP_BWD_RANK_STATS, ...) bytes):
 *   stats_rank[0][h][slot'] = -LSE * log2(e),  stats_rank[1][h][slot'] = -D
 * for the Hq/U heads of the rank, where slot' pads every position chunk of
 * the rank to a multiple of 128 slots (padding: -inf and 0) so that each
 * 128-slot query tile starts on a 512-byte boundary.  lse_rank [Hq/U][T]. */
int cp_attn_bwd_delta(const cp_plan_t *plan, const void *o_rank, const void *do_rank,
                      const float *lse_rank, float *stats_rank, cudaStream_t stream);

/* Backward contributions of ring step s (fp32):
 *   dq_rank [T][Hq/U][d]: rank a's dQ, from the visiting chunk's keys;
 *   dk_chunk, dv_chunk [T][Hkv/U][d]: the visiting chunk's dK, dV, from
 *   rank a's queries (the buffers travel with the chunk).
 * stats_rank is rank a's buffer from cp_attn_bwd_delta.
 * Step 0 (every chunk at its owner) writes all three, zeros where nothing
 * is visible; steps s > 0 add to them.  After the R steps of every rank,
 * rank a's dQ equals its rows of cp_attn_bwd's dq and each chunk's dk/dv
 * equal its owner's rows of cp_attn_bwd's dk/dv (the same products; the
 * fp32 sums are taken per ring step, so the results agree within fp32
 * rounding, not bit for bit). */
int cp_attn_bwd_step(const cp_plan_t *plan, int rank, int step, const void *q_rank,
                     const void *do_rank, const float *stats_rank, const void *k_chunk,
                     const void *v_chunk, float *dq_rank, float *dk_chunk, float *dv_chunk,
                     cudaStream_t stream);

/* Merge n_parts normalised attention partials over disjoint key sets
 * ([MTX] "Split heads or rotate KV": partial computation and merge):
 *   o_parts   [n_parts][rows][H][d] fp32, lse_parts [n_parts][H][rows] fp32
 *   o_out     [rows][H][d] bf16,          lse_out   [H][rows] fp32
 *   lse = m + ln(sum_p exp(lse_p - m)), m = max_p lse_p;
 *   o   = sum_p exp(lse_p - lse) o_p;   all parts -inf => o = 0, lse = -inf.
 * Parts are folded in index order.  d in {64, 128}. */
int cp_merge_lse(int n_parts, int rows, int H, int d, const float *o_parts,
                 const float *lse_parts, void *o_out, float *lse_out, cudaStream_t stream);

/* Debug table of the forward's tile classes (no counterpart in the pages: it
 * exposes which work the kernel skips).  For every work item of the plan's
 * forward -- a block of up to 256 query slots of one attention rank inside
 * one contiguous-position chunk, split into query tiles 0 and 1 of up to 128
 * rows -- the K/V tiles the kernel walks, in its order (ring steps s = 0..R-1,
 * source rank (r - s) mod R, that rank's chunks in slot order, 128-slot tiles
 * from each chunk's start; with the all-gather exchange, 128-position tiles
 * in position order; with emit_partials, one item per ring step), as rows of
 * 8 int32 {a, q0, len, step, kpos0, klen, class0, class1}: attention rank a,
 * first query slot q0, length len and ring step (-1: all steps) of the item,
 * first key position and length of the tile, and per query tile: 0 = not
 * seen (no MMA, no softmax pass), 1 = seen and masked, 2 = wholly visible
 * (mask skipped).  Items appear in the plan's launch order.  host_rows (host,
 * capacity rows of 8) may be null with
 * capacity 0 to ask for the count.  *n_rows = rows in the table.  Returns
 * CP_ERR_WORKSPACE if capacity is too small, CP_ERR_UNSUPPORTED if the table
 * would need more than 1 GiB of device scratch.  Synchronous: allocates and
 * frees device scratch, synchronises `stream`. */
int cp_tile_classes(const cp_plan_t *plan, int32_t *host_rows, int64_t capacity, int64_t *n_rows,
                    cudaStream_t stream);

/* Self-test of the device-side failure detection (no counterpart in the
 * pages: it checks this library's own bounded waits).  Launches one small
 * kernel in which one role waits on a barrier that nothing completes: after
 * limit_us microseconds (1 .. 1000000) it gives up, records
 * CP_ERR_DEVICE_TIMEOUT in the status word read by cp_get_status and raises
 * the CTA's abort flag; a second role, waiting on a barrier only the first
 * would have completed, must leave on that flag.  out3 (host, 3 ints):
 * [0] = 1 if the first wait timed out, [1] = 1 if the second left on the
 * abort, [2] = the second wait's duration in microseconds.  Synchronises
 * `stream`; the status word is left set for cp_get_status to read.  No
 * fault or trap: the context stays usable. */
int cp_selftest_wait_timeout(int32_t limit_us, int32_t *out3, cudaStream_t stream);

/* Self-test of the bounds record (no counterpart in the pages).  Launches
 * a 64-block kernel in which block `block` (0 .. 63) checks an index one
 * past the end of a small device buffer with the record routine of the
 * CP_DEBUG checks: the check fails, {CP_ERR_DEVICE_BOUNDS, block, line,
 * file id 1} is recorded in the status words (unless an earlier error is
 * already held there) and the store is skipped, so nothing outside the
 * buffer is touched.  *line (host) receives the source line the kernel
 * recorded.  Works in release and debug builds alike; synchronises
 * `stream`; the record is left for cp_get_status_detail to read. */
int cp_selftest_bounds(int32_t block, int32_t *line, cudaStream_t stream);

/* Rates behind the kernels' rooflines (no counterpart in the pages), each
 * timed with the SM clock inside one CTA per SM on the current device:
 * out2 (host, 2 doubles): [0] = ex2.approx.f32 results per SM clock (the
 * softmax's one exponential per visible query-key pair runs on this pipe),
 * [1] = SM clocks per tcgen05.mma M128 N128 K16 bf16 with A in tensor
 * memory and B in shared memory, back to back from one issuing warp.
 * Synchronous (allocates and frees a little device memory).  Returns
 * CP_ERR_ARCH on a device other than sm_103. */
int cp_measure_rates(double *out2, cudaStream_t stream);

/* SM clocks per warp-wide check of an mbarrier phase that has already
 * completed (mbarrier.try_wait in all 32 lanes, then a vote), measured as a
 * dependent chain in one warp (no counterpart in the pages): the fixed cost
 * that the MMA-issuing warp of each kernel pays at every barrier check
 * between two groups of MMAs.  *cycles (host, 1 double).  Synchronous;
 * CP_ERR_INVALID_ARG for a null pointer, CP_ERR_ARCH on a device other than
 * sm_103. */
int cp_measure_barrier_check(double *cycles, cudaStream_t stream);

/* Allocation-free variant of the emit-partials forward (no counterpart in
 * the paper: it exists for callers, not for the method).
 *
 * Some callers cannot call cudaMalloc at all: a plugin running inside a host
 * framework that owns the device allocator, a runtime whose device-memory
 * budget is fixed at start-up, or a latency-critical loop that must not
 * take cudaMalloc's implicit device synchronisation.  This entry point
 * computes exactly what cp_attn_fwd computes for a plan created with
 * emit_partials = 1 (per-ring-step partials, then their merge), but keeps the
 * partials in a static device array of CP_NOALLOC_SCRATCH_BYTES compiled into
 * the library instead of a caller-provided workspace, and calls no
 * allocating function.  The caller still passes q, k, v, o, lse (same
 * layouts as cp_attn_fwd).
 *  - Every GPU that loads the library holds the array until the process exits.
 *  - The first call on a device resolves the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  The per-device address cache is atomic, so
 *    first calls from several host threads at once are safe.
 *  - All calls share the one array: calls whose kernels overlap on the GPU
 *    (different streams, no ordering between them) race on it.  Every
 *    partial a call reads was written earlier by the same call, so nothing
 *    needs clearing between calls.
 *  - Returns CP_ERR_WORKSPACE if the partials need more than
 *    CP_NOALLOC_SCRATCH_BYTES (R * L * Hq * (d + 1) * 4 bytes, each part
 *    rounded up to 256), CP_ERR_INVALID_ARG if the plan was not created with
 *    emit_partials = 1. */
#define CP_NOALLOC_SCRATCH_BYTES (8u << 20)
int cp_attn_fwd_noalloc(const cp_plan_t *plan, const void *q, const void *k, const void *v,
                        void *o, float *lse, cudaStream_t stream);

/* Synchronise `stream`, then read and clear the device status word:
 * *dev_code = 0 or the first CP_ERR_DEVICE_* code any kernel recorded since
 * the last call.  Returns CP_OK or CP_ERR_CUDA. */
int cp_get_status(cudaStream_t stream, int32_t *dev_code);

/* As cp_get_status, with the whole record: out4 (host, 4 ints) = {code,
 * block, source line, file id}.  The last three are set only for
 * CP_ERR_DEVICE_BOUNDS, which only debug builds record (file ids: 1 the C-ABI
 * layer, 2 the forward kernel, 3 the backward kernels, 4 reshard and
 * gather, 5 merge); otherwise 0.  Reads and clears all four words.
 *
 * Debug builds (compiled with -DCP_DEBUG, the library libcpattn_debug.so)
 * check every work item, global index and TMA coordinate of the kernels;
 * a failed check records CP_ERR_DEVICE_BOUNDS here and skips the access
 * (a TMA load is still issued: the hardware fills out-of-range rows with
 * zeros).  Release builds contain no checks. */
int cp_get_status_detail(cudaStream_t stream, int32_t *out4);

/* 1 if this library was built with -DCP_DEBUG, else 0. */
int cp_debug_build(void);

/* Static string for a return code. */
const char *cp_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* CP_ATTN_H */
