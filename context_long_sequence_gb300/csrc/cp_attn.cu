// cp_attn.cu -- the C ABI (include/cp_attn.h): plan validation and tables,
// workspace sizing, argument checks, and the order of kernel launches for
// each entry point.  Host code only; the kernels live in attn_fwd.cu,
// attn_bwd.cu, reshard.cu and merge.cu.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#define CP_TU_ID ::cpattn::kTuCpAttn
#include "cp_attn.h"
#include "debug.cuh"
#include "kernels.h"
#include "ptx.cuh"

using cpattn::AttnGeom;
using cpattn::WorkItem;

// Device status words: [0] the first device-side error code since the last
// cp_get_status(); for a bounds record of a debug build [1] the block, [2]
// the source line and [3] the file id of the failed check.
__device__ int32_t g_cp_status[4];

namespace {
// NVTX range around one phase of an entry point, for timeline tools and for
// `ncu --nvtx` filters.  Host-side: it brackets the asynchronous launches of
// the phase, not their execution.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace

struct cp_plan {
  cp_plan_desc_t desc;
  std::vector<int32_t> offsets;  // empty: one document
  int P, n, T, chunk, nchunks;
  float scale;
  bool on_device;
  int device;
  std::vector<int32_t> chunk_pos;  // balanced layout: [R][nchunks] first position of each chunk
  int32_t* d_chunk_pos;          // device copy, or null
  std::vector<int32_t> chunk_own;  // balanced layout: position chunk -> r * nchunks + k
  int32_t* d_chunk_own;          // device copy, or null
  int32_t* d_doc_start;          // [L] or null
  int32_t* d_doc_end;            // [L] or null
  WorkItem* d_items_fused;       // forward: 256-row query blocks, all ring steps
  int n_items_fused;
  WorkItem* d_items_byu;         // the same grouped by Ulysses member (stream-major launch order), or null
  int n_items_u;                 // items per member
  WorkItem* d_items_q_byu;       // backward query tiles grouped by Ulysses member, or null
  int n_items_q_u;
  WorkItem* d_items_kv_byu;      // backward key tiles grouped by Ulysses member, or null
  int n_items_kv_u;
  WorkItem* d_items_q;           // backward dQ: 128-row query tiles
  int n_items_q;
  WorkItem* d_items_steps;       // emit-partials: one item per (256-row query block, ring step)
  int n_items_steps;
  WorkItem* d_items_kv;          // backward: key tiles
  int n_items_kv;
  WorkItem* d_items_rank;        // the fused list grouped by attention rank (cp_attn_fwd_rank)
  std::vector<int> rank_item_off;  // [P + 1] offsets into d_items_rank
  WorkItem* d_items_q_rank;      // backward query tiles grouped by attention rank (cp_attn_bwd_step)
  std::vector<int> q_rank_off;   // [P + 1]
  WorkItem* d_items_kv_rank;     // backward key tiles grouped by owner rank (cp_attn_bwd_step)
  std::vector<int> kv_rank_off;  // [P + 1]
};

namespace {

constexpr int kTile = 128;

// Device address of the status words on the current device, resolved once
// per device (an atomic cache: concurrent first calls store the same value).
int32_t* status_ptr() {
  static std::atomic<int32_t*> ptrs[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  int32_t* cached = ptrs[dev].load(std::memory_order_acquire);
  if (!cached) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_cp_status) != cudaSuccess) return nullptr;
    cached = static_cast<int32_t*>(p);
    ptrs[dev].store(cached, std::memory_order_release);
  }
  return cached;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int doc_start_host(const cp_plan* p, int pos) {
  if (p->offsets.empty()) return 0;
  auto it = std::upper_bound(p->offsets.begin(), p->offsets.end(), pos);
  return *(it - 1);
}

// Geometry for the kernels (device tables) or for host-side walks of the
// same index arithmetic (host copy of the chunk table).
AttnGeom geom(const cp_plan* p, bool on_host = false) {
  AttnGeom g;
  const cp_plan_desc_t& d = p->desc;
  g.L = d.L;
  g.R = d.ring_degree;
  g.U = d.ulysses_degree;
  g.T = p->T;
  g.Hq_loc = d.Hq / d.ulysses_degree;
  g.Hkv_loc = d.Hkv / d.ulysses_degree;
  g.G = d.Hq / d.Hkv;
  g.layout = d.layout;
  g.chunk = p->chunk;
  g.nchunks = p->nchunks;
  g.chunk_pos = p->chunk_pos.empty() ? nullptr : (on_host ? p->chunk_pos.data() : p->d_chunk_pos);
  g.chunk_owner = p->chunk_own.empty() ? nullptr : (on_host ? p->chunk_own.data() : p->d_chunk_own);
  g.kv_global = d.kv_exchange == CP_KV_ALLGATHER ? 1 : 0;
  g.scale = p->scale;
  g.doc_start = p->d_doc_start;
  g.doc_end = p->d_doc_end;
  return g;
}

// Number of 128-key tiles the forward kernel visits for a query tile (the
// same walk as the kernel's, evaluated on the host for scheduling).
int visited_tiles(const cp_plan* p, const AttnGeom& g, int r, int q0, int len, int s_begin, int s_end) {
  const int qpos0 = cpattn::slot_pos(g, r, q0);
  const int qpos_last = qpos0 + len - 1;
  const int lo_min = doc_start_host(p, qpos0);
  if (g.kv_global) return qpos_last / kTile - lo_min / kTile + 1;
  int count = 0;
  for (int s = s_begin; s < s_end; ++s) {
    const int src = (r - s + g.R) % g.R;
    for (int ch = 0; ch < p->nchunks; ++ch) {
      const int cpos0 = cpattn::slot_pos(g, src, ch * g.chunk);
      const int lo = std::max(cpos0, lo_min);
      const int hi = std::min(cpos0 + g.chunk - 1, qpos_last);
      if (lo > hi) continue;
      count += (hi - cpos0) / kTile - (lo - cpos0) / kTile + 1;
    }
  }
  return count;
}

// The forward over every rank and ring step in one launch: the items
// grouped by Ulysses member, launched stream-major (see FwdArgs), when the
// grouping exists; else the plain longest-first list.
void set_fused_items(const cp_plan* p, cpattn::FwdArgs& a) {
  if (p->d_items_byu) {
    a.items = p->d_items_byu;
    a.stream_major = 1;
    a.n_items_u = p->n_items_u;
  } else {
    a.items = p->d_items_fused;
  }
  a.n_items = p->n_items_fused;
}

// `items` (longest first) grouped by Ulysses member u = a % U, keeping the
// order within each group; empty when the members' counts differ.
std::vector<WorkItem> group_by_member(const std::vector<WorkItem>& items, int U, int* per_member) {
  std::vector<WorkItem> out;
  std::vector<int> cnt(U, 0);
  for (int uu = 0; uu < U; ++uu)
    for (const WorkItem& it : items)
      if (it.a % U == uu) {
        out.push_back(it);
        ++cnt[uu];
      }
  *per_member = cnt[0];
  if (std::count(cnt.begin(), cnt.end(), cnt[0]) != U) out.clear();
  return out;
}

// Query blocks of `rows` slots, ordered by descending work (longest first
// onto the SMs).
std::vector<WorkItem> build_items(const cp_plan* p, bool per_step, int rows) {
  const AttnGeom g = geom(p, true);
  struct Keyed {
    int work;
    WorkItem it;
  };
  std::vector<Keyed> v;
  const int A = g.R * g.U;
  for (int a = 0; a < A; ++a) {
    const int r = a / g.U;
    for (int ch = 0; ch < p->nchunks; ++ch)
      for (int t0 = 0; t0 < p->chunk; t0 += rows) {
        const int q0 = ch * p->chunk + t0;
        const int len = std::min(rows, p->chunk - t0);
        if (per_step) {
          for (int s = 0; s < g.R; ++s)
            v.push_back({visited_tiles(p, g, r, q0, len, s, s + 1), WorkItem{a, q0, len, s}});
        } else {
          v.push_back({visited_tiles(p, g, r, q0, len, 0, g.R), WorkItem{a, q0, len, -1}});
        }
      }
  }
  std::stable_sort(v.begin(), v.end(), [](const Keyed& x, const Keyed& y) { return x.work > y.work; });
  std::vector<WorkItem> out(v.size());
  for (size_t i = 0; i < v.size(); ++i) out[i] = v[i].it;
  return out;
}

// Work-balanced layout ([L3P] "Long context changes more than attention
// cost": split by actual attention work; [MTX] "Split heads or rotate KV":
// causal load balancing).  m*R equal chunks; a query at position i costs
// i - doc_start(i) + 1 visible keys.  Chunks go, from most to least work
// (equal work: lower chunk first), to the least-loaded rank that still holds
// fewer than m chunks (equal load: lower rank first); each rank keeps its
// chunks in position order.  Fills p->chunk_pos[r * m + k].
void balanced_chunk_table(cp_plan* p) {
  const int R = p->desc.ring_degree, m = p->nchunks, C = R * m, c = p->chunk;
  std::vector<long long> work(C, 0);
  for (int j = 0; j < C; ++j) {
    int ds = doc_start_host(p, j * c);
    for (int i = j * c; i < (j + 1) * c; ++i) {
      if (!p->offsets.empty() && std::binary_search(p->offsets.begin(), p->offsets.end(), i)) ds = i;
      work[j] += i - ds + 1;
    }
  }
  std::vector<int> order(C);
  for (int j = 0; j < C; ++j) order[j] = j;
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return work[x] > work[y]; });
  std::vector<long long> load(R, 0);
  std::vector<std::vector<int>> held(R);
  for (int j : order) {
    int best = -1;
    for (int r = 0; r < R; ++r)
      if (static_cast<int>(held[r].size()) < m && (best < 0 || load[r] < load[best])) best = r;
    held[best].push_back(j);
    load[best] += work[j];
  }
  p->chunk_pos.assign(static_cast<size_t>(C), 0);
  for (int r = 0; r < R; ++r) {
    std::sort(held[r].begin(), held[r].end());
    for (int k = 0; k < m; ++k) p->chunk_pos[static_cast<size_t>(r) * m + k] = held[r][k] * c;
  }
  p->chunk_own.assign(static_cast<size_t>(C), 0);
  for (int e = 0; e < C; ++e) p->chunk_own[p->chunk_pos[e] / c] = e;
}

int doc_end_host(const cp_plan* p, int pos) {
  if (p->offsets.empty()) return p->desc.L;
  return *std::upper_bound(p->offsets.begin(), p->offsets.end(), pos);
}

// Number of (query tile, query head) steps the backward's key-tile kernel
// walks for a key tile (the kernel's walk, evaluated on the host).
int visited_q_tiles(const cp_plan* p, const AttnGeom& g, int src, int k0, int len) {
  const int kpos0 = cpattn::slot_pos(g, src, k0);
  const int hi_max = doc_end_host(p, kpos0 + len - 1) - 1;
  int count = 0;
  for (int s = 0; s < g.R; ++s) {
    const int rr = (src + s) % g.R;
    for (int ch = 0; ch < p->nchunks; ++ch) {
      const int cpos0 = cpattn::slot_pos(g, rr, ch * g.chunk);
      const int lo = std::max(cpos0, kpos0);
      const int hi = std::min(cpos0 + g.chunk - 1, hi_max);
      if (lo > hi) continue;
      count += (hi - cpos0) / kTile - (lo - cpos0) / kTile + 1;
    }
  }
  return count;
}

// Key tiles of every attention rank a = src * U + u, ordered by descending work.
std::vector<WorkItem> build_kv_items(const cp_plan* p) {
  const AttnGeom g = geom(p, true);
  std::vector<std::pair<int, WorkItem>> v;
  for (int a = 0; a < g.R * g.U; ++a)
    for (int ch = 0; ch < p->nchunks; ++ch)
      for (int t0 = 0; t0 < p->chunk; t0 += kTile) {
        const int k0 = ch * p->chunk + t0;
        const int len = std::min(kTile, p->chunk - t0);
        v.push_back({visited_q_tiles(p, g, a / g.U, k0, len), WorkItem{a, k0, len, -1}});
      }
  std::stable_sort(v.begin(), v.end(), [](const std::pair<int, WorkItem>& x, const std::pair<int, WorkItem>& y) {
    return x.first > y.first;
  });
  std::vector<WorkItem> out(v.size());
  for (size_t i = 0; i < v.size(); ++i) out[i] = v[i].second;
  return out;
}

// A copy of `items` grouped by attention rank (stable: each group keeps the
// list's order), with the group offsets [P + 1].
std::vector<WorkItem> group_by_rank(const std::vector<WorkItem>& items, int P, std::vector<int>* off) {
  std::vector<WorkItem> by_rank(items);
  std::stable_sort(by_rank.begin(), by_rank.end(), [](const WorkItem& x, const WorkItem& y) { return x.a < y.a; });
  off->assign(P + 1, 0);
  for (const WorkItem& it : by_rank) ++(*off)[it.a + 1];
  for (int a = 0; a < P; ++a) (*off)[a + 1] += (*off)[a];
  return by_rank;
}

template <typename T>
int upload(const std::vector<T>& h, T** d) {
  *d = nullptr;
  if (h.empty()) return CP_OK;
  if (cudaMalloc(reinterpret_cast<void**>(d), h.size() * sizeof(T)) != cudaSuccess) return CP_ERR_CUDA;
  if (cudaMemcpy(*d, h.data(), h.size() * sizeof(T), cudaMemcpyHostToDevice) != cudaSuccess) return CP_ERR_CUDA;
  return CP_OK;
}

int check_device(const cp_plan* p) {
  if (!p->on_device) return CP_ERR_CUDA;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CP_ERR_CUDA;
  if (dev != p->device) return CP_ERR_INVALID_ARG;
  return CP_OK;
}

struct FwdWorkspace {
  size_t opart, lsepart, kall, vall, total;
};

FwdWorkspace fwd_workspace(const cp_plan* p) {
  const cp_plan_desc_t& d = p->desc;
  const size_t L = d.L;
  FwdWorkspace w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align256(bytes);
    return at;
  };
  if (d.emit_partials) {
    w.opart = take(static_cast<size_t>(d.ring_degree) * L * d.Hq * d.d * 4);
    w.lsepart = take(static_cast<size_t>(d.ring_degree) * L * d.Hq * 4);
  }
  if (d.kv_exchange == CP_KV_ALLGATHER) {  // the gathered K and V, in position order
    w.kall = take(L * d.Hkv * d.d * 2);
    w.vall = take(L * d.Hkv * d.d * 2);
  }
  w.total = off;
  return w;
}

struct BwdWorkspace {
  size_t nlse, nd, total;
};

// Query-tile-aligned length of one chunk in the backward's row statistics.
int chunk_pad_of(const cp_plan* p) { return (p->chunk + kTile - 1) / kTile * kTile; }

// Floats of one attention rank's statistics array (-LSE*log2e or -D):
// Hq/U heads x nchunks x chunk_pad slots.
size_t rank_ld_floats(const cp_plan* p) {
  return static_cast<size_t>(p->desc.Hq / p->desc.ulysses_degree) * p->nchunks * chunk_pad_of(p);
}

// The row statistics (-LSE*log2e and -D, chunk-padded).  With U > 1 the
// kernels address the sequence-sharded tensors directly: no copies.
BwdWorkspace bwd_workspace(const cp_plan* p) {
  BwdWorkspace w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align256(bytes);
    return at;
  };
  w.nlse = take(static_cast<size_t>(p->P) * rank_ld_floats(p) * 4);
  w.nd = take(static_cast<size_t>(p->P) * rank_ld_floats(p) * 4);
  w.total = off;
  return w;
}

}  // namespace

extern "C" {

int cp_plan_create(const cp_plan_desc_t* desc, cp_plan_t** out) {
  if (!desc || !out) return CP_ERR_INVALID_ARG;
  const cp_plan_desc_t& d = *desc;
  if (d.version != CP_ATTN_PLAN_VERSION) return CP_ERR_INVALID_ARG;
  if (d.L <= 0 || d.Hq <= 0 || d.Hkv <= 0 || d.ulysses_degree <= 0 || d.ring_degree <= 0) return CP_ERR_INVALID_ARG;
  if (d.Hq % d.Hkv) return CP_ERR_INVALID_ARG;
  if (d.layout != CP_LAYOUT_CONTIGUOUS && d.layout != CP_LAYOUT_ZIGZAG && d.layout != CP_LAYOUT_BALANCED)
    return CP_ERR_INVALID_ARG;
  if (d.layout == CP_LAYOUT_BALANCED && d.chunks_per_rank < 1) return CP_ERR_INVALID_ARG;
  if (d.num_docs < 0) return CP_ERR_INVALID_ARG;
  if (d.out_fp32 != 0 && d.out_fp32 != 1) return CP_ERR_INVALID_ARG;
  if (d.emit_partials != 0 && d.emit_partials != 1) return CP_ERR_INVALID_ARG;
  if (!(d.softmax_scale >= 0.f) || std::isinf(d.softmax_scale)) return CP_ERR_INVALID_ARG;
  if (d.d != 64 && d.d != 128) return CP_ERR_UNSUPPORTED;
  if (d.causal != 1) return CP_ERR_UNSUPPORTED;
  if (d.Hkv % d.ulysses_degree) return CP_ERR_UNSUPPORTED;  // KV heads cap the A2A degree
  const int R = d.ring_degree, U = d.ulysses_degree;
  const int nchunks = d.layout == CP_LAYOUT_CONTIGUOUS ? 1 : d.layout == CP_LAYOUT_ZIGZAG ? 2 : d.chunks_per_rank;
  if (static_cast<long long>(nchunks) * R > d.L || d.L % (static_cast<long long>(nchunks) * R))
    return CP_ERR_INVALID_ARG;
  const int T = d.L / R;
  if (T % U) return CP_ERR_INVALID_ARG;
  if (d.emit_partials && U != 1) return CP_ERR_UNSUPPORTED;
  if (d.kv_exchange != CP_KV_RING && d.kv_exchange != CP_KV_ALLGATHER) return CP_ERR_INVALID_ARG;
  if (d.kv_exchange == CP_KV_ALLGATHER && (U != 1 || d.emit_partials)) return CP_ERR_UNSUPPORTED;
  // Index arithmetic in the kernels is 32-bit for positions and slots.
  if (static_cast<long long>(d.L) * U >= (1LL << 31)) return CP_ERR_UNSUPPORTED;

  cp_plan* p = new (std::nothrow) cp_plan();
  if (!p) return CP_ERR_INVALID_ARG;
  p->desc = d;
  p->desc.doc_offsets = nullptr;
  if (d.num_docs > 1) {
    if (!d.doc_offsets) {
      delete p;
      return CP_ERR_INVALID_ARG;
    }
    p->offsets.assign(d.doc_offsets, d.doc_offsets + d.num_docs + 1);
    bool ok = p->offsets.front() == 0 && p->offsets.back() == d.L;
    for (int i = 0; i < d.num_docs && ok; ++i) ok = p->offsets[i] < p->offsets[i + 1];
    if (!ok) {
      delete p;
      return CP_ERR_INVALID_ARG;
    }
  }
  p->P = R * U;
  p->T = T;
  p->n = T / U;
  p->nchunks = nchunks;
  p->chunk = T / p->nchunks;
  if (d.layout == CP_LAYOUT_BALANCED) balanced_chunk_table(p);
  p->d_chunk_pos = p->d_chunk_own = nullptr;
  p->scale = d.softmax_scale > 0.f ? d.softmax_scale : 1.0f / std::sqrt(static_cast<float>(d.d));
  p->on_device = false;
  p->d_doc_start = p->d_doc_end = nullptr;
  p->d_items_fused = p->d_items_q = p->d_items_steps = p->d_items_kv = p->d_items_rank = nullptr;
  p->d_items_q_rank = p->d_items_kv_rank = p->d_items_byu = p->d_items_q_byu = p->d_items_kv_byu = nullptr;
  p->n_items_u = p->n_items_q_u = p->n_items_kv_u = 0;
  p->n_items_fused = p->n_items_q = p->n_items_steps = p->n_items_kv = 0;

  // Device tables, when a CUDA device is present (host-only use -- index
  // maps, workspace sizes -- works without one).
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) == cudaSuccess && ndev > 0) {
    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
      delete p;
      return CP_ERR_CUDA;
    }
    if (prop.major != 10 || prop.minor != 3) {
      delete p;
      return CP_ERR_ARCH;
    }
    p->device = dev;
    int rc = CP_OK;
    if (!p->offsets.empty()) {
      std::vector<int32_t> ds(d.L), de(d.L);
      for (int i = 0; i < d.num_docs; ++i)
        for (int x = p->offsets[i]; x < p->offsets[i + 1]; ++x) {
          ds[x] = p->offsets[i];
          de[x] = p->offsets[i + 1];
        }
      rc = upload(ds, &p->d_doc_start);
      if (rc == CP_OK) rc = upload(de, &p->d_doc_end);
    }
    if (rc == CP_OK) rc = upload(p->chunk_pos, &p->d_chunk_pos);
    if (rc == CP_OK) rc = upload(p->chunk_own, &p->d_chunk_own);
    std::vector<WorkItem> fused = build_items(p, false, 2 * kTile);
    p->n_items_fused = static_cast<int>(fused.size());
    if (rc == CP_OK) rc = upload(fused, &p->d_items_fused);
    // The same items grouped by rank, each group keeping the longest-first order.
    if (rc == CP_OK) rc = upload(group_by_rank(fused, p->P, &p->rank_item_off), &p->d_items_rank);
    // And grouped by Ulysses member u = a % U (longest first within each),
    // when every member has the same number of items.
    if (rc == CP_OK) rc = upload(group_by_member(fused, U, &p->n_items_u), &p->d_items_byu);
    if (rc == CP_OK) {
      std::vector<WorkItem> qt = build_items(p, false, kTile);
      p->n_items_q = static_cast<int>(qt.size());
      rc = upload(qt, &p->d_items_q);
      if (rc == CP_OK) rc = upload(group_by_rank(qt, p->P, &p->q_rank_off), &p->d_items_q_rank);
      if (rc == CP_OK) rc = upload(group_by_member(qt, U, &p->n_items_q_u), &p->d_items_q_byu);
    }
    if (rc == CP_OK && d.emit_partials) {
      std::vector<WorkItem> steps = build_items(p, true, 2 * kTile);
      p->n_items_steps = static_cast<int>(steps.size());
      rc = upload(steps, &p->d_items_steps);
    }
    if (rc == CP_OK) {
      std::vector<WorkItem> kv = build_kv_items(p);
      p->n_items_kv = static_cast<int>(kv.size());
      rc = upload(kv, &p->d_items_kv);
      if (rc == CP_OK) rc = upload(group_by_rank(kv, p->P, &p->kv_rank_off), &p->d_items_kv_rank);
      if (rc == CP_OK) rc = upload(group_by_member(kv, U, &p->n_items_kv_u), &p->d_items_kv_byu);
    }
    if (rc != CP_OK) {
      cudaFree(p->d_items_q_rank);
      cudaFree(p->d_items_kv_rank);
      cudaFree(p->d_items_byu);
      cudaFree(p->d_items_q_byu);
      cudaFree(p->d_items_kv_byu);
      cudaFree(p->d_items_rank);
      cudaFree(p->d_chunk_pos);
      cudaFree(p->d_chunk_own);
      cudaFree(p->d_doc_start);
      cudaFree(p->d_doc_end);
      cudaFree(p->d_items_fused);
      cudaFree(p->d_items_q);
      cudaFree(p->d_items_steps);
      cudaFree(p->d_items_kv);
      delete p;
      return rc;
    }
    p->on_device = true;
  }
  *out = p;
  return CP_OK;
}

void cp_plan_destroy(cp_plan_t* p) {
  if (!p) return;
  if (p->on_device) {
    cudaFree(p->d_items_q_rank);
    cudaFree(p->d_items_kv_rank);
    cudaFree(p->d_items_byu);
    cudaFree(p->d_items_q_byu);
    cudaFree(p->d_items_kv_byu);
    cudaFree(p->d_items_rank);
    cudaFree(p->d_chunk_pos);
    cudaFree(p->d_chunk_own);
    cudaFree(p->d_doc_start);
    cudaFree(p->d_doc_end);
    cudaFree(p->d_items_fused);
    cudaFree(p->d_items_q);
    cudaFree(p->d_items_steps);
    cudaFree(p->d_items_kv);
  }
  delete p;
}

int cp_index_map(const cp_plan_t* p, int32_t* host_out) {
  if (!p || !host_out) return CP_ERR_INVALID_ARG;
  const AttnGeom g = geom(p, true);
  // Sequence-sharded slot order: rank g = r*U + u holds ring-local slots
  // [u*n, (u+1)*n) of ring rank r, so the slot order is ring rank major.
  for (int r = 0; r < g.R; ++r)
    for (int t = 0; t < g.T; ++t) host_out[static_cast<size_t>(r) * g.T + t] = cpattn::slot_pos(g, r, t);
  return CP_OK;
}

int cp_workspace_size(const cp_plan_t* p, int op, size_t* bytes) {
  if (!p || !bytes) return CP_ERR_INVALID_ARG;
  if (op == CP_OP_FWD)
    *bytes = fwd_workspace(p).total;
  else if (op == CP_OP_BWD)
    *bytes = bwd_workspace(p).total;
  else if (op == CP_OP_BWD_RANK_STATS)
    *bytes = 2 * rank_ld_floats(p) * 4;
  else
    return CP_ERR_INVALID_ARG;
  return CP_OK;
}

namespace {
// Argument checks of one reshard; *bytes = size of its input (= output).
int check_reshard_job(const cp_plan_t* p, const cp_reshard_job_t& j, size_t* bytes) {
  if (!j.in || !j.out) return CP_ERR_INVALID_ARG;
  if (j.direction != CP_SEQ_TO_HEAD && j.direction != CP_HEAD_TO_SEQ) return CP_ERR_INVALID_ARG;
  if (j.tensor_kind != CP_TOKEN_MAJOR && j.tensor_kind != CP_HEAD_MAJOR) return CP_ERR_INVALID_ARG;
  const int U = p->desc.ulysses_degree;
  if (j.H <= 0 || j.row_elems <= 0 || j.elem_bytes <= 0 || j.H % U) return CP_ERR_INVALID_ARG;
  if (j.tensor_kind == CP_HEAD_MAJOR && j.row_elems != 1) return CP_ERR_INVALID_ARG;
  if (!aligned16(j.in) || !aligned16(j.out)) return CP_ERR_ALIGNMENT;
  *bytes = static_cast<size_t>(p->desc.L) * j.H * j.row_elems * j.elem_bytes;
  return CP_OK;
}

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const char* x = static_cast<const char*>(a);
  const char* y = static_cast<const char*>(b);
  return x < y + nb && y < x + na;
}
}  // namespace

int ulysses_reshard(const cp_plan_t* p, int direction, int tensor_kind, int H, int row_elems, int elem_bytes,
                    const void* in, void* out, cudaStream_t stream) {
  if (!p) return CP_ERR_INVALID_ARG;
  const cp_reshard_job_t job{direction, tensor_kind, H, row_elems, elem_bytes, in, out};
  return ulysses_reshard_batch(p, 1, &job, stream);
}

int ulysses_reshard_batch(const cp_plan_t* p, int n_jobs, const cp_reshard_job_t* jobs, cudaStream_t stream) {
  if (!p || !jobs || n_jobs < 1 || n_jobs > CP_RESHARD_MAX_JOBS) return CP_ERR_INVALID_ARG;
  size_t bytes[CP_RESHARD_MAX_JOBS];
  for (int i = 0; i < n_jobs; ++i) {
    const int rc = check_reshard_job(p, jobs[i], &bytes[i]);
    if (rc != CP_OK) return rc;
  }
  // The jobs run concurrently: no output may overlap any input or another output.
  for (int i = 0; i < n_jobs; ++i)
    for (int k = 0; k < n_jobs; ++k) {
      if (overlap(jobs[i].out, bytes[i], jobs[k].in, bytes[k])) return CP_ERR_INVALID_ARG;
      if (k != i && overlap(jobs[i].out, bytes[i], jobs[k].out, bytes[k])) return CP_ERR_INVALID_ARG;
    }
  int rc = check_device(p);
  if (rc != CP_OK) return rc;
  cpattn::ReshardSpec spec[CP_RESHARD_MAX_JOBS];
  for (int i = 0; i < n_jobs; ++i)
    spec[i] = cpattn::ReshardSpec{jobs[i].H, jobs[i].row_elems, jobs[i].direction, jobs[i].tensor_kind,
                                  jobs[i].elem_bytes, jobs[i].in, jobs[i].out};
  NvtxRange range("ulysses_reshard");
  return cpattn::launch_reshard_batch(p->desc.ring_degree, p->desc.ulysses_degree, p->n, spec, n_jobs, stream,
                                      status_ptr());
}

int cp_attn_fwd(const cp_plan_t* p, const void* q, const void* k, const void* v, void* o, float* lse,
                void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!p || !q || !k || !v || !o || !lse) return CP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      (workspace && !aligned16(workspace)))
    return CP_ERR_ALIGNMENT;
  int rc = check_device(p);
  if (rc != CP_OK) return rc;
  const FwdWorkspace w = fwd_workspace(p);
  if (w.total > 0 && (!workspace || workspace_bytes < w.total)) return CP_ERR_WORKSPACE;
  const cp_plan_desc_t& d = p->desc;
  char* ws = static_cast<char*>(workspace);
  NvtxRange call("cp_attn_fwd");
  cpattn::FwdArgs a{};
  a.g = geom(p);
  a.d = d.d;
  a.o_fp32 = d.out_fp32;
  a.status = status_ptr();
  if (!a.status) return CP_ERR_CUDA;
  if (d.ulysses_degree == 1) {
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.lse = lse;
    if (d.emit_partials) {
      a.o_part = reinterpret_cast<float*>(ws + w.opart);
      a.lse_part = reinterpret_cast<float*>(ws + w.lsepart);
      a.items = p->d_items_steps;
      a.n_items = p->n_items_steps;
      {
        NvtxRange phase("attention_partials");
        if ((rc = cpattn::launch_attn_fwd(a, stream))) return rc;
      }
      NvtxRange phase("merge");
      return cpattn::launch_merge(d.ring_degree, d.ring_degree, p->T, d.Hq, d.d, a.o_part, a.lse_part, o, lse,
                                  d.out_fp32, stream, a.status);
    }
    if (d.kv_exchange == CP_KV_ALLGATHER) {
      // All-gather: K and V of every rank to their positions, then each
      // rank's queries attend over the gathered sequence.
      const long long row_bytes = static_cast<long long>(d.Hkv) * d.d * 2;
      NvtxRange phase("gather_kv");
      if ((rc = cpattn::launch_gather_rows(a.g, row_bytes, k, ws + w.kall, stream, a.status)) ||
          (rc = cpattn::launch_gather_rows(a.g, row_bytes, v, ws + w.vall, stream, a.status)))
        return rc;
      a.k = ws + w.kall;
      a.v = ws + w.vall;
    }
    set_fused_items(p, a);
    NvtxRange phase("attention");
    return cpattn::launch_attn_fwd(a, stream);
  }
  // Ulysses / USP: with every rank in this GPU's memory, the two exchanges
  // ([MTX] "Split heads or rotate KV": tokens to heads before attention,
  // heads to tokens after it) are the kernel's addressing.  Ring rank r's U
  // members hold its T ring-local slots in order, so member u's head-sharded
  // rows are the sequence-sharded rows r*T + t restricted to its heads: the
  // kernel reads Q, K, V and writes O and LSE in the API layout directly.
  // ulysses_reshard is the same exchange as a copy, for callers that want
  // the head-sharded tensors (cp_attn_fwd_local, the backward).
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.seq_io = 1;
  set_fused_items(p, a);
  NvtxRange phase("attention");
  return cpattn::launch_attn_fwd(a, stream);
}

int cp_attn_fwd_local(const cp_plan_t* p, const void* q, const void* k, const void* v, void* o, float* lse,
                      cudaStream_t stream) {
  if (!p || !q || !k || !v || !o || !lse) return CP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return CP_ERR_ALIGNMENT;
  int rc = check_device(p);
  if (rc != CP_OK) return rc;
  cpattn::FwdArgs a{};
  a.g = geom(p);
  a.d = p->desc.d;
  a.o_fp32 = p->desc.out_fp32;
  a.status = status_ptr();
  if (!a.status) return CP_ERR_CUDA;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  set_fused_items(p, a);
  NvtxRange call("cp_attn_fwd_local");
  return cpattn::launch_attn_fwd(a, stream);
}

int cp_attn_fwd_rank(const cp_plan_t* p, int rank, const void* q, const void* k, const void* v, void* o, float* lse,
                     cudaStream_t stream) {
  if (!p || !q || !k || !v || !o || !lse) return CP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return CP_ERR_ALIGNMENT;
  if (rank < 0 || rank >= p->P) return CP_ERR_INVALID_ARG;
  int rc = check_device(p);
  if (rc != CP_OK) return rc;
  cpattn::FwdArgs a{};
  a.g = geom(p);
  a.d = p->desc.d;
  a.o_fp32 = p->desc.out_fp32;
  a.status = status_ptr();
  if (!a.status) return CP_ERR_CUDA;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.items = p->d_items_rank + p->rank_item_off[rank];
  a.n_items = p->rank_item_off[rank + 1] - p->rank_item_off[rank];
  NvtxRange call("cp_attn_fwd_rank");
  return cpattn::launch_attn_fwd(a, stream);
}

int cp_attn_bwd(const cp_plan_t* p, const void* q, const void* k, const void* v, const void* o, const float* lse,
                const void* dO, float* dq, float* dk, float* dv, void* workspace, size_t workspace_bytes,
                cudaStream_t stream) {
  if (!p || !q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return CP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dO) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || (workspace && !aligned16(workspace)))
    return CP_ERR_ALIGNMENT;
  int rc = check_device(p);
  if (rc != CP_OK) return rc;
  const BwdWorkspace w = bwd_workspace(p);
  if (!workspace || workspace_bytes < w.total) return CP_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cpattn::BwdArgs a{};
  a.g = geom(p);
  a.g.kv_global = 0;  // the backward walks the ring order over the owners' K/V slots
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.dO = dO;
  a.o_fp32 = p->desc.out_fp32;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.nlse = reinterpret_cast<float*>(ws + w.nlse);
  a.nd = reinterpret_cast<float*>(ws + w.nd);
  a.chunk_pad = chunk_pad_of(p);
  a.items_q = p->d_items_q;
  a.n_items_q = p->n_items_q;
  a.items_kv = p->d_items_kv;
  a.n_items_kv = p->n_items_kv;
  if (p->d_items_q_byu && p->d_items_kv_byu) {  // stream-major launch order (see BwdArgs)
    a.items_q = p->d_items_q_byu;
    a.items_kv = p->d_items_kv_byu;
    a.stream_major = 1;
    a.n_items_q_u = p->n_items_q_u;
    a.n_items_kv_u = p->n_items_kv_u;
  }
  a.d = p->desc.d;
  a.status = status_ptr();
  if (!a.status) return CP_ERR_CUDA;
  const cp_plan_desc_t& d = p->desc;
  NvtxRange call("cp_attn_bwd");
  // Ulysses / USP: the forward's exchanges run in reverse for the gradients
  // ([MTX] "Split heads or rotate KV").  As in the forward, with every rank
  // in this GPU's memory they are the kernels' addressing: member u of ring
  // rank r reads q, k, v, o, dO, LSE and writes dq, dk, dv at rows r*T.. and
  // its own heads of the sequence-sharded tensors.
  a.seq_io = d.ulysses_degree > 1 ? 1 : 0;
  NvtxRange phase("attention_bwd");
  return cpattn::launch_attn_bwd(a, stream);
}

int cp_attn_fwd_step(const cp_plan_t* p, int rank, int step, const void* q_rank, const void* k_chunk,
                     const void* v_chunk, float* o_part, float* lse_part, cudaStream_t stream) {
  if (!p || !q_rank || !k_chunk || !v_chunk || !o_part || !lse_part) return CP_ERR_INVALID_ARG;
  if (!aligned16(q_rank) || !aligned16(k_chunk) || !aligned16(v_chunk) || !aligned16(o_part) || !aligned16(lse_part))
    return CP_ERR_ALIGNMENT;
  if (rank < 0 || rank >= p->P || step < 0 || step >= p->desc.ring_degree) return CP_ERR_INVALID_ARG;
  if (p->desc.kv_exchange != CP_KV_RING) return CP_ERR_UNSUPPORTED;
  int rc = check_device(p);
  if (rc != CP_OK) return rc;
  cpattn::FwdArgs a{};
  a.g = geom(p);
  a.d = p->desc.d;
  a.status = status_ptr();
  if (!a.status) return CP_ERR_CUDA;
  a.q = q_rank;
  a.k = k_chunk;
  a.v = v_chunk;
  a.o = o_part;  // unused in partial mode; non-null for the launcher
  a.lse = lse_part;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.items = p->d_items_rank + p->rank_item_off[rank];
  a.n_items = p->rank_item_off[rank + 1] - p->rank_item_off[rank];
  a.rank_local = 1;
  a.step = step;
  NvtxRange call("cp_attn_fwd_step");
  return cpattn::launch_attn_fwd(a, stream);
}

int cp_attn_bwd_delta(const cp_plan_t* p, const void* o_rank, const void* do_rank, const float* lse_rank,
                      float* stats_rank, cudaStream_t stream) {
  if (!p || !o_rank || !do_rank || !lse_rank || !stats_rank) return CP_ERR_INVALID_ARG;
  if (!aligned16(o_rank) || !aligned16(do_rank) || !aligned16(lse_rank) || !aligned16(stats_rank))
    return CP_ERR_ALIGNMENT;
  int rc = check_device(p);
  if (rc != CP_OK) return rc;
  cpattn::BwdArgs a{};
  a.g = geom(p);
  a.g.kv_global = 0;
  a.o = o_rank;
  a.dO = do_rank;
  a.lse = lse_rank;
  a.o_fp32 = p->desc.out_fp32;
  a.nlse = stats_rank;
  a.nd = stats_rank + rank_ld_floats(p);
  a.chunk_pad = chunk_pad_of(p);
  // The launcher also builds the four tensor maps: point them at valid rows.
  a.q = a.k = a.v = do_rank;
  a.d = p->desc.d;
  a.rank_local = 1;
  a.phases = 1;
  a.status = status_ptr();
  if (!a.status) return CP_ERR_CUDA;
  NvtxRange call("cp_attn_bwd_delta");
  return cpattn::launch_attn_bwd(a, stream);
}

int cp_attn_bwd_step(const cp_plan_t* p, int rank, int step, const void* q_rank, const void* do_rank,
                     const float* stats_rank, const void* k_chunk, const void* v_chunk, float* dq_rank,
                     float* dk_chunk, float* dv_chunk, cudaStream_t stream) {
  if (!p || !q_rank || !do_rank || !stats_rank || !k_chunk || !v_chunk || !dq_rank || !dk_chunk || !dv_chunk)
    return CP_ERR_INVALID_ARG;
  if (!aligned16(q_rank) || !aligned16(do_rank) || !aligned16(stats_rank) || !aligned16(k_chunk) ||
      !aligned16(v_chunk) || !aligned16(dq_rank) || !aligned16(dk_chunk) || !aligned16(dv_chunk))
    return CP_ERR_ALIGNMENT;
  const int R = p->desc.ring_degree, U = p->desc.ulysses_degree;
  if (rank < 0 || rank >= p->P || step < 0 || step >= R) return CP_ERR_INVALID_ARG;
  if (p->desc.kv_exchange != CP_KV_RING) return CP_ERR_UNSUPPORTED;
  int rc = check_device(p);
  if (rc != CP_OK) return rc;
  const int r = rank / U, u = rank % U;
  const int a_src = ((r - step + R) % R) * U + u;  // owner of the visiting chunk
  cpattn::BwdArgs a{};
  a.g = geom(p);
  a.g.kv_global = 0;
  a.q = q_rank;
  a.dO = do_rank;
  a.nlse = const_cast<float*>(stats_rank);  // read only: phases exclude the delta kernel
  a.nd = const_cast<float*>(stats_rank) + rank_ld_floats(p);
  a.chunk_pad = chunk_pad_of(p);
  a.k = k_chunk;
  a.v = v_chunk;
  a.o = do_rank;  // not read (the delta phase is excluded)
  a.dq = dq_rank;
  a.dk = dk_chunk;
  a.dv = dv_chunk;
  a.items_q = p->d_items_q_rank + p->q_rank_off[rank];
  a.n_items_q = p->q_rank_off[rank + 1] - p->q_rank_off[rank];
  a.items_kv = p->d_items_kv_rank + p->kv_rank_off[a_src];
  a.n_items_kv = p->kv_rank_off[a_src + 1] - p->kv_rank_off[a_src];
  a.d = p->desc.d;
  a.rank_local = 1;
  a.step = step;
  a.accumulate = step > 0;  // step 0 writes every row; later steps add
  a.phases = 2 | 4;
  a.status = status_ptr();
  if (!a.status) return CP_ERR_CUDA;
  NvtxRange call("cp_attn_bwd_step");
  return cpattn::launch_attn_bwd(a, stream);
}

int cp_tile_classes(const cp_plan_t* p, int32_t* host_rows, int64_t capacity, int64_t* n_rows, cudaStream_t stream) {
  if (!p || !n_rows || capacity < 0 || (capacity > 0 && !host_rows)) return CP_ERR_INVALID_ARG;
  int rc = check_device(p);
  if (rc != CP_OK) return rc;
  const cp_plan_desc_t& d = p->desc;
  cpattn::FwdArgs a{};
  a.g = geom(p);
  a.d = d.d;
  a.status = status_ptr();
  if (!a.status) return CP_ERR_CUDA;
  const bool steps = d.emit_partials && d.ulysses_degree == 1;
  a.items = steps ? p->d_items_steps : p->d_items_fused;
  a.n_items = steps ? p->n_items_steps : p->n_items_fused;
  // Upper bound on the tiles one item walks: every chunk of every ring step
  // it covers, plus one for a chunk-unaligned start (position order when the
  // K/V are all-gathered).
  const long long per_chunk = (p->chunk + kTile - 1) / kTile + 1;
  const long long stride = a.g.kv_global ? (d.L + kTile - 1) / kTile + 1
                                         : static_cast<long long>(steps ? 1 : d.ring_degree) * p->nchunks * per_chunk;
  const long long cells = static_cast<long long>(a.n_items) * stride * 8;
  if (stride > 0x7fffffffLL || cells * 4 > (1LL << 30)) return CP_ERR_UNSUPPORTED;  // a debug call: 1 GiB at most
  *n_rows = 0;
  if (a.n_items == 0) return CP_OK;
  int32_t* d_rows = nullptr;
  int32_t* d_counts = nullptr;
  if (cudaMalloc(&d_rows, cells * 4) != cudaSuccess) return CP_ERR_CUDA;
  if (cudaMalloc(&d_counts, static_cast<size_t>(a.n_items) * 4) != cudaSuccess) {
    cudaFree(d_rows);
    return CP_ERR_CUDA;
  }
  std::vector<int32_t> counts(a.n_items), rows;
  rc = cpattn::launch_tile_classes(a, d_rows, d_counts, static_cast<int>(stride), stream);
  if (rc == CP_OK &&
      (cudaMemcpyAsync(counts.data(), d_counts, counts.size() * 4, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
       cudaStreamSynchronize(stream) != cudaSuccess))
    rc = CP_ERR_CUDA;
  long long total = 0;
  for (int i = 0; rc == CP_OK && i < a.n_items; ++i) {
    if (counts[i] > stride) rc = CP_ERR_UNSUPPORTED;  // the bound above is wrong: report, never truncate
    total += counts[i];
  }
  if (rc == CP_OK && host_rows && capacity >= total) {
    rows.resize(static_cast<size_t>(cells));
    if (cudaMemcpy(rows.data(), d_rows, cells * 4, cudaMemcpyDeviceToHost) != cudaSuccess) rc = CP_ERR_CUDA;
    long long o = 0;
    for (int i = 0; rc == CP_OK && i < a.n_items; ++i) {
      std::memcpy(host_rows + o * 8, rows.data() + static_cast<size_t>(i) * stride * 8,
                  static_cast<size_t>(counts[i]) * 8 * 4);
      o += counts[i];
    }
  }
  cudaFree(d_rows);
  cudaFree(d_counts);
  if (rc != CP_OK) return rc;
  *n_rows = total;
  return (host_rows && capacity < total) ? CP_ERR_WORKSPACE : CP_OK;
}

int cp_merge_lse(int n_parts, int rows, int H, int d, const float* o_parts, const float* lse_parts, void* o_out,
                 float* lse_out, cudaStream_t stream) {
  if (n_parts <= 0 || rows < 0 || H <= 0 || !o_parts || !lse_parts || !o_out || !lse_out) return CP_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return CP_ERR_UNSUPPORTED;
  if (!aligned16(o_parts) || !aligned16(lse_parts) || !aligned16(o_out) || !aligned16(lse_out))
    return CP_ERR_ALIGNMENT;
  NvtxRange call("cp_merge_lse");
  return cpattn::launch_merge(1, n_parts, rows, H, d, o_parts, lse_parts, o_out, lse_out, 0, stream, status_ptr());
}

int cp_get_status_detail(cudaStream_t stream, int32_t* out4) {
  if (!out4) return CP_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return CP_ERR_CUDA;
  int32_t rec[4] = {0, 0, 0, 0};
  const int32_t zero[4] = {0, 0, 0, 0};
  if (cudaMemcpyFromSymbol(rec, g_cp_status, sizeof(rec)) != cudaSuccess) return CP_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_cp_status, zero, sizeof(zero)) != cudaSuccess) return CP_ERR_CUDA;
  std::memcpy(out4, rec, sizeof(rec));
  return CP_OK;
}

int cp_get_status(cudaStream_t stream, int32_t* dev_code) {
  if (!dev_code) return CP_ERR_INVALID_ARG;
  int32_t rec[4];
  const int rc = cp_get_status_detail(stream, rec);
  if (rc != CP_OK) return rc;
  *dev_code = rec[0];
  return CP_OK;
}

int cp_debug_build(void) {
#ifdef CP_DEBUG
  return 1;
#else
  return 0;
#endif
}

const char* cp_strerror(int code) {
  switch (code) {
    case CP_OK: return "ok";
    case CP_ERR_INVALID_ARG: return "invalid argument";
    case CP_ERR_UNSUPPORTED: return "unsupported configuration";
    case CP_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
    case CP_ERR_CUDA: return "CUDA error";
    case CP_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case CP_ERR_DEVICE_BOUNDS: return "device-side index check failed";
    case CP_ERR_WORKSPACE: return "workspace missing or too small";
    case CP_ERR_ARCH: return "device is not sm_103";
    default: return "unknown error";
  }
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Self-test of the bounded waits (cp_selftest_wait_timeout).
//
// Two roles of one CTA, as in the attention kernels: warp 0 waits on an
// mbarrier that nothing will ever complete; after `limit_ns` its wait gives
// up, records CP_ERR_DEVICE_TIMEOUT and raises the CTA's abort flag.  Warp 1
// waits (with the production 2 s limit) on a barrier that only warp 0 would
// have completed, and must leave because of the abort flag, long before its
// own limit.  out[0] = 1 if warp 0 timed out, out[1] = 1 if warp 1 left on
// the abort, out[2] = warp 1's wait in microseconds.  No fault, no trap: the
// kernel returns normally and the context stays usable.
namespace {
__global__ void selftest_wait_kernel(uint64_t limit_ns, int32_t* status, int32_t* out) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    cpattn::mbar_init(cpattn::smem_u32(&bars[0]), 1);
    cpattn::mbar_init(cpattn::smem_u32(&bars[1]), 1);
    abort_flag = 0;
    cpattn::fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort = &abort_flag;
  if (warp == 0 && lane == 0) {
    const bool ok = cpattn::mbar_wait_limit(cpattn::smem_u32(&bars[0]), 0, abort, status, limit_ns);
    out[0] = ok ? 0 : 1;
  } else if (warp == 1 && lane == 0) {
    const uint64_t t0 = cpattn::globaltimer_ns();
    const bool ok = cpattn::mbar_wait(cpattn::smem_u32(&bars[1]), 0, abort, status);
    out[1] = (!ok && *abort) ? 1 : 0;
    out[2] = static_cast<int32_t>((cpattn::globaltimer_ns() - t0) / 1000);
  }
}
}  // namespace

extern "C" int cp_selftest_wait_timeout(int32_t limit_us, int32_t* out3, cudaStream_t stream) {
  if (limit_us <= 0 || limit_us > 1000000 || !out3) return CP_ERR_INVALID_ARG;
  int32_t* st = status_ptr();
  if (!st) return CP_ERR_CUDA;
  int32_t* d_out = nullptr;
  if (cudaMalloc(&d_out, 3 * sizeof(int32_t)) != cudaSuccess) return CP_ERR_CUDA;
  int rc = CP_OK;
  if (cudaMemsetAsync(d_out, 0, 3 * sizeof(int32_t), stream) != cudaSuccess) rc = CP_ERR_CUDA;
  if (rc == CP_OK) {
    selftest_wait_kernel<<<1, 64, 0, stream>>>(static_cast<uint64_t>(limit_us) * 1000, st, d_out);
    if (cudaGetLastError() != cudaSuccess) rc = CP_ERR_CUDA;
  }
  if (rc == CP_OK && (cudaMemcpyAsync(out3, d_out, 3 * sizeof(int32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
                      cudaStreamSynchronize(stream) != cudaSuccess))
    rc = CP_ERR_CUDA;
  cudaFree(d_out);
  return rc;
}

// ---------------------------------------------------------------------------
// Self-test of the bounds record (cp_selftest_bounds).
//
// Block `block` of a small grid checks the index one past the end of a
// 32-element buffer with the same record routine the CP_DEBUG checks use;
// the check fails, the record is written and the store is skipped.  Nothing
// outside the buffer is touched.  The kernel also stores the source line it
// recorded in buf[0], so the host can compare it with the record.
namespace {
__global__ void selftest_bounds_kernel(int32_t* status, int32_t* buf, int block) {
  if (static_cast<int>(blockIdx.x) != block || threadIdx.x != 0) return;
  const int n = 32, idx = n;  // one past the end
  const bool in = idx < n;
  const int line = __LINE__;
  if (!in) cpattn::debug_bounds_fail(status, line, cpattn::kTuCpAttn);
  if (in) buf[idx] = 1;
  buf[0] = line;
}
}  // namespace

extern "C" int cp_selftest_bounds(int32_t block, int32_t* line, cudaStream_t stream) {
  if (block < 0 || block >= 64 || !line) return CP_ERR_INVALID_ARG;
  int32_t* st = status_ptr();
  if (!st) return CP_ERR_CUDA;
  int32_t* d_buf = nullptr;
  if (cudaMalloc(&d_buf, 32 * sizeof(int32_t)) != cudaSuccess) return CP_ERR_CUDA;
  int rc = CP_OK;
  selftest_bounds_kernel<<<64, 32, 0, stream>>>(st, d_buf, block);
  if (cudaGetLastError() != cudaSuccess ||
      cudaMemcpyAsync(line, d_buf, sizeof(int32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    rc = CP_ERR_CUDA;
  cudaFree(d_buf);
  return rc;
}

// ---------------------------------------------------------------------------
// Rates behind the kernels' rooflines (cp_measure_rates): exp2 results per
// SM clock on the MUFU pipe (the softmax's one exponential per visible pair)
// and SM clocks per tcgen05.mma M128 N128 K16 (bf16, A in TMEM, B in shared
// memory: the PV form), each timed with clock64 inside one CTA per SM.
namespace {
constexpr int kRateEx2Threads = 512, kRateEx2Chains = 16, kRateEx2Iters = 1000;
constexpr int kRateMmaGroups = 200;

__global__ void __launch_bounds__(kRateEx2Threads) rate_ex2_kernel(unsigned long long* cyc, float* sink) {
  float a[kRateEx2Chains];
#pragma unroll
  for (int i = 0; i < kRateEx2Chains; ++i) a[i] = -1e-3f * static_cast<float>(threadIdx.x + i);
  __syncthreads();
  const unsigned long long t0 = clock64();
  for (int it = 0; it < kRateEx2Iters; ++it) {
#pragma unroll
    for (int i = 0; i < kRateEx2Chains; ++i) a[i] = cpattn::ex2_approx(a[i]) - 1.0f;  // stays in (-1, 0]
  }
  __syncthreads();
  const unsigned long long t1 = clock64();
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kRateEx2Chains; ++i) acc += a[i];
  if (acc == 1.0f) sink[threadIdx.x] = acc;  // never true; keeps the chains live
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

constexpr uint32_t kRateMmaSmem = 120 * 1024;  // one CTA per SM

__global__ void __launch_bounds__(128, 1) rate_mma_kernel(unsigned long long* cyc, int32_t* status) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sB = cpattn::smem_u32(sm);  // 32 KB: a 128 x 128 bf16 tile, two 64-column halves
  const uint32_t bar = cpattn::smem_u32(sm + 32768);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + 32768 + 16);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 32768 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sm)[i] = make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);
  if (threadIdx.x == 0) {
    cpattn::mbar_init(bar, 1);
    cpattn::fence_mbar_init();
  }
  if (warp == 0) {
    cpattn::tmem_alloc(cpattn::smem_u32(slot), 512);
    cpattn::tmem_relinquish();
  }
  cpattn::fence_proxy_async_smem();
  cpattn::tc_fence_before();
  __syncthreads();
  cpattn::tc_fence_after();
  const uint32_t tm = *slot;
  if (warp == 1) {
    constexpr uint32_t idesc = cpattn::idesc_bf16_f32(128, 128, 1);
    const uint64_t b = cpattn::smem_desc_sw128(sB, 128 * 128, 1024);
    const unsigned long long t0 = clock64();
    for (int it = 0; it < kRateMmaGroups; ++it) {
      cpattn::mma_bf16_ts_k64_warp(tm, tm + 256, b, idesc, 1u);
      cpattn::mma_bf16_ts_k64_warp(tm, tm + 256 + 32, b + 512, idesc, 1u);
    }
    cpattn::mma_commit_warp(bar);
    cpattn::mbar_wait(bar, 0, nullptr, status);
    if (lane == 0) cyc[blockIdx.x] = clock64() - t0;
  }
  cpattn::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    cpattn::tc_fence_after();
    cpattn::tmem_dealloc(tm, 512);
  }
}
}  // namespace

extern "C" int cp_measure_rates(double* out2, cudaStream_t stream) {
  if (!out2) return CP_ERR_INVALID_ARG;
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return CP_ERR_CUDA;
  if (major != 10 || minor != 3) return CP_ERR_ARCH;
  int32_t* st = status_ptr();
  if (!st) return CP_ERR_CUDA;
  unsigned long long* d_cyc = nullptr;
  float* d_sink = nullptr;
  if (cudaMalloc(&d_cyc, 2 * sms * sizeof(unsigned long long)) != cudaSuccess) return CP_ERR_CUDA;
  if (cudaMalloc(&d_sink, kRateEx2Threads * sizeof(float)) != cudaSuccess) {
    cudaFree(d_cyc);
    return CP_ERR_CUDA;
  }
  int rc = CP_OK;
  if (cudaFuncSetAttribute(rate_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRateMmaSmem) !=
      cudaSuccess)
    rc = CP_ERR_CUDA;
  // Each kernel runs twice and the second run is kept: the first launch of
  // the tensor-core kernel in a process runs measurably slower.
  for (int rep = 0; rc == CP_OK && rep < 2; ++rep) {
    rate_ex2_kernel<<<sms, kRateEx2Threads, 0, stream>>>(d_cyc, d_sink);
    rate_mma_kernel<<<sms, 128, kRateMmaSmem, stream>>>(d_cyc + sms, st);
    if (cudaGetLastError() != cudaSuccess) rc = CP_ERR_CUDA;
  }
  std::vector<unsigned long long> cyc(2 * sms);
  if (rc == CP_OK && (cudaMemcpyAsync(cyc.data(), d_cyc, cyc.size() * sizeof(unsigned long long),
                                      cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
                      cudaStreamSynchronize(stream) != cudaSuccess))
    rc = CP_ERR_CUDA;
  cudaFree(d_cyc);
  cudaFree(d_sink);
  if (rc != CP_OK) return rc;
  double ex2 = 0, mma = 0;
  for (int i = 0; i < sms; ++i) {
    ex2 += static_cast<double>(kRateEx2Threads) * kRateEx2Chains * kRateEx2Iters / static_cast<double>(cyc[i]);
    mma += static_cast<double>(cyc[sms + i]) / (kRateMmaGroups * 8.0);
  }
  out2[0] = ex2 / sms;
  out2[1] = mma / sms;
  return CP_OK;
}

// Latency of one warp-wide check of an mbarrier phase that has already
// completed (try_wait in every lane, then a vote): what the MMA-issuing
// warps pay at each wait between two MMA groups, pipe idle or not.  One warp,
// a dependent chain: each check's barrier depends on the previous result.
namespace {
constexpr int kRateBarChecks = 256;

__global__ void rate_bar_kernel(unsigned long long* cyc, int32_t* status) {
  __shared__ __align__(8) uint64_t bars[2];
  const uint32_t b0 = cpattn::smem_u32(&bars[0]);
  if (threadIdx.x == 0) {
    cpattn::mbar_init(b0, 1);
    cpattn::mbar_init(b0 + 8, 1);
    cpattn::fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {  // phase 0 of both completes
    cpattn::mbar_arrive(b0);
    cpattn::mbar_arrive(b0 + 8);
  }
  __syncwarp();
  uint32_t sel = 0;
  const unsigned long long t0 = clock64();
  for (int i = 0; i < kRateBarChecks; ++i) {
    const bool ok = __all_sync(0xffffffffu, cpattn::mbar_wait(b0 + 8u * sel, 0, nullptr, status));
    sel = ok ? (sel ^ 1u) : sel;
  }
  const unsigned long long t1 = clock64();
  if (threadIdx.x == 0) {
    cyc[0] = t1 - t0;
    cyc[1] = sel;
  }
}
}  // namespace

extern "C" int cp_measure_barrier_check(double* cycles, cudaStream_t stream) {
  if (!cycles) return CP_ERR_INVALID_ARG;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return CP_ERR_CUDA;
  if (major != 10 || minor != 3) return CP_ERR_ARCH;
  int32_t* st = status_ptr();
  if (!st) return CP_ERR_CUDA;
  unsigned long long* d_cyc = nullptr;
  if (cudaMalloc(&d_cyc, 2 * sizeof(unsigned long long)) != cudaSuccess) return CP_ERR_CUDA;
  int rc = CP_OK;
  // Twice; the second run is kept.
  for (int rep = 0; rc == CP_OK && rep < 2; ++rep) {
    rate_bar_kernel<<<1, 32, 0, stream>>>(d_cyc, st);
    if (cudaGetLastError() != cudaSuccess) rc = CP_ERR_CUDA;
  }
  unsigned long long cyc[2] = {0, 0};
  if (rc == CP_OK && (cudaMemcpyAsync(cyc, d_cyc, sizeof(cyc), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
                      cudaStreamSynchronize(stream) != cudaSuccess))
    rc = CP_ERR_CUDA;
  cudaFree(d_cyc);
  if (rc != CP_OK) return rc;
  *cycles = static_cast<double>(cyc[0]) / kRateBarChecks;
  return CP_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free emit-partials forward (cp_attn_fwd_noalloc).
//
// For callers that cannot allocate device memory (see the header): the
// per-ring-step partials live in this file-scope device array instead of a
// caller workspace.  Host code may not use the array's name as an address
// (in host code it is only a stand-in for the symbol), so its device address
// is resolved once per device with cudaGetSymbolAddress while that device is
// current, and that address is what the kernels receive.

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[CP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
// Per-device cache of the resolved address.  Atomic, so that host threads
// making their first call on one device at the same time are well defined:
// each resolves the same address and stores the same value.
std::atomic<void*> g_noalloc_addr[kMaxDevices];

// Device address of g_noalloc_scratch on the current device (set-up on the
// first call per device; nullptr if it could not be resolved).
void* noalloc_scratch_addr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* cached = g_noalloc_addr[dev].load(std::memory_order_acquire);
  if (!cached) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_noalloc_addr[dev].store(ptr, std::memory_order_release);
    cached = ptr;
  }
  return cached;
}

}  // namespace

extern "C" int cp_attn_fwd_noalloc(const cp_plan_t* p, const void* q, const void* k, const void* v, void* o,
                                   float* lse, cudaStream_t stream) {
  if (!p || !q || !k || !v || !o || !lse) return CP_ERR_INVALID_ARG;
  if (!p->desc.emit_partials || p->desc.ulysses_degree != 1) return CP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return CP_ERR_ALIGNMENT;
  int rc = check_device(p);
  if (rc != CP_OK) return rc;
  const cp_plan_desc_t& d = p->desc;
  const size_t R = d.ring_degree, L = d.L;
  const size_t o_bytes = align256(R * L * d.Hq * d.d * 4);
  const size_t lse_bytes = align256(R * L * d.Hq * 4);
  if (o_bytes + lse_bytes > CP_NOALLOC_SCRATCH_BYTES) return CP_ERR_WORKSPACE;
  char* scratch = static_cast<char*>(noalloc_scratch_addr());
  if (!scratch) return CP_ERR_CUDA;
  cpattn::FwdArgs a{};
  a.g = geom(p);
  a.d = d.d;
  a.o_fp32 = d.out_fp32;
  a.status = status_ptr();
  if (!a.status) return CP_ERR_CUDA;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.o_part = reinterpret_cast<float*>(scratch);
  a.lse_part = reinterpret_cast<float*>(scratch + o_bytes);
  a.items = p->d_items_steps;
  a.n_items = p->n_items_steps;
  rc = cpattn::launch_attn_fwd(a, stream);
  if (rc != CP_OK) return rc;
  return cpattn::launch_merge(d.ring_degree, d.ring_degree, p->T, d.Hq, d.d, a.o_part, a.lse_part, o, lse,
                              d.out_fp32, stream, a.status);
}
