"""CPU oracle for context-parallel causal attention (fp64, numpy).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module.  The CUDA path never
calls it and shares no code with it.

Sources (web pages; the citation names the page and its section):

* [MTX] nougat.kr, "MaxText long-context training and KV parallelism":
  section "Why KV comes back together even after splitting the input"
  (causal dependency: a query needs the K/V of every earlier token);
  section "Split heads or rotate KV" (A2A/Ulysses: attention is independent
  per head, tokens->heads before attention and back after; P2P/ring: each
  chip keeps its queries, visits one KV chunk at a time and merges partial
  results; GQA: the KV-head count caps the A2A degree; USP = A2A groups x
  ring; causal load balancing).
* [ULY] aionda.blog, "Ulysses sequence parallelism for long-context
  training": section "Current state" (all-to-all along the sequence axis,
  each GPU computes a subset of heads).
* [L3P] siliconandsystems.com, "Llama 3 parallelism": section "Four
  parallelisms secure different resources" (CP must keep the mask that
  separates packed documents) and "Long context changes more than attention
  cost" (balance by actual attention work; activation recompute).

The pages never write the attention formula out.  This module takes the
textbook definition of scaled dot-product softmax attention:

    s_ik  = scale * <q_i, k_k>                 scale = 1/sqrt(d) by default
    M(i,k) = [pos_k <= pos_i] and [doc(pos_k) == doc(pos_i)]
    LSE_i = log sum_{k in M(i,.)} exp(s_ik)    (natural log)
    O_i   = sum_{k in M(i,.)} exp(s_ik - LSE_i) v_k

with an empty visible set giving the partial (O=0, LSE=-inf).  Query head h
reads KV head floor(h / G), G = Hq/Hkv.  Rows are independent under this
definition, so computing a subset of rows (sampled rows, or rows a few
hundred at a time to bound memory) is the definition itself, not a
re-ordering of it.

Parity status: every function here is pinned by the not-gpu tests (closed
forms, a library attention routine, brute force, finite differences and the
invariants the pages imply); none is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf

# --------------------------------------------------------------------------
# Masks
# --------------------------------------------------------------------------


def doc_start_of(pos: np.ndarray, offsets) -> np.ndarray:
    """Start position of the packed document holding each position.

    ``offsets`` = [0, end_0, end_1, ..., L]; None means one document.
    [L3P] "Four parallelisms secure different resources": the document mask
    must survive context parallelism.
    """
    pos = np.asarray(pos, dtype=np.int64)
    if offsets is None:
        return np.zeros_like(pos)
    offsets = np.asarray(offsets, dtype=np.int64)
    idx = np.searchsorted(offsets, pos, side="right") - 1
    return offsets[idx]


def visible(q_pos, k_pos, offsets=None, causal=True) -> np.ndarray:
    """Boolean [nq, nk]: M(i,k) = [pos_k <= pos_i] and same document.

    [MTX] "Why KV comes back together": under causal attention each query
    needs the K/V of all earlier tokens.
    """
    q_pos = np.asarray(q_pos, dtype=np.int64)[:, None]
    k_pos = np.asarray(k_pos, dtype=np.int64)[None, :]
    m = np.ones((q_pos.shape[0], k_pos.shape[1]), dtype=bool)
    if causal:
        m &= k_pos <= q_pos
    if offsets is not None:
        m &= doc_start_of(k_pos, offsets) == doc_start_of(q_pos, offsets)
    return m


# --------------------------------------------------------------------------
# Attention (the plain definition)
# --------------------------------------------------------------------------


def _scale_of(d, scale):
    return 1.0 / math.sqrt(d) if scale is None else float(scale)


def _f64(x):
    """fp64 numpy copy of an array or a (CPU) torch tensor (exact for bf16/fp32)."""
    if hasattr(x, "detach"):
        import torch
        return x.detach().to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def attention_rows(q, k, v, rows=None, q_pos=None, k_pos=None, offsets=None,
                   causal=True, scale=None, heads=None):
    """O and LSE of the query rows ``rows`` (default: all) for ``heads``
    (default: all query heads).

    q [nq, Hq, d], k, v [nk, Hkv, d] (numpy arrays or CPU torch tensors of
    any float type, evaluated in fp64); q_pos / k_pos give each row's global
    position (default 0..n-1).  Returns O [len(rows), len(heads), d] float64
    and LSE [len(heads), len(rows)] float64.  A row with no visible key
    yields O = 0, LSE = -inf.
    """
    nq, Hq, d = q.shape
    nk, Hkv, _ = k.shape
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    sc = _scale_of(d, scale)
    rows = np.arange(nq) if rows is None else np.asarray(rows, dtype=np.int64)
    heads = list(range(Hq)) if heads is None else [int(h) for h in heads]
    q_pos = np.arange(nq) if q_pos is None else np.asarray(q_pos, dtype=np.int64)
    k_pos = np.arange(nk) if k_pos is None else np.asarray(k_pos, dtype=np.int64)
    # Memory bound: a block of rows times all keys stays near 2^24 scores.
    row_block = max(1, min(256, (1 << 24) // max(nk, 1)))
    O = np.zeros((len(rows), len(heads), d))
    LSE = np.full((len(heads), len(rows)), NEG_INF)
    kv_cache = {}
    for hi, h in enumerate(heads):
        j = h // G                                              # GQA: KV head of query head h
        if j not in kv_cache:
            kv_cache.clear()
            kv_cache[j] = (_f64(k[:, j, :]), _f64(v[:, j, :]))
        Kj, Vj = kv_cache[j]
        for b0 in range(0, len(rows), row_block):
            rb = rows[b0:b0 + row_block]
            M = visible(q_pos[rb], k_pos, offsets, causal)      # [nb, nk]
            any_vis = M.any(axis=1)
            S = sc * (_f64(q[rb, h, :]) @ Kj.T)                 # [nb, nk]
            S = np.where(M, S, NEG_INF)
            m = np.where(any_vis, S.max(axis=1), 0.0)
            with np.errstate(divide="ignore"):
                lse = m + np.log(np.exp(S - m[:, None]).sum(axis=1))
            P = np.exp(S - np.where(any_vis, lse, 0.0)[:, None])
            P[~any_vis] = 0.0
            O[b0:b0 + len(rb), hi, :] = P @ Vj
            LSE[hi, b0:b0 + len(rb)] = np.where(any_vis, lse, NEG_INF)
    return O, LSE


def attention(q, k, v, offsets=None, causal=True, scale=None):
    """Full attention of a global sequence: all rows, positions 0..L-1."""
    return attention_rows(q, k, v, offsets=offsets, causal=causal, scale=scale)


def attention_bwd(q, k, v, do, offsets=None, causal=True, scale=None):
    """Gradients of the attention above, fp64 (plain definition).

    With P = exp(S - LSE) (the forward's probabilities, recomputed from the
    saved LSE as activation recompute does, [L3P] "Long context changes more
    than attention cost"):
        dV_j = sum_{h in group j} P_h^T dO_h
        dP_h = dO_h V_j^T
        D_i  = sum_c dO_ic O_ic
        dS_h = P_h * (dP_h - D)
        dQ_h = scale dS_h K_j
        dK_j = sum_{h in group j} scale dS_h^T Q_h
    Returns (O, LSE, dQ, dK, dV), all float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    L, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    sc = _scale_of(d, scale)
    O, LSE = attention(q, k, v, offsets=offsets, causal=causal, scale=scale)
    M = visible(np.arange(L), np.arange(L), offsets, causal)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(Hq):
        j = h // G
        S = np.where(M, sc * (q[:, h, :] @ k[:, j, :].T), NEG_INF)
        P = np.exp(S - LSE[h][:, None])
        P[~M] = 0.0
        dv[:, j, :] += P.T @ do[:, h, :]
        dP = do[:, h, :] @ v[:, j, :].T
        D = (do[:, h, :] * O[:, h, :]).sum(axis=1)
        dS = P * (dP - D[:, None])
        dq[:, h, :] = sc * (dS @ k[:, j, :])
        dk[:, j, :] += sc * (dS.T @ q[:, h, :])
    return O, LSE, dq, dk, dv


def attention_bwd_rows(q, k, v, do, q_rows=(), key_rows=(), offsets=None, causal=True, scale=None,
                       q_heads=None, kv_heads=None, row_block=None):
    """Selected gradient rows, fp64, from the same definition as
    attention_bwd: dQ at query rows ``q_rows`` for ``q_heads`` and dK, dV at
    key rows ``key_rows`` for ``kv_heads`` (global order, positions 0..L-1).

    Each needed query row's O and LSE come from attention_rows; then, per
    query head h and KV head j = floor(h/G), with P = exp(S - LSE) over the
    visible pairs, dP = dO V^T, D = rowsum(dO * O), dS = P (dP - D):
    dQ_i = scale sum_k dS_ik K_k,  dV_k = sum_h sum_i P_ik dO_i,
    dK_k = scale sum_h sum_i dS_ik Q_i.  A dQ row needs P and dS against
    every key; a dK/dV row needs them only in its own column, for every
    query that sees the key (all later positions of its document), so P and
    dS are formed only for those columns.  Query rows are taken
    ``row_block`` at a time (default: about 2^24 scores per block) to bound
    memory; rows are independent, so this is the definition itself.
    Returns (dq [nq, len(q_heads), d], dk, dv [nk, len(kv_heads), d]).
    """
    L, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    sc = _scale_of(d, scale)
    q_rows = np.asarray(q_rows, dtype=np.int64)
    key_rows = np.asarray(key_rows, dtype=np.int64)
    q_heads = list(range(Hq)) if q_heads is None else [int(h) for h in q_heads]
    kv_heads = list(range(Hkv)) if kv_heads is None else [int(j) for j in kv_heads]
    dq = np.zeros((len(q_rows), len(q_heads), d))
    dk = np.zeros((len(key_rows), len(kv_heads), d))
    dv = np.zeros((len(key_rows), len(kv_heads), d))
    all_pos = np.arange(L)
    blk = row_block or max(1, min(1024, (1 << 24) // max(L, 1)))

    def row_terms(rows, h, cols):
        """P, dS of query rows `rows` of head h against the keys `cols`."""
        j = h // G
        O, LSE = attention_rows(q, k, v, rows=rows, offsets=offsets, causal=causal, scale=scale, heads=[h])
        Kc, Vc = _f64(k[cols, j, :]), _f64(v[cols, j, :])
        Qr, dOr = _f64(q[rows, h, :]), _f64(do[rows, h, :])
        M = visible(rows, cols, offsets, causal)
        S = sc * (Qr @ Kc.T)
        P = np.where(M, np.exp(S - LSE[0][:, None]), 0.0)
        dP = dOr @ Vc.T
        D = (dOr * O[:, 0, :]).sum(axis=1)
        dS = P * (dP - D[:, None])
        return P, dS, Qr, dOr, Kc

    if len(q_rows):
        for hi, h in enumerate(q_heads):
            for b0 in range(0, len(q_rows), blk):
                rb = q_rows[b0:b0 + blk]
                _, dS, _, _, Kc = row_terms(rb, h, all_pos)
                dq[b0:b0 + len(rb), hi, :] = sc * (dS @ Kc)
    if len(key_rows):
        vis = visible(all_pos, key_rows, offsets, causal)          # [L, nk]: query sees key
        need = np.nonzero(vis.any(axis=1))[0]
        for ji, j in enumerate(kv_heads):
            for h in range(j * G, (j + 1) * G):
                for b0 in range(0, len(need), blk):
                    P, dS, Qr, dOr, _ = row_terms(need[b0:b0 + blk], h, key_rows)
                    dv[:, ji, :] += P.T @ dOr
                    dk[:, ji, :] += sc * (dS.T @ Qr)
    return dq, dk, dv


# --------------------------------------------------------------------------
# Context-parallel restatement: index maps, merge, reshard, ring, USP
# --------------------------------------------------------------------------

LAYOUT_CONTIGUOUS = 0
LAYOUT_ZIGZAG = 1
LAYOUT_BALANCED = 2


def chunk_work(L: int, n_chunks: int, offsets=None) -> np.ndarray:
    """Attention work of each of n_chunks equal position chunks: the number
    of visible (query, key) pairs whose query lies in the chunk.  A query at
    position i sees i - doc_start(i) + 1 keys (causal, same document)."""
    c = L // n_chunks
    pos = np.arange(L, dtype=np.int64)
    per_query = pos - doc_start_of(pos, offsets) + 1
    return per_query.reshape(n_chunks, c).sum(axis=1)


def balanced_chunks(L: int, R: int, chunks_per_rank: int, offsets=None):
    """Chunk lists of the work-balanced layout ([L3P] "Long context changes
    more than attention cost": split by actual attention work, not by
    position; [MTX] "Split heads or rotate KV": causal load balancing).

    Reading: the sequence is cut into C = m*R equal chunks (m =
    chunks_per_rank).  Taking the chunks from most to least work (equal work:
    lower chunk index first), each goes to the rank with the least work so
    far among the ranks that still hold fewer than m chunks (equal work:
    lower rank first).  Each rank keeps its chunks in position order.
    Returns a list of R lists of chunk indices.
    """
    m = chunks_per_rank
    C = m * R
    if m < 1 or L % C:
        raise ValueError("chunks_per_rank * R must divide L")
    work = chunk_work(L, C, offsets)
    order = sorted(range(C), key=lambda j: (-int(work[j]), j))
    load = [0] * R
    held = [[] for _ in range(R)]
    for j in order:
        best = None
        for r in range(R):
            if len(held[r]) < m and (best is None or load[r] < load[best]):
                best = r
        held[best].append(j)
        load[best] += int(work[j])
    return [sorted(h) for h in held]


def ring_positions(L: int, R: int, layout: int, offsets=None, chunks_per_rank: int = 4) -> np.ndarray:
    """Global position of every slot, rank-major: out[r*(L/R) + t].

    Contiguous: rank r holds positions [r*L/R, (r+1)*L/R).
    Zigzag (the reading of [MTX] "Split heads or rotate KV" / [L3P] "Long
    context": balance by actual attention work): the sequence is cut into 2R
    chunks of c = L/(2R); rank r holds chunk r followed by chunk 2R-1-r.
    Balanced: the chunks of ``balanced_chunks`` (which reads the document
    offsets), concatenated in each rank's order.
    """
    if layout == LAYOUT_BALANCED:
        lists = balanced_chunks(L, R, chunks_per_rank, offsets)
        c = L // (chunks_per_rank * R)
        return np.concatenate([np.arange(j * c, (j + 1) * c, dtype=np.int64)
                               for chunks in lists for j in chunks])
    if layout == LAYOUT_CONTIGUOUS:
        if L % R:
            raise ValueError("R must divide L")
        return np.arange(L, dtype=np.int64)
    if L % (2 * R):
        raise ValueError("2R must divide L for zigzag")
    c = L // (2 * R)
    out = np.empty(L, dtype=np.int64)
    for r in range(R):
        base = r * 2 * c
        out[base:base + c] = r * c + np.arange(c)
        out[base + c:base + 2 * c] = (2 * R - 1 - r) * c + np.arange(c)
    return out


def shard(x_global: np.ndarray, positions: np.ndarray) -> np.ndarray:
    """Rank-major sharded copy: slot t of the result holds position positions[t]."""
    return x_global[positions]


def unshard(x_slots: np.ndarray, positions: np.ndarray) -> np.ndarray:
    out = np.empty_like(x_slots)
    out[positions] = x_slots
    return out


def merge_pair(o_a, lse_a, o_b, lse_b):
    """Merge two normalised partials over disjoint key sets.

    [MTX] "Split heads or rotate KV": ring attention computes a partial with
    each visiting KV chunk and merges the results.  Reading: with
    l = log(e^la + e^lb) the exact merge is O = e^(la-l) O_a + e^(lb-l) O_b;
    (0, -inf) is the empty partial and the identity.
    o_*: [n, H, d], lse_*: [H, n].
    """
    o_a = np.asarray(o_a, dtype=np.float64)
    o_b = np.asarray(o_b, dtype=np.float64)
    lse_a = np.asarray(lse_a, dtype=np.float64)
    lse_b = np.asarray(lse_b, dtype=np.float64)
    m = np.maximum(lse_a, lse_b)
    empty = np.isneginf(m)
    ms = np.where(empty, 0.0, m)
    wa = np.exp(lse_a - ms)
    wb = np.exp(lse_b - ms)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, NEG_INF, ms + np.log(wa + wb))
    ls = np.where(empty, 0.0, lse)
    ca = np.where(empty, 0.0, np.exp(lse_a - ls))               # [H, n]
    cb = np.where(empty, 0.0, np.exp(lse_b - ls))
    o = ca.T[:, :, None] * o_a + cb.T[:, :, None] * o_b
    return o, lse


def merge(parts):
    """Merge a list of (O, LSE) partials in list order (ring order)."""
    o, lse = parts[0]
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    for o_b, lse_b in parts[1:]:
        o, lse = merge_pair(o, lse, o_b, lse_b)
    return o, lse


def ulysses_seq_to_head(x: np.ndarray, U: int) -> np.ndarray:
    """All-to-all #1 of one Ulysses group: [U][n][H][d] -> [U][U*n][H/U][d].

    Y_u[s*n + t, h'] = X_s[t, u*H/U + h']  ([MTX] "Split heads or rotate KV":
    before attention each chip swaps its token shard of all heads for the
    full group sequence of a subset of heads; [ULY] "Current state").
    """
    U_, n, H = x.shape[:3]
    assert U_ == U and H % U == 0
    Hl = H // U
    y = np.empty((U, U * n, Hl) + x.shape[3:], dtype=x.dtype)
    for u in range(U):
        for s in range(U):
            y[u, s * n:(s + 1) * n] = x[s, :, u * Hl:(u + 1) * Hl]
    return y


def ulysses_head_to_seq(y: np.ndarray, U: int) -> np.ndarray:
    """All-to-all #2, the inverse: [U][U*n][H/U][d] -> [U][n][H][d]."""
    U_, Un, Hl = y.shape[:3]
    assert U_ == U and Un % U == 0
    n = Un // U
    x = np.empty((U, n, Hl * U) + y.shape[3:], dtype=y.dtype)
    for u in range(U):
        for s in range(U):
            x[s, :, u * Hl:(u + 1) * Hl] = y[u, s * n:(s + 1) * n]
    return x


def ulysses_lse_head_to_seq(lse: np.ndarray, U: int) -> np.ndarray:
    """Inverse reshard of LSE: [U][H/U][U*n] -> [U][H][n]."""
    U_, Hl, Un = lse.shape
    n = Un // U
    out = np.empty((U, Hl * U, n), dtype=lse.dtype)
    for u in range(U):
        for s in range(U):
            out[s, u * Hl:(u + 1) * Hl, :] = lse[u, :, s * n:(s + 1) * n]
    return out


def ring_partials(q_r, k_ranks, v_ranks, q_pos, k_pos_ranks, r, offsets=None,
                  causal=True, scale=None, rows=None):
    """Partials of ring rank r, one per ring step s (source (r - s) mod R).

    [MTX] "Split heads or rotate KV": P2P keeps token sharding; each chip
    computes part of attention with the KV chunk it holds now and passes the
    chunk on.  Reading: the chunk received at step s comes from rank (r - s)
    mod R.  Each partial is normalised; an empty one is (0, -inf).
    """
    R = len(k_ranks)
    parts = []
    for s in range(R):
        src = (r - s) % R
        parts.append(attention_rows(q_r, k_ranks[src], v_ranks[src], rows=rows,
                                    q_pos=q_pos, k_pos=k_pos_ranks[src],
                                    offsets=offsets, causal=causal, scale=scale))
    return parts


def ring_forward(q, k, v, R, layout=LAYOUT_CONTIGUOUS, offsets=None, causal=True,
                 scale=None, return_partials=False, chunks_per_rank=4):
    """Ring (P2P) CP forward over R ranks on global-order inputs.

    Returns per-rank O [R][n][Hq][d] and LSE [R][Hq][n] in slot order (and the
    per-step partials if asked).
    """
    L = q.shape[0]
    n = L // R
    pos = ring_positions(L, R, layout, offsets, chunks_per_rank)
    qs, ks, vs = shard(q, pos), shard(k, pos), shard(v, pos)
    k_ranks = [ks[r * n:(r + 1) * n] for r in range(R)]
    v_ranks = [vs[r * n:(r + 1) * n] for r in range(R)]
    kpos = [pos[r * n:(r + 1) * n] for r in range(R)]
    O, LSE, allparts = [], [], []
    for r in range(R):
        parts = ring_partials(qs[r * n:(r + 1) * n], k_ranks, v_ranks, kpos[r], kpos, r,
                              offsets=offsets, causal=causal, scale=scale)
        o, lse = merge(parts)
        O.append(o)
        LSE.append(lse)
        allparts.append(parts)
    if return_partials:
        return np.stack(O), np.stack(LSE), allparts
    return np.stack(O), np.stack(LSE)


def attention_bwd_partial(q, do, o, lse, k, v, q_pos, k_pos, offsets=None, causal=True, scale=None):
    """Contribution of one visiting key block to the gradients, fp64: the
    a7 formulas of attention_bwd restricted to the pairs (i, k) with query i
    in this block (positions q_pos) and key k in the visiting block
    (positions k_pos), using the full forward's O and LSE of the queries
    (P = exp(S - LSE) with the saved LSE, D = rowsum(dO * O)).  This is the
    backward of one ring step ([MTX] "Split heads or rotate KV": partial
    results per visiting chunk; the chunk's dK, dV travel with it).
    q, do, o [nq, Hq, d]; lse [Hq, nq]; k, v [nk, Hkv, d].
    Returns (dq [nq, Hq, d], dk, dv [nk, Hkv, d]) to be summed over steps."""
    q, do, o = (np.asarray(x, dtype=np.float64) for x in (_f64(q), _f64(do), _f64(o)))
    k, v = np.asarray(_f64(k), dtype=np.float64), np.asarray(_f64(v), dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    nq, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    sc = _scale_of(d, scale)
    M = visible(np.asarray(q_pos), np.asarray(k_pos), offsets, causal)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(Hq):
        j = h // G
        qh, doh, kj, vj = q[:, h, :], do[:, h, :], k[:, j, :], v[:, j, :]
        with np.errstate(invalid="ignore"):
            P = np.where(M, np.exp(sc * (qh @ kj.T) - lse[h][:, None]), 0.0)
        dv[:, j, :] += P.T @ doh
        dP = doh @ vj.T
        D = (doh * o[:, h, :]).sum(axis=1)
        dS = P * (dP - D[:, None])
        dq[:, h, :] = sc * (dS @ kj)
        dk[:, j, :] += sc * (dS.T @ qh)
    return dq, dk, dv


def allgather_forward(q, k, v, R, layout=LAYOUT_CONTIGUOUS, offsets=None, causal=True,
                      scale=None, chunks_per_rank=4):
    """All-gather CP forward ([MTX] "Why KV comes back together": every chip
    gathers the K/V of all chips and computes attention for the tokens it
    holds; [L3P] "Four parallelisms secure different resources": the packed
    documents' mask is kept).  The gathered K/V is the global sequence, so
    rank r attends with its own query rows over every key position.
    Returns per-rank O [R][n][Hq][d] and LSE [R][Hq][n] in slot order.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)     # exact for bf16 / fp32 inputs
    L = q.shape[0]
    n = L // R
    pos = ring_positions(L, R, layout, offsets, chunks_per_rank)
    k_all = unshard(shard(k, pos), pos)      # all-gather: the shards put back in position order
    v_all = unshard(shard(v, pos), pos)
    key_pos = np.arange(L, dtype=np.int64)
    O, LSE = [], []
    for r in range(R):
        rows = pos[r * n:(r + 1) * n]
        o, lse = attention_rows(q, k_all, v_all, rows=rows, k_pos=key_pos,
                                offsets=offsets, causal=causal, scale=scale)
        O.append(o)
        LSE.append(lse)
    return np.stack(O), np.stack(LSE)


def usp_forward(q, k, v, U, R, layout=LAYOUT_CONTIGUOUS, offsets=None, causal=True,
                scale=None, chunks_per_rank=4):
    """USP = Ulysses groups x ring ([MTX] "Split heads or rotate KV").

    Rank g = r*U + u (Ulysses innermost).  Member u of ring rank r holds the
    ring-local slots [u*n, (u+1)*n), n = L/(R*U), of ring rank r's shard.
    Steps: reshard seq->head inside each Ulysses group, ring attention over r
    for each head group u, reshard O and LSE head->seq.
    Returns O [P][n][Hq][d] and LSE [P][Hq][n], rank-major.
    """
    L, Hq, d = q.shape
    Hkv = k.shape[1]
    if Hkv % U:
        raise ValueError("Ulysses degree must divide the KV-head count")
    T = L // R                      # ring shard length
    n = T // U                      # per-rank tokens
    pos = ring_positions(L, R, layout, offsets, chunks_per_rank)
    qs, ks, vs = shard(q, pos), shard(k, pos), shard(v, pos)

    def group(x, r):                # [U][n][H][d] of ring rank r
        return x[r * T:(r + 1) * T].reshape((U, n) + x.shape[1:])

    qh = [ulysses_seq_to_head(group(qs, r), U) for r in range(R)]   # [U][T][Hq/U][d]
    kh = [ulysses_seq_to_head(group(ks, r), U) for r in range(R)]
    vh = [ulysses_seq_to_head(group(vs, r), U) for r in range(R)]
    kpos = [pos[r * T:(r + 1) * T] for r in range(R)]
    O = np.empty((R * U, n, Hq, d))
    LSE = np.empty((R * U, Hq, n))
    for r in range(R):
        o_u, l_u = [], []
        for u in range(U):
            parts = ring_partials(qh[r][u], [kh[s][u] for s in range(R)],
                                  [vh[s][u] for s in range(R)], kpos[r], kpos, r,
                                  offsets=offsets, causal=causal, scale=scale)
            o, lse = merge(parts)
            o_u.append(o)
            l_u.append(lse)
        O[r * U:(r + 1) * U] = ulysses_head_to_seq(np.stack(o_u), U)
        LSE[r * U:(r + 1) * U] = ulysses_lse_head_to_seq(np.stack(l_u), U)
    return O, LSE


def visible_pairs(L: int, offsets=None, causal=True) -> int:
    """Number of visible (query, key) pairs: the useful-work count."""
    if offsets is None:
        return L * (L + 1) // 2 if causal else L * L
    lens = np.diff(np.asarray(offsets, dtype=np.int64))
    return int((lens * (lens + 1) // 2).sum()) if causal else int((lens * lens).sum())


def rank_visible_pairs(L, R, layout, offsets=None, chunks_per_rank=4):
    """Visible pairs whose query sits on each ring rank (the rank's work)."""
    pos = ring_positions(L, R, layout, offsets, chunks_per_rank)
    n = L // R
    ds = doc_start_of(np.arange(L), offsets)
    out = []
    for r in range(R):
        p = pos[r * n:(r + 1) * n]
        out.append(int((p - ds[p] + 1).sum()))
    return out
