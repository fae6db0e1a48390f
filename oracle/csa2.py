"""CPU oracle for CSA2 sparse decode attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
(``cpu_baseline`` and ``--impl reference``) may call it.  It shares no code,
constants or helpers with the CUDA library; its inputs come from the seeded
generator in ``sparse_attention_decode_index_gb300.workloads`` (which holds
no arithmetic of the method).

What it computes, in plain numpy, without blocking, fusion or reordering:

* indexer score of a compressed entry ``j`` for one query --
  ``s_j = sum_h w_h * ReLU(q_h . k_j)``.  The architecture page only says the
  indexer is "derived from section 4.2.1" of a report the pages do not
  include (k-a.in "DeepSeek V4.1 Flash", bullet "CSA2 reuse"); this weighted
  multi-head ReLU form is the plainest reading that gives the configured
  "8 heads x dim 64 with per-head weights" a meaning (without a per-head
  nonlinearity the heads would collapse into one).  Scores are computed in
  float64, which is exact for the integer-valued indexer data of the
  workloads (every partial sum is an integer far below 2**53).
* hierarchical indexer -- block summary keys (mean of a block's keys,
  optionally rounded half-to-even to integers), block scores with the same
  formula, a pool of the top ``min(P, NB)`` blocks, then token scores over
  the pooled blocks' entries (page 1 "DeepSeek V4.1 Flash made encoders
  cool": the hierarchical sparse indexer narrows candidates to blocks; page 3
  bullet "Hierarchical indexer": at most 16,384 candidates).
* exact Top-K -- a full sort under the total order (score descending, index
  ascending); the selected set is returned in ascending index order, padded
  with -1 (page 3 bullet "Sparse attention": Top-512).
* attention -- one softmax per query head over the selected main-KV rows
  plus the SWA rows, in float64 on the decoded inputs (page 3 bullet "Sparse
  attention": Top-512 main-KV entries plus a 128-token SWA window).
* cache maintenance -- appending compressed entries at ``n_valid`` with the
  summary keys of the touched blocks recomputed, and pushing a decoded token
  into a ring-shaped SWA window (page 3 bullets "Hierarchical indexer" and
  "Sparse attention"; the compression operator that makes the entries is
  not described by the pages, so entries are inputs).
* layer groups -- Full computes fresh indices, Reindex computes fresh
  indices with its own indexer query over the shared keys, Reuse takes the
  latest indices; every layer has its own query and SWA KV (page 3, "CSA2
  with cross-layer reuse", mode table and the sentence after it).  A pure
  sliding-window layer (page 3 figure caption: the first two encoder layers)
  attends its SWA rows only.

Parity pins: every function above is pinned by ``tests/test_oracle_pins.py``
(textbook dense attention, closed forms, brute-force selection, a
hand-worked golden case, hierarchical == flat when the pool covers every
block, Reuse == Full indices).  The toy workload's own values are parity
unpinned beyond its structural counts: the page says its scores are made-up
illustrations and prints none of them.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional

import numpy as np

FULL, REINDEX, REUSE, SWA = 0, 1, 2, 3


# ----------------------------------------------------------------------------
# decoding of the stored element types
# ----------------------------------------------------------------------------

def to_f64(x: np.ndarray) -> np.ndarray:
    """Decode stored values to float64: uint16 arrays hold bf16 bit patterns."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (8 significant bits, ties to even)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                      # x = m * 2**e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0), e - 8)


# ----------------------------------------------------------------------------
# indexer
# ----------------------------------------------------------------------------

def indexer_scores(q_idx: np.ndarray, w: np.ndarray, keys: np.ndarray, relu: bool = True) -> np.ndarray:
    """s_j = sum_h w_h * ReLU(q_h . k_j) for every row k_j of ``keys``.

    q_idx [HI, dI], w [HI], keys [n, dI] (float64) -> [n] float64.
    """
    dots = keys @ q_idx.T                   # [n, HI]
    if relu:
        dots = np.maximum(dots, 0.0)
    return dots @ w


def block_keys(keys: np.ndarray, n_valid: int, block: int, round_to_int: bool,
               store_bf16: bool = False) -> np.ndarray:
    """Block summary keys: the mean of each block's valid keys.

    Blocks are ``block`` consecutive entries; the last block may be partial
    and then averages only its valid entries.  With ``round_to_int`` the mean
    is rounded half-to-even to an integer (the 128K Reindex workload's
    "rounded to integers"); otherwise, when the keys are stored as bf16,
    the mean is rounded to bf16 for storage.
    """
    nb = -(-n_valid // block)
    out = np.zeros((nb, keys.shape[1]), dtype=np.float64)
    for j in range(nb):
        rows = keys[j * block: min((j + 1) * block, n_valid)]
        mean = rows.sum(axis=0) / rows.shape[0]
        if round_to_int:
            mean = np.rint(mean)
        elif store_bf16:
            mean = round_bf16(mean)
        out[j] = mean
    return out


def kv_append(k_main, v_main, k_idx, kb, n_valid, n_new, k_new, v_new, kidx_new, *, block: int,
              round_to_int: bool, store_bf16: bool = True):
    """Append ``n_new[b]`` compressed entries per query at position ``n_valid[b]``.

    The cache arrays are copied and returned (rows are moved as stored, so bf16
    bit patterns stay bit patterns).  Entries that would land past the cache's
    end are dropped.  When ``kb`` (float64 summary keys, [B, NB, dI]) is given,
    every block that a new position falls in gets its summary key recomputed
    from the updated indexer keys with ``block_keys``; other blocks keep their
    values.  Returns (k_main, v_main, k_idx, kb, n_valid, dropped) where
    dropped[b] counts the entries that did not fit.
    """
    k_main, v_main, k_idx = np.array(k_main), np.array(v_main), np.array(k_idx)
    kb = None if kb is None else np.array(kb, dtype=np.float64)
    n_valid = np.array(n_valid, dtype=np.int64)
    B, N = k_main.shape[0], k_main.shape[1]
    dropped = np.zeros(B, dtype=np.int64)
    for b in range(B):
        nv0 = int(n_valid[b])
        m = min(int(n_new[b]), N - nv0)
        dropped[b] = int(n_new[b]) - m
        k_main[b, nv0:nv0 + m] = k_new[b, :m]
        v_main[b, nv0:nv0 + m] = v_new[b, :m]
        k_idx[b, nv0:nv0 + m] = kidx_new[b, :m]
        nv1 = nv0 + m
        if kb is not None and m > 0:
            keys = block_keys(to_f64(k_idx[b]), nv1, block, round_to_int, store_bf16=store_bf16)
            for j in range(nv0 // block, (nv1 - 1) // block + 1):
                kb[b, j] = keys[j]
        n_valid[b] = nv1
    return k_main, v_main, k_idx, kb, n_valid, dropped


def swa_append(k_swa, v_swa, head, n_swa, k_tok, v_tok):
    """Push token b into query b's SWA ring: row ``head[b]`` takes it, ``head``
    advances modulo the window, ``n_swa`` grows up to the window.  Returns
    updated copies (k_swa, v_swa, head, n_swa)."""
    k_swa, v_swa = np.array(k_swa), np.array(v_swa)
    head, n_swa = np.array(head, dtype=np.int64), np.array(n_swa, dtype=np.int64)
    W = k_swa.shape[1]
    for b in range(k_swa.shape[0]):
        k_swa[b, head[b]] = k_tok[b]
        v_swa[b, head[b]] = v_tok[b]
        head[b] = (head[b] + 1) % W
        n_swa[b] = min(n_swa[b] + 1, W)
    return k_swa, v_swa, head, n_swa


# ----------------------------------------------------------------------------
# exact Top-K
# ----------------------------------------------------------------------------

def select_topk(scores: np.ndarray, ids: np.ndarray, k: int) -> np.ndarray:
    """Exact Top-k under (score descending, id ascending).

    Returns the selected ids in ascending order, padded with -1 to length k.
    NaN scores are treated as -inf.
    """
    scores = np.where(np.isnan(scores), -np.inf, scores)
    order = np.lexsort((ids, -scores))      # primary key: -score; secondary: id
    chosen = np.sort(ids[order[:min(k, len(ids))]])
    out = np.full(k, -1, dtype=np.int64)
    out[:len(chosen)] = chosen
    return out


def pool_blocks(q_idx, w, kb, n_blocks: int, pool: int, relu: bool = True) -> np.ndarray:
    """Hierarchical first stage: the top min(pool, n_blocks) blocks, ascending."""
    s = indexer_scores(q_idx, w, kb[:n_blocks], relu)
    sel = select_topk(s, np.arange(n_blocks), min(pool, n_blocks))
    return sel[sel >= 0]


def pooled_entries(pool: np.ndarray, n_valid: int, block: int) -> np.ndarray:
    """Entries of the pooled blocks that are valid, in ascending order."""
    ent = (pool[:, None] * block + np.arange(block)[None, :]).reshape(-1)
    return ent[ent < n_valid]


def layer_indices(q_idx, w, keys, kb, n_valid: int, *, topk: int, block: int, pool: int,
                  hier: bool, relu: bool = True) -> Dict[str, np.ndarray]:
    """Fresh Top-K indices of one indexing layer (Full or Reindex) for one query.

    Flat: score entries 0..n_valid-1.  Hierarchical: score all blocks, keep the
    pool, score the pooled blocks' entries.  Then exact Top-K.
    """
    res = {}
    if hier:
        nb = -(-n_valid // block)
        pl = pool_blocks(q_idx, w, kb, nb, pool, relu)
        cand = pooled_entries(pl, n_valid, block)
        res["pool"] = pl
    else:
        cand = np.arange(n_valid)
    s = indexer_scores(q_idx, w, keys[cand], relu)
    res["cand"] = cand
    res["scores"] = s
    res["idx"] = select_topk(s, cand, topk)
    return res


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------

def attend(q: np.ndarray, k_rows: np.ndarray, v_rows: np.ndarray, scale: float):
    """Softmax attention of every query head over the given rows.

    q [H, dk], k_rows [n, dk], v_rows [n, dv] -> out [H, dv], lse [H]
    (lse = log sum_j exp(scale * q . k_j), natural log).  With no rows at all
    the output is zero and lse is -inf.
    """
    H = q.shape[0]
    if k_rows.shape[0] == 0:
        return np.zeros((H, v_rows.shape[1])), np.full(H, -np.inf)
    logits = scale * (q @ k_rows.T)          # [H, n]
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    l = e.sum(axis=1, keepdims=True)
    out = (e @ v_rows) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse


def sparse_attention(q, k_main, v_main, idx, k_swa, v_swa, n_swa: int, scale: float):
    """One query: attention over main rows ``idx`` (entries < 0 skipped) plus SWA rows 0..n_swa-1."""
    sel = idx[idx >= 0]
    k_rows = np.concatenate([k_main[sel], k_swa[:n_swa]], axis=0)
    v_rows = np.concatenate([v_main[sel], v_swa[:n_swa]], axis=0)
    return attend(q, k_rows, v_rows, scale)


# ----------------------------------------------------------------------------
# layer groups
# ----------------------------------------------------------------------------

def run_group(wl, *, queries: Optional[List[int]] = None, want_attention: bool = True,
              relu: Optional[bool] = None) -> List[Dict[str, object]]:
    """Run a whole layer group on the CPU.

    ``wl`` is a ``workloads.Workload``.  Returns, per layer, a dict with
    ``idx`` [B', K] (the index set the layer attended with), ``out``
    [B', H, dv] and ``lse`` [B', H] (if ``want_attention``), and for indexing
    layers the per-query intermediates (``pool``, ``cand``, ``scores``).
    ``queries`` restricts the run to a subset of the batch (sampled parity).
    With ``shape.tokens`` = T > 1 the caches hold one sequence per T queries
    and query b reads sequence b // T; every other array is per query.
    """
    sh = wl.shape
    tokens = max(1, int(getattr(sh, "tokens", 1)))
    relu = bool(sh.relu) if relu is None else relu
    scale = sh.scale if sh.scale > 0 else 1.0 / math.sqrt(sh.k_dim)
    qs = list(range(sh.batch)) if queries is None else list(queries)
    bf16 = sh.dtype == "bf16"
    results: List[Dict[str, object]] = [dict() for _ in wl.layers]
    for bi, b in enumerate(qs):
        n_valid = int(wl.n_valid[b])
        n_swa = int(wl.n_swa[b])
        seq = b // tokens
        keys = to_f64(wl.k_idx[seq])
        kb = None
        if any(L.hier for L in wl.layers):
            kb = block_keys(keys, n_valid, sh.block, bool(wl.round_block_keys), store_bf16=bf16)
        k_main = to_f64(wl.k_main[seq]) if want_attention else None
        v_main = to_f64(wl.v_main[seq]) if want_attention else None
        cur = None
        for li, L in enumerate(wl.layers):
            r = results[li]
            if L.mode == SWA:
                if want_attention:
                    out, lse = attend(to_f64(L.q[b]), to_f64(L.k_swa[b])[:n_swa], to_f64(L.v_swa[b])[:n_swa],
                                      scale)
                    r.setdefault("out", np.zeros((len(qs), sh.q_heads, sh.v_dim)))[bi] = out
                    r.setdefault("lse", np.zeros((len(qs), sh.q_heads)))[bi] = lse
                continue
            if L.mode == REUSE:
                if cur is None:
                    raise ValueError("a Reuse layer needs an earlier indexing layer in the group")
                idx = cur
            else:
                lr = layer_indices(to_f64(L.q_idx[b]), to_f64(L.w_idx[b]), keys, kb, n_valid,
                                   topk=sh.topk, block=sh.block, pool=sh.pool_blocks,
                                   hier=bool(L.hier), relu=relu)
                idx = lr["idx"]
                for key in ("pool", "cand", "scores"):
                    if key in lr:
                        r.setdefault(key, [None] * len(qs))[bi] = lr[key]
                cur = idx
            r.setdefault("idx", np.zeros((len(qs), sh.topk), dtype=np.int64))[bi] = idx
            if want_attention:
                out, lse = sparse_attention(to_f64(L.q[b]), k_main, v_main, idx,
                                            to_f64(L.k_swa[b]), to_f64(L.v_swa[b]), n_swa, scale)
                r.setdefault("out", np.zeros((len(qs), sh.q_heads, sh.v_dim)))[bi] = out
                r.setdefault("lse", np.zeros((len(qs), sh.q_heads)))[bi] = lse
    return results


def group_counts(modes: List[object]) -> Dict[str, int]:
    """Counts over a layer pattern: CSA2 layers, layers storing global KV, indexer layers.

    ``modes`` holds FULL/REINDEX/REUSE, and SWA (or the string "swa") for a
    pure sliding-window layer.  Only Full layers compute (store) their own main KV;
    Full and Reindex layers run an indexer (page 3, mode table).
    """
    csa2 = [m for m in modes if m not in ("swa", SWA)]
    return {
        "layers": len(modes),
        "csa2": len(csa2),
        "kv_storing": sum(1 for m in csa2 if m == FULL),
        "indexers": sum(1 for m in csa2 if m in (FULL, REINDEX)),
    }
