"""Pins for the CPU oracle: checks against things the pages and mathematics fix.

None of these compares the oracle with itself.  Each check would fail on a
plausible slip in the oracle (dropped ReLU or weight, wrong tie-break
direction, transposed operand, missing SWA rows, wrong softmax scale, wrong
rounding mode, pool not sorted, Reuse recomputing its indices).
"""
import heapq
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import FULL, REINDEX, REUSE
from sparse_attention_decode_index_gb300 import workloads as W


GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- hand-worked toy

def test_golden_toy16_hand():
    g = _load("toy16_hand.json")
    keys = np.array(g["keys"], dtype=np.float64)[:, None]
    q = np.ones((1, 1))
    w = np.ones(1)
    n_valid, blk, pool, k = g["n_valid"], g["block"], g["pool"], g["topk"]

    kb_unr = oracle.block_keys(keys, n_valid, blk, round_to_int=False)
    kb_r = oracle.block_keys(keys, n_valid, blk, round_to_int=True)
    assert kb_unr[:, 0].tolist() == g["block_means"]
    assert kb_r[:, 0].tolist() == g["block_keys_rounded"]
    assert oracle.indexer_scores(q, w, kb_r).tolist() == g["block_scores_rounded"]

    nb = len(g["block_means"])
    assert oracle.pool_blocks(q, w, kb_r, nb, pool).tolist() == g["pool_rounded"]
    assert oracle.pool_blocks(q, w, kb_unr, nb, pool).tolist() == g["pool_unrounded"]

    r = oracle.layer_indices(q, w, keys, kb_r, n_valid, topk=k, block=blk, pool=pool, hier=True)
    assert r["cand"].tolist() == g["candidates_rounded"]
    assert r["scores"].tolist() == g["candidate_scores_rounded"]
    assert r["idx"].tolist() == g["top3_hier_rounded"]
    r = oracle.layer_indices(q, w, keys, kb_unr, n_valid, topk=k, block=blk, pool=pool, hier=True)
    assert r["idx"].tolist() == g["top3_hier_unrounded"]
    r = oracle.layer_indices(q, w, keys, None, n_valid, topk=k, block=blk, pool=pool, hier=False)
    assert r["idx"].tolist() == g["top3_flat"]

    # attention reads the 3 selected entries plus the 4 window tokens
    n_keys = int((r["idx"] >= 0).sum()) + g["swa"]
    assert n_keys == g["attended_keys"]


def test_toy16_structure():
    """Counts fixed by the page's toy: 12 candidates -> 6 blocks -> pool 4 -> 8 -> Top-3, 7 keys."""
    for seed in range(5):
        wl = W.toy16(seed)
        res = oracle.run_group(wl)
        r = res[0]
        assert int(wl.n_valid[0]) == 12 and int(wl.n_swa[0]) == 4
        assert len(r["pool"][0]) == 4
        assert len(r["cand"][0]) == 8
        idx = r["idx"][0]
        assert (idx >= 0).sum() == 3 and np.all(idx[idx >= 0] < 12)
        assert np.all(np.diff(idx) > 0)
        assert set(idx.tolist()) <= set(r["cand"][0].tolist())
        assert r["out"].shape == (1, 4, 16)


# ---------------------------------------------------------------- indexer

def test_indexer_scores_match_integer_loops():
    rng = np.random.default_rng(7)
    for relu in (True, False):
        for _ in range(20):
            HI, dI, n = rng.integers(1, 5), rng.integers(1, 9), rng.integers(1, 12)
            q = rng.integers(-4, 5, size=(HI, dI))
            k = rng.integers(-4, 5, size=(n, dI))
            w = rng.integers(1, 4, size=HI)
            want = []
            for j in range(n):
                s = 0
                for h in range(HI):
                    d = sum(int(q[h, i]) * int(k[j, i]) for i in range(dI))
                    if relu and d < 0:
                        d = 0
                    s += int(w[h]) * d
                want.append(s)
            got = oracle.indexer_scores(q.astype(np.float64), w.astype(np.float64),
                                        k.astype(np.float64), relu)
            assert got.tolist() == [float(x) for x in want]


def test_block_keys_rounding_half_even_and_partial_block():
    # blocks of 2: sums 1, 3, -1, -3, 5 -> means .5, 1.5, -.5, -1.5, 2.5 -> 0, 2, -0, -2, 2
    keys = np.array([0, 1, 1, 2, 0, -1, -1, -2, 2, 3, 7], dtype=np.float64)[:, None]
    kb = oracle.block_keys(keys, 11, 2, round_to_int=True)
    assert kb[:, 0].tolist() == [0.0, 2.0, 0.0, -2.0, 2.0, 7.0]    # last block holds entry 10 only
    kb = oracle.block_keys(keys, 9, 2, round_to_int=False)
    assert kb[:, 0].tolist() == [0.5, 1.5, -0.5, -1.5, 2.0]      # n_valid = 9: last block = entry 8


def test_block_keys_stored_as_bf16_round_the_mean_to_nearest_even():
    """Unrounded block means stored as bf16 (the fp32-free path of the summary keys): the mean
    of the block's valid keys, computed exactly, then rounded once to bf16, ties to even.
    Hand values (bf16 keeps 8 significant bits; the step above 1 is 2^-7):
      [1, 1 + 2^-7]        -> 1 + 2^-8, halfway between 1 and 1 + 2^-7      -> 1 (even)
      [1, 1 + 3 * 2^-7]    -> 1 + 1.5 * 2^-7, halfway                        -> 1 + 2^-6 (even)
      [2, 3]               -> 2.5, a bf16 value                              -> 2.5
      [1, 1, 2] (partial)  -> 4/3 = 1.0101...b; 8 bits keep 1 + 43 * 2^-7    -> 1.3359375"""
    keys = np.array([1.0, 1 + 2 ** -7, 1.0, 1 + 3 * 2 ** -7, 2.0, 3.0, 1.0, 1.0, 2.0], dtype=np.float64)
    # blocks of 2 over the first 6 keys, then a block of 4 holding 3 valid keys
    kb2 = oracle.block_keys(keys[:6, None], 6, 2, round_to_int=False, store_bf16=True)
    assert kb2[:, 0].tolist() == [1.0, 1 + 2 ** -6, 2.5]
    kb4 = oracle.block_keys(keys[6:, None], 3, 4, round_to_int=False, store_bf16=True)
    assert kb4[:, 0].tolist() == [1 + 43 * 2 ** -7]
    # without bf16 storage the plain means come back
    kb2f = oracle.block_keys(keys[:6, None], 6, 2, round_to_int=False, store_bf16=False)
    assert kb2f[:, 0].tolist() == [1 + 2 ** -8, 1 + 1.5 * 2 ** -7, 2.5]


def test_bf16_decode_and_rounding():
    bits = np.array([0x3F80, 0xC000, 0x3FC0, 0x0000, 0x4080, 0xBE00], dtype=np.uint16)
    assert oracle.to_f64(bits).tolist() == [1.0, -2.0, 1.5, 0.0, 4.0, -0.125]
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1); 1 + 3*2^-8 -> 1 + 2^-6
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 3.0, -(1 + 2 ** -8), 1 + 2 ** -9])
    assert oracle.round_bf16(x).tolist() == [1.0, 1 + 2 ** -6, 3.0, -1.0, 1.0]
    # the generator's rounding agrees with the oracle's decoding on exact values
    v = np.array([1.0, -2.0, 0.5, 3.0, -4.0], dtype=np.float32)
    assert oracle.to_f64(W.f32_to_bf16_bits(v)).tolist() == v.tolist()


# ---------------------------------------------------------------- Top-K

def _heap_topk(scores, ids, k):
    """Independent selection: k smallest of (-score, id) with heapq."""
    s = [(-math.inf if math.isnan(x) else x) for x in scores]
    best = heapq.nsmallest(min(k, len(ids)), zip([-x for x in s], ids))
    out = sorted(i for _, i in best)
    return out + [-1] * (k - len(out))


def test_topk_matches_heap_selection_with_ties():
    rng = np.random.default_rng(11)
    for _ in range(300):
        n = int(rng.integers(0, 40))
        k = int(rng.integers(1, 45))
        scores = rng.integers(-3, 4, size=n).astype(np.float64)
        ids = np.sort(rng.choice(1000, size=n, replace=False))
        assert oracle.select_topk(scores, ids, k).tolist() == _heap_topk(scores.tolist(), ids.tolist(), k)


def test_topk_special_cases():
    ids = np.arange(10)
    # all equal: the lowest ids win
    assert oracle.select_topk(np.zeros(10), ids, 4).tolist() == [0, 1, 2, 3]
    # k >= n: everything, padded with -1
    assert oracle.select_topk(np.arange(3.0), np.arange(3), 5).tolist() == [0, 1, 2, -1, -1]
    # strict order: the largest scores, returned in ascending id order
    assert oracle.select_topk(np.array([1.0, 9, 3, 7, 5]), np.arange(5), 2).tolist() == [1, 3]
    # NaN ranks like -inf (below every finite score; ties with -inf by id)
    s = np.array([np.nan, -np.inf, 0.0, np.nan])
    assert oracle.select_topk(s, np.arange(4), 2).tolist() == [0, 2]


# ---------------------------------------------------------------- hierarchy / modes

def _group(shape, modes, n_valid, seed=3, hier_full=0):
    return W.make_workload(shape, modes, seed=seed, n_valid=n_valid, hier_full=hier_full)


def test_hierarchical_equals_flat_when_pool_covers_every_block():
    for relu in (1, 0):
        sh = W.Shape(batch=3, n_entries=104, idx_heads=3, idx_dim=8, block=8, pool_blocks=13,
                     topk=20, q_heads=2, k_dim=8, v_dim=4, swa=4, relu=relu)
        wl_h = _group(sh, [FULL], n_valid=[104, 97, 1], hier_full=1)
        wl_f = _group(sh, [FULL], n_valid=[104, 97, 1], hier_full=0)
        rh = oracle.run_group(wl_h, want_attention=False)[0]
        rf = oracle.run_group(wl_f, want_attention=False)[0]
        assert np.array_equal(rh["idx"], rf["idx"])
        # and a smaller pool does restrict the candidates to 8 * pool entries
        sh2 = W.Shape(**{**sh.__dict__, "pool_blocks": 3})
        r2 = oracle.run_group(_group(sh2, [FULL], n_valid=[104, 97, 1], hier_full=1),
                              want_attention=False)[0]
        assert len(r2["cand"][0]) == 24 and len(r2["cand"][2]) == 1


def test_reuse_layers_return_the_indexing_layers_indices():
    sh = W.Shape(batch=2, n_entries=64, idx_heads=2, idx_dim=8, block=8, pool_blocks=4,
                 topk=6, q_heads=2, k_dim=8, v_dim=4, swa=4)
    wl = W.make_workload(sh, [FULL, REUSE, REUSE, REINDEX, REUSE], seed=5)
    res = oracle.run_group(wl)
    assert np.array_equal(res[1]["idx"], res[0]["idx"])
    assert np.array_equal(res[2]["idx"], res[0]["idx"])
    assert np.array_equal(res[4]["idx"], res[3]["idx"])
    # each layer still uses its own query: outputs differ between Full and Reuse
    assert not np.allclose(res[0]["out"], res[1]["out"])
    with pytest.raises(ValueError):
        oracle.run_group(W.make_workload(sh, [REUSE], seed=5))


def test_group_counts_of_the_40_layer_pattern():
    enc = W.encoder_stack_modes()
    dec = W.decoder_group_modes()
    assert len(enc) == 20 and len(dec) == 20
    c = oracle.group_counts(enc + dec)
    assert c == {"layers": 40, "csa2": 38, "kv_storing": 4, "indexers": 8}
    assert REINDEX not in enc


# ---------------------------------------------------------------- attention

def _naive_dense(q, k, v, scale):
    """Textbook attention with python loops (fp64)."""
    H, dv = len(q), len(v[0])
    out, lse = [], []
    for h in range(H):
        logits = [scale * sum(q[h][i] * k[j][i] for i in range(len(q[h]))) for j in range(len(k))]
        m = max(logits)
        e = [math.exp(x - m) for x in logits]
        s = sum(e)
        out.append([sum(e[j] * v[j][c] for j in range(len(k))) / s for c in range(dv)])
        lse.append(m + math.log(s))
    return np.array(out), np.array(lse)


def _ratio1_case(T, Wn, K, H, dk, dv, seed):
    """Ratio-1 sequence of T tokens; query at T-1; entries 0..T-1-W, window the rest."""
    rng = np.random.default_rng(seed)
    k_tok = rng.standard_normal((T, dk))
    v_tok = rng.standard_normal((T, dv))
    q = rng.standard_normal((H, dk))
    q_idx = rng.integers(-4, 5, size=(2, 4)).astype(np.float64)
    k_idx = rng.integers(-4, 5, size=(T, 4)).astype(np.float64)
    n_swa = min(Wn, T)
    n_valid = T - n_swa
    return k_tok, v_tok, q, q_idx, k_idx, n_valid, n_swa


@pytest.mark.parametrize("T,Wn,K", [(24, 8, 16), (9, 8, 16), (5, 8, 4), (16, 4, 12)])
def test_sparse_equals_dense_causal_attention_naive(T, Wn, K):
    k_tok, v_tok, q, q_idx, k_idx, n_valid, n_swa = _ratio1_case(T, Wn, K, 3, 5, 4, T)
    sel = oracle.layer_indices(q_idx, np.ones(2), k_idx, None, n_valid, topk=K, block=2, pool=0,
                               hier=False)["idx"]
    scale = 1 / math.sqrt(5)
    out, lse = oracle.sparse_attention(q, k_tok, v_tok, sel, k_tok[n_valid:], v_tok[n_valid:],
                                       n_swa, scale)
    ref_out, ref_lse = _naive_dense(q.tolist(), k_tok.tolist(), v_tok.tolist(), scale)
    assert np.allclose(out, ref_out, rtol=0, atol=1e-12)
    assert np.allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_sparse_equals_dense_attention_sdpa_at_512_plus_128():
    torch = pytest.importorskip("torch")
    T, Wn, K, H, dk, dv = 640, 128, 512, 4, 192, 128
    k_tok, v_tok, q, q_idx, k_idx, n_valid, n_swa = _ratio1_case(T, Wn, K, H, dk, dv, 1)
    sel = oracle.layer_indices(q_idx, np.ones(2), k_idx, None, n_valid, topk=K, block=8, pool=0,
                               hier=False)["idx"]
    assert (sel >= 0).sum() == 512
    out, lse = oracle.sparse_attention(q, k_tok, v_tok, sel, k_tok[n_valid:], v_tok[n_valid:],
                                       n_swa, 1 / math.sqrt(dk))
    qt = torch.tensor(q)[:, None, :]                    # [H, 1, dk]
    kt = torch.tensor(k_tok)[None].expand(H, T, dk)
    vt = torch.tensor(v_tok)[None].expand(H, T, dv)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[:, 0, :].numpy()
    assert np.allclose(out, ref, rtol=0, atol=1e-12)
    ref_lse = torch.logsumexp(torch.einsum("hd,td->ht", torch.tensor(q), torch.tensor(k_tok))
                              / math.sqrt(dk), dim=1).numpy()
    assert np.allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(2)
    H, dk, dv, N = 3, 6, 5, 30
    k_main = rng.standard_normal((N, dk))
    v_main = rng.standard_normal((N, dv))
    k_swa = rng.standard_normal((4, dk))
    v_swa = rng.standard_normal((4, dv))
    idx = np.array([3, 7, 19, -1, -1])
    # q = 0: uniform weights -> mean of the attended V rows, lse = log(n)
    out, lse = oracle.sparse_attention(np.zeros((H, dk)), k_main, v_main, idx, k_swa, v_swa, 4, 0.7)
    want = np.concatenate([v_main[[3, 7, 19]], v_swa]).mean(axis=0)
    assert np.allclose(out, want[None, :], atol=1e-13) and np.allclose(lse, math.log(7))
    # a single attended key -> its V row, lse = scale * q.k
    q = rng.standard_normal((H, dk))
    out, lse = oracle.sparse_attention(q, k_main, v_main, np.array([11, -1]), k_swa, v_swa, 0, 0.3)
    assert np.allclose(out, v_main[11][None, :], atol=1e-13)
    assert np.allclose(lse, 0.3 * q @ k_main[11], atol=1e-13)
    # no key at all -> zero output, lse = -inf
    out, lse = oracle.sparse_attention(q, k_main, v_main, np.array([-1]), k_swa, v_swa, 0, 0.3)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    # invariance under a permutation of the cache rows (indices remapped)
    perm = rng.permutation(N)
    inv = np.argsort(perm)
    idx = np.array([0, 5, 9, 28])
    a, la = oracle.sparse_attention(q, k_main, v_main, idx, k_swa, v_swa, 4, 0.4)
    b, lb = oracle.sparse_attention(q, k_main[perm], v_main[perm], inv[idx], k_swa, v_swa, 4, 0.4)
    assert np.allclose(a, b, atol=1e-13) and np.allclose(la, lb, atol=1e-13)
    # the softmax scale multiplies the logits (a doubled scale != the original)
    c, _ = oracle.sparse_attention(q, k_main, v_main, idx, k_swa, v_swa, 4, 0.8)
    assert not np.allclose(a, c)


def test_swa_layer_is_window_only_attention():
    """A pure sliding-window layer equals textbook attention over its window rows."""
    sh = W.Shape(batch=2, n_entries=64, idx_heads=2, idx_dim=8, block=8, pool_blocks=0, topk=6, q_heads=2,
                 k_dim=5, v_dim=3, swa=7)
    wl = W.make_workload(sh, [W.SWA, W.FULL, W.SWA], seed=9, n_swa=[7, 3])
    res = oracle.run_group(wl)
    for li in (0, 2):
        L = wl.layers[li]
        for b in range(2):
            ns = int(wl.n_swa[b])
            ref_out, ref_lse = _naive_dense(oracle.to_f64(L.q[b]).tolist(), oracle.to_f64(L.k_swa[b])[:ns].tolist(),
                                            oracle.to_f64(L.v_swa[b])[:ns].tolist(), 1 / math.sqrt(5))
            assert np.allclose(res[li]["out"][b], ref_out, atol=1e-12)
            assert np.allclose(res[li]["lse"][b], ref_lse, atol=1e-12)
    assert "idx" not in res[0]


# ---------------------------------------------------------------- cache maintenance (append)

def _bf16_ints(rng, shape):
    return W.f32_to_bf16_bits(rng.integers(-4, 5, shape).astype(np.float32))


def test_kv_append_in_steps_equals_the_cache_written_at_once():
    """Entries appended in random-sized steps, some past the cache's end, give the
    cache written in one go: the rows in arrival order, n_valid capped at N, and
    summary keys equal to block_keys over the final cache (blocks past the
    valid entries untouched)."""
    rng = np.random.default_rng(5)
    B, N, dk, dv, dI, blk = 3, 37, 3, 2, 4, 8
    start = np.array([0, 11, 30])
    k_main = rng.integers(0, 60000, (B, N, dk)).astype(np.uint16)     # rows past n_valid: arbitrary
    v_main = rng.integers(0, 60000, (B, N, dv)).astype(np.uint16)
    k_idx = _bf16_ints(rng, (B, N, dI))
    nb = -(-N // blk)
    kb = np.zeros((B, nb, dI))
    for b in range(B):
        nbv = -(-int(start[b]) // blk)
        kb[b, :nbv] = oracle.block_keys(oracle.to_f64(k_idx[b]), int(start[b]), blk, True)
    T = 40                                                              # more than fits for every query
    ks = rng.integers(0, 60000, (B, T, dk)).astype(np.uint16)
    vs = rng.integers(0, 60000, (B, T, dv)).astype(np.uint16)
    xs = _bf16_ints(rng, (B, T, dI))
    cur = (k_main, v_main, k_idx, kb, start.copy())
    fed = np.zeros(B, dtype=np.int64)
    dropped = np.zeros(B, dtype=np.int64)
    while (fed < T).any():
        n_new = np.minimum(rng.integers(0, 5, B), T - fed)
        mx = int(n_new.max()) if n_new.max() > 0 else 1
        take = lambda a, d: np.stack([np.pad(a[b, fed[b]:fed[b] + n_new[b]], ((0, mx - n_new[b]), (0, 0)))
                                      for b in range(B)])
        *cur, dr = oracle.kv_append(*cur, n_new, take(ks, dk), take(vs, dv), take(xs, dI), block=blk,
                                    round_to_int=True)
        fed += n_new
        dropped += dr
    k1, v1, x1, kb1, nv1 = cur
    for b in range(B):
        fit = N - start[b]
        assert nv1[b] == N and dropped[b] == T - fit
        assert np.array_equal(k1[b, :start[b]], k_main[b, :start[b]])
        assert np.array_equal(k1[b, start[b]:], ks[b, :fit])
        assert np.array_equal(v1[b, start[b]:], vs[b, :fit])
        assert np.array_equal(x1[b, start[b]:], xs[b, :fit])
        full = oracle.block_keys(oracle.to_f64(x1[b]), N, blk, True)
        assert np.array_equal(kb1[b], full)


def test_kv_append_touches_only_the_blocks_of_the_new_positions():
    keys = np.arange(40, dtype=np.float64).reshape(20, 2)        # entry e has keys (2e, 2e+1)
    k_idx = np.zeros((1, 24, 2))
    k_idx[0, :20] = keys
    kb = np.full((1, 3, 2), 99.0)                                # stale values everywhere
    new = np.array([[[100.0, 101.0], [102.0, 103.0]]])
    _, _, x, kb1, nv, dr = oracle.kv_append(np.zeros((1, 24, 1)), np.zeros((1, 24, 1)), k_idx, kb, [15], [2],
                                            np.zeros((1, 2, 1)), np.zeros((1, 2, 1)), new, block=8,
                                            round_to_int=False, store_bf16=False)
    assert nv.tolist() == [17] and dr.tolist() == [0]
    assert x[0, 15].tolist() == [100.0, 101.0] and x[0, 16].tolist() == [102.0, 103.0]
    # block 1 holds entries 8..15: keys 16..29 (even) / 17..31 (odd) with entry 15 replaced by (100, 101)
    assert kb1[0, 1].tolist() == [(sum(range(16, 30, 2)) + 100) / 8, (sum(range(17, 31, 2)) + 101) / 8]
    assert kb1[0, 2].tolist() == [102.0, 103.0]                 # block 2 holds entry 16 only
    assert kb1[0, 0].tolist() == [99.0, 99.0]                   # block 0 untouched


def test_swa_ring_holds_the_last_w_tokens():
    from collections import deque
    Wn, T, B = 5, 13, 2
    rng = np.random.default_rng(9)
    toks = rng.integers(0, 60000, (T, B, 3)).astype(np.uint16)
    k_swa = np.zeros((B, Wn, 3), dtype=np.uint16)
    v_swa = np.zeros((B, Wn, 3), dtype=np.uint16)
    head, n = np.zeros(B, dtype=np.int64), np.zeros(B, dtype=np.int64)
    last = [deque(maxlen=Wn) for _ in range(B)]
    for t in range(T):
        k_swa, v_swa, head, n = oracle.swa_append(k_swa, v_swa, head, n, toks[t], toks[t] + 1)
        for b in range(B):
            last[b].append(tuple(toks[t, b]))
            assert n[b] == min(t + 1, Wn) and head[b] == (t + 1) % Wn
            assert sorted(tuple(r) for r in k_swa[b, :n[b]]) == sorted(last[b])
            assert sorted(tuple(r) for r in v_swa[b, :n[b]]) == sorted(tuple(np.array(x) + 1) for x in last[b])


def test_attention_over_the_ring_equals_attention_oldest_first():
    rng = np.random.default_rng(3)
    H, dk, dv, Wn, N = 4, 6, 5, 7, 20
    q = rng.standard_normal((H, dk))
    k_main, v_main = rng.standard_normal((N, dk)), rng.standard_normal((N, dv))
    idx = np.array([3, 8, 11, -1])
    k_old, v_old = rng.standard_normal((Wn, dk)), rng.standard_normal((Wn, dv))
    shift = 4                                                    # ring after Wn + 4 appends
    ring = np.roll(np.arange(Wn), shift)
    a = oracle.sparse_attention(q, k_main, v_main, idx, k_old, v_old, Wn, 0.4)
    b = oracle.sparse_attention(q, k_main, v_main, idx, k_old[ring], v_old[ring], Wn, 0.4)
    np.testing.assert_allclose(a[0], b[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- several tokens per sequence

def test_decoder_replay_shares_caches_and_slides_the_windows():
    """With T tokens per sequence the oracle reads sequence b // T; copying that
    sequence's caches to every query gives the same result.  The workload's
    windows slide by one raw token per query, and n_valid is causal at ratio 4."""
    T = 8
    wl = W.decoder_replay(2, T, 1000, n_entries=256, pool=8, modes=[FULL, REINDEX, REUSE], seed=1)
    pos = 1000 - T + np.arange(T)
    assert wl.n_valid.tolist() == list((pos + 1) // 4) * 2
    for L in wl.layers:
        for b in range(2 * T - 1):
            if b % T != T - 1:        # consecutive tokens of one sequence: the window moves by one row
                assert np.array_equal(L.k_swa[b, 1:], L.k_swa[b + 1, :-1])
    import dataclasses
    rep = lambda a: np.repeat(a, T, axis=0)
    flat = dataclasses.replace(wl, shape=dataclasses.replace(wl.shape, tokens=1), k_main=rep(wl.k_main),
                               v_main=rep(wl.v_main), k_idx=rep(wl.k_idx))
    qs = [0, 3, 9, 15]
    a, b = oracle.run_group(wl, queries=qs), oracle.run_group(flat, queries=qs)
    for x, y in zip(a, b):
        assert np.array_equal(x["idx"], y["idx"]) and np.array_equal(x["out"], y["out"])


def test_tokens_of_one_sequence_see_their_own_partial_last_block():
    """Two query tokens of one sequence (shape.tokens = 2) share its indexer keys but have
    different causal counts, so their partial last blocks differ.  Hand case, blocks of 2,
    a pool of one block, Top-1, one indexer head with q = w = 1 (score = the key):
      keys 1, 1, 0, 9, 5, 5
      token 0, n_valid 3: block keys 1, 0 (its last block holds entry 2 only) -> pool [0]
                          -> candidates 0, 1 (scores 1, 1) -> Top-1 [0] (tie: lowest id)
      token 1, n_valid 4: block keys 1, rint(4.5) = 4 -> pool [1] -> candidates 2, 3
                          (scores 0, 9) -> Top-1 [3]
    Block keys taken over the sequence's whole cache would give token 0 the pool [1]
    and the index [2] (entry 3 lies past its n_valid)."""
    sh = W.Shape(batch=2, n_entries=6, idx_heads=1, idx_dim=1, block=2, pool_blocks=1, topk=1, q_heads=1,
                 k_dim=1, v_dim=1, swa=1, dtype="f32", tokens=2)
    one = np.ones((2, 1, 1), dtype=np.float32)
    layer = W.Layer(mode=REINDEX, hier=1, q=one, k_swa=one.copy(), v_swa=one.copy(), q_idx=one.copy(),
                    w_idx=np.ones((2, 1), dtype=np.float32))
    keys = np.array([1, 1, 0, 9, 5, 5], dtype=np.float32)[None, :, None]
    wl = W.Workload(name="tokens_hand", shape=sh, k_main=keys.copy(), v_main=keys.copy(), k_idx=keys,
                    n_valid=np.array([3, 4], dtype=np.int32), n_swa=np.array([0, 0], dtype=np.int32),
                    layers=[layer], round_block_keys=1)
    r = oracle.run_group(wl)[0]
    assert [p.tolist() for p in r["pool"]] == [[0], [1]]
    assert [c.tolist() for c in r["cand"]] == [[0, 1], [2, 3]]
    assert r["idx"].tolist() == [[0], [3]]
    # attention reads the selected entry's K/V (no window): out = its value row
    assert r["out"][:, 0, 0].tolist() == [1.0, 9.0]
