"""Per-entry-point parity of the CUDA path against the CPU oracle (through the C ABI)."""
import math

import numpy as np
import pytest

import oracle
from sparse_attention_decode_index_gb300 import workloads as W
from tests.gpu_helpers import (assert_no_device_error, bf16, compare_attention, f32, i32, lib_ready,
                               need_gpu, torch)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    need_gpu()
    return lib_ready()


def _shape(**kw):
    base = dict(batch=3, n_entries=2048, idx_heads=8, idx_dim=64, block=8, pool_blocks=64, topk=512,
                q_heads=64, k_dim=192, v_dim=128, swa=128)
    base.update(kw)
    return W.Shape(**base)


def _int_keys(rng, shape):
    return W.f32_to_bf16_bits(rng.integers(-4, 5, size=shape).astype(np.float32))


# ------------------------------------------------------------------ block keys

@pytest.mark.parametrize("round_to_int", [1, 0])
def test_block_keys(csa2, round_to_int):
    rng = np.random.default_rng(1)
    sh = _shape(batch=4, n_entries=200)
    k_idx = _int_keys(rng, (4, 200, 64))
    n_valid = np.array([200, 197, 1, 0], dtype=np.int32)
    nb = 25
    kb = torch.full((4, nb, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = csa2.workspace(sh)
    csa2.block_keys(sh, bf16(k_idx), i32(n_valid), kb, ws, round_to_int=bool(round_to_int))
    got = kb.float().cpu().numpy()
    for b in range(4):
        want = oracle.block_keys(oracle.to_f64(k_idx[b]), int(n_valid[b]), 8, bool(round_to_int),
                                 store_bf16=True)
        nbv = want.shape[0]
        assert np.array_equal(got[b, :nbv], want), f"query {b}"
        assert np.all(got[b, nbv:] == 0)
    assert_no_device_error(csa2, ws)


# ------------------------------------------------------------------ indexer

@pytest.mark.parametrize("relu", [1, 0])
def test_index_tokens_flat_fast(csa2, relu):
    rng = np.random.default_rng(2)
    N = 2048 + 136
    sh = _shape(batch=5, n_entries=N, relu=relu)
    k_idx = _int_keys(rng, (5, N, 64))
    q_idx = _int_keys(rng, (5, 8, 64))
    w = rng.integers(1, 4, size=(5, 8)).astype(np.float32)
    n_valid = np.array([N, N - 1, 129, 1, 0], dtype=np.int32)
    assert csa2.fast_path(sh)[0]
    ws = csa2.workspace(sh)
    scores = torch.full((5, N), -7.0, dtype=torch.float32, device="cuda")
    cand = torch.full((5, N), -9, dtype=torch.int32, device="cuda")
    n_cand = torch.zeros(5, dtype=torch.int32, device="cuda")
    csa2.index_tokens(sh, bf16(q_idx), f32(w), bf16(k_idx), i32(n_valid), scores, ws, cand_out=cand,
                      n_cand_out=n_cand)
    s = scores.cpu().numpy()
    c = cand.cpu().numpy()
    assert n_cand.cpu().numpy().tolist() == n_valid.tolist()
    for b in range(5):
        n = int(n_valid[b])
        want = oracle.indexer_scores(oracle.to_f64(q_idx[b]), w[b].astype(np.float64),
                                     oracle.to_f64(k_idx[b, :n]), bool(relu))
        assert np.array_equal(s[b, :n].astype(np.float64), want), f"query {b}"
        assert np.array_equal(c[b, :n], np.arange(n))
        assert np.all(s[b, n:] == -7.0)
    assert_no_device_error(csa2, ws)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_index_tokens_flat_generic(csa2, dtype):
    rng = np.random.default_rng(3)
    N = 300
    sh = _shape(batch=2, n_entries=N, idx_heads=3, idx_dim=5, dtype=dtype)
    assert not csa2.fast_path(sh)[0]
    ki = rng.integers(-4, 5, size=(2, N, 5)).astype(np.float32)
    qi = rng.integers(-4, 5, size=(2, 3, 5)).astype(np.float32)
    w = rng.integers(1, 4, size=(2, 3)).astype(np.float32)
    if dtype == "bf16":
        k_dev, q_dev = bf16(W.f32_to_bf16_bits(ki)), bf16(W.f32_to_bf16_bits(qi))
    else:
        k_dev, q_dev = f32(ki), f32(qi)
    n_valid = np.array([N, 77], dtype=np.int32)
    ws = csa2.workspace(sh)
    scores = torch.zeros((2, N), dtype=torch.float32, device="cuda")
    csa2.index_tokens(sh, q_dev, f32(w), k_dev, i32(n_valid), scores, ws)
    s = scores.cpu().numpy()
    for b in range(2):
        n = int(n_valid[b])
        want = oracle.indexer_scores(qi[b].astype(np.float64), w[b].astype(np.float64),
                                     ki[b, :n].astype(np.float64))
        assert np.array_equal(s[b, :n].astype(np.float64), want)


@pytest.mark.parametrize("fast", [True, False])
def test_index_blocks_and_pooled_tokens(csa2, fast):
    rng = np.random.default_rng(4)
    N, P = 4096, 64
    kw = dict(batch=4, n_entries=N, pool_blocks=P)
    if not fast:
        kw.update(idx_heads=4, idx_dim=16)
    sh = _shape(**kw)
    HI, dI = sh.idx_heads, sh.idx_dim
    assert csa2.fast_path(sh)[0] == fast
    k_idx = _int_keys(rng, (4, N, dI))
    q_idx = _int_keys(rng, (4, HI, dI))
    w = rng.integers(1, 4, size=(4, HI)).astype(np.float32)
    n_valid = np.array([N, N - 5, 8 * P - 3, 100], dtype=np.int32)     # last: fewer blocks than the pool
    ws = csa2.workspace(sh)
    kb = torch.zeros((4, N // 8, dI), dtype=torch.bfloat16, device="cuda")
    csa2.block_keys(sh, bf16(k_idx), i32(n_valid), kb, ws, round_to_int=True)
    pool = torch.full((4, P), -5, dtype=torch.int32, device="cuda")
    n_pool = torch.zeros(4, dtype=torch.int32, device="cuda")
    csa2.index_blocks(sh, bf16(q_idx), f32(w), kb, i32(n_valid), pool, n_pool, ws)
    L = P * 8
    scores = torch.zeros((4, L), dtype=torch.float32, device="cuda")
    cand = torch.zeros((4, L), dtype=torch.int32, device="cuda")
    n_cand = torch.zeros(4, dtype=torch.int32, device="cuda")
    csa2.index_tokens(sh, bf16(q_idx), f32(w), bf16(k_idx), i32(n_valid), scores, ws, pool=pool, n_pool=n_pool,
                      cand_out=cand, n_cand_out=n_cand)
    pool_h, np_h = pool.cpu().numpy(), n_pool.cpu().numpy()
    s, c, nc = scores.cpu().numpy(), cand.cpu().numpy(), n_cand.cpu().numpy()
    for b in range(4):
        n = int(n_valid[b])
        keys = oracle.to_f64(k_idx[b])
        kbo = oracle.block_keys(keys, n, 8, True)
        want_pool = oracle.pool_blocks(oracle.to_f64(q_idx[b]), w[b].astype(np.float64), kbo, kbo.shape[0], P)
        npl = len(want_pool)
        assert int(np_h[b]) == npl
        assert pool_h[b, :npl].tolist() == want_pool.tolist(), f"pool of query {b}"
        assert np.all(pool_h[b, npl:] == -1)
        assert int(nc[b]) == npl * 8
        ent = (want_pool[:, None] * 8 + np.arange(8)[None, :]).reshape(-1)
        ok = ent < n
        assert c[b, :npl * 8].tolist() == np.where(ok, ent, -1).tolist()
        want_s = oracle.indexer_scores(oracle.to_f64(q_idx[b]), w[b].astype(np.float64), keys[ent[ok]])
        assert np.array_equal(s[b, :npl * 8][ok].astype(np.float64), want_s)
    assert_no_device_error(csa2, ws)


# ------------------------------------------------------------------ Top-K

@pytest.mark.parametrize("n,k,spread", [(10, 512, 3), (700, 512, 3), (4096, 2048, 50), (16384, 512, 400),
                                        (16384, 512, 2), (20000, 512, 1000), (300000, 512, 5000),
                                        (16384, 1, 0), (5000, 4999, 7)])
def test_topk_exact(csa2, n, k, spread):
    rng = np.random.default_rng(n + k)
    B = 3
    sh = _shape(batch=B, n_entries=max(n, 16), topk=min(k, 1024), swa=0, pool_blocks=0)
    sc = rng.integers(-spread, spread + 1, size=(B, n)).astype(np.float32)
    sc[1] = np.round(sc[1] * 0.37, 2).astype(np.float32)                         # non-integer values
    if n > 3:
        sc[2, :3] = [np.nan, -0.0, 0.0]
    n_cand = np.array([n, max(n - 11, 0), n // 2], dtype=np.int32)
    ws = csa2.workspace(sh)
    idx = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
    vals = torch.zeros((B, k), dtype=torch.float32, device="cuda")
    csa2.topk(sh, f32(sc), k, idx, ws, n_cand=i32(n_cand), score_out=vals)
    got = idx.cpu().numpy()
    gv = vals.cpu().numpy()
    for b in range(B):
        m = int(n_cand[b])
        want = oracle.select_topk(sc[b, :m].astype(np.float64), np.arange(m), k)
        assert got[b].tolist() == want.tolist(), f"row {b}"
        sel = want >= 0
        ref = sc[b][want[sel]].astype(np.float64)
        ref = np.where(np.isnan(ref), -np.inf, ref)
        assert np.array_equal(gv[b][sel].astype(np.float64), ref)
    assert_no_device_error(csa2, ws)


def test_topk_candidate_ids_and_skips(csa2):
    rng = np.random.default_rng(9)
    B, n, k = 2, 3000, 100
    sh = _shape(batch=B, n_entries=n, topk=k, pool_blocks=0)
    sc = rng.integers(0, 20, size=(B, n)).astype(np.float32)
    ids = np.sort(rng.choice(10 ** 6, size=(B, n), replace=False), axis=1).astype(np.int32)
    ids[0, ::7] = -1                                                                 # skipped positions
    ws = csa2.workspace(sh)
    idx = torch.zeros((B, k), dtype=torch.int32, device="cuda")
    csa2.topk(sh, f32(sc), k, idx, ws, cand=i32(ids))
    got = idx.cpu().numpy()
    for b in range(B):
        keep = ids[b] >= 0
        want = oracle.select_topk(sc[b][keep].astype(np.float64), ids[b][keep].astype(np.int64), k)
        assert got[b].tolist() == want.tolist()


# ------------------------------------------------------------------ attention

def _attn_case(rng, B, N, H, dk, dv, K, Wn, dtype="bf16"):
    def draw(shape, div):
        x = rng.standard_normal(shape).astype(np.float32) / np.float32(div)
        return W.f32_to_bf16_bits(x) if dtype == "bf16" else x
    q = draw((B, H, dk), 1.0)
    km, vm = draw((B, N, dk), math.sqrt(dk)), draw((B, N, dv), math.sqrt(dv))
    ks, vs = draw((B, Wn, dk), math.sqrt(dk)), draw((B, Wn, dv), math.sqrt(dv))
    idx = np.full((B, K), -1, dtype=np.int32)
    for b in range(B):
        m = [K, K, K // 3, 0, 7][b % 5]
        idx[b, :m] = np.sort(rng.choice(N, size=m, replace=False))
    return q, km, vm, ks, vs, idx


@pytest.mark.parametrize("fast", [True, False])
def test_sparse_attn(csa2, fast):
    rng = np.random.default_rng(5)
    if fast:
        B, N, H, dk, dv, K, Wn = 6, 3000, 64, 192, 128, 512, 128
        dtype = "bf16"
    else:
        B, N, H, dk, dv, K, Wn = 5, 300, 4, 24, 40, 32, 16
        dtype = "f32"
    sh = _shape(batch=B, n_entries=N, q_heads=H, k_dim=dk, v_dim=dv, topk=K, swa=Wn, dtype=dtype, pool_blocks=0)
    assert csa2.fast_path(sh)[1] == fast
    q, km, vm, ks, vs, idx = _attn_case(rng, B, N, H, dk, dv, K, Wn, dtype)
    n_swa = np.array([Wn, 5, Wn, 0, 0, Wn][:B], dtype=np.int32)
    up = bf16 if dtype == "bf16" else f32
    out = torch.full((B, H, dv), 3.0, dtype=torch.float32, device="cuda")
    lse = torch.zeros((B, H), dtype=torch.float32, device="cuda")
    ws = csa2.workspace(sh)
    csa2.sparse_attn(sh, up(q), up(km), up(vm), i32(idx), up(ks), up(vs), i32(n_swa), out, ws, lse=lse)
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    ref_o = np.zeros((B, H, dv))
    ref_l = np.zeros((B, H))
    for b in range(B):
        ref_o[b], ref_l[b] = oracle.sparse_attention(oracle.to_f64(q[b]), oracle.to_f64(km[b]),
                                                     oracle.to_f64(vm[b]), idx[b].astype(np.int64),
                                                     oracle.to_f64(ks[b]), oracle.to_f64(vs[b]), int(n_swa[b]),
                                                     1 / math.sqrt(dk))
    e, le = compare_attention(o, l, ref_o, ref_l, atol=1e-2 if fast else 1e-4)
    print(f"sparse_attn fast={fast}: max-abs out {e:.2e} lse {le:.2e}")
    assert_no_device_error(csa2, ws)


@pytest.mark.parametrize("K,Wn", [(128, 16), (256, 32), (384, 64), (700, 64), (800, 64), (896, 128)])
def test_sparse_attn_cluster_sizes(csa2, K, Wn):
    """Clusters of 1, 2, 3, 5, 6 and 7 CTAs (the smallest C with ceil(K / C) + ceil(Wn / C) <= 160
    slots; K + Wn <= 1024 keeps C below 8): every CTA merges ceil(64 / C) heads, the last fewer
    when C does not divide 64."""
    rng = np.random.default_rng(K + Wn)
    B, N, H, dk, dv = 5, 3000, 64, 192, 128
    sh = _shape(batch=B, n_entries=N, q_heads=H, k_dim=dk, v_dim=dv, topk=K, swa=Wn, pool_blocks=0)
    assert csa2.fast_path(sh)[1]
    q, km, vm, ks, vs, idx = _attn_case(rng, B, N, H, dk, dv, K, Wn)
    n_swa = np.array([Wn, 3, 0, 0, 1], dtype=np.int32)   # row 3: no key at all (lse -inf, output 0)
    for b in range(B):   # window rows past the count are not part of the window: NaN must not leak
        ks[b, n_swa[b]:] = 0x7fc0
        vs[b, n_swa[b]:] = 0x7fc0
    out = torch.full((B, H, dv), 3.0, dtype=torch.float32, device="cuda")
    lse = torch.zeros((B, H), dtype=torch.float32, device="cuda")
    ws = csa2.workspace(sh)
    csa2.sparse_attn(sh, bf16(q), bf16(km), bf16(vm), i32(idx), bf16(ks), bf16(vs), i32(n_swa), out, ws, lse=lse)
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    ref_o, ref_l = np.zeros((B, H, dv)), np.zeros((B, H))
    for b in range(B):
        ref_o[b], ref_l[b] = oracle.sparse_attention(oracle.to_f64(q[b]), oracle.to_f64(km[b]),
                                                     oracle.to_f64(vm[b]), idx[b].astype(np.int64),
                                                     oracle.to_f64(ks[b]), oracle.to_f64(vs[b]), int(n_swa[b]),
                                                     1 / math.sqrt(dk))
    compare_attention(o, l, ref_o, ref_l, atol=1e-2)
    assert_no_device_error(csa2, ws)


def test_sparse_attn_flags_out_of_range_index(csa2):
    rng = np.random.default_rng(6)
    B, N = 2, 1000
    sh = _shape(batch=B, n_entries=N, pool_blocks=0)
    q, km, vm, ks, vs, idx = _attn_case(rng, B, N, 64, 192, 128, 512, 128)
    bad = idx.copy()
    bad[0, 3] = N + 5                       # outside the cache: must be skipped and reported
    out = torch.zeros((B, 64, 128), dtype=torch.float32, device="cuda")
    ws = csa2.workspace(sh)
    n_swa = i32(np.full(B, 128))
    csa2.sparse_attn(sh, bf16(q), bf16(km), bf16(vm), i32(bad), bf16(ks), bf16(vs), n_swa, out, ws)
    st, bits = csa2.read_device_error(ws)
    assert st == -5 and bits & 1
    assert csa2.read_device_error(ws)[0] == 0            # cleared by the read
    skipped = bad[0].astype(np.int64)
    skipped[3] = -1
    ref, _ = oracle.sparse_attention(oracle.to_f64(q[0]), oracle.to_f64(km[0]), oracle.to_f64(vm[0]), skipped,
                                     oracle.to_f64(ks[0]), oracle.to_f64(vs[0]), 128, 1 / math.sqrt(192))
    assert np.abs(out.cpu().numpy()[0] - ref).max() <= 1e-2


# ------------------------------------------------------------------ fused scoring + Top-k

@pytest.mark.parametrize("mode", ["flat", "pooled", "generic"])
def test_index_topk_fused(csa2, mode):
    rng = np.random.default_rng(12)
    B, N, P, K = 5, 4096, 64, 256
    kw = dict(batch=B, n_entries=N, pool_blocks=P, topk=K)
    if mode == "generic":
        kw.update(idx_heads=4, idx_dim=16)
    sh = _shape(**kw)
    HI, dI = sh.idx_heads, sh.idx_dim
    k_idx = _int_keys(rng, (B, N, dI))
    q_idx = _int_keys(rng, (B, HI, dI))
    w = rng.integers(1, 4, size=(B, HI)).astype(np.float32)
    n_valid = np.array([N, N - 5, 8 * P - 3, 100, 0], dtype=np.int32)
    ws = csa2.workspace(sh)
    pool = n_pool = None
    if mode != "flat":
        kb = torch.zeros((B, N // 8, dI), dtype=torch.bfloat16, device="cuda")
        csa2.block_keys(sh, bf16(k_idx), i32(n_valid), kb, ws, round_to_int=True)
        pool = torch.zeros((B, P), dtype=torch.int32, device="cuda")
        n_pool = torch.zeros(B, dtype=torch.int32, device="cuda")
        csa2.index_blocks(sh, bf16(q_idx), f32(w), kb, i32(n_valid), pool, n_pool, ws)
    for k in (K, 37):
        idx = torch.full((B, k), -9, dtype=torch.int32, device="cuda")
        n_out = torch.zeros(B, dtype=torch.int32, device="cuda")
        csa2.index_topk(sh, bf16(q_idx), f32(w), bf16(k_idx), i32(n_valid), k, idx, ws, pool=pool, n_pool=n_pool,
                        n_out=n_out)
        got = idx.cpu().numpy()
        for b in range(B):
            keys = oracle.to_f64(k_idx[b])
            n = int(n_valid[b])
            kb_o = oracle.block_keys(keys, n, 8, True) if mode != "flat" else None
            r = oracle.layer_indices(oracle.to_f64(q_idx[b]), w[b].astype(np.float64), keys, kb_o, n, topk=k,
                                     block=8, pool=P, hier=mode != "flat")
            assert got[b].tolist() == r["idx"].tolist(), f"{mode} k={k} query {b}"
            assert int(n_out.cpu().numpy()[b]) == int((r["idx"] >= 0).sum())
    assert_no_device_error(csa2, ws)


@pytest.mark.parametrize("mode", ["flat", "pooled"])
def test_index_topk_fused_clusters_of_16(csa2, mode):
    """Small batches over many rows take clusters of 16 CTAs (a non-portable size): 32,768
    flat rows (2,048 per CTA), or a pool of 2,048 blocks (16,384 rows, 1,024 per CTA).
    Integer keys tie heavily; one query is ragged, one nearly empty."""
    rng = np.random.default_rng(16)
    B, N, P = 3, 32768, 2048
    sh = _shape(batch=B, n_entries=N, pool_blocks=P if mode == "pooled" else 0, topk=512)
    k_idx = _int_keys(rng, (B, N, sh.idx_dim))
    q_idx = _int_keys(rng, (B, sh.idx_heads, sh.idx_dim))
    w = rng.integers(1, 4, size=(B, sh.idx_heads)).astype(np.float32)
    n_valid = np.array([N, 20001, 777], dtype=np.int32)
    ws = csa2.workspace(sh)
    pool = n_pool = None
    if mode == "pooled":
        kb = torch.zeros((B, N // 8, sh.idx_dim), dtype=torch.bfloat16, device="cuda")
        csa2.block_keys(sh, bf16(k_idx), i32(n_valid), kb, ws, round_to_int=True)
        pool = torch.zeros((B, P), dtype=torch.int32, device="cuda")
        n_pool = torch.zeros(B, dtype=torch.int32, device="cuda")
        csa2.index_blocks(sh, bf16(q_idx), f32(w), kb, i32(n_valid), pool, n_pool, ws)
    for k in (512, 37):
        idx = torch.full((B, k), -9, dtype=torch.int32, device="cuda")
        csa2.index_topk(sh, bf16(q_idx), f32(w), bf16(k_idx), i32(n_valid), k, idx, ws, pool=pool, n_pool=n_pool)
        got = idx.cpu().numpy()
        for b in range(B):
            keys = oracle.to_f64(k_idx[b])
            n = int(n_valid[b])
            kb_o = oracle.block_keys(keys, n, 8, True) if mode == "pooled" else None
            r = oracle.layer_indices(oracle.to_f64(q_idx[b]), w[b].astype(np.float64), keys, kb_o, n, topk=k,
                                     block=8, pool=P, hier=mode == "pooled")
            assert got[b].tolist() == r["idx"].tolist(), f"{mode} k={k} query {b}"
    assert_no_device_error(csa2, ws)


@pytest.mark.parametrize("group,spread", [(1000, 2), (1000, 1), (340, 1), (280, 1), (280, 2)])
def test_index_topk_fused_large_threshold_bin(csa2, group, spread):
    """Fused flat scoring + Top-k when the bin holding the k-th score gathers `group`
    keys: one-hot queries make every score 8 * k_idx[:, 0], with 100 rows at 2,560,
    `group` rows at 1,000 or 1,008 (one bin; all 1,000 when spread is 1, a tie across
    the CTAs), the rest at 0.  1,000 and 340 gathered keys take the radix passes over
    the gathered keys; 280 (at most 304 words with padding) take the rank-count finish."""
    rng = np.random.default_rng(41)
    B, N, K = 2, 4096, 256
    sh = _shape(batch=B, n_entries=N, topk=K, pool_blocks=0)
    col0 = np.zeros((B, N), dtype=np.float32)
    for b in range(B):
        rows = rng.permutation(N)
        col0[b, rows[:100]] = 320.0
        col0[b, rows[100:100 + group]] = 125.0 + rng.integers(0, spread, size=group)
    k_f = np.zeros((B, N, sh.idx_dim), dtype=np.float32)
    k_f[:, :, 0] = col0
    k_f[:, :, 1:] = rng.integers(-4, 5, size=(B, N, sh.idx_dim - 1))   # ignored by the one-hot queries
    k_idx = W.f32_to_bf16_bits(k_f)
    q_f = np.zeros((B, sh.idx_heads, sh.idx_dim), dtype=np.float32)
    q_f[:, :, 0] = 1.0
    q_idx = W.f32_to_bf16_bits(q_f)
    w = np.ones((B, sh.idx_heads), dtype=np.float32)
    n_valid = np.array([N, N - 3], dtype=np.int32)
    ws = csa2.workspace(sh)
    idx = torch.full((B, K), -9, dtype=torch.int32, device="cuda")
    csa2.index_topk(sh, bf16(q_idx), f32(w), bf16(k_idx), i32(n_valid), K, idx, ws)
    got = idx.cpu().numpy()
    for b in range(B):
        r = oracle.layer_indices(oracle.to_f64(q_idx[b]), w[b].astype(np.float64), oracle.to_f64(k_idx[b]), None,
                                 int(n_valid[b]), topk=K, block=8, pool=0, hier=False)
        assert got[b].tolist() == r["idx"].tolist(), f"group {group} spread {spread} query {b}"
    assert_no_device_error(csa2, ws)


@pytest.mark.parametrize("case", ["outlier", "relu_off"])
def test_index_topk_pooled_wide_or_negative_scores(csa2, case):
    """Pooled scoring + Top-k when the 256 fixed bins below the top score hold fewer than
    k keys (one score 2**100 times the rest: the first pass is redone over [min, max]),
    and with ReLU off, where most scores are negative."""
    rng = np.random.default_rng(31)
    B, N, P, K = 3, 4096, 64, 256
    sh = _shape(batch=B, n_entries=N, pool_blocks=P, topk=K, relu=0 if case == "relu_off" else 1)
    k_idx = _int_keys(rng, (B, N, sh.idx_dim))
    if case == "outlier":
        big = W.f32_to_bf16_bits(np.array([2.0 ** 100], dtype=np.float32))[0]
        for b in range(B):
            k_idx[b, 1000 + 37 * b] = big                    # every dim 2**100: score ~2**100 times the rest
    q_idx = _int_keys(rng, (B, sh.idx_heads, sh.idx_dim))
    if case == "outlier":
        q_idx[:, :, :] = W.f32_to_bf16_bits(np.array([1.0], dtype=np.float32))[0]   # positive dot products
    w = rng.integers(1, 4, size=(B, sh.idx_heads)).astype(np.float32)
    n_valid = np.array([N, N - 11, 3000], dtype=np.int32)
    ws = csa2.workspace(sh)
    kb = torch.zeros((B, N // 8, sh.idx_dim), dtype=torch.bfloat16, device="cuda")
    csa2.block_keys(sh, bf16(k_idx), i32(n_valid), kb, ws, round_to_int=True)
    pool = torch.zeros((B, P), dtype=torch.int32, device="cuda")
    n_pool = torch.zeros(B, dtype=torch.int32, device="cuda")
    csa2.index_blocks(sh, bf16(q_idx), f32(w), kb, i32(n_valid), pool, n_pool, ws)
    idx = torch.full((B, K), -9, dtype=torch.int32, device="cuda")
    csa2.index_topk(sh, bf16(q_idx), f32(w), bf16(k_idx), i32(n_valid), K, idx, ws, pool=pool, n_pool=n_pool)
    got = idx.cpu().numpy()
    for b in range(B):
        keys = oracle.to_f64(k_idx[b])
        n = int(n_valid[b])
        kb_o = oracle.block_keys(keys, n, 8, True)
        r = oracle.layer_indices(oracle.to_f64(q_idx[b]), w[b].astype(np.float64), keys, kb_o, n, topk=K,
                                 block=8, pool=P, hier=True, relu=case != "relu_off")
        assert got[b].tolist() == r["idx"].tolist(), f"{case} query {b}"
    assert_no_device_error(csa2, ws)


# ------------------------------------------------------------------ bounded device waits

def test_bounded_wait_gives_up_and_reports_timeout(csa2):
    """A stage barrier that nothing completes (csa2_debug_wait_timeout leaves out the copy
    of every CTA's first tile): the waits give up after 20 us, the kernel returns, the
    error word says CSA2_ERR_TIMEOUT (bit 2), every write stayed inside the output, and
    the same workspace and stream then serve a normal call that matches the oracle."""
    sh = _shape(batch=4, n_entries=4096, pool_blocks=0)
    wl = W.make_workload(sh, [W.FULL], seed=3, cfg_id=61, n_valid=[4096, 4000, 700, 64])
    d = csa2.upload(wl)
    L = d["layers"][0]
    assert_no_device_error(csa2, d["ws"])
    idx = torch.full((sh.batch, sh.topk), -7, dtype=torch.int32, device="cuda")
    csa2.debug_wait_timeout(sh, L["q_idx"], L["w_idx"], d["k_idx"], d["n_valid"], sh.topk, idx, 20000, d["ws"])
    st, bits = csa2.read_device_error(d["ws"])
    assert st == -6 and bits & 4, (st, bits)          # CSA2_ERR_TIMEOUT
    # every CTA gave up on its first tile and offered no candidate
    assert np.all(idx.cpu().numpy() == -1)
    csa2.index_topk(sh, L["q_idx"], L["w_idx"], d["k_idx"], d["n_valid"], sh.topk, idx, d["ws"])
    ref = oracle.run_group(wl, want_attention=False)[0]["idx"]
    assert np.array_equal(idx.cpu().numpy(), ref)
    assert_no_device_error(csa2, d["ws"])
