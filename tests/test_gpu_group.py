"""Layer-group parity (csa2_layer_group through the C ABI) on every named workload
and on ragged / edge-case groups, against the CPU oracle."""
import numpy as np
import pytest

import oracle
from oracle import FULL, REINDEX, REUSE, SWA
from sparse_attention_decode_index_gb300 import workloads as W
from tests.gpu_helpers import assert_no_device_error, compare_attention, lib_ready, need_gpu, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    need_gpu()
    return lib_ready()


def run_gpu(csa2, wl):
    d = csa2.upload(wl)
    sh = wl.shape
    if any(L.hier for L in wl.layers):
        csa2.block_keys(sh, d["k_idx"], d["n_valid"], d["kb"], d["ws"], round_to_int=bool(wl.round_block_keys))
    csa2.layer_group(sh, d["layers"], d["k_main"], d["v_main"], d["k_idx"], d["kb"], d["n_valid"], d["n_swa"],
                     d["ws"])
    torch.cuda.synchronize()
    return d


def check_group(csa2, wl, d, queries=None, atol=1e-2):
    qs = list(range(wl.shape.batch)) if queries is None else list(queries)
    ref = oracle.run_group(wl, queries=qs)
    worst = 0.0
    cur = None
    for li, L in enumerate(wl.layers):
        y, r = d["layers"][li], ref[li]
        if L.mode == SWA:
            pass
        elif L.mode != REUSE:
            got = y["idx_out"].cpu().numpy()[qs]
            assert np.array_equal(got, r["idx"]), f"layer {li} ({W.MODE_NAMES[L.mode]}): indices differ"
            cur = y["idx_out"]
        else:
            assert "idx_out" not in y or y.get("idx_out") is None
            assert np.array_equal(cur.cpu().numpy()[qs], r["idx"])
        e, _ = compare_attention(y["out"].cpu().numpy()[qs], y["lse"].cpu().numpy()[qs], r["out"], r["lse"],
                                 atol=atol)
        worst = max(worst, e)
    assert_no_device_error(csa2, d["ws"])
    return worst


@pytest.mark.parametrize("name", ["full_b8_8k", "enc_b32_32k", "reindex_b64_128k", "dec_b16_1m",
                                  "dec_b16_1m_hier", "enc_stack_b32_32k", "dec_b64_128k"])
def test_named_workload(csa2, name):
    """Every query of the named workload at full size, in the launch configuration the bench
    times (one csa2_layer_group call), against the oracle: indices bit-exact, outputs within 1e-2."""
    wl = W.named(name)
    d = run_gpu(csa2, wl)
    worst = check_group(csa2, wl, d)
    print(f"{name}: indices bit-exact, max-abs attention error {worst:.2e}")
    del d
    torch.cuda.empty_cache()


def _toy_margin_ok(wl, tol=1e-4):
    """Indices of the fp32 toy are compared only when no selection boundary is a near tie."""
    b = 0
    L = wl.layers[0]
    keys = oracle.to_f64(wl.k_idx[b])
    q, w = oracle.to_f64(L.q_idx[b]), oracle.to_f64(L.w_idx[b])
    n = int(wl.n_valid[b])
    kb = oracle.block_keys(keys, n, wl.shape.block, False)
    for s, k in ((oracle.indexer_scores(q, w, kb), wl.shape.pool_blocks),):
        ss = np.sort(s)[::-1]
        if len(ss) > k and ss[k - 1] - ss[k] < tol:
            return False
    r = oracle.layer_indices(q, w, keys, kb, n, topk=wl.shape.topk, block=wl.shape.block,
                             pool=wl.shape.pool_blocks, hier=True)
    ss = np.sort(r["scores"])[::-1]
    k = wl.shape.topk
    return not (len(ss) > k and ss[k - 1] - ss[k] < tol)


@pytest.mark.parametrize("seed", range(6))
def test_toy16(csa2, seed):
    wl = W.toy16(seed)
    if not _toy_margin_ok(wl):
        pytest.skip(f"seed {seed}: a selection boundary is within 1e-4 (fp32 vs fp64 scores)")
    d = run_gpu(csa2, wl)
    check_group(csa2, wl, d, atol=1e-4)


def test_golden_toy16_hand_on_gpu(csa2):
    """The hand-worked 16-token case (tests/golden/toy16_hand.json) through the GPU path."""
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "toy16_hand.json")) as f:
        g = json.load(f)
    keys = np.zeros((1, 16, 1), dtype=np.float32)
    keys[0, :12, 0] = g["keys"]
    sh = W.Shape(batch=1, n_entries=16, idx_heads=1, idx_dim=1, block=2, pool_blocks=4, topk=3, q_heads=1,
                 k_dim=1, v_dim=1, swa=4, dtype="f32")
    for rnd, pool_key, top_key in ((1, "pool_rounded", "top3_hier_rounded"),
                                   (0, "pool_unrounded", "top3_hier_unrounded")):
        ws = csa2.workspace(sh)
        k_dev = torch.from_numpy(keys).cuda()
        n_valid = torch.tensor([12], dtype=torch.int32, device="cuda")
        kb = torch.zeros((1, 8, 1), dtype=torch.float32, device="cuda")
        q = torch.ones((1, 1, 1), dtype=torch.float32, device="cuda")
        w = torch.ones((1, 1), dtype=torch.float32, device="cuda")
        csa2.block_keys(sh, k_dev, n_valid, kb, ws, round_to_int=bool(rnd))
        key = "block_keys_rounded" if rnd else "block_means"
        assert kb.cpu().numpy()[0, :6, 0].tolist() == g[key]
        pool = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
        npool = torch.zeros(1, dtype=torch.int32, device="cuda")
        csa2.index_blocks(sh, q, w, kb, n_valid, pool, npool, ws)
        assert pool.cpu().numpy()[0].tolist() == g[pool_key]
        scores = torch.zeros((1, 8), dtype=torch.float32, device="cuda")
        cand = torch.zeros((1, 8), dtype=torch.int32, device="cuda")
        ncand = torch.zeros(1, dtype=torch.int32, device="cuda")
        csa2.index_tokens(sh, q, w, k_dev, n_valid, scores, ws, pool=pool, n_pool=npool, cand_out=cand,
                          n_cand_out=ncand)
        if rnd:
            assert cand.cpu().numpy()[0].tolist() == g["candidates_rounded"]
            assert scores.cpu().numpy()[0].tolist() == g["candidate_scores_rounded"]
        idx = torch.zeros((1, 3), dtype=torch.int32, device="cuda")
        csa2.topk(sh, scores, 3, idx, ws, cand=cand, n_cand=ncand)
        assert idx.cpu().numpy()[0].tolist() == g[top_key]
    # flat selection
    scores = torch.zeros((1, 16), dtype=torch.float32, device="cuda")
    csa2.index_tokens(sh, q, w, k_dev, n_valid, scores, ws)
    idx = torch.zeros((1, 3), dtype=torch.int32, device="cuda")
    csa2.topk(sh, scores, 3, idx, ws, n_cand=n_valid)
    assert idx.cpu().numpy()[0].tolist() == g["top3_flat"]


def _small_group(modes, *, batch=6, n_entries=2048, pool=64, topk=512, swa=128, n_valid=None, n_swa=None,
                 seed=11, hier_full=0, **kw):
    sh = W.Shape(batch=batch, n_entries=n_entries, pool_blocks=pool, topk=topk, swa=swa, **kw)
    return W.make_workload(sh, modes, seed=seed, n_valid=n_valid, n_swa=n_swa, hier_full=hier_full)


def test_decoder_pattern_ragged(csa2):
    """Full + 3 Reuse + [Reindex + 3 Reuse] x 4 with ragged contexts (short, partial blocks, < K)."""
    n_valid = [2048, 2047, 1000, 513, 100, 0]
    n_swa = [128, 128, 64, 1, 0, 128]
    wl = _small_group(W.decoder_group_modes(), n_valid=n_valid, n_swa=n_swa, pool=32)
    d = run_gpu(csa2, wl)
    check_group(csa2, wl, d)


def test_hierarchical_full_layer_and_pool_covering_all_blocks(csa2):
    """A hierarchical Full layer whose pool covers every block equals the flat one."""
    wl_h = _small_group([FULL, REUSE], pool=256, hier_full=1, n_valid=[2048, 2041, 600, 9, 2048, 1])
    wl_f = _small_group([FULL, REUSE], pool=256, hier_full=0, n_valid=[2048, 2041, 600, 9, 2048, 1])
    dh, df = run_gpu(csa2, wl_h), run_gpu(csa2, wl_f)
    assert torch.equal(dh["layers"][0]["idx_out"], df["layers"][0]["idx_out"])
    check_group(csa2, wl_h, dh)


def test_all_equal_scores_pick_lowest_indices(csa2):
    wl = _small_group([FULL, REINDEX, REUSE], batch=2, pool=16)
    wl.k_idx[:] = W.f32_to_bf16_bits(np.ones(1, dtype=np.float32))[0]      # every key identical
    for L in wl.layers:
        if L.q_idx is not None:
            L.q_idx[:] = W.f32_to_bf16_bits(np.ones(1, dtype=np.float32))[0]
    wl.layers[1].hier = 1
    d = run_gpu(csa2, wl)
    idx0 = d["layers"][0]["idx_out"].cpu().numpy()
    assert np.array_equal(idx0, np.tile(np.arange(512), (2, 1)))
    # the hierarchical Reindex keeps the 16 lowest blocks, then the lowest 128 entries... of those
    idx1 = d["layers"][1]["idx_out"].cpu().numpy()
    assert np.array_equal(idx1[:, :128], np.tile(np.arange(128), (2, 1)))
    assert np.all(idx1[:, 128:] == -1)
    check_group(csa2, wl, d)


def test_small_topk_and_window_batch_one(csa2):
    wl = _small_group([FULL, REUSE, REINDEX], batch=1, n_entries=4096, topk=64, swa=16, pool=8,
                      n_valid=[3001])
    d = run_gpu(csa2, wl)
    check_group(csa2, wl, d)


def test_swa_layers_anywhere_in_a_group(csa2):
    """Pure sliding-window layers need no indices: first, between and after CSA2 layers."""
    wl = _small_group([SWA, FULL, SWA, REUSE, REINDEX, SWA], n_valid=[2048, 1500, 9, 0, 2048, 700],
                      n_swa=[128, 0, 5, 128, 1, 64], pool=32)
    d = run_gpu(csa2, wl)
    check_group(csa2, wl, d)


@pytest.mark.parametrize("modes", [[FULL, REINDEX, REUSE], [SWA, REINDEX, REUSE, FULL]])
def test_several_tokens_per_sequence_share_the_caches(csa2, modes):
    """A decoder replay: 2 sequences x 16 consecutive tokens, caches shared per sequence,
    each token with its own causal n_valid (ragged within the last blocks), its own
    sliding window and its own block summary keys."""
    wl = W.decoder_replay(2, 16, 8192, n_entries=2048, pool=64, modes=modes, seed=7)
    assert wl.k_main.shape[0] == 2 and wl.shape.batch == 32
    d = run_gpu(csa2, wl)
    check_group(csa2, wl, d)


def test_tokens_of_one_sequence_hand_case_on_gpu(csa2):
    """The oracle pin's hand case (two tokens of one sequence with different partial last
    blocks) through the GPU path: pools [0] / [1], indices [0] / [3]."""
    sh = W.Shape(batch=2, n_entries=6, idx_heads=1, idx_dim=1, block=2, pool_blocks=1, topk=1, q_heads=1,
                 k_dim=1, v_dim=1, swa=1, dtype="f32", tokens=2)
    one = np.ones((2, 1, 1), dtype=np.float32)
    layer = W.Layer(mode=REINDEX, hier=1, q=one, k_swa=one.copy(), v_swa=one.copy(), q_idx=one.copy(),
                    w_idx=np.ones((2, 1), dtype=np.float32))
    keys = np.array([1, 1, 0, 9, 5, 5], dtype=np.float32)[None, :, None]
    wl = W.Workload(name="tokens_hand", shape=sh, k_main=keys.copy(), v_main=keys.copy(), k_idx=keys,
                    n_valid=np.array([3, 4], dtype=np.int32), n_swa=np.array([0, 0], dtype=np.int32),
                    layers=[layer], round_block_keys=1)
    d = run_gpu(csa2, wl)
    assert d["layers"][0]["idx_out"].cpu().numpy().tolist() == [[0], [3]]
    assert d["layers"][0]["out"].cpu().numpy()[:, 0, 0].tolist() == [1.0, 9.0]
    check_group(csa2, wl, d, atol=1e-6)
