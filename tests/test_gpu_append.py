"""Decode-step cache maintenance on the GPU (csa2_kv_append, csa2_swa_append through
the C ABI) against the CPU oracle: caches, block summary keys and counters
bit for bit, and a layer group run on the maintained caches."""
import dataclasses

import numpy as np
import pytest

import oracle
from oracle import FULL, REINDEX, REUSE
from sparse_attention_decode_index_gb300 import workloads as W
from tests.gpu_helpers import assert_no_device_error, bf16, compare_attention, i32, lib_ready, need_gpu, torch

pytestmark = pytest.mark.gpu

BAD_COUNT = 2


@pytest.fixture(scope="module")
def csa2():
    need_gpu()
    return lib_ready()


def _bits(t):
    """Device bf16 tensor -> uint16 bit patterns."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _rows(rng, shape, d):
    return W.f32_to_bf16_bits((rng.standard_normal(shape) / np.sqrt(d)).astype(np.float32))


def _int_rows(rng, shape):
    return W.f32_to_bf16_bits(rng.integers(-4, 5, shape).astype(np.float32))


def test_kv_append_matches_oracle(csa2):
    rng = np.random.default_rng(21)
    sh = W.Shape(batch=7, n_entries=256, pool_blocks=8)
    B, N, nb = sh.batch, sh.n_entries, -(-sh.n_entries // sh.block)
    k_main = _rows(rng, (B, N, sh.k_dim), sh.k_dim)
    v_main = _rows(rng, (B, N, sh.v_dim), sh.v_dim)
    k_idx = _int_rows(rng, (B, N, sh.idx_dim))
    n_valid = np.array([0, 1, 7, 8, 100, 250, 255])
    d_k, d_v, d_x, d_nv = bf16(k_main), bf16(v_main), bf16(k_idx), i32(n_valid)
    d_kb = torch.zeros((B, nb, sh.idx_dim), dtype=torch.bfloat16, device="cuda")
    ws = csa2.workspace(sh)
    csa2.block_keys(sh, d_x, d_nv, d_kb, ws, round_to_int=True)
    kb = np.zeros((B, nb, sh.idx_dim))
    for b in range(B):
        kb[b, :-(-int(n_valid[b]) // sh.block)] = oracle.block_keys(oracle.to_f64(k_idx[b]), int(n_valid[b]),
                                                                    sh.block, True)
    state = (k_main, v_main, k_idx, kb, n_valid)
    for step, n_new in enumerate(([1, 3, 1, 8, 0, 2, 1], [8, 0, 2, 1, 5, 9, 0])):
        n_new = np.array(n_new)
        mx = int(n_new.max())
        k_new = _rows(rng, (B, mx, sh.k_dim), sh.k_dim)
        v_new = _rows(rng, (B, mx, sh.v_dim), sh.v_dim)
        x_new = _int_rows(rng, (B, mx, sh.idx_dim))
        csa2.kv_append(sh, i32(n_new), bf16(k_new), bf16(v_new), bf16(x_new), d_k, d_v, d_x, d_kb, d_nv, ws)
        *state, dropped = oracle.kv_append(*state, n_new, k_new, v_new, x_new, block=sh.block, round_to_int=True)
        st, bits = csa2.read_device_error(ws)
        if dropped.any():                                  # step 2: query 5 overflows (255 + ... > 256)
            assert bits & BAD_COUNT, f"step {step}: entries past the cache's end were not reported"
        else:
            assert st == 0, f"step {step}: unexpected device error {bits:#x}"
        k1, v1, x1, kb1, nv1 = state
        assert np.array_equal(d_nv.cpu().numpy(), nv1)
        assert np.array_equal(_bits(d_k), k1) and np.array_equal(_bits(d_v), v1) and np.array_equal(_bits(d_x), x1)
        got_kb = oracle.to_f64(_bits(d_kb))
        for b in range(B):
            nbv = -(-int(nv1[b]) // sh.block)
            assert np.array_equal(got_kb[b, :nbv], kb1[b, :nbv]), f"step {step} query {b}: block keys differ"
    # the incrementally kept keys equal the ones computed from scratch
    kb2 = torch.zeros_like(d_kb)
    csa2.block_keys(sh, d_x, d_nv, kb2, ws, round_to_int=True)
    assert torch.equal(kb2, d_kb)
    assert_no_device_error(csa2, ws)


def test_kv_append_without_block_keys_and_f32(csa2):
    rng = np.random.default_rng(4)
    sh = W.Shape(batch=3, n_entries=64, pool_blocks=0, dtype="f32")
    B, N = sh.batch, sh.n_entries
    k = rng.standard_normal((B, N, sh.k_dim)).astype(np.float32)
    v = rng.standard_normal((B, N, sh.v_dim)).astype(np.float32)
    x = rng.standard_normal((B, N, sh.idx_dim)).astype(np.float32)
    nv = np.array([0, 30, 63])
    n_new = np.array([2, 0, 1])
    kn = rng.standard_normal((B, 2, sh.k_dim)).astype(np.float32)
    vn = rng.standard_normal((B, 2, sh.v_dim)).astype(np.float32)
    xn = rng.standard_normal((B, 2, sh.idx_dim)).astype(np.float32)
    dev = [torch.from_numpy(a).cuda() for a in (k, v, x)]
    d_nv = i32(nv)
    ws = csa2.workspace(sh)
    csa2.kv_append(sh, i32(n_new), *(torch.from_numpy(a).cuda() for a in (kn, vn, xn)), *dev, None, d_nv, ws)
    k1, v1, x1, _, nv1, dropped = oracle.kv_append(k, v, x, None, nv, n_new, kn, vn, xn, block=sh.block,
                                                   round_to_int=False)
    assert not dropped.any()
    assert np.array_equal(d_nv.cpu().numpy(), nv1)
    for got, want in zip(dev, (k1, v1, x1)):
        assert np.array_equal(got.cpu().numpy(), want)
    assert_no_device_error(csa2, ws)


@pytest.mark.parametrize("dtype,steps", [("bf16", 131), ("f32", 20)])
def test_swa_append_rings_match_oracle(csa2, dtype, steps):
    """Three layers' rings, wrapping around the 128-row (bf16) window."""
    rng = np.random.default_rng(17)
    sh = W.Shape(batch=4, n_entries=64, pool_blocks=0, swa=128 if dtype == "bf16" else 16, dtype=dtype)
    B, Wn, L = sh.batch, sh.swa, 3
    f = dtype == "f32"

    def draw(shape, d):
        a = (rng.standard_normal(shape) / np.sqrt(d)).astype(np.float32)
        return a if f else W.f32_to_bf16_bits(a)

    def dev(a):
        return torch.from_numpy(a).cuda() if f else bf16(a)

    ks = [draw((B, Wn, sh.k_dim), sh.k_dim) for _ in range(L)]
    vs = [draw((B, Wn, sh.v_dim), sh.v_dim) for _ in range(L)]
    n_swa = np.array([0, 5, Wn - 1, Wn])
    head = n_swa % Wn
    d_ks, d_vs = [dev(a) for a in ks], [dev(a) for a in vs]
    d_head, d_n = i32(head), i32(n_swa)
    ws = csa2.workspace(sh)
    for _ in range(steps):
        kt = [draw((B, sh.k_dim), sh.k_dim) for _ in range(L)]
        vt = [draw((B, sh.v_dim), sh.v_dim) for _ in range(L)]
        csa2.swa_append(sh, [(dev(kt[l]), dev(vt[l]), d_ks[l], d_vs[l]) for l in range(L)], d_head, d_n, ws)
        for l in range(L):
            ks[l], vs[l], h1, n1 = oracle.swa_append(ks[l], vs[l], head, n_swa, kt[l], vt[l])
        head, n_swa = h1, n1
    assert np.array_equal(d_head.cpu().numpy(), head) and np.array_equal(d_n.cpu().numpy(), n_swa)
    for l in range(L):
        got_k = d_ks[l].cpu().numpy() if f else _bits(d_ks[l])
        got_v = d_vs[l].cpu().numpy() if f else _bits(d_vs[l])
        assert np.array_equal(got_k, ks[l]) and np.array_equal(got_v, vs[l])
    assert_no_device_error(csa2, ws)


def test_decode_steps_then_layer_group_match_oracle(csa2):
    """Three decode steps of cache maintenance (every layer's SWA ring, plus new
    compressed entries on some steps), then a Full (flat) + Reindex (hierarchical)
    + Reuse group on the maintained caches, against the oracle run on the caches
    the oracle maintained.  The hierarchical layer sees the incrementally kept
    block keys; the oracle computes them from scratch."""
    rng = np.random.default_rng(31)
    sh = W.Shape(batch=4, n_entries=2048, pool_blocks=128)
    n_valid0 = np.array([600, 1021, 1500, 2040])
    n_swa0 = np.array([128, 50, 127, 0])
    wl = W.make_workload(sh, [FULL, REINDEX, REUSE], seed=5, n_valid=n_valid0, n_swa=n_swa0)
    d = csa2.upload(wl)
    csa2.block_keys(sh, d["k_idx"], d["n_valid"], d["kb"], d["ws"], round_to_int=True)
    B, Wn = sh.batch, sh.swa
    head = n_swa0 % Wn
    d_head = i32(head)
    k_main, v_main, k_idx, n_valid, n_swa = wl.k_main, wl.v_main, wl.k_idx, n_valid0.copy(), n_swa0.copy()
    swa = [(L.k_swa, L.v_swa) for L in wl.layers]
    for step, n_new in enumerate(([1, 0, 4, 3], [0, 0, 0, 0], [2, 1, 9, 8])):
        slots, toks = [], []
        for l, L in enumerate(d["layers"]):
            kt = _rows(rng, (B, sh.k_dim), sh.k_dim)
            vt = _rows(rng, (B, sh.v_dim), sh.v_dim)
            toks.append((kt, vt))
            slots.append((bf16(kt), bf16(vt), L["k_swa"], L["v_swa"]))
        csa2.swa_append(sh, slots, d_head, d["n_swa"], d["ws"])
        for l in range(len(swa)):
            ks, vs, h1, n1 = oracle.swa_append(swa[l][0], swa[l][1], head, n_swa, *toks[l])
            swa[l] = (ks, vs)
        head, n_swa = h1, n1
        n_new = np.array(n_new)
        mx = max(1, int(n_new.max()))
        k_new = _rows(rng, (B, mx, sh.k_dim), sh.k_dim)
        v_new = _rows(rng, (B, mx, sh.v_dim), sh.v_dim)
        x_new = _int_rows(rng, (B, mx, sh.idx_dim))
        csa2.kv_append(sh, i32(n_new), bf16(k_new), bf16(v_new), bf16(x_new), d["k_main"], d["v_main"], d["k_idx"],
                       d["kb"], d["n_valid"], d["ws"])
        k_main, v_main, k_idx, _, n_valid, dropped = oracle.kv_append(
            k_main, v_main, k_idx, None, n_valid, n_new, k_new, v_new, x_new, block=sh.block, round_to_int=True)
    assert dropped.tolist() == [0, 0, 0, 3]                # query 3: 2040 + 3 + 8 > 2048
    st, bits = csa2.read_device_error(d["ws"])
    assert bits & BAD_COUNT
    live = dataclasses.replace(
        wl, k_main=k_main, v_main=v_main, k_idx=k_idx, n_valid=n_valid.astype(np.int32),
        n_swa=n_swa.astype(np.int32),
        layers=[dataclasses.replace(L, k_swa=swa[l][0], v_swa=swa[l][1]) for l, L in enumerate(wl.layers)])
    csa2.layer_group(sh, d["layers"], d["k_main"], d["v_main"], d["k_idx"], d["kb"], d["n_valid"], d["n_swa"],
                     d["ws"])
    torch.cuda.synchronize()
    ref = oracle.run_group(live)
    cur = None
    for l, L in enumerate(wl.layers):
        y, r = d["layers"][l], ref[l]
        if L.mode != REUSE:
            cur = y["idx_out"].cpu().numpy()
        assert np.array_equal(cur, r["idx"]), f"layer {l}: indices differ"
        compare_attention(y["out"].cpu().numpy(), y["lse"].cpu().numpy(), r["out"], r["lse"])
    assert_no_device_error(csa2, d["ws"])
