"""The context-parallel helper kernels one by one (csa2_shard_slice,
csa2_shard_counts, csa2_concat_parts, csa2_merge_attn) against their stated
definitions, written out here with numpy on small cases."""
import math

import numpy as np
import pytest

from tests.gpu_helpers import f32, i32, lib_ready, need_gpu, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    need_gpu()
    return lib_ready()


def _slice_ref(ids, lo, hi, delta, ld_out):
    out = np.full((ids.shape[0], ld_out), -1, dtype=np.int32)
    n = np.zeros(ids.shape[0], dtype=np.int32)
    for b, row in enumerate(ids):
        kept = [int(i) + delta for i in row if i >= 0 and lo <= i < hi]
        n[b] = min(len(kept), ld_out)
        out[b, :n[b]] = kept[:ld_out]
    return out, n


@pytest.mark.parametrize("lo,hi,delta", [(0, 1000, 4096), (300, 700, -300), (-50, 200, 7)])
def test_shard_slice_keeps_the_range_in_order(csa2, lo, hi, delta):
    """The range's ids in their order, shifted and compacted; -1 pads are dropped even
    when the range starts below 0."""
    rng = np.random.default_rng(lo + 1000)
    B, ld = 5, 700                                   # 700 ids: several 256-id sweeps of the kernel
    ids = np.full((B, ld), -1, dtype=np.int32)
    for b in range(B):
        m = [ld, 500, 3, 0, 257][b]
        ids[b, :m] = rng.integers(0, 1000, size=m)
    out = torch.full((B, ld), -9, dtype=torch.int32, device="cuda")
    n_out = torch.zeros(B, dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    csa2.shard_slice(i32(ids), lo, hi, delta, out, ws, n_out=n_out)
    ref, n_ref = _slice_ref(ids, lo, hi, delta, ld)
    np.testing.assert_array_equal(out.cpu().numpy(), ref)
    np.testing.assert_array_equal(n_out.cpu().numpy(), n_ref)
    assert csa2.read_device_error(ws)[0] == 0


def test_shard_slice_reports_a_row_that_overflows(csa2):
    ids = i32(np.arange(40, dtype=np.int32).reshape(1, 40))
    out = torch.full((1, 16), -9, dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    csa2.shard_slice(ids, 0, 40, 0, out, ws)
    np.testing.assert_array_equal(out.cpu().numpy()[0], np.arange(16))   # the first 16, the rest dropped
    st, bits = csa2.read_device_error(ws)
    assert st != 0 and bits & 2                                            # bit 1: bad count


@pytest.mark.parametrize("div", [1, 8])
def test_shard_counts(csa2, div):
    n_valid = np.array([0, 1, 999, 1000, 1001, 1999, 2000, 2001, 5000], dtype=np.int32)
    e0, n_loc = 1000, 1000
    out = torch.full((len(n_valid),), -9, dtype=torch.int32, device="cuda")
    csa2.shard_counts(i32(n_valid), e0, n_loc, out, div=div)
    ref = [math.ceil(min(max(int(n) - e0, 0), n_loc) / div) for n in n_valid]
    assert out.cpu().numpy().tolist() == ref


def test_concat_parts(csa2):
    rng = np.random.default_rng(3)
    G, B, k = 3, 4, 5
    ids = rng.integers(-1, 100, size=(G, B, k)).astype(np.int32)
    sc = rng.standard_normal((G, B, k)).astype(np.float32)
    ids_out = torch.empty((B, G * k), dtype=torch.int32, device="cuda")
    sc_out = torch.empty((B, G * k), dtype=torch.float32, device="cuda")
    csa2.concat_parts(i32(ids), f32(sc), ids_out, sc_out)
    np.testing.assert_array_equal(ids_out.cpu().numpy(), ids.transpose(1, 0, 2).reshape(B, G * k))
    np.testing.assert_array_equal(sc_out.cpu().numpy(), sc.transpose(1, 0, 2).reshape(B, G * k))


def test_merge_attn_combines_partials_by_their_lse(csa2):
    """out = sum_g w_g out_g / sum_g w_g with w_g = exp(lse_g - max lse); parts with
    lse = -inf add nothing; a row with no key anywhere gives out 0 and lse -inf."""
    rng = np.random.default_rng(4)
    G, R, dv = 4, 6, 40
    out_p = rng.standard_normal((G, R, dv)).astype(np.float32)
    lse_p = (3 * rng.standard_normal((G, R))).astype(np.float32)
    lse_p[1, 2] = -np.inf            # one empty part
    lse_p[:, 5] = -np.inf            # a row with no key at all
    out = torch.full((R, dv), 7.0, dtype=torch.float32, device="cuda")
    lse = torch.zeros(R, dtype=torch.float32, device="cuda")
    csa2.merge_attn(f32(out_p), f32(lse_p), out, lse)
    o64, l64 = out_p.astype(np.float64), lse_p.astype(np.float64)
    ref_o, ref_l = np.zeros((R, dv)), np.full(R, -np.inf)
    for r in range(R):
        live = np.isfinite(l64[:, r])
        if not live.any():
            continue
        M = l64[live, r].max()
        w = np.exp(l64[live, r] - M)
        ref_o[r] = (w[:, None] * o64[live, r]).sum(0) / w.sum()
        ref_l[r] = M + np.log(w.sum())
    got_o, got_l = out.cpu().numpy(), lse.cpu().numpy()
    assert np.abs(got_o - ref_o).max() < 1e-5
    fin = np.isfinite(ref_l)
    assert np.abs(got_l[fin] - ref_l[fin]).max() < 1e-5
    assert np.all(np.isneginf(got_l[~fin])) and np.all(got_o[~fin] == 0)
