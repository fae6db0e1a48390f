"""csa2_layer_group_static: the layer group for callers that cannot allocate.

Some callers cannot provide a device workspace -- a plugin whose host
framework owns every device allocation, or a decode loop that must not call
cudaMalloc.  The static entry point runs on the library's own device scratch
instead.  This test calls it through the C ABI twice in a row and checks each
result against csa2_layer_group with a caller-provided workspace.  It lives in
a file of its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest

from sparse_attention_decode_index_gb300 import workloads as W
from tests.gpu_helpers import lib_ready, need_gpu, torch

pytestmark = pytest.mark.gpu


def _outputs(d):
    return [(y["out"].clone(), y["lse"].clone(), None if y.get("idx_out") is None else y["idx_out"].clone())
            for y in d["layers"]]


def test_static_scratch_layer_group_matches_workspace_version():
    need_gpu()
    csa2 = lib_ready()
    sh = W.Shape(batch=6, n_entries=4096, pool_blocks=128)
    wl = W.make_workload(sh, [W.FULL, W.REUSE, W.REINDEX, W.REUSE], seed=21, cfg_id=77,
                         n_valid=[4096, 4001, 700, 3, 4096, 2222], n_swa=[128, 128, 17, 0, 128, 64])
    d = csa2.upload(wl)
    csa2.block_keys(sh, d["k_idx"], d["n_valid"], d["kb"], d["ws"], round_to_int=True)
    args = (d["k_main"], d["v_main"], d["k_idx"], d["kb"], d["n_valid"], d["n_swa"])

    csa2.layer_group(sh, d["layers"], *args, d["ws"])
    torch.cuda.synchronize()
    want = _outputs(d)

    for _ in range(2):                       # two calls in a row on the shared scratch
        for y in d["layers"]:
            y["out"].fill_(float("nan"))
            y["lse"].fill_(float("nan"))
            if y.get("idx_out") is not None:
                y["idx_out"].fill_(-7)
        csa2.layer_group_static(sh, d["layers"], *args)
        torch.cuda.synchronize()
        got = _outputs(d)
        for (wo, wl_, wi), (go, gl, gi) in zip(want, got):
            if wi is not None:
                assert torch.equal(gi, wi), "indices differ from the workspace version"
            assert float((go - wo).abs().max()) <= 1e-2
            assert float((gl - wl_).abs().max()) <= 1e-2


def test_static_scratch_rejects_shapes_beyond_its_size():
    need_gpu()
    csa2 = lib_ready()
    sh = W.Shape(batch=16, n_entries=262144, pool_blocks=2048)      # needs ~42 MiB of scratch
    assert csa2.workspace_bytes(sh) > 32 << 20
    lib = csa2.lib()
    s = csa2.c_shape(sh)
    layers = (csa2.CLayer * 1)()
    fake = ctypes.c_void_p(0x7f0000000000)
    st = lib.csa2_layer_group_static(ctypes.byref(s), layers, 1, fake, fake, fake, fake, fake, fake, None)
    assert st == -3                          # CSA2_ERR_WORKSPACE, nothing enqueued
