"""csa2_layer_group_static: the layer group for callers that cannot allocate.

Some callers cannot provide a device workspace -- a plugin whose host
framework owns every device allocation, or a decode loop that must not call
cudaMalloc.  The static entry point runs on the library's own device scratch
instead, and the cache-maintenance calls accept no workspace at all.  These
tests go through the C ABI the way such a caller would: the block summary keys
are built with no workspace, the group runs twice in a row on the static
scratch, and each result is checked against the CPU oracle and against
csa2_layer_group with a caller-provided workspace.  A device-side range
problem on this path is read back through csa2_read_static_device_error.
The file sorts last so that pytest collects it after every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
from sparse_attention_decode_index_gb300 import workloads as W
from tests.gpu_helpers import compare_attention, lib_ready, need_gpu, torch

pytestmark = pytest.mark.gpu


def _outputs(d):
    return [(y["out"].clone(), y["lse"].clone(), None if y.get("idx_out") is None else y["idx_out"].clone())
            for y in d["layers"]]


def _small_group():
    sh = W.Shape(batch=6, n_entries=4096, pool_blocks=128)
    wl = W.make_workload(sh, [W.FULL, W.REUSE, W.REINDEX, W.REUSE], seed=21, cfg_id=77,
                         n_valid=[4096, 4001, 700, 3, 4096, 2222], n_swa=[128, 128, 17, 0, 128, 64])
    return sh, wl


def test_static_scratch_layer_group_matches_oracle_and_workspace_version():
    need_gpu()
    csa2 = lib_ready()
    csa2.read_static_device_error()          # start from a clear static error word
    sh, wl = _small_group()
    d = csa2.upload(wl)
    # a caller without a workspace builds the block summary keys with ws = NULL
    csa2.block_keys(sh, d["k_idx"], d["n_valid"], d["kb"], None, round_to_int=True)
    args = (d["k_main"], d["v_main"], d["k_idx"], d["kb"], d["n_valid"], d["n_swa"])

    csa2.layer_group(sh, d["layers"], *args, d["ws"])
    torch.cuda.synchronize()
    want = _outputs(d)
    ref = oracle.run_group(wl)

    for _ in range(2):                       # two calls in a row on the shared scratch
        for y in d["layers"]:
            y["out"].fill_(float("nan"))
            y["lse"].fill_(float("nan"))
            if y.get("idx_out") is not None:
                y["idx_out"].fill_(-7)
        csa2.layer_group_static(sh, d["layers"], *args)
        torch.cuda.synchronize()
        got = _outputs(d)
        cur = None
        for li, ((wo, wl_, wi), (go, gl, gi)) in enumerate(zip(want, got)):
            r = ref[li]
            if wi is not None:
                assert torch.equal(gi, wi), "indices differ from the workspace version"
                assert np.array_equal(gi.cpu().numpy(), r["idx"]), f"layer {li}: indices differ from the oracle"
                cur = gi
            else:
                assert np.array_equal(cur.cpu().numpy(), r["idx"])
            assert float((go - wo).abs().max()) <= 1e-2
            assert float((gl - wl_).abs().max()) <= 1e-2
            compare_attention(go.cpu().numpy(), gl.cpu().numpy(), r["out"], r["lse"])
        st, bits = csa2.read_static_device_error()
        assert st == 0, f"static error word set: status {st}, bits {bits:#x}"


def test_static_scratch_reports_device_errors_through_its_own_reader():
    """A window count beyond W is clamped by the attention kernels and recorded in the
    static scratch's error word, which csa2_read_static_device_error returns and clears."""
    need_gpu()
    csa2 = lib_ready()
    csa2.read_static_device_error()
    sh, wl = _small_group()
    d = csa2.upload(wl)
    csa2.block_keys(sh, d["k_idx"], d["n_valid"], d["kb"], None, round_to_int=True)
    d["n_swa"][0] = sh.swa + 3
    csa2.layer_group_static(sh, d["layers"], d["k_main"], d["v_main"], d["k_idx"], d["kb"], d["n_valid"],
                            d["n_swa"])
    st, bits = csa2.read_static_device_error()
    assert st == -5 and bits & 2, (st, bits)  # CSA2_ERR_DEVICE_CHECK, bad-count bit
    assert csa2.read_static_device_error() == (0, 0)       # cleared by the read
    # the caller's own workspace saw nothing: the static path never touches it
    assert csa2.read_device_error(d["ws"]) == (0, 0)


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
