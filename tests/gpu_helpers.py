"""Shared helpers for the GPU parity tests (imported only by tests)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from sparse_attention_decode_index_gb300 import build as _build  # noqa: E402

ATOL = 1e-2          # attention outputs: max-abs error bound against the fp64 oracle


def lib_ready():
    _build.build()
    from sparse_attention_decode_index_gb300 import csa2
    csa2.lib()
    return csa2


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def bf16(arr):
    """bf16 bit patterns (uint16 numpy) -> device bf16 tensor."""
    a = np.ascontiguousarray(arr)
    return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)


def i32(arr):
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.int32)).cuda()


def f32(arr):
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).cuda()


def assert_no_device_error(csa2, ws):
    st, detail = csa2.read_device_error(ws)
    assert st == 0, f"device error word set: status {st}, bits {detail:#x}"


def compare_attention(out_gpu, lse_gpu, out_ref, lse_ref, atol=ATOL):
    out_gpu = np.asarray(out_gpu, dtype=np.float64)
    err = np.abs(out_gpu - out_ref)
    fin = np.isfinite(lse_ref)
    lerr = np.abs(np.asarray(lse_gpu, dtype=np.float64)[fin] - lse_ref[fin]) if fin.any() else np.zeros(1)
    assert np.all(np.isneginf(np.asarray(lse_gpu)[~fin])), "lse must be -inf where no key is attended"
    assert err.max() <= atol, f"max-abs output error {err.max():.3e} > {atol}"
    assert lerr.max() <= atol, f"max-abs lse error {lerr.max():.3e} > {atol}"
    return float(err.max()), float(lerr.max())
