"""C ABI checks that need no GPU: the library builds, loads and exports every
function declared in include/csa2.h, and host-side validation rejects bad
arguments with the documented status before anything is enqueued (the fake
pointers below are never dereferenced)."""
import ctypes
import os
import re

import pytest

from sparse_attention_decode_index_gb300 import build as B
from sparse_attention_decode_index_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa2.h")

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, -1, -2, -3


@pytest.fixture(scope="module")
def csa2():
    B.build()
    from sparse_attention_decode_index_gb300 import csa2 as m
    m.lib()
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_\w+)\s*\(", text)))


def test_header_declares_the_planned_entry_points():
    names = declared_functions()
    for n in ("csa2_index_blocks", "csa2_index_tokens", "csa2_topk", "csa2_sparse_attn", "csa2_layer_group",
              "csa2_block_keys", "csa2_workspace_bytes", "csa2_status_str", "csa2_read_device_error",
              "csa2_kv_append", "csa2_swa_append"):
        assert n in names


def test_library_exports_every_declared_function(csa2):
    lib = csa2.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(csa2.exported_symbols())


def _shape(**kw):
    base = dict(batch=4, n_entries=4096, pool_blocks=64)
    base.update(kw)
    return W.Shape(**base)


FAKE = 0x7f0000000000           # 256-byte aligned, never dereferenced
MIS = FAKE + 8                   # not 16-byte aligned


def test_workspace_bytes_and_shape_validation(csa2):
    lib = csa2.lib()
    good = csa2.c_shape(_shape())
    n = lib.csa2_workspace_bytes(ctypes.byref(good))
    assert n > 4 * 4096 * 8 and n % 256 == 0
    for bad in (dict(batch=0), dict(topk=0), dict(block=0), dict(dtype=7), dict(relu=2), dict(topk=1000, swa=100),
                dict(idx_heads=65), dict(pool_blocks=9000), dict(swa=-1)):
        kw = dict(_shape().__dict__)
        kw.update(bad)
        s = csa2.CShape(*[(1 if k == "dtype" and v == "bf16" else v) if not isinstance(v, str) else 0
                          for k, v in kw.items()])
        assert lib.csa2_workspace_bytes(ctypes.byref(s)) == 0, bad
    assert lib.csa2_workspace_bytes(None) == 0


def test_entry_points_reject_bad_arguments_before_launch(csa2):
    lib = csa2.lib()
    sh = _shape()
    s = csa2.c_shape(sh)
    wsb = lib.csa2_workspace_bytes(ctypes.byref(s))
    # null pointers
    assert lib.csa2_sparse_attn(ctypes.byref(s), None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, wsb,
                                None) == INVALID
    assert lib.csa2_index_tokens(ctypes.byref(s), FAKE, FAKE, None, FAKE, None, None, FAKE, None, None, FAKE, wsb,
                                 None) == INVALID
    assert lib.csa2_topk(ctypes.byref(s), None, 100, None, None, 10, FAKE, None, FAKE, wsb, None) == INVALID
    assert lib.csa2_block_keys(ctypes.byref(s), FAKE, None, 1, FAKE, FAKE, wsb, None) == INVALID
    # misaligned bulk-copied arrays on the fast path
    assert lib.csa2_sparse_attn(ctypes.byref(s), MIS, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, wsb,
                                None) == INVALID
    assert lib.csa2_index_tokens(ctypes.byref(s), FAKE, FAKE, MIS, FAKE, None, None, FAKE, None, None, FAKE, wsb,
                                 None) == INVALID
    # workspace too small / misaligned / missing
    assert lib.csa2_sparse_attn(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE,
                                wsb - 1, None) == WORKSPACE
    assert lib.csa2_topk(ctypes.byref(s), FAKE, 100, None, None, 10, FAKE, None, FAKE + 16, wsb, None) == WORKSPACE
    assert lib.csa2_index_blocks(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, wsb, None) == WORKSPACE
    # hierarchical stage without a pool
    s0 = csa2.c_shape(_shape(pool_blocks=0))
    wsb0 = lib.csa2_workspace_bytes(ctypes.byref(s0))
    assert lib.csa2_index_blocks(ctypes.byref(s0), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, wsb0,
                                 None) == INVALID
    # pooled token scoring needs cand_out and n_cand_out
    assert lib.csa2_index_tokens(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, wsb,
                                 None) == INVALID
    # Top-k larger than a chunk, and merges that would not shrink the list
    assert lib.csa2_topk(ctypes.byref(s), FAKE, 100, None, None, 20000, FAKE, None, FAKE, wsb, None) == UNSUPPORTED
    assert lib.csa2_topk(ctypes.byref(s), FAKE, 40000, None, None, 9000, FAKE, None, FAKE, wsb, None) == UNSUPPORTED


def test_append_entry_points_reject_bad_arguments_before_launch(csa2):
    lib = csa2.lib()
    s = csa2.c_shape(_shape())
    wsb = lib.csa2_workspace_bytes(ctypes.byref(s))
    ok_args = [FAKE] * 9          # n_new, k_new, v_new, kidx_new, k_main, v_main, k_idx, kb, n_valid

    def kv(max_new=1, args=None, rnd=1, ws=FAKE, bytes_=wsb):
        a = ok_args if args is None else args
        return lib.csa2_kv_append(ctypes.byref(s), max_new, *a, rnd, ws, bytes_, None)

    assert kv(max_new=-1) == INVALID                         # negative row count
    assert kv(max_new=10 ** 9) == INVALID                    # more rows than the cache holds
    assert kv(args=[None] + ok_args[1:]) == INVALID           # n_new missing
    assert kv(args=ok_args[:1] + [None] + ok_args[2:]) == INVALID   # k_new missing while max_new > 0
    assert kv(args=ok_args[:8] + [None]) == INVALID           # n_valid missing
    assert kv(rnd=2) == INVALID
    assert kv(bytes_=wsb - 1) == WORKSPACE
    assert kv(ws=FAKE + 16) == WORKSPACE                      # misaligned workspace
    slot = csa2.CSwaSlot(FAKE, FAKE, FAKE, FAKE)
    slots = (csa2.CSwaSlot * 2)(slot, slot)
    sp = ctypes.cast(slots, ctypes.c_void_p)

    def swa(shape_, sl=sp, n=2, head=FAKE, n_swa=FAKE, bytes_=None):
        b_ = lib.csa2_workspace_bytes(ctypes.byref(shape_)) if bytes_ is None else bytes_
        return lib.csa2_swa_append(ctypes.byref(shape_), sl, n, head, n_swa, FAKE, b_, None)

    assert swa(csa2.c_shape(_shape(swa=0))) == INVALID       # no window
    assert swa(s, n=0) == INVALID
    assert swa(s, n=65) == INVALID                            # more layers than one call takes
    assert swa(s, sl=None) == INVALID
    assert swa(s, head=None) == INVALID
    assert swa(s, bytes_=wsb - 1) == WORKSPACE
    bad = (csa2.CSwaSlot * 2)(slot, csa2.CSwaSlot(FAKE, None, FAKE, FAKE))
    assert swa(s, sl=ctypes.cast(bad, ctypes.c_void_p)) == INVALID


def test_tokens_per_sequence_rules(csa2):
    lib = csa2.lib()
    bad = csa2.c_shape(_shape(batch=6, tokens=4))                  # 6 queries are not whole sequences of 4
    assert lib.csa2_workspace_bytes(ctypes.byref(bad)) == 0
    s = csa2.c_shape(_shape(batch=8, tokens=4))
    wsb = lib.csa2_workspace_bytes(ctypes.byref(s))
    assert wsb > 0
    UNSUP = -2
    assert lib.csa2_kv_append(ctypes.byref(s), 1, *([FAKE] * 9), 1, FAKE, wsb, None) == UNSUP
    slot = (csa2.CSwaSlot * 1)(csa2.CSwaSlot(FAKE, FAKE, FAKE, FAKE))
    assert lib.csa2_swa_append(ctypes.byref(s), ctypes.cast(slot, ctypes.c_void_p), 1, FAKE, FAKE, FAKE, wsb,
                               None) == UNSUP


def _layers(csa2, modes, hier=None):
    arr = (csa2.CLayer * len(modes))()
    for i, m in enumerate(modes):
        arr[i] = csa2.CLayer(m, (hier or [0] * len(modes))[i], FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None)
    return arr


def test_layer_group_mode_rules(csa2):
    lib = csa2.lib()
    s = csa2.c_shape(_shape())
    wsb = lib.csa2_workspace_bytes(ctypes.byref(s))

    def call(modes, hier=None, kb=FAKE, n=None):
        ls = _layers(csa2, modes, hier)
        return lib.csa2_layer_group(ctypes.byref(s), ls, len(modes) if n is None else n, FAKE, FAKE, FAKE, kb,
                                    FAKE, FAKE, FAKE, wsb, None)

    assert call([W.REUSE, W.FULL]) == INVALID                 # Reuse needs an earlier indexing layer
    assert call([W.FULL, 7]) == INVALID                       # unknown mode
    assert call([W.REINDEX], hier=[1], kb=None) == INVALID    # hierarchical without block keys
    assert call([W.FULL], n=0) == INVALID
    ls = _layers(csa2, [W.FULL, W.REUSE])
    ls[1].q = MIS                                             # misaligned query of a later layer
    assert lib.csa2_layer_group(ctypes.byref(s), ls, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, wsb,
                                None) == INVALID
    ls = _layers(csa2, [W.FULL])
    ls[0].w_idx = None                                        # indexing layer without weights
    assert lib.csa2_layer_group(ctypes.byref(s), ls, 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, wsb,
                                None) == INVALID


def test_status_strings_and_fast_path_selection(csa2):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert csa2.status_str(code)
    assert csa2.fast_path(_shape()) == (True, True)
    assert csa2.fast_path(W.toy16().shape) == (False, False)
    assert csa2.fast_path(_shape(idx_heads=4)) == (False, True)
    assert csa2.fast_path(_shape(topk=1000, swa=24)) == (True, True)     # 8 CTAs of 128 slots
