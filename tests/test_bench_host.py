"""Host-side logic of bench.py (CPU): the algorithmic byte count behind the
roofline, the query slicing of the CPU baseline, and the traffic records."""
import json
import os
import shutil

import numpy as np
import pytest

import bench
from sparse_attention_decode_index_gb300 import workloads as W


def test_algorithmic_bytes_of_the_headline_step_per_query():
    """One Reindex query at 128K context (32,768 entries, 4,096 blocks of 8, a pool of
    2,048 blocks): 4,096 block keys and 16,384 pooled token keys of 64 bf16, 512 selected
    plus 128 window rows of K (192 bf16) and V (128 bf16), Q (64 x 192 bf16) and the fp32
    output (64 x 128)."""
    wl = W.named("reindex_b64_128k", batch=2)
    per_query = {"indexer_blocks": 4096 * 128, "indexer_tokens": 16384 * 128, "selected_kv": 512 * 640,
                 "swa_kv": 128 * 640, "q": 64 * 192 * 2, "out": 64 * 128 * 4}
    ab = bench.algorithmic_bytes(wl)
    for key, v in per_query.items():
        assert ab[key] == 2 * v, key
    assert ab["total"] == 2 * sum(per_query.values())
    assert 64 * sum(per_query.values()) == 197_656_576          # the full batch of 64


def test_reuse_layers_read_the_selected_rows_again_but_count_once():
    """A Reuse layer attends the indices of the layer before it: its selected rows are
    counted with that layer, its own query, window and output separately."""
    wl = W.named("enc_b32_32k", batch=1)                    # Full + 5 Reuse
    ab = bench.algorithmic_bytes(wl)
    assert ab["selected_kv"] == 512 * 640
    assert ab["swa_kv"] == 6 * 128 * 640
    assert ab["q"] == 6 * 64 * 192 * 2 and ab["out"] == 6 * 64 * 128 * 4


def test_slice_queries_maps_tokens_to_their_sequence_caches():
    wl = W.decoder_replay(2, 3, 64, n_entries=16, pool=0, modes=[W.FULL, W.REUSE])
    assert wl.shape.tokens == 3 and wl.shape.batch == 6
    sub = bench.slice_queries(wl, [4, 1])                    # sequence 1 token 1, sequence 0 token 1
    assert sub.shape.batch == 2 and sub.shape.tokens == 1
    np.testing.assert_array_equal(sub.k_main, wl.k_main[[1, 0]])
    np.testing.assert_array_equal(sub.k_idx, wl.k_idx[[1, 0]])
    np.testing.assert_array_equal(sub.n_valid, wl.n_valid[[4, 1]])
    for L, Ls in zip(wl.layers, sub.layers):
        np.testing.assert_array_equal(Ls.q, L.q[[4, 1]])
        np.testing.assert_array_equal(Ls.k_swa, L.k_swa[[4, 1]])


def _copy_sources(tmp_path, monkeypatch):
    csrc = os.path.join(bench.ROOT, "sparse_attention_decode_index_gb300", "csrc")
    dst = tmp_path / "sparse_attention_decode_index_gb300" / "csrc"
    shutil.copytree(csrc, dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return dst


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    before = bench.kernel_source_hash("index_select_pooled")
    dst = _copy_sources(tmp_path, monkeypatch)
    assert bench.kernel_source_hash("index_select_pooled") == before
    p = dst / "fused.cu"
    text = p.read_text()
    p.write_text(text.replace("namespace csa2 {", "// a note\n\n/* and a\n   block */\nnamespace csa2 {   // x", 1))
    assert bench.kernel_source_hash("index_select_pooled") == before
    p.write_text(text.replace("constexpr int kStages = 5;", "constexpr int kStages = 4;", 1))
    assert bench.kernel_source_hash("index_select_pooled") != before


def test_traffic_record_is_used_only_while_the_sources_match(tmp_path, monkeypatch):
    wl = W.named("full_b8_8k", batch=1)
    _copy_sources(tmp_path, monkeypatch)
    (tmp_path / "profiles").mkdir()
    rec = {"dram_bytes_per_launch": 1234, "source_sha256_16": bench.kernel_source_hash("index_select_flat")}
    path = tmp_path / "profiles" / f"index_select_flat__{wl.name}.traffic.json"
    path.write_text(json.dumps(rec))
    assert bench.profiled_traffic(wl, "index_select_flat")[0] == 1234
    path.write_text(json.dumps({**rec, "source_sha256_16": "0" * 16}))
    value, why = bench.profiled_traffic(wl, "index_select_flat")
    assert value is None and "changed" in why
    path.unlink()
    assert bench.profiled_traffic(wl, "index_select_flat")[0] is None


@pytest.mark.parametrize("path", sorted(p for p in os.listdir(os.path.join(bench.ROOT, "profiles"))
                                        if p.endswith(".traffic.json")))
def test_committed_traffic_records_are_well_formed(path):
    kind, workload = path[:-len(".traffic.json")].split("__")
    assert kind in bench.KERNEL_SOURCES
    assert workload in W.WORKLOADS
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", path)))
    assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    assert len(rec["source_sha256_16"]) == 16
    assert "--clock-control none" in rec["command"]
