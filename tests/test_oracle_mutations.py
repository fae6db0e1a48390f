"""The oracle's pins catch plausible mistakes.

Each case plants one slip in the oracle (on the CPU, through monkeypatch) and
checks that at least one pin of ``test_oracle_pins`` fails with it.
"""
import numpy as np
import pytest

import oracle
import oracle.csa2 as C
from tests import test_oracle_pins as P

PINS = [P.test_golden_toy16_hand, P.test_indexer_scores_match_integer_loops,
        P.test_block_keys_rounding_half_even_and_partial_block,
        P.test_topk_matches_heap_selection_with_ties, P.test_topk_special_cases,
        P.test_hierarchical_equals_flat_when_pool_covers_every_block,
        P.test_reuse_layers_return_the_indexing_layers_indices,
        P.test_attention_closed_forms, P.test_toy16_structure,
        lambda: P.test_sparse_equals_dense_causal_attention_naive(24, 8, 16),
        P.test_kv_append_in_steps_equals_the_cache_written_at_once,
        P.test_kv_append_touches_only_the_blocks_of_the_new_positions,
        P.test_swa_ring_holds_the_last_w_tokens,
        P.test_block_keys_stored_as_bf16_round_the_mean_to_nearest_even,
        P.test_tokens_of_one_sequence_see_their_own_partial_last_block]


def _topk_highest_id_wins(scores, ids, k):
    scores = np.where(np.isnan(scores), -np.inf, scores)
    order = np.lexsort((-ids, -scores))
    chosen = np.sort(ids[order[:min(k, len(ids))]])
    out = np.full(k, -1, dtype=np.int64)
    out[:len(chosen)] = chosen
    return out


def _scores_without_relu(q_idx, w, keys, relu=True):
    return (keys @ q_idx.T) @ w


def _scores_without_weights(q_idx, w, keys, relu=True):
    d = keys @ q_idx.T
    return (np.maximum(d, 0.0) if relu else d).sum(axis=1)


def _block_keys_half_up(keys, n_valid, block, round_to_int, store_bf16=False):
    nb = -(-n_valid // block)
    out = np.zeros((nb, keys.shape[1]))
    for j in range(nb):
        rows = keys[j * block: min((j + 1) * block, n_valid)]
        m = rows.sum(axis=0) / rows.shape[0]
        out[j] = np.floor(m + 0.5) if round_to_int else m
    return out


def _attention_without_swa(q, k_main, v_main, idx, k_swa, v_swa, n_swa, scale):
    sel = idx[idx >= 0]
    return C.attend(q, k_main[sel], v_main[sel], scale)


def _attend_without_scale(q, k_rows, v_rows, scale):
    return _orig_attend(q, k_rows, v_rows, 1.0)


def _pooled_entries_off_by_one(pool, n_valid, block):
    ent = (pool[:, None] * block + 1 + np.arange(block)[None, :]).reshape(-1)
    return ent[ent < n_valid]


def _pool_unsorted(q_idx, w, kb, n_blocks, pool, relu=True):
    s = C.indexer_scores(q_idx, w, kb[:n_blocks], relu)
    order = np.lexsort((np.arange(n_blocks), -s))
    return order[:min(pool, n_blocks)]


def _block_keys_bf16_truncated(keys, n_valid, block, round_to_int, store_bf16=False):
    nb = -(-n_valid // block)
    out = np.zeros((nb, keys.shape[1]))
    for j in range(nb):
        rows = keys[j * block: min((j + 1) * block, n_valid)]
        m = rows.sum(axis=0) / rows.shape[0]
        if round_to_int:
            m = np.rint(m)
        elif store_bf16:
            mm, e = np.frexp(m)
            m = np.ldexp(np.trunc(mm * 256.0), e - 8)
        out[j] = m
    return out


def _block_keys_bf16_not_rounded(keys, n_valid, block, round_to_int, store_bf16=False):
    return _orig_block_keys(keys, n_valid, block, round_to_int, store_bf16=False)


def _block_keys_whole_cache(keys, n_valid, block, round_to_int, store_bf16=False):
    # a token's summary keys taken over its sequence's whole cache, not its own valid prefix
    return _orig_block_keys(keys, keys.shape[0], block, round_to_int, store_bf16=store_bf16)


_orig_block_keys = C.block_keys
_orig_attend = C.attend
_orig_kv_append = C.kv_append
_orig_swa_append = C.swa_append


def _kv_append_one_slot_late(k_main, v_main, k_idx, kb, n_valid, *rest, **kw):
    return _orig_kv_append(k_main, v_main, k_idx, kb, np.asarray(n_valid) + 1, *rest, **kw)


def _kv_append_stale_last_block(k_main, v_main, k_idx, kb, n_valid, n_new, k_new, v_new, kidx_new, *, block,
                                round_to_int, store_bf16=True):
    # recomputes only the blocks that were already valid before the append
    k1, v1, x1, kb1, nv1, dr = _orig_kv_append(k_main, v_main, k_idx, None, n_valid, n_new, k_new, v_new, kidx_new,
                                               block=block, round_to_int=round_to_int, store_bf16=store_bf16)
    if kb is not None:
        kb1 = np.array(kb, dtype=np.float64)
        for b in range(len(nv1)):
            nv0 = int(n_valid[b])
            keys = C.block_keys(C.to_f64(x1[b]), int(nv1[b]), block, round_to_int, store_bf16=store_bf16)
            for j in range(nv0 // block, -(-nv0 // block)):
                kb1[b, j] = keys[j]
    return k1, v1, x1, kb1, nv1, dr


def _swa_append_head_stuck(k_swa, v_swa, head, n_swa, k_tok, v_tok):
    k1, v1, _, n1 = _orig_swa_append(k_swa, v_swa, head, n_swa, k_tok, v_tok)
    return k1, v1, np.array(head), n1


MUTATIONS = {
    "tie-break keeps the highest id": ("select_topk", _topk_highest_id_wins),
    "ReLU dropped": ("indexer_scores", _scores_without_relu),
    "head weights dropped": ("indexer_scores", _scores_without_weights),
    "block keys rounded half up": ("block_keys", _block_keys_half_up),
    "SWA rows dropped": ("sparse_attention", _attention_without_swa),
    "softmax scale dropped": ("attend", _attend_without_scale),
    "pooled entries shifted by one": ("pooled_entries", _pooled_entries_off_by_one),
    "pool left in score order": ("pool_blocks", _pool_unsorted),
    "appended entries land one slot late": ("kv_append", _kv_append_one_slot_late),
    "summary key of a newly opened block not computed": ("kv_append", _kv_append_stale_last_block),
    "SWA ring head never advances": ("swa_append", _swa_append_head_stuck),
    "bf16 block means truncated instead of rounded": ("block_keys", _block_keys_bf16_truncated),
    "bf16 block means stored unrounded": ("block_keys", _block_keys_bf16_not_rounded),
    "a token's block keys taken over the whole cache": ("block_keys", _block_keys_whole_cache),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_fails_a_pin(name, monkeypatch):
    fn, bad = MUTATIONS[name]
    monkeypatch.setattr(C, fn, bad)
    monkeypatch.setattr(oracle, fn, bad)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed.append(getattr(pin, "__name__", "pin"))
    assert failed, f"no pin caught: {name}"
