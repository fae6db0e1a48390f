"""Seeded synthetic CSA2 decode workloads.

This module only draws random tensors with the shapes and value
distributions of the workloads; it contains none of the method's
arithmetic (no scoring, selection, block summaries or attention).  Both the
CPU oracle and the CUDA path consume what it produces, so neither side ever
derives an input from the other.

bf16 tensors are returned as their raw 16-bit patterns (numpy ``uint16``),
obtained from float32 draws by round-to-nearest-even; fp32 tensors (the toy
workload) are returned as ``float32``.

Workloads (sizes from the DeepSeek-V4.1-Flash architecture page,
"CSA2 with cross-layer reuse" and its bullet list: Top-512 main-KV entries
plus a 128-token SWA window, blocks of 8, a pool of at most 2,048 blocks):

* ``toy16`` -- the page's 16-token illustration ("How Full, Reuse and
  Reindex pick tokens"): query at position 15, one compressed entry per
  token, Top-3, SWA window 4, blocks of 2, a 4-block pool, Full mode.
  4 query heads of dim 16, one shared KV head, 2 indexer heads of dim 8,
  fp32 N(0,1) values.
* ``full_b8_8k`` -- one Full layer, batch 8, 8,192 tokens at ratio 4
  (2,048 entries), flat indexer.
* ``enc_b32_32k`` -- encoder group Full + 5 Reuse, batch 32, 32,768 tokens at
  ratio 4 (8,192 entries).
* ``reindex_b64_128k`` -- one hierarchical Reindex layer, batch 64,
  131,072 tokens at ratio 4 (32,768 entries = 4,096 blocks of 8), pool of
  2,048 blocks.
* ``dec_b16_1m`` -- decoder group Full + 3 Reuse + [Reindex + 3 Reuse] x 4,
  batch 16, 1,048,576 tokens at ratio 4 (262,144 entries).
* ``dec_b16_1m_hier`` -- ``dec_b16_1m`` with its Full layer hierarchical too
  (block scoring over 32,768 blocks and a pool of 2,048 instead of the flat
  scan of 262,144 entries).
* ``enc_stack_b32_32k`` -- the whole 20-layer encoder stack SWA, SWA,
  [Full + 5 Reuse] x 3 at the shapes of ``enc_b32_32k`` (pure SWA layers attend
  their window only).
* ``dec_b64_128k`` -- the decoder group of ``dec_b16_1m`` at the context and
  batch of ``reindex_b64_128k`` (batch 64, 32,768 entries, pool of 2,048).
* ``replay_t128_128k`` -- one sequence's last 128 prompt tokens through the
  decoder group at 128K context, caches shared by the tokens.

Value recipe: main and SWA keys N(0,1)/sqrt(k_dim), values
N(0,1)/sqrt(v_dim), queries N(0,1), all rounded to bf16; indexer queries
and keys are bf16 integers uniform on {-4..4}; indexer head weights are
fp32 integers uniform on {1,2,3}.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import List, Optional

import numpy as np

FULL, REINDEX, REUSE, SWA = 0, 1, 2, 3
MODE_NAMES = {FULL: "full", REINDEX: "reindex", REUSE: "reuse", SWA: "swa"}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    u = u + (((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF))
    return (u >> np.uint32(16)).astype(np.uint16)


@dataclasses.dataclass
class Shape:
    batch: int
    n_entries: int        # capacity of the main-KV / indexer-key caches per sequence
    idx_heads: int = 8
    idx_dim: int = 64
    block: int = 8
    pool_blocks: int = 2048
    topk: int = 512
    q_heads: int = 64
    k_dim: int = 192
    v_dim: int = 128
    swa: int = 128
    scale: float = 0.0    # 0 -> 1/sqrt(k_dim)
    relu: int = 1
    dtype: str = "bf16"   # "bf16" or "f32"
    tokens: int = 1       # query tokens per sequence: the caches are [batch / tokens, n_entries, ...]

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale > 0 else 1.0 / float(np.sqrt(self.k_dim))


@dataclasses.dataclass
class Layer:
    mode: int
    hier: int                        # 1: hierarchical block pool before token scoring
    q: np.ndarray                    # [B, H, k_dim]
    k_swa: np.ndarray                # [B, W, k_dim]
    v_swa: np.ndarray                # [B, W, v_dim]
    q_idx: Optional[np.ndarray] = None   # [B, HI, dI]  (Full / Reindex)
    w_idx: Optional[np.ndarray] = None   # [B, HI] float32


@dataclasses.dataclass
class Workload:
    name: str
    shape: Shape
    k_main: np.ndarray               # [B, N, k_dim]
    v_main: np.ndarray               # [B, N, v_dim]
    k_idx: np.ndarray                # [B, N, dI]
    n_valid: np.ndarray              # [B] int32: valid compressed entries per query
    n_swa: np.ndarray                # [B] int32: valid SWA rows (oldest first)
    layers: List[Layer]
    round_block_keys: int = 1        # block summary keys rounded to integers
    note: str = ""


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(k) for k in key]))


_CHUNK = 1 << 21                     # values per independently seeded chunk
_THREADS = max(1, min(16, os.cpu_count() or 1))
_INT_BF16 = None


def _int_table():
    global _INT_BF16
    if _INT_BF16 is None:
        _INT_BF16 = f32_to_bf16_bits(np.arange(-4, 5, dtype=np.float32))
    return _INT_BF16


def _draw(shape, key, kind: str, div: float = 1.0, bf16: bool = True) -> np.ndarray:
    """Draw a tensor in fixed chunks, chunk c from the stream (*key, c).

    ``kind``: "normal" (N(0,1)/div) or "int" (uniform integers on {-4..4}).
    The result does not depend on the number of threads used.
    """
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16 if bf16 else np.float32)
    scale = np.float32(1.0 / div)

    def work(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        rng = _rng(*key, c)
        if kind == "int":
            code = rng.integers(0, 9, size=hi - lo, dtype=np.int8)
            out[lo:hi] = _int_table()[code] if bf16 else (code.astype(np.float32) - 4)
            return
        x = rng.standard_normal(size=hi - lo, dtype=np.float32)
        if div != 1.0:
            x *= scale
        out[lo:hi] = f32_to_bf16_bits(x) if bf16 else x

    chunks = range(-(-n // _CHUNK))
    if len(chunks) > 1 and _THREADS > 1:
        with ThreadPoolExecutor(_THREADS) as ex:
            list(ex.map(work, chunks))
    else:
        for c in chunks:
            work(c)
    return out.reshape(shape)


def _weights(rng, shape):
    return rng.integers(1, 4, size=shape, dtype=np.int32).astype(np.float32)


# mode patterns ---------------------------------------------------------------

def encoder_group_modes(n_reuse: int = 5) -> List[int]:
    """One encoder group: Full followed by ``n_reuse`` Reuse layers."""
    return [FULL] + [REUSE] * n_reuse


def encoder_stack_modes() -> List[int]:
    """Encoder stack of the architecture figure: SWA, SWA, then [Full + 5 Reuse] x 3 (20 layers)."""
    return [SWA, SWA] + encoder_group_modes(5) * 3


def decoder_group_modes() -> List[int]:
    """Decoder stack: Full + 3 Reuse, then [Reindex + 3 Reuse] x 4 (20 layers)."""
    return [FULL] + [REUSE] * 3 + ([REINDEX] + [REUSE] * 3) * 4


def make_workload(shape: Shape, modes: List[int], *, seed: int = 0, cfg_id: int = 99,
                  n_valid=None, n_swa=None, hier_full: int = 0, hier_reindex: int = 1,
                  int_indexer: bool = True, name: str = "custom",
                  round_block_keys: int = 1) -> Workload:
    """Draw every tensor of a layer group.

    ``seed`` and ``cfg_id`` select the stream; tensor ``t`` of layer ``l`` uses
    the sub-stream (seed, cfg_id, t, l).  ``n_valid``/``n_swa`` default to
    the full capacity; pass arrays (or callables of the rng) for ragged cases.
    """
    B, N = shape.batch, shape.n_entries
    S = B // max(1, shape.tokens)     # cache sequences
    f32 = shape.dtype == "f32"

    def kv(key, shp, d):
        return _draw(shp, key, "normal", 1.0 if f32 else float(np.sqrt(d)), bf16=not f32)

    def q_of(key, shp):
        return _draw(shp, key, "normal", 1.0, bf16=not f32)

    def idxv(key, shp):
        if f32 or not int_indexer:
            return _draw(shp, key, "normal", 1.0, bf16=not f32)
        return _draw(shp, key, "int")

    k_main = kv((seed, cfg_id, 1), (S, N, shape.k_dim), shape.k_dim)
    v_main = kv((seed, cfg_id, 2), (S, N, shape.v_dim), shape.v_dim)
    k_idx = idxv((seed, cfg_id, 3), (S, N, shape.idx_dim))
    if n_valid is None:
        n_valid = np.full(B, N, dtype=np.int32)
    if n_swa is None:
        n_swa = np.full(B, shape.swa, dtype=np.int32)
    layers = []
    for l, mode in enumerate(modes):
        q = q_of((seed, cfg_id, 10, l), (B, shape.q_heads, shape.k_dim))
        k_swa = kv((seed, cfg_id, 11, l), (B, shape.swa, shape.k_dim), shape.k_dim)
        v_swa = kv((seed, cfg_id, 12, l), (B, shape.swa, shape.v_dim), shape.v_dim)
        q_idx = w = None
        if mode in (FULL, REINDEX):
            q_idx = idxv((seed, cfg_id, 13, l), (B, shape.idx_heads, shape.idx_dim))
            if f32:
                w = np.ones((B, shape.idx_heads), dtype=np.float32)
            else:
                w = _weights(_rng(seed, cfg_id, 14, l), (B, shape.idx_heads))
        hier = hier_full if mode == FULL else (hier_reindex if mode == REINDEX else 0)
        if shape.pool_blocks <= 0:
            hier = 0
        layers.append(Layer(mode=mode, hier=hier, q=q, k_swa=k_swa, v_swa=v_swa,
                            q_idx=q_idx, w_idx=w))
    return Workload(name=name, shape=shape, k_main=k_main, v_main=v_main, k_idx=k_idx,
                    n_valid=np.asarray(n_valid, dtype=np.int32),
                    n_swa=np.asarray(n_swa, dtype=np.int32), layers=layers,
                    round_block_keys=round_block_keys)


def decoder_replay(sequences: int, tokens: int, context: int, *, n_entries: int, pool: int, modes: List[int],
                   seed: int = 0, cfg_id: int = 6, ratio: int = 4, name: str = "replay") -> Workload:
    """The last ``tokens`` prompt tokens of each sequence run through a decoder
    group together (architecture page, "Asymmetric encoder-decoder": a
    128-token decoder replay).  Token t of a sequence sits at position
    p = context - tokens + t.  It sees the compressed entries that end at or
    before p, (p + 1) // ratio of them, and an SWA window of its own last
    min(W, p + 1) raw tokens, oldest first.  The windows of consecutive tokens
    are slices of one raw-token K/V stream per sequence, so they overlap as
    they do in a model.  Caches are per sequence, everything else per token.
    """
    B = sequences * tokens
    shape = Shape(batch=B, n_entries=n_entries, pool_blocks=pool, tokens=tokens)
    W = shape.swa
    pos = context - tokens + np.arange(tokens)
    n_valid = np.tile(np.minimum((pos + 1) // ratio, n_entries), sequences).astype(np.int32)
    n_swa = np.tile(np.minimum(W, pos + 1), sequences).astype(np.int32)
    wl = make_workload(shape, modes, seed=seed, cfg_id=cfg_id, n_valid=n_valid, n_swa=n_swa, name=name)
    span = tokens + W - 1                       # raw tokens covered by all windows of a sequence
    for l, L in enumerate(wl.layers):
        raw_k = _draw((sequences, span, shape.k_dim), (seed, cfg_id, 20, l), "normal", float(np.sqrt(shape.k_dim)))
        raw_v = _draw((sequences, span, shape.v_dim), (seed, cfg_id, 21, l), "normal", float(np.sqrt(shape.v_dim)))
        for s_ in range(sequences):
            for t in range(tokens):
                b = s_ * tokens + t
                n = int(n_swa[b])                # window rows: raw positions p - n + 1 .. p
                L.k_swa[b, :n] = raw_k[s_, t + W - n: t + W]
                L.v_swa[b, :n] = raw_v[s_, t + W - n: t + W]
    wl.note = f"{sequences} x {tokens} replayed tokens at {context} tokens, ratio {ratio}"
    return wl


def toy16(seed: int = 0) -> Workload:
    """The page's 16-token illustration, with one compressed entry per token.

    Token rows 0..15 carry K/V; the query sits at position 15.  The SWA
    window holds the last 4 tokens (12..15) and the compressed candidates are
    the tokens before it (0..11), so no token is attended twice.
    """
    T, W = 16, 4
    shape = Shape(batch=1, n_entries=T, idx_heads=2, idx_dim=8, block=2, pool_blocks=4,
                  topk=3, q_heads=4, k_dim=16, v_dim=16, swa=W, dtype="f32")
    rng = _rng(seed, 0, 1)
    k_tok = rng.standard_normal(size=(1, T, 16), dtype=np.float32)
    v_tok = _rng(seed, 0, 2).standard_normal(size=(1, T, 16), dtype=np.float32)
    k_idx = _rng(seed, 0, 3).standard_normal(size=(1, T, 8), dtype=np.float32)
    q = _rng(seed, 0, 10).standard_normal(size=(1, 4, 16), dtype=np.float32)
    q_idx = _rng(seed, 0, 13).standard_normal(size=(1, 2, 8), dtype=np.float32)
    w = np.ones((1, 2), dtype=np.float32)
    layer = Layer(mode=FULL, hier=1, q=q, k_swa=np.ascontiguousarray(k_tok[:, T - W:]),
                  v_swa=np.ascontiguousarray(v_tok[:, T - W:]), q_idx=q_idx, w_idx=w)
    return Workload(name="toy16", shape=shape, k_main=k_tok, v_main=v_tok, k_idx=k_idx,
                    n_valid=np.array([T - W], dtype=np.int32),
                    n_swa=np.array([W], dtype=np.int32), layers=[layer],
                    round_block_keys=0,
                    note="page-3 toy: 16 tokens, query at 15, Top-3, SWA 4, blocks of 2, pool 4")


# named workloads -------------------------------------------------------------

WORKLOADS = {
    "toy16": dict(cfg_id=0),
    "full_b8_8k": dict(cfg_id=1, batch=8, n_entries=2048, modes=[FULL], pool=0, context=8192),
    "enc_b32_32k": dict(cfg_id=2, batch=32, n_entries=8192, modes=encoder_group_modes(5),
                        pool=0, context=32768),
    "reindex_b64_128k": dict(cfg_id=3, batch=64, n_entries=32768, modes=[REINDEX], pool=2048,
                             context=131072),
    "enc_stack_b32_32k": dict(cfg_id=5, batch=32, n_entries=8192, modes=encoder_stack_modes(), pool=0,
                              context=32768),
    "dec_b16_1m": dict(cfg_id=4, batch=16, n_entries=262144, modes=decoder_group_modes(),
                       pool=2048, context=1048576),
    # the 1M decoder group with its Full layer hierarchical too (block scoring and a
    # 2,048-block pool instead of the 262,144-entry flat scan)
    "dec_b16_1m_hier": dict(cfg_id=4, batch=16, n_entries=262144, modes=decoder_group_modes(),
                            pool=2048, context=1048576, hier_full=1),
    # the 20-layer decoder group at the 128K Reindex workload's context and batch
    "dec_b64_128k": dict(cfg_id=7, batch=64, n_entries=32768, modes=decoder_group_modes(), pool=2048,
                         context=131072),
    # one sequence's 128-token decoder replay through the 20-layer decoder group at 128K context
    "replay_t128_128k": dict(cfg_id=6, sequences=1, tokens=128, n_entries=32768, modes=decoder_group_modes(),
                             pool=2048, context=131072),
}


def named(name: str, seed: int = 0, batch: Optional[int] = None) -> Workload:
    """Build a named workload (optionally with a smaller batch for sampling)."""
    if name == "toy16":
        return toy16(seed)
    spec = WORKLOADS[name]
    if "tokens" in spec:
        return decoder_replay(spec["sequences"], spec["tokens"], spec["context"], n_entries=spec["n_entries"],
                              pool=spec["pool"], modes=spec["modes"], seed=seed, cfg_id=spec["cfg_id"], name=name)
    shape = Shape(batch=batch or spec["batch"], n_entries=spec["n_entries"],
                  pool_blocks=spec["pool"])
    wl = make_workload(shape, spec["modes"], seed=seed, cfg_id=spec["cfg_id"], name=name,
                       hier_full=spec.get("hier_full", 0))
    wl.note = f"{spec['context']} tokens at ratio 4"
    return wl
