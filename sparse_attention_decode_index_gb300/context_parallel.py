"""Context parallelism for CSA2 decode: one long sequence per query split over
G ranks by block-aligned ranges of its compressed entries.

The pages describe no multi-GPU scheme.  The split keeps the method's
results because its selection order (score descending, entry id ascending)
is a strict total order -- the Top-k of a union equals the Top-k of the union
of each part's Top-k list -- and because softmax partials over disjoint key
sets combine exactly by their log-sum-exp.  The architecture page k-a.in
"DeepSeek V4.1 Flash", bullet "Hierarchical indexer" (at most 16,384
candidates whatever the context length), is what keeps the exchanged lists
small for long contexts.

Per indexing layer, each rank (holding entries [e0, e0 + n_loc) of every
sequence) runs:

1. hierarchical layers: its local block scores and local pool of the top
   min(P, local blocks) blocks, with their scores; all-gather of the G pools;
   the exact global pool of min(P, NB) blocks; the pooled entries of its own
   blocks;
2. its local token scores (pooled, or flat over its valid entries) and local
   exact Top-K with scores;
3. all-gather of the G (id, score) lists; the exact global Top-K (identical on
   every rank);

and per layer (Reuse layers reuse the latest global Top-K):

4. attention partials (out, lse) over the selected entries it holds, plus the
   SWA rows on the one rank that owns the window;
5. all-gather of the partials and their merge in fixed rank order.

Every step runs in libcsa2's kernels (``CudaOps``); the exchanges are the
communicator's all-gathers (``TorchComm``: ``torch.distributed``, NCCL on GPU
ranks).  The ops and the communicator are parameters, so the orchestration
can also be driven by other implementations of the same steps.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence, Tuple

import torch

from . import csa2

FULL, REINDEX, REUSE, SWA = csa2.FULL, csa2.REINDEX, csa2.REUSE, csa2.SWA


@dataclasses.dataclass(frozen=True)
class ShardPlan:
    """Block-aligned split of n_entries compressed entries over `world` ranks."""
    n_entries: int
    world: int
    block: int

    def blocks_per_rank(self) -> int:
        nb = -(-self.n_entries // self.block)
        return -(-nb // self.world)

    def entries(self, rank: int) -> Tuple[int, int]:
        """(e0, n_loc): the entry range [e0, e0 + n_loc) held by `rank` (n_loc may be 0)."""
        per = self.blocks_per_rank() * self.block
        e0 = min(rank * per, self.n_entries)
        return e0, min(per, self.n_entries - e0)


class TorchComm:
    """All-gather through torch.distributed (one process per rank)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def all_gather(self, t: torch.Tensor) -> torch.Tensor:
        t = t.contiguous()
        out = torch.empty((self.world,) + tuple(t.shape), dtype=t.dtype, device=t.device)
        self.dist.all_gather(list(out.unbind(0)), t, group=self.group)
        return out


class CudaOps:
    """The per-rank steps on this rank's GPU, through libcsa2.

    `shape` is the global problem shape (n_entries = the whole context).
    The rank's caches are [B, n_loc, ...] slices; its workspaces are sized for
    the local token stage and the local block stage."""

    def __init__(self, shape, plan: ShardPlan, rank: int, device=None):
        self.device = torch.device(device or "cuda")
        self.plan = plan
        self.rank = rank
        self.e0, self.n_loc = plan.entries(rank)
        self.cap = max(plan.blocks_per_rank() * plan.block, plan.block)   # every rank's cache capacity
        self.shape = dataclasses.replace(shape, n_entries=self.cap)
        self.nb_cap = self.cap // plan.block
        self.shape_blocks = dataclasses.replace(shape, n_entries=self.nb_cap, pool_blocks=max(shape.pool_blocks, 0))
        self.ws = csa2.workspace(self.shape, self.device)
        self.ws_blocks = csa2.workspace(self.shape_blocks, self.device)
        self._const = {}

    def _i32(self, *shape):
        return torch.empty(shape, dtype=torch.int32, device=self.device)

    def _f32(self, *shape):
        return torch.empty(shape, dtype=torch.float32, device=self.device)

    # counts ----------------------------------------------------------------
    def local_counts(self, n_valid, div: int = 1):
        out = self._i32(n_valid.shape[0])
        csa2.shard_counts(n_valid, self.e0, self.n_loc, out, div=div)
        return out

    def block_keys(self, k_idx, n_valid_loc, kb, round_to_int: bool = True):
        csa2.block_keys(self.shape, k_idx, n_valid_loc, kb, self.ws, round_to_int=round_to_int)

    # selection --------------------------------------------------------------
    def block_topk(self, q_idx, w, kb, n_blocks_loc, pool: int):
        """Local pool: the top min(pool, local blocks) blocks (local ids, ascending) and their scores."""
        B = q_idx.shape[0]
        sc = self._f32(B, self.nb_cap)
        csa2.index_tokens(self.shape_blocks, q_idx, w, kb, n_blocks_loc, sc, self.ws_blocks)
        ids, s = self._i32(B, pool), self._f32(B, pool)
        csa2.topk(self.shape_blocks, sc, pool, ids, self.ws_blocks, n_cand=n_blocks_loc, score_out=s)
        return ids, s

    def token_topk(self, q_idx, w, k_idx, n_valid_loc, k: int, pool_loc=None, n_pool_loc=None):
        """Local exact Top-k (local entry ids, ascending) and scores, flat or over a local pool."""
        B = q_idx.shape[0]
        ids, s = self._i32(B, k), self._f32(B, k)
        if pool_loc is None:
            sc = self._f32(B, self.cap)
            csa2.index_tokens(self.shape, q_idx, w, k_idx, n_valid_loc, sc, self.ws)
            csa2.topk(self.shape, sc, k, ids, self.ws, n_cand=n_valid_loc, score_out=s)
        else:
            P = pool_loc.shape[1]
            sc, cand, nc = self._f32(B, P * self.plan.block), self._i32(B, P * self.plan.block), self._i32(B)
            csa2.index_tokens(self.shape, q_idx, w, k_idx, n_valid_loc, sc, self.ws, pool=pool_loc, n_pool=n_pool_loc,
                              cand_out=cand, n_cand_out=nc)
            csa2.topk(self.shape, sc, k, ids, self.ws, cand=cand, n_cand=nc, score_out=s)
        return ids, s

    def slice_ids(self, ids, lo: int, hi: int, delta: int, ld_out: Optional[int] = None):
        out = self._i32(ids.shape[0], ld_out or ids.shape[1])
        n = self._i32(ids.shape[0])
        csa2.shard_slice(ids, lo, hi, delta, out, self.ws, n_out=n)
        return out, n

    def merge_topk(self, ids_parts, scores_parts, k: int):
        """Exact Top-k over the gathered [G, B, k'] (global id, score) lists; ids ascending, -1 padded."""
        G, B, kp = ids_parts.shape
        ids_all, sc_all = self._i32(B, G * kp), self._f32(B, G * kp)
        csa2.concat_parts(ids_parts, scores_parts, ids_all, sc_all)
        out = self._i32(B, k)
        csa2.topk(self.shape_blocks, sc_all, k, out, self.ws_blocks, cand=ids_all)
        return out

    # attention ----------------------------------------------------------------
    def attention(self, q, k_main, v_main, idx_loc, k_swa, v_swa, n_swa):
        B, H = q.shape[0], q.shape[1]
        out, lse = self._f32(B, H, self.shape.v_dim), self._f32(B, H)
        csa2.sparse_attn(self.shape, q, k_main, v_main, idx_loc, k_swa, v_swa, n_swa, out, self.ws, lse=lse)
        return out, lse

    def merge_attention(self, outs, lses):
        out, lse = self._f32(*outs.shape[1:]), self._f32(*lses.shape[1:])
        csa2.merge_attn(outs, lses, out, lse)
        return out, lse

    def no_rows(self, B: int, K: int):
        """An index list with no main row (made once per size)."""
        key = ("none", B, K)
        if key not in self._const:
            self._const[key] = torch.full((B, K), -1, dtype=torch.int32, device=self.device)
        return self._const[key]

    def zero_counts(self, B: int):
        """Window counts of a rank that does not own the window (made once per size)."""
        key = ("zero", B)
        if key not in self._const:
            self._const[key] = torch.zeros(B, dtype=torch.int32, device=self.device)
        return self._const[key]


def run_group(ops, comm, plan: ShardPlan, shape, layers: Sequence[Dict], k_main, v_main, k_idx, kb, n_valid, n_swa,
              swa_owner: Optional[int] = None, round_block_keys: bool = True) -> List[Dict[str, torch.Tensor]]:
    """One rank's part of a layer group under context parallelism.

    k_main / v_main / k_idx are this rank's [B, cap, ...] cache slices (entries
    [e0, e0 + n_loc) of every sequence, rows past n_loc unused), kb is a
    [B, cap / block, dI] buffer for its block summary keys (filled here when a
    layer is hierarchical), n_valid [B] the global valid counts, n_swa [B] the
    window fill counts, and `layers` the per-layer dicts of
    ``csa2.layer_group`` (q, q_idx, w_idx, k_swa, v_swa).  The window belongs
    to rank `swa_owner` (default: the last rank, which holds the newest
    entries).  Returns, per layer, the merged ``out`` [B, H, dv] and ``lse``
    [B, H] (identical on every rank) and, for indexing layers, the global
    ``idx`` [B, K].
    """
    rank, G = comm.rank, comm.world
    if G != plan.world:
        raise ValueError("the plan's world size differs from the communicator's")
    if getattr(shape, "tokens", 1) > 1:
        raise ValueError("context parallelism serves one query token per sequence")
    owner = G - 1 if swa_owner is None else swa_owner
    e0, n_loc = plan.entries(rank)
    blk = plan.block
    b0, nb_loc_cap = e0 // blk, -(-n_loc // blk)
    K, P = shape.topk, shape.pool_blocks
    B = n_valid.shape[0]
    nv_loc = ops.local_counts(n_valid, 1)
    n_swa_eff = n_swa if rank == owner else ops.zero_counts(B)
    hier = any(int(L.get("hier", 0)) for L in layers)
    nb_loc = None
    if hier:
        if P < 1:
            raise ValueError("a hierarchical layer needs pool_blocks > 0")
        ops.block_keys(k_idx, nv_loc, kb, round_to_int=round_block_keys)
        nb_loc = ops.local_counts(n_valid, blk)
    results: List[Dict[str, torch.Tensor]] = []
    cur = None
    for L in layers:
        mode = int(L["mode"])
        r: Dict[str, torch.Tensor] = {}
        if mode in (FULL, REINDEX):
            if int(L.get("hier", 0)):
                ids_b, sc_b = ops.block_topk(L["q_idx"], L["w_idx"], kb, nb_loc, P)
                gids_b, _ = ops.slice_ids(ids_b, 0, nb_loc_cap, b0)
                pool_g = ops.merge_topk(comm.all_gather(gids_b), comm.all_gather(sc_b), P)
                pool_loc, npool_loc = ops.slice_ids(pool_g, b0, b0 + nb_loc_cap, -b0)
                ids_t, sc_t = ops.token_topk(L["q_idx"], L["w_idx"], k_idx, nv_loc, K, pool_loc, npool_loc)
            else:
                ids_t, sc_t = ops.token_topk(L["q_idx"], L["w_idx"], k_idx, nv_loc, K)
            gids_t, _ = ops.slice_ids(ids_t, 0, n_loc, e0)
            cur = ops.merge_topk(comm.all_gather(gids_t), comm.all_gather(sc_t), K)
            r["idx"] = cur
        elif mode == REUSE:
            if cur is None:
                raise ValueError("a Reuse layer needs an earlier Full or Reindex layer in the group")
        elif mode != SWA:
            raise ValueError(f"unknown layer mode {mode}")
        if mode == SWA:
            idx_loc = ops.no_rows(B, K)
        else:
            idx_loc, _ = ops.slice_ids(cur, e0, e0 + n_loc, -e0)
        out_l, lse_l = ops.attention(L["q"], k_main, v_main, idx_loc, L["k_swa"], L["v_swa"], n_swa_eff)
        r["out"], r["lse"] = ops.merge_attention(comm.all_gather(out_l), comm.all_gather(lse_l))
        results.append(r)
    return results


def shard_caches(t: torch.Tensor, plan: ShardPlan, rank: int) -> torch.Tensor:
    """The [B, cap, ...] slice of a [B, N, ...] cache that `rank` holds (zero rows past its range)."""
    e0, n_loc = plan.entries(rank)
    cap = max(plan.blocks_per_rank() * plan.block, plan.block)
    out = torch.zeros((t.shape[0], cap) + tuple(t.shape[2:]), dtype=t.dtype, device=t.device)
    out[:, :n_loc] = t[:, e0:e0 + n_loc]
    return out
