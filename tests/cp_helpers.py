"""Test helpers for the context-parallel orchestration (imported only by tests).

* ``OracleOps`` -- the per-rank steps of ``context_parallel.run_group``
  computed on the CPU with the oracle's functions (scores, exact Top-k,
  attention) and plain numpy for the id bookkeeping and the partial merge, so
  that the orchestration and its exchanges can run as gloo processes.
* ``ThreadComm`` -- an all-gather between threads of one process (ranks
  emulated on one device; the ranks' kernels never wait on one another, only
  the host threads meet at the exchanges).
"""
import math
import threading

import numpy as np
import torch

import oracle


class ThreadComm:
    """All-gather among `world` threads; one instance per rank sharing `state`."""

    def __init__(self, rank, world, state):
        self.rank, self.world, self.state = rank, world, state

    @staticmethod
    def shared(world):
        return {"barrier": threading.Barrier(world), "slots": [None] * world}

    def all_gather(self, t):
        st = self.state
        st["slots"][self.rank] = t.contiguous()
        st["barrier"].wait()
        out = torch.stack(st["slots"], 0)
        st["barrier"].wait()
        return out


class OracleOps:
    """CPU steps for one rank holding entries [e0, e0 + n_loc); float64 data, int32 ids."""

    def __init__(self, shape, plan, rank):
        self.shape, self.plan, self.rank = shape, plan, rank
        self.e0, self.n_loc = plan.entries(rank)
        self.blk = plan.block
        self.scale = 1.0 / math.sqrt(shape.k_dim)

    def local_counts(self, n_valid, div=1):
        return ((n_valid - self.e0).clamp(0, self.n_loc) + div - 1) // div

    def block_keys(self, k_idx, n_valid_loc, kb, round_to_int=True):
        for b in range(k_idx.shape[0]):
            n = int(n_valid_loc[b])
            kb[b].zero_()
            if n:
                kk = oracle.block_keys(k_idx[b].numpy(), n, self.blk, round_to_int)
                kb[b, :kk.shape[0]] = torch.from_numpy(kk)

    def _topk(self, s, ids, k):
        sel = oracle.select_topk(s, ids, k)
        pos = {int(i): j for j, i in enumerate(ids)}
        sc = np.array([s[pos[int(i)]] if i >= 0 else -np.inf for i in sel])
        return sel, sc

    def block_topk(self, q_idx, w, kb, n_blocks_loc, pool):
        B = q_idx.shape[0]
        ids, scs = np.full((B, pool), -1), np.full((B, pool), -np.inf)
        for b in range(B):
            nb = int(n_blocks_loc[b])
            s = oracle.indexer_scores(q_idx[b].numpy(), w[b].numpy(), kb[b, :nb].numpy())
            ids[b], scs[b] = self._topk(s, np.arange(nb), pool)
        return torch.from_numpy(ids.astype(np.int32)), torch.from_numpy(scs)

    def token_topk(self, q_idx, w, k_idx, n_valid_loc, k, pool_loc=None, n_pool_loc=None):
        B = q_idx.shape[0]
        ids, scs = np.full((B, k), -1), np.full((B, k), -np.inf)
        for b in range(B):
            n = int(n_valid_loc[b])
            if pool_loc is None:
                cand = np.arange(n)
            else:
                cand = oracle.pooled_entries(pool_loc[b, :int(n_pool_loc[b])].numpy().astype(np.int64), n, self.blk)
            s = oracle.indexer_scores(q_idx[b].numpy(), w[b].numpy(), k_idx[b].numpy()[cand])
            ids[b], scs[b] = self._topk(s, cand, k)
        return torch.from_numpy(ids.astype(np.int32)), torch.from_numpy(scs)

    def slice_ids(self, ids, lo, hi, delta, ld_out=None):
        ids_np = ids.numpy()
        ld = ld_out or ids_np.shape[1]
        out, n = np.full((ids_np.shape[0], ld), -1), np.zeros(ids_np.shape[0])
        for b, row in enumerate(ids_np):
            kept = [int(i) + delta for i in row if lo <= i < hi]
            out[b, :len(kept)] = kept
            n[b] = len(kept)
        return torch.from_numpy(out.astype(np.int32)), torch.from_numpy(n.astype(np.int32))

    def merge_topk(self, ids_parts, scores_parts, k):
        G, B, kp = ids_parts.shape
        out = np.full((B, k), -1)
        for b in range(B):
            ids = ids_parts[:, b].reshape(-1).numpy().astype(np.int64)
            sc = scores_parts[:, b].reshape(-1).numpy()
            keep = ids >= 0
            out[b] = oracle.select_topk(sc[keep], ids[keep], k)
        return torch.from_numpy(out.astype(np.int32))

    def attention(self, q, k_main, v_main, idx_loc, k_swa, v_swa, n_swa):
        B, H = q.shape[0], q.shape[1]
        out, lse = np.zeros((B, H, v_main.shape[2])), np.zeros((B, H))
        for b in range(B):
            out[b], lse[b] = oracle.sparse_attention(q[b].numpy(), k_main[b].numpy(), v_main[b].numpy(),
                                                     idx_loc[b].numpy().astype(np.int64), k_swa[b].numpy(),
                                                     v_swa[b].numpy(), int(n_swa[b]), self.scale)
        return torch.from_numpy(out), torch.from_numpy(lse)

    def merge_attention(self, outs, lses):
        o, l = outs.numpy(), lses.numpy()
        M = l.max(axis=0)
        safe = np.where(np.isneginf(M), 0.0, M)
        w = np.where(np.isneginf(l), 0.0, np.exp(l - safe[None]))
        S = w.sum(axis=0)
        out = np.where(S[..., None] > 0, (w[..., None] * o).sum(axis=0) / np.where(S > 0, S, 1)[..., None], 0.0)
        lse = np.where(S > 0, safe + np.log(np.where(S > 0, S, 1)), -np.inf)
        return torch.from_numpy(out), torch.from_numpy(lse)

    def no_rows(self, B, K):
        return torch.full((B, K), -1, dtype=torch.int32)

    def zero_counts(self, B):
        return torch.zeros(B, dtype=torch.int32)
