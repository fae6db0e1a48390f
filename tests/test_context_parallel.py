"""Context parallelism (one long sequence per query split over ranks by block-aligned
entry ranges) on the CPU: the orchestration of context_parallel.run_group, its three
exchanges and its id bookkeeping, run as world-size 2 and 4 gloo process groups with
oracle-backed per-rank steps (tests/cp_helpers.OracleOps).  The merged result on every
rank must equal the oracle run on the unsharded sequence: the same indices (the
selection order is a strict total order) and the same attention up to rounding."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import oracle  # noqa: E402
from sparse_attention_decode_index_gb300 import context_parallel as CP  # noqa: E402
from sparse_attention_decode_index_gb300 import workloads as W  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _workload(hier_full=0):
    sh = W.Shape(batch=3, n_entries=2048, pool_blocks=32, topk=64, q_heads=8, k_dim=32, v_dim=16, swa=16)
    modes = [W.FULL, W.REUSE, W.REINDEX, W.REUSE, W.SWA]
    return W.make_workload(sh, modes, seed=5, cfg_id=80, n_valid=[2048, 1500, 37], n_swa=[16, 9, 0],
                           hier_full=hier_full)


def _rank_main(rank, world, port, out, hier_full=0):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from tests.cp_helpers import OracleOps
        wl = _workload(hier_full)
        sh = wl.shape
        plan = CP.ShardPlan(sh.n_entries, world, sh.block)
        f = lambda a: torch.from_numpy(np.ascontiguousarray(oracle.to_f64(a)))   # noqa: E731
        caches = [CP.shard_caches(f(x), plan, rank) for x in (wl.k_main, wl.v_main, wl.k_idx)]
        layers = [dict(mode=L.mode, hier=L.hier, q=f(L.q), k_swa=f(L.k_swa), v_swa=f(L.v_swa),
                       q_idx=None if L.q_idx is None else f(L.q_idx), w_idx=None if L.w_idx is None else f(L.w_idx))
                  for L in wl.layers]
        cap = caches[0].shape[1]
        kb = torch.zeros((sh.batch, cap // sh.block, sh.idx_dim), dtype=torch.float64)
        res = CP.run_group(OracleOps(sh, plan, rank), CP.TorchComm(), plan, sh, layers, *caches, kb,
                           torch.from_numpy(wl.n_valid.astype(np.int32)), torch.from_numpy(wl.n_swa.astype(np.int32)))
        ref = oracle.run_group(wl)
        cur = None
        for li, (L, r, g) in enumerate(zip(wl.layers, ref, res)):
            if L.mode in (W.FULL, W.REINDEX):
                assert np.array_equal(g["idx"].numpy(), r["idx"]), f"layer {li}: indices differ"
                cur = g["idx"]
            if L.mode == W.REUSE:
                assert np.array_equal(cur.numpy(), r["idx"])
            np.testing.assert_allclose(g["out"].numpy(), r["out"], rtol=0, atol=1e-9, err_msg=f"layer {li} out")
            fin = np.isfinite(r["lse"])
            np.testing.assert_allclose(g["lse"].numpy()[fin], r["lse"][fin], rtol=0, atol=1e-9)
            assert np.all(np.isneginf(g["lse"].numpy()[~fin]))
        out[rank] = "ok"
    except Exception as e:  # reported to the parent
        out[rank] = f"{type(e).__name__}: {e}"
        raise
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,hier_full", [(2, 0), (4, 0), (3, 1)])
def test_context_parallel_group_equals_the_unsharded_oracle_with_gloo(world, hier_full):
    """World sizes 2 and 4 split the 256 blocks evenly; 3 splits them 86 / 86 / 84 and also
    runs the Full layer hierarchically (its pool of 32 blocks then comes from three ranks)."""
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out, hier_full)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert dict(out) == {r: "ok" for r in range(world)}, dict(out)
    assert all(p.exitcode == 0 for p in procs)


def test_shard_plan_is_block_aligned_and_covers_the_context():
    for n, world, blk in ((2048, 4, 8), (2048, 3, 8), (2000, 4, 8), (16, 8, 2), (8, 4, 8)):
        plan = CP.ShardPlan(n, world, blk)
        covered = []
        for r in range(world):
            e0, n_loc = plan.entries(r)
            assert e0 % blk == 0 and n_loc >= 0
            covered.extend(range(e0, e0 + n_loc))
        assert covered == list(range(n)), (n, world, blk)
