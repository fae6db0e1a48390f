"""Context parallelism through the CUDA kernels (context_parallel.CudaOps and libcsa2's
shard, concat and merge kernels), with the ranks emulated by threads on one GPU: the
ranks' kernels never wait on one another, only the host threads meet at the
all-gathers.  The merged result of every rank must match the oracle on the unsharded
sequence: indices bit-exact, attention within 1e-2."""
import threading

import numpy as np
import pytest

import oracle
from sparse_attention_decode_index_gb300 import context_parallel as CP
from sparse_attention_decode_index_gb300 import workloads as W
from tests.cp_helpers import ThreadComm
from tests.gpu_helpers import compare_attention, lib_ready, need_gpu, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    need_gpu()
    return lib_ready()


@pytest.mark.parametrize("world", [2, 4])
def test_context_parallel_on_emulated_ranks_matches_the_oracle(csa2, world):
    sh = W.Shape(batch=4, n_entries=16384, pool_blocks=256)
    modes = [W.FULL, W.REUSE, W.REINDEX, W.REUSE, W.SWA]
    wl = W.make_workload(sh, modes, seed=9, cfg_id=81, n_valid=[16384, 12001, 3000, 700], n_swa=[128, 128, 5, 0])
    d = csa2.upload(wl)
    plan = CP.ShardPlan(sh.n_entries, world, sh.block)
    state = ThreadComm.shared(world)
    state["barrier"] = threading.Barrier(world, timeout=120)
    results, errors = [None] * world, [None] * world

    def run(r):
        try:
            torch.cuda.set_device(0)
            ops = CP.CudaOps(sh, plan, r)
            caches = [CP.shard_caches(d[k], plan, r) for k in ("k_main", "v_main", "k_idx")]
            kb = torch.zeros((sh.batch, ops.nb_cap, sh.idx_dim), dtype=torch.bfloat16, device="cuda")
            results[r] = CP.run_group(ops, ThreadComm(r, world, state), plan, sh, d["layers"], *caches, kb,
                                      d["n_valid"], d["n_swa"])
            torch.cuda.synchronize()
            st, bits = csa2.read_device_error(ops.ws)
            assert st == 0, f"rank {r}: device error bits {bits:#x}"
        except Exception as e:   # re-raised in the test thread
            errors[r] = e
            state["barrier"].abort()

    threads = [threading.Thread(target=run, args=(r,)) for r in range(world)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    for e in errors:
        if e is not None:
            raise e
    ref = oracle.run_group(wl)
    for r in range(world):
        cur = None
        for li, (L, want, got) in enumerate(zip(wl.layers, ref, results[r])):
            if L.mode in (W.FULL, W.REINDEX):
                assert np.array_equal(got["idx"].cpu().numpy(), want["idx"]), f"rank {r} layer {li}: indices differ"
                cur = got["idx"]
            if L.mode == W.REUSE:
                assert np.array_equal(cur.cpu().numpy(), want["idx"])
            compare_attention(got["out"].cpu().numpy(), got["lse"].cpu().numpy(), want["out"], want["lse"])
