"""The data-parallel shard plan: batch rows split over ranks, one exchange (the sum of the
per-shard dW and db partials, taken in rank order).

CPU: two gloo ranks each run the fp64 oracle on their row shard, all_gather their partials,
reduce them in rank order and must reproduce the full-batch oracle.  GPU: the same plan with
G shards run one after another on one GPU through the library, merged by reduce_axis0."""
import os
import socket

import numpy as np
import pytest

from recurrent_cfc_cell_gb300 import inputs
from recurrent_cfc_cell_gb300.shard import shard_inputs, shard_rows


def test_shard_rows_partition():
    for B in (1, 5, 32, 33, 2048):
        for world in (1, 2, 3, 8):
            spans = [shard_rows(B, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == B
            for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
                assert a1 == b0
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_rows(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, w, q):
    import torch
    import torch.distributed as dist

    import oracle

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    inp = inputs.make_inputs(w)
    a, b = shard_rows(w.B, world, rank)
    o = oracle.step(shard_inputs(inp, a, b))
    # The one exchange: gather every rank's dW / db partial, then reduce in rank order.
    part = torch.from_numpy(np.concatenate([o["dW"].ravel(), o["db"].ravel()]))
    gathered = [torch.empty_like(part) for _ in range(world)]
    dist.all_gather(gathered, part)
    stacked = torch.stack(gathered).numpy()
    merged = oracle.reduce_axis0(stacked)
    n_dW = o["dW"].size
    q.put((rank, a, b, merged[:n_dW], merged[n_dW:], o["H"], o["du"], o["dh0"]))
    dist.destroy_process_group()


def test_two_gloo_ranks_reproduce_the_full_batch_oracle():
    import torch.multiprocessing as mp

    import oracle

    w = inputs.custom(B=5, K=6, n_x=4, C=8, seed=21)
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, w, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    full = oracle.step(inputs.make_inputs(w))
    dW0 = results[0][3]
    for rank, a, b, dW, db, H, du, dh0 in results:
        assert np.array_equal(dW, dW0)  # every rank holds bitwise the same merged gradient
        assert oracle.rel_err(dW.reshape(full["dW"].shape), full["dW"]) <= 1e-12
        assert oracle.rel_err(db.reshape(full["db"].shape), full["db"]) <= 1e-12
        assert oracle.rel_err(H, full["H"][:, a:b]) <= 1e-15
        assert oracle.rel_err(du, full["du"][:, a:b]) <= 1e-12
        assert oracle.rel_err(dh0, full["dh0"][a:b]) <= 1e-12


@pytest.mark.gpu
def test_gpu_shards_merged_by_reduce_axis0_match_full_batch():
    import torch

    import oracle
    from gpu_helpers import GRAD_TOL
    from recurrent_cfc_cell_gb300 import build
    from recurrent_cfc_cell_gb300.shard import merge_grads_gpu
    from recurrent_cfc_cell_gb300.step import KLoopStep, to_device

    build.build()
    w = inputs.CONFIGS[1]
    inp = inputs.make_inputs(w)
    G = 3
    dWs, dbs = [], []
    for r in range(G):
        a, b = shard_rows(w.B, G, r)
        sub = {k: np.ascontiguousarray(v) for k, v in shard_inputs(inp, a, b).items()}
        st = KLoopStep(b - a, w.K, w.C, w.n_x).bind(**to_device(sub))
        st.run()
        dWs.append(st.dW.clone())
        dbs.append(st.db.clone())
    dW, db = merge_grads_gpu(dWs, dbs)
    dW2, db2 = merge_grads_gpu(dWs, dbs)
    torch.cuda.synchronize()
    assert torch.equal(dW, dW2) and torch.equal(db, db2)
    ref = oracle.step(inp)
    assert oracle.rel_err(dW.cpu().numpy(), ref["dW"]) <= GRAD_TOL
    assert oracle.rel_err(db.cpu().numpy(), ref["db"]) <= GRAD_TOL
