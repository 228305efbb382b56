"""Data-parallel sharding of the CfC K-loop step over batch rows.

Batch rows are independent through the forward recurrence and the BPTT recurrence, so a batch
of B sequences splits into contiguous row shards, one per rank, with W replicated.  The only
exchange is the sum of the per-shard weight and bias gradients (and of nothing else: H, du and
dh0 of a row belong to its shard).  The sum is taken deterministically: the per-shard partials
are gathered in rank order and reduced with reduce_axis0, whose summation order depends only on
the sizes, so every rank gets bitwise the same dW and db.
"""
from __future__ import annotations


def shard_rows(B: int, world: int, rank: int) -> tuple[int, int]:
    """[start, stop) of the contiguous batch rows owned by `rank` (sizes differ by at most 1)."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    base, extra = divmod(B, world)
    start = rank * base + min(rank, extra)
    stop = start + base + (1 if rank < extra else 0)
    return start, stop


def shard_inputs(inp: dict, start: int, stop: int) -> dict:
    """Rows [start, stop) of the per-row inputs; W and b are replicated."""
    return {"u": inp["u"][:, start:stop], "h0": inp["h0"][start:stop], "W": inp["W"],
            "b": inp["b"], "ts": inp["ts"][:, start:stop], "dH": inp["dH"][:, start:stop]}


def merge_grads_gpu(partials_dW, partials_db):
    """Sum per-shard dW / db partials (lists in rank order of CUDA tensors) with reduce_axis0."""
    import torch

    from . import _lib

    dW_stack = torch.stack([p.reshape(-1) for p in partials_dW]).contiguous()
    db_stack = torch.stack([p.reshape(-1) for p in partials_db]).contiguous()
    dW = torch.empty(partials_dW[0].shape, dtype=torch.float32, device=dW_stack.device)
    db = torch.empty(partials_db[0].shape, dtype=torch.float32, device=db_stack.device)
    _lib.reduce_axis0(dW_stack, dW.view(-1))
    _lib.reduce_axis0(db_stack, db.view(-1))
    return dW, db
