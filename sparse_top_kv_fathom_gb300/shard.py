"""Row sharding across ranks (one process per GPU).

Rows (layer or session, KV head) are independent in the decode step, so a
multi-GPU run splits them across ranks with no exchange on the data path; the
only collectives are the harness's barrier and the max-over-ranks of the timed
region.  Works with any torch.distributed backend (nccl on GPUs, gloo on CPU).
"""
import torch


def partition(total, world, rank):
    """Contiguous, balanced [start, stop) of `total` units for `rank` of `world`."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    base, extra = divmod(total, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def _initialized():
    return torch.distributed.is_available() and torch.distributed.is_initialized()


def reduce_scalar(x, op="max", device="cpu"):
    """Reduce one float over all ranks (identity when not distributed)."""
    if not _initialized():
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    ops = {"max": torch.distributed.ReduceOp.MAX, "sum": torch.distributed.ReduceOp.SUM,
           "min": torch.distributed.ReduceOp.MIN}
    torch.distributed.all_reduce(t, op=ops[op])
    return float(t.item())


def barrier():
    if _initialized():
        torch.distributed.barrier()
