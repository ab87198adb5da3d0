"""Partition of the forward pass over several GPUs by heads (host logic only).

The (batch, head) pairs of the forward pass are independent problems: each
query tile needs only the K/V of its own head, so the B*H heads can be
split across GPUs with no exchange on the data path (the CUDA book, ch. 15,
section 15.1, change 2: the (query tile x head x batch) units form the grid,
and no unit waits on another). Rank r of W owns one contiguous slice of the
flattened B*H heads, holds its own Q, K, V, O and LSE for that slice and
runs the single-GPU forward on it as a [1, heads, N, D] problem.

Only gathering the sharded outputs into one tensor needs a collective
(gather_heads); it is optional and outside the computation.
"""
from __future__ import annotations


def head_slice(total_heads: int, world: int, rank: int) -> tuple[int, int]:
    """[start, stop) of the flattened heads rank `rank` of `world` owns.

    Contiguous and balanced: the first total_heads % world ranks own one head
    more than the others, so slice sizes differ by at most one. A rank past
    the number of heads owns an empty slice.
    """
    if total_heads < 0 or world < 1 or not 0 <= rank < world:
        raise ValueError("need total_heads >= 0, world >= 1 and 0 <= rank < world")
    base, extra = divmod(total_heads, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def slice_bytes(start: int, stop: int, N: int, D: int, elem_bytes: int = 2) -> dict:
    """Byte offsets and sizes of a head slice inside the contiguous [B, H, N, D]
    tensors (16-bit elements by default) and the fp32 [B, H, N] LSE."""
    if not 0 <= start <= stop:
        raise ValueError("need 0 <= start <= stop")
    head = N * D * elem_bytes
    return {"tensor_offset": start * head, "tensor_bytes": (stop - start) * head,
            "lse_offset": start * N * 4, "lse_bytes": (stop - start) * N * 4}


def local_view(t, start: int, stop: int):
    """The slice of a [B, H, N, ...] tensor that holds flattened heads [start, stop),
    as a contiguous [1, stop - start, N, ...] view (no copy)."""
    B, H = t.shape[0], t.shape[1]
    flat = t.reshape(B * H, *t.shape[2:])
    return flat[start:stop].unsqueeze(0)


def gather_heads(local, total_heads: int, world: int, rank: int, group=None):
    """All-gather the ranks' head slices of one output ([1, heads, N, ...] each,
    the slices of head_slice) into the full [total_heads, N, ...] tensor on
    every rank. Slices are padded to the largest one for the collective."""
    import torch
    import torch.distributed as dist
    start, stop = head_slice(total_heads, world, rank)
    if local.shape[1] != stop - start:
        raise ValueError(f"rank {rank} holds {local.shape[1]} heads, its slice has {stop - start}")
    biggest = -(-total_heads // world)
    tail = tuple(local.shape[2:])
    pad = torch.zeros((biggest, *tail), dtype=local.dtype, device=local.device)
    pad[:stop - start] = local[0]
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad, group=group)
    pieces = []
    for r in range(world):
        a, b = head_slice(total_heads, world, r)
        pieces.append(parts[r][:b - a])
    return torch.cat(pieces, dim=0)
