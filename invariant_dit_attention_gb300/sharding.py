"""Head-sharded runs of the attention core across GPUs (one process per GPU).

The path has no exchange step between heads: split a layer's heads across the
ranks, give each rank its heads as contiguous [S, H_r, 128] tensors (as a
column-split QKV projection produces them) and run them through a handle of
H_r heads; every rank's out, lse, dq, dk and dv are then bitwise the one-GPU
results for those heads.  Only the q/k norm weights are shared by all heads, so
their gradient needs every rank's heads: each rank takes the per-(sample,
head) partials of its last backward (h3attn_norm_weight_grad_partials), the
ranks gather them in global head order, and every rank reduces the gathered
partials with h3attn_combine_norm_weight_grads, the library's own fixed order
(per sample over heads ascending, then over samples).  The result is bitwise
the one-GPU gradient whatever the number of ranks.  The pages' precedent is the
WS2 parallel layer (ws2_comm.py in the changed-file list of the
"ws1_full_h3_transformer" page, RL-Kernel PR #571).

This module is host logic and collectives only; the reductions run in the
library's kernels.
"""

from __future__ import annotations

import torch


def head_range(rank: int, world_size: int, num_heads: int) -> tuple:
    """Heads [lo, hi) of `rank` when `num_heads` are split into `world_size`
    contiguous blocks, the first num_heads % world_size ranks one head larger."""
    if not (0 <= rank < world_size) or num_heads < world_size:
        raise ValueError(f"cannot split {num_heads} heads over {world_size} ranks (rank {rank})")
    base, extra = divmod(num_heads, world_size)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def gather_head_partials(local: torch.Tensor, num_heads: int, group=None) -> torch.Tensor:
    """All-gather every rank's [n, H_r, 128] per-(sample, head) partials into
    [n, num_heads, 128] in global head order (ranks hold contiguous head
    blocks, see head_range).  Works on any backend whose tensors `local` lives
    on (gloo: CPU, nccl: CUDA)."""
    import torch.distributed as dist
    ws = dist.get_world_size(group)
    rank = dist.get_rank(group)
    lo, hi = head_range(rank, ws, num_heads)
    if local.shape[1] != hi - lo:
        raise ValueError(f"rank {rank} holds {local.shape[1]} heads, expected {hi - lo}")
    width = max(h1 - h0 for h0, h1 in (head_range(r, ws, num_heads) for r in range(ws)))
    padded = torch.zeros((local.shape[0], width, local.shape[2]), dtype=local.dtype, device=local.device)
    padded[:, :hi - lo] = local
    parts = [torch.empty_like(padded) for _ in range(ws)]
    dist.all_gather(parts, padded.contiguous(), group=group)
    out = [parts[r][:, :h1 - h0] for r, (h0, h1) in enumerate(head_range(r, ws, num_heads) for r in range(ws))]
    return torch.cat(out, dim=1).contiguous()


def sharded_norm_weight_grads(handle, num_samples: int, num_heads: int, group=None, stream=None) -> dict:
    """After `handle.backward` on this rank's heads: the norm-weight gradients of
    all heads, reduced in the library's fixed order (bitwise the one-GPU
    result).  Returns dq_norm_w, dk_norm_w [128] and the per-sample [n, 128]."""
    from .h3attn import combine_norm_weight_grads
    pq, pk = handle.norm_weight_grad_partials(num_samples, stream=stream)
    res = {}
    for name, part in (("dq_norm_w", pq), ("dk_norm_w", pk)):
        full = gather_head_partials(part, num_heads, group)
        per_sample, total = combine_norm_weight_grads(full, stream=stream)
        res[name], res[name + "_per_sample"] = total, per_sample
    return res
