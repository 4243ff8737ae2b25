"""Host logic of head-sharded runs on CPU: how the heads are split, and the
gather of every rank's per-(sample, head) norm-weight partials in global head
order, with two and three gloo ranks (one process per rank, as one process
runs per GPU).  The reduction after the gather is the library's fixed order
(per sample over heads ascending, then over samples ascending); written out
here in float32 with numpy, its bits after the gather must be those of the
one-process reduction for every split.  The GPU kernels of that reduction
are checked against the same order in tests/test_gpu_sharding.py."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from invariant_dit_attention_gb300.sharding import head_range


def fixed_order_reduce(partials: np.ndarray):
    """float32 [n, H, 128] -> per-sample [n, 128] (heads added in ascending
    order, one rounding per addition) and total [128] (samples ascending)."""
    n, H, _ = partials.shape
    per = np.zeros((n, 128), np.float32)
    for s in range(n):
        acc = np.zeros(128, np.float32)
        for h in range(H):
            acc = acc + partials[s, h]
        per[s] = acc
    tot = np.zeros(128, np.float32)
    for s in range(n):
        tot = tot + per[s]
    return per, tot


def _partials(n, H, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((n, H, 128)) * np.exp(rng.uniform(-8, 8, (n, H, 1)))).astype(np.float32)


@pytest.mark.parametrize("ws,H", [(1, 7), (2, 48), (3, 48), (2, 5), (4, 6), (5, 5)])
def test_head_range_splits_every_head_once_in_order(ws, H):
    ranges = [head_range(r, ws, H) for r in range(ws)]
    assert ranges[0][0] == 0 and ranges[-1][1] == H
    assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
    sizes = [hi - lo for lo, hi in ranges]
    assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1


def test_head_range_rejects_more_ranks_than_heads():
    with pytest.raises(ValueError):
        head_range(0, 4, 3)


def test_fixed_order_is_order_sensitive():
    """The reduction order matters in float32 (so fixing it is not vacuous):
    adding the heads in another order changes bits on these partials."""
    p = _partials(3, 48, 11)
    per, _ = fixed_order_reduce(p)
    rev, _ = fixed_order_reduce(p[:, ::-1].copy())
    assert not np.array_equal(per, rev)


def _digest(a: np.ndarray) -> str:
    import hashlib
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, H, out):
    import torch.distributed as dist

    from invariant_dit_attention_gb300.sharding import gather_head_partials
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        full = _partials(4, H, 1234)
        lo, hi = head_range(rank, ws, H)
        local = torch.from_numpy(full[:, lo:hi].copy())
        gathered = gather_head_partials(local, H).numpy()
        per, tot = fixed_order_reduce(gathered)
        out.put((rank, _digest(gathered), _digest(per), _digest(tot)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("ws,H", [(2, 48), (3, 48), (2, 5)])
def test_gloo_ranks_gather_partials_in_head_order_and_reduce_to_the_one_process_bits(ws, H):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, H, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in range(ws))  # read before joining: a full pipe blocks a child's exit
    for p in procs:
        p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    full = _partials(4, H, 1234)
    per, tot = fixed_order_reduce(full)
    for rank, g, per_r, tot_r in res:
        assert g == _digest(full), f"rank {rank}: gathered partials differ"
        assert per_r == _digest(per) and tot_r == _digest(tot), f"rank {rank}: reduction bits differ"
