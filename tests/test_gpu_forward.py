"""Forward parity of the CUDA path against the FP64 oracle, through the C ABI."""

import numpy as np
import pytest
import torch

from invariant_dit_attention_gb300 import workloads as W
from tests.helpers import (FWD_MAX_ABS, FWD_REL_L2, LSE_MAX_ABS, make_handle, max_abs, max_abs_scaled, need_gpu,
                           np64, oracle_forward, rel_l2, sample_rows, workload)

pytestmark = pytest.mark.gpu


def _run_fwd(inp, H=None, max_samples=64):
    from invariant_dit_attention_gb300.h3attn import to_device
    H = H or inp.num_heads
    h = make_handle(H, max(inp.total_tokens, 1), max_samples)
    d = to_device(inp)
    out, lse = h.forward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
    torch.cuda.synchronize()
    h.check()
    return out, lse, h, d


def _check_rows(out, lse, ref_out, ref_lse, rows=None):
    o = np64(out)
    l = lse.cpu().numpy().astype(np.float64)
    if rows is not None:
        o, ref_out = o[rows], ref_out[rows]
        l, ref_lse = l[:, rows], ref_lse[:, rows]
    assert np.isfinite(o).all()
    e, m = rel_l2(o, ref_out), max_abs_scaled(o, ref_out)
    assert e <= FWD_REL_L2, f"rel-L2 {e:.3e}"
    assert m <= FWD_MAX_ABS, f"max-abs (scaled by max(1, |ref|)) {m:.3e}, raw {max_abs(o, ref_out):.3e}"
    assert max_abs(l, ref_lse) <= LSE_MAX_ABS
    return e, m


def test_forward_tiny_packed_full():
    need_gpu()
    w, inp = workload("tiny_packed")
    out, lse, _, _ = _run_fwd(inp)
    ref, ref_lse = oracle_forward("tiny_packed", inp)
    _check_rows(out, lse, ref, ref_lse)


def test_forward_single_925_full():
    need_gpu()
    w, inp = workload("single_925")
    out, lse, _, _ = _run_fwd(inp)
    ref, ref_lse = oracle_forward("single_925", inp)
    _check_rows(out, lse, ref, ref_lse)


@pytest.mark.parametrize("name", ["single_4253_outliers", "packed_13539"])
def test_forward_full_size_sampled_rows(name):
    need_gpu()
    w, inp = workload(name)
    out, lse, _, _ = _run_fwd(inp)
    rows = sample_rows(inp.seg_offsets.tolist(), per_sample=16)
    ref, ref_lse = oracle_forward(name, inp, rows=rows)
    _check_rows(out, lse, ref, ref_lse, rows)
    assert torch.isfinite(out.float()).all()


# 40 samples of 1 to 300 tokens (a seeded draw): many items, many tile tails
MANY_SAMPLES = [int(x) for x in np.random.default_rng(40).integers(1, 301, size=40)]
# 50 samples of 1 to 60 tokens (a seeded draw): many short items, most of them tails
FIFTY_SAMPLES = [int(x) for x in np.random.default_rng(50).integers(1, 61, size=50)]


@pytest.mark.parametrize("lengths", [[1], [1, 1, 1], [63, 64, 65], [127, 128, 129], [5, 300, 7, 1, 200],
                                     [257, 3], [255, 256], MANY_SAMPLES, FIFTY_SAMPLES])
def test_forward_ragged_lengths_full(lengths):
    need_gpu()
    inp = W.make_inputs([W.SampleLayout(n_text=2, grid=(1, 1, L - 2)) if L > 2 else L for L in lengths],
                        6, seed=sum(lengths))
    out, lse, _, _ = _run_fwd(inp)
    ref, ref_lse = oracle_forward(("ragged", tuple(lengths)), inp)
    _check_rows(out, lse, ref, ref_lse)


def test_single_token_sample_returns_v_exactly():
    need_gpu()
    inp = W.make_inputs([1, 9, 1], 4, seed=3)
    out, _, _, d = _run_fwd(inp)
    assert torch.equal(out[0], d["v"][0])
    assert torch.equal(out[10], d["v"][10])


def test_identical_keys_average_values():
    need_gpu()
    inp = W.make_inputs([40], 2, seed=4)
    inp.k[:] = inp.k[0]
    inp.pos.zero_()
    out, _, _, d = _run_fwd(inp)
    mean = inp.v.double().mean(0)
    assert max_abs(np64(out), np.broadcast_to(mean.numpy(), out.shape)) < 1e-2


def test_rope_identity_at_zero_positions_matches_oracle():
    need_gpu()
    inp = W.make_inputs([100, 28], 3, seed=5)
    inp.pos.zero_()
    out, lse, _, _ = _run_fwd(inp)
    ref, ref_lse = oracle_forward("zero_pos", inp)
    _check_rows(out, lse, ref, ref_lse)


def test_empty_batch_is_noop():
    need_gpu()
    h = make_handle(4, 16)
    z = torch.zeros((0, 4, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(128, device="cuda")
    pos = [torch.zeros(0, dtype=torch.int32, device="cuda")] * 3
    seg = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = h.forward(z, z, z, w, w, pos, seg, num_samples=0)
    assert out.numel() == 0
    h.check()


def test_bad_offsets_are_reported_by_device_status():
    need_gpu()
    from invariant_dit_attention_gb300.h3attn import ERR_INVALID_ARG, OK, to_device
    inp = W.make_inputs([10, 20], 2, seed=6)
    h = make_handle(2, 64)
    d = to_device(inp)
    for bad in ([0, 20, 10], [1, 10, 30], [0, 10, 31], [0, 10, 10]):
        seg = torch.tensor(bad, dtype=torch.int32, device="cuda")
        h.forward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], seg, num_samples=2)
        assert h.device_status() == ERR_INVALID_ARG
        assert h.device_status() == OK  # cleared
    out, lse = h.forward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
    assert h.device_status() == OK


def test_host_side_argument_errors():
    need_gpu()
    from invariant_dit_attention_gb300.h3attn import ERR_CAPACITY, ERR_INVALID_ARG, H3AttnError, to_device
    inp = W.make_inputs([10, 20], 2, seed=7)
    h = make_handle(2, 16, max_samples=1)
    d = to_device(inp)
    with pytest.raises(H3AttnError) as e:
        h.forward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
    assert e.value.status == ERR_CAPACITY
    h2 = make_handle(2, 64)
    qm = torch.empty(30 * 2 * 128 + 1, dtype=torch.bfloat16, device="cuda")[1:].view(30, 2, 128)
    with pytest.raises(H3AttnError) as e:
        h2.forward(qm, d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
    assert e.value.status == ERR_INVALID_ARG


@pytest.mark.parametrize("tensor", ["q", "k"])
def test_fp16_range_of_the_rotated_rows(tensor):
    """q^ and k^ are kept as fp16: a finite normed and rotated value beyond its range is a
    device error (status INVALID_ARG, then cleared).  A normed row has |n_c| <= sqrt(128)
    and a rotation keeps a pair's length, so |q^|, |k^| <= sqrt(128) max|w|: the per-value
    check runs only when 16 max|w| reaches 60000, and below that nothing can be flagged.
    A one-hot row in an unrotated channel reaches the bound exactly."""
    need_gpu()
    from invariant_dit_attention_gb300.h3attn import ERR_INVALID_ARG, OK, to_device
    inp = W.make_inputs([40, 24], 2, seed=11)
    h = make_handle(2, 64)
    d = to_device(inp)
    x = d[tensor].clone()
    x[5, 1, :] = 0
    x[5, 1, 100] = 1.0
    wname = "q_norm_w" if tensor == "q" else "k_norm_w"

    def run(w, rows):
        args = dict(d)
        args[tensor] = rows
        args[wname] = w
        return h.forward(args["q"], args["k"], args["v"], args["q_norm_w"], args["k_norm_w"], args["pos"],
                         args["seg_offsets"])

    w = torch.ones(128, device="cuda")
    w[100] = 6000.0  # sqrt(128) * 6000 = 67882 > 65504
    run(w, x)
    assert h.device_status() == ERR_INVALID_ARG
    assert h.device_status() == OK
    # a non-finite row is not a range error, also where the check runs
    nan_rows = x.clone()
    nan_rows[5, 1, 100] = float("nan")
    run(w, nan_rows)
    assert h.device_status() == OK
    w[100] = 3000.0  # 33941: inside the range, the per-value check is skipped
    out, lse = run(w, x)
    assert h.device_status() == OK
    assert bool(torch.isfinite(out.float()).all()) and bool(torch.isfinite(lse).all())
