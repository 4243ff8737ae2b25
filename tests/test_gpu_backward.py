"""Backward parity of the CUDA path against the FP64 oracle, through the C ABI."""

import numpy as np
import pytest
import torch

from invariant_dit_attention_gb300 import workloads as W
from tests.helpers import BWD_REL_L2, make_handle, need_gpu, np64, oracle_backward, rel_l2, workload

pytestmark = pytest.mark.gpu


def run_fwd_bwd(inp, max_samples=64, store_ds="auto"):
    from invariant_dit_attention_gb300.h3attn import to_device
    h = make_handle(inp.num_heads, max(inp.total_tokens, 1), max_samples, store_ds=store_ds)
    d = to_device(inp)
    out, lse = h.forward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
    g = h.backward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"], out, lse,
                   d["dout"])
    torch.cuda.synchronize()
    h.check()
    return out, lse, g


def check_grads(g, ref, n_samples):
    for name in ("dq", "dk", "dv"):
        x = np64(g[name])
        assert np.isfinite(x).all(), name
        e = rel_l2(x, ref[name])
        assert e <= BWD_REL_L2, f"{name} rel-L2 {e:.3e}"
    for name in ("dq_norm_w", "dk_norm_w"):
        e = rel_l2(np64(g[name]), ref[name])
        assert e <= BWD_REL_L2, f"{name} rel-L2 {e:.3e}"
        ps = np64(g[name + "_per_sample"])[:n_samples]
        e = rel_l2(ps, ref[name + "_per_sample"])
        assert e <= BWD_REL_L2, f"{name} per-sample rel-L2 {e:.3e}"


def test_backward_tiny_packed():
    need_gpu()
    inp = W.make_inputs(W.WORKLOADS["tiny_packed"].samples, 4, seed=1001, with_grad=True)
    _, _, g = run_fwd_bwd(inp)
    check_grads(g, oracle_backward("tiny_bwd", inp), inp.num_samples)


@pytest.mark.parametrize("lengths", [[1, 64, 65], [129, 2, 200], [300]])
def test_backward_ragged(lengths):
    need_gpu()
    inp = W.make_inputs(lengths, 6, seed=7 + sum(lengths), with_grad=True)
    _, _, g = run_fwd_bwd(inp)
    check_grads(g, oracle_backward(("ragged_bwd", tuple(lengths)), inp), inp.num_samples)


@pytest.mark.parametrize("store_ds", [False, True])
def test_backward_both_dq_paths(store_ds):
    """dQ from the dS the dK/dV kernel stored, and dQ recomputing S and dP."""
    need_gpu()
    inp = W.make_inputs([1, 64, 65, 300], 6, seed=321, with_grad=True)
    _, _, g = run_fwd_bwd(inp, store_ds=store_ds)
    check_grads(g, oracle_backward("both_dq_paths", inp), inp.num_samples)


def test_backward_single_925():
    need_gpu()
    w, base = workload("single_925")
    inp = W.make_inputs(w.samples, w.num_heads, w.seed, with_grad=True)
    _, _, g = run_fwd_bwd(inp)
    check_grads(g, oracle_backward("bwd_925", inp), 1)


@pytest.mark.slow
def test_backward_full_4253_outliers():
    need_gpu()
    w, inp = workload("fwd_bwd_4253")
    _, _, g = run_fwd_bwd(inp)
    check_grads(g, oracle_backward("fwd_bwd_4253", inp), 1)
