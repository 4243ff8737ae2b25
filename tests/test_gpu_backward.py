"""Backward parity of the CUDA path against the FP64 oracle, through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
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


# 24 samples of 1 to 200 tokens (a seeded draw)
MANY_SAMPLES = [int(x) for x in np.random.default_rng(24).integers(1, 201, size=24)]
# 50 samples of 1 to 60 tokens (a seeded draw): many short items, most of them tails
FIFTY_SAMPLES = [int(x) for x in np.random.default_rng(50).integers(1, 61, size=50)]


@pytest.mark.parametrize("lengths", [[1, 64, 65], [129, 2, 200], [300], [127, 128, 129], [255, 256, 257],
                                     MANY_SAMPLES, FIFTY_SAMPLES])
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


# ---- the backward as the bench times it: the packed batch of 12 + 925 + 4253 + 8349
# tokens with the stored dS.  The dS blocks of one head of this pack number
# 1 + 64 + 1156 + 4356 = 5577 (32 KB each): at 24 heads they take 4.39 GB, past
# 2^32 bytes of workspace; at 48 heads 8.77 GB, with block indices up to 267,696.

def _bench_pack_inputs(num_heads):
    w = W.WORKLOADS["packed_13539"]
    return W.make_inputs(w.samples, num_heads, w.seed, w.std, w.outlier_frac, w.outlier_scale, with_grad=True)


def _ds_bytes(inp):
    blocks = sum(((L + 127) // 128) ** 2 for L in inp.meta["lengths"]) * inp.num_heads
    return blocks * 128 * 128 * 2


@pytest.mark.slow
def test_backward_bench_pack_24_heads_full_oracle():
    """Every gradient of the 13539-token pack at 24 heads (4.39 GB of stored dS)
    against the full FP64 backward: dq, dk, dv, the total and per-sample weight
    gradients."""
    need_gpu()
    inp = _bench_pack_inputs(24)
    assert _ds_bytes(inp) > (1 << 32)
    _, _, g = run_fwd_bwd(inp, max_samples=8, store_ds=True)
    check_grads(g, oracle_backward("bench_pack_24", inp), inp.num_samples)


@pytest.mark.slow
def test_backward_bench_pack_48_heads_first_and_last_heads():
    """The bench's own inputs (48 heads, seed as the bench draws them, stored dS
    of 8.77 GB): dq, dk, dv of heads 0-1 and 46-47 against the oracle restricted
    to those heads.  Heads 46-47 of the later-ranked samples own the highest
    block indices and byte offsets of the stored dS."""
    need_gpu()
    inp = _bench_pack_inputs(48)
    assert _ds_bytes(inp) > 8 * (1 << 30)
    _, _, g = run_fwd_bwd(inp, max_samples=8, store_ds=True)
    for lo, hi in ((0, 2), (46, 48)):
        ref = oracle.backward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets,
                              inp.dout, heads=(lo, hi))
        for name in ("dq", "dk", "dv"):
            x = np64(g[name][:, lo:hi])
            assert np.isfinite(x).all(), (name, lo, hi)
            e = rel_l2(x, ref[name][:, lo:hi])
            assert e <= BWD_REL_L2, f"{name} heads [{lo}, {hi}) rel-L2 {e:.3e}"


def test_backward_reuse_of_forward_rows_is_bitwise_the_recomputation():
    """With reuse_qk_hat the backward skips the norm/RoPE pass when the handle's
    last forward computed q^/k^ from the same tensors; the gradients must be the
    recomputing handle's bits, also when another forward ran in between (then
    the rows are recomputed)."""
    need_gpu()
    from invariant_dit_attention_gb300.h3attn import to_device
    a = W.make_inputs([300, 129, 1], 6, seed=515, with_grad=True)
    b = W.make_inputs([300, 129, 1], 6, seed=516, with_grad=True)
    da, db = to_device(a), to_device(b)
    on = make_handle(6, a.total_tokens, 4, reuse_qk_hat=True)
    off = make_handle(6, a.total_tokens, 4, reuse_qk_hat=False)

    def fargs(d):
        return (d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])

    out_a, lse_a = (t.clone() for t in off.forward(*fargs(da)))
    ref = {k: v.clone() for k, v in off.backward(*fargs(da), out_a, lse_a, da["dout"]).items()}
    on.forward(*fargs(da))
    g1 = {k: v.clone() for k, v in on.backward(*fargs(da), out_a, lse_a, da["dout"]).items()}
    on.forward(*fargs(da))
    on.forward(*fargs(db))  # the workspace now holds b's rows
    g2 = on.backward(*fargs(da), out_a, lse_a, da["dout"])
    torch.cuda.synchronize()
    on.check()
    off.check()
    for k in ref:
        assert torch.equal(g1[k], ref[k]), f"reused rows: {k}"
        assert torch.equal(g2[k], ref[k]), f"rows of another forward in between: {k}"
