"""h3attn_qkv_forward: the QKV projection with the q/k norm and RoPE fused into
its epilogue, then the attention forward ("ws1_one_h3_block" page of
RL-Kernel, PR #539, Bindings table: the block's QKV projection feeding
q_norm/k_norm and rope_q/rope_k).

The fused call must give bitwise what the separate calls give (h3attn_linear,
split into q, k, v, then h3attn_forward), and the oracle's result within the
usual tolerances."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from invariant_dit_attention_gb300 import workloads as W
from tests.helpers import (FWD_MAX_ABS, FWD_REL_L2, LSE_MAX_ABS, make_handle, max_abs, max_abs_scaled, need_gpu,
                           np64, rel_l2)

pytestmark = pytest.mark.gpu


def _inputs(layouts, H, in_features, seed, bias=True, **kw):
    inp = W.make_inputs(layouts, H, seed=seed, **kw)
    g = torch.Generator().manual_seed(seed + 1)
    S, D = inp.total_tokens, H * 128
    x = torch.randn(S, in_features, generator=g).to(torch.bfloat16)
    w = (torch.randn(3 * D, in_features, generator=g) / in_features ** 0.5).to(torch.bfloat16)
    b = (0.1 * torch.randn(3 * D, generator=g)) if bias else None
    return inp, x, w, b


def _fused(inp, x, w, b, **hkw):
    from invariant_dit_attention_gb300.h3attn import to_device
    H = inp.num_heads
    h = make_handle(H, max(inp.total_tokens, 1), 64, **hkw)
    d = to_device(inp)
    q, k, v, out, lse = h.qkv_forward(x.cuda(), w.cuda(), None if b is None else b.cuda(), d["q_norm_w"],
                                      d["k_norm_w"], d["pos"], d["seg_offsets"])
    torch.cuda.synchronize()
    h.check()
    h.close()
    return [t.cpu() for t in (q, k, v, out, lse)]


def _separate(inp, x, w, b):
    from invariant_dit_attention_gb300.h3attn import linear, to_device
    S, H = inp.total_tokens, inp.num_heads
    D = H * 128
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = linear(x.cuda(), w.cuda(), None if b is None else b.cuda(), error_flags=flags)
    q, k, v = (y[:, i * D:(i + 1) * D].reshape(S, H, 128).contiguous() for i in range(3))
    h = make_handle(H, max(S, 1), 64)
    d = to_device(inp)
    out, lse = h.forward(q, k, v, d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    h.check()
    h.close()
    return [t.cpu() for t in (q, k, v, out, lse)]


def _same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


CASES = {
    "tiny_packed_H4_in256": (W.WORKLOADS["tiny_packed"].samples, 4, 256, 3),
    "ragged_H6_in384": ([W.SampleLayout(n_text=7, grid=(2, 5, 13), n_audio=3), W.SampleLayout(n_text=1),
                         W.SampleLayout(n_text=33, grid=(1, 8, 9))], 6, 384, 4),
    "odd_heads_H3_in128": ([W.SampleLayout(n_text=5, grid=(1, 6, 7), n_audio=9), 130], 3, 128, 5),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_fused_equals_separate_calls_bitwise(case):
    need_gpu()
    layouts, H, fin, seed = CASES[case]
    inp, x, w, b = _inputs(layouts, H, fin, seed)
    fused, sep = _fused(inp, x, w, b), _separate(inp, x, w, b)
    for name, a, c in zip(("q", "k", "v", "out", "lse"), fused, sep):
        assert _same_bits(a, c), f"{case}: {name} differs from the separate calls"


def test_fused_without_bias_equals_separate_calls_bitwise():
    need_gpu()
    layouts, H, fin, seed = CASES["ragged_H6_in384"]
    inp, x, w, _ = _inputs(layouts, H, fin, seed + 10, bias=False)
    fused, sep = _fused(inp, x, w, None), _separate(inp, x, w, None)
    for name, a, c in zip(("q", "k", "v", "out", "lse"), fused, sep):
        assert _same_bits(a, c), name


@pytest.mark.parametrize("case", ["tiny_packed_H4_in256", "ragged_H6_in384"])
def test_fused_matches_oracle(case):
    """q, k, v against the FP64 projection; out and lse against the FP64 forward
    of the q, k, v the call produced."""
    need_gpu()
    layouts, H, fin, seed = CASES[case]
    inp, x, w, b = _inputs(layouts, H, fin, seed)
    q, k, v, out, lse = _fused(inp, x, w, b)
    S, D = inp.total_tokens, H * 128
    y_ref = oracle.linear(x, w, b)
    for i, t in enumerate((q, k, v)):
        ref = y_ref[:, i * D:(i + 1) * D].reshape(S, H, 128)
        assert rel_l2(np64(t), ref) <= FWD_REL_L2 and max_abs_scaled(np64(t), ref) <= FWD_MAX_ABS
    out_ref, lse_ref = oracle.forward(q, k, v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets)
    assert rel_l2(np64(out), out_ref) <= FWD_REL_L2
    assert max_abs_scaled(np64(out), out_ref) <= FWD_MAX_ABS
    assert max_abs(np64(lse), lse_ref) <= LSE_MAX_ABS


@pytest.mark.parametrize("case", ["tiny_packed_H4_in256", "ragged_H6_in384"])
def test_fused_matches_oracle_end_to_end(case):
    """x to out through the oracle alone: the FP64 projection of x, rounded to
    bf16 as the projection's outputs are (nearest even), then the FP64 forward
    of those rows; compared with the fused call's out and lse."""
    need_gpu()
    layouts, H, fin, seed = CASES[case]
    inp, x, w, b = _inputs(layouts, H, fin, seed)
    _, _, _, out, lse = _fused(inp, x, w, b)
    S, D = inp.total_tokens, H * 128
    y_ref = torch.from_numpy(oracle.linear(x, w, b)).to(torch.bfloat16)  # one rounding of the FP64 result
    q_r, k_r, v_r = (y_ref[:, i * D:(i + 1) * D].reshape(S, H, 128).contiguous() for i in range(3))
    out_ref, lse_ref = oracle.forward(q_r, k_r, v_r, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets)
    assert rel_l2(np64(out), out_ref) <= FWD_REL_L2
    assert max_abs_scaled(np64(out), out_ref) <= FWD_MAX_ABS
    assert max_abs(np64(lse), lse_ref) <= LSE_MAX_ABS


def test_fused_full_size_pack_bitwise():
    """The 12 + 925 + 4253 + 8349 pack at H = 48 with a 6144-wide input
    (W_qkv 18432 x 6144): fused and separate calls agree bit for bit."""
    need_gpu()
    w_, _ = W.make_workload("packed_13539")
    inp, x, w, b = _inputs(w_.samples, 48, 6144, 21)
    fused, sep = _fused(inp, x, w, b), _separate(inp, x, w, b)
    for name, a, c in zip(("q", "k", "v", "out", "lse"), fused, sep):
        assert _same_bits(a, c), name


def test_fused_argument_errors():
    need_gpu()
    from invariant_dit_attention_gb300.h3attn import H3AttnError, to_device
    layouts, H, fin, seed = CASES["tiny_packed_H4_in256"]
    inp, x, w, b = _inputs(layouts, H, fin, seed)
    d = to_device(inp)
    h = make_handle(H, inp.total_tokens, 8)
    with pytest.raises(H3AttnError) as e:  # in_features not a multiple of 64
        h.qkv_forward(x[:, :96].contiguous().cuda(), w[:, :96].contiguous().cuda(), b.cuda(), d["q_norm_w"],
                      d["k_norm_w"], d["pos"], d["seg_offsets"])
    assert e.value.status == 2
    with pytest.raises(H3AttnError) as e:  # misaligned x
        xm = torch.empty(x.numel() + 8, dtype=torch.bfloat16, device="cuda")[1:1 + x.numel()].view(x.shape)
        h.qkv_forward(xm, w.cuda(), b.cuda(), d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
    assert e.value.status == 1
    h.close()
    hc = make_handle(H, inp.total_tokens, 8, key_order="canonical")
    with pytest.raises(H3AttnError) as e:  # the fused call is packed-order only
        hc.qkv_forward(x.cuda(), w.cuda(), b.cuda(), d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
    assert e.value.status == 2
    hc.close()
