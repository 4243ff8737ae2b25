"""h3attn_linear (the QKV / output projection either side of the attention
core) against the FP64 oracle, and its row invariance, through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import FWD_MAX_ABS, FWD_REL_L2, lib_built, max_abs_scaled, need_gpu, rel_l2

pytestmark = pytest.mark.gpu


def _data(rows, k, n, bias, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, k, generator=g).to(torch.bfloat16)
    w = (torch.randn(n, k, generator=g) / k ** 0.5).to(torch.bfloat16)
    b = torch.randn(n, generator=g) if bias else None
    return x, w, b


def _run(x, w, b):
    from invariant_dit_attention_gb300.h3attn import linear
    flags = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    y = linear(x.cuda(), w.cuda(), None if b is None else b.cuda(), error_flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    return y


@pytest.mark.parametrize("rows,k,n,bias", [(1, 64, 32, False), (127, 128, 288, True), (129, 256, 512, True),
                                           (300, 512, 800, False), (200, 6144, 256, True)])
def test_linear_matches_oracle(rows, k, n, bias):
    need_gpu()
    lib_built()
    x, w, b = _data(rows, k, n, bias, seed=rows + k + n)
    y = _run(x, w, b).double().cpu().numpy()
    ref = oracle.linear(x, w, b)
    assert np.isfinite(y).all()
    assert rel_l2(y, ref) <= FWD_REL_L2 and max_abs_scaled(y, ref) <= FWD_MAX_ABS


def test_linear_rows_are_invariant_bitwise():
    need_gpu()
    lib_built()
    x, w, b = _data(300, 256, 512, True, seed=11)
    y = _run(x, w, b)
    assert torch.equal(_run(x, w, b), y)  # repeat
    for a, e in ((0, 1), (5, 133), (130, 300), (299, 300)):
        assert torch.equal(_run(x[a:e], w, b), y[a:e]), (a, e)


def test_linear_projection_sized_sampled_rows():
    """The block's projection at the bench size: 13539 tokens, 6144 -> 6144."""
    need_gpu()
    lib_built()
    x, w, b = _data(13539, 6144, 6144, True, seed=12)
    y = _run(x, w, b)
    rows = np.sort(np.random.default_rng(3).choice(13539, size=48, replace=False))
    ref = oracle.linear(x, w, b, rows=rows)
    got = y[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    assert rel_l2(got, ref) <= FWD_REL_L2 and max_abs_scaled(got, ref) <= FWD_MAX_ABS


def test_linear_argument_errors_and_empty():
    need_gpu()
    lib_built()
    from invariant_dit_attention_gb300.h3attn import ERR_INVALID_ARG, ERR_UNSUPPORTED, H3AttnError, linear
    x = torch.zeros(4, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(64, 128, dtype=torch.bfloat16, device="cuda")
    for xx, ww, st in ((x[:, :100].contiguous(), w[:, :100].contiguous(), ERR_UNSUPPORTED),
                       (x, torch.zeros(48, 128, dtype=torch.bfloat16, device="cuda"), ERR_UNSUPPORTED)):
        with pytest.raises(H3AttnError) as e:
            linear(xx, ww)
        assert e.value.status == st
    xm = torch.zeros(4 * 128 + 1, dtype=torch.bfloat16, device="cuda")[1:].view(4, 128)
    with pytest.raises(H3AttnError) as e:
        linear(xm, w)
    assert e.value.status == ERR_INVALID_ARG
    out = torch.full((0, 64), 1.0, dtype=torch.bfloat16, device="cuda")
    assert linear(x[:0], w, out=out).shape == (0, 64)
