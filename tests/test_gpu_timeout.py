"""Bounded on-device waits, made to run out on purpose.

Every wait of the tensor-core kernels gives up after a clock budget.  A test
hook (h3attn_debug_stall) makes one role of one kernel wait once on a barrier
that nothing completes, with a short budget: the call must then fail closed -
h3attn_device_status reports TIMEOUT - and the kernel must unwind without
leaving bulk copies or tensor-core products in flight and release its tensor
memory, so that the next call on the same handle is an ordinary one with
oracle-parity results.  This is the strict mode of the "ws1_full_h3_transformer"
page (RL-Kernel PR #571), Scope / Known limitations: a failure closes rather
than falling back.  No GPU fault, trap or endless wait is involved.
"""

import numpy as np
import pytest
import torch

from invariant_dit_attention_gb300 import workloads as W
from tests.helpers import (BWD_REL_L2, FWD_MAX_ABS, FWD_REL_L2, make_handle, max_abs_scaled, need_gpu, np64,
                           oracle_backward, oracle_forward, rel_l2)

pytestmark = pytest.mark.gpu

ROLES = ("producer", "mma", "consumer")
BUDGET = 2_000_000  # clock cycles, about 1 ms: the stalled wait's limit


def _inputs():
    # ragged samples: several items per kernel, tail tiles, a one-token sample
    return W.make_inputs([300, 129, 1], 4, seed=9090, with_grad=True)


def _expect_timeout(h):
    from invariant_dit_attention_gb300.h3attn import ERR_TIMEOUT
    st = h.device_status()
    assert st == ERR_TIMEOUT, f"device status {st}, expected TIMEOUT"
    assert h.device_status() == 0, "the error word is cleared once read"


@pytest.mark.parametrize("role", ROLES)
def test_forward_wait_runs_out_and_next_call_is_clean(role):
    need_gpu()
    from invariant_dit_attention_gb300.h3attn import to_device
    inp = _inputs()
    d = to_device(inp)
    h = make_handle(4, inp.total_tokens, 4)
    args = (d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
    ref_out, ref_lse = (t.clone() for t in h.forward(*args))
    h.check()
    h.debug_stall("fwd", role, BUDGET)
    h.forward(*args)
    _expect_timeout(h)
    out, lse = h.forward(*args)
    h.check()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    o_ref, _ = oracle_forward("timeout_9090", inp)
    o = np64(out)
    assert rel_l2(o, o_ref) <= FWD_REL_L2 and max_abs_scaled(o, o_ref) <= FWD_MAX_ABS


@pytest.mark.parametrize("kernel,store_ds", [("dkdv", True), ("dq", True), ("dq", False)])
@pytest.mark.parametrize("role", ROLES)
def test_backward_wait_runs_out_and_next_call_is_clean(kernel, store_ds, role):
    need_gpu()
    from invariant_dit_attention_gb300.h3attn import to_device
    inp = _inputs()
    d = to_device(inp)
    h = make_handle(4, inp.total_tokens, 4, store_ds=store_ds)
    fargs = (d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
    out, lse = h.forward(*fargs)

    def bwd():
        return h.backward(*fargs, out, lse, d["dout"])

    ref = {k: v.clone() for k, v in bwd().items()}
    h.check()
    h.debug_stall(kernel, role, BUDGET)
    bwd()
    _expect_timeout(h)
    g = bwd()
    h.check()
    for name, t in ref.items():
        assert torch.equal(g[name], t), name
    r = oracle_backward("timeout_9090_bwd", inp)
    for name in ("dq", "dk", "dv", "dq_norm_w", "dk_norm_w"):
        assert rel_l2(np64(g[name]), r[name]) <= BWD_REL_L2, name


@pytest.mark.parametrize("role", ROLES)
def test_qkv_projection_wait_runs_out_and_next_call_is_clean(role):
    need_gpu()
    from invariant_dit_attention_gb300.h3attn import to_device
    inp = _inputs()
    d = to_device(inp)
    S, H, D = inp.total_tokens, 2, 256
    g = torch.Generator().manual_seed(5)
    x = torch.randn(S, D, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(3 * H * 128, D, generator=g) / D ** 0.5).to(torch.bfloat16).cuda()
    b = (0.1 * torch.randn(3 * H * 128, generator=g)).cuda()
    h = make_handle(H, S, 4)

    def call():
        return h.qkv_forward(x, w, b, d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])

    ref = [t.clone() for t in call()]
    h.check()
    h.debug_stall("qkv", role, BUDGET)
    call()
    _expect_timeout(h)
    res = call()
    h.check()
    for a, r in zip(res, ref):
        assert torch.equal(a, r)


def test_stall_request_is_cleared_by_the_call_that_reads_it():
    need_gpu()
    from invariant_dit_attention_gb300.h3attn import to_device
    inp = _inputs()
    d = to_device(inp)
    h = make_handle(4, inp.total_tokens, 4)
    args = (d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
    h.debug_stall("dkdv", "mma", BUDGET)  # the next call is a forward: no dK/dV kernel runs
    h.forward(*args)
    h.check()
    out, lse = h.forward(*args)
    h.backward(*args, out, lse, d["dout"])  # the request was cleared: no stall here
    h.check()
    h.debug_stall("fwd", "mma", BUDGET)
    h.debug_stall(None)  # cancelled
    h.forward(*args)
    h.check()
