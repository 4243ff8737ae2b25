"""h3attn_forward_static: the forward for callers that cannot allocate device memory.

Hosts that hand a library a fixed memory pool (an inference server's plugin
slot, a process under a device-memory budget) cannot let it call cudaMalloc
while serving.  This entry point keeps its scratch in a static device array of
the library instead; its results must match h3attn_forward's on the same
inputs, call after call.  Collected last on purpose (file name).
"""

import numpy as np
import pytest
import torch

from invariant_dit_attention_gb300 import workloads as W
from tests.helpers import (FWD_MAX_ABS, FWD_REL_L2, LSE_MAX_ABS, lib_built, make_handle, max_abs, max_abs_scaled,
                           need_gpu, np64, oracle_forward, rel_l2)

pytestmark = pytest.mark.gpu


def test_static_scratch_forward_matches_handle_forward_twice():
    need_gpu()
    lib_built()
    from invariant_dit_attention_gb300.h3attn import forward_static, to_device
    inp = W.make_inputs([W.S925, 300, 1, 129], 24, seed=4242)
    d = to_device(inp)
    h = make_handle(24, inp.total_tokens, 8)
    ref_out, ref_lse = h.forward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
    torch.cuda.synchronize()
    h.check()
    flags = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(d["q"], float("nan"))
        lse = torch.full((24, inp.total_tokens), float("nan"), device="cuda")
        forward_static(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"],
                       out=out, lse=lse, error_flags=flags)
        torch.cuda.synchronize()
        assert int(flags.item()) == 0, f"call {call}: device error flags {int(flags.item())}"
        o, r = np64(out), np64(ref_out)
        assert np.isfinite(o).all()
        assert rel_l2(o, r) <= FWD_REL_L2 and max_abs_scaled(o, r) <= FWD_MAX_ABS, f"call {call}"
        # same kernels on the same inputs: the results are in fact bitwise equal
        assert torch.equal(out, ref_out), f"call {call}: out differs from h3attn_forward"
        assert torch.equal(lse, ref_lse), f"call {call}: lse differs from h3attn_forward"
    # and against the FP64 oracle, independently of h3attn_forward
    o_ref, lse_ref = oracle_forward("static_scratch_4242", inp)
    o = np64(out)
    assert rel_l2(o, o_ref) <= FWD_REL_L2 and max_abs_scaled(o, o_ref) <= FWD_MAX_ABS
    assert max_abs(np64(lse), lse_ref) <= LSE_MAX_ABS


def test_static_scratch_forward_raises_on_device_errors_without_flags():
    """With error_flags omitted the binding checks the device word itself: an
    invalid seg_offsets array (not increasing) must raise, not pass silently."""
    need_gpu()
    lib_built()
    from invariant_dit_attention_gb300.h3attn import ERR_INVALID_ARG, H3AttnError, forward_static, to_device
    inp = W.make_inputs([200, 100], 4, seed=77)
    d = to_device(inp)
    bad = torch.tensor([0, 200, 100, 300], dtype=torch.int32, device="cuda")
    with pytest.raises(H3AttnError) as e:
        forward_static(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], bad)
    assert e.value.status == ERR_INVALID_ARG
    # a valid call right after is clean
    out, _ = forward_static(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
    torch.cuda.synchronize()
    assert np.isfinite(np64(out)).all()


def test_static_scratch_forward_rejects_sizes_beyond_its_limit():
    need_gpu()
    lib_built()
    from invariant_dit_attention_gb300.h3attn import (ERR_CAPACITY, STATIC_MAX_TOKEN_HEADS, H3AttnError,
                                                      forward_static)
    H = 64
    S = STATIC_MAX_TOKEN_HEADS // H + 1
    q = torch.zeros((S, H, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(128, device="cuda")
    pos = [torch.zeros(S, dtype=torch.int32, device="cuda")] * 3
    seg = torch.tensor([0, S], dtype=torch.int32, device="cuda")
    with pytest.raises(H3AttnError) as e:
        forward_static(q, q, q, w, w, pos, seg)
    assert e.value.status == ERR_CAPACITY
