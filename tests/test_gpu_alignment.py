"""Output pointers that are 16-byte aligned but not 32-byte aligned.

The boundary promises only 16-byte alignment for every tensor (include/h3attn.h).
The forward's out rows and the backward's dv rows are written with 32-byte
stores when the caller's pointer allows it and with 16-byte stores otherwise;
both must give the same bits, write every element of the tensor and nothing
outside it.  The samples have ragged tails, so rows past a sample end (which
the stores skip) fall inside the tiles.
"""

import pytest
import torch

from invariant_dit_attention_gb300 import workloads as W
from tests.helpers import make_handle, need_gpu

pytestmark = pytest.mark.gpu

GUARD = 64  # bf16 elements on each side of the tensor
SENTINEL = 0x7FA5  # a NaN bit pattern no kernel writes


def _guarded(shape, offset_elems, device):
    """A bf16 tensor of `shape` placed `offset_elems` after a 256-byte aligned start,
    with GUARD sentinel elements before and after it."""
    n = 1
    for s in shape:
        n *= s
    buf = torch.empty(offset_elems + GUARD + n + GUARD, dtype=torch.bfloat16, device=device)
    buf.view(torch.int16).fill_(SENTINEL)
    lo = offset_elems + GUARD
    return buf, buf[lo:lo + n].view(shape), lo, n


def _check_guards(buf, lo, n):
    raw = buf.view(torch.int16)
    assert bool((raw[:lo] == SENTINEL).all()), "a store landed before the tensor"
    assert bool((raw[lo + n:] == SENTINEL).all()), "a store landed after the tensor"
    assert not bool((raw[lo:lo + n] == SENTINEL).any()), "an element of the tensor was not written"


@pytest.mark.parametrize("lengths", [[925, 130, 1], [300]])
def test_outputs_at_16_byte_offsets_match_32_byte_aligned_ones(lengths):
    need_gpu()
    from invariant_dit_attention_gb300.h3attn import to_device
    inp = W.make_inputs(lengths, 4, seed=71 + sum(lengths), with_grad=True)
    d = to_device(inp)
    S, H = d["q"].shape[0], d["q"].shape[1]
    h = make_handle(H, S, len(lengths))
    res = {}
    for name, off in (("a32", 16), ("a16", 8)):  # 16 bf16 = 32 bytes past an aligned start; 8 = 16 bytes
        obuf, out, olo, on = _guarded((S, H, 128), off, d["q"].device)
        assert out.data_ptr() % 32 == (0 if name == "a32" else 16)
        out, lse = h.forward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"],
                             out=out)
        grads = {"dq_norm_w": torch.empty(128, dtype=torch.float32, device=out.device),
                 "dk_norm_w": torch.empty(128, dtype=torch.float32, device=out.device)}
        bufs = {}
        for k in ("dq", "dk", "dv"):
            bufs[k] = _guarded((S, H, 128), off, out.device)
            grads[k] = bufs[k][1]
        h.backward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"], out, lse,
                   d["dout"], grads=grads)
        torch.cuda.synchronize()
        h.check()
        _check_guards(obuf, olo, on)
        for k, (b, _, lo, n) in bufs.items():
            _check_guards(b, lo, n)
        res[name] = {"out": out.clone(), "lse": lse.clone(), **{k: grads[k].clone() for k in ("dq", "dk", "dv")}}
    h.close()
    for k in res["a32"]:
        assert torch.equal(res["a32"][k].view(torch.int16) if res["a32"][k].dtype == torch.bfloat16 else res["a32"][k],
                           res["a16"][k].view(torch.int16) if res["a16"][k].dtype == torch.bfloat16 else res["a16"][k]), k
