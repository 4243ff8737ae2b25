"""Head-sharded runs on one GPU: the heads split into contiguous blocks, each
block run through a handle of its own (as each GPU of a head-sharded run
would), give bitwise the outputs and gradients of one all-heads call; the
norm-weight gradient, gathered as per-(sample, head) partials in head order
and reduced with h3attn_combine_norm_weight_grads, is bitwise the one-call
gradient for every split.  The reduction kernels follow the library's fixed
order, checked bitwise against that order written out in numpy float32."""

import numpy as np
import pytest
import torch

from invariant_dit_attention_gb300 import workloads as W
from invariant_dit_attention_gb300.sharding import head_range
from tests.helpers import make_handle, need_gpu
from tests.test_sharding_cpu import _partials, fixed_order_reduce

pytestmark = pytest.mark.gpu


def _run(inp_dev, H, S, n):
    h = make_handle(H, S, 8)
    d = inp_dev
    out, lse = h.forward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
    g = h.backward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"], out, lse,
                   d["dout"])
    pq, pk = h.norm_weight_grad_partials(n)
    torch.cuda.synchronize()
    h.check()
    return out, lse, g, pq, pk


@pytest.mark.parametrize("world", [2, 3, 5])
def test_head_shards_give_the_one_call_bits(world):
    need_gpu()
    from invariant_dit_attention_gb300.h3attn import combine_norm_weight_grads, to_device
    H = 10
    inp = W.make_inputs([W.S925, 300, 129, 1], H, seed=606, with_grad=True)
    S, n = inp.total_tokens, inp.num_samples
    d = to_device(inp)
    out, lse, g, pq, pk = _run(d, H, S, n)
    outs, lses, grads, parts_q, parts_k = [], [], [], [], []
    for r in range(world):
        lo, hi = head_range(r, world, H)
        dr = dict(d)
        for name in ("q", "k", "v", "dout"):
            dr[name] = d[name][:, lo:hi].contiguous()
        o, l_, gr, a, b = _run(dr, hi - lo, S, n)
        outs.append(o); lses.append(l_); grads.append(gr); parts_q.append(a); parts_k.append(b)
    assert torch.equal(torch.cat(outs, 1), out)
    assert torch.equal(torch.cat(lses, 0), lse)
    for name in ("dq", "dk", "dv"):
        assert torch.equal(torch.cat([gr[name] for gr in grads], 1), g[name]), name
    for name, parts, full in (("dq_norm_w", parts_q, pq), ("dk_norm_w", parts_k, pk)):
        gathered = torch.cat(parts, 1).contiguous()
        assert torch.equal(gathered, full), f"{name}: per-(sample, head) partials"
        per, tot = combine_norm_weight_grads(gathered)
        torch.cuda.synchronize()
        assert torch.equal(tot, g[name]), f"{name}: total"
        assert torch.equal(per, g[name + "_per_sample"][:n]), f"{name}: per sample"


def test_combine_kernel_follows_the_fixed_order_bitwise():
    need_gpu()
    from invariant_dit_attention_gb300.h3attn import combine_norm_weight_grads
    p = _partials(5, 48, 77)
    per, tot = combine_norm_weight_grads(torch.from_numpy(p).cuda())
    torch.cuda.synchronize()
    ref_per, ref_tot = fixed_order_reduce(p)
    assert np.array_equal(per.cpu().numpy().view(np.uint32), ref_per.view(np.uint32))
    assert np.array_equal(tot.cpu().numpy().view(np.uint32), ref_tot.view(np.uint32))


def test_backward_weight_gradient_is_the_fixed_order_reduction_of_its_partials():
    need_gpu()
    from invariant_dit_attention_gb300.h3attn import to_device
    H = 6
    inp = W.make_inputs([300, 129, 1], H, seed=707, with_grad=True)
    d = to_device(inp)
    _, _, g, pq, pk = _run(d, H, inp.total_tokens, inp.num_samples)
    for name, part in (("dq_norm_w", pq), ("dk_norm_w", pk)):
        ref_per, ref_tot = fixed_order_reduce(part.cpu().numpy())
        assert np.array_equal(g[name].cpu().numpy().view(np.uint32), ref_tot.view(np.uint32)), name
        assert np.array_equal(g[name + "_per_sample"].cpu().numpy().view(np.uint32), ref_per.view(np.uint32)), name
