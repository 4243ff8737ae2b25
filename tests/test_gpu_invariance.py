"""Bitwise repeatability and batch invariance (alone vs packed), forward and backward.

The defining property of the strict path on the "ws1_full_h3_transformer"
page (RL-Kernel PR #571), rollout-vs-train control: a sample's results are
bitwise identical whether it runs alone (rollout) or packed with others
(train), and from run to run.
"""

import hashlib

import numpy as np
import pytest
import torch

from invariant_dit_attention_gb300 import workloads as W
from tests.helpers import make_handle, need_gpu, workload

pytestmark = pytest.mark.gpu


def _fwd(h, inp):
    from invariant_dit_attention_gb300.h3attn import to_device
    d = to_device(inp)
    out, lse = h.forward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
    return out, lse, d


def _fwd_bwd(h, inp):
    out, lse, d = _fwd(h, inp)
    g = h.backward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"], out, lse,
                   d["dout"])
    return out, lse, g


def _idx(items, x):
    return next(i for i, y in enumerate(items) if y is x)


def _sha(t):
    return hashlib.sha256(t.contiguous().view(torch.uint8).cpu().numpy().tobytes()).hexdigest()


def _fp(t):
    """The library's device-side fingerprint (h3attn_fingerprint) of a tensor."""
    from invariant_dit_attention_gb300.h3attn import fingerprint, fingerprint_value
    return fingerprint_value(fingerprint(t.contiguous()))


@pytest.mark.parametrize("store_ds", [False, True])
def test_backward_alone_vs_packed_both_dq_paths(store_ds):
    """dq, dk, dv and the per-sample weight gradients of each sample, alone and
    packed with others, on both dQ paths (stored dS, recomputed S and dP)."""
    need_gpu()
    from invariant_dit_attention_gb300.h3attn import to_device
    parts = [W.make_inputs([W.SampleLayout(n_text=5, grid=(2, 6, 11), n_audio=4)], 6, seed=41, with_grad=True),
             W.make_inputs([130, 1], 6, seed=42, with_grad=True)]
    packed = W.pack(parts)

    def run(inp):
        h = make_handle(6, inp.total_tokens, 8, store_ds=store_ds)
        d = to_device(inp)
        out, lse = h.forward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
        g = h.backward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"], out, lse,
                       d["dout"])
        torch.cuda.synchronize()
        h.check()
        h.close()
        return {k: v.cpu() for k, v in g.items()}

    gp = run(packed)
    seg = packed.seg_offsets.tolist()
    for s in range(packed.num_samples):
        ga = run(W.slice_sample(packed, s))
        a, b = seg[s], seg[s + 1]
        for name in ("dq", "dk", "dv"):
            assert _sha(ga[name]) == _sha(gp[name][a:b]), f"sample {s} {name}"
        for name in ("dq_norm_w_per_sample", "dk_norm_w_per_sample"):
            assert _sha(ga[name][0]) == _sha(gp[name][s]), f"sample {s} {name}"


def test_many_samples_alone_vs_packed_forward_and_backward():
    """Twelve samples of 1 to 400 tokens packed together: every sample's out, lse,
    dq, dk, dv and per-sample weight gradients are the bits it gets alone."""
    need_gpu()
    from invariant_dit_attention_gb300.h3attn import to_device
    lengths = [int(x) for x in np.random.default_rng(12).integers(1, 401, size=12)]
    packed = W.make_inputs(lengths, 4, seed=12, with_grad=True)

    def run(inp):
        h = make_handle(4, inp.total_tokens, 16)
        d = to_device(inp)
        out, lse = h.forward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
        g = h.backward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"], out, lse,
                       d["dout"])
        torch.cuda.synchronize()
        h.check()
        h.close()
        r = {k: v.cpu() for k, v in g.items()}
        r["out"], r["lse"] = out.cpu(), lse.cpu()
        return r

    rp = run(packed)
    seg = packed.seg_offsets.tolist()
    for s in range(packed.num_samples):
        ra = run(W.slice_sample(packed, s))
        a, b = seg[s], seg[s + 1]
        for name in ("out", "dq", "dk", "dv"):
            assert _sha(ra[name]) == _sha(rp[name][a:b]), f"sample {s} ({lengths[s]} tokens) {name}"
        assert _sha(ra["lse"]) == _sha(rp["lse"][:, a:b].contiguous()), f"sample {s} lse"
        for name in ("dq_norm_w_per_sample", "dk_norm_w_per_sample"):
            assert _sha(ra[name][0]) == _sha(rp[name][s]), f"sample {s} {name}"


def test_forward_repeat_bitwise_925():
    need_gpu()
    w, inp = workload("single_925")
    h = make_handle(w.num_heads, inp.total_tokens)
    digests = set()
    fps = set()
    for _ in range(3):
        out, lse, _ = _fwd(h, inp)
        digests.add((_sha(out), _sha(lse)))
        fps.add((_fp(out), _fp(lse)))  # compared on the device, without copying the outputs back
    h.check()
    assert len(digests) == 1 and len(fps) == 1


def test_forward_alone_vs_packed_13539():
    need_gpu()
    w, inp = workload("packed_13539")
    h = make_handle(w.num_heads, inp.total_tokens)
    out, lse, _ = _fwd(h, inp)
    seg = inp.seg_offsets.tolist()
    for s in range(inp.num_samples):
        a, b = seg[s], seg[s + 1]
        o1, l1, _ = _fwd(h, W.slice_sample(inp, s))
        assert torch.equal(o1, out[a:b]), f"sample {s} out differs"
        assert torch.equal(l1, lse[:, a:b]), f"sample {s} lse differs"
    h.check()


def _packings(parts):
    """Alternative packings of the same samples: reversed, shifted by odd-sized fillers."""
    filler5 = W.make_inputs([5], parts[0].num_heads, seed=99)
    filler77 = W.make_inputs([77], parts[0].num_heads, seed=98)
    yield list(reversed(parts))
    yield [filler5] + parts
    yield [filler77] + list(reversed(parts)) + [filler5]


def test_forward_packing_variants_bitwise():
    need_gpu()
    H = 8
    parts = [W.make_inputs([L], H, seed=10 + L) for L in (300, 129, 64, 1)]
    for p in parts[1:]:  # one model: the same norm weights for every sample
        p.q_norm_w, p.k_norm_w = parts[0].q_norm_w, parts[0].k_norm_w
    h = make_handle(H, 2048, 16)
    alone = [tuple(t.clone() for t in _fwd(h, p)[:2]) for p in parts]
    for packing in _packings(parts):
        packing[0].q_norm_w, packing[0].k_norm_w = parts[0].q_norm_w, parts[0].k_norm_w
        packed = W.pack(packing)
        out, lse, _ = _fwd(h, packed)
        seg = packed.seg_offsets.tolist()
        for i, p in enumerate(packing):
            j = next((j for j, x in enumerate(parts) if x is p), None)
            if j is None:
                continue
            a, b = seg[i], seg[i + 1]
            assert torch.equal(alone[j][0], out[a:b]), f"sample {j} out differs"
            assert torch.equal(alone[j][1], lse[:, a:b]), f"sample {j} lse differs"
    h.check()


def test_forward_nonfinite_neighbour_does_not_leak():
    need_gpu()
    H = 4
    clean = W.make_inputs([200], H, seed=21)
    dirty = W.make_inputs([150], H, seed=22)
    dirty.q[3, 1, 5] = float("nan")
    dirty.k[10] = float("inf")
    dirty.v[0] = float("nan")
    dirty.v[149] = float("-inf")
    dirty.q_norm_w, dirty.k_norm_w = clean.q_norm_w, clean.k_norm_w
    h = make_handle(H, 1024, 8)
    o_alone, l_alone, _ = _fwd(h, clean)
    for packing in ([clean, dirty], [dirty, clean]):
        packed = W.pack(packing)
        out, lse, _ = _fwd(h, packed)
        i = _idx(packing, clean)
        a, b = packed.seg_offsets[i].item(), packed.seg_offsets[i + 1].item()
        assert torch.equal(o_alone, out[a:b])
        assert torch.equal(l_alone, lse[:, a:b])


def test_backward_repeat_and_packed_with_925_bitwise():
    need_gpu()
    w, inp = workload("fwd_bwd_4253")
    w2, s925 = workload("single_925")
    other = W.make_inputs(w2.samples, w.num_heads, seed=77, with_grad=True)
    other.q_norm_w, other.k_norm_w = inp.q_norm_w, inp.k_norm_w
    h = make_handle(w.num_heads, inp.total_tokens + 925, 4)
    runs, fps = [], []
    for _ in range(3):
        _, _, g = _fwd_bwd(h, inp)
        runs.append({k: v.clone() for k, v in g.items()})
        fps.append({k: _fp(v) for k, v in g.items()})
    for r, f in zip(runs[1:], fps[1:]):
        for k in r:
            assert torch.equal(r[k], runs[0][k]), f"repeat differs in {k}"
            assert f[k] == fps[0][k], f"device fingerprint of {k} differs"
    for packing in ([inp, other], [other, inp]):
        packed = W.pack(packing)
        _, _, g = _fwd_bwd(h, packed)
        i = _idx(packing, inp)
        a, b = packed.seg_offsets[i].item(), packed.seg_offsets[i + 1].item()
        for k in ("dq", "dk", "dv"):
            assert torch.equal(g[k][a:b], runs[0][k]), f"packed {k} differs"
        assert torch.equal(g["dq_norm_w_per_sample"][i], runs[0]["dq_norm_w_per_sample"][0])
        assert torch.equal(g["dk_norm_w_per_sample"][i], runs[0]["dk_norm_w_per_sample"][0])
    h.check()
