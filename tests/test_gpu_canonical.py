"""The canonical key order (H3ATTN_KEY_ORDER_CANONICAL) on the GPU.

Control H-C3 in the Results of the "ws1_one_h3_block" page of RL-Kernel
(PR #539): permuting a sample's packed rows together with their positions
changes output rows when attention sums keys in packed order.  With the
canonical order every output bit must be independent of that permutation,
while results stay within the oracle's tolerances, stay identical alone vs
packed, and the order itself must equal the oracle's exactly (integer work).
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from invariant_dit_attention_gb300 import workloads as W
from tests.helpers import (BWD_REL_L2, FWD_MAX_ABS, FWD_REL_L2, LSE_MAX_ABS, make_handle, max_abs, max_abs_scaled,
                           need_gpu, np64, oracle_backward, oracle_forward, rel_l2, workload)

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "canonical_order_small.json")
GRADS = ("dq", "dk", "dv")
WGRADS = ("dq_norm_w", "dk_norm_w", "dq_norm_w_per_sample", "dk_norm_w_per_sample")


def _run(inp, key_order="canonical", backward=True, max_samples=64, store_ds="auto"):
    from invariant_dit_attention_gb300.h3attn import to_device
    h = make_handle(inp.num_heads, max(inp.total_tokens, 1), max_samples, key_order=key_order, store_ds=store_ds)
    d = to_device(inp)
    out, lse = h.forward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"])
    g = None
    if backward:
        g = h.backward(d["q"], d["k"], d["v"], d["q_norm_w"], d["k_norm_w"], d["pos"], d["seg_offsets"], out, lse,
                       d["dout"])
    torch.cuda.synchronize()
    h.check()
    res = {"out": out.cpu(), "lse": lse.cpu()}
    if g is not None:
        res.update({k: v.cpu() for k, v in g.items()})
    h.close()
    return res


def _gpu_order(inp, with_dout):
    from invariant_dit_attention_gb300.h3attn import to_device
    h = make_handle(inp.num_heads, max(inp.total_tokens, 1), 64)
    d = to_device(inp)
    perm = h.canonical_order(d["q"], d["k"], d["v"], d["pos"], d["seg_offsets"],
                             dout=d["dout"] if with_dout else None)
    torch.cuda.synchronize()
    h.check()
    h.close()
    return perm.cpu().numpy().astype(np.int64)


def _same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def _ties_batch():
    """Two text-only samples (every position (0, 0, 0)): the rows decide the
    order, with tokens whose k rows agree and tokens duplicated exactly."""
    inp = W.make_inputs([W.SampleLayout(n_text=40), W.SampleLayout(n_text=9)], 3, seed=77, with_grad=True)
    q, k, v, do = inp.q.clone(), inp.k.clone(), inp.v.clone(), inp.dout.clone()
    k[5] = k[3]            # equal k rows: v decides
    k[6], v[6] = k[3], v[3]  # equal k and v rows: q decides
    for src, dst in ((1, 30), (2, 31), (44, 47)):  # exact duplicates (all inputs)
        q[dst], k[dst], v[dst], do[dst] = q[src], k[src], v[src], do[src]
    return W.Inputs(q, k, v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets, do, meta=inp.meta)


def test_order_matches_the_hand_worked_fixture():
    need_gpu()
    g = json.load(open(GOLDEN))
    S = len(g["pos_t"])
    t = {}
    for name in ("k", "v", "q", "dout"):
        x = torch.zeros(S, g["heads"], 128)
        for tok, ch, val in g["entries"][name]:
            x[tok, 0, ch] = val
        t[name] = x.to(torch.bfloat16)
    inp = W.Inputs(t["q"], t["k"], t["v"], torch.ones(128), torch.ones(128),
                   torch.tensor([g["pos_t"], g["pos_h"], g["pos_w"]], dtype=torch.int32),
                   torch.tensor(g["seg_offsets"], dtype=torch.int32), t["dout"])
    assert _gpu_order(inp, False).tolist() == g["perm_without_dout"]
    assert _gpu_order(inp, True).tolist() == g["perm_with_dout"]


@pytest.mark.parametrize("case", ["tiny_packed", "single_925", "ties", "packed_13539"])
def test_order_equals_oracle(case):
    need_gpu()
    if case == "ties":
        inp = _ties_batch()
    else:
        w, base = workload(case)
        inp = W.make_inputs(w.samples, w.num_heads, w.seed, w.std, w.outlier_frac, w.outlier_scale,
                            with_grad=True)
    for with_dout in (False, True):
        want = oracle.canonical_order(inp.pos, inp.seg_offsets, inp.k, inp.v, inp.q,
                                      inp.dout if with_dout else None)
        got = _gpu_order(inp, with_dout)
        assert np.array_equal(got, want), f"{case} dout={with_dout}: {int((got != want).sum())} slots differ"


@pytest.mark.parametrize("case", ["tiny_packed", "single_925"])
def test_canonical_parity_with_oracle(case):
    need_gpu()
    w, base = workload(case)
    inp = W.make_inputs(w.samples, w.num_heads, w.seed, with_grad=True)
    r = _run(inp)
    out_ref, lse_ref = oracle_forward(("canon_fwd", case), inp)
    assert rel_l2(np64(r["out"]), out_ref) <= FWD_REL_L2
    assert max_abs_scaled(np64(r["out"]), out_ref) <= FWD_MAX_ABS
    assert max_abs(np64(r["lse"]), lse_ref) <= LSE_MAX_ABS
    ref = oracle_backward(("canon_bwd", case), inp)
    for name in GRADS + ("dq_norm_w", "dk_norm_w"):
        e = rel_l2(np64(r[name]), ref[name])
        assert e <= BWD_REL_L2, f"{name} rel-L2 {e:.3e}"
    for name in ("dq_norm_w_per_sample", "dk_norm_w_per_sample"):
        e = rel_l2(np64(r[name])[:inp.num_samples], ref[name])
        assert e <= BWD_REL_L2, f"{name} rel-L2 {e:.3e}"


def _invariance_cases():
    return ["tiny_packed", "single_925", "ties", "ragged"]


def _case_inputs(case):
    if case == "ties":
        return _ties_batch()
    if case == "ragged":
        return W.make_inputs([W.SampleLayout(n_text=7, grid=(2, 5, 13), n_audio=3), W.SampleLayout(n_text=1),
                              W.SampleLayout(n_text=33, grid=(1, 8, 9))], 6, seed=99, with_grad=True)
    w, _ = workload(case)
    return W.make_inputs(w.samples, w.num_heads, w.seed, w.std, w.outlier_frac, w.outlier_scale, with_grad=True)


def _check_invariant(base, inp, seeds, store_ds="auto"):
    for seed in seeds:
        pin, sigma = W.permute_within_samples(inp, seed)
        r = _run(pin, store_ds=store_ds)
        idx = torch.from_numpy(sigma)
        assert _same_bits(r["out"], base["out"][idx]), f"out, permutation {seed}"
        assert _same_bits(r["lse"], base["lse"][:, idx]), f"lse, permutation {seed}"
        for name in GRADS:
            assert _same_bits(r[name], base[name][idx]), f"{name}, permutation {seed}"
        for name in WGRADS:
            assert _same_bits(r[name], base[name]), f"{name}, permutation {seed}"


@pytest.mark.parametrize("case", _invariance_cases())
def test_canonical_results_do_not_depend_on_the_packed_order(case):
    need_gpu()
    inp = _case_inputs(case)
    _check_invariant(_run(inp), inp, (1, 2))


def test_canonical_invariance_with_dq_recomputing_s_and_dp():
    """The same property on the dQ path that recomputes S and dP (store_ds off)."""
    need_gpu()
    inp = _case_inputs("ragged")
    _check_invariant(_run(inp, store_ds=False), inp, (1,), store_ds=False)


def test_packed_order_does_depend_on_it():
    """The control itself: with the packed order, permuting the 925-token
    sample's rows changes output bits (the pages saw 79 to 2199 rows move)."""
    need_gpu()
    inp = _case_inputs("single_925")
    base = _run(inp, key_order="packed")
    pin, sigma = W.permute_within_samples(inp, 1)
    r = _run(pin, key_order="packed")
    a = r["out"].view(torch.int16).reshape(inp.total_tokens, -1)
    b = base["out"][torch.from_numpy(sigma)].view(torch.int16).reshape(inp.total_tokens, -1)
    changed = int((a != b).any(dim=1).sum())
    print(f"packed order: {changed} of {inp.total_tokens} output rows changed")
    assert changed > 0


def test_canonical_alone_vs_packed_bitwise():
    need_gpu()
    parts = [_case_inputs("ragged"), _case_inputs("tiny_packed")]
    parts[1] = W.make_inputs(W.WORKLOADS["tiny_packed"].samples, 6, seed=5, with_grad=True)
    packed = W.pack(parts)
    rp = _run(packed)
    seg = packed.seg_offsets.tolist()
    for s in range(packed.num_samples):
        a, b = seg[s], seg[s + 1]
        alone = W.slice_sample(packed, s)
        ra = _run(alone)
        assert _same_bits(ra["out"], rp["out"][a:b]), f"sample {s} out"
        assert _same_bits(ra["lse"], rp["lse"][:, a:b]), f"sample {s} lse"
        for name in GRADS:
            assert _same_bits(ra[name], rp[name][a:b]), f"sample {s} {name}"
        for name in ("dq_norm_w_per_sample", "dk_norm_w_per_sample"):
            assert _same_bits(ra[name][0], rp[name][s]), f"sample {s} {name}"


def test_duplicate_tokens_get_identical_results():
    need_gpu()
    inp = _ties_batch()
    r = _run(inp)
    for x, y in ((1, 30), (2, 31)):
        for name in ("out",) + GRADS:
            assert _same_bits(r[name][x], r[name][y]), f"{name} of duplicates {x}, {y}"
        assert _same_bits(r["lse"][:, x], r["lse"][:, y])


def test_full_size_13539_canonical():
    """The 12 + 925 + 4253 + 8349 pack at H = 48: forward parity on sampled rows
    and bitwise invariance of forward and backward under one permutation."""
    need_gpu()
    w, base = workload("packed_13539")
    inp = W.make_inputs(w.samples, w.num_heads, w.seed, with_grad=True)
    r = _run(inp)
    rows = np.random.default_rng(0).choice(inp.total_tokens, 48, replace=False)
    rows.sort()
    out_ref, lse_ref = oracle_forward(("canon_13539", "rows"), inp, rows=rows)
    got = np64(r["out"])[rows]
    assert rel_l2(got, out_ref[rows]) <= FWD_REL_L2
    assert max_abs_scaled(got, out_ref[rows]) <= FWD_MAX_ABS
    assert max_abs(np64(r["lse"])[:, rows], lse_ref[:, rows]) <= LSE_MAX_ABS
    _check_invariant(r, inp, (3,))
