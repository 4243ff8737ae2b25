"""Pins of the FP64 oracle to facts other than itself (CPU only).

Each test ties one part of the oracle to a library routine it does not call, a
closed form, an invariant, or finite differences, chosen so that a plausible
slip (dropped eps, wrong pair layout, sign of the sine, wrong frequency
exponent, transposed operand, missing scale, cross-sample leakage, wrong chain
rule) fails at least one of them.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from invariant_dit_attention_gb300 import workloads as W

D = 128
SECTIONS = (16, 24, 24)
THETA = 10000.0
EPS = 1e-6


def _rand_inputs(lengths, H, seed, std=1.0):
    layouts = [W.SampleLayout(grid=(1, 1, L)) if i % 2 else W.SampleLayout(n_audio=L)
               for i, L in enumerate(lengths)]
    return W.make_inputs(layouts, H, seed, std=std, with_grad=True)


def _complex_rope(y, pos, sections=SECTIONS, theta=THETA):
    """Rotation written as complex multiplication: (u + i v) * exp(i p f)."""
    y = np.array(y, dtype=np.float64, copy=True)
    off = 0
    for a, n in enumerate(sections):
        half = n // 2
        f = theta ** (-np.arange(0, n, 2, dtype=np.float64) / n)
        ang = np.asarray(pos[a], dtype=np.float64)[:, None] * f[None, :]
        z = y[:, :, off:off + half] + 1j * y[:, :, off + half:off + n]
        z = z * np.exp(1j * ang)[:, None, :]
        y[:, :, off:off + half] = z.real
        y[:, :, off + half:off + n] = z.imag
        off += n
    return y


def _block_mask(seg):
    S = int(seg[-1])
    ids = np.zeros(S, dtype=np.int64)
    for s in range(len(seg) - 1):
        ids[int(seg[s]):int(seg[s + 1])] = s
    return torch.from_numpy(ids[:, None] == ids[None, :])


# ----------------------------------------------------------------- RMSNorm


def test_rmsnorm_matches_torch_rms_norm():
    inp = _rand_inputs([5, 9], 3, seed=11)
    zero = torch.zeros_like(inp.pos)
    y, n, r = oracle.norm_rope(inp.q, inp.q_norm_w, zero)
    x = inp.q.to(torch.float64)
    ref = F.rms_norm(x, (D,), weight=inp.q_norm_w.to(torch.float64), eps=EPS)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)
    ref_n = F.rms_norm(x, (D,), eps=EPS).numpy()
    np.testing.assert_allclose(n, ref_n, rtol=1e-12, atol=1e-12)
    # r is 1/rms: n = x * r
    np.testing.assert_allclose(n, x.numpy() * r[..., None], rtol=1e-13, atol=1e-13)


def test_rmsnorm_scale_invariance_and_constant_vector():
    inp = _rand_inputs([6], 2, seed=12)
    zero = torch.zeros_like(inp.pos)
    x = inp.q.to(torch.float32)
    y1, _, _ = oracle.norm_rope(x, inp.q_norm_w, zero)
    y2, _, _ = oracle.norm_rope(x * 4.0, inp.q_norm_w, zero)
    # eps = 1e-6 against mean squares ~1 and ~16: relative change below 1e-6
    np.testing.assert_allclose(y1, y2, rtol=1e-6, atol=1e-7)
    # constant vector c: output = c / sqrt(c^2 + eps) * w
    c = 0.75
    xc = torch.full((1, 1, D), c)
    w = torch.ones(D)
    yc, _, _ = oracle.norm_rope(xc, w, torch.zeros(3, 1, dtype=torch.int32))
    np.testing.assert_allclose(yc, np.full((1, 1, D), c / math.sqrt(c * c + EPS)), rtol=1e-14)
    # mean of squares of (output / w) is 1 up to eps
    yn, _, _ = oracle.norm_rope(x, torch.ones(D), zero)
    np.testing.assert_allclose((yn ** 2).mean(-1), 1.0, rtol=1e-5)


# -------------------------------------------------------------------- RoPE


def test_rope_identity_at_zero_positions():
    inp = _rand_inputs([7, 4], 2, seed=13)
    zero = torch.zeros_like(inp.pos)
    y, n, _ = oracle.norm_rope(inp.q, inp.q_norm_w, zero)
    np.testing.assert_array_equal(y, n * inp.q_norm_w.double().numpy())


def test_rope_matches_complex_rotation_and_keeps_tail():
    inp = _rand_inputs([11, 6], 3, seed=14)
    pos = torch.randint(0, 120, inp.pos.shape, generator=torch.Generator().manual_seed(3), dtype=torch.int32)
    y, n, _ = oracle.norm_rope(inp.k, inp.k_norm_w, pos)
    z = n * inp.k_norm_w.double().numpy()
    ref = _complex_rope(z, pos.numpy())
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    # channels past the rotary span (64..127) are untouched, bit for bit
    np.testing.assert_array_equal(y[..., 64:], z[..., 64:])


def test_rope_unit_vector_angles():
    """Angle of channel pair (o+j, o+j+n/2) is p * theta^(-2j/n), per axis."""
    offs = np.cumsum([0] + list(SECTIONS))
    for a, n in enumerate(SECTIONS):
        for j in range(n // 2):
            x = torch.zeros(1, 1, D)
            x[0, 0, offs[a] + j] = 1.0
            p = 37
            pos = torch.zeros(3, 1, dtype=torch.int32)
            pos[a, 0] = p
            y, _, _ = oracle.norm_rope(x, torch.ones(D), pos, eps=0.0)
            gain = math.sqrt(D)  # RMSNorm of a one-hot vector scales it by sqrt(128)
            u, v = y[0, 0, offs[a] + j] / gain, y[0, 0, offs[a] + j + n // 2] / gain
            ang = p * THETA ** (-2.0 * j / n)
            assert u == pytest.approx(math.cos(ang), abs=1e-12)
            assert v == pytest.approx(math.sin(ang), abs=1e-12)
            others = np.delete(y[0, 0], [offs[a] + j, offs[a] + j + n // 2])
            assert np.all(others == 0.0)


def test_rope_norm_preserving_and_relative_position():
    inp = _rand_inputs([9], 2, seed=15)
    rng = np.random.default_rng(5)
    pos = torch.from_numpy(rng.integers(0, 50, size=(3, 9)).astype(np.int32))
    shift = torch.from_numpy(rng.integers(-20, 30, size=(3, 1)).astype(np.int32))
    yq0, nq, _ = oracle.norm_rope(inp.q, inp.q_norm_w, pos)
    yk0, _, _ = oracle.norm_rope(inp.k, inp.k_norm_w, pos)
    yq1, _, _ = oracle.norm_rope(inp.q, inp.q_norm_w, pos + shift)
    yk1, _, _ = oracle.norm_rope(inp.k, inp.k_norm_w, pos + shift)
    # every rotated pair keeps its length
    z = nq * inp.q_norm_w.double().numpy()
    offs = np.cumsum([0] + list(SECTIONS))
    for a, n in enumerate(SECTIONS):
        h = n // 2
        lo, hi = offs[a], offs[a] + h
        np.testing.assert_allclose(yq0[..., lo:hi] ** 2 + yq0[..., lo + h:hi + h] ** 2,
                                   z[..., lo:hi] ** 2 + z[..., lo + h:hi + h] ** 2, rtol=1e-12)
    # scores depend only on position differences (shift every axis of every token)
    s0 = np.einsum("ihc,jhc->hij", yq0, yk0)
    s1 = np.einsum("ihc,jhc->hij", yq1, yk1)
    np.testing.assert_allclose(s0, s1, rtol=1e-10, atol=1e-10)


def test_rope_axis_separation():
    """Changing one axis' position changes only that axis' channel section."""
    inp = _rand_inputs([5], 1, seed=16)
    pos = torch.ones(3, 5, dtype=torch.int32) * 3
    y0, _, _ = oracle.norm_rope(inp.q, inp.q_norm_w, pos)
    offs = np.cumsum([0] + list(SECTIONS))
    for a in range(3):
        p2 = pos.clone()
        p2[a] += 7
        y1, _, _ = oracle.norm_rope(inp.q, inp.q_norm_w, p2)
        changed = np.any(y0 != y1, axis=(0, 1))
        expect = np.zeros(D, dtype=bool)
        expect[offs[a]:offs[a + 1]] = True
        np.testing.assert_array_equal(changed, expect)


# --------------------------------------------------------------- attention


def _library_forward(inp, dtype=torch.float64, sections=SECTIONS):
    """RMSNorm (torch), RoPE (complex multiply), masked SDPA (torch), float64."""
    q = F.rms_norm(inp.q.to(dtype), (D,), weight=inp.q_norm_w.to(dtype), eps=EPS)
    k = F.rms_norm(inp.k.to(dtype), (D,), weight=inp.k_norm_w.to(dtype), eps=EPS)
    q = torch.from_numpy(_complex_rope(q.numpy(), inp.pos.numpy(), sections))
    k = torch.from_numpy(_complex_rope(k.numpy(), inp.pos.numpy(), sections))
    mask = _block_mask(inp.seg_offsets.numpy())
    out = F.scaled_dot_product_attention(q.permute(1, 0, 2), k.permute(1, 0, 2),
                                         inp.v.to(dtype).permute(1, 0, 2), attn_mask=mask)
    return out.permute(1, 0, 2).numpy()


def test_attention_matches_torch_sdpa_with_block_mask():
    inp = _rand_inputs([12, 20, 3], 4, seed=17)
    out, lse = oracle.forward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets)
    ref = _library_forward(inp)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_lse_matches_torch_logsumexp():
    inp = _rand_inputs([10, 6], 2, seed=18)
    out, lse = oracle.forward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets)
    yq, _, _ = oracle.norm_rope(inp.q, inp.q_norm_w, inp.pos)
    yk, _, _ = oracle.norm_rope(inp.k, inp.k_norm_w, inp.pos)
    scores = torch.einsum("ihc,jhc->hij", torch.from_numpy(yq), torch.from_numpy(yk)) / math.sqrt(D)
    mask = _block_mask(inp.seg_offsets.numpy())
    ref = torch.logsumexp(scores.masked_fill(~mask, -math.inf), dim=-1).numpy()
    np.testing.assert_allclose(lse, ref, rtol=1e-13)


def test_zero_queries_give_uniform_weights_and_log_length():
    inp = _rand_inputs([5, 8], 2, seed=19)
    qz = torch.zeros_like(inp.q)
    out, lse = oracle.forward(qz, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets)
    v = inp.v.double().numpy()
    for s, (a, b) in enumerate([(0, 5), (5, 13)]):
        np.testing.assert_allclose(lse[:, a:b], math.log(b - a), rtol=1e-14)
        np.testing.assert_allclose(out[a:b], np.broadcast_to(v[a:b].mean(0), out[a:b].shape), rtol=1e-12)


def test_softmax_rows_sum_to_one_and_are_probabilities():
    L, H = 9, 1
    inp = _rand_inputs([L], H, seed=20)
    ones = torch.ones_like(inp.v)
    out, _ = oracle.forward(inp.q, inp.k, ones, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets)
    np.testing.assert_allclose(out, 1.0, rtol=1e-14)
    # one-hot values read the probabilities out: rows are >= 0 and sum to 1
    vi = torch.zeros(L, H, D)
    for j in range(L):
        vi[j, 0, j] = 1.0
    out, _ = oracle.forward(inp.q, inp.k, vi, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets)
    P = out[:, 0, :L]
    assert np.all(P >= 0)
    np.testing.assert_allclose(P.sum(-1), 1.0, rtol=1e-14)
    yq, _, _ = oracle.norm_rope(inp.q, inp.q_norm_w, inp.pos)
    yk, _, _ = oracle.norm_rope(inp.k, inp.k_norm_w, inp.pos)
    sc = torch.from_numpy(yq[:, 0] @ yk[:, 0].T / math.sqrt(D))
    np.testing.assert_allclose(P, torch.softmax(sc, -1).numpy(), rtol=1e-12)


def test_single_token_sample_returns_its_value():
    inp = _rand_inputs([1, 6, 1], 3, seed=21)
    out, lse = oracle.forward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets)
    v = inp.v.double().numpy()
    np.testing.assert_array_equal(out[0], v[0])
    np.testing.assert_array_equal(out[7], v[7])


def test_identical_keys_average_values():
    inp = _rand_inputs([7], 2, seed=22)
    k = inp.k.clone()
    k[:] = k[0]
    pos = torch.zeros_like(inp.pos)  # same position too, so the rotated keys are equal
    out, _ = oracle.forward(inp.q, k, inp.v, inp.q_norm_w, inp.k_norm_w, pos, inp.seg_offsets)
    v = inp.v.double().numpy()
    np.testing.assert_allclose(out, np.broadcast_to(v.mean(0), out.shape), rtol=1e-12, atol=1e-15)


def test_no_leakage_across_segments():
    inp = _rand_inputs([6, 9, 4], 2, seed=23)
    out0, lse0 = oracle.forward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets)
    for t in (inp.q, inp.k, inp.v):
        t[6:15] = float("nan")
    t = inp.k
    t[7, 0, 3] = float("inf")
    out1, lse1 = oracle.forward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets)
    keep = np.r_[0:6, 15:19]
    np.testing.assert_array_equal(out0[keep], out1[keep])
    np.testing.assert_array_equal(lse0[:, keep], lse1[:, keep])


def test_key_value_permutation_equivariance_within_segment():
    inp = _rand_inputs([5, 11], 3, seed=24)
    out0, lse0 = oracle.forward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets)
    perm = np.r_[0:5, 5 + np.random.default_rng(1).permutation(11)]
    # keys and values (with their positions) permuted, queries fixed
    yq, _, _ = oracle.norm_rope(inp.q, inp.q_norm_w, inp.pos)
    yk, _, _ = oracle.norm_rope(inp.k, inp.k_norm_w, inp.pos)
    out1, lse1 = oracle.attention(yq, yk[perm], inp.v[perm], inp.seg_offsets)
    np.testing.assert_allclose(out1, out0, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse1, lse0, rtol=1e-14)
    # permuting whole tokens permutes the outputs
    out2, _ = oracle.forward(inp.q[perm], inp.k[perm], inp.v[perm], inp.q_norm_w, inp.k_norm_w,
                             inp.pos[:, perm], inp.seg_offsets)
    np.testing.assert_allclose(out2, out0[perm], rtol=1e-12, atol=1e-14)


def test_row_and_head_subsets_match_full():
    inp = _rand_inputs([13, 7], 4, seed=25)
    full, lse = oracle.forward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets)
    sub, lsub = oracle.forward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets,
                               heads=(1, 3), rows=[0, 12, 13, 19])
    np.testing.assert_array_equal(sub[[0, 12, 13, 19], 1:3], full[[0, 12, 13, 19], 1:3])
    assert np.isnan(sub[1]).all() and np.isnan(sub[:, 0]).all()


# ---------------------------------------------------------------- backward


def test_backward_matches_torch_autograd_of_library_forward():
    inp = _rand_inputs([6, 10], 3, seed=26)
    g = oracle.backward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets, inp.dout)
    q = inp.q.double().requires_grad_()
    k = inp.k.double().requires_grad_()
    v = inp.v.double().requires_grad_()
    wq = inp.q_norm_w.double().requires_grad_()
    wk = inp.k_norm_w.double().requires_grad_()

    def rope_t(y, pos):
        parts, off = [], 0
        for a, n in enumerate(SECTIONS):
            h = n // 2
            f = THETA ** (-torch.arange(0, n, 2, dtype=torch.float64) / n)
            ang = pos[a].double()[:, None] * f[None, :]
            z = torch.complex(y[..., off:off + h], y[..., off + h:off + n]) * torch.polar(
                torch.ones_like(ang), ang)[:, None, :]
            parts += [z.real, z.imag]
            off += n
        return torch.cat(parts + [y[..., off:]], dim=-1)

    yq = rope_t(F.rms_norm(q, (D,), weight=wq, eps=EPS), inp.pos)
    yk = rope_t(F.rms_norm(k, (D,), weight=wk, eps=EPS), inp.pos)
    mask = _block_mask(inp.seg_offsets.numpy())
    out = F.scaled_dot_product_attention(yq.permute(1, 0, 2), yk.permute(1, 0, 2), v.permute(1, 0, 2),
                                         attn_mask=mask).permute(1, 0, 2)
    (out * inp.dout.double()).sum().backward()
    for name, t in (("dq", q), ("dk", k), ("dv", v), ("dq_norm_w", wq), ("dk_norm_w", wk)):
        np.testing.assert_allclose(g[name], t.grad.numpy(), rtol=1e-9, atol=1e-11, err_msg=name)


def test_backward_matches_central_finite_differences():
    inp = _rand_inputs([4, 5], 2, seed=27)
    args = dict(pos=inp.pos, seg_offsets=inp.seg_offsets)
    tensors = {"q": inp.q.float(), "k": inp.k.float(), "v": inp.v.float(),
               "q_norm_w": inp.q_norm_w.clone(), "k_norm_w": inp.k_norm_w.clone()}
    do = inp.dout.double().numpy()
    g = oracle.backward(tensors["q"], tensors["k"], tensors["v"], tensors["q_norm_w"],
                        tensors["k_norm_w"], inp.pos, inp.seg_offsets, inp.dout)

    def loss(t):
        out, _ = oracle.forward(t["q"], t["k"], t["v"], t["q_norm_w"], t["k_norm_w"], **args)
        return float((out * do).sum())

    h = 2.0 ** -10  # exact in fp32 for |x| < 2^13
    rng = np.random.default_rng(0)
    gkey = {"q": "dq", "k": "dk", "v": "dv", "q_norm_w": "dq_norm_w", "k_norm_w": "dk_norm_w"}
    for name, t in tensors.items():
        flat = t.view(-1)
        idx = rng.choice(flat.numel(), size=min(24, flat.numel()), replace=False)
        for i in idx:
            x0 = float(flat[i])
            flat[i] = x0 + h
            lp = loss(tensors)
            flat[i] = x0 - h
            lm = loss(tensors)
            flat[i] = x0
            fd = (lp - lm) / (2 * h)
            an = g[gkey[name]].reshape(-1)[i]
            assert an == pytest.approx(fd, rel=2e-5, abs=2e-6), (name, int(i))


def test_per_sample_weight_gradients_sum_to_total_and_are_local():
    inp = _rand_inputs([5, 7, 3], 2, seed=28)
    g = oracle.backward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets, inp.dout)
    np.testing.assert_allclose(g["dq_norm_w_per_sample"].sum(0), g["dq_norm_w"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(g["dk_norm_w_per_sample"].sum(0), g["dk_norm_w"], rtol=1e-13, atol=1e-13)
    # a sample's gradients equal those of the sample run alone
    alone = W.slice_sample(inp, 1)
    ga = oracle.backward(alone.q, alone.k, alone.v, alone.q_norm_w, alone.k_norm_w, alone.pos,
                         alone.seg_offsets, alone.dout)
    np.testing.assert_allclose(ga["dq"], g["dq"][5:12], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(ga["dv"], g["dv"][5:12], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(ga["dk_norm_w"], g["dk_norm_w_per_sample"][1], rtol=1e-12, atol=1e-14)


# ------------------------------------------------------ 96-channel rotary span

SECTIONS96 = (32, 32, 32)


def test_rope_96_channel_span_matches_complex_rotation_and_keeps_tail():
    """The pages' own rotary width ("ws1_one_h3_block" page, Tests: 96 of the 128
    channels rotate), as sections 32/32/32: complex rotation on the first 96
    channels, the last 32 untouched."""
    inp = _rand_inputs([10, 7], 3, seed=41)
    pos = torch.randint(0, 90, inp.pos.shape, generator=torch.Generator().manual_seed(9), dtype=torch.int32)
    y, n, _ = oracle.norm_rope(inp.q, inp.q_norm_w, pos, sections=SECTIONS96)
    z = n * inp.q_norm_w.double().numpy()
    np.testing.assert_allclose(y, _complex_rope(z, pos.numpy(), SECTIONS96), rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(y[..., 96:], z[..., 96:])


def test_attention_96_channel_span_matches_torch_sdpa_with_block_mask():
    inp = _rand_inputs([9, 14], 2, seed=42)
    inp.pos = torch.randint(0, 40, inp.pos.shape, generator=torch.Generator().manual_seed(10), dtype=torch.int32)
    out, _ = oracle.forward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos, inp.seg_offsets,
                            sections=SECTIONS96)
    np.testing.assert_allclose(out, _library_forward(inp, sections=SECTIONS96), rtol=1e-11, atol=1e-12)
