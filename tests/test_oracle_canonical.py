"""Pins of the canonical token order (oracle.canonical_order).

The order makes the attention core's sums independent of how a sample's tokens
are packed: the "ws1_one_h3_block" page of RL-Kernel (PR #539), Results,
control H-C3, shows packed-order key sums change output rows when a sample's
rows are permuted with their positions.  The order is: position (t, h, w) as
signed integers, then the k, v, q (and dout) rows as unsigned 16-bit bf16 bit
patterns in memory order, then packed index.

Each pin is a check on an implementation: the oracle passes all of them and a
plausible mistake planted in a copy (ties broken by index, numeric instead of
bit order, axes reversed, samples ignored, dout ignored, only a prefix of the
rows compared) fails at least one."""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from invariant_dit_attention_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "canonical_order_small.json")


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).reshape(t.shape[0], -1)


def _golden_inputs():
    g = json.load(open(GOLDEN))
    S, H = len(g["pos_t"]), g["heads"]
    pos = torch.tensor([g["pos_t"], g["pos_h"], g["pos_w"]], dtype=torch.int32)
    seg = torch.tensor(g["seg_offsets"], dtype=torch.int32)
    t = {}
    for name in ("k", "v", "q", "dout"):
        x = torch.zeros(S, H, 128)
        for tok, ch, val in g["entries"][name]:
            x[tok, 0, ch] = val
        t[name] = x.to(torch.bfloat16)
    return g, pos, seg, t


def _small_batch(seed=11, heads=2):
    # text tokens share position (0, 0, 0): the content decides their order
    layouts = [W.SampleLayout(n_text=6, grid=(1, 2, 3), n_audio=3), W.SampleLayout(n_text=1),
               W.SampleLayout(n_text=5, grid=(2, 1, 2), n_audio=1)]
    return W.make_inputs(layouts, heads, seed=seed, with_grad=True)


def _less_equal(a, b):
    """Independent comparator: element-by-element loop over the sort keys of two
    tokens given as (pos tuple, [uint16 rows]); True if a <= b."""
    if a[0] != b[0]:
        return a[0] < b[0]
    for ra, rb in zip(a[1], b[1]):
        for x, y in zip(ra.tolist(), rb.tolist()):
            if x != y:
                return x < y
    return True


def _token(inp, i, with_dout):
    pos = tuple(int(inp.pos[ax, i]) for ax in range(3))
    rows = [_bits(inp.k)[i], _bits(inp.v)[i], _bits(inp.q)[i]]
    if with_dout:
        rows.append(_bits(inp.dout)[i])
    return pos, rows


def pin_golden(co):
    """The hand-worked example under tests/golden, without and with dout."""
    g, pos, seg, t = _golden_inputs()
    a = co(pos, seg, t["k"], t["v"], t["q"])
    b = co(pos, seg, t["k"], t["v"], t["q"], t["dout"])
    return list(a) == g["perm_without_dout"] and list(b) == g["perm_with_dout"]


def pin_permutation_within_samples(co):
    """Each sample's slots hold exactly that sample's tokens."""
    inp = _small_batch()
    perm = np.asarray(co(inp.pos, inp.seg_offsets, inp.k, inp.v, inp.q))
    seg = [int(x) for x in inp.seg_offsets]
    return all(sorted(perm[a:b].tolist()) == list(range(a, b)) for a, b in zip(seg[:-1], seg[1:]))


def pin_sorted(co):
    """Adjacent slots are in order under an element-by-element comparator."""
    inp = _small_batch(seed=12)
    for with_dout in (False, True):
        perm = co(inp.pos, inp.seg_offsets, inp.k, inp.v, inp.q, inp.dout if with_dout else None)
        seg = [int(x) for x in inp.seg_offsets]
        for a, b in zip(seg[:-1], seg[1:]):
            for c in range(a, b - 1):
                if not _less_equal(_token(inp, perm[c], with_dout), _token(inp, perm[c + 1], with_dout)):
                    return False
    return True


def _canonical_content(inp, perm, with_dout):
    parts = [inp.pos[:, perm].numpy().T.astype(np.int64)]
    for t in (inp.k, inp.v, inp.q) + ((inp.dout,) if with_dout else ()):
        parts.append(_bits(t)[perm].astype(np.int64))
    return np.concatenate(parts, axis=1)


def pin_invariance(co):
    """Permuting a sample's tokens (with their positions) leaves the canonical
    sequence of token contents unchanged, bit for bit."""
    inp = _small_batch(seed=13)
    for with_dout in (False, True):
        base = _canonical_content(inp, co(inp.pos, inp.seg_offsets, inp.k, inp.v, inp.q,
                                          inp.dout if with_dout else None), with_dout)
        for seed in (1, 2, 3):
            pin, _ = W.permute_within_samples(inp, seed)
            perm = co(pin.pos, pin.seg_offsets, pin.k, pin.v, pin.q, pin.dout if with_dout else None)
            if not np.array_equal(_canonical_content(pin, perm, with_dout), base):
                return False
    return True


def pin_late_difference(co):
    """Tokens equal in position and in all rows but the last q element are still
    put in one order whatever their packed order."""
    S, H = 8, 2
    base = W.make_inputs([W.SampleLayout(n_text=1)], H, seed=5)
    q = base.q.repeat(S, 1, 1).clone()
    k, v = base.k.repeat(S, 1, 1).clone(), base.v.repeat(S, 1, 1).clone()
    q[:, H - 1, 127] = torch.arange(S, dtype=torch.float32).to(torch.bfloat16)
    inp = W.Inputs(q, k, v, base.q_norm_w, base.k_norm_w, torch.zeros(3, S, dtype=torch.int32),
                   torch.tensor([0, S], dtype=torch.int32))
    want = _canonical_content(inp, co(inp.pos, inp.seg_offsets, inp.k, inp.v, inp.q), False)
    for seed in (4, 5):
        pin, _ = W.permute_within_samples(inp, seed)
        if not np.array_equal(_canonical_content(pin, co(pin.pos, pin.seg_offsets, pin.k, pin.v, pin.q),
                                                 False), want):
            return False
    return True


PINS = (pin_golden, pin_permutation_within_samples, pin_sorted, pin_invariance, pin_late_difference)


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_canonical_order_passes_pin(pin):
    assert pin(oracle.canonical_order)


def _planted(kind):
    """A copy of the canonical order with one mistake."""
    def co(pos, seg_offsets, k, v, q, dout=None):
        pos = np.asarray(pos, dtype=np.int64)
        seg = [int(x) for x in seg_offsets]
        rows = [_bits(t) for t in (k, v, q) + ((dout,) if dout is not None and kind != "ignores_dout" else ())]
        if kind == "numeric_order":
            rows = [t.contiguous().float().numpy().reshape(t.shape[0], -1)
                    for t in (k, v, q) + ((dout,) if dout is not None else ())]
        if kind == "prefix_only":
            rows = [r[:, :2] for r in rows]
        axes = (2, 1, 0) if kind == "axes_reversed" else (0, 1, 2)

        def key(i):
            p = tuple(int(pos[a, i]) for a in axes)
            if kind == "index_ties":
                return p + (i,)
            return p + tuple(tuple(r[i].tolist()) for r in rows) + (i,)
        if kind == "ignores_samples":
            return np.asarray(sorted(range(pos.shape[1]), key=key))
        perm = []
        for a, b in zip(seg[:-1], seg[1:]):
            perm += sorted(range(a, b), key=key)
        return np.asarray(perm)
    return co


PLANTS = ("index_ties", "numeric_order", "axes_reversed", "ignores_samples", "ignores_dout", "prefix_only")


def test_planted_copy_without_mistake_passes_every_pin():
    co = _planted("none")
    assert all(pin(co) for pin in PINS)


@pytest.mark.parametrize("kind", PLANTS)
def test_planted_mistake_fails_a_pin(kind):
    co = _planted(kind)
    failed = [pin.__name__ for pin in PINS if not pin(co)]
    assert failed, f"no pin caught the planted mistake {kind}"


def test_full_size_pack_order_is_within_samples_and_sorted_by_position():
    """The 13539-token pack (12 + 925 + 4253 + 8349): slots stay inside their
    samples and positions are non-decreasing; ties only among text tokens."""
    _, inp = W.make_workload("packed_13539")
    perm = oracle.canonical_order(inp.pos, inp.seg_offsets, inp.k, inp.v, inp.q)
    seg = [int(x) for x in inp.seg_offsets]
    pos = inp.pos.numpy().astype(np.int64)
    for a, b in zip(seg[:-1], seg[1:]):
        sl = perm[a:b]
        assert sorted(sl.tolist()) == list(range(a, b))
        keys = [tuple(pos[:, i]) for i in sl]
        assert keys == sorted(keys)
