"""The synthetic input recipe (text, then a t x h x w video grid, then audio
per sample; seeded draws), checked by hand-written expectations on CPU."""

import numpy as np
import torch

from invariant_dit_attention_gb300 import workloads as W


def test_sample_layouts_have_the_stated_lengths():
    assert [s.length for s in (W.S925, W.S4253, W.S8349)] == [925, 4253, 8349]
    assert W.S925.n_text == 32 and W.S925.grid == (2, 16, 25) and W.S925.n_audio == 93
    w = W.WORKLOADS["packed_13539"]
    assert [s.length for s in w.samples] == [12, 925, 4253, 8349] and w.num_heads == 48
    _, inp = W.make_workload("packed_13539")
    assert inp.total_tokens == 13539 and inp.seg_offsets.tolist() == [0, 12, 937, 5190, 13539]


def test_positions_text_then_video_grid_then_audio():
    lay = W.SampleLayout(n_text=2, grid=(2, 2, 3), n_audio=3)
    want = [(0, 0, 0)] * 2
    want += [(t, h, w) for t in range(2) for h in range(2) for w in range(3)]  # t-major, then h, then w
    want += [(t, 0, 0) for t in range(3)]
    assert [tuple(int(x) for x in lay.positions()[:, i]) for i in range(lay.length)] == want


def test_draws_are_seeded_bf16_and_ordered():
    a = W.make_inputs([W.SampleLayout(n_text=5)], 2, seed=9, with_grad=True)
    b = W.make_inputs([W.SampleLayout(n_text=5)], 2, seed=9, with_grad=True)
    c = W.make_inputs([W.SampleLayout(n_text=5)], 2, seed=10, with_grad=True)
    for name in ("q", "k", "v", "dout"):
        x, y = getattr(a, name), getattr(b, name)
        assert x.dtype == torch.bfloat16 and x.shape == (5, 2, 128)
        assert torch.equal(x, y) and not torch.equal(x, getattr(c, name))
    assert a.q_norm_w.dtype == torch.float32 and torch.equal(a.q_norm_w, b.q_norm_w)
    # the draw order is q, k, v, w_q, w_k, dO: q is the generator's first draw
    rng = np.random.default_rng(9)
    q0 = torch.from_numpy(rng.standard_normal((5, 2, 128), dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(q0, a.q)


def test_outlier_workload_mix():
    """0.5 N(0, 1), with about 1% of the elements multiplied by 20."""
    w, inp = W.make_workload("single_4253_outliers")
    x = inp.q.float().abs().flatten()
    # |0.5 N| > 4 happens ~1e-15 of the time, so |x| > 4 counts the outliers
    # with |20 * 0.5 N| > 4, i.e. |N| > 0.4: 0.01 * 0.6892 of the elements
    frac_big = float((x > 4.0).float().mean())
    assert 0.0066 < frac_big < 0.0072
    core = x[x <= 4.0]
    assert abs(float(core.pow(2).mean().sqrt()) - 0.5) < 0.02


def test_pack_and_slice_round_trip():
    inp = W.make_inputs([W.SampleLayout(n_text=3, grid=(1, 2, 2)), 5, W.SampleLayout(n_audio=4)], 3, seed=2,
                        with_grad=True)
    parts = [W.slice_sample(inp, s) for s in range(inp.num_samples)]
    back = W.pack(parts)
    for name in ("q", "k", "v", "dout", "pos", "seg_offsets"):
        assert torch.equal(getattr(back, name), getattr(inp, name)), name


def test_permute_within_samples_moves_whole_tokens():
    inp = W.make_inputs([W.SampleLayout(n_text=6), W.SampleLayout(grid=(1, 3, 3))], 2, seed=4, with_grad=True)
    per, sigma = W.permute_within_samples(inp, seed=1)
    seg = inp.seg_offsets.tolist()
    for a, b in zip(seg[:-1], seg[1:]):
        assert sorted(sigma[a:b].tolist()) == list(range(a, b))
    idx = torch.from_numpy(sigma)
    for name in ("q", "k", "v", "dout"):
        assert torch.equal(getattr(per, name), getattr(inp, name)[idx]), name
    assert torch.equal(per.pos, inp.pos[:, idx])
