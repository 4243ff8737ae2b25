"""Seeded synthetic inputs for the packed MiniMax-H3 attention core.

This module only builds inputs: token layouts, (t, h, w) position ids, segment
offsets and seeded random tensors.  It holds none of the method's arithmetic
(no normalisation, rotation or attention), so both the CUDA path and the FP64
oracle can be fed from it.

Layout of one packed sample (the FL2VA packing named on the ws1_one_h3_block
page, section "What"): text tokens first, then a video grid, then audio tokens.
Positions are 0-based integers:

* text  -> (0, 0, 0) for every token;
* video -> (t, h, w) grid coordinates, t-major, then h, then w;
* audio -> (t, 0, 0) with t = 0, 1, ..., n_audio - 1.

Values are drawn with numpy's PCG64 generator (``default_rng(seed)``) in the
order q, k, v, q_norm_w, k_norm_w, dO, then rounded to bfloat16 (tensors) or
kept as float32 (norm weights).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

HEAD_DIM = 128


@dataclass(frozen=True)
class SampleLayout:
    """Token layout of one sample: text, then a t x h x w video grid, then audio."""

    n_text: int = 0
    grid: tuple = (0, 0, 0)
    n_audio: int = 0

    @property
    def n_video(self) -> int:
        t, h, w = self.grid
        return t * h * w

    @property
    def length(self) -> int:
        return self.n_text + self.n_video + self.n_audio

    def positions(self) -> np.ndarray:
        """int32 array [3, L]: rows are the t, h and w position of each token."""
        pos = np.zeros((3, self.length), dtype=np.int32)
        o = self.n_text
        t, h, w = self.grid
        if self.n_video:
            tt, hh, ww = np.meshgrid(np.arange(t), np.arange(h), np.arange(w), indexing="ij")
            pos[0, o:o + self.n_video] = tt.reshape(-1)
            pos[1, o:o + self.n_video] = hh.reshape(-1)
            pos[2, o:o + self.n_video] = ww.reshape(-1)
        o += self.n_video
        pos[0, o:o + self.n_audio] = np.arange(self.n_audio, dtype=np.int32)
        return pos


# Sample layouts of the five workloads.
TINY_A = SampleLayout(grid=(1, 3, 4))                          # 12 tokens
TINY_B = SampleLayout(grid=(1, 4, 5))                          # 20 tokens
S925 = SampleLayout(n_text=32, grid=(2, 16, 25), n_audio=93)   # 925 tokens
S4253 = SampleLayout(n_text=128, grid=(6, 24, 28), n_audio=93)  # 4253 tokens
S8349 = SampleLayout(n_text=64, grid=(11, 24, 31), n_audio=101)  # 8349 tokens
S12 = SampleLayout(grid=(1, 3, 4))                             # 12 tokens

assert S925.length == 925 and S4253.length == 4253 and S8349.length == 8349


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: samples, heads and value distribution."""

    name: str
    samples: tuple
    num_heads: int
    seed: int
    std: float = 1.0            # q/k/v ~ std * N(0, 1)
    outlier_frac: float = 0.0   # independent per-element Bernoulli mask
    outlier_scale: float = 1.0  # masked entries multiplied by this before rounding
    with_grad: bool = False     # also draw dO ~ N(0, 1)
    rope_sections: tuple = (16, 24, 24)
    rope_theta: float = 10000.0
    eps: float = 1e-6

    @property
    def lengths(self) -> list:
        return [s.length for s in self.samples]

    @property
    def total_tokens(self) -> int:
        return sum(self.lengths)

    def fwd_flops(self) -> float:
        """4 * H * d * sum_s L_s^2: the two per-sample GEMMs QK^T and PV."""
        return 4.0 * self.num_heads * HEAD_DIM * float(sum(L * L for L in self.lengths))


WORKLOADS = {
    "tiny_packed": Workload("tiny_packed", (TINY_A, TINY_B), 4, seed=1001),
    "single_925": Workload("single_925", (S925,), 24, seed=1002),
    "single_4253_outliers": Workload("single_4253_outliers", (S4253,), 48, seed=1003,
                                     std=0.5, outlier_frac=0.01, outlier_scale=20.0),
    "packed_13539": Workload("packed_13539", (S12, S925, S4253, S8349), 48, seed=1004),
    "fwd_bwd_4253": Workload("fwd_bwd_4253", (S4253,), 48, seed=1005,
                             std=0.5, outlier_frac=0.01, outlier_scale=20.0, with_grad=True),
}


@dataclass
class Inputs:
    """Host-side inputs of one workload (CPU tensors)."""

    q: torch.Tensor            # bf16 [S, H, 128]
    k: torch.Tensor            # bf16 [S, H, 128]
    v: torch.Tensor            # bf16 [S, H, 128]
    q_norm_w: torch.Tensor     # f32 [128]
    k_norm_w: torch.Tensor     # f32 [128]
    pos: torch.Tensor          # int32 [3, S] (t, h, w)
    seg_offsets: torch.Tensor  # int32 [n + 1]
    dout: torch.Tensor | None = None  # bf16 [S, H, 128]
    meta: dict = field(default_factory=dict)

    @property
    def total_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def num_samples(self) -> int:
        return int(self.seg_offsets.numel() - 1)


def _draw(rng, shape, std, outlier_frac, outlier_scale):
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if outlier_frac > 0.0:
        mask = rng.random(shape, dtype=np.float32) < outlier_frac
        x[mask] *= np.float32(outlier_scale)
    return torch.from_numpy(x).to(torch.bfloat16)


def make_inputs(samples, num_heads: int, seed: int, std: float = 1.0,
                outlier_frac: float = 0.0, outlier_scale: float = 1.0,
                with_grad: bool = False) -> Inputs:
    """Draw one packed batch for the given sample layouts (or plain lengths)."""
    layouts = [s if isinstance(s, SampleLayout) else SampleLayout(n_text=int(s)) for s in samples]
    lengths = [s.length for s in layouts]
    S = sum(lengths)
    rng = np.random.default_rng(seed)
    shape = (S, num_heads, HEAD_DIM)
    q = _draw(rng, shape, std, outlier_frac, outlier_scale)
    k = _draw(rng, shape, std, outlier_frac, outlier_scale)
    v = _draw(rng, shape, std, outlier_frac, outlier_scale)
    wq = torch.from_numpy((1.0 + 0.1 * rng.standard_normal(HEAD_DIM)).astype(np.float32))
    wk = torch.from_numpy((1.0 + 0.1 * rng.standard_normal(HEAD_DIM)).astype(np.float32))
    dout = None
    if with_grad:
        dout = torch.from_numpy(rng.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)
    pos = torch.from_numpy(np.concatenate([s.positions() for s in layouts], axis=1)
                           if layouts else np.zeros((3, 0), np.int32))
    seg = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32))
    return Inputs(q, k, v, wq, wk, pos.contiguous(), seg, dout,
                  meta={"lengths": lengths, "seed": seed})


def make_workload(name: str) -> tuple:
    """Inputs of one named workload; returns (Workload, Inputs)."""
    w = WORKLOADS[name]
    return w, make_inputs(w.samples, w.num_heads, w.seed, w.std, w.outlier_frac,
                          w.outlier_scale, w.with_grad)


def slice_sample(inp: Inputs, s: int) -> Inputs:
    """Sample ``s`` of a packed batch as a batch of its own (same values)."""
    a, b = int(inp.seg_offsets[s]), int(inp.seg_offsets[s + 1])
    return Inputs(inp.q[a:b].clone(), inp.k[a:b].clone(), inp.v[a:b].clone(),
                  inp.q_norm_w.clone(), inp.k_norm_w.clone(), inp.pos[:, a:b].contiguous(),
                  torch.tensor([0, b - a], dtype=torch.int32),
                  None if inp.dout is None else inp.dout[a:b].clone(),
                  meta={"lengths": [b - a]})


def pack(parts: list) -> Inputs:
    """Concatenate single- or multi-sample batches into one packed batch.

    All parts must share head count and norm weights (the first part's are used).
    """
    lengths = []
    for p in parts:
        lengths += [int(p.seg_offsets[i + 1] - p.seg_offsets[i]) for i in range(p.num_samples)]
    seg = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32))
    dout = None
    if all(p.dout is not None for p in parts):
        dout = torch.cat([p.dout for p in parts])
    return Inputs(torch.cat([p.q for p in parts]), torch.cat([p.k for p in parts]),
                  torch.cat([p.v for p in parts]), parts[0].q_norm_w.clone(),
                  parts[0].k_norm_w.clone(), torch.cat([p.pos for p in parts], dim=1).contiguous(),
                  seg, dout, meta={"lengths": lengths})


def permute_within_samples(inp: Inputs, seed: int) -> tuple:
    """The same batch with each sample's tokens in a seeded random order: every
    per-token input (q, k, v, positions, dout) moves with its token.  Returns
    (permuted Inputs, sigma) with row r of the result = row sigma[r] of ``inp``."""
    rng = np.random.default_rng(seed)
    seg = [int(x) for x in inp.seg_offsets]
    sigma = np.concatenate([a + rng.permutation(b - a) for a, b in zip(seg[:-1], seg[1:])]
                           ) if len(seg) > 1 else np.zeros(0, np.int64)
    idx = torch.from_numpy(sigma.astype(np.int64))
    out = Inputs(inp.q[idx].contiguous(), inp.k[idx].contiguous(), inp.v[idx].contiguous(),
                 inp.q_norm_w.clone(), inp.k_norm_w.clone(), inp.pos[:, idx].contiguous(),
                 inp.seg_offsets.clone(), None if inp.dout is None else inp.dout[idx].contiguous(),
                 meta=dict(inp.meta, permuted_seed=seed))
    return out, sigma
