"""Shared helpers of the test suite: error metrics, library handles, oracle cache."""

import functools
import os

import numpy as np
import pytest
import torch

import oracle
from invariant_dit_attention_gb300 import workloads as W

# Tolerances against the FP64 oracle: forward rel-L2 <= 5e-3 and max-abs <= 2e-2
# on the bf16 outputs, backward rel-L2 <= 1e-2.  The lse bound follows from
# rounding q^ and k^ to fp16 (2^-11 relative per element): a score moves by at
# most about 2^-10 |q^||k^| scale, about 1e-3 for unit-RMS heads, and lse moves
# by no more than the largest score shift; 1e-2 leaves room for the outlier
# workloads' larger rows.
FWD_REL_L2 = 5e-3
FWD_MAX_ABS = 2e-2
BWD_REL_L2 = 1e-2
LSE_MAX_ABS = 1e-2


def rel_l2(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm((x - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))


def max_abs_scaled(x, ref):
    """max |x - ref| / max(1, |ref|): the absolute error where outputs are O(1),
    relative beyond (a bf16 output of magnitude 8 is quantised in steps of 1/16)."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(x - ref) / np.maximum(1.0, np.abs(ref))))


def max_abs(x, ref):
    return float(np.max(np.abs(np.asarray(x, np.float64) - np.asarray(ref, np.float64))))


def np64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@functools.lru_cache(maxsize=None)
def lib_built():
    from invariant_dit_attention_gb300 import build
    return build.build()


def make_handle(H, max_tokens, max_samples=64, **kw):
    lib_built()
    from invariant_dit_attention_gb300.h3attn import H3Attn
    return H3Attn(H, max_tokens, max_samples, **kw)


@functools.lru_cache(maxsize=None)
def workload(name):
    return W.make_workload(name)


_oracle_cache = {}


def oracle_forward(key, inp, rows=None):
    k = ("fwd", key, None if rows is None else tuple(rows))
    if k not in _oracle_cache:
        _oracle_cache[k] = oracle.forward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos,
                                          inp.seg_offsets, rows=rows)
    return _oracle_cache[k]


def oracle_backward(key, inp):
    k = ("bwd", key)
    if k not in _oracle_cache:
        _oracle_cache[k] = oracle.backward(inp.q, inp.k, inp.v, inp.q_norm_w, inp.k_norm_w, inp.pos,
                                           inp.seg_offsets, inp.dout)
    return _oracle_cache[k]


def sample_rows(seg, per_sample=24, seed=0):
    """Rows spanning every sample: ends, tile boundaries around 64/128, random."""
    rng = np.random.default_rng(seed)
    rows = set()
    seg = [int(x) for x in seg]
    for a, b in zip(seg[:-1], seg[1:]):
        L = b - a
        for r in (0, 1, L - 1, L - 2, 63, 64, 127, 128, 129, L - 65, (L // 128) * 128 - 1, (L // 128) * 128):
            if 0 <= r < L:
                rows.add(a + r)
        for r in rng.integers(0, L, size=min(per_sample, L)):
            rows.add(a + int(r))
    return sorted(rows)
