"""FP64 CPU oracle of the MiniMax-H3 attention core (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
and never touches a GPU.  The arithmetic lives in ``h3ref.c`` (plain C, double
precision, OpenMP over rows); this module compiles it on first use and converts
arguments.

Every function takes the exact values that the GPU path is fed (bf16 tensors
and fp32 norm weights, widened without rounding) and returns float64 arrays.
"""

from __future__ import annotations

import ctypes
import math
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "h3ref.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libh3ref.so")
_lib = None

D = 128


class Params(ctypes.Structure):
    _fields_ = [("sections", ctypes.c_int * 3), ("theta", ctypes.c_double),
                ("eps", ctypes.c_double), ("scale", ctypes.c_double)]


def build(force: bool = False, defines=(), out: str | None = None) -> str:
    """Compile h3ref.c into a shared library (gcc, -O2, OpenMP).

    ``defines``/``out`` build a variant elsewhere (the pin tests use this to plant
    a mistake in a copy and check that some pin catches it).
    """
    path = out or _LIB_PATH
    if (not force and not defines and os.path.exists(path)
            and os.path.getmtime(path) >= os.path.getmtime(_SRC)):
        return path
    os.makedirs(os.path.dirname(path), exist_ok=True)
    tmp = path + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", *[f"-D{d}" for d in defines], _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


def use_library(path: str | None):
    """Bind the module to another build of h3ref.c (None: the default build)."""
    global _lib
    _lib = None if path is None else _bind(ctypes.CDLL(path))


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    fp = ctypes.POINTER(ctypes.c_float)
    ip = ctypes.POINTER(ctypes.c_int32)
    up = ctypes.POINTER(ctypes.c_uint8)
    pp = ctypes.POINTER(Params)
    lib.h3ref_norm_rope.argtypes = [fp, ctypes.c_int, ctypes.c_int, fp, ip, ip, ip, pp, dp, dp, dp]
    lib.h3ref_norm_rope.restype = None
    lib.h3ref_attention.argtypes = [dp, dp, fp, ctypes.c_int, ctypes.c_int, ip, ctypes.c_int,
                                    ctypes.c_double, ctypes.c_int, ctypes.c_int, up, dp, dp]
    lib.h3ref_attention.restype = None
    lib.h3ref_forward.argtypes = [fp, fp, fp, fp, fp, ip, ip, ip, ip, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_int, pp, ctypes.c_int, ctypes.c_int, up, dp, dp]
    lib.h3ref_forward.restype = ctypes.c_int
    lib.h3ref_backward.argtypes = [fp, fp, fp, fp, fp, ip, ip, ip, ip, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, pp, fp, ctypes.c_int, ctypes.c_int,
                                   dp, dp, dp, dp, dp, dp, dp]
    lib.h3ref_backward.restype = ctypes.c_int
    lib.h3ref_num_threads.argtypes = []
    lib.h3ref_num_threads.restype = ctypes.c_int
    return lib


def _f32(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor (bf16 widened exactly to fp32)
        import torch
        x = x.detach().to(torch.float32).cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _params(sections, theta, eps, scale) -> Params:
    p = Params()
    p.sections[:] = list(sections)
    p.theta, p.eps = float(theta), float(eps)
    p.scale = float(1.0 / math.sqrt(D) if scale is None else scale)
    return p


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return int(_load().h3ref_num_threads())


def norm_rope(x, w, pos, sections=(16, 24, 24), theta=10000.0, eps=1e-6):
    """y = RoPE(RMSNorm(x) * w) for x [S, H, 128]; returns (y, n, r) in float64.

    n = x / sqrt(mean x^2 + eps) (before the weight), r = 1 / sqrt(mean x^2 + eps).
    """
    lib = _load()
    x, w, pos = _f32(x), _f32(w), _i32(pos)
    S, H = x.shape[0], x.shape[1]
    y = np.empty((S, H, D)); n = np.empty((S, H, D)); r = np.empty((S, H))
    p = _params(sections, theta, eps, None)
    lib.h3ref_norm_rope(_ptr(x, ctypes.c_float), S, H, _ptr(w, ctypes.c_float),
                        _ptr(pos[0], ctypes.c_int32), _ptr(pos[1], ctypes.c_int32),
                        _ptr(pos[2], ctypes.c_int32), ctypes.byref(p),
                        _ptr(y, ctypes.c_double), _ptr(n, ctypes.c_double), _ptr(r, ctypes.c_double))
    return y, n, r


def attention(yq, yk, v, seg_offsets, scale=None, heads=None, rows=None):
    """Segment-masked softmax attention of already rotated q^, k^ (float64).

    Returns (out [S, H, 128], lse [H, S]); entries of skipped heads/rows are NaN.
    """
    lib = _load()
    yq = np.ascontiguousarray(yq, dtype=np.float64)
    yk = np.ascontiguousarray(yk, dtype=np.float64)
    v, seg = _f32(v), _i32(seg_offsets)
    S, H = yq.shape[0], yq.shape[1]
    h_lo, h_hi = (0, H) if heads is None else heads
    mask = None
    if rows is not None:
        mask = np.zeros(S, dtype=np.uint8)
        mask[np.asarray(rows)] = 1
    out = np.full((S, H, D), np.nan); lse = np.full((H, S), np.nan)
    lib.h3ref_attention(_ptr(yq, ctypes.c_double), _ptr(yk, ctypes.c_double), _ptr(v, ctypes.c_float),
                        S, H, _ptr(seg, ctypes.c_int32), len(seg) - 1,
                        float(1.0 / math.sqrt(D) if scale is None else scale), h_lo, h_hi,
                        None if mask is None else _ptr(mask, ctypes.c_uint8),
                        _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double))
    return out, lse


def forward(q, k, v, q_norm_w, k_norm_w, pos, seg_offsets, sections=(16, 24, 24),
            theta=10000.0, eps=1e-6, scale=None, heads=None, rows=None):
    """Forward of the attention core: returns (out [S, H, 128], lse [H, S]) in float64.

    ``heads`` = (lo, hi) restricts the heads computed, ``rows`` restricts the query
    rows; skipped entries are NaN.
    """
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    wq, wk, pos, seg = _f32(q_norm_w), _f32(k_norm_w), _i32(pos), _i32(seg_offsets)
    S, H = q.shape[0], q.shape[1]
    h_lo, h_hi = (0, H) if heads is None else heads
    mask = None
    if rows is not None:
        mask = np.zeros(S, dtype=np.uint8)
        mask[np.asarray(rows)] = 1
    out = np.full((S, H, D), np.nan); lse = np.full((H, S), np.nan)
    p = _params(sections, theta, eps, scale)
    rc = lib.h3ref_forward(_ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float), _ptr(v, ctypes.c_float),
                           _ptr(wq, ctypes.c_float), _ptr(wk, ctypes.c_float),
                           _ptr(pos[0], ctypes.c_int32), _ptr(pos[1], ctypes.c_int32),
                           _ptr(pos[2], ctypes.c_int32), _ptr(seg, ctypes.c_int32), len(seg) - 1,
                           S, H, ctypes.byref(p), h_lo, h_hi,
                           None if mask is None else _ptr(mask, ctypes.c_uint8),
                           _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc:
        raise MemoryError("oracle forward: allocation failed")
    return out, lse


def backward(q, k, v, q_norm_w, k_norm_w, pos, seg_offsets, dout, sections=(16, 24, 24),
             theta=10000.0, eps=1e-6, scale=None, heads=None):
    """Gradients of sum(out * dout): returns a dict of float64 arrays.

    Keys: dq, dk, dv [S, H, 128]; dq_norm_w, dk_norm_w [128];
    dq_norm_w_per_sample, dk_norm_w_per_sample [n_samples, 128].
    """
    lib = _load()
    q, k, v, do = _f32(q), _f32(k), _f32(v), _f32(dout)
    wq, wk, pos, seg = _f32(q_norm_w), _f32(k_norm_w), _i32(pos), _i32(seg_offsets)
    S, H = q.shape[0], q.shape[1]
    nseg = len(seg) - 1
    h_lo, h_hi = (0, H) if heads is None else heads
    dq = np.full((S, H, D), np.nan); dk = np.full((S, H, D), np.nan); dv = np.full((S, H, D), np.nan)
    dwq = np.zeros(D); dwk = np.zeros(D)
    dwq_s = np.zeros((max(nseg, 1), D)); dwk_s = np.zeros((max(nseg, 1), D))
    p = _params(sections, theta, eps, scale)
    c = ctypes.c_double
    rc = lib.h3ref_backward(_ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float), _ptr(v, ctypes.c_float),
                            _ptr(wq, ctypes.c_float), _ptr(wk, ctypes.c_float),
                            _ptr(pos[0], ctypes.c_int32), _ptr(pos[1], ctypes.c_int32),
                            _ptr(pos[2], ctypes.c_int32), _ptr(seg, ctypes.c_int32), nseg,
                            S, H, ctypes.byref(p), _ptr(do, ctypes.c_float), h_lo, h_hi,
                            _ptr(dq, c), _ptr(dk, c), _ptr(dv, c), _ptr(dwq, c), _ptr(dwk, c),
                            _ptr(dwq_s, c), _ptr(dwk_s, c))
    if rc:
        raise MemoryError("oracle backward: allocation failed")
    return {"dq": dq, "dk": dk, "dv": dv, "dq_norm_w": dwq, "dk_norm_w": dwk,
            "dq_norm_w_per_sample": dwq_s[:nseg], "dk_norm_w_per_sample": dwk_s[:nseg]}


def linear(x, w, bias=None, rows=None):
    """y = x w^T (+ bias) in float64: the block's QKV / output projection either
    side of the attention core ("ws1_one_h3_block" page of RL-Kernel, PR #539,
    Bindings table).  x [rows, in] and w [out, in] as fed to the GPU (bf16,
    widened exactly), bias FP32 [out] or None; ``rows`` selects output rows.
    The product is the library matmul (numpy, float64): the definition itself."""
    xs = _f32(x).astype(np.float64)
    if rows is not None:
        xs = xs[np.asarray(rows)]
    y = xs @ _f32(w).astype(np.float64).T
    if bias is not None:
        y = y + _f32(bias).astype(np.float64)[None, :]
    return y


def _bf16_bits(x) -> np.ndarray:
    """Bit patterns of a bf16 tensor (torch bfloat16, or numpy uint16 already) as
    uint16, one row per token: [S, everything else flattened in memory order]."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().cpu().contiguous()
        if x.dtype != torch.bfloat16:
            raise TypeError("canonical_order: bf16 tensors expected")
        x = x.view(torch.int16).numpy().view(np.uint16)
    x = np.ascontiguousarray(np.asarray(x))
    if x.dtype != np.uint16:
        raise TypeError("canonical_order: bf16 bit patterns (uint16) expected")
    return x.reshape(x.shape[0], -1)


def canonical_order(pos, seg_offsets, k, v, q, dout=None):
    """Canonical order of each sample's tokens, the order in which a
    packing-permutation-invariant attention sums keys (and queries, in the
    backward).  The "ws1_one_h3_block" page of RL-Kernel (PR #539), Results,
    control H-C3, reports that permuting the packed rows of a sample
    together with their positions changes output rows because attention sums
    keys in packed order; an order fixed by the tokens themselves settles it.

    Within each sample the tokens are sorted by
      1. their position (t, h, w), as signed integers, t first;
      2. then their k row, v row, q row and (when given) dout row, each taken
         over all heads in memory order and compared as a sequence of bf16 bit
         patterns read as unsigned 16-bit integers (a total order on bits, not
         the numeric order of the values);
      3. then their packed index (the tokens compared equal here are identical
         in every input, so which comes first changes no result).
    Returns perm (int64 [S]): perm[c] is the packed index of the token in
    canonical slot c; the slots of sample s are seg[s] .. seg[s+1]-1.
    The content comparison only runs inside groups of equal position."""
    pos = _i32(pos)
    seg = [int(x) for x in _i32(seg_offsets)]
    rows = [_bf16_bits(t) for t in (k, v, q) + ((dout,) if dout is not None else ())]
    S = pos.shape[1]
    perm = np.empty(S, dtype=np.int64)
    for s in range(len(seg) - 1):
        a, b = seg[s], seg[s + 1]
        by_pos = sorted(range(a, b), key=lambda i: (int(pos[0, i]), int(pos[1, i]), int(pos[2, i]), i))
        out = []
        g = 0
        while g < len(by_pos):
            e = g
            p0 = tuple(int(pos[ax, by_pos[g]]) for ax in range(3))
            while e < len(by_pos) and tuple(int(pos[ax, by_pos[e]]) for ax in range(3)) == p0:
                e += 1
            group = by_pos[g:e]
            if len(group) > 1:
                # big-endian bytes of uint16 words compare like the words themselves
                group = sorted(group, key=lambda i: tuple(r[i].astype(">u2").tobytes() for r in rows) + (i,))
            out.extend(group)
            g = e
        perm[a:b] = out
    return perm


if __name__ == "__main__":  # `python -m oracle` compiles the library
    print(build(force="--force" in sys.argv))
