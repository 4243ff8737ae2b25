"""Python binding of libh3attn.so (include/h3attn.h): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
passes device pointers of torch tensors and the current CUDA stream, and turns
non-OK status codes into exceptions.  There is no fallback: if the library is
missing or the device is not an sm_103 GPU, calls raise.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libh3attn.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CAPACITY, ERR_CUDA, ERR_TIMEOUT = range(6)

# Entry points declared in include/h3attn.h.
EXPORTS = ("h3attn_create", "h3attn_destroy", "h3attn_forward", "h3attn_backward",
           "h3attn_device_status", "h3attn_set_stage_timing", "h3attn_stage_times", "h3attn_forward_static",
           "h3attn_linear", "h3attn_canonical_order", "h3attn_qkv_forward", "h3attn_debug_stall",
           "h3attn_norm_weight_grad_partials", "h3attn_combine_norm_weight_grads", "h3attn_fingerprint",
           "h3attn_debug_exp2", "h3attn_status_string")

# Limits of h3attn_forward_static's built-in scratch (include/h3attn.h).
STATIC_MAX_TOKEN_HEADS = 131072
STATIC_MAX_SAMPLES = 2048

STAGES = ("plan", "prologue", "fwd", "bwd_delta", "bwd_dkdv", "bwd_dq", "bwd_dw", "bwd_rows", "order", "permute",
          "qkv")

# Key orders (include/h3attn.h, H3ATTN_KEY_ORDER_*).
KEY_ORDERS = {"packed": 0, "canonical": 1}

# Test hook h3attn_debug_stall (include/h3attn.h, H3ATTN_STALL_*): kernels and roles.
STALL_KERNELS = {"fwd": 1, "dkdv": 2, "dq": 3, "qkv": 4}
STALL_ROLES = {"producer": 1, "mma": 2, "consumer": 3}


class H3AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class Config(ctypes.Structure):
    _fields_ = [("num_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float), ("rope_sections", ctypes.c_int * 3),
                ("rope_pairing", ctypes.c_int), ("softmax_scale", ctypes.c_float),
                ("max_tokens", ctypes.c_int), ("max_samples", ctypes.c_int), ("key_order", ctypes.c_int),
                ("store_ds", ctypes.c_int), ("reuse_qk_hat", ctypes.c_int)]


def stored_ds_bytes(num_heads: int, max_tokens: int, max_samples: int) -> int:
    """Workspace of the stored dS blocks (include/h3attn.h, store_ds)."""
    t128 = (max_tokens + 127) // 128
    return num_heads * t128 * (t128 + max_samples) * 128 * 128 * 2


# store_ds="auto" turns the stored dS on while its workspace stays below this.
STORED_DS_AUTO_LIMIT = 32 << 30


_lib = None


def load_library(path: str = LIB_PATH):
    """Loads libh3attn.so (built by invariant_dit_attention_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libh3attn.so not built at {path}; run invariant_dit_attention_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    lib.h3attn_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(vp)]
    lib.h3attn_create.restype = i32
    lib.h3attn_destroy.argtypes = [vp]
    lib.h3attn_destroy.restype = i32
    lib.h3attn_forward.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.POINTER(vp), vp, i32, i32, vp, vp, vp]
    lib.h3attn_forward.restype = i32
    lib.h3attn_backward.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.POINTER(vp), vp, i32, i32, vp, vp, vp,
                                    vp, vp, vp, vp, vp, vp, vp, vp]
    lib.h3attn_backward.restype = i32
    lib.h3attn_device_status.argtypes = [vp, vp]
    lib.h3attn_device_status.restype = i32
    lib.h3attn_set_stage_timing.argtypes = [vp, i32]
    lib.h3attn_set_stage_timing.restype = i32
    lib.h3attn_stage_times.argtypes = [vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(i32), i32]
    lib.h3attn_stage_times.restype = i32
    lib.h3attn_forward_static.argtypes = [ctypes.POINTER(Config), vp, vp, vp, vp, vp, ctypes.POINTER(vp), vp,
                                          i32, i32, vp, vp, vp, vp]
    lib.h3attn_forward_static.restype = i32
    lib.h3attn_linear.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp, vp]
    lib.h3attn_linear.restype = i32
    lib.h3attn_canonical_order.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(vp), vp, i32, i32, vp, vp]
    lib.h3attn_canonical_order.restype = i32
    lib.h3attn_qkv_forward.argtypes = [vp, vp, i32, vp, vp, vp, vp, ctypes.POINTER(vp), vp, i32, i32, vp, vp, vp, vp,
                                       vp, vp]
    lib.h3attn_qkv_forward.restype = i32
    lib.h3attn_norm_weight_grad_partials.argtypes = [vp, vp, vp, vp]
    lib.h3attn_norm_weight_grad_partials.restype = i32
    lib.h3attn_combine_norm_weight_grads.argtypes = [vp, i32, i32, vp, vp, vp]
    lib.h3attn_combine_norm_weight_grads.restype = i32
    lib.h3attn_fingerprint.argtypes = [vp, ctypes.c_uint64, vp, vp]
    lib.h3attn_fingerprint.restype = i32
    lib.h3attn_debug_exp2.argtypes = [vp, vp, i32, i32, vp]
    lib.h3attn_debug_exp2.restype = i32
    lib.h3attn_debug_stall.argtypes = [vp, i32, i32, ctypes.c_longlong]
    lib.h3attn_debug_stall.restype = i32
    lib.h3attn_status_string.argtypes = [i32]
    lib.h3attn_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().h3attn_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != OK:
        raise H3AttnError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _pos_array(pos):
    arr = (ctypes.c_void_p * 3)()
    for a in range(3):
        arr[a] = pos[a].data_ptr()
    return arr


class H3Attn:
    """A handle of the library: configuration plus its bounded device workspace."""

    def __init__(self, num_heads: int, max_tokens: int, max_samples: int = 64, eps: float = 1e-6,
                 rope_theta: float = 10000.0, rope_sections=(16, 24, 24), softmax_scale: float = 0.0,
                 key_order: str = "packed", store_ds="auto", reuse_qk_hat: bool = True):
        """``key_order``: "packed" sums over a sample's tokens in memory order,
        "canonical" in an order fixed by the tokens themselves, so that results
        do not depend on how each sample's tokens are permuted.
        ``store_ds``: True keeps dS from the dK/dV kernel for the dQ kernel (see
        ``stored_ds_bytes`` for its workspace), False recomputes it, "auto"
        stores it while the workspace stays under STORED_DS_AUTO_LIMIT.
        ``reuse_qk_hat``: the backward reuses the rotated q^/k^ rows that the
        handle's last forward computed from the same tensors (their contents
        must not change in between, as a training step's saved tensors do not);
        False recomputes them in every backward."""
        lib = load_library()
        if key_order not in KEY_ORDERS:
            raise ValueError(f"key_order must be one of {sorted(KEY_ORDERS)}")
        cfg = Config()
        cfg.num_heads, cfg.head_dim, cfg.eps, cfg.rope_theta = num_heads, 128, eps, rope_theta
        cfg.rope_sections[:] = list(rope_sections)
        cfg.rope_pairing, cfg.softmax_scale = 0, softmax_scale
        cfg.max_tokens, cfg.max_samples = max_tokens, max_samples
        cfg.key_order = KEY_ORDERS[key_order]
        if store_ds == "auto":
            store_ds = stored_ds_bytes(num_heads, max_tokens, max_samples) <= STORED_DS_AUTO_LIMIT
        cfg.store_ds = 1 if store_ds else 0
        cfg.reuse_qk_hat = 1 if reuse_qk_hat else 0
        self.store_ds = bool(store_ds)
        h = ctypes.c_void_p()
        _check(lib.h3attn_create(ctypes.byref(cfg), ctypes.byref(h)), "h3attn_create")
        self._h = h
        self._lib = lib
        self.num_heads = num_heads
        self.scale = softmax_scale if softmax_scale else 1.0 / math.sqrt(128)
        self.key_order = key_order

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.h3attn_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, q, k, v, q_norm_w, k_norm_w, pos, seg_offsets, num_samples=None,
                out=None, lse=None, want_lse=True, stream=None):
        """out = attention core forward; returns (out, lse or None). Tensors on the device."""
        S, H = q.shape[0], q.shape[1]
        n = int(seg_offsets.numel() - 1) if num_samples is None else num_samples
        if out is None:
            out = torch.empty_like(q)
        if lse is None and want_lse:
            lse = torch.empty((H, S), dtype=torch.float32, device=q.device)
        st = self._lib.h3attn_forward(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(q_norm_w), _ptr(k_norm_w),
                                      _pos_array(pos), _ptr(seg_offsets), n, S, _ptr(out), _ptr(lse),
                                      _stream(stream))
        _check(st, "h3attn_forward")
        return out, lse

    def backward(self, q, k, v, q_norm_w, k_norm_w, pos, seg_offsets, out, lse, dout, num_samples=None,
                 grads=None, per_sample=True, stream=None):
        """Returns a dict: dq, dk, dv, dq_norm_w, dk_norm_w (+ per-sample weight gradients)."""
        S = q.shape[0]
        n = int(seg_offsets.numel() - 1) if num_samples is None else num_samples
        dev = q.device
        if grads is None:
            grads = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
                     "dq_norm_w": torch.empty(128, dtype=torch.float32, device=dev),
                     "dk_norm_w": torch.empty(128, dtype=torch.float32, device=dev)}
            if per_sample:
                grads["dq_norm_w_per_sample"] = torch.empty((max(n, 1), 128), dtype=torch.float32, device=dev)
                grads["dk_norm_w_per_sample"] = torch.empty((max(n, 1), 128), dtype=torch.float32, device=dev)
        st = self._lib.h3attn_backward(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(q_norm_w), _ptr(k_norm_w),
                                       _pos_array(pos), _ptr(seg_offsets), n, S, _ptr(out), _ptr(lse),
                                       _ptr(dout), _ptr(grads["dq"]), _ptr(grads["dk"]), _ptr(grads["dv"]),
                                       _ptr(grads["dq_norm_w"]), _ptr(grads["dk_norm_w"]),
                                       _ptr(grads.get("dq_norm_w_per_sample")),
                                       _ptr(grads.get("dk_norm_w_per_sample")), _stream(stream))
        _check(st, "h3attn_backward")
        return grads

    def qkv_forward(self, x, w_qkv, b_qkv, q_norm_w, k_norm_w, pos, seg_offsets, num_samples=None, q=None, k=None,
                    v=None, out=None, lse=None, want_lse=True, stream=None):
        """h3attn_qkv_forward: [q | k | v] = x w_qkv^T (+ b_qkv) with the q/k norm and
        RoPE fused into the projection, then the attention forward.  x bf16 [S, in],
        w_qkv bf16 [3 H 128, in] (q, k, v heads).  Returns (q, k, v, out, lse)."""
        S = x.shape[0]
        H = self.num_heads
        n = int(seg_offsets.numel() - 1) if num_samples is None else num_samples
        dev = x.device
        q = torch.empty((S, H, 128), dtype=torch.bfloat16, device=dev) if q is None else q
        k = torch.empty((S, H, 128), dtype=torch.bfloat16, device=dev) if k is None else k
        v = torch.empty((S, H, 128), dtype=torch.bfloat16, device=dev) if v is None else v
        out = torch.empty((S, H, 128), dtype=torch.bfloat16, device=dev) if out is None else out
        if lse is None and want_lse:
            lse = torch.empty((H, S), dtype=torch.float32, device=dev)
        st = self._lib.h3attn_qkv_forward(self._h, _ptr(x), x.shape[1], _ptr(w_qkv), _ptr(b_qkv), _ptr(q_norm_w),
                                          _ptr(k_norm_w), _pos_array(pos), _ptr(seg_offsets), n, S, _ptr(q), _ptr(k),
                                          _ptr(v), _ptr(out), _ptr(lse), _stream(stream))
        _check(st, "h3attn_qkv_forward")
        return q, k, v, out, lse

    def canonical_order(self, q, k, v, pos, seg_offsets, dout=None, num_samples=None, perm=None, stream=None):
        """h3attn_canonical_order: int32 [S] device tensor, perm[c] = packed index
        of the token in canonical slot c (dout joins the sort when given)."""
        S = q.shape[0]
        n = int(seg_offsets.numel() - 1) if num_samples is None else num_samples
        if perm is None:
            perm = torch.empty(S, dtype=torch.int32, device=q.device)
        st = self._lib.h3attn_canonical_order(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _pos_array(pos),
                                              _ptr(seg_offsets), n, S, _ptr(perm), _stream(stream))
        _check(st, "h3attn_canonical_order")
        return perm

    def set_stage_timing(self, enable: bool):
        _check(self._lib.h3attn_set_stage_timing(self._h, 1 if enable else 0), "h3attn_set_stage_timing")

    def stage_times(self) -> dict:
        """{stage: (total_ms, launches)} since the last read; waits for the recorded events."""
        n = len(STAGES)
        ms = (ctypes.c_float * n)()
        cnt = (ctypes.c_int * n)()
        _check(self._lib.h3attn_stage_times(self._h, ms, cnt, n), "h3attn_stage_times")
        return {STAGES[i]: (float(ms[i]), int(cnt[i])) for i in range(n)}

    def norm_weight_grad_partials(self, num_samples, out_q=None, out_k=None, stream=None):
        """h3attn_norm_weight_grad_partials: the last backward's per-(sample, head)
        norm-weight gradient partials, float32 [num_samples, H, 128] each for
        q_norm_w and k_norm_w (device tensors).  Returns (dq_partials, dk_partials)."""
        dev = torch.device("cuda", torch.cuda.current_device())
        shape = (num_samples, self.num_heads, 128)
        out_q = torch.empty(shape, dtype=torch.float32, device=dev) if out_q is None else out_q
        out_k = torch.empty(shape, dtype=torch.float32, device=dev) if out_k is None else out_k
        _check(self._lib.h3attn_norm_weight_grad_partials(self._h, _ptr(out_q), _ptr(out_k), _stream(stream)),
               "h3attn_norm_weight_grad_partials")
        return out_q, out_k

    def debug_stall(self, kernel: str | None, role: str = "mma", budget_cycles: int = 2_000_000):
        """h3attn_debug_stall (test hook): the next forward / backward / QKV call
        makes ``role`` of ``kernel`` wait once on a barrier nothing completes, for
        at most ``budget_cycles``; that call then reports ERR_TIMEOUT through
        device_status().  ``kernel=None`` cancels a request."""
        k = 0 if kernel is None else STALL_KERNELS[kernel]
        _check(self._lib.h3attn_debug_stall(self._h, k, STALL_ROLES[role], int(budget_cycles)), "h3attn_debug_stall")

    def device_status(self, stream=None) -> int:
        """Waits for the stream; returns (and clears) errors recorded on the device."""
        return int(self._lib.h3attn_device_status(self._h, _stream(stream)))

    def check(self, stream=None):
        _check(self.device_status(stream), "device")


# Bits of the device error word (the static forward's error_flags, h3attn_linear's).
_DEVICE_ERROR_STATUS = ((2, ERR_TIMEOUT), (1, ERR_INVALID_ARG), (4, ERR_INVALID_ARG))


def _raise_device_flags(flags, stream, where):
    """Waits for the stream and raises on a nonzero device error word."""
    (torch.cuda.current_stream() if stream is None else stream).synchronize()
    bits = int(flags.item())
    for bit, status in _DEVICE_ERROR_STATUS:
        if bits & bit:
            raise H3AttnError(status, f"{where} (device error bits {bits:#x})")


def forward_static(q, k, v, q_norm_w, k_norm_w, pos, seg_offsets, num_heads=None, eps=1e-6,
                   rope_theta=10000.0, rope_sections=(16, 24, 24), softmax_scale=0.0, num_samples=None,
                   out=None, lse=None, want_lse=True, error_flags=None, stream=None):
    """h3attn_forward_static: the forward with no handle and no device allocation
    inside the library (for hosts that forbid cudaMalloc while serving).

    ``out`` and ``lse`` are caller-owned device tensors; when not given they are
    created here with torch (``lse`` only if ``want_lse``).  ``error_flags``
    (int32 [1] on the device): when given, the call's device-side error bits
    are written there on the stream and checking them is the caller's job; when
    omitted, a zeroed word is created here and the binding waits for the stream
    and raises H3AttnError if the device reported an error (invalid
    seg_offsets, a wait that timed out, an fp16 range overflow).
    Returns (out, lse).
    """
    lib = load_library()
    S, H = q.shape[0], q.shape[1] if num_heads is None else num_heads
    cfg = Config()
    cfg.num_heads, cfg.head_dim, cfg.eps, cfg.rope_theta = H, 128, eps, rope_theta
    cfg.rope_sections[:] = list(rope_sections)
    cfg.rope_pairing, cfg.softmax_scale, cfg.max_tokens, cfg.max_samples = 0, softmax_scale, 0, 0
    cfg.key_order = KEY_ORDERS["packed"]
    n = int(seg_offsets.numel() - 1) if num_samples is None else num_samples
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((H, S), dtype=torch.float32, device=q.device)
    own_flags = error_flags is None
    if own_flags:
        error_flags = torch.zeros(1, dtype=torch.int32, device=q.device)
    st = lib.h3attn_forward_static(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(q_norm_w), _ptr(k_norm_w),
                                   _pos_array(pos), _ptr(seg_offsets), n, S, _ptr(out), _ptr(lse),
                                   _ptr(error_flags), _stream(stream))
    _check(st, "h3attn_forward_static")
    if own_flags and S > 0:
        _raise_device_flags(error_flags, stream, "h3attn_forward_static")
    return out, lse


def combine_norm_weight_grads(partials, per_sample=None, total=None, stream=None):
    """h3attn_combine_norm_weight_grads: per-(sample, head) norm-weight partials
    float32 [n, H, 128] (device, heads in global order) reduced in the library's
    fixed order, per sample over heads, then over samples.  Returns
    (per_sample [n, 128], total [128])."""
    lib = load_library()
    n, H = int(partials.shape[0]), int(partials.shape[1])
    partials = partials.contiguous()
    if per_sample is None:
        per_sample = torch.empty((max(n, 1), 128), dtype=torch.float32, device=partials.device)
    if total is None:
        total = torch.empty(128, dtype=torch.float32, device=partials.device)
    _check(lib.h3attn_combine_norm_weight_grads(_ptr(partials), n, H, _ptr(per_sample), _ptr(total), _stream(stream)),
           "h3attn_combine_norm_weight_grads")
    return per_sample[:n], total


def debug_exp2(x, path: str, stream=None):
    """h3attn_debug_exp2 (test hook): 2^x on the device by the SFU path ("sfu")
    or the FMA-pipe polynomial path ("poly") of the attention kernels."""
    lib = load_library()
    x = x.contiguous()
    y = torch.empty_like(x)
    _check(lib.h3attn_debug_exp2(_ptr(x), _ptr(y), x.numel(), {"sfu": 0, "poly": 1}[path], _stream(stream)),
           "h3attn_debug_exp2")
    return y


def fingerprint(t, out=None, stream=None):
    """h3attn_fingerprint of a contiguous device tensor's bytes.  Returns the
    device int64 [1] tensor holding it (read it with ``fingerprint_value``);
    nothing is copied to the host here."""
    lib = load_library()
    if not t.is_contiguous():
        raise ValueError("fingerprint: contiguous tensor expected")
    if out is None:
        out = torch.empty(1, dtype=torch.int64, device=t.device)
    _check(lib.h3attn_fingerprint(_ptr(t), t.numel() * t.element_size(), _ptr(out), _stream(stream)),
           "h3attn_fingerprint")
    return out


def fingerprint_value(fp) -> int:
    """The fingerprint as an unsigned 64-bit Python integer."""
    return int(fp.item()) & 0xFFFFFFFFFFFFFFFF


def linear(x, w, bias=None, out=None, error_flags=None, stream=None):
    """h3attn_linear: y = x w^T (+ bias) on the tensor cores, row-invariant.

    x bf16 [rows, in], w bf16 [out, in], bias FP32 [out] or None.  ``out`` and
    ``error_flags`` (int32 [1]) are caller-owned device tensors, created here
    with torch when not given.  Returns y bf16 [rows, out].
    """
    lib = load_library()
    rows, k = x.shape
    n = w.shape[0]
    if out is None:
        out = torch.empty((rows, n), dtype=torch.bfloat16, device=x.device)
    if error_flags is None:
        error_flags = torch.zeros(1, dtype=torch.int32, device=x.device)
    st = lib.h3attn_linear(_ptr(x), rows, k, _ptr(w), n, _ptr(bias), _ptr(out), _ptr(error_flags), _stream(stream))
    _check(st, "h3attn_linear")
    return out


def to_device(inp, device="cuda"):
    """Moves a workloads.Inputs to the device (pos as three int32 arrays)."""
    d = {"q": inp.q.to(device), "k": inp.k.to(device), "v": inp.v.to(device),
         "q_norm_w": inp.q_norm_w.to(device), "k_norm_w": inp.k_norm_w.to(device),
         "pos": [inp.pos[a].contiguous().to(device) for a in range(3)],
         "seg_offsets": inp.seg_offsets.to(device)}
    if inp.dout is not None:
        d["dout"] = inp.dout.to(device)
    return d
