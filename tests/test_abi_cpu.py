"""The C-ABI library builds for sm_103a, loads, exports every declared entry
point, and rejects bad configurations on the host (no GPU needed)."""

import ctypes
import os
import re
import subprocess

import pytest

from tests.helpers import lib_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "h3attn.h")).read()
    return sorted(set(re.findall(r"^\S.*?\b(h3attn_[a-z0-9_]+)\(", text, flags=re.M)))


def test_header_declares_the_binding_exports():
    from invariant_dit_attention_gb300.h3attn import EXPORTS
    assert declared_symbols() == sorted(EXPORTS)


def test_library_exports_every_declared_symbol():
    path = lib_built()
    lib = ctypes.CDLL(path)
    nm = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (h3attn_\w+)", nm))
    for name in declared_symbols():
        assert hasattr(lib, name)
        assert name in exported, name


def test_status_strings():
    from invariant_dit_attention_gb300 import h3attn
    lib_built()
    names = [h3attn.status_string(s) for s in range(6)]
    assert names[0] == "ok" and len(set(names)) == 6
    assert h3attn.status_string(99) == "unknown status"


def _cfg(**kw):
    from invariant_dit_attention_gb300.h3attn import Config
    c = Config()
    c.num_heads, c.head_dim, c.eps, c.rope_theta = 4, 128, 1e-6, 10000.0
    c.rope_sections[:] = [16, 24, 24]
    c.rope_pairing, c.softmax_scale, c.max_tokens, c.max_samples = 0, 0.0, 64, 4
    for k, v in kw.items():
        if k == "rope_sections":
            c.rope_sections[:] = v
        else:
            setattr(c, k, v)
    return c


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=64), 2), (dict(rope_pairing=1), 2), (dict(rope_sections=[12, 24, 24]), 2),
    (dict(rope_sections=[64, 64, 8]), 2), (dict(num_heads=0), 1), (dict(max_tokens=0), 1),
    (dict(max_samples=0), 1), (dict(eps=-1.0), 1), (dict(key_order=2), 1), (dict(key_order=-1), 1),
    (dict(store_ds=2), 1), (dict(reuse_qk_hat=2), 1), (dict(store_ds=1, num_heads=48, max_tokens=1 << 22), 3),
])
def test_create_rejects_bad_config_on_host(kw, status):
    from invariant_dit_attention_gb300.h3attn import load_library
    lib_built()
    lib = load_library()
    h = ctypes.c_void_p()
    assert lib.h3attn_create(ctypes.byref(_cfg(**kw)), ctypes.byref(h)) == status
    assert not h.value


def test_null_handle_and_pointers_rejected():
    from invariant_dit_attention_gb300.h3attn import load_library
    lib_built()
    lib = load_library()
    assert lib.h3attn_create(None, None) == 1
    pos = (ctypes.c_void_p * 3)()
    assert lib.h3attn_forward(None, None, None, None, None, None, pos, None, 1, 4, None, None, None) == 1
    assert lib.h3attn_device_status(None, None) == 1
    assert lib.h3attn_destroy(None) == 0


def test_static_forward_and_new_entry_points_reject_on_host():
    """Checks that need no device: the static forward offers only the packed key
    order; the fused QKV forward and the canonical-order call reject a null
    handle."""
    from invariant_dit_attention_gb300.h3attn import load_library
    lib_built()
    lib = load_library()
    pos = (ctypes.c_void_p * 3)()
    assert lib.h3attn_forward_static(ctypes.byref(_cfg(key_order=1)), None, None, None, None, None, pos, None,
                                     1, 4, None, None, None, None) == 2
    assert lib.h3attn_qkv_forward(None, None, 64, None, None, None, None, pos, None, 1, 4, None, None, None, None,
                                  None, None) == 1
    assert lib.h3attn_canonical_order(None, None, None, None, None, pos, None, 1, 4, None, None) == 1


def test_binding_checks_and_stored_ds_workspace_size():
    """Python-side checks before the library is asked for a handle, and the
    stored-dS workspace size the "auto" setting compares with its limit."""
    from invariant_dit_attention_gb300.h3attn import STORED_DS_AUTO_LIMIT, H3Attn, stored_ds_bytes
    lib_built()
    with pytest.raises(ValueError):
        H3Attn(4, 64, 4, key_order="sorted")
    # H ceil(T/128) (ceil(T/128) + N) blocks of 128 x 128 fp16
    assert stored_ds_bytes(48, 13539, 8) == 48 * 106 * 114 * 32768
    assert stored_ds_bytes(48, 13539, 8) < STORED_DS_AUTO_LIMIT < stored_ds_bytes(48, 32768, 8)


def test_debug_stall_rejects_bad_arguments_without_a_gpu():
    from invariant_dit_attention_gb300 import h3attn
    lib_built()
    lib = h3attn.load_library()
    assert lib.h3attn_debug_stall(None, 1, 1, 1000) == h3attn.ERR_INVALID_ARG
