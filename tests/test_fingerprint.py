"""h3attn_fingerprint: the device fingerprint of a buffer's bytes equals, bit
for bit, the same definition evaluated on the host (written out here from the
definition in include/h3attn.h), for sizes that hit the 8-byte tail and the
grid-stride loop; and it changes when a byte changes or two words swap."""

import numpy as np
import pytest
import torch

from tests.helpers import lib_built, need_gpu

M64 = (1 << 64) - 1
G = 0x9E3779B97F4A7C15


def _mix(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def fingerprint_ref(b: bytes) -> int:
    """mix( sum_i mix(w_i + (i + 1) G) + len ) mod 2^64, w_i little-endian words."""
    n = len(b)
    w = np.frombuffer(b + b"\0" * ((-n) % 8), dtype="<u8")
    with np.errstate(over="ignore"):
        x = _mix(w + np.arange(1, len(w) + 1, dtype=np.uint64) * np.uint64(G))
        s = int(np.sum(x, dtype=np.uint64)) if len(w) else 0
    return int(_mix(np.array([(s + n) & M64], dtype=np.uint64))[0])


def test_reference_changes_with_any_byte_and_with_word_order():
    rng = np.random.default_rng(3)
    b = bytearray(rng.integers(0, 256, 1000, dtype=np.uint8).tobytes())
    f = fingerprint_ref(bytes(b))
    for pos in (0, 7, 8, 500, 999):
        c = bytearray(b)
        c[pos] ^= 1
        assert fingerprint_ref(bytes(c)) != f
    swapped = bytearray(b)
    swapped[0:8], swapped[8:16] = b[8:16], b[0:8]
    assert fingerprint_ref(bytes(swapped)) != f
    assert fingerprint_ref(bytes(b) + b"\0") != f  # the length is part of it
    assert fingerprint_ref(b"") == int(_mix(np.array([0], dtype=np.uint64))[0])


def test_mix_is_the_splitmix64_finaliser():
    # splitmix64 seeded with 0: the first output is mix(G) = 0xe220a8397b1dcdaf
    assert int(_mix(np.array([G], dtype=np.uint64))[0]) == 0xE220A8397B1DCDAF


@pytest.mark.gpu
@pytest.mark.parametrize("nbytes", [0, 1, 7, 8, 9, 2048 * 8 + 5, 10 * (1 << 20) + 3])
def test_device_fingerprint_equals_the_host_definition(nbytes):
    need_gpu()
    lib_built()
    from invariant_dit_attention_gb300.h3attn import fingerprint, fingerprint_value
    rng = np.random.default_rng(nbytes)
    host = rng.integers(0, 256, max(nbytes, 1), dtype=np.uint8)[:nbytes]
    dev = torch.from_numpy(host.copy()).cuda() if nbytes else torch.empty(0, dtype=torch.uint8, device="cuda")
    fp = fingerprint(dev)
    torch.cuda.synchronize()
    assert fingerprint_value(fp) == fingerprint_ref(host.tobytes())


@pytest.mark.gpu
def test_device_fingerprint_of_a_bf16_tensor_and_a_one_bit_change():
    need_gpu()
    lib_built()
    from invariant_dit_attention_gb300.h3attn import fingerprint, fingerprint_value
    t = torch.randn(925, 24, 128, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).cuda()
    a = fingerprint_value(fingerprint(t))
    assert a == fingerprint_ref(t.cpu().view(torch.int16).numpy().tobytes())
    u = t.clone()
    u.view(torch.int16)[500, 3, 7] ^= 1
    assert fingerprint_value(fingerprint(u)) != a
