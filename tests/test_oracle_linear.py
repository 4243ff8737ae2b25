"""Pins of the projection oracle (oracle.linear): y = x w^T (+ b).

Each pin is written as a check on an implementation; the oracle must pass all
of them, and plausible mistakes planted in copies of it (a transposed weight,
a dropped or misplaced bias, a dropped term of the sum) must each fail one."""

import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


def pin_brute_force(lin):
    """Against explicit sums on tiny inputs (pure Python loops)."""
    x, w = _rand((3, 5), 1), _rand((4, 5), 2)
    b = torch.randn(4, generator=torch.Generator().manual_seed(3))
    y = lin(x, w, b)
    xf, wf, bf = x.float().tolist(), w.float().tolist(), b.tolist()
    for r in range(3):
        for n in range(4):
            s = bf[n]
            for k in range(5):
                s += xf[r][k] * wf[n][k]
            if abs(y[r][n] - s) > 1e-9:
                return False
    return True


def pin_one_hot(lin):
    """A one-hot row e_j picks column j of the weight, plus the bias."""
    w = _rand((6, 8), 4)
    b = torch.randn(6, generator=torch.Generator().manual_seed(5))
    for j in range(8):
        x = torch.zeros(1, 8, dtype=torch.bfloat16)
        x[0, j] = 1.0
        y = lin(x, w, b)
        if not np.array_equal(y[0], w.float().numpy()[:, j].astype(np.float64) + b.numpy().astype(np.float64)):
            return False
    return True


def pin_identity(lin):
    """The identity weight and no bias return x itself, exactly."""
    x = _rand((5, 16), 6)
    y = lin(x, torch.eye(16, dtype=torch.bfloat16), None)
    return np.array_equal(y, x.float().numpy().astype(np.float64))


def pin_linear_in_x(lin):
    """y(2 x1 + x2) = 2 y(x1) + y(x2); small integer inputs keep 2 x1 + x2 exact in bf16."""
    g = torch.Generator().manual_seed(7)
    x1 = torch.randint(-4, 5, (4, 32), generator=g).to(torch.bfloat16)
    x2 = torch.randint(-4, 5, (4, 32), generator=g).to(torch.bfloat16)
    w = _rand((24, 32), 9)
    y = lin((2 * x1.float() + x2.float()).to(torch.bfloat16), w, None)
    ref = 2.0 * lin(x1, w, None) + lin(x2, w, None)
    return np.allclose(y, ref, rtol=1e-12, atol=1e-12)


PINS = (pin_brute_force, pin_one_hot, pin_identity, pin_linear_in_x)


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_linear_passes_pin(pin):
    assert pin(oracle.linear)


def _planted(kind):
    def lin(x, w, b=None):
        xs = np.asarray(x.float().numpy(), dtype=np.float64)
        ws = np.asarray(w.float().numpy(), dtype=np.float64)
        if kind == "transposed_weight":
            y = xs @ ws if ws.shape[0] == xs.shape[1] else np.zeros((xs.shape[0], ws.shape[0]))
        elif kind == "dropped_term":
            y = xs[:, :-1] @ ws[:, :-1].T
        else:
            y = xs @ ws.T
        if b is not None and kind != "dropped_bias":
            bs = np.asarray(b.numpy(), dtype=np.float64)
            y = y + (bs[:, None][: y.shape[0]] if kind == "bias_on_rows" and bs.shape[0] >= y.shape[0] else bs[None, :])
        return y
    return lin


@pytest.mark.parametrize("kind", ["transposed_weight", "dropped_term", "dropped_bias", "bias_on_rows"])
def test_planted_mistakes_are_caught(kind):
    lin = _planted(kind)
    assert not all(pin(lin) for pin in PINS), kind
