"""Sensitivity of the oracle pins: a mistake planted in a copy of the oracle
(on the CPU, compiled with -DH3REF_PLANT=n) must make at least one pin fail."""

import os

import pytest

import oracle
from tests import test_oracle_pins as pins

PLANTS = {
    1: "sine sign flipped in the forward rotation",
    2: "interleaved channel pairs instead of rotate-half",
    3: "frequency exponent -j/n instead of -2j/n",
    4: "eps added outside the square root",
    5: "sum of squares not divided by 128",
    6: "softmax scale dropped",
    7: "one key past the segment end attended",
    8: "weight gradient sums g*n*w instead of g*n",
    9: "mean term dropped from the RMSNorm backward",
    10: "inverse rotation not applied in the backward",
    11: "softmax-Jacobian row term dropped from dS",
}

PIN_TESTS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]


@pytest.mark.parametrize("plant", sorted(PLANTS))
def test_planted_mistake_fails_a_pin(plant, tmp_path):
    lib = oracle.build(defines=[f"H3REF_PLANT={plant}"], out=os.path.join(tmp_path, f"libh3ref_{plant}.so"))
    oracle.use_library(lib)
    failed = []
    try:
        for t in PIN_TESTS:
            try:
                t()
            except AssertionError:
                failed.append(t.__name__)
    finally:
        oracle.use_library(None)
    assert failed, f"no pin caught planted mistake {plant}: {PLANTS[plant]}"
