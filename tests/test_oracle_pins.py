"""The fp64 oracle against what the pages and the mathematics fix (CPU only)."""

import pytest

import pins
from oracle import oracle as orc


@pytest.fixture(scope="module")
def lib():
    return orc.load()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(lib, pin):
    pin(lib)


def test_golden_fixture_is_self_consistent():
    # the page's kernel is b·a^k and its outputs are the kernel's causal
    # convolution with u: the fixture must say the same thing twice
    g = pins.read_golden()
    a, b, u = g["a"][0], g["b"][0], g["u"]
    assert g["kernel"] == pytest.approx([b * a ** k for k in range(3)], rel=1e-12)
    conv = [sum(g["kernel"][k] * u[t - k] for k in range(t + 1)) for t in range(3)]
    assert conv == pytest.approx(g["y"], rel=1e-12)
