"""The fp64 oracle against its pins (CPU only)."""

import numpy as np
import pytest

from oracle import oracle as O
from tests import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    ok, detail = pin(O.load())
    assert ok, detail


def test_stack_prefix_matches_full():
    # Causality: the first P rows of an L-layer stack depend only on the first P inputs.
    dims = O.Dims(2, 24, 16, 4, 4, 32, 5)
    layers = [P.tiny_params(16, 4, 32, seed=80 + l) for l in range(3)]
    x = np.random.default_rng(90).normal(size=(2, 24, 16))
    full = O.stack_forward(dims, x, layers)
    pre = O.stack_forward(dims, x, layers, prefix=9)
    assert np.max(np.abs(pre - full[:, :9])) <= 1e-13


def test_stack_is_layer_chain():
    dims = O.Dims(1, 12, 8, 2, 4, 16, 3)
    layers = [P.tiny_params(8, 2, 16, seed=100 + l) for l in range(2)]
    x = np.random.default_rng(91).normal(size=(1, 12, 8))
    y = O.block_forward(dims, O.block_forward(dims, x, layers[0]), layers[1])
    assert np.array_equal(O.stack_forward(dims, x, layers), y)


def test_threads_do_not_change_results():
    dims = O.Dims(2, 16, 16, 4, 4, 32, 6)
    p = P.tiny_params(16, 4, 32, seed=110)
    x = np.random.default_rng(111).normal(size=(2, 16, 16))
    a = O.block_forward(dims, x, p, threads=1)
    b = O.block_forward(dims, x, p, threads=5)
    assert np.array_equal(a, b)


def _serial_mutants():
    """Plausible mistakes in the serial block's composition (each must break a pin)."""
    real = O.serial_block_forward

    def parallel_instead(dims, x, p, rows=None, threads=0, lib=None):
        return O.block_forward(dims, x, p, rows=rows, threads=threads, lib=lib)

    def literal_eq3(dims, x, p, rows=None, threads=0, lib=None):
        # y = x + MLP(LN(x + Attn(LN(x)))): the attention term left out of the output
        y = real(dims, x, p, rows=rows, threads=threads, lib=lib)
        _, st = O.block_forward(dims, x, p, rows=rows, threads=threads, keep_stages=True,
                                lib=lib)
        return y - st["att_proj"].reshape(y.shape)

    def first_ln_twice(dims, x, p, rows=None, threads=0, lib=None):
        q = {k: v for k, v in p.items() if k not in ("ln2_gamma", "ln2_beta")}
        return real(dims, x, q, rows=rows, threads=threads, lib=lib)

    return [parallel_instead, literal_eq3, first_ln_twice]


@pytest.mark.parametrize("mutant", _serial_mutants(), ids=lambda f: f.__name__)
def test_serial_pins_catch_mutant(mutant, monkeypatch):
    monkeypatch.setattr(O, "serial_block_forward", mutant)
    serial_pins = [P.pin_serial_library, P.pin_serial_reduces_to_parallel,
                   P.pin_serial_first_order, P.pin_serial_rows_mode]
    assert not all(pin(O.load())[0] for pin in serial_pins)
