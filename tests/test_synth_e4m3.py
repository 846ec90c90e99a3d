"""Pins of the E4M3 input rounding (the FP8 activation workloads).

The values follow from the OCP 8-bit floating point format E4M3 ("e4m3fn"):
bias 7, three mantissa bits, no infinities, largest finite 448 (code 0x7E),
NaN at 0x7F / 0xFF, subnormals in steps of 2^-9.  A slip in the generator
(a wrong bias, a dropped subnormal branch, ties rounded up instead of to
even, no saturation) fails one of these.
"""

import numpy as np
import pytest
import torch

from tensor_train_compressed_tt_gb300 import synth


@pytest.mark.parametrize("value,code", [
    (1.0, 0x38), (-2.0, 0xC0), (448.0, 0x7E), (-448.0, 0xFE), (2.0 ** -6, 0x08),
    (2.0 ** -9, 0x01), (7 * 2.0 ** -9, 0x07), (0.0, 0x00), (1.75, 0x3E), (0.3125, 0x2A),
])
def test_codes_of_format_values(value, code):
    v = synth.round_e4m3(np.array([value]))
    assert v[0] == value
    assert synth.e4m3_bytes(v)[0] == code
    assert synth.e4m3_values(np.array([code], np.uint8))[0] == value


def test_ties_round_to_even_and_saturate():
    x = np.array([1.0625, 1.1875, 3 * 2.0 ** -10, 2.0 ** -10, 500.0, -1e6, 464.0, 0.9999])
    want = np.array([1.0, 1.25, 2 * 2.0 ** -9, 0.0, 448.0, -448.0, 448.0, 1.0])
    np.testing.assert_array_equal(synth.round_e4m3(x), want.astype(np.float32))


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = synth.e4m3_values(codes)
    assert np.all(np.isfinite(vals))
    np.testing.assert_array_equal(synth.round_e4m3(vals), vals)
    nz = codes != 0x80   # -0 encodes back to 0x80 as well, but compare magnitudes apart
    np.testing.assert_array_equal(synth.e4m3_bytes(vals)[nz], codes[nz])
    assert np.isnan(synth.e4m3_values(np.array([0x7F, 0xFF], np.uint8))).all()


def test_midpoints_go_to_the_even_neighbour():
    pos = np.sort(synth.e4m3_values(np.arange(0, 0x7F, dtype=np.uint8)).astype(np.float64))
    mid = (pos[:-1] + pos[1:]) / 2
    got = synth.round_e4m3(mid).astype(np.float64)
    codes = synth.e4m3_bytes(got)
    assert np.all(codes % 2 == 0)
    assert np.all((got == pos[:-1]) | (got == pos[1:]))


def test_matches_torch_float8_on_random_values():
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 40.0)])
    x = np.clip(x, -448.0, 448.0).astype(np.float32)
    ours = synth.e4m3_bytes(synth.round_e4m3(x))
    theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # signed zeros may differ in the sign bit only
    same = (ours == theirs) | (((ours & 0x7F) == 0) & ((theirs & 0x7F) == 0))
    assert same.all()


def test_e4m3_workload_inputs_are_representable():
    w = synth.WORKLOADS["tt768_e4m3"]
    inp = synth.draw(w, seed=0, tokens=64)
    for a in (inp.x, inp.dy):
        np.testing.assert_array_equal(synth.e4m3_values(synth.e4m3_bytes(a)), a)
    assert np.abs(inp.x).max() <= 448.0
