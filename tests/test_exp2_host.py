"""The kernels' software exp2, through its host twin (same operation sequence),
against the exact 2**x (float64), exhaustively over the bf16 inputs and densely
over fp32 inputs. The device copy is compared bit for bit with this twin in the
GPU tests."""
import numpy as np
import pytest

import oracle
from fa_testing_lib import fa_exp2_poly_host


def test_every_negative_bf16_input():
    bits = (np.arange(0x8000, 0x10000, dtype=np.uint32) << 16).view(np.float32)
    xs = bits[np.isfinite(bits) & (bits >= -125.0)]
    got = np.array([fa_exp2_poly_host(float(x)) for x in xs], dtype=np.float64)
    rel = np.abs(got / oracle.exp2_exact(xs.astype(np.float64)) - 1)
    assert rel.max() <= 2.0 ** -13


def test_dense_fp32_inputs_including_stale_max_margin():
    xs = np.linspace(-125.0, 8.0, 200001).astype(np.float32)
    got = np.array([fa_exp2_poly_host(float(x)) for x in xs], dtype=np.float64)
    rel = np.abs(got / oracle.exp2_exact(xs.astype(np.float64)) - 1)
    assert rel.max() <= 2.0 ** -13


@pytest.mark.parametrize("x,want", [(0.0, 1.0), (-1.0, 0.5), (-127.0, 0.0), (-1e30, 0.0),
                                    (float("-inf"), 0.0), (3.0, 8.0)])
def test_special_values(x, want):
    assert fa_exp2_poly_host(x) == want
