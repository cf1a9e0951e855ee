"""The comparison the GPU parity tests use, on the CPU: what passes and what
fails the bf16 bar."""
import numpy as np
import pytest
import torch

from tests.parity_util import check_close


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float64)).to(torch.bfloat16).double().numpy()


def test_rounding_alone_passes_on_a_tiny_output():
    # values just above a power of two: rounding to bf16 alone costs more than 3e-3
    want = np.array([-0.529496, 0.5021, 1.0117, -2.0233])
    got = _bf16(want)
    assert np.linalg.norm(got - want) / np.linalg.norm(want) > 3e-3
    check_close(got, want, torch.bfloat16, "rounded oracle")


def test_a_planted_error_fails_on_a_tiny_output():
    want = np.array([-0.529496, 0.5021, 1.0117, -2.0233])
    with pytest.raises(AssertionError):
        check_close(_bf16(want * 1.01), want, torch.bfloat16, "1% off, stored in bf16")


def test_the_bar_stays_3e3_on_a_large_output():
    want = np.random.default_rng(0).standard_normal(100_000)
    check_close(_bf16(want), want, torch.bfloat16, "rounded oracle")
    with pytest.raises(AssertionError, match=r"> 3\.000e-03"):
        check_close(_bf16(want * 1.004), want, torch.bfloat16, "0.4% off, stored in bf16")


def test_fp32_bar_is_max_abs():
    want = np.linspace(-1, 1, 101)
    check_close(want + 0.9e-4, want, torch.float32, "within 1e-4 of max")
    with pytest.raises(AssertionError):
        check_close(want + 1.1e-4, want, torch.float32, "beyond 1e-4 of max")
