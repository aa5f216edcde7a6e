"""The all-heads comparison of the GPU parity tests, checked on the CPU: the
oracle's own full result passes it, and an error planted in any one value
head (or a NaN anywhere) fails it, also in heads past the first batch."""

import numpy as np
import pytest
import torch

from chunked_gated_delta_chunk_gb300 import inputs
from tests.harness import TOL_BF16, compare_all_heads, run_oracle


def _full(p):
    r = run_oracle(p)
    res = {"out": torch.from_numpy(r["out"]), "state_out": torch.from_numpy(r["state_out"])}
    if "conv_state_out" in r:
        res["conv_state_out"] = torch.from_numpy(r["conv_state_out"])
    return res


@pytest.fixture(scope="module")
def problem():
    return inputs.make_problem(81, [37, 5, 70], 2, 8, 16, 16, conv_kernel=4)


def test_oracle_result_passes(problem):
    errs = compare_all_heads(_full(problem), problem, TOL_BF16, batch=3)
    assert errs["out"] < 1e-12 and errs["state_out"] < 1e-12


@pytest.mark.parametrize("head", [0, 4, 7])
def test_planted_error_in_one_head_fails(problem, head):
    res = _full(problem)
    res["out"][10, head, 3] += 0.1 * float(res["out"].abs().max())
    with pytest.raises(AssertionError):
        compare_all_heads(res, problem, TOL_BF16, batch=3)


def test_nan_anywhere_fails(problem):
    res = _full(problem)
    res["state_out"][2, 7, 0, 0] = float("nan")
    with pytest.raises(AssertionError):
        compare_all_heads(res, problem, TOL_BF16, batch=3)


def test_conv_state_off_by_one_ulp_fails(problem):
    res = _full(problem)
    cs = res["conv_state_out"]
    cs[1, -1, 0] = float(np.nextafter(float(cs[1, -1, 0]), np.inf))
    with pytest.raises(AssertionError):
        compare_all_heads(res, problem, TOL_BF16, batch=3)
