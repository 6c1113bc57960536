"""The stored W fixtures still match the oracle bit for bit (drift guard)."""

import numpy as np
import pytest

import oracle
from tests.golden.write_golden import CASES, case_name, load


@pytest.mark.parametrize("case", CASES, ids=[case_name(*c) for c in CASES])
def test_oracle_reproduces_stored_w(case):
    stored = load()[case_name(*case)]
    W = oracle.mixing_matrix(case[0], case[1], case[2], local_thres=case[3], exp_sigma=case[4])
    assert np.array_equal(W.view(np.uint32), stored.view(np.uint32))
