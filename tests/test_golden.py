"""The oracle against its recorded outputs (tests/golden/oracle_small.json,
written by tests/golden/make_golden.py from the oracle alone): a regression
record of the oracle's arithmetic, next to the pins that tie it to the
pages' definitions."""
import importlib.util
import json
import os

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def golden():
    with open(os.path.join(HERE, "golden", "oracle_small.json")) as f:
        return json.load(f)


def test_oracle_reproduces_its_recorded_outputs(golden):
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(HERE, "golden", "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    now = mg.compute()
    for name, recorded in golden["inputs"].items():  # the seeded inputs themselves are stable
        for k_, v_ in recorded.items():
            np.testing.assert_array_equal(np.asarray(now["inputs"][name][k_]), np.asarray(v_), err_msg=k_)
    for name, recorded in golden["expected"].items():
        np.testing.assert_allclose(np.asarray(now["expected"][name]), np.asarray(recorded),
                                   rtol=1e-12, atol=1e-14, err_msg=name)


def test_recorded_chunked_form_equals_recorded_recurrence(golden):
    """Within the fixture itself: the third sequence's chunked-form outputs
    (chunk size 3, so the last chunk is ragged) equal the recurrence's rows
    3..6 and its final state."""
    o = np.asarray(golden["expected"]["recurrence_o"])[3:7]
    s = np.asarray(golden["expected"]["recurrence_state"])[2]
    np.testing.assert_allclose(np.asarray(golden["expected"]["chunked_o_seq3"]), o, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(np.asarray(golden["expected"]["chunked_state_seq3"]), s, rtol=1e-10, atol=1e-12)
