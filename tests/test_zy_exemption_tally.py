"""The near-boundary exemptions of the whole GPU parity suite, after its verification tests.

Every check_verify call (tests/parity_util.py) adds its draws -- ratio tests and resampling
draws the oracle took -- and its exempt divergences (a GPU decision differing from the oracle's
where the uniform lies within 1e-6 of the boundary, which fp32 sums cannot resolve) to one
tally.  The verification step's contract allows fewer than 1e-5 of the draws to be exempt; with
the suite's draw count that means none.  The file is named so that pytest collects it after the
parity tests and before the no-allocation test."""
import pytest

import parity_util as PU

pytestmark = pytest.mark.gpu


def test_suite_exemptions_below_bar():
    if PU.TALLY["calls"] == 0:
        pytest.skip("no verification parity test ran in this session")
    draws, exempt = PU.TALLY["draws"], PU.TALLY["exempt"]
    print(f"suite: {PU.TALLY['calls']} verification checks, {draws} draws, {exempt} exempt")
    assert draws > 0
    assert exempt < 1e-5 * draws, (exempt, draws)
