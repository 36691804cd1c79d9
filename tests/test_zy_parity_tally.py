"""The excused-decision rule on the session's totals.

A GPU decision may differ from the oracle's only where the oracle's margin
is below 1e-5 relative (an accept test, a race, a top-p boundary), and such
excused decisions must stay below 1e-4 of all decisions. Each parity test
adds its counts to ``parity.TALLY``; this module, collected after every
parity test module and before the no-allocation test, checks the bound per
workload over everything the session compared, with no allowance of one
excused decision per test. Run on its own (nothing compared yet) it skips.
"""
import pytest

import parity

pytestmark = pytest.mark.gpu


def test_excused_decisions_below_the_bound_per_workload():
    totals = parity.totals_by_workload()
    if not totals:
        pytest.skip("no parity comparison ran in this session")
    print("\n" + "\n".join(parity.tally_lines()))
    for w, t in totals.items():
        assert t["excused"] < parity.EXCUSED_FRACTION * t["decisions"] or t["excused"] == 0, (w, t)
