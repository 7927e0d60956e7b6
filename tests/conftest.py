"""Shared pytest setup: the ``gpu`` marker and import paths."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def repo_root():
    return ROOT


def pytest_terminal_summary(terminalreporter):
    """Rounding-tie statistics of the parity checks run in this session: how
    often the oracle took the GPU's q_c rounding of a tie-zone element, how
    many nope Q_B values were ambiguous, and the elements outside one BF16 ulp."""
    import sys as _sys

    pu = _sys.modules.get("tests.parity_util")
    if pu is None or not pu.SESSION["steps_checked"]:
        return
    s = pu.SESSION
    terminalreporter.write_line(
        "parity ties: {steps_checked} steps checked; q_c tie-zone elements that took the other "
        "rounding: {q_c_ties_taken} (in {steps_with_q_c_tie} steps); ambiguous nope Q_B values: "
        "{q_ambiguous}; elements outside one BF16 ulp: q_c {q_c_plain_fails}, q_pe "
        "{q_pe_plain_fails}, q_latent {q_latent_plain_fails} of {q_latent_elems}; lowest "
        "within-1-ulp fraction {worst_plain_frac:.6f}".format(**s))
