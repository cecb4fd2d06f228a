"""The parity errors each GPU test measured, gathered for the summary that
``conftest.py`` prints at the end of a run (one line per test), so that a run
shows the errors next to the bounds they were held to, not only pass / fail."""

RECORD = None   # pytest's record_property of the running test (set by conftest)


def report(**errors):
    """Attach measured errors (name -> float) to the running test's report."""
    if RECORD is not None:
        RECORD("parity", {k: float(v) for k, v in errors.items()})
