"""Counts of fully compared and flagged (near-tie) sequences per parity case, filled by
the GPU parity tests and printed by conftest at the end of the run."""
RESULTS = {}
