"""Tolerated differences counted by the GPU parity tests: top-p decisions
that flip inside the band around round_D(1 - p), and min-p decisions inside
their relative band.  The tests add one record per workload; the summary
hook in conftest.py prints them at the end of the run, so they show even
under ``pytest -q``.  Nothing here computes any part of the filter."""

RECORDS = []


def record(name, rows, flips, what="top-p flips inside the band"):
    RECORDS.append((str(name), int(rows), int(flips), what))
