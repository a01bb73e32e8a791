"""Near-threshold exclusions seen by the GPU parity tests in this session.

Every comparison with the oracle records how many sequences (or draft rows) it
compared and how many the oracle flagged as lying within 1e-6 of a decision
threshold; conftest prints the table at the end of the run.
"""
RECORDS = []


def record(case, compared, flagged, unit="sequences"):
    RECORDS.append((str(case), int(compared), int(flagged), unit))
