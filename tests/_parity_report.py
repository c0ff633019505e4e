"""Largest |gpu - oracle| / bound seen by each GPU parity test of this session (the bound
is oracle.tolerance), printed at the end of the run and written as JSON to the file named
by GMMFR_PARITY_REPORT when that variable is set."""
import json
import os

RATIOS = {}


def record(ratio: float, what: str = "") -> None:
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    key = test + (f" [{what}]" if what else "")
    RATIOS[key] = max(RATIOS.get(key, 0.0), float(ratio))


def write() -> None:
    path = os.environ.get("GMMFR_PARITY_REPORT")
    if path and RATIOS:
        os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
        with open(path, "w") as f:
            json.dump(RATIOS, f, indent=1, sort_keys=True)
