import importlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    # the oracle mutation test: GMMFR_ORACLE_PY_MUTANT = "<module>=<path>" runs the pins with the
    # functions of <module> (an oracle module) replaced by those of a mutated copy of its source
    spec = os.environ.get("GMMFR_ORACLE_PY_MUTANT")
    if spec:
        name, path = spec.split("=", 1)
        mod = importlib.import_module(name)
        ns = {"__name__": name + "_mutant", "__file__": mod.__file__}
        exec(compile(open(path).read(), path, "exec"), ns)
        for k, v in ns.items():
            if callable(v) and getattr(v, "__module__", None) == ns["__name__"]:
                setattr(mod, k, v)


def pytest_terminal_summary(terminalreporter):
    """Largest err/bound of each GPU parity comparison (tests/_parity_report.py)."""
    rep = sys.modules.get("_parity_report")
    if rep is None or not rep.RATIOS:
        return
    terminalreporter.write_sep("-", "parity: max |gpu - oracle| / (1e-4 * absb + 1e-6)")
    for k in sorted(rep.RATIOS):
        terminalreporter.write_line(f"{rep.RATIOS[k]:.4f}  {k}")
    terminalreporter.write_line(f"overall max {max(rep.RATIOS.values()):.4f} over {len(rep.RATIOS)} comparisons")
    rep.write()
