import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The per-comparison parity errors of the run (see parity_tol.py)."""
    from parity_tol import LSE_TOL, OUT_TOL, RECORD
    if not RECORD:
        return
    lines = [f"| test | case | rows | max abs dout | max abs dout, abs(o) < 4 | max abs dlse | max abs o |",
             "|---|---|---|---|---|---|---|"]
    for test, case, rows, e_out, e_small, e_lse, omax in RECORD:
        lines.append(f"| {test} | {case} | {rows} | {e_out:.3e} | {e_small:.3e} | {e_lse:.3e} | "
                     f"{omax:.3f} |")
    tr = terminalreporter
    tr.write_sep("-", f"parity errors (bound: {OUT_TOL} where |o| < 4, else {OUT_TOL} + half a "
                      f"bf16 ulp; LSE {LSE_TOL})")
    for ln in lines:
        tr.write_line(ln)
    path = os.environ.get("PK_PARITY_SUMMARY")
    if path:
        with open(path, "w") as f:
            f.write("# Parity errors of the GPU tests against the fp64 oracle\n\n")
            f.write(f"Bound: max abs error {OUT_TOL} on bf16 outputs (where |o_oracle| >= 4, "
                    f"{OUT_TOL} + half a bf16 ulp of o), {LSE_TOL} on the fp32 LSE.  "
                    f"Exception: the all-E4M3 cases (test_parity_fp8_pv.py, cases "
                    f"without '/uniform') are held to a sanity bound of 0.1 on the output, "
                    f"their errors recorded here.\n\n")
            f.write("Command: `PK_PARITY_SUMMARY=<file> python -m pytest "
                    + " ".join(config.invocation_params.args) + "`\n\n")
            f.write("\n".join(lines) + "\n")
