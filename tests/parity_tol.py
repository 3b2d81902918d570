"""The parity rule shared by every GPU comparison against the fp64 oracle,
and a record of the errors each comparison saw.

Outputs: |out_gpu - out_oracle| <= 1e-2 on every bf16 output element.  Where
|out_oracle| >= 4, half a bf16 unit in the last place of the output is
0.0156, more than 1e-2, so no bf16 value can meet the literal bound there:
those elements may err by 1e-2 plus that half ulp.  LSE: |lse_gpu -
lse_oracle| <= 1e-3 (natural log, fp32).  Rows that see no key of their range
must come back as exactly out = 0 and lse = -inf.

Every comparison appends (test, case, rows, max|dout|, max|dout| where
|o| < 4, max|dlse|, max|o|) to RECORD; ``tests/conftest.py`` prints the table
at the end of the run and writes it as markdown to the file named by the
PK_PARITY_SUMMARY environment variable, when set."""
import os

import numpy as np

OUT_TOL = 1e-2
LSE_TOL = 1e-3
RECORD = []


def half_ulp_bf16(x):
    """Half a bf16 unit in the last place at |x| (8 significant bits)."""
    a = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return 0.5 * np.exp2(np.floor(np.log2(a)) - 7)


def out_allowance(out_oracle):
    """1e-2, plus the output's half ulp only where |o| >= 4."""
    return np.where(np.abs(out_oracle) >= 4.0, OUT_TOL + half_ulp_bf16(out_oracle), OUT_TOL)


def check(case, out_g, lse_g, out_o, lse_o, out_bound=None):
    """Assert the rule on (rows of) one launch's outputs and record the errors.
    ``out_bound``: a path whose arithmetic cannot meet the output rule (E4M3
    softmax weights) is held to this looser bound instead, its errors recorded
    all the same; the LSE rule and the empty-row rule stay."""
    empty = np.isneginf(lse_o)
    assert (np.isneginf(lse_g) == empty).all(), "rows without keys must give lse = -inf"
    assert (out_g[np.broadcast_to(empty.T[..., None], out_g.shape)] == 0).all()
    fin = ~empty
    assert np.isfinite(out_g).all() and np.isfinite(lse_g[fin]).all()
    if out_o.size == 0:
        return
    err = np.abs(out_g - out_o)
    small = np.abs(out_o) < 4.0
    e_out = float(err.max())
    e_small = float(err[small].max()) if small.any() else 0.0
    e_lse = float(np.abs(lse_g[fin] - lse_o[fin]).max()) if fin.any() else 0.0
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    RECORD.append((test, case, int(out_o.shape[0]), e_out, e_small, e_lse,
                   float(np.abs(out_o).max())))
    print(f"{case}: max|dout|={e_out:.3e} (|o|<4: {e_small:.3e}) max|dlse|={e_lse:.3e} "
          f"max|o|={np.abs(out_o).max():.3f}")
    bad = err > (out_allowance(out_o) if out_bound is None else out_bound)
    assert not bad.any(), (case, e_out, float(err[bad].max()))
    assert e_lse <= LSE_TOL, (case, e_lse)
