"""Shared helpers for the parity tests: device transfer and the acceptance
metrics (max-abs and relative RMS on O, absolute error on LSE)."""
import numpy as np

# Acceptance bar for the CUDA path against the fp64 oracle (bf16 output,
# fp32 log-sum-exp).  rel_rms = ||O_gpu - O_ref||_2 / ||O_ref||_2.
MAX_ABS = 2e-2
REL_RMS = 5e-3
LSE_ABS = 1e-3


def to_dev(a, dev):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def metrics(got_o, got_l, ref_o, ref_l):
    go = np.asarray(got_o, np.float64)
    err = np.abs(go - ref_o)
    max_abs = float(err.max()) if err.size else 0.0
    den = float((ref_o ** 2).sum())
    rel_rms = float(np.sqrt((err ** 2).sum() / den)) if den > 0 else float(np.sqrt((err ** 2).sum()))
    lse_err = 0.0
    same_inf = True
    if got_l is not None:
        gl = np.asarray(got_l, np.float64)
        fin = np.isfinite(ref_l)
        same_inf = bool(np.array_equal(np.isfinite(gl), fin)) and bool(np.all(gl[~fin] == -np.inf))
        if fin.any():
            lse_err = float(np.abs(gl[fin] - ref_l[fin]).max())
    return dict(max_abs=max_abs, rel_rms=rel_rms, lse_err=lse_err, same_inf=same_inf,
                finite=bool(np.all(np.isfinite(go))))


def assert_parity(m, label=""):
    assert m["finite"], "%s: non-finite output" % label
    assert m["same_inf"], "%s: LSE -inf pattern differs" % label
    assert m["max_abs"] <= MAX_ABS, "%s: max_abs %.3e" % (label, m["max_abs"])
    assert m["rel_rms"] <= REL_RMS, "%s: rel_rms %.3e" % (label, m["rel_rms"])
    assert m["lse_err"] <= LSE_ABS, "%s: lse_err %.3e" % (label, m["lse_err"])
