"""Shared comparison helpers for the GPU parity tests (tolerances stated once)."""
import numpy as np

# Forward: O max-abs <= 2e-2 and relative Frobenius <= 1e-2; LSE abs <= 1e-3.
# Backward: relative Frobenius <= 2e-2 for dQ, dK, dV.
O_MAX_ABS = 2e-2
O_REL_FRO = 1e-2
LSE_ABS = 1e-3
GRAD_REL_FRO = 2e-2


def rel_fro(got, ref):
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(np.asarray(got, np.float64) - ref) / (den if den > 0 else 1.0))


def check_fwd(o_got, lse_got, o_ref, lse_ref, what=""):
    o_got = np.asarray(o_got, np.float64)
    lse_got = np.asarray(lse_got, np.float64)
    assert np.isfinite(o_got).all() and np.isfinite(lse_got).all(), f"{what}: non-finite output"
    e_max = float(np.abs(o_got - o_ref).max()) if o_ref.size else 0.0
    e_fro = rel_fro(o_got, o_ref) if o_ref.size else 0.0
    e_lse = float(np.abs(lse_got - lse_ref).max()) if lse_ref.size else 0.0
    assert e_max <= O_MAX_ABS, f"{what}: O max abs err {e_max:.3e}"
    assert e_fro <= O_REL_FRO, f"{what}: O rel Frobenius err {e_fro:.3e}"
    assert e_lse <= LSE_ABS, f"{what}: LSE abs err {e_lse:.3e}"
    return e_max, e_fro, e_lse
