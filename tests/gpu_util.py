"""Helpers shared by the GPU tests: device copies and tolerance checks against the oracle."""
import numpy as np

# Tolerances: max-abs 2e-3 on O and 1e-4 on LSE (fp32 accumulation, f16 P operand), and
# the RMSE of O within 3e-4, the bound "KVARN KV Performance optimizations" (item 9) accepts
# for chunked-window parity (a change of floating-point reduction order only).
TOL_O = 2e-3
TOL_LSE = 1e-4
TOL_RMSE_O = 3e-4


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_close(out, lse, want_o, want_l, tol_o=TOL_O, tol_l=TOL_LSE, tol_rmse=TOL_RMSE_O):
    o = out.detach().cpu().numpy().astype(np.float64).reshape(want_o.shape)
    l = lse.detach().cpu().numpy().astype(np.float64).reshape(want_l.shape)
    empty = np.isneginf(want_l)
    assert np.array_equal(np.isneginf(l), empty), "empty rows differ"
    assert np.all(np.isfinite(o)), "non-finite output"
    if np.any(~empty):
        err_l = np.max(np.abs(l[~empty] - want_l[~empty]))
        assert err_l <= tol_l, f"LSE max-abs {err_l:.3e} > {tol_l}"
    err_o = np.max(np.abs(o - want_o)) if o.size else 0.0
    assert err_o <= tol_o, f"O max-abs {err_o:.3e} > {tol_o}"
    rmse = float(np.sqrt(np.mean((o - want_o) ** 2))) if o.size else 0.0
    assert rmse <= tol_rmse, f"O RMSE {rmse:.3e} > {tol_rmse}"
    assert np.all(o[empty] == 0.0)
    return float(err_o), float(np.max(np.abs(l[~empty] - want_l[~empty])) if np.any(~empty) else 0.0)


def rmse(out, want_o):
    o = out.detach().cpu().numpy().astype(np.float64).reshape(want_o.shape)
    return float(np.sqrt(np.mean((o - want_o) ** 2)))
