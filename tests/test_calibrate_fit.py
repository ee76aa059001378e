"""Host logic of the per-shard cost calibration (no GPU): the least-squares
fit of shard times against workload measures, and the imbalance ratio."""
import numpy as np
import pytest

from context_document_masked_gb300 import calibrate as cal


def _rows(coef, launch, n=9, seed=0, noise=0.0):
    rng = np.random.default_rng(seed)
    rows = []
    for _ in range(n):
        r = {"pairs": float(rng.integers(10_000, 5_000_000)), "tiles": float(rng.integers(10, 3000)),
             "qt": float(rng.integers(1, 60))}
        y = launch + coef[0] * r["tiles"] + coef[1] * r["qt"]
        r["ms"] = y * (1.0 + noise * rng.standard_normal())
        rows.append(r)
    return rows


def test_fit_recovers_exact_linear_cost_with_launch_term():
    rows = _rows((2.5e-4, 1.5e-3), launch=0.02)
    f = cal.fit(rows, ("tiles", "qt"), "ms")
    assert f["coef"]["tiles"] == pytest.approx(2.5e-4, rel=1e-9)
    assert f["coef"]["qt"] == pytest.approx(1.5e-3, rel=1e-9)
    assert f["coef"]["launch"] == pytest.approx(0.02, rel=1e-9)
    assert f["r2"] == pytest.approx(1.0, abs=1e-12)
    assert f["max_rel_err"] < 1e-9


def test_fit_without_intercept_is_through_the_origin():
    rows = _rows((3e-4, 0.0), launch=0.0)
    f = cal.fit(rows, ("tiles",), "ms", intercept=False)
    assert set(f["coef"]) == {"tiles"}
    assert f["coef"]["tiles"] == pytest.approx(3e-4, rel=1e-9)
    # A launch cost the model cannot express shows up as residual error.
    g = cal.fit(_rows((3e-4, 0.0), launch=0.05), ("tiles",), "ms", intercept=False)
    assert g["max_rel_err"] > 0.01 and g["r2"] < 1.0


def test_fit_reports_residuals_of_noisy_data():
    rows = _rows((2e-4, 1e-3), launch=0.01, n=40, seed=3, noise=0.02)
    f = cal.fit(rows, ("tiles", "qt"), "ms")
    y = np.array([r["ms"] for r in rows])
    x = np.array([[r["tiles"], r["qt"], 1.0] for r in rows])
    c = np.array([f["coef"]["tiles"], f["coef"]["qt"], f["coef"]["launch"]])
    pred = x @ c
    assert f["max_rel_err"] == pytest.approx(float(np.max(np.abs(pred - y) / y)))
    assert f["r2"] == pytest.approx(1 - ((y - pred) ** 2).sum() / ((y - y.mean()) ** 2).sum())
    # Least squares: the residual is orthogonal to every regressor column.
    assert np.abs(x.T @ (y - pred)).max() < 1e-6 * np.abs(x.T @ y).max()


def test_imbalance_is_max_over_mean():
    assert cal.imbalance([3.0, 3.0, 3.0]) == 1.0
    assert cal.imbalance([1.0, 2.0, 3.0]) == pytest.approx(1.5)
    assert cal.imbalance([0.5, 4.0]) == pytest.approx(4.0 / 2.25)
