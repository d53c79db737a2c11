"""Parity bars for attention outputs against the fp64 oracle.

Two bars, both applied to every compared element:

* the acceptance bar: max |got - want| <= 2e-2 and mean |got - want| <= 2e-3;
* the bf16-floor bar, which is what catches a kernel that silently drops keys.
  An exact method whose result is rounded once to bf16 is off by at most half
  a bf16 ulp, at most 2^-8 |want|.  The kernels also round P to bf16 for the
  P V product.  That rounding gives each weight a relative error of at most
  2^-9, spread over all keys, so the error it adds is a small multiple of
  2^-9 times the row's rms, not of the element.  Each element must therefore
  stay within

      |got - want| <= 2^-8 |want| + ROW_K * 2^-8 * rms(want row),

  and the mean error over all compared elements must stay within
  FLOOR_MEAN_K times the mean error of the bf16-rounded oracle (the floor).

With N(0, 1) inputs and scale 1/sqrt(D), a row's output shrinks roughly as
1/sqrt(ctx).  One dropped 16-key block then moves the output by about as
much as the acceptance bar's mean-abs at ctx ~ 4000, and by far less at
ctx 30 000, where the floor bar still rejects it.  The CPU test
`test_floor_bar_rejects_a_dropped_block` pins this: the floor bar accepts
the bf16-rounded oracle and rejects the oracle with one block dropped.

Each check is recorded; conftest prints the per-case floor ratio and worst
element at the end of the run.
"""

from __future__ import annotations

import numpy as np

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
ROW_K = 3.0
FLOOR_MEAN_K = 3.0

RECORDS: list[dict] = []


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), exactly:
    a scaling by a power of two, numpy's round-half-even, and the scaling back
    are all exact in float64 for the magnitudes attention outputs take."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = (x != 0) & np.isfinite(x)
    e = np.floor(np.log2(np.abs(x[nz])))
    ulp = np.exp2(e - 7)                      # 8 significant bits
    out[nz] = np.round(x[nz] / ulp) * ulp
    out[~np.isfinite(x)] = x[~np.isfinite(x)]
    return out


def _as_f64(got) -> np.ndarray:
    try:
        import torch
        if isinstance(got, torch.Tensor):
            return got.detach().to(torch.float64).cpu().numpy()
    except ImportError:   # pragma: no cover
        pass
    return np.asarray(got, dtype=np.float64)


def evaluate(got, want: np.ndarray, head_dim: int | None = None) -> dict:
    """Errors of `got` against the oracle `want`, and both bars' verdicts."""
    want = np.asarray(want, dtype=np.float64)
    d = head_dim or want.shape[-1]
    g = _as_f64(got).reshape(-1, d)
    w = want.reshape(-1, d)
    err = np.abs(g - w)
    finite = bool(np.all(np.isfinite(g)))
    floor = np.abs(bf16_round(w) - w)
    rms = np.sqrt(np.mean(w * w, axis=1, keepdims=True))
    bound = 2.0 ** -8 * np.abs(w) + ROW_K * 2.0 ** -8 * rms
    over = err / np.maximum(bound, 1e-300)
    worst = np.unravel_index(int(np.argmax(over)), over.shape) if over.size else (0, 0)
    floor_mean = float(floor.mean()) if floor.size else 0.0
    mean_err = float(err.mean()) if err.size else 0.0
    r = {
        "n": int(err.size),
        "finite": finite,
        "max_abs": float(err.max()) if err.size else 0.0,
        "mean_abs": mean_err,
        "floor_mean": floor_mean,
        "floor_ratio": mean_err / floor_mean if floor_mean > 0 else (0.0 if mean_err == 0 else np.inf),
        "worst_bound_ratio": float(over[worst]) if over.size else 0.0,
        "worst_row": int(worst[0]),
        "worst_col": int(worst[1]),
        "worst_got": float(g[worst]) if over.size else 0.0,
        "worst_want": float(w[worst]) if over.size else 0.0,
        "elements_over_bound": int(np.count_nonzero(err > bound)),
    }
    r["acceptance_ok"] = finite and r["max_abs"] <= MAX_ABS and r["mean_abs"] <= MEAN_ABS
    r["floor_ok"] = (finite and r["elements_over_bound"] == 0 and
                     (floor_mean == 0 and mean_err == 0 or r["floor_ratio"] <= FLOOR_MEAN_K))
    return r


def check(got, want: np.ndarray, what: str = "", head_dim: int | None = None) -> dict:
    """Assert both bars; record the case for the end-of-run summary."""
    r = evaluate(got, want, head_dim)
    RECORDS.append({"what": what, **r})
    assert r["finite"], f"{what}: non-finite output"
    assert r["acceptance_ok"], (f"{what}: max|err| {r['max_abs']:.3e} mean|err| "
                                f"{r['mean_abs']:.3e} (bar {MAX_ABS:g} / {MEAN_ABS:g})")
    assert r["floor_ok"], (
        f"{what}: bf16-floor bar: {r['elements_over_bound']} of {r['n']} elements over "
        f"2^-8|want| + {ROW_K:g}*2^-8*rms(row); worst row {r['worst_row']} col {r['worst_col']} "
        f"got {r['worst_got']:.6g} want {r['worst_want']:.6g} ({r['worst_bound_ratio']:.2f}x "
        f"its bound); mean|err| / floor = {r['floor_ratio']:.2f} (bar {FLOOR_MEAN_K:g})")
    return r


def summary_lines() -> list[str]:
    lines = []
    for r in RECORDS:
        lines.append(f"{r['what'][:58]:58s} n={r['n']:>10d} max={r['max_abs']:.2e} "
                     f"mean={r['mean_abs']:.2e} floor={r['floor_mean']:.2e} "
                     f"ratio={r['floor_ratio']:.2f} worst/bound={r['worst_bound_ratio']:.2f}")
    return lines
