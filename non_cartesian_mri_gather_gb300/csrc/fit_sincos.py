"""Fit the FMA-pipe polynomial sin/cos used by the gather kernels.

    python non_cartesian_mri_gather_gb300/csrc/fit_sincos.py   # rewrites sincos_poly.cuh

Form.  Phases are in cycles: the kernels need sin(2 pi t) and cos(2 pi t).
A half-period reduction, n = rint(2t) and u = t - n/2 in [-1/4, 1/4] (exact
in float32), gives

    sin(2 pi t) = (-1)^n sin(2 pi u),   cos(2 pi t) = (-1)^n cos(2 pi u)

(a shift by half a period only flips both signs), so only u in [-1/4, 1/4]
has to be approximated.  With w = u^2:

    sin(2 pi u) ~= u * (a0 + a1 w + ... )      cos(2 pi u) ~= b0 + b1 w + ...

Two sets are fitted: a short one for the fast mode's FMA-pipe share of
sin/cos (next to the hardware approximations) and a longer one for the
accurate mode, which uses it for every sin/cos.

Method.  Each polynomial is the discrete minimax (Chebyshev) approximation on
a dense Chebyshev grid of w in [0, 1/16], found by linear programming:
minimise e subject to -e <= weight(w) * (p(w) - f(w)) <= e at every grid
point (absolute error of sin and cos; the weight u turns the sin fit into an
absolute-error fit of u*p).  Coefficients are rounded to float32 one at a
time, from the constant term up, each later coefficient refitted with the
earlier ones held at their float32 values.  The float32 evaluation error of
sin/cos, in the kernels' operation order, is then measured on a dense grid of
t in [-1/2, 1/2] (float32 FMA emulated in float64).  The coefficients come
from this fit only; none is taken from a math library.
"""
from __future__ import annotations

import math
import os

import numpy as np
from scipy.optimize import linprog

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "sincos_poly.cuh")

# (sin coefficients, cos coefficients) of each set
FAST = (4, 5)
ACCURATE = (5, 6)


def minimax(f, weight, degree: int, lo: float, hi: float, fixed=None, n: int = 4000) -> np.ndarray:
    """Coefficients c_0..c_degree (ascending) minimising max |weight*(sum c_j w^j - f)|
    over a Chebyshev grid of [lo, hi], with the coefficients in `fixed` (index ->
    value) held."""
    fixed = fixed or {}
    k = np.arange(n)
    w = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * (k + 0.5) / n)
    w = np.concatenate([[lo, hi], w])
    V = np.vander(w, degree + 1, increasing=True) * weight(w)[:, None]
    r = f(w) * weight(w) - sum(V[:, j] * v for j, v in fixed.items())
    free = [j for j in range(degree + 1) if j not in fixed]
    m = len(free)
    # variables: the free coefficients, e; minimise e
    cost = np.zeros(m + 1)
    cost[-1] = 1.0
    A = np.block([[V[:, free], -np.ones((len(w), 1))], [-V[:, free], -np.ones((len(w), 1))]])
    b = np.concatenate([r, -r])
    res = linprog(cost, A_ub=A, b_ub=b, bounds=[(None, None)] * m + [(0, None)], method="highs")
    assert res.success, res.message
    c = np.zeros(degree + 1)
    for j, v in fixed.items():
        c[j] = v
    c[free] = res.x[:m]
    return c


def minimax_f32(f, weight, degree: int, lo: float, hi: float) -> np.ndarray:
    """minimax() with the coefficients rounded to float32 one at a time."""
    fixed = {}
    for j in range(degree + 1):
        fixed[j] = float(np.float32(minimax(f, weight, degree, lo, hi, fixed)[j]))
    return np.array([fixed[j] for j in range(degree + 1)], dtype=np.float32)


def _sin_over_u(w):  # sin(2 pi u) / u, limit 2 pi at u = 0
    u = np.sqrt(w)
    out = np.full_like(w, 2 * math.pi)
    nz = u > 1e-12
    out[nz] = np.sin(2 * math.pi * u[nz]) / u[nz]
    return out


def fit(n_s: int, n_c: int):
    lo, hi = 0.0, 1.0 / 16.0
    a = minimax_f32(_sin_over_u, lambda w: np.sqrt(w) + 1e-300, n_s - 1, lo, hi)
    b = minimax_f32(lambda w: np.cos(2 * math.pi * np.sqrt(w)), lambda w: np.ones_like(w), n_c - 1, lo, hi)
    return a, b


def fma32(a, b, c):
    return (np.asarray(a, np.float64) * np.asarray(b, np.float64) + np.asarray(c, np.float64)).astype(np.float32)


def mul32(a, b):
    return (np.asarray(a, np.float64) * np.asarray(b, np.float64)).astype(np.float32)


def eval32(t, a, b, leading_fma: bool):
    """float32 evaluation of sin(2 pi t), cos(2 pi t) in the kernels' operation
    order: the half-period reduction, the polynomials (the sin polynomial as
    u * (a0 + w * q) with a final FMA when leading_fma, else by Horner's rule
    and one multiply by u), the sign flip."""
    t = np.asarray(t, np.float32)
    n = np.rint(2.0 * t.astype(np.float64))
    u = fma32(n, -0.5, t)  # exact
    w = mul32(u, u)
    if leading_fma:
        q = np.full_like(w, a[-1])
        for c in a[-2:0:-1]:
            q = fma32(q, w, c)
        s = fma32(a[0], u, mul32(mul32(u, w), q))
    else:
        q = np.full_like(w, a[-1])
        for c in a[-2::-1]:
            q = fma32(q, w, c)
        s = mul32(q, u)
    cpoly = np.full_like(w, b[-1])
    for c in b[-2::-1]:
        cpoly = fma32(cpoly, w, c)
    sign = np.where(np.mod(n, 2) == 0, 1.0, -1.0).astype(np.float32)
    return s * sign, cpoly * sign


def max_err(a, b, leading_fma: bool, n=4_000_001):
    t = np.linspace(-0.5, 0.5, n).astype(np.float32)
    s, c = eval32(t, a, b, leading_fma)
    t64 = t.astype(np.float64)
    return (float(np.max(np.abs(s - np.sin(2 * math.pi * t64)))),
            float(np.max(np.abs(c - np.cos(2 * math.pi * t64)))))


def main():
    sets = {}
    for name, (n_s, n_c), lead in (("Fast", FAST, False), ("Accurate", ACCURATE, True)):
        a, b = fit(n_s, n_c)
        es, ec = max_err(a, b, lead)
        sets[name] = (a, b, es, ec)
        print(f"{name}: sin {n_s} coefficients, cos {n_c}: max |sin err| {es:.3e}  max |cos err| {ec:.3e}")
    fmt = lambda v: f"{float(v):.9e}f"
    body = []
    for name, (a, b, es, ec) in sets.items():
        body.append(f"""// {name.lower()} set: max |sin error| = {es:.3e}, max |cos error| = {ec:.3e}
constexpr int k{name}SinTerms = {len(a)};
constexpr int k{name}CosTerms = {len(b)};
__device__ constexpr float k{name}Sin[k{name}SinTerms] = {{{", ".join(fmt(v) for v in a)}}};
__device__ constexpr float k{name}Cos[k{name}CosTerms] = {{{", ".join(fmt(v) for v in b)}}};""")
    with open(OUT, "w") as f:
        f.write("""// sincos_poly.cuh - GENERATED by fit_sincos.py; do not edit by hand.
//
// sin(2 pi u), cos(2 pi u) for u in [-1/4, 1/4] (cycles, after the
// half-period reduction u = t - rint(2t)/2), w = u^2:
//   sin(2 pi u) ~= u * (a0 + a1 w + ... ),   cos(2 pi u) ~= b0 + b1 w + ...
// Discrete minimax fits (linear programming on a Chebyshev grid), the
// coefficients rounded to float32 one at a time with the rest refitted.
// Errors: float32 evaluation in the kernels' operation order, measured on
// t in [-1/2, 1/2] including the reduction and the sign flip (the accurate
// set's sin polynomial ends in the FMA a0 * u + u * w * (a1 + ...)).
#pragma once

namespace fhd {
namespace poly {
""" + "\n".join(body) + """
}  // namespace poly
}  // namespace fhd
""")
    print("wrote", OUT)


if __name__ == "__main__":
    main()
