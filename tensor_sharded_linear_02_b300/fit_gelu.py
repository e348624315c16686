"""Derives the constants of the epilogue's normal-tail function (run by
hand; prints C constants; not used at build or run time).

The epilogue needs h(x) = Phi(-|x|) = erfc(z) / 2, z = |x| / sqrt(2), with
an error small RELATIVE to h over the whole range (GeLU(x) = x h for x < 0
shrinks like exp(-x^2 / 2)).  It uses the functional form of the
Chebyshev-fitted complementary error function in Press, Teukolsky,
Vetterling & Flannery, "Numerical Recipes in C", 2nd ed., section 6.2:

    erfc(z) = t exp(-z^2 + P(t)),   t = 1 / (1 + z / 2),

where P is a polynomial.  As z runs over [0, inf), t runs over (0, 1] and
f(t) = ln(erfc(z) exp(z^2) / t) is smooth on [0, 1] (it tends to
-ln(2 sqrt(pi) (1 - t)) ... at t -> 0 through the asymptote
erfc(z) exp(z^2) ~ 1 / (z sqrt(pi))), so a low-degree polynomial fits it.
The fit here is a least-squares Chebyshev fit of degree DEG over t in
[T_MIN, 1] (z up to about 20, x up to about 28, beyond the range where
h is above fp32's smallest normal), converted to the power basis and folded
for the kernel's base-2 exponential and the factor 1/2:

    h = t * 2^(G(t) - x^2 * log2(e) / 2),   G(t) = log2(e) (P(t) - ln 2).

Written with scipy's erfcx (scaled complementary error function) as the
reference.
"""
import numpy as np
from scipy.special import erfc, erfcx

DEG = 7
T_MIN = 0.09
LOG2E = 1.0 / np.log(2.0)


def fit():
    k = np.arange(20001)
    t = 0.5 * (1 - np.cos(np.pi * (k + 0.5) / k.size)) * (1 - T_MIN) + T_MIN  # Chebyshev nodes
    z = 2.0 * (1.0 / t - 1.0)
    f = np.log(erfcx(z) / t)
    cheb = np.polynomial.chebyshev.Chebyshev.fit(t, f, DEG, domain=[T_MIN, 1.0])
    P = cheb.convert(kind=np.polynomial.Polynomial, domain=[T_MIN, 1.0], window=[T_MIN, 1.0])
    p = P.coef.copy()
    g = LOG2E * p
    g[0] -= 1.0
    return g


def h_model(x, g):
    """h from the folded form, in double."""
    u = np.abs(x)
    t = 1.0 / (1.0 + u / (2.0 * np.sqrt(2.0)))
    G = np.polynomial.polynomial.polyval(t, g)
    return t * np.exp2(G - x * x * LOG2E / 2.0)


if __name__ == "__main__":
    g = fit()
    x = np.linspace(0, 26, 2000001)
    ref = 0.5 * erfc(x / np.sqrt(2.0))
    rel = np.abs(h_model(x, g) - ref) / ref
    print(f"// degree {DEG}, t in [{T_MIN}, 1]: max relative error of h in double "
          f"{rel.max():.2e} (x = {x[rel.argmax()]:.3f}) over |x| <= 26")
    for i, c in enumerate(g):
        print(f"constexpr float GELU_G{i} = {float(np.float32(c)):.9e}f;  // {float(c):.17e}")
