"""Derivation of the 2^f polynomial used by the log-prob kernel (logprob.cu, exp2_poly2).

Fits 2^f on [-1/2, 1/2] with a degree-6 polynomial by least squares of the
relative error on Chebyshev nodes (close to the minimax fit), rounds the
coefficients to fp32 and reports the relative error of the fp32 Horner
evaluation. Run: python fit_exp2_poly.py. Not used at build or run time.
"""
import numpy as np

deg = 6
k = np.arange(4000)
f = 0.5 * np.cos((2 * k + 1) * np.pi / (2 * len(k)))
A = np.vander(f, deg + 1, increasing=True)
c, *_ = np.linalg.lstsq(A / (2.0 ** f)[:, None], np.ones_like(f), rcond=None)  # relative error
c32 = c.astype(np.float32)
print("coefficients (fp32, degree 0..6):", [float(x) for x in c32])
g = np.linspace(-0.5, 0.5, 2000001).astype(np.float32)
p = np.full_like(g, c32[deg])
for j in range(deg - 1, -1, -1):
    p = (p * g + c32[j]).astype(np.float32)
rel = p.astype(np.float64) / 2.0 ** g.astype(np.float64) - 1
exact = np.polyval(c[::-1], g.astype(np.float64)) / 2.0 ** g.astype(np.float64) - 1
print("fit relative error (fp64 coefficients): max %.3g" % np.abs(exact).max())
print("fp32 Horner relative error: max %.3g, mean %.3g" % (np.abs(rel).max(), rel.mean()))
