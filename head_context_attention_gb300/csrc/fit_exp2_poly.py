"""Fit the polynomial used for the FMA-pipe exp2 in the attention kernels.

2^x = 2^n * 2^f with n = round(x), f = x - n in [-1/2, 1/2]; 2^f is replaced by
p(f) = 1 + c1 f + c2 f^2 + c3 f^3 (constant term fixed at exactly 1 so that the
clamped input -127 maps to +0.0).  c1..c3 minimise the maximum relative error
on [-1/2, 1/2] (a discrete minimax problem on a dense grid, solved exactly as
a linear program).  Prints the coefficients as float32
literals and the error of the float32 evaluation (Horner, fused multiply-add).

    python fit_exp2_poly.py
"""
import numpy as np


def fit(deg=3, npts=4001):
    """Discrete minimax of the relative error, solved as a linear program:
    minimise E subject to |sum_j c_j x^j / 2^x - (1 - 2^-x)| <= E on a grid."""
    from scipy.optimize import linprog

    xs = np.linspace(-0.5, 0.5, npts)
    A = np.stack([xs ** j for j in range(1, deg + 1)], axis=1) / (2.0 ** xs)[:, None]
    b = 1.0 - 1.0 / 2.0 ** xs
    # variables: c_1..c_deg, E ; rows: A c - E <= b and -A c - E <= -b
    ones = np.ones((npts, 1))
    A_ub = np.vstack([np.hstack([A, -ones]), np.hstack([-A, -ones])])
    b_ub = np.concatenate([b, -b])
    cost = np.zeros(deg + 1)
    cost[-1] = 1.0
    res = linprog(cost, A_ub=A_ub, b_ub=b_ub, bounds=[(None, None)] * (deg + 1), method="highs")
    if not res.success:
        raise RuntimeError(res.message)
    return res.x[:deg].astype(np.float32)


def eval_f32(c, x):
    x = np.asarray(x, dtype=np.float32)
    x = np.maximum(x, np.float32(-127.0))
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    r = (t - magic).astype(np.float32)
    f = (x - r).astype(np.float32)
    p = np.float32(c[2])
    p = (p * f + np.float32(c[1])).astype(np.float32)
    p = (p * f + np.float32(c[0])).astype(np.float32)
    p = (p * f + np.float32(1.0)).astype(np.float32)
    n = (t.view(np.int32) - magic.view(np.int32)).astype(np.int32)
    return (p.view(np.int32) + (n << 23)).view(np.float32)


if __name__ == "__main__":
    c = fit()
    print("coefficients:", ", ".join(f"{v:.9e}f" for v in c))
    xs = np.linspace(-126, 8, 2000001, dtype=np.float64)
    got = eval_f32(c, xs.astype(np.float32)).astype(np.float64)
    ref = np.exp2(xs.astype(np.float32).astype(np.float64))
    rel = np.abs(got / ref - 1.0)
    print(f"max relative error on [-126, 8]: {rel.max():.3e} (2^{np.log2(rel.max()):.2f})")
    print("exp2(-127) ->", eval_f32(c, [-127.0])[0], " exp2(-inf) ->", eval_f32(c, [-np.inf])[0])
