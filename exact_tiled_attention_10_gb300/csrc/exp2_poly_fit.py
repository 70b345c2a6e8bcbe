"""Derives the coefficients of the polynomial exp2 used by the forward softmax.

Method (textbook range reduction + minimax approximation):
    2^x = 2^r * 2^f,   r = round(x) (an integer),   f = x - r in [-1/2, 1/2]
and 2^f is approximated on [-1/2, 1/2] by the degree-3 polynomial
    q(f) = c0 + c1 f + c2 f^2 + c3 f^3
that minimises the maximum RELATIVE error max |q(f) / 2^f - 1|.  The minimax
polynomial is found with the Remez exchange algorithm on the weighted error
e(f) = (q(f) - 2^f) / 2^f, in float64.  2^r is applied by adding r to the
float32 exponent field, so the overall relative error is that of q.

Run:  python exp2_poly_fit.py      (prints the coefficients and the error)
The printed values are the constants kExp2C0..C3 in ptx.cuh.
"""
import numpy as np

DEG = 3
A, B = -0.5, 0.5


def remez(deg=DEG, iters=40):
    n = deg + 2
    # initial reference: Chebyshev extrema mapped to [A, B]
    k = np.arange(n)
    ref = (A + B) / 2 + (B - A) / 2 * np.cos(np.pi * k[::-1] / (n - 1))
    grid = np.linspace(A, B, 200001)
    f = lambda x: np.exp2(x)
    for _ in range(iters):
        # solve  sum_i c_i x_j^i - f(x_j) = (-1)^j E f(x_j)   for c, E
        M = np.zeros((n, n))
        for j, x in enumerate(ref):
            M[j, :deg + 1] = x ** np.arange(deg + 1)
            M[j, deg + 1] = -((-1) ** j) * f(x)
        sol = np.linalg.solve(M, f(ref))
        c, E = sol[:deg + 1], sol[deg + 1]
        err = (np.polyval(c[::-1], grid) - f(grid)) / f(grid)
        # new reference: extrema of the error between sign changes
        sign = np.sign(err)
        idx = np.where(np.diff(sign) != 0)[0]
        bounds = np.concatenate([[0], idx + 1, [len(grid)]])
        ext = [seg[np.argmax(np.abs(err[seg]))] for seg in
               (np.arange(bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1))]
        ext = np.array(ext)
        if len(ext) > n:  # keep the n largest alternating points
            while len(ext) > n:
                drop = np.argmin(np.abs(err[ext]))
                ext = np.delete(ext, drop)
        if len(ext) == n:
            ref = grid[ext]
    return c, np.max(np.abs(err))


if __name__ == "__main__":
    c, e = remez()
    for i, ci in enumerate(c):
        print("c%d = %.9e" % (i, ci))
    print("max relative error on [-1/2, 1/2]: %.3e" % e)
    # the same error with the coefficients rounded to float32 and Horner in float32
    cf = c.astype(np.float32)
    x = np.linspace(A, B, 100001).astype(np.float32)
    q = cf[3]
    for ci in (cf[2], cf[1], cf[0]):
        q = (q * x + ci).astype(np.float32)
    print("float32 Horner max relative error: %.3e" % np.max(np.abs(q / np.exp2(x.astype(np.float64)) - 1)))
