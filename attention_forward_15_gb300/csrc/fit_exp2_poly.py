"""Fit the polynomial the kernel uses for part of its exp2 evaluations.

exp2(x) = 2^j * 2^f with j = round(x) and f = x - j in [-1/2, 1/2]
(Cody-Waite style range reduction; the rounding is done by adding 1.5 * 2^23
in fp32, which leaves round(x) in the low mantissa bits).  2^f is approximated
by the degree-3 polynomial with minimal maximum RELATIVE error on [-1/2, 1/2],
found with the Remez exchange algorithm (equioscillation of the relative
error at n + 2 points).  The coefficients are rounded to fp32 and printed;
they are pasted into attn_fwd_kernel.cuh (kExp2Poly).

    python fit_exp2_poly.py       # prints coefficients and the error bound
"""
import numpy as np


def remez_exp2(n: int, a: float = -0.5, b: float = 0.5, iters: int = 40):
    m = n + 2
    x = 0.5 * (a + b) + 0.5 * (b - a) * np.cos(np.pi * np.arange(m)[::-1] / (m - 1))
    grid = np.linspace(a, b, 400001)
    for _ in range(iters):
        A = np.zeros((m, m))
        for i in range(m):
            A[i, :n + 1] = x[i] ** np.arange(n + 1)
            A[i, n + 1] = -((-1) ** i) * 2.0 ** x[i]
        sol = np.linalg.solve(A, 2.0 ** x)
        c = sol[:n + 1]
        err = (np.polyval(c[::-1], grid) - 2.0 ** grid) / 2.0 ** grid
        sign_change = np.where(np.diff(np.sign(err)) != 0)[0]
        edges = np.concatenate(([0], sign_change + 1, [len(grid)]))
        new_x = [grid[s0 + np.argmax(np.abs(err[s0:s1]))] for s0, s1 in zip(edges[:-1], edges[1:])]
        if len(new_x) != m:
            break
        x = np.array(new_x)
    return c


def max_rel_error_fp32(c32) -> float:
    """Error of the whole fp32 evaluation (reduction + Horner) over x in [-30, 8]."""
    x = np.linspace(-30.0, 8.0, 2000001).astype(np.float32)
    return float(np.max(np.abs(emulate(x, c32) / np.exp2(x.astype(np.float64)) - 1.0)))


def emulate(x, c32):
    """The kernel's steps in fp32 (numpy), for checking the error bound."""
    x = np.maximum(x.astype(np.float32), np.float32(-125.0))
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    j = (t - magic).astype(np.float32)
    f = (x - j).astype(np.float32)
    p = np.float32(c32[3])
    for k in (2, 1, 0):
        p = (p * f + np.float32(c32[k])).astype(np.float32)
    bits = p.view(np.uint32).astype(np.uint64) + (t.view(np.uint32).astype(np.uint64) << np.uint64(23))
    return (bits & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32).astype(np.float64)


if __name__ == "__main__":
    c = remez_exp2(3)
    c32 = [float(np.float32(v)) for v in c]
    print("coefficients (c0..c3):", ", ".join(f"{v:.9g}f" for v in c32))
    print("max relative error (fp32 evaluation, x in [-30, 8]):", max_rel_error_fp32(c32))
