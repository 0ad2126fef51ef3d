"""2^x on the FMA pipe: the coefficients the attention kernel uses for part of its softmax
exponentials, and a bit-level CPU model of its fp32 arithmetic.

Method.  Range reduction by the power of two (the base-2 form of Cody and Waite's argument
reduction, which is exact in base 2): x = n + f with n = floor(x) and f in [0, 1), so that
2^x = 2^n * 2^f; 2^n goes into the exponent field with one integer add.  2^f on [0, 1] is a
polynomial of low degree whose coefficients minimise the maximum RELATIVE error, found here with
the Remez exchange algorithm (E. Ya. Remez, 1934): solve for the polynomial that equioscillates
on n+2 reference points, move the references to the extrema of the new error curve, repeat.

The kernel evaluates, per value (fp32, round to nearest unless said otherwise):
    x  = max(x, -126)
    j  = x + 1.5 * 2^23, rounded toward -inf      (the low mantissa bits of j hold floor(x))
    f  = x - (j - 1.5 * 2^23)                     (exact: f in [0, 1))
    p  = ((c3 f + c2) f + c1) f + c0              (Horner, fused multiply-adds)
    2^x ~= bits(p) + (bits(j) << 23)              (integer add into the exponent field)
The clamp keeps the exponent field from wrapping: with x >= -126 the sum above is at worst a
tiny positive subnormal (p(0) = c0 is just below 1), never a NaN; values below 2^-126 do not
matter next to a softmax row whose largest term is near 1.  The fp32 coefficients the kernel
spells out are what `fit()` returns, rounded to fp32.  Run `python -m streaming_causal_video_gb300.exp2_poly` to print them.
"""
import numpy as np

MAGIC = 12582912.0            # 1.5 * 2^23


def fit(degree: int = 3, iters: int = 30, grid: int = 20001):
    """Minimax (relative error) coefficients c0..c_degree of 2^f on [0, 1], by Remez exchange,
    and the maximum relative error of the fp64 polynomial."""
    n = degree
    xs = np.linspace(0.0, 1.0, grid)
    # initial references: Chebyshev extrema mapped to [0, 1]
    ref = 0.5 - 0.5 * np.cos(np.pi * np.arange(n + 2) / (n + 1))
    c = None
    for _ in range(iters):
        # p(x_i) - 2^x_i = (-1)^i E 2^x_i   ->   sum_k c_k x_i^k - (-1)^i E 2^x_i = 2^x_i
        A = np.zeros((n + 2, n + 2))
        for i, x in enumerate(ref):
            A[i, :n + 1] = x ** np.arange(n + 1)
            A[i, n + 1] = -((-1.0) ** i) * 2.0 ** x
        sol = np.linalg.solve(A, 2.0 ** ref)
        c = sol[:n + 1]
        err = np.polyval(c[::-1], xs) / 2.0 ** xs - 1.0
        # new references: the extremum of each run of equal error sign
        sign = np.sign(err)
        bounds = np.flatnonzero(np.diff(sign) != 0) + 1
        runs = np.split(np.arange(grid), bounds)
        ext = [r[np.argmax(np.abs(err[r]))] for r in runs if len(r)]
        if len(ext) != n + 2:
            break
        new_ref = xs[ext]
        if np.allclose(new_ref, ref, atol=1e-12):
            ref = new_ref
            break
        ref = new_ref
    err = np.polyval(c[::-1], xs) / 2.0 ** xs - 1.0
    return [float(v) for v in c], float(np.abs(err).max())


def _f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def _fma_f32(a, b, c):
    """fp32 fused multiply-add: the exact product (48 bits fit in fp64) plus c, rounded once to
    fp64 and then to fp32 (a double rounding; it can differ from one rounding only on
    exact fp64 ties, immaterial for the error bound checked with it)."""
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def model_f32(x, coeffs32):
    """The kernel's fp32 evaluation of 2^x, bit for bit (up to the fma note above), for x <= 127;
    x below -126 is clamped to -126."""
    x = np.maximum(_f32(x), np.float32(-126.0))
    # j = x + MAGIC rounded toward -inf: floor(x) + MAGIC exactly for |x| < 2^22
    j = _f32(np.floor(x.astype(np.float64)) + MAGIC)
    f = (x.astype(np.float64) - (j.astype(np.float64) - MAGIC)).astype(np.float32)
    c = [np.float32(v) for v in coeffs32]
    p = np.full(f.shape, c[-1], np.float32)
    for ck in c[-2::-1]:
        p = _fma_f32(p, f, np.full(f.shape, ck, np.float32))
    bits = (p.view(np.uint32).astype(np.uint64) + ((j.view(np.uint32).astype(np.uint64) << 23) & 0xFFFFFFFF)) \
        & 0xFFFFFFFF
    return bits.astype(np.uint32).view(np.float32)


if __name__ == "__main__":
    for d in (3, 4):
        c, e = fit(d)
        print("degree %d: max relative error %.3e" % (d, e))
        print("  " + ", ".join("%.9ef" % np.float32(v) for v in c))
