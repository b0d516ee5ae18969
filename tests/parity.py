"""Parity bars used by the GPU tests.

fp32: max abs error <= 1e-4 against the fp64 oracle.
bf16: max abs error <= 2e-2 and per-row cosine >= 0.999, one row being one
(token, head) vector of head_dim elements (the pages' parity bar is cosine >=
0.999 on outputs: page "packed-encoders 0.1.0", section "Benchmarks").
Gradients (check_grad): the same, except that the cosine bar skips rows whose
exact norm is below a tenth of the tensor's median row norm. Such a row is a
near-cancellation of terms whose bf16 rounding (P and dS before the MMAs, and
the bf16 output that Delta = rowsum(dO o O) is formed from) exceeds the row
itself, so its direction is not determined at bf16; it keeps the absolute bar.
"""

import numpy as np

FP32_ATOL = 1e-4
BF16_ATOL = 2e-2
BF16_COS = 0.999


def to64(t):
    if hasattr(t, "detach"):
        return t.detach().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


def row_cosine(got, want):
    got = got.reshape(-1, got.shape[-1])
    want = want.reshape(-1, want.shape[-1])
    num = np.sum(got * want, axis=1)
    den = np.linalg.norm(got, axis=1) * np.linalg.norm(want, axis=1)
    cos = np.where(den > 0, num / np.where(den > 0, den, 1.0), 1.0)
    # Rows whose reference is exactly zero compare by absolute error only.
    return cos


def check(got, want, dtype: str, what: str = "", cos_min_norm_frac: float = 0.0):
    got, want = to64(got), to64(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = float(np.abs(got - want).max()) if got.size else 0.0
    if dtype == "fp32":
        assert err <= FP32_ATOL, f"{what}: max abs error {err:.3e} > {FP32_ATOL}"
        return {"max_abs": err}
    assert err <= BF16_ATOL, f"{what}: max abs error {err:.3e} > {BF16_ATOL}"
    cos = row_cosine(got, want)
    if cos_min_norm_frac > 0 and cos.size:
        norms = np.linalg.norm(want.reshape(-1, want.shape[-1]), axis=1)
        cos = cos[norms >= cos_min_norm_frac * np.median(norms)]
    worst = float(cos.min()) if cos.size else 1.0
    assert worst >= BF16_COS, f"{what}: min per-row cosine {worst:.6f} < {BF16_COS}"
    return {"max_abs": err, "min_cos": worst}


GRAD_COS_MIN_NORM_FRAC = 0.1


def check_grad(got, want, dtype: str, what: str = ""):
    return check(got, want, dtype, what, cos_min_norm_frac=GRAD_COS_MIN_NORM_FRAC)
