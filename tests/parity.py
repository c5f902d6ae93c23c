"""Element-wise comparison of a CUDA result with the float64 oracle.

Tolerance, against the unrounded float64 oracle on outputs of O(1) scale:
  fp16: max |err| <= 1e-2 and mean |err| <= 1e-3 (the stated bound).
  bf16: the same bound scaled by the ratio of the unit roundoffs,
        2^-8 / 2^-11 = 8: max <= 8e-2, mean <= 8e-3. A bf16 output rounded
        perfectly from the exact value already has a mean error near 1.1e-3
        and a maximum near 1.2e-2 at these sizes, so the unscaled bound is
        below bf16's own rounding floor.
"""
import numpy as np

TOL = {"f16": (1e-2, 1e-3), "bf16": (8e-2, 8e-3)}


def errors(got, ref):
    g = got.detach().float().cpu().double().numpy()
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.isfinite(g).all(), "non-finite values in the CUDA result"
    e = np.abs(g - r)
    return float(e.max()), float(e.mean())


def assert_close(got, ref, dtype, what=""):
    mx, mean = errors(got, ref)
    tmax, tmean = TOL[dtype]
    assert mx <= tmax and mean <= tmean, f"{what}: max|err| {mx:.3e} (<= {tmax}), mean {mean:.3e} (<= {tmean})"
    return mx, mean


def sample_rows(M, n=256, seed=0):
    """Sorted sample of n rows, always with the first and the last."""
    if M <= n:
        return np.arange(M)
    rng = np.random.default_rng([seed, M])
    mid = rng.choice(np.arange(1, M - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, M - 1], mid]))
