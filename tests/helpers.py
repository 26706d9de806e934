"""Shared test helpers: tolerance checks and oracle runs on synthetic inputs."""

import numpy as np

# Forward and backward floating-point outputs must satisfy both bounds.
MAX_ERR_OVER_RMS = 2e-2
REL_FROBENIUS = 5e-3


def err_stats(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    maxerr = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    fro = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    return maxerr, rms, fro


def assert_close(got, ref, name, bf16_rounding=False):
    """Both bounds.  With ``bf16_rounding`` the max bound also allows one bf16
    rounding step of |ref| per element (2^-8 relative): used only where the
    output is so heavy-tailed (a rank-one dW from a single token) that the
    rounding of the largest element to the bf16 output alone exceeds
    2e-2 * rms."""
    maxerr, rms, fro = err_stats(got, ref)
    if bf16_rounding:
        excess = np.abs(np.asarray(got, np.float64) - ref) - (MAX_ERR_OVER_RMS * rms + 2.0 ** -8 * np.abs(ref))
        assert excess.max() <= 0, f"{name}: error beyond 2e-2*rms + one bf16 step"
    else:
        assert maxerr <= MAX_ERR_OVER_RMS * rms, f"{name}: max|err| {maxerr:.3e} > {MAX_ERR_OVER_RMS} * rms {rms:.3e}"
    assert fro <= REL_FROBENIUS, f"{name}: relative Frobenius error {fro:.3e} > {REL_FROBENIUS}"


def assert_codes_match(got, ref, name, min_exact=0.999):
    """E4M3 codes decided from float32 values computed in a different order:
    all within one step of the grid, at least `min_exact` identical."""
    got = np.asarray(got, np.uint8)
    ref = np.asarray(ref, np.uint8)
    assert got.shape == ref.shape, name
    # signed position on the grid: magnitude code with the sign applied
    def ordinal(c):
        m = (c & 0x7F).astype(np.int32)
        return np.where(c & 0x80, -m, m)
    diff = np.abs(ordinal(got) - ordinal(ref))
    # +0 / -0 (0x00 / 0x80) both have ordinal 0
    assert diff.max() <= 1, f"{name}: a code is more than one grid step off"
    exact = float(np.mean(got == ref)) if got.size else 1.0
    zero_sign = np.mean(((got & 0x7F) == 0) & ((ref & 0x7F) == 0) & (got != ref)) if got.size else 0.0
    assert exact + zero_sign >= min_exact, f"{name}: only {exact:.6f} of the codes are identical"


def assert_chain_close(got, ref, name, codes_agree, bf16_rounding=False):
    """A gradient from the GPU's run against the oracle's whole chain, in which
    an FP8-quantised intermediate (dY, or the MLP's dpre) carries the oracle's
    own codes.  Where the two sides' float32 values of that intermediate fall
    on either side of an E4M3 rounding boundary, both codes are correct and
    they differ by one grid step.  One step on a value near the amax is
    amax / 14, and it moves a whole row of the gradient by that times the
    other operand's row: relative to 2e-2 * rms(ref) of a sum over T terms
    that is ~ 15 * amax / (sqrt(T) * rms) of the intermediate, above 1 at a
    few hundred tokens.  The relative Frobenius error of such a step is
    ~ 1 / sqrt(T * N), far inside its bound.  So the Frobenius bound is always
    applied, and the max bound as well when the codes agree everywhere."""
    if codes_agree:
        assert_close(got, ref, name, bf16_rounding)
        return
    _, _, fro = err_stats(got, ref)
    assert fro <= REL_FROBENIUS, f"{name}: relative Frobenius error {fro:.3e} > {REL_FROBENIUS}"

