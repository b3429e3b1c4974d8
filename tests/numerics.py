"""Tolerances of the MoE block's floating-point outputs.

The bar (stated for the block's outputs): max |err| <= 2e-2 * rms(ref) and
mean relative error <= 2e-3, the mean relative error taken normwise,
sum|got - ref| / sum|ref|, against the float64 oracle before any rounding.
The same bar is applied to the router logits and routing weights."""
import numpy as np

MAX_ABS_VS_RMS = 2e-2
MEAN_REL = 2e-3


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(err.max()) / max(rms, 1e-300), float(err.sum()) / max(float(np.abs(ref).sum()), 1e-300)


def assert_close(got, ref, what=""):
    max_rel_rms, mean_rel = errors(got, ref)
    assert max_rel_rms <= MAX_ABS_VS_RMS and mean_rel <= MEAN_REL, (
        f"{what}: max|err|/rms = {max_rel_rms:.3e} (bar {MAX_ABS_VS_RMS}), "
        f"mean rel = {mean_rel:.3e} (bar {MEAN_REL})")
    return max_rel_rms, mean_rel


def bf16_bits_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
