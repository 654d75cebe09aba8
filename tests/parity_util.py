"""Comparison helpers shared by the GPU parity tests (no attention arithmetic here).

Tolerances for bf16 / fp16 / fp32(TF32) inputs with fp32 accumulation, against
the fp64 oracle: max |dO| <= 2e-2, mean |dO| <= 2e-3, |dlse| <= 1e-2 on finite
rows; a row the oracle reports as fully masked (lse = -inf) must come back with
lse = -inf and O = 0 exactly.
"""
import numpy as np

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_ABS = 1e-2


def compare(out, lse, ref_o, ref_l, o_max=O_MAX_ABS, o_mean=O_MEAN_ABS, lse_abs=LSE_ABS):
    """out/lse: GPU results (torch or numpy) for the same rows as ref_o/ref_l."""
    o = np.asarray(out.float().cpu().double().numpy() if hasattr(out, "cpu") else out, dtype=np.float64)
    l = np.asarray(lse.cpu().double().numpy() if hasattr(lse, "cpu") else lse, dtype=np.float64)
    ref_o = np.asarray(ref_o, dtype=np.float64)
    ref_l = np.asarray(ref_l, dtype=np.float64)
    assert o.shape == ref_o.shape and l.shape == ref_l.shape
    assert not np.isnan(o).any(), "NaN in O"
    assert not np.isnan(l).any(), "NaN in lse"
    masked = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(l), masked), "fully masked rows differ"
    if masked.any():
        assert np.all(o[masked] == 0.0), "fully masked rows must give O = 0"
    err = np.abs(o - ref_o)
    dl = np.abs(l[~masked] - ref_l[~masked]) if (~masked).any() else np.zeros(1)
    stats = {"o_max": float(err.max()) if err.size else 0.0, "o_mean": float(err.mean()) if err.size else 0.0,
             "lse_max": float(dl.max())}
    assert stats["o_max"] <= o_max, stats
    assert stats["o_mean"] <= o_mean, stats
    assert stats["lse_max"] <= lse_abs, stats
    return stats
