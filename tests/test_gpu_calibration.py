"""The calibration study on a small case: errors finite and bounded, FP8
closer to FP32 than NVFP4 on every distribution, and on sparse x20 outliers
the amax-based global scale at least as good as a scale four times smaller
(which saturates the outliers)."""
import pytest

pytestmark = pytest.mark.gpu


def test_calibration_study_small():
    from nvfp4_quantized_paged_gb300.calibration import study
    rows = study(device="cuda", B=2, L=1024, Hq=8, Hkv=2, factors=(0.25, 1.0, 4.0))
    assert len(rows) == 4 * (1 + 3)
    for r in rows:
        assert r["cache_err"] == 0
        assert 0.0 < r["rel_l2"] < float("inf"), r
        if r["factor"] == 1.0:  # the amax rule; moved scales may saturate (x0.25 on outliers: ~0.7)
            assert r["rel_l2"] < 0.5, r
    by = {(r["dist"], r["prec"], r["factor"]): r["rel_l2"] for r in rows}
    for d in ("normal", "element_outliers", "channel_outliers", "lognormal_channels"):
        assert by[(d, "fp8", 1.0)] < by[(d, "nvfp4", 1.0)], d
    assert by[("element_outliers", "nvfp4", 1.0)] <= by[("element_outliers", "nvfp4", 0.25)]
