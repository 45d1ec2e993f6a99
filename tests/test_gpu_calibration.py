"""The GPU calibration (oscar_calibrate_layer, through the C ABI) against the oracle's
fp64 numpy calibration, on the same seeded activations:

- the covariances C_Q and C_S (A.1) to 1e-10 relative (fp64 on both sides, different
  summation orders);
- the rotations R_K = U_Q H P and R_V = U_S H P (A.2, A.3) to 1e-6 (both rounded to fp32
  from fp64 eigenbases: Jacobi on the GPU, LAPACK in the oracle);
- the clip thresholds (A.4) to 1e-6 relative (the same order statistic);
- the Hadamard-only rotation exactly.
"""
import numpy as np
import pytest
import torch

from int2_rotated_kv_rotate_gb300 import calibrate, workloads as wl
from oracle import calibration as ocal

pytestmark = pytest.mark.gpu

SEED = 31


def _inputs(w, layer):
    q, k, v = wl.gen_calibration(w, SEED, layer, device="cuda")
    return (q, k, v), (q.float().cpu().numpy(), k.float().cpu().numpy(), v.float().cpu().numpy())


@pytest.mark.parametrize("name,gqa,tokens", [("g4", 4, 2048), ("g8", 8, 512), ("ragged_n", 4, 777)])
def test_gpu_calibration_matches_the_oracle(name, gqa, tokens):
    w = wl.scaled(wl.WORKLOADS["qwen3_8b_layer"], name=f"calib_{name}", n_q_heads=2 * gqa, n_kv_heads=2,
                  calib_tokens=tokens)
    dev, host = _inputs(w, 1)
    RK, RV, cK, cV, C = calibrate.calibrate_layer_gpu(*dev, w.clip_percentile, covariances=True)
    q, k, v = host
    G = w.gqa
    C = C.cpu().numpy()
    for h in range(w.n_kv_heads):
        qh = q[:, h * G:(h + 1) * G]
        cq = ocal.query_covariance(qh)
        cs = ocal.score_value_covariance(qh, k[:, h], v[:, h])
        for got, ref, what in ((C[h], cq, "C_Q"), (C[w.n_kv_heads + h], cs, "C_S")):
            err = np.abs(got - ref).max() / np.abs(ref).max()
            assert err < 1e-10, f"{name} head {h} {what}: relative error {err:.2e}"
    oRK, oRV, ocK, ocV = ocal.calibrate_layer(q, k, v, w.clip_percentile)
    assert np.abs(RK - oRK).max() < 1e-6 and np.abs(RV - oRV).max() < 1e-6
    np.testing.assert_allclose(cK, ocK, rtol=1e-6)
    np.testing.assert_allclose(cV, ocV, rtol=1e-6)
    for R in list(RK) + list(RV):
        R64 = R.astype(np.float64)
        assert np.abs(R64.T @ R64 - np.eye(128)).max() < 1e-6


def test_gpu_hadamard_only_calibration_is_exact():
    w = wl.scaled(wl.WORKLOADS["qwen3_8b_layer"], name="calib_had", n_q_heads=8, n_kv_heads=2, calib_tokens=1000)
    dev, host = _inputs(w, 0)
    RK, RV, cK, cV = calibrate.calibrate_layer_gpu(*dev, w.clip_percentile, rotation="hadamard")
    oRK, oRV, ocK, ocV = ocal.calibrate_layer(*host, w.clip_percentile, rotation="hadamard")
    assert np.array_equal(RK, oRK) and np.array_equal(RV, oRV)
    np.testing.assert_allclose(cK, ocK, rtol=1e-7)
    np.testing.assert_allclose(cV, ocV, rtol=1e-7)


def test_gpu_calibration_of_a_benchmark_layer():
    """The 32B-shaped capacity workload's layer shape (64 query / 8 kv heads, 2048 tokens),
    as the benchmark calibrates it: rotations and clips against the oracle."""
    w = wl.WORKLOADS["qwen3_32b_capacity"]
    dev, host = _inputs(w, 5)
    RK, RV, cK, cV = calibrate.calibrate_layer_gpu(*dev, w.clip_percentile)
    torch.cuda.synchronize()
    oRK, oRV, ocK, ocV = ocal.calibrate_layer(*host, w.clip_percentile)
    assert np.abs(RK - oRK).max() < 1e-6 and np.abs(RV - oRV).max() < 1e-6
    np.testing.assert_allclose(cK, ocK, rtol=1e-6)
    np.testing.assert_allclose(cV, ocV, rtol=1e-6)
