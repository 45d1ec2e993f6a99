"""The Hadamard-only rotation switch (the ablation the OSCAR technical summary compares
against, sections 1 and 4): R = H_Had P_br for keys and values, no covariance basis.
CPU checks of both calibrations against an independent construction; the GPU path takes
R as an input, so its parity with these rotations is in the GPU parity tests."""
import math

import numpy as np
import pytest

from int2_rotated_kv_rotate_gb300 import calibrate, workloads as wl
from oracle import calibration as ocal


def _sylvester_bitrev(d):
    # built here from the definitions: H[i][j] = (-1)^popcount(i & j) / sqrt(d), and P_br
    # sends basis vector e_j to e_rev(j), so column j of H P is column rev(j) of H
    bits = d.bit_length() - 1
    H = np.array([[(-1) ** bin(i & j).count("1") for j in range(d)] for i in range(d)], np.float64) / math.sqrt(d)
    rev = [int(format(j, f"0{bits}b")[::-1], 2) for j in range(d)]
    return H[:, rev]


def _calibration_inputs():
    w = wl.scaled(wl.WORKLOADS["tiny"], calib_tokens=256)
    q, k, v = wl.gen_calibration(w, 7, 0)
    return w, q.float().numpy(), k.float().numpy(), v.float().numpy()


def test_oracle_hadamard_only_rotation_is_h_p_and_clips_are_percentiles():
    w, q, k, v = _calibration_inputs()
    RK, RV, cK, cV = ocal.calibrate_layer(q, k, v, w.clip_percentile, rotation="hadamard")
    R = _sylvester_bitrev(q.shape[-1]).astype(np.float32)
    for h in range(k.shape[1]):
        assert np.array_equal(RK[h], R) and np.array_equal(RV[h], R)
        # clip: nearest-rank percentile of |R^T x| over tokens x channels (brute force)
        for X, c in ((k[:, h], cK[h]), (v[:, h], cV[h])):
            a = np.sort(np.abs(X.astype(np.float64) @ R.astype(np.float64)).ravel())
            rank = math.ceil(w.clip_percentile / 100 * a.size - 1e-9)
            assert np.float32(a[rank - 1]) == np.float32(c)


def test_product_hadamard_only_calibration_matches_the_oracle():
    w, q, k, v = _calibration_inputs()
    a = calibrate.calibrate_layer(q, k, v, w.clip_percentile, rotation="hadamard")
    b = ocal.calibrate_layer(q, k, v, w.clip_percentile, rotation="hadamard")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    np.testing.assert_allclose(a[2], b[2], rtol=1e-6)
    np.testing.assert_allclose(a[3], b[3], rtol=1e-6)


def test_the_two_rotations_differ_and_unknown_names_are_rejected():
    w, q, k, v = _calibration_inputs()
    osc = calibrate.calibrate_layer(q, k, v, w.clip_percentile)
    had = calibrate.calibrate_layer(q, k, v, w.clip_percentile, rotation="hadamard")
    assert not np.array_equal(osc[0], had[0])
    with pytest.raises(ValueError):
        calibrate.calibrate_layer(q, k, v, w.clip_percentile, rotation="identity")


def test_product_oscar_calibration_matches_the_oracle():
    """The product's CPU calibration in OSCAR mode (covariance eigenbases) against the
    oracle's: the same rotations to 1e-6 and the same clip thresholds."""
    w = wl.scaled(wl.WORKLOADS["qwen3_8b_layer"], n_q_heads=8, n_kv_heads=2, calib_tokens=1024)
    q, k, v = wl.gen_calibration(w, 17, 3)
    q, k, v = q.float().numpy(), k.float().numpy(), v.float().numpy()
    a = calibrate.calibrate_layer(q, k, v, w.clip_percentile)
    b = ocal.calibrate_layer(q, k, v, w.clip_percentile)
    assert np.abs(a[0] - b[0]).max() < 1e-6 and np.abs(a[1] - b[1]).max() < 1e-6
    np.testing.assert_allclose(a[2], b[2], rtol=1e-6)
    np.testing.assert_allclose(a[3], b[3], rtol=1e-6)
    assert not np.array_equal(a[0], a[1])  # keys and values get their own bases
