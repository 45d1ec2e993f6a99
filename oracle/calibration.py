"""Offline calibration, oracle side (TEST INFRASTRUCTURE ONLY): plain numpy, fp64.

Follows the offline phase of the OSCAR technical summary, section 2.2-A, step by step:
  A.1  C_Q = (1/N) sum_n q_n^T q_n          (query-aware key target)
       C_S = (1/N) V^T S^T S V             (score-aware value target, S = attention probs)
  A.2  eigendecomposition of C_Q, C_S  ->  eigenbases U_Q, U_S
  A.3  R_K = U_Q H_Had P_br,  R_V = U_S H_Had P_br
  A.4  per-layer clip thresholds estimated on the rotated calibration activations
Readings where the page is silent: with grouped-query attention the G query heads of a
kv-head are pooled (N counts token x head pairs); S is the causal softmax of
q k^T / sqrt(d); eigenvalues are sorted descending and each eigenvector's largest-|.|
entry is made positive; H_Had is the full-size Sylvester matrix scaled by 1/sqrt(d);
P_br maps basis vector e_j to e_rev(j); the clip is the nearest-rank percentile of
|R^T x| over every token and channel of the calibration set.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np


def hadamard(d: int) -> np.ndarray:
    """Normalised Sylvester Hadamard matrix: H[i, j] = (-1)^popcount(i & j) / sqrt(d)."""
    assert d & (d - 1) == 0
    i = np.arange(d)[:, None]
    j = np.arange(d)[None, :]
    parity = np.vectorize(lambda v: bin(int(v)).count("1") & 1)(i & j)
    return (1.0 - 2.0 * parity) / math.sqrt(d)


def bit_reverse(j: int, bits: int) -> int:
    out = 0
    for _ in range(bits):
        out = (out << 1) | (j & 1)
        j >>= 1
    return out


def bitrev_permutation(d: int) -> np.ndarray:
    """P_br as a matrix: column j is the basis vector e_rev(j)."""
    bits = d.bit_length() - 1
    P = np.zeros((d, d))
    for j in range(d):
        P[bit_reverse(j, bits), j] = 1.0
    return P


def query_covariance(Q: np.ndarray) -> np.ndarray:
    """C_Q from queries Q [N, G, d] of one kv-head: mean of q^T q over all N*G rows."""
    X = Q.reshape(-1, Q.shape[-1]).astype(np.float64)
    return X.T @ X / X.shape[0]


def attention_probs(Qh: np.ndarray, K: np.ndarray) -> np.ndarray:
    """Causal softmax(q k^T / sqrt(d)) for one query head: [N, N]."""
    d = Qh.shape[-1]
    logits = Qh.astype(np.float64) @ K.astype(np.float64).T / math.sqrt(d)
    N = logits.shape[0]
    logits[np.triu_indices(N, k=1)] = -np.inf
    logits -= logits.max(axis=1, keepdims=True)
    e = np.exp(logits)
    return e / e.sum(axis=1, keepdims=True)


def score_value_covariance(Q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """C_S = (1/(G N)) sum_h V^T S_h^T S_h V for the G query heads sharing K, V."""
    N, G, d = Q.shape
    Vd = V.astype(np.float64)
    C = np.zeros((d, d))
    for h in range(G):
        S = attention_probs(Q[:, h, :], K)
        O = S @ Vd
        C += O.T @ O
    return C / (G * N)


def eig_desc(C: np.ndarray):
    """Eigenvalues descending, eigenvectors as columns, largest-|.| entry positive."""
    w, U = np.linalg.eigh(C)
    order = np.argsort(w)[::-1]
    w, U = w[order], U[:, order].copy()
    for k in range(U.shape[1]):
        i = int(np.argmax(np.abs(U[:, k])))
        if U[i, k] < 0:
            U[:, k] = -U[:, k]
    return w, U


def compose_rotation(U: np.ndarray) -> np.ndarray:
    """R = U H_Had P_br (fp64)."""
    d = U.shape[0]
    return U @ hadamard(d) @ bitrev_permutation(d)


def nearest_rank_percentile(values: np.ndarray, pct: float) -> float:
    """Nearest-rank percentile: the ceil(pct/100 * n)-th smallest value (1-based)."""
    v = np.sort(np.asarray(values, dtype=np.float64).reshape(-1))
    n = v.size
    # exact decimal arithmetic: 99.9 / 100 * 1000 must be 999, not 999.0000000000001
    rank = max(1, math.ceil(Fraction(repr(float(pct))) / 100 * n))
    return float(v[rank - 1])


def clip_threshold(R: np.ndarray, X: np.ndarray, pct: float) -> float:
    """Percentile of |R^T x| over tokens x channels; X [N, d] in the original basis."""
    rotated = X.astype(np.float64) @ R.astype(np.float64)
    return nearest_rank_percentile(np.abs(rotated), pct)


def calibrate_head(Q: np.ndarray, K: np.ndarray, V: np.ndarray, pct: float, rotation: str = "oscar"):
    """(R_K, R_V, clip_K, clip_V) for one kv-head; Q [N, G, d], K and V [N, d] (float).
    rotation "hadamard" is the ablation without the covariance eigenbasis (U = I): the
    Hadamard-only rotation of the OSCAR technical summary's sections 1 and 4."""
    if rotation == "hadamard":
        U_Q = U_S = np.eye(Q.shape[-1])
    else:
        _, U_Q = eig_desc(query_covariance(Q))
        _, U_S = eig_desc(score_value_covariance(Q, K, V))
    R_K = compose_rotation(U_Q).astype(np.float32)
    R_V = compose_rotation(U_S).astype(np.float32)
    clip_K = np.float32(clip_threshold(R_K, K, pct))
    clip_V = np.float32(clip_threshold(R_V, V, pct))
    return R_K, R_V, float(clip_K), float(clip_V)


def calibrate_layer(Q: np.ndarray, K: np.ndarray, V: np.ndarray, pct: float, rotation: str = "oscar"):
    """Per kv-head calibration of one layer.  Q [N, H_q, d]; K, V [N, H_kv, d].

    Returns R_K, R_V fp32 [H_kv, d, d] and clip_K, clip_V fp32 [H_kv].
    """
    N, Hq, d = Q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    RK = np.zeros((Hkv, d, d), np.float32)
    RV = np.zeros((Hkv, d, d), np.float32)
    cK = np.zeros(Hkv, np.float32)
    cV = np.zeros(Hkv, np.float32)
    for h in range(Hkv):
        RK[h], RV[h], cK[h], cV[h] = calibrate_head(Q[:, h * G:(h + 1) * G, :], K[:, h, :], V[:, h, :], pct,
                                                    rotation)
    return RK, RV, cK, cV
