"""Offline calibration of the rotations and clip thresholds (CPU, fp64).

OSCAR technical summary (gist.science), §2.2-A: from a small calibration set,
  A.1  query-aware key target C_Q = (1/N) sum q^T q and score-aware value target
       C_S = (1/N) V^T S^T S V (S = attention probabilities);
  A.2  eigenbases U_Q, U_S of C_Q and C_S;
  A.3  R_K = U_Q H_Had P_br, R_V = U_S H_Had P_br (Hadamard, then bit-reversal
       permutation to interleave high- and low-variance channels inside groups);
  A.4  per-layer clip thresholds estimated on the rotated calibration activations.
This module produces the inputs of oscar_set_layer_params; it is not on the decode path.
Readings where the page is silent: grouped query heads are pooled per kv-head, S is the
causal softmax of q k^T / sqrt(d), eigenvalues descending with each eigenvector's
largest-magnitude entry positive, H_Had is the Sylvester matrix / sqrt(d), the clip is
the nearest-rank percentile of |R^T x| over all tokens and channels.
"""
from __future__ import annotations

import math

import numpy as np


def sylvester_hadamard(d: int) -> np.ndarray:
    """Normalised Sylvester Hadamard matrix by repeated doubling [[H, H], [H, -H]]."""
    H = np.ones((1, 1))
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    assert H.shape[0] == d, "head_dim must be a power of two"
    return H / math.sqrt(d)


def bit_reversal_order(d: int) -> np.ndarray:
    """perm[j] = j with its log2(d) bits reversed."""
    bits = int(math.log2(d))
    j = np.arange(d)
    out = np.zeros(d, dtype=np.int64)
    for b in range(bits):
        out |= ((j >> b) & 1) << (bits - 1 - b)
    return out


def rotation_from_eigenbasis(U: np.ndarray) -> np.ndarray:
    """R = U H P_br; P_br sends e_j to e_rev(j), so column j of R is column rev(j) of U H."""
    UH = U @ sylvester_hadamard(U.shape[0])
    return UH[:, bit_reversal_order(U.shape[0])]


def sorted_eigenbasis(C: np.ndarray) -> np.ndarray:
    vals, vecs = np.linalg.eigh(C)
    vecs = vecs[:, ::-1]
    pivot = np.abs(vecs).argmax(axis=0)
    signs = np.sign(vecs[pivot, np.arange(vecs.shape[1])])
    signs[signs == 0] = 1.0
    return vecs * signs


def causal_attention_outputs(Qh: np.ndarray, K: np.ndarray, V: np.ndarray, block: int = 256) -> np.ndarray:
    """O = softmax_causal(Qh K^T / sqrt(d)) V for one query head, in row blocks."""
    n, d = Qh.shape
    out = np.empty((n, V.shape[1]))
    inv = 1.0 / math.sqrt(d)
    for r0 in range(0, n, block):
        r1 = min(n, r0 + block)
        logits = (Qh[r0:r1] @ K[:r1].T) * inv
        rows = np.arange(r0, r1)[:, None]
        logits[np.arange(r1)[None, :] > rows] = -np.inf
        logits -= logits.max(axis=1, keepdims=True)
        w = np.exp(logits)
        w /= w.sum(axis=1, keepdims=True)
        out[r0:r1] = w @ V[:r1]
    return out


def nearest_rank(values: np.ndarray, percentile: float) -> float:
    flat = np.asarray(values, dtype=np.float64).ravel()
    # rank = ceil(p/100 * n) evaluated on the decimal percentile (99.9 -> 999/10 exactly)
    num, den = _decimal_ratio(percentile)
    k = max(1, -(-(num * flat.size) // (den * 100)))
    return float(np.partition(flat, k - 1)[k - 1])


def _decimal_ratio(p: float):
    text = repr(float(p))
    if "e" in text or "E" in text:
        return float(p).as_integer_ratio()
    whole, _, frac = text.partition(".")
    den = 10 ** len(frac)
    return int(whole + frac), den


ROTATIONS = ("oscar", "hadamard")


def _check_rotation(rotation: str) -> None:
    if rotation not in ROTATIONS:
        raise ValueError(f"rotation must be one of {ROTATIONS}, not {rotation!r}")


def calibrate_kv_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, percentile: float = 99.9,
                      rotation: str = "oscar"):
    """q [N, G, d], k and v [N, d] -> (R_K, R_V) fp32 [d, d], (clip_K, clip_V) fp32.
    rotation "oscar": R = U H P with U the sorted eigenbasis of C_Q (keys) or C_S (values);
    "hadamard": the ablation without the covariance basis, R = H P for both (the
    Hadamard-only rotation that the OSCAR technical summary compares against, sections 1
    and 4)."""
    _check_rotation(rotation)
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n, G, d = q.shape
    if rotation == "hadamard":
        R_K = R_V = rotation_from_eigenbasis(np.eye(d)).astype(np.float32)
    else:
        flat_q = q.reshape(n * G, d)
        C_Q = np.einsum("ni,nj->ij", flat_q, flat_q) / (n * G)
        C_S = np.zeros((d, d))
        for h in range(G):
            O = causal_attention_outputs(q[:, h, :], k, v)
            C_S += O.T @ O
        C_S /= n * G
        R_K = rotation_from_eigenbasis(sorted_eigenbasis(C_Q)).astype(np.float32)
        R_V = rotation_from_eigenbasis(sorted_eigenbasis(C_S)).astype(np.float32)
    clip_K = np.float32(nearest_rank(np.abs(k @ R_K.astype(np.float64)), percentile))
    clip_V = np.float32(nearest_rank(np.abs(v @ R_V.astype(np.float64)), percentile))
    return R_K, R_V, clip_K, clip_V


def calibrate_layer(q, k, v, percentile: float = 99.9, rotation: str = "oscar"):
    """q [N, H_q, d], k and v [N, H_kv, d] (array-like) -> R_K, R_V [H_kv, d, d],
    clip_K, clip_V [H_kv] (fp32 numpy).  rotation: "oscar" or "hadamard" (the ablation)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    Hkv = k.shape[1]
    G = q.shape[1] // Hkv
    d = q.shape[2]
    RK = np.empty((Hkv, d, d), np.float32)
    RV = np.empty((Hkv, d, d), np.float32)
    cK = np.empty(Hkv, np.float32)
    cV = np.empty(Hkv, np.float32)
    for h in range(Hkv):
        RK[h], RV[h], cK[h], cV[h] = calibrate_kv_head(q[:, h * G:(h + 1) * G], k[:, h], v[:, h], percentile,
                                                       rotation)
    return RK, RV, cK, cV


def clip_rank(n_values: int, percentile: float) -> int:
    """1-based nearest rank of a percentile among n values: ceil(p / 100 * n), evaluated on
    the decimal percentile (99.9 is 999/10 exactly)."""
    num, den = _decimal_ratio(percentile)
    return max(1, -(-(num * n_values) // (den * 100)))


def calibrate_layer_gpu(q, k, v, percentile: float = 99.9, rotation: str = "oscar", covariances: bool = False):
    """The same calibration on the GPU, in fp64, by the library's CUDA kernels
    (oscar_calibrate_layer: covariances, causal attention, Jacobi eigenbases, R = U H P,
    radix-selected clip).  q [N, H_q, d], k and v [N, H_kv, d] bf16 torch tensors on the
    device.  Returns fp32 numpy R_K, R_V [H_kv, d, d] and clip_K, clip_V [H_kv] (and, with
    covariances=True, the fp64 covariances [2 H_kv, d, d] as a torch tensor: C_Q of every
    kv-head, then C_S)."""
    import torch

    from . import _native as N

    _check_rotation(rotation)
    q, k, v = (t.to(torch.bfloat16).contiguous() for t in (q, k, v))
    n, hq, d = q.shape
    hkv = k.shape[1]
    dev = q.device
    ws = torch.empty(N.oscar_calibration_workspace_bytes(n, hq, hkv), dtype=torch.uint8, device=dev)
    RK = torch.empty((hkv, d, d), dtype=torch.float32, device=dev)
    RV = torch.empty_like(RK)
    cK = torch.empty(hkv, dtype=torch.float32, device=dev)
    cV = torch.empty_like(cK)
    C = torch.zeros((2 * hkv, d, d), dtype=torch.float64, device=dev) if covariances else None
    N.oscar_calibrate_layer(q, k, v, clip_rank(n * d, percentile),
                            N.OSCAR_ROTATION_HADAMARD if rotation == "hadamard" else N.OSCAR_ROTATION_OSCAR,
                            RK, RV, cK, cV, ws, covariances=C)
    out = (RK.cpu().numpy(), RV.cpu().numpy(), cK.cpu().numpy(), cV.cpu().numpy())
    return out + (C,) if covariances else out
