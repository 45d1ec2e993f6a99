"""Whole-cache oracle (TEST INFRASTRUCTURE ONLY): layers x requests x kv-heads of streams.

Built only from the plain calls in this package; used by the parity tests to produce
expected INT2 rows, scale/zero words, BF16 sink and ring contents and fp64 decode
outputs from the same seeded inputs the CUDA path receives.
"""
from __future__ import annotations

import numpy as np

from . import Stream, bf16_decode, decode, decode_folded


def as_bits(t) -> np.ndarray:
    """bf16 torch tensor (any device) -> uint16 numpy bit patterns."""
    import torch

    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


class OracleCache:
    """Mixed-precision cache of one workload shape, kept per (layer, request, kv-head)."""

    def __init__(self, n_layers, n_requests, n_kv_heads, head_dim, group, n_sink, window, capacity, R_K, R_V, clip_K,
                 clip_V):
        self.n_layers, self.n_requests, self.Hkv = n_layers, n_requests, n_kv_heads
        self.d, self.g, self.S, self.W = head_dim, group, n_sink, window
        self.R_K = np.asarray(R_K, np.float32)  # [layers, H_kv, d, d]
        self.R_V = np.asarray(R_V, np.float32)
        self.clip_K = np.asarray(clip_K, np.float32)  # [layers, H_kv]
        self.clip_V = np.asarray(clip_V, np.float32)
        cap = capacity if np.ndim(capacity) else [capacity] * n_requests
        self.streams = [[[(Stream(head_dim, group, n_sink, window, cap[r], self.R_K[l, h], self.clip_K[l, h]),
                           Stream(head_dim, group, n_sink, window, cap[r], self.R_V[l, h], self.clip_V[l, h]))
                          for h in range(n_kv_heads)] for r in range(n_requests)] for l in range(n_layers)]

    def append(self, layer: int, request: int, k_bits: np.ndarray, v_bits: np.ndarray) -> None:
        """k_bits, v_bits: uint16 [n, H_kv, d]."""
        for h in range(self.Hkv):
            K, V = self.streams[layer][request][h]
            K.append(np.ascontiguousarray(k_bits[:, h, :]))
            V.append(np.ascontiguousarray(v_bits[:, h, :]))

    def share_prefix(self, dst: int, src: int, n_tokens: int) -> None:
        for l in range(self.n_layers):
            for h in range(self.Hkv):
                for t in range(2):
                    self.streams[l][dst][h][t].share_from(self.streams[l][src][h][t], n_tokens)

    def decode(self, layer: int, request: int, q_bits: np.ndarray) -> np.ndarray:
        """q_bits uint16 [H_q, d] -> fp64 [H_q, d]."""
        Hq = q_bits.shape[0]
        G = Hq // self.Hkv
        out = np.zeros((Hq, self.d))
        for h in range(self.Hkv):
            K, V = self.streams[layer][request][h]
            out[h * G:(h + 1) * G] = decode(np.ascontiguousarray(q_bits[h * G:(h + 1) * G]), K, V, self.R_K[layer, h],
                                            self.R_V[layer, h])
        return out

    def decode_folded(self, layer: int, request: int, qt_bits: np.ndarray) -> np.ndarray:
        """decode() with the rotations folded into the model's projections: qt_bits are the
        rotated queries (uint16 [H_q, d]); fp64 [H_q, d] in the rotated basis."""
        Hq = qt_bits.shape[0]
        G = Hq // self.Hkv
        out = np.zeros((Hq, self.d))
        for h in range(self.Hkv):
            K, V = self.streams[layer][request][h]
            out[h * G:(h + 1) * G] = decode_folded(np.ascontiguousarray(qt_bits[h * G:(h + 1) * G]), K, V)
        return out

    def length(self, request: int) -> int:
        return self.streams[0][request][0][0].length

    def history_end(self, request: int) -> int:
        return self.streams[0][request][0][0].history_end


def bf16_reference(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray) -> np.ndarray:
    """Plain attention over bf16 K, V: q [H_q, d], k and v [L, H_kv, d] -> fp64 [H_q, d]."""
    Hq, d = q_bits.shape
    Hkv = k_bits.shape[1]
    G = Hq // Hkv
    out = np.zeros((Hq, d))
    for h in range(Hkv):
        out[h * G:(h + 1) * G] = bf16_decode(np.ascontiguousarray(q_bits[h * G:(h + 1) * G]),
                                             np.ascontiguousarray(k_bits[:, h, :]),
                                             np.ascontiguousarray(v_bits[:, h, :]))
    return out
