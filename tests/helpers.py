"""Shared test helpers: build the CUDA cache and the oracle cache from the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

from int2_rotated_kv_rotate_gb300 import KVCache, workloads as wl
from int2_rotated_kv_rotate_gb300 import _native as N
from oracle import calibration as ocal
from oracle.model import OracleCache, as_bits

# tolerance on decode outputs (fp32 output vs the oracle's fp64 attention on the same
# dequantised values): max-abs and relative L2 error
MAX_ABS = 2e-2
REL_L2 = 5e-3


def oracle_params(w: wl.Workload, seed: int, n_layers: int, rotation: str = "oscar"):
    """Rotations and clips per layer from the oracle's calibration (inputs to both sides)."""
    RK, RV, cK, cV = [], [], [], []
    for layer in range(n_layers):
        q, k, v = wl.gen_calibration(w, seed, layer)
        a, b, c, d = ocal.calibrate_layer(q.float().numpy(), k.float().numpy(), v.float().numpy(), w.clip_percentile,
                                          rotation=rotation)
        RK.append(a)
        RV.append(b)
        cK.append(c)
        cV.append(d)
    return np.stack(RK), np.stack(RV), np.stack(cK), np.stack(cV)


def make_pair(w: wl.Workload, seed: int, n_layers: int, n_requests: int, max_len: int, fmt=N.OSCAR_FORMAT_INT2,
              params=None, extra_pages: int = 8):
    ppr = (max_len + 63) // 64 + 1
    cache = KVCache(fmt=fmt, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, group=w.group, n_sink=w.n_sink,
                    window=w.window, n_layers=n_layers, max_requests=n_requests,
                    max_pages=n_requests * ppr + extra_pages, max_pages_per_request=ppr)
    int2 = fmt in (N.OSCAR_FORMAT_INT2, N.OSCAR_FORMAT_INT2_CM)
    if params is None and int2:
        params = oracle_params(w, seed, n_layers)
    oc = None
    if int2:
        RK, RV, cK, cV = params
        for layer in range(n_layers):
            cache.set_layer_params(layer, RK[layer], RV[layer], cK[layer], cV[layer])
        oc = OracleCache(n_layers, n_requests, w.n_kv_heads, w.head_dim, w.group, w.n_sink, w.window, max_len + 64,
                         RK, RV, cK, cV)
    return cache, oc, params


def check_stream(cache: KVCache, layer: int, slot: int, kvh: int, kv: int, st, label: str = "", positions=None):
    """One (request, kv-head, K|V) stream of the cache against an oracle.Stream: INT2 rows,
    scale/zero words, sinks and ring slots, bit-exact."""
    L, H, S, W = st.length, st.history_end, st.S, st.W
    gL, gH, _ = cache.info(slot)
    assert (gL, gH) == (L, H), f"{label}: lengths {(gL, gH)} != {(L, H)}"
    pos = list(range(S, H)) if positions is None else [p for p in positions if S <= p < H]
    if pos:
        rows, sz = cache.int2_rows(layer, slot, kvh, kv, pos)
        exp_rows = st.rows[pos]
        exp_sz = st.sz[pos].view(np.int16)
        bad = np.nonzero((rows.numpy() != exp_rows).any(axis=1))[0]
        assert bad.size == 0, f"{label} layer {layer} kvh {kvh} kv {kv}: {bad.size} code rows differ, first pos {pos[bad[0]]}"
        badz = np.nonzero((sz.numpy() != exp_sz).any(axis=1))[0]
        assert badz.size == 0, f"{label} layer {layer} kvh {kvh} kv {kv}: {badz.size} scale/zero differ, first pos {pos[badz[0]]}"
    n_s = min(L, S)
    if n_s:
        got = cache.sink_tokens(layer, slot, kvh, kv)[:n_s].numpy().view(np.uint16)
        assert np.array_equal(got, st.sink[:n_s]), f"{label}: sink tokens differ"
    if L > H:
        ring = cache.ring_tokens(layer, slot, kvh, kv).numpy().view(np.uint16)
        idx = [p % W for p in range(H, L)]
        assert np.array_equal(ring[idx], st.ring[idx]), f"{label}: ring tokens differ"


def check_pages(cache: KVCache, oc: OracleCache, layer: int, slot: int, req: int, kvhs=None, positions=None):
    """INT2 rows, scale/zero words, sinks and ring slots: bit-exact."""
    assert cache.info(slot)[:2] == (oc.length(req), oc.history_end(req))
    kvhs = range(oc.Hkv) if kvhs is None else kvhs
    for kvh in kvhs:
        for kv in range(2):
            check_stream(cache, layer, slot, kvh, kv, oc.streams[layer][req][kvh][kv], positions=positions)


def compare_decode(out_f32: torch.Tensor, out_bf16: torch.Tensor, ref: np.ndarray, label: str = ""):
    got = out_f32.detach().cpu().double().numpy()
    assert np.isfinite(got).all(), f"{label}: non-finite output"
    err = np.abs(got - ref).max() if ref.size else 0.0
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err <= MAX_ABS, f"{label}: max-abs error {err:.3e} > {MAX_ABS}"
    if np.linalg.norm(ref) > 0:
        assert rel <= REL_L2, f"{label}: rel-L2 error {rel:.3e} > {REL_L2}"
    # the bf16 output is the round-to-nearest-even of the fp32 output
    assert torch.equal(out_bf16.detach().cpu(), out_f32.detach().cpu().to(torch.bfloat16)), f"{label}: bf16 != rne(fp32)"
    return err, rel


def bits(t: torch.Tensor) -> np.ndarray:
    return as_bits(t)
