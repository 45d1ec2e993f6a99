"""Seeded synthetic workloads for the 2-bit rotated KV-cache hot path.

This module only draws numbers: shapes, lengths and random bf16 tensors.  It holds none
of the method's arithmetic (no rotation, quantisation or attention), so both the CUDA
path and the CPU oracle may take their inputs from it.

Distribution (the pages give no dataset for the kernels; their accuracy suites need
trained weights): K, V and q are bf16 draws from N(0, 1).  Four seeded K channels are
scaled x20 and two seeded V channels x8 (channel outliers, the failure case described in
the OSCAR technical summary, section 1).  From the 8B-shaped layer on, every token
vector is also scaled by its own log-normal(0, 0.5) factor (token-norm variation, the
effect the OScaR abstract names).

Generation is block-wise: tokens of one (layer, stream) are drawn in blocks of
BLOCK_TOKENS, each block from its own seeded generator, so any position range can be
regenerated on its own.  A stream is a request, or the shared prefix of a group of
requests (positions below the prefix length).  CPU and CUDA generators give different
numbers for the same seed: a test draws on one device and copies to the host for the
oracle.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Optional

import torch

BLOCK_TOKENS = 4096


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    description: str
    batch: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    context: int  # context length per request (max for ragged mixes)
    group: int  # quantisation group size along head_dim
    page: int
    n_sink: int
    window: int
    lognormal_sigma: float  # 0 = no per-token norm variation
    k_outlier_channels: int = 4
    k_outlier_scale: float = 20.0
    v_outlier_channels: int = 2
    v_outlier_scale: float = 8.0
    calib_tokens: int = 2048
    clip_percentile: float = 99.9
    append_per_step: int = 0  # tokens appended per request per decode step
    ragged_min: int = 0  # ragged mix: lengths uniform in [ragged_min, context]
    prefix_group: int = 0  # ragged mix: requests per shared-prefix group
    prefix_tokens: int = 0  # ragged mix: shared prefix length
    chunk_appenders: int = 0  # ragged mix: requests that append a chunk each step
    chunk_tokens: int = 0

    @property
    def gqa(self) -> int:
        return self.n_q_heads // self.n_kv_heads


WORKLOADS = {
    "tiny": Workload(
        name="tiny",
        description="B1, 1 layer, 8q/2kv, d128, L4096 = 4 sink + 128 recent + 3964 INT2, g128, page 64",
        batch=1, n_layers=1, n_q_heads=8, n_kv_heads=2, head_dim=128, context=4096, group=128, page=64,
        n_sink=4, window=128, lognormal_sigma=0.0),
    "qwen3_8b_layer": Workload(
        name="qwen3_8b_layer",
        description="Qwen3-8B-shaped layer: B1, 32q/8kv, d128, L32768 (4 sink + 128 recent BF16), g128, page 64, "
                    "36 layers, 16 tokens appended + 1 decoded per layer-step",
        batch=1, n_layers=36, n_q_heads=32, n_kv_heads=8, head_dim=128, context=32768, group=128, page=64,
        n_sink=4, window=128, lognormal_sigma=0.5, append_per_step=16),
    "long_batch": Workload(
        name="long_batch",
        description="B8 x 100000, 32q/8kv, d128, g32, page 64, 4 sink + 256 recent BF16",
        batch=8, n_layers=1, n_q_heads=32, n_kv_heads=8, head_dim=128, context=100000, group=32, page=64,
        n_sink=4, window=256, lognormal_sigma=0.5),
    "qwen3_32b_capacity": Workload(
        name="qwen3_32b_capacity",
        description="Qwen3-32B-shaped capacity run: B28 x 100000, 64q/8kv (GQA 8), d128, g128, 64 layers resident, "
                    "4 sink + 128 recent BF16",
        batch=28, n_layers=64, n_q_heads=64, n_kv_heads=8, head_dim=128, context=100000, group=128, page=64,
        n_sink=4, window=128, lognormal_sigma=0.5),
    "ragged_prefix": Workload(
        name="ragged_prefix",
        description="64 requests, L uniform in [1024, 131072], groups of 8 sharing a 16384-token prefix, 32q/8kv, "
                    "g128; per step all decode 1 token and 8 append a 512-token chunk",
        batch=64, n_layers=1, n_q_heads=32, n_kv_heads=8, head_dim=128, context=131072, group=128, page=64,
        n_sink=4, window=128, lognormal_sigma=0.5, append_per_step=1, ragged_min=1024, prefix_group=8,
        prefix_tokens=16384, chunk_appenders=8, chunk_tokens=512),
}


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields replaced (smaller parity cases)."""
    return dataclasses.replace(w, **changes)


def _seed(*parts) -> int:
    h = hashlib.sha256(repr(parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _generator(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*parts))
    return g


def outlier_channels(w: Workload, seed: int):
    """Seeded outlier channel indices (K, V); the same for every layer and head."""
    g = _generator("cpu", "outliers", w.name, seed)
    perm = torch.randperm(w.head_dim, generator=g)
    k_idx = sorted(perm[: w.k_outlier_channels].tolist())
    perm = torch.randperm(w.head_dim, generator=g)
    v_idx = sorted(perm[: w.v_outlier_channels].tolist())
    return k_idx, v_idx


def _channel_scale(w: Workload, idx, scale, device) -> torch.Tensor:
    s = torch.ones(w.head_dim, dtype=torch.float32, device=device)
    if len(idx):
        s[torch.tensor(idx, device=device)] = scale
    return s


def _draw_block(w: Workload, seed: int, layer: int, stream: str, block: int, device) -> tuple:
    """One block of BLOCK_TOKENS tokens of K and V, fp32 [BLOCK_TOKENS, H_kv, d]."""
    g = _generator(device, "kv", w.name, seed, layer, stream, block)
    shape = (BLOCK_TOKENS, w.n_kv_heads, w.head_dim)
    k = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    k_idx, v_idx = outlier_channels(w, seed)
    k *= _channel_scale(w, k_idx, w.k_outlier_scale, device)
    v *= _channel_scale(w, v_idx, w.v_outlier_scale, device)
    if w.lognormal_sigma > 0:
        nk = torch.randn(shape[:2], generator=g, device=device, dtype=torch.float32)
        nv = torch.randn(shape[:2], generator=g, device=device, dtype=torch.float32)
        k *= torch.exp(w.lognormal_sigma * nk).unsqueeze(-1)
        v *= torch.exp(w.lognormal_sigma * nv).unsqueeze(-1)
    return k, v


def _stream_of(w: Workload, request: int, position: int) -> str:
    if w.prefix_tokens and position < w.prefix_tokens:
        return f"prefix{request // w.prefix_group}"
    return f"req{request}"


def gen_kv(w: Workload, seed: int, layer: int, request: int, start: int, n: int, device="cpu"):
    """K and V of positions [start, start+n) of one request: bf16 [n, H_kv, d] each."""
    ks, vs = [], []
    p = start
    end = start + n
    while p < end:
        stream = _stream_of(w, request, p)
        # the stream changes at the prefix boundary; never draw across it
        stop = end
        if w.prefix_tokens and p < w.prefix_tokens:
            stop = min(stop, w.prefix_tokens)
        block = p // BLOCK_TOKENS
        bstart = block * BLOCK_TOKENS
        take = min(stop, bstart + BLOCK_TOKENS) - p
        k, v = _draw_block(w, seed, layer, stream, block, device)
        ks.append(k[p - bstart: p - bstart + take])
        vs.append(v[p - bstart: p - bstart + take])
        p += take
    if not ks:
        shape = (0, w.n_kv_heads, w.head_dim)
        return (torch.empty(shape, dtype=torch.bfloat16, device=device),
                torch.empty(shape, dtype=torch.bfloat16, device=device))
    return torch.cat(ks).to(torch.bfloat16), torch.cat(vs).to(torch.bfloat16)


def gen_q(w: Workload, seed: int, layer: int, step: int, n_req: int, device="cpu") -> torch.Tensor:
    """Decode queries, bf16 [n_req, H_q, d]."""
    g = _generator(device, "q", w.name, seed, layer, step)
    q = torch.randn((n_req, w.n_q_heads, w.head_dim), generator=g, device=device, dtype=torch.float32)
    return q.to(torch.bfloat16)


def gen_calibration(w: Workload, seed: int, layer: int, device="cpu"):
    """Calibration activations for one layer: q [N, H_q, d], k and v [N, H_kv, d] (bf16)."""
    g = _generator(device, "calib", w.name, seed, layer)
    n = w.calib_tokens
    q = torch.randn((n, w.n_q_heads, w.head_dim), generator=g, device=device, dtype=torch.float32)
    shape = (n, w.n_kv_heads, w.head_dim)
    k = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    k_idx, v_idx = outlier_channels(w, seed)
    k *= _channel_scale(w, k_idx, w.k_outlier_scale, device)
    v *= _channel_scale(w, v_idx, w.v_outlier_scale, device)
    if w.lognormal_sigma > 0:
        k *= torch.exp(w.lognormal_sigma * torch.randn(shape[:2], generator=g, device=device)).unsqueeze(-1)
        v *= torch.exp(w.lognormal_sigma * torch.randn(shape[:2], generator=g, device=device)).unsqueeze(-1)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def context_lengths(w: Workload, seed: int):
    """Context length of every request (uniform for fixed workloads, seeded for ragged)."""
    if not w.ragged_min:
        return [w.context] * w.batch
    g = _generator("cpu", "lengths", w.name, seed)
    lo, hi = w.ragged_min, w.context
    u = torch.randint(lo, hi + 1, (w.batch,), generator=g)
    return [int(x) for x in u.tolist()]


def shared_prefix_tokens(w: Workload, length: int) -> int:
    """Tokens of a request that map its group's shared prefix pages.

    Only full pages below the request's recent window are shared (they are never
    rewritten): min(prefix, floor((L - W) / page) * page), and 0 without sharing.
    """
    if not w.prefix_tokens:
        return 0
    usable = (length - w.window) // w.page * w.page
    return max(0, min(w.prefix_tokens, usable))


def chunk_appenders(w: Workload, step: int):
    """Requests that append a chunk at a given step: one per prefix group, rotating."""
    if not w.chunk_appenders:
        return []
    groups = max(1, w.batch // max(1, w.prefix_group))
    per = max(1, w.chunk_appenders // groups)
    out = []
    for gi in range(groups):
        for j in range(per):
            out.append(gi * w.prefix_group + (step * per + j) % w.prefix_group)
    return sorted(out[: w.chunk_appenders])


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)
