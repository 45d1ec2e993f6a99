"""Parity at the benchmark workloads' full sizes, in the launch configuration bench.py
times: the workload's whole batch at its context lengths, filled by the bench's own code
(prefix owners first, sharers mapping the owners' pages), then the bench's first step
(its per-request appends, chunk appenders included) as one fused append + decode call
under the automatic plan, so the CTA shape, the schedule and the merge are the bench's.
One layer is built: every layer of a step runs the same plan.

The cache is checked on samples the oracle can compute one by one: it rebuilds only the
sampled (request, kv-head) streams from the same seeded tokens (a sharer's stream takes
its prefix from the owner's, as the cache does).  Their stored K and V streams (INT2 rows,
scale/zero words, sinks, ring) must match bit for bit, and their outputs the oracle's
fp64 attention within the parity tests' tolerance (max-abs 2e-2, relative L2 5e-3 on the
fp32 output, bf16 output = RNE of it).
"""
import os
import sys

import numpy as np
import pytest
import torch

import oracle
from int2_rotated_kv_rotate_gb300 import KVCache, workloads as wl
from oracle import calibration as ocal
from oracle.model import as_bits

from helpers import check_stream, compare_decode

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402  (the plan and the context fill are the bench's own)

pytestmark = pytest.mark.gpu

SEED = 4242


def _samples(w, plan, shared, n_new):
    """(request, kv-head) pairs: the first and last request, a prefix sharer and a
    chunk appender where the workload has them."""
    B = plan.B
    picks = [0, B - 1]
    picks += [r for r in range(B) if shared[r] > 0][:1]
    picks += [r for r in range(B) if n_new[r] > 1][:1]
    return [(r, (3 * i + r) % w.n_kv_heads) for i, r in enumerate(dict.fromkeys(picks))]


def _stream_pair(w, RK, RV, cK, cV, h, capacity):
    return (oracle.Stream(w.head_dim, w.group, w.n_sink, w.window, capacity, RK[h], cK[h]),
            oracle.Stream(w.head_dim, w.group, w.n_sink, w.window, capacity, RV[h], cV[h]))


def _append_pieces(sk, sv, kb, vb, a, b):
    """Tokens [a, b) (kb, vb hold them from a on) in the fill's pieces."""
    for s in range(a, b, bench.FILL_CHUNK):
        e = min(s + bench.FILL_CHUNK, b)
        sk.append(np.ascontiguousarray(kb[s - a:e - a]))
        sv.append(np.ascontiguousarray(vb[s - a:e - a]))


def _head_bits(w, r, start, n, h, dev):
    # the same device draws the fill used, then the sampled head copied to the host
    k, v = wl.gen_kv(w, SEED, 0, r, start, n, device=dev)
    return as_bits(k[:, h]), as_bits(v[:, h])


@pytest.mark.parametrize("name", ["qwen3_8b_layer", "long_batch", "qwen3_32b_capacity", "ragged_prefix"])
def test_full_size_sampled_heads(name):
    w = wl.WORKLOADS[name]
    dev = torch.device("cuda")
    plan = bench.Plan(w, SEED, 1, 1)
    B, G, Hkv = plan.B, w.gqa, w.n_kv_heads
    cur, n_new = plan.steps[0]
    qc, kc, vc = wl.gen_calibration(w, SEED, 0)
    RK, RV, cK, cV = ocal.calibrate_layer(qc.float().numpy(), kc.float().numpy(), vc.float().numpy(),
                                          w.clip_percentile)
    ppr = (plan.max_len() + 63) // 64 + 2
    pages = sum((L + 63) // 64 + 1 for L in plan.final) + 8
    cache = KVCache(n_q_heads=w.n_q_heads, n_kv_heads=Hkv, group=w.group, n_sink=w.n_sink, window=w.window,
                    n_layers=1, max_requests=B, max_pages=pages, max_pages_per_request=ppr, device=dev)
    try:
        cache.set_layer_params(0, RK, RV, cK, cV)
        slots = [cache.alloc() for _ in range(B)]
        shared = bench.fill_context(cache, w, SEED, 1, slots, plan.lengths, dev)
        torch.cuda.synchronize()
        # the checked step: the bench's call
        cache.reserve(slots, n_new)
        cache.plan(slots)
        ks, vs = zip(*[wl.gen_kv(w, SEED, 0, r, cur[r], n_new[r], device=dev) for r in range(B)])
        q = wl.gen_q(w, SEED, 0, 0, B, device=dev)
        out32 = torch.empty(q.shape, dtype=torch.float32, device=dev)
        out = cache.append_decode(0, torch.cat(ks).contiguous(), torch.cat(vs).contiguous(), q, out_f32=out32)
        torch.cuda.synchronize()
        cache.commit()
        st, flags = cache.status()
        assert st == 0 and flags == 0, f"device flags {flags:#x}"
        qb = as_bits(q)
        for r, h in _samples(w, plan, shared, n_new):
            L, n = cur[r], n_new[r]
            sk, sv = _stream_pair(w, RK, RV, cK, cV, h, L + n + 64)
            start = 0
            if shared[r]:
                # the owner's stream far enough that the shared tokens are history, then shared
                src = r - r % w.prefix_group
                n_src = min(plan.lengths[src], shared[r] + w.window)
                ok, ov = _stream_pair(w, RK, RV, cK, cV, h, n_src + 64)
                kb, vb = _head_bits(w, src, 0, n_src, h, dev)
                _append_pieces(ok, ov, kb, vb, 0, n_src)
                sk.share_from(ok, shared[r])
                sv.share_from(ov, shared[r])
                start = shared[r]
            kb, vb = _head_bits(w, r, start, L + n - start, h, dev)
            _append_pieces(sk, sv, kb[:L - start], vb[:L - start], start, L)
            sk.append(np.ascontiguousarray(kb[L - start:]))  # the step's tokens, as one append
            sv.append(np.ascontiguousarray(vb[L - start:]))
            label = f"{name} req {r} (L {L} + {n}, shared {shared[r]}) kv-head {h}"
            # the stored stream after the step, bit for bit, then the step's output
            check_stream(cache, 0, slots[r], h, 0, sk, label)
            check_stream(cache, 0, slots[r], h, 1, sv, label)
            ref = oracle.decode(np.ascontiguousarray(qb[r, h * G:(h + 1) * G]), sk, sv, RK[h], RV[h])
            compare_decode(out32[r, h * G:(h + 1) * G], out[r, h * G:(h + 1) * G], ref, label)
    finally:
        cache.close()
