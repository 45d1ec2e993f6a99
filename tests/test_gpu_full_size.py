"""Parity at the benchmark workloads' full sizes, in the launch configuration bench.py
times: the workload's whole batch at its context lengths, filled by the bench's own code
(prefix owners first, sharers mapping the owners' pages), then the bench's first step
(its per-request appends, chunk appenders included) as one fused append + decode call
per layer under the automatic plan, so the CTA shape, the schedule and the merge are the
bench's.

Coverage:
- the 8B-shaped layer, the long batch and the ragged shared-prefix mix (one layer each):
  every (request, kv-head) stream of the layer is rebuilt by the oracle from the same
  seeded tokens (a sharer's stream takes its prefix from the owner's, as the cache does);
  all of its stored rows (INT2 codes, scale/zero words, sinks, ring) must match bit for
  bit, and every request's output the oracle's fp64 attention within the parity tests'
  tolerance (max-abs 2e-2, relative L2 5e-3 on the fp32 output, bf16 = RNE of it);
- the 32B-shaped capacity run (64 layers resident): layer 0 and one seeded random layer
  the same way, and in every other layer a seeded 1 % sample of the INT2 pages (whole
  4096-token blocks of the seeded generator, every kv-head and K|V), bit for bit against
  the oracle's rotation and quantizer applied to those tokens.
The oracle's work runs on all host cores (one stream per thread; its C calls release the
interpreter lock).
"""
import os
import random
import sys
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from int2_rotated_kv_rotate_gb300 import KVCache, workloads as wl
from int2_rotated_kv_rotate_gb300 import _native as N
from oracle import calibration as ocal
from oracle.model import as_bits

from helpers import MAX_ABS, REL_L2, check_stream

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402  (the plan and the context fill are the bench's own)

pytestmark = pytest.mark.gpu

SEED = 4242


def _stream_pair(w, RK, RV, cK, cV, h, capacity):
    return (oracle.Stream(w.head_dim, w.group, w.n_sink, w.window, capacity, RK[h], cK[h]),
            oracle.Stream(w.head_dim, w.group, w.n_sink, w.window, capacity, RV[h], cV[h]))


def _append_pieces(sk, sv, kb, vb, a, b):
    """Tokens [a, b) (kb, vb hold them from a on) in the fill's pieces."""
    for s in range(a, b, bench.FILL_CHUNK):
        e = min(s + bench.FILL_CHUNK, b)
        sk.append(np.ascontiguousarray(kb[s - a:e - a]))
        sv.append(np.ascontiguousarray(vb[s - a:e - a]))


def _calibration(w, layer):
    qc, kc, vc = wl.gen_calibration(w, SEED, layer)
    return ocal.calibrate_layer(qc.float().numpy(), kc.float().numpy(), vc.float().numpy(), w.clip_percentile)


def _check_layer(w, cache, slots, plan, shared, layer, params, q_bits, out32, out, cur, n_new):
    """Every (request, kv-head) of one layer: stored rows bit for bit, outputs in tolerance.
    Requests one at a time (their tokens drawn on the device as the fill drew them, copied to
    the host), the kv-heads of a request on parallel threads; a prefix owner's streams are
    kept until its group's sharers have taken their prefix from them."""
    RK, RV, cK, cV = params
    B, G, Hkv = plan.B, w.gqa, w.n_kv_heads
    dev = torch.device("cuda")
    o32 = out32.detach().cpu().double().numpy()
    threads = max(1, (os.cpu_count() or 8) // Hkv)
    owner_streams = {}

    def one(r, h, kb, vb):
        oracle.set_threads(threads)  # this worker's own OpenMP thread count
        L, n, start = cur[r], n_new[r], shared[r]
        sk, sv = _stream_pair(w, RK, RV, cK, cV, h, L + n + 64)
        if start:
            ok_, ov = owner_streams[(r - r % w.prefix_group, h)]
            sk.share_from(ok_, start)
            sv.share_from(ov, start)
        _append_pieces(sk, sv, kb[:L - start, h], vb[:L - start, h], start, L)
        sk.append(np.ascontiguousarray(kb[L - start:, h]))  # the step's tokens, as one append
        sv.append(np.ascontiguousarray(vb[L - start:, h]))
        ref = oracle.decode(np.ascontiguousarray(q_bits[r, h * G:(h + 1) * G]), sk, sv, RK[h], RV[h])
        return sk, sv, ref

    worst = [0.0, 0.0]
    with ThreadPoolExecutor(max_workers=Hkv) as ex:
        for r in range(B):
            start = shared[r]
            k, v = wl.gen_kv(w, SEED, layer, r, start, cur[r] + n_new[r] - start, device=dev)
            kb, vb = as_bits(k), as_bits(v)
            del k, v
            results = list(ex.map(lambda h: one(r, h, kb, vb), range(Hkv)))
            for h, (sk, sv, ref) in enumerate(results):
                label = f"{w.name} layer {layer} req {r} (L {cur[r]} + {n_new[r]}, shared {start}) kv-head {h}"
                check_stream(cache, layer, slots[r], h, 0, sk, label)
                check_stream(cache, layer, slots[r], h, 1, sv, label)
                got = o32[r, h * G:(h + 1) * G]
                err = np.abs(got - ref).max()
                rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
                assert np.isfinite(got).all() and err <= MAX_ABS and rel <= REL_L2, \
                    f"{label}: max-abs {err:.3e} rel {rel:.3e}"
                worst = [max(worst[0], err), max(worst[1], rel)]
                if w.prefix_tokens and r % w.prefix_group == 0:
                    owner_streams[(r, h)] = (sk, sv)
            if w.prefix_tokens and r % w.prefix_group == w.prefix_group - 1:
                for h in range(Hkv):
                    owner_streams.pop((r - r % w.prefix_group, h), None)
    assert torch.equal(out.detach().cpu(), out32.detach().cpu().to(torch.bfloat16))
    return worst


def _check_page_sample(w, cache, slots, plan, layer, params, H_now, rng, frac=0.01):
    """A seeded sample of whole 4096-token blocks of INT2 history in one layer: every
    kv-head's K and V rows of the block's INT2 positions against the oracle's rotation and
    quantizer applied to those tokens."""
    RK, RV, cK, cV = params
    B, Hkv = plan.B, w.n_kv_heads
    blocks = [(r, b) for r in range(B) for b in range(-(-H_now[r] // wl.BLOCK_TOKENS))]
    pick = rng.sample(blocks, max(1, round(frac * len(blocks))))
    dev = torch.device("cuda")
    checked = 0
    for r, b in pick:
        a = max(b * wl.BLOCK_TOKENS, w.n_sink)
        e = min((b + 1) * wl.BLOCK_TOKENS, H_now[r])
        if e <= a:
            continue
        k, v = wl.gen_kv(w, SEED, layer, r, a, e - a, device=dev)
        kb, vb = as_bits(k), as_bits(v)
        pos = list(range(a, e))
        for h in range(Hkv):
            for kv, xb, R, c in ((0, kb, RK, cK), (1, vb, RV, cV)):
                # a stream with no sinks and no window quantises every token it is given:
                # the oracle's rotation and quantizer of exactly these tokens
                st = oracle.Stream(w.head_dim, w.group, 0, 0, len(pos), R[h], c[h])
                st.append(np.ascontiguousarray(xb[:, h]))
                rows, sz = cache.int2_rows(layer, slots[r], h, kv, pos)
                assert np.array_equal(rows.numpy(), st.rows[:len(pos)]), f"layer {layer} req {r} block {b}"
                assert np.array_equal(sz.numpy(), st.sz[:len(pos)].view(np.int16)), \
                    f"layer {layer} req {r} block {b} scale/zero"
                checked += len(pos)
    return checked


@pytest.mark.parametrize("fmt", [pytest.param(N.OSCAR_FORMAT_INT2, id="tm"), pytest.param(N.OSCAR_FORMAT_INT2_CM, id="cm")])
@pytest.mark.parametrize("name", ["qwen3_8b_layer", "long_batch", "ragged_prefix", "qwen3_32b_capacity"])
def test_full_size_every_head(name, fmt):
    """Both INT2 formats: the token-major one (the bench's headline) and the channel-major
    one with the tcgen05 decode (the bench's int2_cm_format line)."""
    w = wl.WORKLOADS[name]
    dev = torch.device("cuda")
    n_layers = w.n_layers if name == "qwen3_32b_capacity" else 1
    plan = bench.Plan(w, SEED, n_layers, 1)
    B = plan.B
    cur, n_new = plan.steps[0]
    ppr = (plan.max_len() + 63) // 64 + 2
    pages = sum((L + 63) // 64 + 1 for L in plan.final) + 8
    rng = random.Random(SEED)
    full_layers = [0] if n_layers == 1 else [0, rng.randrange(1, n_layers)]
    cache = KVCache(fmt=fmt, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, group=w.group, n_sink=w.n_sink,
                    window=w.window, n_layers=n_layers, max_requests=B, max_pages=pages, max_pages_per_request=ppr,
                    device=dev)
    try:
        params = {}
        for layer in range(n_layers):
            # the oracle's calibration for the layers checked in full; the others take the
            # product's GPU calibration (their pages are checked against the same inputs)
            if layer in full_layers:
                params[layer] = _calibration(w, layer)
            else:
                from int2_rotated_kv_rotate_gb300 import calibrate

                qc, kc, vc = wl.gen_calibration(w, SEED, layer, device=dev)
                params[layer] = calibrate.calibrate_layer_gpu(qc, kc, vc, w.clip_percentile)
            cache.set_layer_params(layer, *params[layer])
        slots = [cache.alloc() for _ in range(B)]
        shared = bench.fill_context(cache, w, SEED, n_layers, slots, plan.lengths, dev)
        torch.cuda.synchronize()
        # the checked step: the bench's call on every layer
        cache.reserve(slots, n_new)
        cache.plan(slots)
        outs = {}
        for layer in range(n_layers):
            ks, vs = zip(*[wl.gen_kv(w, SEED, layer, r, cur[r], n_new[r], device=dev) for r in range(B)])
            q = wl.gen_q(w, SEED, layer, 0, B, device=dev)
            out32 = torch.empty(q.shape, dtype=torch.float32, device=dev)
            out = cache.append_decode(layer, torch.cat(ks).contiguous(), torch.cat(vs).contiguous(), q,
                                      out_f32=out32)
            if layer in full_layers:
                outs[layer] = (as_bits(q), out32, out)
        torch.cuda.synchronize()
        cache.commit()
        st, flags = cache.status()
        assert st == 0 and flags == 0, f"device flags {flags:#x}"
        for layer in full_layers:
            qb, out32, out = outs[layer]
            _check_layer(w, cache, slots, plan, shared, layer, params[layer], qb, out32, out, cur, n_new)
        if n_layers > 1:
            H_now = [cache.info(s)[1] for s in slots]
            sampled = 0
            for layer in range(n_layers):
                if layer not in full_layers:
                    sampled += _check_page_sample(w, cache, slots, plan, layer, params[layer], H_now, rng)
            assert sampled > 0
    finally:
        cache.close()
