"""The throughput-mode serving loop (continuous batching at a fixed budget) against the
oracle: a pool too small for every request at once, so requests queue, are admitted as
others finish and free their pages, and map their group's shared prefix from a prefix
holder.  Every decode output of every step is checked against the oracle's attention over
a private copy of the request's tokens (the same tokens, rebuilt on the host from the
token pools); the INT2 rows of the running requests are checked bit for bit every few
steps; at the end the pool holds only the prefix holders' pages, and none once they are
freed.  The BF16 cache runs the same loop at the same budget, checked against plain
attention."""
import numpy as np
import pytest
import torch

import oracle
from int2_rotated_kv_rotate_gb300 import serving, workloads as wl
from int2_rotated_kv_rotate_gb300 import _native as N
from oracle import calibration as ocal
from oracle.model import as_bits, bf16_reference

from helpers import check_stream, compare_decode

pytestmark = pytest.mark.gpu

SEED = 2718


def _shape():
    return wl.scaled(wl.WORKLOADS["qwen3_8b_layer"], name="serving_test", n_layers=2, n_q_heads=8, n_kv_heads=2,
                     window=64, calib_tokens=512)


def _params(w):
    out = [[], [], [], []]
    for layer in range(w.n_layers):
        q, k, v = wl.gen_calibration(w, SEED, layer)
        for i, a in enumerate(ocal.calibrate_layer(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                                   w.clip_percentile)):
            out[i].append(a)
    return [np.stack(a) for a in out]


class Mirror:
    """The oracle's private copy of every request's tokens, built lazily from the pools."""

    def __init__(self, w, tokens, prefix, params):
        self.w, self.prefix = w, prefix
        self.K, self.V, self.Q = as_bits(tokens.K), as_bits(tokens.V), as_bits(tokens.Q)
        self.tokens = tokens
        self.params = params
        self.streams = {}  # (rid, layer, kvh) -> (K stream, V stream)
        self.plain = {}  # (rid, layer) -> list of (k bits, v bits) rows (BF16 reference)

    def rows(self, r, layer, a, n):
        idx = torch.cat([self.tokens.rows(layer, s, p, m) for s, p, m in
                         [(serving.TokenSource.stream(r, p, self.prefix), p, 1) for p in range(a, a + n)]]).cpu()
        return self.K[idx.numpy()], self.V[idx.numpy()]

    def int2_streams(self, r, layer, upto):
        w = self.w
        RK, RV, cK, cV = self.params
        out = []
        for h in range(w.n_kv_heads):
            key = (r.rid, layer, h)
            if key not in self.streams:
                self.streams[key] = (
                    oracle.Stream(128, w.group, w.n_sink, w.window, 1 << 14, RK[layer, h], cK[layer, h]),
                    oracle.Stream(128, w.group, w.n_sink, w.window, 1 << 14, RV[layer, h], cV[layer, h]))
            sk, sv = self.streams[key]
            if sk.length < upto:
                kb, vb = self.rows(r, layer, sk.length, upto - sk.length)
                sk.append(np.ascontiguousarray(kb[:, h]))
                sv.append(np.ascontiguousarray(vb[:, h]))
            out.append((sk, sv))
        return out


@pytest.mark.parametrize("fmt", [N.OSCAR_FORMAT_INT2, N.OSCAR_FORMAT_INT2_CM, N.OSCAR_FORMAT_BF16])
def test_serving_loop_against_the_oracle(fmt):
    w = _shape()
    prefix = 384
    tokens = serving.TokenSource(w, SEED, pool_tokens=4096)
    int2 = fmt in (N.OSCAR_FORMAT_INT2, N.OSCAR_FORMAT_INT2_CM)
    params = _params(w) if int2 else None
    reqs = serving.make_requests(9, (450, 1400), (3, 14), n_groups=2, seed=SEED)
    # about three or four requests at once at this budget
    per_token = w.n_layers * w.n_kv_heads * 2 * (36 if int2 else 256)
    budget = N.oscar_cache_device_bytes(N.oscar_config(fmt, 128, w.n_q_heads, w.n_kv_heads, w.group, 64, w.n_sink,
                                                       w.window, w.n_layers, 16, 1, 40)) + 3500 * per_token
    loop = serving.ServingLoop(w, fmt, budget, tokens, layer_params=params, max_requests=16, max_len=2560,
                               prefix_tokens=prefix, prefill_chunk=1000)
    free0 = loop.cache.stats()[0]
    mirror = Mirror(w, tokens, prefix, params)
    G = w.gqa
    checked = [0]

    def on_output(step, layer, reqs_, K, V, q, out, o32):
        torch.cuda.synchronize()
        qb = as_bits(q)
        for i, r in enumerate(reqs_):
            L = r.length + 1  # the step appends the request's next token first
            if int2:
                ref = np.zeros((w.n_q_heads, 128))
                for h, (sk, sv) in enumerate(mirror.int2_streams(r, layer, L)):
                    ref[h * G:(h + 1) * G] = oracle.decode(np.ascontiguousarray(qb[i, h * G:(h + 1) * G]), sk, sv,
                                                           params[0][layer, h], params[1][layer, h])
            else:
                kb, vb = mirror.rows(r, layer, 0, L)
                ref = bf16_reference(qb[i], kb, vb)
            compare_decode(o32[i], out[i], ref, f"fmt {fmt} step {step} layer {layer} request {r.rid} (L {L})")
            checked[0] += 1

    def on_step(step, done):
        if not int2 or step % 4:
            return
        for r in loop.running:
            for layer in range(w.n_layers):
                for h, (sk, sv) in enumerate(mirror.int2_streams(r, layer, r.length)):
                    check_stream(loop.cache, layer, r.slot, h, 0, sk, f"request {r.rid} step {step}")
                    check_stream(loop.cache, layer, r.slot, h, 1, sv, f"request {r.rid} step {step}")

    st = loop.run(reqs, on_output=on_output, on_step=on_step)
    assert st["completed"] == len(reqs) and st["generated"] == sum(r.gen for r in reqs)
    assert checked[0] == st["generated"] * w.n_layers
    assert 1 < st["max_batch"] < len(reqs), st  # requests queued, and several ran at once
    assert st["prefix_hits"] > 0 and st["shared_tokens"] > 0
    status, flags = loop.cache.status()
    assert status == 0 and flags == 0
    holder_pages = sum(loop.cache.info(s)[2] for s in loop.holders.values())
    assert loop.cache.stats()[0] == free0 - holder_pages
    for s in list(loop.holders.values()):
        loop.cache.free(s)
    loop.holders = {}
    assert loop.cache.stats() == (free0, 16)
    loop.close()
