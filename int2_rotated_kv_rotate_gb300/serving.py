"""Throughput-mode serving over one cache: continuous batching at a fixed HBM budget.

The OSCAR technical summary (gist.science) reports, for large batches, up to 7x the
throughput of BF16 under the same memory budget (section 4), and runs the INT2 kernel
inside a serving framework with paged KV and prefix caching (section 2.2-B).  This module
is the analogue for this library: one loop that admits requests while the pool's pages
allow, prefills their prompts (mapping a group's shared prefix from a prefix holder
instead of recomputing it: a prefix-cache hit), decodes one token per running request per
step through the library's calls, and frees a request's pages when it finishes.  The same
loop runs the INT2 cache and the uncompressed BF16 cache, each sized to the same byte
budget; the number of requests that fit at once is what differs.

Scheduling: first come, first served.  A request is admitted when a slot is free and the
free pages cover its final length on top of what the running requests will still need
(so a running request never runs out of pages).  A prefix holder is a slot that holds
one group's prefix tokens and stays resident once made.

Tokens: K, V and q rows come from seeded pools on the device, indexed by (layer, stream,
position), where the stream is the group's prefix below the prefix length and the
request's own beyond it, so shared prefixes really are the same tokens and any token can
be rebuilt on the host (the tests' oracle does).  The model that would produce them is
out of scope: these are the cache's inputs.
"""
from __future__ import annotations

import dataclasses
import time
from typing import Callable, Optional

import torch

from . import _native as N

_INT2 = (N.OSCAR_FORMAT_INT2, N.OSCAR_FORMAT_INT2_CM)  # both INT2 page formats
from . import workloads as wl
from .cache import KVCache


@dataclasses.dataclass
class Request:
    rid: int
    prompt: int  # context tokens before generation
    gen: int  # tokens generated (decode steps)
    group: int = -1  # shared-prefix group, -1 = none
    slot: int = -1
    length: int = 0
    generated: int = 0
    shared: int = 0  # prompt tokens mapped from the group's prefix holder


def make_requests(n: int, prompt_range, gen_range, n_groups: int, seed: int):
    """n seeded requests: prompt and generation lengths uniform in the given ranges, every
    request in one of n_groups shared-prefix groups (round robin)."""
    g = torch.Generator().manual_seed(seed)
    p = torch.randint(prompt_range[0], prompt_range[1] + 1, (n,), generator=g).tolist()
    o = torch.randint(gen_range[0], gen_range[1] + 1, (n,), generator=g).tolist()
    return [Request(rid=i, prompt=int(p[i]), gen=int(o[i]), group=(i % n_groups) if n_groups else -1)
            for i in range(n)]


class TokenSource:
    """K, V (bf16 [P, H_kv, d]) and q (bf16 [P, H_q, d]) pools; the row of (layer, stream,
    position) is pool[(A * stream + B * layer + position) mod P]."""

    A, B = 7919, 104729

    def __init__(self, w: wl.Workload, seed: int, pool_tokens: int = 8192, device="cuda"):
        self.P = pool_tokens
        self.K, self.V = wl.gen_kv(wl.scaled(w, prefix_tokens=0), seed, 0, 0, 0, pool_tokens, device=device)
        self.Q = wl.gen_q(w, seed, 0, 0, pool_tokens, device=device)
        self.device = torch.device(device)

    @staticmethod
    def stream(req: Request, position: int, prefix_tokens: int) -> int:
        if req.group >= 0 and position < prefix_tokens:
            return 1_000_000 + req.group
        return req.rid

    def rows(self, layer: int, stream: int, start: int, n: int) -> torch.Tensor:
        base = (self.A * stream + self.B * layer + start) % self.P
        return (torch.arange(n, device=self.device) + base) % self.P

    def index(self, layer: int, pieces) -> torch.Tensor:
        """Pool rows of the pieces [(stream, start, n)] concatenated."""
        parts = [self.rows(layer, s, a, n) for s, a, n in pieces if n > 0]
        if not parts:
            return torch.empty(0, dtype=torch.long, device=self.device)
        return torch.cat(parts)


def pages_needed(fmt: int, L: int, S: int, W: int) -> int:
    """Pages of a request of length L (the library's rule: INT2 pages hold history rows only)."""
    if fmt in _INT2:
        H = max(S, L - W)
        return -(-H // 64) if H > S else 0
    return -(-L // 64)


def cache_for_budget(w: wl.Workload, fmt: int, budget_bytes: int, max_requests: int, max_len: int, device):
    """The cache with the most pages whose device block fits the budget."""
    ppr = -(-max_len // 64) + 2

    def cfg(pages):
        return N.oscar_config(fmt, w.head_dim, w.n_q_heads, w.n_kv_heads, w.group, 64, w.n_sink, w.window, w.n_layers,
                              max_requests, pages, ppr)

    lo, hi = 1, 1 << 24
    if N.oscar_cache_device_bytes(cfg(lo)) > budget_bytes:
        raise ValueError(f"a budget of {budget_bytes} bytes holds no page")
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if N.oscar_cache_device_bytes(cfg(mid)) <= budget_bytes:
            lo = mid
        else:
            hi = mid - 1
    return KVCache(fmt=fmt, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, group=w.group, n_sink=w.n_sink,
                   window=w.window, n_layers=w.n_layers, max_requests=max_requests, max_pages=lo,
                   max_pages_per_request=ppr, device=device)


class ServingLoop:
    """Continuous batching over one cache (INT2 or BF16) of workload shape w."""

    def __init__(self, w: wl.Workload, fmt: int, budget_bytes: int, tokens: TokenSource, layer_params=None,
                 max_requests: int = 128, max_len: int = 1 << 16, prefix_tokens: int = 0,
                 prefill_chunk: int = 16384, device="cuda"):
        self.w, self.fmt, self.tokens = w, fmt, tokens
        self.S = w.n_sink if fmt in _INT2 else 0
        self.W = w.window if fmt in _INT2 else 0
        self.prefix = prefix_tokens
        self.prefill_chunk = prefill_chunk
        self.cache = cache_for_budget(w, fmt, budget_bytes, max_requests, max_len, device)
        if fmt in _INT2:
            RK, RV, cK, cV = layer_params
            for layer in range(w.n_layers):
                self.cache.set_layer_params(layer, RK[layer], RV[layer], cK[layer], cV[layer])
        self.holders = {}  # group -> holder slot
        self.stats = dict(steps=0, generated=0, completed=0, prefill_tokens=0, shared_tokens=0, prefix_hits=0,
                          max_batch=0, batch_sum=0, decode_s=0.0, wall_s=0.0, max_pages_used=0)

    # ------------------------------------------------------------------ pages
    def _need(self, L: int) -> int:
        return pages_needed(self.fmt, L, self.S, self.W)

    def _shareable(self) -> int:
        """Prefix tokens a request maps from its group's holder (full pages the holder will
        never rewrite)."""
        if not self.prefix:
            return 0
        held = self.prefix if self.fmt not in _INT2 else max(self.S, self.prefix - self.W)
        return held // 64 * 64

    # ------------------------------------------------------------------ appends
    def _append(self, reqs, starts, counts):
        """Append tokens [start, start + count) of each request (as one reservation)."""
        c = self.cache
        slots = [r.slot for r in reqs]
        c.reserve(slots, counts)
        for layer in range(self.w.n_layers):
            pieces = []
            for r, a, n in zip(reqs, starts, counts):
                pieces += self._pieces(r, a, n)
            idx = self.tokens.index(layer, pieces)
            K = self.tokens.K.index_select(0, idx)
            V = self.tokens.V.index_select(0, idx)
            c.append(layer, K, V)
        c.commit()

    def _pieces(self, r: Request, a: int, n: int):
        """(stream, start, count) pieces of tokens [a, a + n) of request r."""
        out = []
        p = a
        while p < a + n:
            stop = a + n
            if r.group >= 0 and p < self.prefix:
                stop = min(stop, self.prefix)
            out.append((TokenSource.stream(r, p, self.prefix), p, stop - p))
            p = stop
        return out

    def _holder(self, group: int) -> Optional[int]:
        """The group's prefix holder slot (made on first use if the pool allows)."""
        if group in self.holders:
            return self.holders[group]
        free_pages, free_slots = self.cache.stats()
        if free_slots < 2 or free_pages - self._future_pages() < self._need(self.prefix):
            return None
        h = Request(rid=-1 - group, prompt=self.prefix, gen=0, group=group)
        h.slot = self.cache.alloc()
        self._append([h], [0], [self.prefix])
        self.holders[group] = h.slot
        return h.slot

    def _future_pages(self) -> int:
        """Pages the running requests will still take before they finish."""
        return sum(max(0, self._need(r.prompt + r.gen) - max(self._need(r.length), r.shared // 64))
                   for r in self.running)

    def _admit(self, waiting) -> list:
        admitted = []
        while waiting:
            r = waiting[0]
            free_pages, free_slots = self.cache.stats()
            if free_slots == 0:
                break
            sh = 0
            if r.group >= 0 and self.prefix and r.prompt >= self.prefix + self.W:
                sh = self._shareable()
            if sh and self._holder(r.group) is None:
                sh = 0
            free_pages, free_slots = self.cache.stats()
            own = self._need(r.prompt + r.gen) - sh // 64
            if free_slots == 0 or free_pages - self._future_pages() < own:
                break
            waiting.pop(0)
            r.slot = self.cache.alloc()
            if sh:
                self.cache.share_prefix(r.slot, self.holders[r.group], sh)
                r.shared = sh
                self.stats["shared_tokens"] += sh
                self.stats["prefix_hits"] += 1
            r.length = sh
            admitted.append(r)
            self.running.append(r)
        # prefill the admitted prompts, in chunks
        while admitted:
            batch, starts, counts, total = [], [], [], 0
            for r in admitted:
                n = min(r.prompt - r.length, self.prefill_chunk - total)
                if n <= 0:
                    continue
                batch.append(r)
                starts.append(r.length)
                counts.append(n)
                total += n
                if total >= self.prefill_chunk:
                    break
            if not batch:
                break
            self._append(batch, starts, counts)
            for r, n in zip(batch, counts):
                r.length += n
                self.stats["prefill_tokens"] += n
            admitted = [r for r in admitted if r.length < r.prompt]
        return admitted

    # ------------------------------------------------------------------ decode
    def _decode_step(self, on_output: Optional[Callable]):
        c = self.cache
        reqs = self.running
        slots = [r.slot for r in reqs]
        c.reserve(slots, [1] * len(reqs))
        c.plan(slots)
        # pool rows of every request's new token and query, all layers: row = (A * stream +
        # B * layer + position) mod P, one device tensor per step
        tk = self.tokens
        base = torch.tensor([[TokenSource.A * TokenSource.stream(r, r.length, self.prefix) + r.length,
                              TokenSource.A * (r.rid + 17) + r.length] for r in reqs], dtype=torch.long)
        rows = ((base.to(tk.device)[None] + TokenSource.B * torch.arange(self.w.n_layers, device=tk.device)[:, None, None])
                % tk.P)  # [layer, request, (token, query)]
        for layer in range(self.w.n_layers):
            idx, qi = rows[layer, :, 0], rows[layer, :, 1]
            K = tk.K.index_select(0, idx)
            V = tk.V.index_select(0, idx)
            q = tk.Q.index_select(0, qi)
            o32 = torch.empty(q.shape, dtype=torch.float32, device=q.device) if on_output else None
            if self.fmt in _INT2:
                out = c.append_decode(layer, K, V, q, out_f32=o32)
            else:
                c.bf16_append(layer, K, V)
                out = c.decode(layer, q, out_f32=o32)
            if on_output:
                on_output(self.stats["steps"], layer, list(reqs), K, V, q, out, o32)
        c.commit()
        for r in reqs:
            r.length += 1
            r.generated += 1

    def _warm_gathers(self, n_max: int) -> None:
        """Run the step's gathers once for every batch size (set-up, untimed): the first use
        of a torch gather of a given size can stall for seconds while its device code loads."""
        tk = self.tokens
        idx = torch.zeros((self.w.n_layers, n_max, 2), dtype=torch.long, device=tk.device)
        for n in range(1, n_max + 1):
            for t in (tk.K, tk.V, tk.Q):
                t.index_select(0, idx[0, :n, 0])
        base = torch.zeros((n_max, 2), dtype=torch.long)
        _ = ((base.to(tk.device)[None] + TokenSource.B * torch.arange(self.w.n_layers, device=tk.device)[:, None, None])
             % tk.P)
        torch.cuda.synchronize(tk.device)

    def run(self, requests, on_output: Optional[Callable] = None, on_step: Optional[Callable] = None):
        """Serve every request to completion; returns the statistics."""
        waiting = list(requests)
        self._warm_gathers(min(len(requests), self.cache.cfg.max_requests))
        self.running = []
        st = self.stats
        free0 = self.cache.stats()[0]
        dev = self.tokens.device
        ev = []
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        while waiting or self.running:
            self._admit(waiting)
            if not self.running:
                raise RuntimeError(f"request {waiting[0].rid} does not fit the budget even alone")
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            self._decode_step(on_output)
            e1.record()
            ev.append((e0, e1))
            n = len(self.running)
            st["steps"] += 1
            st["generated"] += n
            st["batch_sum"] += n
            st["max_batch"] = max(st["max_batch"], n)
            st["max_pages_used"] = max(st["max_pages_used"], free0 - self.cache.stats()[0])
            done = [r for r in self.running if r.generated >= r.gen]
            for r in done:
                self.cache.free(r.slot)
                r.slot = -1
                st["completed"] += 1
            self.running = [r for r in self.running if r.generated < r.gen]
            if on_step:
                on_step(st["steps"], done)
        torch.cuda.synchronize(dev)
        st["wall_s"] = time.perf_counter() - t0
        st["decode_s"] = sum(a.elapsed_time(b) for a, b in ev) / 1000.0
        st["mean_batch"] = st["batch_sum"] / max(1, st["steps"])
        st["tokens_per_s"] = st["generated"] / st["wall_s"]
        st["decode_tokens_per_s"] = st["generated"] / max(st["decode_s"], 1e-9)
        st["pool_pages"] = self.cache.cfg.max_pages
        return st

    def close(self):
        for slot in self.holders.values():
            self.cache.free(slot)
        self.holders = {}
        self.cache.close()
