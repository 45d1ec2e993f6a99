"""Failure paths on the GPU, made on the host (nothing here faults, traps or hangs a GPU).

- A bounded wait that runs out: the fused append + decode launch is planned to expect
  one more append signal than its append tasks send (host-side fault injection: a signal
  that never arrives), with a short wait limit.  The kernel returns, the status word
  carries OSCAR_FLAG_TIMEOUT, the outputs are finite, and after oscar_get_status the
  cache serves the next step exactly like the oracle.
- NaN and infinite K/V inputs: the format's reading (bf16 NaN is 0x7FFF; on the INT2 path
  fminf/fmaxf map NaN to the clip and infinities to +-clip) gives codes and scale/zero
  words bit-identical to the oracle's, through quantize_append and the fused step, and
  the decode over such history stays finite and within tolerance.
"""
import numpy as np
import pytest
import torch

from int2_rotated_kv_rotate_gb300 import workloads as wl
from int2_rotated_kv_rotate_gb300 import _native as N

from helpers import bits, check_pages, compare_decode, make_pair

pytestmark = pytest.mark.gpu

SEED = 777


def _rows(w, layer, reqs, starts, counts):
    ks, vs = [], []
    for r, s0, n in zip(reqs, starts, counts):
        k, v = wl.gen_kv(w, SEED, layer, r, s0, n, device="cuda")
        ks.append(k)
        vs.append(v)
    return torch.cat(ks).contiguous(), torch.cat(vs).contiguous()


def _oracle_append(oc, layer, reqs, counts, K, V):
    kb, vb = bits(K), bits(V)
    off = 0
    for r, n in zip(reqs, counts):
        oc.append(layer, r, kb[off:off + n], vb[off:off + n])
        off += n


def test_bounded_wait_runs_out_and_the_cache_recovers():
    w = wl.scaled(wl.WORKLOADS["tiny"], name="timeout", lognormal_sigma=0.5)
    reqs, lens = [0, 1], [1500, 700]
    cache, oc, _ = make_pair(w, SEED, 1, 2, 2000)
    slots = [cache.alloc() for _ in reqs]
    cache.reserve(slots, lens)
    K, V = _rows(w, 0, reqs, [0, 0], lens)
    cache.quantize_append(0, K, V)
    _oracle_append(oc, 0, reqs, lens, K, V)
    cache.commit()
    pos = list(lens)
    # the step whose waits run out: ~4096 polls of about 0.1-0.3 us instead of ~a second
    N.oscar_set_wait_limit(cache.handle, 4096)
    counts = [16, 1]
    cache.reserve(slots, counts)
    N.oscar_inject_fault(cache.handle, N.OSCAR_FAULT_LOST_APPEND_SIGNAL)
    cache.plan(slots)
    K, V = _rows(w, 0, reqs, pos, counts)
    q = wl.gen_q(w, SEED, 0, 0, 2, device="cuda")
    out32 = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    cache.append_decode(0, K, V, q, out_f32=out32)
    assert N.oscar_last_launch_count() == 1  # the fused launch, where the waits are
    torch.cuda.synchronize()
    st, flags = cache.status()
    assert flags & N.OSCAR_FLAG_TIMEOUT and st == 6, f"status {st} flags {flags:#x}"
    assert torch.isfinite(out32).all()
    cache.commit()
    _oracle_append(oc, 0, reqs, counts, K, V)
    pos = [p + n for p, n in zip(pos, counts)]
    for i, s in enumerate(slots):
        check_pages(cache, oc, 0, s, i)  # the append tasks themselves ran to the end
    # the next steps, with the default limit, behave like the oracle (counters were reset)
    N.oscar_set_wait_limit(cache.handle, 0)
    for step, counts in enumerate(([16, 1], [1, 16])):
        cache.reserve(slots, counts)
        cache.plan(slots)
        K, V = _rows(w, 0, reqs, pos, counts)
        q = wl.gen_q(w, SEED, 0, step + 1, 2, device="cuda")
        o32 = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        out = cache.append_decode(0, K, V, q, out_f32=o32)
        torch.cuda.synchronize()
        cache.commit()
        _oracle_append(oc, 0, reqs, counts, K, V)
        pos = [p + n for p, n in zip(pos, counts)]
        st, flags = cache.status()
        assert st == 0 and flags == 0, f"step {step}: flags {flags:#x}"
        qb = bits(q)
        for i, s in enumerate(slots):
            check_pages(cache, oc, 0, s, i)
            compare_decode(o32[i], out[i], oc.decode(0, i, qb[i]), f"after timeout step {step} req {i}")
    cache.close()


def _poison(x: torch.Tensor, rng: np.random.Generator, rows, per_row: int = 3):
    """NaN, +inf and -inf in a few channels of the given token rows (all kv-heads)."""
    x = x.clone()
    specials = [float("nan"), float("inf"), float("-inf")]
    for t in rows:
        for h in range(x.shape[1]):
            ch = rng.choice(x.shape[2], size=per_row, replace=False)
            for j, c in enumerate(ch):
                x[t, h, int(c)] = specials[(t + h + j) % 3]
    return x


@pytest.mark.parametrize("group,window", [(128, 128), (32, 64)])
def test_nan_and_inf_inputs_quantize_like_the_oracle(group, window):
    w = wl.scaled(wl.WORKLOADS["tiny"], name=f"nan_{group}", group=group, window=window, lognormal_sigma=0.5)
    cache, oc, _ = make_pair(w, SEED, 1, 1, 1400)
    slot = cache.alloc()
    rng = np.random.default_rng(5)
    pos = 0
    # 300 plain tokens, then a chunk with NaN / inf tokens: the chunk's early tokens go
    # straight to INT2, its last ones land in the ring and are evicted by the next appends
    for n, bad in ((300, False), (400, True), (1, False), (200, False), (17, False)):
        K, V = wl.gen_kv(w, SEED, 0, 0, pos, n, device="cuda")
        if bad:
            rows = list(range(0, n, 7)) + list(range(n - 40, n, 3))
            K, V = _poison(K, rng, rows), _poison(V, rng, rows[::2])
        cache.reserve([slot], [n])
        cache.quantize_append(0, K.contiguous(), V.contiguous())
        cache.commit()
        _oracle_append(oc, 0, [0], [n], K, V)
        pos += n
        torch.cuda.synchronize()
        check_pages(cache, oc, 0, slot, 0)
    assert oc.history_end(0) >= 700  # every poisoned token is INT2 history by now
    cache.plan([slot])
    q = wl.gen_q(w, SEED, 0, 0, 1, device="cuda")
    o32 = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    out = cache.decode(0, q, out_f32=o32)
    torch.cuda.synchronize()
    st, flags = cache.status()
    assert st == 0 and flags == 0
    compare_decode(o32[0], out[0], oc.decode(0, 0, bits(q)[0]), "decode over NaN/inf history")
    cache.close()


def test_nan_and_inf_inputs_in_the_fused_step():
    """No recent window: every new token beyond the sinks goes straight to INT2 inside the
    one-launch append + decode, poisoned tokens included."""
    w = wl.scaled(wl.WORKLOADS["tiny"], name="nan_fused", window=0, lognormal_sigma=0.5)
    cache, oc, _ = make_pair(w, SEED, 1, 2, 1200)
    slots = [cache.alloc(), cache.alloc()]
    rng = np.random.default_rng(9)
    lens = [900, 300]
    cache.reserve(slots, lens)
    K, V = _rows(w, 0, [0, 1], [0, 0], lens)
    cache.quantize_append(0, K, V)
    cache.commit()
    _oracle_append(oc, 0, [0, 1], lens, K, V)
    pos = list(lens)
    for step, counts in enumerate(([16, 16], [1, 16], [16, 1])):
        cache.reserve(slots, counts)
        cache.plan(slots)
        K, V = _rows(w, 0, [0, 1], pos, counts)
        K, V = _poison(K, rng, range(0, K.shape[0], 2)), _poison(V, rng, range(1, V.shape[0], 3))
        q = wl.gen_q(w, SEED, 0, step, 2, device="cuda")
        o32 = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        out = cache.append_decode(0, K, V, q, out_f32=o32)
        assert N.oscar_last_launch_count() == 1
        torch.cuda.synchronize()
        cache.commit()
        _oracle_append(oc, 0, [0, 1], counts, K, V)
        pos = [p + n for p, n in zip(pos, counts)]
        st, flags = cache.status()
        assert st == 0 and flags == 0
        qb = bits(q)
        for i, s in enumerate(slots):
            check_pages(cache, oc, 0, s, i)
            compare_decode(o32[i], out[i], oc.decode(0, i, qb[i]), f"fused NaN step {step} req {i}")
    cache.close()
