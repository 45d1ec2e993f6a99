"""The decode entry point that allocates nothing (oscar_decode_attention_noalloc).

Some callers cannot allocate device memory at all (a plugin inside a framework that owns
every device allocation, a serving loop that may not allocate once running), so they
cannot hand the decode a workspace.  This entry point uses a fixed scratch array inside
the library instead.  Here it is called through the C ABI twice in a row, with different
queries, and each output is checked against the ordinary entry point's output on the
same plan: both run the same kernel on the same plan, so they must agree bit for bit.
The scratch keeps whatever the previous call left in it, so a larger multi-wave plan of
another cache (its items taken from the work-queue counters) runs through the same
scratch first; a wrong scratch offset or a read of stale partials would show.  Both INT2
layouts (token-major values, and channel-major values on the tensor-core decode) run
through it.  This file runs last so that a failure here cannot hide any other test.
"""
import numpy as np
import pytest
import torch

from int2_rotated_kv_rotate_gb300 import KVCache, workloads as wl
from int2_rotated_kv_rotate_gb300 import _native as N

from helpers import MAX_ABS, REL_L2, make_pair

pytestmark = pytest.mark.gpu

SEED = 99


def close(a: torch.Tensor, b: torch.Tensor):
    x, y = a.double().cpu().numpy(), b.double().cpu().numpy()
    err = np.abs(x - y).max()
    rel = np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-30)
    return err <= MAX_ABS and rel <= REL_L2, (err, rel)


FORMATS = pytest.mark.parametrize("fmt", [N.OSCAR_FORMAT_INT2, N.OSCAR_FORMAT_INT2_CM], ids=["tm", "cm"])


def _filled(w, lens, fmt=N.OSCAR_FORMAT_INT2):
    cache, _, _ = make_pair(w, SEED, 1, len(lens), max(lens), fmt=fmt)
    slots = [cache.alloc() for _ in lens]
    ks, vs = [], []
    for r, n in enumerate(lens):
        k, v = wl.gen_kv(w, SEED, 0, r, 0, n, device="cuda")
        ks.append(k)
        vs.append(v)
    cache.reserve(slots, lens)
    cache.quantize_append(0, torch.cat(ks).contiguous(), torch.cat(vs).contiguous())
    cache.commit()
    return cache, slots


def _both(cache, q):
    """(workspace decode, no-allocation decode) fp32 outputs, and the no-alloc bf16 output."""
    ref = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    cache.decode(0, q, out_f32=ref)
    out = torch.empty_like(q)
    out32 = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    N.oscar_decode_attention_noalloc(cache.handle, 0, q, out, out32)
    torch.cuda.synchronize()
    return ref, out32, out


@FORMATS
def test_noalloc_decode_matches_workspace_decode_twice(fmt):
    w = wl.scaled(wl.WORKLOADS["tiny"], name="noalloc", lognormal_sigma=0.5)
    cache, slots = _filled(w, [1500, 700], fmt)
    cache.plan(slots, max_split_pages=3)
    assert N.oscar_decode_workspace_bytes(cache.handle) <= 8 << 20
    for step in range(2):  # two calls in a row share (and leave behind) the library scratch
        q = wl.gen_q(w, SEED, 0, step, 2, device="cuda")
        ref, out32, out = _both(cache, q)
        ok, (err, rel) = close(out32, ref)
        assert ok, f"call {step}: max-abs {err:.3e}, rel-L2 {rel:.3e}"
        assert torch.equal(out32, ref), f"call {step}: the two entry points differ"
        assert torch.equal(out.cpu(), out32.cpu().to(torch.bfloat16))
    st, flags = cache.status()
    assert st == 0 and flags == 0


@FORMATS
def test_noalloc_after_a_larger_multi_wave_plan_of_another_cache(fmt):
    """A plan of single-page items, several times more than the resident CTAs (so the CTAs
    take them from the work-queue counters), fills much of the scratch; then a smaller plan
    of the first cache reuses it.  Both agree with the workspace path bit for bit."""
    big_w = wl.scaled(wl.WORKLOADS["tiny"], name="noalloc_waves", n_q_heads=32, n_kv_heads=8, lognormal_sigma=0.5)
    big, big_slots = _filled(big_w, [6000, 5000], fmt)
    big.plan(big_slots, max_split_pages=1)
    n_items, _, _ = big.plan_info()
    assert n_items > 2 * torch.cuda.get_device_properties(0).multi_processor_count
    assert N.oscar_decode_workspace_bytes(big.handle) <= 8 << 20
    w = wl.scaled(wl.WORKLOADS["tiny"], name="noalloc_small", lognormal_sigma=0.5)
    small, small_slots = _filled(w, [1300, 400], fmt)
    for step in range(2):
        q = wl.gen_q(big_w, SEED, 0, step, 2, device="cuda")
        ref, out32, _ = _both(big, q)
        assert torch.equal(out32, ref), f"large plan, call {step}"
        small.plan(small_slots, max_split_pages=2 + step)
        q = wl.gen_q(w, SEED, 0, step, 2, device="cuda")
        ref, out32, _ = _both(small, q)
        assert torch.equal(out32, ref), f"small plan after the large one, call {step}"
    for c in (big, small):
        st, flags = c.status()
        assert st == 0 and flags == 0
        c.close()


def test_noalloc_rejects_plans_beyond_the_fixed_scratch():
    # GQA 8: one partial is 8 x 130 fp32; 2048+ single-page items exceed 8 MiB
    w = wl.scaled(wl.WORKLOADS["qwen3_32b_capacity"], name="noalloc_big", n_layers=1, batch=1, context=16384)
    cache, _, _ = make_pair(w, SEED, 1, 1, 16384, params=(np.stack([np.eye(128, dtype=np.float32)] * 8)[None],
                                                          np.stack([np.eye(128, dtype=np.float32)] * 8)[None],
                                                          np.ones((1, 8), np.float32) * 50,
                                                          np.ones((1, 8), np.float32) * 50))
    slot = cache.alloc()
    k, v = wl.gen_kv(w, SEED, 0, 0, 0, 16384, device="cuda")
    cache.reserve([slot], [16384])
    cache.quantize_append(0, k, v)
    cache.commit()
    cache.plan([slot], max_split_pages=1)
    assert N.oscar_decode_workspace_bytes(cache.handle) > 8 << 20
    q = wl.gen_q(w, SEED, 0, 0, 1, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(N.OscarError) as ei:
        N.oscar_decode_attention_noalloc(cache.handle, 0, q, out)
    assert ei.value.status == 1 and "8388608" in str(ei.value)
