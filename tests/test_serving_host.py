"""Host logic of the serving loop (CPU): request generation, the token pools' stream
mapping (a group's shared prefix is the same tokens for every request of the group) and
the page rule it budgets with."""
import torch

from int2_rotated_kv_rotate_gb300 import serving, workloads as wl
from int2_rotated_kv_rotate_gb300 import _native as N


def test_requests_are_seeded_and_grouped():
    a = serving.make_requests(10, (100, 200), (3, 9), n_groups=3, seed=5)
    b = serving.make_requests(10, (100, 200), (3, 9), n_groups=3, seed=5)
    assert [(r.prompt, r.gen, r.group) for r in a] == [(r.prompt, r.gen, r.group) for r in b]
    assert all(100 <= r.prompt <= 200 and 3 <= r.gen <= 9 for r in a)
    assert [r.group for r in a] == [i % 3 for i in range(10)]
    assert serving.make_requests(4, (1, 2), (1, 2), n_groups=0, seed=1)[0].group == -1


def test_prefix_tokens_are_shared_within_a_group_only():
    w = wl.scaled(wl.WORKLOADS["tiny"], name="serving_host")
    src = serving.TokenSource(w, 3, pool_tokens=512, device="cpu")
    r0, r1, r2 = (serving.Request(rid=i, prompt=300, gen=1, group=g) for i, g in ((0, 0), (1, 0), (2, 1)))
    prefix = 128
    rows = lambda r, a, n, layer=0: src.index(layer, [(serving.TokenSource.stream(r, p, prefix), p, 1)  # noqa: E731
                                                      for p in range(a, a + n)])
    assert torch.equal(rows(r0, 0, prefix), rows(r1, 0, prefix))  # same group: same prefix tokens
    assert not torch.equal(rows(r0, 0, prefix), rows(r2, 0, prefix))  # another group
    assert not torch.equal(rows(r0, prefix, 50), rows(r1, prefix, 50))  # beyond the prefix: own tokens
    assert not torch.equal(rows(r0, 0, prefix, layer=0), rows(r0, 0, prefix, layer=1))
    assert int(rows(r0, 0, 600).max()) < 512 and src.K.shape == (512, w.n_kv_heads, 128)


def test_page_rule():
    # INT2: pages hold history rows [S, H), H = max(S, L - W); BF16: every token
    I, B = N.OSCAR_FORMAT_INT2, N.OSCAR_FORMAT_BF16
    assert serving.pages_needed(I, 100, 4, 128) == 0
    assert serving.pages_needed(I, 132, 4, 128) == 0
    assert serving.pages_needed(I, 133, 4, 128) == 1
    assert serving.pages_needed(I, 128 + 64 + 1, 4, 128) == 2
    assert serving.pages_needed(I, 1000, 4, 0) == 16
    assert serving.pages_needed(B, 1, 0, 0) == 1 and serving.pages_needed(B, 128, 0, 0) == 2
