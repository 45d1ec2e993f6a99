"""Pins for the CPU oracle: checks against what the pages and mathematics fix, not against
the oracle itself (CPU only).

- calibration: Hadamard and bit-reversal identities, orthogonality, eigen residuals, the
  literal covariance formulas on tiny inputs by brute force, the Hadamard-only special
  case against scipy's Hadamard routine, nearest-rank percentiles on known arrays;
- rotation chain and bf16 rounding: bit-exact against exact rational arithmetic;
- quantizer: hand-derived groups, code optimality, the scale/2 error bound;
- packing: hand-derived golden rows (tests/golden/pack_layout.json);
- append state machine: chunking invariance, routing, prefix sharing = private copy;
- decode: brute-force softmax attention, change-of-basis invariance, one-token and
  equal-logit closed forms, INT2 streams against explicit dequantisation.
"""
import json
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import calibration as cal

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- helpers
def bits(x_f32) -> np.ndarray:
    """bf16 bit patterns of float values through torch's RNE conversion (library routine)."""
    t = torch.as_tensor(np.asarray(x_f32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def round_frac(v: Fraction, mant_bits: int) -> float:
    """Exact round-to-nearest-even of a rational to a binary format with mant_bits
    significand bits (24 = binary32, 8 = bfloat16), exponent range of binary32."""
    if v == 0:
        return 0.0
    sign = -1.0 if v < 0 else 1.0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    quantum = Fraction(2) ** (e - (mant_bits - 1))
    m = a / quantum
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * float(n * quantum)


def fma_f32_exact(a: float, b: float, c: float) -> float:
    return round_frac(Fraction(a) * Fraction(b) + Fraction(c), 24)


def random_orthogonal(d, seed):
    g = np.random.default_rng(seed)
    Q, Rm = np.linalg.qr(g.standard_normal((d, d)))
    return (Q * np.sign(np.diag(Rm))).astype(np.float32)


def signed_permutation(d, seed):
    g = np.random.default_rng(seed)
    P = np.zeros((d, d), np.float32)
    perm = g.permutation(d)
    P[np.arange(d), perm] = g.choice([-1.0, 1.0], size=d)
    return P


# ----------------------------------------------------------------------------- calibration
def test_hadamard_matches_scipy_and_is_orthogonal():
    import scipy.linalg

    d = 128
    H = cal.hadamard(d)
    Hint = np.rint(H * math.sqrt(d)).astype(np.int64)
    assert np.array_equal(Hint, scipy.linalg.hadamard(d))
    assert np.array_equal(Hint @ Hint.T, d * np.eye(d, dtype=np.int64))


def test_bit_reversal_permutation():
    d = 128
    hand = {0: 0, 1: 64, 2: 32, 3: 96, 5: 80, 6: 48, 64: 1, 127: 127, 100: 19}
    for j, r in hand.items():
        assert cal.bit_reverse(j, 7) == r
    P = cal.bitrev_permutation(d)
    assert np.array_equal(P @ P, np.eye(d))  # involution
    assert np.array_equal(P.T @ P, np.eye(d))
    for j, r in hand.items():
        e = np.zeros(d)
        e[j] = 1
        assert np.argmax(P @ e) == r


def test_hadamard_only_special_case():
    """U = I gives R = H_Had P_br: column j of R is column rev(j) of scipy's Hadamard / sqrt(d)."""
    import scipy.linalg

    d = 128
    R = cal.compose_rotation(np.eye(d))
    Hs = scipy.linalg.hadamard(d) / math.sqrt(d)
    for j in range(d):
        assert np.allclose(R[:, j], Hs[:, cal.bit_reverse(j, 7)], atol=0, rtol=0)


def test_query_covariance_brute_force():
    g = np.random.default_rng(3)
    N, G, d = 5, 2, 6
    Q = g.standard_normal((N, G, d))
    C = np.zeros((d, d))
    for n in range(N):
        for h in range(G):
            for i in range(d):
                for j in range(d):
                    C[i, j] += Q[n, h, i] * Q[n, h, j]
    C /= N * G
    assert np.allclose(cal.query_covariance(Q), C, atol=1e-13)


def test_score_value_covariance_is_vt_st_s_v():
    """C_S = (1/N) V^T S^T S V, S the causal softmax, built here element by element."""
    g = np.random.default_rng(4)
    N, G, d = 6, 2, 4
    Q = g.standard_normal((N, G, d))
    K = g.standard_normal((N, d))
    V = g.standard_normal((N, d))
    C = np.zeros((d, d))
    for h in range(G):
        S = np.zeros((N, N))
        for i in range(N):
            w = [math.exp(sum(Q[i, h, c] * K[j, c] for c in range(d)) / math.sqrt(d)) for j in range(i + 1)]
            for j in range(i + 1):
                S[i, j] = w[j] / sum(w)
        C += V.T @ S.T @ S @ V
    C /= N * G
    assert np.allclose(cal.score_value_covariance(Q, K, V), C, atol=1e-13)


def test_eigendecomposition_residual_order_and_sign():
    g = np.random.default_rng(5)
    A = g.standard_normal((128, 64))
    C = A @ A.T / 64 + np.diag(np.linspace(0, 1, 128))
    w, U = cal.eig_desc(C)
    assert np.all(np.diff(w) <= 0)
    assert np.linalg.norm(C @ U - U * w) < 1e-8 * np.linalg.norm(C)
    assert np.allclose(U.T @ U, np.eye(128), atol=1e-12)
    for k in range(128):
        assert U[np.argmax(np.abs(U[:, k])), k] > 0


def test_nearest_rank_percentile():
    v = np.arange(1, 1001, dtype=np.float64)
    np.random.default_rng(0).shuffle(v)
    assert cal.nearest_rank_percentile(v, 99.9) == 999
    assert cal.nearest_rank_percentile(v, 50) == 500
    assert cal.nearest_rank_percentile(v, 100) == 1000
    assert cal.nearest_rank_percentile(v, 0.05) == 1
    assert cal.nearest_rank_percentile(np.array([7.0]), 99.9) == 7.0


def test_calibrated_rotations_are_orthogonal():
    from int2_rotated_kv_rotate_gb300 import workloads as wl

    w = wl.WORKLOADS["tiny"]
    q, k, v = wl.gen_calibration(w, 11, 0)
    RK, RV, cK, cV = cal.calibrate_layer(q.float().numpy(), k.float().numpy(), v.float().numpy(), 99.9)
    for R in list(RK) + list(RV):
        R64 = R.astype(np.float64)
        assert np.abs(R64.T @ R64 - np.eye(128)).max() < 1e-6
    # clip is an order statistic of |R^T x|: about 0.1% of calibration entries exceed it
    for h in range(w.n_kv_heads):
        rot = np.abs(k[:, h].float().numpy().astype(np.float64) @ RK[h].astype(np.float64))
        frac = np.mean(rot > cK[h])
        assert frac <= 0.001 + 1e-9 and frac > 0.0005
    assert np.all(cK > 0) and np.all(cV > 0)


# ----------------------------------------------------------------------------- bf16 + rotation
def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(6)
    x = np.concatenate([
        g.standard_normal(2000).astype(np.float32) * 10,
        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 3.0e38, 1e-40, -1e-41, 0.0, -0.0,
                  np.inf, -np.inf], np.float32),
    ])
    ours = oracle.f32_to_bf16(x)
    assert np.array_equal(ours, bits(x))
    assert oracle.f32_to_bf16(np.array([np.nan], np.float32))[0] == 0x7FFF


def test_rotation_chain_bit_exact_against_rationals():
    d = 128
    R = random_orthogonal(d, 7)
    g = np.random.default_rng(8)
    x = bits(g.standard_normal((3, d)) * np.array([20.0 if c in (3, 77) else 1.0 for c in range(d)]))
    r = oracle.rotate(R, x)
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    for t in range(x.shape[0]):
        for j in range(d):
            acc = 0.0
            for i in range(d):
                acc = fma_f32_exact(float(R[i, j]), float(xf[t, i]), acc)
            expect = round_frac(Fraction(acc), 8)
            got = float(oracle.bf16_to_f32(r[t, j]))
            assert got == expect, (t, j, got, expect)


def test_rotation_identity_and_permutation():
    d = 128
    g = np.random.default_rng(9)
    x = bits(g.standard_normal((5, d)))
    assert np.array_equal(oracle.rotate(np.eye(d, dtype=np.float32), x), x)
    P = signed_permutation(d, 10)
    r = oracle.rotate(P, x)
    # r = P^T x exactly (one nonzero term per output; sign flip is exact in bf16)
    expect = oracle.bf16_to_f32(x).astype(np.float64) @ P.astype(np.float64)
    assert np.array_equal(oracle.bf16_to_f32(r).astype(np.float64), expect)


# ----------------------------------------------------------------------------- quantizer
def group_token(values):
    return bits(np.asarray(values, np.float32))


def test_quantizer_hand_examples():
    inf = float("inf")
    # values 0,1,2,3 repeated: s = 1, z = 0, codes = values
    r = group_token([c % 4 for c in range(128)])
    row, sz = oracle.quantize_token(r, 128, inf)
    assert list(sz) == list(bits([1.0, 0.0]))
    assert list(oracle.unpack_row(row)) == [c % 4 for c in range(128)]
    # constant group: s = 0, every code 0, dequantised value = z exactly
    row, sz = oracle.quantize_token(group_token([1.5] * 128), 128, inf)
    assert list(sz) == list(bits([0.0, 1.5]))
    assert not row.any()
    assert np.all(oracle.dequant_token(row, sz, 128) == 1.5)
    # clipping at c = 10: [100, -100, 0, 0, ...] -> x = [10, -10, 0 ...];
    # s = bf16(20/3) = 6.65625, z = -10; codes 3, 0, round(10/6.65625 = 1.50235) = 2
    vals = [0.0] * 128
    vals[0], vals[1] = 100.0, -100.0
    row, sz = oracle.quantize_token(group_token(vals), 128, 10.0)
    assert list(sz) == list(bits([6.65625, -10.0]))
    codes = oracle.unpack_row(row)
    assert codes[0] == 3 and codes[1] == 0 and np.all(codes[2:] == 2)
    # g = 32: each group gets its own scale/zero
    vals = [float(c // 32) * 10 + (c % 4) for c in range(128)]
    row, sz = oracle.quantize_token(group_token(vals), 32, inf)
    assert list(sz) == list(bits([1.0, 0.0, 1.0, 10.0, 1.0, 20.0, 1.0, 30.0]))
    assert list(oracle.unpack_row(row)) == [c % 4 for c in range(128)]


@pytest.mark.parametrize("g_size", [128, 32])
def test_quantizer_codes_nearest_and_error_bound(g_size):
    rng = np.random.default_rng(12)
    for trial in range(40):
        scale = float(rng.choice([0.01, 1.0, 7.0, 300.0]))
        clip = float(rng.choice([np.inf, 2.0 * scale]))
        r = bits(rng.standard_normal(128) * scale)
        row, sz = oracle.quantize_token(r, g_size, clip)
        codes = oracle.unpack_row(row)
        x = np.clip(oracle.bf16_to_f32(r).astype(np.float64), -clip, clip)
        xhat = oracle.dequant_token(row, sz, g_size).astype(np.float64)
        for grp in range(128 // g_size):
            sl = slice(grp * g_size, (grp + 1) * g_size)
            s = float(oracle.bf16_to_f32(sz[2 * grp]))
            z = float(oracle.bf16_to_f32(sz[2 * grp + 1]))
            mn, mx = x[sl].min(), x[sl].max()
            assert abs(z - mn) <= abs(mn) * 2 ** -8 + 1e-38
            assert abs(s - (mx - mn) / 3) <= (mx - mn) / 3 * 2 ** -8 + 1e-38
            for i in range(grp * g_size, (grp + 1) * g_size):
                u = (Fraction(float(x[i])) - Fraction(z)) / Fraction(s)
                c = int(codes[i])
                # nearest level, ties within fp32 rounding of the quotient allowed either way
                best = min(range(4), key=lambda k: abs(u - k))
                assert c == best or abs(abs(u - c) - abs(u - best)) < 1e-5, (u, c, best)
            bound = 0.5 * s + abs(z - mn) + 3 * abs(s - (mx - mn) / 3) + 1e-6 * max(1.0, np.abs(x[sl]).max())
            assert np.abs(x[sl] - xhat[sl]).max() <= bound


def test_history_bytes_per_token():
    """72 B per token-head for g = 128 (2.25 bits/element), 96 B for g = 32 (3.0 bits)."""
    r = bits(np.linspace(-1, 1, 128))
    for g, expect in ((128, 72), (32, 96)):
        row, sz = oracle.quantize_token(r, g, 5.0)
        per_tensor = row.nbytes + sz.nbytes
        assert 2 * per_tensor == expect
        assert per_tensor * 8 / 128 == {128: 2.25, 32: 3.0}[g]
    assert 16 / 2.25 == pytest.approx(7.11, abs=0.01)  # vs BF16 at long context


# ----------------------------------------------------------------------------- packing
def test_pack_layout_golden():
    with open(os.path.join(GOLDEN, "pack_layout.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        codes = np.zeros(128, np.uint8)
        if "pattern" in case:
            codes[:] = [eval(case["pattern"], {"c": c}) for c in range(128)]  # noqa: S307 (fixture text)
        for c, v in case.get("set", {}).items():
            codes[int(c)] = v
        row = oracle.pack_row(codes)
        assert row.tolist() == [int(b, 16) for b in case["row_hex"]], case["name"]
        assert np.array_equal(oracle.unpack_row(row), codes)


def test_pack_roundtrip_random():
    rng = np.random.default_rng(13)
    for _ in range(50):
        codes = rng.integers(0, 4, 128).astype(np.uint8)
        assert np.array_equal(oracle.unpack_row(oracle.pack_row(codes)), codes)
    positions = sorted(oracle.code_bitpos(c) for c in range(128))
    assert positions == list(range(0, 256, 2))  # a bijection onto the 128 two-bit fields


# ----------------------------------------------------------------------------- state machine
def make_streams(S=4, W=64, g=128, cap=600, seed=14, clip=3.0):
    R = random_orthogonal(128, seed)
    return [oracle.Stream(128, g, S, W, cap, R, clip) for _ in range(2)], R


def stream_state(s):
    """Logical content: sinks held, ring slots of positions [H, L), INT2 rows of [S, H)."""
    L, H = s.length, s.history_end
    ring = b"".join(s.ring[p % s.W].tobytes() for p in range(H, L))
    rows = s.rows[s.S:H].tobytes() if s.S < H else b""
    sz = s.sz[s.S:H].tobytes() if s.S < H else b""
    return (L, H, s.sink[:min(L, s.S)].tobytes(), ring, rows, sz)


@pytest.mark.parametrize("W", [64, 16, 0])
def test_append_chunking_invariance_and_routing(W):
    rng = np.random.default_rng(15)
    x = bits(rng.standard_normal((500, 128)) * 2)
    (a, b), R = make_streams(W=W)
    a.append(x)
    pos = 0
    while pos < 500:
        n = int(rng.choice([1, 2, 3, 17, 64, 100]))
        b.append(x[pos:pos + n])
        pos += n
        # invariant after every append: exactly the last W tokens beyond the sinks are BF16
        assert b.history_end == max(b.S, b.length - W)
    assert stream_state(a) == stream_state(b)
    r = oracle.rotate(R, x)
    for p in range(500):
        route = a.route(p)
        if route == "sink":
            assert np.array_equal(a.sink[p], r[p])
        elif route == "ring":
            assert np.array_equal(a.ring[p % W], r[p])
        else:
            row, sz = oracle.quantize_token(r[p], 128, 3.0)
            assert np.array_equal(a.rows[p], row) and np.array_equal(a.sz[p], sz)


def test_prefix_share_equals_private_copy():
    rng = np.random.default_rng(16)
    x = bits(rng.standard_normal((400, 128)))
    (src, dst), _ = make_streams(W=64)
    (priv, _unused), _ = make_streams(W=64)
    src.append(x[:300])
    n = 192  # full pages below src's window (history end 236)
    dst.share_from(src, n)
    dst.append(x[n:400])
    priv.append(x[:400])
    assert stream_state(dst) == stream_state(priv)


# ----------------------------------------------------------------------------- decode
def brute_attention(q, K, V):
    """softmax(q K^T / sqrt(d)) V in fp64, written out directly."""
    out = np.zeros((q.shape[0], K.shape[1]))
    for h in range(q.shape[0]):
        logits = np.array([np.dot(q[h], K[t]) / math.sqrt(K.shape[1]) for t in range(K.shape[0])])
        w = np.exp(logits - logits.max())
        out[h] = (w[:, None] * V).sum(0) / w.sum()
    return out


def f64(b):
    return oracle.bf16_to_f32(b).astype(np.float64)


def test_decode_bf16_bypass_identity_rotation():
    """W >= L and R = I: every token stays BF16 and decode is plain softmax attention."""
    rng = np.random.default_rng(17)
    I = np.eye(128, dtype=np.float32)
    K = oracle.Stream(128, 128, 4, 64, 64, I, 1.0)
    V = oracle.Stream(128, 128, 4, 64, 64, I, 1.0)
    xk, xv = bits(rng.standard_normal((50, 128)) * 3), bits(rng.standard_normal((50, 128)))
    K.append(xk)
    V.append(xv)
    q = bits(rng.standard_normal((4, 128)))
    got = oracle.decode(q, K, V, I, I)
    assert np.allclose(got, brute_attention(f64(q), f64(xk), f64(xv)), atol=1e-12, rtol=0)


@pytest.mark.parametrize("exact", [True, False])
def test_decode_change_of_basis_invariance(exact):
    """Scores in the rotated basis with q~ = R_K^T q and o = R_V o~ equal plain attention
    over the stored tokens mapped back to the original basis."""
    rng = np.random.default_rng(18)
    RK = signed_permutation(128, 19) if exact else random_orthogonal(128, 19)
    RV = signed_permutation(128, 20) if exact else random_orthogonal(128, 20)
    K = oracle.Stream(128, 128, 4, 64, 64, RK, 1.0)
    V = oracle.Stream(128, 128, 4, 64, 64, RV, 1.0)
    xk, xv = bits(rng.standard_normal((40, 128)) * 3), bits(rng.standard_normal((40, 128)))
    K.append(xk)
    V.append(xv)
    q = bits(rng.standard_normal((4, 128)))
    got = oracle.decode(q, K, V, RK, RV)
    stored_k = np.array([f64(K.sink[p]) if p < 4 else f64(K.ring[p % 64]) for p in range(40)])
    stored_v = np.array([f64(V.sink[p]) if p < 4 else f64(V.ring[p % 64]) for p in range(40)])
    back_k = stored_k @ RK.astype(np.float64).T  # x = R r
    back_v = stored_v @ RV.astype(np.float64).T
    assert np.allclose(got, brute_attention(f64(q), back_k, back_v), atol=1e-10, rtol=0)
    if exact:  # the rotation is exact, so this is attention over the original tokens
        assert np.allclose(got, brute_attention(f64(q), f64(xk), f64(xv)), atol=1e-12, rtol=0)


@pytest.mark.parametrize("exact", [True, False])
def test_folded_decode_is_attention_in_the_rotated_basis(exact):
    """With the rotations folded into the model's projections the oracle takes q~ (bf16)
    and returns o~: plain attention of q~ over the stored rotated keys and values (INT2
    history dequantised by hand here); with a signed permutation (exact rotations) o~ is
    R_V^T of the unfolded decode of q."""
    rng = np.random.default_rng(31)
    RK = signed_permutation(128, 32) if exact else random_orthogonal(128, 32)
    RV = signed_permutation(128, 33) if exact else random_orthogonal(128, 33)
    K = oracle.Stream(128, 32, 4, 64, 320, RK, 4.0)
    V = oracle.Stream(128, 32, 4, 64, 320, RV, 4.0)
    xk, xv = bits(rng.standard_normal((300, 128)) * 2), bits(rng.standard_normal((300, 128)))
    K.append(xk)
    V.append(xv)
    q = bits(rng.standard_normal((4, 128)))
    qt = bits((f64(q) @ RK.astype(np.float64)))  # q~ = R_K^T q (rows), rounded to bf16

    def stored(st, p):
        route = st.route(p)
        if route == "sink":
            return f64(st.sink[p])
        if route == "ring":
            return f64(st.ring[p % 64])
        return oracle.dequant_token(st.rows[p], st.sz[p], 32).astype(np.float64)

    sk = np.array([stored(K, p) for p in range(300)])
    sv = np.array([stored(V, p) for p in range(300)])
    assert K.route(100) == "int2"
    got = oracle.decode_folded(qt, K, V)
    assert np.allclose(got, brute_attention(f64(qt), sk, sv), atol=1e-12, rtol=0)
    if exact:  # q~ is exact, so the folded output is R_V^T times the unfolded one
        full = oracle.decode(q, K, V, RK, RV)
        assert np.allclose(got, full @ RV.astype(np.float64), atol=1e-12, rtol=0)
    assert not np.any(oracle.decode_folded(np.zeros((2, 128), np.uint16), oracle.Stream(128, 32, 4, 64, 8, RK, 1.0),
                                           oracle.Stream(128, 32, 4, 64, 8, RV, 1.0)))


def test_decode_single_token_and_equal_logits():
    rng = np.random.default_rng(21)
    RK, RV = signed_permutation(128, 22), signed_permutation(128, 23)
    K = oracle.Stream(128, 128, 4, 8, 64, RK, 1.0)
    V = oracle.Stream(128, 128, 4, 8, 64, RV, 1.0)
    xk, xv = bits(rng.standard_normal((1, 128))), bits(rng.standard_normal((1, 128)))
    K.append(xk)
    V.append(xv)
    q = bits(rng.standard_normal((2, 128)) * 5)
    got = oracle.decode(q, K, V, RK, RV)
    assert np.array_equal(got, np.repeat(f64(xv), 2, axis=0))  # one token: o = v exactly
    xk2, xv2 = bits(rng.standard_normal((13, 128))), bits(rng.standard_normal((13, 128)))
    K.append(xk2)
    V.append(xv2)
    zero_q = np.zeros((2, 128), np.uint16)
    got = oracle.decode(zero_q, K, V, RK, RV)
    allv = np.concatenate([f64(xv), f64(xv2)])
    # equal logits: uniform weights over the 14 stored values (positions 4, 5 now INT2)
    Vals = []
    for p in range(14):
        route = V.route(p)
        r = V.sink[p] if route == "sink" else (V.ring[p % 8] if route == "ring" else None)
        Vals.append(f64(r) if r is not None else oracle.dequant_token(V.rows[p], V.sz[p], 128).astype(np.float64))
    expect = np.mean(np.array(Vals) @ RV.astype(np.float64).T, axis=0)
    assert np.allclose(got, np.repeat(expect[None], 2, axis=0), atol=1e-12, rtol=0)
    assert V.route(4) == "int2" and np.abs(expect - allv.mean(0)).max() > 0  # INT2 error is visible


@pytest.mark.parametrize("g_size", [128, 32])
def test_decode_int2_stream_against_explicit_dequantisation(g_size):
    rng = np.random.default_rng(24)
    RK, RV = random_orthogonal(128, 25), random_orthogonal(128, 26)
    K = oracle.Stream(128, g_size, 4, 32, 400, RK, 9.0)
    V = oracle.Stream(128, g_size, 4, 32, 400, RV, 4.0)
    xk = bits(rng.standard_normal((300, 128)) * np.where(np.arange(128) % 37 == 0, 20, 1))
    xv = bits(rng.standard_normal((300, 128)))
    for chunk in np.array_split(np.arange(300), 7):
        K.append(xk[chunk])
        V.append(xv[chunk])
    q = bits(rng.standard_normal((4, 128)))
    got = oracle.decode(q, K, V, RK, RV)

    def stored(S, p):
        route = S.route(p)
        if route == "sink":
            return f64(S.sink[p])
        if route == "ring":
            return f64(S.ring[p % S.W])
        return oracle.dequant_token(S.rows[p], S.sz[p], g_size).astype(np.float64)

    Ks = np.array([stored(K, p) for p in range(300)])
    Vs = np.array([stored(V, p) for p in range(300)])
    qt = f64(q) @ RK.astype(np.float64)
    expect = brute_attention(qt, Ks, Vs) @ RV.astype(np.float64).T
    assert np.allclose(got, expect, atol=1e-11, rtol=0)


def test_decode_empty_context_is_zero():
    I = np.eye(128, dtype=np.float32)
    K = oracle.Stream(128, 128, 4, 8, 8, I, 1.0)
    V = oracle.Stream(128, 128, 4, 8, 8, I, 1.0)
    assert not oracle.decode(bits(np.ones((2, 128))), K, V, I, I).any()


# ----------------------------------------------------------------------------- quantizer ties
def test_quantizer_rounds_exact_ties_to_even():
    """Groups whose (x - z) / s lands exactly on 0.5, 1.5 and 2.5 take codes 0, 2 and 2
    (round half to even); rounding half away from zero would give 1, 2 and 3."""
    inf = float("inf")
    cases = [
        ([0.0, 3.0] + [0.5, 1.5, 2.5] * 42, [1.0, 0.0]),  # s = 1, z = 0
        ([0.0, 6.0] + [1.0, 3.0, 5.0] * 42, [2.0, 0.0]),  # s = 2, z = 0
        ([-1.0, 2.0] + [-0.5, 0.5, 1.5] * 42, [1.0, -1.0]),  # s = 1, z = -1
    ]
    for vals, sz_expect in cases:
        row, sz = oracle.quantize_token(group_token(vals), 128, inf)
        assert list(sz) == list(bits(sz_expect))
        codes = oracle.unpack_row(row)
        assert codes[0] == 0 and codes[1] == 3
        assert list(codes[2:]) == [0, 2, 2] * 42, vals[:5]
    # g = 32: each group on its own, ties in every group
    vals = []
    for grp in range(4):
        base = float(4 * grp)
        vals += [base, base + 3.0] + [base + 0.5, base + 1.5, base + 2.5] * 10
    row, sz = oracle.quantize_token(group_token(vals), 32, inf)
    codes = oracle.unpack_row(row)
    for grp in range(4):
        assert list(codes[32 * grp:32 * grp + 32]) == [0, 3] + [0, 2, 2] * 10


# ----------------------------------------------------------------------------- BF16 comparison decode
def softmax_attention_loops(qf, Kf, Vf):
    """softmax(q K^T / sqrt(d)) V spelled out token by token with Python floats."""
    G, d = qf.shape
    out = np.zeros((G, d))
    for h in range(G):
        logits = []
        for t in range(Kf.shape[0]):
            logits.append(math.fsum(float(qf[h, c]) * float(Kf[t, c]) for c in range(d)) / math.sqrt(d))
        m = max(logits)
        w = [math.exp(x - m) for x in logits]
        tot = math.fsum(w)
        for t in range(Kf.shape[0]):
            out[h] += (w[t] / tot) * Vf[t]
    return out


@pytest.mark.parametrize("L,G", [(1, 4), (2, 8), (7, 4), (64, 8), (129, 4)])
def test_bf16_comparison_decode_brute_force(L, G):
    """The uncompressed comparison's reference: plain attention over every one of the L
    tokens, with the 1/sqrt(d) logit scale (sharp logits make a dropped scale or a
    dropped token visible)."""
    rng = np.random.default_rng(100 + L)
    K = bits(rng.standard_normal((L, 128)) * 4)
    V = bits(rng.standard_normal((L, 128)) * np.where(np.arange(128) % 50 == 0, 8.0, 1.0))
    q = bits(rng.standard_normal((G, 128)))
    got = oracle.bf16_decode(q, K, V)
    assert np.allclose(got, softmax_attention_loops(f64(q), f64(K), f64(V)), atol=1e-12, rtol=0)


def test_bf16_comparison_decode_closed_forms():
    rng = np.random.default_rng(120)
    K = bits(rng.standard_normal((1, 128)) * 3)
    V = bits(rng.standard_normal((1, 128)))
    q = bits(rng.standard_normal((4, 128)) * 7)
    # one token: every head's output is that token's value, exactly
    assert np.array_equal(oracle.bf16_decode(q, K, V), np.repeat(f64(V), 4, axis=0))
    # equal logits (q = 0): the mean of the values
    K = bits(rng.standard_normal((37, 128)) * 3)
    V = bits(rng.standard_normal((37, 128)))
    got = oracle.bf16_decode(np.zeros((8, 128), np.uint16), K, V)
    assert np.allclose(got, np.repeat(f64(V).mean(0)[None], 8, axis=0), atol=1e-14, rtol=0)
    # two tokens with logits a and b: weights 1 / (1 + e^(b - a)) and the rest
    K = np.zeros((2, 128), np.uint16)
    K[0, 0] = bits([2.0])[0]
    K[1, 0] = bits([-1.0])[0]
    V = bits(rng.standard_normal((2, 128)))
    q = np.zeros((1, 128), np.uint16)
    q[0, 0] = bits([math.sqrt(128.0) * 0.5])[0]  # exact in bf16? sqrt(128)/2 is not: use its bf16 value
    qv = float(f64(q)[0, 0])
    a, b = qv * 2.0 / math.sqrt(128), qv * -1.0 / math.sqrt(128)
    w0 = 1.0 / (1.0 + math.exp(b - a))
    expect = w0 * f64(V)[0] + (1 - w0) * f64(V)[1]
    assert np.allclose(oracle.bf16_decode(q, K, V)[0], expect, atol=1e-14, rtol=0)
    # no tokens: zeros
    assert not oracle.bf16_decode(q, np.zeros((0, 128), np.uint16), np.zeros((0, 128), np.uint16)).any()


# ----------------------------------------------------------------------------- calibration wiring
def independent_hadamard_bitrev(d):
    """H_Had from its entries, (-1)^popcount(i & j) / sqrt(d), and the bit-reversal map."""
    nbits = d.bit_length() - 1
    H = np.array([[(-1) ** bin(i & j).count("1") for j in range(d)] for i in range(d)], np.float64) / math.sqrt(d)
    rev = [int(format(j, f"0{nbits}b")[::-1], 2) for j in range(d)]
    P = np.zeros((d, d))
    P[rev, np.arange(d)] = 1.0  # column j of P_br is e_rev(j)
    return H, P, rev


def test_compose_rotation_order_with_a_general_basis():
    """R = U H_Had P_br for a U that is not the identity: column j of R is U H e_rev(j),
    and none of the other orders of the three factors gives the same matrix."""
    d = 128
    U = random_orthogonal(d, 31).astype(np.float64)
    H, P, rev = independent_hadamard_bitrev(d)
    R = cal.compose_rotation(U)
    for j in range(d):
        assert np.allclose(R[:, j], U @ H[:, rev[j]], atol=1e-13, rtol=0), j
    # (H_Had and P_br commute, since H_Had[rev i][rev j] = H_Had[i][j], so U P_br H_Had is the
    # same matrix; every order that moves U is not)
    assert np.abs(U @ P @ H - U @ H @ P).max() < 1e-13
    for wrong in (H @ U @ P, P @ H @ U, H @ P @ U, P @ U @ H):
        assert np.abs(R - wrong).max() > 0.1


def rows_with_covariance(U, sigma, n, seed):
    """n rows x with (1/n) sum x^T x = U diag(sigma^2) U^T (exact up to fp64 rounding)."""
    g = np.random.default_rng(seed)
    Z, _ = np.linalg.qr(g.standard_normal((n, U.shape[0])))  # orthonormal columns
    return math.sqrt(n) * Z @ np.diag(sigma) @ U.T


def causal_softmax_rows(Qh, K):
    """S[i, j] = exp(l_ij) / sum_{j' <= i} exp(l_ij') for j <= i, l = q_i . k_j / sqrt(d), row by row."""
    n, d = Qh.shape
    S = np.zeros((n, n))
    for i in range(n):
        l = K[:i + 1] @ Qh[i] / math.sqrt(d)
        e = np.exp(l - l.max())
        S[i, :i + 1] = e / e.sum()
    return S


def test_calibrate_head_recovers_the_key_eigenbasis_and_wires_values_to_c_s():
    """Key queries with a known covariance U diag(sigma^2) U^T: the key rotation's basis
    U_Q = R_K P_br^T H_Had^T is U with its columns in descending-variance order, each with its
    largest-magnitude entry positive.  The value rotation's basis diagonalises C_S (built
    here from its definition, V^T S^T S V / N pooled over the query heads) with the
    eigenvalues descending, and it is not the key basis."""
    d, N, G = 128, 384, 2
    U_true = random_orthogonal(d, 40).astype(np.float64)
    sigma = np.geomspace(4.0, 0.25, d)  # distinct, descending
    Q = rows_with_covariance(U_true, sigma, N * G, 41).reshape(N, G, d)
    g = np.random.default_rng(42)
    K = g.standard_normal((N, d))
    V = g.standard_normal((N, d)) * np.geomspace(6.0, 0.5, d)  # anisotropic values, a different basis
    RK, RV, cK, cV = cal.calibrate_head(Q, K, V, 99.9)
    H, P, _ = independent_hadamard_bitrev(d)
    U_K = RK.astype(np.float64) @ P.T @ H.T
    expect = U_true.copy()
    for k in range(d):
        i = int(np.argmax(np.abs(expect[:, k])))
        if expect[i, k] < 0:
            expect[:, k] = -expect[:, k]
    assert np.abs(U_K - expect).max() < 1e-5
    C_S = np.zeros((d, d))
    for h in range(G):
        O = causal_softmax_rows(Q[:, h], K) @ V
        C_S += O.T @ O
    C_S /= N * G
    U_V = RV.astype(np.float64) @ P.T @ H.T
    D = U_V.T @ C_S @ U_V
    diag = np.diag(D)
    assert np.abs(D - np.diag(diag)).max() < 1e-5 * diag.max()
    assert np.all(np.diff(diag) <= 1e-6 * diag.max()) and diag[0] > 2 * diag[-1]
    # wiring: the key basis does not diagonalise C_S, nor the value basis C_Q
    C_Q = U_true @ np.diag(sigma ** 2) @ U_true.T
    DK = U_K.T @ C_S @ U_K
    DV = U_V.T @ C_Q @ U_V
    assert np.abs(DK - np.diag(np.diag(DK))).max() > 1e-2 * diag.max()
    assert np.abs(DV - np.diag(np.diag(DV))).max() > 1e-2 * sigma[0] ** 2
