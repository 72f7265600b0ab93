"""Pins for the oracle's building blocks (CPU only).

Every check compares against something other than the oracle's own formula:
a closed form, a special case that reduces to a textbook identity or a library
routine (scipy), or brute force.
"""
import math
import os

import numpy as np
import pytest
import scipy.special

from oracle import llama as L
from oracle import quant as Q

GOLD = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


# ------------------------------------------------------------------ RMSNorm
def test_rmsnorm_unit_rms_closed_form():
    # With g = 1, y = x / sqrt(m + eps) so rms(y) = sqrt(m / (m + eps)), m = mean(x^2).
    for eps in (1e-5, 1e-2, 0.5):
        x = rng.standard_normal(257) * 3.0
        m = np.mean(x * x)
        y = L.rmsnorm(x, np.ones_like(x), eps)
        assert np.sqrt(np.mean(y * y)) == pytest.approx(math.sqrt(m / (m + eps)), rel=1e-13)


def test_rmsnorm_gain_is_elementwise_and_scale_invariant():
    x = rng.standard_normal(64)
    g = rng.standard_normal(64)
    y1 = L.rmsnorm(x, np.ones(64), 0.0)
    assert np.allclose(L.rmsnorm(x, g, 0.0), y1 * g, rtol=1e-14)
    assert np.allclose(L.rmsnorm(7.5 * x, np.ones(64), 0.0), y1, rtol=1e-13)


# ------------------------------------------------------------------ RoPE
def test_rope_golden_unit_vectors():
    rows = np.loadtxt(os.path.join(GOLD, "rope_hd4.txt"))
    # the fixture itself is cos/sin of 1 and of fp32(0.01)
    a1 = float(np.float32(1e4 ** -0.5))
    assert rows[0, 0] == pytest.approx(math.cos(1.0), abs=1e-15)
    assert rows[0, 2] == pytest.approx(math.sin(1.0), abs=1e-15)
    assert rows[1, 3] == pytest.approx(math.sin(a1), abs=1e-15)
    out = np.stack([L.rope(np.eye(4)[j], 1, 1e4) for j in range(4)])
    assert np.allclose(out, rows, atol=1e-15)


def test_rope_matches_complex_rotation():
    # rotate-half RoPE == multiplying (x_i + i x_{i+h}) by exp(i * angle_i)
    hd, theta = 64, 1e4
    v = rng.standard_normal((3, hd))
    for pos in (0, 1, 17, 1000, 8191):
        ang = (np.float32(pos) * (theta ** (-(2.0 * np.arange(hd // 2)) / hd)).astype(np.float32)).astype(np.float32)
        z = (v[:, : hd // 2] + 1j * v[:, hd // 2:]) * np.exp(1j * ang.astype(np.float64))
        want = np.concatenate([z.real, z.imag], axis=1)
        assert np.allclose(L.rope(v, pos, theta), want, rtol=1e-13, atol=1e-14)


def test_rope_norm_identity_and_relative_position():
    hd = 128
    q, k = rng.standard_normal(hd), rng.standard_normal(hd)
    assert np.allclose(L.rope(q, 0, 5e5), q, rtol=0, atol=0)
    for pos in (1, 77, 8000):
        assert np.linalg.norm(L.rope(q, pos, 5e5)) == pytest.approx(np.linalg.norm(q), rel=1e-13)
    # <R(p)q, R(p')k> depends on p - p' only (up to the fp32 angle rounding)
    d1 = L.rope(q, 10, 1e4) @ L.rope(k, 7, 1e4)
    d2 = L.rope(q, 103, 1e4) @ L.rope(k, 100, 1e4)
    assert d1 == pytest.approx(d2, rel=1e-4, abs=1e-5)


# ------------------------------------------------------------------ softmax / attention
def test_softmax_rows_sum_to_one_and_match_scipy():
    s = rng.standard_normal((5, 33)) * 10
    p = L.softmax(s)
    assert np.allclose(p.sum(axis=-1), 1.0, rtol=0, atol=1e-15)
    assert np.allclose(p, scipy.special.softmax(s, axis=-1), rtol=1e-13)
    assert np.allclose(L.softmax(s + 1000.0), p, rtol=1e-12)


def test_attention_single_position_returns_v():
    q, K, V = rng.standard_normal(64), rng.standard_normal((1, 64)), rng.standard_normal((1, 64))
    assert np.array_equal(L.attention_head(q, K, V), V[0])


def test_attention_zero_keys_is_mean_of_values():
    V = rng.standard_normal((9, 64))
    out = L.attention_head(rng.standard_normal(64), np.zeros((9, 64)), V)
    assert np.allclose(out, V.mean(axis=0), rtol=1e-13)


def test_attention_matches_scipy_weights():
    q, K, V = rng.standard_normal(128), rng.standard_normal((40, 128)), rng.standard_normal((40, 128))
    w = scipy.special.softmax(np.array([K[j] @ q for j in range(40)]) / math.sqrt(128))
    assert np.allclose(L.attention_head(q, K, V), sum(w[j] * V[j] for j in range(40)), rtol=1e-12)


def test_gqa_equals_mha_with_repeated_heads():
    hq, hkv, n, hd = 8, 2, 11, 16
    q = rng.standard_normal((hq, hd))
    K, V = rng.standard_normal((hkv, n, hd)), rng.standard_normal((hkv, n, hd))
    rep = hq // hkv
    K_rep = np.stack([K[i // rep] for i in range(hq)])
    V_rep = np.stack([V[i // rep] for i in range(hq)])
    mha = L.gqa_attention(q, K_rep, V_rep)
    assert np.array_equal(L.gqa_attention(q, K, V), mha)
    # contiguous grouping: head 3 uses kv head 0, head 4 uses kv head 1
    assert np.allclose(mha[3], L.attention_head(q[3], K[0], V[0]))
    assert np.allclose(mha[4], L.attention_head(q[4], K[1], V[1]))


# ------------------------------------------------------------------ SwiGLU / argmax
def test_silu_special_values_and_scipy():
    assert L.silu(0.0) == 0.0
    assert L.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    assert abs(L.silu(-40.0)) < 1e-15
    x = rng.standard_normal(100) * 4
    assert np.allclose(L.silu(x), x * scipy.special.expit(x), rtol=1e-14)
    assert np.allclose(L.swiglu(x, x[::-1]), x * scipy.special.expit(x) * x[::-1], rtol=1e-14)


def test_argmax_lowest_index_on_ties():
    v = np.array([0.5, 2.0, -1.0, 2.0, 2.0])
    assert L.argmax_lowest(v) == 1 == int(np.argmax(v))
    assert L.argmax_lowest(np.array([-3.0, -3.0])) == 0
    with pytest.raises(ValueError):
        L.argmax_lowest(np.array([0.0, np.nan]))


# ------------------------------------------------------------------ bf16 storage rounding
def test_round_to_bf16_brute_force():
    # nearest bf16 value by brute force over neighbouring bit patterns, ties to even
    x = np.concatenate([rng.standard_normal(2000) * 0.05, [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8)]])
    got = L.round_to_bf16(x)
    for xi, gi in zip(x, got):
        f = np.float32(xi)
        hi = int(np.array([f]).view(np.uint32)[0]) >> 16
        cands = [(c << 16) for c in (hi - 1, hi, hi + 1)]
        vals = [float(np.array([c], np.uint32).view(np.float32)[0]) for c in cands]
        d = [abs(v - float(f)) for v in vals]
        best = min(d)
        winners = [c for c, dd in zip(cands, d) if dd == best]
        win = [c for c in winners if ((c >> 16) & 1) == 0] if len(winners) > 1 else winners
        assert gi == float(np.array([win[0]], np.uint32).view(np.float32)[0])


# ------------------------------------------------------------------ quantisers
def test_int8_quant_brute_force_rows():
    w = (rng.standard_normal((6, 96)) * 0.02).astype(np.float32)
    w[2] = 0.0
    w[3, 5] = 0.04 * 1.0          # a row with one large element
    q, s = Q.quantize_int8_rows(w)
    assert s.dtype == np.float16 and q.dtype == np.int8
    assert s[2] == 0 and not q[2].any()
    for r in range(6):
        if s[r] == 0:
            continue
        sr = np.float32(s[r])
        # scale: fp16 rounding of fp32(max|w| / 127)
        assert s[r] == np.float16(np.float32(np.abs(w[r]).max()) / np.float32(127))
        for k in range(96):
            cands = np.arange(-127, 128)
            err = np.abs(np.float32(w[r, k] / sr) - cands)
            best = cands[err == err.min()]
            want = best[best % 2 == 0][0] if len(best) > 1 else best[0]
            assert q[r, k] == want
        # error bound |w - q s| <= s/2 wherever no clamping happened
        deq = Q.dequant_int8(q[r:r + 1], s[r:r + 1])[0]
        unclamped = np.abs(w[r] / sr) <= 127
        assert np.all(np.abs(w[r] - deq)[unclamped] <= sr / 2 * (1 + 1e-6))


def test_int8_idempotent_on_grid():
    s = np.float16(0.00042)
    q0 = rng.integers(-127, 128, (3, 64)).astype(np.int8)
    q0[:, 0] = 127
    w = q0.astype(np.float32) * np.float32(s)
    q, s2 = Q.quantize_int8_rows(w)
    assert np.all(s2 == s) and np.array_equal(q, q0)


def test_int4_group_quant_and_packing():
    w = (rng.standard_normal((4, 256)) * 0.02).astype(np.float32)
    w[1, 128:] = 0.0
    q, s = Q.quantize_int4_g128(w)
    assert s.shape == (4, 2) and s[1, 1] == 0 and not q[1, 128:].any()
    assert q.min() >= -7 and q.max() <= 7
    for r in range(4):
        for g in range(2):
            blk = w[r, g * 128:(g + 1) * 128]
            assert s[r, g] == np.float16(np.float32(np.abs(blk).max()) / np.float32(7))
            if s[r, g] == 0:
                continue
            sr = np.float32(s[r, g])
            for k in range(128):
                cands = np.arange(-7, 8)
                err = np.abs(np.float32(blk[k] / sr) - cands)
                best = cands[err == err.min()]
                want = best[best % 2 == 0][0] if len(best) > 1 else best[0]
                assert q[r, g * 128 + k] == want
    packed = Q.pack_int4_nibbles(q)
    assert packed.shape == (4, 128)
    assert np.array_equal(Q.unpack_int4_nibbles(packed), q)


def test_int4_nibble_golden():
    lines = open(os.path.join(GOLD, "int4_nibbles.txt")).read().splitlines()
    qv = np.array([int(t) for t in lines[1].split()[1:]], np.int8)[None, :]
    bv = np.array([int(t, 16) for t in lines[2].split()[1:]], np.uint8)[None, :]
    assert np.array_equal(Q.pack_int4_nibbles(qv), bv)
    assert np.array_equal(Q.unpack_int4_nibbles(bv), qv)


def test_dequant_exact_in_fp32():
    q = rng.integers(-127, 128, (5, 32)).astype(np.int8)
    s = (rng.random(5) * 0.01).astype(np.float16)
    d = Q.dequant_int8(q, s)
    exact = q.astype(np.float64) * s.astype(np.float64)[:, None]
    assert np.array_equal(d.astype(np.float64), exact)


# ----------------------------------------------------------------- FP8 E4M3
def test_e4m3_golden_values():
    import os
    from oracle import quant as Q
    v = Q.e4m3_values()
    path = os.path.join(os.path.dirname(__file__), "golden", "e4m3_values.txt")
    for ln in open(path):
        if ln.startswith("#") or not ln.strip():
            continue
        code, want = ln.split()
        got = v[int(code, 16)]
        if want == "nan":
            assert np.isnan(got)
        else:
            assert got == float(want) and np.signbit(got) == want.startswith("-"), (code, got, want)
    assert np.sum(np.isnan(v)) == 2 and np.nanmax(v) == 448.0


def test_e4m3_rounding_brute_force():
    """Every value rounds to the nearest finite E4M3 value, ties to the even
    code, magnitudes above 448 to 448 (brute force over the whole table)."""
    from oracle import quant as Q
    v = Q.e4m3_values()
    finite = [c for c in range(256) if not np.isnan(v[c])]
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(4000) * 40, rng.standard_normal(2000) * 0.01,
                        (v[finite] + np.roll(v[finite], 1)) / 2,  # midpoints: the ties
                        np.array([500.0, -1000.0, 2.0 ** -10, 3 * 2.0 ** -11])]).astype(np.float32)
    codes = Q.f32_to_e4m3(x)
    for xi, c in zip(x.astype(np.float64), codes):
        a = min(abs(xi), 448.0) * (1 if xi >= 0 else -1)
        d = np.array([abs(v[f] - a) for f in finite])
        best = np.flatnonzero(d == d.min())
        cands = [finite[i] for i in best]
        if len(cands) > 1:  # a tie: the even code (the zeros count as one value)
            cands = [f for f in cands if f % 2 == 0 and not (f == 0x80)] or cands
        assert int(c) in cands or (v[int(c)] == 0 and all(v[f] == 0 for f in cands)), (xi, hex(c), cands)


def test_fp8_quantiser_properties():
    from oracle import quant as Q
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((6, 256)) * 0.02).astype(np.float32)
    w[2, 128:] = 0.0  # an all-zero group: scale 0, codes 0
    codes, s = Q.quantize_fp8_g128(w)
    deq = Q.dequant_fp8(codes, s)
    assert s[2, 1] == 0 and not codes[2, 128:].any()
    # the dequantised value is exact in fp32 and within half a code spacing of w
    v = Q.e4m3_values()
    for r in range(6):
        for g in range(2):
            sc = float(s[r, g])
            if sc == 0:
                continue
            x = w[r, 128 * g:128 * g + 128].astype(np.float64) / sc
            q = v[codes[r, 128 * g:128 * g + 128]]
            spacing = np.maximum(2.0 ** (np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -6))) - 3), 2.0 ** -9)
            assert np.all(np.abs(x - q) <= spacing / 2 + 1e-12)
    # idempotent on grid values
    c2, s2 = Q.quantize_fp8_g128(deq)
    assert np.array_equal(c2, codes) and np.array_equal(s2, s)
