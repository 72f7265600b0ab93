"""Weight-only quantisation (W8A16 per-row, W4A16 group-128) and dequantisation.

The AutoMegaKernel explainer ("Key contributions": int8 weight-only kernels
that are greedy-lossless, int4 kernels that cut weight traffic 2.42x and are
lossy) fixes only "symmetric, per output channel, fp16 scale = max|w|/127"
for int8 and "symmetric group-128, fp16 scales" for int4.  Readings taken for
what is left open:

* int8: s = fp16(fp32(max_k |w_rk|) / 127) with both roundings to nearest
  even; q = clamp(round_half_even(fp32(w) / fp32(s)), -127, 127); s == 0 gives
  q == 0.
* int4: groups of 128 consecutive k per row; s = fp16(fp32(max|w|) / 7);
  q = clamp(round_half_even(w / s), -7, 7); stored as two's-complement
  nibbles, the even k in the low nibble.
* Dequantisation is w' = fp32(q) * fp32(s), which is exact in float32
  (at most 4 + 11 significant bits), so it is checked bit for bit.
"""
import numpy as np


def _fp16_of_fp32(x):
    return np.asarray(x, np.float32).astype(np.float16)


def _round_half_even_div(w32, s32):
    """round_half_even(fp32(w / s)) with an fp32 division."""
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (w32 / s32).astype(np.float32)
    return np.rint(r)          # numpy rint rounds half to even


def quantize_int8_rows(w):
    """w: float32 [N, K] (bf16-exact values).  Returns (q int8 [N,K], s float16 [N])."""
    w = np.asarray(w, np.float32)
    amax = np.max(np.abs(w), axis=1)
    s16 = _fp16_of_fp32(amax / np.float32(127.0))
    s32 = s16.astype(np.float32)[:, None]
    q = np.zeros(w.shape, np.int8)
    nz = s32[:, 0] != 0
    r = _round_half_even_div(w[nz], s32[nz])
    q[nz] = np.clip(r, -127, 127).astype(np.int8)
    return q, s16


def quantize_int4_g128(w, group=128):
    """w: float32 [N, K], K % 128 == 0.  Returns (q int8 [N,K] in [-7,7], s float16 [N, K/128])."""
    w = np.asarray(w, np.float32)
    n, k = w.shape
    assert k % group == 0
    g = w.reshape(n, k // group, group)
    amax = np.max(np.abs(g), axis=2)
    s16 = _fp16_of_fp32(amax / np.float32(7.0))
    s32 = s16.astype(np.float32)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = _round_half_even_div(g, s32)
    r = np.where(s32 == 0, 0.0, r)
    q = np.clip(r, -7, 7).astype(np.int8).reshape(n, k)
    return q, s16


def pack_int4_nibbles(q):
    """q int8 [N, K] in [-8, 7] -> uint8 [N, K/2]; even k in the low nibble."""
    u = (np.asarray(q).astype(np.int16) & 0xF).astype(np.uint8)
    return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def unpack_int4_nibbles(b):
    """Inverse of pack_int4_nibbles (sign-extends each nibble)."""
    b = np.asarray(b, np.uint8)
    lo = (b & 0xF).astype(np.int8)
    hi = (b >> 4).astype(np.int8)
    lo = np.where(lo >= 8, lo - 16, lo).astype(np.int8)
    hi = np.where(hi >= 8, hi - 16, hi).astype(np.int8)
    out = np.empty((b.shape[0], b.shape[1] * 2), np.int8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


def dequant_int8(q, s16):
    """w' = fp32(q) * fp32(s), float32 [N, K]."""
    return (np.asarray(q).astype(np.float32) * s16.astype(np.float32)[:, None]).astype(np.float32)


def dequant_int4(q, s16, group=128):
    n, k = q.shape
    s = np.repeat(s16.astype(np.float32), group, axis=1)
    return (np.asarray(q).astype(np.float32) * s).astype(np.float32)


# ----------------------------------------------------------------- FP8 E4M3, block-scaled
# The Netra Kernel summary ("TL;DR": FP8 serving ops) names FP8; the pages fix
# no format details for weights.  Readings: the OCP FP8
# E4M3 format (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0
# holds the subnormals m * 2^-9; S.1111.111 is NaN and there is no infinity, so
# the largest finite magnitude is 1.75 * 2^8 = 448), one fp16 scale per 128
# consecutive k of a row (as for int4): s = fp16(fp32(max|w|) / 448), codes =
# E4M3 nearest to fp32(w) / fp32(s), ties to the even code, s == 0 -> 0.

def e4m3_values():
    """float64 value of each of the 256 codes (NaN for the two NaN codes)."""
    v = np.empty(256)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 7
        if e == 15 and m == 7:
            v[c] = np.nan
        elif e == 0:
            v[c] = sign * m * 2.0 ** -9
        else:
            v[c] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return v


def f32_to_e4m3(x):
    """Round float32 values to the nearest E4M3 code (ties to the even code),
    clamping magnitudes to 448; returns uint8 codes."""
    x = np.asarray(x, np.float32).astype(np.float64)
    vals = e4m3_values()[:0x7F]              # the 127 non-negative finite codes, ascending
    a = np.minimum(np.abs(x), 448.0)
    hi = np.searchsorted(vals, a, side="left").clip(0, len(vals) - 1)
    lo = (hi - 1).clip(0, len(vals) - 1)
    dlo, dhi = a - vals[lo], vals[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(a == vals[lo], lo, code).astype(np.uint8)
    return np.where(np.signbit(x) & (code != 0), code | 0x80, code).astype(np.uint8)


def quantize_fp8_g128(w, group=128):
    """w: float32 [N, K], K % 128 == 0.  Returns (codes uint8 [N, K], s float16 [N, K/128])."""
    w = np.asarray(w, np.float32)
    n, k = w.shape
    assert k % group == 0
    g = w.reshape(n, k // group, group)
    amax = np.max(np.abs(g), axis=2)
    s16 = _fp16_of_fp32(amax / np.float32(448.0))
    s32 = s16.astype(np.float32)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (g / s32).astype(np.float32)
    r = np.where(s32 == 0, np.float32(0), r)
    return f32_to_e4m3(r).reshape(n, k), s16


def dequant_fp8(codes, s16, group=128):
    """w' = fp32(e4m3(code)) * fp32(s): exact in float32 (4 + 11 significant bits)."""
    v = e4m3_values()[np.asarray(codes, np.uint8)].astype(np.float32)
    s = np.repeat(s16.astype(np.float32), group, axis=1)
    return (v * s).astype(np.float32)


GEMV_TENSORS = ("wq", "wk", "wv", "wo", "wgate", "wup", "wdown")


def quantised_model_weights(shape, weights, wdtype, base_dtype="bf16"):
    """Dequantised float64 copies of every GEMV weight (LM head included).

    The embedding and the norm gains stay in their storage type.  Returns a
    dict usable as ``llama.Model(..., dequantised=...)`` plus the raw
    quantised (q, s) pairs for byte comparisons."""
    from .llama import bf16_bits_to_f64, fp16_bits_to_f64
    widen = bf16_bits_to_f64 if base_dtype == "bf16" else fp16_bits_to_f64
    names = [f"l{i}.{t}" for i in range(shape.n_layers) for t in GEMV_TENSORS] + ["lm_head"]
    deq, raw = {}, {}
    for nm in names:
        w32 = widen(weights[nm]).astype(np.float32)
        if wdtype == "int8":
            q, s = quantize_int8_rows(w32)
            deq[nm] = dequant_int8(q, s).astype(np.float64)
        elif wdtype == "int4":
            q, s = quantize_int4_g128(w32)
            deq[nm] = dequant_int4(q, s).astype(np.float64)
        elif wdtype == "fp8":
            q, s = quantize_fp8_g128(w32)
            deq[nm] = dequant_fp8(q, s).astype(np.float64)
        else:
            raise ValueError(wdtype)
        raw[nm] = (q, s)
    return deq, raw
