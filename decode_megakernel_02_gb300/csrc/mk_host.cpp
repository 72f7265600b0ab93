// Host side of the library that needs no GPU: contract checks, the packed
// weight layout, the packer and the weight-only quantisers.
//
// Packing follows the "GEMV-friendly tiles" the decode path streams: each
// GEMV is a set of contiguous rows, read once per token by exactly one CTA
// (AutoMegaKernel explainer, "Problem definition": the floor is
// weight_bytes / HBM bandwidth, so every weight byte is read once).
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "mk_host.h"

namespace mk {

static thread_local std::string g_err;

void set_error(const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
}
const char* thread_error() { return g_err.c_str(); }

// ------------------------------------------------------------------ fp16 <-> fp32
// IEEE-754 binary16 conversion, round to nearest even (written from the format
// definition: 1 sign, 5 exponent (bias 15), 10 fraction bits).
uint16_t f32_to_f16_rne(float f) {
    uint32_t x;
    std::memcpy(&x, &f, 4);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ax = x & 0x7FFFFFFFu;
    if (ax > 0x7F800000u) return sign | 0x7E00u;  // NaN
    if (ax == 0x7F800000u) return sign | 0x7C00u; // Inf
    int e = (int)(ax >> 23) - 127;
    uint32_t m = ax & 0x7FFFFFu;
    if (e > 15) return sign | 0x7C00u;
    if (e >= -14) {
        uint32_t mant = m >> 13, rem = m & 0x1FFFu;
        uint32_t h = ((uint32_t)(e + 15) << 10) | mant;
        if (rem > 0x1000u || (rem == 0x1000u && (mant & 1u))) h += 1;  // may carry into exp/Inf
        return sign | (uint16_t)h;
    }
    if (ax < 0x00800000u) return sign;            // fp32 subnormal: far below fp16 range
    uint32_t m24 = m | 0x800000u;                 // value = m24 * 2^(e-23); unit 2^-24
    int s = -(e + 1);                             // bits dropped (>= 14)
    if (s > 24) return sign;
    uint32_t q = m24 >> s, r = m24 & ((1u << s) - 1u), half = 1u << (s - 1);
    if (r > half || (r == half && (q & 1u))) q += 1;
    return sign | (uint16_t)q;
}

float f16_to_f32(uint16_t h) {
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1Fu, m = h & 0x3FFu, x;
    if (e == 0) {
        if (m == 0) {
            x = sign;
        } else {  // subnormal: m * 2^-24
            float v = (float)m * 5.9604644775390625e-08f;
            std::memcpy(&x, &v, 4);
            x |= sign;
        }
    } else if (e == 31) {
        x = sign | 0x7F800000u | (m << 13);
    } else {
        x = sign | ((e - 15 + 127) << 23) | (m << 13);
    }
    float f;
    std::memcpy(&f, &x, 4);
    return f;
}

static inline float bf16_to_f32(uint16_t b) {
    uint32_t x = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &x, 4);
    return f;
}

float base_to_f32(uint16_t v, int base) { return base == MK_W_FP16 ? f16_to_f32(v) : bf16_to_f32(v); }

// ------------------------------------------------------------------ quantisers
// W8A16 per output row: s = fp16(fp32(max|w|) / 127), q = clamp(rne(w / s), +-127).
void quant_row_int8(const float* w, int64_t k, int8_t* q, uint16_t* s16) {
    float amax = 0.f;
    for (int64_t i = 0; i < k; ++i) amax = std::max(amax, std::fabs(w[i]));
    uint16_t sh = f32_to_f16_rne(amax / 127.0f);
    float s = f16_to_f32(sh);
    *s16 = sh;
    for (int64_t i = 0; i < k; ++i) {
        if (s == 0.f) {
            q[i] = 0;
            continue;
        }
        float r = std::nearbyint(w[i] / s);  // default rounding mode: half to even
        r = std::min(127.f, std::max(-127.f, r));
        q[i] = (int8_t)r;
    }
}

// W4A16 with one scale per 128 consecutive k: s = fp16(fp32(max|w|) / 7).
void quant_row_int4(const float* w, int64_t k, int8_t* q, uint16_t* s16) {
    for (int64_t g = 0; g < k / 128; ++g) {
        const float* wg = w + g * 128;
        float amax = 0.f;
        for (int i = 0; i < 128; ++i) amax = std::max(amax, std::fabs(wg[i]));
        uint16_t sh = f32_to_f16_rne(amax / 7.0f);
        float s = f16_to_f32(sh);
        s16[g] = sh;
        for (int i = 0; i < 128; ++i) {
            if (s == 0.f) {
                q[g * 128 + i] = 0;
                continue;
            }
            float r = std::nearbyint(wg[i] / s);
            r = std::min(7.f, std::max(-7.f, r));
            q[g * 128 + i] = (int8_t)r;
        }
    }
}

// FP8 E4M3 (OCP 8-bit floating point: 1 sign, 4 exponent bits with bias 7, 3
// mantissa bits; exponent 0 holds the subnormals m * 2^-9; S.1111.111 is NaN;
// 448 is the largest magnitude), rounded to nearest, ties to even, clamped to
// 448.  Codes ascend with the value, so the code is the rounded mantissa step
// count on the 2^-9 grid (subnormals) or (e + 7) * 8 + round(a * 2^(3 - e)) - 8
// for a in [2^e, 2^(e+1)): a carry past 8 lands on the next exponent's code.
uint8_t f32_to_e4m3_rne(float f) {
    uint32_t x;
    std::memcpy(&x, &f, 4);
    const uint8_t sign = (uint8_t)((x >> 24) & 0x80u);
    const float a = std::fabs(f);
    if (a >= 448.f) return sign | 0x7Eu;
    int code;
    if (a < 0.015625f) {  // below 2^-6: the subnormal grid
        code = (int)std::nearbyint(a * 512.f);
    } else {
        int e;
        std::frexp(a, &e);  // a = m * 2^e with m in [0.5, 1)
        e -= 1;             // a in [2^e, 2^(e+1))
        code = (e + 7) * 8 + (int)std::nearbyint(std::ldexp(a, 3 - e)) - 8;
    }
    if (code > 0x7E) code = 0x7E;
    return code == 0 ? 0 : (uint8_t)(sign | code);
}

// FP8 E4M3 with one scale per 128 consecutive k: s = fp16(fp32(max|w|) / 448).
void quant_row_fp8(const float* w, int64_t k, uint8_t* q, uint16_t* s16) {
    for (int64_t g = 0; g < k / 128; ++g) {
        const float* wg = w + g * 128;
        float amax = 0.f;
        for (int i = 0; i < 128; ++i) amax = std::max(amax, std::fabs(wg[i]));
        const uint16_t sh = f32_to_f16_rne(amax / 448.0f);
        const float s = f16_to_f32(sh);
        s16[g] = sh;
        for (int i = 0; i < 128; ++i) q[g * 128 + i] = s == 0.f ? 0 : f32_to_e4m3_rne(wg[i] / s);
    }
}

// ------------------------------------------------------------------ contract
static bool pow2_le(int v, int hi) { return v >= 1 && v <= hi; }

mk_status check_desc(const mk_model_desc* d) {
    if (!d) {
        set_error("desc is NULL");
        return MK_ERR_INVALID_ARG;
    }
    if (d->flags & (MK_FLAG_PROJ_BIAS | MK_FLAG_TIED_HEAD | MK_FLAG_ROPE_SCALING)) {
        set_error("unsupported model variant flags 0x%x (biased projections, tied head or rope "
                  "scaling are outside the contract)", d->flags);
        return MK_ERR_UNSUPPORTED;
    }
    if (d->n_layers < 1 || d->d_model < 1 || d->n_q_heads < 1 || d->n_kv_heads < 1 ||
        d->d_ffn < 1 || d->vocab < 1 || d->max_seq < 1 || !(d->rms_eps > 0.f) ||
        !(d->rope_theta > 1.f)) {
        set_error("non-positive dimension, eps or theta");
        return MK_ERR_INVALID_ARG;
    }
    if (d->head_dim != 64 && d->head_dim != 128) {
        set_error("head_dim %d: only 64 and 128 are supported", d->head_dim);
        return MK_ERR_UNSUPPORTED;
    }
    if (d->n_q_heads % d->n_kv_heads || !pow2_le(d->n_q_heads / d->n_kv_heads, MAX_REP)) {
        set_error("n_q_heads %d / n_kv_heads %d: need an integer group of at most %d",
                  d->n_q_heads, d->n_kv_heads, MAX_REP);
        return MK_ERR_UNSUPPORTED;
    }
    int qd = d->n_q_heads * d->head_dim;
    if (d->d_model % 128 || d->d_ffn % 128 || qd % 128) {
        set_error("d_model %d, d_ffn %d and q_dim %d must be multiples of 128", d->d_model,
                  d->d_ffn, qd);
        return MK_ERR_UNSUPPORTED;
    }
    if (d->d_model > MAX_K || d->d_ffn > MAX_K || qd > MAX_K) {
        set_error("a GEMV reduction length exceeds %d", MAX_K);
        return MK_ERR_UNSUPPORTED;
    }
    if (d->wdtype == MK_W_INT4_G128) {  // the rows a GEMV task streams: d_model, q_dim, and d_ffn when the FFN is not fused
        const int kmax = std::max(std::max(d->d_model, qd),
                                  ffn_fused(d->wdtype, d->base_dtype, d->d_model) ? 0 : d->d_ffn);
        if (kmax > INT4_MAX_ROW_K) {
            set_error("int4 rows of %d codes: at most %d are supported", kmax, INT4_MAX_ROW_K);
            return MK_ERR_UNSUPPORTED;
        }
    }
    if (d->vocab >= (1 << KEY_IDX_BITS)) {
        set_error("vocab %d >= %d", d->vocab, 1 << KEY_IDX_BITS);
        return MK_ERR_UNSUPPORTED;
    }
    if (d->base_dtype != MK_W_BF16 && d->base_dtype != MK_W_FP16) {
        set_error("base_dtype %d must be MK_W_BF16 or MK_W_FP16", d->base_dtype);
        return MK_ERR_UNSUPPORTED;
    }
    const bool quant = d->wdtype == MK_W_INT8_ROW || d->wdtype == MK_W_INT4_G128 || d->wdtype == MK_W_FP8_E4M3;
    if (d->wdtype != d->base_dtype && !quant) {
        set_error("wdtype %d must equal base_dtype or be a quantised type", d->wdtype);
        return MK_ERR_UNSUPPORTED;
    }
    if (quant && d->base_dtype != MK_W_BF16) {
        set_error("quantised weights are packed from bf16 sources only");
        return MK_ERR_UNSUPPORTED;
    }
    return MK_OK;
}

// ------------------------------------------------------------------ layout
static int64_t up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

int64_t row_stride(int64_t K, int wdtype) {
    switch (wdtype) {
        case MK_W_INT8_ROW: return up(K + 2, 16);                 // codes + fp16 scale
        case MK_W_INT4_G128: return up(K / 2 + 2 * (K / 128), 16); // nibbles + fp16 scales
        case MK_W_FP8_E4M3: return up(K + 2 * (K / 128), 16);      // E4M3 codes + fp16 scales
        default: return up(2 * K, 16);
    }
}

BlobLayout blob_layout(const mk_model_desc* d) {
    BlobLayout b{};
    int64_t qd = (int64_t)d->n_q_heads * d->head_dim, kd = (int64_t)d->n_kv_heads * d->head_dim;
    b.down_cols = ffn_fused(d->wdtype, d->base_dtype, d->d_model);
    b.row_qkv = row_stride(d->d_model, d->wdtype);
    b.row_o = row_stride(qd, d->wdtype);
    b.row_gu = row_stride(d->d_model, d->wdtype);
    b.row_down = row_stride(d->d_ffn, d->wdtype);
    b.row_lm = row_stride(d->d_model, d->wdtype);
    b.norm_bytes = up(2 * (int64_t)d->d_model, 256);
    int64_t o = 0;
    b.l_attn_norm = o; o += b.norm_bytes;
    b.l_ffn_norm = o; o += b.norm_bytes;
    b.l_qkv = o; o = up(o + (qd + 2 * kd) * b.row_qkv, 256);
    b.l_o = o; o = up(o + (int64_t)d->d_model * b.row_o, 256);
    b.l_gu = o; o = up(o + 2 * (int64_t)d->d_ffn * b.row_gu, 256);
    b.l_down = o; o = up(o + (int64_t)d->d_model * b.row_down, 256);
    b.layer_bytes = o;
    int64_t g = b.layer_bytes * d->n_layers;
    b.final_norm = g; g += b.norm_bytes;
    b.lm = g; g = up(g + (int64_t)d->vocab * b.row_lm, 256);
    b.embed = g; g = up(g + (int64_t)d->vocab * d->d_model * 2, 256);
    b.total = g;
    return b;
}

// Placement of a tensor: region offset, stride, first row and row step inside
// the region (gate/up are interleaved row by row), rows, cols.
struct Place {
    int64_t off, stride;
    int32_t first, step, rows, cols;
    bool gemv;
};

static bool place(const mk_model_desc* d, int tensor, int layer, Place* p) {
    BlobLayout b = blob_layout(d);
    int32_t qd = d->n_q_heads * d->head_dim, kd = d->n_kv_heads * d->head_dim;
    bool per_layer = tensor >= MK_T_ATTN_NORM && tensor != MK_T_EMBED && tensor != MK_T_LM_HEAD &&
                     tensor != MK_T_FINAL_NORM;
    if (per_layer && (layer < 0 || layer >= d->n_layers)) return false;
    int64_t lb = per_layer ? b.layer_bytes * layer : 0;
    *p = Place{0, 0, 0, 1, 0, 0, true};
    switch (tensor) {
        case MK_T_EMBED: *p = {b.embed, 2 * (int64_t)d->d_model, 0, 1, d->vocab, d->d_model, false}; break;
        case MK_T_LM_HEAD: *p = {b.lm, b.row_lm, 0, 1, d->vocab, d->d_model, true}; break;
        case MK_T_FINAL_NORM: *p = {b.final_norm, 0, 0, 1, 1, d->d_model, false}; break;
        case MK_T_ATTN_NORM: *p = {lb + b.l_attn_norm, 0, 0, 1, 1, d->d_model, false}; break;
        case MK_T_FFN_NORM: *p = {lb + b.l_ffn_norm, 0, 0, 1, 1, d->d_model, false}; break;
        case MK_T_WQ: *p = {lb + b.l_qkv, b.row_qkv, 0, 1, qd, d->d_model, true}; break;
        case MK_T_WK: *p = {lb + b.l_qkv, b.row_qkv, qd, 1, kd, d->d_model, true}; break;
        case MK_T_WV: *p = {lb + b.l_qkv, b.row_qkv, qd + kd, 1, kd, d->d_model, true}; break;
        case MK_T_WO: *p = {lb + b.l_o, b.row_o, 0, 1, d->d_model, qd, true}; break;
        case MK_T_WGATE: *p = {lb + b.l_gu, b.row_gu, 0, 2, d->d_ffn, d->d_model, true}; break;
        case MK_T_WUP: *p = {lb + b.l_gu, b.row_gu, 1, 2, d->d_ffn, d->d_model, true}; break;
        case MK_T_WDOWN: *p = {lb + b.l_down, b.down_cols ? 0 : b.row_down, 0, 1, d->d_model, d->d_ffn, true}; break;
        default: return false;
    }
    return true;
}

}  // namespace mk

using namespace mk;

extern "C" {

mk_status mk_packed_size(const mk_model_desc* desc, size_t* bytes) {
    mk_status st = check_desc(desc);
    if (st) return st;
    if (!bytes) {
        set_error("bytes is NULL");
        return MK_ERR_INVALID_ARG;
    }
    *bytes = (size_t)blob_layout(desc).total;
    return MK_OK;
}

mk_status mk_tensor_layout(const mk_model_desc* desc, int32_t tensor, int32_t layer, size_t* offset,
                           size_t* stride, int32_t* first_row, int32_t* row_step, int32_t* rows) {
    mk_status st = check_desc(desc);
    if (st) return st;
    Place p;
    if (!place(desc, tensor, layer, &p)) {
        set_error("bad tensor id %d or layer %d", tensor, layer);
        return MK_ERR_INVALID_ARG;
    }
    if (offset) *offset = (size_t)p.off;
    if (stride) *stride = (size_t)p.stride;
    if (first_row) *first_row = p.first;
    if (row_step) *row_step = p.step;
    if (rows) *rows = p.rows;
    return MK_OK;
}

mk_status mk_pack_tensor(const mk_model_desc* desc, int32_t tensor, int32_t layer,
                         const void* src_host, void* blob_host, size_t blob_bytes) {
    mk_status st = check_desc(desc);
    if (st) return st;
    if (!src_host || !blob_host) {
        set_error("NULL source or blob");
        return MK_ERR_INVALID_ARG;
    }
    BlobLayout b = blob_layout(desc);
    if (blob_bytes < (size_t)b.total) {
        set_error("blob has %zu bytes, layout needs %lld", blob_bytes, (long long)b.total);
        return MK_ERR_INVALID_ARG;
    }
    Place p;
    if (!place(desc, tensor, layer, &p)) {
        set_error("bad tensor id %d or layer %d", tensor, layer);
        return MK_ERR_INVALID_ARG;
    }
    const uint16_t* src = (const uint16_t*)src_host;
    uint8_t* blob = (uint8_t*)blob_host;
    if (!p.gemv) {  // embedding and norm gains: stored as given
        std::memcpy(blob + p.off, src, (size_t)p.rows * p.cols * 2);
        return MK_OK;
    }
    const int64_t K = p.cols;
    std::vector<float> wf;
    std::vector<int8_t> q;
    std::vector<uint16_t> s16;
    for (int32_t r = 0; r < p.rows; ++r) {
        uint8_t* dst = blob + p.off + (int64_t)(p.first + (int64_t)r * p.step) * p.stride;
        const uint16_t* row = src + (int64_t)r * K;
        if (p.stride == 0 && desc->wdtype == desc->base_dtype) {
            // W_down in column blocks: row r of block c at (c * rows + r) * 16 bytes
            for (int64_t c = 0; c < K / 8; ++c) std::memcpy(blob + p.off + (c * p.rows + r) * 16, row + c * 8, 16);
            continue;
        }
        if (p.stride) std::memset(dst, 0, (size_t)p.stride);
        if (desc->wdtype == desc->base_dtype) {
            std::memcpy(dst, row, (size_t)K * 2);
            continue;
        }
        wf.resize(K);
        q.resize(K);
        for (int64_t k = 0; k < K; ++k) wf[k] = base_to_f32(row[k], desc->base_dtype);
        if (p.stride == 0) {
            // Quantised W_down in column blocks of 16 bytes: block c holds the
            // codes of units [c * BU, (c + 1) * BU) of every row r at
            // (c * rows + r) * 16; after the blocks come the fp16 scales, per
            // row (int8, [rows]) or per 128-unit group ([K / 128][rows]).
            const int64_t BU = ffn_block(desc->wdtype), rows = p.rows;
            uint8_t* codes = blob + p.off;
            uint16_t* scales = (uint16_t*)(blob + p.off + rows * K * 16 / BU);
            if (desc->wdtype == MK_W_INT8_ROW) {
                uint16_t sc;
                quant_row_int8(wf.data(), K, q.data(), &sc);
                for (int64_t c = 0; c < K / BU; ++c) std::memcpy(codes + (c * rows + r) * 16, q.data() + c * BU, 16);
                std::memcpy(scales + r, &sc, 2);
            } else if (desc->wdtype == MK_W_FP8_E4M3) {
                s16.resize(K / 128);
                quant_row_fp8(wf.data(), K, (uint8_t*)q.data(), s16.data());
                for (int64_t c = 0; c < K / BU; ++c) std::memcpy(codes + (c * rows + r) * 16, q.data() + c * BU, 16);
                for (int64_t g = 0; g < K / 128; ++g) std::memcpy(scales + g * rows + r, &s16[g], 2);
            } else {
                s16.resize(K / 128);
                quant_row_int4(wf.data(), K, q.data(), s16.data());
                for (int64_t c = 0; c < K / BU; ++c)
                    for (int64_t k = 0; k < BU; k += 2)
                        codes[(c * rows + r) * 16 + k / 2] = (uint8_t)(((uint8_t)q[c * BU + k] & 0xF) |
                                                                       (((uint8_t)q[c * BU + k + 1] & 0xF) << 4));
                for (int64_t g = 0; g < K / 128; ++g) std::memcpy(scales + g * rows + r, &s16[g], 2);
            }
            continue;
        }
        if (desc->wdtype == MK_W_INT8_ROW) {
            uint16_t s;
            quant_row_int8(wf.data(), K, q.data(), &s);
            std::memcpy(dst, q.data(), (size_t)K);
            std::memcpy(dst + K, &s, 2);
        } else if (desc->wdtype == MK_W_FP8_E4M3) {
            s16.resize(K / 128);
            quant_row_fp8(wf.data(), K, (uint8_t*)q.data(), s16.data());
            std::memcpy(dst, q.data(), (size_t)K);
            std::memcpy(dst + K, s16.data(), s16.size() * 2);
        } else {
            s16.resize(K / 128);
            quant_row_int4(wf.data(), K, q.data(), s16.data());
            for (int64_t k = 0; k < K; k += 2)
                dst[k / 2] = (uint8_t)(((uint8_t)q[k] & 0xF) | (((uint8_t)q[k + 1] & 0xF) << 4));
            std::memcpy(dst + K / 2, s16.data(), s16.size() * 2);
        }
    }
    return MK_OK;
}

mk_status mk_quantize_int8(const float* w, int64_t n, int64_t k, int8_t* q, uint16_t* s16) {
    if (!w || !q || !s16 || n < 0 || k < 1) {
        set_error("bad quantiser arguments");
        return MK_ERR_INVALID_ARG;
    }
    for (int64_t r = 0; r < n; ++r) quant_row_int8(w + r * k, k, q + r * k, s16 + r);
    return MK_OK;
}

mk_status mk_quantize_int4(const float* w, int64_t n, int64_t k, int8_t* q, uint16_t* s16) {
    if (!w || !q || !s16 || n < 0 || k < 128 || k % 128) {
        set_error("bad quantiser arguments (k must be a positive multiple of 128)");
        return MK_ERR_INVALID_ARG;
    }
    for (int64_t r = 0; r < n; ++r) quant_row_int4(w + r * k, k, q + r * k, s16 + r * (k / 128));
    return MK_OK;
}

mk_status mk_quantize_fp8(const float* w, int64_t n, int64_t k, uint8_t* q, uint16_t* s16) {
    if (!w || !q || !s16 || n < 0 || k < 128 || k % 128) {
        set_error("bad quantiser arguments (k must be a positive multiple of 128)");
        return MK_ERR_INVALID_ARG;
    }
    for (int64_t r = 0; r < n; ++r) quant_row_fp8(w + r * k, k, q + r * k, s16 + r * (k / 128));
    return MK_OK;
}

mk_status mk_kv_cache_size(const mk_model_desc* desc, size_t* bytes) {
    mk_status st = check_desc(desc);
    if (st) return st;
    if (!bytes) {
        set_error("bytes is NULL");
        return MK_ERR_INVALID_ARG;
    }
    *bytes = (size_t)desc->n_layers * 2 * desc->n_kv_heads * desc->max_seq * desc->head_dim * 2;
    return MK_OK;
}

}  // extern "C"
