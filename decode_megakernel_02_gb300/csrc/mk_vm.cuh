// The persistent decode kernel ("VM") for sm_103a.
//
// AutoMegaKernel explainer, "Methodology", Layer 0: one cooperative
// threadblock per SM, each owning a local queue that it walks in global
// topological order with wait -> dispatch -> signal, synchronised by
// monotonic counters instead of locks.  Kog monokernel tutorial: the whole
// decode loop (LM head and token selection included) stays resident, the
// host never re-enters per token, and batch-1 projections are GEMVs on the
// vector ALUs, not matrix-core GEMMs.
//
// GB300 design (differs from the pages' kernels):
//  * Weight streaming is split from compute.  Weight bytes never depend on
//    activations, so one producer warp per CTA walks the CTA's whole queue
//    ahead of the consumers and keeps a ring of shared-memory slots filled
//    with 1-D bulk TMA copies (cp.async.bulk + mbarrier complete_tx), across
//    counter waits and across steps.  HBM keeps streaming while consumers
//    wait on a dependency; the ring depth is the pipelining depth.
//  * Eight consumer warps own the arithmetic: each thread owns fixed 8-wide
//    k-groups of the input vector in registers (fp32), reads 16/8/4-byte
//    weight groups from shared memory (conflict-free), accumulates in fp32
//    and reduces each slot's rows with a transposed warp reduction.
//  * Counters are u32 words on their own 128-byte lines; a wait is an
//    ld.acquire.gpu spin with a %globaltimer watchdog; a signal is a
//    __threadfence + red.release.gpu.add.  Thresholds scale with the global
//    step (epoch), so counters never need a reset between steps or launches.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mk_internal.h"

// Device code of the decode kernel, included by one translation unit per
// weight type (each instantiates vm_kernel for head_dim 64 and 128).
#pragma once

namespace mk {

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// The same test, but a thread whose phase is not complete is suspended for up
// to `ns` nanoseconds (woken early when the phase completes) instead of
// returning at once: spinning waiters then issue almost nothing.
__device__ __forceinline__ bool mbar_wait_hint(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
constexpr uint32_t SUSPEND_NS = 20000;
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
        "%2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}
// Fire-and-forget prefetch of [src, src + bytes) from HBM into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_volatile(const uint32_t* p) {
    return *(const volatile uint32_t*)p;
}
// Named barrier 1 among the NT consumer threads only (the producer warp never joins).
__device__ __forceinline__ void bar_consumers() { asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory"); }

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }
__device__ __forceinline__ float half_bits_to_f32(uint32_t b) {
    return __half2float(__ushort_as_half((unsigned short)b));
}
template <int BASE>
__device__ __forceinline__ float base_to_f32(uint32_t b) {
    return BASE == MK_W_FP16 ? half_bits_to_f32(b) : bf16_bits_to_f32(b);
}
__device__ __forceinline__ float round_bf16(float v) {
    return __bfloat162float(__float2bfloat16_rn(v));
}

// ------------------------------------------------------------------ dequantisation
// int8 code -> exact float: the byte (q + 128) is placed in the low mantissa
// bits of 2^23 and the bias 2^23 + 128 is subtracted (both steps exact).
__device__ __forceinline__ float i8_to_f32(uint32_t word_xor80, int k) {
    return __uint_as_float(__byte_perm(word_xor80, 0x4B000000u, 0x7540u + k)) - 8388736.0f;
}
// int4 code (two's-complement nibble n of a word XOR 0x88888888) -> exact float.
__device__ __forceinline__ float i4_to_f32(uint32_t word_xor88, int n) {
    return __uint_as_float(((word_xor88 >> (4 * n)) & 0xFu) | 0x4B000000u) - 8388616.0f;
}

// ------------------------------------------------------------------ shared memory
// Scratch of one attention task; its space is reused by the split-KV merge of
// the O prologue (a CTA never runs both at once).
struct AttnScratch {
    float q[MAX_REP * 128];         // roped, scaled queries of one KV group
    float kcur[128], vcur[128];     // this step's K and V (bf16-rounded)
    float sc[MAX_REP * ATTN_TILE];  // scores / probabilities of a tile
    uint16_t sv[ATTN_TILE * 128];   // V rows of the current tile (bf16)
};
struct MergeScratch {
    float mw[MAX_HC];               // per (head, chunk) max, then weight
    float ml[MAX_HC];               // per (head, chunk) sum
};

struct Shared {
    float norm[NW];                 // RMSNorm sum of squares
    float gpart[NW][2][8][NW];      // [group][parity][row][warp]: partial sums of shared rows
    unsigned long long keys[NW];    // per-warp LM argmax keys
    union {
        AttnScratch at;
        MergeScratch mg;
    };
    float m[MAX_REP], l[MAX_REP], alpha[MAX_REP];
    int32_t flag;                   // broadcast of a counter-wait result
    int32_t abort;                  // a warp gave up inside a task
    int32_t tok;                    // broadcast of the step's input token
    uint32_t consumed, issued;      // ring bookkeeping for the exit drain
    unsigned long long prod_wait_ns;   // trace: producer time waiting for free slots
    unsigned long long full_wait_ns;   // trace: consumer warp 0 time waiting for filled slots
    unsigned long long bars[2 * 16]; // full[16], empty[16]
};

struct Ctx {
    const VmParams* p;
    Shared* sh;
    uint8_t* ring;
    float* xs;          // the task's input vector (K floats)
    float rstd;         // scale of xs applied when the fragments are loaded (RMSNorm)
    int tid, lane, warp;
    uint32_t slot_seq;  // ring slots consumed so far (identical in every consumer warp)
    int slot_i;         // slot_seq % n_slots
    uint32_t slot_phase;  // (slot_seq / n_slots) & 1
    bool abort;
};

__device__ __forceinline__ uint32_t full_bar(Ctx& c, int i) { return smem_u32(&c.sh->bars[i]); }
__device__ __forceinline__ uint32_t empty_bar(Ctx& c, int i) { return smem_u32(&c.sh->bars[16 + i]); }

__device__ __forceinline__ bool aborted(const VmParams& p) { return ld_volatile(p.status) != 0; }

static __device__ void raise_error(const VmParams& p, uint32_t code, uint32_t task, uint32_t detail) {
    if (atomicCAS(p.status, 0u, code) == 0u) {
        p.status[1] = task;
        p.status[2] = detail;
    }
}

// Consumer wait on a counter: thread 0 spins, the rest learn the outcome at
// the named barrier.  An abort raised anywhere (another CTA, or one of this
// CTA's warps inside the previous task) stops every consumer warp here.
static __device__ __forceinline__ bool wait_counters(Ctx& c, const DevTask& t, int task_id, int step) {
    const VmParams& p = *c.p;
    if (c.tid == 0) {
        int ok = c.sh->abort ? 0 : 1;
        const uint32_t e = (uint32_t)(p.epoch0 + step);
        for (int w = 0; w < t.n_waits && ok; ++w) {
            const uint32_t* ctr = p.counters + (size_t)t.wait_ctr[w] * CTR_STRIDE;
            const uint32_t target = (uint32_t)t.wait_cnt[w] * (e + 1u + (uint32_t)t.wait_off[w]);
            if ((int32_t)(ld_acquire(ctr) - target) >= 0) continue;
            const uint64_t t0 = gtimer();
            for (uint32_t it = 1;; ++it) {
                if ((int32_t)(ld_acquire(ctr) - target) >= 0) break;
                if ((it & 63u) == 0u) {
                    if (aborted(p)) {
                        ok = 0;
                        break;
                    }
                    if (gtimer() - t0 > (uint64_t)p.watchdog_ns) {
                        raise_error(p, DEV_TIMEOUT, (uint32_t)task_id, (uint32_t)step);
                        ok = 0;
                        break;
                    }
                }
            }
        }
        c.sh->flag = ok;
    }
    bar_consumers();
    return c.sh->flag != 0;
}

// The consumer barrier orders every consumer thread's writes of the task
// before thread 0's release-add; a gpu-scope release is cumulative over
// writes that happen before it, so the waiting CTA's acquire sees them all.
__device__ __forceinline__ void signal_counter(Ctx& c, const DevTask& t) {
    bar_consumers();
    if (c.tid == 0 && t.signal_ctr >= 0 && !c.sh->abort)
        red_release_add(c.p->counters + (size_t)t.signal_ctr * CTR_STRIDE, 1u);
}

// One warp waits for ring slot `seq`: lane 0 polls with the watchdog and the
// abort flag, the warp learns the outcome by shuffle.  Every warp waits for
// every slot of its tasks (also slots holding none of its rows) before it
// releases the slot, so releases never run ahead of fills.
static __device__ __forceinline__ bool warp_wait_full(Ctx& c, int i, uint32_t par, uint32_t seq) {
    const VmParams& p = *c.p;
    int ok = 1;
    const uint64_t tw0 = (p.trace && c.warp == 0 && c.lane == 0) ? gtimer() : 0;
    if (c.lane == 0 && !mbar_try_wait(full_bar(c, i), par)) {
        const uint64_t t0 = gtimer();
        for (uint32_t it = 1;; ++it) {
            if (mbar_wait_hint(full_bar(c, i), par, SUSPEND_NS)) break;
            if ((it & 15u) == 0u) {
                if (aborted(p)) {
                    ok = 0;
                    break;
                }
                if (gtimer() - t0 > (uint64_t)p.watchdog_ns) {
                    raise_error(p, DEV_TIMEOUT, 0xFFFF0000u | (uint32_t)i, seq);
                    ok = 0;
                    break;
                }
            }
        }
    }
    if (tw0) c.sh->full_wait_ns += gtimer() - tw0;
    // Lane 0's acquire of the completed phase, then the warp barrier, orders
    // every lane's reads of the slot after the bulk copy (waits by all 32
    // lanes on one mbarrier word would serialise in shared memory).
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// ------------------------------------------------------------------ tokens
__device__ __forceinline__ unsigned long long key_tag(uint32_t epoch) {
    return (unsigned long long)(epoch + 1u);
}
__device__ __forceinline__ uint32_t float_order(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Token fed at step s.  Called by thread 0; broadcast through shared memory.
static __device__ __forceinline__ int step_token(const VmParams& p, int step) {
    int tok;
    if (p.forced) {
        tok = __ldg(p.forced + step);
    } else if (step == 0) {
        tok = p.pending >= 0 ? p.pending : (int)__ldcg((const unsigned int*)p.status + 3);
    } else {
        unsigned long long k = __ldcg(p.key);
        if ((k >> 49) != key_tag((uint32_t)(p.epoch0 + step - 1))) {
            raise_error(p, DEV_BAD_KEY, 0xFFFFFFFEu, (uint32_t)step);
            return -1;
        }
        tok = (int)((1u << KEY_IDX_BITS) - 1u - (uint32_t)(k & ((1ull << KEY_IDX_BITS) - 1ull)));
    }
    if (tok < 0 || tok >= p.V) {
        raise_error(p, DEV_BAD_TOKEN, 0xFFFFFFFDu, (uint32_t)step);
        return -1;
    }
    return tok;
}

// ------------------------------------------------------------------ GEMV inputs
// Each prologue writes the task's input vector (K floats) into c.xs with all
// consumer threads and ends with a consumer barrier.

// RMSNorm(x) * gain, x from the residual stream or (layer 0) an embedding row.
// The gain loads are issued together with the x loads (one memory round trip).
template <int BASE>
static __device__ __forceinline__ void prologue_rmsnorm(Ctx& c, const float* x, const uint16_t* emb_row, const uint16_t* gain, int K,
                                 float eps) {
    float ss = 0.f;
    for (int g = c.tid; g < (K >> 3); g += NT) {
        const uint4 graw = __ldg((const uint4*)(gain + 8 * g));
        float v[8];
        if (emb_row) {
            const uint4 raw = __ldg((const uint4*)(emb_row + 8 * g));
            const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[2 * i] = base_to_f32<BASE>(wv[i] & 0xFFFFu);
                v[2 * i + 1] = base_to_f32<BASE>(wv[i] >> 16);
            }
        } else {
            const float4 a = __ldcg((const float4*)(x + 8 * g));
            const float4 b = __ldcg((const float4*)(x + 8 * g + 4));
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
        const uint32_t gv[4] = {graw.x, graw.y, graw.z, graw.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // x * gain now; the common 1/rms factor is applied below
            v[2 * i] *= base_to_f32<BASE>(gv[i] & 0xFFFFu);
            v[2 * i + 1] *= base_to_f32<BASE>(gv[i] >> 16);
        }
        *(float4*)(c.xs + 8 * g) = make_float4(v[0], v[1], v[2], v[3]);
        *(float4*)(c.xs + 8 * g + 4) = make_float4(v[4], v[5], v[6], v[7]);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if (c.lane == 0) c.sh->norm[c.warp] = ss;
    bar_consumers();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) tot += c.sh->norm[w];
    c.rstd = rsqrtf(tot / (float)K + eps);  // applied to the fragments by gemv_rows
}

// Merge the split-KV partials of every query head into the attention output:
// o = sum_c e^(m_c - M) acc_c / sum_c e^(m_c - M) l_c.  The (max, sum) pairs of
// all heads are read cooperatively and turned into per-chunk weights in
// shared memory; each thread then reads its chunk accumulators with batches
// of independent loads.
static __device__ __forceinline__ void prologue_attention(Ctx& c) {
    const VmParams& p = *c.p;
    const int C = p.C, HC = p.Hq * C;
    float* wgt = c.sh->mg.mw;  // [Hq][C]
    for (int i = c.tid; i < HC; i += NT) wgt[i] = __ldcg(p.part_ml + 2 * i);        // m
    for (int i = c.tid; i < HC; i += NT) c.sh->mg.ml[i] = __ldcg(p.part_ml + 2 * i + 1);  // l
    bar_consumers();
    if (c.tid < p.Hq) {
        float* wh = wgt + c.tid * C;
        const float* lh = c.sh->mg.ml + c.tid * C;
        float M = -3.0e38f;
        for (int ch = 0; ch < C; ++ch) M = fmaxf(M, wh[ch]);
        float den = 0.f;
        for (int ch = 0; ch < C; ++ch) {
            wh[ch] = expf(wh[ch] - M);
            den = fmaf(wh[ch], lh[ch], den);
        }
        const float inv = 1.f / den;
        for (int ch = 0; ch < C; ++ch) wh[ch] *= inv;
    }
    bar_consumers();
    for (int g = c.tid; g < (p.q_dim >> 3); g += NT) {
        const int hq = (8 * g) / p.hd, d0 = (8 * g) % p.hd;
        const float* wh = wgt + hq * C;
        const float* base = p.part_acc + (size_t)hq * C * p.hd + d0;
        float o[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int c0 = 0; c0 < C; c0 += 4) {
            float4 a[4][2];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int ch = min(c0 + k, C - 1);
                a[k][0] = __ldcg((const float4*)(base + (size_t)ch * p.hd));
                a[k][1] = __ldcg((const float4*)(base + (size_t)ch * p.hd + 4));
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float w = c0 + k < C ? wh[c0 + k] : 0.f;
                o[0] = fmaf(w, a[k][0].x, o[0]); o[1] = fmaf(w, a[k][0].y, o[1]);
                o[2] = fmaf(w, a[k][0].z, o[2]); o[3] = fmaf(w, a[k][0].w, o[3]);
                o[4] = fmaf(w, a[k][1].x, o[4]); o[5] = fmaf(w, a[k][1].y, o[5]);
                o[6] = fmaf(w, a[k][1].z, o[6]); o[7] = fmaf(w, a[k][1].w, o[7]);
            }
        }
        *(float4*)(c.xs + 8 * g) = make_float4(o[0], o[1], o[2], o[3]);
        *(float4*)(c.xs + 8 * g + 4) = make_float4(o[4], o[5], o[6], o[7]);
    }
    c.rstd = 1.f;
    bar_consumers();
}

// ------------------------------------------------------------------ GEMV rows
// Packed fp32 FMA on register pairs (sm_100+): {d.x, d.y} = {a.x*b.x + c.x, a.y*b.y + c.y}.
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
    return (unsigned long long)__float_as_uint(lo) | ((unsigned long long)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float sum2(unsigned long long v) {
    return __uint_as_float((uint32_t)v) + __uint_as_float((uint32_t)(v >> 32));
}

// The lane's partial dot product of one packed weight row with its register
// fragment xr of the input vector (no cross-lane reduction).  Lane L of a
// row's warp group owns the 8-wide k-groups L, L + S, ..., L + (NG-1) S
// (S = 32 * warps per row): the 32 lanes of a warp read consecutive
// 16/8/4-byte groups, so shared-memory reads have no bank conflicts.  NG is
// a compile-time count so that all loads of the row are issued before the
// arithmetic; only the last group can lie past K and is zeroed by `tail_ok`.
template <int WT, int NG>
__device__ __forceinline__ float row_partial(const uint8_t* row, int K, int L, int S, bool tail_ok,
                                             const unsigned long long (&xr)[MAXG][4]) {
    if constexpr (WT == MK_W_BF16 || WT == MK_W_FP16) {
        uint4 w[NG];
#pragma unroll
        for (int j = 0; j < NG; ++j)
            w[j] = (j < NG - 1 || tail_ok) ? *(const uint4*)(row + (L + S * j) * 16) : make_uint4(0, 0, 0, 0);
        unsigned long long a0 = 0ull, a1 = 0ull;
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const uint32_t wv[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                unsigned long long wp;
                if constexpr (WT == MK_W_BF16) {
                    wp = pack2(__uint_as_float(wv[i] << 16), __uint_as_float(wv[i] & 0xFFFF0000u));
                } else {
                    const float2 f = __half22float2(*(const __half2*)&wv[i]);
                    wp = pack2(f.x, f.y);
                }
                if (i & 1) a1 = ffma2(wp, xr[j][i], a1);
                else a0 = ffma2(wp, xr[j][i], a0);
            }
        }
        return sum2(a0) + sum2(a1);
    } else if constexpr (WT == MK_W_INT8_ROW) {
        uint2 w[NG];
#pragma unroll
        for (int j = 0; j < NG; ++j)
            w[j] = (j < NG - 1 || tail_ok) ? *(const uint2*)(row + (L + S * j) * 8) : make_uint2(0x80808080u, 0x80808080u);
        unsigned long long a0 = 0ull, a1 = 0ull;
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const uint32_t u0 = w[j].x ^ 0x80808080u, u1 = w[j].y ^ 0x80808080u;
            a0 = ffma2(pack2(i8_to_f32(u0, 0), i8_to_f32(u0, 1)), xr[j][0], a0);
            a1 = ffma2(pack2(i8_to_f32(u0, 2), i8_to_f32(u0, 3)), xr[j][1], a1);
            a0 = ffma2(pack2(i8_to_f32(u1, 0), i8_to_f32(u1, 1)), xr[j][2], a0);
            a1 = ffma2(pack2(i8_to_f32(u1, 2), i8_to_f32(u1, 3)), xr[j][3], a1);
        }
        return sum2(a0) + sum2(a1);
    } else {  // int4: group-128 scales follow the nibbles
        uint32_t w[NG];
        float sc[NG];
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const bool ok = j < NG - 1 || tail_ok;
            const int g = L + S * j;
            w[j] = ok ? *(const uint32_t*)(row + g * 4) : 0x88888888u;
            sc[j] = ok ? half_bits_to_f32(*(const uint16_t*)(row + K / 2 + 2 * (g >> 4))) : 0.f;
        }
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const uint32_t u = w[j] ^ 0x88888888u;
            unsigned long long p = ffma2(pack2(i4_to_f32(u, 0), i4_to_f32(u, 1)), xr[j][0], 0ull);
            p = ffma2(pack2(i4_to_f32(u, 2), i4_to_f32(u, 3)), xr[j][1], p);
            p = ffma2(pack2(i4_to_f32(u, 4), i4_to_f32(u, 5)), xr[j][2], p);
            p = ffma2(pack2(i4_to_f32(u, 6), i4_to_f32(u, 7)), xr[j][3], p);
            if (j & 1) a1 = fmaf(sc[j], sum2(p), a1);
            else a0 = fmaf(sc[j], sum2(p), a0);
        }
        return a0 + a1;
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ void bar_group(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ float silu(float g) { return g / (1.f + __expf(-g)); }

// Reduce v[0..N) (N a power of two <= 32) over the 32 lanes: log2(N) halving
// steps in which each lane sends half of its remaining values, then plain
// butterfly steps.  Lane l ends with the total of v[l >> (5 - log2 N)].
template <int N>
__device__ __forceinline__ float transpose_reduce(float (&v)[N], int lane) {
    constexpr int B = N >= 32 ? 5 : N >= 16 ? 4 : N >= 8 ? 3 : N >= 4 ? 2 : N >= 2 ? 1 : 0;
#pragma unroll
    for (int n = N, off = 16; n > 1; n >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
        }
    }
#pragma unroll
    for (int off = 16 >> B; off >= 1; off >>= 1) v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], off);
    return v[0];
}

// One GEMV task: rows [row0, row0 + nrows) in ring slots of rps = RW * ngroups
// rows; warp group grp owns rows [grp*RW, grp*RW + RW) of every slot (a gate/up
// pair stays inside one group).  Per slot a warp: waits (lane 0), computes the
// lane partials of its RW rows, releases the slot (its arrival on the slot's
// empty barrier; NW arrivals complete it), then reduces all RW rows with one
// transposed warp reduction, combines the warps of a shared row (group
// barrier) and writes the results from RW lanes in parallel.  No CTA-wide
// barrier inside.  After a failed wait a warp keeps walking the slots without
// touching them, so group barriers stay balanced; the task-end barrier then
// stops the CTA.  `xin` is the input vector (shared or, from_global, device
// memory).
template <int WT, int BASE, int NG, int RW>
static __device__ __forceinline__ void gemv_rows(Ctx& c, const int op, const int layer, const int row0, const int nrows, const int K,
                          const int row_bytes, const int g, const float* xin, const bool from_global, int step,
                          int tok, float& best_v, int& best_i) {
    const VmParams& p = *c.p;
    const int ngroups = NW / g;
    const int grp = c.warp / g, wig = c.warp % g;
    const int L = wig * 32 + c.lane, S = 32 * g;
    const int G = K >> 3;
    const bool tail_ok = L + S * (NG - 1) < G;
    const float xscale = from_global ? 1.f : c.rstd;
    unsigned long long xr[MAXG][4];
#pragma unroll
    for (int j = 0; j < NG; ++j) {
        const int gi = (j < NG - 1 || tail_ok) ? L + S * j : 0;
        float4 a, b;
        if (from_global) {
            a = __ldcg((const float4*)(xin + 8 * gi));
            b = __ldcg((const float4*)(xin + 8 * gi + 4));
        } else {
            a = *(const float4*)(xin + 8 * gi);
            b = *(const float4*)(xin + 8 * gi + 4);
        }
        const bool ok = j < NG - 1 || tail_ok;
        const float f = xscale;
        xr[j][0] = ok ? pack2(a.x * f, a.y * f) : 0ull;
        xr[j][1] = ok ? pack2(a.z * f, a.w * f) : 0ull;
        xr[j][2] = ok ? pack2(b.x * f, b.y * f) : 0ull;
        xr[j][3] = ok ? pack2(b.z * f, b.w * f) : 0ull;
    }
    constexpr int B = RW >= 8 ? 3 : RW >= 4 ? 2 : 1;  // log2(RW)
    const int rps = RW * ngroups;
    const int n_slots = p.n_slots, slot_bytes = p.slot_bytes;
    // after the reduction lane l holds row (l >> (5 - B)) of the group's RW rows
    const int my_r = c.lane >> (5 - B);
    const bool writer = (c.lane & ((32 >> B) - 1)) == 0;
    bool dead = false;
    int par = 0;
    uint32_t seq = c.slot_seq;
    int si = c.slot_i;
    uint32_t phase = c.slot_phase;
    for (int r0 = 0; r0 < nrows; r0 += rps) {
        const int rows_here = min(rps, nrows - r0);
        const int first = grp * RW;  // first row of this group inside the slot
        const int row_g = row0 + r0 + first + my_r;  // global row this lane may finish
        const bool has_row = first + my_r < rows_here;
        // residual input of this lane's row, requested before the slot arrives
        float resid = 0.f;
        if (writer && has_row && !dead) {
            if (op == OP_DOWN || (op == OP_O && layer > 0)) {
                resid = __ldcg(p.x + row_g);
            } else if (op == OP_O) {
                const uint16_t* e = (const uint16_t*)(p.w + p.embed) + (size_t)tok * p.d;
                resid = base_to_f32<BASE>(__ldg(e + row_g));
            }
        }
        if (!dead) dead = !warp_wait_full(c, si, phase, seq);
        const uint8_t* slot = c.ring + (size_t)si * slot_bytes;
        float v[RW];
        float scale = 1.f;
#pragma unroll
        for (int r = 0; r < RW; ++r)
            v[r] = (!dead && first + r < rows_here)
                       ? row_partial<WT, NG>(slot + (size_t)(first + r) * row_bytes, K, L, S, tail_ok, xr)
                       : 0.f;
        if constexpr (WT == MK_W_INT8_ROW) {
            if (writer && has_row && !dead) scale = half_bits_to_f32(*(const uint16_t*)(slot + (size_t)(first + my_r) * row_bytes + K));
        }
        __syncwarp();
        if (c.lane == 0 && !dead) mbar_arrive(empty_bar(c, si));  // the slot is no longer read
        float tot = transpose_reduce<RW>(v, c.lane);
        if (g > 1) {
            float* scr = &c.sh->gpart[grp][par][0][0];  // [row][warp]
            if (writer) scr[my_r * NW + wig] = tot;
            bar_group(2 + grp, S);
            if (wig == 0 && writer) {
                tot = 0.f;
                for (int w = 0; w < g; ++w) tot += scr[my_r * NW + w];
            }
            par ^= 1;
        }
        if constexpr (WT == MK_W_INT8_ROW) tot *= scale;
        if (op == OP_GU) {  // rows alternate gate, up: the up total sits one row further
            const float up = __shfl_down_sync(0xFFFFFFFFu, tot, 32 >> B);
            if (wig == 0 && writer && has_row && !dead && !(my_r & 1)) p.h[row_g >> 1] = silu(tot) * up;
        } else if (wig == 0 && writer && has_row && !dead) {
            if (op == OP_LM) {
                if (p.logits) p.logits[(size_t)step * p.V + row_g] = tot;
                if (tot > best_v) {  // rows ascend per lane: the first maximum is kept
                    best_v = tot;
                    best_i = row_g;
                }
            } else if (op == OP_QKV) {
                p.qkv[row_g] = tot;
            } else {  // O and down: residual add
                p.x[row_g] = resid + tot;
            }
        }
        ++seq;
        if (++si == n_slots) {
            si = 0;
            phase ^= 1u;
        }
    }
    c.slot_seq = seq;
    c.slot_i = si;
    c.slot_phase = phase;
    if (dead && c.lane == 0) c.sh->abort = 1;
}

template <int WT, int BASE>
static __device__ __forceinline__ void gemv_task(Ctx& c, const DevTask& task, const float* xin, bool from_global, int step, int tok,
                          float& best_v, int& best_i) {
    const int op = task.op, layer = task.layer, row0 = task.row0, nrows = task.nrows, K = task.K;
    const int row_bytes = task.row_bytes, g = task.wpr, rw = task.rw;
    const int S = 32 * g, ng = ((K >> 3) + S - 1) / S;
#define MK_ROWS(N, R) gemv_rows<WT, BASE, N, R>(c, op, layer, row0, nrows, K, row_bytes, g, xin, from_global, step, tok, best_v, best_i)
#define MK_NG(R)                         \
    switch (ng) {                        \
        case 1: MK_ROWS(1, R); break;    \
        case 2: MK_ROWS(2, R); break;    \
        case 3: MK_ROWS(3, R); break;    \
        case 4: MK_ROWS(4, R); break;    \
        case 5: MK_ROWS(5, R); break;    \
        case 6: MK_ROWS(6, R); break;    \
        case 7: MK_ROWS(7, R); break;    \
        default: MK_ROWS(8, R); break;   \
    }
    if (rw >= 8) {
        MK_NG(8)
    } else if (rw == 4) {
        MK_NG(4)
    } else {
        MK_NG(2)
    }
#undef MK_NG
#undef MK_ROWS
}

// ------------------------------------------------------------------ attention
template <int DPL>
__device__ __forceinline__ void load_kv_row(const uint16_t* rowp, int lane, float (&f)[DPL]) {
    if constexpr (DPL == 2) {
        const uint32_t w = __ldcg((const unsigned int*)(rowp + lane * 2));
        f[0] = bf16_bits_to_f32(w & 0xFFFFu);
        f[1] = bf16_bits_to_f32(w >> 16);
    } else {
        const uint2 w = __ldcg((const uint2*)(rowp + lane * 4));
        f[0] = bf16_bits_to_f32(w.x & 0xFFFFu);
        f[1] = bf16_bits_to_f32(w.x >> 16);
        f[2] = bf16_bits_to_f32(w.y & 0xFFFFu);
        f[3] = bf16_bits_to_f32(w.y >> 16);
    }
}

// One (KV head, chunk) task: RoPE for the group's queries and this step's
// key, K/V append at pos (last chunk only), then an online-softmax pass over
// the chunk's positions in tiles of ATTN_TILE.  Warp w owns positions
// w, w+8, ... of a tile for the scores (its K rows in registers) and stages
// their V rows in shared memory; for P.V each thread owns fixed output
// elements (head, dim).  The first tile's rows are requested before the
// queries are rotated, so cache reads overlap the qkv reads.  Writes
// (max, sum, unnormalised output) per query head.
template <int HD>
static __device__ __forceinline__ void attn_task(Ctx& c, const DevTask& t, int step) {
    const VmParams& p = *c.p;
    Shared& sh = *c.sh;
    constexpr int DPL = HD / 32;            // dims per lane
    constexpr int PPW = ATTN_TILE / NW;     // positions per warp per tile
    constexpr int OPT = MAX_REP * HD / NT;  // output elements per thread (upper bound)
    const int rep = p.Hq / p.Hkv, g = t.row0, ch = t.nrows, C = t.K, l = t.layer;
    const int pos = p.pos0 + step, len = pos + 1;
    const int j0 = (int)((int64_t)ch * len / C), j1 = (int)((int64_t)(ch + 1) * len / C);
    const float scale = rsqrtf((float)HD);
    constexpr int half = HD / 2;
    const size_t head_stride = (size_t)p.max_seq * HD;
    uint16_t* kbase = p.kv + (((size_t)l * 2 + 0) * p.Hkv + g) * head_stride;
    uint16_t* vbase = p.kv + (((size_t)l * 2 + 1) * p.Hkv + g) * head_stride;

    float kf[PPW][DPL];
    uint32_t vraw[PPW][DPL / 2];
    auto load_tile = [&](int jt, int n) {
#pragma unroll
        for (int k = 0; k < PPW; ++k) {
            const int jj = c.warp + NW * k, j = jt + jj;
            if (jj < n && j != pos) {
                load_kv_row<DPL>(kbase + (size_t)j * HD, c.lane, kf[k]);
                if constexpr (DPL == 2) {
                    vraw[k][0] = __ldcg((const unsigned int*)(vbase + (size_t)j * HD + c.lane * 2));
                } else {
                    const uint2 w = __ldcg((const uint2*)(vbase + (size_t)j * HD + c.lane * 4));
                    vraw[k][0] = w.x;
                    vraw[k][1] = w.y;
                }
            }
        }
    };
    auto stage_v = [&](int jt, int n) {  // V rows -> shared memory (pos from this step's value)
#pragma unroll
        for (int k = 0; k < PPW; ++k) {
            const int jj = c.warp + NW * k, j = jt + jj;
            if (jj < n) {
                uint32_t* dst = (uint32_t*)(sh.at.sv + jj * HD + c.lane * DPL);
#pragma unroll
                for (int i = 0; i < DPL / 2; ++i) {
                    if (j == pos) {
                        dst[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(sh.at.vcur[c.lane * DPL + 2 * i])) |
                                 ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(sh.at.vcur[c.lane * DPL + 2 * i + 1])) << 16);
                    } else {
                        dst[i] = vraw[k][i];
                    }
                }
                if (j == pos) {
#pragma unroll
                    for (int i = 0; i < DPL; ++i) kf[k][i] = sh.at.kcur[c.lane * DPL + i];
                }
            }
        }
    };
    if (j1 > j0) load_tile(j0, min(ATTN_TILE, j1 - j0));

    for (int i = c.tid; i < (rep + 1) * half; i += NT) {
        const int hh = i / half, dd = i % half;
        const float* src = hh < rep ? p.qkv + (size_t)(g * rep + hh) * HD : p.qkv + p.q_dim + (size_t)g * HD;
        const float x1 = __ldcg(src + dd), x2 = __ldcg(src + dd + half);
        const float ang = __fmul_rn((float)pos, __ldg(p.inv_freq + dd));
        float sn, cs;
        sincosf(ang, &sn, &cs);
        const float o1 = x1 * cs - x2 * sn, o2 = x2 * cs + x1 * sn;
        if (hh < rep) {
            sh.at.q[hh * HD + dd] = o1 * scale;
            sh.at.q[hh * HD + dd + half] = o2 * scale;
        } else {
            sh.at.kcur[dd] = round_bf16(o1);
            sh.at.kcur[dd + half] = round_bf16(o2);
        }
    }
    for (int i = c.tid; i < HD; i += NT)
        sh.at.vcur[i] = round_bf16(__ldcg(p.qkv + p.q_dim + p.kv_dim + (size_t)g * HD + i));
    if (c.tid < rep) {
        sh.m[c.tid] = -1.0e30f;
        sh.l[c.tid] = 0.f;
    }
    bar_consumers();
    if (ch == C - 1) {
        for (int i = c.tid; i < HD; i += NT) {
            kbase[(size_t)pos * HD + i] = __bfloat16_as_ushort(__float2bfloat16_rn(sh.at.kcur[i]));
            vbase[(size_t)pos * HD + i] = __bfloat16_as_ushort(__float2bfloat16_rn(sh.at.vcur[i]));
        }
    }
    float acc[OPT];
#pragma unroll
    for (int e = 0; e < OPT; ++e) acc[e] = 0.f;

    for (int jt = j0; jt < j1; jt += ATTN_TILE) {
        const int n = min(ATTN_TILE, j1 - jt);
        if (jt != j0) load_tile(jt, n);
        stage_v(jt, n);
        // scores for (position k, head h), four heads at a time: PPW*4 partial
        // sums per lane, transposed so that lane pairs hold the totals
        for (int h0 = 0; h0 < rep; h0 += 4) {
            float v[PPW * 4];
#pragma unroll
            for (int k = 0; k < PPW; ++k)
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) {
                    float sacc = 0.f;
                    if (h0 + hh < rep) {
#pragma unroll
                        for (int i = 0; i < DPL; ++i) sacc = fmaf(sh.at.q[(h0 + hh) * HD + c.lane * DPL + i], kf[k][i], sacc);
                    }
                    v[k * 4 + hh] = sacc;
                }
            const float sc = transpose_reduce<PPW * 4>(v, c.lane);
            constexpr int SH = PPW * 4 >= 32 ? 0 : PPW * 4 >= 16 ? 1 : 2;
            const int idx = c.lane >> SH, k = idx >> 2, hh = idx & 3, jj = c.warp + NW * k;
            if ((c.lane & ((1 << SH) - 1)) == 0 && h0 + hh < rep && jj < n) sh.at.sc[(h0 + hh) * ATTN_TILE + jj] = sc;
        }
        bar_consumers();
        if (c.warp < rep) {  // online softmax statistics: warp h owns query head h
            const int h = c.warp;
            const float a = c.lane < n ? sh.at.sc[h * ATTN_TILE + c.lane] : -3.0e38f;
            float mt = a;
#pragma unroll
            for (int o = 16; o; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, o));
            const float m_old = sh.m[h], m_new = fmaxf(m_old, mt);
            const float pa = c.lane < n ? expf(a - m_new) : 0.f;
            if (c.lane < n) sh.at.sc[h * ATTN_TILE + c.lane] = pa;
            const float ls = warp_sum(pa);
            if (c.lane == 0) {
                const float al = expf(m_old - m_new);
                sh.alpha[h] = al;
                sh.l[h] = sh.l[h] * al + ls;
                sh.m[h] = m_new;
            }
        }
        bar_consumers();
#pragma unroll
        for (int e = 0; e < OPT; ++e) {
            const int oe = c.tid + NT * e, h = oe / HD, dd = oe % HD;
            if (h < rep) {
                float a = acc[e] * sh.alpha[h];
                const float* pr = sh.at.sc + h * ATTN_TILE;
                for (int jj = 0; jj < n; ++jj) a = fmaf(pr[jj], bf16_bits_to_f32(sh.at.sv[jj * HD + dd]), a);
                acc[e] = a;
            }
        }
        bar_consumers();  // the next tile overwrites scores and V rows
    }
#pragma unroll
    for (int e = 0; e < OPT; ++e) {
        const int oe = c.tid + NT * e, h = oe / HD, dd = oe % HD;
        if (h < rep) p.part_acc[(((size_t)(g * rep + h)) * C + ch) * HD + dd] = acc[e];
    }
    if (c.tid < rep) {
        float* ml = p.part_ml + ((size_t)(g * rep + c.tid) * C + ch) * 2;
        ml[0] = sh.m[c.tid];
        ml[1] = sh.l[c.tid];
    }
}

// ------------------------------------------------------------------ producer
__device__ __forceinline__ bool streams_weights(const VmParams& p, int op) {
    return op == OP_QKV || op == OP_O || op == OP_GU || op == OP_DOWN || (op == OP_LM && !p.skip_lm);
}

// Walks the weight chunks of this CTA's queue in consumption order.  The
// current task's fields stay in registers, so the task table is read once
// per task, not once per chunk.
struct ChunkCursor {
    int s, qi, r0;
    int nrows, rps, row_bytes;  // current streaming task (nrows == 0: none loaded)
    const uint8_t* base;
};

// Advance to the next weight chunk (rows r0 .. r0 + rps of a streaming task);
// returns false at the end of the launch.
__device__ __forceinline__ bool next_chunk(const VmParams& p, int q0, int q1, ChunkCursor& k, const uint8_t*& src,
                                           uint32_t& bytes) {
    for (;;) {
        if (k.r0 < k.nrows) {
            src = k.base + (int64_t)k.r0 * k.row_bytes;
            bytes = (uint32_t)(min(k.rps, k.nrows - k.r0) * k.row_bytes);
            k.r0 += k.rps;
            return true;
        }
        // load the next streaming task
        k.nrows = 0;
        k.r0 = 0;
        if (k.qi >= q1) {
            if (++k.s >= p.n_steps) return false;
            k.qi = q0;
        }
        const DevTask& t = p.tasks[__ldg(p.queue + k.qi)];
        ++k.qi;
        const int op = __ldg(&t.op);
        if (streams_weights(p, op)) {
            k.nrows = __ldg(&t.nrows);
            k.rps = __ldg(&t.rps);
            k.row_bytes = __ldg(&t.row_bytes);
            k.base = p.w + __ldg((const long long*)&t.w_off);
        }
    }
}

// The weight-streaming lane.  Weights never depend on activations, so it
// walks the CTA's queue ahead of the consumers through every counter wait and
// every step: an L2 cursor keeps up to l2_ahead bytes requested from HBM into
// L2 (bulk prefetches, nothing to wait for), and the ring cursor copies chunk
// after chunk into the shared-memory slots as the consumers free them.
static __device__ __forceinline__ void producer_lane(Ctx& c) {
    const VmParams& p = *c.p;
    const uint64_t pol = evict_first_policy();
    const int q0 = p.queue_off[blockIdx.x], q1 = p.queue_off[blockIdx.x + 1];
    const int n_slots = p.n_slots;
    uint32_t seq = 0, phase = 0;  // phase: parity of the current use of slot si
    int si = 0;
    ChunkCursor ring{0, q0, 0, 0, 1, 0, nullptr}, pf{0, q0, 0, 0, 1, 0, nullptr};
    int64_t ring_bytes = 0, pf_bytes = 0;
    bool pf_done = p.l2_ahead <= 0;
    const uint8_t* src;
    uint32_t bytes;
    while (next_chunk(p, q0, q1, ring, src, bytes)) {
        ring_bytes += bytes;
        while (!pf_done && pf_bytes < ring_bytes + p.l2_ahead) {
            const uint8_t* psrc;
            uint32_t pbytes;
            if (!next_chunk(p, q0, q1, pf, psrc, pbytes)) {
                pf_done = true;
                break;
            }
            if (pf_bytes + pbytes > ring_bytes - bytes) bulk_prefetch_l2(psrc, pbytes);  // not yet in the ring
            pf_bytes += pbytes;
        }
        if (seq >= (uint32_t)n_slots) {  // wait for the previous use of slot si to be released
            const uint32_t par = phase ^ 1u;
            const uint64_t tw0 = p.trace ? gtimer() : 0;
            if (!mbar_try_wait(empty_bar(c, si), par)) {
                const uint64_t t0 = gtimer();
                bool stop = false;
                for (uint32_t it = 1;; ++it) {
                    if (mbar_wait_hint(empty_bar(c, si), par, SUSPEND_NS)) break;
                    if ((it & 15u) == 0u) {
                        if (aborted(p)) {
                            stop = true;
                            break;
                        }
                        if (gtimer() - t0 > (uint64_t)p.watchdog_ns) {
                            raise_error(p, DEV_TIMEOUT, 0xFFFE0000u | (uint32_t)si, seq);
                            stop = true;
                            break;
                        }
                    }
                }
                if (stop) break;
            }
            if (tw0) c.sh->prod_wait_ns += gtimer() - tw0;
        }
        mbar_expect_tx(full_bar(c, si), bytes);
        bulk_g2s(smem_u32(c.ring + (size_t)si * p.slot_bytes), src, bytes, full_bar(c, si), pol);
        ++seq;
        if (++si == n_slots) {
            si = 0;
            phase ^= 1u;
        }
    }
    c.sh->issued = seq;
}

static __device__ __forceinline__ void producer(Ctx& c) {
    if (c.lane == 0) producer_lane(c);
    __syncwarp();  // the warp reaches the final CTA barrier converged
}

// ------------------------------------------------------------------ consumer
template <int WT, int BASE, int HD>
static __device__ __forceinline__ void consumer(Ctx& c) {
    const VmParams& p = *c.p;
    const int q0 = p.queue_off[blockIdx.x], q1 = p.queue_off[blockIdx.x + 1];
    for (int s = 0; s < p.n_steps && !c.abort; ++s) {
        for (int qi = q0; qi < q1 && !c.abort; ++qi) {
            const int tid_ = __ldg(p.queue + qi);
            const DevTask* tp = p.tasks + tid_;
            DevTask t;  // fields read once into registers (read-only data path)
            t.op = __ldg(&tp->op);
            t.layer = __ldg(&tp->layer);
            t.row0 = __ldg(&tp->row0);
            t.nrows = __ldg(&tp->nrows);
            t.K = __ldg(&tp->K);
            t.row_bytes = __ldg(&tp->row_bytes);
            t.rps = __ldg(&tp->rps);
            t.wpr = __ldg(&tp->wpr);
            t.rw = __ldg(&tp->rw);
            t.n_waits = __ldg(&tp->n_waits);
            t.wait_ctr[0] = __ldg(&tp->wait_ctr[0]);
            t.wait_ctr[1] = __ldg(&tp->wait_ctr[1]);
            t.wait_cnt[0] = __ldg(&tp->wait_cnt[0]);
            t.wait_cnt[1] = __ldg(&tp->wait_cnt[1]);
            t.wait_off[0] = __ldg(&tp->wait_off[0]);
            t.wait_off[1] = __ldg(&tp->wait_off[1]);
            t.signal_ctr = __ldg(&tp->signal_ctr);
            const uint64_t t_start = p.trace ? gtimer() : 0;
            if (!wait_counters(c, t, tid_, s)) {
                c.abort = true;
                break;
            }
            const uint64_t t_waited = p.trace ? gtimer() : 0;
            int tok = 0;
            if (t.layer == 0 && (t.op == OP_QKV || t.op == OP_O)) {
                if (c.tid == 0) c.sh->tok = step_token(p, s);
                bar_consumers();
                tok = c.sh->tok;
                if (tok < 0) {
                    c.abort = true;
                    break;
                }
            }
            float best_v = -3.0e38f;
            int best_i = 0;
            const bool gemv = t.op == OP_QKV || t.op == OP_O || t.op == OP_GU || t.op == OP_DOWN ||
                              (t.op == OP_LM && !p.skip_lm);
            if (gemv) {
                switch (t.op) {
                    case OP_QKV: {
                        const uint16_t* gain = (const uint16_t*)(p.w + p.layer_bytes * t.layer + p.l_attn_norm);
                        const uint16_t* emb = t.layer == 0 ? (const uint16_t*)(p.w + p.embed) + (size_t)tok * p.d : nullptr;
                        prologue_rmsnorm<BASE>(c, p.x, emb, gain, p.d, p.eps);
                        break;
                    }
                    case OP_GU:
                        prologue_rmsnorm<BASE>(c, p.x, nullptr,
                                               (const uint16_t*)(p.w + p.layer_bytes * t.layer + p.l_ffn_norm), p.d, p.eps);
                        break;
                    case OP_LM:
                        prologue_rmsnorm<BASE>(c, p.x, nullptr, (const uint16_t*)(p.w + p.final_norm), p.d, p.eps);
                        break;
                    case OP_O: prologue_attention(c); break;
                    default: break;  // down reads h straight from device memory
                }
                if (t.op == OP_DOWN) gemv_task<WT, BASE>(c, t, p.h, true, s, tok, best_v, best_i);
                else gemv_task<WT, BASE>(c, t, c.xs, false, s, tok, best_v, best_i);
                if (t.op == OP_LM) {  // per-lane bests -> the warp's key (largest value, lowest index)
                    unsigned long long key = (key_tag((uint32_t)(p.epoch0 + s)) << 49) |
                                             ((unsigned long long)float_order(best_v) << KEY_IDX_BITS) |
                                             (unsigned long long)((1u << KEY_IDX_BITS) - 1u - (uint32_t)best_i);
#pragma unroll
                    for (int o = 16; o; o >>= 1) {
                        const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, key, o);
                        key = other > key ? other : key;
                    }
                    if (c.lane == 0) c.sh->keys[c.warp] = key;
                }
            } else if (t.op == OP_ATTN) {
                attn_task<HD>(c, t, s);
            } else if (t.op == OP_FIN) {
                if (c.tid == 0 && !p.skip_lm) {
                    const unsigned long long k = __ldcg(p.key);
                    if ((k >> 49) != key_tag((uint32_t)(p.epoch0 + s))) {
                        raise_error(p, DEV_BAD_KEY, (uint32_t)tid_, (uint32_t)s);
                    } else {
                        const int id = (int)((1u << KEY_IDX_BITS) - 1u - (uint32_t)(k & ((1ull << KEY_IDX_BITS) - 1ull)));
                        if (p.out_ids) p.out_ids[s] = id;
                        p.status[3] = (uint32_t)id;
                    }
                }
            }
            bar_consumers();
            if (t.op == OP_LM && !p.skip_lm && c.tid == 0 && !c.sh->abort) {
                // block argmax: largest value, lowest index on ties
                unsigned long long key = 0;
                for (int w = 0; w < NW; ++w) key = c.sh->keys[w] > key ? c.sh->keys[w] : key;
                atomicMax(p.key, key);
            }
            signal_counter(c, t);
            if (c.sh->abort) {  // read after the barrier: the same in every consumer thread
                c.abort = true;
                break;
            }
            if (p.trace && c.tid == 0) {
                const int k = s * (q1 - q0) + (qi - q0);
                if (k < p.trace_cap) {
                    unsigned long long* r = p.trace + ((size_t)blockIdx.x * p.trace_cap + k) * 8;
                    r[0] = (unsigned long long)tid_ | ((unsigned long long)s << 32);
                    r[1] = t_start;
                    r[2] = t_waited;
                    r[3] = gtimer();
                    r[4] = c.sh->full_wait_ns;
                    r[5] = c.slot_seq;
                    r[6] = *(volatile unsigned long long*)&c.sh->prod_wait_ns;
                    r[7] = 0;
                }
            }
        }
    }
    if (c.tid == 0) c.sh->consumed = c.slot_seq;
}

template <int WT, int BASE, int HD>
__global__ void __launch_bounds__(THREADS, 1) vm_kernel(const VmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Ctx c;
    c.p = &p;
    c.ring = smem_raw;
    c.xs = (float*)(smem_raw + (size_t)p.n_slots * p.slot_bytes);
    c.sh = (Shared*)(smem_raw + (size_t)p.n_slots * p.slot_bytes + (size_t)p.xs_floats * 4);
    c.tid = threadIdx.x;
    c.lane = threadIdx.x & 31;
    c.warp = threadIdx.x >> 5;
    c.slot_seq = 0;
    c.slot_i = 0;
    c.slot_phase = 0;
    c.abort = false;
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.n_slots; ++i) {
            mbar_init(full_bar(c, i), 1);
            mbar_init(empty_bar(c, i), NW);  // one arrival per consumer warp
        }
        c.sh->abort = 0;
        c.sh->prod_wait_ns = 0;
        c.sh->full_wait_ns = 0;
        c.sh->issued = 0;
        c.sh->consumed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (c.warp == NW) producer(c);
    else consumer<WT, BASE, HD>(c);
    __syncthreads();
    // Exit drain: after an abort the producer may have copies in flight into
    // slots nobody consumed; wait (bounded) for them before the CTA exits.
    if (threadIdx.x == 0) {
        const uint32_t issued = c.sh->issued, consumed = c.sh->consumed;
        for (uint32_t s = consumed; s < issued; ++s) {
            const int i = (int)(s % (uint32_t)p.n_slots);
            const uint32_t par = (s / (uint32_t)p.n_slots) & 1u;
            const uint64_t t0 = gtimer();
            while (!mbar_try_wait(full_bar(c, i), par) && gtimer() - t0 < (uint64_t)p.watchdog_ns) {
            }
        }
    }
}


}  // namespace mk
