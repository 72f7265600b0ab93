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
struct Shared {
    float red[2][NW * 32];          // slot reductions (double buffered)
    float norm[NW];                 // RMSNorm sum of squares
    float q[MAX_REP * 128];         // roped, scaled queries of one KV group
    float kcur[128], vcur[128];     // this step's K and V (bf16-rounded)
    float sc[MAX_REP * ATTN_TILE];  // scores / probabilities of a tile
    float o[MAX_REP * 128];         // attention output accumulator
    float m[MAX_REP], l[MAX_REP], alpha[MAX_REP];
    int32_t flag;                   // broadcast of a counter-wait result
    int32_t slot_ok;                // broadcast of a ring-slot wait result
    int32_t tok;                    // broadcast of the step's input token
    uint32_t consumed, issued;      // ring bookkeeping for the exit drain
    unsigned long long bars[2 * 16]; // full[16], empty[16]
};

struct Ctx {
    const VmParams* p;
    Shared* sh;
    uint8_t* ring;
    int tid, lane, warp;
    uint32_t slot_seq;   // slots consumed so far (consumer side)
    bool abort;
};

__device__ __forceinline__ uint32_t full_bar(Ctx& c, int i) { return smem_u32(&c.sh->bars[i]); }
__device__ __forceinline__ uint32_t empty_bar(Ctx& c, int i) { return smem_u32(&c.sh->bars[16 + i]); }

__device__ __forceinline__ bool aborted(const VmParams& p) { return ld_volatile(p.status) != 0; }

__device__ void raise_error(const VmParams& p, uint32_t code, uint32_t task, uint32_t detail) {
    if (atomicCAS(p.status, 0u, code) == 0u) {
        p.status[1] = task;
        p.status[2] = detail;
    }
}

// Consumer wait on a counter: thread 0 spins, the rest learn the outcome at
// the named barrier.  Returns false on abort or watchdog expiry.
__device__ bool wait_counters(Ctx& c, const DevTask& t, int task_id, int step) {
    const VmParams& p = *c.p;
    if (c.tid == 0) {
        int ok = 1;
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

__device__ __forceinline__ void signal_counter(Ctx& c, const DevTask& t) {
    bar_consumers();  // every consumer thread's writes precede the release
    if (c.tid == 0 && t.signal_ctr >= 0) {
        __threadfence();
        red_release_add(c.p->counters + (size_t)t.signal_ctr * CTR_STRIDE, 1u);
    }
}

// Wait for ring slot `seq` to be filled.  Thread 0 alone decides (with the
// watchdog and the abort flag) and the decision reaches every consumer thread
// through the named barrier, so all of them take the same path afterwards.
// Once the phase has completed it cannot flip again before this CTA releases
// the slot, so the other threads' own try_wait succeeds at once.
__device__ bool wait_full(Ctx& c, uint32_t seq) {
    const VmParams& p = *c.p;
    const int i = (int)(seq % (uint32_t)p.n_slots);
    const uint32_t par = (seq / (uint32_t)p.n_slots) & 1u;
    if (c.tid == 0) {
        int ok = 1;
        if (!mbar_try_wait(full_bar(c, i), par)) {
            const uint64_t t0 = gtimer();
            for (uint32_t it = 1;; ++it) {
                if (mbar_try_wait(full_bar(c, i), par)) break;
                if ((it & 255u) == 0u) {
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
        c.sh->slot_ok = ok;
    }
    bar_consumers();
    if (!c.sh->slot_ok) return false;
    if (c.tid != 0)
        while (!mbar_try_wait(full_bar(c, i), par)) {
        }
    return true;
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
__device__ int step_token(const VmParams& p, int step) {
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
// Each consumer thread owns the k-groups g = tid + j*NT (8 consecutive k each).
__device__ __forceinline__ int n_groups(int K, int tid) {
    const int G = K >> 3;
    return tid < G ? (G - tid + NT - 1) / NT : 0;
}

template <int BASE>
__device__ void load_rmsnorm(Ctx& c, const float* x, const uint16_t* emb_row, const uint16_t* gain,
                             int K, float eps, float (&xf)[MAXG][8]) {
    const int ng = n_groups(K, c.tid);
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < MAXG; ++j) {
        if (j < ng) {
            const int g = c.tid + j * NT;
            if (emb_row) {
                uint4 raw = __ldg((const uint4*)(emb_row + 8 * g));
                uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    xf[j][2 * i] = base_to_f32<BASE>(wv[i] & 0xFFFFu);
                    xf[j][2 * i + 1] = base_to_f32<BASE>(wv[i] >> 16);
                }
            } else {
                float4 a = __ldcg((const float4*)(x + 8 * g));
                float4 b = __ldcg((const float4*)(x + 8 * g + 4));
                xf[j][0] = a.x; xf[j][1] = a.y; xf[j][2] = a.z; xf[j][3] = a.w;
                xf[j][4] = b.x; xf[j][5] = b.y; xf[j][6] = b.z; xf[j][7] = b.w;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) ss = fmaf(xf[j][i], xf[j][i], ss);
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if (c.lane == 0) c.sh->norm[c.warp] = ss;
    bar_consumers();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) tot += c.sh->norm[w];
    const float rstd = rsqrtf(tot / (float)K + eps);
#pragma unroll
    for (int j = 0; j < MAXG; ++j) {
        if (j < ng) {
            const int g = c.tid + j * NT;
            uint4 raw = __ldg((const uint4*)(gain + 8 * g));
            uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xf[j][2 * i] *= rstd * base_to_f32<BASE>(wv[i] & 0xFFFFu);
                xf[j][2 * i + 1] *= rstd * base_to_f32<BASE>(wv[i] >> 16);
            }
        }
    }
}

__device__ void load_vector(Ctx& c, const float* v, int K, float (&xf)[MAXG][8]) {
    const int ng = n_groups(K, c.tid);
#pragma unroll
    for (int j = 0; j < MAXG; ++j) {
        if (j < ng) {
            const int g = c.tid + j * NT;
            float4 a = __ldcg((const float4*)(v + 8 * g));
            float4 b = __ldcg((const float4*)(v + 8 * g + 4));
            xf[j][0] = a.x; xf[j][1] = a.y; xf[j][2] = a.z; xf[j][3] = a.w;
            xf[j][4] = b.x; xf[j][5] = b.y; xf[j][6] = b.z; xf[j][7] = b.w;
        }
    }
}

// Merge the split-KV partials of every query head into the attention output
// (the thread's own k-groups of the O projection input).
__device__ void load_attention(Ctx& c, float (&xf)[MAXG][8]) {
    const VmParams& p = *c.p;
    const int ng = n_groups(p.q_dim, c.tid);
#pragma unroll
    for (int j = 0; j < MAXG; ++j) {
        if (j < ng) {
            const int g = c.tid + j * NT;
            const int hq = (8 * g) / p.hd, d0 = (8 * g) % p.hd;
            const float* ml = p.part_ml + (size_t)hq * p.C * 2;
            float M = -3.0e38f;
            for (int ch = 0; ch < p.C; ++ch) M = fmaxf(M, __ldcg(ml + 2 * ch));
            float den = 0.f, o[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            for (int ch = 0; ch < p.C; ++ch) {
                const float wgt = expf(__ldcg(ml + 2 * ch) - M);
                den = fmaf(wgt, __ldcg(ml + 2 * ch + 1), den);
                const float* a = p.part_acc + ((size_t)hq * p.C + ch) * p.hd + d0;
                float4 a0 = __ldcg((const float4*)a), a1 = __ldcg((const float4*)(a + 4));
                o[0] = fmaf(wgt, a0.x, o[0]); o[1] = fmaf(wgt, a0.y, o[1]);
                o[2] = fmaf(wgt, a0.z, o[2]); o[3] = fmaf(wgt, a0.w, o[3]);
                o[4] = fmaf(wgt, a1.x, o[4]); o[5] = fmaf(wgt, a1.y, o[5]);
                o[6] = fmaf(wgt, a1.z, o[6]); o[7] = fmaf(wgt, a1.w, o[7]);
            }
            const float inv = 1.f / den;
#pragma unroll
            for (int i = 0; i < 8; ++i) xf[j][i] = o[i] * inv;
        }
    }
}

// ------------------------------------------------------------------ GEMV slot kernels
// Accumulate acc[r] = sum_k w[r][k] * x[k] over this thread's k-groups for the
// `rows` rows of one ring slot.
template <int WT, int RP>
__device__ __forceinline__ void slot_dot(const uint8_t* slot, int rows, int row_bytes, int K, int tid,
                                         const float (&xf)[MAXG][8], float (&acc)[RP]) {
    const int ng = n_groups(K, tid);
    constexpr int JM = maxg_for(RP);
#pragma unroll
    for (int r = 0; r < RP; ++r) acc[r] = 0.f;
#pragma unroll
    for (int j = 0; j < JM; ++j) {
        if (j < ng) {
            const int g = tid + j * NT;
            if constexpr (WT == MK_W_BF16 || WT == MK_W_FP16) {
#pragma unroll
                for (int r = 0; r < RP; ++r) {
                    if (r < rows) {
                        const uint4 w = *(const uint4*)(slot + r * row_bytes + g * 16);
                        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
                        float a = acc[r];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            float lo, hi;
                            if constexpr (WT == MK_W_BF16) {
                                lo = __uint_as_float(wv[i] << 16);
                                hi = __uint_as_float(wv[i] & 0xFFFF0000u);
                            } else {
                                const float2 f = __half22float2(*(const __half2*)&wv[i]);
                                lo = f.x;
                                hi = f.y;
                            }
                            a = fmaf(lo, xf[j][2 * i], a);
                            a = fmaf(hi, xf[j][2 * i + 1], a);
                        }
                        acc[r] = a;
                    }
                }
            } else if constexpr (WT == MK_W_INT8_ROW) {
#pragma unroll
                for (int r = 0; r < RP; ++r) {
                    if (r < rows) {
                        const uint2 w = *(const uint2*)(slot + r * row_bytes + g * 8);
                        const uint32_t u0 = w.x ^ 0x80808080u, u1 = w.y ^ 0x80808080u;
                        float a = acc[r];
#pragma unroll
                        for (int i = 0; i < 4; ++i) a = fmaf(i8_to_f32(u0, i), xf[j][i], a);
#pragma unroll
                        for (int i = 0; i < 4; ++i) a = fmaf(i8_to_f32(u1, i), xf[j][4 + i], a);
                        acc[r] = a;
                    }
                }
            } else {  // int4, group-128 scales after the nibbles
#pragma unroll
                for (int r = 0; r < RP; ++r) {
                    if (r < rows) {
                        const uint8_t* row = slot + r * row_bytes;
                        const uint32_t u = *(const uint32_t*)(row + g * 4) ^ 0x88888888u;
                        const float s = half_bits_to_f32(*(const uint16_t*)(row + K / 2 + 2 * (g >> 4)));
                        float part = 0.f;
#pragma unroll
                        for (int i = 0; i < 8; ++i) part = fmaf(i4_to_f32(u, i), xf[j][i], part);
                        acc[r] = fmaf(s, part, acc[r]);
                    }
                }
            }
        }
    }
}

// Reduce acc[0..RP) over all NT consumer threads.  Returns, in lanes
// t < RP of warp 0, the total of row t.  Contains one consumer barrier.
template <int RP>
__device__ __forceinline__ float reduce_rows(Ctx& c, float (&acc)[RP], float* red) {
    constexpr int B = (RP >= 32) ? 5 : (RP >= 16) ? 4 : (RP >= 8) ? 3 : (RP >= 4) ? 2 : (RP >= 2) ? 1 : 0;
    // transposed reduction: each halving step sends half of the remaining rows
#pragma unroll
    for (int n = RP, off = 16; n > 1; n >>= 1, off >>= 1) {
        const bool upper = (c.lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? acc[i] : acc[i + n / 2];
            const float keep = upper ? acc[i + n / 2] : acc[i];
            acc[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
        }
    }
#pragma unroll
    for (int off = 16 >> B; off >= 1; off >>= 1) acc[0] += __shfl_xor_sync(0xFFFFFFFFu, acc[0], off);
    if ((c.lane & ((32 >> B) - 1)) == 0) red[c.warp * 32 + (c.lane >> (5 - B))] = acc[0];
    bar_consumers();
    float tot = 0.f;
    if (c.warp == 0 && c.lane < RP) {
#pragma unroll
        for (int w = 0; w < NW; ++w) tot += red[w * 32 + c.lane];
    }
    return tot;
}

__device__ __forceinline__ float silu(float g) { return g / (1.f + __expf(-g)); }

// One GEMV task: rows [row0, row0 + nrows) of the packed tensor, slot by slot.
template <int WT, int BASE, int RP>
__device__ void gemv_task(Ctx& c, const DevTask& t, int step, const float (&xf)[MAXG][8], int tok,
                          float& best_v, int& best_i) {
    const VmParams& p = *c.p;
    for (int r0 = 0; r0 < t.nrows; r0 += t.rps) {
        const int rows = min(t.rps, t.nrows - r0);
        const uint32_t seq = c.slot_seq;
        if (!wait_full(c, seq)) {
            c.abort = true;
            return;
        }
        const int si = (int)(seq % (uint32_t)p.n_slots);
        const uint8_t* slot = c.ring + (size_t)si * p.slot_bytes;
        float acc[RP];
        slot_dot<WT, RP>(slot, rows, t.row_bytes, t.K, c.tid, xf, acc);
        float tot = reduce_rows<RP>(c, acc, c.sh->red[seq & 1]);
        if (c.warp == 0) {
            const int r = t.row0 + r0 + c.lane;  // global row of this lane
            if constexpr (WT == MK_W_INT8_ROW) {
                if (c.lane < rows) tot *= half_bits_to_f32(*(const uint16_t*)(slot + c.lane * t.row_bytes + t.K));
            }
            __syncwarp();
            if (c.lane == 0) mbar_arrive(empty_bar(c, si));  // all reads of the slot are done
            if (t.op == OP_GU) {
                const float up = __shfl_down_sync(0xFFFFFFFFu, tot, 1);
                if (c.lane < rows && !(c.lane & 1)) p.h[r >> 1] = silu(tot) * up;
            } else if (c.lane < rows) {
                switch (t.op) {
                    case OP_QKV: p.qkv[r] = tot; break;
                    case OP_O: {
                        float xin;
                        if (t.layer == 0) {
                            const uint16_t* e = (const uint16_t*)(p.w + p.embed) + (size_t)tok * p.d;
                            xin = base_to_f32<BASE>(__ldg(e + r));
                        } else {
                            xin = __ldcg(p.x + r);
                        }
                        p.x[r] = xin + tot;
                        break;
                    }
                    case OP_DOWN: p.x[r] = __ldcg(p.x + r) + tot; break;
                    case OP_LM:
                        if (p.logits) p.logits[(size_t)step * p.V + r] = tot;
                        if (tot > best_v) {  // rows ascend: the first maximum is kept
                            best_v = tot;
                            best_i = r;
                        }
                        break;
                    default: break;
                }
            }
        }
        c.slot_seq = seq + 1;
    }
}

// ------------------------------------------------------------------ attention
// One (KV head, chunk) task: RoPE for the group's queries and this step's key,
// append K/V at pos (last chunk only), then an online-softmax pass over the
// chunk's positions; writes (max, sum, unnormalised output) per query head.
template <int HD>
__device__ void attn_task(Ctx& c, const DevTask& t, int step) {
    const VmParams& p = *c.p;
    Shared& sh = *c.sh;
    constexpr int DPL = HD / 32;  // dims per lane
    const int rep = p.Hq / p.Hkv, g = t.row0, ch = t.nrows, C = t.K, l = t.layer;
    const int pos = p.pos0 + step, len = pos + 1;
    const int j0 = (int)((int64_t)ch * len / C), j1 = (int)((int64_t)(ch + 1) * len / C);
    const float scale = rsqrtf((float)HD);
    constexpr int half = HD / 2;
    for (int i = c.tid; i < (rep + 1) * half; i += NT) {
        const int hh = i / half, dd = i % half;
        const float* src = hh < rep ? p.qkv + (size_t)(g * rep + hh) * HD : p.qkv + p.q_dim + (size_t)g * HD;
        const float x1 = __ldcg(src + dd), x2 = __ldcg(src + dd + half);
        const float ang = __fmul_rn((float)pos, __ldg(p.inv_freq + dd));
        float sn, cs;
        sincosf(ang, &sn, &cs);
        const float o1 = x1 * cs - x2 * sn, o2 = x2 * cs + x1 * sn;
        if (hh < rep) {
            sh.q[hh * HD + dd] = o1 * scale;
            sh.q[hh * HD + dd + half] = o2 * scale;
        } else {
            sh.kcur[dd] = round_bf16(o1);
            sh.kcur[dd + half] = round_bf16(o2);
        }
    }
    for (int i = c.tid; i < HD; i += NT) sh.vcur[i] = round_bf16(__ldcg(p.qkv + p.q_dim + p.kv_dim + (size_t)g * HD + i));
    for (int i = c.tid; i < rep * HD; i += NT) sh.o[i] = 0.f;
    if (c.tid < rep) {
        sh.m[c.tid] = -1.0e30f;
        sh.l[c.tid] = 0.f;
    }
    bar_consumers();
    const size_t head_stride = (size_t)p.max_seq * HD;
    uint16_t* kbase = p.kv + (((size_t)l * 2 + 0) * p.Hkv + g) * head_stride;
    uint16_t* vbase = p.kv + (((size_t)l * 2 + 1) * p.Hkv + g) * head_stride;
    if (ch == C - 1) {
        for (int i = c.tid; i < HD; i += NT) {
            kbase[(size_t)pos * HD + i] = __bfloat16_as_ushort(__float2bfloat16_rn(sh.kcur[i]));
            vbase[(size_t)pos * HD + i] = __bfloat16_as_ushort(__float2bfloat16_rn(sh.vcur[i]));
        }
    }
    float qr[MAX_REP][DPL];
#pragma unroll
    for (int h = 0; h < MAX_REP; ++h)
#pragma unroll
        for (int i = 0; i < DPL; ++i) qr[h][i] = h < rep ? sh.q[h * HD + c.lane * DPL + i] : 0.f;
    float acc[MAX_REP][DPL];
#pragma unroll
    for (int h = 0; h < MAX_REP; ++h)
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[h][i] = 0.f;

    for (int jt = j0; jt < j1; jt += ATTN_TILE) {
        const int n = min(ATTN_TILE, j1 - jt);
        // scores: warp per position, lanes split the head dims
        for (int jj = c.warp; jj < n; jj += NW) {
            const int j = jt + jj;
            float kf[DPL];
            if (j == pos) {
#pragma unroll
                for (int i = 0; i < DPL; ++i) kf[i] = sh.kcur[c.lane * DPL + i];
            } else if constexpr (DPL == 2) {
                const uint32_t kw = __ldcg((const unsigned int*)(kbase + (size_t)j * HD + c.lane * 2));
                kf[0] = bf16_bits_to_f32(kw & 0xFFFFu);
                kf[1] = bf16_bits_to_f32(kw >> 16);
            } else {
                const uint2 kw = __ldcg((const uint2*)(kbase + (size_t)j * HD + c.lane * 4));
                kf[0] = bf16_bits_to_f32(kw.x & 0xFFFFu);
                kf[1] = bf16_bits_to_f32(kw.x >> 16);
                kf[2] = bf16_bits_to_f32(kw.y & 0xFFFFu);
                kf[3] = bf16_bits_to_f32(kw.y >> 16);
            }
#pragma unroll
            for (int h = 0; h < MAX_REP; ++h) {
                if (h < rep) {
                    float s = 0.f;
#pragma unroll
                    for (int i = 0; i < DPL; ++i) s = fmaf(qr[h][i], kf[i], s);
#pragma unroll
                    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
                    if (c.lane == 0) sh.sc[h * ATTN_TILE + jj] = s;
                }
            }
        }
        bar_consumers();
        // online softmax statistics: warp h handles query head h
        if (c.warp < rep) {
            const int h = c.warp;
            const float a = c.lane < n ? sh.sc[h * ATTN_TILE + c.lane] : -3.0e38f;
            const float b = c.lane + 32 < n ? sh.sc[h * ATTN_TILE + c.lane + 32] : -3.0e38f;
            float mt = fmaxf(a, b);
#pragma unroll
            for (int o = 16; o; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, o));
            const float m_old = sh.m[h], m_new = fmaxf(m_old, mt);
            const float pa = c.lane < n ? expf(a - m_new) : 0.f;
            const float pb = c.lane + 32 < n ? expf(b - m_new) : 0.f;
            if (c.lane < n) sh.sc[h * ATTN_TILE + c.lane] = pa;
            if (c.lane + 32 < n) sh.sc[h * ATTN_TILE + c.lane + 32] = pb;
            float ls = pa + pb;
#pragma unroll
            for (int o = 16; o; o >>= 1) ls += __shfl_xor_sync(0xFFFFFFFFu, ls, o);
            if (c.lane == 0) {
                const float al = expf(m_old - m_new);
                sh.alpha[h] = al;
                sh.l[h] = sh.l[h] * al + ls;
                sh.m[h] = m_new;
            }
        }
        bar_consumers();
        // P.V: warp per position, lanes split the head dims
#pragma unroll
        for (int h = 0; h < MAX_REP; ++h) {
            if (h < rep) {
                const float al = sh.alpha[h];
#pragma unroll
                for (int i = 0; i < DPL; ++i) acc[h][i] *= al;
            }
        }
        for (int jj = c.warp; jj < n; jj += NW) {
            const int j = jt + jj;
            float vf[DPL];
            if (j == pos) {
#pragma unroll
                for (int i = 0; i < DPL; ++i) vf[i] = sh.vcur[c.lane * DPL + i];
            } else if constexpr (DPL == 2) {
                const uint32_t vw = __ldcg((const unsigned int*)(vbase + (size_t)j * HD + c.lane * 2));
                vf[0] = bf16_bits_to_f32(vw & 0xFFFFu);
                vf[1] = bf16_bits_to_f32(vw >> 16);
            } else {
                const uint2 vw = __ldcg((const uint2*)(vbase + (size_t)j * HD + c.lane * 4));
                vf[0] = bf16_bits_to_f32(vw.x & 0xFFFFu);
                vf[1] = bf16_bits_to_f32(vw.x >> 16);
                vf[2] = bf16_bits_to_f32(vw.y & 0xFFFFu);
                vf[3] = bf16_bits_to_f32(vw.y >> 16);
            }
#pragma unroll
            for (int h = 0; h < MAX_REP; ++h) {
                if (h < rep) {
                    const float pj = sh.sc[h * ATTN_TILE + jj];
#pragma unroll
                    for (int i = 0; i < DPL; ++i) acc[h][i] = fmaf(pj, vf[i], acc[h][i]);
                }
            }
        }
        bar_consumers();  // the next tile overwrites the scores
    }
#pragma unroll
    for (int h = 0; h < MAX_REP; ++h)
        if (h < rep)
#pragma unroll
            for (int i = 0; i < DPL; ++i) atomicAdd(&sh.o[h * HD + c.lane * DPL + i], acc[h][i]);
    bar_consumers();
    for (int i = c.tid; i < rep * HD; i += NT) {
        const int h = i / HD, dd = i % HD;
        p.part_acc[(((size_t)(g * rep + h)) * C + ch) * HD + dd] = sh.o[i];
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

__device__ void producer_lane(Ctx& c) {
    const VmParams& p = *c.p;
    const uint64_t pol = evict_first_policy();
    const int q0 = p.queue_off[blockIdx.x], q1 = p.queue_off[blockIdx.x + 1];
    uint32_t seq = 0;
    bool stop = false;
    for (int s = 0; s < p.n_steps && !stop; ++s) {
        for (int qi = q0; qi < q1 && !stop; ++qi) {
            const DevTask& t = p.tasks[p.queue[qi]];
            if (!streams_weights(p, t.op)) continue;
            for (int r0 = 0; r0 < t.nrows; r0 += t.rps) {
                const int rows = min(t.rps, t.nrows - r0);
                const uint32_t bytes = (uint32_t)(rows * t.row_bytes);
                const int si = (int)(seq % (uint32_t)p.n_slots);
                if (seq >= (uint32_t)p.n_slots) {
                    const uint32_t par = ((seq / (uint32_t)p.n_slots) & 1u) ^ 1u;
                    if (!mbar_try_wait(empty_bar(c, si), par)) {
                        const uint64_t t0 = gtimer();
                        for (uint32_t it = 1;; ++it) {
                            if (mbar_try_wait(empty_bar(c, si), par)) break;
                            if ((it & 255u) == 0u) {
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
                }
                mbar_expect_tx(full_bar(c, si), bytes);
                bulk_g2s(smem_u32(c.ring + (size_t)si * p.slot_bytes), p.w + t.w_off + (int64_t)r0 * t.row_bytes,
                         bytes, full_bar(c, si), pol);
                ++seq;
            }
        }
    }
    c.sh->issued = seq;
}

__device__ void producer(Ctx& c) {
    if (c.lane == 0) producer_lane(c);
    __syncwarp();  // the warp reaches the final CTA barrier converged
}

// ------------------------------------------------------------------ consumer
template <int WT, int BASE>
__device__ void consumer(Ctx& c) {
    const VmParams& p = *c.p;
    const int q0 = p.queue_off[blockIdx.x], q1 = p.queue_off[blockIdx.x + 1];
    float xf[MAXG][8];
    for (int s = 0; s < p.n_steps && !c.abort; ++s) {
        for (int qi = q0; qi < q1 && !c.abort; ++qi) {
            const int tid_ = p.queue[qi];
            const DevTask t = p.tasks[tid_];
            if (!wait_counters(c, t, tid_, s)) {
                c.abort = true;
                break;
            }
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
            switch (t.op) {
                case OP_QKV: {
                    const uint16_t* gain = (const uint16_t*)(p.w + p.layer_bytes * t.layer + p.l_attn_norm);
                    const uint16_t* emb = t.layer == 0 ? (const uint16_t*)(p.w + p.embed) + (size_t)tok * p.d : nullptr;
                    load_rmsnorm<BASE>(c, p.x, emb, gain, p.d, p.eps, xf);
                    break;
                }
                case OP_GU: {
                    const uint16_t* gain = (const uint16_t*)(p.w + p.layer_bytes * t.layer + p.l_ffn_norm);
                    load_rmsnorm<BASE>(c, p.x, nullptr, gain, p.d, p.eps, xf);
                    break;
                }
                case OP_LM:
                    if (!p.skip_lm) load_rmsnorm<BASE>(c, p.x, nullptr, (const uint16_t*)(p.w + p.final_norm), p.d, p.eps, xf);
                    break;
                case OP_O: load_attention(c, xf); break;
                case OP_DOWN: load_vector(c, p.h, p.F, xf); break;
                default: break;
            }
            if (t.op == OP_ATTN) {
                if (p.hd == 64) attn_task<64>(c, t, s);
                else attn_task<128>(c, t, s);
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
            } else if (!(t.op == OP_LM && p.skip_lm)) {
                switch (t.rp_log2) {
                    case 0: gemv_task<WT, BASE, 1>(c, t, s, xf, tok, best_v, best_i); break;
                    case 1: gemv_task<WT, BASE, 2>(c, t, s, xf, tok, best_v, best_i); break;
                    case 2: gemv_task<WT, BASE, 4>(c, t, s, xf, tok, best_v, best_i); break;
                    case 3: gemv_task<WT, BASE, 8>(c, t, s, xf, tok, best_v, best_i); break;
                    case 4: gemv_task<WT, BASE, 16>(c, t, s, xf, tok, best_v, best_i); break;
                    default: gemv_task<WT, BASE, 32>(c, t, s, xf, tok, best_v, best_i); break;
                }
                if (c.abort) break;
                if (t.op == OP_LM && c.warp == 0) {
                    // block argmax: largest value, lowest index on ties
                    unsigned long long key = (key_tag((uint32_t)(p.epoch0 + s)) << 49) |
                                             ((unsigned long long)float_order(best_v) << KEY_IDX_BITS) |
                                             (unsigned long long)((1u << KEY_IDX_BITS) - 1u - (uint32_t)best_i);
#pragma unroll
                    for (int o = 16; o; o >>= 1) {
                        const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, key, o);
                        key = other > key ? other : key;
                    }
                    if (c.lane == 0) atomicMax(p.key, key);
                }
            }
            signal_counter(c, t);
        }
    }
    if (c.tid == 0) c.sh->consumed = c.slot_seq;
}

template <int WT, int BASE>
__global__ void __launch_bounds__(THREADS, 1) vm_kernel(const VmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Ctx c;
    c.p = &p;
    c.ring = smem_raw;
    c.sh = (Shared*)(smem_raw + (size_t)p.n_slots * p.slot_bytes);
    c.tid = threadIdx.x;
    c.lane = threadIdx.x & 31;
    c.warp = threadIdx.x >> 5;
    c.slot_seq = 0;
    c.abort = false;
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.n_slots; ++i) {
            mbar_init(full_bar(c, i), 1);
            mbar_init(empty_bar(c, i), 1);
        }
        c.sh->issued = 0;
        c.sh->consumed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (c.warp == NW) producer(c);
    else consumer<WT, BASE>(c);
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

// ------------------------------------------------------------------ launch
template <int WT, int BASE>
static const void* kernel_ptr() {
    return (const void*)vm_kernel<WT, BASE>;
}

const void* vm_kernel_for(int wdtype, int base) {
    if (base == MK_W_FP16) return wdtype == MK_W_FP16 ? kernel_ptr<MK_W_FP16, MK_W_FP16>() : nullptr;
    switch (wdtype) {
        case MK_W_BF16: return kernel_ptr<MK_W_BF16, MK_W_BF16>();
        case MK_W_INT8_ROW: return kernel_ptr<MK_W_INT8_ROW, MK_W_BF16>();
        case MK_W_INT4_G128: return kernel_ptr<MK_W_INT4_G128, MK_W_BF16>();
        default: return nullptr;
    }
}

size_t vm_shared_bytes(int n_slots, int slot_bytes) {
    return (size_t)n_slots * slot_bytes + sizeof(Shared);
}

// ------------------------------------------------------------------ test kernels
// Dequantise a packed tensor with the decode kernel's own code -> float path.
template <int WT>
__global__ void dequant_kernel(const uint8_t* rows, int64_t stride, int first, int step, int nrows, int K,
                               float* out) {
    const int r = blockIdx.x;
    if (r >= nrows) return;
    const uint8_t* row = rows + (int64_t)(first + (int64_t)r * step) * stride;
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        float v;
        if constexpr (WT == MK_W_INT8_ROW) {
            const uint32_t word = *(const uint32_t*)(row + (k & ~3)) ^ 0x80808080u;
            v = i8_to_f32(word, k & 3) * half_bits_to_f32(*(const uint16_t*)(row + K));
        } else if constexpr (WT == MK_W_INT4_G128) {
            const uint32_t word = *(const uint32_t*)(row + (k >> 3) * 4) ^ 0x88888888u;
            v = i4_to_f32(word, k & 7) * half_bits_to_f32(*(const uint16_t*)(row + K / 2 + 2 * (k >> 7)));
        } else if constexpr (WT == MK_W_FP16) {
            v = half_bits_to_f32(((const uint16_t*)row)[k]);
        } else {
            v = bf16_bits_to_f32(((const uint16_t*)row)[k]);
        }
        out[(int64_t)r * K + k] = v;
    }
}

cudaError_t launch_dequant(int wdtype, const uint8_t* rows, int64_t stride, int first, int step, int nrows,
                           int K, float* out, cudaStream_t st) {
    dim3 grid(nrows), block(256);
    switch (wdtype) {
        case MK_W_INT8_ROW: dequant_kernel<MK_W_INT8_ROW><<<grid, block, 0, st>>>(rows, stride, first, step, nrows, K, out); break;
        case MK_W_INT4_G128: dequant_kernel<MK_W_INT4_G128><<<grid, block, 0, st>>>(rows, stride, first, step, nrows, K, out); break;
        case MK_W_FP16: dequant_kernel<MK_W_FP16><<<grid, block, 0, st>>>(rows, stride, first, step, nrows, K, out); break;
        default: dequant_kernel<MK_W_BF16><<<grid, block, 0, st>>>(rows, stride, first, step, nrows, K, out); break;
    }
    return cudaGetLastError();
}

// A wait that can never be satisfied, with the same watchdog as the VM: the
// kernel must give up, report DEV_TIMEOUT and return.
__global__ void watchdog_kernel(uint32_t* ctr, uint32_t* status, int64_t limit_ns) {
    if (threadIdx.x != 0) return;
    const uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if ((int32_t)(ld_acquire(ctr) - 1u) >= 0) {
            status[0] = DEV_OK;
            return;
        }
        if ((it & 63u) == 0u && gtimer() - t0 > (uint64_t)limit_ns) {
            status[0] = DEV_TIMEOUT;
            return;
        }
    }
}

cudaError_t launch_watchdog(uint32_t* ctr, uint32_t* status, int64_t limit_ns, cudaStream_t st) {
    watchdog_kernel<<<1, 32, 0, st>>>(ctr, status, limit_ns);
    return cudaGetLastError();
}

}  // namespace mk
