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
//  * Each warp streams its own weight rows through a private ring of
//    shared-memory slots filled by 16-byte cp.async.cg copies (no mbarriers,
//    no cross-warp hand-off).  A bulk-copy ring shared by the CTA capped the
//    stream near 4.7 TB/s with the full GEMV arithmetic; per-warp rings reach
//    ~7.1 TB/s.
//  * Weight bytes never depend on activations, so the per-warp stream runs
//    ahead across task boundaries and counter waits: the copies of the next
//    task's first rows are in flight while this warp waits or reduces.
//  * Warp groups own whole rows: each lane holds a fixed fragment of the
//    input vector in registers (fp32 pairs for packed fma.rn.f32x2; for int8
//    and int4 codes, the bytes of a 24-bit fixed-point copy for dp4a) and the
//    rows of a batch are reduced with one transposed warp reduction; large K
//    is split over 2-8 warps that combine through shared memory.
//  * Counters are u32 words on their own 128-byte lines; a wait is an
//    ld.acquire.gpu spin with a %globaltimer watchdog; a signal is a
//    red.release.gpu.add after a CTA barrier.  Thresholds scale with the
//    global step (epoch), so counters never need a reset between steps or
//    launches.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mk_internal.h"

// Device code of the decode kernel, included by one translation unit per
// weight type (each instantiates vm_kernel for head_dim 64 and 128).
#pragma once

namespace mk {

// ------------------------------------------------------------------ PTX helpers
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
// Named barrier 1 among all NT threads of the CTA.
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
// Two FP8 E4M3 codes (the low 16 bits, first code in the low byte) -> exact
// floats, through the hardware conversion to a half pair (every E4M3 value is
// a half value).
__device__ __forceinline__ unsigned long long e4m3x2_pair(uint32_t two) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
    const float2 f = __half22float2(*(const __half2*)&h);
    return (unsigned long long)__float_as_uint(f.x) | ((unsigned long long)__float_as_uint(f.y) << 32);
}

// ------------------------------------------------------------------ shared memory
// Layout: [input vector of a GEMV task | attention scratch] (one region: a
// CTA runs one task at a time and a GEMV task reads its input vector into
// registers before it ends) [Shared] [task records] [weight rings].
// Scratch of one attention task.
struct AttnScratch {
    float q[MAX_REP * 128];         // roped, scaled queries of one KV group
    float kcur[128], vcur[128];     // this step's K and V (bf16-rounded)
    float sc[MAX_REP * ATTN_TILE];  // scores of a tile, [head][position]
    float pt[ATTN_TILE * MAX_REP];  // probabilities of a tile, [position][head]
    uint16_t sv[ATTN_TILE * 128];   // V rows of the current tile (bf16); after the last
                                    // tile, the P.V partial sums of the position subsets
};
static_assert(4 * (NT / 64) * 128 * sizeof(float) <= sizeof(AttnScratch::sv), "P.V subset sums, four heads");
struct MergeScratch {
    float mw[MAX_HC];               // per (head, chunk) max, then weight
    float ml[MAX_HC];               // per (head, chunk) sum
};

struct Shared {
    float norm[NW];                 // RMSNorm sum of squares
    float nmax[NW];                 // per-warp max |input| of an integer-dot task
    float gpart[NW][2][8][NW];      // [group][parity][row][warp]: partial sums of shared rows
    unsigned long long keys[NW];    // per-warp LM argmax keys
    MergeScratch mg;
    float m[MAX_REP], l[MAX_REP], alpha[MAX_REP];
    int32_t flag;                   // broadcast of a counter-wait result
    int32_t abort;                  // set when this CTA must stop
    int32_t tok;                    // broadcast of the step's input token
    unsigned long long t_waited;    // trace: when the current task's wait completed
    unsigned long long t_ph[3];     // trace: input ready (prologue done / q,k,v arrived), compute done,
                                    // task body done (before the signal)
};

// Weights per 16-byte chunk of a packed row's codes.
template <int WT>
__host__ __device__ constexpr int wpc() {
    return WT == MK_W_INT8_ROW || WT == MK_W_FP8_E4M3 ? 16 : WT == MK_W_INT4_G128 ? 32 : 8;
}
// Weights with one fp16 scale per 128 consecutive k of a row.
template <int WT>
__host__ __device__ constexpr bool group_scaled() { return WT == MK_W_INT4_G128 || WT == MK_W_FP8_E4M3; }

template <int WT>
__host__ __device__ constexpr int rw_of() {  // rows per batch
    return gemv_batch_rows(WT);
}
// Trailer bytes per row in a slot: the row's scales (int8: one fp16, copied
// as one 16-byte chunk; int4 and fp8: one fp16 per 128 k of a row of at most
// INT4_MAX_ROW_K (int4) or MAX_K (fp8) codes).
template <int WT>
__host__ __device__ constexpr int trailer_of() {
    return WT == MK_W_INT8_ROW    ? 16
           : WT == MK_W_INT4_G128 ? 2 * INT4_MAX_ROW_K / 128
           : WT == MK_W_FP8_E4M3  ? 2 * MAX_K / 128
                                  : 0;
}

template <int WT>
__host__ __device__ constexpr int ring_slot_bytes() {
    return rw_of<WT>() * (64 / wpc<WT>()) * 512 + rw_of<WT>() * trailer_of<WT>();
}
template <int WT>
__host__ __device__ constexpr int ring_slots() {  // slots that fit beside the other shared memory
    return WT == MK_W_INT4_G128 || WT == MK_W_FP8_E4M3 ? 5 : 3;
}
static_assert(ring_slot_bytes<MK_W_INT8_ROW>() >= ffn_slot_lines(MK_W_INT8_ROW) * 512, "column lines of a slot");
static_assert(ring_slot_bytes<MK_W_INT4_G128>() >= ffn_slot_lines(MK_W_INT4_G128) * 512, "column lines of a slot");
static_assert(ring_slot_bytes<MK_W_FP8_E4M3>() >= ffn_slot_lines(MK_W_FP8_E4M3) * 512, "column lines of a slot");

struct WarpStream {
    int s, qi;               // cursor: step, next record of the CTA's table
    int q, nb, ngroups, grp;  // current phase: next batch of this warp, batches, batch step, first batch
    // row phase: rows, row stride, chunks per lane per row, trailer chunks, lane stride, lane offset, code bytes.
    // column phase (OP_FFN down projection): nrows = column blocks, row_bytes = block stride,
    // nl = 512-byte lines per block of this warp's rows, tlc = blocks per batch.
    int nrows, row_bytes, nl, tlc, S, lofs, code_bytes;
    const uint8_t* base;     // the task's first row (column phase: this warp's part of the first block)
    int si;                  // ring slot of the next issue
    int cols;                // 1 in a column phase
    int ffn_blocks;          // column blocks of the OP_FFN task whose row phase is current (0: none)
    const uint8_t* base2;    // that task's first down-projection column block
    bool done;
};

__host__ __device__ constexpr size_t up128(size_t v) { return (v + 127) / 128 * 128; }
__host__ __device__ constexpr size_t region0_bytes(int xs_floats) {
    return up128((size_t)xs_floats * 4 > sizeof(AttnScratch) ? (size_t)xs_floats * 4 : sizeof(AttnScratch));
}
__host__ __device__ constexpr size_t table_offset(int xs_floats) { return region0_bytes(xs_floats) + up128(sizeof(Shared)); }
__host__ __device__ constexpr size_t ring_offset(int xs_floats, int tab_cap) {
    return table_offset(xs_floats) + up128((size_t)tab_cap * sizeof(TaskRec));
}

struct Ctx {
    const VmParams* p;
    Shared* sh;
    AttnScratch* at;    // overlaps xs
    const TaskRec* tab; // this CTA's task records (shared memory)
    int nrec, q0;       // records in the table; queue index of the first
    uint8_t* ring;      // this warp's weight ring (ring_slots x ring_slot_bytes)
    WarpStream ws;      // this warp's weight-stream cursor (shared-memory ring)
    int rs;             // ring slot of the next batch to compute
    float* xs;          // the task's input vector (K floats, shared memory)
    float rstd;         // scale of xs applied when the fragments are loaded (RMSNorm)
    float xscale;       // step D of the input planes of an integer-dot task
    int tid, lane, warp;
    bool abort;
    int deferred;       // batches of this task that issued no copy: issued after the signal
    int cur;            // queue slot of the running task
};

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
static __device__ __forceinline__ bool wait_counters(Ctx& c, const TaskRec& t, int task_id, int step) {
    const VmParams& p = *c.p;
    if (c.tid == 0) {
        int ok = c.sh->abort ? 0 : 1;
        const uint32_t e = (uint32_t)(p.epoch0 + step);
        for (int w = 0; w < t.n_waits && ok; ++w) {
            const uint32_t* ctr = p.counters + (size_t)t.wait_ctr[w] * CTR_STRIDE;
            const uint32_t target = (uint32_t)t.wait_cnt[w] * (e + 1u - ((t.wait_prev >> w) & 1u));
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
        if (p.trace) c.sh->t_waited = gtimer();
    }
    bar_consumers();
    return c.sh->flag != 0;
}

// Tagged values carry their own completion.  The QKV rows are stored as one
// 64-bit word each: the fp32 result in the low half and a tag naming the
// (step, layer) that wrote it in the high half, with gpu-scope relaxed
// accesses, which are single-copy atomic for aligned 64-bit words.  A reader
// that sees the tag it expects therefore sees that step's value, with no
// counter, barrier or fence on the producer's side; it orders nothing else,
// so only data whose readers poll the tags travels this way.  Tags start at
// 1 after every reset of the synchronisation state (which zeroes the words).
__device__ __forceinline__ uint32_t qkv_tag(const VmParams& p, int step, int layer) {
    return 1u + (uint32_t)(p.epoch0 + step) * (uint32_t)p.L + (uint32_t)layer;
}
__device__ __forceinline__ void st_tagged(unsigned long long* a, float v, uint32_t tag) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(a),
                 "l"(((unsigned long long)tag << 32) | (unsigned long long)__float_as_uint(v))
                 : "memory");
}
__device__ __forceinline__ unsigned long long ld_tagged(const unsigned long long* a) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
    return v;
}
// Re-read the word at a until it carries `tag` (v holds a first read).
// False after an abort or when the watchdog expires (the error is raised).
__device__ __forceinline__ bool poll_tagged(const VmParams& p, const unsigned long long* a, uint32_t tag,
                                            unsigned long long& v, int task_id, int step) {
    if ((uint32_t)(v >> 32) == tag) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        v = ld_tagged(a);
        if ((uint32_t)(v >> 32) == tag) return true;
        if ((it & 63u) == 0u) {
            if (aborted(p)) return false;
            if (gtimer() - t0 > (uint64_t)p.watchdog_ns) {
                raise_error(p, DEV_TIMEOUT, (uint32_t)task_id, (uint32_t)step);
                return false;
            }
        }
    }
}
// Consumer barrier that also ANDs a predicate over the consumer threads.
__device__ __forceinline__ bool bar_consumers_and(bool ok) {
    int r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.s32 pi, %1, 0;\n\tbar.red.and.pred po, 1, %2, pi;\n\t"
        "selp.s32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((int)ok), "n"(NT)
        : "memory");
    return r != 0;
}

// The consumer barrier orders every consumer thread's writes of the task
// before the release-add by lane 0 of warp sw; a gpu-scope release is
// cumulative over writes that happen before it, so the waiting CTA's acquire
// sees them all.
__device__ __forceinline__ void signal_counter(Ctx& c, const TaskRec& t, int sw) {
    bar_consumers();
    if (c.warp == sw && c.lane == 0 && t.signal_ctr >= 0 && !c.sh->abort)
        red_release_add(c.p->counters + (size_t)t.signal_ctr * CTR_STRIDE, 1u);
}

// The warp that releases a task's signal.  A gpu-scope release waits for
// every weight copy its warp still has in flight (about one HBM latency
// right after the warp has run ahead into the next task), so the signal
// goes to the first warp of the last warp group: with batches dealt out
// round-robin that group has the fewest, and its copies usually land while
// the other groups finish.
__device__ __forceinline__ int signal_warp(const TaskRec& t, bool gemv) {
    if (!gemv) return NW - 1;
    const int g = t.wpr;
    return NW - g;
}

// ------------------------------------------------------------------ tokens
__device__ __forceinline__ unsigned long long key_tag(uint32_t epoch) {
    return (unsigned long long)(epoch + 1u);
}
// Order-preserving map of an fp32 value to u32.  -0 is first made +0, so the
// two zeros are equal keys and a tie between them goes to the lower index,
// as with a plain comparison of the values.
__device__ __forceinline__ uint32_t float_order(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ------------------------------------------------------------------ sampling
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
// as 1, 2, 3", SC 2011): ten rounds, each of two 32 x 32 -> 64-bit products
// whose halves are mixed with the other two words and the key; the key is
// bumped by two Weyl constants between rounds.  Counter (c0, c1, 0, 0); the
// first output word is returned.
__device__ __forceinline__ uint32_t philox_x0(uint32_t c0, uint32_t c1, uint32_t k0, uint32_t k1) {
    uint32_t c2 = 0u, c3 = 0u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return c0;
}
// Gumbel-max score of token i fed at position pos: logit / T - log(-log(u)),
// u = (2 (x >> 9) + 1) 2^-24 of the draw x for counter (i, pos); u is exact in
// fp32 and lies in (0, 1).  Out of line: it sits in the LM-head epilogue of
// the GEMV loop, which must keep its registers.
static __device__ __noinline__ float sample_score(float logit, uint32_t i, uint32_t pos, float inv_temp,
                                                  uint32_t k0, uint32_t k1) {
    const uint32_t x = philox_x0(i, pos, k0, k1);
    const float u = __uint2float_rn(2u * (x >> 9) + 1u) * 5.9604644775390625e-8f;
    return fmaf(logit, inv_temp, -logf(-logf(u)));
}
// 56-bit selection key of (value, index): the larger value wins, then the
// lower index.  Zero is below every key of a finite value.
__device__ __forceinline__ unsigned long long sel_key(float v, uint32_t idx) {
    return ((unsigned long long)float_order(v) << 24) | (unsigned long long)(0xFFFFFFu - idx);
}
__device__ __forceinline__ float sel_value(unsigned long long k) {
    const uint32_t u = (uint32_t)(k >> 24);
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}
__device__ __forceinline__ uint32_t sel_index(unsigned long long k) { return 0xFFFFFFu - (uint32_t)(k & 0xFFFFFFu); }

// The LM-head tasks' argmax of step s (once all of them have signalled).
static __device__ __forceinline__ int key_token(const VmParams& p, int step) {
    const unsigned long long k = __ldcg(p.key);
    if ((k >> 49) != key_tag((uint32_t)(p.epoch0 + step))) {
        raise_error(p, DEV_BAD_KEY, 0xFFFFFFFEu, (uint32_t)step);
        return -1;
    }
    return (int)((1u << KEY_IDX_BITS) - 1u - (uint32_t)(k & ((1ull << KEY_IDX_BITS) - 1ull)));
}

// Token selected at step s - 1 (s >= 1), once that step's token is final:
// written by its token-select task, else the LM-head tasks' argmax key.
static __device__ __forceinline__ int selected_token(const VmParams& p, int step) {
    if (p.tokw) {
        const unsigned long long k = __ldcg(p.tokw);
        if ((uint32_t)(k >> 32) != (uint32_t)(p.epoch0 + step)) {
            raise_error(p, DEV_BAD_KEY, 0xFFFFFFFEu, (uint32_t)step);
            return -1;
        }
        return (int)(uint32_t)k;
    }
    return key_token(p, step - 1);
}

// Token fed at step s.  Called by thread 0; broadcast through shared memory.
static __device__ __forceinline__ int step_token(const VmParams& p, int step) {
    int tok;
    if (p.forced) {
        tok = __ldg(p.forced + step);
    } else if (step == 0) {
        tok = p.pending >= 0 ? p.pending : (int)__ldcg((const unsigned int*)p.status + 3);
    } else {
        tok = selected_token(p, step);
        if (tok < 0) return -1;
    }
    if (tok < 0 || tok >= p.V) {
        raise_error(p, DEV_BAD_TOKEN, 0xFFFFFFFDu, (uint32_t)step);
        return -1;
    }
    return tok;
}

// ------------------------------------------------------------------ integer dot products
// int8 and int4 rows multiply their codes in 32-bit integers.  The GEMV input
// is held as a fixed-point copy X = rint(x / D), D a power of two with
// max|x| / D in [2^21, 2^22), stored as three byte planes: byte 0 and byte 1
// of X (unsigned) and byte 2 (signed), so that X = b2 2^16 + b1 2^8 + b0
// exactly.  X keeps 24 significant bits against max|x|, as many as fp32 keeps
// for the largest elements.  A 16-byte chunk of codes then takes dp4a
// instructions against the planes: int8 codes are signed bytes as stored, and
// each int4 nibble, masked into the high half of its byte, is the signed byte
// 16 q.  Every product and sum is exact, and one fp32 combination per row
// (int8) or per chunk (int4, whose group scale changes from chunk to chunk)
// rebuilds the dot product.
template <int WT>
__host__ __device__ constexpr bool idot_type() { return WT == MK_W_INT8_ROW || WT == MK_W_INT4_G128; }
// Byte planes of the input (24 bits).  Two planes (16 bits) against int4
// codes lose too much: the teacher-forced gate fails on the tiny model.
template <int WT>
__host__ __device__ constexpr int n_planes() { return 3; }
constexpr int PIECE_IT = 2;  // groups of 8 inputs a thread holds while the step D is found: K <= 8 NT PIECE_IT

// Byte offset of element k inside a plane.  int8 chunks take k in order.  An
// int4 code word holds 8 k with the even k in the low nibbles, so each 8 k of
// an int4 plane are stored as [k0 k2 k4 k6 | k1 k3 k5 k7]: the even word
// pairs with the low nibbles of the code word, the odd word with the high.
template <int WT>
__device__ __forceinline__ int plane_pos(int k) {
    if constexpr (WT == MK_W_INT4_G128) return (k & ~7) | ((k & 1) << 2) | ((k >> 1) & 3);
    else return k;
}
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {  // signed bytes of a, unsigned of b
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {  // signed bytes of both
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// 1 / D for a vector whose largest magnitude is m (1 when m is 0).  D = 2^E
// with m / D in [2^(8 NP - 3), 2^(8 NP - 2)), so |X| <= 2^(8 NP - 2) and the
// top byte of X (signed) is X >> 8 (NP - 1).
template <int NP>
__device__ __forceinline__ float fixed_inv_step(float m) {
    if (!(m > 0.f)) return 1.f;
    const int e = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127;  // floor(log2 m) for normal m
    const int E = max(-126, min(e - (8 * NP - 3), 126));
    return __uint_as_float((uint32_t)(127 - E) << 23);
}
// Planes of four values: P[p] holds byte p of a, b, c, d (in that order).
__device__ __forceinline__ void planes4(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t (&P)[3]) {
    const uint32_t ab_lo = __byte_perm(a, b, 0x5140), cd_lo = __byte_perm(c, d, 0x5140);  // [a0 b0 a1 b1]
    const uint32_t ab_hi = __byte_perm(a, b, 0x7362), cd_hi = __byte_perm(c, d, 0x7362);  // [a2 b2 a3 b3]
    P[0] = __byte_perm(ab_lo, cd_lo, 0x5410);
    P[1] = __byte_perm(ab_lo, cd_lo, 0x7632);
    P[2] = __byte_perm(ab_hi, cd_hi, 0x5410);
}
// Stores the planes of elements 8g .. 8g+7 (X: their fixed-point values) of a
// K-element vector whose plane p starts at pl + p K.
template <int WT>
__device__ __forceinline__ void put_planes8(uint8_t* pl, int K, int g, const int (&X)[8]) {
    uint32_t A[3], B[3];
    if constexpr (WT == MK_W_INT4_G128) {
        planes4(X[0], X[2], X[4], X[6], A);
        planes4(X[1], X[3], X[5], X[7], B);
    } else {
        planes4(X[0], X[1], X[2], X[3], A);
        planes4(X[4], X[5], X[6], X[7], B);
    }
#pragma unroll
    for (int p = 0; p < n_planes<WT>(); ++p) *(uint2*)(pl + (size_t)p * K + 8 * g) = make_uint2(A[p], B[p]);
}
// sum over a chunk pair of 4 words of 4-byte products, as an fp32 value of
// the fixed-point sum: S0 + 2^8 S1 + 2^16 S2
__device__ __forceinline__ float planes_combine(int s0, int s1, int s2) {
    return fmaf((float)s2, 65536.f, fmaf((float)s1, 256.f, (float)s0));
}
template <int NP>
__device__ __forceinline__ float planes_sum(const int (&s)[NP]) {
    if constexpr (NP == 3) return planes_combine(s[0], s[1], s[2]);
    else return fmaf((float)s[1], 256.f, (float)s[0]);
}
// The lane's partial dot product of one row, in units of D: xp holds the
// planes of the lane's chunks L + S*j (int8: one uint4 per plane; int4: two,
// plane p at xp[j][2p], xp[j][2p + 1]).  int4 chunks carry their group
// scale in sc[j]; int8 takes its row scale after the warp reduction.
template <int WT, int NG>
__device__ __forceinline__ float chunks_idot(const uint4 (&w)[NG], const float (&sc)[NG],
                                             const uint4 (&xp)[NG][WT == MK_W_INT4_G128 ? 2 * n_planes<WT>() : 3]) {
    if constexpr (WT == MK_W_INT8_ROW) {
        int s[2][3] = {{0, 0, 0}, {0, 0, 0}};  // two sets: shorter dependency chains
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const uint32_t wv[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
            const uint32_t p0[4] = {xp[j][0].x, xp[j][0].y, xp[j][0].z, xp[j][0].w};
            const uint32_t p1[4] = {xp[j][1].x, xp[j][1].y, xp[j][1].z, xp[j][1].w};
            const uint32_t p2[4] = {xp[j][2].x, xp[j][2].y, xp[j][2].z, xp[j][2].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                s[j & 1][0] = dp4a_su(wv[i], p0[i], s[j & 1][0]);
                s[j & 1][1] = dp4a_su(wv[i], p1[i], s[j & 1][1]);
                s[j & 1][2] = dp4a_ss(wv[i], p2[i], s[j & 1][2]);
            }
        }
        return planes_combine(s[0][0] + s[1][0], s[0][1] + s[1][1], s[0][2] + s[1][2]);
    } else {  // int4: lo = 16 q of the even k, hi = 16 q of the odd k
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const uint32_t wv[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
            constexpr int NP = n_planes<WT>();
            int s[NP];
#pragma unroll
            for (int p = 0; p < NP; ++p) s[p] = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t lo = (wv[i] << 4) & 0xF0F0F0F0u, hi = wv[i] & 0xF0F0F0F0u;
#pragma unroll
                for (int p = 0; p < NP; ++p) {  // the top plane is signed
                    const uint4 A = xp[j][2 * p + (i >> 1)];
                    const uint32_t ev = (i & 1) ? A.z : A.x, od = (i & 1) ? A.w : A.y;
                    if (p < NP - 1) {
                        s[p] = dp4a_su(lo, ev, s[p]);
                        s[p] = dp4a_su(hi, od, s[p]);
                    } else {
                        s[p] = dp4a_ss(lo, ev, s[p]);
                        s[p] = dp4a_ss(hi, od, s[p]);
                    }
                }
            }
            acc = fmaf(sc[j], planes_sum<NP>(s), acc);
        }
        return acc * 0.0625f;
    }
}

// ------------------------------------------------------------------ GEMV inputs
// Position (in floats) of float4 unit u of a K-float input vector in c.xs.
// Unit u belongs to the 16-byte weight chunk u >> lq4 of a row (2^lq4 units
// per chunk); the units of equal rank in their chunk form one plane, so the
// 32 lanes of a warp, which read the same rank of 32 consecutive chunks,
// touch 512 consecutive bytes (no bank conflicts).
__device__ __forceinline__ int xs_pos(int u, int K, int lq4) {
    const int nch = K >> (lq4 + 2);
    return ((u & ((1 << lq4) - 1)) * nch + (u >> lq4)) * 4;
}
// Each prologue writes the task's input vector into c.xs with all consumer
// threads and ends with a consumer barrier: K floats in planes (IW = 0), or
// for an integer-dot task (IW = the weight type) the three byte planes of its
// fixed-point copy and the step D in c.xscale.  An integer-dot prologue keeps
// its inputs in registers (groups 8g .. 8g+7 for g = tid + it NT) until the
// block-wide max |x| fixes D.

// The planes of the kept inputs times f0, given m = max |kept input|.
template <int IW>
__device__ __forceinline__ void write_planes(Ctx& c, const float (&keep)[PIECE_IT][8], int K, float f0, float m) {
    const float inv = fixed_inv_step<n_planes<IW>()>(m * f0);
    const float f = f0 * inv;
#pragma unroll
    for (int it = 0; it < PIECE_IT; ++it) {
        const int g = c.tid + it * NT;
        if (g < (K >> 3)) {
            int X[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) X[i] = __float2int_rn(keep[it][i] * f);
            put_planes8<IW>((uint8_t*)c.xs, K, g, X);
        }
    }
    c.xscale = 1.f / inv;  // a power of two: exact
    bar_consumers();
}
// Block-wide max of the threads' m (one consumer barrier); every thread gets it.
__device__ __forceinline__ float block_max(Ctx& c, float m) {
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (c.lane == 0) c.sh->nmax[c.warp] = m;
    bar_consumers();
    float r = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) r = fmaxf(r, c.sh->nmax[w]);
    return r;
}

// RMSNorm(x) * gain, x from the residual stream or (layer 0) an embedding row.
// The gain loads are issued together with the x loads (one memory round trip).
template <int BASE, int IW>
static __device__ __forceinline__ void prologue_rmsnorm(Ctx& c, const float* x, const uint16_t* emb_row, const uint16_t* gain, int K,
                                 float eps, int lq4) {
    float ss = 0.f, mx = 0.f;
    auto load8 = [&](int g, float (&v)[8]) {  // v = x[8g, 8g + 8) * gain, ss += x^2
        const uint4 graw = __ldg((const uint4*)(gain + 8 * g));
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
        for (int i = 0; i < 4; ++i) {  // x * gain now; the common 1/rms factor is applied later
            v[2 * i] *= base_to_f32<BASE>(gv[i] & 0xFFFFu);
            v[2 * i + 1] *= base_to_f32<BASE>(gv[i] >> 16);
        }
    };
    float keep[IW ? PIECE_IT : 1][8];
    if constexpr (IW == 0) {
        for (int g = c.tid; g < (K >> 3); g += NT) {
            float v[8];
            load8(g, v);
            *(float4*)(c.xs + xs_pos(2 * g, K, lq4)) = make_float4(v[0], v[1], v[2], v[3]);
            *(float4*)(c.xs + xs_pos(2 * g + 1, K, lq4)) = make_float4(v[4], v[5], v[6], v[7]);
        }
    } else {
#pragma unroll
        for (int it = 0; it < PIECE_IT; ++it) {
            const int g = c.tid + it * NT;
            if (g < (K >> 3)) {
                load8(g, keep[it]);
#pragma unroll
                for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(keep[it][i]));
            }
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
        if constexpr (IW != 0) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    }
    if (c.lane == 0) {
        c.sh->norm[c.warp] = ss;
        if constexpr (IW != 0) c.sh->nmax[c.warp] = mx;
    }
    bar_consumers();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) tot += c.sh->norm[w];
    c.rstd = rsqrtf(tot / (float)K + eps);  // applied to the fragments by gemv_rows
    if constexpr (IW != 0) {
        float m = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) m = fmaxf(m, c.sh->nmax[w]);
        write_planes<IW>(c, keep, K, c.rstd, m);
    }
}

// Merge the split-KV partials of every query head into the attention output:
// o = sum_c e^(m_c - M) l_c a_c / sum_c e^(m_c - M) l_c, M = max_c m_c, where
// a_c is chunk c's output normalised by its own sum l_c.
// One pass with a running maximum: each thread reads, for its 8 outputs,
// every chunk's (max, sum) and partial accumulators itself (up to 8 chunks'
// loads in flight at once) and rescales as the maximum grows, so the merge
// costs about one round trip to L2 and no block barrier.
__device__ __forceinline__ void merge8(const VmParams& p, int g, float (&o)[8]) {
    const int C = p.C;
    const int hq = (8 * g) / p.hd, d0 = (8 * g) % p.hd;
    const int cp = blockIdx.x % PART_COPIES;  // this CTA's copy of the partials
    const float* ml = p.part_ml + ((size_t)cp * p.Hq + hq) * C * 2;
    const uint16_t* base = p.part_acc + ((size_t)cp * p.Hq + hq) * C * p.hd + d0;
    float M = -3.0e38f, den = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = 0.f;
    for (int c0 = 0; c0 < C; c0 += 8) {
        float mm[8], ll[8];
        uint4 a[8];  // eight fp16 accumulators
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int ch = min(c0 + k, C - 1);
            const float2 v = __ldcg((const float2*)(ml + 2 * ch));  // (max, sum) in one load
            mm[k] = v.x;
            ll[k] = v.y;
            a[k] = __ldcg((const uint4*)(base + (size_t)ch * p.hd));
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (c0 + k >= C) break;
            const float Mn = fmaxf(M, mm[k]);
            const float r = expf(M - Mn), w = expf(mm[k] - Mn);
            M = Mn;
            const float wl = w * ll[k];  // the chunk's weight: its partials are acc / l
            den = fmaf(den, r, wl);
            const uint32_t h4[4] = {a[k].x, a[k].y, a[k].z, a[k].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                o[2 * i] = fmaf(o[2 * i], r, wl * half_bits_to_f32(h4[i] & 0xFFFFu));
                o[2 * i + 1] = fmaf(o[2 * i + 1], r, wl * half_bits_to_f32(h4[i] >> 16));
            }
        }
    }
    const float inv = 1.f / den;
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] *= inv;
}
template <int IW>
static __device__ __forceinline__ void prologue_attention(Ctx& c, int lq4) {
    const VmParams& p = *c.p;
    c.rstd = 1.f;
    if constexpr (IW == 0) {
        for (int g = c.tid; g < (p.q_dim >> 3); g += NT) {
            float o[8];
            merge8(p, g, o);
            *(float4*)(c.xs + xs_pos(2 * g, p.q_dim, lq4)) = make_float4(o[0], o[1], o[2], o[3]);
            *(float4*)(c.xs + xs_pos(2 * g + 1, p.q_dim, lq4)) = make_float4(o[4], o[5], o[6], o[7]);
        }
        bar_consumers();
    } else {
        float keep[PIECE_IT][8], mx = 0.f;
#pragma unroll
        for (int it = 0; it < PIECE_IT; ++it) {
            const int g = c.tid + it * NT;
            if (g < (p.q_dim >> 3)) {
                merge8(p, g, keep[it]);
#pragma unroll
                for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(keep[it][i]));
            }
        }
        write_planes<IW>(c, keep, p.q_dim, 1.f, block_max(c, mx));
    }
}

// OP_MERGE: the split-KV merge of KV group g's query heads, written once to
// att[g * rep * hd ...] for every O task to read.  Each thread produces four
// outputs from all chunks, with the running maximum of prologue_attention.
static __device__ __forceinline__ void merge_task(Ctx& c, const TaskRec& t) {
    const VmParams& p = *c.p;
    const int C = p.C, rep = p.Hq / p.Hkv, g = t.row0;
    for (int u = c.tid; u < rep * (p.hd >> 2); u += NT) {
        const int hq = g * rep + (4 * u) / p.hd, d0 = (4 * u) % p.hd;
        const int cp = blockIdx.x % PART_COPIES;
        const float* ml = p.part_ml + ((size_t)cp * p.Hq + hq) * C * 2;
        const uint16_t* base = p.part_acc + ((size_t)cp * p.Hq + hq) * C * p.hd + d0;
        float M = -3.0e38f, den = 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c0 = 0; c0 < C; c0 += 8) {
            float2 mlv[8];
            uint2 a[8];  // four fp16 accumulators
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int ch = min(c0 + k, C - 1);
                mlv[k] = __ldcg((const float2*)(ml + 2 * ch));
                a[k] = __ldcg((const uint2*)(base + (size_t)ch * p.hd));
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (c0 + k >= C) break;
                const float Mn = fmaxf(M, mlv[k].x);
                const float r = expf(M - Mn), w = expf(mlv[k].x - Mn);
                M = Mn;
                const float wl = w * mlv[k].y;  // the chunk's weight: its partials are acc / l
                den = fmaf(den, r, wl);
                o.x = fmaf(o.x, r, wl * half_bits_to_f32(a[k].x & 0xFFFFu));
                o.y = fmaf(o.y, r, wl * half_bits_to_f32(a[k].x >> 16));
                o.z = fmaf(o.z, r, wl * half_bits_to_f32(a[k].y & 0xFFFFu));
                o.w = fmaf(o.w, r, wl * half_bits_to_f32(a[k].y >> 16));
            }
        }
        const float inv = 1.f / den;
        const float4 r = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
#pragma unroll
        for (int k = 0; k < PART_COPIES; ++k) *(float4*)(p.att + (size_t)k * p.q_dim + (size_t)hq * p.hd + d0) = r;
    }
}

// O prologue when merge tasks ran: the merged attention output, copied from
// att into c.xs (planes).
template <int IW>
static __device__ __forceinline__ void prologue_att_copy(Ctx& c, int lq4) {
    const VmParams& p = *c.p;
    const float* att = p.att + (size_t)(blockIdx.x % PART_COPIES) * p.q_dim;
    c.rstd = 1.f;
    if constexpr (IW == 0) {
        for (int u = c.tid; u < (p.q_dim >> 2); u += NT)
            *(float4*)(c.xs + xs_pos(u, p.q_dim, lq4)) = __ldcg((const float4*)(att + 4 * u));
        bar_consumers();
    } else {
        float keep[PIECE_IT][8], mx = 0.f;
#pragma unroll
        for (int it = 0; it < PIECE_IT; ++it) {
            const int g = c.tid + it * NT;
            if (g < (p.q_dim >> 3)) {
                const float4 a = __ldcg((const float4*)(att + 8 * g)), b = __ldcg((const float4*)(att + 8 * g + 4));
                keep[it][0] = a.x; keep[it][1] = a.y; keep[it][2] = a.z; keep[it][3] = a.w;
                keep[it][4] = b.x; keep[it][5] = b.y; keep[it][6] = b.z; keep[it][7] = b.w;
#pragma unroll
                for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(keep[it][i]));
            }
        }
        write_planes<IW>(c, keep, p.q_dim, 1.f, block_max(c, mx));
    }
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

// The lane's partial dot product over its chunks of one row: w[j] is chunk
// L + S*j of the row's codes, xr holds the matching input values as fp32
// pairs (WPC/2 pairs per chunk).  int4 and fp8 chunks carry their group-128
// scale in sc[j] (a chunk of 32 or 16 codes never straddles a group).
template <int WT, int NG>
__device__ __forceinline__ float chunks_dot(const uint4 (&w)[NG], const float (&sc)[NG],
                                            const unsigned long long (&xr)[NG * wpc<WT>() / 2]) {
    constexpr int HP = wpc<WT>() / 2;  // pairs per chunk
    unsigned long long a0 = 0ull, a1 = 0ull;
    float f0 = 0.f, f1 = 0.f;
#pragma unroll
    for (int j = 0; j < NG; ++j) {
        const uint32_t wv[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
        if constexpr (WT == MK_W_BF16 || WT == MK_W_FP16) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                unsigned long long wp;
                if constexpr (WT == MK_W_BF16) {
                    wp = pack2(__uint_as_float(wv[i] << 16), __uint_as_float(wv[i] & 0xFFFF0000u));
                } else {
                    const float2 f = __half22float2(*(const __half2*)&wv[i]);
                    wp = pack2(f.x, f.y);
                }
                if (i & 1) a1 = ffma2(wp, xr[j * HP + i], a1);
                else a0 = ffma2(wp, xr[j * HP + i], a0);
            }
        } else if constexpr (WT == MK_W_INT8_ROW) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t u = wv[i] ^ 0x80808080u;
                a0 = ffma2(pack2(i8_to_f32(u, 0), i8_to_f32(u, 1)), xr[j * HP + 2 * i], a0);
                a1 = ffma2(pack2(i8_to_f32(u, 2), i8_to_f32(u, 3)), xr[j * HP + 2 * i + 1], a1);
            }
        } else if constexpr (WT == MK_W_FP8_E4M3) {
            unsigned long long pa = 0ull, pb = 0ull;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                pa = ffma2(e4m3x2_pair(wv[i]), xr[j * HP + 2 * i], pa);
                pb = ffma2(e4m3x2_pair(wv[i] >> 16), xr[j * HP + 2 * i + 1], pb);
            }
            if (j & 1) f1 = fmaf(sc[j], sum2(pa) + sum2(pb), f1);
            else f0 = fmaf(sc[j], sum2(pa) + sum2(pb), f0);
        } else {  // int4
            unsigned long long pa = 0ull, pb = 0ull;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t u = wv[i] ^ 0x88888888u;
                pa = ffma2(pack2(i4_to_f32(u, 0), i4_to_f32(u, 1)), xr[j * HP + 4 * i], pa);
                pb = ffma2(pack2(i4_to_f32(u, 2), i4_to_f32(u, 3)), xr[j * HP + 4 * i + 1], pb);
                pa = ffma2(pack2(i4_to_f32(u, 4), i4_to_f32(u, 5)), xr[j * HP + 4 * i + 2], pa);
                pb = ffma2(pack2(i4_to_f32(u, 6), i4_to_f32(u, 7)), xr[j * HP + 4 * i + 3], pb);
            }
            if (j & 1) f1 = fmaf(sc[j], sum2(pa) + sum2(pb), f1);
            else f0 = fmaf(sc[j], sum2(pa) + sum2(pb), f0);
        }
    }
    if constexpr (group_scaled<WT>()) return f0 + f1;
    else return sum2(a0) + sum2(a1);
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

// ------------------------------------------------------------------ weight stream
// Each warp streams the weight rows it will multiply through a private ring
// of NB shared-memory slots with cp.async (16 bytes per lane per copy), NB - 1
// batches ahead of the batch it computes.  The warp's sequence of batches is
// fixed by the schedule (tasks in queue order, for each GEMV task the batches
// q = grp, grp + ngroups, ... of its warp group), so the copies run ahead
// across counter waits and across tasks: a task usually starts with its first
// batches already on chip.  A slot holds RW = rw_of<WT>() rows (2 for 16-bit
// and fp8 codes, 4 for int8 and int4): the lane's chunks j of each row at
// [(r * NGM + j) * 512 + lane * 16] and the row's quantisation trailer
// (scales) at [RW * NGM * 512 + r * TRAILER], TRAILER = trailer_of<WT>().

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gsrc)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Move the cursor to this warp's next batch; false at the end of the launch.
template <int WT>
__device__ __forceinline__ bool stream_next(const Ctx& c, WarpStream& w) {
    const VmParams& p = *c.p;
    for (;;) {
        if (w.q < w.nb) return true;
        if (w.ffn_blocks) {  // the row phase of an OP_FFN task is done: its column blocks follow
            const int R = p.d / NW;  // output rows of this warp
            const int SL = ffn_slot_lines(p.wdtype);
            w.cols = 1;
            w.nl = R / 32;                                      // 512-byte lines per block of this warp's rows
            w.tlc = w.nl <= SL ? (SL / w.nl) * w.nl : SL;       // lines per batch (whole blocks, or a part)
            w.nrows = w.ffn_blocks * w.nl;                      // lines of the task
            w.row_bytes = p.d * 16;
            w.base = w.base2 + (size_t)c.warp * R * 16;
            w.lofs = c.lane * 16;
            w.nb = (w.nrows + w.tlc - 1) / w.tlc;
            w.q = 0;
            w.ngroups = 1;
            w.ffn_blocks = 0;
            continue;
        }
        if (w.qi >= c.nrec) {
            if (++w.s >= p.n_steps) return false;
            w.qi = 0;
        }
        const TaskRec& t = c.tab[w.qi++];
        const int op = t.op;
        w.nb = 0;
        w.q = 0;
        w.cols = 0;
        if (!(op == OP_QKV || op == OP_O || op == OP_GU || op == OP_DOWN || op == OP_FFN ||
              (op == OP_LM && !p.skip_lm)))
            continue;
        if (op == OP_FFN) {
            const int BU = ffn_block(p.wdtype);
            w.ffn_blocks = t.nrows / (2 * BU);
            w.base2 = p.w + p.layer_bytes * t.layer + p.l_down + (size_t)(t.row0 / (2 * BU)) * p.d * 16;
        }
        const int K = t.K, g = t.wpr;
        const int L = (c.warp % g) * 32 + c.lane;
        w.nrows = t.nrows;
        w.row_bytes = (int)t.row_bytes16 * 16;
        w.ngroups = NW / g;
        w.grp = c.warp / g;
        w.S = 32 * g;
        const int code_bytes = p.wdtype == MK_W_INT8_ROW || p.wdtype == MK_W_FP8_E4M3 ? K
                               : p.wdtype == MK_W_INT4_G128                             ? K / 2
                                                                                        : 2 * K;
        const int CHc = code_bytes / 16;
        w.nl = L < CHc ? (CHc - L + w.S - 1) / w.S : 0;  // this lane's chunks of a row
        w.tlc = (w.row_bytes - code_bytes) / 16;
        w.base = p.w + (size_t)t.w_off16 * 16;
        w.lofs = L * 16;
        w.code_bytes = code_bytes;
        w.nb = (w.nrows + rw_of<WT>() - 1) / rw_of<WT>();
        w.q = w.grp;
    }
}

// Issue the copies of the cursor's batch into ring slot w.si (or an empty
// group after the last batch), then advance.
template <int WT>
__device__ __forceinline__ void stream_issue(Ctx& c) {
    constexpr int NGM = 64 / wpc<WT>();
    WarpStream& w = c.ws;
    const int lane = c.lane;
    if (!w.done && stream_next<WT>(c, w)) {
        uint8_t* slot = c.ring + (size_t)w.si * ring_slot_bytes<WT>() + lane * 16;
        const int64_t jstep = (int64_t)w.S * 16;
        if (w.cols) {  // lines q*tlc .. of the task: line i is line i % nl of block i / nl
            int seg, m = 0, lines;
            if constexpr (WT == MK_W_BF16 || WT == MK_W_FP16) {  // whole blocks: tlc / nl of them
                seg = w.q * (16 / w.nl);
                lines = min(w.tlc, w.nrows - w.q * w.tlc);
            } else {
                if (w.tlc >= w.nl) {  // whole blocks per batch
                    seg = w.q * (w.tlc / w.nl);
                } else {              // a block spans nl / tlc batches
                    const int bpb = w.nl / w.tlc;
                    seg = w.q / bpb;
                    m = (w.q - seg * bpb) * w.tlc;
                }
                lines = min(w.tlc, w.nrows - w.q * w.tlc);
            }
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                if (k < lines) cp_async16(slot + k * 512, w.base + (size_t)seg * w.row_bytes + m * 512 + w.lofs);
                if (++m == w.nl) {
                    m = 0;
                    ++seg;
                }
            }
        }
        constexpr int RW = rw_of<WT>(), TRAILER = trailer_of<WT>();
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            if (w.cols) break;
            const int row = w.q * RW + r;
            if (row < w.nrows) {
                const uint8_t* rowp = w.base + (int64_t)row * w.row_bytes;
                const uint8_t* src = rowp + w.lofs;
#pragma unroll
                for (int j = 0; j < NGM; ++j)
                    if (j < w.nl) cp_async16(slot + (r * NGM + j) * 512, src + j * jstep);
                if constexpr (!(WT == MK_W_BF16 || WT == MK_W_FP16)) {
                    if (lane < w.tlc)  // the row's scales follow its codes
                        cp_async16(slot + RW * NGM * 512 + r * TRAILER, rowp + w.code_bytes + lane * 16);
                }
            }
        }
        w.q += w.ngroups;
        if (++w.si == ring_slots<WT>()) w.si = 0;
    } else {
        w.done = true;
    }
    cp_async_commit();
}

// Wait until at most n (0 <= n <= N) of the warp's copy groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait_upto(int n) {
    if constexpr (N == 0) {
        cp_async_wait<0>();
    } else {
        if (n >= N) cp_async_wait<N>();
        else cp_async_wait_upto<N - 1>(n);
    }
}

// Wait for the ring slot of the batch about to be computed.  NB - 1 batches
// run ahead.  A batch may defer its issue until after the task's signal
// (defer = true), which keeps the copy's back-pressure off the signal's path:
// a task's last batch always does, and so does every batch of a QKV task
// whose warp computes at most NB - 1 batches of it (each of them was issued
// before the task began).  Callers never follow a deferred batch with one that
// issues, so with k issues pending NB - 1 - k groups follow the current one.
template <int WT>
__device__ __forceinline__ void ring_acquire(Ctx& c, bool defer) {
    constexpr int NB = ring_slots<WT>();
    if (defer) {
        ++c.deferred;
        cp_async_wait_upto<NB - 2>(NB - 1 - c.deferred);
    } else {
        stream_issue<WT>(c);
        cp_async_wait<NB - 1>();
    }
    __syncwarp();
}

// ------------------------------------------------------------------ fused FFN
// Residual buffer holding the input of `layer` (with the fused FFN the two
// buffers alternate by layer; otherwise there is one).
__device__ __forceinline__ float* xbuf(const VmParams& p, int layer) {
    return p.x + (p.fused ? (size_t)(layer & 1) * p.d : 0);
}
// x_mid = x + attention output of the running layer, written by O and read by
// the FFN side.  It has a buffer of its own so that O never overwrites the
// layer input that QKV tasks elsewhere may still be reading.
__device__ __forceinline__ float* xmid(const VmParams& p) { return p.x + 2 * (size_t)p.d; }
// SwiGLU outputs of the running OP_FFN task (the merge scratch is idle then).
static_assert(sizeof(MergeScratch) >= FFN_MAX_UNITS * sizeof(float), "OP_FFN SwiGLU outputs");
__device__ __forceinline__ float* ffn_h(Ctx& c) { return reinterpret_cast<float*>(&c.sh->mg); }

__device__ __forceinline__ void red_add_f32(float* p, float v) {
    asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// Down projection of an OP_FFN task: y[r] = sum over the task's hidden units
// u of Wdown[r][u] * h[u], for every output row r, added into the next
// layer's residual buffer (which O initialised to x_mid).  W_down is packed in
// 16-byte column chunks of BU units (8 bf16/fp16, 16 int8/fp8 or 32 int4 codes):
// block b holds, for r = 0..d-1, the codes of Wdown[r][BU b .. BU (b+1)).
// Warp w owns rows [w*R, (w+1)*R), R = d/8, so a block gives it NL = R/32
// lines of 512 bytes: lane l of line m holds row w*R + 32m + l.  The lane
// keeps one accumulator per line and ends with one red.add per row.  A ring
// batch holds SEGB whole blocks, or (when a block has more lines than a slot
// holds) the part bb of a block.  Scales of quantised codes follow the
// blocks: one per row for int8 (applied before the red.add), one per row and
// 128-unit group for int4 and fp8 (applied to each block's dot product).
template <int WT>
__device__ __forceinline__ unsigned long long col_pair(uint32_t word, int i) {
    if constexpr (WT == MK_W_BF16) {
        (void)i;
        return pack2(__uint_as_float(word << 16), __uint_as_float(word & 0xFFFF0000u));
    } else {
        const float2 f = __half22float2(*(const __half2*)&word);
        (void)i;
        return pack2(f.x, f.y);
    }
}
// The BU inputs of a column block as fp32 pairs (loaded once per block).
template <int WT>
__device__ __forceinline__ void load_h(const float* hs, unsigned long long (&hx)[ffn_block(WT) / 2]) {
#pragma unroll
    for (int i = 0; i < ffn_block(WT) / 4; ++i) {
        const float4 h = *(const float4*)(hs + 4 * i);
        hx[2 * i] = pack2(h.x, h.y);
        hx[2 * i + 1] = pack2(h.z, h.w);
    }
}
// Accumulate one 16-byte column chunk times its inputs into the packed pair
// accumulator a.
template <int WT>
__device__ __forceinline__ void chunk_fma(const uint4 w, const unsigned long long (&hx)[ffn_block(WT) / 2],
                                          unsigned long long& a) {
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
    if constexpr (WT == MK_W_BF16 || WT == MK_W_FP16) {
#pragma unroll
        for (int i = 0; i < 4; ++i) a = ffma2(col_pair<WT>(wv[i], i), hx[i], a);
    } else if constexpr (WT == MK_W_INT8_ROW) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t u = wv[i] ^ 0x80808080u;
            a = ffma2(pack2(i8_to_f32(u, 0), i8_to_f32(u, 1)), hx[2 * i], a);
            a = ffma2(pack2(i8_to_f32(u, 2), i8_to_f32(u, 3)), hx[2 * i + 1], a);
        }
    } else if constexpr (WT == MK_W_FP8_E4M3) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            a = ffma2(e4m3x2_pair(wv[i]), hx[2 * i], a);
            a = ffma2(e4m3x2_pair(wv[i] >> 16), hx[2 * i + 1], a);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t u = wv[i] ^ 0x88888888u;
            a = ffma2(pack2(i4_to_f32(u, 0), i4_to_f32(u, 1)), hx[4 * i], a);
            a = ffma2(pack2(i4_to_f32(u, 2), i4_to_f32(u, 3)), hx[4 * i + 1], a);
            a = ffma2(pack2(i4_to_f32(u, 4), i4_to_f32(u, 5)), hx[4 * i + 2], a);
            a = ffma2(pack2(i4_to_f32(u, 6), i4_to_f32(u, 7)), hx[4 * i + 3], a);
        }
    }
}

// 16-bit weights: SEGB = 16 / NL whole blocks per batch and packed pair
// accumulators, no scales.
template <int WT, int NL>
__device__ __forceinline__ void ffn_cols16(Ctx& c, const TaskRec& t, int layer) {
    const VmParams& p = *c.p;
    constexpr int NB = ring_slots<WT>();
    constexpr int SEGB = 16 / NL;
    const int kc = t.nrows / (2 * ffn_block(WT));
    const int nb2 = (kc + SEGB - 1) / SEGB;
    const float* hs = ffn_h(c);
    unsigned long long acc[NL];
#pragma unroll
    for (int m = 0; m < NL; ++m) acc[m] = 0ull;
    for (int b = 0; b < nb2; ++b) {
        ring_acquire<WT>(c, b == nb2 - 1);
        const uint8_t* slot = c.ring + (size_t)c.rs * ring_slot_bytes<WT>() + c.lane * 16;
#pragma unroll
        for (int sg = 0; sg < SEGB; ++sg) {
            const int seg = b * SEGB + sg;
            if (seg < kc) {
                unsigned long long hx[4];
                load_h<WT>(hs + seg * 8, hx);
#pragma unroll
                for (int m = 0; m < NL; ++m) chunk_fma<WT>(*(const uint4*)(slot + (sg * NL + m) * 512), hx, acc[m]);
            }
        }
        __syncwarp();  // the slot is reused by a later issue of this warp
        if (++c.rs == NB) c.rs = 0;
    }
    float* xo = xbuf(p, layer + 1) + (size_t)c.warp * (p.d / NW) + c.lane;
#pragma unroll
    for (int m = 0; m < NL; ++m) red_add_f32(xo + 32 * m, sum2(acc[m]));
}

// int8 and int4 codes: integer dot products against byte planes of the
// task's SwiGLU outputs (a fixed-point copy with step D_h, built here in the
// input region, which every row batch of the task has finished with).  Each
// lane keeps one int32 sum per line and plane; int8 combines them once per
// row, int4 at each change of 128-unit group (its scale changes there).
static_assert(3 * FFN_MAX_UNITS <= sizeof(AttnScratch), "planes of an OP_FFN task's SwiGLU outputs in the input region");
template <int WT, int NL>
__device__ __forceinline__ void ffn_cols_idot(Ctx& c, const TaskRec& t, int layer) {
    const VmParams& p = *c.p;
    constexpr int NB = ring_slots<WT>();
    constexpr int BU = ffn_block(WT), SL = ffn_slot_lines(WT);
    constexpr int CB = WT == MK_W_INT4_G128 ? 2 : 1;  // 16-byte words of a block per plane
    constexpr int NP = n_planes<WT>();
    const int kc = t.nrows / (2 * BU);
    const int units = kc * BU;
    const float* hs = ffn_h(c);
    float mx = 0.f;
    for (int u = c.tid; u < units; u += NT) mx = fmaxf(mx, fabsf(hs[u]));
    const float inv = fixed_inv_step<NP>(block_max(c, mx));
    uint8_t* hp = (uint8_t*)c.xs;
    for (int u = c.tid; u < units; u += NT) {
        const int X = __float2int_rn(hs[u] * inv);
        const int q = plane_pos<WT>(u);
#pragma unroll
        for (int pp = 0; pp < NP; ++pp) hp[pp * units + q] = (uint8_t)(X >> (8 * pp));
    }
    bar_consumers();
    const float hstep = 1.f / inv;
    const int r0 = c.warp * (p.d / NW) + c.lane;  // row of line 0 of this lane
    const uint16_t* scales = (const uint16_t*)(p.w + p.layer_bytes * layer + p.l_down + (size_t)p.d * (p.F / BU) * 16);
    const int u0 = t.row0 / 2;  // first hidden unit of the task
    int S[NL][NP];
    float acc[NL], sc[NL];
    int sc_group = -1;
#pragma unroll
    for (int m = 0; m < NL; ++m) {
#pragma unroll
        for (int pp = 0; pp < NP; ++pp) S[m][pp] = 0;
        acc[m] = 0.f;
        sc[m] = 0.f;
    }
    uint4 hb[NP * CB];  // the planes of the current block
    auto flush = [&]() {  // int4: the group's sums, scaled
#pragma unroll
        for (int m = 0; m < NL; ++m) {
            acc[m] = fmaf(sc[m], planes_sum<NP>(S[m]), acc[m]);
#pragma unroll
            for (int pp = 0; pp < NP; ++pp) S[m][pp] = 0;
        }
    };
    auto begin_block = [&](int seg) {
        if constexpr (WT == MK_W_INT4_G128) {
            const int g = (u0 + seg * BU) >> 7;
            if (g != sc_group) {
                if (sc_group >= 0) flush();
                sc_group = g;
#pragma unroll
                for (int m = 0; m < NL; ++m) sc[m] = half_bits_to_f32(__ldg(scales + (size_t)g * p.d + r0 + 32 * m));
            }
        }
#pragma unroll
        for (int q = 0; q < NP * CB; ++q)
            hb[q] = *(const uint4*)(hp + (size_t)(q / CB) * units + (size_t)seg * BU + 16 * (q % CB));
    };
    auto line = [&](int m, const uint8_t* src) {
        const uint4 wq = *(const uint4*)src;
        const uint32_t wv[4] = {wq.x, wq.y, wq.z, wq.w};
        if constexpr (WT == MK_W_INT8_ROW) {
            const uint32_t p0[4] = {hb[0].x, hb[0].y, hb[0].z, hb[0].w};
            const uint32_t p1[4] = {hb[1].x, hb[1].y, hb[1].z, hb[1].w};
            const uint32_t p2[4] = {hb[2].x, hb[2].y, hb[2].z, hb[2].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                S[m][0] = dp4a_su(wv[i], p0[i], S[m][0]);
                S[m][1] = dp4a_su(wv[i], p1[i], S[m][1]);
                S[m][2] = dp4a_ss(wv[i], p2[i], S[m][2]);
            }
        } else {  // 16 q of the even units (low nibbles) and of the odd units
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t lo = (wv[i] << 4) & 0xF0F0F0F0u, hi = wv[i] & 0xF0F0F0F0u;
#pragma unroll
                for (int q = 0; q < NP; ++q) {  // the top plane is signed
                    const uint4 A = hb[2 * q + (i >> 1)];
                    const uint32_t ev = (i & 1) ? A.z : A.x, od = (i & 1) ? A.w : A.y;
                    if (q < NP - 1) {
                        S[m][q] = dp4a_su(lo, ev, S[m][q]);
                        S[m][q] = dp4a_su(hi, od, S[m][q]);
                    } else {
                        S[m][q] = dp4a_ss(lo, ev, S[m][q]);
                        S[m][q] = dp4a_ss(hi, od, S[m][q]);
                    }
                }
            }
        }
    };
    if constexpr (NL <= SL) {
        constexpr int SEGB = SL / NL;  // whole blocks per batch
        const int nb2 = (kc + SEGB - 1) / SEGB;
        for (int b = 0; b < nb2; ++b) {
            ring_acquire<WT>(c, b == nb2 - 1);
            const uint8_t* slot = c.ring + (size_t)c.rs * ring_slot_bytes<WT>() + c.lane * 16;
#pragma unroll
            for (int sg = 0; sg < SEGB; ++sg) {
                const int seg = b * SEGB + sg;
                if (seg < kc) {
                    begin_block(seg);
#pragma unroll
                    for (int m = 0; m < NL; ++m) line(m, slot + (sg * NL + m) * 512);
                }
            }
            __syncwarp();  // the slot is reused by a later issue of this warp
            if (++c.rs == NB) c.rs = 0;
        }
    } else {
        constexpr int BPB = NL / SL;  // batches per block
        for (int seg = 0; seg < kc; ++seg) {
            begin_block(seg);
#pragma unroll
            for (int bb = 0; bb < BPB; ++bb) {
                ring_acquire<WT>(c, seg == kc - 1 && bb == BPB - 1);
                const uint8_t* slot = c.ring + (size_t)c.rs * ring_slot_bytes<WT>() + c.lane * 16;
#pragma unroll
                for (int k = 0; k < SL; ++k) line(bb * SL + k, slot + k * 512);
                __syncwarp();
                if (++c.rs == NB) c.rs = 0;
            }
        }
    }
    if constexpr (WT == MK_W_INT4_G128) flush();
    float* xo = xbuf(p, layer + 1) + r0;
#pragma unroll
    for (int m = 0; m < NL; ++m) {
        float v;
        if constexpr (WT == MK_W_INT8_ROW)
            v = planes_combine(S[m][0], S[m][1], S[m][NP - 1]) * hstep * half_bits_to_f32(__ldg(scales + r0 + 32 * m));
        else
            v = acc[m] * (hstep * 0.0625f);
        red_add_f32(xo + 32 * m, v);
    }
}

template <int WT, int NL>
__device__ __forceinline__ void ffn_cols(Ctx& c, const TaskRec& t, int layer) {
    if constexpr (WT == MK_W_BF16 || WT == MK_W_FP16) {
        ffn_cols16<WT, NL>(c, t, layer);
        return;
    }
    if constexpr (idot_type<WT>()) {
        ffn_cols_idot<WT, NL>(c, t, layer);
        return;
    }
    const VmParams& p = *c.p;
    constexpr int NB = ring_slots<WT>();
    constexpr int BU = ffn_block(WT), SL = ffn_slot_lines(WT);
    constexpr bool QUANT = !(WT == MK_W_BF16 || WT == MK_W_FP16);
    const int kc = t.nrows / (2 * BU);
    const float* hs = ffn_h(c);
    const int r0 = c.warp * (p.d / NW) + c.lane;  // row of line 0 of this lane
    // quantised scales: after the codes of all F / BU blocks (d x 16 bytes each)
    const uint16_t* scales =
        QUANT ? (const uint16_t*)(p.w + p.layer_bytes * layer + p.l_down + (size_t)p.d * (p.F / BU) * 16) : nullptr;
    const int u0 = t.row0 / 2;  // first hidden unit of the task
    // 16-bit and int8: packed pair accumulators over the whole task; int4: a
    // float accumulator per line that takes each block's scaled dot product
    unsigned long long acc2[NL];
    float acc[NL], sc[NL];
    int sc_group = -1;
#pragma unroll
    for (int m = 0; m < NL; ++m) {
        acc2[m] = 0ull;
        acc[m] = 0.f;
    }
    unsigned long long hx[BU / 2];
    auto line = [&](int m, const uint8_t* src) {
        if constexpr (group_scaled<WT>()) {
            unsigned long long a = 0ull;
            chunk_fma<WT>(*(const uint4*)src, hx, a);
            acc[m] = fmaf(sc[m], sum2(a), acc[m]);
        } else {
            chunk_fma<WT>(*(const uint4*)src, hx, acc2[m]);
        }
    };
    auto block_scales = [&](int seg) {  // int4, fp8: the scales of block seg's group for this lane's rows
        if constexpr (group_scaled<WT>()) {
            const int g = (u0 + seg * BU) >> 7;
            if (g != sc_group) {
                sc_group = g;
#pragma unroll
                for (int m = 0; m < NL; ++m) sc[m] = half_bits_to_f32(__ldg(scales + (size_t)g * p.d + r0 + 32 * m));
            }
        }
    };
    if constexpr (NL <= SL) {
        constexpr int SEGB = SL / NL;  // whole blocks per batch
        const int nb2 = (kc + SEGB - 1) / SEGB;
        for (int b = 0; b < nb2; ++b) {
            ring_acquire<WT>(c, b == nb2 - 1);
            const uint8_t* slot = c.ring + (size_t)c.rs * ring_slot_bytes<WT>() + c.lane * 16;
#pragma unroll
            for (int sg = 0; sg < SEGB; ++sg) {
                const int seg = b * SEGB + sg;
                if (seg < kc) {
                    block_scales(seg);
                    load_h<WT>(hs + seg * BU, hx);
#pragma unroll
                    for (int m = 0; m < NL; ++m) line(m, slot + (sg * NL + m) * 512);
                }
            }
            __syncwarp();  // the slot is reused by a later issue of this warp
            if (++c.rs == NB) c.rs = 0;
        }
    } else {
        constexpr int BPB = NL / SL;  // batches per block
        for (int seg = 0; seg < kc; ++seg) {
            block_scales(seg);
            load_h<WT>(hs + seg * BU, hx);
#pragma unroll
            for (int bb = 0; bb < BPB; ++bb) {
                ring_acquire<WT>(c, seg == kc - 1 && bb == BPB - 1);
                const uint8_t* slot = c.ring + (size_t)c.rs * ring_slot_bytes<WT>() + c.lane * 16;
#pragma unroll
                for (int k = 0; k < SL; ++k) line(bb * SL + k, slot + k * 512);
                __syncwarp();
                if (++c.rs == NB) c.rs = 0;
            }
        }
    }
    float* xo = xbuf(p, layer + 1) + r0;
#pragma unroll
    for (int m = 0; m < NL; ++m) {
        float v = group_scaled<WT>() ? acc[m] : sum2(acc2[m]);
        if constexpr (WT == MK_W_INT8_ROW) v *= half_bits_to_f32(__ldg(scales + r0 + 32 * m));
        red_add_f32(xo + 32 * m, v);
    }
}

template <int WT>
__device__ __forceinline__ void ffn_down(Ctx& c, const TaskRec& t, int layer) {
    switch (c.p->d / 256) {  // lines per block; the host only fuses these shapes
        case 1: ffn_cols<WT, 1>(c, t, layer); break;
        case 2: ffn_cols<WT, 2>(c, t, layer); break;
        case 4: ffn_cols<WT, 4>(c, t, layer); break;
        case 8: ffn_cols<WT, 8>(c, t, layer); break;
        case 10:
            if constexpr (WT == MK_W_BF16 || WT == MK_W_FP16) ffn_cols<WT, 10>(c, t, layer);
            break;
        case 12:
            if constexpr (WT == MK_W_BF16 || WT == MK_W_FP16) ffn_cols<WT, 12>(c, t, layer);
            break;
        default: ffn_cols<WT, 16>(c, t, layer); break;
    }
}

// One GEMV task.  Warp group grp (g warps sharing each row) owns the batches
// of RW consecutive rows q*RW .. q*RW+RW for q = grp, grp + ngroups, ...; a
// gate/up pair stays inside one batch.  The batches come from the warp's
// stream (already requested before the counter wait).  Returns false when
// the CTA must stop (abort or watchdog), identically in every thread.
template <int WT, int BASE, int NG, bool SEL, int IW>
__device__ bool gemv_run(Ctx& c, const TaskRec& t, int task_id, int step, float& best_v, int& best_i) {
    const VmParams& p = *c.p;
    constexpr int HP = wpc<WT>() / 2;
    constexpr int NGM = 64 / wpc<WT>();
    constexpr int NB = ring_slots<WT>();
    constexpr int RW = rw_of<WT>(), TRAILER = trailer_of<WT>();
    const int op = t.op, layer = t.layer, row0 = t.row0, nrows = t.nrows, K = t.K;
    const int g = t.wpr, ngroups = NW / g;
    const int grp = c.warp / g, wig = c.warp % g;
    const int L = wig * 32 + c.lane, S = 32 * g;
    const int CH = K / wpc<WT>();  // 16-byte chunks of codes per row
    constexpr int LQ4 = wpc<WT>() == 8 ? 1 : wpc<WT>() == 16 ? 2 : 3;  // log2(float4 units per chunk)

    if (!wait_counters(c, t, task_id, step)) return false;
    int tok = 0;
    if (layer == 0 && (op == OP_QKV || op == OP_O)) {
        if (c.tid == 0) c.sh->tok = step_token(p, step);
        bar_consumers();
        tok = c.sh->tok;
        if (tok < 0) return false;
    }
    const float* xin = c.xs;
    bool from_global = false;
    switch (op) {
        case OP_QKV: {
            const uint16_t* gain = (const uint16_t*)(p.w + p.layer_bytes * layer + p.l_attn_norm);
            const uint16_t* emb = layer == 0 ? (const uint16_t*)(p.w + p.embed) + (size_t)tok * p.d : nullptr;
            prologue_rmsnorm<BASE, IW>(c, xbuf(p, layer), emb, gain, p.d, p.eps, LQ4);
            break;
        }
        case OP_GU:
        case OP_FFN:
            prologue_rmsnorm<BASE, IW>(c, xmid(p), nullptr,
                                   (const uint16_t*)(p.w + p.layer_bytes * layer + p.l_ffn_norm), p.d, p.eps, LQ4);
            break;
        case OP_LM:
            prologue_rmsnorm<BASE, IW>(c, xbuf(p, p.L), nullptr, (const uint16_t*)(p.w + p.final_norm), p.d, p.eps, LQ4);
            break;
        case OP_O:
            if (p.merge_tasks) prologue_att_copy<IW>(c, LQ4);
            else prologue_attention<IW>(c, LQ4);
            break;
        default:  // down reads h straight from device memory
            xin = p.h;
            from_global = true;
            break;
    }
    if (p.trace && c.tid == 0) c.sh->t_ph[0] = gtimer();
    // the lane's fragment of the input vector: k of chunk L + S*j (an
    // integer-dot task: the bytes of the three planes for those k)
    unsigned long long xr[IW ? 1 : NG * HP];
    uint4 xp[NG][IW == MK_W_INT4_G128 ? 2 * n_planes<IW>() : 3];
    if constexpr (IW != 0) {
        constexpr int CB = IW == MK_W_INT4_G128 ? 2 : 1;  // 16-byte words per chunk and plane
        const uint8_t* pl = (const uint8_t*)c.xs;
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const int cidx = L + S * j;
            const bool ok = cidx < CH;
#pragma unroll
            for (int q = 0; q < n_planes<IW>() * CB; ++q)
                xp[j][q] = ok ? *(const uint4*)(pl + (size_t)(q / CB) * K + (size_t)cidx * 16 * CB + 16 * (q % CB))
                              : make_uint4(0, 0, 0, 0);
        }
    } else {
        const float f = from_global ? 1.f : c.rstd;
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const int cidx = L + S * j;
            const bool ok = cidx < CH;
            const int cc = ok ? cidx : 0;
#pragma unroll
            for (int i = 0; i < HP / 2; ++i) {
                float4 v;
                if (from_global) v = __ldcg((const float4*)(xin + cc * wpc<WT>() + 4 * i));  // natural layout
                else v = *(const float4*)(xin + (i * CH + cc) * 4);                         // planes (xs_pos)
                xr[j * HP + 2 * i] = ok ? pack2(v.x * f, v.y * f) : 0ull;
                xr[j * HP + 2 * i + 1] = ok ? pack2(v.z * f, v.w * f) : 0ull;
            }
        }
    }
    // Rows shared by g > 1 warps: each warp leaves its partial sums in a
    // [row][warp] table (the input-vector region, free once every warp holds
    // its fragment) and the rows are finished after the loop, so the warps of
    // a group never wait for each other per batch.
    const bool defer = g > 1 && nrows * g <= p.xs_floats;
    float* part = c.xs;
    if (defer) bar_consumers();
    constexpr int B = RW >= 8 ? 3 : RW >= 4 ? 2 : RW >= 2 ? 1 : 0;  // log2(RW)
    const int my_r = c.lane >> (5 - B);                              // row of the batch this lane finishes
    const bool writer = (c.lane & ((32 >> B) - 1)) == 0;
    int par = 0;
    const int nbatches = (nrows + RW - 1) / RW;
    // QKV leads the layer's latency-bound chain: when all of this warp's
    // batches are already in flight, none of them issues a copy before the signal.
    const bool defer_all = op == OP_QKV && (nbatches - grp + ngroups - 1) / ngroups <= ring_slots<WT>() - 1;
    for (int q = grp; q < nbatches; q += ngroups) {
        const int rb = q * RW;
        const int row_g = row0 + rb + my_r;
        const bool has_row = rb + my_r < nrows;
        float resid = 0.f;  // residual input of this lane's row
        if (writer && has_row && !defer) {
            if (op == OP_DOWN) {
                resid = __ldcg(xmid(p) + row_g);
            } else if (op == OP_O && layer > 0) {
                resid = __ldcg(xbuf(p, layer) + row_g);
            } else if (op == OP_O) {
                const uint16_t* e = (const uint16_t*)(p.w + p.embed) + (size_t)tok * p.d;
                resid = base_to_f32<BASE>(__ldg(e + row_g));
            }
        }
        // keep NB - 1 batches in flight beyond this one, then wait for this one
        ring_acquire<WT>(c, op != OP_FFN && (q + ngroups >= nbatches || defer_all));
        const uint8_t* slot = c.ring + (size_t)c.rs * ring_slot_bytes<WT>();
        float v[RW], rsv[RW];
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            uint4 w[NG];
            float sc[NG];
            // Chunks past the row's end and rows past the task's end read
            // whatever the slot holds: zeros (the ring is cleared at start) or
            // finite weights of an earlier batch.  Their input values are
            // zero and their results are discarded, so no test is needed.
#pragma unroll
            for (int j = 0; j < NG; ++j) {
                w[j] = *(const uint4*)(slot + (r * NGM + j) * 512 + c.lane * 16);
                if constexpr (group_scaled<WT>())  // chunks per 128-k group: 4 (int4), 8 (fp8)
                    sc[j] = half_bits_to_f32(*(const uint16_t*)(slot + RW * NGM * 512 + r * TRAILER +
                                                                2 * (((L + S * j) >> (WT == MK_W_INT4_G128 ? 2 : 3)) &
                                                                     (TRAILER / 2 - 1))));
                else
                    sc[j] = 0.f;
            }
            if constexpr (IW != 0) v[r] = chunks_idot<WT, NG>(w, sc, xp) * c.xscale;
            else v[r] = chunks_dot<WT, NG>(w, sc, xr);
            if constexpr (WT == MK_W_INT8_ROW)
                rsv[r] = half_bits_to_f32(*(const uint16_t*)(slot + RW * NGM * 512 + r * TRAILER));
            else
                rsv[r] = 1.f;
        }
        __syncwarp();  // the slot is reused by a later issue of this warp
        if (++c.rs == NB) c.rs = 0;
        float tot = transpose_reduce<RW>(v, c.lane);
        if (g > 1 && !defer) {
            float* scr = &c.sh->gpart[grp][par][0][0];  // [row][warp]
            if (writer) scr[my_r * NW + wig] = tot;
            bar_group(2 + grp, S);
            if (wig == 0 && writer) {
                tot = 0.f;
                for (int ww = 0; ww < g; ++ww) tot += scr[my_r * NW + ww];
            }
            par ^= 1;
        }
        if constexpr (WT == MK_W_INT8_ROW) {
            float scale = rsv[0];
#pragma unroll
            for (int r = 1; r < RW; ++r) scale = my_r == r ? rsv[r] : scale;
            tot *= scale;
        }
        if (defer) {
            if (writer && has_row) part[(rb + my_r) * g + wig] = tot;
            continue;
        }
        if (op == OP_GU || op == OP_FFN) {  // rows alternate gate, up: the up total sits one row further
            const float up = __shfl_down_sync(0xFFFFFFFFu, tot, 32 >> B);
            if (wig == 0 && writer && has_row && !(my_r & 1)) {
                if (op == OP_GU) p.h[row_g >> 1] = silu(tot) * up;
                else ffn_h(c)[(rb + my_r) >> 1] = silu(tot) * up;
            }
        } else if (wig == 0 && writer && has_row) {
            if (op == OP_LM) {
                if (p.logits) p.logits[(size_t)step * p.V + row_g] = tot;
                float v = tot;
                if constexpr (SEL) {
                    if (p.top_k > 0) ffn_h(c)[rb + my_r] = tot;  // the CTA's top-k is taken after the loop
                    else if (p.inv_temp > 0.f)
                        v = sample_score(tot, (uint32_t)row_g, (uint32_t)(p.pos0 + step), p.inv_temp, p.seed_lo,
                                         p.seed_hi);
                }
                if (v > best_v) {  // rows ascend per lane: the first maximum is kept
                    best_v = v;
                    best_i = row_g;
                }
            } else if (op == OP_QKV) {
                st_tagged(p.qkv + row_g, tot, qkv_tag(p, step, layer));
            } else if (op == OP_O) {  // residual add: x_mid, and with the fused FFN the copy it adds into
                xmid(p)[row_g] = resid + tot;
                if (p.fused) xbuf(p, layer + 1)[row_g] = resid + tot;
            } else {  // down: residual add
                xbuf(p, layer)[row_g] = resid + tot;
            }
        }
    }
    if (p.trace && c.tid == 0) c.sh->t_ph[1] = gtimer();
    if (defer) {  // finish the shared rows: sum the warps' partials, then the epilogue
        bar_consumers();
        for (int rr = c.tid; rr < nrows; rr += NT) {
            const int row_g = row0 + rr;
            float tot = 0.f;
            for (int w = 0; w < g; ++w) tot += part[rr * g + w];
            if (op == OP_GU || op == OP_FFN) {  // gate rows are even, their up row follows
                if (!(rr & 1) && rr + 1 < nrows) {
                    float up = 0.f;
                    for (int w = 0; w < g; ++w) up += part[(rr + 1) * g + w];
                    if (op == OP_GU) p.h[row_g >> 1] = silu(tot) * up;
                    else ffn_h(c)[rr >> 1] = silu(tot) * up;
                }
            } else if (op == OP_LM) {
                if (p.logits) p.logits[(size_t)step * p.V + row_g] = tot;
                float v = tot;
                if constexpr (SEL) {
                    if (p.top_k > 0) ffn_h(c)[rr] = tot;
                    else if (p.inv_temp > 0.f)
                        v = sample_score(tot, (uint32_t)row_g, (uint32_t)(p.pos0 + step), p.inv_temp, p.seed_lo,
                                         p.seed_hi);
                }
                if (v > best_v) {  // rows ascend per thread: the first maximum is kept
                    best_v = v;
                    best_i = row_g;
                }
            } else if (op == OP_QKV) {
                st_tagged(p.qkv + row_g, tot, qkv_tag(p, step, layer));
            } else {  // O and down: residual add
                float resid;
                if (op == OP_DOWN) resid = __ldcg(xmid(p) + row_g);
                else if (layer > 0) resid = __ldcg(xbuf(p, layer) + row_g);
                else resid = base_to_f32<BASE>(__ldg((const uint16_t*)(p.w + p.embed) + (size_t)tok * p.d + row_g));
                if (op == OP_O) {
                    xmid(p)[row_g] = resid + tot;
                    if (p.fused) xbuf(p, layer + 1)[row_g] = resid + tot;
                } else {
                    xbuf(p, layer)[row_g] = resid + tot;
                }
            }
        }
    }
    return true;
}

template <int WT, int BASE, bool SEL>
__device__ __forceinline__ bool gemv_task(Ctx& c, const TaskRec& t, int task_id, int step, float& best_v, int& best_i) {
    const int S = 32 * t.wpr, CH = t.K / wpc<WT>(), ng = (CH + S - 1) / S;
    constexpr int NGMAX = 64 / wpc<WT>();  // 8 (16-bit), 4 (int8), 2 (int4)
    if constexpr (idot_type<WT>()) {
        // integer dot products for every task whose input vector a prologue
        // builds in shared memory (not the down rows of an unfused FFN) and
        // whose threads can hold it while the step D is found.  One instance
        // (NGMAX chunks per lane): chunks past a row's end meet zero planes.
        if (t.op != OP_DOWN && t.K <= 8 * NT * PIECE_IT)
            return gemv_run<WT, BASE, NGMAX, SEL, WT>(c, t, task_id, step, best_v, best_i);
    }
#define MK_RUN(N) return gemv_run<WT, BASE, (N <= NGMAX ? N : NGMAX), SEL, 0>(c, t, task_id, step, best_v, best_i)
    switch (ng) {
        case 1: MK_RUN(1);
        case 2: MK_RUN(2);
        case 3: MK_RUN(3);
        case 4: MK_RUN(4);
        case 5: MK_RUN(5);
        case 6: MK_RUN(6);
        case 7: MK_RUN(7);
        default: MK_RUN(8);
    }
#undef MK_RUN
}

// ------------------------------------------------------------------ attention
// One (KV head, chunk) task: RoPE for the group's queries and this step's
// key, K/V append at pos (last chunk only), then an online-softmax pass over
// the chunk's positions in tiles of ATTN_TILE.  Warp w owns positions
// w, w+8, ... of a tile for the scores (its K rows and the queries in
// registers) and stages their V rows in shared memory; for P.V each thread
// owns two adjacent dims of every head over one subset of a tile's positions
// (one V word and one probability vector per position), and the subsets are
// added once after the last tile.  The first tile's rows are requested
// before the queries are rotated, so cache reads overlap the qkv reads.  Writes, per
// query head, the chunk's running max m, its sum l = sum e^(s - m), and its
// output normalised by l (bounded by max|v|, so fp16 holds it at any chunk
// length); a merge weights each chunk by e^(m - M) * l.  Two tiles of cache
// rows are in flight: the first two are requested before this step's q/k/v
// are polled, and each later one as the tile two ahead of it finishes.
template <int HD>
static __device__ __forceinline__ bool attn_task(Ctx& c, const TaskRec& t, int task_id, int step) {
    const VmParams& p = *c.p;
    Shared& sh = *c.sh;
    AttnScratch& at = *c.at;
    constexpr int DPL = HD / 32;            // dims per lane
    constexpr int PPW = ATTN_TILE / NW;     // positions per warp per tile
    constexpr int NDP = HD / 2, NPS = NT / NDP;  // P.V: dim pairs, position subsets
    const int rep = p.Hq / p.Hkv, g = t.row0, ch = t.nrows, C = t.K, l = t.layer;
    const int pos = p.pos0 + step, len = pos + 1;
    const int j0 = (int)((int64_t)ch * len / C), j1 = (int)((int64_t)(ch + 1) * len / C);
    const float scale = rsqrtf((float)HD);
    constexpr int half = HD / 2;
    const size_t head_stride = (size_t)p.max_seq * HD;
    uint16_t* kbase = p.kv + (((size_t)l * 2 + 0) * p.Hkv + g) * head_stride;
    uint16_t* vbase = p.kv + (((size_t)l * 2 + 1) * p.Hkv + g) * head_stride;

    uint32_t kraw[PPW][DPL / 2], kn[PPW][DPL / 2];  // this tile's K and V rows, the next tile's
    uint32_t vraw[PPW][DPL / 2], vn[PPW][DPL / 2];
    // K rows of a tile go to kraw, V rows to vraw, as raw bf16 pairs (widened
    // where they are used, so that a load in flight does not hold the thread
    // up before its wait); the two halves are loaded separately so that the
    // next tile's rows are in flight while this one is computed (V once
    // staged in shared memory, K once the scores are done).
    auto load_rows = [&](uint32_t (&dst)[PPW][DPL / 2], const uint16_t* base, int jt, int n) {
#pragma unroll
        for (int k = 0; k < PPW; ++k) {
            const int jj = c.warp + NW * k, j = jt + jj;
            if (jj < n && j != pos) {
                if constexpr (DPL == 2) {
                    dst[k][0] = __ldcg((const unsigned int*)(base + (size_t)j * HD + c.lane * 2));
                } else {
                    const uint2 w = __ldcg((const uint2*)(base + (size_t)j * HD + c.lane * 4));
                    dst[k][0] = w.x;
                    dst[k][1] = w.y;
                }
            }
        }
    };
    auto stage_v = [&](int jt, int n) {  // V rows -> shared memory (pos from this step's value)
#pragma unroll
        for (int k = 0; k < PPW; ++k) {
            const int jj = c.warp + NW * k, j = jt + jj;
            if (jj < n) {
                uint32_t* dst = (uint32_t*)(at.sv + jj * HD + c.lane * DPL);
#pragma unroll
                for (int i = 0; i < DPL / 2; ++i) {
                    if (j == pos) {
                        dst[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(at.vcur[c.lane * DPL + 2 * i])) |
                                 ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(at.vcur[c.lane * DPL + 2 * i + 1])) << 16);
                    } else {
                        dst[i] = vraw[k][i];
                    }
                }
                if (j == pos) {  // this step's key (already bf16-rounded)
#pragma unroll
                    for (int i = 0; i < DPL / 2; ++i)
                        kraw[k][i] = (__float_as_uint(at.kcur[c.lane * DPL + 2 * i]) >> 16) |
                                     (__float_as_uint(at.kcur[c.lane * DPL + 2 * i + 1]) & 0xFFFF0000u);
                }
            }
        }
    };
    // The chunk's first cache rows are requested before this step's q/k/v
    // arrive: rows of earlier positions were written by earlier steps, whose
    // writers the wait of this CTA's previous task already ordered before us.
    if (j1 > j0) {
        load_rows(kraw, kbase, j0, min(ATTN_TILE, j1 - j0));
        load_rows(vraw, vbase, j0, min(ATTN_TILE, j1 - j0));
    }
    if (j0 + ATTN_TILE < j1) {
        load_rows(kn, kbase, j0 + ATTN_TILE, min(ATTN_TILE, j1 - j0 - ATTN_TILE));
        load_rows(vn, vbase, j0 + ATTN_TILE, min(ATTN_TILE, j1 - j0 - ATTN_TILE));
    }
    if (!wait_counters(c, t, task_id, step)) return false;  // counter waits, if any, and aborts

    // The group's query, key and value rows are read as tagged values: each
    // thread polls its words until they carry this step's tag.
    const uint32_t tag = qkv_tag(p, step, l);
    bool ok = true;
    const unsigned long long* vsrc = p.qkv + p.q_dim + p.kv_dim + (size_t)g * HD + c.tid;  // HD <= NT
    unsigned long long wv = c.tid < HD ? ld_tagged(vsrc) : 0ull;
    for (int i = c.tid; i < (rep + 1) * half && ok; i += NT) {
        const int hh = i / half, dd = i % half;
        const unsigned long long* src = hh < rep ? p.qkv + (size_t)(g * rep + hh) * HD : p.qkv + p.q_dim + (size_t)g * HD;
        unsigned long long w1 = ld_tagged(src + dd), w2 = ld_tagged(src + dd + half);
        ok = poll_tagged(p, src + dd, tag, w1, task_id, step) && poll_tagged(p, src + dd + half, tag, w2, task_id, step);
        const float x1 = __uint_as_float((uint32_t)w1), x2 = __uint_as_float((uint32_t)w2);
        const float ang = __fmul_rn((float)pos, __ldg(p.inv_freq + dd));
        float sn, cs;
        sincosf(ang, &sn, &cs);
        const float o1 = x1 * cs - x2 * sn, o2 = x2 * cs + x1 * sn;
        if (hh < rep) {
            at.q[hh * HD + dd] = o1 * scale;
            at.q[hh * HD + dd + half] = o2 * scale;
        } else {
            at.kcur[dd] = round_bf16(o1);
            at.kcur[dd + half] = round_bf16(o2);
        }
    }
    if (c.tid < HD && ok) {
        ok = poll_tagged(p, vsrc, tag, wv, task_id, step);
        at.vcur[c.tid] = round_bf16(__uint_as_float((uint32_t)wv));
    }
    if (c.tid < rep) {
        sh.m[c.tid] = -1.0e30f;
        sh.l[c.tid] = 0.f;
    }
    if (!bar_consumers_and(ok)) return false;
    if (p.trace && c.tid == 0) c.sh->t_ph[0] = gtimer();
    if (ch == C - 1) {
        for (int i = c.tid; i < HD; i += NT) {
            kbase[(size_t)pos * HD + i] = __bfloat16_as_ushort(__float2bfloat16_rn(at.kcur[i]));
            vbase[(size_t)pos * HD + i] = __bfloat16_as_ushort(__float2bfloat16_rn(at.vcur[i]));
        }
    }
    // The queries in registers: lane dims lane*DPL .. +DPL of every head.
    float qr[MAX_REP][DPL];
#pragma unroll
    for (int h = 0; h < MAX_REP; ++h)
#pragma unroll
        for (int i = 0; i < DPL; ++i) qr[h][i] = h < rep ? at.q[h * HD + c.lane * DPL + i] : 0.f;
    // P.V: thread (dp, ps) accumulates dims 2dp, 2dp+1 of every head over the
    // positions ps, ps + NPS, ... of each tile; the NPS partial sums of a
    // head's dim are added after the last tile.
    const int dp = c.tid % NDP, ps = c.tid / NDP;
    float acc[MAX_REP][2];
#pragma unroll
    for (int h = 0; h < MAX_REP; ++h) acc[h][0] = acc[h][1] = 0.f;

    for (int jt = j0; jt < j1; jt += ATTN_TILE) {
        const int n = min(ATTN_TILE, j1 - jt);
        stage_v(jt, n);
        // scores for (position k, head h), four heads at a time: PPW*4 partial
        // sums per lane, transposed so that lane pairs hold the totals
#pragma unroll
        for (int h0 = 0; h0 < MAX_REP; h0 += 4) {
            if (h0 >= rep) break;
            float v[PPW * 4];
#pragma unroll
            for (int k = 0; k < PPW; ++k)
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) {
                    float sacc = 0.f;
#pragma unroll
                    for (int i = 0; i < DPL; ++i)
                        sacc = fmaf(qr[h0 + hh][i],
                                    __uint_as_float((i & 1) ? (kraw[k][i >> 1] & 0xFFFF0000u) : (kraw[k][i >> 1] << 16)),
                                    sacc);
                    v[k * 4 + hh] = sacc;
                }
            const float sc = transpose_reduce<PPW * 4>(v, c.lane);
            constexpr int SH = PPW * 4 >= 32 ? 0 : PPW * 4 >= 16 ? 1 : 2;
            const int idx = c.lane >> SH, k = idx >> 2, hh = idx & 3, jj = c.warp + NW * k;
            if ((c.lane & ((1 << SH) - 1)) == 0 && h0 + hh < rep && jj < n) at.sc[(h0 + hh) * ATTN_TILE + jj] = sc;
        }
        bar_consumers();
        if (c.warp < rep) {  // online softmax statistics: warp h owns query head h
            const int h = c.warp;
            const float a = c.lane < n ? at.sc[h * ATTN_TILE + c.lane] : -3.0e38f;
            float mt = a;
#pragma unroll
            for (int o = 16; o; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, o));
            const float m_old = sh.m[h], m_new = fmaxf(m_old, mt);
            const float pa = c.lane < n ? expf(a - m_new) : 0.f;
            at.pt[c.lane * MAX_REP + h] = pa;
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
        for (int h = 0; h < MAX_REP; ++h) {
            if (h < rep) {
                const float al = sh.alpha[h];
                acc[h][0] *= al;
                acc[h][1] *= al;
            }
        }
        for (int jj = ps; jj < n; jj += NPS) {
            const uint32_t vv = *(const uint32_t*)(at.sv + jj * HD + 2 * dp);
            const float v0 = bf16_bits_to_f32(vv & 0xFFFFu), v1 = bf16_bits_to_f32(vv >> 16);
#pragma unroll
            for (int h0 = 0; h0 < MAX_REP; h0 += 4) {
                if (h0 >= rep) break;
                const float4 pr = *(const float4*)(at.pt + jj * MAX_REP + h0);
                const float pw[4] = {pr.x, pr.y, pr.z, pr.w};
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) {
                    acc[h0 + hh][0] = fmaf(pw[hh], v0, acc[h0 + hh][0]);
                    acc[h0 + hh][1] = fmaf(pw[hh], v1, acc[h0 + hh][1]);
                }
            }
        }
        bar_consumers();  // the next tile overwrites scores and V rows
        // the next tile's rows (requested one tile ago) become current; the
        // tile after it is requested now
        const int j2 = jt + 2 * ATTN_TILE;
#pragma unroll
        for (int k = 0; k < PPW; ++k)
#pragma unroll
            for (int i = 0; i < DPL / 2; ++i) {
                kraw[k][i] = kn[k][i];
                vraw[k][i] = vn[k][i];
            }
        if (j2 < j1) {
            load_rows(kn, kbase, j2, min(ATTN_TILE, j1 - j2));
            load_rows(vn, vbase, j2, min(ATTN_TILE, j1 - j2));
        }
    }
    if (p.trace && c.tid == 0) c.sh->t_ph[1] = gtimer();
    // The position subsets' sums, four heads at a time, through the V tile's
    // region (free: every tile ended with a barrier).
    float* red = reinterpret_cast<float*>(at.sv);  // [ps][head of the round][HD]
#pragma unroll
    for (int h0 = 0; h0 < MAX_REP; h0 += 4) {
        if (h0 >= rep) break;
#pragma unroll
        for (int hh = 0; hh < 4; ++hh)
            *(float2*)(red + ((size_t)ps * 4 + hh) * HD + 2 * dp) = make_float2(acc[h0 + hh][0], acc[h0 + hh][1]);
        bar_consumers();
        for (int oe = c.tid; oe < 4 * HD; oe += NT) {
            const int hh = oe / HD, dd = oe % HD, h = h0 + hh;
            if (h < rep) {  // stored normalised (acc / l), so its range is that of v
                float a = 0.f;
#pragma unroll
                for (int q = 0; q < NPS; ++q) a += red[((size_t)q * 4 + hh) * HD + dd];
                const float lh = sh.l[h];
                const uint16_t v = __half_as_ushort(__float2half_rn(lh > 0.f ? a / lh : 0.f));
#pragma unroll
                for (int k = 0; k < PART_COPIES; ++k)
                    p.part_acc[(((size_t)k * p.Hq + g * rep + h) * C + ch) * HD + dd] = v;
            }
        }
        bar_consumers();  // the next round overwrites the sums
    }
    if (c.tid < rep) {
        const float2 mlv = make_float2(sh.m[c.tid], sh.l[c.tid]);
#pragma unroll
        for (int k = 0; k < PART_COPIES; ++k)
            *(float2*)(p.part_ml + (((size_t)k * p.Hq + g * rep + c.tid) * C + ch) * 2) = mlv;
    }
    return true;
}

// ------------------------------------------------------------------ top-k selection
// This code exists only in the token-selection instantiation of the kernel
// (SEL = true); the greedy instantiation carries none of it.
// Scratch of a block selection, in the input-vector region: the LM-head task
// holds its input fragments in registers by then (its rows are in the merge
// scratch), and the select task has no input vector.
struct SelScratch {
    uint32_t hist[256];
    unsigned long long prefix;
    uint32_t need;       // rank still to find inside the current prefix
    uint32_t count;      // compaction cursor
    unsigned long long best;
};
static_assert(sizeof(SelScratch) <= sizeof(AttnScratch), "selection scratch");
static_assert(LM_MAX_ROWS * sizeof(float) <= sizeof(MergeScratch), "LM rows of a CTA");

// The k-th largest of the n distinct 56-bit keys key(0..n-1) (1 <= k <= n),
// by seven 8-bit radix passes from the top: each pass histograms the digit of
// the keys that share the prefix found so far, and the bin holding rank k
// extends the prefix.  Every consumer thread calls it; all get the result.
template <typename KeyFn>
__device__ __forceinline__ unsigned long long block_kth_largest(Ctx& b, int n, uint32_t k, KeyFn key) {
    SelScratch& ss = *reinterpret_cast<SelScratch*>(b.xs);
    if (b.tid == 0) {
        ss.prefix = 0ull;
        ss.need = k;
    }
    for (int shift = 48; shift >= 0; shift -= 8) {
        for (int i = b.tid; i < 256; i += NT) ss.hist[i] = 0u;
        bar_consumers();
        const unsigned long long pre = ss.prefix;
        for (int i = b.tid; i < n; i += NT) {
            const unsigned long long kk = key(i);
            if ((kk >> (shift + 8)) == (pre >> (shift + 8))) atomicAdd(&ss.hist[(kk >> shift) & 255u], 1u);
        }
        bar_consumers();
        if (b.warp == 0) {  // lane l scans bins 255 - 8l .. 248 - 8l (descending order)
            uint32_t cnt[8], tot = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                cnt[j] = ss.hist[255 - 8 * b.lane - j];
                tot += cnt[j];
            }
            uint32_t before = tot;  // inclusive scan over lanes, then made exclusive
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, before, o);
                if (b.lane >= o) before += v;
            }
            before -= tot;
            const uint32_t need = ss.need;
            if (before < need && need <= before + tot) {  // exactly one lane
                uint32_t acc = before;
                for (int j = 0; j < 8; ++j) {
                    if (need <= acc + cnt[j]) {
                        ss.prefix = pre | ((unsigned long long)(255 - 8 * b.lane - j) << shift);
                        ss.need = need - acc;
                        break;
                    }
                    acc += cnt[j];
                }
            }
        }
        bar_consumers();
    }
    return ss.prefix;
}

// After an LM-head task under top-k sampling: the CTA's k largest logits
// (ties: lower index) become its candidates, as selection keys in
// cand[blockIdx.x][0 .. MAX_TOP_K) (unused slots zero).
static __device__ __forceinline__ void lm_candidates(Ctx& b, int row0, int n) {
    const VmParams& p = *b.p;
    const float* v = reinterpret_cast<const float*>(&b.sh->mg);
    auto key = [&](int i) { return sel_key(v[i], (uint32_t)(row0 + i)); };
    const uint32_t k = (uint32_t)min(p.top_k, n);
    const unsigned long long kth = block_kth_largest(b, n, k, key);
    SelScratch& ss = *reinterpret_cast<SelScratch*>(b.xs);
    unsigned long long* out = p.cand + (size_t)blockIdx.x * MAX_TOP_K;
    if (b.tid == 0) ss.count = 0u;
    for (int j = b.tid + (int)k; j < MAX_TOP_K; j += NT) out[j] = 0ull;
    bar_consumers();
    for (int i = b.tid; i < n; i += NT) {
        const unsigned long long kk = key(i);
        if (kk >= kth) out[atomicAdd(&ss.count, 1u)] = kk;
    }
}

// OP_SELECT (token-select schedules): the step's token from every CTA's
// candidates.  Greedy (T = 0) and full-vocabulary sampling take the LM-head
// tasks' key; top-k sampling takes the global top k of the candidates (the
// top k of the vocabulary, since each CTA sent its own top k) and samples it
// by the largest Gumbel-max score.
static __device__ __forceinline__ void select_task(Ctx& b, int step) {
    const VmParams& p = *b.p;
    if (p.top_k == 0) {
        if (b.tid == 0) {
            const int id = key_token(p, step);
            if (id >= 0) {
                if (p.out_ids) p.out_ids[step] = id;
                p.status[3] = (uint32_t)id;
                p.status[4] = (uint32_t)(step + 1);
                *p.tokw = (unsigned long long)(uint32_t)id | ((unsigned long long)(uint32_t)(p.epoch0 + step + 1) << 32);
            }
        }
        return;
    }
    const int n = (int)gridDim.x * MAX_TOP_K;
    const unsigned long long* cand = p.cand;
    auto key = [&](int i) { return __ldcg(cand + i); };
    const unsigned long long kth = block_kth_largest(b, n, (uint32_t)p.top_k, key);
    SelScratch& ss = *reinterpret_cast<SelScratch*>(b.xs);
    unsigned long long best = 0ull;
    for (int i = b.tid; i < n; i += NT) {
        const unsigned long long kk = __ldcg(cand + i);
        if (kk == 0ull || kk < kth) continue;
        const uint32_t idx = sel_index(kk);
        const float z = sample_score(sel_value(kk), idx, (uint32_t)(p.pos0 + step), p.inv_temp, p.seed_lo, p.seed_hi);
        const unsigned long long zk = sel_key(z, idx);
        best = zk > best ? zk : best;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        best = other > best ? other : best;
    }
    if (b.tid == 0) ss.best = 0ull;
    bar_consumers();
    if (b.lane == 0) atomicMax(&ss.best, best);
    bar_consumers();
    if (b.tid == 0) {
        const uint32_t id = sel_index(ss.best);
        if (p.out_ids) p.out_ids[step] = (int32_t)id;
        p.status[3] = id;
        p.status[4] = (uint32_t)(step + 1);
        *p.tokw = (unsigned long long)id | ((unsigned long long)(uint32_t)(p.epoch0 + step + 1) << 32);
    }
}

// EOS: at the start of step s >= 1 every CTA waits until the previous step's
// token is final (its counter), reads it, and stops when it is eos.  Every
// CTA sees the same token at the same step boundary, so all stop together
// and no task of the stopped step runs.  False also after an abort.
static __device__ __forceinline__ bool eos_continue(Ctx& b, int step) {
    const VmParams& p = *b.p;
    if (b.tid == 0) {
        int go = b.sh->abort ? 0 : 1;
        const uint32_t* ctr = p.counters + (size_t)p.ctr_tok * CTR_STRIDE;
        const uint32_t target = (uint32_t)p.n_tok * (uint32_t)(p.epoch0 + step);
        const uint64_t t0 = gtimer();
        for (uint32_t it = 1; go && (int32_t)(ld_acquire(ctr) - target) < 0; ++it) {
            if ((it & 63u) == 0u) {
                if (aborted(p)) go = 0;
                else if (gtimer() - t0 > (uint64_t)p.watchdog_ns) {
                    raise_error(p, DEV_TIMEOUT, 0xFFFFFFFCu, (uint32_t)step);
                    go = 0;
                }
            }
        }
        if (go) {
            const int tok = selected_token(p, step);  // the previous step's choice (forced or not)
            go = tok >= 0 && tok != p.eos;
        }
        b.sh->flag = go;
    }
    bar_consumers();
    return b.sh->flag != 0;
}

// ------------------------------------------------------------------ consumer
template <int WT, int BASE, int HD, bool SEL>
__device__ __forceinline__ void consumer(Ctx& c) {
    const VmParams& p = *c.p;
    for (int s = 0; s < p.n_steps && !c.abort; ++s) {
        if constexpr (SEL) {
            if (p.eos >= 0 && s > 0 && !p.skip_lm && !eos_continue(c, s)) break;
        }
        for (int qi = 0; qi < c.nrec && !c.abort; ++qi) {
            const TaskRec& t = c.tab[qi];
            const int tid_ = c.q0 + qi;  // queue index: identifies the task in errors and traces
            c.cur = qi;
            const uint64_t t_start = p.trace ? gtimer() : 0;
            if (p.trace && c.tid == 0) c.sh->t_ph[0] = c.sh->t_ph[1] = c.sh->t_ph[2] = 0ull;
            float best_v = -3.0e38f;
            int best_i = 0;
            const bool gemv = t.op == OP_QKV || t.op == OP_O || t.op == OP_GU || t.op == OP_DOWN || t.op == OP_FFN ||
                              (t.op == OP_LM && !p.skip_lm);
            bool ok;
            if (gemv) {
                ok = gemv_task<WT, BASE, SEL>(c, t, tid_, s, best_v, best_i);
                if constexpr (SEL) {
                    if (ok && t.op == OP_LM && p.top_k > 0) {
                        bar_consumers();  // every row of the task is in shared memory
                        lm_candidates(c, t.row0, t.nrows);
                    }
                }
                if (ok && t.op == OP_FFN) {
                    bar_consumers();  // every SwiGLU output of the task is in shared memory
                    ffn_down<WT>(c, t, t.layer);
                }
            } else {
                ok = t.op == OP_ATTN ? attn_task<HD>(c, t, tid_, s) : wait_counters(c, t, tid_, s);
                if (ok && t.op == OP_MERGE) merge_task(c, t);
                if constexpr (SEL) {
                    if (ok && t.op == OP_SELECT && !p.skip_lm) select_task(c, s);
                }
                if (ok && t.op == OP_FIN && c.tid == 0 && !p.skip_lm) {
                    const unsigned long long k = __ldcg(p.key);
                    if ((k >> 49) != key_tag((uint32_t)(p.epoch0 + s))) {
                        raise_error(p, DEV_BAD_KEY, (uint32_t)tid_, (uint32_t)s);
                    } else {
                        const int id = (int)((1u << KEY_IDX_BITS) - 1u - (uint32_t)(k & ((1ull << KEY_IDX_BITS) - 1ull)));
                        if (p.out_ids) p.out_ids[s] = id;
                        p.status[3] = (uint32_t)id;
                        p.status[4] = (uint32_t)(s + 1);
                    }
                }
            }
            if (!ok) {  // decided uniformly (after a consumer barrier)
                c.abort = true;
                break;
            }
            if (gemv && t.op == OP_LM) {  // per-lane bests -> the warp's key (largest value, lowest index)
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
            const int sw = signal_warp(t, gemv);
            if (p.trace && c.tid == 0) c.sh->t_ph[2] = gtimer();
            if (c.warp == sw) cp_async_wait<0>();  // its release then has no copies to wait for
            bar_consumers();
            if (gemv && t.op == OP_LM && c.tid == 0) {
                unsigned long long key = 0;
                for (int w = 0; w < NW; ++w) key = c.sh->keys[w] > key ? c.sh->keys[w] : key;
                atomicMax(p.key, key);
            }
            signal_counter(c, t, sw);
            if (p.trace && c.warp == sw && c.lane == 0) {  // the releasing lane stamps its own slot
                const int k = s * c.nrec + qi;
                if (k < p.trace_cap) p.trace[((size_t)blockIdx.x * p.trace_cap + k) * 8 + 7] = gtimer();
            }
            // The copies the task skipped go out now, unless an attention or
            // merge task follows: it does not use the ring, and its own loads
            // are on the layer's critical path, so the copies wait for its end.
            const int nop = c.tab[qi + 1 < c.nrec ? qi + 1 : 0].op;
            if (!(nop == OP_ATTN || nop == OP_MERGE))
                for (; c.deferred > 0; --c.deferred) stream_issue<WT>(c);
            if (p.trace && c.tid == 0) {
                const int k = s * c.nrec + qi;
                if (k < p.trace_cap) {
                    unsigned long long* r = p.trace + ((size_t)blockIdx.x * p.trace_cap + k) * 8;
                    r[0] = (unsigned long long)tid_ | ((unsigned long long)s << 32);
                    r[1] = t_start;
                    r[2] = c.sh->t_waited;
                    r[3] = gtimer();
                    r[4] = c.sh->t_ph[0];
                    r[5] = c.sh->t_ph[1];
                    r[6] = c.sh->t_ph[2];  // r[7]: written by the releasing lane
                }
            }
        }
    }
}

template <int WT, int BASE, int HD, bool SEL>
__global__ void __launch_bounds__(THREADS, 1) vm_kernel(const VmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Ctx c;
    c.p = &p;
    c.tid = threadIdx.x;
    c.lane = threadIdx.x & 31;
    c.warp = threadIdx.x >> 5;
    c.xs = (float*)smem_raw;
    c.at = (AttnScratch*)smem_raw;
    c.sh = (Shared*)(smem_raw + region0_bytes(p.xs_floats));
    TaskRec* tab = (TaskRec*)(smem_raw + table_offset(p.xs_floats));
    c.tab = tab;
    c.ring = smem_raw + ring_offset(p.xs_floats, p.tab_cap) + (size_t)c.warp * ring_slots<WT>() * ring_slot_bytes<WT>();
    c.rstd = 1.f;
    c.abort = false;
    c.deferred = 0;
    c.rs = 0;
    c.cur = 0;
    c.q0 = p.queue_off[blockIdx.x];
    c.nrec = min(p.queue_off[blockIdx.x + 1] - c.q0, p.tab_cap);  // the host sizes tab_cap to the longest queue
    for (int i = threadIdx.x; i < c.nrec * (int)(sizeof(TaskRec) / 16); i += NT)
        ((uint4*)tab)[i] = __ldg((const uint4*)(p.recs + c.q0) + i);
    c.ws = WarpStream{0, 0, 0, 0, 1, 0, 0, 0, 0, 0, 32, 0, 0, nullptr, 0, 0, 0, nullptr, false};
    if (threadIdx.x == 0) c.sh->abort = 0;
    for (int i = c.lane; i < ring_slots<WT>() * ring_slot_bytes<WT>() / 16; i += 32)  // no stale NaN bit patterns
        ((uint4*)c.ring)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();  // the task table is complete
    for (int i = 0; i < ring_slots<WT>() - 1; ++i) stream_issue<WT>(c);
    consumer<WT, BASE, HD, SEL>(c);
    cp_async_wait<0>();  // no copy may land in shared memory after the CTA exits
}

}  // namespace mk
