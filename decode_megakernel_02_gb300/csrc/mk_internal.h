// Internal definitions shared by the host lowering (C++) and the persistent
// decode kernel (CUDA).  Not part of the public ABI.
#pragma once
#include <stdint.h>

#include "mk.h"

namespace mk {

// Instructions of the VM (AutoMegaKernel explainer, "Methodology", Layer 1:
// GEMV, attention, RMSNorm ... micro-kernels behind one task ABI).
enum Op : int32_t {
    OP_QKV = 1,   // RMSNorm prologue + [Wq;Wk;Wv] GEMV rows -> qkv (fp32, tagged)
    OP_ATTN = 2,  // RoPE + KV append + split-KV GQA attention chunk -> partials
    OP_O = 3,     // merge partials + Wo GEMV rows + residual add -> x
    OP_GU = 4,    // RMSNorm prologue + interleaved gate/up rows + SwiGLU -> h
    OP_DOWN = 5,  // Wdown GEMV rows + residual add -> x
    OP_LM = 6,    // final RMSNorm + LM-head rows + block argmax -> logits, key
    OP_FIN = 7,   // read the step's argmax key -> out id
    OP_FFN = 8,   // RMSNorm prologue + gate/up rows + SwiGLU (kept on chip) + the down
                  // projection's columns of those units, red.add into the next residual
    OP_MERGE = 9, // split-KV merge of one KV group's query heads -> att (O then reads att)
    OP_SELECT = 10  // token-select: the step's top-k sample from every CTA's candidates
};

constexpr int NT = 256;                 // threads per CTA (eight warps)
constexpr int NW = NT / 32;             // warps per CTA
constexpr int THREADS = NT;
constexpr int MAXG = 8;                 // 8-element k groups per lane
constexpr int MAX_K = 8 * NT * MAXG;    // 16384: eight warps x 32 lanes x MAXG groups
constexpr int INT4_MAX_ROW_K = 8192;    // int4 GEMV rows: their fp16 scales (one per 128 k) fill a 128-byte slot trailer
constexpr int MAX_REP = 8;              // query heads per KV head
constexpr int ATTN_TILE = 32;           // positions per online-softmax tile
// Copies of the split-KV partials (and of the merged attention output) that
// their producers write: every O task reads all of them, and CTAs that read
// the same lines at the same moment queue at the L2 slices holding them, so
// CTA b reads copy b % PART_COPIES.
constexpr int PART_COPIES = 4;
constexpr int CTR_STRIDE = 32;          // u32 words between counters (128 B lines)
constexpr int MAX_HC = 1024;            // query heads x split-KV chunks (merge scratch)
constexpr int FFN_MAX_UNITS = 2 * MAX_HC;  // hidden units of one OP_FFN task (its SwiGLU outputs reuse the merge scratch)
constexpr int MAX_TOP_K = MK_MAX_TOP_K;     // top-k candidates per CTA
constexpr int LM_MAX_ROWS = 2 * MAX_HC;     // LM-head rows of one CTA under top-k sampling (kept in the merge scratch)

// Hidden units per 16-byte column chunk of a fused down projection: 8
// (16-bit), 16 (int8) or 32 (int4) codes.
#ifdef __CUDACC__
__host__ __device__
#endif
constexpr int ffn_block(int wdtype) {
    return wdtype == MK_W_INT8_ROW || wdtype == MK_W_FP8_E4M3 ? 16 : wdtype == MK_W_INT4_G128 ? 32 : 8;
}

// 512-byte lines a ring slot holds in the column phase of the fused FFN.
#ifdef __CUDACC__
__host__ __device__
#endif
constexpr int ffn_slot_lines(int wdtype) {
    return wdtype == MK_W_FP8_E4M3 ? 8 : wdtype == MK_W_INT4_G128 ? 8 : 16;
}
// Rows of one GEMV batch (a ring slot): 4 for int8 and int4 codes, whose
// batches would otherwise carry a quarter or half of a 16-bit batch's bytes
// for the same fixed cost per batch; 2 otherwise.
#ifdef __CUDACC__
__host__ __device__
#endif
constexpr int gemv_batch_rows(int wdtype) {
    return wdtype == MK_W_INT8_ROW || wdtype == MK_W_INT4_G128 ? 4 : 2;
}

// The FFN runs fused (OP_FFN) when every warp's share of the d_model output
// rows is a whole number of 32-row lines (d_model % 256 == 0) and the lines
// per column block of a warp's rows (d_model / 256) is one the kernel is built
// for; a block whose lines exceed a ring slot spans several batches.
#ifdef __CUDACC__
__host__ __device__
#endif
constexpr bool ffn_fused(int wdtype, int base_dtype, int d_model) {
    return wdtype == base_dtype
               ? d_model % 256 == 0 && (d_model / 256 == 1 || d_model / 256 == 2 || d_model / 256 == 4 ||
                                        d_model / 256 == 8 || d_model / 256 == 10 || d_model / 256 == 12 ||
                                        d_model / 256 == 16)
               : (wdtype == MK_W_INT8_ROW || wdtype == MK_W_INT4_G128 || wdtype == MK_W_FP8_E4M3) &&
                     d_model % 256 == 0 &&
                     (d_model / 256 == 1 || d_model / 256 == 2 || d_model / 256 == 4 || d_model / 256 == 8 ||
                      d_model / 256 == 16);
}

// Warps that share one weight row: enough that each lane holds at most
// MAXG 8-wide k-groups of the input vector in registers (K <= 2048 * wpr).
#ifdef __CUDACC__
__host__ __device__
#endif
constexpr int warps_per_row(int K) { return K <= 2048 ? 1 : K <= 4096 ? 2 : K <= 8192 ? 4 : 8; }

// One entry of the device task table (one IR task).
struct DevTask {
    int32_t op, layer;
    int32_t row0, nrows;    // GEMV: first row / row count.  ATTN: kv head / chunk
    int32_t K;              // GEMV: reduction length.  ATTN: chunks per head
    int32_t row_bytes;      // GEMV: packed row stride
    int32_t rps;            // GEMV: rows per batch over all warp groups (rw * 8 / wpr)
    int32_t wpr;            // GEMV: warps sharing one row (1, 2, 4, 8)
    int64_t w_off;          // GEMV: blob offset of row0
    int32_t n_waits;
    int32_t wait_ctr[2];
    int32_t wait_cnt[2];
    int32_t wait_off[2];
    int32_t signal_ctr;
    int32_t rw;             // GEMV: rows a warp group keeps in flight (a batch)
};
static_assert(sizeof(DevTask) == 80, "DevTask layout");

// The device's compact copy of a DevTask.  Each CTA keeps the records of its
// own queue (in queue order) in shared memory for the whole launch.
struct TaskRec {
    uint8_t op, n_waits;
    uint16_t layer;
    int32_t row0, nrows;    // as in DevTask
    uint32_t w_off16;       // GEMV: blob offset of row0 / 16
    uint16_t row_bytes16;   // GEMV: packed row stride / 16
    uint16_t K;             // GEMV: reduction length.  ATTN: chunks per head
    uint16_t wait_ctr[2];
    uint16_t wait_cnt[2];
    int16_t signal_ctr;     // -1: none
    uint8_t wpr;
    uint8_t wait_prev;      // bit i: wait i targets the previous step (epoch offset -1)
};
static_assert(sizeof(TaskRec) == 32, "TaskRec layout");

// Byte offsets of the packed weight blob.
struct BlobLayout {
    bool down_cols;     // W_down stored in 16-byte column blocks (fused FFN) instead of rows
    int64_t row_qkv, row_o, row_gu, row_down, row_lm;   // row strides
    int64_t norm_bytes;                                 // bytes per norm-gain vector (padded)
    int64_t layer_bytes;                                // one layer block
    int64_t l_attn_norm, l_ffn_norm, l_qkv, l_o, l_gu, l_down;   // inside a layer block
    int64_t final_norm, lm, embed, total;
};

// Kernel parameters (passed by value).
struct VmParams {
    const uint8_t* w;          // packed blob
    uint16_t* kv;              // bf16 KV cache [L][2][Hkv][max_seq][hd]
    uint32_t* status;          // [0] status, [1] queue index, [2] detail, [3] last token, [4] steps run
    uint32_t* counters;        // n_counters lines of CTR_STRIDE words
    unsigned long long* key;   // the step's packed argmax key
    const TaskRec* recs;       // every CTA's queue, concatenated in queue order
    const int32_t* queue_off;  // [n_sms + 1]: CTA b owns recs[queue_off[b] .. queue_off[b+1])
    const float* inv_freq;     // [hd/2]
    float* x;                  // residual stream [2][d], then x_mid [d]
    unsigned long long* qkv;   // [q_dim + 2 kv_dim] tagged values: fp32 bits | tag << 32
    float* part_ml;            // [PART_COPIES][Hq][C][2]  (running max, sum)
    float* att;                // [PART_COPIES][q_dim] merged attention output (merge tasks; else unused)
    int32_t merge_tasks;       // 1: OP_MERGE tasks merge the partials and O reads att
    uint16_t* part_acc;        // [PART_COPIES][Hq][C][hd] fp16 bit patterns
    float* h;                  // SwiGLU output [F]
    const int32_t* forced;     // nullable: token fed at step s
    int32_t* out_ids;          // nullable: argmax of step s
    float* logits;             // nullable: [n_steps][V]
    // model
    int32_t L, d, Hq, Hkv, hd, F, V, max_seq, wdtype, base_dtype, q_dim, kv_dim, C;
    int32_t fused;             // FFN as OP_FFN: residual buffers alternate by layer (x + (layer & 1) * d)
    float eps;
    int64_t layer_bytes, l_attn_norm, l_ffn_norm, l_down, final_norm, embed;
    // run
    int32_t n_steps, pos0, epoch0, skip_lm;
    int32_t pending;           // token fed at step 0 (no forcing); -1: status[3]
    int32_t xs_floats;         // shared-memory input vector capacity: max(d, q_dim)
    int32_t tab_cap;           // task records a CTA's shared-memory table holds (longest queue)
    int64_t watchdog_ns;
    // token selection
    float inv_temp;            // 1 / temperature (0: greedy argmax)
    int32_t top_k;             // > 0: candidates are the top_k logits (token-select task)
    uint32_t seed_lo, seed_hi; // Philox4x32-10 key
    int32_t eos;               // -1: none; else a launch stops after the step that selects it
    int32_t ctr_tok, n_tok;    // the counter after which the step's token is final, and its producers
    unsigned long long* cand;  // token-select: MAX_TOP_K candidate keys per CTA
    unsigned long long* tokw;  // token-select: the selected token | (epoch + 1) << 32 (nullptr: read the key)
    unsigned long long* trace; // nullable: per-task timestamps [ctas][trace_cap][4]
    int32_t trace_cap;
};

// Status codes written by the device into status[0].
enum : uint32_t { DEV_OK = 0, DEV_TIMEOUT = 1, DEV_BAD_KEY = 2, DEV_BAD_TOKEN = 3 };

// Argmax key: [tag:15][orderable fp32:32][0x1FFFF - index:17].  A larger tag
// (step) always wins, so the word needs no reset between steps.
constexpr int KEY_IDX_BITS = 17;
constexpr int KEY_TAG_MAX = 32767;

}  // namespace mk
