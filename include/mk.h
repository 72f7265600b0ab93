/*
 * mk.h — C ABI of the batch-1 decode megakernel library (libmk.so).
 *
 * One persistent, cooperative sm_103a kernel runs the whole greedy decode loop
 * of a Llama-style dense decoder: one CTA per SM walks its own task queue
 * (wait on a monotonic counter -> run an instruction -> signal a counter), and
 * the host is not re-entered per token.  Sources of the design:
 *   - AutoMegaKernel explainer (gist.science, paper 2606.09682), "Methodology":
 *     Layer 0 VM (one cooperative threadblock per SM, local queue,
 *     wait -> dispatch -> signal, monotonic counters), Layer 1 instructions
 *     (GEMV, attention, RMSNorm), Layer 2 schedule IR + ScheduleConfig, and the
 *     static validate() gate run before any launch.
 *   - Kog MI300X monokernel tutorial (news.creeta.com), "How the monokernel
 *     removes launch overhead": prefill, decode and LM-head sampling in one
 *     resident kernel, no host re-entry per token.
 *   - Netra Kernel summary (aitrends.kr 102888), section details: a runtime that
 *     binds persistent and boundary buffers and launches on a caller-owned
 *     stream behind a C ABI, with exact contracts and no silent fallback.
 *
 * Conventions for every call:
 *   - Every call returns mk_status; nothing throws or aborts across the ABI.
 *   - The caller owns all device memory (packed weights, KV cache, workspace)
 *     and the stream.  The library owns only host-side state and carves its
 *     device tables (tasks, queues, counters, activations) out of the
 *     caller's workspace.
 *   - "host" pointers are ordinary CPU memory; "device" pointers are CUDA
 *     global memory of the device current at mk_create.
 *   - On error, mk_last_error(handle) (or mk_last_error(NULL) for calls that
 *     take no handle) returns a one-line reason; it is valid until the next
 *     call on the same handle / thread.
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* mk_stream_t;

typedef enum {
    MK_OK = 0,
    MK_ERR_INVALID_ARG = 1,      /* null/misaligned pointer, bad size, bad state            */
    MK_ERR_UNSUPPORTED = 2,      /* a model variant outside the contract (biases, odd dims) */
    MK_ERR_SCHEDULE_INVALID = 3, /* the static validator rejected the schedule: no launch   */
    MK_ERR_CAPACITY = 4,         /* pos + n_steps > max_seq, or a buffer is too small       */
    MK_ERR_CUDA = 5,             /* a CUDA runtime call failed                               */
    MK_ERR_TIMEOUT = 6,          /* a device wait gave up (watchdog); state must be reset    */
    MK_ERR_DEVICE = 7            /* the kernel reported an inconsistency (e.g. a stale key)  */
} mk_status;

/* Storage type of the GEMV weights (mk_model_desc.wdtype). */
enum {
    MK_W_BF16 = 0,      /* bf16 rows                                                      */
    MK_W_FP16 = 1,      /* IEEE fp16 rows                                                 */
    MK_W_INT8_ROW = 2,  /* int8, one fp16 scale per output row (W8A16)                     */
    MK_W_INT4_G128 = 3, /* int4 nibbles, one fp16 scale per 128 k of a row (W4A16)         */
    MK_W_FP8_E4M3 = 4   /* FP8 E4M3 codes (OCP format), one fp16 scale per 128 k of a row  */
};

/* Model variants the contract rejects (mk_model_desc.flags). */
enum {
    MK_FLAG_PROJ_BIAS = 1,   /* biased projections: rejected, not silently mis-run          */
    MK_FLAG_TIED_HEAD = 2,   /* LM head tied to the embedding: rejected (head is separate)  */
    MK_FLAG_ROPE_SCALING = 4 /* rope scaling variants: rejected                             */
};

/* Shape of a Llama-style dense decoder (RMSNorm, rotate-half RoPE, GQA,
 * SwiGLU FFN, final RMSNorm, untied LM head).  Contract: head_dim in {64,128},
 * n_q_heads % n_kv_heads == 0, n_q_heads / n_kv_heads <= 8,
 * d_model % 128 == 0, d_ffn % 128 == 0, n_q_heads * head_dim % 128 == 0,
 * vocab < 131072, max_seq >= 1.  base_dtype (MK_W_BF16 or MK_W_FP16) is the
 * storage type of the embedding, the norm gains and the packer's source rows;
 * wdtype may be base_dtype, MK_W_INT8_ROW, MK_W_INT4_G128 or MK_W_FP8_E4M3
 * (bf16 source). */
typedef struct {
    int32_t n_layers, d_model, n_q_heads, n_kv_heads, head_dim, d_ffn, vocab;
    float rms_eps, rope_theta;
    int32_t max_seq;
    int32_t wdtype;
    int32_t base_dtype;
    int32_t flags;
} mk_model_desc;

/* Structural knobs of the lowering (AutoMegaKernel "ScheduleConfig": tiling,
 * SM assignment, pipelining depth).  0 selects the default. */
typedef struct {
    int32_t sms;            /* CTAs (= SMs used); default all SMs of the device              */
    int32_t rows_in_flight; /* weight rows of one batch of a warp group; the only value built
                               is 4 for int8/int4 weights and 2 otherwise (0 selects it)  */
    int32_t attn_chunks;    /* split-KV chunks per KV head; default from max_seq and sms     */
    int32_t watchdog_ms;    /* a device wait gives up after this long; default 1000          */
    int32_t token_select;   /* 1: one more task per step selects the token after the LM
                               head (needed for top-k sampling); 0 (default): the LM-head
                               tasks' block argmax is the selection                       */
    int32_t prefill_chunk;  /* 0 (default): mk_prefill runs the decode kernel over the prompt,
                               one position per step.  A multiple of 128 up to 4096: mk_prefill
                               runs the prompt through tensor-core GEMMs (tcgen05) in chunks of
                               this many tokens (16-bit weights only; the workspace grows by the
                               chunk's activations)                                        */
} mk_schedule_config;

/* ------------------------------------------------------------------ packing
 * The packer lays every GEMV weight out as contiguous rows in one blob, in
 * the order the device streams them: per layer [QKV rows (Wq;Wk;Wv)] [O rows]
 * [gate/up rows interleaved: gate_j, up_j] [down], then the LM head, the
 * norm gains and the embedding.  Quantised rows carry their fp16 scales after
 * the codes; every row starts on a 16-byte boundary.
 * Down projection, when the FFN is fused (d_model / 256 in {1, 2, 4, 8, 16},
 * and also 10 and 12 for 16-bit weights): column blocks of 16 bytes, block b
 * holding for r = 0 .. d_model-1 the codes of Wdown[r][BU b .. BU (b+1)) at
 * offset (b * d_model + r) * 16, BU = 8 (bf16/fp16), 16 (int8) or 32 (int4,
 * even k in the low nibble); quantised blocks are followed by their fp16
 * scales, [d_model] (int8, one per row) or [d_ffn / 128][d_model] (int4).
 * Otherwise rows [d_model][d_ffn] like the other tensors. */
enum {
    MK_T_EMBED = 0, MK_T_LM_HEAD = 1, MK_T_FINAL_NORM = 2, MK_T_ATTN_NORM = 3, MK_T_FFN_NORM = 4,
    MK_T_WQ = 5, MK_T_WK = 6, MK_T_WV = 7, MK_T_WO = 8, MK_T_WGATE = 9, MK_T_WUP = 10,
    MK_T_WDOWN = 11
};

/* Bytes of the packed weight blob for desc.  Errors: INVALID_ARG, UNSUPPORTED. */
mk_status mk_packed_size(const mk_model_desc* desc, size_t* bytes);

/* Pack one tensor into its place in a host blob of mk_packed_size bytes.
 * src_host: row-major [rows][cols] array of base_dtype bit patterns (uint16),
 * shapes as in the standard decoder (Wq [Hq*hd][d], Wk/Wv [Hkv*hd][d],
 * Wo [d][Hq*hd], Wgate/Wup [d_ffn][d], Wdown [d][d_ffn], embed/LM head
 * [vocab][d], norms [d]).  layer is ignored for the embedding, LM head and
 * final norm.  Quantised models quantise here (int8 per row, int4 per
 * 128-group; fp16 scales rounded to nearest even).  Errors: INVALID_ARG
 * (null pointer, bad id/layer, blob too small), UNSUPPORTED. */
mk_status mk_pack_tensor(const mk_model_desc* desc, int32_t tensor, int32_t layer,
                         const void* src_host, void* blob_host, size_t blob_bytes);

/* Byte offset, row stride and row count of a packed tensor inside the blob
 * (rows of Wq/Wk/Wv/Wgate/Wup are interleaved with their siblings: use the
 * stride and first_row to locate them).  A down projection stored in column
 * blocks reports row_stride 0 (layout above).  Errors: INVALID_ARG. */
mk_status mk_tensor_layout(const mk_model_desc* desc, int32_t tensor, int32_t layer,
                           size_t* offset, size_t* row_stride, int32_t* first_row,
                           int32_t* row_step, int32_t* rows);

/* Host quantisers the packer uses (exposed for tests).  w: float32 [n][k]
 * row-major; q: int8 [n][k]; s16: fp16 bit patterns, [n] (int8) or
 * [n][k/128] (int4, k % 128 == 0).  Readings: s = fp16(fp32(max|w|)/127 or 7),
 * q = clamp(round_half_even(fp32(w)/fp32(s)), +-127 or +-7), s == 0 -> q == 0. */
mk_status mk_quantize_int8(const float* w, int64_t n, int64_t k, int8_t* q, uint16_t* s16);
mk_status mk_quantize_int4(const float* w, int64_t n, int64_t k, int8_t* q, uint16_t* s16);
/* FP8 E4M3 block-scaled (Netra Kernel summary, "TL;DR": FP8 ops): per 128 k,
 * s = fp16(fp32(max|w|) / 448); q = the E4M3 code nearest to fp32(w) /
 * fp32(s) (ties to the even code, magnitudes clamped to 448), s == 0 -> 0;
 * q: uint8 codes [n][k], s16 [n][k/128]. */
mk_status mk_quantize_fp8(const float* w, int64_t n, int64_t k, uint8_t* q, uint16_t* s16);

/* ------------------------------------------------------------------ sizes */
/* KV cache bytes: bf16 [n_layers][2 (K,V)][n_kv_heads][max_seq][head_dim]. */
mk_status mk_kv_cache_size(const mk_model_desc* desc, size_t* bytes);

/* Workspace bytes for desc/cfg on n_sms CTAs (n_sms <= 0: the current device's
 * SM count, which needs a CUDA device). */
mk_status mk_workspace_size(const mk_model_desc* desc, const mk_schedule_config* cfg,
                            int32_t n_sms, size_t* bytes);

/* ------------------------------------------------------------------ schedule IR
 * The lowered task DAG (AutoMegaKernel "Layer 2": a typed schedule IR whose
 * tasks are synchronised by monotonic counters).  A task on CTA `sm` runs
 * once per decode step e (epoch): it waits until every (counter, count,
 * epoch_off) satisfies counter >= count * (e + 1 + epoch_off), runs, then adds
 * 1 to signal_ctr (-1: none).  Accesses describe the bytes the instruction
 * touches at epoch e: [lo + e*stride, hi + e*stride + e*grow) of buffer buf.
 *
 * A counter c with ctr_buf[c] = b >= 0 is carried by tagged values instead of
 * a memory word (this library's own device protocol; the pages describe only
 * counters): each value its producers write to b holds the step's tag, and a
 * waiting task polls the values of b it reads until they carry that tag.
 * Such a wait therefore orders the waiting task after the producers' writes
 * of b that it reads, and after nothing else. */
#define MK_IR_MAX_WAITS 2
enum { MK_ACC_READ = 1, MK_ACC_WRITE = 2, MK_ACC_ATOMIC = 3 };
enum { MK_BUF_OUTPUT = 1 };

typedef struct {
    int32_t sm, op, layer;
    int32_t n_waits;
    int32_t wait_ctr[MK_IR_MAX_WAITS];
    int32_t wait_count[MK_IR_MAX_WAITS];
    int32_t wait_epoch_off[MK_IR_MAX_WAITS];
    int32_t signal_ctr;
    int32_t acc_begin, n_acc;
} mk_ir_task;

typedef struct {
    int32_t buf, kind;
    int64_t lo, hi, stride, grow;
} mk_ir_access;

typedef struct {
    int32_t n_sms, n_tasks, n_counters, n_buffers, n_acc;
    mk_ir_task* tasks;
    mk_ir_access* acc;
    int32_t* queue;      /* task ids, SM after SM                                  */
    int32_t* queue_off;  /* [n_sms + 1]: SM s runs queue[queue_off[s] .. queue_off[s+1]) */
    int32_t* buf_flags;  /* [n_buffers]: MK_BUF_OUTPUT marks the step's results      */
    int32_t* ctr_buf;    /* [n_counters]: -1, or the buffer whose tagged values carry
                          * the counter (below)                                     */
} mk_ir;

/* Lower desc/cfg for n_sms CTAs (host only).  *out is library-owned: free it
 * with mk_free_ir.  Its arrays may be edited in place (tests mutate them). */
mk_status mk_build_ir(const mk_model_desc* desc, const mk_schedule_config* cfg, int32_t n_sms,
                      mk_ir** out);
void mk_free_ir(mk_ir* ir);

/* The static validator (AutoMegaKernel "safety gate", validate()): rejects
 * the IR unless it is
 *   well formed  — every id in range, every task queued once on its own SM;
 *   deadlock-free — every wait threshold satisfiable, 1 <= count <= #producers,
 *                   epoch_off in {-1, 0}, and the dependency graph including
 *                   each SM's queue order acyclic;
 *   race-free    — every multi-producer counter joined (count == #producers),
 *                   counter reuse across steps ordered, and every pair of
 *                   conflicting accesses ordered by happens-before over three
 *                   unrolled steps (a wait on a tagged counter counts only
 *                   for accesses to its buffer, and only from the producers
 *                   whose writes overlap the waiter's reads);
 *   tag-complete — every byte of a tagged buffer that a waiter reads is
 *                   written by the counter's producers in the waited step;
 *   correct      — every task's writes reach an output buffer.
 * Returns MK_OK or MK_ERR_SCHEDULE_INVALID with the first reason in `why`
 * (may be NULL).  Host only; no device is touched. */
mk_status mk_validate_ir(const mk_ir* ir, char* why, size_t why_len);

/* Lower and validate in one call (no device work). */
mk_status mk_validate_schedule(const mk_model_desc* desc, const mk_schedule_config* cfg,
                               int32_t n_sms, char* why, size_t why_len);

/* ------------------------------------------------------------------ runtime */
typedef struct mk_handle mk_handle;

/* Check the contract, lower the model, run the static validator and only then
 * upload the schedule into the workspace (async on `stream`).  weights_dev:
 * the packed blob (mk_packed_size bytes, 256-byte aligned); kv_dev: the KV
 * cache (mk_kv_cache_size bytes, 16-byte aligned); workspace_dev:
 * mk_workspace_size bytes, 256-byte aligned.  The device current at this call
 * is the one used by every later call on the handle.  Errors: INVALID_ARG,
 * UNSUPPORTED, CAPACITY (buffer too small), SCHEDULE_INVALID (nothing was
 * written to the device), CUDA. */
mk_status mk_create(const mk_model_desc* desc, const mk_schedule_config* cfg,
                    const void* weights_dev, size_t weights_bytes, void* kv_dev, size_t kv_bytes,
                    void* workspace_dev, size_t workspace_bytes, mk_stream_t stream,
                    mk_handle** out);

/* Prefill: positions 0..n-2 of tokens_host go through the decoder (KV writes
 * only, LM head skipped); afterwards pos = n-1 and the pending token is
 * tokens_host[n-1], which the first decode step feeds.  Resets the sequence
 * (any earlier tokens are discarded).  Synchronous.
 * With mk_schedule_config.prefill_chunk = 0 the decode kernel runs the prompt
 * one position per step in one launch.  With a chunk size C, the prompt goes
 * through the layers C tokens at a time: RMSNorm, then the QKV, O, gate/up
 * and down projections as tensor-core GEMMs (tcgen05.mma, operands staged by
 * TMA, 16-bit activations, fp32 accumulation) with RoPE + KV append, residual
 * and SwiGLU fused into their epilogues, and causal GQA attention of the chunk
 * over the cache (Kog monokernel tutorial: prefill in the same runtime as
 * decode).  Errors: INVALID_ARG (n < 1, token out of range), CAPACITY
 * (n > max_seq), CUDA, TIMEOUT. */
mk_status mk_prefill(mk_handle* h, const int32_t* tokens_host, int32_t n);

/* Greedy decode of n_steps tokens in ONE launch.  Step s feeds the pending
 * token at position pos, writes KV[pos], emits the argmax (lowest index on
 * ties) into out_ids_host[s], then pending <- that id and pos += 1.
 * Synchronous: returns after the ids are on the host.  Errors: INVALID_ARG,
 * CAPACITY (pos + n_steps > max_seq), CUDA, TIMEOUT, DEVICE. */
mk_status mk_decode(mk_handle* h, int32_t n_steps, int32_t* out_ids_host);

/* The same launch without any host synchronisation or copy (the hot path).
 * forced_dev (nullable): int32 [n_steps]; when given, step s feeds
 * forced_dev[s] instead of the pending token / previous argmax (teacher
 * forcing).  out_ids_dev (nullable): int32 [n_steps].
 * logits_dev (nullable): float32 [n_steps][vocab], every step's logits.
 * pos advances by n_steps at once; the pending token stays on the device.
 * Call mk_finish before reading results or trusting the state.  Errors:
 * INVALID_ARG, CAPACITY, CUDA. */
mk_status mk_decode_async(mk_handle* h, int32_t n_steps, const int32_t* forced_dev,
                          int32_t* out_ids_dev, float* logits_dev);

/* Wait for the stream and read the device status word: MK_OK, MK_ERR_TIMEOUT
 * (a wait gave up; mk_create-time state is restored on the next launch) or
 * MK_ERR_DEVICE. */
mk_status mk_finish(mk_handle* h);

/* Sequence state: the next position and the pending token (-1 while it only
 * exists on the device after mk_decode_async). */
mk_status mk_get_state(const mk_handle* h, int32_t* pos, int32_t* pending);

/* Rewind: continue from position pos (<= current pos) feeding `pending`.
 * KV entries at positions >= pos are rewritten by the next steps. */
mk_status mk_set_state(mk_handle* h, int32_t pos, int32_t pending);

/* Launch geometry chosen at mk_create: CTAs, threads per CTA, dynamic shared
 * memory bytes, rows in flight per warp group, tasks in the schedule. */
mk_status mk_get_launch_info(const mk_handle* h, int32_t* ctas, int32_t* threads,
                             int32_t* smem_bytes, int32_t* rows_in_flight, int32_t* n_tasks);

/* Token selection of later mk_decode / mk_decode_async launches (Kog monokernel
 * tutorial, "How the monokernel removes launch overhead": sampling and the
 * end-of-sequence check stay inside the one resident kernel).
 *   temperature: 0 selects greedy argmax (lowest index on ties, the default).
 *     T > 0 draws token i with probability proportional to exp(logit_i / T)
 *     over the candidate set, by the Gumbel-max rule: the candidate with the
 *     largest logit_i / T - log(-log(u_i)) (lowest index on ties), computed in
 *     fp32 inside the LM-head task.
 *   top_k: 0 = every token is a candidate; 1..MK_MAX_TOP_K = the k largest
 *     logits (lower index first among equal logits); needs a handle created
 *     with mk_schedule_config.token_select = 1, else MK_ERR_UNSUPPORTED.
 *   seed: u_i comes from Philox4x32-10 (Salmon et al., SC 2011) with key
 *     (seed low 32 bits, seed high 32 bits) and counter (i, pos, 0, 0), pos
 *     the absolute position of the token being fed; first output word x,
 *     u = (2 * (x >> 9) + 1) * 2^-24.  Draws depend only on (seed, pos, i), so
 *     a decode split over several calls draws as one call does.
 *   eos_id: -1 = none.  Otherwise a launch stops after the step that selects
 *     eos_id: that id is emitted, later steps do not run (no KV writes), and
 *     pos advances by the steps run.  mk_decode fills the rest of
 *     out_ids_host with -1.  After mk_decode_async, call mk_finish before the
 *     next launch (it reads how many steps ran; a launch before it returns
 *     MK_ERR_INVALID_ARG).
 * Errors: INVALID_ARG (NULL, T < 0 or not finite, top_k out of range, eos_id
 * out of range), UNSUPPORTED (top_k on a handle without token_select). */
#define MK_MAX_TOP_K 64
typedef struct {
    float temperature;
    int32_t top_k;
    uint64_t seed;
    int32_t eos_id;
} mk_sampling;
mk_status mk_set_sampling(mk_handle* h, const mk_sampling* s);

/* Steps the last launch ran (n_steps, or fewer after an EOS stop); valid after
 * mk_decode or mk_finish. */
int32_t mk_last_steps(const mk_handle* h);

/* Kernel launches issued by this handle so far (one per prefill/decode call). */
int64_t mk_launch_count(const mk_handle* h);

const char* mk_last_error(const mk_handle* h);
void mk_destroy(mk_handle* h);

/* ------------------------------------------------------------------ allocation-free decode */
/* Largest scratch mk_decode_static accepts (8 MiB; a Llama-3-8B layout with an
 * 8k context needs about 1.6 MiB on 152 SMs). */
#define MK_STATIC_SCRATCH_BYTES (8u << 20)

/* Greedy decode of n_steps tokens from position pos feeding `token`, without a
 * handle or a caller workspace.  The design sources have no counterpart: this
 * is an extra entry point of this library for callers that may not allocate.
 * It runs the same kernel and schedule as mk_create + mk_decode, but the
 * kernel's scratch (schedule tables, sync counters, activations, split-KV
 * partials, token ids) lives in one file-scope device array of
 * MK_STATIC_SCRATCH_BYTES per device; no device memory is allocated.
 *
 * weights_dev: packed blob (mk_packed_size bytes, 256-byte aligned).
 * kv_dev: KV cache (mk_kv_cache_size bytes, 16-byte aligned) whose positions
 *   0..pos-1 already hold the sequence (e.g. written by a handle's mk_prefill);
 *   positions pos..pos+n_steps-1 are written.
 * out_ids_host: int32 [n_steps], the argmax ids (lowest index on ties).
 * logits_dev (nullable): float32 [n_steps][vocab].
 * Synchronous on `stream`.
 *
 * Set-up: the first call on a device looks up the array's address (once per
 * device) and, like every call whose desc or resolved config differs from the
 * previous call's on that device, lowers, validates and uploads the schedule;
 * make that first call before any stream capture.  Every call zeroes the
 * status words, sync counters, argmax key and tagged q/k/v words before its
 * launch; all other scratch is written before it is read.
 * Calls share the one array per device: calls that overlap (other host
 * threads, other streams) race on it.  Calls of this library are serialised
 * by a host lock, and each returns only after its launch has finished.
 * Errors: INVALID_ARG, UNSUPPORTED, CAPACITY (scratch above
 * MK_STATIC_SCRATCH_BYTES, checked first; then buffers too small or
 * pos + n_steps > max_seq), SCHEDULE_INVALID, CUDA, TIMEOUT, DEVICE. */
mk_status mk_decode_static(const mk_model_desc* desc, const mk_schedule_config* cfg,
                           const void* weights_dev, size_t weights_bytes, void* kv_dev,
                           size_t kv_bytes, int32_t pos, int32_t token, int32_t n_steps,
                           int32_t* out_ids_host, float* logits_dev, mk_stream_t stream);

/* ------------------------------------------------------------------ test support */
/* Dequantise one packed GEMV tensor on the device with the same device
 * function the decode kernel uses: out_dev float32 [rows][cols] row-major.
 * Errors: INVALID_ARG, CUDA. */
mk_status mk_debug_dequant(const mk_model_desc* desc, const void* weights_dev, int32_t tensor,
                           int32_t layer, float* out_dev, mk_stream_t stream);

/* Record %globaltimer stamps of every task of later launches into trace_dev,
 * uint64 [ctas][records_per_cta][8] = {queue index | step << 32, task start,
 * wait done, task end, input ready, compute done, body done, signal released}:
 * "input ready" is the end of a GEMV task's prologue or the arrival of an
 * attention task's q/k/v, "compute done" the end of its row batches or tiles
 * (both 0 for other tasks), "body done" the end of the instruction before its
 * signal, "signal released" the counter release (0 for tasks that signal
 * none); "task end" follows the copies issued after the signal.  The queue index is the task's
 * position in the concatenated per-CTA queues (mk_ir.queue holds the task id
 * at each index).  Record k of a CTA is step * queue_len + queue slot, and
 * records past the capacity are dropped.  NULL disables tracing.  The buffer
 * is caller-owned and must outlive the launches. */
mk_status mk_debug_set_trace(mk_handle* h, void* trace_dev, int32_t records_per_cta);

/* Launch a one-CTA kernel that waits on a counter nothing ever signals, with
 * a watchdog of timeout_us; returns MK_ERR_TIMEOUT when the wait gave up
 * cleanly (the context stays usable).  counter_dev: 128 zeroed bytes. */
mk_status mk_debug_watchdog(int32_t timeout_us, void* counter_dev, mk_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MK_H */
