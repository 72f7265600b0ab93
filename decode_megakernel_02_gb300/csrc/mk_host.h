// Host-side internal API shared by the library's C++ translation units.
#pragma once
#include <stdint.h>

#include <string>
#include <vector>

#include "mk_internal.h"

namespace mk {

void set_error(const char* fmt, ...);
const char* thread_error();

uint16_t f32_to_f16_rne(float f);
float f16_to_f32(uint16_t h);
float base_to_f32(uint16_t v, int base);

mk_status check_desc(const mk_model_desc* d);
int64_t row_stride(int64_t K, int wdtype);
BlobLayout blob_layout(const mk_model_desc* d);

// Resolved schedule knobs.
struct Config {
    int sms, rw, C;
    int64_t watchdog_ns;
    bool token_select;        // an OP_SELECT task after the LM head selects each step's token
    int pf_chunk;             // tensor-core prefill chunk (tokens; 0: prefill by the decode kernel)
};
mk_status resolve_config(const mk_model_desc* d, const mk_schedule_config* cfg, int n_sms,
                         Config* out);

// IR buffers of the decode path.
enum Buf : int32_t { B_X = 0, B_QKV, B_PART, B_H, B_LOGITS, B_KEY, B_OUT, B_KV, B_ATT, B_CAND, B_TOKW, B_COUNT };

// Whether the split-KV partials are merged by per-group OP_MERGE tasks (true
// when every O CTA would otherwise read more than 64 KB of partials).
bool merge_tasks(const mk_model_desc* d, const Config& c);

// Result of lowering: the IR (owning storage) and the matching device tables.
struct Lowering {
    std::vector<mk_ir_task> tasks;
    std::vector<mk_ir_access> acc;
    std::vector<std::vector<int32_t>> queues;
    std::vector<DevTask> dev;
    int32_t n_counters = 0;
    // Per counter: -1, or the buffer whose tagged values carry it.  Such a
    // counter has no memory word: its producers' writes of that buffer carry
    // the step's tag and its waiters poll the values they read, so the device
    // records keep neither the signal nor the wait.
    std::vector<int32_t> ctr_buf;
    int64_t bytes_per_sm_max = 0, bytes_per_sm_min = 0;
    int32_t ctr_tok = 0, n_tok = 0;   // the counter after which a step's token is final, its producers
    int32_t lm_rows_max = 0;          // most LM-head rows of one CTA
};
mk_status lower(const mk_model_desc* d, const Config& c, Lowering* out);

// The device tables of a lowering: records in queue order and queue offsets.
// Fails (INVALID_ARG) if a field does not fit its record width.
mk_status device_tables(const Lowering& lw, int n_sms, std::vector<TaskRec>* recs, std::vector<int32_t>* queue,
                        std::vector<int32_t>* queue_off, int32_t* tab_cap);

// Flatten a lowering into a library-owned mk_ir.
mk_ir* to_ir(const Lowering& lw, int n_sms);

// The validator on a flat IR.
mk_status validate_ir(const mk_ir* ir, std::string* why);

// Workspace layout (byte offsets).
struct WsLayout {
    int64_t status, counters, key, tokw, cand, recs, queue_off, inv_freq, x, qkv, part_ml, part_acc, att,
        h, tok, out_ids;
    // tensor-core prefill (pf_chunk > 0): residual, q, and the hi / lo halves of
    // the GEMM inputs (normed x, attention output, SwiGLU output)
    int64_t pf_x, pf_q, pf_h, pf_hl, pf_ao, pf_aol, pf_gu, pf_gul, pf_err;
    int64_t total;
};
WsLayout ws_layout(const mk_model_desc* d, const Config& c, int64_t n_tasks, int32_t n_counters);

}  // namespace mk
