// Lowering of the decoder to a task DAG synchronised by monotonic counters,
// the device tables and the workspace layout.
//
// AutoMegaKernel explainer, "Methodology": Layer 2 lowers the model to a typed
// schedule IR (a task DAG synchronised by monotonic counters) under a
// ScheduleConfig (tiling, SM assignment, pipelining depth).  The safety gate
// that must accept the IR before any launch is in mk_validate.cpp.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <iterator>
#include <numeric>
#include <string>
#include <vector>

#include "mk_host.h"

namespace mk {

static int64_t up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

// ------------------------------------------------------------------ config
mk_status resolve_config(const mk_model_desc* d, const mk_schedule_config* cfg, int n_sms,
                         Config* out) {
    mk_schedule_config z{};
    if (!cfg) cfg = &z;
    if (n_sms < 1) {
        set_error("n_sms %d < 1", n_sms);
        return MK_ERR_INVALID_ARG;
    }
    Config c{};
    c.sms = cfg->sms > 0 ? std::min(cfg->sms, n_sms) : n_sms;
    if (cfg->sms < 0 || cfg->rows_in_flight < 0 || cfg->attn_chunks < 0 || cfg->watchdog_ms < 0) {
        set_error("negative schedule knob");
        return MK_ERR_INVALID_ARG;
    }
    c.rw = gemv_batch_rows(d->wdtype);  // the kernel's batch for this weight type
    if (cfg->rows_in_flight && cfg->rows_in_flight != c.rw) {
        set_error("rows_in_flight %d: only %d is built for this weight type", cfg->rows_in_flight, c.rw);
        return MK_ERR_INVALID_ARG;
    }
    if (cfg->attn_chunks) {
        c.C = cfg->attn_chunks;
    } else {
        int by_len = std::max(1, d->max_seq / 64);
        int by_sms = std::max(1, c.sms / d->n_kv_heads);
        c.C = std::max(1, std::min(std::min(by_len, by_sms), MAX_HC / d->n_q_heads));
    }
    if (c.C < 1 || (int64_t)c.C * d->n_q_heads > MAX_HC) {
        set_error("attn_chunks %d: need 1 <= chunks * n_q_heads <= %d", c.C, MAX_HC);
        return MK_ERR_INVALID_ARG;
    }
    c.watchdog_ns = (int64_t)(cfg->watchdog_ms ? cfg->watchdog_ms : 1000) * 1000000;
    if (cfg->token_select != 0 && cfg->token_select != 1) {
        set_error("token_select %d: 0 or 1", cfg->token_select);
        return MK_ERR_INVALID_ARG;
    }
    c.token_select = cfg->token_select == 1;
    if (cfg->prefill_chunk < 0 || cfg->prefill_chunk % 128 != 0 || cfg->prefill_chunk > 4096) {
        set_error("prefill_chunk %d: 0 or a multiple of 128 up to 4096", cfg->prefill_chunk);
        return MK_ERR_INVALID_ARG;
    }
    c.pf_chunk = cfg->prefill_chunk;
    *out = c;
    return MK_OK;
}

// ------------------------------------------------------------------ lowering
namespace {

struct Builder {
    const mk_model_desc* d;
    Config c;
    Lowering* lw;
    std::vector<int64_t> load;
    int S;
    std::vector<std::vector<mk_ir_access>> tacc;  // accesses per task (flattened at the end)

    // Split `units` (of unit_rows rows, unit_bytes bytes) across the CTAs: every
    // CTA gets units/S, and the remainder goes to the CTAs with the least
    // weight bytes so far, so that total bytes per CTA per token stay level.
    std::vector<std::pair<int, std::pair<int64_t, int64_t>>> split(int64_t units, int64_t unit_bytes) {
        std::vector<int64_t> cnt(S, units / S);
        int64_t rem = units % S;
        std::vector<int> order(S);
        std::iota(order.begin(), order.end(), 0);
        std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return load[a] < load[b]; });
        for (int64_t i = 0; i < rem; ++i) cnt[order[i]] += 1;
        std::vector<std::pair<int, std::pair<int64_t, int64_t>>> out;
        int64_t u = 0;
        for (int s = 0; s < S; ++s) {
            if (!cnt[s]) continue;
            out.push_back({s, {u, u + cnt[s]}});
            load[s] += cnt[s] * unit_bytes;
            u += cnt[s];
        }
        return out;
    }

    int add_task(int sm, const DevTask& t, std::vector<mk_ir_access> acc) {
        mk_ir_task it{};
        it.sm = sm;
        it.op = t.op;
        it.layer = t.layer;
        it.n_waits = t.n_waits;
        for (int i = 0; i < 2; ++i) {
            it.wait_ctr[i] = t.wait_ctr[i];
            it.wait_count[i] = t.wait_cnt[i];
            it.wait_epoch_off[i] = t.wait_off[i];
        }
        it.signal_ctr = t.signal_ctr;
        tacc.push_back(std::move(acc));
        int id = (int)lw->tasks.size();
        lw->tasks.push_back(it);
        lw->dev.push_back(t);
        lw->queues[sm].push_back(id);
        return id;
    }

    void set_wait(const std::vector<int>& ids, int ctr, int cnt, int off) {
        for (int id : ids) {
            mk_ir_task& it = lw->tasks[id];
            DevTask& t = lw->dev[id];
            it.n_waits = t.n_waits = 1;
            it.wait_ctr[0] = t.wait_ctr[0] = ctr;
            it.wait_count[0] = t.wait_cnt[0] = cnt;
            it.wait_epoch_off[0] = t.wait_off[0] = off;
        }
    }
};

mk_ir_access A(int buf, int kind, int64_t lo, int64_t hi, int64_t stride = 0, int64_t grow = 0) {
    mk_ir_access a;
    a.buf = buf;
    a.kind = kind;
    a.lo = lo;
    a.hi = hi;
    a.stride = stride;
    a.grow = grow;
    return a;
}

}  // namespace

// Nominal position for the access model: KV reads cover [0, P0 + e) and the
// step's write lands at P0 + e.
static constexpr int64_t P0 = 1;

bool merge_tasks(const mk_model_desc* d, const Config& c) {
    return (int64_t)d->n_q_heads * c.C * (d->head_dim + 2) * 4 > 64 * 1024;
}

mk_status lower(const mk_model_desc* d, const Config& c, Lowering* lw) {
    *lw = Lowering{};
    Builder B{d, c, lw, std::vector<int64_t>(c.sms, 0), c.sms};
    lw->queues.assign(c.sms, {});
    const int L = d->n_layers, hd = d->head_dim, Hq = d->n_q_heads, Hkv = d->n_kv_heads;
    const int rep = Hq / Hkv, C = c.C;
    const int64_t qd = (int64_t)Hq * hd, kd = (int64_t)Hkv * hd, dm = d->d_model, F = d->d_ffn,
                  V = d->vocab;
    const BlobLayout bl = blob_layout(d);
    // Counters per layer: 0 QKV, 1 attention done, 2 O, 3 FFN / gate-up, 4 down,
    // 5 + g chunks of KV group g (merge tasks only).
    const int CS = 5 + Hkv;
    const int CTR_LM = CS * L;
    const int CTR_TOK = CS * L + 1;  // token-select schedules: the step's token is final
    const bool ts = c.token_select;
    const int64_t CAND_BYTES = (int64_t)MAX_TOP_K * 8;  // one CTA's candidate keys
    lw->n_counters = CS * L + (ts ? 2 : 1);
    lw->ctr_buf.assign(lw->n_counters, -1);
    auto ctr = [&](int l, int k) { return CS * l + k; };
    const bool mt = merge_tasks(d, c);
    const int64_t ML_BYTES = (int64_t)Hq * C * 2 * 4, PART_BYTES = ML_BYTES + (int64_t)Hq * C * hd * 2;
    // Residual buffers: x[2][d].  With the fused FFN the layer-l input lives in
    // x[l & 1]; O(l) writes x_mid into x[l & 1] and x[(l + 1) & 1], and the
    // OP_FFN tasks add their down-projection partials into x[(l + 1) & 1].
    const bool fused = bl.down_cols;
    auto xb = [&](int l) -> int64_t { return fused ? (int64_t)(l & 1) * 4 * dm : 0; };
    const int64_t xm = 8 * dm;  // x_mid: written by O, read by the FFN side

    auto gemv_task = [&](int op, int l, int64_t row0, int64_t nrows, int64_t K, int64_t rb,
                         int64_t region, int unit_rows, int signal) {
        DevTask t{};
        t.op = op;
        t.layer = l;
        t.row0 = (int32_t)row0;
        t.nrows = (int32_t)nrows;
        t.K = (int32_t)K;
        t.row_bytes = (int32_t)rb;
        (void)unit_rows;  // rw >= 2 keeps gate/up pairs inside one warp batch
        t.wpr = warps_per_row((int)K);
        t.rw = c.rw;
        t.rps = c.rw * (NW / t.wpr);
        t.w_off = region + row0 * rb;
        t.signal_ctr = signal;
        return t;
    };

    std::vector<int> prev;  // tasks of the previous stage
    int prev_ctr = -1;
    std::vector<int> first_qkv;
    int fin_sm = -1;
    std::vector<int> lm_ids;

    for (int l = 0; l < L; ++l) {
        const int64_t lb = bl.layer_bytes * l;
        // ---- QKV: RMSNorm(x) -> rows of [Wq; Wk; Wv]
        std::vector<int> ids;
        for (auto& p : B.split(qd + 2 * kd, bl.row_qkv)) {
            int64_t r0 = p.second.first, r1 = p.second.second;
            DevTask t = gemv_task(OP_QKV, l, r0, r1 - r0, dm, bl.row_qkv, lb + bl.l_qkv, 1, ctr(l, 0));
            std::vector<mk_ir_access> acc;
            acc.push_back(l == 0 ? A(ts ? B_TOKW : B_KEY, MK_ACC_READ, 0, 8) : A(B_X, MK_ACC_READ, xb(l), xb(l) + 4 * dm));
            acc.push_back(A(B_QKV, MK_ACC_WRITE, 8 * r0, 8 * r1));
            ids.push_back(B.add_task(p.first, t, acc));
        }
        if (l == 0) {
            first_qkv = ids;
            fin_sm = lw->tasks[ids[0]].sm;
        } else {
            B.set_wait(ids, prev_ctr, (int)prev.size(), 0);
        }
        prev = ids;
        prev_ctr = ctr(l, 0);
        std::vector<char> has_qkv(c.sms, 0);
        for (int id : ids) has_qkv[lw->tasks[id].sm] = 1;
        bool tag_ok = true;  // every CTA of this layer's attention, merge and O tasks ran a QKV task

        // ---- attention: one task per (kv head, chunk), placed on the least-loaded
        // CTAs, no two on one CTA while free CTAs remain (they run in parallel)
        ids.clear();
        const int64_t est = std::max<int64_t>(1, d->max_seq / 2 / C) * hd * 2 * 2;
        std::vector<char> has_attn(c.sms, 0);
        int attn_placed = 0;
        for (int g = 0; g < Hkv; ++g) {
            for (int ch = 0; ch < C; ++ch) {
                if (attn_placed == c.sms) {
                    std::fill(has_attn.begin(), has_attn.end(), 0);
                    attn_placed = 0;
                }
                int sm = -1;
                for (int q = 0; q < c.sms; ++q)
                    if (!has_attn[q] && (sm < 0 || B.load[q] < B.load[sm])) sm = q;
                has_attn[sm] = 1;
                ++attn_placed;
                B.load[sm] += est;
                DevTask t{};
                t.op = OP_ATTN;
                t.layer = l;
                t.row0 = g;
                t.nrows = ch;
                t.K = C;
                t.signal_ctr = mt ? ctr(l, 5 + g) : ctr(l, 1);
                std::vector<mk_ir_access> acc;
                acc.push_back(A(B_QKV, MK_ACC_READ, 8 * (int64_t)g * rep * hd, 8 * (int64_t)(g + 1) * rep * hd));
                acc.push_back(A(B_QKV, MK_ACC_READ, 8 * (qd + (int64_t)g * hd), 8 * (qd + (int64_t)(g + 1) * hd)));
                acc.push_back(A(B_QKV, MK_ACC_READ, 8 * (qd + kd + (int64_t)g * hd),
                                8 * (qd + kd + (int64_t)(g + 1) * hd)));
                // The cache rows of earlier positions are read from before the
                // task's own wait (their writers precede this CTA's previous
                // task), so the read belongs to that previous task.
                const int prev_task = lw->queues[sm].empty() ? -1 : lw->queues[sm].back();
                for (int kv = 0; kv < 2; ++kv) {
                    int64_t base = (((int64_t)l * 2 + kv) * Hkv + g) * d->max_seq * hd * 2;
                    const mk_ir_access hist = A(B_KV, MK_ACC_READ, base, base + P0 * hd * 2, 0, hd * 2);
                    if (prev_task >= 0) B.tacc[prev_task].push_back(hist);
                    else acc.push_back(hist);
                    if (ch == C - 1)  // the chunk holding the newest position appends it
                        acc.push_back(A(B_KV, MK_ACC_WRITE, base + P0 * hd * 2, base + (P0 + 1) * hd * 2, hd * 2, 0));
                }
                for (int k = 0; k < PART_COPIES; ++k)  // every copy of the partials
                    for (int i = g * rep; i < (g + 1) * rep; ++i) {
                        int64_t ml = k * PART_BYTES + ((int64_t)i * C + ch) * 2 * 4,
                                ac = k * PART_BYTES + ML_BYTES + ((int64_t)i * C + ch) * hd * 2;
                        acc.push_back(A(B_PART, MK_ACC_WRITE, ml, ml + 8));
                        acc.push_back(A(B_PART, MK_ACC_WRITE, ac, ac + hd * 2));
                    }
                ids.push_back(B.add_task(sm, t, acc));
                tag_ok = tag_ok && has_qkv[sm];
            }
        }
        B.set_wait(ids, prev_ctr, (int)prev.size(), 0);
        if (mt) {
            // ---- merge of each KV group's chunks, on the CTA of the group's last
            // chunk right after it: att gets the group's query-head outputs
            std::vector<int> mids;
            for (int g = 0; g < Hkv; ++g) {
                const int last = ids[(size_t)g * C + C - 1];
                DevTask t{};
                t.op = OP_MERGE;
                t.layer = l;
                t.row0 = g;
                t.K = C;
                t.signal_ctr = ctr(l, 1);
                std::vector<mk_ir_access> acc;
                const int64_t h0 = (int64_t)g * rep, h1 = h0 + rep;
                const int64_t cpo = (lw->tasks[last].sm % PART_COPIES) * PART_BYTES;  // the CTA's copy
                acc.push_back(A(B_PART, MK_ACC_READ, cpo + h0 * C * 2 * 4, cpo + h1 * C * 2 * 4));
                acc.push_back(A(B_PART, MK_ACC_READ, cpo + ML_BYTES + h0 * C * hd * 2, cpo + ML_BYTES + h1 * C * hd * 2));
                for (int k = 0; k < PART_COPIES; ++k)
                    acc.push_back(A(B_ATT, MK_ACC_WRITE, k * 4 * qd + h0 * hd * 4, k * 4 * qd + h1 * hd * 4));
                const int id = B.add_task(lw->tasks[last].sm, t, acc);
                tag_ok = tag_ok && has_qkv[lw->tasks[last].sm];
                B.set_wait({id}, ctr(l, 5 + g), C, 0);
                mids.push_back(id);
            }
            ids = mids;
        }
        prev = ids;
        prev_ctr = ctr(l, 1);

        // ---- O: merge partials -> rows of Wo, residual add
        ids.clear();
        for (auto& p : B.split(dm, bl.row_o)) {
            int64_t r0 = p.second.first, r1 = p.second.second;
            DevTask t = gemv_task(OP_O, l, r0, r1 - r0, qd, bl.row_o, lb + bl.l_o, 1, ctr(l, 2));
            std::vector<mk_ir_access> acc;
            const int cp = p.first % PART_COPIES;  // the CTA's copy
            if (mt) acc.push_back(A(B_ATT, MK_ACC_READ, cp * 4 * qd, (cp + 1) * 4 * qd));
            else acc.push_back(A(B_PART, MK_ACC_READ, cp * PART_BYTES, (cp + 1) * PART_BYTES));
            if (l == 0) acc.push_back(A(ts ? B_TOKW : B_KEY, MK_ACC_READ, 0, 8));
            else acc.push_back(A(B_X, MK_ACC_READ, xb(l) + 4 * r0, xb(l) + 4 * r1));  // residual
            acc.push_back(A(B_X, MK_ACC_WRITE, xm + 4 * r0, xm + 4 * r1));
            if (fused) acc.push_back(A(B_X, MK_ACC_WRITE, xb(l + 1) + 4 * r0, xb(l + 1) + 4 * r1));
            ids.push_back(B.add_task(p.first, t, acc));
            tag_ok = tag_ok && has_qkv[p.first];
        }
        B.set_wait(ids, prev_ctr, (int)prev.size(), 0);
        // The attention tasks read q/k/v as tagged values and need no counter
        // when every later task of the layer sits on a CTA whose QKV task
        // already acquired the previous layer's results: then the tags order
        // nothing that the counter chain must carry.
        if (tag_ok) lw->ctr_buf[ctr(l, 0)] = B_QKV;
        prev = ids;
        prev_ctr = ctr(l, 2);

        if (fused) {
            // ---- fused FFN: each CTA owns blocks of BU hidden units (one 16-byte
            // column chunk of the down projection): their gate/up rows, SwiGLU
            // in shared memory, and their down-projection column block, added
            // into the next residual buffer
            ids.clear();
            const int64_t BU = ffn_block(d->wdtype);
            const int64_t blocks = F / BU, max_blocks = FFN_MAX_UNITS / BU;
            const int64_t block_bytes = BU * 2 * bl.row_gu + dm * 16;
            for (auto& p : B.split(blocks, block_bytes)) {
                for (int64_t b0 = p.second.first; b0 < p.second.second; b0 += max_blocks) {
                    const int64_t b1 = std::min(p.second.second, b0 + max_blocks);
                    const int64_t u0 = b0 * BU, u1 = b1 * BU;
                    DevTask t = gemv_task(OP_FFN, l, 2 * u0, 2 * (u1 - u0), dm, bl.row_gu, lb + bl.l_gu, 2, ctr(l, 3));
                    std::vector<mk_ir_access> acc;
                    acc.push_back(A(B_X, MK_ACC_READ, xm, xm + 4 * dm));
                    acc.push_back(A(B_X, MK_ACC_ATOMIC, xb(l + 1), xb(l + 1) + 4 * dm));
                    ids.push_back(B.add_task(p.first, t, acc));
                }
            }
            B.set_wait(ids, prev_ctr, (int)prev.size(), 0);
            prev = ids;
            prev_ctr = ctr(l, 3);
            continue;
        }

        // ---- gate/up (interleaved pairs) + SwiGLU
        ids.clear();
        for (auto& p : B.split(F, 2 * bl.row_gu)) {
            int64_t u0 = p.second.first, u1 = p.second.second;
            DevTask t = gemv_task(OP_GU, l, 2 * u0, 2 * (u1 - u0), dm, bl.row_gu, lb + bl.l_gu, 2, ctr(l, 3));
            std::vector<mk_ir_access> acc;
            acc.push_back(A(B_X, MK_ACC_READ, xm, xm + 4 * dm));
            acc.push_back(A(B_H, MK_ACC_WRITE, 4 * u0, 4 * u1));
            ids.push_back(B.add_task(p.first, t, acc));
        }
        B.set_wait(ids, prev_ctr, (int)prev.size(), 0);
        prev = ids;
        prev_ctr = ctr(l, 3);

        // ---- down + residual
        ids.clear();
        for (auto& p : B.split(dm, bl.row_down)) {
            int64_t r0 = p.second.first, r1 = p.second.second;
            DevTask t = gemv_task(OP_DOWN, l, r0, r1 - r0, F, bl.row_down, lb + bl.l_down, 1, ctr(l, 4));
            std::vector<mk_ir_access> acc;
            acc.push_back(A(B_H, MK_ACC_READ, 0, 4 * F));
            acc.push_back(A(B_X, MK_ACC_READ, xm + 4 * r0, xm + 4 * r1));  // residual: x_mid
            acc.push_back(A(B_X, MK_ACC_WRITE, 4 * r0, 4 * r1));
            ids.push_back(B.add_task(p.first, t, acc));
        }
        B.set_wait(ids, prev_ctr, (int)prev.size(), 0);
        prev = ids;
        prev_ctr = ctr(l, 4);
    }

    // ---- final norm + LM head + block argmax
    for (auto& p : B.split(V, bl.row_lm)) {
        int64_t r0 = p.second.first, r1 = p.second.second;
        DevTask t = gemv_task(OP_LM, L, r0, r1 - r0, dm, bl.row_lm, bl.lm, 1, CTR_LM);
        std::vector<mk_ir_access> acc;
        acc.push_back(A(B_X, MK_ACC_READ, xb(L), xb(L) + 4 * dm));
        acc.push_back(A(B_LOGITS, MK_ACC_WRITE, 4 * r0, 4 * r1, 4 * V, 0));
        acc.push_back(A(B_KEY, MK_ACC_ATOMIC, 0, 8));
        if (ts) acc.push_back(A(B_CAND, MK_ACC_WRITE, p.first * CAND_BYTES, (p.first + 1) * CAND_BYTES));
        lm_ids.push_back(B.add_task(p.first, t, acc));
        lw->lm_rows_max = std::max<int32_t>(lw->lm_rows_max, (int32_t)(r1 - r0));
    }
    B.set_wait(lm_ids, prev_ctr, (int)prev.size(), 0);

    // ---- read the key -> out id; on the CTA that starts the next step first.
    // Token-select schedules: OP_SELECT picks the token from every CTA's
    // candidates, publishes it and signals CTR_TOK.
    {
        DevTask t{};
        t.op = ts ? OP_SELECT : OP_FIN;
        t.layer = L;
        t.signal_ctr = ts ? CTR_TOK : -1;
        std::vector<mk_ir_access> acc;
        acc.push_back(A(B_KEY, MK_ACC_READ, 0, 8));
        acc.push_back(A(B_OUT, MK_ACC_WRITE, 0, 4, 4, 0));
        if (ts) {
            acc.push_back(A(B_CAND, MK_ACC_READ, 0, c.sms * CAND_BYTES));
            acc.push_back(A(B_TOKW, MK_ACC_WRITE, 0, 8));
        }
        int id = B.add_task(fin_sm, t, acc);
        B.set_wait({id}, CTR_LM, (int)lm_ids.size(), 0);
    }
    // The first layer of step e waits for the token of step e-1: the LM head's
    // argmax key, or the token-select task's word.
    if (ts) B.set_wait(first_qkv, CTR_TOK, 1, -1);
    else B.set_wait(first_qkv, CTR_LM, (int)lm_ids.size(), -1);
    lw->ctr_tok = ts ? CTR_TOK : CTR_LM;
    lw->n_tok = ts ? 1 : (int)lm_ids.size();

    for (size_t i = 0; i < lw->tasks.size(); ++i) {
        lw->tasks[i].acc_begin = (int32_t)lw->acc.size();
        lw->tasks[i].n_acc = (int32_t)B.tacc[i].size();
        lw->acc.insert(lw->acc.end(), B.tacc[i].begin(), B.tacc[i].end());
    }
    auto mm = std::minmax_element(B.load.begin(), B.load.end());
    lw->bytes_per_sm_min = *mm.first;
    lw->bytes_per_sm_max = *mm.second;
    return MK_OK;
}

mk_status device_tables(const Lowering& lw, int n_sms, std::vector<TaskRec>* recs, std::vector<int32_t>* queue,
                        std::vector<int32_t>* queue_off, int32_t* tab_cap) {
    recs->clear();
    queue->clear();
    queue_off->assign(n_sms + 1, 0);
    *tab_cap = 0;
    for (int s = 0; s < n_sms; ++s) {
        (*queue_off)[s] = (int32_t)queue->size();
        if (s < (int)lw.queues.size()) {
            *tab_cap = std::max(*tab_cap, (int32_t)lw.queues[s].size());
            for (int id : lw.queues[s]) queue->push_back(id);
        }
    }
    (*queue_off)[n_sms] = (int32_t)queue->size();
    for (int id : *queue) {
        DevTask t = lw.dev[id];
        // counters carried by tagged values exist only in the IR
        auto tagged = [&](int ctr) { return ctr >= 0 && ctr < (int)lw.ctr_buf.size() && lw.ctr_buf[ctr] >= 0; };
        if (tagged(t.signal_ctr)) t.signal_ctr = -1;
        for (int w = 0; w < t.n_waits;) {
            if (tagged(t.wait_ctr[w])) {
                for (int v = w; v + 1 < t.n_waits; ++v) {
                    t.wait_ctr[v] = t.wait_ctr[v + 1];
                    t.wait_cnt[v] = t.wait_cnt[v + 1];
                    t.wait_off[v] = t.wait_off[v + 1];
                }
                --t.n_waits;
            } else {
                ++w;
            }
        }
        TaskRec r{};
        bool fits = t.op >= 0 && t.op < 256 && t.layer >= 0 && t.layer < 65536 && t.n_waits >= 0 && t.n_waits <= 2 &&
                    t.w_off >= 0 && (t.w_off & 15) == 0 && (t.w_off >> 4) <= 0xFFFFFFFFll && t.row_bytes >= 0 &&
                    (t.row_bytes & 15) == 0 && (t.row_bytes >> 4) < 65536 && t.K >= 0 && t.K < 65536 &&
                    t.signal_ctr >= -1 && t.signal_ctr < 32768 && t.wpr >= 0 && t.wpr < 256;
        for (int w = 0; w < t.n_waits && fits; ++w)
            fits = t.wait_ctr[w] >= 0 && t.wait_ctr[w] < 65536 && t.wait_cnt[w] >= 0 && t.wait_cnt[w] < 65536 &&
                   (t.wait_off[w] == 0 || t.wait_off[w] == -1);
        if (!fits) {
            set_error("task %d does not fit the device record (blob offset above 64 GiB or a field out of range)", id);
            return MK_ERR_INVALID_ARG;
        }
        r.op = (uint8_t)t.op;
        r.n_waits = (uint8_t)t.n_waits;
        r.layer = (uint16_t)t.layer;
        r.row0 = t.row0;
        r.nrows = t.nrows;
        r.w_off16 = (uint32_t)(t.w_off >> 4);
        r.row_bytes16 = (uint16_t)(t.row_bytes >> 4);
        r.K = (uint16_t)t.K;
        for (int w = 0; w < t.n_waits; ++w) {
            r.wait_ctr[w] = (uint16_t)t.wait_ctr[w];
            r.wait_cnt[w] = (uint16_t)t.wait_cnt[w];
            if (t.wait_off[w] == -1) r.wait_prev |= (uint8_t)(1u << w);
        }
        r.signal_ctr = (int16_t)t.signal_ctr;
        r.wpr = (uint8_t)t.wpr;
        recs->push_back(r);
    }
    return MK_OK;
}

mk_ir* to_ir(const Lowering& lw, int n_sms) {
    mk_ir* ir = new mk_ir{};
    ir->n_sms = n_sms;
    ir->n_tasks = (int32_t)lw.tasks.size();
    ir->n_counters = lw.n_counters;
    ir->n_buffers = B_COUNT;
    ir->n_acc = (int32_t)lw.acc.size();
    ir->tasks = new mk_ir_task[std::max<size_t>(1, lw.tasks.size())];
    std::copy(lw.tasks.begin(), lw.tasks.end(), ir->tasks);
    ir->acc = new mk_ir_access[std::max<size_t>(1, lw.acc.size())];
    std::copy(lw.acc.begin(), lw.acc.end(), ir->acc);
    ir->queue = new int32_t[std::max<size_t>(1, lw.tasks.size())];
    ir->queue_off = new int32_t[n_sms + 1];
    int32_t o = 0;
    for (int s = 0; s < n_sms; ++s) {
        ir->queue_off[s] = o;
        if (s < (int)lw.queues.size())
            for (int id : lw.queues[s]) ir->queue[o++] = id;
    }
    ir->queue_off[n_sms] = o;
    ir->buf_flags = new int32_t[B_COUNT]();
    ir->buf_flags[B_LOGITS] = MK_BUF_OUTPUT;
    ir->buf_flags[B_OUT] = MK_BUF_OUTPUT;
    ir->ctr_buf = new int32_t[std::max(1, lw.n_counters)];
    for (int k = 0; k < lw.n_counters; ++k) ir->ctr_buf[k] = k < (int)lw.ctr_buf.size() ? lw.ctr_buf[k] : -1;
    return ir;
}

WsLayout ws_layout(const mk_model_desc* d, const Config& c, int64_t n_tasks, int32_t n_counters) {
    WsLayout w{};
    int64_t o = 0;
    auto take = [&](int64_t bytes) {
        int64_t at = o;
        o = up(o + bytes, 256);
        return at;
    };
    const int64_t qd = (int64_t)d->n_q_heads * d->head_dim, kd = (int64_t)d->n_kv_heads * d->head_dim;
    w.status = take(256);
    w.counters = take((int64_t)n_counters * CTR_STRIDE * 4);
    w.key = take(64);
    w.tokw = take(64);
    w.cand = take((int64_t)c.sms * MAX_TOP_K * 8);
    w.recs = take(n_tasks * (int64_t)sizeof(TaskRec));
    w.queue_off = take((int64_t)(c.sms + 1) * 4);
    w.inv_freq = take((int64_t)d->head_dim / 2 * 4);
    w.x = take((int64_t)d->d_model * 3 * 4);  // x[2][d], x_mid[d]
    w.qkv = take((qd + 2 * kd) * 8);  // tagged values
    w.part_ml = take((int64_t)PART_COPIES * d->n_q_heads * c.C * 2 * 4);
    w.att = take((int64_t)PART_COPIES * d->n_q_heads * d->head_dim * 4);
    w.part_acc = take((int64_t)PART_COPIES * d->n_q_heads * c.C * d->head_dim * 2);  // fp16
    w.h = take((int64_t)d->d_ffn * 4);
    w.tok = take((int64_t)d->max_seq * 4 + 16);
    w.out_ids = take((int64_t)d->max_seq * 4 + 16);
    if (c.pf_chunk > 0) {  // one chunk's activations
        const int64_t mc = c.pf_chunk;
        w.pf_x = take(mc * d->d_model * 4);
        w.pf_q = take(mc * qd * 4);
        w.pf_h = take(mc * d->d_model * 2);
        w.pf_hl = take(mc * d->d_model * 2);
        w.pf_ao = take(mc * qd * 2);
        w.pf_aol = take(mc * qd * 2);
        w.pf_gu = take(mc * d->d_ffn * 2);
        w.pf_gul = take(mc * d->d_ffn * 2);
        w.pf_err = take(16);
    }
    w.total = o;
    return w;
}

}  // namespace mk

using namespace mk;

extern "C" {

mk_status mk_build_ir(const mk_model_desc* desc, const mk_schedule_config* cfg, int32_t n_sms,
                      mk_ir** out) {
    mk_status st = check_desc(desc);
    if (st) return st;
    if (!out) {
        set_error("out is NULL");
        return MK_ERR_INVALID_ARG;
    }
    Config c;
    if ((st = resolve_config(desc, cfg, n_sms, &c))) return st;
    Lowering lw;
    if ((st = lower(desc, c, &lw))) return st;
    *out = to_ir(lw, c.sms);
    return MK_OK;
}

void mk_free_ir(mk_ir* ir) {
    if (!ir) return;
    delete[] ir->tasks;
    delete[] ir->acc;
    delete[] ir->queue;
    delete[] ir->queue_off;
    delete[] ir->buf_flags;
    delete[] ir->ctr_buf;
    delete ir;
}

}  // extern "C"
