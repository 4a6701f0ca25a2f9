// Continuous-batching scheduler (host code only): requests wait in a FIFO
// queue, are admitted into free KV-cache slots between decode steps and
// leave their slot when they finish, so a batch keeps up to max_batch
// sequences in flight while others come and go.  The per-sequence
// positions it hands out are the ones the decode step already takes (each
// row carries its own sequence slot and position: "Model-agnostic LLM
// inference", section "Supported models" runs each sequence at its own
// position; "LLM inference overview", section "Workload characteristics":
// one weight sweep per step serves every sequence in the batch).
//
// One step of the caller's loop:
//   plan           -> requests to admit (with their slots) and the decode rows
//   prefill admits -> complete_prefill(first token of each admitted request)
//   decode rows    -> complete_step(next token of each row)
// A request is finished after max_new_tokens tokens or at eos_id (kept);
// its slot is free from then on.
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <deque>
#include <new>
#include <string>
#include <vector>

#include "../../include/q3i8.h"

int q3_report_error(int code, const char* msg);  // engine.cu

namespace {

struct Req {
    std::vector<int32_t> prompt;
    int32_t max_new = 0, eos = -1;
    int32_t slot = -1;
    enum State { kQueued, kPrefill, kDecoding, kDone } state = kQueued;
    std::vector<int32_t> out;  // generated tokens
};

int report(int code, const std::string& msg) { return q3_report_error(code, msg.c_str()); }

}  // namespace

struct q3i8_sched {
    int32_t max_batch = 0, max_ctx = 0;
    std::vector<Req> reqs;
    std::deque<int32_t> queue;          // request ids waiting for a slot
    std::vector<int32_t> slot_req;      // slot -> request id, -1 = free
    std::vector<int32_t> pending_fill;  // admitted, prefill result not reported yet
    std::vector<int32_t> rows;          // request ids of the last plan's decode rows
    bool step_open = false;             // a plan's decode rows await complete_step

    void finish_if_done(Req& r) {
        if ((int32_t)r.out.size() >= r.max_new || (r.eos >= 0 && r.out.back() == r.eos)) {
            r.state = Req::kDone;
            slot_req[r.slot] = -1;
        }
    }
};

// Accessors for the device serving loop (engine.cu).
int q3_sched_slots(const q3i8_sched* s) { return s->max_batch; }
int q3_sched_max_ctx(const q3i8_sched* s) { return s->max_ctx; }
const int32_t* q3_sched_prompt(const q3i8_sched* s, int request_id, int32_t* len) {
    if (request_id < 0 || request_id >= (int)s->reqs.size()) {
        *len = 0;
        return nullptr;
    }
    const Req& r = s->reqs[request_id];
    *len = (int32_t)r.prompt.size();
    return r.prompt.data();
}

extern "C" int q3i8_sched_new(int32_t max_batch, int32_t max_ctx, q3i8_sched** out) {
    if (!out) return report(Q3_ERR_INVALID_ARGUMENTS, "sched_new: NULL out");
    if (max_batch < 1 || max_ctx < 2)
        return report(Q3_ERR_INVALID_ARGUMENTS, "sched_new: max_batch must be >= 1 and max_ctx >= 2");
    q3i8_sched* s = new (std::nothrow) q3i8_sched;
    if (!s) return report(Q3_ERR_OOM, "sched_new: out of host memory");
    s->max_batch = max_batch;
    s->max_ctx = max_ctx;
    s->slot_req.assign(max_batch, -1);
    *out = s;
    return Q3_OK;
}

extern "C" void q3i8_sched_destroy(q3i8_sched* s) { delete s; }

extern "C" int q3i8_sched_submit(q3i8_sched* s, const int32_t* prompt, int32_t prompt_len, int32_t max_new_tokens,
                                 int32_t eos_id, int32_t* request_id) {
    if (!s || !prompt || !request_id) return report(Q3_ERR_INVALID_ARGUMENTS, "sched_submit: NULL argument");
    if (prompt_len < 1) return report(Q3_ERR_INVALID_ARGUMENTS, "sched_submit: empty prompt");
    if (max_new_tokens < 1) return report(Q3_ERR_INVALID_ARGUMENTS, "sched_submit: max_new_tokens must be >= 1");
    // the last generated token is never fed back, so a sequence holds
    // prompt_len + max_new_tokens - 1 positions
    if ((long long)prompt_len + max_new_tokens - 1 > s->max_ctx) {
        char buf[160];
        snprintf(buf, sizeof buf, "sched_submit: prompt %d + %d new tokens exceed the %d-position slots", prompt_len,
                 max_new_tokens, s->max_ctx);
        return report(Q3_ERR_CONTEXT, buf);
    }
    Req r;
    r.prompt.assign(prompt, prompt + prompt_len);
    r.max_new = max_new_tokens;
    r.eos = eos_id;
    *request_id = (int32_t)s->reqs.size();
    s->reqs.push_back(std::move(r));
    s->queue.push_back(*request_id);
    return Q3_OK;
}

extern "C" int q3i8_sched_plan(q3i8_sched* s, int32_t* n_admit, int32_t* admit_req, int32_t* admit_slot,
                               int32_t* n_rows, int32_t* row_req, int32_t* row_slot, int32_t* row_pos,
                               int32_t* row_token) {
    if (!s || !n_admit || !admit_req || !admit_slot || !n_rows || !row_req || !row_slot || !row_pos || !row_token)
        return report(Q3_ERR_INVALID_ARGUMENTS, "sched_plan: NULL argument");
    if (!s->pending_fill.empty() || s->step_open)
        return report(Q3_ERR_STATE, "sched_plan: the previous plan's prefill or step was not completed");
    // decode rows: every sequence in flight, in slot order; its last token at
    // the next position (prompt_len + tokens generated - 1)
    int nr = 0;
    s->rows.clear();
    for (int slot = 0; slot < s->max_batch; ++slot) {
        const int32_t id = s->slot_req[slot];
        if (id < 0) continue;
        const Req& r = s->reqs[id];
        row_req[nr] = id;
        row_slot[nr] = slot;
        row_pos[nr] = (int32_t)(r.prompt.size() + r.out.size() - 1);
        row_token[nr] = r.out.back();
        s->rows.push_back(id);
        ++nr;
    }
    // admissions: the queue's head into the lowest free slots
    int na = 0;
    for (int slot = 0; slot < s->max_batch && !s->queue.empty(); ++slot) {
        if (s->slot_req[slot] >= 0) continue;
        const int32_t id = s->queue.front();
        s->queue.pop_front();
        Req& r = s->reqs[id];
        r.slot = slot;
        r.state = Req::kPrefill;
        s->slot_req[slot] = id;
        admit_req[na] = id;
        admit_slot[na] = slot;
        s->pending_fill.push_back(id);
        ++na;
    }
    *n_admit = na;
    *n_rows = nr;
    s->step_open = nr > 0;
    return Q3_OK;
}

extern "C" int q3i8_sched_complete_prefill(q3i8_sched* s, int32_t n, const int32_t* request_ids,
                                           const int32_t* first_tokens) {
    if (!s || (n > 0 && (!request_ids || !first_tokens)))
        return report(Q3_ERR_INVALID_ARGUMENTS, "sched_complete_prefill: NULL argument");
    for (int i = 0; i < n; ++i) {
        const int32_t id = request_ids[i];
        auto it = std::find(s->pending_fill.begin(), s->pending_fill.end(), id);
        if (it == s->pending_fill.end())
            return report(Q3_ERR_STATE, "sched_complete_prefill: request " + std::to_string(id) +
                                            " is not waiting for its prefill");
        s->pending_fill.erase(it);
        Req& r = s->reqs[id];
        r.out.push_back(first_tokens[i]);
        r.state = Req::kDecoding;
        s->finish_if_done(r);
    }
    return Q3_OK;
}

extern "C" int q3i8_sched_complete_step(q3i8_sched* s, int32_t n_rows, const int32_t* tokens) {
    if (!s || (n_rows > 0 && !tokens)) return report(Q3_ERR_INVALID_ARGUMENTS, "sched_complete_step: NULL argument");
    if (!s->step_open && n_rows == 0) return Q3_OK;  // the plan had no rows
    if (!s->step_open || n_rows != (int32_t)s->rows.size())
        return report(Q3_ERR_STATE, "sched_complete_step: the row count does not match the last plan");
    for (int i = 0; i < n_rows; ++i) {
        Req& r = s->reqs[s->rows[i]];
        r.out.push_back(tokens[i]);
        s->finish_if_done(r);
    }
    s->rows.clear();
    s->step_open = false;
    return Q3_OK;
}

extern "C" int32_t q3i8_sched_idle(const q3i8_sched* s) {
    if (!s) return 1;
    if (!s->queue.empty() || !s->pending_fill.empty() || s->step_open) return 0;
    for (int32_t id : s->slot_req)
        if (id >= 0) return 0;
    return 1;
}

extern "C" int q3i8_sched_result(const q3i8_sched* s, int32_t request_id, int32_t* tokens, int32_t cap,
                                 int32_t* n_tokens, int32_t* done) {
    if (!s || !n_tokens || !done || (cap > 0 && !tokens))
        return report(Q3_ERR_INVALID_ARGUMENTS, "sched_result: NULL argument");
    if (request_id < 0 || request_id >= (int32_t)s->reqs.size())
        return report(Q3_ERR_INVALID_ARGUMENTS, "sched_result: unknown request id");
    const Req& r = s->reqs[request_id];
    const int32_t n = (int32_t)r.out.size();
    if (cap > 0) memcpy(tokens, r.out.data(), sizeof(int32_t) * (size_t)std::min(n, cap));
    *n_tokens = n;
    *done = r.state == Req::kDone ? 1 : 0;
    return Q3_OK;
}
