// Rounds fed from host memory: a caller-owned session holds two device sets of a
// round's inputs, the device tree, results and workspace, and a copy stream. The
// caller stages the inputs of the next round (host -> device on the copy stream,
// into the set no round is reading) while the current round runs; each round's
// results go back to host memory on the round's stream right after it. One round
// is dartree_round (DARTree blog post, 3.1 and 3.2: build, prune, verify).
#include <cuda_runtime.h>

#include <new>

#include "dartree.h"

struct dartree_host_session {
    dartree_head head;
    dartree_params p;
    int rows;
    size_t in_bytes[4];  // base logits, block hidden, anchor, target
    void* in[2][4];      // the two device input sets
    dartree_tree tree;
    int32_t* acc;
    int32_t* path;
    int32_t* bonus;
    void* ws;
    size_t ws_bytes;
    void* block;  // the one device allocation holding all of the above
    cudaStream_t copy;
    cudaEvent_t ready[2];  // set b staged
    cudaEvent_t freed[2];  // the round that read set b and its result copies finished
    bool used[2];
    long staged, ran;
};

namespace {

size_t round_up(size_t x) { return (x + 255) / 256 * 256; }

void release(dartree_host_session* s) {
    if (!s) return;
    for (int b = 0; b < 2; ++b) {
        if (s->ready[b]) cudaEventDestroy(s->ready[b]);
        if (s->freed[b]) cudaEventDestroy(s->freed[b]);
    }
    if (s->copy) cudaStreamDestroy(s->copy);
    if (s->block) cudaFree(s->block);
    delete s;
}

}  // namespace

extern "C" {

int dartree_host_session_create(const dartree_head* head, const dartree_params* p, int rows,
                                dartree_host_session** out) {
    if (!head || !p || !out || !head->E || !head->Wq) return DARTREE_EINVAL;
    *out = nullptr;
    if (rows != DARTREE_ROWS_PER_POSITION && rows != DARTREE_ROWS_PER_NODE) return DARTREE_EDTYPE;
    if (head->dtype != DARTREE_F32 && head->dtype != DARTREE_BF16) return DARTREE_EDTYPE;
    if (p->C < 1) return DARTREE_EINVAL;
    const size_t ws = dartree_workspace_bytes(p, head->V, head->H, head->dtype);
    if (ws == 0) return DARTREE_EINVAL;  // shape rejected by the round's own checks
    const size_t es = head->dtype == DARTREE_BF16 ? 2 : 4;
    const size_t C = size_t(p->C), L = size_t(p->L), S = size_t(p->B) + 1, V = size_t(head->V),
                 H = size_t(head->H);
    dartree_host_session* s = new (std::nothrow) dartree_host_session{};
    if (!s) return DARTREE_EINVAL;
    s->head = *head;
    s->p = *p;
    s->rows = rows;
    s->in_bytes[0] = C * L * V * es;
    s->in_bytes[1] = C * L * H * es;
    s->in_bytes[2] = C * 4;
    s->in_bytes[3] = (rows == DARTREE_ROWS_PER_POSITION ? C * L : C * S) * V * es;
    s->ws_bytes = ws;
    // layout of the one allocation
    size_t off = 0;
    size_t in_off[2][4];
    for (int b = 0; b < 2; ++b)
        for (int k = 0; k < 4; ++k) {
            in_off[b][k] = off;
            off += round_up(s->in_bytes[k]);
        }
    const size_t o_tok = off; off += round_up(C * S * 4);
    const size_t o_par = off; off += round_up(C * S * 4);
    const size_t o_dep = off; off += round_up(C * S * 4);
    const size_t o_sco = off; off += round_up(C * S * 4);
    const size_t o_nn = off; off += round_up(C * 4);
    const size_t o_mask = off; off += round_up(C * S * S);
    const size_t o_pos = off; off += round_up(C * S * 4);
    const size_t o_acc = off; off += round_up(C * 4);
    const size_t o_path = off; off += round_up(C * L * 4);
    const size_t o_bonus = off; off += round_up(C * 4);
    const size_t o_ws = off; off += round_up(ws);
    if (cudaMalloc(&s->block, off) != cudaSuccess) {
        cudaGetLastError();
        s->block = nullptr;
        release(s);
        return DARTREE_ECUDA;
    }
    uint8_t* base = static_cast<uint8_t*>(s->block);
    for (int b = 0; b < 2; ++b)
        for (int k = 0; k < 4; ++k) s->in[b][k] = base + in_off[b][k];
    s->tree = dartree_tree{reinterpret_cast<int32_t*>(base + o_tok), reinterpret_cast<int32_t*>(base + o_par),
                           reinterpret_cast<int32_t*>(base + o_dep), reinterpret_cast<float*>(base + o_sco),
                           reinterpret_cast<int32_t*>(base + o_nn), base + o_mask,
                           reinterpret_cast<int32_t*>(base + o_pos)};
    s->acc = reinterpret_cast<int32_t*>(base + o_acc);
    s->path = reinterpret_cast<int32_t*>(base + o_path);
    s->bonus = reinterpret_cast<int32_t*>(base + o_bonus);
    s->ws = base + o_ws;
    bool ok = cudaStreamCreateWithFlags(&s->copy, cudaStreamNonBlocking) == cudaSuccess;
    for (int b = 0; b < 2 && ok; ++b)
        ok = cudaEventCreateWithFlags(&s->ready[b], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&s->freed[b], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        release(s);
        return DARTREE_ECUDA;
    }
    *out = s;
    return DARTREE_OK;
}

void dartree_host_session_destroy(dartree_host_session* s) {
    if (!s) return;
    // the session's memory is freed only once no copy or round uses it
    cudaStreamSynchronize(s->copy);
    for (int b = 0; b < 2; ++b)
        if (s->used[b]) cudaEventSynchronize(s->freed[b]);
    cudaGetLastError();
    release(s);
}

int dartree_host_stage(dartree_host_session* s, const dartree_host_inputs* in) {
    if (!s || !in || !in->base_logits || !in->block_hidden || !in->anchor || !in->target) return DARTREE_EINVAL;
    if (s->staged - s->ran >= 2) return DARTREE_EINVAL;  // both sets hold inputs no round has read yet
    const int b = int(s->staged % 2);
    if (s->used[b] && cudaStreamWaitEvent(s->copy, s->freed[b], 0) != cudaSuccess) return DARTREE_ECUDA;
    const void* src[4] = {in->base_logits, in->block_hidden, in->anchor, in->target};
    for (int k = 0; k < 4; ++k)
        if (cudaMemcpyAsync(s->in[b][k], src[k], s->in_bytes[k], cudaMemcpyHostToDevice, s->copy) != cudaSuccess)
            return DARTREE_ECUDA;
    if (cudaEventRecord(s->ready[b], s->copy) != cudaSuccess) return DARTREE_ECUDA;
    ++s->staged;
    return DARTREE_OK;
}

int dartree_host_round(dartree_host_session* s, const dartree_host_outputs* out, void* stream) {
    if (!s || !out || !out->accepted_len || !out->path || !out->bonus) return DARTREE_EINVAL;
    if (s->ran >= s->staged) return DARTREE_EINVAL;  // nothing staged
    const int b = int(s->ran % 2);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamWaitEvent(st, s->ready[b], 0) != cudaSuccess) return DARTREE_ECUDA;
    void* const* x = s->in[b];
    if (int e = dartree_round(&s->head, &s->p, x[0], x[1], static_cast<const int32_t*>(x[2]), x[3], s->rows,
                              &s->tree, s->acc, s->path, s->bonus, s->ws, s->ws_bytes, stream)) {
        // (work the call enqueued before failing may still read set b)
        if (cudaEventRecord(s->freed[b], st) == cudaSuccess) s->used[b] = true;
        return e;
    }
    ++s->ran;
    const size_t C = size_t(s->p.C), L = size_t(s->p.L);
    int rc = DARTREE_OK;
    if (cudaMemcpyAsync(out->accepted_len, s->acc, C * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyAsync(out->path, s->path, C * L * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyAsync(out->bonus, s->bonus, C * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        rc = DARTREE_ECUDA;
    // set b may be refilled (and the session freed) once the round and these copies are
    // done (recorded after whatever was enqueued, also when a copy failed)
    if (cudaEventRecord(s->freed[b], st) != cudaSuccess) rc = DARTREE_ECUDA;
    s->used[b] = true;
    return rc;
}

size_t dartree_host_input_bytes(const dartree_host_session* s, int which) {
    if (!s || which < 0 || which > 3) return 0;
    return s->in_bytes[which];
}

}  // extern "C"
