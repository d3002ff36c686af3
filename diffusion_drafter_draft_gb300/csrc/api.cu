// C ABI of the DARTree draft-tree build and verify step: argument checks,
// workspace carving and kernel launches on the caller's stream.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "dartree.h"
#include "kernels.h"

#include <mutex>

namespace {

using namespace dartree;

constexpr size_t kAlign = 256;
constexpr int kMaxGRows = 8192;   // candidate rows of the candidate-side projection path

size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Layout {
    size_t status, cand_tok, cand_val, h[2], s[2], U, z, st_tok, st_par, st_s, st_n, keys, uhl, Eg, Ghi, Glo, total;
    int g_rows;
};

Layout layout_of(const dartree_params& p, int H, int dtype) {
    const size_t C = size_t(p.C), L = size_t(p.L), K = size_t(p.K), W = size_t(p.W), B = size_t(p.B);
    const size_t elem = dtype == DARTREE_BF16 ? 2 : 4;
    Layout l{};
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o += up(bytes); return at; };
    l.status = take(4);
    l.cand_tok = take(C * L * K * 4);
    l.cand_val = take(C * L * K * 4);
    l.h[0] = take(C * W * size_t(H) * elem);
    l.h[1] = take(C * W * size_t(H) * elem);
    l.s[0] = take(C * W * 4);
    l.s[1] = take(C * W * 4);
    l.U = take(C * W * size_t(H) * 4);
    l.z = take(C * W * K * 4);
    l.st_tok = take(C * L * W * 4);
    l.st_par = take(C * L * W * 4);
    l.st_s = take(C * L * W * 4);
    l.st_n = take(C * L * 4);
    l.keys = take((C * L > C * (B + 1) ? C * L : C * (B + 1)) * 8);
    // bf16 hi/lo projection rows for the tensor-core contraction, [C, 32, H]
    l.uhl = take(dtype == DARTREE_BF16 ? C * 32 * size_t(H) * 2 : 0);
    // candidate-side projection path (prepared bf16 heads, small batches): gathered
    // candidate rows and G = E[cand] W_q as a bf16 pair, [C*L*K, H] each
    const size_t g = C * L * K;
    l.g_rows = (dtype == DARTREE_BF16 && K <= 64 && W <= 16 && g <= size_t(kMaxGRows)) ? int(g) : 0;
    l.Eg = take(size_t(l.g_rows) * H * 2);
    l.Ghi = take(size_t(l.g_rows) * H * 2);
    l.Glo = take(size_t(l.g_rows) * H * 2);
    l.total = o;
    return l;
}

bool dtype_ok(int dt) { return dt == DARTREE_F32 || dt == DARTREE_BF16; }

int check_params(const dartree_params* p, int V, int H, int dtype) {
    if (!p) return DARTREE_EINVAL;
    if (!dtype_ok(dtype)) return DARTREE_EDTYPE;
    if (p->C < 0 || p->L < 1 || p->K < 1 || p->W < 1 || p->B < 1 || V < 1 || H < 8) return DARTREE_EINVAL;
    if (H % 8 != 0) return DARTREE_EINVAL;
    if (!(p->beta <= 0.0f)) return DARTREE_EINVAL;  // also rejects NaN
    if (p->K > V) return DARTREE_EINVAL;
    if (p->B > p->L * p->W) return DARTREE_EINVAL;
    if (p->L > DARTREE_MAX_L || p->K > DARTREE_MAX_K || p->W > DARTREE_MAX_W || p->B + 1 > DARTREE_MAX_SLOTS ||
        p->W * p->K > DARTREE_MAX_CHILDREN)
        return DARTREE_EUNSUPPORTED;
    return DARTREE_OK;
}

int check_ws(const void* ws, size_t have, size_t need) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0 || have < need) return DARTREE_EWORKSPACE;
    return DARTREE_OK;
}

template <typename P>
P* at(void* ws, size_t off) { return reinterpret_cast<P*>(static_cast<uint8_t*>(ws) + off); }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// S8 + S9 from a supertree: the fused one-CTA-per-request kernel when the
// supertree holds at most 256 nodes, else the radix prune and the mask kernel.
int finish_tree(const dartree_params* p, const dartree_supertree* sp, const int32_t* anchor, dartree_tree* tree,
                int* status, cudaStream_t s) {
    if (finish_supported(p->L, p->W))
        return launch_finish(p->C, p->L, p->W, p->B, sp->tok, sp->par, sp->score, sp->n, anchor, tree->tok,
                             tree->par, tree->depth, tree->score, tree->n_nodes, tree->mask, tree->pos, nullptr,
                             nullptr, nullptr, nullptr, status, s, true);
    if (int e = launch_prune(p->C, p->L, p->W, p->B, sp->tok, sp->par, sp->score, sp->n, anchor, tree->tok, tree->par,
                             tree->depth, tree->score, tree->n_nodes, status, s))
        return e;
    if (tree->mask)
        return launch_mask(p->C, p->L, p->B, tree->par, tree->depth, tree->n_nodes, tree->mask, tree->pos, s);
    return DARTREE_OK;
}

// Workspace of the node-by-node heap search: status, candidate table, gathered
// candidate rows and the G pair, and the popped nodes' states.
struct HeapLayout {
    size_t status, cand_tok, cand_val, Eg, Ghi, Glo, hws, total;
};
HeapLayout heap_layout(const dartree_params& p, int H) {
    const size_t C = size_t(p.C), L = size_t(p.L), K = size_t(p.K), B = size_t(p.B), g = C * L * K;
    HeapLayout l{};
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o += up(bytes); return at; };
    l.status = take(4);
    l.cand_tok = take(g * 4);
    l.cand_val = take(g * 4);
    l.Eg = take(g * size_t(H) * 2);
    l.Ghi = take(g * size_t(H) * 2);
    l.Glo = take(g * size_t(H) * 2);
    l.hws = take(C * B * size_t(H) * 2);
    l.total = o;
    return l;
}

int check_heap(const dartree_head* head, const dartree_params* p) {
    if (!head || !p) return DARTREE_EINVAL;
    if (head->dtype != DARTREE_BF16) return DARTREE_EUNSUPPORTED;
    if (p->C < 0 || p->L < 1 || p->K < 1 || p->B < 1 || p->K > head->V) return DARTREE_EINVAL;
    if (!(p->beta <= 0.0f)) return DARTREE_EINVAL;
    // (the G GEMM's shape rule: N = H a multiple of 128; the row gather: H <= 6144)
    if (p->L > DARTREE_MAX_L || !heap_supported(head->H, p->K, p->B) || head->H % 128 != 0 || head->H / 8 > 768)
        return DARTREE_EUNSUPPORTED;
    return DARTREE_OK;
}

}  // namespace

extern "C" {

size_t dartree_heap_workspace_bytes(const dartree_params* p, int V, int H, int dtype) {
    dartree_head h{};
    h.V = V;
    h.H = H;
    h.dtype = dtype;
    if (H < 8 || H % 8 != 0 || check_heap(&h, p) != DARTREE_OK) return 0;
    return heap_layout(*p, H).total;
}

int dartree_heap_build(const dartree_head* head, const dartree_params* p, const void* base_logits,
                       const void* block_hidden, const int32_t* anchor, int32_t* tok, int32_t* parent, int32_t* depth,
                       float* score, void* ws, size_t ws_bytes, void* stream) {
    if (int e = check_heap(head, p)) return e;
    if (p->C == 0) return DARTREE_OK;
    if (!head->E || !head->WqT || !base_logits || !block_hidden || !anchor || !tok || !parent || !depth || !score)
        return DARTREE_EINVAL;
    const HeapLayout l = heap_layout(*p, head->H);
    if (int e = check_ws(ws, ws_bytes, l.total)) return e;
    cudaStream_t s = as_stream(stream);
    int* status = at<int>(ws, l.status);
    int32_t* ct = at<int32_t>(ws, l.cand_tok);
    float* cv = at<float>(ws, l.cand_val);
    uint16_t* Eg = at<uint16_t>(ws, l.Eg);
    const int M = p->C * p->L * p->K;
    // S1 (the same launch copies the candidates' rows when it can), then G = E[cand] W_q
    const TopkGather g{static_cast<const uint16_t*>(head->E), head->H, Eg, head->WqT,
                       reinterpret_cast<uintptr_t>(head->WqT) % 16 == 0 ? size_t(head->H) * head->H * 2 : 0};
    bool gathered = false;
    if (int e = launch_topk(base_logits, p->C * p->L, head->V, p->K, head->dtype, ct, cv, status, s, &g, &gathered))
        return e;
    if (!gathered)
        if (int e = launch_gather_rows(static_cast<const uint16_t*>(head->E), ct, head->H, M, Eg, s)) return e;
    if (int e = launch_gemm_bf16_tc(Eg, head->WqT, M, head->H, head->H, 2, nullptr, at<uint16_t>(ws, l.Ghi), 1,
                                    status, s, at<uint16_t>(ws, l.Glo), true))
        return e;
    return launch_heap_search(head->E, block_hidden, anchor, ct, cv, at<uint16_t>(ws, l.Ghi), at<uint16_t>(ws, l.Glo),
                              p->C, head->H, p->L, p->K, p->B, p->beta, at<uint16_t>(ws, l.hws), tok, parent, depth,
                              score, status, s);
}

const char* dartree_status_string(int s) {
    switch (s) {
        case DARTREE_OK: return "ok";
        case DARTREE_EINVAL: return "invalid argument";
        case DARTREE_EDTYPE: return "unknown dtype or row mode";
        case DARTREE_EWORKSPACE: return "workspace null, misaligned or too small";
        case DARTREE_ECUDA: return "CUDA call or launch failed";
        case DARTREE_ETIMEOUT: return "a bounded device-side wait ran out";
        case DARTREE_EINTERNAL: return "device-side consistency check failed";
        case DARTREE_EUNSUPPORTED: return "sizes beyond the library limits";
        default: return "unknown status";
    }
}

int dartree_head_init(dartree_head* head, const void* E, const void* Wq, int V, int H, int dtype) {
    if (!head || !E || !Wq || V < 1 || H < 8 || H % 8 != 0) return DARTREE_EINVAL;
    if (!dtype_ok(dtype)) return DARTREE_EDTYPE;
    head->E = E;
    head->Wq = Wq;
    head->V = V;
    head->H = H;
    head->dtype = dtype;
    head->WqT = nullptr;
    return DARTREE_OK;
}

int dartree_head_prepare(dartree_head* head, void* wqt, void* stream) {
    if (!head || !head->Wq || !wqt || head->H < 8 || (reinterpret_cast<uintptr_t>(wqt) % 16) != 0)
        return DARTREE_EINVAL;
    if (head->dtype != DARTREE_BF16) return DARTREE_EUNSUPPORTED;
    if (int e = launch_transpose_bf16(head->Wq, wqt, head->H, as_stream(stream))) return e;
    head->WqT = wqt;
    return DARTREE_OK;
}

size_t dartree_workspace_bytes(const dartree_params* p, int V, int H, int dtype) {
    if (check_params(p, V, H, dtype) != DARTREE_OK) return 0;
    return layout_of(*p, H, dtype).total;
}

int dartree_read_status(const void* ws, int32_t* status, void* stream) {
    if (!ws || !status) return DARTREE_EINVAL;
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, as_stream(stream)) != cudaSuccess)
        return DARTREE_ECUDA;
    if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return DARTREE_ECUDA;
    *status = v;
    return DARTREE_OK;
}

int dartree_clear_status(void* ws, void* stream) {
    if (!ws) return DARTREE_EINVAL;
    return cudaMemsetAsync(ws, 0, sizeof(int32_t), as_stream(stream)) == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

int dartree_selftest_wait(void* ws, size_t ws_bytes, int which, unsigned limit_us, void* stream) {
    if (which != 0 && which != 1) return DARTREE_EINVAL;
    if (limit_us < 1 || limit_us > 1000000u) return DARTREE_EINVAL;
    if (int e = check_ws(ws, ws_bytes, 2 * kAlign)) return e;
    return launch_selftest_wait(which, at<unsigned>(ws, kAlign), at<int>(ws, 0), uint64_t(limit_us) * 1000ull,
                                as_stream(stream));
}

int dartree_gemm_bf16(const void* A, const void* B, float* D, int M, int N, int K, int32_t* status, void* stream) {
    if (!A || !B || !D || M < 1 || N < 1 || K < 1) return DARTREE_EINVAL;
    if (!gemm_tc_supported(M, N, K)) return DARTREE_EUNSUPPORTED;
    return launch_gemm_bf16_tc(A, B, M, N, K, 0, D, nullptr, 1, status, as_stream(stream));
}

int dartree_topk(const void* logits, int rows, int V, int K, int dtype, int32_t* tok, float* val, void* ws,
                 size_t ws_bytes, void* stream) {
    if (!dtype_ok(dtype)) return DARTREE_EDTYPE;
    if (rows < 0 || V < 1 || K < 1 || K > V) return DARTREE_EINVAL;
    if (K > DARTREE_MAX_K) return DARTREE_EUNSUPPORTED;
    if (rows > 0 && (!logits || !tok || !val)) return DARTREE_EINVAL;
    if (int e = check_ws(ws, ws_bytes, kAlign)) return e;
    return launch_topk(logits, rows, V, K, dtype, tok, val, at<int>(ws, 0), as_stream(stream));
}

static ExpandArgs expand_args(const dartree_head* head, const dartree_params* p, const void* hidden,
                              const int32_t* anchor, const int32_t* cand_tok, const float* cand_val,
                              const dartree_supertree* st, void* ws, const Layout& l) {
    ExpandArgs a{};
    a.E = head->E;
    a.Wq = head->Wq;
    a.V = head->V;
    a.H = head->H;
    a.dtype = head->dtype;
    a.C = p->C;
    a.L = p->L;
    a.K = p->K;
    a.W = p->W;
    a.beta = p->beta;
    a.hidden = hidden;
    a.anchor = anchor;
    a.cand_tok = cand_tok;
    a.cand_val = cand_val;
    a.st_tok = st->tok;
    a.st_par = st->par;
    a.st_s = st->score;
    a.st_n = st->n;
    a.hbuf[0] = at<void>(ws, l.h[0]);
    a.hbuf[1] = at<void>(ws, l.h[1]);
    a.sbuf[0] = at<float>(ws, l.s[0]);
    a.sbuf[1] = at<float>(ws, l.s[1]);
    a.U = at<float>(ws, l.U);
    a.z = at<float>(ws, l.z);
    a.uhl = head->dtype == DARTREE_BF16 ? at<uint16_t>(ws, l.uhl) : nullptr;
    a.WqT = head->WqT;
    a.g_rows = l.g_rows;
    a.Eg = l.g_rows ? at<uint16_t>(ws, l.Eg) : nullptr;
    a.Ghi = l.g_rows ? at<uint16_t>(ws, l.Ghi) : nullptr;
    a.Glo = l.g_rows ? at<uint16_t>(ws, l.Glo) : nullptr;
    a.status = at<int>(ws, l.status);
    return a;
}

static int expand_impl(const dartree_head* head, const dartree_params* p, const void* hidden, const int32_t* anchor,
                       const int32_t* cand_tok, const float* cand_val, const dartree_supertree* st, void* ws,
                       const Layout& l, cudaStream_t stream) {
    return launch_expand(expand_args(head, p, hidden, anchor, cand_tok, cand_val, st, ws, l), stream);
}

// S1 of a whole tree build into ct/cv; when the expansion a describes takes the
// candidate-side projection path, the same launch may also copy the candidates'
// rows of E into a.Eg (a.eg_ready says whether it did).
// With rm, the launch may also write the per-position target row maxima
// (*rm_done says whether it did).
static int topk_for_expand(const dartree_head* head, const dartree_params* p, const void* base_logits, int32_t* ct,
                           float* cv, int* status, ExpandArgs& a, cudaStream_t s, const TopkRowmax* rm = nullptr,
                           bool* rm_done = nullptr) {
    // (the candidate-side projection GEMM that follows streams W_q^T: into L2 meanwhile)
    const TopkGather g{static_cast<const uint16_t*>(head->E), head->H, a.Eg, a.WqT,
                       a.WqT && reinterpret_cast<uintptr_t>(a.WqT) % 16 == 0 ? size_t(head->H) * head->H * 2 : 0};
    bool gathered = false;
    const bool want = expand_g_fits(a);
    if (int e = launch_topk(base_logits, p->C * p->L, head->V, p->K, head->dtype, ct, cv, status, s,
                            want ? &g : nullptr, &gathered, rm, rm_done))
        return e;
    a.eg_ready = gathered;
    return DARTREE_OK;
}

static bool st_ok(const dartree_supertree* st) { return st && st->tok && st->par && st->score && st->n; }

int dartree_expand(const dartree_head* head, const dartree_params* p, const void* block_hidden, const int32_t* anchor,
                   const dartree_candidates* cand, dartree_supertree* st, void* ws, size_t ws_bytes, void* stream) {
    if (!head) return DARTREE_EINVAL;
    if (int e = check_params(p, head->V, head->H, head->dtype)) return e;
    if (p->C == 0) return DARTREE_OK;
    if (!head->E || !head->Wq || !block_hidden || !anchor || !cand || !cand->tok || !cand->logit || !st_ok(st))
        return DARTREE_EINVAL;
    const Layout l = layout_of(*p, head->H, head->dtype);
    if (int e = check_ws(ws, ws_bytes, l.total)) return e;
    return expand_impl(head, p, block_hidden, anchor, cand->tok, cand->logit, st, ws, l, as_stream(stream));
}

int dartree_prune(const dartree_params* p, const dartree_supertree* st, const int32_t* anchor, dartree_tree* tree,
                  void* stream) {
    if (!p || p->C < 0 || p->L < 1 || p->W < 1 || p->B < 1 || p->B > p->L * p->W) return DARTREE_EINVAL;
    if (p->L > DARTREE_MAX_L || p->W > DARTREE_MAX_W || p->B + 1 > DARTREE_MAX_SLOTS) return DARTREE_EUNSUPPORTED;
    if (p->C == 0) return DARTREE_OK;
    if (!st_ok(st) || !anchor || !tree || !tree->tok || !tree->par || !tree->depth || !tree->score || !tree->n_nodes)
        return DARTREE_EINVAL;
    return launch_prune(p->C, p->L, p->W, p->B, st->tok, st->par, st->score, st->n, anchor, tree->tok, tree->par,
                        tree->depth, tree->score, tree->n_nodes, nullptr, as_stream(stream));
}

int dartree_tree_mask(const dartree_params* p, dartree_tree* tree, void* stream) {
    if (!p || p->C < 0 || p->L < 1 || p->B < 1) return DARTREE_EINVAL;
    if (p->L > DARTREE_MAX_L || p->B + 1 > DARTREE_MAX_SLOTS) return DARTREE_EUNSUPPORTED;
    if (p->C == 0) return DARTREE_OK;
    if (!tree || !tree->par || !tree->depth || !tree->n_nodes || !tree->mask || !tree->pos) return DARTREE_EINVAL;
    return launch_mask(p->C, p->L, p->B, tree->par, tree->depth, tree->n_nodes, tree->mask, tree->pos,
                       as_stream(stream));
}

int dartree_build_tree(const dartree_head* head, const dartree_params* p, const void* base_logits,
                       const void* block_hidden, const int32_t* anchor, dartree_tree* tree, dartree_supertree* st,
                       dartree_candidates* cand, void* ws, size_t ws_bytes, void* stream) {
    if (!head) return DARTREE_EINVAL;
    if (int e = check_params(p, head->V, head->H, head->dtype)) return e;
    if (p->C == 0) return DARTREE_OK;
    if (!head->E || !head->Wq || !base_logits || !block_hidden || !anchor || !tree || !tree->tok || !tree->par ||
        !tree->depth || !tree->score || !tree->n_nodes)
        return DARTREE_EINVAL;
    if ((tree->mask == nullptr) != (tree->pos == nullptr)) return DARTREE_EINVAL;
    if (st && !st_ok(st)) return DARTREE_EINVAL;
    if (cand && (!cand->tok || !cand->logit)) return DARTREE_EINVAL;
    const Layout l = layout_of(*p, head->H, head->dtype);
    if (int e = check_ws(ws, ws_bytes, l.total)) return e;
    cudaStream_t s = as_stream(stream);
    int32_t* ct = cand ? cand->tok : at<int32_t>(ws, l.cand_tok);
    float* cv = cand ? cand->logit : at<float>(ws, l.cand_val);
    dartree_supertree wst{at<int32_t>(ws, l.st_tok), at<int32_t>(ws, l.st_par), at<float>(ws, l.st_s),
                          at<int32_t>(ws, l.st_n)};
    const dartree_supertree* sp = st ? st : &wst;
    int* status = at<int>(ws, l.status);
    ExpandArgs a = expand_args(head, p, block_hidden, anchor, ct, cv, sp, ws, l);
    if (int e = topk_for_expand(head, p, base_logits, ct, cv, status, a, s)) return e;
    // S8-S9 inside the expansion launch when its path can take them
    const FinishOut fo{tree->tok, tree->par, tree->depth, tree->score, tree->n_nodes, tree->mask, tree->pos,
                       nullptr, nullptr, nullptr, nullptr};
    bool fin_done = false;
    a.B = p->B;
    a.fin = &fo;
    a.fin_done = &fin_done;
    if (int e = launch_expand(a, s)) return e;
    if (fin_done) return DARTREE_OK;
    return finish_tree(p, sp, anchor, tree, status, s);
}

int dartree_round(const dartree_head* head, const dartree_params* p, const void* base_logits,
                  const void* block_hidden, const int32_t* anchor, const void* target, int rows, dartree_tree* tree,
                  int32_t* accepted_len, int32_t* path, int32_t* bonus, void* ws, size_t ws_bytes, void* stream) {
    if (!head) return DARTREE_EINVAL;
    if (int e = check_params(p, head->V, head->H, head->dtype)) return e;
    if (rows != DARTREE_ROWS_PER_POSITION && rows != DARTREE_ROWS_PER_NODE) return DARTREE_EDTYPE;
    if (p->C == 0) return DARTREE_OK;
    if (!head->E || !head->Wq || !base_logits || !block_hidden || !anchor || !target || !tree || !tree->tok ||
        !tree->par || !tree->depth || !tree->score || !tree->n_nodes || !accepted_len || !path || !bonus)
        return DARTREE_EINVAL;
    if ((tree->mask == nullptr) != (tree->pos == nullptr)) return DARTREE_EINVAL;
    const Layout l = layout_of(*p, head->H, head->dtype);
    if (int e = check_ws(ws, ws_bytes, l.total)) return e;
    cudaStream_t s = as_stream(stream);
    int32_t* ct = at<int32_t>(ws, l.cand_tok);
    float* cv = at<float>(ws, l.cand_val);
    const dartree_supertree st{at<int32_t>(ws, l.st_tok), at<int32_t>(ws, l.st_par), at<float>(ws, l.st_s),
                               at<int32_t>(ws, l.st_n)};
    int* status = at<int>(ws, l.status);
    unsigned long long* rowkeys = at<unsigned long long>(ws, l.keys);
    const bool per_pos = rows == DARTREE_ROWS_PER_POSITION;
    // S1 first. The target-row maxima (per-position rows) come from the cluster
    // top-K launch itself when it can; otherwise they run on a side stream forked
    // after S1, overlapping the expansion, which leaves most SMs idle for small
    // batches (forked before S1 they would compete with it for HBM)
    ExpandArgs a = expand_args(head, p, block_hidden, anchor, ct, cv, &st, ws, l);
    // on the candidate-side path the projection GEMM's idle warps take the bf16 row
    // maxima (the top-K launch only clears their keys)
    const bool gemm_rm = per_pos && head->dtype == DARTREE_BF16 && expand_g_fits(a) &&
                         reinterpret_cast<uintptr_t>(target) % 16 == 0 && (size_t(head->V) * 2) % 16 == 0;
    const TopkRowmax rm{target, rowkeys, gemm_rm};
    bool rm_done = false;
    if (int e = topk_for_expand(head, p, base_logits, ct, cv, status, a, s, per_pos ? &rm : nullptr, &rm_done))
        return e;
    if (gemm_rm && rm_done) {
        a.rm_target = target;
        a.rm_keys = rowkeys;
    } else if (gemm_rm) {
        rm_done = false;  // keys not cleared: the maxima are taken below instead
    }
    std::unique_lock<std::recursive_mutex> lock(side_mutex(), std::defer_lock);
    SideStreams* side = nullptr;
    if (per_pos && !rm_done) {
        lock.lock();
        side = side_streams(s);
        if (side) {
            if (cudaEventRecord(side->fork[0], s) != cudaSuccess ||
                cudaStreamWaitEvent(side->s[0], side->fork[0], 0) != cudaSuccess)
                return DARTREE_ECUDA;
            if (int e = launch_rowmax_position(p->C, p->L, head->V, head->dtype, target, rowkeys, side->s[0])) return e;
            if (cudaEventRecord(side->join[0], side->s[0]) != cudaSuccess) return DARTREE_ECUDA;
        } else {
            lock.unlock();
            if (int e = launch_rowmax_position(p->C, p->L, head->V, head->dtype, target, rowkeys, s)) return e;
        }
    }
    // S8-S10 inside the expansion launch when its path can take them and the row
    // maxima are complete before it starts (not on a side stream)
    const FinishOut fo{tree->tok, tree->par, tree->depth, tree->score, tree->n_nodes, tree->mask, tree->pos,
                       per_pos ? rowkeys : nullptr, accepted_len, path, bonus};
    bool fin_done = false;
    if (!side) {
        a.B = p->B;
        a.fin = &fo;
        a.fin_done = &fin_done;
    }
    if (int e = launch_expand(a, s)) return e;
    if (side && cudaStreamWaitEvent(s, side->join[0], 0) != cudaSuccess) return DARTREE_ECUDA;
    if (fin_done)
        return per_pos ? DARTREE_OK
                       : launch_verify(p->C, p->L, p->B, tree->tok, tree->par, tree->depth, tree->n_nodes, target,
                                       rows, head->V, head->dtype, rowkeys, accepted_len, path, bonus, status, s);
    if (per_pos && finish_supported(p->L, p->W))  // (set-up overlapping the expansion's tail)
        return launch_finish(p->C, p->L, p->W, p->B, st.tok, st.par, st.score, st.n, anchor, tree->tok, tree->par,
                             tree->depth, tree->score, tree->n_nodes, tree->mask, tree->pos, rowkeys, accepted_len,
                             path, bonus, status, s, true);
    if (int e = finish_tree(p, &st, anchor, tree, status, s)) return e;
    if (per_pos)
        return launch_walk_position(p->C, p->L, p->B, tree->tok, tree->par, tree->depth, tree->n_nodes, rowkeys,
                                    accepted_len, path, bonus, status, s);
    return launch_verify(p->C, p->L, p->B, tree->tok, tree->par, tree->depth, tree->n_nodes, target, rows, head->V,
                         head->dtype, rowkeys, accepted_len, path, bonus, status, s);
}

int dartree_verify(const dartree_params* p, const dartree_tree* tree, const void* target, int rows, int V, int dtype,
                   int32_t* accepted_len, int32_t* path, int32_t* bonus, void* ws, size_t ws_bytes, void* stream) {
    if (!p || p->C < 0 || p->L < 1 || p->B < 1 || V < 1) return DARTREE_EINVAL;
    if (!dtype_ok(dtype) || (rows != DARTREE_ROWS_PER_POSITION && rows != DARTREE_ROWS_PER_NODE))
        return DARTREE_EDTYPE;
    if (p->L > DARTREE_MAX_L || p->B + 1 > DARTREE_MAX_SLOTS) return DARTREE_EUNSUPPORTED;
    if (p->C == 0) return DARTREE_OK;
    if (!tree || !tree->tok || !tree->par || !tree->depth || !tree->n_nodes || !target || !accepted_len || !path ||
        !bonus)
        return DARTREE_EINVAL;
    const size_t keys_bytes = size_t(p->C) * (p->L > p->B + 1 ? p->L : p->B + 1) * 8;
    if (int e = check_ws(ws, ws_bytes, kAlign + keys_bytes)) return e;
    // row keys sit right after the status word (scratch of the build is dead by then)
    const size_t keys_off = kAlign;
    return launch_verify(p->C, p->L, p->B, tree->tok, tree->par, tree->depth, tree->n_nodes, target, rows, V, dtype,
                         at<unsigned long long>(ws, keys_off), accepted_len, path, bonus, at<int>(ws, 0),
                         as_stream(stream));
}

int dartree_verify_sample(const dartree_params* p, const dartree_tree* tree, const void* target, int rows, int V,
                          int dtype, float temperature, uint64_t seed, int32_t* accepted_len, int32_t* path,
                          int32_t* bonus, void* ws, size_t ws_bytes, void* stream) {
    if (!p || p->C < 0 || p->L < 1 || p->B < 1 || V < 1) return DARTREE_EINVAL;
    if (!(temperature > 0.0f) || !isfinite(temperature)) return DARTREE_EINVAL;
    if (!dtype_ok(dtype) || (rows != DARTREE_ROWS_PER_POSITION && rows != DARTREE_ROWS_PER_NODE))
        return DARTREE_EDTYPE;
    if (p->L > DARTREE_MAX_L || p->B + 1 > DARTREE_MAX_SLOTS) return DARTREE_EUNSUPPORTED;
    if (p->C == 0) return DARTREE_OK;
    if (!tree || !tree->tok || !tree->par || !tree->depth || !tree->n_nodes || !target || !accepted_len || !path ||
        !bonus)
        return DARTREE_EINVAL;
    const size_t keys_bytes = size_t(p->C) * (p->L > p->B + 1 ? p->L : p->B + 1) * 8;
    if (int e = check_ws(ws, ws_bytes, kAlign + keys_bytes)) return e;
    return launch_verify_sample(p->C, p->L, p->B, tree->tok, tree->par, tree->depth, tree->n_nodes, target, rows, V,
                                dtype, temperature, seed, at<unsigned long long>(ws, kAlign), accepted_len, path,
                                bonus, at<int>(ws, 0), as_stream(stream));
}

size_t dartree_lm_head_workspace_bytes(int R, int V, int H, int K) {
    if (!lmhead_supported(R, V, H, K)) return 0;
    return kAlign + up(lmhead_part_bytes(R < 64 ? R : 64, V, K));
}

int dartree_lm_head_topk(const void* hidden, const void* W_lm, int R, int V, int H, int K, int dtype, int32_t* tok,
                         float* val, void* ws, size_t ws_bytes, void* stream) {
    if (R < 0 || V < 1 || H < 1 || K < 1 || K > V) return DARTREE_EINVAL;
    if (!dtype_ok(dtype)) return DARTREE_EDTYPE;
    if (dtype != DARTREE_BF16) return DARTREE_EUNSUPPORTED;  // bf16 tensor-core operands
    if (R == 0) return DARTREE_OK;
    if (!lmhead_supported(R, V, H, K)) return DARTREE_EUNSUPPORTED;
    if (!hidden || !W_lm || !tok || !val || reinterpret_cast<uintptr_t>(hidden) % 16 != 0 ||
        reinterpret_cast<uintptr_t>(W_lm) % 16 != 0)
        return DARTREE_EINVAL;
    if (int e = check_ws(ws, ws_bytes, dartree_lm_head_workspace_bytes(R, V, H, K))) return e;
    return launch_lmhead_topk(hidden, W_lm, R, V, H, K, tok, val, at<unsigned long long>(ws, kAlign),
                              at<int>(ws, 0), as_stream(stream));
}

static bool attn_params_ok(const dartree_attn_params* p) {
    return p && attn_supported(p->C, p->S, p->Hq, p->Hkv, p->D, p->N) && p->theta > 0.f && isfinite(p->theta);
}

size_t dartree_tree_attention_workspace_bytes(const dartree_attn_params* p) {
    if (!attn_params_ok(p)) return 0;
    return attn_plan(p->C, p->S, p->Hq, p->Hkv, p->N).total;
}

int dartree_tree_attention(const dartree_attn_params* p, const void* q, const void* k_tree, const void* v_tree,
                           const void* k_cache, const void* vt_cache, const int32_t* n_ctx, const dartree_tree* tree,
                           void* out, void* ws, size_t ws_bytes, void* stream) {
    if (!p || p->C < 0) return DARTREE_EINVAL;
    if (!attn_params_ok(p)) return DARTREE_EUNSUPPORTED;
    if (p->C == 0) return DARTREE_OK;
    auto al16 = [](const void* x) { return x && reinterpret_cast<uintptr_t>(x) % 16 == 0; };
    if (!al16(q) || !al16(k_tree) || !al16(v_tree) || !al16(out) || !n_ctx || !tree || !tree->mask || !tree->pos ||
        !tree->n_nodes || (p->N > 0 && (!al16(k_cache) || !al16(vt_cache))))
        return DARTREE_EINVAL;
    const AttnPlan pl = attn_plan(p->C, p->S, p->Hq, p->Hkv, p->N);
    if (int e = check_ws(ws, ws_bytes, pl.total)) return e;
    return launch_tree_attention(p->C, p->S, p->Hq, p->Hkv, p->N, double(p->theta), q, k_tree, v_tree, k_cache,
                                 vt_cache, n_ctx, tree->mask, tree->pos, tree->n_nodes, out, ws, pl,
                                 as_stream(stream));
}

int dartree_adaptive_budget(int C, int* B, int* W) {
    if (C < 1 || !B || !W) return DARTREE_EINVAL;
    const bool reduced = C >= DARTREE_REDUCED_BUDGET_FROM_C;
    *B = reduced ? 32 : 64;
    *W = reduced ? 3 : 12;
    return DARTREE_OK;
}

}  // extern "C"
