// Per-kernel launch timing: while enabled, every library kernel launch is
// bracketed by two CUDA events recorded on its own stream; reading the totals
// synchronises those events. Used to measure the dominant kernel of a round.
// Off by default; not meant for launches captured into a CUDA graph.
#include <mutex>
#include <vector>

#include "dartree.h"
#include "kernels.h"

namespace dartree {

namespace {
struct Pair {
    cudaEvent_t a, b;
};
std::mutex g_mu;
bool g_on = false;
std::vector<Pair> g_pairs[KID_COUNT];
std::vector<cudaEvent_t> g_free;

cudaEvent_t take_event() {
    if (!g_free.empty()) {
        cudaEvent_t e = g_free.back();
        g_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return e;
}
void release_all() {
    for (auto& v : g_pairs) {
        for (auto& p : v) {
            g_free.push_back(p.a);
            g_free.push_back(p.b);
        }
        v.clear();
    }
}
const char* const kNames[KID_COUNT] = {
    "topk_rows_kernel",  "topk_stream_kernel", "gemm_bf16_tc_kernel", "contract_tc_kernel",
    "expand_g_kernel",   "gather_rows_kernel", "select_kernel",       "state_kernel",
    "heap_search_kernel",  "finish_kernel",    "prune_kernel",        "mask_kernel",
    "rowmax_kernel",     "walk_kernel",        "rowsample_kernel",    "lmhead_topk_kernel",
    "lmhead_merge_kernel", "attn_prep_kernel", "attn_kernel", "attn_combine_kernel", "other"};
}  // namespace

KTimer::KTimer(int id, cudaStream_t s) : id_(id), s_(s), b_(nullptr) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_on || id < 0 || id >= KID_COUNT) return;
    cudaEvent_t a = take_event(), b = take_event();
    if (!a || !b) return;
    if (cudaEventRecord(a, s) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    g_pairs[id].push_back(Pair{a, b});
    b_ = b;
}

KTimer::~KTimer() {
    if (b_ && cudaEventRecord(static_cast<cudaEvent_t>(b_), s_) != cudaSuccess) cudaGetLastError();
}

}  // namespace dartree

using namespace dartree;

extern "C" {

int dartree_timing(int enable) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (enable) {
        if (cudaDeviceSynchronize() != cudaSuccess) return DARTREE_ECUDA;
        release_all();
    }
    g_on = enable != 0;
    return DARTREE_OK;
}

int dartree_timing_read(int kernel_id, int* launches, double* total_ms) {
    if (kernel_id < 0 || kernel_id >= KID_COUNT || !launches || !total_ms) return DARTREE_EINVAL;
    std::lock_guard<std::mutex> lk(g_mu);
    double ms = 0.0;
    for (auto& p : g_pairs[kernel_id]) {
        if (cudaEventSynchronize(p.b) != cudaSuccess) return DARTREE_ECUDA;
        float x = 0.f;
        if (cudaEventElapsedTime(&x, p.a, p.b) != cudaSuccess) return DARTREE_ECUDA;
        ms += x;
    }
    *launches = int(g_pairs[kernel_id].size());
    *total_ms = ms;
    return DARTREE_OK;
}

const char* dartree_kernel_name(int kernel_id) {
    if (kernel_id < 0 || kernel_id >= KID_COUNT) return "unknown";
    return kNames[kernel_id];
}

}  // extern "C"
