// Library-owned side streams for the forks inside a call: the target-row maxima
// of dartree_round, and the second half of a large batch's expansion. One set
// per (device, caller stream), created on its first use, so that two callers
// on two streams fork onto different side streams and never wait for each
// other. Forks and joins go through events, so they are captured with the
// caller's stream into a CUDA graph (the set must exist before the capture
// starts: make one call on that stream first).
#include "kernels.h"

namespace dartree {

namespace {
constexpr int kMaxSets = 256;
SideStreams g_side[kMaxSets];
int g_nside = 0;
std::recursive_mutex g_side_mu;
}  // namespace

std::recursive_mutex& side_mutex() { return g_side_mu; }

SideStreams* side_streams(cudaStream_t caller) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::recursive_mutex> lock(g_side_mu);
    for (int i = 0; i < g_nside; ++i)
        if (g_side[i].dev == dev && g_side[i].caller == caller) return g_side[i].ok ? &g_side[i] : nullptr;
    if (g_nside == kMaxSets) return nullptr;
    SideStreams& ss = g_side[g_nside++];
    ss.dev = dev;
    ss.caller = caller;
    for (int i = 0; i < 2; ++i) {
        if (cudaStreamCreateWithFlags(&ss.s[i], cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&ss.fork[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&ss.join[i], cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;  // stays in the table as not usable
        }
    }
    ss.ok = true;
    return &ss;
}

}  // namespace dartree
