// Library-owned side streams (one set per device, created on first use) for the
// forks inside a call: the target-row maxima of dartree_round, and the second
// half of a large batch's expansion. Forks and joins go through events, so they
// are captured with the caller's stream into a CUDA graph.
#include "kernels.h"

namespace dartree {

namespace {
SideStreams g_side[64];
std::recursive_mutex g_side_mu;
}  // namespace

std::recursive_mutex& side_mutex() { return g_side_mu; }

SideStreams* side_streams() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    SideStreams& ss = g_side[dev];
    if (!ss.ok) {
        for (int i = 0; i < 2; ++i) {
            if (cudaStreamCreateWithFlags(&ss.s[i], cudaStreamNonBlocking) != cudaSuccess ||
                cudaEventCreateWithFlags(&ss.fork[i], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&ss.join[i], cudaEventDisableTiming) != cudaSuccess) {
                cudaGetLastError();
                return nullptr;
            }
        }
        ss.ok = true;
    }
    return &ss;
}

}  // namespace dartree
