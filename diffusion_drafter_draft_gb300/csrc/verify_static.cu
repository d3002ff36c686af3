// dartree_verify_static: the S10 verification with its scratch in a fixed
// device array instead of a caller workspace.
//
// Some callers cannot allocate device memory where they verify: a serving loop
// that hands all free HBM to its own caching allocator at start-up, or a plugin
// reached through a plain C interface that has no allocator handle. For them
// this entry point takes only inputs and outputs. Its scratch (one 64-bit row
// key per target row, after a 256-byte header that is not used) lives in
// g_verify_scratch below, a file-scope device array of kStaticVerifyBytes that
// every GPU which loads the library keeps until the process exits. With no
// status word the caller could read, a malformed tree (which dartree_verify
// reports as DARTREE_EINTERNAL in its workspace) goes unreported here.
#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>

#include "dartree.h"
#include "kernels.h"

namespace {

constexpr size_t kStaticVerifyBytes = DARTREE_STATIC_VERIFY_BYTES;
constexpr size_t kKeysOffset = 256;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_verify_scratch[kStaticVerifyBytes];

std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_verify_scratch on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
int scratch_on_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DARTREE_ECUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || !p) return DARTREE_ECUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return DARTREE_OK;
}

}  // namespace

extern "C" int dartree_verify_static(const dartree_params* p, const dartree_tree* tree, const void* target, int rows,
                                     int V, int dtype, int32_t* accepted_len, int32_t* path, int32_t* bonus,
                                     void* stream) {
    if (!p || p->C < 0 || p->L < 1 || p->B < 1 || V < 1) return DARTREE_EINVAL;
    if ((dtype != DARTREE_F32 && dtype != DARTREE_BF16) ||
        (rows != DARTREE_ROWS_PER_POSITION && rows != DARTREE_ROWS_PER_NODE))
        return DARTREE_EDTYPE;
    if (p->L > DARTREE_MAX_L || p->B + 1 > DARTREE_MAX_SLOTS) return DARTREE_EUNSUPPORTED;
    const size_t keys = size_t(p->C) * size_t(p->L > p->B + 1 ? p->L : p->B + 1) * sizeof(unsigned long long);
    if (kKeysOffset + keys > kStaticVerifyBytes) return DARTREE_EUNSUPPORTED;
    if (p->C == 0) return DARTREE_OK;
    if (!tree || !tree->tok || !tree->par || !tree->depth || !tree->n_nodes || !target || !accepted_len || !path ||
        !bonus)
        return DARTREE_EINVAL;
    void* base = nullptr;
    if (int e = scratch_on_current_device(&base)) return e;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* b = static_cast<uint8_t*>(base);
    // the previous call's row keys stay in the array; launch_verify clears the ones
    // it uses before the row maxima are taken
    return dartree::launch_verify(p->C, p->L, p->B, tree->tok, tree->par, tree->depth, tree->n_nodes, target, rows,
                                  V, dtype, reinterpret_cast<unsigned long long*>(b + kKeysOffset), accepted_len,
                                  path, bonus, nullptr, s);
}
