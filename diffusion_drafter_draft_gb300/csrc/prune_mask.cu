// S8: deferred pruning (DARTree blog post, 3.1 "Basic flow": one global top-B
// over the supertree; Lemma 1: for beta <= 0 the set is prefix-closed and equals
// best-first heap popping on the materialised supertree).
// S9: tree-attention mask and position ids (blog post, 3.2).
#include "common.cuh"
#include "kernels.h"

namespace dartree {

constexpr int PR_NT = 256;

// Global order: s desc, depth asc, rank asc. Output depth-major, rank within
// a depth; parents remapped from rank to slot id.
__global__ void __launch_bounds__(PR_NT) prune_kernel(int L, int W, int B, const int32_t* __restrict__ st_tok,
                                                      const int32_t* __restrict__ st_par, const float* __restrict__ st_s,
                                                      const int32_t* __restrict__ st_n, const int32_t* __restrict__ anchor,
                                                      int32_t* __restrict__ tok, int32_t* __restrict__ par,
                                                      int32_t* __restrict__ depth, float* __restrict__ score,
                                                      int32_t* __restrict__ n_nodes, int* status) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int r = blockIdx.x;
    const int n = L * W;
    uint64_t* keys = reinterpret_cast<uint64_t*>(smem);        // n
    int* slot = reinterpret_cast<int*>(keys + n);              // n
    uint32_t* hist = reinterpret_cast<uint32_t*>(slot + n);    // 256
    uint32_t* bcast = hist + 256;                              // 8
    int* wtot = reinterpret_cast<int*>(bcast + 8);             // 32
    int* total = wtot + 32;                                    // 8
    const int32_t* sn = st_n + size_t(r) * L;
    const size_t base = size_t(r) * L * W;

    int valid = 0;
    for (int q = threadIdx.x; q < n; q += PR_NT) {
        const int dm1 = q / W, k = q % W;
        uint64_t key = 0;
        if (k < sn[dm1]) {
            const float s = st_s[base + q] + 0.f;
            key = (uint64_t(ord_f32(s)) << 32) | (uint64_t(0xffffu - uint32_t(dm1 + 1)) << 16) | (0xffffu - uint32_t(k));
            ++valid;
        }
        keys[q] = key;
    }
    // count valid nodes
    int nv = 0;
    {
        int tot;
        block_exclusive_scan<PR_NT>(valid, wtot, total);
        tot = *total;
        __syncthreads();
        nv = tot;
    }
    const int N = min(B, nv);
    uint64_t prefix = ~0ull, mask = ~0ull;
    bool ok = true;
    if (N > 0) ok = block_select_top<PR_NT>(keys, n, N, hist, bcast, prefix, mask);
    if (!ok && threadIdx.x == 0) set_status(status, DARTREE_EINTERNAL);

    // slots: exclusive scan of chosen flags in (depth, rank) order, by contiguous runs
    const int per = (n + PR_NT - 1) / PR_NT;
    const int lo = min(n, int(threadIdx.x) * per), hi = min(n, lo + per);
    int cnt = 0;
    for (int q = lo; q < hi; ++q) cnt += (ok && N > 0 && keys[q] != 0 && selected(keys[q], prefix, mask));
    int run = block_exclusive_scan<PR_NT>(cnt, wtot, total);
    for (int q = lo; q < hi; ++q) {
        const bool ch = ok && N > 0 && keys[q] != 0 && selected(keys[q], prefix, mask);
        slot[q] = ch ? 1 + run : -1;
        run += ch;
    }
    __syncthreads();
    const int chosen = *total;
    const int S = B + 1;
    int32_t* t_tok = tok + size_t(r) * S;
    int32_t* t_par = par + size_t(r) * S;
    int32_t* t_dep = depth + size_t(r) * S;
    float* t_sc = score + size_t(r) * S;
    for (int j = threadIdx.x; j < S; j += PR_NT) {
        if (j == 0) { t_tok[0] = anchor[r]; t_par[0] = -1; t_dep[0] = 0; t_sc[0] = 0.f; }
        else if (j > chosen) { t_tok[j] = -1; t_par[j] = -1; t_dep[j] = -1; t_sc[j] = 0.f; }
    }
    for (int q = threadIdx.x; q < n; q += PR_NT) {
        const int j = slot[q];
        if (j < 0 || j > B) continue;
        const int dm1 = q / W;
        int ps = 0;
        if (dm1 > 0) {
            const int pr = st_par[base + q];
            ps = (pr >= 0 && pr < W) ? slot[(dm1 - 1) * W + pr] : -1;
            if (ps < 0) set_status(status, DARTREE_EINTERNAL);  // the chosen set is not prefix-closed
        }
        t_tok[j] = st_tok[base + q];
        t_par[j] = ps;
        t_dep[j] = dm1 + 1;
        t_sc[j] = st_s[base + q];
    }
    if (threadIdx.x == 0) {
        n_nodes[r] = 1 + chosen;
        if (chosen != N) set_status(status, DARTREE_EINTERNAL);
    }
}

int launch_prune(int C, int L, int W, int B, const int32_t* st_tok, const int32_t* st_par, const float* st_s,
                 const int32_t* st_n, const int32_t* anchor, int32_t* tok, int32_t* par, int32_t* depth,
                 float* score, int32_t* n_nodes, int* status, cudaStream_t stream) {
    if (C == 0) return DARTREE_OK;
    const size_t n = size_t(L) * W;
    const size_t smem = n * 8 + n * 4 + 256 * 4 + 8 * 4 + 32 * 4 + 8 * 4 + 16;
    if (cudaFuncSetAttribute(prune_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
        return DARTREE_ECUDA;
    {
        KTimer kt_(KID_PRUNE, stream);
        prune_kernel<<<C, PR_NT, smem, stream>>>(L, W, B, st_tok, st_par, st_s, st_n, anchor, tok, par, depth, score,
                                                n_nodes, status);
    }
    return cudaGetLastError() == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

// --------------------------------------------------------------------------- mask + position ids

constexpr int MK_NT = 256;

// mask[i][j] = 1 iff j < n, i < n, depth[j] <= depth[i] and the ancestor of i at
// depth depth[j] is j. anc[i][delta] is filled by walking up from every slot.
__global__ void __launch_bounds__(MK_NT) mask_kernel(int L, int B, const int32_t* __restrict__ par,
                                                     const int32_t* __restrict__ depth,
                                                     const int32_t* __restrict__ n_nodes, uint8_t* __restrict__ mask,
                                                     int32_t* __restrict__ pos) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int r = blockIdx.x;
    const int S = B + 1;
    int16_t* anc = reinterpret_cast<int16_t*>(smem);     // S x (L+1)
    int16_t* dep = anc + size_t(S) * (L + 1);            // S
    const int n = min(S, max(0, n_nodes[r]));
    const int32_t* pr = par + size_t(r) * S;
    const int32_t* dp = depth + size_t(r) * S;
    for (int i = threadIdx.x; i < S; i += MK_NT) {
        const int di = i < n ? min(max(dp[i], 0), L) : -1;
        dep[i] = int16_t(di);
        if (di >= 0) {
            int b = i;
            for (int dd = di; dd >= 0; --dd) {
                anc[size_t(i) * (L + 1) + dd] = int16_t(b);
                b = (b >= 0 && b < S) ? pr[b] : -1;
            }
        }
        pos[size_t(r) * S + i] = di;
    }
    __syncthreads();
    uint8_t* m = mask + size_t(r) * S * S;
    const int total = S * S;
    for (int e = threadIdx.x * 4; e < total; e += MK_NT * 4) {
        uint32_t word = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int x = e + q;
            if (x >= total) break;
            const int i = x / S, j = x % S;
            const int di = dep[i], dj = dep[j];
            const bool on = di >= 0 && dj >= 0 && dj <= di && anc[size_t(i) * (L + 1) + dj] == j;
            word |= uint32_t(on) << (8 * q);
        }
        if (e + 4 <= total && (reinterpret_cast<uintptr_t>(m + e) & 3) == 0) {
            *reinterpret_cast<uint32_t*>(m + e) = word;
        } else {
            for (int q = 0; q < 4 && e + q < total; ++q) m[e + q] = uint8_t(word >> (8 * q));
        }
    }
}

int launch_mask(int C, int L, int B, const int32_t* par, const int32_t* depth, const int32_t* n_nodes,
                uint8_t* mask, int32_t* pos, cudaStream_t stream) {
    if (C == 0) return DARTREE_OK;
    const int S = B + 1;
    const size_t smem = size_t(S) * (L + 1) * 2 + size_t(S) * 2 + 16;
    if (cudaFuncSetAttribute(mask_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
        return DARTREE_ECUDA;
    {
        KTimer kt_(KID_MASK, stream);
        mask_kernel<<<C, MK_NT, smem, stream>>>(L, B, par, depth, n_nodes, mask, pos);
    }
    return cudaGetLastError() == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

}  // namespace dartree
