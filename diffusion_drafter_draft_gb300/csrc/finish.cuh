// S8-S10 of one request by one CTA of FN_NT threads (DARTree blog post, 3.1
// "Basic flow", deferred pruning and Lemma 1: one global top-B over the
// supertree, prefix-closed for beta <= 0; 3.2: tree-attention mask, position ids
// and the greedy longest accepted prefix), for supertrees of at most FN_NT
// nodes. Used by the finish kernel (supertree read from global memory) and by
// the candidate-side cluster expansion, which runs it in one CTA of the cluster
// right after its last depth, from the supertree it holds in shared memory.
//
// Every supertree node's global rank under (score desc, depth asc, rank asc) is
// counted against all keys in shared memory (broadcast reads); the nodes of rank
// below B are chosen and take slots in (depth, rank) order by a block scan. Tree
// arrays, ancestor table and mask are built in shared memory, and the walk
// follows the per-position target row maxima computed beforehand.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace dartree {

constexpr int FN_NT = 256;  // one supertree node per thread

struct FnSmem {
    size_t keys, slot, ttok, tpar, tdep, anc, rowk, next, wtot, misc, bytes;
};
__host__ __device__ inline FnSmem fn_smem(int L, int B) {
    const size_t S = size_t(B) + 1;
    FnSmem f{};
    size_t o = 0;
    auto take = [&](size_t b) { size_t at = o; o = (o + b + 15) / 16 * 16; return at; };
    f.keys = take(FN_NT * 8);
    f.slot = take(FN_NT * 4);
    f.ttok = take(S * 4);
    f.tpar = take(S * 4);
    f.tdep = take(S * 4);
    f.anc = take(S * (size_t(L) + 1) * 2);
    f.rowk = take(size_t(L) * 8);
    f.next = take(S * 4);
    f.wtot = take(32 * 4);
    f.misc = take(16);
    f.bytes = o;
    return f;
}

// Key of supertree node (depth dm1 + 1, rank k) with score word ord_f32(score):
// larger keys come first in the global order.
__device__ __forceinline__ uint64_t finish_key(uint32_t score_ord, int dm1, int k) {
    return (uint64_t(score_ord) << 32) | (uint64_t(0xffffu - uint32_t(dm1 + 1)) << 16) | (0xffffu - uint32_t(k));
}

// Called by all FN_NT threads of the CTA for request r. Thread q < L*W holds
// supertree node q = (depth - 1) * W + rank: key (0 = no node), token, parent
// rank, score. smem: fn_smem(L, B).bytes, 16-byte aligned. WALK: o.rowkeys is set.
template <bool WALK>
__device__ void finish_request(int r, int L, int W, int B, uint8_t* smem, uint64_t key, int s_tok, int s_par,
                               float s_sc, int dm1, int anchor_tok, const FinishOut& o, int* status) {
    const FnSmem fl = fn_smem(L, B);
    uint64_t* keys = reinterpret_cast<uint64_t*>(smem + fl.keys);
    int* slot = reinterpret_cast<int*>(smem + fl.slot);
    int* ttok = reinterpret_cast<int*>(smem + fl.ttok);
    int* tpar = reinterpret_cast<int*>(smem + fl.tpar);
    int* tdep = reinterpret_cast<int*>(smem + fl.tdep);
    int16_t* anc = reinterpret_cast<int16_t*>(smem + fl.anc);
    int* wtot = reinterpret_cast<int*>(smem + fl.wtot);
    int* misc = reinterpret_cast<int*>(smem + fl.misc);  // [0] scan total
    uint64_t* rowk = reinterpret_cast<uint64_t*>(smem + fl.rowk);
    int* next = reinterpret_cast<int*>(smem + fl.next);  // accepted child of every slot, or INT_MAX
    const int n = L * W, S = B + 1, q = threadIdx.x;
    int32_t* tok = o.tok;
    int32_t* par = o.par;
    int32_t* depth = o.depth;
    float* score = o.score;
    int32_t* n_nodes = o.n_nodes;
    uint8_t* mask = o.mask;
    int32_t* pos = o.pos;
    int32_t* accepted = o.accepted;
    int32_t* path = o.path;
    int32_t* bonus = o.bonus;
    keys[q] = key;
    if (WALK)
        for (int d = q; d < L; d += FN_NT) rowk[d] = o.rowkeys[size_t(r) * L + d];
    const int nv = __syncthreads_count(key != 0);
    const int N = min(B, nv);
    // ---- global rank: keys above this one (all threads read the same pair at once)
    int above = 0;
    {
        const ulonglong2* k2 = reinterpret_cast<const ulonglong2*>(keys);
        const int n2 = (n + 1) / 2;
#pragma unroll 4
        for (int i = 0; i < n2; ++i) {
            const ulonglong2 v = k2[i];
            above += (v.x > key) + (v.y > key);
        }
    }
    const bool ch = key != 0 && above < N;
    // ---- slots in (depth, rank) order
    const int ex = block_exclusive_scan<FN_NT>(ch ? 1 : 0, wtot, misc);
    const int chosen = misc[0];
    slot[q] = ch ? 1 + ex : -1;
    for (int j = q; j < S; j += FN_NT) {
        if (j == 0) { ttok[0] = anchor_tok; tpar[0] = -1; tdep[0] = 0; }
        else if (j > chosen) { ttok[j] = -1; tpar[j] = -1; tdep[j] = -1; }
    }
    __syncthreads();
    int32_t* t_tok = tok + size_t(r) * S;
    int32_t* t_par = par + size_t(r) * S;
    int32_t* t_dep = depth + size_t(r) * S;
    float* t_sc = score + size_t(r) * S;
    if (ch) {
        const int j = 1 + ex;
        int ps = 0;
        if (dm1 > 0) {
            ps = (s_par >= 0 && s_par < W) ? slot[(dm1 - 1) * W + s_par] : -1;
            if (ps < 0) set_status(status, DARTREE_EINTERNAL);  // the chosen set is not prefix-closed
        }
        if (j < S) {
            ttok[j] = s_tok;
            tpar[j] = ps;
            tdep[j] = dm1 + 1;
        }
    }
    __syncthreads();
    for (int j = q; j < S; j += FN_NT) {
        t_tok[j] = ttok[j];
        t_par[j] = tpar[j];
        t_dep[j] = tdep[j];
    }
    if (ch && 1 + ex < S) t_sc[1 + ex] = s_sc;
    for (int j = q; j < S; j += FN_NT)
        if (j == 0 || j > chosen) t_sc[j] = 0.f;
    if (q == 0) {
        n_nodes[r] = 1 + chosen;
        if (chosen != N) set_status(status, DARTREE_EINTERNAL);
    }
    const int nn = min(S, 1 + chosen);
    // ---- mask and position ids: anc[i][delta] = ancestor of slot i at depth delta
    if (mask) {
        for (int i = q; i < S; i += FN_NT) {
            const int di = i < nn ? min(max(tdep[i], 0), L) : -1;
            if (di >= 0) {
                int b = i;
                for (int dd = di; dd >= 0; --dd) {
                    anc[size_t(i) * (L + 1) + dd] = int16_t(b);
                    b = (b >= 0 && b < S) ? tpar[b] : -1;
                }
            }
            pos[size_t(r) * S + i] = di;
        }
        __syncthreads();
        uint8_t* m = mask + size_t(r) * S * S;
        const int total = S * S;
        for (int e = q * 4; e < total; e += FN_NT * 4) {
            uint32_t word = 0;
            const int i0 = e / S;
            int i = i0, j = e - i0 * S;  // (row, column) of byte e, then stepped
            const int di = i < nn ? tdep[i] : -1;
            const int di2 = i + 1 < nn ? tdep[i + 1] : -1;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (e + u >= total) break;
                const int dii = i == i0 ? di : di2;
                const int dj = j < nn ? tdep[j] : -1;
                const bool on = dii >= 0 && dj >= 0 && dj <= dii && anc[size_t(i) * (L + 1) + dj] == j;
                word |= uint32_t(on) << (8 * u);
                if (++j == S) { j = 0; ++i; }
            }
            if (e + 4 <= total && (reinterpret_cast<uintptr_t>(m + e) & 3) == 0) {
                *reinterpret_cast<uint32_t*>(m + e) = word;
            } else {
                for (int u = 0; u < 4 && e + u < total; ++u) m[e + u] = uint8_t(word >> (8 * u));
            }
        }
    }
    // ---- greedy walk with per-position row maxima: every slot's accepted child
    //      (the lowest slot whose parent it is and whose token is the argmax of
    //      the parent's row) in parallel, then one thread follows the chain
    if (WALK) {
        for (int j = q; j < S; j += FN_NT) next[j] = 0x7fffffff;
        __syncthreads();
        for (int j = 1 + q; j < nn; j += FN_NT) {
            const int p = tpar[j];
            const int dp = (p >= 0 && p < nn) ? tdep[p] : -1;
            if (dp >= 0 && dp < L && ttok[j] == int(0xffffffffu - uint32_t(rowk[dp]))) atomicMin(&next[p], j);
        }
        __syncthreads();
        if (q == 0) {
            int cur = 0, acc = 0, bon = -1;
            for (int step = 0; step <= L; ++step) {
                const int d = tdep[cur];
                if (d < 0 || d >= L) break;
                const int f = next[cur];
                if (f == 0x7fffffff) { bon = int(0xffffffffu - uint32_t(rowk[d])); break; }
                if (acc < L) path[size_t(r) * L + acc] = f;
                ++acc;
                cur = f;
            }
            accepted[r] = acc;
            bonus[r] = bon;
            misc[1] = acc;
        }
        __syncthreads();
        for (int u = misc[1] + q; u < L; u += FN_NT) path[size_t(r) * L + u] = -1;
    }
}

}  // namespace dartree
