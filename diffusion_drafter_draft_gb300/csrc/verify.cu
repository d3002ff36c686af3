// S10: greedy longest accepted prefix (DARTree blog post, 3.2: all draft tokens
// are verified in one target pass with the tree-attention mask and the longest
// valid prefix is kept).
//
// Walk: from the root, t = argmax of the current slot's target row (lowest token
// id among equal maxima, i.e. the largest key (value, ~token)); move to the child
// carrying t while one exists.
//  - per-position rows [C, L, V]: the row of a slot depends only on its depth,
//    so all C*L row maxima are computed in parallel first, then one warp per
//    request walks the tree;
//  - per-node rows [C, B+1, V]: only the rows on the accepted path are read; one
//    thread-block cluster per request computes each row's maximum (partials
//    exchanged through distributed shared memory) and takes the next step.
// A walk that would take more than L steps can only come from a malformed tree
// (a parent that is not one depth above its child); it stops there and records
// DARTREE_EINTERNAL in the status word (when one is given).
//
// At a temperature T > 0 the same walks run on a drawn token instead of the row's
// maximum: t = argmax_v (x_v / T + G_v), G_v = -log(-log U_v) (a Gumbel-max draw from
// softmax(row / T)), lowest token id among equal values. U_v comes from
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
// 1, 2, 3", SC 2011) with key (seed low word, seed high word), counter
// (v / 4, row, request, 0), output word v % 4, U = (2 (word >> 9) + 1) 2^-24; row is
// the slot's depth for per-position rows and the slot index for per-node rows. Every
// emitted token is then a draw of the target at temperature T, so the output
// distribution is the target's own (the lossless claim of the DARTree blog post,
// section 4; the pages print no rule for T > 0, this is the plainest lossless one
// for deterministically chosen children).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace dartree {

// Philox4x32-10 from its published definition: ten rounds of two 32x32 -> 64-bit
// products, the key bumped by the Weyl increments before every round but the first.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    }
    return c;
}

// What a row's winning token is: the maximum (greedy) or a draw at temperature T.
struct Draw {
    float temp;       // T > 0
    uint32_t k0, k1;  // seed words
    uint32_t row, request;
};

// x_v / T + G_v in float32 for the uniform word w of token v.
__device__ __forceinline__ float perturb(float x, uint32_t w, float temp) {
    const float u = float(int((w >> 9) * 2u + 1u)) * 5.9604644775390625e-8f;  // exact: odd < 2^24, times 2^-24
    const float g = -logf(-logf(u));
    return __fadd_rn(__fdiv_rn(x, temp), g);
}

template <typename T>
__device__ __forceinline__ float elem_f32(const T* row, int q) {
    if constexpr (sizeof(T) == 2) return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(row)[q]);
    else return row[q];
}

// Key (value, ~token) of token q of the row: its own value, or its perturbed value.
template <typename T, bool DRAW>
__device__ __forceinline__ uint64_t elem_key(const T* __restrict__ row, int q, const Draw& dr) {
    if constexpr (DRAW) {
        const uint4 w = philox4x32_10(make_uint4(uint32_t(q) >> 2, dr.row, dr.request, 0u), dr.k0, dr.k1);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        const float y = perturb(elem_f32<T>(row, q), ws[q & 3], dr.temp);
        return (uint64_t(ord_f32(y)) << 32) | (0xffffffffu - uint32_t(q));
    } else {
        return (uint64_t(ValueKey<T>::ord(row[q])) << 32) | (0xffffffffu - uint32_t(q));
    }
}

// Largest key over row[lo, hi) for this thread's share of the elements.
template <typename T, bool DRAW = false>
__device__ __forceinline__ uint64_t seg_max_key(const T* __restrict__ row, int lo, int hi, bool vec_ok,
                                                const Draw& dr = Draw{}) {
    constexpr int VEC = ValueKey<T>::VEC;
    uint64_t best = 0;
    int i = lo;
    if (vec_ok) {
        const int a = min(hi, int((lo + VEC - 1) / VEC * VEC));
        for (int q = lo + threadIdx.x; q < a; q += blockDim.x) {
            const uint64_t k = elem_key<T, DRAW>(row, q, dr);
            best = k > best ? k : best;
        }
        const int nv = (hi - a) / VEC;
        const uint4* v4 = reinterpret_cast<const uint4*>(row + a);
        for (int q = threadIdx.x; q < nv; q += blockDim.x) {
            const uint4 v = __ldg(v4 + q);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            const int b = a + q * VEC;  // a multiple of VEC (4 or 8): whole Philox blocks
            uint32_t nz[VEC];
            if constexpr (DRAW) {
#pragma unroll
                for (int h = 0; h < VEC / 4; ++h) {
                    const uint4 z =
                        philox4x32_10(make_uint4(uint32_t(b) / 4u + h, dr.row, dr.request, 0u), dr.k0, dr.k1);
                    nz[4 * h] = z.x;
                    nz[4 * h + 1] = z.y;
                    nz[4 * h + 2] = z.z;
                    nz[4 * h + 3] = z.w;
                }
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                uint32_t o;
                if constexpr (DRAW) {
                    float x;
                    if constexpr (VEC == 8) x = bf16_bits_to_float((w[e >> 1] >> ((e & 1) * 16)) & 0xffffu);
                    else x = __uint_as_float(w[e]);
                    o = ord_f32(perturb(x, nz[e], dr.temp));
                } else {
                    if constexpr (VEC == 8) o = ord_bf16((w[e >> 1] >> ((e & 1) * 16)) & 0xffffu);
                    else o = ord_f32(__uint_as_float(w[e]));
                }
                const uint64_t k = (uint64_t(o) << 32) | (0xffffffffu - uint32_t(b + e));
                best = k > best ? k : best;
            }
        }
        i = a + nv * VEC;
    }
    for (int q = i + threadIdx.x; q < hi; q += blockDim.x) {
        const uint64_t k = elem_key<T, DRAW>(row, q, dr);
        best = k > best ? k : best;
    }
    return best;
}

// ----------------------------------------------------------------------------- per-position rows

constexpr int RM_NT = 256;

// Row maxima (DRAW = false) or drawn tokens (DRAW = true) of [C*L, V] rows; row
// index = request * L + depth. One CTA per (segment, row); keys combined by atomicMax.
template <typename T, bool DRAW>
__device__ __forceinline__ void row_keys(const T* __restrict__ x, int V, int seg, int L, Draw dr,
                                         unsigned long long* __restrict__ keys) {
    const int row = blockIdx.y;
    const int lo = blockIdx.x * seg, hi = min(V, lo + seg);
    const T* r = x + size_t(row) * V;
    const bool vec_ok = (reinterpret_cast<uintptr_t>(r) % 16) == 0;
    if constexpr (DRAW) {
        dr.request = uint32_t(row / L);
        dr.row = uint32_t(row % L);
    }
    uint64_t k = seg_max_key<T, DRAW>(r, lo, hi, vec_ok, dr);
    k = warp_max_u64(k);
    __shared__ uint64_t red[RM_NT / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = k;
    __syncthreads();
    if (threadIdx.x < 32) {
        uint64_t v = threadIdx.x < RM_NT / 32 ? red[threadIdx.x] : 0;
        v = warp_max_u64(v);
        if (threadIdx.x == 0) atomicMax(keys + row, (unsigned long long)v);
    }
}

template <typename T>
__global__ void __launch_bounds__(RM_NT) rowmax_kernel(const T* __restrict__ x, int V, int seg,
                                                       unsigned long long* __restrict__ keys) {
    row_keys<T, false>(x, V, seg, 1, Draw{}, keys);
}

template <typename T>
__global__ void __launch_bounds__(RM_NT) rowsample_kernel(const T* __restrict__ x, int V, int seg, int L, Draw dr,
                                                          unsigned long long* __restrict__ keys) {
    row_keys<T, true>(x, V, seg, L, dr, keys);
}

__global__ void walk_position_kernel(int L, int B, const int32_t* __restrict__ tok, const int32_t* __restrict__ par,
                                     const int32_t* __restrict__ depth, const int32_t* __restrict__ n_nodes,
                                     const unsigned long long* __restrict__ keys, int32_t* __restrict__ accepted,
                                     int32_t* __restrict__ path, int32_t* __restrict__ bonus, int* status) {
    const int r = blockIdx.x;
    const int lane = threadIdx.x;
    const int S = B + 1;
    const int n = min(S, n_nodes[r]);
    const int32_t* tk = tok + size_t(r) * S;
    const int32_t* pr = par + size_t(r) * S;
    const int32_t* dp = depth + size_t(r) * S;
    int cur = 0, acc = 0, bon = -1;
    for (int step = 0;; ++step) {
        if (step > L) {  // more steps than depths: malformed tree
            if (lane == 0) set_status(status, DARTREE_EINTERNAL);
            break;
        }
        const int d = dp[cur];
        if (d < 0 || d >= L) break;
        const int t = int(0xffffffffu - uint32_t(keys[size_t(r) * L + d]));
        int found = -1;
        for (int j0 = 1; j0 < n && found < 0; j0 += 32) {
            const int j = j0 + lane;
            const bool hit = j < n && pr[j] == cur && tk[j] == t;
            const uint32_t b = __ballot_sync(0xffffffffu, hit);
            if (b) found = j0 + __ffs(b) - 1;
        }
        if (found < 0) { bon = t; break; }
        if (lane == 0 && acc < L) path[size_t(r) * L + acc] = found;
        ++acc;
        cur = found;
    }
    for (int q = acc + lane; q < L; q += 32) path[size_t(r) * L + q] = -1;
    if (lane == 0) { accepted[r] = acc; bonus[r] = bon; }
}

// ----------------------------------------------------------------------------- per-node rows

constexpr int WK_NT = 512;

template <typename T, bool DRAW>
__global__ void __launch_bounds__(WK_NT) walk_node_kernel(int L, int B, int V, int seg, Draw dr,
                                                          const T* __restrict__ target,
                                                          const int32_t* __restrict__ tok,
                                                          const int32_t* __restrict__ par,
                                                          const int32_t* __restrict__ n_nodes,
                                                          int32_t* __restrict__ accepted, int32_t* __restrict__ path,
                                                          int32_t* __restrict__ bonus, int* status) {
    __shared__ uint64_t part[2][8];
    __shared__ uint64_t red[WK_NT / 32];
    __shared__ int found_s;
    const uint32_t S = cluster_nctarank(), cr = cluster_ctarank();
    const int r = blockIdx.x / S;
    const int SL = B + 1;
    const int n = min(SL, n_nodes[r]);
    const int32_t* tk = tok + size_t(r) * SL;
    const int32_t* pr = par + size_t(r) * SL;
    const int lo = int(cr) * seg, hi = min(V, lo + seg);
    int cur = 0, acc = 0, bon = -1;
    for (int step = 0; step <= L; ++step) {
        const T* row = target + (size_t(r) * SL + cur) * V;
        const bool vec_ok = (reinterpret_cast<uintptr_t>(row) % 16) == 0;
        dr.request = uint32_t(r);
        dr.row = uint32_t(cur);
        uint64_t k = warp_max_u64(seg_max_key<T, DRAW>(row, lo, hi, vec_ok, dr));
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = k;
        if (threadIdx.x == 0) found_s = 0x7fffffff;
        __syncthreads();
        if (threadIdx.x < 32) {
            uint64_t v = threadIdx.x < WK_NT / 32 ? red[threadIdx.x] : 0;
            v = warp_max_u64(v);
            if (threadIdx.x < S) st_dsmem_u64(dsmem_addr(&part[step & 1][cr], threadIdx.x), v);
        }
        cluster_sync();
        uint64_t best = 0;
        for (uint32_t q = 0; q < S; ++q) best = part[step & 1][q] > best ? part[step & 1][q] : best;
        const int t = int(0xffffffffu - uint32_t(best));
        for (int j = 1 + threadIdx.x; j < n; j += WK_NT)
            if (pr[j] == cur && tk[j] == t) atomicMin(&found_s, j);
        __syncthreads();
        const int f = found_s;
        __syncthreads();
        if (f == 0x7fffffff) { bon = t; break; }
        if (cr == 0 && threadIdx.x == 0 && acc < L) path[size_t(r) * L + acc] = f;
        ++acc;
        cur = f;
        if (acc > L) {  // more steps than depths: malformed tree
            if (cr == 0 && threadIdx.x == 0) set_status(status, DARTREE_EINTERNAL);
            break;
        }
    }
    if (cr == 0) {
        for (int q = acc + threadIdx.x; q < L; q += WK_NT) path[size_t(r) * L + q] = -1;
        if (threadIdx.x == 0) { accepted[r] = acc; bonus[r] = bon; }
    }
}

// ----------------------------------------------------------------------------- host

// Row maxima of per-position target rows [C*L, V] into keys (value, ~token).
template <typename T, bool DRAW = false>
static int launch_rowmax_t(int rows, int V, const void* target, unsigned long long* keys, cudaStream_t stream,
                           int L = 1, Draw dr = Draw{}) {
    if (cudaMemsetAsync(keys, 0, size_t(rows) * sizeof(unsigned long long), stream) != cudaSuccess)
        return DARTREE_ECUDA;
    // a draw costs a Philox block per 4 tokens and two logarithms per token: more CTAs
    int splits = ((DRAW ? 4 : 2) * num_sms() + rows - 1) / rows;
    const int min_seg = DRAW ? 1024 : 4096;
    if (splits > (V + min_seg - 1) / min_seg) splits = (V + min_seg - 1) / min_seg;
    if (splits < 1) splits = 1;
    int seg = (V + splits - 1) / splits;
    seg = (seg + 7) / 8 * 8;
    splits = (V + seg - 1) / seg;
    {
        KTimer kt_(DRAW ? KID_ROWSAMPLE : KID_ROWMAX, stream);
        if constexpr (DRAW)
            rowsample_kernel<T>
                <<<dim3(splits, rows), RM_NT, 0, stream>>>(static_cast<const T*>(target), V, seg, L, dr, keys);
        else
            rowmax_kernel<T><<<dim3(splits, rows), RM_NT, 0, stream>>>(static_cast<const T*>(target), V, seg, keys);
    }
    return cudaGetLastError() == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

int launch_walk_position(int C, int L, int B, const int32_t* tok, const int32_t* par, const int32_t* depth,
                         const int32_t* n_nodes, const unsigned long long* keys, int32_t* accepted, int32_t* path,
                         int32_t* bonus, int* status, cudaStream_t stream) {
    if (C == 0) return DARTREE_OK;
    {
        KTimer kt_(KID_WALK, stream);
        walk_position_kernel<<<C, 32, 0, stream>>>(L, B, tok, par, depth, n_nodes, keys, accepted, path, bonus,
                                                   status);
    }
    return cudaGetLastError() == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

int launch_rowmax_position(int C, int L, int V, int dtype, const void* target, unsigned long long* keys,
                           cudaStream_t stream) {
    if (C == 0) return DARTREE_OK;
    return dtype == DARTREE_BF16 ? launch_rowmax_t<bf16_t>(C * L, V, target, keys, stream)
                                 : launch_rowmax_t<float>(C * L, V, target, keys, stream);
}

template <typename T, bool DRAW>
static int launch_verify_t(int C, int L, int B, const int32_t* tok, const int32_t* par, const int32_t* depth,
                           const int32_t* n_nodes, const void* target, int rows_mode, int V,
                           unsigned long long* keys, int32_t* accepted, int32_t* path, int32_t* bonus,
                           int* status, cudaStream_t stream, Draw dr) {
    const T* tg = static_cast<const T*>(target);
    if (rows_mode == DARTREE_ROWS_PER_POSITION) {
        if (int e = launch_rowmax_t<T, DRAW>(C * L, V, target, keys, stream, L, dr)) return e;
        {
            KTimer kt_(KID_WALK, stream);
            walk_position_kernel<<<C, 32, 0, stream>>>(L, B, tok, par, depth, n_nodes, keys, accepted, path, bonus,
                                                       status);
        }
        return cudaGetLastError() == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
    }
    const int S = 8;
    int seg = (V + S - 1) / S;
    seg = (seg + 7) / 8 * 8;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(C) * S);
    cfg.blockDim = dim3(WK_NT);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    {
        KTimer kt_(KID_WALK, stream);
        e = cudaLaunchKernelEx(&cfg, walk_node_kernel<T, DRAW>, L, B, V, seg, dr, tg, tok, par, n_nodes, accepted,
                               path, bonus, status);
    }
    return e == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

int launch_verify(int C, int L, int B, const int32_t* tok, const int32_t* par, const int32_t* depth,
                  const int32_t* n_nodes, const void* target, int rows_mode, int V, int dtype,
                  unsigned long long* keys, int32_t* accepted, int32_t* path, int32_t* bonus, int* status,
                  cudaStream_t stream) {
    if (C == 0) return DARTREE_OK;
    if (dtype == DARTREE_BF16)
        return launch_verify_t<bf16_t, false>(C, L, B, tok, par, depth, n_nodes, target, rows_mode, V, keys,
                                              accepted, path, bonus, status, stream, Draw{});
    return launch_verify_t<float, false>(C, L, B, tok, par, depth, n_nodes, target, rows_mode, V, keys, accepted,
                                         path, bonus, status, stream, Draw{});
}

int launch_verify_sample(int C, int L, int B, const int32_t* tok, const int32_t* par, const int32_t* depth,
                         const int32_t* n_nodes, const void* target, int rows_mode, int V, int dtype, float temp,
                         uint64_t seed, unsigned long long* keys, int32_t* accepted, int32_t* path, int32_t* bonus,
                         int* status, cudaStream_t stream) {
    if (C == 0) return DARTREE_OK;
    const Draw dr{temp, uint32_t(seed & 0xffffffffu), uint32_t(seed >> 32), 0u, 0u};
    if (dtype == DARTREE_BF16)
        return launch_verify_t<bf16_t, true>(C, L, B, tok, par, depth, n_nodes, target, rows_mode, V, keys,
                                             accepted, path, bonus, status, stream, dr);
    return launch_verify_t<float, true>(C, L, B, tok, par, depth, n_nodes, target, rows_mode, V, keys, accepted,
                                        path, bonus, status, stream, dr);
}

}  // namespace dartree
