// Node-by-node best-first search with one correction-head evaluation per popped
// node: the "heap pop -> correction" drafting that DARTree's deferred pruning
// replaces (DARTree blog post, section 2, latency breakdown, and section 4.3,
// Table 2: the same tree built by popping nodes one at a time and running the
// head on each). It reuses S1 and the candidate-side projection (G = E[cand] W_q)
// of the deferred path, so the two differ only in the search.
//
// One CTA of 512 threads per request keeps every pushed child's key in shared
// memory (K per expansion: the root's, then one expansion per popped node). Step t:
//   pop    the largest key (block-wide maximum; a popped key is cleared);
//   state  h_t = RMSNorm(h_parent + E[tok] + H_d[depth-1]) (bf16, as the deferred
//          path stores it), the parent's row read back from the workspace;
//   expand if depth < L: z[c] = L^base[depth, c] + <h_t, G_c> / sqrt(H) for the K
//          candidates of position `depth` (G as its bf16 pair, every warp a quarter
//          of the candidates), log-softmax over the K, and the K children's keys.
// Keys order children by (score desc, depth asc, push order asc): the push order
// (expansion index * K + candidate rank) is the order a binary heap with that key
// and an insertion counter pops equal scores in.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace dartree {

constexpr int HP_NT = 512, HP_NW = HP_NT / 32;
constexpr int HP_MAXK = 64, HP_MAXB = 256, HP_MAXH = 8192;

struct HeapArgs {
    const uint16_t* E;
    const uint16_t* hidden;
    const int32_t* anchor;
    const int32_t* cand_tok;
    const float* cand_val;
    const uint16_t* Ghi;
    const uint16_t* Glo;
    int H, L, K, B;
    float beta, inv_sqrt_h;
    uint16_t* hws;  // [C, B, H] popped nodes' states
    int32_t* o_tok;
    int32_t* o_par;
    int32_t* o_dep;
    float* o_sc;
    int* status;
};

// Key of a pushed child: score, then shallower depth, then earlier push.
__device__ __forceinline__ uint64_t heap_key(float s, int depth, int push) {
    s += 0.f;  // -0 -> +0
    return (uint64_t(ord_f32(s)) << 32) | (uint64_t(0xffffu - uint32_t(depth)) << 16) | (0xffffu - uint32_t(push));
}

__global__ void __launch_bounds__(HP_NT, 1) heap_search_kernel(HeapArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int H = a.H, L = a.L, K = a.K, B = a.B;
    uint64_t* keys = reinterpret_cast<uint64_t*>(smem);              // [(B + 1) * K]
    uint64_t* wbest = keys + size_t(B + 1) * K;                       // [HP_NW]
    float* hcur = reinterpret_cast<float*>(wbest + HP_NW);            // [H] state of the node being expanded
    float* zc = hcur + H;                                             // [HP_MAXK]
    float* wsum = zc + HP_MAXK;                                       // [HP_NW]
    int* widx = reinterpret_cast<int*>(wsum + HP_NW);                 // [HP_NW]
    int* pdep = widx + HP_NW;                                         // [HP_MAXB] depth of every popped node
    int* misc = pdep + HP_MAXB;                                       // [0] winner
    const int r = blockIdx.x, lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const size_t hrow = size_t(r) * B;

    // root: h = E[anchor], score 0, depth 0
    const uint16_t* er = a.E + size_t(a.anchor[r]) * H;
    for (int f = threadIdx.x; f < H; f += HP_NT) hcur[f] = bf16_bits_to_float(er[f]);
    int nd = 0;        // depth of the node being expanded
    float ns = 0.f;    // its score
    __syncthreads();
    for (int t = 0; t <= B; ++t) {
        // ---- expansion t (t = 0: the root) of a node at depth nd < L: its K children
        if (nd < L) {
            const size_t crow = (size_t(r) * L + nd) * K;
            for (int c = wid; c < K; c += HP_NW) {
                const uint4* gh = reinterpret_cast<const uint4*>(a.Ghi + (crow + c) * H);
                const uint4* gl = reinterpret_cast<const uint4*>(a.Glo + (crow + c) * H);
                float ah = 0.f, al = 0.f;
                for (int v = lane; v < H / 8; v += 32) {
                    const uint4 x = __ldg(gh + v), y = __ldg(gl + v);
                    const uint32_t wx[4] = {x.x, x.y, x.z, x.w}, wy[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float hv = hcur[v * 8 + i];
                        const int sh = (i & 1) ? 16 : 0;
                        ah = fmaf(hv, bf16_bits_to_float((wx[i >> 1] >> sh) & 0xffffu), ah);
                        al = fmaf(hv, bf16_bits_to_float((wy[i >> 1] >> sh) & 0xffffu), al);
                    }
                }
                ah = warp_sum(ah);
                al = warp_sum(al);
                if (lane == 0) zc[c] = a.cand_val[crow + c] + (ah + al) * a.inv_sqrt_h;
            }
            __syncthreads();
            if (wid == 0) {  // log-softmax over the K candidates, the children's keys
                float zv[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) zv[h] = lane + 32 * h < K ? zc[lane + 32 * h] : -INFINITY;
                const float mx = warp_max(fmaxf(zv[0], zv[1]));
                float se = 0.f;
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    if (lane + 32 * h < K) se += expf(zv[h] - mx);
                se = warp_sum(se);
                const float lse = mx + logf(se);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c = lane + 32 * h;
                    if (c < K) keys[size_t(t) * K + c] = heap_key((ns + (zv[h] - lse)) + a.beta, nd + 1, t * K + c);
                }
            }
        } else {
            for (int c = threadIdx.x; c < K; c += HP_NT) keys[size_t(t) * K + c] = 0ull;
        }
        __syncthreads();
        if (t == B) break;
        // ---- pop the best pushed key (keys are distinct: the push order is in the low bits)
        uint64_t best = 0;
        int bi = -1;
        for (int i = threadIdx.x; i < (t + 1) * K; i += HP_NT) {
            const uint64_t k = keys[i];
            if (k > best) {
                best = k;
                bi = i;
            }
        }
        {
            const uint64_t wb = warp_max_u64(best);
            const uint32_t m = __ballot_sync(0xffffffffu, best == wb && wb != 0);
            const int wbi = __shfl_sync(0xffffffffu, bi, m ? __ffs(m) - 1 : 0);
            if (lane == 0) {
                wbest[wid] = wb;
                widx[wid] = m ? wbi : -1;
            }
        }
        __syncthreads();
        if (wid == 0) {
            const uint64_t v = lane < HP_NW ? wbest[lane] : 0ull;
            const uint64_t w = warp_max_u64(v);
            const uint32_t m = __ballot_sync(0xffffffffu, lane < HP_NW && v == w && w != 0);
            if (lane == 0) misc[0] = m ? widx[__ffs(m) - 1] : -1;
        }
        __syncthreads();
        const int e = misc[0];
        if (e < 0) {  // fewer nodes than the budget (cannot happen for B <= L * K): empty slots
            for (int q = t + threadIdx.x; q < B; q += HP_NT) {
                a.o_tok[hrow + q] = -1;
                a.o_par[hrow + q] = -1;
                a.o_dep[hrow + q] = -1;
                a.o_sc[hrow + q] = 0.f;
            }
            break;
        }
        const uint64_t key = keys[e];
        const int j = e / K, c = e - j * K;               // expansion j: the root (0) or pop j - 1
        const int depth = j == 0 ? 1 : pdep[j - 1] + 1;
        const float sc = f32_from_ord(uint32_t(key >> 32));
        const int tok = a.cand_tok[(size_t(r) * L + depth - 1) * K + c];
        __syncthreads();  // every thread read the winner before its key is cleared
        if (threadIdx.x == 0) {
            keys[e] = 0ull;
            pdep[t] = depth;
            a.o_tok[hrow + t] = tok;
            a.o_par[hrow + t] = j - 1;
            a.o_dep[hrow + t] = depth;
            a.o_sc[hrow + t] = sc;
        }
        // ---- state of the popped node: RMSNorm(h_parent + E[tok] + H_d[depth-1]) in bf16
        const uint16_t* hp = j == 0 ? er : a.hws + (hrow + j - 1) * H;
        const uint16_t* et = a.E + size_t(tok) * H;
        const uint16_t* hd = a.hidden + (size_t(r) * L + depth - 1) * H;
        float ss = 0.f;
        for (int f = threadIdx.x; f < H; f += HP_NT) {
            const float x = (bf16_bits_to_float(hp[f]) + bf16_bits_to_float(et[f])) + bf16_bits_to_float(hd[f]);
            hcur[f] = x;
            ss = fmaf(x, x, ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) wsum[wid] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < HP_NW; ++w) tot += wsum[w];
        const float inv = 1.0f / sqrtf(tot / float(H) + 1e-6f);
        uint16_t* hw = a.hws + (hrow + t) * H;
        for (int f = threadIdx.x; f < H; f += HP_NT) {
            const uint16_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hcur[f] * inv));
            hw[f] = b;
            hcur[f] = bf16_bits_to_float(b);
        }
        nd = depth;
        ns = sc;
        __syncthreads();
    }
}

size_t heap_smem_bytes(int H, int K, int B) {
    return size_t(B + 1) * K * 8 + HP_NW * 8 + size_t(H) * 4 + HP_MAXK * 4 + HP_NW * 8 + HP_MAXB * 4 + 16;
}

bool heap_supported(int H, int K, int B) {
    return K >= 1 && K <= HP_MAXK && B >= 1 && B <= HP_MAXB && H % 8 == 0 && H <= HP_MAXH &&
           heap_smem_bytes(H, K, B) <= 200 * 1024;
}

int launch_heap_search(const void* E, const void* hidden, const int32_t* anchor, const int32_t* cand_tok,
                       const float* cand_val, const uint16_t* Ghi, const uint16_t* Glo, int C, int H, int L, int K,
                       int B, float beta, uint16_t* hws, int32_t* tok, int32_t* par, int32_t* depth, float* score,
                       int* status, cudaStream_t stream) {
    if (C == 0) return DARTREE_OK;
    if (!heap_supported(H, K, B)) return DARTREE_EUNSUPPORTED;
    const size_t smem = heap_smem_bytes(H, K, B);
    if (cudaFuncSetAttribute(heap_search_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
        cudaSuccess)
        return DARTREE_ECUDA;
    HeapArgs x{static_cast<const uint16_t*>(E), static_cast<const uint16_t*>(hidden), anchor, cand_tok, cand_val,
               Ghi, Glo, H, L, K, B, beta, 1.0f / sqrtf(float(H)), hws, tok, par, depth, score, status};
    {
        KTimer kt_(KID_HEAP, stream);
        heap_search_kernel<<<C, HP_NT, smem, stream>>>(x);
    }
    return cudaGetLastError() == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

}  // namespace dartree
