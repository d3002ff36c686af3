// S2-S7: depth-wise tree expansion with the stand-in correction head
// (DARTree blog post, 3.1 "Basic flow": depth-wise expansion, scoring function,
// per-depth pruning; the ainews.surl.tw article: all active branches are
// processed in batches, one tree depth at a time).
//
// Per depth d = 1..L, over all C requests at once:
//   proj     U[m, :] = W_q h_m              (all C*P parents in one matrix product)
//   contract z[r, p, c] = L^base[r, d-1, c] + <U[r*P+p], E[cand_c]> / sqrt(H)
//   select   log q = z - logsumexp_c z; s = s_p + log q + beta;
//            keep the top-W children by (s desc, flat index p*K+c asc);
//            h_child = RMSNorm(h_p + E[tok] + H_d[d-1]) stored in the input type.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace dartree {

// --------------------------------------------------------------------------- root

template <typename T>
__global__ void root_init_kernel(const T* __restrict__ E, const int32_t* __restrict__ anchor, int H,
                                 T* __restrict__ h0, float* __restrict__ s0) {
    const int r = blockIdx.x;
    const T* e = E + size_t(anchor[r]) * H;
    for (int j = threadIdx.x; j < H; j += blockDim.x) h0[size_t(r) * H + j] = e[j];
    if (threadIdx.x == 0) s0[r] = 0.f;
}

// --------------------------------------------------------------------------- projection (CUDA cores)

constexpr int PJ_TM = 32, PJ_TN = 64, PJ_TK = 32, PJ_NT = 256;

template <typename T>
__global__ void __launch_bounds__(PJ_NT) proj_simple_kernel(const T* __restrict__ h, const T* __restrict__ Wq,
                                                            float* __restrict__ U, int M, int H) {
    __shared__ float hs[PJ_TK][PJ_TM + 1];
    __shared__ float ws[PJ_TK][PJ_TN + 1];
    const int m0 = blockIdx.y * PJ_TM, n0 = blockIdx.x * PJ_TN;
    const int tm = threadIdx.x / 16, tn = threadIdx.x % 16;  // 2 rows x 4 cols per thread
    float acc[2][4] = {};
    for (int k0 = 0; k0 < H; k0 += PJ_TK) {
        for (int i = threadIdx.x; i < PJ_TM * PJ_TK; i += PJ_NT) {
            const int mm = i / PJ_TK, kk = i % PJ_TK;
            const int m = m0 + mm, k = k0 + kk;
            hs[kk][mm] = (m < M && k < H) ? to_float(h[size_t(m) * H + k]) : 0.f;
        }
        for (int i = threadIdx.x; i < PJ_TN * PJ_TK; i += PJ_NT) {
            const int nn = i / PJ_TK, kk = i % PJ_TK;
            const int n = n0 + nn, k = k0 + kk;
            ws[kk][nn] = (n < H && k < H) ? to_float(Wq[size_t(n) * H + k]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < PJ_TK; ++kk) {
            const float a0 = hs[kk][tm * 2], a1 = hs[kk][tm * 2 + 1];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float b = ws[kk][tn + 16 * q];
                acc[0][q] = fmaf(a0, b, acc[0][q]);
                acc[1][q] = fmaf(a1, b, acc[1][q]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < 2; ++a) {
        const int m = m0 + tm * 2 + a;
        if (m >= M) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int n = n0 + tn + 16 * q;
            if (n < H) U[size_t(m) * H + n] = acc[a][q];
        }
    }
}

// --------------------------------------------------------------------------- candidate contraction (CUDA cores)

constexpr int CT_NT = 256, CT_CPW = 4, CT_PT = 16;  // candidates per warp, parents per pass

template <typename T>
__device__ __forceinline__ void load4(const T* p, float (&v)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&v)[4]) {
    const float4 x = *reinterpret_cast<const float4*>(p);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
template <>
__device__ __forceinline__ void load4<bf16_t>(const bf16_t* p, float (&v)[4]) {
    const uint2 x = *reinterpret_cast<const uint2*>(p);
    v[0] = bf16_bits_to_float(x.x & 0xffffu); v[1] = bf16_bits_to_float(x.x >> 16);
    v[2] = bf16_bits_to_float(x.y & 0xffffu); v[3] = bf16_bits_to_float(x.y >> 16);
}

template <typename T>
__global__ void __launch_bounds__(CT_NT) contract_simple_kernel(const float* __restrict__ U, const T* __restrict__ E,
                                                                const int32_t* __restrict__ cand_tok,
                                                                const float* __restrict__ cand_val,
                                                                float* __restrict__ z, int P, int K, int H, int L,
                                                                int d, float inv_sqrt_h) {
    const int r = blockIdx.y;
    const size_t crow = (size_t(r) * L + (d - 1)) * K;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int cbase = (blockIdx.x * (CT_NT / 32) + wid) * CT_CPW;
    if (cbase >= K) return;
    const T* erow[CT_CPW];
#pragma unroll
    for (int q = 0; q < CT_CPW; ++q) {
        const int c = min(cbase + q, K - 1);
        erow[q] = E + size_t(cand_tok[crow + c]) * H;
    }
    for (int p0 = 0; p0 < P; p0 += CT_PT) {
        float acc[CT_PT][CT_CPW];
#pragma unroll
        for (int p = 0; p < CT_PT; ++p)
#pragma unroll
            for (int q = 0; q < CT_CPW; ++q) acc[p][q] = 0.f;
        for (int j = lane * 4; j < H; j += 128) {
            float e[CT_CPW][4];
#pragma unroll
            for (int q = 0; q < CT_CPW; ++q) load4<T>(erow[q] + j, e[q]);
#pragma unroll
            for (int p = 0; p < CT_PT; ++p) {
                if (p0 + p < P) {
                    float u[4];
                    load4<float>(U + (size_t(r) * P + p0 + p) * H + j, u);
#pragma unroll
                    for (int q = 0; q < CT_CPW; ++q)
                        acc[p][q] = fmaf(u[0], e[q][0], fmaf(u[1], e[q][1], fmaf(u[2], e[q][2], fmaf(u[3], e[q][3], acc[p][q]))));
                }
            }
        }
#pragma unroll
        for (int p = 0; p < CT_PT; ++p) {
            if (p0 + p >= P) break;
#pragma unroll
            for (int q = 0; q < CT_CPW; ++q) {
                const float s = warp_sum(acc[p][q]);
                const int c = cbase + q;
                if (lane == 0 && c < K)
                    z[(size_t(r) * P + p0 + p) * K + c] = cand_val[crow + c] + s * inv_sqrt_h;
            }
        }
    }
}

// --------------------------------------------------------------------------- select: softmax, score, top-W, state

constexpr int SL_NT = 512;
constexpr int SL_NW = SL_NT / 32;

// One depth's log-softmax, scores, top-W and state update for the per-depth
// (large batch) path, one CTA per request: the selection runs once, then the
// kept children's state rows are built in parallel, one group of warps per row.
template <typename T>
__global__ void __launch_bounds__(SL_NT) select_kernel(
    const float* __restrict__ z, const float* __restrict__ s_cur, const T* __restrict__ h_cur,
    const int32_t* __restrict__ cand_tok,  // [C, L, K] base of the table
    const T* __restrict__ E, const T* __restrict__ hidden, int P, int K, int W, int H, int L, int d, float beta,
    int32_t* __restrict__ st_tok, int32_t* __restrict__ st_par, float* __restrict__ st_s, int32_t* __restrict__ st_n,
    T* __restrict__ h_next, float* __restrict__ s_next, int update_state, int* status) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int r = blockIdx.x;
    const int n = P * K;
    const int n_keep = min(W, n);
    uint64_t* keys = reinterpret_cast<uint64_t*>(smem);         // n
    uint64_t* cands = keys + n;                                  // 16 * W
    uint64_t* sel = cands + SL_NW * W;                           // W
    float* lse = reinterpret_cast<float*>(sel + W);              // P
    // (no reduction scratch: state rows are built by state_kernel)
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const float* zr = z + size_t(r) * P * K;
    const int32_t* ct = cand_tok + (size_t(r) * L + (d - 1)) * K;
    (void)status;

    for (int p = wid; p < P; p += SL_NW) {
        float m = -INFINITY;
        for (int c = lane; c < K; c += 32) m = fmaxf(m, zr[size_t(p) * K + c]);
        m = warp_max(m);
        float sum = 0.f;
        for (int c = lane; c < K; c += 32) sum += expf(zr[size_t(p) * K + c] - m);
        sum = warp_sum(sum);
        if (lane == 0) lse[p] = m + logf(sum);
    }
    __syncthreads();
    for (int f = threadIdx.x; f < n; f += SL_NT) {
        const int p = f / K;
        float sc = (s_cur[size_t(r) * P + p] + (zr[f] - lse[p])) + beta;
        sc += 0.f;
        keys[f] = (uint64_t(ord_f32(sc)) << 32) | (0xffffffffu - uint32_t(f));
    }
    __syncthreads();
    block_top_keys<SL_NT>(keys, n, n_keep, cands, sel);

    const size_t sto = (size_t(r) * L + (d - 1)) * W;
    for (int k = threadIdx.x; k < W; k += SL_NT) {
        if (k < n_keep) {
            const uint64_t key = sel[k];
            const uint32_t f = 0xffffffffu - uint32_t(key);
            const float sc = f32_from_ord(uint32_t(key >> 32));
            st_tok[sto + k] = ct[f % uint32_t(K)];
            st_par[sto + k] = int(f / uint32_t(K));
            st_s[sto + k] = sc;
            s_next[size_t(r) * n_keep + k] = sc;
        } else {
            st_tok[sto + k] = -1;
            st_par[sto + k] = -1;
            st_s[sto + k] = 0.f;
        }
    }
    if (threadIdx.x == 0) st_n[size_t(r) * L + (d - 1)] = n_keep;
    (void)h_cur; (void)E; (void)hidden; (void)H; (void)h_next; (void)update_state;
}

// The same selection for W <= 16, P <= 16 and K <= 1024, one CTA per request:
// warp p takes parent row p with its K logits in registers (EPL per lane): the
// log-softmax and scores (the same arithmetic in the same order as above), then
// the row's best m = min(W, K) keys by m rounds of "largest remaining key of the
// warp", sorted into a list. The 16 lists (empty beyond P) are merged by a
// bitonic tree of 16-key merges.
template <int EPL>
__global__ void __launch_bounds__(SL_NT) select_rows_kernel(
    const float* __restrict__ z, const float* __restrict__ s_cur, const int32_t* __restrict__ cand_tok, int P, int K,
    int W, int L, int d, float beta, int32_t* __restrict__ st_tok, int32_t* __restrict__ st_par,
    float* __restrict__ st_s, int32_t* __restrict__ st_n, float* __restrict__ s_next) {
    __shared__ uint64_t lists[16 * 16];
    __shared__ uint64_t mrg[2 * 8 * 16];
    const int r = blockIdx.x;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int n = P * K, n_keep = min(W, n), m = min(n_keep, K);
    if (wid < P) {
        const int p = wid;
        const float* zr = z + (size_t(r) * P + p) * K;
        float zv[EPL];
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const int c = lane + 32 * j;
            zv[j] = c < K ? zr[c] : -INFINITY;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < EPL; ++j) mx = fmaxf(mx, zv[j]);
        mx = warp_max(mx);
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < EPL; ++j)
            if (lane + 32 * j < K) sum += expf(zv[j] - mx);
        sum = warp_sum(sum);
        const float lse = mx + logf(sum);
        const float sp = s_cur[size_t(r) * P + p];
        uint64_t v[EPL];
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const int c = lane + 32 * j;
            v[j] = 0ull;
            if (c < K) {
                float sc = (sp + (zv[j] - lse)) + beta;
                sc += 0.f;
                v[j] = (uint64_t(ord_f32(sc)) << 32) | (0xffffffffu - uint32_t(p * K + c));
            }
        }
        for (int k = 0; k < m; ++k) {
            uint64_t lm = 0;
#pragma unroll
            for (int j = 0; j < EPL; ++j) lm = v[j] > lm ? v[j] : lm;
            const uint64_t w = warp_max_key64(lm);
            if (w != 0 && lm == w) {
#pragma unroll
                for (int j = 0; j < EPL; ++j)
                    if (v[j] == w) v[j] = 0;
            }
            if (lane == 0) lists[p * 16 + k] = w;
        }
    }
    __syncthreads();
    // merge tree: level 1, warp w merges lists 2w and 2w + 1
    const int hl = lane & 15;
    uint64_t v = 0;
    if (wid < 8) {
        const int q = 2 * wid + (lane >> 4);
        v = (q < P && hl < m) ? lists[q * 16 + hl] : 0ull;
        v = xg_merge16(v);
        if (lane < 16) mrg[wid * 16 + lane] = v;
    }
    __syncthreads();
    int in = 0;
    for (int nm = 4; nm >= 1; nm >>= 1) {
        if (wid < nm) {
            v = mrg[in * 128 + (2 * wid + (lane >> 4)) * 16 + hl];
            v = xg_merge16(v);
            if (lane < 16) mrg[(1 - in) * 128 + wid * 16 + lane] = v;
        }
        in = 1 - in;
        __syncthreads();
    }
    const int32_t* ct = cand_tok + (size_t(r) * L + (d - 1)) * K;
    const size_t sto = (size_t(r) * L + (d - 1)) * W;
    for (int k = threadIdx.x; k < W; k += SL_NT) {
        if (k < n_keep) {
            const uint64_t key = mrg[in * 128 + k];
            const uint32_t f = 0xffffffffu - uint32_t(key);
            const float sc = f32_from_ord(uint32_t(key >> 32));
            st_tok[sto + k] = ct[f % uint32_t(K)];
            st_par[sto + k] = int(f / uint32_t(K));
            st_s[sto + k] = sc;
            s_next[size_t(r) * n_keep + k] = sc;
        } else {
            st_tok[sto + k] = -1;
            st_par[sto + k] = -1;
            st_s[sto + k] = 0.f;
        }
    }
    if (threadIdx.x == 0) st_n[size_t(r) * L + (d - 1)] = n_keep;
}

template <int EPL>
static void launch_select_rows(const ExpandArgs& a, const float* s_cur, int P, int d, float* s_next, cudaStream_t st) {
    select_rows_kernel<EPL><<<a.C, SL_NT, 0, st>>>(a.z, s_cur, a.cand_tok, P, a.K, a.W, a.L, d, a.beta, a.st_tok,
                                                   a.st_par, a.st_s, a.st_n, s_next);
}

// true when select_rows_kernel covers the shape (and was launched)
static bool select_rows(const ExpandArgs& a, const float* s_cur, int P, int d, float* s_next, cudaStream_t st) {
    if (P > 16 || a.W > 16 || a.K > 1024) return false;
    if (a.K <= 64) launch_select_rows<2>(a, s_cur, P, d, s_next, st);
    else if (a.K <= 128) launch_select_rows<4>(a, s_cur, P, d, s_next, st);
    else if (a.K <= 256) launch_select_rows<8>(a, s_cur, P, d, s_next, st);
    else if (a.K <= 512) launch_select_rows<16>(a, s_cur, P, d, s_next, st);
    else launch_select_rows<32>(a, s_cur, P, d, s_next, st);
    return true;
}

// State rows of the kept children of one depth: h = RMSNorm(h_p + E[tok] +
// H_d[d-1]) in the storage type. Grid (n_keep, C), one CTA per row; parent and
// token come from the supertree entries just written. Every thread holds up to
// two 16-byte vectors of each input in registers, so all loads are in flight
// together.
constexpr int SU_NT = 256;

template <typename T>
__global__ void __launch_bounds__(SU_NT) state_kernel(const T* __restrict__ h_cur, const T* __restrict__ E,
                                                      const T* __restrict__ hidden,
                                                      const int32_t* __restrict__ st_tok,
                                                      const int32_t* __restrict__ st_par, int P, int W, int H, int L,
                                                      int d, T* __restrict__ h_next) {
    __shared__ float red[SU_NT / 32];
    const int k = blockIdx.x, r = blockIdx.y, n_keep = gridDim.x;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const size_t o = (size_t(r) * L + (d - 1)) * W + k;
    const T* hp = h_cur + (size_t(r) * P + st_par[o]) * H;
    const T* e = E + size_t(st_tok[o]) * H;
    const T* hd = hidden + (size_t(r) * L + (d - 1)) * H;
    T* out = h_next + (size_t(r) * n_keep + k) * H;
    constexpr int VE = 16 / sizeof(T), VR = 2;
    const int nv = H / VE;
    float xr[VR][VE];
    float ss = 0.f;
    uint4 vo[VR], ve[VR], vh[VR];
#pragma unroll
    for (int i = 0; i < VR; ++i) {
        const int v = threadIdx.x + i * SU_NT;
        if (v < nv) {
            vo[i] = __ldcg(reinterpret_cast<const uint4*>(hp) + v);  // written by the previous depth
            ve[i] = reinterpret_cast<const uint4*>(e)[v];
            vh[i] = reinterpret_cast<const uint4*>(hd)[v];
        }
    }
#pragma unroll
    for (int i = 0; i < VR; ++i) {
        if (int(threadIdx.x) + i * SU_NT < nv) {
            const T* po = reinterpret_cast<const T*>(&vo[i]);
            const T* pe = reinterpret_cast<const T*>(&ve[i]);
            const T* ph = reinterpret_cast<const T*>(&vh[i]);
#pragma unroll
            for (int j = 0; j < VE; ++j) {
                xr[i][j] = (to_float(po[j]) + to_float(pe[j])) + to_float(ph[j]);
                ss = fmaf(xr[i][j], xr[i][j], ss);
            }
        }
    }
    for (int v = threadIdx.x + VR * SU_NT; v < nv; v += SU_NT)  // rows wider than the registers
        for (int j = 0; j < VE; ++j) {
            const float x = (to_float(hp[v * VE + j]) + to_float(e[v * VE + j])) + to_float(hd[v * VE + j]);
            ss = fmaf(x, x, ss);
        }
    ss = warp_sum(ss);
    if (lane == 0) red[wid] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < SU_NT / 32; ++w) tot += red[w];
    const float rs = sqrtf(tot / float(H) + 1e-6f);
#pragma unroll
    for (int i = 0; i < VR; ++i) {
        const int v = threadIdx.x + i * SU_NT;
        if (v < nv) {
            uint4 ov;
            T* pw = reinterpret_cast<T*>(&ov);
#pragma unroll
            for (int j = 0; j < VE; ++j) pw[j] = from_float<T>(xr[i][j] / rs);
            reinterpret_cast<uint4*>(out)[v] = ov;
        }
    }
    for (int v = threadIdx.x + VR * SU_NT; v < nv; v += SU_NT)
        for (int j = 0; j < VE; ++j) {
            const float x = (to_float(hp[v * VE + j]) + to_float(e[v * VE + j])) + to_float(hd[v * VE + j]);
            out[v * VE + j] = from_float<T>(x / rs);
        }
}

static size_t select_smem(int P, int K, int W) {
    const size_t n = size_t(P) * K;
    return n * 8 + size_t(SL_NW) * W * 8 + size_t(W) * 8 + size_t(P) * 4 + SL_NW * 4 + 16;
}

// --------------------------------------------------------------------------- host loop

template <typename T>
static int launch_expand_t(const ExpandArgs& a, cudaStream_t st) {
    const T* E = static_cast<const T*>(a.E);
    const T* Wq = static_cast<const T*>(a.Wq);
    const T* hid = static_cast<const T*>(a.hidden);
    T* hb[2] = {static_cast<T*>(a.hbuf[0]), static_cast<T*>(a.hbuf[1])};
    {
        KTimer kt_(KID_OTHER, st);
        root_init_kernel<T><<<a.C, 256, 0, st>>>(E, a.anchor, a.H, hb[0], a.sbuf[0]);
    }
    const size_t smax = select_smem(a.W, a.K, a.W);
    if (cudaFuncSetAttribute(select_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smax)) != cudaSuccess)
        return DARTREE_ECUDA;
    const float inv_sqrt_h = 1.0f / sqrtf(float(a.H));
    int cur = 0, P = 1;
    for (int d = 1; d <= a.L; ++d) {
        const int M = a.C * P;
        dim3 pg((a.H + PJ_TN - 1) / PJ_TN, (M + PJ_TM - 1) / PJ_TM);
        const bool tc_proj = sizeof(T) == 2 && gemm_tc_supported(M, a.H, a.H);
        if (tc_proj && a.uhl && contract_tc_supported(P, a.H)) {
            // tensor cores for both: U as bf16 hi/lo pairs, then the gathered contraction
            if (int e = launch_gemm_bf16_tc(hb[cur], Wq, M, a.H, a.H, 1, nullptr, a.uhl, P, a.status, st, nullptr,
                                            false, nullptr, a.split))
                return e;
            if (int e = launch_contract_tc(E, a.uhl, a.cand_tok, a.cand_val, a.z, a.C, P, a.K, a.H, a.L, d,
                                           inv_sqrt_h, a.status, st))
                return e;
        } else {
            if (tc_proj) {
                if (int e = launch_gemm_bf16_tc(hb[cur], Wq, M, a.H, a.H, 0, a.U, nullptr, 1, a.status, st)) return e;
            } else {
                {
                    KTimer kt_(KID_OTHER, st);
                    proj_simple_kernel<T><<<pg, PJ_NT, 0, st>>>(hb[cur], Wq, a.U, M, a.H);
                }
            }
            dim3 cg((a.K + (CT_NT / 32) * CT_CPW - 1) / ((CT_NT / 32) * CT_CPW), a.C);
            {
                KTimer kt_(KID_CONTRACT, st);
                contract_simple_kernel<T><<<cg, CT_NT, 0, st>>>(a.U, E, a.cand_tok, a.cand_val, a.z, P, a.K, a.H, a.L, d,
                                                                inv_sqrt_h);
            }
        }
        const int n_keep = P * a.K < a.W ? P * a.K : a.W;
        {
            KTimer kt_(KID_SELECT, st);
            if (!select_rows(a, a.sbuf[cur], P, d, a.sbuf[1 - cur], st))
                select_kernel<T><<<a.C, SL_NT, select_smem(P, a.K, a.W), st>>>(
                    a.z, a.sbuf[cur], hb[cur], a.cand_tok, E, hid, P, a.K, a.W, a.H, a.L, d, a.beta, a.st_tok,
                    a.st_par, a.st_s, a.st_n, hb[1 - cur], a.sbuf[1 - cur], d < a.L ? 1 : 0, a.status);
        }
        if (d < a.L)
            {
                KTimer kt_(KID_STATE, st);
                state_kernel<T><<<dim3(n_keep, a.C), SU_NT, 0, st>>>(hb[cur], E, hid, a.st_tok, a.st_par, P, a.W, a.H,
                                                                   a.L, d, hb[1 - cur]);
            }
        cur = 1 - cur;
        P = n_keep;
    }
    return cudaGetLastError() == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

constexpr int kSplitMinC = 32;  // requests from which a batch expands as two halves

int launch_expand(const ExpandArgs& a, cudaStream_t stream) {
    bool done = false;
    if (int e = try_launch_expand_g(a, stream, &done)) return e;
    if (done) return DARTREE_OK;
    auto run = [&](const ExpandArgs& x, cudaStream_t st) {
        return x.dtype == DARTREE_BF16 ? launch_expand_t<bf16_t>(x, st) : launch_expand_t<float>(x, st);
    };
    // A large batch runs as two halves of requests on two streams, so that one
    // half's projection GEMM (tensor cores, L2) overlaps the other half's
    // candidate-row contraction (HBM). Requests are independent; every
    // per-request buffer is indexed from the half's first request.
    std::unique_lock<std::recursive_mutex> lock(side_mutex());
    SideStreams* side = a.C >= kSplitMinC ? side_streams(stream) : nullptr;
    if (!side) return run(a, stream);
    const int c0 = a.C / 2, r0 = c0;
    const size_t eb = a.dtype == DARTREE_BF16 ? 2 : 4;
    ExpandArgs h0 = a, h1 = a;
    h0.fin = h1.fin = nullptr;  // the per-depth path leaves S8-S10 to the caller
    h0.split = h1.split = true;
    h0.C = c0;
    h1.C = a.C - c0;
    h1.hidden = static_cast<const uint8_t*>(a.hidden) + size_t(r0) * a.L * a.H * eb;
    h1.anchor = a.anchor + r0;
    h1.cand_tok = a.cand_tok + size_t(r0) * a.L * a.K;
    h1.cand_val = a.cand_val + size_t(r0) * a.L * a.K;
    h1.st_tok = a.st_tok + size_t(r0) * a.L * a.W;
    h1.st_par = a.st_par + size_t(r0) * a.L * a.W;
    h1.st_s = a.st_s + size_t(r0) * a.L * a.W;
    h1.st_n = a.st_n + size_t(r0) * a.L;
    for (int i = 0; i < 2; ++i) {
        h1.hbuf[i] = static_cast<uint8_t*>(a.hbuf[i]) + size_t(r0) * a.W * a.H * eb;
        h1.sbuf[i] = a.sbuf[i] + size_t(r0) * a.W;
    }
    h1.U = a.U + size_t(r0) * a.W * a.H;
    h1.z = a.z + size_t(r0) * a.W * a.K;
    if (a.uhl) h1.uhl = a.uhl + size_t(r0) * 32 * a.H;
    if (cudaEventRecord(side->fork[1], stream) != cudaSuccess ||
        cudaStreamWaitEvent(side->s[1], side->fork[1], 0) != cudaSuccess)
        return DARTREE_ECUDA;
    if (int e = run(h0, stream)) return e;
    if (int e = run(h1, side->s[1])) return e;
    if (cudaEventRecord(side->join[1], side->s[1]) != cudaSuccess || cudaStreamWaitEvent(stream, side->join[1], 0) != cudaSuccess)
        return DARTREE_ECUDA;
    return DARTREE_OK;
}

}  // namespace dartree
