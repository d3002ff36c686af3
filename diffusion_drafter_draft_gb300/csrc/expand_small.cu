// S2-S7 for small batches (C * W parents per depth fit in one CTA's shared
// memory): one persistent kernel runs all L depths (DARTree blog post, 3.1
// "Basic flow", depth-wise expansion; the whole tree is built with one batched
// correction per depth instead of one head call per node).
//
// Latency, not bandwidth, bounds this regime, so the design minimises grid-wide
// synchronisation: one grid barrier per depth.
//   * The grid is a set of 8-CTA clusters, one CTA per SM. CTA b owns a slice of
//     nf ~ H/G output features of W_q, kept in its shared memory when it fits.
//   * Phase B (per depth): U[:, slice] = h . W_q[slice]^T for all C*P parents
//     (bf16 mma.sync, fp32 accumulation; a 16 x nf tile per CTA is far below a
//     tcgen05 tile), then partial logits zp[m, c] = sum_{f in slice} U[m, f] *
//     E[cand_c, f]. The cluster sums its 8 partials through distributed shared
//     memory and writes one partial per cluster to global memory.
//   * Grid barrier.
//   * Phase A: each CTA sums 1/8 of the entries over the clusters (fixed order:
//     deterministic) and broadcasts them to its cluster peers; every CTA then
//     holds all logits and selects the top-W children of every request itself
//     (log-softmax, s = s_p + log q + beta, key (s desc, flat index asc)).
//   * State update: the cluster computes the new rows h = RMSNorm(h_p + E[tok] +
//     H_d[d-1]) (each CTA 1/8 of the rows) and writes each row into the shared
//     memory of all 8 peers; cluster 0 also keeps a copy in global memory, from
//     which the next depth reads parent rows.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace dartree {

constexpr int XS_NT = 512;
constexpr int XS_NW = XS_NT / 32;
constexpr int XS_CL = 8;        // CTAs per cluster
constexpr int XS_MAXC = 16;     // requests (one selection warp each at least)
constexpr int XS_MTMAX = 3;     // 16-row mma tiles: C*W <= 48
constexpr int XS_NTMAX = 4;     // 8-feature mma tiles: nf <= 32
constexpr int XS_ZSTAGE = 4096; // floats staged for the cross-cluster sum

__host__ __device__ constexpr size_t xs_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Row stride (elements) of the embedding slices: an odd number of 4-byte words,
// so 32 lanes reading 32 consecutive candidates hit 32 different banks.
__host__ __device__ constexpr int xs_es_stride(int nfp, int elem) {
    return ((nfp * elem / 4) % 2 == 1) ? nfp : nfp + 4 / elem;
}

struct XsLayout {
    size_t h, Ws, U, Es, ctok, zfull, zp, red, keys, sel_flat, sel_par, sel_tok, sel_s, sp, zstage, misc, mbar, total;
};

// rows: C*W, hp: padded row length (elements), nfp: padded features, zs: C*W*K,
// wq_rows: nonzero when W_q rows are kept in shared memory
__host__ __device__ inline XsLayout xs_layout(int rows, int hp, int elem, int nfp, int C, int K, int zs, int W,
                                              int wq_rows) {
    XsLayout l{};
    size_t o = 0;
    auto take = [&](size_t b) { size_t at = o; o = xs_up(o + b, 16); return at; };
    l.h = take(xs_up(size_t(rows), 16) * hp * elem);  // whole 16-row mma tiles
    l.Ws = take(size_t(wq_rows ? nfp : 0) * hp * elem); // whole 8-row mma tiles
    l.U = take(size_t(rows) * nfp * 4);
    l.Es = take(size_t(C) * K * xs_es_stride(nfp, elem) * elem);
    l.ctok = take(size_t(C) * K * 4);
    l.zfull = take(size_t(zs) * 4);
    l.zp = take(size_t(zs) * 4);
    l.red = take(size_t(XS_NW) * 16 * nfp * 4);
    l.keys = take(size_t(zs) * 8);
    l.sel_flat = take(size_t(C) * W * 4);
    l.sel_par = take(size_t(C) * W * 4);
    l.sel_tok = take(size_t(C) * W * 4);
    l.sel_s = take(size_t(C) * W * 4);
    l.sp = take(size_t(C) * W * 4);
    l.zstage = take(size_t(XS_ZSTAGE) * 4);
    l.misc = take(64 * 4);
    l.mbar = take(16);
    l.total = o;
    return l;
}

struct XsArgs {
    const void* E;
    const void* Wq;
    const void* hidden;
    const int32_t* anchor;
    const int32_t* cand_tok;
    const float* cand_val;
    int V, H, C, L, K, W;
    float beta, inv_sqrt_h;
    int32_t* st_tok;
    int32_t* st_par;
    float* st_s;
    int32_t* st_n;
    void* hglob[2];    // [C*W, H] storage type
    float* zpart;      // [Q, C*W*K]
    unsigned* bar;     // grid barrier counter, zero at launch
    int* status;
    int G, Q, hp, nfp, use_mma, wq_smem;
};

__device__ __forceinline__ void st_dsmem_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w) : "memory");
}
__device__ __forceinline__ void st_dsmem_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_u32(p)));
}

// bf16 tensor-core projection with MT 16-row tiles: U[m][f] = sum_j h[m][j] * W_q[f0+f][j].
// h rows (stride hp) are in shared memory; W_q rows are in shared memory (wsm,
// stride hp, nfp rows allocated) or read from global memory (wsm null, wg = row f0).
// Warps split the k dimension; partial tiles are summed in warp order (deterministic).
template <int MT>
__device__ void project_mma(const uint16_t* hb, int hp, int M, int H, const uint16_t* __restrict__ wg,
                            const uint16_t* wsm, int nf, int nfp, float* U, float* red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int nt = (nf + 7) / 8, ksteps = H / 16;
    float acc[MT][XS_NTMAX][4];
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int j = 0; j < XS_NTMAX; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;
    // ldmatrix row addresses: lane l feeds row (l % 8) of 8x8 matrix l / 8
    const int lm = lane >> 3, lr = lane & 7;
    constexpr int KB = MT == 1 ? 4 : 2;  // k-steps whose W_q fragments are in flight together
    for (int ks0 = wid; ks0 < ksteps; ks0 += KB * XS_NW) {
        uint32_t b[KB][XS_NTMAX][2];
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            const int k0 = (ks0 + kb * XS_NW) * 16;
            if (wsm) {
#pragma unroll
                for (int np = 0; np < XS_NTMAX / 2; ++np) {
                    if (k0 < H && 2 * np < nt) {
                        uint32_t r[4];
                        // matrices: (tile 2np, k lo), (2np, k hi), (2np+1, k lo), (2np+1, k hi). With an
                        // odd tile count the last pair's second tile is not allocated: its lanes
                        // address the last allocated row instead (values unused).
                        const int wrow = min((2 * np + (lm >> 1)) * 8 + lr, nfp - 1);
                        ldsm_x4(r, wsm + size_t(wrow) * hp + k0 + (lm & 1) * 8);
                        b[kb][2 * np][0] = r[0];
                        b[kb][2 * np][1] = r[1];
                        b[kb][2 * np + 1][0] = r[2];
                        b[kb][2 * np + 1][1] = r[3];
                    } else {
                        b[kb][2 * np][0] = b[kb][2 * np][1] = b[kb][2 * np + 1][0] = b[kb][2 * np + 1][1] = 0u;
                    }
                }
            } else {
#pragma unroll
                for (int ni = 0; ni < XS_NTMAX; ++ni) {
                    const int f = ni * 8 + g;
                    if (k0 < H && ni < nt && f < nf) {
                        const uint16_t* wr = wg + size_t(f) * H + k0 + 2 * t;
                        b[kb][ni][0] = __ldg(reinterpret_cast<const unsigned int*>(wr));
                        b[kb][ni][1] = __ldg(reinterpret_cast<const unsigned int*>(wr + 8));
                    } else {
                        b[kb][ni][0] = b[kb][ni][1] = 0u;
                    }
                }
            }
        }
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            const int k0 = (ks0 + kb * XS_NW) * 16;
            if (k0 >= H) break;
#pragma unroll
            for (int mi = 0; mi < MT; ++mi) {
                uint32_t a[4];
                // matrices: (rows lo, k lo), (rows hi, k lo), (rows lo, k hi), (rows hi, k hi);
                // rows up to 16*MT-1 are allocated (padded to whole tiles)
                ldsm_x4(a, hb + size_t(mi * 16 + (lm & 1) * 8 + lr) * hp + k0 + (lm >> 1) * 8);
#pragma unroll
                for (int ni = 0; ni < XS_NTMAX; ++ni)
                    if (ni < nt) mma_bf16_16816(acc[mi][ni], a, b[kb][ni]);
            }
        }
    }
#pragma unroll
    for (int mi = 0; mi < MT; ++mi) {
#pragma unroll
        for (int ni = 0; ni < XS_NTMAX; ++ni) {
            if (ni < nt) {
                float* rw = red + size_t(wid) * 16 * nfp;
                const int c = ni * 8 + 2 * t;
                rw[g * nfp + c] = acc[mi][ni][0];
                rw[g * nfp + c + 1] = acc[mi][ni][1];
                rw[(g + 8) * nfp + c] = acc[mi][ni][2];
                rw[(g + 8) * nfp + c + 1] = acc[mi][ni][3];
            }
        }
        __syncthreads();
        for (int e = threadIdx.x; e < 16 * nf; e += XS_NT) {
            const int rr = e / nf, f = e % nf, m = mi * 16 + rr;
            if (m < M) {
                float s = 0.f;
#pragma unroll
                for (int w = 0; w < XS_NW; ++w) s += red[size_t(w) * 16 * nfp + rr * nfp + f];
                U[size_t(m) * nfp + f] = s;
            }
        }
        __syncthreads();
    }
}

// U[m][f] = sum_j h[m][j] * W_q[f0 + f][j], m < M, f < nf (fp32, row stride nfp).
template <typename T>
__device__ void project_slice(const T* h, int hp, int M, int H, const T* __restrict__ Wq, const T* wsm, int f0,
                              int nf, int nfp, float* U, float* red, int use_mma) {
    if constexpr (sizeof(T) == 2) {
        if (use_mma) {
            const uint16_t* hb = reinterpret_cast<const uint16_t*>(h);
            const uint16_t* wg = reinterpret_cast<const uint16_t*>(Wq) + size_t(f0) * H;
            const uint16_t* ws = reinterpret_cast<const uint16_t*>(wsm);
            const int mt = (M + 15) / 16;
            if (mt == 1) project_mma<1>(hb, hp, M, H, wg, ws, nf, nfp, U, red);
            else if (mt == 2) project_mma<2>(hb, hp, M, H, wg, ws, nf, nfp, U, red);
            else project_mma<3>(hb, hp, M, H, wg, ws, nf, nfp, U, red);
            return;
        }
    }
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    (void)red;
    for (int e = wid; e < M * nf; e += XS_NW) {
        const int m = e / nf, f = e % nf;
        const T* hr = h + size_t(m) * hp;
        const T* wr = wsm ? wsm + size_t(f) * hp : Wq + size_t(f0 + f) * H;
        float s = 0.f;
        for (int j = lane; j < H; j += 32) s = fmaf(to_float(hr[j]), to_float(wr[j]), s);
        s = warp_sum(s);
        if (lane == 0) U[size_t(m) * nfp + f] = s;
    }
    __syncthreads();
}

// Warp-wide maximum of unique 64-bit keys: redux on the high word, then on the
// low word among the lanes holding that high word.
__device__ __forceinline__ uint64_t warp_max_key(uint64_t v) {
    const uint32_t hi = uint32_t(v >> 32), lo = uint32_t(v);
    const uint32_t mh = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t ml = __reduce_max_sync(0xffffffffu, hi == mh ? lo : 0u);
    return (uint64_t(mh) << 32) | ml;
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}

template <typename T>
__global__ void __launch_bounds__(XS_NT, 1) expand_small_kernel(XsArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int C = a.C, L = a.L, K = a.K, W = a.W, H = a.H, hp = a.hp, nfp = a.nfp;
    const int zs = C * W * K;
    const int G = a.G;
    const int b = blockIdx.x;
    const int base_nf = H / G, extra = H % G;
    const int nf = base_nf + (b < extra ? 1 : 0);
    const int f0 = b * base_nf + (b < extra ? b : extra);
    const XsLayout lay = xs_layout(C * W, hp, sizeof(T), nfp, C, K, zs, W, a.wq_smem);
    T* h = reinterpret_cast<T*>(smem + lay.h);
    T* Ws = a.wq_smem ? reinterpret_cast<T*>(smem + lay.Ws) : nullptr;
    float* U = reinterpret_cast<float*>(smem + lay.U);
    T* Es = reinterpret_cast<T*>(smem + lay.Es);
    int* ctok = reinterpret_cast<int*>(smem + lay.ctok);
    float* zfull = reinterpret_cast<float*>(smem + lay.zfull);
    float* zp = reinterpret_cast<float*>(smem + lay.zp);
    float* red = reinterpret_cast<float*>(smem + lay.red);
    uint64_t* keys = reinterpret_cast<uint64_t*>(smem + lay.keys);
    int* sel_flat = reinterpret_cast<int*>(smem + lay.sel_flat);
    int* sel_par = reinterpret_cast<int*>(smem + lay.sel_par);
    int* sel_tok = reinterpret_cast<int*>(smem + lay.sel_tok);
    float* sel_s = reinterpret_cast<float*>(smem + lay.sel_s);
    float* sp = reinterpret_cast<float*>(smem + lay.sp);
    float* zstage = reinterpret_cast<float*>(smem + lay.zstage);
    unsigned* misc = reinterpret_cast<unsigned*>(smem + lay.misc);
    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + lay.mbar);
    const int ess = xs_es_stride(nfp, sizeof(T));

    const uint32_t cr = cluster_ctarank();
    const int q = b / XS_CL;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const T* E = static_cast<const T*>(a.E);
    const T* Wq = static_cast<const T*>(a.Wq);
    const T* hid = static_cast<const T*>(a.hidden);
    T* hg[2] = {static_cast<T*>(a.hglob[0]), static_cast<T*>(a.hglob[1])};
    const int nes = C * K * nf;

    if (threadIdx.x == 0) misc[0] = 0;  // timed-out flag
    {
        const size_t hrows = xs_up(size_t(C) * W, 16);
        uint32_t* hz = reinterpret_cast<uint32_t*>(h);
        for (size_t i = threadIdx.x; i < hrows * hp * sizeof(T) / 4; i += XS_NT) hz[i] = 0u;
        if (Ws) {
            uint32_t* wz = reinterpret_cast<uint32_t*>(Ws + size_t(nf) * hp);
            for (size_t i = threadIdx.x; i < size_t(nfp - nf) * hp * sizeof(T) / 4; i += XS_NT) wz[i] = 0u;
        }
    }
    __syncthreads();
    // this CTA's W_q rows stay in shared memory for all depths
    bool w_loaded = true;
    if (Ws) {
        if (threadIdx.x == 0) { mbar_init(mbar, 1); fence_mbar_init(); }
        __syncthreads();
        if (threadIdx.x == 0) {
            const uint32_t rb = uint32_t(H) * sizeof(T);
            mbar_arrive_expect_tx(mbar, rb * uint32_t(nf));
            for (int f = 0; f < nf; ++f) bulk_g2s(Ws + size_t(f) * hp, Wq + size_t(f0 + f) * H, rb, mbar);
        }
    }
    // block hidden rows of every position: warm L2 (read once per depth by the state update)
    for (size_t o = size_t(b) * XS_NT + threadIdx.x; o * 128 < size_t(C) * L * H * sizeof(T); o += size_t(G) * XS_NT)
        prefetch_l2(reinterpret_cast<const uint8_t*>(hid) + o * 128);
    // root: h = E[anchor], s = 0
    for (int e = threadIdx.x; e < C * H; e += XS_NT) {
        const int r = e / H, j = e % H;
        const T v = E[size_t(a.anchor[r]) * H + j];
        h[size_t(r) * hp + j] = v;
        if (b == 0) hg[0][size_t(r) * H + j] = v;
    }
    for (int r = threadIdx.x; r < C; r += XS_NT) sp[r] = 0.f;
    // embedding slices and candidate tokens of position 0
    for (int e = threadIdx.x; e < nes; e += XS_NT) {
        const int rc = e / nf, f = e % nf, r = rc / K, c = rc % K;
        Es[size_t(rc) * ess + f] = E[size_t(a.cand_tok[(size_t(r) * L) * K + c]) * H + f0 + f];
    }
    for (int e = threadIdx.x; e < C * K; e += XS_NT) ctok[e] = a.cand_tok[(size_t(e / K) * L) * K + e % K];
    if (Ws) w_loaded = mbar_wait_bounded(mbar, 0, a.status);
    __syncthreads();

    int P = 1, M = C;
    unsigned epoch = 0;
    for (int d = 1; d <= L; ++d) {
        // ---------------- phase B: projection of this CTA's feature slice, partial logits
        // warm L2 with the embedding rows of this position's candidates (state update reads them)
        {
            const int lines_per_row = int((size_t(H) * sizeof(T) + 127) / 128);
            const int nlines = C * K * lines_per_row;
            for (int i = b * XS_NT + int(threadIdx.x); i < nlines; i += G * XS_NT) {
                const int rc = i / lines_per_row, ln = i % lines_per_row;
                prefetch_l2(reinterpret_cast<const uint8_t*>(E + size_t(ctok[rc]) * H) + size_t(ln) * 128);
            }
        }
        project_slice<T>(h, hp, M, H, Wq, Ws, f0, nf, nfp, U, red, a.use_mma);
        const int ne = M * K;
        for (int e = threadIdx.x; e < ne; e += XS_NT) {
            const int m = e / K, c = e % K, r = m / P;
            const float* u = U + size_t(m) * nfp;
            const T* es = Es + (size_t(r) * K + c) * ess;
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
            int f = 0;
            for (; f + 4 <= nf; f += 4) {
                s0 = fmaf(u[f], to_float(es[f]), s0);
                s1 = fmaf(u[f + 1], to_float(es[f + 1]), s1);
                s2 = fmaf(u[f + 2], to_float(es[f + 2]), s2);
                s3 = fmaf(u[f + 3], to_float(es[f + 3]), s3);
            }
            for (; f < nf; ++f) s0 = fmaf(u[f], to_float(es[f]), s0);
            zp[e] = (s0 + s1) + (s2 + s3);
        }
        cluster_sync();
        {
            const int share = (ne + XS_CL - 1) / XS_CL;
            const int e0 = int(cr) * share, e1 = min(ne, e0 + share);
            for (int e = e0 + threadIdx.x; e < e1; e += XS_NT) {
                float v[XS_CL];
#pragma unroll
                for (int x = 0; x < XS_CL; ++x) v[x] = ld_dsmem_f32(dsmem_addr(&zp[e], uint32_t(x)));
                float s = 0.f;
#pragma unroll
                for (int x = 0; x < XS_CL; ++x) s += v[x];
                a.zpart[size_t(q) * zs + e] = s;
            }
        }
        ++epoch;
        grid_barrier(a.bar, epoch * unsigned(G), a.status, &misc[0]);

        // ---------------- phase A
        // next position's embedding slices: loads in flight during this phase
        T epre[4];
        const bool more = d < L;
        if (more) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int e = threadIdx.x + i * XS_NT;
                if (e < nes) {
                    const int rc = e / nf, f = e % nf, r = rc / K, c = rc % K;
                    epre[i] = E[size_t(a.cand_tok[(size_t(r) * L + d) * K + c]) * H + f0 + f];
                }
            }
        }
        {
            const int share = (ne + XS_CL - 1) / XS_CL;
            const int e0 = int(cr) * share, e1 = min(ne, e0 + share), cnt = max(0, e1 - e0);
            // stage all clusters' partials of this CTA's share (one round of loads)
            const bool staged = cnt * a.Q <= XS_ZSTAGE;
            if (staged) {
                for (int i = threadIdx.x; i < cnt * a.Q; i += XS_NT) {
                    const int qq = i / cnt, e = e0 + i % cnt;
                    zstage[i] = __ldcg(a.zpart + size_t(qq) * zs + e);
                }
                __syncthreads();
            }
            for (int e = e0 + threadIdx.x; e < e1; e += XS_NT) {
                float s = 0.f;
                if (staged) {
                    for (int qq = 0; qq < a.Q; ++qq) s += zstage[qq * cnt + (e - e0)];
                } else {
                    for (int qq = 0; qq < a.Q; ++qq) s += __ldcg(a.zpart + size_t(qq) * zs + e);
                }
                const int m = e / K, c = e % K, r = m / P;
                const float z = a.cand_val[(size_t(r) * L + (d - 1)) * K + c] + s * a.inv_sqrt_h;
                for (uint32_t x = 0; x < XS_CL; ++x) st_dsmem_f32(dsmem_addr(&zfull[e], x), z);
            }
        }
        cluster_sync();
        const int n = P * K;
        const int n_keep = min(W, n);
        // log-softmax per parent, then keys (s desc, flat index p*K + c asc)
        for (int m = wid; m < M; m += XS_NW) {
            const float* zr = zfull + size_t(m) * K;
            float mx = -INFINITY;
            for (int c = lane; c < K; c += 32) mx = fmaxf(mx, zr[c]);
            mx = warp_max(mx);
            float se = 0.f;
            for (int c = lane; c < K; c += 32) se += expf(zr[c] - mx);
            se = warp_sum(se);
            const float lse = mx + logf(se);
            const float spm = sp[m];
            const int r = m / P, p = m % P;
            for (int c = lane; c < K; c += 32) {
                float s = (spm + (zr[c] - lse)) + a.beta;
                s += 0.f;
                const uint32_t f = uint32_t(p * K + c);
                keys[size_t(r) * n + f] = (uint64_t(ord_f32(s)) << 32) | (0xffffffffu - f);
            }
        }
        __syncthreads();
        // top-W per request in two levels: each of the request's warps keeps the best
        // n_keep keys of a slice of its children (rounds of "largest key below the
        // previous one"), then one warp merges those lists.
        {
            const int wpr = max(1, XS_NW / C);  // warps per request
            uint64_t* cands = reinterpret_cast<uint64_t*>(red);  // [C][wpr][n_keep]
            const int r = wid / wpr, part = wid % wpr;
            if (r < C) {
                const uint64_t* kr = keys + size_t(r) * n;
                const int per = (n + wpr - 1) / wpr;
                const int lo = part * per, hi = min(n, lo + per);
                // up to 4 keys per lane stay in registers; longer slices loop over shared memory
                uint64_t kv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) kv[i] = (lo + lane + 32 * i < hi) ? kr[lo + lane + 32 * i] : 0ull;
                const bool inreg = hi - lo <= 128;
                uint64_t prev = ~0ull;
                for (int k = 0; k < n_keep; ++k) {
                    uint64_t best = 0;
                    if (inreg) {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (kv[i] < prev && kv[i] > best) best = kv[i];
                    } else {
                        for (int f = lo + lane; f < hi; f += 32) {
                            const uint64_t v = kr[f];
                            if (v < prev && v > best) best = v;
                        }
                    }
                    best = warp_max_key(best);
                    prev = best;
                    if (lane == 0) cands[(size_t(r) * wpr + part) * n_keep + k] = best;
                }
            }
            __syncthreads();
            if (part == 0 && r < C) {
                const uint64_t* cr_ = cands + size_t(r) * wpr * n_keep;
                const int m = wpr * n_keep;
                uint64_t kv[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) kv[i] = (lane + 32 * i < m) ? cr_[lane + 32 * i] : 0ull;
                const bool inreg = m <= 256;
                uint64_t prev = ~0ull;
                for (int k = 0; k < n_keep; ++k) {
                    uint64_t best = 0;
                    if (inreg) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            if (kv[i] < prev && kv[i] > best) best = kv[i];
                    } else {
                        for (int f = lane; f < m; f += 32) {
                            const uint64_t v = cr_[f];
                            if (v < prev && v > best) best = v;
                        }
                    }
                    best = warp_max_key(best);
                    prev = best;
                    if (lane == 0) {
                        sel_flat[r * W + k] = int(0xffffffffu - uint32_t(best));
                        sel_s[r * W + k] = f32_from_ord(uint32_t(best >> 32));
                    }
                }
            }
        }
        __syncthreads();
        for (int e = threadIdx.x; e < C * n_keep; e += XS_NT) {
            const int r = e / n_keep, k = e % n_keep;
            const int f = sel_flat[r * W + k];
            sel_par[r * W + k] = f / K;
            sel_tok[r * W + k] = ctok[r * K + f % K];
        }
        __syncthreads();
        if (b == 0) {
            for (int e = threadIdx.x; e < C * W; e += XS_NT) {
                const int r = e / W, k = e % W;
                const size_t o = (size_t(r) * L + (d - 1)) * W + k;
                a.st_tok[o] = k < n_keep ? sel_tok[e] : -1;
                a.st_par[o] = k < n_keep ? sel_par[e] : -1;
                a.st_s[o] = k < n_keep ? sel_s[e] : 0.f;
            }
            for (int r = threadIdx.x; r < C; r += XS_NT) a.st_n[size_t(r) * L + (d - 1)] = n_keep;
        }
        if (!more) break;

        // ---------------- state update: this CTA's new rows (qrow = cr, cr+8, ...) in
        // parallel, one thread group per row; each row goes to all 8 peers
        const int Mn = C * n_keep;
        const T* hold = hg[(d - 1) & 1];
        T* hnew = hg[d & 1];
        {
            constexpr int VE = 16 / sizeof(T);
            const int nv = H / VE;
            const int nrow = Mn > int(cr) ? (Mn - int(cr) + XS_CL - 1) / XS_CL : 0;  // rows of this CTA
            const int wpg = nrow > 0 ? max(1, XS_NW / nrow) : XS_NW;                   // warps per row
            const int grp = wid / wpg, gl = threadIdx.x - grp * wpg * 32, gsz = wpg * 32;
            const bool mine = grp < nrow;
            int qrow = 0;
            const T *ho = nullptr, *er = nullptr, *hd = nullptr;
            constexpr int VR = 2;  // vectors per thread held in registers
            float xr[VR][VE];
            float ss = 0.f;
            if (mine) {
                qrow = int(cr) + grp * XS_CL;
                const int r = qrow / n_keep, k = qrow % n_keep;
                const int par = sel_par[r * W + k], tok = sel_tok[r * W + k];
                ho = hold + (size_t(r) * P + par) * H;
                er = E + size_t(tok) * H;
                hd = hid + (size_t(r) * L + (d - 1)) * H;
                uint4 vo[VR], ve[VR], vh[VR];
#pragma unroll
                for (int i = 0; i < VR; ++i) {
                    const int v = gl + i * gsz;
                    if (v < nv) {
                        vo[i] = __ldcg(reinterpret_cast<const uint4*>(ho) + v);  // written this launch
                        ve[i] = reinterpret_cast<const uint4*>(er)[v];
                        vh[i] = reinterpret_cast<const uint4*>(hd)[v];
                    }
                }
#pragma unroll
                for (int i = 0; i < VR; ++i) {
                    const int v = gl + i * gsz;
                    if (v < nv) {
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
                for (int v = gl + VR * gsz; v < nv; v += gsz) {  // rows wider than the registers
                    const uint4 wo = __ldcg(reinterpret_cast<const uint4*>(ho) + v);
                    const uint4 we = reinterpret_cast<const uint4*>(er)[v];
                    const uint4 wh = reinterpret_cast<const uint4*>(hd)[v];
                    const T* po = reinterpret_cast<const T*>(&wo);
                    const T* pe = reinterpret_cast<const T*>(&we);
                    const T* ph = reinterpret_cast<const T*>(&wh);
                    for (int j = 0; j < VE; ++j) {
                        const float y = (to_float(po[j]) + to_float(pe[j])) + to_float(ph[j]);
                        ss = fmaf(y, y, ss);
                    }
                }
            }
            ss = warp_sum(ss);
            float* rowred = red;
            if (lane == 0) rowred[wid] = ss;
            __syncthreads();
            if (mine) {
                float tot = 0.f;
                for (int w = grp * wpg; w < (grp + 1) * wpg; ++w) tot += rowred[w];
                const float rs = sqrtf(tot / float(H) + 1e-6f);
                uint4* hrow = reinterpret_cast<uint4*>(h + size_t(qrow) * hp);
                auto emit = [&](int v, const float* x) {
                    uint4 out;
                    T* pw = reinterpret_cast<T*>(&out);
#pragma unroll
                    for (int j = 0; j < VE; ++j) pw[j] = from_float<T>(x[j] / rs);
#pragma unroll
                    for (int xx = 0; xx < XS_CL; ++xx) st_dsmem_v4(dsmem_addr(hrow + v, uint32_t(xx)), out);
                    if (q == 0) reinterpret_cast<uint4*>(hnew + size_t(qrow) * H)[v] = out;
                };
#pragma unroll
                for (int i = 0; i < VR; ++i) {
                    const int v = gl + i * gsz;
                    if (v < nv) emit(v, xr[i]);
                }
                for (int v = gl + VR * gsz; v < nv; v += gsz) {
                    const uint4 wo = __ldcg(reinterpret_cast<const uint4*>(ho) + v);
                    const uint4 we = reinterpret_cast<const uint4*>(er)[v];
                    const uint4 wh = reinterpret_cast<const uint4*>(hd)[v];
                    const T* po = reinterpret_cast<const T*>(&wo);
                    const T* pe = reinterpret_cast<const T*>(&we);
                    const T* ph = reinterpret_cast<const T*>(&wh);
                    float x[VE];
                    for (int j = 0; j < VE; ++j) x[j] = (to_float(po[j]) + to_float(pe[j])) + to_float(ph[j]);
                    emit(v, x);
                }
            }
        }
        // next position's slices and tokens (the loads were issued at the top of phase A)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = threadIdx.x + i * XS_NT;
            if (e < nes) Es[size_t(e / nf) * ess + e % nf] = epre[i];
        }
        for (int e = threadIdx.x + 4 * XS_NT; e < nes; e += XS_NT) {
            const int rc = e / nf, f = e % nf, r = rc / K, c = rc % K;
            Es[size_t(rc) * ess + f] = E[size_t(a.cand_tok[(size_t(r) * L + d) * K + c]) * H + f0 + f];
        }
        for (int e = threadIdx.x; e < C * K; e += XS_NT) ctok[e] = a.cand_tok[(size_t(e / K) * L + d) * K + e % K];
        for (int e = threadIdx.x; e < Mn; e += XS_NT) sp[e] = sel_s[(e / n_keep) * W + e % n_keep];
        cluster_sync();  // every peer's rows have landed
        P = n_keep;
        M = Mn;
    }
    if (Ws && !w_loaded && threadIdx.x == 0) mbar_wait_bounded(mbar, 0, nullptr);
    cluster_sync();  // no CTA leaves while a peer may still address its shared memory
}

// --------------------------------------------------------------------------- host

constexpr size_t kSmemBudget = 227 * 1024;

struct XsPlan {
    int G = 0, Q = 0, hp = 0, nfp = 0, use_mma = 0, wq_smem = 0;
    size_t smem = 0;
};

template <typename T>
static bool xs_plan(const ExpandArgs& a, XsPlan& pl) {
    if (a.C > XS_MAXC || a.C * a.W > XS_MTMAX * 16 || a.H % 8 != 0) return false;
    const int elem = sizeof(T);
    pl.hp = a.H + 16 / elem;  // one 16-byte pad per row: conflict-free fragment loads
    pl.use_mma = (elem == 2 && a.H % 16 == 0) ? 1 : 0;
    int max_clusters = 0;
    auto kern = expand_small_kernel<T>;
    // size with the largest plausible grid first, then refine nf for the real grid
    for (int pass = 0; pass < 2; ++pass) {
        const int G = pass == 0 ? num_sms() : pl.G;
        const int nfmax = (a.H + G - 1) / G;
        pl.nfp = int(xs_up(nfmax, 8));
        if (pl.nfp > XS_NTMAX * 8) return false;
        XsLayout l = xs_layout(a.C * a.W, pl.hp, elem, pl.nfp, a.C, a.K, a.C * a.W * a.K, a.W, 1);
        pl.wq_smem = l.total <= kSmemBudget ? 1 : 0;
        if (!pl.wq_smem) l = xs_layout(a.C * a.W, pl.hp, elem, pl.nfp, a.C, a.K, a.C * a.W * a.K, a.W, 0);
        pl.smem = l.total;
        if (pl.smem > kSmemBudget) return false;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(pl.smem)) != cudaSuccess)
            return false;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) return false;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(XS_CL);
        cfg.blockDim = dim3(XS_NT);
        cfg.dynamicSmemBytes = pl.smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = XS_CL;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg) != cudaSuccess || max_clusters < 1) {
            cudaGetLastError();
            return false;
        }
        const int Gr = max_clusters * XS_CL;
        if (pass == 1 && Gr != pl.G) return false;
        pl.G = Gr;
        pl.Q = max_clusters;
        if (a.H < pl.G) return false;
    }
    return true;
}

template <typename T>
static int launch_small_t(const ExpandArgs& a, const XsPlan& pl, cudaStream_t st) {
    XsArgs x{};
    x.E = a.E;
    x.Wq = a.Wq;
    x.hidden = a.hidden;
    x.anchor = a.anchor;
    x.cand_tok = a.cand_tok;
    x.cand_val = a.cand_val;
    x.V = a.V;
    x.H = a.H;
    x.C = a.C;
    x.L = a.L;
    x.K = a.K;
    x.W = a.W;
    x.beta = a.beta;
    x.inv_sqrt_h = 1.0f / sqrtf(float(a.H));
    x.st_tok = a.st_tok;
    x.st_par = a.st_par;
    x.st_s = a.st_s;
    x.st_n = a.st_n;
    x.hglob[0] = a.hbuf[0];
    x.hglob[1] = a.hbuf[1];
    x.zpart = a.zpart;
    x.bar = a.bar;
    x.status = a.status;
    x.G = pl.G;
    x.Q = pl.Q;
    x.hp = pl.hp;
    x.nfp = pl.nfp;
    x.use_mma = pl.use_mma;
    x.wq_smem = pl.wq_smem;
    if (cudaMemsetAsync(a.bar, 0, sizeof(unsigned), st) != cudaSuccess) return DARTREE_ECUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(pl.G);
    cfg.blockDim = dim3(XS_NT);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = XS_CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    KTimer kt_(KID_EXPAND_SMALL, st);
    return cudaLaunchKernelEx(&cfg, expand_small_kernel<T>, x) == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

int try_launch_expand_small(const ExpandArgs& a, cudaStream_t stream, bool* launched) {
    *launched = false;
    if (!a.zpart || !a.bar) return DARTREE_OK;
    XsPlan pl;
    if (a.dtype == DARTREE_BF16) {
        if (!xs_plan<bf16_t>(a, pl) || pl.Q > a.zpart_clusters) return DARTREE_OK;
        *launched = true;
        return launch_small_t<bf16_t>(a, pl, stream);
    }
    if (!xs_plan<float>(a, pl) || pl.Q > a.zpart_clusters) return DARTREE_OK;
    *launched = true;
    return launch_small_t<float>(a, pl, stream);
}

}  // namespace dartree
