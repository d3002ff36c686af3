// S2-S7 for small batches with a prepared bf16 head: candidate-side projection.
//
// The stand-in head's corrected logit is bilinear in the parent state and the
// candidate embedding (DARTree blog post, 3.1, depth-wise expansion):
//
//   z[p, c] = L^base[d-1, c] + <W_q h_p, E[c]> / sqrt(H) = L^base[d-1, c] + <h_p, G_c> / sqrt(H),
//   G_c = W_q^T E[c]   (G[c, j] = sum_i E[c, i] W_q[i, j]).
//
// The candidates of every position are known after S1, so G for all C*L*K of
// them is one tcgen05 GEMM per round (gathered E rows x W_q, using the head's
// prepared W_q^T as the K-major operand), stored as a bf16 pair G = G_hi + G_lo.
// Each depth then contracts the P parents with the K candidates of its position
// in one batch: z = h . G_hi^T + h . G_lo^T (mma.sync, fp32 accumulation), with
// no dependence on W_q, so one thread-block cluster per request runs all L
// depths: CTA q of the cluster owns H/CS features of h and G, the partial logits
// are summed through distributed shared memory, every CTA selects the same top-W
// children, and each CTA normalises its own feature slice of the new states
// (the RMSNorm sum of squares is all-reduced across the cluster). Nothing leaves
// the cluster between depths.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace dartree {

constexpr int XG_NT = 256;
constexpr int XG_NW = XG_NT / 32;
constexpr int XG_MAXK = 64;   // candidates per position (one 8-candidate mma tile per warp)
constexpr int XG_MAXW = 16;   // parents per depth (one 16-row mma tile)
constexpr int XG_MAXCAND = 8192;

__host__ __device__ constexpr size_t xg_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct XgLayout {
    size_t hs, gs, es, hds, zp, zfull, keys, ssp, sel, cands, misc, total;
};

// fs: features per CTA, fp = fs + 8 (padded row), cs: cluster size
__host__ __device__ inline XgLayout xg_layout(int fs, int K, int cs) {
    const int fp = fs + 8;
    XgLayout l{};
    size_t o = 0;
    auto take = [&](size_t b) { size_t at = o; o = xg_up(o + b, 16); return at; };
    l.hs = take(size_t(2) * XG_MAXW * fp * 2);   // h slices, current and next
    l.gs = take(size_t(2) * K * fp * 2);         // G_hi, G_lo slices of one position
    l.es = take(size_t(K) * fs * 2);             // E slices of one position
    l.hds = take(size_t(fs) * 2);                // H_d slice of one position
    l.zp = take(size_t(XG_MAXW) * K * 4);
    l.zfull = take(size_t(XG_MAXW) * K * 4);
    l.keys = take(size_t(XG_MAXW) * K * 8);
    l.ssp = take(size_t(cs) * XG_MAXW * 4);
    l.sel = take(size_t(XG_MAXW) * 16);
    l.cands = take(size_t(XG_NW) * XG_MAXW * 8);
    l.misc = take(64 * 4);
    l.total = o;
    return l;
}

struct XgArgs {
    const uint16_t* E;
    const uint16_t* hidden;
    const int32_t* anchor;
    const int32_t* cand_tok;
    const float* cand_val;
    const uint16_t* Ghi;
    const uint16_t* Glo;
    int H, L, K, W, cs;
    float beta, inv_sqrt_h;
    int32_t* st_tok;
    int32_t* st_par;
    float* st_s;
    int32_t* st_n;
    int* status;
};

__device__ __forceinline__ void xg_cp16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void xg_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void xg_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void xg_ldsm_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_u32(p)));
}
__device__ __forceinline__ void xg_mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void st_dsmem_f32x(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_dsmem_f32x(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// G_hi/G_lo slices of position pos, by cp.async (one group).
__device__ __forceinline__ void xg_load_g(const XgArgs& a, int r, int pos, int f0, int fs, uint16_t* gs) {
    const int fp = fs + 8, K = a.K, H = a.H;
    const int cpr = fs / 8;  // 16-byte chunks per slice row
    const size_t crow = (size_t(r) * a.L + pos) * K;
    for (int i = threadIdx.x; i < 2 * K * cpr; i += XG_NT) {
        const int hl = i / (K * cpr), c = (i / cpr) % K, j = i % cpr;
        const uint16_t* src = (hl ? a.Glo : a.Ghi) + (crow + c) * H + f0 + j * 8;
        xg_cp16(gs + (size_t(hl) * K + c) * fp + j * 8, src);
    }
    xg_commit();
}

// E slices of the candidates of position pos and the H_d slice of pos (one group).
__device__ __forceinline__ void xg_load_e(const XgArgs& a, int r, int pos, int f0, int fs, uint16_t* es,
                                          uint16_t* hds) {
    const int K = a.K, H = a.H;
    const int cpr = fs / 8;
    const size_t crow = (size_t(r) * a.L + pos) * K;
    for (int i = threadIdx.x; i < K * cpr; i += XG_NT) {
        const int c = i / cpr, j = i % cpr;
        xg_cp16(es + size_t(c) * fs + j * 8, a.E + size_t(a.cand_tok[crow + c]) * H + f0 + j * 8);
    }
    for (int j = threadIdx.x; j < cpr; j += XG_NT)
        xg_cp16(hds + j * 8, a.hidden + (size_t(r) * a.L + pos) * H + f0 + j * 8);
    xg_commit();
}

__global__ void __launch_bounds__(XG_NT, 1) expand_g_kernel(XgArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int CS = a.cs, H = a.H, L = a.L, K = a.K, W = a.W;
    const int fs = H / CS, fp = fs + 8;
    const XgLayout lay = xg_layout(fs, K, CS);
    uint16_t* hs = reinterpret_cast<uint16_t*>(smem + lay.hs);
    uint16_t* gs = reinterpret_cast<uint16_t*>(smem + lay.gs);
    uint16_t* es = reinterpret_cast<uint16_t*>(smem + lay.es);
    uint16_t* hds = reinterpret_cast<uint16_t*>(smem + lay.hds);
    float* zp = reinterpret_cast<float*>(smem + lay.zp);
    float* zfull = reinterpret_cast<float*>(smem + lay.zfull);
    uint64_t* keys = reinterpret_cast<uint64_t*>(smem + lay.keys);
    float* ssp = reinterpret_cast<float*>(smem + lay.ssp);
    uint64_t* selk = reinterpret_cast<uint64_t*>(smem + lay.sel);   // kept keys, descending
    int* selx = reinterpret_cast<int*>(selk + XG_MAXW);             // [0..W): parent rank, [W..2W): candidate
    uint64_t* cands = reinterpret_cast<uint64_t*>(smem + lay.cands);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + lay.misc);
    float* spar = reinterpret_cast<float*>(misc + 32);              // parent scores (<= 16)

    const uint32_t cr = cluster_ctarank();
    const int r = blockIdx.x / CS;
    const int f0 = int(cr) * fs;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;

    // root: h = E[anchor] (this CTA's slice), s = 0; rows 1..15 zero
    for (int i = threadIdx.x; i < 2 * XG_MAXW * fp; i += XG_NT) hs[i] = 0;
    __syncthreads();
    for (int f = threadIdx.x; f < fs; f += XG_NT) hs[f] = a.E[size_t(a.anchor[r]) * H + f0 + f];
    if (threadIdx.x < XG_MAXW) spar[threadIdx.x] = 0.f;
    xg_load_g(a, r, 0, f0, fs, gs);
    xg_load_e(a, r, 0, f0, fs, es, hds);
    int cur = 0, P = 1;

    for (int d = 1; d <= L; ++d) {
        const int pos = d - 1;
        xg_wait_all();
        __syncthreads();
        // ---- partial logits over this CTA's features: zp[p][c] = h_p . (G_hi + G_lo)_c
        {
            const uint16_t* hb = hs + size_t(cur) * XG_MAXW * fp;
            const int lm = lane >> 3, lr = lane & 7, g = lane >> 2, t = lane & 3;
            for (int ct = wid; ct * 8 < K; ct += XG_NW) {  // 8 candidates per tile
                float acc_hi[4] = {0.f, 0.f, 0.f, 0.f}, acc_lo[4] = {0.f, 0.f, 0.f, 0.f};
                for (int k0 = 0; k0 < fs; k0 += 16) {
                    uint32_t af[4], bf[4];
                    xg_ldsm_x4(af, hb + size_t((lm & 1) * 8 + lr) * fp + k0 + (lm >> 1) * 8);
                    // matrices: (hi, k lo), (hi, k hi), (lo, k lo), (lo, k hi)
                    xg_ldsm_x4(bf, gs + (size_t(lm >> 1) * K + ct * 8 + lr) * fp + k0 + (lm & 1) * 8);
                    xg_mma(acc_hi, af, bf[0], bf[1]);
                    xg_mma(acc_lo, af, bf[2], bf[3]);
                }
                const int c = ct * 8 + 2 * t;
                if (g < P) {
                    zp[g * K + c] = acc_hi[0] + acc_lo[0];
                    zp[g * K + c + 1] = acc_hi[1] + acc_lo[1];
                }
                if (g + 8 < P) {
                    zp[(g + 8) * K + c] = acc_hi[2] + acc_lo[2];
                    zp[(g + 8) * K + c + 1] = acc_hi[3] + acc_lo[3];
                }
            }
        }
        __syncthreads();
        if (d < L) xg_load_g(a, r, pos + 1, f0, fs, gs);  // this depth is done with gs
        cluster_sync();
        // ---- cluster sum of this CTA's share of the entries, broadcast to every peer
        const int ne = P * K;
        {
            const int share = (ne + CS - 1) / CS;
            const int e0 = int(cr) * share, e1 = min(ne, e0 + share);
            for (int e = e0 + threadIdx.x; e < e1; e += XG_NT) {
                float s = 0.f;
                for (int q = 0; q < CS; ++q) s += ld_dsmem_f32x(dsmem_addr(&zp[e], uint32_t(q)));
                const float z = a.cand_val[(size_t(r) * L + pos) * K + e % K] + s * a.inv_sqrt_h;
                for (int q = 0; q < CS; ++q) st_dsmem_f32x(dsmem_addr(&zfull[e], uint32_t(q)), z);
            }
        }
        cluster_sync();
        // ---- log-softmax, scores, top-W (identical in every CTA)
        for (int p = wid; p < P; p += XG_NW) {
            const float* zr = zfull + p * K;
            float mx = -INFINITY;
            for (int c = lane; c < K; c += 32) mx = fmaxf(mx, zr[c]);
            mx = warp_max(mx);
            float se = 0.f;
            for (int c = lane; c < K; c += 32) se += expf(zr[c] - mx);
            se = warp_sum(se);
            const float lse = mx + logf(se);
            for (int c = lane; c < K; c += 32) {
                float s = (spar[p] + (zr[c] - lse)) + a.beta;
                s += 0.f;
                const uint32_t f = uint32_t(p * K + c);
                keys[f] = (uint64_t(ord_f32(s)) << 32) | (0xffffffffu - f);
            }
        }
        __syncthreads();
        const int n_keep = min(W, ne);
        block_top_keys<XG_NT>(keys, ne, n_keep, cands, selk);
        if (threadIdx.x < n_keep) {
            const uint32_t f = 0xffffffffu - uint32_t(selk[threadIdx.x]);
            selx[threadIdx.x] = int(f) / K;
            selx[XG_MAXW + threadIdx.x] = int(f) % K;
        }
        __syncthreads();
        if (cr == 0) {
            for (int k = threadIdx.x; k < W; k += XG_NT) {
                const size_t o = (size_t(r) * L + pos) * W + k;
                if (k < n_keep) {
                    a.st_tok[o] = a.cand_tok[(size_t(r) * L + pos) * K + selx[XG_MAXW + k]];
                    a.st_par[o] = selx[k];
                    a.st_s[o] = f32_from_ord(uint32_t(selk[k] >> 32));
                } else {
                    a.st_tok[o] = -1;
                    a.st_par[o] = -1;
                    a.st_s[o] = 0.f;
                }
            }
            if (threadIdx.x == 0) a.st_n[size_t(r) * L + pos] = n_keep;
        }
        if (d == L) break;
        // ---- state update of this CTA's feature slice; the RMSNorm sum of squares
        // is all-reduced over the cluster
        const uint16_t* hb = hs + size_t(cur) * XG_MAXW * fp;
        uint16_t* hn = hs + size_t(1 - cur) * XG_MAXW * fp;
        for (int k = wid; k < n_keep; k += XG_NW) {
            const uint16_t* hp = hb + size_t(selx[k]) * fp;
            const uint16_t* er = es + size_t(selx[XG_MAXW + k]) * fs;
            float ss = 0.f;
            for (int f = lane; f < fs; f += 32) {
                const float x = (bf16_bits_to_float(hp[f]) + bf16_bits_to_float(er[f])) + bf16_bits_to_float(hds[f]);
                ss = fmaf(x, x, ss);
            }
            ss = warp_sum(ss);
            if (lane < CS) st_dsmem_f32x(dsmem_addr(&ssp[int(cr) * XG_MAXW + k], uint32_t(lane)), ss);
        }
        cluster_sync();
        for (int k = wid; k < n_keep; k += XG_NW) {
            float tot = 0.f;
            for (int q = 0; q < CS; ++q) tot += ssp[q * XG_MAXW + k];
            const float rs = sqrtf(tot / float(H) + 1e-6f);
            const uint16_t* hp = hb + size_t(selx[k]) * fp;
            const uint16_t* er = es + size_t(selx[XG_MAXW + k]) * fs;
            for (int f = lane; f < fs; f += 32) {
                const float x = (bf16_bits_to_float(hp[f]) + bf16_bits_to_float(er[f])) + bf16_bits_to_float(hds[f]);
                hn[size_t(k) * fp + f] = __bfloat16_as_ushort(__float2bfloat16_rn(x / rs));
            }
        }
        for (int i = threadIdx.x; i < (XG_MAXW - n_keep) * fs; i += XG_NT)  // unused rows stay zero
            hn[size_t(n_keep + i / fs) * fp + i % fs] = 0;
        if (threadIdx.x < n_keep) spar[threadIdx.x] = f32_from_ord(uint32_t(selk[threadIdx.x] >> 32));
        __syncthreads();
        xg_load_e(a, r, pos + 1, f0, fs, es, hds);  // this depth is done with es, hds
        cur = 1 - cur;
        P = n_keep;
    }
    xg_wait_all();
    cluster_sync();  // no CTA leaves while a peer may still address its shared memory
}

// --------------------------------------------------------------------------- gathers, transpose

__global__ void gather_rows_kernel(const uint16_t* __restrict__ E, const int32_t* __restrict__ idx, int H,
                                   uint16_t* __restrict__ out) {
    const int m = blockIdx.x;
    const uint4* src = reinterpret_cast<const uint4*>(E + size_t(idx[m]) * H);
    uint4* dst = reinterpret_cast<uint4*>(out + size_t(m) * H);
    for (int v = threadIdx.x; v < H / 8; v += blockDim.x) dst[v] = src[v];
}

__global__ void transpose_bf16_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst, int H) {
    __shared__ uint16_t tile[32][33];
    const int x0 = blockIdx.x * 32, y0 = blockIdx.y * 32;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int y = y0 + i, x = x0 + threadIdx.x;
        if (y < H && x < H) tile[i][threadIdx.x] = src[size_t(y) * H + x];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int y = x0 + i, x = y0 + threadIdx.x;
        if (y < H && x < H) dst[size_t(y) * H + x] = tile[threadIdx.x][i];
    }
}

int launch_transpose_bf16(const void* src, void* dst, int H, cudaStream_t stream) {
    dim3 grid((H + 31) / 32, (H + 31) / 32), block(32, 8);
    transpose_bf16_kernel<<<grid, block, 0, stream>>>(static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst), H);
    return cudaGetLastError() == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

// --------------------------------------------------------------------------- host

static bool xg_cluster_ok(int cs, size_t smem) {
    auto kern = expand_g_kernel;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    cudaLaunchConfig_t q{};
    q.gridDim = dim3(unsigned(cs));
    q.blockDim = dim3(XG_NT);
    q.dynamicSmemBytes = smem;
    cudaLaunchAttribute qa[1];
    qa[0].id = cudaLaunchAttributeClusterDimension;
    qa[0].val.clusterDim.x = cs;
    qa[0].val.clusterDim.y = 1;
    qa[0].val.clusterDim.z = 1;
    q.attrs = qa;
    q.numAttrs = 1;
    int nc = 0;
    if (cudaOccupancyMaxActiveClusters(&nc, kern, &q) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return nc >= 1;
}

int try_launch_expand_g(const ExpandArgs& a, cudaStream_t stream, bool* launched) {
    *launched = false;
    if (a.dtype != DARTREE_BF16 || !a.WqT || !a.Eg || !a.Ghi || !a.Glo) return DARTREE_OK;
    const int M = a.C * a.L * a.K;
    if (M > a.g_rows || a.K > XG_MAXK || a.K % 8 != 0 || a.W > XG_MAXW) return DARTREE_OK;
    if (!gemm_tc_supported(M, a.H, a.H)) return DARTREE_OK;
    int cs = 0;
    size_t smem = 0;
    for (int c : {16, 8}) {
        if (a.H % (c * 16) != 0) continue;
        const size_t sm = xg_layout(a.H / c, a.K, c).total;
        if (sm <= 227 * 1024 && xg_cluster_ok(c, sm)) { cs = c; smem = sm; break; }
    }
    if (!cs) return DARTREE_OK;
    *launched = true;
    gather_rows_kernel<<<M, 256, 0, stream>>>(static_cast<const uint16_t*>(a.E), a.cand_tok, a.H, a.Eg);
    if (cudaGetLastError() != cudaSuccess) return DARTREE_ECUDA;
    if (int e = launch_gemm_bf16_tc(a.Eg, a.WqT, M, a.H, a.H, 2, nullptr, a.Ghi, 1, a.status, stream, a.Glo)) return e;
    XgArgs x{};
    x.E = static_cast<const uint16_t*>(a.E);
    x.hidden = static_cast<const uint16_t*>(a.hidden);
    x.anchor = a.anchor;
    x.cand_tok = a.cand_tok;
    x.cand_val = a.cand_val;
    x.Ghi = a.Ghi;
    x.Glo = a.Glo;
    x.H = a.H;
    x.L = a.L;
    x.K = a.K;
    x.W = a.W;
    x.cs = cs;
    x.beta = a.beta;
    x.inv_sqrt_h = 1.0f / sqrtf(float(a.H));
    x.st_tok = a.st_tok;
    x.st_par = a.st_par;
    x.st_s = a.st_s;
    x.st_n = a.st_n;
    x.status = a.status;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(a.C) * cs);
    cfg.blockDim = dim3(XG_NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, expand_g_kernel, x) == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

}  // namespace dartree
