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
// depths. CTA q of the cluster owns H/CS features of h, G and E, and parent
// rows p with p mod CS = q. Per depth, three exchanges through distributed
// shared memory, each made of st.async stores that count their bytes on the
// receiver's mbarrier (no cluster barrier: a receiver waits for exactly the
// data it needs, and a sender never waits):
//
//   1. partial logits over the CTA's features (mma.sync), each parent row sent
//      to its owner's shared memory (reduce-scatter);
//   2. the owner sums the CS partials of its rows in a fixed order, takes the
//      log-softmax and scores, ranks the row's candidates by counting, and
//      broadcasts the row's best min(W, K) keys, sorted, to every CTA;
//   3. every CTA merges the P sorted lists with a bitonic merge tree (pairs of
//      16-key lists per warp, four levels), so all of them take the same top-W;
//      the kept children's state slices x = h_p + E[tok] + H_d[d-1] are formed,
//      partial sums of squares exchanged, and the slices normalised into the
//      next parent buffer.
//
// The candidate table of the request sits in shared memory (it arrives, with the
// root row E[anchor], by bulk copy on the first prefetch's barrier). The G, E and
// H_d slices of the next position arrive by TMA while the current depth runs: G
// as 32-column tiles with 64-byte swizzle (conflict-free ldmatrix), E as one tile
// of the gathered candidate rows, H_d as one bulk copy, all completing on one
// mbarrier. Waits are bounded; a wait that runs out records a timeout and the
// CTA keeps taking part in every cluster barrier, so no peer is left waiting.
#include <math.h>

#include "common.cuh"
#include "finish.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace dartree {

constexpr int XG_NT = 256;
constexpr int XG_NW = XG_NT / 32;
constexpr int XG_MAXK = 64;   // candidates per position: two per lane in the score pass
constexpr int XG_MAXW = 16;   // parents per depth: one 16-row mma tile

__host__ __device__ constexpr size_t xg_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct XgLayout {
    size_t gs, hs, es, hds, ctok, cval, zred, rkeys, lists, mrg, ssq, sel, spar, stout, fgk, ftree, fnext, frow,
        fcnt, floc, fbits, mbar, total;
};

constexpr int XG_GB = 32;  // columns of one swizzled G tile (64 bytes)

// fs: features per CTA (a multiple of 32, at most 256), cs: cluster size, B: node
// budget of the S8-S10 run after the last depth (0: none)
__host__ __device__ inline XgLayout xg_layout(int fs, int K, int cs, int L, int B) {
    const size_t fp = size_t(fs) + 8;
    const size_t rpo = XG_MAXW / cs;  // parent rows per owner
    XgLayout l{};
    size_t o = 0;
    auto take = [&](size_t b, size_t al) { o = xg_up(o, al); size_t at = o; o += b; return at; };
    l.gs = take(2 * size_t(K) * fs * 2, 1024);        // G_hi, G_lo: fs/32 swizzled tiles [K][32] each
    l.hs = take(2 * XG_MAXW * fp * 2, 128);          // parent state slices, two buffers of 16 padded rows
    l.es = take(2 * size_t(K) * fs * 2, 128);        // E slices [K][fs], two positions
    l.hds = take(2 * size_t(fs) * 2, 128);           // H_d slices, two positions
    l.ctok = take(size_t(L) * K * 4, 16);            // candidate table of the request
    l.cval = take(size_t(L) * K * 4, 16);
    l.zred = take(size_t(cs) * rpo * K * 4, 16);     // partial logits of the owned rows [q][slot][c]
    l.rkeys = take(rpo * size_t(K) * 8, 16);         // keys of the owned rows
    l.lists = take(size_t(XG_MAXW) * XG_MAXW * 8, 16);  // best keys of every row, sorted [p][j]
    l.mrg = take(2 * size_t(XG_NW) * 16 * 8, 16);        // merge tree levels, ping-pong
    l.ssq = take(size_t(cs) * XG_MAXW * 4, 16);      // partial sums of squares [q][k]
    l.sel = take(size_t(XG_MAXW) * 8 + 2 * XG_MAXW * 4, 16);
    l.spar = take(size_t(XG_MAXW) * 4, 16);
    l.stout = take(size_t(L) * XG_MAXW * 8 + size_t(L) * 4, 16);  // supertree of the request, written at the end
    // S8-S10 after the last depth (B + 1 slots)
    const size_t S = size_t(B) + 1;
    l.fgk = take(size_t(L) * XG_MAXW * 8, 16);       // keys in the global order [L][16]
    l.ftree = take(4 * S * 4, 16);                   // slot arrays: token, parent, depth, score
    l.fnext = take(S * 4, 16);                       // accepted child of every slot
    l.frow = take(size_t(L) * 8, 16);                // per-position target row maxima
    l.fcnt = take(2 * size_t(L) * 4, 16);            // chosen per depth (received), first slot per depth
    l.floc = take(64 * 4, 16);                       // chosen per local depth; totals
    l.fbits = take(size_t(XG_NW) * 32 * 4, 16);      // one ancestor bitset per warp (S <= 1024)
    l.mbar = take(5 * 8, 8);                         // prefetch barrier; exchanges A, B, C; chosen counts F
    l.total = o;
    return l;
}

struct XgArgs {
    const uint16_t* E;
    const uint16_t* hidden;
    const int32_t* anchor;
    const int32_t* cand_tok;
    const float* cand_val;
    int H, L, K, W;
    float beta, inv_sqrt_h;
    int32_t* st_tok;
    int32_t* st_par;
    float* st_s;
    int32_t* st_n;
    int* status;
    int fin;       // run S8-S10 (and the walk when fo.rowkeys is set) after the last depth
    int B;
    FinishOut fo;
};

__device__ __forceinline__ void xg_ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void xg_mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Remote stores into a peer CTA's shared memory that count their bytes on the
// peer's mbarrier (addr and bar: shared::cluster addresses from mapa).
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];"
                 :: "r"(addr), "f"(v), "r"(bar) : "memory");
}
__device__ __forceinline__ void st_async_v2f32(uint32_t addr, float x, float y, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
                 :: "r"(addr), "f"(x), "f"(y), "r"(bar) : "memory");
}
__device__ __forceinline__ void st_async_u32(uint32_t addr, uint32_t v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                 :: "r"(addr), "r"(v), "r"(bar) : "memory");
}
__device__ __forceinline__ void st_async_b64(uint32_t addr, uint64_t v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];"
                 :: "r"(addr), "l"(v), "r"(bar) : "memory");
}

// Sum over the 16 lanes of a half-warp (every lane of the warp takes part).
__device__ __forceinline__ float half_sum(float v) {
#pragma unroll
    for (int m = 8; m; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

// S8-S10 of request r after the last depth, by the whole cluster (DARTree blog
// post, 3.1: deferred pruning, one global top-B over the supertree, prefix-closed
// for beta <= 0 (Lemma 1); 3.2: tree-attention mask, position ids, greedy longest
// accepted prefix). Every CTA holds the same supertree: the kept keys of every
// depth, sorted. In the global order (score desc, depth asc, rank asc) the
// chosen set is the top min(B, nodes), and within a depth it is a prefix of the
// sorted keys, so a depth's choice is one number: CTA q ranks the keys of depths
// q, q + CS, ... against all keys (a warp per key), and sends each such depth's
// chosen count to every CTA (st.async counted on barrier F). With all counts,
// every CTA lays out the slots (depth-major, rank within a depth) and the parents'
// slots itself. CTA 0 writes the tree arrays, CTA q the mask rows i = q mod CS,
// and CTA 1 (CTA 0 for a cluster of one) follows the greedy walk over the
// per-position target row maxima. Remote stores into this CTA all completed before
// the last depth's list barrier, and no copy is in flight.
template <int CS>
__device__ void xg_finish(const XgArgs& a, uint8_t* smem, const XgLayout& lay, int r, uint32_t cr,
                          const uint64_t* stkey, const int* stn, const int32_t* ctok) {
    const int L = a.L, K = a.K, S = a.B + 1;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint64_t* fgk = reinterpret_cast<uint64_t*>(smem + lay.fgk);
    int* ttok = reinterpret_cast<int*>(smem + lay.ftree);
    int* tpar = ttok + S;
    int* tdep = ttok + 2 * S;
    float* tsc = reinterpret_cast<float*>(ttok + 3 * S);
    int* fnext = reinterpret_cast<int*>(smem + lay.fnext);
    uint64_t* frow = reinterpret_cast<uint64_t*>(smem + lay.frow);
    int* fcnt = reinterpret_cast<int*>(smem + lay.fcnt);  // [L] chosen per depth
    int* foff = fcnt + L;                                 // [L] first slot of every depth
    int* floc = reinterpret_cast<int*>(smem + lay.floc);  // [0..8) chosen per local depth, [32] total
    uint32_t* fbits = reinterpret_cast<uint32_t*>(smem + lay.fbits);
    uint64_t* mbF = reinterpret_cast<uint64_t*>(smem + lay.mbar) + 4;
    const uint32_t walker = CS > 1 ? 1u : 0u;
    const bool walk = a.fo.rowkeys != nullptr && cr == walker;
    const int nd = L * XG_MAXW;
    if (walk)  // (the global loads overlap the ranking)
        for (int d = threadIdx.x; d < L; d += XG_NT) frow[d] = a.fo.rowkeys[size_t(r) * L + d];
    for (int i = threadIdx.x; i < nd; i += XG_NT) {
        const int dm1 = i / XG_MAXW, k = i % XG_MAXW;
        fgk[i] = k < stn[dm1] ? finish_key(uint32_t(stkey[i] >> 32), dm1, k) : 0ull;
    }
    if (threadIdx.x < 64) floc[threadIdx.x] = 0;
    if (threadIdx.x == 0) mbar_arrive_expect_tx(mbF, uint32_t(L * 4));
    __syncthreads();
    int nv = 0;
    // (loops over shared memory are unrolled so that their loads are in flight together)
#pragma unroll 16
    for (int d = 0; d < L; ++d) nv += stn[d];
    const int N = min(a.B, nv);
    // ranks of the keys of depths cr, cr + CS, ...: a warp per key, lanes over all keys
    const int nloc = (L - int(cr) + CS - 1) / CS;
    for (int i = wid; i < nloc * XG_MAXW; i += XG_NW) {
        const int dl = i / XG_MAXW, k = i % XG_MAXW, dm1 = int(cr) + dl * CS;
        if (k >= stn[dm1]) continue;  // uniform across the warp
        const uint64_t x = fgk[dm1 * XG_MAXW + k];
        int c = 0;
        for (int j0 = lane; j0 < nd; j0 += 32 * 8) {  // 8 unconditional loads in flight
            uint64_t y[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) y[u] = fgk[min(j0 + 32 * u, nd - 1)];
#pragma unroll
            for (int u = 0; u < 8; ++u) c += (j0 + 32 * u < nd && y[u] > x) ? 1 : 0;
        }
        c = __reduce_add_sync(0xffffffffu, c);
        if (lane == 0 && c < N) atomicAdd(&floc[dl], 1);
    }
    __syncthreads();
    for (int t = threadIdx.x; t < nloc * CS; t += XG_NT) {
        const int dl = t / CS, q = t % CS, dm1 = int(cr) + dl * CS;
        st_async_u32(mapa_u32(smem_u32(fcnt + dm1), uint32_t(q)), uint32_t(floc[dl]),
                     mapa_u32(smem_u32(mbF), uint32_t(q)));
    }
    mbar_wait_bounded(mbF, 0, a.status);  // every depth's chosen count
    // first slot of every depth: 1 + chosen counts of the depths above (L <= 64)
    if (wid == 0) {
        const int v0 = lane < L ? fcnt[lane] : 0, v1 = lane + 32 < L ? fcnt[lane + 32] : 0;
        int s0 = v0, s1 = v1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y0 = __shfl_up_sync(0xffffffffu, s0, o), y1 = __shfl_up_sync(0xffffffffu, s1, o);
            if (lane >= o) { s0 += y0; s1 += y1; }
        }
        const int t0 = __shfl_sync(0xffffffffu, s0, 31);
        if (lane < L) foff[lane] = 1 + s0 - v0;
        if (lane + 32 < L) foff[lane + 32] = 1 + t0 + s1 - v1;
        if (lane == 31) floc[32] = t0 + s1;
    }
    __syncthreads();
    const int chosen = floc[32], nn = min(S, 1 + chosen);
    if (cr == 0 && threadIdx.x == 0 && chosen != N) set_status(a.status, DARTREE_EINTERNAL);
    // slot arrays (parents as slots: a chosen node's parent must be chosen)
    for (int i = threadIdx.x; i < nd; i += XG_NT) {
        const int dm1 = i / XG_MAXW, k = i % XG_MAXW;
        if (k < fcnt[dm1]) {
            const int j = foff[dm1] + k;
            const uint64_t sk = stkey[i];
            const uint32_t f = 0xffffffffu - uint32_t(sk);
            const int pr = int(f) / K;
            int ps = 0;
            if (dm1 > 0) {
                ps = pr < fcnt[dm1 - 1] ? foff[dm1 - 1] + pr : -1;
                if (ps < 0 && cr == 0) set_status(a.status, DARTREE_EINTERNAL);  // not prefix-closed
            }
            if (j < S) {
                ttok[j] = ctok[dm1 * K + int(f) % K];
                tpar[j] = ps;
                tdep[j] = dm1 + 1;
                tsc[j] = f32_from_ord(uint32_t(sk >> 32));
            }
        }
    }
    for (int j = threadIdx.x; j < S; j += XG_NT) {
        if (j == 0) {
            ttok[0] = a.anchor[r];
            tpar[0] = -1;
            tdep[0] = 0;
            tsc[0] = 0.f;
        } else if (j >= nn) {
            ttok[j] = tpar[j] = tdep[j] = -1;
            tsc[j] = 0.f;
        }
    }
    __syncthreads();
    if (cr == 0) {
        for (int j = threadIdx.x; j < S; j += XG_NT) {
            const size_t o = size_t(r) * S + j;
            a.fo.tok[o] = ttok[j];
            a.fo.par[o] = tpar[j];
            a.fo.depth[o] = tdep[j];
            a.fo.score[o] = tsc[j];
            if (a.fo.pos) a.fo.pos[o] = tdep[j];
        }
        if (threadIdx.x == 0) a.fo.n_nodes[r] = 1 + chosen;
    }
    // S9: mask rows i = cr (mod CS), a warp per row: the ancestor-or-self bitset of
    // slot i (a walk up its parents), then one byte per column
    if (a.fo.mask) {
        uint32_t* bits = fbits + wid * 32;
        const int nw = (S + 31) / 32;
        for (int i = int(cr) + wid * CS; i < S; i += CS * XG_NW) {
            if (lane < nw) bits[lane] = 0u;
            __syncwarp();
            if (lane == 0 && i < nn) {
                int b = i;
                for (int g = 0; g <= L && b >= 0 && b < S; ++g) {
                    bits[b >> 5] |= 1u << (b & 31);
                    b = tpar[b];
                }
            }
            __syncwarp();
            uint8_t* row = a.fo.mask + (size_t(r) * S + i) * S;
            for (int j = lane; j < S; j += 32) row[j] = uint8_t((bits[j >> 5] >> (j & 31)) & 1u);
            __syncwarp();
        }
    }
    // S10 with per-position row maxima: every slot's accepted child (the lowest slot
    // under it whose token is the argmax of its row), then one thread follows them
    if (walk) {
        for (int j = threadIdx.x; j < S; j += XG_NT) fnext[j] = 0x7fffffff;
        __syncthreads();
        for (int j = 1 + threadIdx.x; j < nn; j += XG_NT) {
            const int p = tpar[j];
            const int dp = (p >= 0 && p < nn) ? tdep[p] : -1;
            if (dp >= 0 && dp < L && ttok[j] == int(0xffffffffu - uint32_t(frow[dp]))) atomicMin(&fnext[p], j);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int cur = 0, acc = 0, bon = -1;
            for (int step = 0; step <= L; ++step) {
                const int d = tdep[cur];
                if (d < 0 || d >= L) break;
                const int f = fnext[cur];
                if (f == 0x7fffffff) {
                    bon = int(0xffffffffu - uint32_t(frow[d]));
                    break;
                }
                if (acc < L) a.fo.path[size_t(r) * L + acc] = f;
                ++acc;
                cur = f;
            }
            a.fo.accepted[r] = acc;
            a.fo.bonus[r] = bon;
            floc[33] = acc;
        }
        __syncthreads();
        for (int u = floc[33] + threadIdx.x; u < L; u += XG_NT) a.fo.path[size_t(r) * L + u] = -1;
    }
}

template <int CS>
__global__ void __launch_bounds__(XG_NT, 1) expand_g_kernel(XgArgs a, const __grid_constant__ CUtensorMap tm_ghi,
                                                             const __grid_constant__ CUtensorMap tm_glo,
                                                             const __grid_constant__ CUtensorMap tm_eg) {
    constexpr int RPO = XG_MAXW / CS;  // parent rows per owner
    extern __shared__ __align__(1024) uint8_t smem[];
    const int H = a.H, L = a.L, K = a.K, W = a.W;
    const int fs = H / CS, fp = fs + 8, cpr = fs / 8, nb = fs / XG_GB;
    const XgLayout lay = xg_layout(fs, K, CS, L, a.fin ? a.B : 0);
    uint8_t* gs = smem + lay.gs;
    uint16_t* hs = reinterpret_cast<uint16_t*>(smem + lay.hs);
    uint16_t* es = reinterpret_cast<uint16_t*>(smem + lay.es);
    uint16_t* hds = reinterpret_cast<uint16_t*>(smem + lay.hds);
    int32_t* ctok = reinterpret_cast<int32_t*>(smem + lay.ctok);
    float* cval = reinterpret_cast<float*>(smem + lay.cval);
    float* zred = reinterpret_cast<float*>(smem + lay.zred);
    uint64_t* rkeys = reinterpret_cast<uint64_t*>(smem + lay.rkeys);
    uint64_t* lists = reinterpret_cast<uint64_t*>(smem + lay.lists);
    uint64_t* mrg = reinterpret_cast<uint64_t*>(smem + lay.mrg);
    float* ssq = reinterpret_cast<float*>(smem + lay.ssq);
    uint64_t* selk = reinterpret_cast<uint64_t*>(smem + lay.sel);  // kept keys, descending
    int* selx = reinterpret_cast<int*>(selk + XG_MAXW);            // [0..16): parent rank, [16..32): candidate
    float* spar = reinterpret_cast<float*>(smem + lay.spar);       // parent scores
    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + lay.mbar);  // prefetch
    uint64_t* mbA = mbar + 1;  // partial logits of the owned rows
    uint64_t* mbB = mbar + 2;  // row lists
    uint64_t* mbC = mbar + 3;  // partial sums of squares (mbar + 4: chosen counts of S8, in xg_finish)
    uint64_t* stkey = reinterpret_cast<uint64_t*>(smem + lay.stout);  // [L][16] kept keys (0 = none)
    int* stn = reinterpret_cast<int*>(stkey + size_t(L) * XG_MAXW);    // [L] kept per depth

    const uint32_t cr = cluster_ctarank();
    const int r = blockIdx.x / CS;
    const int f0 = int(cr) * fs;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;

    // G (and, with_e, the E and H_d slices) of position pos, with `extra` more bytes
    // expected on the barrier; one thread
    auto prefetch = [&](int pos, bool with_e, uint32_t extra) {
        const int row = (r * L + pos) * K;  // first candidate row of the position in G and E[cand]
        mbar_arrive_expect_tx(mbar, uint32_t((2 + (with_e ? 1 : 0)) * K * fs * 2 + (with_e ? fs * 2 : 0)) + extra);
        for (int b = 0; b < nb; ++b) {
            tc::tma_load_2d(gs + size_t(b) * K * 64, &tm_ghi, f0 + b * XG_GB, row, mbar);
            tc::tma_load_2d(gs + size_t(nb + b) * K * 64, &tm_glo, f0 + b * XG_GB, row, mbar);
        }
        if (with_e) {
            tc::tma_load_2d(es + size_t(pos & 1) * K * fs, &tm_eg, f0, row, mbar);
            bulk_g2s(hds + size_t(pos & 1) * fs, a.hidden + (size_t(r) * L + pos) * H + f0, uint32_t(fs * 2), mbar);
        }
    };

    griddep_launch_dependents();
    const uint32_t tbl = uint32_t(L * K * 4);  // bytes of the candidate tokens (and of their values)
    if (threadIdx.x == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(&mbar[i], 1);
        fence_mbar_init();
        // root: h = E[anchor] (this CTA's slice), on the first prefetch's barrier (the
        // head and the anchor are not written by the kernels before this one)
        bulk_g2s(hs, a.E + size_t(a.anchor[r]) * H + f0, uint32_t(fs * 2), mbar);
        spar[0] = 0.f;
    }
    __syncthreads();
    cluster_sync();  // every peer's exchange barriers are initialised before any store targets them
    // the candidates, their rows and G come from the kernels before this one: G of
    // position 0 and the candidate table arrive with the root row on one barrier
    griddep_wait();
    if (threadIdx.x == 0) {
        prefetch(0, L > 1, uint32_t(fs * 2) + 2 * tbl);
        bulk_g2s(ctok, a.cand_tok + size_t(r) * L * K, tbl, mbar);
        bulk_g2s(cval, a.cand_val + size_t(r) * L * K, tbl, mbar);
    }
    int issued = 1, waited = 0;  // prefetch phases (uniform across the CTA)
    bool pf_ok = true;           // false once a prefetch wait ran out: no further prefetches
    int cur = 0, P = 1;

    for (int d = 1; d <= L; ++d) {
        const int pos = d - 1;
        const int ne = P * K;
        const int n_keep = min(W, ne);
        const int m = min(n_keep, K);  // keys per row list
        const uint32_t par = uint32_t(pos) & 1u;
        int owned = 0;  // owned rows of this depth
        for (int sl = 0; sl < RPO; ++sl) owned += int(cr) + CS * sl < P;
        // a timed-out prefetch wait records ETIMEOUT and the CTA carries on with the
        // exchanges, so that no peer is left waiting for its data
        if (pf_ok) pf_ok = __syncthreads_and(mbar_wait_bounded(mbar, uint32_t(waited) & 1u, a.status) ? 1 : 0) != 0;
        else __syncthreads();
        if (pf_ok) waited = issued;
        // ---- 1. partial logits over this CTA's features, each row to its owner
        {
            const uint16_t* hb = hs + size_t(cur) * XG_MAXW * fp;
            const int lm = lane >> 3, lr = lane & 7, g = lane >> 2, t = lane & 3;
            const uint32_t z0 = smem_u32(zred), g0 = smem_u32(gs);
            for (int ct = wid; ct * 8 < K; ct += XG_NW) {  // 8 candidates per tile
                const int n = ct * 8 + lr;                 // candidate row this lane addresses
                // matrices: (hi, k lo), (hi, k hi), (lo, k lo), (lo, k hi)
                const uint32_t brow = g0 + uint32_t(((lm >> 1) * nb * K + n) * 64);
                const uint32_t sw = uint32_t((n >> 1) & 3);
                // two accumulator chains per operand (even and odd k-steps), summed in a
                // fixed order at the end
                float acc_hi[4] = {0.f, 0.f, 0.f, 0.f}, acc_lo[4] = {0.f, 0.f, 0.f, 0.f};
                float acc_hi2[4] = {0.f, 0.f, 0.f, 0.f}, acc_lo2[4] = {0.f, 0.f, 0.f, 0.f};
                auto kstep = [&](int k0, float (&ah)[4], float (&al)[4]) {
                    uint32_t af[4], bf[4];
                    xg_ldsm_x4(af, smem_u32(hb + size_t((lm & 1) * 8 + lr) * fp + k0 + (lm >> 1) * 8));
                    const uint32_t chunk = uint32_t(((k0 & 31) >> 3) + (lm & 1));
                    xg_ldsm_x4(bf, brow + uint32_t((k0 >> 5) * K * 64) + ((chunk ^ sw) << 4));
                    xg_mma(ah, af, bf[0], bf[1]);
                    xg_mma(al, af, bf[2], bf[3]);
                };
                int k0 = 0;
                for (; k0 + 16 < fs; k0 += 32) {  // fs is a multiple of 32
                    kstep(k0, acc_hi, acc_lo);
                    kstep(k0 + 16, acc_hi2, acc_lo2);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc_hi[i] += acc_hi2[i];
                    acc_lo[i] += acc_lo2[i];
                }
                const int c = ct * 8 + 2 * t;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int p = g + 8 * hh;
                    if (p < P) {
                        const uint32_t off = z0 + uint32_t(((int(cr) * RPO + p / CS) * K + c) * 4);
                        const uint32_t ow = uint32_t(p % CS);
                        st_async_v2f32(mapa_u32(off, ow), acc_hi[2 * hh] + acc_lo[2 * hh],
                                       acc_hi[2 * hh + 1] + acc_lo[2 * hh + 1], mapa_u32(smem_u32(mbA), ow));
                    }
                }
            }
        }
        // arm this depth's exchange barriers (data that lands before the arrival
        // only drives the transaction count negative for a while)
        if (threadIdx.x == 0) {
            // one arrival per phase: a barrier whose previous phase did not complete
            // (a wait that ran out) gets none, and the status records the timeout
            auto arm = [&](uint64_t* b, uint32_t bytes) {
                if (mbar_try_wait(b, par ^ 1u)) mbar_arrive_expect_tx(b, bytes);
                else set_status(a.status, DARTREE_ETIMEOUT);
            };
            arm(mbA, uint32_t(owned * CS * K * 4));
            arm(mbB, uint32_t(P * m * 8));
            if (d < L) arm(mbC, uint32_t(CS * n_keep * 4));
        }
        __syncthreads();  // gs free
        // ---- 2. owned rows: z, log-softmax, scores (warp s: row slot s)
        if (wid < RPO) {
            const int p = int(cr) + CS * wid;
            if (p < P) {
                mbar_wait_bounded(mbA, par, a.status);  // the CS partials of the owned rows
                float zv[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c = lane + 32 * h;
                    zv[h] = -INFINITY;
                    if (c < K) {
                        float sacc = 0.f;
#pragma unroll
                        for (int q = 0; q < CS; ++q) sacc += zred[(q * RPO + wid) * K + c];
                        zv[h] = cval[pos * K + c] + sacc * a.inv_sqrt_h;
                    }
                }
                const float mx = f32_from_ord(__reduce_max_sync(0xffffffffu, ord_f32(fmaxf(zv[0], zv[1]))));
                float se = 0.f;
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    if (lane + 32 * h < K) se += expf(zv[h] - mx);
                se = warp_sum(se);
                const float lse = mx + logf(se);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c = lane + 32 * h;
                    if (c < K) {
                        float sc = (spar[p] + (zv[h] - lse)) + a.beta;
                        sc += 0.f;  // -0 -> +0
                        const uint32_t f = uint32_t(p * K + c);
                        rkeys[wid * K + c] = (uint64_t(ord_f32(sc)) << 32) | (0xffffffffu - f);
                    }
                }
            }
        } else if (threadIdx.x == 32 * RPO && pf_ok && d < L) {
            prefetch(pos + 1, d + 1 < L, 0);
        }
        if (pf_ok && d < L) ++issued;
        __syncthreads();
        // rank of every owned key within its row (4 lanes per key), best m broadcast
        for (int item = threadIdx.x >> 2; item < RPO * K; item += XG_NT / 4) {
            const int slot = item / K, i = item % K, qd = threadIdx.x & 3;
            const int p = int(cr) + CS * slot;
            const bool live = p < P;
            int cnt = 0;
            uint64_t x = 0;
            if (live) {
                x = rkeys[slot * K + i];
                // K <= 64: the 16 loads are unconditional (clamped index), so they are
                // all in flight together
                uint64_t y[XG_MAXK / 4];
#pragma unroll
                for (int jj = 0; jj < XG_MAXK / 4; ++jj) y[jj] = rkeys[slot * K + min(qd + 4 * jj, K - 1)];
#pragma unroll
                for (int jj = 0; jj < XG_MAXK / 4; ++jj) cnt += (qd + 4 * jj < K && y[jj] > x) ? 1 : 0;
            }
            cnt += __shfl_xor_sync(0xffffffffu, cnt, 1);
            cnt += __shfl_xor_sync(0xffffffffu, cnt, 2);
            if (live && cnt < m) {
                // lane qd writes the key to CTAs qd, qd + 4, ...
                const uint32_t off = smem_u32(lists + p * XG_MAXW + cnt);
                for (int q = qd; q < CS; q += 4)
                    st_async_b64(mapa_u32(off, uint32_t(q)), x, mapa_u32(smem_u32(mbB), uint32_t(q)));
            }
        }
        mbar_wait_bounded(mbB, par, a.status);  // every row list
        // ---- 3. top-W: bitonic merge tree over the 16 row lists (slots past m or P
        //         are empty = 0); level 1: warp w merges lists 2w and 2w + 1
        {
            const int hl = lane & 15, q = 2 * wid + (lane >> 4);
            uint64_t v = (q < P && hl < m) ? lists[q * XG_MAXW + hl] : 0ull;
            v = xg_merge16(v);
            if (lane < 16) mrg[wid * 16 + lane] = v;
            __syncthreads();
            // level 2: warps 0..3
            if (wid < 4) {
                v = mrg[(2 * wid + (lane >> 4)) * 16 + hl];
                v = xg_merge16(v);
                if (lane < 16) mrg[XG_NW * 16 + wid * 16 + lane] = v;
            }
            __syncthreads();
            // levels 3 and 4 in warp 0: lists 0+1 and 2+3, then the two results
            if (wid == 0) {
                const uint64_t ab = xg_merge16(mrg[XG_NW * 16 + (lane >> 4) * 16 + hl]);
                const uint64_t cd = xg_merge16(mrg[XG_NW * 16 + (2 + (lane >> 4)) * 16 + hl]);
                const uint32_t lo = __shfl_up_sync(0xffffffffu, uint32_t(cd), 16);
                const uint32_t hi = __shfl_up_sync(0xffffffffu, uint32_t(cd >> 32), 16);
                const uint64_t x = xg_merge16(lane < 16 ? ab : ((uint64_t(hi) << 32) | lo));
                if (lane < n_keep) {
                    const uint32_t f = 0xffffffffu - uint32_t(x);
                    selk[lane] = x;
                    selx[lane] = int(f) / K;
                    selx[XG_MAXW + lane] = int(f) % K;
                }
            }
        }
        __syncthreads();
        // supertree entries stay in shared memory until the depth loop ends (global
        // stores inside the loop would hold up the release of the next cluster barrier)
        if (threadIdx.x < XG_MAXW) stkey[pos * XG_MAXW + threadIdx.x] = threadIdx.x < n_keep ? selk[threadIdx.x] : 0ull;
        if (threadIdx.x == 0) stn[pos] = n_keep;
        if (d == L) break;  // no remote access follows barrier B of the last depth
        // ---- state slices of the kept children: half-warp k owns row k, its lane
        //      j the 8-feature chunks j and j + 16
        const uint16_t* hb = hs + size_t(cur) * XG_MAXW * fp;
        uint16_t* hn = hs + size_t(1 - cur) * XG_MAXW * fp;
        const uint16_t* eb = es + size_t(pos & 1) * K * fs;
        const uint16_t* hdb = hds + size_t(pos & 1) * fs;
        const int k = threadIdx.x >> 4, hl = threadIdx.x & 15;
        const bool row_ok = k < n_keep;
        float x[2][8];
        {
            float ss = 0.f;
            if (row_ok) {
                const uint16_t* hp = hb + size_t(selx[k]) * fp;
                const uint16_t* er = eb + size_t(selx[XG_MAXW + k]) * fs;
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int j = hl + 16 * cc;
                    if (j < cpr) {
                        const uint4 vp = *reinterpret_cast<const uint4*>(hp + j * 8);
                        const uint4 ve = *reinterpret_cast<const uint4*>(er + j * 8);
                        const uint4 vh = *reinterpret_cast<const uint4*>(hdb + j * 8);
                        const uint32_t* wp = reinterpret_cast<const uint32_t*>(&vp);
                        const uint32_t* we = reinterpret_cast<const uint32_t*>(&ve);
                        const uint32_t* wh = reinterpret_cast<const uint32_t*>(&vh);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int sh = (i & 1) ? 16 : 0;
                            const float xv = (bf16_bits_to_float((wp[i >> 1] >> sh) & 0xffffu) +
                                              bf16_bits_to_float((we[i >> 1] >> sh) & 0xffffu)) +
                                             bf16_bits_to_float((wh[i >> 1] >> sh) & 0xffffu);
                            x[cc][i] = xv;
                            ss = fmaf(xv, xv, ss);
                        }
                    }
                }
            }
            ss = half_sum(ss);  // both half-warps of a warp take part
            if (row_ok && hl < CS)
                st_async_f32(mapa_u32(smem_u32(ssq + int(cr) * XG_MAXW + k), uint32_t(hl)), ss,
                             mapa_u32(smem_u32(mbC), uint32_t(hl)));
        }
        mbar_wait_bounded(mbC, par, a.status);  // every partial sum of squares
        if (row_ok) {
            // the CS partial sums in four fixed chains; reciprocal square root in
            // one instruction (its error is far below the bf16 rounding of h)
            float t4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int q = 0; q < CS; ++q) t4[q & 3] += ssq[q * XG_MAXW + k];
            const float tot = (t4[0] + t4[1]) + (t4[2] + t4[3]);
            const float inv = rsqrtf(tot / float(H) + 1e-6f);
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int j = hl + 16 * cc;
                if (j < cpr) {
                    uint32_t w4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        w4[i] = uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(x[cc][2 * i] * inv))) |
                                (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(x[cc][2 * i + 1] * inv))) << 16);
                    *reinterpret_cast<uint4*>(hn + size_t(k) * fp + j * 8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
            }
        }
        if (threadIdx.x < n_keep) spar[threadIdx.x] = f32_from_ord(uint32_t(selk[threadIdx.x] >> 32));
        cur = 1 - cur;
        P = n_keep;
    }
    // the supertree: CTA q writes depths q, q + CS, ...
    __syncthreads();
    for (int pd = int(cr); pd < L; pd += CS) {
        const int nk = stn[pd];
        for (int k = threadIdx.x; k < W; k += XG_NT) {
            const size_t o = (size_t(r) * L + pd) * W + k;
            const uint64_t key = k < XG_MAXW ? stkey[pd * XG_MAXW + k] : 0ull;
            if (k < nk) {
                const uint32_t f = 0xffffffffu - uint32_t(key);
                a.st_tok[o] = ctok[pd * K + int(f) % K];
                a.st_par[o] = int(f) / K;
                a.st_s[o] = f32_from_ord(uint32_t(key >> 32));
            } else {
                a.st_tok[o] = -1;
                a.st_par[o] = -1;
                a.st_s[o] = 0.f;
            }
        }
        if (threadIdx.x == 0) a.st_n[size_t(r) * L + pd] = nk;
    }
    // a prefetch still in flight (only after a timed-out wait) lands before the CTA leaves
    if (!pf_ok) mbar_wait_bounded(mbar, uint32_t(waited) & 1u, a.status);
    if (a.fin) xg_finish<CS>(a, smem, lay, r, cr, stkey, stn, ctok);
}

// --------------------------------------------------------------------------- gathers, transpose

// out[m] = E[idx[m]]: GR_ROWS rows per CTA, every load of a thread issued before
// its stores.
constexpr int GR_ROWS = 8, GR_NT = 256, GR_MAXV = 3;  // rows of up to GR_MAXV * GR_NT vectors
__global__ void __launch_bounds__(GR_NT) gather_rows_kernel(const uint16_t* __restrict__ E,
                                                            const int32_t* __restrict__ idx, int H, int M,
                                                            uint16_t* __restrict__ out) {
    const int nv = H / 8;
    uint4 v[GR_ROWS][GR_MAXV];
#pragma unroll
    for (int i = 0; i < GR_ROWS; ++i) {
        const int m = blockIdx.x * GR_ROWS + i;
        if (m < M) {
            const uint4* src = reinterpret_cast<const uint4*>(E + size_t(idx[m]) * H);
#pragma unroll
            for (int j = 0; j < GR_MAXV; ++j)
                if (int(threadIdx.x) + j * GR_NT < nv) v[i][j] = __ldg(src + threadIdx.x + j * GR_NT);
        }
    }
#pragma unroll
    for (int i = 0; i < GR_ROWS; ++i) {
        const int m = blockIdx.x * GR_ROWS + i;
        if (m < M) {
            uint4* dst = reinterpret_cast<uint4*>(out + size_t(m) * H);
#pragma unroll
            for (int j = 0; j < GR_MAXV; ++j)
                if (int(threadIdx.x) + j * GR_NT < nv) dst[threadIdx.x + j * GR_NT] = v[i][j];
        }
    }
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

int launch_gather_rows(const uint16_t* E, const int32_t* idx, int H, int M, uint16_t* out, cudaStream_t stream) {
    if (M == 0) return DARTREE_OK;
    if (H % 8 != 0 || H / 8 > GR_MAXV * GR_NT) return DARTREE_EUNSUPPORTED;
    {
        KTimer kt_(KID_GATHER, stream);
        gather_rows_kernel<<<(M + GR_ROWS - 1) / GR_ROWS, GR_NT, 0, stream>>>(E, idx, H, M, out);
    }
    return cudaGetLastError() == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

int launch_transpose_bf16(const void* src, void* dst, int H, cudaStream_t stream) {
    dim3 grid((H + 31) / 32, (H + 31) / 32), block(32, 8);
    {
        KTimer kt_(KID_OTHER, stream);
        transpose_bf16_kernel<<<grid, block, 0, stream>>>(static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst), H);
    }
    return cudaGetLastError() == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

// --------------------------------------------------------------------------- host

template <int CS>
static bool xg_cluster_ok(size_t smem) {
    auto kern = expand_g_kernel<CS>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess ||
        (CS > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)) {
        cudaGetLastError();
        return false;
    }
    cudaLaunchConfig_t q{};
    q.gridDim = dim3(unsigned(CS));
    q.blockDim = dim3(XG_NT);
    q.dynamicSmemBytes = smem;
    cudaLaunchAttribute qa[1];
    qa[0].id = cudaLaunchAttributeClusterDimension;
    qa[0].val.clusterDim.x = CS;
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

template <int CS>
static int xg_launch(const XgArgs& x, const CUtensorMap& ghi, const CUtensorMap& glo, const CUtensorMap& eg, int C,
                     size_t smem, cudaStream_t stream) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(C) * CS);
    cfg.blockDim = dim3(XG_NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();  // the prologue overlaps the GEMM's tail
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    KTimer kt_(KID_EXPAND_G, stream);
    return cudaLaunchKernelEx(&cfg, expand_g_kernel<CS>, x, ghi, glo, eg) == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

// Features per CTA for cluster size cs: whole 32-column G tiles, at most 256 (one
// 16-byte chunk per lane in the state update, one E tile).
static bool xg_fs_ok(int H, int cs) { return H % (cs * XG_GB) == 0 && H / cs <= 256; }

// Cluster size of the path for these arguments (0: it does not apply) and its
// shared memory.
// Whether the launch also runs S8-S10 (a.fin given and the supertree small enough).
static bool xg_fin(const ExpandArgs& a) {
    return a.fin && a.fin_done && a.B >= 1 && a.B + 1 <= 1024 && a.L * XG_MAXW <= 4096;
}

static int xg_plan(const ExpandArgs& a, size_t* smem) {
    if (a.dtype != DARTREE_BF16 || !a.WqT || !a.Eg || !a.Ghi || !a.Glo) return 0;
    if (reinterpret_cast<uintptr_t>(a.E) % 16 != 0) return 0;  // the root row arrives by a bulk copy
    const int M = a.C * a.L * a.K;
    if (M > a.g_rows || a.K > XG_MAXK || a.K % 8 != 0 || a.W > XG_MAXW) return 0;
    if (!gemm_tc_supported(M, a.H, a.H) || a.H / 8 > GR_MAXV * GR_NT) return 0;
    const int fin_b = xg_fin(a) ? a.B : 0;
    auto need = [&](int cs) { return xg_layout(a.H / cs, a.K, cs, a.L, fin_b).total; };
    if (xg_fs_ok(a.H, 16)) {
        const size_t sm = need(16);
        if (sm <= 227 * 1024 && xg_cluster_ok<16>(sm)) { *smem = sm; return 16; }
    }
    if (xg_fs_ok(a.H, 8)) {
        const size_t sm = need(8);
        if (sm <= 227 * 1024 && xg_cluster_ok<8>(sm)) { *smem = sm; return 8; }
    }
    return 0;
}

bool expand_g_fits(const ExpandArgs& a) {
    size_t smem = 0;
    return xg_plan(a, &smem) != 0;
}

int try_launch_expand_g(const ExpandArgs& a, cudaStream_t stream, bool* launched) {
    *launched = false;
    size_t smem = 0;
    const int cs = xg_plan(a, &smem);
    if (!cs) return DARTREE_OK;
    const int M = a.C * a.L * a.K;
    *launched = true;
    if (!a.eg_ready) {
        {
            KTimer kt_(KID_GATHER, stream);
            gather_rows_kernel<<<(M + GR_ROWS - 1) / GR_ROWS, GR_NT, 0, stream>>>(
                static_cast<const uint16_t*>(a.E), a.cand_tok, a.H, M, a.Eg);
        }
        if (cudaGetLastError() != cudaSuccess) return DARTREE_ECUDA;
    }
    // the GEMM's W_q^T tiles and set-up overlap the previous kernel's tail
    const GemmRowmax grm{static_cast<const uint16_t*>(a.rm_target), a.C * a.L, a.V, a.rm_keys};
    if (int e = launch_gemm_bf16_tc(a.Eg, a.WqT, M, a.H, a.H, 2, nullptr, a.Ghi, 1, a.status, stream, a.Glo, true,
                                    a.rm_target ? &grm : nullptr))
        return e;
    const int fs = a.H / cs;
    CUtensorMap ghi, glo, eg;
    if (!make_tensor_map_bf16(&ghi, a.Ghi, M, a.H, XG_GB, a.K, 64) ||
        !make_tensor_map_bf16(&glo, a.Glo, M, a.H, XG_GB, a.K, 64) ||
        !make_tensor_map_bf16(&eg, a.Eg, M, a.H, fs, a.K, 0))
        return DARTREE_ECUDA;
    XgArgs x{};
    x.E = static_cast<const uint16_t*>(a.E);
    x.hidden = static_cast<const uint16_t*>(a.hidden);
    x.anchor = a.anchor;
    x.cand_tok = a.cand_tok;
    x.cand_val = a.cand_val;
    x.H = a.H;
    x.L = a.L;
    x.K = a.K;
    x.W = a.W;
    x.beta = a.beta;
    x.inv_sqrt_h = 1.0f / sqrtf(float(a.H));
    x.st_tok = a.st_tok;
    x.st_par = a.st_par;
    x.st_s = a.st_s;
    x.st_n = a.st_n;
    x.status = a.status;
    if (xg_fin(a)) {
        x.fin = 1;
        x.B = a.B;
        x.fo = *a.fin;
        *a.fin_done = true;
    }
    return cs == 16 ? xg_launch<16>(x, ghi, glo, eg, a.C, smem, stream) : xg_launch<8>(x, ghi, glo, eg, a.C, smem, stream);
}

}  // namespace dartree
