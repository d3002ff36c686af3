// Tree attention of the verification pass: every drafted token of the pruned tree
// is checked in one target forward pass with a tree-attention mask (DARTree blog
// post, "3.2"). One attention layer over a KV cache:
//   slot j of request c, query head h (key/value head g = h / (Hq / Hkv)) attends to
//   the request's n_ctx cached keys and to the tree slots mask[c, j, :] marks
//   (ancestor-or-self, from S9), with rotary embedding at position n_ctx + pos[c, j]
//   (pos = depth, from S9); scores scaled by 1 / sqrt(D).
//
// Launch 1 (attn_prep_kernel: one CTA per (4 slots of a 128-slot block, request), then
//   one per (request, key/value head)): rotate the tree's queries and keys (angles
//   reduced in double precision), writing Qr [C, Hkv, grp*S, D] (row hg*S + j: the
//   grp query heads of a group stacked) and Kt [C, Hkv, 128, D], and transpose the
//   tree's values, Vtt [C, Hkv, D, 128]; unused and padding slots are zero.
// Launch 2 (attn_kernel, CTA = (chunk of key blocks, 128-row tile of a group's
//   query rows, (request, group))): warp 0 loads, per 128-key block, the keys and
//   transposed values with TMA (128-byte swizzle) into two-stage rings, keys one block
//   ahead of values (a key block is released as soon as its scores are formed);
//   warp 1 issues S = Q K^T into one of two TMEM score buffers and O += P V^T into a
//   TMEM accumulator, both with the A operand (Q, P) in tensor memory so that shared
//   memory serves only the key/value operands and the copies; warps 2-9 (two threads
//   per query row, each on half of the keys and of O) first store the query tile into
//   tensor memory, then per block mask, take the running maximum (log2 domain; O and
//   the sums are rescaled only when the maximum grows by more than 2^8) and write P
//   in bf16 over the block's scores (so P_i V^T runs while block i+1's weights are
//   formed), and at the end either normalise and write the output (one chunk) or
//   write the chunk's partial (O, max, sum).
// Launch 3 (attn_combine_kernel, several chunks only): merges the partials of a row.
// The prefix blocks come first, the tree block (keys = the tree's slots) last.
// Every mbarrier wait is bounded; a wait that runs out records DARTREE_ETIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace dartree {

constexpr int AT_D = 128;        // head dimension
constexpr int AT_BM = 128;       // query rows per tile
constexpr int AT_BN = 128;       // keys per block
constexpr int AT_NT = 320;       // producer, MMA, 8 softmax warps (two per TMEM lane quarter)
constexpr int AT_SMX = 256;      // softmax threads
constexpr int AT_ST = 2;         // stages of the key and of the value ring
constexpr int AT_MAXMT = 3;      // query-row tiles per group (grp * S <= 384)
constexpr float AT_RESCALE = 8.0f;  // log2 growth of the maximum that forces a rescale

// Shared memory holds only the key/value rings (the MMAs' B operands): the query
// tile and the weights P are A operands read from tensor memory.
struct AtSmem {
    static constexpr size_t PANEL = size_t(128) * 64 * 2;  // 128 rows x 64 bf16, swizzled
    static constexpr size_t RING_OFF = 0;                   // AT_ST stages x (K 2 panels, V^T 2 panels), K
                                                            // and V filled and released separately
    static constexpr size_t STAGE = 4 * PANEL;
    static constexpr size_t XCH_OFF = RING_OFF + AT_ST * STAGE;  // float [2 halves][128 rows]
    static constexpr size_t BAR_OFF = XCH_OFF + 2 * 128 * 4;
    // qf, kfull[AT_ST], kempty[AT_ST], vfull[AT_ST], vempty[AT_ST], sfull[2], sfree[2], pfull[2], odone[2]
    static constexpr size_t SLOT_OFF = BAR_OFF + 8 * (1 + 4 * AT_ST + 8);
    static constexpr size_t TOTAL = SLOT_OFF + 16 + 1024;
};
static_assert(AtSmem::TOTAL <= 227 * 1024, "attention tile fits in shared memory");

struct AtArgs {
    int C, S, Hq, Hkv, N, grp, rows;  // rows = grp * S
    int nchunk, per;                  // key blocks per chunk
    const int32_t* n_ctx;
    const uint8_t* mask;              // [C, S, S]
    const int32_t* n_nodes;
    uint16_t* out;                    // [C, S, Hq, D] bf16 (one chunk)
    float* part_o;                    // [C*Hkv, mtiles, nchunk, 128, D]
    float* part_ml;                   // [C*Hkv, mtiles, nchunk, 128, 2]
    int* status;
    const uint16_t* qr;               // [C*Hkv, rows, D] rotated queries (from attn_prep_kernel)
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    return uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(a))) |
           (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(b))) << 16);
}

// ----------------------------------------------------------------------------- prep

// Rotary inverse frequencies theta^(-2i/D), i < D/2, computed once on the host in double.
struct RopeFreq {
    double inv[AT_D / 2];
};

// The rotation, one CTA per (AT_RSLOTS slots of a 128-slot block, request). The slots'
// D/2 rotation angles (position * inv_freq_i, reduced to [-pi, pi] in double; sine and
// cosine in float) go to shared memory, one per thread; then 8 threads per (slot, head
// unit) rotate 8 pairs (i, i + D/2) each with 16-byte loads and stores. Head units: the
// Hq query heads, then the Hkv key heads.
constexpr int AT_PREP_NT = 256;
constexpr int AT_RSLOTS = AT_PREP_NT / (AT_D / 2);  // 4 slots per CTA: one angle per thread

__device__ __forceinline__ void attn_rotate_slots(const uint16_t* __restrict__ q, const uint16_t* __restrict__ kt,
                                                  const int32_t* n_ctx, const int32_t* pos, const int32_t* n_nodes,
                                                  int S, int Hq, int Hkv, const RopeFreq& fr, uint16_t* __restrict__ Qr,
                                                  uint16_t* __restrict__ Kr, int j0, int c, float (*cs)[AT_D / 2],
                                                  float (*sn)[AT_D / 2]) {
    const int grp = Hq / Hkv, half = AT_D / 2;
    const int nn = n_nodes[c];
    {
        const int sl = threadIdx.x / half, i = threadIdx.x % half, j = j0 + sl;
        if (j < S && j < nn) {
            const double p = double(n_ctx[c]) + double(pos[size_t(c) * S + j]);
            const double a = p * fr.inv[i];
            const double k = rint(a * 0.15915494309189535);           // 1 / (2 pi)
            const float r = float(fma(-k, 6.283185307179586, a));    // 2 pi
            sincosf(r, &sn[sl][i], &cs[sl][i]);
        }
    }
    __syncthreads();
    const int t = threadIdx.x & 7, i0 = t * 8;  // pairs i0 .. i0 + 7
    const int units = Hq + Hkv;
    for (int w8 = threadIdx.x >> 3; w8 < AT_RSLOTS * units; w8 += AT_PREP_NT / 8) {
        const int sl = w8 / units, u = w8 - sl * units, j = j0 + sl;
        if (u < Hq && j >= S) continue;  // query rows exist for real slots only
        const bool used = j < S && j < nn;
        const uint16_t* src;
        uint16_t* dst;
        if (u < Hq) {
            const int g = u / grp, hg = u - g * grp;
            src = q + ((size_t(c) * S + j) * Hq + u) * AT_D;
            dst = Qr + ((size_t(c) * Hkv + g) * (size_t(grp) * S) + size_t(hg) * S + j) * AT_D;
        } else {
            const int g = u - Hq;
            src = kt + ((size_t(c) * S + j) * Hkv + g) * AT_D;
            dst = Kr + ((size_t(c) * Hkv + g) * AT_BN + j) * AT_D;
        }
        uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
        if (used) {
            const uint4 x4 = reinterpret_cast<const uint4*>(src + i0)[0];
            const uint4 y4 = reinterpret_cast<const uint4*>(src + half + i0)[0];
            const uint32_t xs[4] = {x4.x, x4.y, x4.z, x4.w}, ys[4] = {y4.x, y4.y, y4.z, y4.w};
            uint32_t ro[4], rh[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                float a2[2], b2[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int i = i0 + 2 * w + e;
                    const float x = bf16_bits_to_float((xs[w] >> (16 * e)) & 0xffffu);
                    const float y = bf16_bits_to_float((ys[w] >> (16 * e)) & 0xffffu);
                    a2[e] = x * cs[sl][i] - y * sn[sl][i];
                    b2[e] = y * cs[sl][i] + x * sn[sl][i];
                }
                ro[w] = pack_bf16x2(a2[0], a2[1]);
                rh[w] = pack_bf16x2(b2[0], b2[1]);
            }
            lo = make_uint4(ro[0], ro[1], ro[2], ro[3]);
            hi = make_uint4(rh[0], rh[1], rh[2], rh[3]);
        }
        reinterpret_cast<uint4*>(dst + i0)[0] = lo;
        reinterpret_cast<uint4*>(dst + half + i0)[0] = hi;
    }
}

// The tree's values transposed, Vtt[c, g, d, j] = v_tree[c, j, g, d] (zero for unused
// and padding slots): one CTA per (request, key/value head), through a shared tile;
// 16-byte loads along d (8 values of one slot) and 16-byte stores along j (8 slots
// of one dimension).
constexpr int AT_VT_PITCH = AT_BN + 8;  // halfwords per tile row (rows stay 16-byte aligned)

__device__ __forceinline__ void attn_transpose_values(const uint16_t* __restrict__ vt, const int32_t* n_nodes, int S,
                                                      int Hkv, uint16_t* __restrict__ Vtt, int cg,
                                                      uint16_t (*tile)[AT_VT_PITCH]) {
    const int c = cg / Hkv, g = cg - c * Hkv;
    const int n = min(S, n_nodes[c]);
    constexpr int DV = AT_D / 8;  // 16-byte vectors per slot
    for (int e = threadIdx.x; e < AT_BN * DV; e += AT_PREP_NT) {  // a warp: 32 slots, one vector each
        const int j = e % AT_BN, d0 = (e / AT_BN) * 8;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (j < n) w = *reinterpret_cast<const uint4*>(vt + ((size_t(c) * S + j) * Hkv + g) * AT_D + d0);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) tile[d0 + q][j] = uint16_t(ws[q >> 1] >> ((q & 1) * 16));
    }
    __syncthreads();
    uint4* dst = reinterpret_cast<uint4*>(Vtt + size_t(cg) * AT_D * AT_BN);
    constexpr int JV = AT_BN / 8;  // 16-byte vectors per transposed row
    for (int e = threadIdx.x; e < AT_D * JV; e += AT_PREP_NT) {
        const int d = e / JV, j0 = (e - d * JV) * 8;
        dst[e] = *reinterpret_cast<const uint4*>(&tile[d][j0]);
    }
}

// One launch for both: the first (128 / AT_RSLOTS) C CTAs rotate AT_RSLOTS slots of a
// request each, the next C * Hkv CTAs transpose the values of one (request, key/value head).
__global__ void __launch_bounds__(AT_PREP_NT) attn_prep_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ kt, const uint16_t* __restrict__ v, const int32_t* n_ctx,
    const int32_t* pos, const int32_t* n_nodes, int C, int S, int Hq, int Hkv, const __grid_constant__ RopeFreq fr,
    uint16_t* __restrict__ Qr, uint16_t* __restrict__ Kr, uint16_t* __restrict__ Vtt) {
    __shared__ __align__(16) uint16_t tile[AT_D][AT_VT_PITCH];       // [d][j]: the transpose's tile
    __shared__ float cs[AT_RSLOTS][AT_D / 2], sn[AT_RSLOTS][AT_D / 2];  // the rotation's angles
    constexpr int PER = AT_BN / AT_RSLOTS;  // rotation CTAs per request
    const int b = int(blockIdx.x), nrot = PER * C;
    if (b < nrot)
        attn_rotate_slots(q, kt, n_ctx, pos, n_nodes, S, Hq, Hkv, fr, Qr, Kr, (b % PER) * AT_RSLOTS, b / PER, cs, sn);
    else
        attn_transpose_values(v, n_nodes, S, Hkv, Vtt, b - nrot, tile);
}

// ----------------------------------------------------------------------------- attention

__global__ void __launch_bounds__(AT_NT, 1) attn_kernel(const __grid_constant__ CUtensorMap tmK,
                                                        const __grid_constant__ CUtensorMap tmVt,
                                                        const __grid_constant__ CUtensorMap tmKt,
                                                        const __grid_constant__ CUtensorMap tmVtt, AtArgs a) {
    using L = AtSmem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
    uint64_t* qf = bars;                     // the query tile is in tensor memory
    uint64_t* kfull = bars + 1;              // [AT_ST]: key block landed, by stage
    uint64_t* kempty = kfull + AT_ST;        // [AT_ST]: S = Q K^T done with it
    uint64_t* vfull = kempty + AT_ST;        // [AT_ST]: value block landed
    uint64_t* vempty = vfull + AT_ST;        // [AT_ST]: P V^T done with it
    uint64_t* sfull = vempty + AT_ST;        // [2]: S written, by TMEM score buffer
    uint64_t* sfree = sfull + 2;
    uint64_t* pfull = sfree + 2;             // [2]: P written, by P buffer
    uint64_t* odone = pfull + 2;             // [2]: P V^T done, by P buffer
    uint32_t* slot = reinterpret_cast<uint32_t*>(smem + L::SLOT_OFF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunk = blockIdx.x, mt = blockIdx.y, cg = blockIdx.z;
    const int c = cg / a.Hkv, g = cg - c * a.Hkv;
    const int nctx = min(max(a.n_ctx[c], 0), a.N);
    const int nbp = (nctx + AT_BN - 1) / AT_BN;  // prefix blocks; block nbp = the tree
    const int b0 = chunk * a.per, b1 = min(nbp + 1, b0 + a.per);
    const int nblk = b1 > b0 ? b1 - b0 : 0;

    if (threadIdx.x == 0) {
        mbar_init(qf, AT_SMX / 32);
        for (int s = 0; s < AT_ST; ++s) {
            mbar_init(&kfull[s], 1);
            mbar_init(&kempty[s], 1);
            mbar_init(&vfull[s], 1);
            mbar_init(&vempty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sfull[s], 1);
            mbar_init(&sfree[s], AT_SMX / 32);
            mbar_init(&pfull[s], AT_SMX / 32);
            mbar_init(&odone[s], 1);
        }
        fence_mbar_init();
    }
    if (warp == 1) tc::tmem_alloc(slot, 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // TMEM columns: S buffers at 0 and 128 (P_i overwrites S_i in place: the 64 keys of
    // half h as 32 packed bf16 pairs at 128 s + 64 h), O at 256, Q at 384 (d pairs)
    const uint32_t tmem = *slot;
    griddep_launch_dependents();
    griddep_wait();

    if (warp == 0) {
        if (lane == 0 && nblk > 0) {  // producer
            // key blocks run AT_ST - 1 ahead of value blocks: K_i+AT_ST-1 needs only S_i-1
            // done, V_i needs P_i-AT_ST V^T done
            auto load_k = [&](int i) -> bool {
                const int s = i % AT_ST, b = b0 + i;
                if (i >= AT_ST && !mbar_wait_bounded(&kempty[s], uint32_t((i / AT_ST) & 1) ^ 1u, a.status))
                    return false;
                uint8_t* st = smem + L::RING_OFF + size_t(s) * L::STAGE;
                mbar_arrive_expect_tx(&kfull[s], uint32_t(2 * L::PANEL));
                if (b < nbp) {  // prefix block: K_cache rows
                    const int kr = cg * a.N + b * AT_BN;
                    tc::tma_load_2d(st, &tmK, 0, kr, &kfull[s]);
                    tc::tma_load_2d(st + L::PANEL, &tmK, 64, kr, &kfull[s]);
                } else {        // the tree block
                    tc::tma_load_2d(st, &tmKt, 0, cg * AT_BN, &kfull[s]);
                    tc::tma_load_2d(st + L::PANEL, &tmKt, 64, cg * AT_BN, &kfull[s]);
                }
                return true;
            };
            auto load_v = [&](int i) -> bool {
                const int s = i % AT_ST, b = b0 + i;
                if (i >= AT_ST && !mbar_wait_bounded(&vempty[s], uint32_t((i / AT_ST) & 1) ^ 1u, a.status))
                    return false;
                uint8_t* st = smem + L::RING_OFF + size_t(s) * L::STAGE + 2 * L::PANEL;
                mbar_arrive_expect_tx(&vfull[s], uint32_t(2 * L::PANEL));
                if (b < nbp) {  // V^T_cache columns
                    tc::tma_load_2d(st, &tmVt, b * AT_BN, cg * AT_D, &vfull[s]);
                    tc::tma_load_2d(st + L::PANEL, &tmVt, b * AT_BN + 64, cg * AT_D, &vfull[s]);
                } else {
                    tc::tma_load_2d(st, &tmVtt, 0, cg * AT_D, &vfull[s]);
                    tc::tma_load_2d(st + L::PANEL, &tmVtt, 64, cg * AT_D, &vfull[s]);
                }
                return true;
            };
            constexpr int lead = AT_ST - 1;
            int nk = 0, nv = 0;  // blocks issued
            bool ok = true;
            for (int i = 0; i < lead && i < nblk && ok; ++i) {
                ok = load_k(i);
                if (ok) nk = i + 1;
            }
            for (int i = 0; i < nblk && ok; ++i) {
                if (i + lead < nblk) {
                    ok = load_k(i + lead);
                    if (ok) nk = i + lead + 1;
                }
                if (ok) {
                    ok = load_v(i);
                    if (ok) nv = i + 1;
                }
            }
            // copies issued and not yet seen complete land before the CTA can exit
            for (int q = nk - 1; q >= 0 && q >= nk - AT_ST; --q)
                mbar_wait_bounded(&kfull[q % AT_ST], uint32_t(q / AT_ST) & 1u, a.status);
            for (int q = nv - 1; q >= 0 && q >= nv - AT_ST; --q)
                mbar_wait_bounded(&vfull[q % AT_ST], uint32_t(q / AT_ST) & 1u, a.status);
        }
    } else if (warp == 1) {
        if (lane == 0 && nblk > 0) {  // MMA issuer
            constexpr uint32_t idesc = tc::idesc_bf16_f32(AT_BM, AT_BN);
            bool ok = mbar_wait_bounded(qf, 0, a.status);
            auto pv = [&](int i) -> bool {  // O += P_i V_i^T, then release stage i
                if (!mbar_wait_bounded(&pfull[i & 1], uint32_t(i >> 1) & 1u, a.status) ||
                    !mbar_wait_bounded(&vfull[i % AT_ST], uint32_t(i / AT_ST) & 1u, a.status))
                    return false;
                tc::fence_after_sync();
                const uint32_t st = smem_u32(smem + L::RING_OFF + size_t(i % AT_ST) * L::STAGE);
                const uint32_t ta = tmem + uint32_t((i & 1) * AT_BN);  // P_i, keys 64 p + 16 kk at 64 p + 8 kk
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const uint64_t db = tc::desc_sw128_kmajor(st + uint32_t((2 + p) * L::PANEL));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_bf16_ts(tmem + 256, ta + uint32_t(64 * p + 8 * kk), db + 2u * kk, idesc,
                                        i > 0 || p > 0 || kk > 0);
                }
                tc::mma_commit(&odone[i & 1]);
                tc::mma_commit(&vempty[i % AT_ST]);
                return true;
            };
            for (int i = 0; i < nblk && ok; ++i) {
                const int s = i & 1;
                if (i >= 2 && !mbar_wait_bounded(&sfree[s], uint32_t((i >> 1) - 1) & 1u, a.status)) break;
                if (!mbar_wait_bounded(&kfull[i % AT_ST], uint32_t(i / AT_ST) & 1u, a.status)) break;
                tc::fence_after_sync();
                const uint32_t st = smem_u32(smem + L::RING_OFF + size_t(i % AT_ST) * L::STAGE);
#pragma unroll
                for (int p = 0; p < 2; ++p) {  // S_i = Q K_i^T over the two 64-wide d panels
                    const uint64_t db = tc::desc_sw128_kmajor(st + uint32_t(p * L::PANEL));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_bf16_ts(tmem + uint32_t(s * AT_BN), tmem + 384u + uint32_t(32 * p + 8 * kk),
                                        db + 2u * kk, idesc, p > 0 || kk > 0);
                }
                tc::mma_commit(&sfull[s]);
                tc::mma_commit(&kempty[i % AT_ST]);
                if (i >= 1 && !pv(i - 1)) {
                    ok = false;
                    break;
                }
            }
            if (ok) pv(nblk - 1);
        }
    } else {
        // softmax warps 2..9: one query row per pair of threads (TMEM lane = row in the
        // tile); `half` takes keys [64 half, 64 half + 64) of every block and the same
        // columns of O. The halves agree on the running maximum through shared memory.
        const int quarter = warp & 3, half = (warp - 2) >> 2;
        const int rt = quarter * 32 + lane;                 // row in the tile
        const int R = mt * AT_BM + rt;                      // row in the group
        const bool real = R < a.rows;
        const int hg = real ? R / a.S : 0, j = real ? R - hg * a.S : 0;
        const int nn = a.n_nodes[c];
        const bool live = real && j < nn;
        // a warp whose 32 rows are all padding (the last tile of a group) forms no
        // weights: its rows of P are never read into a real output row
        const bool warp_real = __any_sync(0xffffffffu, real);
        const uint32_t trow = tmem + (uint32_t(quarter * 32) << 16);
        const uint32_t col0 = uint32_t(half * 64);          // this thread's key / O columns
        const float sl2 = 1.4426950408889634f / sqrtf(float(AT_D));  // log2(e) / sqrt(D)
        float* xch = reinterpret_cast<float*>(smem + L::XCH_OFF);
        auto ex2 = [](float x) {
            float y;
            asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
            return y;
        };
        // this thread's half of its query row (d in [64 half, 64 half + 64)) into TMEM
        {
            uint32_t v[32];
            const uint4* src = reinterpret_cast<const uint4*>(a.qr + (size_t(cg) * a.rows + R) * AT_D + col0);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint4 x = real ? src[q] : make_uint4(0, 0, 0, 0);
                v[4 * q] = x.x;
                v[4 * q + 1] = x.y;
                v[4 * q + 2] = x.z;
                v[4 * q + 3] = x.w;
            }
            tc::tmem_st32(trow + 384u + uint32_t(32 * half), v);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(qf);
        }
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int i = 0; i < nblk; ++i) {
            const int s = i & 1, b = b0 + i;
            ok = ok && __all_sync(0xffffffffu, mbar_wait_bounded(&sfull[s], uint32_t(i >> 1) & 1u, a.status));
            // visibility of this thread's 64 keys as a bit mask
            uint64_t vis = 0;
            if (live) {
                if (b < nbp) {
                    const int nv = min(max(nctx - b * AT_BN - int(col0), 0), 64);
                    vis = nv >= 64 ? ~0ull : ((1ull << nv) - 1ull);
                } else {
                    const uint8_t* mrow = a.mask + (size_t(c) * a.S + j) * a.S + col0;
                    const int nv = min(max(a.S - int(col0), 0), 64);
                    for (int q = 0; q < nv; ++q) vis |= uint64_t(mrow[q] != 0) << q;
                }
            }
            // pass 1: this half's maximum of the raw scores over the visible keys
            float mx = -INFINITY;
            if (ok && warp_real) {
                tc::fence_after_sync();
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 32) {
                    uint32_t v[32];
                    tc::tmem_ld32(trow + uint32_t(s * AT_BN) + col0 + uint32_t(c0), v);
                    const uint32_t bits = uint32_t(vis >> c0);
#pragma unroll
                    for (int e = 0; e < 32; ++e) mx = fmaxf(mx, (bits >> e) & 1u ? __uint_as_float(v[e]) : -INFINITY);
                }
            }
            xch[half * 128 + rt] = mx;  // (the second barrier: read before the next block writes)
            asm volatile("bar.sync 2, %0;" :: "n"(AT_SMX) : "memory");
            mx = fmaxf(mx, xch[(half ^ 1) * 128 + rt]);
            asm volatile("bar.sync 2, %0;" :: "n"(AT_SMX) : "memory");
            mx = mx > -INFINITY ? mx * sl2 : mx;
            // a new running maximum (beyond the slack) rescales O and the sums; that
            // needs the previous P V^T complete. TMEM accesses are warp-wide: lanes
            // without a new maximum scale by 1.
            const bool grow = ok && mx > m_used + AT_RESCALE;
            const float f = grow && m_used > -INFINITY ? exp2f(m_used - mx) : 1.0f;
            if (i >= 1 && warp_real && __any_sync(0xffffffffu, grow && m_used > -INFINITY)) {
                ok = ok && __all_sync(0xffffffffu, mbar_wait_bounded(&odone[(i - 1) & 1], uint32_t((i - 1) >> 1) & 1u,
                                                                     a.status));
                if (ok) {
                    tc::fence_after_sync();
#pragma unroll 1
                    for (int c0 = 0; c0 < 64; c0 += 32) {
                        uint32_t v[32];
                        tc::tmem_ld32(trow + 256u + col0 + uint32_t(c0), v);
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * f);
                        tc::tmem_st32(trow + 256u + col0 + uint32_t(c0), v);
                    }
                }
            }
            if (grow) {
                l *= f;
                m_used = mx;
            }
            // pass 2: P = 2^(s sl2 - m) in bf16 over S_i's first 32 columns of this half
            // (the chunk read before its packed weights are stored); the sum of the
            // unrounded weights. P_i-2 V^T, which read this buffer, ran before S_i.
            if (ok && warp_real) {
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 32) {
                    uint32_t v[32];
                    tc::tmem_ld32(trow + uint32_t(s * AT_BN) + col0 + uint32_t(c0), v);
                    const uint32_t bits = uint32_t(vis >> c0);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float p0 = (bits >> e) & 1u ? ex2(fmaf(__uint_as_float(v[e]), sl2, -m_used)) : 0.f;
                        const float p1 =
                            (bits >> (e + 1)) & 1u ? ex2(fmaf(__uint_as_float(v[e + 1]), sl2, -m_used)) : 0.f;
                        l += p0 + p1;
                        const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                        pk[e / 2] = *reinterpret_cast<const uint32_t*>(&h2);
                    }
                    tc::tmem_st16_async(trow + uint32_t(s * AT_BN) + col0 + uint32_t(c0 / 2), pk);
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
            }
            __syncwarp();
            if (lane == 0 && ok) {
                mbar_arrive(&sfree[s]);
                mbar_arrive(&pfull[s]);
            }
        }
        // the row's total sum: both halves
        xch[half * 128 + rt] = l;
        asm volatile("bar.sync 2, %0;" :: "n"(AT_SMX) : "memory");
        l += xch[(half ^ 1) * 128 + rt];
        // the last block's P V^T, then the row out (this half's 64 columns)
        if (nblk > 0)
            ok = ok && __all_sync(0xffffffffu, mbar_wait_bounded(&odone[(nblk - 1) & 1], uint32_t((nblk - 1) >> 1) & 1u,
                                                                 a.status));
        const bool has = ok && nblk > 0 && l > 0.f;
        if (ok && nblk > 0) tc::fence_after_sync();
        const int h = g * a.grp + hg;
        if (a.nchunk == 1) {  // (TMEM loads warp-wide; padding rows load and drop)
            uint4* dst = reinterpret_cast<uint4*>(a.out + ((size_t(c) * a.S + j) * a.Hq + h) * AT_D + col0);
            const float inv = has ? 1.0f / l : 0.f;
#pragma unroll 1
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t v[32];
                if (ok && nblk > 0) tc::tmem_ld32(trow + 256u + col0 + uint32_t(c0), v);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = has && live ? pack_bf16x2(__uint_as_float(v[2 * e]) * inv, __uint_as_float(v[2 * e + 1]) * inv)
                                        : 0u;
                if (real)
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dst[c0 / 8 + q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
        } else {
            // (padding rows are never combined: nothing is written for them)
            const size_t pr = ((size_t(cg) * gridDim.y + mt) * a.nchunk + chunk) * AT_BM + rt;
            float4* dst = reinterpret_cast<float4*>(a.part_o + pr * AT_D + col0);
#pragma unroll 1
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t v[32];
                if (ok && nblk > 0) tc::tmem_ld32(trow + 256u + col0 + uint32_t(c0), v);
                if (real)
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        dst[c0 / 4 + q] = has ? make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                            __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]))
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (half == 0 && real) {
                a.part_ml[pr * 2] = has ? m_used : -INFINITY;
                a.part_ml[pr * 2 + 1] = has ? l : 0.f;
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

// ----------------------------------------------------------------------------- combine

// One warp per (request, group, tile row): merge the chunks' partials and write
// the row's output (bf16), zero for padding-free unused slots.
__global__ void __launch_bounds__(256) attn_combine_kernel(AtArgs a, int mtiles) {
    const int w = int(blockIdx.x) * 8 + int(threadIdx.x >> 5), lane = threadIdx.x & 31;
    const int total = a.C * a.Hkv * mtiles * AT_BM;
    griddep_wait();
    if (w >= total) return;
    const int rt = w % AT_BM, mt = (w / AT_BM) % mtiles, cg = w / (AT_BM * mtiles);
    const int R = mt * AT_BM + rt;
    if (R >= a.rows) return;
    const int c = cg / a.Hkv, g = cg - c * a.Hkv;
    const int hg = R / a.S, j = R - hg * a.S, h = g * a.grp + hg;
    const bool live = j < a.n_nodes[c];
    const size_t pr0 = (size_t(cg) * mtiles + mt) * a.nchunk * AT_BM + rt;  // chunk k: pr0 + k * AT_BM
    // the chunks' (max, sum) pairs, lane k taking chunks k, k + 32, ... (independent loads)
    float mloc = -INFINITY;
    for (int k = lane; k < a.nchunk; k += 32) {
        const float2 ml = reinterpret_cast<const float2*>(a.part_ml)[pr0 + size_t(k) * AT_BM];
        if (ml.y > 0.f) mloc = fmaxf(mloc, ml.x);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
    const float mmax = mloc;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lsum = 0.f;
    if (live && mmax > -INFINITY)
        for (int k0 = 0; k0 < a.nchunk; k0 += 32) {
            // lane t: chunk k0 + t's weight 2^(m - mmax) (0 for an empty chunk)
            float fk = 0.f;
            if (k0 + lane < a.nchunk) {
                const float2 ml = reinterpret_cast<const float2*>(a.part_ml)[pr0 + size_t(k0 + lane) * AT_BM];
                if (ml.y > 0.f) {
                    fk = exp2f(ml.x - mmax);
                    lsum += fk * ml.y;
                }
            }
            const int nk = min(32, a.nchunk - k0);
            // the chunks' rows of O, eight loads in flight
            for (int t0 = 0; t0 < nk; t0 += 8) {
                float4 o[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (t0 + u < nk)
                        o[u] = reinterpret_cast<const float4*>(a.part_o + (pr0 + size_t(k0 + t0 + u) * AT_BM) * AT_D)[lane];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float f = __shfl_sync(0xffffffffu, fk, (t0 + u) & 31);
                    if (t0 + u < nk && f > 0.f) {
                        acc.x += f * o[u].x;
                        acc.y += f * o[u].y;
                        acc.z += f * o[u].z;
                        acc.w += f * o[u].w;
                    }
                }
            }
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
    uint2 pk = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    reinterpret_cast<uint2*>(a.out + ((size_t(c) * a.S + j) * a.Hq + h) * AT_D)[lane] = pk;
}

// ----------------------------------------------------------------------------- host

bool attn_supported(int C, int S, int Hq, int Hkv, int D, int N) {
    return C >= 0 && S >= 1 && S <= AT_BN && Hkv >= 1 && Hq >= Hkv && Hq % Hkv == 0 && D == AT_D && N >= 0 &&
           N % 8 == 0 && (Hq / Hkv) * S <= AT_MAXMT * AT_BM;
}

static int attn_mtiles(int S, int grp) { return (grp * S + AT_BM - 1) / AT_BM; }

AttnPlan attn_plan(int C, int S, int Hq, int Hkv, int N) {
    AttnPlan p{};
    const int grp = Hq / Hkv, mt = attn_mtiles(S, grp);
    const int blocks = (N + AT_BN - 1) / AT_BN + 1;  // most prefix blocks + the tree block
    const long base = long(C) * Hkv * mt;
    // as many chunks of a tile's key blocks as one wave of CTAs holds (one per SM):
    // a second, partial wave costs a CTA's fixed prologue and epilogue again
    int want = base > 0 ? int(long(num_sms()) / base) : 1;
    if (want < 1) want = 1;
    if (want > blocks) want = blocks;
    p.per = (blocks + want - 1) / want;
    p.nchunk = (blocks + p.per - 1) / p.per;
    p.mtiles = mt;
    size_t off = 256;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += (bytes + 255) / 256 * 256;
        return o;
    };
    p.qr = take(size_t(C) * Hkv * grp * S * AT_D * 2);
    p.kt = take(size_t(C) * Hkv * AT_BN * AT_D * 2);
    p.vtt = take(size_t(C) * Hkv * AT_D * AT_BN * 2);
    if (p.nchunk > 1) {
        p.part_o = take(size_t(C) * Hkv * mt * p.nchunk * AT_BM * AT_D * 4);
        p.part_ml = take(size_t(C) * Hkv * mt * p.nchunk * AT_BM * 2 * 4);
    }
    p.total = off;
    return p;
}

int launch_tree_attention(int C, int S, int Hq, int Hkv, int N, double theta, const void* q, const void* k_tree,
                          const void* v_tree, const void* k_cache, const void* vt_cache, const int32_t* n_ctx,
                          const uint8_t* mask, const int32_t* pos, const int32_t* n_nodes, void* out, void* ws,
                          const AttnPlan& pl, cudaStream_t stream) {
    if (C == 0) return DARTREE_OK;
    uint8_t* w = static_cast<uint8_t*>(ws);
    int* status = reinterpret_cast<int*>(w);
    uint16_t* Qr = reinterpret_cast<uint16_t*>(w + pl.qr);
    uint16_t* Kt = reinterpret_cast<uint16_t*>(w + pl.kt);
    uint16_t* Vtt = reinterpret_cast<uint16_t*>(w + pl.vtt);
    const int grp = Hq / Hkv;
    RopeFreq fr;
    for (int i = 0; i < AT_D / 2; ++i) fr.inv[i] = pow(theta, -2.0 * double(i) / double(AT_D));
    {
        KTimer kt_(KID_ATTN_PREP, stream);
        attn_prep_kernel<<<(AT_BN / AT_RSLOTS) * C + C * Hkv, AT_PREP_NT, 0, stream>>>(
            static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k_tree), static_cast<const uint16_t*>(v_tree),
            n_ctx, pos, n_nodes, C, S, Hq, Hkv, fr, Qr, Kt, Vtt);
    }
    if (cudaGetLastError() != cudaSuccess) return DARTREE_ECUDA;
    CUtensorMap tk, tvt, tkt, tvtt;
    const int rows = grp * S;
    // an empty cache (N = 0) still needs valid maps: point them at the tree block
    const bool cache = N > 0;
    if (!make_tensor_map_bf16(&tk, cache ? k_cache : Kt, cache ? C * Hkv * N : C * Hkv * AT_BN, AT_D, 64, AT_BN,
                              128) ||
        !make_tensor_map_bf16(&tvt, cache ? vt_cache : Vtt, C * Hkv * AT_D, cache ? N : AT_BN, 64, AT_D, 128) ||
        !make_tensor_map_bf16(&tkt, Kt, C * Hkv * AT_BN, AT_D, 64, AT_BN, 128) ||
        !make_tensor_map_bf16(&tvtt, Vtt, C * Hkv * AT_D, AT_BN, 64, AT_D, 128))
        return DARTREE_ECUDA;
    AtArgs a{C, S, Hq, Hkv, N, grp, rows, pl.nchunk, pl.per, n_ctx, mask, n_nodes, static_cast<uint16_t*>(out),
             pl.nchunk > 1 ? reinterpret_cast<float*>(w + pl.part_o) : nullptr,
             pl.nchunk > 1 ? reinterpret_cast<float*>(w + pl.part_ml) : nullptr, status, Qr};
    const size_t smem = AtSmem::TOTAL;
    if (cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
        return DARTREE_ECUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(pl.nchunk, pl.mtiles, C * Hkv);
    cfg.blockDim = dim3(AT_NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    {
        KTimer kt_(KID_ATTN, stream);
        e = cudaLaunchKernelEx(&cfg, attn_kernel, tk, tvt, tkt, tvtt, a);
    }
    if (e != cudaSuccess) return DARTREE_ECUDA;
    if (pl.nchunk > 1) {
        const int warps = C * Hkv * pl.mtiles * AT_BM;
        cudaLaunchConfig_t c2{};
        c2.gridDim = dim3((warps + 7) / 8);
        c2.blockDim = dim3(256);
        c2.stream = stream;
        c2.attrs = attr;
        c2.numAttrs = 1;
        {
            KTimer kt_(KID_ATTN_COMBINE, stream);
            e = cudaLaunchKernelEx(&c2, attn_combine_kernel, a, pl.mtiles);
        }
        if (e != cudaSuccess) return DARTREE_ECUDA;
    }
    return DARTREE_OK;
}

}  // namespace dartree
