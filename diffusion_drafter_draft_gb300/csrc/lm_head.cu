// The block drafter's LM head fused with S1 (candidate generation, DARTree blog
// post 3.1: keep the top-K tokens of every block position's base logits): the
// base logits L[r, v] = <h_r, W_lm[v]> are formed on the tensor cores and reduced
// to per-row candidates on chip, so they never reach global memory.
//
// Launch 1 (lmhead_topk_kernel<NR>, one CTA per SM): CTA b owns a contiguous run of
// 128-row tiles of W_lm [V, H]. Warp 0's elected thread streams each tile's 64-wide
// k blocks (W_lm 128 x 64 and the NR hidden rows x 64, 128-byte swizzle) with TMA
// into a ring; warp 1's elected thread issues tcgen05.mma (M = 128 vocabulary rows,
// N = NR hidden rows) into one of two TMEM accumulators; warps 2-5 read the other
// accumulator (one vocabulary row per thread, NR logits) while the next tile
// streams, and append to row r's candidate buffer every key
// (ord(logit) << 32 | ~token) above the row's current threshold. A buffer that
// could overflow with the next tile is sorted and cut to its K best first (the
// threshold becomes its K-th key; the cut is a radix selection in registers). At
// the end each row's buffer is cut to its K best, sorted and written out: K keys
// per (row, CTA), largest first.
// Launch 2 (lmhead_merge_kernel, one CTA per row): the K largest keys among the
// row's CTA lists, sorted, written as (token, logit). Only keys at or above the
// K-th largest list maximum can qualify; when those are few they are sorted
// directly, else a radix selection over all the lists runs.
// Keys are distinct (the token is in the low bits), so the result is the exact
// top-K of the fp32 logits under (logit desc, token asc).
// Every mbarrier wait is bounded; a wait that runs out records DARTREE_ETIMEOUT.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace dartree {

constexpr int LM_BM = 128, LM_BK = 64;
constexpr int LM_NT = 192;          // 6 warps: producer, MMA, 4 x epilogue
constexpr int LM_CAP = 256;         // candidate buffer per row (>= K + 128)
constexpr int LM_MAXK = LM_CAP - LM_BM;
constexpr int LM_MAXROWS = 64;      // hidden rows per pass over W_lm

template <int NR>
struct LmSmem {
    static constexpr size_t A_BYTES = size_t(LM_BM) * LM_BK * 2;
    static constexpr size_t B_BYTES = size_t(NR) * LM_BK * 2;
    static constexpr size_t STAGE = A_BYTES + B_BYTES;  // a multiple of 1024
    static constexpr size_t CAND = size_t(NR) * LM_CAP * 8;
    static constexpr int STAGES_FIT = int((200 * 1024 - CAND) / STAGE);
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr size_t CAND_OFF = STAGE * STAGES;
    static constexpr size_t THR_OFF = CAND_OFF + CAND;           // u64 [NR]
    static constexpr size_t CNT_OFF = THR_OFF + size_t(NR) * 8;  // int [NR]
    static constexpr size_t HIST_OFF = CNT_OFF + size_t(NR) * 4 + 8;  // (+ error flag) u32 [4][256]
    static constexpr size_t BAR_OFF = HIST_OFF + 4 * 256 * 4;          // full[S], empty[S], accf[2], acce[2]
    static constexpr size_t SLOT_OFF = BAR_OFF + 8 * (2 * STAGES + 4);
    static constexpr size_t TOTAL = SLOT_OFF + 16 + 1024;        // + alignment slack
    static constexpr uint32_t TMEM_COLS = 2 * NR < 32 ? 32 : 2 * NR;
    static_assert(STAGES >= 2, "ring of at least two stages");
    static_assert(STAGE % 1024 == 0, "stages keep the swizzle atoms aligned");
};

struct LmArgs {
    int r0;          // first hidden row of this pass
    int R;           // hidden rows of this pass (<= NR)
    int V, H, K;
    int tiles;       // ceil(V / 128)
    unsigned long long* part;  // [R, gridDim.x, K] keys
    int* status;
};

// In-place descending bitonic sort of n (a power of two, <= LM_CAP) keys in shared
// memory by one warp.
__device__ __forceinline__ void warp_sort_desc(uint64_t* s, int n) {
    const int lane = threadIdx.x & 31;
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int t = lane; t < n / 2; t += 32) {
                const int i = 2 * t - (t & (j - 1)), l = i + j;  // i: t with a zero bit inserted at j
                const uint64_t a = s[i], b = s[l];
                const bool desc = (i & k) == 0;
                if ((a < b) == desc) {
                    s[i] = b;
                    s[l] = a;
                }
            }
            __syncwarp();
        }
    }
}

// Cut row r's buffer (cnt <= LM_CAP distinct keys) to its K largest keys, in any
// order, by one warp: radix selection 8 bits at a time from the top, in registers
// (LM_CAP / 32 keys per lane) with a 256-bin histogram in shared memory. The
// selection stops at the first digit whose bin holds exactly the keys still
// needed; the threshold becomes the smallest kept key.
__device__ __forceinline__ void cut_row(uint64_t* buf, int* cnt, uint64_t* thr, int K, uint32_t* hist) {
    constexpr int PER = LM_CAP / 32;
    const int lane = threadIdx.x & 31;
    const int n = *cnt;
    if (n <= K) {  // nothing to drop; the threshold stays (0 while the row holds fewer than K)
        if (lane == 0 && n == K) {
            uint64_t m = ~0ull;
            for (int i = 0; i < n; ++i) m = buf[i] < m ? buf[i] : m;
            *thr = m;
        }
        __syncwarp();
        return;
    }
    uint64_t k[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) k[j] = lane + 32 * j < n ? buf[lane + 32 * j] : 0ull;
    uint64_t prefix = 0, pmask = 0;
    uint32_t need = uint32_t(K);
    for (int shift = 56; shift >= 0; shift -= 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j) hist[lane * 8 + j] = 0;
        __syncwarp();
#pragma unroll
        for (int j = 0; j < PER; ++j)
            if (lane + 32 * j < n && (k[j] & pmask) == prefix) atomicAdd(&hist[(k[j] >> shift) & 0xffu], 1u);
        __syncwarp();
        uint32_t c[8], tot = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {  // this lane's digits, descending: 255 - 8 lane - j
            c[j] = hist[255 - 8 * lane - j];
            tot += c[j];
        }
        uint32_t incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        uint32_t run = incl - tot, digit = 0, left = 0, inbin = 0;
        const bool mine = run < need && incl >= need;
        if (mine) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (run + c[j] >= need) {
                    digit = uint32_t(255 - 8 * lane - j);
                    left = need - run;
                    inbin = c[j];
                    break;
                }
                run += c[j];
            }
        }
        const int src = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
        digit = __shfl_sync(0xffffffffu, digit, src < 0 ? 0 : src);
        left = __shfl_sync(0xffffffffu, left, src < 0 ? 0 : src);
        inbin = __shfl_sync(0xffffffffu, inbin, src < 0 ? 0 : src);
        __syncwarp();
        prefix |= uint64_t(digit) << shift;
        pmask |= uint64_t(0xffu) << shift;
        need = left;
        if (src < 0 || inbin == left) break;  // every key of this bin is kept
    }
    // keep the keys at or above the prefix: exactly K (keys distinct)
    uint32_t base = 0;
    uint64_t mn = ~0ull;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const bool keep = lane + 32 * j < n && (k[j] & pmask) >= prefix;
        const uint32_t m = __ballot_sync(0xffffffffu, keep);
        const uint32_t at = base + __popc(m & ((1u << lane) - 1u));
        if (keep && at < uint32_t(LM_CAP)) {
            buf[at] = k[j];
            mn = k[j] < mn ? k[j] : mn;
        }
        base += __popc(m);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t y = __shfl_xor_sync(0xffffffffu, mn, o);
        mn = y < mn ? y : mn;
    }
    if (lane == 0) {
        *cnt = int(base < uint32_t(K) ? base : uint32_t(K));
        *thr = mn;
    }
    __syncwarp();
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

template <int NR>
__global__ void __launch_bounds__(LM_NT, 1) lmhead_topk_kernel(const __grid_constant__ CUtensorMap tmW,
                                                               const __grid_constant__ CUtensorMap tmH, LmArgs a) {
    using S = LmSmem<NR>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* cand = reinterpret_cast<uint64_t*>(smem + S::CAND_OFF);
    uint64_t* thr = reinterpret_cast<uint64_t*>(smem + S::THR_OFF);
    int* cnt = reinterpret_cast<int*>(smem + S::CNT_OFF);
    uint32_t* hists = reinterpret_cast<uint32_t*>(smem + S::HIST_OFF);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF);
    uint64_t* empty = full + S::STAGES;
    uint64_t* accf = empty + S::STAGES;
    uint64_t* acce = accf + 2;
    uint32_t* slot = reinterpret_cast<uint32_t*>(smem + S::SLOT_OFF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // this CTA's tiles: a contiguous run, the first `rem` CTAs one longer
    const int G = int(gridDim.x), b = int(blockIdx.x);
    const int per = a.tiles / G, rem = a.tiles % G;
    const int t0 = b * per + (b < rem ? b : rem);
    const int nt = per + (b < rem ? 1 : 0);
    const int nk = a.H / LM_BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(&accf[q], 1);
            mbar_init(&acce[q], 4);
        }
        fence_mbar_init();
    }
    for (int r = threadIdx.x; r <= NR; r += LM_NT) {
        cnt[r] = 0;  // cnt[NR]: the epilogue's error flag
        if (r < NR) thr[r] = 0ull;
    }
    if (warp == 1) tc::tmem_alloc(slot, S::TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *slot;
    griddep_launch_dependents();
    griddep_wait();  // the hidden rows may come from the launch before

    if (warp == 0) {
        if (lane == 0) {  // producer: TMA ring over (tile, k block)
            int step = 0;
            bool ok = true;
            for (int i = 0; i < nt && ok; ++i) {
                const int tile = t0 + i;
                for (int kb = 0; kb < nk; ++kb, ++step) {
                    const int s = step % S::STAGES;
                    const uint32_t ph = uint32_t(step / S::STAGES) & 1u;
                    if (step >= S::STAGES && !mbar_wait_bounded(&empty[s], ph ^ 1u, a.status)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + size_t(s) * S::STAGE;
                    mbar_arrive_expect_tx(&full[s], uint32_t(S::STAGE));
                    tc::tma_load_2d(st, &tmW, kb * LM_BK, tile * LM_BM, &full[s]);
                    tc::tma_load_2d(st + S::A_BYTES, &tmH, kb * LM_BK, a.r0, &full[s]);
                }
            }
            if (!ok) {  // let the copies already issued land before the CTA can exit
                for (int q = step - 1; q >= 0 && q >= step - S::STAGES; --q)
                    mbar_wait_bounded(&full[q % S::STAGES], uint32_t(q / S::STAGES) & 1u, a.status);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            constexpr uint32_t idesc = tc::idesc_bf16_f32(LM_BM, NR);
            int step = 0;
            bool ok = true;
            for (int i = 0; i < nt && ok; ++i) {
                const int q = i & 1;
                if (i >= 2 && !mbar_wait_bounded(&acce[q], uint32_t((i >> 1) - 1) & 1u, a.status)) break;
                tc::fence_after_sync();
                const uint32_t acc = tmem + uint32_t(q * NR);
                for (int kb = 0; kb < nk; ++kb, ++step) {
                    const int s = step % S::STAGES;
                    if (!mbar_wait_bounded(&full[s], uint32_t(step / S::STAGES) & 1u, a.status)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t sa = smem_u32(smem + size_t(s) * S::STAGE);
                    const uint64_t da = tc::desc_sw128_kmajor(sa);
                    const uint64_t db = tc::desc_sw128_kmajor(sa + uint32_t(S::A_BYTES));
#pragma unroll
                    for (int kk = 0; kk < LM_BK / 16; ++kk)
                        tc::mma_bf16(acc, da + 2u * kk, db + 2u * kk, idesc, kb > 0 || kk > 0);
                    tc::mma_commit(&empty[s]);
                }
                if (ok) tc::mma_commit(&accf[q]);
            }
        }
    } else {
        // epilogue warps 2..5: TMEM lane quarter (warp % 4) = vocabulary rows 32 (warp % 4) ..
        const int quarter = warp & 3;
        const int ew = warp - 2;  // 0..3: which rows this warp cuts
        const uint32_t trow = tmem + (uint32_t(quarter * 32) << 16);
        // every epilogue warp runs the same barriers whatever happens: a warp whose
        // bounded wait ran out raises epi_err, and from then on all of them skip the work
        volatile int* epi_err = cnt + NR;  // one int after the counters
        bool ok = true;
        for (int i = 0; i < nt; ++i) {
            const int q = i & 1;
            const bool got =
                __all_sync(0xffffffffu, ok && mbar_wait_bounded(&accf[q], uint32_t(i >> 1) & 1u, a.status)) != 0;
            uint32_t v[NR];
            if (got) {
                tc::fence_after_sync();
#pragma unroll
                for (int c = 0; c < NR; c += 16) {
                    uint32_t r16[16];
                    tc::tmem_ld16(trow + uint32_t(q * NR + c), r16);
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[c + j] = r16[j];
                }
                tc::fence_before_sync();
            }
            __syncwarp();
            if (lane == 0) {
                if (got) mbar_arrive(&acce[q]);
                else *epi_err = 1;
            }
            epi_bar();
            ok = *epi_err == 0;
            if (ok)  // rows that a full tile could overflow are cut first
                for (int r = ew; r < a.R; r += 4)
                    if (cnt[r] > LM_CAP - LM_BM)
                        cut_row(cand + size_t(r) * LM_CAP, &cnt[r], &thr[r], a.K, hists + ew * 256);
            epi_bar();
            if (!ok) continue;
            const int tok = (t0 + i) * LM_BM + quarter * 32 + lane;
            const bool in = tok < a.V;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r >= a.R) break;
                const uint64_t key = (uint64_t(ord_f32(__uint_as_float(v[r]))) << 32) | (0xffffffffu - uint32_t(tok));
                const bool pass = in && key > thr[r];
                const uint32_t m = __ballot_sync(0xffffffffu, pass);
                if (m) {
                    int base = 0;
                    if (lane == 0) base = atomicAdd(&cnt[r], __popc(m));
                    base = __shfl_sync(0xffffffffu, base, 0);
                    if (pass) cand[size_t(r) * LM_CAP + base + __popc(m & ((1u << lane) - 1u))] = key;
                }
            }
        }
        // final cut of every row, K keys per (row, CTA); zero keys pad a short list
        epi_bar();
        for (int r = ew; r < a.R; r += 4) {
            uint64_t* buf = cand + size_t(r) * LM_CAP;
            cut_row(buf, &cnt[r], &thr[r], a.K, hists + ew * 256);
            {  // the list sorted (descending): the merge reads each list's maximum first
                const int n = cnt[r];
                int p = 32;
                while (p < a.K) p <<= 1;
                for (int q = n + lane; q < p; q += 32) buf[q] = 0ull;
                __syncwarp();
                warp_sort_desc(buf, p);
            }
            unsigned long long* dst = a.part + (size_t(r) * G + b) * a.K;
            for (int k = lane; k < a.K; k += 32) dst[k] = k < cnt[r] ? buf[k] : 0ull;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tmem, S::TMEM_COLS);
}

// ----------------------------------------------------------------------------- merge

constexpr int LMM_NT = 512;

// Row r: the K largest of n keys (K lists of every CTA), sorted, as (token, logit).
__global__ void __launch_bounds__(LMM_NT) lmhead_merge_kernel(const unsigned long long* __restrict__ part, int n,
                                                              int K, int32_t* __restrict__ tok,
                                                              float* __restrict__ val) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint64_t* keys = reinterpret_cast<uint64_t*>(smem);      // [n]
    uint32_t* hist = reinterpret_cast<uint32_t*>(keys + n);  // [256]
    uint64_t* sel = reinterpret_cast<uint64_t*>(hist + 256); // [LM_CAP] (K <= LM_MAXK)
    __shared__ uint32_t s_digit, s_need, s_inbin, s_nsel;
    const int r = blockIdx.x;
    if (threadIdx.x == 0) {
        s_digit = 0;
        s_need = 1;
        s_inbin = 0;
    }
    __shared__ uint64_t s_lb;
    griddep_wait();
    for (int i = threadIdx.x; i < n; i += LMM_NT) keys[i] = part[size_t(r) * n + i];
    __syncthreads();
    // Every list is sorted, so its first key is its maximum; with at least K lists, the
    // K-th largest list maximum is a lower bound of the K-th largest key (K distinct
    // keys reach it). The keys at or above it are usually few: those are sorted directly.
    const int G = n / K;
    if (G >= K && G <= LM_CAP) {
        if (threadIdx.x == 0) {
            s_nsel = 0;
            s_lb = 0;  // (no list maximum of rank K - 1: every key qualifies)
        }
        for (int b = threadIdx.x; b < G; b += LMM_NT) sel[b] = keys[b * K];
        __syncthreads();
        if (int(threadIdx.x) < G) {  // the list maximum of rank K - 1 (keys distinct)
            const uint64_t m = sel[threadIdx.x];
            int rank = 0;
            for (int b = 0; b < G; ++b) rank += sel[b] > m ? 1 : 0;
            if (rank == K - 1) s_lb = m;
        }
        __syncthreads();
        const uint64_t lb = s_lb;
        for (int b = threadIdx.x; b < G; b += LMM_NT)
            for (int k = 0; k < K && keys[b * K + k] >= lb; ++k) {
                const uint32_t at = atomicAdd(&s_nsel, 1u);
                if (at < uint32_t(LM_CAP)) sel[at] = keys[b * K + k];
            }
        __syncthreads();
        const uint32_t nsel = s_nsel;
        if (nsel <= uint32_t(LM_CAP)) {  // each candidate's rank is its output position
            if (threadIdx.x < nsel) {
                const uint64_t key = sel[threadIdx.x];
                int rank = 0;
                for (uint32_t q = 0; q < nsel; ++q) rank += sel[q] > key ? 1 : 0;
                if (rank < K) {
                    tok[size_t(r) * K + rank] = int32_t(0xffffffffu - uint32_t(key));
                    val[size_t(r) * K + rank] = f32_from_ord(uint32_t(key >> 32));
                }
            }
            return;
        }
        __syncthreads();
    }
    // otherwise: radix selection of the K-th largest key, 8 bits at a time from the top;
    // prefix/pmask: the bits fixed so far. It stops at the first digit whose bin holds
    // exactly the keys still needed.
    uint64_t prefix = 0, pmask = 0;
    uint32_t need = uint32_t(K);
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += LMM_NT) hist[i] = 0;
        __syncthreads();
        for (int i0 = 0; i0 < n; i0 += LMM_NT) {  // equal digits of a warp add once
            const int i = i0 + int(threadIdx.x);
            const uint64_t k = i < n ? keys[i] : 0ull;
            const bool in = i < n && (k & pmask) == prefix;
            const uint32_t d = in ? uint32_t(k >> shift) & 0xffu : 0x100u;
            const uint32_t same = __match_any_sync(0xffffffffu, d);
            if (in && (threadIdx.x & 31) == uint32_t(__ffs(same) - 1)) atomicAdd(&hist[d], uint32_t(__popc(same)));
        }
        __syncthreads();
        if (threadIdx.x < 32) {  // the digit where the count from the top reaches `need`
            const int lane = threadIdx.x;
            uint32_t c[8], tot = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {  // lane owns digits 255 - 8 lane - j (descending)
                c[j] = hist[255 - 8 * lane - j];
                tot += c[j];
            }
            uint32_t incl = tot;  // inclusive scan over lanes (descending digit order)
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            uint32_t run = incl - tot;
            const bool mine = run < need && incl >= need;
            if (mine) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (run + c[j] >= need) {
                        s_digit = uint32_t(255 - 8 * lane - j);
                        s_need = need - run;
                        s_inbin = c[j];
                        break;
                    }
                    run += c[j];
                }
            }
        }
        __syncthreads();
        prefix |= uint64_t(s_digit) << shift;
        pmask |= uint64_t(0xffu) << shift;
        need = s_need;
        const bool whole = s_inbin == s_need;  // every key of the bin is kept
        __syncthreads();
        if (whole) break;
    }
    // keep every key at or above the prefix in the fixed bits (exactly K, keys distinct)
    if (threadIdx.x == 0) s_nsel = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += LMM_NT) {
        const uint64_t k = keys[i];
        if ((k & pmask) >= prefix) {
            const uint32_t at = atomicAdd(&s_nsel, 1u);
            if (at < uint32_t(LM_CAP)) sel[at] = k;  // exactly K unless the lists were not written
        }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        int p = 32;
        while (p < K) p <<= 1;
        for (int i = K + threadIdx.x; i < p; i += 32) sel[i] = 0ull;
        __syncwarp();
        warp_sort_desc(sel, p);
        for (int k = threadIdx.x; k < K; k += 32) {
            const uint64_t key = sel[k];
            tok[size_t(r) * K + k] = int32_t(0xffffffffu - uint32_t(key));
            val[size_t(r) * K + k] = f32_from_ord(uint32_t(key >> 32));
        }
    }
}

// ----------------------------------------------------------------------------- host

bool lmhead_supported(int R, int V, int H, int K) {
    return R >= 1 && V >= K && V >= 1 && K >= 1 && K <= LM_MAXK && H >= LM_BK && H % LM_BK == 0;
}

int lmhead_grid(int V) {
    const int tiles = (V + LM_BM - 1) / LM_BM;
    return tiles < num_sms() ? tiles : num_sms();
}

size_t lmhead_part_bytes(int R, int V, int K) { return size_t(R) * lmhead_grid(V) * K * 8; }

static size_t merge_smem(int n) { return size_t(n) * 8 + 256 * 4 + LM_CAP * 8; }

template <int NR>
static int launch_lmhead_nr(const CUtensorMap& tw, const CUtensorMap& th, const LmArgs& a, int G,
                            cudaStream_t stream, bool pdl) {
    const size_t smem = LmSmem<NR>::TOTAL;
    auto kern = lmhead_topk_kernel<NR>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
        return DARTREE_ECUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(LM_NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e;
    {
        KTimer kt_(KID_LMHEAD, stream);
        e = cudaLaunchKernelEx(&cfg, kern, tw, th, a);
    }
    return e == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

int launch_lmhead_topk(const void* hidden, const void* W, int R, int V, int H, int K, int32_t* tok, float* val,
                       unsigned long long* part, int* status, cudaStream_t stream) {
    if (R == 0) return DARTREE_OK;
    if (!lmhead_supported(R, V, H, K)) return DARTREE_EUNSUPPORTED;
    const int G = lmhead_grid(V);
    const int n = G * K;
    const size_t msmem = merge_smem(n);
    if (msmem > 200 * 1024) return DARTREE_EUNSUPPORTED;
    if (cudaFuncSetAttribute(lmhead_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(msmem)) !=
        cudaSuccess)
        return DARTREE_ECUDA;
    CUtensorMap tw, th16, th32, th64;
    if (!make_tensor_map_bf16(&tw, W, V, H, LM_BK, LM_BM, 128) ||
        !make_tensor_map_bf16(&th16, hidden, R, H, LM_BK, 16, 128) ||
        !make_tensor_map_bf16(&th32, hidden, R, H, LM_BK, 32, 128) ||
        !make_tensor_map_bf16(&th64, hidden, R, H, LM_BK, 64, 128))
        return DARTREE_ECUDA;
    for (int r0 = 0; r0 < R; r0 += LM_MAXROWS) {  // one pass over W_lm per 64 hidden rows
        const int rr = R - r0 < LM_MAXROWS ? R - r0 : LM_MAXROWS;
        const int nr = rr <= 16 ? 16 : rr <= 32 ? 32 : 64;  // rows past R load as zeros
        LmArgs a{r0, rr, V, H, K, (V + LM_BM - 1) / LM_BM, part, status};
        int e = nr == 16   ? launch_lmhead_nr<16>(tw, th16, a, G, stream, r0 > 0)
                : nr == 32 ? launch_lmhead_nr<32>(tw, th32, a, G, stream, r0 > 0)
                           : launch_lmhead_nr<64>(tw, th64, a, G, stream, r0 > 0);
        if (e) return e;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(rr);
        cfg.blockDim = dim3(LMM_NT);
        cfg.dynamicSmemBytes = msmem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1] = {pdl_attribute()};
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t ce;
        {
            KTimer kt_(KID_LMMERGE, stream);
            ce = cudaLaunchKernelEx(&cfg, lmhead_merge_kernel, static_cast<const unsigned long long*>(part), n, K,
                                    tok + size_t(r0) * K, val + size_t(r0) * K);
        }
        if (ce != cudaSuccess) return DARTREE_ECUDA;
    }
    return DARTREE_OK;
}

}  // namespace dartree
