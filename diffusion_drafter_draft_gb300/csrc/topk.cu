// S1: per-position top-K of the base logits (DARTree blog post, 3.1 "Basic flow",
// candidate generation: keep the top-K tokens of every position).
//
// One thread-block cluster per row. Each CTA stages a contiguous chunk of the
// row in shared memory with TMA bulk copies (a single HBM read of the row) and
// works on orderable keys (value, ~token), so ties go to the lower token id:
//   1. while the pieces land, every thread keeps the 4 largest maxima of its
//      vectors (a branch-free min/max network); each CTA takes the j-th largest
//      of its threads' 4th-largest values (a bitwise search, j = ceil(K / 4S)),
//      and the minimum over the cluster is a value c with at least K elements
//      >= c (every CTA holds j threads with 4 vectors reaching it);
//   2. elements >= c (typically 2-20x K of them) are written to the leader CTA
//      through distributed shared memory at offsets from a cluster-wide scan;
//   3. the leader sorts the candidates (after a radix select of exactly K when
//      more than 1024 passed) and writes the first K.
// If more than TK_CAP elements pass the filter (heavy ties), the cluster falls
// back to an exact radix select of the K-th value with ordered tie compaction.
#include "common.cuh"
#include "kernels.h"

namespace dartree {

constexpr int TK_NT = 256;

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int TK_CAP = 4096;      // at most this many candidate keys gathered by the leader CTA
constexpr int TK_FB = 1024;       // keys of the exact fallback (K <= 1024)
constexpr int TK_PIECE = 16384;   // bytes per bulk copy (one mbarrier each)
constexpr int TK_MAXP = 16;       // at most 16 pieces (256 KB chunk)
constexpr int TK_STASH = 8;       // candidate keys a thread keeps in registers

// The data chunk doubles as the leader's candidate buffer once the filter pass
// has read it (peers write candidates only after the pass, behind a cluster
// barrier), so a CTA needs little more than its chunk of shared memory.
struct TopkSmem {
    size_t data, hist, hsum, misc, wtot, mbar, fb, total;
    int cap;  // candidate keys the data region holds
};

__host__ __device__ inline TopkSmem topk_smem_layout(int chunk, int elem) {
    TopkSmem s{};
    const size_t data = align_up(size_t(chunk) * elem, 128);
    s.data = 0;
    size_t off = data;
    s.hist = off; off += 2 * 256 * 4;
    s.hsum = off; off += 256 * 4;
    s.misc = off; off += 64 * 4;
    s.wtot = off; off += 32 * 4;
    s.mbar = off; off += 8 * TK_MAXP;
    off = align_up(off, 16);
    s.fb = off; off += size_t(TK_FB) * 8;
    s.total = off;
    const size_t cap = data / 8;
    s.cap = int(cap < size_t(TK_CAP) ? cap : size_t(TK_CAP));
    return s;
}

// Largest orderable key among the VEC elements of one 16-byte vector.
__device__ __forceinline__ uint32_t vec_max_ord(uint4 v, bf16_t*) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&v.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&v.w);
    const __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
    const uint32_t mb = *reinterpret_cast<const uint32_t*>(&m);
    const uint32_t lo = ord_bf16(mb & 0xffffu), hi = ord_bf16(mb >> 16);
    return lo > hi ? lo : hi;
}
__device__ __forceinline__ uint32_t vec_max_ord(uint4 v, float*) {
    return ord_f32(fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                         fmaxf(__uint_as_float(v.z), __uint_as_float(v.w))));
}
__device__ __forceinline__ uint32_t vec_elem_ord(uint4 v, int e, bf16_t*) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    return ord_bf16((w[e >> 1] >> ((e & 1) * 16)) & 0xffffu);
}
__device__ __forceinline__ uint32_t vec_elem_ord(uint4 v, int e, float*) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    return ord_f32(__uint_as_float(w[e]));
}

// Calls f(index_in_chunk, ord_key) for the thread's owned run [lo, hi) in order.
template <typename T, class F>
__device__ __forceinline__ void for_owned(const T* buf, int lo, int hi, F&& f) {
    constexpr int VEC = ValueKey<T>::VEC;
    int i = lo;
    for (; i + VEC <= hi; i += VEC) {
        uint4 v = *reinterpret_cast<const uint4*>(buf + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        if constexpr (VEC == 8) {
#pragma unroll
            for (int e = 0; e < 8; ++e) f(i + e, ord_bf16((w[e >> 1] >> ((e & 1) * 16)) & 0xffffu));
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) f(i + e, ord_f32(__uint_as_float(w[e])));
        }
    }
    for (; i < hi; ++i) f(i, ValueKey<T>::ord(buf[i]));
}

// Exact K-th largest of the values produced by `each` over the whole cluster,
// counting only values >= lo. On success v = that value and rem = how many of
// the values equal to v belong to the top K.
template <int KBITS, class Each>
__device__ bool cluster_select_kth(Each&& each, uint32_t lo, uint32_t K, uint32_t* hist2, uint32_t* hsum,
                                   uint32_t* misc, uint32_t S, uint32_t& v, uint32_t& rem) {
    uint32_t prefix = 0, r = K;
    int pass = 0;
    for (int shift = KBITS - 8; shift >= 0; shift -= 8, ++pass) {
        uint32_t* h = hist2 + (pass & 1) * 256;
        for (int i = threadIdx.x; i < 256; i += TK_NT) h[i] = 0;
        __syncthreads();
        const uint32_t hi_mask = (shift + 8 >= 32) ? 0u : (0xffffffffu << (shift + 8));
        const uint32_t want = prefix & hi_mask;
        each([&](int, uint32_t x) {
            if (x >= lo && (x & hi_mask) == want) atomicAdd(&h[(x >> shift) & 255u], 1u);
        });
        cluster_sync();
        for (int i = threadIdx.x; i < 256; i += TK_NT) {
            uint32_t s = 0;
            for (uint32_t c = 0; c < S; ++c) s += ld_dsmem_u32(dsmem_addr(&h[i], c));
            hsum[i] = s;
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            uint32_t rr = r, d;
            pick_digit_warp(hsum, rr, d);
            if (threadIdx.x == 0) { misc[0] = d; misc[1] = rr; }
        }
        __syncthreads();
        const uint32_t d = misc[0];
        const uint32_t nr = misc[1];
        __syncthreads();
        if (d == 0xffffffffu) return false;  // same outcome in every CTA: sums are shared
        prefix |= d << shift;
        r = nr;
    }
    v = prefix;
    rem = r;
    return true;
}

// Bitonic sort, descending, of n (a power of two, <= EPT*NT) keys: thread t holds
// elements t + e*NT (e < EPT) in registers. Partners closer than 32 are exchanged
// with warp shuffles, partners in the same thread directly, and only strides of
// 32..NT/2 go through shared memory.
template <int NT, int EPT>
__device__ __forceinline__ void sort_desc_regs(uint64_t* a, int n) {
    const int t = threadIdx.x;
    uint64_t v[EPT];
#pragma unroll
    for (int e = 0; e < EPT; ++e) v[e] = (t + e * NT < n) ? a[t + e * NT] : 0ull;
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j >= NT) {
                const int ej = j / NT;
#pragma unroll
                for (int es = 1; es < EPT; es <<= 1) {  // static partner slots (register indices)
                    if (es != ej) continue;
#pragma unroll
                    for (int e = 0; e < EPT; ++e) {
                        const int pe = e ^ es;
                        if (pe > e) {
                            const int i = t + e * NT;
                            const bool desc = (i & k) == 0;
                            const uint64_t x = v[e], y = v[pe];
                            const bool sw = desc ? (x < y) : (x > y);
                            v[e] = sw ? y : x;
                            v[pe] = sw ? x : y;
                        }
                    }
                }
            } else if (j >= 32) {
                __syncthreads();
#pragma unroll
                for (int e = 0; e < EPT; ++e)
                    if (t + e * NT < n) a[t + e * NT] = v[e];
                __syncthreads();
#pragma unroll
                for (int e = 0; e < EPT; ++e) {
                    const int i = t + e * NT;
                    if (i < n) {
                        const uint64_t p = a[i ^ j];
                        const bool lower = (i & j) == 0, desc = (i & k) == 0;
                        v[e] = (lower == desc) ? (p > v[e] ? p : v[e]) : (p < v[e] ? p : v[e]);
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < EPT; ++e) {
                    const int i = t + e * NT;
                    const uint64_t p = shfl_xor_u64(v[e], j);
                    const bool lower = (i & j) == 0, desc = (i & k) == 0;
                    v[e] = (lower == desc) ? (p > v[e] ? p : v[e]) : (p < v[e] ? p : v[e]);
                }
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < EPT; ++e)
        if (t + e * NT < n) a[t + e * NT] = v[e];
    __syncthreads();
}

template <int NT>
__device__ __forceinline__ void sort_desc(uint64_t* a, int n) {
    if (n <= NT) sort_desc_regs<NT, 1>(a, n);
    else if (n <= 2 * NT) sort_desc_regs<NT, 2>(a, n);
    else sort_desc_regs<NT, 4>(a, n);  // callers sort at most 1024 keys
}

// Exact selection used when the filter leaves more than TK_CAP candidates (heavy
// ties, constant rows): radix select of the K-th largest value over the whole
// chunk, then ordered compaction of the ties in token order. Writes the K keys
// to the leader's cand[0..K) (unsorted).
template <typename T>
__device__ bool topk_exact_fallback(const T* buf, int n, int c0, int K, uint32_t S, uint32_t cr, uint32_t* hist,
                                    uint32_t* hsum, uint32_t* misc, int* wtot, uint64_t* cand) {
    constexpr int VEC = ValueKey<T>::VEC;
    constexpr int KBITS = ValueKey<T>::BITS;
    const int per = int(align_up((n + TK_NT - 1) / TK_NT, VEC));
    const int lo = min(n, int(threadIdx.x) * per);
    const int hi = min(n, lo + per);
    auto each = [&](auto&& f) { for_owned<T>(buf, lo, hi, f); };
    if (threadIdx.x == 0) misc[10] = 0;
    uint32_t t = 0, rem = 0;
    bool ok = cluster_select_kth<KBITS>(each, 0u, uint32_t(K), hist, hsum, misc, S, t, rem);
    if (!ok) { t = 0xffffffffu; rem = 0; }
    const uint32_t n_gt = uint32_t(K) - rem;
    const uint32_t leader_ctr = dsmem_addr(&misc[10], 0);
    const uint32_t leader_cand = dsmem_addr(cand, 0);
    each([&](int i, uint32_t o) {
        if (o > t) {
            const uint32_t p = atom_add_dsmem_u32(leader_ctr, 1u);
            if (p < n_gt) st_dsmem_u64(leader_cand + 8u * p, (uint64_t(o) << 32) | (0xffffffffu - uint32_t(c0 + i)));
        }
    });
    int cnt = 0;
    each([&](int, uint32_t o) { cnt += (o == t); });
    const int excl = block_exclusive_scan<TK_NT>(cnt, wtot, reinterpret_cast<int*>(&misc[16]));
    cluster_sync();
    uint32_t rank = uint32_t(excl);
    for (uint32_t q = 0; q < cr; ++q) rank += ld_dsmem_u32(dsmem_addr(&misc[16], q));
    each([&](int i, uint32_t o) {
        if (o == t) {
            if (rank < rem)
                st_dsmem_u64(leader_cand + 8u * (n_gt + rank), (uint64_t(o) << 32) | (0xffffffffu - uint32_t(c0 + i)));
            ++rank;
        }
    });
    cluster_sync();
    return ok && (cr != 0 || misc[10] == n_gt);
}

// Bitonic sort, descending, of one 32-bit value per lane.
__device__ __forceinline__ uint32_t warp_sort_desc_u32(uint32_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int d = k >> 1; d >= 1; d >>= 1) {
            const uint32_t o = __shfl_xor_sync(0xffffffffu, v, d);
            const bool keep_max = ((lane & d) == 0) == ((lane & k) == 0);
            v = keep_max ? max(v, o) : min(v, o);
        }
    }
    return v;
}

template <typename T>
__global__ void __launch_bounds__(TK_NT, 4) topk_rows_kernel(const T* __restrict__ x, int V, int K, int jsel,
                                                          int chunk, int use_bulk, int32_t* __restrict__ out_tok,
                                                          float* __restrict__ out_val, int* status,
                                                          const uint16_t* __restrict__ gE, int gH,
                                                          uint16_t* __restrict__ gout, const T* __restrict__ tgt,
                                                          unsigned long long* __restrict__ tkeys,
                                                          const uint8_t* __restrict__ pre, unsigned long long pre_bytes) {
    extern __shared__ __align__(1024) uint8_t smem[];
    griddep_launch_dependents();
    constexpr int VEC = ValueKey<T>::VEC;
    const uint32_t S = cluster_nctarank(), cr = cluster_ctarank();
    const int row = blockIdx.x / S;
    const int c0 = int(cr) * chunk;
    const int n = max(0, min(V, c0 + chunk) - c0);
    const TopkSmem L = topk_smem_layout(chunk, sizeof(T));
    T* buf = reinterpret_cast<T*>(smem);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + L.hist);
    uint32_t* hsum = reinterpret_cast<uint32_t*>(smem + L.hsum);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L.misc);
    int* wtot = reinterpret_cast<int*>(smem + L.wtot);
    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + L.mbar);
    uint64_t* cand = reinterpret_cast<uint64_t*>(smem + L.data);  // after the filter pass
    uint64_t* fb = reinterpret_cast<uint64_t*>(smem + L.fb);
    const T* src = x + size_t(row) * V + c0;
    const int nvec = n / VEC;
    constexpr int VPP = TK_PIECE / 16;  // vectors per piece
    const uint32_t bytes = uint32_t(n) * sizeof(T);
    const int npieces = use_bulk ? int((bytes + TK_PIECE - 1) / TK_PIECE) : 0;

    // misc: [2] CTA min, [3] leader min, [4] leader count, [8..] scans
    if (tkeys && !tgt && cr == 0 && threadIdx.x == 0) tkeys[row] = 0ull;  // the maxima come later
    if (threadIdx.x < 64) misc[threadIdx.x] = (threadIdx.x == 2 || threadIdx.x == 3) ? 0xffffffffu : 0u;
    if (use_bulk) {
        if (threadIdx.x == 0) {
            for (int p = 0; p < npieces; ++p) mbar_init(&mbar[p], 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int p = 0; p < npieces; ++p) {
                const uint32_t o = uint32_t(p) * TK_PIECE;
                const uint32_t b = bytes - o < uint32_t(TK_PIECE) ? bytes - o : uint32_t(TK_PIECE);
                mbar_arrive_expect_tx(&mbar[p], b);
                bulk_g2s(reinterpret_cast<uint8_t*>(buf) + o, reinterpret_cast<const uint8_t*>(src) + o, b, &mbar[p]);
            }
        }
    } else {
        for (int i = threadIdx.x; i < n; i += TK_NT) buf[i] = src[i];
        __syncthreads();
    }

    // maximum key (ord(value) << 32 | ~index) of this chunk of the row's target
    // logits (verification), read while the chunk's copy is in flight; rows of
    // whole 16-byte vectors
    uint64_t tbest = 0;
    if (tgt) {
        const T* ts = tgt + size_t(row) * V + c0;
#pragma unroll 4
        for (int v = threadIdx.x; v < nvec; v += TK_NT) {
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(ts) + v);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const uint64_t k = (uint64_t(vec_elem_ord(w, e, static_cast<T*>(nullptr))) << 32) |
                                   (0xffffffffu - uint32_t(c0 + v * VEC + e));
                tbest = k > tbest ? k : tbest;
            }
        }
        for (int i = nvec * VEC + int(threadIdx.x); i < n; i += TK_NT) {
            const uint64_t k = (uint64_t(ValueKey<T>::ord(ts[i])) << 32) | (0xffffffffu - uint32_t(c0 + i));
            tbest = k > tbest ? k : tbest;
        }
        tbest = warp_max_u64(tbest);
        if ((threadIdx.x & 31) == 0) reinterpret_cast<uint64_t*>(hsum)[threadIdx.x >> 5] = tbest;
    }

    // pass 1: the 4 largest maxima of the vectors t, t+NT, ... (piece by piece as they land)
    uint32_t t0 = 0, t1 = 0, t2 = 0, t3 = 0;
    auto ins = [&](uint32_t vm) {
        t3 = max(t3, min(t2, vm));
        t2 = max(t2, min(t1, vm));
        t1 = max(t1, min(t0, vm));
        t0 = max(t0, vm);
    };
    bool loaded = true;
    if (use_bulk) {
        for (int p = 0; p < npieces; ++p) {
            if (!mbar_wait_bounded(&mbar[p], 0, status)) loaded = false;
            const int v1 = min(nvec, (p + 1) * VPP);
            for (int v = p * VPP + int(threadIdx.x); v < v1; v += TK_NT)
                ins(vec_max_ord(reinterpret_cast<const uint4*>(buf)[v], static_cast<T*>(nullptr)));
        }
    } else {
        for (int v = threadIdx.x; v < nvec; v += TK_NT)
            ins(vec_max_ord(reinterpret_cast<const uint4*>(buf)[v], static_cast<T*>(nullptr)));
    }
    for (int i = nvec * VEC + int(threadIdx.x); i < n; i += TK_NT) ins(ValueKey<T>::ord(buf[i]));
    // lower bound c, per CTA the larger of two bounds, then minimised over the
    // cluster: the CTA's j1-th largest vector maximum (j1 = ceil(K / S): j1 distinct
    // elements reach it) and its jsel-th largest 4th-largest vector maximum (4 * jsel
    // elements reach it, 4 * jsel * S >= K). Every CTA then has at least K / S
    // elements >= c. The first bound is the tighter one when a thread reads few
    // vectors, the second when it reads many.
    // Both are found 4 bits at a time: per digit value d, each warp counts (ballots)
    // its threads reaching prefix | d, lanes 1..15 for c1 and 17..31 for c4; after
    // one barrier every warp sums the warps' counts and takes the largest digit
    // whose count suffices (the counts fall with d), so all warps agree.
    // With j1, jsel <= 4 (few keys per CTA) the bounds are read off sorted lists
    // instead: each warp sorts its t0 and t3, its 4 largest of each go to shared
    // memory, and every warp sorts those 32 (they hold the CTA's 4 largest).
    const int j1 = (K + int(S) - 1) / int(S);
    if (j1 <= 4 && jsel <= 4) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        static_assert(TK_NT / 32 * 4 == 32, "8 warps x 4 keys");
        const uint32_t s0 = warp_sort_desc_u32(t0), s3 = warp_sort_desc_u32(t3);
        if (lane < 4) { hist[warp * 4 + lane] = s0; hist[32 + warp * 4 + lane] = s3; }
        __syncthreads();
        const uint32_t a0 = warp_sort_desc_u32(hist[lane]), a3 = warp_sort_desc_u32(hist[32 + lane]);
        const uint32_t c1 = __shfl_sync(0xffffffffu, a0, j1 - 1), c4 = __shfl_sync(0xffffffffu, a3, jsel - 1);
        if (threadIdx.x == 0) misc[2] = c1 > c4 ? c1 : c4;
    } else {
        constexpr int KB = ValueKey<T>::BITS;
        static_assert(KB % 4 == 0, "whole digits");
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        uint32_t c1 = 0, c4 = 0;
        uint32_t* wc = hist;  // [2][TK_NT / 32][32] per-warp counts, double-buffered
        for (int sh = KB - 4, it = 0; sh >= 0; sh -= 4, ++it) {
            uint32_t mine = 0;
#pragma unroll
            for (uint32_t d = 1; d < 16; ++d) {
                const uint32_t b1 = __ballot_sync(0xffffffffu, t0 >= (c1 | (d << sh)));
                const uint32_t b4 = __ballot_sync(0xffffffffu, t3 >= (c4 | (d << sh)));
                if (uint32_t(lane) == d) mine = __popc(b1);
                if (uint32_t(lane) == d + 16) mine = __popc(b4);
            }
            uint32_t* buf = wc + (it & 1) * TK_NT;
            buf[warp * 32 + lane] = mine;
            __syncthreads();
            uint32_t tot = 0;
#pragma unroll
            for (int w = 0; w < TK_NT / 32; ++w) tot += buf[w * 32 + lane];
            const bool ok1 = lane >= 1 && lane < 16 && j1 <= TK_NT && tot >= uint32_t(j1);
            const bool ok4 = lane >= 17 && tot >= uint32_t(jsel);
            const uint32_t m1 = __ballot_sync(0xffffffffu, ok1), m4 = __ballot_sync(0xffffffffu, ok4);
            if (m1) c1 |= uint32_t(31 - __clz(m1)) << sh;
            if (m4) c4 |= uint32_t(31 - __clz(m4) - 16) << sh;
        }
        if (threadIdx.x == 0) misc[2] = c1 > c4 ? c1 : c4;
    }
    __syncthreads();
    cluster_sync();  // every CTA's misc is initialised before remote atomics
    if (threadIdx.x == 0) {
        uint32_t old;
        asm volatile("atom.shared::cluster.min.u32 %0, [%1], %2;" : "=r"(old) : "r"(dsmem_addr(&misc[3], 0)), "r"(misc[2]) : "memory");
        if (tgt) {  // the CTA's target maximum into its slot misc[32 + 2 cr] of the leader
            uint64_t m = 0;
            for (int w = 0; w < TK_NT / 32; ++w) {
                const uint64_t x = reinterpret_cast<const uint64_t*>(hsum)[w];
                m = x > m ? x : m;
            }
            st_dsmem_u64(dsmem_addr(&misc[32 + 2 * cr], 0), m);
        }
    }
    cluster_sync();
    const uint32_t c = ld_dsmem_u32(dsmem_addr(&misc[3], 0));

    // pass 2: candidates >= c; a few per thread stay in registers
    uint64_t stash[TK_STASH];
    int cnt = 0;
    auto consider = [&](uint32_t o, int i) {
        if (o >= c) {
            const uint64_t key = (uint64_t(o) << 32) | (0xffffffffu - uint32_t(c0 + i));
#pragma unroll
            for (int q = 0; q < TK_STASH; ++q)
                if (q == cnt) stash[q] = key;
            ++cnt;
        }
    };
    for (int v = threadIdx.x; v < nvec; v += TK_NT) {
        const uint4 w = reinterpret_cast<const uint4*>(buf)[v];
        if (vec_max_ord(w, static_cast<T*>(nullptr)) >= c) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) consider(vec_elem_ord(w, e, static_cast<T*>(nullptr)), v * VEC + e);
        }
    }
    for (int i = nvec * VEC + int(threadIdx.x); i < n; i += TK_NT) consider(ValueKey<T>::ord(buf[i]), i);
    if (gout) {  // the rows of E the copy at the end may need: into L2 now
#pragma unroll
        for (int q = 0; q < TK_STASH; ++q)
            if (q < cnt) prefetch_l2_bulk(gE + size_t(0xffffffffu - uint32_t(stash[q])) * gH, uint32_t(gH) * 2u);
    }
    const int over = __syncthreads_or(cnt > TK_STASH);  // a thread with more candidates than registers
    if (threadIdx.x == 0) misc[9] = uint32_t(over);
    const int excl = block_exclusive_scan<TK_NT>(cnt, wtot, reinterpret_cast<int*>(&misc[8]));
    cluster_sync();  // CTA totals visible
    // the rows have streamed: this CTA's share of the next launch's operand into L2
    // (HBM is idle for the rest of this launch), in 16-byte multiples
    if (pre && threadIdx.x == 0) {
        const unsigned long long per = (pre_bytes / gridDim.x + 15) & ~15ull, b0 = per * blockIdx.x;
        for (unsigned long long o = b0; o < b0 + per && o < pre_bytes; o += 65536)
            prefetch_l2_bulk(pre + o, uint32_t(min(65536ull, min(b0 + per, pre_bytes) - o)));
    }
    if (tgt && cr == 0 && threadIdx.x == 0) {
        uint64_t m = 0;
#pragma unroll 16
        for (uint32_t q = 0; q < S; ++q) {
            const uint64_t x = *reinterpret_cast<const uint64_t*>(&misc[32 + 2 * q]);
            m = x > m ? x : m;
        }
        tkeys[row] = m;
    }
    // every CTA's candidate count and overflow flag: lane q reads CTA q's (one
    // remote load each, all in flight together), then the warp sums them
    uint32_t base, total, anyover;
    {
        const uint32_t lane = threadIdx.x & 31u;
        uint32_t tq = 0, oq = 0;
        if (lane < S) {
            tq = ld_dsmem_u32(dsmem_addr(&misc[8], lane));
            oq = ld_dsmem_u32(dsmem_addr(&misc[9], lane));
        }
        base = __reduce_add_sync(0xffffffffu, lane < cr ? tq : 0u);
        total = __reduce_add_sync(0xffffffffu, tq);
        anyover = __reduce_or_sync(0xffffffffu, oq);
    }
    // the same decision in every CTA: the totals and flags are shared
    const bool fits = total >= uint32_t(K) && total <= uint32_t(L.cap) && !anyover;
    // few candidates (one per thread): every CTA ranks the leader's list itself
    // (no sort, no further exchange); else the leader sorts or selects
    const bool spread = fits && total <= uint32_t(TK_NT);
    if (fits) {
        const uint32_t leader_cand = dsmem_addr(cand, 0);
        const uint32_t pos = base + uint32_t(excl);
#pragma unroll
        for (int q = 0; q < TK_STASH; ++q)
            if (q < cnt) st_dsmem_u64(leader_cand + 8u * (pos + q), stash[q]);
        cluster_sync();
    } else {
        // uniform across the cluster: every CTA summed the same totals
        if (!topk_exact_fallback<T>(buf, n, c0, K, S, cr, hist, hsum, misc, wtot, fb))
            if (threadIdx.x == 0) set_status(status, DARTREE_EINTERNAL);
    }

    // leader: up to TK_FB candidates are sorted directly; more are cut to exactly K
    // by a radix select first
    if (spread) {
        // rank of a key = number of larger keys (keys are distinct: the index is
        // in the low half). Every CTA copies the leader's list, then arrives on the
        // cluster barrier (the leader's shared memory may go once all have), ranks
        // every key, and copies the rows of ranks cr, cr + S, ... < K; the leader
        // writes the K outputs.
        const int n = int(total);
        uint64_t key = 0;
        if (int(threadIdx.x) < n) key = cr == 0 ? cand[threadIdx.x] : ld_dsmem_u64(dsmem_addr(&cand[threadIdx.x], 0));
        if (cr != 0 && int(threadIdx.x) < n) cand[threadIdx.x] = key;
        cluster_arrive_release();
        __syncthreads();
        int32_t* ranked = reinterpret_cast<int32_t*>(fb);  // token of each rank < K
        if (int(threadIdx.x) < n) {
            int larger = 0;
            for (int j0 = 0; j0 < n; j0 += 8) {  // 8 unconditional loads in flight
                uint64_t y[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) y[u] = cand[min(j0 + u, n - 1)];
#pragma unroll
                for (int u = 0; u < 8; ++u) larger += (j0 + u < n && y[u] > key) ? 1 : 0;
            }
            if (larger < K) {
                const int32_t t = int32_t(0xffffffffu - uint32_t(key));
                if (cr == 0) {
                    out_tok[size_t(row) * K + larger] = t;
                    out_val[size_t(row) * K + larger] = ValueKey<T>::value(uint32_t(key >> 32));
                }
                ranked[larger] = (t >= 0 && t < V) ? t : 0;
            }
        }
        if (gout) {
            __syncthreads();
            const int nmine = (K - int(cr) + int(S) - 1) / int(S);
            const int nv = gH / 8, tot = nmine * nv;
            constexpr int GU = 8;  // 16-byte loads in flight per thread
            for (int b = threadIdx.x; b < tot; b += GU * TK_NT) {
                uint4 v[GU];
#pragma unroll
                for (int u = 0; u < GU; ++u) {
                    const int i = b + u * TK_NT;
                    if (i < tot) {
                        const int j = i / nv, c = i - j * nv;
                        const int32_t t = ranked[int(cr) + j * int(S)];
                        v[u] = __ldg(reinterpret_cast<const uint4*>(gE + size_t(t) * gH) + c);
                    }
                }
#pragma unroll
                for (int u = 0; u < GU; ++u) {
                    const int i = b + u * TK_NT;
                    if (i < tot) {
                        const int j = i / nv, c = i - j * nv;
                        reinterpret_cast<uint4*>(gout + (size_t(row) * K + int(cr) + j * int(S)) * gH)[c] = v[u];
                    }
                }
            }
        }
        cluster_wait_acquire();
        if (use_bulk && !loaded && threadIdx.x == 0)
            for (int p = 0; p < npieces; ++p) mbar_wait_bounded(&mbar[p], 0, nullptr);
        return;
    }

    int np = 1;
    while (np < int(total)) np <<= 1;
    if (cr == 0 && fits && np <= TK_FB && np <= L.cap) {
        for (int i = int(total) + threadIdx.x; i < np; i += TK_NT) cand[i] = 0;
        __syncthreads();
        sort_desc<TK_NT>(cand, np);
        for (int i = threadIdx.x; i < K; i += TK_NT) {
            const uint64_t k = cand[i];
            const int32_t t = int32_t(0xffffffffu - uint32_t(k));
            out_tok[size_t(row) * K + i] = t;
            out_val[size_t(row) * K + i] = ValueKey<T>::value(uint32_t(k >> 32));
            if (gout) reinterpret_cast<int32_t*>(hist)[i] = t;
        }
    } else if (cr == 0) {
        if (fits) {
            uint64_t prefix = 0, mask = 0;
            uint64_t* orand = reinterpret_cast<uint64_t*>(hsum);  // 16 words of scratch
            const bool ok = block_select_top_agg<TK_NT>(cand, int(total), K, hist, misc + 32, orand, prefix, mask);
            if (threadIdx.x == 0) { misc[40] = 0; if (!ok) set_status(status, DARTREE_EINTERNAL); }
            __syncthreads();
            for (int i = threadIdx.x; i < int(total); i += TK_NT) {
                const uint64_t k = cand[i];
                if (ok && selected(k, prefix, mask)) {
                    const uint32_t q = atomicAdd(&misc[40], 1u);
                    if (q < uint32_t(K)) fb[q] = k;
                }
            }
            __syncthreads();
            if (threadIdx.x == 0 && misc[40] != uint32_t(K)) set_status(status, DARTREE_EINTERNAL);
            for (int i = min(int(misc[40]), K) + threadIdx.x; i < K; i += TK_NT) fb[i] = 0;
        }
        int kp = 1;
        while (kp < K) kp <<= 1;
        for (int i = K + threadIdx.x; i < kp; i += TK_NT) fb[i] = 0;
        __syncthreads();
        sort_desc<TK_NT>(fb, kp);
        for (int i = threadIdx.x; i < K; i += TK_NT) {
            const uint64_t k = fb[i];
            const int32_t t = int32_t(0xffffffffu - uint32_t(k));
            out_tok[size_t(row) * K + i] = t;
            out_val[size_t(row) * K + i] = ValueKey<T>::value(uint32_t(k >> 32));
            if (gout) reinterpret_cast<int32_t*>(hist)[i] = t;
        }
    }
    if (gout) {
        // rows of E for the K tokens, ranks cr, cr + S, ... copied by this CTA: the
        // leader's tokens (its hist, K <= 512) are read first, then the cluster
        // barrier's arrival releases them while the copies run
        int32_t* mine = reinterpret_cast<int32_t*>(fb);  // TK_FB * 2 >= 512 entries
        cluster_sync();
        const int nmine = (K - int(cr) + int(S) - 1) / int(S);
        const uint32_t ltok = dsmem_addr(hist, 0);
        for (int j = threadIdx.x; j < nmine; j += TK_NT) {
            const int32_t t = int32_t(ld_dsmem_u32(ltok + 4u * uint32_t(int(cr) + j * int(S))));
            mine[j] = (t >= 0 && t < V) ? t : 0;  // an invalid token (error status set) reads row 0
        }
        __syncthreads();
        cluster_arrive_release();
        const int nv = gH / 8, total = nmine * nv;
        constexpr int GU = 8;  // 16-byte loads in flight per thread
        for (int b = threadIdx.x; b < total; b += GU * TK_NT) {
            uint4 v[GU];
#pragma unroll
            for (int u = 0; u < GU; ++u) {
                const int i = b + u * TK_NT;
                if (i < total) {
                    const int j = i / nv, c = i - j * nv;
                    v[u] = __ldg(reinterpret_cast<const uint4*>(gE + size_t(mine[j]) * gH) + c);
                }
            }
#pragma unroll
            for (int u = 0; u < GU; ++u) {
                const int i = b + u * TK_NT;
                if (i < total) {
                    const int j = i / nv, c = i - j * nv;
                    reinterpret_cast<uint4*>(gout + (size_t(row) * K + int(cr) + j * int(S)) * gH)[c] = v[u];
                }
            }
        }
        cluster_wait_acquire();
    }
    if (use_bulk && !loaded && threadIdx.x == 0)
        for (int p = 0; p < npieces; ++p) mbar_wait_bounded(&mbar[p], 0, nullptr);
}

// --------------------------------------------------------------------------- many rows: one CTA per row

// With at least two rows per SM, one CTA per row reads its row once with 16-byte
// vector loads, several in flight per thread, and needs no cluster barrier:
//   1. every thread keeps the 4 largest maxima of the vectors it reads (a
//      branch-free min/max network), and the 16-bit maximum of every 32-byte
//      group of the row goes to shared memory; the largest c such that
//      ceil(K/4) threads hold a 4th-largest vector maximum >= c (a bitwise
//      search with __syncthreads_count) has at least K elements >= c: that
//      many threads each read 4 vectors holding an element >= c;
//   2. only the groups whose maximum reaches c (a few percent) are read again
//      and their elements >= c written to a candidate buffer at block-scan
//      offsets;
//   3. exactly the K best are selected (radix) and sorted as in the cluster
//      kernel. More than TS_CAP candidates (heavy ties) take the exact radix
//      select over the row instead.
// Four CTAs share an SM.
constexpr int TS_NT = 256;
constexpr int TS_UNROLL = 8;    // vector loads in flight per thread
constexpr int TS_CAP = 2048;    // candidate keys

struct TsSmem {
    size_t gmax, cand, fb, hist, hsum, misc, wtot, total;
};
// nvec: 16-byte vectors per row (two per group)
__host__ __device__ inline TsSmem ts_smem(int nvec) {
    TsSmem s{};
    size_t o = 0;
    auto take = [&](size_t b, size_t a) { o = align_up(o, a); size_t at = o; o += b; return at; };
    s.gmax = take(size_t((nvec + 1) / 2) * 2, 16);
    s.cand = take(size_t(TS_CAP) * 8, 16);
    s.fb = take(size_t(TK_FB) * 8, 16);
    s.hist = take(2 * 256 * 4, 16);
    s.hsum = take(256 * 4, 16);
    s.misc = take(64 * 4, 16);
    s.wtot = take(32 * 4, 16);
    s.total = o;
    return s;
}

template <typename T>
__global__ void __launch_bounds__(TS_NT, 4) topk_stream_kernel(const T* __restrict__ x, int V, int K,
                                                            int32_t* __restrict__ out_tok,
                                                            float* __restrict__ out_val, int* status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int VEC = ValueKey<T>::VEC;
    constexpr int KBITS = ValueKey<T>::BITS;
    const int nvec = int(size_t(V) * sizeof(T) / 16);
    const TsSmem L = ts_smem(nvec);
    uint16_t* gmax = reinterpret_cast<uint16_t*>(smem + L.gmax);  // 16-bit key maximum of vectors 2g, 2g + 1
    uint64_t* cand = reinterpret_cast<uint64_t*>(smem + L.cand);
    uint64_t* fb = reinterpret_cast<uint64_t*>(smem + L.fb);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + L.hist);
    uint32_t* hsum = reinterpret_cast<uint32_t*>(smem + L.hsum);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L.misc);
    int* wtot = reinterpret_cast<int*>(smem + L.wtot);
    const int row = blockIdx.x;
    const T* src = x + size_t(row) * V;
    const uint4* rv = reinterpret_cast<const uint4*>(src);
    const int lane = threadIdx.x & 31;

    if (threadIdx.x < 64) misc[threadIdx.x] = 0;
    __syncthreads();
    // ---- pass 1: vectors t, t + NT, ... (TS_UNROLL loads issued before any is
    //      used): the thread's 4 largest vector maxima and the group maxima
    uint32_t t0 = 0, t1 = 0, t2 = 0, t3 = 0;
    auto insert = [&](uint32_t vm) {  // t0 >= t1 >= t2 >= t3: the 4 largest vector maxima
        t3 = max(t3, min(t2, vm));
        t2 = max(t2, min(t1, vm));
        t1 = max(t1, min(t0, vm));
        t0 = max(t0, vm);
    };
    constexpr int SHIFT16 = KBITS - 16;  // 16-bit group keys: the top bits of the key
    // lanes 2i and 2i+1 hold the two vectors of one group (v = base + lane, base even)
    auto group_max = [&](int v, uint32_t vm, bool valid) {
        uint32_t g16 = valid ? (vm >> SHIFT16) : 0u;
        g16 = max(g16, __shfl_xor_sync(0xffffffffu, g16, 1));
        if ((lane & 1) == 0 && v < nvec) gmax[v >> 1] = uint16_t(g16);
    };
    {
        int v0 = int(threadIdx.x) & ~31;  // warp-uniform trip counts (group maxima use shuffles)
        for (; v0 + (TS_UNROLL - 1) * TS_NT < nvec; v0 += TS_UNROLL * TS_NT) {
            uint4 w[TS_UNROLL];
            bool ok[TS_UNROLL];
#pragma unroll
            for (int u = 0; u < TS_UNROLL; ++u) {
                const int v = v0 + lane + u * TS_NT;
                ok[u] = v < nvec;
                w[u] = ok[u] ? __ldg(rv + v) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < TS_UNROLL; ++u) {
                const uint32_t vm = ok[u] ? vec_max_ord(w[u], static_cast<T*>(nullptr)) : 0u;
                insert(vm);
                group_max(v0 + lane + u * TS_NT, vm, ok[u]);
            }
        }
        for (; v0 < nvec; v0 += TS_NT) {
            const int v = v0 + lane;
            const bool ok = v < nvec;
            const uint4 w = ok ? __ldg(rv + v) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t vm = ok ? vec_max_ord(w, static_cast<T*>(nullptr)) : 0u;
            insert(vm);
            group_max(v, vm, ok);
        }
    }
    // ---- lower bound: largest c with at least ceil(K/4) threads' 4th-largest
    //      vector maximum >= c
    const int j4 = (K + 3) / 4;
    uint32_t c = 0;
    for (int b = KBITS - 1; b >= 0; --b) {
        const uint32_t trial = c | (1u << b);
        if (__syncthreads_count(t3 >= trial) >= j4) c = trial;
    }
    // ---- pass 2: only the groups whose maximum reaches c are read again (gmax is
    //      complete: the bound's barriers follow pass 1). Their indices are placed
    //      in fb by a block scan; then every thread counts the elements >= c of
    //      its hit groups (two groups' loads in flight), a second scan gives the
    //      offsets, and the same groups (now in L1) are read once more to write
    //      the candidate keys.
    const uint32_t c16 = c >> SHIFT16;
    const int ngroups = (nvec + 1) / 2;
    int nh = 0;
    for (int g = threadIdx.x; g < ngroups; g += TS_NT) nh += uint32_t(gmax[g]) >= c16;
    const int hx = block_exclusive_scan<TS_NT>(nh, wtot, reinterpret_cast<int*>(&misc[4]));
    const int nhits = int(misc[4]);
    uint32_t* hits = reinterpret_cast<uint32_t*>(fb);
    constexpr int TS_HITCAP = TK_FB * 2;  // u32 entries of fb
    const bool hits_fit = nhits <= TS_HITCAP;
    if (hits_fit) {
        int o = hx;
        for (int g = threadIdx.x; g < ngroups; g += TS_NT)
            if (uint32_t(gmax[g]) >= c16) hits[o++] = uint32_t(g);
    }
    __syncthreads();
    // f(vector index, vector) over the vectors of this thread's hit groups
    auto over_hits = [&](auto&& f) {
        for (int h = threadIdx.x; h < nhits; h += 2 * TS_NT) {
            const int h2 = h + TS_NT;
            const int va = 2 * int(hits[h]), vb = h2 < nhits ? 2 * int(hits[h2]) : -1;
            const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
            const uint4 w0 = __ldg(rv + va);
            const uint4 w1 = va + 1 < nvec ? __ldg(rv + va + 1) : zero;
            const uint4 w2 = vb >= 0 ? __ldg(rv + vb) : zero;
            const uint4 w3 = (vb >= 0 && vb + 1 < nvec) ? __ldg(rv + vb + 1) : zero;
            f(va, w0);
            if (va + 1 < nvec) f(va + 1, w1);
            if (vb >= 0) {
                f(vb, w2);
                if (vb + 1 < nvec) f(vb + 1, w3);
            }
        }
    };
    int cnt = 0;
    if (hits_fit)
        over_hits([&](int, uint4 w) {
            if (vec_max_ord(w, static_cast<T*>(nullptr)) < c) return;
#pragma unroll
            for (int e = 0; e < VEC; ++e) cnt += vec_elem_ord(w, e, static_cast<T*>(nullptr)) >= c;
        });
    const int excl = block_exclusive_scan<TS_NT>(cnt, wtot, reinterpret_cast<int*>(&misc[0]));
    const uint32_t total = hits_fit ? misc[0] : 0xffffffffu;
    if (total <= uint32_t(TS_CAP)) {
        uint32_t pos = uint32_t(excl);
        over_hits([&](int vi, uint4 w) {
            if (vec_max_ord(w, static_cast<T*>(nullptr)) < c) return;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const uint32_t o = vec_elem_ord(w, e, static_cast<T*>(nullptr));
                if (o >= c) cand[pos++] = (uint64_t(o) << 32) | (0xffffffffu - uint32_t(vi * VEC + e));
            }
        });
    }
    __syncthreads();
    if (total >= uint32_t(K) && total <= uint32_t(TS_CAP)) {
        uint64_t prefix = 0, mask = 0;
        uint64_t* orand = reinterpret_cast<uint64_t*>(hsum);
        const bool ok = block_select_top_agg<TS_NT>(cand, int(total), K, hist, misc + 32, orand, prefix, mask);
        if (threadIdx.x == 0) { misc[40] = 0; if (!ok) set_status(status, DARTREE_EINTERNAL); }
        __syncthreads();
        for (int i = threadIdx.x; i < int(total); i += TS_NT) {
            const uint64_t k = cand[i];
            if (ok && selected(k, prefix, mask)) {
                const uint32_t q = atomicAdd(&misc[40], 1u);
                if (q < uint32_t(K)) fb[q] = k;
            }
        }
        __syncthreads();
        if (threadIdx.x == 0 && misc[40] != uint32_t(K)) set_status(status, DARTREE_EINTERNAL);
        for (int i = min(int(misc[40]), K) + threadIdx.x; i < K; i += TS_NT) fb[i] = 0;
    } else {
        // heavy ties: exact radix select over the row read from global memory
        // (a one-CTA cluster)
        if (!topk_exact_fallback<T>(src, V, 0, K, 1u, 0u, hist, hsum, misc, wtot, fb))
            if (threadIdx.x == 0) set_status(status, DARTREE_EINTERNAL);
    }
    int kp = 1;
    while (kp < K) kp <<= 1;
    for (int i = K + threadIdx.x; i < kp; i += TS_NT) fb[i] = 0;
    __syncthreads();
    sort_desc<TS_NT>(fb, kp);
    for (int i = threadIdx.x; i < K; i += TS_NT) {
        const uint64_t k = fb[i];
        out_tok[size_t(row) * K + i] = int32_t(0xffffffffu - uint32_t(k));
        out_val[size_t(row) * K + i] = ValueKey<T>::value(uint32_t(k >> 32));
    }
}

// --------------------------------------------------------------------------- host side

static int g_num_sms = 0;

int num_sms() {
    if (!g_num_sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 148;
    }
    return g_num_sms;
}

template <typename T>
static int launch_topk_t(const void* x, int rows, int V, int K, int32_t* tok, float* val, int* status,
                         cudaStream_t stream, const TopkGather* g, const TopkRowmax* rm, int max_s = 16) {
    const int elem = sizeof(T);
    const int VEC = 16 / elem;
    int S = 1;
    auto chunk_of = [&](int s) { return int(align_up((V + s - 1) / s, VEC)); };
    // ~40 KB chunks: several CTAs per SM overlap their loads with the other CTAs'
    // passes; with few rows, up to 16-CTA clusters so that the rows still cover the GPU
    while (S < 8 && size_t(chunk_of(S)) * elem > 40 * 1024) S *= 2;
    while (S < max_s && rows * S < 2 * num_sms() && size_t(chunk_of(2 * S)) * elem >= 16 * 1024) S *= 2;
    const int chunk = chunk_of(S);
    const TopkSmem L = topk_smem_layout(chunk, elem);
    const int jsel = (K + 4 * S - 1) / (4 * S);  // threads per CTA holding the bound (<= TK_NT)
    const int use_bulk = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && ((size_t(V) * elem) % 16 == 0);
    auto kern = topk_rows_kernel<T>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(L.total)) != cudaSuccess)
        return DARTREE_ECUDA;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return DARTREE_ECUDA;
    if (S > 8) {  // 16-CTA clusters need a GPC with 16 free SMs: keep 8 when none can run
        cudaLaunchConfig_t q{};
        q.gridDim = dim3(unsigned(S));
        q.blockDim = dim3(TK_NT);
        q.dynamicSmemBytes = L.total;
        cudaLaunchAttribute qa[1];
        qa[0].id = cudaLaunchAttributeClusterDimension;
        qa[0].val.clusterDim.x = S;
        qa[0].val.clusterDim.y = 1;
        qa[0].val.clusterDim.z = 1;
        q.attrs = qa;
        q.numAttrs = 1;
        int nc = 0;
        if (cudaOccupancyMaxActiveClusters(&nc, kern, &q) != cudaSuccess || nc < 1) {
            cudaGetLastError();
            return launch_topk_t<T>(x, rows, V, K, tok, val, status, stream, g, rm, 8);
        }
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(rows) * S);
    cfg.blockDim = dim3(TK_NT);
    cfg.dynamicSmemBytes = L.total;
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
        KTimer kt_(KID_TOPK_ROWS, stream);
        e = cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const T*>(x), V, K, jsel, chunk, use_bulk, tok, val,
                               status, g ? g->E : nullptr, g ? g->H : 0, g ? g->out : nullptr,
                               rm && !rm->zero_only ? static_cast<const T*>(rm->target) : nullptr,
                               rm ? rm->keys : nullptr, g ? static_cast<const uint8_t*>(g->pre) : nullptr,
                               g ? (unsigned long long)g->pre_bytes : 0ull);
    }
    return e == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

template <typename T>
static int launch_topk_stream(const void* x, int rows, int V, int K, int32_t* tok, float* val, int* status,
                              cudaStream_t stream) {
    const TsSmem L = ts_smem(int(size_t(V) * sizeof(T) / 16));
    auto kern = topk_stream_kernel<T>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(L.total)) != cudaSuccess)
        return DARTREE_ECUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(rows));
    cfg.blockDim = dim3(TS_NT);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];  // a one-CTA cluster: the exact fallback uses cluster barriers
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    {
        KTimer kt_(KID_TOPK_STREAM, stream);
        e = cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const T*>(x), V, K, tok, val, status);
    }
    // (rows are read with plain vector loads: 16-byte aligned rows)
    return e == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

// One CTA per row once the rows cover the SMs twice and every row starts on a
// 16-byte boundary; else one cluster per row.
static bool use_stream(const void* x, int rows, int V, int K, int elem) {
    return rows >= 2 * num_sms() && K <= 4 * TS_NT && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
           (size_t(V) * elem) % 16 == 0;
}

// The cluster kernel copies the gathered rows itself (K <= 512 tokens fit the
// leader's histogram, rows of whole 16-byte vectors).
static bool gather_ok(const TopkGather* g, int K) {
    return g && g->E && g->out && K <= 512 && g->H > 0 && g->H % 8 == 0 &&
           (reinterpret_cast<uintptr_t>(g->E) | reinterpret_cast<uintptr_t>(g->out)) % 16 == 0;
}

int launch_topk(const void* x, int rows, int V, int K, int dtype, int32_t* tok, float* val, int* status,
                cudaStream_t stream, const TopkGather* g, bool* gathered, const TopkRowmax* rm, bool* rm_done) {
    if (gathered) *gathered = false;
    if (rm_done) *rm_done = false;
    if (rows == 0) return DARTREE_OK;
    const int elem = dtype == DARTREE_BF16 ? 2 : 4;
    if (use_stream(x, rows, V, K, elem))
        return dtype == DARTREE_BF16 ? launch_topk_stream<bf16_t>(x, rows, V, K, tok, val, status, stream)
                                     : launch_topk_stream<float>(x, rows, V, K, tok, val, status, stream);
    const TopkGather* gg = gather_ok(g, K) ? g : nullptr;
    // the target rows are read with 16-byte vector loads
    const TopkRowmax* rr = rm && rm->keys &&
                                   (rm->zero_only || (rm->target && reinterpret_cast<uintptr_t>(rm->target) % 16 == 0 &&
                                                      (size_t(V) * elem) % 16 == 0))
                               ? rm
                               : nullptr;
    const int e = dtype == DARTREE_BF16 ? launch_topk_t<bf16_t>(x, rows, V, K, tok, val, status, stream, gg, rr)
                                        : launch_topk_t<float>(x, rows, V, K, tok, val, status, stream, gg, rr);
    if (gathered) *gathered = e == DARTREE_OK && gg != nullptr;
    if (rm_done) *rm_done = e == DARTREE_OK && rr != nullptr;
    return e;
}

}  // namespace dartree
