// S1: per-position top-K of the base logits (DARTree blog post, 3.1 "Basic flow",
// candidate generation: keep the top-K tokens of every position).
//
// One thread-block cluster per row. Each CTA stages a contiguous chunk of the
// row in shared memory with one TMA bulk copy (a single HBM read of the row),
// then the cluster runs an exact radix select on orderable value keys:
//   1. every thread's maximum over its owned run of elements is a "group max";
//      the K-th largest group max c is a lower bound of the K-th largest value
//      (K groups each hold an element >= c), so only elements >= c can matter;
//   2. exact K-th largest value t among elements >= c, 8 bits per pass, with the
//      per-CTA histograms summed through distributed shared memory;
//   3. all elements > t, plus the first (K - #>t) elements == t in token order
//      (ties go to the lower token id), are written to the leader CTA;
//   4. the leader sorts the K composite keys (value, ~token) and writes them out.
#include "common.cuh"
#include "kernels.h"

namespace dartree {

constexpr int TK_NT = 512;

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct TopkSmem {
    size_t hist, hsum, misc, wtot, mbar, cand, total;
};

__host__ __device__ inline TopkSmem topk_smem_layout(int chunk, int elem, int kpad) {
    TopkSmem s{};
    size_t off = align_up(size_t(chunk) * elem, 128);
    s.hist = off; off += 2 * 256 * 4;
    s.hsum = off; off += 256 * 4;
    s.misc = off; off += 64 * 4;
    s.wtot = off; off += 32 * 4;
    s.mbar = off; off += 16;
    off = align_up(off, 16);
    s.cand = off; off += size_t(kpad) * 8;
    s.total = off;
    return s;
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

template <typename T>
__global__ void __launch_bounds__(TK_NT) topk_rows_kernel(const T* __restrict__ x, int V, int K, int kpad,
                                                          int chunk, int use_bulk, int32_t* __restrict__ out_tok,
                                                          float* __restrict__ out_val, int* status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int VEC = ValueKey<T>::VEC;
    constexpr int KBITS = ValueKey<T>::BITS;
    const uint32_t S = cluster_nctarank(), cr = cluster_ctarank();
    const int row = blockIdx.x / S;
    const int c0 = int(cr) * chunk;
    const int n = max(0, min(V, c0 + chunk) - c0);
    const TopkSmem L = topk_smem_layout(chunk, sizeof(T), kpad);
    T* buf = reinterpret_cast<T*>(smem);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + L.hist);
    uint32_t* hsum = reinterpret_cast<uint32_t*>(smem + L.hsum);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L.misc);
    int* wtot = reinterpret_cast<int*>(smem + L.wtot);
    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + L.mbar);
    uint64_t* cand = reinterpret_cast<uint64_t*>(smem + L.cand);
    const T* src = x + size_t(row) * V + c0;

    if (threadIdx.x < 64) misc[threadIdx.x] = 0;
    bool loaded = true;
    if (use_bulk) {
        if (threadIdx.x == 0) { mbar_init(mbar, 1); fence_mbar_init(); }
        __syncthreads();
        if (threadIdx.x == 0) {
            const uint32_t bytes = uint32_t(n) * sizeof(T);
            mbar_arrive_expect_tx(mbar, bytes);
            constexpr uint32_t PIECE = 32768;
            for (uint32_t o = 0; o < bytes; o += PIECE) {
                const uint32_t b = bytes - o < PIECE ? bytes - o : PIECE;
                bulk_g2s(reinterpret_cast<uint8_t*>(buf) + o, reinterpret_cast<const uint8_t*>(src) + o, b, mbar);
            }
        }
        loaded = mbar_wait_bounded(mbar, 0, status);
    } else {
        for (int i = threadIdx.x; i < n; i += TK_NT) buf[i] = src[i];
    }
    __syncthreads();

    // owned run of this thread (multiple of the 16-byte vector)
    const int per = int(align_up((n + TK_NT - 1) / TK_NT, VEC));
    const int lo = min(n, int(threadIdx.x) * per);
    const int hi = min(n, lo + per);
    auto each = [&](auto&& f) { for_owned<T>(buf, lo, hi, f); };

    // 1. lower bound c from the group maxima
    uint32_t gm = 0;
    each([&](int, uint32_t o) { gm = o > gm ? o : gm; });
    uint32_t c = 0, dummy = 0;
    bool ok = true;
    if (S * TK_NT >= uint32_t(K)) {
        ok = cluster_select_kth<KBITS>([&](auto&& f) { f(0, gm); }, 0u, uint32_t(K), hist, hsum, misc, S, c, dummy);
    }
    // 2. exact K-th largest value t among elements >= c
    uint32_t t = 0, rem = 0;
    if (ok) ok = cluster_select_kth<KBITS>(each, c, uint32_t(K), hist, hsum, misc, S, t, rem);
    if (!ok) { t = 0xffffffffu; rem = 0; }  // select nothing; the status records the failure
    const uint32_t n_gt = uint32_t(K) - rem;

    // 3a. elements > t go to the leader in any order
    const uint32_t leader_ctr = dsmem_addr(&misc[8], 0);
    const uint32_t leader_cand = dsmem_addr(cand, 0);
    each([&](int i, uint32_t o) {
        if (o > t) {
            const uint32_t p = atom_add_dsmem_u32(leader_ctr, 1u);
            if (p < n_gt) st_dsmem_u64(leader_cand + 8u * p, (uint64_t(o) << 32) | (0xffffffffu - uint32_t(c0 + i)));
        }
    });
    // 3b. the first rem elements == t in token order
    int cnt = 0;
    each([&](int, uint32_t o) { cnt += (o == t); });
    const int excl = block_exclusive_scan<TK_NT>(cnt, wtot, reinterpret_cast<int*>(&misc[16]));
    cluster_sync();
    uint32_t rank = uint32_t(excl);
    for (uint32_t q = 0; q < cr; ++q) rank += ld_dsmem_u32(dsmem_addr(&misc[16], q));
    each([&](int i, uint32_t o) {
        if (o == t) {
            if (rank < rem) st_dsmem_u64(leader_cand + 8u * (n_gt + rank), (uint64_t(o) << 32) | (0xffffffffu - uint32_t(c0 + i)));
            ++rank;
        }
    });
    cluster_sync();

    // 4. leader sorts and writes
    if (cr == 0) {
        if (threadIdx.x == 0 && (!ok || misc[8] != n_gt)) set_status(status, DARTREE_EINTERNAL);
        for (int i = K + threadIdx.x; i < kpad; i += TK_NT) cand[i] = 0;
        if (!ok) for (int i = threadIdx.x; i < K; i += TK_NT) cand[i] = 0;
        __syncthreads();
        bitonic_sort_desc<TK_NT>(cand, kpad);
        for (int i = threadIdx.x; i < K; i += TK_NT) {
            const uint64_t k = cand[i];
            out_tok[size_t(row) * K + i] = int32_t(0xffffffffu - uint32_t(k));
            out_val[size_t(row) * K + i] = ValueKey<T>::value(uint32_t(k >> 32));
        }
    }
    if (use_bulk && !loaded && threadIdx.x == 0) mbar_wait_bounded(mbar, 0, nullptr);
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
                         cudaStream_t stream) {
    const int elem = sizeof(T);
    const int VEC = 16 / elem;
    int S = 1;
    auto chunk_of = [&](int s) { return int(align_up((V + s - 1) / s, VEC)); };
    while (S < 8 && (size_t(chunk_of(S)) * elem > 96 * 1024 ||
                     (rows * S < 2 * num_sms() && size_t(chunk_of(2 * S)) * elem >= 16 * 1024)))
        S *= 2;
    const int chunk = chunk_of(S);
    int kpad = 1;
    while (kpad < K) kpad <<= 1;
    const TopkSmem L = topk_smem_layout(chunk, elem, kpad);
    const int use_bulk = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && ((size_t(V) * elem) % 16 == 0);
    auto kern = topk_rows_kernel<T>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(L.total)) != cudaSuccess)
        return DARTREE_ECUDA;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return DARTREE_ECUDA;
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
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const T*>(x), V, K, kpad, chunk, use_bulk,
                                       tok, val, status);
    return e == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

int launch_topk(const void* x, int rows, int V, int K, int dtype, int32_t* tok, float* val, int* status,
                cudaStream_t stream) {
    if (rows == 0) return DARTREE_OK;
    if (dtype == DARTREE_BF16) return launch_topk_t<bf16_t>(x, rows, V, K, tok, val, status, stream);
    return launch_topk_t<float>(x, rows, V, K, tok, val, status, stream);
}

}  // namespace dartree
