// Shared device helpers for the DARTree kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "dartree.h"

namespace dartree {

// ----------------------------------------------------------------------------- storage types

// bf16 is handled as raw bits; widening to float is exact (bits << 16).
struct bf16_t { uint16_t bits; };

__device__ __forceinline__ float to_float(float v) { return v; }
__device__ __forceinline__ float to_float(bf16_t v) { return __uint_as_float(uint32_t(v.bits) << 16); }
__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

template <typename T> __device__ __forceinline__ T from_float(float v);
template <> __device__ __forceinline__ float from_float<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16_t from_float<bf16_t>(float v) {
    return bf16_t{__bfloat16_as_ushort(__float2bfloat16_rn(v))};
}

// ----------------------------------------------------------------------------- orderable keys
// Larger key = larger value. -0.0 is folded onto +0.0 so that they tie.

__device__ __forceinline__ uint32_t ord_f32(float v) {
    uint32_t u = __float_as_uint(v);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float f32_from_ord(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}
__device__ __forceinline__ uint32_t ord_bf16(uint32_t b) {
    if (b == 0x8000u) b = 0u;
    return (b & 0x8000u) ? (~b & 0xffffu) : (b | 0x8000u);
}
__device__ __forceinline__ float f32_from_ord_bf16(uint32_t o) {
    uint32_t b = (o & 0x8000u) ? (o & 0x7fffu) : (~o & 0xffffu);
    return bf16_bits_to_float(b);
}

template <typename T> struct ValueKey;
template <> struct ValueKey<float> {
    static constexpr int BITS = 32;
    static constexpr int VEC = 4;  // elements per 16-byte vector
    __device__ static uint32_t ord(float v) { return ord_f32(v); }
    __device__ static float value(uint32_t o) { return f32_from_ord(o); }
};
template <> struct ValueKey<bf16_t> {
    static constexpr int BITS = 16;
    static constexpr int VEC = 8;
    __device__ static uint32_t ord(bf16_t v) { return ord_bf16(v.bits); }
    __device__ static float value(uint32_t o) { return f32_from_ord_bf16(o); }
};

// ----------------------------------------------------------------------------- status word

__device__ __forceinline__ void set_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s for any device-side wait

// ----------------------------------------------------------------------------- warp/block reductions

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m) {
    uint32_t lo = uint32_t(v), hi = uint32_t(v >> 32);
    lo = __shfl_xor_sync(0xffffffffu, lo, m);
    hi = __shfl_xor_sync(0xffffffffu, hi, m);
    return (uint64_t(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl_idx_u64(uint64_t v, int src) {
    const uint32_t lo = __shfl_sync(0xffffffffu, uint32_t(v), src);
    const uint32_t hi = __shfl_sync(0xffffffffu, uint32_t(v >> 32), src);
    return (uint64_t(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
    for (int m = 16; m; m >>= 1) { uint64_t o = shfl_xor_u64(v, m); v = o > v ? o : v; }
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
    for (int m = 16; m; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
    for (int m = 16; m; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

// ----------------------------------------------------------------------------- clusters / DSMEM

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r; asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r)); return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r; asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r)); return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Split cluster barrier: arrive once this thread's accesses to peers' shared memory
// are done, wait (before exiting) until every peer has arrived.
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Programmatic dependent launch. griddep_wait: the grids this one was launched
// behind (with the programmatic stream serialization attribute) have completed and
// their writes are visible; a no-op for a grid launched without the attribute.
// griddep_launch_dependents: the next grid of the stream, if launched with the
// attribute, may start (its CTAs run their prologue, then wait in griddep_wait).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_u32(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// Address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
    uint32_t r; asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t addr) {
    uint32_t v; asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory"); return v;
}
__device__ __forceinline__ uint64_t ld_dsmem_u64(uint32_t addr) {
    uint64_t v; asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory"); return v;
}
__device__ __forceinline__ void st_dsmem_u64(uint32_t addr, uint64_t v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" :: "r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_dsmem_u32(uint32_t addr, uint32_t v) {
    uint32_t old; asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
    return old;
}

// ----------------------------------------------------------------------------- mbarrier + bulk copy

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// Bounded wait on an mbarrier phase. Returns false (and records ETIMEOUT) when
// the phase did not complete within limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int* status,
                                                  uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) { set_status(status, DARTREE_ETIMEOUT); return false; }
    }
    return true;
}
// 1-D bulk copy global -> own shared memory, completion counted on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// Prefetch of `bytes` (a multiple of 16, 16-byte aligned address) into L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src), "r"(bytes) : "memory");
}

// 1-D bulk copy from own shared memory into a peer CTA's shared memory; completion
// (bytes) is counted on the peer's mbarrier. remote_dst and remote_bar are
// shared::cluster addresses (mapa); all addresses and bytes multiples of 16.
__device__ __forceinline__ void bulk_s2cluster(uint32_t remote_dst, const void* src, uint32_t bytes,
                                               uint32_t remote_bar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(remote_dst), "r"(smem_u32(src)), "r"(bytes), "r"(remote_bar) : "memory");
}

// ----------------------------------------------------------------------------- grid barrier

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_gpu_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Grid-wide barrier on a monotonic counter; target = G * epoch. The wait is
// bounded: after limit_ns it records DARTREE_ETIMEOUT and gives up (later
// barriers of the same launch then skip their waits).
__device__ __forceinline__ void grid_barrier(unsigned* ctr, unsigned target, int* status, unsigned* timed_out,
                                             uint64_t limit_ns = kWaitLimitNs) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        red_release_gpu_add(ctr, 1u);
        if (!*timed_out) {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_gpu(ctr) < target) {
                if (globaltimer_ns() - t0 > limit_ns) {
                    set_status(status, DARTREE_ETIMEOUT);
                    *timed_out = 1;
                    break;
                }
            }
        }
    }
    __syncthreads();
}

// ----------------------------------------------------------------------------- block helpers

// Exclusive scan of one int per thread over a block of NT threads (NT multiple of 32, <= 1024).
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
    for (int o = 1; o < 32; o <<= 1) { int y = __shfl_up_sync(0xffffffffu, x, o); if (lane >= o) x += y; }
    if (lane == 31) warp_tot[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int w = lane < NT / 32 ? warp_tot[lane] : 0;
        int s = w;
        for (int o = 1; o < 32; o <<= 1) { int y = __shfl_up_sync(0xffffffffu, s, o); if (lane >= o) s += y; }
        if (lane < NT / 32) warp_tot[lane] = s - w;
        if (lane == 31) *total = s;
    }
    __syncthreads();
    int r = warp_tot[wid] + x - v;
    __syncthreads();
    return r;
}

// Bitonic sort of n (power of two) 64-bit keys in shared memory, descending.
template <int NT>
__device__ __forceinline__ void bitonic_sort_desc(uint64_t* a, int n) {
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += NT) {
                int ixj = i ^ j;
                if (ixj > i) {
                    uint64_t x = a[i], y = a[ixj];
                    bool first_half = (i & k) == 0;
                    if (first_half ? (x < y) : (x > y)) { a[i] = y; a[ixj] = x; }
                }
            }
            __syncthreads();
        }
    }
}

// Find the digit d (0..255) holding the rem-th largest element given a 256-bin
// histogram; rem is reduced by the count of larger digits. One warp.
__device__ __forceinline__ void pick_digit_warp(const uint32_t* hist, uint32_t& rem, uint32_t& digit) {
    const int lane = threadIdx.x & 31;
    // lane l owns bins 255-8l .. 248-8l (descending)
    uint32_t c[8], s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) { c[i] = hist[255 - 8 * lane - i]; s += c[i]; }
    uint32_t inc = s;
    for (int o = 1; o < 32; o <<= 1) { uint32_t y = __shfl_up_sync(0xffffffffu, inc, o); if (lane >= o) inc += y; }
    uint32_t exc = inc - s;
    bool mine = exc < rem && rem <= inc;
    uint32_t ballot = __ballot_sync(0xffffffffu, mine);
    uint32_t d = 0, r = rem;
    if (mine) {
        uint32_t acc = exc;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (acc + c[i] >= rem) { d = 255 - 8 * lane - i; r = rem - acc; break; }
            acc += c[i];
        }
    }
    int src = ballot ? __ffs(ballot) - 1 : 0;
    digit = __shfl_sync(0xffffffffu, d, src);
    rem = __shfl_sync(0xffffffffu, r, src);
    if (!ballot) { digit = 0xffffffffu; }
}

// Block-level selection of the N largest of n unique 64-bit keys (radix select,
// MSD 8 bits at a time). On return every thread knows (prefix, mask): a key is
// selected iff (key & mask) >= prefix... with the rule below. Exactly N keys satisfy
// sel(k) = ((k & mask) > prefix) || ((k & mask) == prefix).
// Returns false when the histogram did not account for N keys (internal error).
template <int NT>
__device__ bool block_select_top(const uint64_t* keys, int n, int N, uint32_t* hist, uint32_t* bcast,
                                 uint64_t& prefix_out, uint64_t& mask_out) {
    uint64_t prefix = 0, mask = 0;
    uint32_t rem = (uint32_t)N;
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += NT) hist[i] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += NT) {
            uint64_t k = keys[i];
            if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            uint32_t r = rem, d;
            pick_digit_warp(hist, r, d);
            if (threadIdx.x == 0) { bcast[0] = d; bcast[1] = r; bcast[2] = d == 0xffffffffu ? 0 : hist[d]; }
        }
        __syncthreads();
        uint32_t d = bcast[0];
        if (d == 0xffffffffu) return false;
        uint32_t r = bcast[1], cnt = bcast[2];
        __syncthreads();
        prefix |= uint64_t(d) << shift;
        mask |= uint64_t(0xffu) << shift;
        rem = r;
        if (cnt == rem) break;  // every key of this bin is selected
    }
    prefix_out = prefix;
    mask_out = mask;
    return true;
}

// Same contract as block_select_top, for keys that share long common prefixes
// (candidate scores cluster in a narrow range): the bytes above the highest bit
// where any two keys differ are skipped, and each warp adds one count per
// distinct digit (lanes with equal digits are merged with match.any), which keeps
// shared-memory atomics uncontended.
template <int NT>
__device__ bool block_select_top_agg(const uint64_t* keys, int n, int N, uint32_t* hist, uint32_t* bcast,
                                     uint64_t* orand, uint64_t& prefix_out, uint64_t& mask_out) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    // bits where the keys differ: OR of (key ^ keys[0])
    uint64_t x = 0;
    const uint64_t k0 = n > 0 ? keys[0] : 0ull;
    for (int i = threadIdx.x; i < n; i += NT) x |= keys[i] ^ k0;
    for (int m = 16; m; m >>= 1) x |= shfl_xor_u64(x, m);
    if (lane == 0) orand[wid] = x;
    __syncthreads();
    uint64_t diff = 0;
    for (int w = 0; w < NT / 32; ++w) diff |= orand[w];
    __syncthreads();
    if (diff == 0) {  // a single distinct key (n == 1)
        prefix_out = k0;
        mask_out = ~0ull;
        return N <= n;
    }
    const int top = 63 - __clzll(static_cast<long long>(diff));
    int shift = (top / 8) * 8;
    uint64_t mask = (shift + 8 >= 64) ? 0ull : (~0ull << (shift + 8));
    uint64_t prefix = k0 & mask;
    uint32_t rem = uint32_t(N);
    const int nfull = (n + NT - 1) / NT * NT;
    for (; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += NT) hist[i] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < nfull; i += NT) {
            const bool in = i < n && (keys[i] & mask) == prefix;
            const uint32_t dg = in ? uint32_t(keys[i] >> shift) & 255u : 256u;
            const uint32_t peers = __match_any_sync(0xffffffffu, dg);
            if (in && lane == __ffs(peers) - 1) atomicAdd(&hist[dg], uint32_t(__popc(peers)));
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            uint32_t r = rem, d;
            pick_digit_warp(hist, r, d);
            if (threadIdx.x == 0) { bcast[0] = d; bcast[1] = r; bcast[2] = d == 0xffffffffu ? 0 : hist[d]; }
        }
        __syncthreads();
        const uint32_t d = bcast[0], r = bcast[1], cnt = bcast[2];
        __syncthreads();
        if (d == 0xffffffffu) return false;
        prefix |= uint64_t(d) << shift;
        mask |= uint64_t(0xffu) << shift;
        rem = r;
        if (cnt == rem) break;  // every key of this bin is selected
    }
    prefix_out = prefix;
    mask_out = mask;
    return true;
}

__device__ __forceinline__ bool selected(uint64_t k, uint64_t prefix, uint64_t mask) {
    return (k & mask) >= prefix;
}

// Warp-wide maximum of unique 64-bit keys (redux on the high word, then on the
// low word among the lanes holding that high word).
__device__ __forceinline__ uint64_t warp_max_key64(uint64_t v) {
    const uint32_t hi = uint32_t(v >> 32), lo = uint32_t(v);
    const uint32_t mh = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t ml = __reduce_max_sync(0xffffffffu, hi == mh ? lo : 0u);
    return (uint64_t(mh) << 32) | ml;
}

// The n_keep largest keys of keys[0..n), descending, into out[0..n_keep) (all
// threads of the block; unique keys). Two levels: every warp keeps the best
// n_keep of its slice by rounds of "largest key below the previous one", then
// warp 0 merges the per-warp lists the same way.
template <int NT>
__device__ void block_top_keys(const uint64_t* keys, int n, int n_keep, uint64_t* cands, uint64_t* out) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int per = (n + (NT / 32) - 1) / (NT / 32);
    const int lo = wid * per, hi = min(n, lo + per);
    uint64_t prev = ~0ull;
    for (int k = 0; k < n_keep; ++k) {
        uint64_t best = 0;
        for (int f = lo + lane; f < hi; f += 32) {
            const uint64_t v = keys[f];
            if (v < prev && v > best) best = v;
        }
        best = warp_max_key64(best);
        prev = best;
        if (lane == 0) cands[wid * n_keep + k] = best;
    }
    __syncthreads();
    if (wid == 0) {
        const int m = (NT / 32) * n_keep;
        prev = ~0ull;
        for (int k = 0; k < n_keep; ++k) {
            uint64_t best = 0;
            for (int f = lane; f < m; f += 32) {
                const uint64_t v = cands[f];
                if (v < prev && v > best) best = v;
            }
            best = warp_max_key64(best);
            prev = best;
            if (lane == 0) out[k] = best;
        }
    }
    __syncthreads();
}

// Bitonic sort, descending, of the 32*EPL keys a warp holds (element lane*EPL + j
// in register j; EPL a power of two); partners in other lanes come by shuffles.
template <int EPL>
__device__ __forceinline__ void warp_bitonic_desc(uint64_t (&v)[EPL]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32 * EPL; k <<= 1) {
#pragma unroll
        for (int d = k >> 1; d >= 1; d >>= 1) {
            if (d >= EPL) {
#pragma unroll
                for (int j = 0; j < EPL; ++j) {
                    const int e = lane * EPL + j;
                    const uint64_t o = shfl_xor_u64(v[j], d / EPL);
                    const bool keep_max = ((e & d) == 0) == ((e & k) == 0);
                    v[j] = keep_max ? (v[j] > o ? v[j] : o) : (v[j] < o ? v[j] : o);
                }
            } else {
#pragma unroll
                for (int j = 0; j < EPL; ++j) {
                    if ((j & d) == 0) {
                        const bool desc = ((lane * EPL + j) & k) == 0;
                        const uint64_t x = v[j], y = v[j | d];
                        if (desc ? (x < y) : (x > y)) { v[j] = y; v[j | d] = x; }
                    }
                }
            }
        }
    }
}

// Top 16 of two descending 16-key lists held by the two half-warps (lane l of
// half-warp h holds element l of list h), sorted descending into lanes 0..15:
// the element-wise maximum of one list and the other reversed is bitonic and
// holds the 16 largest; a bitonic merge (distances 8, 4, 2, 1) sorts it.
__device__ __forceinline__ uint64_t xg_merge16(uint64_t v) {
    const int lane = threadIdx.x & 31;
    const uint32_t lo = __shfl_sync(0xffffffffu, uint32_t(v), 31 - lane);
    const uint32_t hi = __shfl_sync(0xffffffffu, uint32_t(v >> 32), 31 - lane);
    const uint64_t o = (uint64_t(hi) << 32) | lo;
    uint64_t c = v > o ? v : o;
#pragma unroll
    for (int d = 8; d; d >>= 1) {
        const uint64_t p = shfl_xor_u64(c, d);
        c = ((lane & d) == 0) ? (c > p ? c : p) : (c < p ? c : p);
    }
    return c;
}

}  // namespace dartree
