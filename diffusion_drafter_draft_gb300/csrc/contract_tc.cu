// S4 on tensor cores for large batches: the parent x candidate contraction of one
// depth (DARTree blog post, 3.1, depth-wise expansion), for every request r:
//
//   z[r, p, c] = L^base[r, d-1, c] + <u_{r,p}, E[cand_{r,c}]> / sqrt(H)
//
// as D[c, j] = E[cand_c] . B_r[j]^T with B_r = [u_hi(p=0..15); u_lo(p=0..15)]
// (u split into a bf16 pair by the projection's epilogue, so u is used to about
// 16 significant bits), and z = cand + (D[c, p] + D[c, 16+p]) / sqrt(H).
//
// One CTA per (request, 128-candidate tile). The candidate rows are a gather
// (8 KB rows of a 151936-row table), so four producer warps copy each row's
// 128-byte k-slice with 16-byte cp.async into a 128-byte-swizzled stage (the
// layout tcgen05 reads) and arrive on the stage's mbarrier when their copies
// land; warp 4 issues tcgen05.mma (M=128, N=32) into TMEM and frees the stage
// with tcgen05.commit; warps 0-3 then write z from TMEM. All waits are bounded.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace dartree {

constexpr int CC_BM = 128, CC_BN = 32, CC_BK = 64, CC_STAGES = 4, CC_NT = 160;
constexpr size_t CC_A = size_t(CC_BM) * CC_BK * 2;   // 16 KB
constexpr size_t CC_B = size_t(CC_BN) * CC_BK * 2;   // 4 KB
constexpr size_t CC_STAGE = CC_A + CC_B;
constexpr size_t CC_BAR = CC_STAGE * CC_STAGES;
constexpr size_t CC_SMEM = CC_BAR + 8 * (2 * CC_STAGES + 1) + 16 + 1024;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// Arrive on `bar` when all of this thread's earlier cp.async copies have landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_u32(bar)) : "memory");
}

__global__ void __launch_bounds__(CC_NT, 1) contract_tc_kernel(const uint16_t* __restrict__ E,
                                                               const uint16_t* __restrict__ uhl,  // [C, 32, H]
                                                               const int32_t* __restrict__ cand_tok,
                                                               const float* __restrict__ cand_val, float* __restrict__ z,
                                                               int P, int K, int H, int L, int d, float inv_sqrt_h,
                                                               int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + CC_BAR);
    uint64_t* empty = full + CC_STAGES;
    uint64_t* accum = empty + CC_STAGES;
    uint32_t* slot = reinterpret_cast<uint32_t*>(accum + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.y, c0 = blockIdx.x * CC_BM;
    const size_t crow = (size_t(r) * L + (d - 1)) * K;
    const int nk = H / CC_BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < CC_STAGES; ++s) { mbar_init(&full[s], 128); mbar_init(&empty[s], 1); }
        mbar_init(accum, 1);
        fence_mbar_init();
    }
    if (warp == 4) tc::tmem_alloc(slot, CC_BN);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *slot;

    if (warp < 4) {
        // producers: thread t copies candidate row t (8 x 16 B per k block) and 2 chunks of B
        const int i = threadIdx.x;
        const int c = c0 + i;
        const bool valid = c < K;
        const uint16_t* arow = E + size_t(cand_tok[crow + (valid ? c : 0)]) * H;
        const uint16_t* brow = uhl + (size_t(r) * CC_BN) * H;
        const uint32_t sw = uint32_t(i & 7);
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % CC_STAGES;
            const uint32_t ph = uint32_t(kb / CC_STAGES) & 1u;
            if (!mbar_wait_bounded(&empty[s], ph ^ 1u, status)) break;
            const uint32_t sa = smem_u32(smem + s * CC_STAGE);
            const uint16_t* src = arow + kb * CC_BK;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                cp_async16(sa + uint32_t(i) * 128u + ((uint32_t(j) ^ sw) << 4), src + j * 8, valid ? 16u : 0u);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int ch = i * 2 + q;          // 256 chunks: 32 rows x 8
                const int br = ch >> 3, bj = ch & 7;
                cp_async16(sa + uint32_t(CC_A) + uint32_t(br) * 128u + ((uint32_t(bj) ^ uint32_t(br & 7)) << 4),
                           brow + size_t(br) * H + kb * CC_BK + bj * 8, 16u);
            }
            cp_async_arrive(&full[s]);
        }
    } else if (lane == 0) {
        // MMA issuer
        constexpr uint32_t idesc = tc::idesc_bf16_f32(CC_BM, CC_BN);
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % CC_STAGES;
            const uint32_t ph = uint32_t(kb / CC_STAGES) & 1u;
            if (!mbar_wait_bounded(&full[s], ph, status)) break;
            fence_proxy_async_smem();  // cp.async writes -> tensor-core reads
            tc::fence_after_sync();
            const uint32_t sa = smem_u32(smem + s * CC_STAGE);
            const uint64_t da = tc::desc_sw128_kmajor(sa);
            const uint64_t db = tc::desc_sw128_kmajor(sa + uint32_t(CC_A));
#pragma unroll
            for (int kk = 0; kk < CC_BK / 16; ++kk)
                tc::mma_bf16(tmem, da + 2u * kk, db + 2u * kk, idesc, kb > 0 || kk > 0);
            tc::mma_commit(&empty[s]);
        }
        tc::mma_commit(accum);
    }
    __syncwarp();

    if (warp < 4) {
        const bool have = mbar_wait_bounded(accum, 0, status);
        tc::fence_after_sync();
        uint32_t v[32];
        tc::tmem_ld32(tmem + (uint32_t(warp * 32) << 16), v);
        const int c = c0 + warp * 32 + lane;
        if (have && c < K) {
            const float base = cand_val[crow + c];
#pragma unroll
            for (int p = 0; p < 16; ++p)
                if (p < P)
                    z[(size_t(r) * P + p) * K + c] =
                        base + (__uint_as_float(v[p]) + __uint_as_float(v[16 + p])) * inv_sqrt_h;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 4) tc::tmem_dealloc(tmem, CC_BN);
}

bool contract_tc_supported(int P, int H) { return P >= 1 && P <= 16 && H % CC_BK == 0; }

int launch_contract_tc(const void* E, const uint16_t* uhl, const int32_t* cand_tok, const float* cand_val, float* z,
                       int C, int P, int K, int H, int L, int d, float inv_sqrt_h, int* status, cudaStream_t stream) {
    if (!contract_tc_supported(P, H)) return DARTREE_EUNSUPPORTED;
    if (cudaFuncSetAttribute(contract_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(CC_SMEM)) !=
        cudaSuccess)
        return DARTREE_ECUDA;
    dim3 grid((K + CC_BM - 1) / CC_BM, C);
    contract_tc_kernel<<<grid, CC_NT, CC_SMEM, stream>>>(static_cast<const uint16_t*>(E), uhl, cand_tok, cand_val, z,
                                                         P, K, H, L, d, inv_sqrt_h, status);
    return cudaGetLastError() == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

}  // namespace dartree
