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
// (8 KB rows of a 151936-row table). Each stage holds a 128-element k-slice of
// every row (two 128-byte swizzle atoms, the layout tcgen05 reads); the four
// producer warps copy it with 16-byte cp.async, 16 lanes per row so that every
// instruction reads two whole 256-byte row segments, and arrive on the stage's
// mbarrier when their copies land. Warp 4 issues tcgen05.mma (M=128, N=32) into
// TMEM and frees the stage with tcgen05.commit; warps 0-3 then write z from
// TMEM. All waits are bounded.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace dartree {

constexpr int CC_BM = 128, CC_BN = 32, CC_BK = 128, CC_STAGES = 4, CC_NT = 160;
constexpr int CC_ATOMS = CC_BK / 64;                  // 64-element swizzle atoms per stage row
constexpr size_t CC_A_ATOM = size_t(CC_BM) * 128;     // 16 KB: 128 rows x 128 B
constexpr size_t CC_B_ATOM = size_t(CC_BN) * 128;     // 4 KB
constexpr size_t CC_A = CC_A_ATOM * CC_ATOMS;
constexpr size_t CC_B = CC_B_ATOM * CC_ATOMS;
constexpr size_t CC_STAGE = CC_A + CC_B;
constexpr size_t CC_BAR = CC_STAGE * CC_STAGES;
constexpr size_t CC_SMEM = CC_BAR + 8 * (2 * CC_STAGES + 1) + 16 + 128 * 4 + 1024;

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

    int* rowtok = reinterpret_cast<int*>(accum + 2);  // 128 candidate tokens of this tile (-1 = none)
    if (warp < 4) {
        const int c = c0 + int(threadIdx.x);
        rowtok[threadIdx.x] = c < K ? cand_tok[crow + c] : -1;
        asm volatile("bar.sync 1, 128;" ::: "memory");  // producers only
        // producers: per stage, warp w copies rows 32w..32w+31 (two rows per instruction,
        // 16 lanes x 16 B = one 256-byte row segment each) and 4 chunks of B per thread
        const int half = lane >> 4, j = lane & 15;       // j: 16-byte chunk within the 256-byte slice
        const uint32_t atom_off = uint32_t(j >> 3), jj = uint32_t(j & 7);
        const uint16_t* brow = uhl + (size_t(r) * CC_BN) * H;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % CC_STAGES;
            const uint32_t ph = uint32_t(kb / CC_STAGES) & 1u;
            if (!mbar_wait_bounded(&empty[s], ph ^ 1u, status)) break;
            const uint32_t sa = smem_u32(smem + s * CC_STAGE);
            const int k0 = kb * CC_BK + j * 8;
#pragma unroll 4
            for (int q = 0; q < 16; ++q) {
                const int row = warp * 32 + 2 * q + half;
                const int tk = rowtok[row];
                const uint32_t dst = sa + atom_off * uint32_t(CC_A_ATOM) + uint32_t(row) * 128u +
                                     ((jj ^ uint32_t(row & 7)) << 4);
                cp_async16(dst, E + size_t(tk < 0 ? 0 : tk) * H + k0, tk < 0 ? 0u : 16u);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int ch = int(threadIdx.x) * 4 + q;   // 512 chunks: 32 rows x 16
                const int br = ch >> 4, bj = ch & 15;
                const uint32_t dst = sa + uint32_t(CC_A) + uint32_t(bj >> 3) * uint32_t(CC_B_ATOM) +
                                     uint32_t(br) * 128u + ((uint32_t(bj & 7) ^ uint32_t(br & 7)) << 4);
                cp_async16(dst, brow + size_t(br) * H + kb * CC_BK + bj * 8, 16u);
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
#pragma unroll
            for (int kk = 0; kk < CC_BK / 16; ++kk) {
                // 16-element step kk: atom kk/4, 32-byte offset (kk%4) inside the atom
                const uint64_t da = tc::desc_sw128_kmajor(sa + uint32_t(kk >> 2) * uint32_t(CC_A_ATOM)) + 2u * (kk & 3);
                const uint64_t db =
                    tc::desc_sw128_kmajor(sa + uint32_t(CC_A) + uint32_t(kk >> 2) * uint32_t(CC_B_ATOM)) + 2u * (kk & 3);
                tc::mma_bf16(tmem, da, db, idesc, kb > 0 || kk > 0);
            }
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
// (H % 128 == 0: every stage is a whole 128-element k-slice)

int launch_contract_tc(const void* E, const uint16_t* uhl, const int32_t* cand_tok, const float* cand_val, float* z,
                       int C, int P, int K, int H, int L, int d, float inv_sqrt_h, int* status, cudaStream_t stream) {
    if (!contract_tc_supported(P, H)) return DARTREE_EUNSUPPORTED;
    if (cudaFuncSetAttribute(contract_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(CC_SMEM)) !=
        cudaSuccess)
        return DARTREE_ECUDA;
    dim3 grid((K + CC_BM - 1) / CC_BM, C);
    {
        KTimer kt_(KID_CONTRACT, stream);
        contract_tc_kernel<<<grid, CC_NT, CC_SMEM, stream>>>(static_cast<const uint16_t*>(E), uhl, cand_tok, cand_val, z,
                                                             P, K, H, L, d, inv_sqrt_h, status);
    }
    return cudaGetLastError() == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

}  // namespace dartree
