// tcgen05 GEMM for the per-depth parent projection (S3, DARTree blog post 3.1:
// the correction head runs on all surviving parents of a depth in one matrix
// operation): U[m, :] = h_m W_q^T for all C*P parents at once.
//
//   D[M, N] = A[M, K] . B[N, K]^T, A and B bf16 K-major, fp32 accumulation in TMEM.
//
// One 128 x BN tile per CTA (cta_group::1). Warp 0's elected thread streams
// 128 x 64 and BN x 64 tiles with TMA (128-byte swizzle) into a ring of as many
// stages as shared memory holds (4 for BN = 256, 6 for BN = 160 or 128);
// warp 1's elected thread issues tcgen05.mma (4 per 64-wide k block) and
// releases each stage with tcgen05.commit; all 8 warps then read the
// accumulator from TMEM (one row per thread; warps w and w + 4 share the TMEM
// lanes of rows 32 (w mod 4) ... and take alternate 32-column chunks) and write
// the epilogue:
//   mode 0: fp32 D (row-major, ld = N);
//   mode 1: the contraction's operand, U split into a bf16 pair (hi = bf16(u),
//           lo = bf16(u - hi)), row m = r*P + p going to rows r*32 + p and
//           r*32 + 16 + p of a [requests, 32, N] buffer;
//   mode 2: the same pair into two [M, N] buffers.
// The bf16 pairs are staged in shared memory (the drained operand ring) and
// written row by row, so that consecutive lanes store consecutive 16 bytes.
// Every mbarrier wait is bounded; a wait that runs out records DARTREE_ETIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace dartree {

constexpr int GT_BM = 128, GT_BK = 64, GT_NT = 256;

struct GemmOut {
    int mode;          // 0: fp32 d32; 1: hi/lo bf16 pairs into hilo (row remap); 2: hi -> hilo, lo -> lo2
    float* d32;
    uint16_t* hilo;
    uint16_t* lo2;     // mode 2: [M, N]
    int P;             // mode 1: rows per request (<= 16)
    GemmRowmax rm;     // rm.target null: none
};

// Maxima keys (ord(value) << 32 | ~token) of bf16 rows: warps 2 and 3 of every CTA
// (idle while the ring streams) take segments of the rows, spread over the grid,
// and merge them with one 64-bit atomic max per warp and segment. The keys were
// cleared by the launch before this one, whose completion griddep_wait ensures.
struct RowmaxSeg {
    int spr, per, nvr, nb, b;
};
__device__ __forceinline__ RowmaxSeg rowmax_seg(const GemmRowmax& rm) {
    RowmaxSeg g;
    g.nb = int(gridDim.x * gridDim.y);
    g.b = int(blockIdx.y * gridDim.x + blockIdx.x);
    g.spr = (g.nb + rm.rows - 1) / rm.rows;  // segments per row
    g.nvr = rm.V / 8;                        // 16-byte vectors per row
    g.per = (g.nvr + g.spr - 1) / g.spr;
    return g;
}
// Before the dependency wait (the rows are inputs, not written by the launch before):
// this CTA's segments into L2, one bulk prefetch per 16 KB.
__device__ void gemm_rowmax_prefetch(const GemmRowmax& rm) {
    const RowmaxSeg g = rowmax_seg(rm);
    for (int item = g.b; item < rm.rows * g.spr; item += g.nb) {
        const int row = item / g.spr, seg = item - row * g.spr;
        const int v0 = seg * g.per, v1 = min(g.nvr, v0 + g.per);
        const uint4* src = reinterpret_cast<const uint4*>(rm.target + size_t(row) * rm.V);
        for (int v = v0 + (threadIdx.x - 64) * 1024; v < v1; v += 64 * 1024)
            prefetch_l2_bulk(src + v, uint32_t(min(1024, v1 - v)) * 16u);
    }
}
__device__ void gemm_rowmax(const GemmRowmax& rm) {
    const int lane = threadIdx.x & 31, t = threadIdx.x - 64;  // 0..63
    const RowmaxSeg g = rowmax_seg(rm);
    constexpr int U = 8;  // loads in flight per thread
    for (int item = g.b; item < rm.rows * g.spr; item += g.nb) {
        const int row = item / g.spr, seg = item - row * g.spr;
        const int v0 = seg * g.per, v1 = min(g.nvr, v0 + g.per);
        const uint4* src = reinterpret_cast<const uint4*>(rm.target + size_t(row) * rm.V);
        uint64_t best = 0;
        for (int vb = v0 + t; vb < v1; vb += 64 * U) {
            uint4 w[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (vb + u * 64 < v1) w[u] = __ldg(src + vb + u * 64);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = vb + u * 64;
                if (v >= v1) break;
                const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t o = ord_bf16((ws[e >> 1] >> ((e & 1) * 16)) & 0xffffu);
                    const uint64_t k = (uint64_t(o) << 32) | (0xffffffffu - uint32_t(v * 8 + e));
                    best = k > best ? k : best;
                }
            }
        }
        best = warp_max_u64(best);
        if (lane == 0 && best) atomicMax(rm.keys + row, (unsigned long long)best);
    }
}

template <int BN>
struct GtSmem {
    static constexpr size_t A_BYTES = size_t(GT_BM) * GT_BK * 2;
    static constexpr size_t B_BYTES = size_t(BN) * GT_BK * 2;
    static constexpr size_t STAGE = A_BYTES + B_BYTES;      // a multiple of 1024 (swizzle atoms)
    // as many stages as fit next to the barriers (more bytes in flight per SM)
    static constexpr int STAGES = int((220 * 1024) / STAGE) > 8 ? 8 : int((220 * 1024) / STAGE);
    static constexpr size_t BAR = STAGE * STAGES;          // full[S], empty[S], accum
    static constexpr size_t SLOT = BAR + 8 * (2 * STAGES + 1);
    static constexpr size_t TOTAL = SLOT + 16 + 1024;      // + alignment slack
    static constexpr uint32_t TMEM_COLS = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
    // epilogue staging of the bf16 pair in the drained ring: rows padded by 16
    // bytes, so a warp's 16-byte row stores fall on all 32 banks
    static constexpr int EPI_PITCH = BN * 2 + 16;
    static_assert(size_t(2) * GT_BM * EPI_PITCH <= BAR, "epilogue staging fits in the operand ring");
};

template <int BN>
__global__ void __launch_bounds__(GT_NT, 1) gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                                                                const __grid_constant__ CUtensorMap tmB, int M,
                                                                int N, int K, GemmOut out, int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using L = GtSmem<BN>;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR);
    uint64_t* empty = full + L::STAGES;
    uint64_t* accum = empty + L::STAGES;
    uint32_t* slot = reinterpret_cast<uint32_t*>(smem + L::SLOT);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * GT_BM, n0 = blockIdx.x * BN;
    const int nk = (K + GT_BK - 1) / GT_BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < L::STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        mbar_init(accum, 1);
        fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(slot, L::TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *slot;

    griddep_launch_dependents();
    if ((warp == 2 || warp == 3) && out.rm.target) gemm_rowmax_prefetch(out.rm);
    if (warp == 0 && lane == 0) {
        // producer: TMA ring. B is not written by the previous kernel of the stream:
        // the first stages' B tiles load before the dependency wait, A after it.
        const int npre = nk < L::STAGES ? nk : L::STAGES;
        for (int kb = 0; kb < npre; ++kb) {
            mbar_arrive_expect_tx(&full[kb], uint32_t(L::STAGE));
            tc::tma_load_2d(smem + kb * L::STAGE + L::A_BYTES, &tmB, kb * GT_BK, n0, &full[kb]);
        }
        griddep_wait();
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % L::STAGES;
            const uint32_t ph = uint32_t(kb / L::STAGES) & 1u;
            uint8_t* sa = smem + s * L::STAGE;
            if (kb >= npre) {
                if (!mbar_wait_bounded(&empty[s], ph ^ 1u, status)) break;
                mbar_arrive_expect_tx(&full[s], uint32_t(L::STAGE));
                tc::tma_load_2d(sa + L::A_BYTES, &tmB, kb * GT_BK, n0, &full[s]);
            }
            tc::tma_load_2d(sa, &tmA, kb * GT_BK, m0, &full[s]);
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer (its bounded waits start once the operands can arrive)
        griddep_wait();
        constexpr uint32_t idesc = tc::idesc_bf16_f32(GT_BM, BN);
        bool ok = true;
        for (int kb = 0; kb < nk && ok; ++kb) {
            const int s = kb % L::STAGES;
            const uint32_t ph = uint32_t(kb / L::STAGES) & 1u;
            if (!mbar_wait_bounded(&full[s], ph, status)) { ok = false; break; }
            tc::fence_after_sync();
            const uint32_t sa = smem_u32(smem + s * L::STAGE);
            const uint64_t da = tc::desc_sw128_kmajor(sa);
            const uint64_t db = tc::desc_sw128_kmajor(sa + uint32_t(L::A_BYTES));
#pragma unroll
            for (int kk = 0; kk < GT_BK / 16; ++kk)  // 16 elements = 32 B = +2 in the encoded address
                tc::mma_bf16(tmem, da + 2u * kk, db + 2u * kk, idesc, kb > 0 || kk > 0);
            tc::mma_commit(&empty[s]);
        }
        tc::mma_commit(accum);
    }
    __syncwarp();
    griddep_wait();  // (the producer's wait already covers the operands; this orders the stores)
    if ((warp == 2 || warp == 3) && out.rm.target) gemm_rowmax(out.rm);

    // epilogue: TMEM -> registers -> global. Warps w and w + 4 share TMEM lanes
    // 32 (w mod 4) ... and take alternate 32-column chunks of their rows.
    const bool have = __syncthreads_and(mbar_wait_bounded(accum, 0, status) ? 1 : 0) != 0;
    tc::fence_after_sync();
    const int quarter = warp & 3, cfirst = (warp >> 2) * 32;
    const int m = m0 + quarter * 32 + lane;
    const uint32_t trow = tmem + (uint32_t(quarter * 32) << 16);
    if (out.mode == 0) {
        for (int c0 = cfirst; c0 < BN; c0 += 64) {
            uint32_t r[32];
            tc::tmem_ld32(trow + uint32_t(c0), r);
            const int n = n0 + c0;
            if (!have || m >= M || n >= N) continue;
            float4* dst = reinterpret_cast<float4*>(out.d32 + size_t(m) * N + n);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                     __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        }
    } else if (have) {
        // bf16 pair: every thread splits its row into shared memory (the operand
        // ring is drained: every stage was consumed by the MMAs that completed),
        // then the tile is written row by row, consecutive lanes on consecutive
        // 16-byte chunks of a row
        constexpr int PITCH = L::EPI_PITCH;
        uint8_t* sh = smem;
        uint8_t* sl = smem + GT_BM * PITCH;
        const int rl = quarter * 32 + lane;
        for (int c0 = cfirst; c0 < BN; c0 += 64) {
            uint32_t r[32];
            tc::tmem_ld32(trow + uint32_t(c0), r);
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {  // two columns per conversion (each rounded to nearest even)
                const float u0 = __uint_as_float(r[2 * j]), u1 = __uint_as_float(r[2 * j + 1]);
                const __nv_bfloat162 h = __floats2bfloat162_rn(u0, u1);
                const __nv_bfloat162 l = __floats2bfloat162_rn(u0 - __low2float(h), u1 - __high2float(h));
                hi[j] = *reinterpret_cast<const uint32_t*>(&h);
                lo[j] = *reinterpret_cast<const uint32_t*>(&l);
            }
            uint4* dh = reinterpret_cast<uint4*>(sh + size_t(rl) * PITCH + size_t(c0) * 2);
            uint4* dl = reinterpret_cast<uint4*>(sl + size_t(rl) * PITCH + size_t(c0) * 2);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                dh[j] = make_uint4(hi[4 * j], hi[4 * j + 1], hi[4 * j + 2], hi[4 * j + 3]);
                dl[j] = make_uint4(lo[4 * j], lo[4 * j + 1], lo[4 * j + 2], lo[4 * j + 3]);
            }
        }
        __syncthreads();
        constexpr int CPR = BN / 8;  // 16-byte chunks per row
        for (int i = threadIdx.x; i < GT_BM * CPR; i += GT_NT) {
            const int rr = i / CPR, cc = i - rr * CPR, mm = m0 + rr;
            if (mm >= M || n0 >= N) continue;
            const uint4 vh = *reinterpret_cast<const uint4*>(sh + size_t(rr) * PITCH + cc * 16);
            const uint4 vl = *reinterpret_cast<const uint4*>(sl + size_t(rr) * PITCH + cc * 16);
            uint16_t* gh;
            uint16_t* gl;
            if (out.mode == 2) {
                gh = out.hilo + size_t(mm) * N + n0;
                gl = out.lo2 + size_t(mm) * N + n0;
            } else {
                const int rq = mm / out.P, p = mm % out.P;
                gh = out.hilo + (size_t(rq) * 32 + p) * N + n0;
                gl = out.hilo + (size_t(rq) * 32 + 16 + p) * N + n0;
            }
            reinterpret_cast<uint4*>(gh)[cc] = vh;
            reinterpret_cast<uint4*>(gl)[cc] = vl;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, L::TMEM_COLS);
}

// --------------------------------------------------------------------------- host

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool make_tensor_map_bf16(CUtensorMap* map, const void* base, int rows, int cols, int box_cols, int box_rows,
                          int swizzle_bytes) {
    auto fn = encode_fn();
    if (!fn) return false;
    CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
    if (swizzle_bytes == 32) sw = CU_TENSOR_MAP_SWIZZLE_32B;
    else if (swizzle_bytes == 64) sw = CU_TENSOR_MAP_SWIZZLE_64B;
    else if (swizzle_bytes == 128) sw = CU_TENSOR_MAP_SWIZZLE_128B;
    else if (swizzle_bytes != 0) return false;
    cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
    cuuint32_t box[2] = {cuuint32_t(box_cols), cuuint32_t(box_rows)};
    cuuint32_t es[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Operand tiles of the GEMM: box = 64 columns x box_rows rows, 128-byte swizzle.
static bool make_map(CUtensorMap* map, const void* base, int rows, int cols, int box_rows) {
    return make_tensor_map_bf16(map, base, rows, cols, GT_BK, box_rows, 128);
}

bool gemm_tc_supported(int M, int N, int K) {
    return M > 0 && N > 0 && K > 0 && N % 128 == 0 && K % 8 == 0 && encode_fn() != nullptr;
}

template <int BN>
static int launch_gemm_bn(const void* A, const void* B, int M, int N, int K, const GemmOut& o, int* status,
                          cudaStream_t stream, bool pdl) {
    CUtensorMap ta, tb;
    if (!make_map(&ta, A, M, K, GT_BM) || !make_map(&tb, B, N, K, BN)) return DARTREE_ECUDA;
    const size_t smem = GtSmem<BN>::TOTAL;
    auto kern = gemm_bf16_tc_kernel<BN>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
        return DARTREE_ECUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(N / BN, (M + GT_BM - 1) / GT_BM);
    cfg.blockDim = dim3(GT_NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e;
    {
        KTimer kt_(KID_GEMM, stream);
        e = cudaLaunchKernelEx(&cfg, kern, ta, tb, M, N, K, o, status);
    }
    return e == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

int launch_gemm_bf16_tc(const void* A, const void* B, int M, int N, int K, int mode, float* d32, uint16_t* hilo,
                        int P, int* status, cudaStream_t stream, uint16_t* lo2, bool pdl, const GemmRowmax* rm,
                        bool shared_sms) {
    if (!gemm_tc_supported(M, N, K)) return DARTREE_EUNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) % 16) return DARTREE_EINVAL;
    if (mode == 1 && (P < 1 || P > 16 || !hilo)) return DARTREE_EINVAL;
    if (mode == 0 && !d32) return DARTREE_EINVAL;
    if (mode == 2 && (!hilo || !lo2)) return DARTREE_EINVAL;
    if (rm && (!rm->target || !rm->keys || rm->rows < 1 || rm->V % 8 != 0 ||
               reinterpret_cast<uintptr_t>(rm->target) % 16 != 0))
        return DARTREE_EINVAL;
    GemmOut o{mode, d32, hilo, lo2, P, rm ? *rm : GemmRowmax{nullptr, 0, 0, nullptr}};
    // Tile width: the operand bytes a CTA streams per k block (its ingest time)
    // times the number of waves of CTAs over the SMs, smallest wins.
    const int mt = (M + GT_BM - 1) / GT_BM, sms = num_sms();
    int best = 128;
    long best_cost = -1;
    for (int bn : {256, 160, 128}) {
        if (N % bn != 0) continue;
        const long tiles = long(mt) * (N / bn), waves = (tiles + sms - 1) / sms;
        // beside other work (the per-depth projection of one half of a split batch,
        // next to the other half's contraction) the operand bytes all its CTAs stream
        // count, not its own span
        const long cost = shared_sms ? tiles * (GT_BM + bn) : waves * (GT_BM + bn);
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = bn; }
    }
    if (best == 256) return launch_gemm_bn<256>(A, B, M, N, K, o, status, stream, pdl);
    if (best == 160) return launch_gemm_bn<160>(A, B, M, N, K, o, status, stream, pdl);
    return launch_gemm_bn<128>(A, B, M, N, K, o, status, stream, pdl);
}

}  // namespace dartree
