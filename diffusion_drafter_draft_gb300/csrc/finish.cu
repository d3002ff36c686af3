// S8-S10 for one request per CTA when the supertree holds at most 256 nodes
// (finish.cuh): the supertree is read from global memory.
#include "common.cuh"
#include "finish.cuh"
#include "kernels.h"

namespace dartree {

template <bool WALK>
__global__ void __launch_bounds__(FN_NT) finish_kernel(int L, int W, int B, const int32_t* __restrict__ st_tok,
                                                       const int32_t* __restrict__ st_par,
                                                       const float* __restrict__ st_s,
                                                       const int32_t* __restrict__ st_n,
                                                       const int32_t* __restrict__ anchor, FinishOut o,
                                                       int* status) {
    extern __shared__ __align__(16) uint8_t smem[];
    griddep_wait();  // the supertree comes from the kernel before this one
    const int r = blockIdx.x, n = L * W, q = threadIdx.x;
    const size_t base = size_t(r) * L * W;
    // ---- keys of the supertree nodes (0 = no node)
    uint64_t key = 0;
    int s_tok = -1, s_par = -1, dm1 = 0;
    float s_sc = 0.f;
    if (q < n) {
        dm1 = q / W;
        const int k = q % W;
        if (k < st_n[size_t(r) * L + dm1]) {
            s_sc = st_s[base + q];
            s_tok = st_tok[base + q];
            s_par = st_par[base + q];
            key = finish_key(ord_f32(s_sc + 0.f), dm1, k);
        }
    }
    finish_request<WALK>(r, L, W, B, smem, key, s_tok, s_par, s_sc, dm1, anchor[r], o, status);
}

bool finish_supported(int L, int W) { return L * W <= FN_NT; }

int launch_finish(int C, int L, int W, int B, const int32_t* st_tok, const int32_t* st_par, const float* st_s,
                  const int32_t* st_n, const int32_t* anchor, int32_t* tok, int32_t* par, int32_t* depth,
                  float* score, int32_t* n_nodes, uint8_t* mask, int32_t* pos, const unsigned long long* rowkeys,
                  int32_t* accepted, int32_t* path, int32_t* bonus, int* status, cudaStream_t stream, bool pdl) {
    if (C == 0) return DARTREE_OK;
    if (!finish_supported(L, W)) return DARTREE_EUNSUPPORTED;
    const size_t smem = fn_smem(L, B).bytes;
    const bool walk = rowkeys != nullptr;
    auto kern = walk ? finish_kernel<true> : finish_kernel<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
        return DARTREE_ECUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(C));
    cfg.blockDim = dim3(FN_NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const FinishOut o{tok, par, depth, score, n_nodes, mask, pos, rowkeys, accepted, path, bonus};
    cudaError_t e;
    {
        KTimer kt_(KID_FINISH, stream);
        e = cudaLaunchKernelEx(&cfg, kern, L, W, B, st_tok, st_par, st_s, st_n, anchor, o, status);
    }
    return e == cudaSuccess ? DARTREE_OK : DARTREE_ECUDA;
}

}  // namespace dartree
