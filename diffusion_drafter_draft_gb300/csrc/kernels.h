// Host-side launchers of the DARTree kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <stdint.h>

namespace dartree {

// Side streams for forks inside one call (0: target-row maxima of a round, 1: the
// second half of a large batch's expansion), one set per (device, caller stream),
// so that callers on different streams never wait for each other's forks.
// Enqueue under side_mutex().
struct SideStreams {
    int dev = -1;
    cudaStream_t caller = nullptr;
    cudaStream_t s[2] = {nullptr, nullptr};
    cudaEvent_t fork[2] = {nullptr, nullptr}, join[2] = {nullptr, nullptr};
    bool ok = false;
};
// The set of `caller` on the current device (created on its first use); nullptr
// when it cannot be created or the table of sets is full (the call then runs
// without forks, on the caller's stream alone).
SideStreams* side_streams(cudaStream_t caller);
std::recursive_mutex& side_mutex();

// Kernel ids of the launch timing (dartree_timing): one per kernel family.
enum KernelId {
    KID_TOPK_ROWS = 0, KID_TOPK_STREAM, KID_GEMM, KID_CONTRACT, KID_EXPAND_G, KID_GATHER, KID_SELECT,
    KID_STATE, KID_HEAP, KID_FINISH, KID_PRUNE, KID_MASK, KID_ROWMAX, KID_WALK, KID_ROWSAMPLE, KID_LMHEAD,
    KID_LMMERGE, KID_ATTN_PREP, KID_ATTN, KID_ATTN_COMBINE, KID_OTHER,
    KID_COUNT
};
// Brackets the launches of its scope with timing events when timing is enabled.
struct KTimer {
    KTimer(int id, cudaStream_t s);
    ~KTimer();
    KTimer(const KTimer&) = delete;
    KTimer& operator=(const KTimer&) = delete;
    int id_;
    cudaStream_t s_;
    void* b_;
};

int num_sms();

// Launch attribute of programmatic dependent launch: the kernel may start while the
// previous kernel of the stream finishes; it calls griddep_wait before it touches
// anything that kernel (or one before it) writes.
inline cudaLaunchAttribute pdl_attribute() {
    cudaLaunchAttribute a{};
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
}

// Rows of a bf16 [V, H] matrix copied, per top-K row r and rank i, to out[r*K + i]
// by the top-K launch itself (the candidate rows of the candidate-side projection).
struct TopkGather {
    const uint16_t* E;
    int H;
    uint16_t* out;
    const void* pre = nullptr;  // a range the launch after this one reads (16-byte aligned, a multiple of
    size_t pre_bytes = 0;       // 16 bytes): prefetched into L2 while the rows stream, or none
};

// Maxima keys (ord(value) << 32 | ~index) of per-position target rows [rows, V],
// the same dtype as the top-K rows, computed by the top-K launch itself; with
// zero_only the launch only clears keys (a later launch takes the maxima).
struct TopkRowmax {
    const void* target;
    unsigned long long* keys;  // [rows]
    bool zero_only;
};

// Per-position target row maxima taken by the otherwise idle warps of the
// candidate-side projection GEMM (bf16 rows [rows, V], keys cleared beforehand).
struct GemmRowmax {
    const uint16_t* target;
    int rows, V;
    unsigned long long* keys;
};

// S1: top-K of `rows` rows of V values. With g, *gathered tells whether the rows of
// g->E were copied too, with rm, *rm_done whether the target row maxima were
// written (only some launch shapes do either; otherwise the caller does).
int launch_topk(const void* x, int rows, int V, int K, int dtype, int32_t* tok, float* val, int* status,
                cudaStream_t stream, const TopkGather* g = nullptr, bool* gathered = nullptr,
                const TopkRowmax* rm = nullptr, bool* rm_done = nullptr);

// Outputs of S8-S10 (the tree arrays of dartree_tree; mask/pos and the walk are optional).
struct FinishOut {
    int32_t* tok;
    int32_t* par;
    int32_t* depth;
    float* score;
    int32_t* n_nodes;
    uint8_t* mask;                      // null: no mask and position ids
    int32_t* pos;
    const unsigned long long* rowkeys;  // [C, L] per-position target row maxima; null: no walk
    int32_t* accepted;
    int32_t* path;
    int32_t* bonus;
};

struct ExpandArgs {
    const void* E;
    const void* Wq;
    int V, H, dtype;
    int C, L, K, W;
    float beta;
    const void* hidden;       // [C, L, H]
    const int32_t* anchor;    // [C]
    const int32_t* cand_tok;  // [C, L, K]
    const float* cand_val;    // [C, L, K]
    int32_t* st_tok;          // [C, L, W]
    int32_t* st_par;          // [C, L, W]
    float* st_s;              // [C, L, W]
    int32_t* st_n;            // [C, L]
    void* hbuf[2];            // [C, W, H] storage type, ping-pong
    float* sbuf[2];           // [C, W]
    float* U;                 // [C*W, H]
    float* z;                 // [C, W, K]
    uint16_t* uhl;            // [C, 32, H] bf16 hi/lo projection rows (tensor-core contraction), or null
    const void* WqT;          // [H, H] W_q transposed (prepared head), or null
    uint16_t* Eg;             // [C*L*K, H] gathered candidate rows (candidate-side projection path)
    bool eg_ready;            // Eg already holds E[cand_tok] (copied by the top-K launch)
    uint16_t* Ghi;            // [C*L*K, H] G = E[cand] W_q, bf16 high part
    uint16_t* Glo;            // [C*L*K, H] low part
    int g_rows;               // rows the Eg/G buffers hold (0: path unavailable)
    bool split;               // one part of a batch split across streams (per-depth path)
    int* status;
    // Optional per-position target row maxima (bf16 rows [C*L, V]) taken inside the
    // candidate-side path's GEMM launch (keys cleared by the top-K launch)
    const void* rm_target;
    unsigned long long* rm_keys;
    // Optional S8-S10 in the same launch (candidate-side path, L*W <= 256): the
    // path that takes it sets *fin_done; otherwise the caller runs them.
    int B;
    const FinishOut* fin;
    bool* fin_done;
};

// 2-D bf16 TMA descriptor of a row-major [rows, cols] tensor, box box_cols x box_rows,
// swizzle 0 (none), 32, 64 or 128 bytes. False when the driver refuses it.
bool make_tensor_map_bf16(CUtensorMap* map, const void* base, int rows, int cols, int box_cols, int box_rows,
                          int swizzle_bytes);
// out[m] = E[idx[m]] for m < M (rows of H bf16, H / 8 <= 768).
int launch_gather_rows(const uint16_t* E, const int32_t* idx, int H, int M, uint16_t* out, cudaStream_t stream);

// Node-by-node best-first search (one head evaluation per popped node) over the
// candidates of S1 and the candidate-side G pair; outputs [C, B] in pop order.
bool heap_supported(int H, int K, int B);
int launch_heap_search(const void* E, const void* hidden, const int32_t* anchor, const int32_t* cand_tok,
                       const float* cand_val, const uint16_t* Ghi, const uint16_t* Glo, int C, int H, int L, int K,
                       int B, float beta, uint16_t* hws, int32_t* tok, int32_t* par, int32_t* depth, float* score,
                       int* status, cudaStream_t stream);

// Transpose of an H x H bf16 matrix (head preparation).
int launch_transpose_bf16(const void* src, void* dst, int H, cudaStream_t stream);

// Candidate-side projection path (small batches, prepared bf16 head); *launched = false
// when the shape does not fit it. expand_g_fits: whether it would launch.
bool expand_g_fits(const ExpandArgs& a);
int try_launch_expand_g(const ExpandArgs& a, cudaStream_t stream, bool* launched);

// tcgen05 GEMM D[M,N] = A[M,K] . B[N,K]^T (bf16 in, fp32 accumulate).
// mode 0: fp32 d32 [M,N]; mode 1: bf16 hi/lo pairs into hilo [M/P, 32, N];
// mode 2: bf16 hi into hilo [M,N] and lo into lo2 [M,N].
// pdl: programmatic dependent launch (A may be written by the previous kernel; B and
// the outputs are not touched by it).
bool gemm_tc_supported(int M, int N, int K);
// shared_sms: the launch runs beside other work (the other half of a split batch):
// its tile width is chosen by the operand bytes all its CTAs stream, not by its span.
int launch_gemm_bf16_tc(const void* A, const void* B, int M, int N, int K, int mode, float* d32, uint16_t* hilo,
                        int P, int* status, cudaStream_t stream, uint16_t* lo2 = nullptr, bool pdl = false,
                        const GemmRowmax* rm = nullptr, bool shared_sms = false);

// tcgen05 contraction of one depth: z[r,p,c] from gathered candidate rows and uhl.
bool contract_tc_supported(int P, int H);
int launch_contract_tc(const void* E, const uint16_t* uhl, const int32_t* cand_tok, const float* cand_val, float* z,
                       int C, int P, int K, int H, int L, int d, float inv_sqrt_h, int* status, cudaStream_t stream);

// S2-S7 over all depths.
int launch_expand(const ExpandArgs& a, cudaStream_t stream);

// S8: deferred prune.
int launch_prune(int C, int L, int W, int B, const int32_t* st_tok, const int32_t* st_par, const float* st_s,
                 const int32_t* st_n, const int32_t* anchor, int32_t* tok, int32_t* par, int32_t* depth,
                 float* score, int32_t* n_nodes, int* status, cudaStream_t stream);

// S9: mask and position ids.
int launch_mask(int C, int L, int B, const int32_t* par, const int32_t* depth, const int32_t* n_nodes,
                uint8_t* mask, int32_t* pos, cudaStream_t stream);

// S10: verification.
// Row maxima (value, ~token) of per-position target rows [C*L, V] (keys zeroed first).
int launch_rowmax_position(int C, int L, int V, int dtype, const void* target, unsigned long long* keys,
                           cudaStream_t stream);

// S10 walk over per-position row maxima computed by launch_rowmax_position.
// status (may be null): DARTREE_EINTERNAL when the tree is malformed.
int launch_walk_position(int C, int L, int B, const int32_t* tok, const int32_t* par, const int32_t* depth,
                         const int32_t* n_nodes, const unsigned long long* keys, int32_t* accepted, int32_t* path,
                         int32_t* bonus, int* status, cudaStream_t stream);

// S8-S9 (and S10 with per-position row maxima when rowkeys is not null) for one
// request per CTA; supertrees of at most 256 nodes (finish_supported).
bool finish_supported(int L, int W);
int launch_finish(int C, int L, int W, int B, const int32_t* st_tok, const int32_t* st_par, const float* st_s,
                  const int32_t* st_n, const int32_t* anchor, int32_t* tok, int32_t* par, int32_t* depth,
                  float* score, int32_t* n_nodes, uint8_t* mask, int32_t* pos, const unsigned long long* rowkeys,
                  int32_t* accepted, int32_t* path, int32_t* bonus, int* status, cudaStream_t stream,
                  bool pdl = false);

// S10 (row maxima + walk); status (may be null): DARTREE_EINTERNAL when the tree is malformed.
int launch_verify(int C, int L, int B, const int32_t* tok, const int32_t* par, const int32_t* depth,
                  const int32_t* n_nodes, const void* target, int rows_mode, int V, int dtype,
                  unsigned long long* keys, int32_t* accepted, int32_t* path, int32_t* bonus, int* status,
                  cudaStream_t stream);

// S10 at a temperature T > 0: the same walks on Gumbel-max draws (Philox4x32-10 noise).
int launch_verify_sample(int C, int L, int B, const int32_t* tok, const int32_t* par, const int32_t* depth,
                         const int32_t* n_nodes, const void* target, int rows_mode, int V, int dtype, float temp,
                         uint64_t seed, unsigned long long* keys, int32_t* accepted, int32_t* path, int32_t* bonus,
                         int* status, cudaStream_t stream);

// The LM head fused with S1: tok/val [R, K] = top-K of hidden [R, H] x W[V, H]^T per
// row (bf16 operands, fp32 logits); part: lmhead_part_bytes of scratch.
bool lmhead_supported(int R, int V, int H, int K);
size_t lmhead_part_bytes(int R, int V, int K);
int launch_lmhead_topk(const void* hidden, const void* W, int R, int V, int H, int K, int32_t* tok, float* val,
                       unsigned long long* part, int* status, cudaStream_t stream);

// Tree attention of the verification pass (one layer, D = 128): workspace plan and launch.
struct AttnPlan {
    int nchunk, per, mtiles;              // key-block chunks per row tile, blocks per chunk, row tiles per group
    size_t qr, kt, vtt, part_o, part_ml;  // workspace offsets (status word at 0)
    size_t total;
};
bool attn_supported(int C, int S, int Hq, int Hkv, int D, int N);
AttnPlan attn_plan(int C, int S, int Hq, int Hkv, int N);
int launch_tree_attention(int C, int S, int Hq, int Hkv, int N, double theta, const void* q, const void* k_tree,
                          const void* v_tree, const void* k_cache, const void* vt_cache, const int32_t* n_ctx,
                          const uint8_t* mask, const int32_t* pos, const int32_t* n_nodes, void* out, void* ws,
                          const AttnPlan& pl, cudaStream_t stream);

// Bounded-wait self-test (which = 0: mbarrier, 1: grid barrier on ctr).
int launch_selftest_wait(int which, unsigned* ctr, int* status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace dartree
