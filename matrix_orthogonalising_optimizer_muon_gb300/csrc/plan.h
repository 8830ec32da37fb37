// Host-side internals of the library shared by its C entry points (plan.cu,
// step.cu, capi.cu): the plan object, its buckets, launch lists and workspace
// layout, tensor-map encoding and the argument checks.  Not part of the C ABI.
#pragma once
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/muon.h"
#include "kernels.h"

namespace muon_impl {
using namespace muon;

// Quintic coefficients of the Newton-Schulz step ("Muon is Scalable" blog, eq. (2)).
constexpr float kNsA = 3.4445f;
constexpr float kNsB = -4.7750f;
constexpr float kNsC = 2.0315f;
// Limit on Newton-Schulz steps of the Gram-form recursion.  It carries G in 11
// significant bits (fp16); rounding can leave a null-space eigenvalue of G slightly
// negative, and each step multiplies such an eigenvalue by about p(0)^2 = a^2 ~ 11.9,
// so on rank-deficient or large square inputs it grows to O(1) and diverges after
// about six steps.  Five steps (the pages' choice) keep it below 1e-2.
constexpr int kMaxNsSteps = 5;            // one segment of the fp16 Gram recursion
constexpr int kMaxNsStepsRestart = 100;    // with restarts (opts.max_ns_steps)
constexpr int kMaxDim = 1 << 20;        // per-dimension limit of the library
constexpr int kMaxR = 32768;            // r x r workspace limit of the library

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 3-D tensor map over `batch` row-major matrices (rows x inner, leading dim ld,
// item stride rows * ld), 128-byte swizzle, zero fill outside the extents.
inline bool make_map(CUtensorMap* map, void* base, bool bf16, uint64_t inner, uint64_t rows, uint64_t batch, uint64_t ld,
              uint32_t box_inner, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const uint64_t esz = 2;   // bf16 or fp16
    cuuint64_t dims[3] = {inner, rows, batch};
    cuuint64_t strides[2] = {ld * esz, ld * rows * esz};
    cuuint32_t box[3] = {box_inner, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D view (64 columns, rows, cols / 64 column chunks, batch) of `batch` row-major
// matrices with cols % 64 == 0, so every box stays inside its rows: boxes (64, 128, 1, 1)
// are K-major operand blocks at (0, row, k / 64, item), boxes (64, 64, 2, 1) two 64-column
// chunks of 64 rows (an MN-major operand block, or a mirrored one) at (0, k, row / 64, item).
inline bool make_map4(CUtensorMap* map, void* base, bool bf16, uint64_t cols, uint64_t rows, uint64_t batch, uint64_t ld,
               uint32_t box_rows, uint32_t box_chunks) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || cols % 64 != 0) return false;
    cuuint64_t dims[4] = {64, rows, cols / 64, batch};
    cuuint64_t strides[3] = {ld * 2, 128, ld * rows * 2};
    cuuint32_t box[4] = {64, box_rows, box_chunks, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, base, dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// W of one matrix (fp32, stored m x n row-major, 16-byte aligned, n % 4 == 0) in 32 x 32
// boxes with 128-byte swizzle: exactly the staged layout of a W piece of the final product.
inline bool make_w_piece_map(CUtensorMap* map, void* W, uint64_t m, uint64_t n) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {n, m};
    cuuint64_t strides[1] = {n * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, W, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// Store map over `batch` r x r row-major matrices (leading dim ld): 32 x 32 boxes
// in the 64-byte-swizzled shared layout the pair kernel's epilogue stages.
inline bool make_out_map(CUtensorMap* map, void* base, bool bf16, uint64_t r, uint64_t batch, uint64_t ld) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const uint64_t esz = 2;
    cuuint64_t dims[3] = {r, r, batch};
    cuuint64_t strides[2] = {ld * esz, ld * r * esz};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// CTA pairs left to the batched products of a plan that also holds fused
// (r <= 128) matrices, or 0 to run the two one after the other.  Estimates at
// full GPU: the fused kernel moves its bytes at about 5.1 TB/s; the batched side
// is a chain of 16 dependent launches (about 20 us each when small) plus its
// FLOPs at about 1.2 PFLOP/s.  The batched side gets the share of CTA pairs its
// estimate holds of the total, within [1/8, 1/2] of them; when it is the larger
// part it runs after the fused kernel on every SM instead (a persistent launch
// keeps its CTA pairs to the end, after the fused kernel has finished).
inline int choose_chain_clusters(double fused_bytes, double chain_flops, int max_pairs) {
    const double t_fused = fused_bytes / 5.1e12;
    const double t_chain = 16 * 20e-6 + chain_flops / 1.2e15;
    if (t_chain >= t_fused) return 0;
    const int k = (int)std::lround(max_pairs * t_chain / (t_chain + t_fused));
    return std::min(std::max(k, std::max(1, max_pairs / 8)), max_pairs / 2);
}

inline long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }
inline long long round_up(long long a, long long b) { return ceil_div(a, b) * b; }

struct Bucket {
    int r = 0, c = 0, batch = 0;
    bool fused = false;     // r <= 128: whole step in the fused one-matrix-per-CTA kernel
    bool f32 = false;       // r <= 128, nearly square: whole step in fp32 on CUDA cores (ns_f32_kernel)
    int split = 0;          // batched precision: 0 plain, 1 r x r buffers and Q in two parts, 2 also X0
    bool batched() const { return !fused && !f32; }   // r x r buffers in the workspace, grouped products
    int chunk = 0;          // workspace chunk (see muon_plan_opts.workspace_bytes)
    long long ut1_off = -1; // second X buffer (restarted NS segments), element offset like ut_off
    CUtensorMap ut1_a, ut1_b, ut1_mn;
    int ldr = 0;   // leading dim of r x r buffers (multiple of 8)
    int ldu = 0;   // leading dim of X0 rows (multiple of 8)
    std::vector<int> mats;
    int slot_base = 0;
    long long ut_off = 0;   // element offset of item 0 in the X0 workspace
    float gscale = 1.f;     // G is carried as s G, s = 2^round(log2 r)
    __half* G[2] = {nullptr, nullptr};
    __half* P = nullptr;
    __half* T = nullptr;
    __half* Q[2] = {nullptr, nullptr};
    __nv_bfloat16* Qb = nullptr;
    int* d_item_mat = nullptr;
    float* Odbg = nullptr;
    CUtensorMap ut_a, ut_b, ut_mn, qb_a;
    CUtensorMap ga[2], gb[2], pa, pb, tb, qb[2];
    CUtensorMap qa[2], ta;   // 128-row boxes of Q and T (B halves of the CTA-pair kernel)
    CUtensorMap og[2], op, ot, oq[2], oqb;   // store maps of G, P, T, Q (fp16) and Qb (bf16)
    // 4-D maps of lower-triangle launches (r % 64 == 0 and c % 64 == 0): K-major (..k) and
    // mirror / MN-major (..t) boxes of X0, the second X buffer and the r x r buffers
    CUtensorMap utk, utt, ut1k, ut1t, gk[2], gt[2], pk, pt, tk, tt, qk[2], qt[2], qbk, qbt;
};

struct ListDev {
    int* list = nullptr;
    long long* blk = nullptr;
    int n = 0;
    long long blocks = 0;
};

}  // namespace muon_impl

using namespace muon_impl;

struct muon_plan_s {
    int device = 0;
    int sm_count = 0;
    int pair_clusters = 0;   // co-resident CTA pairs for the 2-SM kernel (0: 1-SM kernel only)
    int tuned = 0;           // candidates muon_plan_tune measured (0: not tuned)
    // fused (r <= 128) and batched matrices in one chunk: the batched products' stream
    // and fork/join events (created when a chunk overlaps the two)
    cudaStream_t s2 = nullptr;
    cudaEvent_t fork_ev = nullptr, join_ev = nullptr;
    float* ones = nullptr;   // per matrix 1.0 (alpha of the iterates after a restart)
    double* diff = nullptr;  // muon_debug_update_error's partial sums (2 + 2 kDiffParts doubles)
    muon_dtype gdt = MUON_F32;
    muon_plan_opts opts{};
    std::vector<muon_shape> shapes;
    std::vector<int64_t> full_rows;   // opts.full_rows copied (dim-0 shard plans), else empty
    std::vector<int32_t> prec_of;     // opts.precision_of copied (per-matrix precision), else empty
    long long colsq_len = 0;          // floats of the shard calls' colsq buffer
    std::vector<MatDev> mats;
    std::vector<int> mat_bucket, mat_item;
    std::vector<Bucket> buckets;

    void* ws = nullptr;
    size_t ws_bytes = 0;
    __nv_bfloat16* ut = nullptr;
    MatDev* d_mats = nullptr;
    float* partials = nullptr;
    float* cpartials = nullptr;
    float* rowinv = nullptr;
    float* alpha = nullptr;
    int* status = nullptr;
    unsigned char* d_transposed = nullptr;
    void** d_ptrs = nullptr;   // [G(n) | M(n) | W(n)]

    ListDev rn_rows[kRowClasses], rn_stats, rn_final, rn_apply;   // rows by length class
    // NS steps run chunk by chunk; the chunks' X0 and r x r buffers share (alias) one
    // workspace region.  One chunk unless opts.workspace_bytes caps the workspace.
    struct Chunk {
        std::vector<int> buckets;
        ListDev mom_rows, mom_tiles, all;
        ListDev rn_rows[kRowClasses], rn_stats, rn_final, rn_apply;   // RowNorm of this chunk (muon_step_host)
        int chain_clusters = 0;   // CTA pairs for the batched products beside the fused kernel
        int chain_est = 0;        // the work estimate's choice (chunks with fused and batched work)
        bool mixed = false;       // the chunk holds both fused and batched matrices
        bool lower_ok = false;    // every batched bucket on the pair kernel has r and c multiples of 64
        bool lower = false;       // its pair-kernel products store symmetric results as the lower triangle
    };
    std::vector<Chunk> chunks;

    void** h_pinned = nullptr;
    // per matrix: W piece map of the final product (re-encoded when the parameter pointers
    // change) and its validity; pinned host staging (n maps, then n bytes) and device copy
    CUtensorMap* h_wmap = nullptr;
    CUtensorMap* d_wmap = nullptr;
    unsigned char* d_wmap_ok = nullptr;
    std::vector<void*> h_cache;
    cudaEvent_t upload_ev = nullptr;
    bool uploaded = false;

    // opts.timing: one event group per step since the last muon_stage_times call
    // Per chunk c, events e[7c + k].  NS: e[0] momentum | e[1] fused r <= 128 | e[6],
    // batched SYRK from e[6] (or, split, from e[1] beside the fused kernel) | e[2] r x r |
    // e[3] final | e[4].  RowNorm: e[0] .. e[5] of chunk 0.
    struct StepEvents {
        std::vector<cudaEvent_t> e;
        std::vector<char> split;
        bool ns = false;
    };
    std::vector<StepEvents> evs;
    size_t n_timed = 0;
    double flops[3] = {0, 0, 0};   // summed over the timed steps
    int last_launches = 0;

    // muon_step_host: copy streams (in, out) and events, created on first use.
    // in_ev[c]: chunk c's gradients are on the device; out_ev[c]: chunk c's
    // parameters are final; entry_ev: the caller's stream before the step;
    // end_ev: the last copy back.
    struct HostCopy {
        cudaStream_t in = nullptr, out = nullptr;
        std::vector<cudaEvent_t> in_ev, out_ev;
        cudaEvent_t entry_ev = nullptr, end_ev = nullptr;
    } hc;
};

namespace muon_impl {

// The last CUDA error this thread turned into MUON_ERR_CUDA (muon_last_error_detail).
cudaError_t& last_cuda_error();

inline muon_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return MUON_OK;
    last_cuda_error() = e;
    return MUON_ERR_CUDA;
}

#define MUON_TRY(expr)                                    \
    do {                                                  \
        cudaError_t e__ = (expr);                         \
        if (e__ != cudaSuccess) {                         \
            last_cuda_error() = e__;                      \
            return MUON_ERR_CUDA;                         \
        }                                                 \
    } while (0)

inline bool finite_nonneg(float x) { return std::isfinite(x) && x >= 0.f; }

// Every params / momentum / grads range must be disjoint from every other.
muon_status check_pointers(const muon_plan_s* p, float* const* params, const void* const* grads,
                           float* const* momentum);

muon_status check_device(const muon_plan_s* p);

// Copies the per-call pointer tables to the device when they changed.
muon_status upload_pointers(muon_plan_s* p, float* const* params, const void* const* grads, float* const* momentum,
                            cudaStream_t s);

ElemArgs elem_args(const muon_plan_s* p, const ListDev& l, float mu, float lr, float wd, float eps);

int sym_tiles(int r);

GemmProblem problem(int M, int N, int K, int batch, bool sym, int epi);

// Event group for the next timed step (the last group is reused past the cap).
muon_plan_s::StepEvents* next_events(muon_plan_s* p);

void free_plan(muon_plan_s* p);

// Workspace offsets and per-chunk RowNorm lists of a plan, from plan_layout.
struct Layout {
    bool restarts = false;   // opts.max_ns_steps > 0: second X buffer, every matrix batched
    size_t o_mats = 0, o_part = 0, o_cpart = 0, o_inv = 0, o_alpha = 0, o_status = 0, o_tr = 0, o_ptrs = 0,
           o_items = 0, o_ones = 0, o_diff = 0, o_wmap = 0, o_wmap_ok = 0, o_odbg = 0, o_lists = 0, o_prefix = 0, o_region = 0;
    std::vector<size_t> o_ut, o_ut1, o_rr, o_qb;   // per bucket: X0, second X, r x r, bf16 Q (in the region)
    std::vector<int> rnr_list, rnc_list;           // RowNorm: row-wise and column-wise matrices
};

// Argument checks of muon_plan_create and muon_plan_workspace_size.
muon_status check_plan_args(const muon_shape* shapes, int32_t n, muon_dtype grad_dtype,
                            const muon_plan_opts* opts);

// The host part of planning, from p->shapes and p->opts alone (no CUDA call):
// orientation, buckets, chunks and the workspace layout; sets p->mats, p->buckets,
// p->chunks, p->mat_bucket, p->mat_item and p->ws_bytes.  MUON_ERR_OOM when
// opts.workspace_bytes cannot hold the largest single matrix.
muon_status plan_layout(muon_plan_s* p, Layout& L);

}  // namespace muon_impl
