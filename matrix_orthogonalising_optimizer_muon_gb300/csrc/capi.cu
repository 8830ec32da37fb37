// C ABI of the Muon step (include/muon.h): planner, argument validation and the
// stream-ordered launch sequence.  Host code only; kernels live in gemm.cu and
// elementwise.cu.
//
// Step (mode NS), per plan, every kernel grouped over all matrices:
//   momentum (m <= n)  |  momentum + transpose (m > n)  |  1/||U||_F
//   G0 = a^2 X X^T                                         (one launch, all buckets)
//   k = 1..J:  P = aI + bG + cG^2;  {Q' = P Q, T = P P};  G' = G T
//   O = a Q X fused with W -= lr (0.2 sqrt(c) O + wd W)    (one launch, all buckets)
// (Gram Newton-Schulz from DMuon's technical summary; coefficients, Nesterov
// input, normalisation and eq. (4) from the "Muon is Scalable" blog summary;
// orientation and RowNorm from the DiT paper sec. 3.1.)
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/muon.h"
#include "kernels.h"

using namespace muon;

namespace {

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

EncodeTiledFn encode_fn() {
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
bool make_map(CUtensorMap* map, void* base, bool bf16, uint64_t inner, uint64_t rows, uint64_t batch, uint64_t ld,
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
bool make_map4(CUtensorMap* map, void* base, bool bf16, uint64_t cols, uint64_t rows, uint64_t batch, uint64_t ld,
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
bool make_w_piece_map(CUtensorMap* map, void* W, uint64_t m, uint64_t n) {
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
bool make_out_map(CUtensorMap* map, void* base, bool bf16, uint64_t r, uint64_t batch, uint64_t ld) {
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
int choose_chain_clusters(double fused_bytes, double chain_flops, int max_pairs) {
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

}  // namespace

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

namespace {
thread_local cudaError_t g_last_cuda_error = cudaSuccess;
}  // namespace

void muon::record_cuda_error(cudaError_t e) { g_last_cuda_error = e; }

namespace {

muon_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return MUON_OK;
    g_last_cuda_error = e;
    return MUON_ERR_CUDA;
}

#define MUON_TRY(expr)                                    \
    do {                                                  \
        cudaError_t e__ = (expr);                         \
        if (e__ != cudaSuccess) {                         \
            g_last_cuda_error = e__;                      \
            return MUON_ERR_CUDA;                         \
        }                                                 \
    } while (0)

bool finite_nonneg(float x) { return std::isfinite(x) && x >= 0.f; }

// Every params / momentum / grads range must be disjoint from every other.
muon_status check_pointers(const muon_plan_s* p, float* const* params, const void* const* grads,
                           float* const* momentum) {
    if (!params || !grads || !momentum) return MUON_ERR_INVALID_ARG;
    const size_t n = p->shapes.size();
    const size_t gsz = p->gdt == MUON_BF16 ? 2 : 4;
    std::vector<std::pair<uintptr_t, uintptr_t>> ranges;
    ranges.reserve(3 * n);
    for (size_t i = 0; i < n; ++i) {
        if (!params[i] || !grads[i] || !momentum[i]) return MUON_ERR_INVALID_ARG;
        const size_t numel = (size_t)p->shapes[i].rows * (size_t)p->shapes[i].cols;
        const uintptr_t w = reinterpret_cast<uintptr_t>(params[i]);
        const uintptr_t g = reinterpret_cast<uintptr_t>(grads[i]);
        const uintptr_t m = reinterpret_cast<uintptr_t>(momentum[i]);
        ranges.push_back({w, w + numel * 4});
        ranges.push_back({m, m + numel * 4});
        ranges.push_back({g, g + numel * gsz});
    }
    std::sort(ranges.begin(), ranges.end());
    for (size_t k = 1; k < ranges.size(); ++k)
        if (ranges[k].first < ranges[k - 1].second) return MUON_ERR_INVALID_ARG;
    return MUON_OK;
}

muon_status check_device(const muon_plan_s* p) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_CUDA;
    return dev == p->device ? MUON_OK : MUON_ERR_INVALID_ARG;
}

// Copies the per-call pointer tables to the device when they changed.
muon_status upload_pointers(muon_plan_s* p, float* const* params, const void* const* grads, float* const* momentum,
                            cudaStream_t s) {
    const size_t n = p->shapes.size();
    bool same = p->uploaded;
    for (size_t i = 0; same && i < n; ++i)
        same = p->h_cache[i] == grads[i] && p->h_cache[n + i] == momentum[i] && p->h_cache[2 * n + i] == params[i];
    if (same) return MUON_OK;
    if (p->uploaded) MUON_TRY(cudaEventSynchronize(p->upload_ev));   // pinned buffer free again
    for (size_t i = 0; i < n; ++i) {
        p->h_cache[i] = const_cast<void*>(grads[i]);
        p->h_cache[n + i] = momentum[i];
        p->h_cache[2 * n + i] = params[i];
    }
    std::memcpy(p->h_pinned, p->h_cache.data(), 3 * n * sizeof(void*));
    MUON_TRY(cudaMemcpyAsync(p->d_ptrs, p->h_pinned, 3 * n * sizeof(void*), cudaMemcpyHostToDevice, s));
    if (p->h_wmap) {   // W piece maps follow the parameter pointers (tensor-core final products)
        unsigned char* ok = reinterpret_cast<unsigned char*>(p->h_wmap + n);
        for (size_t i = 0; i < n; ++i) {
            const MatDev& md = p->mats[i];
            const Bucket& bk = p->buckets[p->mat_bucket[i]];
            const bool usable = (bk.batched() || bk.fused) && md.n % 4 == 0 &&
                                (reinterpret_cast<uintptr_t>(params[i]) & 15) == 0;
            ok[i] = usable && make_w_piece_map(&p->h_wmap[i], params[i], (uint64_t)md.m, (uint64_t)md.n) ? 1 : 0;
        }
        MUON_TRY(cudaMemcpyAsync(p->d_wmap, p->h_wmap, n * sizeof(CUtensorMap), cudaMemcpyHostToDevice, s));
        MUON_TRY(cudaMemcpyAsync(p->d_wmap_ok, ok, n, cudaMemcpyHostToDevice, s));
    }
    MUON_TRY(cudaEventRecord(p->upload_ev, s));
    p->uploaded = true;
    return MUON_OK;
}

ElemArgs elem_args(const muon_plan_s* p, const ListDev& l, float mu, float lr, float wd, float eps) {
    ElemArgs a{};
    const size_t n = p->shapes.size();
    a.mats = p->d_mats;
    a.list = l.list;
    a.nlist = l.n;
    a.list_blk = l.blk;
    a.G = const_cast<const void* const*>(p->d_ptrs);
    a.M = reinterpret_cast<float* const*>(p->d_ptrs + n);
    a.W = reinterpret_cast<float* const*>(p->d_ptrs + 2 * n);
    a.ut = p->ut;
    a.partials = p->partials;
    a.alpha = p->alpha;
    a.rowinv = p->rowinv;
    a.mu = mu;
    a.lr = lr;
    a.wd = wd;
    a.eps = eps;
    a.grad_bf16 = p->gdt == MUON_BF16;
    a.check_finite = p->opts.check_finite ? 1 : 0;
    a.status = p->status;
    return a;
}

int sym_tiles(int r) {
    const int tm = (int)ceil_div(r, kBM);
    int t = 0;
    for (int i = 0; i < tm; ++i) t += i / 2 + 1;
    return t;
}

GemmProblem problem(int M, int N, int K, int batch, bool sym, int epi) {
    GemmProblem q{};
    q.M = M;
    q.N = N;
    q.K = K;
    q.batch = batch;
    q.tiles_m = (int)ceil_div(M, kBM);
    q.tiles_n = (int)ceil_div(N, kBN);
    q.tiles_per_item = sym ? sym_tiles(M) : q.tiles_m * q.tiles_n;
    q.sym = sym ? 1 : 0;
    q.epi = epi;
    return q;
}

// 4-D maps of one operand for lower-triangle launches.
struct Maps4 {
    const CUtensorMap* k = nullptr;   // K-major boxes (64, 128, 1, 1)
    const CUtensorMap* t = nullptr;   // mirror / MN-major boxes (64, 64, 2, 1)
    bool sym = false;                 // a symmetric buffer stored as its lower triangle
};

// Collects problems into grouped launches of up to kMaxProblems.
struct Grouper {
    muon_plan_s* p;
    cudaStream_t s;
    bool bf16;
    bool lower;         // lower-triangle launches (the chunk's Chunk::lower)
    bool wtma = false;  // final products whose every matrix has a W map: W pieces by TMA
    int clusters = 0;   // CTA pairs for the pair kernel, CTAs for the one-SM kernel
    int grid1 = 0;
    GemmLaunch L1;   // 1-SM kernel, 128 x 256 tiles
    GemmLaunch L2;   // CTA-pair kernel, 256 x 256 tiles
    muon_status st = MUON_OK;
    int launches = 0;
    Grouper(muon_plan_s* plan, cudaStream_t stream, bool is_bf16, bool lower_tri, int pair_clusters, int sm_grid)
        : p(plan), s(stream), bf16(is_bf16), lower(lower_tri), clusters(pair_clusters), grid1(sm_grid) {
        reset(L1);
        reset(L2);
    }
    void reset(GemmLaunch& L) {
        std::memset(&L, 0, sizeof(L));
        L.status = p->status;
    }
    static void push(GemmLaunch& L, const CUtensorMap& a, const CUtensorMap& b, GemmProblem q) {
        q.tile_begin = L.total_tiles;
        L.mapA[L.nprob] = a;
        L.mapB[L.nprob] = b;
        L.prob[L.nprob] = q;
        L.nprob++;
        L.total_tiles += q.tiles_per_item * q.batch;
    }
    // a128: A with 128-row boxes; b256 / b128: B with 256- / 128-row boxes (the
    // same map for an MN-major B).  Problems with more than 128 rows go to the
    // CTA-pair kernel (each CTA loads 128 rows of A and 128 of B).
    // oc / oc2: store maps of a symmetric problem's outputs (tma_out set by the
    // caller); the pair kernel then writes them with TMA stores.
    // a4 / b4: the operands' 4-D maps, used by lower-triangle launches (B of an
    // MN-major problem through b4.t).
    // og: for a polynomial product, the store map of its G' input (32 x 32 boxes), through
    // which the pair kernel's epilogue loads G' by TMA.
    void add(const CUtensorMap& a128, const CUtensorMap& b256, const CUtensorMap& b128, GemmProblem q,
             const CUtensorMap* oc, const CUtensorMap* oc2, Maps4 a4, Maps4 b4, const CUtensorMap* og = nullptr) {
        if (q.a_split || q.b_split || q.out_split) q.tma_out = 0;   // split parts: per-thread stores
        q.gin_tma = 0;
        if (q.M > kBM && p->pair_clusters > 0) {
            if (L2.nprob == kMaxProblems) flush2();
            q.tiles_m = (int)ceil_div(q.M, 256);
            q.tiles_n = (int)ceil_div(q.N, 256);
            q.tiles_per_item = q.sym ? q.tiles_m * (q.tiles_m + 1) / 2 : q.tiles_m * q.tiles_n;
            if (!q.sym || !oc || ((q.tma_out & kTmaOutC2) && !oc2)) q.tma_out = 0;
            if (q.tma_out) {
                L2.mapC[L2.nprob] = *oc;
                if (oc2) L2.mapC2[L2.nprob] = *oc2;
                if (og && q.epi == kEpiPoly) {
                    L2.mapG[L2.nprob] = *og;
                    q.gin_tma = 1;
                }
            }
            if (lower) {
                q.lower_out = q.sym;
                q.sym_a = a4.sym;
                q.sym_b = b4.sym && !q.b_mn;
                L2.mapAt[L2.nprob] = a4.t ? *a4.t : *a4.k;
                L2.mapBt[L2.nprob] = b4.t ? *b4.t : *b4.k;
                push(L2, *a4.k, b4.k ? *b4.k : *b4.t, q);
            } else {
                push(L2, a128, b128, q);
            }
        } else {
            if (L1.nprob == kMaxProblems) flush1();
            q.tma_out = 0;
            push(L1, a128, b256, q);
        }
    }
    void flush1() {
        if (L1.nprob == 0) return;
        if (st == MUON_OK) {
            st = cuda_status(gemm_launch(L1, bf16, grid1, s));
            ++launches;
        }
        reset(L1);
    }
    void flush2() {
        if (L2.nprob == 0) return;
        if (st == MUON_OK) {
            st = cuda_status(gemm2_launch(L2, bf16, clusters, s, lower, wtma));
            ++launches;
        }
        reset(L2);
    }
    void flush() {
        flush2();
        flush1();
    }
};

constexpr size_t kMaxTimedSteps = 4096;

// Event group for the next timed step (the last group is reused past the cap).
muon_plan_s::StepEvents* next_events(muon_plan_s* p) {
    if (p->n_timed < p->evs.size()) return &p->evs[p->n_timed++];
    if (p->evs.size() >= kMaxTimedSteps) return &p->evs.back();
    muon_plan_s::StepEvents g{};
    try {
        g.e.assign(7 * p->chunks.size(), nullptr);
        g.split.assign(p->chunks.size(), 0);
        p->evs.reserve(p->evs.size() + 1);   // the push_back below cannot throw
    } catch (...) {
        return nullptr;   // host memory
    }
    for (auto& e : g.e)
        if (cudaEventCreate(&e) != cudaSuccess) {
            for (auto& x : g.e)
                if (x) cudaEventDestroy(x);
            return nullptr;
        }
    p->evs.push_back(std::move(g));
    p->n_timed = p->evs.size();
    return &p->evs.back();
}

void free_plan(muon_plan_s* p) {
    if (!p) return;
    if (p->ws) cudaFree(p->ws);
    if (p->h_pinned) cudaFreeHost(p->h_pinned);
    if (p->h_wmap) cudaFreeHost(p->h_wmap);
    if (p->upload_ev) cudaEventDestroy(p->upload_ev);
    if (p->fork_ev) cudaEventDestroy(p->fork_ev);
    if (p->join_ev) cudaEventDestroy(p->join_ev);
    if (p->s2) cudaStreamDestroy(p->s2);
    if (p->hc.in) cudaStreamDestroy(p->hc.in);
    if (p->hc.out) cudaStreamDestroy(p->hc.out);
    for (cudaEvent_t e : p->hc.in_ev)
        if (e) cudaEventDestroy(e);
    for (cudaEvent_t e : p->hc.out_ev)
        if (e) cudaEventDestroy(e);
    if (p->hc.entry_ev) cudaEventDestroy(p->hc.entry_ev);
    if (p->hc.end_ev) cudaEventDestroy(p->hc.end_ev);
    for (auto& g : p->evs)
        for (auto& e : g.e)
            if (e) cudaEventDestroy(e);
    delete p;
}

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
                            const muon_plan_opts* opts) {
    if (!shapes || n <= 0) return MUON_ERR_INVALID_ARG;
    if (grad_dtype != MUON_F32 && grad_dtype != MUON_BF16) return MUON_ERR_UNSUPPORTED;
    for (int i = 0; i < n; ++i) {
        if (shapes[i].rows <= 0 || shapes[i].cols <= 0) return MUON_ERR_INVALID_ARG;
        if (shapes[i].rows > kMaxDim || shapes[i].cols > kMaxDim) return MUON_ERR_UNSUPPORTED;
        if (std::min(shapes[i].rows, shapes[i].cols) > kMaxR) return MUON_ERR_UNSUPPORTED;
    }
    if (opts && (opts->max_ns_steps < 0 || opts->max_ns_steps > kMaxNsStepsRestart || opts->chunks < 0 ||
                 opts->workspace_bytes < 0))
        return MUON_ERR_INVALID_ARG;
    if (opts && opts->full_rows)
        for (int i = 0; i < n; ++i)
            if (opts->full_rows[i] < shapes[i].rows || opts->full_rows[i] > kMaxDim) return MUON_ERR_INVALID_ARG;
    return MUON_OK;
}

// The host part of planning, from p->shapes and p->opts alone (no CUDA call):
// orientation, buckets, chunks and the workspace layout; sets p->mats, p->buckets,
// p->chunks, p->mat_bucket, p->mat_item and p->ws_bytes.  MUON_ERR_OOM when
// opts.workspace_bytes cannot hold the largest single matrix.
muon_status plan_layout(muon_plan_s* p, Layout& L) {
    const int n = (int)p->shapes.size();
    // ---- orient; group by oriented shape (r, c) in order of first appearance
    // (DiT paper sec. 3.1; DMuon batching)
    p->mats.resize(n);
    p->mat_bucket.resize(n);
    p->mat_item.resize(n);
    std::vector<std::pair<int, int>> group_rc;
    std::vector<int> group_lv;   // per group: the matrices' opts.precision_of entry (0: the plan's rule)
    std::vector<std::vector<int>> group_mats;
    for (int i = 0; i < n; ++i) {
        MatDev& md = p->mats[i];
        std::memset(&md, 0, sizeof(md));
        md.m = p->shapes[i].rows;
        md.n = p->shapes[i].cols;
        md.r = (int)std::min(md.m, md.n);
        md.c = (int)std::max(md.m, md.n);
        md.transposed = md.m > md.n;
        md.scale = 0.2f * std::sqrt((float)md.c);   // blog eq. (4)
        if (!p->full_rows.empty()) {   // a dim-0 shard: RowNorm axis and scale of the full matrix
            const long long fm = p->full_rows[i];
            md.transposed = fm > md.n;
            md.scale = 0.2f * std::sqrt((float)std::max(fm, md.n));
        }
        size_t g = 0;
        const int lv = p->prec_of.empty() ? 0 : p->prec_of[i];
        while (g < group_rc.size() &&
               !(group_rc[g].first == md.r && group_rc[g].second == md.c && group_lv[g] == lv))
            ++g;
        if (g == group_rc.size()) {
            group_rc.push_back({md.r, md.c});
            group_lv.push_back(lv);
            group_mats.emplace_back();
        }
        group_mats[g].push_back(i);
    }

    // ---- workspace: a fixed part (per-matrix tables, partial sums, pointer tables,
    // launch lists, debug copies of O) and a region for the X0 and r x r buffers of
    // one chunk of matrices, shared by all chunks (they run one after the other)
    const bool restarts = L.restarts = p->opts.max_ns_steps > 0;   // second X buffer, batched path for all
    // fp32 path (opts.small_fp32): 0 nearly square (c < 1.25 r) matrices with r <= 128,
    // > 0 every matrix with r <= 128, < 0 none; never in plans with restarts
    auto is_f32 = [&](int r, int c) {
        if (restarts || p->opts.small_fp32 < 0 || r > kF32MaxR) return false;
        return p->opts.small_fp32 > 0 || 4LL * c < 5LL * r;
    };
    const bool fused_ok = !p->opts.generic_small && !restarts;
    auto is_fused = [&](int r, int c) { return fused_ok && r <= kSmallMaxR && !is_f32(r, c); };
    // split precision of a batched bucket (opts.precision, opts.split_max_r)
    // lv: the matrices' opts.precision_of entry (< 0 plain, 1 or 2 that level, 0 the plan's rule)
    auto split_of = [&](int r, int c, int lv) -> int {
        if (is_fused(r, c) || is_f32(r, c)) return 0;
        if (lv != 0) return lv < 0 ? 0 : (lv >= 2 ? 2 : 1);
        if (p->opts.precision < 0) return 0;
        if (p->opts.precision > 0) return p->opts.precision >= 2 ? 2 : 1;
        const int rmax = p->opts.split_max_r > 0 ? p->opts.split_max_r : 1024;
        return (4LL * c < 5LL * r && r <= rmax) ? 1 : 0;
    };
    // region bytes of a bucket of `batch` matrices, exactly as laid out below: its X0
    // (and second X) buffer and, batched, its seven r x r buffers, each rounded to 256
    // (split buffers hold two parts per matrix)
    const bool sharded = !p->full_rows.empty();   // RowNorm only: no NS buffers
    auto bucket_bytes = [&](int r, int c, int lv, long long batch) -> long long {
        if (sharded) return 0;
        const int sp = split_of(r, c, lv);
        const long long x = round_up(batch * r * round_up(c, 8) * 2 * (sp == 2 ? 2 : 1), 256);
        const long long rr = round_up(batch * r * round_up(r, 8) * 2 * (sp ? 2 : 1), 256);
        return (restarts ? 2 : 1) * x + (is_fused(r, c) || is_f32(r, c) ? 0 : 7 * rr);
    };
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = (size_t)round_up((long long)(off + bytes), 256);
        return o;
    };
    // momentum / RowNorm bookkeeping per matrix (not chunked)
    long long mom_part = 0, col_part = 0, inv_elems = 0;
    for (int i = 0; i < n; ++i) {
        MatDev& md = p->mats[i];
        md.nblk = (int)(md.transposed ? ceil_div(md.m, kTileRows) * ceil_div(md.n, kTile)
                                      : ceil_div(md.m * md.n, kMomElemsPerBlock));
        md.part_off = mom_part;
        mom_part += md.nblk;
        if (md.transposed) {
            md.cpart_off = col_part;
            col_part += ceil_div(md.m, kColSlab) * md.n;
            md.inv_off = inv_elems;
            inv_elems += round_up(md.n, 4);
            L.rnc_list.push_back(i);
        } else {
            L.rnr_list.push_back(i);
        }
    }
    p->colsq_len = sharded ? inv_elems : 0;
    L.o_mats = take(sizeof(MatDev) * n);
    L.o_part = take(sizeof(float) * std::max<long long>(mom_part, 1));
    L.o_cpart = take(sizeof(float) * std::max<long long>(col_part, 1));
    L.o_inv = take(sizeof(float) * std::max<long long>(inv_elems, 1));
    L.o_alpha = take(sizeof(float) * n);
    L.o_status = take(sizeof(int));
    L.o_tr = take((size_t)n);
    L.o_ptrs = take(sizeof(void*) * 3 * n);
    L.o_items = take(sizeof(int) * n);   // item -> plan matrix, per bucket slice
    L.o_ones = take(sizeof(float) * n);
    L.o_diff = take(sizeof(double) * (2 + 2 * kDiffParts));
    L.o_wmap = take(sizeof(CUtensorMap) * n);   // W piece maps (slices are 256-byte aligned)
    L.o_wmap_ok = take((size_t)n);
    L.o_odbg = p->opts.keep_update ? take([&] {
        size_t t = 0;
        for (int i = 0; i < n; ++i) t += (size_t)round_up(p->mats[i].m * p->mats[i].n * 4, 256);
        return t;
    }()) : 0;
    // launch lists: per chunk the momentum rows / tiles / all lists and its six
    // RowNorm lists (rows in three length classes, column statistics, finalize,
    // apply), and the six RowNorm lists of the whole plan.  Chunks partition the
    // matrices (n chunks at most); a list of k matrices takes max(k, 1) ints and k + 1
    // prefixes.  Momentum lists: 2 per matrix plus 3 per chunk, at most 5n; chunk
    // RowNorm lists (rows once, column matrices three times): at most 3n + 6n; the
    // plan's: 3n + 6.  17n + 6 <= 17n + 16 of each.
    L.o_lists = take(sizeof(int) * (size_t)(17 * n + 16));
    L.o_prefix = take(sizeof(long long) * (size_t)(17 * n + 16));
    const size_t fixed_bytes = off;

    // ---- chunks: matrices in group order, a new chunk whenever the region would
    // exceed what the cap leaves after the fixed part (one chunk without a cap)
    const long long cap = p->opts.workspace_bytes;
    double region_cap = 1e300;
    if (cap > 0) {
        region_cap = (double)cap - (double)fixed_bytes;
        double need = 0;
        for (int i = 0; i < n; ++i)
            need = std::max(need, (double)bucket_bytes(p->mats[i].r, p->mats[i].c,
                                                       p->prec_of.empty() ? 0 : p->prec_of[i], 1));
        if (region_cap < need) return MUON_ERR_OOM;   // the cap cannot hold even the largest single matrix
    }
    if (p->opts.chunks > 1) {   // about opts.chunks chunks, each at least one matrix
        double total = 0, largest = 0;
        for (int i = 0; i < n; ++i) {
            const double b =
                (double)bucket_bytes(p->mats[i].r, p->mats[i].c, p->prec_of.empty() ? 0 : p->prec_of[i], 1);
            total += b;
            largest = std::max(largest, b);
        }
        const double per = total / p->opts.chunks;
        region_cap = std::min(region_cap, std::max(per, largest));
    }
    {
        long long used = 0;   // region bytes of the current chunk, exactly
        p->chunks.emplace_back();
        for (size_t g = 0; g < group_rc.size(); ++g) {
            const int r = group_rc[g].first, c = group_rc[g].second, lv = group_lv[g];
            int cur = -1;   // bucket of this group in the current chunk
            for (int i : group_mats[g]) {
                const long long k = cur < 0 ? 0 : (long long)p->buckets[cur].mats.size();
                long long grow = bucket_bytes(r, c, lv, k + 1) - (k > 0 ? bucket_bytes(r, c, lv, k) : 0);
                if ((double)(used + grow) > region_cap && used > 0) {
                    p->chunks.emplace_back();
                    used = 0;
                    cur = -1;
                    grow = bucket_bytes(r, c, lv, 1);
                }
                if (cur < 0) {
                    Bucket nb{};   // value-initialised: the tensor maps are filled in later
                    nb.r = r;
                    nb.c = c;
                    nb.ldr = (int)round_up(r, 8);
                    nb.ldu = (int)round_up(c, 8);
                    nb.fused = is_fused(r, c);
                    nb.f32 = is_f32(r, c);
                    nb.split = split_of(r, c, lv);
                    nb.chunk = (int)p->chunks.size() - 1;
                    p->buckets.push_back(nb);
                    cur = (int)p->buckets.size() - 1;
                    p->chunks.back().buckets.push_back(cur);
                }
                used += grow;
                p->mat_bucket[i] = cur;
                p->mat_item[i] = (int)p->buckets[cur].mats.size();
                p->buckets[cur].mats.push_back(i);
            }
        }
    }
    // region offsets: each chunk's buckets laid out from the start of the region
    size_t region_bytes = 0;
    std::vector<size_t>& o_ut = L.o_ut;
    std::vector<size_t>& o_ut1 = L.o_ut1;
    std::vector<size_t>& o_rr = L.o_rr;
    std::vector<size_t>& o_qb = L.o_qb;
    o_ut.assign(p->buckets.size(), 0);
    o_ut1.assign(p->buckets.size(), 0);
    o_rr.assign(p->buckets.size(), 0);
    o_qb.assign(p->buckets.size(), 0);
    {
        int slots = 0;
        for (auto& ch : p->chunks) {
            size_t roff = 0;
            auto rtake = [&](size_t bytes) {
                const size_t o = roff;
                roff = (size_t)round_up((long long)(roff + bytes), 256);
                return o;
            };
            for (int k : ch.buckets) {
                Bucket& b = p->buckets[k];
                b.batch = (int)b.mats.size();
                b.slot_base = slots;
                slots += b.batch;
                const size_t xparts = b.split == 2 ? 2 : 1, rparts = b.split ? 2 : 1;
                if (sharded) continue;   // RowNorm only: no X0 or r x r buffers
                o_ut[k] = rtake((size_t)b.batch * b.r * b.ldu * 2 * xparts);
                if (restarts) o_ut1[k] = rtake((size_t)b.batch * b.r * b.ldu * 2 * xparts);
                if (b.batched()) {
                    const size_t rr = (size_t)b.batch * b.r * b.ldr * 2 * rparts;
                    o_rr[k] = rtake(rr);   // G0 (fp16, scaled)
                    for (int q = 0; q < 5; ++q) rtake(rr);   // G1, P, T, Q0, Q1
                    o_qb[k] = rtake(rr);   // bf16 Q for the final product
                }
            }
            region_bytes = std::max(region_bytes, roff);
        }
    }
    L.o_region = take(std::max<size_t>(region_bytes, 256));
    for (int i = 0; i < n; ++i) {
        MatDev& md = p->mats[i];
        const Bucket& b = p->buckets[p->mat_bucket[i]];
        md.slot = b.slot_base + p->mat_item[i];
        md.ldu = b.ldu;
        md.x_split = b.split == 2 ? 1 : 0;   // hi part of item i at 2i, lo at 2i + 1
        md.ut_off = (long long)(o_ut[p->mat_bucket[i]] / 2) +
                    (long long)p->mat_item[i] * b.r * b.ldu * (md.x_split ? 2 : 1);
    }
    p->ws_bytes = off;
    // the packing counts the region exactly, so a cap is never exceeded; kept as a guard
    if (cap > 0 && (long long)off > cap) return MUON_ERR_OOM;
    return MUON_OK;
}

}  // namespace

extern "C" {

const char* muon_last_error_detail(void) {
    return g_last_cuda_error == cudaSuccess ? "no CUDA error recorded" : cudaGetErrorString(g_last_cuda_error);
}

const char* muon_status_string(muon_status s) {
    switch (s) {
        case MUON_OK: return "MUON_OK";
        case MUON_ERR_INVALID_ARG: return "MUON_ERR_INVALID_ARG: invalid argument";
        case MUON_ERR_UNSUPPORTED: return "MUON_ERR_UNSUPPORTED: unsupported dtype or size";
        case MUON_ERR_OOM: return "MUON_ERR_OOM: workspace allocation failed";
        case MUON_ERR_CUDA: return "MUON_ERR_CUDA: CUDA runtime or launch error";
        case MUON_ERR_TIMEOUT: return "MUON_ERR_TIMEOUT: a bounded device wait expired";
        case MUON_ERR_NONFINITE: return "MUON_ERR_NONFINITE: a non-finite input norm (opts.check_finite)";
    }
    return "MUON_ERR_UNKNOWN";
}

// Everything of muon_plan_create after the argument checks.  On failure it frees p;
// a host allocation that throws leaves p to the caller.
static muon_status plan_build(muon_plan_s* p, const muon_shape* shapes, int32_t n, muon_dtype grad_dtype,
                              const muon_plan_opts* opts, muon_plan* out) {
    if (cudaGetDevice(&p->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess ||
        !encode_fn()) {
        free_plan(p);
        return MUON_ERR_CUDA;
    }
    p->gdt = grad_dtype;
    if (opts) p->opts = *opts;
    p->shapes.assign(shapes, shapes + n);
    if (p->opts.full_rows) p->full_rows.assign(p->opts.full_rows, p->opts.full_rows + n);
    if (p->opts.precision_of) p->prec_of.assign(p->opts.precision_of, p->opts.precision_of + n);
    p->opts.full_rows = nullptr;   // read during creation only
    p->opts.precision_of = nullptr;

    Layout L;
    {
        const muon_status st = plan_layout(p, L);
        if (st != MUON_OK) {
            free_plan(p);
            return st;
        }
    }
    const bool restarts = L.restarts;
    if (cudaMalloc(&p->ws, p->ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        free_plan(p);
        return MUON_ERR_OOM;
    }
    char* base = static_cast<char*>(p->ws);
    p->ut = reinterpret_cast<__nv_bfloat16*>(base + L.o_region);
    p->d_mats = reinterpret_cast<MatDev*>(base + L.o_mats);
    p->partials = reinterpret_cast<float*>(base + L.o_part);
    p->cpartials = reinterpret_cast<float*>(base + L.o_cpart);
    p->rowinv = reinterpret_cast<float*>(base + L.o_inv);
    p->alpha = reinterpret_cast<float*>(base + L.o_alpha);
    p->status = reinterpret_cast<int*>(base + L.o_status);
    p->d_transposed = reinterpret_cast<unsigned char*>(base + L.o_tr);
    p->d_ptrs = reinterpret_cast<void**>(base + L.o_ptrs);
    p->ones = reinterpret_cast<float*>(base + L.o_ones);
    p->diff = reinterpret_cast<double*>(base + L.o_diff);
    p->d_wmap = reinterpret_cast<CUtensorMap*>(base + L.o_wmap);
    p->d_wmap_ok = reinterpret_cast<unsigned char*>(base + L.o_wmap_ok);

    std::vector<unsigned char> tr(n);
    for (int i = 0; i < n; ++i) tr[i] = (unsigned char)p->mats[i].transposed;
    bool ok = cudaMemcpy(p->d_mats, p->mats.data(), sizeof(MatDev) * n, cudaMemcpyHostToDevice) == cudaSuccess;
    ok = ok && cudaMemcpy(p->d_transposed, tr.data(), n, cudaMemcpyHostToDevice) == cudaSuccess;
    ok = ok && cudaMemset(p->status, 0, sizeof(int)) == cudaSuccess;
    ok = ok && cudaMemset(p->rowinv, 0, L.o_alpha - L.o_inv) == cudaSuccess;
    ok = ok && cudaMemset(p->d_ptrs, 0, sizeof(void*) * 3 * n) == cudaSuccess;
    {
        const std::vector<float> one(n, 1.f);
        ok = ok && cudaMemcpy(p->ones, one.data(), sizeof(float) * n, cudaMemcpyHostToDevice) == cudaSuccess;
    }

    // launch lists (int lists then long long prefixes, carved from their slices)
    int* list_cursor = reinterpret_cast<int*>(base + L.o_lists);
    long long* prefix_cursor = reinterpret_cast<long long*>(base + L.o_prefix);
    auto upload_list = [&](const std::vector<int>& v, ListDev& d, int kind) {
        d.list = list_cursor;
        d.blk = prefix_cursor;
        d.n = (int)v.size();
        list_cursor += std::max<size_t>(v.size(), 1);
        prefix_cursor += v.size() + 1;
        std::vector<long long> pre(v.size() + 1, 0);
        for (size_t j = 0; j < v.size(); ++j) {
            const MatDev& md = p->mats[v[j]];
            long long nb = 0;
            switch (kind) {
                case 0: case 1: nb = md.nblk; break;
                case 2: nb = 1; break;
                case 3: nb = md.m; break;
                case 4: nb = ceil_div(md.m, kColSlab) * ceil_div(md.n, kColWidth); break;
                case 5: nb = ceil_div(md.n, kElemThreads); break;
                case 6: nb = ceil_div(md.m * md.n, kApplyElemsPerBlock); break;
            }
            pre[j + 1] = pre[j] + nb;
        }
        d.blocks = pre.back();
        if (ok && !v.empty()) ok = cudaMemcpy(d.list, v.data(), sizeof(int) * v.size(), cudaMemcpyHostToDevice) == cudaSuccess;
        if (ok) ok = cudaMemcpy(d.blk, pre.data(), sizeof(long long) * pre.size(), cudaMemcpyHostToDevice) == cudaSuccess;
    };
    for (auto& ch : p->chunks) {
        std::vector<int> rows, tiles, all;
        for (int k : ch.buckets)
            for (int i : p->buckets[k].mats) {
                (p->mats[i].transposed ? tiles : rows).push_back(i);
                all.push_back(i);
            }
        upload_list(rows, ch.mom_rows, 0);
        upload_list(tiles, ch.mom_tiles, 1);
        upload_list(all, ch.all, 2);
        for (int cl = 0; cl < kRowClasses; ++cl) {
            std::vector<int> rc;
            for (int i : rows)
                if (rownorm_row_class(p->mats[i].n) == cl) rc.push_back(i);
            upload_list(rc, ch.rn_rows[cl], 3);
        }
        upload_list(tiles, ch.rn_stats, 4);
        upload_list(tiles, ch.rn_final, 5);
        upload_list(tiles, ch.rn_apply, 6);
    }
    for (int cl = 0; cl < kRowClasses; ++cl) {
        std::vector<int> rc;
        for (int i : L.rnr_list)
            if (rownorm_row_class(p->mats[i].n) == cl) rc.push_back(i);
        upload_list(rc, p->rn_rows[cl], 3);
    }
    upload_list(L.rnc_list, p->rn_stats, 4);
    upload_list(L.rnc_list, p->rn_final, 5);
    upload_list(L.rnc_list, p->rn_apply, 6);

    int* item_cursor = reinterpret_cast<int*>(base + L.o_items);
    size_t odbg_off = L.o_odbg;
    for (size_t k = 0; ok && k < p->buckets.size(); ++k) {
        Bucket& b = p->buckets[k];
        b.d_item_mat = item_cursor;
        item_cursor += b.batch;
        ok = cudaMemcpy(b.d_item_mat, b.mats.data(), sizeof(int) * b.batch, cudaMemcpyHostToDevice) == cudaSuccess;
        if (!p->full_rows.empty()) continue;   // dim-0 shard plans run RowNorm only: no NS buffers
        b.gscale = std::ldexp(1.f, (int)std::lround(std::log2((double)b.r)));
        b.ut_off = (long long)(L.o_ut[k] / 2);
        if (p->opts.keep_update) {
            b.Odbg = reinterpret_cast<float*>(base + odbg_off);
            odbg_off += (size_t)round_up((long long)b.batch * b.r * b.c * 4, 256);
        }
        __nv_bfloat16* ut = p->ut + b.ut_off;
        const int xb = b.batch * (b.split == 2 ? 2 : 1);   // X items (two parts per matrix at level 2)
        const int rb = b.batch * (b.split ? 2 : 1);        // r x r items
        ok = ok && make_map(&b.ut_a, ut, true, b.c, b.r, xb, b.ldu, 64, kBM);
        ok = ok && make_map(&b.ut_b, ut, true, b.c, b.r, xb, b.ldu, 64, kBN);
        ok = ok && make_map(&b.ut_mn, ut, true, b.c, b.r, xb, b.ldu, 64, 64);
        const bool aligned4 = b.batched() && !b.split && b.r % 64 == 0 && b.c % 64 == 0;
        if (aligned4) {
            ok = ok && make_map4(&b.utk, ut, true, b.c, b.r, b.batch, b.ldu, 128, 1);
            ok = ok && make_map4(&b.utt, ut, true, b.c, b.r, b.batch, b.ldu, 64, 2);
        }
        if (restarts) {
            b.ut1_off = (long long)(L.o_ut1[k] / 2);
            __nv_bfloat16* ut1 = p->ut + b.ut1_off;
            ok = ok && make_map(&b.ut1_a, ut1, true, b.c, b.r, xb, b.ldu, 64, kBM);
            ok = ok && make_map(&b.ut1_b, ut1, true, b.c, b.r, xb, b.ldu, 64, kBN);
            ok = ok && make_map(&b.ut1_mn, ut1, true, b.c, b.r, xb, b.ldu, 64, 64);
            if (aligned4) {
                ok = ok && make_map4(&b.ut1k, ut1, true, b.c, b.r, b.batch, b.ldu, 128, 1);
                ok = ok && make_map4(&b.ut1t, ut1, true, b.c, b.r, b.batch, b.ldu, 64, 2);
            }
        }
        if (!b.batched()) continue;   // the one-CTA kernels keep their r x r operands on chip
        const size_t rr = (size_t)rb * b.r * b.ldr;
        const size_t step = (size_t)round_up((long long)rr * 2, 256);
        char* rbase = base + L.o_region + L.o_rr[k];
        b.G[0] = reinterpret_cast<__half*>(rbase);
        b.G[1] = reinterpret_cast<__half*>(rbase + step);
        b.P = reinterpret_cast<__half*>(rbase + 2 * step);
        b.T = reinterpret_cast<__half*>(rbase + 3 * step);
        b.Q[0] = reinterpret_cast<__half*>(rbase + 4 * step);
        b.Q[1] = reinterpret_cast<__half*>(rbase + 5 * step);
        b.Qb = reinterpret_cast<__nv_bfloat16*>(base + L.o_region + L.o_qb[k]);
        ok = ok && make_map(&b.qb_a, b.Qb, true, b.r, b.r, rb, b.ldr, 64, kBM);
        for (int g = 0; g < 2; ++g) {
            ok = ok && make_map(&b.ga[g], b.G[g], false, b.r, b.r, rb, b.ldr, 64, kBM);
            ok = ok && make_map(&b.gb[g], b.G[g], false, b.r, b.r, rb, b.ldr, 64, kBN);
            ok = ok && make_map(&b.qb[g], b.Q[g], false, b.r, b.r, rb, b.ldr, 64, kBN);
            ok = ok && make_map(&b.qa[g], b.Q[g], false, b.r, b.r, rb, b.ldr, 64, kBM);
        }
        ok = ok && make_map(&b.pa, b.P, false, b.r, b.r, rb, b.ldr, 64, kBM);
        ok = ok && make_map(&b.pb, b.P, false, b.r, b.r, rb, b.ldr, 64, kBN);
        ok = ok && make_map(&b.tb, b.T, false, b.r, b.r, rb, b.ldr, 64, kBN);
        ok = ok && make_map(&b.ta, b.T, false, b.r, b.r, rb, b.ldr, 64, kBM);
        for (int g = 0; g < 2; ++g) {
            ok = ok && make_out_map(&b.og[g], b.G[g], false, b.r, rb, b.ldr);
            ok = ok && make_out_map(&b.oq[g], b.Q[g], false, b.r, rb, b.ldr);
        }
        ok = ok && make_out_map(&b.op, b.P, false, b.r, rb, b.ldr);
        ok = ok && make_out_map(&b.ot, b.T, false, b.r, rb, b.ldr);
        ok = ok && make_out_map(&b.oqb, b.Qb, true, b.r, rb, b.ldr);
        if (aligned4) {
            auto kt = [&](CUtensorMap* k, CUtensorMap* t, void* buf, bool bf) {
                return make_map4(k, buf, bf, b.r, b.r, b.batch, b.ldr, 128, 1) &&
                       make_map4(t, buf, bf, b.r, b.r, b.batch, b.ldr, 64, 2);
            };
            for (int g = 0; g < 2; ++g) {
                ok = ok && kt(&b.gk[g], &b.gt[g], b.G[g], false);
                ok = ok && kt(&b.qk[g], &b.qt[g], b.Q[g], false);
            }
            ok = ok && kt(&b.pk, &b.pt, b.P, false) && kt(&b.tk, &b.tt, b.T, false) && kt(&b.qbk, &b.qbt, b.Qb, true);
        }
    }
    ok = ok && cudaMallocHost(&p->h_pinned, sizeof(void*) * 3 * n) == cudaSuccess;
    ok = ok && cudaMallocHost(&p->h_wmap, (sizeof(CUtensorMap) + 1) * n) == cudaSuccess;
    ok = ok && cudaMemset(p->d_wmap_ok, 0, n) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&p->upload_ev, cudaEventDisableTiming) == cudaSuccess;
    ok = ok && gemm_prepare(p->device) == cudaSuccess;
    ok = ok && ns_f32_prepare() == cudaSuccess;
    if (ok && !p->opts.single_sm_gemm) {
        int clusters = 0;
        ok = gemm2_max_clusters(&clusters) == cudaSuccess;
        p->pair_clusters = clusters;
    }
    for (auto& ch : p->chunks) {   // lower-triangle storage where the 4-D operand view is exact
        bool aligned = true;
        for (int k : ch.buckets) {
            const Bucket& b = p->buckets[k];
            if (b.batched() && b.r > kBM) aligned = aligned && !b.split && b.r % 64 == 0 && b.c % 64 == 0;
        }
        ch.lower_ok = p->pair_clusters > 0 && aligned;
        ch.lower = ch.lower_ok && !p->opts.full_symmetric;
    }
    if (ok && p->pair_clusters > 1) {
        bool any = false;
        for (auto& ch : p->chunks) {
            double fused_bytes = 0, chain_flops = 0;
            for (int k : ch.buckets) {
                const Bucket& b = p->buckets[k];
                const double r = b.r, c = b.c;
                if (b.fused)
                    fused_bytes += 12.0 * r * c * b.batch;
                else if (b.batched())
                    chain_flops += (3.0 * r * r * c + 17.0 * r * r * r) * b.batch;
            }
            if (fused_bytes > 0 && chain_flops > 0) {
                const int kmax = std::min(p->pair_clusters - 1, (p->sm_count - 2) / 2);
                ch.mixed = true;
                ch.chain_est = std::max(std::min(choose_chain_clusters(fused_bytes, chain_flops, p->pair_clusters),
                                                 kmax), 0);
                const int k = p->opts.chain_clusters == 0 ? ch.chain_est
                                                          : std::min(std::max(p->opts.chain_clusters, 0), kmax);
                ch.chain_clusters = k;
                any = true;   // the second stream also serves muon_plan_tune's candidates
            }
        }
        if (any)
            ok = cudaStreamCreateWithFlags(&p->s2, cudaStreamNonBlocking) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p->fork_ev, cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p->join_ev, cudaEventDisableTiming) == cudaSuccess;
    }
    ok = ok && cudaDeviceSynchronize() == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        free_plan(p);
        return MUON_ERR_CUDA;
    }
    p->h_cache.assign(3 * n, nullptr);
    *out = p;
    return MUON_OK;
}

muon_status muon_plan_create(const muon_shape* shapes, int32_t n, muon_dtype grad_dtype, const muon_plan_opts* opts,
                             muon_plan* out) {
    if (!out) return MUON_ERR_INVALID_ARG;
    *out = nullptr;
    const muon_status bad = check_plan_args(shapes, n, grad_dtype, opts);
    if (bad != MUON_OK) return bad;
    muon_plan_s* p = new (std::nothrow) muon_plan_s();
    if (!p) return MUON_ERR_OOM;
    try {
        return plan_build(p, shapes, n, grad_dtype, opts, out);
    } catch (...) {   // std::vector's bad_alloc / length_error: host memory
        free_plan(p);
        return MUON_ERR_OOM;
    }
}

muon_status muon_partition(const muon_shape* shapes, int32_t n, int32_t world, const double* cost, int32_t* owner,
                           double* load) {
    if (!shapes || n <= 0 || !owner || world < 1 || world > 65536) return MUON_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        if (shapes[i].rows <= 0 || shapes[i].cols <= 0 || shapes[i].rows > kMaxDim || shapes[i].cols > kMaxDim)
            return MUON_ERR_INVALID_ARG;
        if (cost && !(std::isfinite(cost[i]) && cost[i] >= 0.0)) return MUON_ERR_INVALID_ARG;
    }
    try {
        std::vector<double> c(n);
        for (int i = 0; i < n; ++i) {
            if (cost) {
                c[i] = cost[i];
                continue;
            }
            const double r = (double)std::min(shapes[i].rows, shapes[i].cols);
            const double cc = (double)std::max(shapes[i].rows, shapes[i].cols);
            const double t_mem = 24.0 * r * cc / 6.8e12;
            const double t_tc = r <= kSmallMaxR ? 0.0 : (3.0 * r * r * cc + 17.0 * r * r * r) / 1.5e15;
            c[i] = std::max(t_mem, t_tc);
        }
        std::vector<int> order(n);
        for (int i = 0; i < n; ++i) order[i] = i;
        std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return c[a] > c[b]; });
        std::vector<double> l(world, 0.0);
        for (int i : order) {
            int best = 0;
            for (int r = 1; r < world; ++r)
                if (l[r] < l[best]) best = r;
            owner[i] = best;
            l[best] += c[i];
        }
        if (load)
            for (int r = 0; r < world; ++r) load[r] = l[r];
        return MUON_OK;
    } catch (...) {   // host memory
        return MUON_ERR_OOM;
    }
}

muon_status muon_plan_workspace_size(const muon_shape* shapes, int32_t n, muon_dtype grad_dtype,
                                     const muon_plan_opts* opts, int64_t* bytes, int32_t* n_buckets,
                                     int32_t* n_chunks) {
    const muon_status bad = check_plan_args(shapes, n, grad_dtype, opts);
    if (bad != MUON_OK) return bad;
    try {
        muon_plan_s plan;   // host fields only: nothing is created on the device
        if (opts) plan.opts = *opts;
        plan.shapes.assign(shapes, shapes + n);
        if (plan.opts.full_rows) plan.full_rows.assign(plan.opts.full_rows, plan.opts.full_rows + n);
        if (plan.opts.precision_of) plan.prec_of.assign(plan.opts.precision_of, plan.opts.precision_of + n);
        plan.opts.full_rows = nullptr;
        plan.opts.precision_of = nullptr;
        Layout L;
        const muon_status st = plan_layout(&plan, L);
        if (st != MUON_OK) return st;
        if (bytes) *bytes = (int64_t)plan.ws_bytes;
        if (n_buckets) *n_buckets = (int32_t)plan.buckets.size();
        if (n_chunks) *n_chunks = (int32_t)plan.chunks.size();
        return MUON_OK;
    } catch (...) {   // host memory
        return MUON_ERR_OOM;
    }
}

void muon_plan_destroy(muon_plan p) {
    if (!p) return;
    cudaDeviceSynchronize();
    free_plan(p);
}

// The RowNorm kernels over one set of lists (m <= n rows; m > n column statistics,
// finalize, apply).
static muon_status rownorm_launch(muon_plan_s* p, const ListDev* rows, const ListDev& stats,
                                  const ListDev& fin, const ListDev& apply, float lr, float wd, float mu, float eps,
                                  cudaStream_t s, int* launches) {
    ElemArgs a{};
    for (int cl = 0; cl < kRowClasses; ++cl) {
        a = elem_args(p, rows[cl], mu, lr, wd, eps);
        MUON_TRY(launch_rownorm_rows(a, rows[cl].blocks, rownorm_class_vec(cl), s));
        *launches += rows[cl].blocks > 0;
    }
    a = elem_args(p, stats, mu, lr, wd, eps);
    a.partials = p->cpartials;
    MUON_TRY(launch_rownorm_colstats(a, stats.blocks, s));
    a = elem_args(p, fin, mu, lr, wd, eps);
    a.partials = p->cpartials;
    MUON_TRY(launch_rownorm_colfinal(a, fin.blocks, s));
    a = elem_args(p, apply, mu, lr, wd, eps);
    MUON_TRY(launch_rownorm_colapply(a, apply.blocks, s));
    *launches += stats.blocks > 0 ? 3 : 0;
    return MUON_OK;
}

muon_status muon_rownorm_step(muon_plan p, float* const* params, const void* const* grads, float* const* momentum,
                              float lr, float wd, float mu, float eps, void* stream) {
    if (!p) return MUON_ERR_INVALID_ARG;
    if (!p->full_rows.empty()) return MUON_ERR_UNSUPPORTED;   // the shard calls sum norms across shards
    if (!finite_nonneg(lr) || !finite_nonneg(wd) || !std::isfinite(mu) || mu < 0.f || mu >= 1.f ||
        !std::isfinite(eps) || eps <= 0.f)
        return MUON_ERR_INVALID_ARG;
    muon_status st = check_pointers(p, params, grads, momentum);
    if (st != MUON_OK) return st;
    if ((st = check_device(p)) != MUON_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = upload_pointers(p, params, grads, momentum, s)) != MUON_OK) return st;
    muon_plan_s::StepEvents* se = nullptr;
    if (p->opts.timing && !(se = next_events(p))) return MUON_ERR_CUDA;
    if (se) {
        se->ns = false;
        MUON_TRY(cudaEventRecord(se->e[0], s));
    }
    int launches = 0;
    if ((st = rownorm_launch(p, p->rn_rows, p->rn_stats, p->rn_final, p->rn_apply, lr, wd, mu, eps, s,
                             &launches)) != MUON_OK)
        return st;
    if (se) MUON_TRY(cudaEventRecord(se->e[5], s));
    p->last_launches = launches;
    return MUON_OK;
}

// Checks shared by the two shard calls.
static muon_status shard_check(muon_plan_s* p, float* const* params, const void* const* grads,
                               float* const* momentum, float lr, float wd, float mu, float eps, const void* colsq) {
    if (!p) return MUON_ERR_INVALID_ARG;
    if (p->full_rows.empty()) return MUON_ERR_UNSUPPORTED;
    if (!finite_nonneg(lr) || !finite_nonneg(wd) || !std::isfinite(mu) || mu < 0.f || mu >= 1.f ||
        !std::isfinite(eps) || eps <= 0.f || (p->colsq_len > 0 && !colsq))
        return MUON_ERR_INVALID_ARG;
    muon_status st = check_pointers(p, params, grads, momentum);
    if (st != MUON_OK) return st;
    return check_device(p);
}

muon_status muon_rownorm_shard_stats(muon_plan p, float* const* params, const void* const* grads,
                                     float* const* momentum, float lr, float wd, float mu, float eps, float* colsq,
                                     void* stream) {
    muon_status st = shard_check(p, params, grads, momentum, lr, wd, mu, eps, colsq);
    if (st != MUON_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = upload_pointers(p, params, grads, momentum, s)) != MUON_OK) return st;
    int launches = 0;
    ElemArgs a{};
    for (int cl = 0; cl < kRowClasses; ++cl) {   // rows complete in the shard: the whole step
        a = elem_args(p, p->rn_rows[cl], mu, lr, wd, eps);
        MUON_TRY(launch_rownorm_rows(a, p->rn_rows[cl].blocks, rownorm_class_vec(cl), s));
        launches += p->rn_rows[cl].blocks > 0;
    }
    a = elem_args(p, p->rn_stats, mu, lr, wd, eps);   // momentum and slab sums of U^2
    a.partials = p->cpartials;
    MUON_TRY(launch_rownorm_colstats(a, p->rn_stats.blocks, s));
    a = elem_args(p, p->rn_final, mu, lr, wd, eps);   // this shard's column sums into colsq
    a.partials = p->cpartials;
    MUON_TRY(launch_rownorm_colsum(a, p->rn_final.blocks, colsq, s));
    launches += p->rn_stats.blocks > 0 ? 2 : 0;
    p->last_launches = launches;
    return MUON_OK;
}

muon_status muon_rownorm_shard_apply(muon_plan p, float* const* params, const void* const* grads,
                                     float* const* momentum, float lr, float wd, float mu, float eps,
                                     const float* colsq, void* stream) {
    muon_status st = shard_check(p, params, grads, momentum, lr, wd, mu, eps, colsq);
    if (st != MUON_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = upload_pointers(p, params, grads, momentum, s)) != MUON_OK) return st;
    ElemArgs a = elem_args(p, p->rn_final, mu, lr, wd, eps);
    MUON_TRY(launch_rownorm_colinv(a, p->rn_final.blocks, colsq, s));
    a = elem_args(p, p->rn_apply, mu, lr, wd, eps);
    MUON_TRY(launch_rownorm_colapply(a, p->rn_apply.blocks, s));
    p->last_launches = p->rn_apply.blocks > 0 ? 2 : 0;
    return MUON_OK;
}

muon_status muon_step(muon_plan p, float* const* params, const void* const* grads, float* const* momentum, float lr,
                      float wd, float mu, int32_t ns_steps, muon_mode mode, void* stream) {
    if (!p) return MUON_ERR_INVALID_ARG;
    if (mode == MUON_MODE_ROWNORM) return muon_rownorm_step(p, params, grads, momentum, lr, wd, mu, 1e-8f, stream);
    if (mode != MUON_MODE_NS) return MUON_ERR_INVALID_ARG;
    return muon_step_ex(p, params, grads, momentum, lr, wd, mu, ns_steps, nullptr, 0, stream);
}

// Host side of muon_step_host inside the NS step: the chunk's gradients arrive on
// hc.in (in_ev), its parameters go back on hc.out.
struct HostIO {
    float* const* params_host;   // may be null
};

static muon_status ns_step(muon_plan p, float* const* params, const void* const* grads, float* const* momentum,
                           float lr, float wd, float mu, int32_t ns_steps, const float* coeffs, int32_t restart,
                           void* stream, const HostIO* io);

muon_status muon_step_ex(muon_plan p, float* const* params, const void* const* grads, float* const* momentum,
                         float lr, float wd, float mu, int32_t ns_steps, const float* coeffs, int32_t restart,
                         void* stream) {
    return ns_step(p, params, grads, momentum, lr, wd, mu, ns_steps, coeffs, restart, stream, nullptr);
}

static muon_status ns_step(muon_plan p, float* const* params, const void* const* grads, float* const* momentum,
                           float lr, float wd, float mu, int32_t ns_steps, const float* coeffs, int32_t restart,
                           void* stream, const HostIO* io) {
    if (!p) return MUON_ERR_INVALID_ARG;
    if (!p->full_rows.empty()) return MUON_ERR_UNSUPPORTED;   // dim-0 shard plans: RowNorm only
    const int max_steps = p->opts.max_ns_steps > 0 ? p->opts.max_ns_steps : kMaxNsSteps;
    if (!finite_nonneg(lr) || !finite_nonneg(wd) || !std::isfinite(mu) || mu < 0.f || mu >= 1.f ||
        ns_steps < 0 || ns_steps > max_steps || restart < 0 || restart > kMaxNsSteps)
        return MUON_ERR_INVALID_ARG;
    if (coeffs && !(std::isfinite(coeffs[0]) && std::isfinite(coeffs[1]) && std::isfinite(coeffs[2])))
        return MUON_ERR_INVALID_ARG;
    const float ca = coeffs ? coeffs[0] : kNsA, cb = coeffs ? coeffs[1] : kNsB, cc = coeffs ? coeffs[2] : kNsC;
    // segments of at most `period` Gram steps (one segment unless restarted)
    const int period = restart > 0 ? restart : kMaxNsSteps;
    const int nseg = ns_steps == 0 ? 1 : (ns_steps + period - 1) / period;
    if (nseg > 1 && p->opts.max_ns_steps <= 0) return MUON_ERR_UNSUPPORTED;
    muon_status st = check_pointers(p, params, grads, momentum);
    if (st != MUON_OK) return st;
    if ((st = check_device(p)) != MUON_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = upload_pointers(p, params, grads, momentum, s)) != MUON_OK) return st;
    muon_plan_s::StepEvents* se = nullptr;
    if (p->opts.timing && !(se = next_events(p))) return MUON_ERR_CUDA;
    const int n = (int)p->shapes.size();
    int launches = 0;

    // algorithmic tensor FLOPs of the GEMM stages (the fused r <= 128 step is
    // HBM-bound and timed as a stage of its own)
    double fl_syrk = 0, fl_rr = 0, fl_final = 0;
    for (auto& b : p->buckets) {
        if (!b.batched()) continue;
        const double r = b.r, c = b.c;
        for (int sg = 0; sg < nseg; ++sg) {   // per segment: SYRK, 4Js-3 r x r products, r x c product
            const int Js = sg == nseg - 1 ? ns_steps - sg * period : period;
            fl_syrk += b.batch * r * r * c;
            fl_final += b.batch * 2.0 * r * r * c;
            const int nrr = Js == 0 ? 0 : (Js == 1 ? 1 : 4 * Js - 3);
            fl_rr += b.batch * (double)nrr * r * r * r;
        }
    }
    if (se) {
        p->flops[0] += fl_syrk;
        p->flops[1] += fl_rr;
        p->flops[2] += fl_final;
    }
    if (se) se->ns = true;
    for (size_t ci = 0; ci < p->chunks.size(); ++ci) {
        const muon_plan_s::Chunk& ch = p->chunks[ci];
        cudaEvent_t* ev = se ? &se->e[7 * ci] : nullptr;
        if (io) MUON_TRY(cudaStreamWaitEvent(s, p->hc.in_ev[ci], 0));   // this chunk's gradients
        // ---- momentum, Nesterov, sum of squares, bf16 X0 (oriented), for this chunk
        if (ev) MUON_TRY(cudaEventRecord(ev[0], s));
        ElemArgs a = elem_args(p, ch.mom_rows, mu, lr, wd, 0.f);
        MUON_TRY(launch_momentum_rows(a, ch.mom_rows.blocks, s));
        launches += ch.mom_rows.blocks > 0;
        a = elem_args(p, ch.mom_tiles, mu, lr, wd, 0.f);
        MUON_TRY(launch_momentum_tiles(a, ch.mom_tiles.blocks, s));
        launches += ch.mom_tiles.blocks > 0;
        a = elem_args(p, ch.all, mu, lr, wd, 0.f);
        MUON_TRY(launch_norm_finalize(a, s));
        ++launches;
        if (ev) MUON_TRY(cudaEventRecord(ev[1], s));


        // Plans with both fused and batched matrices run them side by side: the batched
        // products on p->s2 (forked here, joined after the final product) with
        // chain_clusters CTA pairs, the fused kernel on the remaining SMs.
        const bool split = ch.chain_clusters > 0;
        cudaStream_t sc = split ? p->s2 : s;
        const int gc_clusters = split ? ch.chain_clusters : p->pair_clusters;
        const int g_grid1 = split ? 2 * ch.chain_clusters : p->sm_count;
        const int fused_grid = split ? p->sm_count - 2 * ch.chain_clusters : p->sm_count;
        if (se) se->split[ci] = split;
        if (split) {
            MUON_TRY(cudaEventRecord(p->fork_ev, s));
            MUON_TRY(cudaStreamWaitEvent(p->s2, p->fork_ev, 0));
        }

        // ---- r <= 128: the whole step of each matrix (SYRK, recursion, final product +
        // update) in one fused launch, on all SMs but those left to the batched products
        {
            GemmLaunch Ls;
            std::memset(&Ls, 0, sizeof(Ls));
            Ls.status = p->status;
            float* const* W = reinterpret_cast<float* const*>(p->d_ptrs + 2 * n);
            auto flush_small = [&]() -> muon_status {
                if (Ls.nprob == 0) return MUON_OK;
                const muon_status st2 = cuda_status(ns_small_launch(Ls, fused_grid, s));
                ++launches;
                std::memset(&Ls, 0, sizeof(Ls));
                Ls.status = p->status;
                return st2;
            };
            for (int bk : ch.buckets) {
                Bucket& b = p->buckets[bk];
                if (!b.fused) continue;
                if (Ls.nprob == kMaxProblems && (st = flush_small()) != MUON_OK) return st;
                GemmProblem q = problem(b.r, b.c, b.r, b.batch, false, kEpiApply);
                q.tiles_per_item = 1;
                q.tile_begin = Ls.total_tiles;
                q.alpha = p->alpha + b.slot_base;
                q.item_mat = b.d_item_mat;
                q.W = W;
                q.wmap = p->d_wmap;        // W pieces by TMA for the matrices with a valid map
                q.wmap_ok = p->d_wmap_ok;
                q.transposed = p->d_transposed;
                q.Odbg = b.Odbg;
                q.lr = lr;
                q.wd = wd;
                q.scale = 0.2f * std::sqrt((float)b.c);
                q.out_scale = b.gscale;
                q.coef_a = ca;
                q.coef_b = cb / b.gscale;
                q.coef_c = cc / (b.gscale * b.gscale);
                q.ns_steps = ns_steps;
                Ls.mapA[Ls.nprob] = b.ut_a;
                Ls.mapB[Ls.nprob] = b.ut_mn;
                Ls.prob[Ls.nprob] = q;
                Ls.nprob++;
                Ls.total_tiles += b.batch;
            }
            if ((st = flush_small()) != MUON_OK) return st;
        }
        // ---- small nearly square matrices: the whole step in fp32 on CUDA cores
        {
            F32Launch Lf;
            std::memset(&Lf, 0, sizeof(Lf));
            auto reset_f32 = [&]() {
                std::memset(&Lf, 0, sizeof(Lf));
                Lf.mats = p->d_mats;
                Lf.G = const_cast<const void* const*>(p->d_ptrs);
                Lf.M = reinterpret_cast<float* const*>(p->d_ptrs + n);
                Lf.W = reinterpret_cast<float* const*>(p->d_ptrs + 2 * n);
                Lf.mu = mu;
                Lf.lr = lr;
                Lf.wd = wd;
                Lf.grad_bf16 = p->gdt == MUON_BF16;
            };
            auto flush_f32 = [&]() -> muon_status {
                if (Lf.nprob == 0) return MUON_OK;
                const muon_status st2 = cuda_status(ns_f32_launch(Lf, fused_grid, s));
                ++launches;
                reset_f32();
                return st2;
            };
            reset_f32();
            for (int bk : ch.buckets) {
                Bucket& b = p->buckets[bk];
                if (!b.f32) continue;
                if (Lf.nprob == kMaxProblems && (st = flush_f32()) != MUON_OK) return st;
                F32Problem& q = Lf.prob[Lf.nprob++];
                q.r = b.r;
                q.c = b.c;
                q.batch = b.batch;
                q.item_begin = Lf.total;
                q.ns_steps = ns_steps;
                q.item_mat = b.d_item_mat;
                q.alpha = p->alpha + b.slot_base;
                q.Odbg = b.Odbg;
                q.coef_a = ca;
                q.coef_b = cb;
                q.coef_c = cc;
                q.scale = 0.2f * std::sqrt((float)b.c);
                Lf.total += b.batch;
            }
            if ((st = flush_f32()) != MUON_OK) return st;
        }
        if (ev) MUON_TRY(cudaEventRecord(ev[6], s));


        // ---- batched matrices: NS in segments of at most `period` Gram steps; between
        // segments the iterate goes to the other X buffer (xc: 0 X0, 1 the second)
        for (int sg = 0, xc = 0; sg < nseg; ++sg, xc ^= 1) {
            const bool first = sg == 0, last = sg == nseg - 1;
            const int Js = last ? ns_steps - sg * period : period;
            // ---- G0' = s alpha^2 X0 X0^T (lower triangle, mirrored), all buckets in one launch
            {
                Grouper g(p, sc, true, ch.lower, gc_clusters, g_grid1);
                for (int bk : ch.buckets) {
                    Bucket& b = p->buckets[bk];
                    if (!b.batched()) continue;
                    GemmProblem q = problem(b.r, b.r, b.c, b.batch, true, kEpiSyrk);
                    q.a_split = q.b_split = b.split == 2;
                    q.out_split = b.split != 0;
                    q.C = b.G[0];
                    q.strideC = (long long)b.r * b.ldr;
                    q.ldc = b.ldr;
                    q.alpha = (first ? p->alpha : p->ones) + b.slot_base;
                    q.out_scale = b.gscale;
                    q.tma_out = kTmaOutC;
                    if (xc == 0)
                        g.add(b.ut_a, b.ut_b, b.ut_a, q, &b.og[0], nullptr, {&b.utk}, {&b.utk});
                    else
                        g.add(b.ut1_a, b.ut1_b, b.ut1_a, q, &b.og[0], nullptr, {&b.ut1k}, {&b.ut1k});
                }
                g.flush();
                if (g.st != MUON_OK) return g.st;
                launches += g.launches;
            }
            if (ev && first) MUON_TRY(cudaEventRecord(ev[2], sc));


            // ---- Newton-Schulz in the Gram space (fp16 operands, G carried as s G)
            const int J = Js;
            int gc = 0;   // current G buffer
            int qc = 0;   // current Q buffer
            auto rr_problem = [](const Bucket& b, int epi) {
                GemmProblem q = problem(b.r, b.r, b.r, b.batch, true, epi);
                q.strideC = (long long)b.r * b.ldr;
                q.ldc = b.ldr;
                q.a_split = q.b_split = q.out_split = b.split != 0;   // every r x r operand and result
                return q;
            };
            for (int k = 1; k <= J; ++k) {
                {   // P = aI + (b/s) G' + (c/s^2) G'^2 (at k = 1 this is also Q_1)
                    Grouper g(p, sc, false, ch.lower, gc_clusters, g_grid1);
                    for (int bk : ch.buckets) {
                    Bucket& b = p->buckets[bk];
                    if (!b.batched()) continue;
                        GemmProblem q = rr_problem(b, kEpiPoly);
                        q.C = b.P;
                        if (k == 1 && J > 1) q.C2 = b.Q[0];
                        if (k == 1 && J == 1) q.Cb = b.Qb;
                        q.Gin = b.G[gc];
                        q.coef_a = ca;
                        q.coef_b = cb / b.gscale;
                        q.coef_c = cc / (b.gscale * b.gscale);
                        // fp16 P (and the fp16 copy Q_1): TMA stores; P with a bf16 Q_1 (J = 1): per thread
                        q.tma_out = q.Cb ? 0 : (kTmaOutC | (q.C2 ? kTmaOutC2 : 0));
                        const Maps4 g4{&b.gk[gc], &b.gt[gc], true};
                        g.add(b.ga[gc], b.gb[gc], b.ga[gc], q, &b.op, q.C2 ? &b.oq[0] : nullptr, g4, g4, &b.og[gc]);
                    }
                    g.flush();
                    if (g.st != MUON_OK) return g.st;
                    launches += g.launches;
                }
                {   // Q' = P Q (k >= 2) and T = P P (k < J), independent: one launch
                    Grouper g(p, sc, false, ch.lower, gc_clusters, g_grid1);
                    for (int bk : ch.buckets) {
                    Bucket& b = p->buckets[bk];
                    if (!b.batched()) continue;
                        if (k >= 2) {
                            GemmProblem q = rr_problem(b, kEpiPlain);
                            if (k < J) {
                                q.C = b.Q[qc ^ 1];
                                q.tma_out = kTmaOutC;
                                g.add(b.pa, b.qb[qc], b.qa[qc], q, &b.oq[qc ^ 1], nullptr, {&b.pk, &b.pt, true},
                                      {&b.qk[qc], &b.qt[qc], true});
                            } else {
                                q.Cb = b.Qb;
                                q.tma_out = kTmaOutC | kTmaOutBf16;
                                g.add(b.pa, b.qb[qc], b.qa[qc], q, &b.oqb, nullptr, {&b.pk, &b.pt, true},
                                      {&b.qk[qc], &b.qt[qc], true});
                            }
                        }
                        if (k < J) {
                            GemmProblem q = rr_problem(b, kEpiPlain);
                            q.C = b.T;
                            q.tma_out = kTmaOutC;
                            g.add(b.pa, b.pb, b.pa, q, &b.ot, nullptr, {&b.pk, &b.pt, true}, {&b.pk, &b.pt, true});
                        }
                    }
                    g.flush();
                    if (g.st != MUON_OK) return g.st;
                    launches += g.launches;
                    if (k >= 2) qc ^= 1;
                }
                if (k < J) {   // G'' = G' T
                    Grouper g(p, sc, false, ch.lower, gc_clusters, g_grid1);
                    for (int bk : ch.buckets) {
                    Bucket& b = p->buckets[bk];
                    if (!b.batched()) continue;
                        GemmProblem q = rr_problem(b, kEpiPlain);
                        q.C = b.G[gc ^ 1];
                        q.tma_out = kTmaOutC;
                        g.add(b.ga[gc], b.tb, b.ta, q, &b.og[gc ^ 1], nullptr, {&b.gk[gc], &b.gt[gc], true},
                              {&b.tk, &b.tt, true});
                    }
                    g.flush();
                    if (g.st != MUON_OK) return g.st;
                    launches += g.launches;
                    gc ^= 1;
                }
            }
            if (J == 0) {
                for (int bk : ch.buckets) {
                    Bucket& b = p->buckets[bk];
                    if (!b.batched()) continue;
                    MUON_TRY(launch_identity_bf16(b.Qb, b.r, b.ldr, b.batch, b.split != 0, sc));
                    ++launches;
                }
            }
            if (ev && last) MUON_TRY(cudaEventRecord(ev[3], sc));

            // ---- last segment: O = alpha Q X, fused W <- W - lr (s O + wd W) in the stored
            // layout; earlier segments: X' = alpha Q X (bf16) into the other X buffer
            {
                Grouper g(p, sc, true, ch.lower, gc_clusters, g_grid1);
                if (last) {   // W pieces by TMA when every batched matrix of the chunk has a W map
                    const unsigned char* wok = reinterpret_cast<const unsigned char*>(p->h_wmap + n);
                    bool all = true;
                    for (int bk : ch.buckets)
                        if (p->buckets[bk].batched())
                            for (int i : p->buckets[bk].mats) all = all && wok[i];
                    g.wtma = all;
                }
                float* const* W = reinterpret_cast<float* const*>(p->d_ptrs + 2 * n);
                for (int bk : ch.buckets) {
                    Bucket& b = p->buckets[bk];
                    if (!b.batched()) continue;
                    GemmProblem q = problem(b.r, b.c, b.r, b.batch, false, last ? kEpiApply : kEpiXout);
                    q.b_mn = 1;
                    q.a_split = b.split != 0;             // Q in two bf16 parts
                    q.b_split = b.split == 2;             // X in two bf16 parts
                    q.out_split = !last && b.split == 2;  // X' between segments
                    q.alpha = (first ? p->alpha : p->ones) + b.slot_base;
                    if (last) {
                        q.item_mat = b.d_item_mat;
                        q.W = W;
                        q.wmap = p->d_wmap;
                        q.wmap_ok = p->d_wmap_ok;
                        q.transposed = p->d_transposed;
                        q.Odbg = b.Odbg;
                        q.lr = lr;
                        q.wd = wd;
                        q.scale = 0.2f * std::sqrt((float)b.c);
                    } else {
                        q.Cb = p->ut + (xc == 0 ? b.ut1_off : b.ut_off);
                        q.ldc = b.ldu;
                        q.strideC = (long long)b.r * b.ldu;
                    }
                    const CUtensorMap& xm = xc == 0 ? b.ut_mn : b.ut1_mn;
                    g.add(b.qb_a, xm, xm, q, nullptr, nullptr, {&b.qbk, &b.qbt, true},
                          {nullptr, xc == 0 ? &b.utt : &b.ut1t});
                }
                g.flush();
                if (g.st != MUON_OK) return g.st;
                launches += g.launches;
            }
            if (ev && last) MUON_TRY(cudaEventRecord(ev[4], sc));
        }
        if (split) {
            MUON_TRY(cudaEventRecord(p->join_ev, p->s2));
            MUON_TRY(cudaStreamWaitEvent(s, p->join_ev, 0));
        }
        if (io && io->params_host) {   // this chunk's parameters are final: copy them back
            MUON_TRY(cudaEventRecord(p->hc.out_ev[ci], s));
            MUON_TRY(cudaStreamWaitEvent(p->hc.out, p->hc.out_ev[ci], 0));
            for (int bk : ch.buckets)
                for (int i : p->buckets[bk].mats)
                    MUON_TRY(cudaMemcpyAsync(io->params_host[i], params[i],
                                             (size_t)(p->mats[i].m * p->mats[i].n) * sizeof(float),
                                             cudaMemcpyDefault, p->hc.out));
        }
    }
    p->last_launches = launches;
    return MUON_OK;
}

// Copy streams and events of muon_step_host, created on first use.
static muon_status host_copy_setup(muon_plan_s* p) {
    auto& h = p->hc;
    if (h.in) return MUON_OK;
    const size_t nc = p->chunks.size();
    bool ok = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&h.entry_ev, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&h.end_ev, cudaEventDisableTiming) == cudaSuccess;
    bool host_ok = true;
    try {
        h.in_ev.assign(nc, nullptr);
        h.out_ev.assign(nc, nullptr);
    } catch (...) {
        ok = host_ok = false;   // host memory
    }
    for (size_t c = 0; ok && c < nc; ++c)
        ok = cudaEventCreateWithFlags(&h.in_ev[c], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&h.out_ev[c], cudaEventDisableTiming) == cudaSuccess;
    if (ok) return MUON_OK;
    if (host_ok) g_last_cuda_error = cudaGetLastError();
    if (h.in) cudaStreamDestroy(h.in);
    if (h.out) cudaStreamDestroy(h.out);
    h.in = h.out = nullptr;
    for (cudaEvent_t& e : h.in_ev)
        if (e) cudaEventDestroy(e);
    for (cudaEvent_t& e : h.out_ev)
        if (e) cudaEventDestroy(e);
    h.in_ev.clear();
    h.out_ev.clear();
    if (h.entry_ev) cudaEventDestroy(h.entry_ev);
    if (h.end_ev) cudaEventDestroy(h.end_ev);
    h.entry_ev = h.end_ev = nullptr;
    return host_ok ? MUON_ERR_CUDA : MUON_ERR_OOM;
}

muon_status muon_step_host(muon_plan p, float* const* params, const void* const* grads, float* const* momentum,
                           const void* const* grads_host, float* const* params_host, float lr, float wd,
                           float mu, int32_t ns_steps, muon_mode mode, void* stream) {
    if (!p || !grads_host) return MUON_ERR_INVALID_ARG;
    if (!p->full_rows.empty()) return MUON_ERR_UNSUPPORTED;
    const int n = (int)p->shapes.size();
    for (int i = 0; i < n; ++i)
        if (!grads_host[i] || (params_host && !params_host[i])) return MUON_ERR_INVALID_ARG;
    // every check of the step itself before anything is enqueued
    const int max_steps = p->opts.max_ns_steps > 0 ? p->opts.max_ns_steps : kMaxNsSteps;
    if (!finite_nonneg(lr) || !finite_nonneg(wd) || !std::isfinite(mu) || mu < 0.f || mu >= 1.f)
        return MUON_ERR_INVALID_ARG;
    if (mode == MUON_MODE_NS) {
        if (ns_steps < 0 || ns_steps > max_steps) return MUON_ERR_INVALID_ARG;
    } else if (mode != MUON_MODE_ROWNORM) {
        return MUON_ERR_INVALID_ARG;
    }
    muon_status st = check_pointers(p, params, grads, momentum);
    if (st != MUON_OK) return st;
    if ((st = check_device(p)) != MUON_OK) return st;
    if ((st = host_copy_setup(p)) != MUON_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t gsz = p->gdt == MUON_BF16 ? 2 : 4;
    auto& h = p->hc;
    // gradients in, chunk by chunk, after the caller's earlier work (which may still read grads)
    MUON_TRY(cudaEventRecord(h.entry_ev, s));
    MUON_TRY(cudaStreamWaitEvent(h.in, h.entry_ev, 0));
    for (size_t ci = 0; ci < p->chunks.size(); ++ci) {
        for (int bk : p->chunks[ci].buckets)
            for (int i : p->buckets[bk].mats)
                MUON_TRY(cudaMemcpyAsync(const_cast<void*>(grads[i]), grads_host[i],
                                         (size_t)(p->mats[i].m * p->mats[i].n) * gsz, cudaMemcpyDefault, h.in));
        MUON_TRY(cudaEventRecord(h.in_ev[ci], h.in));
    }
    if (mode == MUON_MODE_NS) {
        const HostIO io{params_host};
        st = ns_step(p, params, grads, momentum, lr, wd, mu, ns_steps, nullptr, 0, stream, &io);
        if (st != MUON_OK) return st;
    } else {   // RowNorm, chunk by chunk like the NS step
        if ((st = upload_pointers(p, params, grads, momentum, s)) != MUON_OK) return st;
        int launches = 0;
        for (size_t ci = 0; ci < p->chunks.size(); ++ci) {
            const muon_plan_s::Chunk& ch = p->chunks[ci];
            MUON_TRY(cudaStreamWaitEvent(s, h.in_ev[ci], 0));
            if ((st = rownorm_launch(p, ch.rn_rows, ch.rn_stats, ch.rn_final, ch.rn_apply, lr, wd, mu, 1e-8f, s,
                                     &launches)) != MUON_OK)
                return st;
            if (!params_host) continue;
            MUON_TRY(cudaEventRecord(h.out_ev[ci], s));
            MUON_TRY(cudaStreamWaitEvent(h.out, h.out_ev[ci], 0));
            for (int bk : ch.buckets)
                for (int i : p->buckets[bk].mats)
                    MUON_TRY(cudaMemcpyAsync(params_host[i], params[i],
                                             (size_t)(p->mats[i].m * p->mats[i].n) * sizeof(float),
                                             cudaMemcpyDefault, h.out));
        }
        p->last_launches = launches;
    }
    if (params_host) {   // the caller's stream covers the copies back
        MUON_TRY(cudaEventRecord(h.end_ev, h.out));
        MUON_TRY(cudaStreamWaitEvent(s, h.end_ev, 0));
    }
    return MUON_OK;
}

muon_status muon_plan_tune(muon_plan p, float* const* params, const void* const* grads, float* const* momentum,
                           float lr, float wd, float mu, int32_t reps, float* ms_out, void* stream) {
    if (!p || reps < 1 || reps > 100) return MUON_ERR_INVALID_ARG;
    if (!p->full_rows.empty()) return MUON_ERR_UNSUPPORTED;
    muon_status st = check_pointers(p, params, grads, momentum);
    if (st != MUON_OK) return st;
    // candidates: CTA pairs beside the fused kernel (none, the estimate, half and one and a
    // half times it; only while opts.chain_clusters leaves the choice to the plan) and
    // symmetric r x r results stored as the lower triangle or whole
    bool mixed = false;
    for (const auto& ch : p->chunks) mixed = mixed || (ch.mixed && ch.chain_est > 0);
    const float scales[4] = {1.f, 0.f, 0.5f, 1.5f};
    const int n_scales = mixed && p->opts.chain_clusters == 0 && p->s2 ? 4 : 1;
    bool lower_choice = false;   // chunks where lower-triangle storage is a choice
    for (const auto& ch : p->chunks) lower_choice = lower_choice || ch.lower_ok;
    const bool lowers[2] = {true, false};
    const int n_lowers = lower_choice && !p->opts.full_symmetric ? 2 : 1;
    const int kmax = std::min(p->pair_clusters - 1, (p->sm_count - 2) / 2);
    auto apply = [&](float sc, bool q) {
        for (auto& ch : p->chunks)
            if (ch.mixed && p->opts.chain_clusters == 0)
                ch.chain_clusters = sc == 0.f ? 0 : std::min(std::max((int)std::lround(ch.chain_est * sc), 1), kmax);
        for (auto& ch : p->chunks) ch.lower = ch.lower_ok && !p->opts.full_symmetric && q;
    };
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        g_last_cuda_error = cudaGetLastError();
        if (e0) cudaEventDestroy(e0);
        return MUON_ERR_CUDA;
    }
    float best = 0.f, best_sc = 1.f;
    bool best_q = true;
    int tried = 0;
    for (int si = 0; si < n_scales; ++si) {
        for (int qi = 0; qi < n_lowers; ++qi) {
            const float sc = scales[si];
            const bool q = lowers[qi];
            apply(sc, q);
            st = muon_step_ex(p, params, grads, momentum, lr, wd, mu, kMaxNsSteps, nullptr, 0, stream);   // warm-up
            if (st == MUON_OK && cudaEventRecord(e0, s) != cudaSuccess) st = MUON_ERR_CUDA;
            for (int i = 0; st == MUON_OK && i < reps; ++i)
                st = muon_step_ex(p, params, grads, momentum, lr, wd, mu, kMaxNsSteps, nullptr, 0, stream);
            float ms = 0.f;
            if (st == MUON_OK && (cudaEventRecord(e1, s) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
                                  cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess))
                st = MUON_ERR_CUDA;
            if (st != MUON_OK) break;
            ms /= (float)reps;
            if (tried == 0 || ms < best) {
                best = ms;
                best_sc = sc;
                best_q = q;
            }
            ++tried;
        }
        if (st != MUON_OK) break;
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    apply(best_sc, best_q);
    if (st != MUON_OK) return st;
    p->tuned = tried;
    if (ms_out) *ms_out = best;
    return muon_sync(p, stream);
}

muon_status muon_sync(muon_plan p, void* stream) {
    if (!p) return MUON_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MUON_ERR_CUDA;
    int st = 0;
    MUON_TRY(cudaMemcpy(&st, p->status, sizeof(int), cudaMemcpyDeviceToHost));
    if (st != 0) {
        MUON_TRY(cudaMemset(p->status, 0, sizeof(int)));
        // a timeout replaces the word; non-finite norms are or-ed into it
        return (st & kStatusTimeoutMask) ? MUON_ERR_TIMEOUT : MUON_ERR_NONFINITE;
    }
    return MUON_OK;
}

muon_status muon_debug_wait_timeout(muon_plan p, int32_t limit_us, void* stream) {
    if (!p || limit_us < 1 || limit_us > 1000000) return MUON_ERR_INVALID_ARG;
    if (check_device(p) != MUON_OK) return MUON_ERR_INVALID_ARG;
    return cuda_status(
        launch_wait_selftest(p->status, 1000ull * (unsigned long long)limit_us, static_cast<cudaStream_t>(stream)));
}

muon_status muon_debug_copy_update(muon_plan p, int32_t i, float* dst, void* stream) {
    if (!p || !dst || i < 0 || i >= (int)p->shapes.size()) return MUON_ERR_INVALID_ARG;
    if (!p->opts.keep_update) return MUON_ERR_INVALID_ARG;
    const Bucket& b = p->buckets[p->mat_bucket[i]];
    const size_t numel = (size_t)b.r * b.c;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(dst, b.Odbg + (size_t)p->mat_item[i] * numel, numel * sizeof(float), cudaMemcpyDefault, s) !=
        cudaSuccess)
        return MUON_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

muon_status muon_debug_update_error(muon_plan p, int32_t i, const float* ref, double* rel, void* stream) {
    if (!p || !ref || !rel || i < 0 || i >= (int)p->shapes.size()) return MUON_ERR_INVALID_ARG;
    if (!p->opts.keep_update || !p->full_rows.empty()) return MUON_ERR_INVALID_ARG;
    const Bucket& b = p->buckets[p->mat_bucket[i]];
    const long long numel = (long long)b.r * b.c;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MUON_TRY(launch_sq_diff(b.Odbg + (size_t)p->mat_item[i] * numel, ref, numel, p->diff, s));
    double sums[2] = {0.0, 0.0};
    MUON_TRY(cudaMemcpyAsync(sums, p->diff, sizeof(sums), cudaMemcpyDeviceToHost, s));
    MUON_TRY(cudaStreamSynchronize(s));
    *rel = sums[1] > 0.0 ? std::sqrt(sums[0] / sums[1]) : std::sqrt(sums[0]);
    return MUON_OK;
}

muon_status muon_debug_copy_workspace(muon_plan p, int32_t i, int32_t which, void* dst, int32_t* ld,
                                      void* stream) {
    if (!p || !dst || !ld || i < 0 || i >= (int)p->shapes.size() || which < 0 || which > 8)
        return MUON_ERR_INVALID_ARG;
    const Bucket& b = p->buckets[p->mat_bucket[i]];
    // the fused kernel keeps its r x r operands on chip: only X0 and alpha exist
    if (!b.batched() && which >= 1 && which <= 7) return MUON_ERR_UNSUPPORTED;
    // split buffers hold two parts per matrix (hi at 2 item, lo at 2 item + 1): the hi part is copied
    const int item = p->mat_item[i] * (which >= 1 && which <= 7 && b.split ? 2 : 1);
    const int xitem = p->mat_item[i] * (b.split == 2 ? 2 : 1);
    const size_t rr = (size_t)b.r * b.ldr;
    const void* src = nullptr;
    size_t bytes = 0;
    *ld = b.ldr;
    switch (which) {
        case 0:
            src = p->ut + b.ut_off + (size_t)xitem * b.r * b.ldu;
            bytes = (size_t)b.r * b.ldu * 2;
            *ld = b.ldu;
            break;
        case 1: case 2: src = b.G[which - 1] + item * rr; bytes = rr * 2; break;
        case 3: src = b.P + item * rr; bytes = rr * 2; break;
        case 4: src = b.T + item * rr; bytes = rr * 2; break;
        case 5: case 6: src = b.Q[which - 5] + item * rr; bytes = rr * 2; break;
        case 7: src = b.Qb + item * rr; bytes = rr * 2; break;
        case 8: src = p->alpha + p->mats[i].slot; bytes = 4; *ld = 1; break;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (which >= 1 && which <= 7 && b.r > kBM && p->chunks[b.chunk].lower) {
        // lower-triangle storage (256 x 256 tiles at or below the diagonal): rebuild the upper part
        std::vector<uint16_t> h;
        try {
            h.resize(rr);
        } catch (...) {
            return MUON_ERR_OOM;   // host memory
        }
        if (cudaMemcpyAsync(h.data(), src, bytes, cudaMemcpyDefault, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return MUON_ERR_CUDA;
        for (int row = 0; row < b.r; ++row)
            for (int col = (row / 256 + 1) * 256; col < b.r; ++col)
                h[(size_t)row * b.ldr + col] = h[(size_t)col * b.ldr + row];
        if (cudaMemcpyAsync(dst, h.data(), bytes, cudaMemcpyDefault, s) != cudaSuccess) return MUON_ERR_CUDA;
        return cudaStreamSynchronize(s) == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
    }
    if (cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, s) != cudaSuccess) return MUON_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

muon_status muon_plan_info(muon_plan p, muon_plan_info_t* info) {
    if (!p || !info) return MUON_ERR_INVALID_ARG;
    info->n_matrices = (int32_t)p->shapes.size();
    info->n_buckets = (int32_t)p->buckets.size();
    info->workspace_bytes = (int64_t)p->ws_bytes;
    info->launches_last_step = p->last_launches;
    info->n_chunks = (int32_t)p->chunks.size();
    int lower = 0;
    for (const auto& ch : p->chunks) lower += ch.lower ? 1 : 0;
    info->lower_chunks = lower;
    info->tuned_candidates = p->tuned;
    int chain = 0;
    for (const auto& ch : p->chunks) chain = std::max(chain, ch.chain_clusters);
    info->chain_clusters = chain;
    info->sm_count = p->sm_count;
    int nsplit = 0, nf32 = 0;
    for (const auto& b : p->buckets) {
        nsplit += b.split ? 1 : 0;
        nf32 += b.f32 ? 1 : 0;
    }
    info->split_buckets = nsplit;
    info->fp32_buckets = nf32;
    info->colsq_len = (int64_t)p->colsq_len;
    return MUON_OK;
}

muon_status muon_stage_times(muon_plan p, float* ms, double* flops, int32_t n_stages) {
    if (!p || !ms || n_stages < 0 || n_stages > 6) return MUON_ERR_INVALID_ARG;
    if (p->n_timed == 0) return MUON_ERR_INVALID_ARG;
    double acc[6] = {0, 0, 0, 0, 0, 0};
    // NS steps: momentum e[0] -> e[1]; fused e[1] -> e[6]; SYRK from e[6] (after the
    // fused kernel) or, split, from e[1] (beside it) to e[2]; r x r e[2] -> e[3];
    // final e[3] -> e[4]
    for (size_t g = 0; g < p->n_timed; ++g) {
        const auto& se = p->evs[g];
        float t = 0.f;
        if (se.ns) {
            for (size_t c = 0; c < p->chunks.size(); ++c) {   // stages summed over the chunks
                const cudaEvent_t* e = &se.e[7 * c];
                if (cudaEventSynchronize(e[4]) != cudaSuccess || cudaEventSynchronize(e[6]) != cudaSuccess)
                    return MUON_ERR_CUDA;
                const int from[5] = {0, se.split[c] ? 1 : 6, 2, 3, 1}, to[5] = {1, 2, 3, 4, 6},
                          slot[5] = {0, 1, 2, 3, 5};
                for (int k = 0; k < 5; ++k) {
                    if (cudaEventElapsedTime(&t, e[from[k]], e[to[k]]) != cudaSuccess) return MUON_ERR_CUDA;
                    acc[slot[k]] += t;
                }
            }
        } else {
            if (cudaEventSynchronize(se.e[5]) != cudaSuccess) return MUON_ERR_CUDA;
            if (cudaEventElapsedTime(&t, se.e[0], se.e[5]) != cudaSuccess) return MUON_ERR_CUDA;
            acc[4] += t;
        }
    }
    for (int k = 0; k < n_stages; ++k) ms[k] = (float)acc[k];
    if (flops)
        for (int k = 0; k < 3; ++k) flops[k] = p->flops[k];
    p->n_timed = 0;
    p->flops[0] = p->flops[1] = p->flops[2] = 0;
    return MUON_OK;
}

}  // extern "C"
