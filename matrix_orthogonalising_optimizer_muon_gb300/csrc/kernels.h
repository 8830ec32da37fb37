// Kernel parameter blocks and launch entry points shared by the host planner
// (plan.cu, step.cu, capi.cu) and the kernel translation units (gemm.cu, ns_small.cu,
// ns_f32.cu, elementwise.cu, noalloc.cu).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace muon {

// Codes of the plan's device status word (read and cleared by muon_sync).
enum DeviceStatus : int {
    kStatusOk = 0,
    kStatusTimeoutProducer = 0x101,
    kStatusTimeoutMma = 0x102,
    kStatusTimeoutEpilogue = 0x103,
    kStatusTimeoutSelftest = 0x1ff,   // muon_debug_wait_timeout
    kStatusTimeoutMask = 0xfff,       // timeouts replace the word (atomicExch)
    kStatusNonFinite = 0x10000,       // a non-finite input norm (atomicOr; opts.check_finite)
};

// ------------------------------------------------------------------ GEMM
// Tile of one tensor-core product: BM x BN output, one tcgen05.mma M=128 N=256.
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kStages = 4;      // 1-SM kernel: 48 KB per stage
#ifndef MUON_PAIR_STAGES
#define MUON_PAIR_STAGES 5
#endif
constexpr int kStages2 = MUON_PAIR_STAGES;   // 2-SM kernel: 32 KB per stage per CTA
constexpr int kMaxProblems = 8;
#ifndef MUON_EPI_WARPS
#define MUON_EPI_WARPS 8
#endif
// 4: one warp per TMEM lane quarter; 8: two, each on half of the 256 columns
constexpr int kEpiWarps = MUON_EPI_WARPS;
constexpr int kGemmThreads = 32 * (2 + kEpiWarps);   // warp 0 TMA, warp 1 MMA + TMEM, warps 2.. epilogue

enum Epilogue : int {
    kEpiSyrk = 0,    // C = s alpha^2 acc                          (G0' = s X0 X0^T)
    kEpiPoly = 1,    // C = a I + b' Gin + c' acc                  (P = aI + bG + cG^2 in scaled G')
    kEpiPlain = 2,   // C = acc                                    (P Q, P P, G' T)
    kEpiApply = 3,   // W -= lr (s_w alpha acc + wd W), stored layout (final O = Q X0)
    kEpiXout = 4,    // Cb = alpha acc, bf16 r x c (X' = Q X between restarted NS segments)
};

// One batched product C_item = A_item * B_item^T (A: M x K, B: N x K as loaded
// by TMA; B may be MN-major, i.e. stored K x N).  Operands are 2-byte: bf16 for
// the SYRK and the final product, fp16 for the r x r recursion.  With sym = 1
// the output is symmetric (M = N): only tiles touching the lower triangle are
// computed and each lower element is also written to its mirror position.
// Launch with programmatic stream serialisation (see pdl_trigger / pdl_wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// As launch_pdl, with clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                      unsigned cluster_x, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

struct GemmProblem {
    int M, N, K, batch;
    int tiles_m, tiles_n, tiles_per_item, tile_begin;
    int sym, b_mn, epi, ns_steps;   // ns_steps: Newton-Schulz iterations (fused r <= 128 kernel)
    // fp16 outputs (row-major, leading dim ldc, batch stride strideC); C2 an optional copy
    __half* C;
    __half* C2;
    long long strideC;
    int ldc, pad1;
    // optional bf16 copy of the output (same leading dim and stride)
    __nv_bfloat16* Cb;
    // kEpiPoly: G' input of the polynomial (same leading dim and stride)
    const __half* Gin;
    // per-item 1/||U||_F (kEpiSyrk uses its square, kEpiApply the value)
    const float* alpha;
    float coef_a, coef_b, coef_c, out_scale;
    // kEpiApply
    const int* item_mat;               // item -> plan matrix index
    float* const* W;                   // plan matrix index -> params pointer
    const unsigned char* transposed;   // plan matrix index -> stored as c x r
    float* Odbg;                       // optional O (fp32, stored layout), item stride M*N
    float lr, wd, scale, pad3;
    // symmetric outputs of the CTA-pair kernel written with TMA stores from shared
    // memory: kTmaOutC (staged values via mapC), kTmaOutC2 (also via mapC2),
    // kTmaOutBf16 (staged as bf16, else fp16); 0: per-thread stores
    int tma_out;
    // CTA-pair kernel with lower-triangle storage (launches of chunks whose batched
    // matrices have r and c multiples of 64): symmetric r x r results are stored as
    // their 256 x 256 pair tiles at or below the diagonal, the diagonal tiles whole and
    // exactly symmetric.  lower_out: this output is stored so (no mirror below the
    // diagonal tile).  sym_a / sym_b: that operand is stored so; its 64-deep k-blocks
    // beyond the operand rows' diagonal tile are read from the mirror position.
    int lower_out, sym_a, sym_b;
    // Split precision (launches of plans that carry an operand as two 2-byte parts,
    // value = hi + lo): a split buffer holds 2 x batch items, hi of item i at 2i and lo
    // at 2i + 1.  a_split / b_split: that operand is split, and the product runs as
    // K-concatenated passes over the parts, (hi, hi), (hi, lo), (lo, hi) when both are
    // split, (hi), (lo) of the split one otherwise, all into one fp32 accumulator.
    // out_split: the output (C, C2, Cb) is written as hi = round(v), lo = round(v - hi).
    // kEpiPoly reads its G' input split when a_split is set.  Per-thread stores only.
    int a_split, b_split, out_split;
    // kEpiPoly on the CTA-pair kernel with TMA-stored output: the G' input is read by TMA
    // (mapG, 32 x 32 boxes) into the epilogue warp's shared memory, one chunk ahead
    int gin_tma;
    int pad4;
    // kEpiApply on the CTA-pair kernel: per plan matrix, a tensor map of W (fp32, stored
    // layout, 32 x 32 boxes with 128-byte swizzle: the layout of a staged W piece).  The host
    // launches the TMA W path only when every matrix of the launch has a valid map (W 16-byte
    // aligned, stored row length a multiple of 4); wmap_ok holds the validity per matrix.
    const CUtensorMap* wmap;
    const unsigned char* wmap_ok;
};
constexpr int kTmaOutC = 1, kTmaOutC2 = 2, kTmaOutBf16 = 4;

// K-concatenated passes of a (possibly split) product and the parts each reads.
__host__ __device__ __forceinline__ int split_passes(const GemmProblem& P) {
    return (P.a_split && P.b_split) ? 3 : ((P.a_split || P.b_split) ? 2 : 1);
}
// For k-block kbt of the concatenated product (nkb k-blocks per pass): the k-block
// within the pass and the batch coordinates of A and B (item, or 2 item + part).
__host__ __device__ __forceinline__ void split_coords(const GemmProblem& P, int kbt, int nkb, int item, int* kb,
                                                      int* za, int* zb) {
    const int pass = kbt / nkb;
    *kb = kbt - pass * nkb;
    const bool both = P.a_split && P.b_split;
    const int a_lo = P.a_split ? (both ? pass == 2 : pass == 1) : 0;
    const int b_lo = P.b_split ? (pass == 1) : 0;
    *za = P.a_split ? 2 * item + a_lo : item;
    *zb = P.b_split ? 2 * item + b_lo : item;
}

struct GemmLaunch {
    CUtensorMap mapA[kMaxProblems];
    CUtensorMap mapB[kMaxProblems];
    CUtensorMap mapC[kMaxProblems];    // 32 x 32 store boxes (64-byte swizzle) of the outputs
    CUtensorMap mapC2[kMaxProblems];
    // Lower-triangle launches view every operand as (64 columns, rows, column chunks,
    // batch): mapA / mapB then hold K-major boxes (64, 128, 1, 1) at (0, row, k / 64, item)
    // and mapAt / mapBt mirror boxes (64, 64, 2, 1) at (0, k, row / 64, item), MN-major in
    // shared memory (mapBt also serves an MN-major B such as X0 in the final product).
    CUtensorMap mapAt[kMaxProblems];
    CUtensorMap mapBt[kMaxProblems];
    CUtensorMap mapG[kMaxProblems];    // kEpiPoly with gin_tma: its G' input, 32 x 32 boxes (64-byte swizzle)
    GemmProblem prob[kMaxProblems];
    int nprob;
    int total_tiles;
    int* status;
    int pad;
};
static_assert(sizeof(GemmLaunch) <= 32764, "a GemmLaunch must fit the kernel parameter space");

size_t gemm_smem_bytes();
cudaError_t gemm_prepare(int device);   // sets the dynamic shared-memory limit once
// bf16 = true: bf16 operands (SYRK, final product); false: fp16 operands (r x r products)
cudaError_t gemm_launch(const GemmLaunch& L, bool bf16, int grid, cudaStream_t s);
// CTA-pair kernel (cluster of 2, tcgen05 cta_group::2, 256 x 256 tiles); problems
// use pair tiling: tiles_m = ceil(M / 256), tiles_n = ceil(N / 256).
// lower: the lower-triangle variant (4-D operand maps, lower_out / sym_a / sym_b honoured).
cudaError_t gemm2_max_clusters(int* out);
// wtma: a launch of final products whose every matrix has a valid W map (GemmProblem::wmap).
cudaError_t gemm2_launch(const GemmLaunch& L, bool bf16, int clusters, cudaStream_t s, bool lower, bool wtma);
// Whole NS step (SYRK, r x r recursion, final product + fused update) of matrices
// with r <= 128, one matrix per CTA at a time.  One problem per bucket: M = r,
// N = c, batch = matrices, tile_begin = prefix over matrices; mapA = X with
// 64 x 128 boxes, mapB = X with 64 x 64 boxes (MN-major); epilogue fields as
// kEpiApply plus out_scale = s, coef_a/b/c = a, b/s, c/s^2 and ns_steps.
constexpr int kSmallMaxR = 128;
cudaError_t ns_small_prepare();   // sets the fused kernel's dynamic shared-memory limit
cudaError_t ns_small_launch(const GemmLaunch& L, int grid, cudaStream_t s);

// ------------------------------------------------------------------ elementwise
// Per plan matrix, resident on the device.
struct MatDev {
    long long m, n;          // stored shape
    int r, c;                // oriented: r = min, c = max
    int transposed;          // m > n
    int slot;                // bucket-item slot (alpha table)
    long long ut_off;        // element offset of X0 (bf16, r x ldu) in the X0 workspace
    int ldu;                 // leading dim of X0 rows (multiple of 8)
    int nblk;                // momentum blocks of this matrix (= its partial sums)
    long long part_off;      // offset of its momentum partial sums
    long long cpart_off;     // offset of its RowNorm column partial sums (m > n)
    long long inv_off;       // offset of its RowNorm per-column inverse norms (m > n)
    float scale;             // 0.2 * sqrt(c)
    int x_split;             // X0 kept as bf16 hi and lo parts (lo at ut_off + r * ldu)
};

struct ElemArgs {
    const MatDev* mats;
    const int* list;           // plan matrix indices covered by this launch
    int nlist;
    int pad;
    const long long* list_blk; // prefix block offsets, nlist + 1 entries
    const void* const* G;      // per plan matrix
    float* const* M;
    float* const* W;
    __nv_bfloat16* ut;         // X0 workspace
    float* partials;           // block partial sums
    float* alpha;              // per slot
    float* rowinv;             // per-row inverse norms (RowNorm, transposed matrices)
    float mu, lr, wd, eps;
    int grad_bf16;
    int check_finite;          // record a non-finite norm in *status (kStatusNonFinite)
    int* status;
};

// Momentum + Nesterov + partial sum of squares + bf16 X0 in the oriented layout.
cudaError_t launch_momentum_rows(const ElemArgs& a, long long blocks, cudaStream_t s);   // m <= n
cudaError_t launch_momentum_tiles(const ElemArgs& a, long long blocks, cudaStream_t s);  // m > n (transpose)
// alpha[slot] = 1 / sqrt(sum of partials) (0 for a zero input); one warp per matrix.
cudaError_t launch_norm_finalize(const ElemArgs& a, cudaStream_t s);
// Fill a batch of r x r bf16 identities (ns_steps = 0).
// split: q holds 2 x batch items (hi, lo per matrix); the lo parts are filled with zeros.
cudaError_t launch_identity_bf16(__nv_bfloat16* q, int r, int ld, int batch, bool split, cudaStream_t s);
// RowNorm: rows of the stored matrix (m <= n), one block per row, fused apply; rows of
// up to 1024 vec elements in registers (vec 2, 4 or 8), longer ones in two passes.
constexpr int kRowClasses = 3;   // launch classes by row length: <= 2048, <= 4096, longer
inline int rownorm_row_class(long long n) { return n <= 2048 ? 0 : (n <= 4096 ? 1 : 2); }
inline int rownorm_class_vec(int cls) { return 2 << cls; }
cudaError_t launch_rownorm_rows(const ElemArgs& a, long long blocks, int vec, cudaStream_t s);
// RowNorm, m > n: column statistics, finalize, apply.
cudaError_t launch_rownorm_colstats(const ElemArgs& a, long long blocks, cudaStream_t s);
cudaError_t launch_rownorm_colfinal(const ElemArgs& a, long long blocks, cudaStream_t s);
// Dim-0 shards: column sums of U^2 of this shard into out (per matrix at inv_off, padded
// to 4 with zeros; blocks as colfinal over ceil(round_up(n, 4) / threads)), and inverse
// norms from the sums over all shards.
cudaError_t launch_rownorm_colsum(const ElemArgs& a, long long blocks, float* out, cudaStream_t s);
cudaError_t launch_rownorm_colinv(const ElemArgs& a, long long blocks, const float* colsq, cudaStream_t s);
cudaError_t launch_rownorm_colapply(const ElemArgs& a, long long blocks, cudaStream_t s);

// Block geometry the planner needs to size grids and partial-sum buffers.
constexpr int kElemThreads = 256;
constexpr int kMomVecPerThread = 4;                                  // 8-element vectors per thread
constexpr long long kMomElemsPerBlock = 8LL * kElemThreads * kMomVecPerThread;   // rows kernel
#ifndef MUON_TILE_COLS
#define MUON_TILE_COLS 64
#endif
constexpr int kTile = MUON_TILE_COLS;                                // transpose tile: stored columns ...
constexpr int kTileTpr = kTile / 4;                                  // threads per stored row (float4 each)
constexpr int kTileRpp = kElemThreads / kTileTpr;                    // stored rows per pass of the block
#ifndef MUON_TILE_ROWS
#define MUON_TILE_ROWS 128
#endif
constexpr int kTileRows = MUON_TILE_ROWS;                            // ... x kTileRows stored rows
static_assert(kTileRows % 32 == 0 && kTileRows <= 128, "transpose tile rows");
static_assert(kTile % 32 == 0 && kTile <= 128 && kTileRows % kTileRpp == 0 && kTile * (kTileRows + 1) * 4 <= 40000,
              "transpose tile columns");
constexpr int kColSlab = 64;                                         // RowNorm column-stat rows per block
constexpr int kColWidth = 4 * kElemThreads;                          // columns per column-stat block
constexpr long long kApplyElemsPerBlock = 4LL * kElemThreads * 4;    // RowNorm col apply

// ------------------------------------------------------------------ fp32 step of small near-square matrices
// Whole NS step (SYRK, r x r recursion, final product + update) in fp32 on CUDA
// cores, one matrix per CTA, for matrices with r <= kF32MaxR.  U is recomputed
// from the new momentum and the gradient (mu M + G), so the X0 workspace is not read.
constexpr int kF32MaxR = 128;
struct F32Problem {
    int r, c, batch, item_begin;   // oriented shape, matrices, first launch item
    int ns_steps, pad;
    const int* item_mat;           // item -> plan matrix index
    const float* alpha;            // per item 1/||U||_F
    float* Odbg;                   // optional O (fp32, stored layout), item stride r*c
    float coef_a, coef_b, coef_c, scale;
};
struct F32Launch {
    F32Problem prob[kMaxProblems];
    int nprob, total;
    const MatDev* mats;
    const void* const* G;
    float* const* M;
    float* const* W;
    float mu, lr, wd;
    int grad_bf16;
};
cudaError_t ns_f32_prepare();   // sets the kernel's dynamic shared-memory limit
cudaError_t ns_f32_launch(const F32Launch& L, int grid, cudaStream_t s);

// Sums of (a - b)^2 and b^2 over n floats (fp64, fixed order) into scratch[0], scratch[1];
// scratch holds 2 + 2 kDiffParts doubles of device memory.
constexpr int kDiffParts = 256;
cudaError_t launch_sq_diff(const float* a, const float* b, long long n, double* scratch, cudaStream_t s);

// Remembers a CUDA error for muon_last_error_detail (this host thread's last one).
void record_cuda_error(cudaError_t e);

// bounded-wait self test: one mbarrier wait that nothing completes (limit in ns)
cudaError_t launch_wait_selftest(int* status, unsigned long long limit_ns, cudaStream_t s);

}  // namespace muon
