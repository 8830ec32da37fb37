// Batched, grouped tensor-core products of the Gram Newton-Schulz iteration on
// sm_103a: TMA-fed shared-memory pipeline, tcgen05.mma (kind::f16) with the
// accumulator in TMEM, warp-specialised persistent CTAs.
//
// Products (DMuon, "Gram Newton-Schulz": the recursion runs on r x r matrices;
// SYRK-style symmetric products compute only the lower triangle):
//   G0' = s alpha^2 X X^T            bf16 x bf16 -> fp32, K = c   (kEpiSyrk, symmetric)
//   P   = aI + (b/s) G' + (c/s^2) G'G'  fp16 x fp16 -> fp32, K = r (kEpiPoly, symmetric)
//   Q'  = P Q,  T = P P,  G'' = G' T    fp16 x fp16 -> fp32, K = r (kEpiPlain, symmetric)
//   O   = alpha Q X                  bf16 x bf16 -> fp32, K = r   (kEpiApply: fused
//                                    W -= lr (0.2 sqrt(c) O + wd W), blog eq. (4))
// G is carried scaled, G' = s G with s = 2^round(log2 r), so every r x r value
// sits in fp16's normal range: sigma_max(X0) <= ||X0||_F = 1 bounds |G'| by
// 1.44 s, |P| by 3.45 and |Q| by 3.45^J.  fp16 keeps 11 significant bits (as
// tf32) at the bf16 tensor rate.  Every r x r product of commuting polynomials
// in G0 is symmetric, so all of them are lower-triangle products.
#include "kernels.h"
#include "ptx.cuh"

namespace muon {

struct GemmCfg {
    static constexpr int BK = 64;                        // one 128-byte swizzle row of K
    static constexpr int ESZ = 2;
    static constexpr int UK = 16;                        // K of one tcgen05.mma kind::f16
    static constexpr int A_BYTES = kBM * BK * ESZ;       // 16 KB
    static constexpr int B_BYTES = kBN * BK * ESZ;       // 32 KB
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int MN_CHUNK_BYTES = 64 * BK * ESZ; // one 64-wide MN-major chunk of B
    static constexpr int BAR_OFFSET = kStages * STAGE_BYTES;
    static constexpr int SMEM_BYTES = BAR_OFFSET + 256 + 1024;   // + barriers + alignment slack
};

size_t gemm_smem_bytes() { return GemmCfg::SMEM_BYTES; }

struct TileCoord {
    int p, item, m0, n0;
};

__device__ __forceinline__ TileCoord decode_tile(const GemmLaunch& L, int t) {
    int p = 0;
    while (p + 1 < L.nprob && t >= L.prob[p + 1].tile_begin) ++p;
    const GemmProblem& P = L.prob[p];
    const int local = t - P.tile_begin;
    const int item = local / P.tiles_per_item;
    const int tl = local - item * P.tiles_per_item;
    int tm, tn;
    if (P.sym) {
        // Row tm of 128 has floor(tm/2)+1 column tiles of 256 touching the lower triangle.
        tm = 0;
        int acc = 0;
        for (;;) {
            const int cnt = (tm >> 1) + 1;
            if (tl < acc + cnt) {
                tn = tl - acc;
                break;
            }
            acc += cnt;
            ++tm;
        }
    } else {
        // M fastest: consecutive CTAs share the same (large) B column tile in L2.
        tm = tl % P.tiles_m;
        tn = tl / P.tiles_m;
    }
    return {p, item, tm * kBM, tn * kBN};
}

// Waits that must finish even after an abort (draining our own async work).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitTimeoutNs) break;
    }
}

// fp16 conversions saturate at +-65504 instead of overflowing to inf.  For
// ns_steps >= 9 the null-space eigenvalue of Q (exactly a^J on a rank-deficient
// input) exceeds fp16's range; saturating keeps it finite, so its product with
// the exactly-zero null-space component of X0 stays 0 rather than NaN.
__device__ __forceinline__ float sat_half(float x) {
    return (x != x) ? x : fminf(fmaxf(x, -65504.f), 65504.f);   // a NaN stays NaN
}
__device__ __forceinline__ __half to_half(float x) { return __float2half_rn(sat_half(x)); }
__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    __half2 h = __floats2half2_rn(sat_half(a), sat_half(b));
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf162(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// ------------------------------------------------------------------ epilogues
// v[j] is element (row, col0 + j) of a symmetric result.  The lower part goes to
// (row, col), its mirror to (col, row).  Rows beyond M are masked (their lanes
// still took part in the collective TMEM load).
__device__ __forceinline__ void store_sym(const GemmProblem& P, int item, int row, int col0, const float (&v)[32]) {
    if (row >= P.M) return;
    const long long ib = item * P.strideC;
    __half* C = P.C ? P.C + ib : nullptr;
    __half* C2 = P.C2 ? P.C2 + ib : nullptr;
    __nv_bfloat16* Cb = P.Cb ? P.Cb + ib : nullptr;
    const long long rbase = (long long)row * P.ldc + col0;
    const bool full = (col0 + 31 <= row) && (col0 + 31 < P.N);
    if (full) {
        if (C || C2) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 h = make_uint4(pack_half2(v[8 * q], v[8 * q + 1]), pack_half2(v[8 * q + 2], v[8 * q + 3]),
                                           pack_half2(v[8 * q + 4], v[8 * q + 5]),
                                           pack_half2(v[8 * q + 6], v[8 * q + 7]));
                if (C) reinterpret_cast<uint4*>(C + rbase)[q] = h;
                if (C2) reinterpret_cast<uint4*>(C2 + rbase)[q] = h;
            }
        }
        if (Cb) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                reinterpret_cast<uint4*>(Cb + rbase)[q] =
                    make_uint4(pack_bf162(v[8 * q], v[8 * q + 1]), pack_bf162(v[8 * q + 2], v[8 * q + 3]),
                               pack_bf162(v[8 * q + 4], v[8 * q + 5]), pack_bf162(v[8 * q + 6], v[8 * q + 7]));
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int col = col0 + j;
            if (col <= row && col < P.N) {
                if (C) C[rbase + j] = to_half(v[j]);
                if (C2) C2[rbase + j] = to_half(v[j]);
                if (Cb) Cb[rbase + j] = __float2bfloat16_rn(v[j]);
            }
        }
    }
    // mirror: for fixed j the warp's lanes write consecutive entries of row `col`
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const int col = col0 + j;
        if (col < row && col < P.N) {
            const long long idx = (long long)col * P.ldc + row;
            if (C) C[idx] = to_half(v[j]);
            if (C2) C2[idx] = to_half(v[j]);
            if (Cb) Cb[idx] = __float2bfloat16_rn(v[j]);
        }
    }
}

// Final product epilogue, in two phases so the 32 W loads of a chunk are all in
// flight at once (and overlap the TMEM load): apply_load, then apply_store.
struct ApplyCtx {
    float* W;
    float* O;
    long long base;     // index of element (row, col0) in the stored layout
    long long stride;   // index step per column: 1 (m <= n) or M (stored transposed)
    bool vec;           // 8 float4 per chunk (m <= n, aligned, no tail)
};

__device__ __forceinline__ ApplyCtx apply_ctx(const GemmProblem& P, int item, int row, int col0) {
    ApplyCtx c;
    const int mat = P.item_mat[item];
    c.W = P.W[mat];
    c.O = P.Odbg ? P.Odbg + (long long)item * P.M * P.N : nullptr;
    if (P.transposed[mat] == 0) {
        // stored layout = oriented layout: element (row, col) at row * N + col
        c.base = (long long)row * P.N + col0;
        c.stride = 1;
        c.vec = (col0 + 31 < P.N) && ((P.N & 3) == 0) && ((reinterpret_cast<uintptr_t>(c.W) & 15) == 0);
    } else {
        // stored as c x r: oriented (row, col) lives at col * M + row, so the
        // warp's lanes (consecutive rows) touch consecutive addresses
        c.base = (long long)col0 * P.M + row;
        c.stride = P.M;
        c.vec = false;
    }
    return c;
}

__device__ __forceinline__ void apply_load(const GemmProblem& P, const ApplyCtx& c, int row, int col0,
                                           float (&w)[32]) {
    if (row >= P.M) return;
    if (c.vec) {
        const float4* w4 = reinterpret_cast<const float4*>(c.W + c.base);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 t = w4[q];
            w[4 * q] = t.x;
            w[4 * q + 1] = t.y;
            w[4 * q + 2] = t.z;
            w[4 * q + 3] = t.w;
        }
    } else {
        const float* base = c.W + c.base;
        const int st = (int)c.stride;   // 1 or M (< 2^20): 32-bit offsets keep few registers live
        const int nj = min(32, P.N - col0);
#pragma unroll
        for (int j = 0; j < 32; ++j) w[j] = (j < nj) ? base[j * st] : 0.f;
    }
}

// Debug copy of O = alpha * acc (plans with keep_update only).  Kept out of line
// so its registers do not weigh on the fused update of every other plan.
__device__ __noinline__ void store_debug_update(const GemmProblem& P, const ApplyCtx& c, int row, int col0, float al,
                                                const uint32_t (&raw)[32]) {
    if (c.vec) {
        float4* o4 = reinterpret_cast<float4*>(c.O + c.base);
        for (int q = 0; q < 8; ++q)
            o4[q] = make_float4(al * __uint_as_float(raw[4 * q]), al * __uint_as_float(raw[4 * q + 1]),
                                al * __uint_as_float(raw[4 * q + 2]), al * __uint_as_float(raw[4 * q + 3]));
    } else {
        float* base = c.O + c.base;
        const int st = (int)c.stride;
        const int nj = min(32, P.N - col0);
        for (int j = 0; j < nj; ++j) base[j * st] = al * __uint_as_float(raw[j]);
    }
}

__device__ __forceinline__ void apply_store(const GemmProblem& P, const ApplyCtx& c, int item, int row, int col0,
                                            const uint32_t (&raw)[32], float (&w)[32]) {
    if (row >= P.M) return;
    const float al = P.alpha[item];
    const float lr = P.lr, wd = P.wd, s = P.scale;
    const int st = (int)c.stride;   // 1 or M (< 2^20): 32-bit offsets keep few registers live
    const int nj = min(32, P.N - col0);
#pragma unroll
    for (int j = 0; j < 32; ++j) w[j] = w[j] - lr * (s * (al * __uint_as_float(raw[j])) + wd * w[j]);
    if (c.vec) {
        float4* w4 = reinterpret_cast<float4*>(c.W + c.base);
#pragma unroll
        for (int q = 0; q < 8; ++q) w4[q] = make_float4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    } else {
        float* base = c.W + c.base;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j < nj) base[j * st] = w[j];
    }
    if (c.O) store_debug_update(P, c, row, col0, al, raw);
}

__device__ __forceinline__ void epilogue_chunk(const GemmProblem& P, int item, int row, int col0,
                                               const uint32_t (&raw)[32]) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw[j]);
    if (P.epi == kEpiSyrk) {
        const float al = P.alpha[item];
        const float k = P.out_scale * al * al;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= k;
    } else if (P.epi == kEpiPoly) {
        // P = a I + b' G' + c' G'^2, with G' read (8 values at a time) from the fp16
        // input the MMA used
        const __half* Grow = P.Gin + item * P.strideC + (long long)(row < P.M ? row : 0) * P.ldc + col0;
        const bool vec = (row < P.M) && (col0 + 31 < P.N);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float g[8];
            if (vec) {
                const uint4 t = reinterpret_cast<const uint4*>(Grow)[q];
                const uint32_t w4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w4[e]));
                    g[2 * e] = f.x;
                    g[2 * e + 1] = f.y;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    g[e] = (row < P.M && col0 + 8 * q + e < P.N) ? __half2float(Grow[8 * q + e]) : 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int j = 8 * q + e;
                v[j] = P.coef_c * v[j] + P.coef_b * g[e] + ((col0 + j == row) ? P.coef_a : 0.f);
            }
        }
    }
    store_sym(P, item, row, col0, v);
}

// ------------------------------------------------------------------ kernel
template <bool BF16>
__global__ void __maxnreg__(200) gemm_kernel(const __grid_constant__ GemmLaunch L) {
    using Cfg = GemmCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::BAR_OFFSET);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull + a, 1);
            mbar_init(tempty + a, kEpiWarps);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int p = 0; p < L.nprob; ++p) {
            tma_prefetch_desc(&L.mapA[p]);
            tma_prefetch_desc(&L.mapB[p]);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 2 * kBN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < L.total_tiles; t += gridDim.x) {
                const TileCoord tc = decode_tile(L, t);
                const GemmProblem& P = L.prob[tc.p];
                const int kblocks = (P.K + Cfg::BK - 1) / Cfg::BK;
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const uint32_t s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!mbar_wait(empty + s, ph ^ 1u, abort_flag, L.status, kStatusTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + s * Cfg::STAGE_BYTES;
                    uint8_t* sb = sa + Cfg::A_BYTES;
                    mbar_arrive_expect_tx(full + s, Cfg::STAGE_BYTES);
                    tma_load_3d(sa, &L.mapA[tc.p], full + s, kb * Cfg::BK, tc.m0, tc.item);
                    if (!P.b_mn) {
                        tma_load_3d(sb, &L.mapB[tc.p], full + s, kb * Cfg::BK, tc.n0, tc.item);
                    } else {
#pragma unroll
                        for (int q = 0; q < kBN / 64; ++q)
                            tma_load_3d(sb + q * Cfg::MN_CHUNK_BYTES, &L.mapB[tc.p], full + s, tc.n0 + 64 * q,
                                        kb * Cfg::BK, tc.item);
                    }
                }
            }
            if (!ok) {
                // let the copies already issued land before the CTA exits
                const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0u;
                for (uint32_t j = first; j < it; ++j) mbar_drain(full + (j % kStages), (j / kStages) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer (one thread)
            uint32_t it = 0;
            int local = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < L.total_tiles; t += gridDim.x, ++local) {
                const TileCoord tc = decode_tile(L, t);
                const GemmProblem& P = L.prob[tc.p];
                const int kblocks = (P.K + Cfg::BK - 1) / Cfg::BK;
                const uint32_t acc = local & 1;
                const uint32_t aph = (local >> 1) & 1u;
                if (!mbar_wait(tempty + acc, aph ^ 1u, abort_flag, L.status, kStatusTimeoutMma)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * kBN;
                const uint32_t idesc = idesc_make(BF16, kBM, kBN, false, P.b_mn != 0);
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const uint32_t s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!mbar_wait(full + s, ph, abort_flag, L.status, kStatusTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + s * Cfg::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + Cfg::A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < Cfg::BK / Cfg::UK; ++kk) {
                        const uint64_t ad = sdesc_sw128(a_addr + kk * Cfg::UK * Cfg::ESZ, 0, 1024);
                        const uint64_t bd =
                            P.b_mn ? sdesc_sw128(b_addr + kk * Cfg::UK * 128, Cfg::MN_CHUNK_BYTES, 1024)
                                   : sdesc_sw128(b_addr + kk * Cfg::UK * Cfg::ESZ, 0, 1024);
                        mma_f16kind(d_tmem, ad, bd, idesc, (kb | kk) != 0);
                    }
                    mma_commit(empty + s);   // frees the stage when these MMAs finish
                }
                if (!ok) break;
                mma_commit(tfull + acc);     // accumulator ready for the epilogue
            }
            // all MMAs issued by this thread complete before TMEM is released
            mma_commit(drain);
            mbar_drain(drain, 0);
        }
    } else {
        // ---------------- epilogue: TMEM lane quarter = warp % 4; warps 2-5 take
        // columns 0-127 of the tile, warps 6-9 columns 128-255
        const int wq = warp & 3;
        const int c_begin = ((warp - 2) >> 2) * (kBN * 4 / kEpiWarps);
        int local = 0;
        for (int t = blockIdx.x; t < L.total_tiles; t += gridDim.x, ++local) {
            const TileCoord tc = decode_tile(L, t);
            const GemmProblem& P = L.prob[tc.p];
            const uint32_t acc = local & 1;
            const uint32_t aph = (local >> 1) & 1u;
            if (!mbar_wait(tfull + acc, aph, abort_flag, L.status, kStatusTimeoutEpilogue)) break;
            tc_fence_after();
            const int row = tc.m0 + wq * 32 + lane;
            const int warp_row_max = tc.m0 + wq * 32 + 31;
            const uint32_t tbase = tmem_base + acc * kBN + (static_cast<uint32_t>(wq * 32) << 16);
            for (int cc = c_begin; cc < c_begin + kBN * 4 / kEpiWarps; cc += 32) {
                const int col0 = tc.n0 + cc;
                if (col0 >= P.N) break;                              // warp-uniform
                if (P.sym && col0 > warp_row_max) break;             // whole chunk above the diagonal
                uint32_t raw[32];
                tmem_ld32(tbase + cc, raw);
                if (P.epi == kEpiApply) {
                    const ApplyCtx ac = apply_ctx(P, tc.item, row < P.M ? row : 0, col0);
                    float w[32];
                    apply_load(P, ac, row, col0, w);   // in flight with the TMEM load
                    tmem_ld_wait();
                    apply_store(P, ac, tc.item, row, col0, raw, w);
                } else {
                    tmem_ld_wait();
                    epilogue_chunk(P, tc.item, row, col0, raw);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty + acc);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 2 * kBN);
    }
}

// ------------------------------------------------------------------ 2-SM kernel
// A cluster of two CTAs on two SMs computes one 256 x 256 tile with
// tcgen05.mma.cta_group::2 (M = 256): each CTA stages its own 128 rows of A
// and one half (128 rows) of B, so each SM moves 32 KB through shared memory
// per k-block of 4.2 MFLOP instead of 48 KB per 4.2 MFLOP on one SM alone.
// The even CTA (leader) issues the MMAs; both CTAs' TMA loads signal the
// leader's `full` barrier; MMA completion is multicast to both CTAs.
struct Gemm2Cfg {
    static constexpr int BK = 64;
    static constexpr int ESZ = 2;
    static constexpr int UK = 16;
    static constexpr int A_BYTES = 128 * BK * ESZ;       // this CTA's 128 rows of A
    static constexpr int B_BYTES = 128 * BK * ESZ;       // this CTA's half of B
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int MN_CHUNK_BYTES = 64 * BK * ESZ;
    static constexpr int BAR_OFFSET = kStages2 * STAGE_BYTES;
    static constexpr int SMEM_BYTES = BAR_OFFSET + 256 + 1024;
};

// Pair tiles: (tm2, tn) of 256 x 256; the CTA of rank `rank` owns rows
// 256 tm2 + 128 rank .. + 127.  Symmetric outputs keep tn <= tm2.
__device__ __forceinline__ TileCoord decode_pair_tile(const GemmLaunch& L, int t, uint32_t rank) {
    int p = 0;
    while (p + 1 < L.nprob && t >= L.prob[p + 1].tile_begin) ++p;
    const GemmProblem& P = L.prob[p];
    const int local = t - P.tile_begin;
    const int item = local / P.tiles_per_item;
    const int tl = local - item * P.tiles_per_item;
    int tm, tn;
    if (P.sym) {
        tm = 0;
        int acc = 0;
        for (;;) {
            if (tl < acc + tm + 1) {
                tn = tl - acc;
                break;
            }
            acc += tm + 1;
            ++tm;
        }
    } else {
        tm = tl % P.tiles_m;
        tn = tl / P.tiles_m;
    }
    return {p, item, tm * 256 + 128 * (int)rank, tn * 256};
}

template <bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(200)
    gemm2_kernel(const __grid_constant__ GemmLaunch L) {
    using Cfg = Gemm2Cfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::BAR_OFFSET);
    uint64_t* empty = full + kStages2;
    uint64_t* tfull = empty + kStages2;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster_id = blockIdx.x >> 1;
    const int nclusters = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages2; ++s) {
            mbar_init(full + s, 1);    // leader: its expect_tx arrival + both CTAs' bytes
            mbar_init(empty + s, 1);   // both: the leader's multicast commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull + a, 1);   // both: the leader's multicast commit
            mbar_init(tempty + a, 2 * kEpiWarps);   // leader: every epilogue warp of both CTAs
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int p = 0; p < L.nprob; ++p) {
            tma_prefetch_desc(&L.mapA[p]);
            tma_prefetch_desc(&L.mapB[p]);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, 2 * kBN);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();   // barriers of both CTAs initialised before any remote signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs)
            uint32_t it = 0;
            bool ok = true;
            for (int t = cluster_id; ok && t < L.total_tiles; t += nclusters) {
                const TileCoord tc = decode_pair_tile(L, t, rank);
                const GemmProblem& P = L.prob[tc.p];
                const int kblocks = (P.K + Cfg::BK - 1) / Cfg::BK;
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const uint32_t s = it % kStages2;
                    const uint32_t ph = (it / kStages2) & 1u;
                    if (!mbar_wait_cluster(empty + s, ph ^ 1u, abort_flag, L.status, kStatusTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + s * Cfg::STAGE_BYTES;
                    uint8_t* sb = sa + Cfg::A_BYTES;
                    const uint32_t fb = mapa_shared(smem_u32(full + s), 0);
                    if (leader) mbar_arrive_expect_tx(full + s, 2 * Cfg::STAGE_BYTES);
                    tma_load_3d_pair(sa, &L.mapA[tc.p], fb, kb * Cfg::BK, tc.m0, tc.item);
                    const int nb = tc.n0 + 128 * (int)rank;
                    if (!P.b_mn) {
                        tma_load_3d_pair(sb, &L.mapB[tc.p], fb, kb * Cfg::BK, nb, tc.item);
                    } else {
                        tma_load_3d_pair(sb, &L.mapB[tc.p], fb, nb, kb * Cfg::BK, tc.item);
                        tma_load_3d_pair(sb + Cfg::MN_CHUNK_BYTES, &L.mapB[tc.p], fb, nb + 64, kb * Cfg::BK,
                                         tc.item);
                    }
                }
            }
            if (!ok) {
                // copies already issued signal the leader; give them time to land
                const unsigned long long t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 2000000ull) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (one thread of the even CTA)
            uint32_t it = 0;
            int local = 0;
            bool ok = true;
            for (int t = cluster_id; ok && t < L.total_tiles; t += nclusters, ++local) {
                const TileCoord tc = decode_pair_tile(L, t, rank);
                const GemmProblem& P = L.prob[tc.p];
                const int kblocks = (P.K + Cfg::BK - 1) / Cfg::BK;
                const uint32_t acc = local & 1;
                const uint32_t aph = (local >> 1) & 1u;
                if (!mbar_wait_cluster(tempty + acc, aph ^ 1u, abort_flag, L.status, kStatusTimeoutMma)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * kBN;
                const uint32_t idesc = idesc_make(BF16, 256, kBN, false, P.b_mn != 0);
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const uint32_t s = it % kStages2;
                    const uint32_t ph = (it / kStages2) & 1u;
                    if (!mbar_wait_cluster(full + s, ph, abort_flag, L.status, kStatusTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + s * Cfg::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + Cfg::A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < Cfg::BK / Cfg::UK; ++kk) {
                        const uint64_t ad = sdesc_sw128(a_addr + kk * Cfg::UK * Cfg::ESZ, 0, 1024);
                        const uint64_t bd =
                            P.b_mn ? sdesc_sw128(b_addr + kk * Cfg::UK * 128, Cfg::MN_CHUNK_BYTES, 1024)
                                   : sdesc_sw128(b_addr + kk * Cfg::UK * Cfg::ESZ, 0, 1024);
                        mma_f16kind_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0);
                    }
                    mma_commit_pair(empty + s, 3);   // frees the stage in both CTAs
                }
                if (!ok) break;
                mma_commit_pair(tfull + acc, 3);     // both CTAs' accumulators ready
            }
            mma_commit_pair(drain, 1);
            mbar_drain(drain, 0);
        }
    } else {
        // ---------------- epilogue of both CTAs, each on its own TMEM: lane quarter =
        // warp % 4; warps 2-5 take columns 0-127 of the tile, warps 6-9 columns 128-255
        const int wq = warp & 3;
        const int c_begin = ((warp - 2) >> 2) * (kBN * 4 / kEpiWarps);
        const uint32_t tempty_leader = mapa_shared(smem_u32(tempty), 0);
        int local = 0;
        for (int t = cluster_id; t < L.total_tiles; t += nclusters, ++local) {
            const TileCoord tc = decode_pair_tile(L, t, rank);
            const GemmProblem& P = L.prob[tc.p];
            const uint32_t acc = local & 1;
            const uint32_t aph = (local >> 1) & 1u;
            if (!mbar_wait_cluster(tfull + acc, aph, abort_flag, L.status, kStatusTimeoutEpilogue)) break;
            tc_fence_after();
            const int row = tc.m0 + wq * 32 + lane;
            const int warp_row_max = tc.m0 + wq * 32 + 31;
            const uint32_t tbase = tmem_base + acc * kBN + (static_cast<uint32_t>(wq * 32) << 16);
            for (int cc = c_begin; cc < c_begin + kBN * 4 / kEpiWarps; cc += 32) {
                const int col0 = tc.n0 + cc;
                if (col0 >= P.N) break;
                if (P.sym && col0 > warp_row_max) break;
                uint32_t raw[32];
                tmem_ld32(tbase + cc, raw);
                if (P.epi == kEpiApply) {
                    const ApplyCtx ac = apply_ctx(P, tc.item, row < P.M ? row : 0, col0);
                    float w[32];
                    apply_load(P, ac, row, col0, w);
                    tmem_ld_wait();
                    apply_store(P, ac, tc.item, row, col0, raw, w);
                } else {
                    tmem_ld_wait();
                    epilogue_chunk(P, tc.item, row, col0, raw);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader)
                    mbar_arrive(tempty + acc);
                else
                    mbar_arrive_remote(tempty_leader + acc * 8);
            }
        }
    }

    tc_fence_before();
    cluster_sync();   // all pair MMAs done and both TMEMs drained
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, 2 * kBN);
    }
}

// ------------------------------------------------------------------ fused kernel for r <= 128
// One CTA runs the whole step of one matrix with r <= 128 (persistent over the
// matrices of the launch): the SYRK streams X once, all 4J-3 r x r products
// run on operands kept in shared memory (128 x 128 fp16, 128-byte swizzled
// K-major, the layout TMA would write) with accumulators in TMEM, and the final
// product streams X again in 128-column MN-major chunks into the fused W
// update.  Rows and columns of the r x r operands beyond r are written as zero,
// so the padded recursion is block-diagonal and leaves rows < r unchanged.
constexpr int kSmallRing = 3;                       // X stream ring (SYRK k-blocks, final chunks)
constexpr int kSmallThreads = 320;                  // warp 0 TMA, warp 1 MMA + TMEM, warps 2-9 epilogue
struct SmallCfg {
    static constexpr int SLOT = 32768;              // 16 KB SYRK k-block or 32 KB 128-column chunk
    static constexpr int MAT = 128 * 128 * 2;       // one 128 x 128 2-byte operand
    static constexpr int GS = kSmallRing * SLOT;    // G' (fp16)
    static constexpr int PS = GS + MAT;             // P (fp16)
    static constexpr int QS = PS + MAT;             // Q (fp16)
    static constexpr int TS = QS + MAT;             // T (fp16); then Q_J (bf16) for the final product
    static constexpr int BAR = TS + MAT;
    static constexpr int SMEM_BYTES = BAR + 256 + 1024;
};

// byte offset of element (row, col) of a 128 x 128 2-byte operand in the
// 128-byte-swizzled K-major layout: two 64-column atoms of 128 rows x 128 B
__device__ __forceinline__ uint32_t op_off(int row, int col) {
    return (uint32_t)((col >> 6) * 16384 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) + ((col & 7) << 1));
}

// 32 values v of row `row`, columns [col0, col0 + 32), of a symmetric result into an
// operand buffer (fp16 or bf16): the lower part (col <= row) is stored directly and
// mirrored to (col, row), so the stored operand is exactly symmetric (a K-major B
// operand is read transposed); zero outside the r x r block.  Each element is
// written by exactly one thread.
template <bool BF16OUT>
__device__ __forceinline__ void op_store32(uint8_t* buf, int row, int col0, int r, float (&x)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = (row < r && col0 + j < r) ? x[j] : 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int c8 = col0 + 8 * q;
        if (c8 + 7 <= row) {
            uint4 pk;
            if (BF16OUT)
                pk = make_uint4(pack_bf162(x[8 * q], x[8 * q + 1]), pack_bf162(x[8 * q + 2], x[8 * q + 3]),
                                pack_bf162(x[8 * q + 4], x[8 * q + 5]), pack_bf162(x[8 * q + 6], x[8 * q + 7]));
            else
                pk = make_uint4(pack_half2(x[8 * q], x[8 * q + 1]), pack_half2(x[8 * q + 2], x[8 * q + 3]),
                                pack_half2(x[8 * q + 4], x[8 * q + 5]), pack_half2(x[8 * q + 6], x[8 * q + 7]));
            *reinterpret_cast<uint4*>(buf + op_off(row, c8)) = pk;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (c8 + e <= row) {
                    if (BF16OUT)
                        *reinterpret_cast<__nv_bfloat16*>(buf + op_off(row, c8 + e)) = __float2bfloat16_rn(x[8 * q + e]);
                    else
                        *reinterpret_cast<__half*>(buf + op_off(row, c8 + e)) = to_half(x[8 * q + e]);
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const int col = col0 + j;
        if (col < row) {
            if (BF16OUT)
                *reinterpret_cast<__nv_bfloat16*>(buf + op_off(col, row)) = __float2bfloat16_rn(x[j]);
            else
                *reinterpret_cast<__half*>(buf + op_off(col, row)) = to_half(x[j]);
        }
    }
}

__device__ __forceinline__ void op_load32_half(const uint8_t* buf, int row, int col0, float (&g)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 t = *reinterpret_cast<const uint4*>(buf + op_off(row, col0 + 8 * q));
        const uint32_t w4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w4[e]));
            g[8 * q + 2 * e] = f.x;
            g[8 * q + 2 * e + 1] = f.y;
        }
    }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Kinds of on-chip steps, in the order the MMA thread and the epilogue walk them.
enum SmallStep : int { kSmSyrk = 0, kSmPoly = 1, kSmPair = 2, kSmGT = 3, kSmIdentity = 4 };

// Epilogue of one on-chip step for this thread's row (TMEM lane = row).
__device__ __forceinline__ void small_step_epilogue(int step, int k, int J, const GemmProblem& P, int item,
                                                    uint8_t* smem, uint32_t tmem_row, int row, int c_begin) {
    const int r = P.M;
    for (int cc = c_begin; cc < c_begin + 64; cc += 32) {
        uint32_t raw[32];
        float v[32];
        if (step == kSmIdentity) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = (cc + j == row) ? 1.f : 0.f;
            op_store32<true>(smem + SmallCfg::TS, row, cc, r, v);
            continue;
        }
        tmem_ld32(tmem_row + cc, raw);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw[j]);
        if (step == kSmSyrk) {
            const float al = P.alpha[item];
            const float sc = P.out_scale * al * al;
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= sc;
            op_store32<false>(smem + SmallCfg::GS, row, cc, r, v);
        } else if (step == kSmPoly) {
            float g[32];
            op_load32_half(smem + SmallCfg::GS, row, cc, g);
#pragma unroll
            for (int j = 0; j < 32; ++j)
                v[j] = P.coef_c * v[j] + P.coef_b * g[j] + ((cc + j == row) ? P.coef_a : 0.f);
            op_store32<false>(smem + SmallCfg::PS, row, cc, r, v);
            if (k == 1 && J > 1) op_store32<false>(smem + SmallCfg::QS, row, cc, r, v);
            if (k == 1 && J == 1) op_store32<true>(smem + SmallCfg::TS, row, cc, r, v);
        } else if (step == kSmPair) {
            // accumulator 0: Q' = P Q (k >= 2); accumulator 1: T = P P (k < J)
            if (k >= 2) {
                if (k < J)
                    op_store32<false>(smem + SmallCfg::QS, row, cc, r, v);
                else
                    op_store32<true>(smem + SmallCfg::TS, row, cc, r, v);
            }
            if (k < J) {
                tmem_ld32(tmem_row + 128 + cc, raw);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw[j]);
                op_store32<false>(smem + SmallCfg::TS, row, cc, r, v);
            }
        } else {   // kSmGT: G'' = G' T
            op_store32<false>(smem + SmallCfg::GS, row, cc, r, v);
        }
    }
}

// L2 prefetch of the W entries the fused update of oriented rows [0, M) x columns
// [n0, n0 + 128) reads, issued by the producer with the X chunk (two or three chunks
// ahead of the epilogue).  Only whole 16-byte-aligned in-bounds row segments.
__device__ __forceinline__ void prefetch_w_chunk(const GemmProblem& P, int item, int n0) {
    const int mat = P.item_mat[item];
    const float* W = P.W[mat];
    if ((reinterpret_cast<uintptr_t>(W) & 15) || (P.M & 3) || (P.N & 3)) return;
    const int c_end = min(n0 + 128, P.N);
    if (P.transposed[mat] == 0) {
        const uint32_t bytes = (uint32_t)(c_end - n0) * 4u;
        for (int r = 0; r < P.M; ++r) prefetch_l2_bulk(W + (long long)r * P.N + n0, bytes);
    } else {
        const uint32_t bytes = (uint32_t)P.M * 4u;
        for (int c = n0; c < c_end; ++c) prefetch_l2_bulk(W + (long long)c * P.M, bytes);
    }
}

__global__ void __launch_bounds__(kSmallThreads, 1) ns_small_kernel(const __grid_constant__ GemmLaunch L) {
    using Cfg = SmallCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::BAR);
    uint64_t* empty = full + kSmallRing;
    uint64_t* mma_done = empty + kSmallRing;
    uint64_t* epi_done = mma_done + 1;
    uint64_t* accf_full = epi_done + 1;
    uint64_t* accf_empty = accf_full + 2;
    uint64_t* drain = accf_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSmallRing; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(mma_done, 1);
        mbar_init(epi_done, 8);
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_full + b, 1);
            mbar_init(accf_empty + b, 8);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int p = 0; p < L.nprob; ++p) {
            tma_prefetch_desc(&L.mapA[p]);
            tma_prefetch_desc(&L.mapB[p]);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer: per matrix, the SYRK k-blocks then the final chunks
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < L.total_tiles; t += gridDim.x) {
                int p = 0;
                while (p + 1 < L.nprob && t >= L.prob[p + 1].tile_begin) ++p;
                const GemmProblem& P = L.prob[p];
                const int item = t - P.tile_begin;
                const int kbs = (P.N + 63) / 64;
                const int nch = (P.N + 127) / 128;
                for (int q = 0; ok && q < kbs + nch; ++q, ++it) {
                    const uint32_t s = it % kSmallRing;
                    const uint32_t ph = (it / kSmallRing) & 1u;
                    if (!mbar_wait(empty + s, ph ^ 1u, abort_flag, L.status, kStatusTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    uint8_t* slot = smem + s * Cfg::SLOT;
                    if (q < kbs) {
                        mbar_arrive_expect_tx(full + s, 16384);
                        tma_load_3d(slot, &L.mapA[p], full + s, q * 64, 0, item);
                    } else {
                        const int n0 = (q - kbs) * 128;
                        prefetch_w_chunk(P, item, n0);
                        mbar_arrive_expect_tx(full + s, 32768);
#pragma unroll
                        for (int j = 0; j < 2; ++j)
#pragma unroll
                            for (int h = 0; h < 2; ++h)
                                tma_load_3d(slot + j * 16384 + h * 8192, &L.mapB[p], full + s, n0 + 64 * j, 64 * h,
                                            item);
                    }
                }
            }
            if (!ok) {
                const uint32_t first = it > (uint32_t)kSmallRing ? it - kSmallRing : 0u;
                for (uint32_t j = first; j < it; ++j) mbar_drain(full + (j % kSmallRing), (j / kSmallRing) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            uint32_t it = 0, sc = 0, fc = 0;
            bool ok = true;
            const uint32_t gs = smem_u32(smem + Cfg::GS), ps = smem_u32(smem + Cfg::PS);
            const uint32_t qs = smem_u32(smem + Cfg::QS), ts = smem_u32(smem + Cfg::TS);
            const uint32_t id_h = idesc_make(false, 128, 128, false, false);   // fp16 operands
            const uint32_t id_b = idesc_make(true, 128, 128, false, false);    // bf16 SYRK
            const uint32_t id_f = idesc_make(true, 128, 128, false, true);     // bf16 final, B MN-major
            auto rr = [&](uint32_t a, uint32_t b, uint32_t d) {   // 128 x 128 x 128 from smem operands
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_f16kind(d, sdesc_sw128(a + off, 0, 1024), sdesc_sw128(b + off, 0, 1024), id_h, kk != 0);
                }
            };
            auto finish_step = [&]() -> bool {   // commit, then wait for the epilogue of this step
                mma_commit(mma_done);
                const bool w = mbar_wait(epi_done, sc & 1u, abort_flag, L.status, kStatusTimeoutMma);
                ++sc;
                tc_fence_after();
                return w;
            };
            for (int t = blockIdx.x; ok && t < L.total_tiles; t += gridDim.x) {
                int p = 0;
                while (p + 1 < L.nprob && t >= L.prob[p + 1].tile_begin) ++p;
                const GemmProblem& P = L.prob[p];
                const int J = P.ns_steps;
                const int kbs = (P.N + 63) / 64;
                const int nch = (P.N + 127) / 128;
                // G0 = X X^T (A and B are the same staged tile)
                for (int kb = 0; ok && kb < kbs; ++kb, ++it) {
                    const uint32_t s = it % kSmallRing;
                    if (!mbar_wait(full + s, (it / kSmallRing) & 1u, abort_flag, L.status, kStatusTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = smem_u32(smem + s * Cfg::SLOT);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t d = sdesc_sw128(a + kk * 32, 0, 1024);
                        mma_f16kind(tmem_base, d, d, id_b, (kb | kk) != 0);
                    }
                    mma_commit(empty + s);
                }
                if (!ok || !finish_step()) break;
                for (int k = 1; ok && k <= J; ++k) {
                    rr(gs, gs, tmem_base);                                    // G'^2
                    if (!finish_step()) { ok = false; break; }
                    if (k >= 2 || k < J) {
                        if (k >= 2) rr(ps, qs, tmem_base);                    // P Q
                        if (k < J) rr(ps, ps, tmem_base + 128);               // P P
                        if (!finish_step()) { ok = false; break; }
                    }
                    if (k < J) {
                        rr(gs, ts, tmem_base);                                // G' T
                        if (!finish_step()) { ok = false; break; }
                    }
                }
                if (!ok) break;
                if (J == 0 && !finish_step()) break;                          // Q = I written by the epilogue
                // O = Q X, 128 columns at a time, into alternating accumulators
                for (int ch = 0; ch < nch; ++ch, ++it, ++fc) {
                    const uint32_t b = fc & 1u;
                    if (!mbar_wait(accf_empty + b, ((fc >> 1) & 1u) ^ 1u, abort_flag, L.status, kStatusTimeoutMma) ||
                        !mbar_wait(full + (it % kSmallRing), (it / kSmallRing) & 1u, abort_flag, L.status,
                                   kStatusTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t bs = smem_u32(smem + (it % kSmallRing) * Cfg::SLOT);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = sdesc_sw128(ts + (kk >> 2) * 16384 + (kk & 3) * 32, 0, 1024);
                        const uint64_t bd = sdesc_sw128(bs + kk * 2048, 16384, 1024);
                        mma_f16kind(tmem_base + 256 + 128 * b, ad, bd, id_f, kk != 0);
                    }
                    mma_commit(empty + (it % kSmallRing));
                    mma_commit(accf_full + b);
                }
            }
            mma_commit(drain);
            mbar_drain(drain, 0);
        }
    } else {
        // ---------------- epilogue warps 2..9: row = TMEM lane (warp % 4 picks the lane
        // quarter); warps 2-5 take columns 0-63 of each 128-column block, warps 6-9 64-127
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const int c_begin = ((warp - 2) >> 2) * 64;
        const uint32_t tmem_row = tmem_base + (static_cast<uint32_t>(wq * 32) << 16);
        uint32_t sc = 0, fc = 0;
        bool ok = true;
        auto step = [&](int kind, int k, int J, const GemmProblem& P, int item) -> bool {
            if (!mbar_wait(mma_done, sc & 1u, abort_flag, L.status, kStatusTimeoutEpilogue)) return false;
            ++sc;
            tc_fence_after();
            small_step_epilogue(kind, k, J, P, item, smem, tmem_row, row, c_begin);
            fence_proxy_async_smem();   // operand writes visible to the tensor core
            // and to the other epilogue warps (the next step reads mirrored rows)
            asm volatile("bar.sync 1, 256;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(epi_done);
            return true;
        };
        for (int t = blockIdx.x; ok && t < L.total_tiles; t += gridDim.x) {
            int p = 0;
            while (p + 1 < L.nprob && t >= L.prob[p + 1].tile_begin) ++p;
            const GemmProblem& P = L.prob[p];
            const int item = t - P.tile_begin;
            const int J = P.ns_steps;
            const int nch = (P.N + 127) / 128;
            ok = step(kSmSyrk, 0, J, P, item);
            for (int k = 1; ok && k <= J; ++k) {
                ok = step(kSmPoly, k, J, P, item);
                if (ok && (k >= 2 || k < J)) ok = step(kSmPair, k, J, P, item);
                if (ok && k < J) ok = step(kSmGT, k, J, P, item);
            }
            if (ok && J == 0) ok = step(kSmIdentity, 0, J, P, item);
            for (int ch = 0; ok && ch < nch; ++ch, ++fc) {
                const uint32_t b = fc & 1u;
                // this warp's two 32-column pieces of the chunk; the first piece's W loads go
                // out before the wait for the accumulator
                const int col_a = ch * 128 + c_begin, col_b = col_a + 32;
                float w[32];
                ApplyCtx ac = apply_ctx(P, item, row < P.M ? row : 0, col_a < P.N ? col_a : 0);
                if (col_a < P.N) apply_load(P, ac, row, col_a, w);
                if (!mbar_wait(accf_full + b, (fc >> 1) & 1u, abort_flag, L.status, kStatusTimeoutEpilogue)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tacc = tmem_row + 256 + 128 * b + c_begin;
                if (col_a < P.N) {
                    uint32_t raw[32];
                    tmem_ld32(tacc, raw);
                    tmem_ld_wait();
                    apply_store(P, ac, item, row, col_a, raw, w);
                }
                if (col_b < P.N) {
                    ac = apply_ctx(P, item, row < P.M ? row : 0, col_b);
                    uint32_t raw[32];
                    tmem_ld32(tacc + 32, raw);
                    apply_load(P, ac, row, col_b, w);
                    tmem_ld_wait();
                    apply_store(P, ac, item, row, col_b, raw, w);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(accf_empty + b);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

cudaError_t gemm_prepare(int device) {
    (void)device;
    cudaError_t e =
        cudaFuncSetAttribute(gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, GemmCfg::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 GemmCfg::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm2_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Gemm2Cfg::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm2_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Gemm2Cfg::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(ns_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SmallCfg::SMEM_BYTES);
    return e;
}

cudaError_t ns_small_launch(const GemmLaunch& L, int grid, cudaStream_t s) {
    if (L.total_tiles <= 0) return cudaSuccess;
    if (grid > L.total_tiles) grid = L.total_tiles;
    ns_small_kernel<<<grid, kSmallThreads, SmallCfg::SMEM_BYTES, s>>>(L);
    return cudaGetLastError();
}

cudaError_t gemm2_max_clusters(int* out) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = Gemm2Cfg::SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, gemm2_kernel<true>, &cfg);
}

cudaError_t gemm2_launch(const GemmLaunch& L, bool bf16, int clusters, cudaStream_t s) {
    if (L.total_tiles <= 0) return cudaSuccess;
    if (clusters > L.total_tiles) clusters = L.total_tiles;
    if (clusters < 1) clusters = 1;
    if (bf16)
        gemm2_kernel<true><<<2 * clusters, kGemmThreads, Gemm2Cfg::SMEM_BYTES, s>>>(L);
    else
        gemm2_kernel<false><<<2 * clusters, kGemmThreads, Gemm2Cfg::SMEM_BYTES, s>>>(L);
    return cudaGetLastError();
}

cudaError_t gemm_launch(const GemmLaunch& L, bool bf16, int grid, cudaStream_t s) {
    if (L.total_tiles <= 0) return cudaSuccess;
    if (grid > L.total_tiles) grid = L.total_tiles;
    if (bf16)
        gemm_kernel<true><<<grid, kGemmThreads, GemmCfg::SMEM_BYTES, s>>>(L);
    else
        gemm_kernel<false><<<grid, kGemmThreads, GemmCfg::SMEM_BYTES, s>>>(L);
    return cudaGetLastError();
}

}  // namespace muon
