// Device helpers shared by the tensor-core kernels: bounded drain waits,
// saturating fp16 packing, and the epilogues that write symmetric fp16/bf16
// results or apply the fused weight update.
#pragma once
#include "kernels.h"
#include "ptx.cuh"

namespace muon {

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
    if (c.O) {   // debug copy of O = alpha acc (plans that keep the update)
        float* o = c.O + c.base;
        if (c.vec) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
                reinterpret_cast<float4*>(o)[q] =
                    make_float4(al * __uint_as_float(raw[4 * q]), al * __uint_as_float(raw[4 * q + 1]),
                                al * __uint_as_float(raw[4 * q + 2]), al * __uint_as_float(raw[4 * q + 3]));
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < nj) o[j * st] = al * __uint_as_float(raw[j]);
        }
    }
}

// L2 prefetch of what the epilogue of this warp will read for its part of a tile:
// rows [row0, row0 + 32) x columns [col0, col0 + ncols) of W (kEpiApply, stored
// layout) or of G' (kEpiPoly).  Issued while the tile's main loop runs, so the
// epilogue's loads hit L2.  Only whole, 16-byte-aligned in-bounds segments.
__device__ __forceinline__ void prefetch_epilogue_inputs(const GemmProblem& P, int item, int row0, int col0,
                                                         int ncols, int lane) {
    if (col0 >= P.N || row0 >= P.M) return;
    const int nc = min(ncols, P.N - col0);
    if (P.epi == kEpiApply) {
        const int mat = P.item_mat[item];
        const float* W = P.W[mat];
        if (reinterpret_cast<uintptr_t>(W) & 15) return;
        if (P.transposed[mat] == 0) {
            // one oriented row per lane: nc contiguous floats
            const int row = row0 + lane;
            if ((P.N & 3) || row >= P.M) return;
            const uint32_t bytes = (uint32_t)(nc & ~3) * 4u;
            if (bytes) prefetch_l2_bulk(W + (long long)row * P.N + col0, bytes);
        } else {
            // stored c x r: each oriented column is a contiguous run of rows
            const int nr = min(32, P.M - row0);
            if ((P.M & 3) || (row0 & 3)) return;
            const uint32_t bytes = (uint32_t)(nr & ~3) * 4u;
            if (bytes == 0) return;
            for (int c = lane; c < nc; c += 32) prefetch_l2_bulk(W + (long long)(col0 + c) * P.M + row0, bytes);
        }
    } else if (P.epi == kEpiPoly) {
        const int row = row0 + lane;
        if (row >= P.M || (P.ldc & 7)) return;
        const uint32_t bytes = (uint32_t)(nc & ~7) * 2u;
        if (bytes) prefetch_l2_bulk(P.Gin + item * P.strideC + (long long)row * P.ldc + col0, bytes);
    }
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

}  // namespace muon
