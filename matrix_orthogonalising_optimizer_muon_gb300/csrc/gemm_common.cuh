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
// Writes the chunk to the outputs C, C2 (fp16) and Cb (bf16) given (any may be null),
// at batch item `item`, with the problem's shape and strides.
__device__ __forceinline__ void store_sym_to(const GemmProblem& P, __half* C0, __half* C20, __nv_bfloat16* Cb0,
                                             int item, int row, int col0, const float (&v)[32]);

// out_split: hi = round(v) to item 2i, lo = round(v - hi) to item 2i + 1 (fp16 for C
// and C2, bf16 for Cb, each rounded in its own format).
__device__ __forceinline__ void store_sym(const GemmProblem& P, int item, int row, int col0, const float (&v)[32]) {
    if (!P.out_split) {
        store_sym_to(P, P.C, P.C2, P.Cb, item, row, col0, v);
        return;
    }
    if (row >= P.M) return;
    float hi[32], lo[32];
    if (P.C || P.C2) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            hi[j] = __half2float(to_half(v[j]));
            lo[j] = v[j] - hi[j];
        }
        store_sym_to(P, P.C, P.C2, nullptr, 2 * item, row, col0, hi);
        store_sym_to(P, P.C, P.C2, nullptr, 2 * item + 1, row, col0, lo);
    }
    if (P.Cb) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            hi[j] = __bfloat162float(__float2bfloat16_rn(v[j]));
            lo[j] = v[j] - hi[j];
        }
        store_sym_to(P, nullptr, nullptr, P.Cb, 2 * item, row, col0, hi);
        store_sym_to(P, nullptr, nullptr, P.Cb, 2 * item + 1, row, col0, lo);
    }
}

__device__ __forceinline__ void store_sym_to(const GemmProblem& P, __half* C0, __half* C20, __nv_bfloat16* Cb0,
                                             int item, int row, int col0, const float (&v)[32]) {
    if (row >= P.M) return;
    const long long ib = item * P.strideC;
    __half* C = C0 ? C0 + ib : nullptr;
    __half* C2 = C20 ? C20 + ib : nullptr;
    __nv_bfloat16* Cb = Cb0 ? Cb0 + ib : nullptr;
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
        const int gi = P.a_split ? 2 * item : item;
        if (bytes) prefetch_l2_bulk(P.Gin + gi * P.strideC + (long long)row * P.ldc + col0, bytes);
    }
}

__device__ __forceinline__ uint32_t stage64_off(int y, int x);

// Values of one 32-column chunk of a symmetric result for this thread's row:
// kEpiSyrk scales, kEpiPoly adds a I + b' G', kEpiPlain passes the accumulator.
// gin_s (kEpiPoly, may be null): the warp's 32 x 32 block of G' already in shared
// memory (64-byte-swizzled rows, row = lane), instead of per-thread global loads.
__device__ __forceinline__ void epilogue_values(const GemmProblem& P, int item, int row, int col0,
                                                const uint32_t (&raw)[32], float (&v)[32],
                                                const uint8_t* gin_s = nullptr) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw[j]);
    if (P.epi == kEpiSyrk) {
        const float al = P.alpha[item];
        const float k = P.out_scale * al * al;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= k;
    } else if (P.epi == kEpiPoly && gin_s != nullptr) {
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 t = *reinterpret_cast<const uint4*>(gin_s + stage64_off(lane, 8 * q));
            const uint32_t w4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w4[e]));
                const int j = 8 * q + 2 * e;
                v[j] = P.coef_c * v[j] + P.coef_b * f.x + ((col0 + j == row) ? P.coef_a : 0.f);
                v[j + 1] = P.coef_c * v[j + 1] + P.coef_b * f.y + ((col0 + j + 1 == row) ? P.coef_a : 0.f);
            }
        }
    } else if (P.epi == kEpiPoly) {
        // P = a I + b' G' + c' G'^2, with G' read (8 values at a time) from the fp16
        // input the MMA used
        const int gi = P.a_split ? 2 * item : item;   // split: G' = hi (item 2i) + lo (item 2i + 1)
        const __half* Grow = P.Gin + gi * P.strideC + (long long)(row < P.M ? row : 0) * P.ldc + col0;
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
            if (P.a_split) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    g[e] += (row < P.M && col0 + 8 * q + e < P.N) ? __half2float(Grow[P.strideC + 8 * q + e]) : 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int j = 8 * q + e;
                v[j] = P.coef_c * v[j] + P.coef_b * g[e] + ((col0 + j == row) ? P.coef_a : 0.f);
            }
        }
    }
}

// X' = alpha acc as bf16 rows (ldc, item stride strideC): the iterate handed from one
// restarted Newton-Schulz segment to the next (not symmetric: rows only).
__device__ __forceinline__ void store_xout(const GemmProblem& P, int item, int row, int col0,
                                           const uint32_t (&raw)[32]) {
    if (row >= P.M) return;
    const float al = P.alpha[item];
    if (P.out_split) {   // X' as bf16 hi (item 2i) and lo (item 2i + 1)
        __nv_bfloat16* hi = P.Cb + 2 * item * P.strideC + (long long)row * P.ldc + col0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (col0 + j < P.N) {
                const float x = al * __uint_as_float(raw[j]);
                const __nv_bfloat16 h = __float2bfloat16_rn(x);
                hi[j] = h;
                hi[P.strideC + j] = __float2bfloat16_rn(x - __bfloat162float(h));
            }
        }
        return;
    }
    __nv_bfloat16* dst = P.Cb + item * P.strideC + (long long)row * P.ldc + col0;
    if (col0 + 31 < P.N && (P.ldc & 7) == 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t* r = raw + 8 * q;
            reinterpret_cast<uint4*>(dst)[q] = make_uint4(
                pack_bf162(al * __uint_as_float(r[0]), al * __uint_as_float(r[1])),
                pack_bf162(al * __uint_as_float(r[2]), al * __uint_as_float(r[3])),
                pack_bf162(al * __uint_as_float(r[4]), al * __uint_as_float(r[5])),
                pack_bf162(al * __uint_as_float(r[6]), al * __uint_as_float(r[7])));
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (col0 + j < P.N) dst[j] = __float2bfloat16_rn(al * __uint_as_float(raw[j]));
    }
}

__device__ __forceinline__ void epilogue_chunk(const GemmProblem& P, int item, int row, int col0,
                                               const uint32_t (&raw)[32]) {
    if (P.epi == kEpiXout) {
        store_xout(P, item, row, col0, raw);
        return;
    }
    float v[32];
    epilogue_values(P, item, row, col0, raw, v);
    store_sym(P, item, row, col0, v);
}

// The same chunk written through shared memory with TMA stores: the warp's 32 x 32
// block (rows R0 .. R0 + 31, columns col0 .. col0 + 31) is staged in `stl` as 64-byte
// rows in the 64-byte-swizzled layout of the store box, and, for blocks below the
// diagonal, its transpose in `stm`; lane 0 stores them at (col0, R0) and (R0, col0).
// A block on the diagonal (col0 == R0) is staged as its lower triangle plus the
// mirror of it and stored once, so the output is exactly symmetric (the products
// read B transposed) and every element is written exactly once.  Rows and columns
// beyond the matrix fall outside the store box's extents and are not written.
__device__ __forceinline__ uint32_t stage64_off(int y, int x) {   // 2-byte element (y, x), x < 32
    return (uint32_t)(y * 64 + ((((x >> 3) ^ ((y >> 1) & 3))) << 4) + ((x & 7) << 1));
}

__device__ __forceinline__ void epilogue_chunk_tma(const GemmProblem& P, const CUtensorMap* mc,
                                                   const CUtensorMap* mc2, int item, int R0, int col0, int lane,
                                                   const uint32_t (&raw)[32], uint8_t* stl, uint8_t* stm,
                                                   const uint8_t* gin_s = nullptr) {
    float v[32];
    epilogue_values(P, item, R0 + lane, col0, raw, v, gin_s);
    const bool diag = col0 == R0;
    // the transposed block goes to the mirror position unless the output is stored as
    // its lower triangle and the block lies below the diagonal 256 x 256 tile
    const bool mirror = !diag && (!P.lower_out || ((R0 ^ col0) & ~255) == 0);
    const bool bf = (P.tma_out & kTmaOutBf16) != 0;
    if (lane == 0) bulk_wait_read<0>();   // the previous chunk's stores have read the staging
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float* x = v + 8 * q;
        const uint4 pk = bf ? make_uint4(pack_bf162(x[0], x[1]), pack_bf162(x[2], x[3]), pack_bf162(x[4], x[5]),
                                         pack_bf162(x[6], x[7]))
                            : make_uint4(pack_half2(x[0], x[1]), pack_half2(x[2], x[3]), pack_half2(x[4], x[5]),
                                         pack_half2(x[6], x[7]));
        *reinterpret_cast<uint4*>(stl + stage64_off(lane, 8 * q)) = pk;
    }
    if (diag) {
        __syncwarp();   // rows staged; the upper triangle becomes the mirror of the lower
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (j < lane) {
                const unsigned short h = bf ? __bfloat16_as_ushort(__float2bfloat16_rn(v[j]))
                                            : __half_as_ushort(to_half(v[j]));
                *reinterpret_cast<unsigned short*>(stl + stage64_off(j, lane)) = h;
            }
        }
    } else if (mirror) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const unsigned short h = bf ? __bfloat16_as_ushort(__float2bfloat16_rn(v[j]))
                                        : __half_as_ushort(to_half(v[j]));
            *reinterpret_cast<unsigned short*>(stm + stage64_off(j, lane)) = h;
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // staging visible to the TMA unit
    __syncwarp();
    if (lane == 0) {
        if (P.tma_out & kTmaOutC) tma_store_3d(mc, stl, col0, R0, item);
        if (P.tma_out & kTmaOutC2) tma_store_3d(mc2, stl, col0, R0, item);
        if (mirror) {
            if (P.tma_out & kTmaOutC) tma_store_3d(mc, stm, R0, col0, item);
            if (P.tma_out & kTmaOutC2) tma_store_3d(mc2, stm, R0, col0, item);
        }
        bulk_commit();
    }
}

// ------------------------------------------------------------------ W staging (fused update)
// A piece is oriented rows [rw, rw + 32) x columns [col0, col0 + 32) of one
// matrix, staged in its stored orientation: 32 lines of 128 B (a line is an
// oriented row when W is stored r x c, an oriented column when stored c x r),
// 16-byte chunks XOR-swizzled by line so that both the coalesced copies and the
// one-row-per-thread update are free of bank conflicts.
constexpr int kWPiece = 32 * 32 * 4;   // one 32 x 32 fp32 piece of W

struct WPiece {
    float* W;        // the matrix, stored layout
    long long ld;    // stored leading dimension: N (r x c) or M (c x r)
    int M, N;        // oriented extent
    bool tr;         // stored c x r
    bool vec;        // 16-byte copies possible
};

// item < 0: an empty context (problems without the fused update)
__device__ __forceinline__ WPiece w_piece_ctx(const GemmProblem& P, int item) {
    WPiece c;
    c.M = P.M;
    c.N = P.N;
    if (item < 0) {
        c.W = nullptr;
        c.ld = 0;
        c.tr = false;
        c.vec = false;
        return c;
    }
    const int mat = P.item_mat[item];
    c.W = P.W[mat];
    c.tr = P.transposed[mat] != 0;
    c.ld = c.tr ? P.M : P.N;
    c.vec = ((c.ld & 3) == 0) && ((reinterpret_cast<uintptr_t>(c.W) & 15) == 0);
    return c;
}

__device__ __forceinline__ uint32_t stage_off(int line, int e) {   // element e (0..31) of a line
    return (uint32_t)(line * 128 + ((((e >> 2) ^ (line & 7))) << 4) + ((e & 3) << 2));
}

// Global address and validity of staged element (line, e) of the piece at (rw, col0).
__device__ __forceinline__ float* w_elem(const WPiece& c, int rw, int col0, int line, int e, bool& ok) {
    int row, col;
    if (c.tr) {
        col = col0 + line;
        row = rw + e;
    } else {
        row = rw + line;
        col = col0 + e;
    }
    ok = row < c.M && col < c.N;
    return c.tr ? c.W + (long long)col * c.ld + row : c.W + (long long)row * c.ld + col;
}

// Issue the copies of one piece into `buf` (one commit group per call).
__device__ __forceinline__ void w_piece_load(const WPiece& c, int rw, int col0, uint32_t buf, int lane) {
    if (col0 < c.N && rw < c.M) {
        if (c.vec) {
            // lanes 8i..8i+7 take the eight 16-byte chunks of line 4s + i
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const int line = 4 * s + (lane >> 3), e = 4 * (lane & 7);
                bool ok;
                const float* g = w_elem(c, rw, col0, line, e, ok);
                if (ok) cp_async_16(buf + stage_off(line, e), g);
            }
        } else {
#pragma unroll 4
            for (int line = 0; line < 32; ++line) {
                bool ok;
                const float* g = w_elem(c, rw, col0, line, lane, ok);
                if (ok) cp_async_4(buf + stage_off(line, lane), g);
            }
        }
    }
    cp_async_commit();
}

// Write a staged piece back to global memory with the same coalesced mapping.
__device__ __forceinline__ void w_piece_store(const WPiece& c, int rw, int col0, const uint8_t* buf, int lane) {
    if (col0 >= c.N || rw >= c.M) return;
    if (c.vec) {
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const int line = 4 * s + (lane >> 3), e = 4 * (lane & 7);
            bool ok;
            float* g = w_elem(c, rw, col0, line, e, ok);
            if (ok) *reinterpret_cast<float4*>(g) = *reinterpret_cast<const float4*>(buf + stage_off(line, e));
        }
    } else {
#pragma unroll 4
        for (int line = 0; line < 32; ++line) {
            bool ok;
            float* g = w_elem(c, rw, col0, line, lane, ok);
            if (ok) *g = *reinterpret_cast<const float*>(buf + stage_off(line, lane));
        }
    }
}

// The fused update of this thread's row of a staged piece:
// w -= lr (scale alpha acc + wd w), acc the 32 accumulator columns of the row.
// Plans that keep the update also write O = alpha acc (fp32, stored layout).
__device__ __forceinline__ void w_piece_update(const GemmProblem& P, const WPiece& c, int item, int rw, int col0,
                                               uint8_t* buf, int lane, const uint32_t (&acc)[32]) {
    const float al = P.alpha[item];
    const float lr = P.lr, wd = P.wd, s = P.scale;
    if (!c.tr) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float4* p = reinterpret_cast<float4*>(buf + stage_off(lane, 4 * q));
            float4 w = *p;
            w.x -= lr * (s * (al * __uint_as_float(acc[4 * q])) + wd * w.x);
            w.y -= lr * (s * (al * __uint_as_float(acc[4 * q + 1])) + wd * w.y);
            w.z -= lr * (s * (al * __uint_as_float(acc[4 * q + 2])) + wd * w.z);
            w.w -= lr * (s * (al * __uint_as_float(acc[4 * q + 3])) + wd * w.w);
            *p = w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            float* p = reinterpret_cast<float*>(buf + stage_off(j, lane));
            const float w = *p;
            *p = w - lr * (s * (al * __uint_as_float(acc[j])) + wd * w);
        }
    }
    if (P.Odbg != nullptr) {
        float* O = P.Odbg + (long long)item * P.M * P.N;
        const int row = rw + lane;
        if (row < c.M) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const long long idx = c.tr ? (long long)(col0 + j) * c.ld + row : (long long)row * c.ld + col0 + j;
                if (col0 + j < c.N) O[idx] = al * __uint_as_float(acc[j]);
            }
        }
    }
}

}  // namespace muon
