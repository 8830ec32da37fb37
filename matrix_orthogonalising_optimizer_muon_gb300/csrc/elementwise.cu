// HBM-streaming kernels of the Muon step (no tensor cores):
//  * momentum:  M <- mu M + G,  U = mu M + G  ("Muon is Scalable" blog, eq. (1) and the
//    Nesterov input), per-block partial sums of U^2 for ||U||_F (Background,
//    X0 = M/||M||_F), and U written as bf16 in the ORIENTED layout (DiT paper
//    sec. 3.1: transposed when m > n) so every tensor-core operand is K-major.
//  * norm finalize: alpha = 1/||U||_F per matrix, fixed-order (deterministic) sum.
//  * RowNorm (DiT paper sec. 3.1, R_eps over rows of the oriented matrix) fused
//    with momentum and the update W <- W - lr (0.2 sqrt(c) R + wd W) (blog eq. (4)).
// Reductions never use floating-point atomics, so results are bitwise
// reproducible run to run.
#include "kernels.h"
#include "ptx.cuh"

namespace muon {

namespace {

__device__ __forceinline__ bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
__device__ __forceinline__ bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7) == 0; }

// Largest i with list_blk[i] <= b (list_blk is a prefix over the launch list).
__device__ __forceinline__ int find_entry(const long long* list_blk, int nlist, long long b) {
    int lo = 0, hi = nlist - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (list_blk[mid] <= b)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Fixed-order block sum; the result is returned to every thread.
__device__ __forceinline__ float block_sum_all(float v, float* sred) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) sred[w] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += sred[i];
        sred[32] = t;
    }
    __syncthreads();
    const float t = sred[32];
    __syncthreads();
    return t;
}

template <bool BF16>
__device__ __forceinline__ float load_g(const void* G, long long e) {
    if (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(G)[e]);
    return reinterpret_cast<const float*>(G)[e];
}

// 4 consecutive gradient values; G + e must be 8-byte (bf16) / 16-byte (fp32) aligned.
template <bool BF16>
__device__ __forceinline__ float4 load_g4(const void* G, long long e) {
    if (BF16) {
        const uint2 raw = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(G) + e);
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
        const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
        return make_float4(fa.x, fa.y, fb.x, fb.y);
    }
    return *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(G) + e);
}

template <bool BF16>
__device__ __forceinline__ bool g_vec_ok(const void* G) {
    return BF16 ? aligned8(G) : aligned16(G);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// ------------------------------------------------------------------ momentum, m <= n
template <bool BF16>
__global__ void __launch_bounds__(kElemThreads) k_momentum_rows(const ElemArgs a) {
    pdl_trigger();
    pdl_wait();
    __shared__ float sred[33];
    const long long b = blockIdx.x;
    const int li = find_entry(a.list_blk, a.nlist, b);
    const int mi = a.list[li];
    const MatDev md = a.mats[mi];
    const long long blk = b - a.list_blk[li];
    const long long numel = md.m * md.n;
    const void* G = a.G[mi];
    float* M = a.M[mi];
    __nv_bfloat16* U = a.ut + md.ut_off;
    const float mu = a.mu;
    float ss = 0.f;
    const long long e0 = blk * kMomElemsPerBlock;
    const bool vec = (md.n % 8 == 0) && g_vec_ok<BF16>(G) && aligned16(M);
    if (vec) {
        // n % 8 == 0 means ldu == n: X0 has the stored layout and the same index
#pragma unroll
        for (int k = 0; k < kMomVecPerThread; ++k) {
            const long long e = e0 + ((long long)k * kElemThreads + threadIdx.x) * 8;
            if (e < numel) {
                const float4 g0 = load_g4<BF16>(G, e), g1 = load_g4<BF16>(G, e + 4);
                float4* m4 = reinterpret_cast<float4*>(M + e);
                float4 m0 = m4[0], m1 = m4[1];
                m0.x = mu * m0.x + g0.x; m0.y = mu * m0.y + g0.y; m0.z = mu * m0.z + g0.z; m0.w = mu * m0.w + g0.w;
                m1.x = mu * m1.x + g1.x; m1.y = mu * m1.y + g1.y; m1.z = mu * m1.z + g1.z; m1.w = mu * m1.w + g1.w;
                m4[0] = m0;
                m4[1] = m1;
                const float u0 = mu * m0.x + g0.x, u1 = mu * m0.y + g0.y, u2 = mu * m0.z + g0.z, u3 = mu * m0.w + g0.w;
                const float u4 = mu * m1.x + g1.x, u5 = mu * m1.y + g1.y, u6 = mu * m1.z + g1.z, u7 = mu * m1.w + g1.w;
                ss += u0 * u0 + u1 * u1 + u2 * u2 + u3 * u3 + u4 * u4 + u5 * u5 + u6 * u6 + u7 * u7;
                uint4 pk;
                pk.x = pack_bf16x2(u0, u1);
                pk.y = pack_bf16x2(u2, u3);
                pk.z = pack_bf16x2(u4, u5);
                pk.w = pack_bf16x2(u6, u7);
                *reinterpret_cast<uint4*>(U + e) = pk;
                if (md.x_split) {   // lo part: u - bf16(u), itself rounded to bf16
                    const float v[8] = {u0, u1, u2, u3, u4, u5, u6, u7};
                    const uint32_t h[4] = {pk.x, pk.y, pk.z, pk.w};
                    uint32_t l[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 hf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&h[q]));
                        l[q] = pack_bf16x2(v[2 * q] - hf.x, v[2 * q + 1] - hf.y);
                    }
                    *reinterpret_cast<uint4*>(U + (long long)md.r * md.ldu + e) = make_uint4(l[0], l[1], l[2], l[3]);
                }
            }
        }
    } else {
        for (int k = 0; k < 8 * kMomVecPerThread; ++k) {
            const long long e = e0 + (long long)k * kElemThreads + threadIdx.x;
            if (e < numel) {
                const long long i = e / md.n, j = e - i * md.n;
                const float g = load_g<BF16>(G, e);
                const float m = mu * M[e] + g;
                M[e] = m;
                const float u = mu * m + g;
                ss += u * u;
                const __nv_bfloat16 h = __float2bfloat16_rn(u);
                U[i * md.ldu + j] = h;
                if (md.x_split) U[(long long)md.r * md.ldu + i * md.ldu + j] = __float2bfloat16_rn(u - __bfloat162float(h));
            }
        }
    }
    const float tot = block_sum_all(ss, sred);
    if (threadIdx.x == 0) a.partials[md.part_off + blk] = tot;
}

// ------------------------------------------------------------------ momentum, m > n (transpose to r x c)
template <bool BF16>
__global__ void __launch_bounds__(kElemThreads) k_momentum_tiles(const ElemArgs a) {
    pdl_trigger();
    pdl_wait();
    __shared__ float tile[kTile][kTileRows + 1];   // [stored col][stored row]
    __shared__ float sred[33];
    const long long b = blockIdx.x;
    const int li = find_entry(a.list_blk, a.nlist, b);
    const int mi = a.list[li];
    const MatDev md = a.mats[mi];
    const long long blk = b - a.list_blk[li];
    const long long tiles_n = (md.n + kTile - 1) / kTile;
    const long long i0 = (blk / tiles_n) * kTileRows;
    const long long j0 = (blk % tiles_n) * kTile;
    const void* G = a.G[mi];
    float* M = a.M[mi];
    __nv_bfloat16* U = a.ut + md.ut_off;   // r x ldu with r = n, c = m
    const float mu = a.mu;
    const int t = threadIdx.x;
    float ss = 0.f;
    const bool full = (i0 + kTileRows <= md.m) && (j0 + kTile <= md.n) && (md.n % 4 == 0) && g_vec_ok<BF16>(G) &&
                      aligned16(M);
    const int cq = t % kTileTpr, rr = t / kTileTpr;
    if (full) {
        // G and M of kTileAhead passes are loaded before the first of their M stores (which
        // the compiler may not move loads across): 96 B in flight per thread instead of 24
        // (momentum of the 56 transposed 18944 x 3584 matrices 14.8 -> 13.9 ms per step)
        constexpr int kPasses = kTileRows / kTileRpp;
        constexpr int kTileAhead = kPasses < 4 ? kPasses : 4;
        static_assert(kPasses % kTileAhead == 0, "passes per load batch");
#pragma unroll
        for (int p0 = 0; p0 < kPasses; p0 += kTileAhead) {
            float4 gv[kTileAhead], mv[kTileAhead];
#pragma unroll
            for (int q = 0; q < kTileAhead; ++q) {
                const long long e = (i0 + rr + kTileRpp * (p0 + q)) * md.n + j0 + 4 * cq;
                gv[q] = load_g4<BF16>(G, e);
                mv[q] = *reinterpret_cast<const float4*>(M + e);
            }
#pragma unroll
            for (int q = 0; q < kTileAhead; ++q) {
                const int p = p0 + q;
                const long long e = (i0 + rr + kTileRpp * p) * md.n + j0 + 4 * cq;
                const float4 g = gv[q];
                float4 m = mv[q];
                m.x = mu * m.x + g.x; m.y = mu * m.y + g.y; m.z = mu * m.z + g.z; m.w = mu * m.w + g.w;
                *reinterpret_cast<float4*>(M + e) = m;
                const float u0 = mu * m.x + g.x, u1 = mu * m.y + g.y, u2 = mu * m.z + g.z, u3 = mu * m.w + g.w;
                ss += u0 * u0 + u1 * u1 + u2 * u2 + u3 * u3;
                tile[4 * cq + 0][rr + kTileRpp * p] = u0;
                tile[4 * cq + 1][rr + kTileRpp * p] = u1;
                tile[4 * cq + 2][rr + kTileRpp * p] = u2;
                tile[4 * cq + 3][rr + kTileRpp * p] = u3;
            }
        }
    } else {
#pragma unroll
        for (int p = 0; p < kTileRows / kTileRpp; ++p) {
            const long long i = i0 + rr + kTileRpp * p;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const long long j = j0 + 4 * cq + q;
                float u = 0.f;
                if (i < md.m && j < md.n) {
                    const long long e = i * md.n + j;
                    const float g = load_g<BF16>(G, e);
                    const float m = mu * M[e] + g;
                    M[e] = m;
                    u = mu * m + g;
                    ss += u * u;
                }
                tile[4 * cq + q][rr + kTileRpp * p] = u;
            }
        }
    }
    __syncthreads();
    // X0 row jj = stored column j0 + jj; its elements are stored rows i0 .. i0 + kTileRows - 1.
    // Warp w writes X0 rows 8w .. 8w + 7; lane l takes elements l, l + 32, l + 64, l + 96,
    // so the shared reads hit 32 banks and each store covers 64 contiguous bytes.
    {
        const int lane = t & 31, wid = t >> 5;
#pragma unroll 2
        for (int r = 0; r < kTile / (kElemThreads / 32); ++r) {
            const int jj = wid * (kTile / (kElemThreads / 32)) + r;
            const long long gj = j0 + jj;
            if (gj < md.n) {
                __nv_bfloat16* dst = U + gj * md.ldu + i0;
#pragma unroll
                for (int q = 0; q < kTileRows / 32; ++q) {
                    const int ii = lane + 32 * q;
                    if (i0 + ii < md.m) {
                        const float u = tile[jj][ii];
                        const __nv_bfloat16 h = __float2bfloat16_rn(u);
                        dst[ii] = h;
                        if (md.x_split) dst[(long long)md.r * md.ldu + ii] = __float2bfloat16_rn(u - __bfloat162float(h));
                    }
                }
            }
        }
    }
    const float tot = block_sum_all(ss, sred);
    if (t == 0) a.partials[md.part_off + blk] = tot;
}

// ------------------------------------------------------------------ 1/||U||_F
__global__ void k_norm_finalize(const ElemArgs a) {
    pdl_trigger();
    pdl_wait();
    const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= a.nlist) return;
    const MatDev md = a.mats[a.list[w]];
    double s = 0.0;
    for (int k = lane; k < md.nblk; k += 32) s += (double)a.partials[md.part_off + k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) {
        a.alpha[md.slot] = s > 0.0 ? (float)(1.0 / sqrt(s)) : 0.f;
        if (a.check_finite && !isfinite(s)) atomicOr(a.status, kStatusNonFinite);
    }
}

__global__ void k_identity_bf16(__nv_bfloat16* q, int r, int ld, long long total, int split) {
    pdl_trigger();
    pdl_wait();
    const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= total) return;
    const long long per = (long long)r * ld;
    const long long w = e % per;
    const long long i = w / ld, j = w % ld;
    const bool lo_part = split && ((e / per) & 1);
    q[e] = __float2bfloat16_rn((i == j && !lo_part) ? 1.f : 0.f);
}

// ------------------------------------------------------------------ RowNorm, m <= n (stored rows)
// VEC float4 groups per thread kept in registers (rows <= 1024 VEC elements).  The
// planner launches rows of up to 2048, 4096 and more elements with VEC = 2, 4 and 8,
// so short rows do not hold the registers (and the occupancy) of the longest.
template <bool BF16, int VEC>
__global__ void __launch_bounds__(kElemThreads) k_rownorm_rows(const ElemArgs a) {
    pdl_trigger();
    pdl_wait();
    __shared__ float sred[33];
    const long long b = blockIdx.x;
    const int li = find_entry(a.list_blk, a.nlist, b);
    const int mi = a.list[li];
    const MatDev md = a.mats[mi];
    const long long row = b - a.list_blk[li];
    const long long n = md.n;
    const long long base = row * n;
    const void* G = a.G[mi];
    float* M = a.M[mi] + base;
    float* W = a.W[mi] + base;
    const float mu = a.mu, lr = a.lr, wd = a.wd, s = md.scale;
    const int t = threadIdx.x;
    const bool reg = (n % 4 == 0) && (n <= 4LL * kElemThreads * VEC) && g_vec_ok<BF16>(G) &&
                     aligned16(M) && aligned16(W);
    float ss = 0.f;
    if (reg) {
        // Rows of up to 4096 elements load W with G and M, so all three streams are in
        // flight across the row reduction.  Longer rows (VEC = 8) load W after it: holding
        // W too took 80-94 registers (3 blocks per SM) against 64 (4 blocks), and the
        // extra resident rows keep more loads in flight (RowNorm step of the DiT set 7.10
        // -> 6.85 ms in a same-box comparison).
        constexpr bool kEarlyW = VEC < 8;
        float4 u[VEC], wv[VEC];
        if (kEarlyW) {
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const long long j = 4LL * (v * kElemThreads + t);
                if (j < n) wv[v] = *reinterpret_cast<const float4*>(W + j);
            }
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const long long j = 4LL * (v * kElemThreads + t);
            if (j < n) {
                const float4 g = load_g4<BF16>(G, base + j);
                float4 m = *reinterpret_cast<float4*>(M + j);
                m.x = mu * m.x + g.x; m.y = mu * m.y + g.y; m.z = mu * m.z + g.z; m.w = mu * m.w + g.w;
                *reinterpret_cast<float4*>(M + j) = m;
                u[v] = make_float4(mu * m.x + g.x, mu * m.y + g.y, mu * m.z + g.z, mu * m.w + g.w);
                ss += u[v].x * u[v].x + u[v].y * u[v].y + u[v].z * u[v].z + u[v].w * u[v].w;
            }
        }
        const float tot = block_sum_all(ss, sred);
        if (a.check_finite && t == 0 && !isfinite(tot)) atomicOr(a.status, kStatusNonFinite);
        const float inv = 1.f / fmaxf(sqrtf(tot), a.eps);
        const float k = s * inv;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const long long j = 4LL * (v * kElemThreads + t);
            if (j < n) {
                float4 w = kEarlyW ? wv[v] : *reinterpret_cast<const float4*>(W + j);
                w.x = w.x - lr * (k * u[v].x + wd * w.x);
                w.y = w.y - lr * (k * u[v].y + wd * w.y);
                w.z = w.z - lr * (k * u[v].z + wd * w.z);
                w.w = w.w - lr * (k * u[v].w + wd * w.w);
                *reinterpret_cast<float4*>(W + j) = w;
            }
        }
    } else {
        // long or unaligned rows: second pass recomputes U from G and the new M
        for (long long j = t; j < n; j += kElemThreads) {
            const float g = load_g<BF16>(G, base + j);
            const float m = mu * M[j] + g;
            M[j] = m;
            const float u = mu * m + g;
            ss += u * u;
        }
        const float tot = block_sum_all(ss, sred);
        if (a.check_finite && t == 0 && !isfinite(tot)) atomicOr(a.status, kStatusNonFinite);
        const float inv = 1.f / fmaxf(sqrtf(tot), a.eps);
        const float k = s * inv;
        for (long long j = t; j < n; j += kElemThreads) {
            const float g = load_g<BF16>(G, base + j);
            const float u = mu * M[j] + g;
            const float w = W[j];
            W[j] = w - lr * (k * u + wd * w);
        }
    }
}

// ------------------------------------------------------------------ RowNorm, m > n (stored columns)
// Block: stored rows [i0, i0 + kColSlab) x columns [j0, j0 + kColWidth); partial
// column sums of U^2 go to partials[cpart_off + slab * n + j].
template <bool BF16>
__global__ void __launch_bounds__(kElemThreads) k_rownorm_colstats(const ElemArgs a) {
    pdl_trigger();
    pdl_wait();
    const long long b = blockIdx.x;
    const int li = find_entry(a.list_blk, a.nlist, b);
    const int mi = a.list[li];
    const MatDev md = a.mats[mi];
    const long long blk = b - a.list_blk[li];
    const long long n = md.n, m = md.m;
    const long long tiles_j = (n + kColWidth - 1) / kColWidth;
    const long long slab = blk / tiles_j;
    const long long j = (blk % tiles_j) * kColWidth + 4LL * threadIdx.x;
    const long long i0 = slab * kColSlab;
    const long long i1 = (i0 + kColSlab < m) ? i0 + kColSlab : m;
    const void* G = a.G[mi];
    float* M = a.M[mi];
    const float mu = a.mu;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    if (j >= n) return;
    const bool vec = (n % 4 == 0) && g_vec_ok<BF16>(G) && aligned16(M);
    if (vec) {
#pragma unroll 4
        for (long long i = i0; i < i1; ++i) {
            const long long e = i * n + j;
            const float4 g = load_g4<BF16>(G, e);
            float4 mm = *reinterpret_cast<float4*>(M + e);
            mm.x = mu * mm.x + g.x; mm.y = mu * mm.y + g.y; mm.z = mu * mm.z + g.z; mm.w = mu * mm.w + g.w;
            *reinterpret_cast<float4*>(M + e) = mm;
            const float u0 = mu * mm.x + g.x, u1 = mu * mm.y + g.y, u2 = mu * mm.z + g.z, u3 = mu * mm.w + g.w;
            s0 += u0 * u0;
            s1 += u1 * u1;
            s2 += u2 * u2;
            s3 += u3 * u3;
        }
    } else {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (long long i = i0; i < i1; ++i) {
            for (int q = 0; q < 4; ++q) {
                if (j + q < n) {
                    const long long e = i * n + j + q;
                    const float g = load_g<BF16>(G, e);
                    const float mm = mu * M[e] + g;
                    M[e] = mm;
                    const float u = mu * mm + g;
                    acc[q] += u * u;
                }
            }
        }
        s0 = acc[0]; s1 = acc[1]; s2 = acc[2]; s3 = acc[3];
    }
    float* dst = a.partials + md.cpart_off + slab * n + j;
    dst[0] = s0;
    if (j + 1 < n) dst[1] = s1;
    if (j + 2 < n) dst[2] = s2;
    if (j + 3 < n) dst[3] = s3;
}

// inv[j] = 1 / max(||U[:, j]||_2, eps): fixed-order sum over the row slabs.
__global__ void __launch_bounds__(kElemThreads) k_rownorm_colfinal(const ElemArgs a) {
    pdl_trigger();
    pdl_wait();
    const long long b = blockIdx.x;
    const int li = find_entry(a.list_blk, a.nlist, b);
    const MatDev md = a.mats[a.list[li]];
    const long long j = (b - a.list_blk[li]) * kElemThreads + threadIdx.x;
    if (j >= md.n) return;
    const long long slabs = (md.m + kColSlab - 1) / kColSlab;
    float s = 0.f;
    for (long long k = 0; k < slabs; ++k) s += a.partials[md.cpart_off + k * md.n + j];
    if (a.check_finite && !isfinite(s)) atomicOr(a.status, kStatusNonFinite);
    a.rowinv[md.inv_off + j] = 1.f / fmaxf(sqrtf(s), a.eps);
}

// Dim-0 shards: this shard's column sums of U^2 (fixed slab order) into out[inv_off + j],
// the padding up to a multiple of 4 written as 0, for the caller to sum across shards.
__global__ void __launch_bounds__(kElemThreads) k_rownorm_colsum(const ElemArgs a, float* out) {
    pdl_trigger();
    pdl_wait();
    const long long b = blockIdx.x;
    const int li = find_entry(a.list_blk, a.nlist, b);
    const MatDev md = a.mats[a.list[li]];
    const long long j = (b - a.list_blk[li]) * kElemThreads + threadIdx.x;
    const long long npad = (md.n + 3) / 4 * 4;
    if (j >= npad) return;
    float s = 0.f;
    if (j < md.n) {
        const long long slabs = (md.m + kColSlab - 1) / kColSlab;
        for (long long k = 0; k < slabs; ++k) s += a.partials[md.cpart_off + k * md.n + j];
    }
    out[md.inv_off + j] = s;
}

// inv[j] = 1 / max(sqrt(colsq[j]), eps) from column sums already summed over the shards.
__global__ void __launch_bounds__(kElemThreads) k_rownorm_colinv(const ElemArgs a, const float* colsq) {
    pdl_trigger();
    pdl_wait();
    const long long b = blockIdx.x;
    const int li = find_entry(a.list_blk, a.nlist, b);
    const MatDev md = a.mats[a.list[li]];
    const long long j = (b - a.list_blk[li]) * kElemThreads + threadIdx.x;
    if (j >= md.n) return;
    const float s = colsq[md.inv_off + j];
    if (a.check_finite && !isfinite(s)) atomicOr(a.status, kStatusNonFinite);
    a.rowinv[md.inv_off + j] = 1.f / fmaxf(sqrtf(s), a.eps);
}

// W <- W - lr (s * U * inv[col] + wd W), U recomputed from G and the stored new M.
template <bool BF16>
__global__ void __launch_bounds__(kElemThreads) k_rownorm_colapply(const ElemArgs a) {
    pdl_trigger();
    pdl_wait();
    const long long b = blockIdx.x;
    const int li = find_entry(a.list_blk, a.nlist, b);
    const int mi = a.list[li];
    const MatDev md = a.mats[mi];
    const long long blk = b - a.list_blk[li];
    const long long n = md.n, numel = md.m * md.n;
    const void* G = a.G[mi];
    const float* M = a.M[mi];
    float* W = a.W[mi];
    const float* inv = a.rowinv + md.inv_off;
    const float mu = a.mu, lr = a.lr, wd = a.wd, s = md.scale;
    const long long e0 = blk * kApplyElemsPerBlock;
    const bool vec = (n % 4 == 0) && g_vec_ok<BF16>(G) && aligned16(M) && aligned16(W);
    if (vec) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const long long e = e0 + 4LL * (k * kElemThreads + threadIdx.x);
            if (e < numel) {
                const long long j = e % n;
                const float4 g = load_g4<BF16>(G, e);
                const float4 mm = *reinterpret_cast<const float4*>(M + e);
                const float4 iv = *reinterpret_cast<const float4*>(inv + j);
                float4 w = *reinterpret_cast<float4*>(W + e);
                w.x = w.x - lr * (s * iv.x * (mu * mm.x + g.x) + wd * w.x);
                w.y = w.y - lr * (s * iv.y * (mu * mm.y + g.y) + wd * w.y);
                w.z = w.z - lr * (s * iv.z * (mu * mm.z + g.z) + wd * w.z);
                w.w = w.w - lr * (s * iv.w * (mu * mm.w + g.w) + wd * w.w);
                *reinterpret_cast<float4*>(W + e) = w;
            }
        }
    } else {
        for (int k = 0; k < 16; ++k) {
            const long long e = e0 + (long long)k * kElemThreads + threadIdx.x;
            if (e < numel) {
                const long long j = e % n;
                const float u = mu * M[e] + load_g<BF16>(G, e);
                const float w = W[e];
                W[e] = w - lr * (s * inv[j] * u + wd * w);
            }
        }
    }
}

}  // namespace

cudaError_t launch_momentum_rows(const ElemArgs& a, long long blocks, cudaStream_t s) {
    if (blocks <= 0) return cudaSuccess;
    if (a.grad_bf16)
        return launch_pdl(k_momentum_rows<true>, dim3((unsigned)blocks), dim3(kElemThreads), 0, s, a);
    else
        return launch_pdl(k_momentum_rows<false>, dim3((unsigned)blocks), dim3(kElemThreads), 0, s, a);
}
cudaError_t launch_momentum_tiles(const ElemArgs& a, long long blocks, cudaStream_t s) {
    if (blocks <= 0) return cudaSuccess;
    if (a.grad_bf16)
        return launch_pdl(k_momentum_tiles<true>, dim3((unsigned)blocks), dim3(kElemThreads), 0, s, a);
    else
        return launch_pdl(k_momentum_tiles<false>, dim3((unsigned)blocks), dim3(kElemThreads), 0, s, a);
}
cudaError_t launch_norm_finalize(const ElemArgs& a, cudaStream_t s) {
    if (a.nlist <= 0) return cudaSuccess;
    const int warps_per_block = kElemThreads / 32;
    const int blocks = (a.nlist + warps_per_block - 1) / warps_per_block;
    return launch_pdl(k_norm_finalize, dim3(blocks), dim3(kElemThreads), 0, s, a);
}
cudaError_t launch_identity_bf16(__nv_bfloat16* q, int r, int ld, int batch, bool split, cudaStream_t s) {
    const long long total = (long long)r * ld * batch * (split ? 2 : 1);
    if (total <= 0) return cudaSuccess;
    return launch_pdl(k_identity_bf16, dim3((unsigned)((total + 255) / 256)), dim3(256), 0, s, q, r, ld, total,
                      split ? 1 : 0);
}
cudaError_t launch_rownorm_rows(const ElemArgs& a, long long blocks, int vec, cudaStream_t s) {
    if (blocks <= 0) return cudaSuccess;
    const dim3 g((unsigned)blocks), b(kElemThreads);
    if (vec <= 2)
        return a.grad_bf16 ? launch_pdl(k_rownorm_rows<true, 2>, g, b, 0, s, a)
                           : launch_pdl(k_rownorm_rows<false, 2>, g, b, 0, s, a);
    if (vec <= 4)
        return a.grad_bf16 ? launch_pdl(k_rownorm_rows<true, 4>, g, b, 0, s, a)
                           : launch_pdl(k_rownorm_rows<false, 4>, g, b, 0, s, a);
    return a.grad_bf16 ? launch_pdl(k_rownorm_rows<true, 8>, g, b, 0, s, a)
                       : launch_pdl(k_rownorm_rows<false, 8>, g, b, 0, s, a);
}
cudaError_t launch_rownorm_colstats(const ElemArgs& a, long long blocks, cudaStream_t s) {
    if (blocks <= 0) return cudaSuccess;
    if (a.grad_bf16)
        return launch_pdl(k_rownorm_colstats<true>, dim3((unsigned)blocks), dim3(kElemThreads), 0, s, a);
    else
        return launch_pdl(k_rownorm_colstats<false>, dim3((unsigned)blocks), dim3(kElemThreads), 0, s, a);
}
cudaError_t launch_rownorm_colfinal(const ElemArgs& a, long long blocks, cudaStream_t s) {
    if (blocks <= 0) return cudaSuccess;
    return launch_pdl(k_rownorm_colfinal, dim3((unsigned)blocks), dim3(kElemThreads), 0, s, a);
}
cudaError_t launch_rownorm_colsum(const ElemArgs& a, long long blocks, float* out, cudaStream_t s) {
    if (blocks <= 0) return cudaSuccess;
    return launch_pdl(k_rownorm_colsum, dim3((unsigned)blocks), dim3(kElemThreads), 0, s, a, out);
}
cudaError_t launch_rownorm_colinv(const ElemArgs& a, long long blocks, const float* colsq, cudaStream_t s) {
    if (blocks <= 0) return cudaSuccess;
    return launch_pdl(k_rownorm_colinv, dim3((unsigned)blocks), dim3(kElemThreads), 0, s, a, colsq);
}
cudaError_t launch_rownorm_colapply(const ElemArgs& a, long long blocks, cudaStream_t s) {
    if (blocks <= 0) return cudaSuccess;
    if (a.grad_bf16)
        return launch_pdl(k_rownorm_colapply<true>, dim3((unsigned)blocks), dim3(kElemThreads), 0, s, a);
    else
        return launch_pdl(k_rownorm_colapply<false>, dim3((unsigned)blocks), dim3(kElemThreads), 0, s, a);
}

// ------------------------------------------------------------------ relative difference (debug / tuning)
// Sums of (a - b)^2 and b^2 over n floats in fp64: kDiffParts blocks write their partial
// sums (fixed order inside a block), one block adds them in order into out[0], out[1].
__global__ void __launch_bounds__(kElemThreads) k_diff_partial(const float* a, const float* b, long long n,
                                                               double* part) {
    __shared__ double sd[kElemThreads], sb[kElemThreads];
    double d = 0.0, bb = 0.0;
    for (long long e = (long long)blockIdx.x * kElemThreads + threadIdx.x; e < n;
         e += (long long)gridDim.x * kElemThreads) {
        const double x = a[e], y = b[e];
        d += (x - y) * (x - y);
        bb += y * y;
    }
    sd[threadIdx.x] = d;
    sb[threadIdx.x] = bb;
    __syncthreads();
    for (int w = kElemThreads / 2; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) {
            sd[threadIdx.x] += sd[threadIdx.x + w];
            sb[threadIdx.x] += sb[threadIdx.x + w];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        part[2 * blockIdx.x] = sd[0];
        part[2 * blockIdx.x + 1] = sb[0];
    }
}

__global__ void k_diff_final(const double* part, int nparts, double* out) {
    if (threadIdx.x != 0) return;
    double d = 0.0, bb = 0.0;
    for (int k = 0; k < nparts; ++k) {
        d += part[2 * k];
        bb += part[2 * k + 1];
    }
    out[0] = d;
    out[1] = bb;
}

cudaError_t launch_sq_diff(const float* a, const float* b, long long n, double* scratch, cudaStream_t s) {
    k_diff_partial<<<kDiffParts, kElemThreads, 0, s>>>(a, b, n, scratch + 2);
    k_diff_final<<<1, 32, 0, s>>>(scratch + 2, kDiffParts, scratch);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ bounded-wait self test
// One wait on an mbarrier whose phase nothing completes: the bounded wait gives
// up after limit_ns, raises the abort flag and records kStatusTimeoutSelftest in
// the status word, and the kernel returns (the same path every tensor-core kernel
// takes when a TMA load or an MMA commit never arrives).
__global__ void k_wait_selftest(int* status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    mbar_wait(&bar, 0, &abort_flag, status, kStatusTimeoutSelftest, limit_ns);
}

cudaError_t launch_wait_selftest(int* status, unsigned long long limit_ns, cudaStream_t s) {
    k_wait_selftest<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace muon
