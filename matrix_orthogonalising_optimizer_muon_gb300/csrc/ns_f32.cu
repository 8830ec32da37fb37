// Muon NS step in fp32 on CUDA cores for small, nearly square matrices
// (r <= 128): one CTA per matrix (persistent over the matrices of the launch).
//
// Why a separate path: a square (or nearly square) Gaussian matrix has
// singular values close to zero, and the quintic maps them through f^J, whose
// slope near zero is a^J (about 485 for J = 5).  Rounding of the Gram
// recursion to 11 bits (fp16) and of Q to 8 bits (bf16) moves those directions
// by a few percent of O's norm, so the tensor-core recipe misses a 2e-2
// relative bound on such matrices.  Their cost is small (r <= 128), so this
// kernel runs the same Gram recursion entirely in fp32:
//
//   G0 = X0 X0^T;  P_k = aI + bG + cG^2;  Q_k = P_k Q_{k-1};  G_k = G_{k-1} P_k^2;
//   O = Q_J X0   (DMuon, "Gram Newton-Schulz"),
//   W <- W - lr (0.2 sqrt(max(m, n)) O + wd W)   ("Muon is Scalable" blog, eq. (4)),
//
// with X0 = O(U)/||U||_F (blog, Background; orientation from "Scaling Muon for
// Diffusion Transformers" sec. 3.1).  U = mu M + G is recomputed here from the
// momentum the momentum kernel has just written and the gradient, in the same
// fp32 arithmetic, so the bf16 X0 workspace is not used.
//
// Every r x r matrix of the recursion is a polynomial in G0, hence symmetric,
// so each product A B is evaluated as A^T B: both operands are read along rows
// of shared memory (k-major), which makes every operand load a contiguous
// 16-byte vector.  Shared memory holds three 128 x 128 fp32 buffers (G, P, Q);
// products that overwrite one of their operands keep the result in registers
// across a block barrier.  Rows and columns beyond r stay exactly zero.
#include "kernels.h"
#include "ptx.cuh"

namespace muon {
namespace {

constexpr int kF32Threads = 256;          // 16 x 16 threads, 8 x 8 outputs each
constexpr int kDim = 128;                 // operands padded to 128 x 128
constexpr int kLds = 132;                 // row stride (floats): rows stay 16-byte aligned
constexpr int kBuf = kDim * kLds;         // floats per buffer
constexpr int kF32Smem = 3 * kBuf * 4;    // G, P, Q: 202,752 bytes

// Output row / column q (0..7) of thread index t4 (0..15): {4 t4 .. 4 t4 + 3} and
// {64 + 4 t4 .. 64 + 4 t4 + 3}, so a warp's 16-byte operand loads cover 256
// contiguous bytes (no bank conflict) or are broadcasts.
__device__ __forceinline__ int own(int t4, int q) { return ((q >> 2) << 6) + 4 * t4 + (q & 3); }

// acc[i][j] (+)= sum_{k < K} A[k][own(ty, i)] * B[k][own(tx, j)]
template <bool ACCUMULATE>
__device__ __forceinline__ void mm_t(const float* A, const float* B, int K, int ty, int tx, float (&acc)[8][8]) {
    if (!ACCUMULATE) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    }
    const float* a_p = A + 4 * ty;
    const float* b_p = B + 4 * tx;
#pragma unroll 2
    for (int k = 0; k < K; ++k) {
        const float4 a0 = *reinterpret_cast<const float4*>(a_p + k * kLds);
        const float4 a1 = *reinterpret_cast<const float4*>(a_p + k * kLds + 64);
        const float4 b0 = *reinterpret_cast<const float4*>(b_p + k * kLds);
        const float4 b1 = *reinterpret_cast<const float4*>(b_p + k * kLds + 64);
        const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
}

// C[own(ty, i)][own(tx, j)] = acc[i][j], zero outside the leading r x r block.
__device__ __forceinline__ void store_tile(float* C, int r, int ty, int tx, const float (&acc)[8][8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = own(ty, i);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int col = own(tx, 4 * h);
            float4 v;
            v.x = (row < r && col + 0 < r) ? acc[i][4 * h + 0] : 0.f;
            v.y = (row < r && col + 1 < r) ? acc[i][4 * h + 1] : 0.f;
            v.z = (row < r && col + 2 < r) ? acc[i][4 * h + 2] : 0.f;
            v.w = (row < r && col + 3 < r) ? acc[i][4 * h + 3] : 0.f;
            *reinterpret_cast<float4*>(C + row * kLds + col) = v;
        }
    }
}

template <bool BF16>
__device__ __forceinline__ float grad_at(const void* G, long long e) {
    if (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(G)[e]);
    return reinterpret_cast<const float*>(G)[e];
}

template <bool BF16>
__global__ void __launch_bounds__(kF32Threads, 1) ns_f32_kernel(const __grid_constant__ F32Launch L) {
    extern __shared__ float4 smem4[];
    float* Gs = reinterpret_cast<float*>(smem4);
    float* Ps = Gs + kBuf;
    float* Qs = Ps + kBuf;
    pdl_trigger();
    pdl_wait();   // momentum and 1/||U||_F of the previous kernels are complete from here on
    const int t = threadIdx.x;
    const int tx = t & 15, ty = t >> 4;
    const float mu = L.mu;
    for (int g = blockIdx.x; g < L.total; g += gridDim.x) {
        int p = 0;
        while (p + 1 < L.nprob && g >= L.prob[p + 1].item_begin) ++p;
        const F32Problem& P = L.prob[p];
        const int item = g - P.item_begin;
        const int mi = P.item_mat[item];
        const MatDev md = L.mats[mi];
        const int r = P.r, c = P.c;
        const long long ld = md.n;   // stored row length
        const bool tr = md.transposed != 0;
        const float* M = L.M[mi];
        const void* Gp = L.G[mi];
        float* W = L.W[mi];
        const float al = P.alpha[item];
        float acc[8][8];

        // ---- G0 = al^2 X X^T over 128-column chunks of X (k-major in Ps: Ps[k][i] = X[i][k0 + k])
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
        for (int k0 = 0; k0 < c; k0 += kDim) {
            const int kn = min(kDim, c - k0);
            for (int e = t; e < kDim * kDim; e += kF32Threads) {
                // stored rows are contiguous: run along the stored column index
                const int i = tr ? (e & (kDim - 1)) : (e >> 7);
                const int k = tr ? (e >> 7) : (e & (kDim - 1));
                float u = 0.f;
                if (i < r && k < kn) {
                    const long long idx = tr ? (long long)(k0 + k) * ld + i : (long long)i * ld + k0 + k;
                    u = fmaf(mu, M[idx], grad_at<BF16>(Gp, idx));
                }
                Ps[k * kLds + i] = u;
            }
            __syncthreads();
            mm_t<true>(Ps, Ps, kn, ty, tx, acc);
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] *= al * al;
        store_tile(Gs, r, ty, tx, acc);
        __syncthreads();

        // ---- J Gram steps
        const int J = P.ns_steps;
        const float ca = P.coef_a, cb = P.coef_b, cc = P.coef_c;
        for (int k = 1; k <= J; ++k) {
            mm_t<false>(Gs, Gs, r, ty, tx, acc);   // G^2
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int row = own(ty, i);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int col = own(tx, j);
                    acc[i][j] = cc * acc[i][j] + cb * Gs[row * kLds + col] + (row == col ? ca : 0.f);
                }
            }
            store_tile(Ps, r, ty, tx, acc);   // P_k (P_{k-1} is no longer read)
            if (k == 1) store_tile(Qs, r, ty, tx, acc);   // Q_1 = P_1
            __syncthreads();
            if (k >= 2) {   // Q_k = P_k Q_{k-1}, in place
                mm_t<false>(Ps, Qs, r, ty, tx, acc);
                __syncthreads();
                store_tile(Qs, r, ty, tx, acc);
            }
            if (k < J) {   // G_k = (G_{k-1} P_k) P_k, in place twice
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    mm_t<false>(Gs, Ps, r, ty, tx, acc);
                    __syncthreads();
                    store_tile(Gs, r, ty, tx, acc);
                    __syncthreads();
                }
            }
            __syncthreads();
        }
        if (J == 0) {   // Q_0 = I
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = own(ty, i) == own(tx, j) ? 1.f : 0.f;
            store_tile(Qs, r, ty, tx, acc);
            __syncthreads();
        }

        // ---- O = al Q X over 128-column chunks of X (Ps[k][j] = X[k][j0 + j]), fused update
        const float lr = L.lr, wd = L.wd, s = P.scale;
        float* Od = P.Odbg ? P.Odbg + (long long)item * r * c : nullptr;
        for (int j0 = 0; j0 < c; j0 += kDim) {
            const int jn = min(kDim, c - j0);
            for (int e = t; e < kDim * kDim; e += kF32Threads) {
                const int k = tr ? (e & (kDim - 1)) : (e >> 7);
                const int j = tr ? (e >> 7) : (e & (kDim - 1));
                float u = 0.f;
                if (k < r && j < jn) {
                    const long long idx = tr ? (long long)(j0 + j) * ld + k : (long long)k * ld + j0 + j;
                    u = fmaf(mu, M[idx], grad_at<BF16>(Gp, idx));
                }
                Ps[k * kLds + j] = u;
            }
            __syncthreads();
            mm_t<false>(Qs, Ps, r, ty, tx, acc);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int row = own(ty, i);
                if (row >= r) continue;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int col = own(tx, j);
                    if (col >= jn) continue;
                    const long long idx = tr ? (long long)(j0 + col) * ld + row : (long long)row * ld + j0 + col;
                    const float o = al * acc[i][j];
                    const float w = W[idx];
                    W[idx] = w - lr * (s * o + wd * w);
                    if (Od) Od[idx] = o;
                }
            }
            __syncthreads();   // Ps is restaged for the next chunk
        }
    }
}

}  // namespace

cudaError_t ns_f32_prepare() {
    cudaError_t e = cudaFuncSetAttribute(ns_f32_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kF32Smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(ns_f32_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kF32Smem);
}

cudaError_t ns_f32_launch(const F32Launch& L, int grid, cudaStream_t s) {
    if (L.total <= 0) return cudaSuccess;
    if (grid > L.total) grid = L.total;
    if (L.grad_bf16) return launch_pdl(ns_f32_kernel<true>, dim3(grid), dim3(kF32Threads), kF32Smem, s, L);
    return launch_pdl(ns_f32_kernel<false>, dim3(grid), dim3(kF32Threads), kF32Smem, s, L);
}

}  // namespace muon
