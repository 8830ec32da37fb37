// RowNorm step for one matrix that allocates no device memory.
//
// Who needs it: callers that are not allowed to call cudaMalloc themselves or
// to have a library call it for them.  Typical cases are frameworks that own
// every device byte through their own pooling allocator (a stray cudaMalloc
// bypasses their accounting and can fail once the pool has reserved the
// device), processes running under a hard per-process memory budget, and
// latency-critical loops where cudaMalloc / cudaFree would implicitly
// synchronise the device.  The planned API (muon_plan_create) allocates its
// workspace once; this entry point instead uses a fixed scratch array that is
// part of the library image.
//
// Scratch: `g_rownorm_scratch`, a file-scope __device__ array of
// kNoAllocScratchFloats floats (4 MiB) that every GPU which loads the library
// keeps until the process exits; its device address is looked up on every
// call.  When m > n the RowNorm rows are the stored columns, so their norms need
// a second pass: per-slab column sums of U^2 and
// the per-column inverse norms are kept in this array.  Every scratch word a
// call reads is written earlier in the same call, so nothing has to be
// cleared between calls; calls that overlap on the GPU (different streams, or
// several host threads) share the array and race.
#include <cmath>

#include "../../include/muon.h"
#include "kernels.h"

namespace muon {
namespace {

constexpr long long kNoAllocScratchFloats = 1LL << 20;   // 4 MiB

static __device__ __align__(256) float g_rownorm_scratch[kNoAllocScratchFloats];

// Device address of the scratch array in the current context.  In host code the
// array's name is only a stand-in, so the kernels always receive this address.
// It is looked up on every call (a host-side query: no allocation, no
// synchronisation), so a context that was reset and re-created gets the array's
// new address; the first lookup on a device may load the library's device code.
cudaError_t scratch_address(float** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_rownorm_scratch);
    if (e != cudaSuccess) return e;
    *out = static_cast<float*>(p);
    return cudaSuccess;
}

template <bool BF16>
__device__ __forceinline__ float grad_at(const void* G, long long e) {
    if (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(G)[e]);
    return reinterpret_cast<const float*>(G)[e];
}

// m <= n: one block per stored row (the oriented rows); two passes over the
// row so any length works.  Same arithmetic as the planned RowNorm step.
template <bool BF16>
__global__ void __launch_bounds__(kElemThreads) nk_rows(const void* G, float* M, float* W, long long n, float mu,
                                                        float lr, float wd, float eps, float scale) {
    __shared__ float sred[33];
    const long long base = (long long)blockIdx.x * n;
    float ss = 0.f;
    for (long long j = threadIdx.x; j < n; j += kElemThreads) {
        const float g = grad_at<BF16>(G, base + j);
        const float m = mu * M[base + j] + g;
        M[base + j] = m;
        const float u = mu * m + g;
        ss += u * u;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) sred[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int i = 0; i < kElemThreads / 32; ++i) t += sred[i];
        sred[32] = t;
    }
    __syncthreads();
    const float k = scale / fmaxf(sqrtf(sred[32]), eps);
    for (long long j = threadIdx.x; j < n; j += kElemThreads) {
        const float u = mu * M[base + j] + grad_at<BF16>(G, base + j);
        const float w = W[base + j];
        W[base + j] = w - lr * (k * u + wd * w);
    }
}

// m > n, pass 1: momentum and per-slab column sums of U^2 into scratch.
template <bool BF16>
__global__ void __launch_bounds__(kElemThreads) nk_colstats(const void* G, float* M, long long m, long long n,
                                                            float mu, float* partials) {
    const long long tiles_j = (n + kElemThreads - 1) / kElemThreads;
    const long long slab = blockIdx.x / tiles_j;
    const long long j = (blockIdx.x % tiles_j) * kElemThreads + threadIdx.x;
    if (j >= n) return;
    const long long i0 = slab * kColSlab;
    const long long i1 = (i0 + kColSlab < m) ? i0 + kColSlab : m;
    float s = 0.f;
    for (long long i = i0; i < i1; ++i) {
        const long long e = i * n + j;
        const float g = grad_at<BF16>(G, e);
        const float mm = mu * M[e] + g;
        M[e] = mm;
        const float u = mu * mm + g;
        s += u * u;
    }
    partials[slab * n + j] = s;
}

// m > n, pass 2: inverse column norms (fixed slab order) into scratch.
__global__ void __launch_bounds__(kElemThreads) nk_colfinal(const float* partials, float* inv, long long m,
                                                            long long n, float eps) {
    const long long j = (long long)blockIdx.x * kElemThreads + threadIdx.x;
    if (j >= n) return;
    const long long slabs = (m + kColSlab - 1) / kColSlab;
    float s = 0.f;
    for (long long k = 0; k < slabs; ++k) s += partials[k * n + j];
    inv[j] = 1.f / fmaxf(sqrtf(s), eps);
}

// m > n, pass 3: the update with U recomputed from G and the new M.
template <bool BF16>
__global__ void __launch_bounds__(kElemThreads) nk_colapply(const void* G, const float* M, float* W, long long m,
                                                            long long n, const float* inv, float mu, float lr,
                                                            float wd, float scale) {
    const long long e = (long long)blockIdx.x * kElemThreads + threadIdx.x;
    if (e >= m * n) return;
    const long long j = e % n;
    const float u = mu * M[e] + grad_at<BF16>(G, e);
    const float w = W[e];
    W[e] = w - lr * (scale * inv[j] * u + wd * w);
}

template <bool BF16>
cudaError_t launch_all(float* W, const void* G, float* M, long long m, long long n, float lr, float wd, float mu,
                       float eps, float* scratch, cudaStream_t s) {
    const float scale = 0.2f * sqrtf((float)(m > n ? m : n));   // 0.2 sqrt(max(m, n)), blog eq. (4)
    if (m <= n) {
        nk_rows<BF16><<<(unsigned)m, kElemThreads, 0, s>>>(G, M, W, n, mu, lr, wd, eps, scale);
        return cudaGetLastError();
    }
    const long long slabs = (m + kColSlab - 1) / kColSlab;
    float* partials = scratch;
    float* inv = scratch + slabs * n;
    const long long tiles_j = (n + kElemThreads - 1) / kElemThreads;
    nk_colstats<BF16><<<(unsigned)(slabs * tiles_j), kElemThreads, 0, s>>>(G, M, m, n, mu, partials);
    nk_colfinal<<<(unsigned)tiles_j, kElemThreads, 0, s>>>(partials, inv, m, n, eps);
    nk_colapply<BF16><<<(unsigned)((m * n + kElemThreads - 1) / kElemThreads), kElemThreads, 0, s>>>(
        G, M, W, m, n, inv, mu, lr, wd, scale);
    return cudaGetLastError();
}

}  // namespace
}  // namespace muon

extern "C" muon_status muon_rownorm_matrix_noalloc(float* param, const void* grad, float* momentum, int64_t rows,
                                                   int64_t cols, muon_dtype grad_dtype, float lr, float wd,
                                                   float mu, float eps, void* stream) {
    using namespace muon;
    if (!param || !grad || !momentum || rows <= 0 || cols <= 0) return MUON_ERR_INVALID_ARG;
    if (grad_dtype != MUON_F32 && grad_dtype != MUON_BF16) return MUON_ERR_UNSUPPORTED;
    if (!std::isfinite(lr) || lr < 0.f || !std::isfinite(wd) || wd < 0.f || !std::isfinite(mu) || mu < 0.f ||
        mu >= 1.f || !std::isfinite(eps) || eps <= 0.f)
        return MUON_ERR_INVALID_ARG;
    if (rows > (1LL << 31) / 2 || cols > (1LL << 31) / 2) return MUON_ERR_UNSUPPORTED;
    if (rows > cols) {
        // scratch: ceil(rows / 64) slab sums per column + one inverse norm per column
        const long long need = ((rows + kColSlab - 1) / kColSlab) * cols + cols;
        if (need > kNoAllocScratchFloats) return MUON_ERR_UNSUPPORTED;
    }
    if ((long long)rows * cols / kElemThreads >= (1LL << 31)) return MUON_ERR_UNSUPPORTED;
    const size_t gsz = grad_dtype == MUON_BF16 ? 2 : 4;
    const uintptr_t w = reinterpret_cast<uintptr_t>(param), g = reinterpret_cast<uintptr_t>(grad),
                    mo = reinterpret_cast<uintptr_t>(momentum);
    const size_t numel = (size_t)rows * (size_t)cols;
    auto overlap = [](uintptr_t a, size_t na, uintptr_t b, size_t nb) { return a < b + nb && b < a + na; };
    if (overlap(w, numel * 4, mo, numel * 4) || overlap(w, numel * 4, g, numel * gsz) ||
        overlap(mo, numel * 4, g, numel * gsz))
        return MUON_ERR_INVALID_ARG;
    float* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return MUON_ERR_CUDA;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    e = grad_dtype == MUON_BF16 ? launch_all<true>(param, grad, momentum, rows, cols, lr, wd, mu, eps, scratch, s)
                                : launch_all<false>(param, grad, momentum, rows, cols, lr, wd, mu, eps, scratch, s);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return MUON_ERR_CUDA;
    }
    return MUON_OK;
}
