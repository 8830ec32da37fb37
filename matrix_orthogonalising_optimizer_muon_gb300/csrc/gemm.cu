// Batched, grouped tensor-core products of the Gram Newton-Schulz iteration on
// sm_103a: TMA-fed shared-memory pipeline, tcgen05.mma with the accumulator in
// TMEM, warp-specialised persistent CTAs.
//
// Products (DMuon, "Gram Newton-Schulz": the recursion runs on r x r matrices;
// SYRK-style symmetric products compute only the lower triangle):
//   G0 = alpha^2 * X X^T            bf16 x bf16 -> fp32, K = c     (kEpiSyrk, symmetric)
//   P  = aI + bG + c * (G G)        tf32 x tf32 -> fp32, K = r     (kEpiPoly, symmetric)
//   Q' = P Q,  T = P P,  G' = G T   tf32 x tf32 -> fp32, K = r     (kEpiPlain, symmetric)
//   O  = alpha * Q X                bf16 x bf16 -> fp32, K = r     (kEpiApply, fused update
//                                   W -= lr (0.2 sqrt(c) O + wd W), blog eq. (4))
// Every r x r product of commuting polynomials in G0 is symmetric, so all of
// them are lower-triangle products.  r x r outputs are stored already rounded
// to tf32 (nearest even) because the next product reads them as tf32 operands.
#include "kernels.h"
#include "ptx.cuh"

namespace muon {

template <bool TF32>
struct GemmCfg {
    static constexpr int BK = TF32 ? 32 : 64;            // one 128-byte swizzle row of K
    static constexpr int ESZ = TF32 ? 4 : 2;
    static constexpr int UK = TF32 ? 8 : 16;             // K of one tcgen05.mma
    static constexpr int A_BYTES = kBM * BK * ESZ;       // 16 KB
    static constexpr int B_BYTES = kBN * BK * ESZ;       // 32 KB
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int MN_CHUNK_BYTES = 64 * BK * ESZ; // one 64-wide MN-major chunk of B
    static constexpr int BAR_OFFSET = kStages * STAGE_BYTES;
    static constexpr int SMEM_BYTES = BAR_OFFSET + 256 + 1024;   // + barriers + alignment slack
};

size_t gemm_smem_bytes(bool tf32) {
    return tf32 ? GemmCfg<true>::SMEM_BYTES : GemmCfg<false>::SMEM_BYTES;
}

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

// ------------------------------------------------------------------ epilogues
__device__ __forceinline__ void store_sym(const GemmProblem& P, int item, int row, int col0, const float (&v)[32]) {
    // v[j] is element (row, col0 + j).  Lower part goes to (row, col), its
    // mirror to (col, row).  Rows beyond M are masked (their lanes still ran
    // the collective TMEM load).
    if (row >= P.M) return;
    float* C = P.C ? P.C + item * P.strideC : nullptr;
    float* C2 = P.C2 ? P.C2 + item * P.strideC : nullptr;
    __nv_bfloat16* Cb = P.Cb ? P.Cb + item * P.strideCb : nullptr;
    const bool full = (col0 + 31 <= row) && (col0 + 31 < P.N);
    if (full) {
        if (C) {
            float4* dst = reinterpret_cast<float4*>(C + (long long)row * P.ldc + col0);
#pragma unroll
            for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
        if (C2) {
            float4* dst = reinterpret_cast<float4*>(C2 + (long long)row * P.ldc + col0);
#pragma unroll
            for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
        if (Cb) {
            uint4* dst = reinterpret_cast<uint4*>(Cb + (long long)row * P.ldcb + col0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                __nv_bfloat162 h0 = __floats2bfloat162_rn(v[8 * q + 0], v[8 * q + 1]);
                __nv_bfloat162 h1 = __floats2bfloat162_rn(v[8 * q + 2], v[8 * q + 3]);
                __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * q + 4], v[8 * q + 5]);
                __nv_bfloat162 h3 = __floats2bfloat162_rn(v[8 * q + 6], v[8 * q + 7]);
                uint4 pk;
                pk.x = *reinterpret_cast<uint32_t*>(&h0);
                pk.y = *reinterpret_cast<uint32_t*>(&h1);
                pk.z = *reinterpret_cast<uint32_t*>(&h2);
                pk.w = *reinterpret_cast<uint32_t*>(&h3);
                dst[q] = pk;
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int col = col0 + j;
            if (col <= row && col < P.N) {
                if (C) C[(long long)row * P.ldc + col] = v[j];
                if (C2) C2[(long long)row * P.ldc + col] = v[j];
                if (Cb) Cb[(long long)row * P.ldcb + col] = __float2bfloat16_rn(v[j]);
            }
        }
    }
    // mirror: for fixed j the warp's lanes write consecutive rows of row `col`
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const int col = col0 + j;
        if (col < row && col < P.N) {
            if (C) C[(long long)col * P.ldc + row] = v[j];
            if (C2) C2[(long long)col * P.ldc + row] = v[j];
            if (Cb) Cb[(long long)col * P.ldcb + row] = __float2bfloat16_rn(v[j]);
        }
    }
}

__device__ __forceinline__ void epilogue_chunk(const GemmProblem& P, int item, int row, int col0,
                                               const uint32_t (&raw)[32]) {
    float v[32];
    if (P.epi == kEpiApply) {
        if (row >= P.M) return;
        const float al = P.alpha[item];
        const int mat = P.item_mat[item];
        float* W = P.W[mat];
        const bool tr = P.transposed[mat] != 0;
        float* O = P.Odbg ? P.Odbg + (long long)item * P.M * P.N : nullptr;
        const float lr = P.lr, wd = P.wd, s = P.scale;
        if (!tr) {
            // stored layout = oriented layout: element (row, col) at row * N + col
            const long long base = (long long)row * P.N + col0;
            const bool vec = (col0 + 31 < P.N) && ((P.N & 3) == 0) && ((reinterpret_cast<uintptr_t>(W) & 15) == 0);
            if (vec) {
                float4* w4 = reinterpret_cast<float4*>(W + base);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float4 w = w4[q];
                    const float o0 = al * __uint_as_float(raw[4 * q + 0]);
                    const float o1 = al * __uint_as_float(raw[4 * q + 1]);
                    const float o2 = al * __uint_as_float(raw[4 * q + 2]);
                    const float o3 = al * __uint_as_float(raw[4 * q + 3]);
                    w.x = w.x - lr * (s * o0 + wd * w.x);
                    w.y = w.y - lr * (s * o1 + wd * w.y);
                    w.z = w.z - lr * (s * o2 + wd * w.z);
                    w.w = w.w - lr * (s * o3 + wd * w.w);
                    w4[q] = w;
                    if (O) {
                        O[base + 4 * q + 0] = o0;
                        O[base + 4 * q + 1] = o1;
                        O[base + 4 * q + 2] = o2;
                        O[base + 4 * q + 3] = o3;
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    if (col0 + j < P.N) {
                        const float o = al * __uint_as_float(raw[j]);
                        const float w = W[base + j];
                        W[base + j] = w - lr * (s * o + wd * w);
                        if (O) O[base + j] = o;
                    }
                }
            }
        } else {
            // stored as c x r: oriented (row, col) lives at col * M + row; lanes
            // (consecutive rows) write consecutive addresses
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int col = col0 + j;
                if (col < P.N) {
                    const long long idx = (long long)col * P.M + row;
                    const float o = al * __uint_as_float(raw[j]);
                    const float w = W[idx];
                    W[idx] = w - lr * (s * o + wd * w);
                    if (O) O[idx] = o;
                }
            }
        }
        return;
    }
    if (P.epi == kEpiSyrk) {
        const float al = P.alpha[item];
        const float a2 = al * al;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = round_tf32(a2 * __uint_as_float(raw[j]));
    } else if (P.epi == kEpiPoly) {
        // P = a I + b G + c G^2; G read from the (tf32-valued) input
        float g[32];
        if (row < P.M) {
            const float* Grow = P.Gin + item * P.strideG + (long long)row * P.ldg + col0;
            if (col0 + 31 < P.N) {
                const float4* g4 = reinterpret_cast<const float4*>(Grow);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 t = g4[q];
                    g[4 * q] = t.x;
                    g[4 * q + 1] = t.y;
                    g[4 * q + 2] = t.z;
                    g[4 * q + 3] = t.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) g[j] = (col0 + j < P.N) ? Grow[j] : 0.f;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) g[j] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            float x = P.coef_c * __uint_as_float(raw[j]) + P.coef_b * g[j];
            if (col0 + j == row) x += P.coef_a;
            v[j] = round_tf32(x);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = round_tf32(__uint_as_float(raw[j]));
    }
    store_sym(P, item, row, col0, v);
}

// ------------------------------------------------------------------ kernel
template <bool TF32>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(const __grid_constant__ GemmLaunch L) {
    using Cfg = GemmCfg<TF32>;
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
            mbar_init(tempty + a, 4);
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
                const uint32_t idesc = idesc_make(TF32, kBM, kBN, false, P.b_mn != 0);
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
                        if (TF32)
                            mma_tf32(d_tmem, ad, bd, idesc, (kb | kk) != 0);
                        else
                            mma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0);
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
        // ---------------- epilogue: warps 2..5, TMEM lane quarter = warp % 4
        const int wq = warp & 3;
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
            for (int cc = 0; cc < kBN; cc += 32) {
                const int col0 = tc.n0 + cc;
                if (col0 >= P.N) break;                              // warp-uniform
                if (P.sym && col0 > warp_row_max) break;             // whole chunk above the diagonal
                uint32_t raw[32];
                tmem_ld32(tbase + cc, raw);
                tmem_ld_wait();
                epilogue_chunk(P, tc.item, row, col0, raw);
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

cudaError_t gemm_prepare(int device) {
    (void)device;
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         GemmCfg<false>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                GemmCfg<true>::SMEM_BYTES);
}

cudaError_t gemm_launch(const GemmLaunch& L, bool tf32, int grid, cudaStream_t s) {
    if (L.total_tiles <= 0) return cudaSuccess;
    if (grid > L.total_tiles) grid = L.total_tiles;
    if (tf32)
        gemm_kernel<true><<<grid, kGemmThreads, GemmCfg<true>::SMEM_BYTES, s>>>(L);
    else
        gemm_kernel<false><<<grid, kGemmThreads, GemmCfg<false>::SMEM_BYTES, s>>>(L);
    return cudaGetLastError();
}

}  // namespace muon
