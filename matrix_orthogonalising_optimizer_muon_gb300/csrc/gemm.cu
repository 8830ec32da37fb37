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
#include "gemm_common.cuh"

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

// ------------------------------------------------------------------ kernel
template <bool BF16>
__global__ void __maxnreg__(168) gemm_kernel(const __grid_constant__ GemmLaunch L) {
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
    pdl_trigger();
    pdl_wait();   // the previous kernel of the stream is complete from here on

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < L.total_tiles; t += gridDim.x) {
                const TileCoord tc = decode_tile(L, t);
                const GemmProblem& P = L.prob[tc.p];
                const int nkb = (P.K + Cfg::BK - 1) / Cfg::BK;
                const int kblocks = nkb * split_passes(P);
                for (int kbt = 0; kbt < kblocks; ++kbt, ++it) {
                    const uint32_t s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!mbar_wait_idle(empty + s, ph ^ 1u, abort_flag, L.status, kStatusTimeoutProducer, false)) {
                        ok = false;
                        break;
                    }
                    int kb, za, zb;   // split passes: the part of A and B this k-block reads
                    split_coords(P, kbt, nkb, tc.item, &kb, &za, &zb);
                    uint8_t* sa = smem + s * Cfg::STAGE_BYTES;
                    uint8_t* sb = sa + Cfg::A_BYTES;
                    mbar_arrive_expect_tx(full + s, Cfg::STAGE_BYTES);
                    tma_load_3d(sa, &L.mapA[tc.p], full + s, kb * Cfg::BK, tc.m0, za);
                    if (!P.b_mn) {
                        tma_load_3d(sb, &L.mapB[tc.p], full + s, kb * Cfg::BK, tc.n0, zb);
                    } else {
#pragma unroll
                        for (int q = 0; q < kBN / 64; ++q)
                            tma_load_3d(sb + q * Cfg::MN_CHUNK_BYTES, &L.mapB[tc.p], full + s, tc.n0 + 64 * q,
                                        kb * Cfg::BK, zb);
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
                const int kblocks = (P.K + Cfg::BK - 1) / Cfg::BK * split_passes(P);
                const uint32_t acc = local & 1;
                const uint32_t aph = (local >> 1) & 1u;
                if (!mbar_wait_idle(tempty + acc, aph ^ 1u, abort_flag, L.status, kStatusTimeoutMma, false)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * kBN;
                const uint32_t idesc = idesc_make(BF16, kBM, kBN, false, P.b_mn != 0);
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const uint32_t s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!mbar_wait_idle(full + s, ph, abort_flag, L.status, kStatusTimeoutMma, false)) {
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
            if (P.epi == kEpiApply || P.epi == kEpiPoly)
                prefetch_epilogue_inputs(P, tc.item, tc.m0 + wq * 32, tc.n0 + c_begin, kBN * 4 / kEpiWarps, lane);
            if (!mbar_wait_idle(tfull + acc, aph, abort_flag, L.status, kStatusTimeoutEpilogue, false)) break;
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
                    tmem_ld32(tbase + cc, raw);
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
    // per epilogue warp: 2 x 2 KB store staging, then 2 x 2 KB of the polynomial's G' blocks
    static constexpr int OUT_OFFSET = kStages2 * STAGE_BYTES;
    static constexpr int OUT_WARP = 8192;
    static constexpr int OUT_BYTES = kEpiWarps * OUT_WARP;
    static constexpr int BAR_OFFSET = OUT_OFFSET + OUT_BYTES;
    static constexpr int SMEM_BYTES = BAR_OFFSET + 512 + 1024;
};
static_assert(Gemm2Cfg::SMEM_BYTES <= 232448, "CTA-pair kernel exceeds the shared memory of one CTA");

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

// A k-block [k0, k0 + 64) of rows starting at `row0` of a lower-stored symmetric
// operand lies beyond the rows' 256-row diagonal tile: it is read from the mirror
// position (rows k0.., columns row0..), MN-major.
__device__ __forceinline__ bool upper_block(bool sym, int k0, int row0) {
    return sym && k0 >= (row0 & ~255) + 256;
}

// L2 prefetch of the polynomial's G' input for this CTA's part of a tile (rows m0 ..
// m0 + 127, columns n0 .. n0 + 255), issued by the producer when the tile's loads start:
// four tensor prefetches of the A operand's boxes (64 columns x 128 rows), in place of
// one bulk prefetch per row from the epilogue warps.  (The final product's W keeps the
// epilogue warps' row prefetches: the same through two 128 x 128 W boxes from the
// producer measured 5 % slower on that stage.)
template <bool LOWER>
__device__ __forceinline__ void tile_prefetch(const GemmLaunch& L, const GemmProblem& P, const TileCoord& tc) {
    if (tc.m0 >= P.M) return;
    if (P.epi == kEpiPoly) {
        for (int q = 0; q < 4 && tc.n0 + 64 * q < P.N; ++q) {
            if constexpr (LOWER) {
                tma_prefetch_4d(&L.mapA[tc.p], 0, tc.m0, (tc.n0 >> 6) + q, tc.item);
            } else {
                const int za = P.a_split ? 2 * tc.item : tc.item;
                tma_prefetch_3d(&L.mapA[tc.p], tc.n0 + 64 * q, tc.m0, za);
                if (P.a_split) tma_prefetch_3d(&L.mapA[tc.p], tc.n0 + 64 * q, tc.m0, za + 1);
            }
        }
    }
}

// LOWER = false: operands through 3-D maps, symmetric outputs stored whole.
// LOWER = true: every operand through a 4-D map of 64-column chunks, one box per
// operand per stage whichever way it is read (the map and the coordinates are
// selected per k-block, no branch around the TMA issue); symmetric outputs stored
// as their lower triangle (lower_out) and read back through the mirror (sym_a /
// sym_b).  The same MMAs on the same operand values in the same order: both give
// bitwise the same results.
// WTMA (bf16 only): final products whose every matrix has a W map move their W pieces by TMA;
// the cp.async path is compiled out of that instantiation and the TMA one out of the others,
// which keeps each within the 168 registers a 10-warp CTA gets.
template <bool BF16, bool LOWER, bool WTMA>
__global__ void __maxnreg__(168) gemm2_kernel(const __grid_constant__ GemmLaunch L) {
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
    uint64_t* gbar = reinterpret_cast<uint64_t*>(tmem_slot + 2);   // per epilogue warp: its two G' blocks

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t q = rank & 1u;      // CTA within the pair
    const uint32_t lead = 0;           // the even CTA: MMA issuer, owner of the full / tempty barriers
    const bool leader = q == 0;
    const int cluster_id = blockIdx.x >> 1;
    const int nclusters = gridDim.x >> 1;
    auto decode = [&](int t) { return decode_pair_tile(L, t, q); };

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
        for (int w = 0; w < 2 * kEpiWarps; ++w) mbar_init(gbar + w, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int p = 0; p < L.nprob; ++p) {
            tma_prefetch_desc(&L.mapA[p]);
            tma_prefetch_desc(&L.mapB[p]);
            if (LOWER && L.prob[p].sym_a) tma_prefetch_desc(&L.mapAt[p]);
            if (LOWER && (L.prob[p].sym_b || L.prob[p].b_mn)) tma_prefetch_desc(&L.mapBt[p]);
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
    pdl_trigger();
    pdl_wait();   // the previous kernel of the stream is complete from here on

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs)
            uint32_t it = 0;
            bool ok = true;
            for (int t = cluster_id; ok && t < L.total_tiles; t += nclusters) {
                const TileCoord tc = decode(t);
                const GemmProblem& P = L.prob[tc.p];
                const int nkb = (P.K + Cfg::BK - 1) / Cfg::BK;
                const int kblocks = LOWER ? nkb : nkb * split_passes(P);
                tile_prefetch<LOWER>(L, P, tc);
                // lower-triangle launches: the problem's fields and maps read once per tile
                const bool sym_a = P.sym_a != 0, sym_b = P.sym_b != 0, bmn = P.b_mn != 0;
                const CUtensorMap* mA = &L.mapA[tc.p];
                const CUtensorMap* mAt = &L.mapAt[tc.p];
                const CUtensorMap* mB = &L.mapB[tc.p];
                const CUtensorMap* mBt = &L.mapBt[tc.p];
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const uint32_t s = it % kStages2;
                    const uint32_t ph = (it / kStages2) & 1u;
                    if (!mbar_wait_idle(empty + s, ph ^ 1u, abort_flag, L.status, kStatusTimeoutProducer, true)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + s * Cfg::STAGE_BYTES;
                    uint8_t* sb = sa + Cfg::A_BYTES;
                    const uint32_t fb = mapa_shared(smem_u32(full + s), lead);
                    if (leader) mbar_arrive_expect_tx(full + s, 2 * Cfg::STAGE_BYTES);
                    const int nb = tc.n0 + 128 * (int)q;
                    if constexpr (LOWER) {
                        // one 4-D box per operand: K-major at (0, row, kb) or the mirror at (0, k0, row / 64)
                        const int k0 = kb * Cfg::BK;
                        const bool at = upper_block(sym_a, k0, tc.m0);
                        const bool bt = bmn || upper_block(sym_b, k0, tc.n0);
                        tma_load_4d_pair(sa, at ? mAt : mA, fb, 0, at ? k0 : tc.m0, at ? (tc.m0 >> 6) : kb, tc.item);
                        tma_load_4d_pair(sb, bt ? mBt : mB, fb, 0, bt ? k0 : nb, bt ? (nb >> 6) : kb, tc.item);
                        continue;
                    }
                    int kr, za, zb;   // split passes: the part of A and B this k-block reads
                    split_coords(P, kb, nkb, tc.item, &kr, &za, &zb);
                    tma_load_3d_pair(sa, &L.mapA[tc.p], fb, kr * Cfg::BK, tc.m0, za);
                    if (!P.b_mn) {
                        tma_load_3d_pair(sb, &L.mapB[tc.p], fb, kr * Cfg::BK, nb, zb);
                    } else {
                        tma_load_3d_pair(sb, &L.mapB[tc.p], fb, nb, kr * Cfg::BK, zb);
                        tma_load_3d_pair(sb + Cfg::MN_CHUNK_BYTES, &L.mapB[tc.p], fb, nb + 64, kr * Cfg::BK, zb);
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
                const TileCoord tc = decode(t);
                const GemmProblem& P = L.prob[tc.p];
                const int kblocks = (P.K + Cfg::BK - 1) / Cfg::BK * (LOWER ? 1 : split_passes(P));
                const uint32_t acc = local & 1;
                const uint32_t aph = (local >> 1) & 1u;
                if (!mbar_wait_idle(tempty + acc, aph ^ 1u, abort_flag, L.status, kStatusTimeoutMma, true)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * kBN;
                const uint32_t idesc = idesc_make(BF16, 256, kBN, false, P.b_mn != 0);
                // lower-triangle launches: k-block where A / B switch to the mirror (MN-major)
                const int a_sw = P.sym_a ? ((tc.m0 & ~255) + 256) / Cfg::BK : 1 << 30;
                const int b_sw = P.b_mn ? 0 : (P.sym_b ? ((tc.n0 & ~255) + 256) / Cfg::BK : 1 << 30);
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const uint32_t s = it % kStages2;
                    const uint32_t ph = (it / kStages2) & 1u;
                    if (!mbar_wait_idle(full + s, ph, abort_flag, L.status, kStatusTimeoutMma, true)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + s * Cfg::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + Cfg::A_BYTES;
                    if constexpr (LOWER) {
                        const bool a_mn = kb >= a_sw, b_mn = kb >= b_sw;
                        const uint32_t id = idesc_make(BF16, 256, kBN, a_mn, b_mn);
#pragma unroll
                        for (int kk = 0; kk < Cfg::BK / Cfg::UK; ++kk) {
                            constexpr int MN = Cfg::MN_CHUNK_BYTES;
                            const uint64_t ad = a_mn ? sdesc_sw128(a_addr + kk * Cfg::UK * 128, MN, 1024)
                                                     : sdesc_sw128(a_addr + kk * Cfg::UK * Cfg::ESZ, 0, 1024);
                            const uint64_t bd = b_mn ? sdesc_sw128(b_addr + kk * Cfg::UK * 128, MN, 1024)
                                                     : sdesc_sw128(b_addr + kk * Cfg::UK * Cfg::ESZ, 0, 1024);
                            mma_f16kind_pair(d_tmem, ad, bd, id, (kb | kk) != 0);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < Cfg::BK / Cfg::UK; ++kk) {
                            const uint64_t ad = sdesc_sw128(a_addr + kk * Cfg::UK * Cfg::ESZ, 0, 1024);
                            const uint64_t bd =
                                P.b_mn ? sdesc_sw128(b_addr + kk * Cfg::UK * 128, Cfg::MN_CHUNK_BYTES, 1024)
                                       : sdesc_sw128(b_addr + kk * Cfg::UK * Cfg::ESZ, 0, 1024);
                            mma_f16kind_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0);
                        }
                    }
                    mma_commit_pair(empty + s, 0x3);   // frees the stage in both CTAs
                }
                if (!ok) break;
                mma_commit_pair(tfull + acc, (uint16_t)(3u << lead));   // both CTAs' accumulators ready
            }
            mma_commit_pair(drain, (uint16_t)(1u << rank));
            mbar_drain(drain, 0);
        }
    } else {
        // ---------------- epilogue of both CTAs, each on its own TMEM: lane quarter =
        // warp % 4; warps 2-5 take columns 0-127 of the tile, warps 6-9 columns 128-255
        const int wq = warp & 3;
        const int c_begin = ((warp - 2) >> 2) * (kBN * 4 / kEpiWarps);
        const uint32_t tempty_leader = mapa_shared(smem_u32(tempty), lead);
        uint8_t* stage_l = smem + Cfg::OUT_OFFSET + (warp - 2) * Cfg::OUT_WARP;
        uint8_t* gin_buf = stage_l + 4096;            // two 2 KB blocks of G'
        uint64_t* gb = gbar + 2 * (warp - 2);
        uint32_t gph = 0;                             // phase bit per G' buffer (bits 0, 1)
        uint32_t gpend = 0;                           // G' loads in flight (bits 0, 1)
        int local = 0;
        for (int t = cluster_id; t < L.total_tiles; t += nclusters, ++local) {
            const TileCoord tc = decode(t);
            const GemmProblem& P = L.prob[tc.p];
            const uint32_t acc = local & 1;
            const uint32_t aph = (local >> 1) & 1u;
            if (BF16 && P.epi == kEpiApply)   // (the polynomial's G' is prefetched by the producer)
                prefetch_epilogue_inputs(P, tc.item, tc.m0 + wq * 32, tc.n0 + c_begin, kBN * 4 / kEpiWarps, lane);
            // Final product with a W map: this warp's W pieces (rows R0w .. R0w + 31, its 32-column
            // chunks) come by TMA into two 4 KB buffers (the shared memory the symmetric stores and
            // the G' blocks use in other launches), the first two while the MMAs run, each next one
            // once the previous store from its buffer has read it; box coordinates are those of
            // the stored layout.  wn: the pieces this warp processes.
            const CUtensorMap* wm = nullptr;
            bool wtr = false;
            int wn = 0;
            const int R0w = tc.m0 + wq * 32;
            if (WTMA && P.epi == kEpiApply) {   // (the host launches WTMA only when every map is valid)
                const int mat = P.item_mat[tc.item];
                if (R0w < P.M) {
                    wm = &P.wmap[mat];
                    wtr = P.transposed[mat] != 0;
                    while (wn < 4 && tc.n0 + c_begin + 32 * wn < P.N) ++wn;
                    if (lane == 0 && wn > 0) bulk_wait_read<0>();   // earlier stores have read the buffers
                    for (int k = 0; k < 2 && k < wn; ++k) {
                        if (lane == 0) {
                            const int c0 = tc.n0 + c_begin + 32 * k;
                            mbar_arrive_expect_tx(gb + k, kWPiece);
                            tma_load_2d(stage_l + 4096 * k, wm, gb + k, wtr ? R0w : c0, wtr ? c0 : R0w);
                        }
                        gpend |= 1u << k;
                    }
                }
            }
            // The polynomial's G' blocks (rows R0 .. R0 + 31, this warp's 32-column chunks) come
            // by TMA into the warp's two G' buffers, the first two while the MMAs run, each next
            // one as soon as its buffer has been read.  gn: the chunks this warp processes.
            int gn = 0;
            const bool gt = !BF16 && P.epi == kEpiPoly && P.gin_tma;
            if (gt) {
                const int wrmax = tc.m0 + wq * 32 + 31;
                while (gn < 4 && tc.n0 + c_begin + 32 * gn < P.N && tc.n0 + c_begin + 32 * gn <= wrmax) ++gn;
                for (int k = 0; k < 2 && k < gn; ++k) {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(gb + k, 2048);
                        tma_load_3d(gin_buf + 2048 * k, &L.mapG[tc.p], gb + k, tc.n0 + c_begin + 32 * k,
                                    tc.m0 + wq * 32, tc.item);
                    }
                    gpend |= 1u << k;
                }
            }
            if (!mbar_wait_idle(tfull + acc, aph, abort_flag, L.status, kStatusTimeoutEpilogue, true)) break;
            tc_fence_after();
            const int row = tc.m0 + wq * 32 + lane;
            const int warp_row_max = tc.m0 + wq * 32 + 31;
            const uint32_t tbase = tmem_base + acc * kBN + (static_cast<uint32_t>(wq * 32) << 16);
            // fp16 launches carry only r x r products (kEpiPoly, kEpiPlain); the final product's
            // W pieces exist in the bf16 instantiations alone
            const WPiece wc = w_piece_ctx(P, BF16 && P.epi == kEpiApply ? tc.item : -1);
            bool gabort = false;
            for (int cc = c_begin, kc = 0; cc < c_begin + kBN * 4 / kEpiWarps; cc += 32, ++kc) {
                const int col0 = tc.n0 + cc;
                if (col0 >= P.N) break;
                if (P.sym && col0 > warp_row_max) break;
                uint32_t raw[32];
                if (WTMA && P.epi == kEpiApply) {   // this chunk's W piece (chunk kc, buffer kc % 2)
                    if (wm == nullptr) break;       // rows beyond the matrix: no pieces
                    const uint32_t bsel = kc & 1;
                    if (!mbar_wait_idle(gb + bsel, (gph >> bsel) & 1u, abort_flag, L.status, kStatusTimeoutEpilogue,
                                        false)) {
                        gabort = true;
                        break;
                    }
                    gph ^= 1u << bsel;
                    gpend &= ~(1u << bsel);
                    uint8_t* wbuf = stage_l + 4096 * bsel;
                    tmem_ld32(tbase + cc, raw);
                    tmem_ld_wait();
                    w_piece_update(P, wc, tc.item, R0w, col0, wbuf, lane, raw);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // updates visible to TMA
                    __syncwarp();
                    const bool more = kc + 2 < wn;
                    if (lane == 0) {
                        tma_store_2d(wm, wbuf, wtr ? R0w : col0, wtr ? col0 : R0w);
                        bulk_commit();
                        if (more) {
                            const int c2 = col0 + 64;
                            bulk_wait_read<0>();   // the store has read the piece: its buffer is free
                            mbar_arrive_expect_tx(gb + bsel, kWPiece);
                            tma_load_2d(wbuf, wm, gb + bsel, wtr ? R0w : c2, wtr ? c2 : R0w);
                        }
                    }
                    if (more) gpend |= 1u << bsel;
                    __syncwarp();
                    continue;
                }
                if (BF16 && !WTMA && P.epi == kEpiApply) {
                    // W piece (rows R0.., columns col0..) in with coalesced cp.async, updated
                    // in shared memory, out with coalesced 16-byte stores
                    const int R0 = tc.m0 + wq * 32;
                    w_piece_load(wc, R0, col0, smem_u32(stage_l), lane);
                    tmem_ld32(tbase + cc, raw);
                    tmem_ld_wait();
                    cp_async_wait<0>();
                    __syncwarp();
                    if (R0 < P.M) w_piece_update(P, wc, tc.item, R0, col0, stage_l, lane, raw);
                    __syncwarp();
                    w_piece_store(wc, R0, col0, stage_l, lane);
                    __syncwarp();
                    continue;
                }
                if (P.tma_out) {
                    const uint8_t* gin_s = nullptr;
                    if (!BF16 && gt) {   // this chunk's G' block (chunk kc, buffer kc % 2)
                        const uint32_t bsel = kc & 1;
                        if (!mbar_wait_idle(gb + bsel, (gph >> bsel) & 1u, abort_flag, L.status, kStatusTimeoutEpilogue,
                                            false)) {
                            gabort = true;
                            break;
                        }
                        gph ^= 1u << bsel;
                        gpend &= ~(1u << bsel);
                        gin_s = gin_buf + 2048 * bsel;
                    }
                    tmem_ld32(tbase + cc, raw);
                    tmem_ld_wait();
                    epilogue_chunk_tma(P, &L.mapC[tc.p], &L.mapC2[tc.p], tc.item, tc.m0 + wq * 32, col0, lane, raw,
                                       stage_l, stage_l + 2048, gin_s);
                    if (!BF16 && gt && kc + 2 < gn) {   // every lane has read the block: load chunk kc + 2 into it
                        const uint32_t bsel = kc & 1;
                        __syncwarp();
                        if (lane == 0) {
                            mbar_arrive_expect_tx(gb + bsel, 2048);
                            tma_load_3d(gin_buf + 2048 * bsel, &L.mapG[tc.p], gb + bsel, col0 + 64, tc.m0 + wq * 32,
                                        tc.item);
                        }
                        gpend |= 1u << bsel;
                    }
                } else {
                    tmem_ld32(tbase + cc, raw);
                    tmem_ld_wait();
                    epilogue_chunk(P, tc.item, row, col0, raw);
                }
            }
            if (gabort) break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader)
                    mbar_arrive(tempty + acc);
                else
                    mbar_arrive_remote(tempty_leader + acc * 8);
            }
        }
        for (int k = 0; k < 2; ++k)   // G' loads still in flight after an abort
            if (gpend & (1u << k)) mbar_drain(gb + k, (gph >> k) & 1u);
        if (lane == 0) bulk_wait<0>();   // TMA stores of the staging complete before the CTA exits
    }

    tc_fence_before();
    cluster_sync();   // all pair MMAs done and both TMEMs drained
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, 2 * kBN);
    }
}

cudaError_t gemm_prepare(int device) {
    (void)device;
    cudaError_t e =
        cudaFuncSetAttribute(gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, GemmCfg::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 GemmCfg::SMEM_BYTES);
    const int n = Gemm2Cfg::SMEM_BYTES;
    const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gemm2_kernel<true, false, false>, a, n);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gemm2_kernel<false, false, false>, a, n);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gemm2_kernel<true, true, false>, a, n);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gemm2_kernel<false, true, false>, a, n);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gemm2_kernel<true, false, true>, a, n);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gemm2_kernel<true, true, true>, a, n);
    if (e == cudaSuccess) e = ns_small_prepare();
    return e;
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
    return cudaOccupancyMaxActiveClusters(out, gemm2_kernel<true, false, false>, &cfg);
}

cudaError_t gemm2_launch(const GemmLaunch& L, bool bf16, int clusters, cudaStream_t s, bool lower, bool wtma) {
    if (L.total_tiles <= 0) return cudaSuccess;
    if (clusters > L.total_tiles) clusters = L.total_tiles;
    if (clusters < 1) clusters = 1;
    const dim3 grid(2 * clusters), blk(kGemmThreads);
    const size_t sm = Gemm2Cfg::SMEM_BYTES;
    if (bf16 && wtma)
        return lower ? launch_pdl_cluster(gemm2_kernel<true, true, true>, grid, blk, sm, s, 2u, L)
                     : launch_pdl_cluster(gemm2_kernel<true, false, true>, grid, blk, sm, s, 2u, L);
    if (lower)
        return bf16 ? launch_pdl_cluster(gemm2_kernel<true, true, false>, grid, blk, sm, s, 2u, L)
                    : launch_pdl_cluster(gemm2_kernel<false, true, false>, grid, blk, sm, s, 2u, L);
    return bf16 ? launch_pdl_cluster(gemm2_kernel<true, false, false>, grid, blk, sm, s, 2u, L)
                : launch_pdl_cluster(gemm2_kernel<false, false, false>, grid, blk, sm, s, 2u, L);
}

cudaError_t gemm_launch(const GemmLaunch& L, bool bf16, int grid, cudaStream_t s) {
    if (L.total_tiles <= 0) return cudaSuccess;
    if (grid > L.total_tiles) grid = L.total_tiles;
    if (bf16)
        return launch_pdl(gemm_kernel<true>, dim3(grid), dim3(kGemmThreads), GemmCfg::SMEM_BYTES, s, L);
    else
        return launch_pdl(gemm_kernel<false>, dim3(grid), dim3(kGemmThreads), GemmCfg::SMEM_BYTES, s, L);
}

}  // namespace muon