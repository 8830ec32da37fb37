// Fused Muon NS step for matrices with r <= 128 on sm_103a: one CTA per matrix
// (persistent), SYRK, the whole Gram recursion on shared-memory operands, and the
// final product with the fused weight update, in one launch.
//
// DMuon, "Gram Newton-Schulz": G0 = X0 X0^T, P_k = aI + bG + cG^2,
// Q_k = P_k Q_{k-1}, G_k = G_{k-1} P_k^2, O = Q_J X0; the Muon update
// W -= lr (0.2 sqrt(max(m, n)) O + wd W) (Moonlight blog, eq. (4)) is fused into
// the final product's epilogue.
#include "kernels.h"
#include "ptx.cuh"
#include "gemm_common.cuh"

namespace muon {

// One CTA runs the whole step of one matrix with r <= 128 (persistent over the
// matrices of the launch).  The SYRK streams X once in 128-column k-blocks; all
// 4J-3 r x r products run on operands kept in shared memory (128 x 128, 2-byte,
// 128-byte swizzled, row-major) with accumulators in TMEM; the final product
// streams X again in 128-column chunks into the fused W update.
//
// Every r x r product is a plain row-major product C = A B: A is read K-major and
// B MN-major from the same row-major layout, so no operand has to be stored
// symmetric and each epilogue thread writes only its own row.  Rows and columns
// beyond r are written as zero, so the padded recursion is block-diagonal and
// leaves rows < r unchanged.
//
// The W update of the final product goes through shared memory: each epilogue
// warp streams its 32 x 32 fp32 pieces of W in (two pieces ahead of the one it
// updates), updates them from the accumulator and writes them back.  With a W
// tensor map for the matrix (32 x 32 fp32 boxes, 128-byte swizzle: the staged
// piece layout) the pieces move by TMA tile loads and stores, one instruction
// per piece each way, the stores asynchronous; otherwise by cp.async and
// coalesced 16-byte stores.  The staging uses the r x r operand buffers, which
// the final product does not read; with one NS step the last on-chip epilogue
// still reads and writes them, so the epilogue warps meet before staging W, and
// every warp's stores have read its staging before the next matrix's epilogues
// write operands there.
constexpr int kSmallRing = 3;                       // X stream ring (SYRK k-blocks, final chunks)
constexpr int kSmallThreads = 320;                  // warp 0 TMA, warp 1 MMA + TMEM, warps 2-9 epilogue
constexpr int kSmallEpiWarps = 8;
constexpr int kWBufs = 3;                           // pieces in flight per epilogue warp
struct SmallCfg {
    static constexpr int SLOT = 32768;              // one 128-column k-block or chunk of X (bf16)
    static constexpr int MAT = 128 * 128 * 2;       // one 128 x 128 2-byte operand
    static constexpr int GS = kSmallRing * SLOT;    // G' (fp16)
    static constexpr int PS = GS + MAT;             // P (fp16)
    static constexpr int QS = PS + MAT;             // Q (fp16)
    static constexpr int TS = QS + MAT;             // T (fp16); then Q_J (bf16) for the final product
    static constexpr int STAGE = GS;                // W staging of the final phase: GS, PS, QS
    static constexpr int BAR = TS + MAT;
    static constexpr int WBAR = BAR + 256;          // per epilogue warp, one mbarrier per W buffer
    static constexpr int SMEM_BYTES = BAR + 512 + 1024;
};
static_assert(kSmallEpiWarps * kWBufs * 8 <= 256, "W buffer barriers");
static_assert(SmallCfg::SMEM_BYTES <= 232448, "fused kernel exceeds the shared memory of one CTA");
static_assert(kSmallEpiWarps * kWBufs * kWPiece <= 3 * SmallCfg::MAT, "W staging must fit in GS, PS, QS");

// byte offset of element (row, col) of a 128 x 128 2-byte operand in the
// 128-byte-swizzled layout: two 64-column atoms of 128 rows x 128 B.  Read
// K-major (A) it is the matrix; read MN-major (B) it is the same matrix.
__device__ __forceinline__ uint32_t op_off(int row, int col) {
    return (uint32_t)((col >> 6) * 16384 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) + ((col & 7) << 1));
}

// 32 values of row `row`, columns [col0, col0 + 32), into an operand buffer
// (fp16 saturating, or bf16); zero outside the r x r block.
template <bool BF16OUT>
__device__ __forceinline__ void op_store_row(uint8_t* buf, int row, int col0, int r, const float (&x)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = (row < r && col0 + 8 * q + e < r) ? x[8 * q + e] : 0.f;
        uint4 pk;
        if (BF16OUT)
            pk = make_uint4(pack_bf162(y[0], y[1]), pack_bf162(y[2], y[3]), pack_bf162(y[4], y[5]),
                            pack_bf162(y[6], y[7]));
        else
            pk = make_uint4(pack_half2(y[0], y[1]), pack_half2(y[2], y[3]), pack_half2(y[4], y[5]),
                            pack_half2(y[6], y[7]));
        *reinterpret_cast<uint4*>(buf + op_off(row, col0 + 8 * q)) = pk;
    }
}

__device__ __forceinline__ void op_load_row_half(const uint8_t* buf, int row, int col0, float (&g)[32]) {
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

// Epilogue of one on-chip step for this thread's row (TMEM lane = row), columns
// [c_begin, c_begin + 64).
__device__ __forceinline__ void small_step_epilogue(int step, int k, int J, const GemmProblem& P, int item,
                                                    uint8_t* smem, uint32_t tmem_row, int row, int c_begin) {
    const int r = P.M;
    for (int cc = c_begin; cc < c_begin + 64; cc += 32) {
        float v[32];
        if (step == kSmIdentity) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = (cc + j == row) ? 1.f : 0.f;
            op_store_row<true>(smem + SmallCfg::TS, row, cc, r, v);
            continue;
        }
        {
            uint32_t raw[32];
            tmem_ld32(tmem_row + cc, raw);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw[j]);
        }
        if (step == kSmSyrk) {
            const float al = P.alpha[item];
            const float sc = P.out_scale * al * al;
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= sc;
            op_store_row<false>(smem + SmallCfg::GS, row, cc, r, v);
        } else if (step == kSmPoly) {
            {
                float g[32];
                op_load_row_half(smem + SmallCfg::GS, row, cc, g);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    v[j] = P.coef_c * v[j] + P.coef_b * g[j] + ((cc + j == row) ? P.coef_a : 0.f);
            }
            op_store_row<false>(smem + SmallCfg::PS, row, cc, r, v);
            if (k == 1 && J > 1) op_store_row<false>(smem + SmallCfg::QS, row, cc, r, v);
            if (k == 1 && J == 1) op_store_row<true>(smem + SmallCfg::TS, row, cc, r, v);
        } else if (step == kSmPair) {
            // accumulator 0: Q' = P Q (k >= 2); accumulator 1: T = P P (k < J)
            if (k >= 2) {
                if (k < J)
                    op_store_row<false>(smem + SmallCfg::QS, row, cc, r, v);
                else
                    op_store_row<true>(smem + SmallCfg::TS, row, cc, r, v);
            }
            if (k < J) {
                uint32_t raw[32];
                tmem_ld32(tmem_row + 128 + cc, raw);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw[j]);
                op_store_row<false>(smem + SmallCfg::TS, row, cc, r, v);
            }
        } else {   // kSmGT: G'' = G' T
            op_store_row<false>(smem + SmallCfg::GS, row, cc, r, v);
        }
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
    uint64_t* stage_free = drain + 1;
    uint64_t* rr_free = stage_free + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rr_free + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint64_t* wbar = reinterpret_cast<uint64_t*>(smem + Cfg::WBAR);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int w = 0; w < kSmallEpiWarps * kWBufs; ++w) mbar_init(wbar + w, 1);
        for (int s = 0; s < kSmallRing; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(mma_done, 1);
        mbar_init(epi_done, kSmallEpiWarps);
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_full + b, 1);
            mbar_init(accf_empty + b, kSmallEpiWarps);
        }
        mbar_init(drain, 1);
        mbar_init(stage_free, kSmallEpiWarps);
        mbar_init(rr_free, kSmallEpiWarps);
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
    pdl_trigger();
    pdl_wait();   // the previous kernel of the stream is complete from here on

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer: per matrix, the SYRK k-blocks then the final chunks,
            // 128 columns of X (32 KB) per ring slot
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < L.total_tiles; t += gridDim.x) {
                int p = 0;
                while (p + 1 < L.nprob && t >= L.prob[p + 1].tile_begin) ++p;
                const GemmProblem& P = L.prob[p];
                const int item = t - P.tile_begin;
                const int nch = (P.N + 127) / 128;
                for (int q = 0; ok && q < 2 * nch; ++q, ++it) {
                    const uint32_t s = it % kSmallRing;
                    const uint32_t ph = (it / kSmallRing) & 1u;
                    if (!mbar_wait_idle(empty + s, ph ^ 1u, abort_flag, L.status, kStatusTimeoutProducer, false)) {
                        ok = false;
                        break;
                    }
                    uint8_t* slot = smem + s * Cfg::SLOT;
                    mbar_arrive_expect_tx(full + s, 32768);
                    if (q < nch) {
                        // SYRK k-block: X[:, 128q .. 128q + 127] K-major, two 64-column boxes
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            tma_load_3d(slot + j * 16384, &L.mapA[p], full + s, q * 128 + 64 * j, 0, item);
                    } else {
                        // final chunk: the same columns MN-major (two 64-column x 64-row boxes each)
                        const int n0 = (q - nch) * 128;
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
            const uint32_t id_h = idesc_make(false, 128, 128, false, true);    // fp16 r x r: B MN-major
            const uint32_t id_b = idesc_make(true, 128, 128, false, false);    // bf16 SYRK: X X^T
            const uint32_t id_f = idesc_make(true, 128, 128, false, true);     // bf16 final, B MN-major
            // 128 x 128 x 128 product A B of row-major smem operands: A K-major, B MN-major
            auto rr = [&](uint32_t a, uint32_t b, uint32_t d) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = sdesc_sw128(a + (kk >> 2) * 16384 + (kk & 3) * 32, 0, 1024);
                    const uint64_t bd = sdesc_sw128(b + kk * 2048, 16384, 1024);
                    mma_f16kind(d, ad, bd, id_h, kk != 0);
                }
            };
            auto finish_step = [&]() -> bool {   // commit, then wait for the epilogue of this step
                mma_commit(mma_done);
                const bool w =
                    mbar_wait_idle(epi_done, sc & 1u, abort_flag, L.status, kStatusTimeoutMma, false);
                ++sc;
                tc_fence_after();
                return w;
            };
            for (int t = blockIdx.x; ok && t < L.total_tiles; t += gridDim.x) {
                int p = 0;
                while (p + 1 < L.nprob && t >= L.prob[p + 1].tile_begin) ++p;
                const GemmProblem& P = L.prob[p];
                const int J = P.ns_steps;
                const int nch = (P.N + 127) / 128;
                // G0 = X X^T (A and B are the same staged k-block)
                for (int kb = 0; ok && kb < nch; ++kb, ++it) {
                    const uint32_t s = it % kSmallRing;
                    if (!mbar_wait_idle(full + s, (it / kSmallRing) & 1u, abort_flag, L.status, kStatusTimeoutMma,
                                        false)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = smem_u32(smem + s * Cfg::SLOT);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t d = sdesc_sw128(a + (kk >> 2) * 16384 + (kk & 3) * 32, 0, 1024);
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
                    if (!mbar_wait_idle(accf_empty + b, ((fc >> 1) & 1u) ^ 1u, abort_flag, L.status,
                                        kStatusTimeoutMma, false) ||
                        !mbar_wait_idle(full + (it % kSmallRing), (it / kSmallRing) & 1u, abort_flag, L.status,
                                        kStatusTimeoutMma, false)) {
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
        uint8_t* stage = smem + Cfg::STAGE + (warp - 2) * kWBufs * kWPiece;
        const uint32_t stage_u32 = smem_u32(stage);
        uint64_t* wb = wbar + kWBufs * (warp - 2);
        uint32_t wph = 0;    // phase bit per W buffer (TMA path)
        uint32_t wpend = 0;  // W loads in flight per buffer (TMA path)
        uint32_t sc = 0, fc = 0, mc = 0, jc = 0;
        bool ok = true;
        auto step = [&](int kind, int k, int J, const GemmProblem& P, int item) -> bool {
            if (!mbar_wait_idle(mma_done, sc & 1u, abort_flag, L.status, kStatusTimeoutEpilogue, false))
                return false;
            ++sc;
            tc_fence_after();
            small_step_epilogue(kind, k, J, P, item, smem, tmem_row, row, c_begin);
            fence_proxy_async_smem();   // operand writes visible to the tensor core
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
            if (ok && J == 1) {
                // the last on-chip epilogue (the polynomial) reads G' and writes P in the
                // buffers the W staging reuses: every warp leaves it before any stages W
                __syncwarp();
                if (lane == 0) mbar_arrive(rr_free);
                ok = mbar_wait_idle(rr_free, jc & 1u, abort_flag, L.status, kStatusTimeoutEpilogue, false);
                ++jc;
            }
            if (!ok) break;
            // Final product: this warp's pieces are (chunk ch, half h) at oriented rows
            // [32 wq, 32 wq + 32) and columns 128 ch + c_begin + 32 h; piece i lives in
            // staging buffer i % kWBufs, loaded kWBufs - 1 pieces ahead.
            const WPiece wc = w_piece_ctx(P, item);
            const int rw = wq * 32;
            const int npieces = 2 * nch;
            auto piece_col = [&](int i) { return (i >> 1) * 128 + c_begin + 32 * (i & 1); };
            const int mat = P.item_mat[item];
            const CUtensorMap* wm = (P.wmap != nullptr && rw < P.M && P.wmap_ok[mat]) ? P.wmap + mat : nullptr;
            if (wm != nullptr) {
                // TMA pieces: box coordinates in the stored layout; piece i in buffer i % kWBufs,
                // loaded kWBufs - 1 pieces ahead once the store of the piece before it has read
                // the buffer
                const bool wtr = P.transposed[mat] != 0;
                auto issue = [&](int i) {
                    const int c0 = piece_col(i), bs = i % kWBufs;
                    mbar_arrive_expect_tx(wb + bs, kWPiece);
                    tma_load_2d(stage + bs * kWPiece, wm, wb + bs, wtr ? rw : c0, wtr ? c0 : rw);
                };
#pragma unroll 1
                for (int i = 0; i < kWBufs - 1 && i < npieces; ++i) {
                    if (piece_col(i) >= P.N) continue;
                    if (lane == 0) issue(i);
                    wpend |= 1u << (i % kWBufs);
                }
#pragma unroll 1
                for (int i = 0; i < npieces; ++i) {
                    const int h = i & 1;
                    const uint32_t b = fc & 1u;
                    const int col0 = piece_col(i);
                    const int ahead = i + kWBufs - 1;
                    if (ahead < npieces && piece_col(ahead) < P.N) {
                        if (lane == 0) {
                            bulk_wait_read<0>();
                            issue(ahead);
                        }
                        wpend |= 1u << (ahead % kWBufs);
                    }
                    if (h == 0) {
                        if (!mbar_wait_idle(accf_full + b, (fc >> 1) & 1u, abort_flag, L.status,
                                            kStatusTimeoutEpilogue, false)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    uint32_t acc[32];
                    tmem_ld32(tmem_row + 256 + 128 * b + c_begin + 32 * h, acc);
                    tmem_ld_wait();
                    if (h == 1) {   // both halves read: the accumulator may be reused
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(accf_empty + b);
                        ++fc;
                    }
                    if (col0 < P.N) {
                        const int bs = i % kWBufs;
                        if (!mbar_wait_idle(wb + bs, (wph >> bs) & 1u, abort_flag, L.status, kStatusTimeoutEpilogue,
                                            false)) {
                            ok = false;
                            break;
                        }
                        wph ^= 1u << bs;
                        wpend &= ~(1u << bs);
                        uint8_t* buf = stage + bs * kWPiece;
                        w_piece_update(P, wc, item, rw, col0, buf, lane, acc);
                        fence_proxy_async_smem();   // the updated piece visible to the TMA store
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(wm, buf, wtr ? rw : col0, wtr ? col0 : rw);
                            bulk_commit();
                        }
                    }
                    __syncwarp();
                }
                if (lane == 0) bulk_wait_read<0>();   // the stores have read the staging
                __syncwarp();
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(stage_free);
                ok = mbar_wait_idle(stage_free, mc & 1u, abort_flag, L.status, kStatusTimeoutEpilogue, false);
                ++mc;
                continue;
            }
#pragma unroll 1
            for (int i = 0; i < kWBufs - 1; ++i) {
                if (i < npieces) w_piece_load(wc, rw, piece_col(i), stage_u32 + i * kWPiece, lane);
                else cp_async_commit();
            }
#pragma unroll 1
            for (int i = 0; i < npieces; ++i) {
                const int h = i & 1;
                const uint32_t b = fc & 1u;
                const int col0 = piece_col(i);
                const int ahead = i + kWBufs - 1;
                if (ahead < npieces) w_piece_load(wc, rw, piece_col(ahead), stage_u32 + (ahead % kWBufs) * kWPiece, lane);
                else cp_async_commit();
                if (h == 0) {
                    if (!mbar_wait_idle(accf_full + b, (fc >> 1) & 1u, abort_flag, L.status, kStatusTimeoutEpilogue,
                                        false)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                uint32_t acc[32];
                tmem_ld32(tmem_row + 256 + 128 * b + c_begin + 32 * h, acc);
                tmem_ld_wait();
                if (h == 1) {   // both halves read: the accumulator may be reused
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(accf_empty + b);
                    ++fc;
                }
                cp_async_wait<kWBufs - 1>();   // piece i has landed (this thread's copies) ...
                __syncwarp();                   // ... and every lane's
                uint8_t* buf = stage + (i % kWBufs) * kWPiece;
                if (col0 < P.N && rw < P.M) w_piece_update(P, wc, item, rw, col0, buf, lane, acc);
                __syncwarp();
                w_piece_store(wc, rw, col0, buf, lane);
                __syncwarp();                   // buffer free for the load issued kWBufs - 1 pieces on
            }
            cp_async_wait<0>();
            if (!ok) break;
            // the next matrix's epilogue writes operands over the staging of every warp:
            // all warps leave the final phase first
            __syncwarp();
            if (lane == 0) mbar_arrive(stage_free);
            ok = mbar_wait_idle(stage_free, mc & 1u, abort_flag, L.status, kStatusTimeoutEpilogue, false);
            ++mc;
        }
        cp_async_wait<0>();
        for (int k = 0; k < kWBufs; ++k)   // TMA W loads still in flight after an abort
            if (wpend & (1u << k)) mbar_drain(wb + k, (wph >> k) & 1u);
        if (lane == 0) bulk_wait<0>();     // TMA W stores complete before the CTA exits
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

cudaError_t ns_small_prepare() {
    return cudaFuncSetAttribute(ns_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SmallCfg::SMEM_BYTES);
}

cudaError_t ns_small_launch(const GemmLaunch& L, int grid, cudaStream_t s) {
    if (L.total_tiles <= 0) return cudaSuccess;
    if (grid > L.total_tiles) grid = L.total_tiles;
    return launch_pdl(ns_small_kernel, dim3(grid), dim3(kSmallThreads), SmallCfg::SMEM_BYTES, s, L);
}

}  // namespace muon
