// The stream-ordered launch sequence of the Muon step (include/muon.h: muon_step,
// muon_step_ex, muon_step_host, the RowNorm steps).  Host code only; the kernels live in
// gemm.cu, ns_small.cu, ns_f32.cu and elementwise.cu.
//
// Step (mode NS), per plan, every kernel grouped over all matrices:
//   momentum (m <= n)  |  momentum + transpose (m > n)  |  1/||U||_F
//   G0 = a^2 X X^T                                         (one launch, all buckets)
//   k = 1..J:  P = aI + bG + cG^2;  {Q' = P Q, T = P P};  G' = G T
//   O = a Q X fused with W -= lr (0.2 sqrt(c) O + wd W)    (one launch, all buckets)
// (Gram Newton-Schulz from DMuon's technical summary; coefficients, Nesterov
// input, normalisation and eq. (4) from the "Muon is Scalable" blog summary;
// orientation and RowNorm from the DiT paper sec. 3.1.)
#include "plan.h"

namespace {

// 4-D maps of one operand for lower-triangle launches.
struct Maps4 {
    const CUtensorMap* k = nullptr;   // K-major boxes (64, 128, 1, 1)
    const CUtensorMap* t = nullptr;   // mirror / MN-major boxes (64, 64, 2, 1)
    bool sym = false;                 // a symmetric buffer stored as its lower triangle
};

// Collects problems into grouped launches of up to kMaxProblems.
struct Grouper {
    muon_plan_s* p;
    cudaStream_t s;
    bool bf16;
    bool lower;         // lower-triangle launches (the chunk's Chunk::lower)
    bool wtma = false;  // final products whose every matrix has a W map: W pieces by TMA
    int clusters = 0;   // CTA pairs for the pair kernel, CTAs for the one-SM kernel
    int grid1 = 0;
    GemmLaunch L1;   // 1-SM kernel, 128 x 256 tiles
    GemmLaunch L2;   // CTA-pair kernel, 256 x 256 tiles
    muon_status st = MUON_OK;
    int launches = 0;
    Grouper(muon_plan_s* plan, cudaStream_t stream, bool is_bf16, bool lower_tri, int pair_clusters, int sm_grid)
        : p(plan), s(stream), bf16(is_bf16), lower(lower_tri), clusters(pair_clusters), grid1(sm_grid) {
        reset(L1);
        reset(L2);
    }
    void reset(GemmLaunch& L) {
        std::memset(&L, 0, sizeof(L));
        L.status = p->status;
    }
    static void push(GemmLaunch& L, const CUtensorMap& a, const CUtensorMap& b, GemmProblem q) {
        q.tile_begin = L.total_tiles;
        L.mapA[L.nprob] = a;
        L.mapB[L.nprob] = b;
        L.prob[L.nprob] = q;
        L.nprob++;
        L.total_tiles += q.tiles_per_item * q.batch;
    }
    // a128: A with 128-row boxes; b256 / b128: B with 256- / 128-row boxes (the
    // same map for an MN-major B).  Problems with more than 128 rows go to the
    // CTA-pair kernel (each CTA loads 128 rows of A and 128 of B).
    // oc / oc2: store maps of a symmetric problem's outputs (tma_out set by the
    // caller); the pair kernel then writes them with TMA stores.
    // a4 / b4: the operands' 4-D maps, used by lower-triangle launches (B of an
    // MN-major problem through b4.t).
    // og: for a polynomial product, the store map of its G' input (32 x 32 boxes), through
    // which the pair kernel's epilogue loads G' by TMA.
    void add(const CUtensorMap& a128, const CUtensorMap& b256, const CUtensorMap& b128, GemmProblem q,
             const CUtensorMap* oc, const CUtensorMap* oc2, Maps4 a4, Maps4 b4, const CUtensorMap* og = nullptr) {
        if (q.a_split || q.b_split || q.out_split) q.tma_out = 0;   // split parts: per-thread stores
        q.gin_tma = 0;
        if (q.M > kBM && p->pair_clusters > 0) {
            if (L2.nprob == kMaxProblems) flush2();
            q.tiles_m = (int)ceil_div(q.M, 256);
            q.tiles_n = (int)ceil_div(q.N, 256);
            q.tiles_per_item = q.sym ? q.tiles_m * (q.tiles_m + 1) / 2 : q.tiles_m * q.tiles_n;
            if (!q.sym || !oc || ((q.tma_out & kTmaOutC2) && !oc2)) q.tma_out = 0;
            if (q.tma_out) {
                L2.mapC[L2.nprob] = *oc;
                if (oc2) L2.mapC2[L2.nprob] = *oc2;
                if (og && q.epi == kEpiPoly) {
                    L2.mapG[L2.nprob] = *og;
                    q.gin_tma = 1;
                }
            }
            if (lower) {
                q.lower_out = q.sym;
                q.sym_a = a4.sym;
                q.sym_b = b4.sym && !q.b_mn;
                L2.mapAt[L2.nprob] = a4.t ? *a4.t : *a4.k;
                L2.mapBt[L2.nprob] = b4.t ? *b4.t : *b4.k;
                push(L2, *a4.k, b4.k ? *b4.k : *b4.t, q);
            } else {
                push(L2, a128, b128, q);
            }
        } else {
            if (L1.nprob == kMaxProblems) flush1();
            q.tma_out = 0;
            push(L1, a128, b256, q);
        }
    }
    void flush1() {
        if (L1.nprob == 0) return;
        if (st == MUON_OK) {
            st = cuda_status(gemm_launch(L1, bf16, grid1, s));
            ++launches;
        }
        reset(L1);
    }
    void flush2() {
        if (L2.nprob == 0) return;
        if (st == MUON_OK) {
            st = cuda_status(gemm2_launch(L2, bf16, clusters, s, lower, wtma));
            ++launches;
        }
        reset(L2);
    }
    void flush() {
        flush2();
        flush1();
    }
};


}  // namespace

extern "C" {

// The RowNorm kernels over one set of lists (m <= n rows; m > n column statistics,
// finalize, apply).
static muon_status rownorm_launch(muon_plan_s* p, const ListDev* rows, const ListDev& stats,
                                  const ListDev& fin, const ListDev& apply, float lr, float wd, float mu, float eps,
                                  cudaStream_t s, int* launches) {
    ElemArgs a{};
    for (int cl = 0; cl < kRowClasses; ++cl) {
        a = elem_args(p, rows[cl], mu, lr, wd, eps);
        MUON_TRY(launch_rownorm_rows(a, rows[cl].blocks, rownorm_class_vec(cl), s));
        *launches += rows[cl].blocks > 0;
    }
    a = elem_args(p, stats, mu, lr, wd, eps);
    a.partials = p->cpartials;
    MUON_TRY(launch_rownorm_colstats(a, stats.blocks, s));
    a = elem_args(p, fin, mu, lr, wd, eps);
    a.partials = p->cpartials;
    MUON_TRY(launch_rownorm_colfinal(a, fin.blocks, s));
    a = elem_args(p, apply, mu, lr, wd, eps);
    MUON_TRY(launch_rownorm_colapply(a, apply.blocks, s));
    *launches += stats.blocks > 0 ? 3 : 0;
    return MUON_OK;
}

muon_status muon_rownorm_step(muon_plan p, float* const* params, const void* const* grads, float* const* momentum,
                              float lr, float wd, float mu, float eps, void* stream) {
    if (!p) return MUON_ERR_INVALID_ARG;
    if (!p->full_rows.empty()) return MUON_ERR_UNSUPPORTED;   // the shard calls sum norms across shards
    if (!finite_nonneg(lr) || !finite_nonneg(wd) || !std::isfinite(mu) || mu < 0.f || mu >= 1.f ||
        !std::isfinite(eps) || eps <= 0.f)
        return MUON_ERR_INVALID_ARG;
    muon_status st = check_pointers(p, params, grads, momentum);
    if (st != MUON_OK) return st;
    if ((st = check_device(p)) != MUON_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = upload_pointers(p, params, grads, momentum, s)) != MUON_OK) return st;
    muon_plan_s::StepEvents* se = nullptr;
    if (p->opts.timing && !(se = next_events(p))) return MUON_ERR_CUDA;
    if (se) {
        se->ns = false;
        MUON_TRY(cudaEventRecord(se->e[0], s));
    }
    int launches = 0;
    if ((st = rownorm_launch(p, p->rn_rows, p->rn_stats, p->rn_final, p->rn_apply, lr, wd, mu, eps, s,
                             &launches)) != MUON_OK)
        return st;
    if (se) MUON_TRY(cudaEventRecord(se->e[5], s));
    p->last_launches = launches;
    return MUON_OK;
}

// Checks shared by the two shard calls.
static muon_status shard_check(muon_plan_s* p, float* const* params, const void* const* grads,
                               float* const* momentum, float lr, float wd, float mu, float eps, const void* colsq) {
    if (!p) return MUON_ERR_INVALID_ARG;
    if (p->full_rows.empty()) return MUON_ERR_UNSUPPORTED;
    if (!finite_nonneg(lr) || !finite_nonneg(wd) || !std::isfinite(mu) || mu < 0.f || mu >= 1.f ||
        !std::isfinite(eps) || eps <= 0.f || (p->colsq_len > 0 && !colsq))
        return MUON_ERR_INVALID_ARG;
    muon_status st = check_pointers(p, params, grads, momentum);
    if (st != MUON_OK) return st;
    return check_device(p);
}

muon_status muon_rownorm_shard_stats(muon_plan p, float* const* params, const void* const* grads,
                                     float* const* momentum, float lr, float wd, float mu, float eps, float* colsq,
                                     void* stream) {
    muon_status st = shard_check(p, params, grads, momentum, lr, wd, mu, eps, colsq);
    if (st != MUON_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = upload_pointers(p, params, grads, momentum, s)) != MUON_OK) return st;
    int launches = 0;
    ElemArgs a{};
    for (int cl = 0; cl < kRowClasses; ++cl) {   // rows complete in the shard: the whole step
        a = elem_args(p, p->rn_rows[cl], mu, lr, wd, eps);
        MUON_TRY(launch_rownorm_rows(a, p->rn_rows[cl].blocks, rownorm_class_vec(cl), s));
        launches += p->rn_rows[cl].blocks > 0;
    }
    a = elem_args(p, p->rn_stats, mu, lr, wd, eps);   // momentum and slab sums of U^2
    a.partials = p->cpartials;
    MUON_TRY(launch_rownorm_colstats(a, p->rn_stats.blocks, s));
    a = elem_args(p, p->rn_final, mu, lr, wd, eps);   // this shard's column sums into colsq
    a.partials = p->cpartials;
    MUON_TRY(launch_rownorm_colsum(a, p->rn_final.blocks, colsq, s));
    launches += p->rn_stats.blocks > 0 ? 2 : 0;
    p->last_launches = launches;
    return MUON_OK;
}

muon_status muon_rownorm_shard_apply(muon_plan p, float* const* params, const void* const* grads,
                                     float* const* momentum, float lr, float wd, float mu, float eps,
                                     const float* colsq, void* stream) {
    muon_status st = shard_check(p, params, grads, momentum, lr, wd, mu, eps, colsq);
    if (st != MUON_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = upload_pointers(p, params, grads, momentum, s)) != MUON_OK) return st;
    ElemArgs a = elem_args(p, p->rn_final, mu, lr, wd, eps);
    MUON_TRY(launch_rownorm_colinv(a, p->rn_final.blocks, colsq, s));
    a = elem_args(p, p->rn_apply, mu, lr, wd, eps);
    MUON_TRY(launch_rownorm_colapply(a, p->rn_apply.blocks, s));
    p->last_launches = p->rn_apply.blocks > 0 ? 2 : 0;
    return MUON_OK;
}

muon_status muon_step(muon_plan p, float* const* params, const void* const* grads, float* const* momentum, float lr,
                      float wd, float mu, int32_t ns_steps, muon_mode mode, void* stream) {
    if (!p) return MUON_ERR_INVALID_ARG;
    if (mode == MUON_MODE_ROWNORM) return muon_rownorm_step(p, params, grads, momentum, lr, wd, mu, 1e-8f, stream);
    if (mode != MUON_MODE_NS) return MUON_ERR_INVALID_ARG;
    return muon_step_ex(p, params, grads, momentum, lr, wd, mu, ns_steps, nullptr, 0, stream);
}

// Host side of muon_step_host inside the NS step: the chunk's gradients arrive on
// hc.in (in_ev), its parameters go back on hc.out.
struct HostIO {
    float* const* params_host;   // may be null
};

static muon_status ns_step(muon_plan p, float* const* params, const void* const* grads, float* const* momentum,
                           float lr, float wd, float mu, int32_t ns_steps, const float* coeffs, int32_t restart,
                           void* stream, const HostIO* io);

muon_status muon_step_ex(muon_plan p, float* const* params, const void* const* grads, float* const* momentum,
                         float lr, float wd, float mu, int32_t ns_steps, const float* coeffs, int32_t restart,
                         void* stream) {
    return ns_step(p, params, grads, momentum, lr, wd, mu, ns_steps, coeffs, restart, stream, nullptr);
}

static muon_status ns_step(muon_plan p, float* const* params, const void* const* grads, float* const* momentum,
                           float lr, float wd, float mu, int32_t ns_steps, const float* coeffs, int32_t restart,
                           void* stream, const HostIO* io) {
    if (!p) return MUON_ERR_INVALID_ARG;
    if (!p->full_rows.empty()) return MUON_ERR_UNSUPPORTED;   // dim-0 shard plans: RowNorm only
    const int max_steps = p->opts.max_ns_steps > 0 ? p->opts.max_ns_steps : kMaxNsSteps;
    if (!finite_nonneg(lr) || !finite_nonneg(wd) || !std::isfinite(mu) || mu < 0.f || mu >= 1.f ||
        ns_steps < 0 || ns_steps > max_steps || restart < 0 || restart > kMaxNsSteps)
        return MUON_ERR_INVALID_ARG;
    if (coeffs && !(std::isfinite(coeffs[0]) && std::isfinite(coeffs[1]) && std::isfinite(coeffs[2])))
        return MUON_ERR_INVALID_ARG;
    const float ca = coeffs ? coeffs[0] : kNsA, cb = coeffs ? coeffs[1] : kNsB, cc = coeffs ? coeffs[2] : kNsC;
    // segments of at most `period` Gram steps (one segment unless restarted)
    const int period = restart > 0 ? restart : kMaxNsSteps;
    const int nseg = ns_steps == 0 ? 1 : (ns_steps + period - 1) / period;
    if (nseg > 1 && p->opts.max_ns_steps <= 0) return MUON_ERR_UNSUPPORTED;
    muon_status st = check_pointers(p, params, grads, momentum);
    if (st != MUON_OK) return st;
    if ((st = check_device(p)) != MUON_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = upload_pointers(p, params, grads, momentum, s)) != MUON_OK) return st;
    muon_plan_s::StepEvents* se = nullptr;
    if (p->opts.timing && !(se = next_events(p))) return MUON_ERR_CUDA;
    const int n = (int)p->shapes.size();
    int launches = 0;

    // algorithmic tensor FLOPs of the GEMM stages (the fused r <= 128 step is
    // HBM-bound and timed as a stage of its own)
    double fl_syrk = 0, fl_rr = 0, fl_final = 0;
    for (auto& b : p->buckets) {
        if (!b.batched()) continue;
        const double r = b.r, c = b.c;
        for (int sg = 0; sg < nseg; ++sg) {   // per segment: SYRK, 4Js-3 r x r products, r x c product
            const int Js = sg == nseg - 1 ? ns_steps - sg * period : period;
            fl_syrk += b.batch * r * r * c;
            fl_final += b.batch * 2.0 * r * r * c;
            const int nrr = Js == 0 ? 0 : (Js == 1 ? 1 : 4 * Js - 3);
            fl_rr += b.batch * (double)nrr * r * r * r;
        }
    }
    if (se) {
        p->flops[0] += fl_syrk;
        p->flops[1] += fl_rr;
        p->flops[2] += fl_final;
    }
    if (se) se->ns = true;
    for (size_t ci = 0; ci < p->chunks.size(); ++ci) {
        const muon_plan_s::Chunk& ch = p->chunks[ci];
        cudaEvent_t* ev = se ? &se->e[7 * ci] : nullptr;
        if (io) MUON_TRY(cudaStreamWaitEvent(s, p->hc.in_ev[ci], 0));   // this chunk's gradients
        // ---- momentum, Nesterov, sum of squares, bf16 X0 (oriented), for this chunk
        if (ev) MUON_TRY(cudaEventRecord(ev[0], s));
        ElemArgs a = elem_args(p, ch.mom_rows, mu, lr, wd, 0.f);
        MUON_TRY(launch_momentum_rows(a, ch.mom_rows.blocks, s));
        launches += ch.mom_rows.blocks > 0;
        a = elem_args(p, ch.mom_tiles, mu, lr, wd, 0.f);
        MUON_TRY(launch_momentum_tiles(a, ch.mom_tiles.blocks, s));
        launches += ch.mom_tiles.blocks > 0;
        a = elem_args(p, ch.all, mu, lr, wd, 0.f);
        MUON_TRY(launch_norm_finalize(a, s));
        ++launches;
        if (ev) MUON_TRY(cudaEventRecord(ev[1], s));


        // Plans with both fused and batched matrices run them side by side: the batched
        // products on p->s2 (forked here, joined after the final product) with
        // chain_clusters CTA pairs, the fused kernel on the remaining SMs.
        const bool split = ch.chain_clusters > 0;
        cudaStream_t sc = split ? p->s2 : s;
        const int gc_clusters = split ? ch.chain_clusters : p->pair_clusters;
        const int g_grid1 = split ? 2 * ch.chain_clusters : p->sm_count;
        const int fused_grid = split ? p->sm_count - 2 * ch.chain_clusters : p->sm_count;
        if (se) se->split[ci] = split;
        if (split) {
            MUON_TRY(cudaEventRecord(p->fork_ev, s));
            MUON_TRY(cudaStreamWaitEvent(p->s2, p->fork_ev, 0));
        }

        // ---- r <= 128: the whole step of each matrix (SYRK, recursion, final product +
        // update) in one fused launch, on all SMs but those left to the batched products
        {
            GemmLaunch Ls;
            std::memset(&Ls, 0, sizeof(Ls));
            Ls.status = p->status;
            float* const* W = reinterpret_cast<float* const*>(p->d_ptrs + 2 * n);
            auto flush_small = [&]() -> muon_status {
                if (Ls.nprob == 0) return MUON_OK;
                const muon_status st2 = cuda_status(ns_small_launch(Ls, fused_grid, s));
                ++launches;
                std::memset(&Ls, 0, sizeof(Ls));
                Ls.status = p->status;
                return st2;
            };
            for (int bk : ch.buckets) {
                Bucket& b = p->buckets[bk];
                if (!b.fused) continue;
                if (Ls.nprob == kMaxProblems && (st = flush_small()) != MUON_OK) return st;
                GemmProblem q = problem(b.r, b.c, b.r, b.batch, false, kEpiApply);
                q.tiles_per_item = 1;
                q.tile_begin = Ls.total_tiles;
                q.alpha = p->alpha + b.slot_base;
                q.item_mat = b.d_item_mat;
                q.W = W;
                q.wmap = p->d_wmap;        // W pieces by TMA for the matrices with a valid map
                q.wmap_ok = p->d_wmap_ok;
                q.transposed = p->d_transposed;
                q.Odbg = b.Odbg;
                q.lr = lr;
                q.wd = wd;
                q.scale = 0.2f * std::sqrt((float)b.c);
                q.out_scale = b.gscale;
                q.coef_a = ca;
                q.coef_b = cb / b.gscale;
                q.coef_c = cc / (b.gscale * b.gscale);
                q.ns_steps = ns_steps;
                Ls.mapA[Ls.nprob] = b.ut_a;
                Ls.mapB[Ls.nprob] = b.ut_mn;
                Ls.prob[Ls.nprob] = q;
                Ls.nprob++;
                Ls.total_tiles += b.batch;
            }
            if ((st = flush_small()) != MUON_OK) return st;
        }
        // ---- small nearly square matrices: the whole step in fp32 on CUDA cores
        {
            F32Launch Lf;
            std::memset(&Lf, 0, sizeof(Lf));
            auto reset_f32 = [&]() {
                std::memset(&Lf, 0, sizeof(Lf));
                Lf.mats = p->d_mats;
                Lf.G = const_cast<const void* const*>(p->d_ptrs);
                Lf.M = reinterpret_cast<float* const*>(p->d_ptrs + n);
                Lf.W = reinterpret_cast<float* const*>(p->d_ptrs + 2 * n);
                Lf.mu = mu;
                Lf.lr = lr;
                Lf.wd = wd;
                Lf.grad_bf16 = p->gdt == MUON_BF16;
            };
            auto flush_f32 = [&]() -> muon_status {
                if (Lf.nprob == 0) return MUON_OK;
                const muon_status st2 = cuda_status(ns_f32_launch(Lf, fused_grid, s));
                ++launches;
                reset_f32();
                return st2;
            };
            reset_f32();
            for (int bk : ch.buckets) {
                Bucket& b = p->buckets[bk];
                if (!b.f32) continue;
                if (Lf.nprob == kMaxProblems && (st = flush_f32()) != MUON_OK) return st;
                F32Problem& q = Lf.prob[Lf.nprob++];
                q.r = b.r;
                q.c = b.c;
                q.batch = b.batch;
                q.item_begin = Lf.total;
                q.ns_steps = ns_steps;
                q.item_mat = b.d_item_mat;
                q.alpha = p->alpha + b.slot_base;
                q.Odbg = b.Odbg;
                q.coef_a = ca;
                q.coef_b = cb;
                q.coef_c = cc;
                q.scale = 0.2f * std::sqrt((float)b.c);
                Lf.total += b.batch;
            }
            if ((st = flush_f32()) != MUON_OK) return st;
        }
        if (ev) MUON_TRY(cudaEventRecord(ev[6], s));


        // ---- batched matrices: NS in segments of at most `period` Gram steps; between
        // segments the iterate goes to the other X buffer (xc: 0 X0, 1 the second)
        for (int sg = 0, xc = 0; sg < nseg; ++sg, xc ^= 1) {
            const bool first = sg == 0, last = sg == nseg - 1;
            const int Js = last ? ns_steps - sg * period : period;
            // ---- G0' = s alpha^2 X0 X0^T (lower triangle, mirrored), all buckets in one launch
            {
                Grouper g(p, sc, true, ch.lower, gc_clusters, g_grid1);
                for (int bk : ch.buckets) {
                    Bucket& b = p->buckets[bk];
                    if (!b.batched()) continue;
                    GemmProblem q = problem(b.r, b.r, b.c, b.batch, true, kEpiSyrk);
                    q.a_split = q.b_split = b.split == 2;
                    q.out_split = b.split != 0;
                    q.C = b.G[0];
                    q.strideC = (long long)b.r * b.ldr;
                    q.ldc = b.ldr;
                    q.alpha = (first ? p->alpha : p->ones) + b.slot_base;
                    q.out_scale = b.gscale;
                    q.tma_out = kTmaOutC;
                    if (xc == 0)
                        g.add(b.ut_a, b.ut_b, b.ut_a, q, &b.og[0], nullptr, {&b.utk}, {&b.utk});
                    else
                        g.add(b.ut1_a, b.ut1_b, b.ut1_a, q, &b.og[0], nullptr, {&b.ut1k}, {&b.ut1k});
                }
                g.flush();
                if (g.st != MUON_OK) return g.st;
                launches += g.launches;
            }
            if (ev && first) MUON_TRY(cudaEventRecord(ev[2], sc));


            // ---- Newton-Schulz in the Gram space (fp16 operands, G carried as s G)
            const int J = Js;
            int gc = 0;   // current G buffer
            int qc = 0;   // current Q buffer
            auto rr_problem = [](const Bucket& b, int epi) {
                GemmProblem q = problem(b.r, b.r, b.r, b.batch, true, epi);
                q.strideC = (long long)b.r * b.ldr;
                q.ldc = b.ldr;
                q.a_split = q.b_split = q.out_split = b.split != 0;   // every r x r operand and result
                return q;
            };
            for (int k = 1; k <= J; ++k) {
                {   // P = aI + (b/s) G' + (c/s^2) G'^2 (at k = 1 this is also Q_1)
                    Grouper g(p, sc, false, ch.lower, gc_clusters, g_grid1);
                    for (int bk : ch.buckets) {
                    Bucket& b = p->buckets[bk];
                    if (!b.batched()) continue;
                        GemmProblem q = rr_problem(b, kEpiPoly);
                        q.C = b.P;
                        if (k == 1 && J > 1) q.C2 = b.Q[0];
                        if (k == 1 && J == 1) q.Cb = b.Qb;
                        q.Gin = b.G[gc];
                        q.coef_a = ca;
                        q.coef_b = cb / b.gscale;
                        q.coef_c = cc / (b.gscale * b.gscale);
                        // fp16 P (and the fp16 copy Q_1): TMA stores; P with a bf16 Q_1 (J = 1): per thread
                        q.tma_out = q.Cb ? 0 : (kTmaOutC | (q.C2 ? kTmaOutC2 : 0));
                        const Maps4 g4{&b.gk[gc], &b.gt[gc], true};
                        g.add(b.ga[gc], b.gb[gc], b.ga[gc], q, &b.op, q.C2 ? &b.oq[0] : nullptr, g4, g4, &b.og[gc]);
                    }
                    g.flush();
                    if (g.st != MUON_OK) return g.st;
                    launches += g.launches;
                }
                {   // Q' = P Q (k >= 2) and T = P P (k < J), independent: one launch
                    Grouper g(p, sc, false, ch.lower, gc_clusters, g_grid1);
                    for (int bk : ch.buckets) {
                    Bucket& b = p->buckets[bk];
                    if (!b.batched()) continue;
                        if (k >= 2) {
                            GemmProblem q = rr_problem(b, kEpiPlain);
                            if (k < J) {
                                q.C = b.Q[qc ^ 1];
                                q.tma_out = kTmaOutC;
                                g.add(b.pa, b.qb[qc], b.qa[qc], q, &b.oq[qc ^ 1], nullptr, {&b.pk, &b.pt, true},
                                      {&b.qk[qc], &b.qt[qc], true});
                            } else {
                                q.Cb = b.Qb;
                                q.tma_out = kTmaOutC | kTmaOutBf16;
                                g.add(b.pa, b.qb[qc], b.qa[qc], q, &b.oqb, nullptr, {&b.pk, &b.pt, true},
                                      {&b.qk[qc], &b.qt[qc], true});
                            }
                        }
                        if (k < J) {
                            GemmProblem q = rr_problem(b, kEpiPlain);
                            q.C = b.T;
                            q.tma_out = kTmaOutC;
                            g.add(b.pa, b.pb, b.pa, q, &b.ot, nullptr, {&b.pk, &b.pt, true}, {&b.pk, &b.pt, true});
                        }
                    }
                    g.flush();
                    if (g.st != MUON_OK) return g.st;
                    launches += g.launches;
                    if (k >= 2) qc ^= 1;
                }
                if (k < J) {   // G'' = G' T
                    Grouper g(p, sc, false, ch.lower, gc_clusters, g_grid1);
                    for (int bk : ch.buckets) {
                    Bucket& b = p->buckets[bk];
                    if (!b.batched()) continue;
                        GemmProblem q = rr_problem(b, kEpiPlain);
                        q.C = b.G[gc ^ 1];
                        q.tma_out = kTmaOutC;
                        g.add(b.ga[gc], b.tb, b.ta, q, &b.og[gc ^ 1], nullptr, {&b.gk[gc], &b.gt[gc], true},
                              {&b.tk, &b.tt, true});
                    }
                    g.flush();
                    if (g.st != MUON_OK) return g.st;
                    launches += g.launches;
                    gc ^= 1;
                }
            }
            if (J == 0) {
                for (int bk : ch.buckets) {
                    Bucket& b = p->buckets[bk];
                    if (!b.batched()) continue;
                    MUON_TRY(launch_identity_bf16(b.Qb, b.r, b.ldr, b.batch, b.split != 0, sc));
                    ++launches;
                }
            }
            if (ev && last) MUON_TRY(cudaEventRecord(ev[3], sc));

            // ---- last segment: O = alpha Q X, fused W <- W - lr (s O + wd W) in the stored
            // layout; earlier segments: X' = alpha Q X (bf16) into the other X buffer
            {
                Grouper g(p, sc, true, ch.lower, gc_clusters, g_grid1);
                if (last) {   // W pieces by TMA when every batched matrix of the chunk has a W map
                    const unsigned char* wok = reinterpret_cast<const unsigned char*>(p->h_wmap + n);
                    bool all = true;
                    for (int bk : ch.buckets)
                        if (p->buckets[bk].batched())
                            for (int i : p->buckets[bk].mats) all = all && wok[i];
                    g.wtma = all;
                }
                float* const* W = reinterpret_cast<float* const*>(p->d_ptrs + 2 * n);
                for (int bk : ch.buckets) {
                    Bucket& b = p->buckets[bk];
                    if (!b.batched()) continue;
                    GemmProblem q = problem(b.r, b.c, b.r, b.batch, false, last ? kEpiApply : kEpiXout);
                    q.b_mn = 1;
                    q.a_split = b.split != 0;             // Q in two bf16 parts
                    q.b_split = b.split == 2;             // X in two bf16 parts
                    q.out_split = !last && b.split == 2;  // X' between segments
                    q.alpha = (first ? p->alpha : p->ones) + b.slot_base;
                    if (last) {
                        q.item_mat = b.d_item_mat;
                        q.W = W;
                        q.wmap = p->d_wmap;
                        q.wmap_ok = p->d_wmap_ok;
                        q.transposed = p->d_transposed;
                        q.Odbg = b.Odbg;
                        q.lr = lr;
                        q.wd = wd;
                        q.scale = 0.2f * std::sqrt((float)b.c);
                    } else {
                        q.Cb = p->ut + (xc == 0 ? b.ut1_off : b.ut_off);
                        q.ldc = b.ldu;
                        q.strideC = (long long)b.r * b.ldu;
                    }
                    const CUtensorMap& xm = xc == 0 ? b.ut_mn : b.ut1_mn;
                    g.add(b.qb_a, xm, xm, q, nullptr, nullptr, {&b.qbk, &b.qbt, true},
                          {nullptr, xc == 0 ? &b.utt : &b.ut1t});
                }
                g.flush();
                if (g.st != MUON_OK) return g.st;
                launches += g.launches;
            }
            if (ev && last) MUON_TRY(cudaEventRecord(ev[4], sc));
        }
        if (split) {
            MUON_TRY(cudaEventRecord(p->join_ev, p->s2));
            MUON_TRY(cudaStreamWaitEvent(s, p->join_ev, 0));
        }
        if (io && io->params_host) {   // this chunk's parameters are final: copy them back
            MUON_TRY(cudaEventRecord(p->hc.out_ev[ci], s));
            MUON_TRY(cudaStreamWaitEvent(p->hc.out, p->hc.out_ev[ci], 0));
            for (int bk : ch.buckets)
                for (int i : p->buckets[bk].mats)
                    MUON_TRY(cudaMemcpyAsync(io->params_host[i], params[i],
                                             (size_t)(p->mats[i].m * p->mats[i].n) * sizeof(float),
                                             cudaMemcpyDefault, p->hc.out));
        }
    }
    p->last_launches = launches;
    return MUON_OK;
}

// Copy streams and events of muon_step_host, created on first use.
static muon_status host_copy_setup(muon_plan_s* p) {
    auto& h = p->hc;
    if (h.in) return MUON_OK;
    const size_t nc = p->chunks.size();
    bool ok = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&h.entry_ev, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&h.end_ev, cudaEventDisableTiming) == cudaSuccess;
    bool host_ok = true;
    try {
        h.in_ev.assign(nc, nullptr);
        h.out_ev.assign(nc, nullptr);
    } catch (...) {
        ok = host_ok = false;   // host memory
    }
    for (size_t c = 0; ok && c < nc; ++c)
        ok = cudaEventCreateWithFlags(&h.in_ev[c], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&h.out_ev[c], cudaEventDisableTiming) == cudaSuccess;
    if (ok) return MUON_OK;
    if (host_ok) last_cuda_error() = cudaGetLastError();
    if (h.in) cudaStreamDestroy(h.in);
    if (h.out) cudaStreamDestroy(h.out);
    h.in = h.out = nullptr;
    for (cudaEvent_t& e : h.in_ev)
        if (e) cudaEventDestroy(e);
    for (cudaEvent_t& e : h.out_ev)
        if (e) cudaEventDestroy(e);
    h.in_ev.clear();
    h.out_ev.clear();
    if (h.entry_ev) cudaEventDestroy(h.entry_ev);
    if (h.end_ev) cudaEventDestroy(h.end_ev);
    h.entry_ev = h.end_ev = nullptr;
    return host_ok ? MUON_ERR_CUDA : MUON_ERR_OOM;
}

muon_status muon_step_host(muon_plan p, float* const* params, const void* const* grads, float* const* momentum,
                           const void* const* grads_host, float* const* params_host, float lr, float wd,
                           float mu, int32_t ns_steps, muon_mode mode, void* stream) {
    if (!p || !grads_host) return MUON_ERR_INVALID_ARG;
    if (!p->full_rows.empty()) return MUON_ERR_UNSUPPORTED;
    const int n = (int)p->shapes.size();
    for (int i = 0; i < n; ++i)
        if (!grads_host[i] || (params_host && !params_host[i])) return MUON_ERR_INVALID_ARG;
    // every check of the step itself before anything is enqueued
    const int max_steps = p->opts.max_ns_steps > 0 ? p->opts.max_ns_steps : kMaxNsSteps;
    if (!finite_nonneg(lr) || !finite_nonneg(wd) || !std::isfinite(mu) || mu < 0.f || mu >= 1.f)
        return MUON_ERR_INVALID_ARG;
    if (mode == MUON_MODE_NS) {
        if (ns_steps < 0 || ns_steps > max_steps) return MUON_ERR_INVALID_ARG;
    } else if (mode != MUON_MODE_ROWNORM) {
        return MUON_ERR_INVALID_ARG;
    }
    muon_status st = check_pointers(p, params, grads, momentum);
    if (st != MUON_OK) return st;
    if ((st = check_device(p)) != MUON_OK) return st;
    if ((st = host_copy_setup(p)) != MUON_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t gsz = p->gdt == MUON_BF16 ? 2 : 4;
    auto& h = p->hc;
    // gradients in, chunk by chunk, after the caller's earlier work (which may still read grads)
    MUON_TRY(cudaEventRecord(h.entry_ev, s));
    MUON_TRY(cudaStreamWaitEvent(h.in, h.entry_ev, 0));
    for (size_t ci = 0; ci < p->chunks.size(); ++ci) {
        for (int bk : p->chunks[ci].buckets)
            for (int i : p->buckets[bk].mats)
                MUON_TRY(cudaMemcpyAsync(const_cast<void*>(grads[i]), grads_host[i],
                                         (size_t)(p->mats[i].m * p->mats[i].n) * gsz, cudaMemcpyDefault, h.in));
        MUON_TRY(cudaEventRecord(h.in_ev[ci], h.in));
    }
    if (mode == MUON_MODE_NS) {
        const HostIO io{params_host};
        st = ns_step(p, params, grads, momentum, lr, wd, mu, ns_steps, nullptr, 0, stream, &io);
        if (st != MUON_OK) return st;
    } else {   // RowNorm, chunk by chunk like the NS step
        if ((st = upload_pointers(p, params, grads, momentum, s)) != MUON_OK) return st;
        int launches = 0;
        for (size_t ci = 0; ci < p->chunks.size(); ++ci) {
            const muon_plan_s::Chunk& ch = p->chunks[ci];
            MUON_TRY(cudaStreamWaitEvent(s, h.in_ev[ci], 0));
            if ((st = rownorm_launch(p, ch.rn_rows, ch.rn_stats, ch.rn_final, ch.rn_apply, lr, wd, mu, 1e-8f, s,
                                     &launches)) != MUON_OK)
                return st;
            if (!params_host) continue;
            MUON_TRY(cudaEventRecord(h.out_ev[ci], s));
            MUON_TRY(cudaStreamWaitEvent(h.out, h.out_ev[ci], 0));
            for (int bk : ch.buckets)
                for (int i : p->buckets[bk].mats)
                    MUON_TRY(cudaMemcpyAsync(params_host[i], params[i],
                                             (size_t)(p->mats[i].m * p->mats[i].n) * sizeof(float),
                                             cudaMemcpyDefault, h.out));
        }
        p->last_launches = launches;
    }
    if (params_host) {   // the caller's stream covers the copies back
        MUON_TRY(cudaEventRecord(h.end_ev, h.out));
        MUON_TRY(cudaStreamWaitEvent(s, h.end_ev, 0));
    }
    return MUON_OK;
}

}  // extern "C"
