// The plan's remaining C entry points (include/muon.h): launch tuning, status, timing
// and the debug copies.  Host code only.
#include "plan.h"

extern "C" {

muon_status muon_plan_tune(muon_plan p, float* const* params, const void* const* grads, float* const* momentum,
                           float lr, float wd, float mu, int32_t reps, float* ms_out, void* stream) {
    if (!p || reps < 1 || reps > 100) return MUON_ERR_INVALID_ARG;
    if (!p->full_rows.empty()) return MUON_ERR_UNSUPPORTED;
    muon_status st = check_pointers(p, params, grads, momentum);
    if (st != MUON_OK) return st;
    // candidates: CTA pairs beside the fused kernel (none, the estimate, half and one and a
    // half times it; only while opts.chain_clusters leaves the choice to the plan) and
    // symmetric r x r results stored as the lower triangle or whole
    bool mixed = false;
    for (const auto& ch : p->chunks) mixed = mixed || (ch.mixed && ch.chain_est > 0);
    const float scales[4] = {1.f, 0.f, 0.5f, 1.5f};
    const int n_scales = mixed && p->opts.chain_clusters == 0 && p->s2 ? 4 : 1;
    bool lower_choice = false;   // chunks where lower-triangle storage is a choice
    for (const auto& ch : p->chunks) lower_choice = lower_choice || ch.lower_ok;
    const bool lowers[2] = {true, false};
    const int n_lowers = lower_choice && !p->opts.full_symmetric ? 2 : 1;
    const int kmax = std::min(p->pair_clusters - 1, (p->sm_count - 2) / 2);
    auto apply = [&](float sc, bool q) {
        for (auto& ch : p->chunks)
            if (ch.mixed && p->opts.chain_clusters == 0)
                ch.chain_clusters = sc == 0.f ? 0 : std::min(std::max((int)std::lround(ch.chain_est * sc), 1), kmax);
        for (auto& ch : p->chunks) ch.lower = ch.lower_ok && !p->opts.full_symmetric && q;
    };
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        last_cuda_error() = cudaGetLastError();
        if (e0) cudaEventDestroy(e0);
        return MUON_ERR_CUDA;
    }
    float best = 0.f, best_sc = 1.f;
    bool best_q = true;
    int tried = 0;
    for (int si = 0; si < n_scales; ++si) {
        for (int qi = 0; qi < n_lowers; ++qi) {
            const float sc = scales[si];
            const bool q = lowers[qi];
            apply(sc, q);
            st = muon_step_ex(p, params, grads, momentum, lr, wd, mu, kMaxNsSteps, nullptr, 0, stream);   // warm-up
            if (st == MUON_OK && cudaEventRecord(e0, s) != cudaSuccess) st = MUON_ERR_CUDA;
            for (int i = 0; st == MUON_OK && i < reps; ++i)
                st = muon_step_ex(p, params, grads, momentum, lr, wd, mu, kMaxNsSteps, nullptr, 0, stream);
            float ms = 0.f;
            if (st == MUON_OK && (cudaEventRecord(e1, s) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
                                  cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess))
                st = MUON_ERR_CUDA;
            if (st != MUON_OK) break;
            ms /= (float)reps;
            if (tried == 0 || ms < best) {
                best = ms;
                best_sc = sc;
                best_q = q;
            }
            ++tried;
        }
        if (st != MUON_OK) break;
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    apply(best_sc, best_q);
    if (st != MUON_OK) return st;
    p->tuned = tried;
    if (ms_out) *ms_out = best;
    return muon_sync(p, stream);
}

muon_status muon_sync(muon_plan p, void* stream) {
    if (!p) return MUON_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MUON_ERR_CUDA;
    int st = 0;
    MUON_TRY(cudaMemcpy(&st, p->status, sizeof(int), cudaMemcpyDeviceToHost));
    if (st != 0) {
        MUON_TRY(cudaMemset(p->status, 0, sizeof(int)));
        // a timeout replaces the word; non-finite norms are or-ed into it
        return (st & kStatusTimeoutMask) ? MUON_ERR_TIMEOUT : MUON_ERR_NONFINITE;
    }
    return MUON_OK;
}

muon_status muon_debug_wait_timeout(muon_plan p, int32_t limit_us, void* stream) {
    if (!p || limit_us < 1 || limit_us > 1000000) return MUON_ERR_INVALID_ARG;
    if (check_device(p) != MUON_OK) return MUON_ERR_INVALID_ARG;
    return cuda_status(
        launch_wait_selftest(p->status, 1000ull * (unsigned long long)limit_us, static_cast<cudaStream_t>(stream)));
}

muon_status muon_debug_copy_update(muon_plan p, int32_t i, float* dst, void* stream) {
    if (!p || !dst || i < 0 || i >= (int)p->shapes.size()) return MUON_ERR_INVALID_ARG;
    if (!p->opts.keep_update) return MUON_ERR_INVALID_ARG;
    const Bucket& b = p->buckets[p->mat_bucket[i]];
    const size_t numel = (size_t)b.r * b.c;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(dst, b.Odbg + (size_t)p->mat_item[i] * numel, numel * sizeof(float), cudaMemcpyDefault, s) !=
        cudaSuccess)
        return MUON_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

muon_status muon_debug_update_error(muon_plan p, int32_t i, const float* ref, double* rel, void* stream) {
    if (!p || !ref || !rel || i < 0 || i >= (int)p->shapes.size()) return MUON_ERR_INVALID_ARG;
    if (!p->opts.keep_update || !p->full_rows.empty()) return MUON_ERR_INVALID_ARG;
    const Bucket& b = p->buckets[p->mat_bucket[i]];
    const long long numel = (long long)b.r * b.c;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MUON_TRY(launch_sq_diff(b.Odbg + (size_t)p->mat_item[i] * numel, ref, numel, p->diff, s));
    double sums[2] = {0.0, 0.0};
    MUON_TRY(cudaMemcpyAsync(sums, p->diff, sizeof(sums), cudaMemcpyDeviceToHost, s));
    MUON_TRY(cudaStreamSynchronize(s));
    *rel = sums[1] > 0.0 ? std::sqrt(sums[0] / sums[1]) : std::sqrt(sums[0]);
    return MUON_OK;
}

muon_status muon_debug_copy_workspace(muon_plan p, int32_t i, int32_t which, void* dst, int32_t* ld,
                                      void* stream) {
    if (!p || !dst || !ld || i < 0 || i >= (int)p->shapes.size() || which < 0 || which > 8)
        return MUON_ERR_INVALID_ARG;
    const Bucket& b = p->buckets[p->mat_bucket[i]];
    // the fused kernel keeps its r x r operands on chip: only X0 and alpha exist
    if (!b.batched() && which >= 1 && which <= 7) return MUON_ERR_UNSUPPORTED;
    // split buffers hold two parts per matrix (hi at 2 item, lo at 2 item + 1): the hi part is copied
    const int item = p->mat_item[i] * (which >= 1 && which <= 7 && b.split ? 2 : 1);
    const int xitem = p->mat_item[i] * (b.split == 2 ? 2 : 1);
    const size_t rr = (size_t)b.r * b.ldr;
    const void* src = nullptr;
    size_t bytes = 0;
    *ld = b.ldr;
    switch (which) {
        case 0:
            src = p->ut + b.ut_off + (size_t)xitem * b.r * b.ldu;
            bytes = (size_t)b.r * b.ldu * 2;
            *ld = b.ldu;
            break;
        case 1: case 2: src = b.G[which - 1] + item * rr; bytes = rr * 2; break;
        case 3: src = b.P + item * rr; bytes = rr * 2; break;
        case 4: src = b.T + item * rr; bytes = rr * 2; break;
        case 5: case 6: src = b.Q[which - 5] + item * rr; bytes = rr * 2; break;
        case 7: src = b.Qb + item * rr; bytes = rr * 2; break;
        case 8: src = p->alpha + p->mats[i].slot; bytes = 4; *ld = 1; break;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (which >= 1 && which <= 7 && b.r > kBM && p->chunks[b.chunk].lower) {
        // lower-triangle storage (256 x 256 tiles at or below the diagonal): rebuild the upper part
        std::vector<uint16_t> h;
        try {
            h.resize(rr);
        } catch (...) {
            return MUON_ERR_OOM;   // host memory
        }
        if (cudaMemcpyAsync(h.data(), src, bytes, cudaMemcpyDefault, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return MUON_ERR_CUDA;
        for (int row = 0; row < b.r; ++row)
            for (int col = (row / 256 + 1) * 256; col < b.r; ++col)
                h[(size_t)row * b.ldr + col] = h[(size_t)col * b.ldr + row];
        if (cudaMemcpyAsync(dst, h.data(), bytes, cudaMemcpyDefault, s) != cudaSuccess) return MUON_ERR_CUDA;
        return cudaStreamSynchronize(s) == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
    }
    if (cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, s) != cudaSuccess) return MUON_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

muon_status muon_plan_info(muon_plan p, muon_plan_info_t* info) {
    if (!p || !info) return MUON_ERR_INVALID_ARG;
    info->n_matrices = (int32_t)p->shapes.size();
    info->n_buckets = (int32_t)p->buckets.size();
    info->workspace_bytes = (int64_t)p->ws_bytes;
    info->launches_last_step = p->last_launches;
    info->n_chunks = (int32_t)p->chunks.size();
    int lower = 0;
    for (const auto& ch : p->chunks) lower += ch.lower ? 1 : 0;
    info->lower_chunks = lower;
    info->tuned_candidates = p->tuned;
    int chain = 0;
    for (const auto& ch : p->chunks) chain = std::max(chain, ch.chain_clusters);
    info->chain_clusters = chain;
    info->sm_count = p->sm_count;
    int nsplit = 0, nf32 = 0;
    for (const auto& b : p->buckets) {
        nsplit += b.split ? 1 : 0;
        nf32 += b.f32 ? 1 : 0;
    }
    info->split_buckets = nsplit;
    info->fp32_buckets = nf32;
    info->colsq_len = (int64_t)p->colsq_len;
    return MUON_OK;
}

muon_status muon_stage_times(muon_plan p, float* ms, double* flops, int32_t n_stages) {
    if (!p || !ms || n_stages < 0 || n_stages > 6) return MUON_ERR_INVALID_ARG;
    if (p->n_timed == 0) return MUON_ERR_INVALID_ARG;
    double acc[6] = {0, 0, 0, 0, 0, 0};
    // NS steps: momentum e[0] -> e[1]; fused e[1] -> e[6]; SYRK from e[6] (after the
    // fused kernel) or, split, from e[1] (beside it) to e[2]; r x r e[2] -> e[3];
    // final e[3] -> e[4]
    for (size_t g = 0; g < p->n_timed; ++g) {
        const auto& se = p->evs[g];
        float t = 0.f;
        if (se.ns) {
            for (size_t c = 0; c < p->chunks.size(); ++c) {   // stages summed over the chunks
                const cudaEvent_t* e = &se.e[7 * c];
                if (cudaEventSynchronize(e[4]) != cudaSuccess || cudaEventSynchronize(e[6]) != cudaSuccess)
                    return MUON_ERR_CUDA;
                const int from[5] = {0, se.split[c] ? 1 : 6, 2, 3, 1}, to[5] = {1, 2, 3, 4, 6},
                          slot[5] = {0, 1, 2, 3, 5};
                for (int k = 0; k < 5; ++k) {
                    if (cudaEventElapsedTime(&t, e[from[k]], e[to[k]]) != cudaSuccess) return MUON_ERR_CUDA;
                    acc[slot[k]] += t;
                }
            }
        } else {
            if (cudaEventSynchronize(se.e[5]) != cudaSuccess) return MUON_ERR_CUDA;
            if (cudaEventElapsedTime(&t, se.e[0], se.e[5]) != cudaSuccess) return MUON_ERR_CUDA;
            acc[4] += t;
        }
    }
    for (int k = 0; k < n_stages; ++k) ms[k] = (float)acc[k];
    if (flops)
        for (int k = 0; k < 3; ++k) flops[k] = p->flops[k];
    p->n_timed = 0;
    p->flops[0] = p->flops[1] = p->flops[2] = 0;
    return MUON_OK;
}

}  // extern "C"
