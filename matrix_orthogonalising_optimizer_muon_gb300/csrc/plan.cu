// The plan: host-side planning (orientation, buckets, chunks, workspace layout), its
// device part (one workspace allocation, tensor maps, launch lists), the argument checks
// and pointer upload every step shares, and the plan's C entry points (create, size,
// destroy, owner partition, status strings).
#include "plan.h"

namespace muon_impl {

namespace {
thread_local cudaError_t g_last_cuda_error = cudaSuccess;
}  // namespace

cudaError_t& last_cuda_error() { return g_last_cuda_error; }

// Every params / momentum / grads range must be disjoint from every other.
muon_status check_pointers(const muon_plan_s* p, float* const* params, const void* const* grads,
                           float* const* momentum) {
    if (!params || !grads || !momentum) return MUON_ERR_INVALID_ARG;
    const size_t n = p->shapes.size();
    const size_t gsz = p->gdt == MUON_BF16 ? 2 : 4;
    std::vector<std::pair<uintptr_t, uintptr_t>> ranges;
    ranges.reserve(3 * n);
    for (size_t i = 0; i < n; ++i) {
        if (!params[i] || !grads[i] || !momentum[i]) return MUON_ERR_INVALID_ARG;
        const size_t numel = (size_t)p->shapes[i].rows * (size_t)p->shapes[i].cols;
        const uintptr_t w = reinterpret_cast<uintptr_t>(params[i]);
        const uintptr_t g = reinterpret_cast<uintptr_t>(grads[i]);
        const uintptr_t m = reinterpret_cast<uintptr_t>(momentum[i]);
        ranges.push_back({w, w + numel * 4});
        ranges.push_back({m, m + numel * 4});
        ranges.push_back({g, g + numel * gsz});
    }
    std::sort(ranges.begin(), ranges.end());
    for (size_t k = 1; k < ranges.size(); ++k)
        if (ranges[k].first < ranges[k - 1].second) return MUON_ERR_INVALID_ARG;
    return MUON_OK;
}

muon_status check_device(const muon_plan_s* p) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_CUDA;
    return dev == p->device ? MUON_OK : MUON_ERR_INVALID_ARG;
}

// Copies the per-call pointer tables to the device when they changed.
muon_status upload_pointers(muon_plan_s* p, float* const* params, const void* const* grads, float* const* momentum,
                            cudaStream_t s) {
    const size_t n = p->shapes.size();
    bool same = p->uploaded;
    for (size_t i = 0; same && i < n; ++i)
        same = p->h_cache[i] == grads[i] && p->h_cache[n + i] == momentum[i] && p->h_cache[2 * n + i] == params[i];
    if (same) return MUON_OK;
    if (p->uploaded) MUON_TRY(cudaEventSynchronize(p->upload_ev));   // pinned buffer free again
    for (size_t i = 0; i < n; ++i) {
        p->h_cache[i] = const_cast<void*>(grads[i]);
        p->h_cache[n + i] = momentum[i];
        p->h_cache[2 * n + i] = params[i];
    }
    std::memcpy(p->h_pinned, p->h_cache.data(), 3 * n * sizeof(void*));
    MUON_TRY(cudaMemcpyAsync(p->d_ptrs, p->h_pinned, 3 * n * sizeof(void*), cudaMemcpyHostToDevice, s));
    if (p->h_wmap) {   // W piece maps follow the parameter pointers (tensor-core final products)
        unsigned char* ok = reinterpret_cast<unsigned char*>(p->h_wmap + n);
        for (size_t i = 0; i < n; ++i) {
            const MatDev& md = p->mats[i];
            const Bucket& bk = p->buckets[p->mat_bucket[i]];
            const bool usable = (bk.batched() || bk.fused) && md.n % 4 == 0 &&
                                (reinterpret_cast<uintptr_t>(params[i]) & 15) == 0;
            ok[i] = usable && make_w_piece_map(&p->h_wmap[i], params[i], (uint64_t)md.m, (uint64_t)md.n) ? 1 : 0;
        }
        MUON_TRY(cudaMemcpyAsync(p->d_wmap, p->h_wmap, n * sizeof(CUtensorMap), cudaMemcpyHostToDevice, s));
        MUON_TRY(cudaMemcpyAsync(p->d_wmap_ok, ok, n, cudaMemcpyHostToDevice, s));
    }
    MUON_TRY(cudaEventRecord(p->upload_ev, s));
    p->uploaded = true;
    return MUON_OK;
}

ElemArgs elem_args(const muon_plan_s* p, const ListDev& l, float mu, float lr, float wd, float eps) {
    ElemArgs a{};
    const size_t n = p->shapes.size();
    a.mats = p->d_mats;
    a.list = l.list;
    a.nlist = l.n;
    a.list_blk = l.blk;
    a.G = const_cast<const void* const*>(p->d_ptrs);
    a.M = reinterpret_cast<float* const*>(p->d_ptrs + n);
    a.W = reinterpret_cast<float* const*>(p->d_ptrs + 2 * n);
    a.ut = p->ut;
    a.partials = p->partials;
    a.alpha = p->alpha;
    a.rowinv = p->rowinv;
    a.mu = mu;
    a.lr = lr;
    a.wd = wd;
    a.eps = eps;
    a.grad_bf16 = p->gdt == MUON_BF16;
    a.check_finite = p->opts.check_finite ? 1 : 0;
    a.status = p->status;
    return a;
}

int sym_tiles(int r) {
    const int tm = (int)ceil_div(r, kBM);
    int t = 0;
    for (int i = 0; i < tm; ++i) t += i / 2 + 1;
    return t;
}

GemmProblem problem(int M, int N, int K, int batch, bool sym, int epi) {
    GemmProblem q{};
    q.M = M;
    q.N = N;
    q.K = K;
    q.batch = batch;
    q.tiles_m = (int)ceil_div(M, kBM);
    q.tiles_n = (int)ceil_div(N, kBN);
    q.tiles_per_item = sym ? sym_tiles(M) : q.tiles_m * q.tiles_n;
    q.sym = sym ? 1 : 0;
    q.epi = epi;
    return q;
}

// Timed steps kept between muon_stage_times calls.
constexpr size_t kMaxTimedSteps = 4096;

// Event group for the next timed step (the last group is reused past the cap).
muon_plan_s::StepEvents* next_events(muon_plan_s* p) {
    if (p->n_timed < p->evs.size()) return &p->evs[p->n_timed++];
    if (p->evs.size() >= kMaxTimedSteps) return &p->evs.back();
    muon_plan_s::StepEvents g{};
    try {
        g.e.assign(7 * p->chunks.size(), nullptr);
        g.split.assign(p->chunks.size(), 0);
        p->evs.reserve(p->evs.size() + 1);   // the push_back below cannot throw
    } catch (...) {
        return nullptr;   // host memory
    }
    for (auto& e : g.e)
        if (cudaEventCreate(&e) != cudaSuccess) {
            for (auto& x : g.e)
                if (x) cudaEventDestroy(x);
            return nullptr;
        }
    p->evs.push_back(std::move(g));
    p->n_timed = p->evs.size();
    return &p->evs.back();
}

void free_plan(muon_plan_s* p) {
    if (!p) return;
    if (p->ws) cudaFree(p->ws);
    if (p->h_pinned) cudaFreeHost(p->h_pinned);
    if (p->h_wmap) cudaFreeHost(p->h_wmap);
    if (p->upload_ev) cudaEventDestroy(p->upload_ev);
    if (p->fork_ev) cudaEventDestroy(p->fork_ev);
    if (p->join_ev) cudaEventDestroy(p->join_ev);
    if (p->s2) cudaStreamDestroy(p->s2);
    if (p->hc.in) cudaStreamDestroy(p->hc.in);
    if (p->hc.out) cudaStreamDestroy(p->hc.out);
    for (cudaEvent_t e : p->hc.in_ev)
        if (e) cudaEventDestroy(e);
    for (cudaEvent_t e : p->hc.out_ev)
        if (e) cudaEventDestroy(e);
    if (p->hc.entry_ev) cudaEventDestroy(p->hc.entry_ev);
    if (p->hc.end_ev) cudaEventDestroy(p->hc.end_ev);
    for (auto& g : p->evs)
        for (auto& e : g.e)
            if (e) cudaEventDestroy(e);
    delete p;
}

// Argument checks of muon_plan_create and muon_plan_workspace_size.
muon_status check_plan_args(const muon_shape* shapes, int32_t n, muon_dtype grad_dtype,
                            const muon_plan_opts* opts) {
    if (!shapes || n <= 0) return MUON_ERR_INVALID_ARG;
    if (grad_dtype != MUON_F32 && grad_dtype != MUON_BF16) return MUON_ERR_UNSUPPORTED;
    for (int i = 0; i < n; ++i) {
        if (shapes[i].rows <= 0 || shapes[i].cols <= 0) return MUON_ERR_INVALID_ARG;
        if (shapes[i].rows > kMaxDim || shapes[i].cols > kMaxDim) return MUON_ERR_UNSUPPORTED;
        if (std::min(shapes[i].rows, shapes[i].cols) > kMaxR) return MUON_ERR_UNSUPPORTED;
    }
    if (opts && (opts->max_ns_steps < 0 || opts->max_ns_steps > kMaxNsStepsRestart || opts->chunks < 0 ||
                 opts->workspace_bytes < 0))
        return MUON_ERR_INVALID_ARG;
    if (opts && opts->full_rows)
        for (int i = 0; i < n; ++i)
            if (opts->full_rows[i] < shapes[i].rows || opts->full_rows[i] > kMaxDim) return MUON_ERR_INVALID_ARG;
    return MUON_OK;
}

// The host part of planning, from p->shapes and p->opts alone (no CUDA call):
// orientation, buckets, chunks and the workspace layout; sets p->mats, p->buckets,
// p->chunks, p->mat_bucket, p->mat_item and p->ws_bytes.  MUON_ERR_OOM when
// opts.workspace_bytes cannot hold the largest single matrix.
muon_status plan_layout(muon_plan_s* p, Layout& L) {
    const int n = (int)p->shapes.size();
    // ---- orient; group by oriented shape (r, c) in order of first appearance
    // (DiT paper sec. 3.1; DMuon batching)
    p->mats.resize(n);
    p->mat_bucket.resize(n);
    p->mat_item.resize(n);
    std::vector<std::pair<int, int>> group_rc;
    std::vector<int> group_lv;   // per group: the matrices' opts.precision_of entry (0: the plan's rule)
    std::vector<std::vector<int>> group_mats;
    for (int i = 0; i < n; ++i) {
        MatDev& md = p->mats[i];
        std::memset(&md, 0, sizeof(md));
        md.m = p->shapes[i].rows;
        md.n = p->shapes[i].cols;
        md.r = (int)std::min(md.m, md.n);
        md.c = (int)std::max(md.m, md.n);
        md.transposed = md.m > md.n;
        md.scale = 0.2f * std::sqrt((float)md.c);   // blog eq. (4)
        if (!p->full_rows.empty()) {   // a dim-0 shard: RowNorm axis and scale of the full matrix
            const long long fm = p->full_rows[i];
            md.transposed = fm > md.n;
            md.scale = 0.2f * std::sqrt((float)std::max(fm, md.n));
        }
        size_t g = 0;
        const int lv = p->prec_of.empty() ? 0 : p->prec_of[i];
        while (g < group_rc.size() &&
               !(group_rc[g].first == md.r && group_rc[g].second == md.c && group_lv[g] == lv))
            ++g;
        if (g == group_rc.size()) {
            group_rc.push_back({md.r, md.c});
            group_lv.push_back(lv);
            group_mats.emplace_back();
        }
        group_mats[g].push_back(i);
    }

    // ---- workspace: a fixed part (per-matrix tables, partial sums, pointer tables,
    // launch lists, debug copies of O) and a region for the X0 and r x r buffers of
    // one chunk of matrices, shared by all chunks (they run one after the other)
    const bool restarts = L.restarts = p->opts.max_ns_steps > 0;   // second X buffer, batched path for all
    // fp32 path (opts.small_fp32): 0 nearly square (c < 1.25 r) matrices with r <= 128,
    // > 0 every matrix with r <= 128, < 0 none; never in plans with restarts
    auto is_f32 = [&](int r, int c) {
        if (restarts || p->opts.small_fp32 < 0 || r > kF32MaxR) return false;
        return p->opts.small_fp32 > 0 || 4LL * c < 5LL * r;
    };
    const bool fused_ok = !p->opts.generic_small && !restarts;
    auto is_fused = [&](int r, int c) { return fused_ok && r <= kSmallMaxR && !is_f32(r, c); };
    // split precision of a batched bucket (opts.precision, opts.split_max_r)
    // lv: the matrices' opts.precision_of entry (< 0 plain, 1 or 2 that level, 0 the plan's rule)
    auto split_of = [&](int r, int c, int lv) -> int {
        if (is_fused(r, c) || is_f32(r, c)) return 0;
        if (lv != 0) return lv < 0 ? 0 : (lv >= 2 ? 2 : 1);
        if (p->opts.precision < 0) return 0;
        if (p->opts.precision > 0) return p->opts.precision >= 2 ? 2 : 1;
        const int rmax = p->opts.split_max_r > 0 ? p->opts.split_max_r : 1024;
        return (4LL * c < 5LL * r && r <= rmax) ? 1 : 0;
    };
    // region bytes of a bucket of `batch` matrices, exactly as laid out below: its X0
    // (and second X) buffer and, batched, its seven r x r buffers, each rounded to 256
    // (split buffers hold two parts per matrix)
    const bool sharded = !p->full_rows.empty();   // RowNorm only: no NS buffers
    auto bucket_bytes = [&](int r, int c, int lv, long long batch) -> long long {
        if (sharded) return 0;
        const int sp = split_of(r, c, lv);
        const long long x = round_up(batch * r * round_up(c, 8) * 2 * (sp == 2 ? 2 : 1), 256);
        const long long rr = round_up(batch * r * round_up(r, 8) * 2 * (sp ? 2 : 1), 256);
        return (restarts ? 2 : 1) * x + (is_fused(r, c) || is_f32(r, c) ? 0 : 7 * rr);
    };
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = (size_t)round_up((long long)(off + bytes), 256);
        return o;
    };
    // momentum / RowNorm bookkeeping per matrix (not chunked)
    long long mom_part = 0, col_part = 0, inv_elems = 0;
    for (int i = 0; i < n; ++i) {
        MatDev& md = p->mats[i];
        md.nblk = (int)(md.transposed ? ceil_div(md.m, kTileRows) * ceil_div(md.n, kTile)
                                      : ceil_div(md.m * md.n, kMomElemsPerBlock));
        md.part_off = mom_part;
        mom_part += md.nblk;
        if (md.transposed) {
            md.cpart_off = col_part;
            col_part += ceil_div(md.m, kColSlab) * md.n;
            md.inv_off = inv_elems;
            inv_elems += round_up(md.n, 4);
            L.rnc_list.push_back(i);
        } else {
            L.rnr_list.push_back(i);
        }
    }
    p->colsq_len = sharded ? inv_elems : 0;
    L.o_mats = take(sizeof(MatDev) * n);
    L.o_part = take(sizeof(float) * std::max<long long>(mom_part, 1));
    L.o_cpart = take(sizeof(float) * std::max<long long>(col_part, 1));
    L.o_inv = take(sizeof(float) * std::max<long long>(inv_elems, 1));
    L.o_alpha = take(sizeof(float) * n);
    L.o_status = take(sizeof(int));
    L.o_tr = take((size_t)n);
    L.o_ptrs = take(sizeof(void*) * 3 * n);
    L.o_items = take(sizeof(int) * n);   // item -> plan matrix, per bucket slice
    L.o_ones = take(sizeof(float) * n);
    L.o_diff = take(sizeof(double) * (2 + 2 * kDiffParts));
    L.o_wmap = take(sizeof(CUtensorMap) * n);   // W piece maps (slices are 256-byte aligned)
    L.o_wmap_ok = take((size_t)n);
    L.o_odbg = p->opts.keep_update ? take([&] {
        size_t t = 0;
        for (int i = 0; i < n; ++i) t += (size_t)round_up(p->mats[i].m * p->mats[i].n * 4, 256);
        return t;
    }()) : 0;
    // launch lists: per chunk the momentum rows / tiles / all lists and its six
    // RowNorm lists (rows in three length classes, column statistics, finalize,
    // apply), and the six RowNorm lists of the whole plan.  Chunks partition the
    // matrices (n chunks at most); a list of k matrices takes max(k, 1) ints and k + 1
    // prefixes.  Momentum lists: 2 per matrix plus 3 per chunk, at most 5n; chunk
    // RowNorm lists (rows once, column matrices three times): at most 3n + 6n; the
    // plan's: 3n + 6.  17n + 6 <= 17n + 16 of each.
    L.o_lists = take(sizeof(int) * (size_t)(17 * n + 16));
    L.o_prefix = take(sizeof(long long) * (size_t)(17 * n + 16));
    const size_t fixed_bytes = off;

    // ---- chunks: matrices in group order, a new chunk whenever the region would
    // exceed what the cap leaves after the fixed part (one chunk without a cap)
    const long long cap = p->opts.workspace_bytes;
    double region_cap = 1e300;
    if (cap > 0) {
        region_cap = (double)cap - (double)fixed_bytes;
        double need = 0;
        for (int i = 0; i < n; ++i)
            need = std::max(need, (double)bucket_bytes(p->mats[i].r, p->mats[i].c,
                                                       p->prec_of.empty() ? 0 : p->prec_of[i], 1));
        if (region_cap < need) return MUON_ERR_OOM;   // the cap cannot hold even the largest single matrix
    }
    if (p->opts.chunks > 1) {   // about opts.chunks chunks, each at least one matrix
        double total = 0, largest = 0;
        for (int i = 0; i < n; ++i) {
            const double b =
                (double)bucket_bytes(p->mats[i].r, p->mats[i].c, p->prec_of.empty() ? 0 : p->prec_of[i], 1);
            total += b;
            largest = std::max(largest, b);
        }
        const double per = total / p->opts.chunks;
        region_cap = std::min(region_cap, std::max(per, largest));
    }
    {
        long long used = 0;   // region bytes of the current chunk, exactly
        p->chunks.emplace_back();
        for (size_t g = 0; g < group_rc.size(); ++g) {
            const int r = group_rc[g].first, c = group_rc[g].second, lv = group_lv[g];
            int cur = -1;   // bucket of this group in the current chunk
            for (int i : group_mats[g]) {
                const long long k = cur < 0 ? 0 : (long long)p->buckets[cur].mats.size();
                long long grow = bucket_bytes(r, c, lv, k + 1) - (k > 0 ? bucket_bytes(r, c, lv, k) : 0);
                if ((double)(used + grow) > region_cap && used > 0) {
                    p->chunks.emplace_back();
                    used = 0;
                    cur = -1;
                    grow = bucket_bytes(r, c, lv, 1);
                }
                if (cur < 0) {
                    Bucket nb{};   // value-initialised: the tensor maps are filled in later
                    nb.r = r;
                    nb.c = c;
                    nb.ldr = (int)round_up(r, 8);
                    nb.ldu = (int)round_up(c, 8);
                    nb.fused = is_fused(r, c);
                    nb.f32 = is_f32(r, c);
                    nb.split = split_of(r, c, lv);
                    nb.chunk = (int)p->chunks.size() - 1;
                    p->buckets.push_back(nb);
                    cur = (int)p->buckets.size() - 1;
                    p->chunks.back().buckets.push_back(cur);
                }
                used += grow;
                p->mat_bucket[i] = cur;
                p->mat_item[i] = (int)p->buckets[cur].mats.size();
                p->buckets[cur].mats.push_back(i);
            }
        }
    }
    // region offsets: each chunk's buckets laid out from the start of the region
    size_t region_bytes = 0;
    std::vector<size_t>& o_ut = L.o_ut;
    std::vector<size_t>& o_ut1 = L.o_ut1;
    std::vector<size_t>& o_rr = L.o_rr;
    std::vector<size_t>& o_qb = L.o_qb;
    o_ut.assign(p->buckets.size(), 0);
    o_ut1.assign(p->buckets.size(), 0);
    o_rr.assign(p->buckets.size(), 0);
    o_qb.assign(p->buckets.size(), 0);
    {
        int slots = 0;
        for (auto& ch : p->chunks) {
            size_t roff = 0;
            auto rtake = [&](size_t bytes) {
                const size_t o = roff;
                roff = (size_t)round_up((long long)(roff + bytes), 256);
                return o;
            };
            for (int k : ch.buckets) {
                Bucket& b = p->buckets[k];
                b.batch = (int)b.mats.size();
                b.slot_base = slots;
                slots += b.batch;
                const size_t xparts = b.split == 2 ? 2 : 1, rparts = b.split ? 2 : 1;
                if (sharded) continue;   // RowNorm only: no X0 or r x r buffers
                o_ut[k] = rtake((size_t)b.batch * b.r * b.ldu * 2 * xparts);
                if (restarts) o_ut1[k] = rtake((size_t)b.batch * b.r * b.ldu * 2 * xparts);
                if (b.batched()) {
                    const size_t rr = (size_t)b.batch * b.r * b.ldr * 2 * rparts;
                    o_rr[k] = rtake(rr);   // G0 (fp16, scaled)
                    for (int q = 0; q < 5; ++q) rtake(rr);   // G1, P, T, Q0, Q1
                    o_qb[k] = rtake(rr);   // bf16 Q for the final product
                }
            }
            region_bytes = std::max(region_bytes, roff);
        }
    }
    L.o_region = take(std::max<size_t>(region_bytes, 256));
    for (int i = 0; i < n; ++i) {
        MatDev& md = p->mats[i];
        const Bucket& b = p->buckets[p->mat_bucket[i]];
        md.slot = b.slot_base + p->mat_item[i];
        md.ldu = b.ldu;
        md.x_split = b.split == 2 ? 1 : 0;   // hi part of item i at 2i, lo at 2i + 1
        md.ut_off = (long long)(o_ut[p->mat_bucket[i]] / 2) +
                    (long long)p->mat_item[i] * b.r * b.ldu * (md.x_split ? 2 : 1);
    }
    p->ws_bytes = off;
    // the packing counts the region exactly, so a cap is never exceeded; kept as a guard
    if (cap > 0 && (long long)off > cap) return MUON_ERR_OOM;
    return MUON_OK;
}

}  // namespace muon_impl

void muon::record_cuda_error(cudaError_t e) { muon_impl::last_cuda_error() = e; }

extern "C" {

const char* muon_last_error_detail(void) {
    return last_cuda_error() == cudaSuccess ? "no CUDA error recorded" : cudaGetErrorString(last_cuda_error());
}

const char* muon_status_string(muon_status s) {
    switch (s) {
        case MUON_OK: return "MUON_OK";
        case MUON_ERR_INVALID_ARG: return "MUON_ERR_INVALID_ARG: invalid argument";
        case MUON_ERR_UNSUPPORTED: return "MUON_ERR_UNSUPPORTED: unsupported dtype or size";
        case MUON_ERR_OOM: return "MUON_ERR_OOM: workspace allocation failed";
        case MUON_ERR_CUDA: return "MUON_ERR_CUDA: CUDA runtime or launch error";
        case MUON_ERR_TIMEOUT: return "MUON_ERR_TIMEOUT: a bounded device wait expired";
        case MUON_ERR_NONFINITE: return "MUON_ERR_NONFINITE: a non-finite input norm (opts.check_finite)";
    }
    return "MUON_ERR_UNKNOWN";
}

// Everything of muon_plan_create after the argument checks.  On failure it frees p;
// a host allocation that throws leaves p to the caller.
static muon_status plan_build(muon_plan_s* p, const muon_shape* shapes, int32_t n, muon_dtype grad_dtype,
                              const muon_plan_opts* opts, muon_plan* out) {
    if (cudaGetDevice(&p->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess ||
        !encode_fn()) {
        free_plan(p);
        return MUON_ERR_CUDA;
    }
    p->gdt = grad_dtype;
    if (opts) p->opts = *opts;
    p->shapes.assign(shapes, shapes + n);
    if (p->opts.full_rows) p->full_rows.assign(p->opts.full_rows, p->opts.full_rows + n);
    if (p->opts.precision_of) p->prec_of.assign(p->opts.precision_of, p->opts.precision_of + n);
    p->opts.full_rows = nullptr;   // read during creation only
    p->opts.precision_of = nullptr;

    Layout L;
    {
        const muon_status st = plan_layout(p, L);
        if (st != MUON_OK) {
            free_plan(p);
            return st;
        }
    }
    const bool restarts = L.restarts;
    if (cudaMalloc(&p->ws, p->ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        free_plan(p);
        return MUON_ERR_OOM;
    }
    char* base = static_cast<char*>(p->ws);
    p->ut = reinterpret_cast<__nv_bfloat16*>(base + L.o_region);
    p->d_mats = reinterpret_cast<MatDev*>(base + L.o_mats);
    p->partials = reinterpret_cast<float*>(base + L.o_part);
    p->cpartials = reinterpret_cast<float*>(base + L.o_cpart);
    p->rowinv = reinterpret_cast<float*>(base + L.o_inv);
    p->alpha = reinterpret_cast<float*>(base + L.o_alpha);
    p->status = reinterpret_cast<int*>(base + L.o_status);
    p->d_transposed = reinterpret_cast<unsigned char*>(base + L.o_tr);
    p->d_ptrs = reinterpret_cast<void**>(base + L.o_ptrs);
    p->ones = reinterpret_cast<float*>(base + L.o_ones);
    p->diff = reinterpret_cast<double*>(base + L.o_diff);
    p->d_wmap = reinterpret_cast<CUtensorMap*>(base + L.o_wmap);
    p->d_wmap_ok = reinterpret_cast<unsigned char*>(base + L.o_wmap_ok);

    std::vector<unsigned char> tr(n);
    for (int i = 0; i < n; ++i) tr[i] = (unsigned char)p->mats[i].transposed;
    bool ok = cudaMemcpy(p->d_mats, p->mats.data(), sizeof(MatDev) * n, cudaMemcpyHostToDevice) == cudaSuccess;
    ok = ok && cudaMemcpy(p->d_transposed, tr.data(), n, cudaMemcpyHostToDevice) == cudaSuccess;
    ok = ok && cudaMemset(p->status, 0, sizeof(int)) == cudaSuccess;
    ok = ok && cudaMemset(p->rowinv, 0, L.o_alpha - L.o_inv) == cudaSuccess;
    ok = ok && cudaMemset(p->d_ptrs, 0, sizeof(void*) * 3 * n) == cudaSuccess;
    {
        const std::vector<float> one(n, 1.f);
        ok = ok && cudaMemcpy(p->ones, one.data(), sizeof(float) * n, cudaMemcpyHostToDevice) == cudaSuccess;
    }

    // launch lists (int lists then long long prefixes, carved from their slices)
    int* list_cursor = reinterpret_cast<int*>(base + L.o_lists);
    long long* prefix_cursor = reinterpret_cast<long long*>(base + L.o_prefix);
    auto upload_list = [&](const std::vector<int>& v, ListDev& d, int kind) {
        d.list = list_cursor;
        d.blk = prefix_cursor;
        d.n = (int)v.size();
        list_cursor += std::max<size_t>(v.size(), 1);
        prefix_cursor += v.size() + 1;
        std::vector<long long> pre(v.size() + 1, 0);
        for (size_t j = 0; j < v.size(); ++j) {
            const MatDev& md = p->mats[v[j]];
            long long nb = 0;
            switch (kind) {
                case 0: case 1: nb = md.nblk; break;
                case 2: nb = 1; break;
                case 3: nb = md.m; break;
                case 4: nb = ceil_div(md.m, kColSlab) * ceil_div(md.n, kColWidth); break;
                case 5: nb = ceil_div(md.n, kElemThreads); break;
                case 6: nb = ceil_div(md.m * md.n, kApplyElemsPerBlock); break;
            }
            pre[j + 1] = pre[j] + nb;
        }
        d.blocks = pre.back();
        if (ok && !v.empty()) ok = cudaMemcpy(d.list, v.data(), sizeof(int) * v.size(), cudaMemcpyHostToDevice) == cudaSuccess;
        if (ok) ok = cudaMemcpy(d.blk, pre.data(), sizeof(long long) * pre.size(), cudaMemcpyHostToDevice) == cudaSuccess;
    };
    for (auto& ch : p->chunks) {
        std::vector<int> rows, tiles, all;
        for (int k : ch.buckets)
            for (int i : p->buckets[k].mats) {
                (p->mats[i].transposed ? tiles : rows).push_back(i);
                all.push_back(i);
            }
        upload_list(rows, ch.mom_rows, 0);
        upload_list(tiles, ch.mom_tiles, 1);
        upload_list(all, ch.all, 2);
        for (int cl = 0; cl < kRowClasses; ++cl) {
            std::vector<int> rc;
            for (int i : rows)
                if (rownorm_row_class(p->mats[i].n) == cl) rc.push_back(i);
            upload_list(rc, ch.rn_rows[cl], 3);
        }
        upload_list(tiles, ch.rn_stats, 4);
        upload_list(tiles, ch.rn_final, 5);
        upload_list(tiles, ch.rn_apply, 6);
    }
    for (int cl = 0; cl < kRowClasses; ++cl) {
        std::vector<int> rc;
        for (int i : L.rnr_list)
            if (rownorm_row_class(p->mats[i].n) == cl) rc.push_back(i);
        upload_list(rc, p->rn_rows[cl], 3);
    }
    upload_list(L.rnc_list, p->rn_stats, 4);
    upload_list(L.rnc_list, p->rn_final, 5);
    upload_list(L.rnc_list, p->rn_apply, 6);

    int* item_cursor = reinterpret_cast<int*>(base + L.o_items);
    size_t odbg_off = L.o_odbg;
    for (size_t k = 0; ok && k < p->buckets.size(); ++k) {
        Bucket& b = p->buckets[k];
        b.d_item_mat = item_cursor;
        item_cursor += b.batch;
        ok = cudaMemcpy(b.d_item_mat, b.mats.data(), sizeof(int) * b.batch, cudaMemcpyHostToDevice) == cudaSuccess;
        if (!p->full_rows.empty()) continue;   // dim-0 shard plans run RowNorm only: no NS buffers
        b.gscale = std::ldexp(1.f, (int)std::lround(std::log2((double)b.r)));
        b.ut_off = (long long)(L.o_ut[k] / 2);
        if (p->opts.keep_update) {
            b.Odbg = reinterpret_cast<float*>(base + odbg_off);
            odbg_off += (size_t)round_up((long long)b.batch * b.r * b.c * 4, 256);
        }
        __nv_bfloat16* ut = p->ut + b.ut_off;
        const int xb = b.batch * (b.split == 2 ? 2 : 1);   // X items (two parts per matrix at level 2)
        const int rb = b.batch * (b.split ? 2 : 1);        // r x r items
        ok = ok && make_map(&b.ut_a, ut, true, b.c, b.r, xb, b.ldu, 64, kBM);
        ok = ok && make_map(&b.ut_b, ut, true, b.c, b.r, xb, b.ldu, 64, kBN);
        ok = ok && make_map(&b.ut_mn, ut, true, b.c, b.r, xb, b.ldu, 64, 64);
        const bool aligned4 = b.batched() && !b.split && b.r % 64 == 0 && b.c % 64 == 0;
        if (aligned4) {
            ok = ok && make_map4(&b.utk, ut, true, b.c, b.r, b.batch, b.ldu, 128, 1);
            ok = ok && make_map4(&b.utt, ut, true, b.c, b.r, b.batch, b.ldu, 64, 2);
        }
        if (restarts) {
            b.ut1_off = (long long)(L.o_ut1[k] / 2);
            __nv_bfloat16* ut1 = p->ut + b.ut1_off;
            ok = ok && make_map(&b.ut1_a, ut1, true, b.c, b.r, xb, b.ldu, 64, kBM);
            ok = ok && make_map(&b.ut1_b, ut1, true, b.c, b.r, xb, b.ldu, 64, kBN);
            ok = ok && make_map(&b.ut1_mn, ut1, true, b.c, b.r, xb, b.ldu, 64, 64);
            if (aligned4) {
                ok = ok && make_map4(&b.ut1k, ut1, true, b.c, b.r, b.batch, b.ldu, 128, 1);
                ok = ok && make_map4(&b.ut1t, ut1, true, b.c, b.r, b.batch, b.ldu, 64, 2);
            }
        }
        if (!b.batched()) continue;   // the one-CTA kernels keep their r x r operands on chip
        const size_t rr = (size_t)rb * b.r * b.ldr;
        const size_t step = (size_t)round_up((long long)rr * 2, 256);
        char* rbase = base + L.o_region + L.o_rr[k];
        b.G[0] = reinterpret_cast<__half*>(rbase);
        b.G[1] = reinterpret_cast<__half*>(rbase + step);
        b.P = reinterpret_cast<__half*>(rbase + 2 * step);
        b.T = reinterpret_cast<__half*>(rbase + 3 * step);
        b.Q[0] = reinterpret_cast<__half*>(rbase + 4 * step);
        b.Q[1] = reinterpret_cast<__half*>(rbase + 5 * step);
        b.Qb = reinterpret_cast<__nv_bfloat16*>(base + L.o_region + L.o_qb[k]);
        ok = ok && make_map(&b.qb_a, b.Qb, true, b.r, b.r, rb, b.ldr, 64, kBM);
        for (int g = 0; g < 2; ++g) {
            ok = ok && make_map(&b.ga[g], b.G[g], false, b.r, b.r, rb, b.ldr, 64, kBM);
            ok = ok && make_map(&b.gb[g], b.G[g], false, b.r, b.r, rb, b.ldr, 64, kBN);
            ok = ok && make_map(&b.qb[g], b.Q[g], false, b.r, b.r, rb, b.ldr, 64, kBN);
            ok = ok && make_map(&b.qa[g], b.Q[g], false, b.r, b.r, rb, b.ldr, 64, kBM);
        }
        ok = ok && make_map(&b.pa, b.P, false, b.r, b.r, rb, b.ldr, 64, kBM);
        ok = ok && make_map(&b.pb, b.P, false, b.r, b.r, rb, b.ldr, 64, kBN);
        ok = ok && make_map(&b.tb, b.T, false, b.r, b.r, rb, b.ldr, 64, kBN);
        ok = ok && make_map(&b.ta, b.T, false, b.r, b.r, rb, b.ldr, 64, kBM);
        for (int g = 0; g < 2; ++g) {
            ok = ok && make_out_map(&b.og[g], b.G[g], false, b.r, rb, b.ldr);
            ok = ok && make_out_map(&b.oq[g], b.Q[g], false, b.r, rb, b.ldr);
        }
        ok = ok && make_out_map(&b.op, b.P, false, b.r, rb, b.ldr);
        ok = ok && make_out_map(&b.ot, b.T, false, b.r, rb, b.ldr);
        ok = ok && make_out_map(&b.oqb, b.Qb, true, b.r, rb, b.ldr);
        if (aligned4) {
            auto kt = [&](CUtensorMap* k, CUtensorMap* t, void* buf, bool bf) {
                return make_map4(k, buf, bf, b.r, b.r, b.batch, b.ldr, 128, 1) &&
                       make_map4(t, buf, bf, b.r, b.r, b.batch, b.ldr, 64, 2);
            };
            for (int g = 0; g < 2; ++g) {
                ok = ok && kt(&b.gk[g], &b.gt[g], b.G[g], false);
                ok = ok && kt(&b.qk[g], &b.qt[g], b.Q[g], false);
            }
            ok = ok && kt(&b.pk, &b.pt, b.P, false) && kt(&b.tk, &b.tt, b.T, false) && kt(&b.qbk, &b.qbt, b.Qb, true);
        }
    }
    ok = ok && cudaMallocHost(&p->h_pinned, sizeof(void*) * 3 * n) == cudaSuccess;
    ok = ok && cudaMallocHost(&p->h_wmap, (sizeof(CUtensorMap) + 1) * n) == cudaSuccess;
    ok = ok && cudaMemset(p->d_wmap_ok, 0, n) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&p->upload_ev, cudaEventDisableTiming) == cudaSuccess;
    ok = ok && gemm_prepare(p->device) == cudaSuccess;
    ok = ok && ns_f32_prepare() == cudaSuccess;
    if (ok && !p->opts.single_sm_gemm) {
        int clusters = 0;
        ok = gemm2_max_clusters(&clusters) == cudaSuccess;
        p->pair_clusters = clusters;
    }
    for (auto& ch : p->chunks) {   // lower-triangle storage where the 4-D operand view is exact
        bool aligned = true;
        for (int k : ch.buckets) {
            const Bucket& b = p->buckets[k];
            if (b.batched() && b.r > kBM) aligned = aligned && !b.split && b.r % 64 == 0 && b.c % 64 == 0;
        }
        ch.lower_ok = p->pair_clusters > 0 && aligned;
        ch.lower = ch.lower_ok && !p->opts.full_symmetric;
    }
    if (ok && p->pair_clusters > 1) {
        bool any = false;
        for (auto& ch : p->chunks) {
            double fused_bytes = 0, chain_flops = 0;
            for (int k : ch.buckets) {
                const Bucket& b = p->buckets[k];
                const double r = b.r, c = b.c;
                if (b.fused)
                    fused_bytes += 12.0 * r * c * b.batch;
                else if (b.batched())
                    chain_flops += (3.0 * r * r * c + 17.0 * r * r * r) * b.batch;
            }
            if (fused_bytes > 0 && chain_flops > 0) {
                const int kmax = std::min(p->pair_clusters - 1, (p->sm_count - 2) / 2);
                ch.mixed = true;
                ch.chain_est = std::max(std::min(choose_chain_clusters(fused_bytes, chain_flops, p->pair_clusters),
                                                 kmax), 0);
                const int k = p->opts.chain_clusters == 0 ? ch.chain_est
                                                          : std::min(std::max(p->opts.chain_clusters, 0), kmax);
                ch.chain_clusters = k;
                any = true;   // the second stream also serves muon_plan_tune's candidates
            }
        }
        if (any)
            ok = cudaStreamCreateWithFlags(&p->s2, cudaStreamNonBlocking) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p->fork_ev, cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p->join_ev, cudaEventDisableTiming) == cudaSuccess;
    }
    ok = ok && cudaDeviceSynchronize() == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        free_plan(p);
        return MUON_ERR_CUDA;
    }
    p->h_cache.assign(3 * n, nullptr);
    *out = p;
    return MUON_OK;
}

muon_status muon_plan_create(const muon_shape* shapes, int32_t n, muon_dtype grad_dtype, const muon_plan_opts* opts,
                             muon_plan* out) {
    if (!out) return MUON_ERR_INVALID_ARG;
    *out = nullptr;
    const muon_status bad = check_plan_args(shapes, n, grad_dtype, opts);
    if (bad != MUON_OK) return bad;
    muon_plan_s* p = new (std::nothrow) muon_plan_s();
    if (!p) return MUON_ERR_OOM;
    try {
        return plan_build(p, shapes, n, grad_dtype, opts, out);
    } catch (...) {   // std::vector's bad_alloc / length_error: host memory
        free_plan(p);
        return MUON_ERR_OOM;
    }
}

muon_status muon_partition(const muon_shape* shapes, int32_t n, int32_t world, const double* cost, int32_t* owner,
                           double* load) {
    if (!shapes || n <= 0 || !owner || world < 1 || world > 65536) return MUON_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        if (shapes[i].rows <= 0 || shapes[i].cols <= 0 || shapes[i].rows > kMaxDim || shapes[i].cols > kMaxDim)
            return MUON_ERR_INVALID_ARG;
        if (cost && !(std::isfinite(cost[i]) && cost[i] >= 0.0)) return MUON_ERR_INVALID_ARG;
    }
    try {
        std::vector<double> c(n);
        for (int i = 0; i < n; ++i) {
            if (cost) {
                c[i] = cost[i];
                continue;
            }
            const double r = (double)std::min(shapes[i].rows, shapes[i].cols);
            const double cc = (double)std::max(shapes[i].rows, shapes[i].cols);
            const double t_mem = 24.0 * r * cc / 6.8e12;
            const double t_tc = r <= kSmallMaxR ? 0.0 : (3.0 * r * r * cc + 17.0 * r * r * r) / 1.5e15;
            c[i] = std::max(t_mem, t_tc);
        }
        std::vector<int> order(n);
        for (int i = 0; i < n; ++i) order[i] = i;
        std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return c[a] > c[b]; });
        std::vector<double> l(world, 0.0);
        for (int i : order) {
            int best = 0;
            for (int r = 1; r < world; ++r)
                if (l[r] < l[best]) best = r;
            owner[i] = best;
            l[best] += c[i];
        }
        if (load)
            for (int r = 0; r < world; ++r) load[r] = l[r];
        return MUON_OK;
    } catch (...) {   // host memory
        return MUON_ERR_OOM;
    }
}

muon_status muon_plan_workspace_size(const muon_shape* shapes, int32_t n, muon_dtype grad_dtype,
                                     const muon_plan_opts* opts, int64_t* bytes, int32_t* n_buckets,
                                     int32_t* n_chunks) {
    const muon_status bad = check_plan_args(shapes, n, grad_dtype, opts);
    if (bad != MUON_OK) return bad;
    try {
        muon_plan_s plan;   // host fields only: nothing is created on the device
        if (opts) plan.opts = *opts;
        plan.shapes.assign(shapes, shapes + n);
        if (plan.opts.full_rows) plan.full_rows.assign(plan.opts.full_rows, plan.opts.full_rows + n);
        if (plan.opts.precision_of) plan.prec_of.assign(plan.opts.precision_of, plan.opts.precision_of + n);
        plan.opts.full_rows = nullptr;
        plan.opts.precision_of = nullptr;
        Layout L;
        const muon_status st = plan_layout(&plan, L);
        if (st != MUON_OK) return st;
        if (bytes) *bytes = (int64_t)plan.ws_bytes;
        if (n_buckets) *n_buckets = (int32_t)plan.buckets.size();
        if (n_chunks) *n_chunks = (int32_t)plan.chunks.size();
        return MUON_OK;
    } catch (...) {   // host memory
        return MUON_ERR_OOM;
    }
}

void muon_plan_destroy(muon_plan p) {
    if (!p) return;
    cudaDeviceSynchronize();
    free_plan(p);
}

}  // extern "C"
