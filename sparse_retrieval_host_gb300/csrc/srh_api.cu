// Host side of the C ABI: context creation, validation, pinned pools, launches,
// the attention's static work plan and the native host loop (srh_hostloop_*).
//
// Guards restated from PocketLLM "FlashMemory 1M 上下文显存优化使用文档":
//   * section 关键参数调优 item 1 and 故障排查 error 2: GPU_CHUNKS must be >=
//     index_topk unless the test-only reduction flag is set;
//   * section 关键参数调优 item 2 and 故障排查 error 3: the pinned pools must fit
//     the cap, reported as "required_mib=... cap_mib=...";
//   * section 故障排查, the swap auto-disable note: a layer whose capacity fits in
//     the staging slots does not swap (its chunk c lives in staging row c);
//   * section 故障排查 error 4: a selected chunk that was never stored is an error
//     (raised on the device, reported by srh_check_error).
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>

#include "srh_internal.cuh"

using namespace srh;

namespace {

std::string g_create_error;

const char* kErrText[] = {
    "ok",
    "invalid argument",
    "pinned cache exceeds cap",
    "selected chunk before it was stored",
    "CUDA error",
    "device wait timed out",
    "out of memory",
    "index out of bounds on the device",
    "attention operand beyond the fp16 range",
};

int fail(srh_ctx* ctx, int code, const std::string& msg) {
    if (ctx) ctx->last_error = msg;
    else g_create_error = msg;
    return code;
}

int cuda_fail(srh_ctx* ctx, cudaError_t e, const char* where) {
    std::string m = std::string(where) + ": " + cudaGetErrorString(e);
    return fail(ctx, SRH_ERR_CUDA, m);
}

#define SRH_CUDA(ctx, call)                                   \
    do {                                                      \
        cudaError_t e_ = (call);                              \
        if (e_ != cudaSuccess) return cuda_fail(ctx, e_, #call); \
    } while (0)

long long cap_of(long long ctx_len, int ratio) { return (ctx_len + ratio - 1) / ratio; }


int validate_config(const srh_config* c, std::string* why) {
    if (!c) { *why = "config is NULL"; return SRH_ERR_INVALID; }
    if (c->batch < 1) { *why = "batch must be >= 1"; return SRH_ERR_INVALID; }
    if (c->n_layers < 1) { *why = "n_layers must be >= 1"; return SRH_ERR_INVALID; }
    if (c->kv_dim != SRH_KV_DIM) { *why = "kv_dim must be 512"; return SRH_ERR_INVALID; }
    if (c->window != SRH_WINDOW) { *why = "window must be 128"; return SRH_ERR_INVALID; }
    if (c->gpu_chunks < 1 || c->gpu_chunks > kMaxGpuChunks) {
        *why = "gpu_chunks must be in [1, 4096]"; return SRH_ERR_INVALID;
    }
    if (c->index_topk < 1 || c->index_topk > kMaxSelect) {
        *why = "index_topk must be in [1, 4096]"; return SRH_ERR_INVALID;
    }
    if (c->gpu_chunks < c->index_topk && !c->allow_topk_reduction) {
        *why = "POCKETLLM_GGUF_KV_SWAP_GPU_CHUNKS must be >= index_topk";
        return SRH_ERR_INVALID;
    }
    if (c->src_ratio < 1) { *why = "src_ratio must be >= 1"; return SRH_ERR_INVALID; }
    if (!c->layer_ratio) { *why = "layer_ratio is NULL"; return SRH_ERR_INVALID; }
    if (c->context_len < 1) { *why = "context_len must be >= 1"; return SRH_ERR_INVALID; }
    const long long n_src = cap_of(c->context_len, c->src_ratio);
    if (n_src > (1LL << 30)) { *why = "context too long"; return SRH_ERR_INVALID; }
    for (int l = 0; l < c->n_layers; ++l) {
        const int r = c->layer_ratio[l];
        if (r < c->src_ratio || r % c->src_ratio != 0) {
            *why = "every layer ratio must be a multiple of src_ratio";
            return SRH_ERR_INVALID;
        }
    }
    const int S = c->max_select > 0 ? c->max_select : c->index_topk;
    if (S < c->index_topk || S > kMaxSelect) {
        *why = "max_select must be in [index_topk, 4096]"; return SRH_ERR_INVALID;
    }
    if (lru_smem_bytes(S, c->gpu_chunks) > 227 * 1024) {
        *why = "max_select + gpu_chunks too large for one LRU block"; return SRH_ERR_INVALID;
    }
    return SRH_OK;
}

unsigned long long pinned_bytes(const srh_config* c) {
    unsigned long long t = 0;
    for (int l = 0; l < c->n_layers; ++l)
        t += (unsigned long long)c->batch * cap_of(c->context_len, c->layer_ratio[l]) *
             SRH_KV_DIM * sizeof(float);
    return t;
}

void free_ctx(srh_ctx* ctx) {
    if (!ctx) return;
    cudaDeviceSynchronize();
    for (float* p : ctx->pool_host) if (p) cudaFreeHost(p);
    for (auto& ld : ctx->h_layers) {
        cudaFree(ld.host_ready);
        cudaFree(ld.slot_of);
        cudaFree(ld.slot_logical);
        cudaFree(ld.lru_order);
        cudaFree(ld.adapt);
    }
    cudaFree(ctx->d_layers);
    cudaFree(ctx->d_swap_layers);
    cudaFree(ctx->d_stats);
    cudaFree(ctx->d_err);
    cudaFree(ctx->d_hist);
    cudaFree(ctx->d_cand);
    cudaFree(ctx->d_cand_cnt);
    cudaFree(ctx->d_miss);
    cudaFree(ctx->d_miss_count);
    cudaFree(ctx->d_sink);
    cudaFree(ctx->d_segs);
    cudaFree(ctx->d_cta_begin);
    cudaFree(ctx->d_part_o);
    cudaFree(ctx->d_part_ml);
    cudaFree(ctx->d_merges);
    cudaFree(ctx->d_merge_cnt);
    if (ctx->ev_resolved) cudaEventDestroy(ctx->ev_resolved);
    if (ctx->ev_gathered) cudaEventDestroy(ctx->ev_gathered);
    delete ctx;
}

// The static attention plan of one lsa_attend scope (the pairs (layer, seq)
// of `layers`). A pair holds 128 window rows (fp32, 2 KiB each) plus at most
// min(S, cap) staged rows (fp16, 1 KiB each). A CTA runs its rows in tiles of
// up to 128 rows, each tile a serial chain (rows in, two products, softmax);
// it holds ~218 KB of shared memory and 512 threads of 128 registers, so one
// runs per SM, and a plan never has more CTAs than SMs (every CTA becomes
// resident, which the merge waits rely on).
//   * One wave, when every pair's tiles fit on CTAs of their own: each pair is
//     cut into k chunks of at most one tile, balanced by bytes (the largest
//     chunk as small as k chunks of <= 128 rows allow); k starts at the pair's
//     tile count and the pairs with the largest chunks get one more CTA each,
//     all together, while the SMs last. No CTA starts a second pair (a second
//     query load and epilogue).
//   * Otherwise stream-K: the scope's tiles, in (layer, seq, row) order and
//     weighted by their bytes, cut into at most SMs contiguous ranges of
//     equal bytes to the nearest tile.
// A pair spread over several CTAs is merged by those CTAs, each taking one
// share, once all its partials are written. CTAs whose first tile holds only
// window rows come first: that tile needs no earlier kernel's output, and the
// CTAs launched first run it while those kernels finish. The plan depends only
// on the configuration, so the same rows give the same bits whichever slots
// hold them.
void plan_scope(srh_ctx* ctx, const std::vector<int>& layers, std::vector<AttnSeg>* segs,
                std::vector<int>* cta_begin, std::vector<MergeItem>* merges, AttnPlan* plan) {
    const int B = ctx->B;
    const long long N = ctx->sm_count;
    constexpr long long kT = kAttnTile;
    std::vector<int> lbs;
    std::vector<long long> rows;
    for (int l : layers)
        for (int b = 0; b < B; ++b) {
            lbs.push_back(l * B + b);
            rows.push_back(kWindow + std::min<long long>(ctx->S, ctx->caps[l]));
        }
    const size_t P = lbs.size();
    // KiB of rows [0, r) of a pair: window rows 2, staged rows 1
    auto cost_to = [](long long r) { return r <= kWindow ? 2 * r : 2LL * kWindow + (r - kWindow); };
    // Cut rows [0, n) into chunks of at most kT rows and M KiB, each as long as
    // it can be; returns the chunk count (or -1 if a row exceeds M) and the ends.
    auto pack = [&](long long n, long long M, std::vector<long long>* ends) -> long long {
        long long r = 0, c = 0;
        while (r < n) {
            const long long w = r < kWindow ? std::min({kWindow - r, M / 2, kT, n - r}) : 0;
            long long e = r + w, room = M - 2 * w;
            if (e >= kWindow && e - r < kT) e += std::min({n - e, room, kT - (e - r)});
            if (e == r) return -1;
            if (ends) ends->push_back(e);
            r = e;
            ++c;
        }
        return c;
    };
    // the smallest largest-chunk of a pair cut into at most k such chunks
    auto best = [&](long long n, long long k) {
        long long lo = 2, hi = 2 * kT;
        while (lo < hi) {
            const long long m = (lo + hi) / 2;
            const long long c = pack(n, m, nullptr);
            if (c >= 0 && c <= k) hi = m;
            else lo = m + 1;
        }
        return lo;
    };
    struct Raw { size_t p; int r0, r1; };
    std::vector<Raw> raw;
    std::vector<int> begin;
    long long tiles_all = 0;
    for (long long r : rows) tiles_all += (r + kT - 1) / kT;
    const bool one_wave = tiles_all <= N;
    if (one_wave) {
        // A CTA's fixed costs (its queries, the dependent-load chain, the epilogue
        // and the merge wait) outweigh the rows below about one staged tile: a
        // pair gets more chunks than tiles only down to 128 KiB each, and at most
        // attend_max_splits() chunks (what a merge combines).
        std::vector<long long> k(P), kmax(P), top(P);
        long long used = 0;
        for (size_t p = 0; p < P; ++p) {
            k[p] = (rows[p] + kT - 1) / kT;
            kmax[p] = std::max(k[p], std::min<long long>(attend_max_splits(), cost_to(rows[p]) / 128));
            top[p] = best(rows[p], k[p]);
            used += k[p];
        }
        for (;;) {
            long long mx = 0;
            for (size_t p = 0; p < P; ++p) mx = std::max(mx, top[p]);
            std::vector<size_t> at;
            bool room = true;
            for (size_t p = 0; p < P; ++p)
                if (top[p] == mx) {
                    at.push_back(p);
                    room = room && k[p] < kmax[p];
                }
            if (!room || used + (long long)at.size() > N) break;
            for (size_t p : at) top[p] = best(rows[p], ++k[p]);
            used += (long long)at.size();
        }
        for (size_t p = 0; p < P; ++p) {
            std::vector<long long> ends;
            pack(rows[p], top[p], &ends);
            long long prev = 0;
            for (long long e : ends) {
                begin.push_back((int)raw.size());
                raw.push_back(Raw{p, (int)prev, (int)e});
                prev = e;
            }
        }
    } else {
        // stream-K over whole tiles, weighted by bytes
        struct Tile { size_t p; long long r0, r1, c; };
        std::vector<Tile> tl;
        long long total = 0;
        for (size_t p = 0; p < P; ++p)
            for (long long r0 = 0; r0 < rows[p]; r0 += kT) {
                const long long r1 = std::min(r0 + kT, rows[p]);
                tl.push_back(Tile{p, r0, r1, cost_to(r1) - cost_to(r0)});
                total += tl.back().c;
            }
        const long long n = std::min<long long>(N, (long long)tl.size());
        size_t t = 0;
        long long acc = 0;
        for (long long j = 0; j < n && t < tl.size(); ++j) {
            // the range ends at the tile boundary nearest to (j + 1) / n of the bytes,
            // leaving at least one tile for each remaining range
            const long long goal = (j + 1) * total / n;
            size_t e = t + 1;
            long long a = acc + tl[t].c;
            while (e < tl.size() && (long long)(tl.size() - e) > n - j - 1 && 2 * (a + tl[e].c) <= 2 * goal + tl[e].c) {
                a += tl[e].c;
                ++e;
            }
            if (j == n - 1) {
                for (; e < tl.size(); ++e) a += tl[e].c;
            }
            begin.push_back((int)raw.size());
            for (size_t i = t; i < e; ++i) {
                if (!raw.empty() && (int)raw.size() > begin.back() && raw.back().p == tl[i].p &&
                    raw.back().r1 == tl[i].r0)
                    raw.back().r1 = (int)tl[i].r1;
                else
                    raw.push_back(Raw{tl[i].p, (int)tl[i].r0, (int)tl[i].r1});
            }
            t = e;
            acc = a;
        }
    }
    plan->seg0 = (int)segs->size();
    plan->cta0 = (int)cta_begin->size();
    plan->merge0 = (int)merges->size();
    plan->n_ctas = (int)begin.size();
    plan->one_wave = one_wave ? 1 : 0;
    // pairs with more than one segment write partials, in row order
    std::vector<int> n_parts(P, 0), merge_of(P, -1), seen(P, 0);
    for (const Raw& x : raw) ++n_parts[x.p];
    int slot = 0;
    for (const Raw& x : raw) {
        if (n_parts[x.p] > 1 && merge_of[x.p] < 0) {
            merge_of[x.p] = (int)merges->size() - plan->merge0;
            merges->push_back(MergeItem{lbs[x.p], slot, n_parts[x.p], 0});
            slot += n_parts[x.p];
        }
    }
    std::vector<AttnSeg> tmp;
    for (const Raw& x : raw) {
        const int mi = merge_of[x.p];
        int sl = -1, part = 0;
        if (mi >= 0) {
            part = seen[x.p]++;
            sl = (*merges)[plan->merge0 + mi].first + part;
        }
        tmp.push_back(AttnSeg{lbs[x.p], x.r0, x.r1, sl, mi, part});
    }
    // CTAs whose first tile holds only window rows first, otherwise in plan order
    const int nct = (int)begin.size();
    auto window_first = [&](int j) {
        const Raw& x = raw[begin[j]];
        return x.r0 < kWindow && (x.r0 == 0 || x.r1 <= kWindow);
    };
    std::vector<int> order;
    for (int pass = 0; pass < 2; ++pass)
        for (int j = 0; j < nct; ++j)
            if (window_first(j) == (pass == 0)) order.push_back(j);
    for (int j : order) {
        const int e = j + 1 < nct ? begin[j + 1] : (int)raw.size();
        cta_begin->push_back((int)segs->size() - plan->seg0);
        for (int i = begin[j]; i < e; ++i) segs->push_back(tmp[i]);
    }
    cta_begin->push_back((int)segs->size() - plan->seg0);
    plan->n_segs = (int)raw.size();
    plan->n_merges = (int)merges->size() - plan->merge0;
    plan->n_slots = slot;
}

// The plan's invariants, which the kernel relies on: at most one CTA per SM;
// every pair of the scope covered once, in row order, by its segments (parts
// 0 .. ns-1 of a split pair contiguous from row 0, within the merge limit); a
// CTA takes part in at most attend_max_duties() split pairs.
bool plan_valid(const srh_ctx* ctx, const std::vector<int>& layers, const std::vector<AttnSeg>& segs,
                const std::vector<int>& cta_begin, const std::vector<MergeItem>& merges, const AttnPlan& pl) {
    if (pl.n_ctas < 1 || pl.n_ctas > ctx->sm_count) return false;
    std::vector<std::vector<AttnSeg>> by_lb((size_t)ctx->L * ctx->B);
    for (int j = 0; j < pl.n_ctas; ++j) {
        const int a = cta_begin[pl.cta0 + j], b = cta_begin[pl.cta0 + j + 1];
        if (a < 0 || b < a || b > pl.n_segs) return false;
        int duties = 0;
        for (int i = a; i < b; ++i) {
            const AttnSeg& g = segs[pl.seg0 + i];
            if (g.lb < 0 || g.lb >= ctx->L * ctx->B || g.r1 <= g.r0) return false;
            if (g.slot >= 0) ++duties;
            by_lb[g.lb].push_back(g);
        }
        if (duties > attend_max_duties()) return false;
    }
    if (cta_begin[pl.cta0] != 0 || cta_begin[pl.cta0 + pl.n_ctas] != pl.n_segs) return false;
    for (int l : layers)
        for (int b = 0; b < ctx->B; ++b) {
            std::vector<AttnSeg>& v = by_lb[(size_t)l * ctx->B + b];
            const long long rows = kWindow + std::min<long long>(ctx->S, ctx->caps[l]);
            if (v.empty()) return false;
            std::sort(v.begin(), v.end(), [](const AttnSeg& x, const AttnSeg& y) { return x.r0 < y.r0; });
            const int ns = (int)v.size();
            if (ns > attend_max_splits()) return false;
            for (int i = 0; i < ns; ++i) {
                if (v[i].r0 != (i == 0 ? 0 : v[i - 1].r1)) return false;
                if (ns == 1) {
                    if (v[i].slot >= 0) return false;
                    continue;
                }
                if (v[i].merge < 0 || v[i].merge >= pl.n_merges || v[i].part != i) return false;
                const MergeItem& m = merges[pl.merge0 + v[i].merge];
                if (m.ns != ns || m.lb != v[i].lb || v[i].slot != m.first + i || m.first + ns > pl.n_slots) return false;
            }
            if (v[ns - 1].r1 != rows) return false;
        }
    return true;
}

// Plans [0] for all layers and [1 + l] for layer l alone.
bool plan_attention(srh_ctx* ctx, std::vector<AttnSeg>* segs, std::vector<int>* cta_begin,
                    std::vector<MergeItem>* merges) {
    ctx->plans.assign(ctx->L + 1, AttnPlan{});
    std::vector<int> all(ctx->L);
    for (int l = 0; l < ctx->L; ++l) all[l] = l;
    plan_scope(ctx, all, segs, cta_begin, merges, &ctx->plans[0]);
    for (int l = 0; l < ctx->L; ++l) plan_scope(ctx, {l}, segs, cta_begin, merges, &ctx->plans[1 + l]);
    ctx->max_slots = 0;
    for (const AttnPlan& p : ctx->plans) ctx->max_slots = std::max(ctx->max_slots, p.n_slots);
    bool ok = plan_valid(ctx, all, *segs, *cta_begin, *merges, ctx->plans[0]);
    for (int l = 0; ok && l < ctx->L; ++l) ok = plan_valid(ctx, {l}, *segs, *cta_begin, *merges, ctx->plans[1 + l]);
    return ok;
}

}  // namespace

extern "C" {

const char* srh_error_string(int code) {
    if (code > 0 || code < -8) return "unknown error";
    return kErrText[-code];
}

const char* srh_last_error(srh_ctx* ctx) {
    return ctx ? ctx->last_error.c_str() : g_create_error.c_str();
}

int srh_pinned_required_bytes(const srh_config* cfg, unsigned long long* out) {
    std::string why;
    if (!out) return SRH_ERR_INVALID;
    const int rc = validate_config(cfg, &why);
    if (rc != SRH_OK) return fail(nullptr, rc, why);
    *out = pinned_bytes(cfg);
    return SRH_OK;
}

int srh_attend_plan_info(const srh_config* cfg, int sm_count, int layer, long long* info) {
    std::string why;
    if (!info || sm_count <= 0) return fail(nullptr, SRH_ERR_INVALID, "info is NULL or sm_count <= 0");
    const int rc = validate_config(cfg, &why);
    if (rc != SRH_OK) return fail(nullptr, rc, why);
    if (layer < -1 || layer >= cfg->n_layers) return fail(nullptr, SRH_ERR_INVALID, "layer out of range");
    srh_ctx* ctx = new (std::nothrow) srh_ctx();
    if (!ctx) return fail(nullptr, SRH_ERR_NOMEM, "host allocation failed");
    ctx->B = cfg->batch;
    ctx->L = cfg->n_layers;
    ctx->G = cfg->gpu_chunks;
    ctx->S = cfg->max_select > 0 ? cfg->max_select : cfg->index_topk;
    ctx->sm_count = sm_count;
    for (int l = 0; l < ctx->L; ++l) ctx->caps.push_back(cap_of(cfg->context_len, cfg->layer_ratio[l]));
    std::vector<AttnSeg> segs;
    std::vector<int> cta_begin;
    std::vector<MergeItem> merges;
    const bool ok = plan_attention(ctx, &segs, &cta_begin, &merges);
    const AttnPlan& pl = ctx->plans[layer + 1];
    long long worst = 0;
    for (int j = 0; j < pl.n_ctas; ++j) {
        long long c = 0;
        for (int i = cta_begin[pl.cta0 + j]; i < cta_begin[pl.cta0 + j + 1]; ++i) {
            const AttnSeg& g = segs[pl.seg0 + i];
            auto to = [](long long r) { return r <= kWindow ? 2 * r : 2LL * kWindow + (r - kWindow); };
            c += to(g.r1) - to(g.r0);
        }
        worst = std::max(worst, c);
    }
    info[0] = pl.n_ctas;
    info[1] = pl.n_segs;
    info[2] = pl.n_merges;
    info[3] = worst;
    info[4] = pl.one_wave;
    info[5] = ok ? 1 : 0;
    delete ctx;
    return SRH_OK;
}

int srh_create(const srh_config* cfg, srh_ctx** out) {
    if (!out) return fail(nullptr, SRH_ERR_INVALID, "out is NULL");
    *out = nullptr;
    std::string why;
    int rc = validate_config(cfg, &why);
    if (rc != SRH_OK) return fail(nullptr, rc, why);

    const unsigned long long need = pinned_bytes(cfg);
    if (cfg->pinned_cap_bytes && need > cfg->pinned_cap_bytes) {
        char buf[160];
        std::snprintf(buf, sizeof buf,
                      "POCKETLLM_GGUF_KV_SWAP pinned cache exceeds cap: required_mib=%llu cap_mib=%llu",
                      (need + (1ull << 20) - 1) >> 20,
                      (unsigned long long)(cfg->pinned_cap_bytes >> 20));
        return fail(nullptr, SRH_ERR_PINNED_CAP, buf);
    }

    srh_ctx* ctx = new (std::nothrow) srh_ctx();
    if (!ctx) return fail(nullptr, SRH_ERR_NOMEM, "host allocation failed");
    ctx->cfg = *cfg;
    ctx->B = cfg->batch;
    ctx->L = cfg->n_layers;
    ctx->G = cfg->gpu_chunks;
    ctx->S = cfg->max_select > 0 ? cfg->max_select : cfg->index_topk;
    ctx->n_src = cap_of(cfg->context_len, cfg->src_ratio);
    ctx->ratios.assign(cfg->layer_ratio, cfg->layer_ratio + cfg->n_layers);
    ctx->cfg.layer_ratio = nullptr;

    auto bail = [&](int code, const std::string& msg) {
        g_create_error = msg;
        free_ctx(ctx);
        return code;
    };
    cudaError_t e = cudaGetDevice(&ctx->device);
    if (e != cudaSuccess) return bail(SRH_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    e = cudaDeviceGetAttribute(&ctx->sm_count, cudaDevAttrMultiProcessorCount, ctx->device);
    if (e != cudaSuccess) return bail(SRH_ERR_CUDA, cudaGetErrorString(e));
    e = set_select_attrs();
    if (e == cudaSuccess) e = set_lru_attrs();
    if (e == cudaSuccess) e = set_attend_attrs();
    if (e == cudaSuccess) e = set_score_tc_attrs();
    if (e != cudaSuccess) return bail(SRH_ERR_CUDA, std::string("kernel attributes: ") + cudaGetErrorString(e));

    const int B = ctx->B, G = ctx->G;
    ctx->h_layers.resize(ctx->L);
    ctx->pool_host.assign(ctx->L, nullptr);
    ctx->pool_dev.assign(ctx->L, nullptr);
    ctx->ready_host.resize(ctx->L);
    ctx->resident_dirty.assign(ctx->L, 0);
    for (int l = 0; l < ctx->L; ++l) {
        const long long cap = cap_of(cfg->context_len, ctx->ratios[l]);
        ctx->caps.push_back(cap);
        ctx->swap.push_back(cap > G ? 1 : 0);
        LayerDev& ld = ctx->h_layers[l];
        ld = LayerDev{};
        ld.cap = cap;
        ld.ratio = ctx->ratios[l];
        ld.swap = cap > G ? 1 : 0;
        const size_t pool_bytes = (size_t)B * cap * kKvDim * sizeof(float);
        void* hp = nullptr;
        if ((cfg->flags & SRH_FLAG_TEST_FAIL_HOST_ALLOC) && l == ctx->L - 1) {
            return bail(SRH_ERR_NOMEM, "cudaHostAlloc failed (injected by SRH_FLAG_TEST_FAIL_HOST_ALLOC)");
        }
        e = cudaHostAlloc(&hp, pool_bytes, cudaHostAllocMapped | cudaHostAllocPortable);
        if (e != cudaSuccess) {
            return bail(SRH_ERR_NOMEM, std::string("cudaHostAlloc: ") + cudaGetErrorString(e));
        }
        ctx->pool_host[l] = static_cast<float*>(hp);
        void* dp = nullptr;
        e = cudaHostGetDevicePointer(&dp, hp, 0);
        if (e != cudaSuccess) return bail(SRH_ERR_CUDA, std::string("cudaHostGetDevicePointer: ") + cudaGetErrorString(e));
        ctx->pool_dev[l] = static_cast<float*>(dp);
        ld.pool = ctx->pool_dev[l];
        ctx->ready_host[l].assign((size_t)B * cap, 0);
        e = cudaMalloc(&ld.host_ready, (size_t)B * cap);
        if (e == cudaSuccess) e = cudaMemset(ld.host_ready, 0, (size_t)B * cap);
        if (e == cudaSuccess && ld.swap) {
            e = cudaMalloc(&ld.slot_of, sizeof(int) * (size_t)B * cap);
            if (e == cudaSuccess) e = cudaMemset(ld.slot_of, 0xff, sizeof(int) * (size_t)B * cap);
            if (e == cudaSuccess) e = cudaMalloc(&ld.slot_logical, sizeof(int) * (size_t)B * G);
            if (e == cudaSuccess) e = cudaMemset(ld.slot_logical, 0xff, sizeof(int) * (size_t)B * G);
            if (e == cudaSuccess) e = cudaMalloc(&ld.lru_order, sizeof(int) * (size_t)B * G);
            if (e == cudaSuccess) {
                std::vector<int> order((size_t)B * G);
                for (int b = 0; b < B; ++b)
                    for (int q = 0; q < G; ++q) order[(size_t)b * G + q] = q;   // slot 0 at the back
                e = cudaMemcpy(ld.lru_order, order.data(), sizeof(int) * order.size(), cudaMemcpyHostToDevice);
            }
            if (e == cudaSuccess) e = cudaMalloc(&ld.adapt, sizeof(AdaptState) * (size_t)B);
            if (e == cudaSuccess) {
                std::vector<AdaptState> st((size_t)B, AdaptState{G, G, 0, 0, 0, 0});   // all slots in use
                e = cudaMemcpy(ld.adapt, st.data(), sizeof(AdaptState) * st.size(), cudaMemcpyHostToDevice);
            }
        }
        if (e != cudaSuccess) return bail(SRH_ERR_NOMEM, std::string("device state: ") + cudaGetErrorString(e));
    }

    std::vector<int> swl;
    ctx->swap_pos.assign(ctx->L, -1);
    for (int l = 0; l < ctx->L; ++l)
        if (ctx->swap[l]) {
            ctx->swap_pos[l] = (int)swl.size();
            swl.push_back(l);
        }
    ctx->n_swap = (int)swl.size();
    e = cudaMalloc(&ctx->d_swap_layers, sizeof(int) * std::max<size_t>(swl.size(), 1));
    if (e == cudaSuccess && !swl.empty())
        e = cudaMemcpy(ctx->d_swap_layers, swl.data(), sizeof(int) * swl.size(), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return bail(SRH_ERR_NOMEM, std::string("device state: ") + cudaGetErrorString(e));
    e = cudaMalloc(&ctx->d_layers, sizeof(LayerDev) * ctx->L);
    if (e == cudaSuccess)
        e = cudaMemcpy(ctx->d_layers, ctx->h_layers.data(), sizeof(LayerDev) * ctx->L, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_stats, sizeof(unsigned long long) * kStatCount);
    if (e == cudaSuccess) e = cudaMemset(ctx->d_stats, 0, sizeof(unsigned long long) * kStatCount);
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_err, sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemset(ctx->d_err, 0, sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_hist, sizeof(uint32_t) * kHistBins * B);
    if (e == cudaSuccess) e = cudaMemset(ctx->d_hist, 0, sizeof(uint32_t) * kHistBins * B);
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_cand, sizeof(unsigned long long) * select_cand_cap() * B);
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_cand_cnt, sizeof(int) * B);
    if (e == cudaSuccess) e = cudaMemset(ctx->d_cand_cnt, 0, sizeof(int) * B);
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_miss, sizeof(int2) * (size_t)ctx->L * B * ctx->S);
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_miss_count, sizeof(int) * (size_t)ctx->L * B);
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_sink, sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemset(ctx->d_miss_count, 0, sizeof(int) * (size_t)ctx->L * B);
    if (e != cudaSuccess) return bail(SRH_ERR_NOMEM, std::string("device scratch: ") + cudaGetErrorString(e));

    std::vector<AttnSeg> segs;
    std::vector<int> cta_begin;
    std::vector<MergeItem> merges;
    if (!plan_attention(ctx, &segs, &cta_begin, &merges))
        return bail(SRH_ERR_INVALID, "internal: the attention plan breaks its invariants for this configuration");
    e = cudaMalloc(&ctx->d_segs, sizeof(AttnSeg) * segs.size());
    if (e == cudaSuccess)
        e = cudaMemcpy(ctx->d_segs, segs.data(), sizeof(AttnSeg) * segs.size(), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_cta_begin, sizeof(int) * cta_begin.size());
    if (e == cudaSuccess)
        e = cudaMemcpy(ctx->d_cta_begin, cta_begin.data(), sizeof(int) * cta_begin.size(), cudaMemcpyHostToDevice);
    const size_t slots = (size_t)std::max(ctx->max_slots, 1);
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_part_o, sizeof(uint16_t) * slots * SRH_MAX_HEADS * kKvDim);
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_part_ml, sizeof(float) * slots * kAttnMlStride);
    if (e == cudaSuccess && !merges.empty()) e = cudaMalloc(&ctx->d_merges, sizeof(MergeItem) * merges.size());
    if (e == cudaSuccess && !merges.empty())
        e = cudaMemcpy(ctx->d_merges, merges.data(), sizeof(MergeItem) * merges.size(), cudaMemcpyHostToDevice);
    if (e == cudaSuccess && !merges.empty())
        e = cudaMalloc(&ctx->d_merge_cnt, sizeof(unsigned long long) * merges.size());
    if (e == cudaSuccess && !merges.empty())
        e = cudaMemset(ctx->d_merge_cnt, 0, sizeof(unsigned long long) * merges.size());
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ctx->ev_resolved, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ctx->ev_gathered, cudaEventDisableTiming);
    if (e != cudaSuccess) return bail(SRH_ERR_NOMEM, std::string("attention scratch: ") + cudaGetErrorString(e));
    *out = ctx;
    return SRH_OK;
}

void srh_destroy(srh_ctx* ctx) { free_ctx(ctx); }

float* srh_pool_host_ptr(srh_ctx* ctx, int layer, int seq) {
    if (!ctx || layer < 0 || layer >= ctx->L || seq < 0 || seq >= ctx->B) return nullptr;
    return ctx->pool_host[layer] + (size_t)seq * ctx->caps[layer] * kKvDim;
}

int srh_mark_stored(srh_ctx* ctx, int layer, int seq, long long c0, long long n) {
    if (!ctx) return SRH_ERR_INVALID;
    if (layer < 0 || layer >= ctx->L || seq < 0 || seq >= ctx->B)
        return fail(ctx, SRH_ERR_INVALID, "layer or seq out of range");
    const long long cap = ctx->caps[layer];
    if (c0 < 0 || n < 0 || c0 + n > cap) return fail(ctx, SRH_ERR_INVALID, "chunk range out of bounds");
    if (n == 0) return SRH_OK;
    uint8_t* hr = ctx->ready_host[layer].data() + (size_t)seq * cap;
    std::memset(hr + c0, 1, (size_t)n);
    SRH_CUDA(ctx, cudaMemcpy(ctx->h_layers[layer].host_ready + (size_t)seq * cap + c0, hr + c0, (size_t)n,
                             cudaMemcpyHostToDevice));
    if (!ctx->swap[layer]) ctx->resident_dirty[layer] = 1;
    // read each stored page once from the device: the first reads of a host
    // page are the slow ones, and this keeps them out of the decode steps
    const cudaError_t e = launch_touch(ctx->pool_dev[layer] + ((size_t)seq * cap + c0) * kKvDim, n * kKvDim,
                                       ctx->d_sink, ctx->sm_count, 0);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "srh_mark_stored touch");
    SRH_CUDA(ctx, cudaStreamSynchronize(0));
    return SRH_OK;
}

int kvswap_store(srh_ctx* ctx, int layer, int seq, long long c0, int n, const float* d_rows,
                 srh_stream_t stream) {
    if (!ctx) return SRH_ERR_INVALID;
    if (!d_rows) return fail(ctx, SRH_ERR_INVALID, "NULL pointer");
    if (layer < 0 || layer >= ctx->L || seq < 0 || seq >= ctx->B)
        return fail(ctx, SRH_ERR_INVALID, "layer or seq out of range");
    const long long cap = ctx->caps[layer];
    if (c0 < 0 || n < 0 || c0 + n > cap) return fail(ctx, SRH_ERR_INVALID, "chunk range out of bounds");
    if (((uintptr_t)d_rows) & 15) return fail(ctx, SRH_ERR_INVALID, "rows must be 16-byte aligned");
    if (n == 0) return SRH_OK;
    // a layer that does not swap gets its staging rows written directly once the
    // staging is bound; before that, the next kvswap_stage fills them
    if (!ctx->swap[layer] && !ctx->staging) ctx->resident_dirty[layer] = 1;
    const cudaError_t e = launch_store(ctx->d_layers, layer, ctx->B, ctx->G, seq, c0, n, d_rows, ctx->staging,
                                       ctx->d_err, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "kvswap_store launch");
    std::memset(ctx->ready_host[layer].data() + (size_t)seq * cap + c0, 1, (size_t)n);
    ctx->stored_bytes += (unsigned long long)n * kKvDim * sizeof(float);
    return SRH_OK;
}

int srh_layer_info(srh_ctx* ctx, int layer, long long* cap, int* swap_enabled) {
    if (!ctx || layer < 0 || layer >= ctx->L) return SRH_ERR_INVALID;
    if (cap) *cap = ctx->caps[layer];
    if (swap_enabled) *swap_enabled = ctx->swap[layer];
    return SRH_OK;
}

int srh_max_select(srh_ctx* ctx) { return ctx ? ctx->S : SRH_ERR_INVALID; }

namespace {
int score_impl(srh_ctx* ctx, const uint16_t* d_keys, int key_sets, int n, const uint16_t* d_q, float scale,
               const float* bias3, int ensemble, float* d_scores, srh_stream_t stream) {
    if (!ctx) return SRH_ERR_INVALID;
    if (!d_keys || !d_q || !bias3 || !d_scores) return fail(ctx, SRH_ERR_INVALID, "NULL pointer");
    if (n < 1 || n > ctx->n_src) return fail(ctx, SRH_ERR_INVALID, "n must be in [1, source capacity]");
    if (ensemble != SRH_ENSEMBLE_MAX && ensemble != SRH_ENSEMBLE_MEAN)
        return fail(ctx, SRH_ERR_INVALID, "unknown ensemble");
    if (((uintptr_t)d_keys | (uintptr_t)d_q) & 15) return fail(ctx, SRH_ERR_INVALID, "keys/queries must be 16-byte aligned");
    if (!std::isfinite(scale)) return fail(ctx, SRH_ERR_INVALID, "scale must be finite");
    // After a threshold selection, the pass also appends the chunks above that
    // threshold to the candidate list, and builds no histogram: the next
    // selection with the same threshold uses the list and skips its own pass
    // over the scores (a top-k selection rebuilds the histogram).
    const bool fused = ctx->thresh_hint_valid;
    CandSink sink{0u, nullptr, nullptr, 0};
    if (fused) sink = CandSink{ordered_key(ctx->thresh_hint), ctx->d_cand, ctx->d_cand_cnt, select_cand_cap()};
    const cudaError_t e = launch_score(d_keys, n, ctx->B, d_q, scale, bias3, ensemble, d_scores,
                                       fused ? nullptr : ctx->d_hist, ctx->d_err, ctx->sm_count,
                                       (cudaStream_t)stream, key_sets, !fused && !ctx->hist_clean, sink,
                                       fused && !ctx->cand_clean);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "fm_score launch");
    if (fused) {
        ctx->cand_clean = false;
        ctx->cand_scores = d_scores;
        ctx->cand_n = n;
        ctx->cand_thresh = ctx->thresh_hint;
        ctx->hist_scores = nullptr;
        ctx->hist_n = -1;
    } else {
        ctx->hist_clean = false;
        ctx->hist_scores = d_scores;
        ctx->hist_n = n;
        ctx->cand_scores = nullptr;
    }
    return SRH_OK;
}
}  // namespace

int fm_score(srh_ctx* ctx, const uint16_t* d_keys, int n, const uint16_t* d_q, float scale,
             const float* bias3, int ensemble, float* d_scores, srh_stream_t stream) {
    return score_impl(ctx, d_keys, 1, n, d_q, scale, bias3, ensemble, d_scores, stream);
}

int fm_score_multi(srh_ctx* ctx, const uint16_t* d_keys3, int n, const uint16_t* d_q, float scale,
                   const float* bias3, int ensemble, float* d_scores, srh_stream_t stream) {
    return score_impl(ctx, d_keys3, 3, n, d_q, scale, bias3, ensemble, d_scores, stream);
}

int fm_quantize_keys(srh_ctx* ctx, const uint16_t* d_keys, int n, uint8_t* d_codes, float* d_kscale,
                     srh_stream_t stream) {
    if (!ctx) return SRH_ERR_INVALID;
    if (!d_keys || !d_codes || !d_kscale) return fail(ctx, SRH_ERR_INVALID, "NULL pointer");
    if (n < 1 || n > ctx->n_src) return fail(ctx, SRH_ERR_INVALID, "n must be in [1, source capacity]");
    if (((uintptr_t)d_keys | (uintptr_t)d_codes | (uintptr_t)d_kscale) & 15)
        return fail(ctx, SRH_ERR_INVALID, "keys/codes/scales must be 16-byte aligned");
    const cudaError_t e = launch_quantize_keys(d_keys, (long long)ctx->B * n, d_codes, d_kscale, ctx->sm_count,
                                               (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "fm_quantize_keys launch");
    return SRH_OK;
}

int fm_score_fp8(srh_ctx* ctx, const uint8_t* d_codes, const float* d_kscale, int n, const uint16_t* d_q,
                 float scale, const float* bias3, int ensemble, float* d_scores, srh_stream_t stream) {
    if (!ctx) return SRH_ERR_INVALID;
    if (!d_codes || !d_kscale || !d_q || !bias3 || !d_scores) return fail(ctx, SRH_ERR_INVALID, "NULL pointer");
    if (n < 1 || n > ctx->n_src) return fail(ctx, SRH_ERR_INVALID, "n must be in [1, source capacity]");
    if (ensemble != SRH_ENSEMBLE_MAX && ensemble != SRH_ENSEMBLE_MEAN)
        return fail(ctx, SRH_ERR_INVALID, "unknown ensemble");
    if (((uintptr_t)d_codes | (uintptr_t)d_q) & 15) return fail(ctx, SRH_ERR_INVALID, "codes/queries must be 16-byte aligned");
    if (((uintptr_t)d_kscale) & 3) return fail(ctx, SRH_ERR_INVALID, "scales must be 4-byte aligned");
    if (!std::isfinite(scale)) return fail(ctx, SRH_ERR_INVALID, "scale must be finite");
    const cudaError_t e = launch_score_fp8(d_codes, d_kscale, n, ctx->B, d_q, scale, bias3, ensemble, d_scores,
                                           ctx->d_hist, ctx->sm_count, (cudaStream_t)stream, !ctx->hist_clean);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "fm_score_fp8 launch");
    ctx->hist_clean = false;
    ctx->hist_scores = d_scores;
    ctx->hist_n = n;
    ctx->cand_scores = nullptr;   // this pass builds no candidate list
    return SRH_OK;
}

int fm_select(srh_ctx* ctx, const float* d_scores, int n, int mode, int k, float tau, int clamp,
              int32_t* d_sel, int32_t* d_count, srh_stream_t stream) {
    if (!ctx) return SRH_ERR_INVALID;
    if (!d_scores || !d_sel || !d_count) return fail(ctx, SRH_ERR_INVALID, "NULL pointer");
    if (n < 1 || n > ctx->n_src) return fail(ctx, SRH_ERR_INVALID, "n must be in [1, source capacity]");
    float thresh = 0.f;
    if (mode == SRH_SELECT_TOPK) {
        if (k < 1 || k > ctx->S) return fail(ctx, SRH_ERR_INVALID, "k must be in [1, max_select]");
    } else if (mode == SRH_SELECT_THRESH) {
        if (!(tau > 0.f && tau < 1.f)) return fail(ctx, SRH_ERR_INVALID, "tau must be in (0, 1)");
        if (clamp < 0 || clamp > ctx->S || clamp > ctx->G)
            return fail(ctx, SRH_ERR_INVALID, "clamp must be in [0, min(max_select, gpu_chunks)]");
        thresh = (float)std::log((double)tau / (1.0 - (double)tau));
    } else {
        return fail(ctx, SRH_ERR_INVALID, "unknown selection mode");
    }
    cudaStream_t st = (cudaStream_t)stream;
    if (mode == SRH_SELECT_THRESH) {
        const bool have_list = ctx->cand_scores == d_scores && ctx->cand_n == n && ctx->cand_thresh == thresh;
        ctx->thresh_hint_valid = true;     // the next scoring pass builds the list for this threshold
        ctx->thresh_hint = thresh;
        if (have_list) {
            // the scoring pass appended every chunk above the threshold: select from that list
            ctx->cand_scores = nullptr;
            const cudaError_t e = launch_select(d_scores, n, ctx->B, mode, k, thresh, clamp, ctx->S, nullptr, d_sel,
                                                d_count, st, ctx->d_cand, ctx->d_cand_cnt, select_cand_cap(),
                                                ctx->chained);
            if (e != cudaSuccess) return cuda_fail(ctx, e, "fm_select launch");
            ctx->cand_clean = true;   // the select kernel zeroes the counts it reads
            return SRH_OK;
        }
    } else {
        ctx->thresh_hint_valid = false;
    }
    ctx->cand_scores = nullptr;
    uint32_t* hist = nullptr;
    bool chained = ctx->chained;   // the select kernel follows a kernel of this call or of fm_score
    if (mode == SRH_SELECT_TOPK || clamp > 0) {
        if (ctx->hist_scores == d_scores && ctx->hist_n == n) {
            hist = ctx->d_hist;
        } else {
            const cudaError_t e = launch_hist(d_scores, n, ctx->B, ctx->d_hist, st, !ctx->hist_clean);
            ctx->hist_clean = false;
            if (e != cudaSuccess) return cuda_fail(ctx, e, "fm_select histogram");
            hist = ctx->d_hist;
            chained = true;
        }
    }
    ctx->hist_scores = nullptr;   // one use per scoring pass
    ctx->hist_n = -1;
    const unsigned long long* cand = nullptr;
    if (n > kCollectMinN) {
        const int K = mode == SRH_SELECT_TOPK ? std::min(k, n) : clamp;
        const cudaError_t ec = launch_collect(d_scores, n, ctx->B, mode, K, thresh, hist, ctx->d_cand,
                                              ctx->d_cand_cnt, select_cand_cap(), st, !ctx->cand_clean, chained);
        ctx->cand_clean = false;
        if (ec != cudaSuccess) return cuda_fail(ctx, ec, "fm_select candidate pass");
        cand = ctx->d_cand;
        chained = true;
    }
    const cudaError_t e = launch_select(d_scores, n, ctx->B, mode, k, thresh, clamp, ctx->S, hist, d_sel,
                                        d_count, st, cand, ctx->d_cand_cnt, select_cand_cap(), chained);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "fm_select launch");
    if (hist) ctx->hist_clean = true;   // the select kernel zeroes the rows it reads
    if (cand) ctx->cand_clean = true;   // ... and the candidate counts
    return SRH_OK;
}

int kvswap_stage(srh_ctx* ctx, int layer, const int32_t* d_sel, const int32_t* d_count,
                 uint16_t* d_staging, int32_t* d_phys, int32_t* d_count_l, srh_stream_t main,
                 srh_stream_t side) {
    if (!ctx) return SRH_ERR_INVALID;
    if (!d_sel || !d_count || !d_staging || !d_phys || !d_count_l) return fail(ctx, SRH_ERR_INVALID, "NULL pointer");
    if (layer < -1 || layer >= ctx->L) return fail(ctx, SRH_ERR_INVALID, "layer out of range");
    if (((uintptr_t)d_staging) & 31) return fail(ctx, SRH_ERR_INVALID, "staging must be 32-byte aligned");
    if (ctx->staging && ctx->staging != d_staging)
        return fail(ctx, SRH_ERR_INVALID, "d_staging differs from the buffer bound on the first call");
    ctx->staging = d_staging;
    cudaStream_t sm = (cudaStream_t)main, ss = (cudaStream_t)side;
    const int l0 = layer < 0 ? 0 : layer;
    const int nl = layer < 0 ? ctx->L : 1;
    // swap-disabled layers: (re)copy their stored chunks once
    for (int l = l0; l < l0 + nl; ++l) {
        if (ctx->swap[l] || !ctx->resident_dirty[l]) continue;
        cudaError_t e = launch_resident_fill(ctx->pool_dev[l], ctx->h_layers[l].host_ready, ctx->caps[l], l,
                                             ctx->B, ctx->G, d_staging, ctx->d_err, sm);
        if (e != cudaSuccess) return cuda_fail(ctx, e, "resident fill");
        ctx->resident_dirty[l] = 0;
        unsigned long long ready = 0;
        for (uint8_t v : ctx->ready_host[l]) ready += v;
        ctx->resident_fill_bytes += ready * kKvDim * sizeof(float);
    }
    long long dedup_cap = 0, mirror_cap = 0;
    for (int l = l0; l < l0 + nl; ++l) {
        if (ctx->ratios[l] != ctx->cfg.src_ratio) dedup_cap = std::max(dedup_cap, ctx->caps[l]);
        if (ctx->swap[l] && ctx->caps[l] <= kLruMirrorMax) mirror_cap = std::max(mirror_cap, ctx->caps[l]);
    }
    cudaError_t e = launch_lru(ctx->d_layers, l0, nl, ctx->B, ctx->G, ctx->S, ctx->cfg.src_ratio, dedup_cap, mirror_cap,
                               d_sel, d_count, d_phys, d_count_l, ctx->d_miss, ctx->d_miss_count, ctx->d_stats,
                               ctx->d_err, ctx->adapt, sm, ctx->chained);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "kvswap_stage LRU launch");
    // The gather is a wide kernel of its own, over the swapped layers only: a
    // boundary step's misses are rows of host pages the GPU may not have read
    // recently, so many must be in flight at once. On the main stream it
    // directly follows the resolve kernel (chained); with a side stream it
    // runs there, joined by events. A call with no swapped layer has none.
    const int sw0 = layer < 0 ? 0 : ctx->swap_pos[layer];
    const int n_sw = layer < 0 ? ctx->n_swap : (sw0 >= 0 ? 1 : 0);
    if (n_sw > 0) {
        if (ss && ss != sm) {
            SRH_CUDA(ctx, cudaEventRecord(ctx->ev_resolved, sm));
            SRH_CUDA(ctx, cudaStreamWaitEvent(ss, ctx->ev_resolved, 0));
        } else {
            ss = sm;
        }
        e = launch_gather(ctx->d_layers, ctx->d_swap_layers + sw0, n_sw, nl, ctx->B, ctx->G, ctx->S, ctx->d_miss,
                          ctx->d_miss_count, d_staging, ctx->d_err, ctx->sm_count, ss, ss == sm);
        if (e != cudaSuccess) return cuda_fail(ctx, e, "kvswap_stage gather launch");
        if (ss != sm) {
            SRH_CUDA(ctx, cudaEventRecord(ctx->ev_gathered, ss));
            SRH_CUDA(ctx, cudaStreamWaitEvent(sm, ctx->ev_gathered, 0));
        }
    }
    ++ctx->stage_calls;
    return SRH_OK;
}

int lsa_attend(srh_ctx* ctx, int layer, const uint16_t* d_q, int n_heads, const float* d_window,
               const uint16_t* d_staging, const int32_t* d_phys, const int32_t* d_count_l, float* d_out,
               srh_stream_t stream) {
    if (!ctx) return SRH_ERR_INVALID;
    if (!d_q || !d_window || !d_staging || !d_phys || !d_count_l || !d_out)
        return fail(ctx, SRH_ERR_INVALID, "NULL pointer");
    if (layer < -1 || layer >= ctx->L) return fail(ctx, SRH_ERR_INVALID, "layer out of range");
    if (n_heads != 16 && n_heads != 32 && n_heads != 64)
        return fail(ctx, SRH_ERR_INVALID, "n_heads must be 16, 32 or 64");
    if (((uintptr_t)d_q | (uintptr_t)d_out) & 15 || ((uintptr_t)d_window | (uintptr_t)d_staging) & 31)
        return fail(ctx, SRH_ERR_INVALID, "q/out must be 16-byte aligned, window/staging 32-byte aligned");
    const AttnPlan& pl = ctx->plans[layer + 1];
    const cudaError_t e = launch_attend(ctx->d_segs + pl.seg0, ctx->d_cta_begin + pl.cta0, pl.n_ctas,
                                        ctx->d_merges + pl.merge0, ctx->d_merge_cnt + pl.merge0, n_heads, ctx->B,
                                        ctx->G, ctx->S, d_q, d_window, d_staging, d_phys, d_count_l, d_out,
                                        ctx->d_part_o, ctx->d_part_ml, ctx->d_err, (cudaStream_t)stream,
                                        ctx->chained);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "lsa_attend launch");
    return SRH_OK;
}

int srh_set_adaptive(srh_ctx* ctx, const srh_adaptive* p) {
    if (!ctx) return SRH_ERR_INVALID;
    AdaptParams ap{};
    const int G = ctx->G;
    int g_next = G;
    if (p && p->enabled) {
        const int lo_g = ctx->cfg.allow_topk_reduction ? 1 : ctx->cfg.index_topk;
        if (p->g_max < 1 || p->g_max > G) return fail(ctx, SRH_ERR_INVALID, "g_max must be in [1, gpu_chunks]");
        if (p->g_min < lo_g || p->g_min > p->g_max)
            return fail(ctx, SRH_ERR_INVALID, "g_min must be in [index_topk, g_max]");
        if (p->g_init < p->g_min || p->g_init > p->g_max)
            return fail(ctx, SRH_ERR_INVALID, "g_init must be in [g_min, g_max]");
        if (p->epoch < 1 || p->delta < 1) return fail(ctx, SRH_ERR_INVALID, "epoch and delta must be >= 1");
        if (p->lo_permille < 0 || p->lo_permille > p->hi_permille || p->hi_permille > 1000)
            return fail(ctx, SRH_ERR_INVALID, "need 0 <= lo_permille <= hi_permille <= 1000");
        ap = AdaptParams{1, p->g_min, p->g_max, p->epoch, p->lo_permille, p->hi_permille, p->delta};
        g_next = p->g_init;
    }
    SRH_CUDA(ctx, cudaDeviceSynchronize());
    std::vector<AdaptState> st((size_t)ctx->B);
    for (int l = 0; l < ctx->L; ++l) {
        if (!ctx->swap[l]) continue;
        AdaptState* d = ctx->h_layers[l].adapt;
        SRH_CUDA(ctx, cudaMemcpy(st.data(), d, sizeof(AdaptState) * st.size(), cudaMemcpyDeviceToHost));
        for (auto& a : st) {
            a.g_next = g_next;
            a.ep_steps = 0;
            a.ep_hits = a.ep_sel = 0;
        }
        SRH_CUDA(ctx, cudaMemcpy(d, st.data(), sizeof(AdaptState) * st.size(), cudaMemcpyHostToDevice));
    }
    ctx->adapt = ap;
    return SRH_OK;
}

int srh_get_active_slots(srh_ctx* ctx, int* out) {
    if (!ctx) return SRH_ERR_INVALID;
    if (!out) return fail(ctx, SRH_ERR_INVALID, "NULL pointer");
    SRH_CUDA(ctx, cudaDeviceSynchronize());
    std::vector<AdaptState> st((size_t)ctx->B);
    for (int l = 0; l < ctx->L; ++l) {
        if (ctx->swap[l]) {
            SRH_CUDA(ctx, cudaMemcpy(st.data(), ctx->h_layers[l].adapt, sizeof(AdaptState) * st.size(),
                                     cudaMemcpyDeviceToHost));
            for (int b = 0; b < ctx->B; ++b) out[(size_t)l * ctx->B + b] = st[b].g;
        } else {
            for (int b = 0; b < ctx->B; ++b) out[(size_t)l * ctx->B + b] = (int)ctx->caps[l];
        }
    }
    return SRH_OK;
}

int srh_set_chained(srh_ctx* ctx, int on) {
    if (!ctx) return SRH_ERR_INVALID;
    ctx->chained = on != 0;
    return SRH_OK;
}

int srh_get_stats(srh_ctx* ctx, srh_stats* out) {
    if (!ctx || !out) return SRH_ERR_INVALID;
    SRH_CUDA(ctx, cudaDeviceSynchronize());
    unsigned long long s[kStatCount];
    SRH_CUDA(ctx, cudaMemcpy(s, ctx->d_stats, sizeof s, cudaMemcpyDeviceToHost));
    std::memset(out, 0, sizeof *out);
    out->hits = s[kStatHits];
    out->misses = s[kStatMisses];
    out->h2d_bytes = s[kStatMisses] * kKvDim * sizeof(float);
    out->d2h_bytes = ctx->stored_bytes;
    out->resident_fill_bytes = ctx->resident_fill_bytes;
    out->stage_calls = ctx->stage_calls;
    out->selected = s[kStatSelected];
    int sw = 0;
    for (int v : ctx->swap) sw += v;
    out->swapped_layers = sw;
    out->n_layers = ctx->L;
    return SRH_OK;
}

int srh_reset_stats(srh_ctx* ctx) {
    if (!ctx) return SRH_ERR_INVALID;
    SRH_CUDA(ctx, cudaDeviceSynchronize());
    SRH_CUDA(ctx, cudaMemset(ctx->d_stats, 0, sizeof(unsigned long long) * kStatCount));
    SRH_CUDA(ctx, cudaDeviceSynchronize());
    ctx->stage_calls = 0;
    ctx->stored_bytes = 0;
    return SRH_OK;
}

int srh_selftest_wait_timeout(srh_ctx* ctx, int limit_us, srh_stream_t stream) {
    if (!ctx) return SRH_ERR_INVALID;
    if (limit_us < 1 || limit_us > 2000000) return fail(ctx, SRH_ERR_INVALID, "limit_us must be in [1, 2000000]");
    const cudaError_t e = launch_wait_selftest(ctx->d_err, (unsigned long long)limit_us * 1000ull,
                                               (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "srh_selftest_wait_timeout launch");
    return SRH_OK;
}

}  // extern "C"

struct srh_hostloop {
    srh_ctx* ctx = nullptr;
    cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
    cudaEvent_t ev_in[2] = {}, ev_done[2] = {}, ev_out[2] = {};
    cudaGraph_t graph[2] = {};
    cudaGraphExec_t exec[2] = {};
    uint16_t* fm_q[2] = {};
    uint16_t* q[2] = {};
    float* out[2] = {};
    int32_t* sel[2] = {};
    int32_t* count[2] = {};
    size_t fmq_bytes = 0, q_bytes = 0, out_bytes = 0, sel_bytes = 0, count_bytes = 0;
};

namespace {

void hostloop_free(srh_hostloop* lp) {
    if (!lp) return;
    for (cudaStream_t s : {lp->s_in, lp->s_comp, lp->s_out})
        if (s) cudaStreamSynchronize(s);
    for (int k = 0; k < 2; ++k) {
        if (lp->exec[k]) cudaGraphExecDestroy(lp->exec[k]);
        if (lp->graph[k]) cudaGraphDestroy(lp->graph[k]);
        for (cudaEvent_t e : {lp->ev_in[k], lp->ev_done[k], lp->ev_out[k]})
            if (e) cudaEventDestroy(e);
    }
    for (cudaStream_t s : {lp->s_in, lp->s_comp, lp->s_out})
        if (s) cudaStreamDestroy(s);
    delete lp;
}

}  // namespace

extern "C" {

int srh_hostloop_create(srh_ctx* ctx, const uint16_t* d_keys, int n, float* d_scores, uint16_t* d_staging,
                        int32_t* d_phys, int32_t* d_count_l, const float* d_window, int n_heads, float scale,
                        const float* bias3, int ensemble, int mode, int k, float tau, int clamp,
                        uint16_t* const d_fm_q[2], uint16_t* const d_q[2], float* const d_out[2],
                        int32_t* const d_sel[2], int32_t* const d_count[2], srh_stream_t stream,
                        srh_hostloop** out) {
    if (!ctx || !out) return SRH_ERR_INVALID;
    *out = nullptr;
    if (!d_keys || !d_scores || !d_staging || !d_phys || !d_count_l || !d_window || !bias3 || !d_fm_q || !d_q ||
        !d_out || !d_sel || !d_count)
        return fail(ctx, SRH_ERR_INVALID, "NULL pointer");
    for (int s = 0; s < 2; ++s)
        if (!d_fm_q[s] || !d_q[s] || !d_out[s] || !d_sel[s] || !d_count[s])
            return fail(ctx, SRH_ERR_INVALID, "NULL step buffer");
    if (n_heads != 16 && n_heads != 32 && n_heads != 64) return fail(ctx, SRH_ERR_INVALID, "n_heads must be 16, 32 or 64");
    srh_hostloop* lp = new (std::nothrow) srh_hostloop;
    if (!lp) return fail(ctx, SRH_ERR_NOMEM, "host loop");
    lp->ctx = ctx;
    const size_t LB = (size_t)ctx->L * ctx->B;
    lp->fmq_bytes = (size_t)ctx->B * 3 * 8 * 128 * sizeof(uint16_t);
    lp->q_bytes = LB * n_heads * kKvDim * sizeof(uint16_t);
    lp->out_bytes = LB * n_heads * kKvDim * sizeof(float);
    lp->sel_bytes = (size_t)ctx->B * ctx->S * sizeof(int32_t);
    lp->count_bytes = (size_t)ctx->B * sizeof(int32_t);
    for (int s = 0; s < 2; ++s) {
        lp->fm_q[s] = d_fm_q[s];
        lp->q[s] = d_q[s];
        lp->out[s] = d_out[s];
        lp->sel[s] = d_sel[s];
        lp->count[s] = d_count[s];
    }
    auto bail = [&](int code) {
        hostloop_free(lp);
        return code;
    };
    cudaError_t e = cudaSuccess;
    for (cudaStream_t* s : {&lp->s_in, &lp->s_comp, &lp->s_out})
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
    for (int s = 0; s < 2 && e == cudaSuccess; ++s)
        for (cudaEvent_t* ev : {&lp->ev_in[s], &lp->ev_done[s], &lp->ev_out[s]})
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "host loop streams and events"));
    // the work already on the caller's stream comes first
    if (e == cudaSuccess) e = cudaEventRecord(lp->ev_in[0], (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(lp->s_comp, lp->ev_in[0], 0);
    if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "host loop start"));
    const bool was_chained = ctx->chained;   // the caller's setting, restored after each capture
    for (int s = 0; s < 2; ++s) {
        e = cudaStreamBeginCapture(lp->s_comp, cudaStreamCaptureModeThreadLocal);
        if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "host loop capture"));
        ctx->chained = false;                 // the graph's first kernel has no predecessor
        int rc = fm_score(ctx, d_keys, n, lp->fm_q[s], scale, bias3, ensemble, d_scores, lp->s_comp);
        if (rc == SRH_OK) {
            ctx->chained = true;
            rc = fm_select(ctx, d_scores, n, mode, k, tau, clamp, lp->sel[s], lp->count[s], lp->s_comp);
            if (rc == SRH_OK)
                rc = kvswap_stage(ctx, -1, lp->sel[s], lp->count[s], d_staging, d_phys, d_count_l, lp->s_comp,
                                  nullptr);
            if (rc == SRH_OK)
                rc = lsa_attend(ctx, -1, lp->q[s], n_heads, d_window, d_staging, d_phys, d_count_l, lp->out[s],
                                lp->s_comp);
        }
        ctx->chained = was_chained;
        cudaGraph_t g = nullptr;
        const cudaError_t ec = cudaStreamEndCapture(lp->s_comp, &g);
        if (rc != SRH_OK) {
            if (g) cudaGraphDestroy(g);
            return bail(rc);
        }
        if (ec != cudaSuccess) return bail(cuda_fail(ctx, ec, "host loop capture"));
        lp->graph[s] = g;
        e = cudaGraphInstantiate(&lp->exec[s], g, 0);
        if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "host loop graph instantiate"));
    }
    *out = lp;
    return SRH_OK;
}

int srh_hostloop_step(srh_hostloop* lp, long long i, const uint16_t* h_fm_q, const uint16_t* h_q, float* h_out,
                      int32_t* h_sel, int32_t* h_count) {
    if (!lp) return SRH_ERR_INVALID;
    srh_ctx* ctx = lp->ctx;
    if (i < 0 || !h_fm_q || !h_q || !h_out || !h_sel || !h_count) return fail(ctx, SRH_ERR_INVALID, "host loop step arguments");
    const int s = (int)(i & 1);
    // set s was last read by step i - 2: its inputs are refilled after that step finished
    SRH_CUDA(ctx, cudaStreamWaitEvent(lp->s_in, lp->ev_done[s], 0));
    SRH_CUDA(ctx, cudaMemcpyAsync(lp->fm_q[s], h_fm_q, lp->fmq_bytes, cudaMemcpyHostToDevice, lp->s_in));
    SRH_CUDA(ctx, cudaMemcpyAsync(lp->q[s], h_q, lp->q_bytes, cudaMemcpyHostToDevice, lp->s_in));
    SRH_CUDA(ctx, cudaEventRecord(lp->ev_in[s], lp->s_in));
    // and its outputs are overwritten after step i - 2's outputs left the device
    SRH_CUDA(ctx, cudaStreamWaitEvent(lp->s_comp, lp->ev_in[s], 0));
    SRH_CUDA(ctx, cudaStreamWaitEvent(lp->s_comp, lp->ev_out[s], 0));
    SRH_CUDA(ctx, cudaGraphLaunch(lp->exec[s], lp->s_comp));
    SRH_CUDA(ctx, cudaEventRecord(lp->ev_done[s], lp->s_comp));
    SRH_CUDA(ctx, cudaStreamWaitEvent(lp->s_out, lp->ev_done[s], 0));
    SRH_CUDA(ctx, cudaMemcpyAsync(h_out, lp->out[s], lp->out_bytes, cudaMemcpyDeviceToHost, lp->s_out));
    SRH_CUDA(ctx, cudaMemcpyAsync(h_sel, lp->sel[s], lp->sel_bytes, cudaMemcpyDeviceToHost, lp->s_out));
    SRH_CUDA(ctx, cudaMemcpyAsync(h_count, lp->count[s], lp->count_bytes, cudaMemcpyDeviceToHost, lp->s_out));
    SRH_CUDA(ctx, cudaEventRecord(lp->ev_out[s], lp->s_out));
    return SRH_OK;
}

int srh_hostloop_wait(srh_hostloop* lp, long long i) {
    if (!lp || i < 0) return SRH_ERR_INVALID;
    SRH_CUDA(lp->ctx, cudaEventSynchronize(lp->ev_out[i & 1]));
    return SRH_OK;
}

int srh_hostloop_sync(srh_hostloop* lp) {
    if (!lp) return SRH_ERR_INVALID;
    for (cudaStream_t s : {lp->s_in, lp->s_comp, lp->s_out}) SRH_CUDA(lp->ctx, cudaStreamSynchronize(s));
    return SRH_OK;
}

void srh_hostloop_destroy(srh_hostloop* lp) { hostloop_free(lp); }

int srh_check_error(srh_ctx* ctx) {
    if (!ctx) return SRH_ERR_INVALID;
    SRH_CUDA(ctx, cudaDeviceSynchronize());
    uint32_t w = 0;
    SRH_CUDA(ctx, cudaMemcpy(&w, ctx->d_err, sizeof w, cudaMemcpyDeviceToHost));
    SRH_CUDA(ctx, cudaMemset(ctx->d_err, 0, sizeof w));
    SRH_CUDA(ctx, cudaDeviceSynchronize());
    if (w & kErrNotStored) return fail(ctx, SRH_ERR_NOT_STORED, "GGUF KV swap selected chunk before it was stored");
    if (w & kErrBounds) return fail(ctx, SRH_ERR_BOUNDS, "a device index was out of bounds");
    if (w & kErrTimeout) return fail(ctx, SRH_ERR_TIMEOUT, "a device wait timed out");
    if (w & kErrRange)
        return fail(ctx, SRH_ERR_RANGE, "an attention query or latent value is beyond +-65504 (fp16 range)");
    return SRH_OK;
}

}  // extern "C"
