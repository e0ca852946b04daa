// C ABI entry points, context set-up and the pipelined decode step.
//
// The decode step follows "DualDecoder: Accelerate Long Context LLM Inference
// by Predictive Prefetch": the prediction for the next step comes from the
// speculative query through the same landmarks (§4.1, §5.2); prefetches run on
// a low-priority stream and misses on a high-priority urgent stream (Fig. 10);
// two ping-pong halves hold the sparse KV of consecutive layers, reuse ordered
// by CUDA events (§5.4, Fig. 11); the prefetch for global layer n + 2 is issued
// once layer n's attention has released its half (§5.3).
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <functional>
#include <initializer_list>
#include <string>
#include <vector>

#include "kvo_internal.cuh"
#include "resident_assign.cuh"

struct kvo_ctx {
    kvo::Ctx c;
};

namespace {

thread_local std::string g_err;

kvo_status fail(kvo::Ctx* c, kvo_status st, const std::string& msg) {
    if (c) c->err = msg; else g_err = msg;
    return st;
}

kvo_status cuda_fail(kvo::Ctx* c, cudaError_t e, const char* what) {
    std::string m = std::string(what) + ": " + cudaGetErrorString(e);
    if (c) c->err = m; else g_err = m;
    return e == cudaErrorMemoryAllocation ? KVO_ERR_OOM : KVO_ERR_CUDA;
}

#define KVO_CUDA(c, expr)                                                   \
    do {                                                                    \
        cudaError_t e_ = (expr);                                            \
        if (e_ != cudaSuccess) return cuda_fail((c), e_, #expr);            \
    } while (0)

template <typename T>
cudaError_t dalloc(T** p, size_t bytes, size_t* acc) {
    *p = nullptr;
    if (bytes == 0) bytes = 16;
    cudaError_t e = cudaMalloc((void**)p, bytes);
    if (e == cudaSuccess && acc) *acc += bytes;
    return e;
}

// Partial-result buffers of the attention kernels, for `items` work items.
cudaError_t part_alloc(kvo::Ctx& c, int items) {
    if (items <= c.att_part_cap) return cudaSuccess;
    if (c.att_part_o) cudaFree(c.att_part_o);
    if (c.att_part_ml) cudaFree(c.att_part_ml);
    c.att_part_o = nullptr;
    c.att_part_ml = nullptr;
    c.att_part_cap = 0;
    const size_t rows = 2 * c.r <= 16 ? 2 * c.r : c.r;   // room for co-batched speculative rows
    // two sets: a chain step runs two layers' hit passes side by side
    cudaError_t e = dalloc(&c.att_part_o, sizeof(float) * 2 * items * rows * c.d, nullptr);
    if (e == cudaSuccess) e = dalloc(&c.att_part_ml, sizeof(float) * 2 * items * rows * 2, nullptr);
    if (e == cudaSuccess) c.att_part_cap = items;
    return e;
}

// Work items of the TMA-staged attention kernel: the tiles of every group
// (sparse part, then window part; window tiles up to the largest window the
// context can hold), group after group, split into `grid` contiguous ranges of
// equal cost -- a tile costs 1, and each part costs kItemCost more, the price
// of the work-item epilogue a range pays where it enters a part -- with their
// bounds rounded to a multiple of the CTA's warps (so the warps of an item get
// equal tile counts), each range cut at part boundaries.  Pure host logic;
// returns the grid used (at least 1, at most the tile count).
int64_t plan_tma_items(int G, int sp_tokens, int w_tokens, int64_t grid, std::vector<int4>& items,
                       std::vector<int32_t>& cta) {
    const int64_t sp_tiles = (sp_tokens + kvo::ATT_TILE - 1) / kvo::ATT_TILE;
    const int64_t w_tiles = (w_tokens + kvo::ATT_TILE - 1) / kvo::ATT_TILE;
    const int64_t per_g = sp_tiles + w_tiles, T = per_g * G;
    grid = std::max<int64_t>(1, std::min<int64_t>(grid, T));
    items.clear();
    cta.assign(grid + 1, 0);
    // parts in tile order with their first tile and first cost unit
    // epilogue of a work item, in tiles: per-CTA timing on the Llama-shaped
    // layer put it at ~4.4 us, the time of ~12 tiles (partial write, ticket
    // round trip, group merge)
    constexpr int64_t kItemCost = 12;
    std::vector<int64_t> p_t0, p_c0, p_len;
    int64_t cost = 0;
    for (int g = 0; g < G; ++g)
        for (int part = 0; part < 2; ++part) {
            const int64_t len = part == 0 ? sp_tiles : w_tiles;
            if (len == 0) continue;
            p_t0.push_back(g * per_g + (part == 0 ? 0 : sp_tiles));
            p_c0.push_back(cost);
            p_len.push_back(len);
            cost += kItemCost + len;
        }
    auto tile_at = [&](int64_t x) -> int64_t {      // tile where cost point x falls (part starts absorb their extra)
        const size_t i = (size_t)(std::upper_bound(p_c0.begin(), p_c0.end(), x) - p_c0.begin()) - 1;
        return p_t0[i] + std::min(p_len[i], std::max<int64_t>(0, x - p_c0[i] - kItemCost));
    };
    auto bound = [&](int64_t j) {
        if (j == grid) return T;
        const int64_t b = tile_at(cost * j / grid);
        return std::min(T, b - b % kvo::ATT_WARPS);
    };
    for (int64_t j = 0; j < grid; ++j) {
        cta[j] = (int32_t)items.size();
        int64_t t = bound(j);
        const int64_t hi = bound(j + 1);
        while (t < hi) {
            const int g = (int)(t / per_g);
            const int64_t off = t - g * per_g;
            const bool sparse = off < sp_tiles;
            const int64_t n = std::min(hi - t, sparse ? sp_tiles - off : per_g - off);
            items.push_back(make_int4(g, sparse ? 0 : 1, (int)(sparse ? off : off - sp_tiles), (int)n));
            t += n;
        }
    }
    cta[grid] = (int32_t)items.size();
    return grid;
}

// The selection kernel: a cluster per group where the group's CTAs fit one
// (at most 8, the portable cluster size; shorter groups' extra CTAs score no
// rows), else the ticket kernel.  Automatically only where the ticket
// kernel's single-CTA tail is long and exposed: more than 4 keys per thread
// (groups of more than 1024 blocks) in a grid of one wave, so no other
// group's scoring runs beside the tails.  Measured, 20 isolated calls each:
// wide_budget (64 groups x ~4000 blocks, 8 CTAs per cluster) 43.0 -> 39.6 us;
// llama3_8b_decode (1008 blocks per group) 17.4 / 17.6 us, long_ctx_predict
// (2.5 waves) 138.5 / 140.8 us, and the Llama chain step 2.10 / 2.15 ms with
// the ticket / cluster kernel.
// Pure host logic (kvo_plan_select): returns the cluster's CTA count, or 0.
static int select_cluster_ctas(int impl, int chunks_max, int64_t n_ctas, int Cmax, int sms) {
    const int S = std::max(1, chunks_max);
    const bool exposed = Cmax > 4 * kvo::SEL_THREADS && n_ctas <= 4 * (int64_t)sms;
    const bool want = impl == 2 || (impl == 1 && exposed);
    return want && S <= 8 ? S : 0;
}

static void set_sel_clu(kvo::Ctx& c) {
    c.sel_clu = select_cluster_ctas(c.sel_impl, c.sel_chunks_max, c.n_sel_items, c.Cmax, c.sel_sms);
}

// Rows per thread of the selection kernels (1, 2 or 4; 256 threads per CTA)
// for groups of Ccap[g] candidate blocks on `sms` SMs holding 4 selection CTAs
// each: 1024 rows per CTA when that gives ~8 CTAs per SM or more; otherwise
// 512 or 256, whichever needs fewer waves (256 on a tie: more CTAs share the
// HBM).  Pure host logic (kvo_plan_select).
static int select_rows_per_thread(int G, const int32_t* Ccap, int sms) {
    int64_t n[3] = {0, 0, 0};
    for (int g = 0; g < G; ++g)
        for (int i = 0; i < 3; ++i) {
            const int rows = kvo::SEL_THREADS << i;
            n[i] += (Ccap[g] + rows - 1) / rows;
        }
    const int64_t slots = 4 * (int64_t)std::max(1, sms);
    auto waves = [&](int64_t x) { return (x + slots - 1) / slots; };
    if (n[2] >= 8 * (int64_t)std::max(1, sms)) return 4;
    return waves(n[1]) < waves(n[0]) ? 2 : 1;
}

kvo_status build_tma_plan(kvo::Ctx& c, kvo::Ctx::TmaPlan& pl, int64_t grid) {
    const int w_max = c.max_append > 0 ? c.W + c.B - 1 : c.W;
    std::vector<int4> items;
    std::vector<int32_t> cta, first(c.G, 0), count(c.G, 0);
    grid = plan_tma_items(c.G, c.k * c.B, w_max, grid, items, cta);
    for (size_t i = 0; i < items.size(); ++i) {
        const int g = items[i].x;
        if (count[g] == 0) first[g] = (int32_t)i;
        ++count[g];
    }
    auto F = [](void* p) { if (p) cudaFree(p); };
    F(pl.items); F(pl.cta); F(pl.first); F(pl.count);
    pl = kvo::Ctx::TmaPlan{};
    KVO_CUDA(&c, part_alloc(c, (int)items.size()));
    KVO_CUDA(&c, dalloc(&pl.items, sizeof(int4) * items.size(), nullptr));
    KVO_CUDA(&c, dalloc(&pl.cta, sizeof(int32_t) * cta.size(), nullptr));
    KVO_CUDA(&c, dalloc(&pl.first, sizeof(int32_t) * c.G, nullptr));
    KVO_CUDA(&c, dalloc(&pl.count, sizeof(int32_t) * c.G, nullptr));
    KVO_CUDA(&c, cudaMemcpy(pl.items, items.data(), sizeof(int4) * items.size(), cudaMemcpyHostToDevice));
    KVO_CUDA(&c, cudaMemcpy(pl.cta, cta.data(), sizeof(int32_t) * cta.size(), cudaMemcpyHostToDevice));
    KVO_CUDA(&c, cudaMemcpy(pl.first, first.data(), sizeof(int32_t) * c.G, cudaMemcpyHostToDevice));
    KVO_CUDA(&c, cudaMemcpy(pl.count, count.data(), sizeof(int32_t) * c.G, cudaMemcpyHostToDevice));
    pl.grid = (int)grid;
    pl.n_items = (int)items.size();
    return KVO_OK;
}

// Both plans: the whole device, and the decode step's share of it (each flat
// gather CTA reserves most of its SM's shared memory, so no attention CTA
// lands on those SMs while a prefetch runs beside the attention).  An explicit
// grid (tma_ctas > 0) applies to both.  Callers synchronise first.
kvo_status build_tma_plans(kvo::Ctx& c) {
    const int64_t dev = (int64_t)c.tma_per_sm * c.n_sms;
    int held = 0;
    if (c.gather_engine == 3 && c.gather_reserve_smem >= 64 * 1024)
        held = std::min(c.gather_ctas > 0 ? c.gather_ctas : 2 * c.n_sms, c.n_sms - 1);
    const int64_t step = (int64_t)c.tma_per_sm * (c.n_sms - held);
    // group-split clusters: as many CTAs per group as the resident CTAs allow,
    // 1 .. 8 (the portable cluster size); chosen automatically only when the
    // groups' CTAs then fill at least 3/4 of the slots -- fewer groups leave
    // SMs idle, and the persistent kernel's balanced tile ranges measured
    // faster there (the Llama layer beside the decode step's gather: 128 CTAs
    // on 228 slots; 64-73 us live against 78-85 us for 256 clusters' CTAs)
    auto plan_clu = [&](int i, int64_t slots) {
        if (c.att_cluster > 0) {
            c.clu_S[i] = c.att_cluster;
            c.clu_use[i] = true;
            return;
        }
        const int64_t G = std::max(1, c.G);
        const int64_t S = std::max<int64_t>(1, std::min<int64_t>(8, slots / G));
        c.clu_S[i] = (int)S;
        c.clu_use[i] = 4 * G * S >= 3 * slots;
    };
    plan_clu(0, (int64_t)c.clu_per_sm * c.n_sms);
    plan_clu(1, (int64_t)c.clu_per_sm * (c.n_sms - held));
    if (kvo_status st = build_tma_plan(c, c.tma[0], c.tma_ctas > 0 ? c.tma_ctas : dev)) return st;
    return build_tma_plan(c, c.tma[1], c.tma_ctas > 0 ? c.tma_ctas : step);
}

void free_ctx(kvo::Ctx& c) {
    auto F = [](void* p) { if (p) cudaFree(p); };
    F(c.g_off); F(c.g_C); F(c.g_len); F(c.g_wstart); F(c.g_wlen);
    for (void* p : c.ring_k) F(p);
    for (void* p : c.ring_v) F(p);
    F(c.d_ring_k); F(c.d_ring_v); F(c.d_host_k); F(c.d_host_v); F(c.d_lm);
    for (void* p : c.lm) F(p);
    for (int i = 0; i < 2; ++i) { F(c.pp_k[i]); F(c.pp_v[i]); }
    for (void* p : c.res_k) F(p);
    for (void* p : c.res_v) F(p);
    F(c.res_map); F(c.res_slots); F(c.res_dslot); F(c.res_pf_ids); F(c.res_pf_cnt); F(c.res_pf_dslot);
    F(c.res_fetched); F(c.res_pfbit); F(c.res_stat); F(c.res_pol); F(c.res_pol_ticket); F(c.res_hit_slot); F(c.res_hit_cnt); F(c.res_oA); F(c.res_lA); F(c.mp_part_o); F(c.mp_part_ml); F(c.mp_done);
    F(c.sel_keys); F(c.sel_hist); F(c.sel_done); F(c.sel_items); F(c.sel_nchunks);
    F(c.runs); F(c.nruns);
    F(c.att_items); F(c.att_first); F(c.att_count); F(c.att_part_o); F(c.att_part_ml); F(c.att_done);
    for (auto& pl : c.tma) { F(pl.items); F(pl.cta); F(pl.first); F(pl.count); }
    F(c.status);
    if (c.h_runs) cudaFreeHost(c.h_runs);
    if (c.h_nruns) cudaFreeHost(c.h_nruns);
    F(c.st_true); F(c.st_pred); F(c.st_miss); F(c.st_miss_cnt); F(c.st_slot);
    for (auto* E : {&c.ev_eager, &c.ev_graph}) {
        for (auto* v : {&E->sel, &E->attn, &E->pref, &E->urg, &E->hit, &E->rassign, &E->rpref})
            for (cudaEvent_t e : *v) if (e) cudaEventDestroy(e);
        if (E->start) cudaEventDestroy(E->start);
    }
    if (c.ev_gin) cudaEventDestroy(c.ev_gin);
    if (c.ev_gout) cudaEventDestroy(c.ev_gout);
    for (cudaGraphExec_t g : c.gexec) if (g) cudaGraphExecDestroy(g);
    for (cudaEvent_t e : c.prof_pool) if (e) cudaEventDestroy(e);
    for (cudaStream_t s : {c.s_compute, c.s_prefetch, c.s_urgent, c.s_urgent2, c.s_hit, c.s_graph}) if (s) cudaStreamDestroy(s);
}

// Records a timing event on `s` when profiling is on; returns its pool index or -1.
cudaError_t prof_mark(kvo::Ctx& c, cudaStream_t s, int* idx) {
    *idx = -1;
    if (!c.prof_on) return cudaSuccess;
    if (c.prof_used == (int)c.prof_pool.size()) {
        cudaEvent_t e;
        cudaError_t err = cudaEventCreate(&e);
        if (err != cudaSuccess) return err;
        c.prof_pool.push_back(e);
    }
    *idx = c.prof_used++;
    return cudaEventRecord(c.prof_pool[*idx], s);
}

cudaStream_t pick(const kvo::Ctx& c, kvo_stream_t s) { return s ? (cudaStream_t)s : c.s_compute; }

kvo_status init_impl(kvo::Ctx& c, const kvo_config* cfg, void* const* k_host, void* const* v_host,
                     const void* const* k_win, const void* const* v_win) {
    if (!cfg || !k_host || !v_host || !cfg->seq_lens) return fail(&c, KVO_ERR_INVALID, "null config, host arrays or seq_lens");
    c.cfg = *cfg;
    c.batch = cfg->batch; c.Hq = cfg->n_q_heads; c.Hkv = cfg->n_kv_heads; c.d = cfg->head_dim;
    c.B = cfg->block_size; c.k = cfg->top_k; c.W = cfg->window; c.L = cfg->n_layers;
    if (c.batch < 1 || c.Hkv < 1 || c.Hq < c.Hkv || c.Hq % c.Hkv) return fail(&c, KVO_ERR_INVALID, "bad batch or head counts");
    c.r = c.Hq / c.Hkv;
    if (c.r > 16) return fail(&c, KVO_ERR_INVALID, "n_q_heads / n_kv_heads must be <= 16");
    if (c.d != 64 && c.d != 128) return fail(&c, KVO_ERR_INVALID, "head_dim must be 64 or 128");
    if (c.B < 1 || c.k < 1 || c.k > 8192 || c.W < 0 || c.L < 1)
        return fail(&c, KVO_ERR_INVALID, "need block_size >= 1, 1 <= top_k <= 8192, window >= 0, n_layers >= 1");
    if (c.W > 0 && (!k_win || !v_win)) return fail(&c, KVO_ERR_INVALID, "window > 0 needs k_win and v_win");
    c.max_append = cfg->max_append;
    if (c.max_append < 0) return fail(&c, KVO_ERR_INVALID, "max_append must be >= 0");
    if (c.max_append > 0 && (c.W == 0 || c.W % c.B))
        return fail(&c, KVO_ERR_INVALID, "max_append > 0 needs window > 0 and window % block_size == 0");
    c.Wcap = c.max_append > 0 ? c.W + c.B : c.W;
    if (cfg->resident < 0 || cfg->resident > 1) return fail(&c, KVO_ERR_INVALID, "resident must be 0 or 1");
    c.resident = cfg->resident == 1;
    c.G = c.batch * c.Hkv;
    c.lens.assign(cfg->seq_lens, cfg->seq_lens + c.batch);
    std::vector<int64_t> off(c.G);
    std::vector<int32_t> C(c.G), Ccap(c.G), glen(c.G), gws(c.G), gwl(c.G);
    int64_t tok = 0;
    for (int b = 0; b < c.batch; ++b) {
        const int64_t n = c.lens[b];
        if (n < c.W || (n - c.W) % c.B) return fail(&c, KVO_ERR_INVALID, "each len must be >= window with (len - window) % block_size == 0");
        const int64_t Cb = (n - c.W) / c.B;
        const int64_t cap = n + c.max_append;            // rows reserved per (request, KV head)
        const int64_t Cc = (cap - c.W) / c.B;            // most candidate blocks the request can reach
        if (Cb < c.k) return fail(&c, KVO_ERR_INVALID, "top_k exceeds the candidate blocks of a request");
        if (Cc > (1 << 30)) return fail(&c, KVO_ERR_INVALID, "too many candidate blocks");
        for (int g = 0; g < c.Hkv; ++g) {
            const int i = b * c.Hkv + g;
            off[i] = (tok * c.Hkv + (int64_t)g * cap) * c.d;
            C[i] = (int32_t)Cb;
            Ccap[i] = (int32_t)Cc;
            glen[i] = (int32_t)n;
            gws[i] = c.Wcap ? (int32_t)((Cb * c.B) % c.Wcap) : 0;
            gwl[i] = c.W;
        }
        c.Cmax = std::max<int>(c.Cmax, (int)Cc);
        tok += cap;
    }
    c.h_off = off;
    c.h_Ccap = Ccap;
    // host caches: page-locked and device-addressable
    for (int l = 0; l < c.L; ++l) {
        for (int kv = 0; kv < 2; ++kv) {
            void* hp = kv ? v_host[l] : k_host[l];
            if (!hp) return fail(&c, KVO_ERR_INVALID, "null host K/V pointer");
            cudaPointerAttributes a{};
            cudaError_t e = cudaPointerGetAttributes(&a, hp);
            if (e != cudaSuccess) return cuda_fail(&c, e, "cudaPointerGetAttributes(host K/V)");
            if (a.type != cudaMemoryTypeHost || !a.devicePointer)
                return fail(&c, KVO_ERR_INVALID, "host K/V must be page-locked, device-mapped memory (cudaHostAlloc / cudaHostRegister)");
            if ((uintptr_t)a.devicePointer % 16) return fail(&c, KVO_ERR_INVALID, "host K/V must be 16-byte aligned");
            (kv ? c.v_host : c.k_host).push_back((const uint16_t*)a.devicePointer);
        }
        if (c.W > 0) {
            for (int kv = 0; kv < 2; ++kv) {
                const void* wp = kv ? v_win[l] : k_win[l];
                if (!wp) return fail(&c, KVO_ERR_INVALID, "null window pointer");
                cudaPointerAttributes a{};
                cudaError_t e = cudaPointerGetAttributes(&a, wp);
                if (e != cudaSuccess) return cuda_fail(&c, e, "cudaPointerGetAttributes(window)");
                if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
                    return fail(&c, KVO_ERR_INVALID, "window K/V must be device memory");
                if ((uintptr_t)wp % 16) return fail(&c, KVO_ERR_INVALID, "window K/V must be 16-byte aligned");
                (kv ? c.v_win : c.k_win).push_back((const uint16_t*)wp);
            }
        } else {
            c.k_win.push_back(nullptr);
            c.v_win.push_back(nullptr);
        }
    }
    // streams: urgent > compute > prefetch
    int least = 0, greatest = 0;
    KVO_CUDA(&c, cudaDeviceGetStreamPriorityRange(&least, &greatest));
    KVO_CUDA(&c, cudaStreamCreateWithPriority(&c.s_compute, cudaStreamNonBlocking, (least + greatest) / 2));
    KVO_CUDA(&c, cudaStreamCreateWithPriority(&c.s_prefetch, cudaStreamNonBlocking, least));
    KVO_CUDA(&c, cudaStreamCreateWithPriority(&c.s_urgent, cudaStreamNonBlocking, greatest));
    KVO_CUDA(&c, cudaStreamCreateWithPriority(&c.s_urgent2, cudaStreamNonBlocking, greatest));
    KVO_CUDA(&c, cudaStreamCreateWithPriority(&c.s_hit, cudaStreamNonBlocking, (least + greatest) / 2));
    size_t sb = 0;
    KVO_CUDA(&c, dalloc(&c.g_off, sizeof(int64_t) * c.G, &sb));
    KVO_CUDA(&c, dalloc(&c.g_C, sizeof(int32_t) * c.G, &sb));
    KVO_CUDA(&c, cudaMemcpy(c.g_off, off.data(), sizeof(int64_t) * c.G, cudaMemcpyHostToDevice));
    KVO_CUDA(&c, cudaMemcpy(c.g_C, C.data(), sizeof(int32_t) * c.G, cudaMemcpyHostToDevice));
    if (c.max_append > 0) {
        KVO_CUDA(&c, dalloc(&c.g_len, sizeof(int32_t) * c.G, &sb));
        KVO_CUDA(&c, dalloc(&c.g_wstart, sizeof(int32_t) * c.G, &sb));
        KVO_CUDA(&c, dalloc(&c.g_wlen, sizeof(int32_t) * c.G, &sb));
        KVO_CUDA(&c, cudaMemcpy(c.g_len, glen.data(), sizeof(int32_t) * c.G, cudaMemcpyHostToDevice));
        KVO_CUDA(&c, cudaMemcpy(c.g_wstart, gws.data(), sizeof(int32_t) * c.G, cudaMemcpyHostToDevice));
        KVO_CUDA(&c, cudaMemcpy(c.g_wlen, gwl.data(), sizeof(int32_t) * c.G, cudaMemcpyHostToDevice));
        // window rings, filled from the caller's windows
        const size_t ring_bytes = (size_t)c.G * c.Wcap * c.d * sizeof(uint16_t);
        c.ring_k.assign(c.L, nullptr);
        c.ring_v.assign(c.L, nullptr);
        for (int l = 0; l < c.L; ++l) {
            KVO_CUDA(&c, dalloc(&c.ring_k[l], ring_bytes, &sb));
            KVO_CUDA(&c, dalloc(&c.ring_v[l], ring_bytes, &sb));
            KVO_CUDA(&c, kvo::launch_ring_fill(c, l, c.k_win[l], c.v_win[l], c.s_compute));
            c.k_win[l] = c.ring_k[l];
            c.v_win[l] = c.ring_v[l];
        }
        KVO_CUDA(&c, dalloc(&c.d_ring_k, sizeof(void*) * c.L, &sb));
        KVO_CUDA(&c, dalloc(&c.d_ring_v, sizeof(void*) * c.L, &sb));
        KVO_CUDA(&c, dalloc(&c.d_host_k, sizeof(void*) * c.L, &sb));
        KVO_CUDA(&c, dalloc(&c.d_host_v, sizeof(void*) * c.L, &sb));
        KVO_CUDA(&c, dalloc(&c.d_lm, sizeof(void*) * c.L, &sb));
        KVO_CUDA(&c, cudaMemcpy(c.d_ring_k, c.ring_k.data(), sizeof(void*) * c.L, cudaMemcpyHostToDevice));
        KVO_CUDA(&c, cudaMemcpy(c.d_ring_v, c.ring_v.data(), sizeof(void*) * c.L, cudaMemcpyHostToDevice));
        KVO_CUDA(&c, cudaMemcpy(c.d_host_k, c.k_host.data(), sizeof(void*) * c.L, cudaMemcpyHostToDevice));
        KVO_CUDA(&c, cudaMemcpy(c.d_host_v, c.v_host.data(), sizeof(void*) * c.L, cudaMemcpyHostToDevice));
    }
    // landmarks
    c.lm_bytes = (size_t)c.G * c.Cmax * c.d * (c.B > 1 ? 4 : 2);
    c.lm.assign(c.L, nullptr);
    for (int l = 0; l < c.L; ++l) {
        KVO_CUDA(&c, dalloc((char**)&c.lm[l], c.lm_bytes, nullptr));
        KVO_CUDA(&c, cudaMemsetAsync(c.lm[l], 0, c.lm_bytes, c.s_compute));
        KVO_CUDA(&c, kvo::launch_landmarks(c, l, c.s_compute));
    }
    if (c.max_append > 0)
        KVO_CUDA(&c, cudaMemcpy(c.d_lm, c.lm.data(), sizeof(void*) * c.L, cudaMemcpyHostToDevice));
    // ping-pong halves
    const size_t half = (size_t)c.G * 2 * c.k * c.B * c.d * sizeof(uint16_t);
    for (int i = 0; i < 2; ++i) {
        KVO_CUDA(&c, dalloc(&c.pp_k[i], half, nullptr));
        KVO_CUDA(&c, dalloc(&c.pp_v[i], half, nullptr));
        KVO_CUDA(&c, cudaMemsetAsync(c.pp_k[i], 0, half, c.s_compute));
        KVO_CUDA(&c, cudaMemsetAsync(c.pp_v[i], 0, half, c.s_compute));
    }
    c.pp_bytes = 4 * half;
    if (c.resident) {
        // per-layer resident block sets and their slot tables (every slot empty)
        c.res_k.assign(c.L, nullptr);
        c.res_v.assign(c.L, nullptr);
        for (int l = 0; l < c.L; ++l) {
            KVO_CUDA(&c, dalloc(&c.res_k[l], half, nullptr));
            KVO_CUDA(&c, dalloc(&c.res_v[l], half, nullptr));
            KVO_CUDA(&c, cudaMemsetAsync(c.res_k[l], 0, half, c.s_compute));
            KVO_CUDA(&c, cudaMemsetAsync(c.res_v[l], 0, half, c.s_compute));
        }
        const size_t lg = (size_t)c.L * c.G;
        KVO_CUDA(&c, dalloc(&c.res_map, sizeof(int32_t) * lg * c.Cmax, &sb));
        KVO_CUDA(&c, dalloc(&c.res_slots, sizeof(int32_t) * lg * 2 * c.k, &sb));
        KVO_CUDA(&c, cudaMemsetAsync(c.res_map, 0xff, sizeof(int32_t) * lg * c.Cmax, c.s_compute));
        KVO_CUDA(&c, cudaMemsetAsync(c.res_slots, 0xff, sizeof(int32_t) * lg * 2 * c.k, c.s_compute));
        KVO_CUDA(&c, dalloc(&c.res_dslot, sizeof(int32_t) * lg * c.k, &sb));
        KVO_CUDA(&c, dalloc(&c.res_pf_ids, sizeof(int32_t) * lg * c.k, &sb));
        KVO_CUDA(&c, dalloc(&c.res_pf_cnt, sizeof(int32_t) * lg, &sb));
        KVO_CUDA(&c, dalloc(&c.res_pf_dslot, sizeof(int32_t) * lg * c.k, &sb));
        KVO_CUDA(&c, dalloc(&c.res_fetched, sizeof(unsigned long long) * 2, &sb));
        const size_t rows = (size_t)c.batch * c.Hq;
        KVO_CUDA(&c, dalloc(&c.res_hit_slot, sizeof(int32_t) * lg * c.k, &sb));
        KVO_CUDA(&c, dalloc(&c.res_hit_cnt, sizeof(int32_t) * lg, &sb));
        // one per layer: a layer's hit pass never waits for an earlier layer's merge
        KVO_CUDA(&c, dalloc(&c.res_oA, sizeof(float) * c.L * rows * c.d, &sb));
        KVO_CUDA(&c, dalloc(&c.res_lA, sizeof(float) * c.L * rows, &sb));
        KVO_CUDA(&c, cudaMemsetAsync(c.res_fetched, 0, sizeof(unsigned long long) * 2, c.s_compute));
        KVO_CUDA(&c, dalloc(&c.res_pfbit, (size_t)c.L * c.G * 2 * c.k, &sb));
        KVO_CUDA(&c, dalloc(&c.res_stat, sizeof(unsigned long long) * 2 * c.L, &sb));
        KVO_CUDA(&c, dalloc(&c.res_pol, sizeof(unsigned long long) * 8 * c.L, &sb));
        KVO_CUDA(&c, dalloc(&c.res_pol_ticket, sizeof(uint32_t) * c.L, &sb));
        KVO_CUDA(&c, cudaMemsetAsync(c.res_pfbit, 0, (size_t)c.L * c.G * 2 * c.k, c.s_compute));
        KVO_CUDA(&c, cudaMemsetAsync(c.res_stat, 0, sizeof(unsigned long long) * 2 * c.L, c.s_compute));
        KVO_CUDA(&c, cudaMemsetAsync(c.res_pol_ticket, 0, sizeof(uint32_t) * c.L, c.s_compute));
        c.res_pending.assign(c.L, 0);
        KVO_CUDA(&c, kvo::prepare_resident(c));
        KVO_CUDA(&c, kvo::prepare_select_assign(c));
    }
    // selection scratch and work items
    const size_t Cmax4 = (size_t)((c.Cmax + 3) & ~3);
    KVO_CUDA(&c, dalloc(&c.sel_keys, sizeof(uint32_t) * 2 * c.G * Cmax4, &sb));
    KVO_CUDA(&c, dalloc(&c.sel_hist, sizeof(uint32_t) * 2 * c.G * 256, &sb));
    KVO_CUDA(&c, dalloc(&c.sel_done, sizeof(uint32_t) * c.G, &sb));
    KVO_CUDA(&c, cudaMemsetAsync(c.sel_hist, 0, sizeof(uint32_t) * 2 * c.G * 256, c.s_compute));
    KVO_CUDA(&c, cudaMemsetAsync(c.sel_done, 0, sizeof(uint32_t) * c.G, c.s_compute));
    std::vector<int2> sel_items;
    std::vector<int32_t> nch(c.G);
    {
        int dev = 0, sms = 0;
        KVO_CUDA(&c, cudaGetDevice(&dev));
        KVO_CUDA(&c, cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
        c.sel_sms = std::max(1, sms);
    }
    c.sel_rpt = select_rows_per_thread(c.G, Ccap.data(), c.sel_sms);
    const int sel_rows = kvo::SEL_THREADS * c.sel_rpt;
    for (int g = 0; g < c.G; ++g) {
        nch[g] = (Ccap[g] + sel_rows - 1) / sel_rows;     // rows past the current C_b are skipped
        for (int j = 0; j < nch[g]; ++j) sel_items.push_back(make_int2(g, j));
        c.sel_chunks_max = std::max(c.sel_chunks_max, nch[g]);
    }
    c.n_sel_items = (int)sel_items.size();
    set_sel_clu(c);
    KVO_CUDA(&c, dalloc(&c.sel_items, sizeof(int2) * sel_items.size(), &sb));
    KVO_CUDA(&c, dalloc(&c.sel_nchunks, sizeof(int32_t) * c.G, &sb));
    KVO_CUDA(&c, cudaMemcpy(c.sel_items, sel_items.data(), sizeof(int2) * sel_items.size(), cudaMemcpyHostToDevice));
    KVO_CUDA(&c, cudaMemcpy(c.sel_nchunks, nch.data(), sizeof(int32_t) * c.G, cudaMemcpyHostToDevice));
    // run scratch: [2][G][k] int4 + [2][G]
    KVO_CUDA(&c, dalloc(&c.runs, sizeof(int32_t) * 4 * 2 * (size_t)c.G * c.k, &sb));
    KVO_CUDA(&c, dalloc(&c.nruns, sizeof(int32_t) * 2 * c.G, &sb));
    // attention work items
    std::vector<int4> att;
    std::vector<int32_t> afirst(c.G), acount(c.G);
    const int sp_tiles = (c.k * c.B + kvo::ATT_TILE - 1) / kvo::ATT_TILE;
    const int w_max = c.max_append > 0 ? c.W + c.B - 1 : c.W;   // the window may grow to W + B - 1
    const int w_tiles = (w_max + kvo::ATT_TILE - 1) / kvo::ATT_TILE;
    for (int g = 0; g < c.G; ++g) {
        afirst[g] = (int)att.size();
        for (int t = 0; t < sp_tiles; t += kvo::ATT_TILES_PER_ITEM)
            att.push_back(make_int4(g, 0, t, std::min(kvo::ATT_TILES_PER_ITEM, sp_tiles - t)));
        for (int t = 0; t < w_tiles; t += kvo::ATT_TILES_PER_ITEM)
            att.push_back(make_int4(g, 1, t, std::min(kvo::ATT_TILES_PER_ITEM, w_tiles - t)));
        acount[g] = (int)att.size() - afirst[g];
    }
    c.n_att_items = (int)att.size();
    KVO_CUDA(&c, dalloc(&c.att_items, sizeof(int4) * att.size(), &sb));
    KVO_CUDA(&c, dalloc(&c.att_first, sizeof(int32_t) * c.G, &sb));
    KVO_CUDA(&c, dalloc(&c.att_count, sizeof(int32_t) * c.G, &sb));
    KVO_CUDA(&c, cudaMemcpy(c.att_items, att.data(), sizeof(int4) * att.size(), cudaMemcpyHostToDevice));
    KVO_CUDA(&c, cudaMemcpy(c.att_first, afirst.data(), sizeof(int32_t) * c.G, cudaMemcpyHostToDevice));
    KVO_CUDA(&c, cudaMemcpy(c.att_count, acount.data(), sizeof(int32_t) * c.G, cudaMemcpyHostToDevice));
    KVO_CUDA(&c, part_alloc(c, (int)att.size()));
    KVO_CUDA(&c, dalloc(&c.att_done, sizeof(uint32_t) * 2 * c.G, &sb));
    KVO_CUDA(&c, cudaMemsetAsync(c.att_done, 0, sizeof(uint32_t) * 2 * c.G, c.s_compute));
    KVO_CUDA(&c, kvo::prepare_attention(c));
    if (c.resident) {   // partials of the fetched-block attention of chain steps
        const size_t parts = (size_t)c.G * kvo::merge_part_split(c) * c.r;
        KVO_CUDA(&c, dalloc(&c.mp_part_o, sizeof(float) * parts * c.d, &sb));
        KVO_CUDA(&c, dalloc(&c.mp_part_ml, sizeof(float) * parts * 2, &sb));
        KVO_CUDA(&c, dalloc(&c.mp_done, sizeof(uint32_t) * c.G, &sb));
        KVO_CUDA(&c, cudaMemsetAsync(c.mp_done, 0, sizeof(uint32_t) * c.G, c.s_compute));
    }
    KVO_CUDA(&c, kvo::prepare_lowrank());
    c.lr_coef.assign(c.L, nullptr);
    c.lr_basis.assign(c.L, nullptr);
    c.lr_rank.assign(c.L, 0);
    KVO_CUDA(&c, dalloc(&c.status, sizeof(int32_t), &sb));
    KVO_CUDA(&c, cudaMemsetAsync(c.status, 0, sizeof(int32_t), c.s_compute));
    // decode-step state
    const size_t lgk = (size_t)c.L * c.G * c.k;
    KVO_CUDA(&c, dalloc(&c.st_true, sizeof(int32_t) * lgk, &sb));
    KVO_CUDA(&c, dalloc(&c.st_pred, sizeof(int32_t) * 2 * lgk, &sb));
    KVO_CUDA(&c, dalloc(&c.st_miss, sizeof(int32_t) * lgk, &sb));
    KVO_CUDA(&c, dalloc(&c.st_miss_cnt, sizeof(int32_t) * c.L * c.G, &sb));
    KVO_CUDA(&c, dalloc(&c.st_slot, sizeof(int32_t) * lgk, &sb));
    c.scratch_bytes = sb;
    for (auto* E : {&c.ev_eager, &c.ev_graph}) {
        for (auto* v : {&E->sel, &E->attn, &E->urg, &E->hit}) {
            v->assign(c.L, nullptr);
            for (auto& e : *v) KVO_CUDA(&c, cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
        }
        E->pref.assign(2, nullptr);
        for (auto& e : E->pref) KVO_CUDA(&c, cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
        for (auto* v : {&E->rassign, &E->rpref}) {
            v->assign(c.resident ? c.L : 0, nullptr);
            for (auto& e : *v) KVO_CUDA(&c, cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
        }
        KVO_CUDA(&c, cudaEventCreateWithFlags(&E->start, cudaEventDisableTiming));
    }
    KVO_CUDA(&c, cudaEventCreateWithFlags(&c.ev_gin, cudaEventDisableTiming));
    KVO_CUDA(&c, cudaEventCreateWithFlags(&c.ev_gout, cudaEventDisableTiming));
    KVO_CUDA(&c, cudaStreamCreateWithPriority(&c.s_graph, cudaStreamNonBlocking, (least + greatest) / 2));
    KVO_CUDA(&c, kvo::prepare_gather_tma());
    KVO_CUDA(&c, kvo::prepare_gather_flat());
    KVO_CUDA(&c, cudaStreamSynchronize(c.s_compute));
    return build_tma_plans(c);
}

kvo_status check_ctx(kvo_ctx* ctx) { return ctx ? KVO_OK : fail(nullptr, KVO_ERR_INVALID, "null context"); }

// buffer ids: 0, 1 ping-pong halves; 2 + l the resident set of layer l (resident mode)
bool buf_ok(const kvo::Ctx& c, int buf) { return buf == 0 || buf == 1 || (c.resident && buf >= 2 && buf < 2 + c.L); }

}  // namespace

void kvo::set_last_error(const char* msg) { g_err = msg ? msg : ""; }

extern "C" {

kvo_status kv_offload_init(const kvo_config* cfg, void* const* k_host, void* const* v_host,
                           const void* const* k_win, const void* const* v_win, kvo_ctx** out) {
    if (!out) return fail(nullptr, KVO_ERR_INVALID, "null output pointer");
    *out = nullptr;
    kvo_ctx* ctx = new (std::nothrow) kvo_ctx;
    if (!ctx) return fail(nullptr, KVO_ERR_OOM, "host allocation failed");
    kvo_status st = init_impl(ctx->c, cfg, k_host, v_host, k_win, v_win);
    if (st != KVO_OK) {
        g_err = ctx->c.err;
        free_ctx(ctx->c);
        delete ctx;
        return st;
    }
    *out = ctx;
    return KVO_OK;
}

kvo_status kv_offload_destroy(kvo_ctx* ctx) {
    if (!ctx) return KVO_OK;
    for (cudaStream_t s : {ctx->c.s_compute, ctx->c.s_prefetch, ctx->c.s_urgent, ctx->c.s_urgent2, ctx->c.s_hit, ctx->c.s_graph})
        if (s) cudaStreamSynchronize(s);
    free_ctx(ctx->c);
    delete ctx;
    return KVO_OK;
}

kvo_status select_topk(kvo_ctx* ctx, int layer, const void* q, const void* q_spec, int32_t* idx_true,
                       int32_t* idx_pred, kvo_stream_t stream) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (layer < 0 || layer >= c.L) return fail(&c, KVO_ERR_INVALID, "layer out of range");
    if (!q || !idx_true) return fail(&c, KVO_ERR_INVALID, "null q or idx_true");
    if (q_spec && !idx_pred) return fail(&c, KVO_ERR_INVALID, "q_spec given without idx_pred");
    KVO_CUDA(&c, kvo::launch_select(c, layer, q, q_spec, idx_true, q_spec ? idx_pred : nullptr, pick(c, stream),
                                    nullptr, true));
    return KVO_OK;
}

kvo_status index_diff(kvo_ctx* ctx, const int32_t* idx_true, const int32_t* idx_pred, int32_t* miss_idx,
                      int32_t* miss_cnt, int32_t* slot_of_true, kvo_stream_t stream) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (!idx_true || !miss_idx || !miss_cnt || !slot_of_true) return fail(&c, KVO_ERR_INVALID, "null pointer argument");
    KVO_CUDA(&c, kvo::launch_index_diff(c, idx_true, idx_pred, miss_idx, miss_cnt, slot_of_true, pick(c, stream)));
    return KVO_OK;
}

kvo_status gather_coalesced(kvo_ctx* ctx, int layer, int buf, const int32_t* idx, const int32_t* cnt, int slot_base,
                            int urgent, int32_t* runs_out, int32_t* n_runs_out, kvo_stream_t stream) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (layer < 0 || layer >= c.L) return fail(&c, KVO_ERR_INVALID, "layer out of range");
    if (!buf_ok(c, buf)) return fail(&c, KVO_ERR_INVALID, "buf must be 0 or 1 (or 2 + layer with resident = 1)");
    if (!idx) return fail(&c, KVO_ERR_INVALID, "null idx");
    if (slot_base < 0 || slot_base > c.k) return fail(&c, KVO_ERR_INVALID, "slot_base must be in [0, k]");
    if (runs_out && ((uintptr_t)runs_out % 16)) return fail(&c, KVO_ERR_INVALID, "runs_out must be 16-byte aligned");
    const int u = urgent ? 1 : 0;
    cudaStream_t s = stream ? (cudaStream_t)stream : (u ? c.s_urgent : c.s_prefetch);
    int32_t* runs = runs_out ? runs_out : c.runs + (size_t)u * 4 * c.G * c.k;
    int32_t* nruns = n_runs_out ? n_runs_out : c.nruns + (size_t)u * c.G;
    KVO_CUDA(&c, kvo::launch_coalesce(c, idx, cnt, slot_base, runs, nruns, s));
    if (c.gather_engine == 3)
        KVO_CUDA(&c, kvo::launch_gather_flat(c, layer, buf, idx, cnt, slot_base, s));
    else
        KVO_CUDA(&c, kvo::launch_gather(c, layer, buf, runs, nruns, s));
    return KVO_OK;
}

kvo_status sparse_decode_attn(kvo_ctx* ctx, int layer, int buf, const void* q, const int32_t* slot_of_true, float* o,
                              float* lse, int fuse_window_merge, kvo_stream_t stream) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (layer < 0 || layer >= c.L) return fail(&c, KVO_ERR_INVALID, "layer out of range");
    if (!buf_ok(c, buf)) return fail(&c, KVO_ERR_INVALID, "buf must be 0 or 1 (or 2 + layer with resident = 1)");
    if (!q || !slot_of_true || !o || !lse) return fail(&c, KVO_ERR_INVALID, "null pointer argument");
    KVO_CUDA(&c, kvo::launch_attention(c, layer, buf, q, nullptr, slot_of_true, o, lse, nullptr, nullptr,
                                       fuse_window_merge ? 1 : 0, pick(c, stream)));
    return KVO_OK;
}

kvo_status merge_lse(const float* o1, const float* lse1, const float* o2, const float* lse2, float* o, float* lse,
                     int rows, int d, kvo_stream_t stream) {
    if (rows < 0 || d < 1) return fail(nullptr, KVO_ERR_INVALID, "rows must be >= 0 and d >= 1");
    if (rows > 0 && (!o1 || !lse1 || !o2 || !lse2 || !o || !lse))
        return fail(nullptr, KVO_ERR_INVALID, "null pointer argument");
    if (rows > 0 && (lse == lse1 || lse == lse2)) return fail(nullptr, KVO_ERR_INVALID, "lse must not alias lse1 or lse2");
    cudaError_t e = kvo::launch_merge_lse(o1, lse1, o2, lse2, o, lse, rows, d, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "merge_lse launch");
    return KVO_OK;
}

// Enqueues one decode step ordered after `s_user` (which waits for all of it).
// Host state (parity, prediction) is not changed here.
static kvo_status decode_step_body(kvo_ctx* ctx, const void* q, const void* q_spec, float* o, float* lse,
                                   float* o_spec, float* lse_spec, cudaStream_t s_user, bool join_prefetch) {
    kvo::Ctx& c = ctx->c;
    kvo::Ctx::EvSet& E = join_prefetch ? c.ev_graph : c.ev_eager;
    const size_t gk = (size_t)c.G * c.k;
    const size_t q_layer = (size_t)c.batch * c.Hq * c.d;
    const size_t o_layer = q_layer, lse_layer = (size_t)c.batch * c.Hq;
    const int par = c.step_parity;
    int32_t* pred_cur = c.st_pred + (size_t)par * c.L * gk;
    int32_t* pred_next = c.st_pred + (size_t)(1 - par) * c.L * gk;
    const bool have = c.have_pred;
    int32_t* runs_pf = c.runs;
    int32_t* nruns_pf = c.nruns;
    int32_t* runs_ur = c.runs + (size_t)4 * gk;
    int32_t* nruns_ur = c.nruns + c.G;

    KVO_CUDA(&c, cudaEventRecord(E.start, s_user));
    for (cudaStream_t s : {c.s_compute, c.s_prefetch, c.s_urgent}) KVO_CUDA(&c, cudaStreamWaitEvent(s, E.start, 0));
    // launch wrapper: timing events around the launch when profiling is on
    int cur_layer = -1;
    auto timed = [&](int kind, cudaStream_t s, auto&& launch) -> cudaError_t {
        int e0, e1;
        cudaError_t e = prof_mark(c, s, &e0);
        if (e != cudaSuccess) return e;
        e = launch();
        if (e != cudaSuccess) return e;
        e = prof_mark(c, s, &e1);
        if (e != cudaSuccess) return e;
        if (e0 >= 0) {
            c.prof_recs.push_back({kind, e0, cur_layer});
            c.prof_recs.push_back({-1, e1, cur_layer});
        }
        return cudaSuccess;
    };

    // prefetch of a layer: the prediction list into slots [0, k) of its half
    auto prefetch = [&](int layer, int buf, const int32_t* pred, cudaEvent_t after) -> kvo_status {
        cur_layer = layer;
        KVO_CUDA(&c, cudaStreamWaitEvent(c.s_prefetch, after, 0));
        if (c.gather_engine == 3) {
            KVO_CUDA(&c, timed(kvo::PK_GATHER_PREFETCH, c.s_prefetch, [&] {
                return kvo::launch_gather_flat(c, layer, buf, pred, nullptr, 0, c.s_prefetch);
            }));
        } else {
            KVO_CUDA(&c, timed(kvo::PK_COALESCE, c.s_prefetch, [&] {
                return kvo::launch_coalesce(c, pred, nullptr, 0, runs_pf, nruns_pf, c.s_prefetch);
            }));
            KVO_CUDA(&c, timed(kvo::PK_GATHER_PREFETCH, c.s_prefetch,
                               [&] { return kvo::launch_gather(c, layer, buf, runs_pf, nruns_pf, c.s_prefetch); }));
        }
        KVO_CUDA(&c, cudaEventRecord(E.pref[buf], c.s_prefetch));
        return KVO_OK;
    };
    // A prefetch into each half is outstanding at step start when the previous
    // step issued one (layers 0 and 1, or layer 0 when n_layers == 1).
    // Half of layer l: parity of the global layer index step * L + l.
    auto half_of = [&](int l) { return (c.step_parity * (c.L & 1) + l) & 1; };
    // Inside a graph capture the previous step's prefetches are complete before
    // the graph starts (the launch waits for the prefetch stream), and waiting
    // on their events would tie the graph to work outside it.
    const bool prior_pref = have && !join_prefetch;
    bool pref_ready[2] = {false, false};
    pref_ready[half_of(0)] = prior_pref;
    if (c.L >= 2) pref_ready[half_of(1)] = prior_pref;
    for (int l = 0; l < c.L; ++l) {
        cur_layer = l;
        const int buf = half_of(l);
        const void* ql = (const char*)q + l * q_layer * 2;
        const void* qsl = q_spec ? (const char*)q_spec + l * q_layer * 2 : nullptr;
        int32_t* T = q_spec ? c.st_true + l * gk : pred_next + l * gk;
        int32_t* slot = c.st_slot + l * gk;
        int32_t* miss = c.st_miss + l * gk;
        int32_t* mcnt = c.st_miss_cnt + (size_t)l * c.G;
        // 1. retrieval index (true; speculative -> next step's prediction)
        KVO_CUDA(&c, timed(kvo::PK_SELECT, c.s_compute, [&] {
            return kvo::launch_select(c, l, ql, qsl, T, q_spec ? pred_next + l * gk : nullptr, c.s_compute);
        }));
        // 2. diff against the prediction made one step earlier
        KVO_CUDA(&c, timed(kvo::PK_DIFF, c.s_compute, [&] {
            return kvo::launch_index_diff(c, T, have ? pred_cur + l * gk : nullptr, miss, mcnt, slot, c.s_compute);
        }));
        KVO_CUDA(&c, cudaEventRecord(E.sel[l], c.s_compute));
        // single-layer model: the next step's prefetch can start now, into the other half
        if (c.L == 1) {
            kvo_status st = prefetch(l, buf ^ 1, pred_next + l * gk, E.sel[l]);
            if (st) return st;
        }
        // 3. urgent gather of the misses into slots [k, 2k)
        cur_layer = l;
        KVO_CUDA(&c, cudaStreamWaitEvent(c.s_urgent, E.sel[l], 0));
        if (c.lr_rank[l] > 0) {
            // low-rank layer: only V crosses the link (urgent stream) while the missed
            // keys are rebuilt on the GPU (compute stream, before the attention that reads them)
            KVO_CUDA(&c, timed(kvo::PK_GATHER_URGENT, c.s_urgent, [&] {
                return kvo::launch_gather_flat(c, l, buf, miss, mcnt, c.k, c.s_urgent, nullptr, 2);
            }));
            KVO_CUDA(&c, timed(kvo::PK_RECON, c.s_compute, [&] {
                return kvo::launch_lowrank_k(c, l, buf, miss, mcnt, c.k, nullptr, c.s_compute);
            }));
        } else if (c.gather_engine == 3) {
            KVO_CUDA(&c, timed(kvo::PK_GATHER_URGENT, c.s_urgent,
                               [&] { return kvo::launch_gather_flat(c, l, buf, miss, mcnt, c.k, c.s_urgent); }));
        } else {
            KVO_CUDA(&c, timed(kvo::PK_COALESCE, c.s_urgent, [&] {
                return kvo::launch_coalesce(c, miss, mcnt, c.k, runs_ur, nruns_ur, c.s_urgent);
            }));
            KVO_CUDA(&c, timed(kvo::PK_GATHER_URGENT, c.s_urgent,
                               [&] { return kvo::launch_gather(c, l, buf, runs_ur, nruns_ur, c.s_urgent); }));
        }
        KVO_CUDA(&c, cudaEventRecord(E.urg[l], c.s_urgent));
        // 4. attention once the misses and this half's prefetch have landed
        KVO_CUDA(&c, cudaStreamWaitEvent(c.s_compute, E.urg[l], 0));
        if (pref_ready[buf]) KVO_CUDA(&c, cudaStreamWaitEvent(c.s_compute, E.pref[buf], 0));
        KVO_CUDA(&c, timed(kvo::PK_ATTENTION, c.s_compute, [&] {
            return kvo::launch_attention(c, l, buf, ql, o_spec ? qsl : nullptr, slot, o + l * o_layer,
                                         lse + l * lse_layer, o_spec ? o_spec + l * o_layer : nullptr,
                                         lse_spec ? lse_spec + l * lse_layer : nullptr, 1, c.s_compute, true);
        }));
        KVO_CUDA(&c, cudaEventRecord(E.attn[l], c.s_compute));
        pref_ready[buf] = false;
        // 5. this half is free: prefetch global layer l + 2
        if (c.L >= 2) {
            const int t = l + 2;
            if (t < c.L) {
                if (have) {
                    kvo_status st = prefetch(t, buf, pred_cur + t * gk, E.attn[l]);
                    if (st) return st;
                    pref_ready[buf] = true;
                }
            } else {
                kvo_status st = prefetch(t - c.L, buf, pred_next + (t - c.L) * gk, E.attn[l]);
                if (st) return st;
            }
        }
    }
    // The caller's stream waits for the outputs (compute and urgent streams).
    // The prefetches issued for the next step stay in flight: the next step's
    // attention waits for them through ev_pref, and nothing before it reads or
    // overwrites what they touch.  A graph capture joins them too.
    for (cudaStream_t s : {c.s_compute, c.s_urgent, c.s_prefetch}) {
        if (s == c.s_prefetch && !join_prefetch) break;
        KVO_CUDA(&c, cudaEventRecord(E.start, s));
        KVO_CUDA(&c, cudaStreamWaitEvent(s_user, E.start, 0));
    }
    return KVO_OK;
}

// A resident step whose kernels form one chain: no speculative query, no
// prefetch of an earlier step in flight, no layer with low-rank keys.
static bool resident_alone(const kvo::Ctx& c, const void* q_spec) {
    if (q_spec) return false;
    for (int l = 0; l < c.L; ++l)
        if (c.res_pending[l] || c.lr_rank[l] > 0) return false;
    return true;
}

// Decode step with per-layer resident block sets (cross-step delta prefetch).
// Per layer l: select (true index, and with q_spec the prediction for the next
// step); urgent assign (T resident, sparing the prediction fetched for this
// step) and urgent gather of just the blocks that were missing; attention over
// the layer's resident set; then, with q_spec, prefetch assign (next step's
// prediction resident, sparing T) and its gather on the low-priority stream.
// Ordering: the next step's select of layer l waits for this step's prefetch
// assign of l (it reads T and the slot table), and its attention for the
// prefetch gather; urgent copies never touch slots of the prediction being
// prefetched, because the urgent assign spares them.
// Without a speculative query (nothing in flight, no low-rank layer) the step
// is one chain on the compute stream; its attention is split around the
// urgent copy (see below), and so is a speculative step's when no layer is
// low-rank.
static kvo_status decode_step_resident(kvo_ctx* ctx, const void* q, const void* q_spec, float* o, float* lse,
                                       float* o_spec, float* lse_spec, cudaStream_t s_user) {
    kvo::Ctx& c = ctx->c;
    kvo::Ctx::EvSet& E = c.ev_eager;
    const size_t gk = (size_t)c.G * c.k;
    const size_t q_layer = (size_t)c.batch * c.Hq * c.d;
    const size_t o_layer = q_layer, lse_layer = (size_t)c.batch * c.Hq;
    const int par = c.step_parity;
    int32_t* pred_cur = c.st_pred + (size_t)par * c.L * gk;
    int32_t* pred_next = c.st_pred + (size_t)(1 - par) * c.L * gk;
    const bool have = c.have_pred;
    // Without speculation, with no prefetch of an earlier step still in flight
    // and no layer rebuilding keys beside its copies, the step is four chains:
    // the compute stream selects and assigns layer after layer; two urgent
    // streams take the layers in turn, each copying a layer's missing blocks
    // once its assign is done and attending to the layer's resident blocks
    // beside the copy (a dependent launch that follows the copy's SMs, so the
    // copy keeps them); the attention stream (the prefetch stream, idle without
    // speculation) attends to the fetched blocks once they have landed and
    // merges.  So layer l + 1's copy starts while layer l's hit pass runs, and
    // the host link, HBM and the selection of later layers stay busy together.
    const bool alone_step = resident_alone(c, q_spec);
    const cudaStream_t sc = c.s_compute;                          // select, assign (and attention when speculating)
    const cudaStream_t sa = alone_step ? c.s_prefetch : sc;       // attention
    // A speculative step splits attention too when no layer rebuilds keys (a
    // whole-layer attention would share the hit passes' scratch): its hit pass
    // is launched plainly, at the compute stream's priority, on a stream of its
    // own beside the copy.  (At the urgent streams' priority its CTAs took SMs
    // ahead of the prefetch gathers that keep the link busy: always-prefetch
    // steps on long context slowed from 1.08 to 1.34-1.48 ms.)
    bool spec_split = q_spec && !alone_step && c.att_impl >= 1 && !o_spec;
    for (int l = 0; l < c.L && spec_split; ++l) spec_split = c.lr_rank[l] == 0;

    KVO_CUDA(&c, cudaEventRecord(E.start, s_user));
    for (cudaStream_t s : {c.s_compute, c.s_prefetch, c.s_urgent, c.s_urgent2, c.s_hit})
        KVO_CUDA(&c, cudaStreamWaitEvent(s, E.start, 0));
    int cur_layer = -1;
    auto timed = [&](int kind, cudaStream_t s, auto&& launch) -> cudaError_t {
        int e0, e1;
        cudaError_t e = prof_mark(c, s, &e0);
        if (e != cudaSuccess) return e;
        e = launch();
        if (e != cudaSuccess) return e;
        e = prof_mark(c, s, &e1);
        if (e != cudaSuccess) return e;
        if (e0 >= 0) {
            c.prof_recs.push_back({kind, e0, cur_layer});
            c.prof_recs.push_back({-1, e1, cur_layer});
        }
        return cudaSuccess;
    };
    for (int l = 0; l < c.L; ++l) {
        cur_layer = l;
        const int buf = 2 + l;
        const void* ql = (const char*)q + l * q_layer * 2;
        const void* qsl = q_spec ? (const char*)q_spec + l * q_layer * 2 : nullptr;
        int32_t* T = q_spec ? c.st_true + l * gk : pred_next + l * gk;
        int32_t* slot = c.st_slot + l * gk;
        int32_t* miss = c.st_miss + l * gk;
        int32_t* mcnt = c.st_miss_cnt + (size_t)l * c.G;
        int32_t* dsl = c.res_dslot + l * gk;
        int32_t* hit_slot = c.res_hit_slot + l * gk;       // per layer: layer l + 1's assign runs beside
        int32_t* hit_cnt = c.res_hit_cnt + (size_t)l * c.G;  // layer l's attention in a split step
        const cudaStream_t su = alone_step && (l & 1) ? c.s_urgent2 : c.s_urgent;   // urgent copies
        const bool pending = c.res_pending[l] != 0;
        // the previous step's prefetch of this layer has read T and written the slot table
        if (pending) KVO_CUDA(&c, cudaStreamWaitEvent(sc, E.rassign[l], 0));
        // A split step attends to the blocks resident already and the window
        // beside the urgent copies, to the fetched blocks after them, and merges
        // the two results by log-sum-exp.  A chain step's hit pass is a dependent
        // launch of the copy (under graph replay it starts beside the copy;
        // launched stream by stream it did not -- a chain step took 0.76 ms
        // instead of 0.50 on long context -- so steps that are not replayed
        // split only with a speculative query, their hit pass on a stream of
        // its own).
        const bool split = (alone_step && c.att_impl >= 1 && !o_spec && c.lr_rank[l] == 0) || spec_split;
        // 1. retrieval index (true; speculative -> next step's prediction), and
        // 2. urgent assign: T resident, sparing the prediction fetched for this
        // step -- without a speculative query, in the selection kernel itself
        if (!q_spec) {
            const kvo::ResAssignArgs aa =
                kvo::resident_assign_args(c, l, T, have ? pred_cur + l * gk : nullptr, miss, mcnt, dsl, slot, 0, -1,
                                          split ? hit_slot : nullptr, split ? hit_cnt : nullptr);
            KVO_CUDA(&c, timed(kvo::PK_SELECT, sc, [&] {
                return kvo::launch_select(c, l, ql, nullptr, T, nullptr, sc, &aa);
            }));
        } else {
            KVO_CUDA(&c, timed(kvo::PK_SELECT, sc, [&] {
                return kvo::launch_select(c, l, ql, qsl, T, pred_next + l * gk, sc);
            }));
            KVO_CUDA(&c, timed(kvo::PK_DIFF, sc, [&] {
                return kvo::launch_resident_assign(c, l, T, have ? pred_cur + l * gk : nullptr, miss, mcnt, dsl, slot,
                                                   0, sc, -1, split ? hit_slot : nullptr, split ? hit_cnt : nullptr);
            }));
        }
        // 3. urgent gather of the blocks that were missing
        KVO_CUDA(&c, cudaEventRecord(E.sel[l], sc));
        KVO_CUDA(&c, cudaStreamWaitEvent(su, E.sel[l], 0));
        // In-flight prefetch copies of this layer land first when nothing is spared
        // (no prediction).  (A chain step has none in flight; a speculative hit
        // pass waits for them itself.)
        if (pending && !have) KVO_CUDA(&c, cudaStreamWaitEvent(su, E.rpref[l], 0));
        const int urg_mask = c.lr_rank[l] > 0 ? 2 : 3;      // low-rank layer: V only, keys rebuilt
        KVO_CUDA(&c, timed(kvo::PK_GATHER_URGENT, su, [&] {
            return kvo::launch_gather_flat(c, l, buf, miss, mcnt, 0, su, dsl, urg_mask);
        }));
        if (split) {
            // the hits' result has a buffer per layer; the partials and tickets of the
            // persistent kernel alternate by layer parity, so each set serves the
            // layers of one stream (a chain step's urgent streams take the layers
            // in turn; a speculative step's hit passes share one stream)
            float* oA = c.res_oA + (size_t)l * o_layer;
            float* lA = c.res_lA + (size_t)l * lse_layer;
            if (alone_step) {
                // hits + window beside the copy: a programmatic dependent of the copy,
                // dispatched once the copy's SM-exclusive CTAs are all resident (so it
                // cannot take their SMs), completing after it
                KVO_CUDA(&c, timed(kvo::PK_ATTENTION, su, [&] {
                    return kvo::launch_attention(c, l, buf, ql, nullptr, hit_slot, oA, lA, nullptr, nullptr, 1, su,
                                                 true, hit_cnt, true, l & 1);
                }));
            } else {
                // hits + window on their own stream once the assign has listed them
                // and the blocks prefetched for this step have landed
                const cudaStream_t sh = c.s_hit;
                KVO_CUDA(&c, cudaStreamWaitEvent(sh, E.sel[l], 0));
                if (pending) KVO_CUDA(&c, cudaStreamWaitEvent(sh, E.rpref[l], 0));
                KVO_CUDA(&c, timed(kvo::PK_ATTENTION, sh, [&] {
                    return kvo::launch_attention(c, l, buf, ql, nullptr, hit_slot, oA, lA, nullptr, nullptr, 1, sh,
                                                 true, hit_cnt, false, l & 1);
                }));
                KVO_CUDA(&c, cudaEventRecord(E.hit[l], sh));
                KVO_CUDA(&c, cudaStreamWaitEvent(sa, E.hit[l], 0));
            }
            // the fetched blocks once they have landed, merged with the hits
            KVO_CUDA(&c, cudaEventRecord(E.urg[l], su));
            KVO_CUDA(&c, cudaStreamWaitEvent(sa, E.urg[l], 0));
            KVO_CUDA(&c, timed(kvo::PK_ATTENTION, sa, [&] {
                return kvo::launch_attn_merge_part(c, buf, ql, dsl, mcnt, oA, lA, o + l * o_layer,
                                                   lse + l * lse_layer, sa);
            }));
            KVO_CUDA(&c, cudaEventRecord(E.attn[l], sa));
            c.res_pending[l] = 0;
        } else {
            if (c.lr_rank[l] > 0)           // keys rebuilt on the compute stream, beside the V copies
                KVO_CUDA(&c, timed(kvo::PK_RECON, sc, [&] {
                    return kvo::launch_lowrank_k(c, l, buf, miss, mcnt, 0, dsl, sc);
                }));
            // 4. attention over the resident set once the urgent and prefetched blocks have landed
            KVO_CUDA(&c, cudaEventRecord(E.urg[l], su));
            KVO_CUDA(&c, cudaStreamWaitEvent(sa, E.urg[l], 0));
            if (pending) KVO_CUDA(&c, cudaStreamWaitEvent(sc, E.rpref[l], 0));
            c.res_pending[l] = 0;
            KVO_CUDA(&c, timed(kvo::PK_ATTENTION, sa, [&] {
                return kvo::launch_attention(c, l, buf, ql, o_spec ? qsl : nullptr, slot, o + l * o_layer,
                                             lse + l * lse_layer, o_spec ? o_spec + l * o_layer : nullptr,
                                             lse_spec ? lse_spec + l * lse_layer : nullptr, 1, sa, true);
            }));
            KVO_CUDA(&c, cudaEventRecord(E.attn[l], sa));
        }
        // 5. prefetch of the next step's prediction, sparing T (with the adaptive
        // policy the assign fetches nothing while the layer's prefetches do not pay)
        if (q_spec) {
            int32_t* pids = c.res_pf_ids + l * gk;
            int32_t* pcnt = c.res_pf_cnt + (size_t)l * c.G;
            int32_t* pdsl = c.res_pf_dslot + l * gk;
            KVO_CUDA(&c, cudaStreamWaitEvent(c.s_prefetch, E.attn[l], 0));
            KVO_CUDA(&c, timed(kvo::PK_DIFF, c.s_prefetch, [&] {
                return kvo::launch_resident_assign(c, l, pred_next + l * gk, T, pids, pcnt, pdsl, nullptr, 1,
                                                   c.s_prefetch, c.res_budget);
            }));
            KVO_CUDA(&c, cudaEventRecord(E.rassign[l], c.s_prefetch));
            KVO_CUDA(&c, timed(kvo::PK_GATHER_PREFETCH, c.s_prefetch,
                               [&] { return kvo::launch_gather_flat(c, l, buf, pids, pcnt, 0, c.s_prefetch, pdsl); }));
            KVO_CUDA(&c, cudaEventRecord(E.rpref[l], c.s_prefetch));
            c.res_pending[l] = 1;
        }
    }
    // the caller's stream waits for the outputs; prefetches stay in flight (a
    // chain step's attention stream is joined)
    for (cudaStream_t s : {c.s_compute, c.s_urgent, c.s_prefetch, c.s_urgent2, c.s_hit}) {
        if (s == c.s_prefetch && !alone_step) continue;
        KVO_CUDA(&c, cudaEventRecord(E.start, s));
        KVO_CUDA(&c, cudaStreamWaitEvent(s_user, E.start, 0));
    }
    return KVO_OK;
}

static void drop_graphs(kvo::Ctx& c) {
    for (auto& g : c.gexec)
        if (g) { cudaGraphExecDestroy(g); g = nullptr; }
}

// Replay the step graph of this step's parity, capturing it first when it is
// missing or was captured for other buffers.  The replay waits for the
// caller's stream and for `after` (work of earlier stream-launched steps it
// must follow); the compute stream and the caller's stream wait for it.
static kvo_status graph_step(kvo::Ctx& c, std::initializer_list<const void*> key_list, cudaStream_t s_user,
                             cudaStream_t after, const std::function<kvo_status()>& body) {
    const int par = c.step_parity;
    const void* key[6];
    int n = 0;
    for (const void* p : key_list) key[n++] = p;
    bool same = c.gexec[par] != nullptr;
    for (int i = 0; i < 6 && same; ++i) same = c.gkey[par][i] == key[i];
    if (!same) {
        if (c.gexec[par]) { cudaGraphExecDestroy(c.gexec[par]); c.gexec[par] = nullptr; }
        KVO_CUDA(&c, cudaStreamBeginCapture(c.s_graph, cudaStreamCaptureModeThreadLocal));
        kvo_status st = body();
        cudaGraph_t g = nullptr;
        cudaError_t e = cudaStreamEndCapture(c.s_graph, &g);
        if (st != KVO_OK) { if (g) cudaGraphDestroy(g); return st; }
        if (e != cudaSuccess) return cuda_fail(&c, e, "cudaStreamEndCapture(decode step)");
        e = cudaGraphInstantiate(&c.gexec[par], g, 0);
        cudaGraphDestroy(g);
        if (e != cudaSuccess) { c.gexec[par] = nullptr; return cuda_fail(&c, e, "cudaGraphInstantiate(decode step)"); }
        for (int i = 0; i < 6; ++i) c.gkey[par][i] = key[i];
    }
    KVO_CUDA(&c, cudaEventRecord(c.ev_gin, s_user));
    KVO_CUDA(&c, cudaStreamWaitEvent(c.s_graph, c.ev_gin, 0));
    KVO_CUDA(&c, cudaEventRecord(c.ev_gin, after));
    KVO_CUDA(&c, cudaStreamWaitEvent(c.s_graph, c.ev_gin, 0));
    KVO_CUDA(&c, cudaGraphLaunch(c.gexec[par], c.s_graph));
    KVO_CUDA(&c, cudaEventRecord(c.ev_gout, c.s_graph));
    KVO_CUDA(&c, cudaStreamWaitEvent(s_user, c.ev_gout, 0));
    KVO_CUDA(&c, cudaStreamWaitEvent(c.s_compute, c.ev_gout, 0));
    return KVO_OK;
}

static kvo_status decode_step_impl(kvo_ctx* ctx, const void* q, const void* q_spec, float* o, float* lse,
                                   float* o_spec, float* lse_spec, kvo_stream_t stream) {
    kvo::Ctx& c = ctx->c;
    cudaStream_t s_user = pick(c, stream);
    if (c.resident && c.use_graphs && c.have_pred && !c.prof_on && resident_alone(c, q_spec)) {
        // a chain step: replayed from the graph of its parity
        kvo_status st = graph_step(c, {q, q_spec, o, lse, o_spec, lse_spec}, s_user, c.s_compute, [&] {
            return decode_step_resident(ctx, q, q_spec, o, lse, o_spec, lse_spec, c.s_graph);
        });
        if (st != KVO_OK) return st;
    } else if (c.resident) {
        kvo_status st = decode_step_resident(ctx, q, q_spec, o, lse, o_spec, lse_spec, s_user);
        if (st != KVO_OK) return st;
    } else if (c.use_graphs && c.have_pred && !c.prof_on) {
        // prefetches an earlier stream-launched step left in flight finish first
        kvo_status st = graph_step(c, {q, q_spec, o, lse, o_spec, lse_spec}, s_user, c.s_prefetch, [&] {
            return decode_step_body(ctx, q, q_spec, o, lse, o_spec, lse_spec, c.s_graph, true);
        });
        if (st != KVO_OK) return st;
    } else {
        kvo_status st = decode_step_body(ctx, q, q_spec, o, lse, o_spec, lse_spec, s_user, false);
        if (st != KVO_OK) return st;
    }
    c.have_pred = true;
    c.step_parity ^= 1;
    return KVO_OK;
}

kvo_status kvo_set_graphs(kvo_ctx* ctx, int enable) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    if (enable && ctx->c.gather_engine == 4)
        return fail(&ctx->c, KVO_ERR_STATE, "graph replay needs a device-side gather engine (not engine 4)");
    for (cudaStream_t s : {ctx->c.s_compute, ctx->c.s_prefetch, ctx->c.s_urgent, ctx->c.s_urgent2, ctx->c.s_hit, ctx->c.s_graph})
        cudaStreamSynchronize(s);
    drop_graphs(ctx->c);
    ctx->c.use_graphs = enable != 0;
    return KVO_OK;
}

kvo_status kvo_decode_step(kvo_ctx* ctx, const void* q, const void* q_spec, float* o, float* lse,
                           kvo_stream_t stream) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    if (!q || !o || !lse) return fail(&ctx->c, KVO_ERR_INVALID, "null q, o or lse");
    return decode_step_impl(ctx, q, q_spec, o, lse, nullptr, nullptr, stream);
}

kvo_status kvo_decode_step_dual(kvo_ctx* ctx, const void* q, const void* q_spec, float* o, float* lse,
                                float* o_spec, float* lse_spec, kvo_stream_t stream) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (!q || !q_spec || !o || !lse || !o_spec || !lse_spec) return fail(&c, KVO_ERR_INVALID, "null pointer argument");
    if (2 * c.r > 16) return fail(&c, KVO_ERR_INVALID, "co-batching needs 2 * n_q_heads / n_kv_heads <= 16");
    return decode_step_impl(ctx, q, q_spec, o, lse, o_spec, lse_spec, stream);
}

kvo_status sparse_decode_attn_cobatch(kvo_ctx* ctx, int layer, int buf, const void* q, const void* q_spec,
                                      const int32_t* slot_of_true, float* o, float* lse, float* o_spec,
                                      float* lse_spec, int fuse_window_merge, kvo_stream_t stream) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (layer < 0 || layer >= c.L) return fail(&c, KVO_ERR_INVALID, "layer out of range");
    if (!buf_ok(c, buf)) return fail(&c, KVO_ERR_INVALID, "buf must be 0 or 1 (or 2 + layer with resident = 1)");
    if (!q || !q_spec || !slot_of_true || !o || !lse || !o_spec || !lse_spec)
        return fail(&c, KVO_ERR_INVALID, "null pointer argument");
    if (2 * c.r > 16) return fail(&c, KVO_ERR_INVALID, "co-batching needs 2 * n_q_heads / n_kv_heads <= 16");
    KVO_CUDA(&c, kvo::launch_attention(c, layer, buf, q, q_spec, slot_of_true, o, lse, o_spec, lse_spec,
                                       fuse_window_merge ? 1 : 0, pick(c, stream)));
    return KVO_OK;
}

kvo_status kvo_append(kvo_ctx* ctx, const void* k_new, const void* v_new, kvo_stream_t stream) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (!k_new || !v_new) return fail(&c, KVO_ERR_INVALID, "null k_new or v_new");
    if (c.max_append == 0) return fail(&c, KVO_ERR_STATE, "context built with max_append == 0");
    if (c.appended >= c.max_append) return fail(&c, KVO_ERR_STATE, "append capacity used up");
    KVO_CUDA(&c, kvo::launch_append(c, k_new, v_new, pick(c, stream)));
    ++c.appended;
    return KVO_OK;
}

kvo_status kvo_reset_prediction(kvo_ctx* ctx) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    for (cudaStream_t s : {ctx->c.s_compute, ctx->c.s_prefetch, ctx->c.s_urgent, ctx->c.s_urgent2, ctx->c.s_hit, ctx->c.s_graph}) cudaStreamSynchronize(s);
    ctx->c.have_pred = false;
    ctx->c.step_parity = 0;
    return KVO_OK;
}

kvo_status kvo_get_stream(kvo_ctx* ctx, int which, kvo_stream_t* out) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    if (!out || which < 0 || which > 2) return fail(&ctx->c, KVO_ERR_INVALID, "bad stream selector");
    *out = which == 0 ? ctx->c.s_compute : which == 1 ? ctx->c.s_prefetch : ctx->c.s_urgent;
    return KVO_OK;
}

kvo_status kvo_device_status(kvo_ctx* ctx, int32_t* code_out, kvo_stream_t stream) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (stream) KVO_CUDA(&c, cudaStreamSynchronize((cudaStream_t)stream));
    for (cudaStream_t s : {c.s_compute, c.s_prefetch, c.s_urgent, c.s_urgent2, c.s_hit}) KVO_CUDA(&c, cudaStreamSynchronize(s));
    int32_t v = 0;
    KVO_CUDA(&c, cudaMemcpy(&v, c.status, sizeof(v), cudaMemcpyDeviceToHost));
    KVO_CUDA(&c, cudaMemset(c.status, 0, sizeof(int32_t)));
    if (code_out) *code_out = v;
    if (v) return fail(&c, KVO_ERR_DEVICE, "device status word " + std::to_string(v));
    return KVO_OK;
}

kvo_status kvo_landmarks(kvo_ctx* ctx, int layer, void* dst, kvo_stream_t stream) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (layer < 0 || layer >= c.L || !dst) return fail(&c, KVO_ERR_INVALID, "bad layer or null dst");
    KVO_CUDA(&c, kvo::copy_landmarks_logical(c, layer, dst, pick(c, stream)));
    return KVO_OK;
}

kvo_status kvo_buffer(kvo_ctx* ctx, int buf, void** k_out, void** v_out) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    if (!buf_ok(ctx->c, buf) || !k_out || !v_out) return fail(&ctx->c, KVO_ERR_INVALID, "bad buf or null output");
    *k_out = ctx->c.buf_k(buf);
    *v_out = ctx->c.buf_v(buf);
    return KVO_OK;
}

kvo_status kvo_info(kvo_ctx* ctx, int64_t* out4) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    if (!out4) return fail(&ctx->c, KVO_ERR_INVALID, "null output");
    out4[0] = ctx->c.Cmax;
    out4[1] = (int64_t)ctx->c.lm_bytes;
    out4[2] = (int64_t)ctx->c.pp_bytes;
    out4[3] = (int64_t)ctx->c.scratch_bytes;
    return KVO_OK;
}

kvo_status kvo_resident_slots(kvo_ctx* ctx, int layer, int32_t* slots_out) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (!c.resident) return fail(&c, KVO_ERR_STATE, "context built with resident = 0");
    if (layer < 0 || layer >= c.L || !slots_out) return fail(&c, KVO_ERR_INVALID, "bad layer or null output");
    for (cudaStream_t s : {c.s_compute, c.s_prefetch, c.s_urgent, c.s_urgent2, c.s_hit}) KVO_CUDA(&c, cudaStreamSynchronize(s));
    const size_t n = (size_t)c.G * 2 * c.k;
    KVO_CUDA(&c, cudaMemcpy(slots_out, c.res_slots + (size_t)layer * n, sizeof(int32_t) * n, cudaMemcpyDeviceToHost));
    return KVO_OK;
}

kvo_status kvo_set_lowrank_keys(kvo_ctx* ctx, int layer, int rank, const void* coef, const void* basis) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (layer < 0 || layer >= c.L) return fail(&c, KVO_ERR_INVALID, "bad layer");
    if (rank < 0 || rank > 64) return fail(&c, KVO_ERR_INVALID, "rank must be in 0..64");
    if (rank > 0 && (!coef || !basis)) return fail(&c, KVO_ERR_INVALID, "rank > 0 needs coef and basis");
    for (cudaStream_t s : {c.s_compute, c.s_prefetch, c.s_urgent, c.s_urgent2, c.s_hit, c.s_graph}) KVO_CUDA(&c, cudaStreamSynchronize(s));
    drop_graphs(c);
    c.lr_rank[layer] = rank;
    c.lr_coef[layer] = rank > 0 ? (const uint16_t*)coef : nullptr;
    c.lr_basis[layer] = rank > 0 ? (const uint16_t*)basis : nullptr;
    return KVO_OK;
}

kvo_status kvo_set_prefetch_budget(kvo_ctx* ctx, int blocks) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (!c.resident) return fail(&c, KVO_ERR_STATE, "context built with resident = 0");
    if (blocks < -1) return fail(&c, KVO_ERR_INVALID, "blocks must be >= -1");
    for (cudaStream_t s : {c.s_compute, c.s_prefetch, c.s_urgent, c.s_urgent2, c.s_hit}) KVO_CUDA(&c, cudaStreamSynchronize(s));
    c.res_budget = blocks;
    return KVO_OK;
}

kvo_status kvo_set_spec_policy(kvo_ctx* ctx, int mode) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (!c.resident) return fail(&c, KVO_ERR_STATE, "context built with resident = 0");
    if (mode < 0 || mode > 1) return fail(&c, KVO_ERR_INVALID, "mode must be 0 or 1");
    for (cudaStream_t s : {c.s_compute, c.s_prefetch, c.s_urgent, c.s_urgent2, c.s_hit, c.s_graph})
        KVO_CUDA(&c, cudaStreamSynchronize(s));
    drop_graphs(c);
    // every layer starts a fresh window with its prefetch on
    std::vector<unsigned long long> init(8 * (size_t)c.L, 0ull);
    for (int l = 0; l < c.L; ++l) init[8 * l] = 1;
    KVO_CUDA(&c, cudaMemcpy(c.res_pol, init.data(), sizeof(unsigned long long) * 8 * c.L, cudaMemcpyHostToDevice));
    c.spec_policy = mode;
    return KVO_OK;
}

kvo_status kvo_spec_stats(kvo_ctx* ctx, int64_t* out3) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (!c.resident) return fail(&c, KVO_ERR_STATE, "context built with resident = 0");
    if (!out3) return fail(&c, KVO_ERR_INVALID, "null output");
    for (cudaStream_t s : {c.s_compute, c.s_prefetch, c.s_urgent, c.s_urgent2, c.s_hit}) KVO_CUDA(&c, cudaStreamSynchronize(s));
    std::vector<unsigned long long> h(2 * (size_t)c.L), p(8 * (size_t)c.L);
    KVO_CUDA(&c, cudaMemcpy(h.data(), c.res_stat, sizeof(unsigned long long) * 2 * c.L, cudaMemcpyDeviceToHost));
    KVO_CUDA(&c, cudaMemcpy(p.data(), c.res_pol, sizeof(unsigned long long) * 8 * c.L, cudaMemcpyDeviceToHost));
    for (int l = 0; l < c.L; ++l) {
        out3[3 * l + 0] = (int64_t)h[2 * l];
        out3[3 * l + 1] = (int64_t)h[2 * l + 1];
        out3[3 * l + 2] = c.spec_policy == 1 ? (p[8 * l] ? 1 : 0) : 1;
    }
    return KVO_OK;
}

kvo_status kvo_resident_fetched(kvo_ctx* ctx, int64_t* out2, int reset) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (!c.resident) return fail(&c, KVO_ERR_STATE, "context built with resident = 0");
    if (!out2) return fail(&c, KVO_ERR_INVALID, "null output");
    for (cudaStream_t s : {c.s_compute, c.s_prefetch, c.s_urgent, c.s_urgent2, c.s_hit}) KVO_CUDA(&c, cudaStreamSynchronize(s));
    unsigned long long h[2];
    KVO_CUDA(&c, cudaMemcpy(h, c.res_fetched, sizeof(h), cudaMemcpyDeviceToHost));
    out2[0] = (int64_t)h[0];
    out2[1] = (int64_t)h[1];
    if (reset) KVO_CUDA(&c, cudaMemset(c.res_fetched, 0, sizeof(h)));
    return KVO_OK;
}

kvo_status kvo_plan_select(int n_groups, const int32_t* blocks_per_group, int n_sms, int impl, int32_t* out4) {
    if (n_groups <= 0 || !blocks_per_group || n_sms <= 0 || impl < 0 || impl > 2 || !out4) {
        kvo::set_last_error("kvo_plan_select: need n_groups, n_sms > 0, impl in 0..2, non-null arrays");
        return KVO_ERR_INVALID;
    }
    int Cmax = 0;
    for (int g = 0; g < n_groups; ++g) {
        if (blocks_per_group[g] < 0) {
            kvo::set_last_error("kvo_plan_select: negative block count");
            return KVO_ERR_INVALID;
        }
        Cmax = std::max(Cmax, (int)blocks_per_group[g]);
    }
    const int rpt = select_rows_per_thread(n_groups, blocks_per_group, n_sms);
    const int rows = kvo::SEL_THREADS * rpt;
    int64_t n_ctas = 0;
    int chunks_max = 0;
    for (int g = 0; g < n_groups; ++g) {
        const int n = (blocks_per_group[g] + rows - 1) / rows;
        n_ctas += n;
        chunks_max = std::max(chunks_max, n);
    }
    out4[0] = rpt;
    out4[1] = chunks_max;
    out4[2] = (int32_t)std::min<int64_t>(n_ctas, INT32_MAX);
    out4[3] = select_cluster_ctas(impl, chunks_max, n_ctas, Cmax, n_sms);
    return KVO_OK;
}

kvo_status kvo_plan_attention(int n_groups, int sparse_tokens, int window_tokens, int grid, int32_t* items_out,
                              int items_cap, int32_t* cta_out, int32_t* n_items_out, int32_t* grid_out) {
    if (n_groups <= 0 || sparse_tokens < 0 || window_tokens < 0 || sparse_tokens + window_tokens <= 0 || grid <= 0 ||
        items_cap < 0 || !n_items_out || !grid_out) {
        kvo::set_last_error("kvo_plan_attention: need n_groups, grid > 0, token counts >= 0 (not both 0), non-null counts");
        return KVO_ERR_INVALID;
    }
    std::vector<int4> items;
    std::vector<int32_t> cta;
    const int64_t used = plan_tma_items(n_groups, sparse_tokens, window_tokens, grid, items, cta);
    *n_items_out = (int32_t)items.size();
    *grid_out = (int32_t)used;
    if (items_out) {
        if ((size_t)items_cap < items.size()) {
            kvo::set_last_error("kvo_plan_attention: items_cap below the item count (see n_items_out)");
            return KVO_ERR_INVALID;
        }
        for (size_t i = 0; i < items.size(); ++i) {
            items_out[4 * i + 0] = items[i].x; items_out[4 * i + 1] = items[i].y;
            items_out[4 * i + 2] = items[i].z; items_out[4 * i + 3] = items[i].w;
        }
    }
    if (cta_out)
        for (size_t j = 0; j < cta.size(); ++j) cta_out[j] = cta[j];
    return KVO_OK;
}

kvo_status kvo_set_gather_shape(kvo_ctx* ctx, int ctas, int threads, int unroll) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    for (cudaStream_t s : {ctx->c.s_compute, ctx->c.s_prefetch, ctx->c.s_urgent, ctx->c.s_urgent2, ctx->c.s_hit, ctx->c.s_graph}) cudaStreamSynchronize(s);
    drop_graphs(ctx->c);
    const int max_threads = ctx->c.gather_engine == 3 ? 1024 : kvo::GATHER_THREADS;
    if (ctas < 0 || ctas > 65535 || threads < 32 || threads > max_threads || threads % 32 ||
        (unroll != 1 && unroll != 2 && unroll != 4))
        return fail(&ctx->c, KVO_ERR_INVALID,
                    "need 0 <= ctas <= 65535, threads a multiple of 32 (<= 256; <= 1024 for engine 3), unroll 1|2|4");
    ctx->c.gather_ctas = ctas;
    ctx->c.gather_threads = threads;
    ctx->c.gather_unroll = unroll;
    return build_tma_plans(ctx->c);   // the step's attention plan depends on the gather's SMs
}

kvo_status kvo_set_gather_reserve(kvo_ctx* ctx, int smem_bytes) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    for (cudaStream_t s : {ctx->c.s_compute, ctx->c.s_prefetch, ctx->c.s_urgent, ctx->c.s_urgent2, ctx->c.s_hit, ctx->c.s_graph}) cudaStreamSynchronize(s);
    drop_graphs(ctx->c);
    if (smem_bytes < 0 || smem_bytes > 227 * 1024 - 128)
        return fail(&ctx->c, KVO_ERR_INVALID, "0 <= smem_bytes <= 232320 (227 KiB less 128 bytes)");
    ctx->c.gather_reserve_smem = smem_bytes;
    return build_tma_plans(ctx->c);   // the step's attention plan depends on the gather's SMs
}

kvo_status kvo_set_gather_engine(kvo_ctx* ctx, int engine, int drivers) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    for (cudaStream_t s : {ctx->c.s_compute, ctx->c.s_prefetch, ctx->c.s_urgent, ctx->c.s_urgent2, ctx->c.s_hit, ctx->c.s_graph}) cudaStreamSynchronize(s);
    drop_graphs(ctx->c);
    // engine 1: 4 batches per driver; engine 2: 8 batches per driver (one driver per CTA)
    if (engine < 0 || engine > 4 || drivers < 0 || drivers > 4096)
        return fail(&ctx->c, KVO_ERR_INVALID, "engine must be 0..4 and 0 <= drivers <= 4096");
    kvo::Ctx& c = ctx->c;
    if (engine == 4) {
        // the copy engine reads the run list back: pinned staging, and no graph
        // capture (the host waits for the list inside the step)
        if (!c.h_runs) KVO_CUDA(&c, cudaHostAlloc((void**)&c.h_runs, sizeof(int32_t) * 4 * (size_t)c.G * c.k,
                                                  cudaHostAllocDefault));
        if (!c.h_nruns) KVO_CUDA(&c, cudaHostAlloc((void**)&c.h_nruns, sizeof(int32_t) * c.G, cudaHostAllocDefault));
        c.use_graphs = false;
    }
    ctx->c.gather_engine = engine == 0 ? 0 : engine == 3 ? 3 : engine == 4 ? 4 : 1;
    // each engine starts from its own default launch shape
    if (engine == 3) {
        ctx->c.gather_ctas = 38; ctx->c.gather_threads = 1024; ctx->c.gather_unroll = 2;
        ctx->c.gather_reserve_smem = 200 * 1024;
    } else {
        ctx->c.gather_ctas = 0; ctx->c.gather_threads = 128; ctx->c.gather_unroll = 1;
        ctx->c.gather_reserve_smem = 0;
    }
    ctx->c.gather_stages = engine == 2 ? 8 : 4;
    ctx->c.gather_drivers = drivers;
    return build_tma_plans(ctx->c);   // the step's attention plan depends on the gather's SMs
}

kvo_status kvo_set_attn_impl(kvo_ctx* ctx, int impl, int ctas) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    if (impl < 0 || impl > 2 || ctas < 0 || (impl == 2 && ctas > 8))
        return fail(&ctx->c, KVO_ERR_INVALID,
                    "attention implementation must be 0, 1 or 2, ctas >= 0, and ctas <= 8 for implementation 2");
    for (cudaStream_t s : {ctx->c.s_compute, ctx->c.s_prefetch, ctx->c.s_urgent, ctx->c.s_urgent2, ctx->c.s_hit, ctx->c.s_graph}) cudaStreamSynchronize(s);
    drop_graphs(ctx->c);
    ctx->c.att_impl = impl;
    ctx->c.tma_ctas = impl == 2 ? 0 : ctas;
    ctx->c.att_cluster = impl == 2 ? ctas : 0;
    return build_tma_plans(ctx->c);
}

kvo_status kvo_set_select_impl(kvo_ctx* ctx, int impl) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (impl < 0 || impl > 2) return fail(&c, KVO_ERR_INVALID, "selection implementation must be 0, 1 or 2");
    for (cudaStream_t s : {c.s_compute, c.s_prefetch, c.s_urgent, c.s_urgent2, c.s_hit, c.s_graph})
        KVO_CUDA(&c, cudaStreamSynchronize(s));
    drop_graphs(c);
    c.sel_impl = impl;
    set_sel_clu(c);
    return KVO_OK;
}

kvo_status kvo_set_wait_test(kvo_ctx* ctx, int64_t limit_ns, int skip_tile) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (limit_ns < 1000000 || limit_ns > 10000000000LL || skip_tile < -1)
        return fail(&c, KVO_ERR_INVALID, "need 1 ms <= limit_ns <= 10 s and skip_tile >= -1");
    for (cudaStream_t s : {c.s_compute, c.s_prefetch, c.s_urgent, c.s_urgent2, c.s_hit, c.s_graph}) KVO_CUDA(&c, cudaStreamSynchronize(s));
    drop_graphs(c);
    c.att_wait_ns = limit_ns;
    c.att_skip_tile = skip_tile;
    return KVO_OK;
}

kvo_status kvo_profile(kvo_ctx* ctx, int enable) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    c.prof_on = enable != 0;
    c.prof_recs.clear();
    c.prof_used = 0;
    return KVO_OK;
}

kvo_status kvo_profile_read(kvo_ctx* ctx, double* ms_out, int64_t* launches_out, int n_kinds) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (!ms_out || !launches_out || n_kinds < kvo::PK_COUNT) return fail(&c, KVO_ERR_INVALID, "need 7 output slots");
    for (int i = 0; i < n_kinds; ++i) { ms_out[i] = 0.0; launches_out[i] = 0; }
    for (size_t i = 0; i + 1 < c.prof_recs.size(); i += 2) {
        cudaEvent_t a = c.prof_pool[c.prof_recs[i].ev], b = c.prof_pool[c.prof_recs[i + 1].ev];
        KVO_CUDA(&c, cudaEventSynchronize(b));
        float ms = 0.f;
        KVO_CUDA(&c, cudaEventElapsedTime(&ms, a, b));
        ms_out[c.prof_recs[i].kind] += ms;
        launches_out[c.prof_recs[i].kind] += 1;
    }
    c.prof_recs.clear();
    c.prof_used = 0;
    return KVO_OK;
}

kvo_status kvo_profile_trace(kvo_ctx* ctx, double* start_ms, double* end_ms, int32_t* kind, int32_t* layer,
                             int cap, int* n_out) {
    if (check_ctx(ctx)) return KVO_ERR_INVALID;
    kvo::Ctx& c = ctx->c;
    if (!n_out || cap < 0 || (cap > 0 && (!start_ms || !end_ms || !kind || !layer)))
        return fail(&c, KVO_ERR_INVALID, "bad trace output arguments");
    const int n = (int)(c.prof_recs.size() / 2);
    *n_out = n;
    if (n == 0) return KVO_OK;
    cudaEvent_t base = c.prof_pool[c.prof_recs[0].ev];
    for (int i = 0; i < n && i < cap; ++i) {
        cudaEvent_t a = c.prof_pool[c.prof_recs[2 * i].ev], b = c.prof_pool[c.prof_recs[2 * i + 1].ev];
        KVO_CUDA(&c, cudaEventSynchronize(b));
        float t0 = 0.f, t1 = 0.f;
        KVO_CUDA(&c, cudaEventElapsedTime(&t0, base, a));
        KVO_CUDA(&c, cudaEventElapsedTime(&t1, base, b));
        start_ms[i] = t0;
        end_ms[i] = t1;
        kind[i] = c.prof_recs[2 * i].kind;
        layer[i] = c.prof_recs[2 * i].layer;
    }
    return KVO_OK;
}

const char* kvo_last_error(const kvo_ctx* ctx) {
    if (ctx) return ctx->c.err.c_str();
    return g_err.c_str();
}

}  // extern "C"
