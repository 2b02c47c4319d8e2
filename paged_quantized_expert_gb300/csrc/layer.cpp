// layer.cpp -- native runtime of one paged MoE layer: a step is
//   route -> permute -> counts to the host (the one sync of a step) ->
//   page_table_update -> refills of the misses on a side stream ->
//   page table to the device -> (compute stream waits for the refills) ->
//   expert FFN over the slot pool -> combine.
//
// Expert-pager article (rand.pepabo.com), "エキスパート重みの階層ページング":
// per-layer VRAM slots managed LRU, copy-in of a missing expert, working buffer
// when a step needs more experts than slots; "重みの圧縮": compressed host pages
// decoded on the GPU as they arrive (one pass pulls and decodes every miss).
// MoE-Gen summary (aibr.jp), "3.中核となる技術的要素": host-to-device transfers
// overlap compute (side stream).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "pqe.h"
#include "pqe_common.cuh"

namespace pqe {
void set_last_cuda_error(cudaError_t e);
}

namespace {

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

struct ScratchMap {
    size_t status, topk_ids, topk_w, counts, offsets, perm_src, inv, page_table, perm_ws, ffn_ws, out_perm, x_in,
        logits_in, y_out, lru, miss, host_pages, page_bytes, total;
    size_t perm_ws_bytes, ffn_ws_bytes, staging_bytes;
};

ScratchMap scratch_map(const pqe_layer_config &c) {
    ScratchMap m{};
    const size_t A = (size_t)c.max_T * c.k;
    size_t off = 0;
    auto take = [&off](size_t bytes) {
        size_t at = off;
        off += up256(bytes == 0 ? 1 : bytes);
        return at;
    };
    m.status = take(sizeof(int32_t));
    m.topk_ids = take(sizeof(int32_t) * A);
    m.topk_w = take(sizeof(float) * A);
    m.counts = take(sizeof(int32_t) * c.E);
    m.offsets = take(sizeof(int32_t) * (c.E + 1));
    m.perm_src = take(sizeof(int32_t) * A);
    m.inv = take(sizeof(int32_t) * A);
    m.page_table = take(sizeof(int32_t) * c.E);
    m.perm_ws_bytes = moe_permute_workspace_size(c.max_T, c.k, c.E);
    m.perm_ws = take(m.perm_ws_bytes);
    m.ffn_ws_bytes = moe_paged_ffn_workspace_size(c.max_T, c.k, c.E, c.H, c.I);
    m.ffn_ws = take(m.ffn_ws_bytes);
    m.out_perm = take(sizeof(uint16_t) * A * c.H);
    m.x_in = take(sizeof(uint16_t) * (size_t)c.max_T * c.H);
    m.logits_in = take(sizeof(float) * (size_t)c.max_T * c.E);
    m.y_out = take(sizeof(uint16_t) * (size_t)c.max_T * c.H);
    // compressed refills are decoded straight from the host pages (no staging);
    // staging_bytes only bounds a compressed page's size
    m.staging_bytes = c.compressed ? pqe_huff_page_bound(c.H, c.I) : 0;
    if (c.device_pager) {
        m.lru = take(pqe_lru_device_bytes(c.E, c.S));
        m.miss = take(sizeof(int32_t) * (3 * (size_t)c.E + 3));
        m.host_pages = take(sizeof(uint64_t) * c.E);
        m.page_bytes = take(sizeof(size_t) * c.E);
    }
    m.total = off;
    return m;
}

// CTAs of the refill kernel in an overlapped step: eight already pull pinned
// host pages at the host link's rate alone; beside the FFN passes 32 did best
// (16 and 64 within 2 us of it at T=64), the rest of the GPU runs the FFN
constexpr int OVERLAP_FILL_CTAS = 32;
// SMs of an FFN pass that runs beside a refill: the passes have slack (each
// runs under a refill at least half its size), and fewer SMs disturb the
// refill less (T=64: 2233 us on all but the refill's SMs, 2224 on 48-96)
constexpr int OVERLAP_FFN_SMS = 64;

bool config_ok(const pqe_layer_config *c) {
    if (!c || c->E < 1 || c->E > 1024 || c->k < 1 || c->k > 32 || c->k > c->E || c->S < 0 || c->W < 0 ||
        c->max_T < 1 || (size_t)c->max_T * c->k >= (1u << 30) || pqe_page_bytes(PQE_FMT_FP8, c->H, c->I) == 0)
        return false;
    // the device pager: at most 1024 slots, a working buffer for any step
    if (c->device_pager && (c->S > 1024 || c->W < c->E)) return false;
    if (c->overlap_groups < 0 || c->overlap_groups > PQE_MAX_OVERLAP_GROUPS ||
        (c->overlap_groups > 0 && !c->device_pager))
        return false;
    return true;
}

}  // namespace

struct pqe_layer {
    pqe_layer_config cfg{};
    pqe_pool pool{};
    std::vector<const void *> host_pages;
    std::vector<size_t> host_bytes;
    const uint8_t *luts = nullptr;
    const uint8_t *expert_fmt = nullptr;
    uint8_t *scratch = nullptr;
    ScratchMap map{};
    pqe_lru *lru = nullptr;
    int32_t *pinned = nullptr;  // counts [E], page table [E], miss expert [E], miss dest [E]
    cudaEvent_t ev_counts = nullptr, ev_fill = nullptr;
    cudaEvent_t ev_lru = nullptr, ev_group[PQE_MAX_OVERLAP_GROUPS] = {};  // overlapped device-pager steps
    cudaEvent_t ev_ffn_begin = nullptr, ev_ffn_end = nullptr;  // caller's, optional
    std::vector<const void *> fill_src;  // [E] scratch for slot_fill_batch / slot_fill_compressed_batch
    std::vector<size_t> fill_bytes;
    std::vector<const uint8_t *> fill_lut13, fill_lut2;
    std::vector<int32_t> fill_dest, fill_expert;
    // optional RAM tier: the step's misses are served from its RAM pages
    pqe_ram_tier *ram = nullptr;
    std::vector<int32_t> ram_need, ram_queued;
    std::vector<const void *> ram_page;
    std::vector<size_t> ram_bytes;
    // pqe_layer_step_host on a device-pager layer: the step's launches captured
    // once per shape and replayed (the first call of a shape runs eagerly)
    struct StepGraph {
        int T;
        const float *w_router;
        bool overlap;
        uint64_t gen;
        int state;  // 0 seen once, 1 exec built, -1 capture failed (eager from then on)
        cudaGraphExec_t exec;
    };
    std::vector<StepGraph> graphs;
    bool step_graphs = true;

    template <class T>
    T *at(size_t off) const {
        return reinterpret_cast<T *>(scratch + off);
    }
};

namespace {

// Records one of the caller's FFN timing events on s. Inside a stream capture
// a plain record only orders streams; an external record becomes an event node
// that each replay of the graph records, so the FFN inside a replayed step can
// be timed too.
cudaError_t record_timing(cudaEvent_t ev, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t ce = cudaStreamIsCapturing(s, &cs);
    if (ce != cudaSuccess) return ce;
    return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                                               : cudaEventRecord(ev, s);
}

// Refills the n pages described by L->fill_* on `side`: one pull+decode pass
// for compressed pages, one bulk pull for FP8 pages.
int refill(pqe_layer *L, int n, cudaStream_t side, int32_t *status) {
    if (n == 0) return PQE_OK;
    if (L->cfg.compressed) {
        for (int i = 0; i < n; ++i) {
            L->fill_lut13[i] = L->luts + (size_t)L->fill_expert[i] * 2 * PQE_HUFF_LUT_BYTES;
            L->fill_lut2[i] = L->fill_lut13[i] + PQE_HUFF_LUT_BYTES;
        }
        return slot_fill_compressed_batch(&L->pool, n, L->fill_dest.data(), L->fill_src.data(),
                                          L->fill_bytes.data(), L->fill_lut13.data(), L->fill_lut2.data(), status,
                                          side, nullptr);
    }
    return slot_fill_batch(&L->pool, n, L->fill_dest.data(), L->fill_src.data(), L->fill_bytes.data(), side,
                           nullptr);
}

}  // namespace

extern "C" {

size_t pqe_layer_scratch_bytes(const pqe_layer_config *cfg) {
    if (!config_ok(cfg)) return 0;
    return scratch_map(*cfg).total;
}

pqe_layer *pqe_layer_create(const pqe_layer_config *cfg, const pqe_pool *pool, const void *const *host_pages,
                            const size_t *host_page_bytes, const uint8_t *luts_dev, const uint8_t *expert_fmt_dev,
                            void *scratch_dev, size_t scratch_bytes) {
    if (!config_ok(cfg) || !pool || !host_pages || !host_page_bytes || !scratch_dev) return nullptr;
    if ((cfg->S > 0 && !pool->base) || (cfg->W > 0 && !pool->wb_base)) return nullptr;
    if (pool->H != cfg->H || pool->I != cfg->I || pool->n_slots != cfg->S || pool->n_wb != cfg->W) return nullptr;
    if (pool->slot_stride != pqe_slot_stride(cfg->H, cfg->I)) return nullptr;
    if (cfg->compressed && !luts_dev) return nullptr;
    if (reinterpret_cast<uintptr_t>(scratch_dev) % 256) return nullptr;
    ScratchMap m = scratch_map(*cfg);
    if (scratch_bytes < m.total) return nullptr;
    for (int e = 0; e < cfg->E; ++e) {
        if (!host_pages[e] || host_page_bytes[e] == 0) return nullptr;
        if (!cfg->compressed && (reinterpret_cast<uintptr_t>(host_pages[e]) % 16 || host_page_bytes[e] % 16))
            return nullptr;
        if (!cfg->compressed && host_page_bytes[e] > pool->slot_stride) return nullptr;
        if (cfg->compressed && (host_page_bytes[e] > m.staging_bytes ||
                                reinterpret_cast<uintptr_t>(host_pages[e]) % 16))
            return nullptr;
    }
    pqe_layer *L = new (std::nothrow) pqe_layer();
    if (!L) return nullptr;
    L->cfg = *cfg;
    L->pool = *pool;
    L->host_pages.assign(host_pages, host_pages + cfg->E);
    L->host_bytes.assign(host_page_bytes, host_page_bytes + cfg->E);
    L->fill_src.assign(cfg->E, nullptr);
    L->fill_bytes.assign(cfg->E, 0);
    L->fill_lut13.assign(cfg->E, nullptr);
    L->fill_lut2.assign(cfg->E, nullptr);
    L->fill_dest.assign(cfg->E, 0);
    L->fill_expert.assign(cfg->E, 0);
    L->luts = luts_dev;
    L->expert_fmt = expert_fmt_dev;
    L->scratch = static_cast<uint8_t *>(scratch_dev);
    L->map = m;
    L->lru = pqe_lru_create(cfg->E, cfg->S);
    cudaError_t e1 = cudaHostAlloc(reinterpret_cast<void **>(&L->pinned), sizeof(int32_t) * 4 * cfg->E,
                                   cudaHostAllocDefault);
    cudaError_t e2 = cudaEventCreateWithFlags(&L->ev_counts, cudaEventDisableTiming);
    cudaError_t e3 = cudaEventCreateWithFlags(&L->ev_fill, cudaEventDisableTiming);
    if (e3 == cudaSuccess && cfg->overlap_groups > 0) {
        e3 = cudaEventCreateWithFlags(&L->ev_lru, cudaEventDisableTiming);
        for (int g = 0; g < cfg->overlap_groups && e3 == cudaSuccess; ++g)
            e3 = cudaEventCreateWithFlags(&L->ev_group[g], cudaEventDisableTiming);
    }
    if (!L->lru || e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess) {
        pqe::set_last_cuda_error(e1 != cudaSuccess ? e1 : (e2 != cudaSuccess ? e2 : e3));
        pqe_layer_destroy(L);
        return nullptr;
    }
    if (cudaMemset(L->at<int32_t>(m.status), 0, sizeof(int32_t)) != cudaSuccess) {
        pqe_layer_destroy(L);
        return nullptr;
    }
    if (cfg->device_pager) {
        std::vector<uint64_t> ptrs(cfg->E);
        for (int e = 0; e < cfg->E; ++e) ptrs[e] = reinterpret_cast<uint64_t>(host_pages[e]);
        if (cudaMemcpy(L->at<void>(m.host_pages), ptrs.data(), sizeof(uint64_t) * cfg->E, cudaMemcpyHostToDevice) !=
                cudaSuccess ||
            cudaMemcpy(L->at<void>(m.page_bytes), host_page_bytes, sizeof(size_t) * cfg->E,
                       cudaMemcpyHostToDevice) != cudaSuccess ||
            pqe_lru_device_init(L->at<void>(m.lru), cfg->E, cfg->S, nullptr) != PQE_OK ||
            cudaDeviceSynchronize() != cudaSuccess) {
            pqe_layer_destroy(L);
            return nullptr;
        }
    }
    return L;
}

void pqe_layer_destroy(pqe_layer *L) {
    if (!L) return;
    if (L->ev_counts) cudaEventDestroy(L->ev_counts);
    if (L->ev_fill) cudaEventDestroy(L->ev_fill);
    if (L->ev_lru) cudaEventDestroy(L->ev_lru);
    for (cudaEvent_t e : L->ev_group)
        if (e) cudaEventDestroy(e);
    if (L->pinned) cudaFreeHost(L->pinned);
    for (auto &g : L->graphs)
        if (g.exec) cudaGraphExecDestroy(g.exec);
    pqe_lru_destroy(L->lru);
    delete L;
}

int pqe_layer_attach_ram_tier(pqe_layer *L, pqe_ram_tier *t) {
    if (!L) return PQE_ERR_INVALID_ARG;
    if (!t) {
        L->ram = nullptr;
        return PQE_OK;
    }
    if (L->cfg.device_pager) return PQE_ERR_UNSUPPORTED;
    const int E = L->cfg.E;
    std::vector<size_t> b(E);
    for (int e = 0; e < E; ++e) {
        b[e] = pqe_ram_tier_page_bytes(t, e);
        if (b[e] == 0) return PQE_ERR_INVALID_ARG;  // the tier has fewer experts than the layer
        if (!L->cfg.compressed && (b[e] > L->pool.slot_stride || b[e] % 16)) return PQE_ERR_INVALID_ARG;
        if (L->cfg.compressed && b[e] > L->map.staging_bytes) return PQE_ERR_INVALID_ARG;
    }
    if (pqe_ram_tier_page_bytes(t, E) != 0) return PQE_ERR_INVALID_ARG;  // more experts than the layer
    L->ram_bytes = std::move(b);
    L->ram_need.assign(E, 0);
    L->ram_queued.assign(E, 0);
    L->ram_page.assign(E, nullptr);
    L->ram = t;
    return PQE_OK;
}

int pqe_layer_set_host_page(pqe_layer *L, int expert, const void *pinned_page, size_t bytes) {
    if (!L || expert < 0 || expert >= L->cfg.E || !pinned_page || bytes == 0) return PQE_ERR_INVALID_ARG;
    if (!L->cfg.compressed && (bytes > L->pool.slot_stride || bytes % 16 ||
                               reinterpret_cast<uintptr_t>(pinned_page) % 16))
        return PQE_ERR_INVALID_ARG;
    if (L->cfg.compressed && (bytes > L->map.staging_bytes || reinterpret_cast<uintptr_t>(pinned_page) % 16))
        return PQE_ERR_INVALID_ARG;
    L->host_pages[expert] = pinned_page;
    L->host_bytes[expert] = bytes;
    if (L->cfg.device_pager) {
        const uint64_t ptr = reinterpret_cast<uint64_t>(pinned_page);
        cudaError_t ce = cudaMemcpy(L->at<uint64_t>(L->map.host_pages) + expert, &ptr, sizeof(ptr),
                                    cudaMemcpyHostToDevice);
        if (ce == cudaSuccess)
            ce = cudaMemcpy(L->at<size_t>(L->map.page_bytes) + expert, &bytes, sizeof(bytes), cudaMemcpyHostToDevice);
        if (ce != cudaSuccess) {
            pqe::set_last_cuda_error(ce);
            return PQE_ERR_CUDA;
        }
        int rc = pqe_lru_device_invalidate(L->at<void>(L->map.lru), L->cfg.E, L->cfg.S, expert, nullptr);
        if (rc) return rc;
        ce = cudaDeviceSynchronize();
        if (ce != cudaSuccess) {
            pqe::set_last_cuda_error(ce);
            return PQE_ERR_CUDA;
        }
    }
    return pqe_lru_invalidate(L->lru, expert);
}

int pqe_layer_device_stats(pqe_layer *L, int64_t *stats, int32_t *slot_expert, int64_t *last_use, int64_t *step,
                           void *stream) {
    if (!L || !L->cfg.device_pager) return PQE_ERR_INVALID_ARG;
    return pqe_lru_device_state(L->at<void>(L->map.lru), L->cfg.E, L->cfg.S, slot_expert, last_use, step, stats,
                                stream);
}

int pqe_layer_buffers(pqe_layer *L, pqe_layer_buffers_t *out) {
    if (!L || !out) return PQE_ERR_INVALID_ARG;
    out->status = L->at<int32_t>(L->map.status);
    out->topk_ids = L->at<int32_t>(L->map.topk_ids);
    out->topk_w = L->at<float>(L->map.topk_w);
    out->counts = L->at<int32_t>(L->map.counts);
    out->offsets = L->at<int32_t>(L->map.offsets);
    out->perm_src = L->at<int32_t>(L->map.perm_src);
    out->inv = L->at<int32_t>(L->map.inv);
    out->page_table = L->at<int32_t>(L->map.page_table);
    out->out_perm = L->at<void>(L->map.out_perm);
    out->x_in = L->at<void>(L->map.x_in);
    out->logits_in = L->at<float>(L->map.logits_in);
    out->y_out = L->at<void>(L->map.y_out);
    return PQE_OK;
}

int pqe_layer_set_step_graphs(pqe_layer *L, int enable) {
    if (!L) return PQE_ERR_INVALID_ARG;
    L->step_graphs = enable != 0;
    return PQE_OK;
}

int pqe_layer_set_ffn_events(pqe_layer *L, void *ev_begin, void *ev_end) {
    if (!L || (!ev_begin) != (!ev_end)) return PQE_ERR_INVALID_ARG;
    L->ev_ffn_begin = reinterpret_cast<cudaEvent_t>(ev_begin);
    L->ev_ffn_end = reinterpret_cast<cudaEvent_t>(ev_end);
    return PQE_OK;
}

int pqe_layer_lru_state(const pqe_layer *L, int32_t *slot_expert, int64_t *last_use, int64_t *step) {
    if (!L) return PQE_ERR_INVALID_ARG;
    return pqe_lru_state(L->lru, slot_expert, last_use, step);
}

int pqe_layer_step(pqe_layer *L, const void *x_dev, const float *w_router_dev, float *logits_dev, int T, void *y_dev,
                   void *stream, void *side_stream, pqe_step_info *info) {
    if (!L || T < 0 || T > L->cfg.max_T || !y_dev || !x_dev || (!w_router_dev && !logits_dev))
        return PQE_ERR_INVALID_ARG;
    const pqe_layer_config &c = L->cfg;
    const ScratchMap &m = L->map;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaStream_t side = side_stream ? reinterpret_cast<cudaStream_t>(side_stream) : s;
    pqe_step_info local{};
    if (T == 0) {
        if (info) *info = local;
        return PQE_OK;
    }
    int32_t *status = L->at<int32_t>(m.status);
    int32_t *ids = L->at<int32_t>(m.topk_ids);
    float *gates = L->at<float>(m.topk_w);
    int32_t *counts = L->at<int32_t>(m.counts);
    int32_t *offsets = L->at<int32_t>(m.offsets);
    int32_t *perm_src = L->at<int32_t>(m.perm_src);
    int32_t *inv = L->at<int32_t>(m.inv);
    int32_t *page_table = L->at<int32_t>(m.page_table);
    void *out_perm = L->at<void>(m.out_perm);
    int rc = moe_route(x_dev, w_router_dev, logits_dev, T, c.H, c.E, c.k, ids, gates, stream);
    if (rc) return rc;
    rc = moe_permute(ids, T, c.k, c.E, counts, offsets, perm_src, inv, L->at<void>(m.perm_ws), m.perm_ws_bytes,
                     status, stream);
    if (rc) return rc;
    if (c.device_pager) {
        // page table, misses and refills stay on the device: nothing blocks the host
        int32_t *miss = L->at<int32_t>(m.miss);
        const size_t *pbytes = L->at<size_t>(m.page_bytes);
        rc = page_table_update_device(L->at<void>(m.lru), c.E, c.S, counts, pbytes, page_table, miss, stream);
        if (rc) return rc;
        const int G = c.overlap_groups;
        if (G > 0 && side != s && !L->ev_ffn_begin) {
            // refills in G groups on the side stream, each by a refill kernel on a few
            // SMs; the FFN in passes on s: the resident experts first, beside the
            // refills, then each group's experts once its pages have landed
            const uint64_t *hp = L->at<uint64_t>(m.host_pages);
            int dev = 0, sms = 0;
            if ((rc = pqe::device_info(dev, sms))) return rc;
            // SMs left to the refills beside the FFN passes: plain pages need 32 CTAs
            // at the host link's rate, compressed ones are decoded by 4 CTAs on each
            // SM the passes leave
            const int reserve = std::max(OVERLAP_FILL_CTAS, sms - OVERLAP_FFN_SMS);
            cudaError_t ce = cudaEventRecord(L->ev_lru, s);
            if (ce == cudaSuccess) ce = cudaStreamWaitEvent(side, L->ev_lru, 0);
            for (int g = 0; g < G && ce == cudaSuccess; ++g) {
                // compressed pages: pulled and decoded by 4 decode CTAs on each SM left to the refill
                if ((rc = c.compressed ? pqe::slot_fill_compressed_device_group(&L->pool, miss, c.E, hp, pbytes,
                                                                                L->luts, g, G, 4 * reserve, status,
                                                                                side)
                                       : pqe::slot_fill_device_group(&L->pool, miss, c.E, hp, pbytes, g, G,
                                                                     OVERLAP_FILL_CTAS, side)))
                    return rc;
                ce = cudaEventRecord(L->ev_group[g], side);
            }
            if (ce != cudaSuccess) {
                pqe::set_last_cuda_error(ce);
                return PQE_ERR_CUDA;
            }
            void *ws = L->at<void>(m.ffn_ws);
            for (int p = 0; p <= G; ++p) {
                if (p > 0 && (ce = cudaStreamWaitEvent(s, L->ev_group[p - 1], 0)) != cudaSuccess) {
                    pqe::set_last_cuda_error(ce);
                    return PQE_ERR_CUDA;
                }
                rc = pqe::moe_paged_ffn_pass(x_dev, perm_src, offsets, page_table, L->expert_fmt, &L->pool, T, c.k,
                                             c.E, out_perm, ws, m.ffn_ws_bytes, status, s, miss, G, p,
                                             p < G ? reserve : 0);
                if (rc) return rc;
            }
            rc = moe_combine(out_perm, inv, gates, T, c.k, c.H, y_dev, stream);
            if (rc) return rc;
            if (info) *info = local;
            return PQE_OK;
        }
        rc = c.compressed ? pqe::slot_fill_compressed_device_group(&L->pool, miss, c.E, L->at<uint64_t>(m.host_pages),
                                                                   pbytes, L->luts, 0, 1, 0, status, s)
                          : slot_fill_device(&L->pool, miss, c.E, L->at<uint64_t>(m.host_pages), pbytes, stream);
        if (rc) return rc;
        if (L->ev_ffn_begin && (rc = (record_timing(L->ev_ffn_begin, s) == cudaSuccess ? 0 : PQE_ERR_CUDA))) return rc;
        rc = moe_paged_ffn(x_dev, perm_src, offsets, page_table, L->expert_fmt, &L->pool, T, c.k, c.E, out_perm,
                           L->at<void>(m.ffn_ws), m.ffn_ws_bytes, status, stream);
        if (rc) return rc;
        if (L->ev_ffn_end && (rc = (record_timing(L->ev_ffn_end, s) == cudaSuccess ? 0 : PQE_ERR_CUDA))) return rc;
        rc = moe_combine(out_perm, inv, gates, T, c.k, c.H, y_dev, stream);
        if (rc) return rc;
        if (info) *info = local;
        return PQE_OK;
    }
    int32_t *counts_h = L->pinned, *pt_h = L->pinned + c.E, *miss_e = L->pinned + 2 * c.E,
            *miss_d = L->pinned + 3 * c.E;
    cudaError_t ce = cudaMemcpyAsync(counts_h, counts, sizeof(int32_t) * c.E, cudaMemcpyDeviceToHost, s);
    if (ce == cudaSuccess) ce = cudaEventRecord(L->ev_counts, s);
    if (ce == cudaSuccess) ce = cudaEventSynchronize(L->ev_counts);
    if (ce != cudaSuccess) {
        pqe::set_last_cuda_error(ce);
        return PQE_ERR_CUDA;
    }
    int32_t nm = 0, wb = 0;
    rc = page_table_update(L->lru, counts_h, pt_h, miss_e, miss_d, &nm, &wb);
    if (rc) return rc;
    for (int e = 0; e < c.E; ++e) local.n_routed += counts_h[e] > 0;
    local.n_miss = nm;
    local.working_buffer = wb;
    for (int i = 0; i < nm; ++i)
        if (miss_d[i] >= L->pool.n_slots + L->pool.n_wb) return PQE_ERR_CAPACITY;
    if (L->ram && nm > 0) {
        // RAM tier: the misses whose pages are in RAM are refilled at once, the
        // others after the paging-file reads have landed
        std::fill(L->ram_need.begin(), L->ram_need.end(), 0);
        for (int i = 0; i < nm; ++i) L->ram_need[miss_e[i]] = 1;
        int32_t nr = 0, rwb = 0;
        rc = pqe_ram_tier_request(L->ram, L->ram_need.data(), L->ram_page.data(), L->ram_queued.data(), &nr, &rwb);
        if (rc) return rc;
        local.n_file_read = nr;
        for (int pass = 0; pass < 2; ++pass) {
            if (pass == 1 && nr > 0 && (rc = pqe_ram_tier_wait(L->ram))) return rc;
            int n = 0;
            for (int i = 0; i < nm; ++i) {
                const int e = miss_e[i];
                if (L->ram_queued[e] != pass) continue;
                L->fill_expert[n] = e;
                L->fill_dest[n] = miss_d[i];
                L->fill_src[n] = L->ram_page[e];
                L->fill_bytes[n] = L->ram_bytes[e];
                ++n;
            }
            if ((rc = refill(L, n, side, status))) return rc;
        }
        for (int i = 0; i < nm; ++i) local.h2d_bytes += (int64_t)L->ram_bytes[miss_e[i]];
    } else if (nm > 0) {
        for (int i = 0; i < nm; ++i) {
            const int e = miss_e[i];
            L->fill_expert[i] = e;
            L->fill_dest[i] = miss_d[i];
            L->fill_src[i] = L->host_pages[e];
            L->fill_bytes[i] = L->host_bytes[e];
            local.h2d_bytes += (int64_t)L->host_bytes[e];
        }
        if ((rc = refill(L, nm, side, status))) return rc;
    }
    if (nm > 0 && side != s) {
        ce = cudaEventRecord(L->ev_fill, side);
        if (ce == cudaSuccess) ce = cudaStreamWaitEvent(s, L->ev_fill, 0);
        if (ce != cudaSuccess) {
            pqe::set_last_cuda_error(ce);
            return PQE_ERR_CUDA;
        }
    }
    ce = cudaMemcpyAsync(page_table, pt_h, sizeof(int32_t) * c.E, cudaMemcpyHostToDevice, s);
    if (ce != cudaSuccess) {
        pqe::set_last_cuda_error(ce);
        return PQE_ERR_CUDA;
    }
    if (L->ev_ffn_begin && (ce = record_timing(L->ev_ffn_begin, s)) != cudaSuccess) {
        pqe::set_last_cuda_error(ce);
        return PQE_ERR_CUDA;
    }
    rc = moe_paged_ffn(x_dev, perm_src, offsets, page_table, L->expert_fmt, &L->pool, T, c.k, c.E, out_perm,
                       L->at<void>(m.ffn_ws), m.ffn_ws_bytes, status, stream);
    if (rc) return rc;
    if (L->ev_ffn_end && (ce = record_timing(L->ev_ffn_end, s)) != cudaSuccess) {
        pqe::set_last_cuda_error(ce);
        return PQE_ERR_CUDA;
    }
    rc = moe_combine(out_perm, inv, gates, T, c.k, c.H, y_dev, stream);
    if (rc) return rc;
    if (info) *info = local;
    return PQE_OK;
}

}  // extern "C"

namespace {

// The launches of one pqe_layer_step for pqe_layer_step_host. A device-pager
// step decides nothing on the host, so its launches for a given step size,
// router mode and stream pair are the same every time: they are captured into
// a CUDA graph on the second call of that shape and replayed from then on.
// Timing events, the legacy default streams (which cannot be captured) and a
// changed launch setting (wait limit, test hooks) fall back to the eager step
// or to a new capture.
constexpr size_t MAX_STEP_GRAPHS = 16;

int step_host_launches(pqe_layer *L, const void *x_in, const float *w_router, float *lg, int T, void *y,
                       cudaStream_t s, void *side_stream, pqe_step_info *info) {
    const bool overlap = side_stream && reinterpret_cast<cudaStream_t>(side_stream) != s;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const bool graphable = L->cfg.device_pager && L->step_graphs && !L->ev_ffn_begin && T > 0 && s &&
                           s != cudaStreamLegacy && s != cudaStreamPerThread &&
                           cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone;
    if (!graphable) return pqe_layer_step(L, x_in, w_router, lg, T, y, s, side_stream, info);
    const uint64_t gen = pqe::launch_settings_generation();
    pqe_layer::StepGraph *g = nullptr;
    for (auto &e : L->graphs)
        if (e.T == T && e.w_router == w_router && e.overlap == overlap) g = &e;
    if (g && g->gen != gen) {  // captured under other settings: start again
        if (g->exec) cudaGraphExecDestroy(g->exec);
        *g = pqe_layer::StepGraph{T, w_router, overlap, gen, 0, nullptr};
        return pqe_layer_step(L, x_in, w_router, lg, T, y, s, side_stream, info);
    }
    if (!g) {
        if (L->graphs.size() >= MAX_STEP_GRAPHS) {
            if (L->graphs.front().exec) cudaGraphExecDestroy(L->graphs.front().exec);
            L->graphs.erase(L->graphs.begin());
        }
        L->graphs.push_back(pqe_layer::StepGraph{T, w_router, overlap, gen, 0, nullptr});
        return pqe_layer_step(L, x_in, w_router, lg, T, y, s, side_stream, info);
    }
    if (g->state < 0) return pqe_layer_step(L, x_in, w_router, lg, T, y, s, side_stream, info);
    if (g->state == 0) {
        cudaError_t ce = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
        if (ce != cudaSuccess) {
            pqe::set_last_cuda_error(ce);
            return PQE_ERR_CUDA;
        }
        const int rc = pqe_layer_step(L, x_in, w_router, lg, T, y, s, side_stream, nullptr);
        cudaGraph_t graph = nullptr;
        ce = cudaStreamEndCapture(s, &graph);
        cudaGraphExec_t exec = nullptr;
        if (rc == PQE_OK && ce == cudaSuccess) ce = cudaGraphInstantiate(&exec, graph, 0);
        if (graph) cudaGraphDestroy(graph);
        if (rc != PQE_OK) {
            (void)cudaGetLastError();
            return rc;
        }
        if (ce != cudaSuccess) {  // not capturable here: this shape steps eagerly from now on
            (void)cudaGetLastError();
            g->state = -1;
            return pqe_layer_step(L, x_in, w_router, lg, T, y, s, side_stream, info);
        }
        g->exec = exec;
        g->state = 1;
    }
    const cudaError_t ce = cudaGraphLaunch(g->exec, s);
    if (ce != cudaSuccess) {
        pqe::set_last_cuda_error(ce);
        return PQE_ERR_CUDA;
    }
    if (info) *info = pqe_step_info{};
    return PQE_OK;
}

}  // namespace

extern "C" {

int pqe_layer_step_host(pqe_layer *L, const void *x_host, const float *w_router_dev, const float *logits_host, int T,
                        void *y_host, void *stream, void *side_stream, pqe_step_info *info) {
    if (!L || T < 0 || T > L->cfg.max_T || !x_host || !y_host || (!w_router_dev && !logits_host))
        return PQE_ERR_INVALID_ARG;
    const pqe_layer_config &c = L->cfg;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void *x_in = L->at<void>(L->map.x_in);
    float *lg = L->at<float>(L->map.logits_in);
    void *y = L->at<void>(L->map.y_out);
    cudaError_t ce = cudaMemcpyAsync(x_in, x_host, sizeof(uint16_t) * (size_t)T * c.H, cudaMemcpyHostToDevice, s);
    if (ce == cudaSuccess && !w_router_dev)
        ce = cudaMemcpyAsync(lg, logits_host, sizeof(float) * (size_t)T * c.E, cudaMemcpyHostToDevice, s);
    if (ce != cudaSuccess) {
        pqe::set_last_cuda_error(ce);
        return PQE_ERR_CUDA;
    }
    int rc = step_host_launches(L, x_in, w_router_dev, w_router_dev ? nullptr : lg, T, y, s, side_stream, info);
    if (rc) return rc;
    ce = cudaMemcpyAsync(y_host, y, sizeof(uint16_t) * (size_t)T * c.H, cudaMemcpyDeviceToHost, s);
    if (ce == cudaSuccess) ce = cudaStreamSynchronize(s);
    if (ce != cudaSuccess) {
        pqe::set_last_cuda_error(ce);
        return PQE_ERR_CUDA;
    }
    return PQE_OK;
}

}  // extern "C"
