// pager.cpp -- host side of the paged expert pool: per-layer LRU page table,
// slot refills from the host tier, per-expert bit-width ranking, error text.
//
// Per-layer slot pools with LRU, copy-in on a miss, and the working buffer
// for a step that needs more experts than slots: expert-pager article
// (rand.pepabo.com), "エキスパート重みの階層ページング". Refills overlap compute:
// MoE-Gen summary (aibr.jp), "3.中核となる技術的要素". Bit-width from
// importance: PagedWeight commentary (spectral-agent.com), "技術的に面白い点".
#include <cmath>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "pqe.h"
#include "pqe_common.cuh"

namespace pqe {

static thread_local cudaError_t g_last_cuda = cudaSuccess;
static std::atomic<uint64_t> g_launches{0};

void set_last_cuda_error(cudaError_t e) { g_last_cuda = e; }

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// polls of a bounded device wait before it gives up, and the test bias of the
// weight stream's phase-2 target (both read at each launch)
static std::atomic<uint32_t> g_wait_limit{DEFAULT_WAIT_LIMIT};
static std::atomic<uint32_t> g_phase2_bias{0};
static std::atomic<int> g_stream_kernel{0};
// bumped by every setter above: a captured launch keeps the values it read,
// so a cached graph of a layer step is rebuilt when this changes
static std::atomic<uint64_t> g_launch_gen{0};

uint64_t launch_settings_generation() { return g_launch_gen.load(std::memory_order_relaxed); }
uint32_t wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }
uint32_t phase2_bias() { return g_phase2_bias.load(std::memory_order_relaxed); }
int stream_kernel_choice() { return g_stream_kernel.load(std::memory_order_relaxed); }

}  // namespace pqe

struct pqe_lru {
    int E = 0, S = 0;
    int64_t step = 0;
    std::vector<int32_t> slot_expert;  // [S], -1 empty
    std::vector<int64_t> last_use;     // [S]
    std::vector<int32_t> expert_slot;  // [E], -1 not resident
    std::vector<uint8_t> needed;       // [E] scratch: member of U this step
};

extern "C" {

const char *pqe_strerror(int code) {
    switch (code) {
    case PQE_OK: return "ok";
    case PQE_ERR_INVALID_ARG: return "invalid argument";
    case PQE_ERR_CUDA: return "CUDA runtime error";
    case PQE_ERR_CAPACITY: return "capacity exceeded";
    case PQE_ERR_CORRUPT: return "corrupt compressed page";
    case PQE_ERR_TIMEOUT: return "timed out";
    case PQE_ERR_UNSUPPORTED: return "unsupported";
    case PQE_ERR_IO: return "paging file I/O error";
    default: return "unknown error";
    }
}

int pqe_abi_version(void) { return 1; }

int pqe_set_wait_limit(uint32_t polls) {
    pqe::g_wait_limit.store(polls ? polls : pqe::DEFAULT_WAIT_LIMIT, std::memory_order_relaxed);
    pqe::g_launch_gen.fetch_add(1, std::memory_order_relaxed);
    return PQE_OK;
}

int pqe_test_set_phase2_bias(uint32_t bias) {
    pqe::g_phase2_bias.store(bias, std::memory_order_relaxed);
    pqe::g_launch_gen.fetch_add(1, std::memory_order_relaxed);
    return PQE_OK;
}

int pqe_test_set_stream_kernel(int kind) {
    if (kind < 0 || kind > 2) return PQE_ERR_INVALID_ARG;
    pqe::g_stream_kernel.store(kind, std::memory_order_relaxed);
    pqe::g_launch_gen.fetch_add(1, std::memory_order_relaxed);
    return PQE_OK;
}

int pqe_last_cuda_error(void) { return (int)pqe::g_last_cuda; }

uint64_t pqe_kernel_launches(void) { return pqe::g_launches.load(std::memory_order_relaxed); }

size_t pqe_page_bytes(int fmt, int H, int I) {
    if (H < 64 || I < 64 || H % 64 || I % 64) return 0;
    const size_t ih = (size_t)I * H;
    if (fmt == PQE_FMT_FP8) return 3 * ih + 4 * (2 * (size_t)I + H);
    if (fmt == PQE_FMT_MXFP4) return 3 * ih / 2 + 3 * ih / 32;
    return 0;
}

size_t pqe_slot_stride(int H, int I) {
    const size_t b = pqe_page_bytes(PQE_FMT_FP8, H, I);
    return b ? (b + 4095) / 4096 * 4096 : 0;
}

pqe_lru *pqe_lru_create(int E, int S) {
    if (E < 1 || S < 0 || E > (1 << 20) || S > (1 << 20)) return nullptr;
    pqe_lru *st = new (std::nothrow) pqe_lru();
    if (!st) return nullptr;
    st->E = E;
    st->S = S;
    st->slot_expert.assign(S, -1);
    st->last_use.assign(S, -1);
    st->expert_slot.assign(E, -1);
    st->needed.assign(E, 0);
    return st;
}

void pqe_lru_destroy(pqe_lru *st) { delete st; }

int pqe_lru_state(const pqe_lru *st, int32_t *slot_expert, int64_t *last_use, int64_t *step) {
    if (!st) return PQE_ERR_INVALID_ARG;
    if (slot_expert) std::copy(st->slot_expert.begin(), st->slot_expert.end(), slot_expert);
    if (last_use) std::copy(st->last_use.begin(), st->last_use.end(), last_use);
    if (step) *step = st->step;
    return PQE_OK;
}

int pqe_lru_invalidate(pqe_lru *st, int expert) {
    if (!st || expert < 0 || expert >= st->E) return PQE_ERR_INVALID_ARG;
    const int s = st->expert_slot[expert];
    if (s >= 0) {
        st->slot_expert[s] = -1;
        st->last_use[s] = -1;
        st->expert_slot[expert] = -1;
    }
    return PQE_OK;
}

int page_table_update(pqe_lru *st, const int32_t *counts_host, int32_t *page_table_host, int32_t *miss_expert,
                      int32_t *miss_dest, int32_t *n_miss, int32_t *working_buffer_mode) {
    if (!st || !counts_host || !page_table_host || !miss_expert || !miss_dest || !n_miss || !working_buffer_mode)
        return PQE_ERR_INVALID_ARG;
    const int E = st->E, S = st->S;
    const int64_t now = st->step;
    int n_needed = 0;
    for (int e = 0; e < E; ++e) {
        st->needed[e] = counts_host[e] > 0;
        n_needed += st->needed[e];
        page_table_host[e] = -1;
    }
    int nm = 0;
    if (n_needed > S) {
        // working-buffer step: the cache is left as it is
        int w = 0;
        for (int e = 0; e < E; ++e) {
            if (!st->needed[e]) continue;
            const int s = st->expert_slot[e];
            if (s >= 0) {
                page_table_host[e] = s;
            } else {
                page_table_host[e] = S + w;
                miss_expert[nm] = e;
                miss_dest[nm] = S + w;
                ++nm;
                ++w;
            }
        }
        *working_buffer_mode = 1;
    } else {
        for (int e = 0; e < E; ++e) {
            const int s = st->expert_slot[e];
            if (st->needed[e] && s >= 0) {
                st->last_use[s] = now;
                page_table_host[e] = s;
            }
        }
        int next_empty = 0;
        for (int e = 0; e < E; ++e) {
            if (!st->needed[e] || st->expert_slot[e] >= 0) continue;
            int victim = -1;
            while (next_empty < S && st->slot_expert[next_empty] >= 0) ++next_empty;
            if (next_empty < S) {
                victim = next_empty;
            } else {
                int64_t best = 0;
                for (int s = 0; s < S; ++s) {
                    const int held = st->slot_expert[s];
                    if (st->needed[held]) continue;
                    if (victim < 0 || st->last_use[s] < best) {
                        victim = s;
                        best = st->last_use[s];
                    }
                }
            }
            if (victim < 0) return PQE_ERR_CAPACITY;  // cannot happen when n_needed <= S
            const int old = st->slot_expert[victim];
            if (old >= 0) st->expert_slot[old] = -1;
            st->slot_expert[victim] = e;
            st->expert_slot[e] = victim;
            st->last_use[victim] = now;
            page_table_host[e] = victim;
            miss_expert[nm] = e;
            miss_dest[nm] = victim;
            ++nm;
        }
        *working_buffer_mode = 0;
    }
    *n_miss = nm;
    st->step = now + 1;
    return PQE_OK;
}

void *pqe_pool_slot_addr(const pqe_pool *pool, int dest) {
    if (!pool || dest < 0 || dest >= pool->n_slots + pool->n_wb) return nullptr;
    if (dest < pool->n_slots) return pool->base ? static_cast<uint8_t *>(pool->base) + (size_t)dest * pool->slot_stride
                                                : nullptr;
    return pool->wb_base ? static_cast<uint8_t *>(pool->wb_base) + (size_t)(dest - pool->n_slots) * pool->slot_stride
                         : nullptr;
}

int slot_fill(const pqe_pool *pool, int dest, const void *pinned_src, size_t bytes, void *stream, void *done_event) {
    uint8_t *dst = static_cast<uint8_t *>(pqe_pool_slot_addr(pool, dest));
    if (!dst || !pinned_src || bytes == 0 || bytes > pool->slot_stride) return PQE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(dst, pinned_src, bytes, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && done_event) e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(done_event), s);
    if (e != cudaSuccess) {
        pqe::set_last_cuda_error(e);
        return PQE_ERR_CUDA;
    }
    return PQE_OK;
}

int pqe_rank_formats(const double *m, int E, int n_hi, uint8_t *fmt) {
    if (!m || !fmt || E < 1 || n_hi < 0) return PQE_ERR_INVALID_ARG;
    std::vector<int> order(E);
    for (int e = 0; e < E; ++e) order[e] = e;
    std::stable_sort(order.begin(), order.end(), [m](int a, int b) { return m[a] > m[b]; });
    for (int e = 0; e < E; ++e) fmt[e] = PQE_FMT_MXFP4;
    for (int r = 0; r < std::min(n_hi, E); ++r) fmt[order[r]] = PQE_FMT_FP8;
    return PQE_OK;
}

int pqe_rank_formats_quality(const double *m, const double *q, int E, int n_hi, uint8_t *fmt) {
    if (!m || !q || !fmt || E < 1 || n_hi < 0) return PQE_ERR_INVALID_ARG;
    std::vector<double> score(E);
    for (int e = 0; e < E; ++e) score[e] = m[e] * q[e];
    return pqe_rank_formats(score.data(), E, n_hi, fmt);
}

int pqe_importance_step(double *m, const int32_t *ids, const float *gates, int T, int k, int E, double alpha,
                        int64_t step, int every, int n_hi, uint8_t *fmt, int32_t *reranked) {
    if (!m || !fmt || E < 1 || T < 1 || k < 1 || every < 1 || (!ids && T) || (!gates && T))
        return PQE_ERR_INVALID_ARG;
    std::vector<double> mass(E, 0.0);
    for (long f = 0; f < (long)T * k; ++f) {
        const int e = ids[f];
        if (e < 0 || e >= E) return PQE_ERR_INVALID_ARG;
        mass[e] += (double)gates[f];
    }
    // three separately rounded operations (the library is built without contraction)
    for (int e = 0; e < E; ++e) m[e] = alpha * m[e] + (1.0 - alpha) * (mass[e] / (double)T);
    const bool rr = (step + 1) % every == 0;
    if (reranked) *reranked = rr ? 1 : 0;
    if (rr) return pqe_rank_formats(m, E, n_hi, fmt);
    return PQE_OK;
}

int64_t pqe_module_batch_size(int E, int k, int H, int I, double hbm_gbs, double fp8_tflops, int granule) {
    if (E < 1 || k < 1 || k > E || pqe_page_bytes(PQE_FMT_FP8, H, I) == 0 || !(hbm_gbs > 0.0) ||
        !(fp8_tflops > 0.0) || granule < 1)
        return 0;
    // per expert with n rows: 6 n H I FLOP against its FP8 page plus
    // 2 H (1 + 1/k) bytes of activations per row (the token's bf16 x, read once
    // for its k rows, and the row's bf16 out_perm)
    const double P = fp8_tflops * 1e12, BW = hbm_gbs * 1e9;
    const double page = (double)pqe_page_bytes(PQE_FMT_FP8, H, I);
    const double den = 6.0 * H * I * BW - P * 2.0 * H * (1.0 + 1.0 / k);
    if (!(den > 0.0)) return 0;  // the activations alone outrun the tensor cores: no knee
    const double n_star = P * page / den;
    const double t_star = std::ceil(n_star * E / k);
    const int64_t g = granule;
    return ((int64_t)t_star + g - 1) / g * g;
}

}  // extern "C"
