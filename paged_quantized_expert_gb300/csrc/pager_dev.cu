// pager_dev.cu -- the per-layer LRU slot pool kept on the GPU, and refills
// driven by a miss list that never leaves the device.
//
// Same rules as the host pager (expert-pager article, rand.pepabo.com,
// "エキスパート重みの階層ページング": per-layer slots, LRU, copy-in of a missing
// expert, a working buffer when a step needs more experts than slots), so the
// two produce bit-identical page tables and slot states. Keeping the state on
// the device removes the one host round trip of a step: routing counts, the
// page table, the miss list and the refill stay on the GPU, and a whole layer
// step can be replayed from a CUDA graph.
//
// Step on one CTA of 1024 threads (E <= 1024, S <= 1024):
//   U = {e : counts[e] > 0};
//   |U| > S: working-buffer step, state untouched, non-resident e in U get
//            S + (rank among them by id);
//   else:    hits refresh last_use; candidate slots are ordered empty-first by
//            index, then by (last_use, index) among slots whose expert is not
//            in U; the i-th miss (ascending id) takes the i-th candidate --
//            the order in which the host assigns victims one at a time.
#include "pqe_common.cuh"

namespace pqe {

struct DevLru {
    int64_t step;
    int64_t stats[4];  // routed experts, misses, working-buffer steps, refill bytes (running totals)
};

// device state layout: DevLru | slot_expert [S] int32 | last_use [S] int64 | expert_slot [E] int32
struct LruView {
    DevLru *hdr;
    int32_t *slot_expert;
    int64_t *last_use;
    int32_t *expert_slot;
};

__host__ __device__ inline size_t lru_bytes(int E, int S) {
    return round_up(sizeof(DevLru), 16) + round_up(4 * (size_t)S, 16) + round_up(8 * (size_t)S, 16) +
           round_up(4 * (size_t)E, 16);
}

__host__ __device__ inline LruView lru_view(void *p, int E, int S) {
    uint8_t *b = static_cast<uint8_t *>(p);
    LruView v;
    v.hdr = reinterpret_cast<DevLru *>(b);
    b += round_up(sizeof(DevLru), 16);
    v.slot_expert = reinterpret_cast<int32_t *>(b);
    b += round_up(4 * (size_t)S, 16);
    v.last_use = reinterpret_cast<int64_t *>(b);
    b += round_up(8 * (size_t)S, 16);
    v.expert_slot = reinterpret_cast<int32_t *>(b);
    (void)E;
    return v;
}

__global__ void lru_init_kernel(void *state, int E, int S) {
    LruView v = lru_view(state, E, S);
    for (int i = threadIdx.x; i < S; i += blockDim.x) {
        v.slot_expert[i] = -1;
        v.last_use[i] = -1;
    }
    for (int i = threadIdx.x; i < E; i += blockDim.x) v.expert_slot[i] = -1;
    if (threadIdx.x == 0) {
        v.hdr->step = 0;
        for (int j = 0; j < 4; ++j) v.hdr->stats[j] = 0;
    }
}

__global__ void lru_invalidate_kernel(void *state, int E, int S, int e) {
    LruView v = lru_view(state, E, S);
    const int s = v.expert_slot[e];
    if (s >= 0) {
        v.slot_expert[s] = -1;
        v.last_use[s] = -1;
        v.expert_slot[e] = -1;
    }
}

// block-wide exclusive scans of three ints per thread at once (any multiple of
// 32 threads up to 1024): one pair of barriers for all three
__device__ __forceinline__ int3 scan3(int3 x, int (*wtot)[33], int3 &total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int3 incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, incl.x, o), b = __shfl_up_sync(0xffffffffu, incl.y, o),
                  c = __shfl_up_sync(0xffffffffu, incl.z, o);
        if (lane >= o) incl = make_int3(incl.x + a, incl.y + b, incl.z + c);
    }
    if (lane == 31) {
        wtot[0][w] = incl.x;
        wtot[1][w] = incl.y;
        wtot[2][w] = incl.z;
    }
    __syncthreads();
    for (int q = w; q < 3; q += nw) {  // the warp totals of component q, scanned by warp q mod nw
        const int c = lane < nw ? wtot[q][lane] : 0;
        int ci = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, ci, o);
            if (lane >= o) ci += n;
        }
        wtot[q][lane] = ci - c;
        if (lane == 31) wtot[q][32] = ci;
    }
    __syncthreads();
    total = make_int3(wtot[0][32], wtot[1][32], wtot[2][32]);
    return make_int3(wtot[0][w] + incl.x - x.x, wtot[1][w] + incl.y - x.y, wtot[2][w] + incl.z - x.z);
}

constexpr uint32_t DF_SEG = 8192;  // bytes a warp of the refill kernel moves per segment

// miss list layout: [0] n_miss, [1] working-buffer flag, [2 .. 2+E) expert,
// [2+E .. 2+2E) destination, [2+2E .. 2+3E+1) first refill segment of each miss
// (prefix over the misses, n_miss + 1 entries). One CTA of max(E, S) threads
// rounded up to a warp: thread t is expert t and slot t.
__global__ void __launch_bounds__(1024) lru_step_kernel(void *state, int E, int S, const int32_t *__restrict__ counts,
                                                        const size_t *__restrict__ page_bytes,
                                                        int32_t *__restrict__ page_table, int32_t *__restrict__ miss) {
    pdl_acquire();  // launched after the previous kernel of the step: wait for its output
    __shared__ int wtot[3][33];
    __shared__ uint8_t needed[1024];
    __shared__ int cand_of_rank[1024];
    __shared__ int s_expert[1024];     // slot -> expert at the start of the step
    __shared__ int64_t s_last[1024];   // slot -> last use at the start of the step
    __shared__ uint8_t s_class[1024];  // slot -> 0 empty, 1 eviction candidate, 2 holds a needed expert
    LruView v = lru_view(state, E, S);
    const int t = threadIdx.x;
    const int64_t now = v.hdr->step;
    const bool need = t < E && counts[t] > 0;
    const int my_slot = t < E ? v.expert_slot[t] : -1;
    const bool miss_e = need && my_slot < 0;
    if (t < E) needed[t] = need ? 1 : 0;
    if (t < S) {
        s_expert[t] = v.slot_expert[t];
        s_last[t] = v.last_use[t];
    }
    // needed experts, misses, and the misses' refill segments, scanned together
    // (the barriers inside also make needed[] and the slot copies visible)
    int3 tot;
    const int3 pre = scan3(make_int3(need ? 1 : 0, miss_e ? 1 : 0,
                                     miss_e ? (int)((page_bytes[t] + DF_SEG - 1) / DF_SEG) : 0),
                           wtot, tot);
    const int nu = tot.x, n_miss = tot.y, n_seg = tot.z;
    const int mrank = pre.y, spos = pre.z;
    int32_t *miss_exp = miss + 2, *miss_dst = miss + 2 + E, *miss_seg = miss + 2 + 2 * E;
    if (miss_e) miss_seg[mrank] = spos;
    if (t == 0) miss_seg[n_miss] = n_seg;
    if (nu > S) {
        // working-buffer step: read residents in place, stage the rest
        if (t < E) page_table[t] = need ? (my_slot >= 0 ? my_slot : S + mrank) : -1;
        if (miss_e) {
            miss_exp[mrank] = t;
            miss_dst[mrank] = S + mrank;
        }
    } else {
        // order candidate slots: empty by index, then resident-not-needed by (last_use, index)
        int key_class = 2;  // 0 empty, 1 candidate, 2 not a candidate
        int64_t lu = 0;
        if (t < S) {
            const int held = s_expert[t];
            lu = s_last[t];
            key_class = held < 0 ? 0 : (needed[held] ? 2 : 1);
            s_class[t] = (uint8_t)key_class;
        }
        __syncthreads();
        int rank = 0;
        if (key_class < 2) {
#pragma unroll 4
            for (int s2 = 0; s2 < S; ++s2) {
                const int c2 = s_class[s2];
                const int64_t l2 = s_last[s2];
                const bool before = c2 < key_class || (c2 == key_class && (c2 == 0 ? s2 < t : (l2 < lu || (l2 == lu && s2 < t))));
                rank += before ? 1 : 0;
            }
            cand_of_rank[rank] = t;
        }
        __syncthreads();
        // hits refresh recency; misses take their victims
        if (need && my_slot >= 0) {
            v.last_use[my_slot] = now;
            page_table[t] = my_slot;
        } else if (t < E) {
            page_table[t] = -1;
        }
        if (miss_e) {
            const int victim = cand_of_rank[mrank];
            const int old = s_expert[victim];
            if (old >= 0) v.expert_slot[old] = -1;
            v.slot_expert[victim] = t;
            v.last_use[victim] = now;
            page_table[t] = victim;
            miss_exp[mrank] = t;
            miss_dst[mrank] = victim;
        }
        __syncthreads();
        if (miss_e) v.expert_slot[t] = cand_of_rank[mrank];
    }
    // refill bytes of this step
    long long bytes = miss_e ? (long long)page_bytes[t] : 0;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
    if ((t & 31) == 0 && bytes) atomicAdd(reinterpret_cast<unsigned long long *>(&v.hdr->stats[3]), (unsigned long long)bytes);
    if (t == 0) {
        miss[0] = n_miss;
        miss[1] = nu > S ? 1 : 0;
        v.hdr->step = now + 1;
        v.hdr->stats[0] += nu;
        v.hdr->stats[1] += n_miss;
        v.hdr->stats[2] += nu > S ? 1 : 0;
    }
}

// refill from a device miss list: warps walk 8 KiB segments of the missed
// pages (one page = ceil(bytes / 8 KiB) segments); pages are located by
// binary search over the per-miss segment prefix written by the LRU step.
// Group g of G takes the misses of rank overlap_group_start(g) .. (g + 1) - 1,
// the grouping the FFN passes of an overlapped step use.
constexpr int DF_THREADS = 512;
constexpr int DF_UNROLL = 16;
static_assert(DF_SEG == 32 * DF_UNROLL * 16, "a warp moves one segment per pass");

__global__ void __launch_bounds__(DF_THREADS) fill_device_kernel(const int32_t *__restrict__ miss, int E,
                                                                 const uint64_t *__restrict__ host_pages,
                                                                 const size_t *__restrict__ page_bytes,
                                                                 uint8_t *__restrict__ base,
                                                                 uint8_t *__restrict__ wb_base, int n_slots,
                                                                 size_t slot_stride, int group, int groups) {
    pdl_acquire();  // launched after the previous kernel of the step: wait for its output
    extern __shared__ uint32_t seg0[];  // [misses of the group + 1]
    const int n_all = miss[0];
    const int m0 = overlap_group_start(group, groups, n_all), m1 = overlap_group_start(group + 1, groups, n_all);
    const int n = m1 - m0;
    const int32_t *mexp = miss + 2 + m0, *mdst = miss + 2 + E + m0, *mseg = miss + 2 + 2 * E + m0;
    for (int i = threadIdx.x; i <= n; i += blockDim.x) seg0[i] = (uint32_t)mseg[i];
    __syncthreads();
    const uint32_t first = seg0[0], total = seg0[n];
    const int lane = threadIdx.x & 31;
    const uint32_t nwarps = gridDim.x * (DF_THREADS / 32);
    for (uint32_t seg = first + blockIdx.x * (DF_THREADS / 32) + (threadIdx.x >> 5); seg < total; seg += nwarps) {
        int lo = 0, hi = n - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (seg0[mid] <= seg) lo = mid;
            else hi = mid - 1;
        }
        const int e = mexp[lo], d = mdst[lo];
        const uint32_t n16 = (uint32_t)(page_bytes[e] / 16);
        const uint32_t b16 = (seg - seg0[lo]) * (DF_SEG / 16);
        const uint4 *src = reinterpret_cast<const uint4 *>(host_pages[e]);
        uint4 *dst = reinterpret_cast<uint4 *>(d < n_slots ? base + (size_t)d * slot_stride
                                                           : wb_base + (size_t)(d - n_slots) * slot_stride);
        uint4 v[DF_UNROLL];
#pragma unroll
        for (int u = 0; u < DF_UNROLL; ++u) {
            const uint32_t w = b16 + u * 32 + lane;
            if (w < n16) v[u] = src[w];
        }
#pragma unroll
        for (int u = 0; u < DF_UNROLL; ++u) {
            const uint32_t w = b16 + u * 32 + lane;
            if (w < n16) dst[w] = v[u];
        }
    }
}

}  // namespace pqe

using namespace pqe;

extern "C" {

size_t pqe_lru_device_bytes(int E, int S) {
    if (E < 1 || E > 1024 || S < 0 || S > 1024) return 0;
    return lru_bytes(E, S);
}

int pqe_lru_device_init(void *state, int E, int S, void *stream) {
    PQE_CHECK_ARG(state && E >= 1 && E <= 1024 && S >= 0 && S <= 1024 && aligned(state, 16));
    lru_init_kernel<<<1, 1024, 0, as_stream(stream)>>>(state, E, S);
    PQE_LAUNCH_CHECK();
    return PQE_OK;
}

int pqe_lru_device_invalidate(void *state, int E, int S, int expert, void *stream) {
    PQE_CHECK_ARG(state && E >= 1 && E <= 1024 && S >= 0 && S <= 1024 && expert >= 0 && expert < E);
    lru_invalidate_kernel<<<1, 1, 0, as_stream(stream)>>>(state, E, S, expert);
    PQE_LAUNCH_CHECK();
    return PQE_OK;
}

int pqe_lru_device_state(const void *state, int E, int S, int32_t *slot_expert, int64_t *last_use, int64_t *step,
                         int64_t *stats, void *stream) {
    PQE_CHECK_ARG(state && E >= 1 && E <= 1024 && S >= 0 && S <= 1024);
    LruView v = lru_view(const_cast<void *>(state), E, S);
    cudaStream_t s = as_stream(stream);
    DevLru hdr;
    PQE_CUDA_TRY(cudaMemcpyAsync(&hdr, v.hdr, sizeof(hdr), cudaMemcpyDeviceToHost, s));
    if (slot_expert && S) PQE_CUDA_TRY(cudaMemcpyAsync(slot_expert, v.slot_expert, 4 * (size_t)S, cudaMemcpyDeviceToHost, s));
    if (last_use && S) PQE_CUDA_TRY(cudaMemcpyAsync(last_use, v.last_use, 8 * (size_t)S, cudaMemcpyDeviceToHost, s));
    PQE_CUDA_TRY(cudaStreamSynchronize(s));
    if (step) *step = hdr.step;
    if (stats)
        for (int j = 0; j < 4; ++j) stats[j] = hdr.stats[j];
    return PQE_OK;
}

int page_table_update_device(void *state, int E, int S, const int32_t *counts, const size_t *page_bytes,
                             int32_t *page_table, int32_t *miss, void *stream) {
    PQE_CHECK_ARG(state && counts && page_bytes && page_table && miss && E >= 1 && E <= 1024 && S >= 0 && S <= 1024);
    const int threads = ((E > S ? E : S) + 31) / 32 * 32;
    return launch_pdl(lru_step_kernel, 1, threads > 0 ? threads : 32, 0, as_stream(stream), state, E, S, counts,
                      page_bytes, page_table, miss);
}

int slot_fill_device(const pqe_pool *pool, const int32_t *miss, int E, const uint64_t *host_pages,
                     const size_t *page_bytes, void *stream) {
    PQE_CHECK_ARG(pool && miss && host_pages && page_bytes && E >= 1 && E <= 1024);
    int dev = 0, sms = 0;
    const int di = device_info(dev, sms);
    if (di != PQE_OK) return di;
    return slot_fill_device_group(pool, miss, E, host_pages, page_bytes, 0, 1, sms, as_stream(stream));
}

}  // extern "C"

namespace pqe {

int slot_fill_device_group(const pqe_pool *pool, const int32_t *miss, int E, const uint64_t *host_pages,
                           const size_t *page_bytes, int group, int groups, int ctas, cudaStream_t s) {
    if (!pool || !miss || !host_pages || !page_bytes || E < 1 || E > 1024 || groups < 1 || group < 0 ||
        group >= groups || ctas < 1)
        return PQE_ERR_INVALID_ARG;
    return launch_pdl(fill_device_kernel, ctas, DF_THREADS, sizeof(uint32_t) * (E + 1), s, miss, E, host_pages,
                      page_bytes, static_cast<uint8_t *>(pool->base), static_cast<uint8_t *>(pool->wb_base),
                      pool->n_slots, pool->slot_stride, group, groups);
}

}  // namespace pqe
