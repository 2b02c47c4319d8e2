// route_permute.cu -- router (top-k + gates), token-to-expert permutation,
// weighted combine, and the page quantisers.
//
// Router: the expert-pager article (rand.pepabo.com), "エキスパート重みの階層
// ページング", only says each token uses a few experts; the plain MoE top-k
// with renormalised softmax gates is used. Permutation: MoE-Gen summary
// (aibr.jp) "3.中核となる技術的要素", module-based batching: the assignments
// are grouped into one contiguous batch per expert.
#include <atomic>

#include "pqe_common.cuh"

namespace pqe {

// ===========================================================================
// K1: route. One warp per token.
// ===========================================================================

struct Cand {
    float v;
    int id;
};

__device__ __forceinline__ bool better(const Cand &a, const Cand &b) {
    return a.v > b.v || (a.v == b.v && a.id < b.id);
}

template <int NV>  // logits held per lane: experts e = lane + 32*i, i < NV
__global__ void __launch_bounds__(256) route_kernel(const uint16_t *__restrict__ x, const float *__restrict__ w_r,
                                                    float *__restrict__ logits, int T, int H, int E, int k,
                                                    int32_t *__restrict__ ids, float *__restrict__ gates) {
    pdl_acquire();  // launched after the previous kernel of the step: wait for its output
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    float lv[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) lv[i] = 0.0f;

    if (w_r != nullptr) {
        // fixed-order fp32 dot: lane l sums h = l, l+32, ... with FMA, then a
        // pairwise xor tree (16, 8, 4, 2, 1); every lane ends with the same bits
        const uint16_t *xt = x + (size_t)t * H;
        for (int e = 0; e < E; ++e) {
            const float *we = w_r + (size_t)e * H;
            float acc = 0.0f;
            for (int h = lane; h < H; h += 32) acc = __fmaf_rn(bf16_to_f32(__ldg(xt + h)), __ldg(we + h), acc);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
            if ((e & 31) == lane) lv[e >> 5] = acc;
            if (logits != nullptr && lane == 0) logits[(size_t)t * E + e] = acc;
        }
    } else {
        const float *lt = logits + (size_t)t * E;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            int e = lane + 32 * i;
            if (e < E) lv[i] = __ldg(lt + e);
        }
    }

    // top-k under `better` (larger value, then lower id): every lane sorts its
    // NV candidates once (bitonic network in registers, best first), then each
    // round the best of the 32 lane heads is the next pick and its lane drops
    // that head. A lane's remaining list is exactly its candidates not yet
    // picked, so round j picks the best candidate left: the same picks, in the
    // same order, as scanning every untaken candidate each round.
    Cand c[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        c[i] = e < E ? Cand{lv[i], e} : Cand{-INFINITY, 0x7fffffff};
    }
#pragma unroll
    for (int size = 2; size <= NV; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1)
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int j = i ^ stride;
                if (j > i) {
                    // best-first within blocks of `size` whose index bit `size` is 0
                    const bool desc = (i & size) == 0;
                    const Cand a = c[i], b = c[j];
                    const bool swap = desc ? better(b, a) : better(a, b);
                    c[i] = swap ? b : a;
                    c[j] = swap ? a : b;
                }
            }
    float top0 = 0.0f, sel_v = 0.0f;
    int sel_id = 0;
    for (int j = 0; j < k; ++j) {
        Cand w = c[0];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            Cand d{__shfl_xor_sync(0xffffffffu, w.v, o), __shfl_xor_sync(0xffffffffu, w.id, o)};
            if (better(d, w)) w = d;
        }
        if ((w.id & 31) == lane) {  // this lane's head was picked: drop it
#pragma unroll
            for (int i = 0; i + 1 < NV; ++i) c[i] = c[i + 1];
            c[NV - 1] = Cand{-INFINITY, 0x7fffffff};
        }
        if (j == 0) top0 = w.v;
        if (lane == j) {  // lane j keeps pick j (k <= 32)
            sel_v = w.v;
            sel_id = w.id;
        }
    }
    // gates: softmax over the k picked, in pick order
    float ex = (lane < k) ? expf(sel_v - top0) : 0.0f;
    float denom = 0.0f;
    for (int j = 0; j < k; ++j) denom += __shfl_sync(0xffffffffu, ex, j);
    if (lane < k) {
        ids[(size_t)t * k + lane] = sel_id;
        gates[(size_t)t * k + lane] = ex / denom;
    }
}

// ===========================================================================
// K2-K4: permutation (deterministic, stable).
//   count:   per-chunk histograms  hist[c][e]
//   scan:    per-expert prefix over chunks, offsets, chunk bases
//   scatter: per-warp stable ranks with match_any, write perm_src / inv
// ===========================================================================

constexpr int PERM_THREADS = 256;
constexpr int PERM_PER_THREAD = 8;
constexpr int PERM_CHUNK = PERM_THREADS * PERM_PER_THREAD;  // 2048 assignments per CTA
constexpr int PERM_WARPS = PERM_THREADS / 32;
constexpr int PERM_WARP_SPAN = PERM_CHUNK / PERM_WARPS;     // 256 consecutive per warp

__global__ void __launch_bounds__(PERM_THREADS) perm_count_kernel(const int32_t *__restrict__ ids, int A, int E,
                                                                   int32_t *__restrict__ hist,
                                                                   int32_t *__restrict__ status) {
    pdl_acquire();  // launched after the previous kernel of the step: wait for its output
    extern __shared__ int32_t sh[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
    __syncthreads();
    int base = blockIdx.x * PERM_CHUNK;
    bool bad = false;
    for (int i = threadIdx.x; i < PERM_CHUNK; i += blockDim.x) {
        int f = base + i;
        if (f < A) {
            int e = __ldg(ids + f);
            if (e >= 0 && e < E) atomicAdd(&sh[e], 1);
            else bad = true;
        }
    }
    if (bad) atomicOr(status, PQE_STATUS_BAD_EXPERT_ID);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)blockIdx.x * E + e] = sh[e];
}

// single CTA of 1024 threads
__global__ void __launch_bounds__(1024) perm_scan_kernel(int32_t *__restrict__ hist, int nchunk, int E, int A,
                                                         int32_t *__restrict__ counts,
                                                         int32_t *__restrict__ offsets,
                                                         int32_t *__restrict__ perm_src) {
    pdl_acquire();  // launched after the previous kernel of the step: wait for its output
    __shared__ int32_t tot[1024];
    __shared__ int32_t warp_sums[32];
    int e = threadIdx.x;
    int run = 0;
    if (e < E) {
        for (int c = 0; c < nchunk; ++c) {
            int v = hist[(size_t)c * E + e];
            hist[(size_t)c * E + e] = run;  // exclusive prefix over chunks
            run += v;
        }
        counts[e] = run;
    }
    tot[e] = (e < E) ? run : 0;
    __syncthreads();
    // exclusive scan of tot over 1024 entries
    int lane = e & 31, w = e >> 5;
    int v = tot[e];
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    if (w == 0) {
        int s = warp_sums[lane];
        int si = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, si, o);
            if (lane >= o) si += n;
        }
        warp_sums[lane] = si - s;
    }
    __syncthreads();
    int excl = warp_sums[w] + incl - v;
    if (e < E) {
        offsets[e] = excl;
        for (int c = 0; c < nchunk; ++c) hist[(size_t)c * E + e] += excl;
    }
    __shared__ int32_t s_valid;
    if (e == E - 1) {
        offsets[E] = excl + v;
        s_valid = excl + v;
    }
    __syncthreads();
    for (int p = s_valid + e; p < A; p += blockDim.x) perm_src[p] = -1;  // only when ids were dropped
}

__global__ void __launch_bounds__(PERM_THREADS) perm_scatter_kernel(const int32_t *__restrict__ ids, int A, int E,
                                                                     const int32_t *__restrict__ chunk_base,
                                                                     int32_t *__restrict__ perm_src,
                                                                     int32_t *__restrict__ inv) {
    pdl_acquire();  // launched after the previous kernel of the step: wait for its output
    extern __shared__ int32_t sh[];  // [PERM_WARPS][E] counts, then bases
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int32_t *wc = sh + (size_t)w * E;
    for (int i = threadIdx.x; i < PERM_WARPS * E; i += blockDim.x) sh[i] = 0;
    __syncthreads();
    const int base = blockIdx.x * PERM_CHUNK + w * PERM_WARP_SPAN;
    const unsigned lt_mask = (1u << lane) - 1u;
    // pass 1: per-warp counts
    for (int r = 0; r < PERM_WARP_SPAN / 32; ++r) {
        int f = base + r * 32 + lane;
        int e = (f < A) ? __ldg(ids + f) : -1;
        bool ok = e >= 0 && e < E;
        unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1);
        if (ok && (peers & lt_mask) == 0) wc[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // exclusive prefix over warps per expert, plus the chunk's global base
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = chunk_base[(size_t)blockIdx.x * E + e];
        for (int q = 0; q < PERM_WARPS; ++q) {
            int c = sh[(size_t)q * E + e];
            sh[(size_t)q * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    // pass 2: positions
    for (int r = 0; r < PERM_WARP_SPAN / 32; ++r) {
        int f = base + r * 32 + lane;
        int e = (f < A) ? __ldg(ids + f) : -1;
        bool ok = e >= 0 && e < E;
        unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1);
        if (f < A) {
            if (ok) {
                int p = wc[e] + __popc(peers & lt_mask);
                perm_src[p] = f;
                inv[f] = p;
            } else {
                inv[f] = -1;
            }
        }
        __syncwarp();
        if (ok && (peers & lt_mask) == 0) wc[e] += __popc(peers);
        __syncwarp();
    }
}

// One chunk (A <= PERM_CHUNK): the count, scan and scatter above in one CTA,
// with the same per-warp ranks, so the result is the same, and without the
// chunk histogram in global memory.
__global__ void __launch_bounds__(PERM_THREADS) perm_single_kernel(const int32_t *__restrict__ ids, int A, int E,
                                                                    int32_t *__restrict__ counts,
                                                                    int32_t *__restrict__ offsets,
                                                                    int32_t *__restrict__ perm_src,
                                                                    int32_t *__restrict__ inv,
                                                                    int32_t *__restrict__ status) {
    pdl_acquire();  // launched after the previous kernel of the step: wait for its output
    extern __shared__ int32_t sh[];  // [PERM_WARPS][E] per-warp counts, then bases
    __shared__ int32_t wsum[PERM_WARPS + 1];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    int32_t *wc = sh + (size_t)w * E;
    for (int i = tid; i < PERM_WARPS * E; i += PERM_THREADS) sh[i] = 0;
    __syncthreads();
    const int base = w * PERM_WARP_SPAN;
    const unsigned lt_mask = (1u << lane) - 1u;
    bool bad = false;
    // pass 1: per-warp counts
    for (int r = 0; r < PERM_WARP_SPAN / 32; ++r) {
        const int f = base + r * 32 + lane;
        const int e = (f < A) ? __ldg(ids + f) : -1;
        const bool ok = e >= 0 && e < E;
        bad |= f < A && !ok;
        const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1);
        if (ok && (peers & lt_mask) == 0) wc[e] += __popc(peers);
        __syncwarp();
    }
    if (bad) atomicOr(status, PQE_STATUS_BAD_EXPERT_ID);
    __syncthreads();
    // totals per expert, their exclusive prefix (thread t takes experts t*ept ..),
    // and each warp's base per expert
    const int ept = (E + PERM_THREADS - 1) / PERM_THREADS;
    int tsum = 0;
    for (int j = 0; j < ept; ++j) {
        const int e = tid * ept + j;
        if (e < E)
            for (int q = 0; q < PERM_WARPS; ++q) tsum += sh[(size_t)q * E + e];
    }
    int incl = tsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int q = 0; q < PERM_WARPS; ++q) {
            const int c = wsum[q];
            wsum[q] = run;
            run += c;
        }
        wsum[PERM_WARPS] = run;
    }
    __syncthreads();
    int run = wsum[w] + incl - tsum;
    for (int j = 0; j < ept; ++j) {
        const int e = tid * ept + j;
        if (e < E) {
            offsets[e] = run;
            const int start = run;
            for (int q = 0; q < PERM_WARPS; ++q) {
                const int c = sh[(size_t)q * E + e];
                sh[(size_t)q * E + e] = run;
                run += c;
            }
            counts[e] = run - start;
        }
    }
    const int valid = wsum[PERM_WARPS];
    if (tid == 0) offsets[E] = valid;
    __syncthreads();
    // pass 2: positions
    for (int r = 0; r < PERM_WARP_SPAN / 32; ++r) {
        const int f = base + r * 32 + lane;
        const int e = (f < A) ? __ldg(ids + f) : -1;
        const bool ok = e >= 0 && e < E;
        const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1);
        if (f < A) {
            if (ok) {
                const int p = wc[e] + __popc(peers & lt_mask);
                perm_src[p] = f;
                inv[f] = p;
            } else {
                inv[f] = -1;
            }
        }
        __syncwarp();
        if (ok && (peers & lt_mask) == 0) wc[e] += __popc(peers);
        __syncwarp();
    }
    for (int p = valid + tid; p < A; p += PERM_THREADS) perm_src[p] = -1;  // only when ids were dropped
}

// ===========================================================================
// K8: combine. One CTA per token, each thread 8 columns (16 bytes).
// ===========================================================================

__global__ void __launch_bounds__(256) combine_kernel(const uint16_t *__restrict__ out_perm,
                                                      const int32_t *__restrict__ inv,
                                                      const float *__restrict__ gates, int T, int k, int H,
                                                      uint16_t *__restrict__ y) {
    pdl_acquire();  // launched after the previous kernel of the step: wait for its output
    const int t = blockIdx.x;
    for (int c8 = threadIdx.x; c8 < H / 8; c8 += blockDim.x) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int j = 0; j < k; ++j) {
            int p = __ldg(inv + (size_t)t * k + j);
            if (p < 0) continue;
            float g = __ldg(gates + (size_t)t * k + j);
            uint4 v = __ldg(reinterpret_cast<const uint4 *>(out_perm + (size_t)p * H) + c8);
            uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] = __fmaf_rn(g, bf16_to_f32((uint16_t)(u[i] & 0xffff)), acc[2 * i]);
                acc[2 * i + 1] = __fmaf_rn(g, bf16_to_f32((uint16_t)(u[i] >> 16)), acc[2 * i + 1]);
            }
        }
        uint4 o;
        o.x = f32_to_bf16_rn(acc[0]) | ((uint32_t)f32_to_bf16_rn(acc[1]) << 16);
        o.y = f32_to_bf16_rn(acc[2]) | ((uint32_t)f32_to_bf16_rn(acc[3]) << 16);
        o.z = f32_to_bf16_rn(acc[4]) | ((uint32_t)f32_to_bf16_rn(acc[5]) << 16);
        o.w = f32_to_bf16_rn(acc[6]) | ((uint32_t)f32_to_bf16_rn(acc[7]) << 16);
        reinterpret_cast<uint4 *>(y + (size_t)t * H)[c8] = o;
    }
}

// ===========================================================================
// Page quantisers (page preparation, not on the per-step path).
// ===========================================================================

__global__ void __launch_bounds__(256) quant_fp8_rows_kernel(const float *__restrict__ w, int cols,
                                                             uint8_t *__restrict__ q, float *__restrict__ scale) {
    __shared__ float red[8];
    const float *wr = w + (size_t)blockIdx.x * cols;
    float amax = 0.0f;
    for (int c = threadIdx.x; c < cols; c += blockDim.x) amax = fmaxf(amax, fabsf(wr[c]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, red[i]);
    const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
    if (threadIdx.x == 0) scale[blockIdx.x] = s;
    uint8_t *qr = q + (size_t)blockIdx.x * cols;
    for (int c = 2 * threadIdx.x; c < cols; c += 2 * blockDim.x) {
        uint16_t v = f32x2_to_e4m3x2(__fdiv_rn(wr[c], s), __fdiv_rn(wr[c + 1], s));
        *reinterpret_cast<uint16_t *>(qr + c) = v;
    }
}

// one warp per 32-element block
__global__ void __launch_bounds__(256) quant_mxfp4_kernel(const uint8_t *__restrict__ q8, const float *__restrict__ s8,
                                                          int rows, int cols, uint8_t *__restrict__ q4,
                                                          uint8_t *__restrict__ x8) {
    const int lane = threadIdx.x & 31;
    const long blk = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int nblk = cols / 32;
    if (blk >= (long)rows * nblk) return;
    const int r = (int)(blk / nblk), b = (int)(blk % nblk);
    const uint8_t code = q8[(size_t)r * cols + b * 32 + lane];
    const float2 f = e4m3x2_to_f32x2(code);
    const float v = __fmul_rn(f.x, s8[r]);
    float amax = fabsf(v);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    uint32_t sb = 0;
    if (amax != 0.0f) {
        uint32_t bits = __float_as_uint(amax);
        int ex = (int)((bits >> 23) & 0xff);
        int E = (ex != 0) ? ex - 127 : (31 - __clz((int)(bits & 0x7fffff))) - 149;  // floor(log2 amax)
        int byte = E - 2 + 127;
        sb = (uint32_t)(byte < 0 ? 0 : (byte > 254 ? 254 : byte));
    }
    const float X = e8m0_to_f32(sb);
    const float qv = __fdiv_rn(v, X);
    const float other = __shfl_down_sync(0xffffffffu, qv, 1);
    if ((lane & 1) == 0) q4[((size_t)r * cols + b * 32 + lane) / 2] = f32x2_to_e2m1x2(qv, other);
    if (lane == 0) x8[(size_t)r * nblk + b] = (uint8_t)sb;
}

// ---------------------------------------------------------------------------
// Scratch of moe_permute_static: a file-scope device array, so that call needs
// no workspace from the caller. Every GPU that loads the library holds it
// until the process exits. Only device code may name it; host code reaches it
// through the per-device address from cudaGetSymbolAddress.
// ---------------------------------------------------------------------------
constexpr size_t PERM_STATIC_WORDS = (size_t)1 << 20;  // 4 MiB of int32 chunk histograms
static __device__ __align__(256) int32_t g_perm_scratch[PERM_STATIC_WORDS];

// One cached address per device. Host threads may make their first call on a
// device at the same time: each looks the address up and stores the same
// value, so relaxed atomics suffice (as for the launch caches of device_info).
static std::atomic<int32_t *> g_perm_scratch_addr[PQE_MAX_DEVICES];

// address of g_perm_scratch on the current device, looked up once per device
static int perm_static_scratch(int32_t **out) {
    int dev = 0;
    PQE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= PQE_MAX_DEVICES) return PQE_ERR_UNSUPPORTED;
    int32_t *p = g_perm_scratch_addr[dev].load(std::memory_order_relaxed);
    if (!p) {
        void *q = nullptr;
        PQE_CUDA_TRY(cudaGetSymbolAddress(&q, g_perm_scratch));
        p = static_cast<int32_t *>(q);
        g_perm_scratch_addr[dev].store(p, std::memory_order_relaxed);
    }
    *out = p;
    return PQE_OK;
}

}  // namespace pqe

using namespace pqe;

extern "C" {

int moe_route(const void *x_bf16, const float *w_router, float *logits, int T, int H, int E, int k,
              int32_t *topk_ids, float *topk_w, void *stream) {
    PQE_CHECK_ARG(T >= 0 && E >= 1 && E <= 1024 && k >= 1 && k <= 32 && k <= E);
    if (T == 0) return PQE_OK;
    PQE_CHECK_ARG(topk_ids && topk_w);
    if (w_router) PQE_CHECK_ARG(x_bf16 && H >= 1);
    else PQE_CHECK_ARG(logits);
    const int warps = 8;
    dim3 grid((T + warps - 1) / warps), block(32 * warps);
    auto s = as_stream(stream);
    const uint16_t *x = static_cast<const uint16_t *>(x_bf16);
    int nv = (E + 31) / 32;
    auto kern = nv <= 1 ? route_kernel<1> : nv <= 2 ? route_kernel<2> : nv <= 4 ? route_kernel<4>
              : nv <= 8 ? route_kernel<8> : nv <= 16 ? route_kernel<16> : route_kernel<32>;
    return launch_pdl(kern, grid, block, 0, s, x, w_router, logits, T, H, E, k, topk_ids, topk_w);
}

size_t moe_permute_workspace_size(int T, int k, int E) {
    if (T < 0 || k < 1 || E < 1) return 0;
    size_t A = (size_t)T * k;
    size_t nchunk = (A + PERM_CHUNK - 1) / PERM_CHUNK;
    if (nchunk == 0) nchunk = 1;
    return round_up(nchunk * (size_t)E * sizeof(int32_t), 256);
}

int moe_permute(const int32_t *topk_ids, int T, int k, int E, int32_t *counts, int32_t *offsets,
                int32_t *perm_src, int32_t *inv, void *ws, size_t ws_bytes, int32_t *status, void *stream) {
    PQE_CHECK_ARG(T >= 0 && k >= 1 && k <= 32 && E >= 1 && E <= 1024);
    PQE_CHECK_ARG(counts && offsets && status);
    auto s = as_stream(stream);
    const long A = (long)T * k;
    PQE_CHECK_ARG(A < (1L << 30));
    if (A == 0) {
        PQE_CUDA_TRY(cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s));
        PQE_CUDA_TRY(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s));
        return PQE_OK;
    }
    PQE_CHECK_ARG(topk_ids && perm_src && inv && ws);
    PQE_CHECK_ARG(ws_bytes >= moe_permute_workspace_size(T, k, E) && aligned(ws, 256));
    const int nchunk = (int)((A + PERM_CHUNK - 1) / PERM_CHUNK);
    const size_t smem = sizeof(int32_t) * PERM_WARPS * E;
    if (smem > 48 * 1024) {
        PQE_CUDA_TRY(cudaFuncSetAttribute(perm_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        PQE_CUDA_TRY(cudaFuncSetAttribute(perm_single_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    }
    if (nchunk == 1)  // one CTA covers the step: one kernel
        return launch_pdl(perm_single_kernel, 1, PERM_THREADS, smem, s, topk_ids, (int)A, E, counts, offsets, perm_src,
                          inv, status);
    int32_t *hist = static_cast<int32_t *>(ws);
    int rc = launch_pdl(perm_count_kernel, nchunk, PERM_THREADS, sizeof(int32_t) * E, s, topk_ids, (int)A, E, hist,
                        status);
    if (rc != PQE_OK) return rc;
    if ((rc = launch_pdl(perm_scan_kernel, 1, 1024, 0, s, hist, nchunk, E, (int)A, counts, offsets, perm_src)))
        return rc;
    return launch_pdl(perm_scatter_kernel, nchunk, PERM_THREADS, smem, s, topk_ids, (int)A, E, hist, perm_src, inv);
}

size_t moe_permute_static_max_words(void) { return PERM_STATIC_WORDS; }

int moe_permute_static(const int32_t *topk_ids, int T, int k, int E, int32_t *counts, int32_t *offsets,
                       int32_t *perm_src, int32_t *inv, int32_t *status, void *stream) {
    PQE_CHECK_ARG(T >= 0 && k >= 1 && k <= 32 && E >= 1 && E <= 1024);
    PQE_CHECK_ARG(counts && offsets && status);
    const size_t need = moe_permute_workspace_size(T, k, E);
    if (need > PERM_STATIC_WORDS * sizeof(int32_t)) return PQE_ERR_CAPACITY;
    int32_t *scratch = nullptr;
    int rc = perm_static_scratch(&scratch);
    if (rc != PQE_OK) return rc;
    // the chunk histograms are written in full by every call before they are
    // read, so nothing has to be cleared between calls
    return moe_permute(topk_ids, T, k, E, counts, offsets, perm_src, inv, scratch, need, status, stream);
}

int moe_combine(const void *out_perm, const int32_t *inv, const float *topk_w, int T, int k, int H, void *y_bf16,
                void *stream) {
    PQE_CHECK_ARG(T >= 0 && k >= 1 && k <= 32 && H >= 8 && H % 8 == 0);
    if (T == 0) return PQE_OK;
    PQE_CHECK_ARG(out_perm && inv && topk_w && y_bf16);
    PQE_CHECK_ARG(aligned(out_perm, 16) && aligned(y_bf16, 16));
    int threads = H / 8 < 256 ? ((H / 8 + 31) / 32) * 32 : 256;
    return launch_pdl(combine_kernel, T, threads, 0, as_stream(stream), static_cast<const uint16_t *>(out_perm), inv,
                      topk_w, T, k, H, static_cast<uint16_t *>(y_bf16));
}

int pqe_quantize_fp8_rows(const float *w, int rows, int cols, uint8_t *q, float *scale, void *stream) {
    PQE_CHECK_ARG(w && q && scale && rows >= 0 && cols >= 2 && cols % 2 == 0);
    if (rows == 0) return PQE_OK;
    quant_fp8_rows_kernel<<<rows, 256, 0, as_stream(stream)>>>(w, cols, q, scale);
    PQE_LAUNCH_CHECK();
    return PQE_OK;
}

int pqe_quantize_mxfp4_rows(const uint8_t *q8, const float *s8, int rows, int cols, uint8_t *q4, uint8_t *x8,
                            void *stream) {
    PQE_CHECK_ARG(q8 && s8 && q4 && x8 && rows >= 0 && cols >= 32 && cols % 32 == 0);
    if (rows == 0) return PQE_OK;
    long blocks = (long)rows * (cols / 32);
    long grid = (blocks + 7) / 8;
    PQE_CHECK_ARG(grid < (1L << 31));
    quant_mxfp4_kernel<<<(unsigned)grid, 256, 0, as_stream(stream)>>>(q8, s8, rows, cols, q4, x8);
    PQE_LAUNCH_CHECK();
    return PQE_OK;
}

int pqe_pack_fp8_page(const float *w13, const float *w2, int H, int I, uint8_t *page, void *stream) {
    PQE_CHECK_ARG(w13 && w2 && page && shape_ok(H, I) && aligned(page, 16));
    const PageLayout L = fp8_layout(H, I);
    int rc = pqe_quantize_fp8_rows(w13, 2 * I, H, page + L.w13, reinterpret_cast<float *>(page + L.s13), stream);
    if (rc != PQE_OK) return rc;
    return pqe_quantize_fp8_rows(w2, H, I, page + L.w2, reinterpret_cast<float *>(page + L.s2), stream);
}

int pqe_pack_mxfp4_page(const uint8_t *fp8_page, int H, int I, uint8_t *fp4_page, void *stream) {
    PQE_CHECK_ARG(fp8_page && fp4_page && shape_ok(H, I) && aligned(fp8_page, 16) && aligned(fp4_page, 16));
    const PageLayout A = fp8_layout(H, I), B = mxfp4_layout(H, I);
    int rc = pqe_quantize_mxfp4_rows(fp8_page + A.w13, reinterpret_cast<const float *>(fp8_page + A.s13), 2 * I, H,
                                     fp4_page + B.w13, fp4_page + B.s13, stream);
    if (rc != PQE_OK) return rc;
    return pqe_quantize_mxfp4_rows(fp8_page + A.w2, reinterpret_cast<const float *>(fp8_page + A.s2), H, I,
                                   fp4_page + B.w2, fp4_page + B.s2, stream);
}

}  // extern "C"
