// ffn_gemv.cu -- expert FFN over the slot pool, weight-streaming CUDA-core path.
//
// For each routed expert e (its page in slot page_table[e]) and each batch
// position p of e: u = W13_e x_t, h = SiLU(u[:I]) * u[I:], out_perm[p] = W2_e h.
// Paging per layer and the w13/w2 weight names: expert-pager article
// (rand.pepabo.com), "エキスパート重みの階層ページング" and "評価"; 4-bit pages:
// PagedWeight commentary (spectral-agent.com), "技術的に面白い点".
//
// This path serves small per-expert batches (decode), where the layer is bound
// by streaming the weights from HBM: every weight byte is read once per group
// of up to NT tokens with 128-bit loads, converted exactly to fp32 and
// multiplied with bf16 activations in fp32. h stays fp32.
#include <atomic>

#include "pqe_common.cuh"
#include "ffn_internal.cuh"

namespace pqe {

// ---------------------------------------------------------------------------
// schedule (one CTA, one thread per expert, ascending id):
//   sched[0] = count, sched[1 + a] = experts for the CUDA-core path;
//   tiles[i] = {expert, first batch row, valid rows, page entry} of the
//   128-row tiles of experts on the tensor-core path, those of FP8 pages
//   first, then those of MXFP4 pages; n_tiles = {all, FP8, MXFP4} counts.
// An expert goes to the tensor cores when tc_min > 0, its batch has at least
// tc_min rows, its page is FP8 or MXFP4 and its page-table entry is inside
// the pool.
// ---------------------------------------------------------------------------
// exclusive scans of four ints per thread at once (blockDim a multiple of 32,
// at most 1024): one pair of barriers for all four
__device__ __forceinline__ int4 block_excl_scan4(int4 v, int (*wt)[33], int4 &total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int4 incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, incl.x, o), b = __shfl_up_sync(0xffffffffu, incl.y, o),
                  c = __shfl_up_sync(0xffffffffu, incl.z, o), d = __shfl_up_sync(0xffffffffu, incl.w, o);
        if (lane >= o) incl = make_int4(incl.x + a, incl.y + b, incl.z + c, incl.w + d);
    }
    if (lane == 31) {
        wt[0][w] = incl.x;
        wt[1][w] = incl.y;
        wt[2][w] = incl.z;
        wt[3][w] = incl.w;
    }
    __syncthreads();
    for (int q = w; q < 4; q += nw) {  // component q's warp totals, scanned by warp q mod nw
        const int c = lane < nw ? wt[q][lane] : 0;
        int ci = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, ci, o);
            if (lane >= o) ci += n;
        }
        wt[q][lane] = ci - c;
        if (lane == 31) wt[q][32] = ci;
    }
    __syncthreads();
    total = make_int4(wt[0][32], wt[1][32], wt[2][32], wt[3][32]);
    return make_int4(wt[0][w] + incl.x - v.x, wt[1][w] + incl.y - v.y, wt[2][w] + incl.z - v.z,
                     wt[3][w] + incl.w - v.w);
}

// With a miss list (an overlapped step), only the experts of pass `pass` are
// scheduled: pass 0 the experts not in the list, pass g + 1 the misses refill
// group g brings (ranks overlap_group_start(g) .. overlap_group_start(g + 1) - 1).
__global__ void __launch_bounds__(1024) ffn_schedule_kernel(FfnArgs a, int tc_min, int32_t *__restrict__ tiles,
                                                            int32_t *__restrict__ n_tiles,
                                                            const int32_t *__restrict__ miss, int groups, int pass) {
    pdl_acquire();  // launched after the previous kernel of the step: wait for its output
    __shared__ int scan_tot[4][33];
    __shared__ int16_t s_pass[1024];
    const int e = threadIdx.x;
    if (miss) {
        if (e < a.E) s_pass[e] = 0;
        __syncthreads();
        const int nm = miss[0];
        for (int r = e; r < nm; r += blockDim.x) {
            int g = 0;
            while (g + 1 < groups && overlap_group_start(g + 1, groups, nm) <= r) ++g;
            s_pass[miss[2 + r]] = (int16_t)(1 + g);
        }
        __syncthreads();
    }
    int n = 0, slot = -1, fmt = PQE_FMT_FP8, p0 = 0;
    if (e < a.E && (!miss || s_pass[e] == pass)) {
        p0 = a.offsets[e];
        n = a.offsets[e + 1] - p0;
        slot = a.page_table[e];
        fmt = a.expert_fmt ? (int)a.expert_fmt[e] : PQE_FMT_FP8;
    }
    if (e < a.E && a.done13) a.done13[e] = 0u;
    if (e == 0 && a.done13) a.done13[a.E] = 0u;  // the tensor-core stream's grab counter
    const bool valid_page = slot >= 0 && slot < a.n_slots + a.n_wb;
    const bool big = n > 0 && tc_min > 0 && n >= tc_min && valid_page;
    // large batches take the tcgen05 path: FP8 pages on the FP8 GEMM, MXFP4 pages
    // on the block-scaled GEMM; everything else (and unknown formats) the weight stream
    const bool tc8 = big && fmt == PQE_FMT_FP8, tc4 = big && fmt == PQE_FMT_MXFP4;
    const bool gemv = n > 0 && !tc8 && !tc4;
    // work weight of a weight-stream expert: its bytes (FP8 4, E2M1 2) plus 3 per
    // further group of 8 tokens (each repeats the conversion and the mma);
    // tiles of 128 batch rows: the FP8 experts' first, then the MXFP4 experts'
    const int wgt = (fmt == PQE_FMT_FP8 ? 4 : 2) + 3 * ((n > 0 ? n - 1 : 0) / 8);
    const int nt8 = tc8 ? (n + 127) / 128 : 0, nt4 = tc4 ? (n + 127) / 128 : 0;
    int4 tot;
    const int4 pre = block_excl_scan4(make_int4(gemv ? 1 : 0, gemv ? wgt : 0, nt8, nt4), scan_tot, tot);
    const int gpos = pre.x, wpos = pre.y, tpos8 = pre.z, tpos4 = pre.w;
    const int total = tot.x, wtot = tot.y, total8 = tot.z, total4 = tot.w;
    if (gemv) {
        a.sched[1 + gpos] = e;
        // the stream kernels read the expert's batch and page from here: one
        // dependent load fewer before their first copies
        a.info[gpos] = make_int4(e, p0, n, info_pack(slot, fmt));
    }
    if (threadIdx.x == 0) a.sched[0] = total;
    if (gemv) a.wpre[gpos] = wpos;
    if (threadIdx.x == 0) a.wpre[total] = wtot;
    const int nt = nt8 + nt4, tpos = tc8 ? tpos8 : total8 + tpos4;
    for (int i = 0; i < nt; ++i) {
        int4 t;
        t.x = e;
        t.y = a.offsets[e] + 128 * i;
        t.z = min(128, n - 128 * i);
        t.w = slot;
        reinterpret_cast<int4 *>(tiles)[tpos + i] = t;
    }
    if (threadIdx.x == 0) {
        n_tiles[0] = total8 + total4;  // all tiles
        n_tiles[1] = total8;           // FP8 tiles: [0, total8)
        n_tiles[2] = total4;           // MXFP4 tiles: [total8, total8 + total4)
    }
}

__device__ __forceinline__ bool page_ok(const FfnArgs &a, int e, int &slot, int &fmt) {
    slot = a.page_table[e];
    fmt = a.expert_fmt ? (int)a.expert_fmt[e] : PQE_FMT_FP8;
    return slot >= 0 && slot < a.n_slots + a.n_wb && (fmt == PQE_FMT_FP8 || fmt == PQE_FMT_MXFP4);
}

// 16 bf16 activations (two uint4 in shared memory) dotted with 16 fp32 weights
__device__ __forceinline__ float dot16_bf16(const float (&w)[16], const uint4 &x0, const uint4 &x1, float acc) {
    const uint32_t xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        acc = __fmaf_rn(w[2 * i], __uint_as_float(xs[i] << 16), acc);
        acc = __fmaf_rn(w[2 * i + 1], __uint_as_float(xs[i] & 0xffff0000u), acc);
    }
    return acc;
}

__device__ __forceinline__ void cvt16_e4m3(const uint4 &v, float (&f)[16]) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 a = e4m3x2_to_f32x2((uint16_t)(u[i] & 0xffff));
        float2 b = e4m3x2_to_f32x2((uint16_t)(u[i] >> 16));
        f[4 * i] = a.x;
        f[4 * i + 1] = a.y;
        f[4 * i + 2] = b.x;
        f[4 * i + 3] = b.y;
    }
}

// 8 bytes of E2M1 pairs -> 16 fp32
__device__ __forceinline__ void cvt16_e2m1(uint32_t lo, uint32_t hi, float (&f)[16]) {
    const uint32_t u[2] = {lo, hi};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            float2 v = e2m1x2_to_f32x2((uint8_t)(u[i] >> (8 * b)));
            f[8 * i + 2 * b] = v.x;
            f[8 * i + 2 * b + 1] = v.y;
        }
    }
}

// ---------------------------------------------------------------------------
// w13 + SwiGLU. Unit = (active expert a, block of 8 gate/up row pairs); one
// warp per pair (gate row j, up row I + j). Tokens in groups of NT, their x
// rows staged in shared memory as bf16.
// ---------------------------------------------------------------------------
template <int NT>
__global__ void __launch_bounds__(256) ffn_w13_gemv_kernel(FfnArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem_raw);  // [NT][H]
    const int H = a.H, I = a.I;
    const int rblocks = I / 8;
    const int units = a.sched[0] * rblocks;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int unit = blockIdx.x; unit < units; unit += gridDim.x) {
    const int act_i = unit / rblocks, rb = unit % rblocks;
    const int e = a.sched[1 + act_i];
    const int p0 = a.offsets[e], n = a.offsets[e + 1] - p0;
    const int j = rb * 8 + warp;
    int slot, fmt;
    if (!page_ok(a, e, slot, fmt)) {
        if (threadIdx.x == 0) atomicOr(a.status, PQE_STATUS_BAD_PAGE);
        if (lane == 0)
            for (int p = p0; p < p0 + n; ++p) a.h[(size_t)p * I + j] = 0.0f;
        continue;
    }
    const uint8_t *page = page_addr(a, slot);
    for (int g0 = 0; g0 < n; g0 += NT) {
        const int nt = min(NT, n - g0);
        __syncthreads();
        for (int i = threadIdx.x; i < nt * (H / 8); i += blockDim.x) {
            const int tt = i / (H / 8), c = i % (H / 8);
            const int tok = a.perm_src[p0 + g0 + tt] / a.k;
            reinterpret_cast<uint4 *>(xs + (size_t)tt * H)[c] =
                __ldg(reinterpret_cast<const uint4 *>(a.x + (size_t)tok * H) + c);
        }
        __syncthreads();
        float ag[NT], au[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) ag[t] = au[t] = 0.0f;
        if (fmt == PQE_FMT_FP8) {
            const uint4 *gr = reinterpret_cast<const uint4 *>(page + (size_t)j * H);
            const uint4 *ur = reinterpret_cast<const uint4 *>(page + (size_t)(I + j) * H);
            for (int c = lane; c < H / 16; c += 32) {
                float wg[16], wu[16];
                cvt16_e4m3(__ldg(gr + c), wg);
                cvt16_e4m3(__ldg(ur + c), wu);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (t < nt) {
                        const uint4 *xr = reinterpret_cast<const uint4 *>(xs + (size_t)t * H + 16 * c);
                        const uint4 x0 = xr[0], x1 = xr[1];
                        ag[t] = dot16_bf16(wg, x0, x1, ag[t]);
                        au[t] = dot16_bf16(wu, x0, x1, au[t]);
                    }
                }
            }
        } else {
            const PageLayout L = mxfp4_layout(H, I);
            const uint4 *gr = reinterpret_cast<const uint4 *>(page + (size_t)j * (H / 2));
            const uint4 *ur = reinterpret_cast<const uint4 *>(page + (size_t)(I + j) * (H / 2));
            const uint8_t *xg = page + L.s13 + (size_t)j * (H / 32);
            const uint8_t *xu = page + L.s13 + (size_t)(I + j) * (H / 32);
            for (int c = lane; c < H / 32; c += 32) {  // 16 bytes = 32 weights = one scale block
                const uint4 vg = __ldg(gr + c), vu = __ldg(ur + c);
                const float sg = e8m0_to_f32(__ldg(xg + c)), su = e8m0_to_f32(__ldg(xu + c));
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float wg[16], wu[16];
                    cvt16_e2m1(half ? vg.z : vg.x, half ? vg.w : vg.y, wg);
                    cvt16_e2m1(half ? vu.z : vu.x, half ? vu.w : vu.y, wu);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        wg[q] *= sg;
                        wu[q] *= su;
                    }
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        if (t < nt) {
                            const uint4 *xr =
                                reinterpret_cast<const uint4 *>(xs + (size_t)t * H + 32 * c + 16 * half);
                            const uint4 x0 = xr[0], x1 = xr[1];
                            ag[t] = dot16_bf16(wg, x0, x1, ag[t]);
                            au[t] = dot16_bf16(wu, x0, x1, au[t]);
                        }
                    }
                }
            }
        }
        float sg = 1.0f, su = 1.0f;
        if (fmt == PQE_FMT_FP8) {
            const PageLayout L = fp8_layout(H, I);
            sg = __ldg(reinterpret_cast<const float *>(page + L.s13) + j);
            su = __ldg(reinterpret_cast<const float *>(page + L.s13) + I + j);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (t < nt) {
                const float g = warp_sum(ag[t]) * sg;
                const float u = warp_sum(au[t]) * su;
                if (lane == 0) a.h[(size_t)(p0 + g0 + t) * I + j] = silu(g) * u;
            }
        }
    }
    __syncthreads();  // x staging is reused by the next unit
    }
}

// ---------------------------------------------------------------------------
// w2. Unit = (active expert a, block of 32 output rows); each warp 4 rows.
// h rows of a token group staged in shared memory (fp32); the CTA's 32
// outputs per token are written as one 64-byte bf16 segment.
// ---------------------------------------------------------------------------
template <int NT>
__global__ void __launch_bounds__(256) ffn_w2_gemv_kernel(FfnArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    float *hs = reinterpret_cast<float *>(smem_raw);  // [NT][I]
    __shared__ float outs[NT][32];
    const int H = a.H, I = a.I;
    const int rblocks = H / 32;
    const int units = a.sched[0] * rblocks;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int unit = blockIdx.x; unit < units; unit += gridDim.x) {
    const int act_i = unit / rblocks, rb = unit % rblocks;
    const int e = a.sched[1 + act_i];
    const int p0 = a.offsets[e], n = a.offsets[e + 1] - p0;
    const int r0 = rb * 32 + warp * 4;
    int slot, fmt;
    const bool ok = page_ok(a, e, slot, fmt);
    const uint8_t *page = page_addr(a, ok ? slot : 0);
    for (int g0 = 0; g0 < n; g0 += NT) {
        const int nt = min(NT, n - g0);
        __syncthreads();
        if (ok) {
            for (int i = threadIdx.x; i < nt * (I / 4); i += blockDim.x) {
                const int tt = i / (I / 4), c = i % (I / 4);
                reinterpret_cast<float4 *>(hs + (size_t)tt * I)[c] =
                    reinterpret_cast<const float4 *>(a.h + (size_t)(p0 + g0 + tt) * I)[c];
            }
        }
        __syncthreads();
        float acc[4][NT];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[r][t] = 0.0f;
        if (ok && fmt == PQE_FMT_FP8) {
            const PageLayout L = fp8_layout(H, I);
            for (int c = lane; c < I / 16; c += 32) {
                float w[4][16];
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    cvt16_e4m3(__ldg(reinterpret_cast<const uint4 *>(page + L.w2 + (size_t)(r0 + r) * I) + c), w[r]);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (t < nt) {
                        const float4 *hr = reinterpret_cast<const float4 *>(hs + (size_t)t * I + 16 * c);
                        float hv[16];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            float4 v = hr[q];
                            hv[4 * q] = v.x;
                            hv[4 * q + 1] = v.y;
                            hv[4 * q + 2] = v.z;
                            hv[4 * q + 3] = v.w;
                        }
#pragma unroll
                        for (int r = 0; r < 4; ++r)
#pragma unroll
                            for (int q = 0; q < 16; ++q) acc[r][t] = __fmaf_rn(w[r][q], hv[q], acc[r][t]);
                    }
                }
            }
        } else if (ok) {
            const PageLayout L = mxfp4_layout(H, I);
            for (int c = lane; c < I / 32; c += 32) {
                uint4 v[4];
                float sc[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    v[r] = __ldg(reinterpret_cast<const uint4 *>(page + L.w2 + (size_t)(r0 + r) * (I / 2)) + c);
                    sc[r] = e8m0_to_f32(__ldg(page + L.s2 + (size_t)(r0 + r) * (I / 32) + c));
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float w[4][16];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        cvt16_e2m1(half ? v[r].z : v[r].x, half ? v[r].w : v[r].y, w[r]);
#pragma unroll
                        for (int q = 0; q < 16; ++q) w[r][q] *= sc[r];
                    }
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        if (t < nt) {
                            const float4 *hr = reinterpret_cast<const float4 *>(hs + (size_t)t * I + 32 * c + 16 * half);
                            float hv[16];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                float4 x4 = hr[q];
                                hv[4 * q] = x4.x;
                                hv[4 * q + 1] = x4.y;
                                hv[4 * q + 2] = x4.z;
                                hv[4 * q + 3] = x4.w;
                            }
#pragma unroll
                            for (int r = 0; r < 4; ++r)
#pragma unroll
                                for (int q = 0; q < 16; ++q) acc[r][t] = __fmaf_rn(w[r][q], hv[q], acc[r][t]);
                        }
                    }
                }
            }
        }
        float s2[4] = {1.0f, 1.0f, 1.0f, 1.0f};
        if (ok && fmt == PQE_FMT_FP8) {
            const PageLayout L = fp8_layout(H, I);
#pragma unroll
            for (int r = 0; r < 4; ++r) s2[r] = __ldg(reinterpret_cast<const float *>(page + L.s2) + r0 + r);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float v = warp_sum(acc[r][t]) * s2[r];
                if (lane == 0 && t < nt) outs[t][warp * 4 + r] = v;
            }
        }
        __syncthreads();
        for (int i = threadIdx.x; i < nt * 32; i += blockDim.x) {
            const int t = i / 32, c = i % 32;
            a.out_perm[(size_t)(p0 + g0 + t) * H + rb * 32 + c] = f32_to_bf16_rn(outs[t][c]);
        }
    }
    if (!ok && threadIdx.x == 0 && n > 0) atomicOr(a.status, PQE_STATUS_BAD_PAGE);
    __syncthreads();  // h staging and outs are reused by the next unit
    }
}

int launch_ffn_gemv(const FfnArgs &args, int max_active, cudaStream_t s) {
    constexpr int NT = 4;
    const size_t smem13 = (size_t)NT * args.H * sizeof(uint16_t);
    const size_t smem2 = (size_t)NT * args.I * sizeof(float);
    if (smem13 > 48 * 1024)
        PQE_CUDA_TRY(cudaFuncSetAttribute(ffn_w13_gemv_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)smem13));
    if (smem2 > 48 * 1024)
        PQE_CUDA_TRY(cudaFuncSetAttribute(ffn_w2_gemv_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)smem2));
    // grid-stride over (expert, row block) units; the unit count is known on the device
    int dev = 0, sms = 0;
    const int di = device_info(dev, sms);
    if (di != PQE_OK) return di;
    const long cap = 8L * sms;
    const long u13 = (long)max_active * (args.I / 8), u2 = (long)max_active * (args.H / 32);
    ffn_w13_gemv_kernel<NT><<<(unsigned)(u13 < cap ? u13 : cap), 256, smem13, s>>>(args);
    PQE_LAUNCH_CHECK();
    ffn_w2_gemv_kernel<NT><<<(unsigned)(u2 < cap ? u2 : cap), 256, smem2, s>>>(args);
    PQE_LAUNCH_CHECK();
    return PQE_OK;
}

// workspace carve-up shared by the size query and the call
struct FfnWs {
    size_t sched, wpre, tiles, n_tiles, done13, info, h, xt, st, xq, sx, hbf, hmax, hq, sh, total;
    int max_tiles;
    bool tc;
};

static FfnWs ffn_ws_layout(int T, int k, int E, int H, int I) {
    FfnWs w{};
    const size_t A = (size_t)T * k;
    // an expert's batch holds at most one row per token (top-k picks distinct
    // experts), so with fewer than TC_MIN_ROWS tokens no batch reaches the
    // tensor cores: no tile buffers, no side chain, the weight stream on every SM
    w.tc = tc_shape_ok(H, I) && T >= TC_MIN_ROWS;
    w.max_tiles = w.tc ? (int)((A + 127) / 128 + (size_t)E) : 0;
    size_t off = 0;
    auto take = [&off](size_t b) {
        const size_t at = off;
        off += round_up(b ? b : 1, 256);
        return at;
    };
    w.sched = take(sizeof(int32_t) * (E + 1));
    w.wpre = take(sizeof(int32_t) * (E + 1));
    w.tiles = take(sizeof(int32_t) * 4 * (size_t)(w.max_tiles ? w.max_tiles : 1));
    w.n_tiles = take(3 * sizeof(int32_t));
    w.done13 = take(sizeof(uint32_t) * (E + 1));
    w.info = take(sizeof(int4) * (size_t)E);
    w.h = take(A * I * sizeof(float));
    if (w.tc) {
        w.xt = take((size_t)T * H);
        w.st = take((size_t)T * sizeof(float));
        w.xq = take(A * H);
        w.sx = take(A * sizeof(float));
        w.hbf = take(A * I * sizeof(uint16_t));
        w.hmax = take(A * sizeof(uint32_t));
        w.hq = take(A * I);
        w.sh = take(A * sizeof(float));
    }
    w.total = off;
    return w;
}

// The side stream of this host thread on the current device, with its fork and
// join events (created on first use; one set per thread, so calls from several
// host threads never share them).
struct SideStream {
    int dev = -1;
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

static int side_stream(int dev, SideStream *&out) {
    thread_local SideStream ss[PQE_MAX_DEVICES];
    if (dev < 0 || dev >= PQE_MAX_DEVICES) return PQE_ERR_UNSUPPORTED;
    SideStream &x = ss[dev];
    if (x.s == nullptr) {
        PQE_CUDA_TRY(cudaStreamCreateWithFlags(&x.s, cudaStreamNonBlocking));
        PQE_CUDA_TRY(cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming));
        PQE_CUDA_TRY(cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming));
        x.dev = dev;
    }
    out = &x;
    return PQE_OK;
}

int device_info(int &dev, int &sms) {
    static std::atomic<int> cache[PQE_MAX_DEVICES];
    PQE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= PQE_MAX_DEVICES) return PQE_ERR_UNSUPPORTED;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        PQE_CUDA_TRY(cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev));
        cache[dev].store(v, std::memory_order_relaxed);
    }
    sms = v;
    return PQE_OK;
}

}  // namespace pqe

using namespace pqe;

extern "C" {

size_t moe_paged_ffn_workspace_size(int T, int k, int E, int H, int I) {
    if (T < 0 || k < 1 || E < 1 || !shape_ok(H, I)) return 0;
    return ffn_ws_layout(T, k, E, H, I).total;
}

int moe_paged_ffn(const void *x_bf16, const int32_t *perm_src, const int32_t *offsets, const int32_t *page_table,
                  const uint8_t *expert_fmt, const pqe_pool *pool, int T, int k, int E, void *out_perm, void *ws,
                  size_t ws_bytes, int32_t *status, void *stream) {
    return pqe::moe_paged_ffn_pass(x_bf16, perm_src, offsets, page_table, expert_fmt, pool, T, k, E, out_perm, ws,
                                   ws_bytes, status, as_stream(stream), nullptr, 1, 0, 0);
}

}  // extern "C"

namespace pqe {

int moe_paged_ffn_pass(const void *x_bf16, const int32_t *perm_src, const int32_t *offsets,
                       const int32_t *page_table, const uint8_t *expert_fmt, const pqe_pool *pool, int T, int k,
                       int E, void *out_perm, void *ws, size_t ws_bytes, int32_t *status, cudaStream_t s,
                       const int32_t *miss, int groups, int pass, int reserve_sms) {
    PQE_CHECK_ARG(pool && T >= 0 && k >= 1 && k <= 32 && E >= 1 && E <= 1024 && k <= E);
    PQE_CHECK_ARG(groups >= 1 && pass >= 0 && pass <= groups && reserve_sms >= 0);
    PQE_CHECK_ARG(shape_ok(pool->H, pool->I));
    if (T == 0) return PQE_OK;
    PQE_CHECK_ARG(x_bf16 && perm_src && offsets && page_table && out_perm && ws && status);
    PQE_CHECK_ARG(pool->n_slots >= 0 && pool->n_wb >= 0 && pool->n_slots + pool->n_wb >= 1);
    PQE_CHECK_ARG(pool->slot_stride == pqe_slot_stride(pool->H, pool->I));
    PQE_CHECK_ARG(pool->n_slots == 0 || (pool->base && aligned(pool->base, 256)));
    PQE_CHECK_ARG(pool->n_wb == 0 || (pool->wb_base && aligned(pool->wb_base, 256)));
    PQE_CHECK_ARG(aligned(x_bf16, 16) && aligned(out_perm, 16) && aligned(ws, 256));
    PQE_CHECK_ARG(ws_bytes >= moe_paged_ffn_workspace_size(T, k, E, pool->H, pool->I));
    FfnArgs args{};
    args.x = static_cast<const uint16_t *>(x_bf16);
    args.perm_src = perm_src;
    args.offsets = offsets;
    args.page_table = page_table;
    args.expert_fmt = expert_fmt;
    args.pool_base = static_cast<const uint8_t *>(pool->base);
    args.wb_base = static_cast<const uint8_t *>(pool->wb_base);
    args.slot_stride = pool->slot_stride;
    args.n_slots = pool->n_slots;
    args.n_wb = pool->n_wb;
    args.T = T;
    args.k = k;
    args.E = E;
    args.H = pool->H;
    args.I = pool->I;
    const FfnWs w = ffn_ws_layout(T, k, E, pool->H, pool->I);
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    args.sched = reinterpret_cast<int32_t *>(wsb + w.sched);
    args.wpre = reinterpret_cast<int32_t *>(wsb + w.wpre);
    args.h = reinterpret_cast<float *>(wsb + w.h);
    args.out_perm = static_cast<uint16_t *>(out_perm);
    args.status = status;
    args.done13 = reinterpret_cast<uint32_t *>(wsb + w.done13);
    args.info = reinterpret_cast<int4 *>(wsb + w.info);
    args.wait_limit = wait_limit();
    args.phase2_bias = phase2_bias();
    const long A = (long)T * k;
    const int max_active = (int)(A < E ? A : E);
    int32_t *tiles = reinterpret_cast<int32_t *>(wsb + w.tiles);
    int32_t *n_tiles = reinterpret_cast<int32_t *>(wsb + w.n_tiles);
    const int sr = launch_pdl(ffn_schedule_kernel, 1, (E + 31) / 32 * 32, 0, s, args, w.tc ? TC_MIN_ROWS : 0, tiles,
                              n_tiles, miss, groups, pass);
    if (sr != PQE_OK) return sr;
    const bool stream_path = stream_shape_ok(pool->H, pool->I);
    int dev = 0, sms = 0;
    const int di = device_info(dev, sms);
    if (di != PQE_OK) return di;
    // SMs left to a refill running beside this pass
    if (reserve_sms > 0) sms = sms - reserve_sms > 2 * TC_SIDE_SMS + 8 ? sms - reserve_sms : 2 * TC_SIDE_SMS + 8;
    // the tensor-core stream on all-FP8 layers once the step routes enough experts
    const int kind = stream_kernel_choice();
    const bool tc_ok = stream_path && expert_fmt == nullptr && stream_tc_shape_ok(pool->H, pool->I);
    const bool use_tc = tc_ok && (kind == 2 || (kind == 0 && max_active >= STREAM_TC_MIN_EXPERTS));
    const int side_sms = use_tc ? TC_SIDE_SMS_TC_STREAM : TC_SIDE_SMS;
    // decode-sized step: the tensor-core batches run beside the weight stream
    const bool side = stream_path && w.tc && A >= TC_MIN_ROWS && A <= (long)DECODE_ROWS_PER_EXPERT * E &&
                      sms > 2 * side_sms;
    SideStream *ss = nullptr;
    if (side) {
        const int r = side_stream(dev, ss);
        if (r != PQE_OK) return r;
        PQE_CUDA_TRY(cudaEventRecord(ss->fork, s));
    }
    // the stream kernel goes out first: from an idle GPU every host step before it
    // is a gap after the schedule kernel
    int rc;
    if (stream_path) {
        const int grid = side ? sms - side_sms : (reserve_sms > 0 ? sms : 0);
        rc = use_tc ? launch_ffn_stream_tc(args, s, grid) : launch_ffn_stream(args, s, grid);
    } else {
        rc = launch_ffn_gemv(args, max_active, s);
    }
    if (side) PQE_CUDA_TRY(cudaStreamWaitEvent(ss->s, ss->fork, 0));
    if (rc != PQE_OK || !w.tc) {
        if (side) {  // close the fork
            PQE_CUDA_TRY(cudaEventRecord(ss->join, ss->s));
            PQE_CUDA_TRY(cudaStreamWaitEvent(s, ss->join, 0));
        }
        return rc;
    }
    TcBuffers b{};
    b.A = A;
    b.tiles = tiles;
    b.n_tiles = n_tiles;
    b.xt = wsb + w.xt;
    b.st = reinterpret_cast<float *>(wsb + w.st);
    b.xq = wsb + w.xq;
    b.sx = reinterpret_cast<float *>(wsb + w.sx);
    b.h = reinterpret_cast<uint16_t *>(wsb + w.hbf);
    b.hmax = reinterpret_cast<uint32_t *>(wsb + w.hmax);
    b.hq = wsb + w.hq;
    b.sh = reinterpret_cast<float *>(wsb + w.sh);
    if (!side) return launch_ffn_tc(args, b, w.max_tiles, s, sms);
    rc = launch_ffn_tc(args, b, w.max_tiles, ss->s, side_sms);
    // the join is recorded even after a failed launch, so the caller's stream never
    // waits on a fork that was left open
    PQE_CUDA_TRY(cudaEventRecord(ss->join, ss->s));
    PQE_CUDA_TRY(cudaStreamWaitEvent(s, ss->join, 0));
    return rc;
}

}  // namespace pqe
