// ffn_stream_tc.cu -- expert FFN for small per-expert batches (decode) on the
// 5th-generation tensor cores: a persistent weight stream whose multiplies are
// tcgen05 MMAs with the expert's weight rows as the 128-row operand.
//
// A routed expert's weights are read once from its slot (expert-pager article,
// rand.pepabo.com, "エキスパート重みの階層ページング"); with at most 8 tokens
// per expert the FFN is bound by that stream from HBM. The weight rows are the
// MMA's M side (128 rows) and the tokens its N side: each token's activations
// are split into two E4M3 terms, hi = E4M3(v) and lo = E4M3(v - hi) with
// v = x / s and s = amax / 448 per token, so that hi + lo = v within 2^-8 |v|;
// the 8 hi and 8 lo columns make N = 16 (the smallest N of an M = 128 MMA),
// and the epilogue adds the two column halves. Weights enter the MMA as the
// page's E4M3 codes, exact; products and sums are fp32 in TMEM.
//
// Work items (per expert):
//   phase 1  item rb: 64 gate rows [64 rb, 64 rb + 64) and the matching up rows
//            [I + 64 rb, ...) as one 128-row tile over K = H; the epilogue
//            computes h[p, 64 rb + j] = SiLU(gate_j . x_p) * (up_j . x_p) (fp32,
//            both sides scaled by their row scale and the token's s), then
//            publishes the item on the expert's phase-1 count
//   phase 2  item rb: w2 rows [128 rb, 128 rb + 128) over K = I;
//            out_perm[p, 128 rb + r] = bf16(w2_r . h_p * s2_r)
// Phase 2 of an expert starts once its phase-1 count is complete (items of any
// CTA): no grid-wide barrier, and the weight stream keeps loading meanwhile.
//
// Work is taken dynamically in grabs: a phase-1 grab is one phase-1 item, a
// phase-2 grab G2 consecutive phase-2 items of one expert (about half the
// bytes of a phase-1 item). Grab g of the step is phase-1 item g for
// g < n1 = experts * (I / 64), else phase-2 grab g - n1; both in the order of
// the active-expert list, so an expert's phase-1 items are taken together and
// its phase-2 grabs long after. CTA c takes grab c first, then the value of a
// global counter plus the grid size, until the grabs run out: a CTA that
// streams faster takes more, and the step ends within about one grab of the
// last CTA.
//
// One CTA per SM (cooperative launch), sixteen warps:
//   warp 14    scheduler (one thread): takes the next grab, reads its expert,
//              batch and page from the schedule's record of the expert, and
//              publishes it in a queue of two entries that every other role
//              reads in order (an entry is reused once each reader has copied
//              it)
//   warp 0     TMA producer (one thread): each stage is 128 weight rows x 128
//              bytes of K, two [64 rows x 128 B] boxes from the page's 3-D map
//              [slot, row, k], 128-byte swizzle, into a ring of 16 KB stages
//   warps 1,15 MMA issuers (one thread each; warp 1 owns TMEM): each issues
//              two of a stage's four kind::f8f6f4 MMAs (K = 32 each) into its
//              own half of one of two accumulators (16 fp32 columns a half),
//              so that a stage costs each thread half the issue time; a stage
//              is released once both have committed it
//   warps 2-5  epilogue, one per TMEM lane quarter, adding the two issuers'
//              halves and each token's hi and lo columns: rows 0-63 of a
//              phase-1 tile are gate rows, 64-127 up rows, so the up warps hand
//              their values to the gate warps through shared memory
//   warps 6-13 activation tiles, one warp per token: for each grab, quantise
//              the expert's token rows (x, or h once its phase-1 count is
//              complete) into a [16 x K] E4M3 tile in the MMA's swizzled
//              layout, double-buffered; each lane loads its whole share of the
//              row into registers before the tile's buffer is free, so the
//              load latency overlaps the MMAs still reading that buffer. A step
//              of at most 8 tokens has all of x and perm_src staged in shared
//              memory first, so its phase-1 tiles need no global load
// Every wait is bounded: on expiry PQE_STATUS_TIMEOUT is set, the waiting role
// stops, the CTA drains the copies and MMAs it issued, frees its TMEM and
// returns.
#include <cuda.h>

#include <atomic>

#include "ffn_internal.cuh"
#include "pqe_common.cuh"
#include "tc_ptx.cuh"

namespace pqe {
namespace sw {
using namespace ptx;

constexpr int W_TMA = 0, W_MMA = 1, W_EPI0 = 2, W_ACT0 = 6, W_SCHED = 14, W_MMA1 = 15;  // warp roles
constexpr int EPI_WARPS = 4, ACT_WARPS = 8, MMA_ISSUERS = 2;
constexpr int THREADS = 32 * (W_MMA1 + 1);
constexpr int QN = 2;                   // grabs in the queue
constexpr int NTOK = 8;                 // tokens of one expert batch on this path (one activation warp each)
constexpr int XCH = 5;                  // 16-element chunks of an x row per lane at most (H <= 2560)
constexpr int HCH = 2;                  // 16-element chunks of an h row per lane at most (I <= 1024)
constexpr int MMA_N = 2 * NTOK;         // hi and lo columns
constexpr int ROWS = 128;               // weight rows per item (the MMA's M)
constexpr int KSTEP = 128;              // bytes of K per stage (one swizzle-atom row)
constexpr uint32_t STAGE_BYTES = ROWS * KSTEP;
constexpr uint32_t BOX_BYTES = 64 * KSTEP;      // one TMA box: 64 rows
constexpr uint32_t ACT_STEP = MMA_N * KSTEP;    // activation tile bytes per K step
constexpr int MAX_STAGES = 9, MIN_STAGES = 3;
constexpr uint32_t ACC_COLS = MMA_ISSUERS * MMA_N;  // fp32 columns of one accumulator: a half per issuer
constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;        // two accumulators
// every reader of a queue entry copies it and then frees it
constexpr uint32_t QFREE_COUNT = 1 + MMA_ISSUERS + ACT_WARPS + EPI_WARPS;
// instruction descriptor, kind::f8f6f4: D f32, A and B E4M3, both K-major, N = 16, M = 128
constexpr uint32_t IDESC = (1u << 4) | ((uint32_t)(MMA_N >> 3) << 17) | ((uint32_t)(ROWS >> 4) << 24);
// phase-1 work counted per item on the expert's count: the unit of that count is
// 8 gate/up row pairs of one token group, and an item holds 64 pairs of at most
// NTOK tokens (one group)
constexpr uint32_t COUNT_PER_ITEM = 64 / 8;
static_assert(TC_MIN_ROWS <= NTOK + 1, "batches on this path hold at most NTOK rows");
static_assert(ACT_WARPS == NTOK, "one activation warp per token of a batch");

struct Geo {
    int stages;
    uint32_t act_off, act_bytes;  // two activation tiles of act_bytes
    uint32_t xb_off;              // [2][64][NTOK] fp32: up-row values for the gate warps
    uint32_t ts_off;              // [2][NTOK] fp32: token scales of each activation tile
    uint32_t q_off;               // Grab [QN]: the queue
    uint32_t xs_off, xs_bytes;    // steps of at most NTOK tokens: x [T][H] bf16, then perm_src [T k], staged
    uint32_t bar_off, tmem_off, smem_bytes;
};

// one grab as the scheduler publishes it: row blocks [rb0, rb0 + nrb) of one
// expert's phase; phase 0 marks the end of the work
struct Grab {
    int phase, e, p0, n, slot, valid, rb0, nrb;
};

// position in the stage ring: stage s and the parity of its current fill
struct Ring {
    int s = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void next(int stages) {
        if (++s == stages) {
            s = 0;
            ph ^= 1u;
        }
    }
};

// bounded wait without sleeping between polls (try_wait itself suspends the
// thread for a while): a sleeping waiter wakes late, and every wait here is on
// the stream's critical path; false after `limit` polls
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// a ready barrier costs one poll; otherwise the bounded wait
__device__ __forceinline__ bool mbar_ready(uint32_t bar, uint32_t parity, uint32_t limit) {
    return mbar_try_wait(bar, parity) || wait_bar(bar, parity, limit);
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// two fp32 -> packed E4M3 pair (lo in the low byte), round to nearest even, saturating
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// packed E4M3 pair -> the two values (exact)
__device__ __forceinline__ void e4m3x2_val(uint32_t p, float &lo, float &hi) {
    uint32_t h2;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "r"(p));
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h2));
}

// 16 values already in units of the token scale -> E4M3 codes hi and lo with
// hi + lo = v within 2^-8 |v| (lo holds the rounding error of hi); element i in
// byte i % 4 of word i / 4, K order
__device__ __forceinline__ void split16(const float (&v)[16], uint4 &hi, uint4 &lo) {
    uint32_t h[4] = {0u, 0u, 0u, 0u}, l[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t hp = e4m3x2(v[2 * i], v[2 * i + 1]);
        float b0, b1;
        e4m3x2_val(hp, b0, b1);
        const uint32_t lp = e4m3x2(v[2 * i] - b0, v[2 * i + 1] - b1);
        h[i >> 1] |= hp << (16 * (i & 1));
        l[i >> 1] |= lp << (16 * (i & 1));
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// byte offset of 16-byte chunk j (0..7) of tile row r (0..15) inside one K step
// of the activation tile: 8-row groups of 128-byte rows, 1024 B apart, chunk j
// of row r at position j ^ (r % 8) (the MMA's 128-byte swizzle)
__device__ __forceinline__ uint32_t act_chunk(int r, int j) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// 448 / amax, kept finite for tiny rows (1 for a zero row)
__device__ __forceinline__ float act_factor(float amax) {
    return amax > 0.0f ? fminf(448.0f / amax, 0x1p100f) : 1.0f;
}

// named barriers of the epilogue warps: 1 (all four, AND vote), 3 (all four), 2 (the two gate warps);
// 4 is the activation warps' (staging a small step's x)
__device__ __forceinline__ bool epi_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, "
        "q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(EPI_WARPS * 32)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 3, %0;" ::"n"(EPI_WARPS * 32) : "memory"); }
__device__ __forceinline__ void gate_sync() { asm volatile("bar.sync 2, 64;" ::: "memory"); }

__global__ void __launch_bounds__(THREADS, 1)
    ffn_stream_tc_kernel(const __grid_constant__ CUtensorMap m13c, const __grid_constant__ CUtensorMap m13w,
                         const __grid_constant__ CUtensorMap m2c, const __grid_constant__ CUtensorMap m2w,
                         const FfnArgs a, const Geo g) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int H = a.H, I = a.I;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar_full = sbase + g.bar_off;
    const uint32_t bar_empty = bar_full + 8 * g.stages;
    const uint32_t bar_tfull = bar_empty + 8 * g.stages;  // [2] accumulator written
    const uint32_t bar_tempty = bar_tfull + 16;           // [2] accumulator read
    const uint32_t bar_afull = bar_tempty + 16;           // [2] activation tile written
    const uint32_t bar_aempty = bar_afull + 16;           // [2] activation tile no longer read
    const uint32_t bar_qfull = bar_aempty + 16;           // [QN] queue entry published
    const uint32_t bar_qfree = bar_qfull + 8 * QN;        // [QN] queue entry copied by all of its readers
    const uint32_t bar_drain = bar_qfree + 8 * QN;        // every MMA of the CTA finished
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + g.tmem_off);
    Grab *s_q = reinterpret_cast<Grab *>(smem + g.q_off);
    float *s_ts = reinterpret_cast<float *>(smem + g.ts_off);
    const PageLayout L = fp8_layout(H, I);
    const int per1 = I / 64, per2 = H / ROWS;
    const int nk1 = H / KSTEP, nk2 = I / KSTEP;

    if (warp == W_TMA) {
        if (lane == 0) {
            for (int s = 0; s < g.stages; ++s) {
                mbar_init(bar_full + 8 * s, 1);
                mbar_init(bar_empty + 8 * s, MMA_ISSUERS);
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(bar_tfull + 8 * b, MMA_ISSUERS);
                mbar_init(bar_tempty + 8 * b, EPI_WARPS);
                mbar_init(bar_afull + 8 * b, ACT_WARPS);
                mbar_init(bar_aempty + 8 * b, MMA_ISSUERS + EPI_WARPS);  // the MMAs' commits and each epilogue warp
            }
            for (int q = 0; q < QN; ++q) {
                mbar_init(bar_qfull + 8 * q, 1);
                mbar_init(bar_qfree + 8 * q, QFREE_COUNT);
            }
            mbar_init(bar_drain, MMA_ISSUERS);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&m13c)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&m13w)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&m2c)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&m2w)) : "memory");
        }
    } else if (warp == W_MMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == W_SCHED) {
        // ---------------- scheduler ----------------
        if (lane == 0) {
            const int n_act = __ldg(a.sched);
            const int g2 = H / (2 * I) > 1 ? H / (2 * I) : 1;  // phase-2 items per grab
            const int ng2 = (per2 + g2 - 1) / g2;
            const int n1 = n_act * per1, ng = n1 + n_act * ng2;
            uint32_t *counter = a.done13 + a.E;
            int gi = blockIdx.x;
            bool ok = true;
            for (int q = 0; ok; ++q) {
                Grab gr;
                gr.phase = 0;
                int next = ng;
                if (gi < ng) {
                    int i;
                    if (gi < n1) {
                        i = gi / per1;
                        gr.phase = 1;
                        gr.rb0 = gi - i * per1;
                        gr.nrb = 1;
                    } else {
                        const int r = gi - n1;
                        i = r / ng2;
                        gr.phase = 2;
                        gr.rb0 = (r - i * ng2) * g2;
                        gr.nrb = min(g2, per2 - gr.rb0);
                    }
                    const int4 r = __ldg(a.info + i);  // the schedule's record: expert, batch, page
                    gr.e = r.x;
                    gr.p0 = r.y;
                    gr.n = r.z;
                    gr.slot = info_slot(r.w);
                    gr.valid = gr.slot >= 0 && gr.slot < a.n_slots + a.n_wb && info_fmt(r.w) == PQE_FMT_FP8;
                    // the grab after this one, taken while this one waits for its entry
                    next = (int)gridDim.x + (int)atomicAdd(counter, 1u);
                }
                const int qs = q % QN;
                ok = wait_bar(bar_qfree + 8 * qs, ((uint32_t)(q / QN) & 1u) ^ 1u, a.wait_limit);
                if (!ok) {
                    atomicOr(a.status, PQE_STATUS_TIMEOUT);
                    break;
                }
                s_q[qs] = gr;
                mbar_arrive_plain(bar_qfull + 8 * qs);  // release: the entry is visible to its waiters
                if (gr.phase == 0) break;
                gi = next;
            }
        }
    } else if (warp == W_TMA) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int it = 0;
            Ring rp;
            bool ok = true;
            for (int q = 0; ok; ++q) {
                if (!wait_bar(bar_qfull + 8 * (q % QN), (uint32_t)(q / QN) & 1u, a.wait_limit)) {
                    ok = false;
                    break;
                }
                const Grab gr = s_q[q % QN];
                mbar_arrive_plain(bar_qfree + 8 * (q % QN));
                if (gr.phase == 0) break;
                const bool cache = gr.slot < a.n_slots;
                const int zc = cache ? gr.slot : gr.slot - a.n_slots;
                const CUtensorMap *mp = gr.phase == 1 ? (cache ? &m13c : &m13w) : (cache ? &m2c : &m2w);
                const int nk = gr.phase == 1 ? nk1 : nk2;
                for (int rb = gr.rb0; rb < gr.rb0 + gr.nrb && ok; ++rb) {
                    // the tile's two 64-row boxes
                    const int r_lo = gr.phase == 1 ? 64 * rb : ROWS * rb;
                    const int r_hi = gr.phase == 1 ? I + 64 * rb : ROWS * rb + 64;
                    for (int ks = 0; ks < nk; ++ks, ++it, rp.next(g.stages)) {
                        const int s = rp.s;
                        if (!mbar_ready(bar_empty + 8 * s, rp.ph ^ 1u, a.wait_limit)) {
                            ok = false;
                            break;
                        }
                        const uint32_t dst = sbase + (uint32_t)s * STAGE_BYTES, fb = bar_full + 8 * s;
                        if (gr.valid) {
                            mbar_expect_tx(fb, STAGE_BYTES);
                            tma_load_3d(dst, mp, ks * KSTEP, r_lo, zc, fb);
                            tma_load_3d(dst + BOX_BYTES, mp, ks * KSTEP, r_hi, zc, fb);
                        } else {
                            mbar_arrive_plain(fb);  // no page: nothing to load, the epilogue writes zeros
                        }
                    }
                }
            }
            if (!ok) atomicOr(a.status, PQE_STATUS_TIMEOUT);
            // drain: the stages issued last have landed before the CTA may exit
            for (int j = (it > g.stages ? it - g.stages : 0); j < it; ++j)
                wait_bar(bar_full + 8 * (j % g.stages), (uint32_t)(j / g.stages) & 1u, a.wait_limit);
        }
    } else if (warp == W_MMA || warp == W_MMA1) {
        // ---------------- MMA issuers ----------------
        if (lane == 0) {
            const int mi = warp == W_MMA ? 0 : 1;  // this issuer's K = 32 slices of a stage: 2 mi, 2 mi + 1
            int j = 0;  // items issued (accumulator alternation)
            Ring rp;
            bool ok = true;
            // descriptors of stage 0 and of the two activation tiles; a byte offset
            // o < 256 KB moves a descriptor by o >> 4 (its address field, no carry)
            const uint64_t adesc0 = sw128_desc(sbase);
            const uint64_t bdesc0 = sw128_desc(sbase + g.act_off);
            for (int q = 0; ok; ++q) {
                if (!wait_bar(bar_qfull + 8 * (q % QN), (uint32_t)(q / QN) & 1u, a.wait_limit)) {
                    ok = false;
                    break;
                }
                const Grab gr = s_q[q % QN];
                mbar_arrive_plain(bar_qfree + 8 * (q % QN));
                if (gr.phase == 0) break;
                const int buf = q & 1;
                if (!wait_bar(bar_afull + 8 * buf, (uint32_t)(q >> 1) & 1u, a.wait_limit)) {
                    ok = false;
                    break;
                }
                const int nk = gr.phase == 1 ? nk1 : nk2;
                for (int r = 0; r < gr.nrb && ok; ++r, ++j) {
                    const int acc = j & 1;
                    if (!mbar_ready(bar_tempty + 8 * acc, ((uint32_t)(j >> 1) & 1u) ^ 1u, a.wait_limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)acc * ACC_COLS + (uint32_t)(mi * MMA_N);
                    uint64_t bd = bdesc0 + (uint64_t)(((uint32_t)buf * g.act_bytes) >> 4) + (uint64_t)(4 * mi);
                    for (int ks = 0; ks < nk; ++ks, rp.next(g.stages), bd += ACT_STEP >> 4) {
                        const int s = rp.s;
                        if (!mbar_ready(bar_full + 8 * s, rp.ph, a.wait_limit)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (gr.valid) {
                            // this issuer's two K = 32 slices of the stage's 128-byte rows (+32 B each)
                            const uint64_t ad = adesc0 + (uint64_t)(((uint32_t)s * STAGE_BYTES) >> 4) + (uint64_t)(4 * mi);
                            umma_f8f6f4(d, ad, bd, IDESC, ks != 0);
                            umma_f8f6f4(d, ad + 2, bd + 2, IDESC, 1u);
                        }
                        umma_commit(bar_empty + 8 * s);
                    }
                    if (!ok) break;
                    umma_commit(bar_tfull + 8 * acc);
                }
                if (!ok) break;
                umma_commit(bar_aempty + 8 * buf);
            }
            if (!ok) atomicOr(a.status, PQE_STATUS_TIMEOUT);
            // every issued MMA has finished before TMEM is released (also after a wait gave up mid-item)
            umma_commit(bar_drain);
            wait_bar(bar_drain, 0u, a.wait_limit);
        }
    } else if (warp < W_ACT0) {
        // ---------------- epilogue: TMEM -> h / out_perm ----------------
        const int q4 = warp & 3;        // the TMEM lane quarter this warp may access
        const int m = 32 * q4 + lane;   // tile row
        float *xb = reinterpret_cast<float *>(smem + g.xb_off);
        int j = 0;
        for (int q = 0;; ++q) {
            const bool okq = wait_bar(bar_qfull + 8 * (q % QN), (uint32_t)(q / QN) & 1u, a.wait_limit);
            if (!epi_all(okq)) {
                if (threadIdx.x == 32 * W_EPI0) atomicOr(a.status, PQE_STATUS_TIMEOUT);
                break;
            }
            const Grab f = s_q[q % QN];
            __syncwarp();
            if (lane == 0) mbar_arrive_plain(bar_qfree + 8 * (q % QN));  // copied
            if (f.phase == 0) break;
            const int buf = q & 1;
            bool stop = false;
            for (int r = 0; r < f.nrb; ++r, ++j) {
                const int rb = f.rb0 + r, phase = f.phase, acc = j & 1;
                // this row's scale, read before the accumulator wait
                float srow = 0.0f;
                if (f.valid) {
                    const uint8_t *page = page_addr(a, f.slot);
                    const int row = phase == 1 ? (m < 64 ? 64 * rb + m : I + 64 * rb + (m - 64)) : ROWS * rb + m;
                    srow = __ldg(reinterpret_cast<const float *>(page + (phase == 1 ? L.s13 : L.s2)) + row);
                }
                // the activation tile's scales were written before its barrier completed
                const bool ok = wait_bar(bar_tfull + 8 * acc, (uint32_t)(j >> 1) & 1u, a.wait_limit) &&
                                wait_bar(bar_afull + 8 * buf, (uint32_t)(q >> 1) & 1u, a.wait_limit);
                if (!epi_all(ok)) {
                    if (threadIdx.x == 32 * W_EPI0) atomicOr(a.status, PQE_STATUS_TIMEOUT);
                    stop = true;
                    break;
                }
                tc_fence_after();
                uint32_t d[32];  // issuer 0's hi, lo columns, then issuer 1's
                tmem_ld32(tmem + (uint32_t)acc * ACC_COLS + ((uint32_t)(32 * q4) << 16), d);
                tmem_ld_wait();
                float ts[NTOK];
#pragma unroll
                for (int t = 0; t < NTOK; ++t) ts[t] = s_ts[buf * NTOK + t];
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_plain(bar_tempty + 8 * acc);
                    if (r + 1 == f.nrb) mbar_arrive_plain(bar_aempty + 8 * buf);
                }
                float v[NTOK];
#pragma unroll
                for (int t = 0; t < NTOK; ++t)
                    v[t] = f.valid ? ((__uint_as_float(d[t]) + __uint_as_float(d[MMA_N + t])) +
                                      (__uint_as_float(d[NTOK + t]) + __uint_as_float(d[MMA_N + NTOK + t]))) *
                                         ts[t] * srow
                                   : 0.0f;
                if (phase == 1) {
                    float *x = xb + (j & 1) * 64 * NTOK;
                    if (q4 >= 2) {
                        float4 *o = reinterpret_cast<float4 *>(x + (m - 64) * NTOK);
                        o[0] = make_float4(v[0], v[1], v[2], v[3]);
                        o[1] = make_float4(v[4], v[5], v[6], v[7]);
                    }
                    epi_sync();
                    if (q4 < 2) {
                        const float4 *u4 = reinterpret_cast<const float4 *>(x + m * NTOK);
                        const float4 ua = u4[0], ub = u4[1];
                        const float u[NTOK] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
                        float *hr = a.h + (size_t)f.p0 * I + 64 * rb + m;
#pragma unroll
                        for (int t = 0; t < NTOK; ++t)
                            if (t < f.n) hr[(size_t)t * I] = silu(v[t]) * u[t];
                        __threadfence();
                        gate_sync();
                        if (m == 0) atomicAdd(a.done13 + f.e, COUNT_PER_ITEM);
                    }
                } else {
                    uint16_t *o = a.out_perm + (size_t)f.p0 * H + ROWS * rb + m;
#pragma unroll
                    for (int t = 0; t < NTOK; ++t)
                        if (t < f.n) o[(size_t)t * H] = f32_to_bf16_rn(v[t]);
                }
            }
            if (stop) break;
        }
    } else if (warp < W_SCHED) {
        // ---------------- activation tiles ----------------
        const int aw = warp - W_ACT0;
        bool timed_out = false, counts_expired = false;
        // a small step: all of x and perm_src into shared memory once (no
        // dependent global loads behind the weight copies per phase-1 tile)
        const uint16_t *xsrc = a.x;
        const int32_t *psrc = a.perm_src;
        if (g.xs_bytes) {
            uint4 *xd = reinterpret_cast<uint4 *>(smem + g.xs_off);
            const int nx = a.T * H / 8, np = a.T * a.k, ta = threadIdx.x - 32 * W_ACT0;
            for (int i = ta; i < nx; i += 32 * ACT_WARPS) xd[i] = __ldg(reinterpret_cast<const uint4 *>(a.x) + i);
            int32_t *pd = reinterpret_cast<int32_t *>(smem + g.xs_off + (size_t)a.T * H * 2);
            for (int i = ta; i < np; i += 32 * ACT_WARPS) pd[i] = __ldg(a.perm_src + i);
            asm volatile("bar.sync 4, %0;" ::"n"(32 * ACT_WARPS) : "memory");  // the activation warps only (barrier 4)
            xsrc = reinterpret_cast<const uint16_t *>(xd);
            psrc = pd;
        }
        for (int q = 0;; ++q) {
            const int buf = q & 1;
            int ok = 1;
            if (lane == 0) ok = wait_bar(bar_qfull + 8 * (q % QN), (uint32_t)(q / QN) & 1u, a.wait_limit);
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                timed_out = true;
                break;
            }
            __syncwarp();  // lane 0's acquire orders the other lanes' reads of the entry
            const Grab f = s_q[q % QN];
            __syncwarp();
            if (lane == 0) mbar_arrive_plain(bar_qfree + 8 * (q % QN));
            if (f.phase == 0) break;
            // this warp's token row into registers before its tile buffer is free:
            // the loads are in flight while the MMAs finish with the buffer
            const bool mine = f.valid && aw < f.n;
            uint4 u[2 * XCH];  // x: bf16 pairs; h: fp32 bits, four per entry
#pragma unroll
            for (int i = 0; i < 2 * XCH; ++i) u[i] = make_uint4(0u, 0u, 0u, 0u);
            if (mine && f.phase == 1) {
                const int nch = H / 16;
                const uint4 *xr = reinterpret_cast<const uint4 *>(xsrc + (size_t)(psrc[f.p0 + aw] / a.k) * H);
#pragma unroll
                for (int i = 0; i < XCH; ++i) {
                    const int c = lane + 32 * i;
                    if (c < nch) {
                        u[2 * i] = xr[2 * c];
                        u[2 * i + 1] = xr[2 * c + 1];
                    }
                }
            } else if (mine) {
                // the h row, once all of the expert's phase-1 items are counted
                const uint32_t target = (uint32_t)per1 * COUNT_PER_ITEM + a.phase2_bias;
                int hok = 1;
                if (lane == 0 && !counts_expired) {
                    uint32_t i = 0;
                    while (ld_acquire(a.done13 + f.e) < target) {
                        if (++i > a.wait_limit) {
                            hok = 0;
                            break;
                        }
                        __nanosleep(64);
                    }
                }
                if (!__shfl_sync(0xffffffffu, hok, 0)) {
                    // the tile is built from h as it is, and this warp waits for no later count
                    if (lane == 0) atomicOr(a.status, PQE_STATUS_TIMEOUT);
                    counts_expired = true;
                }
                const int nch = I / 16;
                const float4 *hr = reinterpret_cast<const float4 *>(a.h + (size_t)(f.p0 + aw) * I);
#pragma unroll
                for (int i = 0; i < HCH; ++i) {
                    const int c = lane + 32 * i;
                    if (c < nch) {
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            const float4 v = __ldcg(hr + 4 * c + b);
                            u[4 * i + b] = make_uint4(__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z),
                                                      __float_as_uint(v.w));
                        }
                    }
                }
            }
            if (lane == 0) ok = wait_bar(bar_aempty + 8 * buf, ((uint32_t)(q >> 1) & 1u) ^ 1u, a.wait_limit);
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                timed_out = true;
                break;
            }
            uint8_t *tile = smem + g.act_off + (size_t)buf * g.act_bytes;
            if (!f.valid) {
                if (aw == 0 && lane == 0) atomicOr(a.status, PQE_STATUS_BAD_PAGE);
            } else if (mine) {
                const int t = aw;
                const bool p1 = f.phase == 1;
                float amax = 0.0f;
#pragma unroll
                for (int i = 0; i < 2 * XCH; ++i) {
                    const uint32_t w4[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
#pragma unroll
                    for (int b = 0; b < 4; ++b)
                        amax = p1 ? fmaxf(amax, fmaxf(fabsf(bf16_lo(w4[b])), fabsf(bf16_hi(w4[b]))))
                                  : fmaxf(amax, fabsf(__uint_as_float(w4[b])));
                }
                const float r = act_factor(warp_max(amax));
                if (lane == 0) s_ts[buf * NTOK + t] = 1.0f / r;
                if (p1) {
                    const int nch = H / 16;
#pragma unroll
                    for (int i = 0; i < XCH; ++i) {
                        const int c = lane + 32 * i;
                        if (c < nch) {
                            const uint32_t w8[8] = {u[2 * i].x,     u[2 * i].y,     u[2 * i].z,     u[2 * i].w,
                                                    u[2 * i + 1].x, u[2 * i + 1].y, u[2 * i + 1].z, u[2 * i + 1].w};
                            float v[16];
#pragma unroll
                            for (int b = 0; b < 8; ++b) {
                                v[2 * b] = bf16_lo(w8[b]) * r;
                                v[2 * b + 1] = bf16_hi(w8[b]) * r;
                            }
                            uint4 hi, lo;
                            split16(v, hi, lo);
                            uint8_t *st = tile + (size_t)(c >> 3) * ACT_STEP;
                            *reinterpret_cast<uint4 *>(st + act_chunk(t, c & 7)) = hi;
                            *reinterpret_cast<uint4 *>(st + act_chunk(NTOK + t, c & 7)) = lo;
                        }
                    }
                } else {
                    const int nch = I / 16;
#pragma unroll
                    for (int i = 0; i < HCH; ++i) {
                        const int c = lane + 32 * i;
                        if (c < nch) {
                            float v[16];
#pragma unroll
                            for (int b = 0; b < 4; ++b) {
                                v[4 * b] = __uint_as_float(u[4 * i + b].x) * r;
                                v[4 * b + 1] = __uint_as_float(u[4 * i + b].y) * r;
                                v[4 * b + 2] = __uint_as_float(u[4 * i + b].z) * r;
                                v[4 * b + 3] = __uint_as_float(u[4 * i + b].w) * r;
                            }
                            uint4 hi, lo;
                            split16(v, hi, lo);
                            uint8_t *st = tile + (size_t)(c >> 3) * ACT_STEP;
                            *reinterpret_cast<uint4 *>(st + act_chunk(t, c & 7)) = hi;
                            *reinterpret_cast<uint4 *>(st + act_chunk(NTOK + t, c & 7)) = lo;
                        }
                    }
                }
            }
            // the generic-proxy writes become visible to the MMAs (async proxy)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive_plain(bar_afull + 8 * buf);
        }
        if (timed_out && lane == 0) atomicOr(a.status, PQE_STATUS_TIMEOUT);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == W_MMA) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

// 3-D [slots, rows, cols] uint8 with a slot stride, box [1, 64, 128], 128-byte swizzle
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load(std::memory_order_relaxed);
    if (!f) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            f = reinterpret_cast<EncodeTiledFn>(p);
            fn.store(f, std::memory_order_relaxed);
        }
    }
    return f;
}

static bool map_rows64(CUtensorMap *m, const void *base, uint64_t slots, uint64_t rows, uint64_t cols,
                       uint64_t slot_stride) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[3] = {cols, rows, slots};
    cuuint64_t strides[2] = {cols, slot_stride};
    cuuint32_t box[3] = {(cuuint32_t)KSTEP, 64, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// shared memory of one CTA; a step of T <= NTOK tokens (k per token) stages
// all of x and perm_src once, so that the phase-1 tiles are built on chip
static bool geometry(int H, int I, int T, int k, Geo &g) {
    if (H / 16 > 32 * XCH || I / 16 > 32 * HCH) return false;  // a row's chunks per activation lane
    const int kmax = (H > I ? H : I) / KSTEP;
    g.act_bytes = (uint32_t)kmax * ACT_STEP;
    const uint32_t xb = 2u * 64 * NTOK * 4, ts = 2u * NTOK * 4;
    const uint32_t qb = (uint32_t)round_up(sizeof(Grab) * QN, 16);
    const uint32_t bars = 8u * (2 * MAX_STAGES + 9 + 2 * QN);
    const uint32_t tail = 16;
    g.xs_bytes = (T >= 1 && T <= NTOK) ? (uint32_t)round_up((size_t)T * H * 2 + (size_t)T * k * 4, 16) : 0u;
    const uint32_t fixed = 2 * g.act_bytes + xb + ts + qb + g.xs_bytes + bars + tail;
    const uint32_t budget = 227 * 1024 - 1024;  // less the alignment slack
    if (fixed + MIN_STAGES * STAGE_BYTES > budget) return false;
    int stages = (int)((budget - fixed) / STAGE_BYTES);
    if (stages > MAX_STAGES) stages = MAX_STAGES;
    g.stages = stages;
    g.act_off = (uint32_t)stages * STAGE_BYTES;
    g.xb_off = g.act_off + 2 * g.act_bytes;
    g.ts_off = g.xb_off + xb;
    g.q_off = g.ts_off + ts;
    g.xs_off = g.q_off + qb;
    g.bar_off = g.xs_off + g.xs_bytes;
    g.tmem_off = g.bar_off + bars;
    g.smem_bytes = g.tmem_off + tail + 1024;
    return true;
}

}  // namespace sw

bool stream_tc_shape_ok(int H, int I) {
    sw::Geo g;
    return tc_shape_ok(H, I) && stream_shape_ok(H, I) && sw::geometry(H, I, 0, 1, g);
}

int launch_ffn_stream_tc(const FfnArgs &args, cudaStream_t s, int grid) {
    using namespace sw;
    Geo g;
    if (args.expert_fmt != nullptr || !tc_shape_ok(args.H, args.I) || !geometry(args.H, args.I, args.T, args.k, g))
        return PQE_ERR_UNSUPPORTED;
    const int H = args.H, I = args.I;
    const PageLayout L = fp8_layout(H, I);
    // the working-buffer / cache maps need a non-empty region to encode; an
    // absent region gets a one-slot map over the other base (never selected)
    const uint8_t *cache = args.n_slots ? args.pool_base : args.wb_base;
    const uint8_t *wb = args.n_wb ? args.wb_base : args.pool_base;
    const uint64_t ns = args.n_slots ? args.n_slots : 1, nw = args.n_wb ? args.n_wb : 1;
    CUtensorMap m13c, m13w, m2c, m2w;
    if (!(map_rows64(&m13c, cache + L.w13, ns, 2 * (uint64_t)I, H, args.slot_stride) &&
          map_rows64(&m13w, wb + L.w13, nw, 2 * (uint64_t)I, H, args.slot_stride) &&
          map_rows64(&m2c, cache + L.w2, ns, (uint64_t)H, I, args.slot_stride) &&
          map_rows64(&m2w, wb + L.w2, nw, (uint64_t)H, I, args.slot_stride)))
        return PQE_ERR_UNSUPPORTED;
    static std::atomic<uint32_t> smem_set[PQE_MAX_DEVICES];
    int dev = 0, sms = 0;
    const int di = device_info(dev, sms);
    if (di != PQE_OK) return di;
    if (g.smem_bytes > smem_set[dev].load(std::memory_order_relaxed)) {
        PQE_CUDA_TRY(cudaFuncSetAttribute(ffn_stream_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)g.smem_bytes));
        smem_set[dev].store(g.smem_bytes, std::memory_order_relaxed);
    }
    // cooperative: all CTAs resident at once (phase 2 of an expert waits for
    // phase-1 items of other CTAs); the attribute also holds in a captured graph
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid > 0 && grid < sms ? grid : sms);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = g.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    PQE_CUDA_TRY(cudaLaunchKernelEx(&cfg, ffn_stream_tc_kernel, m13c, m13w, m2c, m2w, args, g));
    count_launch();
    return PQE_OK;
}

}  // namespace pqe
