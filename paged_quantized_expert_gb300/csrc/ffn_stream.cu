// ffn_stream.cu -- expert FFN for small per-expert batches (decode): a
// persistent, bulk-copy-fed weight stream.
//
// The weights of a routed expert are read once from its slot (expert-pager
// article, rand.pepabo.com, "エキスパート重みの階層ページング"); for a handful of
// tokens per expert the layer is bound by that stream from HBM. One CTA per SM
// (cooperative launch), twelve warps: three producers, one combiner, eight
// consumers.
//
// Producers (warps 0-2): their lanes pull the weight rows of a unit (8 gate/up
// row pairs of w13, or 64 rows of w2, plus their scales) into a ring of
// shared-memory stages with one cp.async.bulk per row (2 KB pieces of w2),
// completing on an mbarrier transaction count. A single warp issuing a stage's
// 2 KB copies reaches about 5.1 TB/s on GB300; several warps sharing them
// reach 7 TB/s and more, above a device-to-device copy. Rows land with a small
// pad so that the consumers' fragment loads are free of bank conflicts.
//
// Consumers (warps 4-11) multiply with mma.sync m16n8k16 (f16 inputs, fp32
// accumulate): 16 weight rows are the M side and up to 8 tokens the N side.
// FP8 E4M3 weights convert exactly to f16 (one cvt per two weights); E2M1
// weights too, with their E8M0 block scale applied to each 32-column block's
// partial sum. Activations (bf16 x, fp32 h) are brought to f16 with a
// power-of-two factor per token and per warp slice of K, so products of bf16 x
// are exact (h is rounded to 11 bits) and all sums are fp32. Inside a warp's
// slice the K order is permuted identically for weights and activations, which
// a dot product allows: each lane reads contiguous weight bytes of its rows.
// Phase 1 (w13 + SwiGLU -> h): the 8 warps split K of a 16-row unit. Phase 2
// (w2 -> out_perm): warp w takes 16 of the unit's 64 rows and half of K. Each
// warp hands its partial sums, already multiplied by the rows' scales and the
// tokens' factors (both linear), to a ring of four shared-memory slots.
//
// The combiner (warp 3) reads the slots in the same (unit, token group) order,
// adds the partials and applies SwiGLU (phase 1) or pairs the K halves (phase
// 2), and stores h / out_perm. A consumer waits only when the combiner is four
// steps behind, never for the other consumers.
//
// Each CTA takes a contiguous range of units holding an equal share of the
// work, weighting each expert by its bytes and token groups. Phase 2 of an
// expert starts once all of its phase-1 work (in any CTA) is counted complete,
// which each CTA's combiner publishes per expert: no grid-wide barrier, and
// the producers keep streaming, so phase-2 weights are in flight meanwhile.
// Every wait is bounded: on expiry PQE_STATUS_TIMEOUT is set and the waiter
// moves on.
#include "ffn_internal.cuh"
#include "pqe_common.cuh"

namespace pqe {
namespace st {

constexpr int CONS = 8;                   // consumer warps
constexpr int PROD = 3;                   // producer warps 0 .. PROD-1
constexpr int COMB = PROD;                // the combiner warp
constexpr int CONS0 = PROD + 1;           // first consumer warp
constexpr int THREADS = 32 * (CONS + PROD + 1);
constexpr int RSLOTS = 4;                 // partial-sum slots between the consumers and the combiner
constexpr int MAX_STAGES = 4;
constexpr int PAIRS = 8;                  // w13 gate/up row pairs per unit (16 weight rows)
constexpr int ROWS2 = 64;                 // w2 rows per unit
constexpr int NT = 8;                     // tokens per mma column group
constexpr int NCH_MAX = 5;                // 64-column chunks of K a warp holds at most (H <= 2560, I <= 640)

// shared-memory pitch of a weight row of `len` bytes: FP8 rows are read as
// 16-byte pieces (pitch = 64 mod 128), E2M1 rows as 4-byte pieces (pitch = 16
// mod 128); either way a warp's loads fall on distinct banks
__host__ __device__ inline uint32_t pitch8(int len) { return (uint32_t)round_up((size_t)len, 128) + 64; }
__host__ __device__ inline uint32_t pitch4(int len) { return (uint32_t)round_up((size_t)len, 128) + 16; }
// w2 units land as 2-KiB-class pieces (single-row copies of I bytes stream
// poorly): FP8 as 16 pieces of 4 rows, E2M1 as 8 pieces of 8 rows, each piece
// padded like a row above. An mma row then takes one row from each piece:
// FP8 m-tile mt, mma row g <- unit row 4g + mt; E2M1 m-tile mt, mma rows g and
// g+8 <- unit rows 8g + 2mt and 8g + 2mt + 1.
__host__ __device__ inline uint32_t piece8(int I) { return pitch8(4 * I); }
__host__ __device__ inline uint32_t piece4(int I) { return pitch4(4 * I); }

struct Geo {
    int stages;
    uint32_t stage_bytes;  // multiple of 128
    uint32_t red_off, sched_off, bar_off, smem_bytes;
    uint32_t info_off;  // ExpertInfo array, in int32 words after the work-weight prefix
};

// per active expert, staged in shared memory once per launch
struct ExpertInfo {
    int e, p0, n, slot, fmt, valid;
};

// position in the stage ring: stage s and the parity of its current fill
struct RingPos {
    int s = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void next(int stages) {
        if (++s == stages) {
            s = 0;
            ph ^= 1u;
        }
    }
};

// position in a range of units: schedule entry ea and unit rb of its `per`
// (one division at the start, none per unit)
struct UnitPos {
    int ea, rb;
    __device__ __forceinline__ UnitPos(int u, int per) : ea(u / per), rb(u % per) {}
    __device__ __forceinline__ void next(int per) {
        if (++rb == per) {
            rb = 0;
            ++ea;
        }
    }
    __device__ __forceinline__ void prev(int per) {
        if (rb-- == 0) {
            rb = per - 1;
            --ea;
        }
    }
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, "
            "p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if (i > 16) __nanosleep(64);
    }
    return false;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// two E4M3 codes (low / high 16 bits of w) -> f16x2, exact
__device__ __forceinline__ uint32_t f16x2_e4m3_lo(uint32_t w) {
    uint32_t r;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t}" : "=r"(r) : "r"(w));
    return r;
}
__device__ __forceinline__ uint32_t f16x2_e4m3_hi(uint32_t w) {
    uint32_t r;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h;\n\t}" : "=r"(r) : "r"(w));
    return r;
}

// four bytes of E2M1 pairs -> four f16x2 (byte i -> d[i], low nibble in the low half), exact
__device__ __forceinline__ void f16x2_e2m1x4(uint32_t w, uint32_t (&d)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\tcvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(w));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// D[16 x 8] += A[16 x 16] . B[16 x 8], f16 inputs, fp32 accumulate. Lane (g, c):
// a0/a2 = row g, k pairs (2c, 2c+1) / (2c+8, 2c+9); a1/a3 = row g+8, same k;
// b0/b1 = column g, same k as a0/a2; d = rows g, g+8 x columns 2c, 2c+1.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// power of two s with amax * s in [2^14, 2^15) (inside f16's range), and 1/s
__device__ __forceinline__ void pow2_scale(float amax, float &s, float &inv) {
    int sh = 14 - ((int)((__float_as_uint(amax) >> 23) & 0xffu) - 127);
    if (amax == 0.0f) sh = 0;
    sh = max(-126, min(126, sh));
    s = __uint_as_float((uint32_t)(127 + sh) << 23);
    inv = __uint_as_float((uint32_t)(127 - sh) << 23);
}

// Activation fragments of one token group for a warp's K slice (chunks c0 ..
// c0+nch-1 of 64 columns): lane (g, c) holds token g; v[j][i] is its column
// pair i of chunk j as f16x2. Column order inside a chunk: for FP8 weights lane
// c takes columns 16c .. 16c+15; for E2M1 weights columns 8c .. 8c+7 of each of
// the chunk's two 32-column blocks.
template <int NCH>
struct BFrag {
    uint32_t v[NCH][8];
};

// Column offset (elements) of piece q (0..1 for bf16 x as 8-element pieces,
// 0..3 for fp32 h as 4-element pieces) of chunk `ch` for lane c.
__device__ __forceinline__ int bf16_piece(int ch, int q, int c, bool fp8map) {
    const int base = 64 * ch;
    return fp8map ? base + 16 * c + 8 * q : base + 32 * q + 8 * c;
}
__device__ __forceinline__ int f32_piece(int ch, int q, int c, bool fp8map) {
    const int base = 64 * ch;
    return fp8map ? base + 16 * c + 4 * q : base + (q >> 1) * 32 + 8 * c + 4 * (q & 1);
}

// The token's amax over the warp slice (its four lanes hold it). With amax in
// [2^-4, 2^15) the values convert with factor 1: bf16 x is then exact in f16
// down to amax * 2^-10 and below that off by at most 2^-25 absolute, far
// inside the tolerance; only other amax take a second, scaled pass.
__device__ __forceinline__ bool unit_factor_ok(float amax) {
    return amax == 0.0f || (amax >= 0.0625f && amax < 32768.0f);
}

__device__ __forceinline__ float token_amax(float amax) {
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    return fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
}

// from a bf16 row (x); row == nullptr -> zeros. inv = 1/s of this lane's token.
template <int NCH>
__device__ __forceinline__ void load_bfrag_bf16(const uint16_t *row, int c0, int nch, int c, bool fp8map, BFrag<NCH> &b,
                                                float &inv) {
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (j < nch && row != nullptr)
                v = __ldg(reinterpret_cast<const uint4 *>(row + bf16_piece(c0 + j, q, c, fp8map)));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xffff0000u);
                amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
                b.v[j][4 * q + i] = pack_f16x2(lo, hi);
            }
        }
    }
    amax = token_amax(amax);
    inv = 1.0f;
    if (unit_factor_ok(amax)) return;
    float s;
    pow2_scale(amax, s, inv);
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            if (j < nch && row != nullptr) {
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(row + bf16_piece(c0 + j, q, c, fp8map)));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    b.v[j][4 * q + i] =
                        pack_f16x2(__uint_as_float(w[i] << 16) * s, __uint_as_float(w[i] & 0xffff0000u) * s);
            }
        }
    }
}

// from an fp32 row (h, written earlier in this launch by other CTAs: read at L2)
template <int NCH>
__device__ __forceinline__ void load_bfrag_f32(const float *row, int c0, int nch, int c, bool fp8map, BFrag<NCH> &b,
                                               float &inv) {
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j < nch && row != nullptr)
                v = __ldcg(reinterpret_cast<const float4 *>(row + f32_piece(c0 + j, q, c, fp8map)));
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
            b.v[j][2 * q] = pack_f16x2(v.x, v.y);
            b.v[j][2 * q + 1] = pack_f16x2(v.z, v.w);
        }
    }
    amax = token_amax(amax);
    inv = 1.0f;
    if (unit_factor_ok(amax)) return;
    float s;
    pow2_scale(amax, s, inv);
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (j < nch && row != nullptr) {
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(row + f32_piece(c0 + j, q, c, fp8map)));
                b.v[j][2 * q] = pack_f16x2(v.x * s, v.y * s);
                b.v[j][2 * q + 1] = pack_f16x2(v.z * s, v.w * s);
            }
        }
    }
}

// acc[mma rows g, g+8 x tokens 2c, 2c+1] += W . B over the warp's chunks.
// FP8: mma row g at rows + g * pitch, row g+8 `off8` bytes after it; lane c
// reads bytes 16c .. 16c+15 of each chunk.
// one 64-column chunk of FP8 rows: pa = row g's 16 bytes of the chunk for lane c
template <int NCH>
__device__ __forceinline__ void mma_chunk_fp8(const uint8_t *pa, uint32_t off8, const uint32_t (&bv)[8],
                                              float (&part)[4][4]) {
    const uint4 wa = *reinterpret_cast<const uint4 *>(pa);
    const uint4 wb = *reinterpret_cast<const uint4 *>(pa + off8);
    const uint32_t ua[4] = {wa.x, wa.y, wa.z, wa.w}, ub[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
        mma_f16(part[q], f16x2_e4m3_lo(ua[q]), f16x2_e4m3_lo(ub[q]), f16x2_e4m3_hi(ua[q]), f16x2_e4m3_hi(ub[q]),
                bv[2 * q], bv[2 * q + 1]);
}

template <int NCH>
__device__ __forceinline__ void mma_rows_fp8(const uint8_t *rows, uint32_t pitch, uint32_t off8, int c0, int nch,
                                             int g, int c, const BFrag<NCH> &b, float (&acc)[4]) {
    // four independent accumulator chains (one per k-step of a chunk)
    float part[4][4] = {};
    const uint8_t *base = rows + (size_t)g * pitch + 64 * c0 + 16 * c;
    if (nch == NCH) {  // every warp's slice on the standard shapes: no per-chunk guard
#pragma unroll
        for (int j = 0; j < NCH; ++j) mma_chunk_fp8<NCH>(base + 64 * j, off8, b.v[j], part);
    } else {
#pragma unroll
        for (int j = 0; j < NCH; ++j)
            if (j < nch) mma_chunk_fp8<NCH>(base + 64 * j, off8, b.v[j], part);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] += (part[0][i] + part[1][i]) + (part[2][i] + part[3][i]);
}

// E2M1: rows placed as for FP8; lane c reads bytes 4c .. 4c+3 of each 16-byte
// (32-column) block. E8M0 scales of mma row g at scales + g * spitch, of row
// g+8 `soff8` bytes after them, one byte per block.
// one 64-column chunk (two 32-column blocks) of E2M1 rows; pa = row g's bytes
// of the chunk for lane c, sc = row g's scale of the chunk's first block
template <int NCH>
__device__ __forceinline__ void mma_chunk_fp4(const uint8_t *pa, uint32_t off8, const uint8_t *sc, int soff8,
                                              const uint32_t (&bv)[8], float (&acc)[4]) {
#pragma unroll
    for (int lb = 0; lb < 2; ++lb) {
        uint32_t fa[4], fb[4];
        f16x2_e2m1x4(*reinterpret_cast<const uint32_t *>(pa + 16 * lb), fa);
        f16x2_e2m1x4(*reinterpret_cast<const uint32_t *>(pa + 16 * lb + off8), fb);
        float t[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f16(t, fa[0], fb[0], fa[1], fb[1], bv[4 * lb], bv[4 * lb + 1]);
        mma_f16(t, fa[2], fb[2], fa[3], fb[3], bv[4 * lb + 2], bv[4 * lb + 3]);
        const float sa = e8m0_to_f32(sc[lb]);
        const float sb = e8m0_to_f32(sc[soff8 + lb]);
        acc[0] = __fmaf_rn(sa, t[0], acc[0]);
        acc[1] = __fmaf_rn(sa, t[1], acc[1]);
        acc[2] = __fmaf_rn(sb, t[2], acc[2]);
        acc[3] = __fmaf_rn(sb, t[3], acc[3]);
    }
}

template <int NCH>
__device__ __forceinline__ void mma_rows_fp4(const uint8_t *rows, uint32_t pitch, uint32_t off8,
                                             const uint8_t *scales, int spitch, int soff8, int c0, int nch, int g,
                                             int c, const BFrag<NCH> &b, float (&acc)[4]) {
    const uint8_t *base = rows + (size_t)g * pitch + 32 * c0 + 4 * c;
    const uint8_t *sbase = scales + (size_t)g * spitch + 2 * c0;
    if (nch == NCH) {  // every warp's slice on the standard shapes: no per-chunk guard
#pragma unroll
        for (int j = 0; j < NCH; ++j) mma_chunk_fp4<NCH>(base + 32 * j, off8, sbase + 2 * j, soff8, b.v[j], acc);
    } else {
#pragma unroll
        for (int j = 0; j < NCH; ++j)
            if (j < nch) mma_chunk_fp4<NCH>(base + 32 * j, off8, sbase + 2 * j, soff8, b.v[j], acc);
    }
}

// Units of the expert list in expert-major order, each expert's units weighted
// by its work weight w_a = wpre[a+1] - wpre[a]; unit_at maps a position of the
// weighted line (0 .. wpre[n]*per) to the first unit at or after it.
__device__ __forceinline__ int unit_at(const int32_t *wpre, int n, int per, long pos) {
    if (n == 0 || pos >= (long)wpre[n] * per) return n * per;
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long)wpre[mid] * per <= pos) lo = mid;
        else hi = mid - 1;
    }
    const long w = wpre[lo + 1] - wpre[lo];
    long off = (pos - (long)wpre[lo] * per + w - 1) / w;
    if (off > per) off = per;
    return lo * per + (int)off;
}

// CTA blockIdx.x's units: an equal share of the weighted work, contiguous
__device__ __forceinline__ void unit_range(const int32_t *wpre, int n, int per, int &u0, int &u1) {
    const long total = (n > 0 ? (long)wpre[n] : 0) * per;
    u0 = unit_at(wpre, n, per, total * blockIdx.x / gridDim.x);
    u1 = unit_at(wpre, n, per, total * (blockIdx.x + 1) / gridDim.x);
}

template <int NCH>
__global__ void __launch_bounds__(THREADS, 1) ffn_stream_kernel(const FfnArgs a, const Geo g) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int H = a.H, I = a.I;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + g.bar_off, bar_empty = bar_full + 8 * g.stages;
    const PageLayout L8 = fp8_layout(H, I), L4 = mxfp4_layout(H, I);
    // row pitches of the four stage layouts
    const uint32_t p13_8 = pitch8(H), p13_4 = pitch4(H / 2), q2_8 = piece8(I), q2_4 = piece4(I);
    // the expert list, its work-weight prefix and each expert's batch and page,
    // loaded once by all threads in parallel (no dependent global loads later)
    const int n_act = __ldg(a.sched);
    int32_t *s_wpre = reinterpret_cast<int32_t *>(smem + g.sched_off);  // [n_act + 1]
    ExpertInfo *s_info = reinterpret_cast<ExpertInfo *>(s_wpre + g.info_off);  // [n_act]
    for (int i = threadIdx.x; i <= n_act; i += THREADS) s_wpre[i] = __ldg(a.wpre + i);
    for (int i = threadIdx.x; i < n_act; i += THREADS) {
        const int4 r = __ldg(a.info + i);  // the schedule's record: expert, batch, page
        ExpertInfo f;
        f.e = r.x;
        f.p0 = r.y;
        f.n = r.z;
        f.slot = info_slot(r.w);
        f.fmt = info_fmt(r.w);
        f.valid = f.slot >= 0 && f.slot < a.n_slots + a.n_wb && (f.fmt == PQE_FMT_FP8 || f.fmt == PQE_FMT_MXFP4);
        s_info[i] = f;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < g.stages; ++s) {
            mbar_init(bar_full + 8 * s, PROD);
            mbar_init(bar_empty + 8 * s, CONS);
        }
        // partial-sum slots: rfull[i] takes every consumer lane's arrival, rfree[i] the combiner's lanes
        const uint32_t rb = bar_empty + 8 * g.stages;
        for (int i = 0; i < RSLOTS; ++i) {
            mbar_init(rb + 8 * i, CONS * 32);
            mbar_init(rb + 8 * (RSLOTS + i), 32);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int per13 = I / PAIRS, per2 = H / ROWS2;
    int u13a, u13b, u2a, u2b;
    unit_range(s_wpre, n_act, per13, u13a, u13b);
    unit_range(s_wpre, n_act, per2, u2a, u2b);

    if (warp < PROD) {
        // ---------------- producers: one bulk copy per weight row ----------------
        // copy c of a unit is issued by warp c % PROD, lane c / PROD: the copies of
        // a stage leave from several warps at once, which a single warp's lanes
        // cannot match (one warp's bulk copies are accepted one after another).
        // Each warp posts the bytes of its own copies on the stage's barrier.
        int it = 0;
        RingPos rp;
        bool ok = true;
        const int c = warp + PROD * lane;
        for (int phase = 1; phase <= 2 && ok; ++phase) {
            const int ua = phase == 1 ? u13a : u2a, ub = phase == 1 ? u13b : u2b;
            const int per = phase == 1 ? per13 : per2;
            // phase 2 runs backwards (see the consumers)
            const bool fwd = phase == 1;
            UnitPos up(fwd ? ua : ub - 1, per);
            for (int i = ua; i < ub; ++i, ++it, rp.next(g.stages), fwd ? up.next(per) : up.prev(per)) {
                const int s = rp.s;
                int w_ok = 1;
                if (lane == 0) w_ok = mbar_wait(bar_empty + 8 * s, rp.ph ^ 1u, a.wait_limit) ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
                    ok = false;
                    break;
                }
                const ExpertInfo f = s_info[up.ea];
                const int rb = up.rb;
                const uint32_t dst = sbase + (uint32_t)s * g.stage_bytes;
                const uint32_t fb = bar_full + 8 * s;
                if (!f.valid) {
                    if (lane == 0) mbar_arrive(fb);  // no data: consumers write zeros
                    continue;
                }
                const uint8_t *page = page_addr(a, f.slot);
                const bool fp8 = f.fmt == PQE_FMT_FP8;
                const uint8_t *src = nullptr;
                uint32_t doff = 0, bytes = 0;
                if (phase == 1) {
                    // copies 0..7: gate rows rb*8 .. +7; 8..15: the matching up rows;
                    // 16, 17: the gate and the up rows' scales (FP8 8 fp32 each, E2M1 [8][H/32] E8M0)
                    const uint32_t rowb = fp8 ? (uint32_t)H : (uint32_t)H / 2, pitch = fp8 ? p13_8 : p13_4;
                    const uint32_t scb = fp8 ? 4u * PAIRS : (uint32_t)PAIRS * (H / 32);
                    const size_t scrow = fp8 ? 4 : (size_t)(H / 32);
                    if (c < 2 * PAIRS) {
                        const size_t wr = c < PAIRS ? (size_t)rb * PAIRS + c : (size_t)I + rb * PAIRS + (c - PAIRS);
                        src = page + (fp8 ? L8.w13 : L4.w13) + wr * rowb;
                        doff = (uint32_t)c * pitch;
                        bytes = rowb;
                    } else if (c < 2 * PAIRS + 2) {
                        const int hf = c - 2 * PAIRS;
                        const size_t sr = (size_t)(hf ? I : 0) + (size_t)rb * PAIRS;
                        src = page + (fp8 ? L8.s13 : L4.s13) + sr * scrow;
                        doff = 2 * PAIRS * pitch + (uint32_t)hf * scb;
                        bytes = scb;
                    }
                } else {
                    // pieces of 4 (FP8) or 8 (E2M1) contiguous rows, 4*I bytes each; then the scales
                    const int np = fp8 ? 16 : 8;
                    const uint32_t pb = 4u * I, pitch = fp8 ? q2_8 : q2_4;
                    const uint32_t scb = fp8 ? 4u * ROWS2 : (uint32_t)ROWS2 * (I / 32);
                    const uint8_t *w2 = page + (fp8 ? L8.w2 : L4.w2) + (size_t)rb * ROWS2 * (fp8 ? I : I / 2);
                    if (c < np) {
                        src = w2 + (size_t)c * pb;
                        doff = (uint32_t)c * pitch;
                        bytes = pb;
                    } else if (c == np) {
                        src = page + (fp8 ? L8.s2 + (size_t)rb * ROWS2 * 4 : L4.s2 + (size_t)rb * ROWS2 * (I / 32));
                        doff = (uint32_t)np * pitch;
                        bytes = scb;
                    }
                }
                const uint32_t tot = __reduce_add_sync(0xffffffffu, bytes);
                if (lane == 0) mbar_expect_tx(fb, tot);
                __syncwarp();
                if (bytes) bulk_g2s(dst + doff, src, bytes, fb);
            }
        }
        if (lane == 0) {
            if (!ok) atomicOr(a.status, PQE_STATUS_TIMEOUT);
            // the copies issued last have landed before the CTA may exit
            for (int j = (it > g.stages ? it - g.stages : 0); j < it; ++j)
                mbar_wait(bar_full + 8 * (j % g.stages), (uint32_t)(j / g.stages) & 1u, a.wait_limit);
        }
        return;  // the producer warps take no part in the consumer barriers
    }

    const uint32_t rfull = bar_empty + 8 * g.stages, rfree = rfull + 8 * RSLOTS;
    float4 *red = reinterpret_cast<float4 *>(smem + g.red_off);  // [RSLOTS][CONS][32] partial sums
    const int gq = lane >> 2, cq = lane & 3;                      // mma fragment coordinates

    if (warp == COMB) {
        // ---------------- combiner: partial sums -> h, out_perm ----------------
        // takes the (unit, token group) steps in the consumers' order; slot rc % RSLOTS
        int rc = 0;
        bool timed_out = false;
        // phase 1: lane (gq, cq) holds gate row j = rb*8 + gq and up row j for tokens 2cq, 2cq+1.
        // Once this CTA's units of an expert are combined, their count is published
        // (after the h stores are visible); phase 2 of the expert waits for the
        // counts of all CTAs (done13), not for the whole grid
        UnitPos up1(u13a, per13);
        int run = 0;  // units of the current expert combined here
        for (int u = u13a; u < u13b; ++u, up1.next(per13)) {
            const ExpertInfo f = s_info[up1.ea];
            const int j = up1.rb * PAIRS + gq;
            for (int tg = 0; tg < f.n; tg += NT, ++rc) {
                const int nt = min(NT, f.n - tg), sl = rc % RSLOTS;
                if (!timed_out && !mbar_wait(rfull + 8 * sl, (uint32_t)(rc / RSLOTS) & 1u, a.wait_limit)) timed_out = true;
                const float4 *rs = red + sl * CONS * 32;
                float4 v = rs[lane];
#pragma unroll
                for (int w = 1; w < CONS; ++w) {
                    const float4 t = rs[w * 32 + lane];
                    v.x += t.x;
                    v.y += t.y;
                    v.z += t.z;
                    v.w += t.w;
                }
                mbar_arrive(rfree + 8 * sl);
                const int t0 = 2 * cq;
                if (t0 < nt) a.h[(size_t)(f.p0 + tg + t0) * I + j] = silu(v.x) * v.z;
                if (t0 + 1 < nt) a.h[(size_t)(f.p0 + tg + t0 + 1) * I + j] = silu(v.y) * v.w;
            }
            ++run;
            if (u + 1 == u13b || up1.rb + 1 == per13) {
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(a.done13 + f.e, (uint32_t)(run * ((f.n + NT - 1) / NT)));
                run = 0;
            }
        }
        // phase 2: warps mt and mt + 4 hold the two K halves of m-tile mt
        UnitPos up2(u2b - 1, per2);
        for (int u = u2b - 1; u >= u2a; --u, up2.prev(per2)) {
            const ExpertInfo f = s_info[up2.ea];
            const int r0 = up2.rb * ROWS2;
            const bool fp8 = f.fmt == PQE_FMT_FP8;
            for (int tg = 0; tg < f.n; tg += NT, ++rc) {
                const int nt = min(NT, f.n - tg), sl = rc % RSLOTS;
                if (!timed_out && !mbar_wait(rfull + 8 * sl, (uint32_t)(rc / RSLOTS) & 1u, a.wait_limit)) timed_out = true;
                const float4 *rs = red + sl * CONS * 32;
                float4 v[4];
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    const float4 p = rs[mt * 32 + lane], q = rs[(mt + 4) * 32 + lane];
                    v[mt] = make_float4(p.x + q.x, p.y + q.y, p.z + q.z, p.w + q.w);
                }
                mbar_arrive(rfree + 8 * sl);
                const int t0 = 2 * cq;
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    // unit rows of mma rows gq and gq + 8 in m-tile mt
                    const int ra = fp8 ? 4 * gq + mt : 8 * gq + 2 * mt, rbw = fp8 ? ra + 32 : ra + 1;
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        if (t0 + i < nt) {
                            uint16_t *o = a.out_perm + (size_t)(f.p0 + tg + t0 + i) * H + r0;
                            o[ra] = f32_to_bf16_rn(i ? v[mt].y : v[mt].x);
                            o[rbw] = f32_to_bf16_rn(i ? v[mt].w : v[mt].z);
                        }
                    }
                }
            }
        }
        if (timed_out && lane == 0) atomicOr(a.status, PQE_STATUS_TIMEOUT);
        return;
    }

    // ---------------- consumers ----------------
    // each (unit, token group) step ends with this warp's partials, already
    // multiplied by the rows' scales and the tokens' activation factors, in slot
    // rc % RSLOTS; only a slot the combiner has not yet read makes a warp wait
    const int cw = warp - CONS0;
    RingPos rp;
    int rc = 0;
    bool timed_out = false;
    BFrag<NCH> bf;
    float inv = 1.0f;
    int b_a = -1, b_tg = -1;  // expert and token group bf holds
    int f_a = -1;             // schedule entry f holds
    ExpertInfo f{};
    // the activation factors of this lane's output tokens 2cq, 2cq+1 (they sit in
    // lanes 8cq, 8cq+4 of the fragment), taken when the fragment is loaded
    float i0 = 1.0f, i1 = 1.0f;
    auto take_factors = [&]() {
        i0 = __shfl_sync(0xffffffffu, inv, 8 * cq);
        i1 = __shfl_sync(0xffffffffu, inv, 8 * cq + 4);
    };
    auto hand_off = [&](float s_lo, float s_hi, const float (&acc)[4]) {
        const int sl = rc % RSLOTS;
        if (!timed_out && !mbar_wait(rfree + 8 * sl, ((uint32_t)(rc / RSLOTS) & 1u) ^ 1u, a.wait_limit)) timed_out = true;
        red[(sl * CONS + cw) * 32 + lane] =
            make_float4(acc[0] * i0 * s_lo, acc[1] * i1 * s_lo, acc[2] * i0 * s_hi, acc[3] * i1 * s_hi);
        mbar_arrive(rfull + 8 * sl);
        ++rc;
    };

    // ---- phase 1: gate_j . x_t and up_j . x_t over this warp's chunks [c0, c0 + nch) of K
    {
        const int NC = H / 64, c0 = cw * NC / CONS, nch = (cw + 1) * NC / CONS - c0;
        UnitPos up(u13a, per13);
        for (int u = u13a; u < u13b; ++u, rp.next(g.stages), up.next(per13)) {
            const int s = rp.s;
            const int ua = up.ea;
            if (ua != f_a) {  // the schedule entry changes only at expert boundaries
                f = s_info[ua];
                f_a = ua;
            }
            const int p0 = f.p0, n = f.n;
            const bool fp8 = f.fmt == PQE_FMT_FP8;
            bool valid = f.valid != 0 && !timed_out;
            if (!timed_out && !mbar_wait(bar_full + 8 * s, rp.ph, a.wait_limit)) {
                valid = false;
                timed_out = true;
            }
            const uint8_t *stg = smem + (size_t)s * g.stage_bytes;
            // this unit's row scales, read before the stage is handed back
            float sg = 1.0f, su = 1.0f;
            if (valid && fp8) {
                const float *s13 = reinterpret_cast<const float *>(stg + 2 * PAIRS * p13_8);
                sg = s13[gq];
                su = s13[PAIRS + gq];
            }
            for (int tg = 0; tg < n; tg += NT) {
                const int nt = min(NT, n - tg);
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                if (valid) {
                    if (b_a != ua || b_tg != tg) {
                        const uint16_t *row = nullptr;
                        if (gq < nt) row = a.x + (size_t)(__ldg(a.perm_src + p0 + tg + gq) / a.k) * H;
                        load_bfrag_bf16(row, c0, nch, cq, fp8, bf, inv);
                        take_factors();
                        b_a = ua;
                        b_tg = tg;
                    }
                    if (fp8) mma_rows_fp8(stg, p13_8, 8 * p13_8, c0, nch, gq, cq, bf, acc);
                    else
                        mma_rows_fp4(stg, p13_4, 8 * p13_4, stg + 2 * PAIRS * p13_4, H / 32, 8 * (H / 32), c0, nch, gq,
                                     cq, bf, acc);
                }
                if (tg + NT >= n) {  // last token group: this warp reads the stage no more
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_empty + 8 * s);
                }
                hand_off(sg, su, acc);
            }
        }
    }

    int ready_a = -1;  // expert whose h rows this warp has seen complete
    b_a = -1;
    b_tg = -1;

    // ---- phase 2: out_perm[p, r] = w2_r . h_p; warp cw: rows 16 mt .. 16 mt + 15 of the unit, half kh of K
    {
        const int mt = cw & 3, kh = cw >> 2;
        const int NC = I / 64, c0 = kh * NC / 2, nch = (kh + 1) * NC / 2 - c0;
        // backwards through this CTA's units: it starts with the expert it shares
        // with the next CTA, whose phase-1 share of it that CTA did first, and ends
        // with the one it shares with the previous CTA, whose share came last there
        UnitPos up(u2b - 1, per2);
        for (int u = u2b - 1; u >= u2a; --u, rp.next(g.stages), up.prev(per2)) {
            const int s = rp.s;
            const int ua = up.ea;
            if (ua != f_a) {  // the schedule entry changes only at expert boundaries
                f = s_info[ua];
                f_a = ua;
            }
            const int p0 = f.p0, n = f.n;
            const bool fp8 = f.fmt == PQE_FMT_FP8;
            bool valid = f.valid != 0 && !timed_out;
            if (!timed_out && !mbar_wait(bar_full + 8 * s, rp.ph, a.wait_limit)) {
                valid = false;
                timed_out = true;
            }
            const uint8_t *stg = smem + (size_t)s * g.stage_bytes;
            // unit rows of mma rows gq and gq + 8, and their scales, read before the stage is handed back
            const int ra = fp8 ? 4 * gq + mt : 8 * gq + 2 * mt, rbw = fp8 ? ra + 32 : ra + 1;
            float sa = 1.0f, sb = 1.0f;
            if (valid && fp8) {
                const float *s2 = reinterpret_cast<const float *>(stg + 16 * q2_8);
                sa = s2[ra];
                sb = s2[rbw];
            }
            for (int tg = 0; tg < n; tg += NT) {
                const int nt = min(NT, n - tg);
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                if (valid && ready_a != ua) {
                    // h of this expert: all per13 units x token groups combined (other CTAs included)
                    const uint32_t target = (uint32_t)per13 * (uint32_t)((n + NT - 1) / NT) + a.phase2_bias;
                    int ok = 1;
                    if (lane == 0 && !timed_out) {
                        uint32_t i = 0;
                        while (ld_acquire(a.done13 + f.e) < target) {
                            if (++i > a.wait_limit) {
                                ok = 0;
                                break;
                            }
                            __nanosleep(64);
                        }
                    }
                    if (!__shfl_sync(0xffffffffu, ok, 0)) timed_out = true;
                    ready_a = ua;
                }
                if (valid) {
                    if (b_a != ua || b_tg != tg) {
                        const float *row = gq < nt ? a.h + (size_t)(p0 + tg + gq) * I : nullptr;
                        load_bfrag_f32(row, c0, nch, cq, fp8, bf, inv);
                        take_factors();
                        b_a = ua;
                        b_tg = tg;
                    }
                    if (fp8) mma_rows_fp8(stg + (size_t)mt * I, q2_8, 8 * q2_8, c0, nch, gq, cq, bf, acc);
                    else
                        mma_rows_fp4(stg + (size_t)mt * I, q2_4, I / 2, stg + 8 * q2_4 + (size_t)2 * mt * (I / 32),
                                     8 * (I / 32), I / 32, c0, nch, gq, cq, bf, acc);
                }
                if (tg + NT >= n) {  // last token group: this warp reads the stage no more
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_empty + 8 * s);
                }
                hand_off(sa, sb, acc);
            }
            if (!valid && threadIdx.x == 32 * CONS0 && n > 0 && !timed_out) atomicOr(a.status, PQE_STATUS_BAD_PAGE);
        }
    }
    if (timed_out && lane == 0) atomicOr(a.status, PQE_STATUS_TIMEOUT);
}

// 64-column chunks a consumer warp holds: phase 1 splits H/64 over 8 warps, phase 2 I/64 over 2
static int chunks_per_warp(int H, int I) {
    const int c1 = (H / 64 + CONS - 1) / CONS, c2 = (I / 64 + 1) / 2;
    return c1 > c2 ? c1 : c2;
}

// shared memory of one CTA for experts E (the schedule area is sized by E)
static bool geometry(int H, int I, int E, Geo &g) {
    const uint32_t s13_8 = 2u * PAIRS * pitch8(H) + 8u * PAIRS;
    const uint32_t s13_4 = 2u * PAIRS * pitch4(H / 2) + 2u * PAIRS * (H / 32);
    const uint32_t s2_8 = 16u * piece8(I) + 4u * ROWS2;
    const uint32_t s2_4 = 8u * piece4(I) + (uint32_t)ROWS2 * (I / 32);
    uint32_t sb = s13_8;
    if (s13_4 > sb) sb = s13_4;
    if (s2_8 > sb) sb = s2_8;
    if (s2_4 > sb) sb = s2_4;
    sb = (sb + 127) / 128 * 128;
    const uint32_t redb = (uint32_t)RSLOTS * CONS * 32 * 16;
    g.info_off = (uint32_t)(E + 4);  // >= n_act + 1 prefix entries
    const uint32_t schedb = (uint32_t)round_up(4 * (size_t)g.info_off + sizeof(ExpertInfo) * (size_t)E, 128);
    const uint32_t budget = 227 * 1024 - 1024;
    const uint32_t fixed = redb + schedb + 256;
    if (fixed + 2 * sb > budget) return false;
    int stages = (int)((budget - fixed) / sb);
    if (stages > MAX_STAGES) stages = MAX_STAGES;
    g.stages = stages;
    g.stage_bytes = sb;
    g.red_off = stages * sb;
    g.sched_off = g.red_off + redb;
    g.bar_off = g.sched_off + schedb;
    g.smem_bytes = g.bar_off + 16 * stages + 16 * RSLOTS;
    return true;
}

}  // namespace st

bool stream_shape_ok(int H, int I) {
    st::Geo g;
    // phase 1: the 8 consumer warps split H/64 chunks; phase 2: two warps split I/64 chunks
    return H % st::ROWS2 == 0 && I % st::PAIRS == 0 && H % 64 == 0 && I % 64 == 0 &&
           st::chunks_per_warp(H, I) <= st::NCH_MAX && st::geometry(H, I, 1024, g);
}

int launch_ffn_stream(const FfnArgs &args, cudaStream_t s, int grid) {
    st::Geo g;
    if (!st::geometry(args.H, args.I, args.E, g)) return PQE_ERR_UNSUPPORTED;
    // the shared-memory opt-in is per device
    static uint32_t smem_set[PQE_MAX_DEVICES] = {};
    int dev = 0, sms = 0;
    const int di = device_info(dev, sms);
    if (di != PQE_OK) return di;
    if (g.smem_bytes > smem_set[dev]) {
        PQE_CUDA_TRY(cudaFuncSetAttribute(st::ffn_stream_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)g.smem_bytes));
        PQE_CUDA_TRY(cudaFuncSetAttribute(st::ffn_stream_kernel<5>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)g.smem_bytes));
        smem_set[dev] = g.smem_bytes;
    }
    // cooperative: all CTAs resident at once (phase 2 of an expert waits for
    // phase-1 work of other CTAs); the attribute also holds when the launch is
    // captured into a graph
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid > 0 && grid < sms ? grid : sms);
    cfg.blockDim = dim3(st::THREADS);
    cfg.dynamicSmemBytes = g.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (st::chunks_per_warp(args.H, args.I) <= 4) PQE_CUDA_TRY(cudaLaunchKernelEx(&cfg, st::ffn_stream_kernel<4>, args, g));
    else PQE_CUDA_TRY(cudaLaunchKernelEx(&cfg, st::ffn_stream_kernel<5>, args, g));
    count_launch();
    return PQE_OK;
}

}  // namespace pqe
