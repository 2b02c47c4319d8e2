// ffn_tc.cu -- expert FFN for large per-expert batches on the 5th-generation
// tensor cores (tcgen05, FP8 E4M3 x E4M3 -> fp32 in TMEM), fed by TMA from
// the slot pool through the page table.
//
// Module-based batching (MoE-Gen summary, aibr.jp, "3.中核となる技術的要素")
// gives each expert a batch of hundreds of tokens; the FFN is then a grouped
// GEMM over ragged per-expert segments. The weights are read from the slot
// each expert's page occupies (expert-pager article, rand.pepabo.com,
// "エキスパート重みの階層ページング"): one 3-D TMA tensor map per pool region
// [slot, row, k] with the slot as the outer coordinate.
//
// Per segment of expert e (rows p of the permuted batch, tiles of 128):
//   GEMM1  D[128 x 256] = Xq[p, :] . [W13 gate rows j..j+127 ; up rows I+j..]^T
//          epilogue: u = D * sx[p] * s13[row]; h = SiLU(u_gate) * u_up -> bf16,
//          row amax of h -> hmax[p]
//   hquant hq[p, :] = E4M3(h[p, :] / sh[p]), sh[p] = hmax[p] / 448
//   GEMM2  D[128 x 256] = hq[p, :] . W2[n..n+255, :]^T
//          epilogue: out_perm[p, n..] = D * sh[p] * s2[n] -> bf16
// Activations are quantised once per token to E4M3 (scale amax / 448); a
// gather kernel then copies the E4M3 rows into batch order for TMA (a byte
// copy: each token's row is read from L2, not re-quantised per batch row).
//
// MXFP4 pages (E2M1 weights, one E8M0 scale per 32 along a row) are multiplied
// as they are, by the block-scaled MMA (kind::mxf8f6f4 with .block_scale): E4M3
// activations x E2M1 weights, each 32-element K block scaled by a 2^e pair
// read from TMEM. TMA brings the packed E2M1 rows into 8-bit-footprint smem
// rows (16 values in the low 8 bytes of each 16-byte chunk, the layout the MMA
// reads), so the smem tiles and descriptors are those of FP8. Per stage, four
// scale warps (one per TMEM lane quarter) load the 256 weight rows' E8M0 bytes
// of the stage's four K blocks and write them into a TMEM ring: row n's word at
// lane 32q + n % 32 of every quarter q, column SFB + n / 32 (each quarter's MMA
// datapath reads its own lanes); the activations' scales are all 2^0 (their
// fp32 row scale stays in the epilogue), at lane m, column SFA + m / 32, and the
// MMA's scale-factor ids pick the K block's byte. The scale columns take the
// room of the second accumulator, so MXFP4 items run with one.
//
// Persistent CTA (one per SM, or per SM of a given share) over (M tile,
// N tile) work items, 10 warps: warp 0 issues TMA (one thread), warp 1 owns
// TMEM and issues the MMAs (one thread), warps 2-9 read the accumulator from
// TMEM (two warps per 32-lane quarter, each half of the columns) and run the
// epilogue. 4-stage smem ring of A [128 x 128 B] + B [256 x 128 B] tiles,
// 128-byte swizzle, K-major; two TMEM accumulators so the epilogue of one item
// overlaps the MMAs of the next. The epilogue scales with packed fp32
// multiplies, converts two values per instruction to bf16 and stages 32-column
// chunks in two per-warp shared buffers (the output map's 64-byte swizzle),
// which leave in pairs as TMA stores; rows past an expert's segment are never
// written.
// Every mbarrier wait is bounded: on expiry the CTA sets PQE_STATUS_TIMEOUT,
// drains what it issued (bounded), frees its TMEM and returns.
//
// The kernels after the first of the chain are launched with programmatic
// dependent launch: a kernel may be set up while its predecessor runs. One
// that reads its predecessor's output waits for it (griddepcontrol.wait)
// before its first read; the MXFP4 GEMM of a phase, which needs nothing from
// the FP8 GEMM before it, starts as that GEMM's CTAs drain and waits for it
// only before it exits, so that everything after it still sees both done.
// A kernel lets its successor launch (griddepcontrol.launch_dependents) only
// after its own wait, so a successor never starts before the data its
// predecessor read is complete.
#include <cuda.h>

#include <atomic>

#include "ffn_internal.cuh"
#include "pqe_common.cuh"
#include "tc_ptx.cuh"

namespace pqe {
namespace tc {
using namespace ptx;

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;  // bytes of K per stage (FP8)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 8;  // two per TMEM lane quarter, each taking half the columns
constexpr int SF_WARPS = 4;   // MXFP4: one scale warp per TMEM lane quarter
constexpr int SF_WARP0 = 2 + EPI_WARPS;
__host__ __device__ constexpr int threads_of(bool fp4) { return 64 + 32 * EPI_WARPS + (fp4 ? 32 * SF_WARPS : 0); }
constexpr uint32_t SFA_COL = 256;  // MXFP4: activation scales (4 columns)
constexpr uint32_t SFB_COL = 264;  // MXFP4: weight scales, 8 columns per ring stage
constexpr uint32_t ACC_COLS = 256;       // one fp32 accumulator of BM x BN
constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;  // two: the epilogue of item i overlaps the MMAs of item i+1
constexpr int ROW_CTAS = BM / 8;  // row kernels: CTAs of 8 warps per 128-row tile, one row per warp
// smem: stages | full[S] empty[S] tfull[2] tempty[2] | tmem base | column scales [2][BN] | store buffers
constexpr int SMEM_BAR_OFF = STAGES * STAGE_BYTES;
constexpr int SMEM_TMEM_OFF = SMEM_BAR_OFF + 8 * (2 * STAGES + 4);
// store buffers: per epilogue warp 32 rows x 64 bytes (32 bf16 columns), laid out
// with the 64-byte swizzle the output tensor maps use; 1024-byte aligned
constexpr int EPI_BUF = 32 * 64;
constexpr int EPI_NBUF = 2;  // store buffers per epilogue warp (32-column chunks flushed together)
constexpr int SMEM_EPI_OFF = (SMEM_TMEM_OFF + 4 + 1023) / 1024 * 1024;
constexpr int SMEM_BYTES = SMEM_EPI_OFF + EPI_WARPS * EPI_NBUF * EPI_BUF + 1024;  // + alignment slack

// instruction descriptor, kind::f8f6f4: D f32, A/B E4M3, both K-major, N, M
constexpr uint32_t IDESC = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(BM >> 4) << 24);
// instruction descriptor, kind::mxf8f6f4 with block scaling: A E4M3, B E2M1,
// both K-major, E8M0 scales, N, M; the scale-factor ids (bits 4-5 for B, 29-30
// for A) select the byte of the scale words, i.e. the K block of the stage
constexpr uint32_t IDESC_MX = (0u << 7) | (5u << 10) | ((uint32_t)(BN >> 3) << 17) | (1u << 23) |
                              ((uint32_t)(BM >> 4) << 24);

// programmatic dependent launch: PDL_WAIT_START waits for the predecessor grid
// before the kernel reads anything, PDL_WAIT_END before it exits (a no-op for
// a kernel launched without the attribute)
constexpr int PDL_WAIT_START = 1, PDL_WAIT_END = 2;
__device__ __forceinline__ void pdl_begin(int pdl) {
    if (pdl & PDL_WAIT_START) pdl_wait();
    pdl_trigger();
}

__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accum) {
    umma_f8f6f4(d_tmem, adesc, bdesc, IDESC, accum);
}

// block-scaled MMA on scale words in TMEM (sfa, sfb), K block kb of the stage
__device__ __forceinline__ void umma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t sfa, uint32_t sfb,
                                        uint32_t kb, uint32_t accum) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\ttcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, "
        "%2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(IDESC_MX | (kb << 4) | (kb << 29)), "r"(sfa), "r"(sfb), "r"(accum)
        : "memory");
}

// this warp's 32 TMEM lanes, 4 / 8 consecutive 32-bit columns from taddr
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %1, %1, %1};" ::"r"(taddr), "r"(v) : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// SiLU with the hardware exponential and reciprocal: the activations on this
// path are rounded to E4M3 (3 mantissa bits), far coarser than their error
__device__ __forceinline__ float silu_fast(float z) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + __expf(-z)));
    return z * r;
}

struct GemmArgs {
    const int32_t *tiles;    // [n][4]: expert, first row p0, valid rows, page-table entry
    const int32_t *n_tiles;  // device count of this launch's tiles
    const int32_t *tile_first;  // device index of this launch's first tile (NULL: 0)
    int n_nt;                // N tiles per M tile
    int n_slots;             // entries below this use the cache map,
    int n_wb;                // then n_wb working-buffer entries
    int K;                   // reduction length in bytes (H for GEMM1, I for GEMM2)
    int I;                   // GEMM1: up rows start at I
    int out_cols;            // row length of the output (I for h, H for out_perm)
    int swiglu;              // 1: GEMM1 epilogue, 0: GEMM2 epilogue
    const float *row_scale;  // sx or sh [A]
    const uint8_t *pool_base, *wb_base;
    size_t slot_stride;
    size_t wscale_off;       // FP8: byte offset of the weight row scales in a page (s13 or s2)
    size_t sf_off;           // MXFP4: byte offset of the E8M0 block scales in a page (x13 or x2)
    int sf_row_bytes;        // MXFP4: block-scale bytes per weight row (K / 32)
    uint16_t *out;           // bf16 h [A, I] or out_perm [A, H]
    uint32_t *hmax;          // [A] (GEMM1)
    int32_t *status;
    uint32_t wait_limit;     // polls of a bounded wait before it gives up
    int pdl;                 // PDL_WAIT_START / PDL_WAIT_END
};

// address of the page behind a tile's page-table entry (cache or working buffer)
__device__ __forceinline__ const uint8_t *tile_page(const GemmArgs &a, int slot) {
    if (slot < a.n_slots) return a.pool_base + (size_t)slot * a.slot_stride;
    return a.wb_base + (size_t)(slot - a.n_slots) * a.slot_stride;
}

struct Item {
    int p0, nv, slot, nt, r0, r1;
};

__device__ __forceinline__ Item item_of(const GemmArgs &a, int first, int i) {
    const int4 t = reinterpret_cast<const int4 *>(a.tiles)[first + i / a.n_nt];
    Item it;
    it.p0 = t.y;
    it.nv = t.z;
    it.slot = t.w;
    it.nt = i % a.n_nt;
    // B rows of this N tile: two halves of 128 rows
    it.r0 = a.swiglu ? it.nt * 128 : it.nt * 256;
    it.r1 = a.swiglu ? a.I + it.nt * 128 : it.nt * 256 + 128;
    return it;
}

// a * b for two fp32 pairs in one instruction (sm_100+ packed fp32)
__device__ __forceinline__ float2 mul2(float2 x, float2 y) {
    uint64_t rx, ry, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(rx) : "f"(x.x), "f"(x.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(ry) : "f"(y.x), "f"(y.y));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(rx), "l"(ry));
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(rd));
    return r;
}

// two floats -> bf16x2 (lo in the low half), round to nearest even
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// A warp's 32 output rows x 32 bf16 columns (lane = row, packed = its 64 bytes)
// into one of its shared buffers, in the 64-byte swizzle of the output tensor
// map (16-byte piece v of row r at piece v ^ ((r >> 1) & 3)), which also makes
// the writes conflict-free.
__device__ __forceinline__ void stage_rows32(uint8_t *buf, const uint32_t (&packed)[16], int lane) {
    uint8_t *mine = buf + lane * 64;
    const int sw = (lane >> 1) & 3;
#pragma unroll
    for (int v = 0; v < 4; ++v)
        *reinterpret_cast<uint4 *>(mine + 16 * (v ^ sw)) =
            make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
}

// The n chunks a warp staged for an item (buffers 0..n-1, 32 columns each from
// column col) leave together: a full group of 32 batch rows as n TMA stores in
// one bulk group behind one proxy fence; a partial group (the end of an
// expert's segment) row by row, 8 rows x 64 bytes per instruction, so that no
// row of another expert is written.
__device__ __forceinline__ void flush_rows32(const uint8_t *buf0, int n, const CUtensorMap *tm, int col, int row0,
                                             uint16_t *out, size_t ld, int nrows, int lane) {
    if (nrows == 32) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // writes visible to the TMA unit
        __syncwarp();
        if (lane == 0) {
            for (int c = 0; c < n; ++c)
                asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                                 reinterpret_cast<uint64_t>(tm)),
                             "r"(col + 32 * c), "r"(row0), "r"(smem_u32(buf0 + c * EPI_BUF))
                             : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        return;
    }
    __syncwarp();
    for (int c = 0; c < n; ++c) {
        const uint8_t *buf = buf0 + c * EPI_BUF;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int pc = it * 32 + lane, r = pc >> 2, part = pc & 3;
            if (r < nrows)
                *reinterpret_cast<uint4 *>(out + (size_t)r * ld + 32 * c + 8 * part) =
                    *reinterpret_cast<const uint4 *>(buf + r * 64 + 16 * (part ^ ((r >> 1) & 3)));
        }
    }
    __syncwarp();
}

// barrier among the epilogue warps only (named barrier 1) with an AND vote:
// every epilogue warp takes the same branch
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

// Persistent: CTA b takes work items b, b + G, b + 2G, ... (item = M tile x N
// tile; neighbouring CTAs share an M tile, so its activations stay in L2).
// FP4: the weights are MXFP4 pages (block-scaled MMA, scale warps, one accumulator).
template <bool FP4>
__global__ void __launch_bounds__(threads_of(FP4), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB_cache,
                   const __grid_constant__ CUtensorMap tmB_wb, const __grid_constant__ CUtensorMap tmOut,
                   const GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    constexpr int NBUF = FP4 ? 1 : 2;  // accumulators: the second one's columns hold the scales on the FP4 path
    const int first = a.tile_first ? *a.tile_first : 0;
    const int n_items = *a.n_tiles * a.n_nt;
    if ((int)blockIdx.x >= n_items) {
        if (a.pdl) pdl_wait();  // an idle CTA still orders the grid's completion after its predecessor
        return;
    }
    // 1024-byte alignment for the 128-byte swizzle atoms
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + SMEM_BAR_OFF;
    const uint32_t bar_empty = bar_full + 8 * STAGES;
    const uint32_t bar_tfull = bar_empty + 8 * STAGES;
    const uint32_t bar_tempty = bar_tfull + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + SMEM_TMEM_OFF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const int nk = a.K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, FP4 ? 1 + SF_WARPS : 1);  // FP4: the TMA bytes and the scale warps
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_tfull + 8 * b, 1);
            mbar_init(bar_tempty + 8 * b, EPI_WARPS * 32);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB_cache)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB_wb)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_begin(a.pdl);  // the set-up above may overlap the predecessor; the inputs are read below

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int i = blockIdx.x; i < n_items && ok; i += G) {
                const Item w = item_of(a, first, i);
                // the region the tile's page lies in, and its index there
                const bool cache = w.slot < a.n_slots;
                const CUtensorMap *tmB = cache ? &tmB_cache : &tmB_wb;
                const int zc = cache ? w.slot : w.slot - a.n_slots;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (!mbar_wait(bar_empty + 8 * s, ((uint32_t)(it / STAGES) & 1u) ^ 1u, a.wait_limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + s * STAGE_BYTES, sb = sa + A_BYTES;
                    // packed E2M1 rows count their global bytes (half the smem footprint)
                    mbar_expect_tx(bar_full + 8 * s, FP4 ? A_BYTES + B_BYTES / 2 : STAGE_BYTES);
                    tma_load_2d(sa, &tmA, kb * BK, w.p0, bar_full + 8 * s);
                    tma_load_3d(sb, tmB, kb * BK, w.r0, zc, bar_full + 8 * s);
                    tma_load_3d(sb + B_BYTES / 2, tmB, kb * BK, w.r1, zc, bar_full + 8 * s);
                }
            }
            if (!ok) atomicOr(a.status, PQE_STATUS_TIMEOUT);
            // drain: the stages issued last have landed before the CTA may exit
            for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
                mbar_wait(bar_full + 8 * (j % STAGES), (uint32_t)(j / STAGES) & 1u, a.wait_limit);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int it = 0, local = 0;
            bool ok = true;
            for (int i = blockIdx.x; i < n_items && ok; i += G, ++local) {
                const int b = local % NBUF;
                if (!mbar_wait(bar_tempty + 8 * b, ((uint32_t)(local / NBUF) & 1u) ^ 1u, a.wait_limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)b * ACC_COLS;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (!mbar_wait(bar_full + 8 * s, (uint32_t)(it / STAGES) & 1u, a.wait_limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = sbase + s * STAGE_BYTES, sb = sa + A_BYTES;
                    if constexpr (FP4) {
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k)
                            umma_mx(d, sw128_desc(sa + 32 * k), sw128_desc(sb + 32 * k), tmem + SFA_COL,
                                    tmem + SFB_COL + 8 * s, (uint32_t)k, (kb | k) != 0);
                    } else {
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k)
                            umma_f8(d, sw128_desc(sa + 32 * k), sw128_desc(sb + 32 * k), (kb | k) != 0);
                    }
                    umma_commit(bar_empty + 8 * s);
                }
                umma_commit(bar_tfull + 8 * b);
            }
            if (!ok) atomicOr(a.status, PQE_STATUS_TIMEOUT);
            // every issued MMA has finished before TMEM is released
            if (local > 0)
                mbar_wait(bar_tfull + 8 * ((local - 1) % NBUF), (uint32_t)((local - 1) / NBUF) & 1u, a.wait_limit);
        }
    } else if (FP4 && warp >= SF_WARP0) {
        // ---------------- MXFP4 scale warps: E8M0 block scales -> TMEM ----------------
        const int q = warp & 3;  // the TMEM lane quarter this warp may access
        const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
        tmem_st4(tq + SFA_COL, 0x7F7F7F7Fu);  // the activations' block scales: 2^0
        tmem_st_wait();
        int it = 0;
        bool ok = true;
        for (int i = blockIdx.x; i < n_items && ok; i += G) {
            const Item w = item_of(a, first, i);
            const uint8_t *xs = tile_page(a, w.slot) + a.sf_off;
            for (int kb = 0; kb < nk; ++kb, ++it) {
                const int s = it % STAGES;
                // the MMAs that read this stage's scale columns before have finished
                int e_ok = 1;
                if (lane == 0) e_ok = mbar_wait(bar_empty + 8 * s, ((uint32_t)(it / STAGES) & 1u) ^ 1u, a.wait_limit);
                if (!__shfl_sync(0xffffffffu, e_ok, 0)) {
                    ok = false;
                    break;
                }
                // B row n of the tile: weight row r0 + n (n < 128) or r1 + n - 128; its
                // four scale bytes of this stage's K blocks form one word
                uint32_t v[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int n = lane + 32 * c;
                    const int row = n < 128 ? w.r0 + n : w.r1 + n - 128;
                    v[c] = __ldg(reinterpret_cast<const uint32_t *>(xs + (size_t)row * a.sf_row_bytes) + kb);
                }
                tmem_st8(tq + SFB_COL + 8 * s, v);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_plain(bar_full + 8 * s);
            }
        }
        if (!ok && lane == 0) atomicOr(a.status, PQE_STATUS_TIMEOUT);
    } else {
        // ---------------- epilogue: TMEM -> registers -> global ----------------
        const int q = warp & 3;            // TMEM lane quarter this warp may access
        const int half = (warp - 2) >> 2;  // which half of the tile's columns it finishes
        const int m = 32 * q + lane;
        const int et = threadIdx.x - 64;  // one output column per epilogue thread (BN of them)
        uint8_t *ebuf = smem + SMEM_EPI_OFF + (warp - 2) * EPI_NBUF * EPI_BUF;  // this warp's store buffers
        static_assert(SMEM_BYTES <= 227 * 1024, "shared memory of one CTA");
        int local = 0;
        bool ok = true;
        for (int i = blockIdx.x; i < n_items && ok; i += G, ++local) {
            const Item w = item_of(a, first, i);
            const int b = local % NBUF;
            const int p = w.p0 + m;
            const bool valid = m < w.nv;
            // the weight-row (output column) scales of this warp's columns: output
            // column c < 128 is weight row r0 + c, c >= 128 row r1 + c - 128. They are
            // read with broadcast vector loads; fetched to L1 before the accumulator
            // wait, like this lane's row scale
            // MXFP4 pages have no row scales (their block scales are in the MMA): 1
            const float *wsc = reinterpret_cast<const float *>(tile_page(a, w.slot) + a.wscale_off);
            const float *cs_lo = wsc + w.r0, *cs_hi = wsc + w.r1 - 128;
            const float4 one4 = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
            if (!FP4 && lane < 4) {
                const float *pf = a.swiglu ? (lane < 2 ? cs_lo + 64 * half + 32 * lane : cs_hi + 128 + 64 * half + 32 * (lane - 2))
                                           : (half ? cs_hi + 128 : cs_lo) + 32 * lane;
                asm volatile("prefetch.global.L1 [%0];" ::"l"(pf));
            }
            const float rs = valid ? a.row_scale[p] : 0.0f;
            if (!epi_all(mbar_wait(bar_tfull + 8 * b, (uint32_t)(local / NBUF) & 1u, a.wait_limit))) {
                ok = false;
                if (et == 0) atomicOr(a.status, PQE_STATUS_TIMEOUT);
                break;
            }
            tc_fence_after();
            const uint32_t trow = tmem + (uint32_t)b * ACC_COLS + ((uint32_t)(32 * q) << 16);
            // this warp's 32 rows of the tile: the first, and how many hold batch rows
            uint16_t *wrow = a.out + (size_t)(w.p0 + 32 * q) * a.out_cols;
            const int nrows = min(max(w.nv - 32 * q, 0), 32);
            // the previous item's stores have finished reading this warp's buffers
            if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            __syncwarp();
            const float2 rs2 = make_float2(rs, rs);
            if (a.swiglu) {
                // h columns 64 half .. 64 half + 63 of the item's 128: gate in accumulator
                // columns c, up in c + 128
                float amax = 0.0f;
#pragma unroll 1
                for (int ci = 0; ci < 2; ++ci) {
                    const int c0 = 64 * half + 32 * ci;
                    uint32_t g[32], u[32];
                    tmem_ld32(trow + c0, g);
                    tmem_ld32(trow + 128 + c0, u);
                    tmem_ld_wait();
                    const float4 *cg = reinterpret_cast<const float4 *>(cs_lo + c0);
                    const float4 *cu = reinterpret_cast<const float4 *>(cs_hi + 128 + c0);
                    uint32_t packed[16];
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 sg = FP4 ? one4 : __ldg(cg + j4), su = FP4 ? one4 : __ldg(cu + j4);
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            const int j = 4 * j4 + 2 * t;
                            const float2 gs = mul2(t ? make_float2(sg.z, sg.w) : make_float2(sg.x, sg.y), rs2);
                            const float2 us = mul2(t ? make_float2(su.z, su.w) : make_float2(su.x, su.y), rs2);
                            const float2 gv = mul2(make_float2(__uint_as_float(g[j]), __uint_as_float(g[j + 1])), gs);
                            const float2 uv = mul2(make_float2(__uint_as_float(u[j]), __uint_as_float(u[j + 1])), us);
                            const float2 hv = mul2(make_float2(silu_fast(gv.x), silu_fast(gv.y)), uv);
                            const uint32_t hb = bf16x2_rn(hv.x, hv.y);
                            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(hb << 16)),
                                                     fabsf(__uint_as_float(hb & 0xffff0000u))));
                            packed[j / 2] = hb;
                        }
                    }
                    stage_rows32(ebuf + ci * EPI_BUF, packed, lane);
                }
                flush_rows32(ebuf, 2, &tmOut, w.nt * 128 + 64 * half, w.p0 + 32 * q, wrow + w.nt * 128 + 64 * half,
                             a.out_cols, nrows, lane);
                if (valid) atomicMax(a.hmax + p, __float_as_uint(amax));
            } else {
                // output columns 128 half .. 128 half + 127 of the item's 256, in four
                // 32-column chunks flushed in pairs; the third chunk is computed before
                // the wait for the first pair's stores, which then have its math to finish
                // reading the buffers
                const float *csw = half ? cs_hi : cs_lo;
                auto chunk = [&](int ci, uint32_t (&packed)[16]) {
                    const int c0 = 128 * half + 32 * ci;
                    uint32_t d[32];
                    tmem_ld32(trow + c0, d);
                    tmem_ld_wait();
                    const float4 *c4 = reinterpret_cast<const float4 *>(csw + c0);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 sc = FP4 ? one4 : __ldg(c4 + j4);
                        const float2 s01 = mul2(make_float2(sc.x, sc.y), rs2), s23 = mul2(make_float2(sc.z, sc.w), rs2);
                        const int j = 4 * j4;
                        const float2 v01 = mul2(make_float2(__uint_as_float(d[j]), __uint_as_float(d[j + 1])), s01);
                        const float2 v23 = mul2(make_float2(__uint_as_float(d[j + 2]), __uint_as_float(d[j + 3])), s23);
                        packed[2 * j4] = bf16x2_rn(v01.x, v01.y);
                        packed[2 * j4 + 1] = bf16x2_rn(v23.x, v23.y);
                    }
                };
                uint32_t packed[16];
                chunk(0, packed);
                stage_rows32(ebuf, packed, lane);
                chunk(1, packed);
                stage_rows32(ebuf + EPI_BUF, packed, lane);
                flush_rows32(ebuf, 2, &tmOut, w.nt * 256 + 128 * half, w.p0 + 32 * q, wrow + w.nt * 256 + 128 * half,
                             a.out_cols, nrows, lane);
                chunk(2, packed);
                if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                __syncwarp();
                stage_rows32(ebuf, packed, lane);
                chunk(3, packed);
                stage_rows32(ebuf + EPI_BUF, packed, lane);
                flush_rows32(ebuf, 2, &tmOut, w.nt * 256 + 128 * half + 64, w.p0 + 32 * q,
                             wrow + w.nt * 256 + 128 * half + 64, a.out_cols, nrows, lane);
            }
            // this accumulator may be overwritten by the MMAs of item i + NBUF * G
            tc_fence_before();
            mbar_arrive_plain(bar_tempty + 8 * b);
        }
    }
    // every TMA store of an epilogue warp has completed before the CTA leaves
    if (warp >= 2 && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
    if (a.pdl & PDL_WAIT_END) pdl_wait();
}

// ---------------------------------------------------------------------------
// quantise: xt[t, :] = E4M3(x[t, :] / st[t]), st[t] = amax / 448 (1 for a zero
// row); one warp per token, 8 tokens per CTA, the grid striding over the tokens.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) tc_xquant_kernel(const uint16_t *__restrict__ x, int T, int H,
                                                        uint8_t *__restrict__ xt, float *__restrict__ st) {
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t = (int)blockIdx.x * 8 + warp; t < T; t += (int)gridDim.x * 8) {
        const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
        float amax = 0.0f;
        for (int c = lane; c < H / 8; c += 32) {
            const uint4 v = __ldg(xr + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
                amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xffff0000u))));
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
        const float inv = __fdiv_rn(1.0f, s);
        for (int c = lane; c < H / 8; c += 32) {
            const uint4 v = __ldg(xr + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t q[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const uint16_t lo = f32x2_to_e4m3x2(__uint_as_float(w[2 * i] << 16) * inv,
                                                    __uint_as_float(w[2 * i] & 0xffff0000u) * inv);
                const uint16_t hi = f32x2_to_e4m3x2(__uint_as_float(w[2 * i + 1] << 16) * inv,
                                                    __uint_as_float(w[2 * i + 1] & 0xffff0000u) * inv);
                q[i] = (uint32_t)lo | ((uint32_t)hi << 16);
            }
            reinterpret_cast<uint2 *>(xt + (size_t)t * H)[c] = make_uint2(q[0], q[1]);
        }
        if (lane == 0) st[t] = s;
    }
}

// ---------------------------------------------------------------------------
// gather: row p of the batch <- xt[perm_src[p] / k], sx[p] = st[that token];
// one warp per row, rows of TC tiles (unit u: tile u / 16, rows 8 (u % 16) ..
// +7), the grid striding over the units of the scheduled tiles. Also clears
// hmax for the rows.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) tc_gather_kernel(const uint8_t *__restrict__ xt, const float *__restrict__ st,
                                                        const int32_t *__restrict__ perm_src, int k, int H,
                                                        const int32_t *__restrict__ tiles,
                                                        const int32_t *__restrict__ n_tiles,
                                                        uint8_t *__restrict__ xq, float *__restrict__ sx,
                                                        uint32_t *__restrict__ hmax) {
    pdl_begin(PDL_WAIT_START);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int units = *n_tiles * ROW_CTAS;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int4 tile = reinterpret_cast<const int4 *>(tiles)[u / ROW_CTAS];
        const int m = (u % ROW_CTAS) * 8 + warp;
        if (m >= tile.z) continue;
        const int p = tile.y + m;
        const int t = __ldg(perm_src + p) / k;
        const uint4 *src = reinterpret_cast<const uint4 *>(xt + (size_t)t * H);
        uint4 *dst = reinterpret_cast<uint4 *>(xq + (size_t)p * H);
        for (int c = lane; c < H / 16; c += 32) dst[c] = __ldg(src + c);
        if (lane == 0) {
            sx[p] = __ldg(st + t);
            hmax[p] = 0u;
        }
    }
}

// hq[p, :] = E4M3(h[p, :] / sh[p]), sh[p] = hmax[p] / 448; one warp per row
__global__ void __launch_bounds__(256) tc_hquant_kernel(const uint16_t *__restrict__ h, int I,
                                                        const int32_t *__restrict__ tiles,
                                                        const int32_t *__restrict__ n_tiles,
                                                        const uint32_t *__restrict__ hmax, uint8_t *__restrict__ hq,
                                                        float *__restrict__ sh) {
    pdl_begin(PDL_WAIT_START);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int units = *n_tiles * ROW_CTAS;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int4 tile = reinterpret_cast<const int4 *>(tiles)[u / ROW_CTAS];
        const int m = (u % ROW_CTAS) * 8 + warp;
        if (m >= tile.z) continue;
        const int p = tile.y + m;
        const float amax = __uint_as_float(hmax[p]);
        const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
        const float inv = __fdiv_rn(1.0f, s);
        const uint4 *hr = reinterpret_cast<const uint4 *>(h + (size_t)p * I);
        for (int c = lane; c < I / 8; c += 32) {
            const uint4 v = hr[c];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t q[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const uint16_t lo = f32x2_to_e4m3x2(__uint_as_float(w[2 * i] << 16) * inv,
                                                    __uint_as_float(w[2 * i] & 0xffff0000u) * inv);
                const uint16_t hi = f32x2_to_e4m3x2(__uint_as_float(w[2 * i + 1] << 16) * inv,
                                                    __uint_as_float(w[2 * i + 1] & 0xffff0000u) * inv);
                q[i] = (uint32_t)lo | ((uint32_t)hi << 16);
            }
            reinterpret_cast<uint2 *>(hq + (size_t)p * I)[c] = make_uint2(q[0], q[1]);
        }
        if (lane == 0) sh[p] = s;
    }
}

// ---- host: tensor maps -------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D [rows, cols] uint8, box [128 rows, 128 cols], 128-byte swizzle
static bool map_2d(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {128, 128};
    cuuint32_t es[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D [rows, cols] bf16 output, box [32 rows, 32 cols], 64-byte swizzle (epilogue TMA stores)
static bool map_out(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t es[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D [slots, rows, cols] uint8 with a slot stride, box [1, 128, 128]
static bool map_3d(CUtensorMap *m, const void *base, uint64_t slots, uint64_t rows, uint64_t cols,
                   uint64_t slot_stride) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[3] = {cols, rows, slots};
    cuuint64_t strides[2] = {cols, slot_stride};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D [slots, rows, cols] packed E2M1 (cols values, cols / 2 bytes a row) with a
// slot stride, box [1, 128, 128 values]: each 16 values land in the low half of
// a 16-byte smem chunk (the 8-bit footprint the block-scaled MMA reads), 128-byte
// swizzle. Needs cols % 128 == 0, a 32-byte aligned base, strides % 32 == 0.
static bool map_3d_fp4(CUtensorMap *m, const void *base, uint64_t slots, uint64_t rows, uint64_t cols,
                       uint64_t slot_stride) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[3] = {cols, rows, slots};
    cuuint64_t strides[2] = {cols / 2, slot_stride};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

bool tc_shape_ok(int H, int I) { return H % 256 == 0 && I % 128 == 0 && H >= 256 && I >= 128; }

int launch_ffn_tc(const FfnArgs &args, const TcBuffers &b, int max_tiles, cudaStream_t s, int sm_cap) {
    using namespace tc;
    const int H = args.H, I = args.I;
    const long A = b.A;
    CUtensorMap mx, mh, m13c, m13w, m2c, m2w, f13c, f13w, f2c, f2w, mo1, mo2;
    const PageLayout L = fp8_layout(H, I), L4 = mxfp4_layout(H, I);
    // the working-buffer / cache maps need a non-empty region to encode; an
    // absent region gets a one-slot map over the other base (never selected)
    const uint8_t *cache = args.n_slots ? args.pool_base : args.wb_base;
    const uint8_t *wb = args.n_wb ? args.wb_base : args.pool_base;
    const uint64_t ns = args.n_slots ? args.n_slots : 1, nw = args.n_wb ? args.n_wb : 1;
    bool ok = map_2d(&mx, b.xq, (uint64_t)A, (uint64_t)H) && map_2d(&mh, b.hq, (uint64_t)A, (uint64_t)I) &&
              map_3d(&m13c, cache + L.w13, ns, 2 * (uint64_t)I, H, args.slot_stride) &&
              map_3d(&m13w, wb + L.w13, nw, 2 * (uint64_t)I, H, args.slot_stride) &&
              map_3d(&m2c, cache + L.w2, ns, (uint64_t)H, I, args.slot_stride) &&
              map_3d(&m2w, wb + L.w2, nw, (uint64_t)H, I, args.slot_stride);
    ok = ok && map_out(&mo1, b.h, (uint64_t)A, (uint64_t)I) && map_out(&mo2, args.out_perm, (uint64_t)A, (uint64_t)H);
    // MXFP4 pages, when the layer tags formats
    const bool fp4 = args.expert_fmt != nullptr;
    if (fp4)
        ok = ok && map_3d_fp4(&f13c, cache + L4.w13, ns, 2 * (uint64_t)I, H, args.slot_stride) &&
             map_3d_fp4(&f13w, wb + L4.w13, nw, 2 * (uint64_t)I, H, args.slot_stride) &&
             map_3d_fp4(&f2c, cache + L4.w2, ns, (uint64_t)H, I, args.slot_stride) &&
             map_3d_fp4(&f2w, wb + L4.w2, nw, (uint64_t)H, I, args.slot_stride);
    if (!ok) return PQE_ERR_UNSUPPORTED;
    // the shared-memory opt-in is per device
    static std::atomic<int> attr_set[PQE_MAX_DEVICES];
    int dev = 0, sms = 0;
    const int di = device_info(dev, sms);
    if (di != PQE_OK) return di;
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        PQE_CUDA_TRY(cudaFuncSetAttribute(tc_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          SMEM_BYTES));
        PQE_CUDA_TRY(cudaFuncSetAttribute(tc_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          SMEM_BYTES));
        attr_set[dev].store(1, std::memory_order_relaxed);
    }
    // persistent grids: one CTA per SM (or per SM of the share given), at most one per work item
    const int cap = sm_cap > 0 && sm_cap < sms ? sm_cap : sms;
    const int items1 = max_tiles * (I / 128), items2 = max_tiles * (H / 256);
    const int grid1 = items1 < cap ? items1 : cap, grid2 = items2 < cap ? items2 : cap;
    // row kernels: eight CTAs of 256 threads per SM of the share at most (a full
    // SM), striding over the row units of the tiles the schedule produced
    const int row_units = max_tiles * ROW_CTAS, grid_rows = row_units < 8 * cap ? row_units : 8 * cap;
    const long T = A / args.k, tok_ctas = (T + 7) / 8;
    tc_xquant_kernel<<<(unsigned)(tok_ctas < 8L * cap ? tok_ctas : 8L * cap), 256, 0, s>>>(args.x, (int)T, H, b.xt,
                                                                                          b.st);
    PQE_LAUNCH_CHECK();
    int rc = launch_pdl(tc_gather_kernel, grid_rows, 256, 0, s, (const uint8_t *)b.xt, (const float *)b.st,
                        args.perm_src, args.k, H, (const int32_t *)b.tiles, (const int32_t *)b.n_tiles, b.xq, b.sx,
                        b.hmax);
    if (rc != PQE_OK) return rc;
    // GEMM1 over the FP8 tiles (the first n_tiles[1]), then the MXFP4 tiles (the next n_tiles[2])
    GemmArgs g1{};
    g1.tiles = b.tiles;
    g1.n_tiles = b.n_tiles + 1;
    g1.tile_first = nullptr;
    g1.n_nt = I / 128;
    g1.n_slots = args.n_slots;
    g1.n_wb = args.n_wb;
    g1.K = H;
    g1.I = I;
    g1.out_cols = I;
    g1.swiglu = 1;
    g1.row_scale = b.sx;
    g1.pool_base = args.pool_base;
    g1.wb_base = args.wb_base;
    g1.slot_stride = args.slot_stride;
    g1.wscale_off = L.s13;
    g1.sf_off = L4.s13;
    g1.sf_row_bytes = H / 32;
    g1.out = b.h;
    g1.hmax = b.hmax;
    g1.status = args.status;
    g1.wait_limit = args.wait_limit;
    g1.pdl = PDL_WAIT_START;
    if ((rc = launch_pdl(tc_gemm_kernel<false>, grid1, threads_of(false), SMEM_BYTES, s, mx, m13c, m13w, mo1, g1)))
        return rc;
    // the MXFP4 tiles need nothing from the FP8 GEMM: they start as its CTAs drain
    GemmArgs g1x = g1;
    g1x.n_tiles = b.n_tiles + 2;
    g1x.tile_first = b.n_tiles + 1;
    g1x.pdl = PDL_WAIT_END;
    if (fp4 && (rc = launch_pdl(tc_gemm_kernel<true>, grid1, threads_of(true), SMEM_BYTES, s, mx, f13c, f13w, mo1, g1x)))
        return rc;
    if ((rc = launch_pdl(tc_hquant_kernel, grid_rows, 256, 0, s, (const uint16_t *)b.h, I, (const int32_t *)b.tiles,
                         (const int32_t *)b.n_tiles, (const uint32_t *)b.hmax, b.hq, b.sh)))
        return rc;
    GemmArgs g2 = g1;
    g2.n_nt = H / 256;
    g2.K = I;
    g2.out_cols = H;
    g2.swiglu = 0;
    g2.row_scale = b.sh;
    g2.wscale_off = L.s2;
    g2.sf_off = L4.s2;
    g2.sf_row_bytes = I / 32;
    g2.out = args.out_perm;
    g2.hmax = nullptr;
    g2.pdl = PDL_WAIT_START;
    if ((rc = launch_pdl(tc_gemm_kernel<false>, grid2, threads_of(false), SMEM_BYTES, s, mh, m2c, m2w, mo2, g2)))
        return rc;
    if (fp4) {
        GemmArgs g2x = g2;
        g2x.n_tiles = b.n_tiles + 2;
        g2x.tile_first = b.n_tiles + 1;
        g2x.pdl = PDL_WAIT_END;
        if ((rc = launch_pdl(tc_gemm_kernel<true>, grid2, threads_of(true), SMEM_BYTES, s, mh, f2c, f2w, mo2, g2x)))
            return rc;
    }
    return PQE_OK;
}

}  // namespace pqe
