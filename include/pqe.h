/*
 * pqe.h -- C ABI of libpqe.so: the MoE expert layer over paged, quantized
 * expert weights, on one NVIDIA GB300 (sm_103a).
 *
 * The layer: top-k routing; a token-to-expert permutation that builds one
 * contiguous batch per expert; a SwiGLU expert FFN that reads FP8 (or 4-bit)
 * weights through an expert-to-slot page table into a fixed VRAM slot pool
 * managed LRU per layer; a weighted combine; and GPU decode of host-tier
 * pages whose FP8 exponents are Huffman-coded per row.
 *
 * Sources, cited by page and section:
 *   [EP] vllm-expert-pager article (rand.pepabo.com, 2026-09-18):
 *        "エキスパート重みの階層ページング" (per-layer slot pools, LRU,
 *        working buffer), "重みの圧縮" (per-row exponent Huffman, GPU decode
 *        after the copy), "評価"/表4 (code table resident in VRAM), and the
 *        "w13_weight"/"w2_weight" names of vLLM's FP8 MoE weights.
 *   [MG] MoE-Gen summary (aibr.jp), "3.中核となる技術的要素": module-based
 *        batching (large per-expert batches) and overlap of host-to-device
 *        transfer with compute.
 *   [PW] PagedWeight commentary (spectral-agent.com), "技術的に面白い点":
 *        page-unit weight management, per-expert bit-width from importance.
 *
 * Conventions for every call:
 *   - Return value: PQE_OK (0) or a negative PQE_ERR_* code.
 *   - Pointers marked "device" point to GPU memory owned by the caller
 *     (allocated with any CUDA allocator); the library never frees them and
 *     keeps no reference after the call returns. "host" pointers are CPU
 *     memory; "pinned" means page-locked host memory (cudaHostAlloc).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Device calls are asynchronous on it unless stated otherwise.
 *     Most kernels are launched with programmatic stream serialization, so
 *     one may be set up while the kernel before it on the stream finishes;
 *     none reads memory before the kernels whose output it reads have
 *     completed (griddepcontrol.wait), and none completes before the kernel
 *     launched before it, so ordering on `stream` is that of plain launches.
 *   - Arguments are checked on the host before any launch; a bad argument
 *     returns PQE_ERR_INVALID_ARG and launches nothing.
 *   - Errors found on the device (an out-of-range expert id, a corrupt
 *     compressed stream, a page whose format tag is unknown) are OR-ed into a
 *     caller-owned device int32 `status` word as PQE_STATUS_* bits; kernels
 *     never trap. The caller clears the word and reads it after the stream
 *     is synchronised.
 *   - bf16 tensors are row-major with the innermost dimension contiguous.
 *   - Shape limits: 1 <= k <= 32, k <= E <= 1024; H % 64 == 0, I % 64 == 0;
 *     64 <= H <= 16384, 64 <= I <= 8192; T >= 0 (T == 0 is a no-op).
 */
#ifndef PQE_H
#define PQE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PQE_API __attribute__((visibility("default")))
#else
#define PQE_API
#endif

#define PQE_OK 0
#define PQE_ERR_INVALID_ARG (-1)
#define PQE_ERR_CUDA (-2)
#define PQE_ERR_CAPACITY (-3)
#define PQE_ERR_CORRUPT (-4)
#define PQE_ERR_TIMEOUT (-5)
#define PQE_ERR_UNSUPPORTED (-6)
#define PQE_ERR_IO (-7)

/* bits OR-ed into the device status word */
#define PQE_STATUS_BAD_EXPERT_ID 0x1  /* a routed id outside [0, E) */
#define PQE_STATUS_CORRUPT_STREAM 0x2 /* a compressed row that does not decode */
#define PQE_STATUS_BAD_PAGE 0x4       /* page table entry outside the pool, or unknown format */
#define PQE_STATUS_TIMEOUT 0x8        /* a bounded device wait gave up */

/* page formats (per expert page) */
#define PQE_FMT_FP8 0   /* E4M3 weights, one fp32 scale per output row */
#define PQE_FMT_MXFP4 1 /* E2M1 weights, one E8M0 scale per 32 weights along a row */

/* Message for a PQE_* code; never NULL. */
PQE_API const char *pqe_strerror(int code);

/* Library ABI version (this header: 1). */
PQE_API int pqe_abi_version(void);

/* The cudaError_t of the last PQE_ERR_CUDA returned on this thread. */
PQE_API int pqe_last_cuda_error(void);

/* Kernels this library has launched in this process (all threads). */
PQE_API uint64_t pqe_kernel_launches(void);

/* Every wait inside a kernel of this library (on an mbarrier, or on a count
 * another CTA publishes) is bounded: after `polls` polls it gives up, ORs
 * PQE_STATUS_TIMEOUT into the call's status word, stops waiting for the rest
 * of the launch and lets the kernel run to its end, so the call returns and
 * the CUDA context stays usable (the outputs of that call are then
 * unspecified). Process-wide, read at each launch; 0 restores the default of
 * 2^22 polls (a fraction of a second). */
PQE_API int pqe_set_wait_limit(uint32_t polls);

/* Test hook for the expiry path above, with no GPU fault: adds `bias` to the
 * count of phase-1 work that phase 2 of every expert in the weight-stream FFN
 * kernel waits for, so any nonzero bias makes those waits expire. Process-wide,
 * read at each launch; 0 (the default) in normal use. */
PQE_API int pqe_test_set_phase2_bias(uint32_t bias);

/* Test hook: which weight-stream kernel moe_paged_ffn runs for batches of at
 * most 8 rows. 0 (the default): the tensor-core stream (tcgen05 MMAs on the
 * page's E4M3 codes, activations as two E4M3 terms) when expert_fmt is NULL
 * (every page FP8), the shape allows it and the step routes enough experts,
 * else the CUDA-core stream (mma.sync on f16-converted weights); 1: always the
 * CUDA-core stream; 2: the tensor-core stream wherever it applies. Both compute
 * the same layer; the choice changes rounding only, inside the stated
 * tolerance. Process-wide, read at each launch. PQE_ERR_INVALID_ARG for any
 * other kind. */
PQE_API int pqe_test_set_stream_kernel(int kind);

/* ------------------------------------------------------------------------
 * Expert pages and the slot pool  ([EP] 階層ページング; [PW] page-unit weights)
 *
 * One expert's weights form one page of contiguous bytes; the same byte
 * layout is used in a VRAM slot and in a host-tier buffer, so a refill is one
 * copy. FP8 page (offsets in bytes):
 *   w13 [2I, H] E4M3 at 0        (rows 0..I-1 gate projection, I..2I-1 up)
 *   w2  [H, I]  E4M3 at 2*I*H
 *   s13 [2I]    fp32 at 3*I*H    (per-row scales; weight = e4m3(code) * s)
 *   s2  [H]     fp32 at 3*I*H + 8*I
 * MXFP4 page:
 *   w13 [2I, H/2] E2M1 pairs at 0 (low nibble = even column)
 *   w2  [H, I/2]  E2M1 pairs at I*H
 *   x13 [2I, H/32] E8M0 at 3*I*H/2 (weight = e2m1 * 2^(x - 127))
 *   x2  [H, I/32]  E8M0 at 3*I*H/2 + I*H/16
 * A slot pool is n_slots cache slots of `slot_stride` bytes each (the LRU
 * cache of one layer) plus n_wb working-buffer entries, used when one step
 * needs more than n_slots experts. Page-table entry s < n_slots addresses
 * base + s * slot_stride, entry n_slots + w addresses wb_base + w *
 * slot_stride. The working buffer holds pages for one step only, so layers
 * that run one after another on one stream may share it.
 * ------------------------------------------------------------------------ */

/* Bytes of one page in format fmt; 0 for bad arguments. */
PQE_API size_t pqe_page_bytes(int fmt, int H, int I);

/* Slot stride for (H, I): the FP8 page size rounded up to 4096 bytes. */
PQE_API size_t pqe_slot_stride(int H, int I);

typedef struct pqe_pool {
    void *base;         /* device: n_slots * slot_stride bytes, 256-byte aligned */
    void *wb_base;      /* device: n_wb * slot_stride bytes, 256-byte aligned (NULL if n_wb == 0) */
    size_t slot_stride; /* == pqe_slot_stride(H, I) */
    int32_t n_slots;    /* cache slots */
    int32_t n_wb;       /* working-buffer entries */
    int32_t H, I;
} pqe_pool;

/* Device address of page-table entry `dest` of the pool; NULL if outside it. */
PQE_API void *pqe_pool_slot_addr(const pqe_pool *pool, int dest);

/* Quantise fp32 weights [rows, cols] (device) to E4M3 codes (device, [rows,
 * cols]) with one fp32 scale per row (device, [rows]): s = amax/448 in fp32
 * (1 for an all-zero row), code = RNE_e4m3(w / s) with the quotient in fp32,
 * saturating at 448: FP8 E4M3 weights with one fp32 scale per row, as the
 * workloads' experts are stored; it prepares pages and is not on the per-step path. */
PQE_API int pqe_quantize_fp8_rows(const float *w, int rows, int cols, uint8_t *q, float *scale, void *stream);

/* 4-bit copy of an FP8 matrix ([PW]: lower-bit pages; the FP8 master copy is
 * kept, [EP] 位置づけ). From v = fp32(e4m3(q)) * s (fp32 product), per block
 * of 32 along a row: X = 2^(floor(log2 amax) - 2) as E8M0 (byte 0 for an
 * all-zero block), element RNE_e2m1(v / X) saturating at 6 (OCP MX v1.0).
 * q8 [rows, cols] and s8 [rows] device in; q4 [rows, cols/2] and x8
 * [rows, cols/32] device out. cols % 32 == 0. */
PQE_API int pqe_quantize_mxfp4_rows(const uint8_t *q8, const float *s8, int rows, int cols, uint8_t *q4,
                            uint8_t *x8, void *stream);

/* Pack one FP8 page (device) from fp32 weights w13 [2I, H] and w2 [H, I]
 * (device): both matrices quantised with pqe_quantize_fp8_rows into the
 * page's sections. */
PQE_API int pqe_pack_fp8_page(const float *w13, const float *w2, int H, int I, uint8_t *page, void *stream);

/* Pack the 4-bit page (device) of an FP8 page (device) with
 * pqe_quantize_mxfp4_rows on both matrices. */
PQE_API int pqe_pack_mxfp4_page(const uint8_t *fp8_page, int H, int I, uint8_t *fp4_page, void *stream);

/* ------------------------------------------------------------------------
 * moe_route -- top-k routing ([EP] 階層ページング: each token uses a few
 * experts; [MG] §3). The pages give no formula; the plain MoE reading is used.
 *   logits[t,e] = sum_h x[t,h] * w_router[e,h] in fp32 when w_router is not
 *     NULL; the reduction order is fixed (32 strided partial sums with fused
 *     multiply-add, h = l, l+32, ..., then a pairwise tree over offsets 16, 8,
 *     4, 2, 1), so the logits, and with them the top-k choice, are
 *     reproducible bit for bit.
 *   top-k: the k largest logits, the lower expert id on an exact tie; ids are
 *     ordered by logit descending, then id ascending.
 *   gates: softmax over the k picked (the full softmax renormalised to them).
 * x_bf16   device bf16 [T, H] (read only when w_router != NULL)
 * w_router device fp32 [E, H] or NULL
 * logits   device fp32 [T, E]: output when w_router != NULL (may then be NULL
 *          to skip storing), input otherwise. Inputs must be finite.
 * topk_ids device int32 [T, k] out; topk_w device fp32 [T, k] out.
 * ------------------------------------------------------------------------ */
PQE_API int moe_route(const void *x_bf16, const float *w_router, float *logits, int T, int H, int E, int k,
              int32_t *topk_ids, float *topk_w, void *stream);

/* ------------------------------------------------------------------------
 * moe_permute -- token-to-expert permutation: one contiguous batch per expert
 * ([MG] §3, module-based batching). Stable counting sort of the assignments
 * f = t*k + j by expert id:
 *   counts[e] = #{f : topk_ids[f] == e}; offsets = exclusive prefix sum, E+1;
 *   within an expert, assignments keep ascending f;
 *   perm_src[p] = the f at batch position p; inv[f] = p.
 * The result is unique and deterministic.
 * topk_ids device int32 [T*k]; counts device int32 [E]; offsets device int32
 * [E+1]; perm_src, inv device int32 [T*k]. ws: device scratch of at least
 * moe_permute_workspace_size(T, k, E) bytes, 256-byte aligned. status: device
 * int32; an id outside [0, E) sets PQE_STATUS_BAD_EXPERT_ID and that
 * assignment is dropped from the counts (perm_src/inv then hold -1 for it).
 * ------------------------------------------------------------------------ */
PQE_API size_t moe_permute_workspace_size(int T, int k, int E);
PQE_API int moe_permute(const int32_t *topk_ids, int T, int k, int E, int32_t *counts, int32_t *offsets,
                int32_t *perm_src, int32_t *inv, void *ws, size_t ws_bytes, int32_t *status,
                void *stream);

/* moe_permute_static -- moe_permute without a caller-provided workspace.
 * The pages have no counterpart of this call. It exists for callers that
 * cannot hand the library scratch memory: a plugin inside a framework that
 * owns all device memory and exposes no allocator to it, or a steady-state
 * serving loop that must not call cudaMalloc/cudaFree because those
 * synchronise the device. Its scratch is one file-scope device array of
 * moe_permute_static_max_words() int32 (4 MiB), held on every GPU that loads
 * the library until the process exits; calls with T*k*E beyond it (more
 * than 1M chunk-histogram words, i.e. ceil(T*k/2048)*E > 1048576) return
 * PQE_ERR_CAPACITY. The call allocates nothing. The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture. All calls share
 * the one array, so calls that overlap on the GPU (other streams, other host
 * threads) race and corrupt each other's results; issue them in one stream
 * order. Results are identical to moe_permute's. The looked-up address is
 * cached for the life of the process: after cudaDeviceReset (or anything else
 * that tears down and recreates the device's context) it is stale, and the
 * call must not be used on that device again. */
PQE_API size_t moe_permute_static_max_words(void);
PQE_API int moe_permute_static(const int32_t *topk_ids, int T, int k, int E, int32_t *counts, int32_t *offsets,
                               int32_t *perm_src, int32_t *inv, int32_t *status, void *stream);

/* ------------------------------------------------------------------------
 * moe_paged_ffn -- grouped SwiGLU expert FFN over the slot pool ([EP]
 * 階層ページング for the paging, 評価 for w13/w2; [PW] for 4-bit pages).
 * For each expert e with a non-empty batch, its page is read from slot
 * page_table[e] of the pool, and for each batch position p in
 * [offsets[e], offsets[e+1]), with token t = perm_src[p] / k:
 *   u = W13_e x_t;  h = SiLU(u[0:I]) * u[I:2I];  out_perm[p] = W2_e h.
 * x_bf16     device bf16 [T, H]
 * perm_src, offsets: from moe_permute (device)
 * page_table device int32 [E]: slot of each routed expert, -1 if unrouted
 * expert_fmt device uint8 [E]: PQE_FMT_* of each expert's page, or NULL for
 *            all FP8
 * pool       host struct describing the device slot pool
 * out_perm   device bf16 [T*k, H] out
 * ws         device scratch, >= moe_paged_ffn_workspace_size(...) bytes
 * status     device int32; a routed expert whose slot is outside the pool or
 *            whose format is unknown sets PQE_STATUS_BAD_PAGE and its rows of
 *            out_perm are zero.
 * Work is dispatched on the device per expert batch: batches of at most 8
 * rows take the weight stream (mma.sync on the SMs' tensor pipe as a
 * dot-product engine), larger ones the tcgen05 tensor-core path.
 * Streams: all work is ordered after earlier work on `stream`, and later work
 * on `stream` is ordered after all of it. For decode-sized steps (T*k at most
 * 4*E) the tensor-core batches run on a side stream that the library creates
 * once per host thread and device (non-blocking, never destroyed). It is
 * forked from `stream` with an event after the call's first kernel and joined
 * back with another before the call returns. The call can be captured into a
 * CUDA graph (the fork and join become graph edges). Make one call before the
 * first capture on a host thread, so that the side stream and its events
 * exist.
 * ------------------------------------------------------------------------ */
PQE_API size_t moe_paged_ffn_workspace_size(int T, int k, int E, int H, int I);
PQE_API int moe_paged_ffn(const void *x_bf16, const int32_t *perm_src, const int32_t *offsets,
                  const int32_t *page_table, const uint8_t *expert_fmt, const pqe_pool *pool, int T,
                  int k, int E, void *out_perm, void *ws, size_t ws_bytes, int32_t *status,
                  void *stream);

/* ------------------------------------------------------------------------
 * moe_combine -- y[t] = sum_j topk_w[t,j] * out_perm[inv[t*k+j]] with fp32
 * accumulation in ascending j, bf16 output (the weighted sum that closes a
 * MoE layer; the pages do not spell it out).
 * out_perm device bf16 [T*k, H]; inv device int32 [T*k]; topk_w device fp32
 * [T, k]; y device bf16 [T, H] out. An inv entry of -1 contributes nothing.
 * ------------------------------------------------------------------------ */
PQE_API int moe_combine(const void *out_perm, const int32_t *inv, const float *topk_w, int T, int k, int H,
                void *y_bf16, void *stream);

/* ------------------------------------------------------------------------
 * Per-layer LRU slot pool on the host ([EP] 階層ページング: each MoE layer owns
 * its slots, one expert per slot, managed LRU; a miss is copied in; a step
 * that needs more experts than slots switches to a working buffer).
 * Rules (the pages say only "LRU"):
 *   U = {e : counts[e] > 0}.
 *   |U| > S: working-buffer step; slot state untouched (no eviction, no
 *     recency update); resident experts are read in place; every
 *     non-resident e in U gets entry S + w, w its rank among them by id.
 *   |U| <= S: hits refresh last_use = step; misses in ascending id take the
 *     lowest empty slot, else the slot with the smallest last_use whose expert
 *     is not in U (ties: lowest slot index).
 *   page_table[e] = slot or S + w for e in U, -1 otherwise; the step counter
 *   advances by one per call.
 * ------------------------------------------------------------------------ */
typedef struct pqe_lru pqe_lru;

/* New state with S empty slots for E experts; NULL on bad arguments. */
PQE_API pqe_lru *pqe_lru_create(int E, int S);
PQE_API void pqe_lru_destroy(pqe_lru *st);

/* Copy out slot->expert [S] (-1 empty), last_use [S] and the step counter. */
PQE_API int pqe_lru_state(const pqe_lru *st, int32_t *slot_expert, int64_t *last_use, int64_t *step);

/* Forget expert e's resident copy (its slot becomes empty), e.g. after its
 * page changed format. */
PQE_API int pqe_lru_invalidate(pqe_lru *st, int expert);

/* One step (host only, no CUDA call). counts_host [E] in; page_table_host
 * [E] out; miss_expert / miss_dest [E] out: the n_miss experts to copy and
 * their destination (slot, or S + w); working_buffer_mode out (0/1). */
PQE_API int page_table_update(pqe_lru *st, const int32_t *counts_host, int32_t *page_table_host,
                      int32_t *miss_expert, int32_t *miss_dest, int32_t *n_miss,
                      int32_t *working_buffer_mode);

/* ------------------------------------------------------------------------
 * slot_fill -- refill one slot from the host tier ([EP] 階層ページング: a
 * missing expert is copied from its RAM slot; [MG] §3: transfers overlap
 * compute). One cudaMemcpyAsync of `bytes` from pinned_src (pinned host, one
 * page in the layout above) to slot `dest` of the pool, on `stream` (a side
 * stream), then cudaEventRecord(done_event) if done_event is not NULL.
 * bytes <= pool->slot_stride.
 * ------------------------------------------------------------------------ */
PQE_API int slot_fill(const pqe_pool *pool, int dest, const void *pinned_src, size_t bytes, void *stream,
              void *done_event);

/* slot_fill_batch -- refill n entries of the pool with one kernel launch per
 * 128 pages: page i is read from host_src[i] (pinned host memory, which
 * kernels can address directly under unified addressing) and written to
 * entry dest[i]; bytes[i] <= slot_stride, a multiple of 16, both addresses
 * 16-byte aligned. dest, host_src, bytes are host arrays. Asynchronous on
 * `stream`; done_event recorded after the last launch if not NULL. The SMs
 * pull the pages over the host link, so one launch (per 128 pages) covers
 * every miss of a step at the link's bandwidth. */
PQE_API int slot_fill_batch(const pqe_pool *pool, int n, const int32_t *dest, const void *const *host_src,
                            const size_t *bytes, void *stream, void *done_event);

/* ------------------------------------------------------------------------
 * GPU-resident pager: the same LRU rules with the state in device memory, so
 * a step needs no host round trip (the counts, page table, miss list and
 * refill stay on the GPU). State: pqe_lru_device_bytes(E, S) bytes of device
 * memory, 16-byte aligned, owned by the caller; E <= 1024, S <= 1024.
 * ------------------------------------------------------------------------ */
PQE_API size_t pqe_lru_device_bytes(int E, int S);

/* All slots empty, step 0, counters 0 (asynchronous on stream). */
PQE_API int pqe_lru_device_init(void *state, int E, int S, void *stream);

/* Forget expert e's resident copy (asynchronous on stream). */
PQE_API int pqe_lru_device_invalidate(void *state, int E, int S, int expert, void *stream);

/* Copy the state to the host (synchronises the stream): slot_expert [S],
 * last_use [S], step, and running totals stats[4] = routed experts, misses,
 * working-buffer steps, refill bytes. Any output may be NULL. */
PQE_API int pqe_lru_device_state(const void *state, int E, int S, int32_t *slot_expert, int64_t *last_use,
                                 int64_t *step, int64_t *stats, void *stream);

/* page_table_update on the device, one CTA: counts [E] (device) ->
 * page_table [E] (device) and miss (device int32 [3E + 3]): [0] number of
 * misses, [1] working-buffer flag, [2, 2+E) missed experts in ascending id,
 * [2+E, 2+2E) their destinations, [2+2E, 3+3E) prefix of their refill
 * segments. page_bytes [E] (device): bytes of each expert's host page. */
PQE_API int page_table_update_device(void *state, int E, int S, const int32_t *counts, const size_t *page_bytes,
                                     int32_t *page_table, int32_t *miss, void *stream);

/* Refill every page of a device miss list from pinned host memory:
 * host_pages [E] (device array of the pinned page addresses), page_bytes [E]
 * (device). One persistent kernel; no host involvement. */
PQE_API int slot_fill_device(const pqe_pool *pool, const int32_t *miss, int E, const uint64_t *host_pages,
                             const size_t *page_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Compressed host tier ([EP] 重みの圧縮: per row of each expert weight matrix
 * the FP8 exponent field is Huffman-coded, the rest kept raw; decoded on the
 * GPU right after the copy to VRAM; 表4: the code table stays in VRAM).
 * Format (the pages fix only the above):
 *   symbol = (byte >> 3) & 15; raw nibble = (byte >> 7) << 3 | (byte & 7);
 *   one canonical prefix code per matrix (w13 and w2 of each expert), lengths
 *   <= 12, optimal for the matrix's symbol histogram (package-merge; at equal
 *   weight a symbol item precedes a package, symbols by id, packages by
 *   creation order); canonical code values in (length, symbol) order;
 *   each row its own MSB-first bitstream of uint32 words starting on a word
 *   boundary; rows cut into chunks of 64 symbols with a uint16 bit offset per
 *   chunk (so every chunk must start below bit 65536 of its row: the encoder
 *   refuses a page where one would not, with PQE_ERR_CAPACITY); raw nibbles
 *   two per byte, low nibble = even column.
 * Compressed page: a 256-byte header then 256-byte aligned sections:
 *   scales (s13 then s2, fp32), w13 {row_word [2I+1] u32, chunk_bit
 *   [2I*H/64] u16, nibbles [2I*H/2], words}, w2 {row_word [H+1], chunk_bit
 *   [H*I/64], nibbles [H*I/2], words}.
 * Code table (kept in VRAM, [EP] 表4): 4096 little-endian uint32 entries per
 * matrix (PQE_HUFF_LUT_BYTES), built from the code lengths; the entry of a
 * 12-bit window w (the next bits of a stream, MSB first) describes the whole
 * code words at the front of w, at most 5: bits 0-3 their total length, bits
 * 4-6 their number n, bits 7-10 the length of the first, bits 12-31 their
 * symbols, 4 bits each, the first lowest, unused slots zero. A window that no
 * code word prefixes reads length 0, n = 1, first length 0 and bit 11 set.
 * One lookup thus decodes up to 5 symbols.
 * ------------------------------------------------------------------------ */

#define PQE_HUFF_LUT_BYTES 16384

/* Upper bound of a compressed FP8 page for (H, I). */
PQE_API size_t pqe_huff_page_bound(int H, int I);

/* Host: compress one FP8 page (host bytes, layout above) into out (host,
 * out_cap bytes). Writes the page size to *out_bytes and the two code tables
 * to lut13 / lut2 (host, PQE_HUFF_LUT_BYTES each). PQE_ERR_CAPACITY when out
 * is too small or a row's chunk offsets do not fit 16 bits (such a page stays
 * uncompressed). */
PQE_API int pqe_huff_encode_page(const uint8_t *fp8_page, int H, int I, void *out, size_t out_cap,
                         size_t *out_bytes, uint8_t *lut13, uint8_t *lut2);

/* Code lengths [16] of a compressed page's two matrices (host page). */
PQE_API int pqe_huff_page_lengths(const void *comp_page, uint8_t *len13, uint8_t *len2);

/* Host: the code table (PQE_HUFF_LUT_BYTES, layout above) of canonical code
 * lengths [16]. */
PQE_API int pqe_huff_build_lut(const uint8_t *lengths, uint8_t *lut);

/* fp8_exp_huff_decode -- GPU decode of one compressed page (device, 256-byte
 * aligned) into an FP8 page (device, e.g. a slot, 16-byte aligned). lut13 /
 * lut2: resident device code tables of that expert (16-byte aligned). A row
 * that does not decode sets PQE_STATUS_CORRUPT_STREAM; its bytes are then
 * unspecified. comp_bytes bounds every read. */
PQE_API int fp8_exp_huff_decode(const void *comp_page, size_t comp_bytes, const uint8_t *lut13,
                        const uint8_t *lut2, int H, int I, uint8_t *fp8_page, int32_t *status,
                        void *stream);

/* fp8_exp_huff_decode_batch -- n pages in one kernel launch (one per 128
 * pages), all of shape (H, I). Host arrays [n]: comp_pages[i] is a compressed
 * page in device memory OR in pinned host memory (kernels read pinned memory
 * directly over the host link, so a host-tier page is pulled and decoded in
 * the same pass, [EP] 重みの圧縮: decoded on the GPU as it arrives);
 * comp_bytes[i] bounds its reads; lut13[i], lut2[i] are its device code tables;
 * fp8_pages[i] its device destination. Every pointer 16-byte aligned; the
 * destinations must not overlap each other or any source. Status as for
 * fp8_exp_huff_decode; a corrupt page does not disturb the others. */
PQE_API int fp8_exp_huff_decode_batch(int n, const void *const *comp_pages, const size_t *comp_bytes,
                                      const uint8_t *const *lut13, const uint8_t *const *lut2, int H, int I,
                                      uint8_t *const *fp8_pages, int32_t *status, void *stream);

/* slot_fill_compressed -- H2D copy of a compressed page (pinned) into a device
 * staging buffer, then fp8_exp_huff_decode into slot `dest`, both on
 * `stream`; done_event recorded after the decode. */
PQE_API int slot_fill_compressed(const pqe_pool *pool, int dest, const void *pinned_comp, size_t comp_bytes,
                         void *staging, size_t staging_bytes, const uint8_t *lut13,
                         const uint8_t *lut2, int32_t *status, void *stream, void *done_event);

/* slot_fill_compressed_batch -- refill n entries of the pool from compressed
 * host pages without a staging copy: fp8_exp_huff_decode_batch reads each
 * page (pinned, 16-byte aligned, comp_bytes[i] bytes) over the host link and
 * writes the decoded FP8 page into entry dest[i]. dest, pinned_comp,
 * comp_bytes, lut13, lut2 are host arrays [n] (lut pointers: device code
 * tables). Asynchronous on `stream`; done_event recorded after the last
 * launch if not NULL. */
PQE_API int slot_fill_compressed_batch(const pqe_pool *pool, int n, const int32_t *dest,
                                       const void *const *pinned_comp, const size_t *comp_bytes,
                                       const uint8_t *const *lut13, const uint8_t *const *lut2, int32_t *status,
                                       void *stream, void *done_event);

/* ------------------------------------------------------------------------
 * Host-RAM tier and paging file ([EP] エキスパート重みの階層ページング: each
 * MoE layer owns slots in VRAM and in host RAM, one expert per slot, both
 * tiers LRU, slot counts per layer; an expert missing from VRAM is copied from
 * its RAM slot. [EP] SSD階層: at start-up all experts of all layers are written
 * into one paging file on SSD; an expert missing from RAM too is read from it
 * by a host thread into a RAM slot, with O_DIRECT. [EP] 重みの圧縮: the RAM and
 * SSD tiers may hold compressed pages.)
 * Reading (the pages say only "LRU"): the RAM tier is accessed by the VRAM
 * tier's misses; its step is page_table_update's LRU step, with S = RAM
 * slots, over the set of experts the VRAM tier missed; a step whose set is
 * larger than S reads the missing pages into W RAM working entries and leaves
 * the RAM slots as they are. Host only.
 * ------------------------------------------------------------------------ */

/* Write n pages (host memory, bytes[i] each) into a new paging file at
 * `path`, each at a 4096-byte aligned offset (offsets[i] out, host) and padded
 * with zeros to a multiple of 4096 bytes. PQE_ERR_IO on a file error. */
PQE_API int pqe_paging_file_write(const char *path, int n, const void *const *pages, const size_t *bytes,
                                  uint64_t *offsets);

typedef struct pqe_ram_tier_config {
    int32_t E;           /* experts of the layer */
    int32_t S;           /* RAM slots (RAM_SLOTS) */
    int32_t W;           /* RAM working entries, for a step that needs more than S pages from RAM */
    int32_t n_threads;   /* reader threads, 1..64 */
    int32_t direct_io;   /* 1: read with O_DIRECT where the file system allows it */
    int32_t pad;
    uint64_t slot_bytes; /* bytes per RAM slot: a multiple of 4096, >= every page rounded up to 4096 */
} pqe_ram_tier_config;

typedef struct pqe_ram_tier pqe_ram_tier;

/* The RAM tier of one layer: expert e's page is bytes[e] bytes at offsets[e]
 * (4096-aligned) of the paging file `path`. ram: pinned host memory of (S + W)
 * * slot_bytes bytes, 4096-byte aligned, owned by the caller (entry s < S is
 * RAM slot s, S + w working entry w). Starts the reader threads. NULL on bad
 * arguments or when the file cannot be opened. */
PQE_API pqe_ram_tier *pqe_ram_tier_create(const pqe_ram_tier_config *cfg, const char *path,
                                          const uint64_t *offsets, const size_t *bytes, void *ram);
/* Stops the reader threads (after the queued reads) and closes the file. */
PQE_API void pqe_ram_tier_destroy(pqe_ram_tier *t);

/* One RAM-tier step. need [E] (host): nonzero for the experts whose pages are
 * wanted from RAM this step. Runs the LRU step, queues a file read for every
 * page not in RAM, and returns without waiting for them. Out (host, [E]):
 * ram_page[e], the RAM address of e's page (NULL if not needed);
 * read_queued[e], 1 when that page is being read from the file (valid only
 * after pqe_ram_tier_wait); *n_read, the pages read; *working, 1 for a
 * working-entry step. Waits first for the reads of the previous call. A step
 * needing more working entries than W returns PQE_ERR_CAPACITY. The caller
 * must not let the GPU read a RAM slot that a later call may refill (the
 * layer runtime orders its refills before its next step's routing read-back). */
PQE_API int pqe_ram_tier_request(pqe_ram_tier *t, const int32_t *need, const void **ram_page,
                                 int32_t *read_queued, int32_t *n_read, int32_t *working);

/* Blocks until every queued read has landed. PQE_ERR_IO if one failed. */
PQE_API int pqe_ram_tier_wait(pqe_ram_tier *t);

/* LRU state of the RAM slots (see pqe_lru_state) and running totals
 * stats[4] = pages read, bytes read, working-entry steps, O_DIRECT in use
 * (0/1). Any output may be NULL. */
PQE_API int pqe_ram_tier_state(const pqe_ram_tier *t, int32_t *slot_expert, int64_t *last_use, int64_t *step,
                               int64_t *stats);

/* Bytes of expert e's page (0 for a bad argument). */
PQE_API size_t pqe_ram_tier_page_bytes(const pqe_ram_tier *t, int expert);

/* ------------------------------------------------------------------------
 * Per-expert bit-width from importance ([PW] 技術的に面白い点: the router's
 * choices estimate each expert's importance; important experts keep more
 * bits). Importance m_e is an exponential moving average of the gate mass
 * per token: m_e <- alpha*m_e + (1-alpha) * (sum_{t,j: ids=e} g[t,j]) / T,
 * summed in ascending (t, j) in fp64. After steps every-1, 2*every-1, ... the
 * experts are ranked (m descending, ties to the lower id); the top n_hi get
 * PQE_FMT_FP8, the rest PQE_FMT_MXFP4. Host only.
 * m host fp64 [E] in/out; ids host int32 [T*k]; gates host fp32 [T*k];
 * fmt host uint8 [E] in/out; *reranked set to 1 when the formats were
 * re-ranked at this step.
 * ------------------------------------------------------------------------ */
PQE_API int pqe_importance_step(double *m, const int32_t *ids, const float *gates, int T, int k, int E,
                        double alpha, int64_t step, int every, int n_hi, uint8_t *fmt,
                        int32_t *reranked);

/* Rank without an update: the top n_hi of m get FP8, the rest MXFP4. */
PQE_API int pqe_rank_formats(const double *m, int E, int n_hi, uint8_t *fmt);

/* Quality-aware ranking ([PW] 技術的に面白い点, the feedback loop that tracks
 * quantisation error and adjusts bit widths; the scoring is a reading): expert
 * e's score is m[e] * q[e], its importance times q[e], the relative output
 * error of its 4-bit page measured on sampled tokens (pqe_expert_quant_error:
 * sqrt(sums[0] / sums[1])); the top n_hi scores keep FP8, the rest MXFP4, ties
 * to the lower id. m, q host double [E]; fmt host uint8 [E] out. Host-only. */
PQE_API int pqe_rank_formats_quality(const double *m, const double *q, int E, int n_hi, uint8_t *fmt);

/* The 4-bit quality proxy of one expert ([PW] 技術的に面白い点): runs n
 * sampled tokens x (device bf16 [n, H], 16-byte aligned) through the expert's
 * FP8 page and its MXFP4 page (device, in the layouts of pqe_page_layout),
 * both through moe_paged_ffn exactly as the layer runs them, and writes
 *   sums[0] = sum_t ||y4(x_t) - y8(x_t)||^2,  sums[1] = sum_t ||y8(x_t)||^2
 * (device double [2], fp64, deterministic order) computed from the bf16
 * outputs. Scratch: ws (device, 256-byte aligned) of at least
 * pqe_quality_workspace_size(n, H, I) bytes; both pages are copied into it.
 * status: device int32, as for moe_paged_ffn. Asynchronous on stream. */
PQE_API size_t pqe_quality_workspace_size(int n, int H, int I);
PQE_API int pqe_expert_quant_error(const void *x_bf16, int n, const uint8_t *page_fp8, const uint8_t *page_fp4,
                                   int H, int I, double *sums, void *ws, size_t ws_bytes, int32_t *status,
                                   void *stream);

/* Module-batch sizer: how many tokens to accumulate before running a layer so
 * that its expert FFN turns from weight-bound to compute-bound ([MG] 3.中核と
 * なる技術的要素: tokens are accumulated into large per-expert batches;
 * 6.今後の調査・学習の方向性: choosing the batch size). On the roofline of the
 * given ceilings (HBM GB/s, dense FP8 TFLOP/s), an expert with n rows does
 * 6 n H I FLOP against its FP8 page (pqe_page_bytes) plus a = 2 H (1 + 1/k)
 * bytes of activations per row (the token's bf16 x read once for its k rows,
 * the row's bf16 out_perm); it is compute-bound from
 *   n* = P * page / (6 H I BW - a P)   rows,
 * so with tokens routed evenly over E experts, k per token, T* = E n* / k.
 * Returns T* rounded up to a multiple of granule (>= 1), or 0 for invalid
 * arguments or when no batch reaches the knee (6 H I BW <= a P). Host-only. */
PQE_API int64_t pqe_module_batch_size(int E, int k, int H, int I, double hbm_gbs, double fp8_tflops, int granule);

/* ------------------------------------------------------------------------
 * Layer runtime -- one MoE layer over its own slot pool, one call per step.
 * A step: moe_route -> moe_permute -> per-expert counts to the host (the one
 * host synchronisation of a step; the LRU state lives on the host) ->
 * page_table_update -> every miss refilled by one slot_fill_batch (or
 * slot_fill_compressed_batch) on the side stream -> the compute stream waits
 * for the refills -> page table
 * to the device -> moe_paged_ffn -> moe_combine. Sources: [EP]
 * 階層ページング and 重みの圧縮; [MG] §3 (transfers on their own stream).
 * ------------------------------------------------------------------------ */
typedef struct pqe_layer_config {
    int32_t E, H, I, k;
    int32_t S;          /* cache slots */
    int32_t W;          /* working-buffer entries; pool->n_slots == S, pool->n_wb == W */
    int32_t max_T;      /* largest token count of a step */
    int32_t compressed; /* host pages are compressed pages (decoded after the copy) */
    int32_t device_pager; /* 1: LRU state and refills on the GPU, no host synchronisation in a step
                             (compressed host pages are pulled and decoded by a kernel that reads the
                             step's miss list on the device) */
    int32_t overlap_groups; /* device pager with a side stream given to the step: 0 refills every miss,
                               then runs the FFN once; G >= 1 (at most PQE_MAX_OVERLAP_GROUPS) refills
                               the misses in G groups on the side stream (a refill kernel on 32 CTAs)
                               while the FFN runs in passes on the step's stream: first the experts
                               already resident, then each group once its pages have landed (transfers
                               overlapped with compute, MoE-Gen summary, 3.中核となる技術的要素). The
                               FFN timing events of pqe_layer_set_ffn_events select the single pass. */
} pqe_layer_config;

#define PQE_MAX_OVERLAP_GROUPS 16

typedef struct pqe_step_info {
    int32_t n_routed;       /* |U|: experts with a non-empty batch */
    int32_t n_miss;         /* pages copied in by this step */
    int32_t working_buffer; /* 1 when |U| > S */
    int32_t n_file_read;    /* pages read from the paging file by the RAM tier (0 without one) */
    int64_t h2d_bytes;      /* bytes of host pages copied by this step */
} pqe_step_info;

typedef struct pqe_layer_buffers_t {
    int32_t *status;   /* device status word of the layer's kernels */
    int32_t *topk_ids; /* [max_T*k] of the last step */
    float *topk_w;
    int32_t *counts, *offsets, *perm_src, *inv, *page_table;
    void *out_perm;    /* bf16 [max_T*k, H] */
    void *x_in;        /* bf16 [max_T, H] staging used by pqe_layer_step_host */
    float *logits_in;  /* fp32 [max_T, E] staging used by pqe_layer_step_host */
    void *y_out;       /* bf16 [max_T, H] staging used by pqe_layer_step_host */
} pqe_layer_buffers_t;

typedef struct pqe_layer pqe_layer;

/* Device scratch a layer needs (0 for a bad config). */
PQE_API size_t pqe_layer_scratch_bytes(const pqe_layer_config *cfg);

/* host_pages [E]: pinned pointer of each expert's page (compressed page when
 * cfg->compressed), host_page_bytes [E] its size; luts_dev: device code tables
 * [E][2][PQE_HUFF_LUT_BYTES] (w13 then w2), required when compressed (host
 * pages then 16-byte aligned);
 * expert_fmt_dev: device [E] PQE_FMT_* or NULL (all FP8); scratch_dev:
 * device, 256-byte aligned, >= pqe_layer_scratch_bytes(cfg). The layer keeps
 * these pointers (caller-owned) and allocates only small pinned host buffers
 * and two CUDA events of its own. NULL on bad arguments or allocation failure. */
PQE_API pqe_layer *pqe_layer_create(const pqe_layer_config *cfg, const pqe_pool *pool,
                                    const void *const *host_pages, const size_t *host_page_bytes,
                                    const uint8_t *luts_dev, const uint8_t *expert_fmt_dev,
                                    void *scratch_dev, size_t scratch_bytes);
PQE_API void pqe_layer_destroy(pqe_layer *L);

/* Serve the layer's refills from a RAM tier (host pager only; the tier's E
 * must equal the layer's, its pages fit the layer's format: FP8 pages of at
 * most slot_stride bytes, or compressed pages when cfg->compressed). From
 * then on a VRAM miss is copied from the expert's RAM page instead of
 * host_pages: the step asks the tier for the step's misses, refills at once
 * those already in RAM, waits for the file reads, then refills the rest. The
 * layer does not own the tier; NULL detaches it. */
PQE_API int pqe_layer_attach_ram_tier(pqe_layer *L, pqe_ram_tier *t);

/* Point expert e at a new host page (e.g. after its format changed) and
 * forget its resident copy, so its next use refills the slot. */
PQE_API int pqe_layer_set_host_page(pqe_layer *L, int expert, const void *pinned_page, size_t bytes);

/* Device pointers of the layer's internal buffers. */
PQE_API int pqe_layer_buffers(pqe_layer *L, pqe_layer_buffers_t *out);

/* Optional CUDA events (timing-enabled, created by the caller) recorded on
 * the compute stream right before and right after the FFN of the next step;
 * NULL, NULL to stop. For measuring the FFN inside whole steps. A step
 * captured into a CUDA graph records them as event nodes, so each replay
 * records them again. */
PQE_API int pqe_layer_set_ffn_events(pqe_layer *L, void *ev_begin, void *ev_end);

/* pqe_layer_step_host's graph replays on (enable != 0, the default) or off
 * (every call steps eagerly). The layer keeps its graphs until destroyed. */
PQE_API int pqe_layer_set_step_graphs(pqe_layer *L, int enable);

/* The layer's LRU state (see pqe_lru_state). */
PQE_API int pqe_layer_lru_state(const pqe_layer *L, int32_t *slot_expert, int64_t *last_use, int64_t *step);

/* One step on device inputs: x_dev bf16 [T, H]; either w_router_dev fp32
 * [E, H] (logits computed, written to logits_dev if not NULL) or logits_dev
 * fp32 [T, E] given; y_dev bf16 [T, H] out. With the host pager it blocks the
 * host once, until the routing counts are known, and a working-buffer step
 * with more misses than W returns PQE_ERR_CAPACITY; side_stream NULL = refills
 * on `stream`. With the device pager nothing blocks, every launch is on
 * `stream` (the step may be captured in a CUDA graph), W must be >= E, and
 * *info is left zero (the totals are in pqe_layer_device_stats). */
PQE_API int pqe_layer_step(pqe_layer *L, const void *x_dev, const float *w_router_dev, float *logits_dev,
                           int T, void *y_dev, void *stream, void *side_stream, pqe_step_info *info);

/* Device-pager layers: the running totals (routed experts, misses,
 * working-buffer steps, refill bytes) and the LRU state; synchronises. */
PQE_API int pqe_layer_device_stats(pqe_layer *L, int64_t *stats, int32_t *slot_expert, int64_t *last_use,
                                   int64_t *step, void *stream);

/* The same step on host buffers (pinned for asynchronous copies): x_host bf16
 * [T, H] and logits_host fp32 [T, E] are copied in, y_host bf16 [T, H] is
 * copied out; returns after the stream is synchronised. On a device-pager
 * layer, a created (non-default) stream and no FFN timing events, the step's
 * launches between the copies are captured into a CUDA graph on the second
 * call with the same T, router pointer and stream pairing, and replayed on
 * later calls (at most 16 shapes kept per layer, the oldest dropped first;
 * a change of pqe_set_wait_limit or a test hook rebuilds it); the copies and
 * the synchronisation stay outside the graph. */
PQE_API int pqe_layer_step_host(pqe_layer *L, const void *x_host, const float *w_router_dev,
                                const float *logits_host, int T, void *y_host, void *stream,
                                void *side_stream, pqe_step_info *info);

#ifdef __cplusplus
}
#endif

#endif /* PQE_H */
