// ffn_internal.cuh -- argument block shared by the expert-FFN kernels (internal).
#pragma once

#include <stdint.h>

namespace pqe {

struct FfnArgs {
    const uint16_t *x;           // bf16 [T, H]
    const int32_t *perm_src;     // [T*k]
    const int32_t *offsets;      // [E+1]
    const int32_t *page_table;   // [E]
    const uint8_t *expert_fmt;   // [E] or null (all FP8)
    const uint8_t *pool_base;    // cache slots
    const uint8_t *wb_base;      // working-buffer entries
    size_t slot_stride;
    int n_slots;                 // cache slots
    int n_wb;                    // working-buffer entries
    int T, k, E, H, I;
    int32_t *sched;              // [E+1]: count, then active expert ids
    int32_t *wpre;               // [E+1]: prefix of per-expert work weights over sched (stream kernel)
    int4 *info;                  // [E]: per expert of sched, {e, first batch row, batch rows, page entry
                                 // (24 bits, sign-extended) | format << 24}, written by the schedule
    float *h;                    // fp32 [T*k, I]
    uint16_t *out_perm;          // bf16 [T*k, H]
    int32_t *status;
    uint32_t *done13;            // [E + 1] stream kernels: phase-1 work combined per expert, then the
                                 // tensor-core stream's grab counter (all zeroed by the schedule)
    uint32_t wait_limit;         // polls of a bounded wait before it gives up
    uint32_t phase2_bias;        // test hook: added to the phase-2 target (0 in normal use)
};

// the schedule's record of an expert's page-table entry and format
__host__ __device__ __forceinline__ int info_pack(int slot, int fmt) { return (slot & 0x00FFFFFF) | (fmt << 24); }
__host__ __device__ __forceinline__ int info_slot(int w) { return (int)((unsigned)w << 8) >> 8; }
__host__ __device__ __forceinline__ int info_fmt(int w) { return (int)((unsigned)w >> 24); }

// address of page-table entry `slot` (valid: 0 <= slot < n_slots + n_wb)
__device__ __forceinline__ const uint8_t *page_addr(const FfnArgs &a, int slot) {
    return slot < a.n_slots ? a.pool_base + (size_t)slot * a.slot_stride
                            : a.wb_base + (size_t)(slot - a.n_slots) * a.slot_stride;
}

// scratch of the tensor-core path (all device, inside the FFN workspace)
struct TcBuffers {
    long A;
    int32_t *tiles;      // [max_tiles][4]: expert, first batch row, valid rows, page-table entry
    int32_t *n_tiles;    // [3]: all tiles, FP8 tiles (first in the list), MXFP4 tiles (after them)
    uint8_t *xt;         // E4M3 [T, H] activations per token
    float *st;           // [T] their row scales
    uint8_t *xq;         // E4M3 [A, H] the same rows in batch order
    float *sx;           // [A] their row scales
    uint16_t *h;         // bf16 [A, I]
    uint32_t *hmax;      // [A] row amax of h (fp32 bits)
    uint8_t *hq;         // E4M3 [A, I]
    float *sh;           // [A]
};

// batches of at least this many rows (FP8 pages) take the tcgen05 path; the
// weight stream handles up to 8 tokens in one mma column group, so its cost up
// to here is that of reading the weights once
constexpr int TC_MIN_ROWS = 9;

// Decode-sized steps (at most DECODE_ROWS_PER_EXPERT rows per routed expert on
// average) run the tensor-core batches beside the weight stream: the stream
// kernel leaves TC_SIDE_SMS SMs free and the tensor-core kernels, on a side
// stream, use at most that many persistent CTAs. The weight stream is bound
// per SM by its consumers, so it gives up about TC_SIDE_SMS / SMs of its rate,
// while the tensor-core chain (a few latency-bound launches) no longer adds to
// the step.
constexpr int TC_SIDE_SMS = 16;
constexpr int DECODE_ROWS_PER_EXPERT = 4;
// Beside the tensor-core weight stream the side chain gets more SMs: that
// stream takes a larger share of HBM per SM, so with 16 the side chain
// finished last (a T=64 decode step: 97 us against the stream's 89 us; with
// 24, 77 us against 92 us).
constexpr int TC_SIDE_SMS_TC_STREAM = 24;

// The weight stream runs on the tensor cores (ffn_stream_tc.cu) when a layer's
// pages are all FP8 and a step routes at least this many experts: its work
// items are 128-row tiles of whole K, so fewer experts leave SMs without work,
// and the CUDA-core stream (16-row units) is then the faster one.
constexpr int STREAM_TC_MIN_EXPERTS = 32;

bool tc_shape_ok(int H, int I);
bool stream_shape_ok(int H, int I);
// grid: CTAs of the persistent stream kernel, 0 = one per SM
int launch_ffn_stream(const FfnArgs &args, cudaStream_t s, int grid = 0);
// the same FFN on the tensor cores (tcgen05, FP8 pages only: expert_fmt null)
bool stream_tc_shape_ok(int H, int I);
int launch_ffn_stream_tc(const FfnArgs &args, cudaStream_t s, int grid = 0);
int launch_ffn_gemv(const FfnArgs &args, int max_active, cudaStream_t s);
// sm_cap: at most this many persistent GEMM CTAs, 0 = one per SM
int launch_ffn_tc(const FfnArgs &args, const TcBuffers &b, int max_tiles, cudaStream_t s, int sm_cap = 0);

}  // namespace pqe
