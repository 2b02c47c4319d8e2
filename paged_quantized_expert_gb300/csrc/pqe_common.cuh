// pqe_common.cuh -- shared device/host helpers of libpqe (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pqe.h"

namespace pqe {

// ---- host-side error plumbing ----------------------------------------------

void set_last_cuda_error(cudaError_t e);

#define PQE_CUDA_TRY(expr)                                                                     \
    do {                                                                                       \
        cudaError_t pqe_e_ = (expr);                                                           \
        if (pqe_e_ != cudaSuccess) {                                                           \
            ::pqe::set_last_cuda_error(pqe_e_);                                                \
            return PQE_ERR_CUDA;                                                               \
        }                                                                                      \
    } while (0)

#define PQE_CHECK_ARG(cond)                                                                    \
    do {                                                                                       \
        if (!(cond)) return PQE_ERR_INVALID_ARG;                                               \
    } while (0)

// every kernel launch of the library is counted (pqe_kernel_launches)
void count_launch();

#define PQE_LAUNCH_CHECK()                                                                     \
    do {                                                                                       \
        ::pqe::count_launch();                                                                 \
        PQE_CUDA_TRY(cudaGetLastError());                                                      \
    } while (0)

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// ---- programmatic dependent launch -------------------------------------------
// The kernels of a layer step are launched with programmatic stream
// serialization: a kernel may be set up while the one before it on the stream
// still runs. pdl_wait() returns once the preceding grid has completed and its
// writes are visible; pdl_trigger() lets the next kernel be set up. Both are
// no-ops in a kernel launched without the attribute. pdl_acquire() is the
// usual pair at the top of a kernel, before its first global access.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_acquire() {
    pdl_wait();
    pdl_trigger();
}

// ---- internal entry points used by the layer runtime --------------------------

// Refill groups of an overlapped step over n misses: group g of G starts at miss
// rank n - (n >> g) (halves: 1/2, 1/4, ... of the misses, the last group taking
// the rest), so the FFN pass left after the last refill is the smallest, while
// every earlier pass runs beside a refill of at least half its pages.
__host__ __device__ inline int overlap_group_start(int g, int G, int n) {
    return g >= G ? n : n - (g < 31 ? (n >> g) : 0);
}

// refill of group `group` of `groups` of a device miss list (the misses from
// overlap_group_start(group) on) by a grid of `ctas` CTAs
int slot_fill_device_group(const pqe_pool *pool, const int32_t *miss, int E, const uint64_t *host_pages,
                           const size_t *page_bytes, int group, int groups, int ctas, cudaStream_t s);

// compressed refill of group `group` of `groups` of a device miss list: each
// miss's compressed host page (comp_pages[e], comp_bytes[e], device arrays) is
// pulled and decoded into its slot; code tables at luts + e * 2 * LUT bytes;
// `ctas` decode CTAs (0: four per SM)
int slot_fill_compressed_device_group(const pqe_pool *pool, const int32_t *miss, int E, const uint64_t *comp_pages,
                                      const size_t *comp_bytes, const uint8_t *luts, int group, int groups, int ctas,
                                      int32_t *status, cudaStream_t s);

// moe_paged_ffn restricted to one pass of an overlapped step (miss non-null):
// pass 0 takes the experts that were resident (not in the miss list), pass
// g + 1 the misses of refill group g of `groups`; `reserve_sms` SMs are left to
// a refill running beside it
int moe_paged_ffn_pass(const void *x_bf16, const int32_t *perm_src, const int32_t *offsets,
                       const int32_t *page_table, const uint8_t *expert_fmt, const pqe_pool *pool, int T, int k,
                       int E, void *out_perm, void *ws, size_t ws_bytes, int32_t *status, cudaStream_t s,
                       const int32_t *miss, int groups, int pass, int reserve_sms);

template <class T>
struct ident {
    using type = T;
};

// launch with the programmatic-serialization attribute; the arguments convert
// to the kernel's parameter types
template <typename... KArgs>
int launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
               typename ident<KArgs>::type... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    PQE_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, args...));
    count_launch();
    return PQE_OK;
}

// Bounded device waits: polls before a wait gives up (pqe_set_wait_limit), and
// the test bias added to the weight stream's phase-2 target
// (pqe_test_set_phase2_bias); both are read on the host at each launch.
constexpr uint32_t DEFAULT_WAIT_LIMIT = 1u << 22;
uint32_t wait_limit();
uint32_t phase2_bias();
// Test hook (pqe_test_set_stream_kernel): which weight-stream kernel the FFN
// takes, 0 the default choice, 1 the CUDA-core stream, 2 the tensor-core
// stream where it applies; read on the host at each launch.
int stream_kernel_choice();
// Changes whenever one of the settings above does (graphs captured before it
// hold the old values).
uint64_t launch_settings_generation();

// The current device and its SM count, cached per device (a process may drive
// several GPUs; launch attributes such as the dynamic shared-memory opt-in are
// per device too). PQE_OK, PQE_ERR_CUDA, or PQE_ERR_UNSUPPORTED for a device
// index at or above PQE_MAX_DEVICES.
constexpr int PQE_MAX_DEVICES = 64;
int device_info(int &dev, int &sms);

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

__host__ __device__ inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline bool shape_ok(int H, int I) {
    return H >= 64 && H <= 16384 && H % 64 == 0 && I >= 64 && I <= 8192 && I % 64 == 0;
}

// ---- page layout (bytes) ---------------------------------------------------

struct PageLayout {
    size_t w13, w2, s13, s2, bytes;
};

__host__ __device__ inline PageLayout fp8_layout(int H, int I) {
    size_t ih = (size_t)I * H;
    return {0, 2 * ih, 3 * ih, 3 * ih + 8 * (size_t)I, 3 * ih + 8 * (size_t)I + 4 * (size_t)H};
}

__host__ __device__ inline PageLayout mxfp4_layout(int H, int I) {
    size_t ih = (size_t)I * H;
    return {0, ih, 3 * ih / 2, 3 * ih / 2 + ih / 16, 3 * ih / 2 + ih / 16 + ih / 32};
}

// ---- device helpers --------------------------------------------------------

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}

// two E4M3 codes (lo byte -> .x, hi byte -> .y) to fp32, exact
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t v) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
    float2 r;
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tcvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "r"(h2));
    return r;
}

// two E2M1 codes (low nibble -> .x, high nibble -> .y) to fp32, exact
__device__ __forceinline__ float2 e2m1x2_to_f32x2(uint8_t v) {
    uint32_t h2;
    uint16_t w = v;
    asm("{\n\t.reg .b8 b;\n\tcvt.u8.u16 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(h2) : "h"(w));
    float2 r;
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tcvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "r"(h2));
    return r;
}

// fp32 pair -> two E4M3 codes, round to nearest even, saturating (lo <- a, hi <- b)
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

// fp32 pair -> two E2M1 codes in one byte (low nibble <- a, high nibble <- b)
__device__ __forceinline__ uint8_t f32x2_to_e2m1x2(float a, float b) {
    uint16_t r;
    asm("{\n\t.reg .b8 d;\n\tcvt.rn.satfinite.e2m1x2.f32 d, %1, %2;\n\tcvt.u16.u8 %0, d;\n\t}"
        : "=h"(r)
        : "f"(b), "f"(a));
    return (uint8_t)r;
}

// 2^(b - 127) for an E8M0 byte b in [0, 254], as fp32
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
    return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

}  // namespace pqe
