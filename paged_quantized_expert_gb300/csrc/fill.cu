// fill.cu -- refill of many slots from the pinned host tier with one kernel.
//
// Expert-pager article (rand.pepabo.com), "エキスパート重みの階層ページング": a
// missing expert is copied from its host-RAM slot into a VRAM slot. On GB300
// the host tier is reached over NVLink-C2C; pinned host memory is addressable
// from kernels (unified addressing), so the SMs stream every missed page of a
// step in one persistent launch: every warp walks 8 KiB segments of the
// concatenated pages with sixteen 16-byte loads in flight per lane, enough
// outstanding reads to fill the link, which a sequence of per-page copies
// does not.
#include "pqe_common.cuh"

namespace pqe {

constexpr int FILL_MAX = 128;           // pages per launch (kernel parameter block < 4 KiB)
constexpr int FILL_THREADS = 512;
constexpr int FILL_UNROLL = 16;         // 16-byte loads in flight per lane
constexpr uint32_t FILL_SEG = 32 * FILL_UNROLL * 16;  // 8 KiB per warp segment

struct FillBatch {
    const uint4 *src[FILL_MAX];
    uint4 *dst[FILL_MAX];
    uint32_t n16[FILL_MAX];     // 16-byte words per page
    uint32_t seg0[FILL_MAX + 1];  // first segment of each page (prefix), seg0[n] = total
    int n;
};

// persistent: every warp walks segments seg = warp_id + k * n_warps of the
// concatenated pages; segment -> page by binary search over seg0
__global__ void __launch_bounds__(FILL_THREADS) fill_batch_kernel(const __grid_constant__ FillBatch b) {
    const int lane = threadIdx.x & 31;
    const uint32_t nwarps = gridDim.x * (FILL_THREADS / 32);
    const uint32_t total = b.seg0[b.n];
    for (uint32_t seg = blockIdx.x * (FILL_THREADS / 32) + (threadIdx.x >> 5); seg < total; seg += nwarps) {
        int lo = 0, hi = b.n - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (b.seg0[mid] <= seg) lo = mid;
            else hi = mid - 1;
        }
        const uint32_t n16 = b.n16[lo];
        const uint32_t base = (seg - b.seg0[lo]) * (FILL_SEG / 16);
        const uint4 *__restrict__ src = b.src[lo];
        uint4 *__restrict__ dst = b.dst[lo];
        uint4 v[FILL_UNROLL];
#pragma unroll
        for (int u = 0; u < FILL_UNROLL; ++u) {
            const uint32_t w = base + u * 32 + lane;
            if (w < n16) v[u] = src[w];
        }
#pragma unroll
        for (int u = 0; u < FILL_UNROLL; ++u) {
            const uint32_t w = base + u * 32 + lane;
            if (w < n16) dst[w] = v[u];
        }
    }
}

}  // namespace pqe

using namespace pqe;

extern "C" {

int slot_fill_batch(const pqe_pool *pool, int n, const int32_t *dest, const void *const *host_src,
                    const size_t *bytes, void *stream, void *done_event) {
    PQE_CHECK_ARG(pool && n >= 0 && (n == 0 || (dest && host_src && bytes)));
    cudaStream_t s = as_stream(stream);
    for (int i = 0; i < n; ++i) {  // all arguments are checked before the first launch
        uint8_t *d = static_cast<uint8_t *>(pqe_pool_slot_addr(pool, dest[i]));
        const size_t nb = bytes[i];
        PQE_CHECK_ARG(d && host_src[i] && nb > 0 && nb <= pool->slot_stride && nb % 16 == 0);
        PQE_CHECK_ARG(aligned(host_src[i], 16) && aligned(d, 16));
    }
    int dev = 0, sms = 0;
    const int di = device_info(dev, sms);
    if (di != PQE_OK) return di;
    for (int i0 = 0; i0 < n; i0 += FILL_MAX) {
        FillBatch b{};
        b.n = (n - i0 < FILL_MAX) ? n - i0 : FILL_MAX;
        uint32_t segs = 0;
        for (int j = 0; j < b.n; ++j) {
            const size_t nb = bytes[i0 + j];
            b.src[j] = static_cast<const uint4 *>(host_src[i0 + j]);
            b.dst[j] = static_cast<uint4 *>(pqe_pool_slot_addr(pool, dest[i0 + j]));
            b.n16[j] = (uint32_t)(nb / 16);
            b.seg0[j] = segs;
            segs += (uint32_t)((nb + FILL_SEG - 1) / FILL_SEG);
        }
        b.seg0[b.n] = segs;
        const uint32_t warps = FILL_THREADS / 32;
        uint32_t blocks = (segs + warps - 1) / warps;
        if (blocks > (uint32_t)sms) blocks = sms;
        fill_batch_kernel<<<blocks, FILL_THREADS, 0, s>>>(b);
        PQE_LAUNCH_CHECK();
    }
    if (done_event) PQE_CUDA_TRY(cudaEventRecord(reinterpret_cast<cudaEvent_t>(done_event), s));
    return PQE_OK;
}

}  // extern "C"
