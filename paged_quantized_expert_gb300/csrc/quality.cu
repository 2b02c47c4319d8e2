// quality.cu -- the 4-bit quality proxy of one expert: how far its MXFP4
// page's output lies from its FP8 page's on a sample of tokens.
//
// The PagedWeight article ("技術的に面白い点", the quality feedback loop)
// tracks the error that quantisation introduces and feeds it back into the
// choice of bit widths. With no trained model to score, the proxy here is the
// output error itself: for sampled tokens x_t, sum_t ||y4(x_t) - y8(x_t)||^2
// and sum_t ||y8(x_t)||^2, where y8 / y4 run the expert's SwiGLU FFN from its
// FP8 / MXFP4 page. Both pages run through moe_paged_ffn as the two experts of
// a two-slot pool in the caller's workspace, every token routed to both, so
// the proxy measures exactly the arithmetic the layer uses.
#include <algorithm>

#include "pqe_common.cuh"

namespace pqe {
namespace qp {

struct QpWs {
    size_t pool, perm, offsets, table, fmt, out, part, ffn, total;
};

// the n x H outputs are summed by QP_BLOCKS(n H) CTAs of 2048 elements each
// (at most 256), whose fp64 partial pairs one CTA then adds in a fixed order:
// the result depends on n and H only, not on the device
constexpr int QP_CHUNK = 2048;
constexpr int QP_MAX_BLOCKS = 256;
static int qp_blocks(long nH) { return (int)std::min<long>(QP_MAX_BLOCKS, (nH + QP_CHUNK - 1) / QP_CHUNK); }

static QpWs qp_layout(int n, int H, int I) {
    QpWs w{};
    size_t off = 0;
    auto take = [&off](size_t b) {
        const size_t at = off;
        off += round_up(b ? b : 1, 256);
        return at;
    };
    w.pool = take(2 * pqe_slot_stride(H, I));
    w.perm = take(sizeof(int32_t) * 2 * (size_t)n);
    w.offsets = take(sizeof(int32_t) * 3);
    w.table = take(sizeof(int32_t) * 2);
    w.fmt = take(2);
    w.out = take(sizeof(uint16_t) * 2 * (size_t)n * H);
    w.part = take(sizeof(double) * 2 * QP_MAX_BLOCKS);
    w.ffn = take(moe_paged_ffn_workspace_size(n, 2, 2, H, I));
    w.total = off;
    return w;
}

// expert 0 = the FP8 page (slot 0), expert 1 = the MXFP4 page (slot 1); token t
// is routed to both (flat indices 2t and 2t+1), so batch rows 0..n-1 are
// expert 0's and n..2n-1 expert 1's
__global__ void qp_setup_kernel(int n, int32_t *perm, int32_t *offsets, int32_t *table, uint8_t *fmt) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < 2 * n; i += gridDim.x * blockDim.x)
        perm[i] = i < n ? 2 * i : 2 * (i - n) + 1;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        offsets[0] = 0;
        offsets[1] = n;
        offsets[2] = 2 * n;
        table[0] = 0;
        table[1] = 1;
        fmt[0] = PQE_FMT_FP8;
        fmt[1] = PQE_FMT_MXFP4;
    }
}

// fixed-order tree over the 256 threads' fp64 values (d, r); thread 0 ends
// with the totals
__device__ void qp_block_sum(double &d, double &r) {
    __shared__ double sd[256], sr[256];
    sd[threadIdx.x] = d;
    sr[threadIdx.x] = r;
    __syncthreads();
    for (int o = 128; o >= 1; o >>= 1) {
        if ((int)threadIdx.x < o) {
            sd[threadIdx.x] += sd[threadIdx.x + o];
            sr[threadIdx.x] += sr[threadIdx.x + o];
        }
        __syncthreads();
    }
    d = sd[0];
    r = sr[0];
}

// part[2b], part[2b+1] = sum (y4 - y8)^2, sum y8^2 over CTA b's stride of the
// n x H outputs (rows 0..n-1 of out are y8, rows n..2n-1 y4)
__global__ void __launch_bounds__(256) qp_partial_kernel(const uint16_t *__restrict__ out, long nH, double *part) {
    double d2 = 0.0, r2 = 0.0;
    for (long i = (long)blockIdx.x * 256 + threadIdx.x; i < nH; i += (long)gridDim.x * 256) {
        const double y8 = bf16_to_f32(out[i]), y4 = bf16_to_f32(out[nH + i]);
        d2 += (y4 - y8) * (y4 - y8);
        r2 += y8 * y8;
    }
    qp_block_sum(d2, r2);
    if (threadIdx.x == 0) {
        part[2 * blockIdx.x] = d2;
        part[2 * blockIdx.x + 1] = r2;
    }
}

__global__ void __launch_bounds__(256) qp_final_kernel(const double *__restrict__ part, int nb, double *sums) {
    double d2 = 0.0, r2 = 0.0;
    if ((int)threadIdx.x < nb) {
        d2 = part[2 * threadIdx.x];
        r2 = part[2 * threadIdx.x + 1];
    }
    qp_block_sum(d2, r2);
    if (threadIdx.x == 0) {
        sums[0] = d2;
        sums[1] = r2;
    }
}

}  // namespace qp
}  // namespace pqe

using namespace pqe;

extern "C" {

size_t pqe_quality_workspace_size(int n, int H, int I) {
    if (n < 1 || !shape_ok(H, I)) return 0;
    return qp::qp_layout(n, H, I).total;
}

int pqe_expert_quant_error(const void *x_bf16, int n, const uint8_t *page_fp8, const uint8_t *page_fp4, int H, int I,
                           double *sums, void *ws, size_t ws_bytes, int32_t *status, void *stream) {
    PQE_CHECK_ARG(n >= 1 && shape_ok(H, I));
    PQE_CHECK_ARG(x_bf16 && page_fp8 && page_fp4 && sums && ws && status);
    PQE_CHECK_ARG(aligned(x_bf16, 16) && aligned(ws, 256) && aligned(sums, 8));
    PQE_CHECK_ARG(ws_bytes >= pqe_quality_workspace_size(n, H, I));
    const qp::QpWs w = qp::qp_layout(n, H, I);
    uint8_t *b = static_cast<uint8_t *>(ws);
    cudaStream_t s = as_stream(stream);
    const size_t stride = pqe_slot_stride(H, I);
    PQE_CUDA_TRY(cudaMemcpyAsync(b + w.pool, page_fp8, pqe_page_bytes(PQE_FMT_FP8, H, I), cudaMemcpyDeviceToDevice, s));
    PQE_CUDA_TRY(cudaMemcpyAsync(b + w.pool + stride, page_fp4, pqe_page_bytes(PQE_FMT_MXFP4, H, I),
                                 cudaMemcpyDeviceToDevice, s));
    int32_t *perm = reinterpret_cast<int32_t *>(b + w.perm);
    int32_t *offsets = reinterpret_cast<int32_t *>(b + w.offsets);
    int32_t *table = reinterpret_cast<int32_t *>(b + w.table);
    uint8_t *fmt = b + w.fmt;
    qp::qp_setup_kernel<<<(2 * n + 255) / 256, 256, 0, s>>>(n, perm, offsets, table, fmt);
    PQE_LAUNCH_CHECK();
    pqe_pool pool{};
    pool.base = b + w.pool;
    pool.wb_base = nullptr;
    pool.slot_stride = stride;
    pool.n_slots = 2;
    pool.n_wb = 0;
    pool.H = H;
    pool.I = I;
    uint16_t *out = reinterpret_cast<uint16_t *>(b + w.out);
    const int rc = moe_paged_ffn(x_bf16, perm, offsets, table, fmt, &pool, n, 2, 2, out, b + w.ffn,
                                 ws_bytes - w.ffn, status, stream);
    if (rc != PQE_OK) return rc;
    const long nH = (long)n * H;
    const int nb = qp::qp_blocks(nH);
    double *part = reinterpret_cast<double *>(b + w.part);
    qp::qp_partial_kernel<<<nb, 256, 0, s>>>(out, nH, part);
    PQE_LAUNCH_CHECK();
    qp::qp_final_kernel<<<1, 256, 0, s>>>(part, nb, sums);
    PQE_LAUNCH_CHECK();
    return PQE_OK;
}

}  // extern "C"
