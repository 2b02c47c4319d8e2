// huff.cu -- lossless compression of FP8 expert pages for the host tier, and
// its GPU decoder.
//
// Expert-pager article (rand.pepabo.com), "重みの圧縮": FP8 values have a skewed
// exponent, so per row of each expert weight matrix the exponent is Huffman-
// coded; the page is decoded on the GPU right after it is copied to VRAM; the
// code table stays resident in VRAM ("評価", Table 4 discussion).
//
// Format (the article fixes only the above; full statement in pqe.h):
// symbol = E4M3 exponent field, raw nibble = sign | mantissa; one canonical,
// length-limited (<= 12 bits) optimal code per matrix built by package-merge
// (Larmore & Hirschberg 1990); rows are MSB-first uint32 bitstreams starting on
// word boundaries, cut into chunks of 64 symbols with uint16 bit offsets.
//
// GPU decode: one thread per 64-symbol chunk, both code tables staged in
// shared memory, 12-bit window lookup per symbol, 64 output bytes written as
// four 16-byte stores. Every read is bounded by the page size; a bad stream
// sets PQE_STATUS_CORRUPT_STREAM and the thread stops.
#include <algorithm>
#include <cstring>
#include <vector>

#include "pqe_common.cuh"

namespace pqe {

constexpr int HUF_LMAX = 12;
constexpr int HUF_CHUNK = 64;
constexpr uint32_t HUF_MAGIC = 0x48455150u;  // "PQEH"
constexpr uint32_t HUF_VERSION = 1;
constexpr size_t HUF_HEADER = 256;

struct HuffMatrixDesc {
    uint64_t off_row_word, off_chunk_bit, off_nibbles, off_words, n_words;
};

struct HuffHeader {
    uint32_t magic, version;
    int32_t H, I;
    uint8_t len13[16], len2[16];
    uint64_t off_scales;
    HuffMatrixDesc m13, m2;
    uint64_t total_bytes;
};
static_assert(sizeof(HuffHeader) <= HUF_HEADER, "header too large");

// ---- host: code construction ------------------------------------------------

namespace {

struct PmItem {
    uint64_t weight;
    bool pkg;
    int order;          // symbol id, or package creation number
    uint8_t count[16];  // how many times each symbol is inside this item
};

bool pm_less(const PmItem &a, const PmItem &b) {
    if (a.weight != b.weight) return a.weight < b.weight;
    if (a.pkg != b.pkg) return !a.pkg;  // symbol before package
    return a.order < b.order;
}

// optimal prefix-code lengths with max length lmax (package-merge)
bool code_lengths(const uint64_t freq[16], int lmax, uint8_t len[16]) {
    std::memset(len, 0, 16);
    std::vector<PmItem> leaves;
    for (int s = 0; s < 16; ++s) {
        if (!freq[s]) continue;
        PmItem it{freq[s], false, s, {}};
        it.count[s] = 1;
        leaves.push_back(it);
    }
    const int n = (int)leaves.size();
    if (n == 0) return true;
    if (n == 1) {
        len[leaves[0].order] = 1;
        return true;
    }
    if ((1 << lmax) < n) return false;
    std::sort(leaves.begin(), leaves.end(), pm_less);
    std::vector<PmItem> cur = leaves;
    int made = 0;
    for (int level = 1; level < lmax; ++level) {
        std::vector<PmItem> packs;
        for (size_t i = 0; i + 1 < cur.size(); i += 2) {
            PmItem p{cur[i].weight + cur[i + 1].weight, true, made++, {}};
            for (int s = 0; s < 16; ++s) p.count[s] = (uint8_t)(cur[i].count[s] + cur[i + 1].count[s]);
            packs.push_back(p);
        }
        std::vector<PmItem> next(leaves.size() + packs.size());
        std::merge(leaves.begin(), leaves.end(), packs.begin(), packs.end(), next.begin(), pm_less);
        cur.swap(next);
    }
    for (int i = 0; i < 2 * n - 2; ++i)
        for (int s = 0; s < 16; ++s) len[s] = (uint8_t)(len[s] + cur[i].count[s]);
    return true;
}

void canonical_codes(const uint8_t len[16], uint32_t code[16]) {
    // first code of each length (RFC 1951 §3.2.2), then consecutive values in symbol order
    int bl_count[HUF_LMAX + 1] = {0};
    for (int s = 0; s < 16; ++s)
        if (len[s]) bl_count[len[s]]++;
    uint32_t next_code[HUF_LMAX + 1] = {0};
    uint32_t c = 0;
    for (int l = 1; l <= HUF_LMAX; ++l) {
        c = (c + (uint32_t)bl_count[l - 1]) << 1;
        next_code[l] = c;
    }
    for (int s = 0; s < 16; ++s) code[s] = len[s] ? next_code[len[s]]++ : 0;
}

void build_lut(const uint8_t len[16], uint8_t *lut) {
    uint32_t code[16];
    canonical_codes(len, code);
    std::memset(lut, 0, PQE_HUFF_LUT_BYTES);
    for (int s = 0; s < 16; ++s) {
        if (!len[s]) continue;
        const uint32_t lo = code[s] << (HUF_LMAX - len[s]);
        const uint32_t hi = (code[s] + 1) << (HUF_LMAX - len[s]);
        for (uint32_t w = lo; w < hi; ++w) lut[w] = (uint8_t)((s << 4) | len[s]);
    }
}

struct MatrixSizes {
    size_t row_word, chunk_bit, nibbles, words;
};

MatrixSizes matrix_sizes(int rows, int cols, uint64_t n_words) {
    return {sizeof(uint32_t) * ((size_t)rows + 1), sizeof(uint16_t) * (size_t)rows * (cols / HUF_CHUNK),
            (size_t)rows * cols / 2, sizeof(uint32_t) * n_words};
}

// encodes one matrix into dst at the offsets in d (d.n_words set by the caller)
void encode_matrix(const uint8_t *q, int rows, int cols, const uint8_t len[16], uint8_t *page,
                   const HuffMatrixDesc &d) {
    uint32_t code[16];
    canonical_codes(len, code);
    uint32_t *row_word = reinterpret_cast<uint32_t *>(page + d.off_row_word);
    uint16_t *chunk_bit = reinterpret_cast<uint16_t *>(page + d.off_chunk_bit);
    uint8_t *nib = page + d.off_nibbles;
    uint32_t *words = reinterpret_cast<uint32_t *>(page + d.off_words);
    const int nc = cols / HUF_CHUNK;
    uint32_t w = 0;
    for (int r = 0; r < rows; ++r) {
        row_word[r] = w;
        const uint8_t *qr = q + (size_t)r * cols;
        uint64_t acc = 0;  // pending bits, left-aligned count in `nacc`
        int nacc = 0;
        uint32_t bit = 0;
        for (int c = 0; c < cols; ++c) {
            if (c % HUF_CHUNK == 0) chunk_bit[(size_t)r * nc + c / HUF_CHUNK] = (uint16_t)bit;
            const int s = (qr[c] >> 3) & 15;
            acc = (acc << len[s]) | code[s];
            nacc += len[s];
            bit += len[s];
            while (nacc >= 32) {
                words[w++] = (uint32_t)(acc >> (nacc - 32));
                nacc -= 32;
            }
        }
        if (nacc > 0) words[w++] = (uint32_t)(acc << (32 - nacc));
        for (int c = 0; c < cols; c += 2) {
            const uint8_t a = qr[c], b = qr[c + 1];
            const uint8_t na = (uint8_t)(((a >> 4) & 8) | (a & 7));
            const uint8_t nb = (uint8_t)(((b >> 4) & 8) | (b & 7));
            nib[((size_t)r * cols + c) / 2] = (uint8_t)(na | (nb << 4));
        }
    }
    row_word[rows] = w;
}

uint64_t count_words(const uint8_t *q, int rows, int cols, const uint8_t len[16]) {
    uint64_t words = 0;
    for (int r = 0; r < rows; ++r) {
        uint64_t bits = 0;
        for (int c = 0; c < cols; ++c) bits += len[(q[(size_t)r * cols + c] >> 3) & 15];
        words += (bits + 31) / 32;
    }
    return words;
}

void histogram(const uint8_t *q, size_t n, uint64_t freq[16]) {
    std::memset(freq, 0, 16 * sizeof(uint64_t));
    for (size_t i = 0; i < n; ++i) freq[(q[i] >> 3) & 15]++;
}

}  // namespace

// ---- device: decoder --------------------------------------------------------

__device__ __forceinline__ bool in_page(uint64_t off, uint64_t len, uint64_t comp_bytes) {
    return off <= comp_bytes && len <= comp_bytes - off;
}

__global__ void __launch_bounds__(256) huff_decode_kernel(const uint8_t *__restrict__ comp, uint64_t comp_bytes,
                                                          const uint8_t *__restrict__ lut13,
                                                          const uint8_t *__restrict__ lut2, int H, int I,
                                                          uint8_t *__restrict__ out, int32_t *__restrict__ status) {
    __shared__ __align__(16) uint8_t lut[2][PQE_HUFF_LUT_BYTES];
    for (int i = threadIdx.x; i < PQE_HUFF_LUT_BYTES / 16; i += blockDim.x) {
        reinterpret_cast<uint4 *>(lut[0])[i] = __ldg(reinterpret_cast<const uint4 *>(lut13) + i);
        reinterpret_cast<uint4 *>(lut[1])[i] = __ldg(reinterpret_cast<const uint4 *>(lut2) + i);
    }
    __syncthreads();
    if (comp_bytes < HUF_HEADER) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, PQE_STATUS_CORRUPT_STREAM);
        return;
    }
    const HuffHeader hd = *reinterpret_cast<const HuffHeader *>(comp);
    const PageLayout L = fp8_layout(H, I);
    const uint64_t n_scale = 2 * (uint64_t)I + H;
    const uint64_t r13 = 2 * (uint64_t)I, r2 = H;
    const uint64_t nc13 = H / HUF_CHUNK, nc2 = I / HUF_CHUNK;
    bool ok = hd.magic == HUF_MAGIC && hd.version == HUF_VERSION && hd.H == H && hd.I == I &&
              in_page(hd.off_scales, 4 * n_scale, comp_bytes) &&
              in_page(hd.m13.off_row_word, 4 * (r13 + 1), comp_bytes) &&
              in_page(hd.m13.off_chunk_bit, 2 * r13 * nc13, comp_bytes) &&
              in_page(hd.m13.off_nibbles, r13 * H / 2, comp_bytes) &&
              hd.m13.n_words < (comp_bytes >> 2) && in_page(hd.m13.off_words, 4 * hd.m13.n_words, comp_bytes) &&
              in_page(hd.m2.off_row_word, 4 * (r2 + 1), comp_bytes) &&
              in_page(hd.m2.off_chunk_bit, 2 * r2 * nc2, comp_bytes) &&
              in_page(hd.m2.off_nibbles, r2 * I / 2, comp_bytes) &&
              hd.m2.n_words < (comp_bytes >> 2) && in_page(hd.m2.off_words, 4 * hd.m2.n_words, comp_bytes) &&
              (hd.off_scales % 4) == 0 && (hd.m13.off_row_word % 4) == 0 && (hd.m13.off_chunk_bit % 2) == 0 &&
              (hd.m13.off_nibbles % 16) == 0 && (hd.m13.off_words % 4) == 0 && (hd.m2.off_row_word % 4) == 0 &&
              (hd.m2.off_chunk_bit % 2) == 0 && (hd.m2.off_nibbles % 16) == 0 && (hd.m2.off_words % 4) == 0;
    if (!ok) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, PQE_STATUS_CORRUPT_STREAM);
        return;
    }
    const uint64_t gid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // scales are copied raw
    if (gid < n_scale) {
        reinterpret_cast<float *>(out + L.s13)[gid] = reinterpret_cast<const float *>(comp + hd.off_scales)[gid];
    }
    const uint64_t n13 = r13 * nc13, n2 = r2 * nc2;
    if (gid >= n13 + n2) return;
    const bool first = gid < n13;
    const HuffMatrixDesc &d = first ? hd.m13 : hd.m2;
    const uint64_t g = first ? gid : gid - n13;
    const int cols = first ? H : I;
    const uint64_t nc = first ? nc13 : nc2;
    const uint64_t r = g / nc, c = g % nc;
    const uint8_t *lt = lut[first ? 0 : 1];
    const uint32_t *row_word = reinterpret_cast<const uint32_t *>(comp + d.off_row_word);
    const uint32_t *words = reinterpret_cast<const uint32_t *>(comp + d.off_words);
    const uint32_t w0 = row_word[r], w1 = row_word[r + 1];
    if (w1 < w0 || w1 > d.n_words) {
        atomicOr(status, PQE_STATUS_CORRUPT_STREAM);
        return;
    }
    const uint32_t row_bits = (w1 - w0) * 32u;
    uint32_t pos = reinterpret_cast<const uint16_t *>(comp + d.off_chunk_bit)[g];
    const uint4 *nibp = reinterpret_cast<const uint4 *>(comp + d.off_nibbles + (r * cols + c * HUF_CHUNK) / 2);
    const uint4 n0 = nibp[0], n1 = nibp[1];
    const uint32_t nibw[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
    uint32_t outw[16];
    const uint32_t *wr = words + w0;
    const uint32_t nwr = w1 - w0;
#pragma unroll 4
    for (int i = 0; i < HUF_CHUNK; ++i) {
        if (pos >= row_bits) {
            atomicOr(status, PQE_STATUS_CORRUPT_STREAM);
            return;
        }
        const uint32_t wi = pos >> 5, sh = pos & 31;
        const uint64_t two = ((uint64_t)wr[wi] << 32) | (wi + 1 < nwr ? wr[wi + 1] : 0u);
        const uint32_t win = (uint32_t)(two >> (52 - sh)) & 0xFFFu;
        const uint32_t ent = lt[win];
        const uint32_t len = ent & 15u;
        if (len == 0 || pos + len > row_bits) {
            atomicOr(status, PQE_STATUS_CORRUPT_STREAM);
            return;
        }
        pos += len;
        const uint32_t nb = (nibw[i >> 3] >> (4 * (i & 7))) & 15u;
        const uint32_t byte = ((nb & 8u) << 4) | ((ent >> 4) << 3) | (nb & 7u);
        if ((i & 3) == 0) outw[i >> 2] = byte;
        else outw[i >> 2] |= byte << (8 * (i & 3));
    }
    uint4 *dst = reinterpret_cast<uint4 *>(out + (first ? L.w13 : L.w2) + r * cols + c * HUF_CHUNK);
    dst[0] = make_uint4(outw[0], outw[1], outw[2], outw[3]);
    dst[1] = make_uint4(outw[4], outw[5], outw[6], outw[7]);
    dst[2] = make_uint4(outw[8], outw[9], outw[10], outw[11]);
    dst[3] = make_uint4(outw[12], outw[13], outw[14], outw[15]);
}

}  // namespace pqe

using namespace pqe;

extern "C" {

size_t pqe_huff_page_bound(int H, int I) {
    if (!shape_ok(H, I)) return 0;
    const int r13 = 2 * I, r2 = H;
    // worst case: every symbol at the maximum length, plus a padding word per row
    const uint64_t w13 = ((uint64_t)r13 * H * HUF_LMAX + 31) / 32 + r13;
    const uint64_t w2 = ((uint64_t)r2 * I * HUF_LMAX + 31) / 32 + r2;
    const MatrixSizes a = matrix_sizes(r13, H, w13), b = matrix_sizes(r2, I, w2);
    return HUF_HEADER + round_up(4 * (2 * (size_t)I + H), 256) + round_up(a.row_word, 256) +
           round_up(a.chunk_bit, 256) + round_up(a.nibbles, 256) + round_up(a.words, 256) +
           round_up(b.row_word, 256) + round_up(b.chunk_bit, 256) + round_up(b.nibbles, 256) +
           round_up(b.words, 256);
}

int pqe_huff_encode_page(const uint8_t *fp8_page, int H, int I, void *out, size_t out_cap, size_t *out_bytes,
                         uint8_t *lut13, uint8_t *lut2) {
    if (!fp8_page || !out || !out_bytes || !shape_ok(H, I)) return PQE_ERR_INVALID_ARG;
    const PageLayout L = fp8_layout(H, I);
    const uint8_t *q13 = fp8_page + L.w13, *q2 = fp8_page + L.w2;
    const int r13 = 2 * I, r2 = H;
    HuffHeader hd;
    std::memset(&hd, 0, sizeof(hd));
    hd.magic = HUF_MAGIC;
    hd.version = HUF_VERSION;
    hd.H = H;
    hd.I = I;
    uint64_t f13[16], f2[16];
    histogram(q13, (size_t)r13 * H, f13);
    histogram(q2, (size_t)r2 * I, f2);
    if (!code_lengths(f13, HUF_LMAX, hd.len13) || !code_lengths(f2, HUF_LMAX, hd.len2)) return PQE_ERR_CORRUPT;
    const uint64_t nw13 = count_words(q13, r13, H, hd.len13), nw2 = count_words(q2, r2, I, hd.len2);
    size_t off = HUF_HEADER;
    hd.off_scales = off;
    off += round_up(4 * (2 * (size_t)I + H), 256);
    const MatrixSizes a = matrix_sizes(r13, H, nw13), b = matrix_sizes(r2, I, nw2);
    hd.m13.off_row_word = off; off += round_up(a.row_word, 256);
    hd.m13.off_chunk_bit = off; off += round_up(a.chunk_bit, 256);
    hd.m13.off_nibbles = off; off += round_up(a.nibbles, 256);
    hd.m13.off_words = off; off += round_up(a.words, 256);
    hd.m13.n_words = nw13;
    hd.m2.off_row_word = off; off += round_up(b.row_word, 256);
    hd.m2.off_chunk_bit = off; off += round_up(b.chunk_bit, 256);
    hd.m2.off_nibbles = off; off += round_up(b.nibbles, 256);
    hd.m2.off_words = off; off += round_up(b.words, 256);
    hd.m2.n_words = nw2;
    hd.total_bytes = off;
    if (off > out_cap) return PQE_ERR_CAPACITY;
    uint8_t *page = static_cast<uint8_t *>(out);
    std::memset(page, 0, off);
    std::memcpy(page, &hd, sizeof(hd));
    std::memcpy(page + hd.off_scales, fp8_page + L.s13, 4 * (2 * (size_t)I + H));
    encode_matrix(q13, r13, H, hd.len13, page, hd.m13);
    encode_matrix(q2, r2, I, hd.len2, page, hd.m2);
    *out_bytes = off;
    if (lut13) build_lut(hd.len13, lut13);
    if (lut2) build_lut(hd.len2, lut2);
    return PQE_OK;
}

int pqe_huff_page_lengths(const void *comp_page, uint8_t *len13, uint8_t *len2) {
    if (!comp_page) return PQE_ERR_INVALID_ARG;
    HuffHeader hd;
    std::memcpy(&hd, comp_page, sizeof(hd));
    if (hd.magic != HUF_MAGIC || hd.version != HUF_VERSION) return PQE_ERR_CORRUPT;
    if (len13) std::memcpy(len13, hd.len13, 16);
    if (len2) std::memcpy(len2, hd.len2, 16);
    return PQE_OK;
}

// host helper: the canonical code table of given lengths (for tests and setup)
int pqe_huff_build_lut(const uint8_t *lengths, uint8_t *lut) {
    if (!lengths || !lut) return PQE_ERR_INVALID_ARG;
    build_lut(lengths, lut);
    return PQE_OK;
}

int fp8_exp_huff_decode(const void *comp_page, size_t comp_bytes, const uint8_t *lut13, const uint8_t *lut2, int H,
                        int I, uint8_t *fp8_page, int32_t *status, void *stream) {
    PQE_CHECK_ARG(comp_page && lut13 && lut2 && fp8_page && status && shape_ok(H, I));
    PQE_CHECK_ARG(aligned(comp_page, 256) && aligned(fp8_page, 16) && aligned(lut13, 16) && aligned(lut2, 16));
    const uint64_t chunks = (uint64_t)2 * I * (H / HUF_CHUNK) + (uint64_t)H * (I / HUF_CHUNK);
    const uint64_t n_scale = 2 * (uint64_t)I + H;
    const uint64_t threads = chunks > n_scale ? chunks : n_scale;
    const unsigned grid = (unsigned)((threads + 255) / 256);
    huff_decode_kernel<<<grid, 256, 0, as_stream(stream)>>>(static_cast<const uint8_t *>(comp_page), comp_bytes,
                                                            lut13, lut2, H, I, fp8_page, status);
    PQE_LAUNCH_CHECK();
    return PQE_OK;
}

int slot_fill_compressed(const pqe_pool *pool, int dest, const void *pinned_comp, size_t comp_bytes, void *staging,
                         size_t staging_bytes, const uint8_t *lut13, const uint8_t *lut2, int32_t *status,
                         void *stream, void *done_event) {
    uint8_t *dst = static_cast<uint8_t *>(pqe_pool_slot_addr(pool, dest));
    PQE_CHECK_ARG(dst && pinned_comp && staging);
    PQE_CHECK_ARG(comp_bytes >= HUF_HEADER && comp_bytes <= staging_bytes);
    auto s = as_stream(stream);
    PQE_CUDA_TRY(cudaMemcpyAsync(staging, pinned_comp, comp_bytes, cudaMemcpyHostToDevice, s));
    int rc = fp8_exp_huff_decode(staging, comp_bytes, lut13, lut2, pool->H, pool->I, dst, status, stream);
    if (rc != PQE_OK) return rc;
    if (done_event) PQE_CUDA_TRY(cudaEventRecord(reinterpret_cast<cudaEvent_t>(done_event), s));
    return PQE_OK;
}

}  // extern "C"
