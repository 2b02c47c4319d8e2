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
// Code table (resident in VRAM, built on the host from the code lengths): for
// every 12-bit window, the whole code words at its front, at most 5, with
// their symbols and lengths, so one lookup decodes several symbols.
//
// GPU decode: a batch of pages per launch, one CTA per block of chunks of one
// matrix; described with the kernel below.
#include <algorithm>
#include <atomic>
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

// Multi-symbol code table: entry w (a 12-bit window, MSB first) describes the
// whole code words at the front of w, at most 5:
//   bits 0-3   t, their total length (0 when no code word prefixes w),
//   bits 4-6   n, their number (1 when no code word prefixes w),
//   bits 7-10  the length of the first (0 when none),
//   bit 11     set when no code word prefixes w (a corrupt stream),
//   bits 12-31 their symbols, 4 bits each, the first lowest (unused: 0).
// An invalid window thus yields one symbol and consumes no bits, so a decoder
// needs no early exit: it finishes its 64 symbols and reports bit 11.
void build_lut(const uint8_t len[16], uint8_t *lut_bytes) {
    uint32_t code[16];
    canonical_codes(len, code);
    uint8_t one[1 << HUF_LMAX];  // (symbol << 4) | length of the code word that prefixes a window
    std::memset(one, 0, sizeof(one));
    for (int s = 0; s < 16; ++s) {
        if (!len[s]) continue;
        const uint32_t lo = code[s] << (HUF_LMAX - len[s]);
        const uint32_t hi = (code[s] + 1) << (HUF_LMAX - len[s]);
        for (uint32_t w = lo; w < hi; ++w) one[w] = (uint8_t)((s << 4) | len[s]);
    }
    for (uint32_t w = 0; w < (1u << HUF_LMAX); ++w) {
        uint32_t n = 0, pos = 0, l0 = 0, syms = 0;
        while (n < 5) {
            const uint32_t e = one[(w << pos) & ((1u << HUF_LMAX) - 1)], l = e & 15u;
            if (l == 0 || pos + l > (uint32_t)HUF_LMAX) break;  // no whole code word left in the window
            if (n == 0) l0 = l;
            syms |= (e >> 4) << (4 * n);
            pos += l;
            ++n;
        }
        const uint32_t ent = n ? (pos | n << 4 | l0 << 7 | syms << 12) : (1u << 4 | 1u << 11);
        std::memcpy(lut_bytes + 4 * (size_t)w, &ent, 4);  // little-endian u32, as the device reads it
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

// code words of a matrix; false when a chunk would start at bit 65536 or later
// of its row (chunk offsets are 16-bit)
bool count_words(const uint8_t *q, int rows, int cols, const uint8_t len[16], uint64_t *words) {
    *words = 0;
    for (int r = 0; r < rows; ++r) {
        uint64_t bits = 0;
        for (int c = 0; c < cols; ++c) {
            if (c % HUF_CHUNK == 0 && bits > 0xFFFFu) return false;
            bits += len[(q[(size_t)r * cols + c] >> 3) & 15];
        }
        *words += (bits + 31) / 32;
    }
    return true;
}

void histogram(const uint8_t *q, size_t n, uint64_t freq[16]) {
    std::memset(freq, 0, 16 * sizeof(uint64_t));
    for (size_t i = 0; i < n; ++i) freq[(q[i] >> 3) & 15]++;
}

}  // namespace

// ---- device: decoder --------------------------------------------------------
//
// One launch decodes a batch of pages. A CTA takes one block of at most 512
// consecutive 64-symbol chunks of one matrix (whole rows), so the grid is
// pages x blocks per page:
//   1. it loads the block's code table (16 KiB, resident in VRAM), its row word
//      offsets and chunk bit offsets (the source may be device memory or
//      pinned host memory read over the host link);
//   2. it stages the block's code words in shared memory (16-byte loads) and
//      each thread decodes two chunks: two neighbours of one row as a single
//      128-symbol run where rows have an even number of chunks, else two
//      chunks one after the other. One table lookup yields every whole code
//      word at the front of the 12-bit window (up to 5), the exponent nibbles
//      collect in a 64-bit accumulator and leave eight at a time into a shared
//      exponent plane;
//   3. it loads the raw-nibble plane (16-byte loads) and combines it with the
//      exponent plane into FP8 bytes, written with coalesced 16-byte stores.
// Every read is bounded by the page size; a row that does not decode sets
// PQE_STATUS_CORRUPT_STREAM (its bytes are then unspecified).

#ifndef PQE_HD_THREADS
#define PQE_HD_THREADS 256
#endif
#ifndef PQE_HD_SPAN_WORDS
#define PQE_HD_SPAN_WORDS 4096
#endif
constexpr int HD_THREADS = PQE_HD_THREADS;
constexpr int HD_UNIT_CHUNKS = 2 * HD_THREADS;  // chunks per CTA (two per thread)
constexpr int HD_SPAN_WORDS = PQE_HD_SPAN_WORDS; // code words staged per pass
constexpr int HD_SPAN_PAD = 64;                 // zero words after them (a run of two chunks reads <= 49 words ahead)
constexpr int HD_EXP_STRIDE = 9;                // exponent-plane words per chunk: 8 + 1 (bank spread)
constexpr int HD_PAIR_STRIDE = 17;              // per pair of chunks decoded as one run: 16 + 1
static_assert(HD_THREADS * HD_PAIR_STRIDE <= HD_UNIT_CHUNKS * HD_EXP_STRIDE, "pair plane larger than the chunk plane");
constexpr int HD_LUT_WORDS = PQE_HUFF_LUT_BYTES / 4;
constexpr int HD_MAX_PAGES = 128;               // pages per launch (kernel parameter block)
constexpr int HD_RW_WORDS = HD_UNIT_CHUNKS + 4; // row offsets of a block (<= 512 rows + 1)

struct HuffBatch {
    const uint8_t *comp[HD_MAX_PAGES];
    const uint32_t *lut13[HD_MAX_PAGES];
    const uint32_t *lut2[HD_MAX_PAGES];
    uint8_t *out[HD_MAX_PAGES];
    uint64_t comp_bytes[HD_MAX_PAGES];
    int n, H, I;
    int rows13_unit, rows2_unit;  // rows per CTA
    int units13, units2;          // CTAs per matrix
};

constexpr size_t HD_SMEM = sizeof(uint32_t) * (HD_LUT_WORDS + HD_SPAN_WORDS + HD_SPAN_PAD + HD_UNIT_CHUNKS * HD_EXP_STRIDE +
                                               HD_RW_WORDS) +
                           HUF_HEADER + 16;

__device__ __forceinline__ bool in_page(uint64_t off, uint64_t len, uint64_t comp_bytes) {
    return off <= comp_bytes && len <= comp_bytes - off;
}

__device__ bool header_ok(const HuffHeader &hd, uint64_t comp_bytes, int H, int I) {
    const uint64_t n_scale = 2 * (uint64_t)I + H;
    const uint64_t r13 = 2 * (uint64_t)I, r2 = H;
    const uint64_t nc13 = H / HUF_CHUNK, nc2 = I / HUF_CHUNK;
    return hd.magic == HUF_MAGIC && hd.version == HUF_VERSION && hd.H == H && hd.I == I &&
           in_page(hd.off_scales, 4 * n_scale, comp_bytes) &&
           in_page(hd.m13.off_row_word, 4 * (r13 + 1), comp_bytes) &&
           in_page(hd.m13.off_chunk_bit, 2 * r13 * nc13, comp_bytes) &&
           in_page(hd.m13.off_nibbles, r13 * H / 2, comp_bytes) && hd.m13.n_words < (comp_bytes >> 2) &&
           in_page(hd.m13.off_words, round_up(4 * hd.m13.n_words, 16), comp_bytes) &&
           in_page(hd.m2.off_row_word, 4 * (r2 + 1), comp_bytes) &&
           in_page(hd.m2.off_chunk_bit, 2 * r2 * nc2, comp_bytes) &&
           in_page(hd.m2.off_nibbles, r2 * I / 2, comp_bytes) && hd.m2.n_words < (comp_bytes >> 2) &&
           in_page(hd.m2.off_words, round_up(4 * hd.m2.n_words, 16), comp_bytes) && (hd.off_scales % 16) == 0 &&
           (hd.m13.off_row_word % 4) == 0 && (hd.m13.off_chunk_bit % 2) == 0 && (hd.m13.off_nibbles % 16) == 0 &&
           (hd.m13.off_words % 16) == 0 && (hd.m2.off_row_word % 4) == 0 && (hd.m2.off_chunk_bit % 2) == 0 &&
           (hd.m2.off_nibbles % 16) == 0 && (hd.m2.off_words % 16) == 0;
}

// funnel shift left and byte permute, callable on the host as well (the chunk
// decoder below is checked there against the encoder)
__host__ __device__ __forceinline__ uint32_t fshl(uint32_t lo, uint32_t hi, uint32_t sh) {
#ifdef __CUDA_ARCH__
    return __funnelshift_l(lo, hi, sh);
#else
    sh &= 31u;
    return sh ? (hi << sh) | (lo >> (32u - sh)) : hi;
#endif
}

__host__ __device__ __forceinline__ uint32_t bperm(uint32_t x, uint32_t y, uint32_t sel) {
#ifdef __CUDA_ARCH__
    return __byte_perm(x, y, sel);
#else
    const uint64_t v = ((uint64_t)y << 32) | x;
    uint32_t r = 0;
    for (int i = 0; i < 4; ++i) r |= (uint32_t)((v >> (8 * ((sel >> (4 * i)) & 7u))) & 0xFFu) << (8 * i);
    return r;
#endif
}

// Eight exponent nibbles e and eight raw (sign | mantissa) nibbles r, symbol j
// in bits 4j..4j+3 of both, to eight E4M3 bytes (symbol j -> byte j).
__host__ __device__ __forceinline__ uint2 fp8_bytes8(uint32_t e, uint32_t r) {
    const uint32_t e_ev = e & 0x0F0F0F0Fu, e_od = (e >> 4) & 0x0F0F0F0Fu;
    const uint32_t r_ev = r & 0x0F0F0F0Fu, r_od = (r >> 4) & 0x0F0F0F0Fu;
    const uint32_t b_ev = ((r_ev & 0x08080808u) << 4) | (e_ev << 3) | (r_ev & 0x07070707u);
    const uint32_t b_od = ((r_od & 0x08080808u) << 4) | (e_od << 3) | (r_od & 0x07070707u);
    return make_uint2(bperm(b_ev, b_od, 0x5140), bperm(b_ev, b_od, 0x7362));
}

// Decoder state of a run of 64-symbol chunks that follow each other in one
// row's code stream. span: the row's code words, followed by at least
// HD_SPAN_PAD readable words (a run of n chunks reads at most n * 64 * 12 bits
// past its start, and one word more); pos: the next bit of span; eb: the run's exponent words (eight
// nibbles each, first symbol lowest). Every step does the same work (no
// refill or emit branch, which would diverge across the lanes of a warp): the
// 12-bit window is cut from two span words at the bit position, and an
// exponent word is stored once complete.
struct ChunkDec {
    uint32_t pos, acc_lo, acc_hi;  // next bit; pending exponent nibbles
    uint32_t na4, o;               // 4 x pending nibbles; exponent words stored
    uint32_t *eb;

    __host__ __device__ __forceinline__ void init(uint32_t p, uint32_t *e) {
        pos = p;
        acc_lo = acc_hi = na4 = o = 0;
        eb = e;
    }
    __host__ __device__ __forceinline__ uint32_t window(const uint32_t *__restrict__ lut,
                                                       const uint32_t *__restrict__ span) const {
        const uint32_t w = pos >> 5;
        return lut[fshl(span[w + 1], span[w], pos) >> 20];  // fshl shifts by pos mod 32
    }
    __host__ __device__ __forceinline__ void take(uint32_t n4, uint32_t t, uint32_t syms) {
        pos += t;
        acc_lo |= syms << na4;
        acc_hi |= fshl(syms, 0u, na4);
        na4 += n4;
        const bool full = na4 >= 32;
        if (full) eb[o] = acc_lo;
        o += full;
        acc_lo = full ? acc_hi : acc_lo;
        acc_hi = full ? 0u : acc_hi;
        na4 -= full ? 32u : 0u;
    }
    // one lookup taking all of its (at most 5) symbols: while o < words - 1.
    // An invalid window consumes no bits, so once met it is met again by every
    // later lookup: finish() alone checks for it.
    __host__ __device__ __forceinline__ void step(const uint32_t *__restrict__ lut,
                                                  const uint32_t *__restrict__ span) {
        const uint32_t ent = window(lut, span);
        take((ent >> 2) & 0x1Cu, ent & 15u, ent >> 12);
    }
    // the last 8 symbols of a run of `words` exponent words: a lookup with more
    // than needed contributes its first
    __host__ __device__ __forceinline__ void finish(const uint32_t *__restrict__ lut,
                                                    const uint32_t *__restrict__ span, uint32_t words,
                                                    uint32_t &bad) {
        while (o < words) {
            const uint32_t ent = window(lut, span);
            bad |= ent;
            const uint32_t n4 = (ent >> 2) & 0x1Cu;
            if (n4 + na4 <= 32) take(n4, ent & 15u, ent >> 12);
            else take(4u, (ent >> 7) & 15u, (ent >> 12) & 15u);
        }
    }
};

// Decodes NCH consecutive chunks of one row (8 NCH exponent words) starting
// at bit `pos` of span, the row ending at bit `end`. Chunks of a row follow
// each other in its code stream, so a run needs only its first chunk's offset,
// and a lookup that crosses from one of its chunks into the next takes all of
// its symbols. Returns false for a stream that does not decode.
template <int NCH>
__host__ __device__ __forceinline__ bool decode_chunks(const uint32_t *__restrict__ lut,
                                                       const uint32_t *__restrict__ span, uint32_t pos, uint32_t end,
                                                       uint32_t *__restrict__ eb) {
    ChunkDec a;
    a.init(pos, eb);
    uint32_t bad = 0;
    while (a.o < 8 * NCH - 1) a.step(lut, span);
    a.finish(lut, span, 8 * NCH, bad);
    return !(bad & 0x800u) && a.pos <= end;
}

// 16-byte global -> shared copies that complete asynchronously (no register
// staging): the code table is requested at block start and lands while the
// header and the row offsets are read
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// geometry of a page's decode blocks (the same for every page of a layer)
struct HuffGeo {
    int H, I;
    int rows13_unit, rows2_unit;  // rows per block
    int units13, units2;          // blocks per matrix
};

// One decode block: block u of one page (u < units13: w13 rows, else w2 rows),
// the compressed page at `comp`, its code tables, the FP8 page out. Every
// thread of the CTA calls it for the same block.
__device__ void decode_block(const HuffGeo &b, const uint8_t *comp, uint64_t cbytes, const uint32_t *lut13g,
                             const uint32_t *lut2g, uint8_t *page_out, int u, int32_t *__restrict__ status) {
    extern __shared__ __align__(16) uint8_t hd_smem[];
    uint32_t *lut = reinterpret_cast<uint32_t *>(hd_smem);
    uint32_t *span = lut + HD_LUT_WORDS;
    uint32_t *expb = span + HD_SPAN_WORDS + HD_SPAN_PAD;
    uint32_t *rw = expb + HD_UNIT_CHUNKS * HD_EXP_STRIDE;
    HuffHeader *hdr = reinterpret_cast<HuffHeader *>(rw + HD_RW_WORDS);
    int *flag = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(hdr) + HUF_HEADER);

    const int tid = threadIdx.x;
    const int H = b.H, I = b.I;
    const bool first = u < b.units13;

    // 1. code table (asynchronous), header
    const uint4 *lut_g = reinterpret_cast<const uint4 *>(first ? lut13g : lut2g);
    for (int i = tid; i < HD_LUT_WORDS / 4; i += HD_THREADS) cp_async16(reinterpret_cast<uint4 *>(lut) + i, lut_g + i);
    if (tid < (int)(HUF_HEADER / 16) && cbytes >= HUF_HEADER)
        reinterpret_cast<uint4 *>(hdr)[tid] = reinterpret_cast<const uint4 *>(comp)[tid];
    __syncthreads();
    if (tid == 0) *flag = cbytes >= HUF_HEADER && header_ok(*hdr, cbytes, H, I);
    __syncthreads();
    if (!*flag) {
        if (tid == 0 && u == 0) atomicOr(status, PQE_STATUS_CORRUPT_STREAM);
        cp_async_wait_all();  // the table's copies land before the block's shared memory is reused
        return;
    }
    const int rows = first ? 2 * I : H, cols = first ? H : I, nc = cols / HUF_CHUNK;
    const int R = first ? b.rows13_unit : b.rows2_unit;
    const int r0 = (first ? u : u - b.units13) * R;
    const int nr = min(R, rows - r0);
    const int nch = nr * nc;
    const HuffMatrixDesc d = first ? hdr->m13 : hdr->m2;
    const PageLayout L = fp8_layout(H, I);

    // row offsets, chunk offsets, raw nibbles (registers), scales
    const uint32_t *rw_g = reinterpret_cast<const uint32_t *>(comp + d.off_row_word) + r0;
    for (int i = tid; i <= nr; i += HD_THREADS) rw[i] = rw_g[i];
    // rows of an even number of chunks: thread t decodes chunks 2t and 2t + 1
    // as one run (half the lookups that straddle a chunk end, and one loop
    // whose length varies less across a warp); otherwise chunks t and t + 256
    const bool pairs = (nc & 1) == 0;
    const uint16_t *cb_g = reinterpret_cast<const uint16_t *>(comp + d.off_chunk_bit) + (size_t)r0 * nc;
    const int c0 = pairs ? 2 * tid : tid;
    const uint32_t cb0 = c0 < nch ? cb_g[c0] : 0u;
    const uint32_t cb1 = !pairs && tid + HD_THREADS < nch ? cb_g[tid + HD_THREADS] : 0u;
    // the 32-symbol halves of the chunks this thread's warp decodes (half q of
    // chunk q / 2): a warp combines only its own chunks, so no block-wide
    // barrier lies between its decode and its stores
    const int warp = tid >> 5, lane = tid & 31;
    auto half_of = [&](int i) {
        return (pairs ? 128 * warp + 32 * i : (i < 2 ? 64 * warp + 32 * i : 2 * HD_THREADS + 64 * warp + 32 * (i - 2))) +
               lane;
    };
    const uint4 *nib_g = reinterpret_cast<const uint4 *>(comp + d.off_nibbles + (size_t)r0 * cols / 2);
    if (u == 0) {
        const uint4 *sc = reinterpret_cast<const uint4 *>(comp + hdr->off_scales);
        uint4 *so = reinterpret_cast<uint4 *>(page_out + L.s13);
        for (int i = tid; i < (2 * I + H) / 4; i += HD_THREADS) so[i] = sc[i];
    }
    __syncthreads();
    // row offsets: ascending, within the stream, and no row longer than the
    // staging buffer (a row's last chunk starts below bit 65536, as chunk
    // offsets are 16-bit, so a valid row has fewer than 2100 words)
    const uint32_t cap = HD_SPAN_WORDS - 8;
    int bad = 0;
    for (int i = tid; i < nr; i += HD_THREADS) bad |= rw[i + 1] < rw[i] || rw[i + 1] - rw[i] > cap;
    if (tid == 0) bad |= rw[nr] > d.n_words;
    cp_async_wait_all();  // this thread's table copies; the barriers below publish them
    if (__syncthreads_or(bad)) {
        if (tid == 0) atomicOr(status, PQE_STATUS_CORRUPT_STREAM);
        return;
    }

    // 2. rows in groups whose code words fit the staging buffer
    bool ok = true;
    for (int ga = 0; ga < nr;) {
        int lo = ga + 1, hi = nr;  // largest gb with rw[gb] - rw[ga] <= cap
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (rw[mid] - rw[ga] <= cap) lo = mid;
            else hi = mid - 1;
        }
        const int gb = lo;
        const uint64_t byte0 = d.off_words + 4 * (uint64_t)rw[ga];
        const uint64_t a0 = byte0 & ~(uint64_t)15;
        const uint32_t dsh = (uint32_t)(byte0 - a0) / 4;
        const uint64_t a1 = round_up(d.off_words + 4 * (uint64_t)rw[gb], 16);
        const int nq = (int)((a1 - a0) / 16);
        // plain 16-byte loads: the source may be pinned host memory, which
        // asynchronous copies read far slower (compressed refills at 155
        // against 190 GB/s, measured)
        for (int i = tid; i < nq; i += HD_THREADS)
            reinterpret_cast<uint4 *>(span)[i] = *reinterpret_cast<const uint4 *>(comp + a0 + 16 * (uint64_t)i);
        if (tid < HD_SPAN_PAD) span[4 * nq + tid] = 0;
        __syncthreads();
        if (pairs) {
            const int rr = c0 / nc;
            if (c0 < nch && rr >= ga && rr < gb) {
                const uint32_t row0 = 32 * (dsh + rw[rr] - rw[ga]);  // row start, in bits of span
                const uint32_t row_bits = 32 * (rw[rr + 1] - rw[rr]);
                if (cb0 >= row_bits) ok = false;  // a chunk that starts past its row
                else ok &= decode_chunks<2>(lut, span, row0 + cb0, row0 + row_bits, expb + tid * HD_PAIR_STRIDE);
            }
        } else {
#pragma unroll 1
            for (int j = 0; j < 2; ++j) {
                const int c = tid + HD_THREADS * j;
                if (c >= nch) break;
                const int rr = c / nc;
                if (rr < ga || rr >= gb) continue;
                const uint32_t sb = j ? cb1 : cb0;
                const uint32_t row0 = 32 * (dsh + rw[rr] - rw[ga]);
                const uint32_t row_bits = 32 * (rw[rr + 1] - rw[rr]);
                if (sb >= row_bits) {
                    ok = false;
                    continue;
                }
                ok &= decode_chunks<1>(lut, span, row0 + sb, row0 + row_bits, expb + c * HD_EXP_STRIDE);
            }
        }
        if (gb < nr) __syncthreads();  // the next group's words overwrite the staging buffer
        ga = gb;
    }
    if (!ok) atomicOr(status, PQE_STATUS_CORRUPT_STREAM);

    // 3. exponent plane + raw nibbles -> FP8 bytes, 32 per thread and slice,
    // over the halves of the warp's own chunks (their exponent words are this
    // warp's stores)
    uint4 nib[4];  // loaded once the warp's decode is done; other warps' decode hides the latency
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int q = half_of(i);
        nib[i] = q < 2 * nch ? nib_g[q] : make_uint4(0, 0, 0, 0);
    }
    __syncwarp();
    uint4 *dst = reinterpret_cast<uint4 *>(page_out + (first ? L.w13 : L.w2) + (size_t)r0 * cols);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int q = half_of(i);  // 32 symbols: chunk q / 2, half q % 2
        if (q >= 2 * nch) continue;
        const uint32_t *e = expb + (pairs ? (q >> 2) * HD_PAIR_STRIDE + 4 * (q & 3)
                                          : (q >> 1) * HD_EXP_STRIDE + 4 * (q & 1));
        const uint2 a = fp8_bytes8(e[0], nib[i].x), bb = fp8_bytes8(e[1], nib[i].y);
        const uint2 c = fp8_bytes8(e[2], nib[i].z), dd = fp8_bytes8(e[3], nib[i].w);
        dst[2 * q] = make_uint4(a.x, a.y, bb.x, bb.y);
        dst[2 * q + 1] = make_uint4(c.x, c.y, dd.x, dd.y);
    }
}

__global__ void __launch_bounds__(HD_THREADS, 1024 / HD_THREADS) huff_decode_batch_kernel(const __grid_constant__ HuffBatch b,
                                                                          int32_t *__restrict__ status) {
    const int upp = b.units13 + b.units2;
    const int page = blockIdx.x / upp, u = blockIdx.x % upp;
    const HuffGeo g{b.H, b.I, b.rows13_unit, b.rows2_unit, b.units13, b.units2};
    decode_block(g, b.comp[page], b.comp_bytes[page], b.lut13[page], b.lut2[page], b.out[page], u, status);
}

// The misses of a device miss list (layout of the GPU-resident pager: [0] n,
// [2 .. 2+E) expert, [2+E .. 2+2E) destination entry), those of refill group
// `group` of `groups`, pulled from their compressed host pages and decoded
// into their slots: the grid strides over (miss, block) items. Code tables:
// expert e's at luts + e * 2 * PQE_HUFF_LUT_BYTES (w13, then w2).
__global__ void __launch_bounds__(HD_THREADS, 1024 / HD_THREADS)
    huff_decode_device_kernel(const HuffGeo g, const int32_t *__restrict__ miss, int E,
                              const uint64_t *__restrict__ comp_pages, const size_t *__restrict__ comp_bytes,
                              const uint8_t *__restrict__ luts, uint8_t *__restrict__ base, uint8_t *__restrict__ wb_base,
                              int n_slots, size_t slot_stride, int group, int groups, int32_t *__restrict__ status) {
    pdl_acquire();  // launched after the previous kernel of the step: wait for its output
    const int n_all = miss[0];
    const int m0 = overlap_group_start(group, groups, n_all), m1 = overlap_group_start(group + 1, groups, n_all);
    const int upp = g.units13 + g.units2;
    const long items = (long)(m1 - m0) * upp;
    for (long it = blockIdx.x; it < items; it += gridDim.x) {
        const int i = m0 + (int)(it / upp), u = (int)(it % upp);
        const int e = miss[2 + i], d = miss[2 + E + i];
        uint8_t *out = d < n_slots ? base + (size_t)d * slot_stride : wb_base + (size_t)(d - n_slots) * slot_stride;
        const uint32_t *l13 = reinterpret_cast<const uint32_t *>(luts + (size_t)e * 2 * PQE_HUFF_LUT_BYTES);
        decode_block(g, reinterpret_cast<const uint8_t *>(comp_pages[e]), comp_bytes[e], l13,
                     l13 + PQE_HUFF_LUT_BYTES / 4, out, u, status);
        __syncthreads();  // the block's shared memory is reused by the next item
    }
}

// the geometry of the decode blocks of an H x I page
static HuffGeo huff_geo(int H, int I) {
    const int nc13 = H / HUF_CHUNK, nc2 = I / HUF_CHUNK;
    const int R13 = HD_UNIT_CHUNKS / nc13, R2 = HD_UNIT_CHUNKS / nc2;
    return HuffGeo{H, I, R13, R2, (2 * I + R13 - 1) / R13, (H + R2 - 1) / R2};
}

static int decode_attr(int dev) {
    static std::atomic<int> attr_set[PQE_MAX_DEVICES];
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        PQE_CUDA_TRY(cudaFuncSetAttribute(huff_decode_batch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)HD_SMEM));
        PQE_CUDA_TRY(cudaFuncSetAttribute(huff_decode_device_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)HD_SMEM));
        attr_set[dev].store(1, std::memory_order_relaxed);
    }
    return PQE_OK;
}

int slot_fill_compressed_device_group(const pqe_pool *pool, const int32_t *miss, int E, const uint64_t *comp_pages,
                                      const size_t *comp_bytes, const uint8_t *luts, int group, int groups, int ctas,
                                      int32_t *status, cudaStream_t s) {
    if (!pool || !miss || !comp_pages || !comp_bytes || !luts || !status || E < 1 || E > 1024 || groups < 1 ||
        group < 0 || group >= groups || !shape_ok(pool->H, pool->I))
        return PQE_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    int rc = device_info(dev, sms);
    if (rc != PQE_OK || (rc = decode_attr(dev)) != PQE_OK) return rc;
    // the grid strides over the items; by default it fills the GPU (4 decode CTAs per SM)
    return launch_pdl(huff_decode_device_kernel, ctas > 0 ? ctas : 4 * sms, HD_THREADS, HD_SMEM, s, huff_geo(pool->H, pool->I), miss,
                      E, comp_pages, comp_bytes, luts, static_cast<uint8_t *>(pool->base),
                      static_cast<uint8_t *>(pool->wb_base), pool->n_slots, pool->slot_stride, group, groups, status);
}

// launch over n pages (n <= HD_MAX_PAGES per launch)
int launch_decode_batch(int n, const void *const *comp, const size_t *comp_bytes, const uint8_t *const *lut13,
                        const uint8_t *const *lut2, int H, int I, uint8_t *const *out, int32_t *status,
                        cudaStream_t s) {
    int dev = 0, sms = 0;
    int di = device_info(dev, sms);
    if (di != PQE_OK || (di = decode_attr(dev)) != PQE_OK) return di;
    const HuffGeo hg = huff_geo(H, I);
    const int R13 = hg.rows13_unit, R2 = hg.rows2_unit, u13 = hg.units13, u2 = hg.units2;
    for (int i0 = 0; i0 < n; i0 += HD_MAX_PAGES) {
        HuffBatch b{};
        b.n = n - i0 < HD_MAX_PAGES ? n - i0 : HD_MAX_PAGES;
        b.H = H;
        b.I = I;
        b.rows13_unit = R13;
        b.rows2_unit = R2;
        b.units13 = u13;
        b.units2 = u2;
        for (int j = 0; j < b.n; ++j) {
            b.comp[j] = static_cast<const uint8_t *>(comp[i0 + j]);
            b.comp_bytes[j] = comp_bytes[i0 + j];
            b.lut13[j] = reinterpret_cast<const uint32_t *>(lut13[i0 + j]);
            b.lut2[j] = reinterpret_cast<const uint32_t *>(lut2[i0 + j]);
            b.out[j] = out[i0 + j];
        }
        const unsigned grid = (unsigned)b.n * (unsigned)(u13 + u2);
        huff_decode_batch_kernel<<<grid, HD_THREADS, HD_SMEM, s>>>(b, status);
        PQE_LAUNCH_CHECK();
    }
    return PQE_OK;
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
    uint64_t nw13 = 0, nw2 = 0;
    if (!count_words(q13, r13, H, hd.len13, &nw13) || !count_words(q2, r2, I, hd.len2, &nw2))
        return PQE_ERR_CAPACITY;
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
    return launch_decode_batch(1, &comp_page, &comp_bytes, &lut13, &lut2, H, I, &fp8_page, status,
                               as_stream(stream));
}

int fp8_exp_huff_decode_batch(int n, const void *const *comp_pages, const size_t *comp_bytes,
                              const uint8_t *const *lut13, const uint8_t *const *lut2, int H, int I,
                              uint8_t *const *fp8_pages, int32_t *status, void *stream) {
    PQE_CHECK_ARG(n >= 0 && status && shape_ok(H, I));
    if (n == 0) return PQE_OK;
    PQE_CHECK_ARG(comp_pages && comp_bytes && lut13 && lut2 && fp8_pages);
    for (int i = 0; i < n; ++i) {
        PQE_CHECK_ARG(comp_pages[i] && lut13[i] && lut2[i] && fp8_pages[i]);
        PQE_CHECK_ARG(aligned(comp_pages[i], 16) && aligned(fp8_pages[i], 16) && aligned(lut13[i], 16) &&
                      aligned(lut2[i], 16));
    }
    return launch_decode_batch(n, comp_pages, comp_bytes, lut13, lut2, H, I, fp8_pages, status, as_stream(stream));
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

int slot_fill_compressed_batch(const pqe_pool *pool, int n, const int32_t *dest, const void *const *pinned_comp,
                               const size_t *comp_bytes, const uint8_t *const *lut13, const uint8_t *const *lut2,
                               int32_t *status, void *stream, void *done_event) {
    PQE_CHECK_ARG(pool && n >= 0 && status);
    auto s = as_stream(stream);
    if (n > 0) {
        PQE_CHECK_ARG(dest && pinned_comp && comp_bytes && lut13 && lut2);
        std::vector<uint8_t *> dst((size_t)n);
        for (int i = 0; i < n; ++i) {
            dst[i] = static_cast<uint8_t *>(pqe_pool_slot_addr(pool, dest[i]));
            PQE_CHECK_ARG(dst[i] && comp_bytes[i] >= HUF_HEADER);
        }
        const int rc = fp8_exp_huff_decode_batch(n, pinned_comp, comp_bytes, lut13, lut2, pool->H, pool->I,
                                                 dst.data(), status, stream);
        if (rc != PQE_OK) return rc;
    }
    if (done_event) PQE_CUDA_TRY(cudaEventRecord(reinterpret_cast<cudaEvent_t>(done_event), s));
    return PQE_OK;
}

}  // extern "C"
