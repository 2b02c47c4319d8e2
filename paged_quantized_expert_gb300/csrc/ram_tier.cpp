// ram_tier.cpp -- the host-RAM tier of one MoE layer, fed from a paging file.
//
// Expert-pager article (rand.pepabo.com), "エキスパート重みの階層ページング":
// every MoE layer owns slots in VRAM and in host RAM, one expert per slot,
// both tiers managed LRU, slot counts set per layer; an expert missing from
// VRAM is copied from its RAM slot. "SSD階層": when host RAM cannot hold every
// expert, all experts of all layers are written at start-up into one paging
// file on SSD, and an expert missing from RAM as well is read from that file
// by a host thread into a RAM slot (O_DIRECT, so Linux). "重みの圧縮": the RAM
// and SSD tiers may hold the compressed pages.
//
// Reading taken here: the RAM tier is accessed by the VRAM tier's misses, so
// one step of the RAM tier is the LRU step (the VRAM tier's rules, with
// RAM_SLOTS slots) over the set of experts the VRAM tier missed; a step whose
// set exceeds RAM_SLOTS leaves the RAM slots as they are and reads the missing
// pages into RAM working entries, as the VRAM tier does with its working buffer.
//
// The reads run on a pool of reader threads: a step queues one job per 1 MiB
// piece of every page it must read and returns; pqe_ram_tier_wait blocks
// until all have landed. Pages sit in the file at 4096-byte offsets and are
// padded to 4096 bytes, and RAM slots are 4096-byte aligned, so each read is
// valid under O_DIRECT.
#include <fcntl.h>
#include <unistd.h>

#include <atomic>
#include <cerrno>
#include <condition_variable>
#include <cstdint>
#include <cstring>
#include <deque>
#include <mutex>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "pqe.h"

namespace {

constexpr uint64_t FILE_ALIGN = 4096;
constexpr uint64_t READ_PIECE = 1u << 20;

uint64_t up4k(uint64_t x) { return (x + FILE_ALIGN - 1) / FILE_ALIGN * FILE_ALIGN; }

struct ReadJob {
    uint64_t off, len;
    uint8_t *dst;
};

}  // namespace

struct pqe_ram_tier {
    pqe_ram_tier_config cfg{};
    int fd = -1;      // the paging file, with O_DIRECT when the file system allows it
    int fd_buf = -1;  // the same file without O_DIRECT (a direct read refused with EINVAL is retried here)
    std::atomic<int> direct{0};  // O_DIRECT in use
    std::vector<uint64_t> offsets;
    std::vector<size_t> bytes;
    uint8_t *ram = nullptr;
    pqe_lru *lru = nullptr;
    std::vector<int32_t> table, miss_e, miss_d;  // LRU step outputs
    // reader pool
    std::vector<std::thread> threads;
    std::mutex mu;
    std::condition_variable cv_job, cv_done;
    std::deque<ReadJob> jobs;
    int64_t in_flight = 0;  // queued + running
    int io_error = 0;       // errno of the first failed read since the last wait
    bool stop = false;
    // running totals: file reads (pages), bytes read, working-buffer steps
    int64_t n_reads = 0, n_bytes = 0, n_working = 0;

    void worker() {
        for (;;) {
            ReadJob j;
            {
                std::unique_lock<std::mutex> lk(mu);
                cv_job.wait(lk, [&] { return stop || !jobs.empty(); });
                if (jobs.empty()) return;  // stop requested and nothing left
                j = jobs.front();
                jobs.pop_front();
            }
            int err = 0;
            uint64_t done = 0;
            while (done < j.len) {
                const bool dio = direct.load(std::memory_order_relaxed);
                const ssize_t r = pread(dio ? fd : fd_buf, j.dst + done, j.len - done, (off_t)(j.off + done));
                if (r < 0 && errno == EINTR) continue;
                if (r < 0 && errno == EINVAL && dio) {  // the file system refuses direct reads: buffered from now on
                    direct.store(0, std::memory_order_relaxed);
                    continue;
                }
                if (r <= 0) {
                    err = r < 0 ? errno : EIO;  // an error, or the file ended early
                    break;
                }
                done += (uint64_t)r;
            }
            {
                std::lock_guard<std::mutex> lk(mu);
                if (err && !io_error) io_error = err;
                if (--in_flight == 0) cv_done.notify_all();
            }
        }
    }
};

extern "C" {

int pqe_paging_file_write(const char *path, int n, const void *const *pages, const size_t *bytes, uint64_t *offsets) {
    if (!path || n < 0 || (n > 0 && (!pages || !bytes || !offsets))) return PQE_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i)
        if (!pages[i] || bytes[i] == 0) return PQE_ERR_INVALID_ARG;
    const int fd = open(path, O_WRONLY | O_CREAT | O_TRUNC, 0644);
    if (fd < 0) return PQE_ERR_IO;
    std::vector<uint8_t> pad(FILE_ALIGN, 0);
    uint64_t off = 0;
    int rc = PQE_OK;
    for (int i = 0; i < n && rc == PQE_OK; ++i) {
        offsets[i] = off;
        const uint8_t *p = static_cast<const uint8_t *>(pages[i]);
        uint64_t done = 0;
        while (done < bytes[i]) {
            const ssize_t w = pwrite(fd, p + done, bytes[i] - done, (off_t)(off + done));
            if (w < 0 && errno == EINTR) continue;
            if (w <= 0) {
                rc = PQE_ERR_IO;
                break;
            }
            done += (uint64_t)w;
        }
        const uint64_t tail = up4k(bytes[i]) - bytes[i];  // pad each page to 4096 bytes
        if (rc == PQE_OK && tail && pwrite(fd, pad.data(), tail, (off_t)(off + bytes[i])) != (ssize_t)tail)
            rc = PQE_ERR_IO;
        off += up4k(bytes[i]);
    }
    if (close(fd) != 0 && rc == PQE_OK) rc = PQE_ERR_IO;
    return rc;
}

pqe_ram_tier *pqe_ram_tier_create(const pqe_ram_tier_config *cfg, const char *path, const uint64_t *offsets,
                                  const size_t *bytes, void *ram) {
    if (!cfg || !path || !offsets || !bytes || !ram) return nullptr;
    const pqe_ram_tier_config &c = *cfg;
    if (c.E < 1 || c.E > (1 << 20) || c.S < 0 || c.W < 0 || c.n_threads < 1 || c.n_threads > 64 ||
        c.slot_bytes == 0 || c.slot_bytes % FILE_ALIGN || reinterpret_cast<uintptr_t>(ram) % FILE_ALIGN)
        return nullptr;
    for (int e = 0; e < c.E; ++e)
        if (bytes[e] == 0 || up4k(bytes[e]) > c.slot_bytes || offsets[e] % FILE_ALIGN) return nullptr;
    pqe_ram_tier *t = new (std::nothrow) pqe_ram_tier();
    if (!t) return nullptr;
    t->cfg = c;
    t->offsets.assign(offsets, offsets + c.E);
    t->bytes.assign(bytes, bytes + c.E);
    t->ram = static_cast<uint8_t *>(ram);
    t->lru = pqe_lru_create(c.E, c.S);
    t->table.assign(c.E, -1);
    t->miss_e.assign(c.E, 0);
    t->miss_d.assign(c.E, 0);
    if (!t->lru) {
        pqe_ram_tier_destroy(t);
        return nullptr;
    }
    t->fd_buf = open(path, O_RDONLY);
#ifdef O_DIRECT
    if (c.direct_io) t->fd = open(path, O_RDONLY | O_DIRECT);
#endif
    t->direct.store(t->fd >= 0 ? 1 : 0);
    if (t->fd_buf < 0) {
        pqe_ram_tier_destroy(t);
        return nullptr;
    }
    try {
        for (int i = 0; i < c.n_threads; ++i) t->threads.emplace_back([t] { t->worker(); });
    } catch (...) {
        pqe_ram_tier_destroy(t);
        return nullptr;
    }
    return t;
}

void pqe_ram_tier_destroy(pqe_ram_tier *t) {
    if (!t) return;
    {
        std::lock_guard<std::mutex> lk(t->mu);
        t->stop = true;
    }
    t->cv_job.notify_all();
    for (auto &th : t->threads) th.join();
    if (t->fd >= 0) close(t->fd);
    if (t->fd_buf >= 0) close(t->fd_buf);
    pqe_lru_destroy(t->lru);
    delete t;
}

int pqe_ram_tier_wait(pqe_ram_tier *t) {
    if (!t) return PQE_ERR_INVALID_ARG;
    std::unique_lock<std::mutex> lk(t->mu);
    t->cv_done.wait(lk, [&] { return t->in_flight == 0; });
    const int err = t->io_error;
    t->io_error = 0;
    return err ? PQE_ERR_IO : PQE_OK;
}

int pqe_ram_tier_request(pqe_ram_tier *t, const int32_t *need, const void **ram_page, int32_t *read_queued,
                         int32_t *n_read, int32_t *working) {
    if (!t || !need || !ram_page || !read_queued || !n_read || !working) return PQE_ERR_INVALID_ARG;
    // a RAM slot may be the destination of a read still in flight: finish those first
    int rc = pqe_ram_tier_wait(t);
    if (rc) return rc;
    const int E = t->cfg.E, S = t->cfg.S;
    int32_t nm = 0, wb = 0;
    rc = page_table_update(t->lru, need, t->table.data(), t->miss_e.data(), t->miss_d.data(), &nm, &wb);
    if (rc) return rc;
    for (int i = 0; i < nm; ++i)
        if (t->miss_d[i] >= S + t->cfg.W) return PQE_ERR_CAPACITY;
    for (int e = 0; e < E; ++e) {
        ram_page[e] = t->table[e] >= 0 ? t->ram + (size_t)t->table[e] * t->cfg.slot_bytes : nullptr;
        read_queued[e] = 0;
    }
    int64_t bytes = 0;
    {
        std::lock_guard<std::mutex> lk(t->mu);
        for (int i = 0; i < nm; ++i) {
            const int e = t->miss_e[i];
            uint8_t *dst = t->ram + (size_t)t->miss_d[i] * t->cfg.slot_bytes;
            const uint64_t len = up4k(t->bytes[e]);
            for (uint64_t o = 0; o < len; o += READ_PIECE) {
                t->jobs.push_back({t->offsets[e] + o, len - o < READ_PIECE ? len - o : READ_PIECE, dst + o});
                ++t->in_flight;
            }
            read_queued[e] = 1;
            bytes += (int64_t)len;
        }
        t->n_reads += nm;
        t->n_bytes += bytes;
        t->n_working += wb;
    }
    t->cv_job.notify_all();
    *n_read = nm;
    *working = wb;
    return PQE_OK;
}

int pqe_ram_tier_state(const pqe_ram_tier *t, int32_t *slot_expert, int64_t *last_use, int64_t *step,
                       int64_t *stats) {
    if (!t) return PQE_ERR_INVALID_ARG;
    int rc = pqe_lru_state(t->lru, slot_expert, last_use, step);
    if (rc) return rc;
    if (stats) {
        stats[0] = t->n_reads;
        stats[1] = t->n_bytes;
        stats[2] = t->n_working;
        stats[3] = t->direct.load();
    }
    return PQE_OK;
}

size_t pqe_ram_tier_page_bytes(const pqe_ram_tier *t, int expert) {
    if (!t || expert < 0 || expert >= t->cfg.E) return 0;
    return t->bytes[expert];
}

}  // extern "C"
