// zero_ckpt.cu -- sharded checkpoint save and load (host code).  Each rank's
// master, m, v and 16-bit parameters go to a file of their own with a
// checksum per 2^20-element block; a plan of any rank count and stage over the
// same tensor list reads them back, each of its ranks taking the flat
// elements it owns.  The file format is specified in zero_b200.h.
//
// [Z026] sec. 5: a restore at another degree of parallelism regroups ownership
// while keeping the parameter order and each element's moments together, and
// a rank's missing file fails the restore explicitly.  [L32] sec. 4.3: the
// checkpoint holds the sharded optimizer state.
//
// IO engine: the work is a list of jobs, each at most one staging chunk of one
// file's array, pulled by worker threads.  A worker owns two pinned staging
// buffers and a CUDA stream, so the device copy of one chunk overlaps the
// checksum and the file IO of the other.  Files are read and written with
// pread/pwrite at fixed offsets, so several workers share one file.
#include <cuda_runtime.h>
#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <cerrno>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "zero_b200.h"
#include "zero_plan_access.h"
#include "zero_trace.h"

#if !defined(__BYTE_ORDER__) || __BYTE_ORDER__ != __ORDER_LITTLE_ENDIAN__
#error "checkpoint files are little-endian and are written by copying host integers"
#endif

namespace {

using zero::PlanLayout;
using zero::PlanScalars;

constexpr uint64_t BLOCK_ELEMS = 1ull << 20;      // checksum block
constexpr uint64_t CHUNK_ELEMS = 8 * BLOCK_ELEMS;  // staging chunk: whole blocks
constexpr uint64_t HEADER_BYTES = 4096;
constexpr uint64_t FILE_ALIGN = 4096;
constexpr uint32_t VERSION = 1;
constexpr int NARRAYS = 4;                        // master, m, v, params
constexpr int MAX_WORKERS = 32;
constexpr uint64_t GOLDEN = 0x9E3779B97F4A7C15ull;

const char SHARD_MAGIC[8] = {'Z', 'E', 'R', 'O', 'S', 'H', 'D', '1'};
const char MANIFEST_MAGIC[8] = {'Z', 'E', 'R', 'O', 'M', 'A', 'N', '1'};

inline uint64_t esize(int array) { return array == 3 ? 2 : 4; }
inline uint64_t round_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }
inline uint64_t ceil_div(uint64_t x, uint64_t a) { return (x + a - 1) / a; }

inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Position-keyed sum of mixed 8-byte words (see zero_b200.h); four
// independent partial sums keep the multiplier busy.
uint64_t zck64(const void* data, uint64_t bytes, uint64_t w0)
{
    const unsigned char* p = static_cast<const unsigned char*>(data);
    const uint64_t words = bytes / 8;
    uint64_t h0 = 0, h1 = 0, h2 = 0, h3 = 0;
    uint64_t i = 0;
    for (; i + 4 <= words; i += 4) {
        uint64_t x[4];
        std::memcpy(x, p + 8 * i, 32);
        const uint64_t k = (w0 + i + 1) * GOLDEN;
        h0 += mix64(x[0] + k);
        h1 += mix64(x[1] + k + GOLDEN);
        h2 += mix64(x[2] + k + 2 * GOLDEN);
        h3 += mix64(x[3] + k + 3 * GOLDEN);
    }
    for (unsigned j = 0; j < (unsigned)(words & 3); j++, i++) {   // the last 0-3 words
        uint64_t x;
        std::memcpy(&x, p + 8 * i, 8);
        h0 += mix64(x + (w0 + i + 1) * GOLDEN);
    }
    if (bytes % 8) {
        uint64_t x = 0;
        std::memcpy(&x, p + 8 * words, bytes % 8);
        h0 += mix64(x + (w0 + words + 1) * GOLDEN);
    }
    return h0 + h1 + h2 + h3;
}

struct Scalars32 {
    float loss_scale;
    int32_t good_steps;
    int64_t t;
    double beta1_pow;
    double beta2_pow;
};
static_assert(sizeof(Scalars32) == 32, "scalar record is 32 bytes");

struct ManifestRec {
    char magic[8];
    uint32_t version;
    uint32_t size;
    uint64_t psi;
    int32_t nd, stage, dtype, zero;
    uint64_t model_hash;
    Scalars32 sc;
    uint64_t meta_hash;
};
static_assert(offsetof(ManifestRec, psi) == 16 && offsetof(ManifestRec, model_hash) == 40 &&
                  offsetof(ManifestRec, sc) == 48 && offsetof(ManifestRec, meta_hash) == 80 &&
                  sizeof(ManifestRec) == 88,
              "manifest layout");

struct ShardHeader {
    char magic[8];
    uint32_t version;
    uint32_t header_bytes;
    uint64_t psi;
    int32_t nd, stage, dtype, rank;
    uint64_t model_hash;
    Scalars32 sc;
    uint64_t nseg, n, block_elems, nblocks, table_offset;
    uint64_t array_offset[NARRAYS];
    uint64_t file_bytes;
    uint64_t meta_hash;
};
static_assert(offsetof(ShardHeader, psi) == 16 && offsetof(ShardHeader, rank) == 36 &&
                  offsetof(ShardHeader, model_hash) == 40 && offsetof(ShardHeader, sc) == 48 &&
                  offsetof(ShardHeader, nseg) == 80 && offsetof(ShardHeader, array_offset) == 120 &&
                  offsetof(ShardHeader, file_bytes) == 152 &&
                  offsetof(ShardHeader, meta_hash) == 160 && sizeof(ShardHeader) == 168,
              "shard header layout");

// A run of flat elements [gstart, gstart + count) held at element dev_off of
// the device buffers a call passes (stages 0-2: the flat buffers; stage 3:
// the resident shard).
struct Seg {
    uint64_t gstart, count, dev_off;
};

// The elements rank r of a layout owns, in shard order.
std::vector<Seg> rank_segments(const PlanLayout& L, int r)
{
    std::vector<Seg> out;
    if (L.stage <= 2) {
        const uint64_t base = (uint64_t)r * L.shard;
        if (base < L.psi) out.push_back({base, std::min(L.shard, L.psi - base), base});
        return out;
    }
    uint64_t ustart = 0;
    for (size_t u = 0; u < L.unit_len.size(); u++) {
        const uint64_t lo = (uint64_t)r * L.unit_slice[u];
        if (lo < L.unit_len[u])
            out.push_back({ustart + lo, std::min(L.unit_slice[u], L.unit_len[u] - lo),
                           L.unit_off[u]});
        ustart += L.unit_len[u];
    }
    return out;
}

// Padding positions of rank r's shard: [first, first + count) element ranges.
std::vector<std::pair<uint64_t, uint64_t>> rank_padding(const PlanLayout& L, int r)
{
    std::vector<std::pair<uint64_t, uint64_t>> out;
    if (L.stage <= 2) {
        const uint64_t base = (uint64_t)r * L.shard;
        const uint64_t valid = base < L.psi ? std::min(L.shard, L.psi - base) : 0;
        if (valid < L.shard) out.push_back({base + valid, L.shard - valid});
        return out;
    }
    for (size_t u = 0; u < L.unit_len.size(); u++) {
        const uint64_t lo = (uint64_t)r * L.unit_slice[u];
        const uint64_t valid = lo < L.unit_len[u] ? std::min(L.unit_slice[u], L.unit_len[u] - lo) : 0;
        if (valid < L.unit_slice[u])
            out.push_back({L.unit_off[u] + valid, L.unit_slice[u] - valid});
    }
    return out;
}

std::string shard_path(const char* dir, int rank, int nd)
{
    char name[64];
    std::snprintf(name, sizeof(name), "/shard_%05d_of_%05d.zck", rank, nd);
    return std::string(dir) + name;
}

std::string manifest_path(const char* dir) { return std::string(dir) + "/manifest.zck"; }

bool write_all(int fd, const void* data, uint64_t bytes, uint64_t off)
{
    const char* p = static_cast<const char*>(data);
    while (bytes > 0) {
        const ssize_t w = pwrite(fd, p, (size_t)std::min<uint64_t>(bytes, 1ull << 30), (off_t)off);
        if (w < 0 && errno == EINTR) continue;
        if (w <= 0) return false;
        p += w;
        off += (uint64_t)w;
        bytes -= (uint64_t)w;
    }
    return true;
}

bool read_all(int fd, void* data, uint64_t bytes, uint64_t off)
{
    char* p = static_cast<char*>(data);
    while (bytes > 0) {
        const ssize_t r = pread(fd, p, (size_t)std::min<uint64_t>(bytes, 1ull << 30), (off_t)off);
        if (r < 0 && errno == EINTR) continue;
        if (r <= 0) return false;
        p += r;
        off += (uint64_t)r;
        bytes -= (uint64_t)r;
    }
    return true;
}

// First error wins; workers stop at their next job.
struct ErrorSlot {
    std::atomic<int> code{0};
    void set(zero_status_t s)
    {
        int expected = 0;
        code.compare_exchange_strong(expected, (int)s);
    }
    bool failed() const { return code.load(std::memory_order_relaxed) != 0; }
    zero_status_t get() const { return (zero_status_t)code.load(); }
};

struct Worker {
    cudaStream_t stream = nullptr;
    cudaEvent_t ev[2] = {nullptr, nullptr};
    void* buf[2] = {nullptr, nullptr};
};

// Streams and events for `count` workers on `device`, staging from the plan.
struct WorkerSet {
    std::vector<Worker> w;
    ~WorkerSet()
    {
        for (Worker& x : w) {
            for (cudaEvent_t e : x.ev)
                if (e) cudaEventDestroy(e);
            if (x.stream) cudaStreamDestroy(x.stream);
        }
    }
    zero_status_t init(zero_plan_t plan, int count)
    {
        void* const* staging = zero::plan_staging(plan, 2 * count, CHUNK_ELEMS * 4);
        if (!staging) return ZERO_ENOMEM;
        w.resize((size_t)count);
        for (int i = 0; i < count; i++) {
            Worker& x = w[(size_t)i];
            if (cudaStreamCreateWithFlags(&x.stream, cudaStreamNonBlocking) != cudaSuccess ||
                cudaEventCreateWithFlags(&x.ev[0], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&x.ev[1], cudaEventDisableTiming) != cudaSuccess)
                return ZERO_ECUDA;
            x.buf[0] = staging[2 * i];
            x.buf[1] = staging[2 * i + 1];
        }
        return ZERO_OK;
    }
};

int worker_count(size_t jobs)
{
    unsigned hw = std::thread::hardware_concurrency();
    if (hw == 0) hw = 4;
    return (int)std::max<size_t>(1, std::min<size_t>({jobs, (size_t)hw, (size_t)MAX_WORKERS}));
}

// Run fn(worker index) on up to `count` threads (the calling thread is worker
// 0).  Jobs are pulled from a shared counter, so if a thread cannot be started
// the others still run every job.
template <class F>
void run_workers(int count, int device, F fn)
{
    std::vector<std::thread> threads;
    for (int i = 1; i < count; i++) {
        try {
            threads.emplace_back([=]() {
                cudaSetDevice(device);
                fn(i);
            });
        } catch (...) {
            break;
        }
    }
    fn(0);
    for (auto& t : threads) t.join();
}

void scalars_to_rec(const PlanScalars& s, Scalars32* r)
{
    r->loss_scale = s.loss_scale;
    r->good_steps = s.good_steps;
    r->t = s.t;
    r->beta1_pow = s.beta1_pow;
    r->beta2_pow = s.beta2_pow;
}

// ---------------------------------------------------------------- save
struct ShardOut {
    std::string path, tmp;
    int fd = -1;
    ShardHeader h{};
    std::vector<Seg> segs;
    std::vector<uint64_t> cum;         // file element where segment i starts (nseg + 1)
    std::vector<uint64_t> hashes;      // NARRAYS x nblocks
};

struct SaveJob {
    int file, array;
    uint64_t felem, count;
};

zero_status_t write_table_and_header(ShardOut& F)
{
    std::vector<uint64_t> table;
    table.reserve(2 * F.segs.size() + F.hashes.size());
    for (const Seg& s : F.segs) {
        table.push_back(s.gstart);
        table.push_back(s.count);
    }
    table.insert(table.end(), F.hashes.begin(), F.hashes.end());
    F.h.meta_hash = zck64(&F.h, offsetof(ShardHeader, meta_hash), 0) +
                    zck64(table.data(), table.size() * 8, 0);
    std::vector<unsigned char> head(HEADER_BYTES, 0);
    std::memcpy(head.data(), &F.h, sizeof(ShardHeader));
    if (!write_all(F.fd, head.data(), HEADER_BYTES, 0)) return ZERO_EIO;
    if (!table.empty() && !write_all(F.fd, table.data(), table.size() * 8, F.h.table_offset))
        return ZERO_EIO;
    return ZERO_OK;
}

zero_status_t fsync_dir(const char* dir)
{
    const int fd = open(dir, O_RDONLY | O_DIRECTORY);
    if (fd < 0) return ZERO_EIO;
    const int r = fsync(fd);
    close(fd);
    return r == 0 ? ZERO_OK : ZERO_EIO;
}

zero_status_t save_impl(zero_plan_t plan, const char* dir, int rank, const void* const src[NARRAYS],
                        int flags, std::vector<ShardOut>& files)
{
    PlanLayout L;
    zero::plan_layout(plan, &L);
    PlanScalars sc;
    zero_status_t st = zero::plan_scalars_get(plan, &sc);
    if (st != ZERO_OK) return st;
    Scalars32 rec{};
    scalars_to_rec(sc, &rec);

    if (mkdir(dir, 0755) != 0 && errno != EEXIST) return ZERO_EIO;

    const int r0 = rank < 0 ? 0 : rank, r1 = rank < 0 ? L.nd : rank + 1;
    for (int r = r0; r < r1; r++) {
        ShardOut F;
        F.path = shard_path(dir, r, L.nd);
        F.tmp = F.path + ".tmp";
        F.segs = rank_segments(L, r);
        F.cum.push_back(0);
        for (const Seg& s : F.segs) F.cum.push_back(F.cum.back() + s.count);
        const uint64_t n = F.cum.back();
        ShardHeader& h = F.h;
        std::memcpy(h.magic, SHARD_MAGIC, 8);
        h.version = VERSION;
        h.header_bytes = (uint32_t)HEADER_BYTES;
        h.psi = L.psi;
        h.nd = L.nd;
        h.stage = L.stage;
        h.dtype = L.dtype;
        h.rank = r;
        h.model_hash = L.model_hash;
        h.sc = rec;
        h.nseg = F.segs.size();
        h.n = n;
        h.block_elems = BLOCK_ELEMS;
        h.nblocks = ceil_div(n, BLOCK_ELEMS);
        h.table_offset = HEADER_BYTES;
        uint64_t off = round_up(HEADER_BYTES + 16 * h.nseg + 8 * NARRAYS * h.nblocks, FILE_ALIGN);
        for (int a = 0; a < NARRAYS; a++) {
            h.array_offset[a] = off;
            off += round_up(n * esize(a), FILE_ALIGN);
        }
        h.file_bytes = off;
        F.hashes.assign((size_t)(NARRAYS * h.nblocks), 0);
        files.push_back(std::move(F));
    }
    for (ShardOut& F : files) {
        F.fd = open(F.tmp.c_str(), O_WRONLY | O_CREAT | O_TRUNC, 0644);
        if (F.fd < 0) return ZERO_EIO;
        if (ftruncate(F.fd, (off_t)F.h.file_bytes) != 0) return ZERO_EIO;
    }

    // chunk-major order: consecutive jobs, which run at the same time, go to
    // different files (buffered writes to one file serialise on its inode lock)
    std::vector<SaveJob> jobs;
    uint64_t nmax = 0;
    for (const ShardOut& F : files) nmax = std::max(nmax, F.h.n);
    for (uint64_t e = 0; e < nmax; e += CHUNK_ELEMS)
        for (int a = 0; a < NARRAYS; a++)
            for (int f = 0; f < (int)files.size(); f++)
                if (e < files[(size_t)f].h.n)
                    jobs.push_back({f, a, e, std::min(CHUNK_ELEMS, files[(size_t)f].h.n - e)});

    if (!jobs.empty()) {
        const int nw = worker_count(jobs.size());
        WorkerSet ws;
        st = ws.init(plan, nw);
        if (st != ZERO_OK) return st;
        std::atomic<size_t> next{0};
        ErrorSlot err;
        run_workers(nw, L.device, [&](int wi) {
            Worker& W = ws.w[(size_t)wi];
            auto issue = [&](const SaveJob& j, int b) -> bool {
                const ShardOut& F = files[(size_t)j.file];
                const uint64_t es = esize(j.array);
                const char* base = static_cast<const char*>(src[j.array]);
                size_t i = (size_t)(std::upper_bound(F.cum.begin(), F.cum.end(), j.felem) -
                                    F.cum.begin()) - 1;
                uint64_t k = j.felem, out = 0;
                const uint64_t end = j.felem + j.count;
                while (k < end) {
                    const uint64_t take = std::min(end, F.cum[i + 1]) - k;
                    const char* from = base + (F.segs[i].dev_off + (k - F.cum[i])) * es;
                    if (cudaMemcpyAsync(static_cast<char*>(W.buf[b]) + out * es, from, take * es,
                                        cudaMemcpyDeviceToHost, W.stream) != cudaSuccess)
                        return false;
                    out += take;
                    k += take;
                    i++;
                }
                return cudaEventRecord(W.ev[b], W.stream) == cudaSuccess;
            };
            size_t cur = next.fetch_add(1);
            int b = 0;
            if (cur < jobs.size() && !issue(jobs[cur], b)) {
                err.set(ZERO_ECUDA);
                return;
            }
            while (cur < jobs.size() && !err.failed()) {
                const size_t nxt = next.fetch_add(1);
                if (nxt < jobs.size() && !issue(jobs[nxt], 1 - b)) {
                    err.set(ZERO_ECUDA);
                    break;
                }
                if (cudaEventSynchronize(W.ev[b]) != cudaSuccess) {
                    err.set(ZERO_ECUDA);
                    break;
                }
                const SaveJob& j = jobs[cur];
                ShardOut& F = files[(size_t)j.file];
                const uint64_t es = esize(j.array);
                const unsigned char* data = static_cast<const unsigned char*>(W.buf[b]);
                for (uint64_t blk = j.felem / BLOCK_ELEMS; blk * BLOCK_ELEMS < j.felem + j.count;
                     blk++) {
                    const uint64_t e0 = blk * BLOCK_ELEMS;
                    const uint64_t cnt = std::min(BLOCK_ELEMS, F.h.n - e0);
                    F.hashes[(size_t)(j.array * F.h.nblocks + blk)] =
                        zck64(data + (e0 - j.felem) * es, cnt * es, e0 * es / 8);
                }
                if (!write_all(F.fd, data, j.count * es, F.h.array_offset[j.array] + j.felem * es)) {
                    err.set(ZERO_EIO);
                    break;
                }
                cur = nxt;
                b = 1 - b;
            }
            cudaStreamSynchronize(W.stream);
        });
        if (err.failed()) return err.get();
    }

    for (ShardOut& F : files) {
        st = write_table_and_header(F);
        if (st != ZERO_OK) return st;
        if ((flags & ZERO_CKPT_FSYNC) && fsync(F.fd) != 0) return ZERO_EIO;
#ifdef POSIX_FADV_DONTNEED
        if ((flags & ZERO_CKPT_FSYNC) && (flags & ZERO_CKPT_DROP_CACHE))
            posix_fadvise(F.fd, 0, 0, POSIX_FADV_DONTNEED);
#endif
        if (close(F.fd) != 0) {
            F.fd = -1;
            return ZERO_EIO;
        }
        F.fd = -1;
        if (rename(F.tmp.c_str(), F.path.c_str()) != 0) return ZERO_EIO;
        F.tmp.clear();
    }

    if (rank <= 0) {
        ManifestRec m{};
        std::memcpy(m.magic, MANIFEST_MAGIC, 8);
        m.version = VERSION;
        m.size = (uint32_t)sizeof(ManifestRec);
        m.psi = L.psi;
        m.nd = L.nd;
        m.stage = L.stage;
        m.dtype = L.dtype;
        m.model_hash = L.model_hash;
        m.sc = rec;
        m.meta_hash = zck64(&m, offsetof(ManifestRec, meta_hash), 0);
        const std::string path = manifest_path(dir), tmp = path + ".tmp";
        const int fd = open(tmp.c_str(), O_WRONLY | O_CREAT | O_TRUNC, 0644);
        if (fd < 0) return ZERO_EIO;
        bool ok = write_all(fd, &m, sizeof(m), 0);
        if (ok && (flags & ZERO_CKPT_FSYNC)) ok = fsync(fd) == 0;
        ok = (close(fd) == 0) && ok;
        if (!ok || rename(tmp.c_str(), path.c_str()) != 0) {
            unlink(tmp.c_str());
            return ZERO_EIO;
        }
    }
    if (flags & ZERO_CKPT_FSYNC) return fsync_dir(dir);
    return ZERO_OK;
}

// ---------------------------------------------------------------- load
struct ShardIn {
    int fd = -1;
    ShardHeader h{};
    std::vector<uint64_t> seg_start, seg_count;
    std::vector<uint64_t> hashes;
};

struct Piece {                 // a run of flat elements held by one old file
    uint64_t gstart, count;
    int file;
    uint64_t felem;            // element of that file's arrays
};

struct LoadJob {
    int file, array;
    uint64_t felem, count, dst;
};

zero_status_t open_error() { return errno == ENOENT ? ZERO_ENOENT : ZERO_EIO; }

zero_status_t read_manifest(const char* dir, ManifestRec* m)
{
    const int fd = open(manifest_path(dir).c_str(), O_RDONLY);
    if (fd < 0) return open_error();
    const bool ok = read_all(fd, m, sizeof(*m), 0);
    close(fd);
    if (!ok || std::memcmp(m->magic, MANIFEST_MAGIC, 8) != 0 || m->version != VERSION ||
        m->size != sizeof(ManifestRec) || m->nd < 1 || m->nd > 1024 || m->stage < 0 ||
        m->stage > 3 || m->meta_hash != zck64(m, offsetof(ManifestRec, meta_hash), 0))
        return ZERO_ECORRUPT;
    return ZERO_OK;
}

zero_status_t open_shard(const char* dir, const ManifestRec& m, int r, ShardIn* S)
{
    S->fd = open(shard_path(dir, r, m.nd).c_str(), O_RDONLY);
    if (S->fd < 0) return open_error();
    ShardHeader& h = S->h;
    if (!read_all(S->fd, &h, sizeof(h), 0)) return ZERO_ECORRUPT;
    if (std::memcmp(h.magic, SHARD_MAGIC, 8) != 0 || h.version != VERSION ||
        h.header_bytes != HEADER_BYTES || h.psi != m.psi || h.nd != m.nd ||
        h.stage != m.stage || h.dtype != m.dtype || h.rank != r ||
        h.model_hash != m.model_hash || std::memcmp(&h.sc, &m.sc, sizeof(Scalars32)) != 0 ||
        h.block_elems != BLOCK_ELEMS || h.n > m.psi || h.nseg > h.n || h.nseg > (1ull << 24) ||
        h.nblocks != ceil_div(h.n, BLOCK_ELEMS) || h.table_offset != HEADER_BYTES)
        return ZERO_ECORRUPT;
    uint64_t off = round_up(HEADER_BYTES + 16 * h.nseg + 8 * NARRAYS * h.nblocks, FILE_ALIGN);
    for (int a = 0; a < NARRAYS; a++) {
        if (h.array_offset[a] != off) return ZERO_ECORRUPT;
        off += round_up(h.n * esize(a), FILE_ALIGN);
    }
    struct stat stt;
    if (h.file_bytes != off || fstat(S->fd, &stt) != 0 || (uint64_t)stt.st_size < h.file_bytes)
        return ZERO_ECORRUPT;
    std::vector<uint64_t> table((size_t)(2 * h.nseg + NARRAYS * h.nblocks));
    if (!table.empty() && !read_all(S->fd, table.data(), table.size() * 8, h.table_offset))
        return ZERO_ECORRUPT;
    if (h.meta_hash != zck64(&h, offsetof(ShardHeader, meta_hash), 0) +
                           zck64(table.data(), table.size() * 8, 0))
        return ZERO_ECORRUPT;
    uint64_t total = 0;
    for (uint64_t i = 0; i < h.nseg; i++) {
        S->seg_start.push_back(table[(size_t)(2 * i)]);
        S->seg_count.push_back(table[(size_t)(2 * i + 1)]);
        total += table[(size_t)(2 * i + 1)];
    }
    if (total != h.n) return ZERO_ECORRUPT;
    S->hashes.assign(table.begin() + (ptrdiff_t)(2 * h.nseg), table.end());
    return ZERO_OK;
}

zero_status_t load_impl(zero_plan_t plan, const char* dir, int rank, void* const dst[NARRAYS],
                        std::vector<ShardIn>& shards)
{
    PlanLayout L;
    zero::plan_layout(plan, &L);
    PlanScalars now;
    zero_status_t st = zero::plan_scalars_get(plan, &now);     // waits for the last step
    if (st != ZERO_OK) return st;

    ManifestRec m;
    st = read_manifest(dir, &m);
    if (st != ZERO_OK) return st;
    if (m.psi != L.psi || m.model_hash != L.model_hash || m.dtype != L.dtype) return ZERO_EINVAL;

    // every rank file of the saving plan, whether or not this load needs it
    shards.resize((size_t)m.nd);
    for (int r = 0; r < m.nd; r++) {
        st = open_shard(dir, m, r, &shards[(size_t)r]);
        if (st != ZERO_OK) return st;
    }
    // their segments must cover [0, psi) exactly once
    std::vector<Piece> map;
    for (int r = 0; r < m.nd; r++) {
        const ShardIn& S = shards[(size_t)r];
        uint64_t fe = 0;
        for (size_t i = 0; i < S.seg_start.size(); i++) {
            if (S.seg_count[i] > 0) map.push_back({S.seg_start[i], S.seg_count[i], r, fe});
            fe += S.seg_count[i];
        }
    }
    std::sort(map.begin(), map.end(),
              [](const Piece& a, const Piece& b) { return a.gstart < b.gstart; });
    uint64_t covered = 0;
    for (const Piece& p : map) {
        if (p.gstart != covered || p.count > L.psi - covered) return ZERO_ECORRUPT;
        covered += p.count;
    }
    if (covered != L.psi) return ZERO_ECORRUPT;

    // jobs: each target segment cut where the old pieces and the staging chunks end
    const int r0 = rank < 0 ? 0 : rank, r1 = rank < 0 ? L.nd : rank + 1;
    std::vector<LoadJob> jobs;
    for (int r = r0; r < r1; r++)
        for (const Seg& s : rank_segments(L, r)) {
            uint64_t k = s.gstart;
            const uint64_t end = s.gstart + s.count;
            size_t i = (size_t)(std::upper_bound(map.begin(), map.end(), k,
                                                 [](uint64_t g, const Piece& p) {
                                                     return g < p.gstart;
                                                 }) -
                                map.begin()) - 1;
            while (k < end) {
                const Piece& p = map[i];
                const uint64_t take = std::min(end, p.gstart + p.count) - k;
                uint64_t fe = p.felem + (k - p.gstart), left = take;
                uint64_t d = s.dev_off + (k - s.gstart);
                while (left > 0) {
                    const uint64_t c = std::min(left, (fe / CHUNK_ELEMS + 1) * CHUNK_ELEMS - fe);
                    for (int a = 0; a < NARRAYS; a++) jobs.push_back({p.file, a, fe, c, d});
                    fe += c;
                    d += c;
                    left -= c;
                }
                k += take;
                i++;
            }
        }

    const int nw = worker_count(std::max<size_t>(jobs.size(), 1));
    WorkerSet ws;
    st = ws.init(plan, nw);
    if (st != ZERO_OK) return st;

    // from here on device memory changes
    zero::plan_set_poisoned(plan, true);
    for (int r = r0; r < r1; r++)
        for (const auto& pad : rank_padding(L, r))
            for (int a = 0; a < NARRAYS; a++) {
                const uint64_t es = esize(a);
                if (cudaMemsetAsync(static_cast<char*>(dst[a]) + pad.first * es, 0,
                                    pad.second * es, ws.w[0].stream) != cudaSuccess)
                    return ZERO_ECUDA;
            }

    std::atomic<size_t> next{0};
    ErrorSlot err;
    run_workers(nw, L.device, [&](int wi) {
        Worker& W = ws.w[(size_t)wi];
        bool pending[2] = {false, false};
        int b = 0;
        for (size_t ji = next.fetch_add(1); ji < jobs.size() && !err.failed();
             ji = next.fetch_add(1)) {
            const LoadJob& j = jobs[ji];
            const ShardIn& S = shards[(size_t)j.file];
            const uint64_t es = esize(j.array);
            if (pending[b] && cudaEventSynchronize(W.ev[b]) != cudaSuccess) {
                err.set(ZERO_ECUDA);
                break;
            }
            pending[b] = false;
            const uint64_t b0 = j.felem / BLOCK_ELEMS;
            const uint64_t e0 = b0 * BLOCK_ELEMS;
            const uint64_t e1 = std::min(ceil_div(j.felem + j.count, BLOCK_ELEMS) * BLOCK_ELEMS,
                                         S.h.n);
            unsigned char* data = static_cast<unsigned char*>(W.buf[b]);
            if (!read_all(S.fd, data, (e1 - e0) * es, S.h.array_offset[j.array] + e0 * es)) {
                err.set(ZERO_EIO);
                break;
            }
            bool ok = true;
            for (uint64_t e = e0; e < e1 && ok; e += BLOCK_ELEMS) {
                const uint64_t cnt = std::min(BLOCK_ELEMS, S.h.n - e);
                ok = zck64(data + (e - e0) * es, cnt * es, e * es / 8) ==
                     S.hashes[(size_t)(j.array * S.h.nblocks + e / BLOCK_ELEMS)];
            }
            if (!ok) {
                err.set(ZERO_ECORRUPT);
                break;
            }
            if (cudaMemcpyAsync(static_cast<char*>(dst[j.array]) + j.dst * es,
                                data + (j.felem - e0) * es, j.count * es, cudaMemcpyHostToDevice,
                                W.stream) != cudaSuccess ||
                cudaEventRecord(W.ev[b], W.stream) != cudaSuccess) {
                err.set(ZERO_ECUDA);
                break;
            }
            pending[b] = true;
            b = 1 - b;
        }
        if (cudaStreamSynchronize(W.stream) != cudaSuccess) err.set(ZERO_ECUDA);
    });
    if (err.failed()) return err.get();

    PlanScalars sc;
    sc.loss_scale = m.sc.loss_scale;
    sc.good_steps = m.sc.good_steps;
    sc.t = m.sc.t;
    sc.beta1_pow = m.sc.beta1_pow;
    sc.beta2_pow = m.sc.beta2_pow;
    st = zero::plan_scalars_set(plan, sc);
    if (st != ZERO_OK) return st;
    zero::plan_set_poisoned(plan, false);
    return ZERO_OK;
}

bool args_ok(zero_plan_t plan, const char* dir, int rank, const void* const p[NARRAYS])
{
    if (!plan || !dir || !dir[0]) return false;
    const int nd = zero::plan_nd(plan), stage = zero::plan_stage(plan);
    if (rank < -1 || rank >= nd || (rank < 0 && stage == 3)) return false;
    for (int a = 0; a < NARRAYS; a++)
        if (!p[a] || (reinterpret_cast<uintptr_t>(p[a]) & 15u) != 0) return false;
    int dev = -1;
    PlanLayout L;
    zero::plan_layout(plan, &L);
    return cudaGetDevice(&dev) == cudaSuccess && dev == L.device;
}

}  // namespace

extern "C" zero_status_t zero_checkpoint_save(zero_plan_t plan, const char* dir, int rank,
                                              const float* master, const float* m,
                                              const float* v, const void* params, int flags,
                                              void* stream)
{
    zero::TraceRange trace_("zero_checkpoint_save");
    const void* src[NARRAYS] = {master, m, v, params};
    if (!args_ok(plan, dir, rank, src)) return ZERO_EINVAL;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ZERO_ECUDA;
    std::vector<ShardOut> files;
    zero_status_t st;
    try {
        st = save_impl(plan, dir, rank, src, flags, files);
    } catch (const std::bad_alloc&) {
        st = ZERO_ENOMEM;
    } catch (...) {                             // nothing escapes the ABI
        st = ZERO_EIO;
    }
    for (ShardOut& F : files) {                     // on failure: no file under a final name
        if (F.fd >= 0) close(F.fd);
        if (!F.tmp.empty()) unlink(F.tmp.c_str());
    }
    return st;
}

extern "C" zero_status_t zero_checkpoint_load(zero_plan_t plan, const char* dir, int rank,
                                              float* master, float* m, float* v, void* params,
                                              void* stream)
{
    zero::TraceRange trace_("zero_checkpoint_load");
    void* dst[NARRAYS] = {master, m, v, params};
    const void* cdst[NARRAYS] = {master, m, v, params};
    if (!args_ok(plan, dir, rank, cdst)) return ZERO_EINVAL;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ZERO_ECUDA;
    std::vector<ShardIn> shards;
    zero_status_t st;
    try {
        st = load_impl(plan, dir, rank, dst, shards);
    } catch (const std::bad_alloc&) {
        st = ZERO_ENOMEM;
    } catch (...) {
        st = ZERO_EIO;
    }
    for (ShardIn& S : shards)
        if (S.fd >= 0) close(S.fd);
    return st;
}
