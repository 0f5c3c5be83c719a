// Host engine of kvx: validation, chunk planning, the pinned staging ring,
// reusable descriptor buffers, the launch table, device status, the C ABI.
//
// The path of one kvx_copy_batch (PegaFlow issue #408, §Summary: one
// descriptor upload and one copy-kernel launch instead of one memcpy per
// fragment):
//   1. validate the descriptors (arrays, direction, 8-byte alignment, address
//      overflow, chunk capacity; overlap and address kinds at higher levels);
//   2. cut every descriptor into chunks of at most 16 KiB and pack the 32-byte
//      records into a pinned staging slot (the reused pinned descriptor
//      buffers of the vLLM PR #42212 report, §实现拆解 item 3 and §评论区精华:
//      an unpinned buffer makes the "asynchronous" upload synchronous);
//   3. one cudaMemcpyAsync of the table to the slot's device buffer (on a
//      side stream when the caller's stream still has work queued), or none
//      for a small host-link batch, whose table the kernel reads in place;
//   4. one launch of the persistent copy kernel with min(cta_budget, work)
//      CTAs;
//   5. record the slot's event and return: enqueue-only (PegaFlow issue #408,
//      follow-up §2).
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <cerrno>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cctype>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "kvx_internal.h"
#include "kvx_workers.h"

using kvx::Launch;

// ---------------------------------------------------------------------------
// error reporting
// ---------------------------------------------------------------------------
namespace {

thread_local std::string t_err;

int log_level();

kvx_status fail(kvx_status s, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_err = buf;
    if (log_level() >= 1)
        fprintf(stderr, "kvx: status %d: %s\n", (int)s, buf);
    return s;
}

kvx_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(KVX_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define KVX_CUDA_TRY(call)                         \
    do {                                           \
        cudaError_t e_ = (call);                   \
        if (e_ != cudaSuccess)                     \
            return cuda_fail(e_, #call);           \
    } while (0)

// ---------------------------------------------------------------------------
// environment settings (an unknown value is an error on every call, so that a
// typo cannot silently select a default: FreeToken issue #751, §What we
// changed, on its own switch)
// ---------------------------------------------------------------------------
struct TableRow {
    int dir;
    uint64_t max_mean_chunk;  // row applies when mean chunk bytes <= this
    kvx_launch cfg;
    uint64_t min_payload = 0;  // ... and the batch carries at least this many bytes
    bool unmatched_only = false;  // ... and (when set) some chunk's src and dst differ mod 16
    uint64_t max_payload = ~0ull; // ... and at most this many bytes
};

struct EnvSettings {
    int validate = 0;
    int variant = KVX_VARIANT_AUTO;
    int cta_budget = 0;
    int log = 0;
    bool nvtx = false;  // KVX_NVTX=1: NVTX ranges around each entry point and its packing
    bool pdl = true;    // KVX_PDL=0: launch the copy kernels without programmatic dependent launch
    std::vector<TableRow> table;  // KVX_TABLE rows, consulted before the built-in table
    std::string error;
};

// A launch table in a text file: one row per line, `#` starts a comment:
//   dir max_mean_chunk_bytes variant cta_budget threads unroll stages store_policy
//       [assign [min_payload_bytes [phase [max_payload_bytes]]]]
// with dir h2d|d2h|d2d, max_mean_chunk_bytes an integer or "inf", variant
// ldg|bulk|stage, assign static|dynamic|auto (absent or auto: the built-in
// choice for dir), min_payload_bytes an integer (absent: 0), phase any|unmatched
// (unmatched: only batches with a chunk whose src and dst differ mod 16; absent:
// any), max_payload_bytes an integer or "inf" (absent: inf). Rows are tried in
// file order, before the built-in rows.
std::string parse_table(const char *path, std::vector<TableRow> *rows)
{
    FILE *f = fopen(path, "r");
    if (!f)
        return std::string("KVX_TABLE=") + path + ": cannot open";
    char line[512];
    int lineno = 0;
    std::string err;
    while (err.empty() && fgets(line, sizeof line, f)) {
        ++lineno;
        if (char *h = strchr(line, '#'))
            *h = 0;
        char dir[16], maxs[32], var[16], asg[16] = "", minp[32] = "", phase[16] = "", maxp[32] = "";
        int budget, threads, unroll, stages, policy;
        const int got = sscanf(line, "%15s %31s %15s %d %d %d %d %d %15s %31s %15s %31s", dir, maxs, var, &budget,
                               &threads, &unroll, &stages, &policy, asg, minp, phase, maxp);
        if (got <= 0)
            continue;  // blank or comment
        TableRow r{};
        char *end = nullptr;
        r.dir = !strcmp(dir, "h2d") ? KVX_H2D : !strcmp(dir, "d2h") ? KVX_D2H : !strcmp(dir, "d2d") ? KVX_D2D : -1;
        if (!strcmp(maxs, "inf"))
            r.max_mean_chunk = ~0ull;
        else
            r.max_mean_chunk = strtoull(maxs, &end, 10);
        const int variant = !strcmp(var, "ldg")     ? KVX_VARIANT_LDG
                            : !strcmp(var, "bulk")  ? KVX_VARIANT_BULK
                            : !strcmp(var, "stage") ? KVX_VARIANT_STAGE
                                                    : -1;
        const int ph = (got < 11 || !strcmp(phase, "any")) ? 0 : !strcmp(phase, "unmatched") ? 1 : -1;
        r.unmatched_only = ph == 1;
        char *xend = nullptr;
        if (got >= 12 && strcmp(maxp, "inf"))
            r.max_payload = strtoull(maxp, &xend, 10);
        const int assign = (got < 9 || !strcmp(asg, "auto")) ? KVX_ASSIGN_AUTO
                           : !strcmp(asg, "static") ? KVX_ASSIGN_STATIC
                           : !strcmp(asg, "dynamic") ? KVX_ASSIGN_DYNAMIC : -1;
        char *pend = nullptr;
        if (got >= 10)
            r.min_payload = strtoull(minp, &pend, 10);
        if (got < 8 || r.dir < 0 || variant < 0 || (end && *end) || budget < 1 ||
            (threads != 128 && threads != 256 && threads != 512) || (unroll != 2 && unroll != 4 && unroll != 8) ||
            stages < 2 || stages > 12 || policy < 0 || policy > 2 || assign < 0 || (pend && *pend) ||
            (got >= 10 && !isdigit((unsigned char)minp[0])) || ph < 0 || (xend && *xend) ||
            (got >= 12 && strcmp(maxp, "inf") && !isdigit((unsigned char)maxp[0])) ||
            (variant == KVX_VARIANT_STAGE && stages != 2 && stages != 4 && stages != 8)) {
            err = std::string("KVX_TABLE=") + path + ": line " + std::to_string(lineno) +
                  " is not 'dir max_mean_chunk variant cta_budget threads unroll stages store_policy "
                  "[assign [min_payload [phase [max_payload]]]]'";
            break;
        }
        r.cfg = kvx_launch{variant, budget, threads, unroll, stages, policy, assign};
        rows->push_back(r);
    }
    fclose(f);
    return err;
}

const EnvSettings &env()
{
    static EnvSettings s = [] {
        EnvSettings e;
        if (const char *v = getenv("KVX_VALIDATE")) {
            if (!strcmp(v, "0") || !strcmp(v, "1") || !strcmp(v, "2"))
                e.validate = v[0] - '0';
            else
                e.error = std::string("KVX_VALIDATE=") + v + " is not 0, 1 or 2";
        }
        if (const char *v = getenv("KVX_VARIANT")) {
            if (!strcmp(v, "auto"))
                e.variant = KVX_VARIANT_AUTO;
            else if (!strcmp(v, "ldg"))
                e.variant = KVX_VARIANT_LDG;
            else if (!strcmp(v, "bulk"))
                e.variant = KVX_VARIANT_BULK;
            else if (!strcmp(v, "stage"))
                e.variant = KVX_VARIANT_STAGE;
            else
                e.error = std::string("KVX_VARIANT=") + v + " is not auto, ldg, bulk or stage";
        }
        if (const char *v = getenv("KVX_CTA_BUDGET")) {
            char *end = nullptr;
            errno = 0;
            long b = strtol(v, &end, 10);
            if (errno || end == v || *end || b < 0 || b > (1 << 20))
                e.error = std::string("KVX_CTA_BUDGET=") + v + " is not an integer in [0, 2^20]";
            else
                e.cta_budget = (int)b;
        }
        if (const char *v = getenv("KVX_LOG")) {
            if (strlen(v) == 1 && v[0] >= '0' && v[0] <= '2')
                e.log = v[0] - '0';
            else
                e.error = std::string("KVX_LOG=") + v + " is not 0, 1 or 2";
        }
        if (const char *v = getenv("KVX_NVTX")) {
            if (!strcmp(v, "0") || !strcmp(v, "1"))
                e.nvtx = v[0] == '1';
            else
                e.error = std::string("KVX_NVTX=") + v + " is not 0 or 1";
        }
        if (const char *v = getenv("KVX_PDL")) {
            if (!strcmp(v, "0") || !strcmp(v, "1"))
                e.pdl = v[0] == '1';
            else
                e.error = std::string("KVX_PDL=") + v + " is not 0 or 1";
        }
        if (const char *v = getenv("KVX_PACK_THREADS")) {  // read by the worker pool
            char *end = nullptr;
            errno = 0;
            long t = strtol(v, &end, 10);
            if (errno || end == v || *end || t < 0 || t > 64)
                e.error = std::string("KVX_PACK_THREADS=") + v + " is not an integer in [0, 64]";
        }
        if (const char *v = getenv("KVX_TABLE")) {
            std::string err = parse_table(v, &e.table);
            if (!err.empty())
                e.error = err;
        }
        return e;
    }();
    return s;
}

int log_level() { return env().log; }

// An NVTX range for a profiler's timeline (KVX_NVTX=1), nothing otherwise.
struct NvtxRange {
    bool on;
    explicit NvtxRange(const char *name) : on(env().nvtx)
    {
        if (on)
            nvtxRangePushA(name);
    }
    ~NvtxRange()
    {
        if (on)
            nvtxRangePop();
    }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

std::atomic<int> g_validate_level{-1};

int validate_level()
{
    int v = g_validate_level.load(std::memory_order_relaxed);
    return v >= 0 ? v : env().validate;
}

kvx_status check_env()
{
    if (!env().error.empty())
        return fail(KVX_ERR_INVALID_ARG, "%s", env().error.c_str());
    return KVX_OK;
}

// ---------------------------------------------------------------------------
// validation and chunk planning (host only)
// ---------------------------------------------------------------------------
inline uint64_t chunks_of(uint64_t size)
{
    return size / KVX_CHUNK_BYTES + (size % KVX_CHUNK_BYTES != 0);  // no overflow near 2^64
}

struct Range {
    uint64_t lo, hi;
    bool operator<(const Range &o) const { return lo < o.lo; }
};

kvx_status check_overlap(const uint64_t *src, const uint64_t *dst, const uint64_t *sizes, size_t n)
{
    std::vector<Range> d;
    try {
        d.reserve(n);
    } catch (const std::exception &) {  // bad_alloc, or length_error past max_size
        return fail(KVX_ERR_CAPACITY, "out of host memory for the overlap check of %zu descriptors", n);
    }
    for (size_t i = 0; i < n; ++i)
        if (sizes[i])
            d.push_back({dst[i], dst[i] + sizes[i]});
    std::sort(d.begin(), d.end());
    for (size_t k = 1; k < d.size(); ++k)
        if (d[k].lo < d[k - 1].hi)
            return fail(KVX_ERR_OVERLAP, "destination ranges [0x%llx, 0x%llx) and [0x%llx, 0x%llx) overlap",
                        (unsigned long long)d[k - 1].lo, (unsigned long long)d[k - 1].hi,
                        (unsigned long long)d[k].lo, (unsigned long long)d[k].hi);
    // Destination ranges are now disjoint and sorted by start, hence by end:
    // the last one starting before a source range ends is the only candidate.
    for (size_t i = 0; i < n; ++i) {
        if (!sizes[i])
            continue;
        const Range s{src[i], src[i] + sizes[i]};
        auto it = std::lower_bound(d.begin(), d.end(), Range{s.hi, 0});
        if (it != d.begin() && std::prev(it)->hi > s.lo)
            return fail(KVX_ERR_OVERLAP, "descriptor %zu: source range overlaps a destination range", i);
    }
    return KVX_OK;
}

bool kind_ok(uint64_t addr, bool want_host)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, reinterpret_cast<const void *>(addr)) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeManaged)
        return true;
    return want_host ? (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr)
                     : a.type == cudaMemoryTypeDevice;
}

kvx_status check_kinds(const uint64_t *src, const uint64_t *dst, const uint64_t *sizes, size_t n, int dir)
{
    const bool src_host = dir == KVX_H2D, dst_host = dir == KVX_D2H;
    for (size_t i = 0; i < n; ++i) {
        if (!sizes[i])
            continue;
        if (!kind_ok(src[i], src_host) || !kind_ok(src[i] + sizes[i] - 1, src_host))
            return fail(KVX_ERR_NOT_MAPPED, "descriptor %zu: source 0x%llx is not %s memory", i,
                        (unsigned long long)src[i], src_host ? "mapped pinned host" : "device");
        if (!kind_ok(dst[i], dst_host) || !kind_ok(dst[i] + sizes[i] - 1, dst_host))
            return fail(KVX_ERR_NOT_MAPPED, "descriptor %zu: destination 0x%llx is not %s memory", i,
                        (unsigned long long)dst[i], dst_host ? "mapped pinned host" : "device");
    }
    return KVX_OK;
}

// Validate; count chunks and payload bytes, find the longest chunk, count
// the bytes of descriptors whose source, destination and size are all
// multiples of 16 (the bulk copy's condition), and OR together the phases
// (src ^ dst) mod 16 of the non-empty descriptors (0: every chunk matched).
kvx_status validate(const uint64_t *src, const uint64_t *dst, const uint64_t *sizes, size_t n,
                    int dir, int level, uint64_t *n_chunks, uint64_t *payload,
                    uint32_t *max_chunk = nullptr, uint64_t *aligned16 = nullptr, uint64_t *phases = nullptr)
{
    if (dir < KVX_H2D || dir > KVX_D2D)
        return fail(KVX_ERR_INVALID_ARG, "dir %d is not KVX_H2D, KVX_D2H or KVX_D2D", dir);
    if (level < 0 || level > 2)
        return fail(KVX_ERR_INVALID_ARG, "validation level %d is not 0, 1 or 2", level);
    uint64_t chunks = 0, bytes = 0, longest = 0, aligned = 0, phase = 0;
    if (n) {
        if (!src || !dst || !sizes)
            return fail(KVX_ERR_INVALID_ARG, "null descriptor array with n = %zu", n);
        // One branch-free pass over every descriptor; the exact loop below runs
        // only when this pass saw a problem, to name the first bad descriptor.
        static_assert(KVX_CHUNK_BYTES == (1u << 14), "chunk count uses a shift");
        constexpr uint64_t kHuge = 1ull << 40;  // one such descriptor exceeds KVX_MAX_CHUNKS
        uint64_t bad = 0;
        for (size_t i = 0; i < n; ++i) {
            const uint64_t z = sizes[i], s = src[i], d = dst[i];
            const uint64_t live = z ? ~0ull : 0ull;
            bad |= live & (((s | d | z) & 7u) |
                           ((uint64_t)((s == 0) | (d == 0) | (s + z < s) | (d + z < d) | (z > kHuge)) << 3));
            chunks += (z >> 14) + ((z & (KVX_CHUNK_BYTES - 1)) != 0);
            bytes += z;
            aligned += ((s | d | z) & 15u) ? 0 : z;
            phase |= live & (s ^ d) & 15u;
            longest = z > longest ? z : longest;
        }
        if (!bad) {
            if (chunks > KVX_MAX_CHUNKS)
                return fail(KVX_ERR_CAPACITY, "batch needs more than KVX_MAX_CHUNKS (%u) chunks",
                            KVX_MAX_CHUNKS);
        } else {
            chunks = bytes = longest = aligned = phase = 0;
        }
        for (size_t i = 0; bad && i < n; ++i) {
            const uint64_t z = sizes[i];
            if (!z)
                continue;
            const uint64_t s = src[i], d = dst[i];
            if (!s || !d)
                return fail(KVX_ERR_INVALID_ARG, "descriptor %zu: null address", i);
            if ((s | d | z) & 7u)
                return fail(KVX_ERR_ALIGN,
                            "descriptor %zu: src 0x%llx, dst 0x%llx, size %llu not all multiples of 8", i,
                            (unsigned long long)s, (unsigned long long)d, (unsigned long long)z);
            if (s + z < s || d + z < d)
                return fail(KVX_ERR_INVALID_ARG, "descriptor %zu: range wraps the address space", i);
            if (z > kHuge)
                return fail(KVX_ERR_CAPACITY, "descriptor %zu: %llu bytes exceed KVX_MAX_CHUNKS chunks", i,
                            (unsigned long long)z);
            chunks += chunks_of(z);
            bytes += z;
            aligned += ((s | d | z) & 15u) ? 0 : z;
            phase |= (s ^ d) & 15u;
            if (z > longest)
                longest = z;
            if (chunks > KVX_MAX_CHUNKS)
                return fail(KVX_ERR_CAPACITY, "batch needs more than KVX_MAX_CHUNKS (%u) chunks",
                            KVX_MAX_CHUNKS);
        }
    }
    if (level >= 1 && n) {
        kvx_status st = check_overlap(src, dst, sizes, n);
        if (st != KVX_OK)
            return st;
    }
    if (level >= 2 && n) {
        kvx_status st = check_kinds(src, dst, sizes, n, dir);
        if (st != KVX_OK)
            return st;
    }
    if (n_chunks)
        *n_chunks = chunks;
    if (payload)
        *payload = bytes;
    if (max_chunk)
        *max_chunk = (uint32_t)std::min<uint64_t>(longest, KVX_CHUNK_BYTES);
    if (aligned16)
        *aligned16 = aligned;
    if (phases)
        *phases = phase;
    return KVX_OK;
}

// Pack the chunk records of descriptors [a, b) of a validated batch from out[0].
// Chunk k of a descriptor covers bytes [k * 16 KiB, min((k + 1) * 16 KiB, size)).
size_t pack_range(const uint64_t *src, const uint64_t *dst, const uint64_t *sizes, size_t a, size_t b,
                  kvx_chunk *out)
{
    size_t m = 0;
    for (size_t i = a; i < b; ++i) {
        const uint64_t z = sizes[i];
        for (uint64_t o = 0; o < z; o += KVX_CHUNK_BYTES) {
            kvx_chunk &c = out[m++];
            c.src = src[i] + o;
            c.dst = dst[i] + o;
            c.len = (uint32_t)std::min<uint64_t>(KVX_CHUNK_BYTES, z - o);
            c.desc = (uint32_t)i;
            c.reserved = 0;
        }
    }
    return m;
}

// Pack a validated batch that expands to `chunks` records. A large table is
// split over the caller and the worker pool by descriptor ranges, each written
// at its own offset: the copy cannot start before the table is packed. Waking
// sleeping pool threads costs about 20 us on Grace, so only tables of 32 Ki
// records and more (1 MiB, ~100 us for one thread) are split: a MoE call's
// 3,552 records packed in 22 us alone and 40 us split, the pool asleep after
// the previous call's wait.
void pack(const uint64_t *src, const uint64_t *dst, const uint64_t *sizes, size_t n, kvx_chunk *out,
          uint64_t chunks = 0)
{
    constexpr uint64_t kParallelMinChunks = 32768;
    constexpr int kMaxParts = 16;
    kvx::Workers &w = kvx::Workers::get();
    const int parts = std::min<int>({w.threads() + 1, kMaxParts, (int)std::min<size_t>(n, kMaxParts)});
    if (chunks >= kParallelMinChunks && parts > 1) {
        size_t lo[kMaxParts + 1];
        uint64_t off[kMaxParts + 1];
        off[0] = 0;
        for (int p = 0; p <= parts; ++p)
            lo[p] = n * (size_t)p / (size_t)parts;
        for (int p = 0; p < parts; ++p) {
            uint64_t c = 0;
            for (size_t i = lo[p]; i < lo[p + 1]; ++i)
                c += chunks_of(sizes[i]);
            off[p + 1] = off[p] + c;
        }
        if (w.run(parts, [&](int p) { pack_range(src, dst, sizes, lo[p], lo[p + 1], out + off[p]); }))
            return;
    }
    pack_range(src, dst, sizes, 0, n, out);
}

// Validation level 0 and packing in one pass, for the common batch of many
// descriptors that each fit one chunk: record i is descriptor i (a zero-size
// descriptor becomes an empty record, which the kernels skip). Needs cap >= n.
// Returns false (having written garbage) when a descriptor fails a level-0
// check or is longer than one chunk; the caller then takes the exact two-pass
// path, which also reports the first failing descriptor.
struct PackAcc {
    uint64_t bad = 0, bytes = 0, longest = 0, aligned = 0, phase = 0;
};

void pack_fast_range(const uint64_t *src, const uint64_t *dst, const uint64_t *sizes, size_t a, size_t b,
                     kvx_chunk *out, PackAcc &acc)
{
    uint64_t bad = 0, bytes = 0, longest = 0, aligned = 0, phase = 0;
    for (size_t i = a; i < b; ++i) {
        const uint64_t z = sizes[i], s = src[i], d = dst[i];
        const uint64_t live = z ? ~0ull : 0ull;
        bad |= live & (((s | d | z) & 7u) | ((uint64_t)((s == 0) | (d == 0) | (s + z < s) | (d + z < d)) << 3));
        bad |= (uint64_t)(z > KVX_CHUNK_BYTES) << 4;
        bytes += z;
        aligned += ((s | d | z) & 15u) ? 0 : z;
        phase |= live & (s ^ d) & 15u;
        longest = z > longest ? z : longest;
        out[i] = kvx_chunk{s, d, (uint32_t)z, (uint32_t)i, 0};
    }
    acc.bad = bad;
    acc.bytes = bytes;
    acc.longest = longest;
    acc.aligned = aligned;
    acc.phase = phase;
}

bool pack_fast(const uint64_t *src, const uint64_t *dst, const uint64_t *sizes, size_t n,
               kvx_chunk *out, uint64_t *n_chunks, uint64_t *payload, uint32_t *max_chunk, uint64_t *aligned16,
               uint64_t *phases)
{
    // Large batches are split over the calling thread and the worker pool.
    constexpr size_t kParallelMin = 8192, kMinPart = 4096;
    constexpr int kMaxParts = 16;
    PackAcc acc[kMaxParts];
    int parts = 1;
    if (n >= kParallelMin) {
        kvx::Workers &w = kvx::Workers::get();
        parts = std::min<int>({w.threads() + 1, kMaxParts, (int)(n / kMinPart)});
        if (parts > 1 && !w.run(parts, [&](int p) {
                pack_fast_range(src, dst, sizes, n * p / parts, n * (p + 1) / parts, out, acc[p]);
            }))
            parts = 1;
    }
    if (parts == 1)
        pack_fast_range(src, dst, sizes, 0, n, out, acc[0]);
    PackAcc t;
    for (int p = 0; p < parts; ++p) {
        t.bad |= acc[p].bad;
        t.bytes += acc[p].bytes;
        t.longest = std::max(t.longest, acc[p].longest);
        t.aligned += acc[p].aligned;
        t.phase |= acc[p].phase;
    }
    if (t.bad || n > KVX_MAX_CHUNKS)
        return false;
    *n_chunks = n;
    *payload = t.bytes;
    *max_chunk = (uint32_t)t.longest;
    *aligned16 = t.aligned;
    *phases = t.phase;
    return true;
}

// ---------------------------------------------------------------------------
// launch table
// ---------------------------------------------------------------------------
// Rows by direction and mean chunk size, from the calibration sweeps on a
// GB300 (NVLink-C2C host link). The host-link rows target bytes in flight
// rather than threads (FreeToken issue #751, §Measured impact and §Proposal:
// the optimum follows bytes in flight): one direction alone saturates the
// link from about 512 KiB in flight (8 CTAs x 512 threads x 8 x 16 B) up to
// the whole GPU, while H2D and D2H running together peak at about 2 MiB in
// flight per direction (64 CTAs x 256 threads) and lose throughput beyond it,
// as the pages saw PCIe collapse past its optimum; LDG holds the link peak in
// every size class there. D2D of small chunks fills the GPU with LDG (one
// 512-thread CTA per SM: about 120 registers a thread leave room for one); of
// chunks averaging 12 KiB or more, the bulk ring measured faster (3.28-3.36
// TB/s of payload with 608 one-warp CTAs and 96 KiB rings, against 3.24 for
// LDG), so that size class picks it.
//
// Work assignment: over the host link the LDG warps take units from a counter
// (joined KV bursts 329 against 324 GB/s by position; single-direction cells
// unchanged or up to 1.5 % faster). D2D keeps the assignment by position: its
// units take ~1 us, so one counter shared by 2,432 warps contends (4 KiB x
// 65,536 chunks: 2.1 against 3.2 TB/s).
//
// A BULK row applies only to a batch whose bytes are at least 90 % in
// descriptors with 16-byte aligned source, destination and size: the bulk
// kernel moves every other chunk with its single warp, which for D2D chunks of
// 16-28 KiB with 8-byte tails ran at 0.75 TB/s where LDG reaches 3.
//
// D2D, from the mean of 30 L2-flushed launches per shape (the event timer
// ticks in ~1 us, so medians of short launches are coarse), first calibrated
// against LDG with 1,216 CTAs of 128 threads: the bulk ring was fastest for
// batches of 256 MiB and more of full 16 KiB chunks (16 KiB x 32,768: 0.992
// of HBM with 456 CTAs and 96 KiB rings, against 0.985; 64 KiB x 8,192: 0.996
// against 0.985) and LDG for everything else (24 KiB x 21,845, chunks of 16
// and 8 KiB that waste the ring's stages: 0.974 against 0.934 for the ring;
// 16 KiB x 4,096: 0.981 against 0.894, the ring's fill and drain not
// amortised over 64 MiB). The grids below were calibrated later, each shape
// as a stream of batches and alone in the same process.
//
// D2D batches of 128 MiB and more with a chunk whose source and destination
// differ mod 16 (the LDG kernel then runs its re-pairing instance, 118
// registers a thread) take the STAGE kernel: 4 warps a CTA, 4 stages of 4 KiB
// per warp, 1,216 CTAs. Odd-tail cells (sizes 8 mod 16, either side shifted
// by 8 bytes at random): 4 KiB x 65,536 0.916 against 0.877 for LDG, 8 KiB x
// 65,536 0.936 against 0.898, 16 KiB x 32,768 0.948 against 0.921, 28 KiB x
// 18,724 0.942 against 0.920. Smaller ones stay with LDG (16 KiB x 4,096 odd:
// 0.890 LDG against 0.856), as do matched batches (phase-matched LDG: 0.97-0.99).
// More, smaller grids of warps serve STAGE better (two sweeps of stages x
// CTAs, back to back and alone): with chunks longer than one 4 KiB unit, 4
// stages and 3,648 CTAs (8 KiB to 28 KiB odd cells: 0.952-0.976 as a stream
// and alone, against 0.921-0.941 and 0.940-0.952 with 1,216); with chunks of
// one unit, so that each warp has only a few units, 2 stages and 2,432 CTAs
// (4 KiB x 65,536 odd: 0.901 / 0.923 against 0.895 / 0.917; 4 stages lose
// there as the grid grows, 0.756 at 7,296 CTAs).
//
// D2D batches of at most 24 MiB take one 512-thread CTA per SM: timed alone a
// 16 MiB batch is launch-bound with any grid (0.49 of HBM), but as a stream
// of batches (programmatic dependent launch) 152 CTAs hand over to the next
// batch faster than 1,216: 4 KiB x 4,096 back to back 0.845 of HBM, 0.83 with
// 304 x 256, 0.73-0.77 with 1,216 x 128. From 32 MiB up grids of 128-thread
// CTAs are as fast or faster (8 KiB x 4,096: 0.895-0.909 against 0.885).
//
// Above 24 MiB the grid depends on the LDG instance and the payload. The
// phase-matched one (84 registers a thread: 5 CTAs of 128 threads per SM) is
// faster with 1,824 CTAs than with 1,216 on every graded aligned cell, as a
// stream of batches (4 KiB x 65,536: 0.943 -> 0.952, 8 KiB x 65,536: 0.944 ->
// 0.972, 12 KiB x 4,096: 0.864 -> 0.944, 24 KiB x 21,845: 0.950 -> 0.962) and
// timed alone (+0 to +1.3 points); above 48 MiB 3,648 CTAs are faster still
// on every cell (+1.1 points as a stream and +1.0 alone on average; 24 KiB x
// 21,845: 0.960 / 0.976 -> 0.982 / 0.992), up to it 1,824 (12 KiB x 4,096:
// 0.944 against 0.919). From 256 MiB up more CTAs still pay: with static
// assignment a CTA's share of the work is fixed, and a grid many times what
// fits at once lets the block scheduler start a new CTA wherever one has
// finished. With 9,728 CTAs the 256-512 MiB aligned cells read 0.977-0.995 of
// HBM as a stream and 0.992-1.004 alone, above the bulk ring that held this
// class before (16 KiB x 32,768: 0.972 / 0.984 -> 0.992 / 0.998; 32 KiB x
// 16,384: 0.955 / 0.982 -> 0.988 / 0.997 with 4,864; 64 KiB x 8,192: 0.947 /
// 0.988 -> 0.991 / 0.997), so no built-in row picks the ring any more; it stays
// for the tail policy (few one-warp CTAs beside a colocated kernel) and for
// KVX_TABLE rows. Phase-mismatched D2D batches run the one-path
// instance (kvx::kPhaseShift, 79 registers: 6 CTAs per SM) rather than the
// re-pairing one (118 registers): against re-pairing with 1,216 CTAs, with
// 1,824 CTAs odd-tail cells of 28-108 MiB gained +1.0 to +4.0 points as a
// stream (8 KiB x 4,096: 0.780 -> 0.820) and +0 to +2.8 alone (same box,
// alternating builds). Its grid then follows the payload: up to 32 MiB 1,216
// CTAs (8 KiB x 4,096 odd: 0.845 against 0.822 with 1,824), above it 3,040
// (60 / 92 / 108 MiB odd: 0.864 / 0.886 / 0.904 as a stream and 0.922 /
// 0.941 / 0.955 alone, against 0.843 / 0.868 / 0.885 and 0.883 / 0.889 /
// 0.922 with 1,824; 44 MiB even as a stream, +2.8 points alone).
const TableRow kTable[] = {
    {KVX_H2D, ~0ull, {KVX_VARIANT_LDG, 64, 256, 8, 3, 0, KVX_ASSIGN_DYNAMIC}},
    {KVX_D2H, ~0ull, {KVX_VARIANT_LDG, 64, 256, 8, 3, 0, KVX_ASSIGN_DYNAMIC}},
    {KVX_D2D, 4096, {KVX_VARIANT_STAGE, 2432, 128, 8, 2, 0, KVX_ASSIGN_STATIC}, 128ull << 20, true},
    {KVX_D2D, ~0ull, {KVX_VARIANT_STAGE, 3648, 128, 8, 4, 0, KVX_ASSIGN_STATIC}, 128ull << 20, true},
    {KVX_D2D, ~0ull, {KVX_VARIANT_LDG, 152, 512, 8, 3, 0, KVX_ASSIGN_STATIC}, 0, false, 24ull << 20},
    {KVX_D2D, ~0ull, {KVX_VARIANT_LDG, 1216, 128, 8, 3, 0, KVX_ASSIGN_STATIC}, 0, true, 32ull << 20},
    {KVX_D2D, ~0ull, {KVX_VARIANT_LDG, 3040, 128, 8, 3, 0, KVX_ASSIGN_STATIC}, 0, true},
    {KVX_D2D, ~0ull, {KVX_VARIANT_LDG, 1824, 128, 8, 3, 0, KVX_ASSIGN_STATIC}, 0, false, 48ull << 20},
    {KVX_D2D, ~0ull, {KVX_VARIANT_LDG, 9728, 128, 8, 3, 0, KVX_ASSIGN_STATIC}, 256ull << 20},
    {KVX_D2D, ~0ull, {KVX_VARIANT_LDG, 3648, 128, 8, 3, 0, KVX_ASSIGN_STATIC}},
};

int default_assign(int dir) { return dir == KVX_D2D ? KVX_ASSIGN_STATIC : KVX_ASSIGN_DYNAMIC; }

// The shape of a batch that the table rows look at.
struct BatchShape {
    uint64_t mean_chunk = 0;        // payload / chunks
    uint64_t payload = ~0ull;       // bytes (unknown: as large as can be)
    bool aligned = true;            // may take a BULK row
    bool matched = false;           // every chunk's src and dst agree mod 16 (unknown: no)
};

bool row_matches(const TableRow &r, int dir, const BatchShape &b)
{
    return r.dir == dir && b.mean_chunk <= r.max_mean_chunk && b.payload >= r.min_payload &&
           b.payload <= r.max_payload &&
           (b.aligned || r.cfg.variant != KVX_VARIANT_BULK) && (!r.unmatched_only || !b.matched);
}

// The row for a batch of this direction and shape.
kvx_launch table_launch(int dir, const BatchShape &b)
{
    for (const TableRow &r : env().table) {  // KVX_TABLE rows first
        if (row_matches(r, dir, b)) {
            kvx_launch c = r.cfg;
            if (c.assign == KVX_ASSIGN_AUTO)
                c.assign = default_assign(dir);
            return c;
        }
    }
    for (const TableRow &r : kTable)
        if (row_matches(r, dir, b))
            return r.cfg;
    return kTable[0].cfg;
}

// The shape of a validated batch: whether it is aligned enough for a BULK row
// (see the table), its mean chunk and its payload.
BatchShape batch_shape(uint64_t chunks, uint64_t payload, uint64_t aligned16, uint64_t phases)
{
    BatchShape b;
    b.mean_chunk = chunks ? payload / chunks : 0;
    b.payload = payload;
    b.aligned = aligned16 / 9 >= payload / 10;  // at least ~90 % (no overflow near 2^64)
    b.matched = phases == 0;
    return b;
}

// Whether an LDG copy of this direction and payload prefetches its sources into
// L2 while it waits for the grid before it: D2D (sources in HBM) of at most
// kvx::kPrefetchMaxPayload bytes (an unknown payload is ~0: no).
bool prefetch_for(int dir, uint64_t payload)
{
    return env().pdl && dir == KVX_D2D && payload <= kvx::kPrefetchMaxPayload;
}

// Merge explicit settings over env over table and check them.
kvx_status resolve(int dir, const BatchShape &shape, const kvx_launch *want, Launch *out)
{
    kvx_launch t = table_launch(dir, shape);
    const EnvSettings &e = env();
    int variant = (want && want->variant) ? want->variant : (e.variant ? e.variant : t.variant);
    int budget = (want && want->cta_budget) ? want->cta_budget : (e.cta_budget ? e.cta_budget : t.cta_budget);
    int threads = (want && want->threads) ? want->threads : t.threads;
    int unroll = (want && want->unroll) ? want->unroll : t.unroll;
    int stages = (want && want->stages) ? want->stages : t.stages;
    int policy = (want && want->store_policy) ? want->store_policy : t.store_policy;
    int assign = (want && want->assign) ? want->assign : t.assign;
    if (want) {
        if (want->variant < 0 || want->variant > KVX_VARIANT_STAGE)
            return fail(KVX_ERR_INVALID_ARG, "variant %d is not AUTO, LDG, BULK or STAGE", want->variant);
        if (want->cta_budget < 0)
            return fail(KVX_ERR_INVALID_ARG, "cta_budget %d < 0", want->cta_budget);
        if (want->threads && want->threads != 128 && want->threads != 256 && want->threads != 512)
            return fail(KVX_ERR_INVALID_ARG, "threads %d is not 128, 256 or 512", want->threads);
        if (want->unroll && want->unroll != 2 && want->unroll != 4 && want->unroll != 8)
            return fail(KVX_ERR_INVALID_ARG, "unroll %d is not 2, 4 or 8", want->unroll);
        if (want->stages && (want->stages < 2 || want->stages > 12))
            return fail(KVX_ERR_INVALID_ARG, "stages %d is not in 2..12", want->stages);
        if (want->store_policy < 0 || want->store_policy > 2)
            return fail(KVX_ERR_INVALID_ARG, "store_policy %d is not 0, 1 or 2", want->store_policy);
        if (want->assign < 0 || want->assign > KVX_ASSIGN_DYNAMIC)
            return fail(KVX_ERR_INVALID_ARG, "assign %d is not AUTO, STATIC or DYNAMIC", want->assign);
    }
    if (variant == KVX_VARIANT_AUTO)
        variant = t.variant;
    if (variant == KVX_VARIANT_STAGE && stages != 2 && stages != 4 && stages != 8) {
        if (want && want->stages)
            return fail(KVX_ERR_INVALID_ARG, "stages %d is not 2, 4 or 8 for the STAGE variant", want->stages);
        stages = 4;  // the table row was another variant's
    }
    out->variant = variant;
    out->ctas = budget;
    out->threads = threads;
    out->unroll = unroll;
    out->stages = stages;
    out->store_policy = policy;
    out->assign = assign;
    out->matched = shape.matched;
    out->shift = dir == KVX_D2D;  // see kvx::kPhaseShift
    out->pdl = e.pdl;
    out->prefetch = prefetch_for(dir, shape.payload);
    return KVX_OK;
}

void log_batch(const char *entry, int dir, size_t n, uint64_t chunks, uint64_t bytes, const Launch &l)
{
    if (log_level() >= 2)
        fprintf(stderr, "kvx: %s dir=%d n=%zu chunks=%llu bytes=%llu variant=%d ctas=%d threads=%d unroll=%d "
                        "stages=%d assign=%d\n",
                entry, dir, n, (unsigned long long)chunks, (unsigned long long)bytes, l.variant, l.ctas,
                l.threads, l.unroll, l.stages, l.assign);
}

kvx_status is_capturing(cudaStream_t stream, bool *cap)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    KVX_CUDA_TRY(cudaStreamIsCapturing(stream, &cs));
    *cap = cs != cudaStreamCaptureStatusNone;
    return KVX_OK;
}

// ---------------------------------------------------------------------------
// pinned staging ring (per device)
// ---------------------------------------------------------------------------
constexpr int kRingSlots = 8;
constexpr int kMaxDevices = 64;

// Device error flags: kvx::kErrWords words per device in one page of host
// memory, registered with the driver as mapped pinned memory on first use (a
// static array, so no allocation), written by kernels with plain stores and
// read and cleared here by atomic exchanges once the work that may have set
// them has completed.
alignas(4096) unsigned g_err_words[kMaxDevices][16];
static_assert(kvx::kErrWords <= 16, "error flag words per device");
struct ErrMap {
    std::mutex mu;
    bool registered = false;
    unsigned *dev[kMaxDevices] = {};  // device address of each device's words
};
ErrMap g_err_map;

// The device address of `dev`'s error flags (`dev` current in this thread).
// Registers the page on the first call in the process: call it outside
// stream capture (object creation and uncapturable entry points do).
kvx_status err_flags(int dev, unsigned **out)
{
    std::lock_guard<std::mutex> g(g_err_map.mu);
    if (!g_err_map.registered) {
        KVX_CUDA_TRY(cudaHostRegister(g_err_words, sizeof(g_err_words),
                                      cudaHostRegisterMapped | cudaHostRegisterPortable));
        g_err_map.registered = true;
    }
    if (!g_err_map.dev[dev]) {
        void *p = nullptr;
        KVX_CUDA_TRY(cudaHostGetDevicePointer(&p, g_err_words[dev], 0));
        g_err_map.dev[dev] = static_cast<unsigned *>(p);
    }
    *out = g_err_map.dev[dev];
    return KVX_OK;
}

// Read and clear `dev`'s error flags as a kDevErr* bit set.
unsigned take_err(int dev)
{
    unsigned bits = 0;
    for (int i = 0; i < kvx::kErrWords; ++i)
        if (__atomic_exchange_n(&g_err_words[dev][i], 0u, __ATOMIC_ACQ_REL))
            bits |= 1u << i;
    return bits;
}

constexpr size_t kMinSlotChunks = 1 << 16;

struct Slot {
    kvx_chunk *host = nullptr;  // pinned: the table header (kept zero), then the records
    kvx_chunk *host_dev = nullptr;  // the same memory as the device addresses it
    kvx_chunk *dev = nullptr;   // the device table: header, then records
    size_t cap = 0;             // chunks (records after the header)
    cudaEvent_t done = nullptr;
    cudaEvent_t uploaded = nullptr;  // recorded after a side-stream upload of the table
    bool recorded = false;
    bool busy = false;          // held by a caller between acquire and release
    uint64_t stamp = 0;         // release order: larger = more recently packed
};

struct Ring {
    std::mutex mu;
    Slot slots[kRingSlots];
    uint64_t clock = 0;
};

Ring g_rings[kMaxDevices];

kvx_status ring_acquire(int dev, size_t chunks, Slot **out)
{
    if (dev < 0 || dev >= kMaxDevices)
        return fail(KVX_ERR_INVALID_ARG, "device %d out of range", dev);
    Ring &r = g_rings[dev];
    Slot *s = nullptr;
    {
        // Prefer the most recently packed slot whose copy has finished: its
        // pinned pages are still in the CPU caches, so packing into it avoids
        // fetching a cold slot's lines from memory. Otherwise take the least
        // recently used free slot and wait for its copy below.
        std::lock_guard<std::mutex> g(r.mu);
        Slot *warm = nullptr, *oldest = nullptr;
        for (Slot &c : r.slots) {
            if (c.busy)
                continue;
            if (!oldest || c.stamp < oldest->stamp)
                oldest = &c;
            if (c.cap < chunks || (warm && c.stamp <= warm->stamp))
                continue;
            if (c.recorded) {
                if (cudaEventQuery(c.done) != cudaSuccess) {
                    cudaGetLastError();  // cudaErrorNotReady is not sticky; clear it
                    continue;
                }
                c.recorded = false;
            }
            warm = &c;
        }
        s = warm ? warm : oldest;
        if (!s)
            return fail(KVX_ERR_CAPACITY, "all %d staging slots are held by concurrent callers", kRingSlots);
        s->busy = true;
    }
    auto release_on_error = [&](kvx_status st) {
        std::lock_guard<std::mutex> g(r.mu);
        s->busy = false;
        return st;
    };
    if (!s->done) {
        cudaError_t e = cudaEventCreateWithFlags(&s->done, cudaEventDisableTiming);
        if (e != cudaSuccess)
            return release_on_error(cuda_fail(e, "cudaEventCreateWithFlags"));
    }
    if (s->recorded) {  // wait until the copy that last used this slot has finished
        cudaError_t e = cudaEventSynchronize(s->done);
        if (e != cudaSuccess)
            return release_on_error(cuda_fail(e, "cudaEventSynchronize(staging slot)"));
        s->recorded = false;
    }
    if (s->cap < chunks) {
        size_t cap = std::max(chunks, std::max(kMinSlotChunks, 2 * s->cap));
        if (cap > KVX_MAX_CHUNKS)
            cap = std::max<size_t>(chunks, KVX_MAX_CHUNKS);
        if (s->host)
            cudaFreeHost(s->host);
        if (s->dev)
            cudaFree(s->dev);
        s->host = nullptr;
        s->host_dev = nullptr;
        s->dev = nullptr;
        s->cap = 0;
        // mapped: small tables are read in place by the kernel (table_in_place)
        cudaError_t e = cudaHostAlloc(reinterpret_cast<void **>(&s->host),
                                      (cap + kvx::kTableHeader) * sizeof(kvx_chunk),
                                      cudaHostAllocPortable | cudaHostAllocMapped);
        if (e != cudaSuccess)
            return release_on_error(cuda_fail(e, "cudaHostAlloc(staging slot)"));
        memset(s->host, 0, kvx::kTableHeader * sizeof(kvx_chunk));
        e = cudaHostGetDevicePointer(reinterpret_cast<void **>(&s->host_dev), s->host, 0);
        if (e != cudaSuccess) {
            cudaFreeHost(s->host);
            s->host = nullptr;
            return release_on_error(cuda_fail(e, "cudaHostGetDevicePointer(staging slot)"));
        }
        e = cudaMalloc(reinterpret_cast<void **>(&s->dev), (cap + kvx::kTableHeader) * sizeof(kvx_chunk));
        if (e != cudaSuccess) {
            cudaFreeHost(s->host);
            s->host = nullptr;
            s->host_dev = nullptr;
            return release_on_error(cuda_fail(e, "cudaMalloc(staging slot)"));
        }
        s->cap = cap;
    }
    *out = s;
    return KVX_OK;
}

// Side streams of each device (the chunk-table uploads of kvx_copy_batch, and
// those of kvx_copy_batch_noalloc, which wait on the GPU for their table to be
// free and must not hold up the others). Created on first use with the
// device's highest priority, never destroyed.
enum AuxKind { kAuxUpload = 0, kAuxNoalloc = 1, kAuxKinds = 2 };
struct AuxStreams {
    std::mutex mu;
    cudaStream_t s[kAuxKinds] = {};
};
AuxStreams g_aux[kMaxDevices];

cudaError_t aux_stream(int dev, AuxKind kind, cudaStream_t *out)
{
    AuxStreams &a = g_aux[dev];
    std::lock_guard<std::mutex> g(a.mu);
    if (!a.s[kind]) {
        int least = 0, greatest = 0;
        cudaError_t e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
        if (e != cudaSuccess)
            return e;
        e = cudaStreamCreateWithPriority(&a.s[kind], cudaStreamNonBlocking, greatest);
        if (e != cudaSuccess) {
            a.s[kind] = nullptr;
            return e;
        }
    }
    *out = a.s[kind];
    return cudaSuccess;
}

// Upload a packed chunk table from its pinned slot to the slot's device table,
// ordered before whatever is enqueued on `stream` next. ring_acquire returned
// the slot only after the last kernel reading its device table finished, so
// the upload depends on nothing already on `stream`. When `stream` is idle
// (`busy` false) it goes on `stream`; when work is still queued there (a
// transfer worker that submits the next burst while the previous one copies)
// it goes on the upload side stream and `stream` waits for it, so the upload
// overlaps that work instead of idling the link between two copy kernels.
// Whether `stream` still has work queued (cudaErrorNotReady, cleared); other
// errors are returned in *err.
bool stream_busy(cudaStream_t stream, cudaError_t *err)
{
    const cudaError_t q = cudaStreamQuery(stream);
    *err = cudaSuccess;
    if (q == cudaErrorNotReady) {
        cudaGetLastError();  // not sticky; clear it
        return true;
    }
    if (q != cudaSuccess)
        *err = q;
    return false;
}

cudaError_t upload_table(int dev, Slot *s, size_t bytes, cudaStream_t stream, bool busy)
{
    if (!busy)
        return cudaMemcpyAsync(s->dev, s->host, bytes, cudaMemcpyHostToDevice, stream);
    cudaStream_t side = nullptr;
    cudaError_t e = aux_stream(dev, kAuxUpload, &side);
    if (e == cudaSuccess && !s->uploaded)
        e = cudaEventCreateWithFlags(&s->uploaded, cudaEventDisableTiming);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(s->dev, s->host, bytes, cudaMemcpyHostToDevice, side);
    if (e == cudaSuccess)
        e = cudaEventRecord(s->uploaded, side);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(stream, s->uploaded, 0);
    return e;
}

// Small batches skip the table upload: the kernel reads its records from the
// pinned staging slot itself (a unified address), which takes a copy-engine
// operation and its latency off the call (1,024 x 4 KiB H2D, submit + copy +
// status read: 67 -> 72 GB/s; 256 x 4 KiB D2D: 41.7 -> 36.4 us). Only for
// launches that assign units by position (the work counter must stay in
// device memory) and for at most kInPlaceMaxChunks records: a warp then reads
// its records once, where a long launch over a busy link would wait on each
// 32-record batch. A D2D batch does it only when the caller's stream is idle:
// when it is busy, the upload overlaps that work on the side stream and the
// kernel then reads its records from HBM, a shorter round trip than the host
// link's (256 x 4 KiB: 6.5 against 7.4 us).
constexpr uint64_t kInPlaceMaxChunks = 4096;

bool table_in_place(int dir, const kvx::Launch &l, uint64_t chunks, uint32_t max_chunk, bool busy)
{
    return (dir != KVX_D2D || !busy) && chunks <= kInPlaceMaxChunks &&
           !kvx::ldg_dynamic(l, (uint32_t)chunks, max_chunk);
}

void ring_release(int dev, Slot *s, cudaStream_t stream, bool record)
{
    if (record && cudaEventRecord(s->done, stream) == cudaSuccess)
        s->recorded = true;
    std::lock_guard<std::mutex> g(g_rings[dev].mu);
    s->stamp = ++g_rings[dev].clock;
    s->busy = false;
}

// Enqueue the copy over a packed slot: upload its table (or read it in place)
// and launch, then hand the slot back with the copy's completion event.
kvx_status launch_from_slot(int dev, Slot *s, int dir, const kvx::Launch &l, uint64_t chunks,
                            uint32_t max_chunk, cudaStream_t stream)
{
    cudaError_t qe = cudaSuccess;
    const bool busy = stream_busy(stream, &qe);
    if (qe != cudaSuccess) {
        ring_release(dev, s, stream, false);
        return cuda_fail(qe, "cudaStreamQuery");
    }
    kvx_chunk *table = s->host_dev;
    if (!table_in_place(dir, l, chunks, max_chunk, busy)) {
        cudaError_t e =
            upload_table(dev, s, (size_t)(chunks + kvx::kTableHeader) * sizeof(kvx_chunk), stream, busy);
        if (e != cudaSuccess) {
            ring_release(dev, s, stream, false);
            return cuda_fail(e, "chunk table upload");
        }
        table = s->dev;
    }
    unsigned *err = nullptr;
    kvx_status est = err_flags(dev, &err);
    if (est != KVX_OK) {
        ring_release(dev, s, stream, false);
        return est;
    }
    cudaError_t e = kvx::launch_copy(l, table, (uint32_t)chunks, max_chunk, err, stream);
    ring_release(dev, s, stream, true);
    if (e != cudaSuccess)
        return cuda_fail(e, "copy kernel launch");
    return KVX_OK;
}

// Status tokens: an event recorded on the caller's stream, per device a ring
// of kStatusEvents with a generation count each.
constexpr unsigned kStatusEvents = 1024;
struct StatusEvents {
    std::mutex mu;
    cudaEvent_t events[kStatusEvents] = {};
    uint64_t gen[kStatusEvents] = {};
    unsigned next = 0;
};
StatusEvents g_status_events[kMaxDevices];

// The status a word of status bits stands for (kvx_stream_check's answer).
kvx_status bits_status(unsigned bits)
{
    if (bits & kvx::kDevErrTimeout)
        return fail(KVX_ERR_TIMEOUT, "a bounded device wait gave up (status bits 0x%x)", bits);
    if (bits)
        return fail(KVX_ERR_DEVICE_FAULT, "device status bits 0x%x:%s%s%s%s", bits,
                    (bits & kvx::kDevErrBadRecord) ? " inconsistent chunk record (longer than KVX_CHUNK_BYTES, or "
                                                     "src and dst out of phase in a phase-matched launch);" : "",
                    (bits & kvx::kDevErrCount) ? " device list count above its capacity (clamped);" : "",
                    (bits & kvx::kDevErrBadDesc) ? " device list descriptor failed validation (skipped);" : "",
                    (bits & kvx::kDevErrBounds) ? " a chunk outside the debug bounds (skipped);" : "");
    return KVX_OK;
}

// The common case of kvx_copy_batch_ex in one pass over the descriptors:
// level-0 validation fused with packing into the staging slot. Sets *done and
// returns the call's status once it has enqueued (or failed to enqueue) the
// copy; leaves *done false, with nothing enqueued, whenever anything is off
// (capture, a bad descriptor, a full slot), so that the exact path decides.
kvx_status copy_batch_fast(const uint64_t *src, const uint64_t *dst, const uint64_t *sizes, size_t n,
                           int dir, const kvx_launch *want, cudaStream_t stream, bool *done)
{
    *done = false;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
        cudaGetLastError();
        return KVX_OK;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return KVX_OK;
    }
    if (n > KVX_MAX_CHUNKS)
        return KVX_OK;
    Slot *s = nullptr;
    if (ring_acquire(dev, n, &s) != KVX_OK)
        return KVX_OK;
    uint64_t chunks = 0, payload = 0, aligned16 = 0, phases = 0;
    uint32_t max_chunk = 0;
    Launch l;
    bool packed;
    {
        NvtxRange pack_range("kvx pack");
        packed = pack_fast(src, dst, sizes, n, s->host + kvx::kTableHeader, &chunks, &payload, &max_chunk,
                           &aligned16, &phases);
    }
    if (!packed || payload == 0 ||
        resolve(dir, batch_shape(chunks, payload, aligned16, phases), want, &l) != KVX_OK) {
        ring_release(dev, s, stream, false);
        return KVX_OK;
    }
    *done = true;
    log_batch("kvx_copy_batch", dir, n, chunks, payload, l);
    return launch_from_slot(dev, s, dir, l, chunks, max_chunk, stream);
}

}  // namespace

kvx_status kvx::set_error(kvx_status status, const char *message)
{
    return fail(status, "%s", message);
}

namespace {
std::mutex g_handles_mu;
std::unordered_map<const void *, int> g_handles;  // live handle -> its kvx::HandleKind
}  // namespace

bool kvx::handle_add(const void *h, HandleKind kind)
{
    std::lock_guard<std::mutex> g(g_handles_mu);
    try {
        g_handles[h] = kind;
    } catch (const std::bad_alloc &) {
        return false;
    }
    return true;
}

bool kvx::handle_remove(const void *h, HandleKind kind)
{
    std::lock_guard<std::mutex> g(g_handles_mu);
    auto it = g_handles.find(h);
    if (it == g_handles.end() || it->second != kind)
        return false;
    g_handles.erase(it);
    return true;
}

bool kvx::handle_live(const void *h, HandleKind kind)
{
    std::lock_guard<std::mutex> g(g_handles_mu);
    auto it = g_handles.find(h);
    return it != g_handles.end() && it->second == kind;
}

// ---------------------------------------------------------------------------
// descriptor buffers
// ---------------------------------------------------------------------------
struct kvx_desc_buf {
    mutable std::mutex mu;  // uploads, copies and info calls on one buffer take turns
    int device = 0;
    size_t cap = 0;
    kvx_chunk *dev = nullptr;   // header record, then the chunk records
    kvx_chunk *host = nullptr;  // pinned staging, same layout (header kept zero)
    cudaEvent_t upload_done = nullptr;
    cudaEvent_t last_use = nullptr;
    bool upload_recorded = false;
    bool use_recorded = false;
    unsigned long long last_stream = 0;  // cudaStreamGetId of the stream of the last copy
    uint32_t n_chunks = 0;
    uint32_t max_chunk = 0;
    uint64_t payload = 0;
    int dir = KVX_H2D;
    kvx_launch selected{};
    bool matched = false;  // every uploaded chunk's src and dst agree mod 16
    unsigned *err = nullptr;  // the device's error flags
};

struct kvx_devlist {
    int device = 0;
    unsigned *err = nullptr;  // the device's error flags
    uint32_t max_n = 0;
    kvx::DevListMeta *meta = nullptr;  // 256 bytes, then the offsets
    uint64_t *offsets = nullptr;
    cudaEvent_t last_use = nullptr;
    bool use_recorded = false;
    unsigned long long last_stream = 0;  // cudaStreamGetId of the stream of the last copy
    std::mutex mu;
};

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
extern "C" {

const char *kvx_status_string(int s)
{
    switch (s) {
    case KVX_OK: return "KVX_OK";
    case KVX_ERR_INVALID_ARG: return "KVX_ERR_INVALID_ARG";
    case KVX_ERR_ALIGN: return "KVX_ERR_ALIGN";
    case KVX_ERR_OVERLAP: return "KVX_ERR_OVERLAP";
    case KVX_ERR_CAPACITY: return "KVX_ERR_CAPACITY";
    case KVX_ERR_NOT_MAPPED: return "KVX_ERR_NOT_MAPPED";
    case KVX_ERR_CUDA: return "KVX_ERR_CUDA";
    case KVX_ERR_TIMEOUT: return "KVX_ERR_TIMEOUT";
    case KVX_ERR_DEVICE_FAULT: return "KVX_ERR_DEVICE_FAULT";
    case KVX_ERR_CAPTURE: return "KVX_ERR_CAPTURE";
    default: return "KVX_ERR_UNKNOWN";
    }
}

const char *kvx_last_error(void) { return t_err.c_str(); }

int kvx_version(void) { return KVX_VERSION_MAJOR * 100 + KVX_VERSION_MINOR; }

kvx_status kvx_set_validate_level(int level)
{
    if (level < 0 || level > 2)
        return fail(KVX_ERR_INVALID_ARG, "validation level %d is not 0, 1 or 2", level);
    g_validate_level.store(level);
    return KVX_OK;
}

int kvx_get_validate_level(void) { return validate_level(); }

kvx_status kvx_validate(const uint64_t *src, const uint64_t *dst, const uint64_t *sizes, size_t n,
                        int dir, int level)
{
    return validate(src, dst, sizes, n, dir, level, nullptr, nullptr);
}

kvx_status kvx_plan_chunks(const uint64_t *src, const uint64_t *dst, const uint64_t *sizes, size_t n,
                           kvx_chunk *out, size_t max_out, size_t *n_chunks)
{
    uint64_t chunks = 0;
    kvx_status st = validate(src, dst, sizes, n, KVX_H2D, 0, &chunks, nullptr);
    if (st != KVX_OK)
        return st;
    if (n_chunks)
        *n_chunks = (size_t)chunks;
    if (!out)
        return KVX_OK;
    if (chunks > max_out)
        return fail(KVX_ERR_CAPACITY, "batch needs %llu chunks, output holds %zu",
                    (unsigned long long)chunks, max_out);
    pack(src, dst, sizes, n, out, chunks);
    return KVX_OK;
}

kvx_status kvx_default_launch(int dir, uint64_t mean_chunk_bytes, kvx_launch *out)
{
    if (dir < KVX_H2D || dir > KVX_D2D)
        return fail(KVX_ERR_INVALID_ARG, "dir %d is not KVX_H2D, KVX_D2H or KVX_D2D", dir);
    if (!out)
        return fail(KVX_ERR_INVALID_ARG, "null output");
    BatchShape b;
    b.mean_chunk = mean_chunk_bytes;
    b.matched = true;  // 16-byte aligned descriptors
    *out = table_launch(dir, b);
    return KVX_OK;
}

kvx_status kvx_select_launch(const uint64_t *src, const uint64_t *dst, const uint64_t *sizes, size_t n,
                             int dir, const kvx_launch *want, kvx_launch *out)
{
    if (!out)
        return fail(KVX_ERR_INVALID_ARG, "null output");
    kvx_status st = check_env();
    if (st != KVX_OK)
        return st;
    uint64_t chunks = 0, payload = 0, aligned16 = 0, phases = 0;
    uint32_t max_chunk = 0;
    st = validate(src, dst, sizes, n, dir, 0, &chunks, &payload, &max_chunk, &aligned16, &phases);
    if (st != KVX_OK)
        return st;
    Launch l;
    st = resolve(dir, batch_shape(chunks, payload, aligned16, phases), want, &l);
    if (st != KVX_OK)
        return st;
    const bool ldg = l.variant == KVX_VARIANT_LDG, stage = l.variant == KVX_VARIANT_STAGE;
    *out = kvx_launch{l.variant,
                      chunks ? kvx::work_ctas(l, (uint32_t)chunks, max_chunk) : 0,
                      ldg ? l.threads : stage ? 128 : 0,
                      ldg ? l.unroll : 0,
                      ldg ? 0 : l.stages,
                      (ldg || stage) ? l.store_policy : 0,
                      ldg ? (kvx::ldg_dynamic(l, (uint32_t)chunks, max_chunk) ? KVX_ASSIGN_DYNAMIC
                                                                             : KVX_ASSIGN_STATIC)
                          : 0};
    return KVX_OK;
}

kvx_status kvx_copy_batch_ex(const uint64_t *src, const uint64_t *dst, const uint64_t *sizes, size_t n,
                             int dir, const kvx_launch *want, void *stream_)
{
    NvtxRange range("kvx_copy_batch");
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    kvx_status st = check_env();
    if (st != KVX_OK)
        return st;
    if (n && src && dst && sizes && dir >= KVX_H2D && dir <= KVX_D2D && validate_level() == 0) {
        bool done = false;
        st = copy_batch_fast(src, dst, sizes, n, dir, want, stream, &done);
        if (done)
            return st;
    }
    uint64_t chunks = 0, payload = 0, aligned16 = 0, phases = 0;
    uint32_t max_chunk = 0;
    st = validate(src, dst, sizes, n, dir, validate_level(), &chunks, &payload, &max_chunk, &aligned16, &phases);
    if (st != KVX_OK)
        return st;
    Launch l;
    st = resolve(dir, batch_shape(chunks, payload, aligned16, phases), want, &l);
    if (st != KVX_OK)
        return st;
    if (chunks == 0)
        return KVX_OK;
    bool cap = false;
    st = is_capturing(stream, &cap);
    if (st != KVX_OK)
        return st;
    if (cap)
        return fail(KVX_ERR_CAPTURE,
                    "kvx_copy_batch writes a host staging slot; capture kvx_copy_uploaded instead");
    int dev = 0;
    KVX_CUDA_TRY(cudaGetDevice(&dev));
    Slot *s = nullptr;
    st = ring_acquire(dev, (size_t)chunks, &s);
    if (st != KVX_OK)
        return st;
    {
        NvtxRange pack_range("kvx pack");
        pack(src, dst, sizes, n, s->host + kvx::kTableHeader, chunks);
    }
    log_batch("kvx_copy_batch", dir, n, chunks, payload, l);
    return launch_from_slot(dev, s, dir, l, chunks, max_chunk, stream);
}

kvx_status kvx_copy_batch(const uint64_t *src, const uint64_t *dst, const uint64_t *sizes, size_t n,
                          int dir, int cta_budget, void *stream)
{
    if (cta_budget < 0)
        return fail(KVX_ERR_INVALID_ARG, "cta_budget %d < 0", cta_budget);
    kvx_launch l{};
    l.cta_budget = cta_budget;
    return kvx_copy_batch_ex(src, dst, sizes, n, dir, &l, stream);
}

kvx_status kvx_desc_buf_create(size_t max_chunks, kvx_desc_buf **out)
{
    if (!out)
        return fail(KVX_ERR_INVALID_ARG, "null output");
    *out = nullptr;
    if (max_chunks < 1 || max_chunks > KVX_MAX_CHUNKS)
        return fail(KVX_ERR_CAPACITY, "max_chunks %zu not in 1..KVX_MAX_CHUNKS", max_chunks);
    kvx_desc_buf *b = new (std::nothrow) kvx_desc_buf;
    if (!b)
        return fail(KVX_ERR_CAPACITY, "out of host memory");
    cudaError_t e = cudaGetDevice(&b->device);
    if (e == cudaSuccess && (b->device < 0 || b->device >= kMaxDevices)) {
        delete b;
        return fail(KVX_ERR_INVALID_ARG, "device out of range");
    }
    if (e == cudaSuccess) {
        const kvx_status est = err_flags(b->device, &b->err);
        if (est != KVX_OK) {
            delete b;
            return est;
        }
    }
    const size_t bytes = (max_chunks + kvx::kTableHeader) * sizeof(kvx_chunk);
    if (e == cudaSuccess)
        e = cudaMalloc(reinterpret_cast<void **>(&b->dev), bytes);
    if (e == cudaSuccess)
        e = cudaHostAlloc(reinterpret_cast<void **>(&b->host), bytes, cudaHostAllocPortable);
    if (e == cudaSuccess)
        memset(b->host, 0, kvx::kTableHeader * sizeof(kvx_chunk));
    if (e == cudaSuccess)
        e = cudaEventCreateWithFlags(&b->upload_done, cudaEventDisableTiming);
    if (e == cudaSuccess)
        e = cudaEventCreateWithFlags(&b->last_use, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        if (b->dev)
            cudaFree(b->dev);
        if (b->host)
            cudaFreeHost(b->host);
        if (b->upload_done)
            cudaEventDestroy(b->upload_done);
        delete b;
        return cuda_fail(e, "kvx_desc_buf_create");
    }
    b->cap = max_chunks;
    if (!kvx::handle_add(b, kvx::kHandleDescBuf)) {
        cudaFree(b->dev);
        cudaFreeHost(b->host);
        cudaEventDestroy(b->upload_done);
        cudaEventDestroy(b->last_use);
        delete b;
        return fail(KVX_ERR_CAPACITY, "kvx_desc_buf_create: out of host memory");
    }
    *out = b;
    return KVX_OK;
}

kvx_status kvx_upload_descriptors(kvx_desc_buf *b, const uint64_t *src, const uint64_t *dst,
                                  const uint64_t *sizes, size_t n, int dir, void *stream_)
{
    NvtxRange range("kvx_upload_descriptors");
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (!b)
        return fail(KVX_ERR_INVALID_ARG, "null descriptor buffer");
    if (!kvx::handle_live(b, kvx::kHandleDescBuf))
        return fail(KVX_ERR_INVALID_ARG, "not a live descriptor buffer (destroyed, or never created)");
    kvx_status st = check_env();
    if (st != KVX_OK)
        return st;
    uint64_t chunks = 0, payload = 0, aligned16 = 0, phases = 0;
    uint32_t max_chunk = 0;
    st = validate(src, dst, sizes, n, dir, validate_level(), &chunks, &payload, &max_chunk, &aligned16, &phases);
    if (st != KVX_OK)
        return st;
    if (chunks > b->cap)
        return fail(KVX_ERR_CAPACITY, "batch needs %llu chunks, buffer holds %zu",
                    (unsigned long long)chunks, b->cap);
    Launch l;
    st = resolve(dir, batch_shape(chunks, payload, aligned16, phases), nullptr, &l);
    if (st != KVX_OK)
        return st;
    bool cap = false;
    st = is_capturing(stream, &cap);
    if (st != KVX_OK)
        return st;
    if (cap)
        return fail(KVX_ERR_CAPTURE, "kvx_upload_descriptors writes host staging memory");
    std::lock_guard<std::mutex> g(b->mu);
    if (b->upload_recorded) {
        KVX_CUDA_TRY(cudaEventSynchronize(b->upload_done));
        b->upload_recorded = false;
    }
    {
        NvtxRange pack_range("kvx pack");
        pack(src, dst, sizes, n, b->host + kvx::kTableHeader, chunks);
    }
    if (chunks)
        KVX_CUDA_TRY(cudaMemcpyAsync(b->dev, b->host, (size_t)(chunks + kvx::kTableHeader) * sizeof(kvx_chunk),
                                     cudaMemcpyHostToDevice, stream));
    KVX_CUDA_TRY(cudaEventRecord(b->upload_done, stream));
    b->upload_recorded = true;
    b->n_chunks = (uint32_t)chunks;
    b->max_chunk = max_chunk;
    b->payload = payload;
    b->dir = dir;
    b->selected = {l.variant, l.ctas, l.threads, l.unroll, l.stages, l.store_policy, l.assign};
    b->matched = l.matched;
    return KVX_OK;
}

kvx_status kvx_copy_uploaded_ex(kvx_desc_buf *b, const kvx_launch *want, void *stream_)
{
    NvtxRange range("kvx_copy_uploaded");
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (!b)
        return fail(KVX_ERR_INVALID_ARG, "null descriptor buffer");
    if (!kvx::handle_live(b, kvx::kHandleDescBuf))
        return fail(KVX_ERR_INVALID_ARG, "not a live descriptor buffer (destroyed, or never created)");
    kvx_status st = check_env();
    if (st != KVX_OK)
        return st;
    // One call at a time per buffer: the wait on the previous copy, the launch
    // and the record of this one go together, so copies from several threads
    // never overlap on the buffer's table (and its work counter).
    std::lock_guard<std::mutex> g(b->mu);
    kvx_launch merged = b->selected;
    if (want) {
        if (want->variant < 0 || want->variant > KVX_VARIANT_STAGE || want->cta_budget < 0)
            return fail(KVX_ERR_INVALID_ARG, "bad variant %d or cta_budget %d", want->variant,
                        want->cta_budget);
        if (want->variant)
            merged.variant = want->variant;
        if (want->cta_budget)
            merged.cta_budget = want->cta_budget;
        if (want->threads)
            merged.threads = want->threads;
        if (want->unroll)
            merged.unroll = want->unroll;
        if (want->stages)
            merged.stages = want->stages;
        if (want->store_policy)
            merged.store_policy = want->store_policy;
        if (want->assign)
            merged.assign = want->assign;
        // another variant's ring size is not a request for the STAGE ring
        if (want->variant == KVX_VARIANT_STAGE && b->selected.variant != KVX_VARIANT_STAGE && !want->stages &&
            merged.stages != 2 && merged.stages != 4 && merged.stages != 8)
            merged.stages = 0;
    }
    Launch l;
    st = resolve(b->dir, BatchShape{}, &merged, &l);
    if (st != KVX_OK)
        return st;
    l.matched = b->matched;
    l.prefetch = prefetch_for(b->dir, b->payload);
    if (b->n_chunks == 0)
        return KVX_OK;
    bool cap = false;
    st = is_capturing(stream, &cap);
    if (st != KVX_OK)
        return st;
    // Two copies over one table must not overlap: order this one after the
    // buffer's previous copy. On the same stream they are ordered already, and
    // waiting on that copy's event as well would make this launch wait for its
    // completion instead of overlapping its tail (programmatic dependent
    // launch). Streams are compared by cudaStreamGetId, which is never reused,
    // not by handle: a destroyed stream's handle can come back for a new one.
    unsigned long long sid = 0;
    if (!cap) {
        KVX_CUDA_TRY(cudaStreamGetId(stream, &sid));
        if (b->use_recorded && b->last_stream != sid)
            KVX_CUDA_TRY(cudaStreamWaitEvent(stream, b->last_use, 0));
    }
    cudaError_t e = kvx::launch_copy(l, b->dev, b->n_chunks, b->max_chunk, b->err, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "copy kernel launch");
    if (!cap) {
        KVX_CUDA_TRY(cudaEventRecord(b->last_use, stream));
        b->use_recorded = true;
        b->last_stream = sid;
    }
    return KVX_OK;
}

kvx_status kvx_copy_uploaded(kvx_desc_buf *b, int cta_budget, void *stream)
{
    if (cta_budget < 0)
        return fail(KVX_ERR_INVALID_ARG, "cta_budget %d < 0", cta_budget);
    kvx_launch l{};
    l.cta_budget = cta_budget;
    return kvx_copy_uploaded_ex(b, &l, stream);
}

kvx_status kvx_desc_buf_info(const kvx_desc_buf *b, size_t *n_chunks, uint64_t *payload,
                             kvx_launch *selected)
{
    if (!b)
        return fail(KVX_ERR_INVALID_ARG, "null descriptor buffer");
    if (!kvx::handle_live(b, kvx::kHandleDescBuf))
        return fail(KVX_ERR_INVALID_ARG, "not a live descriptor buffer (destroyed, or never created)");
    std::lock_guard<std::mutex> g(b->mu);
    if (n_chunks)
        *n_chunks = b->n_chunks;
    if (payload)
        *payload = b->payload;
    if (selected)
        *selected = b->selected;
    return KVX_OK;
}

kvx_status kvx_desc_buf_destroy(kvx_desc_buf *b)
{
    if (!b)
        return KVX_OK;
    if (!kvx::handle_remove(b, kvx::kHandleDescBuf))
        return fail(KVX_ERR_INVALID_ARG, "not a live descriptor buffer (destroyed, or never created)");
    if (b->upload_recorded)
        cudaEventSynchronize(b->upload_done);
    if (b->use_recorded)
        cudaEventSynchronize(b->last_use);
    cudaFree(b->dev);
    cudaFreeHost(b->host);
    cudaEventDestroy(b->upload_done);
    cudaEventDestroy(b->last_use);
    delete b;
    return KVX_OK;
}

kvx_status kvx_devlist_create(uint32_t max_n, kvx_devlist **out)
{
    if (!out)
        return fail(KVX_ERR_INVALID_ARG, "null output");
    *out = nullptr;
    if (max_n < 1 || max_n > (1u << 24))
        return fail(KVX_ERR_CAPACITY, "max_n %u not in 1..2^24", max_n);
    kvx_devlist *l = new (std::nothrow) kvx_devlist;
    if (!l)
        return fail(KVX_ERR_CAPACITY, "out of host memory");
    l->max_n = max_n;
    cudaError_t e = cudaGetDevice(&l->device);
    if (e == cudaSuccess && (l->device < 0 || l->device >= kMaxDevices)) {
        delete l;
        return fail(KVX_ERR_INVALID_ARG, "device out of range");
    }
    if (e == cudaSuccess) {
        const kvx_status est = err_flags(l->device, &l->err);
        if (est != KVX_OK) {
            delete l;
            return est;
        }
    }
    if (e == cudaSuccess)
        e = cudaMalloc(reinterpret_cast<void **>(&l->meta), 256 + kvx::devlist_scratch_bytes(max_n));
    if (e == cudaSuccess)
        e = cudaEventCreateWithFlags(&l->last_use, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        if (l->meta)
            cudaFree(l->meta);
        delete l;
        return cuda_fail(e, "kvx_devlist_create");
    }
    l->offsets = reinterpret_cast<uint64_t *>(reinterpret_cast<char *>(l->meta) + 256);
    if (!kvx::handle_add(l, kvx::kHandleDevList)) {
        cudaFree(l->meta);
        cudaEventDestroy(l->last_use);
        delete l;
        return fail(KVX_ERR_CAPACITY, "kvx_devlist_create: out of host memory");
    }
    *out = l;
    return KVX_OK;
}

kvx_status kvx_devlist_destroy(kvx_devlist *l)
{
    if (!l)
        return KVX_OK;
    if (!kvx::handle_remove(l, kvx::kHandleDevList))
        return fail(KVX_ERR_INVALID_ARG, "not a live device list (destroyed, or never created)");
    if (l->use_recorded)
        cudaEventSynchronize(l->last_use);
    cudaFree(l->meta);
    cudaEventDestroy(l->last_use);
    delete l;
    return KVX_OK;
}

kvx_status kvx_copy_device_list(kvx_devlist *l, const uint64_t *src, const uint64_t *dst,
                                const uint64_t *sizes, const uint32_t *count, int dir,
                                const kvx_launch *want, void *stream_)
{
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (!l)
        return fail(KVX_ERR_INVALID_ARG, "null device list");
    if (!kvx::handle_live(l, kvx::kHandleDevList))
        return fail(KVX_ERR_INVALID_ARG, "not a live device list (destroyed, or never created)");
    kvx_status st = check_env();
    if (st != KVX_OK)
        return st;
    if (!src || !dst || !sizes || !count)
        return fail(KVX_ERR_INVALID_ARG, "null device array");
    if (((uintptr_t)src | (uintptr_t)dst | (uintptr_t)sizes) & 7u || (uintptr_t)count & 3u)
        return fail(KVX_ERR_ALIGN, "device arrays must be 8-byte aligned (the count 4-byte aligned)");
    if (dir < KVX_H2D || dir > KVX_D2D)
        return fail(KVX_ERR_INVALID_ARG, "dir %d is not KVX_H2D, KVX_D2H or KVX_D2D", dir);
    // Device lists are copied by the LDG variant: start from the table's LDG
    // row for the direction (its small-chunk row) and apply the caller's fields.
    if (want && want->variant && want->variant != KVX_VARIANT_LDG)
        return fail(KVX_ERR_INVALID_ARG, "device lists are copied by the LDG variant only");
    BatchShape list_shape;
    list_shape.matched = true;  // not a STAGE row: the list's phases are not known on the host
    // nor its payload, and the grid is not clamped to the work: take the
    // mid-size rows rather than the largest batches' grids
    list_shape.payload = 48ull << 20;
    kvx_launch merged = table_launch(dir, list_shape);
    if (want) {
        if (want->cta_budget < 0)
            return fail(KVX_ERR_INVALID_ARG, "cta_budget %d < 0", want->cta_budget);
        if (want->cta_budget)
            merged.cta_budget = want->cta_budget;
        if (want->threads)
            merged.threads = want->threads;
        if (want->unroll)
            merged.unroll = want->unroll;
        if (want->store_policy)
            merged.store_policy = want->store_policy;
        if (want->assign)
            merged.assign = want->assign;
    }
    merged.variant = KVX_VARIANT_LDG;
    Launch lc;
    st = resolve(dir, BatchShape{}, &merged, &lc);
    if (st != KVX_OK)
        return st;
    bool cap = false;
    st = is_capturing(stream, &cap);
    if (st != KVX_OK)
        return st;
    // The list's scratch serves one copy at a time: outside capture, order this
    // copy after the list's previous one when that ran on another stream (same
    // stream: ordered already, and a wait would cancel the launch overlap).
    std::lock_guard<std::mutex> g(l->mu);
    unsigned long long sid = 0;
    if (!cap) {
        KVX_CUDA_TRY(cudaStreamGetId(stream, &sid));
        if (l->use_recorded && l->last_stream != sid)
            KVX_CUDA_TRY(cudaStreamWaitEvent(stream, l->last_use, 0));
    }
    cudaError_t e = kvx::launch_devlist(lc, src, dst, sizes, count, l->max_n, l->meta, l->offsets, l->err, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "device-list launch");
    if (!cap) {
        KVX_CUDA_TRY(cudaEventRecord(l->last_use, stream));
        l->use_recorded = true;
        l->last_stream = sid;
    }
    return KVX_OK;
}

kvx_status kvx_status_enqueue(void *stream_, kvx_status_token *tok)
{
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (!tok)
        return fail(KVX_ERR_INVALID_ARG, "null token");
    int dev = 0;
    KVX_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(KVX_ERR_INVALID_ARG, "device %d out of range", dev);
    bool cap = false;
    kvx_status st = is_capturing(stream, &cap);
    if (st != KVX_OK)
        return st;
    if (cap)
        return fail(KVX_ERR_CAPTURE, "a status read waits on the host; enqueue it on the stream that replays the graph");
    unsigned *err = nullptr;
    st = err_flags(dev, &err);  // registers the flags before any kernel could need them
    if (st != KVX_OK)
        return st;
    StatusEvents &w = g_status_events[dev];
    std::lock_guard<std::mutex> g(w.mu);
    const unsigned slot = w.next++ % kStatusEvents;
    if (!w.events[slot])
        KVX_CUDA_TRY(cudaEventCreateWithFlags(&w.events[slot], cudaEventDisableTiming));
    KVX_CUDA_TRY(cudaEventRecord(w.events[slot], stream));
    tok->slot = slot;
    tok->gen = ++w.gen[slot];
    tok->device = dev;
    return KVX_OK;
}

namespace {

kvx_status token_event(const kvx_status_token *tok, cudaEvent_t *ev)
{
    if (!tok || tok->device < 0 || tok->device >= kMaxDevices || tok->slot >= kStatusEvents)
        return fail(KVX_ERR_INVALID_ARG, "not a status token");
    StatusEvents &sw = g_status_events[tok->device];
    std::lock_guard<std::mutex> g(sw.mu);
    if (!sw.events[tok->slot] || sw.gen[tok->slot] != tok->gen)
        return fail(KVX_ERR_INVALID_ARG, "status token expired: %u later reads reused its slot", kStatusEvents);
    *ev = sw.events[tok->slot];
    return KVX_OK;
}

}  // namespace

kvx_status kvx_status_query(const kvx_status_token *tok, int *ready)
{
    if (!ready)
        return fail(KVX_ERR_INVALID_ARG, "null output");
    *ready = 0;
    cudaEvent_t ev = nullptr;
    kvx_status st = token_event(tok, &ev);
    if (st != KVX_OK)
        return st;
    const cudaError_t e = cudaEventQuery(ev);
    if (e == cudaErrorNotReady) {
        cudaGetLastError();
        return KVX_OK;
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaEventQuery(status read)");
    *ready = 1;
    return bits_status(take_err(tok->device));
}

kvx_status kvx_status_wait(const kvx_status_token *tok)
{
    cudaEvent_t ev = nullptr;
    kvx_status st = token_event(tok, &ev);
    if (st != KVX_OK)
        return st;
    KVX_CUDA_TRY(cudaEventSynchronize(ev));
    return bits_status(take_err(tok->device));
}

kvx_status kvx_stream_check(void *stream)
{
    int dev = 0;
    KVX_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(KVX_ERR_INVALID_ARG, "device %d out of range", dev);
    unsigned *err = nullptr;
    kvx_status st = err_flags(dev, &err);
    if (st != KVX_OK)
        return st;
    KVX_CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    return bits_status(take_err(dev));
}

kvx_status kvx_device_query(int *sm_count, size_t *stack_bytes_per_thread, size_t *free_bytes,
                            size_t *total_bytes)
{
    int dev = 0;
    KVX_CUDA_TRY(cudaGetDevice(&dev));
    if (sm_count)
        KVX_CUDA_TRY(cudaDeviceGetAttribute(sm_count, cudaDevAttrMultiProcessorCount, dev));
    if (stack_bytes_per_thread)
        KVX_CUDA_TRY(cudaDeviceGetLimit(stack_bytes_per_thread, cudaLimitStackSize));
    if (free_bytes || total_bytes) {
        size_t f = 0, t = 0;
        KVX_CUDA_TRY(cudaMemGetInfo(&f, &t));
        if (free_bytes)
            *free_bytes = f;
        if (total_bytes)
            *total_bytes = t;
    }
    return KVX_OK;
}

kvx_status kvx_host_alloc(size_t bytes, void **out)
{
    if (!out || !bytes)
        return fail(KVX_ERR_INVALID_ARG, "null output or zero bytes");
    *out = nullptr;
    void *p = nullptr;
    KVX_CUDA_TRY(cudaHostAlloc(&p, bytes, cudaHostAllocMapped | cudaHostAllocPortable));
    void *dp = nullptr;
    cudaError_t e = cudaHostGetDevicePointer(&dp, p, 0);
    if (e != cudaSuccess || dp != p) {
        cudaFreeHost(p);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaHostGetDevicePointer");
        return fail(KVX_ERR_NOT_MAPPED, "device address of pinned memory differs from its host address");
    }
    *out = p;
    return KVX_OK;
}

kvx_status kvx_host_free(void *p)
{
    if (!p)
        return KVX_OK;
    KVX_CUDA_TRY(cudaFreeHost(p));
    return KVX_OK;
}

kvx_status kvx_copy_batch_memcpy(const uint64_t *src, const uint64_t *dst, const uint64_t *sizes,
                                 size_t n, int dir, void *stream_, size_t *n_ranges)
{
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    kvx_status st = check_env();
    if (st != KVX_OK)
        return st;
    st = validate(src, dst, sizes, n, dir, validate_level(), nullptr, nullptr);
    if (st != KVX_OK)
        return st;
    const cudaMemcpyKind kind = dir == KVX_H2D   ? cudaMemcpyHostToDevice
                                : dir == KVX_D2H ? cudaMemcpyDeviceToHost
                                                 : cudaMemcpyDeviceToDevice;
    size_t ranges = 0;
    size_t i = 0;
    while (i < n) {
        if (!sizes[i]) {
            ++i;
            continue;
        }
        uint64_t s = src[i], d = dst[i], z = sizes[i];
        size_t k = i + 1;
        while (k < n && sizes[k] && src[k] == s + z && dst[k] == d + z) {
            z += sizes[k];
            ++k;
        }
        KVX_CUDA_TRY(cudaMemcpyAsync(reinterpret_cast<void *>(d), reinterpret_cast<const void *>(s),
                                     (size_t)z, kind, stream));
        ++ranges;
        i = k;
    }
    if (n_ranges)
        *n_ranges = ranges;
    return KVX_OK;
}

kvx_status kvx_copy_contiguous(uint64_t dst, uint64_t src, uint64_t bytes, int dir, void *stream)
{
    if (dir < KVX_H2D || dir > KVX_D2D)
        return fail(KVX_ERR_INVALID_ARG, "dir %d is not KVX_H2D, KVX_D2H or KVX_D2D", dir);
    if (!bytes)
        return KVX_OK;
    if (!src || !dst)
        return fail(KVX_ERR_INVALID_ARG, "null address");
    const cudaMemcpyKind kind = dir == KVX_H2D   ? cudaMemcpyHostToDevice
                                : dir == KVX_D2H ? cudaMemcpyDeviceToHost
                                                 : cudaMemcpyDeviceToDevice;
    KVX_CUDA_TRY(cudaMemcpyAsync(reinterpret_cast<void *>(dst), reinterpret_cast<const void *>(src),
                                 (size_t)bytes, kind, static_cast<cudaStream_t>(stream)));
    return KVX_OK;
}

kvx_status kvx_debug_bounds(const uint64_t *lo, const uint64_t *hi, size_t n)
{
    if (n > KVX_DEBUG_BOUNDS_MAX)
        return fail(KVX_ERR_CAPACITY, "%zu debug bounds; at most KVX_DEBUG_BOUNDS_MAX (%u)", n,
                    KVX_DEBUG_BOUNDS_MAX);
    if (n && (!lo || !hi))
        return fail(KVX_ERR_INVALID_ARG, "null range array");
    for (size_t i = 0; i < n; ++i)
        if (lo[i] >= hi[i])
            return fail(KVX_ERR_INVALID_ARG, "debug bounds range %zu is empty or reversed", i);
    // the legacy stream's query fails while any stream of the device captures in global mode
    bool cap = false;
    kvx_status st = is_capturing(cudaStreamLegacy, &cap);
    if (st != KVX_OK)
        return st;
    if (cap)
        return fail(KVX_ERR_CAPTURE, "kvx_debug_bounds synchronises the device");
    cudaError_t e = kvx::set_debug_bounds(lo, hi, (uint32_t)n);
    if (e != cudaSuccess)
        return cuda_fail(e, "setting the debug bounds");
    return KVX_OK;
}

kvx_status kvx_selftest_wait_timeout(uint64_t timeout_ns, void *stream)
{
    if (timeout_ns < 1000000ull || timeout_ns > 10000000000ull)
        return fail(KVX_ERR_INVALID_ARG, "timeout_ns %llu not in [1 ms, 10 s]",
                    (unsigned long long)timeout_ns);
    int dev = 0;
    KVX_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(KVX_ERR_INVALID_ARG, "device %d out of range", dev);
    unsigned *err = nullptr;
    kvx_status st = err_flags(dev, &err);
    if (st != KVX_OK)
        return st;
    KVX_CUDA_TRY(kvx::launch_wait_selftest(timeout_ns, err, static_cast<cudaStream_t>(stream)));
    return KVX_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// kvx_copy_batch_noalloc: the same batch copy with no allocation at call time
// ---------------------------------------------------------------------------
namespace {

// The two chunk tables of kvx_copy_batch_noalloc (each its header record, then
// up to KVX_NOALLOC_MAX_CHUNKS records, padded to 256 bytes), in the library's
// own device memory: every GPU that loads the library holds these 4 MiB until
// exit. Calls fill them in turn, so that one call's upload can run while the
// previous call's copy still reads the other table; before an upload
// overwrites a table, the GPU waits for the last copy that read it
// (g_noalloc_read), on whichever stream that copy ran.
constexpr size_t kNoallocRecords = (kvx::kTableHeader + KVX_NOALLOC_MAX_CHUNKS + 7) / 8 * 8;
static __device__ __align__(256) kvx_chunk g_noalloc_table[2][kNoallocRecords];

// Host side of the table, same layout, header kept zero. The first call
// page-locks it (cudaHostRegister of the library's own static memory, as for
// the error flags), so that each upload is one DMA straight from it: a
// pageable copy went through the runtime's own staging buffer first and cost
// a 16,384-chunk batch 7 % of its device time and 30 us of host time. The
// next call packs only once the previous upload has completed (g_noalloc_up).
// Should the registration fail, the copy stays pageable: the runtime then
// stages the bytes before cudaMemcpyAsync returns, and no wait is needed.
alignas(4096) kvx_chunk g_noalloc_stage[kvx::kTableHeader + KVX_NOALLOC_MAX_CHUNKS];
bool g_noalloc_lock_tried = false;
bool g_noalloc_locked = false;
cudaEvent_t g_noalloc_up[kMaxDevices];  // per device: the last upload from the array
int g_noalloc_up_dev = -1;              // device of an upload not yet waited for, or -1
cudaEvent_t g_noalloc_read[kMaxDevices][2];  // per device and table: the last copy that read it
unsigned g_noalloc_next[kMaxDevices];        // per device: the table the next call fills

// Serialises callers from pack to launch: the host array has one owner at a
// time, and calls on one stream enqueue upload and kernel back to back.
std::mutex g_noalloc_mu;

// Device addresses of the two tables per device. In host code the symbol is
// only a host-side stand-in, so the address comes from cudaGetSymbolAddress
// with the device current (first call on each device). The same first call
// maps the library's error flags if no other call did (a registration of a
// static host page, not an allocation).
kvx_chunk *g_noalloc_dev[kMaxDevices][2];
unsigned *g_noalloc_err[kMaxDevices];

// With the lock held: the first call's setup on this device (the table's
// device address, the error flags, the page-locked host array and its upload
// event), then a wait until the previous upload no longer reads the array.
kvx_status noalloc_prepare(int dev)
{
    if (!g_noalloc_dev[dev][0]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_table);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(no-alloc chunk tables)");
        const kvx_status est = err_flags(dev, &g_noalloc_err[dev]);
        if (est != KVX_OK)
            return est;
        for (int t = 0; t < 2; ++t)
            if (!g_noalloc_read[dev][t])
                KVX_CUDA_TRY(cudaEventCreateWithFlags(&g_noalloc_read[dev][t], cudaEventDisableTiming));
        g_noalloc_dev[dev][0] = static_cast<kvx_chunk *>(p);
        g_noalloc_dev[dev][1] = static_cast<kvx_chunk *>(p) + kNoallocRecords;
    }
    if (!g_noalloc_lock_tried) {
        g_noalloc_lock_tried = true;
        g_noalloc_locked = cudaHostRegister(g_noalloc_stage, sizeof(g_noalloc_stage), cudaHostRegisterPortable) ==
                           cudaSuccess;
        if (!g_noalloc_locked)
            cudaGetLastError();  // keep the pageable copy
    }
    if (g_noalloc_locked && !g_noalloc_up[dev])
        KVX_CUDA_TRY(cudaEventCreateWithFlags(&g_noalloc_up[dev], cudaEventDisableTiming));
    if (g_noalloc_up_dev >= 0) {  // the array is still being read by the previous upload
        KVX_CUDA_TRY(cudaEventSynchronize(g_noalloc_up[g_noalloc_up_dev]));
        g_noalloc_up_dev = -1;
    }
    return KVX_OK;
}

// With the lock held and the array packed: upload it into the next table and
// launch. The upload waits for the last copy that read that table. When
// `stream` still has work queued, a page-locked upload goes on the side stream
// and `stream` waits for it, so that it overlaps that work (as kvx_copy_batch's
// uploads do); otherwise it goes on `stream`.
kvx_status noalloc_launch(int dev, const kvx::Launch &l, uint64_t chunks, uint32_t max_chunk, cudaStream_t stream)
{
    const unsigned t = g_noalloc_next[dev];
    kvx_chunk *table = g_noalloc_dev[dev][t];
    cudaError_t qe = cudaSuccess;
    const bool busy = stream_busy(stream, &qe);
    if (qe != cudaSuccess)
        return cuda_fail(qe, "cudaStreamQuery");
    cudaStream_t up = stream;
    if (busy && g_noalloc_locked)
        KVX_CUDA_TRY(aux_stream(dev, kAuxNoalloc, &up));
    KVX_CUDA_TRY(cudaStreamWaitEvent(up, g_noalloc_read[dev][t], 0));
    KVX_CUDA_TRY(cudaMemcpyAsync(table, g_noalloc_stage, (size_t)(chunks + kvx::kTableHeader) * sizeof(kvx_chunk),
                                 cudaMemcpyHostToDevice, up));
    g_noalloc_next[dev] = t ^ 1u;
    if (g_noalloc_locked) {
        cudaError_t ue = cudaEventRecord(g_noalloc_up[dev], up);
        if (ue == cudaSuccess) {
            g_noalloc_up_dev = dev;
            if (up != stream)
                ue = cudaStreamWaitEvent(stream, g_noalloc_up[dev], 0);
        }
        if (ue != cudaSuccess) {
            // No later call could wait for this upload: finish it here, so that
            // it neither reads the host array nor writes the table afterwards.
            cudaStreamSynchronize(up);
            g_noalloc_up_dev = -1;
            return cuda_fail(ue, "no-alloc table upload ordering");
        }
    }
    cudaError_t e = kvx::launch_copy(l, table, (uint32_t)chunks, max_chunk, g_noalloc_err[dev], stream);
    // Recorded whether or not the launch went in: `stream` is past the upload
    // either way, and the next upload into this table waits for the event.
    const cudaError_t re = cudaEventRecord(g_noalloc_read[dev][t], stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "copy kernel launch");
    if (re != cudaSuccess)
        return cuda_fail(re, "cudaEventRecord(no-alloc table read)");
    return KVX_OK;
}

}  // namespace

extern "C" kvx_status kvx_copy_batch_noalloc(const uint64_t *src, const uint64_t *dst,
                                             const uint64_t *sizes, size_t n, int dir, int cta_budget,
                                             void *stream_)
{
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (cta_budget < 0)
        return fail(KVX_ERR_INVALID_ARG, "cta_budget %d < 0", cta_budget);
    kvx_status st = check_env();
    if (st != KVX_OK)
        return st;
    kvx_launch want{};
    want.cta_budget = cta_budget;
    // The common batch (level-0 validation, every descriptor within one chunk)
    // is validated while it is packed, in one pass split over the packing
    // threads, as kvx_copy_batch does; anything else takes the exact path below.
    if (validate_level() == 0 && n && n <= KVX_NOALLOC_MAX_CHUNKS && src && dst && sizes && dir >= KVX_H2D &&
        dir <= KVX_D2D) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        int dev = -1;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess)
            cudaGetLastError();  // the exact path below reports it
        else if (cs == cudaStreamCaptureStatusNone && dev >= 0 && dev < kMaxDevices) {
            std::lock_guard<std::mutex> g(g_noalloc_mu);
            st = noalloc_prepare(dev);
            if (st != KVX_OK)
                return st;
            uint64_t chunks = 0, payload = 0, aligned16 = 0, phases = 0;
            uint32_t max_chunk = 0;
            Launch l;
            if (pack_fast(src, dst, sizes, n, g_noalloc_stage + kvx::kTableHeader, &chunks, &payload, &max_chunk,
                          &aligned16, &phases) &&
                payload && resolve(dir, batch_shape(chunks, payload, aligned16, phases), &want, &l) == KVX_OK) {
                log_batch("kvx_copy_batch_noalloc", dir, n, chunks, payload, l);
                return noalloc_launch(dev, l, chunks, max_chunk, stream);
            }
        }
    }
    uint64_t chunks = 0, payload = 0, aligned16 = 0, phases = 0;
    uint32_t max_chunk = 0;
    st = validate(src, dst, sizes, n, dir, validate_level(), &chunks, &payload, &max_chunk, &aligned16, &phases);
    if (st != KVX_OK)
        return st;
    if (chunks > KVX_NOALLOC_MAX_CHUNKS)
        return fail(KVX_ERR_CAPACITY,
                    "batch needs %llu chunks; kvx_copy_batch_noalloc holds at most KVX_NOALLOC_MAX_CHUNKS "
                    "(%u)", (unsigned long long)chunks, KVX_NOALLOC_MAX_CHUNKS);
    Launch l;
    st = resolve(dir, batch_shape(chunks, payload, aligned16, phases), &want, &l);
    if (st != KVX_OK)
        return st;
    if (chunks == 0)
        return KVX_OK;
    // Under capture the table upload would become a graph node that reads the
    // shared host array at replay time, by then holding another call's records.
    bool cap = false;
    st = is_capturing(stream, &cap);
    if (st != KVX_OK)
        return st;
    if (cap)
        return fail(KVX_ERR_CAPTURE,
                    "kvx_copy_batch_noalloc uploads from a shared host array; capture kvx_copy_uploaded instead");
    int dev = 0;
    KVX_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(KVX_ERR_INVALID_ARG, "device %d out of range", dev);
    std::lock_guard<std::mutex> g(g_noalloc_mu);
    st = noalloc_prepare(dev);
    if (st != KVX_OK)
        return st;
    pack(src, dst, sizes, n, g_noalloc_stage + kvx::kTableHeader, chunks);
    log_batch("kvx_copy_batch_noalloc", dir, n, chunks, payload, l);
    return noalloc_launch(dev, l, chunks, max_chunk, stream);
}
