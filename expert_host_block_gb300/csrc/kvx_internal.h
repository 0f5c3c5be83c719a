// Internal interface between the host engine (kvx_engine.cu) and the device
// kernels (kvx_kernels.cu). Not part of the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kvx.h"

static_assert(sizeof(kvx_chunk) == 32, "chunk records are 32 bytes");

namespace kvx {

// Kinds of device error. Each is reported in its own flag word (kind bit b ->
// word b) of a device's kErrWords mapped pinned words, shared by all streams
// of the device; the host reads them as a bit set.
enum : unsigned {
    kDevErrTimeout = 1u,    // a bounded mbarrier wait gave up
    kDevErrBadRecord = 2u,  // a chunk record longer than KVX_CHUNK_BYTES, or out of phase for its launch
    kDevErrCount = 4u,      // a device-side descriptor count above the list's capacity (clamped)
    kDevErrBadDesc = 8u,    // a device-side descriptor failed validation (skipped)
    kDevErrBounds = 16u,    // a chunk (device list: a descriptor) outside the debug bounds (skipped)
};
constexpr int kErrWords = 5;

// Result of the device-list plan kernel, read by the device-list copy kernel.
struct DevListMeta {
    uint64_t total;      // chunks of the valid descriptors
    uint32_t n;          // descriptors taken (the count, clamped to the capacity)
    uint32_t max_chunk;  // longest chunk, bytes
    unsigned long long next;  // the copy kernel's unit counter (zeroed by the plan kernels)
    uint32_t tiles;      // plan tiles of kListTile descriptors in use
};

// A device list's plan is computed in tiles of this many descriptors: each
// descriptor's chunk offset within its tile, and per tile its first chunk
// (tile base), longest chunk and error bits.
constexpr uint32_t kListTile = 256;

// Bytes of a device list's scratch after its 256-byte DevListMeta: (max_n + 1)
// tile-relative chunk offsets, one 64-bit base and one 32-bit word (longest
// chunk | error bits << 16) per tile.
inline uint32_t devlist_tiles(uint32_t max_n) { return (max_n + kListTile - 1) / kListTile; }
inline size_t devlist_scratch_bytes(uint32_t max_n)
{
    return ((size_t)max_n + 1) * 8 + (size_t)devlist_tiles(max_n) * 12 + 8;
}

// Bounded-wait limit of the bulk kernel's mbarrier waits (ns of %globaltimer).
constexpr uint64_t kBulkWaitNs = 2000000000ull;

// A resolved launch: every field set.
struct Launch {
    int variant;       // KVX_VARIANT_LDG or KVX_VARIANT_BULK
    int ctas;          // grid size (already clamped to the work)
    int threads;       // LDG threads per CTA
    int unroll;        // LDG 16-byte loads in flight per lane
    int stages;        // BULK ring size in units of KVX_CHUNK_BYTES
    int store_policy;  // LDG store cache policy
    int assign;        // LDG: KVX_ASSIGN_STATIC or KVX_ASSIGN_DYNAMIC
    bool matched;      // LDG: every chunk's src and dst agree mod 16 (decided from the packed batch)
    bool shift;        // LDG, not matched: the one-path instance (kPhaseShift) instead of re-pairing
    bool pdl;          // launch with programmatic stream serialisation (KVX_PDL, default on)
    bool prefetch;     // LDG by position: prefetch the first units' sources into L2 before the wait
};

// The LDG kernel's instances (its template argument M), by how they copy a
// chunk whose src and dst differ in phase mod 16.
enum : int {
    kPhaseRepair = 0,   // a phase-matched path and a re-pairing path, chosen per chunk
    kPhaseMatched = 1,  // no such chunk in the batch (checked per record)
    kPhaseShift = 2,    // one path for both phases (source words shifted by 0 or 8 bytes)
};

// LDG kernel flags.
enum : uint32_t {
    kLdgPrefetch = 1u,  // before waiting for the grid before it, prefetch each lane's unit into L2
};

// Batches of at most this many payload bytes prefetch their sources (D2D): with
// the previous batch's writes still in L2, more would push lines out before use
// (4,096 x 16 KiB back to back: 0.91 without, 0.87 with).
constexpr uint64_t kPrefetchMaxPayload = 48ull << 20;

// Every device chunk table starts with one header record that holds the
// dynamic-assignment counters (next unit, warps done); the chunk records
// follow it. The header is zero after every upload (the host staging copy
// keeps it zero) and after every copy (the last warp zeroes it).
constexpr size_t kTableHeader = 1;

// KVX_ASSIGN_DYNAMIC applies to launches with at least this many work units
// per warp; smaller ones are assigned by position.
constexpr uint64_t kDynamicMinUnitsPerWarp = 8;

// Grid needed to give every CTA some work, for a chunk count, the longest
// chunk and the variant.
int work_ctas(const Launch &l, uint32_t n_chunks, uint32_t max_chunk_len);

// Whether an LDG launch takes its units from the table's counter: asked for
// (KVX_ASSIGN_DYNAMIC) and at least kDynamicMinUnitsPerWarp units per warp.
bool ldg_dynamic(const Launch &l, uint32_t n_chunks, uint32_t max_chunk_len);

// Enqueue the copy kernel over a device-resident chunk table: `table` points at
// its header record, n_chunks records follow. max_chunk_len is the longest
// record's len (it sets the LDG kernel's passes per chunk).
cudaError_t launch_copy(const Launch &l, kvx_chunk *table, uint32_t n_chunks,
                        uint32_t max_chunk_len, unsigned *err, cudaStream_t stream);

// Enqueue the plan and copy kernels over a device-resident descriptor list:
// count and arrays in device memory, meta and offsets[max_n + 1] scratch.
// l.ctas is used as is (the work is not known on the host).
cudaError_t launch_devlist(const Launch &l, const uint64_t *src, const uint64_t *dst,
                           const uint64_t *sizes, const uint32_t *count, uint32_t max_n,
                           DevListMeta *meta, uint64_t *offsets, unsigned *err, cudaStream_t stream);


// Set the calling thread's kvx_last_error() message and return `status`.
kvx_status set_error(kvx_status status, const char *message);

// The live handles of the library's opaque objects. Every entry point that
// takes a handle looks it up before touching it, so a destroyed handle, or a
// pointer that never was one, is KVX_ERR_INVALID_ARG instead of a use after
// free. (Destroying a handle while another thread still uses it remains the
// caller's error.)
enum HandleKind : int { kHandleDescBuf = 1, kHandleDevList = 2, kHandleTransfer = 3 };
bool handle_add(const void *h, HandleKind kind);     // false: out of host memory
bool handle_remove(const void *h, HandleKind kind);  // false: not a live handle of that kind
bool handle_live(const void *h, HandleKind kind);

// Replace the current device's debug bounds (kvx_debug_bounds) with the n
// ranges [lo[i], hi[i]); n == 0 turns the check off. Synchronises the device.
cudaError_t set_debug_bounds(const uint64_t *lo, const uint64_t *hi, uint32_t n);

// Enqueue the bounded-wait self-test kernel.
cudaError_t launch_wait_selftest(uint64_t timeout_ns, unsigned *err, cudaStream_t stream);

// Shared memory of a bulk ring of `units` x KVX_CHUNK_BYTES.
size_t bulk_smem_bytes(int units);

}  // namespace kvx
