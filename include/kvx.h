/*
 * kvx: batched, descriptor-driven scatter/gather copies between mapped pinned
 * host memory and HBM, for one NVIDIA GB300 (sm_103a).
 *
 * The operation. A batch is n descriptors (src_i, dst_i, size_i). The result
 * of a batch is the result of one memcpy(dst_i, src_i, size_i) per
 * descriptor; no other byte changes. The pages replace one directional CUDA
 * memcpy per fragment with one descriptor upload and one copy-kernel launch
 * (PegaFlow issue #408, "Kernel transfer backend causes decode TPOT tail
 * spikes under concurrent KV transfers", §Summary), and the copy kernel moves
 * the same bytes as the path it replaces (FreeToken issue #751, "[Perf]
 * Offloaded decode: gather missed experts with a few TMA bulk-copy CTAs",
 * §What we changed; vLLM PR #42212 report, §实现拆解 items 1 and 4).
 *
 * How kvx runs a batch. The host validates the descriptors, cuts each one
 * into chunks of at most KVX_CHUNK_BYTES at 8-byte granularity, packs the
 * 32-byte chunk records into a pinned staging buffer, uploads the table with
 * one cudaMemcpyAsync (small tables are read by the kernel in place
 * instead) and launches one persistent copy kernel on `stream` with at
 * most `cta_budget` CTAs. Every call is enqueue-only: it returns once the
 * work is queued (PegaFlow issue #408, follow-up §2: the transfer backend
 * contract is enqueue-only and never synchronises).
 *
 * Common rules for every entry point below:
 *   - Addresses are plain 64-bit virtual addresses in the unified address
 *     space. Host memory must be mapped pinned memory (kvx_host_alloc, or
 *     cudaHostAlloc with cudaHostAllocMapped on a unified-addressing system)
 *     so that the device can use the same address. kvx does not translate.
 *   - src_i, dst_i and size_i must be multiples of 8 (the 8-byte word
 *     granularity of the vLLM kernel, which the report selects only for
 *     8-byte-aligned pages: vLLM PR #42212 report, §实现拆解 item 2). kvx
 *     rejects other values with KVX_ERR_ALIGN instead of truncating them.
 *     16-byte alignment is not required; it only makes the fast paths apply.
 *   - Destination ranges of one batch must not overlap one another or any
 *     source range of the batch. Source ranges may overlap. Under that rule
 *     the result does not depend on descriptor order, and kvx gives no order
 *     among descriptors. kvx checks it only at validation level >= 1
 *     (kvx_set_validate_level); at level 0 an overlapping batch is undefined.
 *   - A size of 0 is a no-op (its addresses are not checked); n == 0 is a
 *     no-op that returns KVX_OK.
 *   - The caller owns all payload memory and the three descriptor arrays.
 *     The arrays are read during the call only and may be reused when it
 *     returns. The payload must stay valid until the stream reaches the copy.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream) of the
 *     device that is current in the calling thread.
 *   - Back-to-back copies: every copy kernel is launched with programmatic
 *     stream serialisation (programmatic dependent launch). A copy may start
 *     launching while the kernel before it on `stream` still runs; until that
 *     kernel has completed and its writes are visible it reads only its own
 *     chunk table, never payload. The copy also lets the next kernel on
 *     `stream` launch early: a kernel launched after a kvx copy with
 *     cudaLaunchAttributeProgrammaticStreamSerialization must call
 *     cudaGridDependencySynchronize() before it reads the copy's destination
 *     or writes its source, as that attribute requires of every kernel.
 *     Kernels launched without the attribute, copy-engine work and events
 *     are ordered as usual. The environment variable KVX_PDL=0 launches the
 *     copy kernels without the attribute.
 *   - Errors: a non-KVX_OK status means nothing was enqueued, except
 *     KVX_ERR_CUDA from a launch, which may follow a completed table upload.
 *     kvx_last_error() gives a one-line message for the calling thread.
 *     Device-side errors (a bounded wait that gave up) are reported by
 *     kvx_stream_check. No entry point aborts the process or traps the GPU.
 *   - Environment (read once per process; an unknown or malformed value makes
 *     every call fail with KVX_ERR_INVALID_ARG naming the variable, so a typo
 *     never silently selects a default):
 *       KVX_VARIANT=auto|ldg|bulk|stage   override the table's variant
 *       KVX_CTA_BUDGET=<0..2^20>          override the table's grid budget (0: none)
 *       KVX_VALIDATE=0|1|2                initial validation level
 *       KVX_PDL=0|1                       programmatic dependent launch (1)
 *       KVX_LOG=0|1|2                     stderr: failing statuses; + one line a batch
 *       KVX_NVTX=0|1                      NVTX ranges around entry points and packing
 *       KVX_PACK_THREADS=<0..64>          host packing threads for large batches
 *       KVX_TABLE=<file>                  launch-table rows tried before the built-in
 *         ones, one per line ('#' starts a comment):
 *           dir max_mean_chunk variant cta_budget threads unroll stages
 *               store_policy [assign [min_payload [phase [max_payload]]]]
 *         dir h2d|d2h|d2d; max_mean_chunk and max_payload bytes or "inf";
 *         variant ldg|bulk|stage; assign static|dynamic|auto; phase
 *         any|unmatched (unmatched: only batches with a chunk whose source and
 *         destination differ mod 16). A row applies when the batch's mean chunk
 *         and payload fall within its bounds (a bulk row also needs 90 % of the
 *         bytes in 16-byte aligned descriptors); explicit kvx_launch fields
 *         override it.
 *   - Opaque handles (kvx_desc_buf, kvx_devlist, kvx_transfer): kvx keeps a
 *     registry of the live ones, so passing a destroyed handle, or a pointer
 *     that never was one, returns KVX_ERR_INVALID_ARG without touching it
 *     (destroying a handle twice included). Destroying a handle while another
 *     thread is inside a call with it is the caller's error.
 */
#ifndef KVX_H
#define KVX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVX_VERSION_MAJOR 0
#define KVX_VERSION_MINOR 4

/* Largest chunk a descriptor is cut into: 16 KiB, the chunk of the FreeToken
 * gather (FreeToken issue #751, §What we changed: "chunks of up to 16 KiB,
 * each inside one bank row"). */
#define KVX_CHUNK_BYTES 16384u
/* Most chunks one batch may expand to (a 128 MiB chunk table). */
#define KVX_MAX_CHUNKS (1u << 22)

typedef enum kvx_dir {
    KVX_H2D = 0, /* mapped pinned host -> device memory */
    KVX_D2H = 1, /* device memory -> mapped pinned host */
    KVX_D2D = 2  /* device memory -> device memory */
} kvx_dir;

typedef enum kvx_variant {
    KVX_VARIANT_AUTO = 0, /* pick from the calibrated table by direction and size */
    KVX_VARIANT_LDG = 1,  /* 16-byte loads/stores by every lane, several in flight */
    KVX_VARIANT_BULK = 2, /* cp.async.bulk through a shared::cta ring, one issuing lane */
    KVX_VARIANT_STAGE = 3 /* cp.async.bulk loads into a shared::cta ring per warp, 16-byte stores by the
                             whole warp at any 8-byte phase (128 threads a CTA): for batches whose
                             sources and destinations do not agree mod 16 */
} kvx_variant;

/* How the LDG kernel hands work units (one warp pass over a chunk) to warps. */
typedef enum kvx_assign {
    KVX_ASSIGN_AUTO = 0,    /* the table's choice: DYNAMIC for H2D and D2H, STATIC for D2D */
    KVX_ASSIGN_STATIC = 1,  /* unit u to warp u mod (warps in the grid) */
    KVX_ASSIGN_DYNAMIC = 2  /* each warp takes its next unit from a counter kept in the chunk
                               table's device allocation, so warps the link serves faster take
                               more units; two copies over the same table must not overlap.
                               Applies when there are at least 8 units per warp (fewer go by
                               position) */
} kvx_assign;

typedef enum kvx_status {
    KVX_OK = 0,
    KVX_ERR_INVALID_ARG = 1,  /* null array, bad dir/variant/budget, null address, address overflow */
    KVX_ERR_ALIGN = 2,        /* an address or size is not a multiple of 8 */
    KVX_ERR_OVERLAP = 3,      /* (validation level >= 1) destination ranges overlap */
    KVX_ERR_CAPACITY = 4,     /* more than KVX_MAX_CHUNKS chunks, or more than a buffer holds, or the
                                 host heap ran out (no C++ exception ever crosses this boundary) */
    KVX_ERR_NOT_MAPPED = 5,   /* (validation level 2) an address is not of the kind dir names */
    KVX_ERR_CUDA = 6,         /* a CUDA runtime call failed; see kvx_last_error() */
    KVX_ERR_TIMEOUT = 7,      /* a bounded device wait gave up (reported by kvx_stream_check) */
    KVX_ERR_DEVICE_FAULT = 8, /* the device reported an inconsistent chunk record, or a chunk outside
                                 the debug bounds (kvx_debug_bounds) */
    KVX_ERR_CAPTURE = 9       /* the call is not allowed while `stream` is being captured */
} kvx_status;

/* One chunk record of the uploaded table: 32 bytes. `len` <= KVX_CHUNK_BYTES,
 * `desc` is the index of the descriptor the chunk belongs to. */
typedef struct kvx_chunk {
    uint64_t src;
    uint64_t dst;
    uint32_t len;
    uint32_t desc;
    uint64_t reserved;
} kvx_chunk;

/* Launch configuration. Zero in a field means "take it from the calibrated
 * table" (direction and mean chunk size select the row). */
typedef struct kvx_launch {
    int variant;         /* kvx_variant */
    int cta_budget;      /* maximum CTAs; the grid is min(cta_budget, work) */
    int threads;         /* LDG: threads per CTA, one of 128, 256, 512 (STAGE: always 128) */
    int unroll;          /* LDG: 16-byte loads in flight per lane, one of 2, 4, 8 */
    int stages;          /* BULK: shared-memory ring of stages x KVX_CHUNK_BYTES, 2..12; it is cut
                            into stages of the batch's longest chunk (at most 32 stages).
                            STAGE: 4 KiB units each warp keeps in flight, 2, 4 or 8 */
    int store_policy;    /* LDG and STAGE: 0 default, 1 write-through (.wt), 2 streaming (.cs) */
    int assign;          /* LDG: kvx_assign */
} kvx_launch;

/* Opaque, library-owned reusable descriptor buffer (device chunk table plus
 * its pinned staging buffer). */
typedef struct kvx_desc_buf kvx_desc_buf;

/* ---- the batch copy ----------------------------------------------------- */

/* Copy a batch: validate, chunk, pack, upload the chunk table and launch the
 * copy kernel on `stream`: one descriptor upload and one copy-kernel launch in
 * place of one memcpy per fragment (PegaFlow issue #408, §Summary), with the
 * three address/size arrays of the vLLM wrapper `swap_blocks_batch` (vLLM PR
 * #42212 report, §实现拆解 item 1). Enqueue-only (PegaFlow issue #408,
 * follow-up §2). `dir` is a kvx_dir; it selects the table row and
 * what validation level 2 checks (data moves through unified addresses in
 * every direction). `cta_budget`: 0 = calibrated default, > 0 = at most that
 * many CTAs, < 0 = KVX_ERR_INVALID_ARG. Not allowed during stream capture
 * (KVX_ERR_CAPTURE): it writes a pinned staging slot on the host. The staging
 * ring has 8 slots per device; a call takes the most recently used slot whose
 * copy has finished, and waits on the host only when none has (then for the
 * least recently used one). A slot allocates on first use and grows, once, for
 * a batch bigger than it holds. A batch of at most 4,096 chunks whose units
 * the kernel assigns by position is not uploaded (for D2D: only when `stream`
 * is idle): the kernel reads its records from the mapped staging slot.
 * Otherwise, when `stream` still has work queued, the table upload runs on a
 * library side stream (overlapping that work) and the copy kernel waits for
 * it on `stream`. The copy stays ordered after all earlier work on `stream`
 * either way. */
kvx_status kvx_copy_batch(const uint64_t *src_addrs, const uint64_t *dst_addrs,
                          const uint64_t *sizes, size_t n, int dir, int cta_budget,
                          void *stream);

/* kvx_copy_batch with an explicit launch configuration (NULL = all table):
 * the per-device grid limit the pages ask to expose instead of a constant
 * (PegaFlow issue #408, follow-up §Proposed direction, `KernelOptions`
 * `max_grid_blocks`). */
kvx_status kvx_copy_batch_ex(const uint64_t *src_addrs, const uint64_t *dst_addrs,
                             const uint64_t *sizes, size_t n, int dir,
                             const kvx_launch *launch, void *stream);

/* ---- reusable descriptor buffers (pinned staging + device table) -------- */
/* The vLLM transfer keeps three pinned descriptor buffers that it allocates
 * once and reuses for every transfer, so that the H2D copy of the descriptors
 * is truly asynchronous and no transfer allocates (vLLM PR #42212 report,
 * §实现拆解 item 3, `_new_descriptor_buffers`; §评论区精华, pinned memory).
 * A kvx_desc_buf is that buffer, holding the packed chunk table instead of
 * the three arrays, plus its device copy, so that a copy over it is a
 * fixed-shape launch with no host work (FreeToken issue #751, §What we
 * changed: fixed-shape, CUDA-graph capturable). */

/* Create a buffer for up to max_chunks chunk records (1..KVX_MAX_CHUNKS) on
 * the current device. Allocates device and pinned host memory (synchronous),
 * once, for reuse by every upload (vLLM PR #42212 report, §实现拆解 item 3). */
kvx_status kvx_desc_buf_create(size_t max_chunks, kvx_desc_buf **out);

/* Validate, chunk and pack a batch into the buffer's pinned staging area and
 * enqueue its upload on `stream`: the one descriptor upload of a batch
 * (PegaFlow issue #408, §Summary), into the reused pinned buffer (vLLM PR
 * #42212 report, §实现拆解 item 3). Waits on the host only while the buffer's
 * previous upload is still in flight. The caller orders this upload after any
 * kvx_copy_uploaded of the same buffer that is still running on another
 * stream (same stream: ordered already). Not allowed during capture. */
kvx_status kvx_upload_descriptors(kvx_desc_buf *buf, const uint64_t *src_addrs,
                                  const uint64_t *dst_addrs, const uint64_t *sizes,
                                  size_t n, int dir, void *stream);

/* Launch the copy kernel over the uploaded table. No host work besides the
 * launch: fixed shape, allowed inside CUDA graph capture (FreeToken issue
 * #751, §What we changed: the launch is fixed-shape and CUDA-graph
 * capturable). `cta_budget` as in
 * kvx_copy_batch. Two copies of one buffer must not run at the same time (a
 * dynamic-assignment copy keeps its work counter in the buffer): outside
 * capture, each copy first makes `stream` wait for the buffer's previous copy
 * (free when that was on the same stream); graph replays are the caller's to
 * order. Calls on one buffer from several threads are serialised by the
 * buffer (uploads and copies alike), so their copies never overlap. */
kvx_status kvx_copy_uploaded(kvx_desc_buf *buf, int cta_budget, void *stream);

/* kvx_copy_uploaded with an explicit launch configuration (NULL = table): the
 * bounded, device-specific grid of PegaFlow issue #408, follow-up §Proposed
 * direction (`KernelOptions`). */
kvx_status kvx_copy_uploaded_ex(kvx_desc_buf *buf, const kvx_launch *launch, void *stream);

/* Chunks and payload bytes of the last upload, and the launch configuration
 * the table selected for it (the device-aware profile's choice: PegaFlow
 * issue #408, follow-up §Proposed direction). Any output pointer may be
 * NULL. */
kvx_status kvx_desc_buf_info(const kvx_desc_buf *buf, size_t *n_chunks,
                             uint64_t *payload_bytes, kvx_launch *selected);

/* Wait for the buffer's last upload and last copy, then free it. The buffers
 * live as long as their owner wants them reused (vLLM PR #42212 report,
 * §实现拆解 item 3: allocated once and reused, not per transfer). */
kvx_status kvx_desc_buf_destroy(kvx_desc_buf *buf);

/* ---- descriptor lists that live on the device ---------------------------- */

/* A producer on the GPU (a MoE router choosing missed experts, a block manager
 * choosing KV pages) can write the descriptor arrays and their count in device
 * memory. Then the host knows neither, and the copy must be a fixed-shape
 * launch that reads the count on the device, so that it can be captured in a
 * CUDA graph and replayed with new contents (FreeToken issue #751, §What we
 * changed: "the miss count is read on the device, so the launch is
 * fixed-shape and CUDA-graph capturable").
 *
 * A kvx_devlist holds the device scratch of such copies for lists of up to
 * max_n descriptors: the plan results, each descriptor's 64-bit chunk offset
 * within its tile of 256 descriptors, and 12 bytes per tile (its first chunk,
 * longest chunk and error bits): about 8.05 bytes a descriptor. Create it
 * outside capture (it allocates device memory). */
typedef struct kvx_devlist kvx_devlist;

kvx_status kvx_devlist_create(uint32_t max_n, kvx_devlist **out); /* 1 <= max_n <= 2^24 */
kvx_status kvx_devlist_destroy(kvx_devlist *list);                /* waits for its last copy */

/* Enqueue the copy of the device-resident list: d_src, d_dst and d_sizes are
 * device arrays of at least max_n uint64 each (same meaning and rules as the
 * host arrays of kvx_copy_batch), d_count a device uint32 holding n. Three
 * launches on `stream` (two for a list of at most 256 descriptors): the plan,
 * as a tile kernel (up to 304 CTAs: validates tiles of 256 descriptors and
 * scans their chunk counts) and a one-CTA kernel (scans the tile totals), then
 * the LDG copy kernel with launch->cta_budget CTAs (the grid is not clamped to
 * the work, which the host does not know). No host work, no
 * allocation, no synchronisation: allowed inside stream capture; replaying
 * the graph copies whatever the arrays and count hold at replay time.
 * Host-side errors (null or misaligned arrays, bad dir or launch, a BULK
 * variant) return without enqueuing. Device-side problems are reported by
 * kvx_stream_check as KVX_ERR_DEVICE_FAULT: a count above max_n (only max_n
 * descriptors are copied) or a descriptor that fails validation (it is
 * skipped; the others are copied). Overlapping destinations are not
 * detected. The list's scratch is reused by every call, one copy at a time:
 * outside capture each call makes `stream` wait for the list's previous copy
 * when that was on another stream (calls from several threads are serialised
 * by the list); inside capture, copies of one list on different streams of the
 * graph are the caller's to order. */
kvx_status kvx_copy_device_list(kvx_devlist *list, const uint64_t *d_src, const uint64_t *d_dst,
                                const uint64_t *d_sizes, const uint32_t *d_count, int dir,
                                const kvx_launch *launch, void *stream);

/* ---- tail-bounded submission --------------------------------------------- */

/* A transfer cut into pieces of at most chunk_descriptors descriptors, each
 * submitted (through kvx_copy_batch_ex) only after the previous piece has
 * completed on the GPU. This bounds how long a transfer holds SMs and link
 * bandwidth at a time, at the cost of throughput, for serving where a
 * colocated decode's tail latency matters (PegaFlow issue #408, follow-up §2
 * and §Proposed direction: `chunk_descriptors` with event-based completion
 * backpressure; enqueue-only chunking does not help). kvx never blocks: the
 * caller's transfer worker calls kvx_transfer_poll until it reports done,
 * yielding in between. */
typedef struct kvx_transfer kvx_transfer;

kvx_status kvx_transfer_create(kvx_transfer **out);

/* Validate the whole batch (at the current validation level), take a copy of
 * the three arrays (the caller may reuse them on return), and submit the
 * first piece on `stream`. chunk_descriptors == 0 submits the batch as one
 * piece. KVX_ERR_INVALID_ARG while a piece of the previous transfer is still
 * in flight (poll it to done first). */
kvx_status kvx_transfer_start(kvx_transfer *t, const uint64_t *src_addrs, const uint64_t *dst_addrs,
                              const uint64_t *sizes, size_t n, int dir, size_t chunk_descriptors,
                              const kvx_launch *launch, void *stream);

/* Non-blocking: if the piece in flight has completed, submit the next one.
 * *done = 1 once every piece has completed. Start, poll and progress calls on
 * one transfer from several threads take turns (the transfer holds a lock). */
kvx_status kvx_transfer_poll(kvx_transfer *t, int *done);

/* Descriptors submitted so far and in total (either pointer may be NULL). */
kvx_status kvx_transfer_progress(const kvx_transfer *t, size_t *submitted, size_t *total);

/* Wait for the piece in flight, if any, and free the transfer. */
kvx_status kvx_transfer_destroy(kvx_transfer *t);

/* ---- Auto policy -------------------------------------------------------- */

/* Choose the path from the transfer's shape: merged range count (descriptors
 * that continue the previous one in both source and destination merge), total
 * bytes and mean range size (PegaFlow issue #408, §Discussion item 2). A few
 * large ranges go to the copy engines (per-range cudaMemcpyAsync: near the
 * link peak with no SM used): for KVX_POLICY_THROUGHPUT at most 8 ranges whose
 * mean is at least ranges x 256 KiB (where DMA measured faster than the
 * kernel), for KVX_POLICY_TAIL at most 16 ranges averaging at least 1 MiB.
 * Everything else goes to the copy kernel: for THROUGHPUT the variant and
 * launch the calibrated table picks for the batch (kvx_select_launch with no
 * request: LDG or STAGE, or the bulk ring from a KVX_TABLE row), for TAIL the bulk variant with 4
 * one-warp CTAs (the lightest footprint beside a colocated decode). */
typedef enum kvx_policy { KVX_POLICY_THROUGHPUT = 0, KVX_POLICY_TAIL = 1 } kvx_policy;
typedef enum kvx_path {
    KVX_PATH_KERNEL_LDG = 1,
    KVX_PATH_KERNEL_BULK = 2,
    KVX_PATH_DMA = 3,
    KVX_PATH_KERNEL_STAGE = 4
} kvx_path;

/* The path kvx_copy_batch_auto would take (host only; validation level 0). */
kvx_status kvx_auto_path(const uint64_t *src_addrs, const uint64_t *dst_addrs, const uint64_t *sizes,
                         size_t n, int dir, int policy, int *path);

/* Copy a batch along the path kvx_auto_path chooses; *path (may be NULL)
 * receives it. Same rules and errors as kvx_copy_batch. */
kvx_status kvx_copy_batch_auto(const uint64_t *src_addrs, const uint64_t *dst_addrs, const uint64_t *sizes,
                               size_t n, int dir, int policy, void *stream, int *path);

/* ---- host-only helpers (no CUDA call, no GPU needed) -------------------- */

/* Validate a batch at `level` (0: arrays, dir, alignment, overflow, capacity;
 * 1: + destination overlap; 2: + address kinds, which calls the CUDA
 * runtime). Returns the status kvx_copy_batch would return before enqueuing. */
kvx_status kvx_validate(const uint64_t *src_addrs, const uint64_t *dst_addrs,
                        const uint64_t *sizes, size_t n, int dir, int level);

/* The chunk table kvx would upload for a batch. With out == NULL only
 * *n_chunks is set. KVX_ERR_CAPACITY when it needs more than max_out. */
kvx_status kvx_plan_chunks(const uint64_t *src_addrs, const uint64_t *dst_addrs,
                           const uint64_t *sizes, size_t n, kvx_chunk *out,
                           size_t max_out, size_t *n_chunks);

/* The launch kvx_copy_batch_ex(..., want, ...) would make for this batch,
 * computed on the host without a device: validation level 0, the table row
 * for the batch's direction, mean chunk, payload and alignment, then the KVX_*
 * environment and `want` (NULL = none) over it. In *out, cta_budget is the
 * grid actually launched (at most the budget, at most the work; 0 for an
 * empty batch); fields the chosen variant does not use are 0; assign is what
 * the kernel will do (STATIC when DYNAMIC was asked for but the batch has
 * fewer than 8 units per warp). Same errors as kvx_copy_batch's validation. */
kvx_status kvx_select_launch(const uint64_t *src_addrs, const uint64_t *dst_addrs,
                             const uint64_t *sizes, size_t n, int dir, const kvx_launch *want,
                             kvx_launch *out);

/* The calibrated launch configuration for a direction and mean chunk size,
 * for a large batch of 16-byte aligned descriptors. Rows are chosen by
 * direction, mean chunk size and, for some rows, the batch's payload and
 * phases (the D2D grids grow with the payload; the D2D rows that select
 * KVX_VARIANT_STAGE apply only to batches of 128 MiB or more with a chunk
 * whose source and destination differ mod 16). A row that selects
 * KVX_VARIANT_BULK (none of the built-in ones; a KVX_TABLE file may have
 * them) applies only to batches with at least 90 % of their bytes in
 * descriptors whose source, destination and size are multiples of 16. A batch
 * a row does not apply to takes the next matching row. */
kvx_status kvx_default_launch(int dir, uint64_t mean_chunk_bytes, kvx_launch *out);

/* Process-wide validation level for kvx_copy_batch / kvx_upload_descriptors
 * (0..2). Initial value: the KVX_VALIDATE environment variable, else 0. */
kvx_status kvx_set_validate_level(int level);
int kvx_get_validate_level(void);

/* The name of a kvx_status ("KVX_ERR_TIMEOUT"...), for the completion status
 * that the enqueue-only contract reads after the fact (PegaFlow issue #408,
 * follow-up §2: record completion, query it later). Never NULL:
 * "KVX_ERR_UNKNOWN" for a value that is not a kvx_status. */
const char *kvx_status_string(int status);
/* Message of the last non-OK status returned in the calling thread. */
const char *kvx_last_error(void);
int kvx_version(void); /* KVX_VERSION_MAJOR * 100 + KVX_VERSION_MINOR */

/* ---- device status, memory ---------------------------------------------- */

/* Synchronise `stream`, then read and clear the device's error flags: the
 * completion read that the enqueue-only copy leaves to the caller (PegaFlow
 * issue #408, follow-up §2: the transfer backend contract is enqueue-only,
 * so completion is recorded and read later, outside submit). Kernels set the
 * flags (a bounded wait that gave up, an inconsistent chunk record, a
 * device-list count above capacity or a bad device-list descriptor). The
 * flags live in a page of mapped pinned host memory that kvx registers with
 * the driver on its first use in the process (a static page, no allocation);
 * kernels set them with plain stores, so reading them needs no kernel. They
 * are shared by all streams of the device, so an error raised by a kernel on
 * another stream may be reported here. KVX_OK, KVX_ERR_TIMEOUT,
 * KVX_ERR_DEVICE_FAULT or KVX_ERR_CUDA. */
kvx_status kvx_stream_check(void *stream);

/* The current device's SM count, per-thread stack limit and free / total
 * memory (any pointer may be NULL): the inputs of a per-device launch profile,
 * and the check against the sm_120 bulk-copy pitfall, where the
 * cluster-scope destination form made the driver raise the per-thread
 * stack limit and hold 1.37 GiB of device memory (FreeToken issue #751,
 * §What we changed). kvx uses the .shared::cta form, which leaves both
 * unchanged. */
kvx_status kvx_device_query(int *sm_count, size_t *stack_bytes_per_thread, size_t *free_bytes,
                            size_t *total_bytes);

/* The same read without blocking, for a transfer worker that submits the
 * next batch before collecting the previous one (the enqueue-only contract of
 * PegaFlow issue #408, follow-up §2: record completion, poll it later).
 * kvx_status_enqueue records an event behind the work already on `stream`
 * and returns a token; nothing is added to the stream's work, so later work
 * on `stream` does not wait for the read. kvx_status_wait blocks until the
 * stream has reached the token, then reads and clears the device's error
 * flags and returns what kvx_stream_check would have; kvx_status_query does
 * not block (*ready = 0 while the stream has not reached the token;
 * otherwise *ready = 1 and the status). The flags are shared by all streams
 * of the device, so an error that work enqueued after the token (or on
 * another stream) has already raised may be reported by this token rather
 * than the next. Not allowed while `stream` is being captured
 * (KVX_ERR_CAPTURE): read the status after replaying the graph. A token
 * stays valid for the next 1,024 tokens of its device; after that,
 * KVX_ERR_INVALID_ARG. */
typedef struct kvx_status_token {
    uint64_t slot; /* opaque */
    uint64_t gen;  /* opaque */
    int device;
} kvx_status_token;

kvx_status kvx_status_enqueue(void *stream, kvx_status_token *tok);
kvx_status kvx_status_wait(const kvx_status_token *tok);
kvx_status kvx_status_query(const kvx_status_token *tok, int *ready);

/* Mapped, portable pinned host memory (cudaHostAlloc). Fails with
 * KVX_ERR_NOT_MAPPED if the device address differs from the host address
 * (no unified addressing). Synchronous; not for the hot path. */
kvx_status kvx_host_alloc(size_t bytes, void **out);
kvx_status kvx_host_free(void *ptr);

/* ---- baselines (same validation; not the engine) ------------------------ */

/* The direct path the pages compare against: coalesce descriptors that
 * continue the previous one in both source and destination, then one
 * directional cudaMemcpyAsync per merged range (PegaFlow issue #408,
 * §Relevant implementation, MemcpyBackend). *n_ranges (may be NULL) receives
 * the number of memcpy calls issued. */
kvx_status kvx_copy_batch_memcpy(const uint64_t *src_addrs, const uint64_t *dst_addrs,
                                 const uint64_t *sizes, size_t n, int dir, void *stream,
                                 size_t *n_ranges);

/* One contiguous directional cudaMemcpyAsync: the roofline probe of the host
 * link (PegaFlow issue #408, §Results: contiguous pinned-memory DMA). */
kvx_status kvx_copy_contiguous(uint64_t dst, uint64_t src, uint64_t bytes, int dir,
                               void *stream);

/* ---- a batch copy that allocates nothing -------------------------------- */

/* The pages have no counterpart of this entry point; it exists for callers
 * that cannot allocate memory at copy time. kvx_copy_batch allocates its
 * staging ring lazily (cudaHostAlloc and cudaMalloc on a slot's first use,
 * and again, with a device-synchronising cudaFree, when a bigger batch makes a
 * slot grow). Some callers cannot accept that: a serving engine that reserves
 * almost all HBM for its KV cache at start-up leaves later cudaMalloc calls to
 * fail, and a decode loop with a fixed per-step budget cannot absorb an
 * allocation or a device-wide synchronisation in the middle of a step.
 *
 * kvx_copy_batch_noalloc takes the same arguments and moves the same bytes as
 * kvx_copy_batch, with the same validation and error rules, but makes no CUDA
 * device or pinned-host allocation: no cudaMalloc, cudaFree, cudaHostAlloc or
 * cudaHostRegister of new memory. (Host heap use is not excluded: validation
 * levels 1 and 2 sort a heap copy of the ranges, and the first pack of 32 Ki
 * records or more may start the library's packing threads.) Its chunk
 * table lives in one of two fixed arrays of KVX_NOALLOC_MAX_CHUNKS records
 * (2 MiB each) in the library's own device memory, which every GPU that loads
 * the library holds until the process exits; the records are packed into a
 * fixed host array of the same size and copied with one cudaMemcpyAsync from
 * that array into the two device arrays in turn.
 *   - A batch that needs more than KVX_NOALLOC_MAX_CHUNKS chunks returns
 *     KVX_ERR_CAPACITY and enqueues nothing.
 *   - Not allowed while `stream` is being captured (KVX_ERR_CAPTURE): the
 *     table upload reads the shared host array, which a replayed graph would
 *     read again with whatever another call had packed there since. Capture
 *     kvx_copy_uploaded over a kvx_desc_buf instead.
 *   - The first call on a device looks up the device address of the arrays
 *     (cudaGetSymbolAddress) with that device current, creates three events
 *     and, unless another kvx call did, registers the library's static page
 *     of error flags with the driver (cudaHostRegister of existing memory,
 *     not an allocation). The first call in the process also page-locks the
 *     static host array the same way, so that the upload is one DMA from it;
 *     a later call then waits on the host until the previous call's upload
 *     has completed before it packs the array again. If the array cannot be
 *     page-locked, the upload is a pageable copy, which the runtime stages
 *     before returning.
 *   - Each upload into a device array first waits, on the GPU, for the last
 *     copy that read that array, on whatever stream it ran. When `stream`
 *     still has work queued, a page-locked upload runs on a side stream of
 *     the library (created by the first such call on the device) and
 *     `stream` waits for it, so that it overlaps that work; otherwise it runs
 *     on `stream`. Calls from several host threads are serialised until
 *     their copy is enqueued; calls on one stream or on different streams
 *     are both safe.
 *   - Nothing in the arrays has to start at zero: each call writes every
 *     record its kernel reads, and the header record that holds the work
 *     counter. */
#define KVX_NOALLOC_MAX_CHUNKS 65536u

kvx_status kvx_copy_batch_noalloc(const uint64_t *src_addrs, const uint64_t *dst_addrs,
                                  const uint64_t *sizes, size_t n, int dir, int cta_budget,
                                  void *stream);

/* ---- debug bounds: a kernel-side check of every chunk ------------------- */

/* Most address ranges kvx_debug_bounds takes per device. */
#define KVX_DEBUG_BOUNDS_MAX 64u

/* A debugging aid for callers whose descriptors come from code they do not
 * trust yet (a block manager or router that writes addresses). Register the
 * memory that copies may touch, typically the host and device pools: n ranges
 * [lo[i], hi[i]) for the current device, at most KVX_DEBUG_BOUNDS_MAX; n == 0
 * turns the check off (the initial state). While ranges are registered every
 * copy kernel checks each chunk it is about to move: its source bytes and its
 * destination bytes must each lie inside one registered range. A chunk that
 * does not is skipped (its destination is not written) and the device's
 * error flags report it, so the next kvx_stream_check / kvx_status_wait on the
 * device returns KVX_ERR_DEVICE_FAULT; the other chunks are copied. For a
 * device-resident descriptor list the unit is the whole descriptor. The check
 * never traps and never reads or writes outside the registered ranges on a
 * skipped chunk's behalf. It costs one constant-cache read per chunk record
 * while off, and a scan of the ranges per chunk while on.
 * This call synchronises the device (no copy may be in flight while the table
 * changes) and is not allowed during stream capture. KVX_ERR_INVALID_ARG for
 * null arrays with n > 0, or an empty or reversed range; KVX_ERR_CAPACITY for
 * n > KVX_DEBUG_BOUNDS_MAX. The pages describe no such check: it guards
 * against a descriptor that points outside its pools. */
kvx_status kvx_debug_bounds(const uint64_t *lo, const uint64_t *hi, size_t n);

/* ---- self-test of the bounded device wait ------------------------------- */

/* Launch one CTA that waits on an mbarrier nothing ever completes, with the
 * same bounded wait the bulk kernel uses, limited to timeout_ns (1 ms..10 s).
 * The kernel gives up, sets the timeout flag of the device and returns;
 * a following kvx_stream_check returns KVX_ERR_TIMEOUT. Faults nothing. */
kvx_status kvx_selftest_wait_timeout(uint64_t timeout_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KVX_H */
