// Tail-bounded submission: a transfer split into pieces that are submitted one
// at a time, each only after the previous piece has completed.
//
// The pages measured that cutting a burst into smaller enqueue-only launches
// does nothing for a colocated decode's tail; what bounds the tail is real
// completion backpressure: submit one piece, record and query its event,
// yield while it is incomplete, then submit the next. Because the transfer
// backend must not block, that progress belongs in the transfer worker as an
// event-driven state machine (PegaFlow issue #408, follow-up §2 and
// §Proposed direction: `chunk_descriptors` with event-based completion).
// kvx_transfer is that state machine, built on the public batch-copy ABI.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "kvx_internal.h"

struct kvx_transfer {
    std::vector<uint64_t> src, dst, sizes;  // the transfer's own copy of the descriptors
    size_t n = 0, next = 0, piece = 0;
    int dir = KVX_H2D;
    kvx_launch launch{};
    bool has_launch = false;
    cudaStream_t stream = nullptr;
    cudaEvent_t done_ev = nullptr;
    bool in_flight = false;
    int device = 0;
    mutable std::mutex mu;  // start, poll and progress from several threads take turns
};

namespace {

kvx_status submit_piece(kvx_transfer *t)
{
    const size_t k = std::min(t->piece, t->n - t->next);
    kvx_status st = kvx_copy_batch_ex(t->src.data() + t->next, t->dst.data() + t->next,
                                      t->sizes.data() + t->next, k, t->dir,
                                      t->has_launch ? &t->launch : nullptr, t->stream);
    if (st != KVX_OK)
        return st;
    if (cudaEventRecord(t->done_ev, t->stream) != cudaSuccess)
        return kvx::set_error(KVX_ERR_CUDA, "kvx_transfer: cudaEventRecord failed");
    t->next += k;
    t->in_flight = true;
    return KVX_OK;
}

}  // namespace

extern "C" {

kvx_status kvx_transfer_create(kvx_transfer **out)
{
    if (!out)
        return kvx::set_error(KVX_ERR_INVALID_ARG, "kvx_transfer_create: null output");
    *out = nullptr;
    kvx_transfer *t = new (std::nothrow) kvx_transfer;
    if (!t)
        return kvx::set_error(KVX_ERR_CAPACITY, "kvx_transfer_create: out of host memory");
    if (!kvx::handle_add(t, kvx::kHandleTransfer)) {
        delete t;
        return kvx::set_error(KVX_ERR_CAPACITY, "kvx_transfer_create: out of host memory");
    }
    *out = t;
    return KVX_OK;
}

kvx_status kvx_transfer_start(kvx_transfer *t, const uint64_t *src, const uint64_t *dst,
                              const uint64_t *sizes, size_t n, int dir, size_t chunk_descriptors,
                              const kvx_launch *launch, void *stream)
{
    if (!t)
        return kvx::set_error(KVX_ERR_INVALID_ARG, "kvx_transfer_start: null transfer");
    if (!kvx::handle_live(t, kvx::kHandleTransfer))
        return kvx::set_error(KVX_ERR_INVALID_ARG, "kvx_transfer_start: not a live transfer");
    std::lock_guard<std::mutex> g(t->mu);
    if (t->in_flight)
        return kvx::set_error(KVX_ERR_INVALID_ARG,
                              "kvx_transfer_start: a piece of the previous transfer is still in flight");
    kvx_status st = kvx_validate(src, dst, sizes, n, dir, kvx_get_validate_level());
    if (st != KVX_OK)
        return st;
    // Nothing of the previous transfer is in flight: start from an empty one,
    // so that a failure below leaves a transfer with nothing to submit.
    t->n = 0;
    t->next = 0;
    if (n == 0)
        return KVX_OK;
    try {
        t->src.assign(src, src + n);
        t->dst.assign(dst, dst + n);
        t->sizes.assign(sizes, sizes + n);
    } catch (const std::bad_alloc &) {
        return kvx::set_error(KVX_ERR_CAPACITY, "kvx_transfer_start: out of host memory for the descriptors");
    }
    if (!t->done_ev) {
        if (cudaGetDevice(&t->device) != cudaSuccess ||
            cudaEventCreateWithFlags(&t->done_ev, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            t->done_ev = nullptr;
            return kvx::set_error(KVX_ERR_CUDA, "kvx_transfer_start: cannot create its event");
        }
    }
    t->n = n;
    t->piece = chunk_descriptors ? chunk_descriptors : n;
    t->dir = dir;
    t->has_launch = launch != nullptr;
    if (launch)
        t->launch = *launch;
    t->stream = static_cast<cudaStream_t>(stream);
    return submit_piece(t);
}

kvx_status kvx_transfer_poll(kvx_transfer *t, int *done)
{
    if (!t || !done)
        return kvx::set_error(KVX_ERR_INVALID_ARG, "kvx_transfer_poll: null argument");
    if (!kvx::handle_live(t, kvx::kHandleTransfer))
        return kvx::set_error(KVX_ERR_INVALID_ARG, "kvx_transfer_poll: not a live transfer");
    std::lock_guard<std::mutex> g(t->mu);
    *done = 0;
    if (t->in_flight) {
        const cudaError_t e = cudaEventQuery(t->done_ev);
        if (e == cudaErrorNotReady) {
            cudaGetLastError();  // not sticky
            return KVX_OK;
        }
        if (e != cudaSuccess)
            return kvx::set_error(KVX_ERR_CUDA, "kvx_transfer_poll: cudaEventQuery failed");
        t->in_flight = false;
    }
    if (t->next < t->n)
        return submit_piece(t);
    *done = 1;
    return KVX_OK;
}

kvx_status kvx_transfer_progress(const kvx_transfer *t, size_t *submitted, size_t *total)
{
    if (!t)
        return kvx::set_error(KVX_ERR_INVALID_ARG, "kvx_transfer_progress: null transfer");
    if (!kvx::handle_live(t, kvx::kHandleTransfer))
        return kvx::set_error(KVX_ERR_INVALID_ARG, "kvx_transfer_progress: not a live transfer");
    std::lock_guard<std::mutex> g(t->mu);
    if (submitted)
        *submitted = t->next;
    if (total)
        *total = t->n;
    return KVX_OK;
}

kvx_status kvx_transfer_destroy(kvx_transfer *t)
{
    if (!t)
        return KVX_OK;
    if (!kvx::handle_remove(t, kvx::kHandleTransfer))
        return kvx::set_error(KVX_ERR_INVALID_ARG, "kvx_transfer_destroy: not a live transfer");
    if (t->in_flight)
        cudaEventSynchronize(t->done_ev);
    if (t->done_ev)
        cudaEventDestroy(t->done_ev);
    delete t;
    return KVX_OK;
}

}  // extern "C"
