// Auto policy: choose DMA or the copy kernel, and the kernel's shape, from the
// observable shape of a transfer.
//
// The pages propose an Auto policy "based on observable transfer shape, such
// as merged range count, total bytes, and average range size", with separate
// throughput-balanced and tail-bounded operating points chosen per device
// (PegaFlow issue #408, §Discussion item 2 and follow-up §Proposed direction;
// the vLLM report's threshold/minimum-count selection is the same idea, vLLM
// PR #42212 report, §实现拆解 item 2). The GB300 measurements behind the rules
// (H2D, host wall clock from submission to completion):
//   - per-range cudaMemcpyAsync costs about 2.6 us of host submission per
//     range, so it loses to the kernel at every fragmented shape measured
//     (4-64 KiB, 16-65,536 descriptors);
//   - with few large ranges it wins: 1 x 256 KiB 10.5 vs 8.0 GB/s, 1 x 4 MiB
//     92 vs 77, 4 x 1 MiB 82 vs 78; it ties at 16 x 4-16 MiB (180-202 vs
//     188-203) and loses at 16 x 1 MiB (122 vs 149) and at 64 ranges. So the
//     throughput policy takes DMA for at most 8 ranges whose mean is at least
//     ranges x 256 KiB;
//   - the copy engines occupy no SM at all, so the tail policy takes DMA
//     whenever it stays near the link peak (at most 16 ranges of 1 MiB mean);
//   - otherwise: the calibrated table's kernel for the batch (throughput:
//     LDG over the host link, LDG or STAGE for D2D by size and phase, or the
//     bulk ring where a KVX_TABLE file has a row for it); the one-warp bulk CTAs at a budget of 4 cost the
//     colocated decode stand-in the least p99 while still sustaining a paced
//     KV burst (tail).
#include <cuda_runtime.h>

#include "kvx_internal.h"

namespace {

constexpr size_t kDmaMaxRangesThroughput = 8;         // DMA ranges, throughput policy
constexpr uint64_t kDmaMeanPerRange = 256ull << 10;    // ... each averaging ranges x 256 KiB
constexpr size_t kDmaMaxRangesTail = 16;               // DMA ranges, tail policy
constexpr uint64_t kDmaMinMeanTail = 1ull << 20;       // ... averaging at least 1 MiB
constexpr int kTailBudget = 4;                         // bulk CTAs of the tail-bounded policy
constexpr int kTailRing = 3;                           // ... each with a 48 KiB ring (a bigger ring
                                                       // takes shared memory a colocated kernel needs)

// Number of ranges after merging descriptors that continue the previous one
// in both source and destination (the direct path's coalescing).
size_t merged_ranges(const uint64_t *src, const uint64_t *dst, const uint64_t *sizes, size_t n,
                     size_t stop_after)
{
    size_t ranges = 0;
    uint64_t end_s = 0, end_d = 0;
    bool open = false;
    for (size_t i = 0; i < n; ++i) {
        if (!sizes[i])
            continue;
        if (!open || src[i] != end_s || dst[i] != end_d) {
            if (++ranges > stop_after)
                return ranges;
            open = true;
        }
        end_s = src[i] + sizes[i];
        end_d = dst[i] + sizes[i];
    }
    return ranges;
}

}  // namespace

extern "C" {

kvx_status kvx_auto_path(const uint64_t *src, const uint64_t *dst, const uint64_t *sizes, size_t n,
                         int dir, int policy, int *path)
{
    if (!path)
        return kvx::set_error(KVX_ERR_INVALID_ARG, "kvx_auto_path: null output");
    if (policy != KVX_POLICY_THROUGHPUT && policy != KVX_POLICY_TAIL)
        return kvx::set_error(KVX_ERR_INVALID_ARG, "kvx_auto_path: policy is not THROUGHPUT or TAIL");
    kvx_status st = kvx_validate(src, dst, sizes, n, dir, 0);
    if (st != KVX_OK)
        return st;
    uint64_t bytes = 0;
    for (size_t i = 0; i < n; ++i)
        bytes += sizes[i];
    const size_t ranges = merged_ranges(src, dst, sizes, n, kDmaMaxRangesTail);
    bool dma = false;
    if (ranges > 0) {
        const uint64_t mean = bytes / ranges;
        if (policy == KVX_POLICY_TAIL)
            dma = ranges <= kDmaMaxRangesTail && mean >= kDmaMinMeanTail;
        else
            dma = ranges <= kDmaMaxRangesThroughput && mean >= ranges * kDmaMeanPerRange;
    }
    if (dma) {
        *path = KVX_PATH_DMA;
    } else if (policy == KVX_POLICY_TAIL) {
        *path = KVX_PATH_KERNEL_BULK;
    } else {
        kvx_launch l{};
        st = kvx_select_launch(src, dst, sizes, n, dir, nullptr, &l);
        if (st != KVX_OK)
            return st;
        *path = l.variant == KVX_VARIANT_BULK    ? KVX_PATH_KERNEL_BULK
                : l.variant == KVX_VARIANT_STAGE ? KVX_PATH_KERNEL_STAGE
                                                 : KVX_PATH_KERNEL_LDG;
    }
    return KVX_OK;
}

kvx_status kvx_copy_batch_auto(const uint64_t *src, const uint64_t *dst, const uint64_t *sizes, size_t n,
                               int dir, int policy, void *stream, int *path_out)
{
    int path = 0;
    kvx_status st = kvx_auto_path(src, dst, sizes, n, dir, policy, &path);
    if (st != KVX_OK)
        return st;
    if (path_out)
        *path_out = path;
    if (path == KVX_PATH_DMA)
        return kvx_copy_batch_memcpy(src, dst, sizes, n, dir, stream, nullptr);
    if (policy == KVX_POLICY_TAIL) {
        kvx_launch l{};
        l.variant = KVX_VARIANT_BULK;
        l.cta_budget = kTailBudget;
        l.stages = kTailRing;
        return kvx_copy_batch_ex(src, dst, sizes, n, dir, &l, stream);
    }
    return kvx_copy_batch_ex(src, dst, sizes, n, dir, nullptr, stream);  // the table's launch, as reported
}

}  // extern "C"
