/*
 * kvx oracle: the plain CPU definition of a batched descriptor copy.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this file's library.
 * The product path (libkvx.so and its Python binding) never links, imports
 * or calls anything here, and this file includes nothing from the product.
 *
 * What it computes. The pages replace "many directional CUDA memcpy
 * submissions" with one descriptor upload and one copy-kernel launch
 * (PegaFlow issue #408, "Kernel transfer backend causes decode TPOT tail
 * spikes under concurrent KV transfers", §Summary). The replacement must move
 * the same bytes: the vLLM report checks that the kernel "copies the source
 * bytes" (vLLM PR #42212 report, §实现拆解 item 4), and the FreeToken kernel
 * takes "the same arguments and the same bytes" as the kernel it replaces
 * (FreeToken issue #751, §What we changed). So the result has a plain
 * definition: for every descriptor i, the size_i bytes at src_i appear at
 * dst_i, and every other destination byte keeps its value. This file writes
 * that definition out, with no blocking, chunking or reordering.
 *
 * Addresses are given as byte offsets into host snapshot buffers: the caller
 * copies the source pool and the destination pool (with its canary) to host
 * memory, translates each descriptor address to an offset, and compares the
 * whole destination snapshot after this runs.
 *
 * Readings of points the pages leave open (the same readings are listed in
 * the design notes):
 *   - destination ranges of one batch are pairwise disjoint and overlap no
 *     source range of the batch; then the result does not depend on the
 *     order of the descriptors (oracle_ranges_disjoint checks the first part);
 *   - a zero-size descriptor copies nothing; n == 0 is the identity.
 *
 * Pins (tests/test_oracle.py): a pure-Python per-byte brute force over every
 * batch of up to two descriptors in 48-byte pools, sampled three-descriptor
 * batches, the canary / checksum / permutation invariants, published FNV-1a
 * test vectors, per-range checksums against FNV-1a of each slice, and
 * planted mistakes that the pins must catch.
 */
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* The batch definition, one memcpy per descriptor, in descriptor order. */
void oracle_copy_batch(uint8_t *dst_pool, const uint8_t *src_pool,
                       const uint64_t *src_off, const uint64_t *dst_off,
                       const uint64_t *sizes, size_t n)
{
    for (size_t i = 0; i < n; ++i) {
        if (sizes[i] == 0)
            continue;
        memcpy(dst_pool + dst_off[i], src_pool + src_off[i], (size_t)sizes[i]);
    }
}

/*
 * The same definition read per output byte: destination byte j takes the
 * source byte of the descriptor whose destination range holds j, else keeps
 * its value. Quadratic; for the oracle's self-test on tiny pools only.
 */
void oracle_copy_batch_bytewise(uint8_t *dst_pool, size_t dst_pool_bytes,
                                const uint8_t *src_pool,
                                const uint64_t *src_off, const uint64_t *dst_off,
                                const uint64_t *sizes, size_t n)
{
    for (size_t j = 0; j < dst_pool_bytes; ++j) {
        for (size_t i = 0; i < n; ++i) {
            if (j >= dst_off[i] && j < dst_off[i] + sizes[i]) {
                dst_pool[j] = src_pool[src_off[i] + (j - dst_off[i])];
                break;
            }
        }
    }
}

/*
 * 64-bit FNV-1a over len bytes: the per-descriptor checksum used by the
 * invariant "checksum of source range == checksum of destination range".
 * Offset basis 14695981039346656037 and prime 1099511628211 are the published
 * FNV-1a 64-bit parameters.
 */
uint64_t oracle_fnv1a64(const uint8_t *p, size_t len)
{
    uint64_t h = 14695981039346656037ULL;
    for (size_t k = 0; k < len; ++k) {
        h ^= (uint64_t)p[k];
        h *= 1099511628211ULL;
    }
    return h;
}

/* Per-descriptor checksums of n ranges of one pool. */
void oracle_range_checksums(const uint8_t *pool, const uint64_t *off,
                            const uint64_t *sizes, size_t n, uint64_t *out)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = oracle_fnv1a64(pool + off[i], (size_t)sizes[i]);
}

struct oracle_range {
    uint64_t lo, hi;
};

static int range_cmp(const void *a, const void *b)
{
    const struct oracle_range *x = (const struct oracle_range *)a;
    const struct oracle_range *y = (const struct oracle_range *)b;
    if (x->lo < y->lo)
        return -1;
    if (x->lo > y->lo)
        return 1;
    return 0;
}

/*
 * 1 when the non-empty ranges [off_i, off_i + size_i) are pairwise disjoint,
 * 0 when two of them share a byte, -1 when memory runs out. Sort by start,
 * then compare each range with the furthest end seen so far.
 */
int oracle_ranges_disjoint(const uint64_t *off, const uint64_t *sizes, size_t n)
{
    struct oracle_range *r = (struct oracle_range *)malloc((n ? n : 1) * sizeof(*r));
    if (!r)
        return -1;
    size_t m = 0;
    for (size_t i = 0; i < n; ++i) {
        if (sizes[i] == 0)
            continue;
        r[m].lo = off[i];
        r[m].hi = off[i] + sizes[i];
        ++m;
    }
    qsort(r, m, sizeof(*r), range_cmp);
    int ok = 1;
    uint64_t end = 0;
    for (size_t k = 0; k < m; ++k) {
        if (k > 0 && r[k].lo < end) {
            ok = 0;
            break;
        }
        if (r[k].hi > end)
            end = r[k].hi;
    }
    free(r);
    return ok;
}
