/*
 * A C99 client of the kvx C ABI: no Python and no C++, only include/kvx.h,
 * the CUDA runtime for the caller's own device memory and stream, and (as the
 * expected result) the C oracle. It checks that the boundary is usable as a
 * plain C library, the way a serving engine written in C or C++ would call it.
 *
 *   kvx_c_client host   entry points that need no GPU: version, status
 *                        names, validation, the chunk plan of a batch
 *   kvx_c_client copy   on device 0, three hops through the public calls,
 *                        each reading what the hop before wrote:
 *                          H2D  host pool A   -> device pool X  kvx_copy_batch
 *                          D2D  device pool X -> device pool Y  kvx_desc_buf_create,
 *                               kvx_upload_descriptors, kvx_copy_uploaded
 *                          D2H  device pool Y -> host pool B    kvx_copy_batch,
 *                               status through kvx_status_enqueue / kvx_status_wait
 *                        then compares X, Y and B, whole pools with their
 *                        canary, with the oracle applied hop by hop to host
 *                        snapshots of the same inputs.
 *
 * Exit status 0 and a last line starting with "c client ok" on success.
 *
 * The batch copy being checked: one descriptor upload and one copy-kernel
 * launch in place of one memcpy per fragment, moving exactly the bytes a
 * memcpy per descriptor moves (PegaFlow issue #408, §Summary; vLLM PR #42212
 * report, §实现拆解 item 4).
 */
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "kvx.h"

/* The oracle (oracle/kvx_oracle.c, test infrastructure): one memcpy per
 * descriptor on host snapshots addressed by byte offsets. */
void oracle_copy_batch(uint8_t *dst_pool, const uint8_t *src_pool, const uint64_t *src_off,
                       const uint64_t *dst_off, const uint64_t *sizes, size_t n);

#define SLOT 16384u            /* one descriptor per 16 KiB slot */
#define NSLOT 1024u            /* 16 MiB pools */
#define POOL ((size_t)SLOT * NSLOT)
#define NDESC 700u
#define CANARY 0xA5

static int failures = 0;

#define CHECK(cond, ...)                                  \
    do {                                                  \
        if (!(cond)) {                                    \
            fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__); \
            fprintf(stderr, __VA_ARGS__);                 \
            fprintf(stderr, "\n");                        \
            ++failures;                                   \
        }                                                 \
    } while (0)

/* A seeded input generator (splitmix64): pool bytes and descriptor draws. */
static uint64_t rng_state;

static uint64_t next_u64(void)
{
    uint64_t z = (rng_state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static uint64_t below(uint64_t n) { return next_u64() % n; }

/* A hop's descriptors as offsets: n distinct source slots and n distinct
 * destination slots, each start +8 bytes with probability 1/2 (so both phases
 * mod 16 occur), sizes 8 .. 16,376 bytes in steps of 8 that fit their slots. */
static void draw_hop(uint64_t *src_off, uint64_t *dst_off, uint64_t *sizes)
{
    static uint32_t perm_s[NSLOT], perm_d[NSLOT];
    for (uint32_t i = 0; i < NSLOT; ++i) {
        perm_s[i] = i;
        perm_d[i] = i;
    }
    for (uint32_t i = NSLOT - 1; i > 0; --i) {
        uint32_t j = (uint32_t)below(i + 1u), t = perm_s[i];
        perm_s[i] = perm_s[j];
        perm_s[j] = t;
        j = (uint32_t)below(i + 1u);
        t = perm_d[i];
        perm_d[i] = perm_d[j];
        perm_d[j] = t;
    }
    for (uint32_t i = 0; i < NDESC; ++i) {
        const uint64_t so = 8u * below(2), dof = 8u * below(2);
        uint64_t z = 8u * (1u + below(SLOT / 8u - 1u));
        const uint64_t room = SLOT - (so > dof ? so : dof);
        if (z > room)
            z = room;
        src_off[i] = (uint64_t)perm_s[i] * SLOT + so;
        dst_off[i] = (uint64_t)perm_d[i] * SLOT + dof;
        sizes[i] = z;
    }
}

static void add_base(uint64_t *out, const uint64_t *off, const void *base, size_t n)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = (uint64_t)(uintptr_t)base + off[i];
}

/* ---- entry points that need no GPU --------------------------------------- */

static void run_host(void)
{
    static uint64_t so[NDESC], dof[NDESC], z[NDESC], s[NDESC], d[NDESC];
    static kvx_chunk recs[NDESC];
    const char *name;
    size_t n_chunks = 0;
    uint64_t payload = 0, planned = 0;
    int st;

    CHECK(kvx_version() == KVX_VERSION_MAJOR * 100 + KVX_VERSION_MINOR, "version %d", kvx_version());
    for (st = KVX_OK; st <= KVX_ERR_CAPTURE; ++st) {
        name = kvx_status_string(st);
        CHECK(name != NULL && strncmp(name, "KVX_", 4) == 0, "status %d has no name", st);
    }
    CHECK(strcmp(kvx_status_string(99), "KVX_ERR_UNKNOWN") == 0, "unknown status name");

    rng_state = 20261202u;
    draw_hop(so, dof, z);
    add_base(s, so, (const void *)(uintptr_t)(1ull << 32), NDESC);
    add_base(d, dof, (const void *)(uintptr_t)(2ull << 32), NDESC);
    CHECK(kvx_validate(s, d, z, NDESC, KVX_H2D, 0) == KVX_OK, "validate level 0: %s", kvx_last_error());
    CHECK(kvx_validate(s, d, z, NDESC, KVX_D2D, 1) == KVX_OK, "validate level 1: %s", kvx_last_error());
    CHECK(kvx_validate(s, d, z, NDESC, 3, 0) == KVX_ERR_INVALID_ARG, "bad dir accepted");
    z[5] += 4;
    CHECK(kvx_validate(s, d, z, NDESC, KVX_H2D, 0) == KVX_ERR_ALIGN, "size %llu accepted",
          (unsigned long long)z[5]);
    CHECK(kvx_last_error()[0] != '\0', "no message for a failed validation");
    CHECK(kvx_copy_batch(s, d, z, NDESC, KVX_H2D, 0, NULL) == KVX_ERR_ALIGN, "copy_batch accepted a bad size");
    z[5] -= 4;
    d[1] = d[0];  /* two descriptors onto the same destination */
    CHECK(kvx_validate(s, d, z, NDESC, KVX_H2D, 1) == KVX_ERR_OVERLAP, "overlap not found at level 1");
    d[1] = (2ull << 32) + dof[1];
    CHECK(kvx_copy_batch(s, d, z, 0, KVX_H2D, 0, NULL) == KVX_OK, "an empty batch is not a no-op");

    /* every size fits one 16 KiB chunk, so the plan has one record per
       descriptor, covering exactly its bytes */
    CHECK(kvx_plan_chunks(s, d, z, NDESC, NULL, 0, &n_chunks) == KVX_OK && n_chunks == NDESC,
          "plan: %zu chunks for %u descriptors", n_chunks, NDESC);
    CHECK(kvx_plan_chunks(s, d, z, NDESC, recs, NDESC - 1, &n_chunks) == KVX_ERR_CAPACITY,
          "plan: no capacity error");
    CHECK(kvx_plan_chunks(s, d, z, NDESC, recs, NDESC, &n_chunks) == KVX_OK, "plan: %s", kvx_last_error());
    for (size_t i = 0; i < NDESC; ++i) {
        payload += z[i];
        planned += recs[i].len;
        CHECK(recs[i].desc < NDESC && recs[i].src == s[recs[i].desc] && recs[i].dst == d[recs[i].desc] &&
                  recs[i].len == z[recs[i].desc],
              "plan record %zu does not match descriptor %u", i, recs[i].desc);
    }
    CHECK(planned == payload, "plan moves %llu of %llu bytes", (unsigned long long)planned,
          (unsigned long long)payload);
    if (failures == 0)
        printf("c client ok: host entry points (version %d, %zu chunks planned)\n", kvx_version(), n_chunks);
}

/* ---- three hops on device 0 ---------------------------------------------- */

static int cuda_ok(cudaError_t e, const char *what)
{
    if (e != cudaSuccess) {
        fprintf(stderr, "FAIL %s: %s\n", what, cudaGetErrorString(e));
        ++failures;
        return 0;
    }
    return 1;
}

static void compare(const char *name, const uint8_t *got, const uint8_t *want)
{
    for (size_t i = 0; i < POOL; ++i) {
        if (got[i] != want[i]) {
            CHECK(0, "pool %s differs from the oracle at byte %zu (%u, want %u)", name, i, got[i], want[i]);
            return;
        }
    }
}

static void run_copy(void)
{
    static uint64_t so[NDESC], dof[NDESC], z[NDESC], s[NDESC], d[NDESC];
    uint8_t *A = NULL, *B = NULL, *X = NULL, *Y = NULL;
    uint8_t *a = malloc(POOL), *b = malloc(POOL), *x = malloc(POOL), *y = malloc(POOL);
    uint8_t *got = malloc(POOL);
    cudaStream_t st = NULL;
    kvx_desc_buf *buf = NULL;
    kvx_status_token tok;

    if (!a || !b || !x || !y || !got) {
        CHECK(0, "host snapshots: out of memory");
        goto done;
    }
    if (!cuda_ok(cudaSetDevice(0), "cudaSetDevice") ||
        !cuda_ok(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking), "cudaStreamCreate") ||
        !cuda_ok(cudaMalloc((void **)&X, POOL), "cudaMalloc X") ||
        !cuda_ok(cudaMalloc((void **)&Y, POOL), "cudaMalloc Y"))
        goto done;
    CHECK(kvx_host_alloc(POOL, (void **)&A) == KVX_OK && kvx_host_alloc(POOL, (void **)&B) == KVX_OK,
          "kvx_host_alloc: %s", kvx_last_error());
    if (failures)
        goto done;

    rng_state = 20261202u + 7u;
    for (size_t i = 0; i < POOL; i += 8) {
        const uint64_t v = next_u64();
        memcpy(A + i, &v, 8);
    }
    memset(B, CANARY, POOL);
    if (!cuda_ok(cudaMemset(X, CANARY, POOL), "cudaMemset X") ||
        !cuda_ok(cudaMemset(Y, CANARY, POOL), "cudaMemset Y") ||
        !cuda_ok(cudaDeviceSynchronize(), "cudaDeviceSynchronize"))
        goto done;
    memcpy(a, A, POOL);
    memset(b, CANARY, POOL);
    memset(x, CANARY, POOL);
    memset(y, CANARY, POOL);

    /* hop 1: H2D through kvx_copy_batch */
    draw_hop(so, dof, z);
    add_base(s, so, A, NDESC);
    add_base(d, dof, X, NDESC);
    CHECK(kvx_copy_batch(s, d, z, NDESC, KVX_H2D, 0, st) == KVX_OK, "H2D: %s", kvx_last_error());
    oracle_copy_batch(x, a, so, dof, z, NDESC);

    /* hop 2: D2D through a reusable descriptor buffer, copied twice (the second
       copy rewrites the same bytes) */
    draw_hop(so, dof, z);
    add_base(s, so, X, NDESC);
    add_base(d, dof, Y, NDESC);
    CHECK(kvx_desc_buf_create(NDESC, &buf) == KVX_OK, "desc_buf_create: %s", kvx_last_error());
    if (buf) {
        CHECK(kvx_upload_descriptors(buf, s, d, z, NDESC, KVX_D2D, st) == KVX_OK, "upload: %s", kvx_last_error());
        CHECK(kvx_copy_uploaded(buf, 0, st) == KVX_OK, "copy_uploaded: %s", kvx_last_error());
        CHECK(kvx_copy_uploaded(buf, 0, st) == KVX_OK, "copy_uploaded again: %s", kvx_last_error());
    }
    oracle_copy_batch(y, x, so, dof, z, NDESC);

    /* hop 3: D2H through kvx_copy_batch, its status read through a token */
    draw_hop(so, dof, z);
    add_base(s, so, Y, NDESC);
    add_base(d, dof, B, NDESC);
    CHECK(kvx_copy_batch(s, d, z, NDESC, KVX_D2H, 0, st) == KVX_OK, "D2H: %s", kvx_last_error());
    CHECK(kvx_status_enqueue(st, &tok) == KVX_OK, "status_enqueue: %s", kvx_last_error());
    CHECK(kvx_status_wait(&tok) == KVX_OK, "status_wait: %s", kvx_last_error());
    CHECK(kvx_stream_check(st) == KVX_OK, "stream_check: %s", kvx_last_error());
    oracle_copy_batch(b, y, so, dof, z, NDESC);

    compare("B (host)", B, b);
    if (cuda_ok(cudaMemcpy(got, X, POOL, cudaMemcpyDeviceToHost), "read X"))
        compare("X (device)", got, x);
    if (cuda_ok(cudaMemcpy(got, Y, POOL, cudaMemcpyDeviceToHost), "read Y"))
        compare("Y (device)", got, y);
    if (failures == 0)
        printf("c client ok: H2D, D2D (uploaded, twice) and D2H, %u descriptors each, bit-exact against the "
               "oracle\n", NDESC);
done:
    if (buf)
        CHECK(kvx_desc_buf_destroy(buf) == KVX_OK, "desc_buf_destroy: %s", kvx_last_error());
    if (A)
        kvx_host_free(A);
    if (B)
        kvx_host_free(B);
    if (X)
        cudaFree(X);
    if (Y)
        cudaFree(Y);
    if (st)
        cudaStreamDestroy(st);
    free(a);
    free(b);
    free(x);
    free(y);
    free(got);
}

int main(int argc, char **argv)
{
    if (argc != 2 || (strcmp(argv[1], "host") && strcmp(argv[1], "copy"))) {
        fprintf(stderr, "usage: %s host|copy\n", argv[0]);
        return 2;
    }
    if (!strcmp(argv[1], "host"))
        run_host();
    else
        run_copy();
    return failures ? 1 : 0;
}
