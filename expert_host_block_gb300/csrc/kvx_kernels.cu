// Copy kernels of kvx for sm_103a.
//
// The variants walk the same table of 32-byte chunk records ({src, dst,
// len <= 16 KiB, desc}, after a header record) as a persistent grid: work
// unit u goes to worker (u mod workers), where a worker is a warp (LDG, whose
// units are warp passes of at most 512 * U bytes; STAGE, whose units are 4 KiB
// passes) or a CTA (BULK, whose units are chunks). Units are small and of nearly equal size, so handing them out
// round-robin spreads the batch's bytes evenly over the workers, whatever mix
// of descriptor sizes it holds (FreeToken issue #751, §Problem in upstream
// today and §What we changed: split the call's bytes, not its banks, over the
// CTAs). Over the host link, where equal bytes do not take equal time, the
// LDG kernel can instead hand units out from a counter (see the LDG variant).
//
// LDG variant: every lane moves 16-byte words, `U` loads in flight per lane
// before the matching stores (the pages' LDG kernel keeps one 16-byte load in
// flight per thread; FreeToken issue #751, §Problem in upstream today). By
// position, a warp reads the records of its next 32 chunks with one load per
// lane and passes them around with shuffles, so no lane waits on a record
// load per chunk; from the counter, lane 0 fetches the next unit's record
// while the current one copies.
//
// BULK variant: one warp per CTA; lane 0 streams chunks through a ring of
// shared::cta stages with cp.async.bulk loads completed on an mbarrier, then
// cp.async.bulk stores (FreeToken issue #751, §What we changed: a 3-stage
// ring of 16 KiB, one issuing thread per CTA, the .shared::cta destination
// form). Here a stage is as large as the batch's longest chunk, so a ring of
// 4 KiB chunks has many more stages, and loads, in flight than one of 16 KiB
// chunks. Every mbarrier wait is bounded by %globaltimer.
//
// STAGE variant: every warp has its own ring of 4 KiB stages; lane 0 bulk-loads
// the 16-byte blocks holding each unit, the whole warp stores the unit with
// 16-byte stores at the destination's phase. Loads in flight cost shared
// memory instead of registers, which pays off when phases differ.
//
// Unaligned pieces: addresses and sizes are multiples of 8. When src and dst
// have the same phase mod 16, a chunk is an 8-byte head, a 16-byte-word body
// and an 8-byte tail; otherwise aligned 16-byte source words are re-paired
// across neighbouring lanes into aligned 16-byte destination words.
//
// Back to back on a stream (programmatic dependent launch): every copy kernel
// is launched with programmatic stream serialisation and lets the grid after
// it launch as soon as all of its own CTAs are running, so the launch of the
// next batch overlaps this one instead of following its completion. A copy
// kernel reads only its chunk table before it waits for the grid before it
// (griddepcontrol.wait: that grid has completed and its writes are visible);
// a table is written by the host or by a copy on the stream, never by a
// kernel, so the only thing read early is already final. Payload, the
// dynamic-assignment counter and device-list plans are touched only after the
// wait. A grid launched without the attribute returns from the wait at once.
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "kvx_internal.h"

namespace kvx {

namespace {

// Device errors: one flag word per kind (kDevErr* bit b -> word b) in mapped
// pinned host memory, set by a plain store. The host reads and clears the
// words once the stream or event it waits for has completed, so no atomic
// and no extra kernel is needed to report them.
__device__ __forceinline__ void report(unsigned *err, unsigned kind)
{
    *reinterpret_cast<volatile unsigned *>(err + (__ffs(kind) - 1)) = 1u;
}

constexpr unsigned kFull = 0xffffffffu;

// ---- programmatic dependent launch ---------------------------------------------

// Allow the grid launched after this one on the stream to start (it then runs
// only up to its own pdl_wait until this grid completes).
__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the grids this one depends on have completed and their memory
// operations are visible to this grid.
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Ask for [p, p + bytes) to be brought into L2 (p and bytes multiples of 16).
// A hint: it returns no data and needs no completion. Issued before pdl_wait it
// reads nothing stale, because the L2 is where every write to device memory
// lands: a write of the grid before this one updates the line after the
// prefetch brought it in.
__device__ __forceinline__ void prefetch_l2(uint64_t p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---- debug pool bounds -------------------------------------------------------
//
// While ranges are registered (kvx_debug_bounds), every chunk record a copy
// kernel loads is checked: its source bytes and its destination bytes must each
// lie inside one registered range, else the chunk is skipped and kDevErrBounds
// raised. With none registered the check is one read of the constant cache.

__constant__ uint32_t c_bounds_n;
__constant__ uint64_t c_bounds[2 * KVX_DEBUG_BOUNDS_MAX];  // lo, hi of range i at 2i, 2i + 1

__device__ __forceinline__ bool in_bounds(uint64_t a, uint64_t len)
{
    for (uint32_t i = 0; i < c_bounds_n; ++i)
        if (a >= c_bounds[2 * i] && a + len <= c_bounds[2 * i + 1] && a + len >= a)
            return true;
    return false;
}

// ---- global memory access (inline PTX) ----------------------------------

__device__ __forceinline__ uint4 ld16(const unsigned char *p)
{
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint2 ld8(const unsigned char *p)
{
    uint2 v;
    asm volatile("ld.global.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p));
    return v;
}

template <int P>
__device__ __forceinline__ void st16(unsigned char *p, uint4 v)
{
    if constexpr (P == 1)
        asm volatile("st.global.wt.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
    else if constexpr (P == 2)
        asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
    else
        asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
}

template <int P>
__device__ __forceinline__ void st8(unsigned char *p, uint2 v)
{
    if constexpr (P == 1)
        asm volatile("st.global.wt.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
    else if constexpr (P == 2)
        asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
    else
        asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// ---- one warp pass over part of a chunk --------------------------------------
//
// A pass moves up to 512 * U bytes of one chunk: U 16-byte words per lane.
// Pass k of a chunk covers body words [k * 32U, (k + 1) * 32U); pass 0 also
// moves the 8-byte head (and, for matching phases, the tail). All loads of a
// pass are issued before any of its stores, so a lane has U loads (plus at
// most one edge word) in flight.

template <int U>
struct PassBytes {
    static constexpr uint32_t value = 512u * U;
};

// M, the instance (kvx::kPhase*): kPhaseRepair takes the phase-matched path
// below for chunks whose src and dst agree mod 16 and re-pairs 16-byte words
// across lanes for the others (118 registers a thread at U = 8);
// kPhaseMatched is called only for chunks that agree, so the re-pairing path
// is left out (84 registers); kPhaseShift copies every chunk with one path
// (copy_pass_shift, 79 registers).
template <int U, int P, int M>
__device__ __forceinline__ void copy_pass_shift(uint64_t s, uint64_t d, uint32_t len, uint32_t k,
                                                uint32_t lane);

template <int U, int P, int M = kPhaseRepair>
__device__ __forceinline__ void copy_pass(uint64_t s, uint64_t d, uint32_t len, uint32_t k,
                                          uint32_t lane)
{
    if constexpr (M == kPhaseShift) {
        copy_pass_shift<U, P, M>(s, d, len, k, lane);
    } else if (M == kPhaseMatched || ((s ^ d) & 15u) == 0) {
        const uint32_t head = (s & 15u) ? 8u : 0u;  // len >= 8 whenever head != 0
        const uint64_t bs = s + head, bd = d + head;
        const uint32_t blen = len - head;
        const uint32_t n16 = blen >> 4;
        // the edge words of pass 0: lane 0 the head, lane 1 the tail
        bool edge = false;
        uint64_t es = 0, ed = 0;
        if (k == 0) {
            if (lane == 0 && head) {
                edge = true;
                es = s;
                ed = d;
            } else if (lane == 1 && (blen & 15u)) {
                edge = true;
                es = bs + ((uint64_t)n16 << 4);
                ed = bd + ((uint64_t)n16 << 4);
            }
        }
        uint2 e = {0, 0};
        if (edge)
            e = ld8(reinterpret_cast<const unsigned char *>(es));
        const unsigned char *S = reinterpret_cast<const unsigned char *>(bs);
        unsigned char *D = reinterpret_cast<unsigned char *>(bd);
        const uint32_t i0 = k * 32u * U;
        uint4 r[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const uint32_t idx = i0 + 32u * j + lane;
            if (idx < n16)
                r[j] = ld16(S + ((uint64_t)idx << 4));
        }
        if (edge)
            st8<P>(reinterpret_cast<unsigned char *>(ed), e);
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const uint32_t idx = i0 + 32u * j + lane;
            if (idx < n16)
                st16<P>(D + ((uint64_t)idx << 4), r[j]);
        }
    } else if constexpr (M == kPhaseRepair) {
        // Source and destination differ in phase mod 16 (one of them is 8 mod
        // 16). If the source is the 16-aligned one, its first 8 bytes go out as
        // a head word; after that the source is 8 mod 16 and the destination is
        // 16-aligned. Destination word j is then the high half of the aligned
        // source word V[j] and the low half of V[j + 1], where V[0] starts 8
        // bytes before the (remaining) source range. Each V[j] read lies in a
        // 16-byte block that holds source bytes, so no load leaves the pages of
        // the source range; its out-of-range half is never stored.
        bool edge = false;
        uint2 e = {0, 0};
        const uint64_t hd = d;
        if ((s & 15u) == 0) {
            if (k == 0 && lane == 0) {
                edge = true;
                e = ld8(reinterpret_cast<const unsigned char *>(s));
            }
            s += 8;
            d += 8;
            len -= 8;
        }
        const unsigned char *V = reinterpret_cast<const unsigned char *>(s - 8);
        unsigned char *D = reinterpret_cast<unsigned char *>(d);
        const uint32_t n16 = len >> 4;
        const bool tail = (len & 15u) != 0;
        const uint32_t nv = (n16 || tail) ? n16 + 1 : 0;  // source words V[0 .. nv)
        const uint32_t i0 = k * 32u * U;
        uint4 r[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const uint32_t idx = i0 + 32u * j + lane;
            if (idx < nv)
                r[j] = ld16(V + ((uint64_t)idx << 4));
        }
        uint2 x = {0, 0};  // lane 31: the low half of the word after this pass
        const uint32_t ix = i0 + 32u * U;
        if (lane == 31 && ix < nv) {
            const uint4 t = ld16(V + ((uint64_t)ix << 4));
            x = make_uint2(t.x, t.y);
        }
        if (edge)
            st8<P>(reinterpret_cast<unsigned char *>(hd), e);
#pragma unroll
        for (int j = 0; j < U; ++j) {
            uint32_t nx = __shfl_down_sync(kFull, r[j].x, 1);
            uint32_t ny = __shfl_down_sync(kFull, r[j].y, 1);
            if (j + 1 < U) {
                const uint32_t fx = __shfl_sync(kFull, r[j + 1 < U ? j + 1 : j].x, 0);
                const uint32_t fy = __shfl_sync(kFull, r[j + 1 < U ? j + 1 : j].y, 0);
                if (lane == 31) {
                    nx = fx;
                    ny = fy;
                }
            } else if (lane == 31) {
                nx = x.x;
                ny = x.y;
            }
            const uint32_t idx = i0 + 32u * j + lane;
            if (idx < n16)
                st16<P>(D + ((uint64_t)idx << 4), make_uint4(r[j].z, r[j].w, nx, ny));
            else if (idx == n16 && tail)
                st8<P>(D + ((uint64_t)idx << 4), make_uint2(r[j].z, r[j].w));
        }
    }
}

// Every chunk in the destination's frame: an 8-byte head when the destination
// is 8 mod 16, aligned 16-byte destination words, an 8-byte tail. The aligned
// 16-byte source words V[j] start `sh` bytes (0 or 8, the same for the whole
// warp) before the source bytes of destination word j: with sh = 0 word j is
// V[j], with sh = 8 it is the high half of V[j] and the low half of V[j + 1]
// (re-paired across neighbouring lanes). One path for both phases needs no
// more registers than the phase-matched instance; its grid is larger (it
// fits 6 CTAs of 128 threads per SM, the re-pairing instance 4).
template <int U, int P, int M>
__device__ __forceinline__ void copy_pass_shift(uint64_t s, uint64_t d, uint32_t len, uint32_t k,
                                                uint32_t lane)
{
    const uint32_t head = (d & 15u) ? 8u : 0u;  // len >= 8 whenever head != 0
    const uint64_t bs = s + head;
    const uint32_t sh = (uint32_t)(bs & 15u);   // 0 or 8
    const uint32_t blen = len - head;
    const uint32_t n16 = blen >> 4;              // whole destination words
    const bool tail = (blen & 15u) != 0;         // then 8 bytes
    // source words V[0 .. nv): with sh = 8 one more than the destination words
    // (the low half of the last one, and the tail's high half)
    const uint32_t nv = n16 + (((sh || tail) && (n16 || tail)) ? 1u : 0u);
    // Each V[j] lies in a 16-byte block that holds source bytes, so no load
    // leaves the pages of the source range; bytes outside it are never stored.
    const unsigned char *V = reinterpret_cast<const unsigned char *>(bs - sh);
    unsigned char *D = reinterpret_cast<unsigned char *>(d + head);
    const bool edge = k == 0 && lane == 0 && head;  // the head word, pass 0
    uint2 e = {0, 0};
    if (edge)
        e = ld8(reinterpret_cast<const unsigned char *>(s));
    const uint32_t i0 = k * 32u * U;
    uint4 r[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
        const uint32_t idx = i0 + 32u * j + lane;
        if (idx < nv)
            r[j] = ld16(V + ((uint64_t)idx << 4));
    }
    uint2 x = {0, 0};  // sh = 8, lane 31: the low half of the word after this pass
    const uint32_t ix = i0 + 32u * U;
    if (sh && lane == 31 && ix < nv) {
        const uint4 t = ld16(V + ((uint64_t)ix << 4));
        x = make_uint2(t.x, t.y);
    }
    if (edge)
        st8<P>(reinterpret_cast<unsigned char *>(d), e);
#pragma unroll
    for (int j = 0; j < U; ++j) {
        uint32_t nx = 0, ny = 0;
        if (sh) {  // the same for every lane
            nx = __shfl_down_sync(kFull, r[j].x, 1);
            ny = __shfl_down_sync(kFull, r[j].y, 1);
            if (j + 1 < U) {
                const uint32_t fx = __shfl_sync(kFull, r[j + 1 < U ? j + 1 : j].x, 0);
                const uint32_t fy = __shfl_sync(kFull, r[j + 1 < U ? j + 1 : j].y, 0);
                if (lane == 31) {
                    nx = fx;
                    ny = fy;
                }
            } else if (lane == 31) {
                nx = x.x;
                ny = x.y;
            }
        }
        const uint32_t idx = i0 + 32u * j + lane;
        if (idx < n16)
            st16<P>(D + ((uint64_t)idx << 4), sh ? make_uint4(r[j].z, r[j].w, nx, ny) : r[j]);
        else if (idx == n16 && tail)
            st8<P>(D + ((uint64_t)idx << 4), sh ? make_uint2(r[j].z, r[j].w) : make_uint2(r[j].x, r[j].y));
    }
}

// A whole chunk by one warp, pass after pass.
template <int U, int P>
__device__ __forceinline__ void copy_chunk_warp(uint64_t s, uint64_t d, uint32_t len,
                                                uint32_t lane)
{
    for (uint32_t k = 0; k * PassBytes<U>::value < len; ++k)
        copy_pass<U, P>(s, d, len, k, lane);
}

// A chunk record held in one lane's registers.
struct Rec {
    uint64_t s, d;
    uint32_t l;
};

__device__ __forceinline__ Rec load_rec(const kvx_chunk *__restrict__ tab, uint64_t c, unsigned *err)
{
    const uint4 *p = reinterpret_cast<const uint4 *>(tab + c);
    const uint4 a = __ldg(p);
    const uint4 b = __ldg(p + 1);
    Rec r;
    r.s = (uint64_t)a.x | ((uint64_t)a.y << 32);
    r.d = (uint64_t)a.z | ((uint64_t)a.w << 32);
    r.l = b.x;
    if (r.l > KVX_CHUNK_BYTES) {  // never produced by the host planner
        report(err, kDevErrBadRecord);
        r.l = 0;
    }
    if (c_bounds_n && r.l && !(in_bounds(r.s, r.l) && in_bounds(r.d, r.l))) {
        report(err, kDevErrBounds);
        r.l = 0;
    }
    return r;
}

__device__ __forceinline__ Rec shfl_rec(const Rec &r, int src_lane)
{
    Rec o;
    o.s = __shfl_sync(kFull, r.s, src_lane);
    o.d = __shfl_sync(kFull, r.d, src_lane);
    o.l = __shfl_sync(kFull, r.l, src_lane);
    return o;
}

// ---- LDG variant -----------------------------------------------------------

// Work units are warp passes in pass-major order: unit u is pass
// u / n_chunks of chunk u % n_chunks, for `passes` passes per chunk (enough for
// the batch's longest chunk). For a batch of chunks that fit one pass every
// unit is a whole chunk.
//
// Static assignment (ctr == nullptr): unit u goes to warp u mod (warps in the
// grid). Whatever the mix of chunk lengths, no warp ends with more than one
// pass more than another. A warp reads the records of its next 32 units with
// one load per lane and hands them around with shuffles.
//
// Dynamic assignment (ctr != nullptr): warp w copies unit w first, then takes
// one unit at a time from the counter ctr[0]. Over the host link the warps are
// not served equally fast: by position, the first warps of a KV-burst launch
// were done after 60 % of the launch and the last ones set its length. Taking
// units from a counter, every warp stays busy to within about one unit of the
// end. Lane 0 keeps the pipeline: while unit k is copied, the record of unit
// k+1 and the index of unit k+2 are already on their way, so neither latency
// adds to the copy. The last warp to finish (counted in ctr[1]) zeroes both
// words for the next launch over the same table.
// A launch for phase-matched batches (M) copies only chunks whose src and dst
// agree mod 16; the host decides M from the same descriptors it packs, so a
// mismatched record means a bad table: reported and skipped, never copied with
// misaligned 16-byte accesses.
template <int M>
__device__ __forceinline__ bool phase_ok(const Rec &c, uint32_t lane, unsigned *err)
{
    if (M != kPhaseMatched || ((c.s ^ c.d) & 15u) == 0)
        return true;
    if (lane == 0)
        report(err, kDevErrBadRecord);
    return false;
}

__device__ __forceinline__ Rec unit_rec(const kvx_chunk *__restrict__ tab, uint64_t u, uint32_t n_chunks,
                                        uint32_t pass_bytes, uint32_t *pass_out, unsigned *err)
{
    const uint64_t pass = u / n_chunks;
    Rec r = load_rec(tab, u - pass * n_chunks, err);
    if (pass * pass_bytes >= r.l)
        r.l = 0;  // this chunk has no such pass
    *pass_out = (uint32_t)pass;
    return r;
}

// Static assignment with kLdgPrefetch (D2D batches small enough for their
// sources to sit in L2 beside the previous batch's writes): before the wait,
// every lane asks L2 for the source bytes of the unit whose record it holds,
// so a batch launched early fetches its first data while the one before it
// drains (4,096 x 8 KiB back to back: 0.83 -> 0.90 of HBM).
template <int U, int P, int M>
__global__ void __launch_bounds__(512) kvx_copy_ldg_kernel(const kvx_chunk *__restrict__ tab,
                                                            uint32_t n_chunks, uint32_t passes,
                                                            unsigned long long *ctr, unsigned *err,
                                                            uint32_t flags)
{
    pdl_trigger();
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t wpb = blockDim.x >> 5;
    const uint64_t gwarp = (uint64_t)blockIdx.x * wpb + (threadIdx.x >> 5);
    const uint64_t nwarps = (uint64_t)gridDim.x * wpb;
    const uint64_t n_units = (uint64_t)n_chunks * passes;
    if (ctr == nullptr) {
        bool waited = false;  // the first 32 records load before the wait
        for (uint64_t base = gwarp; base < n_units; base += 32u * nwarps) {
            const uint64_t mine = base + (uint64_t)lane * nwarps;
            Rec r = {0, 0, 0};
            uint32_t k = 0;
            if (mine < n_units)
                r = unit_rec(tab, mine, n_chunks, PassBytes<U>::value, &k, err);
            const int cnt = __popc(__ballot_sync(kFull, mine < n_units));
            if (!waited) {
                if ((flags & kLdgPrefetch) && r.l) {
                    // the 16-byte blocks holding this unit's pass (no byte outside them)
                    const uint64_t lo = (r.s + (uint64_t)k * PassBytes<U>::value) & ~15ull;
                    uint64_t hi = r.s + (uint64_t)(k + 1) * PassBytes<U>::value + 16u;
                    if (hi > r.s + r.l)
                        hi = r.s + r.l;
                    prefetch_l2(lo, (uint32_t)(((hi + 15u) & ~15ull) - lo));
                }
                pdl_wait();
                waited = true;
            }
            for (int j = 0; j < cnt; ++j) {
                const Rec c = shfl_rec(r, j);
                const uint32_t kk = __shfl_sync(kFull, k, j);
                if (c.l && phase_ok<M>(c, lane, err))
                    copy_pass<U, P, M>(c.s, c.d, c.l, kk, lane);
            }
        }
        return;
    }
    // lane 0: rc / kc = record and pass of the current unit, nx = the next unit
    uint64_t cur = gwarp;
    unsigned long long nx = 0;
    Rec rc = {0, 0, 0};
    uint32_t kc = 0;
    if (lane == 0 && cur < n_units)
        rc = unit_rec(tab, cur, n_chunks, PassBytes<U>::value, &kc, err);
    // the previous copy over this table zeroes the counter as it ends
    pdl_wait();
    if (lane == 0)
        nx = nwarps + atomicAdd(&ctr[0], 1ull);
    while (cur < n_units) {
        unsigned long long nn = 0;
        Rec rn = {0, 0, 0};
        uint32_t kn = 0;
        if (lane == 0) {
            nn = nwarps + atomicAdd(&ctr[0], 1ull);
            if (nx < n_units)
                rn = unit_rec(tab, nx, n_chunks, PassBytes<U>::value, &kn, err);
        }
        const Rec c = shfl_rec(rc, 0);
        const uint32_t kk = __shfl_sync(kFull, kc, 0);
        if (c.l && phase_ok<M>(c, lane, err))
            copy_pass<U, P, M>(c.s, c.d, c.l, kk, lane);
        cur = __shfl_sync(kFull, nx, 0);
        nx = nn;
        rc = rn;
        kc = kn;
    }
    if (lane == 0) {
        __threadfence();  // this warp's counter updates before its count of done warps
        if (atomicAdd(&ctr[1], 1ull) == nwarps - 1) {
            atomicExch(&ctr[0], 0ull);
            atomicExch(&ctr[1], 0ull);
        }
    }
}

// ---- BULK variant ----------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of the mbarrier to complete, giving up after
// limit_ns of %globaltimer (or 2^28 polls, whichever comes first). The timer
// is read only once a poll has failed: a phase that has already completed
// costs one try_wait.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 0; it < (1u << 28); ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 31u) == 31u && globaltimer() - t0 > limit_ns)
            return false;
    }
    return false;
}

__device__ __forceinline__ void bulk_load(uint32_t dst_smem, uint64_t src, uint32_t bytes,
                                          uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst_smem),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void bulk_store(uint64_t dst, uint32_t src_smem, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(src_smem), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// wait_group.read takes an immediate: dispatch a runtime count in 0..31.
__device__ __noinline__ void bulk_wait_read_n(uint32_t n)
{
#define KVX_WAIT_CASE(i) \
    case i: bulk_wait_read<i>(); return;
    switch (n) {
        KVX_WAIT_CASE(0) KVX_WAIT_CASE(1) KVX_WAIT_CASE(2) KVX_WAIT_CASE(3) KVX_WAIT_CASE(4)
        KVX_WAIT_CASE(5) KVX_WAIT_CASE(6) KVX_WAIT_CASE(7) KVX_WAIT_CASE(8) KVX_WAIT_CASE(9)
        KVX_WAIT_CASE(10) KVX_WAIT_CASE(11) KVX_WAIT_CASE(12) KVX_WAIT_CASE(13) KVX_WAIT_CASE(14)
        KVX_WAIT_CASE(15) KVX_WAIT_CASE(16) KVX_WAIT_CASE(17) KVX_WAIT_CASE(18) KVX_WAIT_CASE(19)
        KVX_WAIT_CASE(20) KVX_WAIT_CASE(21) KVX_WAIT_CASE(22) KVX_WAIT_CASE(23) KVX_WAIT_CASE(24)
        KVX_WAIT_CASE(25) KVX_WAIT_CASE(26) KVX_WAIT_CASE(27) KVX_WAIT_CASE(28) KVX_WAIT_CASE(29)
        KVX_WAIT_CASE(30)
    default: bulk_wait_read<31>(); return;
    }
#undef KVX_WAIT_CASE
}

__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ bool bulk_ok(const Rec &r)
{
    return r.l != 0 && ((r.s | r.d | (uint64_t)r.l) & 15u) == 0;
}

constexpr int kBulkMaxStages = 32;

// The ring is `S` stages of `stage` bytes (the batch's longest chunk rounded
// up to 16 bytes). A bulk store's shared-memory read counts as done only once
// its writes are accepted, so a stage cannot be refilled right after its
// store is issued without waiting a full write latency. The ring is therefore
// split: loads run D = S/2 chunks ahead of the chunk being stored, and up to
// S - D stores stay in flight behind it. Every iteration commits exactly one
// bulk group (a store, or an empty group for a chunk moved by the warp), so
// "the store of the chunk that last used stage s" is always the group S - D
// commits back.
__global__ void __launch_bounds__(32) kvx_copy_bulk_kernel(const kvx_chunk *__restrict__ tab,
                                                           uint32_t n_chunks, uint32_t stage,
                                                           uint32_t S, uint64_t wait_ns, unsigned *err)
{
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t bars[kBulkMaxStages];
    // The record window: chunks [a0, a0 + 64) in slots c & 63. The issuing lane
    // reads records from here; the warp fills it 32 records at a time.
    __shared__ uint64_t w_src[64], w_dst[64];
    __shared__ uint32_t w_len[64];
    const uint32_t lane = threadIdx.x;
    const uint32_t ring0 = smem_u32(ring);
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t D = S / 2;  // loads ahead, >= 1 because S >= 2

    pdl_trigger();
    if (lane == 0) {
        for (uint32_t s = 0; s < S; ++s)
            mbar_init(bar0 + 8u * s, 1);
        mbar_init_fence();
    }

    // Chunks of this CTA: blockIdx.x + k * gridDim.x, k in [0, my_n).
    const uint64_t my_n =
        n_chunks > blockIdx.x ? (n_chunks - 1ull - blockIdx.x) / gridDim.x + 1ull : 0ull;
    // Load records [k0, k0 + 32) into the window; return the batch's bulk-eligibility bits.
    auto load_batch = [&](uint64_t k0) {
        Rec r = {0, 0, 0};
        if (k0 + lane < my_n)
            r = load_rec(tab, (uint64_t)blockIdx.x + (k0 + lane) * gridDim.x, err);
        const uint32_t slot = (uint32_t)((k0 + lane) & 63u);
        w_src[slot] = r.s;
        w_dst[slot] = r.d;
        w_len[slot] = r.l;
        return __ballot_sync(kFull, bulk_ok(r));
    };
    uint64_t a0 = 0;
    uint32_t mask_a = load_batch(0);   // chunks [a0, a0 + 32)
    uint32_t mask_b = load_batch(32);  // chunks [a0 + 32, a0 + 64); the look-ahead k + D < a0 + 64
    __syncwarp();
    pdl_wait();  // records only before this point
    auto eligible = [&](uint64_t c) {
        const uint64_t o = c - a0;
        return ((o < 32u ? mask_a >> o : mask_b >> (o - 32u)) & 1u) != 0;
    };

    uint32_t phase = 0;    // bit s: parity of the next completion of stage s
    uint32_t pending = 0;  // bit s: a load is in flight on stage s
    bool timed_out = false;

    for (uint32_t j = 0; j < D && j < my_n; ++j) {  // prologue: D loads ahead
        if (eligible(j)) {
            if (lane == 0) {
                mbar_arrive_expect_tx(bar0 + 8u * j, w_len[j & 63u]);
                bulk_load(ring0 + j * stage, w_src[j & 63u], w_len[j & 63u], bar0 + 8u * j);
            }
            pending |= 1u << j;
        }
    }

    uint32_t st = 0;      // stage of chunk k: k mod S
    uint32_t sj = D % S;  // stage of chunk k + D
    for (uint64_t k = 0; k < my_n; ++k) {
        if (k == a0 + 32) {  // slide the window: records [a0 + 64, a0 + 96) replace [a0, a0 + 32)
            __syncwarp();
            mask_a = mask_b;
            mask_b = load_batch(a0 + 64);
            a0 += 32;
            __syncwarp();
        }
        const uint32_t slot = (uint32_t)(k & 63u);
        if (eligible(k)) {
            // Lane 0 waits; the outcome is broadcast so the warp stays converged.
            bool ok = true;
            if (lane == 0)
                ok = mbar_wait_bounded(bar0 + 8u * st, (phase >> st) & 1u, wait_ns);
            if (!__shfl_sync(kFull, (int)ok, 0)) {
                timed_out = true;
                break;
            }
            phase ^= 1u << st;
            pending &= ~(1u << st);
            if (lane == 0)
                bulk_store(w_dst[slot], ring0 + st * stage, w_len[slot]);
        } else {
            copy_chunk_warp<4, 0>(w_src[slot], w_dst[slot], w_len[slot], lane);
        }
        if (lane == 0)
            bulk_commit();  // one group per iteration, empty for a warp-moved chunk
        const uint64_t j = k + D;
        if (j < my_n && eligible(j)) {
            // Stage sj last held chunk j - S, whose group is S - D commits back.
            if (lane == 0) {
                const uint32_t js = (uint32_t)(j & 63u);
                bulk_wait_read_n(S - D);
                mbar_arrive_expect_tx(bar0 + 8u * sj, w_len[js]);
                bulk_load(ring0 + sj * stage, w_src[js], w_len[js], bar0 + 8u * sj);
            }
            pending |= 1u << sj;
        }
        st = st + 1 == S ? 0 : st + 1;
        sj = sj + 1 == S ? 0 : sj + 1;
    }

    if (timed_out) {
        if (lane == 0)
            report(err, kDevErrTimeout);
        // Let the loads still in flight land before the shared memory goes away.
        if (lane == 0)
            for (uint32_t s = 0; s < S; ++s)
                if (pending & (1u << s))
                    mbar_wait_bounded(bar0 + 8u * s, (phase >> s) & 1u, wait_ns);
    }
    if (lane == 0)
        bulk_wait_all();
    __syncwarp();
}

// ---- STAGE variant ----------------------------------------------------------
//
// For batches whose chunks' sources and destinations do not agree mod 16 the
// LDG kernel must re-pair 16-byte words across lanes, which costs registers
// (118 a thread: 16 warps per SM) and therefore bytes in flight. Here one lane
// of each warp bulk-loads the 16-byte blocks holding a unit (cp.async.bulk into
// shared::cta, completed on an mbarrier) into a ring of S stages of its own,
// and the whole warp stores the unit from there with 16-byte st.global, reading
// shared memory at whatever 8-byte phase the destination needs. No register
// holds a load in flight, so a warp keeps S units (S x 4 KiB) in flight with
// ~45 registers. Units are warp passes of at most kStageUnit bytes, handed out
// by position as in the LDG kernel; waits are bounded as in the BULK kernel.

constexpr uint32_t kStageUnit = 4096;             // payload bytes per unit
constexpr uint32_t kStageBytes = kStageUnit + 32; // a unit's 16-byte blocks fit in kStageUnit + 16
constexpr int kStageWarps = 4;                    // warps per CTA (128 threads)

// One unit: its source, destination and length (0: the chunk has no such pass).
struct URec {
    uint64_t s, d;
    uint32_t l;
};

__device__ __forceinline__ URec stage_unit(const kvx_chunk *__restrict__ tab, uint64_t u, uint32_t n_chunks,
                                           unsigned *err)
{
    const uint64_t pass = u / n_chunks;
    const Rec r = load_rec(tab, u - pass * n_chunks, err);
    URec o{0, 0, 0};
    const uint64_t off = pass * kStageUnit;
    if (off < r.l) {
        o.s = r.s + off;
        o.d = r.d + off;
        o.l = (uint32_t)(r.l - off < kStageUnit ? r.l - off : kStageUnit);
    }
    return o;
}

__device__ __forceinline__ URec shfl_unit(const URec &r, int src_lane)
{
    URec o;
    o.s = __shfl_sync(kFull, r.s, src_lane);
    o.d = __shfl_sync(kFull, r.d, src_lane);
    o.l = __shfl_sync(kFull, r.l, src_lane);
    return o;
}

__device__ __forceinline__ uint2 lds8(uint32_t a)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

__device__ __forceinline__ uint4 lds16(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

// Order this thread's earlier shared-memory accesses before later bulk copies
// (the async proxy) that write the same shared memory.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Store unit `u` from the stage at shared address `st`, whose byte 0 is the
// global byte (u.s & ~15). Lane 0 writes the 8-byte head that brings the
// destination to 16-byte alignment, all lanes the 16-byte body words, lane 1
// the 8-byte tail.
template <int P>
__device__ __forceinline__ void stage_store(const URec &u, uint32_t st, uint32_t lane)
{
    const uint32_t o = (uint32_t)(u.s & 15u);   // 0 or 8: where the unit's first byte sits in the stage
    const uint32_t hd = (u.d & 15u) ? 8u : 0u;  // len >= 8 whenever hd != 0
    if (hd && lane == 0)
        st8<P>(reinterpret_cast<unsigned char *>(u.d), lds8(st + o));
    const uint32_t ob = o + hd;
    const uint64_t db = u.d + hd;
    const uint32_t blen = u.l - hd;
    const uint32_t nb = blen >> 4;
    if (ob & 15u) {
        for (uint32_t j = lane; j < nb; j += 32u) {
            const uint2 a = lds8(st + ob + 16u * j), b = lds8(st + ob + 16u * j + 8u);
            st16<P>(reinterpret_cast<unsigned char *>(db + 16ull * j), make_uint4(a.x, a.y, b.x, b.y));
        }
    } else {
        for (uint32_t j = lane; j < nb; j += 32u)
            st16<P>(reinterpret_cast<unsigned char *>(db + 16ull * j), lds16(st + ob + 16u * j));
    }
    if ((blen & 15u) && lane == 1)
        st8<P>(reinterpret_cast<unsigned char *>(db + 16ull * nb), lds8(st + ob + 16u * nb));
}

// Warp w copies its units k = 0, 1, ... (unit w + k x warps): lane 0 keeps the
// loads of units k + 1 .. k + S - 1 in flight while the warp stores unit k. The
// records of the warp's units [a0, a0 + 64) sit in two registers per lane (unit
// a0 + i in lane i of wa, a0 + 32 + i of wb), loaded 32 at a time; the
// look-ahead k + S stays below a0 + 64 because S <= 32.
template <int S, int P>
__global__ void __launch_bounds__(kStageWarps * 32) kvx_copy_stage_kernel(const kvx_chunk *__restrict__ tab,
                                                                         uint32_t n_chunks, uint32_t passes,
                                                                         uint64_t wait_ns, unsigned *err)
{
    static_assert(S >= 2 && S <= 32, "stages per warp");
    extern __shared__ __align__(128) unsigned char stage_ring[];
    __shared__ __align__(8) uint64_t bars[kStageWarps][S];
    pdl_trigger();
    const uint32_t lane = threadIdx.x & 31u, wib = threadIdx.x >> 5;
    const uint32_t ring0 = smem_u32(stage_ring) + wib * (uint32_t)S * kStageBytes;
    const uint32_t bar0 = smem_u32(&bars[wib][0]);
    if (lane == 0) {
        for (int s = 0; s < S; ++s)
            mbar_init(bar0 + 8u * s, 1);
        mbar_init_fence();
    }
    __syncwarp();
    const uint64_t gwarp = (uint64_t)blockIdx.x * kStageWarps + wib;
    const uint64_t nwarps = (uint64_t)gridDim.x * kStageWarps;
    const uint64_t n_units = (uint64_t)n_chunks * passes;
    const uint64_t my_n = n_units > gwarp ? (n_units - 1 - gwarp) / nwarps + 1 : 0;
    auto rec_k = [&](uint64_t k) {
        URec r{0, 0, 0};
        if (k < my_n)
            r = stage_unit(tab, gwarp + k * nwarps, n_chunks, err);
        return r;
    };
    uint64_t a0 = 0;
    URec wa = rec_k(lane), wb = rec_k(32u + lane);
    pdl_wait();  // records only before this point
    auto get = [&](uint64_t k) {  // the warp's unit k, k in [a0, a0 + 64); every lane takes part
        const uint64_t o = k - a0;
        const URec x = shfl_unit(wa, (int)(o & 31u)), y = shfl_unit(wb, (int)(o & 31u));
        return o < 32u ? x : y;
    };
    auto issue = [&](const URec &u, uint32_t s) {  // lane 0: load the 16-byte blocks holding u into stage s
        const uint64_t lo = u.s & ~15ull;
        const uint32_t bytes = (uint32_t)(((u.s + u.l + 15u) & ~15ull) - lo);  // <= kStageUnit + 16
        mbar_arrive_expect_tx(bar0 + 8u * s, bytes);
        bulk_load(ring0 + s * kStageBytes, lo, bytes, bar0 + 8u * s);
    };
    uint32_t phase = 0;    // bit s: parity of the next completion of stage s
    uint32_t pending = 0;  // bit s: a load is in flight on stage s
    bool timed_out = false;
    for (uint32_t j = 0; j < (uint32_t)S && j < my_n; ++j) {
        const URec u = get(j);
        if (u.l) {
            if (lane == 0)
                issue(u, j);
            pending |= 1u << j;
        }
    }
    uint32_t st = 0;  // stage of unit k: k mod S
    for (uint64_t k = 0; k < my_n; ++k) {
        if (k == a0 + 32) {
            wa = wb;
            wb = rec_k(a0 + 64 + lane);
            a0 += 32;
        }
        const URec u = get(k);
        if (u.l) {
            bool ok = true;
            if (lane == 0)
                ok = mbar_wait_bounded(bar0 + 8u * st, (phase >> st) & 1u, wait_ns);
            if (!__shfl_sync(kFull, (int)ok, 0)) {
                timed_out = true;
                break;
            }
            phase ^= 1u << st;
            pending &= ~(1u << st);
            stage_store<P>(u, ring0 + st * kStageBytes, lane);
        }
        const uint64_t kn = k + S;
        const URec un = kn < my_n ? get(kn) : URec{0, 0, 0};
        __syncwarp();  // every lane has read stage st
        if (un.l) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(un, st);
            }
            pending |= 1u << st;
        }
        st = st + 1 == (uint32_t)S ? 0 : st + 1;
    }
    if (timed_out && lane == 0) {
        report(err, kDevErrTimeout);
        // let the loads still in flight land before the shared memory goes away
        for (int s = 0; s < S; ++s)
            if (pending & (1u << s))
                mbar_wait_bounded(bar0 + 8u * s, (phase >> s) & 1u, wait_ns);
    }
    __syncwarp();
}

// ---- descriptors that live on the device -------------------------------------
//
// A producer kernel (a MoE router, a block manager on the GPU) writes the
// descriptor arrays and their count in device memory; the host never sees
// them, so the copy is two fixed-shape launches that can be captured in a
// CUDA graph (FreeToken issue #751, §What we changed: the miss count is read
// on the device, so the launch is fixed-shape and capturable). The plan
// kernel validates the list and writes the exclusive scan of chunk counts;
// the copy kernel maps each warp pass to (descriptor, chunk) by binary search
// over that scan.

// The plan, in tiles of kListTile descriptors so that many CTAs share it: the
// tile kernel validates each tile's descriptors, counts their chunks and
// writes each descriptor's chunk offset within the tile, with the tile's
// chunk total, longest chunk and error bits; the base kernel scans the tile
// totals into tile bases and writes the plan results. (One CTA scanning the
// whole list took ~1 us per 1,024 descriptors: 76 us for 65,536.)

// CTA b plans tiles b, b + gridDim.x, ... (kListTile threads). For a list of
// one tile at most (`meta` not null, one CTA) it also writes the plan results
// itself, and the base kernel is not launched.
__global__ void __launch_bounds__(kListTile) kvx_devlist_tile_kernel(
    const uint64_t *__restrict__ src, const uint64_t *__restrict__ dst,
    const uint64_t *__restrict__ sizes, const uint32_t *__restrict__ count, uint32_t max_n,
    uint64_t *__restrict__ offsets, uint64_t *__restrict__ tile_sum, uint32_t *__restrict__ tile_aux,
    DevListMeta *__restrict__ meta, unsigned *err)
{
    constexpr uint32_t kWarps = kListTile / 32;
    __shared__ uint64_t warp_sums[kWarps];
    __shared__ uint32_t warp_aux[kWarps];
    // the list may come from the kernel before this one, and the copy before
    // may still read this list's plan
    pdl_trigger();
    pdl_wait();
    const uint32_t tid = threadIdx.x, lane = tid & 31u, wid = tid >> 5;
    uint32_t n = *count;
    if (n > max_n) {
        if (blockIdx.x == 0 && tid == 0)
            report(err, kDevErrCount);
        n = max_n;
    }
    const uint32_t tiles = (n + kListTile - 1) / kListTile;
    for (uint32_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const uint32_t i = t * kListTile + tid;
        uint64_t c = 0;
        uint32_t m = 0, bad = 0;  // longest chunk, error bits
        if (i < n) {
            const uint64_t z = sizes[i];
            if (z) {
                const uint64_t a = src[i], b = dst[i];
                if (((a | b | z) & 7u) || !a || !b || a + z < a || b + z < b || z > (1ull << 40)) {
                    bad = 1u;  // skipped: contributes no chunks
                } else if (c_bounds_n && !(in_bounds(a, z) && in_bounds(b, z))) {
                    bad = 2u;  // outside the debug bounds: skipped too
                } else {
                    c = z / KVX_CHUNK_BYTES + (z % KVX_CHUNK_BYTES != 0);
                    m = (uint32_t)(z < KVX_CHUNK_BYTES ? z : KVX_CHUNK_BYTES);
                }
            }
        }
        uint64_t x = c;  // inclusive scan within the warp; max and OR across it
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(kFull, x, o);
            if (lane >= (uint32_t)o)
                x += y;
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            m = max(m, __shfl_xor_sync(kFull, m, o));
            bad |= __shfl_xor_sync(kFull, bad, o);
        }
        if (lane == 31)
            warp_sums[wid] = x;
        if (lane == 0)
            warp_aux[wid] = m | (bad << 16);
        __syncthreads();
        uint64_t before = 0, tot = 0;
        uint32_t aux = 0;
#pragma unroll
        for (uint32_t w = 0; w < kWarps; ++w) {
            const uint64_t ws = warp_sums[w];
            before += w < wid ? ws : 0;
            tot += ws;
            const uint32_t wa = warp_aux[w];
            aux = max(aux & 0xffffu, wa & 0xffffu) | ((aux | wa) & ~0xffffu);
        }
        if (i < n)
            offsets[i] = before + x - c;
        if (tid == 0) {
            tile_sum[t] = meta ? 0 : tot;  // a single tile's base is 0
            tile_aux[t] = aux;
            if (meta) {
                meta->total = tot;
                if ((aux >> 16) & 1u)
                    report(err, kDevErrBadDesc);
                if ((aux >> 16) & 2u)
                    report(err, kDevErrBounds);
            }
        }
        __syncthreads();  // warp_sums and warp_aux serve the next tile
    }
    if (meta && tid == 0) {
        if (tiles == 0)
            meta->total = 0;
        meta->n = n;
        meta->max_chunk = tiles ? tile_aux[0] & 0xffffu : 0u;
        meta->next = 0;
        meta->tiles = tiles;
    }
}

// One CTA: the tile totals into tile bases (an exclusive scan, in place), and
// the plan results the copy kernel reads.
__global__ void __launch_bounds__(1024) kvx_devlist_base_kernel(
    const uint32_t *__restrict__ count, uint32_t max_n, DevListMeta *__restrict__ meta,
    uint64_t *__restrict__ tile_base, const uint32_t *__restrict__ tile_aux, unsigned *err)
{
    __shared__ uint64_t warp_sums[32];
    __shared__ uint64_t s_carry;
    __shared__ uint32_t s_max, s_bad;
    pdl_trigger();
    pdl_wait();  // the tile kernel's results
    const uint32_t tid = threadIdx.x, lane = tid & 31u, wid = tid >> 5;
    const uint32_t nwarps = blockDim.x >> 5;
    uint32_t n = *count;
    if (n > max_n)
        n = max_n;
    const uint32_t tiles = (n + kListTile - 1) / kListTile;
    if (tid == 0) {
        s_carry = 0;
        s_max = 0;
        s_bad = 0;
    }
    __syncthreads();
    for (uint32_t base = 0; base < tiles; base += blockDim.x) {
        const uint32_t t = base + tid;
        uint64_t c = 0;
        if (t < tiles) {
            c = tile_base[t];  // the tile's chunk total, until it is replaced by its base below
            const uint32_t aux = tile_aux[t];
            atomicMax(&s_max, aux & 0xffffu);
            atomicOr(&s_bad, aux >> 16);
        }
        uint64_t x = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(kFull, x, o);
            if (lane >= (uint32_t)o)
                x += y;
        }
        if (lane == 31)
            warp_sums[wid] = x;
        __syncthreads();
        if (wid == 0) {  // scan of the warp totals
            uint64_t w = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint64_t y = __shfl_up_sync(kFull, w, o);
                if (lane >= (uint32_t)o)
                    w += y;
            }
            if (lane < nwarps)
                warp_sums[lane] = w;
        }
        __syncthreads();
        if (t < tiles)
            tile_base[t] = s_carry + (wid ? warp_sums[wid - 1] : 0) + x - c;
        __syncthreads();
        if (tid == 0)
            s_carry += warp_sums[nwarps - 1];
        __syncthreads();
    }
    if (tid == 0) {
        meta->total = s_carry;
        meta->n = n;
        meta->max_chunk = s_max;
        meta->next = 0;
        meta->tiles = tiles;
        if (s_bad & 1u)
            report(err, kDevErrBadDesc);
        if (s_bad & 2u)
            report(err, kDevErrBounds);
    }
}

constexpr uint32_t kSmemTiles = 4096;  // tile bases searched in shared memory (lists of up to 1 Mi descriptors)

// The record of unit u of a device list: pass u / total of chunk c = u % total.
// The tile holding c is the last one whose base is at most c (a tile without
// chunks shares its base with the next one, so "last" skips it); within it,
// the descriptor is the last one whose base + offset is at most c (likewise
// past descriptors without chunks). Tile bases are searched in shared memory
// (or global memory for more than kSmemTiles tiles), offsets within the tile
// in global memory: at most log2(kListTile) = 8 dependent loads.
__device__ __forceinline__ Rec devlist_rec(uint64_t u, uint64_t total, uint32_t n, uint32_t tiles, uint32_t unit,
                                           const uint64_t *s_tb, bool in_smem,
                                           const uint64_t *__restrict__ tile_base,
                                           const uint64_t *__restrict__ offsets,
                                           const uint64_t *__restrict__ src, const uint64_t *__restrict__ dst,
                                           const uint64_t *__restrict__ sizes, uint32_t *pass_out)
{
    const uint64_t pass = u / total;
    const uint64_t c = u - pass * total;
    uint32_t lo = 0, hi = tiles;
    while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) >> 1;
        const uint64_t o = in_smem ? s_tb[mid] : __ldg(tile_base + mid);
        if (o <= c)
            lo = mid;
        else
            hi = mid;
    }
    const uint64_t b = in_smem ? s_tb[lo] : __ldg(tile_base + lo);
    uint32_t dlo = lo * kListTile, dhi = dlo + kListTile;
    if (dhi > n)
        dhi = n;
    while (dhi - dlo > 1) {
        const uint32_t mid = (dlo + dhi) >> 1;
        if (b + __ldg(offsets + mid) <= c)
            dlo = mid;
        else
            dhi = mid;
    }
    const uint64_t j = c - b - __ldg(offsets + dlo);
    const uint64_t z = sizes[dlo], off = j * KVX_CHUNK_BYTES;
    Rec r;
    r.s = src[dlo] + off;
    r.d = dst[dlo] + off;
    // off < z always holds for a plan of these arrays; a plan left by another
    // list's copy (scratch used by two copies at once) copies nothing here
    // instead of running past the descriptor
    r.l = off < z ? (uint32_t)(z - off < KVX_CHUNK_BYTES ? z - off : KVX_CHUNK_BYTES) : 0u;
    if (pass * unit >= r.l)
        r.l = 0;
    *pass_out = (uint32_t)pass;
    return r;
}

// Units by position, or (dynamic, with at least kDynamicMinUnitsPerWarp units
// a warp) warp w takes unit w and then one unit at a time from meta->next,
// with the next unit's record on its way while the current one copies, as in
// the LDG kernel. The plan kernel zeroes the counter before every copy, so a
// replayed graph needs no reset.
template <int U, int P>
__global__ void __launch_bounds__(512) kvx_copy_devlist_kernel(
    const uint64_t *__restrict__ src, const uint64_t *__restrict__ dst,
    const uint64_t *__restrict__ sizes, DevListMeta *__restrict__ meta,
    const uint64_t *__restrict__ offsets, const uint64_t *__restrict__ tile_base, bool dynamic)
{
    __shared__ uint64_t s_tb[kSmemTiles];
    pdl_trigger();
    pdl_wait();  // the plan kernels' results
    const uint64_t total = meta->total;
    const uint32_t n = meta->n, tiles = meta->tiles;
    if (total == 0)
        return;
    const bool in_smem = tiles <= kSmemTiles;
    if (in_smem) {
        for (uint32_t i = threadIdx.x; i < tiles; i += blockDim.x)
            s_tb[i] = tile_base[i];
        __syncthreads();
    }
    const uint32_t unit = PassBytes<U>::value;
    const uint32_t passes = meta->max_chunk ? (meta->max_chunk + unit - 1) / unit : 1u;
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t wpb = blockDim.x >> 5;
    const uint64_t gwarp = (uint64_t)blockIdx.x * wpb + (threadIdx.x >> 5);
    const uint64_t nwarps = (uint64_t)gridDim.x * wpb;
    const uint64_t n_units = total * passes;
    if (!dynamic || n_units < kDynamicMinUnitsPerWarp * nwarps) {
        for (uint64_t base = gwarp; base < n_units; base += 32u * nwarps) {
            const uint64_t mine = base + (uint64_t)lane * nwarps;
            Rec r = {0, 0, 0};
            uint32_t k = 0;
            if (mine < n_units)
                r = devlist_rec(mine, total, n, tiles, unit, s_tb, in_smem, tile_base, offsets, src, dst, sizes, &k);
            const int cnt = __popc(__ballot_sync(kFull, mine < n_units));
            for (int jj = 0; jj < cnt; ++jj) {
                const Rec cc = shfl_rec(r, jj);
                const uint32_t kk = __shfl_sync(kFull, k, jj);
                if (cc.l)
                    copy_pass<U, P, kPhaseShift>(cc.s, cc.d, cc.l, kk, lane);
            }
        }
        return;
    }
    unsigned long long *ctr = &meta->next;
    uint64_t cur = gwarp;
    unsigned long long nx = 0;
    Rec rc = {0, 0, 0};
    uint32_t kc = 0;
    if (lane == 0) {
        nx = nwarps + atomicAdd(ctr, 1ull);
        if (cur < n_units)
            rc = devlist_rec(cur, total, n, tiles, unit, s_tb, in_smem, tile_base, offsets, src, dst, sizes, &kc);
    }
    while (cur < n_units) {
        unsigned long long nn = 0;
        Rec rn = {0, 0, 0};
        uint32_t kn = 0;
        if (lane == 0) {
            nn = nwarps + atomicAdd(ctr, 1ull);
            if (nx < n_units)
                rn = devlist_rec(nx, total, n, tiles, unit, s_tb, in_smem, tile_base, offsets, src, dst, sizes, &kn);
        }
        const Rec c = shfl_rec(rc, 0);
        const uint32_t kk = __shfl_sync(kFull, kc, 0);
        if (c.l)
            copy_pass<U, P, kPhaseShift>(c.s, c.d, c.l, kk, lane);
        cur = __shfl_sync(kFull, nx, 0);
        nx = nn;
        rc = rn;
        kc = kn;
    }
}

// ---- the bounded-wait self-test -------------------------------------------

__global__ void kvx_wait_selftest_kernel(uint64_t timeout_ns, unsigned *err)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        mbar_init_fence();
    }
    __syncwarp();
    // Nothing arrives on the barrier, so phase 0 never completes.
    if (threadIdx.x == 0 && !mbar_wait_bounded(b, 0, timeout_ns))
        report(err, kDevErrTimeout);
    __syncwarp();
}

// Launch a kernel on `s`, with programmatic stream serialisation when `pdl`.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(bool pdl, void (*kernel)(KArgs...), int ctas, int threads, size_t smem, cudaStream_t s,
                     Args &&...args)
{
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 1u : 0u;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <int U, int P>
cudaError_t launch_ldg(bool pdl, int ctas, int threads, const kvx_chunk *t, uint32_t n, uint32_t passes,
                       unsigned long long *ctr, int phase, unsigned *err, uint32_t flags, cudaStream_t s)
{
    if (phase == kPhaseMatched)
        return launch_k(pdl, kvx_copy_ldg_kernel<U, P, kPhaseMatched>, ctas, threads, 0, s, t, n, passes, ctr, err,
                        flags);
    if (phase == kPhaseShift)
        return launch_k(pdl, kvx_copy_ldg_kernel<U, P, kPhaseShift>, ctas, threads, 0, s, t, n, passes, ctr, err,
                        flags);
    return launch_k(pdl, kvx_copy_ldg_kernel<U, P, kPhaseRepair>, ctas, threads, 0, s, t, n, passes, ctr, err, flags);
}

template <int U>
cudaError_t launch_ldg_p(const Launch &l, int ctas, const kvx_chunk *t, uint32_t n,
                         uint32_t passes, unsigned long long *ctr, unsigned *err, cudaStream_t s)
{
    const uint32_t flags = (l.prefetch && ctr == nullptr) ? kLdgPrefetch : 0u;
    const int ph = l.matched ? kPhaseMatched : l.shift ? kPhaseShift : kPhaseRepair;
    switch (l.store_policy) {
    case 1: return launch_ldg<U, 1>(l.pdl, ctas, l.threads, t, n, passes, ctr, ph, err, flags, s);
    case 2: return launch_ldg<U, 2>(l.pdl, ctas, l.threads, t, n, passes, ctr, ph, err, flags, s);
    default: return launch_ldg<U, 0>(l.pdl, ctas, l.threads, t, n, passes, ctr, ph, err, flags, s);
    }
}

cudaError_t launch_bulk(bool pdl, int ctas, int ring_units, const kvx_chunk *t, uint32_t n, uint32_t max_chunk_len,
                        unsigned *err, cudaStream_t s)
{
    const uint32_t ring = (uint32_t)bulk_smem_bytes(ring_units);
    uint32_t stage = (max_chunk_len + 15u) & ~15u;
    if (stage < 16u)
        stage = 16u;
    uint32_t S = ring / stage;
    if (S > (uint32_t)kBulkMaxStages)
        S = kBulkMaxStages;
    cudaError_t e = cudaFuncSetAttribute(kvx_copy_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)ring);
    if (e != cudaSuccess)
        return e;
    return launch_k(pdl, kvx_copy_bulk_kernel, ctas, 32, ring, s, t, n, stage, S, kBulkWaitNs, err);
}

template <int S, int P>
cudaError_t launch_stage_sp(bool pdl, int ctas, const kvx_chunk *t, uint32_t n, uint32_t passes, unsigned *err,
                            cudaStream_t s)
{
    const size_t smem = (size_t)kStageWarps * S * kStageBytes;
    cudaError_t e = cudaFuncSetAttribute(kvx_copy_stage_kernel<S, P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    return launch_k(pdl, kvx_copy_stage_kernel<S, P>, ctas, kStageWarps * 32, smem, s, t, n, passes, kBulkWaitNs,
                    err);
}

template <int S>
cudaError_t launch_stage_s(const Launch &l, int ctas, const kvx_chunk *t, uint32_t n, uint32_t passes, unsigned *err,
                           cudaStream_t s)
{
    switch (l.store_policy) {
    case 1: return launch_stage_sp<S, 1>(l.pdl, ctas, t, n, passes, err, s);
    case 2: return launch_stage_sp<S, 2>(l.pdl, ctas, t, n, passes, err, s);
    default: return launch_stage_sp<S, 0>(l.pdl, ctas, t, n, passes, err, s);
    }
}

template <int U>
cudaError_t launch_devlist_p(const Launch &l, const uint64_t *src, const uint64_t *dst,
                            const uint64_t *sizes, DevListMeta *meta, const uint64_t *offsets,
                            const uint64_t *tile_base, bool dyn, cudaStream_t s)
{
    switch (l.store_policy) {
    case 1:
        return launch_k(l.pdl, kvx_copy_devlist_kernel<U, 1>, l.ctas, l.threads, 0, s, src, dst, sizes, meta,
                        offsets, tile_base, dyn);
    case 2:
        return launch_k(l.pdl, kvx_copy_devlist_kernel<U, 2>, l.ctas, l.threads, 0, s, src, dst, sizes, meta,
                        offsets, tile_base, dyn);
    default:
        return launch_k(l.pdl, kvx_copy_devlist_kernel<U, 0>, l.ctas, l.threads, 0, s, src, dst, sizes, meta,
                        offsets, tile_base, dyn);
    }
}

}  // namespace

size_t bulk_smem_bytes(int stages) { return (size_t)stages * KVX_CHUNK_BYTES; }

uint32_t stage_passes(uint32_t max_chunk_len)
{
    const uint32_t p = (max_chunk_len + kStageUnit - 1) / kStageUnit;
    return p ? p : 1u;
}

uint32_t ldg_passes(const Launch &l, uint32_t max_chunk_len)
{
    const uint32_t unit = 512u * (uint32_t)l.unroll;
    const uint32_t p = (max_chunk_len + unit - 1) / unit;
    return p ? p : 1u;
}

// A counter pays off only when every warp has many units to balance; with a
// few units a warp (1,024 x 4 KiB over 512 warps: 2) the positional split,
// with its 32-record batches, is faster (146 against 141 GB/s).
bool ldg_dynamic(const Launch &l, uint32_t n_chunks, uint32_t max_chunk_len)
{
    if (l.variant != KVX_VARIANT_LDG || l.assign != KVX_ASSIGN_DYNAMIC)
        return false;
    const uint64_t warps = (uint64_t)work_ctas(l, n_chunks, max_chunk_len) * (uint64_t)(l.threads / 32);
    return (uint64_t)n_chunks * ldg_passes(l, max_chunk_len) >= kDynamicMinUnitsPerWarp * warps;
}

int work_ctas(const Launch &l, uint32_t n_chunks, uint32_t max_chunk_len)
{
    uint64_t need;
    if (l.variant == KVX_VARIANT_BULK) {
        need = n_chunks;
    } else if (l.variant == KVX_VARIANT_STAGE) {
        need = ((uint64_t)n_chunks * stage_passes(max_chunk_len) + kStageWarps - 1) / kStageWarps;
    } else {
        const uint64_t units = (uint64_t)n_chunks * ldg_passes(l, max_chunk_len);
        need = (units + (uint64_t)(l.threads / 32) - 1) / (uint64_t)(l.threads / 32);
    }
    if (need < 1)
        need = 1;
    return (int)((uint64_t)l.ctas < need ? (uint64_t)l.ctas : need);
}

cudaError_t launch_copy(const Launch &l, kvx_chunk *table, uint32_t n_chunks,
                        uint32_t max_chunk_len, unsigned *err, cudaStream_t stream)
{
    if (n_chunks == 0)
        return cudaSuccess;
    const int ctas = work_ctas(l, n_chunks, max_chunk_len);
    const kvx_chunk *recs = table + kTableHeader;
    if (l.variant == KVX_VARIANT_BULK) {
        return launch_bulk(l.pdl, ctas, l.stages, recs, n_chunks, max_chunk_len, err, stream);
    }
    if (l.variant == KVX_VARIANT_STAGE) {
        const uint32_t passes = stage_passes(max_chunk_len);
        switch (l.stages) {
        case 2: return launch_stage_s<2>(l, ctas, recs, n_chunks, passes, err, stream);
        case 8: return launch_stage_s<8>(l, ctas, recs, n_chunks, passes, err, stream);
        default: return launch_stage_s<4>(l, ctas, recs, n_chunks, passes, err, stream);
        }
    }
    const uint32_t passes = ldg_passes(l, max_chunk_len);
    unsigned long long *ctr =
        ldg_dynamic(l, n_chunks, max_chunk_len) ? reinterpret_cast<unsigned long long *>(table) : nullptr;
    switch (l.unroll) {
    case 2: return launch_ldg_p<2>(l, ctas, recs, n_chunks, passes, ctr, err, stream);
    case 4: return launch_ldg_p<4>(l, ctas, recs, n_chunks, passes, ctr, err, stream);
    default: return launch_ldg_p<8>(l, ctas, recs, n_chunks, passes, ctr, err, stream);
    }
}

cudaError_t launch_devlist(const Launch &l, const uint64_t *src, const uint64_t *dst,
                           const uint64_t *sizes, const uint32_t *count, uint32_t max_n,
                           DevListMeta *meta, uint64_t *offsets, unsigned *err, cudaStream_t stream)
{
    // the scratch after the offsets: tile bases, then tile words (devlist_scratch_bytes)
    const uint32_t tiles_max = devlist_tiles(max_n);
    uint64_t *tile_base = offsets + (size_t)max_n + 1;
    uint32_t *tile_aux = reinterpret_cast<uint32_t *>(tile_base + tiles_max);
    const int tile_ctas = (int)(tiles_max < 304u ? tiles_max : 304u);
    const bool single = tiles_max == 1;  // the tile kernel finishes the plan itself
    cudaError_t e = launch_k(l.pdl, kvx_devlist_tile_kernel, tile_ctas, (int)kListTile, 0, stream, src, dst, sizes,
                             count, max_n, offsets, tile_base, tile_aux, single ? meta : nullptr, err);
    if (e == cudaSuccess && !single)
        e = launch_k(l.pdl, kvx_devlist_base_kernel, 1, 1024, 0, stream, count, max_n, meta, tile_base,
                     static_cast<const uint32_t *>(tile_aux), err);
    if (e != cudaSuccess)
        return e;
    const bool dyn = l.assign == KVX_ASSIGN_DYNAMIC;
    switch (l.unroll) {
    case 2: return launch_devlist_p<2>(l, src, dst, sizes, meta, offsets, tile_base, dyn, stream);
    case 4: return launch_devlist_p<4>(l, src, dst, sizes, meta, offsets, tile_base, dyn, stream);
    default: return launch_devlist_p<8>(l, src, dst, sizes, meta, offsets, tile_base, dyn, stream);
    }
}


cudaError_t set_debug_bounds(const uint64_t *lo, const uint64_t *hi, uint32_t n)
{
    uint64_t pairs[2 * KVX_DEBUG_BOUNDS_MAX];
    for (uint32_t i = 0; i < n; ++i) {
        pairs[2 * i] = lo[i];
        pairs[2 * i + 1] = hi[i];
    }
    // no copy in flight may see a half-written table
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess && n)
        e = cudaMemcpyToSymbol(c_bounds, pairs, sizeof(uint64_t) * 2 * n);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbol(c_bounds_n, &n, sizeof(n));
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    return e;
}

cudaError_t launch_wait_selftest(uint64_t timeout_ns, unsigned *err, cudaStream_t stream)
{
    kvx_wait_selftest_kernel<<<1, 32, 0, stream>>>(timeout_ns, err);
    return cudaGetLastError();
}

}  // namespace kvx
