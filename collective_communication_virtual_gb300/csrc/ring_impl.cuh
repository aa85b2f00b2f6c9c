// ring_impl.cuh -- the staged ring: reduce-scatter and all-gather steps moving chunks
// from virtual rank to virtual rank through device-memory FIFOs.
//
// Structure (NCCL book section 2.2 channels, 2.3 ring, 2.4 protocols):
//  * one CTA per (channel, rank); channel ch owns the sub-range [ch*Lc, (ch+1)*Lc) of
//    every rank block;
//  * rank r receives from r-1 through its own FIFO of 8 slots (NCCL_STEPS) and sends
//    into the FIFO of r+1; a chunk is 4 slots (ALLREDUCE_CHUNKSTEPS), so two chunks can
//    be in flight per hop;
//  * all-reduce = N-1 reduce-scatter stages then N-1 all-gather rounds.  At stage s rank
//    r works on block (r + N - 1 - s) mod N (RingARAlgorithm::getNextSendAddr): stage 0
//    sends its own copy, stages 1..N-2 receive a partial, combine it with their own
//    element and send it on, stage N-1 finishes block r.  All-gather round i sends block
//    (r - i) mod N and receives (r - i - 1) mod N (the ring AllGather of "NCCL Expert
//    Course 17"); the finishing stage and round 0 are one step.
//
// Protocols on the FIFO slots:
//  * Simple: raw payload; the producer publishes a slot by a counter ("tail") after a
//    CTA barrier and a fence, the consumer returns it by another counter ("head");
//  * LL: every 8-byte word is {4 data bytes, 4-byte flag}, written and read as one
//    single-copy-atomic 64-bit access, so a word is valid exactly when its flag matches;
//  * LL128: every 128-byte line is 120 data bytes and an 8-byte flag.  NCCL relies on
//    NVLink delivering a 128-byte line at once, so a reader that sees a line's flag sees
//    its data; within one GPU the PTX memory model orders a flag after data only through
//    a fence.  So a warp stores its lines with their flags (the first line's flag as
//    zero), synchronizes, fences and then sets the first line's flag: the release flag.
//    The reader polls that one flag, fences and synchronizes, then loads the lines and
//    checks their flags as it reads them.
//  Simple counters are 64-bit (launch epoch << 32 | slot count) so values from earlier
//  launches always compare lower; LL flags are (epoch & 0xFF) << 24 | slot count and the
//  host clears the FIFOs whenever that byte wraps.
//
// Every wait is bounded: it gives up after timeoutNs without progress, or when the host
// or another CTA raised an abort, records the reason in the status word and the kernel
// returns.  No trap, no assert.
#pragma once

#include "device.cuh"

namespace vc {

enum { kRecv = 1, kLocal = 2, kOut = 4, kSend = 8 };

template <int DT>
__device__ __forceinline__ uint32_t op_word_rt(int op, uint32_t a, uint32_t b) {
    switch (op) {
    case kSum: return op_word<DT, kSum>(a, b);
    case kProd: return op_word<DT, kProd>(a, b);
    case kMin: return op_word<DT, kMin>(a, b);
    default: return op_word<DT, kMax>(a, b);
    }
}

template <int DT>
__device__ __forceinline__ uint4 op_vec_rt(int op, uint4 a, uint4 b) {
    return make_uint4(op_word_rt<DT>(op, a.x, b.x), op_word_rt<DT>(op, a.y, b.y),
                      op_word_rt<DT>(op, a.z, b.z), op_word_rt<DT>(op, a.w, b.w));
}

// L2 residency.  The ring streams every user byte through once but passes each FIFO slot
// from one SM to another a few microseconds after writing it, so user loads and stores are
// marked to leave L2 first and FIFO stores to stay, which keeps slots in L2 between their
// write and their read instead of sending them through DRAM; a FIFO load marks the line
// as the first to go, since the slot is dead once read.
__device__ __forceinline__ unsigned long long l2_evict_first() {
    unsigned long long p;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ unsigned long long l2_evict_last() {
    unsigned long long p;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint4 ld_user16(const void* p) {
    uint4 v;
    asm("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(l2_evict_first()));
    return v;
}
__device__ __forceinline__ uint2 ld_user8(const void* p) {
    uint2 v;
    asm("ld.global.L1::no_allocate.L2::cache_hint.v2.u32 {%0,%1}, [%2], %3;"
        : "=r"(v.x), "=r"(v.y) : "l"(p), "l"(l2_evict_first()));
    return v;
}
__device__ __forceinline__ void st_user16(void* p, uint4 v) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(l2_evict_first()) : "memory");
}
__device__ __forceinline__ void st_user8(void* p, uint2 v) {
    asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1,%2}, %3;"
                 :: "l"(p), "r"(v.x), "r"(v.y), "l"(l2_evict_first()) : "memory");
}
__device__ __forceinline__ uint4 ld_fifo16(const void* p) {
    uint4 v;
    asm volatile("ld.global.cg.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(l2_evict_first()) : "memory");
    return v;
}
__device__ __forceinline__ uint2 ld_fifo8(const void* p) {
    uint2 v;
    asm volatile("ld.global.cg.L2::cache_hint.v2.u32 {%0,%1}, [%2], %3;"
                 : "=r"(v.x), "=r"(v.y) : "l"(p), "l"(l2_evict_first()) : "memory");
    return v;
}
__device__ __forceinline__ void st_fifo16(void* p, uint4 v) {
    asm volatile("st.global.cg.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(l2_evict_last()) : "memory");
}
// Drop a consumed 128-byte FIFO line from L2 without writing it back to DRAM (its data is
// dead until the producer rewrites it; PTX treats the discard as a weak write of an
// indeterminate value, which the fence before the head word orders before that rewrite).
// Simple slots are discarded (their validity lives in the tail counters) and LL128 slots of
// eager launches; a flag protocol must not discard where the stale DRAM copy the discard
// exposes could hold an old flag of the same value (an LL epoch byte that wrapped, or a
// captured graph replaying its fixed epoch).
__device__ __forceinline__ void discard_l2_line(const void* p) {
    asm volatile("discard.global.L2 [%0], 128;" :: "l"(p) : "memory");
}
__device__ __forceinline__ void st_fifo8(void* p, uint2 v) {
    asm volatile("st.global.cg.L2::cache_hint.v2.u32 [%0], {%1,%2}, %3;"
                 :: "l"(p), "r"(v.x), "r"(v.y), "l"(l2_evict_last()) : "memory");
}

// Load UB bytes of user data (ne valid elements, the rest zero).  ALIGN is the byte
// alignment the caller guarantees for a full unit when `aligned` holds.
template <int ESZ, int UB, int ALIGN>
__device__ __forceinline__ uint4 load_unit(const char* p, int ne, bool aligned) {
    constexpr int UE = UB / ESZ;
    if (aligned && ne == UE) {
        if (UB == 16 && ALIGN == 16) return ld_user16(p);
        const uint2 lo = ld_user8(p);
        if (UB == 8) return make_uint4(lo.x, lo.y, 0u, 0u);
        const uint2 hi = ld_user8(p + 8);
        return make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < UE; i++) {
        if (i < ne) {
            const uint32_t e = ld_elem<ESZ>(p, i);
            if (ESZ == 4) w[i] = e;
            else w[i >> 1] |= e << (16 * (i & 1));
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Store a unit of reduced DT elements as OUT elements (epilogue when `epi`).
template <int DT, int OUT, int UB, int ALIGN>
__device__ __forceinline__ void store_unit(char* p, uint4 v, int ne, bool aligned, bool epi,
                                           bool hasScale, float scale) {
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int OSZ = DTypeOf<OUT>::size;
    constexpr int UE = UB / ESZ;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if (!epi) {
        if (aligned && ne == UE) {
            if (UB == 16 && ALIGN == 16) { st_user16(p, v); return; }
            st_user8(p, make_uint2(v.x, v.y));
            if (UB == 16) st_user8(p + 8, make_uint2(v.z, v.w));
            return;
        }
#pragma unroll
        for (int i = 0; i < UE; i++) {
            if (i < ne) {
                const uint32_t e = ESZ == 4 ? w[i] : ((w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu);
                st_elem<ESZ>(p, i, e);
            }
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < UE; i++) {
        if (i < ne) {
            const uint32_t e = ESZ == 4 ? w[i] : ((w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu);
            float f = elem_to_f32<DT>(e);
            if (hasScale) f = __fmul_rn(f, scale);
            st_elem<OSZ>(p, i, f32_to_elem<OUT>(f));
        }
    }
}

struct RingCtx {
    int ch, r;
    char* myFifo;
    char* nextFifo;
    unsigned long long* myHead;      // I post: slots of my FIFO consumed
    unsigned long long* myTail;      // prev posts: slots of my FIFO produced (Simple)
    unsigned long long* nextHead;    // next posts: credits for my sends
    unsigned long long* nextTail;    // I post: slots of next's FIFO produced (Simple)
    unsigned int sendSeq, recvSeq;
};

// The sequence half of the LL128 line flags a slot receives.  Test hook
// (RingArgs::testBadFlagRank): that rank expects every line flag off by 2^31, as if its
// predecessor had stored wrong ones, and must report the mismatch.
__device__ __forceinline__ unsigned int line_seq(const RingArgs& a, const RingCtx& c) {
    return c.recvSeq + 1u + (c.r == a.testBadFlagRank ? 0x80000000u : 0u);
}

// Test hook (RingArgs::testJitterNs): a pseudo-random sleep of up to testJitterNs
// nanoseconds, different per thread and call, so that tests see other interleavings of
// data stores, flag stores and flag reads than the usual ones.  Off (one uniform branch)
// when testJitterNs is 0.
__device__ __forceinline__ void test_jitter(const RingArgs& a, unsigned salt) {
    if (a.testJitterNs == 0u) return;
    unsigned h = (unsigned)clock() ^ (salt * 0x9E3779B9u) ^ (threadIdx.x * 0x85EBCA6Bu) ^ (blockIdx.x * 0xC2B2AE35u);
    h ^= h >> 15;
    h *= 0x2C1B3C6Du;
    h ^= h >> 12;
    __nanosleep(h % a.testJitterNs);
}

// Acquire/release fence at GPU scope: after a relaxed (volatile) read of a counter or
// flag it completes an acquire, before a relaxed write of one it completes a release (and,
// after a barrier, covers what the other threads stored before the barrier).  Lighter than
// the sequentially consistent fence, which the protocols do not need.
__device__ __forceinline__ void fence_acq_rel() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Give up a wait: record why (abort or timeout); a timeout also raises the device abort
// word so every other waiter gives up too.  Returns false for the caller to pass on.
static __device__ __noinline__ bool wait_failed(const RingArgs& a, int ch, int r, unsigned int seq, bool timedOut) {
    report_error(a.status, a.statusHost, (!timedOut && *a.abortHost) ? vAborted : vTimeout, ch, r, seq);
    if (timedOut) atomicExch(a.abortDev, 1u);
    return false;
}

// A flag-protocol invariant failed (a line flag that does not match after its warp's
// release flag did): record it and raise the device abort word.
static __device__ __noinline__ void protocol_failed(const RingArgs& a, int ch, int r, unsigned int seq) {
    report_error(a.status, a.statusHost, vInternalError, ch, r, seq);
    atomicExch(a.abortDev, 1u);
}

// Checked every 64 polls: an abort raised by the host or another CTA, or this wait's
// deadline.  Returns 0 to keep waiting, 1 aborted, 2 timed out.
__device__ __forceinline__ int wait_check(const RingArgs& a, unsigned long long t0) {
    if (*(volatile unsigned int*)a.abortDev || *a.abortHost) return 1;
    if (global_timer_ns() - t0 > a.timeoutNs) return 2;
    return 0;
}

// Spin until *p >= target (monotonic 64-bit counters), then fence; the value seen goes to
// *seen.  Bounded.
static __device__ __noinline__ bool wait_counter(const RingArgs& a, int ch, int r, const unsigned long long* p,
                                                 unsigned long long target, unsigned int seq,
                                                 unsigned long long* seen) {
    const unsigned long long t0 = global_timer_ns();
    for (unsigned int it = 0;; it++) {
        const unsigned long long v = ld_volatile_u64(p);
        if (v >= target) {
            fence_acq_rel();
            *seen = v;
            return true;
        }
        if ((it & 63u) == 63u) {
            const int why = wait_check(a, t0);
            if (why) return wait_failed(a, ch, r, seq, why == 2);
        }
    }
}

// Spin until the 64-bit flag at p equals target.  Bounded.
static __device__ __noinline__ bool wait_flag64(const RingArgs& a, int ch, int r, const void* p,
                                                unsigned long long target, unsigned int seq) {
    const unsigned long long t0 = global_timer_ns();
    for (unsigned int it = 0;; it++) {
        if (ld_volatile_u64(p) == target) return true;
        if ((it & 63u) == 63u) {
            const int why = wait_check(a, t0);
            if (why) return wait_failed(a, ch, r, seq, why == 2);
        }
    }
}

// Spin until both LL words at p carry `flag`; returns their data halves.  Bounded.
static __device__ __noinline__ bool wait_ll_slow(const RingArgs& a, int ch, int r, const void* p,
                                                 unsigned int flag, uint2* data, unsigned int seq) {
    const unsigned long long t0 = global_timer_ns();
    for (unsigned int it = 0;; it++) {
        unsigned long long w0, w1;
        ld_volatile_u64x2(p, w0, w1);
        if ((unsigned int)(w0 >> 32) == flag && (unsigned int)(w1 >> 32) == flag) {
            *data = make_uint2((unsigned int)w0, (unsigned int)w1);
            return true;
        }
        if ((it & 63u) == 63u) {
            const int why = wait_check(a, t0);
            if (why) return wait_failed(a, ch, r, seq, why == 2);
        }
    }
}

// The counter values thread 0 has seen in this launch: [0] the tail of its own FIFO, [1]
// the head of the next rank's.  Both only grow within a launch, so a slot or a credit
// already covered by a value seen (and fenced after) needs no load: the producer often
// runs several slots ahead, and one head value grants up to kFifoSlots sends.
__device__ __forceinline__ unsigned long long* seen_counters() {
    __shared__ unsigned long long seen[2];
    return seen;
}

// Thread 0 takes the slot credit (and, for Simple, waits for the slot's data); the CTA
// then agrees on success.
template <int PROTO, int kind>
__device__ __forceinline__ bool slot_begin(const RingArgs& a, const RingCtx& c) {
    test_jitter(a, c.recvSeq * 3u + c.sendSeq);
    bool fail = false;
    if (threadIdx.x == 0) {
        unsigned long long* seen = seen_counters();
        if (PROTO == vProtoSimple && (kind & kRecv)) {
            const unsigned long long want = a.epochHi | (c.recvSeq + 1ull);
            if (seen[0] < want) fail = !wait_counter(a, c.ch, c.r, c.myTail, want, c.recvSeq, &seen[0]);
        }
        if (!fail && (kind & kSend) && c.sendSeq >= (unsigned)kFifoSlots) {
            const unsigned long long want = a.epochHi | (c.sendSeq - kFifoSlots + 1ull);
            if (seen[1] < want) fail = !wait_counter(a, c.ch, c.r, c.nextHead, want, c.sendSeq, &seen[1]);
        }
    }
    return !__syncthreads_or(fail);
}

// Publish the slot (Simple tail) and return consumed slots (head).  Call after a barrier.
template <int PROTO, int kind>
__device__ __forceinline__ void slot_end(const RingArgs& a, RingCtx& c) {
    if (threadIdx.x == 0) {
        fence_acq_rel();
        if (PROTO == vProtoSimple && (kind & kSend))
            st_volatile_u64(c.nextTail, a.epochHi | (c.sendSeq + 1ull));
        if (kind & kRecv) st_volatile_u64(c.myHead, a.epochHi | (c.recvSeq + 1ull));
    }
    if (kind & kSend) c.sendSeq++;
    if (kind & kRecv) c.recvSeq++;
}

// Units per thread whose loads are in flight together: as many as fit in the 64
// registers of a thread of a 512-thread CTA, two of which share an SM (LL: two; the
// 16-bit LL128 instances take two lines per lane group at a time in their out-of-line
// step, whose packed ops and bounds need more registers).
template <int PROTO, int ESZ> struct RingUnroll {
    static constexpr int value = PROTO == vProtoLL ? 2 : 4;
    static constexpr int general = ESZ == 2 ? 2 : value;     // LL128's out-of-line step
};

// The general step of an LL128 slot (out of line, so the common whole-line steps keep their
// registers): bounds per lane, element accesses at ragged ends, the epilogue; lane 7 moves
// its 8 data bytes alone, with the line's flag.  Lines Lb + g + k * perIter, as in
// ring_slot.  rseq / sseq: the sequence halves of the received and sent flags.  Returns
// whether a received line's flag did not match (checked where lane 7's place holds payload;
// the release flag has already ordered every line).
template <int DT, int OUT, int kind, int R>
__device__ __noinline__ bool ll128_step_general(const RingArgs& a, const char* rs, char* ss, const char* in,
                                                char* out, unsigned int Lb, unsigned int lines, unsigned int P,
                                                bool epi, unsigned int rseq, unsigned int sseq, unsigned int L0) {
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int OSZ = DTypeOf<OUT>::size;
    const bool aligned = a.aligned != 0;
    const bool hasScale = a.hasScale != 0;
    const unsigned int lane = threadIdx.x & 31, g = lane >> 3, t = lane & 7;
    const unsigned int perIter = (blockDim.x >> 5) * 4;
    const unsigned int halfBase = 112 * lines;
    bool bad = false;
    uint4 v[R], l[R];
#pragma unroll
    for (int k = 0; k < R; k++) {
        const unsigned int L = Lb + g + k * perIter;
        const unsigned int b = t < 7 ? 112 * L + 16 * t : halfBase + 8 * L;   // payload byte
        v[k] = make_uint4(0u, 0u, 0u, 0u);
        l[k] = v[k];
        // lane 7 reads its 8-byte place with the line's flag whether or not the place holds
        // payload
        if ((kind & kRecv) && L < lines && b < P) v[k] = ld_fifo16(rs + (size_t)L * 128 + 16 * t);
        if (L < lines && b < P) {
            if (kind & kLocal) {
                const int ne = (int)(min(t < 7 ? 16u : 8u, P - b) / ESZ);
                l[k] = t < 7 ? load_unit<ESZ, 16, 16>(in + b, ne, aligned)
                             : load_unit<ESZ, 8, 8>(in + b, ne, aligned);
            }
        }
    }
#pragma unroll
    for (int k = 0; k < R; k++) {
        const unsigned int L = Lb + g + k * perIter;
        const unsigned int b = t < 7 ? 112 * L + 16 * t : halfBase + 8 * L;
        if (L >= lines) break;
        if ((kind & kRecv) && t == 7 && b < P)     // the line's flag, in lane 7's place
            bad |= ((v[k].z ^ rseq) | (v[k].w ^ (unsigned int)(a.epochHi >> 32))) != 0u;
        uint4 x = v[k];
        if (b < P) {
            if (kind & kLocal) x = (kind & kRecv) ? op_vec_rt<DT>(a.op, x, l[k]) : l[k];
            if (kind & kOut) {
                const int ne = (int)(min(t < 7 ? 16u : 8u, P - b) / ESZ);
                char* o = out + (size_t)(b / ESZ) * OSZ;
                if (t < 7) store_unit<DT, OUT, 16, 16>(o, x, ne, aligned, epi, hasScale, a.scale);
                else store_unit<DT, OUT, 8, 8>(o, x, ne, aligned, epi, hasScale, a.scale);
            }
        }
        if (kind & kSend) {
            if (t < 7) {
                st_fifo16(ss + (size_t)L * 128 + 16 * t, x);
            } else {
                const bool rel = L == L0;     // the release flag follows the fence
                st_fifo16(ss + (size_t)L * 128 + 112,
                          make_uint4(x.x, x.y, rel ? 0u : sseq, rel ? 0u : (unsigned int)(a.epochHi >> 32)));
            }
        }
    }
    return bad;
}

// One slot of m elements (a slot is at most 16 MiB, so 32-bit offsets).  `in`: user input
// at the slot's first element (kLocal); `out`: user output at the slot's first element
// (kOut).  Each thread takes R units at a time and issues all their loads (FIFO data or
// flags, user data) before combining and storing any of them.
template <int DT, int OUT, int PROTO, int kind>
__device__ __forceinline__ bool ring_slot(const RingArgs& a, RingCtx& c, const char* in, char* out,
                                          unsigned int m, bool epi) {
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int OSZ = DTypeOf<OUT>::size;
    constexpr int R = RingUnroll<PROTO, ESZ>::value;
    const bool aligned = a.aligned != 0;
    const bool hasScale = a.hasScale != 0;
    if (!slot_begin<PROTO, kind>(a, c)) return false;
    const char* rs = c.myFifo + (size_t)(c.recvSeq % kFifoSlots) * a.slotBytes;
    char* ss = c.nextFifo + (size_t)(c.sendSeq % kFifoSlots) * a.slotBytes;
    const unsigned int T = blockDim.x;
    bool fail = false;
    if (PROTO == vProtoSimple) {
        // 16 payload bytes per unit, contiguous in the slot.
        constexpr int UE = 16 / ESZ;
        const unsigned int units = (m + UE - 1) / UE;
        for (unsigned int u0 = threadIdx.x; u0 < units; u0 += R * T) {
            uint4 v[R], l[R];
#pragma unroll
            for (int k = 0; k < R; k++) {
                const unsigned int u = u0 + k * T;
                v[k] = make_uint4(0u, 0u, 0u, 0u);
                l[k] = v[k];
                if (u < units) {
                    if (kind & kRecv) v[k] = ld_fifo16(rs + (size_t)u * 16);
                    if (kind & kLocal) l[k] = load_unit<ESZ, 16, 16>(in + (size_t)u * 16, (int)min((unsigned)UE, m - u * UE), aligned);
                }
            }
#pragma unroll
            for (int k = 0; k < R; k++) {
                const unsigned int u = u0 + k * T;
                if (u >= units) break;
                const int ne = (int)min((unsigned)UE, m - u * UE);
                uint4 x = v[k];
                if (kind & kLocal) x = (kind & kRecv) ? op_vec_rt<DT>(a.op, x, l[k]) : l[k];
                if (kind & kOut)
                    store_unit<DT, OUT, 16, 16>(out + (size_t)u * UE * OSZ, x, ne, aligned, epi, hasScale, a.scale);
                if (kind & kSend) st_fifo16(ss + (size_t)u * 16, x);
            }
            if (kind & kRecv) {
                // The warp read R runs of 32 units (4 lines each); once every lane has used
                // them, lanes 0..4R-1 discard one line each.  Only when every run is whole,
                // which the warp decides alike (ub is the warp's first unit of the round).
                const unsigned int ub = u0 - (threadIdx.x & 31u);
                if (ub + (R - 1) * T + 32 <= units) {
                    __syncwarp();
                    const unsigned int lane = threadIdx.x & 31u;
                    if (lane < 4u * R)
                        discard_l2_line(rs + (size_t)(ub + (lane >> 2) * T) * 16 + 128 * (lane & 3u));
                }
            }
            test_jitter(a, u0);
        }
    } else if (PROTO == vProtoLL) {
        // 8 payload bytes per unit, stored as two {data, flag} 64-bit words.
        constexpr int UE = 8 / ESZ;
        const unsigned int units = (m + UE - 1) / UE;
        const unsigned int rflag = a.llEpoch | ((c.recvSeq + 1u) & 0xFFFFFFu);
        const unsigned long long sflag = (unsigned long long)(a.llEpoch | ((c.sendSeq + 1u) & 0xFFFFFFu)) << 32;
        for (unsigned int u0 = threadIdx.x; u0 < units && !fail; u0 += R * T) {
            unsigned long long w0[R], w1[R];
            uint4 l[R];
#pragma unroll
            for (int k = 0; k < R; k++) {
                const unsigned int u = u0 + k * T;
                w0[k] = w1[k] = 0ull;
                l[k] = make_uint4(0u, 0u, 0u, 0u);
                if (u < units) {
                    if (kind & kRecv) ld_volatile_u64x2(rs + (size_t)u * 16, w0[k], w1[k]);
                    if (kind & kLocal) l[k] = load_unit<ESZ, 8, 8>(in + (size_t)u * 8, (int)min((unsigned)UE, m - u * UE), aligned);
                }
            }
#pragma unroll
            for (int k = 0; k < R; k++) {
                const unsigned int u = u0 + k * T;
                if (u >= units || fail) break;
                const int ne = (int)min((unsigned)UE, m - u * UE);
                uint4 x = make_uint4(0u, 0u, 0u, 0u);
                if (kind & kRecv) {
                    if ((unsigned int)(w0[k] >> 32) == rflag && (unsigned int)(w1[k] >> 32) == rflag) {
                        x.x = (unsigned int)w0[k];
                        x.y = (unsigned int)w1[k];
                    } else {
                        uint2 d;
                        if (!wait_ll_slow(a, c.ch, c.r, rs + (size_t)u * 16, rflag, &d, c.recvSeq)) { fail = true; break; }
                        x.x = d.x;
                        x.y = d.y;
                    }
                }
                if (kind & kLocal) x = (kind & kRecv) ? op_vec_rt<DT>(a.op, x, l[k]) : l[k];
                if (kind & kOut)
                    store_unit<DT, OUT, 8, 8>(out + (size_t)u * UE * OSZ, x, ne, aligned, epi, hasScale, a.scale);
                if (kind & kSend) st_volatile_u64x2(ss + (size_t)u * 16, sflag | x.x, sflag | x.y);
            }
            test_jitter(a, u0);
        }
    } else {
        // LL128: 128-byte lines of 120 payload bytes + an 8-byte flag.  Eight lanes share a
        // line: lanes 0..6 carry 16 payload bytes, lane 7 carries 8 bytes and the flag.
        // Payload layout of a slot of P bytes in `lines` lines: bytes [0, 112 lines) fill the
        // 16-byte places in order (line L, place t holds bytes 112 L + 16 t), and the rest,
        // [112 lines, P), the 8-byte places (line L holds bytes 112 lines + 8 L), so every
        // 16-byte place maps to a 16-byte aligned piece of the user buffer and a warp's 28
        // full places (4 consecutive lines) to 448 contiguous bytes.
        const unsigned int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const unsigned int g = lane >> 3, t = lane & 7;
        const unsigned int P = m * ESZ;
        const unsigned int lines = (P + 119) / 120;
        const unsigned int perIter = (T >> 5) * 4;       // lines the CTA covers per step
        const unsigned long long rflag = a.epochHi | (c.recvSeq + 1ull);
        const unsigned long long sflag = a.epochHi | (c.sendSeq + 1ull);
        // Eager launches carry a 32-bit epoch no other launch used, so no stale copy of a
        // line in DRAM can hold a flag this launch waits for, and consumed lines may be
        // dropped from L2; captured graphs (and the no-alloc path) replay epoch 1 and keep them.
        const bool discardLL128 = a.epochHi != (1ull << 32);
        // The lines of this warp: warp * 4 + j * perIter + (0..3) for j = 0, 1, ...; the q-th
        // of them (q = 4 j + i) is line warp * 4 + (q / 4) * perIter + q % 4.
        const unsigned int mine = lines > warp * 4 ? (lines - warp * 4 + perIter - 1) / perIter * 4 : 0;
        // The warp's first line carries its release flag: written as zero with the data,
        // then, after the warp's data stores, a barrier and a fence, set to the slot's flag.
        // A reader that sees it set (and fences) sees every line the warp stored, so it
        // polls that one flag; the other lines' flags are stored with their data and checked
        // as the data pass reads them.
        const unsigned int L0 = warp * 4;
        if ((kind & kRecv) && mine > 0) {
            const char* fp = rs + (size_t)L0 * 128 + 120;
            if (ld_volatile_u64(fp) != rflag && !wait_flag64(a, c.ch, c.r, fp, rflag, c.recvSeq)) fail = true;
            fence_acq_rel();
            __syncwarp();
        }
        if (!__any_sync(0xFFFFFFFFu, fail)) {
            const unsigned int halfBase = 112 * lines;
            // Steps of R lines per lane group; lane group g takes lines Lb + g + k * perIter.
            for (unsigned int Lb = warp * 4; Lb < lines; Lb += R * perIter) {
                const bool whole = aligned && !epi && halfBase + 8 * (Lb + (R - 1) * perIter + 4) <= P;
                if (whole) {
                    // Every line of the step exists and is full: one 16-byte FIFO access per
                    // lane (lane 7's covers its 8 data bytes and the line's flag; the warp's
                    // first line gets zero there -- never a valid flag -- until the release
                    // flag follows the fence), one 16-byte user access per lane 0..6 and one
                    // 8-byte user access per lane 7 (the four lanes 7 of a step cover 32
                    // contiguous user bytes).  No lane waits on another's load: sharing
                    // 16-byte accesses of lanes 7 through shuffles made the whole warp wait
                    // for them, and cost a fifth of the all-reduce's time.
                    uint4 v[R], l[R];
#pragma unroll
                    for (int k = 0; k < R; k++) {
                        const unsigned int L = Lb + g + k * perIter;
                        v[k] = make_uint4(0u, 0u, 0u, 0u);
                        l[k] = v[k];
                        if (kind & kRecv) v[k] = ld_fifo16(rs + (size_t)L * 128 + 16 * t);
                        if (kind & kLocal) {
                            if (t < 7) {
                                l[k] = ld_user16(in + 112 * L + 16 * t);
                            } else {
                                const uint2 h = ld_user8(in + halfBase + 8 * L);
                                l[k] = make_uint4(h.x, h.y, 0u, 0u);
                            }
                        }
                    }
                    if (kind & kRecv) {
                        // the flag's halves: the launch epoch over the slot's sequence number
                        const unsigned int rlo = line_seq(a, c), hi = (unsigned int)(a.epochHi >> 32);
#pragma unroll
                        for (int k = 0; k < R; k++)
                            if (t == 7) fail |= ((v[k].z ^ rlo) | (v[k].w ^ hi)) != 0u;
                    }
#pragma unroll
                    for (int k = 0; k < R; k++) {
                        const unsigned int L = Lb + g + k * perIter;
                        uint4 x = v[k];
                        if (kind & kLocal) x = (kind & kRecv) ? op_vec_rt<DT>(a.op, x, l[k]) : l[k];
                        if (t == 7) {
                            const bool rel = L == L0;     // the release flag follows the fence
                            x.z = rel ? 0u : c.sendSeq + 1u;
                            x.w = rel ? 0u : (unsigned int)(a.epochHi >> 32);
                        }
                        if (kind & kOut) {
                            if (t < 7) st_user16(out + 112 * L + 16 * t, x);
                            else st_user8(out + halfBase + 8 * L, make_uint2(x.x, x.y));
                        }
                        if (kind & kSend) st_fifo16(ss + (size_t)L * 128 + 16 * t, x);
                    }
                    if ((kind & kRecv) && discardLL128) {
                        // the step's R x 4 lines of the warp, read by every lane: dropped
                        // from L2 (one lane per line) once all have used them
                        __syncwarp();
                        if (lane < 4u * R)
                            discard_l2_line(rs + (size_t)(Lb + (lane >> 2) * perIter + (lane & 3u)) * 128);
                    }
                } else {
                    // the general step takes RG of the step's R lines per lane group at a time
                    constexpr int RG = RingUnroll<PROTO, ESZ>::general;
#pragma unroll
                    for (int h = 0; h < R; h += RG)
                        if (Lb + h * perIter < lines)
                            fail |= ll128_step_general<DT, OUT, kind, RG>(a, rs, ss, in, out, Lb + h * perIter, lines,
                                                                          P, epi, line_seq(a, c), c.sendSeq + 1u, L0);
                }
                test_jitter(a, Lb);
            }
            // In the data pass `fail` marks a line flag that did not match after the release
            // flag did: a broken protocol invariant, reported, and the ring stops.
            if ((kind & kRecv) && __any_sync(0xFFFFFFFFu, fail)) {
                if (lane == 0) protocol_failed(a, c.ch, c.r, c.recvSeq);
                fail = true;
            } else if ((kind & kSend) && mine > 0) {
                // after every lane's data stores: the release flag
                test_jitter(a, 0x5157u);
                __syncwarp();
                if (lane == 0) {
                    fence_acq_rel();
                    st_volatile_u64(ss + (size_t)L0 * 128 + 120, sflag);
                }
            }
        }
    }
    if (__syncthreads_or(fail)) return false;
    slot_end<PROTO, kind>(a, c);
    return true;
}

// One transfer of n elements of one block: ceil(n / slotElems) slots.
template <int DT, int OUT, int PROTO, int kind>
__device__ __forceinline__ bool ring_transfer(const RingArgs& a, RingCtx& c, const char* in, char* out,
                                              size_t n, bool epi) {
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int OSZ = DTypeOf<OUT>::size;
    for (size_t k = 0; k < n; k += a.slotElems) {
        const unsigned int m = (unsigned int)min(a.slotElems, n - k);
        if (!ring_slot<DT, OUT, PROTO, kind>(a, c, (kind & kLocal) ? in + k * ESZ : nullptr,
                                             (kind & kOut) ? out + k * OSZ : nullptr, m, epi))
            return false;
    }
    return true;
}

// Elements of block `blk` owned by channel ch that lie at or beyond offset o of that
// sub-range, capped at one chunk.  Returns the element index of the sub-range start.
__device__ __forceinline__ size_t seg_len(const RingArgs& a, int ch, int blk, size_t o,
                                          size_t* start) {
    const size_t base = (size_t)blk * a.blockElems;
    const size_t lo = base + min((size_t)ch * a.chanElems, a.blockElems);
    size_t hi = base + min((size_t)(ch + 1) * a.chanElems, a.blockElems);
    hi = min(hi, a.count);
    *start = lo;
    if (hi <= lo + o) return 0;
    return min(a.chunkElems, hi - lo - o);
}

template <int DT, int OUT, int PROTO>
__global__ void __launch_bounds__(kRingThreads, 2) k_ring(const __grid_constant__ RingArgs a) {
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int OSZ = DTypeOf<OUT>::size;
    const int N = a.nRanks;
    RingCtx c;
    c.ch = blockIdx.x / N;
    c.r = blockIdx.x - c.ch * N;
    if (c.r == a.testStallRank) return;             // test hook: a rank that never shows up
    const int r = c.r, ch = c.ch;
    const int next = r + 1 == N ? 0 : r + 1;
    const size_t fifoBytes = (size_t)kFifoSlots * a.slotBytes;
    c.myFifo = a.fifo + (size_t)(ch * N + r) * fifoBytes;
    c.nextFifo = a.fifo + (size_t)(ch * N + next) * fifoBytes;
    c.myHead = a.ctrl + (size_t)(ch * N + r) * kCtrlStride;
    c.myTail = c.myHead + 16;
    c.nextHead = a.ctrl + (size_t)(ch * N + next) * kCtrlStride;
    c.nextTail = c.nextHead + 16;
    c.sendSeq = 0;
    c.recvSeq = 0;
    if (threadIdx.x == 0) {                         // only thread 0 reads them
        seen_counters()[0] = 0ull;
        seen_counters()[1] = 0ull;
    }

    const char* mySend = (const char*)a.send[r];
    char* myRecv = (char*)a.recv[r];
    const bool epi = a.hasScale != 0 || OUT != DT;

    // Loop bound: the longest of this channel's block sub-ranges (block 0 is never
    // shorter than the others; broadcast has one block).
    size_t loopLen;
    {
        const size_t lo = min((size_t)ch * a.chanElems, a.blockElems);
        const size_t hi = min(min((size_t)(ch + 1) * a.chanElems, a.blockElems), a.count);
        loopLen = hi > lo ? hi - lo : 0;
    }

    for (size_t o = 0; o < loopLen; o += a.chunkElems) {
        size_t st;
        if (a.coll == vCollAllReduce || a.coll == vCollReduceScatter) {
            // reduce-scatter stages
            int blk = r == 0 ? N - 1 : r - 1;
            size_t n = seg_len(a, ch, blk, o, &st);
            if (!ring_transfer<DT, DT, PROTO, kLocal | kSend>(a, c, mySend + (st + o) * ESZ, nullptr, n, false)) return;
            for (int s = 1; s < N - 1; s++) {
                blk = (r + N - 1 - s) % N;
                n = seg_len(a, ch, blk, o, &st);
                if (!ring_transfer<DT, DT, PROTO, kRecv | kLocal | kSend>(a, c, mySend + (st + o) * ESZ,
                                                  nullptr, n, false)) return;
            }
            n = seg_len(a, ch, r, o, &st);
            if (a.coll == vCollAllReduce) {
                if (!ring_transfer<DT, DT, PROTO, kRecv | kLocal | kOut | kSend>(a, c, mySend + (st + o) * ESZ,
                                                  myRecv + (st + o) * ESZ, n, false)) return;
                // all-gather rounds: receive block (r - i - 1), forward unless last
                for (int i = 0; i < N - 1; i++) {
                    blk = ((r - i - 1) % N + N) % N;
                    n = seg_len(a, ch, blk, o, &st);
                    const bool ok = i < N - 2
                        ? ring_transfer<DT, DT, PROTO, kRecv | kOut | kSend>(a, c, nullptr, myRecv + (st + o) * ESZ, n, false)
                        : ring_transfer<DT, DT, PROTO, kRecv | kOut>(a, c, nullptr, myRecv + (st + o) * ESZ, n, false);
                    if (!ok) return;
                }
            } else {
                // block r lands at recv[r][st - r * rc + o] = recv[r][ch * Lc + o]
                const size_t t0 = st - (size_t)r * a.blockElems + o;
                if (!ring_transfer<DT, OUT, PROTO, kRecv | kLocal | kOut>(a, c, mySend + (st + o) * ESZ,
                                                   myRecv + t0 * OSZ, n, epi)) return;
            }
        } else if (a.coll == vCollAllGather) {
            // own block r: copy to recv[r] at block r and send it on
            size_t n = seg_len(a, ch, r, o, &st);
            const size_t inOff = st - (size_t)r * a.blockElems + o;     // within send[r]
            if (!ring_transfer<DT, DT, PROTO, kLocal | kOut | kSend>(a, c, mySend + inOff * ESZ,
                                              myRecv + (st + o) * ESZ, n, false)) return;
            for (int i = 0; i < N - 1; i++) {
                const int blk = ((r - i - 1) % N + N) % N;
                n = seg_len(a, ch, blk, o, &st);
                const bool ok = i < N - 2
                    ? ring_transfer<DT, DT, PROTO, kRecv | kOut | kSend>(a, c, nullptr, myRecv + (st + o) * ESZ, n, false)
                    : ring_transfer<DT, DT, PROTO, kRecv | kOut>(a, c, nullptr, myRecv + (st + o) * ESZ, n, false);
                if (!ok) return;
            }
        } else {
            // broadcast: a chain root, root+1, ..., root-1
            const int pos = ((r - a.root) % N + N) % N;
            const size_t n = seg_len(a, ch, 0, o, &st);
            char* dst = myRecv + (st + o) * ESZ;
            bool ok;
            if (pos == 0)
                ok = ring_transfer<DT, DT, PROTO, kLocal | kOut | kSend>(
                    a, c, (const char*)a.send[a.root] + (st + o) * ESZ, dst, n, false);
            else if (pos < N - 1)
                ok = ring_transfer<DT, DT, PROTO, kRecv | kOut | kSend>(a, c, nullptr, dst, n, false);
            else
                ok = ring_transfer<DT, DT, PROTO, kRecv | kOut>(a, c, nullptr, dst, n, false);
            if (!ok) return;
        }
    }
}

// Kernel entry for a (type, output type) pair of one protocol, for the host launcher.
#define VC_RING_SELECTOR(NAME, PROTO)                                                      \
    void* NAME(vDataType_t dt, vDataType_t out) {                                          \
        switch (dt) {                                                                      \
        case vFloat32: return (void*)k_ring<kF32, kF32, PROTO>;                            \
        case vFloat16:                                                                     \
            return out == vFloat32 ? (void*)k_ring<kF16, kF32, PROTO>                      \
                                   : (void*)k_ring<kF16, kF16, PROTO>;                     \
        case vBFloat16:                                                                    \
            return out == vFloat32 ? (void*)k_ring<kBF16, kF32, PROTO>                     \
                                   : (void*)k_ring<kBF16, kBF16, PROTO>;                   \
        case vInt32: return (void*)k_ring<kI32, kI32, PROTO>;                              \
        }                                                                                  \
        return nullptr;                                                                    \
    }

}  // namespace vc
