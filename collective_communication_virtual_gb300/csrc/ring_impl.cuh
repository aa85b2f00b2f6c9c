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
//  * LL128: every 128-byte line is 120 data bytes and an 8-byte flag.  A warp stores its
//    lines' data, synchronizes, fences, then stores the flags; the reader polls the
//    flags, fences, synchronizes, then loads the data.  (NCCL relies on NVLink's
//    128-byte atomicity; within one GPU the PTX memory model only orders the flag after
//    the data through the fence, so the fence is explicit here.)
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

__device__ __forceinline__ uint2 ld_stream8(const void* p) {
    uint2 v;
    asm("ld.global.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ void st_stream8(void* p, uint2 v) {
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" :: "l"(p), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ uint2 ld_cg8(const void* p) {
    uint2 v;
    asm volatile("ld.global.cg.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_cg8(void* p, uint2 v) {
    asm volatile("st.global.cg.v2.u32 [%0], {%1,%2};" :: "l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// Load UB bytes of user data (ne valid elements, the rest zero).  ALIGN is the byte
// alignment the caller guarantees for a full unit when `aligned` holds.
template <int ESZ, int UB, int ALIGN>
__device__ __forceinline__ uint4 load_unit(const char* p, int ne, bool aligned) {
    constexpr int UE = UB / ESZ;
    if (aligned && ne == UE) {
        if (UB == 16 && ALIGN == 16) return ld_stream(p);
        const uint2 lo = ld_stream8(p);
        if (UB == 8) return make_uint4(lo.x, lo.y, 0u, 0u);
        const uint2 hi = ld_stream8(p + 8);
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
            if (UB == 16 && ALIGN == 16) { st_stream(p, v); return; }
            st_stream8(p, make_uint2(v.x, v.y));
            if (UB == 16) st_stream8(p + 8, make_uint2(v.z, v.w));
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
    int ch, r, N;
    char* myFifo;
    char* nextFifo;
    unsigned long long* myHead;      // I post: slots of my FIFO consumed
    unsigned long long* myTail;      // prev posts: slots of my FIFO produced (Simple)
    unsigned long long* nextHead;    // next posts: credits for my sends
    unsigned long long* nextTail;    // I post: slots of next's FIFO produced (Simple)
    unsigned int sendSeq, recvSeq;
};

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

// Spin until *p >= target (monotonic 64-bit counters).  Bounded.
static __device__ __noinline__ bool wait_counter(const RingArgs& a, const RingCtx& c,
                                          const unsigned long long* p, unsigned long long target,
                                          unsigned int seq) {
    const unsigned long long t0 = global_timer_ns();
    for (unsigned int it = 0;; it++) {
        if (ld_volatile_u64(p) >= target) { __threadfence(); return true; }
        if ((it & 63u) == 63u) {
            if (*(volatile unsigned int*)a.abortDev || *a.abortHost) {
                report_error(a.status, a.statusHost, *a.abortHost ? vAborted : vTimeout, c.ch, c.r, seq);
                return false;
            }
            if (global_timer_ns() - t0 > a.timeoutNs) {
                report_error(a.status, a.statusHost, vTimeout, c.ch, c.r, seq);
                atomicExch(a.abortDev, 1u);
                return false;
            }
        }
    }
}

// Spin until the 64-bit flag at p equals target.  Bounded.
static __device__ __noinline__ bool wait_flag64(const RingArgs& a, const RingCtx& c, const void* p,
                                         unsigned long long target, unsigned int seq) {
    const unsigned long long t0 = global_timer_ns();
    for (unsigned int it = 0;; it++) {
        if (ld_volatile_u64(p) == target) return true;
        if ((it & 63u) == 63u) {
            if (*(volatile unsigned int*)a.abortDev || *a.abortHost) {
                report_error(a.status, a.statusHost, *a.abortHost ? vAborted : vTimeout, c.ch, c.r, seq);
                return false;
            }
            if (global_timer_ns() - t0 > a.timeoutNs) {
                report_error(a.status, a.statusHost, vTimeout, c.ch, c.r, seq);
                atomicExch(a.abortDev, 1u);
                return false;
            }
        }
    }
}

// Spin until both LL words at p carry `flag`; returns their data halves.  Bounded.
static __device__ __noinline__ bool wait_ll_slow(const RingArgs& a, const RingCtx& c, const void* p,
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
            if (*(volatile unsigned int*)a.abortDev || *a.abortHost) {
                report_error(a.status, a.statusHost, *a.abortHost ? vAborted : vTimeout, c.ch, c.r, seq);
                return false;
            }
            if (global_timer_ns() - t0 > a.timeoutNs) {
                report_error(a.status, a.statusHost, vTimeout, c.ch, c.r, seq);
                atomicExch(a.abortDev, 1u);
                return false;
            }
        }
    }
}

// LL read: one inline attempt, then the bounded spin out of line.
__device__ __forceinline__ bool wait_ll(const RingArgs& a, const RingCtx& c, const void* p,
                                       unsigned int flag, uint2* data, unsigned int seq) {
    unsigned long long w0, w1;
    ld_volatile_u64x2(p, w0, w1);
    if ((unsigned int)(w0 >> 32) == flag && (unsigned int)(w1 >> 32) == flag) {
        *data = make_uint2((unsigned int)w0, (unsigned int)w1);
        return true;
    }
    return wait_ll_slow(a, c, p, flag, data, seq);
}

// Thread 0 takes the slot credit (and, for Simple, waits for the slot's data); the CTA
// then agrees on success.
template <int PROTO>
__device__ __forceinline__ bool slot_begin(const RingArgs& a, const RingCtx& c, int kind) {
    test_jitter(a, c.recvSeq * 3u + c.sendSeq);
    bool fail = false;
    if (threadIdx.x == 0) {
        if (PROTO == vProtoSimple && (kind & kRecv))
            fail = !wait_counter(a, c, c.myTail, a.epochHi | (c.recvSeq + 1ull), c.recvSeq);
        if (!fail && (kind & kSend) && c.sendSeq >= (unsigned)kFifoSlots)
            fail = !wait_counter(a, c, c.nextHead, a.epochHi | (c.sendSeq - kFifoSlots + 1ull), c.sendSeq);
    }
    return !__syncthreads_or(fail);
}

// Publish the slot (Simple tail) and return consumed slots (head).  Call after a barrier.
template <int PROTO>
__device__ __forceinline__ void slot_end(const RingArgs& a, RingCtx& c, int kind) {
    if (threadIdx.x == 0) {
        __threadfence();
        if (PROTO == vProtoSimple && (kind & kSend))
            st_volatile_u64(c.nextTail, a.epochHi | (c.sendSeq + 1ull));
        if (kind & kRecv) st_volatile_u64(c.myHead, a.epochHi | (c.recvSeq + 1ull));
    }
    if (kind & kSend) c.sendSeq++;
    if (kind & kRecv) c.recvSeq++;
}

// Units per thread whose loads are in flight together; the flag protocols hold more per
// unit, so they take fewer to stay within 64 registers (two 512-thread CTAs per SM).
template <int PROTO> struct RingUnroll { static constexpr int value = PROTO == vProtoSimple ? 4 : 2; };

// One slot of m elements.  `in`: user input at the slot's first element (kLocal);
// `out`: user output at the slot's first element (kOut).  Each thread takes R units at a
// time and issues all their loads (FIFO data or flags, user data) before
// combining and storing any of them.
template <int DT, int OUT, int PROTO>
__device__ __forceinline__ bool ring_slot(const RingArgs& a, RingCtx& c, int kind, const char* in,
                                          char* out, size_t m, bool epi) {
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int OSZ = DTypeOf<OUT>::size;
    constexpr int R = RingUnroll<PROTO>::value;
    const bool aligned = a.aligned != 0;
    const bool hasScale = a.hasScale != 0;
    if (!slot_begin<PROTO>(a, c, kind)) return false;
    const char* rs = c.myFifo + (size_t)(c.recvSeq % kFifoSlots) * a.slotBytes;
    char* ss = c.nextFifo + (size_t)(c.sendSeq % kFifoSlots) * a.slotBytes;
    bool fail = false;
    if (PROTO == vProtoSimple) {
        // 16 payload bytes per unit, contiguous in the slot.
        constexpr int UE = 16 / ESZ;
        const size_t units = (m + UE - 1) / UE;
        for (size_t u0 = threadIdx.x; u0 < units; u0 += (size_t)R * blockDim.x) {
            uint4 v[R], l[R];
#pragma unroll
            for (int k = 0; k < R; k++) {
                const size_t u = u0 + (size_t)k * blockDim.x;
                v[k] = make_uint4(0u, 0u, 0u, 0u);
                l[k] = v[k];
                if (u < units) {
                    if (kind & kRecv) v[k] = ld_cg(rs + u * 16);
                    if (kind & kLocal) l[k] = load_unit<ESZ, 16, 16>(in + u * 16, (int)min((size_t)UE, m - u * UE), aligned);
                }
            }
#pragma unroll
            for (int k = 0; k < R; k++) {
                const size_t u = u0 + (size_t)k * blockDim.x;
                if (u >= units) break;
                const int ne = (int)min((size_t)UE, m - u * UE);
                uint4 x = v[k];
                if (kind & kLocal) x = (kind & kRecv) ? op_vec_rt<DT>(a.op, x, l[k]) : l[k];
                if (kind & kOut)
                    store_unit<DT, OUT, 16, 16>(out + u * UE * OSZ, x, ne, aligned, epi, hasScale, a.scale);
                if (kind & kSend) st_cg(ss + u * 16, x);
            }
            test_jitter(a, (unsigned)u0);
        }
    } else if (PROTO == vProtoLL) {
        // 8 payload bytes per unit, stored as two {data, flag} 64-bit words.
        constexpr int UE = 8 / ESZ;
        const size_t units = (m + UE - 1) / UE;
        const unsigned int rflag = a.llEpoch | ((c.recvSeq + 1u) & 0xFFFFFFu);
        const unsigned long long sflag = (unsigned long long)(a.llEpoch | ((c.sendSeq + 1u) & 0xFFFFFFu)) << 32;
        for (size_t u0 = threadIdx.x; u0 < units && !fail; u0 += (size_t)R * blockDim.x) {
            unsigned long long w0[R], w1[R];
            uint4 l[R];
#pragma unroll
            for (int k = 0; k < R; k++) {
                const size_t u = u0 + (size_t)k * blockDim.x;
                w0[k] = w1[k] = 0ull;
                l[k] = make_uint4(0u, 0u, 0u, 0u);
                if (u < units) {
                    if (kind & kRecv) ld_volatile_u64x2(rs + u * 16, w0[k], w1[k]);
                    if (kind & kLocal) l[k] = load_unit<ESZ, 8, 8>(in + u * 8, (int)min((size_t)UE, m - u * UE), aligned);
                }
            }
#pragma unroll
            for (int k = 0; k < R; k++) {
                const size_t u = u0 + (size_t)k * blockDim.x;
                if (u >= units || fail) break;
                const int ne = (int)min((size_t)UE, m - u * UE);
                uint4 x = make_uint4(0u, 0u, 0u, 0u);
                if (kind & kRecv) {
                    if ((unsigned int)(w0[k] >> 32) == rflag && (unsigned int)(w1[k] >> 32) == rflag) {
                        x.x = (unsigned int)w0[k];
                        x.y = (unsigned int)w1[k];
                    } else {
                        uint2 d;
                        if (!wait_ll_slow(a, c, rs + u * 16, rflag, &d, c.recvSeq)) { fail = true; break; }
                        x.x = d.x;
                        x.y = d.y;
                    }
                }
                if (kind & kLocal) x = (kind & kRecv) ? op_vec_rt<DT>(a.op, x, l[k]) : l[k];
                if (kind & kOut)
                    store_unit<DT, OUT, 8, 8>(out + u * UE * OSZ, x, ne, aligned, epi, hasScale, a.scale);
                if (kind & kSend) st_volatile_u64x2(ss + u * 16, sflag | x.x, sflag | x.y);
            }
            test_jitter(a, (unsigned)u0);
        }
    } else {
        // LL128: 128-byte lines of 120 payload bytes + an 8-byte flag.  Eight lanes share a
        // line: lanes 0..6 carry 16 payload bytes, lane 7 carries 8 bytes and the flag.
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nWarps = blockDim.x >> 5;
        const int g = lane >> 3, t = lane & 7;
        const size_t lines = (m * ESZ + 119) / 120;
        const size_t perIter = (size_t)nWarps * 4;
        const unsigned long long rflag = a.epochHi | (c.recvSeq + 1ull);
        const unsigned long long sflag = a.epochHi | (c.sendSeq + 1ull);
        if (kind & kRecv) {
            if (t == 7) {
                // Flags of this lane's lines, 8 loads in flight at a time; only a flag that
                // is not yet set is waited for on its own.
                for (size_t L0 = (size_t)warp * 4 + g; L0 < lines && !fail; L0 += 8 * perIter) {
                    unsigned long long f[8];
#pragma unroll
                    for (int k = 0; k < 8; k++) {
                        const size_t L = L0 + (size_t)k * perIter;
                        f[k] = L < lines ? ld_volatile_u64(rs + L * 128 + 120) : rflag;
                    }
#pragma unroll
                    for (int k = 0; k < 8; k++) {
                        const size_t L = L0 + (size_t)k * perIter;
                        if (f[k] != rflag && !fail && !wait_flag64(a, c, rs + L * 128 + 120, rflag, c.recvSeq))
                            fail = true;
                    }
                }
            }
            __threadfence();
            __syncwarp();
        }
        if (!__any_sync(0xFFFFFFFFu, fail)) {
            const int pb = t < 7 ? 16 * t : 112;              // payload byte offset in the line
            const int UEl = t < 7 ? 16 / ESZ : 8 / ESZ;        // elements of this lane
            for (size_t L0 = (size_t)warp * 4 + g; L0 < lines; L0 += (size_t)R * perIter) {
                uint4 v[R], l[R];
#pragma unroll
                for (int k = 0; k < R; k++) {
                    const size_t L = L0 + (size_t)k * perIter;
                    const size_t e0 = (L * 120 + pb) / ESZ;    // first element of this lane
                    v[k] = make_uint4(0u, 0u, 0u, 0u);
                    l[k] = v[k];
                    if (L < lines && e0 < m) {
                        const int ne = (int)min((size_t)UEl, m - e0);
                        if (kind & kRecv) {
                            if (t < 7) v[k] = ld_cg(rs + L * 128 + 16 * t);
                            else { const uint2 d = ld_cg8(rs + L * 128 + 112); v[k].x = d.x; v[k].y = d.y; }
                        }
                        if (kind & kLocal)
                            l[k] = t < 7 ? load_unit<ESZ, 16, 8>(in + e0 * ESZ, ne, aligned)
                                         : load_unit<ESZ, 8, 8>(in + e0 * ESZ, ne, aligned);
                    }
                }
#pragma unroll
                for (int k = 0; k < R; k++) {
                    const size_t L = L0 + (size_t)k * perIter;
                    const size_t e0 = (L * 120 + pb) / ESZ;
                    if (L >= lines || e0 >= m) continue;
                    const int ne = (int)min((size_t)UEl, m - e0);
                    uint4 x = v[k];
                    if (kind & kLocal) x = (kind & kRecv) ? op_vec_rt<DT>(a.op, x, l[k]) : l[k];
                    if (t < 7) {
                        if (kind & kOut)
                            store_unit<DT, OUT, 16, 8>(out + e0 * OSZ, x, ne, aligned, epi, hasScale, a.scale);
                        if (kind & kSend) st_cg(ss + L * 128 + 16 * t, x);
                    } else {
                        if (kind & kOut)
                            store_unit<DT, OUT, 8, 8>(out + e0 * OSZ, x, ne, aligned, epi, hasScale, a.scale);
                        if (kind & kSend) st_cg8(ss + L * 128 + 112, make_uint2(x.x, x.y));
                    }
                }
                test_jitter(a, (unsigned)L0);
            }
            if (kind & kSend) {
                test_jitter(a, 0x5157u);
                __syncwarp();
                __threadfence();
                if (t == 7)
                    for (size_t L = (size_t)warp * 4 + g; L < lines; L += perIter)
                        st_volatile_u64(ss + L * 128 + 120, sflag);
            }
        }
    }
    if (__syncthreads_or(fail)) return false;
    slot_end<PROTO>(a, c, kind);
    return true;
}

// One transfer of n elements of one block: ceil(n / slotElems) slots.
template <int DT, int OUT, int PROTO>
__device__ __forceinline__ bool ring_transfer(const RingArgs& a, RingCtx& c, int kind,
                                              const char* in, char* out, size_t n, bool epi) {
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int OSZ = DTypeOf<OUT>::size;
    for (size_t k = 0; k < n; k += a.slotElems) {
        const size_t m = min(a.slotElems, n - k);
        if (!ring_slot<DT, OUT, PROTO>(a, c, kind, in ? in + k * ESZ : nullptr,
                                       out ? out + k * OSZ : nullptr, m, epi))
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
    c.N = N;
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
            if (!ring_transfer<DT, DT, PROTO>(a, c, kLocal | kSend, mySend + (st + o) * ESZ, nullptr, n, false)) return;
            for (int s = 1; s < N - 1; s++) {
                blk = (r + N - 1 - s) % N;
                n = seg_len(a, ch, blk, o, &st);
                if (!ring_transfer<DT, DT, PROTO>(a, c, kRecv | kLocal | kSend, mySend + (st + o) * ESZ,
                                                  nullptr, n, false)) return;
            }
            n = seg_len(a, ch, r, o, &st);
            if (a.coll == vCollAllReduce) {
                if (!ring_transfer<DT, DT, PROTO>(a, c, kRecv | kLocal | kOut | kSend, mySend + (st + o) * ESZ,
                                                  myRecv + (st + o) * ESZ, n, false)) return;
                // all-gather rounds: receive block (r - i - 1), forward unless last
                for (int i = 0; i < N - 1; i++) {
                    blk = ((r - i - 1) % N + N) % N;
                    n = seg_len(a, ch, blk, o, &st);
                    const int kind = i < N - 2 ? (kRecv | kOut | kSend) : (kRecv | kOut);
                    if (!ring_transfer<DT, DT, PROTO>(a, c, kind, nullptr, myRecv + (st + o) * ESZ, n, false))
                        return;
                }
            } else {
                // block r lands at recv[r][st - r * rc + o] = recv[r][ch * Lc + o]
                const size_t t0 = st - (size_t)r * a.blockElems + o;
                if (!ring_transfer<DT, OUT, PROTO>(a, c, kRecv | kLocal | kOut, mySend + (st + o) * ESZ,
                                                   myRecv + t0 * OSZ, n, epi)) return;
            }
        } else if (a.coll == vCollAllGather) {
            // own block r: copy to recv[r] at block r and send it on
            size_t n = seg_len(a, ch, r, o, &st);
            const size_t inOff = st - (size_t)r * a.blockElems + o;     // within send[r]
            if (!ring_transfer<DT, DT, PROTO>(a, c, kLocal | kOut | kSend, mySend + inOff * ESZ,
                                              myRecv + (st + o) * ESZ, n, false)) return;
            for (int i = 0; i < N - 1; i++) {
                const int blk = ((r - i - 1) % N + N) % N;
                n = seg_len(a, ch, blk, o, &st);
                const int kind = i < N - 2 ? (kRecv | kOut | kSend) : (kRecv | kOut);
                if (!ring_transfer<DT, DT, PROTO>(a, c, kind, nullptr, myRecv + (st + o) * ESZ, n, false))
                    return;
            }
        } else {
            // broadcast: a chain root, root+1, ..., root-1
            const int pos = ((r - a.root) % N + N) % N;
            const size_t n = seg_len(a, ch, 0, o, &st);
            int kind;
            if (pos == 0) kind = kLocal | kOut | kSend;
            else if (pos < N - 1) kind = kRecv | kOut | kSend;
            else kind = kRecv | kOut;
            const char* src = pos == 0 ? (const char*)a.send[a.root] + (st + o) * ESZ : nullptr;
            if (!ring_transfer<DT, DT, PROTO>(a, c, kind, src, myRecv + (st + o) * ESZ, n, false)) return;
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
