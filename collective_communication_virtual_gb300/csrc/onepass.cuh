// onepass.cuh -- one-pass reduction kernels: all-reduce and reduce-scatter, and their
// launch dispatch for a rank count fixed at compile time (NF) or read at run time (NF = 0).
//
// Every virtual rank's buffer is addressable from one kernel, so instead of moving
// partials from rank to rank (2(N-1) ring steps, "NCCL book" section 2.3) each thread
// reads element e of all N ranks once, reduces them in the ring's order, and writes the
// result once per output: 2*N*S bytes for an all-reduce, the minimum.  This is the
// virtual-rank form of the symmetric-memory kernels that read peers' buffers directly
// (NCCL book chapter 5 section 5; "AI Systems Performance Engineering (3)", NVLS and
// symmetric memory).
//
// Order: block b of the buffer is reduced as ranks b+1, b+2, ..., b (mod N), each partial
// rounded to the data type -- exactly the partial a ring reduce-scatter accumulates
// (RingARAlgorithm::getNextSendAddr: at stage s rank r handles chunk (r + N - 1 - s) mod N).
// Channels own contiguous sub-ranges of every block (NCCL book section 2.2); a channel's
// CTAs stride over its sub-range.  Blocks, channel ranges and 16-byte vectors all start
// on 16-byte boundaries, so a vector never straddles two blocks.
#pragma once

#include "reduce_ring.cuh"

namespace vc {

// Element e of a 16-byte vector held as four 32-bit words (2- or 4-byte elements).
template <int ESZ>
__device__ __forceinline__ uint32_t vec_elem(const uint32_t (&w)[4], int e) {
    return ESZ == 4 ? w[e] : (w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
}

// Per channel the work is (block, unit) pairs, flattened so that small buffers still
// spread over all threads: unit i of block b covers elements [lo_b + i*U, lo_b + (i+1)*U)
// with U = 16 / esz on the vector path (1 otherwise) and lo_b = b*B + ch*Lc.  Only the
// very end of the buffer can cut a vector short; its elements go element by element.
struct ChannelSpan {
    size_t lo;       // first element of this channel's range in block 0
    size_t units;    // units per block (of the full-length range)
};

__device__ __forceinline__ ChannelSpan channel_span(const OnePassArgs& a, int ch, size_t unit) {
    ChannelSpan s;
    const size_t lo = min((size_t)ch * a.chanElems, a.blockElems);
    const size_t hi = min((size_t)(ch + 1) * a.chanElems, a.blockElems);
    s.lo = lo;
    s.units = (hi - lo + unit - 1) / unit;
    return s;
}

// The all-reduce element path for 2-byte types whose outputs all sit at one offset from a
// 16-byte boundary: 16-byte vectors aligned to the outputs, cut from the inputs
// (reduce_vec_ring_realign).  A (block, channel) range has one item per vector plus item 0,
// which takes the elements before the first output boundary and after the last vector.
template <int DT, int OP>
__device__ __forceinline__ void allreduce_realigned16(const OnePassArgs& a, int N, int ch, int cta, size_t stride,
                                                      size_t chEnd, int r0, int r1) {
    constexpr int ESZ = DTypeOf<DT>::size;
    const size_t lo = min((size_t)ch * a.chanElems, a.blockElems);
    const size_t items = (chEnd - lo) / 8 + 2;
    for (size_t j = (size_t)cta * blockDim.x + threadIdx.x; j < items * (size_t)N; j += stride) {
        const int b = (int)(j / items);
        const size_t i = j - (size_t)b * items;
        const size_t base = (size_t)b * a.blockElems;
        const size_t x0 = base + lo, x1 = min(base + chEnd, a.count);
        if (x0 >= x1) continue;
        const uintptr_t d0 = (uintptr_t)((const char*)a.recv[r0] + x0 * ESZ);
        const size_t head = min((size_t)(((16u - (d0 & 15u)) & 15u) / ESZ), x1 - x0);
        const size_t nv = (x1 - x0 - head) / 8;
        const int ob = a.orderRoot >= 0 ? a.orderRoot : b;
        const int first = ob + 1 == N ? 0 : ob + 1;
        if (i == 0) {
            for (size_t x = x0; x < x1; x++) {
                if (x == x0 + head) x += 8 * nv;
                if (x >= x1) break;
                const uint32_t acc = reduce_elem_ring<DT, OP>(a.send, N, first, x);
                for (int r = r0; r < r1; r++) st_elem<ESZ>(a.recv[r], x, acc);
            }
        } else if (i - 1 < nv) {
            const size_t e = x0 + head + 8 * (i - 1);
            const uint4 acc = reduce_vec_ring_realign<DT, OP>(a.send, N, first, e * ESZ);
            for (int r = r0; r < r1; r++) st_stream((char*)a.recv[r] + e * ESZ, acc);
        }
    }
}

// All-reduce, and reduce to root.  grid = nChannels * ctasPerChannel.  VB: 0 (element
// path), 16 or 32 bytes per vector; the 32-byte kernel keeps twice the registers, so it
// runs one 512-thread CTA per SM instead of two.  Reduce to root (a.orderRoot = a.outRoot
// = root) reduces every block in the root's order and writes only recv[root].
template <int DT, int OP, int VB, int NF = 0>
__global__ void __launch_bounds__(kOnePassThreads, VB == 32 ? 1 : 2)
k_allreduce_onepass(const __grid_constant__ OnePassArgs a) {
    pdl_begin();
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int U = VB ? VB / ESZ : 1;
    const int N = NF ? NF : a.nRanks;
    const int ch = blockIdx.x / a.ctasPerChannel;
    const int cta = blockIdx.x - ch * a.ctasPerChannel;
    const size_t stride = (size_t)a.ctasPerChannel * blockDim.x;
    const size_t chEnd = min((size_t)(ch + 1) * a.chanElems, a.blockElems);
    const int r0 = a.outRoot >= 0 ? a.outRoot : 0;
    const int r1 = a.outRoot >= 0 ? a.outRoot + 1 : N;
    if constexpr (VB == 0 && ESZ == 2) {
        bool sameOut = true;       // every output at the same offset from a 16-byte boundary
        for (int r = r0 + 1; r < r1; r++)
            sameOut = sameOut && ((((uintptr_t)a.recv[r]) ^ (uintptr_t)a.recv[r0]) & 15u) == 0;
        if (sameOut) {
            allreduce_realigned16<DT, OP>(a, N, ch, cta, stride, chEnd, r0, r1);
            return;
        }
    }
    if (VB == 0) {
        // element path: warp tiles of 32 * kElemsPerThread elements of one block
        constexpr int TILE = 32 * kElemsPerThread;
        const size_t lo = min((size_t)ch * a.chanElems, a.blockElems);
        const size_t tiles = (chEnd - lo + TILE - 1) / TILE;
        const int lane = threadIdx.x & 31;
        for (size_t w = ((size_t)cta * blockDim.x + threadIdx.x) / 32; w < tiles * (size_t)N; w += stride / 32) {
            const int b = (int)(w / tiles);
            const size_t base = (size_t)b * a.blockElems;
            const size_t e0 = base + lo + (w - (size_t)b * tiles) * TILE + lane;
            const size_t end = min(base + chEnd, a.count);
            const int ob = a.orderRoot >= 0 ? a.orderRoot : b;
            uint32_t acc[kElemsPerThread];
            reduce_elems_ring<DT, OP>(a.send, N, ob + 1 == N ? 0 : ob + 1, e0, end, acc);
            for (int r = r0; r < r1; r++) {
#pragma unroll
                for (int k = 0; k < kElemsPerThread; k++)
                    if (e0 + 32 * (size_t)k < end) st_elem<ESZ>(a.recv[r], e0 + 32 * (size_t)k, acc[k]);
            }
        }
        return;
    }
    const ChannelSpan sp = channel_span(a, ch, U);
    const size_t total = sp.units * (size_t)N;
    for (size_t j = (size_t)cta * blockDim.x + threadIdx.x; j < total; j += stride) {
        const int b = (int)(j / sp.units);
        const size_t i = j - (size_t)b * sp.units;
        const size_t base = (size_t)b * a.blockElems;
        const size_t e = base + sp.lo + i * U;
        const size_t hi = min(base + chEnd, a.count);
        if (e >= hi) continue;
        const int ob = a.orderRoot >= 0 ? a.orderRoot : b;
        const int first = ob + 1 == N ? 0 : ob + 1;
        if (VB && e + U <= hi) {
            const size_t boff = e * ESZ;
            const auto acc = reduce_vec_ring<DT, OP, VB ? VB : 16, NF>(a.send, N, first, boff);
            if (NF && a.outRoot < 0) {
#pragma unroll
                for (int r = 0; r < (NF ? NF : 1); r++) VecOf<VB ? VB : 16>::st((char*)a.recv[r] + boff, acc);
            } else {
                for (int r = r0; r < r1; r++) VecOf<VB ? VB : 16>::st((char*)a.recv[r] + boff, acc);
            }
        } else {
            for (size_t x = e; x < min(e + U, hi); x++) {
                const uint32_t acc = reduce_elem_ring<DT, OP>(a.send, N, first, x);
                for (int r = r0; r < r1; r++) st_elem<ESZ>(a.recv[r], x, acc);
            }
        }
    }
}

// Store a reduced 16-byte vector of DT elements as OUT elements, out = (float)acc * scale
// when hasScale (or a plain store when OUT == DT and no scale).
template <int DT, int OUT>
__device__ __forceinline__ void store_epilogue_vec(void* outBase, size_t outElem, uint4 acc,
                                                   bool hasScale, float scale) {
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int OSZ = DTypeOf<OUT>::size;
    if (DT == OUT && !hasScale) {
        st_stream((char*)outBase + outElem * OSZ, acc);
        return;
    }
    constexpr int VE = 16 / ESZ;
    uint32_t w[4] = {acc.x, acc.y, acc.z, acc.w};
    uint32_t o[VE];
#pragma unroll
    for (int i = 0; i < VE; i++) {
        const uint32_t bits = ESZ == 4 ? w[i] : ((w[i / 2] >> (16 * (i & 1))) & 0xFFFFu);
        float f = elem_to_f32<DT>(bits);
        if (hasScale) f = __fmul_rn(f, scale);
        o[i] = f32_to_elem<OUT>(f);
    }
    if (OSZ == 4) {
#pragma unroll
        for (int q = 0; q < VE / 4; q++)
            st_stream((char*)outBase + (outElem + 4 * q) * 4,
                      make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]));
    } else {
        st_stream((char*)outBase + outElem * 2,
                  make_uint4(o[0] | (o[1] << 16), o[2] | (o[3] << 16), o[4] | (o[5] << 16),
                             o[6] | (o[7] << 16)));
    }
}

template <int DT, int OUT>
__device__ __forceinline__ void store_epilogue_vec(void* outBase, size_t outElem, const V32& acc,
                                                   bool hasScale, float scale) {
    constexpr int VE = 16 / DTypeOf<DT>::size;
    if (DT == OUT && !hasScale) {
        st_stream32((char*)outBase + outElem * DTypeOf<DT>::size, acc);
        return;
    }
    store_epilogue_vec<DT, OUT>(outBase, outElem, acc.lo, hasScale, scale);
    store_epilogue_vec<DT, OUT>(outBase, outElem + VE, acc.hi, hasScale, scale);
}

template <int DT, int OUT>
__device__ __forceinline__ void store_epilogue_elem(void* outBase, size_t outElem, uint32_t acc,
                                                    bool hasScale, float scale) {
    constexpr int OSZ = DTypeOf<OUT>::size;
    if (DT == OUT && !hasScale) {
        st_elem<OSZ>(outBase, outElem, acc);
        return;
    }
    float f = elem_to_f32<DT>(acc);
    if (hasScale) f = __fmul_rn(f, scale);
    st_elem<OSZ>(outBase, outElem, f32_to_elem<OUT>(f));
}

// Reduce-scatter: block r = [r*rc, (r+1)*rc) of every send buffer lands in recv[r].
// a.count = N * rc, a.blockElems = rc.  VB > 0 requires rc * esz % VB == 0.  NF > 0 fixes
// the rank count at compile time (the loads and the fold unroll completely).
template <int DT, int OP, int OUT, int VB, int NF = 0>
__global__ void __launch_bounds__(kOnePassThreads, VB == 32 ? 1 : 2)
k_reduce_scatter_onepass(const __grid_constant__ OnePassArgs a) {
    pdl_begin();
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int U = VB ? VB / ESZ : 1;
    const int N = NF ? NF : a.nRanks;
    const int ch = blockIdx.x / a.ctasPerChannel;
    const int cta = blockIdx.x - ch * a.ctasPerChannel;
    const size_t stride = (size_t)a.ctasPerChannel * blockDim.x;
    const size_t rc = a.blockElems;
    const bool hasScale = a.hasScale != 0;
    const size_t chEnd = min((size_t)(ch + 1) * a.chanElems, rc);
    if constexpr (VB == 0 && NF > 0 && (ESZ == 2 || NF <= 4)) {
        // Blocks off 16 bytes (a ragged block), 2 to 4 ranks (and 8 of 2-byte elements): 16-byte vectors aligned
        // to the inputs, which every rank shares when its buffer starts on a 16-byte boundary,
        // so the loads are those of the vector path.  Warp tiles of 32 x K vectors of one block
        // (lane l takes vectors 32 k + l), so the block arithmetic is done once a tile; the
        // last tile of a (block, channel) range also takes the elements before the first
        // input boundary (the head) and after the last whole vector (the tail).  The
        // outputs sit at one offset from 16 bytes per block: a lane stores the aligned 16
        // bytes made of its vector's last bytes and the next vector's first (a shuffle), so
        // only the edges of a tile go element by element; outputs with an epilogue go
        // element by element.
        constexpr int K = NF <= 4 ? 4 : 1;
        constexpr int VE = 16 / ESZ;                                 // elements per vector
        const size_t lo = min((size_t)ch * a.chanElems, rc);
        const size_t span = chEnd - lo;
        const size_t tiles = span / VE / (32 * K) + 1;
        const bool plainOut = OUT == DT && !hasScale;
        const unsigned int lane = threadIdx.x & 31u;
        for (size_t w = ((size_t)cta * blockDim.x + threadIdx.x) / 32; w < tiles * (size_t)N; w += stride / 32) {
            const int r = (int)(w / tiles);
            const size_t tl = w - (size_t)r * tiles;
            const size_t base = (size_t)r * rc;
            const int first = r + 1 == N ? 0 : r + 1;
            const uintptr_t s0 = (uintptr_t)a.send[first] + (base + lo) * ESZ;
            const size_t head = min((size_t)(((16u - (s0 & 15u)) & 15u) / ESZ), span);
            const size_t nv = (span - head) / VE;
            const size_t b0 = (base + lo + head) * ESZ;              // byte offset of vector 0
            bool aligned = true;
            for (int k = 0; k < N; k++) aligned = aligned && (((uintptr_t)a.send[k] + b0) & 15u) == 0;
            const size_t v0 = tl * (32 * K) + lane;                   // this lane's first vector
            if (aligned) {
                uint4 acc[K];
#pragma unroll
                for (int k = 0; k < K; k++) {
                    const size_t v = v0 + 32 * k;
                    acc[k] = v < nv ? reduce_vec_ring<DT, OP, 16, NF>(a.send, N, first, b0 + 16 * v)
                                    : make_uint4(0u, 0u, 0u, 0u);
                }
                char* out = (char*)a.recv[r] + (lo + head) * ESZ;         // vector v lands at out + 16 v
                const unsigned int d = (unsigned int)((uintptr_t)out & 15u);
#pragma unroll
                for (int k = 0; k < K; k++) {
                    const size_t v = v0 + 32 * k;
                    const uint32_t wd[4] = {acc[k].x, acc[k].y, acc[k].z, acc[k].w};
                    if (plainOut && d != 0) {
                        // lane l + 1 holds vector v + 1 (lane 0 of the next k for lane 31)
                        const uint4 src = (lane == 0 && k + 1 < K) ? acc[k + 1] : acc[k];
                        uint4 nx;
                        nx.x = __shfl_sync(0xFFFFFFFFu, src.x, (lane + 1) & 31u);
                        nx.y = __shfl_sync(0xFFFFFFFFu, src.y, (lane + 1) & 31u);
                        nx.z = __shfl_sync(0xFFFFFFFFu, src.z, (lane + 1) & 31u);
                        nx.w = __shfl_sync(0xFFFFFFFFu, src.w, (lane + 1) & 31u);
                        if (v < nv) {
                            const bool nextHere = v + 1 < nv && !(lane == 31u && k == K - 1);
                            const bool prevHere = !(lane == 0u && k == 0);     // v - 1 >= the tile's first
                            const unsigned int split = (16u - d) / ESZ;         // elements before the boundary
                            char* o = out + 16 * v;
                            if (nextHere) st_stream(o + (16u - d), shift_bytes(acc[k], nx, 16u - d));
#pragma unroll
                            for (int e = 0; e < VE; e++)
                                if ((e < (int)split && !prevHere) || (e >= (int)split && !nextHere))
                                    st_elem<ESZ>(o, e, vec_elem<ESZ>(wd, e));
                        }
                    } else if (v < nv) {
                        if (plainOut) {
                            st_stream(out + 16 * v, acc[k]);
                        } else {
#pragma unroll
                            for (int e = 0; e < VE; e++)
                                store_epilogue_elem<DT, OUT>(a.recv[r], lo + head + VE * v + e, vec_elem<ESZ>(wd, e),
                                                             hasScale, a.scale);
                        }
                    }
                }
            } else {
                // the ranks' blocks at different offsets from 16 bytes: element by element
#pragma unroll
                for (int k = 0; k < K; k++) {
                    const size_t v = v0 + 32 * k;
                    if (v >= nv) continue;
                    for (int e = 0; e < VE; e++) {
                        const size_t t = lo + head + VE * v + e;
                        const uint32_t x = reduce_elem_ring<DT, OP>(a.send, N, first, base + t);
                        store_epilogue_elem<DT, OUT>(a.recv[r], t, x, hasScale, a.scale);
                    }
                }
            }
            if (tl == tiles - 1) {
                // the head (lanes 0..7) and the tail (lanes 8..15), fewer than VE elements each
                const size_t tail = span - head - VE * nv;
                size_t t = ~(size_t)0;
                if (lane < head) t = lo + lane;
                else if (lane >= 8u && lane - 8u < tail) t = lo + head + VE * nv + (lane - 8u);
                if (t != ~(size_t)0) {
                    const uint32_t x = reduce_elem_ring<DT, OP>(a.send, N, first, base + t);
                    store_epilogue_elem<DT, OUT>(a.recv[r], t, x, hasScale, a.scale);
                }
            }
        }
        return;
    }
    if constexpr (VB == 0 && ESZ == 2) {
        // (the run-time rank count: one vector per thread)
        // 2-byte blocks off 16 bytes (a ragged block): 16-byte vectors aligned to the
        // inputs, which every rank shares when its buffer starts on a 16-byte boundary, so
        // the loads are those of the vector path; the 8 results are stored one by one (the
        // outputs are 1/N of the traffic).  Item 0 of a (block, channel) range takes the
        // elements before the first input boundary and after the last whole vector.
        const size_t lo = min((size_t)ch * a.chanElems, rc);
        const size_t span = chEnd - lo;
        const size_t items = span / 8 + 2;
        for (size_t j = (size_t)cta * blockDim.x + threadIdx.x; j < items * (size_t)N; j += stride) {
            const int r = (int)(j / items);
            const size_t i = j - (size_t)r * items;
            const size_t base = (size_t)r * rc;
            const int first = r + 1 == N ? 0 : r + 1;
            const uintptr_t s0 = (uintptr_t)a.send[first] + (base + lo) * ESZ;
            const size_t head = min((size_t)(((16u - (s0 & 15u)) & 15u) / ESZ), span);
            const size_t nv = (span - head) / 8;
            if (i == 0) {
                for (size_t t = lo; t < chEnd; t++) {
                    if (t == lo + head) t += 8 * nv;
                    if (t >= chEnd) break;
                    const uint32_t acc = reduce_elem_ring<DT, OP>(a.send, N, first, base + t);
                    store_epilogue_elem<DT, OUT>(a.recv[r], t, acc, hasScale, a.scale);
                }
            } else if (i - 1 < nv) {
                const size_t t = lo + head + 8 * (i - 1);
                const size_t boff = (base + t) * ESZ;
                bool aligned = true;
                for (int k = 0; k < N; k++) aligned = aligned && (((uintptr_t)a.send[k] + boff) & 15u) == 0;
                if (aligned) {
                    const uint4 acc = reduce_vec_ring<DT, OP, 16>(a.send, N, first, boff);
                    const uint32_t w[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                    for (int k = 0; k < 8; k++)
                        store_epilogue_elem<DT, OUT>(a.recv[r], t + k, (w[k >> 1] >> (16 * (k & 1))) & 0xFFFFu,
                                                     hasScale, a.scale);
                } else {
                    for (int k = 0; k < 8; k++) {
                        const uint32_t acc = reduce_elem_ring<DT, OP>(a.send, N, first, base + t + k);
                        store_epilogue_elem<DT, OUT>(a.recv[r], t + k, acc, hasScale, a.scale);
                    }
                }
            }
        }
        return;
    }
    if (VB == 0) {
        // element path: warp tiles of 32 * kElemsPerThread elements of one block
        constexpr int TILE = 32 * kElemsPerThread;
        const size_t lo = min((size_t)ch * a.chanElems, rc);
        const size_t tiles = (chEnd - lo + TILE - 1) / TILE;
        const int lane = threadIdx.x & 31;
        for (size_t w = ((size_t)cta * blockDim.x + threadIdx.x) / 32; w < tiles * (size_t)N; w += stride / 32) {
            const int r = (int)(w / tiles);
            const size_t t0 = lo + (w - (size_t)r * tiles) * TILE + lane;    // element within block r
            const size_t base = (size_t)r * rc;
            uint32_t acc[kElemsPerThread];
            reduce_elems_ring<DT, OP>(a.send, N, r + 1 == N ? 0 : r + 1, base + t0, base + chEnd, acc);
#pragma unroll
            for (int k = 0; k < kElemsPerThread; k++)
                if (t0 + 32 * (size_t)k < chEnd)
                    store_epilogue_elem<DT, OUT>(a.recv[r], t0 + 32 * (size_t)k, acc[k], hasScale, a.scale);
        }
        return;
    }
    const ChannelSpan sp = channel_span(a, ch, U);
    const size_t total = sp.units * (size_t)N;
    for (size_t j = (size_t)cta * blockDim.x + threadIdx.x; j < total; j += stride) {
        const int r = (int)(j / sp.units);
        const size_t i = j - (size_t)r * sp.units;
        const size_t t = sp.lo + i * U;                 // element within block r
        if (t >= chEnd) continue;
        const size_t base = (size_t)r * rc;
        const int first = r + 1 == N ? 0 : r + 1;
        if (VB && t + U <= chEnd) {
            const auto acc = reduce_vec_ring<DT, OP, VB ? VB : 16, NF>(a.send, N, first, (base + t) * ESZ);
            store_epilogue_vec<DT, OUT>(a.recv[r], t, acc, hasScale, a.scale);
        } else {
            for (size_t x = t; x < min(t + U, chEnd); x++) {
                const uint32_t acc = reduce_elem_ring<DT, OP>(a.send, N, first, base + x);
                store_epilogue_elem<DT, OUT>(a.recv[r], x, acc, hasScale, a.scale);
            }
        }
    }
}

// ---- dispatch --------------------------------------------------------------------------
// Kernels with a compile-time rank count (NF > 0) exist for the vector paths only; the
// element path always takes the run-time kernel.

template <int DT, int OP, int NF>
static cudaError_t ar_launch_vec(const OnePassArgs& a, int vb, int grid, int threads, cudaStream_t s) {
    if (vb == 32) (void)pdl_launch(k_allreduce_onepass<DT, OP, 32, NF>, grid, threads, 0, s, a);
    else if (vb == 16) (void)pdl_launch(k_allreduce_onepass<DT, OP, 16, NF>, grid, threads, 0, s, a);
    else if constexpr (NF == 0) (void)pdl_launch(k_allreduce_onepass<DT, OP, 0>, grid, threads, 0, s, a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

template <int DT, int NF>
static cudaError_t ar_launch_op(const OnePassArgs& a, vRedOp_t op, int vb, int grid, int threads,
                                cudaStream_t s) {
    switch (op) {
    case vSum: return ar_launch_vec<DT, kSum, NF>(a, vb, grid, threads, s);
    case vProd: return ar_launch_vec<DT, kProd, NF>(a, vb, grid, threads, s);
    case vMin: return ar_launch_vec<DT, kMin, NF>(a, vb, grid, threads, s);
    case vMax: return ar_launch_vec<DT, kMax, NF>(a, vb, grid, threads, s);
    }
    return cudaErrorInvalidValue;
}

template <int NF>
static cudaError_t ar_launch(const OnePassArgs& a, vDataType_t dt, vRedOp_t op, int vb, int grid, int threads,
                             cudaStream_t s) {
    switch (dt) {
    case vFloat32: return ar_launch_op<kF32, NF>(a, op, vb, grid, threads, s);
    case vFloat16: return ar_launch_op<kF16, NF>(a, op, vb, grid, threads, s);
    case vBFloat16: return ar_launch_op<kBF16, NF>(a, op, vb, grid, threads, s);
    case vInt32: return ar_launch_op<kI32, NF>(a, op, vb, grid, threads, s);
    }
    return cudaErrorInvalidValue;
}

template <int DT, int OP, int OUT, int NF>
static cudaError_t rs_launch_vec(const OnePassArgs& a, int vb, int grid, int threads, cudaStream_t s) {
    if (vb == 32) (void)pdl_launch(k_reduce_scatter_onepass<DT, OP, OUT, 32, NF>, grid, threads, 0, s, a);
    else if (vb == 16) (void)pdl_launch(k_reduce_scatter_onepass<DT, OP, OUT, 16, NF>, grid, threads, 0, s, a);
    else (void)pdl_launch(k_reduce_scatter_onepass<DT, OP, OUT, 0, NF>, grid, threads, 0, s, a);
    return cudaGetLastError();
}

template <int DT, int OUT, int NF>
static cudaError_t rs_launch_op(const OnePassArgs& a, vRedOp_t op, int vb, int grid, int threads,
                                cudaStream_t s) {
    switch (op) {
    case vSum: return rs_launch_vec<DT, kSum, OUT, NF>(a, vb, grid, threads, s);
    case vProd: return rs_launch_vec<DT, kProd, OUT, NF>(a, vb, grid, threads, s);
    case vMin: return rs_launch_vec<DT, kMin, OUT, NF>(a, vb, grid, threads, s);
    case vMax: return rs_launch_vec<DT, kMax, OUT, NF>(a, vb, grid, threads, s);
    }
    return cudaErrorInvalidValue;
}

template <int NF>
static cudaError_t rs_launch(const OnePassArgs& a, vDataType_t dt, vRedOp_t op, vDataType_t outType, int vb,
                             int grid, int threads, cudaStream_t s) {
    const bool toF32 = outType == vFloat32 && dt != vFloat32;
    if (outType != dt && !toF32) return cudaErrorInvalidValue;
    switch (dt) {
    case vFloat32: return rs_launch_op<kF32, kF32, NF>(a, op, vb, grid, threads, s);
    case vFloat16:
        return toF32 ? rs_launch_op<kF16, kF32, NF>(a, op, vb, grid, threads, s)
                     : rs_launch_op<kF16, kF16, NF>(a, op, vb, grid, threads, s);
    case vBFloat16:
        return toF32 ? rs_launch_op<kBF16, kF32, NF>(a, op, vb, grid, threads, s)
                     : rs_launch_op<kBF16, kBF16, NF>(a, op, vb, grid, threads, s);
    case vInt32: return rs_launch_op<kI32, kI32, NF>(a, op, vb, grid, threads, s);
    }
    return cudaErrorInvalidValue;
}

// The 2-, 3- and 4-rank vector kernels (k_onepass_small.cu).
cudaError_t launch_allreduce_onepass_small(const OnePassArgs& a, vDataType_t dt, vRedOp_t op, int vb, int grid,
                                           int threads, cudaStream_t s);
cudaError_t launch_reduce_scatter_onepass_small(const OnePassArgs& a, vDataType_t dt, vRedOp_t op,
                                                vDataType_t outType, int vb, int grid, int threads,
                                                cudaStream_t s);

}  // namespace vc
