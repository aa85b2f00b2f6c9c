// reduce_ring.cuh -- reduction of one element (or one vector) of every virtual rank in
// the ring's order: block b is reduced as ranks b+1, b+2, ..., b (mod N), each partial
// rounded to the data type, exactly the partial a ring reduce-scatter accumulates
// (RingARAlgorithm::getNextSendAddr, NCCL book section 2.3: at stage s rank r handles
// chunk (r + N - 1 - s) mod N).  Shared by the one-pass and the batched kernels.
#pragma once

#include "device.cuh"

namespace vc {

// Load the VB-byte vector at byte offset `boff` of every rank, starting at rank `first`
// and wrapping, and reduce in that order.  Up to 8 loads are in flight before the first use.
template <int DT, int OP, int VB, int NF = 0>
__device__ __forceinline__ typename VecOf<VB>::T reduce_vec_ring(const void* const* send, int Nrt,
                                                                int first, size_t boff) {
    using VT = typename VecOf<VB>::T;
    const int N = NF ? NF : Nrt;
    if (NF) {
        // rank count known at compile time: all loads issued, then the fold, unrolled
        VT v[NF ? NF : 1];
#pragma unroll
        for (int k = 0; k < NF; k++) {
            const int rk = first + k >= NF ? first + k - NF : first + k;
            v[k] = VecOf<VB>::ld((const char*)send[rk] + boff);
        }
        VT acc = v[0];
#pragma unroll
        for (int k = 1; k < NF; k++) acc = op_vec<DT, OP>(acc, v[k]);
        return acc;
    }
    VT acc = VecOf<VB>::ld((const char*)send[first] + boff);
    int rk = first + 1 == N ? 0 : first + 1;
    for (int k = 1; k < N; k += 8) {
        VT v[8];
#pragma unroll
        for (int j = 0; j < 8; j++) {
            if (k + j < N) {
                v[j] = VecOf<VB>::ld((const char*)send[rk] + boff);
                rk = rk + 1 == N ? 0 : rk + 1;
            }
        }
#pragma unroll
        for (int j = 0; j < 8; j++)
            if (k + j < N) acc = op_vec<DT, OP>(acc, v[j]);
    }
    return acc;
}

// Element path (pointers or blocks that 16-byte vectors cannot cover): a warp reduces 32*K
// consecutive elements, lane l taking elements e0 + 32*k (k < K, e0 = tile start + l), so
// every load and store instruction of the warp is coalesced.  The K elements of up to four
// ranks are loaded before any is folded: plain element loads cannot be moved past the
// stores by the compiler, so one element at a time would wait out a full memory latency
// per rank.  Elements at or beyond `end` are neither loaded nor used.
// STRIDE: element spacing of a thread's K elements (32: warp tiles; 1: K consecutive).
template <int DT, int OP, int STRIDE = 32>
__device__ __forceinline__ void reduce_elems_ring(const void* const* send, int N, int first, size_t e0,
                                                  size_t end, uint32_t (&acc)[kElemsPerThread]) {
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int K = kElemsPerThread;
#pragma unroll
    for (int k = 0; k < K; k++) {
        const size_t e = e0 + STRIDE * (size_t)k;
        acc[k] = e < end ? ld_elem<ESZ>(send[first], e) : 0u;
    }
    int rk = first + 1 == N ? 0 : first + 1;
    for (int n = 1; n < N; n += 4) {
        uint32_t v[4][K];
#pragma unroll
        for (int j = 0; j < 4; j++) {
            if (n + j < N) {
#pragma unroll
                for (int k = 0; k < K; k++) {
                    const size_t e = e0 + STRIDE * (size_t)k;
                    v[j][k] = e < end ? ld_elem<ESZ>(send[rk], e) : 0u;
                }
                rk = rk + 1 == N ? 0 : rk + 1;
            }
        }
#pragma unroll
        for (int j = 0; j < 4; j++) {
            if (n + j < N) {
#pragma unroll
                for (int k = 0; k < K; k++) acc[k] = op_elem<DT, OP>(acc[k], v[j][k]);
            }
        }
    }
}

template <int DT, int OP>
__device__ __forceinline__ uint32_t reduce_elem_ring(const void* const* send, int N, int first, size_t e) {
    constexpr int ESZ = DTypeOf<DT>::size;
    uint32_t acc = ld_elem<ESZ>(send[first], e);
    int rk = first + 1 == N ? 0 : first + 1;
    for (int k = 1; k < N; k++) {
        acc = op_elem<DT, OP>(acc, ld_elem<ESZ>(send[rk], e));
        rk = rk + 1 == N ? 0 : rk + 1;
    }
    return acc;
}

// 16 bytes at byte offset `boff` of every rank, reduced in ring order from rank `first`,
// for offsets that need not be 16-byte aligned: each rank's bytes are cut from the two
// aligned 16-byte blocks that hold them.  The second block always holds some of the 16
// bytes, so no load leaves the aligned blocks of the reduced range.  When every rank sits
// at the same offset from a 16-byte boundary (the usual case: equally aligned buffers) the
// loads are unconditional, so four ranks' loads are in flight before any is folded.
template <int DT, int OP, typename Load>
__device__ __forceinline__ uint4 fold_ring4(int N, int first, Load load) {
    uint4 acc = load(first);
    int rk = first + 1 == N ? 0 : first + 1;
    for (int k = 1; k < N; k += 4) {
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
            if (k + j < N) {
                v[j] = load(rk);
                rk = rk + 1 == N ? 0 : rk + 1;
            }
        }
#pragma unroll
        for (int j = 0; j < 4; j++)
            if (k + j < N) acc = op_vec<DT, OP>(acc, v[j]);
    }
    return acc;
}

template <int DT, int OP>
__device__ __forceinline__ uint4 reduce_vec_ring_realign(const void* const* send, int N, int first, size_t boff) {
    const unsigned sh = (unsigned)(((uintptr_t)send[first] + boff) & 15u);
    bool uniform = true;
    for (int k = 0; k < N; k++) uniform = uniform && (unsigned)(((uintptr_t)send[k] + boff) & 15u) == sh;
    if (!uniform) {
        // ranks at different offsets from a 16-byte boundary: element by element
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        constexpr int ESZ = DTypeOf<DT>::size;
        for (int i = 0; i < 16 / ESZ; i++) {
            const uint32_t e = reduce_elem_ring<DT, OP>(send, N, first, boff / ESZ + i);
            if (ESZ == 4) w[i] = e;
            else w[i >> 1] |= e << (16 * (i & 1));
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (sh == 0)
        return fold_ring4<DT, OP>(N, first, [&](int rk) { return ld_stream((const char*)send[rk] + boff); });
    return fold_ring4<DT, OP>(N, first, [&](int rk) {
        const uint4* q = reinterpret_cast<const uint4*>((const char*)send[rk] + boff - sh);
        return shift_bytes(q[0], q[1], sh);
    });
}

}  // namespace vc
