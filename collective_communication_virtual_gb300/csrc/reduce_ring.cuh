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

}  // namespace vc
