// k_group.cu -- group batching: many one-pass all-reduces of one type and op in one
// launch (NCCL book chapter 6: ncclPrepareTasks aggregates collectives of the same
// function, op and type).  The work table arrives in the kernel's parameter block.
#include "reduce_ring.cuh"

namespace vc {

// Batched all-reduces (group batching, NCCL book chapter 6: ncclPrepareTasks aggregates
// collectives of the same function, op and type into one launch).  Every item keeps its
// own block partition and ring order, so its bits equal a separate vAllReduce.  The work
// units of all items form one flat index space; a thread finds its item by binary search
// over the items' first units, held in shared memory.
template <int DT, int OP, int VB>
__global__ void __launch_bounds__(kOnePassThreads, VB == 32 ? 1 : 2)
k_allreduce_group(const __grid_constant__ GroupArgs a) {
    pdl_begin();
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int U = VB ? VB / ESZ : kElemsPerThread;    // a unit: a vector, or 8 elements
    const GroupItem* items = reinterpret_cast<const GroupItem*>(a.table);
    const void* const* ptrs = reinterpret_cast<const void* const*>(a.table + a.ptrByteOff);
    __shared__ unsigned long long sStart[kMaxGroupItems];
    for (int i = threadIdx.x; i < a.nItems; i += blockDim.x) sStart[i] = items[i].unitStart;
    __syncthreads();
    const int N = a.nRanks;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t j = (size_t)blockIdx.x * blockDim.x + threadIdx.x; j < a.totalUnits; j += stride) {
        int lo = 0, hi = a.nItems - 1;                   // last item with unitStart <= j
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sStart[mid] <= j) lo = mid;
            else hi = mid - 1;
        }
        const GroupItem it = items[lo];
        const void* const* send = ptrs + it.ptrOff;
        void* const* recv = (void* const*)(ptrs + it.ptrOff + N);
        const size_t u = j - it.unitStart;
        const int b = (int)(u / it.unitsPerBlock);
        const size_t e = (size_t)b * it.blockElems + (u - (size_t)b * it.unitsPerBlock) * U;
        const size_t bend = min((size_t)((b + 1) * it.blockElems), (size_t)it.count);
        if (e >= bend) continue;
        const int first = b + 1 == N ? 0 : b + 1;
        if (VB && e + U <= bend) {
            const size_t boff = e * ESZ;
            const auto acc = reduce_vec_ring<DT, OP, VB ? VB : 16>(send, N, first, boff);
            for (int r = 0; r < N; r++) VecOf<VB ? VB : 16>::st((char*)recv[r] + boff, acc);
        } else if (VB) {
            for (size_t x = e; x < min(e + U, bend); x++) {
                const uint32_t acc = reduce_elem_ring<DT, OP>(send, N, first, x);
                for (int r = 0; r < N; r++) st_elem<ESZ>(recv[r], x, acc);
            }
        } else {
            // element path: 8 consecutive elements of up to four ranks loaded before folding
            uint32_t acc[kElemsPerThread];
            reduce_elems_ring<DT, OP, 1>(send, N, first, e, bend, acc);
            for (int r = 0; r < N; r++) {
#pragma unroll
                for (int k = 0; k < kElemsPerThread; k++)
                    if (e + k < bend) st_elem<ESZ>(recv[r], e + k, acc[k]);
            }
        }
    }
}

template <int DT, int OP>
static cudaError_t group_dispatch_vec(const GroupArgs& a, int vb, int grid, int threads, cudaStream_t s) {
    if (vb == 32) (void)pdl_launch(k_allreduce_group<DT, OP, 32>, grid, threads, 0, s, a);
    else if (vb == 16) (void)pdl_launch(k_allreduce_group<DT, OP, 16>, grid, threads, 0, s, a);
    else (void)pdl_launch(k_allreduce_group<DT, OP, 0>, grid, threads, 0, s, a);
    return cudaGetLastError();
}

template <int DT>
static cudaError_t group_dispatch_op(const GroupArgs& a, vRedOp_t op, int vb, int grid, int threads,
                                     cudaStream_t s) {
    switch (op) {
    case vSum: return group_dispatch_vec<DT, kSum>(a, vb, grid, threads, s);
    case vProd: return group_dispatch_vec<DT, kProd>(a, vb, grid, threads, s);
    case vMin: return group_dispatch_vec<DT, kMin>(a, vb, grid, threads, s);
    case vMax: return group_dispatch_vec<DT, kMax>(a, vb, grid, threads, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_allreduce_group(const GroupArgs& a, vDataType_t dt, vRedOp_t op, int vb, int grid,
                                   int threads, cudaStream_t s) {
    switch (dt) {
    case vFloat32: return group_dispatch_op<kF32>(a, op, vb, grid, threads, s);
    case vFloat16: return group_dispatch_op<kF16>(a, op, vb, grid, threads, s);
    case vBFloat16: return group_dispatch_op<kBF16>(a, op, vb, grid, threads, s);
    case vInt32: return group_dispatch_op<kI32>(a, op, vb, grid, threads, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace vc
