// k_copy.cu -- data-movement collectives: all-gather, broadcast, all-to-all (uniform and
// variable).  They move bytes whatever the data type (NCCL book chapter 6: AllGather and
// Broadcast are issued as ncclInt8), so each kernel is instantiated once per element
// size and once for the 16-byte vector path.
//
// All-gather and broadcast read each source vector once and write it to all N receive
// buffers: (N+1)*S bytes, the minimum.  All-to-all copies each of the N*N blocks once.
#include "device.cuh"

namespace vc {

constexpr int kCopyUnroll = 4;     // vectors in flight per thread in the block copies

// Each kernel flattens a channel's work -- (block, unit) pairs, a unit being 16 bytes on
// the vector path and one element otherwise -- to one index strided over the channel's
// CTAs, kCopyUnroll units per thread at a time (all loads, then all stores).  Only the
// end of a block can cut a vector short; those elements are copied one by one.

// All-gather: block s = send[s][ch range], written to recv[r] + s*sc for every r.
template <int ESZ, bool VEC>
__global__ void __launch_bounds__(kOnePassThreads)
k_allgather_onepass(const __grid_constant__ OnePassArgs a) {
    constexpr int U = VEC ? 16 / ESZ : 1;
    const int N = a.nRanks;
    const int ch = blockIdx.x / a.ctasPerChannel;
    const int cta = blockIdx.x - ch * a.ctasPerChannel;
    const size_t stride = (size_t)a.ctasPerChannel * blockDim.x;
    const size_t sc = a.count;
    const size_t lo = min((size_t)ch * a.chanElems, sc);
    const size_t hi = min((size_t)(ch + 1) * a.chanElems, sc);
    const size_t units = (hi - lo + U - 1) / U;
    const size_t total = units * (size_t)N;
    for (size_t j0 = (size_t)cta * blockDim.x + threadIdx.x; j0 < total; j0 += kCopyUnroll * stride) {
        uint4 v[kCopyUnroll];
        uint32_t sv[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; u++) {
            const size_t j = j0 + u * stride;
            if (j >= total) break;
            const int s = (int)(j / units);
            const size_t e = lo + (j - (size_t)s * units) * U;
            if (VEC && e + U <= hi) v[u] = ld_stream((const char*)a.send[s] + e * ESZ);
            else if (!VEC) sv[u] = ld_elem<ESZ>(a.send[s], e);
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; u++) {
            const size_t j = j0 + u * stride;
            if (j >= total) break;
            const int s = (int)(j / units);
            const size_t e = lo + (j - (size_t)s * units) * U;
            const size_t dOff = (size_t)s * sc + e;
            if (VEC && e + U <= hi) {
                for (int r = 0; r < N; r++) st_stream((char*)a.recv[r] + dOff * ESZ, v[u]);
            } else if (!VEC) {
                for (int r = 0; r < N; r++) st_elem<ESZ>(a.recv[r], dOff, sv[u]);
            } else {
                for (size_t x = e; x < hi; x++) {
                    const uint32_t w = ld_elem<ESZ>(a.send[s], x);
                    for (int r = 0; r < N; r++) st_elem<ESZ>(a.recv[r], (size_t)s * sc + x, w);
                }
            }
        }
    }
}

// Broadcast: recv[r][t] = send[root][t] for all r.
template <int ESZ, bool VEC>
__global__ void __launch_bounds__(kOnePassThreads)
k_broadcast_onepass(const __grid_constant__ OnePassArgs a) {
    constexpr int U = VEC ? 16 / ESZ : 1;
    const int N = a.nRanks;
    const int ch = blockIdx.x / a.ctasPerChannel;
    const int cta = blockIdx.x - ch * a.ctasPerChannel;
    const size_t stride = (size_t)a.ctasPerChannel * blockDim.x;
    const size_t lo = min((size_t)ch * a.chanElems, a.count);
    const size_t hi = min((size_t)(ch + 1) * a.chanElems, a.count);
    const size_t units = (hi - lo + U - 1) / U;
    const char* src = (const char*)a.send[a.root];
    for (size_t j0 = (size_t)cta * blockDim.x + threadIdx.x; j0 < units; j0 += kCopyUnroll * stride) {
        uint4 v[kCopyUnroll];
        uint32_t sv[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; u++) {
            const size_t j = j0 + u * stride;
            if (j >= units) break;
            const size_t e = lo + j * U;
            if (VEC && e + U <= hi) v[u] = ld_stream(src + e * ESZ);
            else if (!VEC) sv[u] = ld_elem<ESZ>(src, e);
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; u++) {
            const size_t j = j0 + u * stride;
            if (j >= units) break;
            const size_t e = lo + j * U;
            if (VEC && e + U <= hi) {
                for (int r = 0; r < N; r++) st_stream((char*)a.recv[r] + e * ESZ, v[u]);
            } else if (!VEC) {
                for (int r = 0; r < N; r++) st_elem<ESZ>(a.recv[r], e, sv[u]);
            } else {
                for (size_t x = e; x < hi; x++) {
                    const uint32_t w = ld_elem<ESZ>(src, x);
                    for (int r = 0; r < N; r++) st_elem<ESZ>(a.recv[r], x, w);
                }
            }
        }
    }
}

// Copy [lo, hi) elements from src to dst with kCopyUnroll vectors in flight per thread.
template <int ESZ, bool VEC>
__device__ __forceinline__ void copy_range(const char* src, char* dst, size_t lo, size_t hi,
                                           size_t tid, size_t stride) {
    if (VEC) {
        constexpr int VE = 16 / ESZ;
        const size_t nv = (hi - lo) / VE;
        size_t i = tid;
        for (; i + (kCopyUnroll - 1) * stride < nv; i += kCopyUnroll * stride) {
            uint4 v[kCopyUnroll];
#pragma unroll
            for (int u = 0; u < kCopyUnroll; u++) v[u] = ld_stream(src + (lo + (i + u * stride) * VE) * ESZ);
#pragma unroll
            for (int u = 0; u < kCopyUnroll; u++) st_stream(dst + (lo + (i + u * stride) * VE) * ESZ, v[u]);
        }
        for (; i < nv; i += stride) st_stream(dst + (lo + i * VE) * ESZ, ld_stream(src + (lo + i * VE) * ESZ));
        const size_t tail = lo + nv * VE;
        if (tail + tid < hi) st_elem<ESZ>(dst, tail + tid, ld_elem<ESZ>(src, tail + tid));
    } else {
        for (size_t e = lo + tid; e < hi; e += stride) st_elem<ESZ>(dst, e, ld_elem<ESZ>(src, e));
    }
}

// Uniform all-to-all: recv[j][i*c + t] = send[i][j*c + t].  a.count = c.  The N*N blocks'
// channel ranges are flattened as p = i*N + j, unit within the range.
template <int ESZ, bool VEC>
__global__ void __launch_bounds__(kOnePassThreads)
k_alltoall_onepass(const __grid_constant__ OnePassArgs a) {
    constexpr int U = VEC ? 16 / ESZ : 1;
    const int N = a.nRanks;
    const int ch = blockIdx.x / a.ctasPerChannel;
    const int cta = blockIdx.x - ch * a.ctasPerChannel;
    const size_t stride = (size_t)a.ctasPerChannel * blockDim.x;
    const size_t c = a.count;
    const size_t lo = min((size_t)ch * a.chanElems, c);
    const size_t hi = min((size_t)(ch + 1) * a.chanElems, c);
    const size_t units = (hi - lo + U - 1) / U;
    const size_t total = units * (size_t)N * (size_t)N;
    for (size_t j0 = (size_t)cta * blockDim.x + threadIdx.x; j0 < total; j0 += kCopyUnroll * stride) {
        uint4 v[kCopyUnroll];
        uint32_t sv[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; u++) {
            const size_t jj = j0 + u * stride;
            if (jj >= total) break;
            const size_t p = jj / units;
            const int i = (int)(p / N), j = (int)(p - (size_t)(p / N) * N);
            const size_t e = lo + (jj - p * units) * U;
            const char* src = (const char*)a.send[i] + (size_t)j * c * ESZ;
            if (VEC && e + U <= hi) v[u] = ld_stream(src + e * ESZ);
            else if (!VEC) sv[u] = ld_elem<ESZ>(src, e);
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; u++) {
            const size_t jj = j0 + u * stride;
            if (jj >= total) break;
            const size_t p = jj / units;
            const int i = (int)(p / N), j = (int)(p - (size_t)(p / N) * N);
            const size_t e = lo + (jj - p * units) * U;
            char* dst = (char*)a.recv[j] + (size_t)i * c * ESZ;
            if (VEC && e + U <= hi) {
                st_stream(dst + e * ESZ, v[u]);
            } else if (!VEC) {
                st_elem<ESZ>(dst, e, sv[u]);
            } else {
                const char* src = (const char*)a.send[i] + (size_t)j * c * ESZ;
                for (size_t x = e; x < hi; x++) st_elem<ESZ>(dst, x, ld_elem<ESZ>(src, x));
            }
        }
    }
}

// Variable all-to-all.  The N*N blocks are cut into tiles of a.tileBytes; tiles are
// numbered across all blocks and dealt to CTAs round-robin, so a hot destination's many
// tiles spread over the whole grid.  Every CTA builds the tile prefix sums in shared
// memory from the device tables.
template <int ESZ>
__global__ void __launch_bounds__(kOnePassThreads)
k_alltoallv(const __grid_constant__ A2AvArgs a) {
    __shared__ unsigned long long tileStart[VCOMM_MAX_RANKS * VCOMM_MAX_RANKS + 1];
    __shared__ int sBad;
    const int N = a.nRanks;
    const int NB = N * N;
    const size_t tileElems = a.tileBytes / ESZ;
    if (threadIdx.x == 0) sBad = 0;
    __syncthreads();
    for (int p = threadIdx.x; p < NB; p += blockDim.x) {
        const int i = p / N, j = p - (p / N) * N;
        const int32_t cnt = a.counts[p], so = a.sdispls[p], ro = a.rdispls[j * N + i];
        unsigned long long tiles = 0;
        if (cnt < 0 || so < 0 || ro < 0) sBad = 1;
        else tiles = ((unsigned long long)cnt + tileElems - 1) / tileElems;
        tileStart[p + 1] = tiles;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        tileStart[0] = 0;
        for (int p = 0; p < NB; p++) tileStart[p + 1] += tileStart[p];
        if (sBad && blockIdx.x == 0) report_error(a.status, a.statusHost, vInvalidArgument, 0, 0, 0);
    }
    __syncthreads();
    const unsigned long long nTiles = tileStart[NB];
    int p = 0;
    for (unsigned long long tile = blockIdx.x; tile < nTiles; tile += gridDim.x) {
        while (tileStart[p + 1] <= tile) p++;          // tiles ascend, so p only grows
        const int i = p / N, j = p - (p / N) * N;
        const size_t cnt = (size_t)a.counts[p];
        const size_t k = tile - tileStart[p];
        const size_t lo = k * tileElems, hi = min(lo + tileElems, cnt);
        const char* src = (const char*)a.send[i] + (size_t)a.sdispls[p] * ESZ;
        char* dst = (char*)a.recv[j] + (size_t)a.rdispls[j * N + i] * ESZ;
        const bool vec = ((((uintptr_t)src) | ((uintptr_t)dst)) & 15) == 0;
        if (vec) copy_range<ESZ, true>(src, dst, lo, hi, threadIdx.x, blockDim.x);
        else copy_range<ESZ, false>(src, dst, lo, hi, threadIdx.x, blockDim.x);
    }
}

// ---- dispatch --------------------------------------------------------------------------

#define VC_COPY_LAUNCH(KERNEL)                                                             \
    do {                                                                                   \
        if (elemSize == 4) {                                                               \
            if (vec) KERNEL<4, true><<<grid, threads, 0, s>>>(a);                          \
            else KERNEL<4, false><<<grid, threads, 0, s>>>(a);                             \
        } else if (elemSize == 2) {                                                        \
            if (vec) KERNEL<2, true><<<grid, threads, 0, s>>>(a);                          \
            else KERNEL<2, false><<<grid, threads, 0, s>>>(a);                             \
        } else {                                                                           \
            return cudaErrorInvalidValue;                                                  \
        }                                                                                  \
        return cudaGetLastError();                                                         \
    } while (0)

cudaError_t launch_allgather_onepass(const OnePassArgs& a, int elemSize, bool vec, int grid,
                                     int threads, cudaStream_t s) {
    VC_COPY_LAUNCH(k_allgather_onepass);
}

cudaError_t launch_broadcast_onepass(const OnePassArgs& a, int elemSize, bool vec, int grid,
                                     int threads, cudaStream_t s) {
    VC_COPY_LAUNCH(k_broadcast_onepass);
}

cudaError_t launch_alltoall_onepass(const OnePassArgs& a, int elemSize, bool vec, int grid,
                                    int threads, cudaStream_t s) {
    VC_COPY_LAUNCH(k_alltoall_onepass);
}

cudaError_t launch_alltoallv(const A2AvArgs& a, int grid, int threads, cudaStream_t s) {
    if (a.elemSize == 4) k_alltoallv<4><<<grid, threads, 0, s>>>(a);
    else if (a.elemSize == 2) k_alltoallv<2><<<grid, threads, 0, s>>>(a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace vc
