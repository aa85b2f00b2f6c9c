// k_copy.cu -- data-movement collectives: all-gather, broadcast, all-to-all (uniform and
// variable).  They move bytes whatever the data type (NCCL book chapter 6: AllGather and
// Broadcast are issued as ncclInt8), so each kernel is instantiated once per element
// size and once for the 16-byte vector path; 2-byte copies off 16 bytes have kernels of
// their own (k_*_ragged16).
//
// All-gather and broadcast read each source vector once and write it to all N receive
// buffers: (N+1)*S bytes, the minimum.  All-to-all copies each of the N*N blocks once.
#include <type_traits>

#include "device.cuh"

namespace vc {

// The copy kernels deal tiles (2 to 64 KiB, and CTAs of 64 to 512 threads, chosen by the
// planner) of a channel's block ranges to the channel's CTAs round-robin -- with the
// default flat grid, one tile per CTA: tile t covers elements [lo + k*T, lo + (k+1)*T) of
// block p = t / tilesPerBlock.
// Consecutive CTAs take consecutive tiles of one block, so the grid streams through a
// few blocks at a time, and the index arithmetic costs one division per tile.  Inside a
// tile each thread issues all its loads (up to kCopyUnroll 16-byte vectors) before its
// stores.  Only the end of a block can cut a vector short; those elements are copied one
// by one.

// Element by element: a warp copies 32 * K consecutive elements at a time, lane l taking
// elements e0 + 32 * k, so each warp instruction is coalesced and a warp's K stores to one
// destination cover one contiguous stretch.  A thread loads its K elements before it
// stores any.  A plain loop could not do that: the compiler must assume a store may alias
// the next load, so every load would wait for the previous store.
template <int ESZ>
__device__ __forceinline__ void elem_copy(const char* src, char* const* dst, size_t dstOff, int ndst,
                                          size_t lo, size_t hi) {
    constexpr int K = 8;
    const size_t first = lo + (size_t)(threadIdx.x >> 5) * 32 * K + (threadIdx.x & 31);
    for (size_t e0 = first; e0 < hi; e0 += (size_t)K * blockDim.x) {
        uint32_t w[K];
#pragma unroll
        for (int k = 0; k < K; k++) {
            const size_t e = e0 + 32 * (size_t)k;
            w[k] = e < hi ? ld_elem<ESZ>(src, e) : 0u;
        }
        for (int d = 0; d < ndst; d++) {
            char* o = dst[d] + dstOff * ESZ;
#pragma unroll
            for (int k = 0; k < K; k++) {
                const size_t e = e0 + 32 * (size_t)k;
                if (e < hi) st_elem<ESZ>(o, e, w[k]);
            }
        }
    }
}

// Copy [lo, hi) when 16-byte vectors cannot cover source and destinations at the same
// offsets (a ragged block, or pointers off 16 bytes).  The destinations set the vectors:
// the elements up to their first 16-byte boundary go one by one, then every 16-byte
// destination vector is cut from the two aligned 16-byte source vectors that hold its
// bytes, shifted by the source's offset against the destination; the rest go one by one.
// The second source vector always holds some of the copied bytes, so no load leaves the
// aligned 16-byte blocks the copy reads from.  Destinations at different offsets from a
// 16-byte boundary go element by element.
template <int ESZ>
__device__ __forceinline__ void realign_copy(const char* src, char* const* dst, size_t dstOff, int ndst,
                                             size_t lo, size_t hi) {
    if (hi <= lo) return;
    const uintptr_t d0 = (uintptr_t)(dst[0] + (dstOff + lo) * ESZ);
    for (int d = 1; d < ndst; d++)
        if ((((uintptr_t)(dst[d] + (dstOff + lo) * ESZ)) ^ d0) & 15u) {
            elem_copy<ESZ>(src, dst, dstOff, ndst, lo, hi);
            return;
        }
    constexpr int VE = 16 / ESZ;
    const size_t head = min((size_t)(((16u - (d0 & 15u)) & 15u) / ESZ), hi - lo);
    const size_t m0 = lo + head;
    const size_t nv = (hi - m0) / VE;
    elem_copy<ESZ>(src, dst, dstOff, ndst, lo, m0);
    const char* s0 = src + m0 * ESZ;
    const unsigned sh = (unsigned)((uintptr_t)s0 & 15u);
    const uint4* sa = reinterpret_cast<const uint4*>(s0 - sh);
    constexpr int UN = 4;
    // sh is the same for the whole tile: two loops, so that every load is unconditional
    auto body = [&](auto shifted) {
        for (size_t i0 = threadIdx.x; i0 < nv; i0 += (size_t)UN * blockDim.x) {
            uint4 v[UN];
#pragma unroll
            for (int u = 0; u < UN; u++) {
                const size_t i = i0 + (size_t)u * blockDim.x;
                if (i < nv) {
                    if constexpr (decltype(shifted)::value) v[u] = shift_bytes(sa[i], sa[i + 1], sh);
                    else v[u] = ld_stream(sa + i);
                }
            }
            for (int d = 0; d < ndst; d++) {
                uint4* o = reinterpret_cast<uint4*>(dst[d] + (dstOff + m0) * ESZ);
#pragma unroll
                for (int u = 0; u < UN; u++) {
                    const size_t i = i0 + (size_t)u * blockDim.x;
                    if (i < nv) st_stream(o + i, v[u]);
                }
            }
        }
    };
    if (sh) body(std::true_type{});
    else body(std::false_type{});
    elem_copy<ESZ>(src, dst, dstOff, ndst, m0 + nv * VE, hi);
}

// Copy [lo, hi) elements from src to every dst[0..ndst) (ndst = 1 for all-to-all).
// VB: bytes per vector (16 or 32; 0 = misaligned: realigned 16-byte vectors for 2-byte
// elements when REALIGN, else element by element).  A thread keeps 128 bytes of loads in flight: 8 vectors of 16
// bytes or 4 of 32.
template <int ESZ, int VB, bool REALIGN = true>
__device__ __forceinline__ void tile_copy(const char* src, char* const* dst, size_t dstOff, int ndst,
                                          size_t lo, size_t hi) {
    if (VB) {
        constexpr int VBB = VB ? VB : 16;
        constexpr int VE = VBB / ESZ;
        constexpr int UN = 128 / VBB;
        using VT = typename VecOf<VBB>::T;
        const size_t nv = (hi - lo) / VE;
        for (size_t i0 = threadIdx.x; i0 < nv; i0 += (size_t)UN * blockDim.x) {
            VT v[UN];
#pragma unroll
            for (int u = 0; u < UN; u++) {
                const size_t i = i0 + (size_t)u * blockDim.x;
                if (i < nv) v[u] = VecOf<VBB>::ld(src + (lo + i * VE) * ESZ);
            }
            for (int d = 0; d < ndst; d++) {
                char* o = dst[d] + dstOff * ESZ;
#pragma unroll
                for (int u = 0; u < UN; u++) {
                    const size_t i = i0 + (size_t)u * blockDim.x;
                    if (i < nv) VecOf<VBB>::st(o + (lo + i * VE) * ESZ, v[u]);
                }
            }
        }
        elem_copy<ESZ>(src, dst, dstOff, ndst, lo + nv * VE, hi);
    } else if (REALIGN && ESZ == 2) {
        // measured on GB300: realigned vectors beat 2-byte element copies (ragged bf16
        // all-gather 0.71 -> 0.82 of the copy bandwidth) but lose to 4-byte ones (fp32
        // 0.88 -> 0.87, 3-rank all-to-all 0.85 -> 0.69)
        realign_copy<ESZ>(src, dst, dstOff, ndst, lo, hi);
    } else {
        elem_copy<ESZ>(src, dst, dstOff, ndst, lo, hi);
    }
}

struct TileSpan {
    size_t lo, hi;            // channel range within a block
    size_t tileElems, tilesPerBlock;
};

template <int ESZ>
__device__ __forceinline__ TileSpan tile_span(const OnePassArgs& a, int ch, size_t blockLen) {
    TileSpan t;
    t.lo = min((size_t)ch * a.chanElems, blockLen);
    t.hi = min((size_t)(ch + 1) * a.chanElems, blockLen);
    t.tileElems = a.tileBytes / ESZ;
    t.tilesPerBlock = (t.hi - t.lo + t.tileElems - 1) / t.tileElems;
    return t;
}

// One warp tile of a 2-byte copy off 16 bytes (a ragged block): span elements from src to
// dst[r] + dstOff for r < ndst.  After the head elements that bring src to a 16-byte
// boundary, lane l takes the source vectors 32 k + l of tile tl (K per lane), each loaded
// once, aligned; the destinations share one offset d from 16 bytes, so a lane stores the
// aligned 16 bytes made of its vector's last d bytes and the next vector's first 16 - d
// (a shuffle; the tile's last lane loads the next tile's first vector itself), and only
// the block's first and last vectors go element by element.  The block's last tile
// also copies the head and the tail (lanes 0..7 and 8..15).  Destinations at different
// offsets go element by element.  All lanes of the warp call it with the same tile.
template <int K>
__device__ __forceinline__ void ragged16_tile(const char* src, char* const* dst, int ndst, size_t dstOff,
                                              size_t span, size_t tl, size_t tiles) {
    constexpr int ESZ = 2, VE = 8;
    const unsigned int lane = threadIdx.x & 31u;
    const size_t hs = min((size_t)(((16u - ((uintptr_t)src & 15u)) & 15u) / ESZ), span);
    const size_t nv = (span - hs) / VE;
    const char* sv = src + hs * ESZ;                           // 16-byte aligned
    const size_t o0 = dstOff + hs * ESZ;                       // vector v lands at dst[r] + o0 + 16 v
    const unsigned int d = (unsigned int)(((uintptr_t)dst[0] + o0) & 15u);
    bool same = true;
    for (int r = 1; r < ndst; r++) same = same && ((((uintptr_t)dst[r] + o0) & 15u) == d);
    const size_t v0 = tl * (32 * K) + lane;
    if (same) {
        uint4 x[K];
#pragma unroll
        for (int k = 0; k < K; k++) {
            const size_t v = v0 + 32 * k;
            x[k] = v < nv ? ld_stream(sv + 16 * v) : make_uint4(0u, 0u, 0u, 0u);
        }
        // the tile's last lane also loads the next tile's first vector, so that only the
        // block's first and last vectors go element by element
        const size_t vLast = v0 + 32 * (K - 1);
        const uint4 after = (lane == 31u && d != 0 && vLast + 1 < nv) ? ld_stream(sv + 16 * (vLast + 1))
                                                                       : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int k = 0; k < K; k++) {
            const size_t v = v0 + 32 * k;
            if (d == 0) {
                if (v < nv)
                    for (int r = 0; r < ndst; r++) st_stream(dst[r] + o0 + 16 * v, x[k]);
                continue;
            }
            const uint4 give = (lane == 0u && k + 1 < K) ? x[k + 1] : x[k];
            uint4 nx;
            nx.x = __shfl_sync(0xFFFFFFFFu, give.x, (lane + 1) & 31u);
            nx.y = __shfl_sync(0xFFFFFFFFu, give.y, (lane + 1) & 31u);
            nx.z = __shfl_sync(0xFFFFFFFFu, give.z, (lane + 1) & 31u);
            nx.w = __shfl_sync(0xFFFFFFFFu, give.w, (lane + 1) & 31u);
            if (lane == 31u && k == K - 1) nx = after;
            if (v >= nv) continue;
            const bool nextHere = v + 1 < nv;
            const bool prevHere = v > 0;
            const unsigned int split = (16u - d) / ESZ;        // elements before the boundary
            const uint4 y = shift_bytes(x[k], nx, 16u - d);
            for (int r = 0; r < ndst; r++) {
                char* o = dst[r] + o0 + 16 * v;
                if (nextHere) st_stream(o + (16u - d), y);
                if (!prevHere || !nextHere) {                  // the block's first or last vector
                    const uint32_t wd[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
#pragma unroll
                    for (int e = 0; e < VE; e++)
                        if ((e < (int)split && !prevHere) || (e >= (int)split && !nextHere))
                            st_elem<ESZ>(o, e, (wd[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
                }
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < K; k++) {
            const size_t v = v0 + 32 * k;
            if (v >= nv) continue;
            for (int e = 0; e < VE; e++) {
                const uint32_t x = ld_elem<ESZ>(sv, VE * v + e);
                for (int r = 0; r < ndst; r++) st_elem<ESZ>(dst[r] + o0, VE * v + e, x);
            }
        }
    }
    if (tl == tiles - 1) {
        size_t e = ~(size_t)0;
        if (lane < hs) e = lane;
        else if (lane >= 8u && lane - 8u < span - hs - VE * nv) e = hs + VE * nv + (lane - 8u);
        if (e != ~(size_t)0) {
            const uint32_t x = ld_elem<ESZ>(src, e);
            for (int r = 0; r < ndst; r++) st_elem<ESZ>(dst[r] + dstOff, e, x);
        }
    }
}

// The ragged 2-byte copies on warp tiles of 32 x 2 vectors: two 512-thread CTAs per SM,
// 64 registers.
constexpr int kRaggedK = 2;

__global__ void __launch_bounds__(kOnePassThreads, 2) k_allgather_ragged16(const __grid_constant__ OnePassArgs a) {
    pdl_begin();
    const int N = a.nRanks;
    const int ch = blockIdx.x / a.ctasPerChannel;
    const int cta = blockIdx.x - ch * a.ctasPerChannel;
    const size_t sc = a.count;
    const size_t lo = min((size_t)ch * a.chanElems, sc);
    const size_t span = min((size_t)(ch + 1) * a.chanElems, sc) - lo;
    const size_t tiles = span / 8 / (32 * kRaggedK) + 1;
    const size_t stride = (size_t)a.ctasPerChannel * blockDim.x / 32;
    // gather (a.outRoot = root) writes recv[root] only
    char* const* dsts = a.outRoot >= 0 ? (char* const*)&a.recv[a.outRoot] : (char* const*)a.recv;
    const int nd = a.outRoot >= 0 ? 1 : N;
    for (size_t w = ((size_t)cta * blockDim.x + threadIdx.x) / 32; w < tiles * (size_t)N; w += stride) {
        const int s = (int)(w / tiles);
        ragged16_tile<kRaggedK>((const char*)a.send[s] + lo * 2, dsts, nd, ((size_t)s * sc + lo) * 2, span,
                                w - (size_t)s * tiles, tiles);
    }
}

// Broadcast: the root's block to every receiver.
__global__ void __launch_bounds__(kOnePassThreads, 2) k_broadcast_ragged16(const __grid_constant__ OnePassArgs a) {
    pdl_begin();
    const int ch = blockIdx.x / a.ctasPerChannel;
    const int cta = blockIdx.x - ch * a.ctasPerChannel;
    const size_t lo = min((size_t)ch * a.chanElems, a.count);
    const size_t span = min((size_t)(ch + 1) * a.chanElems, a.count) - lo;
    const size_t tiles = span / 8 / (32 * kRaggedK) + 1;
    const size_t stride = (size_t)a.ctasPerChannel * blockDim.x / 32;
    for (size_t w = ((size_t)cta * blockDim.x + threadIdx.x) / 32; w < tiles; w += stride)
        ragged16_tile<kRaggedK>((const char*)a.send[a.root] + lo * 2, (char* const*)a.recv, a.nRanks, lo * 2, span, w,
                                tiles);
}

// Scatter: block j of the root's buffer to recv[j].
__global__ void __launch_bounds__(kOnePassThreads, 2) k_scatter_ragged16(const __grid_constant__ OnePassArgs a) {
    pdl_begin();
    const int N = a.nRanks;
    const int ch = blockIdx.x / a.ctasPerChannel;
    const int cta = blockIdx.x - ch * a.ctasPerChannel;
    const size_t c = a.count;
    const size_t lo = min((size_t)ch * a.chanElems, c);
    const size_t span = min((size_t)(ch + 1) * a.chanElems, c) - lo;
    const size_t tiles = span / 8 / (32 * kRaggedK) + 1;
    const size_t stride = (size_t)a.ctasPerChannel * blockDim.x / 32;
    for (size_t w = ((size_t)cta * blockDim.x + threadIdx.x) / 32; w < tiles * (size_t)N; w += stride) {
        const int j = (int)(w / tiles);
        char* dst = (char*)a.recv[j];
        ragged16_tile<kRaggedK>((const char*)a.send[a.root] + ((size_t)j * c + lo) * 2, &dst, 1, lo * 2, span,
                                w - (size_t)j * tiles, tiles);
    }
}

__global__ void __launch_bounds__(kOnePassThreads, 2) k_alltoall_ragged16(const __grid_constant__ OnePassArgs a) {
    pdl_begin();
    const int N = a.nRanks;
    const int ch = blockIdx.x / a.ctasPerChannel;
    const int cta = blockIdx.x - ch * a.ctasPerChannel;
    const size_t c = a.count;
    const size_t lo = min((size_t)ch * a.chanElems, c);
    const size_t span = min((size_t)(ch + 1) * a.chanElems, c) - lo;
    const size_t tiles = span / 8 / (32 * kRaggedK) + 1;
    const size_t stride = (size_t)a.ctasPerChannel * blockDim.x / 32;
    for (size_t w = ((size_t)cta * blockDim.x + threadIdx.x) / 32; w < tiles * (size_t)N * N; w += stride) {
        const size_t p = w / tiles;                          // block p = i * N + j: send[i] -> recv[j]
        const int i = (int)(p / N), j = (int)(p - (size_t)i * N);
        char* dst = (char*)a.recv[j];
        ragged16_tile<kRaggedK>((const char*)a.send[i] + ((size_t)j * c + lo) * 2, &dst, 1, ((size_t)i * c + lo) * 2,
                                span, w - p * tiles, tiles);
    }
}

// All-gather: block s = send[s] lands at recv[r] + s*sc for every r.  a.count = sc.
// Gather (a.outRoot = root) writes recv[root] only.
template <int ESZ, int VB>
__global__ void __launch_bounds__(kOnePassThreads, 2)
k_allgather_onepass(const __grid_constant__ OnePassArgs a) {
    pdl_begin();
    const int N = a.nRanks;
    const int ch = blockIdx.x / a.ctasPerChannel;
    const int cta = blockIdx.x - ch * a.ctasPerChannel;
    const size_t sc = a.count;

    const TileSpan sp = tile_span<ESZ>(a, ch, sc);
    const size_t nTiles = sp.tilesPerBlock * (size_t)N;
    char* const* dsts = a.outRoot >= 0 ? (char* const*)&a.recv[a.outRoot] : (char* const*)a.recv;
    const int nd = a.outRoot >= 0 ? 1 : N;
    for (size_t t = cta; t < nTiles; t += a.ctasPerChannel) {
        const int s = (int)(t / sp.tilesPerBlock);
        const size_t k = t - (size_t)s * sp.tilesPerBlock;
        const size_t tlo = sp.lo + k * sp.tileElems, thi = min(tlo + sp.tileElems, sp.hi);
        tile_copy<ESZ, VB>((const char*)a.send[s], dsts, (size_t)s * sc, nd, tlo, thi);
    }
}

// Broadcast: recv[r][t] = send[root][t] for all r.
template <int ESZ, int VB>
__global__ void __launch_bounds__(kOnePassThreads, 2)
k_broadcast_onepass(const __grid_constant__ OnePassArgs a) {
    pdl_begin();
    const int ch = blockIdx.x / a.ctasPerChannel;
    const int cta = blockIdx.x - ch * a.ctasPerChannel;
    const TileSpan sp = tile_span<ESZ>(a, ch, a.count);
    for (size_t k = cta; k < sp.tilesPerBlock; k += a.ctasPerChannel) {
        const size_t tlo = sp.lo + k * sp.tileElems, thi = min(tlo + sp.tileElems, sp.hi);
        tile_copy<ESZ, VB>((const char*)a.send[a.root], (char* const*)a.recv, 0, a.nRanks, tlo, thi);
    }
}

// Uniform all-to-all: recv[j][i*c + t] = send[i][j*c + t].  a.count = c.
template <int ESZ, int VB>
__global__ void __launch_bounds__(kOnePassThreads, 2)
k_alltoall_onepass(const __grid_constant__ OnePassArgs a) {
    pdl_begin();
    const int N = a.nRanks;
    const int ch = blockIdx.x / a.ctasPerChannel;
    const int cta = blockIdx.x - ch * a.ctasPerChannel;
    const size_t c = a.count;
    const TileSpan sp = tile_span<ESZ>(a, ch, c);
    const size_t nTiles = sp.tilesPerBlock * (size_t)N * (size_t)N;
    for (size_t t = cta; t < nTiles; t += a.ctasPerChannel) {
        const size_t p = t / sp.tilesPerBlock;
        const size_t k = t - p * sp.tilesPerBlock;
        const int i = (int)(p / N), j = (int)(p - (p / N) * N);
        const size_t tlo = sp.lo + k * sp.tileElems, thi = min(tlo + sp.tileElems, sp.hi);
        char* dst = (char*)a.recv[j];
        tile_copy<ESZ, VB>((const char*)a.send[i] + (size_t)j * c * ESZ, &dst, (size_t)i * c, 1, tlo, thi);
    }
}

// Scatter: block j of send[root] lands in recv[j].  a.count = recvcount.
template <int ESZ, int VB>
__global__ void __launch_bounds__(kOnePassThreads, 2)
k_scatter_onepass(const __grid_constant__ OnePassArgs a) {
    pdl_begin();
    const int N = a.nRanks;
    const int ch = blockIdx.x / a.ctasPerChannel;
    const int cta = blockIdx.x - ch * a.ctasPerChannel;
    const size_t c = a.count;
    const TileSpan sp = tile_span<ESZ>(a, ch, c);
    const size_t nTiles = sp.tilesPerBlock * (size_t)N;
    for (size_t t = cta; t < nTiles; t += a.ctasPerChannel) {
        const int j = (int)(t / sp.tilesPerBlock);
        const size_t k = t - (size_t)j * sp.tilesPerBlock;
        const size_t tlo = sp.lo + k * sp.tileElems, thi = min(tlo + sp.tileElems, sp.hi);
        char* dst = (char*)a.recv[j];
        tile_copy<ESZ, VB>((const char*)a.send[a.root] + (size_t)j * c * ESZ, &dst, 0, 1, tlo, thi);
    }
}

// Variable all-to-all.  The N*N blocks are cut into tiles of a.tileBytes; tiles are
// numbered across all blocks (sender-major), so a hot destination's many tiles spread
// over the whole grid.  The host cannot size the grid (the tables live on the device), so
// one resident wave of CTAs takes tiles in order from an atomic counter: the tiles in
// flight stay within a narrow window of the buffers, as with the flat grids of the other
// copies.  The last CTA to finish resets the counter for the next launch.  Every CTA
// builds the tile prefix sums in shared memory from the device tables.
// Three copy widths are inlined here, so the kernel keeps 128 registers: one CTA per SM,
// so the grid is one wave of CTAs that take tiles from the counter.
template <int ESZ>
__global__ void __launch_bounds__(kOnePassThreads, 1)
k_alltoallv(const __grid_constant__ A2AvArgs a) {
    pdl_begin();
    __shared__ unsigned long long tileStart[VCOMM_MAX_RANKS * VCOMM_MAX_RANKS + 1];
    __shared__ int sBad;
    __shared__ unsigned int sTile;
    const int N = a.nRanks;
    const int NB = N * N;
    const size_t tileElems = a.tileBytes / ESZ;
    if (threadIdx.x == 0) sBad = 0;
    __syncthreads();
    for (int p = threadIdx.x; p < NB; p += blockDim.x) {
        const int i = p / N, j = p - (p / N) * N;
        const int32_t cnt = a.counts[p], so = a.sdispls[p], ro = a.rdispls[j * N + i];
        unsigned long long tiles = 0;
        if (cnt < 0 || so < 0 || ro < 0 || (cnt > 0 && (!a.send[i] || !a.recv[j]))) sBad = 1;
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
    for (;;) {
        if (threadIdx.x == 0) sTile = atomicAdd(&a.tileCounter[0], 1u);
        __syncthreads();
        const unsigned long long tile = sTile;
        __syncthreads();                               // all have read sTile
        if (tile >= nTiles) break;
        while (tileStart[p + 1] <= tile) p++;          // a CTA's tiles ascend, so p only grows
        const int i = p / N, j = p - (p / N) * N;
        const size_t cnt = (size_t)a.counts[p];
        const size_t k = tile - tileStart[p];
        const size_t lo = k * tileElems, hi = min(lo + tileElems, cnt);
        const char* src = (const char*)a.send[i] + (size_t)a.sdispls[p] * ESZ;
        char* dst = (char*)a.recv[j] + (size_t)a.rdispls[j * N + i] * ESZ;
        const uintptr_t al = ((uintptr_t)src | (uintptr_t)dst) & 31;
        if (al == 0) tile_copy<ESZ, 32>(src, &dst, 0, 1, lo, hi);
        else if ((al & 15) == 0) tile_copy<ESZ, 16>(src, &dst, 0, 1, lo, hi);
        else tile_copy<ESZ, 0, false>(src, &dst, 0, 1, lo, hi);   // element by element: no spills
    }
    // Every CTA has taken its last tile number; the last one out clears the counter.
    if (threadIdx.x == 0 && atomicAdd(&a.tileCounter[1], 1u) == gridDim.x - 1) {
        atomicExch(&a.tileCounter[0], 0u);
        atomicExch(&a.tileCounter[1], 0u);
    }
}

// ---- dispatch --------------------------------------------------------------------------

#define VC_COPY_LAUNCH_ESZ(KERNEL, E)                                                      \
    do {                                                                                   \
        if (vb == 32) (void)pdl_launch(KERNEL<E, 32>, grid, threads, 0, s, a);                           \
        else if (vb == 16) (void)pdl_launch(KERNEL<E, 16>, grid, threads, 0, s, a);                      \
        else (void)pdl_launch(KERNEL<E, 0>, grid, threads, 0, s, a);                                     \
    } while (0)

#define VC_COPY_LAUNCH(KERNEL)                                                             \
    do {                                                                                   \
        if (elemSize == 4) VC_COPY_LAUNCH_ESZ(KERNEL, 4);                                  \
        else if (elemSize == 2) VC_COPY_LAUNCH_ESZ(KERNEL, 2);                             \
        else return cudaErrorInvalidValue;                                                 \
        return cudaGetLastError();                                                         \
    } while (0)

cudaError_t launch_allgather_onepass(const OnePassArgs& a, int elemSize, int vb, int grid,
                                     int threads, cudaStream_t s) {
    if (elemSize == 2 && vb == 0) {
        (void)pdl_launch(k_allgather_ragged16, grid, threads, 0, s, a);
        return cudaGetLastError();
    }
    VC_COPY_LAUNCH(k_allgather_onepass);
}

cudaError_t launch_broadcast_onepass(const OnePassArgs& a, int elemSize, int vb, int grid,
                                     int threads, cudaStream_t s) {
    if (elemSize == 2 && vb == 0) {
        (void)pdl_launch(k_broadcast_ragged16, grid, threads, 0, s, a);
        return cudaGetLastError();
    }
    VC_COPY_LAUNCH(k_broadcast_onepass);
}

cudaError_t launch_alltoall_onepass(const OnePassArgs& a, int elemSize, int vb, int grid,
                                    int threads, cudaStream_t s) {
    if (elemSize == 2 && vb == 0) {
        (void)pdl_launch(k_alltoall_ragged16, grid, threads, 0, s, a);
        return cudaGetLastError();
    }
    VC_COPY_LAUNCH(k_alltoall_onepass);
}

cudaError_t launch_scatter_onepass(const OnePassArgs& a, int elemSize, int vb, int grid,
                                   int threads, cudaStream_t s) {
    if (elemSize == 2 && vb == 0) {
        (void)pdl_launch(k_scatter_ragged16, grid, threads, 0, s, a);
        return cudaGetLastError();
    }
    VC_COPY_LAUNCH(k_scatter_onepass);
}

cudaError_t launch_alltoallv(const A2AvArgs& a, int grid, int threads, cudaStream_t s) {
    if (a.elemSize == 4) (void)pdl_launch(k_alltoallv<4>, grid, threads, 0, s, a);
    else if (a.elemSize == 2) (void)pdl_launch(k_alltoallv<2>, grid, threads, 0, s, a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace vc
