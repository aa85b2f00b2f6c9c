// k_onepass.cu -- one-pass reduction kernels: all-reduce and reduce-scatter.
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

// All-reduce, and reduce to root.  grid = nChannels * ctasPerChannel.  VB: 0 (element
// path), 16 or 32 bytes per vector; the 32-byte kernel keeps twice the registers, so it
// runs one 512-thread CTA per SM instead of two.  Reduce to root (a.orderRoot = a.outRoot
// = root) reduces every block in the root's order and writes only recv[root].
template <int DT, int OP, int VB, int NF = 0>
__global__ void __launch_bounds__(kOnePassThreads, VB == 32 ? 1 : 2)
k_allreduce_onepass(const __grid_constant__ OnePassArgs a) {
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int U = VB ? VB / ESZ : 1;
    const int N = NF ? NF : a.nRanks;
    const int ch = blockIdx.x / a.ctasPerChannel;
    const int cta = blockIdx.x - ch * a.ctasPerChannel;
    const size_t stride = (size_t)a.ctasPerChannel * blockDim.x;
    const ChannelSpan sp = channel_span(a, ch, U);
    const size_t chEnd = min((size_t)(ch + 1) * a.chanElems, a.blockElems);
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
        const int r0 = a.outRoot >= 0 ? a.outRoot : 0;
        const int r1 = a.outRoot >= 0 ? a.outRoot + 1 : N;
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
// a.count = N * rc, a.blockElems = rc.  VB > 0 requires rc * esz % VB == 0.
template <int DT, int OP, int OUT, int VB>
__global__ void __launch_bounds__(kOnePassThreads, VB == 32 ? 1 : 2)
k_reduce_scatter_onepass(const __grid_constant__ OnePassArgs a) {
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int U = VB ? VB / ESZ : 1;
    const int N = a.nRanks;
    const int ch = blockIdx.x / a.ctasPerChannel;
    const int cta = blockIdx.x - ch * a.ctasPerChannel;
    const size_t stride = (size_t)a.ctasPerChannel * blockDim.x;
    const size_t rc = a.blockElems;
    const bool hasScale = a.hasScale != 0;
    const ChannelSpan sp = channel_span(a, ch, U);
    const size_t chEnd = min((size_t)(ch + 1) * a.chanElems, rc);
    const size_t total = sp.units * (size_t)N;
    for (size_t j = (size_t)cta * blockDim.x + threadIdx.x; j < total; j += stride) {
        const int r = (int)(j / sp.units);
        const size_t i = j - (size_t)r * sp.units;
        const size_t t = sp.lo + i * U;                 // element within block r
        if (t >= chEnd) continue;
        const size_t base = (size_t)r * rc;
        const int first = r + 1 == N ? 0 : r + 1;
        if (VB && t + U <= chEnd) {
            const auto acc = reduce_vec_ring<DT, OP, VB ? VB : 16>(a.send, N, first, (base + t) * ESZ);
            store_epilogue_vec<DT, OUT>(a.recv[r], t, acc, hasScale, a.scale);
        } else {
            for (size_t x = t; x < min(t + U, chEnd); x++) {
                const uint32_t acc = reduce_elem_ring<DT, OP>(a.send, N, first, base + x);
                store_epilogue_elem<DT, OUT>(a.recv[r], x, acc, hasScale, a.scale);
            }
        }
    }
}

// Batched all-reduces (group batching, NCCL book chapter 6: ncclPrepareTasks aggregates
// collectives of the same function, op and type into one launch).  Every item keeps its
// own block partition and ring order, so its bits equal a separate vAllReduce.  The work
// units of all items form one flat index space; a thread finds its item by binary search
// over the items' first units, held in shared memory.
template <int DT, int OP, int VB>
__global__ void __launch_bounds__(kOnePassThreads, VB == 32 ? 1 : 2)
k_allreduce_group(const __grid_constant__ GroupArgs a) {
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int U = VB ? VB / ESZ : 1;
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
        } else {
            for (size_t x = e; x < min(e + U, bend); x++) {
                const uint32_t acc = reduce_elem_ring<DT, OP>(send, N, first, x);
                for (int r = 0; r < N; r++) st_elem<ESZ>(recv[r], x, acc);
            }
        }
    }
}

// Double-binary-tree all-reduce, one pass.  A thread loads its vector of every rank
// (8 loads in flight at a time) into a per-thread array, then evaluates the tree in
// post-order with a small stack: a node's partial is its own vector, then OP with child
// 0's partial, then with child 1's.  Both arrays live in local memory (their indices are
// data-independent but known only at run time); the kernel stays HBM-bound.
template <int DT, int OP, int VB>
__global__ void __launch_bounds__(kOnePassThreads, 2)
k_allreduce_tree(const __grid_constant__ TreeArgs a) {
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int U = VB ? VB / ESZ : 1;
    using VT = typename VecOf<VB ? VB : 16>::T;
    const int N = a.nRanks;
    const size_t u0 = (a.split + U - 1) / U;
    const size_t u1 = (a.count - a.split + U - 1) / U;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t j = (size_t)blockIdx.x * blockDim.x + threadIdx.x; j < u0 + u1; j += stride) {
        const int t = j < u0 ? 0 : 1;
        const size_t lo = t == 0 ? 0 : a.split, hi = t == 0 ? a.split : a.count;
        const size_t e = lo + (j - (t == 0 ? 0 : u0)) * U;
        if (VB && e + U <= hi) {
            VT xs[VCOMM_MAX_RANKS];
            for (int k0 = 0; k0 < N; k0 += 8) {
                VT v[8];
#pragma unroll
                for (int q = 0; q < 8; q++)
                    if (k0 + q < N) v[q] = VecOf<VB ? VB : 16>::ld((const char*)a.send[k0 + q] + e * ESZ);
#pragma unroll
                for (int q = 0; q < 8; q++)
                    if (k0 + q < N) xs[k0 + q] = v[q];
            }
            VT stk[kTreeMaxStack];
            int sp = 0;
            for (int i = 0; i < N; i++) {
                const int c = a.nchild[t][i];
                VT acc = xs[a.prog[t][i]];
                for (int q = 0; q < c; q++) acc = op_vec<DT, OP>(acc, stk[sp - c + q]);
                sp -= c;
                stk[sp++] = acc;
            }
            for (int r = 0; r < N; r++) VecOf<VB ? VB : 16>::st((char*)a.recv[r] + e * ESZ, stk[0]);
        } else {
            for (size_t x = e; x < min(e + U, hi); x++) {
                uint32_t stk[kTreeMaxStack];
                int sp = 0;
                for (int i = 0; i < N; i++) {
                    const int c = a.nchild[t][i];
                    uint32_t acc = ld_elem<ESZ>(a.send[a.prog[t][i]], x);
                    for (int q = 0; q < c; q++) acc = op_elem<DT, OP>(acc, stk[sp - c + q]);
                    sp -= c;
                    stk[sp++] = acc;
                }
                for (int r = 0; r < N; r++) st_elem<ESZ>(a.recv[r], x, stk[0]);
            }
        }
    }
}

// The same trees for a rank count fixed at compile time: the post-order program is a
// constant expression, so after unrolling every array index is a constant and the values
// stay in registers.
template <int N>
struct TreeProg {
    signed char prog[2][N];
    signed char nchild[2][N];
};

__host__ __device__ constexpr void btree_links(int n, int r, int* u, int* a, int* b) {
    int step = 1;
    while (step < n && (r & step) == 0) step <<= 1;
    if (r == 0) {
        *u = -1;
        *a = -1;
        *b = n > 1 ? step / 2 : -1;
        return;
    }
    const int up = (r ^ step) | (step << 1);
    *u = up < n ? up : (r ^ step);
    int half = step / 2;
    *a = half > 0 ? r - half : -1;
    *b = -1;
    for (; half > 0; half /= 2) {
        if (r + half < n) {
            *b = r + half;
            break;
        }
    }
}

__host__ __device__ constexpr void dtree_links(int n, int r, int t, int* u, int* a, int* b) {
    if (t == 0) {
        btree_links(n, r, u, a, b);
        return;
    }
    const bool mirror = n % 2 == 0;
    int u0 = -1, a0 = -1, b0 = -1;
    btree_links(n, mirror ? n - 1 - r : (r + n - 1) % n, &u0, &a0, &b0);
    *u = u0 < 0 ? -1 : (mirror ? n - 1 - u0 : (u0 + 1) % n);
    *a = a0 < 0 ? -1 : (mirror ? n - 1 - a0 : (a0 + 1) % n);
    *b = b0 < 0 ? -1 : (mirror ? n - 1 - b0 : (b0 + 1) % n);
}

template <int N>
__host__ __device__ constexpr TreeProg<N> make_tree_prog() {
    TreeProg<N> P{};
    for (int t = 0; t < 2; t++) {
        int root = 0;
        for (int v = 0; v < N; v++) {
            int u = 0, a = 0, b = 0;
            dtree_links(N, v, t, &u, &a, &b);
            if (u < 0) root = v;
        }
        // iterative post-order: (node, children visited) on an explicit stack
        int stackNode[N] = {}, stackState[N] = {};
        int sp = 0, n = 0;
        stackNode[sp] = root;
        stackState[sp] = 0;
        sp++;
        while (sp > 0) {
            const int v = stackNode[sp - 1];
            int u = 0, a = 0, b = 0;
            dtree_links(N, v, t, &u, &a, &b);
            const int st = stackState[sp - 1];
            if (st == 0) {
                stackState[sp - 1] = 1;
                if (a >= 0) { stackNode[sp] = a; stackState[sp] = 0; sp++; }
            } else if (st == 1) {
                stackState[sp - 1] = 2;
                if (b >= 0) { stackNode[sp] = b; stackState[sp] = 0; sp++; }
            } else {
                P.prog[t][n] = (signed char)v;
                P.nchild[t][n] = (signed char)((a >= 0) + (b >= 0));
                n++;
                sp--;
            }
        }
    }
    return P;
}

template <int DT, int OP, int VT_BYTES, int N, int T>
__device__ __forceinline__ typename VecOf<VT_BYTES>::T eval_tree_fixed(const typename VecOf<VT_BYTES>::T (&x)[N]) {
    using VT = typename VecOf<VT_BYTES>::T;
    constexpr TreeProg<N> P = make_tree_prog<N>();
    VT stk[N];
    int sp = 0;
#pragma unroll
    for (int i = 0; i < N; i++) {
        const int c = P.nchild[T][i];
        VT acc = x[P.prog[T][i]];
#pragma unroll
        for (int q = 0; q < 2; q++)
            if (q < c) acc = op_vec<DT, OP>(acc, stk[sp - c + q]);
        sp -= c;
        stk[sp++] = acc;
    }
    return stk[0];
}

template <int DT, int OP, int VB, int N>
__global__ void __launch_bounds__(kOnePassThreads, VB == 32 ? 1 : 2)
k_allreduce_tree_fixed(const __grid_constant__ TreeArgs a) {
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int U = VB / ESZ;
    using VT = typename VecOf<VB>::T;
    const size_t u0 = (a.split + U - 1) / U;
    const size_t u1 = (a.count - a.split + U - 1) / U;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t j = (size_t)blockIdx.x * blockDim.x + threadIdx.x; j < u0 + u1; j += stride) {
        const int t = j < u0 ? 0 : 1;
        const size_t lo = t == 0 ? 0 : a.split, hi = t == 0 ? a.split : a.count;
        const size_t e = lo + (j - (t == 0 ? 0 : u0)) * U;
        if (e + U <= hi) {
            VT x[N];
#pragma unroll
            for (int r = 0; r < N; r++) x[r] = VecOf<VB>::ld((const char*)a.send[r] + e * ESZ);
            const VT acc = t == 0 ? eval_tree_fixed<DT, OP, VB, N, 0>(x) : eval_tree_fixed<DT, OP, VB, N, 1>(x);
#pragma unroll
            for (int r = 0; r < N; r++) VecOf<VB>::st((char*)a.recv[r] + e * ESZ, acc);
        } else {
            for (size_t xx = e; xx < min(e + U, hi); xx++) {
                uint32_t stk[kTreeMaxStack];
                int sp = 0;
                for (int i = 0; i < N; i++) {
                    const int c = a.nchild[t][i];
                    uint32_t acc = ld_elem<ESZ>(a.send[a.prog[t][i]], xx);
                    for (int q = 0; q < c; q++) acc = op_elem<DT, OP>(acc, stk[sp - c + q]);
                    sp -= c;
                    stk[sp++] = acc;
                }
                for (int r = 0; r < N; r++) st_elem<ESZ>(a.recv[r], xx, stk[0]);
            }
        }
    }
}

// ---- dispatch --------------------------------------------------------------------------

template <int DT, int OP>
static cudaError_t ar_dispatch_vec(const OnePassArgs& a, int vb, int grid, int threads,
                                   cudaStream_t s) {
    if (a.nRanks == 8 && vb == 32) k_allreduce_onepass<DT, OP, 32, 8><<<grid, threads, 0, s>>>(a);
    else if (a.nRanks == 8 && vb == 16) k_allreduce_onepass<DT, OP, 16, 8><<<grid, threads, 0, s>>>(a);
    else if (vb == 32) k_allreduce_onepass<DT, OP, 32><<<grid, threads, 0, s>>>(a);
    else if (vb == 16) k_allreduce_onepass<DT, OP, 16><<<grid, threads, 0, s>>>(a);
    else k_allreduce_onepass<DT, OP, 0><<<grid, threads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int DT>
static cudaError_t ar_dispatch_op(const OnePassArgs& a, vRedOp_t op, int vb, int grid, int threads,
                                  cudaStream_t s) {
    switch (op) {
    case vSum: return ar_dispatch_vec<DT, kSum>(a, vb, grid, threads, s);
    case vProd: return ar_dispatch_vec<DT, kProd>(a, vb, grid, threads, s);
    case vMin: return ar_dispatch_vec<DT, kMin>(a, vb, grid, threads, s);
    case vMax: return ar_dispatch_vec<DT, kMax>(a, vb, grid, threads, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_allreduce_onepass(const OnePassArgs& a, vDataType_t dt, vRedOp_t op, int vb,
                                     int grid, int threads, cudaStream_t s) {
    switch (dt) {
    case vFloat32: return ar_dispatch_op<kF32>(a, op, vb, grid, threads, s);
    case vFloat16: return ar_dispatch_op<kF16>(a, op, vb, grid, threads, s);
    case vBFloat16: return ar_dispatch_op<kBF16>(a, op, vb, grid, threads, s);
    case vInt32: return ar_dispatch_op<kI32>(a, op, vb, grid, threads, s);
    }
    return cudaErrorInvalidValue;
}

template <int DT, int OP>
static cudaError_t tree_dispatch_vec(const TreeArgs& a, int vb, int grid, int threads, cudaStream_t s) {
    if (a.nRanks == 8 && vb == 32) k_allreduce_tree_fixed<DT, OP, 32, 8><<<grid, threads, 0, s>>>(a);
    else if (a.nRanks == 8 && vb == 16) k_allreduce_tree_fixed<DT, OP, 16, 8><<<grid, threads, 0, s>>>(a);
    else if (vb == 32) k_allreduce_tree<DT, OP, 32><<<grid, threads, 0, s>>>(a);
    else if (vb == 16) k_allreduce_tree<DT, OP, 16><<<grid, threads, 0, s>>>(a);
    else k_allreduce_tree<DT, OP, 0><<<grid, threads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int DT>
static cudaError_t tree_dispatch_op(const TreeArgs& a, vRedOp_t op, int vb, int grid, int threads,
                                    cudaStream_t s) {
    switch (op) {
    case vSum: return tree_dispatch_vec<DT, kSum>(a, vb, grid, threads, s);
    case vProd: return tree_dispatch_vec<DT, kProd>(a, vb, grid, threads, s);
    case vMin: return tree_dispatch_vec<DT, kMin>(a, vb, grid, threads, s);
    case vMax: return tree_dispatch_vec<DT, kMax>(a, vb, grid, threads, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_allreduce_tree(const TreeArgs& a, vDataType_t dt, vRedOp_t op, int vb, int grid,
                                  int threads, cudaStream_t s) {
    switch (dt) {
    case vFloat32: return tree_dispatch_op<kF32>(a, op, vb, grid, threads, s);
    case vFloat16: return tree_dispatch_op<kF16>(a, op, vb, grid, threads, s);
    case vBFloat16: return tree_dispatch_op<kBF16>(a, op, vb, grid, threads, s);
    case vInt32: return tree_dispatch_op<kI32>(a, op, vb, grid, threads, s);
    }
    return cudaErrorInvalidValue;
}

template <int DT, int OP>
static cudaError_t group_dispatch_vec(const GroupArgs& a, int vb, int grid, int threads, cudaStream_t s) {
    if (vb == 32) k_allreduce_group<DT, OP, 32><<<grid, threads, 0, s>>>(a);
    else if (vb == 16) k_allreduce_group<DT, OP, 16><<<grid, threads, 0, s>>>(a);
    else k_allreduce_group<DT, OP, 0><<<grid, threads, 0, s>>>(a);
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

template <int DT, int OP, int OUT>
static cudaError_t rs_dispatch_vec(const OnePassArgs& a, int vb, int grid, int threads,
                                   cudaStream_t s) {
    if (vb == 32) k_reduce_scatter_onepass<DT, OP, OUT, 32><<<grid, threads, 0, s>>>(a);
    else if (vb == 16) k_reduce_scatter_onepass<DT, OP, OUT, 16><<<grid, threads, 0, s>>>(a);
    else k_reduce_scatter_onepass<DT, OP, OUT, 0><<<grid, threads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int DT, int OUT>
static cudaError_t rs_dispatch_op(const OnePassArgs& a, vRedOp_t op, int vb, int grid,
                                  int threads, cudaStream_t s) {
    switch (op) {
    case vSum: return rs_dispatch_vec<DT, kSum, OUT>(a, vb, grid, threads, s);
    case vProd: return rs_dispatch_vec<DT, kProd, OUT>(a, vb, grid, threads, s);
    case vMin: return rs_dispatch_vec<DT, kMin, OUT>(a, vb, grid, threads, s);
    case vMax: return rs_dispatch_vec<DT, kMax, OUT>(a, vb, grid, threads, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_reduce_scatter_onepass(const OnePassArgs& a, vDataType_t dt, vRedOp_t op,
                                          vDataType_t outType, int vb, int grid, int threads,
                                          cudaStream_t s) {
    const bool toF32 = outType == vFloat32 && dt != vFloat32;
    if (outType != dt && !toF32) return cudaErrorInvalidValue;
    switch (dt) {
    case vFloat32: return rs_dispatch_op<kF32, kF32>(a, op, vb, grid, threads, s);
    case vFloat16:
        return toF32 ? rs_dispatch_op<kF16, kF32>(a, op, vb, grid, threads, s)
                     : rs_dispatch_op<kF16, kF16>(a, op, vb, grid, threads, s);
    case vBFloat16:
        return toF32 ? rs_dispatch_op<kBF16, kF32>(a, op, vb, grid, threads, s)
                     : rs_dispatch_op<kBF16, kBF16>(a, op, vb, grid, threads, s);
    case vInt32: return rs_dispatch_op<kI32, kI32>(a, op, vb, grid, threads, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace vc
