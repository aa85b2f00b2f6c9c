// tree.cuh -- double-binary-tree all-reduce in one pass (NCCL book chapter 4, trees.cc
// ncclGetBtree / ncclGetDtree): the first half of the buffer is reduced up tree 0 and the
// rest up tree 1, every node combining its own element, then child 0's partial, then
// child 1's, and the root's result is written to every rank.
#pragma once

#include <algorithm>

#include "device.cuh"

namespace vc {

// Double-binary-tree all-reduce, one pass, for a rank count known only at run time.  A
// thread walks the tree's post-order program (a node's partial is its own value, then OP
// with child 0's partial, then with child 1's) eight steps at a time: it loads the eight
// nodes' values first, then folds them.  The newest partial stays in registers; the
// partials still waiting for their parent sit on a per-thread stack in shared memory
// (at most 6 deep for N <= 64), since their positions are known only at run time.  The
// vector path moves 16 bytes per rank and runs in CTAs of at most kTreeThreads threads.
constexpr int kTreeThreads = 256;
constexpr int kTreeStackDepth = 8;

template <int DT, int OP, typename T>
__device__ __forceinline__ T tree_op(T a, T b) {
    if constexpr (sizeof(T) == 4) return op_elem<DT, OP>(a, b);
    else return op_vec<DT, OP>(a, b);
}

// Fold one tree's program over the values load(rank) yields; returns the root's partial.
template <int DT, int OP, typename T, typename Load>
__device__ __forceinline__ T eval_tree_runtime(const TreeArgs& a, int t, T (*stk)[kTreeThreads], Load load) {
    const int N = a.nRanks;
    T top{};
    int sp = 0;                       // partials below `top`
    for (int i0 = 0; i0 < N; i0 += 8) {
        T v[8];
#pragma unroll
        for (int q = 0; q < 8; q++)
            if (i0 + q < N) v[q] = load(a.prog[t][i0 + q]);
#pragma unroll
        for (int q = 0; q < 8; q++) {
            if (i0 + q < N) {
                const int c = a.nchild[t][i0 + q];
                T acc = v[q];
                if (c == 2) {
                    acc = tree_op<DT, OP>(acc, stk[--sp][threadIdx.x]);   // child 0, below the top
                    acc = tree_op<DT, OP>(acc, top);                      // child 1, the top
                } else if (c == 1) {
                    acc = tree_op<DT, OP>(acc, top);
                } else if (i0 + q > 0) {
                    stk[sp++][threadIdx.x] = top;                         // a leaf: keep the old top
                }
                top = acc;
            }
        }
    }
    return top;
}

template <int DT, int OP, int VB>
__global__ void __launch_bounds__(kTreeThreads, 4)
k_allreduce_tree(const __grid_constant__ TreeArgs a) {
    static_assert(VB == 0 || VB == 16, "the run-time tree moves 16-byte vectors or elements");
    pdl_begin();
    constexpr int ESZ = DTypeOf<DT>::size;
    constexpr int U = VB ? VB / ESZ : 1;
    using VT = typename VecOf<16>::T;
    __shared__ VT vstk[VB ? kTreeStackDepth : 1][kTreeThreads];
    __shared__ uint32_t estk[kTreeStackDepth][kTreeThreads];
    const int N = a.nRanks;
    const size_t u0 = (a.split + U - 1) / U;
    const size_t u1 = (a.count - a.split + U - 1) / U;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t j = (size_t)blockIdx.x * blockDim.x + threadIdx.x; j < u0 + u1; j += stride) {
        const int t = j < u0 ? 0 : 1;
        const size_t lo = t == 0 ? 0 : a.split, hi = t == 0 ? a.split : a.count;
        const size_t e = lo + (j - (t == 0 ? 0 : u0)) * U;
        if (VB && e + U <= hi) {
            const VT acc = eval_tree_runtime<DT, OP, VT>(a, t, vstk, [&](int r) {
                return VecOf<16>::ld((const char*)a.send[r] + e * ESZ);
            });
            for (int r = 0; r < N; r++) VecOf<16>::st((char*)a.recv[r] + e * ESZ, acc);
        } else {
            for (size_t x = e; x < min(e + U, hi); x++) {
                const uint32_t acc = eval_tree_runtime<DT, OP, uint32_t>(a, t, estk, [&](int r) {
                    return ld_elem<ESZ>(a.send[r], x);
                });
                for (int r = 0; r < N; r++) st_elem<ESZ>(a.recv[r], x, acc);
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
    pdl_begin();
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

// ---- dispatch: NF > 0 is a compile-time rank count (vector paths only), NF = 0 the
// run-time kernels ------------------------------------------------------------------------

template <int DT, int OP, int NF>
static cudaError_t tree_launch_vec(const TreeArgs& a, int vb, int grid, int threads, cudaStream_t s) {
    if constexpr (NF > 0) {
        if (vb == 32) (void)pdl_launch(k_allreduce_tree_fixed<DT, OP, 32, NF>, grid, threads, 0, s, a);
        else if (vb == 16) (void)pdl_launch(k_allreduce_tree_fixed<DT, OP, 16, NF>, grid, threads, 0, s, a);
        else return cudaErrorInvalidValue;
    } else {
        // 16-byte vectors (32-byte alignment implies 16) in CTAs of at most kTreeThreads
        // threads, with the grid grown to keep the same number of threads per vector
        const long long scale = (long long)(vb == 32 ? 2 : 1) * (threads > kTreeThreads ? threads / kTreeThreads : 1);
        const int g = (int)std::min<long long>((long long)grid * scale, (long long)kMaxGridCtas);
        const int th = threads > kTreeThreads ? kTreeThreads : threads;
        if (vb != 0) (void)pdl_launch(k_allreduce_tree<DT, OP, 16>, g, th, 0, s, a);
        else (void)pdl_launch(k_allreduce_tree<DT, OP, 0>, g, th, 0, s, a);
    }
    return cudaGetLastError();
}

template <int DT, int NF>
static cudaError_t tree_launch_op(const TreeArgs& a, vRedOp_t op, int vb, int grid, int threads, cudaStream_t s) {
    switch (op) {
    case vSum: return tree_launch_vec<DT, kSum, NF>(a, vb, grid, threads, s);
    case vProd: return tree_launch_vec<DT, kProd, NF>(a, vb, grid, threads, s);
    case vMin: return tree_launch_vec<DT, kMin, NF>(a, vb, grid, threads, s);
    case vMax: return tree_launch_vec<DT, kMax, NF>(a, vb, grid, threads, s);
    }
    return cudaErrorInvalidValue;
}

template <int NF>
static cudaError_t tree_launch(const TreeArgs& a, vDataType_t dt, vRedOp_t op, int vb, int grid, int threads,
                               cudaStream_t s) {
    switch (dt) {
    case vFloat32: return tree_launch_op<kF32, NF>(a, op, vb, grid, threads, s);
    case vFloat16: return tree_launch_op<kF16, NF>(a, op, vb, grid, threads, s);
    case vBFloat16: return tree_launch_op<kBF16, NF>(a, op, vb, grid, threads, s);
    case vInt32: return tree_launch_op<kI32, NF>(a, op, vb, grid, threads, s);
    }
    return cudaErrorInvalidValue;
}

// The 2- and 4-rank vector kernels (k_tree_more.cu).
cudaError_t launch_allreduce_tree_more(const TreeArgs& a, vDataType_t dt, vRedOp_t op, int vb, int grid,
                                       int threads, cudaStream_t s);

}  // namespace vc
