// k_tree_more.cu -- the double-binary-tree all-reduce vector kernels for 2, 4 and 16
// ranks, with the tree program a compile-time constant.  The run-time kernel keeps every
// rank's vector and its evaluation stack in local memory, because their indices come
// from the program; with the program fixed, the indices are constants and the vectors
// stay in registers.
#include "tree.cuh"

namespace vc {

cudaError_t launch_allreduce_tree_more(const TreeArgs& a, vDataType_t dt, vRedOp_t op, int vb, int grid,
                                       int threads, cudaStream_t s) {
    if (a.nRanks == 2) return tree_launch<2>(a, dt, op, vb, grid, threads, s);
    if (a.nRanks == 4) return tree_launch<4>(a, dt, op, vb, grid, threads, s);
    if (a.nRanks == 16) return tree_launch<16>(a, dt, op, vb, grid, threads, s);
    return cudaErrorInvalidValue;
}

}  // namespace vc
