// k_tree_more.cu -- the double-binary-tree all-reduce vector kernels for 2 and 4 ranks,
// with the tree program a compile-time constant.  The run-time kernel loads 16 bytes of
// each rank per thread, which at two or four ranks leaves too few bytes in flight (0.73
// and 0.95 of the copy bandwidth on GB300, against 0.96 and 1.01 here).
#include "tree.cuh"

namespace vc {

cudaError_t launch_allreduce_tree_more(const TreeArgs& a, vDataType_t dt, vRedOp_t op, int vb, int grid,
                                       int threads, cudaStream_t s) {
    if (a.nRanks == 2) return tree_launch<2>(a, dt, op, vb, grid, threads, s);
    if (a.nRanks == 4) return tree_launch<4>(a, dt, op, vb, grid, threads, s);
    return cudaErrorInvalidValue;
}

}  // namespace vc
