// k_tree.cu -- launch of the double-binary-tree all-reduce kernels of tree.cuh: the
// compile-time program for 8 ranks here, for 2 and 4 ranks in k_tree_more.cu, the
// run-time program for every other rank count and for the element path.
#include "tree.cuh"

namespace vc {

cudaError_t launch_allreduce_tree(const TreeArgs& a, vDataType_t dt, vRedOp_t op, int vb, int grid,
                                  int threads, cudaStream_t s) {
    if (vb != 0 && a.nRanks == 8) return tree_launch<8>(a, dt, op, vb, grid, threads, s);
    if (vb != 0 && (a.nRanks == 2 || a.nRanks == 4))
        return launch_allreduce_tree_more(a, dt, op, vb, grid, threads, s);
    return tree_launch<0>(a, dt, op, vb, grid, threads, s);
}

}  // namespace vc
