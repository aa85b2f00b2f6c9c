// k_onepass.cu -- launch of the one-pass all-reduce (and reduce to root) and reduce-scatter
// kernels of onepass.cuh: compile-time instances for 8 ranks here, for 2 to 4 ranks in
// k_onepass_small.cu, the run-time rank count for every other case and the element path.
#include "onepass.cuh"

namespace vc {

cudaError_t launch_allreduce_onepass(const OnePassArgs& a, vDataType_t dt, vRedOp_t op, int vb,
                                     int grid, int threads, cudaStream_t s) {
    if (vb != 0 && a.nRanks == 8) return ar_launch<8>(a, dt, op, vb, grid, threads, s);
    if (vb != 0 && (a.nRanks >= 2 && a.nRanks <= 4))
        return launch_allreduce_onepass_small(a, dt, op, vb, grid, threads, s);
    return ar_launch<0>(a, dt, op, vb, grid, threads, s);
}

cudaError_t launch_reduce_scatter_onepass(const OnePassArgs& a, vDataType_t dt, vRedOp_t op,
                                          vDataType_t outType, int vb, int grid, int threads,
                                          cudaStream_t s) {
    // 2 to 4 and 8 ranks: compile-time instances of the vector paths and of the element
    // path (warp tiles of vectors that follow the inputs)
    if (a.nRanks == 8) return rs_launch<8>(a, dt, op, outType, vb, grid, threads, s);
    if (a.nRanks >= 2 && a.nRanks <= 4)
        return launch_reduce_scatter_onepass_small(a, dt, op, outType, vb, grid, threads, s);
    return rs_launch<0>(a, dt, op, outType, vb, grid, threads, s);
}

}  // namespace vc
