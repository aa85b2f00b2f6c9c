// k_onepass_small.cu -- the one-pass all-reduce and reduce-scatter vector kernels for 2,
// 3 and 4 ranks, with the rank count fixed at compile time.  The run-time kernel holds room
// for eight vectors per thread, so few threads fit on an SM; with two to four ranks that
// leaves too few bytes in flight to keep HBM busy.  These instances hold only the vectors
// they use.
#include "onepass.cuh"

namespace vc {

cudaError_t launch_allreduce_onepass_small(const OnePassArgs& a, vDataType_t dt, vRedOp_t op, int vb, int grid,
                                           int threads, cudaStream_t s) {
    if (a.nRanks == 2) return ar_launch<2>(a, dt, op, vb, grid, threads, s);
    if (a.nRanks == 3) return ar_launch<3>(a, dt, op, vb, grid, threads, s);
    if (a.nRanks == 4) return ar_launch<4>(a, dt, op, vb, grid, threads, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_reduce_scatter_onepass_small(const OnePassArgs& a, vDataType_t dt, vRedOp_t op,
                                                vDataType_t outType, int vb, int grid, int threads,
                                                cudaStream_t s) {
    if (a.nRanks == 2) return rs_launch<2>(a, dt, op, outType, vb, grid, threads, s);
    if (a.nRanks == 3) return rs_launch<3>(a, dt, op, outType, vb, grid, threads, s);
    if (a.nRanks == 4) return rs_launch<4>(a, dt, op, outType, vb, grid, threads, s);
    return cudaErrorInvalidValue;
}

}  // namespace vc
