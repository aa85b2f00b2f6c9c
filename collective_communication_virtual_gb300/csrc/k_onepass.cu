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
    const bool twoByte = dt == vFloat16 || dt == vBFloat16;
    if (a.nRanks == 8 && (vb != 0 || twoByte)) return rs_launch<8>(a, dt, op, outType, vb, grid, threads, s);
    // 2 to 4 ranks: the vector paths, and the 2-byte element path (two vectors that follow
    // the inputs per thread)
    const bool small = a.nRanks >= 2 && a.nRanks <= 4;
    if (small && (vb != 0 || twoByte))
        return launch_reduce_scatter_onepass_small(a, dt, op, outType, vb, grid, threads, s);
    return rs_launch<0>(a, dt, op, outType, vb, grid, threads, s);
}

}  // namespace vc
