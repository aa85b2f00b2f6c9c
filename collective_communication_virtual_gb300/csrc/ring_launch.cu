// ring_launch.cu -- host side of the staged ring launch: co-residency query and the
// cooperative launch (every CTA of the ring waits on its neighbours, so all of them must
// be resident at once; a cooperative launch guarantees it or fails).
#include "internal.h"

namespace vc {

void* ring_kernel_simple(vDataType_t dt, vDataType_t out);
void* ring_kernel_ll(vDataType_t dt, vDataType_t out);
void* ring_kernel_ll128(vDataType_t dt, vDataType_t out);

static void* ring_kernel(vDataType_t dt, vDataType_t out, vProto_t proto) {
    switch (proto) {
    case vProtoSimple: return ring_kernel_simple(dt, out);
    case vProtoLL: return ring_kernel_ll(dt, out);
    case vProtoLL128: return ring_kernel_ll128(dt, out);
    default: return nullptr;
    }
}

cudaError_t ring_max_coresident(vDataType_t dt, vRedOp_t op, vDataType_t outType, vProto_t proto,
                                int threads, int smCount, int* maxCtas) {
    (void)op;
    void* k = ring_kernel(dt, outType, proto);
    if (!k) return cudaErrorInvalidValue;
    int perSm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&perSm, k, threads, 0);
    if (e != cudaSuccess) return e;
    *maxCtas = perSm * smCount;
    return cudaSuccess;
}

cudaError_t launch_ring(const RingArgs& a, vDataType_t dt, vRedOp_t op, vDataType_t outType,
                        vProto_t proto, int grid, int threads, cudaStream_t s) {
    (void)op;
    void* k = ring_kernel(dt, outType, proto);
    if (!k) return cudaErrorInvalidValue;
    void* args[] = {const_cast<RingArgs*>(&a)};
    return cudaLaunchCooperativeKernel(k, dim3(grid), dim3(threads), args, 0, s);
}

}  // namespace vc
