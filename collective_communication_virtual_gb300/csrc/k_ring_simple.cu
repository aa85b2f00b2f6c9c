// k_ring_simple.cu -- staged ring kernels with the simple protocol (one translation unit per
// protocol so the three compile in parallel).
#include "ring_impl.cuh"

namespace vc {
VC_RING_SELECTOR(ring_kernel_simple, vProtoSimple)
}  // namespace vc
