// k_ring_ll.cu -- staged ring kernels with the ll protocol (one translation unit per
// protocol so the three compile in parallel).
#include "ring_impl.cuh"

namespace vc {
VC_RING_SELECTOR(ring_kernel_ll, vProtoLL)
}  // namespace vc
