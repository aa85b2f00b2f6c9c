// k_ring_ll128.cu -- staged ring kernels with the ll128 protocol (one translation unit per
// protocol so the three compile in parallel).
#include "ring_impl.cuh"

namespace vc {
VC_RING_SELECTOR(ring_kernel_ll128, vProtoLL128)
}  // namespace vc
