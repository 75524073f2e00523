// The fused decode kernel instantiated for at most 16 tokens (MAXT = 16).
#include "moe_decode_kernel.cuh"

namespace moe {

const void* decode_kernel_maxt16(const Shapes& s) { return pick_shape<16, false>(s); }

}  // namespace moe
