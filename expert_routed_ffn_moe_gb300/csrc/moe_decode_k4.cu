// The fused decode kernel instantiated for at most 4 tokens (MAXT = 4).
#include "moe_decode_kernel.cuh"

namespace moe {

const void* decode_kernel_maxt4(const Shapes& s) { return pick_shape<4, false>(s); }

}  // namespace moe
