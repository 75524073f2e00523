// The fused decode kernel instantiated for at most 2 tokens (MAXT = 2).
#include "moe_decode_kernel.cuh"

namespace moe {

const void* decode_kernel_maxt2(const Shapes& s) { return pick_shape<2, false>(s); }

}  // namespace moe
