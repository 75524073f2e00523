// The fused decode kernel instantiated for at most 8 tokens (MAXT = 8).
#include "moe_decode_kernel.cuh"

namespace moe {

const void* decode_kernel_maxt8(const Shapes& s) { return pick_shape<8, false>(s); }

}  // namespace moe
