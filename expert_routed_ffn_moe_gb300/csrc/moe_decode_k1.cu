// The fused decode kernel instantiated for at most 1 token (MAXT = 1).
#include "moe_decode_kernel.cuh"

namespace moe {

const void* decode_kernel_maxt1(const Shapes& s) { return pick_shape<1, false>(s); }

}  // namespace moe
