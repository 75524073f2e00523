// The fused decode kernel on 4-bit weights, instantiated for at most 4 token(s) (MAXT = 4).
#include "moe_decode_kernel.cuh"

namespace moe {

const void* decode_kernel_q4_maxt4(const Shapes& s) { return pick_shape<4, true>(s); }

}  // namespace moe
