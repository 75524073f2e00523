// The fused decode kernel on 4-bit weights, instantiated for at most 1 token(s) (MAXT = 1).
#include "moe_decode_kernel.cuh"

namespace moe {

const void* decode_kernel_q4_maxt1(const Shapes& s) { return pick_shape<1, true>(s); }

}  // namespace moe
