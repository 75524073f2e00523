// The fused decode kernel on 4-bit weights, instantiated for at most 16 token(s) (MAXT = 16).
#include "moe_decode_kernel.cuh"

namespace moe {

const void* decode_kernel_q4_maxt16(const Shapes& s) { return pick_shape<16, true>(s); }

}  // namespace moe
