// The fused decode kernel on 4-bit weights, instantiated for at most 8 token(s) (MAXT = 8).
#include "moe_decode_kernel.cuh"

namespace moe {

const void* decode_kernel_q4_maxt8(const Shapes& s) { return pick_shape<8, true>(s); }

}  // namespace moe
