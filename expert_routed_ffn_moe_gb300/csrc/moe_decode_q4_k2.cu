// The fused decode kernel on 4-bit weights, instantiated for at most 2 token(s) (MAXT = 2).
#include "moe_decode_kernel.cuh"

namespace moe {

const void* decode_kernel_q4_maxt2(const Shapes& s) { return pick_shape<2, true>(s); }

}  // namespace moe
