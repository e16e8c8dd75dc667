// q4mv instantiations for one weight format: groups of 128 columns, f32 scale and bias.
#include "q4mv_kernel.cuh"

namespace abg {
ABG_Q4MV_FORMAT_UNIT(g128, 2, false)
}  // namespace abg
