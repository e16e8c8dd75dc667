// q4mv instantiations for one weight format: groups of 32 columns, bf16 or f16 scale and bias.
#include "q4mv_kernel.cuh"

namespace abg {
ABG_Q4MV_FORMAT_UNIT(g32h, 0, true)
}  // namespace abg
