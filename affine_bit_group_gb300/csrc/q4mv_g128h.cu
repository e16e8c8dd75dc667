// q4mv instantiations for one weight format: groups of 128 columns, bf16 or f16 scale and bias.
#include "q4mv_kernel.cuh"

namespace abg {
ABG_Q4MV_FORMAT_UNIT(g128h, 2, true)
}  // namespace abg
