// Fixed-shape instantiations of the product kernel (q4mv_kernel.cuh) for the
// common row lengths of 2048, 4096 and 6144 columns (groups of 64, f32 scale
// and bias staged in shared memory, block layout 0, 8 rows per item).  Their
// tile sizes and shared-memory offsets are compile-time constants, which
// removes the address arithmetic on run-time sizes from the product loop.
// The planner selects one only when a launch's plan has exactly that shape.
#include "q4mv_kernel.cuh"

namespace abg {

void *q4mv_select_fixed(int cols, bool tree) {
    switch (cols) {
    case 2048: return tree ? kernel_ptr<8, true, true, 0, 1, false, 2048>() : kernel_ptr<8, false, true, 0, 1, false, 2048>();
    case 4096: return tree ? kernel_ptr<8, true, true, 0, 1, false, 4096>() : kernel_ptr<8, false, true, 0, 1, false, 4096>();
    case 6144: return tree ? kernel_ptr<8, true, true, 0, 1, false, 6144>() : kernel_ptr<8, false, true, 0, 1, false, 6144>();
    default: return nullptr;
    }
}

cudaError_t q4mv_status_fixed(unsigned *bits, bool clear) { return read_status_word(bits, clear); }

}  // namespace abg
