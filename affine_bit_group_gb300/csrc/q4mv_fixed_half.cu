// Fixed-shape instantiations of the product kernel (q4mv_kernel.cuh) for
// scale and bias stored as bf16 or f16 (groups of 64 columns, staged in shared
// memory; MLX stores them in the model's 16-bit type), for the row lengths of
// 2048, 4096 and 6144 columns: the same layouts and compile-time tile shapes
// as the f32 instantiations of q4mv_fixed.cu, in a unit of their own so the
// two compile in parallel.  The planner selects one only when a launch's plan
// has exactly that shape.
#include "q4mv_kernel.cuh"

namespace abg {

// rows per item R and block layout: (8, 0) for launches of many tiles, (4, 1)
// for launches of few tiles (16 computing warps, one block per SM), and for
// rows of 6144 columns in launches of many tiles (8, 4) (18 computing warps,
// one block per SM)
template <int R, int L>
void *select_fixed_half(int cols, bool tree) {
    switch (cols) {
    case 2048: return tree ? kernel_ptr<R, true, true, L, 1, true, 2048>() : kernel_ptr<R, false, true, L, 1, true, 2048>();
    case 4096: return tree ? kernel_ptr<R, true, true, L, 1, true, 4096>() : kernel_ptr<R, false, true, L, 1, true, 4096>();
    case 6144: return tree ? kernel_ptr<R, true, true, L, 1, true, 6144>() : kernel_ptr<R, false, true, L, 1, true, 6144>();
    default: return nullptr;
    }
}

void *q4mv_select_fixed_half(int cols, bool tree, int R, int layout) {
    if (R == 8 && layout == 0) return select_fixed_half<8, 0>(cols, tree);
    if (R == 4 && layout == 1) return select_fixed_half<4, 1>(cols, tree);
    if (R == 8 && layout == 4 && cols == 6144)
        return tree ? kernel_ptr<8, true, true, 4, 1, true, 6144>() : kernel_ptr<8, false, true, 4, 1, true, 6144>();
    return nullptr;
}

cudaError_t q4mv_status_fixed_half(unsigned *bits, bool clear) { return read_status_word(bits, clear); }

}  // namespace abg
