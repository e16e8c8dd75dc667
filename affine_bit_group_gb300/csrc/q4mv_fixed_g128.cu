// Fixed-shape instantiations of the product kernel (q4mv_kernel.cuh) for
// groups of 128 columns (scale and bias as f32, bf16 or f16, staged in shared
// memory), for the row lengths of 2048, 4096 and 6144 columns: the same
// layouts and compile-time tile shapes as the 64-column groups of
// q4mv_fixed.cu, in a unit of their own so the units compile in parallel.
// The planner selects one only when a launch's plan has exactly that shape.
#include "q4mv_kernel.cuh"

namespace abg {

namespace {

template <int R, int L, bool H>
void *select_g128(int cols, bool tree) {
    switch (cols) {
    case 2048: return tree ? kernel_ptr<R, true, true, L, 2, H, 2048>() : kernel_ptr<R, false, true, L, 2, H, 2048>();
    case 4096: return tree ? kernel_ptr<R, true, true, L, 2, H, 4096>() : kernel_ptr<R, false, true, L, 2, H, 4096>();
    case 6144: return tree ? kernel_ptr<R, true, true, L, 2, H, 6144>() : kernel_ptr<R, false, true, L, 2, H, 6144>();
    default: return nullptr;
    }
}

template <bool H>
void *select_g128_layout(int cols, bool tree, int R, int layout) {
    if (R == 8 && layout == 0) return select_g128<8, 0, H>(cols, tree);
    if (R == 4 && layout == 1) return select_g128<4, 1, H>(cols, tree);
    if (R == 8 && layout == 4 && cols == 6144)
        return tree ? kernel_ptr<8, true, true, 4, 2, H, 6144>() : kernel_ptr<8, false, true, 4, 2, H, 6144>();
    return nullptr;
}

}  // namespace

void *q4mv_select_fixed_g128(int cols, bool tree, int R, int layout, bool half) {
    return half ? select_g128_layout<true>(cols, tree, R, layout) : select_g128_layout<false>(cols, tree, R, layout);
}

cudaError_t q4mv_status_fixed_g128(unsigned *bits, bool clear) { return read_status_word(bits, clear); }

}  // namespace abg
