// Fixed-shape instantiations of the product kernel (q4mv_kernel.cuh) for
// groups of 32 columns (scale and bias as f32, bf16 or f16, staged in shared
// memory), for the row lengths of 2048, 4096 and 6144 columns: the same
// layouts and compile-time tile shapes as the 64-column groups of
// q4mv_fixed.cu (but the 18-warp layout of 6144 columns), in a unit of their
// own so the units compile in parallel.
// The planner selects one only when a launch's plan has exactly that shape.
#include "q4mv_kernel.cuh"

namespace abg {

namespace {

template <int R, int L, bool H>
void *select_g32(int cols, bool tree) {
    switch (cols) {
    case 2048: return tree ? kernel_ptr<R, true, true, L, 0, H, 2048>() : kernel_ptr<R, false, true, L, 0, H, 2048>();
    case 4096: return tree ? kernel_ptr<R, true, true, L, 0, H, 4096>() : kernel_ptr<R, false, true, L, 0, H, 4096>();
    case 6144: return tree ? kernel_ptr<R, true, true, L, 0, H, 6144>() : kernel_ptr<R, false, true, L, 0, H, 6144>();
    default: return nullptr;
    }
}

template <bool H>
void *select_g32_layout(int cols, bool tree, int R, int layout) {
    if (R == 8 && layout == 0) return select_g32<8, 0, H>(cols, tree);
    if (R == 4 && layout == 1) return select_g32<4, 1, H>(cols, tree);
    return nullptr;  // (no 18-warp layout for 6144 columns: at 32-column groups it spills)
}

}  // namespace

void *q4mv_select_fixed_g32(int cols, bool tree, int R, int layout, bool half) {
    return half ? select_g32_layout<true>(cols, tree, R, layout) : select_g32_layout<false>(cols, tree, R, layout);
}

cudaError_t q4mv_status_fixed_g32(unsigned *bits, bool clear) { return read_status_word(bits, clear); }

}  // namespace abg
