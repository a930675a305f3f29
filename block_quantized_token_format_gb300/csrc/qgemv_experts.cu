// Instantiations of the expert-grouped mat-vec kernel (every format, 1, 2 and 4 rows
// per warp; each kernel holds the bodies for ne = 1..4) and of the one-launch layer.
#include "qgemv_experts.cuh"

namespace qg {

const void* expert_kernel_lookup(int fmt, int rpw) {
#define QG_X(F)                                                            \
    if (fmt == F) {                                                        \
        if (rpw == 1) return (const void*)&qgemv_experts_kernel<F, 1>;     \
        if (rpw == 2) return (const void*)&qgemv_experts_kernel<F, 2>;     \
        if (rpw == 4) return (const void*)&qgemv_experts_kernel<F, 4>;     \
        return nullptr;                                                    \
    }
    QG_X(QG_Q8_0) QG_X(QG_Q4_0) QG_X(QG_AFFINE4_G64) QG_X(QG_BF16)
#undef QG_X
    return nullptr;
}

// The one-launch layer: gate/up pairs need an even number of rows per warp.
const void* expert_layer_kernel_lookup(int fmt, int rpw) {
#define QG_L(F)                                                                \
    if (fmt == F) {                                                            \
        if (rpw == 2) return (const void*)&qgemv_expert_layer_kernel<F, 2>;    \
        if (rpw == 4) return (const void*)&qgemv_expert_layer_kernel<F, 4>;    \
        return nullptr;                                                        \
    }
    QG_L(QG_Q8_0) QG_L(QG_Q4_0) QG_L(QG_AFFINE4_G64) QG_L(QG_BF16)
#undef QG_L
    return nullptr;
}

}  // namespace qg
