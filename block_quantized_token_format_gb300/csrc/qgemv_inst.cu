// Instantiations of the dequant-GEMV kernel for one weight format, selected at
// compile time by QG_INST_FMT (the build compiles this file once per format so
// the formats build in parallel).
#include "qgemv_kernels.cuh"

#ifndef QG_INST_FMT
#error "compile with -DQG_INST_FMT=<0..4>"
#endif

#define QG_CAT2(a, b) a##b
#define QG_CAT(a, b) QG_CAT2(a, b)

namespace qg {

const void* QG_CAT(kernel_lookup_fmt, QG_INST_FMT)(int ntok, int rpw, bool argmax, bool split) {
#define QG_K(NT, R, A) (split ? (const void*)&qgemv_kernel<QG_INST_FMT, NT, R, A, true>       \
                              : (const void*)&qgemv_kernel<QG_INST_FMT, NT, R, A, false>)
#define QG_E(NT, R) \
    if (ntok == NT && rpw == R) return argmax ? QG_K(NT, R, true) : QG_K(NT, R, false);
#define QG_E_NT(NT) QG_E(NT, 1) QG_E(NT, 2) QG_E(NT, 4)
    QG_E_NT(1) QG_E_NT(2) QG_E_NT(3) QG_E_NT(4)
    QG_E(1, 8)                 // 8 rows per warp: ntok 1 and 2
    QG_E(2, 8)
    QG_E(2, 6) QG_E(3, 6)      // 6 rows per warp: ntok 2-3
    QG_E(4, 3) QG_E(4, 5)      // 3 and 5 rows per warp: ntok 4
    QG_E(3, 8) QG_E(4, 6)      // more than 20 outputs: at most 12 warps, 168 registers
#undef QG_E_NT
#undef QG_E
#undef QG_K
    return nullptr;
}

}  // namespace qg
