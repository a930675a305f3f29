// Byte layouts of the four weight formats, shared by the host packer and the
// CUDA launch code.  Canonical layout = the formats' stored bytes; device
// layout = row-interleaved [codes][scales][pad to 16 B] so every row starts on
// a 16-byte boundary and a row prefix of a packed matrix is a packed matrix.
#pragma once

#include <cstdint>
#include <cstddef>

#include "../../include/qgemv.h"

namespace qg {

constexpr int kMaxNtok = 4;
constexpr int kChunkWeights = 16;   // weights per lane-chunk in every kernel

inline bool fmt_valid(int fmt) { return fmt >= QG_Q8_0 && fmt <= QG_BF16; }

// n_in must be a positive multiple of this.
inline int64_t n_in_multiple(int fmt) {
    switch (fmt) {
        case QG_Q8_0: case QG_Q4_0: return 32;
        case QG_AFFINE4_G64: return 64;
        case QG_BF16: return 16;          // one lane-chunk of 16 weights
        default: return 0;
    }
}

inline bool shape_valid(int fmt, int64_t n_out, int64_t n_in) {
    if (!fmt_valid(fmt) || n_out < 1 || n_in < 1) return false;
    if (n_out > (int64_t(1) << 31) - 1 || n_in > (int64_t(1) << 24)) return false;
    return n_in % n_in_multiple(fmt) == 0;
}

// Bytes of one row's codes in the device layout.
inline int64_t codes_bytes(int fmt, int64_t n_in) {
    switch (fmt) {
        case QG_Q8_0: return n_in;
        case QG_Q4_0: case QG_AFFINE4_G64: return n_in / 2;
        case QG_BF16: return 2 * n_in;
        default: return 0;
    }
}

// Bytes of one row's scales (and biases) in the device layout.
inline int64_t scales_bytes(int fmt, int64_t n_in) {
    switch (fmt) {
        case QG_Q8_0: case QG_Q4_0: return (n_in / 32) * 2;
        case QG_AFFINE4_G64: return (n_in / 64) * 4;
        default: return 0;
    }
}

// Canonical (= weight) bytes of one row.
inline int64_t canonical_row_bytes(int fmt, int64_t n_in) {
    return codes_bytes(fmt, n_in) + scales_bytes(fmt, n_in);
}

inline int64_t row_stride(int fmt, int64_t n_in) {
    int64_t b = canonical_row_bytes(fmt, n_in);
    return (b + 15) / 16 * 16;
}

}  // namespace qg
