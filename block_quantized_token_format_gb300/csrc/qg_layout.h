// Byte layouts of the four weight formats, shared by the host packer and the
// CUDA launch code.  Canonical layout = the formats' stored bytes; device
// layout = rows one after the other, each row a run of 16-byte-aligned steps
// of [512 B of codes][their scales][pad], so every row starts on a 16-byte
// boundary, step k of RPW consecutive rows is one box of a 2-D tensor copy
// ([n_out][row stride / 8] elements of 8 bytes), and a row prefix of a packed
// matrix is a packed matrix.
#pragma once

#include <cstdint>
#include <cstddef>

#include "../../include/qgemv.h"

namespace qg {

constexpr int kMaxNtok = 4;
constexpr int kChunkWeights = 16;   // weights per lane-chunk in every kernel

inline bool fmt_valid(int fmt) { return fmt >= QG_Q8_0 && fmt <= QG_Q5_0; }

// n_in must be a positive multiple of this.
inline int64_t n_in_multiple(int fmt) {
    switch (fmt) {
        case QG_Q8_0: case QG_Q4_0: case QG_Q5_0: return 32;
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

// Bytes of one row's codes.
inline int64_t codes_bytes(int fmt, int64_t n_in) {
    switch (fmt) {
        case QG_Q8_0: return n_in;
        case QG_Q4_0: case QG_AFFINE4_G64: case QG_Q5_0: return n_in / 2;
        case QG_BF16: return 2 * n_in;
        default: return 0;
    }
}

// Scale (and bias) bytes that belong to `codes` bytes of codes.
inline int64_t scale_bytes_for(int fmt, int64_t codes) {
    switch (fmt) {
        case QG_Q8_0: return codes / 16;         // one fp16 d per 32 one-byte codes
        case QG_Q4_0: return codes / 8;          // one fp16 d per 16 bytes of nibbles
        case QG_AFFINE4_G64: return codes / 8;   // one (fp16 s, fp16 b) per 32 bytes of nibbles
        case QG_Q5_0: return codes / 16 * 6;     // one (uint32 fifth bits, fp16 d) per 16 bytes of nibbles
        default: return 0;
    }
}

// Canonical (= weight) bytes of one row.
inline int64_t canonical_row_bytes(int fmt, int64_t n_in) {
    const int64_t c = codes_bytes(fmt, n_in);
    return c + scale_bytes_for(fmt, c);
}

// Device layout: every row is a run of steps; a step holds 512 bytes of codes
// (one 16-byte chunk per lane of a warp) followed by the scales of exactly those
// codes, padded to 16 bytes.  Only a row's last step can be shorter.
constexpr int64_t kStepCodeBytes = 512;

inline int64_t steps_per_row(int fmt, int64_t n_in) {
    return (codes_bytes(fmt, n_in) + kStepCodeBytes - 1) / kStepCodeBytes;
}
inline int64_t round16(int64_t b) { return (b + 15) / 16 * 16; }
inline int64_t full_step_bytes(int fmt) { return kStepCodeBytes + scale_bytes_for(fmt, kStepCodeBytes); }
inline int64_t last_step_codes(int fmt, int64_t n_in) {
    return codes_bytes(fmt, n_in) - kStepCodeBytes * (steps_per_row(fmt, n_in) - 1);
}
inline int64_t last_step_bytes(int fmt, int64_t n_in) {
    const int64_t c = last_step_codes(fmt, n_in);
    return round16(c + scale_bytes_for(fmt, c));
}
inline int64_t row_stride(int fmt, int64_t n_in) {
    return (steps_per_row(fmt, n_in) - 1) * full_step_bytes(fmt) + last_step_bytes(fmt, n_in);
}

}  // namespace qg
