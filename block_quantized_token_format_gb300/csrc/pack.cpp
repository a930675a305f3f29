// Host weight packer: fp32 -> canonical block bytes -> device layout.
//
// The quantizer rules are the workload definitions of the formats
// (Q8_0 / Q4_0 named in "Where the time goes on an M2 Max", format table, and
// the opus-mtp-turbo Track 1 report, item 3; the MLX-style affine 4-bit head
// in "perf(speculative): cut the MTP drafter's per-step cost", section "The
// cost model"); the include/qgemv.h comment spells each one out.  All
// arithmetic that decides a code is IEEE fp32 (this file is compiled with
// -ffp-contract=off), so the bytes are the same on every host.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

#include "qg_layout.h"

namespace {

inline uint32_t f32_bits(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }
inline float bits_f32(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }

// IEEE binary32 -> binary16, round to nearest, ties to even (subnormals, inf, nan).
uint16_t f32_to_f16(float f) {
    const uint32_t x = f32_bits(f);
    const uint32_t sign = (x >> 16) & 0x8000u;
    const uint32_t a = x & 0x7FFFFFFFu;
    if (a >= 0x7F800000u) return uint16_t(sign | 0x7C00u | (a > 0x7F800000u ? 0x200u : 0u));
    if (a >= 0x477FF000u) return uint16_t(sign | 0x7C00u);          // >= 65520 rounds to inf
    if (a < 0x38800000u) {                                          // below 2^-14: subnormal half
        if (a < 0x33000000u) return uint16_t(sign);                 // below 2^-25: zero
        const uint32_t e = a >> 23;                                 // 102..112
        const uint32_t m = (a & 0x7FFFFFu) | 0x800000u;
        const uint32_t shift = 126u - e;                            // 14..24
        uint32_t k = m >> shift;
        const uint32_t rem = m & ((1u << shift) - 1u);
        const uint32_t half = 1u << (shift - 1u);
        if (rem > half || (rem == half && (k & 1u))) ++k;
        return uint16_t(sign | k);
    }
    uint32_t r = a - 0x38000000u;                                   // rebias 127 -> 15
    r += 0xFFFu + ((r >> 13) & 1u);
    return uint16_t(sign | (r >> 13));
}

float f16_to_f32(uint16_t h) {
    const uint32_t sign = uint32_t(h & 0x8000u) << 16;
    const uint32_t e = (h >> 10) & 0x1Fu, m = h & 0x3FFu;
    if (e == 0) {
        float v = std::ldexp(float(m), -24);
        return sign ? -v : v;
    }
    if (e == 31) return bits_f32(sign | 0x7F800000u | (m << 13));
    return bits_f32(sign | ((e + 112u) << 23) | (m << 13));
}

uint16_t f32_to_bf16(float f) {
    const uint32_t u = f32_bits(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return uint16_t((u >> 16) | 0x40u);   // quiet NaN
    return uint16_t((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

inline void put16(uint8_t* p, uint16_t v) { p[0] = uint8_t(v); p[1] = uint8_t(v >> 8); }
inline void put32(uint8_t* p, uint32_t v) { for (int i = 0; i < 4; ++i) p[i] = uint8_t(v >> (8 * i)); }

// ------------------------------------------------------------------ one row, fp32 -> canonical

void quant_row_q8_0(const float* w, int64_t n_in, uint8_t* out) {
    for (int64_t b = 0; b < n_in / 32; ++b) {
        const float* v = w + 32 * b;
        float amax = 0.f;
        for (int j = 0; j < 32; ++j) amax = std::max(amax, std::fabs(v[j]));
        const float d = amax / 127.0f;
        uint8_t* blk = out + 34 * b;
        put16(blk, f32_to_f16(d));
        for (int j = 0; j < 32; ++j) {
            float q = d > 0.f ? std::roundf(v[j] / d) : 0.f;
            q = std::min(127.f, std::max(-127.f, q));
            blk[2 + j] = uint8_t(int8_t(q));
        }
    }
}

void quant_row_q4_0(const float* w, int64_t n_in, uint8_t* out) {
    for (int64_t b = 0; b < n_in / 32; ++b) {
        const float* v = w + 32 * b;
        float m = 0.f, amax = -1.f;
        for (int j = 0; j < 32; ++j)
            if (std::fabs(v[j]) > amax) { amax = std::fabs(v[j]); m = v[j]; }   // first on ties
        const float d = m / -8.0f;
        uint8_t q[32];
        for (int j = 0; j < 32; ++j) {
            float c = d != 0.f ? std::roundf(v[j] / d) + 8.f : 8.f;
            q[j] = uint8_t(std::min(15.f, std::max(0.f, c)));
        }
        uint8_t* blk = out + 18 * b;
        put16(blk, f32_to_f16(d));
        for (int j = 0; j < 16; ++j) blk[2 + j] = uint8_t(q[j] | (q[j + 16] << 4));
    }
}

// Q5_0: the Q4_0 rule with 5-bit codes (d = m / -16, q = clamp(roundf(w/d) + 16, 0, 31)).
void quant_row_q5_0(const float* w, int64_t n_in, uint8_t* out) {
    for (int64_t b = 0; b < n_in / 32; ++b) {
        const float* v = w + 32 * b;
        float m = 0.f, amax = -1.f;
        for (int j = 0; j < 32; ++j)
            if (std::fabs(v[j]) > amax) { amax = std::fabs(v[j]); m = v[j]; }   // first on ties
        const float d = m / -16.0f;
        uint8_t q[32];
        uint32_t qh = 0;
        for (int j = 0; j < 32; ++j) {
            float c = d != 0.f ? std::roundf(v[j] / d) + 16.f : 16.f;
            q[j] = uint8_t(std::min(31.f, std::max(0.f, c)));
            qh |= uint32_t(q[j] >> 4) << j;
        }
        uint8_t* blk = out + 22 * b;
        put16(blk, f32_to_f16(d));
        put32(blk + 2, qh);
        for (int j = 0; j < 16; ++j) blk[6 + j] = uint8_t((q[j] & 0xF) | ((q[j + 16] & 0xF) << 4));
    }
}

// Affine rows write into three planes: words, scales, biases.
void quant_row_affine4(const float* w, int64_t n_in, uint8_t* words, uint8_t* scales, uint8_t* biases) {
    for (int64_t g = 0; g < n_in / 64; ++g) {
        const float* v = w + 64 * g;
        float mn = v[0], mx = v[0];
        for (int j = 1; j < 64; ++j) { mn = std::min(mn, v[j]); mx = std::max(mx, v[j]); }
        const uint16_t s16 = f32_to_f16((mx - mn) / 15.0f);
        const uint16_t b16 = f32_to_f16(mn);
        const float s = f16_to_f32(s16), bb = f16_to_f32(b16);
        put16(scales + 2 * g, s16);
        put16(biases + 2 * g, b16);
        for (int k = 0; k < 8; ++k) {
            uint32_t word = 0;
            for (int e = 0; e < 8; ++e) {
                float c = s != 0.f ? std::roundf((v[8 * k + e] - bb) / s) : 0.f;
                c = std::min(15.f, std::max(0.f, c));
                word |= uint32_t(c) << (4 * e);
            }
            put32(words + 4 * (8 * g + k), word);
        }
    }
}

void quant_row_bf16(const float* w, int64_t n_in, uint8_t* out) {
    for (int64_t i = 0; i < n_in; ++i) put16(out + 2 * i, f32_to_bf16(w[i]));
}

// ------------------------------------------------------------------ one row, canonical -> device

// Canonical row pointers (affine has three planes).
struct CanonRow { const uint8_t* a; const uint8_t* s; const uint8_t* b; };

// Q5_0 device record: the fifth bit of element e of a block sits at bit 8b + g of the
// record's word, where g = 2 * (e / 8) + (e % 2) numbers the block's 8 groups of 4
// elements (the even or the odd elements of each 8-element code word) and b = (e % 8) / 2
// is the element's place in its group.  Shifting the word left by 4 - g (right by g - 4)
// and masking with 0x10101010 puts the group's 4 fifth bits at bit 4 of the 4 bytes that
// hold the group's codes in the kernels' integer decode; the 32 positions are distinct.
int q5_fifth_bit_pos(int e) {
    const int g = 2 * (e >> 3) + (e & 1), b = (e & 7) >> 1;
    return 8 * b + g;
}

// The row's codes (device byte / nibble order) followed by all its scales.
void flat_device_row(int fmt, CanonRow c, int64_t n_in, uint8_t* dst) {
    const int64_t cb = qg::codes_bytes(fmt, n_in);
    switch (fmt) {
        case QG_Q8_0:
            for (int64_t b = 0; b < n_in / 32; ++b) {
                const uint8_t* blk = c.a + 34 * b;
                std::memcpy(dst + cb + 2 * b, blk, 2);
                for (int j = 0; j < 32; ++j) dst[32 * b + j] = uint8_t(blk[2 + j] ^ 0x80u);   // q + 128
            }
            break;
        case QG_Q4_0:
            for (int64_t b = 0; b < n_in / 32; ++b) {
                const uint8_t* blk = c.a + 18 * b;
                std::memcpy(dst + cb + 2 * b, blk, 2);
                uint8_t q[32];
                for (int j = 0; j < 16; ++j) { q[j] = blk[2 + j] & 0xF; q[j + 16] = blk[2 + j] >> 4; }
                for (int m = 0; m < 4; ++m) {
                    uint32_t word = 0;
                    for (int e = 0; e < 8; ++e) word |= uint32_t(q[8 * m + e]) << (4 * e);
                    put32(dst + 16 * b + 4 * m, word);
                }
            }
            break;
        case QG_AFFINE4_G64:
            std::memcpy(dst, c.a, size_t(cb));
            for (int64_t g = 0; g < n_in / 64; ++g) {
                std::memcpy(dst + cb + 4 * g, c.s + 2 * g, 2);
                std::memcpy(dst + cb + 4 * g + 2, c.b + 2 * g, 2);
            }
            break;
        case QG_BF16:
            std::memcpy(dst, c.a, size_t(cb));
            break;
        case QG_Q5_0:
            // codes: the low nibbles as Q4_0's words; scales: per block its fifth bits
            // (a uint32 in the order of q5_fifth_bit_pos) and then its fp16 d, 6 bytes.
            for (int64_t b = 0; b < n_in / 32; ++b) {
                const uint8_t* blk = c.a + 22 * b;
                const uint32_t qh = uint32_t(blk[2]) | uint32_t(blk[3]) << 8 | uint32_t(blk[4]) << 16 |
                                    uint32_t(blk[5]) << 24;
                uint32_t rot = 0;
                for (int e = 0; e < 32; ++e) rot |= ((qh >> e) & 1u) << q5_fifth_bit_pos(e);
                put32(dst + cb + 6 * b, rot);
                std::memcpy(dst + cb + 6 * b + 4, blk, 2);
                uint8_t q[32];
                for (int j = 0; j < 16; ++j) { q[j] = blk[6 + j] & 0xF; q[j + 16] = blk[6 + j] >> 4; }
                for (int m = 0; m < 4; ++m) {
                    uint32_t word = 0;
                    for (int e = 0; e < 8; ++e) word |= uint32_t(q[8 * m + e]) << (4 * e);
                    put32(dst + 16 * b + 4 * m, word);
                }
            }
            break;
    }
}

// Scatter a flat [codes][scales] row into its steps of [512 B codes][their scales][pad].
void device_row(int fmt, CanonRow c, int64_t n_in, uint8_t* dst, int64_t stride) {
    thread_local std::vector<uint8_t> flat;
    const int64_t cb = qg::codes_bytes(fmt, n_in);
    flat.assign(size_t(qg::canonical_row_bytes(fmt, n_in)), 0);
    flat_device_row(fmt, c, n_in, flat.data());
    std::memset(dst, 0, size_t(stride));
    const int64_t full = qg::full_step_bytes(fmt);
    for (int64_t k = 0; k < qg::steps_per_row(fmt, n_in); ++k) {
        const int64_t c0 = qg::kStepCodeBytes * k;
        const int64_t ck = std::min(qg::kStepCodeBytes, cb - c0);
        std::memcpy(dst + k * full, flat.data() + c0, size_t(ck));
        std::memcpy(dst + k * full + ck, flat.data() + cb + qg::scale_bytes_for(fmt, c0),
                    size_t(qg::scale_bytes_for(fmt, ck)));
    }
}

CanonRow canon_row(int fmt, const uint8_t* canon, int64_t n_out, int64_t n_in, int64_t r) {
    if (fmt == QG_AFFINE4_G64) {
        const int64_t wb = n_in / 2, sb = (n_in / 64) * 2;
        return {canon + r * wb, canon + n_out * wb + r * sb, canon + n_out * (wb + sb) + r * sb};
    }
    return {canon + r * qg::canonical_row_bytes(fmt, n_in), nullptr, nullptr};
}

void quant_row(int fmt, const float* w, int64_t n_in, uint8_t* canon, int64_t n_out, int64_t r) {
    if (fmt == QG_AFFINE4_G64) {
        const int64_t wb = n_in / 2, sb = (n_in / 64) * 2;
        quant_row_affine4(w, n_in, canon + r * wb, canon + n_out * wb + r * sb,
                          canon + n_out * (wb + sb) + r * sb);
        return;
    }
    uint8_t* out = canon + r * qg::canonical_row_bytes(fmt, n_in);
    if (fmt == QG_Q8_0) quant_row_q8_0(w, n_in, out);
    else if (fmt == QG_Q4_0) quant_row_q4_0(w, n_in, out);
    else if (fmt == QG_Q5_0) quant_row_q5_0(w, n_in, out);
    else quant_row_bf16(w, n_in, out);
}

template <class F>
void parallel_rows(int64_t n_out, int64_t work_per_row, F&& fn) {
    unsigned hw = std::max(1u, std::thread::hardware_concurrency());
    int64_t want = std::max<int64_t>(1, (n_out * work_per_row) / (1 << 20));
    int nt = int(std::min<int64_t>({int64_t(hw), want, n_out, 64}));
    if (nt <= 1) { fn(int64_t(0), n_out); return; }
    std::vector<std::thread> th;
    for (int t = 0; t < nt; ++t) {
        int64_t r0 = n_out * t / nt, r1 = n_out * (t + 1) / nt;
        th.emplace_back([=, &fn] { fn(r0, r1); });
    }
    for (auto& x : th) x.join();
}

}  // namespace

extern "C" {

size_t qg_canonical_bytes(qg_fmt fmt, int64_t n_out, int64_t n_in) {
    if (!qg::shape_valid(fmt, n_out, n_in)) return 0;
    return size_t(n_out * qg::canonical_row_bytes(fmt, n_in));
}

size_t qg_packed_bytes(qg_fmt fmt, int64_t n_out, int64_t n_in) {
    if (!qg::shape_valid(fmt, n_out, n_in)) return 0;
    return size_t(n_out * qg::row_stride(fmt, n_in));
}

int64_t qg_row_stride(qg_fmt fmt, int64_t n_in) {
    if (!qg::shape_valid(fmt, 1, n_in)) return 0;
    return qg::row_stride(fmt, n_in);
}

qg_status qg_quantize(qg_fmt fmt, const float* W, int64_t n_out, int64_t n_in, void* canonical) {
    if (!W || !canonical || !qg::shape_valid(fmt, n_out, n_in)) return QG_EINVAL;
    uint8_t* dst = static_cast<uint8_t*>(canonical);
    parallel_rows(n_out, n_in, [&](int64_t r0, int64_t r1) {
        for (int64_t r = r0; r < r1; ++r) quant_row(fmt, W + r * n_in, n_in, dst, n_out, r);
    });
    return QG_OK;
}

qg_status qg_to_device_layout(qg_fmt fmt, const void* canonical, int64_t n_out, int64_t n_in, void* packed) {
    if (!canonical || !packed || !qg::shape_valid(fmt, n_out, n_in)) return QG_EINVAL;
    const uint8_t* src = static_cast<const uint8_t*>(canonical);
    uint8_t* dst = static_cast<uint8_t*>(packed);
    const int64_t stride = qg::row_stride(fmt, n_in);
    parallel_rows(n_out, n_in, [&](int64_t r0, int64_t r1) {
        for (int64_t r = r0; r < r1; ++r)
            device_row(fmt, canon_row(fmt, src, n_out, n_in, r), n_in, dst + r * stride, stride);
    });
    return QG_OK;
}

qg_status qg_pack(qg_fmt fmt, const float* W, int64_t n_out, int64_t n_in, void* packed) {
    if (!W || !packed || !qg::shape_valid(fmt, n_out, n_in)) return QG_EINVAL;
    uint8_t* dst = static_cast<uint8_t*>(packed);
    const int64_t stride = qg::row_stride(fmt, n_in);
    const int64_t crow = qg::canonical_row_bytes(fmt, n_in);
    parallel_rows(n_out, n_in, [&](int64_t r0, int64_t r1) {
        // A one-row canonical scratch per thread (affine: its three planes for one row).
        std::vector<uint8_t> tmp(static_cast<size_t>(crow));
        for (int64_t r = r0; r < r1; ++r) {
            quant_row(fmt, W + r * n_in, n_in, tmp.data(), 1, 0);
            device_row(fmt, canon_row(fmt, tmp.data(), 1, n_in, 0), n_in, dst + r * stride, stride);
        }
    });
    return QG_OK;
}

}  // extern "C"
