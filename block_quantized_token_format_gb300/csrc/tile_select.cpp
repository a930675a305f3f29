// Per-shape kernel geometry for the dequant-GEMV.
//
// Prior art: the Track 2 Audit & Optimization Report (M5 Metal kernels)
// selects a tile per (format, n_in, n_out, ntok) because one tile does not
// fit all (section 1 item 1; table 2.1 shows tile changes worth up to 2.36x at
// ntok = 3).  Its tuples were measured on Apple GPUs and do not transfer; the
// rules below are for GB300 and are refined by the measured table in
// kTable (filled from sweeps on GB300).
#include "tile_select.h"

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "qg_layout.h"

namespace qg {

bool rpw_ok(int v) { return v >= 1 && v <= 8 && v != 7; }
bool depth_ok(int v) { return v >= 2 && v <= 16; }

namespace {

struct Entry {
    int fmt;
    int64_t n_out_min, n_out_max;   // inclusive range of n_out
    int64_t n_in;                   // 0 = any
    int ntok;                       // 0 = any
    Tile tile;                      // {rpw, depth, warps, ctas}
};

// Measured on GB300 (tile sweeps over rows per warp, ring depth, warps per CTA
// and CTAs per SM, back-to-back launches with early start; the sweep summary is
// in profiles/).  First match wins.  The fifth value, where given, is `pre`: the ring
// stages requested before the wait for the previous kernel (default one): the
// Q8_0 / Q4_0 / Q5_0 / BF16 projections gain 1.5-12% from one stage (same-box A/B
// against the whole ring, after retuning the geometry for it); the 2560 x 2560 matrix,
// BF16 at ntok 1-2 and the heads at ntok 2-4 keep more (the whole ring was 1-5% ahead
// there).
const Entry kTable[] = {
    // Q8_0 (integer chunk dot), n_in 2560: LM heads
    {QG_Q8_0, 65536, INT64_MAX, 2560, 1, {8, 2, 12, 1}},
    {QG_Q8_0, 65536, INT64_MAX, 2560, 2, {6, 2, 16, 1}},
    {QG_Q8_0, 65536, INT64_MAX, 2560, 3, {4, 3, 16, 1, 3}},
    {QG_Q8_0, 65536, INT64_MAX, 2560, 4, {5, 2, 16, 1}},
    // Q8_0, n_in 2560: 11264..65535 rows (the 12288 projection)
    {QG_Q8_0, 11264, 65535, 2560, 4, {4, 2, 12, 1}},
    {QG_Q8_0, 11264, 65535, 2560, 1, {8, 3, 12, 1, 1}},
    {QG_Q8_0, 11264, 65535, 2560, 0, {8, 2, 12, 1}},
    // Q8_0, n_in 2560: 9000..11263 rows (the 10240 projection)
    {QG_Q8_0, 9000, 11263, 2560, 1, {8, 3, 12, 1, 1}},
    {QG_Q8_0, 9000, 11263, 2560, 3, {6, 2, 16, 1}},
    {QG_Q8_0, 9000, 11263, 2560, 0, {6, 2, 12, 1}},
    // Q8_0, n_in 2560: 4096..8999 rows (the 6144 projection)
    {QG_Q8_0, 4096, 8999, 2560, 1, {4, 2, 12, 1, 1}},
    {QG_Q8_0, 4096, 8999, 2560, 3, {4, 2, 16, 1}},
    {QG_Q8_0, 4096, 8999, 2560, 0, {4, 2, 12, 1}},
    // Q8_0, n_in 2560: up to 4095 rows (2560 x 2560)
    {QG_Q8_0, 1, 4095, 2560, 1, {4, 4, 12, 1, 4}},
    {QG_Q8_0, 1, 4095, 2560, 2, {2, 4, 12, 1, 4}},
    {QG_Q8_0, 1, 4095, 2560, 3, {2, 4, 16, 1, 4}},
    {QG_Q8_0, 1, 4095, 2560, 4, {2, 3, 16, 1, 3}},
    // Q8_0, n_in 6144, few rows (6144 -> 2560; split 3: 15 warps = 5 teams)
    {QG_Q8_0, 1, 8191, 6144, 1, {4, 3, 16, 1}},
    {QG_Q8_0, 1, 8191, 6144, 0, {4, 2, 16, 1}},
    // Q4_0 (integer chunk dot) and BF16, 8192 x 2560
    {QG_Q4_0, 4096, 65535, 2560, 1, {4, 2, 16, 1}},
    {QG_Q4_0, 4096, 65535, 2560, 2, {8, 2, 12, 1}},
    {QG_Q4_0, 4096, 65535, 2560, 3, {8, 2, 8, 1}},
    {QG_Q4_0, 4096, 65535, 2560, 4, {5, 2, 16, 1}},
    {QG_BF16, 4096, 65535, 2560, 1, {4, 5, 8, 2, 5}},
    {QG_BF16, 4096, 65535, 2560, 2, {4, 5, 8, 2, 3}},
    {QG_BF16, 4096, 65535, 2560, 3, {4, 3, 16, 1}},
    {QG_BF16, 4096, 65535, 2560, 4, {4, 2, 16, 1}},
    // Q5_0, 8192 x 2560 (integer chunk dot; measured)
    {QG_Q5_0, 4096, 65535, 2560, 1, {8, 2, 12, 1}},
    {QG_Q5_0, 4096, 65535, 2560, 2, {8, 2, 12, 1}},
    {QG_Q5_0, 4096, 65535, 2560, 3, {4, 3, 16, 1}},
    {QG_Q5_0, 4096, 65535, 2560, 4, {4, 3, 16, 1}},
    // affine 4-bit LM head (integer chunk dot)
    {QG_AFFINE4_G64, 65536, INT64_MAX, 0, 1, {8, 2, 12, 1}},
    {QG_AFFINE4_G64, 65536, INT64_MAX, 0, 2, {6, 2, 16, 1, 2}},
    {QG_AFFINE4_G64, 65536, INT64_MAX, 0, 3, {8, 2, 12, 1}},
    {QG_AFFINE4_G64, 65536, INT64_MAX, 0, 4, {5, 2, 16, 1, 2}},
};

}  // namespace

Tile select_tile(int fmt, int64_t n_out, int64_t n_in, int ntok) {
    for (const Entry& e : kTable) {
        if (e.fmt != fmt) continue;
        if (n_out < e.n_out_min || n_out > e.n_out_max) continue;
        if (e.n_in && e.n_in != n_in) continue;
        if (e.ntok && e.ntok != ntok) continue;
        return e.tile;
    }

    // Heuristic for unmeasured shapes: many rows stream 4 per warp (8 at ntok 1) in
    // one 12- or 16-warp CTA per SM with a shallow ring; few rows use 2 rows per warp
    // so that the row groups still spread over every SM.
    Tile t;
    if (n_out >= 65536 && ntok == 1) {
        t = {8, 2, 16, 1};
    } else if (n_out >= 65536) {
        t = {4, 2, 16, 1};
    } else if (n_out >= 8192) {
        t = {4, 2, 12, 1};
    } else if (n_out >= 4096) {
        t = {4, 2, 16, 1};
    } else {
        t = {2, 3, 16, 1};
    }
    (void)n_in;
    return t;
}

// Measured on GB300 for the routed-expert layer (gate/up 1280x2560, down 2560x640,
// Q8_0, 10-21 active experts, integer chunk dot): 4 rows per warp, 12 warps and a
// 3-stage ring; 2 rows x 16 warps is 14% slower, 8 warps 10-20% slower, a 2-stage
// ring 1-1.5% slower.  CTA shares weighted 4 + tokens per group (a 4-token group gets
// 1.6x the CTAs of a 1-token group) cut the layer at ntok 3-4 by 7-10% against equal
// shares (2 + tokens: 3% slower at ntok 4 than 4 + tokens, 8 + tokens 1.5% slower).
Tile select_expert_tile(int fmt, int64_t n_out, int64_t n_in) {
    (void)fmt;
    (void)n_out;
    (void)n_in;
    Tile t;
    t.rpw = 4;
    t.depth = 3;
    t.warps = 12;
    t.ctas = 1;
    t.gw = 4;
    return t;
}

int select_split(int fmt, int64_t n_out, int64_t n_in) {
    // Matrices with 8192 rows or more have row groups for every warp of the GPU
    // (at 4 rows per warp) and short rows gain nothing from a team (measured on
    // GB300: splits of 2, 3 or 5 cost 5-15% at ntok 1 and 13-25% at ntok 4 on
    // 10240-12288 x 2560, and gain at most 1-3% on 2560 x 2560).  Few long rows
    // (2560 x 6144: 12 steps a row, 640 groups for 2280 warps) leave most warps
    // idle while each active one walks its steps alone; a team of about one warp
    // per 4 steps gains ~20% there (split 3 on 2560 x 6144).
    const int64_t spr = steps_per_row(fmt, n_in);
    if (n_out >= 8192 || spr <= 6) return 1;
    int64_t p = (spr + 3) / 4;
    if (p > 4) p = 4;          // measured up to 4; larger splits only through the override
    return int(p);
}

Tile apply_override(Tile t, const TileOverride& o) {
    if (o.rpw > 0) t.rpw = o.rpw;
    if (o.depth > 0) t.depth = o.depth;
    if (o.warps > 0) t.warps = o.warps;
    if (o.ctas > 0) t.ctas = o.ctas;
    if (o.pre > 0) t.pre = o.pre;
    if (o.split > 0) t.split = o.split;
    if (o.gw >= 0) t.gw = o.gw;
    return t;
}

bool parse_tile_spec(const char* spec, TileOverride* out) {
    TileOverride o;
    if (spec == nullptr || *spec == '\0') { *out = o; return true; }
    std::string s(spec);
    size_t pos = 0;
    while (pos < s.size()) {
        size_t end = s.find(',', pos);
        if (end == std::string::npos) end = s.size();
        std::string item = s.substr(pos, end - pos);
        pos = end + 1;
        if (item.empty()) continue;
        size_t eq = item.find('=');
        if (eq == std::string::npos) return false;
        std::string key = item.substr(0, eq), val = item.substr(eq + 1);
        if (val.empty() || val.size() > 3) return false;
        for (char ch : val) if (ch < '0' || ch > '9') return false;
        int v = std::atoi(val.c_str());
        if (key == "rpw") { if (!rpw_ok(v)) return false; o.rpw = v; }
        else if (key == "depth") { if (!depth_ok(v)) return false; o.depth = v; }
        else if (key == "warps") { if (v < 1 || v > 16) return false; o.warps = v; }
        else if (key == "ctas") { if (v < 1 || v > 8) return false; o.ctas = v; }
        else if (key == "pre") { if (!depth_ok(v) && v != 1) return false; o.pre = v; }
        else if (key == "split") { if (v < 1 || v > kMaxSplit) return false; o.split = v; }
        else if (key == "gw") { if (v > 64) return false; o.gw = v; }
        else return false;
    }
    *out = o;
    return true;
}

std::string tile_to_string(const Tile& t) {
    char b[96];
    std::snprintf(b, sizeof b, "rpw=%d,depth=%d,warps=%d,ctas=%d,pre=%d,split=%d", t.rpw, t.depth, t.warps,
                  t.ctas, t.pre, t.split);
    return b;
}

}  // namespace qg
