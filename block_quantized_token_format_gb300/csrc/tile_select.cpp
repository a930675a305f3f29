// Per-shape kernel geometry for the dequant-GEMV.
//
// Prior art: the Track 2 Audit & Optimization Report (M5 Metal kernels)
// selects a tile per (format, n_in, n_out, ntok) because one tile does not
// fit all (section 1 item 1; table 2.1 shows tile changes worth up to 2.36x at
// ntok = 3).  Its tuples were measured on Apple GPUs and do not transfer; the
// rules below are for GB300 and are refined by the measured table in
// kTable (filled from sweeps on GB300).
#include "tile_select.h"

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "qg_layout.h"

namespace qg {

bool rpw_ok(int v) { return v == 1 || v == 2 || v == 4; }
bool depth_ok(int v) { return v >= 2 && v <= 16; }

namespace {

struct Entry {
    int fmt;
    int64_t n_out_min, n_out_max;   // inclusive range of n_out
    int64_t n_in;                   // 0 = any
    int ntok;                       // 0 = any
    Tile tile;
};

// Measured on GB300 (see the sweep summary in profiles/); first match wins.
const Entry kTable[] = {
    {-1, 0, 0, 0, 0, {}},   // sentinel
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
    Tile t;
    // Many rows: 4 rows per warp amortise x reads; few rows: spread them thinner.
    t.rpw = n_out >= 8192 ? 4 : 2;
    t.depth = 2;
    t.warps = 16;
    t.ctas = 1;
    (void)fmt; (void)n_in; (void)ntok;
    return t;
}

Tile apply_override(Tile t, const TileOverride& o) {
    if (o.rpw > 0) t.rpw = o.rpw;
    if (o.depth > 0) t.depth = o.depth;
    if (o.warps > 0) t.warps = o.warps;
    if (o.ctas > 0) t.ctas = o.ctas;
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
        else return false;
    }
    *out = o;
    return true;
}

std::string tile_to_string(const Tile& t) {
    char b[96];
    std::snprintf(b, sizeof b, "rpw=%d,depth=%d,warps=%d,ctas=%d", t.rpw, t.depth, t.warps, t.ctas);
    return b;
}

}  // namespace qg
