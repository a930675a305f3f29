// Per-shape kernel geometry selection (host).
#pragma once

#include <cstdint>
#include <string>

namespace qg {

// One launch geometry.  rpw: rows a warp streams together; depth: stages of the
// warp's shared-memory ring (one 512-byte code step of each of its rows per
// stage); warps: warps per CTA; ctas: CTAs per SM (capped by the occupancy the
// kernel actually reaches); pre: ring stages each warp requests before the wait for
// the previous kernel, the rest once x is staged (0 = one; capped at depth);
// split: warps per team, each streaming one segment of a row group's steps (0 =
// the default for the shape, select_split).
struct Tile {
    int rpw = 2;
    int depth = 2;
    int warps = 16;
    int ctas = 1;
    int pre = 0;
    int split = 0;
    int gw = 0;     // expert kernels: CTA shares per group weighted base + tokens (0 = equal)
};

// Fields left at -1 are not overridden.
struct TileOverride {
    int rpw = -1, depth = -1, warps = -1, ctas = -1, pre = -1, split = -1, gw = -1;
    bool any() const {
        return rpw > 0 || depth > 0 || warps > 0 || ctas > 0 || pre > 0 || split > 0 || gw >= 0;
    }
};

// Default split for a shape.  It depends on (fmt, n_out, n_in) only — never on
// ntok or the tile — because it fixes the order in which a row's partial sums are
// added: every ntok and every tile of one matrix then give bitwise the same rows.
int select_split(int fmt, int64_t n_out, int64_t n_in);

constexpr int kMaxSplit = 8;

// The geometry for a call, before the override and the occupancy cap.
Tile select_tile(int fmt, int64_t n_out, int64_t n_in, int ntok);

// The geometry of the expert-grouped mat-vec (rpw 1, 2 or 4; no split) for one
// expert's shape, before the override and the occupancy cap.
Tile select_expert_tile(int fmt, int64_t n_out, int64_t n_in);

// Apply an override on top of a selected tile.
Tile apply_override(Tile t, const TileOverride& o);

// Parse "rpw=4,depth=4,warps=8,ctas=2,pre=1,split=2,gw=4" (any subset, any order).  Empty -> no
// override.
bool parse_tile_spec(const char* spec, TileOverride* out);

// Allowed values (the instantiated kernels).
bool rpw_ok(int v);
bool depth_ok(int v);

std::string tile_to_string(const Tile& t);

}  // namespace qg
