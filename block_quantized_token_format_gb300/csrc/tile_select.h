// Per-shape kernel geometry selection (host).
#pragma once

#include <cstdint>
#include <string>

namespace qg {

// One launch geometry.  rpw: rows a warp streams together; depth: chunk sets a
// lane keeps in flight; warps: warps per CTA; ctas: CTAs per SM (capped by the
// occupancy the kernel actually reaches).
struct Tile {
    int rpw = 2;
    int depth = 4;
    int warps = 8;
    int ctas = 2;
    int pf = 0;      // L2 bulk-prefetch distance, in row groups of the same warp (0 = off)
};

// Fields left at -1 are not overridden.
struct TileOverride {
    int rpw = -1, depth = -1, warps = -1, ctas = -1, pf = -1;
    bool any() const { return rpw > 0 || depth > 0 || warps > 0 || ctas > 0 || pf >= 0; }
};

// The geometry for a call, before the override and the occupancy cap.
Tile select_tile(int fmt, int64_t n_out, int64_t n_in, int ntok);

// Apply an override on top of a selected tile.
Tile apply_override(Tile t, const TileOverride& o);

// Parse "rpw=4,depth=2,warps=8,ctas=2" (any subset, any order).  Empty -> no override.
bool parse_tile_spec(const char* spec, TileOverride* out);

// Allowed values (the instantiated kernels).
bool rpw_ok(int v);
bool depth_ok(int v);

// Whether (fmt, ntok, rpw, depth) fits in registers without spilling.
bool tile_fits_registers(int fmt, int ntok, int rpw, int depth);

std::string tile_to_string(const Tile& t);

}  // namespace qg
