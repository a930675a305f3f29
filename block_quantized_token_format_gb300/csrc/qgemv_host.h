// Host helpers shared by the library's C ABI translation units (internal; not
// part of the public header).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>            // CUtensorMap (type only)

#include "../../include/qgemv.h"
#include "tile_select.h"

namespace qg {

// One launch's geometry and resources.
struct Plan {
    const void* fn = nullptr;
    Tile tile;
    int grid = 0;
    int threads = 0;
    size_t smem = 0;
    unsigned int* status = nullptr;
    int seg_len = 0;
};

constexpr size_t kStaticSmemReserve = 1024;   // static shared memory a kernel may add

// The current device, its SM count, its opt-in shared memory per block and the
// device address of the status word (cached per device).
qg_status device_info(int* dev, int* sms, int* smem_optin, unsigned int** status);
// Blocks of `fn` resident per SM (raises its dynamic shared memory limit on first use).
int blocks_per_sm(const void* fn, int dev, int optin, int threads, size_t smem);
// Threads per block the kernel allows (its launch bound).
int max_threads(const void* fn);
bool aligned(const void* p, uintptr_t a);
// The packed matrix [n_out][row stride / 8] as a 2-D tensor map, box = one full step
// x rpw rows, zero fill outside (cached per thread).
qg_status encode_weight_map(CUtensorMap* map, int fmt, const void* W, int64_t n_out, int64_t n_in, int rpw);
// Launch options, the tile override and its generation, the wait-limit test hook.
unsigned launch_flags();
void read_env_override();
TileOverride current_override();
uint64_t override_generation();
uint32_t wait_limit();
uint32_t test_extra_tx();

}  // namespace qg
