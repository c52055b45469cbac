// Launch parameters shared by the host dispatcher and the tensor-core kernel.
#pragma once

#include <cstdint>

namespace tmmo {

// Value written to the device status word when a bounded wait runs out.
constexpr int TC_STATUS_TIMEOUT = 1;

struct TcParams {
    int M, N, K;
    int tiles_m, tiles_n, num_tiles;  // output tiles of (128 * CG) x BN
    int k_blocks;                      // ceil(K / 64)
    int dp_tiles;                      // tiles computed whole; the rest are split along K
    int k_splits;                      // K ranges per split tile
    int kb_per_split;                  // K steps per range
    int num_work;                      // dp_tiles + (num_tiles - dp_tiles) * k_splits units
    int group_m;                       // raster group height, in tile rows
    uint32_t idesc;                    // tcgen05 instruction descriptor
    int* status;                       // device status word (never null)
    long long wait_budget;             // clock cycles a single wait may take
    int fault_skip_kblock;             // test hook: K step whose loads are skipped; -1 = none
    const void* C;                     // the output, read as C_in when beta != 0
    float alpha, beta;                 // C = alpha * acc + beta * C_in
};

}  // namespace tmmo
