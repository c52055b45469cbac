// Host-side cost model behind the automatic kernel choice.
//
// The traffic and working-set counts are the closed forms of "Reading a
// matrix multiply through its tiles" ("What fits in local storage?", "Count
// the repeated reads", "Edge tiles still matter"): with no reuse of input
// tiles across output tiles, A is read once per output-column tile
// (M * K * ceil(N / tn) elements), B once per output-row tile
// (K * N * ceil(M / tm)), and C is written once (M * N); one step of the
// loop nest holds a tm x tk A tile, a tk x tn B tile and the tm x tn
// accumulator.  The page itself warns that a count is not a latency, so the
// time estimate combines the count with two measured rates (see
// predict_seconds) and with how evenly the tiles fill the GPU's resident
// CTAs, which the count does not see.
#include <algorithm>
#include <cstdint>

#include "launch.h"

namespace tmmo {

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

void traffic_model(int64_t M, int64_t N, int64_t K, int64_t tm, int64_t tn, int64_t tk,
                   int64_t in_bytes, int64_t acc_bytes, int64_t c_bytes, int64_t out[9])
{
    const int64_t tiles = ceil_div(M, tm) * ceil_div(N, tn);
    out[0] = M * K * ceil_div(N, tn);                            // A elements read
    out[1] = K * N * ceil_div(M, tm);                            // B elements read
    out[2] = M * N;                                              // C elements written
    out[3] = (out[0] + out[1]) * in_bytes + out[2] * c_bytes;    // bytes
    out[4] = 2 * M * N * K;                                      // multiply + add = 2
    out[5] = tiles;
    out[6] = tiles * ceil_div(K, tk);                            // K steps over all tiles
    // Largest step: the first tile is the fullest one (edge tiles are only
    // ever smaller), with its actual extents.
    const int64_t rm = std::min(tm, M), rn = std::min(tn, N), rk = std::min(tk, K);
    out[7] = (M > 0 && N > 0 && K > 0) ? rm * rk * in_bytes + rk * rn * in_bytes + rm * rn * acc_bytes
                                       : 0;
    out[8] = tm * tk * in_bytes + tk * tn * in_bytes + tm * tn * acc_bytes;
}

// Predicted seconds of one product on a tensor-core variant:
//   compute: the tiles run in waves of `units` resident CTAs (pairs for the
//     256 x 256 and 256 x 128 kernels); every wave costs one full tile of MMA work at the
//     variant's measured tile throughput;
//   feed: the traffic model's bytes (tile step tk = 64) at the measured
//     on-chip (L2 -> SM) rate;
// the larger of the two, plus a fixed launch cost.  The rates are the
// GB300 measurements behind this library's kernels (8192^3 and 4096^3
// BF16 runs of each variant); they rank the variants, they do not claim an
// absolute time.
double predict_seconds(int64_t M, int64_t N, int64_t K, int variant, int num_sms, int in_bytes,
                       int out_bytes)
{
    int tile_m, tile_n;
    tc_tile_shape(variant, &tile_m, &tile_n);
    const int units = tc_is_pair(variant) ? std::max(1, num_sms / 2) : std::max(1, num_sms);
    // Sustained dense rate per unit (CTA or CTA pair), in FLOP/s, as measured
    // for each tile shape on GB300.
    const double per_sm = 11.0e12;  // ~1680 TFLOP/s over 152 SMs for the pair kernel
    double eff = 1.0;
    if (variant == TC_256x128)
        eff = 0.68;
    else if (variant == TC_128x256)
        eff = 0.84;
    else if (variant == TC_128x128)
        eff = 0.67;
    const double unit_rate = per_sm * eff * (tc_is_pair(variant) ? 2.0 : 1.0);
    const int64_t tiles = ceil_div(M, tile_m) * ceil_div(N, tile_n);
    const int64_t waves = ceil_div(tiles, units);
    const double tile_flops = 2.0 * tile_m * tile_n * static_cast<double>(K);
    const double t_compute = waves * tile_flops / unit_rate;
    int64_t t[9];
    traffic_model(M, N, K, tile_m, tile_n, 64, in_bytes, 4, out_bytes, t);
    const double l2_rate = 14.0e12;  // bytes/s delivered from L2 to the SMs, measured
    const double t_feed = static_cast<double>(t[3]) / l2_rate;
    // Fixed cost of a launch: a CTA-pair kernel also sets up its clusters and
    // synchronizes both CTAs around TMEM, measured about 2 us more than the
    // single-CTA kernel on one-tile problems (128^3 .. 1024^3 BF16).
    const double t_launch = tc_is_pair(variant) ? 6.0e-6 : 4.0e-6;
    return std::max(t_compute, t_feed) + t_launch;
}

}  // namespace tmmo
