// kq_mmq_exact.cuh -- launch interface of the exact integer MMQ kernel (internal).
#pragma once
#include "kq_internal.cuh"

namespace kq {

struct MmqExactArgs {
    const uint8_t *w;       // native weights (grouped: all experts, expert e at rows [e*N, (e+1)*N))
    const uint8_t *xq;      // activation rows (Q8_K or Q8_1 blocks)
    int64_t M, N, K;        // dense: M token rows; grouped: M unused
    float *y;               // fp32 output rows (dense: [M][ldy]; grouped: [M*top_k][N])
    int64_t ldy;
    int32_t *partials;      // debug mode output
    // routed-expert tiles (grouped mode)
    const int *tile_count;     // [1] number of valid tiles
    const int *tiles;          // [max_tiles][2] = (expert, first row index within the expert's list)
    const int *expert_count;   // [E]
    const int *expert_offset;  // [E]
    const int *lists;          // (token, slot) pair indices grouped by expert
    int rows_per_token, top_k;
};

size_t mmq_exact_smem();
kq_status launch_mmq_exact(int dt, int mode, bool grouped, const MmqExactArgs &a, unsigned grid_y, cudaStream_t st);

}  // namespace kq
