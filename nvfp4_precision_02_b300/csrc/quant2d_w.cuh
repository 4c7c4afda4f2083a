// quant2d_w.cuh -- 2D (16x16) quantisation of W only (no W^T) for sm_103a:
// the quantise half of the expert-weight path (per-expert amax first, then
// this), 2D block scaling of weights ("Nemotron 3 Super -- technical report
// summary", gkm0120.cn, "Infra design" table).  The strip arithmetic is
// k_quant2d's (quant2d_strip_load / quant2d_strip_encode).
#pragma once

#include "quant.cuh"

namespace nvfp4 {

// W only (the expert weights): a CTA of four warps covers 64 rows x 64 NS
// columns; each warp loads its NS strips of 16 x 64 before encoding any, so
// it has NS times the loads in flight of k_quant2d with 1/NS of the CTAs (and
// of the per-CTA set-up: the tensor scale's division, the block's addresses).
template <int NS>
__global__ void __launch_bounds__(128) k_quant2d_w(const uint16_t* __restrict__ w, int64_t rows, int64_t cols,
                                                   int64_t ld, const float* __restrict__ amax,
                                                   uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                   uint8_t* __restrict__ tile_sf, float* __restrict__ amax_copy) {
    const int64_t b = blockIdx.z;
    if (amax_copy != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) amax_copy[b] = amax[b];
    const int64_t rs = (int64_t)blockIdx.y * 64 + 16 * (threadIdx.x >> 5), c0 = (int64_t)blockIdx.x * 64 * NS;
    const uint16_t* wb = w + b * rows * ld;
    uint4 v[NS][4];
#pragma unroll
    for (int j = 0; j < NS; ++j) quant2d_strip_load(wb, rows, cols, ld, rs, c0 + 64 * j, v[j]);
    const float s_enc = tensor_encode_scale(amax[b]);
#pragma unroll
    for (int j = 0; j < NS; ++j) {
        if (c0 + 64 * j >= cols) break;
        uint32_t cw[4], word;
        quant2d_strip_encode(v[j], rows, cols, b, rs, c0 + 64 * j, s_enc, codes, sf, tile_sf, cw, word);
    }
}

}  // namespace nvfp4
