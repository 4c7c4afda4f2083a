// quant.cuh -- HBM-bound NVFP4 quantisers for sm_103a.
//
//   k_amax           tensor (or per batch entry) max |x| of bf16 data
//   k_amax_grouped   per-group max |x| of expert-sorted rows
//   k_quant1d        1x16 blocks, RNE or SR, plain or grouped (per-expert scale)
//   k_quant2d        16x16 tiles, emits W and W^T codes with GEMM-ready scales
//   k_rht            16-point random Hadamard transform along tokens, amax or
//                    transform + quantise into the transposed wgrad operand
//
// Recipe: "Nemotron 3 Super -- technical report summary" (gkm0120.cn),
// "Infra design" table (1D scaling for activations/gradients, 2D for weights,
// RHT + SR); "Nemotron 3 Ultra" report (papercache.org translation), section
// 2.2 (RHT on the wgrad inputs, SR on gradients).
#pragma once

#include <cuda.h>
#include "common.cuh"

namespace nvfp4 {

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ uint32_t absmax_bits(uint4 v, uint32_t acc) {
    // non-negative bf16 values order like their 15-bit magnitudes
    acc = __vmaxu2(acc, v.x & 0x7FFF7FFFu);
    acc = __vmaxu2(acc, v.y & 0x7FFF7FFFu);
    acc = __vmaxu2(acc, v.z & 0x7FFF7FFFu);
    acc = __vmaxu2(acc, v.w & 0x7FFF7FFFu);
    return acc;
}

__device__ __forceinline__ float bits_to_amax(uint32_t acc) {
    const uint32_t m = max(acc & 0xFFFFu, acc >> 16);
    return __uint_as_float(m << 16);
}

// Block-wide max of non-negative floats (as bits) followed by one atomicMax.
__device__ __forceinline__ void block_max_atomic(uint32_t v, float* dst) {
    __shared__ uint32_t s_red[32];
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        const int nw = (blockDim.x + 31) >> 5;
        uint32_t w = lane < nw ? s_red[lane] : 0u;
        w = __reduce_max_sync(0xFFFFFFFFu, w);
        if (lane == 0 && w != 0u) atomicMax(reinterpret_cast<unsigned int*>(dst), w);
    }
}

// ------------------------------------------------------------------ amax
// x: bf16 [batch][rows, cols] (row stride ld, entry stride estride elements);
// amax[b] must be zero on entry.  Units of 8 elements; rows*cols/8 < 2^32.
__global__ void __launch_bounds__(256) k_amax(const uint16_t* __restrict__ x, int64_t rows,
                                              int64_t cols, int64_t ld, int64_t estride,
                                              float* __restrict__ amax) {
    const uint16_t* base = x + (int64_t)blockIdx.y * estride;
    const uint32_t upr = (uint32_t)(cols >> 3);
    const uint64_t units = (uint64_t)rows * upr;
    const bool contiguous = (ld == cols);
    uint32_t acc = 0;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    uint64_t u = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; u + 3 * stride < units; u += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint64_t ui = u + i * stride;
            const uint16_t* p = contiguous ? base + ui * 8
                                           : base + (int64_t)(ui / upr) * ld + (ui % upr) * 8;
            v[i] = __ldg(reinterpret_cast<const uint4*>(p));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) acc = absmax_bits(v[i], acc);
    }
    for (; u < units; u += stride) {
        const uint16_t* p = contiguous ? base + u * 8 : base + (int64_t)(u / upr) * ld + (u % upr) * 8;
        acc = absmax_bits(__ldg(reinterpret_cast<const uint4*>(p)), acc);
    }
    const float m = bits_to_amax(acc);
    block_max_atomic(__float_as_uint(m), amax + blockIdx.y);
}

// ------------------------------------------------------------------ groups
// Shared tables of a grouped launch: clamped row offsets o[0..G] and padded
// scale-row offsets P[0..G] (P[g] = sum_{i<g} ceil(cnt_i/128)*128).  Offsets
// that are out of range or decreasing are clamped (and flagged).
struct GroupTables {
    int32_t* off;              // [G+1]
    int32_t* pad;              // [G+1]
    int32_t* pair = nullptr;   // [G+1], optional: sum_{i<g} ceil(cnt_i/256)*256 (tiles of CTA pairs)
};

// pad_shift: pad[] pads each count to a multiple of 2^pad_shift (7: the
// 128-row scale blocks; 6: the 64-token expert segments of the grouped wgrad).
__device__ void build_group_tables(const int64_t* __restrict__ offsets, int32_t groups,
                                   int64_t rows, GroupTables t, int pad_shift = 7) {
    __shared__ int32_t s_wsum[32];
    // 1) clamped offsets: o[g] = min(max(offsets[g], 0), rows); monotone fix-up
    //    is a running max, computed below together with the scan.
    const int nthreads = blockDim.x;
    const int per = (groups + 1 + nthreads - 1) / nthreads;
    const int g0 = threadIdx.x * per;
    int32_t local_max = 0;
    bool bad = false;
    for (int i = 0; i < per; ++i) {
        const int g = g0 + i;
        if (g <= groups) {
            int64_t v = offsets[g];
            if (v < 0 || v > rows) bad = true;
            v = v < 0 ? 0 : (v > rows ? rows : v);
            if (g == 0 && v != 0) bad = true;
            t.off[g] = (int32_t)v;
        }
    }
    __syncthreads();
    // running max (monotone offsets): per-thread max, then exclusive max-scan
    for (int i = 0; i < per; ++i) {
        const int g = g0 + i;
        if (g <= groups) local_max = max(local_max, t.off[g]);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t incl = local_max;
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl = max(incl, o);
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    int32_t prefix = 0;
    for (int w = 0; w < warp; ++w) prefix = max(prefix, s_wsum[w]);
    int32_t excl = max(prefix, __shfl_up_sync(0xFFFFFFFFu, incl, 1));
    if (lane == 0) excl = prefix;
    __syncthreads();
    int32_t run = excl;
    for (int i = 0; i < per; ++i) {
        const int g = g0 + i;
        if (g <= groups) {
            const int32_t v = t.off[g];
            if (v < run) bad = true;
            run = max(run, v);
            t.off[g] = run;
        }
    }
    __syncthreads();
    // 2) padded rows: exclusive sums of ceil(cnt/2^pad_shift)*2^pad_shift and,
    //    when asked, of ceil(cnt/256)*256 (row tiles of CTA pairs)
    for (int which = 0; which < (t.pair != nullptr ? 2 : 1); ++which) {
        const int sh = which == 0 ? pad_shift : 8;
        int32_t* dst = which == 0 ? t.pad : t.pair;
        int32_t local_sum = 0;
        for (int i = 0; i < per; ++i) {
            const int g = g0 + i;
            if (g < groups) local_sum += ((t.off[g + 1] - t.off[g] + (1 << sh) - 1) >> sh) << sh;
        }
        int32_t inc = local_sum;
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t o = __shfl_up_sync(0xFFFFFFFFu, inc, d);
            if (lane >= d) inc += o;
        }
        __syncthreads();
        if (lane == 31) s_wsum[warp] = inc;
        __syncthreads();
        int32_t base = 0;
        for (int w = 0; w < warp; ++w) base += s_wsum[w];
        int32_t acc = base + inc - local_sum;
        for (int i = 0; i < per; ++i) {
            const int g = g0 + i;
            if (g <= groups) {
                dst[g] = acc;
                if (g < groups) acc += ((t.off[g + 1] - t.off[g] + (1 << sh) - 1) >> sh) << sh;
            }
        }
    }
    if (bad && blockIdx.x == 0) raise_status(DEV_BAD_OFFSETS);
    __syncthreads();
}

// Group of row r (o[g] <= r < o[g+1]); requires o[0] <= r < o[G].
__device__ __forceinline__ int find_group(const int32_t* off, int groups, int32_t r) {
    int lo = 0, hi = groups;      // invariant: off[lo] <= r < off[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= r) lo = mid; else hi = mid;
    }
    return lo;
}

// Rows [rows*w/W, rows*(w+1)/W) of warp w out of W.
__device__ __forceinline__ void warp_rows(int64_t rows, int64_t& r0, int64_t& r1) {
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    r0 = rows * w / nw;
    r1 = rows * (w + 1) / nw;
}

// Per-group amax of expert-sorted rows; amax[g] must be zero on entry.
__global__ void __launch_bounds__(256) k_amax_grouped(const uint16_t* __restrict__ x, int64_t rows,
                                                      int64_t cols, int64_t ld,
                                                      const int64_t* __restrict__ offsets,
                                                      int32_t groups, float* __restrict__ amax) {
    extern __shared__ int32_t s_tab[];
    GroupTables t{s_tab, s_tab + groups + 1};
    build_group_tables(offsets, groups, rows, t);
    int64_t r0, r1;
    warp_rows(rows, r0, r1);
    const int lane = threadIdx.x & 31;
    const int upr = (int)(cols >> 3);
    int g = -1;
    int32_t g_end = 0;
    uint32_t acc = 0;
    for (int64_t r = r0; r < r1; ++r) {
        if (r < t.off[0] || r >= t.off[groups]) continue;
        if (g < 0 || r >= g_end) {
            if (g >= 0) {
                // acc packs two 16-bit maxima: unpack before the warp reduction
                const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, max(acc & 0xFFFFu, acc >> 16));
                if (lane == 0 && m) atomicMax(reinterpret_cast<unsigned int*>(amax + g), m << 16);
            }
            g = find_group(t.off, groups, (int32_t)r);
            g_end = t.off[g + 1];
            acc = 0;
        }
        const uint16_t* row = x + r * ld;
        for (int u = lane; u < upr; u += 32)
            acc = absmax_bits(__ldg(reinterpret_cast<const uint4*>(row + u * 8)), acc);
    }
    if (g >= 0) {
        const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, max(acc & 0xFFFFu, acc >> 16));
        if (lane == 0 && m) atomicMax(reinterpret_cast<unsigned int*>(amax + g), m << 16);
    }
}

// ------------------------------------------------------------------ 1D quantise
// Encode the 8 elements of one half-block (lane pair = one 16-element block).
template <bool SR>
__device__ __forceinline__ uint32_t encode8(const uint4 v, float ratio, bool zero, const PhiloxKeys& key,
                                            uint64_t e0) {
    if (zero) return 0u;
    if (!SR) return e2m1x8_rne_bf16(v, ratio);
    float f[8];
    scale8_bf16(v, ratio, f);
    const uint4 w0 = sr_words(key, e0 >> 2);
    const uint4 w1 = sr_words(key, (e0 >> 2) + 1);
    const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    uint32_t out = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) out |= e2m1_sr(f[j], w[j]) << (4 * j);
    return out;
}

// Element multipliers S_enc / e4m3(c) of every scale code c (entry 0 unused)
// in a warp's 128-float slice of shared memory: lane l computes codes l,
// l + 32, l + 64, l + 96 with the same correctly rounded division as
// element_ratio, so a lookup gives the same bits.
__device__ __forceinline__ void fill_ratio_table(float* tab, float s_enc) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t c = (uint32_t)(lane + 32 * i);
        tab[c] = (c >= 1 && c <= 126) ? element_ratio(s_enc, c) : 0.0f;
    }
    __syncwarp();
}

// Work is cut into segments of 32 blocks (512 elements) of one row.  The
// segments are ordered by 128-row band of the scale layout (groups start on
// a band), and inside a band either row by row (row order: each warp then
// streams contiguous memory) or, when the scale buffer is larger than L2
// can keep half-written (BAND), by 32-block column and then by rows
// i, i+32, i+64, i+96 in turn: those four rows share each 16-byte slot of
// the scale atoms, so every 32-byte scale sector is complete within eight
// segments instead of being written back half-filled.  Band rows past the
// tensor's or the group's end are the padding rows of the scale layout:
// their scale words are written as zeros.
// Warp w of W takes the contiguous range [S*w/W, S*(w+1)/W) of the S
// segments, walks it with a (band, column, row-in-band) counter, and keeps
// the next two segments' loads in flight while it encodes one.  Lane l owns block l
// of a segment: its 16 elements (one 256-bit load), the block amax in
// registers, 8 code bytes; every fourth lane stores the 4 scale bytes of its
// block and the next three as one word (zeros past the row's last block
// fill the scale padding of the last atom column).  The element multiplier
// of a block is looked up in the warp's table of the 127 scale codes,
// refilled when the tensor scale changes (a new expert).
// x: bf16 [rows, cols] (row stride ld); codes [rows, cols/2]; sf swizzled.
// amax: 1 value (or one per group when GROUPED).  SR index e = r*cols + c.
struct Seg16 {
    uint4 a, b;
};

template <bool SR, bool GROUPED, bool BAND>
__global__ void __launch_bounds__(256) k_quant1d(const uint16_t* __restrict__ x, int64_t rows,
                                                 int64_t cols, int64_t ld,
                                                 const float* __restrict__ amax, uint64_t seed,
                                                 uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                 const int64_t* __restrict__ offsets, int32_t groups,
                                                 float* __restrict__ amax_copy) {
    extern __shared__ int32_t s_tab[];
    __shared__ float s_ratio[8][128];
    GroupTables t{s_tab, s_tab + (GROUPED ? groups + 1 : 0)};
    if (GROUPED) build_group_tables(offsets, groups, rows, t);
    if (amax_copy != nullptr && blockIdx.x == 0) {
        const int n = GROUPED ? groups : 1;
        for (int i = threadIdx.x; i < n; i += blockDim.x) amax_copy[i] = amax[i];
    }
    const int lane = threadIdx.x & 31;
    float* ratio_tab = s_ratio[threadIdx.x >> 5];
    const int64_t nb = cols >> 4;                       // blocks of a row
    const int64_t nseg = (nb + 31) >> 5;                // 32-block columns
    const int64_t bands = GROUPED ? (int64_t)(t.pad[groups] >> 7) : (rows + 127) >> 7;
    const int64_t S = bands * nseg * 128;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t s0 = S * w / nw, s1 = S * (w + 1) / nw;
    if (s0 >= s1) return;
    const PhiloxKeys key = philox_keys(seed);
    // one 256-bit load per lane when every block starts 32-byte aligned
    const bool vec32 = ((reinterpret_cast<uintptr_t>(x) & 31) == 0) && ((ld & 15) == 0);
    float s_enc = 1.0f;
    if (!GROUPED) {
        s_enc = tensor_encode_scale(amax[0]);
        fill_ratio_table(ratio_tab, s_enc);
    }
    // The walk: band k, 32-block column j, row rib of the band.
    int64_t k, j;
    int rib;
    if (BAND) {
        rib = 32 * (int)(s0 & 3) + (int)((s0 >> 2) & 31);
        const int64_t kj = s0 >> 7;
        k = kj / nseg;
        j = kj - k * nseg;
    } else {
        k = s0 / (nseg * 128);
        const int64_t rem = s0 - k * nseg * 128;
        rib = (int)(rem / nseg);
        j = rem - (int64_t)rib * nseg;
    }
    // the expert whose scale rows hold band k (grouped): pad[g] <= 128 k < pad[g+1]
    int gk = -1, g = 0;
    int32_t g_lo = 0, g_hi = 0, g_pad = 0;
    auto band_group = [&]() {
        if (GROUPED && k != gk) {
            int lo = 0, hi = groups;
            const int32_t key_row = (int32_t)(k * 128);
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (t.pad[mid] <= key_row) lo = mid; else hi = mid;
            }
            g = lo;
            g_lo = t.off[g];
            g_hi = t.off[g + 1];
            g_pad = t.pad[g];
            gk = (int)k;
        }
    };
    // A segment in flight: its data, data row (-1: a padding row of the scale
    // layout), scale row, 32-block column and expert (rows and scale rows are
    // below 2^31: host checks).
    struct InFlight {
        Seg16 v;
        int32_t r, srow, j, g;
    };
    auto fetch = [&]() {
        InFlight f;
        band_group();
        f.srow = (int32_t)(k * 128 + rib);
        f.r = GROUPED ? ((g_lo + (f.srow - g_pad)) < g_hi ? g_lo + (f.srow - g_pad) : -1)
                      : (f.srow < rows ? f.srow : -1);
        f.j = (int32_t)j;
        f.g = g;
        const int64_t fb = j * 32 + lane;
        f.v = Seg16{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        if (f.r >= 0 && fb < nb) {
            const uint16_t* src = x + (int64_t)f.r * ld + 16 * fb;
            if (vec32) {
                ldg32_stream(src, f.v.a, f.v.b);
            } else {
                f.v.a = __ldg(reinterpret_cast<const uint4*>(src));
                f.v.b = __ldg(reinterpret_cast<const uint4*>(src) + 1);
            }
        }
        if (BAND) {
            // rib: 0, 32, 64, 96, 1, 33, 65, 97, ..., 31, 63, 95, 127, then the next column
            if (rib < 96) rib += 32;
            else if (rib < 127) rib -= 95;
            else { rib = 0; if (++j == nseg) { j = 0; ++k; } }
        } else if (++j == nseg) {
            j = 0;
            if (++rib == 128) { rib = 0; ++k; }
        }
        return f;
    };
    // two segments in flight ahead of the one being encoded
    InFlight cur = fetch(), nxt;
    nxt.r = -1;
    if (s0 + 1 < s1) nxt = fetch();
    int cur_g = -1;
    for (int64_t sg = s0; sg < s1; ++sg) {
        InFlight nxt2;
        nxt2.r = -1;
        if (sg + 2 < s1) nxt2 = fetch();
        const int64_t b = (int64_t)cur.j * 32 + lane;
        uint32_t sc = 0;
        if (cur.r >= 0) {
            if (GROUPED && cur.g != cur_g) {
                cur_g = cur.g;
                s_enc = tensor_encode_scale(amax[cur_g]);
                fill_ratio_table(ratio_tab, s_enc);
            }
            const uint32_t m = bf16x16_absmax(cur.v.a, cur.v.b);
            sc = block_scale(__uint_as_float(m << 16), s_enc);
            const float ratio = ratio_tab[sc];
            uint32_t lo = 0, hi = 0;
            if (sc != 0) {
                if (SR) {
                    const uint64_t e0 = (uint64_t)(uint32_t)cur.r * (uint64_t)cols + (uint64_t)b * 16;
                    lo = encode8<true>(cur.v.a, ratio, false, key, e0);
                    hi = encode8<true>(cur.v.b, ratio, false, key, e0 + 8);
                } else {
                    lo = e2m1x8_rne_bf16(cur.v.a, ratio);
                    hi = e2m1x8_rne_bf16(cur.v.b, ratio);
                }
            }
            if (b < nb) *reinterpret_cast<uint2*>(codes + (int64_t)cur.r * (cols >> 1) + 8 * b) = make_uint2(lo, hi);
        }
        // four consecutive blocks' scales in one word (lanes past the row's end,
        // and every lane of a padding row, hold 0)
        const uint32_t scv = b < nb ? sc : 0u;
        const uint32_t word = scv | (__shfl_down_sync(0xFFFFFFFFu, scv, 1) << 8) |
                              (__shfl_down_sync(0xFFFFFFFFu, scv, 2) << 16) |
                              (__shfl_down_sync(0xFFFFFFFFu, scv, 3) << 24);
        if (b < nb && (lane & 3) == 0) *reinterpret_cast<uint32_t*>(sf + sf_offset(cur.srow, b, cols)) = word;
        cur = nxt;
        nxt = nxt2;
    }
}

// Zero the scale bytes of padding rows: for a plain operand rows [rows,
// pad128(rows)); for a grouped one, rows [P_g + cnt_g, P_g + pad128(cnt_g))
// of every group.  Four bytes (one row, one atom column) per store.
__global__ void __launch_bounds__(256) k_zero_pad_rows(uint8_t* __restrict__ sf, int64_t rows,
                                                       int64_t cols, const int64_t* __restrict__ offsets,
                                                       int32_t groups) {
    extern __shared__ int32_t s_tab[];
    const int64_t catoms = ((cols >> 4) + 3) >> 2;
    if (offsets == nullptr) {
        const int64_t pr = ((rows + 127) >> 7) << 7;
        const int64_t n = (pr - rows) * catoms;
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
             i += (int64_t)gridDim.x * blockDim.x) {
            const int64_t r = rows + i / catoms, a = i % catoms;
            *reinterpret_cast<uint32_t*>(sf + sf_offset(r, a * 4, cols)) = 0u;
        }
        return;
    }
    GroupTables t{s_tab, s_tab + groups + 1};
    build_group_tables(offsets, groups, rows, t);
    // one warp per group
    const int lane = threadIdx.x & 31;
    for (int g = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); g < groups;
         g += gridDim.x * (blockDim.x >> 5)) {
        const int64_t cnt = t.off[g + 1] - t.off[g];
        const int64_t pr = ((cnt + 127) >> 7) << 7;
        const int64_t n = (pr - cnt) * catoms;
        for (int64_t i = lane; i < n; i += 32) {
            const int64_t r = t.pad[g] + cnt + i / catoms, a = i % catoms;
            *reinterpret_cast<uint32_t*>(sf + sf_offset(r, a * 4, cols)) = 0u;
        }
    }
}

// ------------------------------------------------------------------ 2D quantise
// In-register transpose of an 8x8 block of nibbles: a[n] holds row n (column
// k in nibble k); afterwards a[k] holds column k (row n in nibble n).  Three
// stages swap 1x1, 2x2 and 4x4 sub-blocks across the diagonal.
__device__ __forceinline__ void transpose8x8_nibbles(uint32_t (&a)[8]) {
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const uint32_t t = ((a[i] >> 4) ^ a[i + 1]) & 0x0F0F0F0Fu;
        a[i + 1] ^= t;
        a[i] ^= t << 4;
    }
#pragma unroll
    for (int i = 0; i < 8; i += 4)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint32_t t = ((a[i + j] >> 8) ^ a[i + j + 2]) & 0x00FF00FFu;
            a[i + j + 2] ^= t;
            a[i + j] ^= t << 8;
        }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t t = ((a[j] >> 16) ^ a[j + 4]) & 0x0000FFFFu;
        a[j + 4] ^= t;
        a[j] ^= t << 16;
    }
}

// One warp's 16x64 strip (rows rs .. rs+15, columns c0 .. c0+63, four 16x16
// tiles) of batch entry b: loads, tile amax, scales, W codes and the W rows'
// scale words.  Returns the four code words and the strip's scale word (tile
// t in byte t) for the W^T stage.  Lane l handles row (l >> 3) + 4i,
// columns 8*(l & 7) .. +7.
__device__ __forceinline__ void quant2d_strip_load(const uint16_t* __restrict__ wb, int64_t rows, int64_t cols,
                                                   int64_t ld, int64_t rs, int64_t c0, uint4 (&v)[4]) {
    const int lane = threadIdx.x & 31, c8 = lane & 7;
    const bool ok = rs < rows && c0 + 8 * c8 < cols;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t rr = rs + (lane >> 3) + 4 * i;
        v[i] = ok ? __ldg(reinterpret_cast<const uint4*>(wb + rr * ld + c0 + 8 * c8)) : make_uint4(0, 0, 0, 0);
    }
}

__device__ __forceinline__ void quant2d_strip_encode(const uint4 (&v)[4], int64_t rows, int64_t cols, int64_t b,
                                                     int64_t rs, int64_t c0, float s_enc, uint8_t* __restrict__ codes,
                                                     uint8_t* __restrict__ sf, uint8_t* __restrict__ tile_sf,
                                                     uint32_t (&cw)[4], uint32_t& word) {
    const int lane = threadIdx.x & 31, c8 = lane & 7;
    const bool rows_ok = rs < rows;                     // rows % 16 == 0: a strip is all in or all out
    const bool col_ok = c0 + 8 * c8 < cols;             // cols % 16 == 0: 8-column groups are all in or out
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) m = absmax_bits(v[i], m);
    m = max(m & 0xFFFFu, m >> 16);
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
    const uint32_t sc = block_scale(__uint_as_float(m << 16), s_enc);
    const float ratio = sc ? element_ratio(s_enc, sc) : 0.0f;
    const PhiloxKeys no_key{};
#pragma unroll
    for (int i = 0; i < 4; ++i) cw[i] = encode8<false>(v[i], ratio, sc == 0, no_key, 0);
    // scales of the strip's four tiles (tile t is held by lane 2t)
    word = __shfl_sync(0xFFFFFFFFu, sc, 0) | (__shfl_sync(0xFFFFFFFFu, sc, 2) << 8) |
           (__shfl_sync(0xFFFFFFFFu, sc, 4) << 16) | (__shfl_sync(0xFFFFFFFFu, sc, 6) << 24);
    if (!rows_ok) return;
    uint8_t* cb = codes + b * (rows * cols / 2);
    if (col_ok) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t rr = rs + (lane >> 3) + 4 * i;
            *reinterpret_cast<uint32_t*>(cb + rr * (cols / 2) + (c0 + 8 * c8) / 2) = cw[i];
        }
    }
    if (lane < 16)
        *reinterpret_cast<uint32_t*>(sf + b * sf_bytes(rows, cols) + sf_offset(rs + lane, c0 / 16, cols)) = word;
    if (tile_sf != nullptr && lane < 8 && (lane & 1) == 0 && col_ok)
        tile_sf[b * (rows / 16) * (cols / 16) + (rs / 16) * (cols / 16) + c0 / 16 + (lane >> 1)] = (uint8_t)sc;
}

// One 64x64 block (rows r0.., columns c0..) of batch entry b, by 4 warps
// (128 threads): warp w quantises the strip of rows r0 + 16w (as above); for
// W^T the code words go through shared memory and 64 threads each transpose
// one 8x8 nibble block, so that every W^T row receives 32 contiguous bytes.
// Every thread of the block must call it.
struct Quant2dSmem {
    uint32_t cw[64][9];     // code words [row of the block][8-column group] (+1 pad)
    uint32_t sc[4][4];      // tile scales [warp][tile]
};

__device__ __forceinline__ void quant2d_block(const uint16_t* __restrict__ wb, int64_t rows, int64_t cols,
                                              int64_t ld, int64_t b, int64_t r0, int64_t c0, float s_enc,
                                              uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                              uint8_t* __restrict__ codes_t, uint8_t* __restrict__ sf_t,
                                              uint8_t* __restrict__ tile_sf, Quant2dSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t rs = r0 + 16 * warp;
    const bool rows_ok = rs < rows;
    const int c8 = lane & 7;
    uint4 v[4];
    quant2d_strip_load(wb, rows, cols, ld, rs, c0, v);
    uint32_t cw[4], word;
    quant2d_strip_encode(v, rows, cols, b, rs, c0, s_enc, codes, sf, tile_sf, cw, word);
    const int64_t ebytes = rows * cols / 2;
    if (codes_t == nullptr) return;
    // ---- W^T: stage the code words, transpose 8x8 nibble blocks
#pragma unroll
    for (int i = 0; i < 4; ++i) sm.cw[16 * warp + (lane >> 3) + 4 * i][c8] = cw[i];
    if (lane < 4) sm.sc[warp][lane] = rows_ok ? (word >> (8 * lane)) & 0xFFu : 0u;
    __syncthreads();
    if (threadIdx.x < 64) {
        const int ng = threadIdx.x & 7, kg = threadIdx.x >> 3;     // rows 8ng.., columns 8kg..
        uint32_t a[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = sm.cw[8 * ng + j][kg];
        transpose8x8_nibbles(a);
        const bool n_ok = r0 + 8 * ng < rows;
        uint8_t* ctb = codes_t + b * ebytes;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t kk = c0 + 8 * kg + k;                    // W^T row = W column
            if (n_ok && kk < cols) *reinterpret_cast<uint32_t*>(ctb + kk * (rows / 2) + (r0 + 8 * ng) / 2) = a[k];
        }
        // W^T row c0 + t: the scales of the block's four row tiles are 4 contiguous bytes
        const int64_t kk = c0 + threadIdx.x;
        if (kk < cols) {
            const int tj = threadIdx.x >> 4;
            const uint32_t tw = sm.sc[0][tj] | (sm.sc[1][tj] << 8) | (sm.sc[2][tj] << 16) | (sm.sc[3][tj] << 24);
            *reinterpret_cast<uint32_t*>(sf_t + b * sf_bytes(cols, rows) + sf_offset(kk, r0 / 16, rows)) = tw;
        }
    }
    __syncthreads();                                    // shared staging free for the next block
}

// CTA = one 64x64 block (blockIdx.x: columns, blockIdx.y: rows, blockIdx.z:
// batch entry) with the entry's amax already known.
__global__ void __launch_bounds__(128) k_quant2d(const uint16_t* __restrict__ w, int64_t rows,
                                                 int64_t cols, int64_t ld, const float* __restrict__ amax,
                                                 uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                 uint8_t* __restrict__ codes_t, uint8_t* __restrict__ sf_t,
                                                 uint8_t* __restrict__ tile_sf, float* __restrict__ amax_copy) {
    __shared__ Quant2dSmem sm;
    const int64_t b = blockIdx.z;
    if (amax_copy != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) amax_copy[b] = amax[b];
    quant2d_block(w + b * rows * ld, rows, cols, ld, b, (int64_t)blockIdx.y * 64, (int64_t)blockIdx.x * 64,
                  tensor_encode_scale(amax[b]), codes, sf, codes_t, sf_t, tile_sf, sm);
}

// ------------------------------------------------------------------ fused 2D
// Per-entry amax and 2D quantisation of a batched weight [batch, rows, cols]
// (W codes and scales; no W^T) in one launch, reading each element twice
// within a short window so that the second read, for the codes, can hit L2.
// Used for entries too large for k_quant2d_resident (which keeps an entry on
// chip); measured on B300 with the LatentMoE expert weights (5.5 and 21 MB
// per entry), most second reads still missed L2 and this launch took 1.3x the
// time of the two-launch amax + quantise path.
//
// Work is split into items of 16 rows x Q2F_ITEM_COLS columns (16x64 strips
// of 16x16 tiles) of one entry; entry e holds items e*ipe .. (e+1)*ipe - 1.
// Every warp works alone (no block barrier anywhere): warp w of the W warps
// of the grid takes slots w, w + W, w + 2W, ...; slot s is first the amax
// item s (max |w| over the item) and then the quantise item s - lag, with
// lag = ipe + 2W.  A warp keeps the running max and item count of the entry
// it is reducing in registers and publishes them (one atomic max into
// amax[e], then one atomic add into counters[e]) when it moves to another
// entry.  A quantise item of entry e first waits until counters[e] == ipe.
// Every amax item of entry e sits in a slot at least 2W before the first
// quantise item of e, so in the steady state the wait finds the entry
// complete (a margin of W/2 or W/4 made warps wait and ran 1.2-2.7x slower),
// and about one entry plus 2W items pass between the two reads.  The waits cannot deadlock: a quantise item of entry e waits only on
// publications that come before any quantise item of an entry >= e in their
// warp's order, and the launch is cooperative (every warp resident).  Each
// wait is bounded anyway: the first to give up records DEV_TIMEOUT and raises
// counters[batch] (the abort word), after which every warp stops.
// amax[0 .. batch) and counters[0 .. batch] (the last one is the abort word)
// must be zero on entry.
constexpr int Q2F_THREADS = 256;
constexpr int Q2F_STRIPS = 4;                        // 64-column strips of an item
constexpr int64_t Q2F_ITEM_COLS = 64 * Q2F_STRIPS;
constexpr uint64_t Q2F_WAIT_NS = 4000000000ull;

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__global__ void __launch_bounds__(Q2F_THREADS, 2) k_quant2d_fused(const uint16_t* __restrict__ w, int64_t batch,
                                                                  int64_t rows, int64_t cols, int64_t ld,
                                                                  float* __restrict__ amax,
                                                                  uint32_t* __restrict__ counters,
                                                                  uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                                  uint8_t* __restrict__ tile_sf) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (Q2F_THREADS / 32);
    const int64_t wid = (int64_t)blockIdx.x * (Q2F_THREADS / 32) + (threadIdx.x >> 5);
    const int64_t ncc = (cols + Q2F_ITEM_COLS - 1) / Q2F_ITEM_COLS;
    const int64_t ipe = (rows / 16) * ncc;
    const int64_t na = batch * ipe;
    const int64_t lag = ipe + 2 * nw;
    int64_t red_e = -1;              // entry being reduced
    uint32_t red_acc = 0, red_n = 0; // its running max (two bf16 magnitudes) and item count
    int64_t ready_e = -1;            // entry whose amax this warp has seen complete
    float s_enc = 0.0f;
    auto publish = [&]() {
        const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, max(red_acc & 0xFFFFu, red_acc >> 16));
        if (lane == 0) {
            if (m != 0u) atomicMax(reinterpret_cast<unsigned int*>(amax + red_e), m << 16);
            __threadfence();
            atomicAdd(counters + red_e, red_n);
        }
    };
    for (int64_t s = wid; s < na + lag; s += nw) {
        if (s < na) {
            const int64_t e = s / ipe, k = s % ipe;
            if (e != red_e) {
                if (red_e >= 0) publish();
                red_e = e; red_acc = 0; red_n = 0;
            }
            const uint16_t* wb = w + e * rows * ld;
            const int64_t rs = (k / ncc) * 16, cb = (k % ncc) * Q2F_ITEM_COLS;
            uint4 v[Q2F_STRIPS][4];
#pragma unroll
            for (int j = 0; j < Q2F_STRIPS; ++j) quant2d_strip_load(wb, rows, cols, ld, rs, cb + 64 * j, v[j]);
#pragma unroll
            for (int j = 0; j < Q2F_STRIPS; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i) red_acc = absmax_bits(v[j][i], red_acc);
            ++red_n;
        } else if (red_e >= 0) {
            publish();
            red_e = -1;
        }
        const int64_t q = s - lag;
        if (q < 0) continue;
        const int64_t e = q / ipe, k = q % ipe;
        if (e != ready_e) {
            uint32_t am = 0u, ok = 1u;
            if (lane == 0) {
                const uint64_t t0 = globaltimer_ns();
                while (ld_acquire_u32(counters + e) < (uint32_t)ipe) {
                    if (ld_acquire_u32(counters + batch) != 0u) { ok = 0u; break; }
                    if (globaltimer_ns() - t0 > Q2F_WAIT_NS) {
                        raise_status(DEV_TIMEOUT);
                        atomicExch(counters + batch, 1u);
                        ok = 0u;
                        break;
                    }
                    __nanosleep(128);
                }
                if (ok) am = *reinterpret_cast<volatile const uint32_t*>(amax + e);
            }
            if (__shfl_sync(0xFFFFFFFFu, ok, 0) == 0u) return;
            s_enc = tensor_encode_scale(__uint_as_float(__shfl_sync(0xFFFFFFFFu, am, 0)));
            ready_e = e;
        }
        const uint16_t* wb = w + e * rows * ld;
        const int64_t rs = (k / ncc) * 16, cb = (k % ncc) * Q2F_ITEM_COLS;
        uint4 v[Q2F_STRIPS][4];
#pragma unroll
        for (int j = 0; j < Q2F_STRIPS; ++j) quant2d_strip_load(wb, rows, cols, ld, rs, cb + 64 * j, v[j]);
#pragma unroll
        for (int j = 0; j < Q2F_STRIPS; ++j) {
            if (cb + 64 * j >= cols) break;
            uint32_t cw[4], word;
            quant2d_strip_encode(v[j], rows, cols, e, rs, cb + 64 * j, s_enc, codes, sf, tile_sf, cw, word);
        }
    }
    if (red_e >= 0) publish();
}

// ------------------------------------------------------------------ zero codes
// Number of E2M1 codes of magnitude 0 (+0 and -0) among n packed bytes:
// for a nibble value v in 0..7 (sign dropped), v + 7 sets the nibble's bit 3
// exactly when v != 0 and never carries into the next nibble, so the zero
// nibbles are the clear bits 3 of (w & 0x77777777) + 0x77777777.  count
// must be zero on entry.
__device__ __forceinline__ uint32_t zero_nibbles(uint32_t w) {
    return __popc(~((w & 0x77777777u) + 0x77777777u) & 0x88888888u);
}

__global__ void __launch_bounds__(256) k_count_zero_codes(const uint8_t* __restrict__ codes, int64_t nbytes,
                                                          unsigned long long* __restrict__ count) {
    unsigned long long c = 0;
    const int64_t nv = nbytes >> 4;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, nt = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = tid; i < nv; i += nt) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(codes) + i);
        c += zero_nibbles(v.x) + zero_nibbles(v.y) + zero_nibbles(v.z) + zero_nibbles(v.w);
    }
    for (int64_t i = (nv << 4) + tid; i < nbytes; i += nt) {
        const uint32_t b = codes[i];
        c += ((b & 7u) == 0u) + (((b >> 4) & 7u) == 0u);
    }
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
    if ((threadIdx.x & 31) == 0 && c != 0) atomicAdd(count, c);
}

// ------------------------------------------------------------------ PTQ scales
// 1x16 quantisation with each block's E4M3 scale chosen by minimum squared
// error (the NVFP4 PTQ recipe of the "Nemotron 3 Super" summary,
// papers.lianghsun.dev, section 4.2: weight scales calibrated by weight MSE,
// not by the block maximum).  A block whose largest magnitude is 0 gets scale
// 0; otherwise every finite positive E4M3 code c = 1 .. 126 is tried: codes
// q_j = E2M1_RNE(x_j * (S_enc / e4m3(c))) and the FP32 error
// sum_j (x_j - value(q_j) * (e4m3(c) * dec))^2, summed in element order with
// one rounding per operation; the smallest error wins, the largest c on ties.
// One thread per block (its 16 values in registers); the per-code element
// multipliers and reconstruction steps are tables in shared memory.  The
// scale buffer must be zero on entry (its padding stays zero).

// FP32 value of an E2M1 code (sign in bit 3).
__device__ __forceinline__ float e2m1_code_value(uint32_t code) {
    const uint32_t m = code & 7u, e = m >> 1;
    const uint32_t fb = e ? (((e + 126u) << 23) | ((m & 1u) << 22)) : ((m & 1u) ? 0x3F000000u : 0u);
    return __uint_as_float(fb | ((code & 8u) << 28));
}

__global__ void __launch_bounds__(256) k_quant1d_mse(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                                                     int64_t ld, const float* __restrict__ amax,
                                                     uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                     float* __restrict__ amax_copy) {
    __shared__ float s_ratio[128], s_step[128];
    const float s_enc = tensor_encode_scale(amax[0]);
    const float dec = tensor_decode_scale(amax[0]);
    if (threadIdx.x >= 1 && threadIdx.x <= 126) {
        s_ratio[threadIdx.x] = element_ratio(s_enc, threadIdx.x);
        s_step[threadIdx.x] = __fmul_rn(e4m3_to_float(threadIdx.x), dec);
    }
    if (amax_copy != nullptr && blockIdx.x == 0 && threadIdx.x == 0) amax_copy[0] = amax[0];
    __syncthreads();
    const int64_t nb = cols >> 4, total = rows * nb;
    const bool vec = ((ld & 7) == 0) && ((reinterpret_cast<uintptr_t>(x) & 15) == 0);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / nb, b = i - r * nb;
        const uint16_t* src = x + r * ld + 16 * b;
        float xv[16];
        if (vec) {
            const uint4 a0 = __ldg(reinterpret_cast<const uint4*>(src));
            const uint4 a1 = __ldg(reinterpret_cast<const uint4*>(src) + 1);
            const uint32_t w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) { xv[2 * j] = bf16_lo(w[j]); xv[2 * j + 1] = bf16_hi(w[j]); }
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) xv[j] = __uint_as_float((uint32_t)__ldg(src + j) << 16);
        }
        float bamax = 0.0f;
#pragma unroll
        for (int j = 0; j < 16; ++j) bamax = fmaxf(bamax, fabsf(xv[j]));
        uint32_t bestc = 0;
        if (bamax != 0.0f) {
            float best = 0.0f;
            for (uint32_t c = 1; c <= 126; ++c) {
                const float rc = s_ratio[c], st = s_step[c];
                float f[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) f[j] = __fmul_rn(xv[j], rc);
                const float lo8[8] = {f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7]};
                const float hi8[8] = {f[8], f[9], f[10], f[11], f[12], f[13], f[14], f[15]};
                const uint32_t q0 = e2m1x8_rne(lo8), q1 = e2m1x8_rne(hi8);
                float err = 0.0f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const uint32_t q = ((j < 8 ? q0 : q1) >> (4 * (j & 7))) & 15u;
                    const float d = __fsub_rn(xv[j], __fmul_rn(e2m1_code_value(q), st));
                    err = __fadd_rn(err, __fmul_rn(d, d));
                }
                if (bestc == 0 || err <= best) { best = err; bestc = c; }
            }
        }
        uint2 cw = make_uint2(0u, 0u);
        if (bestc != 0) {
            const float rc = s_ratio[bestc];
            float lo8[8], hi8[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) { lo8[j] = __fmul_rn(xv[j], rc); hi8[j] = __fmul_rn(xv[8 + j], rc); }
            cw = make_uint2(e2m1x8_rne(lo8), e2m1x8_rne(hi8));
        }
        // a code row is cols/2 bytes (a multiple of 8): 8-byte stores are aligned
        *reinterpret_cast<uint2*>(codes + r * (cols >> 1) + 8 * b) = cw;
        sf[sf_offset(r, b, cols)] = (uint8_t)bestc;
    }
}

// ------------------------------------------------------------------ FP16 SR
// FP32 -> FP16 with stochastic rounding by the Philox-5 word of each element
// (the SSM-cache recipe of the "Nemotron 3 Super" summary, papers.lianghsun.dev,
// section 4.3).  For m = |x| < 65504 with FP16 neighbours lo <= m < hi and
// p = (m - lo) / (hi - lo), the magnitude becomes hi iff
// u < 256 * ceil(p * 2^24); m >= 65504 saturates to 65504, NaN becomes the
// quiet NaN 0x7E00, the sign is kept.  Integer form:
//   FP16 normal range (m >= 2^-14): the 13 FP32 mantissa bits below the FP16
//     ones are the fraction p * 2^13; adding ~u >> 19 carries into the FP16
//     bits exactly when u >> 19 < that fraction, then the exponent is rebiased;
//   FP16 subnormal range: |x| * 2^24 (exact) splits into the FP16 code floor
//     and the fraction p, compared with u at 2^-24 resolution.
// Identical to the definition for every FP32 pattern (checked exhaustively on
// the host).
__device__ __forceinline__ uint32_t fp16_sr(float x, uint32_t u) {
    const uint32_t bits = __float_as_uint(x);
    const uint32_t mb = bits & 0x7FFFFFFFu;
    const uint32_t sign = (bits >> 16) & 0x8000u;
    if (mb > 0x7F800000u) return sign | 0x7E00u;
    if (mb >= 0x477FE000u) return sign | 0x7BFFu;
    if (mb >= 0x38800000u) return sign | (((mb + (~u >> 19)) >> 13) - (112u << 10));
    const float v = fabsf(x) * 16777216.0f;
    const float fl = floorf(v);
    const uint32_t c = __float2uint_ru((v - fl) * 16777216.0f);
    const uint32_t up = (uint64_t)u < ((uint64_t)c << 8) ? 1u : 0u;
    return sign | ((uint32_t)fl + up);
}

// out[e] = fp16_sr(x[e], word e of (seed, e)): four elements per thread and
// Philox call (counter e / 4), 16-byte loads and 8-byte stores when aligned.
__global__ void __launch_bounds__(256) k_sr_fp16(const float* __restrict__ x, int64_t n, uint64_t seed,
                                                 uint16_t* __restrict__ out) {
    const PhiloxKeys key = philox_keys(seed);
    const bool vec = ((reinterpret_cast<uintptr_t>(x) & 15) == 0) && ((reinterpret_cast<uintptr_t>(out) & 7) == 0);
    const int64_t nq = (n + 3) >> 2;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < nq; q += (int64_t)gridDim.x * blockDim.x) {
        const uint4 w = sr_words(key, (uint64_t)q);
        const int64_t e0 = q << 2;
        if (vec && e0 + 4 <= n) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(x + e0));
            const uint32_t lo = fp16_sr(v.x, w.x) | (fp16_sr(v.y, w.y) << 16);
            const uint32_t hi = fp16_sr(v.z, w.z) | (fp16_sr(v.w, w.w) << 16);
            *reinterpret_cast<uint2*>(out + e0) = make_uint2(lo, hi);
        } else {
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
            for (int i = 0; i < 4 && e0 + i < n; ++i) out[e0 + i] = (uint16_t)fp16_sr(__ldg(x + e0 + i), ws[i]);
        }
    }
}

// Padding of the 2D scale buffers (per batch entry: blockIdx.y).
__global__ void __launch_bounds__(256) k_quant2d_pad(uint8_t* __restrict__ sf, uint8_t* __restrict__ sf_t,
                                                     int64_t rows, int64_t cols) {
    const int b = blockIdx.y;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nt = (int64_t)gridDim.x * blockDim.x;
    zero_sf_padding(sf + b * sf_bytes(rows, cols), rows, cols, tid, nt);
    if (sf_t != nullptr) zero_sf_padding(sf_t + b * sf_bytes(cols, rows), cols, rows, tid, nt);
}

// ------------------------------------------------------------------ RHT
// Two lanes of the butterfly at once: (a0, a1) += (b0, b1) and (b0, b1) =
// old (a0, a1) - (b0, b1), each lane rounded once (add/sub.rn.f32x2, the same
// IEEE operation as __fadd_rn / __fsub_rn, subnormals kept).
__device__ __forceinline__ void addsub2(float& a0, float& a1, float& b0, float& b1) {
    asm("{\n\t.reg .b64 a, b, s, d;\n\t"
        "mov.b64 a, {%0, %1};\n\tmov.b64 b, {%2, %3};\n\t"
        "add.rn.f32x2 s, a, b;\n\tsub.rn.f32x2 d, a, b;\n\t"
        "mov.b64 {%0, %1}, s;\n\tmov.b64 {%2, %3}, d;\n\t}"
        : "+f"(a0), "+f"(a1), "+f"(b0), "+f"(b1));
}

// (a0, a1) *= c, each lane rounded once (mul.rn.f32x2).
__device__ __forceinline__ void mul2(float& a0, float& a1, float c) {
    asm("{\n\t.reg .b64 a, k;\n\tmov.b64 a, {%0, %1};\n\tmov.b64 k, {%2, %2};\n\t"
        "mul.rn.f32x2 a, a, k;\n\tmov.b64 {%0, %1}, a;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(c));
}

// y = 0.25 * H16 * (s .* x) on one 16-token chunk, FP32 butterfly with
// strides 1, 2, 4, 8 (Sylvester order); strides 2, 4 and 8 and the factor
// 1/4 run on pairs of lanes (packed f32x2 operations).  FOLD puts the signs
// into the first stage: s_i x_i is an exact multiply by +-1 and
// s_j x_j + (s_i x_i) one fused multiply-add by +-1, which rounds once like
// the plain add or subtract, so both forms give the same bits.  Measured on
// Ultra dY, the folded form makes the amax and RNE passes up to 9 % faster and
// the SR encoders 1 % slower, so those keep the separate sign flips.  SCALE
// false leaves out the factor 1/4 (for maxima: max RN(|y_i| / 4) =
// RN(max |y_i| / 4), rounding being monotone, so it is applied once to the max).
template <bool FOLD, bool SCALE = true>
__device__ __forceinline__ void rht16(float (&x)[16], uint32_t sign_mask) {
    if (FOLD) {
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            const float si = ((sign_mask >> i) & 1u) ? -1.0f : 1.0f;
            const float sj = ((sign_mask >> (i + 1)) & 1u) ? -1.0f : 1.0f;
            const float a = __fmul_rn(x[i], si), c = x[i + 1];
            x[i] = __fmaf_rn(sj, c, a);
            x[i + 1] = __fmaf_rn(-sj, c, a);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if ((sign_mask >> i) & 1u) x[i] = -x[i];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            const float a = x[i], c = x[i + 1];
            x[i] = __fadd_rn(a, c);
            x[i + 1] = __fsub_rn(a, c);
        }
    }
#pragma unroll
    for (int h = 2; h < 16; h <<= 1)
#pragma unroll
        for (int i = 0; i < 16; i += 2)
            if ((i & h) == 0) addsub2(x[i], x[i + 1], x[i + h], x[i + h + 1]);
    if (SCALE) {
#pragma unroll
        for (int i = 0; i < 16; i += 2) mul2(x[i], x[i + 1], 0.25f);
    }
}

// CTA = 64 tokens x 256 channels, 256 threads.  The tile is staged in
// shared memory with 16-byte loads (element loads when rows are not 16-byte
// aligned); thread t then owns channel c0 + t and the tile's four 16-token
// chunks.
// MODE 0: amax of the transform (amax must be zero on entry).
// MODE 1/2: transform + quantise (RNE / SR) into the transposed operand
// [cols, tokens]: codes_t [cols, tokens/2], sf_t for [cols, tokens].
// GROUPED: x holds expert-sorted tokens (rows of expert g: offsets[g] ..
// offsets[g+1]); expert g's segment, padded with zero tokens to a multiple of
// 64, occupies output columns kpad[g] .. kpad[g+1] of the [cols, kt] operand
// (kpad = sums of the padded counts), is transformed in 16-token chunks and
// quantised with its own amax (amax[g]).  A block covers 64 padded tokens of
// one expert; blocks past kpad[G] do nothing.  Dynamic shared memory: two
// tables of G+1 ints.
// MODE 4 (the dual stochastic encoder of a gradient, one read of each tile):
// MODE 2's transposed RHT operand with seed / amax, and from the same staged
// tile the row-wise 1x16 SR operand [tokens, cols] of the row quantiser
// (seed_row, tensor amax amax_row[0]; SR index e = t * cols + c) into
// codes_r / sf_r, whose zero-magnitude codes are added to *zero_count
// (nullable).  cols % 16 == 0.
struct RowSR {
    const float* amax_row = nullptr;
    uint64_t seed_row = 0;
    uint8_t* codes_r = nullptr;
    uint8_t* sf_r = nullptr;
    unsigned long long* zero_count = nullptr;
    float* amax_row_copy = nullptr;     // receives amax_row[0] (nullable)
};

using RhtTile = uint16_t[256 + 8];

// Row operand of the dual encoder from a staged 64 x 256 tile (token rows t0
// .., channels c0 ..; ntok valid rows): thread tid encodes blocks
// 4 (tid & 3) .. + 3 (64 channels) of token row tid >> 2 with the row SR words
// and stores its codes and scale word.  Returns its zero-magnitude codes.
// The block loop stays rolled: the SR encoders are large, and the smaller
// code made the Ultra dual encoder 7 % faster (fewer instruction-fetch stalls).
__device__ __forceinline__ uint32_t rht_rows_sr(const RhtTile* tile, int tid, int64_t t0, int64_t c0, int ntok,
                                                int64_t cols, const RowSR& rsr, float s_row,
                                                const PhiloxKeys& key_r) {
    const int r = tid >> 2, part = tid & 3;
    const int64_t t = t0 + r;
    uint32_t zeros = 0, word = 0;
    const bool row_ok = r < ntok;
    const int64_t cp = c0 + 64 * part;
    // a code row is cols/2 bytes, a multiple of 8 only: 8-byte stores
    uint8_t* dst = rsr.codes_r + t * (cols >> 1) + (cp >> 1);
#pragma unroll 1
    for (int b = 0; b < 4; ++b) {
        const int64_t c = cp + 16 * b;
        if (!row_ok || c >= cols) break;
        const uint4 va = *reinterpret_cast<const uint4*>(&tile[r][64 * part + 16 * b]);
        const uint4 vb = *reinterpret_cast<const uint4*>(&tile[r][64 * part + 16 * b + 8]);
        const uint32_t m = bf16x16_absmax(va, vb);
        const uint32_t sc = block_scale(__uint_as_float(m << 16), s_row);
        word |= sc << (8 * b);
        uint32_t w0 = 0u, w1 = 0u;
        if (sc != 0) {
            const float ratio = element_ratio(s_row, sc);
            const uint64_t e0 = (uint64_t)t * (uint64_t)cols + (uint64_t)c;
            w0 = encode8<true>(va, ratio, false, key_r, e0);
            w1 = encode8<true>(vb, ratio, false, key_r, e0 + 8);
        }
        zeros += zero_nibbles(w0) + zero_nibbles(w1);
        reinterpret_cast<uint2*>(dst)[b] = make_uint2(w0, w1);
    }
    // four scale columns from a multiple of 4: one word (zeros past cols are
    // the scale padding of the last atom column)
    if (row_ok && cp < cols) *reinterpret_cast<uint32_t*>(rsr.sf_r + sf_offset(t, cp >> 4, cols)) = word;
    return zeros;
}

// Transposed RHT operand from a staged tile: thread tid owns channel c (the
// tile's column tid) and the tile's nchunks 16-token chunks starting at token
// t0 of the [*, ocols] output; each chunk is transformed, block-scaled and
// encoded (SR words of element c * ocols + token, or RNE), then the codes and
// scale bytes are stored (a code row is ocols/2 bytes, a multiple of 8, so
// 8-byte stores are aligned).  The SR chunk loop stays rolled (smaller code:
// 8-13 % faster SR encoders); the RNE one is unrolled (5 % faster RNE pass).
template <bool SR, bool FOLD>
__device__ __forceinline__ void rht_cols_encode(const RhtTile* tile, int tid, int64_t c, int64_t t0, int nchunks,
                                                int64_t ocols, uint32_t sign_mask, float s_enc,
                                                const PhiloxKeys& key, uint8_t* __restrict__ codes_t,
                                                uint8_t* __restrict__ sf_t) {
    uint32_t sfw = 0;
    const int64_t sfc = t0 >> 4;
    if constexpr (SR) {
        uint2* crow = reinterpret_cast<uint2*>(codes_t + c * (ocols >> 1) + (t0 >> 1));
#pragma unroll 1
        for (int j = 0; j < nchunks; ++j) {
            uint32_t p0 = 0u, p1 = 0u;
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __uint_as_float((uint32_t)tile[16 * j + i][tid] << 16);
            rht16<FOLD>(v, sign_mask);
            float bamax = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) bamax = fmaxf(bamax, fabsf(v[i]));
            const uint32_t sc = block_scale(bamax, s_enc);
            sfw |= sc << (8 * j);
            if (sc != 0) {
                const float ratio = element_ratio(s_enc, sc);
                float f[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) f[i] = __fmul_rn(v[i], ratio);
                const uint64_t e0 = (uint64_t)c * (uint64_t)ocols + (uint64_t)(t0 + 16 * j);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 wd = sr_words(key, (e0 >> 2) + q);
                    const uint32_t ws[4] = {wd.x, wd.y, wd.z, wd.w};
                    uint32_t acc = 0u;
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc |= e2m1_sr(f[4 * q + i], ws[i]) << (4 * (4 * (q & 1) + i));
                    if (q < 2) p0 |= acc; else p1 |= acc;
                }
            }
            crow[j] = make_uint2(p0, p1);
        }
        if (nchunks == 4) {
            *reinterpret_cast<uint32_t*>(sf_t + sf_offset(c, sfc, ocols)) = sfw;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (j < nchunks) sf_t[sf_offset(c, sfc + j, ocols)] = (uint8_t)(sfw >> (8 * j));
                else if (sfc + j < ((((ocols >> 4) + 3) >> 2) << 2)) sf_t[sf_offset(c, sfc + j, ocols)] = 0;
            }
        }
    } else {
        uint32_t packed[4][2];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            packed[j][0] = packed[j][1] = 0u;
            if (j >= nchunks) continue;
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __uint_as_float((uint32_t)tile[16 * j + i][tid] << 16);
            rht16<FOLD>(v, sign_mask);
            float bamax = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) bamax = fmaxf(bamax, fabsf(v[i]));
            const uint32_t sc = block_scale(bamax, s_enc);
            sfw |= sc << (8 * j);
            if (sc == 0) continue;
            const float ratio = element_ratio(s_enc, sc);
            float f[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) f[i] = __fmul_rn(v[i], ratio);
            const float lo[8] = {f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7]};
            const float hi[8] = {f[8], f[9], f[10], f[11], f[12], f[13], f[14], f[15]};
            packed[j][0] = e2m1x8_rne(lo);
            packed[j][1] = e2m1x8_rne(hi);
        }
        uint2* crow = reinterpret_cast<uint2*>(codes_t + c * (ocols >> 1) + (t0 >> 1));
        if (nchunks == 4) {
#pragma unroll
            for (int j = 0; j < 4; ++j) crow[j] = make_uint2(packed[j][0], packed[j][1]);
            *reinterpret_cast<uint32_t*>(sf_t + sf_offset(c, sfc, ocols)) = sfw;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (j < nchunks) {
                    crow[j] = make_uint2(packed[j][0], packed[j][1]);
                    sf_t[sf_offset(c, sfc + j, ocols)] = (uint8_t)(sfw >> (8 * j));
                } else if (sfc + j < ((((ocols >> 4) + 3) >> 2) << 2)) {
                    sf_t[sf_offset(c, sfc + j, ocols)] = 0;   // scale-column padding of the last atom column
                }
            }
        }
    }
}

template <int MODE, bool GROUPED = false>
__global__ void __launch_bounds__(256) k_rht(const uint16_t* __restrict__ x, int64_t tokens,
                                             int64_t cols, int64_t ld, uint32_t sign_mask,
                                             float* __restrict__ amax, uint64_t seed,
                                             uint8_t* __restrict__ codes_t, uint8_t* __restrict__ sf_t,
                                             float* __restrict__ amax_copy,
                                             const int64_t* __restrict__ offsets = nullptr, int32_t groups = 1,
                                             int64_t kt = 0, RowSR rsr = RowSR{}) {
    __shared__ __align__(16) uint16_t tile[64][256 + 8];
    const int64_t c0 = (int64_t)blockIdx.x * 256, t0 = (int64_t)blockIdx.y * 64;
    const int tid = threadIdx.x;
    int g = 0;                       // expert of this block (GROUPED)
    int64_t src0 = t0;               // first source token of the block
    int nvalid;                      // source tokens of the block (the rest read as zero)
    int nchunks;                     // 16-token chunks written
    const int64_t ocols = GROUPED ? kt : tokens;   // columns of the output operand
    if (GROUPED) {
        extern __shared__ int32_t s_rtab[];
        GroupTables gt{s_rtab, s_rtab + groups + 1};          // pad = kpad: 64-token segments
        build_group_tables(offsets, groups, tokens, gt, 6);
        if (MODE != 0 && amax_copy != nullptr && blockIdx.x == 0 && blockIdx.y == 0)
            for (int i = tid; i < groups; i += blockDim.x) amax_copy[i] = amax[i];
        if (t0 >= gt.pad[groups]) return;     // block-uniform
        int lo = 0, hi = groups;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (gt.pad[mid] <= t0) lo = mid; else hi = mid;
        }
        g = lo;
        src0 = gt.off[g] + (t0 - gt.pad[g]);
        const int64_t left = gt.off[g + 1] - src0;
        nvalid = left < 0 ? 0 : (left > 64 ? 64 : (int)left);
        nchunks = 4;
    } else {
        if (MODE != 0 && MODE != 3 && amax_copy != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && tid == 0)
            amax_copy[0] = amax[0];
        const int64_t left16 = (tokens - t0) >> 4;
        nchunks = left16 < 4 ? (int)left16 : 4;
        nvalid = 16 * nchunks;
    }
    const int ntok = nvalid;
    const bool vec = ((ld & 7) == 0) && ((reinterpret_cast<uintptr_t>(x) & 15) == 0);
    // ---- stage 64 x 256 bf16 (zeros outside the tensor)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int i = tid + 256 * k;
        const int rr = i >> 5, cc = (i & 31) * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        const int64_t gc = c0 + cc;
        if (rr < ntok && gc < cols) {
            const uint16_t* src = x + (src0 + rr) * ld + gc;
            if (vec && gc + 8 <= cols) {
                v = __ldg(reinterpret_cast<const uint4*>(src));
            } else {
                uint16_t e[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) e[j] = (gc + j < cols) ? __ldg(src + j) : (uint16_t)0;
                v = make_uint4(e[0] | ((uint32_t)e[1] << 16), e[2] | ((uint32_t)e[3] << 16),
                               e[4] | ((uint32_t)e[5] << 16), e[6] | ((uint32_t)e[7] << 16));
            }
        }
        *reinterpret_cast<uint4*>(&tile[rr][cc]) = v;
    }
    __syncthreads();
    const int64_t c = c0 + tid;
    const bool active = c < cols;
    if (MODE == 0 || MODE == 3) {
        // MODE 3 also takes the plain max |x| of the same values (one read
        // gives both tensor amaxes of dY: the row quantiser's and the RHT's);
        // amax_copy then receives the plain one
        float m = 0.0f, mp = 0.0f;
        if (active) {
            for (int j = 0; j < nchunks; ++j) {
                float v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = __uint_as_float((uint32_t)tile[16 * j + i][tid] << 16);
                if (MODE == 3) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) mp = fmaxf(mp, fabsf(v[i]));
                }
                rht16<MODE != 2 && MODE != 4, false>(v, sign_mask);
#pragma unroll
                for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
            }
        }
        m = __fmul_rn(m, 0.25f);                // the transform's factor 1/4, once
        block_max_atomic(__float_as_uint(m), amax + g);
        if (MODE == 3) {
            __syncthreads();                    // the reduction buffer is shared by both calls
            block_max_atomic(__float_as_uint(mp), amax_copy);
        }
        return;
    }
    if (MODE == 4) {
        const float s_row = tensor_encode_scale(rsr.amax_row[0]);
        const PhiloxKeys key_r = philox_keys(rsr.seed_row);
        uint32_t zeros = rht_rows_sr(tile, tid, t0, c0, ntok, cols, rsr, s_row, key_r);
        if (rsr.zero_count != nullptr) {
            zeros = __reduce_add_sync(0xFFFFFFFFu, zeros);
            if ((tid & 31) == 0 && zeros != 0) atomicAdd(rsr.zero_count, (unsigned long long)zeros);
        }
        if (rsr.amax_row_copy != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && tid == 0)
            *rsr.amax_row_copy = rsr.amax_row[0];
    }
    if (!active) return;
    const float s_enc = tensor_encode_scale(amax[g]);
    const PhiloxKeys key = philox_keys(seed);
    rht_cols_encode<MODE == 2 || MODE == 4, MODE != 2 && MODE != 4>(tile, tid, c, t0, nchunks, ocols, sign_mask,
                                                                    s_enc, key, codes_t, sf_t);
}

// Persistent form of k_rht for a dense operand whose rows are 16-byte
// aligned (ld % 8 == 0, cols % 8 == 0): MODE 0 (amax of the transform), 1
// (transform + RNE into the transposed operand) and 3 (both amaxes).  CTA b
// takes tiles b, b + G, ... (tile t: token rows 64 (t / tx) .., channels
// 256 (t % tx) ..); while a tile is transformed from one shared buffer, the
// next tile's rows are copied into the other by cp.async (16-byte copies,
// zero-filled outside the tensor), so a CTA always has a tile in flight.  The
// per-tile arithmetic is that of k_rht; the amaxes are reduced over all of a
// CTA's tiles and published once.  The SR modes stay with k_rht: they are
// bound by the integer pipe, and this kernel's three CTAs per SM (two tile
// buffers each) made the Ultra dual encoder 2 % slower than k_rht's four.
constexpr int RHT_TILE_ELEMS = 64 * (256 + 8);
constexpr int RHT_STREAM_SMEM = 2 * RHT_TILE_ELEMS * 2;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

template <int MODE>
__global__ void __launch_bounds__(256, 3) k_rht_stream(const uint16_t* __restrict__ x, int64_t tokens, int64_t cols,
                                                       int64_t ld, uint32_t sign_mask, float* __restrict__ amax,
                                                       uint8_t* __restrict__ codes_t, uint8_t* __restrict__ sf_t,
                                                       float* __restrict__ amax_copy) {
    static_assert(MODE == 0 || MODE == 1 || MODE == 3, "amax and RNE modes only");
    extern __shared__ __align__(16) uint16_t rht_buf[];
    const int tid = threadIdx.x;
    const int64_t tx = (cols + 255) / 256, total = tx * ((tokens + 63) / 64);
    // stage tile t into buffer b (every thread: eight 16-byte copies)
    auto stage = [&](int64_t t, int b) {
        const int64_t r0 = (t / tx) * 64, c0 = (t % tx) * 256;
        uint16_t* tile = rht_buf + b * RHT_TILE_ELEMS;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = tid + 256 * k;
            const int rr = i >> 5, cc = (i & 31) * 8;
            const bool ok = r0 + rr < tokens && c0 + cc < cols;
            const uint16_t* src = ok ? x + (r0 + rr) * ld + c0 + cc : x;
            cp_async16((uint32_t)__cvta_generic_to_shared(tile + rr * (256 + 8) + cc), src, ok ? 16u : 0u);
        }
        cp_async_commit();
    };
    float s_enc = 1.0f;
    if (MODE == 1) {
        s_enc = tensor_encode_scale(amax[0]);
        if (amax_copy != nullptr && blockIdx.x == 0 && tid == 0) amax_copy[0] = amax[0];
    }
    const PhiloxKeys no_key{};
    float m = 0.0f, mp = 0.0f;
    int b = 0;
    int64_t t = blockIdx.x;
    if (t < total) stage(t, 0);
    for (; t < total; t += gridDim.x, b ^= 1) {
        const int64_t tn = t + gridDim.x;
        if (tn < total) stage(tn, b ^ 1);
        else cp_async_commit();                       // keep one group per iteration
        cp_async_wait1();
        __syncthreads();
        const RhtTile* tile = reinterpret_cast<const RhtTile*>(rht_buf + b * RHT_TILE_ELEMS);
        const int64_t t0 = (t / tx) * 64, c = (t % tx) * 256 + tid;
        const int64_t left16 = (tokens - t0) >> 4;
        const int nchunks = left16 < 4 ? (int)left16 : 4;
        if (c < cols) {
            if (MODE == 0 || MODE == 3) {
                for (int j = 0; j < nchunks; ++j) {
                    float v[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float((uint32_t)tile[16 * j + i][tid] << 16);
                    if (MODE == 3) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) mp = fmaxf(mp, fabsf(v[i]));
                    }
                    rht16<true, false>(v, sign_mask);
#pragma unroll
                    for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
                }
            } else {
                rht_cols_encode<false, true>(tile, tid, c, t0, nchunks, tokens, sign_mask, s_enc, no_key, codes_t,
                                             sf_t);
            }
        }
        __syncthreads();                              // buffer b is refilled two iterations on
    }
    if (MODE == 0 || MODE == 3) {
        m = __fmul_rn(m, 0.25f);                      // the transform's factor 1/4, once
        block_max_atomic(__float_as_uint(m), amax);
        if (MODE == 3) {
            __syncthreads();                          // the reduction buffer is shared by both calls
            block_max_atomic(__float_as_uint(mp), amax_copy);
        }
    }
}

}  // namespace nvfp4
