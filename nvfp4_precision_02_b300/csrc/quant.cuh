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
    int32_t* off;    // [G+1]
    int32_t* pad;    // [G+1]
};

__device__ void build_group_tables(const int64_t* __restrict__ offsets, int32_t groups,
                                   int64_t rows, GroupTables t) {
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
    // 2) padded scale rows: exclusive sum of ceil(cnt/128)*128
    int32_t local_sum = 0;
    for (int i = 0; i < per; ++i) {
        const int g = g0 + i;
        if (g < groups) local_sum += ((t.off[g + 1] - t.off[g] + 127) >> 7) << 7;
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
            t.pad[g] = acc;
            if (g < groups) acc += ((t.off[g + 1] - t.off[g] + 127) >> 7) << 7;
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
__device__ __forceinline__ uint32_t encode8(const uint4 v, float ratio, bool zero, uint64_t seed,
                                            uint64_t e0) {
    if (zero) return 0u;
    float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                  bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
    uint32_t out = 0;
    if (SR) {
        const uint4 w0 = sr_words(seed, e0 >> 2);
        const uint4 w1 = sr_words(seed, (e0 >> 2) + 1);
        const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) out |= e2m1_sr(__fmul_rn(f[j], ratio), w[j]) << (4 * j);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) out |= e2m1_rne(__fmul_rn(f[j], ratio)) << (4 * j);
    }
    return out;
}

// One warp walks a contiguous range of rows; in each row lane pairs own
// 16-element blocks (lane 2j: first 8 elements, lane 2j+1: last 8).
// x: bf16 [rows, cols] (row stride ld); codes [rows, cols/2]; sf swizzled.
// amax: 1 value (or one per group when GROUPED).  SR index e = r*cols + c.
template <bool SR, bool GROUPED>
__global__ void __launch_bounds__(256) k_quant1d(const uint16_t* __restrict__ x, int64_t rows,
                                                 int64_t cols, int64_t ld,
                                                 const float* __restrict__ amax, uint64_t seed,
                                                 uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                 const int64_t* __restrict__ offsets, int32_t groups,
                                                 float* __restrict__ amax_copy) {
    extern __shared__ int32_t s_tab[];
    GroupTables t{s_tab, s_tab + (GROUPED ? groups + 1 : 0)};
    if (GROUPED) build_group_tables(offsets, groups, rows, t);
    if (amax_copy != nullptr && blockIdx.x == 0) {
        const int n = GROUPED ? groups : 1;
        for (int i = threadIdx.x; i < n; i += blockDim.x) amax_copy[i] = amax[i];
    }
    const int lane = threadIdx.x & 31;
    const int upr = (int)(cols >> 3);
    const int64_t nc = cols >> 4, pc = ((nc + 3) >> 2) << 2;
    int64_t r0, r1;
    warp_rows(rows, r0, r1);
    int g = 0;
    int32_t g_begin = 0, g_end = (int32_t)rows, sf_row0 = 0;
    float s_enc = GROUPED ? 1.0f : tensor_encode_scale(amax[0]);
    bool have_g = false;
    for (int64_t r = r0; r < r1; ++r) {
        if (GROUPED) {
            if (r < t.off[0] || r >= t.off[groups]) continue;
            if (!have_g || r >= g_end || r < g_begin) {
                g = find_group(t.off, groups, (int32_t)r);
                g_begin = t.off[g];
                g_end = t.off[g + 1];
                sf_row0 = t.pad[g];
                s_enc = tensor_encode_scale(amax[g]);
                have_g = true;
            }
        }
        const int64_t sr = GROUPED ? sf_row0 + (r - g_begin) : r;
        const uint16_t* row = x + r * ld;
        uint8_t* crow = codes + r * (cols >> 1);
        for (int base = 0; base < upr; base += 64) {
            uint4 v[2];
            bool ok[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int u = base + i * 32 + lane;
                ok[i] = u < upr;
                v[i] = ok[i] ? __ldg(reinterpret_cast<const uint4*>(row + u * 8)) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int u = base + i * 32 + lane;
                uint32_t m = absmax_bits(v[i], 0u);
                m = max(m & 0xFFFFu, m >> 16);
                m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
                const float bamax = __uint_as_float(m << 16);
                const uint32_t s = block_scale(bamax, s_enc);
                const float ratio = s ? element_ratio(s_enc, s) : 0.0f;
                if (ok[i]) {
                    const uint32_t packed = encode8<SR>(v[i], ratio, s == 0, seed,
                                                        (uint64_t)r * (uint64_t)cols + (uint64_t)u * 8);
                    *reinterpret_cast<uint32_t*>(crow + u * 4) = packed;
                    if ((lane & 1) == 0) {
                        const int64_t c = u >> 1;
                        sf[sf_offset(sr, c, cols)] = (uint8_t)s;
                        if (c == nc - 1)
                            for (int64_t cc = nc; cc < pc; ++cc) sf[sf_offset(sr, cc, cols)] = 0;
                    }
                }
            }
        }
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
// CTA tile 64x64 of one batch entry; 128 threads; sub-tile s = tid/8 (4x4 of
// 16x16 tiles); thread k = tid%8 of a sub-tile owns its rows 2k, 2k+1 (for
// W) and its columns 2k, 2k+1 (for W^T).
__global__ void __launch_bounds__(128) k_quant2d(const uint16_t* __restrict__ w, int64_t rows,
                                                 int64_t cols, int64_t ld, const float* __restrict__ amax,
                                                 uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                 uint8_t* __restrict__ codes_t, uint8_t* __restrict__ sf_t,
                                                 uint8_t* __restrict__ tile_sf, float* __restrict__ amax_copy) {
    __shared__ __align__(16) uint16_t tile[64][72];
    const int b = blockIdx.z;
    const int64_t r0 = (int64_t)blockIdx.y * 64, c0 = (int64_t)blockIdx.x * 64;
    const uint16_t* wb = w + (int64_t)b * rows * ld;
    const int tid = threadIdx.x;
    if (amax_copy != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) amax_copy[b] = amax[b];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int i = tid + 128 * j;
        const int rr = i >> 3, cc = (i & 7) * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r0 + rr < rows && c0 + cc < cols)
            v = __ldg(reinterpret_cast<const uint4*>(wb + (r0 + rr) * ld + c0 + cc));
        *reinterpret_cast<uint4*>(&tile[rr][cc]) = v;
    }
    __syncthreads();
    const int st = tid >> 3, k = tid & 7;
    const int sr = (st >> 2) * 16, sc = (st & 3) * 16;        // sub-tile origin in the CTA tile
    const bool valid = (r0 + sr < rows) && (c0 + sc < cols);   // dims are multiples of 16
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 16; ++j) m = max(m, (uint32_t)(tile[sr + 2 * k + i][sc + j] & 0x7FFFu));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
    if (!valid) return;
    const float s_enc = tensor_encode_scale(amax[b]);
    const uint32_t s = block_scale(__uint_as_float(m << 16), s_enc);
    const float ratio = s ? element_ratio(s_enc, s) : 0.0f;
    const int64_t ti = (r0 + sr) >> 4, tj = (c0 + sc) >> 4;
    const int64_t ebytes = rows * cols / 2;
    // W rows
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int rr = sr + 2 * k + i;
        uint32_t lo = 0, hi = 0;
        if (s) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                lo |= e2m1_rne(__fmul_rn(__uint_as_float((uint32_t)tile[rr][sc + j] << 16), ratio)) << (4 * j);
                hi |= e2m1_rne(__fmul_rn(__uint_as_float((uint32_t)tile[rr][sc + 8 + j] << 16), ratio)) << (4 * j);
            }
        }
        const int64_t gr = r0 + rr;
        *reinterpret_cast<uint2*>(codes + b * ebytes + gr * (cols / 2) + (c0 + sc) / 2) = make_uint2(lo, hi);
        sf[b * sf_bytes(rows, cols) + sf_offset(gr, tj, cols)] = (uint8_t)s;
    }
    // W^T rows (columns of W)
    if (codes_t != nullptr) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int cc = sc + 2 * k + i;
            uint32_t lo = 0, hi = 0;
            if (s) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    lo |= e2m1_rne(__fmul_rn(__uint_as_float((uint32_t)tile[sr + j][cc] << 16), ratio)) << (4 * j);
                    hi |= e2m1_rne(__fmul_rn(__uint_as_float((uint32_t)tile[sr + 8 + j][cc] << 16), ratio)) << (4 * j);
                }
            }
            const int64_t gc = c0 + cc;
            *reinterpret_cast<uint2*>(codes_t + b * ebytes + gc * (rows / 2) + (r0 + sr) / 2) = make_uint2(lo, hi);
            sf_t[b * sf_bytes(cols, rows) + sf_offset(gc, ti, rows)] = (uint8_t)s;
        }
    }
    if (tile_sf != nullptr && k == 0) tile_sf[(int64_t)b * (rows / 16) * (cols / 16) + ti * (cols / 16) + tj] = (uint8_t)s;
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
// y = 0.25 * H16 * (s .* x) on one 16-token chunk, FP32 butterfly with
// strides 1, 2, 4, 8 (Sylvester order).
__device__ __forceinline__ void rht16(float (&x)[16], uint32_t sign_mask) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
        if ((sign_mask >> i) & 1u) x[i] = -x[i];
#pragma unroll
    for (int h = 1; h < 16; h <<= 1)
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if ((i & h) == 0) {
                const float a = x[i], c = x[i + h];
                x[i] = __fadd_rn(a, c);
                x[i + h] = __fsub_rn(a, c);
            }
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = __fmul_rn(x[i], 0.25f);
}

// One thread = one channel c and 4 consecutive 16-token chunks (64 tokens).
// MODE 0: amax of the transform (amax must be zero on entry).
// MODE 1/2: transform + quantise (RNE / SR) into the transposed operand
// [cols, tokens]: codes_t [cols, tokens/2], sf_t for [cols, tokens].
template <int MODE>
__global__ void __launch_bounds__(128) k_rht(const uint16_t* __restrict__ x, int64_t tokens,
                                             int64_t cols, int64_t ld, uint32_t sign_mask,
                                             float* __restrict__ amax, uint64_t seed,
                                             uint8_t* __restrict__ codes_t, uint8_t* __restrict__ sf_t,
                                             float* __restrict__ amax_copy) {
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t t0 = (int64_t)blockIdx.y * 64;
    if (MODE != 0 && amax_copy != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
        amax_copy[0] = amax[0];
    const bool active = c < cols;
    const int64_t left16 = (tokens - t0) >> 4;
    const int nchunks = left16 < 4 ? (int)left16 : 4;
    if (MODE == 0) {
        float m = 0.0f;
        if (active) {
            for (int j = 0; j < nchunks; ++j) {
                float v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    v[i] = __uint_as_float((uint32_t)__ldg(x + (t0 + 16 * j + i) * ld + c) << 16);
                rht16(v, sign_mask);
#pragma unroll
                for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
            }
        }
        block_max_atomic(__float_as_uint(m), amax);
        return;
    }
    if (!active) return;
    const float s_enc = tensor_encode_scale(amax[0]);
    uint32_t packed[4][2];
    uint32_t sfw = 0;
    for (int j = 0; j < nchunks; ++j) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            v[i] = __uint_as_float((uint32_t)__ldg(x + (t0 + 16 * j + i) * ld + c) << 16);
        rht16(v, sign_mask);
        float bamax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) bamax = fmaxf(bamax, fabsf(v[i]));
        const uint32_t s = block_scale(bamax, s_enc);
        sfw |= s << (8 * j);
        uint32_t lo = 0, hi = 0;
        if (s) {
            const float ratio = element_ratio(s_enc, s);
            if (MODE == 2) {
                const uint64_t e0 = (uint64_t)c * (uint64_t)tokens + (uint64_t)(t0 + 16 * j);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 w = sr_words(seed, (e0 >> 2) + q);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t code = e2m1_sr(__fmul_rn(v[4 * q + i], ratio), ws[i]);
                        if (q < 2) lo |= code << (4 * (4 * q + i)); else hi |= code << (4 * (4 * (q - 2) + i));
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    lo |= e2m1_rne(__fmul_rn(v[i], ratio)) << (4 * i);
                    hi |= e2m1_rne(__fmul_rn(v[8 + i], ratio)) << (4 * i);
                }
            }
        }
        packed[j][0] = lo;
        packed[j][1] = hi;
    }
    uint8_t* crow = codes_t + c * (tokens >> 1) + (t0 >> 1);
    const int64_t sfc = t0 >> 4;
    // a code row is tokens/2 bytes (a multiple of 8), so 8-byte stores are aligned
    if (nchunks == 4) {
#pragma unroll
        for (int j = 0; j < 4; ++j) reinterpret_cast<uint2*>(crow)[j] = make_uint2(packed[j][0], packed[j][1]);
        *reinterpret_cast<uint32_t*>(sf_t + sf_offset(c, sfc, tokens)) = sfw;
    } else {
        for (int j = 0; j < nchunks; ++j) {
            reinterpret_cast<uint2*>(crow)[j] = make_uint2(packed[j][0], packed[j][1]);
            sf_t[sf_offset(c, sfc + j, tokens)] = (uint8_t)(sfw >> (8 * j));
        }
        for (int j = nchunks; j < 4; ++j) {
            // scale-column padding of the last atom column (tokens/16 % 4 != 0)
            const int64_t cc = sfc + j;
            if (cc < ((((tokens >> 4) + 3) >> 2) << 2)) sf_t[sf_offset(c, cc, tokens)] = 0;
        }
    }
}

}  // namespace nvfp4
