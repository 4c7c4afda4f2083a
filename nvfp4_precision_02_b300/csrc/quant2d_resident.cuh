// quant2d_resident.cuh -- per-entry amax and 2D (16x16) quantisation of a
// batched weight [batch, rows, cols] with one read of HBM, for sm_103a.
//
// Recipe: weights take 2D block scaling ("Nemotron 3 Super -- technical report
// summary", gkm0120.cn, "Infra design" table), each LatentMoE expert with its
// own tensor scale.  The tensor scale needs the entry's max |w| before any
// element can be encoded, so a plain kernel reads every entry twice.
//
// Here the whole GPU works through the entries in order, each CTA (one per SM,
// all resident: cooperative launch) owning the same share of every entry:
//   - the share is a run of units of 16 rows x 256 columns (8 KB of bf16),
//     brought into a ring of shared-memory slots by TMA (2D tiles, zero fill
//     past the last column);
//   - the twelve warps copy each unit, strip by strip (16 rows x 64 columns,
//     4 tiles), into registers and keep each lane's max |w| of the strip; the
//     last of the four warps that read a unit refills its slot with the unit
//     that comes Q2R_SLOTS later, so the ring goes on loading the next
//     entry's share while the CTA waits for this entry's amax;
//   - after its share of entry e the CTA publishes its max (atomic max into
//     amax[e]) and then its unit count (atomic add into counters[e]); once
//     counters[e] holds the entry's unit count, amax[e] is final and the warps
//     encode their strips from registers with the arithmetic of the two-launch
//     path (tile amax, E4M3 scale by block_scale, element multiplier from a
//     per-warp table of the 126 scale codes, E2M1 codes by e2m1x8_rne_bf16,
//     GEMM-ready scale words).
// A warp holds at most Q2R_STRIPS_PER_WARP strips, so a CTA takes at most
// Q2R_MAX_UNITS units of an entry; larger entries use k_quant2d_fused.
// Twelve warps of at most 168 registers (three per SM sub-partition) hide the
// latency of the encoder's dependent steps; all index arithmetic inside the
// loops is 32-bit, from a table of the share's unit coordinates.
//
// Waits are bounded: the first that gives up records DEV_TIMEOUT and raises
// counters[batch] (the abort word); every CTA then stops, after every copy it
// issued has landed.
//
// Each entry costs one grid-wide exchange (about 2 us of atomics, fence and
// polling on B300) and the phases of an entry run one after another, so the
// launch stays above the time of the two-launch path (amax, then quantise)
// for the LatentMoE expert weights; it needs no workspace beyond the counters
// and reads the weights once.
#pragma once

#include "gemm.cuh"   // mbarrier and TMA helpers

namespace nvfp4 {

constexpr int Q2R_WARPS = 12;
constexpr int Q2R_THREADS = 32 * Q2R_WARPS;
constexpr int Q2R_STRIPS_PER_WARP = 6;
constexpr int Q2R_MAX_UNITS = Q2R_STRIPS_PER_WARP * Q2R_WARPS / 4;
constexpr int Q2R_UNIT_COLS = 256;
constexpr int Q2R_SLOT_BYTES = 16 * Q2R_UNIT_COLS * 2;
constexpr int Q2R_SLOTS = 26;
// shared memory: slots | full, empty barriers | per-slot reader and issue
// counts | unit table | per-warp ratio tables | partial maxima, scale, abort
constexpr int Q2R_BAR_OFFSET = Q2R_SLOTS * Q2R_SLOT_BYTES;
constexpr int Q2R_CNT_OFFSET = Q2R_BAR_OFFSET + 16 * Q2R_SLOTS;
constexpr int Q2R_UNIT_OFFSET = Q2R_CNT_OFFSET + 8 * Q2R_SLOTS;
constexpr int Q2R_TAB_OFFSET = Q2R_UNIT_OFFSET + 8 * Q2R_MAX_UNITS;
constexpr int Q2R_RED_OFFSET = Q2R_TAB_OFFSET + 512 * Q2R_WARPS;
constexpr int Q2R_SMEM_BYTES = Q2R_RED_OFFSET + 4 * Q2R_WARPS + 8;

struct Quant2dResidentArgs {
    int64_t batch, rows, cols;
    int64_t units;          // units per entry: rows / 16 * ceil(cols / 256)
    int64_t col_units;      // ceil(cols / 256)
    int32_t pitch;          // bytes per row of a landed unit (the box width)
    float* amax;            // [batch], zero on entry
    uint32_t* counters;     // [batch + 1], zero on entry; counters[batch] is the abort word
    uint8_t* codes;
    uint8_t* sf;
    uint8_t* tile_sf;
};

struct Q2rRing {
    uint32_t slots, full0, empty0;
    uint32_t* readers;      // per slot: strips read so far (four per unit)
    uint32_t* issued;       // per slot: copies issued into it
    const int2* unit;       // per unit of the share: first row, first column
};

// Copy of the k-th unit of this CTA's sequence (entry k / n, unit k % n of
// the share) into its slot.
__device__ __forceinline__ void q2r_issue(const CUtensorMap* map, const Q2rRing& r, uint32_t k, uint32_t n,
                                          uint32_t rows, uint32_t pitch) {
    const uint32_t s = k % Q2R_SLOTS, e = k / n;
    const int2 uc = r.unit[k - e * n];
    mbar_expect_tx(r.full0 + 8 * s, 16u * pitch);
    tma_load_2d(r.slots + s * Q2R_SLOT_BYTES, map, uc.y, (int32_t)(e * rows) + uc.x, r.full0 + 8 * s);
    r.issued[s] += 1u;
}

// Byte offset of scale (r, c) in an entry's GEMM-ready scale layout (the
// 32-bit form of sf_offset; catoms = ceil(cols / 64)).
__device__ __forceinline__ uint32_t sf_offset32(uint32_t r, uint32_t c, uint32_t catoms) {
    return ((r >> 7) * catoms + (c >> 2)) * 512u + (r & 31u) * 16u + ((r >> 5) & 3u) * 4u + (c & 3u);
}

__global__ void __launch_bounds__(Q2R_THREADS, 1) k_quant2d_resident(const __grid_constant__ CUtensorMap map,
                                                                    Quant2dResidentArgs a) {
    extern __shared__ __align__(128) uint8_t q2r_smem[];
    Q2rRing ring;
    ring.slots = smem_u32(q2r_smem);
    ring.full0 = ring.slots + Q2R_BAR_OFFSET;
    ring.empty0 = ring.full0 + 8 * Q2R_SLOTS;
    ring.readers = reinterpret_cast<uint32_t*>(q2r_smem + Q2R_CNT_OFFSET);
    ring.issued = ring.readers + Q2R_SLOTS;
    int2* unit_tab = reinterpret_cast<int2*>(q2r_smem + Q2R_UNIT_OFFSET);
    ring.unit = unit_tab;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, c8 = lane & 7;
    float* ratio_tab = reinterpret_cast<float*>(q2r_smem + Q2R_TAB_OFFSET) + 128 * warp;
    uint32_t* red = reinterpret_cast<uint32_t*>(q2r_smem + Q2R_RED_OFFSET);
    float* s_enc_sh = reinterpret_cast<float*>(red + Q2R_WARPS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + Q2R_WARPS + 1);
    // this CTA's share: units [lo, lo + n) of every entry
    const int64_t lo = (int64_t)blockIdx.x * a.units / gridDim.x;
    const uint32_t n = (uint32_t)(((int64_t)blockIdx.x + 1) * a.units / gridDim.x - lo);
    const uint32_t total = (uint32_t)a.batch * n;
    const uint32_t rows = (uint32_t)a.rows, cols = (uint32_t)a.cols, pitch = (uint32_t)a.pitch;
    const uint32_t half_cols = cols / 2, catoms = (cols / 16 + 3) / 4, tiles_per_row = cols / 16;

    if (threadIdx.x < n) {
        const int64_t u = lo + threadIdx.x;
        unit_tab[threadIdx.x] = make_int2((int)(u / a.col_units) * 16, (int)(u % a.col_units) * Q2R_UNIT_COLS);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < Q2R_SLOTS; ++s) {
            mbar_init(ring.full0 + 8 * s, 1);
            mbar_init(ring.empty0 + 8 * s, 4);       // the four warps that read the unit's strips
            ring.readers[s] = 0u;
            ring.issued[s] = 0u;
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0)
        for (uint32_t k = 0; k < total && k < (uint32_t)Q2R_SLOTS; ++k) q2r_issue(&map, ring, k, n, rows, pitch);

    uint4 v[Q2R_STRIPS_PER_WARP][4];
    uint32_t mt[Q2R_STRIPS_PER_WARP];            // the lane's max magnitude over each strip
    const int nq = 4 * (int)n;
    for (uint32_t e = 0; e < (uint32_t)a.batch; ++e) {
        const uint32_t kbase = e * n;
        // scan: strips to registers, the lane's max of each; the unit's last
        // reader refills its slot
        uint32_t acc = 0;
#pragma unroll
        for (int j = 0; j < Q2R_STRIPS_PER_WARP; ++j) {
            const int q = warp + Q2R_WARPS * j;
            if (q < nq) {
                const uint32_t k = kbase + (q >> 2), s = k % Q2R_SLOTS, ph = (k / Q2R_SLOTS) & 1u;
                const uint32_t col = 64u * (q & 3) + 8u * c8;              // column within the unit
                const bool landed = mbar_wait(ring.full0 + 8 * s, ph, abort_flag);
                const bool in_box = landed && 2u * col < pitch;
                const uint8_t* p = q2r_smem + s * Q2R_SLOT_BYTES + (lane >> 3) * pitch + 2u * col;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    v[j][i] = in_box ? *reinterpret_cast<const uint4*>(p + 4u * i * pitch) : make_uint4(0, 0, 0, 0);
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(ring.empty0 + 8 * s);
                    if ((atomicAdd(ring.readers + s, 1u) & 3u) == 3u && k + Q2R_SLOTS < total &&
                        mbar_wait(ring.empty0 + 8 * s, ph, abort_flag))
                        q2r_issue(&map, ring, k + Q2R_SLOTS, n, rows, pitch);
                }
                mt[j] = max(bf16x16_absmax(v[j][0], v[j][1]), bf16x16_absmax(v[j][2], v[j][3]));
                acc = max(acc, mt[j]);
            } else {
                mt[j] = 0u;
            }
        }
        // publish the share's max and unit count, then wait for the entry's amax
        acc = __reduce_max_sync(0xFFFFFFFFu, acc);
        if (lane == 0) red[warp] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            float s_enc = 0.0f;
            if (!*abort_flag) {
                uint32_t mm = 0;
#pragma unroll
                for (int w = 0; w < Q2R_WARPS; ++w) mm = max(mm, red[w]);
                if (mm != 0u) atomicMax(reinterpret_cast<unsigned int*>(a.amax + e), mm << 16);
                __threadfence();
                atomicAdd(a.counters + e, n);
                const uint64_t t0 = globaltimer_ns();
                while (ld_acquire_u32(a.counters + e) < (uint32_t)a.units) {
                    if (ld_acquire_u32(a.counters + a.batch) != 0u) { *abort_flag = 1; break; }
                    if (globaltimer_ns() - t0 > G_WAIT_NS) {
                        raise_status(DEV_TIMEOUT);
                        atomicExch(a.counters + a.batch, 1u);
                        *abort_flag = 1;
                        break;
                    }
                    __nanosleep(32);
                }
                if (!*abort_flag)
                    s_enc = tensor_encode_scale(__uint_as_float(*reinterpret_cast<volatile const uint32_t*>(a.amax + e)));
            }
            *s_enc_sh = s_enc;
        }
        __syncthreads();
        if (*abort_flag) {
            // nothing is issued any more: stop the other CTAs, then wait until
            // every copy in flight has landed
            if (threadIdx.x == 0) {
                atomicExch(a.counters + a.batch, 1u);
                const uint64_t t0 = globaltimer_ns();
                for (int s = 0; s < Q2R_SLOTS; ++s)
                    if (ring.issued[s] != 0u)
                        while (!mbar_try_wait(ring.full0 + 8 * s, (ring.issued[s] - 1u) & 1u))
                            if (globaltimer_ns() - t0 > G_WAIT_NS) { raise_status(DEV_TIMEOUT); break; }
            }
            return;
        }
        const float s_enc = *s_enc_sh;
        fill_ratio_table(ratio_tab, s_enc);
        uint8_t* codes_e = a.codes + (uint64_t)e * rows * half_cols;
        uint8_t* sf_e = a.sf + (uint64_t)e * (uint64_t)sf_bytes(a.rows, a.cols);
        uint8_t* tile_e = a.tile_sf ? a.tile_sf + (uint64_t)e * (rows / 16) * tiles_per_row : nullptr;
        // encode the share from registers
#pragma unroll
        for (int j = 0; j < Q2R_STRIPS_PER_WARP; ++j) {
            const int q = warp + Q2R_WARPS * j;
            if (q < nq) {
                const int2 uc = unit_tab[q >> 2];
                const uint32_t rs = (uint32_t)uc.x, c0 = (uint32_t)uc.y + 64u * (q & 3);
                if (c0 < cols) {
                    uint32_t m = mt[j];                       // tile amax: lanes 2t, 2t+1 (+8, +16)
                    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
                    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
                    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
                    const uint32_t sc = block_scale(__uint_as_float(m << 16), s_enc);
                    const float ratio = ratio_tab[sc];
                    const bool col_ok = c0 + 8u * c8 < cols;
                    if (col_ok) {
                        uint8_t* cp = codes_e + (rs + (lane >> 3)) * half_cols + (c0 + 8u * c8) / 2;
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            *reinterpret_cast<uint32_t*>(cp + 4u * i * half_cols) =
                                sc ? e2m1x8_rne_bf16(v[j][i], ratio) : 0u;
                    }
                    const uint32_t word = __shfl_sync(0xFFFFFFFFu, sc, 0) | (__shfl_sync(0xFFFFFFFFu, sc, 2) << 8) |
                                          (__shfl_sync(0xFFFFFFFFu, sc, 4) << 16) |
                                          (__shfl_sync(0xFFFFFFFFu, sc, 6) << 24);
                    if (lane < 16) *reinterpret_cast<uint32_t*>(sf_e + sf_offset32(rs + lane, c0 / 16, catoms)) = word;
                    if (tile_e != nullptr && lane < 8 && (lane & 1) == 0 && col_ok)
                        tile_e[(rs / 16) * tiles_per_row + c0 / 16 + (lane >> 1)] = (uint8_t)sc;
                }
            }
        }
    }
}

}  // namespace nvfp4
