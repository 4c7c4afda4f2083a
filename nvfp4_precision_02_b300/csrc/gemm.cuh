// gemm.cuh -- NVFP4 block-scaled GEMM on the 5th-generation tensor cores
// (tcgen05.mma kind::mxf4nvf4, E4M3 scales per 16 elements), sm_103a.
//
// C[m, n] = alpha * sum_k (a_k * sa) * (b_k * sb), FP32 accumulation in TMEM,
// alpha = dec_A * dec_B applied once in the epilogue.  These are the fprop,
// dgrad and wgrad GEMMs of the recipe ("Nemotron 3 Super -- technical report
// summary", gkm0120.cn, "Infra design" table; "Nemotron 3 Ultra" report,
// papercache.org translation, section 2.2) and, with per-expert offsets, the
// LatentMoE routed-expert GEMM ("Nemotron 3 Super" summary,
// papers.lianghsun.dev, section 2.2).
//
// Design (one CTA per SM, persistent over output tiles):
//   tile 128 x 256, K stage 256 FP4 elements (128 B per row, 128B-swizzled
//   TMA boxes), 4 stages of A 16 KB + B 32 KB + scales 6 KB in shared memory.
//   warp 0      TMA producer: A and B boxes by cp.async.bulk.tensor, the scale
//               atoms (512 B each, already in the 128x4 layout) by cp.async.bulk
//   warp 1      allocates TMEM; one lane copies the stage's scales into TMEM
//               (tcgen05.cp 32x128b.warpx4) and issues 4 MMAs 128x256x64
//   warps 2..9  epilogue: tcgen05.ld the 128x256 FP32 accumulator (two warps
//               per TMEM lane quarter, 128 columns each), release it to the
//               MMA warp, scale by alpha, round, store rows to global memory
//   TMEM: accumulator columns 0..255; per stage 16 columns of A scales and
//   32 columns of B scales from column 256.
// Every wait is bounded (DEV_TIMEOUT in the status word, then a clean exit).
#pragma once

#include <cuda.h>
#include "common.cuh"
#include "quant.cuh"   // GroupTables / build_group_tables / find_group

namespace nvfp4 {

constexpr int G_BM = 128, G_BN = 256, G_BK = 256;
constexpr int G_STAGES = 4;
constexpr int G_A_BYTES = G_BM * G_BK / 2;                 // 16384
constexpr int G_B_BYTES = G_BN * G_BK / 2;                 // 32768
constexpr int G_SFA_BYTES = (G_BK / 64) * 512;             // 2048
constexpr int G_SFB_BYTES = 2 * (G_BK / 64) * 512;         // 4096
constexpr int G_STAGE_BYTES = G_A_BYTES + G_B_BYTES + G_SFA_BYTES + G_SFB_BYTES;  // 55296
constexpr int G_THREADS = 320;
constexpr int G_TMEM_COLS = 512;
constexpr int G_SF_COL0 = 256;
constexpr int G_SF_COLS_PER_STAGE = 48;
constexpr int G_BAND = 16;                                   // m-tiles per raster band
constexpr uint64_t G_WAIT_NS = 4000000000ull;                // bounded waits: 4 s

// dynamic shared memory: 1 KB alignment slack, stages, barriers, tables
__host__ __device__ constexpr int gemm_smem_bytes(int groups) {
    return 1024 + G_STAGES * G_STAGE_BYTES + 128 + 2 * 4 * (groups + 1);
}

struct GemmParams {
    int64_t M;                  // rows of A (dense) / total rows R (grouped)
    int64_t N;                  // output columns (n per expert when grouped)
    int64_t K;
    const int64_t* offsets;     // grouped: device [groups+1]; dense: nullptr
    int32_t groups;             // 1 for dense
    const uint8_t* sfa;
    const uint8_t* sfb;
    int64_t sfb_group_stride;   // bytes between experts' B scales (grouped)
    const float* amax_a;        // [groups]
    const float* amax_b;        // [groups]
    void* c;
    int64_t ldc;
    bool vec_store;             // rows of C start 16-byte aligned: vector stores
};

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity.  Gives up (false) when
// the shared abort flag is raised or after G_WAIT_NS, raising the flag and
// DEV_TIMEOUT.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0u) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > G_WAIT_NS) {
                *abort_flag = 1;
                raise_status(DEV_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start >> 4 in bits 0-13, leading
// byte offset >> 4 in 16-29, stride byte offset >> 4 in 32-45, descriptor
// version 1 in bits 46-47, swizzle mode in 61-63 (2 = 128B, 0 = none).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swz << 61);
}

// Instruction descriptor of kind::mxf4nvf4: A and B E2M1 (format 1, bits 7-9
// and 10-12), both K-major, N >> 3 in bits 17-22, E4M3 scales (bit 23 = 0),
// M >> 4 in bits 24-28, scale-factor ids 0.
__host__ __device__ constexpr uint32_t mxf4nvf4_idesc(int m, int n) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
}

#define NVFP4_R32(i) "=r"(v[i]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3])
__device__ __forceinline__ void tc_ld_32x32b_x32(uint32_t taddr, uint32_t* v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : NVFP4_R32(0), NVFP4_R32(4), NVFP4_R32(8), NVFP4_R32(12), NVFP4_R32(16), NVFP4_R32(20),
          NVFP4_R32(24), NVFP4_R32(28)
        : "r"(taddr));
}
#undef NVFP4_R32

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ tiles
struct TileCoord {
    int g;            // group
    int mtg;          // global m-tile index (scale atom row of A)
    int nt;           // n-tile
    int32_t row0;     // first A row of the tile
    int32_t rows;     // valid rows (<= 128)
};

// Tiles are numbered in bands of G_BAND m-tiles: inside a band, the m-tile
// runs fastest, so concurrently resident CTAs share B tiles through L2.
__device__ __forceinline__ TileCoord decode_tile(int64_t t, int mtiles, int ntiles, const int32_t* off,
                                                 const int32_t* pad, int groups) {
    const int64_t band_tiles = (int64_t)G_BAND * ntiles;
    const int band = (int)(t / band_tiles);
    const int64_t local = t - (int64_t)band * band_tiles;
    const int bsize = min(G_BAND, mtiles - band * G_BAND);
    TileCoord c;
    c.mtg = band * G_BAND + (int)(local % bsize);
    c.nt = (int)(local / bsize);
    // group: pad[g] <= 128 * mtg < pad[g+1]
    int lo = 0, hi = groups;
    const int32_t key = c.mtg * 128;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pad[mid] <= key) lo = mid; else hi = mid;
    }
    c.g = lo;
    const int32_t lmt = c.mtg - pad[lo] / 128;
    c.row0 = off[lo] + lmt * 128;
    c.rows = min(128, off[lo + 1] - c.row0);
    return c;
}

// ------------------------------------------------------------------ kernel
template <bool OUT_FP32>
__global__ void __launch_bounds__(G_THREADS, 1)
    k_gemm_nvfp4(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                 const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + G_STAGES * G_STAGE_BYTES);
    // bars: full[4], empty[4], acc_full, acc_empty, drain
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * G_STAGES + 3);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int32_t* tab = reinterpret_cast<int32_t*>(smem + G_STAGES * G_STAGE_BYTES + 128);
    const int groups = p.groups;
    GroupTables gt{tab, tab + groups + 1};

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + G_STAGES);
    const uint32_t acc_full = smem_u32(bars + 2 * G_STAGES), acc_empty = acc_full + 8, drain = acc_full + 16;

    if (threadIdx.x == 0) {
        for (int s = 0; s < G_STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 8);
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_a)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_b)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(G_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (p.offsets != nullptr) {
        build_group_tables(p.offsets, groups, p.M, gt);
    } else if (threadIdx.x == 0) {
        gt.off[0] = 0;
        gt.off[1] = (int32_t)p.M;
        gt.pad[0] = 0;
        gt.pad[1] = (int32_t)(((p.M + 127) >> 7) << 7);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int mtiles = gt.pad[groups] >> 7;
    const int ntiles = (int)((p.N + G_BN - 1) / G_BN);
    const int64_t total = (int64_t)mtiles * ntiles;
    const int kstages = (int)((p.K + G_BK - 1) / G_BK);
    const int katoms = (int)((p.K + 63) / 64);
    const int nrb = (int)((p.N + 127) / 128);            // 128-row scale blocks of one B operand
    const int64_t b_rows_per_group = (p.offsets != nullptr) ? p.N : 0;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int32_t issued_ph[G_STAGES];
            for (int i = 0; i < G_STAGES; ++i) issued_ph[i] = -1;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const TileCoord tc = decode_tile(t, mtiles, ntiles, gt.off, gt.pad, groups);
                const int32_t brow0 = (int32_t)(tc.g * b_rows_per_group + (int64_t)tc.nt * G_BN);
                const uint8_t* sfb_g = p.sfb + (int64_t)tc.g * p.sfb_group_stride;
                const bool rb2 = (tc.nt * 2 + 1) < nrb;
                for (int ks = 0; ks < kstages; ++ks) {
                    if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, abort_flag)) { ok = false; break; }
                    const int na = min(4, katoms - 4 * ks);
                    const uint32_t sfbytes = (uint32_t)na * 512u;
                    const uint32_t bar = full0 + 8 * s;
                    mbar_expect_tx(bar, G_A_BYTES + G_B_BYTES + sfbytes * (rb2 ? 3u : 2u));
                    const uint32_t st = smem_u32(stages + s * G_STAGE_BYTES);
                    tma_load_2d(st, &tm_a, ks * 128, tc.row0, bar);
                    tma_load_2d(st + G_A_BYTES, &tm_b, ks * 128, brow0, bar);
                    bulk_load(st + G_A_BYTES + G_B_BYTES, p.sfa + ((int64_t)tc.mtg * katoms + 4 * ks) * 512, sfbytes, bar);
                    bulk_load(st + G_A_BYTES + G_B_BYTES + G_SFA_BYTES,
                              sfb_g + ((int64_t)(tc.nt * 2) * katoms + 4 * ks) * 512, sfbytes, bar);
                    if (rb2)
                        bulk_load(st + G_A_BYTES + G_B_BYTES + G_SFA_BYTES + 2048,
                                  sfb_g + ((int64_t)(tc.nt * 2 + 1) * katoms + 4 * ks) * 512, sfbytes, bar);
                    issued_ph[s] = (int32_t)ph;
                    if (++s == G_STAGES) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                // let every copy already issued land before the CTA exits
                volatile int never = 0;
                for (int i = 0; i < G_STAGES; ++i)
                    if (issued_ph[i] >= 0) mbar_wait(full0 + 8 * i, (uint32_t)issued_ph[i], &never);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = mxf4nvf4_idesc(G_BM, G_BN);
            int s = 0;
            uint32_t ph = 0, it = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
                const TileCoord tc = decode_tile(t, mtiles, ntiles, gt.off, gt.pad, groups);
                const bool rb2 = (tc.nt * 2 + 1) < nrb;
                (void)tc;
                if (!mbar_wait(acc_empty, (it & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                for (int ks = 0; ks < kstages; ++ks) {
                    if (!mbar_wait(full0 + 8 * s, ph, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const int na = min(4, katoms - 4 * ks);
                    const uint32_t st = smem_u32(stages + s * G_STAGE_BYTES);
                    const uint32_t sfa_t = tmem + G_SF_COL0 + s * G_SF_COLS_PER_STAGE;
                    const uint32_t sfb_t = sfa_t + 16;
                    for (int j = 0; j < na; ++j) {
                        tc_cp_sf(sfa_t + 4 * j, smem_desc(st + G_A_BYTES + G_B_BYTES + 512 * j, 0, 128, 0));
                        tc_cp_sf(sfb_t + 8 * j, smem_desc(st + G_A_BYTES + G_B_BYTES + G_SFA_BYTES + 512 * j, 0, 128, 0));
                        if (rb2)
                            tc_cp_sf(sfb_t + 8 * j + 4,
                                     smem_desc(st + G_A_BYTES + G_B_BYTES + G_SFA_BYTES + 2048 + 512 * j, 0, 128, 0));
                    }
                    for (int j = 0; j < na; ++j) {
                        const uint64_t ad = smem_desc(st + 32 * j, 16, 1024, 2);
                        const uint64_t bd = smem_desc(st + G_A_BYTES + 32 * j, 16, 1024, 2);
                        tc_mma(tmem, ad, bd, idesc, sfa_t + 4 * j, sfb_t + 8 * j, (ks | j) != 0 ? 1u : 0u);
                    }
                    tc_commit(empty0 + 8 * s);
                    if (++s == G_STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                tc_commit(acc_full);
            }
            // every MMA issued by this thread completes before teardown
            tc_commit(drain);
            volatile int never = 0;
            mbar_wait(drain, 0, &never);
        }
    } else {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;                  // TMEM lane quarter this warp may access
        const int h = (warp - 2) >> 2;           // column half
        const int r = q * 32 + lane;             // row inside the tile
        uint32_t it = 0;
        for (int64_t t = blockIdx.x; t < total; t += gridDim.x, ++it) {
            const TileCoord tc = decode_tile(t, mtiles, ntiles, gt.off, gt.pad, groups);
            const float alpha = __fmul_rn(tensor_decode_scale(p.amax_a[tc.g]), tensor_decode_scale(p.amax_b[tc.g]));
            if (!mbar_wait(acc_full, it & 1u, abort_flag)) break;
            tc_fence_after();
            uint32_t v[128];
            const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * 128);
            tc_ld_32x32b_x32(taddr, v);
            tc_ld_32x32b_x32(taddr + 32, v + 32);
            tc_ld_32x32b_x32(taddr + 64, v + 64);
            tc_ld_32x32b_x32(taddr + 96, v + 96);
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
            if (r < tc.rows) {
                const int64_t row = tc.row0 + r;
                const int64_t col0 = (int64_t)tc.nt * G_BN + h * 128;
                if (OUT_FP32) {
                    float* out = reinterpret_cast<float*>(p.c) + row * p.ldc + col0;
#pragma unroll
                    for (int i = 0; i < 128; i += 4) {
                        const float4 o = make_float4(__fmul_rn(alpha, __uint_as_float(v[i])),
                                                     __fmul_rn(alpha, __uint_as_float(v[i + 1])),
                                                     __fmul_rn(alpha, __uint_as_float(v[i + 2])),
                                                     __fmul_rn(alpha, __uint_as_float(v[i + 3])));
                        if (p.vec_store && col0 + i + 4 <= p.N) {
                            *reinterpret_cast<float4*>(out + i) = o;
                        } else {
                            const float oo[4] = {o.x, o.y, o.z, o.w};
                            for (int j = 0; j < 4; ++j)
                                if (col0 + i + j < p.N) out[i + j] = oo[j];
                        }
                    }
                } else {
                    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.c) + row * p.ldc + col0;
#pragma unroll
                    for (int i = 0; i < 128; i += 8) {
                        uint32_t w[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(
                                __fmul_rn(alpha, __uint_as_float(v[i + 2 * j])),
                                __fmul_rn(alpha, __uint_as_float(v[i + 2 * j + 1])));
                            w[j] = *reinterpret_cast<const uint32_t*>(&b2);
                        }
                        if (p.vec_store && col0 + i + 8 <= p.N) {
                            *reinterpret_cast<uint4*>(out + i) = make_uint4(w[0], w[1], w[2], w[3]);
                        } else {
                            const uint16_t* hw = reinterpret_cast<const uint16_t*>(w);
                            for (int j = 0; j < 8; ++j)
                                if (col0 + i + j < p.N) reinterpret_cast<uint16_t*>(out)[i + j] = hw[j];
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(G_TMEM_COLS) : "memory");
    }
}

// ------------------------------------------------------------------ timeout probe
// One block waits on an mbarrier that nothing completes; the bounded wait
// gives up after timeout_ns and records DEV_TIMEOUT.
__global__ void k_wait_probe(uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(b, 0)) return;
        if (globaltimer_ns() - t0 > timeout_ns) {
            raise_status(DEV_TIMEOUT);
            mbar_arrive(b);      // complete the phase so nothing is left pending
            return;
        }
    }
}

}  // namespace nvfp4
