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
// Design (one CTA per SM, persistent over output tiles of 128 x 256):
//   K stage 256 FP4 elements (128 B per row, 128B-swizzled TMA boxes);
//   stages of A 16 KB + B 32 KB + scales 6 KB in shared memory.
//   warp 0        A/B producer: the A and B boxes by cp.async.bulk.tensor
//                 (or, when a code row is not a 16-byte multiple, row copies
//                 into the same swizzled layout by the warp's lanes)
//   warp 22       scale producer: the stage's scale atoms (512 B each,
//                 already in the 128x4 layout) by cp.async.bulk on a landing
//                 barrier of their own, so copy issue is split over two warps
//   warp 1        allocates TMEM; one lane issues the 4 MMAs 128x256x64 of a
//                 stage from one asm block (descriptors advanced in place) and,
//                 while they run, tests (without waiting) whether the next
//                 stage has landed
//   warps 2..5    scale-factor writers, one per TMEM lane quarter: when a
//                 stage lands, each lane reads the 16 bytes it owns of every
//                 128x4 scale atom from shared memory and writes them into
//                 TMEM with tcgen05.st.  In every quarter, column j of an
//                 atom's 4 columns then holds rows 32j .. 32j+31 (the same
//                 replicated layout a 32x128b.warpx4 copy would produce),
//                 which is where the block-scaled MMA reads its scales.
//   warps 6..21   epilogue: four warps per TMEM lane quarter, 64 accumulator
//                 columns each; tcgen05.ld, release the accumulator to the
//                 MMA warp, scale by alpha, round, store.  Outputs whose rows
//                 are 16-byte aligned go through a 2 KB 64B-swizzled staging
//                 buffer per warp and TMA stores of 32-row boxes (32 bf16 or
//                 16 FP32 columns; a warp's direct stores would touch 32 rows
//                 per instruction); other outputs, and rows past the end of an
//                 expert, are stored directly.
//   TMEM: accumulator columns 0..255; per stage 16 columns of A scales and
//   32 columns of B scales from column 256.
//   Moving the scales with tcgen05.st from dedicated warps keeps them off
//   the MMA issue thread: measured on B300, a tcgen05.cp per 512-byte atom
//   cost as much tensor time as half an MMA.
// CTA pairs (the default; cta_group::2, clusters of two CTAs on two SMs):
//   tiles of 256 x 256; each CTA holds its 128 A rows and 128 of the 256 B
//   rows of a stage (38 KB instead of 54 KB per stage: five stages beside the
//   32 KB output staging for dense GEMMs, four for grouped ones, whose group
//   tables take the rest), plus its A scales and all 256 rows of B scales in
//   its own TMEM.
//   Rank 0 issues 256 x 256 x 64 MMAs for both; both CTAs' TMA loads complete
//   on rank 0's full barrier, both CTAs' scale warps and epilogues arrive on
//   rank 0's barriers, and rank 0's commits arrive on the barriers of both.
//   The second m-tile of a pair may lie past its group's end: it is computed
//   and not stored.
// Groups along K (KGROUP, a compile-time variant; the wgrad of the expert
// GEMMs): every group has all m-tiles of the shared M rows x all n-tiles; a
// tile's K slice is the group's 64-padded token segment (TMA boxes at its
// byte column, scale atoms at its atom column, a partial last stage issuing
// fewer MMAs), its C rows start at g * M, and a group without tokens issues
// no MMA and stores zeros.
// Every wait is bounded (DEV_TIMEOUT in the status word, then a clean exit).
#pragma once

#include <cuda.h>
#include "common.cuh"
#include "quant.cuh"   // GroupTables / build_group_tables / find_group

namespace nvfp4 {

constexpr int G_BM = 128, G_BN = 256, G_BK = 256;
constexpr int G_A_BYTES = G_BM * G_BK / 2;                 // 16384
constexpr int G_B_BYTES = G_BN * G_BK / 2;                 // 32768
constexpr int G_SFA_BYTES = (G_BK / 64) * 512;             // 2048: 4 atoms of A scales
constexpr int G_SFB_BYTES = 2 * (G_BK / 64) * 512;         // 4096: 2 row blocks x 4 atoms of B scales
constexpr int G_STAGE_BYTES = G_A_BYTES + G_B_BYTES + G_SFA_BYTES + G_SFB_BYTES;  // 55296
// CTA-pair kernel (cta_group::2, 256 x 256 tiles over two SMs): each CTA holds
// its own 128 A rows and half of the 256 B rows of a stage, and all 256 rows
// of B scales.
constexpr int G2_B_BYTES = G_B_BYTES / 2;                                          // 16384
constexpr int G2_STAGE_BYTES = G_A_BYTES + G2_B_BYTES + G_SFA_BYTES + G_SFB_BYTES;  // 38912
constexpr int G_W_TMA = 0, G_W_MMA = 1, G_W_SF0 = 2, G_W_EPI0 = 6;
constexpr int G_EPI_WARPS = 16;
constexpr int G_W_SFP = G_W_EPI0 + G_EPI_WARPS;             // 22: scale-atom producer
constexpr int G_THREADS = (G_W_SFP + 1) * 32;               // 736
constexpr int G_TMEM_COLS = 512;
constexpr int G_SF_COL0 = 256;
constexpr int G_SF_COLS_PER_STAGE = 48;
constexpr int G_BAND = 16;                                   // m-tiles per raster band (grouped schedules)
constexpr int G_BAND_DENSE = 32;                             // ... and for one dense GEMM
constexpr uint64_t G_WAIT_NS = 4000000000ull;                // bounded waits: 4 s
constexpr int G_BAR_BYTES = 256;                             // barriers, TMEM slot, abort flag

constexpr int G_STORE_WARP_BYTES = 2048;   // staging of one epilogue warp: 32 rows x 64 bytes (32 bf16 or 16 FP32)

// Tile schedules (a compile-time parameter of the kernel): one dense GEMM,
// groups along M (the routed-expert GEMM: per-expert rows and weights), or
// groups along K (the expert wgrad: per-expert token segments).
constexpr int G_DENSE = 0, G_MGROUP = 1, G_KGROUP = 2;

// Shared-memory layout of one CTA (after 1 KB alignment): the stage ring,
// the output staging of the TMA-store epilogue, barriers, group tables.
// A CTA pair keeps five stages with the 32 KB staging when its group tables
// are small (dense GEMMs); the 512-expert tables of a grouped GEMM leave room
// for four.  A single CTA's 54 KB stages leave room for three beside the
// staging, four without it.
template <bool TMA_STORE, bool PAIR = false, bool DENSE = false>
struct GemmLayout {
    static constexpr int STAGE_BYTES = PAIR ? G2_STAGE_BYTES : G_STAGE_BYTES;
    static constexpr int B_BYTES = PAIR ? G2_B_BYTES : G_B_BYTES;
    static constexpr int STAGES = PAIR ? ((TMA_STORE && !DENSE) ? 4 : 5) : (TMA_STORE ? 3 : 4);
    static constexpr int STORE_OFF = STAGES * STAGE_BYTES;
    static constexpr int STORE_BYTES = TMA_STORE ? G_EPI_WARPS * G_STORE_WARP_BYTES : 0;
    static constexpr int BAR_OFF = STORE_OFF + STORE_BYTES;
    static constexpr int TAB_OFF = BAR_OFF + G_BAR_BYTES;
};

// dynamic shared memory: 1 KB alignment slack, layout, group tables (row
// offsets, 128-row padded offsets and, for CTA pairs, 256-row padded offsets)
__host__ __device__ constexpr int gemm_smem_bytes(bool tma_store, int groups, bool pair, bool dense) {
    return 1024 +
           (pair ? (tma_store ? (dense ? GemmLayout<true, true, true>::TAB_OFF : GemmLayout<true, true>::TAB_OFF)
                              : GemmLayout<false, true>::TAB_OFF)
                 : (tma_store ? GemmLayout<true>::TAB_OFF : GemmLayout<false>::TAB_OFF)) +
           (pair ? 3 : 2) * 4 * (groups + 1);
}
static_assert(gemm_smem_bytes(true, 1, true, true) <= 227 * 1024, "dense pair layout exceeds shared memory");
static_assert(gemm_smem_bytes(true, 512, true, false) <= 227 * 1024, "grouped pair layout exceeds shared memory");
static_assert(gemm_smem_bytes(true, 512, false, false) <= 227 * 1024, "grouped layout exceeds shared memory");

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
    float* c_amax;              // nullable: max |C| over the written outputs, per group (zeroed by the host)
    bool vec_store;             // rows of C start 16-byte aligned: vector stores
    // K % 32 == 16: code rows of K/2 bytes are not a 16-byte multiple, which
    // a tensor map's row stride must be; the producer warp then copies the
    // stage's rows itself (single-CTA kernel only)
    bool copy_ab;
    const uint8_t* a_codes;     // copy_ab: A codes [a_rows, K/2]
    const uint8_t* b_codes;     // copy_ab: B codes [b_rows, K/2]
    int64_t a_rows, b_rows;
};

// A stage's 128-byte K window of `nrows` operand rows from row0, copied by
// the 32 lanes of a warp into the layout a 128B-swizzled TMA box gives
// (16-byte chunk c of row r at chunk c ^ (r & 7) of the row's 128 bytes),
// 8 bytes at a time (rows are 8-byte aligned when K % 16 == 0); bytes past
// the row's end or rows past `rows` are zero, as a TMA load fills them.
__device__ __forceinline__ void copy_stage_rows(uint8_t* dst, const uint8_t* __restrict__ src, int64_t rows,
                                                int64_t row_bytes, int64_t row0, int nrows, int64_t kx) {
    const int lane = threadIdx.x & 31;
    for (int it = lane; it < nrows * 16; it += 32) {
        const int r = it >> 4, h = it & 15;
        const int64_t gr = row0 + r, gb = kx + 8 * h;
        uint2 v = make_uint2(0u, 0u);
        if (gr < rows && gb + 8 <= row_bytes) v = __ldg(reinterpret_cast<const uint2*>(src + gr * row_bytes + gb));
        *reinterpret_cast<uint2*>(dst + r * 128 + (((h >> 1) ^ (r & 7)) << 4) + 8 * (h & 1)) = v;
    }
}

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
// DEV_TIMEOUT.  (Barriers that the other CTA of a pair signals are waited on
// the same way: what they announce is TMA data or TMEM traffic, not memory
// written by the signalling thread.)
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

// TMA store of a box from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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


template <bool PAIR>
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
    if (PAIR)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
            : "memory");
    else
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

#define NVFP4_R16(i) "=r"(v[i]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3])
__device__ __forceinline__ void tc_ld_32x32b_x16(uint32_t taddr, uint32_t* v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15}, [%16];"
        : NVFP4_R16(0), NVFP4_R16(4), NVFP4_R16(8), NVFP4_R16(12)
        : "r"(taddr));
}
#undef NVFP4_R16

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }


#define NVFP4_MMA4_ASM(CG)                                                                                   \
    asm volatile(                                                                                            \
        "{\n\t.reg .pred p, t;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"                                   \
        ".reg .b32 sa1, sa2, sa3, sb1, sb2, sb3;\n\t"                                                        \
        "setp.ne.b32 p, %4, 0;\n\t"                                                                          \
        "setp.eq.u32 t, 0, 0;\n\t"                                                                           \
        "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\t"                                \
        "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"                                \
        "add.u32 sa1, %5, 4;\n\tadd.u32 sa2, %5, 8;\n\tadd.u32 sa3, %5, 12;\n\t"                            \
        "add.u32 sb1, %6, 8;\n\tadd.u32 sb2, %6, 16;\n\tadd.u32 sb3, %6, 24;\n\t"                           \
        "tcgen05.mma.cta_group::" #CG ".kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t" \
        "tcgen05.mma.cta_group::" #CG ".kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a1, b1, %3, [sa1], [sb1], t;\n\t" \
        "tcgen05.mma.cta_group::" #CG ".kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a2, b2, %3, [sa2], [sb2], t;\n\t" \
        "tcgen05.mma.cta_group::" #CG ".kind::mxf4nvf4.block_scale.scale_vec::4X [%0], a3, b3, %3, [sa3], [sb3], t;\n\t}" \
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)                          \
        : "memory")

// Four K=64 MMAs covering one 256-wide K stage.  The shared-memory
// descriptors advance by 32 bytes (2 in descriptor units) per MMA inside the
// 128-byte swizzle atom; scale columns advance by 4 (A) and 8 (B).  Only the
// first MMA may start a fresh accumulator.  PAIR: cta_group::2, issued by the
// first CTA of a pair for both (A rows and B rows split between the two
// CTAs' shared memory at the same offsets, each CTA's TMEM holding its rows).
template <bool PAIR>
__device__ __forceinline__ void tc_mma4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                        uint32_t sfb, uint32_t accumulate) {
    if (PAIR) NVFP4_MMA4_ASM(2);
    else NVFP4_MMA4_ASM(1);
}
#undef NVFP4_MMA4_ASM

// One whole K stage from one asm block: the four MMAs of tc_mma4, then the
// commit of the stage to its empty barrier (in both CTAs of a pair), and,
// between the first and the second MMA, a non-blocking test of the next
// stage's two barriers (full and sf_full, parity ph_next).  Returns 1 when
// both had completed.  The tensor pipe accepts an MMA only shortly before it
// can start it, so the issuing thread spends most of a stage blocked in MMA
// issue; testing the next stage's barriers there hides their latency, which
// would otherwise be idle tensor time between stages.
#define NVFP4_MMA4_PEEK_ASM(CG, COMMIT)                                                                      \
    asm volatile(                                                                                            \
        "{\n\t.reg .pred p, t, f1, f2;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"                             \
        ".reg .b32 sa1, sa2, sa3, sb1, sb2, sb3;\n\t"                                                        \
        "setp.ne.b32 p, %5, 0;\n\t"                                                                          \
        "setp.eq.u32 t, 0, 0;\n\t"                                                                           \
        "add.s64 a1, %2, 2;\n\tadd.s64 a2, %2, 4;\n\tadd.s64 a3, %2, 6;\n\t"                                \
        "add.s64 b1, %3, 2;\n\tadd.s64 b2, %3, 4;\n\tadd.s64 b3, %3, 6;\n\t"                                \
        "add.u32 sa1, %6, 4;\n\tadd.u32 sa2, %6, 8;\n\tadd.u32 sa3, %6, 12;\n\t"                            \
        "add.u32 sb1, %7, 8;\n\tadd.u32 sb2, %7, 16;\n\tadd.u32 sb3, %7, 24;\n\t"                           \
        "tcgen05.mma.cta_group::" #CG ".kind::mxf4nvf4.block_scale.scale_vec::4X [%1], %2, %3, %4, [%6], [%7], p;\n\t" \
        "mbarrier.test_wait.parity.shared::cta.b64 f1, [%9], %11;\n\t"                                        \
        "mbarrier.test_wait.parity.shared::cta.b64 f2, [%10], %11;\n\t"                                       \
        "tcgen05.mma.cta_group::" #CG ".kind::mxf4nvf4.block_scale.scale_vec::4X [%1], a1, b1, %4, [sa1], [sb1], t;\n\t" \
        "tcgen05.mma.cta_group::" #CG ".kind::mxf4nvf4.block_scale.scale_vec::4X [%1], a2, b2, %4, [sa2], [sb2], t;\n\t" \
        "tcgen05.mma.cta_group::" #CG ".kind::mxf4nvf4.block_scale.scale_vec::4X [%1], a3, b3, %4, [sa3], [sb3], t;\n\t" \
        COMMIT                                                                                               \
        "and.pred f1, f1, f2;\n\t"                                                                           \
        "selp.u32 %0, 1, 0, f1;\n\t}"                                                                        \
        : "=r"(ready)                                                                                        \
        : "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb), "r"(empty_bar),             \
          "r"(full_next), "r"(sff_next), "r"(ph_next)                                                        \
        : "memory")

template <bool PAIR>
__device__ __forceinline__ uint32_t tc_mma4_commit_peek(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                                        uint32_t sfa, uint32_t sfb, uint32_t accumulate,
                                                        uint32_t empty_bar, uint32_t full_next, uint32_t sff_next,
                                                        uint32_t ph_next) {
    uint32_t ready;
    if (PAIR)
        NVFP4_MMA4_PEEK_ASM(2, "{\n\t.reg .b16 msk;\n\tmov.b16 msk, 3;\n\t"
                               "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%8], msk;\n\t}\n\t");
    else
        NVFP4_MMA4_PEEK_ASM(1, "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%8];\n\t");
    return ready;
}
#undef NVFP4_MMA4_PEEK_ASM

// ------------------------------------------------------------------ CTA pairs
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address in the shared::cluster window of the variable at shared::cta
// address `addr` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrivals on the other CTA's barriers are relaxed: what they announce is
// either TMEM traffic already completed by tcgen05.wait::st / wait::ld (and
// ordered by tcgen05.fence::before_thread_sync) or bytes that the TMA itself
// reports, so no release of this thread's memory writes is needed.  Measured
// on B300, cluster-scope release arrivals made the pair kernel twice as slow
// as the single-CTA one (3.45 ms against 1.81 ms for the Ultra fprop GEMM).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx_cluster(uint32_t cluster_addr, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_addr),
                 "r"(bytes)
                 : "memory");
}

// TMA load into this CTA's shared memory that signals an mbarrier of either
// CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                 uint32_t cluster_bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(cluster_bar)
        : "memory");
}

// Arrive once on the mbarrier at shared::cta offset `bar` in every CTA of
// the pair when the pair MMAs issued so far have completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t mask) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
                 ::"r"(bar), "h"(mask)
                 : "memory");
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// tcgen05.st of 16 / 32 consecutive 32-bit columns into this warp's 32 TMEM lanes.
__device__ __forceinline__ void tc_st_x16(uint32_t taddr, const uint4 (&v)[4]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};" ::"r"(taddr),
        "r"(v[0].x), "r"(v[0].y), "r"(v[0].z), "r"(v[0].w), "r"(v[1].x), "r"(v[1].y), "r"(v[1].z), "r"(v[1].w),
        "r"(v[2].x), "r"(v[2].y), "r"(v[2].z), "r"(v[2].w), "r"(v[3].x), "r"(v[3].y), "r"(v[3].z), "r"(v[3].w)
        : "memory");
}

__device__ __forceinline__ void tc_st_x32(uint32_t taddr, const uint4 (&v)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0].x), "r"(v[0].y), "r"(v[0].z), "r"(v[0].w), "r"(v[1].x), "r"(v[1].y), "r"(v[1].z), "r"(v[1].w),
        "r"(v[2].x), "r"(v[2].y), "r"(v[2].z), "r"(v[2].w), "r"(v[3].x), "r"(v[3].y), "r"(v[3].z), "r"(v[3].w),
        "r"(v[4].x), "r"(v[4].y), "r"(v[4].z), "r"(v[4].w), "r"(v[5].x), "r"(v[5].y), "r"(v[5].z), "r"(v[5].w),
        "r"(v[6].x), "r"(v[6].y), "r"(v[6].z), "r"(v[6].w), "r"(v[7].x), "r"(v[7].y), "r"(v[7].z), "r"(v[7].w)
        : "memory");
}

__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Largest |x| over the first `valid` bf16 values packed two per word in w[0..N)
// (element 2j in the low half of word j), as the 15 magnitude bits.
template <int N>
__device__ __forceinline__ uint32_t bf16_absmax(const uint32_t (&w)[N], int valid) {
    uint32_t acc = 0;
    if (valid >= 2 * N) {
#pragma unroll
        for (int j = 0; j < N; ++j) acc = __vmaxu2(acc, w[j] & 0x7FFF7FFFu);
    } else {
#pragma unroll
        for (int j = 0; j < N; ++j) {
            if (2 * j < valid) acc = max(acc, w[j] & 0x7FFFu);
            if (2 * j + 1 < valid) acc = max(acc, (w[j] >> 16) & 0x7FFFu);
        }
    }
    return max(acc & 0xFFFFu, acc >> 16);
}

// Merge a warp's largest output magnitude (non-negative FP32 bits) into *dst.
__device__ __forceinline__ void warp_amax_to(float* dst, uint32_t fbits) {
    fbits = __reduce_max_sync(0xFFFFFFFFu, fbits);
    if ((threadIdx.x & 31) == 0 && fbits != 0u) atomicMax(reinterpret_cast<unsigned int*>(dst), fbits);
}

// Lane/chunk exchange for coalesced row stores.  On entry lane l holds 32
// words of row l of a 32-row block (chunk c = words 4c .. 4c+3, 16 bytes).
// Three xor-shuffle stages swap lane bits 2..4 with chunk bits 0..2; on exit
// chunk x of lane L holds chunk (L >> 2) of row 4x + (L & 3), so the warp's
// 16-byte store of chunk x writes four whole 128-byte row segments instead of
// 16 bytes in each of 32 rows (8x fewer L1 wavefronts).
__device__ __forceinline__ void rows_to_segments(uint32_t (&w)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const int m = 1 << i;
        const bool up = (lane >> (2 + i)) & 1;
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            if (x & m) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t send = up ? w[4 * x + j] : w[4 * (x | m) + j];
                const uint32_t recv = __shfl_xor_sync(0xFFFFFFFFu, send, 4 << i);
                if (up) w[4 * x + j] = recv;
                else w[4 * (x | m) + j] = recv;
            }
        }
    }
}

// Store a 32-row x 16-chunk block after rows_to_segments: chunk x of lane L
// goes to row row_base + 4x + (L & 3), byte offset 16 * (L >> 2) past
// col_ptr_base (rows ldc_bytes apart).  Rows at or beyond rows_valid and
// bytes at or beyond bytes_valid (of the 128-byte segment) are skipped.
__device__ __forceinline__ void store_segments(const uint32_t (&w)[32], uint8_t* base, int64_t ldc_bytes,
                                               int rows_valid, int bytes_valid) {
    const int lane = threadIdx.x & 31;
    const int cb = 16 * (lane >> 2);
#pragma unroll
    for (int x = 0; x < 8; ++x) {
        const int rr = 4 * x + (lane & 3);
        if (rr >= rows_valid) continue;
        uint8_t* dst = base + (int64_t)rr * ldc_bytes + cb;
        if (cb + 16 <= bytes_valid) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
        } else if (cb < bytes_valid) {
#pragma unroll
            for (int b = 0; b < 8; ++b)
                if (cb + 2 * b < bytes_valid)
                    *reinterpret_cast<uint16_t*>(dst + 2 * b) = (uint16_t)(w[4 * x + b / 2] >> (16 * (b & 1)));
        }
    }
}

// ------------------------------------------------------------------ tiles
struct TileCoord {
    int g;            // group
    int mtg;          // global m-tile index (scale atom row of A)
    int nt;           // n-tile
    int32_t row0;     // first A row of the tile
    int32_t rows;     // valid rows (<= 128)
    int32_t k0 = 0;   // first K element of the tile (groups along K; C rows then start at g * M + row0)
    int32_t ka = -1;  // 64-wide K atoms of the tile; -1: all of K
};

// Tiles are numbered in bands of BAND m-tiles: inside a band, the m-tile
// runs fastest, so concurrently resident CTAs share B tiles through L2 and
// every B tile is read from DRAM about once per band.  Measured on the Ultra
// in_proj GEMMs: bands of 32 m-tiles (4096 rows) took fprop 1.585 -> 1.549 ms
// against 16 and left dgrad and wgrad unchanged (64 slowed them by 6 %); the
// grouped down-projection keeps 16 (32 was 0.7 % slower).
template <int BAND>
__device__ __forceinline__ TileCoord decode_tile(int64_t t, int mtiles, int ntiles, const int32_t* off,
                                                 const int32_t* pad, int groups) {
    const int64_t band_tiles = (int64_t)BAND * ntiles;
    const int band = (int)(t / band_tiles);
    const int64_t local = t - (int64_t)band * band_tiles;
    const int bsize = min(BAND, mtiles - band * BAND);
    TileCoord c;
    c.mtg = band * BAND + (int)(local % bsize);
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

// Tiles of a CTA pair: 256 rows (two 128-row m-tiles of one group, the
// second possibly past the group's end) x 256 columns, numbered in bands of
// BAND / 2 row pairs like decode_tile.  Returns the m-tile of CTA `rank`.
// A second m-tile past the group's end has rows = 0 and takes its partner's
// scale row (mtg), so that its loads stay inside the scale buffer; its
// results are never stored.
template <int BAND>
__device__ __forceinline__ TileCoord decode_pair_tile(int64_t t, int ptiles, int ntiles, const int32_t* off,
                                                      const int32_t* pad, const int32_t* pair, int groups,
                                                      uint32_t rank) {
    constexpr int PB = BAND / 2;
    const int64_t band_tiles = (int64_t)PB * ntiles;
    const int band = (int)(t / band_tiles);
    const int64_t local = t - (int64_t)band * band_tiles;
    const int bsize = min(PB, ptiles - band * PB);
    const int pt = band * PB + (int)(local % bsize);
    TileCoord c;
    c.nt = (int)(local / bsize);
    int lo = 0, hi = groups;
    const int32_t key = pt * 256;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pair[mid] <= key) lo = mid; else hi = mid;
    }
    c.g = lo;
    const int32_t lm = 2 * (pt - pair[lo] / 256) + (int32_t)rank;     // m-tile inside the group
    c.row0 = off[lo] + lm * 128;
    c.rows = max(0, min(128, off[lo + 1] - c.row0));
    c.mtg = pad[lo] / 128 + (c.rows > 0 ? lm : lm - 1);
    return c;
}

// Tiles of a GEMM whose groups split K: for every group, the m-tiles (or
// row pairs) of the shared M rows x the n-tiles, the m-tile fastest.  Group
// g's K slice starts at kpad[g] and spans (kpad[g+1] - kpad[g]) / 64 atoms
// (possibly none: C_g is then zero); its C rows start at g * M + row0.
__device__ __forceinline__ TileCoord decode_kgroup_tile(int64_t t, int mt, int ntiles, const int32_t* kpad,
                                                        int64_t M, int64_t K, bool pair, uint32_t rank) {
    const int64_t per_g = (int64_t)mt * ntiles;
    TileCoord c;
    c.g = (int)(t / per_g);
    const int64_t local = t - (int64_t)c.g * per_g;
    const int m = (int)(local % mt);
    c.nt = (int)(local / mt);
    const int lm = pair ? 2 * m + (int)rank : m;
    c.row0 = lm * 128;
    c.rows = (int32_t)max((int64_t)0, min((int64_t)128, M - (int64_t)c.row0));
    c.mtg = c.rows > 0 ? lm : lm - 1;                  // a pair's ghost m-tile borrows its partner's scales
    // K slices never reach past K (offsets are device data)
    const int32_t k1 = (int32_t)min((int64_t)kpad[c.g + 1], K);
    c.k0 = (int32_t)min((int64_t)kpad[c.g], K);
    c.ka = max(0, k1 - c.k0) / 64;
    return c;
}

__device__ __forceinline__ uint4 ldg_u4(const uint8_t* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

// ------------------------------------------------------------------ kernel
// OUT_FP32: FP32 output, otherwise bf16.  TMA_STORE: the output leaves
// through tm_c (rows 16-byte aligned) in boxes of 32 rows x 64 bytes staged
// in shared memory; otherwise it is stored directly.  SCHED: G_DENSE,
// G_MGROUP or G_KGROUP.
template <bool OUT_FP32, bool TMA_STORE, bool PAIR, int SCHED = G_DENSE>
__global__ void __launch_bounds__(G_THREADS, 1)
    k_gemm_nvfp4(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                 const __grid_constant__ CUtensorMap tm_c, const GemmParams p) {
    constexpr bool KGROUP = SCHED == G_KGROUP;
    using L = GemmLayout<TMA_STORE, PAIR, SCHED == G_DENSE>;
    constexpr int G_STAGES = L::STAGES;
    constexpr int STAGE_BYTES = L::STAGE_BYTES;
    static_assert(G_SF_COL0 + G_STAGES * G_SF_COLS_PER_STAGE <= G_TMEM_COLS, "scale columns exceed TMEM");
    static_assert((4 * G_STAGES + 3) * 8 + 8 <= G_BAR_BYTES, "barriers exceed their space");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
    // bars: full[S] (A, B landed), empty[S], sf_full[S] (scales in TMEM),
    // sf_land[S] (scales landed in shared memory), acc_full, acc_empty, drain
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4 * G_STAGES + 3);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int32_t* tab = reinterpret_cast<int32_t*>(smem + L::TAB_OFF);
    const int groups = p.groups;
    // groups along K: pad[] holds the 64-padded token segments (no pair table)
    GroupTables gt{tab, tab + groups + 1, (PAIR && !KGROUP) ? tab + 2 * (groups + 1) : nullptr};
    // CTA pairs: rank 0 issues the MMAs of both; barriers that collect both
    // CTAs' arrivals (full, sf_full, acc_empty) are rank 0's.
    const uint32_t rank = PAIR ? cluster_rank() : 0u;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + G_STAGES), sff0 = smem_u32(bars + 2 * G_STAGES);
    const uint32_t sfl0 = smem_u32(bars + 3 * G_STAGES);
    const uint32_t acc_full = smem_u32(bars + 4 * G_STAGES), acc_empty = acc_full + 8, drain = acc_full + 16;

    if (threadIdx.x == 0) {
        for (int s = 0; s < G_STAGES; ++s) {
            mbar_init(full0 + 8 * s, PAIR ? 2 : 1);
            mbar_init(empty0 + 8 * s, 1);
            mbar_init(sff0 + 8 * s, PAIR ? 8 : 4);
            mbar_init(sfl0 + 8 * s, 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, PAIR ? 2 * G_EPI_WARPS : G_EPI_WARPS);
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == G_W_TMA && lane == 0 && !p.copy_ab) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_a)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_b)) : "memory");
        if (TMA_STORE) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_c)) : "memory");
    }
    if (warp == G_W_MMA) {
        if (PAIR) {
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                         "r"(G_TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                         "r"(G_TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    if (KGROUP) {
        build_group_tables(p.offsets, groups, p.K, gt, 6);
    } else if (p.offsets != nullptr) {
        build_group_tables(p.offsets, groups, p.M, gt);
    } else if (threadIdx.x == 0) {
        gt.off[0] = 0;
        gt.off[1] = (int32_t)p.M;
        gt.pad[0] = 0;
        gt.pad[1] = (int32_t)(((p.M + 127) >> 7) << 7);
        if (PAIR) { gt.pair[0] = 0; gt.pair[1] = (int32_t)(((p.M + 255) >> 8) << 8); }
    }
    tc_fence_before();
    if (PAIR) cluster_sync();   // both CTAs' barriers initialised before any arrival from the other
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int ntiles = (int)((p.N + G_BN - 1) / G_BN);
    // groups along M: tiles from the padded row tables; groups along K: every
    // group has all m-tiles (or row pairs) of the shared M rows
    const int kg_mt = (int)(PAIR ? (p.M + 255) / 256 : (p.M + 127) / 128);
    const int mtiles = KGROUP ? 0 : gt.pad[groups] >> 7;
    const int ptiles = (PAIR && !KGROUP) ? (gt.pair[groups] >> 8) : 0;
    const int64_t total = KGROUP ? (int64_t)groups * kg_mt * ntiles : (int64_t)(PAIR ? ptiles : mtiles) * ntiles;
    // a pair walks the tiles of its cluster (blockIdx.x / 2), both CTAs alike
    const int64_t t_first = PAIR ? (int64_t)(blockIdx.x >> 1) : (int64_t)blockIdx.x;
    const int64_t t_step = PAIR ? (int64_t)(gridDim.x >> 1) : (int64_t)gridDim.x;
    auto tile_at = [&](int64_t t) {
        if (KGROUP) return decode_kgroup_tile(t, kg_mt, ntiles, gt.pad, p.M, p.K, PAIR, rank);
        constexpr int BAND = SCHED == G_DENSE ? G_BAND_DENSE : G_BAND;
        return PAIR ? decode_pair_tile<BAND>(t, ptiles, ntiles, gt.off, gt.pad, gt.pair, groups, rank)
                    : decode_tile<BAND>(t, mtiles, ntiles, gt.off, gt.pad, groups);
    };
    const int katoms = (int)((p.K + 63) / 64);           // atoms of a whole operand row (scale row stride)
    // K atoms and stages of a tile
    auto tile_atoms = [&](const TileCoord& tc) { return KGROUP ? tc.ka : katoms; };
    const int nrb = (int)((p.N + 127) / 128);            // 128-row scale blocks of one B operand
    const int64_t b_rows_per_group = (p.offsets != nullptr && !KGROUP) ? p.N : 0;

    if (warp == G_W_TMA && !PAIR && p.copy_ab) {
        // ------------------------------------------------ copy producer (A, B; K % 32 == 16)
        int s = 0;
        uint32_t ph = 0;
        for (int64_t t = t_first; t < total; t += t_step) {
            const TileCoord tc = tile_at(t);
            const int64_t brow0 = tc.g * b_rows_per_group + (int64_t)tc.nt * G_BN;
            const int ka = tile_atoms(tc), kst = (ka + 3) / 4;
            bool ok = true;
            for (int ks = 0; ks < kst; ++ks) {
                bool free_ = true;
                if (lane == 0) free_ = mbar_wait(empty0 + 8 * s, ph ^ 1u, abort_flag);
                if (!__shfl_sync(0xFFFFFFFFu, free_, 0)) { ok = false; break; }
                uint8_t* st = stages + s * STAGE_BYTES;
                const int64_t kx = tc.k0 / 2 + ks * 128;
                copy_stage_rows(st, p.a_codes, p.a_rows, p.K / 2, tc.row0, G_BM, kx);
                copy_stage_rows(st + G_A_BYTES, p.b_codes, p.b_rows, p.K / 2, brow0, G_BN, kx);
                fence_proxy_async_smem();         // generic writes, read by the tensor cores
                __syncwarp();
                if (lane == 0) mbar_arrive(full0 + 8 * s);
                if (++s == G_STAGES) { s = 0; ph ^= 1u; }
            }
            if (!ok) break;
        }
    } else if (warp == G_W_TMA) {
        // ------------------------------------------------ TMA producer (A, B)
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0, issued = 0, issued_ph = 0;   // per-stage bits: ever issued, parity of last issue
            bool ok = true;
            for (int64_t t = t_first; t < total && ok; t += t_step) {
                const TileCoord tc = tile_at(t);
                // PAIR: this CTA loads B rows 128 * rank .. + 127 of the 256-row tile
                const int32_t brow0 =
                    (int32_t)(tc.g * b_rows_per_group + (int64_t)tc.nt * G_BN + (PAIR ? 128 * (int64_t)rank : 0));
                const int ka = tile_atoms(tc), kst = (ka + 3) / 4;
                for (int ks = 0; ks < kst; ++ks) {
                    if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, abort_flag)) { ok = false; break; }
                    const uint32_t st = smem_u32(stages + s * STAGE_BYTES);
                    const int32_t kx = tc.k0 / 2 + ks * 128;     // byte column of the K stage
                    if (PAIR) {
                        // A and B of both CTAs complete on rank 0's full barrier
                        const uint32_t bar = mapa_shared(full0 + 8 * s, 0);
                        mbar_expect_tx_cluster(bar, G_A_BYTES + L::B_BYTES);
                        tma_load_2d_pair(st, &tm_a, kx, tc.row0, bar);
                        tma_load_2d_pair(st + G_A_BYTES, &tm_b, kx, brow0, bar);
                    } else {
                        const uint32_t bar = full0 + 8 * s;
                        mbar_expect_tx(bar, G_A_BYTES + G_B_BYTES);
                        tma_load_2d(st, &tm_a, kx, tc.row0, bar);
                        tma_load_2d(st + G_A_BYTES, &tm_b, kx, brow0, bar);
                    }
                    issued |= 1u << s;
                    issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
                    if (++s == G_STAGES) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                // let every copy already issued land before the CTA exits (the
                // other CTA of a pair cannot wait on rank 0's full barrier: it
                // gives its copies a fixed millisecond instead)
                volatile int never = 0;
                for (int i = 0; i < G_STAGES; ++i)
                    if (((issued >> i) & 1u) && rank == 0) mbar_wait(full0 + 8 * i, (issued_ph >> i) & 1u, &never);
                if (PAIR && rank != 0) {
                    const uint64_t t0 = globaltimer_ns();
                    while (globaltimer_ns() - t0 < 1000000ull) __nanosleep(1000);
                }
            }
        }
    } else if (warp == G_W_SFP) {
        // ------------------------------------------------ scale-atom producer
        // The stage's scale atoms (A: 4 atoms of its m-tile, B: 4 atoms of each
        // of the tile's two 128-row blocks) by cp.async.bulk on the stage's
        // landing barrier.  A thread of its own: copy issue takes tens of
        // nanoseconds per copy on this part, and the A/B producer's two tensor
        // copies per stage already take a good part of a stage.
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0, issued = 0, issued_ph = 0;
            bool ok = true;
            for (int64_t t = t_first; t < total && ok; t += t_step) {
                const TileCoord tc = tile_at(t);
                const uint8_t* sfb_g = p.sfb + (int64_t)tc.g * p.sfb_group_stride;
                const bool rb2 = (tc.nt * 2 + 1) < nrb;
                const int ka = tile_atoms(tc), kst = (ka + 3) / 4, kc0 = tc.k0 / 64;
                const uint8_t* sa = p.sfa + ((int64_t)tc.mtg * katoms + kc0) * 512;
                const uint8_t* sb = sfb_g + ((int64_t)(tc.nt * 2) * katoms + kc0) * 512;
                for (int ks = 0; ks < kst; ++ks) {
                    if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, abort_flag)) { ok = false; break; }
                    const int na = min(4, ka - 4 * ks);
                    const uint32_t sfbytes = (uint32_t)na * 512u;
                    const uint32_t ssf = smem_u32(stages + s * STAGE_BYTES) + G_A_BYTES + L::B_BYTES;
                    const uint32_t sbar = sfl0 + 8 * s;
                    mbar_expect_tx(sbar, sfbytes * (rb2 ? 3u : 2u));
                    bulk_load(ssf, sa + 2048 * ks, sfbytes, sbar);
                    bulk_load(ssf + G_SFA_BYTES, sb + 2048 * ks, sfbytes, sbar);
                    if (rb2) bulk_load(ssf + G_SFA_BYTES + 2048, sb + (int64_t)katoms * 512 + 2048 * ks, sfbytes, sbar);
                    issued |= 1u << s;
                    issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
                    if (++s == G_STAGES) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                volatile int never = 0;
                for (int i = 0; i < G_STAGES; ++i)
                    if ((issued >> i) & 1u) mbar_wait(sfl0 + 8 * i, (issued_ph >> i) & 1u, &never);
            }
        }
    } else if (warp == G_W_MMA) {
        // ------------------------------------------------ MMA issuer (rank 0 of a pair)
        // A stage may start when its full barrier (A and B landed, both CTAs'
        // in a pair) and its sf_full barrier (scales in TMEM) have completed.
        // The tensor pipe holds little work ahead of the issuing thread, so
        // every cycle this thread spends between stages is an idle tensor
        // cycle: a whole stage is one asm block that also tests the next
        // stage's barriers while the MMAs issue (`ready`), and the blocking
        // waits run only when that test found them incomplete.
        if (lane == 0 && rank == 0) {
            const uint32_t idesc = mxf4nvf4_idesc(PAIR ? 2 * G_BM : G_BM, G_BN);
            const uint64_t ad0 = smem_desc(smem_u32(stages), 16, 1024, 2);
            const uint64_t bd0 = smem_desc(smem_u32(stages) + G_A_BYTES, 16, 1024, 2);
            int s = 0;
            uint32_t ph = 0, it = 0, ready = 0;
            bool ok = true;
            for (int64_t t = t_first; t < total && ok; t += t_step, ++it) {
                if (!mbar_wait(acc_empty, (it & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                // a tile with no K (an expert without tokens) issues nothing: its
                // epilogue writes zeros
                const int ka = KGROUP ? tile_at(t).ka : katoms, kst = (ka + 3) / 4;
                for (int ks = 0; ks < kst; ++ks) {
                    if (!ready && (!mbar_wait(full0 + 8 * s, ph, abort_flag) || !mbar_wait(sff0 + 8 * s, ph, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int na = min(4, ka - 4 * ks);
                    // descriptor start addresses are in 16-byte units (bits 0-13)
                    const uint64_t soff = (uint64_t)((s * STAGE_BYTES) >> 4);
                    const uint64_t ad = ad0 + soff, bd = bd0 + soff;
                    const uint32_t sfa_t = tmem + G_SF_COL0 + s * G_SF_COLS_PER_STAGE;
                    const uint32_t sfb_t = sfa_t + 16;
                    const int sn = s + 1 == G_STAGES ? 0 : s + 1;
                    const uint32_t phn = s + 1 == G_STAGES ? ph ^ 1u : ph;
                    if (na == 4) {
                        ready = tc_mma4_commit_peek<PAIR>(tmem, ad, bd, idesc, sfa_t, sfb_t, ks != 0 ? 1u : 0u,
                                                          empty0 + 8 * s, full0 + 8 * sn, sff0 + 8 * sn, phn);
                    } else {
                        for (int j = 0; j < na; ++j)
                            tc_mma<PAIR>(tmem, ad + 2 * j, bd + 2 * j, idesc, sfa_t + 4 * j, sfb_t + 8 * j,
                                         (ks | j) != 0 ? 1u : 0u);
                        if (PAIR) tc_commit_pair(empty0 + 8 * s, 3);
                        else tc_commit(empty0 + 8 * s);
                        ready = 0;
                    }
                    s = sn;
                    ph = phn;
                }
                if (!ok) break;
                if (PAIR) tc_commit_pair(acc_full, 3);
                else tc_commit(acc_full);
            }
            // every MMA issued by this thread completes before teardown
            if (PAIR) tc_commit_pair(drain, 1);
            else tc_commit(drain);
            volatile int never = 0;
            mbar_wait(drain, 0, &never);
        }
    } else if (warp < G_W_EPI0) {
        // ------------------------------------------------ scale factors -> TMEM
        // The scale producer lands the stage's scale atoms in shared memory
        // next to A and B (on their own barrier).  Lane i of every quarter
        // copies the 16 bytes at offset 16*i of each 512-byte atom (the 4
        // scales of rows i, i+32, i+64, i+96) into the atom's 4 TMEM columns.
        // The stage's TMEM columns are free once its data has landed: the
        // producers refilled it only after the MMAs of its previous use
        // completed.  In a CTA pair each CTA writes its own A scales and all
        // 256 rows of B scales into its own TMEM.
        const uint32_t tq = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int64_t t = t_first; t < total && ok; t += t_step) {
            const TileCoord tc = tile_at(t);
            const bool rb2 = (tc.nt * 2 + 1) < nrb;
            const int ka = tile_atoms(tc), kst = (ka + 3) / 4;
            for (int ks = 0; ks < kst; ++ks) {
                const int na = min(4, ka - 4 * ks);
                if (!mbar_wait(sfl0 + 8 * s, ph, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint8_t* ssf = stages + s * STAGE_BYTES + G_A_BYTES + L::B_BYTES + lane * 16;
                uint4 va[4], vb[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool in = j < na;
                    va[j] = in ? *reinterpret_cast<const uint4*>(ssf + 512 * j) : make_uint4(0, 0, 0, 0);
                    vb[2 * j] = in ? *reinterpret_cast<const uint4*>(ssf + G_SFA_BYTES + 512 * j) : make_uint4(0, 0, 0, 0);
                    vb[2 * j + 1] = (in && rb2) ? *reinterpret_cast<const uint4*>(ssf + G_SFA_BYTES + 2048 + 512 * j)
                                                : make_uint4(0, 0, 0, 0);
                }
                const uint32_t col = (uint32_t)(G_SF_COL0 + s * G_SF_COLS_PER_STAGE);
                tc_st_x16(tq + col, va);
                tc_st_x32(tq + col + 16, vb);
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (PAIR) mbar_arrive_cluster(mapa_shared(sff0 + 8 * s, 0));
                    else mbar_arrive(sff0 + 8 * s);
                }
                if (++s == G_STAGES) { s = 0; ph ^= 1u; }
            }
        }
    } else {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;                          // TMEM lane quarter this warp may access
        const int chunk = (warp - G_W_EPI0) >> 2;        // 64-column chunk of the tile
        const int r = q * 32 + lane;                     // row inside the tile
        uint32_t it = 0;
        // PAIR: the accumulator of this CTA's 128 rows is released to rank 0
        const uint32_t acc_release = PAIR ? mapa_shared(acc_empty, 0) : acc_empty;
        // output amax: each lane keeps a running max over the tiles of one
        // group; the warp merges it into c_amax[group] when the group changes
        int amax_g = -1;
        uint32_t amax_run = 0;
        for (int64_t t = t_first; t < total; t += t_step, ++it) {
            const TileCoord tc = tile_at(t);
            if (p.c_amax != nullptr && tc.g != amax_g) {
                if (amax_g >= 0) warp_amax_to(p.c_amax + amax_g, amax_run);
                amax_g = tc.g;
                amax_run = 0;
            }
            const float alpha = __fmul_rn(tensor_decode_scale(p.amax_a[tc.g]), tensor_decode_scale(p.amax_b[tc.g]));
            if (!mbar_wait(acc_full, it & 1u, abort_flag)) break;
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(chunk * 64);
            // groups along K: C rows of group g start at g * M; a group without
            // K (an expert without tokens) stores zeros (vmask clears the
            // accumulator words, which no MMA wrote)
            const int32_t crow0 = KGROUP ? tc.g * (int32_t)p.M + tc.row0 : tc.row0;   // < 2^31 (host check)
            const uint32_t vmask = (KGROUP && tc.ka == 0) ? 0u : 0xFFFFFFFFu;
            const int64_t row = crow0 + r;
            const int64_t col0 = (int64_t)tc.nt * G_BN + chunk * 64;
            if (TMA_STORE) {
                // Boxes of 32 rows x 64 bytes (32 bf16 or 16 FP32 columns): load the
                // box's columns from TMEM, scale (and round), then store the box
                // through this warp's 64B-swizzled staging buffer.  The accumulator
                // is released after the last box's load.  A box whose 32 rows all
                // belong to the tile leaves by TMA store; other rows (an expert's
                // last rows in a grouped GEMM) are stored directly.
                constexpr int BOXES = OUT_FP32 ? 4 : 2, BOX_COLS = OUT_FP32 ? 16 : 32, ESZ = OUT_FP32 ? 4 : 2;
                const bool rows_full = (q * 32 + 31) < tc.rows;
                const uint32_t stage_buf = smem_u32(smem + L::STORE_OFF + (warp - G_W_EPI0) * G_STORE_WARP_BYTES);
#pragma unroll
                for (int b = 0; b < BOXES; ++b) {
                    uint32_t w[16];
                    if (OUT_FP32) {
                        tc_ld_32x32b_x16(taddr + 16 * b, w);
                        tc_wait_ld();
                        if (b == BOXES - 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) { if (PAIR) mbar_arrive_cluster(acc_release); else mbar_arrive(acc_empty); }
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(__fmul_rn(alpha, __uint_as_float(w[i] & vmask)));
                    } else {
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            uint32_t v[16];
                            tc_ld_32x32b_x16(taddr + 32 * b + 16 * k, v);
                            tc_wait_ld();
                            if (b == BOXES - 1 && k == 1) {
                                tc_fence_before();
                                __syncwarp();
                                if (lane == 0) { if (PAIR) mbar_arrive_cluster(acc_release); else mbar_arrive(acc_empty); }
                            }
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(alpha, __uint_as_float(v[2 * j] & vmask)),
                                                                                __fmul_rn(alpha, __uint_as_float(v[2 * j + 1] & vmask)));
                                w[8 * k + j] = *reinterpret_cast<const uint32_t*>(&b2);
                            }
                        }
                    }
                    const int64_t cstart = col0 + b * BOX_COLS;
                    if (cstart >= p.N) continue;
                    if (p.c_amax != nullptr) {
                        const int valid = r < tc.rows ? (int)(p.N - cstart >= BOX_COLS ? BOX_COLS : p.N - cstart) : 0;
                        if (OUT_FP32) {
                            uint32_t m = 0;
#pragma unroll
                            for (int i = 0; i < 16; ++i) m = max(m, i < valid ? (w[i] & 0x7FFFFFFFu) : 0u);
                            amax_run = max(amax_run, m);
                        } else {
                            amax_run = max(amax_run, bf16_absmax(w, valid) << 16);
                        }
                    }
                    if (rows_full) {
                        // the staging buffer is free once the previous box has been read
                        if (lane == 0) bulk_wait_read0();
                        __syncwarp();
                        // row `lane`, 16-byte chunk j at lane*64 + 16*(j ^ ((lane >> 1) & 3))
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t addr = stage_buf + lane * 64 + 16 * (j ^ ((lane >> 1) & 3));
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[4 * j]),
                                         "r"(w[4 * j + 1]), "r"(w[4 * j + 2]), "r"(w[4 * j + 3])
                                         : "memory");
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tm_c, stage_buf, (int32_t)cstart, (int32_t)(crow0 + q * 32));
                            bulk_commit();
                        }
                    } else if (r < tc.rows) {
                        uint8_t* out = reinterpret_cast<uint8_t*>(p.c) + (row * p.ldc + cstart) * ESZ;
                        if (cstart + BOX_COLS <= p.N) {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                reinterpret_cast<uint4*>(out)[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                        } else {
#pragma unroll
                            for (int i = 0; i < BOX_COLS; ++i) {
                                if (cstart + i >= p.N) continue;
                                if (OUT_FP32) reinterpret_cast<uint32_t*>(out)[i] = w[i];
                                else reinterpret_cast<uint16_t*>(out)[i] = (uint16_t)(w[i / 2] >> (16 * (i & 1)));
                            }
                        }
                    }
                }
            } else if (OUT_FP32) {
                // two 32-column halves: load, scale, store; release after the second load
                const bool live = r < tc.rows && col0 < p.N;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t v[32];
                    tc_ld_32x32b_x32(taddr + 32 * h, v);
                    tc_wait_ld();
                    if (h == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) { if (PAIR) mbar_arrive_cluster(acc_release); else mbar_arrive(acc_empty); }
                    }
                    const int64_t cstart = col0 + 32 * h;
                    if (cstart >= p.N) continue;
                    if (p.c_amax != nullptr) {
                        // rounding is monotone, so max |alpha x| = alpha max |x|
                        const int valid = r < tc.rows ? (int)(p.N - cstart >= 32 ? 32 : p.N - cstart) : 0;
                        float m = 0.0f;
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            m = fmaxf(m, i < valid ? fabsf(__uint_as_float(v[i] & vmask)) : 0.0f);
                        amax_run = max(amax_run, __float_as_uint(__fmul_rn(alpha, m)));
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__fmul_rn(alpha, __uint_as_float(v[i] & vmask)));
                    if (p.vec_store) {
                        // rows of this warp: crow0 + 32q .. ; 32 columns = 128 bytes per row
                        rows_to_segments(v);
                        store_segments(v, reinterpret_cast<uint8_t*>(reinterpret_cast<float*>(p.c) + (crow0 + q * 32) * p.ldc + cstart),
                                       p.ldc * 4, tc.rows - q * 32, (int)(p.N - cstart >= 32 ? 128 : (p.N - cstart) * 4));
                    } else if (live) {
                        float* out = reinterpret_cast<float*>(p.c) + row * p.ldc + cstart;
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (cstart + i < p.N) out[i] = __uint_as_float(v[i]);
                    }
                }
            } else {
                // 64 columns in four 16-column pieces: load, scale, round; release
                // after the last load; then whole 128-byte row segments per store
                uint32_t w[32];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t v[16];
                    tc_ld_32x32b_x16(taddr + 16 * h, v);
                    tc_wait_ld();
                    if (h == 3) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) { if (PAIR) mbar_arrive_cluster(acc_release); else mbar_arrive(acc_empty); }
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(alpha, __uint_as_float(v[2 * j] & vmask)),
                                                                        __fmul_rn(alpha, __uint_as_float(v[2 * j + 1] & vmask)));
                        w[8 * h + j] = *reinterpret_cast<const uint32_t*>(&b2);
                    }
                }
                if (col0 >= p.N) continue;
                if (p.c_amax != nullptr) {
                    const int valid = r < tc.rows ? (int)(p.N - col0 >= 64 ? 64 : p.N - col0) : 0;
                    amax_run = max(amax_run, bf16_absmax(w, valid) << 16);
                }
                if (p.vec_store) {
                    rows_to_segments(w);
                    store_segments(w, reinterpret_cast<uint8_t*>(reinterpret_cast<uint16_t*>(p.c) + (crow0 + q * 32) * p.ldc + col0),
                                   p.ldc * 2, tc.rows - q * 32, (int)(p.N - col0 >= 64 ? 128 : (p.N - col0) * 2));
                } else if (r < tc.rows) {
                    uint16_t* out = reinterpret_cast<uint16_t*>(p.c) + row * p.ldc + col0;
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        if (col0 + i < p.N) out[i] = (uint16_t)(w[i / 2] >> (16 * (i & 1)));
                }
            }
        }
        if (amax_g >= 0) warp_amax_to(p.c_amax + amax_g, amax_run);
        // every TMA store of this warp has finished before the CTA exits
        if (TMA_STORE && lane == 0) bulk_wait0();
    }

    tc_fence_before();
    if (PAIR) cluster_sync();   // neither CTA leaves while the other may still signal or read it
    else __syncthreads();
    if (warp == G_W_MMA) {
        tc_fence_after();
        if (PAIR)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(G_TMEM_COLS) : "memory");
        else
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
