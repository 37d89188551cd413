// gemm.cu: split-pointer grouped GEMM for sm_103a (tcgen05 + TMEM + TMA).
//
// DWDP §4.2 (Eliminating Split-Weight Merge Overhead): the grouped GEMM of
// the MoE block reads local experts and prefetched remote experts from their
// own buffers instead of a contiguous merged copy.  Here each weight buffer is
// one 3-D TMA tensor map [slots][rows][K]; the per-group table (buffer, slot)
// picks the map and the slot coordinate, so no weight byte is ever moved to
// feed the GEMM.
//
// Kernel organisation (one persistent CTA per SM, 192 threads; NVFP4 224,
// or 352 with the eight-warp drain):
//   warp 0      TMA producer: A tile [128 rows x 128 B] + B tile [256 rows x
//               128 B] per stage, 4-stage mbarrier ring in shared memory
//               (128B swizzle); NVFP4 adds the tiles' block-scale chunks.
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32 accumulators;
//               NVFP4: one accumulator and a ring of block scales) and issues
//               tcgen05.mma (M=128, N=256, 32 bytes of K each) from one thread.
//   warps 2..5  epilogue: tcgen05.ld the accumulator rows of their TMEM lane
//               quarter, hand the accumulator back to warp 1 as soon as the
//               last loads land, apply SiLU(gate)*up or plain conversion,
//               store (NVFP4 option: warps 2..9, two per lane quarter, each
//               draining half of the tile's columns).
//   last warp   NVFP4 only: copies each stage's block scales from shared
//               memory into its TMEM columns (tcgen05.cp) and commits to a
//               per-stage barrier the MMA thread waits on.
// Tiles are enumerated group by group, n-tile by n-tile, m-tile fastest, and
// dealt to CTAs round-robin; CTAs 2c and 2c+1 form a cluster, and when their
// tiles are sibling m-tiles of one weight tile each loads half of it and
// multicasts it to both.  EPI_F32 (the router) may also split K into parts,
// each a tile with its own output plane.  Every wait is bounded (global
// timer); a wait that runs out sets a bit in the device error word and the
// CTA drains its copies and exits.
#include <cuda_bf16.h>

#include <algorithm>

#include "dwdp_internal.h"

namespace dwdp {
namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait

// Instruction descriptors.  kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.  kind::f8f6f4: the same with A and B E4M3
// (format 0).  kind::mxf4nvf4 (block-scaled, D always fp32): bits 4-5 and
// 29-30 select the byte of the B / A scale word (0: scale_vec::4X uses all
// four), A and B E2M1 (format 1), bit 23 = 0 for E4M3 scales, N and M as
// above.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);
constexpr uint32_t kIdescE4M3 = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
constexpr uint32_t kIdescNvfp4 = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

#ifndef DWDP_SF_WARP
#define DWDP_SF_WARP 1
#endif
// Per-format constants.  NVFP4 keeps one accumulator (256 TMEM columns) so
// that the other 256 columns can hold the block scales of the stages in
// flight: per stage 4 K steps x (4 columns of A scales + 8 of B scales).
template <int FMT>
struct Fmt {
    static constexpr int kKElems = FMT == FMT_NVFP4 ? 2 * BK_BYTES : FMT == FMT_E4M3 ? BK_BYTES : BK;  // K per slice
    static constexpr int kXPerSlice = FMT == FMT_BF16 ? BK : BK_BYTES;  // tensor-map x units (bf16 or bytes) per slice
    static constexpr int kSfBytes = FMT == FMT_NVFP4 ? kSfStageBytesA + kSfStageBytesB : 0;
    static constexpr int kStageTx = kStageBytes + kSfBytes;
    static constexpr int kAccBufs = FMT == FMT_NVFP4 ? 1 : 2;
    // NVFP4: a seventh warp copies each stage's block scales into TMEM, so
    // the MMA warp's one thread issues only the MMAs
    static constexpr bool kSfWarp = FMT == FMT_NVFP4 && DWDP_SF_WARP;
};

// Warp roles of one kernel instance: producer (warp 0), MMA (warp 1),
// EPIW epilogue warps, and for NVFP4 the scale-copy warp.  EPIW = 4 is one
// epilogue warp per TMEM lane quarter; EPIW = 8 (NVFP4 only) is two per
// quarter, each taking half of the tile's columns, so the single
// accumulator is drained and handed back sooner.
template <int FMT, int EPIW>
struct Warps {
    static_assert(EPIW == 4 || (EPIW == 8 && FMT == FMT_NVFP4), "8 epilogue warps are an NVFP4 variant");
    static constexpr int kEpiWarps = EPIW;
    static constexpr int kColSplit = EPIW / 4;
    static constexpr int kSfWarpIdx = 2 + EPIW;  // after the producer, MMA and epilogue warps
    static constexpr int kThreads = 32 * (2 + EPIW + (Fmt<FMT>::kSfWarp ? 1 : 0));
};
constexpr int kSfCol0 = BN;                             // NVFP4: first TMEM column of the scale ring
constexpr int kSfColsPerStage = 12 * kSfStepsPerSlice;  // per K step: 4 columns of A scales, 8 of B
static_assert(kSfCol0 + kStages * kSfColsPerStage <= 512, "NVFP4 scale ring must fit in TMEM");

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_timer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
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

// Bounded wait on one phase of an mbarrier.  Returns false when the CTA is
// aborting (another role gave up) or when this wait ran out of time, in which
// case it raises the abort flag and records `code` in the error word.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* err, int code, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort_flag) return false;
            if (global_timer() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicOr(err, code);
                return false;
            }
        }
    }
}

// Bounded wait that ignores the abort flag (used while draining).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, int* err, int code) {
    const uint64_t t0 = global_timer();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer() - t0 > kWaitLimitNs) {
            atomicOr(err, code);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// As tma_load_3d, but the box lands at the same shared-memory offset in every
// CTA of the cluster named in cta_mask, each completing its own mbarrier at
// the same offset.
__device__ __forceinline__ void tma_load_3d_mc(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                               uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(bar), "h"(cta_mask)
        : "memory");
}

// Untiled bulk copy of `bytes` (a multiple of 16, both addresses 16-byte
// aligned) into this CTA's shared memory, completing on bar.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"((uint64_t)src), "r"(bytes), "r"(bar)
        : "memory");
}

// As bulk_load, into the same offset of every CTA in cta_mask.
__device__ __forceinline__ void bulk_load_mc(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                             uint16_t cta_mask) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"((uint64_t)src), "r"(bytes), "r"(bar), "h"(cta_mask)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA in the cluster arrives, then waits for all.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with the swizzle that matches the slice width: rows of BK_BYTES bytes,
// 8-row atoms 8 * BK_BYTES apart (stride byte offset), start address >> 4 in
// bits 0-13, leading byte offset unused for these layouts (1), descriptor
// version 1 at bits 46-47, swizzle mode at bits 61-63 (2 = 128-byte, 4 =
// 64-byte).  The tile base is 1024-byte aligned.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)((8 * BK_BYTES) >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)(BK_BYTES == 128 ? 2 : 4) << 61;
    return d;
}

// Shared-memory descriptor of one 512-byte block-scale chunk for
// tcgen05.cp .32x128b: 32 rows of 16 bytes, no swizzle, 8-row core matrices
// 128 B apart (stride byte offset).
__device__ __forceinline__ uint64_t sf_chunk_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(128 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Copy one chunk into 32 TMEM lanes x 4 columns, replicated into all four
// lane quarters: lane m0 of each quarter, column c + m1 then holds the four
// scales of row 32 m1 + m0 for the K step.
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// The twelve chunks of one stage into its TMEM scale columns starting at tc:
// per 64-element K step j, A's 128 rows at tc + 4 j, B's two 128-row halves
// at tc + 16 + 8 j and tc + 20 + 8 j (sd: descriptor of the stage's first
// chunk; chunk o bytes further has descriptor sd + o / 16, since the
// start-address field holds address / 16 and shared memory addresses stay
// below its 2^14 limit, so the add never carries).
__device__ __forceinline__ void copy_stage_scales(uint32_t tc, uint64_t sd) {
    constexpr int kBCol = 4 * kSfStepsPerSlice;  // B scales follow A's columns
#pragma unroll
    for (int j = 0; j < kSfStepsPerSlice; ++j) {
        tc_cp_sf(tc + 4 * j, sd + (uint64_t)(j * kSfChunkBytes / 16));
        tc_cp_sf(tc + kBCol + 8 * j, sd + (uint64_t)((kSfStageBytesA + j * kSfChunkBytes) / 16));
        tc_cp_sf(tc + kBCol + 4 + 8 * j, sd + (uint64_t)((2 * kSfStageBytesA + j * kSfChunkBytes) / 16));
    }
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// One 128 x 256 MMA step over 32 bytes of K: 16 bf16, 32 E4M3 or 64 NVFP4
// elements (NVFP4: scaled by the E4M3 block scales at sfa / sfb in TMEM).
template <int FMT>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate,
                                       uint32_t sfa = 0, uint32_t sfb = 0) {
    if constexpr (FMT == FMT_NVFP4) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
                d_tmem),
            "l"(adesc), "l"(bdesc), "r"(kIdescNvfp4), "r"(accumulate), "r"(sfa), "r"(sfb)
            : "memory");
    } else if constexpr (FMT == FMT_E4M3) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(kIdescE4M3), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
            : "memory");
    }
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// Commit that arrives on the mbarrier at the same offset in every CTA of
// cta_mask once this thread's MMAs have finished reading shared memory.
__device__ __forceinline__ void tc_commit_mc(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(cta_mask)
        : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
        " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
        " [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

// SiLU(g) * u with the fast reciprocal (a few fp32 ulps; the result is
// rounded to bf16).  For g below about -88, exp(-g) overflows to inf and the
// reciprocal to 0, the limit of SiLU there.
__device__ __forceinline__ float silu_mul(float g, float u) {
    return g * __frcp_rn(1.0f + __expf(-g)) * u;
}

// Store 32 bf16 values (64 bytes) at p (16-byte aligned).
__device__ __forceinline__ void store_bf16x32(void* p, const float* v) {
    uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        q[i] = make_uint4(pack_bf16(v[8 * i + 0], v[8 * i + 1]), pack_bf16(v[8 * i + 2], v[8 * i + 3]),
                          pack_bf16(v[8 * i + 4], v[8 * i + 5]), pack_bf16(v[8 * i + 6], v[8 * i + 7]));
    }
}

template <int FMT>
struct SmemLayout {
    // offsets from the 1024-aligned base
    static constexpr int kA = 0;
    static constexpr int kB = kStages * kABytes;
    static constexpr int kSF = kB + kStages * kBBytes;    // NVFP4: A then B scale chunks per stage
    // full[S], empty[S], tfull[2], tempty[2], mdone, sf_full[S], cpdone
    static constexpr int kBars = kSF + kStages * Fmt<FMT>::kSfBytes;
    static constexpr int kNumBars = 3 * kStages + 6;
    static constexpr int kMisc = kBars + 8 * kNumBars;    // tmem base, abort flag
    static constexpr int kTileStart = kMisc + 16;         // int32[G+1]
};

template <int EPI, int FMT, int EPIW>
__global__ void __launch_bounds__(Warps<FMT, EPIW>::kThreads, 1) grouped_gemm_kernel(const __grid_constant__ GemmArgs p) {
    using SL = SmemLayout<FMT>;
    using F = Fmt<FMT>;
    using WR = Warps<FMT, EPIW>;
    constexpr int KE = F::kKElems;     // K elements per 128-byte slice
    constexpr int KX = F::kXPerSlice;  // the slice's width in tensor-map x units
    constexpr bool kScaled = FMT != FMT_BF16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + SL::kBars;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kStages + 2 + a); };
    const uint32_t mdone_bar = bar0 + 8u * (2 * kStages + 4);
    auto sf_full_bar = [&](int s) { return bar0 + 8u * (2 * kStages + 5 + s); };  // scales of stage s in TMEM
    const uint32_t cpdone_bar = bar0 + 8u * (3 * kStages + 5);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SL::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SL::kMisc + 4);
    int32_t* tile_start = reinterpret_cast<int32_t*>(smem + SL::kTileStart);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_routed = p.n_routed;
    const int G = n_routed + (p.shared_rows > 0 ? 1 : 0);
    const int ntile_cols = (EPI == EPI_SILU) ? (BN / 2) : BN;  // output columns per tile
    const int NT = (p.N + ntile_cols - 1) / ntile_cols;
    const int KB = (p.K + KE - 1) / KE;
    // EPI_F32 K split: a group's tiles are (K part, n-tile, m-tile), part-major
    const int KSPLIT = (EPI == EPI_F32 && p.k_split > 1) ? p.k_split : 1;
    const int NTV = NT * KSPLIT;
    const int KB_PART = (KB + KSPLIT - 1) / KSPLIT;
    // Paired mode: the two CTAs of a cluster hold tiles 2p and 2p+1 (every
    // group has an even number of tiles when NT is even, so a pair never
    // straddles two groups).  When both tiles use the same weight tile (same
    // n-tile: sibling m-tiles) each CTA loads one half of it and multicasts it
    // to both; either way each stage is refilled only after BOTH CTAs' MMAs
    // have finished with it (commits are multicast), so the pair stays in step.
    const bool paired = (EPI != EPI_F32) && (NT % 2 == 0);
    const uint32_t crank = cluster_ctarank();

    // ---- tile counts per group, then an inclusive scan into tile_start ----
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
        int rows = (g < n_routed) ? (p.row_offsets[g + 1] - p.row_offsets[g]) : p.shared_rows;
        if (rows < 0) {
            atomicOr(p.err, DERR_BAD_INDEX);
            rows = 0;
        }
        tile_start[g + 1] = ((rows + BM - 1) / BM) * NTV;
    }
    if (threadIdx.x == 0) {
        tile_start[0] = 0;
        *abort_flag = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), paired ? 2 : 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), WR::kEpiWarps);
        }
        mbar_init(mdone_bar, 1);
        for (int s = 0; s < kStages; ++s) mbar_init(sf_full_bar(s), 1);
        mbar_init(cpdone_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         smem_u32(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_map(&p.tmA[0]);
        prefetch_map(&p.tmA[1]);
        prefetch_map(&p.tmB[0]);
        prefetch_map(&p.tmB[1]);
        prefetch_map(&p.tmB[2]);
    }
    __syncthreads();
    // the peer's barriers must be initialised before anything is multicast into them
    if (paired) cluster_sync();
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base < G; base += 32) {
            const int i = base + lane;
            int v = (i < G) ? tile_start[i + 1] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int t = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += t;
            }
            v += carry;
            if (i < G) tile_start[i + 1] = v;
            carry = __shfl_sync(0xffffffffu, v, 31);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = tile_start[G];

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ----
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int pend[kStages];
#pragma unroll
            for (int s = 0; s < kStages; ++s) pend[s] = -1;
            int g = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                while (tile >= tile_start[g + 1]) ++g;
                const int mt = (tile_start[g + 1] - tile_start[g]) / NTV;
                const int local = tile - tile_start[g];
                const int nv = local / mt, m = local % mt;
                const int part = nv / NT, n = nv - part * NT;
                const int kb_begin = part * KB_PART, kb_end = min(KB, kb_begin + KB_PART);
                const bool routed = g < n_routed;
                const CUtensorMap* ma = routed ? &p.tmA[0] : &p.tmA[1];
                const int a_row = (routed ? p.row_offsets[g] : p.shared_a_row) + m * BM;
                const int2 src = p.bsrc[g];
                const CUtensorMap* mb = &p.tmB[src.x];
                int b_row0, b_row1;
                if (EPI == EPI_SILU) {
                    b_row0 = n * (BN / 2);
                    b_row1 = p.N + n * (BN / 2);
                } else {
                    b_row0 = n * BN;
                    b_row1 = n * BN + BN / 2;
                }
                // the pair shares the weight tile when the peer's tile (tile ^ 1,
                // same group) has the same n-tile
                const bool share = paired && (((local ^ 1) / mt) == n);
                int64_t atile = tile_start[g] / NTV + m;  // NVFP4: the A tile's scale chunks
                if (FMT == FMT_NVFP4 && atile >= p.sfa_tiles) {
                    atomicOr(p.err, DERR_BAD_INDEX);  // inconsistent group rows: read tile 0's scales instead
                    atile = 0;
                }
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.err, DERR_PRODUCER_WAIT)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full_bar(stage);
                    mbar_arrive_expect_tx(fb, F::kStageTx);
                    const uint32_t sa = sbase + SL::kA + stage * kABytes;
                    const uint32_t sb = sbase + SL::kB + stage * kBBytes;
                    tma_load_2d(sa, ma, kb * KX, a_row, fb);
                    if (share) {
                        // my half of the weight tile, into both CTAs' stages
                        const uint32_t off = crank ? (uint32_t)(kBBytes / 2) : 0u;
                        tma_load_3d_mc(sb + off, mb, kb * KX, crank ? b_row1 : b_row0, src.y, fb, (uint16_t)0x3);
                    } else {
                        tma_load_3d(sb, mb, kb * KX, b_row0, src.y, fb);
                        tma_load_3d(sb + kBBytes / 2, mb, kb * KX, b_row1, src.y, fb);
                    }
                    if constexpr (FMT == FMT_NVFP4) {
                        // the tiles' block scales: 4 K steps of A's 128 rows, then
                        // of B's two 128-row halves (multicast like the halves)
                        const uint32_t ss = sbase + SL::kSF + stage * F::kSfBytes;
                        const int64_t KS = p.K / 64;
                        bulk_load(ss, p.sfa + (atile * KS + kb * kSfStepsPerSlice) * kSfChunkBytes, kSfStageBytesA, fb);
                        const uint8_t* bs = p.bsf[src.x] + (int64_t)src.y * p.b_slot_bytes;
                        if (share) {
                            const int64_t rb = (crank ? b_row1 : b_row0) / BM;
                            bulk_load_mc(ss + kSfStageBytesA * (1 + crank), bs + (rb * KS + kb * kSfStepsPerSlice) * kSfChunkBytes,
                                         kSfStageBytesA, fb, (uint16_t)0x3);
                        } else {
                            bulk_load(ss + kSfStageBytesA, bs + ((int64_t)(b_row0 / BM) * KS + kb * kSfStepsPerSlice) * kSfChunkBytes,
                                      kSfStageBytesA, fb);
                            bulk_load(ss + 2 * kSfStageBytesA,
                                      bs + ((int64_t)(b_row1 / BM) * KS + kb * kSfStepsPerSlice) * kSfChunkBytes, kSfStageBytesA, fb);
                        }
                    }
                    pend[stage] = (int)phase;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // never leave a copy in flight into shared memory
#pragma unroll
                for (int s = 0; s < kStages; ++s)
                    if (pend[s] >= 0) mbar_wait_drain(full_bar(s), (uint32_t)pend[s], p.err, DERR_DRAIN_WAIT);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer ------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            int g = 0;
            const uint64_t ad0 = smem_desc(sbase + SL::kA), bd0 = smem_desc(sbase + SL::kB);
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                int nkb = KB;  // k-blocks of this tile (its K part's share when K is split)
                if (KSPLIT > 1) {
                    while (tile >= tile_start[g + 1]) ++g;
                    const int mt = (tile_start[g + 1] - tile_start[g]) / NTV;
                    const int part = ((tile - tile_start[g]) / mt) / NT;
                    nkb = min(KB, (part + 1) * KB_PART) - part * KB_PART;
                }
                if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.err, DERR_MMA_TMEM_WAIT)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);  // NVFP4: acc is always 0
                for (int kb = 0; kb < nkb; ++kb) {
                    // with the scale warp, its commit for this stage also means the
                    // stage's operands have landed (it waited for them first)
                    const uint32_t ready = F::kSfWarp ? sf_full_bar(stage) : full_bar(stage);
                    if (!mbar_wait(ready, phase, abort_flag, p.err, DERR_MMA_FULL_WAIT)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // stage s's tiles sit s * k{A,B}Bytes past stage 0's: add to the
                    // start-address field (address / 16; no carry, as below)
                    const uint64_t ad = ad0 + (uint64_t)(stage * (kABytes / 16));
                    const uint64_t bd = bd0 + (uint64_t)(stage * (kBBytes / 16));
                    if constexpr (FMT == FMT_NVFP4) {
                        // block scales of this stage into its TMEM columns (the MMAs
                        // that last read those columns finished before the stage was
                        // refilled; with the scale warp it has copied them already),
                        // then 4 block-scaled MMAs of 64 elements each
                        const uint32_t ss = sbase + SL::kSF + stage * F::kSfBytes;
                        const uint32_t tc = tmem_base + (uint32_t)(kSfCol0 + stage * kSfColsPerStage);
                        constexpr int kBCol = 4 * kSfStepsPerSlice;  // B scales follow A's columns
                        if constexpr (!F::kSfWarp) copy_stage_scales(tc, sf_chunk_desc(ss));
#pragma unroll
                        for (int kk = 0; kk < BK_BYTES / 32; ++kk)
                            tc_mma<FMT>(d_tmem, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk),
                                        (kb > 0 || kk > 0) ? 1u : 0u, tc + 4 * kk, tc + kBCol + 8 * kk);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < BK_BYTES / 32; ++kk) {
                            // advance 32 bytes (16 bf16 / 32 E4M3) along K inside the swizzle atom
                            tc_mma<FMT>(d_tmem, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk),
                                        (kb > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    // Paired CTAs always free a stage in both CTAs, shared tile or not:
                    // if a pair could drift apart on unshared tiles, the first shared
                    // tile's multicast could land in a stage the slower CTA still reads.
                    if (paired)
                        tc_commit_mc(empty_bar(stage), (uint16_t)0x3);
                    else
                        tc_commit(empty_bar(stage));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(tfull_bar(acc));
                if (++acc == F::kAccBufs) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // all issued MMAs complete before TMEM is released
            tc_commit(mdone_bar);
            mbar_wait_drain(mdone_bar, 0, p.err, DERR_MMA_DONE_WAIT);
        }
    } else if (F::kSfWarp && warp == WR::kSfWarpIdx) {
        // ------------------------------------------------ scale copies ----
        // Stage by stage in the MMA warp's order: once a stage's operands have
        // landed, copy its twelve block-scale chunks into the stage's TMEM
        // scale columns and commit to sf_full[stage], on which the MMA warp
        // waits.  The columns are free again by then: the stage was refilled
        // only after the MMAs that last read them had completed.
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(full_bar(stage), phase, abort_flag, p.err, DERR_MMA_FULL_WAIT)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ss = sbase + SL::kSF + stage * F::kSfBytes;
                    copy_stage_scales(tmem_base + (uint32_t)(kSfCol0 + stage * kSfColsPerStage), sf_chunk_desc(ss));
                    tc_commit(sf_full_bar(stage));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // every copy issued has completed before TMEM is released
            tc_commit(cpdone_bar);
            mbar_wait_drain(cpdone_bar, 0, p.err, DERR_MMA_DONE_WAIT);
        }
    } else {
        // ------------------------------------------------ epilogue --------
        const int quad = warp & 3;  // TMEM lanes [32*quad, 32*quad+32)
        const int half = (warp - 2) / 4;  // which share of the columns (kColSplit shares)
        constexpr int kCS = WR::kColSplit;
        const int row_in_tile = quad * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        int g = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            while (tile >= tile_start[g + 1]) ++g;
            const int mt = (tile_start[g + 1] - tile_start[g]) / NTV;
            const int local = tile - tile_start[g];
            const int nv = local / mt, m = local % mt;
            const int part = nv / NT, n = nv - part * NT;
            const bool routed = g < n_routed;
            const int rows = routed ? (p.row_offsets[g + 1] - p.row_offsets[g]) : p.shared_rows;
            const int64_t d_row0 = routed ? p.row_offsets[g] : p.shared_d_row;
            const int r = m * BM + row_in_tile;
            const int64_t grow = d_row0 + r;
            bool valid = r < rows;
            if (valid && (grow < 0 || grow >= p.d_rows)) {
                atomicOr(p.err, DERR_BAD_INDEX);
                valid = false;
            }
            // E4M3 / NVFP4: dequantize with the A row's scale times the group's weight scale
            float sc = 1.0f;
            if (kScaled && valid) {
                const int64_t arow = (routed ? (int64_t)p.row_offsets[g] : (int64_t)p.shared_a_row) + r;
                sc = __ldg(p.row_scale[routed ? 0 : 1] + arow) * p.gscale[g];
            }

            // the decision must be warp-uniform: tcgen05.ld below is .sync.aligned
            const bool got = mbar_wait(tfull_bar(acc), acc_phase, abort_flag, p.err, DERR_EPI_WAIT);
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quad * 32) << 16);

            if constexpr (F::kAccBufs == 1 && EPI == EPI_BF16) {
                // One accumulator (NVFP4): the next tile's MMAs wait for it, so
                // the row's 256 results go to registers as packed bf16 first,
                // the accumulator is released, and the stores follow.  (The
                // SiLU epilogue keeps the interleaved path below: fully unrolled
                // it ran slower.)
                // this warp's share: columns [cbase, cbase + BN / kCS) of the tile
                const int cbase = half * (BN / kCS);
                uint32_t packed[BN / 2 / kCS];
#pragma unroll
                for (int c = 0; c < BN / 32 / kCS; c += 2) {
                    uint32_t v[2][32];
                    tmem_ld32(taddr + cbase + c * 32, v[0]);
                    tmem_ld32(taddr + cbase + (c + 1) * 32, v[1]);
                    tmem_wait_ld();
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int j = 0; j < 32; j += 2)
                            packed[(c + h) * 16 + j / 2] =
                                pack_bf16(__uint_as_float(v[h][j]) * sc, __uint_as_float(v[h][j + 1]) * sc);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar(acc));
                __nv_bfloat16* D = reinterpret_cast<__nv_bfloat16*>(p.D);
                const int col0 = n * BN + cbase;
                if (valid) {
#pragma unroll
                    for (int c = 0; c < BN / 32 / kCS; ++c) {
                        if (col0 + c * 32 >= p.N) break;
                        uint4* q = reinterpret_cast<uint4*>(D + grow * p.ldd + col0 + c * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            q[i] = make_uint4(packed[c * 16 + 4 * i], packed[c * 16 + 4 * i + 1],
                                              packed[c * 16 + 4 * i + 2], packed[c * 16 + 4 * i + 3]);
                    }
                }
                if (++acc == F::kAccBufs) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
                continue;
            }
            // TMEM loads are issued two chunks (SiLU: two gate + two up chunks)
            // ahead of one wait, so their latencies overlap
            bool released = false;
            if (EPI == EPI_SILU) {
                __nv_bfloat16* D = reinterpret_cast<__nv_bfloat16*>(p.D);
                // this warp's share of the tile's 32-output chunks
                const int c_lo = half * (BN / 2 / 32 / kCS), c_hi = c_lo + BN / 2 / 32 / kCS;
#pragma unroll 1
                for (int c = c_lo; c < c_hi; c += 2) {
                    uint32_t gv[2][32], uv[2][32];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        tmem_ld32(taddr + (c + h) * 32, gv[h]);
                        tmem_ld32(taddr + BN / 2 + (c + h) * 32, uv[h]);
                    }
                    tmem_wait_ld();
                    if (c + 2 >= c_hi) {
                        // the last chunks are in registers: hand the accumulator
                        // back now, so the next tile's MMAs overlap this math
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(tempty_bar(acc));
                        released = true;
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int col = n * (BN / 2) + (c + h) * 32;
                        if (valid && col < p.N) {
                            float o[32];
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                o[j] = silu_mul(__uint_as_float(gv[h][j]) * sc, __uint_as_float(uv[h][j]) * sc);
                            store_bf16x32(D + grow * p.ldd + col, o);
                        }
                    }
                }
            } else if (EPI == EPI_BF16) {
                __nv_bfloat16* D = reinterpret_cast<__nv_bfloat16*>(p.D);
#pragma unroll 1
                for (int c = 0; c < BN / 32; c += 4) {
                    uint32_t v[4][32];
#pragma unroll
                    for (int h = 0; h < 4; ++h) tmem_ld32(taddr + (c + h) * 32, v[h]);
                    tmem_wait_ld();
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const int col = n * BN + (c + h) * 32;
                        if (valid && col < p.N) {
                            float o[32];
#pragma unroll
                            for (int j = 0; j < 32; ++j) o[j] = __uint_as_float(v[h][j]) * sc;
                            store_bf16x32(D + grow * p.ldd + col, o);
                        }
                    }
                }
            } else {
                float* D = reinterpret_cast<float*>(p.D) + (int64_t)part * p.split_stride;
                const float* bias = part == 0 ? p.col_bias : nullptr;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(taddr + c * 32, v);
                    tmem_wait_ld();
                    const int col0 = n * BN + c * 32;
                    if (valid) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int col = col0 + j;
                            if (col < p.N) {
                                float o = __uint_as_float(v[j]);
                                if (bias) o += bias[col];
                                D[grow * p.ldd + col] = o;
                            }
                        }
                    }
                }
            }
            if (!released) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar(acc));
            }
            if (++acc == F::kAccBufs) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    // neither CTA of a pair leaves while the other may still multicast into
    // its shared memory or arrive on its barriers
    if (paired) cluster_sync();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem_base) : "memory");
    }
}

// The bounded-wait check of dwdp_selftest_bounded_wait: one thread waits,
// with the GEMM's own mbar_wait and the given limit, for a phase of an
// mbarrier that nothing arrives at, so the wait runs out and records
// DERR_SELFTEST_WAIT.  The loop reads the global timer, so it always ends.
__global__ void bounded_wait_selftest_kernel(int* err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_wait(smem_u32(&bar), 0u, &abort_flag, err, DERR_SELFTEST_WAIT, limit_ns);
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int* err, uint64_t limit_ns, cudaStream_t stream) {
    bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

template <int FMT>
size_t gemm_smem_bytes(int n_groups) {
    return 1024 + SmemLayout<FMT>::kTileStart + sizeof(int32_t) * (size_t)(n_groups + 1);
}

cudaError_t launch_grouped_gemm(int epi, int fmt, const GemmArgs& args, int n_sms, cudaStream_t stream,
                                bool wide_epilogue) {
    const int G = args.n_routed + (args.shared_rows > 0 ? 1 : 0);
    size_t smem = 0;
    const void* fn = nullptr;
    int threads = Warps<FMT_BF16, 4>::kThreads;
    if (fmt == FMT_NVFP4) {
        smem = gemm_smem_bytes<FMT_NVFP4>(G);
        threads = Warps<FMT_NVFP4, 4>::kThreads;
        if (epi == EPI_SILU && wide_epilogue) {
            fn = (const void*)grouped_gemm_kernel<EPI_SILU, FMT_NVFP4, 8>;
            threads = Warps<FMT_NVFP4, 8>::kThreads;
        } else if (epi == EPI_SILU) {
            fn = (const void*)grouped_gemm_kernel<EPI_SILU, FMT_NVFP4, 4>;
        }
        if (epi == EPI_BF16) fn = (const void*)grouped_gemm_kernel<EPI_BF16, FMT_NVFP4, 4>;
    } else if (fmt == FMT_E4M3) {
        smem = gemm_smem_bytes<FMT_E4M3>(G);
        if (epi == EPI_SILU) fn = (const void*)grouped_gemm_kernel<EPI_SILU, FMT_E4M3, 4>;
        if (epi == EPI_BF16) fn = (const void*)grouped_gemm_kernel<EPI_BF16, FMT_E4M3, 4>;
    } else if (fmt == FMT_BF16) {
        smem = gemm_smem_bytes<FMT_BF16>(G);
        if (epi == EPI_SILU) fn = (const void*)grouped_gemm_kernel<EPI_SILU, FMT_BF16, 4>;
        if (epi == EPI_BF16) fn = (const void*)grouped_gemm_kernel<EPI_BF16, FMT_BF16, 4>;
        if (epi == EPI_F32) fn = (const void*)grouped_gemm_kernel<EPI_F32, FMT_BF16, 4>;
    }
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
    if (e != cudaSuccess) return e;
    // CTAs 2c and 2c+1 form one cluster, so they run on one GPC (one die).
    // The round-robin tile order gives them tiles 2p and 2p+1: sibling
    // m-tiles of one (group, n-tile), which read the same weight tile at the
    // same time and so share it in that die's L2 instead of each die
    // fetching it from HBM.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kClusterCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(kClusterCtas);
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    // persistent grid: every cluster resident at once
    cfg.gridDim = dim3(kClusterCtas * std::min(clusters, n_sms / kClusterCtas));
    void* kargs[] = {const_cast<GemmArgs*>(&args)};
    return cudaLaunchKernelExC(&cfg, fn, kargs);
}

}  // namespace dwdp
