// dwdp_internal.h: declarations shared by the translation units of libdwdp.so.
//
// Kernels live in gemm.cu (split-pointer grouped GEMM, tcgen05 + TMA) and
// route.cu (top-k, grouping, row scatter into expert order, combine, and the
// E4M3 / NVFP4 activation quantizers); dwdp_abi.cu is the C ABI.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the driver is reached through an entry point)
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dwdp.h"

namespace dwdp {

constexpr int kMaxGroups = DWDP_MAX_EXPERTS + 1;  // routed experts + one shared
constexpr int kRouterMaxSplit = 4;                  // K parts of the router GEMM

enum Epilogue : int { EPI_BF16 = 0, EPI_SILU = 1, EPI_F32 = 2 };

// GEMM operand formats (the weight_dtype values of dwdp.h).
enum OperandFormat : int { FMT_BF16 = DWDP_DTYPE_BF16, FMT_E4M3 = DWDP_DTYPE_E4M3, FMT_NVFP4 = DWDP_DTYPE_NVFP4 };

// Tile shape of the grouped GEMM: one CTA computes a 128 x 256 fp32
// accumulator in tensor memory from K slices of BK_BYTES bytes per row staged
// by TMA (128 bytes: 64 bf16, 128 E4M3 or 256 NVFP4 elements, 128-byte
// swizzle, 4 stages; 64 bytes: half of that, 64-byte swizzle, 8 stages).
#ifndef DWDP_SLICE_BYTES
#define DWDP_SLICE_BYTES 128
#endif
constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK_BYTES = DWDP_SLICE_BYTES;
constexpr int BK = BK_BYTES / 2;                // bf16 elements per K slice
constexpr int kStages = 512 / BK_BYTES;         // 192 KiB of A + B stages either way
constexpr int kABytes = BM * BK_BYTES;
constexpr int kBBytes = BN * BK_BYTES;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kClusterCtas = 2;                // CTAs per cluster (co-scheduled on one GPC)

// NVFP4 block scales as the block-scaled MMA takes them: for a row block rb
// (rows 128 rb .. 128 rb + 127) and a K step ks (elements 64 ks .. 64 ks + 63)
// one 512-byte chunk; the E4M3 scale of row 128 rb + 32 m1 + m0 and
// 16-element block kb of the step sits at byte 16 m0 + 4 m1 + kb.  Chunks
// run K step fastest: chunk (rb, ks) starts at (rb * K / 64 + ks) * 512.
// An activation operand's chunks are indexed by the GEMM's A tile instead
// of rb (see GemmArgs::sfa).
constexpr int kSfChunkBytes = 512;
constexpr int kSfStepsPerSlice = BK_BYTES / 32;          // 64-element K steps per K slice
constexpr int kSfStageBytesA = kSfStepsPerSlice * kSfChunkBytes;  // 128 rows x one K slice
constexpr int kSfStageBytesB = 2 * kSfStageBytesA;                // 256 rows x one K slice

// Bytes of one [rows][K] weight tensor (one pool slot) in format fmt:
// bf16 2 per element, E4M3 1, NVFP4 half a byte of code plus 1/16 byte of
// block scale (codes first, then the scale chunks).
inline int64_t weight_slot_bytes(int64_t rows, int64_t K, int fmt) {
    if (fmt == FMT_NVFP4) return rows * K / 2 + rows * K / 16;
    return rows * K * (fmt == FMT_E4M3 ? 1 : 2);
}
// Bytes of one row of GEMM operand codes in format fmt.
inline int64_t operand_row_bytes(int64_t K, int fmt) {
    return fmt == FMT_NVFP4 ? K / 2 : K * (fmt == FMT_E4M3 ? 1 : 2);
}

// Bits of the device error word (kernels OR them in; never trap).
enum DeviceError : int {
    DERR_PRODUCER_WAIT = 1 << 0,
    DERR_MMA_FULL_WAIT = 1 << 1,
    DERR_MMA_TMEM_WAIT = 1 << 2,
    DERR_EPI_WAIT = 1 << 3,
    DERR_DRAIN_WAIT = 1 << 4,
    DERR_MMA_DONE_WAIT = 1 << 5,
    DERR_BAD_INDEX = 1 << 6,
    DERR_NONFINITE_LOGIT = 1 << 7,  // a router logit is NaN or infinite
    DERR_SELFTEST_WAIT = 1 << 8,    // dwdp_selftest_bounded_wait's wait ran out (its expected result)
};

// One-thread kernel whose bounded mbarrier wait (the grouped GEMM's) runs
// out after limit_ns and records DERR_SELFTEST_WAIT in err (gemm.cu).
cudaError_t launch_bounded_wait_selftest(int* err, uint64_t limit_ns, cudaStream_t stream);

// Everything one grouped-GEMM launch needs; passed by value (grid constant).
// Group g < n_routed has rows [row_offsets[g], row_offsets[g+1]) of A0 and D;
// group n_routed (present when shared_rows > 0) has rows
// [shared_a_row, +shared_rows) of A1 and [shared_d_row, +shared_rows) of D.
// Group g reads weight slot bsrc[g].y of buffer tmB[bsrc[g].x].
struct GemmArgs {
    CUtensorMap tmA[2];
    CUtensorMap tmB[3];
    const int32_t* row_offsets;
    int32_t n_routed;
    int32_t shared_rows;
    int32_t shared_a_row;
    int32_t shared_d_row;
    int32_t K;
    int32_t N;      // output columns (EPI_SILU: weight rows = 2N)
    int64_t ldd;    // D row stride, elements
    int64_t d_rows; // rows of D: stores at or beyond it are dropped and flagged
    void* D;
    const float* col_bias;  // EPI_F32: added per column (K part 0 only), may be null
    // EPI_F32 only: K is cut into k_split contiguous parts of ceil(KB / k_split)
    // k-blocks (every part non-empty), each a tile of its own; part s writes
    // its partial sums to D + s * split_stride.  Other epilogues take 1.
    int32_t k_split;
    int64_t split_stride;  // elements
    int* err;
    // E4M3 and NVFP4 operands: the fp32 accumulator is multiplied by the A
    // row's scale (routed rows: row_scale[0][A row], shared rows:
    // row_scale[1][A row]) and by the group's weight scale gscale[g].
    const float* row_scale[2];
    // NVFP4 only.  sfa: the A operand's block-scale chunks, indexed by A tile:
    // the m-th 128-row tile of group g is A tile tile_start[g] / NT + m (groups
    // in order, the shared group last), so its chunks for K step ks start at
    // (atile * K / 64 + ks) * 512.  bsf[b]: start of slot 0's scale chunks in
    // weight buffer b; slot s's chunks are b_slot_bytes further per slot.
    const uint8_t* sfa;
    int64_t sfa_tiles;  // A tiles sfa has room for (a larger tile index is flagged)
    const uint8_t* bsf[3];
    int64_t b_slot_bytes;
    int2 bsrc[kMaxGroups];
    float gscale[kMaxGroups];
};

// TMA tensor maps (dwdp_abi.cu): a rows x K matrix (box 128 rows x BK_BYTES)
// and a weight buffer [slots][rows][K] (box 1 x 128 rows x BK_BYTES), both
// swizzled to BK_BYTES.  K counts elements of format fmt (bf16, E4M3 codes or
// NVFP4 codes, two per byte); a weight slot is weight_slot_bytes apart.
bool encode_rows(CUtensorMap* m, const void* base, uint64_t rows, uint64_t K, int fmt = FMT_BF16);
bool encode_slots(CUtensorMap* m, const void* base, uint64_t slots, uint64_t rows, uint64_t K,
                  int fmt = FMT_BF16);

// Sets the text dwdp_last_error(NULL) returns on this thread (dwdp_abi.cu).
void set_last_error(const char* msg);

// True when p points into device memory of device `dev` (cudaMalloc or
// virtual-memory allocations; not host, managed or another GPU's memory).
// Every buffer a TMA tensor map covers is checked with it before the map is
// encoded, so the GEMM's loads, including the loads it shares between the
// two CTAs of a cluster, only ever read this GPU's own memory.
inline bool is_device_memory_of(const void* p, int dev) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();  // an unknown pointer leaves no sticky error behind
        return false;
    }
    return at.type == cudaMemoryTypeDevice && at.device == dev;
}

// One grouped GEMM launch (gemm.cu) as 2-CTA clusters, one persistent CTA per
// SM.  fmt: both operands bf16, both E4M3 codes, or both NVFP4 codes with
// block scales (GemmArgs::sfa / bsf); K counts elements.  EPI_F32 is bf16 only.
// wide_epilogue: the NVFP4 gate/up GEMM drains its accumulator with eight
// warps instead of four (ignored otherwise).
cudaError_t launch_grouped_gemm(int epi, int fmt, const GemmArgs& args, int n_sms, cudaStream_t stream,
                                bool wide_epilogue = false);

// K parts of the router GEMM (bf16, K = H) for T tokens and E experts: with
// fewer 128-token tiles than SMs, as many parts as still fit one wave of
// n_sms CTAs, at most kRouterMaxSplit, none empty, and parts * T * E fp32
// planes within max_bytes.  Depends only on its arguments, so two callers
// with the same device and shapes split alike (and get the same logits).
inline int router_k_parts(int64_t T, int64_t E, int64_t H, int n_sms, size_t max_bytes) {
    const int64_t tiles = (T + BM - 1) / BM * ((E + BN - 1) / BN);
    const int64_t kb = (H + BK - 1) / BK;
    int parts = 1;
    for (int q = 2; q <= kRouterMaxSplit; ++q)
        if (tiles * q <= n_sms && (q - 1) * ((kb + q - 1) / q) < kb && (size_t)(q * T * E) * 4 <= max_bytes)
            parts = q;
    return parts;
}

// route.cu
// Top-k over logits given as `parts` fp32 planes [T][E] part_stride apart
// (summed in plane order, then bias); z_out, if not null, receives the sums.
// A token with a non-finite logit sets DERR_NONFINITE_LOGIT in err.
cudaError_t launch_topk(const float* logits, int parts, int64_t part_stride, const float* bias, int T, int E,
                        int k, int32_t* ids, float* w, float* z_out, int* err, cudaStream_t s);
cudaError_t launch_group(const int32_t* ids, int n, int E, int32_t* counts, int32_t* offsets,
                         int32_t* perm, int32_t* inv, cudaStream_t s);
// The same grouping in three passes over chunks of 1024 pairs; needs
// group_chunked_scratch_bytes(n, E) of device scratch (E <= 1024).
size_t group_chunked_scratch_bytes(int n, int E);
cudaError_t launch_group_chunked(const int32_t* ids, int n, int E, int32_t* counts, int32_t* offsets, int32_t* perm,
                                 int32_t* inv, int32_t* scratch, cudaStream_t s);
// Expert-ordered token rows: xp[inv[t k + j]] = x[t] for t < T, j < k.
// Rows outside [0, T k) in inv are flagged in err (DERR_BAD_INDEX) and skipped,
// here and in the combine.
cudaError_t launch_gather(const void* x, int H, const int32_t* inv, int T, int k, void* xp, int* err,
                          cudaStream_t s);
// E4M3 rows: codes[r][:] and scale[r] of bf16 rows (scale = amax / 448).
cudaError_t launch_quantize_rows(const void* in, int64_t rows, int cols, void* codes, float* scale, cudaStream_t s);
// x rows to E4M3 as launch_quantize_rows does (xq, sx), each also written to
// its chosen experts' rows: xp[inv[t k + j]] = xq[t], sxp[inv[t k + j]] = sx[t].
cudaError_t launch_quantize_x_e4m3(const void* x, int H, const int32_t* inv, int T, int k, void* xq, float* sx,
                                   void* xp, float* sxp, int* err, cudaStream_t s);
// NVFP4 activations (block scales in the GEMM's A-tile chunk layout): x
// rows quantized once per token and written to the shared-expert copy (xq,
// sx) and to each chosen expert's row of xp / sxp; a rows (routed rows in
// group order, then rows_all - rows_r shared rows).
// sf has room for sf_tiles A tiles; a row that would land beyond is flagged
// in err and not written.
cudaError_t launch_quantize_x_nvfp4(const void* x, int H, int T, int k, const int32_t* ids, const int32_t* inv,
                                    const int32_t* offsets, int E, bool has_shared, void* xq, float* sx, void* xp,
                                    float* sxp, uint8_t* sf, int64_t sf_tiles, int* err, cudaStream_t s);
cudaError_t launch_quantize_a_nvfp4(const void* act, int I, int64_t rows_r, int64_t rows_all, const int32_t* offsets,
                                    int E, void* aq, float* sa, uint8_t* sf, int64_t sf_tiles, int* err,
                                    cudaStream_t s);
cudaError_t launch_combine(const void* y, int H, const int32_t* inv, const float* w, int T, int k,
                           int64_t shared_row0, bool has_shared, void* out, int* err, cudaStream_t s);

}  // namespace dwdp
