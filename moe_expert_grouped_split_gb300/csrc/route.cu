// route.cu: routing, grouping, scatter into expert order, combine and the
// activation quantizers (E4M3, NVFP4) of the DWDP MoE block (memory- and
// latency-bound; coalesced 16-byte accesses, warp-level top-k, no atomics on
// any ordered output so every index is deterministic).
//
// The pages do not print the router; these kernels implement the reading the
// library documents in dwdp.h: fp32 logits, the k largest (ties to the lower
// expert id), the chosen set listed in ascending id, weights = softmax
// renormalised over the chosen set, and (token, slot) pairs grouped by expert
// in ascending flat index t*k+j.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <atomic>

#include "dwdp_internal.h"

namespace dwdp {
namespace {

constexpr int kMaxPerLane = DWDP_MAX_EXPERTS / 32;
constexpr int kQuantWarps = 8;  // warps per block of the NVFP4 quantizers

// Order-preserving key of a logit: a > b as floats iff key(a) > key(b) as
// unsigned; -0 is folded into +0 so equal values tie.  Every finite or
// infinite value has a key >= 0x007FFFFF, so 0 marks "no candidate".  Every
// NaN, whatever its sign or payload, gets the one key 0xFFFFFFFF (above
// +inf), so a token with NaN logits still gets k distinct picks.
__device__ __forceinline__ uint32_t order_key(float x) {
    if (x != x) return 0xFFFFFFFFu;
    const uint32_t u = __float_as_uint(x == 0.0f ? 0.0f : x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// One warp per token.  Lane l holds logits l, l+32, ... (PER of them: E <= 32
// PER) and keeps the best of its own not yet chosen ones.  Each of the k
// rounds takes the warp's largest key, then the lowest expert id holding it
// (ties to the lower id), with two warp reductions; only the lane that owned
// the pick rescans.  The chosen set is then listed in ascending id.
// w_j = exp(z_j - z_max) / sum_i exp(z_i - z_max) over the chosen set (the
// full softmax denominator cancels in the renormalisation).
// The logits arrive as `parts` partial-sum planes part_stride apart (a
// K-split router GEMM), added in plane order; with z_out the sums are stored.
// A token with a logit that is not finite (NaN or +-inf) has no defined
// choice or weights: it is still routed (some k distinct experts) and
// DERR_NONFINITE_LOGIT is set in err.
template <int PER>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, int parts,
                                                   int64_t part_stride, const float* __restrict__ bias,
                                                   int T, int E, int k, int32_t* __restrict__ ids,
                                                   float* __restrict__ w, float* __restrict__ z_out,
                                                   int* __restrict__ err) {
    constexpr int kNone = 0x7fffffff;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float* z = logits + (int64_t)t * E;
    uint32_t key[PER];
    bool finite = true;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int e = lane + 32 * j;
        key[j] = 0u;
        if (e < E) {
            float v = z[e];
            for (int q = 1; q < parts; ++q) v += z[q * part_stride + e];
            if (bias) v += bias[e];
            if (z_out) z_out[(int64_t)t * E + e] = v;
            finite &= isfinite(v);
            key[j] = order_key(v);
        }
    }
    if (!__all_sync(0xffffffffu, finite) && lane == 0) atomicOr(err, DERR_NONFINITE_LOGIT);
    // this lane's best remaining candidate (largest key, lowest id on ties)
    auto best = [&](uint32_t& bk, int& bi) {
        bk = 0u;
        bi = kNone;
#pragma unroll
        for (int j = 0; j < PER; ++j)
            if (key[j] > bk) {
                bk = key[j];
                bi = lane + 32 * j;
            }
    };
    uint32_t lk;
    int li;
    best(lk, li);
    int my_id = -1;  // lane s < k ends up holding the s-th chosen id
    float my_val = 0.0f;
    for (int s = 0; s < k; ++s) {
        const uint32_t gk = __reduce_max_sync(0xffffffffu, lk);
        const int gi = __reduce_min_sync(0xffffffffu, (lk == gk && gk != 0u) ? li : kNone);
        if (gi == kNone) break;  // fewer than k candidates (k <= E is checked on the host)
        if (lane == s) {
            my_id = gi;
            my_val = key_value(gk);
        }
        if ((gi & 31) == lane) {
#pragma unroll
            for (int j = 0; j < PER; ++j)  // (a constant index keeps key[] in registers)
                if (j == (gi >> 5)) key[j] = 0u;
            best(lk, li);
        }
    }
    // rank of my id among the chosen ids -> ascending-id slot
    int rank = 0;
    for (int s = 0; s < k; ++s) {
        const int other = __shfl_sync(0xffffffffu, my_id, s);
        if (lane < k && my_id >= 0 && other >= 0 && other < my_id) ++rank;
    }
    // z_max is the first pick
    const float zmax = __shfl_sync(0xffffffffu, my_val, 0);
    const float ex = (lane < k && my_id >= 0) ? __expf(my_val - zmax) : 0.0f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane < k && my_id >= 0) {
        ids[(int64_t)t * k + rank] = my_id;
        w[(int64_t)t * k + rank] = ex / sum;
    }
}

__device__ __forceinline__ int block_sum(int v, int* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    int s = 0;
    for (int i = 0; i < nw; ++i) s += red[i];
    return s;
}

// counts[e] = #{f : ids[f] == e}; one block per expert scans all pairs.
__global__ void __launch_bounds__(1024) count_kernel(const int32_t* __restrict__ ids, int n,
                                                     int32_t* __restrict__ counts) {
    __shared__ int red[32];
    const int e = blockIdx.x;
    int c = 0;
    const int n4 = n >> 2;
    const int4* ids4 = reinterpret_cast<const int4*>(ids);
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
        const int4 q = ids4[i];
        c += (q.x == e) + (q.y == e) + (q.z == e) + (q.w == e);
    }
    for (int i = (n4 << 2) + threadIdx.x; i < n; i += blockDim.x) c += (ids[i] == e);
    c = block_sum(c, red);
    if (threadIdx.x == 0) counts[e] = c;
}

// Stable placement: block e computes offsets[e] from counts, then walks the
// pairs in flat order; pair f with ids[f] == e gets row offsets[e] + (number
// of earlier pairs of e).  A block-wide exclusive scan of the match flags
// keeps the walk in order.
__global__ void __launch_bounds__(1024) place_kernel(const int32_t* __restrict__ ids, int n, int E,
                                                     const int32_t* __restrict__ counts,
                                                     int32_t* __restrict__ offsets,
                                                     int32_t* __restrict__ perm,
                                                     int32_t* __restrict__ inv) {
    __shared__ int red[32];
    __shared__ int wsum[32];
    const int e = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    int part = 0;
    for (int i = threadIdx.x; i < e; i += blockDim.x) part += counts[i];
    const int base = block_sum(part, red);
    if (threadIdx.x == 0) {
        offsets[e] = base;
        if (e == E - 1) offsets[E] = base + counts[e];
    }
    int running = base;
    for (int start = 0; start < n; start += blockDim.x) {
        const int f = start + threadIdx.x;
        const bool hit = f < n && ids[f] == e;
        const uint32_t ball = __ballot_sync(0xffffffffu, hit);
        const int in_warp = __popc(ball & ((1u << lane) - 1u));
        __syncthreads();
        if (lane == 0) wsum[warp] = __popc(ball);
        __syncthreads();
        int before = 0, total = 0;
        for (int i = 0; i < nw; ++i) {
            const int c = wsum[i];
            if (i < warp) before += c;
            total += c;
        }
        if (hit) {
            const int r = running + before + in_warp;
            perm[r] = f;
            inv[f] = r;
        }
        running += total;
    }
}

// The same grouping as count_kernel + place_kernel, in three passes over
// chunks of kChunk consecutive pairs (one 1024-thread block per chunk):
//   chunk_count:  hist[c][e] = pairs of chunk c routed to expert e
//   chunk_scan:   counts, offsets, and base[c][e] = offsets[e] + pairs of
//                 e in chunks before c
//   chunk_place:  pair f of chunk c with expert e goes to row base[c][e] +
//                 (pairs of e earlier in the chunk), ranked with warp
//                 match_any inside a warp and per-warp counts across warps.
// Every row is the stable (ascending flat index) position, the one
// count_kernel + place_kernel give.
constexpr int kChunk = 1024;

__global__ void __launch_bounds__(kChunk) chunk_count_kernel(const int32_t* __restrict__ ids, int n, int E,
                                                             int32_t* __restrict__ hist) {
    extern __shared__ int h[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
    __syncthreads();
    const int f = blockIdx.x * kChunk + threadIdx.x;
    if (f < n) atomicAdd(&h[ids[f]], 1);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(int64_t)blockIdx.x * E + e] = h[e];
}

// One block of 1024 threads; P = 1024 / (E rounded up to a power of two)
// threads per expert: thread (e, q) owns the q-th run of consecutive chunks
// of expert e.  Pass 1 sums the run, the runs' sums are scanned per expert
// and the experts' totals across experts, and pass 2 rewrites the run's
// counts as bases.  The loads and stores of a run go four at a time, so a
// thread waits on memory a few times instead of once per chunk.
__global__ void __launch_bounds__(1024) chunk_scan_kernel(int32_t* __restrict__ hist, int n_chunks, int E,
                                                          int32_t* __restrict__ counts,
                                                          int32_t* __restrict__ offsets) {
    __shared__ int part[1024];  // per thread: its run's sum, then the run's offset within its expert
    __shared__ int scan[1024];  // per expert: inclusive scan of the totals
    int ep = 1;
    while (ep < E) ep <<= 1;
    const int P = 1024 / ep;  // E <= 1024, so P >= 1
    const int tid = threadIdx.x;
    const int e = tid / P, q = tid % P;
    const bool active = e < E;
    const int per = (n_chunks + P - 1) / P;
    const int c0 = min(n_chunks, q * per), c1 = min(n_chunks, c0 + per);
    int sum = 0;
    if (active) {
        int c = c0;
        for (; c + 4 <= c1; c += 4) {
            int v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = hist[(int64_t)(c + u) * E + e];
            sum += v[0] + v[1] + v[2] + v[3];
        }
        for (; c < c1; ++c) sum += hist[(int64_t)c * E + e];
    }
    part[tid] = sum;
    __syncthreads();
    // per expert: exclusive offsets of its P runs, and its total
    int c_e = 0;
    if (active && q == 0) {
        for (int r = 0; r < P; ++r) {
            const int v = part[tid + r];
            part[tid + r] = c_e;
            c_e += v;
        }
    }
    scan[tid] = 0;
    __syncthreads();
    if (active && q == 0) scan[e] = c_e;
    __syncthreads();
    // inclusive scan over experts (Hillis-Steele in shared memory)
    for (int o = 1; o < 1024; o <<= 1) {
        const int v = (tid >= o) ? scan[tid - o] : 0;
        __syncthreads();
        scan[tid] += v;
        __syncthreads();
    }
    if (active) {
        const int total = scan[e] - (e > 0 ? scan[e - 1] : 0);
        const int base = scan[e] - total;  // pairs of experts before e
        if (q == 0) {
            counts[e] = total;
            offsets[e] = base;
            if (e == E - 1) offsets[E] = scan[e];
        }
        int running = base + part[tid];
        int c = c0;
        for (; c + 4 <= c1; c += 4) {
            int v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = hist[(int64_t)(c + u) * E + e];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                hist[(int64_t)(c + u) * E + e] = running;
                running += v[u];
            }
        }
        for (; c < c1; ++c) {
            const int v = hist[(int64_t)c * E + e];
            hist[(int64_t)c * E + e] = running;
            running += v;
        }
    }
}

__global__ void __launch_bounds__(kChunk) chunk_place_kernel(const int32_t* __restrict__ ids, int n, int E,
                                                             const int32_t* __restrict__ base,
                                                             int32_t* __restrict__ perm,
                                                             int32_t* __restrict__ inv) {
    extern __shared__ uint8_t wc[];  // [32 warps][E]: pairs of e in each warp (<= 32)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wc[i] = 0;
    const int f = blockIdx.x * kChunk + threadIdx.x;
    const bool valid = f < n;
    const int e = valid ? ids[f] : -1;
    __syncthreads();
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int rank_w = __popc(peers & ((1u << lane) - 1u));
    if (valid && lane == __ffs(peers) - 1) wc[warp * E + e] = (uint8_t)__popc(peers);
    __syncthreads();
    if (valid) {
        int before = 0;
        for (int w = 0; w < warp; ++w) before += wc[w * E + e];
        const int r = base[(int64_t)blockIdx.x * E + e] + before + rank_w;
        perm[r] = f;
        inv[f] = r;
    }
}

// Expert-ordered copies of the token rows: xp[inv[t k + j]][:] = x[t][:]
// for every chosen expert j of token t (and sxp[inv[t k + j]] = sx[t] when
// sxp is given).  One warp per token reads its row from HBM once and stores
// it to its k slots, so the pass moves T rows in and T k rows out; walking
// the permuted rows instead reads each token row k times at random
// distances, which L2 does not hold.  The stores are streaming
// (st.global.cs): the gate/up GEMM reads them long after they would have
// left L2.  Each lane keeps four 16-byte loads in flight.  KC > 0 fixes k at
// compile time so the k destinations stay in registers.  A destination row
// outside [0, T k) is flagged in err and not written.
template <int KC>
__global__ void __launch_bounds__(256) scatter_rows_kernel(const uint4* __restrict__ x, int row_vecs,
                                                           const int32_t* __restrict__ inv, int T, int k,
                                                           uint4* __restrict__ xp, const float* __restrict__ sx,
                                                           float* __restrict__ sxp, int* __restrict__ err) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const int kk = KC > 0 ? KC : k;
    const int64_t n_rows = (int64_t)T * kk;
    const int32_t* it = inv + (int64_t)t * kk;
    const uint4* src = x + (int64_t)t * row_vecs;
    uint32_t ok = 0;  // bit j: destination j is in range
    for (int j = 0; j < kk; ++j) {
        const int32_t r = it[j];
        if (r >= 0 && r < n_rows) ok |= 1u << j;
    }
    if (ok != (kk == 32 ? 0xffffffffu : (1u << kk) - 1u) && lane == 0) atomicOr(err, DERR_BAD_INDEX);
    if (sxp != nullptr)
        for (int j = lane; j < kk; j += 32)
            if ((ok >> j) & 1u) sxp[it[j]] = sx[t];
    if constexpr (KC > 0) {
        int64_t dst[KC];
#pragma unroll
        for (int j = 0; j < KC; ++j) dst[j] = (int64_t)it[j] * row_vecs;
        int i = lane;
        for (; i + 96 < row_vecs; i += 128) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = __ldg(src + i + 32 * u);
#pragma unroll
            for (int j = 0; j < KC; ++j)
                if ((ok >> j) & 1u) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) __stcs(xp + dst[j] + i + 32 * u, v[u]);
                }
        }
        for (; i < row_vecs; i += 32) {
            const uint4 v = __ldg(src + i);
#pragma unroll
            for (int j = 0; j < KC; ++j)
                if ((ok >> j) & 1u) __stcs(xp + dst[j] + i, v);
        }
    } else {
        for (int i = lane; i < row_vecs; i += 32) {
            const uint4 v = __ldg(src + i);
            for (int j = 0; j < kk; ++j)
                if ((ok >> j) & 1u) __stcs(xp + (int64_t)it[j] * row_vecs + i, v);
        }
    }
}

template <int KC>
void scatter_rows_launch(const uint4* x, int row_vecs, const int32_t* inv, int T, int k, uint4* xp,
                         const float* sx, float* sxp, int* err, cudaStream_t s) {
    const int warps = 8;
    scatter_rows_kernel<KC><<<(T + warps - 1) / warps, 32 * warps, 0, s>>>(x, row_vecs, inv, T, k, xp, sx, sxp, err);
}

cudaError_t scatter_rows(const void* x, int row_vecs, const int32_t* inv, int T, int k, void* xp, const float* sx,
                         float* sxp, int* err, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    uint4* pv = reinterpret_cast<uint4*>(xp);
    switch (k) {
        case 2: scatter_rows_launch<2>(xv, row_vecs, inv, T, k, pv, sx, sxp, err, s); break;
        case 4: scatter_rows_launch<4>(xv, row_vecs, inv, T, k, pv, sx, sxp, err, s); break;
        case 8: scatter_rows_launch<8>(xv, row_vecs, inv, T, k, pv, sx, sxp, err, s); break;
        default: scatter_rows_launch<0>(xv, row_vecs, inv, T, k, pv, sx, sxp, err, s);
    }
    return cudaGetLastError();
}

__device__ __forceinline__ void acc_bf16x8(float (&a)[8], uint4 q, float s) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        a[2 * i] = fmaf(s, f.x, a[2 * i]);
        a[2 * i + 1] = fmaf(s, f.y, a[2 * i + 1]);
    }
}

// out[t] = sum_j w[t][j] * y[inv[t*k+j]] (slot order), then + y[shared_row0 + t];
// fp32 sums, one bf16 rounding at the end.  One warp per token.
__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ y, int row_vecs,
                                                      const int32_t* __restrict__ inv,
                                                      const float* __restrict__ w, int T, int k,
                                                      int64_t shared_row0, int has_shared,
                                                      uint4* __restrict__ out, int* __restrict__ err) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    int rows[DWDP_MAX_TOPK];
    float ws[DWDP_MAX_TOPK];
    for (int j = 0; j < k; ++j) {
        rows[j] = inv[(int64_t)t * k + j];
        ws[j] = w[(int64_t)t * k + j];
        if (rows[j] < 0 || (int64_t)rows[j] >= (int64_t)T * k) {   // flagged; contributes nothing
            if (lane == 0) atomicOr(err, DERR_BAD_INDEX);
            rows[j] = -1;
        }
    }
    for (int i = lane; i < row_vecs; i += 32) {
        float a[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int j = 0; j < k; ++j)
            if (rows[j] >= 0) acc_bf16x8(a, __ldg(y + (int64_t)rows[j] * row_vecs + i), ws[j]);
        if (has_shared) acc_bf16x8(a, __ldg(y + (shared_row0 + t) * row_vecs + i), 1.0f);
        uint4 o;
        __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
        for (int q = 0; q < 4; ++q) oh[q] = __floats2bfloat162_rn(a[2 * q], a[2 * q + 1]);
        out[(int64_t)t * row_vecs + i] = o;
    }
}

// combine_kernel with k fixed at compile time: the token's rows and weights
// stay in registers and all k (+1) row loads are issued before the sums,
// which are the same fp32 operations in the same order.
template <int KC>
__global__ void __launch_bounds__(256) combine_kernel_k(const uint4* __restrict__ y, int row_vecs,
                                                        const int32_t* __restrict__ inv,
                                                        const float* __restrict__ w, int T,
                                                        int64_t shared_row0, int has_shared,
                                                        uint4* __restrict__ out, int* __restrict__ err) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    int64_t rows[KC];
    float ws[KC];
    bool bad = false;
#pragma unroll
    for (int j = 0; j < KC; ++j) {
        const int32_t r = inv[(int64_t)t * KC + j];
        const bool ok = r >= 0 && (int64_t)r < (int64_t)T * KC;
        bad |= !ok;
        // a row outside [0, T k) is flagged and read as row 0 with weight 0,
        // so the loads stay unconditional and in bounds
        rows[j] = ok ? (int64_t)r * row_vecs : 0;
        ws[j] = ok ? w[(int64_t)t * KC + j] : 0.0f;
    }
    if (bad && lane == 0) atomicOr(err, DERR_BAD_INDEX);
    const int64_t srow = (shared_row0 + t) * row_vecs;
    for (int i = lane; i < row_vecs; i += 32) {
        uint4 q[KC + 1];
#pragma unroll
        for (int j = 0; j < KC; ++j) q[j] = __ldg(y + rows[j] + i);
        if (has_shared) q[KC] = __ldg(y + srow + i);
        float a[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < KC; ++j) acc_bf16x8(a, q[j], ws[j]);
        if (has_shared) acc_bf16x8(a, q[KC], 1.0f);
        uint4 o;
        __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
        for (int c = 0; c < 4; ++c) oh[c] = __floats2bfloat162_rn(a[2 * c], a[2 * c + 1]);
        out[(int64_t)t * row_vecs + i] = o;
    }
}

// Eight bf16 values to E4M3 codes (byte i of the result is value i): the
// binary32 quotient v / s, rounded to nearest even, saturated to +-448.
__device__ __forceinline__ uint2 e4m3_codes8(uint4 q, float s) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
    uint32_t w[2] = {0, 0};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(h[j]);
        const uint32_t c0 = __nv_cvt_float_to_fp8(f.x / s, __NV_SATFINITE, __NV_E4M3);
        const uint32_t c1 = __nv_cvt_float_to_fp8(f.y / s, __NV_SATFINITE, __NV_E4M3);
        w[j >> 1] |= (c0 | (c1 << 8)) << ((j & 1) * 16);
    }
    return make_uint2(w[0], w[1]);
}

// binary32 amax of a warp's bf16 row (exact for bf16 inputs), all lanes
// holding it.
__device__ __forceinline__ float row_amax_bf16(const uint4* __restrict__ src, int nv, int lane) {
    float amax = 0.0f;
    for (int i = lane; i < nv; i += 32) {
        const uint4 q = __ldg(src + i);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(h[j]);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    return amax;
}

// E4M3 rows, one warp per row: amax of the row (binary32, exact for bf16
// inputs), scale = amax / 448 (1 for an all-zero row), code = E4M3 of the
// binary32 quotient v / scale, rounded to nearest even and saturated to
// +-448.  cols is a multiple of 8.
__global__ void __launch_bounds__(256) quantize_rows_kernel(const uint4* __restrict__ in, int64_t rows, int cols,
                                                            uint2* __restrict__ codes, float* __restrict__ scale) {
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (r >= rows) return;
    const int nv = cols / 8;
    const uint4* src = in + r * nv;
    const float amax = row_amax_bf16(src, nv, lane);
    const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    if (lane == 0) scale[r] = s;
    uint2* dst = codes + r * nv;
    for (int i = lane; i < nv; i += 32) dst[i] = e4m3_codes8(__ldg(src + i), s);
}

// x rows to E4M3 once per token, written to the shared expert's copy (xq,
// sx) and straight into each chosen expert's row of xp / sxp (inv[t k + j]),
// so x's codes are not read back for a separate scatter.  One warp per token,
// the same arithmetic as quantize_rows_kernel; the second pass re-reads the
// row from L2.  KC > 0 fixes k at compile time.  A destination outside
// [0, T k) is flagged in err and not written.
template <int KC>
__global__ void __launch_bounds__(256) quantize_x_e4m3_kernel(const uint4* __restrict__ x, int nv,
                                                              const int32_t* __restrict__ inv, int T, int k,
                                                              uint2* __restrict__ xq, float* __restrict__ sx,
                                                              uint2* __restrict__ xp, float* __restrict__ sxp,
                                                              int* __restrict__ err) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const int kk = KC > 0 ? KC : k;
    const int64_t n_rows = (int64_t)T * kk;
    const int32_t* it = inv + (int64_t)t * kk;
    uint32_t ok = 0;  // bit j: destination j is in range
    for (int j = 0; j < kk; ++j) {
        const int32_t r = it[j];
        if (r >= 0 && r < n_rows) ok |= 1u << j;
    }
    if (ok != (kk == 32 ? 0xffffffffu : (1u << kk) - 1u) && lane == 0) atomicOr(err, DERR_BAD_INDEX);
    const uint4* src = x + (int64_t)t * nv;
    const float amax = row_amax_bf16(src, nv, lane);
    const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    if (lane == 0) sx[t] = s;
    for (int j = lane; j < kk; j += 32)
        if ((ok >> j) & 1u) sxp[it[j]] = s;
    uint2* own = xq + (int64_t)t * nv;
    if constexpr (KC > 0) {
        int64_t dst[KC];
#pragma unroll
        for (int j = 0; j < KC; ++j) dst[j] = (int64_t)it[j] * nv;
        for (int i = lane; i < nv; i += 32) {
            const uint2 c = e4m3_codes8(__ldg(src + i), s);
            own[i] = c;
#pragma unroll
            for (int j = 0; j < KC; ++j)
                if ((ok >> j) & 1u) __stcs(xp + dst[j] + i, c);
        }
    } else {
        for (int i = lane; i < nv; i += 32) {
            const uint2 c = e4m3_codes8(__ldg(src + i), s);
            own[i] = c;
            for (int j = 0; j < kk; ++j)
                if ((ok >> j) & 1u) __stcs(xp + (int64_t)it[j] * nv + i, c);
        }
    }
}

// ------------------------------------------------------------- NVFP4 --
// Activation rows to NVFP4 for the block-scaled GEMMs.  Per row of n bf16
// values (n a multiple of 64; a lane takes two adjacent blocks at a time):
// s = amax / 2688 (1 for an all-zero row),
// d = 6 s; per 16-element block, its E4M3 scale sf = E4M3(amax_block / d)
// (round to nearest even, saturating) and, with eff = value(sf) * s, each
// element's E2M1 code of v / eff (round to nearest even, saturating; all
// zero when sf is 0).  Every step is one binary32 operation, so the codes
// are the same integer decisions whoever takes them in binary32.  Codes are
// packed two per byte, element 2i in the low nibble.  Block scales go to the
// chunk layout of the GEMM's A tiles (see kSfChunkBytes): a routed row r of
// group g is row (r - offsets[g]) % 128 of A tile tb[g] + (r - offsets[g]) /
// 128, where tb[g] counts the 128-row tiles of the groups before g; shared
// row i is row i % 128 of A tile tb[E] + i / 128.

// binary32 value of a non-negative E4M3 code (exact): exponent field 0 is
// m * 2^-9, otherwise 2^(e-7) * (1 + m/8).
__device__ __forceinline__ float e4m3_value(uint32_t c) {
    const uint32_t e = (c >> 3) & 15u, m = c & 7u;
    return e == 0 ? (float)m * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Eight binary32 values to eight E2M1 codes (cvt.rn.satfinite), value i in
// bits 4i .. 4i+3.
__device__ __forceinline__ uint32_t e2m1x8(const float* v) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

// 16 bf16 values (two uint4) as binary32.
__device__ __forceinline__ void bf16x16_to_float(const uint4* q, float (&v)[16]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&q[h]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(p[j]);
            v[8 * h + 2 * j] = f.x;
            v[8 * h + 2 * j + 1] = f.y;
        }
    }
}

__device__ __forceinline__ void load_bf16x16(const uint4* src, float (&v)[16]) {
    const uint4 q[2] = {__ldg(src), __ldg(src + 1)};
    bf16x16_to_float(q, v);
}

// The row scale s of one row of nb blocks (two uint4 per block), warp-wide.
__device__ __forceinline__ float nvfp4_row_scale(const uint4* src, int nb, int lane) {
    float amax = 0.0f;
#pragma unroll 4
    for (int b = lane; b < nb; b += 32) {
        float v[16];
        load_bf16x16(src + 2 * b, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    return amax > 0.0f ? amax / 2688.0f : 1.0f;
}

// a / b rounded to nearest even, given y = RN(1/b): Markstein's one-step
// correction (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with
// q = RN(a y), the remainder r = a - b q is exact in one FMA and RN(q + r y)
// is the correctly rounded quotient, for b, 1/b and a/b in the normal range.
// The caller keeps b within [2^-100, 2^100]; a quotient below the normal
// range then has |a| below it too and lies far below 0.25, where every
// rounding gives E2M1 code 0; copysign keeps the sign of a zero quotient.
__device__ __forceinline__ float div_rn_markstein(float a, float b, float y) {
    const float q = __fmul_rn(a, y);
    const float r = fmaf(-q, b, a);
    return copysignf(fmaf(r, y, q), a);
}

// One 16-element block (its two uint4 of bf16 in q): its E4M3 scale code and
// 16 E2M1 codes (8 bytes).
__device__ __forceinline__ uint32_t nvfp4_block(const uint4* q, float s, float d, uint2& codes) {
    float v[16];
    bf16x16_to_float(q, v);
    float ab = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(v[i]));
    const uint32_t sf = __nv_cvt_float_to_fp8(ab / d, __NV_SATFINITE, __NV_E4M3);
    const float eff = e4m3_value(sf) * s;
    if (sf == 0) {
        codes = make_uint2(0u, 0u);
    } else {
        if (eff >= 0x1p-100f && eff <= 0x1p100f) {
            // the 16 quotients v / eff, correctly rounded, from one reciprocal
            const float y = __frcp_rn(eff);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = div_rn_markstein(v[i], eff, y);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = v[i] / eff;
        }
        codes = make_uint2(e2m1x8(v), e2m1x8(v + 8));
    }
    return sf;
}

// Two adjacent blocks (their four uint4 of bf16 in q): their scale codes
// (the first block's in the low byte) and 32 E2M1 codes (16 bytes), so a
// lane stores 16 bytes of codes and 2 adjacent scale bytes at once.
__device__ __forceinline__ uint32_t nvfp4_block_pair(const uint4 (&q)[4], float s, float d, uint4& codes) {
    uint2 c0, c1;
    const uint32_t f0 = nvfp4_block(q, s, d, c0);
    const uint32_t f1 = nvfp4_block(q + 2, s, d, c1);
    codes = make_uint4(c0.x, c0.y, c1.x, c1.y);
    return f0 | (f1 << 8);
}

// The lanes that run the iteration of a two-blocks-per-lane loop (block b =
// 2 lane + 64 i) in which this lane holds block b: lanes l with
// 2 l + 64 i < nb.  nb is a multiple of 4, so the lanes come in pairs.
__device__ __forceinline__ unsigned pair_lanes(int b, int lane, int nb) {
    const int active = min(32, (nb - (b - 2 * lane)) / 2);
    return active >= 32 ? 0xffffffffu : ((1u << active) - 1u);
}

// A row's blocks b, b + 1 (b even) as four uint4, or zeros past the row end.
__device__ __forceinline__ void load_block_pair(const uint4* src, int b, int nb, uint4 (&q)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = b < nb ? __ldg(src + 2 * b + i) : make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ int64_t sf_byte(int64_t atile, int K, int b, int m) {
    return (atile * (K / 64) + (b >> 2)) * kSfChunkBytes + (m & 31) * 16 + (m >> 5) * 4 + (b & 3);
}

// tb[g] for g <= E from the group offsets (warp 0), then a block barrier.
// With no groups (offsets NULL, E = 0) tb[0] = 0.
__device__ __forceinline__ void tile_bases(const int32_t* __restrict__ offsets, int E, int* tb, int* offs) {
    if (offsets == nullptr) {
        if (threadIdx.x == 0) tb[0] = offs[0] = 0;
    } else if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int carry = 0;
        for (int base = 0; base <= E; base += 32) {
            const int g = base + lane;
            int c = 0;
            if (g <= E) offs[g] = offsets[g];
            if (g < E) c = max(0, (offsets[g + 1] - offsets[g] + BM - 1) / BM);  // never negative
            int v = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (g <= E) tb[g] = carry + v - c;  // exclusive
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
    }
    __syncthreads();
}

// x rows (one warp per token t): xq[t] and sx[t] for the shared expert (when
// has_shared), and for each chosen expert j the row r = inv[t k + j] of xp /
// sxp with its block scales, so x is read once.
__global__ void __launch_bounds__(256) quantize_x_nvfp4_kernel(const uint4* __restrict__ x, int H, int T, int k,
                                                               const int32_t* __restrict__ ids,
                                                               const int32_t* __restrict__ inv,
                                                               const int32_t* __restrict__ offsets, int E,
                                                               int has_shared, uint2* __restrict__ xq,
                                                               float* __restrict__ sx, uint2* __restrict__ xp,
                                                               float* __restrict__ sxp, uint8_t* __restrict__ sf,
                                                               int64_t sf_tiles, int* __restrict__ err) {
    __shared__ int tb[DWDP_MAX_EXPERTS + 1], offs[DWDP_MAX_EXPERTS + 1];
    // per warp: the token's destination rows (-1: flagged, skipped) and the
    // byte of block 0's scale in each one's A tile
    __shared__ int32_t dst_row[kQuantWarps][DWDP_MAX_TOPK];
    __shared__ int64_t dst_sf[kQuantWarps][DWDP_MAX_TOPK];
    tile_bases(offsets, E, tb, offs);
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int t = blockIdx.x * (blockDim.x >> 5) + wib;
    if (t >= T) return;
    const int nb = H / 16;
    const uint4* src = x + (int64_t)t * (H / 8);
    const float s = nvfp4_row_scale(src, nb, lane);
    const float d = 6.0f * s;
    const int64_t n_rows = (int64_t)T * k;
    if (lane < k) {
        const int64_t r = inv[(int64_t)t * k + lane];
        const int g = ids[(int64_t)t * k + lane];
        int32_t row = -1;
        int64_t base = 0;
        if (r < 0 || r >= n_rows || g < 0 || g >= E || r < offs[g] || r >= offs[g + 1] ||
            tb[g] + (r - offs[g]) / BM >= sf_tiles) {
            atomicOr(err, DERR_BAD_INDEX);
        } else {
            row = (int32_t)r;
            base = sf_byte(tb[g] + (r - offs[g]) / BM, H, 0, (int)((r - offs[g]) % BM));
            sxp[r] = s;
        }
        dst_row[wib][lane] = row;
        dst_sf[wib][lane] = base;
    }
    if (has_shared && lane == 0) sx[t] = s;
    const int64_t sh_at = tb[E] + t / BM;
    if (has_shared && sh_at >= sf_tiles) {
        if (lane == 0) atomicOr(err, DERR_BAD_INDEX);
        has_shared = 0;
    }
    const int64_t sh_sf = has_shared ? sf_byte(sh_at, H, 0, t % BM) : 0;
    __syncwarp();
    // two blocks per lane (nb is a multiple of 4): 16 bytes of codes and two
    // adjacent scale bytes per destination
    uint4* xq4 = reinterpret_cast<uint4*>(xq);
    uint4* xp4 = reinterpret_cast<uint4*>(xp);
    // the next pair's loads are issued before this pair is converted
    uint4 nxt[4];
    load_block_pair(src, 2 * lane, nb, nxt);
    for (int b = 2 * lane; b < nb; b += 64) {
        uint4 cur[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) cur[i] = nxt[i];
        load_block_pair(src, b + 64, nb, nxt);
        uint4 c;
        const uint32_t f = nvfp4_block_pair(cur, s, d, c) & 0xFFFFu;
        // lanes 2i and 2i+1 hold the four block scales of one 64-element K
        // step (one 4-byte word of each destination's chunk): the even lane
        // stores the word, so each destination gets one store per K step
        const uint32_t f_hi = __shfl_xor_sync(pair_lanes(b, lane, nb), f, 1);
        const bool even = (lane & 1) == 0;
        const uint32_t word = f | (f_hi << 16);
        const int64_t sf_off = (int64_t)(b >> 2) * kSfChunkBytes;  // block b's K step within a row's chunks
        if (has_shared) {
            xq4[(int64_t)t * (H / 32) + b / 2] = c;
            if (even) *reinterpret_cast<uint32_t*>(sf + sh_sf + sf_off) = word;
        }
        for (int j = 0; j < k; ++j) {
            const int32_t r = dst_row[wib][j];
            if (r < 0) continue;
            xp4[(int64_t)r * (H / 32) + b / 2] = c;
            if (even) *reinterpret_cast<uint32_t*>(sf + dst_sf[wib][j] + sf_off) = word;
        }
    }
}

__device__ __forceinline__ void quantize_a_row(const uint4* __restrict__ a, int I, int64_t r, int64_t rows_r,
                                               const int* offs, const int* tb, int E, uint2* __restrict__ aq,
                                               float* __restrict__ sa, uint8_t* __restrict__ sf, int64_t sf_tiles,
                                               int* __restrict__ err, int lane) {
    int64_t at;
    int m;
    if (r < rows_r) {
        // the group holding row r: the last g with offs[g] <= r (non-empty)
        int lo = 0, hi = E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (offs[mid] <= r) lo = mid;
            else hi = mid - 1;
        }
        if (r < offs[lo] || r >= offs[lo + 1]) {
            if (lane == 0 && err) atomicOr(err, DERR_BAD_INDEX);
            return;
        }
        at = tb[lo] + (r - offs[lo]) / BM;
        m = (int)((r - offs[lo]) % BM);
    } else {
        at = tb[E] + (r - rows_r) / BM;
        m = (int)((r - rows_r) % BM);
    }
    if (at >= sf_tiles) {
        if (lane == 0 && err) atomicOr(err, DERR_BAD_INDEX);
        return;
    }
    const int nb = I / 16;
    const uint4* src = a + r * (I / 8);
    const float s = nvfp4_row_scale(src, nb, lane);
    const float d = 6.0f * s;
    if (lane == 0) sa[r] = s;
    const int64_t base = sf_byte(at, I, 0, m);
    uint4* aq4 = reinterpret_cast<uint4*>(aq);
    uint4 nxt[4];
    load_block_pair(src, 2 * lane, nb, nxt);
    for (int b = 2 * lane; b < nb; b += 64) {  // two blocks per lane, next pair loaded ahead, as for x
        uint4 cur[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) cur[i] = nxt[i];
        load_block_pair(src, b + 64, nb, nxt);
        uint4 c;
        const uint32_t f = nvfp4_block_pair(cur, s, d, c) & 0xFFFFu;
        const uint32_t f_hi = __shfl_xor_sync(pair_lanes(b, lane, nb), f, 1);  // as in the x quantizer
        aq4[r * (I / 32) + b / 2] = c;
        if ((lane & 1) == 0) *reinterpret_cast<uint32_t*>(sf + base + (int64_t)(b >> 2) * kSfChunkBytes) = f | (f_hi << 16);
    }
}

// a rows (one warp per row r of rows_all = routed rows then shared rows).
// With rows_r = 0 and no groups this quantizes a plain [rows][I] matrix,
// row r landing in row r % 128 of tile r / 128.
__global__ void __launch_bounds__(256) quantize_a_nvfp4_kernel(const uint4* __restrict__ a, int I, int64_t rows_r,
                                                               int64_t rows_all, const int32_t* __restrict__ offsets,
                                                               int E, uint2* __restrict__ aq, float* __restrict__ sa,
                                                               uint8_t* __restrict__ sf, int64_t sf_tiles,
                                                               int* __restrict__ err) {
    __shared__ int tb[DWDP_MAX_EXPERTS + 1], offs[DWDP_MAX_EXPERTS + 1];
    tile_bases(offsets, E, tb, offs);
    const int lane = threadIdx.x & 31;
    // persistent: each warp takes rows warp, warp + all warps, ... (the tile
    // bases above are computed once per block)
    const int64_t n_warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows_all; r += n_warps)
        quantize_a_row(a, I, r, rows_r, offs, tb, E, aq, sa, sf, sf_tiles, err, lane);
}


}  // namespace

cudaError_t launch_quantize_x_nvfp4(const void* x, int H, int T, int k, const int32_t* ids, const int32_t* inv,
                                    const int32_t* offsets, int E, bool has_shared, void* xq, float* sx, void* xp,
                                    float* sxp, uint8_t* sf, int64_t sf_tiles, int* err, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const int warps = kQuantWarps;  // the kernel's per-warp destination tables assume it
    quantize_x_nvfp4_kernel<<<(T + warps - 1) / warps, 32 * warps, 0, s>>>(
        reinterpret_cast<const uint4*>(x), H, T, k, ids, inv, offsets, E, has_shared ? 1 : 0,
        reinterpret_cast<uint2*>(xq), sx, reinterpret_cast<uint2*>(xp), sxp, sf, sf_tiles, err);
    return cudaGetLastError();
}

// Blocks of quantize_a_nvfp4_kernel resident at once on the current device
// (its persistent grid), looked up once per device.
static int quantize_a_blocks() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quantize_a_nvfp4_kernel, 32 * kQuantWarps, 0) !=
                cudaSuccess)
            return 0;
        n = sms * (per_sm > 0 ? per_sm : 1);
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

cudaError_t launch_quantize_a_nvfp4(const void* act, int I, int64_t rows_r, int64_t rows_all, const int32_t* offsets,
                                    int E, void* aq, float* sa, uint8_t* sf, int64_t sf_tiles, int* err,
                                    cudaStream_t s) {
    if (rows_all <= 0) return cudaSuccess;
    const int warps = kQuantWarps;
    const int cap = quantize_a_blocks();
    if (cap <= 0) return cudaErrorInvalidDevice;
    const int64_t blocks = std::min<int64_t>((rows_all + warps - 1) / warps, cap);
    quantize_a_nvfp4_kernel<<<(unsigned)blocks, 32 * warps, 0, s>>>(
        reinterpret_cast<const uint4*>(act), I, rows_r, rows_all, offsets, E, reinterpret_cast<uint2*>(aq), sa, sf,
        sf_tiles, err);
    return cudaGetLastError();
}

cudaError_t launch_quantize_rows(const void* in, int64_t rows, int cols, void* codes, float* scale, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    const int warps = 8;
    quantize_rows_kernel<<<(unsigned)((rows + warps - 1) / warps), 32 * warps, 0, s>>>(
        reinterpret_cast<const uint4*>(in), rows, cols, reinterpret_cast<uint2*>(codes), scale);
    return cudaGetLastError();
}

cudaError_t launch_quantize_x_e4m3(const void* x, int H, const int32_t* inv, int T, int k, void* xq, float* sx,
                                   void* xp, float* sxp, int* err, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const int warps = 8;
    const dim3 grid((T + warps - 1) / warps), block(32 * warps);
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    uint2* qv = reinterpret_cast<uint2*>(xq);
    uint2* pv = reinterpret_cast<uint2*>(xp);
    switch (k) {
        case 2: quantize_x_e4m3_kernel<2><<<grid, block, 0, s>>>(xv, H / 8, inv, T, k, qv, sx, pv, sxp, err); break;
        case 4: quantize_x_e4m3_kernel<4><<<grid, block, 0, s>>>(xv, H / 8, inv, T, k, qv, sx, pv, sxp, err); break;
        case 8: quantize_x_e4m3_kernel<8><<<grid, block, 0, s>>>(xv, H / 8, inv, T, k, qv, sx, pv, sxp, err); break;
        default: quantize_x_e4m3_kernel<0><<<grid, block, 0, s>>>(xv, H / 8, inv, T, k, qv, sx, pv, sxp, err);
    }
    return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits, int parts, int64_t part_stride, const float* bias, int T, int E,
                        int k, int32_t* ids, float* w, float* z_out, int* err, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const int warps = 8;
    const dim3 grid((T + warps - 1) / warps), block(32 * warps);
    static_assert(kMaxPerLane == 32, "dispatch covers up to 32 logits per lane");
#define DWDP_TOPK(PER) \
    topk_kernel<PER><<<grid, block, 0, s>>>(logits, parts, part_stride, bias, T, E, k, ids, w, z_out, err)
    if (E <= 32) DWDP_TOPK(1);
    else if (E <= 64) DWDP_TOPK(2);
    else if (E <= 128) DWDP_TOPK(4);
    else if (E <= 256) DWDP_TOPK(8);
    else if (E <= 512) DWDP_TOPK(16);
    else DWDP_TOPK(32);
#undef DWDP_TOPK
    return cudaGetLastError();
}

cudaError_t launch_group(const int32_t* ids, int n, int E, int32_t* counts, int32_t* offsets,
                         int32_t* perm, int32_t* inv, cudaStream_t s) {
    count_kernel<<<E, 1024, 0, s>>>(ids, n, counts);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    place_kernel<<<E, 1024, 0, s>>>(ids, n, E, counts, offsets, perm, inv);
    return cudaGetLastError();
}

size_t group_chunked_scratch_bytes(int n, int E) {
    return sizeof(int32_t) * (size_t)((n + kChunk - 1) / kChunk) * (size_t)E;
}

cudaError_t launch_group_chunked(const int32_t* ids, int n, int E, int32_t* counts, int32_t* offsets, int32_t* perm,
                                 int32_t* inv, int32_t* scratch, cudaStream_t s) {
    const int n_chunks = (n + kChunk - 1) / kChunk;
    if (n_chunks == 0) {
        cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s);
        return e != cudaSuccess ? e : cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s);
    }
    chunk_count_kernel<<<n_chunks, kChunk, sizeof(int) * E, s>>>(ids, n, E, scratch);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    chunk_scan_kernel<<<1, 1024, 0, s>>>(scratch, n_chunks, E, counts, offsets);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    chunk_place_kernel<<<n_chunks, kChunk, 32 * E, s>>>(ids, n, E, scratch, perm, inv);
    return cudaGetLastError();
}

cudaError_t launch_gather(const void* x, int H, const int32_t* inv, int T, int k, void* xp, int* err,
                          cudaStream_t s) {
    return scatter_rows(x, H / 8, inv, T, k, xp, nullptr, nullptr, err, s);
}

cudaError_t launch_combine(const void* y, int H, const int32_t* inv, const float* w, int T, int k,
                           int64_t shared_row0, bool has_shared, void* out, int* err, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const int warps = 8;
    const dim3 grid((T + warps - 1) / warps), block(32 * warps);
    const uint4* yv = reinterpret_cast<const uint4*>(y);
    uint4* ov = reinterpret_cast<uint4*>(out);
    const int hs = has_shared ? 1 : 0;
    switch (k) {
        case 2: combine_kernel_k<2><<<grid, block, 0, s>>>(yv, H / 8, inv, w, T, shared_row0, hs, ov, err); break;
        case 4: combine_kernel_k<4><<<grid, block, 0, s>>>(yv, H / 8, inv, w, T, shared_row0, hs, ov, err); break;
        case 8: combine_kernel_k<8><<<grid, block, 0, s>>>(yv, H / 8, inv, w, T, shared_row0, hs, ov, err); break;
        default: combine_kernel<<<grid, block, 0, s>>>(yv, H / 8, inv, w, T, k, shared_row0, hs, ov, err);
    }
    return cudaGetLastError();
}

}  // namespace dwdp
