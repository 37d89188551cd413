// dwdp_abi.cu: the C ABI of libdwdp.so (declared in include/dwdp.h).
//
// Host side of the DWDP single-rank hot path: argument validation, the
// per-layer expert map and its per-expert (buffer, slot) table, TMA tensor
// maps, the double-buffer events, the round-robin prefetch copy plan, and the
// launches of the kernels in gemm.cu and route.cu.  Citations ([DWDP] §n) are
// to "DWDP: Distributed Weight Data Parallelism for High-Performance LLM
// Inference on NVL72".
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <tuple>
#include <memory>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "dwdp_internal.h"

using namespace dwdp;

namespace {

thread_local std::string g_last_error = "";

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct LayerMap {
    bool mapped = false;
    dwdp_pool local{};
    std::vector<dwdp_pool> peers;
    std::vector<int32_t> local_slot, peer_id, peer_slot, stage_slot;
    int n_remote = 0;
    const void* shared_w13 = nullptr;
    const void* shared_w2 = nullptr;
    bool has_local_map = false;
    CUtensorMap local13{}, local2{}, shared13{}, shared2{};
    std::vector<int2> bsrc;  // [E + n_shared]
    std::vector<float> scale13, scale2;  // E4M3 weight scales [E + n_shared] (empty until set)
    std::map<size_t, std::vector<dwdp_copy_slice>> plans;
    // copy plans as CUDA graphs of memcpy nodes, keyed by (chunk, stage, chains)
    std::map<std::tuple<size_t, int, int>, cudaGraphExec_t> graphs;
    void release() {
        for (auto& kv : graphs) cudaGraphExecDestroy(kv.second);
        graphs.clear();
    }
};

}  // namespace

namespace dwdp {

// Rows x K matrix, row-major: a 2-D map with a [128 rows x BK_BYTES] box and
// the swizzle of that width (the canonical K-major layout the MMA
// descriptors expect).
// E4M3 and NVFP4 codes are mapped as bytes.
bool encode_rows(CUtensorMap* m, const void* base, uint64_t rows, uint64_t K, int fmt) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || rows == 0) return false;
    const bool bytes = fmt != FMT_BF16;
    const uint64_t row_bytes = (uint64_t)operand_row_bytes((int64_t)K, fmt);
    cuuint64_t dims[2] = {bytes ? row_bytes : K, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)(bytes ? BK_BYTES : BK_BYTES / 2), BM};
    cuuint32_t es[2] = {1, 1};
    return fn(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, BK_BYTES == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A weight buffer [slots][rows][K]: a 3-D map, box [1 x 128 rows x BK_BYTES];
// slots are weight_slot_bytes apart (NVFP4: the codes of each slot, whose
// block scales follow them).
bool encode_slots(CUtensorMap* m, const void* base, uint64_t slots, uint64_t rows, uint64_t K, int fmt) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || rows == 0 || slots == 0) return false;
    const bool bytes = fmt != FMT_BF16;
    const uint64_t row_bytes = (uint64_t)operand_row_bytes((int64_t)K, fmt);
    cuuint64_t dims[3] = {bytes ? row_bytes : K, rows, slots};
    cuuint64_t strides[2] = {row_bytes, (uint64_t)weight_slot_bytes((int64_t)rows, (int64_t)K, fmt)};
    cuuint32_t box[3] = {(cuuint32_t)(bytes ? BK_BYTES : BK_BYTES / 2), BN / 2, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, BK_BYTES == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

void set_last_error(const char* msg) { g_last_error = msg; }

}  // namespace dwdp

struct dwdp_ctx {
    dwdp_config cfg{};
    int device = 0;
    int n_sms = 0;
    int fmt = FMT_BF16;  // expert weight format (weight_dtype)
    int n_stages = 2;
    void* stage13[DWDP_MAX_STAGES] = {};
    void* stage2[DWDP_MAX_STAGES] = {};
    CUtensorMap stage_map13[DWDP_MAX_STAGES]{}, stage_map2[DWDP_MAX_STAGES]{};
    cudaEvent_t ready[DWDP_MAX_STAGES] = {};
    cudaEvent_t freed[DWDP_MAX_STAGES] = {};
    int stage_layer[DWDP_MAX_STAGES] = {-1, -1, -1, -1};
    std::vector<LayerMap> layers;
    int* d_err = nullptr;
    cudaEvent_t phase[DWDP_PHASE_EVENTS] = {};  // the caller's (dwdp_set_phase_events)
    bool phases_on = false;
    std::string err;
    std::unique_ptr<GemmArgs> args;
    // frees what the context made, also after a dwdp_create that failed half-way
    ~dwdp_ctx() {
        for (int s = 0; s < DWDP_MAX_STAGES; ++s) {
            if (ready[s]) cudaEventDestroy(ready[s]);
            if (freed[s]) cudaEventDestroy(freed[s]);
        }
        for (LayerMap& m : layers) m.release();
        if (d_err) cudaFree(d_err);
    }
};

namespace {

int32_t fail(dwdp_ctx* ctx, int32_t code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (ctx) ctx->err = buf;
    g_last_error = buf;
    return code;
}

int32_t cuda_fail(dwdp_ctx* ctx, cudaError_t e, const char* what) {
    return fail(ctx, DWDP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define DWDP_CUDA(ctx, call)                                   \
    do {                                                       \
        cudaError_t e_ = (call);                               \
        if (e_ != cudaSuccess) return cuda_fail(ctx, e_, #call); \
    } while (0)

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Host-side NVTX range around one ABI call, named with its layer / stage /
// token count, so a timeline tool (nsys, ncu --nvtx) shows which call
// enqueued which kernels and copies; without a tool attached the push and
// pop do nothing.
struct NvtxRange {
    NvtxRange(const char* fmt, ...) {
        char buf[96];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        nvtxRangePushA(buf);
    }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

struct WsLayout {
    size_t logits = 0;  // route: fp32 [T][E] when the caller does not keep logits
    size_t group = 0;   // route: scratch of the chunked grouping
    // moe offsets: gathered rows xp, activations a, expert outputs y; E4M3
    // and NVFP4 contexts also keep x's codes/scales (xq, sx), xp's scales
    // (sxp) and a's codes/scales (aq, sa); NVFP4 adds the block-scale chunks
    // of the two GEMMs' A tiles (sfx, sfa).
    size_t xp = 0, a = 0, y = 0, xq = 0, sx = 0, sxp = 0, aq = 0, sa = 0, sfx = 0, sfa = 0;
    int64_t sf_tiles = 0;  // A tiles sfx / sfa have room for
    size_t route_bytes = 0, moe_bytes = 0;
};

WsLayout ws_layout(const dwdp_config& c, int64_t T) {
    WsLayout L;
    const int64_t H = c.hidden, I = c.inter, E = c.n_experts, k = c.top_k, S = c.n_shared;
    const int fmt = c.weight_dtype;
    L.logits = 0;  // up to kRouterMaxSplit partial-sum planes of the router GEMM
    L.group = align_up((size_t)(kRouterMaxSplit * T * E * 4), 256);
    L.route_bytes = L.group + align_up(group_chunked_scratch_bytes((int)(T * k), (int)E), 256);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += align_up(bytes, 256);
        return at;
    };
    L.xp = take((size_t)(T * k * operand_row_bytes(H, fmt)));
    L.a = take((size_t)(T * (k + S) * I * 2));
    L.y = take((size_t)(T * (k + S) * H * 2));
    if (fmt != FMT_BF16) {
        L.xq = take((size_t)(T * operand_row_bytes(H, fmt)));
        L.sx = take((size_t)T * 4);
        L.sxp = take((size_t)(T * k) * 4);
        L.aq = take((size_t)(T * (k + S) * operand_row_bytes(I, fmt)));
        L.sa = take((size_t)(T * (k + S)) * 4);
    }
    if (fmt == FMT_NVFP4) {
        // A tiles: sum over experts of ceil(rows / 128) <= (T k + 127 E) / 128,
        // plus ceil(T / 128) shared tiles; a tile holds 128 x K / 16 = 8 K scales
        const int64_t tiles = (T * k + 127 * E) / BM + (T + BM - 1) / BM;
        L.sf_tiles = tiles;
        L.sfx = take((size_t)(tiles * H * 8));
        L.sfa = take((size_t)(tiles * I * 8));
    }
    L.moe_bytes = o;
    return L;
}

// The copy plan of [DWDP] §4.3.2 (see dwdp_plan_prefetch in dwdp.h for the
// exact order).  Returns false on an invalid map.
bool build_plan(int32_t E, int64_t H, int64_t I, int fmt, const int32_t* local_slot, const int32_t* peer_id,
                const int32_t* peer_slot, int32_t n_peers, size_t chunk,
                std::vector<dwdp_copy_slice>& plan, std::string& why) {
    plan.clear();
    if (chunk == 0) {
        why = "chunk_bytes must be positive";
        return false;
    }
    std::vector<int64_t> sslot(E, -1);
    int64_t r = 0;
    for (int32_t e = 0; e < E; ++e)
        if (local_slot[e] < 0) {
            if (!peer_id || peer_id[e] < 0 || peer_id[e] >= n_peers || !peer_slot || peer_slot[e] < 0) {
                why = "expert " + std::to_string(e) + " is neither resident nor on a valid peer slot";
                return false;
            }
            sslot[e] = r++;
        }
    const int64_t bytes[2] = {weight_slot_bytes(2 * I, H, fmt), weight_slot_bytes(H, I, fmt)};
    std::vector<std::vector<dwdp_copy_slice>> per(n_peers > 0 ? n_peers : 0);
    for (int32_t p = 0; p < n_peers; ++p) {
        std::vector<dwdp_copy_slice> regions;
        for (int t = 0; t < 2; ++t) {
            for (int32_t e = 0; e < E; ++e) {
                if (sslot[e] < 0 || peer_id[e] != p) continue;
                const int64_t src = (int64_t)peer_slot[e] * bytes[t], dst = sslot[e] * bytes[t];
                if (!regions.empty()) {
                    dwdp_copy_slice& last = regions.back();
                    if (last.tensor == t && last.src_offset + last.nbytes == src &&
                        last.dst_offset + last.nbytes == dst) {
                        last.nbytes += bytes[t];
                        continue;
                    }
                }
                regions.push_back(dwdp_copy_slice{p, t, src, dst, bytes[t]});
            }
        }
        for (const dwdp_copy_slice& reg : regions) {
            for (int64_t done = 0; done < reg.nbytes;) {
                const int64_t n = std::min<int64_t>((int64_t)chunk, reg.nbytes - done);
                per[p].push_back(dwdp_copy_slice{p, reg.tensor, reg.src_offset + done, reg.dst_offset + done, n});
                done += n;
            }
        }
    }
    for (size_t c = 0;; ++c) {
        bool any = false;
        for (int32_t p = 0; p < n_peers; ++p)
            if (c < per[p].size()) {
                plan.push_back(per[p][c]);
                any = true;
            }
        if (!any) break;
    }
    return true;
}

// Records phase event i on s when phase timing is on.
cudaError_t mark(dwdp_ctx* ctx, int i, cudaStream_t s) {
    return ctx->phases_on ? cudaEventRecord(ctx->phase[i], s) : cudaSuccess;
}

int32_t check_device_error_word(dwdp_ctx* ctx) {
    int h = 0;
    DWDP_CUDA(ctx, cudaDeviceSynchronize());
    DWDP_CUDA(ctx, cudaMemcpy(&h, ctx->d_err, sizeof h, cudaMemcpyDeviceToHost));
    if (h != 0) {
        DWDP_CUDA(ctx, cudaMemset(ctx->d_err, 0, sizeof(int)));
        return fail(ctx, DWDP_ERR_DEVICE_CHECK, "device check failed: error bits 0x%x", h);
    }
    return DWDP_OK;
}

}  // namespace

extern "C" {

int32_t dwdp_version(void) { return DWDP_ABI_VERSION; }

const char* dwdp_last_error(const dwdp_ctx* ctx) {
    return ctx ? ctx->err.c_str() : g_last_error.c_str();
}

int32_t dwdp_create(const dwdp_config* cfg, void* const stage_w13[], void* const stage_w2[],
                    dwdp_ctx** out) {
    if (!cfg || !out) return fail(nullptr, DWDP_ERR_INVALID_ARG, "cfg and out must not be NULL");
    *out = nullptr;
    const dwdp_config& c = *cfg;
    if (c.hidden <= 0 || c.inter <= 0 || c.n_experts <= 0 || c.top_k <= 0 || c.max_tokens < 0 ||
        c.n_layers <= 0 || c.stage_slots < 0 || c.n_shared < 0 ||
        (c.weight_dtype != DWDP_DTYPE_BF16 && c.weight_dtype != DWDP_DTYPE_E4M3 &&
         c.weight_dtype != DWDP_DTYPE_NVFP4))
        return fail(nullptr, DWDP_ERR_INVALID_ARG, "config has a non-positive size or an unknown weight_dtype");
    if (c.hidden % 64 || c.inter % 64)
        return fail(nullptr, DWDP_ERR_UNSUPPORTED, "hidden and inter must be multiples of 64");
    if (c.weight_dtype == DWDP_DTYPE_NVFP4 && (c.hidden % 256 || c.inter % 256))
        return fail(nullptr, DWDP_ERR_UNSUPPORTED, "NVFP4: hidden and inter must be multiples of 256");
    if (c.n_experts > DWDP_MAX_EXPERTS || c.top_k > DWDP_MAX_TOPK || c.top_k > c.n_experts ||
        c.n_shared > 1 || c.n_layers > DWDP_MAX_LAYERS)
        return fail(nullptr, DWDP_ERR_UNSUPPORTED, "E <= %d, k <= min(E, %d), n_shared <= 1, layers <= %d",
                    DWDP_MAX_EXPERTS, DWDP_MAX_TOPK, DWDP_MAX_LAYERS);
    if ((int64_t)c.max_tokens * (c.top_k + c.n_shared) >= (int64_t)1 << 31)
        return fail(nullptr, DWDP_ERR_UNSUPPORTED, "max_tokens * (k + n_shared) must stay below 2^31");
    if (c.flags & ~DWDP_FLAG_WIDE_EPILOGUE)
        return fail(nullptr, DWDP_ERR_INVALID_ARG, "unknown flags 0x%x", (unsigned)c.flags);
    const int n_stages = c.n_stages == 0 ? 2 : c.n_stages;
    if (n_stages < 1 || n_stages > DWDP_MAX_STAGES)
        return fail(nullptr, DWDP_ERR_INVALID_ARG, "n_stages must be 0 (= 2) or 1..%d", DWDP_MAX_STAGES);
    if (c.stage_slots > 0) {
        for (int s = 0; s < n_stages; ++s)
            if (!stage_w13 || !stage_w2 || !stage_w13[s] || !stage_w2[s] || !aligned16(stage_w13[s]) ||
                !aligned16(stage_w2[s]))
                return fail(nullptr, DWDP_ERR_INVALID_ARG, "stage buffers must be non-NULL, 16-byte aligned");
    }
    std::unique_ptr<dwdp_ctx> ctx(new dwdp_ctx());
    ctx->cfg = c;
    ctx->n_stages = n_stages;
    ctx->fmt = c.weight_dtype;
    ctx->args.reset(new GemmArgs());
    cudaError_t e = cudaGetDevice(&ctx->device);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaGetDevice");
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, ctx->device);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaGetDeviceProperties");
    if (prop.major != 10 || prop.minor != 3)
        return fail(nullptr, DWDP_ERR_UNSUPPORTED, "libdwdp is built for sm_103a; device is sm_%d%d",
                    prop.major, prop.minor);
    ctx->n_sms = prop.multiProcessorCount;
    if (!encode_fn()) return fail(nullptr, DWDP_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
    if (c.stage_slots > 0)
        for (int s = 0; s < n_stages; ++s)
            if (!is_device_memory_of(stage_w13[s], ctx->device) || !is_device_memory_of(stage_w2[s], ctx->device))
                return fail(nullptr, DWDP_ERR_INVALID_ARG,
                            "stage buffer %d must be device memory of the current device (%d)", s, ctx->device);
    for (int s = 0; s < n_stages; ++s) {
        e = cudaEventCreateWithFlags(&ctx->ready[s], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ctx->freed[s], cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaEventCreate");
    }
    e = cudaMalloc(&ctx->d_err, 256);
    if (e == cudaSuccess) e = cudaMemset(ctx->d_err, 0, 256);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "error word");
    if (c.stage_slots > 0) {
        for (int s = 0; s < n_stages; ++s) {
            ctx->stage13[s] = stage_w13[s];
            ctx->stage2[s] = stage_w2[s];
            if (!encode_slots(&ctx->stage_map13[s], stage_w13[s], c.stage_slots, 2ull * c.inter, c.hidden,
                              ctx->fmt) ||
                !encode_slots(&ctx->stage_map2[s], stage_w2[s], c.stage_slots, c.hidden, c.inter, ctx->fmt))
                return fail(nullptr, DWDP_ERR_CUDA, "tensor map for a stage buffer");
        }
    }
    ctx->layers.resize(c.n_layers);
    ctx->err = "";
    *out = ctx.release();
    return DWDP_OK;
}

void dwdp_destroy(dwdp_ctx* ctx) { delete ctx; }

size_t dwdp_workspace_bytes(const dwdp_ctx* ctx, int32_t T) {
    if (!ctx || T < 0) return 0;
    const WsLayout L = ws_layout(ctx->cfg, T);
    return std::max(L.route_bytes, L.moe_bytes);
}

int32_t dwdp_workspace_region(const dwdp_ctx* ctx, int32_t T, int32_t region, size_t* offset, size_t* bytes) {
    if (!ctx || T < 0 || !offset || !bytes)
        return fail(nullptr, DWDP_ERR_INVALID_ARG, "ctx, offset and bytes must not be NULL; T >= 0");
    const dwdp_config& c = ctx->cfg;
    const WsLayout L = ws_layout(c, T);
    const int64_t H = c.hidden, I = c.inter, k = c.top_k, S = c.n_shared;
    const int fmt = c.weight_dtype;
    const bool q = fmt != FMT_BF16, f4 = fmt == FMT_NVFP4;
    size_t o = 0, n = 0;
    switch (region) {
        case DWDP_WS_XP: o = L.xp; n = (size_t)(T * k * operand_row_bytes(H, fmt)); break;
        case DWDP_WS_A: o = L.a; n = (size_t)(T * (k + S) * I * 2); break;
        case DWDP_WS_Y: o = L.y; n = (size_t)(T * (k + S) * H * 2); break;
        case DWDP_WS_XQ: o = L.xq; n = q ? (size_t)(T * operand_row_bytes(H, fmt)) : 0; break;
        case DWDP_WS_SX: o = L.sx; n = q ? (size_t)T * 4 : 0; break;
        case DWDP_WS_SXP: o = L.sxp; n = q ? (size_t)(T * k) * 4 : 0; break;
        case DWDP_WS_AQ: o = L.aq; n = q ? (size_t)(T * (k + S) * operand_row_bytes(I, fmt)) : 0; break;
        case DWDP_WS_SA: o = L.sa; n = q ? (size_t)(T * (k + S)) * 4 : 0; break;
        case DWDP_WS_SFX: o = L.sfx; n = f4 ? (size_t)(L.sf_tiles * H * 8) : 0; break;
        case DWDP_WS_SFA: o = L.sfa; n = f4 ? (size_t)(L.sf_tiles * I * 8) : 0; break;
        default: return fail(nullptr, DWDP_ERR_INVALID_ARG, "unknown workspace region %d", region);
    }
    *offset = n ? o : 0;
    *bytes = n;
    return DWDP_OK;
}

int32_t dwdp_set_expert_map(dwdp_ctx* ctx, int32_t layer, const dwdp_pool* local, const dwdp_pool* peers,
                            int32_t n_peers, const int32_t* local_slot, const int32_t* peer_id,
                            const int32_t* peer_slot, const void* shared_w13, const void* shared_w2) {
    if (!ctx) return fail(nullptr, DWDP_ERR_INVALID_ARG, "ctx is NULL");
    const dwdp_config& c = ctx->cfg;
    if (layer < 0 || layer >= c.n_layers) return fail(ctx, DWDP_ERR_INVALID_ARG, "layer %d out of range", layer);
    if (!local_slot) return fail(ctx, DWDP_ERR_INVALID_ARG, "local_slot must not be NULL");
    if (n_peers < 0 || n_peers > DWDP_MAX_PEERS || (n_peers > 0 && (!peers || !peer_id || !peer_slot)))
        return fail(ctx, DWDP_ERR_INVALID_ARG, "bad peer arguments");
    const int E = c.n_experts;
    bool any_local = false;
    for (int e = 0; e < E; ++e) {
        if (local_slot[e] >= 0) {
            any_local = true;
            if (!local || local_slot[e] >= local->n_slots)
                return fail(ctx, DWDP_ERR_INVALID_ARG, "expert %d: local slot %d outside the local pool", e,
                            local_slot[e]);
        } else {
            if (n_peers == 0 || peer_id[e] < 0 || peer_id[e] >= n_peers)
                return fail(ctx, DWDP_ERR_INVALID_ARG, "expert %d has no copy (not local, no valid peer)", e);
            if (peer_slot[e] < 0 || peer_slot[e] >= peers[peer_id[e]].n_slots)
                return fail(ctx, DWDP_ERR_INVALID_ARG, "expert %d: peer slot %d outside peer %d's pool", e,
                            peer_slot[e], peer_id[e]);
            const dwdp_pool& pp = peers[peer_id[e]];
            if (!pp.w13 || !pp.w2 || !aligned16(pp.w13) || !aligned16(pp.w2))
                return fail(ctx, DWDP_ERR_INVALID_ARG, "peer %d pool pointers must be non-NULL, 16-byte aligned",
                            peer_id[e]);
        }
    }
    if (any_local && (!local->w13 || !local->w2 || !aligned16(local->w13) || !aligned16(local->w2)))
        return fail(ctx, DWDP_ERR_INVALID_ARG, "local pool pointers must be non-NULL, 16-byte aligned");
    if (c.n_shared && (!shared_w13 || !shared_w2 || !aligned16(shared_w13) || !aligned16(shared_w2)))
        return fail(ctx, DWDP_ERR_INVALID_ARG, "the shared expert's weights are required");
    // the GEMM reads the local pool and the shared expert through tensor maps:
    // they must live in this GPU's memory (peer pools are only copied from)
    if (any_local && (!is_device_memory_of(local->w13, ctx->device) || !is_device_memory_of(local->w2, ctx->device)))
        return fail(ctx, DWDP_ERR_INVALID_ARG, "the local pool must be device memory of the context's device (%d)",
                    ctx->device);
    if (c.n_shared && (!is_device_memory_of(shared_w13, ctx->device) || !is_device_memory_of(shared_w2, ctx->device)))
        return fail(ctx, DWDP_ERR_INVALID_ARG,
                    "the shared expert must be device memory of the context's device (%d)", ctx->device);
    LayerMap m;
    m.local_slot.assign(local_slot, local_slot + E);
    m.peer_id.assign(E, -1);
    m.peer_slot.assign(E, -1);
    if (n_peers > 0) {
        m.peer_id.assign(peer_id, peer_id + E);
        m.peer_slot.assign(peer_slot, peer_slot + E);
        m.peers.assign(peers, peers + n_peers);
    }
    m.stage_slot.assign(E, -1);
    for (int e = 0; e < E; ++e)
        if (local_slot[e] < 0) m.stage_slot[e] = m.n_remote++;
    if (m.n_remote > c.stage_slots)
        return fail(ctx, DWDP_ERR_INVALID_ARG, "%d non-resident experts exceed the %d stage slots", m.n_remote,
                    c.stage_slots);
    if (any_local) {
        m.local = *local;
        if (!encode_slots(&m.local13, local->w13, local->n_slots, 2ull * c.inter, c.hidden, ctx->fmt) ||
            !encode_slots(&m.local2, local->w2, local->n_slots, c.hidden, c.inter, ctx->fmt))
            return fail(ctx, DWDP_ERR_CUDA, "tensor map for the local pool");
        m.has_local_map = true;
    }
    if (c.n_shared) {
        m.shared_w13 = shared_w13;
        m.shared_w2 = shared_w2;
        if (!encode_slots(&m.shared13, shared_w13, 1, 2ull * c.inter, c.hidden, ctx->fmt) ||
            !encode_slots(&m.shared2, shared_w2, 1, c.hidden, c.inter, ctx->fmt))
            return fail(ctx, DWDP_ERR_CUDA, "tensor map for the shared expert");
    }
    m.bsrc.resize(E + c.n_shared);
    for (int e = 0; e < E; ++e)
        m.bsrc[e] = (local_slot[e] >= 0) ? make_int2(0, local_slot[e]) : make_int2(1, m.stage_slot[e]);
    if (c.n_shared) m.bsrc[E] = make_int2(2, 0);
    m.mapped = true;
    m.scale13 = ctx->layers[layer].scale13;
    m.scale2 = ctx->layers[layer].scale2;
    ctx->layers[layer].release();
    ctx->layers[layer] = std::move(m);
    for (int s = 0; s < ctx->n_stages; ++s)
        if (ctx->stage_layer[s] == layer) ctx->stage_layer[s] = -1;  // staged bytes follow the old map
    return DWDP_OK;
}

int32_t dwdp_set_expert_scales(dwdp_ctx* ctx, int32_t layer, const float* w13_scale, const float* w2_scale,
                               float shared_w13_scale, float shared_w2_scale) {
    if (!ctx) return fail(nullptr, DWDP_ERR_INVALID_ARG, "ctx is NULL");
    const dwdp_config& c = ctx->cfg;
    if (c.weight_dtype == DWDP_DTYPE_BF16)
        return fail(ctx, DWDP_ERR_INVALID_ARG, "scales apply to E4M3 and NVFP4 contexts only");
    if (layer < 0 || layer >= c.n_layers) return fail(ctx, DWDP_ERR_INVALID_ARG, "layer %d out of range", layer);
    if (!w13_scale || !w2_scale) return fail(ctx, DWDP_ERR_INVALID_ARG, "scale arrays must not be NULL");
    std::vector<float> s13(w13_scale, w13_scale + c.n_experts), s2(w2_scale, w2_scale + c.n_experts);
    if (c.n_shared) {
        s13.push_back(shared_w13_scale);
        s2.push_back(shared_w2_scale);
    }
    for (size_t i = 0; i < s13.size(); ++i)
        if (!(s13[i] > 0.0f) || !(s2[i] > 0.0f) || !std::isfinite(s13[i]) || !std::isfinite(s2[i]))
            return fail(ctx, DWDP_ERR_INVALID_ARG, "scale %zu must be positive and finite", i);
    ctx->layers[layer].scale13 = std::move(s13);
    ctx->layers[layer].scale2 = std::move(s2);
    return DWDP_OK;
}

int32_t dwdp_plan_prefetch(int32_t n_experts, int32_t hidden, int32_t inter, int32_t weight_dtype,
                           const int32_t* local_slot,
                           const int32_t* peer_id, const int32_t* peer_slot, int32_t n_peers,
                           size_t chunk_bytes, dwdp_copy_slice* out, int64_t max_out, int64_t* n_out) {
    if (n_experts <= 0 || hidden <= 0 || inter <= 0 || weight_dtype < DWDP_DTYPE_BF16 ||
        weight_dtype > DWDP_DTYPE_NVFP4 || !local_slot ||
        !n_out || n_peers < 0 ||
        (max_out > 0 && !out))
        return fail(nullptr, DWDP_ERR_INVALID_ARG, "bad arguments to dwdp_plan_prefetch");
    std::vector<dwdp_copy_slice> plan;
    std::string why;
    if (!build_plan(n_experts, hidden, inter, weight_dtype, local_slot, peer_id, peer_slot, n_peers, chunk_bytes, plan,
                    why))
        return fail(nullptr, DWDP_ERR_INVALID_ARG, "%s", why.c_str());
    *n_out = (int64_t)plan.size();
    for (int64_t i = 0; i < max_out && i < (int64_t)plan.size(); ++i) out[i] = plan[i];
    return DWDP_OK;
}

int32_t dwdp_group_map(int32_t n_experts, int32_t n_ranks, int32_t rank, int32_t* local_slot, int32_t* peer_id,
                       int32_t* peer_slot) {
    if (n_experts <= 0 || n_ranks < 1 || n_ranks > DWDP_MAX_PEERS + 1 || n_ranks > n_experts || rank < 0 ||
        rank >= n_ranks || !local_slot || !peer_id || !peer_slot)
        return fail(nullptr, DWDP_ERR_INVALID_ARG, "need 1 <= n_ranks <= min(E, %d), 0 <= rank < n_ranks and "
                    "non-NULL arrays", DWDP_MAX_PEERS + 1);
    // contiguous blocks: rank q hosts experts [q E / N, (q + 1) E / N)
    auto first = [&](int64_t q) { return (int32_t)(q * n_experts / n_ranks); };
    int32_t home = 0;
    for (int32_t e = 0; e < n_experts; ++e) {
        while (e >= first(home + 1)) ++home;
        const int32_t slot = e - first(home);
        if (home == rank) {
            local_slot[e] = slot;
            peer_id[e] = -1;
            peer_slot[e] = -1;
        } else {
            local_slot[e] = -1;
            peer_id[e] = ((home - rank - 1) % n_ranks + n_ranks) % n_ranks;  // peer p is rank (rank + 1 + p) mod N
            peer_slot[e] = slot;
        }
    }
    return DWDP_OK;
}

int32_t dwdp_route(dwdp_ctx* ctx, const void* x, int32_t T, const void* w_router, const float* logit_bias,
                   const dwdp_route_out* out, void* ws, size_t ws_bytes, dwdp_stream_t stream) {
    const NvtxRange nvtx("dwdp_route T=%d", T);
    if (!ctx) return fail(nullptr, DWDP_ERR_INVALID_ARG, "ctx is NULL");
    const dwdp_config& c = ctx->cfg;
    if (T < 0 || T > c.max_tokens) return fail(ctx, DWDP_ERR_INVALID_ARG, "T=%d outside [0, max_tokens]", T);
    if (!out || !out->topk_ids || !out->topk_w || !out->counts || !out->offsets || !out->perm || !out->inv_perm)
        return fail(ctx, DWDP_ERR_INVALID_ARG, "route outputs must not be NULL (except logits)");
    if (!aligned16(out->topk_ids) || !aligned16(out->topk_w) || !aligned16(out->counts) ||
        !aligned16(out->offsets) || !aligned16(out->perm) || !aligned16(out->inv_perm) ||
        (out->logits && !aligned16(out->logits)) || (logit_bias && !aligned16(logit_bias)))
        return fail(ctx, DWDP_ERR_INVALID_ARG, "route pointers must be 16-byte aligned");
    if (T == 0) {
        DWDP_CUDA(ctx, cudaMemsetAsync(out->counts, 0, sizeof(int32_t) * c.n_experts, stream));
        DWDP_CUDA(ctx, cudaMemsetAsync(out->offsets, 0, sizeof(int32_t) * (c.n_experts + 1), stream));
        return DWDP_OK;
    }
    if (!x || !w_router || !aligned16(x) || !aligned16(w_router))
        return fail(ctx, DWDP_ERR_INVALID_ARG, "x and w_router must be non-NULL, 16-byte aligned");
    if (!is_device_memory_of(x, ctx->device) || !is_device_memory_of(w_router, ctx->device))
        return fail(ctx, DWDP_ERR_INVALID_ARG, "x and w_router must be device memory of the context's device (%d)",
                    ctx->device);
    const WsLayout L = ws_layout(c, T);
    if (!ws || ws_bytes < L.route_bytes || !aligned16(ws))
        return fail(ctx, DWDP_ERR_INVALID_ARG, "workspace too small (%zu < %zu) or unaligned", ws_bytes,
                    L.route_bytes);
    // K split: with fewer 128-token tiles than SMs the router GEMM's K is cut
    // into parts, each a tile writing its own fp32 plane; the top-k kernel
    // adds the planes in order (router_k_parts: deterministic per shape).
    const int parts = router_k_parts(T, c.n_experts, c.hidden, ctx->n_sms,
                                     (size_t)kRouterMaxSplit * T * c.n_experts * 4);
    float* planes = reinterpret_cast<float*>(static_cast<char*>(ws) + L.logits);
    float* logits = (out->logits && parts == 1) ? out->logits : planes;
    int32_t* group_scratch = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + L.group);
    DWDP_CUDA(ctx, mark(ctx, 0, stream));
    GemmArgs& a = *ctx->args;
    if (!encode_rows(&a.tmA[0], x, T, c.hidden) ||
        !encode_slots(&a.tmB[0], w_router, 1, c.n_experts, c.hidden))
        return fail(ctx, DWDP_ERR_CUDA, "tensor map for the router GEMM");
    a.tmA[1] = a.tmA[0];
    a.tmB[1] = a.tmB[2] = a.tmB[0];
    a.row_offsets = nullptr;
    a.n_routed = 0;
    a.shared_rows = T;
    a.shared_a_row = 0;
    a.shared_d_row = 0;
    a.K = c.hidden;
    a.N = c.n_experts;
    a.ldd = c.n_experts;
    a.d_rows = T;
    a.D = logits;
    a.col_bias = logit_bias;
    a.k_split = parts;
    a.split_stride = (int64_t)T * c.n_experts;
    a.err = ctx->d_err;
    a.bsrc[0] = make_int2(0, 0);
    DWDP_CUDA(ctx, launch_grouped_gemm(EPI_F32, FMT_BF16, a, ctx->n_sms, stream));
    DWDP_CUDA(ctx, launch_topk(logits, parts, (int64_t)T * c.n_experts, nullptr, T, c.n_experts, c.top_k,
                               out->topk_ids, out->topk_w, parts > 1 ? out->logits : nullptr, ctx->d_err,
                               stream));
    DWDP_CUDA(ctx, launch_group_chunked(out->topk_ids, T * c.top_k, c.n_experts, out->counts, out->offsets,
                                        out->perm, out->inv_perm, group_scratch, stream));
    DWDP_CUDA(ctx, mark(ctx, 1, stream));
    return DWDP_OK;
}

int32_t dwdp_prefetch_layer(dwdp_ctx* ctx, int32_t layer, int32_t stage, size_t chunk_bytes,
                            dwdp_stream_t const* copy_streams, int32_t n_copy_streams) {
    const NvtxRange nvtx("dwdp_prefetch_layer layer %d -> stage %d", layer, stage);
    if (!ctx) return fail(nullptr, DWDP_ERR_INVALID_ARG, "ctx is NULL");
    const dwdp_config& c = ctx->cfg;
    if (layer < 0 || layer >= c.n_layers) return fail(ctx, DWDP_ERR_INVALID_ARG, "layer %d out of range", layer);
    if (stage < 0 || stage >= ctx->n_stages)
        return fail(ctx, DWDP_ERR_INVALID_ARG, "stage %d outside [0, %d)", stage, ctx->n_stages);
    if (chunk_bytes == 0) return fail(ctx, DWDP_ERR_INVALID_ARG, "chunk_bytes must be positive");
    if (!copy_streams || n_copy_streams < 1 || n_copy_streams > DWDP_MAX_PEERS)
        return fail(ctx, DWDP_ERR_INVALID_ARG, "need 1..%d copy streams", DWDP_MAX_PEERS);
    LayerMap& m = ctx->layers[layer];
    if (!m.mapped) return fail(ctx, DWDP_ERR_NOT_MAPPED, "layer %d has no expert map", layer);
    auto it = m.plans.find(chunk_bytes);
    if (it == m.plans.end()) {
        std::vector<dwdp_copy_slice> plan;
        std::string why;
        if (!build_plan(c.n_experts, c.hidden, c.inter, ctx->fmt, m.local_slot.data(), m.peer_id.data(),
                        m.peer_slot.data(),
                        (int32_t)m.peers.size(), chunk_bytes, plan, why))
            return fail(ctx, DWDP_ERR_INVALID_ARG, "%s", why.c_str());
        it = m.plans.emplace(chunk_bytes, std::move(plan)).first;
    }
    // The plan as one CUDA graph of memcpy nodes (built once per chunk size,
    // stage and chain count): slices of peer p form chain p % n_copy_streams,
    // in plan order, so one launch replaces thousands of host calls and the
    // chains may run on separate copy engines.
    const auto key = std::make_tuple(chunk_bytes, (int)stage, (int)n_copy_streams);
    auto git = m.graphs.find(key);
    if (git == m.graphs.end() && !it->second.empty()) {
        cudaGraph_t g = nullptr;
        DWDP_CUDA(ctx, cudaGraphCreate(&g, 0));
        std::vector<cudaGraphNode_t> tail(n_copy_streams, nullptr);
        char* dst_base[2] = {static_cast<char*>(ctx->stage13[stage]), static_cast<char*>(ctx->stage2[stage])};
        cudaError_t e = cudaSuccess;
        for (const dwdp_copy_slice& sl : it->second) {
            const dwdp_pool& pp = m.peers[sl.peer];
            const char* src = static_cast<const char*>(sl.tensor == 0 ? pp.w13 : pp.w2) + sl.src_offset;
            cudaGraphNode_t& t = tail[sl.peer % n_copy_streams];
            cudaGraphNode_t node;
            e = cudaGraphAddMemcpyNode1D(&node, g, t ? &t : nullptr, t ? 1 : 0, dst_base[sl.tensor] + sl.dst_offset,
                                         src, (size_t)sl.nbytes, cudaMemcpyDefault);
            if (e != cudaSuccess) break;
            t = node;
        }
        cudaGraphExec_t exec = nullptr;
        if (e == cudaSuccess) e = cudaGraphInstantiate(&exec, g, 0);
        cudaGraphDestroy(g);
        if (e != cudaSuccess) return cuda_fail(ctx, e, "building the prefetch graph");
        git = m.graphs.emplace(key, exec).first;
    }
    // The stage may be overwritten only once the last layer that read it is done.
    DWDP_CUDA(ctx, cudaStreamWaitEvent(copy_streams[0], ctx->freed[stage], 0));
    if (git != m.graphs.end()) DWDP_CUDA(ctx, cudaGraphLaunch(git->second, copy_streams[0]));
    DWDP_CUDA(ctx, cudaEventRecord(ctx->ready[stage], copy_streams[0]));
    ctx->stage_layer[stage] = layer;
    return DWDP_OK;
}

int32_t dwdp_moe_layer(dwdp_ctx* ctx, int32_t layer, int32_t stage, const void* x, int32_t T,
                       const dwdp_route_out* route, void* out, void* ws, size_t ws_bytes, dwdp_stream_t stream) {
    const NvtxRange nvtx("dwdp_moe_layer layer %d stage %d T=%d", layer, stage, T);
    if (!ctx) return fail(nullptr, DWDP_ERR_INVALID_ARG, "ctx is NULL");
    const dwdp_config& c = ctx->cfg;
    if (layer < 0 || layer >= c.n_layers) return fail(ctx, DWDP_ERR_INVALID_ARG, "layer %d out of range", layer);
    if (T < 0 || T > c.max_tokens) return fail(ctx, DWDP_ERR_INVALID_ARG, "T=%d outside [0, max_tokens]", T);
    LayerMap& m = ctx->layers[layer];
    if (!m.mapped) return fail(ctx, DWDP_ERR_NOT_MAPPED, "layer %d has no expert map", layer);
    if (m.n_remote > 0) {
        if (stage < 0 || stage >= ctx->n_stages)
        return fail(ctx, DWDP_ERR_INVALID_ARG, "stage %d outside [0, %d)", stage, ctx->n_stages);
        if (ctx->stage_layer[stage] != layer)
            return fail(ctx, DWDP_ERR_NOT_MAPPED, "stage %d holds layer %d, not layer %d", stage,
                        ctx->stage_layer[stage], layer);
    }
    if (T == 0) return DWDP_OK;
    if (!route || !route->topk_w || !route->offsets || !route->perm || !route->inv_perm)
        return fail(ctx, DWDP_ERR_INVALID_ARG, "route outputs must not be NULL");
    if (!x || !out || !aligned16(x) || !aligned16(out) || !aligned16(route->offsets) ||
        !aligned16(route->perm) || !aligned16(route->inv_perm) || !aligned16(route->topk_w))
        return fail(ctx, DWDP_ERR_INVALID_ARG, "x, out and route pointers must be non-NULL, 16-byte aligned");
    const WsLayout L = ws_layout(c, T);
    if (!ws || ws_bytes < L.moe_bytes || !aligned16(ws))
        return fail(ctx, DWDP_ERR_INVALID_ARG, "workspace too small (%zu < %zu) or unaligned", ws_bytes, L.moe_bytes);
    // x and the workspace (xp, a and their codes) are read through tensor maps
    if (!is_device_memory_of(x, ctx->device) || !is_device_memory_of(ws, ctx->device))
        return fail(ctx, DWDP_ERR_INVALID_ARG, "x and ws must be device memory of the context's device (%d)",
                    ctx->device);
    const int64_t k = c.top_k, S = c.n_shared, H = c.hidden, I = c.inter, E = c.n_experts;
    const int64_t rows_r = (int64_t)T * k, rows_all = (int64_t)T * (k + S);
    const int fmt = ctx->fmt;
    const bool scaled = fmt != FMT_BF16;
    if (scaled && m.scale13.size() != m.bsrc.size())
        return fail(ctx, DWDP_ERR_NOT_MAPPED, "layer %d has no weight scales (dwdp_set_expert_scales)", layer);
    char* w = static_cast<char*>(ws);
    void* xp = w + L.xp;
    void* act = w + L.a;
    void* y = w + L.y;
    void* xq = w + L.xq;
    float* sx = reinterpret_cast<float*>(w + L.sx);
    float* sxp = reinterpret_cast<float*>(w + L.sxp);
    void* aq = w + L.aq;
    float* sa = reinterpret_cast<float*>(w + L.sa);
    uint8_t* sfx = reinterpret_cast<uint8_t*>(w + L.sfx);
    uint8_t* sfa = reinterpret_cast<uint8_t*>(w + L.sfa);

    // x goes into expert order first: only the GEMMs read the staged weights,
    // so the copy into the stage may still run meanwhile
    if (fmt == FMT_NVFP4) {
        // x rows to NVFP4 once per token, written to each chosen expert's row
        if (!route->topk_ids || !aligned16(route->topk_ids))
            return fail(ctx, DWDP_ERR_INVALID_ARG, "NVFP4 layers need route->topk_ids");
        DWDP_CUDA(ctx, launch_quantize_x_nvfp4(x, (int)H, (int)T, (int)k, route->topk_ids, route->inv_perm,
                                               route->offsets, (int)E, S > 0, xq, sx, xp, sxp, sfx, L.sf_tiles,
                                               ctx->d_err, stream));
    } else if (fmt == FMT_E4M3) {
        // x rows to E4M3 (per-token scales) once, written to xq and into
        // expert order in the same pass
        DWDP_CUDA(ctx, launch_quantize_x_e4m3(x, (int)H, route->inv_perm, (int)T, (int)k, xq, sx, xp, sxp, ctx->d_err,
                                              stream));
    } else {
        DWDP_CUDA(ctx, launch_gather(x, (int)H, route->inv_perm, (int)T, (int)k, xp, ctx->d_err, stream));
    }
    DWDP_CUDA(ctx, mark(ctx, 2, stream));
    if (m.n_remote > 0) DWDP_CUDA(ctx, cudaStreamWaitEvent(stream, ctx->ready[stage], 0));
    DWDP_CUDA(ctx, mark(ctx, 3, stream));

    GemmArgs& a = *ctx->args;
    // B buffers: 0 = local pool, 1 = the stage, 2 = the shared expert.  Slots
    // no group reads get a copy of a valid map.
    auto set_b = [&](const CUtensorMap& local, const CUtensorMap& stg, const CUtensorMap& shared) {
        const CUtensorMap* valid = m.has_local_map ? &local : (m.n_remote > 0 ? &stg : &shared);
        a.tmB[0] = m.has_local_map ? local : *valid;
        a.tmB[1] = m.n_remote > 0 ? stg : *valid;
        a.tmB[2] = S ? shared : *valid;
    };
    // NVFP4: where each buffer's slot 0 keeps its block scales (after its
    // rows x K / 2 bytes of codes); buffers no group reads get nullptr.
    auto set_bsf = [&](const void* local, const void* stg, const void* shared, int64_t rows, int64_t K) {
        const int64_t codes = rows * K / 2;
        auto at = [&](const void* base) { return base ? static_cast<const uint8_t*>(base) + codes : nullptr; };
        a.bsf[0] = m.has_local_map ? at(local) : nullptr;
        a.bsf[1] = m.n_remote > 0 ? at(stg) : nullptr;
        a.bsf[2] = S ? at(shared) : nullptr;
        a.b_slot_bytes = weight_slot_bytes(rows, K, fmt);
    };
    // G1: a = SiLU(xp W_gate) * (xp W_up); the shared group reads x directly
    // (E4M3: xp / x codes, dequantized in the epilogue by row scale * weight scale).
    if (!encode_rows(&a.tmA[0], xp, rows_r, H, fmt) || !encode_rows(&a.tmA[1], scaled ? xq : x, T, H, fmt))
        return fail(ctx, DWDP_ERR_CUDA, "tensor maps for the gate/up GEMM");
    a.row_scale[0] = sxp;
    a.row_scale[1] = sx;
    set_b(m.local13, ctx->stage_map13[m.n_remote > 0 ? stage : 0], m.shared13);
    a.sfa = sfx;
    a.sfa_tiles = L.sf_tiles;
    if (fmt == FMT_NVFP4)
        set_bsf(m.local.w13, ctx->stage13[m.n_remote > 0 ? stage : 0], m.shared_w13, 2 * I, H);
    a.row_offsets = route->offsets;
    a.n_routed = (int32_t)E;
    a.shared_rows = (int32_t)(T * S);
    a.shared_a_row = 0;
    a.shared_d_row = (int32_t)rows_r;
    a.K = (int32_t)H;
    a.N = (int32_t)I;
    a.ldd = I;
    a.d_rows = rows_all;
    a.D = act;
    a.col_bias = nullptr;
    a.k_split = 1;
    a.err = ctx->d_err;
    for (size_t g = 0; g < m.bsrc.size(); ++g) {
        a.bsrc[g] = m.bsrc[g];
        if (scaled) a.gscale[g] = m.scale13[g];
    }
    DWDP_CUDA(ctx, launch_grouped_gemm(EPI_SILU, fmt, a, ctx->n_sms, stream,
                                       (c.flags & DWDP_FLAG_WIDE_EPILOGUE) != 0));
    DWDP_CUDA(ctx, mark(ctx, 4, stream));
    // G2: y = a W_down (E4M3 / NVFP4: a's rows quantized first; this phase includes it).
    if (fmt == FMT_E4M3) DWDP_CUDA(ctx, launch_quantize_rows(act, rows_all, (int)I, aq, sa, stream));
    if (fmt == FMT_NVFP4)
        DWDP_CUDA(ctx, launch_quantize_a_nvfp4(act, (int)I, rows_r, rows_all, route->offsets, (int)E, aq, sa, sfa,
                                               L.sf_tiles, ctx->d_err, stream));
    if (!encode_rows(&a.tmA[0], scaled ? aq : act, rows_all, I, fmt))
        return fail(ctx, DWDP_ERR_CUDA, "tensor map for the down GEMM");
    a.tmA[1] = a.tmA[0];
    a.row_scale[0] = a.row_scale[1] = sa;
    if (scaled)
        for (size_t g = 0; g < m.bsrc.size(); ++g) a.gscale[g] = m.scale2[g];
    set_b(m.local2, ctx->stage_map2[m.n_remote > 0 ? stage : 0], m.shared2);
    a.sfa = sfa;
    if (fmt == FMT_NVFP4)
        set_bsf(m.local.w2, ctx->stage2[m.n_remote > 0 ? stage : 0], m.shared_w2, H, I);
    a.shared_a_row = (int32_t)rows_r;
    a.shared_d_row = (int32_t)rows_r;
    a.K = (int32_t)I;
    a.N = (int32_t)H;
    a.ldd = H;
    a.d_rows = rows_all;
    a.D = y;
    DWDP_CUDA(ctx, launch_grouped_gemm(EPI_BF16, fmt, a, ctx->n_sms, stream));
    DWDP_CUDA(ctx, mark(ctx, 5, stream));
    // The stage's weights have been read: the next prefetch into it may start.
    if (m.n_remote > 0) DWDP_CUDA(ctx, cudaEventRecord(ctx->freed[stage], stream));
    DWDP_CUDA(ctx, launch_combine(y, (int)H, route->inv_perm, route->topk_w, T, (int)k, rows_r, S > 0, out, ctx->d_err, stream));
    DWDP_CUDA(ctx, mark(ctx, 6, stream));
    return DWDP_OK;
}

int32_t dwdp_quantize_rows(int32_t weight_dtype, const void* x, int64_t rows, int32_t K, void* codes,
                           void* block_scales, float* row_scale, dwdp_stream_t stream) {
    if (weight_dtype != DWDP_DTYPE_E4M3 && weight_dtype != DWDP_DTYPE_NVFP4)
        return fail(nullptr, DWDP_ERR_INVALID_ARG, "weight_dtype must be E4M3 or NVFP4");
    if (rows < 0 || rows >= ((int64_t)1 << 31) || K <= 0 || K % 64)
        return fail(nullptr, DWDP_ERR_INVALID_ARG, "rows in [0, 2^31), K a positive multiple of 64");
    if (rows == 0) return DWDP_OK;
    if (!x || !codes || !row_scale || !aligned16(x) || !aligned16(codes) || !aligned16(row_scale) ||
        (weight_dtype == DWDP_DTYPE_NVFP4 && (!block_scales || !aligned16(block_scales))))
        return fail(nullptr, DWDP_ERR_INVALID_ARG, "pointers must be non-NULL and 16-byte aligned");
    cudaError_t e;
    if (weight_dtype == DWDP_DTYPE_E4M3) {
        e = launch_quantize_rows(x, rows, K, codes, row_scale, stream);
    } else {
        e = launch_quantize_a_nvfp4(x, K, 0, rows, nullptr, 0, codes, row_scale, static_cast<uint8_t*>(block_scales),
                                    (rows + BM - 1) / BM, nullptr, stream);
    }
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "dwdp_quantize_rows");
    return DWDP_OK;
}

int32_t dwdp_wait_stage(dwdp_ctx* ctx, int32_t stage, int32_t timeout_ms) {
    if (!ctx) return fail(nullptr, DWDP_ERR_INVALID_ARG, "ctx is NULL");
    if (stage < 0 || stage >= ctx->n_stages || timeout_ms < 0)
        return fail(ctx, DWDP_ERR_INVALID_ARG, "bad stage or timeout");
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        cudaError_t e = cudaEventQuery(ctx->ready[stage]);
        if (e == cudaSuccess) return DWDP_OK;
        if (e != cudaErrorNotReady) return cuda_fail(ctx, e, "cudaEventQuery");
        const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(std::chrono::steady_clock::now() - t0).count();
        if (ms >= timeout_ms) return fail(ctx, DWDP_ERR_TIMEOUT, "stage %d not ready after %d ms", stage, timeout_ms);
        std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
}

int32_t dwdp_stage_layer(const dwdp_ctx* ctx, int32_t stage) {
    if (!ctx || stage < 0 || stage >= ctx->n_stages) return -1;
    return ctx->stage_layer[stage];
}

int32_t dwdp_set_phase_events(dwdp_ctx* ctx, void* const* events, int32_t n_events) {
    if (!ctx) return fail(nullptr, DWDP_ERR_INVALID_ARG, "ctx is NULL");
    if (!events) {
        ctx->phases_on = false;
        return DWDP_OK;
    }
    if (n_events != DWDP_PHASE_EVENTS) return fail(ctx, DWDP_ERR_INVALID_ARG, "need %d events", DWDP_PHASE_EVENTS);
    // all checked before any is taken: a rejected call leaves the previous set
    for (int i = 0; i < DWDP_PHASE_EVENTS; ++i)
        if (!events[i]) return fail(ctx, DWDP_ERR_INVALID_ARG, "event %d is NULL", i);
    for (int i = 0; i < DWDP_PHASE_EVENTS; ++i) ctx->phase[i] = static_cast<cudaEvent_t>(events[i]);
    ctx->phases_on = true;
    return DWDP_OK;
}

int32_t dwdp_selftest_bounded_wait(dwdp_ctx* ctx, uint32_t limit_us, dwdp_stream_t stream) {
    if (!ctx) return fail(nullptr, DWDP_ERR_INVALID_ARG, "ctx is NULL");
    if (limit_us < 1 || limit_us > 1000000)
        return fail(ctx, DWDP_ERR_INVALID_ARG, "limit_us %u outside [1, 1000000]", limit_us);
    DWDP_CUDA(ctx, launch_bounded_wait_selftest(ctx->d_err, (uint64_t)limit_us * 1000ull, stream));
    return DWDP_OK;
}

int32_t dwdp_device_status(dwdp_ctx* ctx) {
    if (!ctx) return fail(nullptr, DWDP_ERR_INVALID_ARG, "ctx is NULL");
    return check_device_error_word(ctx);
}

int32_t dwdp_grouped_gemm(dwdp_ctx* ctx, int32_t epilogue, const void* a_ptr, int64_t a_rows, int32_t K,
                          int32_t N, const int32_t* row_offsets, int32_t G, const dwdp_pool* bufs, int32_t n_bufs,
                          const int32_t* buf_slot, void* d, dwdp_stream_t stream) {
    if (!ctx) return fail(nullptr, DWDP_ERR_INVALID_ARG, "ctx is NULL");
    if (epilogue < 0 || epilogue > 2) return fail(ctx, DWDP_ERR_INVALID_ARG, "epilogue must be 0, 1 or 2");
    if (G < 1 || G > DWDP_MAX_EXPERTS) return fail(ctx, DWDP_ERR_INVALID_ARG, "G must be in [1, %d]", DWDP_MAX_EXPERTS);
    if (K <= 0 || K % 64) return fail(ctx, DWDP_ERR_UNSUPPORTED, "K must be a positive multiple of 64");
    if (N <= 0 || (epilogue != 2 && N % 64)) return fail(ctx, DWDP_ERR_UNSUPPORTED, "N must be a positive multiple of 64");
    if (a_rows <= 0 || a_rows >= ((int64_t)1 << 31)) return fail(ctx, DWDP_ERR_INVALID_ARG, "a_rows out of range");
    if (!a_ptr || !d || !row_offsets || !bufs || !buf_slot || n_bufs < 1 || n_bufs > 3 || !aligned16(a_ptr) ||
        !aligned16(d) || !aligned16(row_offsets))
        return fail(ctx, DWDP_ERR_INVALID_ARG, "bad pointers or buffer count");
    GemmArgs& a = *ctx->args;
    const uint64_t brows = (epilogue == EPI_SILU) ? 2ull * N : (uint64_t)N;
    for (int b = 0; b < n_bufs; ++b) {
        if (!bufs[b].w13 || !aligned16(bufs[b].w13) || bufs[b].n_slots < 1)
            return fail(ctx, DWDP_ERR_INVALID_ARG, "buffer %d: base must be non-NULL, aligned, n_slots >= 1", b);
        if (!is_device_memory_of(bufs[b].w13, ctx->device))
            return fail(ctx, DWDP_ERR_INVALID_ARG, "buffer %d must be device memory of the context's device (%d)", b,
                        ctx->device);
        if (!encode_slots(&a.tmB[b], bufs[b].w13, bufs[b].n_slots, brows, K))
            return fail(ctx, DWDP_ERR_CUDA, "tensor map for buffer %d", b);
    }
    for (int b = n_bufs; b < 3; ++b) a.tmB[b] = a.tmB[0];
    for (int g = 0; g < G; ++g) {
        const int b = buf_slot[2 * g], s = buf_slot[2 * g + 1];
        if (b < 0 || b >= n_bufs || s < 0 || s >= bufs[b].n_slots)
            return fail(ctx, DWDP_ERR_INVALID_ARG, "group %d: (buffer %d, slot %d) out of range", g, b, s);
        a.bsrc[g] = make_int2(b, s);
    }
    if (!is_device_memory_of(a_ptr, ctx->device))
        return fail(ctx, DWDP_ERR_INVALID_ARG, "a must be device memory of the context's device (%d)", ctx->device);
    if (!encode_rows(&a.tmA[0], a_ptr, (uint64_t)a_rows, K)) return fail(ctx, DWDP_ERR_CUDA, "tensor map for A");
    a.tmA[1] = a.tmA[0];
    a.row_offsets = row_offsets;
    a.n_routed = G;
    a.shared_rows = 0;
    a.shared_a_row = 0;
    a.shared_d_row = 0;
    a.K = K;
    a.N = N;
    a.ldd = N;
    a.d_rows = a_rows;
    a.D = d;
    a.col_bias = nullptr;
    a.k_split = 1;
    a.err = ctx->d_err;
    DWDP_CUDA(ctx, launch_grouped_gemm(epilogue, FMT_BF16, a, ctx->n_sms, stream));
    return DWDP_OK;
}

}  // extern "C"
