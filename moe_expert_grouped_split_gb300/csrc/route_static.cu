// route_static.cu: dwdp_route_static, routing that allocates no device memory.
//
// Some callers cannot call cudaMalloc where they route tokens: a framework
// whose caching allocator owns all device memory and forbids raw
// allocations, a latency-critical serving loop that cannot afford the device
// synchronisation cudaMalloc may imply, or an embedded host that fixes its
// memory budget at start-up.  dwdp_route needs a context (whose creation
// allocates an error word) and a caller workspace for the fp32 logits; this
// entry point needs neither.  Its only scratch (the logits and an error
// word) is the file-scope device array below, which every GPU that loads
// this library holds until the process exits.
#include <cstdio>
#include <mutex>

#include "dwdp_internal.h"

namespace {

constexpr size_t kErrBytes = 256;  // error word, padded so the logits stay aligned
// the logits, plus as much again for the router GEMM's K-split partial sums
// (dwdp_route's split always fits on GPUs with up to 256 SMs)
constexpr size_t kPlaneBytes = 2 * (size_t)DWDP_STATIC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_route_scratch[kErrBytes + kPlaneBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
unsigned char* g_scratch_ptr[kMaxDevices] = {};  // device address of g_route_scratch, per device
int g_n_sms[kMaxDevices] = {};

int32_t fail_static(int32_t code, const char* msg) {
    dwdp::set_last_error(msg);  // read back with dwdp_last_error(NULL)
    return code;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Once per device, with that device current: the device address of the
// scratch array (a host-side use of the symbol itself would be a host
// stand-in, not a device address) and the SM count.
int32_t setup_device(int dev, unsigned char** scratch, int* n_sms) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess) return fail_static(DWDP_ERR_CUDA, cudaGetErrorString(e));
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail_static(DWDP_ERR_CUDA, cudaGetErrorString(e));
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3) return fail_static(DWDP_ERR_UNSUPPORTED, "device is not sm_103");
        g_n_sms[dev] = sms;
        g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
    }
    *scratch = g_scratch_ptr[dev];
    *n_sms = g_n_sms[dev];
    return DWDP_OK;
}

}  // namespace

extern "C" int32_t dwdp_route_static(const void* x, int32_t T, int32_t hidden, int32_t n_experts, int32_t top_k,
                                     const void* w_router, const float* logit_bias, const dwdp_route_out* out,
                                     dwdp_stream_t stream) {
    using namespace dwdp;
    if (hidden <= 0 || hidden % 64 || n_experts <= 0 || n_experts > DWDP_MAX_EXPERTS || top_k <= 0 ||
        top_k > n_experts || top_k > DWDP_MAX_TOPK)
        return fail_static(DWDP_ERR_UNSUPPORTED, "need H a positive multiple of 64, 1 <= k <= E <= 1024, k <= 32");
    if (T < 0 || (int64_t)T * top_k >= ((int64_t)1 << 31))
        return fail_static(DWDP_ERR_INVALID_ARG, "T out of range");
    if ((uint64_t)T * (uint64_t)n_experts * sizeof(float) > DWDP_STATIC_SCRATCH_BYTES)
        return fail_static(DWDP_ERR_INVALID_ARG,
                           "T * n_experts * 4 bytes of logits exceed DWDP_STATIC_SCRATCH_BYTES (16 MiB)");
    if (!out || !out->topk_ids || !out->topk_w || !out->counts || !out->offsets || !out->perm || !out->inv_perm)
        return fail_static(DWDP_ERR_INVALID_ARG, "route outputs must not be NULL (logits is ignored)");
    if (!aligned16(out->topk_ids) || !aligned16(out->topk_w) || !aligned16(out->counts) ||
        !aligned16(out->offsets) || !aligned16(out->perm) || !aligned16(out->inv_perm) ||
        (logit_bias && !aligned16(logit_bias)))
        return fail_static(DWDP_ERR_INVALID_ARG, "route pointers must be 16-byte aligned");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_static(DWDP_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail_static(DWDP_ERR_UNSUPPORTED, "device index too large");
    unsigned char* scratch = nullptr;
    int n_sms = 0;
    const int32_t rc = setup_device(dev, &scratch, &n_sms);
    if (rc != DWDP_OK) return rc;
    if (T == 0) {
        e = cudaMemsetAsync(out->counts, 0, sizeof(int32_t) * n_experts, stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(out->offsets, 0, sizeof(int32_t) * (n_experts + 1), stream);
        return e == cudaSuccess ? DWDP_OK : fail_static(DWDP_ERR_CUDA, cudaGetErrorString(e));
    }
    if (!x || !w_router || !aligned16(x) || !aligned16(w_router))
        return fail_static(DWDP_ERR_INVALID_ARG, "x and w_router must be non-NULL, 16-byte aligned");
    if (!is_device_memory_of(x, dev) || !is_device_memory_of(w_router, dev))
        return fail_static(DWDP_ERR_INVALID_ARG, "x and w_router must be device memory of the current device");
    int* err = reinterpret_cast<int*>(scratch);
    float* logits = reinterpret_cast<float*>(scratch + kErrBytes);
    // the error word keeps the previous call's bits: clear it on this stream
    e = cudaMemsetAsync(err, 0, sizeof(int), stream);
    if (e != cudaSuccess) return fail_static(DWDP_ERR_CUDA, cudaGetErrorString(e));

    static thread_local GemmArgs a;  // ~9 KB of launch parameters, host memory only
    if (!encode_rows(&a.tmA[0], x, T, hidden) || !encode_slots(&a.tmB[0], w_router, 1, n_experts, hidden))
        return fail_static(DWDP_ERR_CUDA, "tensor map for the router GEMM");
    a.tmA[1] = a.tmA[0];
    a.tmB[1] = a.tmB[2] = a.tmB[0];
    a.row_offsets = nullptr;
    a.n_routed = 0;
    a.shared_rows = T;
    a.shared_a_row = 0;
    a.shared_d_row = 0;
    a.K = hidden;
    a.N = n_experts;
    a.ldd = n_experts;
    a.d_rows = T;
    // the same K split as dwdp_route, so the same logits
    const int parts = router_k_parts(T, n_experts, hidden, n_sms, kPlaneBytes);
    a.D = logits;
    a.col_bias = logit_bias;
    a.k_split = parts;
    a.split_stride = (int64_t)T * n_experts;
    a.err = err;
    a.bsrc[0] = make_int2(0, 0);
    e = launch_grouped_gemm(EPI_F32, FMT_BF16, a, n_sms, stream);
    if (e == cudaSuccess)
        e = launch_topk(logits, parts, (int64_t)T * n_experts, nullptr, T, n_experts, top_k, out->topk_ids,
                        out->topk_w, nullptr, err, stream);
    if (e == cudaSuccess)
        e = launch_group(out->topk_ids, T * top_k, n_experts, out->counts, out->offsets, out->perm, out->inv_perm,
                         stream);
    return e == cudaSuccess ? DWDP_OK : fail_static(DWDP_ERR_CUDA, cudaGetErrorString(e));
}

extern "C" int32_t dwdp_route_static_status(dwdp_stream_t stream, int32_t* bits) {
    using namespace dwdp;
    if (bits) *bits = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_static(DWDP_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail_static(DWDP_ERR_UNSUPPORTED, "device index too large");
    unsigned char* scratch = nullptr;
    int n_sms = 0;
    const int32_t rc = setup_device(dev, &scratch, &n_sms);
    if (rc != DWDP_OK) return rc;
    int* err = reinterpret_cast<int*>(scratch);
    int h = 0;
    // read the word after everything already enqueued on the stream, then
    // clear it there, so the next call on this stream starts from zero
    e = cudaMemcpyAsync(&h, err, sizeof h, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && h != 0) {
        e = cudaMemsetAsync(err, 0, sizeof h, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    if (e != cudaSuccess) return fail_static(DWDP_ERR_CUDA, cudaGetErrorString(e));
    if (bits) *bits = h;
    if (h != 0) {
        char buf[160];
        snprintf(buf, sizeof buf, "dwdp_route_static: device check failed: error bits 0x%x%s", h,
                 (h & DERR_NONFINITE_LOGIT) ? " (a router logit is not finite)" : "");
        return fail_static(DWDP_ERR_DEVICE_CHECK, buf);
    }
    return DWDP_OK;
}
