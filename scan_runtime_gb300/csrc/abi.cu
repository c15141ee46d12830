// abi.cu -- host side of the C ABI: version/caps/status, contexts, argument
// validation, kernel selection and error surfacing.  No arithmetic of the
// recurrences happens here; every step runs in the kernels.
//
// ABI style after "SunnyNet 工程化实录：一个 O(N) 架构如何长出自己的 C 推理运行时"
// §6 (stable C ABI: sn_ prefix, opaque handles, packed version, capability
// bits, int32 status codes and dimensions).
#include <cstdint>
#include <cmath>
#include <algorithm>
#include <cstring>
#include <initializer_list>
#include <map>
#include <mutex>
#include <utility>

#include <cudaTypedefs.h>

#include "sn_internal.h"

using namespace sn;

namespace {

constexpr int64_t kMaxElems = int64_t(1) << 40;   // sanity bound on one tensor (4 TB)
constexpr int kDefaultWaitUs = 1000000;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// True when the product of positive dimensions stays within kMaxElems.  Each
// factor is checked by division before it is multiplied in, so the product of
// int32 dimensions never overflows int64.
bool within_elems(std::initializer_list<int64_t> dims) {
    int64_t prod = 1;
    for (int64_t d : dims) {
        if (d <= 0 || d > kMaxElems / prod) return false;
        prod *= d;
    }
    return true;
}

bool overlaps(const void* p, int64_t pbytes, const void* q, int64_t qbytes) {
    if (p == nullptr || q == nullptr || pbytes <= 0 || qbytes <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p), a1 = a0 + (uintptr_t)pbytes;
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(q), b1 = b0 + (uintptr_t)qbytes;
    return a0 < b1 && b0 < a1;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct Buf {
    const void* p;
    int64_t bytes;
    bool out;
};

// Outputs may not overlap any other buffer, except the declared in-place pair.
bool any_bad_overlap(const Buf* bufs, int n, const void* inplace_in, const void* inplace_out) {
    for (int i = 0; i < n; ++i) {
        if (!bufs[i].out || bufs[i].p == nullptr) continue;
        for (int j = 0; j < n; ++j) {
            if (j == i || bufs[j].p == nullptr) continue;
            if (bufs[j].out && j < i) continue;   // each output pair checked once
            const bool pair_ok = (bufs[i].p == inplace_out && bufs[j].p == inplace_in && bufs[i].p == bufs[j].p &&
                                  bufs[i].bytes == bufs[j].bytes);
            if (!pair_ok && overlaps(bufs[i].p, bufs[i].bytes, bufs[j].p, bufs[j].bytes)) return true;
        }
    }
    return false;
}

sn_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SN_OK : SN_E_DEVICE; }

// Make the context's device current for the duration of a call.
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) return;
        ok = (prev == dev) || (cudaSetDevice(dev) == cudaSuccess);
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

uint64_t wait_ns(const SnCtx* c) { return (uint64_t)c->wait_limit_us * 1000ull; }

// The side streams and events of the pipelined chunked delta rule, created
// with the context so that no compute call creates CUDA objects.  Priorities:
// chain > preparation > output, so the serial chain starts as soon as SMs free
// up and the preparation that feeds it runs ahead of the outputs.
bool create_delta_pipe(SnCtx* c) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return false;
    const int mid = greatest < least - 1 ? greatest + 1 : greatest;
    cudaStream_t* sts[3] = {&c->pipe_chain, &c->pipe_prep, &c->pipe_out};
    const int prio[3] = {greatest, mid, least};
    int made_s = 0;
    for (; made_s < 3; ++made_s)
        if (cudaStreamCreateWithPriority(sts[made_s], cudaStreamNonBlocking, prio[made_s]) != cudaSuccess) break;
    int made_e = 0;
    if (made_s == 3)
        for (; made_e < 20; ++made_e)
            if (cudaEventCreateWithFlags(&c->pipe_ev[made_e], cudaEventDisableTiming) != cudaSuccess) break;
    if (made_e < 20) {
        for (int i = 0; i < made_e; ++i) cudaEventDestroy(c->pipe_ev[i]);
        for (int i = 0; i < made_s; ++i) cudaStreamDestroy(*sts[i]);
        return false;
    }
    c->pipe_ready = true;
    return true;
}

}  // namespace

namespace sn {
bool encode_tiled(CUtensorMap* map, int rank, const void* base, const uint64_t* dims,
                  const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128) {
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (g_encode == nullptr) return false;
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)rank, const_cast<void*>(base),
                          reinterpret_cast<const cuuint64_t*>(dims), reinterpret_cast<const cuuint64_t*>(strides_bytes),
                          reinterpret_cast<const cuuint32_t*>(box), estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
bool lookback_supported(const ScanArgs& x);

namespace {
std::mutex g_attr_mutex;
std::map<std::pair<const void*, int>, int> g_attr;     // (kernel, device) -> occupancy (0 = attr only)
}  // namespace

cudaError_t set_smem_attr_once(const void* kern, size_t bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    const auto key = std::make_pair(kern, dev);
    if (g_attr.count(key)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) g_attr[key] = 0;
    return e;
}

cudaError_t occupancy_once(const void* kern, int threads, size_t smem, int* out) {
    cudaError_t e = set_smem_attr_once(kern, smem);
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    int& occ = g_attr[std::make_pair(kern, dev)];
    if (occ == 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem);
        if (e != cudaSuccess) return e;
        if (occ < 1) return cudaErrorInvalidConfiguration;
    }
    *out = occ;
    return cudaSuccess;
}
}  // namespace sn

extern "C" {

uint32_t sn_abi_version(void) { return SN_ABI_VERSION; }

sn_status sn_abi_check(int32_t major) { return major == SN_ABI_VERSION_MAJOR ? SN_OK : SN_E_UNSUPPORTED; }

uint32_t sn_abi_caps(void) {
    return SN_CAP_SCAN_FMA | SN_CAP_SCAN_GATED | SN_CAP_RECUR_DIAG | SN_CAP_RECUR_DELTA | SN_CAP_RECUR_RWKV7 |
           SN_CAP_DECODE | SN_CAP_SCAN_LOOKBACK | SN_CAP_SCAN_BACKWARD | SN_CAP_RECUR_CHUNKED |
           SN_CAP_READOUT | SN_CAP_DELTA_CHUNKED;
}

const char* sn_status_str(sn_status s) {
    switch (s) {
        case SN_OK: return "ok";
        case SN_E_INVAL: return "invalid argument";
        case SN_E_NOMEM: return "workspace missing or too small";
        case SN_E_IO: return "i/o error";
        case SN_E_FORMAT: return "format error";
        case SN_E_UNSUPPORTED: return "unsupported (version, shape or device)";
        case SN_E_DEVICE: return "CUDA runtime error";
        case SN_E_TIMEOUT: return "bounded device-side wait ran out";
        case SN_E_RANGE: return "input value outside the range the kernel supports";
        default: return "unknown status";
    }
}

sn_status sn_ctx_create(int32_t device, SnCtx** out_ctx) {
    if (out_ctx == nullptr) return SN_E_INVAL;
    *out_ctx = nullptr;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess) return SN_E_DEVICE;
    if (device < 0 || device >= ndev) return SN_E_INVAL;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return SN_E_DEVICE;
    if (prop.major != 10 || prop.minor != 3) return SN_E_UNSUPPORTED;
    DeviceGuard g(device);
    if (!g.ok) return SN_E_DEVICE;
    SnCtx* c = new SnCtx();
    std::memset(c, 0, sizeof(SnCtx));
    c->device = device;
    c->sm_count = prop.multiProcessorCount;
    c->cc_major = prop.major;
    c->cc_minor = prop.minor;
    c->wait_limit_us = kDefaultWaitUs;
    c->ws_dirty = true;
    if (cudaMalloc(&c->dstatus, sizeof(SnDevStatus)) != cudaSuccess) {
        delete c;
        return SN_E_DEVICE;
    }
    if (cudaMemset(c->dstatus, 0, sizeof(SnDevStatus)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
        !create_delta_pipe(c)) {
        cudaFree(c->dstatus);
        delete c;
        return SN_E_DEVICE;
    }
    *out_ctx = c;
    return SN_OK;
}

void sn_ctx_free(SnCtx* ctx) {
    if (ctx == nullptr) return;
    DeviceGuard g(ctx->device);
    if (ctx->pipe_ready) {
        for (cudaStream_t st : {ctx->pipe_prep, ctx->pipe_chain, ctx->pipe_out}) {
            cudaStreamSynchronize(st);
            cudaStreamDestroy(st);
        }
        for (cudaEvent_t ev : ctx->pipe_ev) cudaEventDestroy(ev);
    }
    cudaFree(ctx->dstatus);
    delete ctx;
}

sn_status sn_ctx_set_workspace(SnCtx* ctx, void* dev_ptr, int64_t bytes) {
    if (ctx == nullptr || bytes < 0) return SN_E_INVAL;
    if (dev_ptr == nullptr || bytes == 0) {
        ctx->ws = nullptr;
        ctx->ws_bytes = 0;
        return SN_OK;
    }
    if (!aligned(dev_ptr, 256)) return SN_E_INVAL;
    ctx->ws = dev_ptr;
    ctx->ws_bytes = bytes;
    ctx->ws_dirty = true;
    return SN_OK;
}

int64_t sn_workspace_bytes(int32_t op, int32_t B, int32_t T, int32_t N) {
    if ((op != SN_OP_SCAN_FMA && op != SN_OP_SCAN_GATED) || !within_elems({B, T, N})) return -1;
    return std::max(lookback_ws_bytes(B, T, N), scan_fused_applies(T) ? scan_fused_ws_bytes(B, T, N) : 0);
}

sn_status sn_ctx_last_error(SnCtx* ctx) {
    if (ctx == nullptr) return SN_E_INVAL;
    DeviceGuard g(ctx->device);
    int err = 0;
    if (cudaMemcpy(&err, &ctx->dstatus->error, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SN_E_DEVICE;
    if (err != 0) {
        const int zero[2] = {0, 0};
        if (cudaMemcpy(ctx->dstatus, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return SN_E_DEVICE;
    }
    return err;
}

sn_status sn_ctx_set_option(SnCtx* ctx, int32_t key, int32_t value) {
    if (ctx == nullptr) return SN_E_INVAL;
    switch (key) {
        case SN_OPT_SCAN_KERNEL:
            if (value < SN_SCAN_KERNEL_AUTO || value > SN_SCAN_KERNEL_FUSED) return SN_E_INVAL;
            ctx->scan_kernel = value;
            return SN_OK;
        case SN_OPT_WAIT_LIMIT_US:
            if (value < 1) return SN_E_INVAL;
            ctx->wait_limit_us = value;
            return SN_OK;
        case SN_OPT_DEBUG_POISON:
            if (value != 0 && value != 1) return SN_E_INVAL;
            ctx->debug_poison = value;
            return SN_OK;
        case SN_OPT_RECUR_KERNEL:
            if (value != 0 && value != 1) return SN_E_INVAL;
            ctx->recur_kernel = value;
            return SN_OK;
        case SN_OPT_RECUR_TILE:
            if (value != 0 && value != 2 && value != 4 && value != 8) return SN_E_INVAL;
            ctx->recur_tile = value;
            return SN_OK;
        case SN_OPT_DELTA_SEGMENTS:
            if (value < 0 || value > DELTA_MAX_SEGMENTS) return SN_E_INVAL;
            ctx->delta_segments = value;
            return SN_OK;
        default: return SN_E_INVAL;
    }
}

sn_status sn_ctx_get_option(SnCtx* ctx, int32_t key, int32_t* value) {
    if (ctx == nullptr || value == nullptr) return SN_E_INVAL;
    switch (key) {
        case SN_OPT_SCAN_KERNEL: *value = ctx->scan_kernel; return SN_OK;
        case SN_OPT_WAIT_LIMIT_US: *value = ctx->wait_limit_us; return SN_OK;
        case SN_OPT_DEBUG_POISON: *value = ctx->debug_poison; return SN_OK;
        case SN_OPT_LOOKBACK_CHUNK: *value = LB_TC; return SN_OK;
        case SN_OPT_RECUR_KERNEL: *value = ctx->recur_kernel; return SN_OK;
        case SN_OPT_RECUR_TILE: *value = ctx->recur_tile; return SN_OK;
        case SN_OPT_DELTA_SEGMENTS: *value = ctx->delta_segments; return SN_OK;
        default: return SN_E_INVAL;
    }
}

// ------------------------------------------------------------------ scans
static sn_status scan_common(SnCtx* ctx, int32_t B, int32_t T, int32_t N, const float* a, const float* b,
                             const float* s0, float* s_final, float* s_out, void* stream, bool gated) {
    if (ctx == nullptr || a == nullptr || b == nullptr) return SN_E_INVAL;
    if (B <= 0 || T <= 0 || N <= 0) return SN_E_INVAL;
    if (!within_elems({B, T, N})) return SN_E_INVAL;
    const int64_t elems = (int64_t)B * T * N;
    const void* ptrs[5] = {a, b, s0, s_final, s_out};
    for (const void* p : ptrs)
        if (p != nullptr && !aligned(p, 4)) return SN_E_INVAL;
    const int64_t big = elems * 4, small = (int64_t)B * N * 4;
    const Buf bufs[5] = {{a, big, false}, {b, big, false}, {s0, small, false}, {s_final, small, true},
                         {s_out, big, true}};
    // s0 and s_final may be the same buffer (in-place continuation)
    if (any_bad_overlap(bufs, 5, s0, s_final)) return SN_E_INVAL;

    ScanArgs x{B, T, N, a, b, s0, s_final, s_out};
    int kernel = ctx->scan_kernel;
    const int64_t need = lookback_ws_bytes(B, T, N);
    const int64_t need_fused = scan_fused_applies(T) ? scan_fused_ws_bytes(B, T, N) : need;
    if (kernel == SN_SCAN_KERNEL_LOOKBACK || kernel == SN_SCAN_KERNEL_REDUCE_SCAN) {
        if (!lookback_supported(x)) return SN_E_UNSUPPORTED;
        if (ctx->ws == nullptr || ctx->ws_bytes < need) return SN_E_NOMEM;
    } else if (kernel == SN_SCAN_KERNEL_FUSED) {
        if (!lookback_supported(x)) return SN_E_UNSUPPORTED;
        if (ctx->ws == nullptr || ctx->ws_bytes < std::max(need, need_fused)) return SN_E_NOMEM;
    } else if (kernel == SN_SCAN_KERNEL_AUTO) {
        // The sequential kernel keeps the exact per-step bits and is HBM-bound
        // once there are enough channels; chunking along T pays only when the
        // channel count leaves most SMs idle and T is long.  Measured at 2^25
        // elements: a sequential CTA (64 channels) streams about 37 GB/s and
        // reduce-then-scan about 3.3 TB/s, so the two cross near 0.6 CTAs per
        // SM (64 CTAs: 0.156 against 0.123 ms; 128 CTAs: 0.084 against
        // 0.123 ms).  Of the two chunked paths (same bits), reduce-then-scan
        // measured faster wherever the channels are that few.
        const int64_t seq_ctas = (int64_t)B * ((N + 63) / 64);
        const bool few = 5 * seq_ctas < 3 * (int64_t)ctx->sm_count;
        kernel = (few && T >= 8 * LB_TC && lookback_supported(x) && ctx->ws != nullptr && ctx->ws_bytes >= need)
                     ? SN_SCAN_KERNEL_REDUCE_SCAN
                     : SN_SCAN_KERNEL_SEQUENTIAL;
        // the same results in one launch that reads a and b once, where the
        // workspace covers the fused path's words (it measured faster than
        // reduce-then-scan at one column of channel tiles and at eight)
        if (kernel == SN_SCAN_KERNEL_REDUCE_SCAN && scan_fused_applies(T) && ctx->ws_bytes >= need_fused)
            kernel = SN_SCAN_KERNEL_FUSED;
    }
    DeviceGuard g(ctx->device);
    if (!g.ok) return SN_E_DEVICE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (kernel == SN_SCAN_KERNEL_LOOKBACK || kernel == SN_SCAN_KERNEL_FUSED) {
        // The launch epoch wraps after 2^29 - 1 launches, when a tag could meet
        // a stale word of the same value: the tagged words are cleared long
        // before, every 2^24 tagged launches.
        if (++ctx->tagged_calls >= (uint64_t(1) << 24)) {
            ctx->ws_dirty = true;
            ctx->tagged_calls = 1;
        }
    }
    if (kernel == SN_SCAN_KERNEL_LOOKBACK) {
        const int64_t nflags = lookback_flag_count(B, T, N);
        if (ctx->ws_dirty || nflags != ctx->lb_last_flags) {
            // fresh flag and carry-word areas: zero them once, on the caller's
            // stream.  Between clears every launch rewrites all its flags and
            // carry words, and the launch epoch (kept on the device) differs
            // from the previous launch's.
            const int64_t cw_off = lookback_cw_offset(B, T, N);
            if (cudaMemsetAsync(ctx->ws, 0, (size_t)nflags * 4, s) != cudaSuccess ||
                cudaMemsetAsync(static_cast<char*>(ctx->ws) + cw_off, 0, (size_t)(need - cw_off), s) != cudaSuccess ||
                cudaMemsetAsync(&ctx->dstatus->abort_tag, 0, sizeof(unsigned int), s) != cudaSuccess)
                return SN_E_DEVICE;
            ctx->ws_dirty = false;
            ctx->lb_last_flags = nflags;
        }
        return from_cuda(launch_scan_lookback(x, gated, ctx->ws, ctx->debug_poison, ctx->dstatus, wait_ns(ctx),
                                              ctx->sm_count, s));
    }
    if (kernel == SN_SCAN_KERNEL_FUSED && !scan_fused_applies(T)) kernel = SN_SCAN_KERNEL_REDUCE_SCAN;   // same bits
    if (kernel == SN_SCAN_KERNEL_FUSED) {
        // carry words tagged with the look-back kernel's launch epoch, in other
        // places: cleared when the workspace, the geometry or the user changes
        const int64_t sig = -lookback_flag_count(B, T, N);
        if (ctx->ws_dirty || ctx->lb_last_flags != sig) {
            int64_t ta, tb;
            scan_fused_tag_area(B, T, N, &ta, &tb);
            if (cudaMemsetAsync(static_cast<char*>(ctx->ws) + ta, 0, (size_t)tb, s) != cudaSuccess ||
                cudaMemsetAsync(&ctx->dstatus->abort_tag, 0, sizeof(unsigned int), s) != cudaSuccess)
                return SN_E_DEVICE;
            ctx->ws_dirty = false;
            ctx->lb_last_flags = sig;
        }
        bool fell_back = false;
        const cudaError_t e = launch_scan_fused(x, gated, ctx->ws, ctx->debug_poison, ctx->dstatus, wait_ns(ctx),
                                                ctx->sm_count, s, &fell_back);
        if (fell_back) ctx->ws_dirty = true;   // reduce-then-scan's arrays overwrote the tagged words
        return from_cuda(e);
    }
    if (kernel == SN_SCAN_KERNEL_REDUCE_SCAN) {
        ctx->ws_dirty = true;   // its carries overwrite the look-back's carry words
        return from_cuda(launch_scan_reduce_scan(x, gated, ctx->ws, ctx->dstatus, wait_ns(ctx), ctx->sm_count, s));
    }
    return from_cuda(launch_scan_sequential(x, gated, ctx->dstatus, wait_ns(ctx), s));
}

sn_status sn_scan_fma(SnCtx* ctx, int32_t B, int32_t T, int32_t N, const float* a, const float* b,
                      const float* s0, float* s_final, float* s_out, void* stream) {
    return scan_common(ctx, B, T, N, a, b, s0, s_final, s_out, stream, false);
}

sn_status sn_scan_gated(SnCtx* ctx, int32_t B, int32_t T, int32_t N, const float* a, const float* u,
                        const float* s0, float* s_final, float* s_out, void* stream) {
    return scan_common(ctx, B, T, N, a, u, s0, s_final, s_out, stream, true);
}

// ------------------------------------------------------------------ host buffers
// Device staging of sn_scan_host: SN_HOST_SLOTS slots, each holding one chunk
// of `rows` batch rows: a, s0, then per form its input, states and final
// states, every part rounded up to 256 bytes.
namespace {
constexpr int SN_HOST_SLOTS = 3;
int64_t r256(int64_t x) { return (x + 255) / 256 * 256; }
int64_t host_slot_bytes(int64_t rows, int64_t T, int64_t N, int forms) {
    const int64_t big = r256(rows * T * N * 4), small = r256(rows * N * 4);
    return big + small + forms * (2 * big + small);
}
}  // namespace

int64_t sn_scan_host_staging_bytes(int32_t B, int32_t T, int32_t N, int32_t forms_mask, int32_t rows_per_chunk) {
    if (!within_elems({B, T, N}) || forms_mask < 1 || forms_mask > 3 || rows_per_chunk < 1) return -1;
    const int forms = (forms_mask & 1) + ((forms_mask >> 1) & 1);
    const int64_t rows = std::min<int64_t>(rows_per_chunk, B);
    return SN_HOST_SLOTS * host_slot_bytes(rows, T, N, forms);
}

sn_status sn_scan_host(SnCtx* ctx, int32_t B, int32_t T, int32_t N, int32_t rows_per_chunk, const float* a,
                       const float* b, const float* u, const float* s0, float* s_out_fma, float* s_final_fma,
                       float* s_out_gated, float* s_final_gated, void* staging, int64_t staging_bytes,
                       void* stream) {
    if (ctx == nullptr || a == nullptr || (b == nullptr && u == nullptr) || staging == nullptr) return SN_E_INVAL;
    if (B <= 0 || T <= 0 || N <= 0 || rows_per_chunk < 1 || !within_elems({B, T, N})) return SN_E_INVAL;
    const int mask = (b != nullptr ? 1 : 0) | (u != nullptr ? 2 : 0);
    if (staging_bytes < sn_scan_host_staging_bytes(B, T, N, mask, rows_per_chunk) || !aligned(staging, 256))
        return SN_E_INVAL;
    const void* ptrs[9] = {a, b, u, s0, s_out_fma, s_final_fma, s_out_gated, s_final_gated, staging};
    for (const void* p : ptrs)
        if (p != nullptr && !aligned(p, 4)) return SN_E_INVAL;
    const int64_t big = (int64_t)B * T * N * 4, small = (int64_t)B * N * 4;
    const Buf bufs[8] = {{a, big, false},          {b, big, false},           {u, big, false},
                         {s0, small, false},       {s_out_fma, big, true},    {s_final_fma, small, true},
                         {s_out_gated, big, true}, {s_final_gated, small, true}};
    if (any_bad_overlap(bufs, 8, nullptr, nullptr)) return SN_E_INVAL;
    if (!ctx->pipe_ready) return SN_E_DEVICE;
    DeviceGuard g(ctx->device);
    if (!g.ok) return SN_E_DEVICE;

    const int64_t R = std::min<int64_t>(rows_per_chunk, B);
    const int forms = (mask & 1) + ((mask >> 1) & 1);
    const int64_t slot_bytes = host_slot_bytes(R, T, N, forms);
    const int64_t bigR = r256(R * T * N * 4), smallR = r256(R * N * 4);
    cudaStream_t caller = reinterpret_cast<cudaStream_t>(stream);
    cudaStream_t st[SN_HOST_SLOTS] = {ctx->pipe_prep, ctx->pipe_chain, ctx->pipe_out};
    cudaEvent_t fork = ctx->pipe_ev[0];
    // the pipeline starts after the caller's earlier work on `stream`
    if (cudaEventRecord(fork, caller) != cudaSuccess) return SN_E_DEVICE;
    for (int i = 0; i < SN_HOST_SLOTS; ++i)
        if (cudaStreamWaitEvent(st[i], fork, 0) != cudaSuccess) return SN_E_DEVICE;
    const float* rhs[2] = {b, u};
    float* outs[2] = {s_out_fma, s_out_gated};
    float* fins[2] = {s_final_fma, s_final_gated};
    auto h2d = [](void* d, const void* h, int64_t n, cudaStream_t s) {
        return cudaMemcpyAsync(d, h, (size_t)n, cudaMemcpyHostToDevice, s) == cudaSuccess;
    };
    auto d2h = [](void* h, const void* d, int64_t n, cudaStream_t s) {
        return cudaMemcpyAsync(h, d, (size_t)n, cudaMemcpyDeviceToHost, s) == cudaSuccess;
    };
    // chunk ci on stream ci mod 3, in slot ci mod 3: the slot's previous chunk
    // (same stream) has been copied out before this one's copies land
    int ci = 0;
    for (int64_t b0 = 0; b0 < B; b0 += R, ++ci) {
        const int64_t r = std::min<int64_t>(R, B - b0);
        cudaStream_t s = st[ci % SN_HOST_SLOTS];
        char* slot = static_cast<char*>(staging) + (ci % SN_HOST_SLOTS) * slot_bytes;
        float* da = reinterpret_cast<float*>(slot);
        float* ds0 = reinterpret_cast<float*>(slot + bigR);
        const int64_t rb = r * T * N * 4, rs = r * N * 4;
        if (!h2d(da, a + b0 * T * N, rb, s)) return SN_E_DEVICE;
        if (s0 != nullptr && !h2d(ds0, s0 + b0 * N, rs, s)) return SN_E_DEVICE;
        char* p = slot + bigR + smallR;
        for (int f = 0; f < 2; ++f) {
            if (rhs[f] == nullptr) continue;
            float* din = reinterpret_cast<float*>(p);
            float* dout = reinterpret_cast<float*>(p + bigR);
            float* dfin = reinterpret_cast<float*>(p + 2 * bigR);
            p += 2 * bigR + smallR;
            if (!h2d(din, rhs[f] + b0 * T * N, rb, s)) return SN_E_DEVICE;
            // the sequential kernel: exact per-step bits, no workspace (chunks
            // in flight on different streams never share one)
            ScanArgs x{(int)r, T, N, da, din, s0 != nullptr ? ds0 : nullptr, dfin, dout};
            if (launch_scan_sequential(x, f == 1, ctx->dstatus, wait_ns(ctx), s) != cudaSuccess) return SN_E_DEVICE;
            if (outs[f] != nullptr && !d2h(outs[f] + b0 * T * N, dout, rb, s)) return SN_E_DEVICE;
            if (fins[f] != nullptr && !d2h(fins[f] + b0 * N, dfin, rs, s)) return SN_E_DEVICE;
        }
    }
    // the caller's later work on `stream` waits for every chunk
    for (int i = 0; i < SN_HOST_SLOTS; ++i) {
        if (cudaEventRecord(ctx->pipe_ev[1 + i], st[i]) != cudaSuccess ||
            cudaStreamWaitEvent(caller, ctx->pipe_ev[1 + i], 0) != cudaSuccess)
            return SN_E_DEVICE;
    }
    return SN_OK;
}

// ------------------------------------------------------------------ reverse scans
static sn_status scan_backward_common(SnCtx* ctx, BwdArgs& x, bool gated, void* stream) {
    if (ctx == nullptr || x.a == nullptr || x.s == nullptr || x.gs == nullptr || (gated && x.u == nullptr))
        return SN_E_INVAL;
    if (x.B <= 0 || x.T <= 0 || x.N <= 0) return SN_E_INVAL;
    if (!within_elems({x.B, x.T, x.N})) return SN_E_INVAL;
    const int64_t elems = (int64_t)x.B * x.T * x.N;
    const void* ptrs[9] = {x.a, x.u, x.s0, x.s, x.gs, x.gf, x.da, x.dbu, x.ds0};
    for (const void* p : ptrs)
        if (p != nullptr && !aligned(p, 4)) return SN_E_INVAL;
    const int64_t big = elems * 4, small = (int64_t)x.B * x.N * 4;
    const Buf bufs[9] = {{x.a, big, false}, {x.u, big, false},   {x.s0, small, false},
                         {x.s, big, false}, {x.gs, big, false},  {x.gf, small, false},
                         {x.da, big, true}, {x.dbu, big, true},  {x.ds0, small, true}};
    if (any_bad_overlap(bufs, 9, nullptr, nullptr)) return SN_E_INVAL;
    // kernel: the sequential reverse scan, or for few channels and long T the
    // chunked one (SN_OPT_SCAN_KERNEL: either chunked value forces it)
    const int64_t need = scan_backward_chunked_ws_bytes(x.B, x.T, x.N);
    bool chunked;
    if (ctx->scan_kernel == SN_SCAN_KERNEL_LOOKBACK || ctx->scan_kernel == SN_SCAN_KERNEL_REDUCE_SCAN) {
        if (!scan_backward_chunked_supported(x)) return SN_E_UNSUPPORTED;
        if (ctx->ws == nullptr || ctx->ws_bytes < need) return SN_E_NOMEM;
        chunked = true;
    } else if (ctx->scan_kernel == SN_SCAN_KERNEL_AUTO) {
        // A sequential reverse-scan CTA covers 32 channels.  Measured at 2^25
        // elements, the chunked path (about 0.165 ms) wins up to about one such
        // CTA per SM (128 CTAs: 0.208 ms sequential; 192 CTAs: 0.143 ms).
        const int64_t seq_ctas = (int64_t)x.B * ((x.N + 31) / 32);
        chunked = seq_ctas <= ctx->sm_count && x.T >= 8 * LB_TC && scan_backward_chunked_supported(x) &&
                  ctx->ws != nullptr && ctx->ws_bytes >= need;
    } else {
        chunked = false;
    }
    DeviceGuard g(ctx->device);
    if (!g.ok) return SN_E_DEVICE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (chunked) {
        ctx->ws_dirty = true;   // the carries overwrite the look-back flag area
        return from_cuda(launch_scan_backward_chunked(x, gated, ctx->ws, ctx->dstatus, wait_ns(ctx), ctx->sm_count, s));
    }
    return from_cuda(launch_scan_backward(x, gated, ctx->dstatus, wait_ns(ctx), s));
}

sn_status sn_scan_fma_backward(SnCtx* ctx, int32_t B, int32_t T, int32_t N, const float* a, const float* s0,
                               const float* s, const float* grad_s, const float* grad_final, float* grad_a,
                               float* grad_b, float* grad_s0, void* stream) {
    BwdArgs x{B, T, N, a, nullptr, s0, s, grad_s, grad_final, grad_a, grad_b, grad_s0};
    return scan_backward_common(ctx, x, false, stream);
}

sn_status sn_scan_gated_backward(SnCtx* ctx, int32_t B, int32_t T, int32_t N, const float* a, const float* u,
                                 const float* s0, const float* s, const float* grad_s, const float* grad_final,
                                 float* grad_a, float* grad_u, float* grad_s0, void* stream) {
    BwdArgs x{B, T, N, a, u, s0, s, grad_s, grad_final, grad_a, grad_u, grad_s0};
    return scan_backward_common(ctx, x, true, stream);
}

// ------------------------------------------------------------------ matrix recurrences
static bool head_dim_ok(int d) { return d == 64 || d == 128; }

// Argument checks shared by every matrix-recurrence entry point.
static sn_status recur_validate(SnCtx* ctx, const RecurArgs& x) {
    if (ctx == nullptr || x.q == nullptr || x.k == nullptr || x.v == nullptr || x.g == nullptr) return SN_E_INVAL;
    if (x.B <= 0 || x.T <= 0 || x.H <= 0 || x.G <= 0 || x.dk <= 0 || x.dv <= 0) return SN_E_INVAL;
    if (x.H % x.G != 0) return SN_E_INVAL;
    if (!head_dim_ok(x.dk) || !head_dim_ok(x.dv)) return SN_E_UNSUPPORTED;
    if (!within_elems({x.B, x.T, x.H, x.dk}) || !within_elems({x.B, x.T, x.H, x.dv}) ||
        !within_elems({x.B, x.H, x.dk, x.dv}))
        return SN_E_INVAL;
    const int64_t rows = (int64_t)x.B * x.T;
    const void* ptrs[7] = {x.q, x.k, x.v, x.g, x.S_in, x.S_out, x.o};
    for (const void* p : ptrs)
        if (p != nullptr && !aligned(p, 16)) return SN_E_INVAL;
    const int64_t qk = rows * x.G * x.dk * 4, vo = rows * x.H * x.dv * 4;
    const bool per_key = x.kind == RK_DIAG_KEY || x.kind == RK_RWKV7 || x.kind == RK_DIAG_KEY_GATED;
    const int64_t gb = per_key ? rows * x.H * x.dk * 4 : rows * x.H * 4;
    const int64_t sb = (int64_t)x.B * x.H * x.dk * x.dv * 4;
    const Buf bufs[7] = {{x.q, qk, false},   {x.k, qk, false},     {x.v, vo, false}, {x.g, gb, false},
                         {x.S_in, sb, false}, {x.S_out, sb, true}, {x.o, vo, true}};
    if (any_bad_overlap(bufs, 7, x.S_in, x.S_out)) return SN_E_INVAL;
    return SN_OK;
}

static sn_status recur_common(SnCtx* ctx, RecurArgs& x, void* stream) {
    const sn_status v = recur_validate(ctx, x);
    if (v != SN_OK) return v;
    DeviceGuard g(ctx->device);
    if (!g.ok) return SN_E_DEVICE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (x.T == 1 && ctx->recur_kernel == 0 && recur_decode_supported(x))
        return from_cuda(launch_recur_decode(x, ctx->dstatus, wait_ns(ctx), ctx->sm_count, s));
    if (!recur_seq_width_ok(x, ctx->sm_count, ctx->recur_tile)) return SN_E_INVAL;
    return from_cuda(launch_recur_sequence(x, ctx->dstatus, wait_ns(ctx), ctx->sm_count, ctx->recur_tile, s));
}

sn_status sn_recur_diag(SnCtx* ctx, int32_t B, int32_t T, int32_t H, int32_t G, int32_t dk, int32_t dv,
                        int32_t decay_kind, float scale, const float* q, const float* k, const float* v,
                        const float* d, const float* S_in, float* S_out, float* o, void* stream) {
    RecurArgs x{};
    switch (decay_kind) {
        case SN_DECAY_PER_KEY: x.kind = RK_DIAG_KEY; break;
        case SN_DECAY_PER_HEAD: x.kind = RK_DIAG_HEAD; break;
        case SN_DECAY_PER_KEY_GATED: x.kind = RK_DIAG_KEY_GATED; break;
        case SN_DECAY_PER_HEAD_GATED: x.kind = RK_DIAG_HEAD_GATED; break;
        default: return SN_E_INVAL;
    }
    x.B = B; x.T = T; x.H = H; x.G = G; x.dk = dk; x.dv = dv; x.scale = scale;
    x.q = q; x.k = k; x.v = v; x.g = d; x.S_in = S_in; x.S_out = S_out; x.o = o;
    x.state_transposed = false;
    return recur_common(ctx, x, stream);
}

sn_status sn_recur_delta(SnCtx* ctx, int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv, float scale,
                         const float* q, const float* k, const float* v, const float* beta, const float* S_in,
                         float* S_out, float* o, void* stream) {
    RecurArgs x{};
    x.kind = RK_DELTA;
    x.B = B; x.T = T; x.H = H; x.G = H; x.dk = dk; x.dv = dv; x.scale = scale;
    x.q = q; x.k = k; x.v = v; x.g = beta; x.S_in = S_in; x.S_out = S_out; x.o = o;
    x.state_transposed = false;
    return recur_common(ctx, x, stream);
}

sn_status sn_recur_rwkv7(SnCtx* ctx, int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv, const float* q,
                         const float* k, const float* v, const float* w, const float* S_in, float* S_out,
                         float* o, void* stream) {
    RecurArgs x{};
    x.kind = RK_RWKV7;
    x.B = B; x.T = T; x.H = H; x.G = H; x.dk = dk; x.dv = dv; x.scale = 1.0f;
    x.q = q; x.k = k; x.v = v; x.g = w; x.S_in = S_in; x.S_out = S_out; x.o = o;
    x.state_transposed = true;
    return recur_common(ctx, x, stream);
}

sn_status sn_recur_diag_chunked(SnCtx* ctx, int32_t B, int32_t T, int32_t H, int32_t G, int32_t dk, int32_t dv,
                                int32_t decay_kind, float scale, const float* q, const float* k, const float* v,
                                const float* d, const float* S_in, float* S_out, float* o, void* stream) {
    RecurArgs x{};
    switch (decay_kind) {
        case SN_DECAY_PER_KEY: x.kind = RK_DIAG_KEY; break;
        case SN_DECAY_PER_HEAD: x.kind = RK_DIAG_HEAD; break;
        case SN_DECAY_PER_KEY_GATED: x.kind = RK_DIAG_KEY_GATED; break;
        case SN_DECAY_PER_HEAD_GATED: x.kind = RK_DIAG_HEAD_GATED; break;
        default: return SN_E_INVAL;
    }
    x.B = B; x.T = T; x.H = H; x.G = G; x.dk = dk; x.dv = dv; x.scale = scale;
    x.q = q; x.k = k; x.v = v; x.g = d; x.S_in = S_in; x.S_out = S_out; x.o = o;
    x.state_transposed = false;
    const sn_status st = recur_validate(ctx, x);
    if (st != SN_OK) return st;
    if (!chunked_supported(x)) return SN_E_UNSUPPORTED;
    const int64_t need = chunked_ws_bytes(B, T, H, dk, dv);
    if (ctx->ws == nullptr || ctx->ws_bytes < need) return SN_E_NOMEM;
    DeviceGuard g(ctx->device);
    if (!g.ok) return SN_E_DEVICE;
    ctx->ws_dirty = true;   // the chunk states overwrite the look-back flag area
    return from_cuda(launch_recur_chunked(x, ctx->ws, ctx->dstatus, wait_ns(ctx), ctx->sm_count,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

sn_status sn_recur_delta_chunked(SnCtx* ctx, int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv, float scale,
                                 const float* q, const float* k, const float* v, const float* beta,
                                 const float* S_in, float* S_out, float* o, void* stream) {
    RecurArgs x{};
    x.kind = RK_DELTA;
    x.B = B; x.T = T; x.H = H; x.G = H; x.dk = dk; x.dv = dv; x.scale = scale;
    x.q = q; x.k = k; x.v = v; x.g = beta; x.S_in = S_in; x.S_out = S_out; x.o = o;
    x.state_transposed = false;
    const sn_status st = recur_validate(ctx, x);
    if (st != SN_OK) return st;
    if (!delta_chunked_supported(x)) return SN_E_UNSUPPORTED;
    const int64_t need = delta_chunked_ws_bytes(B, T, H, dk, dv);
    if (ctx->ws == nullptr || ctx->ws_bytes < need) return SN_E_NOMEM;
    DeviceGuard g(ctx->device);
    if (!g.ok) return SN_E_DEVICE;
    ctx->ws_dirty = true;   // the chunk tiles overwrite the look-back flag area
    const DeltaPipe pipe{ctx->pipe_prep, ctx->pipe_chain, ctx->pipe_out, ctx->pipe_ev, 20};
    return from_cuda(launch_delta_chunked(x, ctx->ws, ctx->dstatus, wait_ns(ctx), ctx->sm_count, ctx->delta_segments,
                                          ctx->debug_poison != 0, pipe, reinterpret_cast<cudaStream_t>(stream)));
}

int64_t sn_recur_delta_chunked_workspace_bytes(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv) {
    if (!within_elems({B, T, H, dk}) || !within_elems({B, T, H, dv}) || dk > 4096 || dv > 4096) return -1;
    return delta_chunked_ws_bytes(B, T, H, dk, dv);
}

// ------------------------------------------------------------------ readout epilogues
static sn_status readout_check(SnCtx* ctx, int32_t B, int32_t T, int32_t H, int32_t dv, const void* const* ptrs,
                               int nptr) {
    if (ctx == nullptr || B <= 0 || T <= 0 || H <= 0 || dv <= 0) return SN_E_INVAL;
    if (!within_elems({B, T, H, dv})) return SN_E_INVAL;
    if (dv != 64 && dv != 128) return SN_E_UNSUPPORTED;
    for (int i = 0; i < nptr; ++i)
        if (ptrs[i] != nullptr && !aligned(ptrs[i], 16)) return SN_E_INVAL;
    return SN_OK;
}

sn_status sn_readout_norm_gate(SnCtx* ctx, int32_t B, int32_t T, int32_t H, int32_t dv, const float* o,
                               const float* g, const float* w, float eps, float* y, void* stream) {
    if (o == nullptr || g == nullptr || y == nullptr || !(eps >= 0.0f) || !std::isfinite(eps)) return SN_E_INVAL;
    const void* ptrs[4] = {o, g, w, y};
    const sn_status st = readout_check(ctx, B, T, H, dv, ptrs, 4);
    if (st != SN_OK) return st;
    const int64_t rows = (int64_t)B * T * H, big = rows * dv * 4;
    const Buf bufs[4] = {{o, big, false}, {g, big, false}, {w, (int64_t)dv * 4, false}, {y, big, true}};
    if (any_bad_overlap(bufs, 4, o, y)) return SN_E_INVAL;
    DeviceGuard gd(ctx->device);
    if (!gd.ok) return SN_E_DEVICE;
    return from_cuda(launch_readout_norm_gate(rows, dv, o, g, w, eps, y, ctx->sm_count,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

sn_status sn_readout_dskip(SnCtx* ctx, int32_t B, int32_t T, int32_t H, int32_t dv, const float* o,
                           const float* x, const float* D, float* y, void* stream) {
    if (o == nullptr || x == nullptr || D == nullptr || y == nullptr) return SN_E_INVAL;
    const void* ptrs[3] = {o, x, y};
    const sn_status st = readout_check(ctx, B, T, H, dv, ptrs, 3);
    if (st != SN_OK) return st;
    if (!aligned(D, 4)) return SN_E_INVAL;
    const int64_t rows = (int64_t)B * T * H, big = rows * dv * 4;
    const Buf bufs[4] = {{o, big, false}, {x, big, false}, {D, (int64_t)H * 4, false}, {y, big, true}};
    if (any_bad_overlap(bufs, 4, o, y)) return SN_E_INVAL;
    DeviceGuard gd(ctx->device);
    if (!gd.ok) return SN_E_DEVICE;
    return from_cuda(launch_readout_dskip(rows, H, dv, o, x, D, y, ctx->sm_count,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

int64_t sn_recur_chunked_workspace_bytes(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv) {
    if (!within_elems({B, T, H, dk}) || !within_elems({B, T, H, dv}) || dk > 4096 || dv > 4096) return -1;
    return chunked_ws_bytes(B, T, H, dk, dv);
}

}  // extern "C"
