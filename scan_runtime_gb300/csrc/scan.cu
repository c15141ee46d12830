// scan.cu -- tier 1: per-channel first-order scans on sm_103a.
//
// FMA form   s_t = a_t * s_{t-1} + b_t                 ("SunnyNet 工程化实录" §2.1)
// gated form s_t = a_t * s_{t-1} + (1 - a_t) * u_t     ("SunnyNet 工程化实录" §2.1)
//
// Kernels:
//  * scan_seq_tma / scan_seq_ldg -- sequential in T.  Each thread carries its
//    channels' state through all T with one fused multiply-add per step, so the
//    result has the bits of the single-precision definition at every t and is
//    invariant under any segment split ("SunnyNet 工程化实录" §4).  The TMA
//    variant streams [32 x S1_NC] tiles of a and b through an S1_STAGES-deep
//    shared-memory ring fed by a producer warp; s_t leaves as coalesced
//    streaming stores.
//    The LDG variant serves layouts TMA cannot describe (N % 4 != 0 or
//    unaligned base pointers).
//  * scan_step -- the single step (T = 1) of every channel, the same
//    arithmetic, elementwise without the pipeline.
//  * the chunked look-back kernel lives in scan_lookback.cu.
#include <algorithm>
#include <cstdio>

#include "scan_common.cuh"

namespace sn {

// ============================================================ sequential (TMA)
namespace {
// Compile-time shape of the TMA kernel: S1_VEC channels per consumer lane
// (S1_NC = 32 * S1_VEC per CTA), S1_TS steps per stage, S1_STAGES stages.
#ifndef SN_SEQ_VEC
#define SN_SEQ_VEC 2
#endif
#ifndef SN_SEQ_STAGES
#define SN_SEQ_STAGES 4
#endif
constexpr int S1_VEC = SN_SEQ_VEC;
constexpr int S1_NC = 32 * S1_VEC;                // channels per CTA
constexpr int S1_TS = 32;                         // time steps per stage
constexpr int S1_STAGES = SN_SEQ_STAGES;
constexpr int S1_THREADS = 64;                    // warp 0 consumes, warp 1 produces
constexpr uint32_t S1_TILE = S1_TS * S1_NC;       // floats per tensor per stage
constexpr uint32_t S1_STAGE_BYTES = 2 * S1_TILE * 4;
static_assert(S1_VEC == 1 || S1_VEC == 2, "one or two channels per lane");
constexpr size_t S1_SMEM = S1_STAGES * S1_STAGE_BYTES + 2 * S1_STAGES * 8 + 16;

}  // namespace

template <bool GATED>
__global__ void __launch_bounds__(S1_THREADS)
scan_seq_tma(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
             int T, int N, const float* __restrict__ s0, float* __restrict__ s_final,
             float* __restrict__ s_out, SnDevStatus* st, uint64_t wait_ns) {
    extern __shared__ __align__(128) unsigned char smem[];
    float* tiles = reinterpret_cast<float*>(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S1_STAGES * S1_STAGE_BYTES);
    uint64_t* empty = full + S1_STAGES;
    volatile int* ctl = reinterpret_cast<volatile int*>(empty + S1_STAGES);  // [0] abort, [1] issued

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * S1_NC, bi = blockIdx.y;
    const int nst = (T + S1_TS - 1) / S1_TS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S1_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        ctl[0] = 0;
        ctl[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();

    int consumed = 0;
    if (warp == 1) {
        if (lane == 0) {
            int k = 0;
            for (; k < nst; ++k) {
                const int slot = k % S1_STAGES;
                if (k >= S1_STAGES) {
                    const uint32_t par = ((k / S1_STAGES) - 1) & 1;
                    const uint64_t t0 = global_ns();
                    bool ok = mbar_try_wait(&empty[slot], par);
                    while (!ok && !ctl[0]) {
                        if (global_ns() - t0 > wait_ns) break;
                        ok = mbar_try_wait(&empty[slot], par);
                    }
                    if (!ok) {
                        if (!ctl[0]) record_error(st, SN_E_TIMEOUT, (SN_K_SCAN_SEQ << 16) | 1);
                        ctl[0] = 1;
                        break;
                    }
                }
                mbar_arrive_expect_tx(&full[slot], S1_STAGE_BYTES);
                float* dst = tiles + slot * 2 * S1_TILE;
                tma_load_3d(dst, &map_a, &full[slot], n0, k * S1_TS, bi);
                tma_load_3d(dst + S1_TILE, &map_b, &full[slot], n0, k * S1_TS, bi);
            }
            ctl[1] = k;
        }
    } else {
        const int c = n0 + S1_VEC * lane;             // this lane's first channel
        const bool live = c < N;                      // N % 4 == 0 here, so a live lane owns all S1_VEC
        float x[S1_VEC];
#pragma unroll
        for (int v = 0; v < S1_VEC; ++v) x[v] = (s0 != nullptr && live) ? s0[(size_t)bi * N + c + v] : 0.0f;
        auto row = [&](const float* A, const float* Bv, float* out, int i) {
            float av[S1_VEC], bv[S1_VEC];
            if constexpr (S1_VEC == 2) {
                const float2 a2 = *reinterpret_cast<const float2*>(A + i * S1_NC);
                const float2 b2 = *reinterpret_cast<const float2*>(Bv + i * S1_NC);
                av[0] = a2.x; av[1] = a2.y; bv[0] = b2.x; bv[1] = b2.y;
            } else {
                av[0] = A[i * S1_NC];
                bv[0] = Bv[i * S1_NC];
            }
#pragma unroll
            for (int v = 0; v < S1_VEC; ++v) x[v] = __fmaf_rn(av[v], x[v], inj<GATED>(av[v], bv[v]));
            if (out) {
                if constexpr (S1_VEC == 2) st_cs(reinterpret_cast<float2*>(out + (size_t)i * N), make_float2(x[0], x[1]));
                else st_cs(out + (size_t)i * N, x[0]);
            }
        };
        for (int k = 0; k < nst; ++k) {
            const int slot = k % S1_STAGES;
            const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[slot], (k / S1_STAGES) & 1, wait_ns));
            if (!ok) {
                if (lane == 0) {
                    record_error(st, SN_E_TIMEOUT, (SN_K_SCAN_SEQ << 16) | 2);
                    ctl[0] = 1;
                }
                break;
            }
            const float* A = tiles + slot * 2 * S1_TILE + S1_VEC * lane;
            const float* Bv = A + S1_TILE;
            const int t0 = k * S1_TS;
            const int tn = min(S1_TS, T - t0);
            float* out = (s_out != nullptr && live) ? s_out + ((size_t)bi * T + t0) * N + c : nullptr;
            if (tn == S1_TS) {
#pragma unroll
                for (int i = 0; i < S1_TS; ++i) row(A, Bv, out, i);
            } else {
                for (int i = 0; i < tn; ++i) row(A, Bv, out, i);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            ++consumed;
        }
        if (s_final != nullptr && live && consumed == nst) {
#pragma unroll
            for (int v = 0; v < S1_VEC; ++v) s_final[(size_t)bi * N + c + v] = x[v];
        }
    }
    // After an abort, wait (bounded) for copies still in flight into this
    // CTA's shared memory before the CTA retires.
    __syncthreads();
    if (warp == 0 && lane == 0 && ctl[0]) {
        for (int k = consumed; k < ctl[1]; ++k)
            (void)mbar_wait(&full[k % S1_STAGES], (k / S1_STAGES) & 1, wait_ns);
    }
}

// ============================================================ sequential (LDG)
template <bool GATED>
__global__ void __launch_bounds__(128)
scan_seq_ldg(int T, int N, const float* __restrict__ a, const float* __restrict__ b,
             const float* __restrict__ s0, float* __restrict__ s_final, float* __restrict__ s_out) {
    const int c = blockIdx.x * 128 + threadIdx.x;
    const int bi = blockIdx.y;
    if (c >= N) return;
    const size_t base = (size_t)bi * T * N + c;
    float x = (s0 != nullptr) ? s0[(size_t)bi * N + c] : 0.0f;
    constexpr int U = 8;
    int t = 0;
    for (; t + U <= T; t += U) {
        float av[U], bv[U];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            av[i] = __ldcs(a + base + (size_t)(t + i) * N);
            bv[i] = __ldcs(b + base + (size_t)(t + i) * N);
        }
#pragma unroll
        for (int i = 0; i < U; ++i) {
            x = __fmaf_rn(av[i], x, inj<GATED>(av[i], bv[i]));
            if (s_out) __stcs(s_out + base + (size_t)(t + i) * N, x);
        }
    }
    for (; t < T; ++t) {
        const float av = a[base + (size_t)t * N], bv = b[base + (size_t)t * N];
        x = __fmaf_rn(av, x, inj<GATED>(av, bv));
        if (s_out) s_out[base + (size_t)t * N] = x;
    }
    if (s_final) s_final[(size_t)bi * N + c] = x;
}

// ============================================================ launchers

// ============================================================ single step (T = 1)
// One step of every channel, s = fma(a, s0, inj(a, b)), written to s_out and
// s_final: the sequential kernel's arithmetic for T = 1, without its
// pipeline (a single row would fill one stage of its ring).  Elementwise over
// the B * N channels, VEC channels per thread per iteration, one wave of
// grid-stride CTAs.
template <bool GATED, int VEC>
__global__ void __launch_bounds__(256) scan_step(int64_t n, const float* __restrict__ a,
                                                 const float* __restrict__ b, const float* s0, float* s_final,
                                                 float* __restrict__ s_out) {
    const int64_t nv = n / VEC;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += (int64_t)gridDim.x * blockDim.x) {
        float av[VEC], bv[VEC], sv[VEC];
        if constexpr (VEC == 4) {
            const float4 ta = __ldcs(reinterpret_cast<const float4*>(a) + i);
            const float4 tb = __ldcs(reinterpret_cast<const float4*>(b) + i);
            const float4 ts = s0 != nullptr ? *(reinterpret_cast<const float4*>(s0) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            av[0] = ta.x; av[1] = ta.y; av[2] = ta.z; av[3] = ta.w;
            bv[0] = tb.x; bv[1] = tb.y; bv[2] = tb.z; bv[3] = tb.w;
            sv[0] = ts.x; sv[1] = ts.y; sv[2] = ts.z; sv[3] = ts.w;
        } else {
            av[0] = __ldcs(a + i);
            bv[0] = __ldcs(b + i);
            sv[0] = s0 != nullptr ? s0[i] : 0.f;
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) sv[v] = __fmaf_rn(av[v], sv[v], inj<GATED>(av[v], bv[v]));
        if constexpr (VEC == 4) {
            const float4 r = make_float4(sv[0], sv[1], sv[2], sv[3]);
            if (s_out != nullptr) st_cs(reinterpret_cast<float4*>(s_out) + i, r);
            if (s_final != nullptr) st_cs(reinterpret_cast<float4*>(s_final) + i, r);
        } else {
            if (s_out != nullptr) st_cs(s_out + i, sv[0]);
            if (s_final != nullptr) st_cs(s_final + i, sv[0]);
        }
    }
}

static cudaError_t launch_scan_step(const ScanArgs& x, bool gated, cudaStream_t stream) {
    const int64_t n = (int64_t)x.B * x.N;
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const bool vec = n % 4 == 0 && al16(x.a) && al16(x.b) && al16(x.s0) && al16(x.s_final) && al16(x.s_out);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t items = vec ? n / 4 : n;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((items + 255) / 256, (int64_t)sms * 8));
    if (vec) {
        if (gated) scan_step<true, 4><<<grid, 256, 0, stream>>>(n, x.a, x.b, x.s0, x.s_final, x.s_out);
        else scan_step<false, 4><<<grid, 256, 0, stream>>>(n, x.a, x.b, x.s0, x.s_final, x.s_out);
    } else {
        if (gated) scan_step<true, 1><<<grid, 256, 0, stream>>>(n, x.a, x.b, x.s0, x.s_final, x.s_out);
        else scan_step<false, 1><<<grid, 256, 0, stream>>>(n, x.a, x.b, x.s0, x.s_final, x.s_out);
    }
    return cudaGetLastError();
}

cudaError_t launch_scan_sequential(const ScanArgs& x, bool gated, SnDevStatus* st, uint64_t wait_ns,
                                   cudaStream_t stream) {
    if (x.T == 1) return launch_scan_step(x, gated, stream);
    if (scan_tma_ok(x)) {
        CUtensorMap ma, mb;
        if (!make_scan_map(&ma, x.a, x.B, x.T, x.N, S1_NC, S1_TS) ||
            !make_scan_map(&mb, x.b, x.B, x.T, x.N, S1_NC, S1_TS))
            return cudaErrorInvalidValue;
        auto kern = gated ? scan_seq_tma<true> : scan_seq_tma<false>;
        cudaError_t e = set_smem_attr_once((const void*)kern, S1_SMEM);
        if (e != cudaSuccess) return e;
        dim3 grid((x.N + S1_NC - 1) / S1_NC, x.B);
        kern<<<grid, S1_THREADS, S1_SMEM, stream>>>(ma, mb, x.T, x.N, x.s0, x.s_final, x.s_out, st, wait_ns);
    } else {
        dim3 grid((x.N + 127) / 128, x.B);
        if (gated) scan_seq_ldg<true><<<grid, 128, 0, stream>>>(x.T, x.N, x.a, x.b, x.s0, x.s_final, x.s_out);
        else scan_seq_ldg<false><<<grid, 128, 0, stream>>>(x.T, x.N, x.a, x.b, x.s0, x.s_final, x.s_out);
    }
    return cudaGetLastError();
}

}  // namespace sn
