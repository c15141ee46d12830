// scan.cu -- tier 1: per-channel first-order scans on sm_103a.
//
// FMA form   s_t = a_t * s_{t-1} + b_t                 ("SunnyNet 工程化实录" §2.1)
// gated form s_t = a_t * s_{t-1} + (1 - a_t) * u_t     ("SunnyNet 工程化实录" §2.1)
//
// Two kernels:
//  * scan_seq_tma / scan_seq_ldg -- sequential in T.  Each thread carries its
//    channels' state through all T with one fused multiply-add per step, so the
//    result has the bits of the single-precision definition at every t and is
//    invariant under any segment split ("SunnyNet 工程化实录" §4).  The TMA
//    variant streams [32 x 64] tiles of a and b through a 4-stage shared-memory
//    ring fed by a producer warp; s_t leaves as coalesced streaming stores.
//    The LDG variant serves layouts TMA cannot describe (N % 4 != 0 or
//    unaligned base pointers).
//  * scan_lookback -- chunked associative scan over (A, B) pairs for few
//    channels and long T.  Each tile is 32 channels x 128 steps: per-thread
//    folds over 4 steps, a warp-shuffle Kogge-Stone scan over the warp's 4
//    segments, a fixed-order fold across warps, and a decoupled look-back
//    across T chunks.  Carries are defined by the forward fold
//    C_k = fma(A_k, C_{k-1}, B_k), applied one chunk at a time whatever the
//    timing, so the result is deterministic and bit-exact under splits at
//    multiples of 128 steps.  Four tiles per CTA are in flight through a TMA
//    ring; the persistent grid is launched cooperatively so every CTA a tile
//    waits on is resident.
#include <algorithm>
#include <cstdio>

#include "ptx.cuh"
#include "sn_internal.h"

namespace sn {

// ============================================================ sequential (TMA)
namespace {
constexpr int S1_NC = 64;                         // channels per CTA
constexpr int S1_TS = 32;                         // time steps per stage
constexpr int S1_STAGES = 4;
constexpr int S1_THREADS = 64;                    // warp 0 consumes (2 ch/lane), warp 1 produces
constexpr uint32_t S1_TILE = S1_TS * S1_NC;       // floats per tensor per stage
constexpr uint32_t S1_STAGE_BYTES = 2 * S1_TILE * 4;
constexpr size_t S1_SMEM = S1_STAGES * S1_STAGE_BYTES + 2 * S1_STAGES * 8 + 16;

template <bool GATED>
__device__ __forceinline__ float inj(float a, float b) {
    if constexpr (GATED) return __fmul_rn(__fsub_rn(1.0f, a), b);
    else return b;
}
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
        const int c = n0 + 2 * lane;                  // this lane's two channels
        const bool live = c < N;                      // N % 4 == 0 here, so c + 1 < N too
        float x0 = 0.0f, x1 = 0.0f;
        if (s0 != nullptr && live) {
            x0 = s0[(size_t)bi * N + c];
            x1 = s0[(size_t)bi * N + c + 1];
        }
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
            const float* A = tiles + slot * 2 * S1_TILE + 2 * lane;
            const float* Bv = A + S1_TILE;
            const int t0 = k * S1_TS;
            const int tn = min(S1_TS, T - t0);
            float* out = (s_out != nullptr && live) ? s_out + ((size_t)bi * T + t0) * N + c : nullptr;
            if (tn == S1_TS) {
#pragma unroll
                for (int i = 0; i < S1_TS; ++i) {
                    const float2 av = *reinterpret_cast<const float2*>(A + i * S1_NC);
                    const float2 bv = *reinterpret_cast<const float2*>(Bv + i * S1_NC);
                    x0 = __fmaf_rn(av.x, x0, inj<GATED>(av.x, bv.x));
                    x1 = __fmaf_rn(av.y, x1, inj<GATED>(av.y, bv.y));
                    if (out) st_cs(reinterpret_cast<float2*>(out + (size_t)i * N), make_float2(x0, x1));
                }
            } else {
                for (int i = 0; i < tn; ++i) {
                    const float2 av = *reinterpret_cast<const float2*>(A + i * S1_NC);
                    const float2 bv = *reinterpret_cast<const float2*>(Bv + i * S1_NC);
                    x0 = __fmaf_rn(av.x, x0, inj<GATED>(av.x, bv.x));
                    x1 = __fmaf_rn(av.y, x1, inj<GATED>(av.y, bv.y));
                    if (out) st_cs(reinterpret_cast<float2*>(out + (size_t)i * N), make_float2(x0, x1));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            ++consumed;
        }
        if (s_final != nullptr && live && consumed == nst) {
            s_final[(size_t)bi * N + c] = x0;
            s_final[(size_t)bi * N + c + 1] = x1;
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

// ============================================================ look-back
namespace {
constexpr int LB_THREADS = 256;                   // 8 warps
constexpr int LB_SEG = LB_TC / 32;                // steps per thread segment
constexpr uint32_t LB_TILE = LB_TC * LB_NC;       // floats per tensor per tile
constexpr uint32_t LB_TILE_BYTES = 2 * LB_TILE * 4;
constexpr uint32_t LB_AGG = 1u, LB_INCL = 2u;
constexpr int LB_STAGES = 4;                      // tiles in flight per CTA
constexpr size_t LB_SMEM = LB_STAGES * LB_TILE_BYTES + LB_STAGES * 8 + 16;

__device__ __forceinline__ float4 f4mul(float4 x, float4 y) {
    return make_float4(__fmul_rn(x.x, y.x), __fmul_rn(x.y, y.y), __fmul_rn(x.z, y.z), __fmul_rn(x.w, y.w));
}
__device__ __forceinline__ float4 f4fma(float4 x, float4 y, float4 z) {
    return make_float4(__fmaf_rn(x.x, y.x, z.x), __fmaf_rn(x.y, y.y, z.y), __fmaf_rn(x.z, y.z, z.z),
                       __fmaf_rn(x.w, y.w, z.w));
}
__device__ __forceinline__ float4 f4shfl_up(float4 v, int d) {
    return make_float4(__shfl_up_sync(0xffffffffu, v.x, d), __shfl_up_sync(0xffffffffu, v.y, d),
                       __shfl_up_sync(0xffffffffu, v.z, d), __shfl_up_sync(0xffffffffu, v.w, d));
}
template <bool GATED>
__device__ __forceinline__ float4 inj4(float4 a, float4 u) {
    return make_float4(inj<GATED>(a.x, u.x), inj<GATED>(a.y, u.y), inj<GATED>(a.z, u.z), inj<GATED>(a.w, u.w));
}
}  // namespace

int64_t lookback_flag_count(int B, int T, int N) {
    const int64_t ncb = (N + LB_NC - 1) / LB_NC, nch = (T + LB_TC - 1) / LB_TC;
    return (int64_t)B * ncb * nch;
}

int64_t lookback_ws_bytes(int B, int T, int N) {
    const int64_t tiles = lookback_flag_count(B, T, N);
    const int64_t flag_bytes = ((tiles * 4 + 255) / 256) * 256;
    return flag_bytes + tiles * 3 * LB_NC * 4;
}

struct LookbackParams {
    int B, T, N, ncb, nbcb, nchunks, ntiles;
    const float* s0;
    float* s_final;
    float* s_out;
    uint32_t* flags;
    float* dA;
    float* dB;
    float* dC;
    uint32_t tag;        // (epoch << 2) written with each state
    uint32_t want;       // tag the waiters look for (differs from `tag` in poison mode)
    SnDevStatus* st;
    uint64_t wait_ns;
};

template <bool GATED>
__global__ void __launch_bounds__(LB_THREADS, 1)
scan_lookback(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
              const LookbackParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    float* bufs = reinterpret_cast<float*>(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + LB_STAGES * LB_TILE_BYTES);
    __shared__ float4 wA[8][8], wB[8][8];          // per-warp aggregates [warp][quad]
    __shared__ float carry[LB_NC], cfin[LB_NC];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = lane & 7, sub = lane >> 3;
    const int seg = warp * 4 + sub;                 // 0..31, rows [seg*LB_SEG, (seg+1)*LB_SEG)

    if (tid == 0) {
        for (int s = 0; s < LB_STAGES; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    auto tile_coords = [&](int ti, int& k, int& bi, int& cb) {
        k = ti / p.nbcb;
        const int r = ti - k * p.nbcb;
        bi = r / p.ncb;
        cb = r - bi * p.ncb;
    };
    auto issue = [&](int ti, int buf) {
        int k, bi, cb;
        tile_coords(ti, k, bi, cb);
        mbar_arrive_expect_tx(&full[buf], LB_TILE_BYTES);
        float* dst = bufs + buf * 2 * LB_TILE;
        tma_load_3d(dst, &map_a, &full[buf], cb * LB_NC, k * LB_TC, bi);
        tma_load_3d(dst + LB_TILE, &map_b, &full[buf], cb * LB_NC, k * LB_TC, bi);
    };

    int it = 0;
    if (tid == 0) {
        for (int s = 0; s < LB_STAGES - 1; ++s) {
            const int ti = blockIdx.x + s * gridDim.x;
            if (ti < p.ntiles) issue(ti, s);
        }
    }
    for (int ti = blockIdx.x; ti < p.ntiles; ti += gridDim.x, ++it) {
        const int buf = it % LB_STAGES;
        // refill the slot the previous iteration released
        const int ahead = ti + (LB_STAGES - 1) * (int)gridDim.x;
        if (tid == 0 && ahead < p.ntiles) issue(ahead, (it + LB_STAGES - 1) % LB_STAGES);
        int k, bi, cb;
        tile_coords(ti, k, bi, cb);
        const int t0 = k * LB_TC;
        const int n0 = cb * LB_NC;
        const int rows = min(LB_TC, p.T - t0);      // valid rows of this chunk

        if (!__syncthreads_and(mbar_wait(&full[buf], (it / LB_STAGES) & 1, p.wait_ns))) {
            // A copy never landed: report, wait (bounded) for this CTA's copies
            // still in flight, and retire the CTA.
            if (tid == 0) {
                record_error(p.st, SN_E_TIMEOUT, (SN_K_SCAN_LOOKBACK << 16) | 1);
                for (int j = 0; j < LB_STAGES; ++j)
                    if (ti + j * (int)gridDim.x < p.ntiles)
                        (void)mbar_wait(&full[(it + j) % LB_STAGES], ((it + j) / LB_STAGES) & 1, p.wait_ns);
            }
            return;
        }
        const float* sa = bufs + buf * 2 * LB_TILE;
        const float* sb = sa + LB_TILE;

        // ---- phase 1: fold this thread's LB_SEG steps of its 4 channels
        float4 A = make_float4(1.f, 1.f, 1.f, 1.f), Bc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < LB_SEG; ++i) {
            const int r = seg * LB_SEG + i;
            float4 av = *reinterpret_cast<const float4*>(sa + r * LB_NC + 4 * quad);
            float4 bv = inj4<GATED>(av, *reinterpret_cast<const float4*>(sb + r * LB_NC + 4 * quad));
            if (r >= rows) {                         // past T: identity step
                av = make_float4(1.f, 1.f, 1.f, 1.f);
                bv = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            Bc = f4fma(av, Bc, bv);
            A = f4mul(av, A);
        }
        // ---- phase 2a: inclusive scan over the warp's 4 segments (same quad)
#pragma unroll
        for (int d = 8; d < 32; d <<= 1) {
            const float4 Ap = f4shfl_up(A, d), Bp = f4shfl_up(Bc, d);
            if (lane >= d) {
                Bc = f4fma(A, Bp, Bc);
                A = f4mul(A, Ap);
            }
        }
        float4 eA = f4shfl_up(A, 8), eB = f4shfl_up(Bc, 8);   // exclusive within the warp
        if (sub == 0) {
            eA = make_float4(1.f, 1.f, 1.f, 1.f);
            eB = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (sub == 3) {
            wA[warp][quad] = A;
            wB[warp][quad] = Bc;
        }
        __syncthreads();
        // ---- phase 2b: fold the earlier warps' aggregates in warp order
        float4 PA = make_float4(1.f, 1.f, 1.f, 1.f), PB = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < warp; ++j) {
            PB = f4fma(wA[j][quad], PB, wB[j][quad]);
            PA = f4mul(wA[j][quad], PA);
        }
        const float4 EB = f4fma(eA, PB, eB);        // exclusive prefix of this segment
        const float4 EA = f4mul(eA, PA);

        // ---- phase 3: chunk aggregate and look-back (warp 0, lane = channel)
        if (warp == 0) {
            const int n = n0 + lane;
            float CA = 1.f, CB = 0.f;
            const float* pA = reinterpret_cast<const float*>(&wA[0][0]) + lane;
            const float* pB = reinterpret_cast<const float*>(&wB[0][0]) + lane;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                CB = __fmaf_rn(pA[j * 32], CB, pB[j * 32]);
                CA = __fmul_rn(pA[j * 32], CA);
            }
            const int base = bi * p.ncb + cb;
            float cin;
            if (k == 0) {
                cin = (p.s0 != nullptr && n < p.N) ? p.s0[(size_t)bi * p.N + n] : 0.f;
            } else {
                const size_t me = (size_t)ti * LB_NC + lane;
                p.dA[me] = CA;
                p.dB[me] = CB;
                __threadfence();
                __syncwarp();
                if (lane == 0) st_release_gpu(p.flags + ti, p.tag | LB_AGG);
                // windowed look-back: lane l inspects chunk (j - l)
                int j = k - 1;
                int m = -2;                           // chunk whose inclusive carry we take (-1 = s0)
                const uint64_t tstart = global_ns();
                bool timed_out = false;
                while (true) {
                    const int jl = j - lane;
                    uint32_t state = LB_INCL;         // chunks before 0 act as "inclusive = s0"
                    if (jl >= 0) {
                        const uint32_t f = ld_acquire_gpu(p.flags + (size_t)jl * p.nbcb + base);
                        state = ((f & ~3u) == p.want) ? (f & 3u) : 0u;
                    }
                    const uint32_t incl = __ballot_sync(0xffffffffu, state == LB_INCL);
                    const uint32_t none = __ballot_sync(0xffffffffu, state == 0u);
                    if (incl != 0u) {
                        const int l = __ffs(incl) - 1;
                        if ((none & ((1u << l) - 1u)) == 0u) {   // all nearer chunks published
                            m = j - l;
                            break;
                        }
                    } else if (none == 0u) {          // 32 aggregates: look further back
                        j -= 32;
                        continue;
                    }
                    // give up after the limit, or at once if another tile of this
                    // launch already gave up (its successors would only wait too)
                    if (global_ns() - tstart > p.wait_ns ||
                        *reinterpret_cast<volatile const uint32_t*>(&p.st->abort_tag) == p.tag) {
                        timed_out = true;
                        break;
                    }
                }
                __syncwarp();
                if (timed_out) {
                    if (lane == 0) {
                        record_error(p.st, SN_E_TIMEOUT, (SN_K_SCAN_LOOKBACK << 16) | 2);
                        atomicExch(&p.st->abort_tag, p.tag);
                    }
                    cin = 0.f;
                } else {
                    // forward fold from the inclusive carry at m through m+1 .. k-1
                    if (m < 0) cin = (p.s0 != nullptr && n < p.N) ? p.s0[(size_t)bi * p.N + n] : 0.f;
                    else cin = ld_relaxed_gpu(p.dC + ((size_t)m * p.nbcb + base) * LB_NC + lane);
                    for (int i = m + 1; i < k; ++i) {
                        const size_t o = ((size_t)i * p.nbcb + base) * LB_NC + lane;
                        cin = __fmaf_rn(ld_relaxed_gpu(p.dA + o), cin, ld_relaxed_gpu(p.dB + o));
                    }
                }
            }
            const float Ck = __fmaf_rn(CA, cin, CB);
            p.dC[(size_t)ti * LB_NC + lane] = Ck;
            __threadfence();
            __syncwarp();
            if (lane == 0) st_release_gpu(p.flags + ti, p.tag | LB_INCL);
            carry[lane] = cin;
            cfin[lane] = Ck;
            if (k == p.nchunks - 1 && p.s_final != nullptr && n < p.N) p.s_final[(size_t)bi * p.N + n] = Ck;
        }
        __syncthreads();
        // ---- phase 4: states of this thread's segment from its exclusive prefix
        if (p.s_out != nullptr && n0 + 4 * quad < p.N) {
            const float4 cc = *reinterpret_cast<const float4*>(&carry[4 * quad]);
            float4 s = f4fma(EA, cc, EB);
            float* out = p.s_out + ((size_t)bi * p.T + t0) * p.N + n0 + 4 * quad;
#pragma unroll
            for (int i = 0; i < LB_SEG; ++i) {
                const int r = seg * LB_SEG + i;
                if (r < rows) {
                    const float4 av = *reinterpret_cast<const float4*>(sa + r * LB_NC + 4 * quad);
                    const float4 bv = inj4<GATED>(av, *reinterpret_cast<const float4*>(sb + r * LB_NC + 4 * quad));
                    s = f4fma(av, s, bv);
                    if (r == rows - 1) s = *reinterpret_cast<const float4*>(&cfin[4 * quad]);
                    st_cs(reinterpret_cast<float4*>(out + (size_t)r * p.N), s);
                }
            }
        }
        __syncthreads();                              // buffer `buf` free for the next prefetch
    }
}

// ============================================================ launchers
static bool tma_ok(const ScanArgs& x) {
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    return (x.N % 4 == 0) && al16(x.a) && al16(x.b) && (x.s_out == nullptr || al16(x.s_out));
}

static bool make_scan_map(CUtensorMap* m, const float* base, int B, int T, int N, int box_n, int box_t) {
    const uint64_t dims[3] = {(uint64_t)N, (uint64_t)T, (uint64_t)B};
    const uint64_t strides[2] = {(uint64_t)N * 4, (uint64_t)T * N * 4};
    const uint32_t box[3] = {(uint32_t)box_n, (uint32_t)box_t, 1};
    return encode_tiled(m, 3, base, dims, strides, box);
}

cudaError_t launch_scan_sequential(const ScanArgs& x, bool gated, SnDevStatus* st, uint64_t wait_ns,
                                   cudaStream_t stream) {
    if (tma_ok(x)) {
        CUtensorMap ma, mb;
        if (!make_scan_map(&ma, x.a, x.B, x.T, x.N, S1_NC, S1_TS) ||
            !make_scan_map(&mb, x.b, x.B, x.T, x.N, S1_NC, S1_TS))
            return cudaErrorInvalidValue;
        auto kern = gated ? scan_seq_tma<true> : scan_seq_tma<false>;
        static bool attr_set[2] = {false, false};
        if (!attr_set[gated]) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S1_SMEM);
            if (e != cudaSuccess) return e;
            attr_set[gated] = true;
        }
        dim3 grid((x.N + S1_NC - 1) / S1_NC, x.B);
        kern<<<grid, S1_THREADS, S1_SMEM, stream>>>(ma, mb, x.T, x.N, x.s0, x.s_final, x.s_out, st, wait_ns);
    } else {
        dim3 grid((x.N + 127) / 128, x.B);
        if (gated) scan_seq_ldg<true><<<grid, 128, 0, stream>>>(x.T, x.N, x.a, x.b, x.s0, x.s_final, x.s_out);
        else scan_seq_ldg<false><<<grid, 128, 0, stream>>>(x.T, x.N, x.a, x.b, x.s0, x.s_final, x.s_out);
    }
    return cudaGetLastError();
}

bool lookback_supported(const ScanArgs& x) { return tma_ok(x); }

cudaError_t launch_scan_lookback(const ScanArgs& x, bool gated, void* ws, uint32_t epoch, int poison,
                                 SnDevStatus* st, uint64_t wait_ns, int sm_count, cudaStream_t stream) {
    CUtensorMap ma, mb;
    if (!make_scan_map(&ma, x.a, x.B, x.T, x.N, LB_NC, LB_TC) ||
        !make_scan_map(&mb, x.b, x.B, x.T, x.N, LB_NC, LB_TC))
        return cudaErrorInvalidValue;
    LookbackParams p;
    p.B = x.B;
    p.T = x.T;
    p.N = x.N;
    p.ncb = (x.N + LB_NC - 1) / LB_NC;
    p.nbcb = x.B * p.ncb;
    p.nchunks = (x.T + LB_TC - 1) / LB_TC;
    p.ntiles = p.nbcb * p.nchunks;
    p.s0 = x.s0;
    p.s_final = x.s_final;
    p.s_out = x.s_out;
    const int64_t tiles = p.ntiles;
    const int64_t flag_bytes = ((tiles * 4 + 255) / 256) * 256;
    p.flags = reinterpret_cast<uint32_t*>(ws);
    p.dA = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + flag_bytes);
    p.dB = p.dA + tiles * LB_NC;
    p.dC = p.dB + tiles * LB_NC;
    p.tag = epoch << 2;
    p.want = poison ? ((epoch + 1u) << 2) : p.tag;
    p.st = st;
    p.wait_ns = wait_ns;

    auto kern = gated ? scan_lookback<true> : scan_lookback<false>;
    static bool attr_set[2] = {false, false};
    static int occ[2] = {0, 0};
    if (!attr_set[gated]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LB_SMEM);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[gated], kern, LB_THREADS, LB_SMEM);
        if (e != cudaSuccess) return e;
        if (occ[gated] < 1) return cudaErrorInvalidConfiguration;
        attr_set[gated] = true;
    }
    const int grid = std::min<int64_t>(tiles, (int64_t)occ[gated] * sm_count);
    void* args[] = {(void*)&ma, (void*)&mb, (void*)&p};
    cudaError_t e = cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(LB_THREADS), args, LB_SMEM,
                                                stream);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace sn
