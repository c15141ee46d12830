// scan_bwd.cu -- reverse (adjoint) scans: the backward pass of both tier-1
// forms, sm_103a.
//
// Forward step s_t = a_t s_{t-1} + b_t, with b_t = (1 - a_t) u_t in the gated
// form ("SunnyNet 工程化实录" §2.1; the kernels there ship forward, reverse and
// single-step entries, §8).  Given gs_t = dL/ds_t and gf = dL/ds_final:
//   g_{T-1} = gs_{T-1} + gf,    g_t = fma(a_{t+1}, g_{t+1}, gs_t)
//   FMA:   da_t = g_t s_{t-1},           db_t = g_t
//   gated: da_t = g_t (s_{t-1} - u_t),   du_t = g_t (1 - a_t)
//   ds0 = a_0 g_0                        (s_{-1} = s0)
// The kernel runs T backwards per channel, like the forward sequential
// kernel: a producer warp streams [32 x 32] tiles of a, gs, the forward
// states shifted one step (s_{t-1}) and u through a 3- or 4-stage TMA ring, from
// the end of the sequence (the last tile may start at a negative row, which
// TMA fills with zeros); the consumer warp carries g through the steps and
// writes da and db|du with streaming stores.  Every operation is one explicit
// rounding, the order the fp32 CPU reference also uses.
#include <algorithm>

#include "scan_common.cuh"

namespace sn {

namespace {
constexpr int SB_NC = 32;                    // channels per CTA (one per consumer lane)
constexpr int SB_TS = 32;                    // time steps per stage
// Stages per form: 48 KB of ring per CTA either way, so four CTAs fit per SM
// and the grid (32-channel CTAs) runs in one wave.
template <bool GATED>
constexpr int sb_stages() { return GATED ? 3 : 4; }
constexpr int SB_THREADS = 64;               // warp 0 consumes, warp 1 produces
constexpr uint32_t SB_TILE = SB_TS * SB_NC;  // floats per tensor per stage

template <bool GATED>
constexpr int sb_tensors() { return GATED ? 4 : 3; }   // a, gs, s_{t-1}, (u)
template <bool GATED>
constexpr uint32_t sb_stage_bytes() { return sb_tensors<GATED>() * SB_TILE * 4; }
template <bool GATED>
constexpr size_t sb_smem() { return sb_stages<GATED>() * sb_stage_bytes<GATED>() + 2 * sb_stages<GATED>() * 8 + 16; }
// One interior stage of the consumer (no sequence edge inside, every row
// valid), rows SB_TS - 1 down to 0, in the same operation order as the edge
// path.  WA / WB select whether grad_a and grad_b|u are stored; pa, pb point
// at this lane's element of the stage's first row, rows N floats apart.
template <bool GATED, bool WA, bool WB>
__device__ __forceinline__ void bwd_stage(const float* A, const float* Gs, const float* Sp, const float* U,
                                          float* pa, float* pb, size_t N, float& g, float& an) {
#pragma unroll
    for (int i = SB_TS - 1; i >= 0; --i) {
        const float av = A[i * SB_NC], gv = Gs[i * SB_NC], sp = Sp[i * SB_NC];
        g = __fmaf_rn(an, g, gv);
        float oa, ob;
        if constexpr (GATED) {
            oa = __fmul_rn(g, __fsub_rn(sp, U[i * SB_NC]));
            ob = __fmul_rn(g, __fsub_rn(1.0f, av));
        } else {
            oa = __fmul_rn(g, sp);
            ob = g;
        }
        if constexpr (WA) st_cs(pa + (size_t)i * N, oa);
        if constexpr (WB) st_cs(pb + (size_t)i * N, ob);
        an = av;
    }
}

}  // namespace

template <bool GATED>
__global__ void __launch_bounds__(SB_THREADS)
scan_bwd_tma(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_gs,
             const __grid_constant__ CUtensorMap map_s, const __grid_constant__ CUtensorMap map_u, int T, int N,
             const float* __restrict__ s0, const float* __restrict__ gf, float* __restrict__ da,
             float* __restrict__ dbu, float* __restrict__ ds0, SnDevStatus* st, uint64_t wait_ns) {
    constexpr int NT = sb_tensors<GATED>();
    constexpr int SB_STAGES = sb_stages<GATED>();
    extern __shared__ __align__(128) unsigned char smem[];
    float* tiles = reinterpret_cast<float*>(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + SB_STAGES * sb_stage_bytes<GATED>());
    uint64_t* empty = full + SB_STAGES;
    volatile int* ctl = reinterpret_cast<volatile int*>(empty + SB_STAGES);   // [0] abort, [1] issued

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * SB_NC, bi = blockIdx.y;
    const int nst = (T + SB_TS - 1) / SB_TS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SB_STAGES; ++s) {
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
                const int slot = k % SB_STAGES;
                if (k >= SB_STAGES) {
                    const uint32_t par = ((k / SB_STAGES) - 1) & 1;
                    const uint64_t t0 = global_ns();
                    bool ok = mbar_try_wait(&empty[slot], par);
                    while (!ok && !ctl[0]) {
                        if (global_ns() - t0 > wait_ns) break;
                        ok = mbar_try_wait(&empty[slot], par);
                    }
                    if (!ok) {
                        if (!ctl[0]) record_error(st, SN_E_TIMEOUT, (SN_K_SCAN_SEQ << 16) | 5);
                        ctl[0] = 1;
                        break;
                    }
                }
                const int r0 = T - (k + 1) * SB_TS;           // first row of this stage (may be < 0)
                float* dst = tiles + (size_t)slot * NT * SB_TILE;
                mbar_arrive_expect_tx(&full[slot], sb_stage_bytes<GATED>());
                tma_load_3d(dst, &map_a, &full[slot], n0, r0, bi);
                tma_load_3d(dst + SB_TILE, &map_gs, &full[slot], n0, r0, bi);
                tma_load_3d(dst + 2 * SB_TILE, &map_s, &full[slot], n0, r0 - 1, bi);   // s_{t-1}
                if constexpr (GATED) tma_load_3d(dst + 3 * SB_TILE, &map_u, &full[slot], n0, r0, bi);
            }
            ctl[1] = k;
        }
    } else {
        const int c = n0 + lane;                      // this lane's channel
        const bool live = c < N;
        float gfv = 0.f, s0v = 0.f;
        if (live) {
            if (gf != nullptr) gfv = gf[(size_t)bi * N + c];
            if (s0 != nullptr) s0v = s0[(size_t)bi * N + c];
        }
        float g = 0.f, an = 0.f;                      // running adjoint, a_{t+1}
        auto row = [&](const float* A, const float* Gs, const float* Sp, const float* U, int i, int t, bool edge) {
            const float av = A[i * SB_NC], gv = Gs[i * SB_NC];
            float sp = Sp[i * SB_NC];
            if (edge && t == 0) sp = s0v;
            if (edge && t == T - 1) g = __fadd_rn(gv, gfv);
            else g = __fmaf_rn(an, g, gv);
            float oa, ob;
            if constexpr (GATED) {
                oa = __fmul_rn(g, __fsub_rn(sp, U[i * SB_NC]));
                ob = __fmul_rn(g, __fsub_rn(1.0f, av));
            } else {
                oa = __fmul_rn(g, sp);
                ob = g;
            }
            if (live) {
                const size_t off = ((size_t)bi * T + t) * N + c;
                if (da != nullptr) st_cs(da + off, oa);
                if (dbu != nullptr) st_cs(dbu + off, ob);
            }
            an = av;
        };
        for (int k = 0; k < nst; ++k) {
            const int slot = k % SB_STAGES;
            const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[slot], (k / SB_STAGES) & 1, wait_ns));
            if (!ok) {
                if (lane == 0) {
                    record_error(st, SN_E_TIMEOUT, (SN_K_SCAN_SEQ << 16) | 6);
                    ctl[0] = 1;
                }
                break;
            }
            const float* A = tiles + (size_t)slot * NT * SB_TILE + lane;
            const float* Gs = A + SB_TILE;
            const float* Sp = A + 2 * SB_TILE;
            const float* U = A + 3 * SB_TILE;
            const int r0 = T - (k + 1) * SB_TS;
            if (k > 0 && r0 >= 1) {
                // interior stage: neither t = T-1 nor t = 0 occurs, all rows valid;
                // which outputs this lane stores is decided once per stage
                const size_t base = ((size_t)bi * T + r0) * N + c;
                const bool wa = live && da != nullptr, wb = live && dbu != nullptr;
                float* pa = wa ? da + base : nullptr;
                float* pb = wb ? dbu + base : nullptr;
                if (wa && wb) bwd_stage<GATED, true, true>(A, Gs, Sp, U, pa, pb, N, g, an);
                else if (wa) bwd_stage<GATED, true, false>(A, Gs, Sp, U, pa, pb, N, g, an);
                else if (wb) bwd_stage<GATED, false, true>(A, Gs, Sp, U, pa, pb, N, g, an);
                else bwd_stage<GATED, false, false>(A, Gs, Sp, U, pa, pb, N, g, an);
            } else {
                for (int i = SB_TS - 1; i >= max(0, -r0); --i) row(A, Gs, Sp, U, i, r0 + i, true);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            ++consumed;
        }
        if (ds0 != nullptr && live && consumed == nst) ds0[(size_t)bi * N + c] = __fmul_rn(an, g);   // a_0 g_0
    }
    __syncthreads();
    if (warp == 0 && lane == 0 && ctl[0]) {
        for (int k = consumed; k < ctl[1]; ++k)
            (void)mbar_wait(&full[k % SB_STAGES], (k / SB_STAGES) & 1, wait_ns);
    }
}

// Layouts TMA cannot describe: one thread per channel, plain loads.
template <bool GATED>
__global__ void __launch_bounds__(128)
scan_bwd_ldg(int T, int N, const float* __restrict__ a, const float* __restrict__ u,
             const float* __restrict__ s0, const float* __restrict__ s, const float* __restrict__ gs,
             const float* __restrict__ gf, float* __restrict__ da, float* __restrict__ dbu,
             float* __restrict__ ds0) {
    const int c = blockIdx.x * 128 + threadIdx.x;
    const int bi = blockIdx.y;
    if (c >= N) return;
    const size_t base = (size_t)bi * T * N + c;
    const float gfv = gf != nullptr ? gf[(size_t)bi * N + c] : 0.f;
    const float s0v = s0 != nullptr ? s0[(size_t)bi * N + c] : 0.f;
    float g = 0.f, an = 0.f;
    for (int t = T - 1; t >= 0; --t) {
        const size_t x = base + (size_t)t * N;
        const float av = a[x], gv = gs[x];
        const float sp = t > 0 ? s[x - N] : s0v;
        g = (t == T - 1) ? __fadd_rn(gv, gfv) : __fmaf_rn(an, g, gv);
        if constexpr (GATED) {
            if (da != nullptr) da[x] = __fmul_rn(g, __fsub_rn(sp, u[x]));
            if (dbu != nullptr) dbu[x] = __fmul_rn(g, __fsub_rn(1.0f, av));
        } else {
            if (da != nullptr) da[x] = __fmul_rn(g, sp);
            if (dbu != nullptr) dbu[x] = g;
        }
        an = av;
    }
    if (ds0 != nullptr) ds0[(size_t)bi * N + c] = __fmul_rn(an, g);
}

cudaError_t launch_scan_backward(const BwdArgs& x, bool gated, SnDevStatus* st, uint64_t wait_ns,
                                 cudaStream_t stream) {
    auto al16 = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const bool tma = (x.N % 4 == 0) && al16(x.a) && al16(x.gs) && al16(x.s) && al16(x.u);
    if (tma) {
        CUtensorMap ma, mg, ms, mu;
        if (!make_scan_map(&ma, x.a, x.B, x.T, x.N, SB_NC, SB_TS) ||
            !make_scan_map(&mg, x.gs, x.B, x.T, x.N, SB_NC, SB_TS) ||
            !make_scan_map(&ms, x.s, x.B, x.T, x.N, SB_NC, SB_TS))
            return cudaErrorInvalidValue;
        if (gated) {
            if (!make_scan_map(&mu, x.u, x.B, x.T, x.N, SB_NC, SB_TS)) return cudaErrorInvalidValue;
        } else {
            mu = ma;   // unused
        }
        auto kern = gated ? scan_bwd_tma<true> : scan_bwd_tma<false>;
        const size_t smem = gated ? sb_smem<true>() : sb_smem<false>();
        cudaError_t e = set_smem_attr_once((const void*)kern, smem);
        if (e != cudaSuccess) return e;
        dim3 grid((x.N + SB_NC - 1) / SB_NC, x.B);
        kern<<<grid, SB_THREADS, smem, stream>>>(ma, mg, ms, mu, x.T, x.N, x.s0, x.gf, x.da, x.dbu, x.ds0, st,
                                                 wait_ns);
    } else {
        dim3 grid((x.N + 127) / 128, x.B);
        if (gated)
            scan_bwd_ldg<true><<<grid, 128, 0, stream>>>(x.T, x.N, x.a, x.u, x.s0, x.s, x.gs, x.gf, x.da, x.dbu,
                                                         x.ds0);
        else
            scan_bwd_ldg<false><<<grid, 128, 0, stream>>>(x.T, x.N, x.a, x.u, x.s0, x.s, x.gs, x.gf, x.da, x.dbu,
                                                          x.ds0);
    }
    return cudaGetLastError();
}

}  // namespace sn
