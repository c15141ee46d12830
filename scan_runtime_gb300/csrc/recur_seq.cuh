// recur_seq.cuh -- the sequence kernel shared by the three matrix recurrences
// (instantiated per kind in recur_diag.cu, recur_diag_gated.cu,
// recur_delta.cu, recur_rwkv7.cu; the tile of each problem is chosen at the
// end of this file).
//
// All recurrences are written for the state P in R^{dk x dv} (row = key index
// i, column = value index j), whose columns evolve independently:
//   diag   P_t = diag(d_t) P_{t-1} + k_t v_t^T                       GLA / Mamba-2
//   delta  P_t = P_{t-1} + k_t delta_t^T,  delta_t = (v_t - P_{t-1}^T k_t) beta_t
//   rwkv7  P_t = diag(w_t) P_{t-1} + k_t delta_t^T,  delta_t = v_t - P_{t-1}^T k_t
//   readout o_t = scale * P_t^T q_t
// ("SunnyNet 工程化实录：一个 O(N) 架构如何长出自己的 C 推理运行时" §4.1 Mamba-2,
// §4.2 DeltaNet, §4.3 GLA, §5.1 RWKV-7; RWKV-7's S in R^{dv x dk} is P^T, so it
// is the delta template with a per-key decay and beta = 1, loaded and stored
// transposed.)
//
// Work split: one CTA per (batch, head, tile of JT value columns).  A lane
// holds R rows x C columns of P in registers for the whole sequence; LPC =
// dk / R lanes share a group of C columns; W consumer warps take different
// column groups.  Column pairs are packed into f32x2 operations, so every k /
// decay / q value read feeds C state entries.  q, k, per-key decay and the v
// slice arrive through a 3-stage TMA ring fed by a producer warp (per-head
// scalars by 4-byte cp.async on the same mbarrier); o leaves through TMA
// stores.  Each step's operands are read from shared memory PF steps ahead of
// its arithmetic.
//
// Arithmetic per column is fixed by R (rows per lane):
//   * the diag update is fma(d_i, P_ij, k_i * v_j) with the product rounded
//     first (the single-precision definition's order), so the diagonal-decay
//     state has the definition's bits whatever the tile;
//   * a dot product over rows (the delta rule's P^T k and every readout) runs
//     four chains over a lane's rows (row index mod 4) joined as
//     (c0 + c1) + (c2 + c3); the LPC lane partials join over xor partners
//     LPC/2 .. 1.
// The result therefore depends only on the state, the inputs and R: segment
// splits are bit-exact, C, W and PF do not change the bits, and the
// single-step decode kernels reproduce the same order (recur_decode.cu,
// recur_rwkv7.cu).
#pragma once

#include <algorithm>

#include "ptx.cuh"
#include "sn_internal.h"

namespace sn {

constexpr int RS_TS = 16;       // time steps per stage
constexpr int RS_STAGES = 3;
constexpr int RS_OBUF = 3;      // output staging buffers

template <int KIND>
constexpr bool per_key_gate() { return KIND == RK_DIAG_KEY || KIND == RK_RWKV7 || KIND == RK_DIAG_KEY_GATED; }
template <int KIND>
constexpr bool scalar_gate() { return KIND == RK_DIAG_HEAD || KIND == RK_DELTA || KIND == RK_DIAG_HEAD_GATED; }
template <int KIND>
constexpr bool diag_kind() {
    return KIND == RK_DIAG_KEY || KIND == RK_DIAG_HEAD || KIND == RK_DIAG_KEY_GATED || KIND == RK_DIAG_HEAD_GATED;
}
template <int KIND>
constexpr bool gated_injection() { return KIND == RK_DIAG_KEY_GATED || KIND == RK_DIAG_HEAD_GATED; }

// Steps per readout reduction batch: 8, or 16 when 8 steps of C columns do
// not fill a reduction over LPC lanes.
constexpr int readout_batch(int C, int LPC) { return (8 * C) % LPC == 0 ? 8 : 16; }

template <int KIND, int DK, int JT>
struct SeqLayout {
    static constexpr uint32_t q_off = 0;
    static constexpr uint32_t k_off = q_off + RS_TS * DK * 4;
    static constexpr uint32_t g_off = k_off + RS_TS * DK * 4;
    static constexpr uint32_t g_bytes = per_key_gate<KIND>() ? RS_TS * DK * 4 : 128;
    static constexpr uint32_t v_off = g_off + g_bytes;
    static constexpr uint32_t v_bytes = ((RS_TS * JT * 4 + 127) / 128) * 128;
    static constexpr uint32_t stage_bytes = v_off + v_bytes;
    static constexpr uint32_t tx_bytes = 2 * RS_TS * DK * 4 + (per_key_gate<KIND>() ? RS_TS * DK * 4 : 0) +
                                         RS_TS * JT * 4;
    static constexpr uint32_t o_off = RS_STAGES * stage_bytes;
    static constexpr uint32_t o_bytes = ((RS_TS * JT * 4 + 127) / 128) * 128;
    static constexpr uint32_t bar_off = o_off + RS_OBUF * o_bytes;
    static constexpr size_t smem = bar_off + 2 * RS_STAGES * 8 + 128;   // + alignment slack
};

struct SeqParams {
    int T, H, G, dk, dv;
    float scale;
    const float* g;        // per-head scalars (dA or beta) for cp.async
    const float* S_in;
    float* S_out;
    int has_o;
    SnDevStatus* st;
    uint64_t wait_ns;
};

__device__ __forceinline__ float2 f2(float x) { return make_float2(x, x); }

__device__ __forceinline__ float group_sum(float x, int lpc) {
    for (int o = lpc >> 1; o > 0; o >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float2 group_sum2(float2 x, int lpc) {
    return make_float2(group_sum(x.x, lpc), group_sum(x.y, lpc));
}

// Sum NV per-lane values over a group of LPC lanes by recursive halving: at
// offset o a lane keeps the half its bit o selects and adds its partner's copy
// of that half.  Afterwards v[e] (e < NV/LPC) holds the group sum of value
// index sub * (NV/LPC) + e.  The pairing (offsets LPC/2 .. 1) is group_sum's
// and addition is commutative, so each sum has the bits group_sum gives it.
template <int LPC, int NV>
__device__ __forceinline__ void reduce_scatter(float (&v)[NV], int sub) {
#pragma unroll
    for (int lvl = 0; (LPC >> (lvl + 1)) >= 1; ++lvl) {
        const int o = LPC >> (lvl + 1);
        const int c = NV >> lvl;
        const bool upper = (sub & o) != 0;
#pragma unroll
        for (int i = 0; i < c / 2; ++i) {
            const float send = upper ? v[i] : v[i + c / 2];
            const float keep = upper ? v[i + c / 2] : v[i];
            v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, o));
        }
    }
}

template <int R, int LPC>
__device__ __forceinline__ void load_rows(float (&x)[R], const float* row, int sub) {
#pragma unroll
    for (int m = 0; m < R / 4; ++m) {
        const float4 t = *reinterpret_cast<const float4*>(row + (m * LPC + sub) * 4);
        x[4 * m] = t.x; x[4 * m + 1] = t.y; x[4 * m + 2] = t.z; x[4 * m + 3] = t.w;
    }
}

// Operands of one time step for one lane: its rows of k, the per-key gate and
// q, its group's C values of v, and the per-head scalar (dA or beta).
template <int KIND, int R, int C>
struct StepOps {
    float k[R];
    float g[per_key_gate<KIND>() ? R : 1];
    float q[R];
    float2 v[C / 2];
    float s;
};

// Read one step's operands: rows (m * LPC + sub) * 4 + e (m < R/4, e < 4) of
// the row slice kr, gr, qr point into, and the group's C values at vr.
template <int KIND, int R, int C, int LPC>
__device__ __forceinline__ void load_step(StepOps<KIND, R, C>& x, const float* kr, const float* gr, const float* qr,
                                          const float* vr, float gsc, int sub, bool want_o) {
    load_rows<R, LPC>(x.k, kr, sub);
    if constexpr (per_key_gate<KIND>()) load_rows<R, LPC>(x.g, gr, sub);
    if (want_o) load_rows<R, LPC>(x.q, qr, sub);
#pragma unroll
    for (int c = 0; c < C / 2; ++c) x.v[c] = *reinterpret_cast<const float2*>(vr + 2 * c);
    x.s = gsc;
}

// One time step for one lane on its R rows x C columns (packed as C/2 pairs)
// from the step's operands; opart receives this lane's readout partials.
template <int KIND, int R, int C, int LPC>
__device__ __forceinline__ void step_compute(float2 (&P)[R][C / 2], const StepOps<KIND, R, C>& x,
                                             float2 (&opart)[C / 2], bool want_o) {
    constexpr int C2 = C / 2;
    float kv[R];
#pragma unroll
    for (int r = 0; r < R; ++r) kv[r] = x.k[r];
    if constexpr (diag_kind<KIND>()) {
        float dv_[R];
#pragma unroll
        for (int r = 0; r < R; ++r) dv_[r] = per_key_gate<KIND>() ? x.g[per_key_gate<KIND>() ? r : 0] : x.s;
        if constexpr (gated_injection<KIND>()) {
            // convex combination: the injection k_i v_j enters with weight 1 - p_i
#pragma unroll
            for (int r = 0; r < R; ++r) kv[r] = __fmul_rn(__fsub_rn(1.0f, dv_[r]), kv[r]);
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int c = 0; c < C2; ++c) P[r][c] = __ffma2_rn(f2(dv_[r]), P[r][c], __fmul2_rn(f2(kv[r]), x.v[c]));
    } else {
#pragma unroll
        for (int c = 0; c < C2; ++c) {
            float2 u0 = f2(0.f), u1 = f2(0.f), u2 = f2(0.f), u3 = f2(0.f);
#pragma unroll
            for (int m = 0; m < R / 4; ++m) {
                u0 = __ffma2_rn(P[4 * m][c], f2(kv[4 * m]), u0);
                u1 = __ffma2_rn(P[4 * m + 1][c], f2(kv[4 * m + 1]), u1);
                u2 = __ffma2_rn(P[4 * m + 2][c], f2(kv[4 * m + 2]), u2);
                u3 = __ffma2_rn(P[4 * m + 3][c], f2(kv[4 * m + 3]), u3);
            }
            const float2 u = group_sum2(__fadd2_rn(__fadd2_rn(u0, u1), __fadd2_rn(u2, u3)), LPC);
            float2 delta = __fadd2_rn(x.v[c], make_float2(-u.x, -u.y));   // v - u, exactly
            if constexpr (KIND == RK_DELTA) {
                delta = __fmul2_rn(delta, f2(x.s));
#pragma unroll
                for (int r = 0; r < R; ++r) P[r][c] = __ffma2_rn(f2(kv[r]), delta, P[r][c]);
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r)
                    P[r][c] = __ffma2_rn(f2(kv[r]), delta, __fmul2_rn(P[r][c], f2(x.g[per_key_gate<KIND>() ? r : 0])));
            }
        }
    }
    if (!want_o) return;
#pragma unroll
    for (int c = 0; c < C2; ++c) {
        float2 a0 = f2(0.f), a1 = f2(0.f), a2 = f2(0.f), a3 = f2(0.f);
#pragma unroll
        for (int m = 0; m < R / 4; ++m) {
            a0 = __ffma2_rn(P[4 * m][c], f2(x.q[4 * m]), a0);
            a1 = __ffma2_rn(P[4 * m + 1][c], f2(x.q[4 * m + 1]), a1);
            a2 = __ffma2_rn(P[4 * m + 2][c], f2(x.q[4 * m + 2]), a2);
            a3 = __ffma2_rn(P[4 * m + 3][c], f2(x.q[4 * m + 3]), a3);
        }
        opart[c] = __fadd2_rn(__fadd2_rn(a0, a1), __fadd2_rn(a2, a3));
    }
}

// One time step for one lane: load the operands, then compute.  kr, gr, qr
// point at the row slice's k, per-key gate and q rows; vr at the group's C
// values; gsc is the per-head scalar (dA or beta).
template <int KIND, int R, int C, int LPC>
__device__ __forceinline__ void lane_step(float2 (&P)[R][C / 2], const float* kr, const float* gr,
                                          const float* qr, const float* vr, float gsc, int sub,
                                          float2 (&opart)[C / 2], bool want_o) {
    StepOps<KIND, R, C> x;
    load_step<KIND, R, C, LPC>(x, kr, gr, qr, vr, gsc, sub, want_o);
    step_compute<KIND, R, C, LPC>(P, x, opart, want_o);
}

// Tile of the sequence kernel for key dimension DK: R rows x C columns per
// lane, LPC = DK / R lanes per column group, W consumer warps; GEN reads the
// staged operands through generic pointers (see smem_align_generic); PF > 0
// reads each step's operands PF steps ahead of its arithmetic (registers as a
// ring).
template <int DK, int R_, int C_, int W_, bool GEN_, int PF_>
struct SeqTile {
    static constexpr int R = R_, C = C_, LPC = DK / R_, W = W_;
    static constexpr bool GEN = GEN_;
    static constexpr int PF = PF_;                       // steps whose operands are read ahead
    static constexpr int CPW = 32 / LPC;                 // column groups per warp
    static constexpr int JT = W * CPW * C;               // columns per CTA
    static constexpr int NCONS = W;                      // consumer warps
    static constexpr int THREADS = (NCONS + 1) * 32;
    static constexpr int RB = readout_batch(C, LPC);
};

template <int KIND, int DK, class TL>
__global__ void __launch_bounds__(TL::THREADS)
recur_seq(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
          const __grid_constant__ CUtensorMap map_g, const __grid_constant__ CUtensorMap map_v,
          const __grid_constant__ CUtensorMap map_o, const SeqParams p) {
    constexpr int R = TL::R, C = TL::C, LPC = TL::LPC, CPW = TL::CPW, JT = TL::JT;
    constexpr int NCONS = TL::NCONS, RB = TL::RB;
    constexpr int C2 = C / 2;
    constexpr int NV = RB * C;             // readout values per lane per batch
    using L = SeqLayout<KIND, DK, JT>;
    static_assert(R % 4 == 0 && C % 2 == 0 && LPC >= 1 && LPC <= 32 && (LPC & (LPC - 1)) == 0 && R * LPC == DK,
                  "tile shape");
    static_assert(NV % LPC == 0 && RS_TS % RB == 0, "reduction shape");

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = TL::GEN ? smem_align_generic<128>(smem_raw) : smem_align<128>(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::bar_off);
    uint64_t* empty = full + RS_STAGES;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int jt0 = blockIdx.x * JT, h = blockIdx.y, b = blockIdx.z;
    const int grp = h / (p.H / p.G);
    const int T = p.T;
    const int nst = (T + RS_TS - 1) / RS_TS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < RS_STAGES; ++s) {
            mbar_init(&full[s], scalar_gate<KIND>() ? 33 : 1);
            mbar_init(&empty[s], NCONS);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NCONS) {
        // ------------------------------------------------ producer warp
        for (int kk = 0; kk < nst; ++kk) {
            const int slot = kk % RS_STAGES;
            if (kk >= RS_STAGES) {
                const bool ok =
                    __all_sync(0xffffffffu, mbar_wait(&empty[slot], ((kk / RS_STAGES) - 1) & 1, p.wait_ns));
                if (!ok) {
                    if (lane == 0) record_error(p.st, SN_E_TIMEOUT, (SN_K_RECUR_SEQ << 16) | 1);
                    break;       // consumers will time out on `full` and stop too
                }
            }
            unsigned char* sb = smem + slot * L::stage_bytes;
            const int t0 = kk * RS_TS;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[slot], L::tx_bytes);
                tma_load_4d(sb + L::q_off, &map_q, &full[slot], 0, grp, t0, b);
                tma_load_4d(sb + L::k_off, &map_k, &full[slot], 0, grp, t0, b);
                if constexpr (per_key_gate<KIND>()) tma_load_4d(sb + L::g_off, &map_g, &full[slot], 0, h, t0, b);
                tma_load_4d(sb + L::v_off, &map_v, &full[slot], jt0, h, t0, b);
            }
            if constexpr (scalar_gate<KIND>()) {
                if (lane < RS_TS && t0 + lane < T)
                    cp_async_4(sb + L::g_off + 4 * lane, p.g + ((size_t)b * T + t0 + lane) * p.H + h);
                cp_async_mbar_arrive_noinc(&full[slot]);
            }
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    const int gcol = lane / LPC, sub = lane % LPC;
    const int jl0 = (warp * CPW + gcol) * C;             // first column of the group within the tile
    const int j0 = jt0 + jl0;
    const size_t sbase = ((size_t)b * p.H + h) * (size_t)DK * p.dv;

    float2 P[R][C2];
#pragma unroll
    for (int m = 0; m < R / 4; ++m) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int row = (m * LPC + sub) * 4 + e;
#pragma unroll
            for (int c = 0; c < C2; ++c) {
                float x0 = 0.f, x1 = 0.f;
                if (p.S_in != nullptr) {
                    if (KIND == RK_RWKV7) {          // stored (dv, dk): value row, keys contiguous
                        x0 = p.S_in[sbase + (size_t)(j0 + 2 * c) * DK + row];
                        x1 = p.S_in[sbase + (size_t)(j0 + 2 * c + 1) * DK + row];
                    } else {                         // stored (dk, dv)
                        const float2 t =
                            *reinterpret_cast<const float2*>(p.S_in + sbase + (size_t)row * p.dv + j0 + 2 * c);
                        x0 = t.x;
                        x1 = t.y;
                    }
                }
                P[4 * m + e][c] = make_float2(x0, x1);
            }
        }
    }

    const bool want_o = p.has_o != 0;
    // A warp whose stage wait runs out records the error and from then on
    // skips the waits and the arithmetic, but keeps passing the named
    // barriers with the other consumer warps, so none of them is left waiting
    // at a barrier (the other warps time out on the same stage or finish).
    bool failed = false;
    for (int kk = 0; kk < nst; ++kk) {
        const int slot = kk % RS_STAGES;
        if (!failed && !__all_sync(0xffffffffu, mbar_wait(&full[slot], (kk / RS_STAGES) & 1, p.wait_ns))) {
            if (lane == 0) record_error(p.st, SN_E_TIMEOUT, (SN_K_RECUR_SEQ << 16) | 2);
            failed = true;
        }
        const unsigned char* sb = smem + slot * L::stage_bytes;
        const float* qs = reinterpret_cast<const float*>(sb + L::q_off);
        const float* ks = reinterpret_cast<const float*>(sb + L::k_off);
        const float* gs = reinterpret_cast<const float*>(sb + L::g_off);
        const float* gks = gs;
        const float* vs = reinterpret_cast<const float*>(sb + L::v_off);
        float* os = reinterpret_cast<float*>(smem + L::o_off + (kk % RS_OBUF) * L::o_bytes);
        const int tn = min(RS_TS, T - kk * RS_TS);

        // a column's readout sum, scaled, into the output staging
        auto put = [&](int t, int col, float x) { os[t * JT + col] = __fmul_rn(x, p.scale); };
        if (failed) {
            // no arithmetic: fall through to the stage's barriers
        } else if (tn == RS_TS) {
            // Readout partials of RB steps stay in registers and are reduced
            // once over the lane group (no per-step shuffle chain or store).
            constexpr int PF = TL::PF;
            StepOps<KIND, R, C> ring[PF + 1];
            auto fetch = [&](int t) {
                load_step<KIND, R, C, LPC>(ring[t % (PF + 1)], ks + t * DK, gks + t * DK, qs + t * DK,
                                           vs + t * JT + jl0, scalar_gate<KIND>() ? gs[t] : 0.f, sub, want_o);
            };
#pragma unroll
            for (int t = 0; t < PF; ++t) fetch(t);
#pragma unroll
            for (int rb = 0; rb < RS_TS / RB; ++rb) {
                float2 ov[RB][C2];
#pragma unroll
                for (int i = 0; i < RB; ++i) {
                    const int t = rb * RB + i;
                    if (t + PF < RS_TS) fetch(t + PF);
                    step_compute<KIND, R, C, LPC>(P, ring[t % (PF + 1)], ov[i], want_o);
                }
                if (want_o) {
                    float fl[NV];                      // [step][column] readout partials
#pragma unroll
                    for (int i = 0; i < RB; ++i)
#pragma unroll
                        for (int c = 0; c < C2; ++c) {
                            fl[i * C + 2 * c] = ov[i][c].x;
                            fl[i * C + 2 * c + 1] = ov[i][c].y;
                        }
                    reduce_scatter<LPC, NV>(fl, sub);
                    constexpr int PER = NV / LPC;
#pragma unroll
                    for (int e = 0; e < PER; ++e) {
                        const int idx = sub * PER + e;
                        put(rb * RB + idx / C, jl0 + idx % C, fl[e]);
                    }
                }
            }
        } else {
            for (int t = 0; t < tn; ++t) {
                float2 part2[C2];
                lane_step<KIND, R, C, LPC>(P, ks + t * DK, gks + t * DK, qs + t * DK, vs + t * JT + jl0,
                                           scalar_gate<KIND>() ? gs[t] : 0.f, sub, part2, want_o);
                if (want_o) {
#pragma unroll
                    for (int c = 0; c < C2; ++c) {
                        const float2 acc = group_sum2(part2[c], LPC);
                        if (sub == 0) {
                            put(t, jl0 + 2 * c, acc.x);
                            put(t, jl0 + 2 * c + 1, acc.y);
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0 && !failed) mbar_arrive(&empty[slot]);
        if (want_o) {
            fence_proxy_async_smem();
            // the store two stages back read the buffer the next stage writes
            if (threadIdx.x == 0) bulk_wait_read_allbut1();
            named_bar_sync(1, NCONS * 32);
            if (threadIdx.x == 0) {
                tma_store_4d(&map_o, os, jt0, h, kk * RS_TS, b);
                bulk_commit();
            }
        }
    }
    if (threadIdx.x == 0) bulk_wait_all();
    if (failed || p.S_out == nullptr) return;
#pragma unroll
    for (int m = 0; m < R / 4; ++m) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int row = (m * LPC + sub) * 4 + e;
#pragma unroll
            for (int c = 0; c < C2; ++c) {
                const float2 x = P[4 * m + e][c];
                if (KIND == RK_RWKV7) {
                    p.S_out[sbase + (size_t)(j0 + 2 * c) * DK + row] = x.x;
                    p.S_out[sbase + (size_t)(j0 + 2 * c + 1) * DK + row] = x.y;
                } else {
                    *reinterpret_cast<float2*>(p.S_out + sbase + (size_t)row * p.dv + j0 + 2 * c) = x;
                }
            }
        }
    }
}

template <int KIND, int DK, class TL>
cudaError_t run_seq(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, cudaStream_t stream) {
    constexpr int JT = TL::JT;
    using L = SeqLayout<KIND, DK, JT>;
    if (x.dv % JT != 0 || x.dk != DK) return cudaErrorInvalidValue;
    const int gdim = diag_kind<KIND>() ? x.G : x.H;
    CUtensorMap mq, mk, mg, mv, mo;
    const uint64_t dqk[4] = {(uint64_t)DK, (uint64_t)gdim, (uint64_t)x.T, (uint64_t)x.B};
    const uint64_t sqk[3] = {(uint64_t)DK * 4, (uint64_t)gdim * DK * 4, (uint64_t)x.T * gdim * DK * 4};
    const uint32_t bqk[4] = {(uint32_t)DK, 1, RS_TS, 1};
    const uint64_t dg[4] = {(uint64_t)DK, (uint64_t)x.H, (uint64_t)x.T, (uint64_t)x.B};
    const uint64_t sg[3] = {(uint64_t)DK * 4, (uint64_t)x.H * DK * 4, (uint64_t)x.T * x.H * DK * 4};
    const uint64_t dvv[4] = {(uint64_t)x.dv, (uint64_t)x.H, (uint64_t)x.T, (uint64_t)x.B};
    const uint64_t svv[3] = {(uint64_t)x.dv * 4, (uint64_t)x.H * x.dv * 4, (uint64_t)x.T * x.H * x.dv * 4};
    const uint32_t bv[4] = {(uint32_t)JT, 1, RS_TS, 1};
    if (!encode_tiled(&mq, 4, x.q, dqk, sqk, bqk) || !encode_tiled(&mk, 4, x.k, dqk, sqk, bqk) ||
        !encode_tiled(&mv, 4, x.v, dvv, svv, bv))
        return cudaErrorInvalidValue;
    if (per_key_gate<KIND>()) {
        if (!encode_tiled(&mg, 4, x.g, dg, sg, bqk)) return cudaErrorInvalidValue;
    } else {
        mg = mk;   // unused
    }
    if (x.o != nullptr) {
        if (!encode_tiled(&mo, 4, x.o, dvv, svv, bv)) return cudaErrorInvalidValue;
    } else {
        mo = mv;   // unused
    }
    SeqParams p{x.T, x.H, x.G, x.dk, x.dv, x.scale, x.g, x.S_in, x.S_out, x.o != nullptr ? 1 : 0, st, wait_ns};
    auto kern = recur_seq<KIND, DK, TL>;
    cudaError_t e = set_smem_attr_once((const void*)kern, L::smem);
    if (e != cudaSuccess) return e;
    dim3 grid(x.dv / JT, x.H, x.B);
    kern<<<grid, TL::THREADS, L::smem, stream>>>(mq, mk, mg, mv, mo, p);
    return cudaGetLastError();
}

}  // namespace sn

namespace sn {

// Tile choices, measured on the GLA, Mamba-2, DeltaNet and RWKV-7 workloads
// (a sweep of rows and columns per lane, CTA width and operand read-ahead):
//   * diagonal kinds with few warps (the GLA shape): 4 rows x 4 columns,
//     generic operand reads, read-ahead 1; 4-warp CTAs while they fit in one
//     wave, else 2-warp CTAs;
//   * diagonal kinds otherwise (the Mamba-2 shape): 8 rows x 2 columns,
//     4-warp CTAs, read-ahead 1;
//   * the delta rule: 8 rows x 2 columns, 2-warp CTAs, read-ahead 1;
//   * RWKV-7: 8 rows x 2 columns, 4-warp CTAs.
// Only the rows per lane fix the summation order, and they are the ones the
// earlier tiles used, so these tiles give the same bits.  A forced width
// (SN_OPT_RECUR_TILE: 2, 4 or 8 warps) replaces the width.

// Warps the sequence kernel would run with R rows x C columns per lane.
inline int64_t seq_warps(const RecurArgs& x, int R, int C) {
    return (int64_t)x.B * x.H * (x.dv / C) * (x.dk / R) / 32;
}

// Rows per lane of the diagonal-decay kinds: 8 when the problem yields at
// least DIAG_R8_WARPS warps per SM with 8 rows x 4 columns per lane, else 4
// rows, which keeps small problems (B4 H4 128 x 128) at more warps.  The
// single-step decode follows the same rule, so a decode step has the bits of
// a one-step sequence call.
constexpr int DIAG_R8_WARPS = 4;
inline bool diag_eight_rows(const RecurArgs& x, int sm_count) {
    return seq_warps(x, 8, 4) >= (int64_t)DIAG_R8_WARPS * sm_count;
}

// Value columns one consumer warp covers under the tile the dispatch picks.
inline int seq_cols_per_warp(const RecurArgs& x, int sm_count) {
    const bool diag = x.kind == RK_DIAG_KEY || x.kind == RK_DIAG_HEAD || x.kind == RK_DIAG_KEY_GATED ||
                      x.kind == RK_DIAG_HEAD_GATED;
    const bool small = diag && !diag_eight_rows(x, sm_count);
    const int R = small ? 4 : 8, C = small ? 4 : 2;
    return (32 / (x.dk / R)) * C;
}

template <int KIND, int DK, int R, int C, bool GEN, int PF>
cudaError_t run_seq_w(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int w, cudaStream_t stream) {
    switch (w) {
        case 2: return run_seq<KIND, DK, SeqTile<DK, R, C, 2, GEN, PF>>(x, st, wait_ns, stream);
        case 4: return run_seq<KIND, DK, SeqTile<DK, R, C, 4, GEN, PF>>(x, st, wait_ns, stream);
        case 8: return run_seq<KIND, DK, SeqTile<DK, R, C, 8, GEN, PF>>(x, st, wait_ns, stream);
        default: return cudaErrorInvalidValue;
    }
}

// The diagonal kinds (plain and gated) for key dimension DK.
template <int KIND, int DK>
cudaError_t run_seq_diag(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count, int force_w,
                         cudaStream_t stream) {
    if (diag_eight_rows(x, sm_count))
        return run_seq_w<KIND, DK, 8, 2, false, 1>(x, st, wait_ns, force_w ? force_w : 4, stream);
    int w = force_w;
    if (w == 0) {
        constexpr int COLS_PER_WARP = (32 / (DK / 4)) * 4;
        const bool fits4 = x.dv % (4 * COLS_PER_WARP) == 0 &&
                           (int64_t)x.B * x.H * (x.dv / (4 * COLS_PER_WARP)) <= sm_count;
        w = (fits4 || x.dv % (2 * COLS_PER_WARP) != 0) ? 4 : 2;
    }
    return run_seq_w<KIND, DK, 4, 4, true, 1>(x, st, wait_ns, w, stream);
}

}  // namespace sn
