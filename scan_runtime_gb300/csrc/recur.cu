// recur.cu -- tier 2: per-head matrix-state recurrences with readout, sm_103a.
//
// All four recurrences are written for the state P in R^{dk x dv} (row = key
// index i, column = value index j), whose columns evolve independently:
//   diag   P_t = diag(d_t) P_{t-1} + k_t v_t^T                      GLA / Mamba-2
//   delta  P_t = P_{t-1} + k_t delta_t^T,  delta_t = (v_t - P_{t-1}^T k_t) beta_t
//   rwkv7  P_t = diag(w_t) P_{t-1} + k_t delta_t^T,  delta_t = v_t - P_{t-1}^T k_t
//   readout o_t = scale * P_t^T q_t
// RWKV-7's state S in R^{dv x dk} ("SunnyNet 工程化实录" §5.1:
// S_t = S_{t-1}(.)w_t - (S_{t-1}k_t)k_t^T + v_t k_t^T, o_t = S_t q_t) is the
// transpose P = S^T, so it is the delta template with a per-key decay and
// beta = 1; the kernel loads and stores it transposed.  Diag follows
// "SunnyNet 工程化实录" §4.1 and §4.3, delta §4.2.
//
// Sequence kernel: one CTA per (batch, head, tile of JT value columns).  Each
// consumer thread keeps R = dk / LPC rows of one column in registers for the
// whole sequence; LPC lanes share a column and combine their partial dot
// products with xor shuffles.  q, k, per-key decay and the v slice arrive
// through a 3-stage TMA ring fed by a producer warp (per-head scalars by
// cp.async on the same mbarrier); the o slice leaves through TMA stores.  The
// update of diag is fma(d_i, P_ij, k_i * v_j) with the product rounded first,
// the order of the single-precision definition, so its final state has the
// definition's bits.  Reductions use a fixed order, so every result depends
// only on the inputs and segment splits are bit-exact.
//
// Decode kernel (RWKV-7, T == 1): four (batch, head) states per CTA move as
// 16 KB bulk copies into shared memory, four lanes per state row update and
// read out with the sequence kernel's arithmetic, and the new states leave as
// bulk copies (in place allowed).
#include <algorithm>

#include "ptx.cuh"
#include "sn_internal.h"

namespace sn {

namespace {

constexpr int RS_TS = 16;       // time steps per stage
constexpr int RS_STAGES = 3;
constexpr int RS_OBUF = 3;      // output staging buffers

template <int KIND>
constexpr bool per_key_gate() { return KIND == RK_DIAG_KEY || KIND == RK_RWKV7; }
template <int KIND>
constexpr bool scalar_gate() { return KIND == RK_DIAG_HEAD || KIND == RK_DELTA; }

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

__device__ __forceinline__ float group_sum(float x, int lpc) {
    for (int o = lpc >> 1; o > 0; o >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// One time step of one state column held by a lane group of LPC lanes; each
// lane owns rows (m * LPC + sub) * 4 + c of the column (m < R4, c < 4).
// kr, gr, qr point at the step's k, per-key gate and q rows in shared memory;
// vj is the column's value, gsc the per-head scalar (dA or beta).  Returns this
// lane's partial of the unscaled readout; the caller reduces the partials over
// the lane group (group_sum per step, or reduce_scatter per stage -- both use
// the same addition tree, so the bits do not depend on which).
// Every operation is an explicit round-to-nearest intrinsic, so any kernel
// that calls this with the same lane layout produces the same bits.
template <int KIND, int R4, int LPC>
__device__ __forceinline__ float col_step(float (&P)[4 * R4], const float* kr, const float* gr,
                                          const float* qr, float vj, float gsc, int sub, bool want_o) {
    float kv[4 * R4];
#pragma unroll
    for (int m = 0; m < R4; ++m) {
        const float4 x = *reinterpret_cast<const float4*>(kr + (m * LPC + sub) * 4);
        kv[4 * m] = x.x; kv[4 * m + 1] = x.y; kv[4 * m + 2] = x.z; kv[4 * m + 3] = x.w;
    }
    if constexpr (KIND == RK_DIAG_KEY) {
#pragma unroll
        for (int m = 0; m < R4; ++m) {
            const float4 d = *reinterpret_cast<const float4*>(gr + (m * LPC + sub) * 4);
            P[4 * m] = __fmaf_rn(d.x, P[4 * m], __fmul_rn(kv[4 * m], vj));
            P[4 * m + 1] = __fmaf_rn(d.y, P[4 * m + 1], __fmul_rn(kv[4 * m + 1], vj));
            P[4 * m + 2] = __fmaf_rn(d.z, P[4 * m + 2], __fmul_rn(kv[4 * m + 2], vj));
            P[4 * m + 3] = __fmaf_rn(d.w, P[4 * m + 3], __fmul_rn(kv[4 * m + 3], vj));
        }
    } else if constexpr (KIND == RK_DIAG_HEAD) {
#pragma unroll
        for (int r = 0; r < 4 * R4; ++r) P[r] = __fmaf_rn(gsc, P[r], __fmul_rn(kv[r], vj));
    } else {
        // u = column . k: four partial chains, then the lane group
        float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
#pragma unroll
        for (int m = 0; m < R4; ++m) {
            u0 = __fmaf_rn(P[4 * m], kv[4 * m], u0);
            u1 = __fmaf_rn(P[4 * m + 1], kv[4 * m + 1], u1);
            u2 = __fmaf_rn(P[4 * m + 2], kv[4 * m + 2], u2);
            u3 = __fmaf_rn(P[4 * m + 3], kv[4 * m + 3], u3);
        }
        const float u = group_sum(__fadd_rn(__fadd_rn(u0, u1), __fadd_rn(u2, u3)), LPC);
        if constexpr (KIND == RK_DELTA) {
            const float delta = __fmul_rn(__fsub_rn(vj, u), gsc);
#pragma unroll
            for (int r = 0; r < 4 * R4; ++r) P[r] = __fmaf_rn(kv[r], delta, P[r]);
        } else {
            const float delta = __fsub_rn(vj, u);
#pragma unroll
            for (int m = 0; m < R4; ++m) {
                const float4 w = *reinterpret_cast<const float4*>(gr + (m * LPC + sub) * 4);
                P[4 * m] = __fmaf_rn(kv[4 * m], delta, __fmul_rn(P[4 * m], w.x));
                P[4 * m + 1] = __fmaf_rn(kv[4 * m + 1], delta, __fmul_rn(P[4 * m + 1], w.y));
                P[4 * m + 2] = __fmaf_rn(kv[4 * m + 2], delta, __fmul_rn(P[4 * m + 2], w.z));
                P[4 * m + 3] = __fmaf_rn(kv[4 * m + 3], delta, __fmul_rn(P[4 * m + 3], w.w));
            }
        }
    }
    if (!want_o) return 0.f;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int m = 0; m < R4; ++m) {
        const float4 x = *reinterpret_cast<const float4*>(qr + (m * LPC + sub) * 4);
        a0 = __fmaf_rn(P[4 * m], x.x, a0);
        a1 = __fmaf_rn(P[4 * m + 1], x.y, a1);
        a2 = __fmaf_rn(P[4 * m + 2], x.z, a2);
        a3 = __fmaf_rn(P[4 * m + 3], x.w, a3);
    }
    return __fadd_rn(__fadd_rn(a0, a1), __fadd_rn(a2, a3));
}

// Sum NV per-lane values over a group of LPC lanes by recursive halving: at
// offset o a lane keeps the half of its values that its bit o selects and adds
// its partner's copy of that half.  Afterwards v[e] (e < NV/LPC) holds the group
// sum of value index sub * (NV/LPC) + e.  The pairing (offsets LPC/2 .. 1) is
// the one group_sum uses, and addition is commutative, so every sum has the
// bits group_sum would give it.
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

template <int KIND, int DK, int LPC, int W>
__global__ void __launch_bounds__((W + 1) * 32)
recur_seq(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
          const __grid_constant__ CUtensorMap map_g, const __grid_constant__ CUtensorMap map_v,
          const __grid_constant__ CUtensorMap map_o, const SeqParams p) {
    constexpr int R = DK / LPC;            // rows per lane
    constexpr int R4 = R / 4;
    constexpr int CPW = 32 / LPC;          // columns per warp
    constexpr int JT = W * CPW;            // columns per CTA
    using L = SeqLayout<KIND, DK, JT>;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
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
            mbar_init(&empty[s], W);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == W) {
        // ------------------------------------------------ producer warp
        for (int kk = 0; kk < nst; ++kk) {
            const int slot = kk % RS_STAGES;
            if (kk >= RS_STAGES) {
                const bool ok = __all_sync(0xffffffffu, mbar_wait(&empty[slot], ((kk / RS_STAGES) - 1) & 1, p.wait_ns));
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
    const int jl = warp * CPW + gcol;                  // column within the tile
    const int j = jt0 + jl;                            // value column
    const size_t sbase = ((size_t)b * p.H + h) * (size_t)DK * p.dv;

    float P[R];
#pragma unroll
    for (int m = 0; m < R4; ++m) {
        const int r0 = (m * LPC + sub) * 4;
        if (p.S_in == nullptr) {
            P[4 * m] = P[4 * m + 1] = P[4 * m + 2] = P[4 * m + 3] = 0.f;
        } else if (KIND == RK_RWKV7) {                 // stored (dv, dk): row j, keys contiguous
            const float4 x = *reinterpret_cast<const float4*>(p.S_in + sbase + (size_t)j * DK + r0);
            P[4 * m] = x.x; P[4 * m + 1] = x.y; P[4 * m + 2] = x.z; P[4 * m + 3] = x.w;
        } else {                                       // stored (dk, dv)
#pragma unroll
            for (int c = 0; c < 4; ++c) P[4 * m + c] = p.S_in[sbase + (size_t)(r0 + c) * p.dv + j];
        }
    }

    bool failed = false;
    for (int kk = 0; kk < nst; ++kk) {
        const int slot = kk % RS_STAGES;
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[slot], (kk / RS_STAGES) & 1, p.wait_ns));
        if (!ok) {
            if (lane == 0) record_error(p.st, SN_E_TIMEOUT, (SN_K_RECUR_SEQ << 16) | 2);
            failed = true;
            break;
        }
        const unsigned char* sb = smem + slot * L::stage_bytes;
        const float* qs = reinterpret_cast<const float*>(sb + L::q_off);
        const float* ks = reinterpret_cast<const float*>(sb + L::k_off);
        const float* gs = reinterpret_cast<const float*>(sb + L::g_off);
        const float* vs = reinterpret_cast<const float*>(sb + L::v_off);
        float* os = reinterpret_cast<float*>(smem + L::o_off + (kk % RS_OBUF) * L::o_bytes);
        const int tn = min(RS_TS, T - kk * RS_TS);

        const bool want_o = p.has_o != 0;
        if (tn == RS_TS) {
            // Readout partials stay in registers for the whole stage and are
            // reduced once over the lane group, so no shuffle chain or store
            // sits between one step and the next.
            float ov[RS_TS];
#pragma unroll
            for (int i = 0; i < RS_TS; ++i)
                ov[i] = col_step<KIND, R4, LPC>(P, ks + i * DK, gs + i * DK, qs + i * DK, vs[i * JT + jl],
                                                scalar_gate<KIND>() ? gs[i] : 0.f, sub, want_o);
            if (want_o) {
                reduce_scatter<LPC, RS_TS>(ov, sub);
                constexpr int PER = RS_TS / LPC;
#pragma unroll
                for (int e = 0; e < PER; ++e) os[(sub * PER + e) * JT + jl] = __fmul_rn(ov[e], p.scale);
            }
        } else {
            for (int i = 0; i < tn; ++i) {
                const float part = col_step<KIND, R4, LPC>(P, ks + i * DK, gs + i * DK, qs + i * DK,
                                                           vs[i * JT + jl], scalar_gate<KIND>() ? gs[i] : 0.f, sub,
                                                           want_o);
                if (want_o) {
                    const float acc = group_sum(part, LPC);
                    if (sub == 0) os[i * JT + jl] = __fmul_rn(acc, p.scale);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        if (p.has_o) {
            fence_proxy_async_smem();
            // the store two stages back read the buffer the next stage writes
            if (threadIdx.x == 0) bulk_wait_read_allbut1();
            named_bar_sync(1, W * 32);
            if (threadIdx.x == 0) {
                tma_store_4d(&map_o, os, jt0, h, kk * RS_TS, b);
                bulk_commit();
            }
        }
    }
    if (threadIdx.x == 0) bulk_wait_all();
    if (failed || p.S_out == nullptr) return;
#pragma unroll
    for (int m = 0; m < R4; ++m) {
        const int r0 = (m * LPC + sub) * 4;
        if (KIND == RK_RWKV7) {
            *reinterpret_cast<float4*>(p.S_out + sbase + (size_t)j * DK + r0) =
                make_float4(P[4 * m], P[4 * m + 1], P[4 * m + 2], P[4 * m + 3]);
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) p.S_out[sbase + (size_t)(r0 + c) * p.dv + j] = P[4 * m + c];
        }
    }
}

template <int KIND, int DK, int LPC, int W>
cudaError_t run_seq(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, cudaStream_t stream) {
    constexpr int JT = W * (32 / LPC);
    using L = SeqLayout<KIND, DK, JT>;
    const int gdim = (KIND == RK_DIAG_KEY || KIND == RK_DIAG_HEAD) ? x.G : x.H;
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
    auto kern = recur_seq<KIND, DK, LPC, W>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    dim3 grid(x.dv / JT, x.H, x.B);
    kern<<<grid, (W + 1) * 32, L::smem, stream>>>(mq, mk, mg, mv, mo, p);
    return cudaGetLastError();
}

// Lanes per column: the diagonal-decay kinds have no reduction on the
// recurrence path, so they spread a column over more lanes (8 rows each) for
// more warps per SM; delta and RWKV-7 keep 16 rows per lane to shorten the
// per-step dot product that feeds the next state.  The CTA width (consumer
// warps) is chosen so the grid covers the SMs, or forced by
// SN_OPT_RECUR_TILE.
template <int KIND, int DK>
constexpr int lanes_per_col() {
    return (KIND == RK_DIAG_KEY || KIND == RK_DIAG_HEAD) ? DK / 8 : DK / 16;
}

template <int KIND, int DK>
cudaError_t dispatch_width(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count, int force_w,
                           cudaStream_t stream) {
    constexpr int LPC = lanes_per_col<KIND, DK>();
    constexpr int CPW = 32 / LPC;                      // columns per warp
    int w = force_w;
    if (w == 0) {
        // widest CTA that still gives at least one CTA per SM, else the narrowest
        w = 2;
        for (int cand : {8, 4}) {
            if (x.dv % (cand * CPW) != 0) continue;
            const int64_t ctas = (int64_t)x.B * x.H * (x.dv / (cand * CPW));
            if (ctas >= sm_count) { w = cand; break; }
        }
    }
    if (x.dv % (w * CPW) != 0) return cudaErrorInvalidValue;
    switch (w) {
        case 2: return run_seq<KIND, DK, LPC, 2>(x, st, wait_ns, stream);
        case 4: return run_seq<KIND, DK, LPC, 4>(x, st, wait_ns, stream);
        case 8: return run_seq<KIND, DK, LPC, 8>(x, st, wait_ns, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int KIND>
cudaError_t dispatch_seq(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count, int force_w,
                         cudaStream_t stream) {
    if (x.dk == 128) return dispatch_width<KIND, 128>(x, st, wait_ns, sm_count, force_w, stream);
    return dispatch_width<KIND, 64>(x, st, wait_ns, sm_count, force_w, stream);
}

// ============================================================ decode (T == 1)
constexpr int DEC_TILES = 4;                   // (b, h) states per CTA
constexpr int DEC_D = 64;                      // dk = dv = 64
constexpr uint32_t DEC_S_BYTES = DEC_D * DEC_D * 4;
constexpr uint32_t DEC_V_BYTES = DEC_D * 4;
// per tile: S (16 KB) then q, k, w, v rows (256 B each)
constexpr uint32_t DEC_TILE_BYTES = DEC_S_BYTES + 4 * DEC_V_BYTES;
constexpr size_t DEC_SMEM = DEC_TILES * DEC_TILE_BYTES + 8 + 128;
constexpr int DEC_THREADS = DEC_D * 4;       // 4 lanes per state row

__global__ void __launch_bounds__(DEC_THREADS, 3)
recur_decode_rwkv7(int BH, const float* __restrict__ q, const float* __restrict__ k,
                   const float* __restrict__ v, const float* __restrict__ w, const float* S_in, float* S_out,
                   float* __restrict__ o, SnDevStatus* st, uint64_t wait_ns) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + DEC_TILES * DEC_TILE_BYTES);
    const int tid = threadIdx.x;
    const int tile0 = blockIdx.x * DEC_TILES;
    const int ntile = min(DEC_TILES, BH - tile0);

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(bar, ntile * (S_in != nullptr ? DEC_TILE_BYTES : 4 * DEC_V_BYTES));
        for (int t = 0; t < ntile; ++t) {
            unsigned char* tb = smem + t * DEC_TILE_BYTES;
            const size_t bh = (size_t)(tile0 + t);
            if (S_in != nullptr) bulk_load(tb, S_in + bh * DEC_D * DEC_D, DEC_S_BYTES, bar);
            bulk_load(tb + DEC_S_BYTES + 0 * DEC_V_BYTES, q + bh * DEC_D, DEC_V_BYTES, bar);
            bulk_load(tb + DEC_S_BYTES + 1 * DEC_V_BYTES, k + bh * DEC_D, DEC_V_BYTES, bar);
            bulk_load(tb + DEC_S_BYTES + 2 * DEC_V_BYTES, w + bh * DEC_D, DEC_V_BYTES, bar);
            bulk_load(tb + DEC_S_BYTES + 3 * DEC_V_BYTES, v + bh * DEC_D, DEC_V_BYTES, bar);
        }
    }
    const bool ok = __syncthreads_and(mbar_wait(bar, 0, wait_ns));
    if (!ok) {
        if (tid == 0) {
            record_error(st, SN_E_TIMEOUT, (SN_K_RECUR_DECODE << 16) | 1);
            (void)mbar_wait(bar, 0, wait_ns);
        }
        return;
    }
    // Same lane layout and arithmetic as the sequence kernel for dk = 64
    // (4 lanes per state row, 16 keys each, col_step), so one decode step and
    // a one-step sequence call give identical bits.
    const int i = tid >> 2, sub = tid & 3;            // state row (value index), lane in group
    for (int t = 0; t < ntile; ++t) {
        float* S = reinterpret_cast<float*>(smem + t * DEC_TILE_BYTES);
        const float* qv = reinterpret_cast<const float*>(smem + t * DEC_TILE_BYTES + DEC_S_BYTES);
        const float* kv = qv + DEC_D;
        const float* wv = kv + DEC_D;
        const float* vv = wv + DEC_D;
        float4* row = reinterpret_cast<float4*>(S + i * DEC_D);
        float P[16];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float4 x = (S_in != nullptr) ? row[m * 4 + sub] : make_float4(0.f, 0.f, 0.f, 0.f);
            P[4 * m] = x.x; P[4 * m + 1] = x.y; P[4 * m + 2] = x.z; P[4 * m + 3] = x.w;
        }
        const float acc = group_sum(col_step<RK_RWKV7, 4, 4>(P, kv, wv, qv, vv[i], 0.f, sub, o != nullptr), 4);
#pragma unroll
        for (int m = 0; m < 4; ++m) row[m * 4 + sub] = make_float4(P[4 * m], P[4 * m + 1], P[4 * m + 2], P[4 * m + 3]);
        if (o != nullptr && sub == 0) o[(size_t)(tile0 + t) * DEC_D + i] = __fmul_rn(acc, 1.0f);
    }
    if (S_out == nullptr) return;
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
        for (int tt = 0; tt < ntile; ++tt)
            bulk_store(S_out + (size_t)(tile0 + tt) * DEC_D * DEC_D, smem + tt * DEC_TILE_BYTES, DEC_S_BYTES);
        bulk_commit();
        bulk_wait_all();
    }
}

}  // namespace

cudaError_t launch_recur_sequence(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count,
                                  int force_w, cudaStream_t stream) {
    switch (x.kind) {
        case RK_DIAG_KEY: return dispatch_seq<RK_DIAG_KEY>(x, st, wait_ns, sm_count, force_w, stream);
        case RK_DIAG_HEAD: return dispatch_seq<RK_DIAG_HEAD>(x, st, wait_ns, sm_count, force_w, stream);
        case RK_DELTA: return dispatch_seq<RK_DELTA>(x, st, wait_ns, sm_count, force_w, stream);
        case RK_RWKV7: return dispatch_seq<RK_RWKV7>(x, st, wait_ns, sm_count, force_w, stream);
        default: return cudaErrorInvalidValue;
    }
}

bool recur_decode_supported(const RecurArgs& x) {
    return x.kind == RK_RWKV7 && x.T == 1 && x.dk == DEC_D && x.dv == DEC_D;
}

cudaError_t launch_recur_decode(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count,
                                cudaStream_t stream) {
    (void)sm_count;
    static bool attr = false;
    if (!attr) {
        cudaError_t e =
            cudaFuncSetAttribute(recur_decode_rwkv7, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DEC_SMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const int BH = x.B * x.H;
    const int grid = (BH + DEC_TILES - 1) / DEC_TILES;
    recur_decode_rwkv7<<<grid, DEC_THREADS, DEC_SMEM, stream>>>(BH, x.q, x.k, x.v, x.g, x.S_in, x.S_out,
                                                                      x.o, st, wait_ns);
    return cudaGetLastError();
}

}  // namespace sn
