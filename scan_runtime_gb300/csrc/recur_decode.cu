// recur_decode.cu -- batched single-step (T = 1) decode of the diagonal-decay
// kinds (GLA per-key and Mamba-2 per-head decays, plain and gated), of the
// DeltaNet delta rule and of RWKV-7 ("SunnyNet 工程化实录" §4.1-4.3, §5.1; the
// single-step entry that must amortise its call, §2.4).
//
// A decode step reads each (b, h) state once, updates it and writes it back:
// it is bound by the state's bytes.  A thread owns four adjacent value
// columns j0 .. j0 + 3 of one state over 16 key rows, so the state moves as
// 16-byte loads and stores (a row segment of four columns per instruction),
// TPG = dk / 16 threads cover a column quad, and a warp covers 32 / TPG quads.
// k, q and per-key decays of the CTA's states are staged in shared memory and
// read as broadcasts.  The state loads of a CTA's next states are issued
// before the arithmetic of the current ones.
//
// Arithmetic: the update of each entry is the sequence kernel's (recur_seq.cuh):
// diag fma(d_i, P_ij, k_i v_j) with the product rounded first (k_i weighted by
// 1 - d_i in the gated kinds); delta u_j = sum_i P_ij k_i, delta_j = (v_j - u_j)
// beta, P_ij = fma(k_i, delta_j, P_ij); RWKV-7 (P = S^T, S stored value-major)
// delta_j = v_j - u_j, P_ij = fma(k_i, delta_j, P_ij w_i).  Each dot product (u and the readout
// o_j = scale * sum_i P_ij q_i) is summed in the order the sequence kernel
// uses for the same call with R rows per lane: LPC = dk / R virtual lanes,
// each running four chains over its rows (row mod 4) joined as
// (c0 + c1) + (c2 + c3), then the virtual lanes pairwise at offsets LPC/2 ..
// 1.  Thread tau of a quad holds the virtual lanes s = tau (mod TPG), so the
// offsets LPC/2 .. TPG join inside the thread and TPG/2 .. 1 across the
// quad's threads (xor shuffles).  A decode step therefore has the bits of a
// one-step sequence call.
#include "recur_seq.cuh"

namespace sn {
namespace {

constexpr int DD_THREADS = 256;
constexpr int DD_ROWS = 16;          // key rows per thread
#ifndef SN_DECODE_PREF
#define SN_DECODE_PREF 1
#endif
constexpr bool DECODE_PREF = SN_DECODE_PREF != 0;

struct DecodeParams {
    int B, H, G;
    float scale;
    const float* q;      // (B, 1, G, dk)
    const float* k;      // (B, 1, G, dk)
    const float* v;      // (B, 1, H, dv)
    const float* g;      // per-key decays (B, 1, H, dk), or per-head decays / beta (B, 1, H)
    const float* S_in;   // (B, H, dk, dv), NULL = zeros
    float* S_out;        // may equal S_in
    float* o;            // (B, 1, H, dv), may be NULL
};

// Thread tau's rows: entry idx = (kk * (R/4) + m) * 4 + e is row
// (m * LPC + tau + kk * TPG) * 4 + e of the state (virtual lane tau + kk TPG).
template <int DK, int R>
struct QuadRows {
    static constexpr int LPC = DK / R, TPG = DK / DD_ROWS, NL = LPC / TPG;
    static_assert(NL * TPG == LPC && NL * R == DD_ROWS, "row split");
    __device__ static int row(int tau, int idx) {
        const int e = idx & 3, q = idx >> 2, m = q % (R / 4), kk = q / (R / 4);
        return (m * LPC + tau + kk * TPG) * 4 + e;
    }
};

// sum_i P[i][c] x_i for the thread's four columns in the sequence kernel's
// order (see the file comment); every thread of the quad gets the totals.
template <int DK, int R>
__device__ __forceinline__ float4 quad_dot(const float4 (&P)[DD_ROWS], const float* x, int tau) {
    using Q = QuadRows<DK, R>;
    constexpr int NL = Q::NL, TPG = Q::TPG;
    float2 lo[NL], hi[NL];                    // columns (0, 1) and (2, 3), per virtual lane
#pragma unroll
    for (int kk = 0; kk < NL; ++kk) {
        float2 a[4][2];
#pragma unroll
        for (int e = 0; e < 4; ++e) a[e][0] = a[e][1] = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < R / 4; ++m)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int idx = (kk * (R / 4) + m) * 4 + e;
                const float2 xr = f2(x[Q::row(tau, idx)]);
                a[e][0] = __ffma2_rn(make_float2(P[idx].x, P[idx].y), xr, a[e][0]);
                a[e][1] = __ffma2_rn(make_float2(P[idx].z, P[idx].w), xr, a[e][1]);
            }
        lo[kk] = __fadd2_rn(__fadd2_rn(a[0][0], a[1][0]), __fadd2_rn(a[2][0], a[3][0]));
        hi[kk] = __fadd2_rn(__fadd2_rn(a[0][1], a[1][1]), __fadd2_rn(a[2][1], a[3][1]));
    }
    // virtual-lane offsets LPC/2 .. TPG: inside the thread
#pragma unroll
    for (int o = NL / 2; o > 0; o >>= 1)
#pragma unroll
        for (int kk = 0; kk < o; ++kk) {
            lo[kk] = __fadd2_rn(lo[kk], lo[kk + o]);
            hi[kk] = __fadd2_rn(hi[kk], hi[kk + o]);
        }
    // offsets TPG/2 .. 1: across the quad's threads
    float4 s = make_float4(lo[0].x, lo[0].y, hi[0].x, hi[0].y);
#pragma unroll
    for (int o = TPG / 2; o > 0; o >>= 1) {
        s.x = __fadd_rn(s.x, __shfl_xor_sync(0xffffffffu, s.x, o));
        s.y = __fadd_rn(s.y, __shfl_xor_sync(0xffffffffu, s.y, o));
        s.z = __fadd_rn(s.z, __shfl_xor_sync(0xffffffffu, s.z, o));
        s.w = __fadd_rn(s.w, __shfl_xor_sync(0xffffffffu, s.w, o));
    }
    return s;
}

// PREF: the next states' loads are issued before this step's stores (one CTA
// per SM, registers for both); otherwise load, update, store in turn with two
// CTAs per SM.
template <int KIND, int DK, int DV, int R, bool PREF>
__global__ void __launch_bounds__(DD_THREADS, PREF ? 1 : 2) recur_decode_cols(const DecodeParams p) {
    using Q = QuadRows<DK, R>;
    constexpr int TPG = Q::TPG;
    constexpr int QUADS = DV / 4;                      // column quads per state
    constexpr int SPC = DD_THREADS / (QUADS * TPG);    // states per CTA step
    static_assert(SPC >= 1 && SPC * QUADS * TPG == DD_THREADS, "thread split");
    __shared__ float sk[SPC][DK], sq[SPC][DK], sd[SPC][per_key_gate<KIND>() ? DK : 1];
    const int tid = threadIdx.x;
    const int tau = tid % TPG;                         // thread within the quad
    const int qd = (tid / TPG) % QUADS, slot = tid / (TPG * QUADS);
    const int j0 = 4 * qd;
    const int BH = p.B * p.H;
    const int hpg = p.H / p.G;
    const int step = gridDim.x * SPC;

    static_assert(SPC * DK <= DD_THREADS, "one staged vector element per thread");
    constexpr bool TR = KIND == RK_RWKV7;              // S stored (dv, dk): keys contiguous
    // The thread's entries as P[t] = its four columns at row Q::row(tau, t).
    // Stored transposed, four consecutive rows t = 4 blk + e of a column are
    // one 16-byte run; four of them are transposed in registers.
    auto state_load = [&](const float* S, int bh, float4 (&P)[DD_ROWS]) {
        if constexpr (!TR) {
#pragma unroll
            for (int t = 0; t < DD_ROWS; ++t)
                P[t] = *reinterpret_cast<const float4*>(S + ((size_t)bh * DK + Q::row(tau, t)) * DV + j0);
        } else {
#pragma unroll
            for (int blk = 0; blk < DD_ROWS / 4; ++blk) {
                const int r0 = Q::row(tau, 4 * blk);
                float4 c[4];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    c[cc] = *reinterpret_cast<const float4*>(S + ((size_t)bh * DV + j0 + cc) * DK + r0);
                P[4 * blk + 0] = make_float4(c[0].x, c[1].x, c[2].x, c[3].x);
                P[4 * blk + 1] = make_float4(c[0].y, c[1].y, c[2].y, c[3].y);
                P[4 * blk + 2] = make_float4(c[0].z, c[1].z, c[2].z, c[3].z);
                P[4 * blk + 3] = make_float4(c[0].w, c[1].w, c[2].w, c[3].w);
            }
        }
    };
    auto state_store = [&](float* S, int bh, const float4 (&P)[DD_ROWS]) {
        if constexpr (!TR) {
#pragma unroll
            for (int t = 0; t < DD_ROWS; ++t)
                *reinterpret_cast<float4*>(S + ((size_t)bh * DK + Q::row(tau, t)) * DV + j0) = P[t];
        } else {
#pragma unroll
            for (int blk = 0; blk < DD_ROWS / 4; ++blk) {
                const int r0 = Q::row(tau, 4 * blk);
                const float4 a = P[4 * blk], b = P[4 * blk + 1], c = P[4 * blk + 2], d = P[4 * blk + 3];
                *reinterpret_cast<float4*>(S + ((size_t)bh * DV + j0 + 0) * DK + r0) = make_float4(a.x, b.x, c.x, d.x);
                *reinterpret_cast<float4*>(S + ((size_t)bh * DV + j0 + 1) * DK + r0) = make_float4(a.y, b.y, c.y, d.y);
                *reinterpret_cast<float4*>(S + ((size_t)bh * DV + j0 + 2) * DK + r0) = make_float4(a.z, b.z, c.z, d.z);
                *reinterpret_cast<float4*>(S + ((size_t)bh * DV + j0 + 3) * DK + r0) = make_float4(a.w, b.w, c.w, d.w);
            }
        }
    };
    float4 P[DD_ROWS];
    float4 vj;                     // this thread's four values of v
    float gh, kr, qr, dr;          // the per-head scalar; this thread's staged k, q, decay element
    // Issue the loads of the states at `base` (the thread's rows of them) and
    // of their vectors into registers.
    auto load_step = [&](int base) {
        const int bh = base + slot;
        if (bh < BH && p.S_in != nullptr) {
            state_load(p.S_in, bh, P);
        } else {
#pragma unroll
            for (int t = 0; t < DD_ROWS; ++t) P[t] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        vj = make_float4(0.f, 0.f, 0.f, 0.f);
        gh = 0.f;
        if (bh < BH) {
            vj = __ldg(reinterpret_cast<const float4*>(p.v + (size_t)bh * DV + j0));
            if constexpr (!per_key_gate<KIND>()) gh = __ldg(p.g + bh);
        }
        kr = qr = dr = 0.f;
        const int sl = tid / DK, i = tid % DK, vbh = base + sl;
        if (tid < SPC * DK && vbh < BH) {
            const int b = vbh / p.H, h = vbh % p.H;
            const size_t qk = ((size_t)b * p.G + h / hpg) * DK + i;
            kr = __ldg(p.k + qk);
            qr = p.o != nullptr ? __ldg(p.q + qk) : 0.f;
            if constexpr (per_key_gate<KIND>()) dr = __ldg(p.g + (size_t)vbh * DK + i);
        }
    };
    int base = blockIdx.x * SPC;
    if (PREF && base < BH) load_step(base);
    for (; base < BH; base += step) {
        if (!PREF) load_step(base);
        __syncthreads();   // the previous step's readers are done with the staged vectors
        if (tid < SPC * DK) {
            const int sl = tid / DK, i = tid % DK;
            sk[sl][i] = kr;
            sq[sl][i] = qr;
            if constexpr (per_key_gate<KIND>()) sd[sl][i] = dr;
        }
        __syncthreads();
        const int bh = base + slot;
        const bool live = bh < BH;
        const float* kx = sk[slot];
        if constexpr (diag_kind<KIND>()) {
            const float2 vlo = make_float2(vj.x, vj.y), vhi = make_float2(vj.z, vj.w);
#pragma unroll
            for (int t = 0; t < DD_ROWS; ++t) {
                const int i = Q::row(tau, t);
                const float di = per_key_gate<KIND>() ? sd[slot][i] : gh;
                float ki = kx[i];
                if constexpr (gated_injection<KIND>()) ki = __fmul_rn(__fsub_rn(1.0f, di), ki);
                const float2 lo = __ffma2_rn(f2(di), make_float2(P[t].x, P[t].y), __fmul2_rn(f2(ki), vlo));
                const float2 hi = __ffma2_rn(f2(di), make_float2(P[t].z, P[t].w), __fmul2_rn(f2(ki), vhi));
                P[t] = make_float4(lo.x, lo.y, hi.x, hi.y);
            }
        } else {   // RK_DELTA, RK_RWKV7
            const float4 u = quad_dot<DK, R>(P, kx, tau);
            float2 dlo = __fadd2_rn(make_float2(vj.x, vj.y), make_float2(-u.x, -u.y));   // v - u, exactly
            float2 dhi = __fadd2_rn(make_float2(vj.z, vj.w), make_float2(-u.z, -u.w));
            if constexpr (KIND == RK_DELTA) {
                dlo = __fmul2_rn(dlo, f2(gh));
                dhi = __fmul2_rn(dhi, f2(gh));
            }
#pragma unroll
            for (int t = 0; t < DD_ROWS; ++t) {
                const int i = Q::row(tau, t);
                const float2 ki = f2(kx[i]);
                float2 lo = make_float2(P[t].x, P[t].y), hi = make_float2(P[t].z, P[t].w);
                if constexpr (KIND == RK_RWKV7) {
                    const float2 wi = f2(sd[slot][i]);
                    lo = __fmul2_rn(lo, wi);
                    hi = __fmul2_rn(hi, wi);
                }
                lo = __ffma2_rn(ki, dlo, lo);
                hi = __ffma2_rn(ki, dhi, hi);
                P[t] = make_float4(lo.x, lo.y, hi.x, hi.y);
            }
        }
        if (p.o != nullptr) {
            const float4 acc = quad_dot<DK, R>(P, sq[slot], tau);
            if (live && tau == 0)
                *reinterpret_cast<float4*>(p.o + (size_t)bh * DV + j0) =
                    make_float4(__fmul_rn(acc.x, p.scale), __fmul_rn(acc.y, p.scale), __fmul_rn(acc.z, p.scale),
                                __fmul_rn(acc.w, p.scale));
        }
        float4 Pn[DD_ROWS];
#pragma unroll
        for (int t = 0; t < DD_ROWS; ++t) Pn[t] = P[t];
        // (PREF) the next states' loads go out before this step's stores
        if (PREF && base + step < BH) load_step(base + step);
        if (live && p.S_out != nullptr) state_store(p.S_out, bh, Pn);
    }
}

template <int KIND, int R, bool PREF = DECODE_PREF>
cudaError_t run_decode_rows(const RecurArgs& x, const DecodeParams& p, int sm_count, cudaStream_t s) {
    const int BH = x.B * x.H;
    auto go = [&](auto kern, int dk, int dv) -> cudaError_t {
        const int spc = DD_THREADS / ((dv / 4) * (dk / DD_ROWS));
        const int grid = std::min((BH + spc - 1) / spc, (PREF ? 1 : 2) * sm_count);
        kern<<<grid, DD_THREADS, 0, s>>>(p);
        return cudaGetLastError();
    };
    if (x.dk == 128)
        return x.dv == 128 ? go(recur_decode_cols<KIND, 128, 128, R, PREF>, 128, 128)
                           : go(recur_decode_cols<KIND, 128, 64, R, PREF>, 128, 64);
    return x.dv == 128 ? go(recur_decode_cols<KIND, 64, 128, R, PREF>, 64, 128)
                       : go(recur_decode_cols<KIND, 64, 64, R, PREF>, 64, 64);
}

// The rows per lane whose summation order the decode reproduces: the sequence
// kernel's choice for the same call (recur_seq.cuh: for the diagonal kinds 8
// when the problem gives at least 4 warps per SM, else 4; the delta rule and
// RWKV-7 always 8), so a call split into single steps and longer segments
// gives the same bits.
template <int KIND>
cudaError_t run_decode_kind(const RecurArgs& x, const DecodeParams& p, int sm_count, cudaStream_t s) {
    if constexpr (KIND == RK_DELTA || KIND == RK_RWKV7) {
        return run_decode_rows<KIND, 8>(x, p, sm_count, s);
    } else {
        if (diag_eight_rows(x, sm_count)) return run_decode_rows<KIND, 8>(x, p, sm_count, s);
        return run_decode_rows<KIND, 4>(x, p, sm_count, s);
    }
}

}  // namespace

bool recur_decode_cols_supported(const RecurArgs& x) {
    const bool kind_ok = x.kind == RK_DIAG_KEY || x.kind == RK_DIAG_HEAD || x.kind == RK_DIAG_KEY_GATED ||
                         x.kind == RK_DIAG_HEAD_GATED || x.kind == RK_DELTA || x.kind == RK_RWKV7;
    return kind_ok && x.T == 1 && (x.dk == 64 || x.dk == 128) && (x.dv == 64 || x.dv == 128);
}

cudaError_t launch_recur_decode_cols(const RecurArgs& x, int sm_count, cudaStream_t s) {
    DecodeParams p;
    p.B = x.B;
    p.H = x.H;
    p.G = x.G;
    p.scale = x.scale;
    p.q = x.q;
    p.k = x.k;
    p.v = x.v;
    p.g = x.g;
    p.S_in = x.S_in;
    p.S_out = x.S_out;
    p.o = x.o;
    switch (x.kind) {
        case RK_DIAG_KEY: return run_decode_kind<RK_DIAG_KEY>(x, p, sm_count, s);
        case RK_DIAG_HEAD: return run_decode_kind<RK_DIAG_HEAD>(x, p, sm_count, s);
        case RK_DIAG_KEY_GATED: return run_decode_kind<RK_DIAG_KEY_GATED>(x, p, sm_count, s);
        case RK_DIAG_HEAD_GATED: return run_decode_kind<RK_DIAG_HEAD_GATED>(x, p, sm_count, s);
        case RK_RWKV7: return run_decode_kind<RK_RWKV7>(x, p, sm_count, s);
        default: return run_decode_kind<RK_DELTA>(x, p, sm_count, s);
    }
}

}  // namespace sn
