// recur_decode.cu -- batched single-step (T = 1) decode of the diagonal-decay
// kinds (GLA per-key and Mamba-2 per-head decays, plain and gated) and of the
// DeltaNet delta rule ("SunnyNet 工程化实录" §4.1-4.3; the single-step entry
// that must amortise its call, §2.4).
//
// A decode step reads each (b, h) state once, updates it and writes it back:
// it is bound by the state's bytes.  One thread owns one value column j of one
// state and holds its dk entries P[i][j] in registers, so the state streams in
// and out as coalesced rows (a warp covers 32 consecutive columns).  k, q and
// per-key decays of the CTA's states are staged in shared memory and read as
// broadcasts.
//
// Arithmetic: the update of each entry is the sequence kernel's (recur_seq.cuh):
// diag fma(d_i, P_ij, k_i v_j) with the product rounded first (k_i weighted by
// 1 - d_i in the gated kinds); delta u_j = sum_i P_ij k_i, delta_j = (v_j - u_j)
// beta, P_ij = fma(k_i, delta_j, P_ij).  Each dot product (u and the readout
// o_j = scale * sum_i P_ij q_i) is summed in the order the sequence kernel
// uses for the same call with R rows per lane: LPC = dk / R lanes, each
// running four chains over its rows (row mod 4) joined as (c0 + c1) +
// (c2 + c3), then the lanes pairwise at offsets LPC/2 .. 1.  A decode step
// therefore has the bits of a one-step sequence call.
#include "recur_seq.cuh"

namespace sn {
namespace {

constexpr int DD_THREADS = 256;

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

// sum_i p[i] x[i] in the sequence kernel's order with R rows per lane.  With
// HV = 2 a column is split over two threads (lanes l and l ^ 16): this thread
// holds the rows of the virtual lanes s in [hv * LPC/2, (hv + 1) * LPC/2) in
// p[0 .. DK/2), and the first join (offset LPC/2) is the pair's shuffle.
template <int DK, int R, int HV>
__device__ __forceinline__ float seq_dot(const float (&p)[DK / HV], const float* x, int hv) {
    constexpr int LPC = DK / R, LS = LPC / HV;
    float lane[LS];
#pragma unroll
    for (int sl = 0; sl < LS; ++sl) {
        const int s = hv * LS + sl;
        float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < R / 4; ++m)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = (m * LPC + s) * 4 + e;           // row of the state
                a[e] = __fmaf_rn(p[(m * LS + sl) * 4 + e], x[r], a[e]);
            }
        lane[sl] = __fadd_rn(__fadd_rn(a[0], a[1]), __fadd_rn(a[2], a[3]));
    }
    if (HV == 2) {
#pragma unroll
        for (int sl = 0; sl < LS; ++sl) lane[sl] = __fadd_rn(lane[sl], __shfl_xor_sync(0xffffffffu, lane[sl], 16));
    }
#pragma unroll
    for (int o = LS / 2; o > 0; o >>= 1)
#pragma unroll
        for (int sl = 0; sl < o; ++sl) lane[sl] = __fadd_rn(lane[sl], lane[sl + o]);
    return lane[0];
}

// Thread layout: HV threads per value column (2 for dk = 128, so a thread
// holds 64 entries); in a warp, lanes 0-15 and 16-31 take the two halves of
// the same 16 columns.
template <int KIND, int DK, int DV, int R>
__global__ void __launch_bounds__(DD_THREADS, 2) recur_decode_cols(const DecodeParams p) {
    constexpr int HV = DK == 128 ? 2 : 1;
    constexpr int PR = DK / HV;                       // state entries per thread
    constexpr int LPC = DK / R, LS = LPC / HV;
    constexpr int SPC = DD_THREADS / (HV * DV);       // states per CTA step
    __shared__ float sk[SPC][DK], sq[SPC][DK], sd[SPC][per_key_gate<KIND>() ? DK : 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hv = HV == 2 ? lane >> 4 : 0;
    const int cl = HV == 2 ? warp * 16 + (lane & 15) : tid;   // column-thread index in the CTA
    const int slot = cl / DV, j = cl % DV;
    const int BH = p.B * p.H;
    const int hpg = p.H / p.G;
    // row of this thread's e-th entry: entry (m * LS + sl) * 4 + e is row (m * LPC + hv * LS + sl) * 4 + e
    auto row_of = [&](int idx) {
        const int e = idx & 3, q = idx >> 2, m = q / LS, sl = q % LS;
        return (m * LPC + hv * LS + sl) * 4 + e;
    };
    for (int base = blockIdx.x * SPC; base < BH; base += gridDim.x * SPC) {
        __syncthreads();   // the previous step's readers are done with the staged vectors
        for (int idx = tid; idx < SPC * DK; idx += DD_THREADS) {
            const int sl = idx / DK, i = idx % DK, bh = base + sl;
            if (bh < BH) {
                const int b = bh / p.H, h = bh % p.H;
                const size_t qk = ((size_t)b * p.G + h / hpg) * DK + i;
                sk[sl][i] = __ldg(p.k + qk);
                sq[sl][i] = p.o != nullptr ? __ldg(p.q + qk) : 0.f;
                if constexpr (per_key_gate<KIND>()) sd[sl][i] = __ldg(p.g + (size_t)bh * DK + i);
            }
        }
        __syncthreads();
        const int bh = base + slot;
        if (bh >= BH) continue;                       // a whole pair of lanes leaves together
        const size_t sbase = (size_t)bh * DK * DV + j;
        float pc[PR];
#pragma unroll
        for (int t = 0; t < PR; ++t) pc[t] = p.S_in != nullptr ? p.S_in[sbase + (size_t)row_of(t) * DV] : 0.f;
        const float vj = __ldg(p.v + (size_t)bh * DV + j);
        const float* kx = sk[slot];
        if constexpr (diag_kind<KIND>()) {
            const float dh = per_key_gate<KIND>() ? 0.f : __ldg(p.g + bh);
#pragma unroll
            for (int t = 0; t < PR; ++t) {
                const int i = row_of(t);
                const float di = per_key_gate<KIND>() ? sd[slot][i] : dh;
                float ki = kx[i];
                if constexpr (gated_injection<KIND>()) ki = __fmul_rn(__fsub_rn(1.0f, di), ki);
                pc[t] = __fmaf_rn(di, pc[t], __fmul_rn(ki, vj));
            }
        } else {   // RK_DELTA
            const float u = seq_dot<DK, R, HV>(pc, kx, hv);
            const float delta = __fmul_rn(__fadd_rn(vj, -u), __ldg(p.g + bh));
#pragma unroll
            for (int t = 0; t < PR; ++t) pc[t] = __fmaf_rn(kx[row_of(t)], delta, pc[t]);
        }
        if (p.o != nullptr) {
            const float acc = seq_dot<DK, R, HV>(pc, sq[slot], hv);
            if (hv == 0) p.o[(size_t)bh * DV + j] = __fmul_rn(acc, p.scale);
        }
        if (p.S_out != nullptr) {
#pragma unroll
            for (int t = 0; t < PR; ++t) p.S_out[sbase + (size_t)row_of(t) * DV] = pc[t];
        }
    }
}

template <int KIND, int R>
cudaError_t run_decode_rows(const RecurArgs& x, const DecodeParams& p, int sm_count, cudaStream_t s) {
    const int BH = x.B * x.H;
    auto go = [&](auto kern, int dv) -> cudaError_t {
        const int spc = DD_THREADS / ((x.dk == 128 ? 2 : 1) * dv);
        const int grid = std::min((BH + spc - 1) / spc, 4 * sm_count);
        kern<<<grid, DD_THREADS, 0, s>>>(p);
        return cudaGetLastError();
    };
    if (x.dk == 128)
        return x.dv == 128 ? go(recur_decode_cols<KIND, 128, 128, R>, 128) : go(recur_decode_cols<KIND, 128, 64, R>, 64);
    return x.dv == 128 ? go(recur_decode_cols<KIND, 64, 128, R>, 128) : go(recur_decode_cols<KIND, 64, 64, R>, 64);
}

// The rows per lane whose summation order the decode reproduces: the sequence
// kernel's choice for the same call (recur_diag.cu: 8 when the problem gives at
// least 4 warps per SM, else 4; the delta rule always 8), so a call split into
// single steps and longer segments gives the same bits.
template <int KIND>
cudaError_t run_decode_kind(const RecurArgs& x, const DecodeParams& p, int sm_count, cudaStream_t s) {
    if constexpr (KIND == RK_DELTA) {
        return run_decode_rows<KIND, 8>(x, p, sm_count, s);
    } else {
        if (diag_eight_rows(x, sm_count)) return run_decode_rows<KIND, 8>(x, p, sm_count, s);
        return run_decode_rows<KIND, 4>(x, p, sm_count, s);
    }
}

}  // namespace

bool recur_decode_cols_supported(const RecurArgs& x) {
    const bool kind_ok = x.kind == RK_DIAG_KEY || x.kind == RK_DIAG_HEAD || x.kind == RK_DIAG_KEY_GATED ||
                         x.kind == RK_DIAG_HEAD_GATED || x.kind == RK_DELTA;
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
        default: return run_decode_kind<RK_DELTA>(x, p, sm_count, s);
    }
}

}  // namespace sn
