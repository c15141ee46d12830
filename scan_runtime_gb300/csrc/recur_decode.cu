// recur_decode.cu -- batched single-step (T = 1) decode of the diagonal-decay
// kinds (GLA per-key and Mamba-2 per-head decays, plain and gated), of the
// DeltaNet delta rule and of RWKV-7 ("SunnyNet 工程化实录" §4.1-4.3, §5.1; the
// single-step entry that must amortise its call, §2.4).
//
// A decode step reads each (b, h) state once, updates it and writes it back:
// it is bound by the state's bytes.  A persistent CTA per SM streams its
// states through a ring of shared-memory stages (192 KB in all), each filled
// by one bulk copy (cp.async.bulk, completion on the stage's mbarrier) before
// it is used, so the copy engine keeps 128 KB or more per SM in flight while
// the threads update the current stage.  A thread owns four adjacent value
// columns j0 .. j0 + 3 of one state over ROWS key rows: it reads them from
// the stage as 16-byte words, updates them in registers and stores them to
// the state's place in global memory as 16-byte words.  TPG = dk / ROWS
// threads cover a column quad.  In the (dk, dv) layout the quads of a warp
// are its fastest lane index (a warp's 16-byte reads of one row are
// contiguous); in RWKV-7's transposed (dv, dk) layout the threads of a quad
// are (their rows are contiguous).  k, q and per-key decays of the step's
// states are staged in shared memory and read as broadcasts; they, v and the
// per-head scalars are loaded one step ahead into registers.
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
    SnDevStatus* st;
    uint64_t wait_ns;
};

// The tile: ROWS = 16 key rows x 4 value columns per thread, so a step covers
// SPC = THREADS / ((dv / 4) (dk / 16)) states, and 192 KB of such stages are
// in flight.  256 threads (64 KB steps, three stages), except 64 x 64 states:
// 192 threads, three states (48 KB) per step in four stages, so the steps
// split more evenly over the SMs.  (Eight rows at dk = 64, 32 KB steps in six
// stages, measured slower: RWKV-7 decode 0.814 against 0.837 of HBM.)
template <int DK, int DV>
struct RingShape {
    static constexpr int ROWS = 16;
    static constexpr int THREADS = DK == 64 && DV == 64 ? 192 : 256;
    static constexpr int TPG = DK / ROWS;               // threads per column quad
    static constexpr int QUADS = DV / 4;                // column quads per state
    static constexpr int PER_STATE = QUADS * TPG;       // threads per state
    static constexpr int SPC = THREADS / PER_STATE;     // states per step
    static constexpr int QPW = 32 / TPG;                // column quads per warp
    static constexpr uint32_t STATE_BYTES = (uint32_t)DK * DV * 4;
    static constexpr uint32_t STAGE_BYTES = SPC * STATE_BYTES;
    static constexpr int NS = (int)(196608u / STAGE_BYTES);   // stages: 192 KB in all
    static constexpr size_t smem = (size_t)NS * STAGE_BYTES + 64 + 128;   // + barriers, alignment slack
    static_assert(PER_STATE % 32 == 0 && SPC * PER_STATE == THREADS, "thread split");
    static_assert(STAGE_BYTES == (uint32_t)THREADS * ROWS * 16 && NS <= 8, "stages");
};

// Thread tau's ROWS rows: entry idx = (kk * (R/4) + m) * 4 + e is row
// (m * LPC + tau + kk * TPG) * 4 + e of the state (virtual lane tau + kk TPG).
template <int DK, int R, int ROWS>
struct QuadRows {
    static constexpr int LPC = DK / R, TPG = DK / ROWS, NL = LPC / TPG;
    static_assert(NL * TPG == LPC && NL * R == ROWS, "row split");
    __device__ static int row(int tau, int idx) {
        const int e = idx & 3, q = idx >> 2, m = q % (R / 4), kk = q / (R / 4);
        return (m * LPC + tau + kk * TPG) * 4 + e;
    }
};

// sum_i P[i][c] x_i for the thread's four columns in the sequence kernel's
// order (see the file comment); every thread of the quad gets the totals.
// The quad's threads are TS lanes apart.
template <int DK, int R, int ROWS, int TS>
__device__ __forceinline__ float4 quad_dot(const float4 (&P)[ROWS], const float* x, int tau) {
    using Q = QuadRows<DK, R, ROWS>;
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
        s.x = __fadd_rn(s.x, __shfl_xor_sync(0xffffffffu, s.x, o * TS));
        s.y = __fadd_rn(s.y, __shfl_xor_sync(0xffffffffu, s.y, o * TS));
        s.z = __fadd_rn(s.z, __shfl_xor_sync(0xffffffffu, s.z, o * TS));
        s.w = __fadd_rn(s.w, __shfl_xor_sync(0xffffffffu, s.w, o * TS));
    }
    return s;
}

template <int KIND, int DK, int DV, int R>
__global__ void __launch_bounds__(RingShape<DK, DV>::THREADS, 1) recur_decode_ring(const DecodeParams p) {
    using S = RingShape<DK, DV>;
    constexpr int ROWS = S::ROWS, TPG = S::TPG, SPC = S::SPC, QPW = S::QPW, NS = S::NS;
    using Q = QuadRows<DK, R, ROWS>;
    constexpr bool TR = KIND == RK_RWKV7;              // S stored (dv, dk): keys contiguous
    constexpr int TS = TR ? 1 : QPW;                   // lane distance of a quad's threads
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = smem_align<128>(smem_raw);
    float* stages = reinterpret_cast<float*>(base);
    uint64_t* full = reinterpret_cast<uint64_t*>(base + (size_t)NS * S::STAGE_BYTES);
    __shared__ float sk[SPC][DK], sq[SPC][DK], sd[SPC][per_key_gate<KIND>() ? DK : 1];
    static_assert(SPC * DK <= S::THREADS, "one staged vector element per thread");

    const int tid = threadIdx.x;
    const int slot = tid / S::PER_STATE, local = tid % S::PER_STATE;
    const int lw = local >> 5, ln = local & 31;
    const int tau = TR ? ln % TPG : ln / QPW;          // thread within the quad
    const int qd = lw * QPW + (TR ? ln / TPG : ln % QPW);
    const int j0 = 4 * qd;
    const int BH = p.B * p.H;
    const int hpg = p.H / p.G;
    const int nsteps = (BH + SPC - 1) / SPC;
    const int grid = gridDim.x;
    const int mine = (int)blockIdx.x < nsteps ? (nsteps - 1 - (int)blockIdx.x) / grid + 1 : 0;
    const bool have_state = p.S_in != nullptr;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // thread 0: the bulk copy of local step n's states into stage n mod NS
    auto issue = [&](int n) {
        const int first = ((int)blockIdx.x + n * grid) * SPC;
        const uint32_t bytes = (uint32_t)min(SPC, BH - first) * S::STATE_BYTES;
        uint64_t* bar = &full[n % NS];
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load(stages + (size_t)(n % NS) * (S::STAGE_BYTES / 4), p.S_in + (size_t)first * DK * DV, bytes, bar);
    };
    int issued = 0;   // thread 0's count of local steps whose copy went out
    if (have_state && tid == 0)
        for (; issued < min(NS, mine); ++issued) issue(issued);

    // the step's vectors, loaded one step ahead: v and the per-head scalar of
    // this thread's state, one element of k, q and the per-key decays
    float4 vj = make_float4(0.f, 0.f, 0.f, 0.f);
    float gh = 0.f, kr = 0.f, qr = 0.f, dr = 0.f;
    auto load_vec = [&](int gs) {
        const int bh = gs * SPC + slot;
        vj = make_float4(0.f, 0.f, 0.f, 0.f);
        gh = 0.f;
        if (bh < BH) {
            vj = __ldg(reinterpret_cast<const float4*>(p.v + (size_t)bh * DV + j0));
            if constexpr (!per_key_gate<KIND>()) gh = __ldg(p.g + bh);
        }
        kr = qr = dr = 0.f;
        const int sl = tid / DK, i = tid % DK, vbh = gs * SPC + sl;
        if (tid < SPC * DK && vbh < BH) {
            const int b = vbh / p.H, h = vbh % p.H;
            const size_t qk = ((size_t)b * p.G + h / hpg) * DK + i;
            kr = __ldg(p.k + qk);
            qr = p.o != nullptr ? __ldg(p.q + qk) : 0.f;
            if constexpr (per_key_gate<KIND>()) dr = __ldg(p.g + (size_t)vbh * DK + i);
        }
    };
    if (mine > 0) load_vec(blockIdx.x);

    bool ok = true;
    int n = 0;
    for (; n < mine; ++n) {
        const int gs = (int)blockIdx.x + n * grid;
        __syncthreads();   // the previous step's readers are done with its stage and the staged vectors
        if (have_state && tid == 0 && n > 0 && issued < mine) {
            fence_proxy_async_smem();   // those reads before the copy's writes
            issue(issued);              // into the stage step n - 1 used
            ++issued;
        }
        if (tid < SPC * DK) {
            const int sl = tid / DK, i = tid % DK;
            sk[sl][i] = kr;
            sq[sl][i] = qr;
            if constexpr (per_key_gate<KIND>()) sd[sl][i] = dr;
        }
        const float4 vc = vj;
        const float gc = gh;
        if (n + 1 < mine) load_vec(gs + grid);
        const bool got = !have_state || mbar_wait(&full[n % NS], (uint32_t)(n / NS) & 1u, p.wait_ns);
        ok = __syncthreads_and(got);
        if (!ok) break;

        const int bh = gs * SPC + slot;
        const bool live = bh < BH;
        const float* st = stages + (size_t)(n % NS) * (S::STAGE_BYTES / 4) + (size_t)slot * DK * DV;
        float4 P[ROWS];
        if (!have_state) {
#pragma unroll
            for (int t = 0; t < ROWS; ++t) P[t] = make_float4(0.f, 0.f, 0.f, 0.f);
        } else if constexpr (!TR) {
#pragma unroll
            for (int t = 0; t < ROWS; ++t) P[t] = *reinterpret_cast<const float4*>(st + Q::row(tau, t) * DV + j0);
        } else {
            // four consecutive rows of a column are one 16-byte word; four
            // columns' words are transposed in registers
#pragma unroll
            for (int blk = 0; blk < ROWS / 4; ++blk) {
                const int r0 = Q::row(tau, 4 * blk);
                float4 c[4];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) c[cc] = *reinterpret_cast<const float4*>(st + (j0 + cc) * DK + r0);
                P[4 * blk + 0] = make_float4(c[0].x, c[1].x, c[2].x, c[3].x);
                P[4 * blk + 1] = make_float4(c[0].y, c[1].y, c[2].y, c[3].y);
                P[4 * blk + 2] = make_float4(c[0].z, c[1].z, c[2].z, c[3].z);
                P[4 * blk + 3] = make_float4(c[0].w, c[1].w, c[2].w, c[3].w);
            }
        }
        const float* kx = sk[slot];
        if constexpr (diag_kind<KIND>()) {
            const float2 vlo = make_float2(vc.x, vc.y), vhi = make_float2(vc.z, vc.w);
#pragma unroll
            for (int t = 0; t < ROWS; ++t) {
                const int i = Q::row(tau, t);
                const float di = per_key_gate<KIND>() ? sd[slot][i] : gc;
                float ki = kx[i];
                if constexpr (gated_injection<KIND>()) ki = __fmul_rn(__fsub_rn(1.0f, di), ki);
                const float2 lo = __ffma2_rn(f2(di), make_float2(P[t].x, P[t].y), __fmul2_rn(f2(ki), vlo));
                const float2 hi = __ffma2_rn(f2(di), make_float2(P[t].z, P[t].w), __fmul2_rn(f2(ki), vhi));
                P[t] = make_float4(lo.x, lo.y, hi.x, hi.y);
            }
        } else {   // RK_DELTA, RK_RWKV7
            const float4 u = quad_dot<DK, R, ROWS, TS>(P, kx, tau);
            float2 dlo = __fadd2_rn(make_float2(vc.x, vc.y), make_float2(-u.x, -u.y));   // v - u, exactly
            float2 dhi = __fadd2_rn(make_float2(vc.z, vc.w), make_float2(-u.z, -u.w));
            if constexpr (KIND == RK_DELTA) {
                dlo = __fmul2_rn(dlo, f2(gc));
                dhi = __fmul2_rn(dhi, f2(gc));
            }
#pragma unroll
            for (int t = 0; t < ROWS; ++t) {
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
            const float4 acc = quad_dot<DK, R, ROWS, TS>(P, sq[slot], tau);
            if (live && tau == 0)
                *reinterpret_cast<float4*>(p.o + (size_t)bh * DV + j0) =
                    make_float4(__fmul_rn(acc.x, p.scale), __fmul_rn(acc.y, p.scale), __fmul_rn(acc.z, p.scale),
                                __fmul_rn(acc.w, p.scale));
        }
        if (live && p.S_out != nullptr) {
            if constexpr (!TR) {
#pragma unroll
                for (int t = 0; t < ROWS; ++t)
                    *reinterpret_cast<float4*>(p.S_out + ((size_t)bh * DK + Q::row(tau, t)) * DV + j0) = P[t];
            } else {
#pragma unroll
                for (int blk = 0; blk < ROWS / 4; ++blk) {
                    const int r0 = Q::row(tau, 4 * blk);
                    const float4 a = P[4 * blk], b = P[4 * blk + 1], c = P[4 * blk + 2], d = P[4 * blk + 3];
                    float* col = p.S_out + ((size_t)bh * DV + j0) * DK + r0;
                    *reinterpret_cast<float4*>(col) = make_float4(a.x, b.x, c.x, d.x);
                    *reinterpret_cast<float4*>(col + DK) = make_float4(a.y, b.y, c.y, d.y);
                    *reinterpret_cast<float4*>(col + 2 * DK) = make_float4(a.z, b.z, c.z, d.z);
                    *reinterpret_cast<float4*>(col + 3 * DK) = make_float4(a.w, b.w, c.w, d.w);
                }
            }
        }
    }
    if (!ok && tid == 0) {
        record_error(p.st, SN_E_TIMEOUT, (SN_K_RECUR_DECODE << 16) | 1);
        // the copies still in flight land before the CTA leaves
        for (int m = n; m < issued; ++m) (void)mbar_wait(&full[m % NS], (uint32_t)(m / NS) & 1u, p.wait_ns);
    }
}

template <int KIND, int R>
cudaError_t run_decode_rows(const RecurArgs& x, const DecodeParams& p, int sm_count, cudaStream_t s) {
    const int BH = x.B * x.H;
    auto go = [&](auto kern, auto shape) -> cudaError_t {
        using S = decltype(shape);
        cudaError_t e = set_smem_attr_once((const void*)kern, S::smem);
        if (e != cudaSuccess) return e;
        const int grid = std::min((BH + S::SPC - 1) / S::SPC, sm_count);
        kern<<<grid, S::THREADS, S::smem, s>>>(p);
        return cudaGetLastError();
    };
    if (x.dk == 128)
        return x.dv == 128 ? go(recur_decode_ring<KIND, 128, 128, R>, RingShape<128, 128>{})
                           : go(recur_decode_ring<KIND, 128, 64, R>, RingShape<128, 64>{});
    return x.dv == 128 ? go(recur_decode_ring<KIND, 64, 128, R>, RingShape<64, 128>{})
                       : go(recur_decode_ring<KIND, 64, 64, R>, RingShape<64, 64>{});
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

bool recur_decode_ring_supported(const RecurArgs& x) {
    const bool kind_ok = x.kind == RK_DIAG_KEY || x.kind == RK_DIAG_HEAD || x.kind == RK_DIAG_KEY_GATED ||
                         x.kind == RK_DIAG_HEAD_GATED || x.kind == RK_DELTA || x.kind == RK_RWKV7;
    return kind_ok && x.T == 1 && (x.dk == 64 || x.dk == 128) && (x.dv == 64 || x.dv == 128);
}

cudaError_t launch_recur_decode_ring(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count,
                                     cudaStream_t s) {
    DecodeParams p;
    p.st = st;
    p.wait_ns = wait_ns;
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
