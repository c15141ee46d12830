// recur_chunked.cu -- chunked tensor-core form of the diagonal-decay matrix
// recurrence
//     S_t = diag(d_t) S_{t-1} + k_t v_t^T,      o_t = scale * S_t^T q_t
// for per-key decays (GLA, "SunnyNet 工程化实录" §4.3) and per-head decays
// (Mamba-2, same page §4.1), the T-parallel counterpart of the sequence kernel
// in recur_seq.cuh.  The pages keep this state "chunk-scannable" ("我拿同一份
// 权重和 llama.cpp 正面比了一场" §8); this file evaluates it chunk by chunk with
// dense contractions on the fifth-generation tensor cores.
//
// Chunk n holds tokens t = 0..C-1 (C = 128, global index nC + t) and starts
// from state S_n.  With lam_t = sum_{s <= t} log2 d_s (per key, or one scalar
// per head) the chunk's tokens satisfy
//   S_{n+1} = diag(2^{lam_{C-1}}) S_n + sum_j diag(2^{lam_{C-1} - lam_j}) k_j v_j^T
//   o_t     = scale * ( sum_i q_ti 2^{lam_ti} S_n[i, :]
//                     + sum_{j <= t} ( sum_i q_ti k_ji 2^{lam_ti - lam_ji} ) v_j )
// which three kernels evaluate:
//   chunk_state   one CTA per chunk: dS_n^T = V^T Khat with Khat_j = k_j
//                 2^{lam_{C-1} - lam_j} (one tcgen05 product, M = dv), the chunk
//                 decay gamma_n = 2^{lam_{C-1}} and the anchor factor below;
//   chunk_carry   one thread per four entries of a state column: S_{n+1} = gamma_n S_n + dS_n over
//                 the chunks in order (fp32 FMA); the operand S'_n of the chunk
//                 (below, rounded to tf32) is written over dS_n;
//   chunk_output  one CTA per chunk: A = Qt Kt^T masked to j <= t, P = Qt S',
//                 O = A V (three M = C tcgen05 products), o = scale (f_t P + O).
// Per-key decays cannot be pulled out of the dot product over keys, so the
// pair weight 2^{lam_ti - lam_ji} is split through an anchor token m = C/2 - 1:
// Qt = q 2^{lam_t - lam_m}, Kt = k 2^{lam_m - lam_j}, S' = diag(2^{lam_m}) S_n
// and f_t = 1.  Those factors stay within 2^{+-60} as long as the decay
// product between any token of the chunk and the anchor is at least 2^-60 (and
// every decay is positive); a chunk outside that range is flagged by the
// state kernel and its outputs are evaluated step by step in fp32 by the
// output kernel instead (a decay <= 0 records SN_E_RANGE).  Per-head decays
// are scalars per token, so Qt = q, Kt =
// k, S' = S_n, the exact weight 2^{lam_t - lam_j} multiplies A after the
// product and f_t = 2^{lam_t}; they only need positive decays.
//
// Operands are rounded to tf32 (to nearest) and products accumulate in fp32
// in tensor memory, so results carry tf32 rounding (about 1e-3 relative)
// instead of the sequence kernel's exact per-step fp32 arithmetic.
//
// Data movement: every tile a CTA needs is requested before any of it is
// used.  q and k of the output stage arrive by TMA in the 128-byte-swizzled
// operand layout.  The per-key state kernel takes k, d and v by TMA as
// natural [token][feature] tiles and transposes them in shared memory while
// it computes; it also leaves its rounded v^T tile for the output stage,
// which takes it by one bulk copy.  The per-head kernels transpose k and v
// with 4-byte cp.async (lanes covering 8 operand rows x 4 tokens, so the
// scattered shared-memory writes are conflict-free).  The chunk's S' operand
// is one contiguous bulk copy, because the state kernels and chunk_carry keep
// the chunk states in the operand layout.
//
// Shared-memory operands use the K-major no-swizzle core-matrix layout of
// tc.cuh with K extent 128 (every contraction here has K = 128: keys, or the
// chunk's tokens).
#include <type_traits>

#include "chunk_common.cuh"
#include "chunk_output.cuh"

namespace sn {
namespace {

using namespace chunk;

// ------------------------------------------------------------------ chunk_state
// Per-head decays (one CTA per chunk and head; chunk_state_key below takes the
// per-key decays, chunk_state_heads the heads of a group that share k).
template <int DV>
struct StateSmem {
    static constexpr int k_off = 0;                                   // k^T, then Khat^T: rows i, K = t
    static constexpr int v_off = OPF;                                 // v^T: rows c, K = t
    static constexpr int mu_off = v_off + DV * CH;                    // [CH] suffix sums
    static constexpr int om_off = mu_off + CH;                        // [CH] injection weights
    static constexpr int misc_off = om_off + CH;                      // total, barrier, tmem slot
    static constexpr size_t bytes = (size_t)(misc_off + 16) * 4 + 128;
};

template <int DV>
__global__ void __launch_bounds__(NT, 1) chunk_state(const ChunkArgs a) {
    extern __shared__ unsigned char smem_raw[];
    using L = StateSmem<DV>;
    float* base = align128(smem_raw);
    float* Ks = base + L::k_off;
    float* Vs = base + L::v_off;
    float* mu = base + L::mu_off;
    float* om = base + L::om_off;
    float* total_s = base + L::misc_off;
    uint64_t* bar = reinterpret_cast<uint64_t*>(base + L::misc_off + 2);
    uint32_t* slot = reinterpret_cast<uint32_t*>(base + L::misc_off + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const ChunkIdx c = chunk_index(a);

    if (warp == 0) tc::tmem_alloc(slot, DKC);
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }

    const size_t krs = (size_t)a.G * DKC, vrs = (size_t)a.H * DV;
    const size_t row0 = (size_t)c.b * a.T + c.t0;
    copy_transposed<DKC>(Ks, a.k + row0 * krs + (size_t)c.g * DKC, krs, c.nval, warp, lane);
    copy_transposed<DV>(Vs, a.v + row0 * vrs + (size_t)c.h * DV, vrs, c.nval, warp, lane);
    cp_async_commit();

    if (warp == 0) {
        // exclusive suffix sums mu[t] = sum_{s > t} log2 d_s of the per-head decays
        float lg[4], s = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int t = 4 * lane + r;
            const float dt = (t < c.nval && a.d != nullptr) ? __ldg(a.d + (row0 + t) * a.H + c.h) : 1.f;
            lg[r] = (t < c.nval && a.d != nullptr) ? lg2(dt) : 0.f;
            om[t] = a.gated ? 1.f - dt : 1.f;
            s += lg[r];
        }
        float x = s;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_down_sync(FULL, x, off);
            if (lane + off < 32) x += y;
        }
        float acc = x - s;
#pragma unroll
        for (int r = 3; r >= 0; --r) {
            mu[4 * lane + r] = acc;
            acc += lg[r];
        }
        if (lane == 0) {
            total_s[0] = x;
            if (!isfinite(x)) record_error(a.st, SN_E_RANGE, (SN_K_RECUR_CHUNK << 16) | SITE_RANGE_HEAD);
        }
    }
    cp_async_wait_all();
    __syncthreads();

    // Khat^T in place: thread = key row i, half of the tokens; the token
    // weight 2^{mu_t} (times 1 - d_t when gated) is a scalar per token
    const int i = tid & (DKC - 1), half = tid >> 7;
    const int tbeg = (CH / 2) * half;
    {
#pragma unroll 4
        for (int t4 = 0; t4 < CH / 8; ++t4) {
            const int tb = tbeg + 4 * t4;
            const int o = off128(i, tb);
            const float4 kk = ld4(Ks + o);
            st4(Ks + o, tf32x4(kk.x * ex2(mu[tb]) * om[tb], kk.y * ex2(mu[tb + 1]) * om[tb + 1],
                               kk.z * ex2(mu[tb + 2]) * om[tb + 2], kk.w * ex2(mu[tb + 3]) * om[tb + 3]));
        }
    }
    if (half == 0) {
        const size_t gi = (c.bh * a.NC + c.n) * DKC + i;
        a.gam[gi] = ex2(total_s[0]);
        a.anc[gi] = 1.f;
    }
    // v^T rounded in place
    for (int f = tid; f < DV * CH / 4; f += NT) st4(Vs + 4 * f, tf32x4(ld4(Vs + 4 * f)));

    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *slot;
    if (tid == 0) {
        // dS^T (M = dv rows c, N = dk columns i) = v^T (K = t) x Khat^T (K = t)
        tc::gemm_tf32(tmem, Vs, Ks, CH, tc::idesc_tf32(DV, DKC), false);
        tc::commit(bar);
    }
    const bool ok = __syncthreads_and(mbar_wait(bar, 0, a.wait_ns));
    tc::fence_after_sync();
    if (ok) {
        // M = 128: row c in lane c.  M = 64: rows 16q..16q+15 in lanes 32q..32q+15.
        const int lq = warp & 3, ih = warp >> 2;
        const int row = DV == 128 ? 32 * lq + lane : 16 * lq + (lane & 15);
        const bool mine = DV == 128 || lane < 16;
        float* wt = a.W + (c.bh * a.NC + c.n) * (size_t)DV * DKC;
#pragma unroll
        for (int i0 = 64 * ih; i0 < 64 * ih + 64; i0 += 16) {
            float x[16];
            tc::ld16(tmem + ((uint32_t)(32 * lq) << 16) + i0, x);
            if (mine) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    st4(wt + off128(row, i0 + 4 * q), make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]));
            }
        }
    } else if (tid == 0) {
        record_error(a.st, SN_E_TIMEOUT, (SN_K_RECUR_CHUNK << 16) | SITE_STATE_WAIT);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, DKC);
}

// ------------------------------------------------------------------ chunk_state_key
// chunk_state for per-key decays with its tiles by TMA: k, d and v arrive as
// natural [token][feature] boxes (128 tokens x 128 or dv features, rows past
// T filled with zeros), three copies instead of 4-byte transposing copies.
// The threads transpose while they compute: thread (key i, half of the
// tokens) reads its column of k and d (consecutive keys, conflict-free),
// takes log2 d in place, forms Khat in registers, and after a barrier writes
// it in the operand layout over k; v goes the same way (rounded to tf32)
// over its own box.  The product's dS^T leaves tensor memory for shared
// memory (over the consumed decays) and goes out by one bulk copy.  The
// arithmetic and its order are chunk_state's, so are the results.
template <int DV>
struct StateKeySmem {
    static constexpr int k_off = 0;                    // k [t][i], then Khat^T (rows i, K = t)
    static constexpr int d_off = OPF;                  // d [t][i] (log2 d in place), then dS^T
    static constexpr int v_off = 2 * OPF;              // v [t][j], then v^T (rows j, K = t)
    static constexpr int tot_off = v_off + DV * CH;    // [2][DKC] half sums, [2][2][DKC] extremes
    static constexpr int misc_off = tot_off + 6 * DKC; // barriers (k and d, v, product), tmem slot
    static constexpr size_t bytes = (size_t)(misc_off + 16) * 4 + 128;
    static_assert(DV * DKC <= OPF, "dS^T fits over the decays");
};

template <int DV>
__global__ void __launch_bounds__(NT, 1)
chunk_state_key(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_d,
                const __grid_constant__ CUtensorMap map_v, const ChunkArgs a) {
    extern __shared__ unsigned char smem_raw[];
    using L = StateKeySmem<DV>;
    float* base = align128(smem_raw);
    float* Kn = base + L::k_off;
    float* Dn = base + L::d_off;
    float* Vn = base + L::v_off;
    float* tot = base + L::tot_off;
    float* ext = tot + 2 * DKC;
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::misc_off);
    uint32_t* slot = reinterpret_cast<uint32_t*>(base + L::misc_off + 6);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const ChunkIdx c = chunk_index(a);
    if (warp == 0) tc::tmem_alloc(slot, DKC);
    if (tid == 0) {
        for (int q = 0; q < 3; ++q) mbar_init(&bars[q], 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bars[0], 2 * OPF * 4);
        tma_load_3d(Kn, &map_k, &bars[0], c.g * DKC, c.t0, c.b);
        tma_load_3d(Dn, &map_d, &bars[0], c.h * DKC, c.t0, c.b);
        mbar_arrive_expect_tx(&bars[1], DV * CH * 4);
        tma_load_3d(Vn, &map_v, &bars[1], c.h * DV, c.t0, c.b);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *slot;

    const int i = tid & (DKC - 1), half = tid >> 7;
    const int tbeg = (CH / 2) * half;
    bool ok = __syncthreads_and(mbar_wait(&bars[0], 0, a.wait_ns));
    int site = SITE_STATE_WAIT;
    float gam = 1.f, anc = 1.f;
    if (ok) {
        // log2 of the decays in place; gated keys take the weight 1 - d
        float sum = 0.f;
#pragma unroll 4
        for (int t4 = 0; t4 < CH / 8; ++t4) {
            const int tb = tbeg + 4 * t4;
            float lg[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int o = (tb + r) * DKC + i;
                const float dd = Dn[o];
                lg[r] = tb + r < c.nval ? lg2(dd) : 0.f;
                Dn[o] = lg[r];
                if (a.gated) Kn[o] = Kn[o] * (1.f - dd);
            }
            sum += (lg[0] + lg[1]) + (lg[2] + lg[3]);
        }
        tot[half * DKC + i] = sum;
        __syncthreads();
        // Khat_t = k_t 2^{m_t}, m_t the log2 decay of the tokens after t
        float m = half == 0 ? tot[DKC + i] : 0.f;
        float mhi = -INFINITY, mlo = INFINITY;
        float kh[CH / 2];
#pragma unroll
        for (int t4 = CH / 8 - 1; t4 >= 0; --t4) {
            const int tb = tbeg + 4 * t4;
#pragma unroll
            for (int r = 3; r >= 0; --r) {
                const int o = (tb + r) * DKC + i;
                kh[4 * t4 + r] = Kn[o] * ex2(m);
                mhi = fmaxf(mhi, m);
                mlo = fminf(mlo, m);
                m += Dn[o];
            }
        }
        gam = ex2(m);                       // half 0: the whole chunk's log2 decay
        ext[(half * 2 + 0) * DKC + i] = mhi;
        ext[(half * 2 + 1) * DKC + i] = mlo;
        __syncthreads();                    // k and d are read: Khat^T goes over k
#pragma unroll
        for (int t4 = 0; t4 < CH / 8; ++t4)
            st4(Kn + off128(i, tbeg + 4 * t4),
                tf32x4(kh[4 * t4], kh[4 * t4 + 1], kh[4 * t4 + 2], kh[4 * t4 + 3]));
        // the range test of chunk_state (flagged chunks run step by step in the output stage)
        bool wide = false;
        if (half == 0) {
            const float mm = tot[DKC + i];
            const float hi2 = fmaxf(mhi, ext[(2 + 0) * DKC + i]), lo2 = fminf(mlo, ext[(2 + 1) * DKC + i]);
            if (!isfinite(tot[i]) || !isfinite(mm))
                record_error(a.st, SN_E_RANGE, (SN_K_RECUR_CHUNK << 16) | SITE_RANGE_KEY);
            wide = !(hi2 - mm <= RANGE_LOG2 && mm - lo2 <= RANGE_LOG2);
        }
        const bool flagged = __syncthreads_or(wide);
        if (tid == 0) a.bad[c.bh * a.NC + c.n] = flagged ? 1 : 0;
        anc = flagged ? -1.f : ex2(tot[i]); // 2^{lam at the anchor token C/2 - 1}; -1 marks the flag
        if (half == 0) {
            const size_t gi = (c.bh * a.NC + c.n) * DKC + i;
            a.gam[gi] = gam;
            a.anc[gi] = anc;
        }
    }
    if (ok) {
        // v^T rounded, over v: thread = value column j, a run of TPV tokens
        ok = __syncthreads_and(mbar_wait(&bars[1], 0, a.wait_ns));
        if (ok) {
            constexpr int TPV = CH * DV / NT;
            const int j = tid % DV, t0 = (tid / DV) * TPV;
            float vv[TPV];
#pragma unroll
            for (int r = 0; r < TPV; ++r) vv[r] = Vn[(t0 + r) * DV + j];
            __syncthreads();
#pragma unroll
            for (int t4 = 0; t4 < TPV / 4; ++t4)
                st4(Vn + off128(j, t0 + 4 * t4), tf32x4(vv[4 * t4], vv[4 * t4 + 1], vv[4 * t4 + 2], vv[4 * t4 + 3]));
        }
    }
    if (ok) {
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (tid == 0) {
            // dS^T (M = dv rows c, N = dk columns i) = v^T (K = t) x Khat^T (K = t)
            tc::gemm_tf32(tmem, Vn, Kn, CH, tc::idesc_tf32(DV, DKC), false);
            tc::commit(&bars[2]);
            if (a.vt_out != nullptr) {   // the output stage's v operand
                bulk_store(a.vt_out + (c.bh * a.NC + c.n) * (size_t)DV * CH, Vn, DV * CH * 4);
                bulk_commit();
            }
        }
        ok = __syncthreads_and(mbar_wait(&bars[2], 0, a.wait_ns));
        tc::fence_after_sync();
        if (ok) {
            // M = 128: row c in lane c.  M = 64: rows 16q..16q+15 in lanes 32q..32q+15.
            const int lq = warp & 3, ih = warp >> 2;
            const int row = DV == 128 ? 32 * lq + lane : 16 * lq + (lane & 15);
            const bool mine = DV == 128 || lane < 16;
#pragma unroll
            for (int i0 = 64 * ih; i0 < 64 * ih + 64; i0 += 16) {
                float x[16];
                tc::ld16(tmem + ((uint32_t)(32 * lq) << 16) + i0, x);
                if (mine) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        st4(Dn + off128(row, i0 + 4 * q), make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]));
                }
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncthreads();
            if (tid == 0) {
                bulk_store(a.W + (c.bh * a.NC + c.n) * (size_t)DV * DKC, Dn, DV * DKC * 4);
                bulk_commit();
            }
        } else {
            site = SITE_STATE_WAIT;
        }
    }
    if (tid == 0) {
        if (!ok) {
            record_error(a.st, SN_E_TIMEOUT, (SN_K_RECUR_CHUNK << 16) | site);
            // the copies still in flight land before the CTA leaves
            (void)mbar_wait(&bars[0], 0, a.wait_ns);
            (void)mbar_wait(&bars[1], 0, a.wait_ns);
        }
        bulk_wait_all();   // the bulk copies out have read shared memory and landed
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, DKC);
}

// ------------------------------------------------------------------ chunk_state_heads
// Per-head decays with heads sharing k (Mamba-2's groups): the token weight
// 2^{mu_t} is a scalar per token, so it is applied to v instead of k,
// dS^T = (v (.) 2^{mu})^T k, and the transposed k tile is the same for every
// head of the group.  One CTA per SM, each taking an even share of the
// (batch, chunk, group, head) items as segments of consecutive heads of one
// (batch, chunk, group).  k and the heads' v tiles arrive by TMA in their natural
// [token][feature] layout (rows past T read as zeros) and the threads
// transpose them: k once, into the operand layout; each head's v tile,
// scaled by its token weights and rounded, into one of two operand buffers,
// while the next head's tile is already on its way into the other staging
// half.  A head's dS^T goes from tensor memory into the operand buffer its v
// used and out by one bulk copy.  dv = 64.
template <int DV>
struct StateHeadsSmem {
    static constexpr int k_off = 0;                    // k^T operand (rows key, K = t), tf32
    static constexpr int st_off = OPF;                 // staging: k [t][i], then two v tiles [t][j]
    static constexpr int v_off = 2 * OPF;              // [2] (v 2^mu)^T operand (rows value, K = t), then dS^T
    static constexpr int mu_off = v_off + 2 * DV * CH; // [CH] suffix sums of log2 d of the head
    static constexpr int om_off = mu_off + CH;         // [CH] injection weights of the head
    static constexpr int misc_off = om_off + CH;       // total, barriers (k, v0, v1, product), tmem slot
    static constexpr size_t bytes = (size_t)(misc_off + 16) * 4 + 128;
    static_assert(2 * DV * CH <= OPF && DV * DKC <= DV * CH, "buffer sizes");
};

template <int DV>
__global__ void __launch_bounds__(NT, 1)
chunk_state_heads(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                  const ChunkArgs a) {
    extern __shared__ unsigned char smem_raw[];
    using L = StateHeadsSmem<DV>;
    float* base = align128(smem_raw);
    float* Ks = base + L::k_off;
    float* Sg = base + L::st_off;
    float* mu = base + L::mu_off;
    float* om = base + L::om_off;
    float* total_s = base + L::misc_off;
    uint64_t* bk = reinterpret_cast<uint64_t*>(base + L::misc_off + 2);
    uint64_t* bv = bk + 1;                              // [2]
    uint64_t* bm = bk + 3;
    uint32_t* slot = reinterpret_cast<uint32_t*>(base + L::misc_off + 10);
    auto stg = [&](int q) { return Sg + q * DV * CH; };
    auto vop = [&](int q) { return base + L::v_off + q * DV * CH; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // The CTA's share of the (batch, chunk, group, head) items, in that order,
    // as segments of consecutive heads of one (batch, chunk, group).  Heads
    // are counted across segments (q): v staging half, operand buffer and
    // barrier phases follow that count.
    const int hpg = a.H / a.G;
    const int64_t total = (int64_t)a.B * a.NC * a.G * hpg;
    int64_t it = (int64_t)blockIdx.x * total / gridDim.x;
    const int64_t it_end = (int64_t)(blockIdx.x + 1) * total / gridDim.x;

    if (warp == 0) tc::tmem_alloc(slot, DKC);
    if (tid == 0) {
        for (int q = 0; q < 4; ++q) mbar_init(&bk[q], 1);
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *slot;
    int v_issued = 0;   // thread 0's count of v tiles requested (all segments)
    int v_used = 0;     // v tiles waited for (all segments)
    int seg = 0;        // segments begun (k tiles requested)
    bool ok = true;
    int site = SITE_STATE_WAIT;
    while (ok && it < it_end) {
    const int64_t pair = it / hpg;
    const int hin = (int)(it % hpg);
    const int hb = (int)std::min<int64_t>(hpg - hin, it_end - it);   // heads h0 .. h0 + hb - 1
    it += hb;
    const int g = (int)(pair % a.G);
    const int64_t bn = pair / a.G;
    const int n = (int)(bn % a.NC), b = (int)(bn / a.NC);
    const int h0 = g * hpg + hin;
    const int t0 = n * CH, nval = min(CH, a.T - t0);
    const size_t row0 = (size_t)b * a.T + t0;
    const int q0 = v_used;   // the segment's first head in the CTA's count
    if (tid == 0) {
        fence_proxy_async_smem();   // the previous segment's reads of the staging area before this copy
        mbar_arrive_expect_tx(bk, OPF * 4);
        tma_load_3d(Sg, &map_k, bk, g * DKC, t0, b);
    }
    ++seg;
    auto issue_v = [&](int q) {   // thread 0: the segment's head q - q0 v tile into staging half q & 1
        mbar_arrive_expect_tx(&bv[q & 1], DV * CH * 4);
        tma_load_3d(stg(q & 1), &map_v, &bv[q & 1], (h0 + q - q0) * DV, t0, b);
    };
    // warp 0: a head's decays, four tokens per lane, loaded a head ahead of
    // their suffix sums so that the load latency hides behind the other work
    float dr[4];
    auto head_d = [&](int hh) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int t = 4 * lane + r;
            dr[r] = (t < nval && a.d != nullptr) ? __ldg(a.d + (row0 + t) * a.H + hh) : 1.f;
        }
    };
    if (warp == 0) head_d(h0);

    // k^T, rounded: thread (key i, half of the tokens) reads its column
    ok = __syncthreads_and(mbar_wait(bk, (uint32_t)(seg - 1) & 1u, a.wait_ns));
    if (ok) {
        const int i = tid & (DKC - 1), tb0 = (CH / 2) * (tid >> 7);
        float kr[CH / 2];
#pragma unroll
        for (int r = 0; r < CH / 2; ++r) kr[r] = Sg[(tb0 + r) * DKC + i];
        __syncthreads();                                // the staging area is read: the v tiles go there
        if (tid == 0) {
            fence_proxy_async_smem();                   // those reads before the copies' writes
            for (; v_issued < q0 + min(2, hb); ++v_issued) issue_v(v_issued);
        }
#pragma unroll
        for (int t4 = 0; t4 < CH / 8; ++t4)
            st4(Ks + off128(i, tb0 + 4 * t4), tf32x4(kr[4 * t4], kr[4 * t4 + 1], kr[4 * t4 + 2], kr[4 * t4 + 3]));
    }
    for (int hi = 0; hi < hb && ok; ++hi) {
        const int h = h0 + hi, q = q0 + hi, p = q & 1;
        // the bulk copy out of two heads ago has read operand buffer p
        if (tid == 0) bulk_wait_read_allbut1();
        if (warp == 0) {
            // exclusive suffix sums mu[t] = sum_{s > t} log2 d_s of this head
            float lg[4], sm = 0.f;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = 4 * lane + r;
                lg[r] = (t < nval && a.d != nullptr) ? lg2(dr[r]) : 0.f;
                om[t] = a.gated ? 1.f - dr[r] : 1.f;
                sm += lg[r];
            }
            if (hi + 1 < hb) head_d(h + 1);
            float x = sm;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_down_sync(FULL, x, off);
                if (lane + off < 32) x += y;
            }
            float acc = x - sm;
#pragma unroll
            for (int r = 3; r >= 0; --r) {
                mu[4 * lane + r] = acc;
                acc += lg[r];
            }
            if (lane == 0) {
                total_s[0] = x;
                if (!isfinite(x)) record_error(a.st, SN_E_RANGE, (SN_K_RECUR_CHUNK << 16) | SITE_RANGE_HEAD);
            }
        }
        ok = __syncthreads_and(mbar_wait(&bv[p], (uint32_t)(q >> 1) & 1u, a.wait_ns));
        if (!ok) break;
        v_used = q + 1;
        {
            // (v^T (.) 2^{mu_t}), rounded, into operand buffer p: thread = value
            // column j, a run of TPV tokens (a float4 of the operand holds four)
            constexpr int TPV = CH * DV / NT;
            const int j = tid % DV, tq0 = (tid / DV) * TPV;
            const float* sv = stg(p);
            float* vo = vop(p);
#pragma unroll
            for (int t4 = 0; t4 < TPV / 4; ++t4) {
                const int tq = tq0 + 4 * t4;
                const float v0 = sv[tq * DV + j], v1 = sv[(tq + 1) * DV + j];
                const float v2 = sv[(tq + 2) * DV + j], v3 = sv[(tq + 3) * DV + j];
                st4(vo + off128(j, tq), tf32x4(v0 * ex2(mu[tq]) * om[tq], v1 * ex2(mu[tq + 1]) * om[tq + 1],
                                               v2 * ex2(mu[tq + 2]) * om[tq + 2], v3 * ex2(mu[tq + 3]) * om[tq + 3]));
            }
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();                                // staging half p is read; operand p is written
        tc::fence_after_sync();
        if (tid == 0) {
            // dS^T (M = dv rows value, N = dk columns key) = (v 2^mu)^T (K = t) x k^T (K = t)
            tc::gemm_tf32(tmem, vop(p), Ks, CH, tc::idesc_tf32(DV, DKC), false);
            tc::commit(bm);
            if (v_issued < q0 + hb) issue_v(v_issued++);   // two heads ahead, into the half just read
        }
        ok = __syncthreads_and(mbar_wait(bm, (uint32_t)q & 1u, a.wait_ns));
        tc::fence_after_sync();
        if (!ok) break;
        {
            // M = 64: rows 16q .. 16q + 15 in lanes 32q .. 32q + 15; dS^T over the operand it consumed
            const int lq = warp & 3, ih = warp >> 2;
            const int row = 16 * lq + (lane & 15);
            const bool mine = lane < 16;
            float* ds = vop(p);
#pragma unroll
            for (int i0 = 64 * ih; i0 < 64 * ih + 64; i0 += 16) {
                float x[16];
                tc::ld16(tmem + ((uint32_t)(32 * lq) << 16) + i0, x);
                if (mine) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        st4(ds + off128(row, i0 + 4 * q), make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]));
                }
            }
            const size_t bh = (size_t)b * a.H + h;
            if (tid < DKC) {
                const size_t gi = (bh * a.NC + n) * DKC + tid;
                a.gam[gi] = ex2(total_s[0]);
                a.anc[gi] = 1.f;
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncthreads();   // dS^T is in place; tensor memory, mu and the weights are free for the next head
            if (tid == 0) {
                bulk_store(a.W + (bh * a.NC + n) * (size_t)DV * DKC, ds, DV * DKC * 4);
                bulk_commit();
            }
        }
    }
    }   // segments
    if (tid == 0) {
        if (!ok) {
            record_error(a.st, SN_E_TIMEOUT, (SN_K_RECUR_CHUNK << 16) | site);
            // the tiles still in flight land before the CTA leaves
            if (seg > 0) (void)mbar_wait(bk, (uint32_t)(seg - 1) & 1u, a.wait_ns);
            for (int q = v_used; q < v_issued; ++q) (void)mbar_wait(&bv[q & 1], (uint32_t)(q >> 1) & 1u, a.wait_ns);
        }
        bulk_wait_all();
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, DKC);
}

// ------------------------------------------------------------------ chunk_carry
// One thread per entry of a head's dv x dk state tile, in the operand layout.
// S_0 = S_in; for each chunk: W[n] <- tf32(anc_n (.) S_n), S_{n+1} = gamma_n (.) S_n + dS_n.
// V entries per thread: keys i0 .. i0 + V - 1 of one value column, 4 V
// contiguous bytes of every chunk's tile (V = 4 where the grid still fills
// the GPU, else V = 1 for more threads to hide the load latency).
template <int V>
__global__ void __launch_bounds__(256) chunk_carry(const ChunkArgs a, int dv) {
    static_assert(V == 1 || V == 4, "one entry or a 16-byte group");
    using vec = typename std::conditional<V == 4, float4, float>::type;
    const size_t per_head = (size_t)DKC * dv;
    const size_t ev = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * V;
    if (ev >= (size_t)a.B * a.H * per_head) return;
    const size_t bh = ev / per_head;
    const int f = (int)(ev % per_head);
    const int i0 = ((f >> 5) & 31) * 4 + (f & 3);       // first key (K index of the operand)
    const int col = (f >> 10) * 8 + ((f >> 2) & 7);     // value (row of the operand)
    float s[V];
#pragma unroll
    for (int q = 0; q < V; ++q) s[q] = a.S_in != nullptr ? a.S_in[bh * per_head + (size_t)(i0 + q) * dv + col] : 0.f;
    float* w = a.W + bh * a.NC * per_head + f;
    const float* gm = a.gam + bh * a.NC * DKC + i0;
    const float* an = a.anc + bh * a.NC * DKC + i0;
    auto ld = [](const float* p) -> vec {
        if constexpr (V == 4) return ld4(p); else return *p;
    };
    auto ldg = [](const float* p) -> vec {
        if constexpr (V == 4) return ldg4(p); else return __ldg(p);
    };
    // a flagged chunk (chunk_state marks it with anchor -1) keeps its start
    // state in fp32 for the step-by-step evaluation
    auto operand = [&](float anchor, float st) { return anchor < 0.f ? st : tc::to_tf32(anchor * st); };
    auto step = [&](vec ds, vec gg, vec aa, float* out) {
        if constexpr (V == 4) {
            st4(out, make_float4(operand(aa.x, s[0]), operand(aa.y, s[1]), operand(aa.z, s[2]), operand(aa.w, s[3])));
            s[0] = fmaf(gg.x, s[0], ds.x);
            s[1] = fmaf(gg.y, s[1], ds.y);
            s[2] = fmaf(gg.z, s[2], ds.z);
            s[3] = fmaf(gg.w, s[3], ds.w);
        } else {
            *out = operand(aa, s[0]);
            s[0] = fmaf(gg, s[0], ds);
        }
    };
    constexpr int U = 8;
    int n = 0;
    for (; n + U <= a.NC; n += U) {
        vec ds[U], gg[U], aa[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            ds[u] = ld(w + (size_t)(n + u) * per_head);
            gg[u] = ldg(gm + (size_t)(n + u) * DKC);
            aa[u] = ldg(an + (size_t)(n + u) * DKC);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) step(ds[u], gg[u], aa[u], w + (size_t)(n + u) * per_head);
    }
    for (; n < a.NC; ++n)
        step(ld(w + (size_t)n * per_head), ldg(gm + (size_t)n * DKC), ldg(an + (size_t)n * DKC),
             w + (size_t)n * per_head);
    if (a.S_out != nullptr) {
#pragma unroll
        for (int q = 0; q < V; ++q) a.S_out[bh * per_head + (size_t)(i0 + q) * dv + col] = s[q];
    }
}

// ------------------------------------------------------------------ flagged chunks
// Per-key decays strong enough that a chunk's anchor factors would leave
// 2^{+-RANGE_LOG2} (chunk_state flags the chunk): the chunk's outputs are
// evaluated step by step from its start state, which chunk_carry kept in fp32.
// Each step is the sequence kernel's single-precision update
// S_ij = fma(d_i, S_ij, k_i v_j) (k_i weighted by 1 - d_i when gated) and the
// readout o_tj = scale sum_i S_ij q_i, so no factor other than the decays
// themselves appears and any positive decay is exact.  The CTA of chunk_output
// that owns the unit runs this after its tensor-core units (it skipped the
// unit's stores there), in the same shared memory; a thread owns four value
// columns over 16 key rows, the eight threads of a column quad sum the
// readout by xor shuffles.  The tokens stream through shared memory FB at a
// time, double-buffered.
constexpr int FB = 32;               // tokens per staged batch

__device__ __forceinline__ float2 f2(float x) { return make_float2(x, x); }

template <int DV>
struct FixSmem {
    static constexpr int per_batch = FB * (3 * DKC + DV);   // q, k, d rows, then v rows
    static constexpr size_t bytes = (size_t)2 * per_batch * 4 + 128;
};

// Evaluate the flagged unit of chunk c (whole CTA; `base` holds FixSmem bytes).
template <int DV>
__device__ __forceinline__ void fix_unit(const ChunkArgs& a, const ChunkIdx& c, float* base) {
    constexpr int QUADS = DV / 4, TPG = DKC / 16;
    const int tid = threadIdx.x;
    const int tau = tid % TPG, qd = tid / TPG;              // quad qd < QUADS holds columns 4 qd .. 4 qd + 3
    const bool owner = qd < QUADS;
    const int r0 = 16 * tau, j0 = 4 * qd;
    {
        const size_t u = c.bh * a.NC + c.n;
        const int b = c.b, h = c.h, g = c.g;
        const int t0 = c.t0, nval = c.nval;
        // start state: column c's rows r0 .. r0 + 15 are four 16-byte runs of the operand tile
        float2 S[16][2];
        const float* w = a.W + (size_t)u * DV * DKC;
        if (owner) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int r4 = 0; r4 < 4; ++r4) {
                    const float4 x = ld4(w + off128(j0 + c, r0 + 4 * r4));
                    const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if (c & 1) S[4 * r4 + e][c >> 1].y = xs[e];
                        else S[4 * r4 + e][c >> 1].x = xs[e];
                    }
                }
        }
        const size_t krs = (size_t)a.G * DKC, drs = (size_t)a.H * DKC, vrs = (size_t)a.H * DV;
        auto stage = [&](int bt, float* buf) {               // tokens [bt, bt + FB) of the chunk
            for (int f = tid; f < FB * (3 * DKC + DV) / 4; f += NT) {
                const int e4 = 4 * f;
                const int tt = e4 / (3 * DKC + DV), col = e4 % (3 * DKC + DV);
                const size_t row = (size_t)b * a.T + t0 + bt + tt;
                const bool ok = bt + tt < nval;
                const float* src;
                if (col < DKC) src = a.q + row * krs + (size_t)g * DKC + col;
                else if (col < 2 * DKC) src = a.k + row * krs + (size_t)g * DKC + (col - DKC);
                else if (col < 3 * DKC) src = a.d + row * drs + (size_t)h * DKC + (col - 2 * DKC);
                else src = a.v + row * vrs + (size_t)h * DV + (col - 3 * DKC);
                cp_async16(buf + e4, ok ? src : a.q, ok);
            }
            cp_async_commit();
        };
        const int nb = (nval + FB - 1) / FB;
        __syncthreads();                                     // the shared memory is free
        stage(0, base);
        for (int bi = 0; bi < nb; ++bi) {
            float* cur = base + (bi & 1) * FixSmem<DV>::per_batch;
            if (bi + 1 < nb) {
                stage((bi + 1) * FB, base + ((bi + 1) & 1) * FixSmem<DV>::per_batch);
                asm volatile("cp.async.wait_group 1;" ::: "memory");
            } else {
                cp_async_wait_all();
            }
            __syncthreads();
            const int tn = min(FB, nval - bi * FB);
            for (int tt = 0; tt < tn; ++tt) {
                const float* row = cur + tt * (3 * DKC + DV);
                float qv[16], kv[16], dv[16];
#pragma unroll
                for (int r4 = 0; r4 < 4; ++r4) {
                    const float4 q4 = ld4(row + r0 + 4 * r4), k4 = ld4(row + DKC + r0 + 4 * r4),
                                 d4 = ld4(row + 2 * DKC + r0 + 4 * r4);
                    qv[4 * r4] = q4.x; qv[4 * r4 + 1] = q4.y; qv[4 * r4 + 2] = q4.z; qv[4 * r4 + 3] = q4.w;
                    kv[4 * r4] = k4.x; kv[4 * r4 + 1] = k4.y; kv[4 * r4 + 2] = k4.z; kv[4 * r4 + 3] = k4.w;
                    dv[4 * r4] = d4.x; dv[4 * r4 + 1] = d4.y; dv[4 * r4 + 2] = d4.z; dv[4 * r4 + 3] = d4.w;
                }
                const float4 v4 = owner ? ld4(row + 3 * DKC + j0) : make_float4(0.f, 0.f, 0.f, 0.f);
                const float2 vlo = make_float2(v4.x, v4.y), vhi = make_float2(v4.z, v4.w);
                float2 alo[4], ahi[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) alo[e] = ahi[e] = make_float2(0.f, 0.f);
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    const float ki = a.gated ? __fmul_rn(__fsub_rn(1.0f, dv[r]), kv[r]) : kv[r];
                    S[r][0] = __ffma2_rn(f2(dv[r]), S[r][0], __fmul2_rn(f2(ki), vlo));
                    S[r][1] = __ffma2_rn(f2(dv[r]), S[r][1], __fmul2_rn(f2(ki), vhi));
                    alo[r & 3] = __ffma2_rn(S[r][0], f2(qv[r]), alo[r & 3]);
                    ahi[r & 3] = __ffma2_rn(S[r][1], f2(qv[r]), ahi[r & 3]);
                }
                float2 slo = __fadd2_rn(__fadd2_rn(alo[0], alo[1]), __fadd2_rn(alo[2], alo[3]));
                float2 shi = __fadd2_rn(__fadd2_rn(ahi[0], ahi[1]), __fadd2_rn(ahi[2], ahi[3]));
#pragma unroll
                for (int o = TPG / 2; o > 0; o >>= 1) {
                    slo.x = __fadd_rn(slo.x, __shfl_xor_sync(FULL, slo.x, o));
                    slo.y = __fadd_rn(slo.y, __shfl_xor_sync(FULL, slo.y, o));
                    shi.x = __fadd_rn(shi.x, __shfl_xor_sync(FULL, shi.x, o));
                    shi.y = __fadd_rn(shi.y, __shfl_xor_sync(FULL, shi.y, o));
                }
                if (owner && tau == 0 && a.o != nullptr) {
                    float* orow = a.o + (((size_t)b * a.T + t0 + bi * FB + tt) * a.H + h) * DV + j0;
                    st_cs(reinterpret_cast<float4*>(orow), make_float4(a.scale * slo.x, a.scale * slo.y,
                                                                        a.scale * shi.x, a.scale * shi.y));
                }
            }
            __syncthreads();                                 // batch `bi` is read: its buffer can refill
        }
    }
}

// ------------------------------------------------------------------ chunk_output
// The output stage over units i, i + grid, ... (chunk_output.cuh).
template <bool PER_KEY, int DV>
__global__ void __launch_bounds__(NT, 1)
chunk_output(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
             const __grid_constant__ CUtensorMap map_o, const ChunkArgs a) {
    StaticUnits sch{chunk_units(a)};
    output_loop<PER_KEY, DV>(&map_q, &map_k, &map_o, a, sch);
}

// ------------------------------------------------------------------ chunk_output_heads
// Per-head decays where several heads share q and k (Mamba-2's groups): one
// CTA per SM, each taking an even share of the (batch, chunk, group, head)
// items as one or more segments of consecutive heads of one (batch, chunk,
// group).  Q K^T does not depend on the head, so a segment forms it once in
// tensor memory and, head by head, weights a copy of it with that head's
// decays, then adds the head's state and value products.  The next head's S'
// tile, v slice and decay sums are fetched while the current head's products
// run.  dv = 64.
template <int DV>
struct HeadsSmem {
    static constexpr int q_off = 0;                  // Q (tf32)
    static constexpr int a_off = OPF;                // K, then the weighted A of the current head
    static constexpr int s_off = 2 * OPF;            // S'^T of the current head
    static constexpr int v_off = s_off + DV * DKC;   // v^T of the current head
    static constexpr int lam_off = v_off + DV * CH;  // [2][CH] decay prefix sums (two heads)
    static constexpr int om_off = lam_off + 2 * CH;  // [2][CH] injection weights (two heads)
    static constexpr int misc_off = om_off + 2 * CH;
    static constexpr int stage_off = misc_off + 16;  // [8 warps][32 rows][dv / 2] o staging
    static constexpr size_t bytes = (size_t)(stage_off + 8 * 32 * (DV / 2)) * 4 + 128;
};

template <int DV>
__global__ void __launch_bounds__(NT, 1) chunk_output_heads(const ChunkArgs a) {
    extern __shared__ unsigned char smem_raw[];
    using L = HeadsSmem<DV>;
    float* base = align128(smem_raw);
    float* bufQ = base + L::q_off;
    float* bufA = base + L::a_off;
    float* bufS = base + L::s_off;
    float* bufV = base + L::v_off;
    float* lam2 = base + L::lam_off;
    float* om2 = base + L::om_off;
    uint64_t* barS = reinterpret_cast<uint64_t*>(base + L::misc_off);
    uint64_t* barM = reinterpret_cast<uint64_t*>(base + L::misc_off + 2);
    uint32_t* slot = reinterpret_cast<uint32_t*>(base + L::misc_off + 4);
    uint64_t* barO = reinterpret_cast<uint64_t*>(base + L::misc_off + 6);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float* stage = base + L::stage_off + warp * 32 * (DV / 2);   // this warp's o rows
    // Warps 4 and 5 hold rows 0..63 of the right column half, above the
    // diagonal: they weight no block of Q K^T.  Warp 4's first thread issues
    // the products and copies (an issue of 16 products can stall it for a
    // while), warp 5 loads the decays and forms their sums, so that neither
    // delays the warps that weight the blocks.
    constexpr int DWARP = 5;
    const bool issuer = tid == 128;
    // The CTA's share of the (batch, chunk, group, head) items, in that order:
    // segments of consecutive heads of one (batch, chunk, group) each.
    const int hpg = a.H / a.G;
    const int64_t total = (int64_t)a.B * a.NC * a.G * hpg;
    int64_t it = (int64_t)blockIdx.x * total / gridDim.x;
    const int64_t it_end = (int64_t)(blockIdx.x + 1) * total / gridDim.x;
    const size_t tile_floats = (size_t)DV * DKC;

    if (warp == 0) tc::tmem_alloc(slot, 512);
    if (tid == 0) {
        mbar_init(barS, 1);
        mbar_init(barM, 1);
        mbar_init(barO, 1);
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *slot;
    uint32_t ps = 0, pm = 0, po = 0;   // phases of barS, barM and barO waited for
    int o_pending = 0;                 // output products issued and not yet waited for
    bool ok = true;
    while (ok && it < it_end) {
    const int64_t pair = it / hpg;
    const int hin = (int)(it % hpg);
    const int hb = (int)std::min<int64_t>(hpg - hin, it_end - it);   // heads h0 .. h0 + hb - 1
    it += hb;
    const int g = (int)(pair % a.G);
    const int64_t bn = pair / a.G;
    const int n = (int)(bn % a.NC), b = (int)(bn / a.NC);
    const int h0 = g * hpg + hin;
    const int t0 = n * CH, nval = min(CH, a.T - t0);
    const size_t row0 = (size_t)b * a.T + t0;
    auto tile = [&](int h) { return a.W + (((size_t)b * a.H + h) * a.NC + n) * tile_floats; };
    if (issuer) {
        mbar_arrive_expect_tx(barS, DV * DKC * 4);
        bulk_load(bufS, tile(h0), DV * DKC * 4, barS);
    }

    // q, k rows straight into the operand layout
    {
        const int tl = lane & 7, ic = 16 * warp + 4 * (lane >> 3);
        const size_t qrs = (size_t)a.G * DKC;
        const float* qb = a.q + row0 * qrs + (size_t)g * DKC + ic;
        const float* kb = a.k + row0 * qrs + (size_t)g * DKC + ic;
#pragma unroll
        for (int tb = 0; tb < CH / 8; ++tb) {
            const int t = 8 * tb + tl;
            const bool ok = t < nval;
            const size_t src = (size_t)(ok ? t : 0) * qrs;
            cp_async16(bufQ + off128(t, ic), qb + src, ok);
            cp_async16(bufA + off128(t, ic), kb + src, ok);
        }
        cp_async_commit();
    }

    constexpr int TP = CH / (NT / DV);
    const int col = tid % DV, part = tid / DV;
    float vr[TP];
    const size_t vrs = (size_t)a.H * DV;
    auto load_v = [&](int h) {
        const float* vcol = a.v + row0 * vrs + (size_t)h * DV + col;
#pragma unroll
        for (int r = 0; r < TP; ++r) {
            const int t = part * TP + r;
            vr[r] = t < nval ? __ldg(vcol + (size_t)t * vrs) : 0.f;
        }
    };
    // warp DWARP: a head's decays, four tokens per lane, loaded one step ahead of
    // their prefix sums so that the load latency hides behind other work
    float dr[4];
    auto head_d = [&](int h) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int t = 4 * lane + r;
            dr[r] = (t < nval && a.d != nullptr) ? __ldg(a.d + (row0 + t) * a.H + h) : 1.f;
        }
    };
    // warp DWARP: inclusive prefix sums of log2 d of the loaded head into dst, and
    // the keys' injection weights (1 - d when gated) into dst + (om2 - lam2)
    auto head_lam = [&](float* dst) {
        float lg[4], s = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            lg[r] = lg2(dr[r]);
            dst[(om2 - lam2) + 4 * lane + r] = a.gated ? 1.f - dr[r] : 1.f;
            s += lg[r];
        }
        float x = s;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(FULL, x, off);
            if (lane >= off) x += y;
        }
        float acc = x - s;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            acc += lg[r];
            dst[4 * lane + r] = acc;
        }
        if (lane == 31 && !isfinite(x)) record_error(a.st, SN_E_RANGE, (SN_K_RECUR_CHUNK << 16) | SITE_RANGE_HEAD);
    };
    load_v(h0);
    if (warp == DWARP) {
        head_d(h0);
        head_lam(lam2);
    }

    cp_async_wait_all();
    {
        const int tl = lane & 7, ic = 16 * warp + 4 * (lane >> 3);
#pragma unroll
        for (int tb = 0; tb < CH / 8; ++tb) {
            const int o = off128(8 * tb + tl, ic);
            st4(bufQ + o, tf32x4(ld4(bufQ + o)));
            st4(bufA + o, tf32x4(ld4(bufA + o)));
        }
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    ok = __syncthreads_and(mbar_wait(barS, ps & 1u, a.wait_ns));
    tc::fence_after_sync();
    constexpr uint32_t COL_P = 128, COL_O = 128 + 2 * DV;   // tensor-memory columns: A, P[2], O[2]
    if (!ok) {
        if (issuer) {
            record_error(a.st, SN_E_TIMEOUT, (SN_K_RECUR_CHUNK << 16) | SITE_OUT_COPY);
            mbar_wait(barS, ps & 1u, a.wait_ns);   // the copy in flight lands before the CTA leaves
        }
        break;
    }
    ++ps;
    if (issuer) {
        tc::gemm_tf32(tmem, bufQ, bufA, DKC, tc::idesc_tf32(128, 128), false);        // Q K^T
        tc::gemm_tf32(tmem + COL_P, bufQ, bufS, DKC, tc::idesc_tf32(128, DV), false); // P of the first head
        tc::commit(barM);
    }

    const int lq = warp & 3, hf = warp >> 2;
    const int t = 32 * lq + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * lq) << 16);
    // head hi's state and value products go to P[hi & 1] and O[hi & 1], so
    // that head hi's output product runs while head hi - 1's epilogue reads
    // its own pair
    auto col_p = [&](int hi) { return COL_P + (uint32_t)(hi & 1) * DV; };
    auto col_o = [&](int hi) { return COL_O + (uint32_t)(hi & 1) * DV; };
    float fp_prev = 0.f;   // 2^{lam_t} of the previous head (its epilogue's factor)
    // o of head h0 + hi from its P and O.  A warp holds 32 rows x dv / 2
    // values; it passes them through its own staging rows (16-byte slots
    // XOR-swizzled by row, so that neither side conflicts on banks) and
    // writes them back as whole 128-byte lines, eight lanes to a row.
    static_assert(DV / 2 == 32, "one 128-byte line per row and warp");
    auto epilogue = [&](int hi, float fp) {
        if (a.o == nullptr) return;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int c0 = hf * (DV / 2) + 16 * c;
            float pv[16], x[16];
            tc::ld16(lane_base + col_p(hi) + c0, pv);
            tc::ld16(lane_base + col_o(hi) + c0, x);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                st4(stage + 32 * lane + 4 * ((4 * c + q) ^ (lane & 7)),
                    make_float4(a.scale * fmaf(fp, pv[4 * q], x[4 * q]),
                                a.scale * fmaf(fp, pv[4 * q + 1], x[4 * q + 1]),
                                a.scale * fmaf(fp, pv[4 * q + 2], x[4 * q + 2]),
                                a.scale * fmaf(fp, pv[4 * q + 3], x[4 * q + 3])));
        }
        __syncwarp();
        const size_t ors = (size_t)a.H * DV;
        float* ob = a.o + (row0 + 32 * lq) * ors + (size_t)(h0 + hi) * DV + hf * (DV / 2) + 4 * (lane & 7);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = 4 * i + (lane >> 3);
            const float4 v = ld4(stage + 32 * r + 4 * ((lane & 7) ^ (r & 7)));
            if (32 * lq + r < nval) st_cs(reinterpret_cast<float4*>(ob + (size_t)r * ors), v);
        }
        __syncwarp();   // read back before the next head's epilogue writes the rows
    };
    int last = -1;    // the last head of the segment whose output product was issued
    for (int hi = 0; hi < hb && ok; ++hi) {
        const int h = h0 + hi;
        const float* lam = lam2 + (hi & 1) * CH;
        const float* omh = om2 + (hi & 1) * CH;
        if (warp == DWARP && hi + 1 < hb) head_d(h + 1);
        // this head's Q K^T (first head) and P are complete; so is the previous
        // head's output product, which read the A and v^T buffers
        bool w = mbar_wait(barM, pm & 1u, a.wait_ns);
        ++pm;
        if (hi > 0) {
            const bool wo = __syncthreads_and(mbar_wait(barO, po & 1u, a.wait_ns));
            if (wo) {
                ++po;
                --o_pending;
            }
            w = w && wo;
        }
        ok = __syncthreads_and(w);
        tc::fence_after_sync();
        if (!ok) {
            if (tid == 0) record_error(a.st, SN_E_TIMEOUT, (SN_K_RECUR_CHUNK << 16) | SITE_OUT_WAIT1);
            break;
        }
        if (issuer && hi + 1 < hb) {   // the S' buffer is free again
            mbar_arrive_expect_tx(barS, DV * DKC * 4);
            bulk_load(bufS, tile(h + 1), DV * DKC * 4, barS);
        }
        const float lt = lam[t];
#pragma unroll
        for (int j0 = 64 * hf; j0 < 64 * hf + 64; j0 += 16) {
            if (j0 > 32 * lq + 31) {   // above the diagonal for the whole warp: zeros
#pragma unroll
                for (int q = 0; q < 4; ++q) st4(bufA + off128(t, j0 + 4 * q), make_float4(0.f, 0.f, 0.f, 0.f));
                continue;
            }
            float x[16], lj[16], wj[16];
            tc::ld16(lane_base + j0, x);
#pragma unroll
            for (int q = 0; q < 4; ++q) {   // the block's decay sums and weights, broadcast to the warp
                const float4 l4 = ld4(lam + j0 + 4 * q), w4 = ld4(omh + j0 + 4 * q);
                lj[4 * q] = l4.x; lj[4 * q + 1] = l4.y; lj[4 * q + 2] = l4.z; lj[4 * q + 3] = l4.w;
                wj[4 * q] = w4.x; wj[4 * q + 1] = w4.y; wj[4 * q + 2] = w4.z; wj[4 * q + 3] = w4.w;
            }
            if (j0 + 15 <= 32 * lq) {   // below the diagonal for the whole warp
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) x[jj] *= ex2(lt - lj[jj]) * wj[jj];
            } else {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) x[jj] *= j0 + jj <= t ? ex2(lt - lj[jj]) * wj[jj] : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                st4(bufA + off128(t, j0 + 4 * q), tf32x4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]));
        }
#pragma unroll
        for (int t4 = 0; t4 < TP / 4; ++t4)
            st4(bufV + off128(col, part * TP + 4 * t4),
                tf32x4(vr[4 * t4], vr[4 * t4 + 1], vr[4 * t4 + 2], vr[4 * t4 + 3]));
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (issuer) {
            tc::gemm_tf32(tmem + col_o(hi), bufA, bufV, CH, tc::idesc_tf32(128, DV), false);
            tc::commit(barO);
        }
        ++o_pending;
        last = hi;
        if (hi > 0) epilogue(hi - 1, fp_prev);   // while this head's output product runs
        fp_prev = ex2(lt);
        if (hi + 1 < hb) {   // next head's v and decay sums, then its P once its S' tile is in
            load_v(h + 1);
            if (warp == DWARP) head_lam(lam2 + ((hi + 1) & 1) * CH);
            tc::fence_before_sync();
            ok = __syncthreads_and(mbar_wait(barS, ps & 1u, a.wait_ns));
            tc::fence_after_sync();
            if (!ok) {
                if (issuer) {
                    record_error(a.st, SN_E_TIMEOUT, (SN_K_RECUR_CHUNK << 16) | SITE_OUT_COPY);
                    mbar_wait(barS, ps & 1u, a.wait_ns);
                }
                break;
            }
            ++ps;
            if (issuer) {   // P[(hi + 1) & 1] was read by the epilogue above
                tc::gemm_tf32(tmem + col_p(hi + 1), bufQ, bufS, DKC, tc::idesc_tf32(128, DV), false);
                tc::commit(barM);
            }
        }
    }
    if (o_pending > 0) {
        // the segment's last output product, then its epilogue; on an error
        // the wait only drains the tensor pipe before the CTA frees its memory
        const bool w = __syncthreads_and(mbar_wait(barO, po & 1u, a.wait_ns));
        tc::fence_after_sync();
        if (w) {
            ++po;
            --o_pending;
        }
        if (ok && w) epilogue(last, fp_prev);
        if (!w) {
            if (tid == 0) record_error(a.st, SN_E_TIMEOUT, (SN_K_RECUR_CHUNK << 16) | SITE_OUT_WAIT2);
            ok = false;
        }
    }
    }   // segments
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// TMA maps of q and k for the output kernel: (B, T, G * dk) row-major, boxes
// of 32 keys x 128 tokens, 128-byte swizzle.
bool make_qk_maps(const ChunkArgs& a, CUtensorMap* mq, CUtensorMap* mk) {
    const uint64_t dims[3] = {(uint64_t)a.G * DKC, (uint64_t)a.T, (uint64_t)a.B};
    const uint64_t strides[2] = {(uint64_t)a.G * DKC * 4, (uint64_t)a.T * a.G * DKC * 4};
    const uint32_t box[3] = {32, (uint32_t)CH, 1};
    return encode_tiled(mq, 3, a.q, dims, strides, box, true) && encode_tiled(mk, 3, a.k, dims, strides, box, true);
}

// TMA map of o for the output kernel's stores: (B, T, H * dv) row-major,
// boxes of 32 values x 128 tokens, 128-byte swizzle (the staging layout).
// Without o the map is left zero: the kernel then stores nothing.
bool make_o_map(const ChunkArgs& a, int dv, CUtensorMap* mo) {
    *mo = CUtensorMap{};
    if (a.o == nullptr) return true;
    const uint64_t dims[3] = {(uint64_t)a.H * dv, (uint64_t)a.T, (uint64_t)a.B};
    const uint64_t strides[2] = {(uint64_t)a.H * dv * 4, (uint64_t)a.T * a.H * dv * 4};
    const uint32_t box[3] = {32, (uint32_t)CH, 1};
    return encode_tiled(mo, 3, a.o, dims, strides, box, true);
}

// TMA maps of k, d and v for chunk_state_key: (B, T, features) row-major,
// boxes of 128 tokens x all of a head's features (k: 128 keys of the group,
// d: 128 keys of the head, v: dv values of the head), no swizzle.
template <int DV>
bool make_natural_maps(const ChunkArgs& a, CUtensorMap* mk, CUtensorMap* md, CUtensorMap* mv) {
    const uint64_t dk_[3] = {(uint64_t)a.G * DKC, (uint64_t)a.T, (uint64_t)a.B};
    const uint64_t sk_[2] = {(uint64_t)a.G * DKC * 4, (uint64_t)a.T * a.G * DKC * 4};
    const uint64_t dd_[3] = {(uint64_t)a.H * DKC, (uint64_t)a.T, (uint64_t)a.B};
    const uint64_t sd_[2] = {(uint64_t)a.H * DKC * 4, (uint64_t)a.T * a.H * DKC * 4};
    const uint64_t dv_[3] = {(uint64_t)a.H * DV, (uint64_t)a.T, (uint64_t)a.B};
    const uint64_t sv_[2] = {(uint64_t)a.H * DV * 4, (uint64_t)a.T * a.H * DV * 4};
    const uint32_t bk[3] = {DKC, (uint32_t)CH, 1}, bv[3] = {DV, (uint32_t)CH, 1};
    return encode_tiled(mk, 3, a.k, dk_, sk_, bk, false) && encode_tiled(md, 3, a.d, dd_, sd_, bk, false) &&
           encode_tiled(mv, 3, a.v, dv_, sv_, bv, false);
}

// TMA maps of k and v for chunk_state_heads: natural boxes of 128 tokens x
// 128 keys (k) and x dv values (v), no swizzle.
template <int DV>
bool make_heads_maps(const ChunkArgs& a, CUtensorMap* mk, CUtensorMap* mv) {
    const uint64_t dk_[3] = {(uint64_t)a.G * DKC, (uint64_t)a.T, (uint64_t)a.B};
    const uint64_t sk_[2] = {(uint64_t)a.G * DKC * 4, (uint64_t)a.T * a.G * DKC * 4};
    const uint64_t dv_[3] = {(uint64_t)a.H * DV, (uint64_t)a.T, (uint64_t)a.B};
    const uint64_t sv_[2] = {(uint64_t)a.H * DV * 4, (uint64_t)a.T * a.H * DV * 4};
    const uint32_t bk[3] = {DKC, (uint32_t)CH, 1}, bv[3] = {DV, (uint32_t)CH, 1};
    return encode_tiled(mk, 3, a.k, dk_, sk_, bk, false) && encode_tiled(mv, 3, a.v, dv_, sv_, bv, false);
}

template <bool PER_KEY, int DV>
cudaError_t run_chunked(const ChunkArgs& a, int sm_count, cudaStream_t s) {
    constexpr bool HEADS = !PER_KEY && DV == 64;   // per-head decays: heads of a group share Q K^T
    size_t st_bytes;
    size_t out_bytes;
    cudaError_t e;
    if constexpr (HEADS) {
        st_bytes = StateHeadsSmem<DV>::bytes;
        e = set_smem_attr_once((const void*)chunk_state_heads<DV>, st_bytes);
    } else if constexpr (PER_KEY) {
        st_bytes = StateKeySmem<DV>::bytes;
        e = set_smem_attr_once((const void*)chunk_state_key<DV>, st_bytes);
    } else {
        st_bytes = StateSmem<DV>::bytes;
        e = set_smem_attr_once((const void*)chunk_state<DV>, st_bytes);
    }
    if (e != cudaSuccess) return e;
    if constexpr (HEADS) {
        out_bytes = HeadsSmem<DV>::bytes;
        e = set_smem_attr_once((const void*)chunk_output_heads<DV>, out_bytes);
    } else {
        out_bytes = OutSmem<DV>::bytes;
        e = set_smem_attr_once((const void*)chunk_output<PER_KEY, DV>, out_bytes);
    }
    if (e != cudaSuccess) return e;
    const unsigned chunks = (unsigned)((size_t)a.B * a.H * a.NC);
    if constexpr (HEADS) {
        CUtensorMap mk, mv;
        if (!make_heads_maps<DV>(a, &mk, &mv)) return cudaErrorInvalidValue;
        const int64_t items = (int64_t)a.B * a.NC * a.H;   // spread evenly over one CTA per SM
        chunk_state_heads<DV><<<(unsigned)std::min<int64_t>(items, sm_count), NT, st_bytes, s>>>(mk, mv, a);
    } else if constexpr (PER_KEY) {
        CUtensorMap mk, md, mv;
        if (!make_natural_maps<DV>(a, &mk, &md, &mv)) return cudaErrorInvalidValue;
        chunk_state_key<DV><<<chunks, NT, st_bytes, s>>>(mk, md, mv, a);
    } else {
        chunk_state<DV><<<chunks, NT, st_bytes, s>>>(a);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t entries = (size_t)a.B * a.H * DKC * DV;
    if ((int64_t)(entries / 4 + 255) / 256 >= 4 * (int64_t)sm_count)   // four CTAs per SM with 16-byte groups
        chunk_carry<4><<<(unsigned)((entries / 4 + 255) / 256), 256, 0, s>>>(a, DV);
    else
        chunk_carry<1><<<(unsigned)((entries + 255) / 256), 256, 0, s>>>(a, DV);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if constexpr (HEADS) {
        // the (batch, chunk, group, head) items spread evenly over one CTA per SM
        const int64_t items = (int64_t)a.B * a.NC * a.H;
        chunk_output_heads<DV><<<(unsigned)std::min<int64_t>(items, sm_count), NT, out_bytes, s>>>(a);
    } else {
        CUtensorMap mq, mk, mo;
        if (!make_qk_maps(a, &mq, &mk) || !make_o_map(a, DV, &mo)) return cudaErrorInvalidValue;
        chunk_output<PER_KEY, DV><<<(unsigned)std::min<size_t>(chunks, (size_t)sm_count), NT, out_bytes, s>>>(mq, mk, mo,
                                                                                                             a);
    }
    return cudaGetLastError();
}

int64_t round256(int64_t x) { return (x + 255) / 256 * 256; }

}  // namespace

// The output stage alone with unit decays (a.d == nullptr, per-head path):
// o = scale (Q S_n + tril(Q K^T) V) for every chunk, with V and the chunk
// states S_n (operand layout, tf32) supplied by the caller; dv = 128.
cudaError_t chunk::launch_output_unit_decay(const ChunkArgs& a, int max_ctas, cudaStream_t s) {
    const size_t bytes = OutSmem<128>::bytes;
    const cudaError_t e = set_smem_attr_once((const void*)chunk_output<false, 128>, bytes);
    if (e != cudaSuccess) return e;
    const int nsg = a.nsg > 0 ? a.nsg : a.NC;
    const size_t units = (size_t)a.B * a.H * nsg;
    CUtensorMap mq, mk, mo;
    if (!make_qk_maps(a, &mq, &mk) || !make_o_map(a, 128, &mo)) return cudaErrorInvalidValue;
    chunk_output<false, 128><<<(unsigned)std::min<size_t>(units, (size_t)max_ctas), NT, bytes, s>>>(mq, mk, mo, a);
    return cudaGetLastError();
}

const void* chunk::output_unit_decay_kernel() { return (const void*)chunk_output<false, 128>; }
size_t chunk::output_unit_decay_smem() { return OutSmem<128>::bytes; }
bool chunk::output_maps(const ChunkArgs& a, int dv, CUtensorMap* mq, CUtensorMap* mk, CUtensorMap* mo) {
    return make_qk_maps(a, mq, mk) && make_o_map(a, dv, mo);
}

int64_t chunked_ws_bytes(int B, int T, int H, int dk, int dv) {
    const int64_t nc = (T + CH - 1) / CH;
    return round256((int64_t)B * H * nc * dk * dv * 4) + 2 * round256((int64_t)B * H * nc * dk * 4) +
           round256((int64_t)B * H * nc * 4) + round256((int64_t)B * H * nc * dv * CH * 4);
}

bool chunked_supported(const RecurArgs& x) {
    return (x.kind == RK_DIAG_KEY || x.kind == RK_DIAG_HEAD || x.kind == RK_DIAG_KEY_GATED ||
            x.kind == RK_DIAG_HEAD_GATED) &&
           x.dk == DKC && (x.dv == 64 || x.dv == 128);
}

cudaError_t launch_recur_chunked(const RecurArgs& x, void* ws, SnDevStatus* st, uint64_t wait_ns, int sm_count,
                                 cudaStream_t s) {
    ChunkArgs a{};
    a.B = x.B; a.T = x.T; a.H = x.H; a.G = x.G;
    a.NC = (x.T + CH - 1) / CH;
    a.scale = x.scale;
    a.q = x.q; a.k = x.k; a.v = x.v; a.d = x.g;
    a.S_in = x.S_in; a.S_out = x.S_out; a.o = x.o;
    char* p = static_cast<char*>(ws);
    a.W = reinterpret_cast<float*>(p);
    p += round256((int64_t)x.B * x.H * a.NC * x.dk * x.dv * 4);
    a.gam = reinterpret_cast<float*>(p);
    p += round256((int64_t)x.B * x.H * a.NC * x.dk * 4);
    a.anc = reinterpret_cast<float*>(p);
    p += round256((int64_t)x.B * x.H * a.NC * x.dk * 4);
    const bool per_key = x.kind == RK_DIAG_KEY || x.kind == RK_DIAG_KEY_GATED;
    a.bad = per_key ? reinterpret_cast<int*>(p) : nullptr;   // written by chunk_state every call
    p += round256((int64_t)x.B * x.H * a.NC * 4);
    // per key: chunk_state_key leaves its rounded v^T tiles for the output
    // stage (for the heads kernels this measured slower: 0.277 -> 0.289 ms
    // on the Mamba-2 workload, the tiles' extra writes outweighing the
    // 4-byte loads they replace)
    a.vt_out = per_key ? reinterpret_cast<float*>(p) : nullptr;
    a.vt = a.vt_out;
    a.st = st;
    a.wait_ns = wait_ns;
    a.gated = x.kind == RK_DIAG_KEY_GATED || x.kind == RK_DIAG_HEAD_GATED;
    if (x.dv == 128) return per_key ? run_chunked<true, 128>(a, sm_count, s) : run_chunked<false, 128>(a, sm_count, s);
    return per_key ? run_chunked<true, 64>(a, sm_count, s) : run_chunked<false, 64>(a, sm_count, s);
}

}  // namespace sn
