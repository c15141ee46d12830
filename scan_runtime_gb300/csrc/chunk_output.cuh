// chunk_output.cuh -- the output stage of the chunked tensor-core forms (one
// chunk of one head per unit) as a loop over a schedule of units.  Shared by
// recur_chunked.cu (chunk_output: units i, i + grid, ... of a launch) and
// recur_delta_chunked.cu (the fused delta rule: units claimed from a counter,
// each once the chains have written its tiles).
#pragma once

#include "chunk_common.cuh"

namespace sn {
namespace {

using namespace chunk;

// ------------------------------------------------------------------ chunk_output
// Persistent: a CTA takes its units from a schedule (StaticUnits: units i,
// i + grid, ...; a unit is one chunk of one head), and the next unit's
// operands stream in as the current unit frees
// their space: its decays into registers after the rescaling, its S' tile
// into the S buffer after the first two products, its v slice into registers
// after the first epilogue, and its q and k rows into the Q and K buffers
// after the last product.  q and k arrive by TMA in the 128-byte-swizzled
// K-major layout (four 32-key x 128-token boxes each; rows past T are filled
// with zeros), which the first two products read directly.
template <int DV>
struct OutSmem {
    static constexpr int q_off = 0;              // Qt, later the masked A
    static constexpr int k_off = OPF;            // Kt, later v^T
    static constexpr int s_off = 2 * OPF;        // S'^T (rows c, K = i)
    static constexpr int lam_off = s_off + DV * DKC;   // [CH] per-head lam
    static constexpr int om_off = lam_off + CH;        // [CH] per-head injection weights
    static constexpr int misc_off = om_off + CH;
    static constexpr size_t bytes = (size_t)(misc_off + 16) * 4 + 1024;
};

// The schedule of chunk_output: units i, i + grid, ... of the launch, in
// chunk_index order, all of whose tiles exist when the kernel starts.  A
// schedule gives the first and the next unit (thread 0 asks; -1 = none), a
// unit's chunk, and ready(): thread 0 returns from it once the unit's S'
// and v^T tiles may be read (false: it gave up and recorded the error).
struct StaticUnits {
    int units;
    static constexpr bool kDynamic = false;
    __device__ int first() const { return (int)blockIdx.x < units ? (int)blockIdx.x : -1; }
    __device__ int next(int u) const { return u + (int)gridDim.x < units ? u + (int)gridDim.x : -1; }
    __device__ ChunkIdx index(const ChunkArgs& a, int u) const { return chunk_index(a, u); }
    __device__ bool ready(const ChunkArgs&, const ChunkIdx&) const { return true; }
};

// per-key chunks flagged out of the factors' range (recur_chunked.cu)
template <int DV>
struct FixSmem;
template <int DV>
__device__ __forceinline__ void fix_unit(const ChunkArgs& a, const ChunkIdx& c, float* base);

template <bool PER_KEY, int DV, class Units>
__device__ __forceinline__ void output_loop(const CUtensorMap* map_q, const CUtensorMap* map_k,
                                            const CUtensorMap* map_o, const ChunkArgs& a, Units& sch) {
    static_assert(!(PER_KEY && Units::kDynamic), "flagged per-key units run on the static schedule");
    extern __shared__ unsigned char smem_raw[];
    using L = OutSmem<DV>;
    float* base = reinterpret_cast<float*>(smem_align<1024>(smem_raw));
    float* bufQ = base + L::q_off;
    float* bufK = base + L::k_off;
    float* bufS = base + L::s_off;
    float* lam_s = base + L::lam_off;
    float* om_s = base + L::om_off;
    uint64_t* barS = reinterpret_cast<uint64_t*>(base + L::misc_off);       // S' tiles, one per unit
    uint64_t* barM = reinterpret_cast<uint64_t*>(base + L::misc_off + 2);   // products, two per unit
    uint64_t* barV = reinterpret_cast<uint64_t*>(base + L::misc_off + 4);   // v^T tiles, one per unit
    uint64_t* barQ = reinterpret_cast<uint64_t*>(base + L::misc_off + 6);   // q and k tiles, one pair per unit
    uint32_t* slot = reinterpret_cast<uint32_t*>(base + L::misc_off + 8);
    int* s_unit = reinterpret_cast<int*>(base + L::misc_off + 10);          // thread 0's unit, for every thread

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // rescaling of q, k (and the per-key decays): warp = 16 key columns,
    // lane = (token mod 8, 4-column group)
    const int tl = lane & 7, ig = lane >> 3;
    const int ic = 16 * warp + 4 * ig;
    // v slice for the last product, in registers: thread = value column, a run
    // of tokens (unless the caller supplies the v^T operand tiles)
    constexpr int TP = CH / (NT / DV);
    const int col = tid % DV, part = tid / DV;
    // tensor-memory rows: warp quarter lq, token t
    const int lq = warp & 3, hf = warp >> 2;
    const int t = 32 * lq + lane;

    if (warp == 0) tc::tmem_alloc_keep(slot, 256);
    if (tid == 0) {
        mbar_init(barS, 1);
        mbar_init(barM, 1);
        mbar_init(barV, 1);
        mbar_init(barQ, 1);
        fence_mbar_init();
        *s_unit = sch.first();
    }
    __syncthreads();   // barriers initialised before any thread polls them
    tc::fence_after_sync();
    const uint32_t tmem = *slot;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * lq) << 16);

    // operands of the unit being loaded (registers are filled by the loads in flight)
    float vr[TP];
    float4 draw[CH / 8];   // per-key decays, lane mapping of q and k
    float lgh[4];          // per-head decays of tokens 4 lane .. 4 lane + 3 (warp 0)
    int s_loads = 0, v_loads = 0, q_loads = 0;   // copies issued on barS / barV / barQ (thread 0's count)

    auto issue_s = [&](const ChunkIdx& c) {   // thread 0: the chunk's S' operand, one contiguous tile
        mbar_arrive_expect_tx(barS, DV * DKC * 4);
        bulk_load(bufS, a.W + (c.bh * a.NC + c.n) * (size_t)DV * DKC, DV * DKC * 4, barS);
        ++s_loads;
    };
    // thread 0: the q and k tiles, four swizzled 32-key boxes each, on one
    // barrier phase that expects both (k may be requested later than q)
    auto issue_q = [&](const ChunkIdx& c) {
        mbar_arrive_expect_tx(barQ, 2 * OPF * 4);
#pragma unroll
        for (int at = 0; at < DKC / 32; ++at) tma_load_3d(bufQ + at * 4096, map_q, barQ, c.g * DKC + 32 * at, c.t0, c.b);
        ++q_loads;
    };
    auto issue_k = [&](const ChunkIdx& c) {
#pragma unroll
        for (int at = 0; at < DKC / 32; ++at) tma_load_3d(bufK + at * 4096, map_k, barQ, c.g * DKC + 32 * at, c.t0, c.b);
    };
    auto issue_v = [&](const ChunkIdx& c) {   // all threads: the v slice into registers
        if (a.vt != nullptr) return;
        const size_t row0 = (size_t)c.b * a.T + c.t0;
        const size_t vrs = (size_t)a.H * DV;
        const float* vcol = a.v + row0 * vrs + (size_t)c.h * DV + col;
#pragma unroll
        for (int r = 0; r < TP; ++r) {
            const int tt = part * TP + r;
            vr[r] = tt < c.nval ? __ldg(vcol + (size_t)tt * vrs) : 0.f;
        }
    };
    auto issue_d = [&](const ChunkIdx& c) {   // the decays into registers
        const size_t row0 = (size_t)c.b * a.T + c.t0;
        if (PER_KEY) {
            const size_t drs = (size_t)a.H * DKC;
            const float* db = a.d + row0 * drs + (size_t)c.h * DKC + ic;
#pragma unroll
            for (int tb = 0; tb < CH / 8; ++tb) {
                const int tt = 8 * tb + tl;
                draw[tb] = tt < c.nval ? ldg4(db + (size_t)tt * drs) : make_float4(1.f, 1.f, 1.f, 1.f);
            }
        } else if (warp == 0) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int tt = 4 * lane + r;
                lgh[r] = (tt < c.nval && a.d != nullptr) ? __ldg(a.d + (row0 + tt) * a.H + c.h) : 1.f;
            }
        }
    };

    bool ok = true;
    int site = 0;
    const int u0 = *s_unit;
    if (u0 >= 0) {
        const ChunkIdx c0 = sch.index(a, u0);
        if (tid == 0) {
            issue_q(c0);
            issue_k(c0);
            (void)sch.ready(a, c0);   // on a give-up the error is recorded and the copy reads what is there
            issue_s(c0);
        }
        issue_v(c0);
        issue_d(c0);
    }
    for (int u = u0, it = 0; u >= 0; ++it) {
        const ChunkIdx c = sch.index(a, u);
        // thread 0 takes the next unit now; every thread reads it after the q, k barrier
        if (tid == 0) *s_unit = sch.next(u);
        const uint32_t ph = (uint32_t)it & 1;

        // decay prefix sums: per key in registers (the q, k lane mapping), per head in shared memory
        float4 lam[CH / 8];
        float4 lm = make_float4(0.f, 0.f, 0.f, 0.f);
        if (PER_KEY) {
            float4 carry = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int tb = 0; tb < CH / 8; ++tb) {
                float4 x = make_float4(lg2(draw[tb].x), lg2(draw[tb].y), lg2(draw[tb].z), lg2(draw[tb].w));
#pragma unroll
                for (int off = 1; off < 8; off <<= 1) {
                    const float yx = __shfl_up_sync(FULL, x.x, off, 8), yy = __shfl_up_sync(FULL, x.y, off, 8);
                    const float yz = __shfl_up_sync(FULL, x.z, off, 8), yw = __shfl_up_sync(FULL, x.w, off, 8);
                    if (tl >= off) {
                        x.x += yx; x.y += yy; x.z += yz; x.w += yw;
                    }
                }
                x.x += carry.x; x.y += carry.y; x.z += carry.z; x.w += carry.w;
                carry = make_float4(__shfl_sync(FULL, x.x, 7, 8), __shfl_sync(FULL, x.y, 7, 8),
                                    __shfl_sync(FULL, x.z, 7, 8), __shfl_sync(FULL, x.w, 7, 8));
                if (tb == ANCHOR / 8) lm = carry;
                lam[tb] = x;
            }
            // a chunk chunk_state flagged (factors beyond 2^{+-RANGE_LOG2}) runs
            // through here too; its stores are skipped and fix_unit writes them
        } else if (warp == 0) {
            // inclusive prefix sums of log2 d (per head) into lam_s
            float lg[4], sm = 0.f;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                lg[r] = lg2(lgh[r]);
                om_s[4 * lane + r] = a.gated ? 1.f - lgh[r] : 1.f;
                sm += lg[r];
            }
            float x = sm;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(FULL, x, off);
                if (lane >= off) x += y;
            }
            float acc = x - sm;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                acc += lg[r];
                lam_s[4 * lane + r] = acc;
            }
            const float total = __shfl_sync(FULL, x, 31);
            if (lane == 0 && !isfinite(total))
                record_error(a.st, SN_E_RANGE, (SN_K_RECUR_CHUNK << 16) | SITE_RANGE_HEAD);
        }

        // Qt, Kt in place, in the swizzled layout
        ok = __syncthreads_and(mbar_wait(barQ, ph, a.wait_ns));
        if (!ok) {
            site = SITE_OUT_COPY;
            break;
        }
        const int un = *s_unit;
        const bool has_next = un >= 0;
        const ChunkIdx cn = sch.index(a, has_next ? un : u);
#pragma unroll
        for (int tb = 0; tb < CH / 8; ++tb) {
            const int o = off_sw(8 * tb + tl, ic);
            const float4 q4 = ld4(bufQ + o), k4 = ld4(bufK + o);
            if (PER_KEY) {
                const float4 x = lam[tb];
                // gated: the key enters with weight 1 - d (the raw decays are still in draw)
                const float4 w = a.gated ? make_float4(1.f - draw[tb].x, 1.f - draw[tb].y, 1.f - draw[tb].z,
                                                       1.f - draw[tb].w)
                                         : make_float4(1.f, 1.f, 1.f, 1.f);
                st4(bufQ + o, tf32x4(q4.x * ex2(x.x - lm.x), q4.y * ex2(x.y - lm.y), q4.z * ex2(x.z - lm.z),
                                     q4.w * ex2(x.w - lm.w)));
                st4(bufK + o, tf32x4(k4.x * ex2(lm.x - x.x) * w.x, k4.y * ex2(lm.y - x.y) * w.y,
                                     k4.z * ex2(lm.z - x.z) * w.z, k4.w * ex2(lm.w - x.w) * w.w));
            } else {
                const float w = om_s[8 * tb + tl];
                st4(bufQ + o, tf32x4(q4));
                st4(bufK + o, tf32x4(k4.x * w, k4.y * w, k4.z * w, k4.w * w));
            }
        }

        if (has_next) issue_d(cn);   // this unit's decays are consumed: the next unit's stream in
        fence_proxy_async_smem();
        tc::fence_before_sync();
        ok = __syncthreads_and(mbar_wait(barS, ph, a.wait_ns));
        tc::fence_after_sync();
        if (!ok) {
            site = SITE_OUT_COPY;
            break;
        }
        if (tid == 0) {
            tc::gemm_tf32_sw_sw(tmem, bufQ, bufK, tc::idesc_tf32(128, 128), false);          // A (cols 0..127)
            tc::gemm_tf32_sw_plain(tmem + 128, bufQ, bufS, tc::idesc_tf32(128, DV), false);  // P (cols 128..)
            tc::commit(barM);
        }
        ok = __syncthreads_and(mbar_wait(barM, 0, a.wait_ns));
        tc::fence_after_sync();
        if (!ok) {
            site = SITE_OUT_WAIT1;
            break;
        }
        if (tid == 0) {
            // the K buffer is free: the v^T tile streams in; the S buffer is free: the next unit's S'
            if (a.vt != nullptr) {
                mbar_arrive_expect_tx(barV, DV * CH * 4);
                bulk_load(bufK, a.vt + (c.bh * a.NC + c.n) * (size_t)DV * CH, DV * CH * 4, barV);
                ++v_loads;
            }
            if (has_next) {
                (void)sch.ready(a, cn);
                issue_s(cn);
            }
        }
        {
            const float lt = PER_KEY ? 0.f : lam_s[t];
            // masked (and, per head, decay-weighted) A into the Q buffer as the next A operand
#pragma unroll
            for (int j0 = 64 * hf; j0 < 64 * hf + 64; j0 += 16) {
                float x[16];
                tc::ld16(lane_base + j0, x);
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    // selected, not multiplied: an entry above the diagonal may be
                    // infinite (its anchor factors are not a decay product)
                    const int j = j0 + jj;
                    x[jj] = j <= t ? (PER_KEY ? x[jj] : x[jj] * ex2(lt - lam_s[j])) : 0.f;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    st4(bufQ + off128(t, j0 + 4 * q), tf32x4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]));
            }
            if (a.vt == nullptr) {
#pragma unroll
                for (int t4 = 0; t4 < TP / 4; ++t4)
                    st4(bufK + off128(col, part * TP + 4 * t4),
                        tf32x4(vr[4 * t4], vr[4 * t4 + 1], vr[4 * t4 + 2], vr[4 * t4 + 3]));
            }
        }
        if (has_next) issue_v(cn);   // this unit's v slice is in the K buffer: the next unit's streams in
        fence_proxy_async_smem();
        tc::fence_before_sync();
        ok = __syncthreads_and(a.vt == nullptr || mbar_wait(barV, ph, a.wait_ns));
        tc::fence_after_sync();
        if (!ok) {
            site = SITE_OUT_COPY;
            break;
        }
        if (tid == 0) {
            tc::gemm_tf32(tmem, bufQ, bufK, CH, tc::idesc_tf32(128, DV), false);   // O (cols 0..DV-1)
            tc::commit(barM);
        }
        ok = __syncthreads_and(mbar_wait(barM, 1, a.wait_ns));
        tc::fence_after_sync();
        if (!ok) {
            site = SITE_OUT_WAIT2;
            break;
        }
        // The Q buffer is free: the next unit's q streams in.  The unit's o
        // tile goes through the K buffer (128-byte-swizzled 32-column boxes,
        // written row by row without bank conflicts) and out by TMA stores,
        // which clip the rows past T; the next unit's k follows once the
        // stores have read it.  A flagged unit's outputs come from fix_unit.
        if (has_next && tid == 0) issue_q(cn);
        const bool out_unit = a.o != nullptr && !(PER_KEY && __ldg(a.bad + c.bh * a.NC + c.n) != 0);
        if (out_unit) {
            const float fp = PER_KEY ? 1.f : ex2(lam_s[t]);
#pragma unroll
            for (int c0 = hf * (DV / 2); c0 < (hf + 1) * (DV / 2); c0 += 16) {
                float p[16], x[16];
                tc::ld16(lane_base + 128 + c0, p);
                tc::ld16(lane_base + c0, x);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    st4(bufK + off_sw(t, c0 + 4 * q),
                        make_float4(a.scale * fmaf(fp, p[4 * q], x[4 * q]), a.scale * fmaf(fp, p[4 * q + 1], x[4 * q + 1]),
                                    a.scale * fmaf(fp, p[4 * q + 2], x[4 * q + 2]),
                                    a.scale * fmaf(fp, p[4 * q + 3], x[4 * q + 3])));
            }
            fence_proxy_async_smem();
        }
        __syncthreads();
        if (tid == 0) {
            if (out_unit) {
#pragma unroll
                for (int at = 0; at < DV / 32; ++at) tma_store_3d(map_o, bufK + at * 4096, c.h * DV + 32 * at, c.t0, c.b);
                bulk_commit();
                bulk_wait_read_all();
            }
            if (has_next) issue_k(cn);
        }
        // tensor memory and the per-head sums are reused by the next unit
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        u = un;
    }
    if constexpr (PER_KEY) {
        // this CTA's flagged units, step by step (their stores were skipped above)
        if (ok) {
            static_assert(FixSmem<DV>::bytes <= (size_t)L::misc_off * 4,
                          "the fix reuses the operand buffers, not the barriers");
            for (int u = sch.first(); u >= 0; u = sch.next(u)) {
                const ChunkIdx c = chunk_index(a, u);
                if (__ldg(a.bad + c.bh * a.NC + c.n) != 0) fix_unit<DV>(a, c, base);
            }
        }
    }
    if (!ok && tid == 0) {
        record_error(a.st, SN_E_TIMEOUT, (SN_K_RECUR_CHUNK << 16) | site);
        // at most one copy per barrier can still be in flight: let it land
        if (s_loads > 0) (void)mbar_wait(barS, (uint32_t)(s_loads - 1) & 1, a.wait_ns);
        if (v_loads > 0) (void)mbar_wait(barV, (uint32_t)(v_loads - 1) & 1, a.wait_ns);
        if (q_loads > 0) (void)mbar_wait(barQ, (uint32_t)(q_loads - 1) & 1, a.wait_ns);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

}  // namespace
}  // namespace sn
