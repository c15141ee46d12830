// scan_bwd_chunked.cu -- chunked reverse scans (the backward pass of both
// tier-1 forms) for few channels and long T, sm_103a.
//
// The reverse recurrence of the adjoint ("SunnyNet 工程化实录" §2.1 forms; the
// pages ship forward and reverse entries, §8)
//     g_{T-1} = gs_{T-1} + gf,    g_t = fma(a_{t+1}, g_{t+1}, gs_t)
// is a first-order linear recurrence run backwards in time, with multiplier
// alpha_t = a_{t+1} (alpha_{T-1} = 1, g_T = gf).  scan_bwd.cu runs it
// sequentially per channel, which leaves most SMs idle when B * N is small.
// Here it is chunked like the forward reduce-then-scan (scan_lookback.cu):
//   bwd_pass<.., false>  every tile's reverse aggregate (A_k, B_k) per channel;
//   scan_chain<true>     per column, h_k = fma(A_k, h_{k+1}, B_k) from the last
//                        chunk down, h_{nchunks} = gf (h_k = g at the chunk's
//                        first step);
//   bwd_pass<.., true>   every tile's g from its incoming h_{k+1}, and the
//                        gradients: FMA da_t = g_t s_{t-1}, db_t = g_t;
//                        gated da_t = g_t (s_{t-1} - u_t), du_t = g_t (1 - a_t);
//                        ds0 = a_0 g_0.
// A tile holds a as 129 rows (its own steps and the next chunk's first a, the
// alpha of its last step), gs, the forward states shifted one step back (row
// 0 = s_{t0-1}; s0 for the first chunk) and u.  The chunked order rounds
// differently from the sequential kernel (the same tolerance to the
// definition), is deterministic, and splits at multiples of 128 steps give
// the same bits, because the chunk's first g is the chain's value.
#include "scan_tile.cuh"

namespace sn {
namespace {

constexpr int BT_STAGES = 2;
constexpr int BT_AROWS = LB_TC + 1;                       // rows of a per tile
template <bool GATED, bool OUT>
constexpr int bt_tile_floats() {   // a (129 rows), gs, then (outputs) s_{t-1} and (gated) u
    return (BT_AROWS + LB_TC + (OUT ? LB_TC : 0) + (OUT && GATED ? LB_TC : 0)) * LB_NC;
}
template <bool GATED, bool OUT>
constexpr size_t bt_smem() { return (size_t)BT_STAGES * bt_tile_floats<GATED, OUT>() * 4 + BT_STAGES * 8 + 16; }

struct BwdPassParams {
    int B, T, N, ncb, nbcb, nchunks, ntiles;
    const float* a;      // (B, T, N), for a_0 of ds0
    const float* s0;
    const float* gf;
    float* da;
    float* dbu;
    float* ds0;
    float* dA;           // aggregates at agg_index (chunks in groups of four), then the chain's h_k in dC
    float* dB;
    float* dC;
    SnDevStatus* st;
    uint64_t wait_ns;
};

template <bool GATED, bool OUT>
__global__ void __launch_bounds__(LB_THREADS, OUT ? 2 : 3)
bwd_pass(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_g,
         const __grid_constant__ CUtensorMap map_s, const __grid_constant__ CUtensorMap map_u, const BwdPassParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int TF = bt_tile_floats<GATED, OUT>();
    float* bufs = reinterpret_cast<float*>(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)BT_STAGES * TF * 4);
    __shared__ float4 wA[8][8], wB[8][8];
    __shared__ float carry[LB_NC], cfin[LB_NC];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = lane & 7, sub = lane >> 3;
    const int seg = warp * 4 + sub;

    if (tid == 0) {
        for (int s = 0; s < BT_STAGES; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // tiles column-major within a chunk row; the output pass visits them in the
    // opposite order, so it starts on the tiles the aggregate pass read last,
    // which are still in L2
    auto tile_coords = [&](int ti, int& k, int& bi, int& cb) {
        if (OUT) ti = p.ntiles - 1 - ti;
        k = ti / p.nbcb;
        const int r = ti - k * p.nbcb;
        bi = r / p.ncb;
        cb = r - bi * p.ncb;
    };
    constexpr uint32_t A_BYTES = BT_AROWS * LB_NC * 4, T_BYTES = LB_TC * LB_NC * 4;
    auto issue = [&](int ti, int buf) {
        int k, bi, cb;
        tile_coords(ti, k, bi, cb);
        float* dst = bufs + (size_t)buf * TF;
        mbar_arrive_expect_tx(&full[buf], A_BYTES + T_BYTES * (1 + (OUT ? 1 : 0) + (OUT && GATED ? 1 : 0)));
        tma_load_3d(dst, &map_a, &full[buf], cb * LB_NC, k * LB_TC, bi);
        tma_load_3d(dst + BT_AROWS * LB_NC, &map_g, &full[buf], cb * LB_NC, k * LB_TC, bi);
        if (OUT) {
            // the forward states one step back: row 0 is s_{t0 - 1} (row -1 of the sequence is read as zeros)
            tma_load_3d(dst + (BT_AROWS + LB_TC) * LB_NC, &map_s, &full[buf], cb * LB_NC, k * LB_TC - 1, bi);
            if (GATED) tma_load_3d(dst + (BT_AROWS + 2 * LB_TC) * LB_NC, &map_u, &full[buf], cb * LB_NC, k * LB_TC, bi);
        }
    };
    int it = 0;
    if (tid == 0) {
        for (int s = 0; s < BT_STAGES - 1; ++s) {
            const int ti = blockIdx.x + s * gridDim.x;
            if (ti < p.ntiles) issue(ti, s);
        }
    }
    for (int ti = blockIdx.x; ti < p.ntiles; ti += gridDim.x, ++it) {
        const int buf = it % BT_STAGES;
        const int ahead = ti + (BT_STAGES - 1) * (int)gridDim.x;
        if (tid == 0 && ahead < p.ntiles) issue(ahead, (it + BT_STAGES - 1) % BT_STAGES);
        int k, bi, cb;
        tile_coords(ti, k, bi, cb);
        const int t0 = k * LB_TC, n0 = cb * LB_NC;
        const int rows = min(LB_TC, p.T - t0);
        if (!__syncthreads_and(mbar_wait(&full[buf], (it / BT_STAGES) & 1, p.wait_ns))) {
            if (tid == 0) {
                record_error(p.st, SN_E_TIMEOUT, (SN_K_SCAN_LOOKBACK << 16) | 5);
                for (int j = 0; j < BT_STAGES; ++j)
                    if (ti + j * (int)gridDim.x < p.ntiles)
                        (void)mbar_wait(&full[(it + j) % BT_STAGES], ((it + j) / BT_STAGES) & 1, p.wait_ns);
            }
            return;
        }
        float* sa = bufs + (size_t)buf * TF;            // a: rows t0 .. t0 + 128
        float* sg = sa + BT_AROWS * LB_NC;              // gs
        float* ssp = sg + LB_TC * LB_NC;                // s_{t-1} (outputs)
        const float* su = ssp + LB_TC * LB_NC;          // u (gated outputs)
        // the sequence's edges: alpha of step T-1 is 1; s_{-1} is s0
        if (tid < LB_NC) {
            const int n = n0 + tid;
            if (t0 + rows == p.T) sa[rows * LB_NC + tid] = 1.f;
            if (OUT && k == 0) ssp[tid] = (p.s0 != nullptr && n < p.N) ? p.s0[(size_t)bi * p.N + n] : 0.f;
        }
        __syncthreads();
        float4 EA, EB;
        tile_local_scan<false, true>(sa + LB_NC, sg, rows, wA, wB, EA, EB);   // alpha_t = a_{t+1}
        const size_t col = (size_t)bi * p.ncb + cb;
        const int nq = chunk_quads(p.nchunks);
        const size_t me = agg_index(col, nq, k, lane);
        if (warp == 0) {
            if (!OUT) {
                float CA, CB;
                tile_aggregate(wA, wB, lane, CA, CB);
                p.dA[me] = CA;
                p.dB[me] = CB;
            } else {
                const int n = n0 + lane;
                // g entering the tile from above (h_{k+1}), and the tile's own first g (h_k)
                carry[lane] = k == p.nchunks - 1 ? ((p.gf != nullptr && n < p.N) ? p.gf[(size_t)bi * p.N + n] : 0.f)
                                                 : __ldg(p.dC + agg_index(col, nq, k + 1, lane));
                cfin[lane] = __ldg(p.dC + me);
            }
        }
        if (OUT) {
            __syncthreads();
            // g through this thread's segment (positions seg * LB_SEG .., rows rows - 1 - position),
            // then the gradients of each of its rows
            if (n0 + 4 * quad < p.N) {
                float4 g = f4fma(EA, *reinterpret_cast<const float4*>(&carry[4 * quad]), EB);
                const size_t rowN = (size_t)p.N;
                float* pa = p.da != nullptr ? p.da + ((size_t)bi * p.T + t0) * rowN + n0 + 4 * quad : nullptr;
                float* pb = p.dbu != nullptr ? p.dbu + ((size_t)bi * p.T + t0) * rowN + n0 + 4 * quad : nullptr;
#pragma unroll
                for (int i = 0; i < LB_SEG; ++i) {
                    const int pos = seg * LB_SEG + i;
                    if (pos < rows) {
                        const int r = rows - 1 - pos;
                        const float4 al = *reinterpret_cast<const float4*>(sa + (r + 1) * LB_NC + 4 * quad);
                        const float4 gv = *reinterpret_cast<const float4*>(sg + r * LB_NC + 4 * quad);
                        g = f4fma(al, g, gv);
                        if (pos == rows - 1) g = *reinterpret_cast<const float4*>(&cfin[4 * quad]);
                        const float4 sp = *reinterpret_cast<const float4*>(ssp + r * LB_NC + 4 * quad);
                        float4 oa, ob;
                        if (GATED) {
                            const float4 uv = *reinterpret_cast<const float4*>(su + r * LB_NC + 4 * quad);
                            const float4 av = *reinterpret_cast<const float4*>(sa + r * LB_NC + 4 * quad);
                            oa = make_float4(__fmul_rn(g.x, __fsub_rn(sp.x, uv.x)), __fmul_rn(g.y, __fsub_rn(sp.y, uv.y)),
                                             __fmul_rn(g.z, __fsub_rn(sp.z, uv.z)), __fmul_rn(g.w, __fsub_rn(sp.w, uv.w)));
                            ob = make_float4(__fmul_rn(g.x, __fsub_rn(1.f, av.x)), __fmul_rn(g.y, __fsub_rn(1.f, av.y)),
                                             __fmul_rn(g.z, __fsub_rn(1.f, av.z)), __fmul_rn(g.w, __fsub_rn(1.f, av.w)));
                        } else {
                            oa = make_float4(__fmul_rn(g.x, sp.x), __fmul_rn(g.y, sp.y), __fmul_rn(g.z, sp.z),
                                             __fmul_rn(g.w, sp.w));
                            ob = g;
                        }
                        if (pa != nullptr) st_cs(reinterpret_cast<float4*>(pa + (size_t)r * rowN), oa);
                        if (pb != nullptr) st_cs(reinterpret_cast<float4*>(pb + (size_t)r * rowN), ob);
                        if (k == 0 && r == 0 && p.ds0 != nullptr) {
                            const float4 a0 = *reinterpret_cast<const float4*>(sa + 4 * quad);
                            float* d0 = p.ds0 + (size_t)bi * p.N + n0 + 4 * quad;
                            d0[0] = __fmul_rn(a0.x, g.x);
                            d0[1] = __fmul_rn(a0.y, g.y);
                            d0[2] = __fmul_rn(a0.z, g.z);
                            d0[3] = __fmul_rn(a0.w, g.w);
                        }
                    }
                }
            }
        }
        fence_proxy_async_smem();                     // the edge writes precede the buffer's next TMA fill
        __syncthreads();                              // buffer `buf` free for the next prefetch
    }
}

}  // namespace

bool scan_backward_chunked_supported(const BwdArgs& x) {
    auto al16 = [](const void* q) { return q == nullptr || (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    return x.N % 4 == 0 && al16(x.a) && al16(x.u) && al16(x.s) && al16(x.gs) && al16(x.da) && al16(x.dbu);
}

int64_t scan_backward_chunked_ws_bytes(int B, int T, int N) {
    // A, B and C arrays at agg_index: per column, chunks in groups of four
    const int64_t nbcb = (int64_t)B * ((N + LB_NC - 1) / LB_NC);
    return 3 * nbcb * chunk_quads((T + LB_TC - 1) / LB_TC) * LB_NC * 4 * 4;
}

cudaError_t launch_scan_backward_chunked(const BwdArgs& x, bool gated, void* ws, SnDevStatus* st, uint64_t wait_ns,
                                         int sm_count, cudaStream_t stream) {
    CUtensorMap ma, mg, ms, mu;
    if (!make_scan_map(&ma, x.a, x.B, x.T, x.N, LB_NC, BT_AROWS) ||
        !make_scan_map(&mg, x.gs, x.B, x.T, x.N, LB_NC, LB_TC) ||
        !make_scan_map(&ms, x.s, x.B, x.T, x.N, LB_NC, LB_TC) ||
        !make_scan_map(&mu, gated ? x.u : x.gs, x.B, x.T, x.N, LB_NC, LB_TC))
        return cudaErrorInvalidValue;
    BwdPassParams p;
    p.B = x.B;
    p.T = x.T;
    p.N = x.N;
    p.ncb = (x.N + LB_NC - 1) / LB_NC;
    p.nbcb = x.B * p.ncb;
    p.nchunks = (x.T + LB_TC - 1) / LB_TC;
    p.ntiles = p.nbcb * p.nchunks;
    p.a = x.a;
    p.s0 = x.s0;
    p.gf = x.gf;
    p.da = x.da;
    p.dbu = x.dbu;
    p.ds0 = x.ds0;
    const int64_t tiles = p.ntiles;
    const int64_t arr = (int64_t)p.nbcb * chunk_quads(p.nchunks) * LB_NC * 4;   // floats per array
    p.dA = static_cast<float*>(ws);
    p.dB = p.dA + arr;
    p.dC = p.dB + arr;
    p.st = st;
    p.wait_ns = wait_ns;

    auto k_agg = gated ? bwd_pass<true, false> : bwd_pass<false, false>;
    auto k_out = gated ? bwd_pass<true, true> : bwd_pass<false, true>;
    const size_t agg_smem = gated ? bt_smem<true, false>() : bt_smem<false, false>();
    const size_t out_smem = gated ? bt_smem<true, true>() : bt_smem<false, true>();
    int occ_a = 0, occ_o = 0;
    cudaError_t e = occupancy_once((const void*)k_agg, LB_THREADS, agg_smem, &occ_a);
    if (e != cudaSuccess) return e;
    e = occupancy_once((const void*)k_out, LB_THREADS, out_smem, &occ_o);
    if (e != cudaSuccess) return e;
    e = set_smem_attr_once((const void*)scan_chain<true>, CHAIN_SMEM);
    if (e != cudaSuccess) return e;
    k_agg<<<(unsigned)std::min<int64_t>(tiles, (int64_t)occ_a * sm_count), LB_THREADS, agg_smem, stream>>>(ma, mg, ms,
                                                                                                          mu, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const ChainParams cp{p.N, p.ncb, p.nchunks, x.gf, p.dA, p.dB, p.dC, nullptr, st, wait_ns};
    scan_chain<true><<<(unsigned)p.nbcb, 32, CHAIN_SMEM, stream>>>(cp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_out<<<(unsigned)std::min<int64_t>(tiles, (int64_t)occ_o * sm_count), LB_THREADS, out_smem, stream>>>(ma, mg, ms,
                                                                                                          mu, p);
    return cudaGetLastError();
}

}  // namespace sn
