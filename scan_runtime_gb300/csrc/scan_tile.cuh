// scan_tile.cuh -- the chunk-tile machinery shared by the chunked scans
// (scan_lookback.cu: look-back and reduce-then-scan; scan_bwd_chunked.cu: the
// reverse scans): a tile is LB_TC time steps x LB_NC channels in shared memory,
// scanned by 256 threads as 32 segments of LB_SEG steps x 4 channels.
#pragma once

#include "scan_common.cuh"

namespace sn {
namespace {

constexpr int LB_THREADS = 256;                   // 8 warps
constexpr int LB_SEG = LB_TC / 32;                // steps per thread segment
constexpr uint32_t LB_TILE = LB_TC * LB_NC;       // floats per tensor per tile
constexpr uint32_t LB_TILE_BYTES = 2 * LB_TILE * 4;

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
// Local scan of one tile (LB_TC steps x LB_NC channels in shared memory, row
// major): every thread folds its LB_SEG steps of 4 channels, the warp scans
// its four segments, and the earlier warps' aggregates are folded in warp
// order.  Returns this thread's exclusive prefix (EA, EB); wA / wB keep the
// warps' aggregates.  Contains one __syncthreads.  REV scans the valid rows
// from the last to the first (position r is row rows - 1 - r), for the
// reverse recurrences of the backward pass.
template <bool GATED, bool REV = false>
__device__ __forceinline__ void tile_local_scan(const float* sa, const float* sb, int rows, float4 (*wA)[8],
                                                float4 (*wB)[8], float4& EA, float4& EB) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = lane & 7, sub = lane >> 3;
    const int seg = warp * 4 + sub;                 // 0..31, rows [seg*LB_SEG, (seg+1)*LB_SEG)
    // ---- phase 1: fold this thread's LB_SEG steps of its 4 channels
    float4 A = make_float4(1.f, 1.f, 1.f, 1.f), Bc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < LB_SEG; ++i) {
        const int r = seg * LB_SEG + i;             // position in scan order
        const int rr = REV ? max(rows - 1 - r, 0) : r;   // its row of the tile
        float4 av = *reinterpret_cast<const float4*>(sa + rr * LB_NC + 4 * quad);
        float4 bv = inj4<GATED>(av, *reinterpret_cast<const float4*>(sb + rr * LB_NC + 4 * quad));
        if (r >= rows) {                         // past the sequence: identity step
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
    EB = f4fma(eA, PB, eB);                     // exclusive prefix of this segment
    EA = f4mul(eA, PA);
}

// The whole tile's aggregate (A, B) for channel `lane` (warp 0): the warps'
// aggregates folded in warp order.
__device__ __forceinline__ void tile_aggregate(const float4 (*wA)[8], const float4 (*wB)[8], int lane, float& CA,
                                               float& CB) {
    CA = 1.f;
    CB = 0.f;
    const float* pA = reinterpret_cast<const float*>(&wA[0][0]) + lane;
    const float* pB = reinterpret_cast<const float*>(&wB[0][0]) + lane;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        CB = __fmaf_rn(pA[j * 32], CB, pB[j * 32]);
        CA = __fmul_rn(pA[j * 32], CA);
    }
}

// States of this thread's segment from its exclusive prefix and the tile's
// incoming carries (carry[]); the tile's last state is the outgoing carry
// itself (cfin[]), so a split at a multiple of LB_TC continues bit-exactly.
// `out` points at state (t0, n0) of the tile; rows of N floats.
template <bool GATED>
__device__ __forceinline__ void tile_outputs(const float* sa, const float* sb, int rows, const float* carry,
                                             const float* cfin, float4 EA, float4 EB, float* out, int N,
                                             bool active) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = lane & 7, sub = lane >> 3;
    const int seg = warp * 4 + sub;
    if (!active) return;
    const float4 cc = *reinterpret_cast<const float4*>(&carry[4 * quad]);
    float4 s = f4fma(EA, cc, EB);
    out += 4 * quad;
#pragma unroll
    for (int i = 0; i < LB_SEG; ++i) {
        const int r = seg * LB_SEG + i;
        if (r < rows) {
            const float4 av = *reinterpret_cast<const float4*>(sa + r * LB_NC + 4 * quad);
            const float4 bv = inj4<GATED>(av, *reinterpret_cast<const float4*>(sb + r * LB_NC + 4 * quad));
            s = f4fma(av, s, bv);
            if (r == rows - 1) s = *reinterpret_cast<const float4*>(&cfin[4 * quad]);
            st_cs(reinterpret_cast<float4*>(out + (size_t)r * N), s);
        }
    }
}

// Aggregates (A_k, B_k) and carries C_k of the chunked scans' passes, per
// column (channel tile) in groups of four chunks: group g of column col holds
// [channel][chunk 4g .. 4g + 3], 16 bytes per channel.  A column holds
// chunk_quads(nchunks) groups; the slots past the last chunk are padding.
__host__ __device__ __forceinline__ int chunk_quads(int nchunks) { return (nchunks + 3) >> 2; }
__host__ __device__ __forceinline__ size_t agg_index(size_t col, int nq, int k, int ch) {
    return ((col * nq + (k >> 2)) * LB_NC + ch) * 4 + (k & 3);
}

// Carries of the chunked scans, one warp per column (lane = channel):
//   forward (REV = false): C_k = fma(A_k, C_{k-1}, B_k), k = 0 .. nchunks - 1, C_{-1} = init;
//   reverse (REV = true):  C_k = fma(A_k, C_{k+1}, B_k), k = nchunks - 1 .. 0, C_{nchunks} = init;
// with (A_k, B_k) and C_k at agg_index.  The column's aggregates arrive in
// blocks of CHAIN_BLK chunks by bulk copies, CHAIN_STAGES blocks in flight.
// A lane reads four chunks of its channel with one 16-byte shared load per
// array and stores their four carries with one 16-byte global store; within
// a full block the groups are read into registers one batch ahead of the
// FMAs that consume them (two batches in turn, all offsets fixed), so the
// dependent chain is held up neither by load latency nor by a store per
// step.  The stores are global (st.global), so they cannot alias the
// shared-memory operands.
constexpr int CHAIN_BLK = 128;                                    // chunks per block (32 groups)
constexpr int CHAIN_STAGES = 4;
constexpr int CHAIN_QB = 4;                                       // groups per register batch
constexpr uint32_t CHAIN_BLK_FLOATS = CHAIN_BLK * LB_NC;          // one block of one array
constexpr size_t CHAIN_SMEM = (size_t)CHAIN_STAGES * 2 * CHAIN_BLK_FLOATS * 4 + CHAIN_STAGES * 8 + 16;

struct ChainParams {
    int N, ncb, nchunks;
    const float* init;   // (B, N) initial carry, NULL = zeros
    const float* dA;
    const float* dB;
    float* dC;
    float* cin0;         // [column][channel]: the initial carry as read, for the output pass (or NULL)
    SnDevStatus* st;
    uint64_t wait_ns;
};

// Four steps of the chain over one group, in visiting order; returns the
// group's carries in chunk order.
template <bool REV>
__device__ __forceinline__ float4 chain_group(float4 a, float4 b, float& c) {
    float4 r;
    if (!REV) {
        c = __fmaf_rn(a.x, c, b.x); r.x = c;
        c = __fmaf_rn(a.y, c, b.y); r.y = c;
        c = __fmaf_rn(a.z, c, b.z); r.z = c;
        c = __fmaf_rn(a.w, c, b.w); r.w = c;
    } else {
        c = __fmaf_rn(a.w, c, b.w); r.w = c;
        c = __fmaf_rn(a.z, c, b.z); r.z = c;
        c = __fmaf_rn(a.y, c, b.y); r.y = c;
        c = __fmaf_rn(a.x, c, b.x); r.x = c;
    }
    return r;
}

template <bool REV>
__global__ void __launch_bounds__(32) scan_chain(const ChainParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    float* bufs = reinterpret_cast<float*>(smem);                 // [stage][A | B][CHAIN_BLK / 4][LB_NC][4]
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + (size_t)CHAIN_STAGES * 2 * CHAIN_BLK_FLOATS * 4);
    const int lane = threadIdx.x;
    const size_t col = blockIdx.x;
    const int bi = (int)(col / p.ncb), cb = (int)(col % p.ncb);
    const int n = cb * LB_NC + lane;
    const int nq = chunk_quads(p.nchunks);
    const size_t colbase = agg_index(col, nq, 0, 0);
    const int nblk = (p.nchunks + CHAIN_BLK - 1) / CHAIN_BLK;
    // the j-th block visited (0-based) is block blk_of(j); stage j % CHAIN_STAGES
    auto blk_of = [&](int j) { return REV ? nblk - 1 - j : j; };
    auto issue = [&](int j) {   // lane 0
        const int blk = blk_of(j);
        const int c0 = blk * CHAIN_BLK, st = j % CHAIN_STAGES;
        const uint32_t bytes = (uint32_t)chunk_quads(min(CHAIN_BLK, p.nchunks - c0)) * LB_NC * 16;
        mbar_arrive_expect_tx(&bar[st], 2 * bytes);
        bulk_load(bufs + (size_t)st * 2 * CHAIN_BLK_FLOATS, p.dA + colbase + (size_t)c0 * LB_NC, bytes, &bar[st]);
        bulk_load(bufs + (size_t)st * 2 * CHAIN_BLK_FLOATS + CHAIN_BLK_FLOATS, p.dB + colbase + (size_t)c0 * LB_NC,
                  bytes, &bar[st]);
    };
    int issued = 0;
    if (lane == 0) {
        for (int st = 0; st < CHAIN_STAGES; ++st) mbar_init(&bar[st], 1);
        fence_mbar_init();
        for (; issued < min(nblk, CHAIN_STAGES); ++issued) issue(issued);
    }
    issued = __shfl_sync(0xffffffffu, issued, 0);
    float c = (p.init != nullptr && n < p.N) ? p.init[(size_t)bi * p.N + n] : 0.f;
    // The output pass takes its first chunk's carry from here, not from init:
    // init may be the buffer that pass writes its final states to.
    if (p.cin0 != nullptr) p.cin0[col * LB_NC + lane] = c;
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
        const int blk = blk_of(j);
        const int st = j % CHAIN_STAGES;
        ok = __all_sync(0xffffffffu, mbar_wait(&bar[st], (uint32_t)(j / CHAIN_STAGES) & 1, p.wait_ns));
        if (!ok) break;
        const float4* sA = reinterpret_cast<const float4*>(bufs + (size_t)st * 2 * CHAIN_BLK_FLOATS) + lane;
        const float4* sB = sA + CHAIN_BLK_FLOATS / 4;
        float4* dC = reinterpret_cast<float4*>(p.dC + colbase + (size_t)blk * CHAIN_BLK * LB_NC) + lane;
        const int cnt = min(CHAIN_BLK, p.nchunks - blk * CHAIN_BLK);
        // group q of the block (0-based, in visiting order) is group gx(q) of it
#define SN_CHAIN_GX(q) (REV ? CHAIN_BLK / 4 - 1 - (q) : (q))
        if (cnt == CHAIN_BLK) {
            // a full block: two register batches in turn, every offset fixed
            constexpr int NG = CHAIN_BLK / 4;
            float4 a0[CHAIN_QB], b0[CHAIN_QB], a1[CHAIN_QB], b1[CHAIN_QB];
#pragma unroll
            for (int u = 0; u < CHAIN_QB; ++u) {
                a0[u] = sA[SN_CHAIN_GX(u) * LB_NC];
                b0[u] = sB[SN_CHAIN_GX(u) * LB_NC];
            }
#pragma unroll
            for (int q0 = 0; q0 < NG; q0 += 2 * CHAIN_QB) {
#pragma unroll
                for (int u = 0; u < CHAIN_QB; ++u) {
                    a1[u] = sA[SN_CHAIN_GX(q0 + CHAIN_QB + u) * LB_NC];
                    b1[u] = sB[SN_CHAIN_GX(q0 + CHAIN_QB + u) * LB_NC];
                }
#pragma unroll
                for (int u = 0; u < CHAIN_QB; ++u)
                    __stcg(&dC[SN_CHAIN_GX(q0 + u) * LB_NC], chain_group<REV>(a0[u], b0[u], c));
                if (q0 + 2 * CHAIN_QB < NG) {
#pragma unroll
                    for (int u = 0; u < CHAIN_QB; ++u) {
                        a0[u] = sA[SN_CHAIN_GX(q0 + 2 * CHAIN_QB + u) * LB_NC];
                        b0[u] = sB[SN_CHAIN_GX(q0 + 2 * CHAIN_QB + u) * LB_NC];
                    }
                }
#pragma unroll
                for (int u = 0; u < CHAIN_QB; ++u)
                    __stcg(&dC[SN_CHAIN_GX(q0 + CHAIN_QB + u) * LB_NC], chain_group<REV>(a1[u], b1[u], c));
            }
        } else {
            // the partial block (the sequence's last): one chunk at a time
            const float* fA = bufs + (size_t)st * 2 * CHAIN_BLK_FLOATS;
            const float* fB = fA + CHAIN_BLK_FLOATS;
            float* fC = p.dC + colbase + (size_t)blk * CHAIN_BLK * LB_NC;
            for (int q = 0; q < cnt; ++q) {
                const int i = REV ? cnt - 1 - q : q;
                const int o = ((i >> 2) * LB_NC + lane) * 4 + (i & 3);
                c = __fmaf_rn(fA[o], c, fB[o]);
                __stcg(&fC[o], c);
            }
        }
#undef SN_CHAIN_GX
        __syncwarp();                                 // the stage is read
        if (lane == 0 && issued < nblk) issue(issued);
        if (issued < nblk) ++issued;
    }
    if (!ok && lane == 0) {
        record_error(p.st, SN_E_TIMEOUT, (SN_K_SCAN_LOOKBACK << 16) | 4);
        // let this warp's loads still in flight land: the last CHAIN_STAGES issued
        for (int j = max(0, issued - CHAIN_STAGES); j < issued; ++j)
            (void)mbar_wait(&bar[j % CHAIN_STAGES], (uint32_t)(j / CHAIN_STAGES) & 1, p.wait_ns);
    }
}

}  // namespace
}  // namespace sn
