// scan_fused.cu -- the chunked scans of tier 1 for few channels and long T in
// two launches ("SunnyNet 工程化实录" §2.1 forms; §4 bit-exact continuation).
//
// The reduce-then-scan path (scan_lookback.cu) runs three launches: every
// tile's aggregate, a carry chain per column, then every tile's states from
// its carry.  The chain is a serial fold over all chunks of a column (one
// dependent FMA per chunk and channel), so the GPU idles for its length
// between the two passes.  Here the chain runs inside the state pass:
//   1. the aggregate pass (scan_lookback.cu), last tile first, writes every
//      tile's (A_k, B_k);
//   2. one cooperative launch: CTA col < columns is the chain of column col
//      (warp 0, lane = channel), folding C_k = fma(A_k, C_{k-1}, B_k) over the
//      chunks in order with the aggregates staged by bulk copies (FU_CSTAGES
//      blocks of FU_CB chunks in flight) into shared memory, while its warp 1
//      publishes each carry as a 64-bit word that holds the launch's tag
//      beside the carry's bits; the other
//      CTAs compute the states of the tiles first to last (the first ones
//      are the last the aggregate pass read, still in L2), each waiting for
//      the carry word of the chunk before its own.
// A single-copy-atomic 64-bit access reads or writes tag and value together,
// so the chain needs no fence and a state tile no flag: it polls its own
// carry words.  Sharing its SM with state CTAs, a chain folds a chunk in about
// 30 cycles (10 alone), so a column of chunks takes about as long as the
// state tiles of two columns: the path pays where a launch has two columns or
// more, and a single column keeps the reduce-then-scan launches.
// Every operation is the reduce-then-scan path's in the same order (tile local
// scan, aggregate, fold, outputs), so all chunked paths give the same bits.
// The chain waits only on its bulk copies and the state tiles only on the
// chain, every CTA is resident (cooperative launch), and every wait is bounded
// (SN_OPT_WAIT_LIMIT_US): a CTA that gives up records SN_E_TIMEOUT and tags
// the launch, and the others stop waiting at once.  The tags carry the launch
// epoch (kept in device memory, shared with the look-back kernel), so no call
// needs a memset while the geometry stays the same.
#include <algorithm>

#include "scan_tile.cuh"

namespace sn {
namespace {

constexpr int FU_CB = 64;                          // chunks per block of a chain's ring
constexpr int FU_CSTAGES = 4;                      // blocks in flight in a chain CTA
constexpr int FU_STAGES = 2;                       // tiles in flight in a state CTA (2 CTAs per SM: the
                                                   // chain keeps its registers; 3 per SM measured slower)
constexpr uint32_t FU_CARRY = 3u;                  // tag state of a carry word
constexpr uint32_t FU_EPOCH_WRAP = 1u << 29;
constexpr uint32_t FU_CBLK_FLOATS = FU_CB * LB_NC;  // one block of one array (agg_index layout)
constexpr int FU_CQ = 4;                           // carry blocks between the folding and the storing warp
constexpr size_t FU_RING = FU_STAGES * (size_t)LB_TILE_BYTES;
static_assert((size_t)FU_CSTAGES * 2 * FU_CBLK_FLOATS * 4 <= FU_RING, "the chain ring reuses the tile ring");
constexpr size_t FU_CBUF = (size_t)FU_CQ * FU_CBLK_FLOATS * 4;   // the folded carries, [block][group][lane][4]
constexpr int FU_NBAR = FU_STAGES + FU_CSTAGES + 2 * FU_CQ;
constexpr size_t FU_SMEM = FU_RING + FU_CBUF + FU_NBAR * 8 + 16;

struct FusedParams {
    int B, T, N, ncb, nbcb, nchunks, ntiles;
    const float* s0;
    float* s_final;
    float* s_out;
    const float* dA;              // aggregates at agg_index (per column, chunks in groups of four)
    const float* dB;
    unsigned long long* cw;       // carries at agg_index: (tag | FU_CARRY) << 32 | bits of C_k
    unsigned long long* cw0;      // [col][channel]: the same for the initial carry
    SnDevStatus* st;              // error word, abort tag and the launch epoch
    uint64_t wait_ns;
};

__device__ __forceinline__ void st_relaxed_gpu_v2u64(unsigned long long* p, unsigned long long a,
                                                     unsigned long long b) {
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}

template <bool GATED>
__global__ void __launch_bounds__(LB_THREADS, 2)
scan_fused(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b, const FusedParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    // [FU_STAGES] tiles | [FU_CSTAGES] chain ring | [FU_CQ] carries folded | [FU_CQ] carries stored
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + FU_RING + FU_CBUF);
    __shared__ float4 wA[8][8], wB[8][8];
    __shared__ float carry[LB_NC], cfin[LB_NC];
    __shared__ uint32_t s_epoch;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = lane & 7;
    const int nq = chunk_quads(p.nchunks);

    if (tid == 0) {
        for (int s = 0; s < FU_NBAR; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
        const uint32_t last = *reinterpret_cast<volatile const uint32_t*>(&p.st->lb_epoch);
        s_epoch = last + 1 >= FU_EPOCH_WRAP ? 1u : last + 1;
    }
    __syncthreads();
    const uint32_t epoch = s_epoch;
    const uint32_t tag = epoch << 2;
    const unsigned long long hi = (unsigned long long)(tag | FU_CARRY) << 32;
    auto aborted = [&]() { return *reinterpret_cast<volatile const uint32_t*>(&p.st->abort_tag) == tag; };
    auto give_up = [&](int site) {
        record_error(p.st, SN_E_TIMEOUT, (SN_K_SCAN_LOOKBACK << 16) | site);
        atomicExch(&p.st->abort_tag, tag);
    };
    // the launch's last CTA to finish records its epoch for the next launch
    auto finish = [&]() {
        __threadfence();
        if (atomicAdd(&p.st->lb_done, 1u) == gridDim.x - 1) {
            p.st->lb_done = 0;
            p.st->lb_epoch = epoch;
            __threadfence();
        }
    };

    if ((int)blockIdx.x < p.nbcb) {
        // ------------------------------------------------ chain CTA of column blockIdx.x
        // Warp 0 folds the carries into shared memory (FU_CQ blocks deep) and
        // warp 1 publishes them as tagged words, so the dependent FMA chain
        // never waits behind global stores.
        if (warp > 1) return;
        const size_t col = blockIdx.x;
        const int bi = (int)(col / p.ncb), cb = (int)(col % p.ncb);
        const int n = cb * LB_NC + lane;
        float* ring = reinterpret_cast<float*>(smem);             // [stage][A | B][FU_CBLK_FLOATS]
        float* cbuf = reinterpret_cast<float*>(smem + FU_RING);   // [FU_CQ][group][lane][4] carries
        uint64_t* cbar = bar + FU_STAGES;
        uint64_t* cfull = cbar + FU_CSTAGES;                      // [FU_CQ] a block is folded
        uint64_t* cfree = cfull + FU_CQ;                          // [FU_CQ] a block is published
        const size_t colbase = agg_index(col, nq, 0, 0);
        const int nblk = (p.nchunks + FU_CB - 1) / FU_CB;
        // bounded wait that also ends when another CTA or warp gave up
        auto wait_or_abort = [&](uint64_t* b, uint32_t parity) {
            if (mbar_try_wait(b, parity)) return true;
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(b, parity))
                if (global_ns() - t0 > p.wait_ns || aborted()) return false;
            return true;
        };
        if (warp == 1) {
            unsigned long long* cwc = p.cw + colbase;
            bool ok = true;
            for (int j = 0; j < nblk; ++j) {
                const int q = j % FU_CQ;
                ok = __all_sync(0xffffffffu, wait_or_abort(&cfull[q], (uint32_t)(j / FU_CQ) & 1u));
                if (!ok) break;
                const int k0 = j * FU_CB, cnt = min(FU_CB, p.nchunks - k0);
                const float4* src = reinterpret_cast<const float4*>(cbuf + (size_t)q * FU_CBLK_FLOATS) + lane;
                for (int g = 0; g < (cnt + 3) >> 2; ++g) {   // four carries of the lane's channel per group
                    const float4 r = src[g * LB_NC];
                    unsigned long long* d = cwc + ((size_t)((k0 >> 2) + g) * LB_NC + lane) * 4;
                    st_relaxed_gpu_v2u64(d, hi | __float_as_uint(r.x), hi | __float_as_uint(r.y));
                    st_relaxed_gpu_v2u64(d + 2, hi | __float_as_uint(r.z), hi | __float_as_uint(r.w));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&cfree[q]);
            }
            if (!ok && lane == 0) give_up(8);
            named_bar_sync(1, 64);                        // the CTA finishes with the folding warp
            return;
        }
        auto issue = [&](int j) {   // lane 0: block j's aggregates into stage j % FU_CSTAGES
            const int k0 = j * FU_CB, st = j % FU_CSTAGES;
            const uint32_t bytes = (uint32_t)chunk_quads(min(FU_CB, p.nchunks - k0)) * LB_NC * 16;
            mbar_arrive_expect_tx(&cbar[st], 2 * bytes);
            bulk_load(ring + (size_t)st * 2 * FU_CBLK_FLOATS, p.dA + colbase + (size_t)k0 * LB_NC, bytes, &cbar[st]);
            bulk_load(ring + (size_t)st * 2 * FU_CBLK_FLOATS + FU_CBLK_FLOATS, p.dB + colbase + (size_t)k0 * LB_NC,
                      bytes, &cbar[st]);
        };
        int issued = 0;
        if (lane == 0)
            for (; issued < min(nblk, FU_CSTAGES); ++issued) issue(issued);
        issued = __shfl_sync(0xffffffffu, issued, 0);
        // the first chunk's carry is published from here, not read from s0 by
        // the state tiles: a call may write its final states over s0
        float c = (p.s0 != nullptr && n < p.N) ? p.s0[(size_t)bi * p.N + n] : 0.f;
        st_relaxed_gpu_u64(p.cw0 + col * LB_NC + lane, hi | __float_as_uint(c));
        bool ok = true;
        for (int j = 0; j < nblk; ++j) {
            const int st = j % FU_CSTAGES, q = j % FU_CQ;
            ok = __all_sync(0xffffffffu, mbar_wait(&cbar[st], (uint32_t)(j / FU_CSTAGES) & 1, p.wait_ns));
            // the carry buffer q is free once warp 1 has published block j - FU_CQ
            if (ok && j >= FU_CQ)
                ok = __all_sync(0xffffffffu, wait_or_abort(&cfree[q], (uint32_t)(j / FU_CQ - 1) & 1u));
            if (!ok) break;
            const int k0 = j * FU_CB, cnt = min(FU_CB, p.nchunks - k0);
            const float4* sA = reinterpret_cast<const float4*>(ring + (size_t)st * 2 * FU_CBLK_FLOATS) + lane;
            const float4* sB = sA + FU_CBLK_FLOATS / 4;
            float4* dst = reinterpret_cast<float4*>(cbuf + (size_t)q * FU_CBLK_FLOATS) + lane;
            if (cnt == FU_CB) {
                // a full block: the groups are read a batch of four ahead of the
                // FMAs that consume them, so the dependent chain waits on no load
                constexpr int NG = FU_CB / 4, QB = 4;
                float4 a0[QB], b0[QB], a1[QB], b1[QB];
#pragma unroll
                for (int u = 0; u < QB; ++u) {
                    a0[u] = sA[u * LB_NC];
                    b0[u] = sB[u * LB_NC];
                }
#pragma unroll
                for (int g = 0; g < NG; g += 2 * QB) {
#pragma unroll
                    for (int u = 0; u < QB; ++u) {
                        a1[u] = sA[(g + QB + u) * LB_NC];
                        b1[u] = sB[(g + QB + u) * LB_NC];
                    }
#pragma unroll
                    for (int u = 0; u < QB; ++u) {
                        float4 r;
                        c = __fmaf_rn(a0[u].x, c, b0[u].x); r.x = c;
                        c = __fmaf_rn(a0[u].y, c, b0[u].y); r.y = c;
                        c = __fmaf_rn(a0[u].z, c, b0[u].z); r.z = c;
                        c = __fmaf_rn(a0[u].w, c, b0[u].w); r.w = c;
                        dst[(g + u) * LB_NC] = r;
                    }
                    if (g + 2 * QB < NG) {
#pragma unroll
                        for (int u = 0; u < QB; ++u) {
                            a0[u] = sA[(g + 2 * QB + u) * LB_NC];
                            b0[u] = sB[(g + 2 * QB + u) * LB_NC];
                        }
                    }
#pragma unroll
                    for (int u = 0; u < QB; ++u) {
                        float4 r;
                        c = __fmaf_rn(a1[u].x, c, b1[u].x); r.x = c;
                        c = __fmaf_rn(a1[u].y, c, b1[u].y); r.y = c;
                        c = __fmaf_rn(a1[u].z, c, b1[u].z); r.z = c;
                        c = __fmaf_rn(a1[u].w, c, b1[u].w); r.w = c;
                        dst[(g + QB + u) * LB_NC] = r;
                    }
                }
            } else {
                // the sequence's last, partial block: one chunk at a time
                const float* fA = ring + (size_t)st * 2 * FU_CBLK_FLOATS;
                const float* fB = fA + FU_CBLK_FLOATS;
                float* fC = cbuf + (size_t)q * FU_CBLK_FLOATS;
                for (int i = 0; i < cnt; ++i) {
                    const int o = ((i >> 2) * LB_NC + lane) * 4 + (i & 3);
                    c = __fmaf_rn(fA[o], c, fB[o]);
                    fC[o] = c;
                }
            }
            __syncwarp();                                 // the stage is read, the carries are written
            if (lane == 0) mbar_arrive(&cfull[q]);        // (release: warp 1 reads them after its wait)
            if (issued < nblk) {
                if (lane == 0) {
                    fence_proxy_async_smem();             // those reads before the copy's writes
                    issue(issued);
                }
                ++issued;
            }
        }
        if (!ok && lane == 0) {
            give_up(5);
            // the bulk copies still in flight must land before the CTA leaves
            for (int j = max(0, issued - FU_CSTAGES); j < issued; ++j)
                (void)mbar_wait(&cbar[j % FU_CSTAGES], (uint32_t)(j / FU_CSTAGES) & 1, p.wait_ns);
        }
        named_bar_sync(1, 64);                            // and with the publishing warp
        if (lane == 0) finish();
        return;
    }

    // ---------------------------------------------------- state CTAs
    const int w = (int)blockIdx.x - p.nbcb, nw = (int)gridDim.x - p.nbcb;
    const int ni = w < p.ntiles ? (p.ntiles - 1 - w) / nw + 1 : 0;   // tiles w, w + nw, ... (chunk order)
    float* bufs = reinterpret_cast<float*>(smem);
    auto coords = [&](int ti, int& k, int& bi, int& cb) {
        k = ti / p.nbcb;
        const int r = ti - k * p.nbcb;
        bi = r / p.ncb;
        cb = r - bi * p.ncb;
    };
    auto issue = [&](int i, int buf) {
        int k, bi, cb;
        coords(w + i * nw, k, bi, cb);
        mbar_arrive_expect_tx(&bar[buf], LB_TILE_BYTES);
        float* dst = bufs + buf * 2 * LB_TILE;
        tma_load_3d(dst, &map_a, &bar[buf], cb * LB_NC, k * LB_TC, bi);
        tma_load_3d(dst + LB_TILE, &map_b, &bar[buf], cb * LB_NC, k * LB_TC, bi);
    };
    if (tid == 0)
        for (int s = 0; s < FU_STAGES - 1 && s < ni; ++s) issue(s, s);
    for (int i = 0; i < ni; ++i) {
        const int buf = i % FU_STAGES;
        if (tid == 0 && i + FU_STAGES - 1 < ni) issue(i + FU_STAGES - 1, (i + FU_STAGES - 1) % FU_STAGES);
        int k, bi, cb;
        coords(w + i * nw, k, bi, cb);
        const int t0 = k * LB_TC, n0 = cb * LB_NC;
        const int rows = min(LB_TC, p.T - t0);
        if (!__syncthreads_and(mbar_wait(&bar[buf], (uint32_t)(i / FU_STAGES) & 1, p.wait_ns))) {
            if (tid == 0) {
                give_up(6);
                for (int j = i; j < min(ni, i + FU_STAGES); ++j)
                    (void)mbar_wait(&bar[j % FU_STAGES], (uint32_t)(j / FU_STAGES) & 1, p.wait_ns);
            }
            break;
        }
        const float* sa = bufs + buf * 2 * LB_TILE;
        const float* sb = sa + LB_TILE;
        float4 EA, EB;
        tile_local_scan<GATED>(sa, sb, rows, wA, wB, EA, EB);
        const size_t col = (size_t)bi * p.ncb + cb;
        if (warp == 0) {
            float CA, CB;
            tile_aggregate(wA, wB, lane, CA, CB);
            // the incoming carry: chunk k - 1's word (the initial carry's for k = 0)
            const unsigned long long* src =
                k == 0 ? p.cw0 + col * LB_NC + lane : p.cw + agg_index(col, nq, k - 1, lane);
            unsigned long long v = ld_relaxed_gpu_u64(src);
            bool got = true;
            if ((v & 0xffffffff00000000ull) != hi) {
                const uint64_t t0w = global_ns();
                do {
                    if (global_ns() - t0w > p.wait_ns || aborted()) {
                        got = false;
                        break;
                    }
                    // back off: a chain CTA may share this SM, and its warp
                    // folds fastest with the issue slots to itself
                    __nanosleep(200);
                    v = ld_relaxed_gpu_u64(src);
                } while ((v & 0xffffffff00000000ull) != hi);
            }
            got = __all_sync(0xffffffffu, got);
            if (!got && lane == 0) give_up(7);
            const float cin = got ? __uint_as_float((uint32_t)v) : 0.f;
            const float Ck = __fmaf_rn(CA, cin, CB);
            carry[lane] = cin;
            cfin[lane] = Ck;
            const int n = n0 + lane;
            if (k == p.nchunks - 1 && p.s_final != nullptr && n < p.N) p.s_final[(size_t)bi * p.N + n] = Ck;
        }
        __syncthreads();
        tile_outputs<GATED>(sa, sb, rows, carry, cfin, EA, EB, p.s_out + ((size_t)bi * p.T + t0) * p.N + n0, p.N,
                            p.s_out != nullptr && n0 + 4 * quad < p.N);
        __syncthreads();                              // buffer `buf` free for the next load
    }
    if (tid == 0) finish();
}

}  // namespace

// The fused path runs for eight chunks or more (shorter scans take the
// reduce-then-scan launches, which give the same bits).
bool scan_fused_applies(int T) { return (T + LB_TC - 1) / LB_TC >= 8; }

// Workspace of the fused path: the A and B arrays of the aggregate pass, the
// tagged carry words (one per chunk and channel, same layout), the tagged
// initial carries.  Returns the bytes it needs.
int64_t scan_fused_ws_bytes(int B, int T, int N) {
    const int64_t ncb = (N + LB_NC - 1) / LB_NC, nbcb = (int64_t)B * ncb;
    const int64_t nch = (T + LB_TC - 1) / LB_TC;
    const int64_t arr = nbcb * chunk_quads((int)nch) * LB_NC * 4 * 4;   // bytes per f32 array
    return 4 * arr + nbcb * LB_NC * 8;
}

// the tagged words' bytes [a, a + b), which a change of geometry clears
void scan_fused_tag_area(int B, int T, int N, int64_t* a, int64_t* b) {
    const int64_t ncb = (N + LB_NC - 1) / LB_NC, nbcb = (int64_t)B * ncb;
    const int64_t nch = (T + LB_TC - 1) / LB_TC;
    const int64_t arr = nbcb * chunk_quads((int)nch) * LB_NC * 4 * 4;
    *a = 2 * arr;
    *b = 2 * arr + nbcb * LB_NC * 8;
}

cudaError_t launch_scan_fused(const ScanArgs& x, bool gated, void* ws, SnDevStatus* st, uint64_t wait_ns,
                              int sm_count, cudaStream_t stream) {
    CUtensorMap ma, mb;
    if (!make_scan_map(&ma, x.a, x.B, x.T, x.N, LB_NC, LB_TC) ||
        !make_scan_map(&mb, x.b, x.B, x.T, x.N, LB_NC, LB_TC))
        return cudaErrorInvalidValue;
    FusedParams p;
    p.B = x.B;
    p.T = x.T;
    p.N = x.N;
    p.ncb = (x.N + LB_NC - 1) / LB_NC;
    p.nbcb = x.B * p.ncb;
    p.nchunks = (x.T + LB_TC - 1) / LB_TC;
    p.ntiles = p.nbcb * p.nchunks;
    p.s0 = x.s0;
    p.s_final = x.s_final;
    p.s_out = x.s_out;
    const int64_t arr = (int64_t)p.nbcb * chunk_quads(p.nchunks) * LB_NC * 4;   // floats per array
    float* dA = static_cast<float*>(ws);
    float* dB = dA + arr;
    p.dA = dA;
    p.dB = dB;
    p.cw = reinterpret_cast<unsigned long long*>(dB + arr);
    p.cw0 = p.cw + arr;
    p.st = st;
    p.wait_ns = wait_ns;

    auto kern = gated ? scan_fused<true> : scan_fused<false>;
    int occ = 0;
    cudaError_t e = occupancy_once((const void*)kern, LB_THREADS, FU_SMEM, &occ);
    if (e != cudaSuccess) return e;
    // every column's chain CTA plus the state CTAs, all resident (cooperative launch)
    const int64_t resident = (int64_t)occ * sm_count;
    if (resident <= p.nbcb) return cudaErrorInvalidConfiguration;
    e = launch_scan_aggregates(x, gated, dA, dB, st, wait_ns, sm_count, stream);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<int64_t>(resident, p.nbcb + (int64_t)p.ntiles);
    void* args[] = {(void*)&ma, (void*)&mb, (void*)&p};
    e = cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(LB_THREADS), args, FU_SMEM, stream);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace sn
