// scan_fused.cu -- the chunked scans of tier 1 for few channels and long T in
// one launch ("SunnyNet 工程化实录" §2.1 forms; §4 bit-exact continuation).
//
// The reduce-then-scan path (scan_lookback.cu) runs three launches: every
// tile's aggregate, then a carry chain per column, then every tile's states
// from its carry.  The chain is a serial fold over all chunks of a column, so
// between the two passes the GPU waits for it, and the output pass starts on
// tiles long gone from L2.  This kernel runs the same three steps at once:
//   * worker CTAs first compute the aggregates of their tiles (chunk-major,
//     like the aggregate pass) and raise a tagged flag per tile;
//   * one chain CTA per column (blockIdx.x < columns, warp 0, lane = channel)
//     folds C_k = fma(A_k, C_{k-1}, B_k) over the chunks in order, a block of
//     FU_CB chunks at a time as soon as the block's flags are up (the
//     aggregates arrive by bulk copies, up to FU_CSTAGES blocks in flight), and
//     raises a tagged flag per block once its carries are written;
//   * after their last aggregate the workers compute the states of their
//     tiles in reverse order (the tiles they read last are still in L2), each
//     waiting for the flag of the block that holds its incoming carry.
// Every operation is the reduce-then-scan path's in the same order (the tile
// local scan, the aggregate, the fold, the outputs), so all chunked paths
// give the same bits.  Workers never wait during their aggregates, and the
// chain waits only on aggregates, so the waits always end; the grid is
// launched cooperatively (every CTA resident), and every wait is bounded
// (SN_OPT_WAIT_LIMIT_US): a CTA that gives up records SN_E_TIMEOUT and tags
// the launch, and the others stop waiting at once.  Flags carry the launch
// epoch (kept in device memory, shared with the look-back kernel), so no call
// needs a memset while the geometry stays the same.
#include <algorithm>

#include "scan_tile.cuh"

namespace sn {
namespace {

constexpr int FU_CB = 64;                          // chunks per carry block
constexpr int FU_CSTAGES = 4;                      // carry blocks in flight in a chain CTA
constexpr int FU_STAGES = 2;                       // tiles in flight in a worker CTA
constexpr uint32_t FU_AGG = 1u;                    // tile flag state: aggregate written
constexpr uint32_t FU_READY = 2u;                  // block flag state: carries written
constexpr uint32_t FU_EPOCH_WRAP = 1u << 29;
constexpr uint32_t FU_CBLK_FLOATS = FU_CB * LB_NC;  // one block of one array (agg_index layout)
constexpr size_t FU_RING = FU_STAGES * (size_t)LB_TILE_BYTES;
static_assert((size_t)FU_CSTAGES * 2 * FU_CBLK_FLOATS * 4 <= FU_RING, "the chain ring reuses the tile ring");
constexpr size_t FU_SMEM = FU_RING + (FU_STAGES + FU_CSTAGES) * 8 + 16;

struct FusedParams {
    int B, T, N, ncb, nbcb, nchunks, ntiles, nblk;
    const float* s0;
    float* s_final;
    float* s_out;
    uint32_t* tflag;     // per tile ti = k * nbcb + col: tag | FU_AGG
    uint32_t* bflag;     // per (col, carry block): tag | FU_READY
    float* dA;           // aggregates and carries at agg_index (per column, chunks in groups of four)
    float* dB;
    float* dC;
    float* cin0;         // [col][channel]: the initial carry as the chain read it
    SnDevStatus* st;     // error word, abort tag and the launch epoch
    uint64_t wait_ns;
};

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

template <bool GATED>
__global__ void __launch_bounds__(LB_THREADS, 2)
scan_fused(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b, const FusedParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + FU_RING);   // [FU_STAGES] tiles | [FU_CSTAGES] chain
    __shared__ float4 wA[8][8], wB[8][8];
    __shared__ float carry[LB_NC], cfin[LB_NC];
    __shared__ uint32_t s_epoch;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = lane & 7;
    const int nq = chunk_quads(p.nchunks);

    if (tid == 0) {
        for (int s = 0; s < FU_STAGES + FU_CSTAGES; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
        const uint32_t last = *reinterpret_cast<volatile const uint32_t*>(&p.st->lb_epoch);
        s_epoch = last + 1 >= FU_EPOCH_WRAP ? 1u : last + 1;
    }
    __syncthreads();
    const uint32_t epoch = s_epoch;
    const uint32_t tag = epoch << 2;
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
        if (warp != 0) return;
        const size_t col = blockIdx.x;
        const int bi = (int)(col / p.ncb), cb = (int)(col % p.ncb);
        const int n = cb * LB_NC + lane;
        float* ring = reinterpret_cast<float*>(smem);             // [stage][A | B][FU_CBLK_FLOATS]
        uint64_t* cbar = bar + FU_STAGES;
        const size_t colbase = agg_index(col, nq, 0, 0);
        float c = (p.s0 != nullptr && n < p.N) ? p.s0[(size_t)bi * p.N + n] : 0.f;
        // the first chunk's carry comes from here, not from s0: a call may
        // write its final states over s0
        p.cin0[col * LB_NC + lane] = c;
        // block j's aggregates are all written: every tile flag of it carries this launch's tag
        auto ready = [&](int j) {
            const int k0 = j * FU_CB, cnt = min(FU_CB, p.nchunks - k0);
            bool ok = true;
            for (int i = lane; i < cnt; i += 32)
                ok = ok && ld_acquire_gpu(p.tflag + (size_t)(k0 + i) * p.nbcb + col) == (tag | FU_AGG);
            return __all_sync(0xffffffffu, ok);
        };
        auto issue = [&](int j) {   // after `ready`: the aggregates of block j into stage j % FU_CSTAGES
            __syncwarp();                 // every lane's acquire before lane 0's copies
            fence_proxy_async_global();   // the flags' acquire before the bulk copies' reads
            if (lane == 0) {
                const int k0 = j * FU_CB, st = j % FU_CSTAGES;
                const uint32_t bytes = (uint32_t)chunk_quads(min(FU_CB, p.nchunks - k0)) * LB_NC * 16;
                mbar_arrive_expect_tx(&cbar[st], 2 * bytes);
                bulk_load(ring + (size_t)st * 2 * FU_CBLK_FLOATS, p.dA + colbase + (size_t)k0 * LB_NC, bytes, &cbar[st]);
                bulk_load(ring + (size_t)st * 2 * FU_CBLK_FLOATS + FU_CBLK_FLOATS, p.dB + colbase + (size_t)k0 * LB_NC,
                          bytes, &cbar[st]);
            }
        };
        int issued = 0;
        bool ok = true;
        for (int j = 0; j < p.nblk && ok; ++j) {
            // blocks j .. j + FU_CSTAGES - 1 go out as their aggregates appear; block j must
            const int limit = min(p.nblk, j + FU_CSTAGES);
            const uint64_t t0 = global_ns();
            while (issued < limit) {
                if (ready(issued)) {
                    issue(issued);
                    ++issued;
                    continue;
                }
                if (issued > j) break;                                 // something to fold meanwhile
                if (global_ns() - t0 > p.wait_ns || aborted()) {
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
            const int st = j % FU_CSTAGES;
            ok = __all_sync(0xffffffffu, mbar_wait(&cbar[st], (uint32_t)(j / FU_CSTAGES) & 1, p.wait_ns));
            if (!ok) break;
            const int k0 = j * FU_CB, cnt = min(FU_CB, p.nchunks - k0);
            const float* fA = ring + (size_t)st * 2 * FU_CBLK_FLOATS;
            const float* fB = fA + FU_CBLK_FLOATS;
            float* fC = p.dC + colbase + (size_t)k0 * LB_NC;
            for (int g = 0; g < (cnt >> 2); ++g) {                  // whole groups of four chunks
                const float4 a4 = reinterpret_cast<const float4*>(fA)[g * LB_NC + lane];
                const float4 b4 = reinterpret_cast<const float4*>(fB)[g * LB_NC + lane];
                float4 r;
                c = __fmaf_rn(a4.x, c, b4.x); r.x = c;
                c = __fmaf_rn(a4.y, c, b4.y); r.y = c;
                c = __fmaf_rn(a4.z, c, b4.z); r.z = c;
                c = __fmaf_rn(a4.w, c, b4.w); r.w = c;
                __stcg(reinterpret_cast<float4*>(fC) + g * LB_NC + lane, r);
            }
            for (int i = cnt & ~3; i < cnt; ++i) {                  // the sequence's last, partial group
                const int o = ((i >> 2) * LB_NC + lane) * 4 + (i & 3);
                c = __fmaf_rn(fA[o], c, fB[o]);
                __stcg(&fC[o], c);
            }
            __syncwarp();
            if (lane == 0) {
                __threadfence();
                st_release_gpu(p.bflag + col * p.nblk + j, tag | FU_READY);
            }
        }
        if (!ok && lane == 0) {
            give_up(5);
            // the bulk copies still in flight must land before the CTA leaves
            for (int j = max(0, issued - FU_CSTAGES); j < issued; ++j)
                (void)mbar_wait(&cbar[j % FU_CSTAGES], (uint32_t)(j / FU_CSTAGES) & 1, p.wait_ns);
        }
        __syncwarp();
        if (lane == 0) finish();
        return;
    }

    // ---------------------------------------------------- worker CTAs
    const int w = (int)blockIdx.x - p.nbcb, nw = (int)gridDim.x - p.nbcb;
    const int ni = w < p.ntiles ? (p.ntiles - 1 - w) / nw + 1 : 0;   // tiles w, w + nw, ...
    float* bufs = reinterpret_cast<float*>(smem);
    // load idx < ni: aggregate of tile w + idx nw; idx >= ni: states of the tiles in reverse
    auto tile_of = [&](int idx) { return w + (idx < ni ? idx : 2 * ni - 1 - idx) * nw; };
    auto coords = [&](int ti, int& k, int& bi, int& cb) {
        k = ti / p.nbcb;
        const int r = ti - k * p.nbcb;
        bi = r / p.ncb;
        cb = r - bi * p.ncb;
    };
    auto issue = [&](int idx, int buf) {
        int k, bi, cb;
        coords(tile_of(idx), k, bi, cb);
        mbar_arrive_expect_tx(&bar[buf], LB_TILE_BYTES);
        float* dst = bufs + buf * 2 * LB_TILE;
        tma_load_3d(dst, &map_a, &bar[buf], cb * LB_NC, k * LB_TC, bi);
        tma_load_3d(dst + LB_TILE, &map_b, &bar[buf], cb * LB_NC, k * LB_TC, bi);
    };
    const int nload = 2 * ni;
    if (tid == 0)
        for (int s = 0; s < FU_STAGES - 1 && s < nload; ++s) issue(s, s);
    bool ok = true;
    for (int idx = 0; idx < nload; ++idx) {
        const int buf = idx % FU_STAGES;
        if (tid == 0 && idx + FU_STAGES - 1 < nload) issue(idx + FU_STAGES - 1, (idx + FU_STAGES - 1) % FU_STAGES);
        const int ti = tile_of(idx);
        int k, bi, cb;
        coords(ti, k, bi, cb);
        const int t0 = k * LB_TC, n0 = cb * LB_NC;
        const int rows = min(LB_TC, p.T - t0);
        if (!__syncthreads_and(mbar_wait(&bar[buf], (uint32_t)(idx / FU_STAGES) & 1, p.wait_ns))) {
            if (tid == 0) {
                give_up(6);
                for (int j = idx; j < min(nload, idx + FU_STAGES); ++j)
                    (void)mbar_wait(&bar[j % FU_STAGES], (uint32_t)(j / FU_STAGES) & 1, p.wait_ns);
            }
            ok = false;
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
            if (idx < ni) {
                const size_t me = agg_index(col, nq, k, lane);
                p.dA[me] = CA;
                p.dB[me] = CB;
                __syncwarp();
                if (lane == 0) st_release_gpu(p.tflag + ti, tag | FU_AGG);
            } else {
                // the incoming carry: chunk k - 1's, in carry block (k - 1) / FU_CB
                const int kb = k == 0 ? 0 : (k - 1) / FU_CB;
                const uint32_t* bf = p.bflag + col * p.nblk + kb;
                const uint64_t t0w = global_ns();
                bool got = true;
                while (ld_acquire_gpu(bf) != (tag | FU_READY)) {
                    if (global_ns() - t0w > p.wait_ns || aborted()) {
                        got = false;
                        break;
                    }
                }
                got = __all_sync(0xffffffffu, got);
                if (!got && lane == 0) give_up(7);
                const float cin = !got ? 0.f
                                  : k == 0 ? __ldcg(p.cin0 + col * LB_NC + lane)
                                           : __ldcg(p.dC + agg_index(col, nq, k - 1, lane));
                const float Ck = __fmaf_rn(CA, cin, CB);
                carry[lane] = cin;
                cfin[lane] = Ck;
                const int n = n0 + lane;
                if (k == p.nchunks - 1 && p.s_final != nullptr && n < p.N) p.s_final[(size_t)bi * p.N + n] = Ck;
            }
        }
        if (idx >= ni) {
            __syncthreads();
            tile_outputs<GATED>(sa, sb, rows, carry, cfin, EA, EB, p.s_out + ((size_t)bi * p.T + t0) * p.N + n0,
                                p.N, p.s_out != nullptr && n0 + 4 * quad < p.N);
        }
        __syncthreads();                              // buffer `buf` free for the next load
    }
    (void)ok;
    __syncthreads();
    if (tid == 0) finish();
}

}  // namespace

// Workspace of the fused path: the tile flags at the start (where the
// look-back kernel keeps its flags), the reduce-then-scan arrays after them,
// then the block flags.  Returns the bytes it needs (at most the look-back
// workspace in every case it is chosen for: T >= 8 chunks).
int64_t scan_fused_ws_bytes(int B, int T, int N) {
    const int64_t ncb = (N + LB_NC - 1) / LB_NC, nbcb = (int64_t)B * ncb;
    const int64_t nch = (T + LB_TC - 1) / LB_TC, tiles = nbcb * nch;
    const int64_t flag_bytes = ((tiles * 4 + 255) / 256) * 256;
    const int64_t arr = nbcb * chunk_quads((int)nch) * LB_NC * 4 * 4;   // bytes per array
    const int64_t nblk = (nch + FU_CB - 1) / FU_CB;
    return flag_bytes + 3 * arr + nbcb * LB_NC * 4 + nbcb * nblk * 4;
}

// the bytes of the two flag areas a change of geometry must clear: [0, a) and [b, b + c)
void scan_fused_flag_areas(int B, int T, int N, int64_t* a, int64_t* b, int64_t* c) {
    const int64_t ncb = (N + LB_NC - 1) / LB_NC, nbcb = (int64_t)B * ncb;
    const int64_t nch = (T + LB_TC - 1) / LB_TC, tiles = nbcb * nch;
    const int64_t nblk = (nch + FU_CB - 1) / FU_CB;
    *a = ((tiles * 4 + 255) / 256) * 256;
    *c = nbcb * nblk * 4;
    *b = scan_fused_ws_bytes(B, T, N) - *c;
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
    p.nblk = (p.nchunks + FU_CB - 1) / FU_CB;
    p.s0 = x.s0;
    p.s_final = x.s_final;
    p.s_out = x.s_out;
    int64_t fa, fb, fc;
    scan_fused_flag_areas(x.B, x.T, x.N, &fa, &fb, &fc);
    char* base = static_cast<char*>(ws);
    const int64_t arr = (int64_t)p.nbcb * chunk_quads(p.nchunks) * LB_NC * 4;   // floats per array
    p.tflag = reinterpret_cast<uint32_t*>(base);
    p.dA = reinterpret_cast<float*>(base + fa);
    p.dB = p.dA + arr;
    p.dC = p.dB + arr;
    p.cin0 = p.dC + arr;
    p.bflag = reinterpret_cast<uint32_t*>(base + fb);
    p.st = st;
    p.wait_ns = wait_ns;

    auto kern = gated ? scan_fused<true> : scan_fused<false>;
    int occ = 0;
    cudaError_t e = occupancy_once((const void*)kern, LB_THREADS, FU_SMEM, &occ);
    if (e != cudaSuccess) return e;
    // every column's chain CTA plus the workers, all resident (cooperative launch)
    const int64_t resident = (int64_t)occ * sm_count;
    if (resident <= p.nbcb) return cudaErrorInvalidConfiguration;
    const int grid = (int)std::min<int64_t>(resident, p.nbcb + (int64_t)p.ntiles);
    void* args[] = {(void*)&ma, (void*)&mb, (void*)&p};
    e = cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(LB_THREADS), args, FU_SMEM, stream);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace sn
