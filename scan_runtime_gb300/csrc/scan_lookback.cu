// scan_lookback.cu -- chunked associative scans of tier 1 for few channels and
// long T, sm_103a: the decoupled look-back kernel, and the reduce-then-scan
// path (further below) that gives the same bits in three flag-free launches;
// the allocation-free entry point runs the look-back kernel.
//
// Forms as in scan.cu ("SunnyNet 工程化实录" §2.1).  Each tile is 32 channels
// x 128 steps: per-thread folds over 4 steps into (A, B) pairs, a warp-shuffle
// Kogge-Stone scan over the warp's 4 segments, a fixed-order fold across
// warps, and a decoupled look-back across T chunks.  Carries are defined by the
// forward fold C_k = fma(A_k, C_{k-1}, B_k), applied one chunk at a time
// whatever the timing, so the result is deterministic; the last output of
// each chunk is its carry, so splits at multiples of 128 steps are bit-exact
// ("SunnyNet 工程化实录" §4).  The persistent grid is launched cooperatively,
// so every CTA a tile waits on is resident.
#include <algorithm>

#include "scan_tile.cuh"

namespace sn {

// ============================================================ look-back
namespace {
constexpr uint32_t LB_AGG = 1u, LB_INCL = 2u;
constexpr int LB_STAGES = 2;                      // tiles in flight per CTA (3 CTAs per SM)
constexpr uint32_t LB_EPOCH_WRAP = 1u << 29;      // epochs run 1 .. 2^29 - 1 (tags are epoch << 2)
constexpr int LB_FOLD_SOLO = 8;                   // deeper folds are staged by the whole CTA
constexpr int LB_FOLD_B = 24;                     // chunks per staged batch (6 KB of shared memory)
constexpr size_t LB_SMEM = LB_STAGES * LB_TILE_BYTES + LB_STAGES * 8 + 16;

}  // namespace

int64_t lookback_flag_count(int B, int T, int N) {
    const int64_t ncb = (N + LB_NC - 1) / LB_NC, nch = (T + LB_TC - 1) / LB_TC;
    return (int64_t)B * ncb * nch;
}

// Look-back workspace: [ flags: u32 per tile | A | B: f32 per channel and tile |
// carry words: u64 per channel and tile ].  The reduce-then-scan path uses the
// region after the flags for its A, B and C arrays (chunks in groups of four,
// agg_index) and the columns' initial carries; the larger need sets the size.
int64_t lookback_cw_offset(int B, int T, int N) {
    const int64_t tiles = lookback_flag_count(B, T, N);
    return ((tiles * 4 + 255) / 256) * 256 + tiles * 2 * LB_NC * 4;
}

int64_t lookback_ws_bytes(int B, int T, int N) {
    const int64_t tiles = lookback_flag_count(B, T, N);
    const int64_t flag_bytes = ((tiles * 4 + 255) / 256) * 256;
    const int64_t nbcb = (int64_t)B * ((N + LB_NC - 1) / LB_NC);
    const int64_t nq = chunk_quads((T + LB_TC - 1) / LB_TC);
    const int64_t lookback = tiles * (2 * LB_NC * 4 + LB_NC * 8);
    const int64_t reduce_scan = (3 * nbcb * nq * LB_NC * 4 + nbcb * LB_NC) * 4;   // A, B, C groups + cin0
    return flag_bytes + std::max(lookback, reduce_scan);
}

struct LookbackParams {
    int B, T, N, ncb, nbcb, nchunks, ntiles;
    const float* s0;
    float* s_final;
    float* s_out;
    uint32_t* flags;
    float* dA;
    float* dB;
    unsigned long long* cw;   // per tile and channel: (tag | LB_INCL) << 32 | bits of the carry
    uint32_t poison;     // 1: waiters look for a tag no tile publishes (tests the bound)
    SnDevStatus* st;     // error word, abort tag and the launch epoch (lb_epoch, lb_done)
    uint64_t wait_ns;
};

template <bool GATED>
__global__ void __launch_bounds__(LB_THREADS, 3)
scan_lookback(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
              const LookbackParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    float* bufs = reinterpret_cast<float*>(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + LB_STAGES * LB_TILE_BYTES);
    __shared__ float4 wA[8][8], wB[8][8];          // per-warp aggregates [warp][quad]
    __shared__ float carry[LB_NC], cfin[LB_NC];
    __shared__ __align__(16) float stA[LB_FOLD_B][LB_NC], stB[LB_FOLD_B][LB_NC];   // staged aggregates
    __shared__ int s_fold[2];                       // chunks [lo, hi) of a staged fold; hi = 0: none

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = lane & 7;

    // The launch epoch lives in device memory: lb_epoch holds the last launch's
    // (0 = none yet), this launch uses the next one, and the launch's last CTA
    // stores it.  A launch replayed from a CUDA graph thus still gets a fresh
    // tag.  Epochs run 1 .. LB_EPOCH_WRAP - 1, so no tag is 0, the value of
    // cleared flags and of a cleared abort tag.
    __shared__ uint32_t s_epoch;
    if (tid == 0) {
        for (int s = 0; s < LB_STAGES; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
        const uint32_t last = *reinterpret_cast<volatile const uint32_t*>(&p.st->lb_epoch);
        s_epoch = last + 1 >= LB_EPOCH_WRAP ? 1u : last + 1;
    }
    __syncthreads();
    const uint32_t epoch = s_epoch;
    const uint32_t tag = epoch << 2;                          // written with each state
    const uint32_t want = p.poison ? (epoch + 1u) << 2 : tag; // what the waiters look for

    auto tile_coords = [&](int ti, int& k, int& bi, int& cb) {
        k = ti / p.nbcb;
        const int r = ti - k * p.nbcb;
        bi = r / p.ncb;
        cb = r - bi * p.ncb;
    };
    auto issue = [&](int ti, int buf) {
        int k, bi, cb;
        tile_coords(ti, k, bi, cb);
        mbar_arrive_expect_tx(&full[buf], LB_TILE_BYTES);
        float* dst = bufs + buf * 2 * LB_TILE;
        tma_load_3d(dst, &map_a, &full[buf], cb * LB_NC, k * LB_TC, bi);
        tma_load_3d(dst + LB_TILE, &map_b, &full[buf], cb * LB_NC, k * LB_TC, bi);
    };

    int it = 0;
    if (tid == 0) {
        for (int s = 0; s < LB_STAGES - 1; ++s) {
            const int ti = blockIdx.x + s * gridDim.x;
            if (ti < p.ntiles) issue(ti, s);
        }
    }
    for (int ti = blockIdx.x; ti < p.ntiles; ti += gridDim.x, ++it) {
        const int buf = it % LB_STAGES;
        // refill the slot the previous iteration released
        const int ahead = ti + (LB_STAGES - 1) * (int)gridDim.x;
        if (tid == 0 && ahead < p.ntiles) issue(ahead, (it + LB_STAGES - 1) % LB_STAGES);
        int k, bi, cb;
        tile_coords(ti, k, bi, cb);
        const int t0 = k * LB_TC;
        const int n0 = cb * LB_NC;
        const int rows = min(LB_TC, p.T - t0);      // valid rows of this chunk

        if (!__syncthreads_and(mbar_wait(&full[buf], (it / LB_STAGES) & 1, p.wait_ns))) {
            // A copy never landed: report, wait (bounded) for this CTA's copies
            // still in flight, and retire the CTA.
            if (tid == 0) {
                record_error(p.st, SN_E_TIMEOUT, (SN_K_SCAN_LOOKBACK << 16) | 1);
                for (int j = 0; j < LB_STAGES; ++j)
                    if (ti + j * (int)gridDim.x < p.ntiles)
                        (void)mbar_wait(&full[(it + j) % LB_STAGES], ((it + j) / LB_STAGES) & 1, p.wait_ns);
            }
            break;
        }
        const float* sa = bufs + buf * 2 * LB_TILE;
        const float* sb = sa + LB_TILE;

        // ---- phases 1 and 2: the tile's local scan
        float4 EA, EB;
        tile_local_scan<GATED>(sa, sb, rows, wA, wB, EA, EB);

        // ---- phase 3: chunk aggregate and look-back (warp 0, lane = channel)
        const int n = n0 + lane;
        const int base = bi * p.ncb + cb;
        float CA = 1.f, CB = 0.f, cin = 0.f;
        // warp 0: this tile's carry and its outgoing carry words
        auto publish = [&]() {
            const float Ck = __fmaf_rn(CA, cin, CB);
            // The carry word is self-validating (its tag), so it needs no
            // release; the flag only tells a deep look-back where it lies.
            st_relaxed_gpu_u64(p.cw + (size_t)ti * LB_NC + lane,
                               ((unsigned long long)(tag | LB_INCL) << 32) | __float_as_uint(Ck));
            __syncwarp();
            if (lane == 0) st_relaxed_gpu(p.flags + ti, tag | LB_INCL);
            carry[lane] = cin;
            cfin[lane] = Ck;
            if (k == p.nchunks - 1 && p.s_final != nullptr && n < p.N) p.s_final[(size_t)bi * p.N + n] = Ck;
        };
        if (warp == 0) {
            tile_aggregate(wA, wB, lane, CA, CB);
            const uint32_t want_c = want | LB_INCL;   // tag of a carry word this launch wrote
            bool staged = false;
            if (k == 0) {
                cin = (p.s0 != nullptr && n < p.N) ? p.s0[(size_t)bi * p.N + n] : 0.f;
            } else {
                // Usually the predecessor has already published its carry: one
                // load of its carry words (value and tag in one word) finds it.
                unsigned long long w = ld_relaxed_gpu_u64(p.cw + ((size_t)(k - 1) * p.nbcb + base) * LB_NC + lane);
                if (__all_sync(0xffffffffu, (uint32_t)(w >> 32) == want_c)) {
                    cin = __uint_as_float((uint32_t)w);
                } else {
                    // Windowed look-back: lane l inspects chunk (j - l).  Success =
                    // the nearest inclusive carry m with every chunk in (m, k)
                    // published.  The aggregate is published the first time a
                    // probe does not succeed.
                    int j = k - 1;
                    int m = -2;                       // chunk whose inclusive carry we take (-1 = s0)
                    bool published = false;
                    const uint64_t tstart = global_ns();
                    bool timed_out = false;
                    auto give_up = [&]() {
                        return global_ns() - tstart > p.wait_ns ||
                               *reinterpret_cast<volatile const uint32_t*>(&p.st->abort_tag) == tag;
                    };
                    while (true) {
                        const int jl = j - lane;
                        uint32_t state = LB_INCL;     // chunks before 0 act as "inclusive = s0"
                        if (jl >= 0) {
                            const uint32_t f = ld_acquire_gpu(p.flags + (size_t)jl * p.nbcb + base);
                            state = ((f & ~3u) == want) ? (f & 3u) : 0u;
                        }
                        const uint32_t incl = __ballot_sync(0xffffffffu, state == LB_INCL);
                        const uint32_t none = __ballot_sync(0xffffffffu, state == 0u);
                        if (incl != 0u) {
                            const int l = __ffs(incl) - 1;
                            if ((none & ((1u << l) - 1u)) == 0u) {   // all nearer chunks published
                                m = j - l;
                                break;
                            }
                        } else if (none == 0u) {      // 32 aggregates: look further back
                            j -= 32;
                            continue;
                        }
                        if (!published) {             // let successors fold through this chunk
                            const size_t me = (size_t)ti * LB_NC + lane;
                            p.dA[me] = CA;
                            p.dB[me] = CB;
                            __syncwarp();
                            if (lane == 0) st_release_gpu(p.flags + ti, tag | LB_AGG);
                            published = true;
                        }
                        // give up after the limit, or at once if another tile of this
                        // launch already gave up (its successors would only wait too)
                        if (give_up()) {
                            timed_out = true;
                            break;
                        }
                    }
                    if (!timed_out) {
                        // chunk m's flag announced its carry; the carry words
                        // themselves may land a moment later
                        const unsigned long long* cm = p.cw + ((size_t)m * p.nbcb + base) * LB_NC + lane;
                        while (true) {
                            w = ld_relaxed_gpu_u64(cm);
                            if (__all_sync(0xffffffffu, (uint32_t)(w >> 32) == want_c)) break;
                            if (give_up()) {
                                timed_out = true;
                                break;
                            }
                        }
                        cin = __uint_as_float((uint32_t)w);
                    }
                    __syncwarp();
                    if (timed_out) {
                        if (lane == 0) {
                            record_error(p.st, SN_E_TIMEOUT, (SN_K_SCAN_LOOKBACK << 16) | 2);
                            atomicExch(&p.st->abort_tag, tag);
                        }
                        cin = 0.f;
                    } else if (k - 1 - m > LB_FOLD_SOLO) {
                        // a deep fold: the whole CTA stages the aggregates below
                        staged = true;
                        if (lane == 0) {
                            s_fold[0] = m + 1;
                            s_fold[1] = k;
                        }
                    } else {
                        // forward fold from the inclusive carry at m through m+1 .. k-1,
                        // one chunk at a time (loads batched eight chunks ahead)
                        for (int i0 = m + 1; i0 < k; i0 += 8) {
                            float fa[8], fb[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u) {
                                const int i = i0 + u < k ? i0 + u : k - 1;
                                const size_t o = ((size_t)i * p.nbcb + base) * LB_NC + lane;
                                fa[u] = __ldcg(p.dA + o);
                                fb[u] = __ldcg(p.dB + o);
                            }
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                if (i0 + u < k) cin = __fmaf_rn(fa[u], cin, fb[u]);
                        }
                    }
                }
            }
            if (!staged) {
                if (lane == 0) s_fold[1] = 0;
                publish();
            }
        }
        __syncthreads();
        if (s_fold[1] != 0) {
            // Deep fold (many chunks of one column in flight): the CTA loads the
            // aggregates of LB_FOLD_B chunks at a time into shared memory (one
            // L2 round trip per batch), and warp 0 folds them one chunk at a
            // time, C = fma(A_i, C, B_i), as the short fold does.  The flags of
            // these chunks were read with acquire by warp 0 before the barrier.
            const int lo = s_fold[0], hi = s_fold[1];
            const int u = tid >> 3, q4 = tid & 7;   // chunk of the batch, quarter of its 32 channels
            for (int c0 = lo; c0 < hi; c0 += LB_FOLD_B) {
                const int cnt = min(LB_FOLD_B, hi - c0);
                if (u < cnt) {
                    const size_t o = ((size_t)(c0 + u) * p.nbcb + base) * LB_NC + 4 * q4;
                    *reinterpret_cast<float4*>(&stA[u][4 * q4]) = __ldcg(reinterpret_cast<const float4*>(p.dA + o));
                    *reinterpret_cast<float4*>(&stB[u][4 * q4]) = __ldcg(reinterpret_cast<const float4*>(p.dB + o));
                }
                __syncthreads();
                if (warp == 0)
                    for (int v = 0; v < cnt; ++v) cin = __fmaf_rn(stA[v][lane], cin, stB[v][lane]);
                __syncthreads();
            }
            if (warp == 0) publish();
            __syncthreads();
        }
        // ---- phase 4: states of this thread's segment from its exclusive prefix
        tile_outputs<GATED>(sa, sb, rows, carry, cfin, EA, EB, p.s_out + ((size_t)bi * p.T + t0) * p.N + n0, p.N,
                            p.s_out != nullptr && n0 + 4 * quad < p.N);
        __syncthreads();                              // buffer `buf` free for the next prefetch
    }
    // every CTA ends here (also after a copy timeout): the last one records
    // this launch's epoch for the next launch
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(&p.st->lb_done, 1u) == gridDim.x - 1) {
            p.st->lb_done = 0;
            p.st->lb_epoch = epoch;
            __threadfence();
        }
    }
}

bool lookback_supported(const ScanArgs& x) { return scan_tma_ok(x); }

// ============================================================ reduce-then-scan
// For few channel tiles and long T the look-back folds deep: with hundreds of
// a column's chunks in flight at once, each chunk's carry must be folded
// forward through hundreds of predecessors' aggregates, one L2 round trip per
// batch.  This path takes the carries out of the tiles instead:
//   scan_pass<.., false>  every tile's aggregate (A_k, B_k) per channel;
//   scan_chain            per column, the carries C_k = fma(A_k, C_{k-1}, B_k)
//                         over all chunks in order, with the aggregates staged
//                         through shared memory by bulk copies;
//   scan_pass<.., true>   every tile's states from its incoming carry.
// The local scan, the aggregates and the carry chain are the look-back
// kernel's own operations in the same order, so both paths give the same bits.
// a and b are read twice (20 bytes per element instead of 12).
// Workspace: A, B and C arrays at agg_index (per column, chunks in groups of
// four), then the columns' initial carries as the chain read them (the output
// pass takes its first chunk's carry there, since s_final may be s0's buffer).
namespace {

constexpr int PASS_STAGES = 2;                    // tiles in flight per CTA of the two passes (3 CTAs
                                                  // per SM; deeper rings with fewer CTAs measured slower)
constexpr size_t PASS_SMEM = PASS_STAGES * LB_TILE_BYTES + PASS_STAGES * 8 + 16;

struct PassParams {
    int B, T, N, ncb, nbcb, nchunks, ntiles;
    const float* s0;
    float* s_final;
    float* s_out;
    float* dA;
    float* dB;
    float* dC;
    float* cin0;         // [column][channel] initial carries, written by the chain
    SnDevStatus* st;
    uint64_t wait_ns;
};

template <bool GATED, bool OUT>
__global__ void __launch_bounds__(LB_THREADS, 3)
scan_pass(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b, const PassParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    float* bufs = reinterpret_cast<float*>(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + PASS_STAGES * LB_TILE_BYTES);
    __shared__ float4 wA[8][8], wB[8][8];
    __shared__ float carry[LB_NC], cfin[LB_NC];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = lane & 7;

    if (tid == 0) {
        for (int s = 0; s < PASS_STAGES; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // tiles column-major within a chunk row, as the look-back kernel; the output pass visits them in the
    // opposite order, so it starts on the tiles the aggregate pass read last,
    // which are still in L2
    auto tile_coords = [&](int ti, int& k, int& bi, int& cb) {
        if (OUT) ti = p.ntiles - 1 - ti;
        k = ti / p.nbcb;
        const int r = ti - k * p.nbcb;
        bi = r / p.ncb;
        cb = r - bi * p.ncb;
    };
    auto issue = [&](int ti, int buf) {
        int k, bi, cb;
        tile_coords(ti, k, bi, cb);
        mbar_arrive_expect_tx(&full[buf], LB_TILE_BYTES);
        float* dst = bufs + buf * 2 * LB_TILE;
        tma_load_3d(dst, &map_a, &full[buf], cb * LB_NC, k * LB_TC, bi);
        tma_load_3d(dst + LB_TILE, &map_b, &full[buf], cb * LB_NC, k * LB_TC, bi);
    };
    int it = 0;
    if (tid == 0) {
        for (int s = 0; s < PASS_STAGES - 1; ++s) {
            const int ti = blockIdx.x + s * gridDim.x;
            if (ti < p.ntiles) issue(ti, s);
        }
    }
    for (int ti = blockIdx.x; ti < p.ntiles; ti += gridDim.x, ++it) {
        const int buf = it % PASS_STAGES;
        const int ahead = ti + (PASS_STAGES - 1) * (int)gridDim.x;
        if (tid == 0 && ahead < p.ntiles) issue(ahead, (it + PASS_STAGES - 1) % PASS_STAGES);
        int k, bi, cb;
        tile_coords(ti, k, bi, cb);
        const int t0 = k * LB_TC, n0 = cb * LB_NC;
        const int rows = min(LB_TC, p.T - t0);
        if (!__syncthreads_and(mbar_wait(&full[buf], (it / PASS_STAGES) & 1, p.wait_ns))) {
            if (tid == 0) {
                record_error(p.st, SN_E_TIMEOUT, (SN_K_SCAN_LOOKBACK << 16) | 3);
                for (int j = 0; j < PASS_STAGES; ++j)
                    if (ti + j * (int)gridDim.x < p.ntiles)
                        (void)mbar_wait(&full[(it + j) % PASS_STAGES], ((it + j) / PASS_STAGES) & 1, p.wait_ns);
            }
            return;
        }
        const float* sa = bufs + buf * 2 * LB_TILE;
        const float* sb = sa + LB_TILE;
        float4 EA, EB;
        tile_local_scan<GATED>(sa, sb, rows, wA, wB, EA, EB);
        const size_t col = (size_t)bi * p.ncb + cb;
        const int nq = chunk_quads(p.nchunks);
        const size_t me = agg_index(col, nq, k, lane);
        if (warp == 0) {
            float CA, CB;
            tile_aggregate(wA, wB, lane, CA, CB);
            if (!OUT) {
                p.dA[me] = CA;
                p.dB[me] = CB;
            } else {
                const int n = n0 + lane;
                // s0 itself is not read here: a call may write its final states over it
                const float cin =
                    k == 0 ? __ldg(p.cin0 + col * LB_NC + lane) : __ldg(p.dC + agg_index(col, nq, k - 1, lane));
                const float Ck = __fmaf_rn(CA, cin, CB);
                carry[lane] = cin;
                cfin[lane] = Ck;
                if (k == p.nchunks - 1 && p.s_final != nullptr && n < p.N) p.s_final[(size_t)bi * p.N + n] = Ck;
            }
        }
        if (OUT) {
            __syncthreads();
            tile_outputs<GATED>(sa, sb, rows, carry, cfin, EA, EB, p.s_out + ((size_t)bi * p.T + t0) * p.N + n0,
                                p.N, p.s_out != nullptr && n0 + 4 * quad < p.N);
        }
        __syncthreads();                              // buffer `buf` free for the next prefetch
    }
}

}  // namespace

cudaError_t launch_scan_reduce_scan(const ScanArgs& x, bool gated, void* ws, SnDevStatus* st, uint64_t wait_ns,
                                    int sm_count, cudaStream_t stream) {
    CUtensorMap ma, mb;
    if (!make_scan_map(&ma, x.a, x.B, x.T, x.N, LB_NC, LB_TC) ||
        !make_scan_map(&mb, x.b, x.B, x.T, x.N, LB_NC, LB_TC))
        return cudaErrorInvalidValue;
    PassParams p;
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
    const int64_t tiles = p.ntiles;
    const int64_t flag_bytes = ((tiles * 4 + 255) / 256) * 256;
    const int64_t arr = (int64_t)p.nbcb * chunk_quads(p.nchunks) * LB_NC * 4;   // floats per array
    p.dA = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + flag_bytes);
    p.dB = p.dA + arr;
    p.dC = p.dB + arr;
    p.cin0 = p.dC + arr;             // nbcb * 32 floats
    p.st = st;
    p.wait_ns = wait_ns;

    auto k_agg = gated ? scan_pass<true, false> : scan_pass<false, false>;
    auto k_out = gated ? scan_pass<true, true> : scan_pass<false, true>;
    int occ = 0;
    cudaError_t e = occupancy_once((const void*)k_agg, LB_THREADS, PASS_SMEM, &occ);
    if (e != cudaSuccess) return e;
    e = occupancy_once((const void*)k_out, LB_THREADS, PASS_SMEM, &occ);
    if (e != cudaSuccess) return e;
    e = set_smem_attr_once((const void*)scan_chain<false>, CHAIN_SMEM);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<int64_t>(tiles, (int64_t)occ * sm_count);
    k_agg<<<grid, LB_THREADS, PASS_SMEM, stream>>>(ma, mb, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const ChainParams cp{p.N, p.ncb, p.nchunks, x.s0, p.dA, p.dB, p.dC, p.cin0, st, wait_ns};
    scan_chain<false><<<(unsigned)p.nbcb, 32, CHAIN_SMEM, stream>>>(cp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_out<<<grid, LB_THREADS, PASS_SMEM, stream>>>(ma, mb, p);
    return cudaGetLastError();
}

cudaError_t launch_scan_lookback(const ScanArgs& x, bool gated, void* ws, int poison, SnDevStatus* st,
                                 uint64_t wait_ns, int sm_count, cudaStream_t stream) {
    CUtensorMap ma, mb;
    if (!make_scan_map(&ma, x.a, x.B, x.T, x.N, LB_NC, LB_TC) ||
        !make_scan_map(&mb, x.b, x.B, x.T, x.N, LB_NC, LB_TC))
        return cudaErrorInvalidValue;
    LookbackParams p;
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
    const int64_t tiles = p.ntiles;
    const int64_t flag_bytes = ((tiles * 4 + 255) / 256) * 256;
    p.flags = reinterpret_cast<uint32_t*>(ws);
    p.dA = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + flag_bytes);
    p.dB = p.dA + tiles * LB_NC;
    p.cw = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(ws) + lookback_cw_offset(x.B, x.T, x.N));
    p.poison = poison ? 1u : 0u;
    p.st = st;
    p.wait_ns = wait_ns;

    auto kern = gated ? scan_lookback<true> : scan_lookback<false>;
    int occ = 0;
    cudaError_t oe = occupancy_once((const void*)kern, LB_THREADS, LB_SMEM, &occ);
    if (oe != cudaSuccess) return oe;
    const int grid = std::min<int64_t>(tiles, (int64_t)occ * sm_count);
    void* args[] = {(void*)&ma, (void*)&mb, (void*)&p};
    cudaError_t e = cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(LB_THREADS), args, LB_SMEM,
                                                stream);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace sn

// ============================================================ allocation-free entry point
//
// sn_scan_lookback_noalloc runs the look-back scan above with its scratch in a
// file-scope device array instead of a workspace handed over by the caller.
// It is for callers that must not allocate device memory at run time: code
// running under a fixed memory budget or a custom allocator that owns the
// whole device, plugins whose host application forbids cudaMalloc after
// start-up, and paths that cannot create an SnCtx (context creation allocates
// the context's status block).
//
// The array (kNoallocScratchBytes, about 20 MiB) lives on every device that
// loads this library until the process exits.  Layout, fixed for every call:
//   [ status block 256 B | flags: kNoallocMaxTiles x u32 | A | B aggregates |
//     carry words: kNoallocMaxTiles x 32 x u64 ]
// Flags and carry words stay at fixed offsets, so such a word only ever holds
// a tagged value or zero.
#include <atomic>
#include <cstddef>
#include <mutex>

namespace {

constexpr int64_t kNoallocMaxTiles = 40960;
constexpr int64_t kNoallocFlagsOff = 256;
constexpr int64_t kNoallocDataOff = kNoallocFlagsOff + kNoallocMaxTiles * 4;
constexpr int64_t kNoallocCwOff = kNoallocDataOff + kNoallocMaxTiles * 2 * sn::LB_NC * 4;
constexpr int64_t kNoallocScratchBytes = kNoallocCwOff + kNoallocMaxTiles * sn::LB_NC * 8;
static_assert(kNoallocScratchBytes <= (int64_t(24) << 20), "scratch stays within 24 MiB");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kNoallocMaxDevices = 64;

// Calls between two clears of the flag and carry areas at one tile count.
// Every launch rewrites the flags and carry words of all its tiles, so with an
// unchanged tile count a stale word holds the previous launch's tag, never the
// current one; the periodic clear bounds the case in which a launch that gave
// up left some words unwritten, well before the epoch can wrap (2^29 - 1).
constexpr uint64_t kNoallocClearEvery = uint64_t(1) << 24;

struct NoallocDevice {
    bool ready = false;
    unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch on this device
    int sm_count = 0;
    int occ[2] = {0, 0};
    int64_t last_tiles = -1;            // tile count of the previous call (-1: areas need a clear)
    uint64_t calls_since_clear = 0;
};
NoallocDevice g_noalloc[kNoallocMaxDevices];
std::mutex g_noalloc_mutex;

bool nz_overlap(const void* p, int64_t pb, const void* q, int64_t qb) {
    if (p == nullptr || q == nullptr) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p), b0 = reinterpret_cast<uintptr_t>(q);
    return a0 < b0 + (uintptr_t)qb && b0 < a0 + (uintptr_t)pb;
}

}  // namespace

extern "C" sn_status sn_scan_lookback_noalloc(int32_t gated, int32_t B, int32_t T, int32_t N, const float* a,
                                              const float* b, const float* s0, float* s_final, float* s_out,
                                              int32_t* status_out, void* stream) {
    using namespace sn;
    // ---- arguments (checked before anything is enqueued)
    if (a == nullptr || b == nullptr || B <= 0 || T <= 0 || N <= 0 || (gated != 0 && gated != 1))
        return SN_E_INVAL;
    const void* ptrs[6] = {a, b, s0, s_final, s_out, status_out};
    for (const void* q : ptrs)
        if (q != nullptr && (reinterpret_cast<uintptr_t>(q) & 3u) != 0) return SN_E_INVAL;
    // element-count bound checked by division first: B * T * N itself can
    // exceed the int64 range for int32 dimensions
    constexpr int64_t kMaxElems = int64_t(1) << 40;
    if ((int64_t)T > kMaxElems / B / N) return SN_E_INVAL;
    const int64_t big = (int64_t)B * T * N * 4, small = (int64_t)B * N * 4;
    const void* ins[3] = {a, b, s0};
    const int64_t insz[3] = {big, big, small};
    void* outs[3] = {s_final, s_out, status_out};
    const int64_t outsz[3] = {small, big, 4};
    for (int i = 0; i < 3; ++i) {
        for (int j = 0; j < 3; ++j) {
            const bool inplace = (i == 0 && j == 2 && outs[0] == ins[2]);   // s_final may equal s0
            if (!inplace && nz_overlap(outs[i], outsz[i], ins[j], insz[j])) return SN_E_INVAL;
        }
        for (int j = i + 1; j < 3; ++j)
            if (nz_overlap(outs[i], outsz[i], outs[j], outsz[j])) return SN_E_INVAL;
    }
    ScanArgs x{B, T, N, a, b, s0, s_final, s_out};
    if (!scan_tma_ok(x)) return SN_E_UNSUPPORTED;
    const int64_t tiles = lookback_flag_count(B, T, N);
    if (tiles > kNoallocMaxTiles) return SN_E_NOMEM;   // beyond the fixed scratch

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoallocMaxDevices) return SN_E_DEVICE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    auto kern = gated ? scan_lookback<true> : scan_lookback<false>;

    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoallocDevice& d = g_noalloc[dev];
    if (!d.ready) {
        // One-time set-up on this device (the first call; it must precede any
        // stream capture): the array's device address, the kernel's shared
        // memory opt-in and occupancy, and cleared status, flag and carry areas.
        void* sym = nullptr;
        if (cudaGetSymbolAddress(&sym, g_noalloc_scratch) != cudaSuccess || sym == nullptr) return SN_E_DEVICE;
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return SN_E_DEVICE;
        if (prop.major != 10 || prop.minor != 3) return SN_E_UNSUPPORTED;
        for (int g = 0; g < 2; ++g) {
            auto k = g ? scan_lookback<true> : scan_lookback<false>;
            if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LB_SMEM) != cudaSuccess ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.occ[g], k, LB_THREADS, LB_SMEM) != cudaSuccess ||
                d.occ[g] < 1)
                return SN_E_DEVICE;
        }
        if (cudaMemsetAsync(sym, 0, sizeof(SnDevStatus), s) != cudaSuccess) return SN_E_DEVICE;
        d.scratch = static_cast<unsigned char*>(sym);
        d.sm_count = prop.multiProcessorCount;
        d.last_tiles = -1;
        d.ready = true;
    }
    if (tiles != d.last_tiles || d.calls_since_clear >= kNoallocClearEvery) {
        // A different tile count maps tiles onto flag and carry words that an
        // older call of another shape may have tagged: clear both areas (in
        // stream order, before the launch), as the context path does.
        if (cudaMemsetAsync(d.scratch + kNoallocFlagsOff, 0, (size_t)(kNoallocDataOff - kNoallocFlagsOff), s) !=
                cudaSuccess ||
            cudaMemsetAsync(d.scratch + kNoallocCwOff, 0, (size_t)(kNoallocScratchBytes - kNoallocCwOff), s) !=
                cudaSuccess)
            return SN_E_DEVICE;
        d.last_tiles = tiles;
        d.calls_since_clear = 0;
    }
    ++d.calls_since_clear;

    CUtensorMap ma, mb;
    if (!make_scan_map(&ma, a, B, T, N, LB_NC, LB_TC) || !make_scan_map(&mb, b, B, T, N, LB_NC, LB_TC))
        return SN_E_DEVICE;
    SnDevStatus* st = reinterpret_cast<SnDevStatus*>(d.scratch);
    LookbackParams p;
    p.B = B;
    p.T = T;
    p.N = N;
    p.ncb = (N + LB_NC - 1) / LB_NC;
    p.nbcb = B * p.ncb;
    p.nchunks = (T + LB_TC - 1) / LB_TC;
    p.ntiles = p.nbcb * p.nchunks;
    p.s0 = s0;
    p.s_final = s_final;
    p.s_out = s_out;
    p.flags = reinterpret_cast<uint32_t*>(d.scratch + kNoallocFlagsOff);
    p.dA = reinterpret_cast<float*>(d.scratch + kNoallocDataOff);
    p.dB = p.dA + tiles * LB_NC;
    p.cw = reinterpret_cast<unsigned long long*>(d.scratch + kNoallocCwOff);
    p.poison = 0;
    p.st = st;                                    // also holds the launch epoch
    p.wait_ns = 1000000000ull;                    // 1 s bound on every device-side wait
    // this call's error word, error site and abort tag start at zero (the
    // launch epoch after them is kept)
    static_assert(offsetof(SnDevStatus, abort_tag) == 2 * sizeof(int) &&
                      offsetof(SnDevStatus, lb_epoch) == 3 * sizeof(int),
                  "error, site and abort tag precede the epoch");
    if (cudaMemsetAsync(st, 0, 3 * sizeof(int), s) != cudaSuccess) return SN_E_DEVICE;
    const int grid = (int)std::min<int64_t>(tiles, (int64_t)d.occ[gated] * d.sm_count);
    void* args[] = {(void*)&ma, (void*)&mb, (void*)&p};
    if (cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(LB_THREADS), args, LB_SMEM, s) !=
        cudaSuccess)
        return SN_E_DEVICE;
    if (status_out != nullptr &&
        cudaMemcpyAsync(status_out, &st->error, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return SN_E_DEVICE;
    return SN_OK;
}
