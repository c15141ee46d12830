// scan_fused.cu -- the chunked scans of tier 1 for few channels and long T in
// one launch that reads a and b once ("SunnyNet 工程化实录" §2.1 forms; §4
// bit-exact continuation).
//
// The reduce-then-scan path (scan_lookback.cu) reads a and b twice: a pass for
// every tile's aggregate, a carry chain per column, then a pass for the states
// (20 bytes of traffic per element against the 12 the scan needs).  Here one
// cooperative launch keeps each tile in shared memory from its aggregate to
// its states:
//   * state CTAs (persistent, two per SM) take the tiles w, w + nw, ... in
//     chunk order through a ring of FU_STAGES tiles loaded by TMA.  A tile's
//     local scan ends in its aggregate (A_k, B_k), published at once as two
//     tagged 64-bit words per channel; the CTA then scans its next tile and
//     publishes that aggregate too before it waits for the first tile's carry
//     and writes its states;
//   * a chain CTA per column of tiles: warps 2..7 poll the aggregate words, a
//     batch of FU_PB chunks at a time, into a ring in shared memory; warp 0
//     folds C_k = fma(A_k, C_{k-1}, B_k) in chunk order and publishes the
//     carry that ends every group of eight chunks as a tagged word;
//   * a state tile's incoming carry C_{k-1} is the published carry entering
//     its group of eight, followed by the aggregates of the chunks before it
//     in the group, folded in the chain's order.
// A tile's carry thus needs the aggregates of its column up to the end of its
// batch (fewer than FU_PB chunks on), while every CTA publishes one tile
// beyond the one whose carry it awaits: with more state CTAs than FU_PB + 1
// tiles per column no chain waits on a CTA that waits on it, and the launcher
// runs the reduce-then-scan launches (the same bits) otherwise.
// A single-copy-atomic 64-bit access reads or writes tag and value together,
// so no word needs a fence or a separate flag: a reader that sees the
// launch's tag sees the value written with it.
// Every operation is the reduce-then-scan path's in the same order (tile
// local scan, aggregate, fold, outputs), so all chunked paths give the same
// bits.  Every CTA is resident (cooperative launch) and every wait is bounded
// (SN_OPT_WAIT_LIMIT_US): a CTA that gives up records SN_E_TIMEOUT and tags
// the launch, and the others stop waiting at once.  The tags carry the launch
// epoch (kept in device memory, shared with the look-back kernel), so no call
// needs a memset while the geometry stays the same.
#include <algorithm>

#include "scan_tile.cuh"

namespace sn {
namespace {

constexpr int FU_STAGES = 3;                        // tiles in flight in a state CTA
constexpr int FU_CB = 32;                           // chunks per block of a chain's ring
constexpr int FU_PB = 16;                           // chunks per polled batch (a block's halves)
constexpr int FU_NS = 8;                            // blocks in a chain's ring
constexpr int FU_NP = 6;                            // polling warps of a chain CTA (warps 2..7)
constexpr uint32_t FU_AGG = 2u;                     // tag state of an aggregate word
constexpr uint32_t FU_CARRY = 3u;                   // tag state of a carry word
constexpr uint32_t FU_EPOCH_WRAP = 1u << 29;
constexpr uint64_t FU_ABORT_NS = 4000;              // a waiting thread reads the abort word this often
constexpr uint32_t FU_CBLK_FLOATS = FU_CB * LB_NC;  // one block of one array ([group][channel][4])
constexpr int FU_NB = FU_CB / FU_PB;                // batches per block
constexpr size_t FU_RING = FU_STAGES * (size_t)LB_TILE_BYTES;
static_assert((size_t)FU_NS * 2 * FU_CBLK_FLOATS * 4 <= FU_RING, "a chain CTA's ring fits in the tile ring");
static_assert(FU_CB % FU_PB == 0 && FU_PB % 8 == 0, "batches of whole groups of eight chunks");
static_assert(2 + FU_NP == LB_THREADS / 32, "a chain CTA: folding and polling warps");
constexpr int FU_NBAR = FU_STAGES + FU_NS * FU_NB + FU_NS;
constexpr size_t FU_SMEM = FU_RING + FU_NBAR * 8;

struct FusedParams {
    int B, T, N, ncb, nbcb, nchunks, ntiles;
    const float* s0;
    float* s_final;
    float* s_out;
    unsigned long long* aw;       // aggregates [col][chunk][channel][A | B]: (tag | FU_AGG) << 32 | bits
    unsigned long long* cw8;      // [col][m][channel]: (tag | FU_CARRY) << 32 | bits of C_{8m+7}
    unsigned long long* cw0;      // [col][channel]: the same for the initial carry
    SnDevStatus* st;              // error word, abort tag and the launch epoch
    uint64_t wait_ns;
    int poison;                   // 1: state tiles wait for a carry state no CTA writes (tests the bound)
};

__device__ __forceinline__ void st_relaxed_gpu_v2u64(unsigned long long* p, unsigned long long a,
                                                     unsigned long long b) {
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
// Two 64-bit words, each read single-copy atomically (the pair is not).
__device__ __forceinline__ ulonglong2 ld_relaxed_gpu_v2u64(const unsigned long long* p) {
    ulonglong2 v;
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p) : "memory");
    return v;
}

constexpr unsigned long long FU_HI = 0xffffffff00000000ull;
__device__ __forceinline__ float lo_f(unsigned long long w) { return __uint_as_float((uint32_t)w); }

// The launch's tag and its abort and completion bookkeeping.
struct Launch {
    const FusedParams* p;
    uint32_t epoch, tag;
    __device__ bool aborted() const {
        return *reinterpret_cast<volatile const uint32_t*>(&p->st->abort_tag) == tag;
    }
    __device__ void give_up(int site) const {
        record_error(p->st, SN_E_TIMEOUT, (SN_K_SCAN_LOOKBACK << 16) | site);
        atomicExch(&p->st->abort_tag, tag);
    }
    // the launch's last CTA to finish records its epoch for the next launch
    __device__ void finish() const {
        __threadfence();
        if (atomicAdd(&p->st->lb_done, 1u) == gridDim.x - 1) {
            p->st->lb_done = 0;
            p->st->lb_epoch = epoch;
            __threadfence();
        }
    }
    // Whether a wait that began at t0 should end: its time ran out or the
    // launch gave up.  The abort word is a global load (about a microsecond
    // under full HBM traffic), so it is read only every FU_ABORT_NS of
    // waiting, lest each spin take that long to see its own condition.
    __device__ bool expired(uint64_t t0, uint64_t& next) const {
        const uint64_t now = global_ns();
        if (now - t0 > p->wait_ns) return true;
        if (now < next) return false;
        next = now + FU_ABORT_NS;
        return aborted();
    }
    // a barrier phase, waited for at most wait_ns and no longer once the launch gave up
    __device__ bool wait(uint64_t* b, uint32_t parity) const {
        if (mbar_try_wait(b, parity)) return true;
        const uint64_t t0 = global_ns();
        uint64_t next = t0 + FU_ABORT_NS;
        while (!mbar_try_wait(b, parity))
            if (expired(t0, next)) return false;
        return true;
    }
};

// Polling warp of a chain CTA: the blocks j = pw, pw + FU_NP, ... of column
// col's aggregate words into ring stage j % FU_NS, as [group][channel][4]
// floats of A, then of B, one batch of FU_PB chunks at a time (each batch's
// barrier completes on its own).  A batch's words are read at once; those not
// yet tagged by this launch are read again, all together, until every one is.
__device__ __forceinline__ bool chain_poll(const FusedParams& p, const Launch& L, size_t col, int pw, int lane,
                                           float* ring, uint64_t* full, uint64_t* empty) {
    const unsigned long long hi_a = (unsigned long long)(L.tag | FU_AGG) << 32;
    const unsigned long long* awc = p.aw + col * p.nchunks * LB_NC * 2 + lane * 2;
    auto untagged = [&](const ulonglong2& w) { return (w.x & FU_HI) != hi_a || (w.y & FU_HI) != hi_a; };
    const int nblk = (p.nchunks + FU_CB - 1) / FU_CB;
    for (int j = pw; j < nblk; j += FU_NP) {
        const int s = j % FU_NS;
        if (j >= FU_NS && !__all_sync(0xffffffffu, L.wait(&empty[s], (uint32_t)(j / FU_NS - 1) & 1u))) return false;
        const int k0 = j * FU_CB, cnt = min(FU_CB, p.nchunks - k0);
        float4* rA = reinterpret_cast<float4*>(ring + (size_t)s * 2 * FU_CBLK_FLOATS) + lane;
        float4* rB = rA + FU_CBLK_FLOATS / 4;
        for (int c0 = 0; c0 < cnt; c0 += FU_PB) {
            ulonglong2 v[FU_PB];
#pragma unroll
            for (int u = 0; u < FU_PB; ++u) {
                v[u] = make_ulonglong2(hi_a | 0x3f800000ull, hi_a);   // past the last chunk: identity
                if (c0 + u < cnt) v[u] = ld_relaxed_gpu_v2u64(awc + (size_t)(k0 + c0 + u) * LB_NC * 2);
            }
            uint32_t bad = 0;
#pragma unroll
            for (int u = 0; u < FU_PB; ++u)
                if (untagged(v[u])) bad |= 1u << u;
            if (__any_sync(0xffffffffu, bad != 0)) {
                const uint64_t t0 = global_ns();
                uint64_t next = t0 + FU_ABORT_NS;
                do {
                    // (the warp leaves together: the loop's votes need every lane)
                    if (__any_sync(0xffffffffu, L.expired(t0, next))) return false;
                    __nanosleep(64);
#pragma unroll
                    for (int u = 0; u < FU_PB; ++u)
                        if (bad >> u & 1u) v[u] = ld_relaxed_gpu_v2u64(awc + (size_t)(k0 + c0 + u) * LB_NC * 2);
                    bad = 0;
#pragma unroll
                    for (int u = 0; u < FU_PB; ++u)
                        if (untagged(v[u])) bad |= 1u << u;
                } while (__any_sync(0xffffffffu, bad != 0));
            }
#pragma unroll
            for (int g = 0; g < FU_PB / 4; ++g) {
                rA[((c0 >> 2) + g) * LB_NC] = make_float4(lo_f(v[4 * g].x), lo_f(v[4 * g + 1].x),
                                                          lo_f(v[4 * g + 2].x), lo_f(v[4 * g + 3].x));
                rB[((c0 >> 2) + g) * LB_NC] = make_float4(lo_f(v[4 * g].y), lo_f(v[4 * g + 1].y),
                                                          lo_f(v[4 * g + 2].y), lo_f(v[4 * g + 3].y));
            }
            __syncwarp();                             // the batch is in the ring
            if (lane == 0) mbar_arrive(&full[s * FU_NB + c0 / FU_PB]);
        }
    }
    return true;
}

// Folding warp of a chain CTA (lane = channel): C_k = fma(A_k, C_{k-1}, B_k)
// over the column's chunks in order, batch by batch from the ring; every
// C_{8m+7} goes out at once as a tagged word.  Returns false if a wait gave up.
__device__ __forceinline__ bool chain_fold(const FusedParams& p, const Launch& L, size_t col, int lane,
                                           const float* ring, uint64_t* full, uint64_t* empty) {
    const int bi = (int)(col / p.ncb), n = (int)(col % p.ncb) * LB_NC + lane;
    const int nblk = (p.nchunks + FU_CB - 1) / FU_CB, nm = (p.nchunks + 7) >> 3;
    const unsigned long long hi = (unsigned long long)(L.tag | FU_CARRY) << 32;
    unsigned long long* cwc = p.cw8 + col * nm * LB_NC + lane;
    // the first chunk's carry is published from here, not read from s0 by the
    // state tiles: a call may write its final states over s0
    float c = (p.s0 != nullptr && n < p.N) ? p.s0[(size_t)bi * p.N + n] : 0.f;
    st_relaxed_gpu_u64(p.cw0 + col * LB_NC + lane, hi | __float_as_uint(c));
    for (int j = 0; j < nblk; ++j) {
        const int s = j % FU_NS, k0 = j * FU_CB, cnt = min(FU_CB, p.nchunks - k0);
        const float* fA = ring + (size_t)s * 2 * FU_CBLK_FLOATS;
        const float* fB = fA + FU_CBLK_FLOATS;
        for (int i0 = 0; i0 < cnt; i0 += FU_PB) {
            if (!__all_sync(0xffffffffu, L.wait(&full[s * FU_NB + i0 / FU_PB], (uint32_t)(j / FU_NS) & 1u)))
                return false;
            if (cnt - i0 >= FU_PB) {
                // a whole batch: its groups are read before the FMAs that consume them
                constexpr int NG = FU_PB / 4;
                const float4* sA = reinterpret_cast<const float4*>(fA) + (i0 >> 2) * LB_NC + lane;
                const float4* sB = reinterpret_cast<const float4*>(fB) + (i0 >> 2) * LB_NC + lane;
                float4 a[NG], b[NG];
#pragma unroll
                for (int g = 0; g < NG; ++g) {
                    a[g] = sA[g * LB_NC];
                    b[g] = sB[g * LB_NC];
                }
#pragma unroll
                for (int g = 0; g < NG; ++g) {
                    c = __fmaf_rn(a[g].x, c, b[g].x);
                    c = __fmaf_rn(a[g].y, c, b[g].y);
                    c = __fmaf_rn(a[g].z, c, b[g].z);
                    c = __fmaf_rn(a[g].w, c, b[g].w);
                    if (g & 1)   // chunk k0 + i0 + 4g + 3 ends a group of eight
                        st_relaxed_gpu_u64(cwc + (size_t)(((k0 + i0) >> 3) + (g >> 1)) * LB_NC, hi | __float_as_uint(c));
                }
            } else {
                // the sequence's last, partial batch: one chunk at a time
                for (int i = i0; i < cnt; ++i) {
                    const int o = ((i >> 2) * LB_NC + lane) * 4 + (i & 3);
                    c = __fmaf_rn(fA[o], c, fB[o]);
                    if (((k0 + i) & 7) == 7)
                        st_relaxed_gpu_u64(cwc + (size_t)((k0 + i) >> 3) * LB_NC, hi | __float_as_uint(c));
                }
            }
        }
        __syncwarp();                                 // the stage is read
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    return true;
}

template <bool GATED>
__global__ void __launch_bounds__(LB_THREADS, 2)
scan_fused(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
           const __grid_constant__ FusedParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    // [FU_STAGES] tiles (a chain CTA: its ring) | barriers
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + FU_RING);
    __shared__ float4 wA[8][8], wB[8][8];
    __shared__ float carry[LB_NC], cfin[LB_NC];
    __shared__ uint32_t s_epoch;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = lane & 7;

    if (tid == 0) {
        for (int s = 0; s < FU_NBAR; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
        const uint32_t last = *reinterpret_cast<volatile const uint32_t*>(&p.st->lb_epoch);
        s_epoch = last + 1 >= FU_EPOCH_WRAP ? 1u : last + 1;
    }
    __syncthreads();
    Launch L;
    L.p = &p;
    L.epoch = s_epoch;
    L.tag = L.epoch << 2;

    if ((int)blockIdx.x < p.nbcb) {
        // ------------------------------------------------ chain CTA of column blockIdx.x
        float* ring = reinterpret_cast<float*>(smem);
        uint64_t* full = bar + FU_STAGES;             // [FU_NS][FU_NB] a batch of aggregates is in the ring
        uint64_t* empty = full + FU_NS * FU_NB;       // [FU_NS] a block is folded
        if (warp >= 2) {
            if (!chain_poll(p, L, blockIdx.x, warp - 2, lane, ring, full, empty) && lane == 0) L.give_up(9);
            return;
        }
        if (warp == 1) return;   // (no part in a chain)
        if (!chain_fold(p, L, blockIdx.x, lane, ring, full, empty) && lane == 0) L.give_up(5);
        if (lane == 0) L.finish();
        return;
    }

    // ---------------------------------------------------- state CTAs
    const int w = (int)blockIdx.x - p.nbcb, nw = (int)gridDim.x - p.nbcb;
    const int ni = w < p.ntiles ? (p.ntiles - 1 - w) / nw + 1 : 0;   // tiles w, w + nw, ... (chunk order)
    const int nm = (p.nchunks + 7) >> 3;
    const unsigned long long hi_a = (unsigned long long)(L.tag | FU_AGG) << 32;
    const unsigned long long hi_c = (unsigned long long)(L.tag | (p.poison ? 1u : FU_CARRY)) << 32;
    float* bufs = reinterpret_cast<float*>(smem);
    auto coords = [&](int i, int& k, int& bi, int& cb) {
        const int ti = w + i * nw;
        k = ti / p.nbcb;
        const int r = ti - k * p.nbcb;
        bi = r / p.ncb;
        cb = r - bi * p.ncb;
    };
    int issued = 0;                                   // tiles whose loads thread 0 has issued
    auto issue = [&](int i) {
        int k, bi, cb;
        coords(i, k, bi, cb);
        const int buf = i % FU_STAGES;
        mbar_arrive_expect_tx(&bar[buf], LB_TILE_BYTES);
        float* dst = bufs + buf * 2 * LB_TILE;
        tma_load_3d(dst, &map_a, &bar[buf], cb * LB_NC, k * LB_TC, bi);
        tma_load_3d(dst + LB_TILE, &map_b, &bar[buf], cb * LB_NC, k * LB_TC, bi);
        issued = i + 1;
    };
    // tile i's local scan; warp 0 publishes its aggregate and keeps it (CA, CB)
    auto scan_publish = [&](int i, float4& EA, float4& EB, float& CA, float& CB) {
        const int buf = i % FU_STAGES;
        if (!__syncthreads_and(mbar_wait(&bar[buf], (uint32_t)(i / FU_STAGES) & 1, p.wait_ns))) return false;
        int k, bi, cb;
        coords(i, k, bi, cb);
        const float* sa = bufs + buf * 2 * LB_TILE;
        tile_local_scan<GATED>(sa, sa + LB_TILE, min(LB_TC, p.T - k * LB_TC), wA, wB, EA, EB);
        if (warp == 0) {
            tile_aggregate(wA, wB, lane, CA, CB);
            const size_t col = (size_t)bi * p.ncb + cb;
            st_relaxed_gpu_v2u64(p.aw + ((col * p.nchunks + k) * LB_NC + lane) * 2, hi_a | __float_as_uint(CA),
                                 hi_a | __float_as_uint(CB));
        }
        return true;
    };
    // C_{k-1} of tile (col, k), for warp 0 (lane = channel): the published
    // carry entering chunk 8m (the initial carry for m = 0), then the
    // aggregates of chunks 8m .. k - 1 folded in order, as the chain folds
    // them.  All words are read at once, and again until each is tagged.
    auto incoming = [&](size_t col, int k, bool& got) {
        const int m = k >> 3, r = k & 7;
        const unsigned long long* csrc =
            m == 0 ? p.cw0 + col * LB_NC + lane : p.cw8 + (col * nm + (m - 1)) * LB_NC + lane;
        const unsigned long long* asrc = p.aw + ((col * p.nchunks + 8 * m) * LB_NC + lane) * 2;
        auto untagged = [&](const ulonglong2& a) { return (a.x & FU_HI) != hi_a || (a.y & FU_HI) != hi_a; };
        unsigned long long cv = ld_relaxed_gpu_u64(csrc);
        ulonglong2 av[7];
#pragma unroll
        for (int u = 0; u < 7; ++u)
            av[u] = u < r ? ld_relaxed_gpu_v2u64(asrc + u * LB_NC * 2) : make_ulonglong2(hi_a, hi_a);
        auto pending = [&]() {
            bool any = (cv & FU_HI) != hi_c;
#pragma unroll
            for (int u = 0; u < 7; ++u) any |= untagged(av[u]);
            return any;
        };
        got = true;
        if (__any_sync(0xffffffffu, pending())) {
            const uint64_t tw = global_ns();
            uint64_t next = tw + FU_ABORT_NS;
            do {
                if (__any_sync(0xffffffffu, L.expired(tw, next))) {
                    got = false;
                    return 0.f;
                }
                __nanosleep(64);                      // back off: a chain CTA may share this SM
                if ((cv & FU_HI) != hi_c) cv = ld_relaxed_gpu_u64(csrc);
#pragma unroll
                for (int u = 0; u < 7; ++u)
                    if (untagged(av[u])) av[u] = ld_relaxed_gpu_v2u64(asrc + u * LB_NC * 2);
            } while (__any_sync(0xffffffffu, pending()));
        }
        float cin = lo_f(cv);
#pragma unroll
        for (int u = 0; u < 7; ++u)
            if (u < r) cin = __fmaf_rn(lo_f(av[u].x), cin, lo_f(av[u].y));
        return cin;
    };

    const float4 one4 = make_float4(1.f, 1.f, 1.f, 1.f), zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 EA0 = one4, EB0 = zero4, EA1 = one4, EB1 = zero4;
    float CA0 = 1.f, CB0 = 0.f, CA1 = 1.f, CB1 = 0.f;
    int failed = -1;                                  // the tile whose load wait gave up
    // every CTA's first tile is requested alone, so the first tiles of all
    // CTAs (the chains' first chunks) land before the rest of the ring's loads
    if (tid == 0 && ni > 0) issue(0);
    if (ni > 0 && !scan_publish(0, EA0, EB0, CA0, CB0)) failed = 0;
    if (tid == 0 && failed < 0)
        while (issued < min(ni, FU_STAGES)) issue(issued);
    for (int i = 0; failed < 0 && i < ni; ++i) {
        // the next tile's aggregate goes out before this tile's carry is awaited
        if (i + 1 < ni && !scan_publish(i + 1, EA1, EB1, CA1, CB1)) {
            failed = i + 1;
            break;
        }
        int k, bi, cb;
        coords(i, k, bi, cb);
        const int t0 = k * LB_TC, n0 = cb * LB_NC;
        if (warp == 0) {
            bool got;
            const float cin = incoming((size_t)bi * p.ncb + cb, k, got);
            if (!got && lane == 0) L.give_up(7);
            const float Ck = __fmaf_rn(CA0, cin, CB0);
            carry[lane] = cin;
            cfin[lane] = Ck;
            const int n = n0 + lane;
            if (k == p.nchunks - 1 && p.s_final != nullptr && n < p.N) p.s_final[(size_t)bi * p.N + n] = Ck;
        }
        __syncthreads();
        const float* sa = bufs + (i % FU_STAGES) * 2 * LB_TILE;
        tile_outputs<GATED>(sa, sa + LB_TILE, min(LB_TC, p.T - t0), carry, cfin, EA0, EB0,
                            p.s_out + ((size_t)bi * p.T + t0) * p.N + n0, p.N,
                            p.s_out != nullptr && n0 + 4 * quad < p.N);
        __syncthreads();                              // stage i % FU_STAGES is free
        if (tid == 0 && issued < ni) issue(issued);   // tile i + FU_STAGES
        EA0 = EA1;
        EB0 = EB1;
        CA0 = CA1;
        CB0 = CB1;
    }
    if (failed >= 0 && tid == 0) {
        L.give_up(6);
        // the tile loads still in flight land before the CTA leaves
        for (int j = failed; j < issued; ++j)
            (void)mbar_wait(&bar[j % FU_STAGES], (uint32_t)(j / FU_STAGES) & 1, p.wait_ns);
    }
    if (tid == 0) L.finish();
}

}  // namespace

// The fused path runs for eight chunks or more (shorter scans take the
// reduce-then-scan launches, which give the same bits).
bool scan_fused_applies(int T) { return (T + LB_TC - 1) / LB_TC >= 8; }

// Workspace of the fused path, all of it tagged words: the carries ending
// each group of eight chunks (8 bytes per channel and group, allocated as 256
// bytes per group of four chunks and column), the aggregates (16 bytes per
// chunk and channel, chunks padded to groups of four), the initial carries
// (8 bytes per channel of each column).
namespace {
struct FusedLayout {
    int64_t cw8, aw, cw0, total;   // byte offsets and the size
};
FusedLayout fused_layout(int B, int T, int N) {
    const int64_t ncb = (N + LB_NC - 1) / LB_NC, nbcb = (int64_t)B * ncb;
    const int64_t nq = chunk_quads((T + LB_TC - 1) / LB_TC);
    FusedLayout l;
    l.cw8 = 0;
    l.aw = nbcb * nq * 256;
    l.cw0 = l.aw + nbcb * nq * 4 * LB_NC * 16;
    l.total = l.cw0 + nbcb * LB_NC * 8;
    return l;
}
}  // namespace

int64_t scan_fused_ws_bytes(int B, int T, int N) { return fused_layout(B, T, N).total; }

// the tagged words' bytes [a, a + b), which a change of geometry clears
void scan_fused_tag_area(int B, int T, int N, int64_t* a, int64_t* b) {
    *a = 0;
    *b = fused_layout(B, T, N).total;
}

cudaError_t launch_scan_fused(const ScanArgs& x, bool gated, void* ws, int poison, SnDevStatus* st,
                              uint64_t wait_ns, int sm_count, cudaStream_t stream, bool* fell_back) {
    *fell_back = false;
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
    const FusedLayout l = fused_layout(x.B, x.T, x.N);
    unsigned char* base = static_cast<unsigned char*>(ws);
    p.cw8 = reinterpret_cast<unsigned long long*>(base + l.cw8);
    p.aw = reinterpret_cast<unsigned long long*>(base + l.aw);
    p.cw0 = reinterpret_cast<unsigned long long*>(base + l.cw0);
    p.st = st;
    p.wait_ns = wait_ns;
    p.poison = poison;

    auto kern = gated ? scan_fused<true> : scan_fused<false>;
    int occ = 0;
    cudaError_t e = occupancy_once((const void*)kern, LB_THREADS, FU_SMEM, &occ);
    if (e != cudaSuccess) return e;
    // every column's chain CTA plus the state CTAs, all resident (cooperative launch)
    const int64_t resident = (int64_t)occ * sm_count;
    const int grid = (int)std::min<int64_t>(resident, p.nbcb + (int64_t)p.ntiles);
    const int64_t nw = grid - p.nbcb;
    // While a tile waits for its carry, every tile up to nw further on has its
    // aggregate out, and the carry needs those up to FU_PB - 2 chunks of its
    // column further on: more columns than that covers (or a grid without
    // room for them) take the reduce-then-scan launches, which give the same bits.
    if (nw < 1 || (nw < p.ntiles && nw <= (int64_t)(FU_PB + 1) * p.nbcb)) {
        *fell_back = true;   // the caller's tagged area now holds the other path's arrays
        return launch_scan_reduce_scan(x, gated, ws, st, wait_ns, sm_count, stream);
    }
    void* args[] = {(void*)&ma, (void*)&mb, (void*)&p};
    e = cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(LB_THREADS), args, FU_SMEM, stream);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace sn
