// recur_delta_chunked.cu -- chunked tensor-core form of the DeltaNet delta rule
//     delta_t = beta_t (v_t - S_{t-1}^T k_t),   S_t = S_{t-1} + k_t delta_t^T,
//     o_t = scale * S_t^T q_t
// ("SunnyNet 工程化实录" §4.2, "我拿同一份权重和 llama.cpp 正面比了一场" §3),
// the T-parallel counterpart of recur_seq<RK_DELTA>.
//
// Within a chunk of C = 128 tokens starting from state S_n, the deltas solve a
// unit lower-triangular system: delta_t = beta_t (v_t - S_n^T k_t -
// sum_{j<t} (k_t . k_j) delta_j).  With L the strictly lower part of K K^T,
//     T = (I + diag(beta) L)^{-1} diag(beta),   W = T K,   U = T V
//     Delta   = U - W S_n                     (the chunk's deltas, C x dv)
//     S_{n+1} = S_n + K^T Delta
//     O       = scale * (Q S_n + tril(Q K^T) Delta)      (j <= t)
// (the WY / UT form of a product of rank-1 updates).  Three launches:
//   delta_prep    one CTA per chunk: the Gram matrix K K^T on tcgen05 with a
//                 hi/lo tf32 split (three products, close to fp32), the
//                 triangular inverse in fp32 on the CUDA cores (16 x 16
//                 diagonal blocks by column-wise substitution in registers,
//                 then doubling levels 16 -> 32 -> 64 -> 128), W = T K and
//                 U = T V on tcgen05; writes W, U and K^T tiles;
//   delta_chain   one CTA per (batch, head), chunks in order: the state S^T
//                 stays in fp32 registers; per chunk the products W S_n and
//                 K^T Delta run on tcgen05 (tf32 operands); the operand tiles
//                 of every chunk's Delta^T and S_n^T leave by bulk stores;
//   chunk_output  the output kernel of the diagonal-decay form with unit
//                 decays (recur_chunked.cu), bulk-loading Delta^T in place of v.
// For longer sequences the chunks are split into segments that run as a
// pipeline on three side streams (launch_delta_chunked), so the chain of one
// segment overlaps the preparation of the next.
// Supported: dk = dv = 128.  Results carry tf32 rounding (about 1e-3
// relative); splits at multiples of 128 tokens are bit-exact because the state
// crosses chunks in fp32.
#include "chunk_common.cuh"
#include "chunk_output.cuh"

#include <algorithm>

namespace sn {
namespace {

using namespace chunk;

constexpr int LDX = CH + 4;         // row stride of A^T and X (rows of float4)
constexpr int BSZ = 16;             // diagonal block size of the inverse
constexpr int SITE_PREP_WAIT1 = 7, SITE_PREP_WAIT2 = 8, SITE_CHAIN_WAIT = 9, SITE_OUT_READY = 10;

struct DeltaArgs {
    int B, T, H, NC;
    int n0, n1;     // chunks [n0, n1) of this launch (a segment of the sequence)
    const float* k;
    const float* v;
    const float* beta;
    float* Wt;      // per chunk: W (rows t, K = key), operand layout, tf32
    float* KTt;     // per chunk: K^T (rows key, K = t), operand layout, tf32
    float* Ut;      // per chunk: U, rows t of 128 values, 16-byte slots swizzled by row (off_u)
    float* DTt;     // per chunk: Delta^T (rows value, K = t), operand layout, tf32
    float* St;      // per chunk: S_n^T (rows value, K = key), operand layout, tf32
    const float* S_from;   // delta_chain: fp32 state entering chunk n0 (NULL = zeros)
    float* S_to;           // delta_chain: fp32 state after chunk n1 - 1 (NULL = not written)
    SnDevStatus* st;
    uint64_t wait_ns;
    int poison;            // fused kernel: the chains wait for a ready value no CTA writes (tests the bound)
};

// Float offset of U[t][i] in a chunk's U tile: rows of 128 values whose
// 16-byte slots are XOR-swizzled by t mod 8 within each 128-byte line, so that
// delta_prep stages a row per thread without bank conflicts and delta_chain
// still reads a row a line at a time.
__device__ __forceinline__ int off_u(int t, int i) {
    return t * 128 + (i & ~31) + ((((i & 31) >> 2) ^ (t & 7)) << 2) + (i & 3);
}

// ------------------------------------------------------------------ delta_prep
struct PrepSmem {
    static constexpr int b0 = 0;                 // K (hi, 128-byte swizzled), then k [t][i], then K^T operand
    static constexpr int b1 = OPF;               // K (lo, swizzled), then v [t][j], then V^T operand
    static constexpr int b2 = 2 * OPF;           // A^T above the diagonal and X = (I + A)^{-1} on and
                                                 // below it (fp32, stride LDX), then T operand, then W
    static constexpr int beta = b2 + CH * LDX;
    static constexpr int misc = beta + CH;       // barriers (products, K tile, v tile), tmem slot
    static constexpr size_t bytes = (size_t)(misc + 16) * 4 + 1024;
};

// One doubling level of the lower-triangular inverse X = (I + A)^{-1}: for
// every 2S x 2S diagonal block, whose two S x S diagonal blocks X_A (upper
// left) and X_D (lower right) are already inverted, the lower-left block is
//     X_C = -X_D (A_C X_A)
// with A_C the matching block of A (read from A^T).  A^T and X share one
// array (A^T strictly above the diagonal, X on and below it), and the product
// Y = A_C X_A is parked over A_C itself, the upper-right S x S block, once
// every thread has read A_C (no later level reads it; X is zero there and the
// T operand masks it).  Every thread owns RT = S / 16 rows x 4
// columns of one pair's block, so all 256 threads work at every level.  The
// sums skip X_A's and X_D's zero triangles in steps of four; the few entries
// past the triangle that a step still touches sit in a diagonal 16 x 16 block
// above its diagonal, where X holds exact zeros.
// Which block of the level a thread owns: pair block at offset o, rows
// RT rt .. RT rt + RT - 1, columns 4 ct .. 4 ct + 3.  The first product's sum
// shortens with ct and the second's lengthens with rt, so for S = 32 and 64
// each product has its own map (Y goes through shared memory in between): a
// warp takes one or two adjacent values of the length-setting index, and the
// warps sharing a scheduler (w, w + 4) take complementary lengths.  Each
// output's sum keeps its order, so the map does not change the results.
template <int S>
__device__ __forceinline__ void level_map(int tid, bool by_rows, int& o, int& rt, int& ct) {
    constexpr int NCT = S / 4;
    const int w = tid >> 5, lane = tid & 31;
    if constexpr (S == 64) {   // one pair block; a warp: one pair of the length-setting index x 16
        const int kp = w < 4 ? w : 11 - w;
        const int key = 2 * kp + (lane >> 4), other = lane & 15;
        o = 0;
        rt = by_rows ? key : other;
        ct = by_rows ? other : key;
    } else if constexpr (S == 32) {   // two pair blocks
        if (!by_rows) {   // a warp: one pair of column groups x 16 row groups of one pair block
            const int kp = w < 4 ? w : 7 - w;
            ct = 2 * kp + (lane >> 4);
            rt = lane & 15;
            o = w < 4 ? 0 : 2 * S;
        } else {          // a half warp: one pair of row groups x 8 column groups of one pair block
            const int kp = w < 4 ? w : 11 - w;
            rt = 2 * kp + ((lane >> 3) & 1);
            ct = lane & 7;
            o = 2 * S * (lane >> 4);
        }
    } else {
        ct = tid % NCT;
        rt = (tid / NCT) % 16;
        o = 2 * S * (tid / (16 * NCT));
    }
}

template <int S>
__device__ __forceinline__ void inverse_level(float* Xm, const float* AT, int tid) {
    constexpr int RT = S / 16;
    int o, rt, ct;
    level_map<S>(tid, false, o, rt, ct);
    int r0 = RT * rt, c0 = 4 * ct;
    float acc[RT][4] = {};
    // Y[r][c] = sum_{m >= c} A[o + S + r][o + m] X[o + m][o + c]
    for (int m = c0; m < S; m += 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 x = ld4(Xm + (o + m + i) * LDX + o + c0);
            const float* ap = AT + (o + m + i) * LDX + o + S + r0;
            float av[RT];
            if constexpr (RT == 4) {
                const float4 t = ld4(ap);
                av[0] = t.x; av[1] = t.y; av[2] = t.z; av[3] = t.w;
            } else if constexpr (RT == 2) {
                const float2 t = *reinterpret_cast<const float2*>(ap);
                av[0] = t.x; av[1] = t.y;
            } else {
                av[0] = ap[0];
            }
#pragma unroll
            for (int j = 0; j < RT; ++j) {
                acc[j][0] = fmaf(av[j], x.x, acc[j][0]); acc[j][1] = fmaf(av[j], x.y, acc[j][1]);
                acc[j][2] = fmaf(av[j], x.z, acc[j][2]); acc[j][3] = fmaf(av[j], x.w, acc[j][3]);
            }
        }
    }
    __syncthreads();   // A_C is read: Y goes over it
#pragma unroll
    for (int j = 0; j < RT; ++j)
        st4(Xm + (o + r0 + j) * LDX + o + S + c0, make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]));
    __syncthreads();
    // X_C[r][c] = -sum_{m <= r} X[o + S + r][o + S + m] Y[m][c]
    level_map<S>(tid, true, o, rt, ct);
    r0 = RT * rt;
    c0 = 4 * ct;
    float out[RT][4] = {};
    for (int m = 0; m < r0 + RT; m += 4) {
        float4 xd[RT];
#pragma unroll
        for (int j = 0; j < RT; ++j) xd[j] = ld4(Xm + (o + S + r0 + j) * LDX + o + S + m);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 y = ld4(Xm + (o + m + i) * LDX + o + S + c0);
#pragma unroll
            for (int j = 0; j < RT; ++j) {
                const float xv = i == 0 ? xd[j].x : i == 1 ? xd[j].y : i == 2 ? xd[j].z : xd[j].w;
                out[j][0] = fmaf(xv, y.x, out[j][0]); out[j][1] = fmaf(xv, y.y, out[j][1]);
                out[j][2] = fmaf(xv, y.z, out[j][2]); out[j][3] = fmaf(xv, y.w, out[j][3]);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < RT; ++j)
        st4(Xm + (o + S + r0 + j) * LDX + o + c0, make_float4(-out[j][0], -out[j][1], -out[j][2], -out[j][3]));
    __syncthreads();
}

// Tiles by TMA: K in the 128-byte-swizzled operand layout for the Gram
// products (four boxes of 32 keys x 128 tokens), then v as a natural
// [token][feature] box; once the inverse is done the threads transpose v and
// K's tf32 part (still in its buffer) into the V^T and K^T operands; W and U
// leave through shared memory by
// bulk copies.  Rows past T read as zeros.  Units are taken chunk by chunk:
// unit u of the segment is chunk n0 + u / (B H) of head-batch u mod (B H).
// Without a queue a CTA takes the units blockIdx.x, blockIdx.x + gridDim.x,
// ..., so that a grid below the SM count leaves SMs free for the kernels
// beside it; with one (the fused kernel) thread 0 claims units from it, and
// once a unit's tiles are written it sets the unit's ready word.  The next
// unit's K tile is requested as soon as the copies out have read the buffer
// it lands in.
__device__ __forceinline__ void prep_role(const CUtensorMap* map_ks, const CUtensorMap* map_vn, const DeltaArgs& a,
                                          unsigned* queue, unsigned* ready) {
    extern __shared__ unsigned char smem_raw[];
    using L = PrepSmem;
    float* base = reinterpret_cast<float*>(smem_align<1024>(smem_raw));
    float* buf0 = base + L::b0;
    float* buf1 = base + L::b1;
    float* buf2 = base + L::b2;
    float* beta_s = base + L::beta;
    uint64_t* bar = reinterpret_cast<uint64_t*>(base + L::misc);
    uint32_t* slot = reinterpret_cast<uint32_t*>(base + L::misc + 2);
    uint64_t* barK = reinterpret_cast<uint64_t*>(base + L::misc + 4);    // the swizzled K tile
    uint64_t* barT = reinterpret_cast<uint64_t*>(base + L::misc + 6);    // the natural v tile
    int* s_next = reinterpret_cast<int*>(base + L::misc + 8);            // the next unit (thread 0 writes)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int BH = a.B * a.H;
    const int units = BH * (a.n1 - a.n0);
    struct Unit {
        int h, b, t0, nval;
        size_t row0, tile, word;
    };
    auto unit = [&](int u) {
        Unit c;
        const int bh = u % BH, n = a.n0 + u / BH;
        c.h = bh % a.H;
        c.b = bh / a.H;
        c.t0 = n * CH;
        c.nval = min(CH, a.T - c.t0);
        c.row0 = (size_t)c.b * a.T + c.t0;
        c.word = (size_t)bh * a.NC + n;
        c.tile = c.word * (size_t)OPF;
        return c;
    };
    auto next_unit = [&](int u) -> int {   // thread 0
        if (queue != nullptr) {
            const unsigned v = atomicAdd(queue, 1u);
            return v < (unsigned)units ? (int)v : -1;
        }
        return u + (int)gridDim.x < units ? u + (int)gridDim.x : -1;
    };
    auto issue_k = [&](const Unit& c) {   // thread 0: K rows in the swizzled operand layout (rows t, K = key)
        mbar_arrive_expect_tx(barK, OPF * 4);
#pragma unroll
        for (int at = 0; at < DKC / 32; ++at) tma_load_3d(buf0 + at * 4096, map_ks, barK, c.h * DKC + 32 * at, c.t0, c.b);
    };
    int k_loads = 0, t_loads = 0;   // thread 0: K tiles and k, v tile pairs requested
    int64_t pending = -1;           // thread 0: the ready word of the last unit whose tiles left
    auto publish = [&]() {          // thread 0: the tiles are written, then the word (gpu-scope release)
        if (pending < 0) return;
        bulk_wait_all();
        fence_proxy_async_global();
        st_release_gpu(ready + pending, 1u);
        pending = -1;
    };

    if (warp == 0) tc::tmem_alloc_keep(slot, 256);
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(barK, 1);
        mbar_init(barT, 1);
        fence_mbar_init();
        const int u0 = queue != nullptr ? next_unit(-1) : ((int)blockIdx.x < units ? (int)blockIdx.x : -1);
        if (u0 >= 0) {
            issue_k(unit(u0));
            ++k_loads;
        }
        *s_next = u0;
    }
    tc::fence_before_sync();
    __syncthreads();   // the barriers are initialised before any thread polls them
    tc::fence_after_sync();
    const uint32_t tmem = *slot;
    const int tl = lane & 7, ic = 16 * warp + 4 * (lane >> 3);
    const int lq = warp & 3, hf = warp >> 2;
    const int tr = 32 * lq + lane;                           // tensor-memory row of this thread
    const uint32_t lane_base = tmem + ((uint32_t)(32 * lq) << 16);
    bool ok = true;
    int site = SITE_PREP_WAIT1;
    for (int u = *s_next, it = 0; u >= 0; ++it) {
        const Unit c = unit(u);
        const uint32_t ph = (uint32_t)it & 1;
        if (tid < CH) beta_s[tid] = tid < c.nval ? __ldg(a.beta + (c.row0 + tid) * a.H + c.h) : 0.f;
        // thread 0: the last unit's W and U copies out have read the buffers
        // this unit fills (they drain while this unit's K tile arrives)
        if (tid == 0) bulk_wait_read_all();
        ok = __syncthreads_and(mbar_wait(barK, ph, a.wait_ns));
        if (!ok) break;
        if (tid == 0) *s_next = next_unit(u);   // read by every thread at the end of the unit

        // K = hi + lo, both tf32: K K^T ~ hi hi^T + hi lo^T + lo hi^T (elementwise,
        // so the split keeps the swizzled layout)
        for (int f = tid; f < OPF / 4; f += NT) {
            const float4 x = ld4(buf0 + 4 * f);
            const float4 hi = tf32x4(x);
            st4(buf0 + 4 * f, hi);
            st4(buf1 + 4 * f, tf32x4(x.x - hi.x, x.y - hi.y, x.z - hi.z, x.w - hi.w));
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (tid == 0) {
            const uint32_t id = tc::idesc_tf32(128, 128);
            tc::gemm_tf32_sw_sw(tmem, buf0, buf0, id, false);
            tc::gemm_tf32_sw_sw(tmem, buf0, buf1, id, true);
            tc::gemm_tf32_sw_sw(tmem, buf1, buf0, id, true);
            tc::commit(bar);
        }
        ok = __syncthreads_and(mbar_wait(bar, 0, a.wait_ns));
        tc::fence_after_sync();
        if (!ok) break;
        // the natural v tile can stream in now (the Gram products have read
        // the lo part of K, whose buffer it takes) while the inverse runs; the last
        // unit's tiles, stored a few microseconds ago, are published (waiting
        // for them at the end of that unit stalled the CTA)
        if (tid == 0) {
            publish();
            ++t_loads;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(barT, OPF * 4);
            tma_load_3d(buf1, map_vn, barT, c.h * 128, c.t0, c.b);
        }
        // A = diag(beta) strict_lower(K K^T) in fp32, stored transposed: AT[j][t] = A[t][j]
        // (zeros on and below the diagonal, where X goes next)
        float* AT = buf2;
        float* Xm = buf2;
        const float bt = beta_s[tr];
#pragma unroll
        for (int j0 = 64 * hf; j0 < 64 * hf + 64; j0 += 16) {
            float x[16];
            tc::ld16(lane_base + j0, x);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) AT[(j0 + jj) * LDX + tr] = j0 + jj < tr ? bt * x[jj] : 0.f;
        }
        __syncthreads();

        // diagonal blocks of X = (I + A)^{-1}, warp w -> block w, in registers: a
        // lane holds column c of rows rb, rb + 2, ..., and column by column
        // X[r][c] -= A[r][m] X[m][c] for r > m once X[m][c] is final
        {
            const int r0 = BSZ * warp, c = lane & 15, rb = lane >> 4;
            float xr[BSZ / 2];
#pragma unroll
            for (int jj = 0; jj < BSZ / 2; ++jj) xr[jj] = (rb + 2 * jj == c) ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < BSZ - 1; ++m) {
                const float xm = __shfl_sync(FULL, xr[m >> 1], (m & 1) * 16 + c);
#pragma unroll
                for (int jj = 0; jj < BSZ / 2; ++jj) {
                    const int r = rb + 2 * jj;
                    if (r > m) xr[jj] = fmaf(-AT[(r0 + m) * LDX + r0 + r], xm, xr[jj]);
                }
            }
            __syncwarp();   // the block's A^T entries are read: its X (zeros above the diagonal) goes over them
#pragma unroll
            for (int jj = 0; jj < BSZ / 2; ++jj) Xm[(r0 + rb + 2 * jj) * LDX + r0 + c] = xr[jj];
        }
        __syncthreads();
        // the inverse by doubling, 16 -> 32 -> 64 -> 128 (one product pair per level)
        inverse_level<16>(Xm, AT, tid);
        inverse_level<32>(Xm, AT, tid);
        inverse_level<64>(Xm, AT, tid);

        // T = X diag(beta) as the tf32 operand (rows t, K = j), in place through registers
        float4 tv[CH / 8];
#pragma unroll
        for (int tb = 0; tb < CH / 8; ++tb) {
            const int t = 8 * tb + tl;
            // blocks right of the diagonal block are never written: X is zero there
            if ((ic >> 4) > (t >> 4)) {
                tv[tb] = make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
                const float4 x4 = ld4(Xm + t * LDX + ic), b4 = ld4(beta_s + ic);
                tv[tb] = tf32x4(x4.x * b4.x, x4.y * b4.y, x4.z * b4.z, x4.w * b4.w);
            }
        }
        __syncthreads();
#pragma unroll
        for (int tb = 0; tb < CH / 8; ++tb) st4(buf2 + off128(8 * tb + tl, ic), tv[tb]);

        // K^T and V^T, rounded, from K's tf32 part and the natural v tile:
        // thread = feature column i, a half of the tokens, through registers
        ok = __syncthreads_and(mbar_wait(barT, ph, a.wait_ns));
        if (!ok) break;
        {
            const int i = tid & 127, tb0 = (CH / 2) * (tid >> 7);
            float kr[CH / 2], vr[CH / 2];
#pragma unroll
            for (int r = 0; r < CH / 2; ++r) {
                kr[r] = buf0[off_sw(tb0 + r, i)];   // K's hi part: tf32(k) itself
                vr[r] = buf1[(tb0 + r) * 128 + i];
            }
            __syncthreads();
#pragma unroll
            for (int t4 = 0; t4 < CH / 8; ++t4) {
                st4(buf0 + off128(i, tb0 + 4 * t4), tf32x4(kr[4 * t4], kr[4 * t4 + 1], kr[4 * t4 + 2], kr[4 * t4 + 3]));
                st4(buf1 + off128(i, tb0 + 4 * t4), tf32x4(vr[4 * t4], vr[4 * t4 + 1], vr[4 * t4 + 2], vr[4 * t4 + 3]));
            }
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (tid == 0) {
            const uint32_t id = tc::idesc_tf32(128, 128);
            tc::gemm_tf32(tmem, buf2, buf0, CH, id, false);          // W = T K   (cols 0..127)
            tc::gemm_tf32(tmem + 128, buf2, buf1, CH, id, false);    // U = T V   (cols 128..255)
            tc::commit(bar);
        }
        ok = __syncthreads_and(mbar_wait(bar, 1, a.wait_ns));
        tc::fence_after_sync();
        if (!ok) {
            site = SITE_PREP_WAIT2;
            break;
        }
        // W and U through shared memory (the T and V^T operands are
        // consumed) and out by bulk copies, with the K^T operand as it
        // stands (tf32) for the chain
#pragma unroll
        for (int i0 = 64 * hf; i0 < 64 * hf + 64; i0 += 16) {
            float x[16];
            tc::ld16(lane_base + i0, x);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                st4(buf2 + off128(tr, i0 + 4 * q), make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]));
            tc::ld16(lane_base + 128 + i0, x);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                st4(buf1 + off_u(tr, i0 + 4 * q), make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]));
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            // The copy engine works in order: K^T first, then the next unit's
            // K tile into its buffer as soon as it is read, then W.  U (staged
            // in its global layout) leaves by the threads' own 16-byte stores
            // meanwhile, beside the copy engine.
            bulk_store(a.KTt + c.tile, buf0, OPF * 4);
            bulk_commit();
            const int un = *s_next;
            if (un >= 0) {
                bulk_wait_read_all();
                issue_k(unit(un));
                ++k_loads;
            }
            bulk_store(a.Wt + c.tile, buf2, OPF * 4);
            bulk_commit();
            if (ready != nullptr) pending = (int64_t)c.word;
        }
        {
            float4* ug = reinterpret_cast<float4*>(a.Ut + c.tile);
            const float4* us = reinterpret_cast<const float4*>(buf1);
#pragma unroll 4
            for (int f = tid; f < OPF / 4; f += NT) ug[f] = us[f];
        }
        u = *s_next;
    }
    if (!ok && tid == 0) {
        record_error(a.st, SN_E_TIMEOUT, (SN_K_RECUR_CHUNK << 16) | site);
        // the tiles still in flight land before the CTA leaves (a phase
        // already waited for passes at once)
        if (k_loads > 0) (void)mbar_wait(barK, (uint32_t)(k_loads - 1) & 1, a.wait_ns);
        if (t_loads > 0) (void)mbar_wait(barT, (uint32_t)(t_loads - 1) & 1, a.wait_ns);
    }
    if (tid == 0) {
        if (ok) publish();   // the last unit's word
        bulk_wait_all();     // every copy out complete before the CTA exits
        mbar_inval(bar);     // the fused kernel's output stage reuses this memory
        mbar_inval(barK);
        mbar_inval(barT);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

__global__ void __launch_bounds__(NT, 1)
delta_prep(const __grid_constant__ CUtensorMap map_ks, const __grid_constant__ CUtensorMap map_vn, const DeltaArgs a) {
    prep_role(&map_ks, &map_vn, a, nullptr, nullptr);
}

// ------------------------------------------------------------------ delta_chain
struct ChainSmem {
    static constexpr int w_off = 0;          // W_n (rows t, K = key)
    static constexpr int kt_off = OPF;       // K_n^T (rows key, K = t)
    static constexpr int su_off = 2 * OPF;   // S_n^T (rows value, K = key), then Delta^T (rows value, K = t)
    static constexpr int misc = 3 * OPF;
    static constexpr size_t bytes = (size_t)(misc + 16) * 4 + 128;
};

// The chain of head-batch bh over chunks [n0, n1).  With ready words (the
// fused kernel), thread 0 waits, bounded, for a chunk's word before it
// requests the chunk's first tile, and publishes in progress[bh] how many
// chunks have their state and delta tiles written.
__device__ __forceinline__ void chain_role(const DeltaArgs& a, int bh_index, const unsigned* ready,
                                           unsigned* progress) {
    extern __shared__ unsigned char smem_raw[];
    using L = ChainSmem;
    float* base = align128(smem_raw);
    float* Wb = base + L::w_off;
    float* KTb = base + L::kt_off;
    float* SUb = base + L::su_off;
    uint64_t* barW = reinterpret_cast<uint64_t*>(base + L::misc);
    uint64_t* barK = reinterpret_cast<uint64_t*>(base + L::misc + 2);
    uint64_t* barM = reinterpret_cast<uint64_t*>(base + L::misc + 4);
    uint32_t* slot = reinterpret_cast<uint32_t*>(base + L::misc + 6);
    int* s_ok = reinterpret_cast<int*>(base + L::misc + 8);   // thread 0: the first chunk's tiles were requested

    const int tid = threadIdx.x, warp = tid >> 5;
    const size_t bh = (size_t)bh_index;
    const int c = tid & 127, part = tid >> 7;     // value column, half of the keys / tokens
    const int lq = warp & 3;                      // tensor-memory lanes 32 lq .. : rows c
    const int NC = a.NC;
    auto tile = [&](const float* p, int n) { return p + (bh * NC + n) * (size_t)OPF; };
    auto wait_ready = [&](int n) -> bool {   // thread 0: chunk n's W, K^T and U tiles are written
        if (ready == nullptr) return true;
        const uint32_t* w = ready + bh * NC + n;
        const uint32_t want = a.poison ? 2u : 1u;   // poisoned: a value no CTA writes (tests the bound)
        if (ld_acquire_gpu(w) != want) {
            const uint64_t t0 = global_ns();
            while (ld_acquire_gpu(w) != want)
                if (global_ns() - t0 > a.wait_ns) return false;
        }
        fence_proxy_async_global();   // the bulk copies that follow read what the flag published
        return true;
    };
    int w_loads = 0, k_loads = 0;   // bulk loads issued on barW / barK (thread 0's count)

    if (warp == 0) tc::tmem_alloc_keep(slot, 256);
    if (tid == 0) {
        mbar_init(barW, 1);
        mbar_init(barK, 1);
        mbar_init(barM, 1);
        fence_mbar_init();
        const bool r0 = wait_ready(a.n0);
        if (r0) {
            mbar_arrive_expect_tx(barW, OPF * 4);
            bulk_load(Wb, tile(a.Wt, a.n0), OPF * 4, barW);
            mbar_arrive_expect_tx(barK, OPF * 4);
            bulk_load(KTb, tile(a.KTt, a.n0), OPF * 4, barK);
            w_loads = k_loads = 1;
        }
        *s_ok = r0 ? 1 : 0;
    }

    // S^T[c][i] for this part's 64 keys, fp32 in registers for the whole sequence
    float sreg[64];
    const size_t sbase = bh * (size_t)(DKC * 128);
#pragma unroll
    for (int r = 0; r < 64; ++r) sreg[r] = a.S_from != nullptr ? a.S_from[sbase + (size_t)(64 * part + r) * 128 + c] : 0.f;
    auto put_state = [&]() {   // tf32 S_n^T into the operand buffer (then bulk-stored as the chunk's tile)
#pragma unroll
        for (int r4 = 0; r4 < 16; ++r4) {
            const int i = 64 * part + 4 * r4;
            st4(SUb + off128(c, i), tf32x4(sreg[4 * r4], sreg[4 * r4 + 1], sreg[4 * r4 + 2], sreg[4 * r4 + 3]));
        }
    };
    auto store_tile = [&](float* tiles, int n) {   // thread 0: the operand buffer -> a chunk's tile
        bulk_store(tiles + (bh * NC + n) * (size_t)OPF, SUb, OPF * 4);
        bulk_commit();
    };
    float u[64];
    auto load_u = [&](int n) {
        const float* ut = tile(a.Ut, n);
#pragma unroll
        for (int r = 0; r < 64; ++r) u[r] = ut[off_u(64 * part + r, c)];
    };
    put_state();
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    bool ok = *s_ok != 0;
    if (ok) load_u(a.n0);
    if (tid == 0) store_tile(a.St, a.n0);
    const uint32_t tmem = *slot;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * lq) << 16);
    const uint32_t id = tc::idesc_tf32(128, 128);
    uint32_t mpar = 0;
    for (int n = a.n0; ok && n < a.n1; ++n) {
        const uint32_t ph = (uint32_t)(n - a.n0) & 1;   // phase of this launch's n-th tile loads
        ok = __syncthreads_and(mbar_wait(barW, ph, a.wait_ns));
        if (!ok) break;
        if (tid == 0) {   // P[c][t] = sum_i S^T[c][i] W[t][i]  (= (W S_n)^T)
            tc::gemm_tf32(tmem, SUb, Wb, DKC, id, false);
            tc::commit(barM);
            bulk_wait_read_all();   // the S_n tile store has read the buffer the deltas overwrite
            if (progress != nullptr && n > a.n0 + 1 && ((n - 1 - a.n0) & 3) == 0) {
                // every copy but the two newest (Delta_{n-1}, S_n) is complete:
                // chunks before n - 1 have their tiles (issued microseconds ago,
                // so this wait does not hold up the chain); every fourth chunk,
                // since the release is thread 0's, which issues the products
                bulk_wait_allbut2();
                fence_proxy_async_global();
                st_release_gpu(progress + bh, (uint32_t)(n - 1));
            }
        }
        ok = __syncthreads_and(mbar_wait(barM, mpar, a.wait_ns));
        mpar ^= 1;
        tc::fence_after_sync();
        if (!ok) break;
        bool rdy = true;   // thread 0: the next chunk's tiles exist
        if (tid == 0 && n + 1 < a.n1) {
            rdy = wait_ready(n + 1);
            if (rdy) {
                mbar_arrive_expect_tx(barW, OPF * 4);
                bulk_load(Wb, tile(a.Wt, n + 1), OPF * 4, barW);
                ++w_loads;
            }
        }
        // Delta^T[c][t] = U[t][c] - P[c][t] for this part's tokens
#pragma unroll
        for (int q0 = 0; q0 < 64; q0 += 16) {
            float x[16];
            tc::ld16(lane_base + 64 * part + q0, x);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) x[jj] = u[q0 + jj] - x[jj];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                st4(SUb + off128(c, 64 * part + q0 + 4 * q),
                    tf32x4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]));
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
        ok = __syncthreads_and(rdy && mbar_wait(barK, ph, a.wait_ns));
        tc::fence_after_sync();
        if (!ok) break;
        if (tid == 0) {   // D[c][i] = sum_t Delta^T[c][t] K^T[i][t]  (= (K^T Delta)^T)
            tc::gemm_tf32(tmem + 128, SUb, KTb, CH, id, false);
            tc::commit(barM);
            store_tile(a.DTt, n);
        }
        if (n + 1 < a.n1) load_u(n + 1);
        if (tid == 0) bulk_wait_read_all();   // the Delta^T tile store has read the buffer
        ok = __syncthreads_and(mbar_wait(barM, mpar, a.wait_ns));
        mpar ^= 1;
        tc::fence_after_sync();
        if (!ok) break;
        if (tid == 0 && n + 1 < a.n1) {
            mbar_arrive_expect_tx(barK, OPF * 4);
            bulk_load(KTb, tile(a.KTt, n + 1), OPF * 4, barK);
            ++k_loads;
        }
#pragma unroll
        for (int q0 = 0; q0 < 64; q0 += 16) {
            float x[16];
            tc::ld16(lane_base + 128 + 64 * part + q0, x);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) sreg[q0 + jj] += x[jj];
        }
        if (n + 1 < a.n1) put_state();
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (tid == 0 && n + 1 < a.n1) store_tile(a.St, n + 1);
    }
    if (tid == 0) {
        bulk_wait_all();   // every tile store complete before the CTA exits
        if (ok && progress != nullptr) {
            fence_proxy_async_global();
            st_release_gpu(progress + bh, (uint32_t)a.n1);
        }
    }
    if (!ok) {
        if (tid == 0) {
            record_error(a.st, SN_E_TIMEOUT, (SN_K_RECUR_CHUNK << 16) | SITE_CHAIN_WAIT);
            // let copies still in flight land before the CTA exits
            if (w_loads > 0) mbar_wait(barW, (w_loads - 1) & 1, a.wait_ns);
            if (k_loads > 0) mbar_wait(barK, (k_loads - 1) & 1, a.wait_ns);
        }
    } else if (a.S_to != nullptr) {
#pragma unroll
        for (int r = 0; r < 64; ++r) a.S_to[sbase + (size_t)(64 * part + r) * 128 + c] = sreg[r];
    }
    if (tid == 0) {   // the fused kernel's output stage reuses this memory
        mbar_inval(barW);
        mbar_inval(barK);
        mbar_inval(barM);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

__global__ void __launch_bounds__(NT, 1) delta_chain(const DeltaArgs a) {
    chain_role(a, blockIdx.x, nullptr, nullptr);
}

// Output units of the fused kernel, chunk by chunk (all heads of chunk 0,
// then chunk 1, ...), claimed from a counter; a unit's tiles may be read once
// its chain's progress word has passed the unit's chunk.  A wait gives up
// after the limit, or at once when an error is already recorded.
struct QueueUnits {
    int units, BH;
    unsigned* queue;
    const unsigned* progress;
    static constexpr bool kDynamic = true;
    __device__ int claim() const {
        const unsigned v = atomicAdd(queue, 1u);
        return v < (unsigned)units ? (int)v : -1;
    }
    __device__ int first() const { return claim(); }
    __device__ int next(int) const { return claim(); }
    __device__ ChunkIdx index(const ChunkArgs& a, int u) const {
        ChunkIdx c;
        const int bh = u % BH;
        c.n = u / BH;
        c.h = bh % a.H;
        c.b = bh / a.H;
        c.g = c.h / (a.H / a.G);
        c.t0 = c.n * CH;
        c.nval = min(CH, a.T - c.t0);
        c.bh = (size_t)bh;
        return c;
    }
    __device__ bool ready(const ChunkArgs& a, const ChunkIdx& c) const {
        const uint32_t* w = progress + c.bh;
        const uint32_t need = (uint32_t)c.n + 1;
        if (ld_acquire_gpu(w) < need) {
            const uint64_t t0 = global_ns();
            while (ld_acquire_gpu(w) < need) {
                if (*reinterpret_cast<volatile const int*>(&a.st->error) != 0 || global_ns() - t0 > a.wait_ns) {
                    record_error(a.st, SN_E_TIMEOUT, (SN_K_RECUR_CHUNK << 16) | SITE_OUT_READY);
                    return false;
                }
            }
        }
        fence_proxy_async_global();   // the bulk copies that follow read what the word published
        return true;
    }
};

// ------------------------------------------------------------------ delta_fused
// The whole call in one cooperative launch.  CTAs 0 .. B H - 1 run the chains
// over the whole sequence; the others claim preparation units chunk by chunk
// from ctrl[0] and set a unit's ready word (ctrl[2 + bh NC + n]) once its
// tiles are written; a chain publishes in its progress word (after the ready
// words) how many chunks have their state and delta tiles written.  Every CTA
// then claims output units from ctrl[1], chunk by chunk, and computes each
// once its chain's progress has passed it.  Preparation units wait on nothing
// but their own copies, every one is claimed before any output unit, chains
// wait only on ready words and every CTA is resident, so every wait ends
// (each is bounded all the same).  The arithmetic of every unit and chain
// step is the pipeline's, so the bits are too.
__global__ void __launch_bounds__(NT, 1)
delta_fused(const __grid_constant__ CUtensorMap map_ks, const __grid_constant__ CUtensorMap map_vn,
            const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
            const __grid_constant__ CUtensorMap map_o, const DeltaArgs a, const ChunkArgs oc, unsigned* ctrl) {
    const int BH = a.B * a.H;
    unsigned* ready = ctrl + 2;
    unsigned* progress = ready + (size_t)BH * a.NC;
    if ((int)blockIdx.x < BH)
        chain_role(a, blockIdx.x, ready, progress);
    else
        prep_role(&map_ks, &map_vn, a, ctrl, ready);
    if (oc.o != nullptr) {
        QueueUnits sch{BH * a.NC, BH, ctrl + 1, progress};
        output_loop<false, 128>(&map_q, &map_k, &map_o, oc, sch);
    }
}

int64_t round256(int64_t x) { return (x + 255) / 256 * 256; }

}  // namespace

int64_t delta_chunked_ws_bytes(int B, int T, int H, int dk, int dv) {
    const int64_t nc = (T + CH - 1) / CH;
    return 5 * round256((int64_t)B * H * nc * dk * dv * 4) + round256((int64_t)B * H * dk * dv * 4) +
           round256((2 + (int64_t)B * H * (nc + 1)) * 4);
}

bool delta_chunked_supported(const RecurArgs& x) { return x.kind == RK_DELTA && x.dk == DKC && x.dv == 128; }

// Auto: when the chain (one CTA per head) leaves at least half the SMs to
// the other stages, three segments from 12 chunks on and two from 8; more
// segments measured slower (each adds a chain launch, its setup and a slower
// first chunk, about 15 us, to the serial path).
int delta_segments(int NC, int BH, int sm_count, int requested) {
    const bool room = 2 * BH <= sm_count;
    int nseg = requested > 0 ? requested : (room && NC >= 12 ? 3 : room && NC >= 8 ? 2 : 1);
    nseg = std::min(nseg, NC);
    const int len = (NC + nseg - 1) / nseg;
    return (NC + len - 1) / len;
}

// First chunk of segment g (g = nseg: NC).  Three segments split about
// 5 : 7 : 4: a short first segment starts the chain early, a short last one
// leaves little output after it, and the middle one's preparation hides
// behind the first chain (32 chunks: 10, 14, 8, measured 3 % faster than
// 16, 16).  Otherwise equal lengths.
int delta_seg_start(int NC, int nseg, int g) {
    if (g >= nseg) return NC;
    if (nseg == 3) return g == 0 ? 0 : g == 1 ? (5 * NC + 8) / 16 : (12 * NC + 8) / 16;
    return std::min(NC, g * ((NC + nseg - 1) / nseg));
}

// Segments of the chunk sequence run as a pipeline over three side streams:
// the per-chunk preparation on `pipe.prep`, the chain on `pipe.chain` once
// the segment's tiles exist, and the output on `pipe.out` once the chain has
// produced the segment's deltas and states.  The chain of one segment thus
// runs beside the preparation of the next; the chain stream has the highest
// priority and the output stream the lowest.  The fp32 state crosses
// segments through the workspace, so every segmentation gives the same bits.
// Events order the stages (fork from and join to the caller's stream); no
// kernel waits on another.
cudaError_t launch_delta_chunked(const RecurArgs& x, void* ws, SnDevStatus* st, uint64_t wait_ns, int sm_count,
                                 int segments, bool poison, const DeltaPipe& pipe, cudaStream_t s) {
    DeltaArgs d{};
    d.B = x.B; d.T = x.T; d.H = x.H;
    d.NC = (x.T + CH - 1) / CH;
    d.k = x.k; d.v = x.v; d.beta = x.g;
    const int64_t tile_bytes = round256((int64_t)x.B * x.H * d.NC * OPF * 4);
    char* p = static_cast<char*>(ws);
    d.Wt = reinterpret_cast<float*>(p);
    d.KTt = reinterpret_cast<float*>(p + tile_bytes);
    d.Ut = reinterpret_cast<float*>(p + 2 * tile_bytes);
    d.St = reinterpret_cast<float*>(p + 3 * tile_bytes);
    d.DTt = reinterpret_cast<float*>(p + 4 * tile_bytes);
    float* S_mid = reinterpret_cast<float*>(p + 5 * tile_bytes);
    unsigned* ctrl = reinterpret_cast<unsigned*>(p + 5 * tile_bytes + round256((int64_t)x.B * x.H * DKC * 128 * 4));
    d.st = st;
    d.wait_ns = wait_ns;

    // TMA maps of k (swizzled boxes of 32 keys for the Gram products; K^T is
    // transposed from that tile's tf32 part) and v (natural tile):
    // (B, T, H * 128) row-major
    CUtensorMap mks, mvn;
    {
        const uint64_t dims[3] = {(uint64_t)x.H * DKC, (uint64_t)x.T, (uint64_t)x.B};
        const uint64_t strides[2] = {(uint64_t)x.H * DKC * 4, (uint64_t)x.T * x.H * DKC * 4};
        const uint32_t box_sw[3] = {32, (uint32_t)CH, 1}, box_n[3] = {DKC, (uint32_t)CH, 1};
        if (!encode_tiled(&mks, 3, x.k, dims, strides, box_sw, true) ||
            !encode_tiled(&mvn, 3, x.v, dims, strides, box_n, false))
            return cudaErrorInvalidValue;
    }
    cudaError_t e = set_smem_attr_once((const void*)delta_prep, PrepSmem::bytes);
    if (e != cudaSuccess) return e;
    e = set_smem_attr_once((const void*)delta_chain, ChainSmem::bytes);
    if (e != cudaSuccess) return e;
    if (x.o != nullptr) {
        e = set_smem_attr_once(output_unit_decay_kernel(), output_unit_decay_smem());
        if (e != cudaSuccess) return e;
    }

    ChunkArgs c{};
    c.B = x.B; c.T = x.T; c.H = x.H; c.G = x.H; c.NC = d.NC;
    c.scale = x.scale;
    c.q = x.q; c.k = x.k; c.v = nullptr; c.vt = d.DTt; c.d = nullptr;
    c.S_in = nullptr; c.S_out = nullptr; c.o = x.o;
    c.W = d.St; c.gam = nullptr; c.anc = nullptr;
    c.st = st;
    c.wait_ns = wait_ns;

    // Auto: the whole call in one cooperative launch (delta_fused) when the
    // chains leave at least half the SMs to the other stages; on the caller's
    // stream.
    if (segments == 0 && d.NC >= 2 && 2 * x.B * x.H <= sm_count) {
        const size_t fused_bytes = std::max({PrepSmem::bytes, ChainSmem::bytes, output_unit_decay_smem()});
        e = set_smem_attr_once((const void*)delta_fused, fused_bytes);
        if (e != cudaSuccess) return e;
        c.n0 = 0;
        c.nsg = d.NC;
        CUtensorMap mq, mk, mo;
        if (!output_maps(c, 128, &mq, &mk, &mo)) return cudaErrorInvalidValue;
        e = cudaMemsetAsync(ctrl, 0, (size_t)(2 + (int64_t)x.B * x.H * (d.NC + 1)) * 4, s);
        if (e != cudaSuccess) return e;
        d.n0 = 0;
        d.n1 = d.NC;
        d.S_from = x.S_in;
        d.S_to = x.S_out;
        d.poison = poison ? 1 : 0;
        void* args[] = {(void*)&mks, (void*)&mvn, (void*)&mq, (void*)&mk, (void*)&mo, (void*)&d, (void*)&c, (void*)&ctrl};
        return cudaLaunchCooperativeKernel((const void*)delta_fused, dim3((unsigned)sm_count), dim3(NT), args, fused_bytes,
                                           s);
    }

    const int nseg = delta_segments(d.NC, x.B * x.H, sm_count, segments);
    const bool piped = nseg > 1;
    // CTAs for a stage that runs beside a chain (one CTA per head): the SMs
    // the chain leaves, when that is at least half of them
    const int free_sms = sm_count - x.B * x.H;
    const int side = 2 * free_sms >= sm_count ? free_sms : sm_count;
    if (piped && (pipe.prep == nullptr || pipe.chain == nullptr || pipe.out == nullptr || pipe.nev < 2 * nseg + 4))
        return cudaErrorInvalidValue;
    cudaStream_t sp = piped ? pipe.prep : s, sc = piped ? pipe.chain : s, so = piped ? pipe.out : s;
    int ev = 0;
    auto order = [&](cudaStream_t from, cudaStream_t to) -> cudaError_t {   // `to` waits for `from`'s work so far
        if (from == to) return cudaSuccess;
        cudaError_t r = cudaEventRecord(pipe.ev[ev], from);
        if (r == cudaSuccess) r = cudaStreamWaitEvent(to, pipe.ev[ev], 0);
        ++ev;
        return r;
    };
    e = cudaSuccess;
    if (piped) {   // fork: the side streams wait for the caller's earlier work
        e = cudaEventRecord(pipe.ev[ev++], s);
        for (cudaStream_t side : {sp, sc, so})
            if (e == cudaSuccess) e = cudaStreamWaitEvent(side, pipe.ev[0], 0);
    }

    for (int g = 0; g < nseg && e == cudaSuccess; ++g) {
        d.n0 = delta_seg_start(d.NC, nseg, g);
        d.n1 = delta_seg_start(d.NC, nseg, g + 1);
        // persistent CTAs: the first segment's on every SM; a later one runs
        // beside the chain of the segment before and leaves the chain's SMs
        // free, so that the chain starts as soon as its inputs exist
        const int units = x.B * x.H * (d.n1 - d.n0);
        delta_prep<<<(unsigned)std::min(units, g > 0 ? side : sm_count), NT, PrepSmem::bytes, sp>>>(mks, mvn, d);
        e = cudaGetLastError();
        if (e == cudaSuccess) e = order(sp, sc);
        if (e != cudaSuccess) break;
        d.S_from = g == 0 ? x.S_in : S_mid;
        d.S_to = g == nseg - 1 ? x.S_out : S_mid;
        delta_chain<<<(unsigned)((size_t)x.B * x.H), NT, ChainSmem::bytes, sc>>>(d);
        e = cudaGetLastError();
        if (e != cudaSuccess || x.o == nullptr) continue;
        e = order(sc, so);
        if (e != cudaSuccess) break;
        c.n0 = d.n0;
        c.nsg = d.n1 - d.n0;
        // persistent output CTAs; one of a segment whose successor's chain is
        // still to run leaves that chain's SMs free as well
        e = launch_output_unit_decay(c, g + 1 < nseg ? side : sm_count, so);
    }
    // join: the caller's stream waits for the side streams, also after an error
    for (cudaStream_t side : {sp, sc, so}) {
        const cudaError_t ej = order(side, s);
        if (e == cudaSuccess) e = ej;
    }
    return e;
}

}  // namespace sn
