// recur_rwkv7.cu -- RWKV-7 rank-1 removal ("SunnyNet 工程化实录" §5.1):
// the sequence kernel (template in recur_seq.cuh, 8 rows x 4 columns per lane)
// and the batched single-step decode kernel.
//
// Decode (T == 1, dk = dv = 64): four (batch, head) states per CTA arrive as
// 16 KB bulk copies plus their q, k, w, v rows; each state is updated and read
// out with the sequence kernel's lane_step and lane layout (8 rows per lane,
// 8 lanes per column group), so a decode call has the bits of a one-step
// sequence call; the new states leave as bulk copies (in place allowed).
#include "recur_seq.cuh"

namespace sn {

cudaError_t launch_recur_rwkv7_seq(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count,
                                   int force_w, cudaStream_t stream) {
    if (x.dk == 128) return run_seq_width<RK_RWKV7, 128, 8, 4>(x, st, wait_ns, sm_count, force_w, stream);
    return run_seq_width<RK_RWKV7, 64, 8, 4>(x, st, wait_ns, sm_count, force_w, stream);
}

namespace {

constexpr int DEC_TILES = 4;                   // (b, h) states per CTA
constexpr int DEC_D = 64;                      // dk = dv = 64
constexpr int DEC_R = 8;                       // rows (keys) per lane, as the sequence kernel
constexpr int DEC_LPC = DEC_D / DEC_R;         // 8 lanes per column group
constexpr int DEC_C = 2;                       // value columns per lane group
constexpr int DEC_THREADS = (DEC_D / DEC_C) * DEC_LPC;   // 256
constexpr uint32_t DEC_S_BYTES = DEC_D * DEC_D * 4;
constexpr uint32_t DEC_V_BYTES = DEC_D * 4;
// per tile: S (16 KB) then q, k, w, v rows (256 B each)
constexpr uint32_t DEC_TILE_BYTES = DEC_S_BYTES + 4 * DEC_V_BYTES;
constexpr size_t DEC_SMEM = DEC_TILES * DEC_TILE_BYTES + 8 + 128;

__global__ void __launch_bounds__(DEC_THREADS, 3)
recur_decode_rwkv7(int BH, const float* __restrict__ q, const float* __restrict__ k,
                   const float* __restrict__ v, const float* __restrict__ w, const float* S_in, float* S_out,
                   float* __restrict__ o, SnDevStatus* st, uint64_t wait_ns) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_align<128>(smem_raw);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + DEC_TILES * DEC_TILE_BYTES);
    const int tid = threadIdx.x;
    const int tile0 = blockIdx.x * DEC_TILES;
    const int ntile = min(DEC_TILES, BH - tile0);

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(bar, ntile * (S_in != nullptr ? DEC_TILE_BYTES : 4 * DEC_V_BYTES));
        for (int t = 0; t < ntile; ++t) {
            unsigned char* tb = smem + t * DEC_TILE_BYTES;
            const size_t bh = (size_t)(tile0 + t);
            if (S_in != nullptr) bulk_load(tb, S_in + bh * DEC_D * DEC_D, DEC_S_BYTES, bar);
            bulk_load(tb + DEC_S_BYTES + 0 * DEC_V_BYTES, q + bh * DEC_D, DEC_V_BYTES, bar);
            bulk_load(tb + DEC_S_BYTES + 1 * DEC_V_BYTES, k + bh * DEC_D, DEC_V_BYTES, bar);
            bulk_load(tb + DEC_S_BYTES + 2 * DEC_V_BYTES, w + bh * DEC_D, DEC_V_BYTES, bar);
            bulk_load(tb + DEC_S_BYTES + 3 * DEC_V_BYTES, v + bh * DEC_D, DEC_V_BYTES, bar);
        }
    }
    const bool ok = __syncthreads_and(mbar_wait(bar, 0, wait_ns));
    if (!ok) {
        if (tid == 0) {
            record_error(st, SN_E_TIMEOUT, (SN_K_RECUR_DECODE << 16) | 1);
            (void)mbar_wait(bar, 0, wait_ns);
        }
        return;
    }
    const int grpi = tid / DEC_LPC, sub = tid % DEC_LPC;
    const int i0 = grpi * DEC_C;                       // first value row (column of P) of the group
    for (int t = 0; t < ntile; ++t) {
        float* S = reinterpret_cast<float*>(smem + t * DEC_TILE_BYTES);
        const float* qv = reinterpret_cast<const float*>(smem + t * DEC_TILE_BYTES + DEC_S_BYTES);
        const float* kv = qv + DEC_D;
        const float* wv = kv + DEC_D;
        const float* vv = wv + DEC_D;
        float2 P[DEC_R][DEC_C / 2];
#pragma unroll
        for (int m = 0; m < DEC_R / 4; ++m) {
            const int r0 = (m * DEC_LPC + sub) * 4;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (S_in != nullptr) {
                a = *reinterpret_cast<const float4*>(S + i0 * DEC_D + r0);
                b = *reinterpret_cast<const float4*>(S + (i0 + 1) * DEC_D + r0);
            }
            P[4 * m][0] = make_float2(a.x, b.x);
            P[4 * m + 1][0] = make_float2(a.y, b.y);
            P[4 * m + 2][0] = make_float2(a.z, b.z);
            P[4 * m + 3][0] = make_float2(a.w, b.w);
        }
        float2 part[DEC_C / 2];
        lane_step<RK_RWKV7, DEC_R, DEC_C, DEC_LPC>(P, kv, wv, qv, vv + i0, 0.f, sub, part, o != nullptr);
        __syncwarp();
#pragma unroll
        for (int m = 0; m < DEC_R / 4; ++m) {
            const int r0 = (m * DEC_LPC + sub) * 4;
            *reinterpret_cast<float4*>(S + i0 * DEC_D + r0) =
                make_float4(P[4 * m][0].x, P[4 * m + 1][0].x, P[4 * m + 2][0].x, P[4 * m + 3][0].x);
            *reinterpret_cast<float4*>(S + (i0 + 1) * DEC_D + r0) =
                make_float4(P[4 * m][0].y, P[4 * m + 1][0].y, P[4 * m + 2][0].y, P[4 * m + 3][0].y);
        }
        if (o != nullptr) {
            const float2 acc = group_sum2(part[0], DEC_LPC);
            if (sub == 0) {
                o[(size_t)(tile0 + t) * DEC_D + i0] = __fmul_rn(acc.x, 1.0f);
                o[(size_t)(tile0 + t) * DEC_D + i0 + 1] = __fmul_rn(acc.y, 1.0f);
            }
        }
    }
    if (S_out == nullptr) return;
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
        for (int tt = 0; tt < ntile; ++tt)
            bulk_store(S_out + (size_t)(tile0 + tt) * DEC_D * DEC_D, smem + tt * DEC_TILE_BYTES, DEC_S_BYTES);
        bulk_commit();
        bulk_wait_read_all();   // shared memory must outlive the copies' reads; the writes finish on their own
    }
}

}  // namespace

bool recur_decode_supported(const RecurArgs& x) {
    return (x.kind == RK_RWKV7 && x.T == 1 && x.dk == DEC_D && x.dv == DEC_D) || recur_decode_cols_supported(x);
}

cudaError_t launch_recur_decode(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count,
                                cudaStream_t stream) {
    if (x.kind != RK_RWKV7) return launch_recur_decode_cols(x, sm_count, stream);   // recur_decode.cu
    cudaError_t e = set_smem_attr_once((const void*)recur_decode_rwkv7, DEC_SMEM);
    if (e != cudaSuccess) return e;
    const int BH = x.B * x.H;
    const int grid = (BH + DEC_TILES - 1) / DEC_TILES;
    recur_decode_rwkv7<<<grid, DEC_THREADS, DEC_SMEM, stream>>>(BH, x.q, x.k, x.v, x.g, x.S_in, x.S_out, x.o, st,
                                                               wait_ns);
    return cudaGetLastError();
}

}  // namespace sn
