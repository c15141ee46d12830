// readout.cu -- readout epilogues applied to a recurrence's output o_t, each
// one pass over HBM with every step of the epilogue fused:
//   norm_gate  y = RMSNorm(o) * w * silu(g) over the dv values of each
//              (b, t, h), normalised first and gated after (GLA's readout,
//              "SunnyNet 工程化实录" §4.3);
//   dskip      y = o + D_h * x, the skip connection of a Mamba-2 head (same
//              page, §4.1).
// Both are HBM bound: 12 bytes per element (read o and g|x, write y).
#include <cmath>

#include "ptx.cuh"
#include "sn_internal.h"

namespace sn {
namespace {

constexpr int RT = 256;                 // threads per CTA
constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ float4 ldg4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// One row of DV values per group of DV / 4 lanes (a float4 each); the sum of
// squares reduces over the group with xor shuffles.  The loop runs per warp,
// so every lane reaches every shuffle; rows past the end are masked.
template <int DV>
__global__ void __launch_bounds__(RT) norm_gate_kernel(int64_t rows, const float* o, const float* g,
                                                       const float* w, float eps, float* y) {
    constexpr int GL = DV / 4;            // lanes per row
    constexpr int RPW = 32 / GL;          // rows per warp
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane / GL, gl = lane % GL;
    const float4 w4 = w != nullptr ? ldg4(w + 4 * gl) : make_float4(1.f, 1.f, 1.f, 1.f);
    const int64_t stride = (int64_t)gridDim.x * (RT / 32) * RPW;
    for (int64_t r0 = ((int64_t)blockIdx.x * (RT / 32) + warp) * RPW; r0 < rows; r0 += stride) {
        const int64_t r = r0 + sub;
        const bool ok = r < rows;
        const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 o4 = ok ? ldg4(o + r * DV + 4 * gl) : zero;
        const float4 g4 = ok ? ldg4(g + r * DV + 4 * gl) : zero;
        float ss = fmaf(o4.x, o4.x, fmaf(o4.y, o4.y, fmaf(o4.z, o4.z, o4.w * o4.w)));
#pragma unroll
        for (int off = GL / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(FULL, ss, off);
        const float inv = rsqrtf(fmaf(ss, 1.0f / DV, eps));
        if (ok)
            st_cs(reinterpret_cast<float4*>(y + r * DV + 4 * gl),
                  make_float4(o4.x * inv * w4.x * silu(g4.x), o4.y * inv * w4.y * silu(g4.y),
                              o4.z * inv * w4.z * silu(g4.z), o4.w * inv * w4.w * silu(g4.w)));
    }
}

// y = o + D_h x over float4 groups; dv4 = dv / 4 groups per row.
__global__ void __launch_bounds__(RT) dskip_kernel(int64_t n4, int H, int dv4, const float* o, const float* x,
                                                   const float* D, float* y) {
    const int64_t stride = (int64_t)gridDim.x * RT;
    for (int64_t i = (int64_t)blockIdx.x * RT + threadIdx.x; i < n4; i += stride) {
        const int64_t row = i / dv4;
        const float d = __ldg(D + (int)(row % H));
        const float4 o4 = ldg4(o + 4 * i), x4 = ldg4(x + 4 * i);
        st_cs(reinterpret_cast<float4*>(y + 4 * i),
              make_float4(fmaf(d, x4.x, o4.x), fmaf(d, x4.y, o4.y), fmaf(d, x4.z, o4.z), fmaf(d, x4.w, o4.w)));
    }
}

unsigned grid_for(int64_t items, int64_t per_cta, int sm_count) {
    const int64_t want = (items + per_cta - 1) / per_cta;
    const int64_t cap = (int64_t)sm_count * (2048 / RT);   // one wave of full SMs
    return (unsigned)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_readout_norm_gate(int64_t rows, int dv, const float* o, const float* g, const float* w, float eps,
                                     float* y, int sm_count, cudaStream_t s) {
    if (dv == 128) {
        norm_gate_kernel<128><<<grid_for(rows, (RT / 32) * 1, sm_count), RT, 0, s>>>(rows, o, g, w, eps, y);
    } else {
        norm_gate_kernel<64><<<grid_for(rows, (RT / 32) * 2, sm_count), RT, 0, s>>>(rows, o, g, w, eps, y);
    }
    return cudaGetLastError();
}

cudaError_t launch_readout_dskip(int64_t rows, int H, int dv, const float* o, const float* x, const float* D,
                                 float* y, int sm_count, cudaStream_t s) {
    const int64_t n4 = rows * (dv / 4);
    dskip_kernel<<<grid_for(n4, RT, sm_count), RT, 0, s>>>(n4, H, dv / 4, o, x, D, y);
    return cudaGetLastError();
}

}  // namespace sn
