// scan_common.cuh -- pieces shared by the two scan kernels' files.
#pragma once

#include "ptx.cuh"
#include "sn_internal.h"

namespace sn {

// Injection term of the two forms: b (FMA form) or (1 - a) * u (gated form),
// each operation rounded to nearest.
template <bool GATED>
__device__ __forceinline__ float inj(float a, float b) {
    if constexpr (GATED) return __fmul_rn(__fsub_rn(1.0f, a), b);
    else return b;
}

// TMA can describe the (B, T, N) tensors: rows 16-byte aligned.
inline bool scan_tma_ok(const ScanArgs& x) {
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    return (x.N % 4 == 0) && al16(x.a) && al16(x.b) && (x.s_out == nullptr || al16(x.s_out));
}

// 3-D tensor map over a (B, T, N) fp32 tensor with a [box_t x box_n] box.
inline bool make_scan_map(CUtensorMap* m, const float* base, int B, int T, int N, int box_n, int box_t) {
    const uint64_t dims[3] = {(uint64_t)N, (uint64_t)T, (uint64_t)B};
    const uint64_t strides[2] = {(uint64_t)N * 4, (uint64_t)T * N * 4};
    const uint32_t box[3] = {(uint32_t)box_n, (uint32_t)box_t, 1};
    return encode_tiled(m, 3, base, dims, strides, box);
}

}  // namespace sn
