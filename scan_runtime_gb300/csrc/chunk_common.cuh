// chunk_common.cuh -- definitions shared by the chunked tensor-core kernels
// (recur_chunked.cu: diagonal decays; recur_delta_chunked.cu: the delta rule):
// chunk geometry, the kernels' argument block, the K-major operand layout
// with K extent 128, async-copy and tf32 helpers.
#pragma once

#include <cmath>

#include "ptx.cuh"
#include "sn_internal.h"
#include "tc.cuh"

namespace sn {
namespace chunk {

constexpr int CH = 128;                 // tokens per chunk
constexpr int DKC = 128;                // key dimension
constexpr int NT = 256;                 // threads per CTA
constexpr int ANCHOR = CH / 2 - 1;      // anchor token of the per-key factors
constexpr float RANGE_LOG2 = 60.0f;     // bound on |lam_t - lam_anchor| (log2 units)
constexpr int OPF = CH * DKC;           // floats per 128 x 128 operand
constexpr unsigned FULL = 0xffffffffu;

struct ChunkArgs {
    int B, T, H, G, NC;
    float scale;
    const float* q;
    const float* k;
    const float* v;
    const float* d;
    const float* S_in;
    float* S_out;
    float* o;
    float* W;       // per (b, h, chunk) a dv x dk tile in operand layout: dS^T, then S'^T
    float* gam;     // (B, H, NC, dk): chunk decay gamma_n per key
    float* anc;     // (B, H, NC, dk): anchor factor 2^{lam_m} (1 for per-head decays, -1 for flagged chunks)
    int* bad;       // (B, H, NC): per-key decays whose anchor factors leave 2^{+-RANGE_LOG2}
    const float* vt;   // optional: per chunk a v^T operand tile (rows value, K = token, tf32)
                       // that replaces v in the output stage (bulk-loaded)
    float* vt_out;     // optional: where chunk_state stores its rounded v^T tile per chunk
    SnDevStatus* st;
    uint64_t wait_ns;
    int n0, nsg;       // the output kernel alone: chunks [n0, n0 + nsg) (nsg = 0: all NC chunks)
    int gated;         // gated injection: key i of token t enters weighted by 1 - d (per key or per head)
};

// sites recorded with SN_E_TIMEOUT / SN_E_RANGE
constexpr int SITE_STATE_WAIT = 1, SITE_OUT_WAIT1 = 2, SITE_OUT_WAIT2 = 3, SITE_RANGE_KEY = 4,
              SITE_RANGE_HEAD = 5, SITE_OUT_COPY = 6;

__device__ __forceinline__ int off128(int r, int k) {
    return (r >> 3) * 1024 + (k >> 2) * 32 + (r & 7) * 4 + (k & 3);
}

// Float offset of element (r, k) of a 128 x 128 operand in the 128-byte-swizzled
// K-major layout (tc.cuh): atom k / 32 (16 KB), row r (128 B), 16-byte chunk
// (k mod 32) / 4 XOR (r mod 8).
__device__ __forceinline__ int off_sw(int r, int k) {
    return (k >> 5) * 4096 + r * 32 + ((((k & 31) >> 2) ^ (r & 7)) << 2) + (k & 3);
}

__device__ __forceinline__ float4 ldg4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 tf32x4(float a, float b, float c, float d) {
    return make_float4(tc::to_tf32(a), tc::to_tf32(b), tc::to_tf32(c), tc::to_tf32(d));
}
__device__ __forceinline__ float4 tf32x4(float4 x) { return tf32x4(x.x, x.y, x.z, x.w); }

// cp.async of 4 / 16 bytes; `valid` false writes zeros (the source is not read).
__device__ __forceinline__ void cp_async4(float* dst, const float* src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async16(float* dst, const float* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Base-2 exponential and logarithm from the SFU instructions (ex2.approx /
// lg2.approx, relative error ~2^-22; subnormals flush to zero): far below the
// tf32 rounding of the operands they scale.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float* align128(unsigned char* p) {
    return reinterpret_cast<float*>(smem_align<128>(p));
}

struct ChunkIdx {
    int b, h, n, g, t0, nval;
    size_t bh;
};

// Units (one chunk of one head each) of a launch: B * H * (nsg or NC).
__device__ __forceinline__ int chunk_units(const ChunkArgs& a) { return a.B * a.H * (a.nsg > 0 ? a.nsg : a.NC); }

__device__ __forceinline__ ChunkIdx chunk_index(const ChunkArgs& a, int unit) {
    ChunkIdx c;
    c.h = unit % a.H;
    const int bn = unit / a.H;
    const int nsg = a.nsg > 0 ? a.nsg : a.NC;
    c.n = a.n0 + bn % nsg;
    c.b = bn / nsg;
    c.g = c.h / (a.H / a.G);
    c.t0 = c.n * CH;
    c.nval = min(CH, a.T - c.t0);
    c.bh = (size_t)c.b * a.H + c.h;
    return c;
}

__device__ __forceinline__ ChunkIdx chunk_index(const ChunkArgs& a) { return chunk_index(a, (int)blockIdx.x); }

// Transposing copy of a (tokens x R) slab of a row-major global array into the
// operand layout (rows = the R columns of the array, K = tokens): element
// (t, r) of rows base[t * rs + r] lands at off128(r, t).  Lanes cover 8 rows x
// 4 tokens (32 distinct banks); tokens >= nval are zero.
template <int R>
__device__ __forceinline__ void copy_transposed(float* dst, const float* base, size_t rs, int nval, int warp,
                                                int lane) {
    const int rl = lane & 7, tq = lane >> 3;
    constexpr int RB = R / 8;
#pragma unroll 8
    for (int p = warp; p < RB * (CH / 4); p += NT / 32) {
        const int r = (p % RB) * 8 + rl;
        const int t = (p / RB) * 4 + tq;
        const bool ok = t < nval;
        cp_async4(dst + off128(r, t), base + (size_t)(ok ? t : 0) * rs + r, ok);
    }
}

// recur_chunked.cu: the output kernel alone with unit decays (d == nullptr),
// dv = 128 (used by the chunked delta rule), over chunks [n0, n0 + nsg) on at
// most max_ctas CTAs (fewer CTAs than units: persistent CTAs); the kernel and
// its shared-memory size, for opting in before the launches.
cudaError_t launch_output_unit_decay(const ChunkArgs& a, int max_ctas, cudaStream_t s);
const void* output_unit_decay_kernel();
size_t output_unit_decay_smem();
// The output stage's TMA maps (q and k swizzled boxes; o, zero without o).
bool output_maps(const ChunkArgs& a, int dv, CUtensorMap* mq, CUtensorMap* mk, CUtensorMap* mo);

}  // namespace chunk
}  // namespace sn
