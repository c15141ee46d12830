// recur_rwkv7.cu -- RWKV-7 rank-1 removal ("SunnyNet 工程化实录" §5.1): the
// sequence kernel (template in recur_seq.cuh, 8 rows x 2 columns per lane,
// 4-warp CTAs) and the entry to the single-step decode (recur_decode.cu, which
// decodes every kind; a decode step has the bits of a one-step sequence call).
#include "recur_seq.cuh"

namespace sn {

cudaError_t launch_recur_rwkv7_seq(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int, int force_w,
                                   cudaStream_t stream) {
    const int w = force_w ? force_w : 4;
    if (x.dk == 128) return run_seq_w<RK_RWKV7, 128, 8, 2, false, 0>(x, st, wait_ns, w, stream);
    return run_seq_w<RK_RWKV7, 64, 8, 2, false, 0>(x, st, wait_ns, w, stream);
}

bool recur_decode_supported(const RecurArgs& x) { return recur_decode_ring_supported(x); }

cudaError_t launch_recur_decode(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count,
                                cudaStream_t stream) {
    return launch_recur_decode_ring(x, st, wait_ns, sm_count, stream);   // recur_decode.cu
}

}  // namespace sn
