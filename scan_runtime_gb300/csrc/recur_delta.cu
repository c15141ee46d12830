// recur_delta.cu -- DeltaNet delta rule ("SunnyNet 工程化实录" §4.2).
// Kernel template in recur_seq.cuh; 8 rows x 2 columns per lane, 2-warp CTAs,
// operands read one step ahead.
#include "recur_seq.cuh"

namespace sn {

cudaError_t launch_recur_delta_seq(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int, int force_w,
                                   cudaStream_t stream) {
    const int w = force_w ? force_w : 2;
    if (x.dk == 128) return run_seq_w<RK_DELTA, 128, 8, 2, false, 1>(x, st, wait_ns, w, stream);
    return run_seq_w<RK_DELTA, 64, 8, 2, false, 1>(x, st, wait_ns, w, stream);
}

}  // namespace sn
