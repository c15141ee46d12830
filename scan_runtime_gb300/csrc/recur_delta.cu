// recur_delta.cu -- DeltaNet delta rule ("SunnyNet 工程化实录" §4.2).
// Kernel template in recur_seq.cuh; 8 rows x 4 columns per lane.
#include "recur_seq.cuh"

namespace sn {

cudaError_t launch_recur_delta_seq(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count,
                                   int force_w, cudaStream_t stream) {
    if (x.dk == 128) return run_seq_width<RK_DELTA, 128, 8, 4>(x, st, wait_ns, sm_count, force_w, stream);
    return run_seq_width<RK_DELTA, 64, 8, 4>(x, st, wait_ns, sm_count, force_w, stream);
}

}  // namespace sn
