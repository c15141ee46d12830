// recur.cu -- dispatch of the tier-2 matrix recurrences to their kernels
// (recur_diag.cu, recur_diag_gated.cu, recur_delta.cu, recur_rwkv7.cu;
// template in recur_seq.cuh).
#include "recur_seq.cuh"

namespace sn {

cudaError_t launch_recur_diag_seq(const RecurArgs&, SnDevStatus*, uint64_t, int, int, cudaStream_t);
cudaError_t launch_recur_diag_gated_seq(const RecurArgs&, SnDevStatus*, uint64_t, int, int, cudaStream_t);
cudaError_t launch_recur_delta_seq(const RecurArgs&, SnDevStatus*, uint64_t, int, int, cudaStream_t);
cudaError_t launch_recur_rwkv7_seq(const RecurArgs&, SnDevStatus*, uint64_t, int, int, cudaStream_t);

bool recur_seq_width_ok(const RecurArgs& x, int sm_count, int width) {
    if (width == 0) return true;
    if (width != 2 && width != 4 && width != 8) return false;
    return x.dv % (width * seq_cols_per_warp(x, sm_count)) == 0;   // the tile of recur_seq.cuh
}

cudaError_t launch_recur_sequence(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count,
                                  int force_width, cudaStream_t stream) {
    switch (x.kind) {
        case RK_DIAG_KEY:
        case RK_DIAG_HEAD: return launch_recur_diag_seq(x, st, wait_ns, sm_count, force_width, stream);
        case RK_DIAG_KEY_GATED:
        case RK_DIAG_HEAD_GATED: return launch_recur_diag_gated_seq(x, st, wait_ns, sm_count, force_width, stream);
        case RK_DELTA: return launch_recur_delta_seq(x, st, wait_ns, sm_count, force_width, stream);
        case RK_RWKV7: return launch_recur_rwkv7_seq(x, st, wait_ns, sm_count, force_width, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sn
