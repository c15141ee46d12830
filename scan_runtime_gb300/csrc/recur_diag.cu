// recur_diag.cu -- diagonal-decay matrix recurrence (GLA per-key decay,
// Mamba-2 per-head scalar decay with grouped k/q): "SunnyNet 工程化实录" §4.1,
// §4.3.  Kernel template and tile choice in recur_seq.cuh.
#include "recur_seq.cuh"

namespace sn {

cudaError_t launch_recur_diag_seq(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count, int force_w,
                                  cudaStream_t stream) {
    if (x.kind == RK_DIAG_KEY)
        return x.dk == 128 ? run_seq_diag<RK_DIAG_KEY, 128>(x, st, wait_ns, sm_count, force_w, stream)
                           : run_seq_diag<RK_DIAG_KEY, 64>(x, st, wait_ns, sm_count, force_w, stream);
    return x.dk == 128 ? run_seq_diag<RK_DIAG_HEAD, 128>(x, st, wait_ns, sm_count, force_w, stream)
                       : run_seq_diag<RK_DIAG_HEAD, 64>(x, st, wait_ns, sm_count, force_w, stream);
}

}  // namespace sn
