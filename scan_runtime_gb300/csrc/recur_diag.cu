// recur_diag.cu -- diagonal-decay matrix recurrence (GLA per-key decay,
// Mamba-2 per-head scalar decay with grouped k/q): "SunnyNet 工程化实录" §4.1,
// §4.3.  Kernel template in recur_seq.cuh.
#include "recur_seq.cuh"

namespace sn {

namespace {
// 8 or 4 rows per lane by diag_eight_rows (recur_seq.cuh).
template <int KIND>
cudaError_t diag_dispatch(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count, int force_w,
                          cudaStream_t stream) {
    const bool many = diag_eight_rows(x, sm_count);
    if (x.dk == 128)
        return many ? run_seq_width<KIND, 128, 8, 4>(x, st, wait_ns, sm_count, force_w, stream)
                    : run_seq_width<KIND, 128, 4, 4>(x, st, wait_ns, sm_count, force_w, stream);
    return many ? run_seq_width<KIND, 64, 8, 4>(x, st, wait_ns, sm_count, force_w, stream)
                : run_seq_width<KIND, 64, 4, 4>(x, st, wait_ns, sm_count, force_w, stream);
}
}  // namespace

cudaError_t launch_recur_diag_seq(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count, int force_w,
                                  cudaStream_t stream) {
    if (x.kind == RK_DIAG_KEY) return diag_dispatch<RK_DIAG_KEY>(x, st, wait_ns, sm_count, force_w, stream);
    return diag_dispatch<RK_DIAG_HEAD>(x, st, wait_ns, sm_count, force_w, stream);
}

}  // namespace sn
