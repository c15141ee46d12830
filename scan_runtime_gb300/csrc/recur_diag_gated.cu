// recur_diag_gated.cu -- the gated (convex-combination) matrix state
//   S_t = diag(p_t) S_{t-1} + diag(1 - p_t) k_t v_t^T,   o_t = scale * S_t^T q_t
// with the gate per key or per head: the association-memory branch of
// "我拿同一份权重和 llama.cpp 正面比了一场：我手写的 C 内核，慢了 1.1–1.7 倍" §8 and
// HGRN2's recurrence structure (§4 there).  Same kernel template and tile
// choice as recur_diag.cu; the injection's k is scaled by (1 - p) first.
#include "recur_seq.cuh"

namespace sn {

cudaError_t launch_recur_diag_gated_seq(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count,
                                        int force_w, cudaStream_t stream) {
    if (x.kind == RK_DIAG_KEY_GATED)
        return x.dk == 128 ? run_seq_diag<RK_DIAG_KEY_GATED, 128>(x, st, wait_ns, sm_count, force_w, stream)
                           : run_seq_diag<RK_DIAG_KEY_GATED, 64>(x, st, wait_ns, sm_count, force_w, stream);
    return x.dk == 128 ? run_seq_diag<RK_DIAG_HEAD_GATED, 128>(x, st, wait_ns, sm_count, force_w, stream)
                       : run_seq_diag<RK_DIAG_HEAD_GATED, 64>(x, st, wait_ns, sm_count, force_w, stream);
}

}  // namespace sn
