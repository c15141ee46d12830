// sn_internal.h -- definitions shared by the host ABI layer and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/sn_abi.h"

// Per-context device status block (256 bytes, zeroed at creation).
struct SnDevStatus {
    int error;   // first device-side error of any launch (SN_E_*), 0 = none
    int site;    // where it happened: (kernel id << 16) | wait site
    unsigned int abort_tag;   // tag of a look-back launch in which a tile gave up waiting
    unsigned int lb_epoch;    // epoch of the last look-back launch, 0 = none (stored by its last CTA)
    unsigned int lb_done;     // CTAs of the running look-back launch that have finished
    int pad[59];
};
static_assert(sizeof(SnDevStatus) == 256, "status block is 256 bytes");

// Kernel ids used in SnDevStatus::site.
enum SnKernelId : int {
    SN_K_SCAN_SEQ = 1,
    SN_K_SCAN_LOOKBACK = 2,
    SN_K_RECUR_SEQ = 3,
    SN_K_RECUR_DECODE = 4,
    SN_K_RECUR_CHUNK = 5,
};

struct SnCtx {
    int device;
    int sm_count;
    int cc_major, cc_minor;
    SnDevStatus* dstatus;       // device status block (owned)
    // caller-owned workspace for the chunked look-back scan
    void* ws;
    int64_t ws_bytes;
    bool ws_dirty;              // flag area must be cleared before next use
    int64_t lb_last_flags;      // layout of the tagged flags last cleared: the look-back kernel's flag
                                // count, or minus the fused path's tile count
    uint64_t tagged_calls;      // look-back and fused launches since the tagged words were last cleared
    // options
    int scan_kernel;
    int wait_limit_us;
    int debug_poison;
    int recur_kernel;
    int recur_tile;             // forced consumer warps per CTA of the sequence kernel (0 = auto)
    int delta_segments;         // segments of the pipelined chunked delta rule (0 = auto)
    // side streams and events of the pipelined chunked delta rule (created with the context)
    cudaStream_t pipe_prep, pipe_chain, pipe_out;
    cudaEvent_t pipe_ev[20];
    bool pipe_ready;
};

namespace sn {

// Layout of the chunked look-back scan (shared with the host for workspace
// sizing): NC channels x TC time steps per tile.
constexpr int LB_NC = 32;
constexpr int LB_TC = 128;

// Returns the workspace bytes of the look-back scan for (B, T, N).
int64_t lookback_ws_bytes(int B, int T, int N);
int64_t lookback_cw_offset(int B, int T, int N);
int64_t lookback_flag_count(int B, int T, int N);

// Opt `kern` into `bytes` of dynamic shared memory on the current device (once
// per kernel and device; function attributes are per device).
cudaError_t set_smem_attr_once(const void* kern, size_t bytes);
// Resident CTAs per SM of `kern` on the current device (cached per device).
cudaError_t occupancy_once(const void* kern, int threads, size_t smem, int* out);


// tensor-map encoder (driver entry point fetched through the runtime)
bool encode_tiled(CUtensorMap* map, int rank, const void* base, const uint64_t* dims,
                  const uint64_t* strides_bytes /* rank-1 entries */, const uint32_t* box, bool swizzle128 = false);

struct ScanArgs {
    int B, T, N;
    const float* a;
    const float* b;   // b (FMA form) or u (gated form)
    const float* s0;
    float* s_final;
    float* s_out;
};

// Reverse (adjoint) scan arguments: forward states s (B, T, N), direct
// gradients gs (B, T, N), final-state gradient gf (B, N), outputs da, db|du
// (B, T, N) and ds0 (B, N); u only for the gated form.
struct BwdArgs {
    int B, T, N;
    const float* a;
    const float* u;
    const float* s0;
    const float* s;
    const float* gs;
    const float* gf;
    float* da;
    float* dbu;
    float* ds0;
};

// Launchers (return a CUDA error code; validation happens before).
cudaError_t launch_scan_backward(const BwdArgs& x, bool gated, SnDevStatus* st, uint64_t wait_ns,
                                 cudaStream_t stream);
// Chunked reverse scans (scan_bwd_chunked.cu), for few channels and long T:
// 16-byte aligned tensors with N % 4 == 0; workspace bytes (at the start of
// the context workspace, which the look-back scan's sizes cover).
bool scan_backward_chunked_supported(const BwdArgs& x);
int64_t scan_backward_chunked_ws_bytes(int B, int T, int N);
cudaError_t launch_scan_backward_chunked(const BwdArgs& x, bool gated, void* ws, SnDevStatus* st, uint64_t wait_ns,
                                         int sm_count, cudaStream_t stream);
cudaError_t launch_scan_sequential(const ScanArgs& x, bool gated, SnDevStatus* st, uint64_t wait_ns,
                                   cudaStream_t stream);
cudaError_t launch_scan_lookback(const ScanArgs& x, bool gated, void* ws, int poison, SnDevStatus* st,
                                 uint64_t wait_ns, int sm_count, cudaStream_t stream);
// Reduce-then-scan (scan_lookback.cu): the look-back kernel's results in three
// launches without flags, for few channel tiles and long T; same workspace.
cudaError_t launch_scan_reduce_scan(const ScanArgs& x, bool gated, void* ws, SnDevStatus* st, uint64_t wait_ns,
                                    int sm_count, cudaStream_t stream);
// The same results in one cooperative launch (scan_fused.cu) that reads a and
// b once: state CTAs publish each tile's aggregate and wait for its carry,
// which a chain CTA per column of tiles folds.  Whether it runs (eight chunks
// or more; else the reduce-then-scan launches run), the workspace bytes it
// needs, and the tagged area [a, a + b) a change of geometry clears.
bool scan_fused_applies(int T);
int64_t scan_fused_ws_bytes(int B, int T, int N);
void scan_fused_tag_area(int B, int T, int N, int64_t* a, int64_t* b);
// *fell_back is set when the launch ran the reduce-then-scan launches instead
// (too many columns for the fused path's progress rule).
cudaError_t launch_scan_fused(const ScanArgs& x, bool gated, void* ws, int poison, SnDevStatus* st,
                              uint64_t wait_ns, int sm_count, cudaStream_t stream, bool* fell_back);

enum RecurKind : int {
    RK_DIAG_KEY = 0,
    RK_DIAG_HEAD = 1,
    RK_DELTA = 2,
    RK_RWKV7 = 3,
    RK_DIAG_KEY_GATED = 4,     // injection scaled by (1 - d_i): convex-combination state
    RK_DIAG_HEAD_GATED = 5,
};

struct RecurArgs {
    int kind;
    int B, T, H, G, dk, dv;
    float scale;
    const float* q;
    const float* k;
    const float* v;
    const float* g;     // decay d (per key or per head), beta (delta) or w (rwkv7)
    const float* S_in;
    float* S_out;
    float* o;
    bool state_transposed;   // S stored (dv, dk) (RWKV-7) instead of (dk, dv)
};

cudaError_t launch_recur_sequence(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count,
                                  int force_width, cudaStream_t stream);
// Whether a forced CTA width (SN_OPT_RECUR_TILE; 0 = auto) suits the problem:
// the value dimension must be a multiple of the columns a CTA of that width covers.
bool recur_seq_width_ok(const RecurArgs& x, int sm_count, int width);
cudaError_t launch_recur_decode(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count,
                                cudaStream_t stream);
bool recur_decode_supported(const RecurArgs& x);
// recur_decode.cu: T == 1 of every kind (diagonal decays, the delta rule, RWKV-7)
bool recur_decode_ring_supported(const RecurArgs& x);
cudaError_t launch_recur_decode_ring(const RecurArgs& x, SnDevStatus* st, uint64_t wait_ns, int sm_count,
                                     cudaStream_t stream);

// Chunked tensor-core form of the delta rule (recur_delta_chunked.cu).
int64_t delta_chunked_ws_bytes(int B, int T, int H, int dk, int dv);
bool delta_chunked_supported(const RecurArgs& x);
// At most DELTA_MAX_SEGMENTS segments; a pipeline of n segments uses 2 n + 4
// events.  delta_segments: the segment count used for NC chunks of BH heads
// (requested 0 = auto).
constexpr int DELTA_MAX_SEGMENTS = 8;
struct DeltaPipe {
    cudaStream_t prep, chain, out;
    cudaEvent_t* ev;
    int nev;
};
int delta_segments(int NC, int BH, int sm_count, int requested);
cudaError_t launch_delta_chunked(const RecurArgs& x, void* ws, SnDevStatus* st, uint64_t wait_ns, int sm_count,
                                 int segments, bool poison, const DeltaPipe& pipe, cudaStream_t stream);

// Readout epilogues (readout.cu).
cudaError_t launch_readout_norm_gate(int64_t rows, int dv, const float* o, const float* g, const float* w, float eps,
                                     float* y, int sm_count, cudaStream_t stream);
cudaError_t launch_readout_dskip(int64_t rows, int H, int dv, const float* o, const float* x, const float* D,
                                 float* y, int sm_count, cudaStream_t stream);

// Chunked tensor-core form of the diagonal-decay recurrence (recur_chunked.cu).
int64_t chunked_ws_bytes(int B, int T, int H, int dk, int dv);
bool chunked_supported(const RecurArgs& x);
cudaError_t launch_recur_chunked(const RecurArgs& x, void* ws, SnDevStatus* st, uint64_t wait_ns, int sm_count,
                                 cudaStream_t stream);

}  // namespace sn
