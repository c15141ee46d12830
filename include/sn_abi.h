/*
 * sn_abi.h -- stable C ABI of the GB300 linear-recurrence library (libsn).
 *
 * The library computes the unified linear-recurrence state update of O(N)
 * sequence models on one NVIDIA GB300 GPU (sm_103a):
 *   tier 1  per-channel first-order scans (FMA and gated forms);
 *   tier 2  per-head matrix-state recurrences with readout (diagonal decay
 *           for GLA / Mamba-2, the DeltaNet delta rule, RWKV-7 rank-1
 *           removal), including batched single-step (T = 1) decode.
 *
 * Sources, cited by page title and section:
 *   [P1] "SunnyNet 工程化实录：一个 O(N) 架构如何长出自己的 C 推理运行时"
 *   [P2] "我拿同一份权重和 llama.cpp 正面比了一场：我手写的 C 内核，慢了 1.1–1.7 倍"
 *
 * ABI conventions follow [P1] §6 (stable C ABI):
 *   - every symbol carries the sn_ prefix; handles are opaque;
 *   - the version is packed as (MAJOR << 16) | (MINOR << 8) | PATCH;
 *   - capability bits SN_CAP_*; callers must ignore bits they do not know;
 *   - sn_status is a fixed int32_t; array dimensions are int32_t;
 *   - a caller passes SN_ABI_VERSION_MAJOR to sn_abi_check() and must refuse
 *     the library when it returns SN_E_UNSUPPORTED.
 *
 * Memory and ownership (all compute calls):
 *   - every tensor argument is a DEVICE pointer to contiguous, row-major fp32
 *     data owned by the caller; the library never frees or retains it;
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *     default stream.  Calls are asynchronous: they validate, enqueue the
 *     kernel on `stream` and return.  Outputs are valid once the stream has
 *     reached that point;
 *   - compute calls never allocate device memory and never create streams or
 *     events.  The only device memory the library owns is a 256-byte status
 *     block per context (allocated by sn_ctx_create, which also creates the
 *     context's side streams and events) and the static scratch array of
 *     sn_scan_lookback_noalloc; the caller hands over the rest with
 *     sn_ctx_set_workspace;
 *   - an initial-state pointer may be NULL (zero initial state); a final-state
 *     or per-step output pointer may be NULL (not written);
 *   - the initial and final state may be the same buffer (in-place
 *     continuation); any other overlap between an output and an input or
 *     another output is rejected with SN_E_INVAL.
 *
 * Errors:
 *   - argument errors are detected on the host before anything is enqueued;
 *     outputs are then left untouched;
 *   - SN_E_DEVICE reports a CUDA runtime error at launch;
 *   - device-side failures (a bounded wait that ran out) are recorded in the
 *     context's status block; sn_ctx_last_error() returns and clears them
 *     once the caller has synchronised the stream.
 *
 * Thread safety: a context may be used from one host thread at a time, and
 * calls that use the context's workspace must be ordered on one stream.
 */
#ifndef SN_ABI_H
#define SN_ABI_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SN_ABI_VERSION_MAJOR 1
#define SN_ABI_VERSION_MINOR 0
#define SN_ABI_VERSION_PATCH 0
#define SN_ABI_VERSION \
    ((SN_ABI_VERSION_MAJOR << 16) | (SN_ABI_VERSION_MINOR << 8) | SN_ABI_VERSION_PATCH)

typedef int32_t sn_status;

/* Status codes.  The first six are the ones [P1] §6 fixes; the last three are
 * extensions of this library. */
#define SN_OK             0
#define SN_E_INVAL       (-1)  /* bad argument: NULL, dim <= 0, overlap, misalignment */
#define SN_E_NOMEM       (-2)  /* workspace missing or too small */
#define SN_E_IO          (-3)  /* reserved by the ABI (no file I/O here) */
#define SN_E_FORMAT      (-4)  /* reserved by the ABI (no file formats here) */
#define SN_E_UNSUPPORTED (-5)  /* major-version mismatch, head dim not compiled, device not sm_103 */
#define SN_E_DEVICE      (-6)  /* CUDA runtime error (launch failure, bad stream, ...) */
#define SN_E_TIMEOUT     (-7)  /* a bounded device-side wait ran out (see sn_ctx_last_error) */
#define SN_E_RANGE       (-8)  /* an input value outside what a kernel supports (see sn_recur_diag_chunked) */

/* Capability bits returned by sn_abi_caps(). */
#define SN_CAP_SCAN_FMA    (1u << 0)   /* sn_scan_fma */
#define SN_CAP_SCAN_GATED  (1u << 1)   /* sn_scan_gated */
#define SN_CAP_RECUR_DIAG  (1u << 2)   /* sn_recur_diag */
#define SN_CAP_RECUR_DELTA (1u << 3)   /* sn_recur_delta */
#define SN_CAP_RECUR_RWKV7 (1u << 4)   /* sn_recur_rwkv7 */
#define SN_CAP_DECODE      (1u << 5)   /* dedicated T == 1 decode kernels */
#define SN_CAP_SCAN_LOOKBACK (1u << 6) /* chunked scan with look-back carries */
#define SN_CAP_SCAN_BACKWARD (1u << 7) /* sn_scan_fma_backward, sn_scan_gated_backward */
#define SN_CAP_RECUR_CHUNKED (1u << 8) /* sn_recur_diag_chunked (tensor-core chunked form) */
#define SN_CAP_READOUT       (1u << 9) /* sn_readout_norm_gate, sn_readout_dskip */
#define SN_CAP_DELTA_CHUNKED (1u << 10) /* sn_recur_delta_chunked (tensor-core chunked delta rule) */

/* Decay layouts of sn_recur_diag. */
#define SN_DECAY_PER_KEY        0   /* d is (B, T, H, dk): one decay per key row (GLA)        */
#define SN_DECAY_PER_HEAD       1   /* d is (B, T, H):     one scalar decay per head (Mamba-2) */
#define SN_DECAY_PER_KEY_GATED  2   /* as PER_KEY, injection weighted by (1 - d_i)             */
#define SN_DECAY_PER_HEAD_GATED 3   /* as PER_HEAD, injection weighted by (1 - d)              */

/* Context options (sn_ctx_set_option / sn_ctx_get_option). */
#define SN_OPT_SCAN_KERNEL      1  /* 0 auto (default), 1 sequential-in-T, 2 chunked look-back,
                                      3 chunked reduce-then-scan, 4 chunked fused (forward scans) */
#define SN_OPT_WAIT_LIMIT_US    2  /* bound on any device-side wait, microseconds (default 1e6) */
#define SN_OPT_DEBUG_POISON     3  /* 1: the look-back and fused scan kernels and the fused delta-rule kernel wait for a word no CTA writes (tests the bound) */
#define SN_OPT_LOOKBACK_CHUNK   4  /* read-only: time steps per look-back chunk */
#define SN_OPT_RECUR_KERNEL     5  /* 0 auto (default: T == 1 uses decode), 1 always the sequence kernel */
#define SN_OPT_RECUR_TILE       6  /* sequence kernel: 0 auto (default), or 2, 4, 8 consumer warps per CTA
                                      (the same bits for every width); a width whose CTA columns the value
                                      dimension does not divide would fail with SN_E_INVAL before any
                                      launch (no compiled tile and head size has such a width) */
#define SN_OPT_DELTA_SEGMENTS   7  /* sn_recur_delta_chunked: 0 auto (default): one cooperative launch of
                                      the preparation, the chains and the output stage, where the
                                      chains (one CTA per head and batch row) leave at least half the SMs,
                                      else a segmented pipeline; or 1..8 segments of the chunk sequence run
                                      as a pipeline (same bits for every value) */

#define SN_SCAN_KERNEL_AUTO       0
#define SN_SCAN_KERNEL_SEQUENTIAL 1
#define SN_SCAN_KERNEL_LOOKBACK   2
#define SN_SCAN_KERNEL_REDUCE_SCAN 3   /* the look-back kernel's results in three flag-free passes */
#define SN_SCAN_KERNEL_FUSED       4   /* the same results in one launch that reads a and b once, a
                                          carry chain per column running beside the tiles (forward scans;
                                          T < 1024, or B * ceil(N / 32) above about SMs / 9, runs
                                          reduce-then-scan) */

/* Operation ids for sn_workspace_bytes(). */
#define SN_OP_SCAN_FMA   1
#define SN_OP_SCAN_GATED 2

typedef struct SnCtx SnCtx;

/* ---------------------------------------------------------------- meta */

/* Packed version of the loaded library ((MAJOR << 16) | (MINOR << 8) | PATCH). */
uint32_t sn_abi_version(void);

/* SN_OK when `major` equals the library's major version, else
 * SN_E_UNSUPPORTED (the caller must refuse the library).  [P1] §6. */
sn_status sn_abi_check(int32_t major);

/* Capability bits (SN_CAP_*).  Unknown bits must be ignored by callers. */
uint32_t sn_abi_caps(void);

/* Static, NUL-terminated description of a status code (never NULL). */
const char* sn_status_str(sn_status s);

/* ---------------------------------------------------------------- context */

/* Create a context bound to CUDA device `device`.  Allocates the context's
 * 256-byte device status block on that device and creates the CUDA objects
 * the pipelined chunked delta rule runs on (three non-blocking streams and 20
 * events, see sn_recur_delta_chunked), so that no compute call creates CUDA
 * objects.  sn_ctx_free releases all of them.  Errors: SN_E_INVAL (NULL
 * out_ctx, bad device index), SN_E_UNSUPPORTED (device is not sm_103),
 * SN_E_DEVICE (CUDA failure).  On error *out_ctx is set to NULL. */
sn_status sn_ctx_create(int32_t device, SnCtx** out_ctx);

/* Free a context (NULL is a no-op).  The caller must have synchronised all
 * streams that still use it. */
void sn_ctx_free(SnCtx* ctx);

/* Hand the context a caller-owned device workspace (used only by the chunked
 * look-back scan).  `dev_ptr` must be 256-byte aligned; `bytes` >= 0; a NULL
 * pointer or 0 bytes removes it.  The library never frees it.  The first
 * look-back launch after this call (or after another chunked path used the
 * workspace) clears the flag and carry-word areas with cudaMemsetAsync on that
 * launch's stream. */
sn_status sn_ctx_set_workspace(SnCtx* ctx, void* dev_ptr, int64_t bytes);

/* Workspace bytes the chunked scans need for this problem (op =
 * SN_OP_SCAN_FMA or SN_OP_SCAN_GATED): with columns = B * ceil(N / 32),
 * chunks = ceil(T / 128) and tiles = columns * chunks, the larger of
 *   a flag word per tile rounded up to 256 bytes, plus the larger of 512
 *   bytes per tile and columns * (1536 * ceil(chunks / 4) + 128) bytes
 *   (the look-back and reduce-then-scan kernels), and
 *   columns * (2304 * ceil(chunks / 4) + 256) bytes from eight chunks on
 *   (the fused kernel's tagged carry and aggregate words);
 * 0 for an op that needs none, -1 on invalid arguments. */
int64_t sn_workspace_bytes(int32_t op, int32_t B, int32_t T, int32_t N);

/* Return and clear the first device-side error recorded in the context's
 * status block (SN_OK if none).  Synchronous: call it after the stream that
 * ran the work has been synchronised. */
sn_status sn_ctx_last_error(SnCtx* ctx);

/* Set / read a context option (SN_OPT_*).  SN_E_INVAL for an unknown key or
 * out-of-range value; SN_OPT_LOOKBACK_CHUNK is read-only. */
sn_status sn_ctx_set_option(SnCtx* ctx, int32_t key, int32_t value);
sn_status sn_ctx_get_option(SnCtx* ctx, int32_t key, int32_t* value);

/* ---------------------------------------------------------------- tier 1 */

/* FMA-form scan, per channel n of each batch row b, for t = 0..T-1:
 *     s_t = a_t * s_{t-1} + b_t,      s_{-1} = s0          ([P1] §2.1)
 * evaluated in fp32 with one fused multiply-add per step.
 *   a, b   : (B, T, N) inputs;      s_out  : (B, T, N) all states, may be NULL
 *   s0     : (B, N), NULL = zeros;  s_final: (B, N) state after t = T-1, may be NULL
 * The sequential kernel (the default whenever it fills the GPU) gives the
 * same bits as the single-precision definition at every t, so splitting a
 * sequence into segments and carrying s_final -> s0 reproduces the full run
 * bit for bit ([P1] §4).  For few channels and long T the call chunks T
 * instead: automatically the fused path where the workspace covers it, else
 * reduce-then-scan; or, by SN_OPT_SCAN_KERNEL, any
 * of those two or the decoupled look-back kernel; all three give the same
 * bits, are deterministic and are bit-exact under splits at multiples of
 * SN_OPT_LOOKBACK_CHUNK.  Calls may be captured in a CUDA graph and replayed:
 * the look-back and fused kernels keep their launch epoch in device memory,
 * so every replay tags its flags and carry words afresh.
 * Pointers need 4-byte alignment; N % 4 == 0 with 16-byte aligned a, b and
 * s_out enables the TMA path.  Errors: SN_E_INVAL, SN_E_NOMEM (look-back
 * forced without enough workspace), SN_E_DEVICE. */
sn_status sn_scan_fma(SnCtx* ctx, int32_t B, int32_t T, int32_t N,
                      const float* a, const float* b, const float* s0,
                      float* s_final, float* s_out, void* stream);

/* Gated-form scan ([P1] §2.1):
 *     s_t = a_t * s_{t-1} + (1 - a_t) * u_t
 * evaluated in fp32 as s = fma(a_t, s, (1 - a_t) * u_t) with the injection
 * rounded after each of its two operations.  Arguments as sn_scan_fma with
 * u in place of b. */
sn_status sn_scan_gated(SnCtx* ctx, int32_t B, int32_t T, int32_t N,
                        const float* a, const float* u, const float* s0,
                        float* s_final, float* s_out, void* stream);

/* Device staging bytes sn_scan_host needs: forms_mask 1 (FMA), 2 (gated) or
 * 3 (both); three slots of rows = min(rows_per_chunk, B) batch rows, each
 * slot r256(rows T N 4) + r256(rows N 4) + forms * (2 r256(rows T N 4) +
 * r256(rows N 4)) bytes with r256 rounding up to a multiple of 256.  -1 on
 * invalid arguments. */
int64_t sn_scan_host_staging_bytes(int32_t B, int32_t T, int32_t N, int32_t forms_mask, int32_t rows_per_chunk);

/* Both scan forms over HOST buffers, the transfers part of the call
 * ([P1] §2.1 forms; §2.4, the call overhead that a batch-wide call must
 * amortise).  a, b, u, s0 (host, same shapes as sn_scan_fma / sn_scan_gated;
 * b = NULL skips the FMA form, u = NULL the gated form, at least one given;
 * s0 NULL = zeros) are copied to the device in chunks of rows_per_chunk batch
 * rows, scanned there, and each given output (s_out_*: (B, T, N), s_final_*:
 * (B, N), host, may be NULL) is copied back.  Three chunks are in flight at
 * once on the context's three pipeline streams (the host-to-device copy of
 * one, the kernels of another and the device-to-host copy of a third
 * overlap), each chunk in its own slot of `staging` (caller-owned device
 * memory, 256-byte aligned, at least sn_scan_host_staging_bytes bytes).
 * Every chunk runs the sequential kernel, so the results have the bits of
 * sn_scan_fma / sn_scan_gated with that kernel (the fp32 definition's) and
 * no context workspace is used.  The call is asynchronous: the pipeline
 * starts after the earlier work on `stream`, and `stream` waits for all of
 * it, so synchronise `stream` before reading the outputs.  Pinned host
 * memory lets the copies overlap; pageable memory works, slower.  One call
 * at a time per context (the pipeline streams are the context's).
 * Outputs may not overlap any other buffer.  Errors: SN_E_INVAL (NULL a,
 * neither b nor u, dims, alignment, overlap, staging too small or not
 * 256-byte aligned), SN_E_DEVICE. */
sn_status sn_scan_host(SnCtx* ctx, int32_t B, int32_t T, int32_t N, int32_t rows_per_chunk,
                       const float* a, const float* b, const float* u, const float* s0,
                       float* s_out_fma, float* s_final_fma, float* s_out_gated, float* s_final_gated,
                       void* staging, int64_t staging_bytes, void* stream);

/* Reverse (adjoint) scan of the FMA form: the backward pass of sn_scan_fma
 * (the pages' kernels pair a forward scan with a reverse scan, [P1] §8).
 * Given the forward states and gs_t = dL/ds_t, gf = dL/ds_final:
 *     g_{T-1} = gs_{T-1} + gf,    g_t = gs_t + a_{t+1} g_{t+1}  (one fma per step)
 *     grad_a_t = g_t s_{t-1},     grad_b_t = g_t,     grad_s0 = a_0 g_0   (s_{-1} = s0)
 *   a, s (forward states s_out), grad_s : (B, T, N), required
 *   s0, grad_final : (B, N), NULL = zeros
 *   grad_a, grad_b : (B, T, N), grad_s0 : (B, N), each may be NULL (not written)
 * Runs T backwards per channel (the fp32 definition's bits); N % 4 == 0 with
 * 16-byte aligned tensors uses TMA, anything else plain loads.  For few
 * channels and long T, with a context workspace of sn_workspace_bytes() bytes
 * set, the call instead chunks T (per-chunk reverse aggregates, a carry chain,
 * then the gradients): chosen automatically there, forced by either chunked
 * SN_OPT_SCAN_KERNEL value (then SN_E_NOMEM without the workspace, and
 * SN_E_UNSUPPORTED unless N % 4 == 0 and every tensor is 16-byte aligned).  It
 * rounds in a different order (within 1e-5 of the definition, deterministic)
 * and overwrites the workspace.  Errors: SN_E_INVAL, SN_E_DEVICE, and those. */
sn_status sn_scan_fma_backward(SnCtx* ctx, int32_t B, int32_t T, int32_t N,
                               const float* a, const float* s0, const float* s,
                               const float* grad_s, const float* grad_final,
                               float* grad_a, float* grad_b, float* grad_s0, void* stream);

/* Reverse scan of the gated form (backward pass of sn_scan_gated): g as in
 * sn_scan_fma_backward, then
 *     grad_a_t = g_t (s_{t-1} - u_t),   grad_u_t = g_t (1 - a_t),   grad_s0 = a_0 g_0.
 * u : (B, T, N) required; other arguments as sn_scan_fma_backward. */
sn_status sn_scan_gated_backward(SnCtx* ctx, int32_t B, int32_t T, int32_t N,
                                 const float* a, const float* u, const float* s0, const float* s,
                                 const float* grad_s, const float* grad_final,
                                 float* grad_a, float* grad_u, float* grad_s0, void* stream);

/* ---------------------------------------------------------------- tier 2 */

/* Diagonal-decay matrix recurrence per (batch b, head h):
 *     S_t = diag(d_t) S_{t-1} + k_t v_t^T,     o_t = scale * S_t^T q_t
 * ([P1] §4.3 GLA with per-key decay; [P1] §4.1 / [P2] §3 Mamba-2 with one
 * scalar decay dA = exp(dt*A) per head, B_g and C_g shared by a group of
 * heads, dt folded into v by the caller).  Decays are linear (not log).
 *   q, k : (B, T, G, dk)   head h reads group h / (H / G)
 *   v, o : (B, T, H, dv)   o may be NULL
 *   d    : (B, T, H, dk) for SN_DECAY_PER_KEY, (B, T, H) for SN_DECAY_PER_HEAD
 *   S_in, S_out : (B, H, dk, dv), row = key index, column = value index;
 *          S_in NULL = zeros; S_out may be NULL or equal S_in.
 * The gated layouts give the convex-combination state
 *     S_t = diag(d_t) S_{t-1} + diag(1 - d_t) k_t v_t^T
 * of the association-memory branch ([P2] §8; HGRN2's recurrence structure,
 * [P2] §4), computed as S = fma(d_i, S, ((1 - d_i) * k_i) * v_j).
 * Requires H % G == 0, dk in {64, 128}, dv in {64, 128} and 16-byte aligned
 * pointers (else SN_E_UNSUPPORTED / SN_E_INVAL).  Deterministic; the result
 * depends only on the inputs, so segment splits are bit-exact. */
sn_status sn_recur_diag(SnCtx* ctx, int32_t B, int32_t T, int32_t H, int32_t G,
                        int32_t dk, int32_t dv, int32_t decay_kind, float scale,
                        const float* q, const float* k, const float* v,
                        const float* d, const float* S_in, float* S_out,
                        float* o, void* stream);

/* DeltaNet delta rule per (b, h) ([P1] §4.2, [P2] §3):
 *     delta_t = (v_t - S_{t-1}^T k_t) * beta_t
 *     S_t     = S_{t-1} + k_t delta_t^T,       o_t = scale * S_t^T q_t
 *   q, k : (B, T, H, dk);  v, o : (B, T, H, dv);  beta : (B, T, H)
 *   S_in, S_out : (B, H, dk, dv) as in sn_recur_diag.
 * Requirements and guarantees as sn_recur_diag. */
sn_status sn_recur_delta(SnCtx* ctx, int32_t B, int32_t T, int32_t H,
                         int32_t dk, int32_t dv, float scale,
                         const float* q, const float* k, const float* v,
                         const float* beta, const float* S_in, float* S_out,
                         float* o, void* stream);

/* RWKV-7 matrix state with rank-1 removal per (b, h) ([P1] §5.1):
 *     S_t = S_{t-1} (.) w_t - (S_{t-1} k_t) k_t^T + v_t k_t^T,   o_t = S_t q_t
 * with w_t scaling key column j of every row and the removal formed from the
 * state before decay.
 *   q, k, w : (B, T, H, dk);  v, o : (B, T, H, dv)
 *   S_in, S_out : (B, H, dv, dk), row = value index, column = key index.
 * T == 1 runs the batched single-step decode kernel (state-bandwidth bound,
 * in place when S_in == S_out).  Requirements as sn_recur_diag. */
sn_status sn_recur_rwkv7(SnCtx* ctx, int32_t B, int32_t T, int32_t H,
                         int32_t dk, int32_t dv,
                         const float* q, const float* k, const float* v,
                         const float* w, const float* S_in, float* S_out,
                         float* o, void* stream);

/* Chunked tensor-core form of sn_recur_diag for all four decay layouts: the
 * same recurrence and readout, evaluated T-parallel in chunks of 128 tokens
 * (the gated layouts are the same recurrence with every key weighted by
 * 1 - d, [P2] §8).  The state is carried from
 * chunk to chunk ([P2] §8 keeps the association memory "chunk-scannable";
 * [P1] §4.3 GLA, §4.1 Mamba-2), and inside a chunk
 *     S_{n+1} = diag(D_n) S_n + sum_j diag(D_n / D_j) k_j v_j^T
 *     o_t     = scale * ( (q_t (.) D_t)^T S_n + sum_{j <= t} (q_t (.) D_t / D_j)^T k_j v_j )
 * with D_t the product of the chunk's decays up to token t (computed in log2
 * space), as three dense contractions per chunk on the tensor cores
 * (tcgen05, tf32 operands rounded to nearest, fp32 accumulation) plus an
 * fp32 chain over the chunk states.
 *
 * Arguments, layouts and state conventions are those of sn_recur_diag.
 * Accuracy: tf32 rounding of the operands, about 1e-3 relative (the
 * sequence kernel of sn_recur_diag is exact fp32 per step); results do not
 * depend on timing, but a segment split changes the chunk grid and so the
 * rounding.
 * Requirements: dk == 128, dv in {64, 128} (else SN_E_UNSUPPORTED); 16-byte aligned pointers; a
 * context workspace of at least sn_recur_chunked_workspace_bytes() bytes
 * (else SN_E_NOMEM), which the call overwrites (a later look-back scan on the
 * same context clears its flag area again).  Decays must be positive: a
 * decay <= 0 (or NaN) records SN_E_RANGE in the context's status block
 * (outputs are then unspecified; use sn_recur_diag).  Per-key decays enter
 * the products through factors anchored at the chunk's token 63; a chunk in
 * which the decay product between some token and the anchor leaves
 * [2^-60, 2^60] has its outputs evaluated step by step in fp32 from the
 * chunk's start state instead (exact per step; slower than the tensor-core
 * products, so strong decays cost time, not accuracy). */
sn_status sn_recur_diag_chunked(SnCtx* ctx, int32_t B, int32_t T, int32_t H, int32_t G,
                                int32_t dk, int32_t dv, int32_t decay_kind, float scale,
                                const float* q, const float* k, const float* v,
                                const float* d, const float* S_in, float* S_out,
                                float* o, void* stream);

/* Workspace bytes sn_recur_diag_chunked needs: B * H * ceil(T / 128) chunk
 * states of dk x dv floats, two vectors of dk floats per chunk, one int32 per
 * chunk and a 128 x dv tile of v per chunk (each part rounded up to 256
 * bytes); -1 on invalid arguments. */
int64_t sn_recur_chunked_workspace_bytes(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv);

/* Chunked tensor-core form of sn_recur_delta: the same delta rule and readout
 * ([P1] §4.2), evaluated T-parallel in chunks of 128 tokens.  Inside a chunk
 * the deltas solve a unit lower-triangular system (the WY form of the chunk's
 * rank-1 updates):
 *     T = (I + diag(beta) L)^{-1} diag(beta),   L = strictly lower part of K K^T
 *     Delta = T V - (T K) S_n,   S_{n+1} = S_n + K^T Delta,
 *     O = scale * (Q S_n + tril(Q K^T) Delta)
 * The Gram matrix uses a hi/lo tf32 split and the triangular inverse runs in
 * fp32; the remaining products use tf32 operands with fp32 accumulation, and
 * the state crosses chunks in fp32.
 * Arguments and layouts as sn_recur_delta.  Accuracy about 1e-3 relative
 * (tf32); splits at multiples of 128 tokens are bit-exact.  Requires dk = dv
 * = 128 (else SN_E_UNSUPPORTED), 16-byte aligned pointers and a context
 * workspace of at least sn_recur_delta_chunked_workspace_bytes() bytes (else
 * SN_E_NOMEM), which the call overwrites.
 * Streams: by default (SN_OPT_DELTA_SEGMENTS 0, with B*H at most half the
 * SMs) the call runs on `stream` alone as one cooperative launch, whose
 * chains wait, bounded, for the preparation of each chunk and whose output
 * units wait for their chains (SN_E_TIMEOUT past SN_OPT_WAIT_LIMIT_US).
 * Otherwise, for more than a
 * few chunks, it splits the sequence into segments and runs the chain of one
 * segment beside the preparation of the next on side streams the context
 * created with it (sn_ctx_create); the call itself creates no stream or
 * event.  The
 * side streams wait for `stream`'s earlier work and `stream` waits for them
 * before its later work, so to the caller the call is ordered on `stream`
 * like any other (also under stream capture).  A context is not for use from
 * two host threads at once. */
sn_status sn_recur_delta_chunked(SnCtx* ctx, int32_t B, int32_t T, int32_t H,
                                 int32_t dk, int32_t dv, float scale,
                                 const float* q, const float* k, const float* v,
                                 const float* beta, const float* S_in, float* S_out,
                                 float* o, void* stream);

/* Workspace bytes sn_recur_delta_chunked needs: five tiles of dk x dv floats
 * per chunk of 128 tokens and head (W, K^T, U, the chunk state and the
 * chunk's deltas), one fp32 dk x dv state per head (carried between
 * segments) and 4 * (2 + B * H * (chunks + 1)) bytes of control words,
 * each kind rounded up to 256 bytes; -1 on invalid arguments. */
int64_t sn_recur_delta_chunked_workspace_bytes(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv);

/* ---------------------------------------------------------------- readout epilogues */

/* GLA readout epilogue ([P1] §4.3: the readout is followed by RMSNorm(o) and
 * the output gate, normalised first and gated after), one pass per element:
 *     y_j = o_j / sqrt(mean_j(o_j^2) + eps) * w_j * silu(g_j),
 *     silu(z) = z / (1 + exp(-z)),
 * with the mean over the dv values of each (b, t, h).
 *   o, g, y : (B, T, H, dv); y may equal o (in place), no other overlap
 *   w       : (dv,) norm weight shared by the heads, NULL = 1
 *   eps     : >= 0 (eps = 0 and an all-zero row give NaN, as the definition)
 * fp32 (rsqrt and exp from the CUDA math library); within 1e-5 normwise of
 * the fp64 definition.  Requires dv in {64, 128} (else SN_E_UNSUPPORTED) and
 * 16-byte aligned pointers.  Errors: SN_E_INVAL, SN_E_UNSUPPORTED, SN_E_DEVICE. */
sn_status sn_readout_norm_gate(SnCtx* ctx, int32_t B, int32_t T, int32_t H, int32_t dv,
                               const float* o, const float* g, const float* w, float eps,
                               float* y, void* stream);

/* Mamba-2 skip connection added to each head's readout:
 *     y = o + D_h * x,   one fused multiply-add per element.
 *   o, x, y : (B, T, H, dv); y may equal o;  D : (H,)
 * Requirements and errors as sn_readout_norm_gate. */
sn_status sn_readout_dskip(SnCtx* ctx, int32_t B, int32_t T, int32_t H, int32_t dv,
                           const float* o, const float* x, const float* D, float* y, void* stream);

/* ---------------------------------------------------------------- allocation-free variant */

/* Maximum look-back tiles of sn_scan_lookback_noalloc: a call needs
 * B * ceil(N / 32) * ceil(T / 128) <= SN_NOALLOC_MAX_TILES. */
#define SN_NOALLOC_MAX_TILES 40960

/* The chunked look-back scan without a context and without any device
 * allocation.  The pages have no counterpart of this entry point: it exists
 * for callers that cannot allocate device memory at run time -- code under a
 * fixed memory budget or an allocator that owns the whole device, plugins
 * whose host application forbids cudaMalloc after start-up, and paths that
 * cannot create an SnCtx (sn_ctx_create allocates a status block).
 *
 * It computes what sn_scan_fma (gated = 0) or sn_scan_gated (gated = 1)
 * computes with SN_OPT_SCAN_KERNEL = SN_SCAN_KERNEL_LOOKBACK, with the same
 * bits.  Its scratch is a file-scope device array of about 20 MiB that every
 * GPU which loads libsn holds until the process exits; problems needing more than
 * SN_NOALLOC_MAX_TILES tiles are rejected with SN_E_NOMEM.  Arguments as
 * sn_scan_fma, except: N % 4 == 0 and 16-byte aligned a, b, s_out are
 * required (else SN_E_UNSUPPORTED); the device is the calling thread's current
 * device; `status_out` (device pointer to one int32, may be NULL) receives, in
 * stream order, SN_OK or SN_E_TIMEOUT if a bounded device-side wait (1 s) ran
 * out during this call.
 *
 * The first call on a device sets the device up (it looks up the array's
 * device address and clears the array's status words with a cudaMemsetAsync
 * on `stream`), so that first call should come before any stream capture.  A
 * call whose tile count differs from the previous call's on that device (and
 * every 2^24-th call) also clears the flag and carry-word areas: two more
 * memsets on `stream`.  Every call enqueues one small memset (this call's
 * error word, error site and abort tag), the kernel and, if status_out is
 * given, a 4-byte device-to-device copy.  All calls on a device share the one array, which
 * keeps the last call's contents: calls that may overlap on the GPU (other
 * streams, other host threads) race on it and must be serialised by the
 * caller.  No cudaMalloc, cudaFree or other allocating routine is called. */
sn_status sn_scan_lookback_noalloc(int32_t gated, int32_t B, int32_t T, int32_t N,
                                   const float* a, const float* b, const float* s0,
                                   float* s_final, float* s_out, int32_t* status_out,
                                   void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SN_ABI_H */
