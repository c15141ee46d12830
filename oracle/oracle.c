/*
 * oracle.c -- plain, sequential CPU reference for the linear-recurrence state
 * update.  TEST INFRASTRUCTURE ONLY: nothing in the product library links or
 * calls this file.  Only the tests, the smoke check of the build entry point
 * and the CPU-baseline leg of the benchmark may load it.
 *
 * Sources (cited by page title and section):
 *   [P1] "SunnyNet 工程化实录：一个 O(N) 架构如何长出自己的 C 推理运行时"
 *        (developer.aliyun.com article 1773847)
 *   [P2] "我拿同一份权重和 llama.cpp 正面比了一场：我手写的 C 内核，慢了 1.1–1.7 倍"
 *        (developer.aliyun.com article 1775078)
 *
 * Every routine is the plain definition written out: loops over batch, head
 * (or channel), then time in increasing order, with no blocking, chunking,
 * fusion or reordering.  Inputs are the exact fp32 tensors that the GPU
 * receives.  Two precisions:
 *   *_f64  every operation in double (the primary reference);
 *   *_f32  every operation in float, with fmaf() exactly where the canonical
 *          single-precision order below uses a fused multiply-add.  Built with
 *          -ffp-contract=off so the compiler adds no fusion of its own.
 *
 * Layouts (row-major, last index fastest):
 *   scans   a, b|u, s_out : (B, T, N)      s0, s_final : (B, N)
 *   diag    q, k          : (B, T, G, dk)  v, o : (B, T, H, dv)
 *           d             : (B, T, H, dk) per-key, or (B, T, H) per-head
 *           S             : (B, H, dk, dv)   (key index i = row, value j = col)
 *   delta   q, k          : (B, T, H, dk)  v, o : (B, T, H, dv)  beta : (B, T, H)
 *           S             : (B, H, dk, dv)
 *   rwkv7   q, k, w       : (B, T, H, dk)  v, o : (B, T, H, dv)
 *           S             : (B, H, dv, dk)   (value index i = row, key j = col)
 * A NULL initial state means zero; a NULL output is not written.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef int32_t i32;
typedef int64_t i64;

#define ORC_DECAY_PER_KEY        0
#define ORC_DECAY_PER_HEAD       1
#define ORC_DECAY_PER_KEY_GATED  2
#define ORC_DECAY_PER_HEAD_GATED 3

/* ------------------------------------------------------------------------ */
/* Tier 1: per-channel first-order scans.                                    */
/* ------------------------------------------------------------------------ */

/* FMA form s_t = a_t * s_{t-1} + b_t, from s_{-1} = s0.  [P1] §2.1. */
void orc_scan_fma_f64(i32 B, i32 T, i32 N, const float* a, const float* b,
                      const double* s0, double* s_final, double* s_out)
{
    for (i64 bi = 0; bi < B; ++bi) {
        for (i64 n = 0; n < N; ++n) {
            double s = s0 ? s0[bi * N + n] : 0.0;
            for (i64 t = 0; t < T; ++t) {
                i64 x = (bi * T + t) * N + n;
                s = (double)a[x] * s + (double)b[x];
                if (s_out) s_out[x] = s;
            }
            if (s_final) s_final[bi * N + n] = s;
        }
    }
}

/* Same recurrence in float.  Canonical single-precision order: one fused
 * multiply-add per step, s = fma(a_t, s, b_t).  [P1] §2.1. */
void orc_scan_fma_f32(i32 B, i32 T, i32 N, const float* a, const float* b,
                      const float* s0, float* s_final, float* s_out)
{
    for (i64 bi = 0; bi < B; ++bi) {
        for (i64 n = 0; n < N; ++n) {
            float s = s0 ? s0[bi * N + n] : 0.0f;
            for (i64 t = 0; t < T; ++t) {
                i64 x = (bi * T + t) * N + n;
                s = fmaf(a[x], s, b[x]);
                if (s_out) s_out[x] = s;
            }
            if (s_final) s_final[bi * N + n] = s;
        }
    }
}

/* Gated form s_t = a_t * s_{t-1} + (1 - a_t) * u_t.  [P1] §2.1. */
void orc_scan_gated_f64(i32 B, i32 T, i32 N, const float* a, const float* u,
                        const double* s0, double* s_final, double* s_out)
{
    for (i64 bi = 0; bi < B; ++bi) {
        for (i64 n = 0; n < N; ++n) {
            double s = s0 ? s0[bi * N + n] : 0.0;
            for (i64 t = 0; t < T; ++t) {
                i64 x = (bi * T + t) * N + n;
                double at = (double)a[x];
                s = at * s + (1.0 - at) * (double)u[x];
                if (s_out) s_out[x] = s;
            }
            if (s_final) s_final[bi * N + n] = s;
        }
    }
}

/* Float gated form.  Canonical order: the injection (1 - a_t) * u_t is formed
 * first with two rounded operations, then one fused multiply-add carries the
 * state: s = fma(a_t, s, (1 - a_t) * u_t).  [P1] §2.1 writes the injection as
 * a separate product term, which this order keeps. */
void orc_scan_gated_f32(i32 B, i32 T, i32 N, const float* a, const float* u,
                        const float* s0, float* s_final, float* s_out)
{
    for (i64 bi = 0; bi < B; ++bi) {
        for (i64 n = 0; n < N; ++n) {
            float s = s0 ? s0[bi * N + n] : 0.0f;
            for (i64 t = 0; t < T; ++t) {
                i64 x = (bi * T + t) * N + n;
                float at = a[x];
                float inj = (1.0f - at) * u[x];
                s = fmaf(at, s, inj);
                if (s_out) s_out[x] = s;
            }
            if (s_final) s_final[bi * N + n] = s;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Tier 2: per-head matrix-state recurrences with readout.                   */
/* ------------------------------------------------------------------------ */

/* Diagonal decay (GLA per-key decay, Mamba-2 per-head scalar decay):
 *   S_t = diag(d_t) S_{t-1} + k_t v_t^T,   o_t = scale * S_t^T q_t,
 * and its gated (convex-combination) form, the matrix-valued association
 * memory of [P2] §8 and HGRN2's structure ([P2] §4):
 *   S_t = diag(p_t) S_{t-1} + diag(1 - p_t) k_t v_t^T     (decay kinds 2, 3).
 * [P1] §4.3 (GLA: decay on the key dimension, readout S^T q with scale),
 * [P1] §4.1 and [P2] §3 (Mamba-2: scalar dA per head, B_g shared by the heads
 * of a group, dt folded into the injected value by the caller).
 * Head h reads k and q of group h / (H / G). */
void orc_recur_diag_f64(i32 B, i32 T, i32 H, i32 G, i32 dk, i32 dv,
                        i32 decay_kind, double scale,
                        const float* q, const float* k, const float* v,
                        const float* d, const double* S_in, double* S_out,
                        double* o)
{
    i32 hpg = H / G;
    double* S = (double*)malloc(sizeof(double) * (size_t)dk * (size_t)dv);
    for (i64 bi = 0; bi < B; ++bi) {
        for (i64 h = 0; h < H; ++h) {
            i64 g = h / hpg;
            i64 sbase = (bi * H + h) * (i64)dk * dv;
            for (i64 e = 0; e < (i64)dk * dv; ++e) S[e] = S_in ? S_in[sbase + e] : 0.0;
            for (i64 t = 0; t < T; ++t) {
                const float* qt = q + ((bi * T + t) * G + g) * dk;
                const float* kt = k + ((bi * T + t) * G + g) * dk;
                const float* vt = v + ((bi * T + t) * H + h) * dv;
                for (i64 i = 0; i < dk; ++i) {
                    int per_key = (decay_kind == ORC_DECAY_PER_KEY || decay_kind == ORC_DECAY_PER_KEY_GATED);
                    int gated = (decay_kind == ORC_DECAY_PER_KEY_GATED || decay_kind == ORC_DECAY_PER_HEAD_GATED);
                    double di = per_key ? (double)d[((bi * T + t) * H + h) * dk + i]
                                        : (double)d[(bi * T + t) * H + h];
                    double ki = gated ? (1.0 - di) * (double)kt[i] : (double)kt[i];
                    for (i64 j = 0; j < dv; ++j)
                        S[i * dv + j] = di * S[i * dv + j] + ki * (double)vt[j];
                }
                if (o) {
                    for (i64 j = 0; j < dv; ++j) {
                        double acc = 0.0;
                        for (i64 i = 0; i < dk; ++i) acc += S[i * dv + j] * (double)qt[i];
                        o[((bi * T + t) * H + h) * dv + j] = scale * acc;
                    }
                }
            }
            if (S_out) for (i64 e = 0; e < (i64)dk * dv; ++e) S_out[sbase + e] = S[e];
        }
    }
    free(S);
}

/* Float diagonal decay.  Canonical update order: the injection k_i * v_j is
 * rounded first (gated kinds: ((1 - p_i) * k_i) * v_j, each product rounded),
 * then one fused multiply-add applies the decay,
 * S_ij = fma(d_i, S_ij, k_i * v_j) -- exactly the FMA-form scan of [P1] §2.1
 * with a = d_i and b = k_i * v_j, which is the elementwise decomposition that
 * [P1] §4.3 states for GLA.  The readout sums over i in increasing order. */
void orc_recur_diag_f32(i32 B, i32 T, i32 H, i32 G, i32 dk, i32 dv,
                        i32 decay_kind, float scale,
                        const float* q, const float* k, const float* v,
                        const float* d, const float* S_in, float* S_out,
                        float* o)
{
    i32 hpg = H / G;
    float* S = (float*)malloc(sizeof(float) * (size_t)dk * (size_t)dv);
    for (i64 bi = 0; bi < B; ++bi) {
        for (i64 h = 0; h < H; ++h) {
            i64 g = h / hpg;
            i64 sbase = (bi * H + h) * (i64)dk * dv;
            for (i64 e = 0; e < (i64)dk * dv; ++e) S[e] = S_in ? S_in[sbase + e] : 0.0f;
            for (i64 t = 0; t < T; ++t) {
                const float* qt = q + ((bi * T + t) * G + g) * dk;
                const float* kt = k + ((bi * T + t) * G + g) * dk;
                const float* vt = v + ((bi * T + t) * H + h) * dv;
                for (i64 i = 0; i < dk; ++i) {
                    int per_key = (decay_kind == ORC_DECAY_PER_KEY || decay_kind == ORC_DECAY_PER_KEY_GATED);
                    int gated = (decay_kind == ORC_DECAY_PER_KEY_GATED || decay_kind == ORC_DECAY_PER_HEAD_GATED);
                    float di = per_key ? d[((bi * T + t) * H + h) * dk + i] : d[(bi * T + t) * H + h];
                    float ki = gated ? (1.0f - di) * kt[i] : kt[i];
                    for (i64 j = 0; j < dv; ++j) {
                        float inj = ki * vt[j];
                        S[i * dv + j] = fmaf(di, S[i * dv + j], inj);
                    }
                }
                if (o) {
                    for (i64 j = 0; j < dv; ++j) {
                        float acc = 0.0f;
                        for (i64 i = 0; i < dk; ++i) acc = acc + S[i * dv + j] * qt[i];
                        o[((bi * T + t) * H + h) * dv + j] = scale * acc;
                    }
                }
            }
            if (S_out) for (i64 e = 0; e < (i64)dk * dv; ++e) S_out[sbase + e] = S[e];
        }
    }
    free(S);
}

/* DeltaNet delta rule, rank-1 form:
 *   delta_t = (v_t - S_{t-1}^T k_t) * beta_t,
 *   S_t = S_{t-1} + k_t delta_t^T,   o_t = scale * S_t^T q_t.
 * [P1] §4.2 and [P2] §3.  The readout uses the updated state S_t. */
void orc_recur_delta_f64(i32 B, i32 T, i32 H, i32 dk, i32 dv, double scale,
                         const float* q, const float* k, const float* v,
                         const float* beta, const double* S_in, double* S_out,
                         double* o)
{
    double* S = (double*)malloc(sizeof(double) * (size_t)dk * (size_t)dv);
    for (i64 bi = 0; bi < B; ++bi) {
        for (i64 h = 0; h < H; ++h) {
            i64 sbase = (bi * H + h) * (i64)dk * dv;
            for (i64 e = 0; e < (i64)dk * dv; ++e) S[e] = S_in ? S_in[sbase + e] : 0.0;
            for (i64 t = 0; t < T; ++t) {
                i64 row = (bi * T + t) * H + h;
                const float* qt = q + row * dk;
                const float* kt = k + row * dk;
                const float* vt = v + row * dv;
                double bt = (double)beta[row];
                for (i64 j = 0; j < dv; ++j) {
                    double u = 0.0;
                    for (i64 i = 0; i < dk; ++i) u += S[i * dv + j] * (double)kt[i];
                    double delta = ((double)vt[j] - u) * bt;
                    for (i64 i = 0; i < dk; ++i) S[i * dv + j] += (double)kt[i] * delta;
                }
                if (o) {
                    for (i64 j = 0; j < dv; ++j) {
                        double acc = 0.0;
                        for (i64 i = 0; i < dk; ++i) acc += S[i * dv + j] * (double)qt[i];
                        o[row * dv + j] = scale * acc;
                    }
                }
            }
            if (S_out) for (i64 e = 0; e < (i64)dk * dv; ++e) S_out[sbase + e] = S[e];
        }
    }
    free(S);
}

/* Float DeltaNet, same loop order, sums over i in increasing order. */
void orc_recur_delta_f32(i32 B, i32 T, i32 H, i32 dk, i32 dv, float scale,
                         const float* q, const float* k, const float* v,
                         const float* beta, const float* S_in, float* S_out,
                         float* o)
{
    float* S = (float*)malloc(sizeof(float) * (size_t)dk * (size_t)dv);
    for (i64 bi = 0; bi < B; ++bi) {
        for (i64 h = 0; h < H; ++h) {
            i64 sbase = (bi * H + h) * (i64)dk * dv;
            for (i64 e = 0; e < (i64)dk * dv; ++e) S[e] = S_in ? S_in[sbase + e] : 0.0f;
            for (i64 t = 0; t < T; ++t) {
                i64 row = (bi * T + t) * H + h;
                const float* qt = q + row * dk;
                const float* kt = k + row * dk;
                const float* vt = v + row * dv;
                float bt = beta[row];
                for (i64 j = 0; j < dv; ++j) {
                    float u = 0.0f;
                    for (i64 i = 0; i < dk; ++i) u = u + S[i * dv + j] * kt[i];
                    float delta = (vt[j] - u) * bt;
                    for (i64 i = 0; i < dk; ++i) S[i * dv + j] = S[i * dv + j] + kt[i] * delta;
                }
                if (o) {
                    for (i64 j = 0; j < dv; ++j) {
                        float acc = 0.0f;
                        for (i64 i = 0; i < dk; ++i) acc = acc + S[i * dv + j] * qt[i];
                        o[row * dv + j] = scale * acc;
                    }
                }
            }
            if (S_out) for (i64 e = 0; e < (i64)dk * dv; ++e) S_out[sbase + e] = S[e];
        }
    }
    free(S);
}

/* RWKV-7 matrix state with rank-1 removal, S in R^{dv x dk}:
 *   S_t = S_{t-1} (.) w_t - (S_{t-1} k_t) k_t^T + v_t k_t^T,   o_t = S_t q_t.
 * [P1] §5.1.  w_t multiplies key column j of every row; the removal term is
 * formed from the state before decay, as the formula is written. */
void orc_recur_rwkv7_f64(i32 B, i32 T, i32 H, i32 dk, i32 dv,
                         const float* q, const float* k, const float* v,
                         const float* w, const double* S_in, double* S_out,
                         double* o)
{
    double* S = (double*)malloc(sizeof(double) * (size_t)dk * (size_t)dv);
    for (i64 bi = 0; bi < B; ++bi) {
        for (i64 h = 0; h < H; ++h) {
            i64 sbase = (bi * H + h) * (i64)dk * dv;
            for (i64 e = 0; e < (i64)dk * dv; ++e) S[e] = S_in ? S_in[sbase + e] : 0.0;
            for (i64 t = 0; t < T; ++t) {
                i64 row = (bi * T + t) * H + h;
                const float* qt = q + row * dk;
                const float* kt = k + row * dk;
                const float* wt = w + row * dk;
                const float* vt = v + row * dv;
                for (i64 i = 0; i < dv; ++i) {
                    double sk = 0.0;
                    for (i64 j = 0; j < dk; ++j) sk += S[i * dk + j] * (double)kt[j];
                    for (i64 j = 0; j < dk; ++j)
                        S[i * dk + j] = S[i * dk + j] * (double)wt[j]
                                        - sk * (double)kt[j]
                                        + (double)vt[i] * (double)kt[j];
                }
                if (o) {
                    for (i64 i = 0; i < dv; ++i) {
                        double acc = 0.0;
                        for (i64 j = 0; j < dk; ++j) acc += S[i * dk + j] * (double)qt[j];
                        o[row * dv + i] = acc;
                    }
                }
            }
            if (S_out) for (i64 e = 0; e < (i64)dk * dv; ++e) S_out[sbase + e] = S[e];
        }
    }
    free(S);
}

/* Float RWKV-7, same loop order. */
void orc_recur_rwkv7_f32(i32 B, i32 T, i32 H, i32 dk, i32 dv,
                         const float* q, const float* k, const float* v,
                         const float* w, const float* S_in, float* S_out,
                         float* o)
{
    float* S = (float*)malloc(sizeof(float) * (size_t)dk * (size_t)dv);
    for (i64 bi = 0; bi < B; ++bi) {
        for (i64 h = 0; h < H; ++h) {
            i64 sbase = (bi * H + h) * (i64)dk * dv;
            for (i64 e = 0; e < (i64)dk * dv; ++e) S[e] = S_in ? S_in[sbase + e] : 0.0f;
            for (i64 t = 0; t < T; ++t) {
                i64 row = (bi * T + t) * H + h;
                const float* qt = q + row * dk;
                const float* kt = k + row * dk;
                const float* wt = w + row * dk;
                const float* vt = v + row * dv;
                for (i64 i = 0; i < dv; ++i) {
                    float sk = 0.0f;
                    for (i64 j = 0; j < dk; ++j) sk = sk + S[i * dk + j] * kt[j];
                    for (i64 j = 0; j < dk; ++j)
                        S[i * dk + j] = S[i * dk + j] * wt[j] - sk * kt[j] + vt[i] * kt[j];
                }
                if (o) {
                    for (i64 i = 0; i < dv; ++i) {
                        float acc = 0.0f;
                        for (i64 j = 0; j < dk; ++j) acc = acc + S[i * dk + j] * qt[j];
                        o[row * dv + i] = acc;
                    }
                }
            }
            if (S_out) for (i64 e = 0; e < (i64)dk * dv; ++e) S_out[sbase + e] = S[e];
        }
    }
    free(S);
}

/* ------------------------------------------------------------------------ */
/* Tier 1 backward: the reverse (adjoint) scans of both forms.               */
/* ------------------------------------------------------------------------ */
/* With gs_t = dL/ds_t given for every t and gf = dL/ds_final, the total
 * adjoint of the state runs backward in time:
 *     g_{T-1} = gs_{T-1} + gf,     g_t = gs_t + a_{t+1} g_{t+1}   (t < T-1)
 * and the input gradients follow from the forward step
 * s_t = a_t s_{t-1} + b_t (b_t = (1 - a_t) u_t in the gated form):
 *     FMA:   da_t = g_t s_{t-1},            db_t = g_t
 *     gated: da_t = g_t (s_{t-1} - u_t),    du_t = g_t (1 - a_t)
 *     ds0 = a_0 g_0,   with s_{-1} = s0.
 * This is the reverse scan that the forward kernels of "SunnyNet 工程化实录"
 * §8 (three entries: forward scan, reverse scan, single step) pair with.
 * s holds the forward states s_t (B, T, N); gs, gf, s0 may be NULL (zeros);
 * outputs may be NULL.  `u` is NULL for the FMA form. */
static void orc_scan_bwd_f64(int gated, i32 B, i32 T, i32 N, const float* a, const float* u,
                             const double* s0, const double* s, const float* gs, const float* gf,
                             double* da, double* dbu, double* ds0)
{
    for (i64 bi = 0; bi < B; ++bi) {
        for (i64 n = 0; n < N; ++n) {
            double g = 0.0;
            for (i64 t = T - 1; t >= 0; --t) {
                i64 x = (bi * T + t) * N + n;
                double gst = gs ? (double)gs[x] : 0.0;
                if (t == T - 1) g = gst + (gf ? (double)gf[bi * N + n] : 0.0);
                else g = gst + (double)a[x + N] * g;
                double sprev = (t > 0) ? s[x - N] : (s0 ? s0[bi * N + n] : 0.0);
                if (gated) {
                    if (da) da[x] = g * (sprev - (double)u[x]);
                    if (dbu) dbu[x] = g * (1.0 - (double)a[x]);
                } else {
                    if (da) da[x] = g * sprev;
                    if (dbu) dbu[x] = g;
                }
            }
            if (ds0) ds0[bi * N + n] = (double)a[bi * T * N + n] * g;
        }
    }
}

/* Float order: g_{T-1} = gs + gf (one add), g_t = fma(a_{t+1}, g_{t+1}, gs_t),
 * each gradient product rounded once after its rounded difference. */
static void orc_scan_bwd_f32(int gated, i32 B, i32 T, i32 N, const float* a, const float* u,
                             const float* s0, const float* s, const float* gs, const float* gf,
                             float* da, float* dbu, float* ds0)
{
    for (i64 bi = 0; bi < B; ++bi) {
        for (i64 n = 0; n < N; ++n) {
            float g = 0.0f;
            for (i64 t = T - 1; t >= 0; --t) {
                i64 x = (bi * T + t) * N + n;
                float gst = gs ? gs[x] : 0.0f;
                if (t == T - 1) g = gst + (gf ? gf[bi * N + n] : 0.0f);
                else g = fmaf(a[x + N], g, gst);
                float sprev = (t > 0) ? s[x - N] : (s0 ? s0[bi * N + n] : 0.0f);
                if (gated) {
                    if (da) da[x] = g * (sprev - u[x]);
                    if (dbu) dbu[x] = g * (1.0f - a[x]);
                } else {
                    if (da) da[x] = g * sprev;
                    if (dbu) dbu[x] = g;
                }
            }
            if (ds0) ds0[bi * N + n] = a[bi * T * N + n] * g;
        }
    }
}

void orc_scan_fma_bwd_f64(i32 B, i32 T, i32 N, const float* a, const double* s0, const double* s,
                          const float* gs, const float* gf, double* da, double* db, double* ds0)
{
    orc_scan_bwd_f64(0, B, T, N, a, NULL, s0, s, gs, gf, da, db, ds0);
}

void orc_scan_gated_bwd_f64(i32 B, i32 T, i32 N, const float* a, const float* u, const double* s0,
                            const double* s, const float* gs, const float* gf, double* da, double* du,
                            double* ds0)
{
    orc_scan_bwd_f64(1, B, T, N, a, u, s0, s, gs, gf, da, du, ds0);
}

void orc_scan_fma_bwd_f32(i32 B, i32 T, i32 N, const float* a, const float* s0, const float* s,
                          const float* gs, const float* gf, float* da, float* db, float* ds0)
{
    orc_scan_bwd_f32(0, B, T, N, a, NULL, s0, s, gs, gf, da, db, ds0);
}

void orc_scan_gated_bwd_f32(i32 B, i32 T, i32 N, const float* a, const float* u, const float* s0,
                            const float* s, const float* gs, const float* gf, float* da, float* du,
                            float* ds0)
{
    orc_scan_bwd_f32(1, B, T, N, a, u, s0, s, gs, gf, da, du, ds0);
}

/* ------------------------------------------------------------------------ */
/* Readout epilogues: the step applied to the readout o_t.                   */
/* ------------------------------------------------------------------------ */
/* GLA output: y = RMSNorm(o) * silu(g), normalised first and gated after
 * ([P1] §4.3).  Per row of dv values (one (b, t, h)):
 *     ms  = (1 / dv) * sum_j o_j^2
 *     y_j = o_j / sqrt(ms + eps) * w_j * g_j / (1 + exp(-g_j))
 * with w the norm's per-channel weight (NULL = 1).  In double. */
void orc_readout_norm_gate_f64(i64 rows, i32 dv, const float* o, const float* g, const float* w,
                               double eps, double* y)
{
    for (i64 r = 0; r < rows; ++r) {
        const float* orow = o + r * dv;
        const float* grow = g + r * dv;
        double ms = 0.0;
        for (i32 j = 0; j < dv; ++j) ms += (double)orow[j] * (double)orow[j];
        ms /= (double)dv;
        const double inv = 1.0 / sqrt(ms + eps);
        for (i32 j = 0; j < dv; ++j) {
            const double gj = (double)grow[j];
            const double silu = gj / (1.0 + exp(-gj));
            const double wj = w ? (double)w[j] : 1.0;
            y[r * dv + j] = (double)orow[j] * inv * wj * silu;
        }
    }
}

/* Mamba-2 skip connection: y = o + D_h * x for every row (b, t, h) of dv
 * values, h = row mod H (rows ordered (b, t, h)).  In double. */
void orc_readout_dskip_f64(i64 rows, i32 H, i32 dv, const float* o, const float* x, const float* D, double* y)
{
    for (i64 r = 0; r < rows; ++r) {
        const double dh = (double)D[r % H];
        for (i32 j = 0; j < dv; ++j)
            y[r * dv + j] = (double)o[r * dv + j] + dh * (double)x[r * dv + j];
    }
}
