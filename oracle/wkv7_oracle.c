/*
 * WKV7 oracle: plain, slow, double-precision CPU statement of the RWKV-7
 * WKV7 state recurrence, its exact adjoint and the single-token decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the test suite, the smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * Sources (web pages, cited by title and section):
 *   [timemix]  "Foundry/cuda_kernels/timemix.cu" -- header comment (layouts:
 *              WKV7 vectors [B][T][H][N], state [B][H][N][N]); k_composites
 *              (the kernel's two composite vectors A = -kk, B = kk*a_gate);
 *              the WKV7 launch in tm_fwd_device (one recurrence per (b,h)).
 *   [model]    "infotheory/backends/rwkvzip/rwkv7/model.rs" --
 *              accumulate_token_step_gradients, "WKV kernel backward" block
 *              (state rows = value index, columns = key index; grad_r taken
 *              from the post-update state s_new; u = s_old * kk taken from the
 *              pre-update state; the carried state gradient is scaled by w
 *              per column and receives a rank-1 term along the key vector);
 *              online_train_segment_tbptt (a checkpoint is the state held
 *              before each replay chunk).
 *
 * What is computed, for every (b,h) independently, N = head size:
 *
 *   S <- s0 (or zeros)
 *   for t = 0 .. T-1:
 *       if t % L == 0:  ckpt[t/L] = S                    (state before token t)
 *       sa[i]   = sum_j S[i][j] * a_t[j]                   (pre-update state)
 *       S[i][j] = S[i][j]*w_t[j] + sa[i]*b_t[j] + v_t[i]*k_t[j]
 *       y_t[i]  = sum_j S[i][j] * r_t[j]                   (post-update state)
 *   sT = S
 *
 * The backward is the exact reverse-mode adjoint of those three lines, with
 * every intermediate state kept (no checkpoint replay, no algebraic shortcut).
 * Where the pages are silent, the reading taken is the plainest one: the
 * interval L only decides where checkpoints are copied, s0 == NULL means a
 * zero state and dsT == NULL a zero final-state gradient.
 *
 * Every function returns 0 on success, -1 on a bad argument, -2 when memory
 * cannot be allocated.  Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared.
 */
#include <stdlib.h>
#include <string.h>
#include <stddef.h>

/* offset of element n of token t, head h, batch b in a [B][T][H][N] tensor */
static size_t vec_at(int b, int t, int h, int n, int T, int H, int N)
{
    return (((size_t)b * T + t) * H + h) * N + n;
}

/* offset of state (b,h) in a [B][H][N][N] tensor */
static size_t state_at(int b, int h, int H, int N)
{
    return ((size_t)b * H + h) * N * N;
}

int oracle_ckpt_count(int T, int L)
{
    if (T < 0 || L < 1) return -1;
    return (T + L - 1) / L;
}

/*
 * Forward.  r,w,k,v,a,b,y: [B][T][H][N]; s0, sT: [B][H][N][N] (either may be
 * NULL); ckpt: [B][H][ceil(T/L)][N][N] or NULL.
 */
int oracle_wkv7_forward(int B, int T, int H, int N, int L,
                        const double *r, const double *w, const double *k,
                        const double *v, const double *a, const double *b,
                        const double *s0, double *y, double *sT, double *ckpt)
{
    if (B < 0 || T < 0 || H < 0 || N < 1 || L < 1) return -1;
    double *S = (double *)malloc((size_t)N * N * sizeof(double));
    double *sa = (double *)malloc((size_t)N * sizeof(double));
    if (!S || !sa) { free(S); free(sa); return -2; }
    const int nck = (T + L - 1) / L;

    for (int bi = 0; bi < B; ++bi) {
        for (int h = 0; h < H; ++h) {
            if (s0) memcpy(S, s0 + state_at(bi, h, H, N), (size_t)N * N * sizeof(double));
            else    memset(S, 0, (size_t)N * N * sizeof(double));

            for (int t = 0; t < T; ++t) {
                const size_t o = vec_at(bi, t, h, 0, T, H, N);
                if (ckpt && t % L == 0) {
                    double *dst = ckpt + (((size_t)bi * H + h) * nck + t / L) * N * N;
                    memcpy(dst, S, (size_t)N * N * sizeof(double));
                }
                for (int i = 0; i < N; ++i) {
                    double acc = 0.0;
                    for (int j = 0; j < N; ++j) acc += S[i * N + j] * a[o + j];
                    sa[i] = acc;
                }
                for (int i = 0; i < N; ++i)
                    for (int j = 0; j < N; ++j)
                        S[i * N + j] = S[i * N + j] * w[o + j] + sa[i] * b[o + j] + v[o + i] * k[o + j];
                if (y) {
                    for (int i = 0; i < N; ++i) {
                        double acc = 0.0;
                        for (int j = 0; j < N; ++j) acc += S[i * N + j] * r[o + j];
                        y[o + i] = acc;
                    }
                }
            }
            if (sT) memcpy(sT + state_at(bi, h, H, N), S, (size_t)N * N * sizeof(double));
        }
    }
    free(S);
    free(sa);
    return 0;
}

/*
 * Backward: the adjoint of the forward above.  Inputs as for the forward plus
 * dy [B][T][H][N] and dsT [B][H][N][N] (NULL = zero).  Outputs dr..db
 * [B][T][H][N] are written (not accumulated); ds0 [B][H][N][N] may be NULL.
 *
 * Per (b,h): the states Sh[0..T] (Sh[0] = s0, Sh[t+1] = state after token t)
 * and sa_t are recomputed and kept in full; then, walking t from T-1 down to 0
 * with G = dL/dSh[t+1]:
 *     G      += dy_t r_t^T                 (y_t = Sh[t+1] r_t)
 *     dr_t    = Sh[t+1]^T dy_t
 *     dv_t    = G k_t,     dk_t = G^T v_t,     db_t = G^T sa_t
 *     dsa     = G b_t,     dw_t[j] = sum_i G[i][j] Sh[t][i][j]
 *     da_t    = Sh[t]^T dsa                (sa_t = Sh[t] a_t)
 *     G       = G diag(w_t) + dsa a_t^T    (now dL/dSh[t])
 * and finally ds0 = G.
 */
int oracle_wkv7_backward(int B, int T, int H, int N,
                         const double *r, const double *w, const double *k,
                         const double *v, const double *a, const double *b,
                         const double *s0, const double *dy, const double *dsT,
                         double *dr, double *dw, double *dk, double *dv,
                         double *da, double *db, double *ds0)
{
    if (B < 0 || T < 0 || H < 0 || N < 1) return -1;
    const size_t NN = (size_t)N * N;
    double *Sh = (double *)malloc(((size_t)T + 1) * NN * sizeof(double));
    double *SA = (double *)malloc(((size_t)T + 1) * N * sizeof(double));
    double *G = (double *)malloc(NN * sizeof(double));
    double *dsa = (double *)malloc((size_t)N * sizeof(double));
    if (!Sh || !SA || !G || !dsa) { free(Sh); free(SA); free(G); free(dsa); return -2; }

    for (int bi = 0; bi < B; ++bi) {
        for (int h = 0; h < H; ++h) {
            /* recompute and keep every state */
            if (s0) memcpy(Sh, s0 + state_at(bi, h, H, N), NN * sizeof(double));
            else    memset(Sh, 0, NN * sizeof(double));
            for (int t = 0; t < T; ++t) {
                const size_t o = vec_at(bi, t, h, 0, T, H, N);
                const double *Sp = Sh + (size_t)t * NN;
                double *Sn = Sh + ((size_t)t + 1) * NN;
                double *sa = SA + (size_t)t * N;
                for (int i = 0; i < N; ++i) {
                    double acc = 0.0;
                    for (int j = 0; j < N; ++j) acc += Sp[i * N + j] * a[o + j];
                    sa[i] = acc;
                }
                for (int i = 0; i < N; ++i)
                    for (int j = 0; j < N; ++j)
                        Sn[i * N + j] = Sp[i * N + j] * w[o + j] + sa[i] * b[o + j] + v[o + i] * k[o + j];
            }

            /* reverse sweep */
            if (dsT) memcpy(G, dsT + state_at(bi, h, H, N), NN * sizeof(double));
            else     memset(G, 0, NN * sizeof(double));
            for (int t = T - 1; t >= 0; --t) {
                const size_t o = vec_at(bi, t, h, 0, T, H, N);
                const double *Sp = Sh + (size_t)t * NN;
                const double *Sn = Sh + ((size_t)t + 1) * NN;
                const double *sa = SA + (size_t)t * N;

                for (int i = 0; i < N; ++i)
                    for (int j = 0; j < N; ++j) G[i * N + j] += dy[o + i] * r[o + j];

                for (int j = 0; j < N; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < N; ++i) acc += Sn[i * N + j] * dy[o + i];
                    dr[o + j] = acc;
                }
                for (int i = 0; i < N; ++i) {
                    double acc_v = 0.0, acc_sa = 0.0;
                    for (int j = 0; j < N; ++j) {
                        acc_v += G[i * N + j] * k[o + j];
                        acc_sa += G[i * N + j] * b[o + j];
                    }
                    dv[o + i] = acc_v;
                    dsa[i] = acc_sa;
                }
                for (int j = 0; j < N; ++j) {
                    double acc_k = 0.0, acc_b = 0.0, acc_w = 0.0, acc_a = 0.0;
                    for (int i = 0; i < N; ++i) {
                        acc_k += G[i * N + j] * v[o + i];
                        acc_b += G[i * N + j] * sa[i];
                        acc_w += G[i * N + j] * Sp[i * N + j];
                        acc_a += Sp[i * N + j] * dsa[i];
                    }
                    dk[o + j] = acc_k;
                    db[o + j] = acc_b;
                    dw[o + j] = acc_w;
                    da[o + j] = acc_a;
                }
                for (int i = 0; i < N; ++i)
                    for (int j = 0; j < N; ++j)
                        G[i * N + j] = G[i * N + j] * w[o + j] + dsa[i] * a[o + j];
            }
            if (ds0) memcpy(ds0 + state_at(bi, h, H, N), G, NN * sizeof(double));
        }
    }
    free(Sh);
    free(SA);
    free(G);
    free(dsa);
    return 0;
}

/*
 * Single-token decode (the streaming-inference update of [model], module
 * header: single-token inference is the primary use).  r..b, y: [B][H][N];
 * state: [B][H][N][N], updated in place.  Same arithmetic as one forward step.
 */
int oracle_wkv7_decode_step(int B, int H, int N,
                            const double *r, const double *w, const double *k,
                            const double *v, const double *a, const double *b,
                            double *state, double *y)
{
    if (B < 0 || H < 0 || N < 1 || !state) return -1;
    double *sa = (double *)malloc((size_t)N * sizeof(double));
    if (!sa) return -2;
    for (int bi = 0; bi < B; ++bi) {
        for (int h = 0; h < H; ++h) {
            double *S = state + state_at(bi, h, H, N);
            const size_t o = ((size_t)bi * H + h) * N;
            for (int i = 0; i < N; ++i) {
                double acc = 0.0;
                for (int j = 0; j < N; ++j) acc += S[i * N + j] * a[o + j];
                sa[i] = acc;
            }
            for (int i = 0; i < N; ++i)
                for (int j = 0; j < N; ++j)
                    S[i * N + j] = S[i * N + j] * w[o + j] + sa[i] * b[o + j] + v[o + i] * k[o + j];
            for (int i = 0; i < N; ++i) {
                double acc = 0.0;
                for (int j = 0; j < N; ++j) acc += S[i * N + j] * r[o + j];
                y[o + i] = acc;
            }
        }
    }
    free(sa);
    return 0;
}
