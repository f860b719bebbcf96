/*
 * fp64 CPU oracle for the gated delta rule -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
 * arm may load this library.  The product path (the CUDA library) never calls
 * it and shares no code with it.
 *
 * What it computes: the token-by-token recurrence, exactly as the pages define
 * it, in double precision, one (sequence, head) chain at a time.
 *
 *   "TileLang 实战：KDA 从零到一 -- Gated DeltaNet", opening equation and
 *   §1.1 (table of the three update rules):
 *       S_t = S_{t-1} ( alpha_t (I - beta_t k_t k_t^T) ) + beta_t v_t k_t^T
 *   "Gated Delta Network (GDN)", eq. 4 (same rule) and eq. 12 (decode form,
 *   o_t = S_t q_t: the read happens after the write).
 *   "You Could Have Come Up With Kimi Delta Attention", the five-line
 *   recurrent update in the transposed layout: decay the state first, predict
 *   with the decayed state, form the residual beta (v - prediction), write the
 *   rank-1 correction, then read with scale * q.  KDA replaces the scalar
 *   retention by a per-key-channel vector exp(g_t) that scales the rows (key
 *   channels) of the transposed state.
 *
 * The paper state S is d_v x d_k; like the pages' kernels we hold its
 * transpose h = S^T (d_k x d_v), which is also the API's state layout
 * [N, H, d_k, d_v].  In that layout one step is
 *     h      <- diag(a) h                a = exp(g_t) (scalar or d_k-vector)
 *     p      =  h^T k_t                  (d_v)
 *     r      =  beta_t (v_t - p)
 *     h      <- h + k_t r^T
 *     o_t    =  scale * h^T q_t
 * which expands to alpha S + beta (v - alpha S k) k^T, i.e. the rule above
 * (first page, §2.3, the additive rewrite with d_r).  g is the natural log
 * of the retention (log alpha).
 *
 * Sequences: without cu_seqlens there are B chains per head, each T tokens.
 * With cu_seqlens (B must be 1) sequence n spans tokens [cu[n], cu[n+1]) and
 * its state starts from initial_state[n] -- nothing leaks across a sequence
 * boundary ("Gated Delta Network (GDN)", §6, terminology notes).
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int gdn_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One chain: tokens t0 .. t0+len-1 of batch row b, head hh.
 * Token index t addresses q[((b*T + t)*H + hh)*dk + i]. */
static void run_chain(const double* q, const double* k, const double* v,
                      const double* g, const double* beta, double scale,
                      const double* h0, double* o, double* hT,
                      long b, long t0, long len, long T, long H, long hh,
                      long dk, long dv, int gate_per_channel,
                      double* h, double* p, double* a) {
    if (h0) memcpy(h, h0, sizeof(double) * (size_t)(dk * dv));
    else memset(h, 0, sizeof(double) * (size_t)(dk * dv));

    for (long t = t0; t < t0 + len; ++t) {
        const long tok = (b * T + t) * H + hh;          /* (b, t, hh) */
        const double* kt = k + tok * dk;
        const double* qt = q + tok * dk;
        const double* vt = v + tok * dv;
        double* ot = o + tok * dv;
        const double bt = beta[tok];

        /* retention: scalar exp(g) for GDN, per key channel for KDA */
        if (gate_per_channel) {
            for (long i = 0; i < dk; ++i) a[i] = exp(g[tok * dk + i]);
        } else {
            const double s = exp(g[tok]);
            for (long i = 0; i < dk; ++i) a[i] = s;
        }
        /* forget first: h <- diag(a) h (row i of h is key channel i) */
        for (long i = 0; i < dk; ++i) {
            double* hi = h + i * dv;
            for (long j = 0; j < dv; ++j) hi[j] *= a[i];
        }
        /* predict with the decayed state: p = h^T k */
        for (long j = 0; j < dv; ++j) p[j] = 0.0;
        for (long i = 0; i < dk; ++i) {
            const double ki = kt[i];
            const double* hi = h + i * dv;
            for (long j = 0; j < dv; ++j) p[j] += hi[j] * ki;
        }
        /* residual r = beta (v - p), then the rank-1 write h += k r^T */
        for (long j = 0; j < dv; ++j) p[j] = bt * (vt[j] - p[j]);
        for (long i = 0; i < dk; ++i) {
            const double ki = kt[i];
            double* hi = h + i * dv;
            for (long j = 0; j < dv; ++j) hi[j] += ki * p[j];
        }
        /* read after the write: o = scale * h^T q */
        for (long j = 0; j < dv; ++j) ot[j] = 0.0;
        for (long i = 0; i < dk; ++i) {
            const double qi = qt[i] * scale;
            const double* hi = h + i * dv;
            for (long j = 0; j < dv; ++j) ot[j] += hi[j] * qi;
        }
    }
    if (hT) memcpy(hT, h, sizeof(double) * (size_t)(dk * dv));
}

/*
 * Layouts (row-major, contiguous):
 *   q, k  [B, T, H, dk]      v, o  [B, T, H, dv]
 *   g     [B, T, H]  (gate_per_channel = 0, GDN)  or [B, T, H, dk] (KDA)
 *   beta  [B, T, H]
 *   h0,hT [N, H, dk, dv]     N = n_seqs with cu_seqlens, else B; either may be NULL
 *   cu_seqlens int32 [n_seqs + 1] (host memory) or NULL
 * Returns 0 on success, a negative code for inconsistent arguments.
 * n_threads <= 0 uses the OpenMP default.
 */
int gdn_oracle_forward(const double* q, const double* k, const double* v,
                       const double* g, const double* beta, double scale,
                       const double* h0, double* o, double* hT,
                       const int* cu_seqlens, int n_seqs,
                       int B, int T, int H, int dk, int dv,
                       int gate_per_channel, int n_threads) {
    if (!q || !k || !v || !g || !beta || !o) return -1;
    if (B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0) return -2;
    long N = B;
    if (cu_seqlens) {
        if (B != 1 || n_seqs < 0) return -3;
        if (cu_seqlens[0] != 0 || cu_seqlens[n_seqs] != T) return -4;
        for (int n = 0; n < n_seqs; ++n)
            if (cu_seqlens[n + 1] < cu_seqlens[n]) return -5;
        N = n_seqs;
    }
    const long chains = N * (long)H;
    int rc = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel
    {
        double* h = (double*)malloc(sizeof(double) * (size_t)dk * (size_t)dv);
        double* p = (double*)malloc(sizeof(double) * (size_t)dv);
        double* a = (double*)malloc(sizeof(double) * (size_t)dk);
        const int ok = (h && p && a);
        if (!ok) {
#pragma omp atomic write
            rc = -6;
        }
        /* every thread reaches the work-sharing loop; one without buffers skips */
#pragma omp for schedule(dynamic, 1)
        for (long c = 0; c < chains; ++c) {
            if (!ok) continue;
            const long n = c / H, hh = c % H;
            long b, t0, len;
            if (cu_seqlens) { b = 0; t0 = cu_seqlens[n]; len = cu_seqlens[n + 1] - cu_seqlens[n]; }
            else { b = n; t0 = 0; len = T; }
            const long sidx = (n * H + hh) * (long)dk * dv;
            run_chain(q, k, v, g, beta, scale, h0 ? h0 + sidx : NULL, o,
                      hT ? hT + sidx : NULL, b, t0, len, T, H, hh, dk, dv,
                      gate_per_channel, h, p, a);
        }
        free(h); free(p); free(a);
    }
    return rc;
}

/*
 * Backward of the recurrence above -- the gradients of
 *     L = sum_t <dO_t, o_t> + <dhT, h_final>
 * with respect to q, k, v, g (the log retention), beta and the initial state.
 * The pages print the chunkwise backward of the ungated delta rule
 * ("阅读笔记：DeltaNet 在 FLA 中的代码实现", 二、反向传播, steps 1-6); the
 * gradients themselves are fixed by the forward recurrence, so the oracle
 * takes them by reverse-mode differentiation of the token steps, in the order
 * the forward wrote them:
 *     a   = diag(alpha) h_prev        p = a^T k       r = beta (v - p)
 *     h   = a + k r^T                 o = scale h^T q
 * Walking t from the last token to the first with G = dL/dh_t:
 *     G  += scale q dO^T              dq = scale h dO
 *     dr  = G^T k                     dk = G r + a dp
 *     dbeta = <dr, v - p>             dv = beta dr          dp = -beta dr
 *     da  = G + k dp^T                d alpha_i = sum_j da_ij h_prev_ij
 *     dg  = alpha * d alpha (per channel; summed over channels for GDN)
 *     G  <- diag(alpha) da            (dL/dh_prev)
 * and the initial state's gradient is the final G.  Every state of the chain
 * is kept (len + 1 of them), so this is for the small sizes the tests use.
 */
static int back_chain(const double* q, const double* k, const double* v,
                      const double* g, const double* beta, double scale,
                      const double* h0, const double* dout, const double* dhT,
                      double* dq, double* dkk, double* dvv, double* dg, double* dbeta,
                      double* dh0, long b, long t0, long len, long T, long H,
                      long hh, long dk, long dv, int gate_per_channel) {
    const size_t S = (size_t)dk * (size_t)dv;
    double* hs = (double*)malloc(sizeof(double) * S * (size_t)(len + 1));
    double* G = (double*)malloc(sizeof(double) * S);
    double* a = (double*)malloc(sizeof(double) * S);
    double* al = (double*)malloc(sizeof(double) * (size_t)dk);
    double* p = (double*)malloc(sizeof(double) * (size_t)dv);
    double* r = (double*)malloc(sizeof(double) * (size_t)dv);
    double* dr = (double*)malloc(sizeof(double) * (size_t)dv);
    double* dp = (double*)malloc(sizeof(double) * (size_t)dv);
    if (!hs || !G || !a || !al || !p || !r || !dr || !dp) {
        free(hs); free(G); free(a); free(al); free(p); free(r); free(dr); free(dp);
        return -6;
    }
    /* forward, keeping h_{t0-1+s} in hs[s] */
    if (h0) memcpy(hs, h0, sizeof(double) * S);
    else memset(hs, 0, sizeof(double) * S);
    for (long s = 0; s < len; ++s) {
        const long tok = (b * T + t0 + s) * H + hh;
        const double* kt = k + tok * dk;
        const double* vt = v + tok * dv;
        const double bt = beta[tok];
        const double* hp = hs + (size_t)s * S;
        double* hn = hs + (size_t)(s + 1) * S;
        for (long i = 0; i < dk; ++i)
            al[i] = exp(gate_per_channel ? g[tok * dk + i] : g[tok]);
        for (long j = 0; j < dv; ++j) p[j] = 0.0;
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) p[j] += al[i] * hp[i * dv + j] * kt[i];
        for (long j = 0; j < dv; ++j) r[j] = bt * (vt[j] - p[j]);
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) hn[i * dv + j] = al[i] * hp[i * dv + j] + kt[i] * r[j];
    }
    /* backward */
    if (dhT) memcpy(G, dhT, sizeof(double) * S);
    else memset(G, 0, sizeof(double) * S);
    for (long s = len - 1; s >= 0; --s) {
        const long tok = (b * T + t0 + s) * H + hh;
        const double* kt = k + tok * dk;
        const double* qt = q + tok * dk;
        const double* vt = v + tok * dv;
        const double* dot = dout + tok * dv;
        const double bt = beta[tok];
        const double* hp = hs + (size_t)s * S;        /* h_{t-1} */
        const double* hn = hs + (size_t)(s + 1) * S;  /* h_t */
        for (long i = 0; i < dk; ++i)
            al[i] = exp(gate_per_channel ? g[tok * dk + i] : g[tok]);
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) a[i * dv + j] = al[i] * hp[i * dv + j];
        for (long j = 0; j < dv; ++j) p[j] = 0.0;
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) p[j] += a[i * dv + j] * kt[i];
        for (long j = 0; j < dv; ++j) r[j] = bt * (vt[j] - p[j]);
        /* the read o = scale h^T q */
        for (long i = 0; i < dk; ++i) {
            double sq = 0.0;
            for (long j = 0; j < dv; ++j) {
                G[i * dv + j] += scale * qt[i] * dot[j];
                sq += hn[i * dv + j] * dot[j];
            }
            dq[tok * dk + i] = scale * sq;
        }
        /* the write h = a + k r^T */
        for (long j = 0; j < dv; ++j) {
            double s2 = 0.0;
            for (long i = 0; i < dk; ++i) s2 += G[i * dv + j] * kt[i];
            dr[j] = s2;
        }
        double db = 0.0;
        for (long j = 0; j < dv; ++j) {
            db += dr[j] * (vt[j] - p[j]);
            dvv[tok * dv + j] = bt * dr[j];
            dp[j] = -bt * dr[j];
        }
        dbeta[tok] = db;
        double dgs = 0.0;
        for (long i = 0; i < dk; ++i) {
            double kd = 0.0, sa = 0.0;
            for (long j = 0; j < dv; ++j) {
                kd += G[i * dv + j] * r[j] + a[i * dv + j] * dp[j];
                const double dai = G[i * dv + j] + kt[i] * dp[j];   /* dL/da */
                sa += dai * hp[i * dv + j];
                G[i * dv + j] = al[i] * dai;                        /* dL/dh_{t-1} */
            }
            dkk[tok * dk + i] = kd;
            if (gate_per_channel) dg[tok * dk + i] = al[i] * sa;
            else dgs += al[i] * sa;
        }
        if (!gate_per_channel) dg[tok] = dgs;
    }
    if (dh0) memcpy(dh0, G, sizeof(double) * S);
    free(hs); free(G); free(a); free(al); free(p); free(r); free(dr); free(dp);
    return 0;
}

/*
 * Layouts as gdn_oracle_forward, plus
 *   dout  [B, T, H, dv] (dL/do)        dhT [N, H, dk, dv] or NULL (dL/d final state)
 *   dq, dk [B, T, H, dk]   dv [B, T, H, dv]   dg like g   dbeta [B, T, H]
 *   dh0   [N, H, dk, dv] or NULL
 */
int gdn_oracle_backward(const double* q, const double* k, const double* v,
                        const double* g, const double* beta, double scale,
                        const double* h0, const double* dout, const double* dhT,
                        double* dq, double* dk_out, double* dv_out, double* dg,
                        double* dbeta, double* dh0,
                        const int* cu_seqlens, int n_seqs,
                        int B, int T, int H, int dk, int dv,
                        int gate_per_channel, int n_threads) {
    if (!q || !k || !v || !g || !beta || !dout || !dq || !dk_out || !dv_out || !dg || !dbeta) return -1;
    if (B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0) return -2;
    long N = B;
    if (cu_seqlens) {
        if (B != 1 || n_seqs < 0) return -3;
        if (cu_seqlens[0] != 0 || cu_seqlens[n_seqs] != T) return -4;
        for (int n = 0; n < n_seqs; ++n)
            if (cu_seqlens[n + 1] < cu_seqlens[n]) return -5;
        N = n_seqs;
    }
    const long chains = N * (long)H;
    int rc = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (long c = 0; c < chains; ++c) {
        const long n = c / H, hh = c % H;
        long b, t0, len;
        if (cu_seqlens) { b = 0; t0 = cu_seqlens[n]; len = cu_seqlens[n + 1] - cu_seqlens[n]; }
        else { b = n; t0 = 0; len = T; }
        const long sidx = (n * H + hh) * (long)dk * dv;
        const int e = back_chain(q, k, v, g, beta, scale, h0 ? h0 + sidx : NULL, dout,
                                 dhT ? dhT + sidx : NULL, dq, dk_out, dv_out, dg, dbeta,
                                 dh0 ? dh0 + sidx : NULL, b, t0, len, T, H, hh, dk, dv,
                                 gate_per_channel);
        if (e) {
#pragma omp atomic write
            rc = e;
        }
    }
    return rc;
}
