/*
 * iha_oracle.c -- plain fp64 CPU oracle for the Interleaved Head Attention (IHA)
 * forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or load
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header or table with the CUDA library.
 *
 * Sources (cited by page title and section):
 *   [IHA]  "交錯頭注意力機制" -- summary of "Interleaved Head Attention"
 *          (Duvvuri et al., arXiv 2602.21371v1), section 4, Algorithm 1
 *          (pseudo-head mixing, stacking, per-head attention, unstack and
 *          R contraction, head concatenation); section 3.1 Definition 1 (MHA).
 *   [ATT]  "注意力机制" (llm-from-scratch, chapter 5): eq. (5.9) softmax read,
 *          eq. (5.11) softmax on the allowed set, Algorithm 5.1 (strict
 *          single-head attention with finite checks and row sums), eq. (5.12)
 *          causality by absolute position.
 *
 * Mask convention (Algorithm 1 itself has no mask; the figure caption of [IHA]
 * section 4 speaks of a sliding window): stacked pseudo-token (j, t) may read
 * pseudo-token (j', t') iff
 *      mode 0: always;
 *      mode 1: t' <= t;
 *      mode 2: t' <= t and t - t' < window.
 * The mask depends on original token positions only, never on the stacked row
 * index ([ATT] eq. (5.12): visibility by absolute position).
 *
 * Arithmetic: every value in double; inputs are the exact values a device would
 * receive (bf16 or fp32 values widened to double).  Loops follow the pages'
 * formulas literally; the only freedom taken is loop order for memory streaming
 * in the projection (a sum over k is a sum over k).
 *
 * Every function here is pinned by tests against values the pages print, closed
 * forms and invariants (see tests/test_oracle_pins.py).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_EINVAL (-1)
#define OR_EEMPTY (-2)   /* a legal query row with an empty allowed set ([ATT] Alg. 5.1) */
#define OR_ENONFINITE (-3)
#define OR_EROWSUM (-4)
#define OR_ENOMEM (-5)

typedef long long i64;

/* ------------------------------------------------------------------------- */
/* Softmax read on an allowed set: [ATT] eq. (5.11), Algorithm 5.1 steps 3-5. */
/* u[S]: scaled scores; allowed[S]: 1 = may read; V[S][dv] row-major.          */
/* Writes a[S] (0 on forbidden positions) if a != NULL, and o[dv].            */
/* ------------------------------------------------------------------------- */
int iha_oracle_softmax_read(const double *u, const unsigned char *allowed, int S,
                            const double *V, int dv, double *a, double *o)
{
    if (S <= 0 || dv <= 0 || !u || !allowed || !V || !o) return OR_EINVAL;
    int any = 0;
    double c = -INFINITY;
    for (int j = 0; j < S; j++) {
        if (!allowed[j]) continue;
        if (!isfinite(u[j])) return OR_ENONFINITE;
        if (!any || u[j] > c) c = u[j];
        any = 1;
    }
    if (!any) return OR_EEMPTY;
    double z = 0.0;
    for (int j = 0; j < S; j++)
        if (allowed[j]) z += exp(u[j] - c);
    /* at least one term equals exp(0) = 1, so z >= 1 */
    for (int r = 0; r < dv; r++) o[r] = 0.0;
    double rowsum = 0.0;
    for (int j = 0; j < S; j++) {
        double aj = allowed[j] ? exp(u[j] - c) / z : 0.0;
        if (a) a[j] = aj;
        rowsum += aj;
        if (aj != 0.0)
            for (int r = 0; r < dv; r++) o[r] += aj * V[(i64)j * dv + r];
    }
    if (fabs(rowsum - 1.0) > 1e-12) return OR_EROWSUM;
    return OR_OK;
}

/* may stacked token at original position tq read the one at tk? */
static int visible(int mask_mode, int window, int tq, int tk)
{
    if (mask_mode == 0) return 1;
    if (tk > tq) return 0;
    if (mask_mode == 2 && tq - tk >= window) return 0;
    return 1;
}

/* ------------------------------------------------------------------------- */
/* simple static-stride parallel for                                          */
/* ------------------------------------------------------------------------- */
typedef void (*item_fn)(void *ctx, i64 item);
typedef struct { item_fn fn; void *ctx; i64 n; int tid, nth; } pf_arg;

static void *pf_worker(void *p)
{
    pf_arg *a = (pf_arg *)p;
    for (i64 i = a->tid; i < a->n; i += a->nth) a->fn(a->ctx, i);
    return NULL;
}

static void parallel_for(i64 n, int nthreads, item_fn fn, void *ctx)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((i64)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    pthread_t th[256];
    pf_arg args[256];
    int started[256];
    for (int t = 0; t < nthreads; t++) {
        args[t].fn = fn; args[t].ctx = ctx; args[t].n = n;
        args[t].tid = t; args[t].nth = nthreads;
        started[t] = (t > 0) && pthread_create(&th[t], NULL, pf_worker, &args[t]) == 0;
    }
    /* thread 0 runs inline; any thread that failed to start runs inline too */
    for (int t = 0; t < nthreads; t++)
        if (!started[t]) pf_worker(&args[t]);
    for (int t = 1; t < nthreads; t++)
        if (started[t]) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------------- */
/* IHA forward, Algorithm 1 of [IHA] section 4.                               */
/* ------------------------------------------------------------------------- */
typedef struct {
    /* problem */
    const double *X, *W[3], *alpha[3], *R;
    const double *XW[3];   /* optional precomputed X W_s, [B][N][H*d]; NULL = compute here */
    int B, N, H, d, P, mask_mode, window, stack_order;
    /* current batch element and token sets */
    int b;
    int ntq;          /* number of query tokens */
    const int *tq;    /* query tokens, ascending */
    int klo, khi;     /* key/value tokens needed: [klo, khi] */
    /* workspaces */
    double *proj[3];  /* [s]: unmixed X W^(m): [H][ntok][d], tokens indexed by slot */
    double *mixed[3]; /* [s]: pseudo-heads Q~_{h,j}: [H][P][ntok][d] */
    int nslot;        /* number of token slots = khi - klo + 1 */
    int *tok_of;      /* slot -> token (klo + slot) */
    double *pbar;     /* P-bar rows of queried tokens: [H][P][ntq][d] */
    double *weights;  /* optional [H][PN][PN] in stacked order (full runs only) */
    int err;
    pthread_mutex_t lock;
} fwd_ctx;

static void set_err(fwd_ctx *c, int e)
{
    pthread_mutex_lock(&c->lock);
    if (c->err == OR_OK) c->err = e;
    pthread_mutex_unlock(&c->lock);
}

/* Step "pseudo-head mixing", first half: X W_s^(m) for every head m and every
 * needed token (one item = one token slot, all three of Q, K, V). */
static void item_project(void *vc, i64 slot)
{
    fwd_ctx *c = (fwd_ctx *)vc;
    const int D = c->H * c->d, Hd = c->H * c->d, H = c->H, d = c->d;
    const int t = c->tok_of[slot];
    const double *x = c->X ? c->X + ((i64)c->b * c->N + t) * D : NULL;
    double *acc = (double *)malloc(sizeof(double) * Hd);
    if (!acc) { set_err(c, OR_ENOMEM); return; }
    for (int s = 0; s < 3; s++) {
        if (c->XW[s]) {
            /* projections supplied by the caller (a library matmul) */
            memcpy(acc, c->XW[s] + ((i64)c->b * c->N + t) * Hd, sizeof(double) * Hd);
        } else {
            /* acc[col] = sum_k x[k] * W[k][col], col = m*d + cc (column block m = W^(m)) */
            for (int col = 0; col < Hd; col++) acc[col] = 0.0;
            for (int k = 0; k < D; k++) {
                const double xk = x[k];
                const double *wrow = c->W[s] + (i64)k * Hd;
                for (int col = 0; col < Hd; col++) acc[col] += xk * wrow[col];
            }
        }
        for (int m = 0; m < H; m++)
            for (int cc = 0; cc < d; cc++)
                c->proj[s][((i64)m * c->nslot + slot) * d + cc] = acc[m * d + cc];
    }
    free(acc);
}

/* Step "pseudo-head mixing", second half:
 *   Q~_{h,j}[t] = sum_m alpha_Q[m][h][j] * (X W_Q^(m))[t]   (same for K, V). */
static void item_mix(void *vc, i64 slot)
{
    fwd_ctx *c = (fwd_ctx *)vc;
    const int H = c->H, P = c->P, d = c->d;
    for (int s = 0; s < 3; s++)
        for (int h = 0; h < H; h++)
            for (int j = 0; j < P; j++) {
                double *dst = c->mixed[s] + (((i64)h * P + j) * c->nslot + slot) * d;
                for (int cc = 0; cc < d; cc++) dst[cc] = 0.0;
                for (int m = 0; m < H; m++) {
                    const double a = c->alpha[s][((i64)m * H + h) * P + j];
                    const double *src = c->proj[s] + ((i64)m * c->nslot + slot) * d;
                    for (int cc = 0; cc < d; cc++) dst[cc] += a * src[cc];
                }
            }
}

/* Stacking: the stacked sequence of head h has length P*N.
 * stack_order 0 (Algorithm 1 as printed, row concatenation):
 *     row = j*N + t.
 * stack_order 1 (interleaved, as the figure caption words it):
 *     row = t*P + j.
 * Both carry the original position t with the row; the mask reads only t. */
static i64 stacked_row(const fwd_ctx *c, int j, int t)
{
    return c->stack_order == 0 ? (i64)j * c->N + t : (i64)t * c->P + j;
}

/* Step "attention (per head)": for head h and stacked query row (j, t):
 *   S_h = Q-bar_h K-bar_h^T / sqrt(d);  P-bar_h = softmax(S_h) V-bar_h,
 * the softmax taken over the allowed set of [ATT] eq. (5.11).
 * One item = (h, query token index qi); all P rows j of that token.
 * The key rows of head h are visited in stacked order (j-major for
 * stack_order 0, t-major for 1). */
static void item_attend(void *vc, i64 item)
{
    fwd_ctx *c = (fwd_ctx *)vc;
    const int P = c->P, d = c->d, N = c->N;
    const int h = (int)(item / c->ntq), qi = (int)(item % c->ntq);
    const int t = c->tq[qi];
    const int nt = c->nslot;              /* key tokens klo..khi, slot = t2 - klo */
    const int nk = nt * P;                /* key rows of the stacked sequence */
    const double scale = 1.0 / sqrt((double)d);
    const double *Kh = c->mixed[1] + (i64)h * P * nt * d;   /* [P][nt][d] */
    const double *Vh = c->mixed[2] + (i64)h * P * nt * d;
    double *u = (double *)malloc(sizeof(double) * nk);
    double *a = (double *)malloc(sizeof(double) * nk);
    unsigned char *al = (unsigned char *)malloc(nk);
    double *vt = NULL;                    /* t-major copy of V-bar_h (stack_order 1) */
    if (!u || !a || !al) { set_err(c, OR_ENOMEM); goto done; }
    if (c->stack_order == 1) {
        vt = (double *)malloc(sizeof(double) * (i64)nk * d);
        if (!vt) { set_err(c, OR_ENOMEM); goto done; }
        for (int s2 = 0; s2 < nt; s2++)
            for (int j2 = 0; j2 < P; j2++)
                memcpy(vt + ((i64)s2 * P + j2) * d, Vh + ((i64)j2 * nt + s2) * d, sizeof(double) * d);
    }

    for (int j = 0; j < P; j++) {
        const double *q = c->mixed[0] + (((i64)h * P + j) * nt + (t - c->klo)) * d;
        for (int n = 0; n < nk; n++) {
            const int j2 = c->stack_order == 0 ? n / nt : n % P;
            const int s2 = c->stack_order == 0 ? n % nt : n / P;
            const double *k = Kh + ((i64)j2 * nt + s2) * d;
            double dot = 0.0;
            for (int cc = 0; cc < d; cc++) dot += q[cc] * k[cc];
            u[n] = dot * scale;
            al[n] = (unsigned char)visible(c->mask_mode, c->window, t, c->klo + s2);
        }
        double *o = c->pbar + (((i64)h * P + j) * c->ntq + qi) * d;
        int e = iha_oracle_softmax_read(u, al, nk, c->stack_order == 0 ? Vh : vt, d, a, o);
        if (e != OR_OK) { set_err(c, e); goto done; }
        if (c->weights) {
            const i64 PN = (i64)P * N;
            double *wrow = c->weights + ((i64)h * PN + stacked_row(c, j, t)) * PN;
            for (int n = 0; n < nk; n++) {
                const int j2 = c->stack_order == 0 ? n / nt : n % P;
                const int s2 = c->stack_order == 0 ? n % nt : n / P;
                wrow[stacked_row(c, j2, c->klo + s2)] = a[n];
            }
        }
    }
done:
    free(u); free(a); free(al); free(vt);
}

/* Steps "unstack and contract (HP -> H)" and "concatenate heads":
 *   O_h[t] = sum_{h'} sum_j R[h][h'*P + j] * P_{h',j}[t]   (0-based indices),
 * where P_{h',j} is the j-th length-N block of P-bar_{h'} (unstacking);
 *   X~[t] = [O_1[t], ..., O_H[t]].  One item = one query token. */
typedef struct { fwd_ctx *c; double *out; i64 out_row0; } contract_ctx;
static void item_contract(void *vc, i64 qi)
{
    contract_ctx *cc = (contract_ctx *)vc;
    fwd_ctx *c = cc->c;
    const int H = c->H, P = c->P, d = c->d;
    double *dst = cc->out + (cc->out_row0 + qi) * (i64)H * d;
    for (int h = 0; h < H; h++) {
        double *oh = dst + (i64)h * d;
        for (int r = 0; r < d; r++) oh[r] = 0.0;
        for (int h2 = 0; h2 < H; h2++)
            for (int j = 0; j < P; j++) {
                const double rr = c->R[(i64)h * (H * P) + h2 * P + j];
                const double *pb = c->pbar + (((i64)h2 * P + j) * c->ntq + qi) * d;
                for (int r = 0; r < d; r++) oh[r] += rr * pb[r];
            }
    }
}

/*
 * iha_oracle_forward
 *   X      [B][N][D]      D = H*d
 *   W_s    [D][H*d]       column block m (columns m*d .. m*d+d-1) is W_s^(m)
 *   alpha_s [H][H][P]     alpha_s[m][h][j]
 *   R      [H][H*P]       R[h][h'*P + j]
 *   sel    optional list of n_sel output rows (b*N + t), each b's tokens ascending;
 *          NULL = every (b, t) in order.
 *   out    [n_sel or B*N][H*d]
 *   weights optional [B][H][P*N][P*N] attention weights in stacked order
 *          (only with sel == NULL).
 * Returns 0 or a negative error code.
 */
static int forward_impl(const double *X, const double *W_Q, const double *W_K, const double *W_V,
                        const double *XW_Q, const double *XW_K, const double *XW_V,
                        const double *alpha_Q, const double *alpha_K, const double *alpha_V,
                        const double *R, int B, int N, int H, int d, int P,
                        int mask_mode, int window, int stack_order,
                        const i64 *sel, int n_sel, double *out, double *weights, int nthreads)
{
    if (!alpha_Q || !alpha_K || !alpha_V || !R || !out) return OR_EINVAL;
    if (B <= 0 || N <= 0 || H <= 0 || d <= 0 || P <= 0) return OR_EINVAL;
    if (mask_mode < 0 || mask_mode > 2) return OR_EINVAL;
    if (mask_mode == 2 && window < 1) return OR_EINVAL;
    if (stack_order != 0 && stack_order != 1) return OR_EINVAL;
    if (sel && weights) return OR_EINVAL;
    if (sel && n_sel <= 0) return OR_EINVAL;

    fwd_ctx c;
    memset(&c, 0, sizeof c);
    c.X = X; c.W[0] = W_Q; c.W[1] = W_K; c.W[2] = W_V;
    c.XW[0] = XW_Q; c.XW[1] = XW_K; c.XW[2] = XW_V;
    c.alpha[0] = alpha_Q; c.alpha[1] = alpha_K; c.alpha[2] = alpha_V; c.R = R;
    c.B = B; c.N = N; c.H = H; c.d = d; c.P = P;
    c.mask_mode = mask_mode; c.window = window; c.stack_order = stack_order;
    pthread_mutex_init(&c.lock, NULL);

    const i64 total = sel ? n_sel : (i64)B * N;
    int *tq = (int *)malloc(sizeof(int) * N);
    c.tok_of = (int *)malloc(sizeof(int) * N);
    if (!tq || !c.tok_of) { free(tq); free(c.tok_of); return OR_ENOMEM; }
    int rc = OR_OK;

    i64 pos = 0;   /* next entry of sel (or of the full enumeration) */
    while (pos < total && rc == OR_OK) {
        /* gather the query tokens of the next batch element */
        const i64 first = sel ? sel[pos] : pos;
        if (first < 0 || first >= (i64)B * N) { rc = OR_EINVAL; break; }
        const int b = (int)(first / N);
        i64 end = pos;
        int nq = 0;
        while (end < total) {
            const i64 r = sel ? sel[end] : end;
            if (r < 0 || r >= (i64)B * N) { rc = OR_EINVAL; break; }
            if ((int)(r / N) != b) break;
            const int t = (int)(r % N);
            if (nq > 0 && t <= tq[nq - 1]) { rc = OR_EINVAL; break; }  /* ascending */
            tq[nq++] = t;
            end++;
        }
        if (rc != OR_OK) break;

        /* key/value tokens any of these queries can read */
        int klo = 0, khi = N - 1;
        if (mask_mode >= 1) khi = tq[nq - 1];
        if (mask_mode == 2) { klo = tq[0] - window + 1; if (klo < 0) klo = 0; }

        /* token slots: the key range; every query token lies inside it
         * (mode 0: all tokens; modes 1, 2: klo <= tq[0] and khi = tq[nq-1]) */
        int ns = 0;
        for (int t = klo; t <= khi; t++) c.tok_of[ns++] = t;

        c.b = b; c.ntq = nq; c.tq = tq; c.klo = klo; c.khi = khi; c.nslot = ns;
        const i64 pe = (i64)H * ns * d, me = (i64)H * P * ns * d;
        for (int s = 0; s < 3; s++) {
            c.proj[s] = (double *)malloc(sizeof(double) * pe);
            c.mixed[s] = (double *)malloc(sizeof(double) * me);
        }
        c.pbar = (double *)malloc(sizeof(double) * (i64)H * P * nq * d);
        c.weights = weights ? weights + (i64)b * H * ((i64)P * N) * ((i64)P * N) : NULL;
        int ok = c.pbar != NULL;
        for (int s = 0; s < 3; s++) ok = ok && c.proj[s] && c.mixed[s];
        if (!ok) rc = OR_ENOMEM;

        if (rc == OR_OK) {
            c.err = OR_OK;
            parallel_for(ns, nthreads, item_project, &c);
            if (c.err == OR_OK) parallel_for(ns, nthreads, item_mix, &c);
            if (c.err == OR_OK) parallel_for((i64)H * nq, nthreads, item_attend, &c);
            if (c.err == OR_OK) {
                contract_ctx cc = { &c, out, pos };
                parallel_for(nq, nthreads, item_contract, &cc);
            }
            rc = c.err;
        }
        for (int s = 0; s < 3; s++) { free(c.proj[s]); free(c.mixed[s]); c.proj[s] = c.mixed[s] = NULL; }
        free(c.pbar); c.pbar = NULL;
        pos = end;
    }
    free(tq); free(c.tok_of);
    pthread_mutex_destroy(&c.lock);
    return rc;
}

int iha_oracle_forward(const double *X, const double *W_Q, const double *W_K, const double *W_V,
                       const double *alpha_Q, const double *alpha_K, const double *alpha_V,
                       const double *R, int B, int N, int H, int d, int P,
                       int mask_mode, int window, int stack_order,
                       const i64 *sel, int n_sel, double *out, double *weights, int nthreads)
{
    if (!X || !W_Q || !W_K || !W_V) return OR_EINVAL;
    return forward_impl(X, W_Q, W_K, W_V, NULL, NULL, NULL, alpha_Q, alpha_K, alpha_V, R,
                        B, N, H, d, P, mask_mode, window, stack_order, sel, n_sel, out, weights, nthreads);
}

/* The same forward pass starting from the per-head projections: XW_s [B][N][H*d]
 * holds X W_s, whose column block m is X W_s^(m) (the first half of the mixing step). */
int iha_oracle_forward_from_projections(const double *XW_Q, const double *XW_K, const double *XW_V,
                                        const double *alpha_Q, const double *alpha_K, const double *alpha_V,
                                        const double *R, int B, int N, int H, int d, int P,
                                        int mask_mode, int window, int stack_order,
                                        const i64 *sel, int n_sel, double *out, double *weights, int nthreads)
{
    if (!XW_Q || !XW_K || !XW_V) return OR_EINVAL;
    return forward_impl(NULL, NULL, NULL, NULL, XW_Q, XW_K, XW_V, alpha_Q, alpha_K, alpha_V, R,
                        B, N, H, d, P, mask_mode, window, stack_order, sel, n_sel, out, weights, nthreads);
}

/* ------------------------------------------------------------------------- */
/* Plain multi-head attention, [IHA] section 3.1 Definition 1, written on its */
/* own (no code shared with the IHA routine above) so that IHA's inclusion of */
/* MHA (Theorem 2) can be checked between two independent loops:              */
/*   head_m = softmax(X W_Q^(m) (X W_K^(m))^T / sqrt(d)) X W_V^(m),           */
/*   MHA(X) = [head_1, ..., head_H],                                          */
/* with the same by-position mask (modes 0, 1, 2).                            */
/* ------------------------------------------------------------------------- */
typedef struct {
    const double *X, *WQ, *WK, *WV;
    int B, N, H, d, mask_mode, window;
    const i64 *sel; int n_sel;
    double *out;
    int err;
} mha_ctx;

static void mha_item(void *vc, i64 item)
{
    mha_ctx *c = (mha_ctx *)vc;
    const int H = c->H, d = c->d, N = c->N, D = H * d, Hd = H * d;
    const i64 row = c->sel ? c->sel[item] : item;
    const int b = (int)(row / N), t = (int)(row % N);
    double *q = (double *)malloc(sizeof(double) * d);
    double *kv = (double *)malloc(sizeof(double) * 2 * d);
    double *sc = (double *)malloc(sizeof(double) * N);
    double *vals = (double *)malloc(sizeof(double) * (i64)N * d);
    if (!q || !kv || !sc || !vals) { c->err = OR_ENOMEM; goto done; }
    for (int m = 0; m < H; m++) {
        const double *xt = c->X + ((i64)b * N + t) * D;
        for (int cc = 0; cc < d; cc++) {
            double s = 0.0;
            for (int k = 0; k < D; k++) s += xt[k] * c->WQ[(i64)k * Hd + m * d + cc];
            q[cc] = s;
        }
        double best = -INFINITY;
        int nvis = 0;
        for (int t2 = 0; t2 < N; t2++) {
            int vis = 1;
            if (c->mask_mode >= 1 && t2 > t) vis = 0;
            if (c->mask_mode == 2 && t - t2 >= c->window) vis = 0;
            if (!vis) { sc[t2] = NAN; continue; }
            const double *x2 = c->X + ((i64)b * N + t2) * D;
            for (int cc = 0; cc < d; cc++) {
                double sk = 0.0, sv = 0.0;
                for (int k = 0; k < D; k++) {
                    sk += x2[k] * c->WK[(i64)k * Hd + m * d + cc];
                    sv += x2[k] * c->WV[(i64)k * Hd + m * d + cc];
                }
                kv[cc] = sk;
                vals[(i64)t2 * d + cc] = sv;
            }
            double dot = 0.0;
            for (int cc = 0; cc < d; cc++) dot += q[cc] * kv[cc];
            sc[t2] = dot / sqrt((double)d);
            if (sc[t2] > best) best = sc[t2];
            nvis++;
        }
        if (nvis == 0) { c->err = OR_EEMPTY; goto done; }
        double z = 0.0;
        for (int t2 = 0; t2 < N; t2++) if (!isnan(sc[t2])) z += exp(sc[t2] - best);
        double *o = c->out + (c->sel ? item : row) * (i64)D + (i64)m * d;
        for (int cc = 0; cc < d; cc++) o[cc] = 0.0;
        for (int t2 = 0; t2 < N; t2++) {
            if (isnan(sc[t2])) continue;
            const double w = exp(sc[t2] - best) / z;
            for (int cc = 0; cc < d; cc++) o[cc] += w * vals[(i64)t2 * d + cc];
        }
    }
done:
    free(q); free(kv); free(sc); free(vals);
}

int iha_oracle_mha(const double *X, const double *W_Q, const double *W_K, const double *W_V,
                   int B, int N, int H, int d, int mask_mode, int window,
                   const i64 *sel, int n_sel, double *out, int nthreads)
{
    if (!X || !W_Q || !W_K || !W_V || !out) return OR_EINVAL;
    if (B <= 0 || N <= 0 || H <= 0 || d <= 0) return OR_EINVAL;
    if (mask_mode < 0 || mask_mode > 2 || (mask_mode == 2 && window < 1)) return OR_EINVAL;
    mha_ctx c = { X, W_Q, W_K, W_V, B, N, H, d, mask_mode, window, sel, n_sel, out, OR_OK };
    parallel_for(sel ? n_sel : (i64)B * N, nthreads, mha_item, &c);
    return c.err;
}

/* Parameter count of one IHA module ([IHA] Theorem 2): the element counts of
 * the arrays iha_oracle_forward reads besides X -- three projections W_s of
 * D x (H d), three mixing tensors alpha_s of H x H x P, and R of H x (H P). */
long long iha_oracle_param_count(int D, int H, int d, int P)
{
    const long long proj = 3LL * D * ((long long)H * d);
    const long long mix = 3LL * H * H * P;
    const long long contract = (long long)H * ((long long)H * P);
    return proj + mix + contract;
}
