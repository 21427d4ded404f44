/*
 * conv_oracle.c -- CPU oracle for the 2-D convolution forward pass (FPROP).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or table with the CUDA
 * library.
 *
 * What it computes (the plain definition, written out):
 *
 *   y[n,k,p,q] = act( alpha * sum_{c<C} sum_{r<R} sum_{s<S}
 *                        X(n, c, p*u + r*dh - pad_top, q*v + s*dw - pad_left) * w[k,c,r,s]
 *                     + beta * y_in[n,k,p,q] + bias[k] )
 *
 * with X(...) = 0 outside [0,H) x [0,W) (zero padding) and act = identity or
 * max(0, .).  Sources:
 *   - "maxDNN: An Efficient Convolution Kernel for Deep Learning with Maxwell
 *     GPUs", method section: every output coordinate is the product of the
 *     input receptive field with the filter weights (a dot product over
 *     c, r, s).
 *   - "cuDNN: Efficient Primitives for Deep Learning", method section: tensors
 *     and filters are addressed through descriptors with arbitrary strides;
 *     non-square inputs and asymmetric padding are supported (method and
 *     findings sections).
 *   - "High Performance Zero-Memory Overhead Direct Convolutions", method
 *     section: direct convolution, no packing.
 * The filter is not flipped (cross-correlation).  Dilation enters as r*dh and
 * s*dw, and the output extent uses the dilated filter extent dh*(R-1)+1 with
 * a floor: a partial last window is dropped.  Bottom/right padding only
 * changes the output extent.
 *
 * All arithmetic is FP64, in the loop order n, k, p, q, c, r, s, on the
 * values given (the caller passes the same BF16/TF32-rounded inputs the GPU
 * reads, widened exactly to double).  Alongside y it returns
 * bound[n,k,p,q] = sum |x*w| (FP64), the scale of the parity tolerance.
 *
 * Element addresses go through caller-given strides (in elements), so a
 * layout (NCHW, NHWC, a padded view) changes addressing only.
 *
 * Threads: plain pthreads split the (n,k) pairs; the thread count is the
 * caller's.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

typedef long long i64;

typedef struct {
    const double *x;
    i64 xs[4];            /* strides of x for n, c, h, w */
    const double *w;
    i64 ws[4];            /* strides of w for k, c, r, s */
    double *y;            /* output, strides ys for n, k, p, q */
    i64 ys[4];
    double *bound;        /* sum |x*w|, same strides as y; may be NULL */
    const double *y_in;   /* beta term input, same strides as y; may be NULL */
    const double *bias;   /* K values; may be NULL */
    int N, C, H, W, K, R, S;
    int pt, pb, pl, pr;   /* pads: top, bottom, left, right */
    int u, v, dh, dw;     /* strides and dilations */
    double alpha, beta;
    int relu;
    i64 P, Q;
} oracle_problem;

/* Number of window positions along one axis: the count of o >= 0 with
 * o*stride + dil*(filt-1) <= in - 1 + pad_lo + pad_hi, i.e. the dilated
 * window fits inside the padded input. */
i64 oracle_out_extent(i64 in, i64 pad_lo, i64 pad_hi, i64 filt, i64 dil, i64 stride)
{
    if (in <= 0 || filt <= 0 || dil <= 0 || stride <= 0 || pad_lo < 0 || pad_hi < 0)
        return -1;
    i64 eff = dil * (filt - 1) + 1;
    i64 span = in + pad_lo + pad_hi - eff;
    if (span < 0)
        return 0;
    return span / stride + 1;
}

/* One output element: the receptive-field dot product, then the epilogue. */
static void oracle_one(const oracle_problem *pr, i64 n, i64 k, i64 p, i64 q,
                       double *val_out, double *bnd_out)
{
    double acc = 0.0, bnd = 0.0;
    for (i64 c = 0; c < pr->C; ++c) {
        for (i64 r = 0; r < pr->R; ++r) {
            i64 h = p * pr->u + r * pr->dh - pr->pt;
            if (h < 0 || h >= pr->H)
                continue;                       /* zero padding row */
            for (i64 s = 0; s < pr->S; ++s) {
                i64 wi = q * pr->v + s * pr->dw - pr->pl;
                if (wi < 0 || wi >= pr->W)
                    continue;                   /* zero padding column */
                double xv = pr->x[n * pr->xs[0] + c * pr->xs[1] + h * pr->xs[2] + wi * pr->xs[3]];
                double wv = pr->w[k * pr->ws[0] + c * pr->ws[1] + r * pr->ws[2] + s * pr->ws[3]];
                acc += xv * wv;
                bnd += fabs(xv * wv);
            }
        }
    }
    double val = pr->alpha * acc;
    i64 yoff = n * pr->ys[0] + k * pr->ys[1] + p * pr->ys[2] + q * pr->ys[3];
    if (pr->beta != 0.0 && pr->y_in)
        val += pr->beta * pr->y_in[yoff];
    if (pr->bias)
        val += pr->bias[k];
    if (pr->relu && val < 0.0)
        val = 0.0;
    *val_out = val;
    *bnd_out = bnd;
}

typedef struct {
    const oracle_problem *pr;
    i64 first, last;      /* range of flattened (n,k) pairs */
} oracle_slice;

static void *oracle_worker(void *arg)
{
    const oracle_slice *sl = (const oracle_slice *)arg;
    const oracle_problem *pr = sl->pr;
    for (i64 nk = sl->first; nk < sl->last; ++nk) {
        i64 n = nk / pr->K, k = nk % pr->K;
        for (i64 p = 0; p < pr->P; ++p) {
            for (i64 q = 0; q < pr->Q; ++q) {
                double val, bnd;
                oracle_one(pr, n, k, p, q, &val, &bnd);
                i64 yoff = n * pr->ys[0] + k * pr->ys[1] + p * pr->ys[2] + q * pr->ys[3];
                pr->y[yoff] = val;
                if (pr->bound)
                    pr->bound[yoff] = bnd;
            }
        }
    }
    return NULL;
}

static int oracle_fill(oracle_problem *pr,
                       const double *x, const i64 *xs, const double *w, const i64 *ws,
                       double *y, const i64 *ys, double *bound,
                       int N, int C, int H, int W, int K, int R, int S,
                       int pt, int pb, int pl, int prt, int u, int v, int dh, int dw,
                       double alpha, double beta, const double *y_in, const double *bias, int relu)
{
    if (!x || !w || !xs || !ws || !ys)
        return 1;
    if (N < 0 || C <= 0 || H <= 0 || W <= 0 || K <= 0 || R <= 0 || S <= 0)
        return 1;
    pr->x = x; pr->w = w; pr->y = y; pr->bound = bound; pr->y_in = y_in; pr->bias = bias;
    for (int i = 0; i < 4; ++i) {
        pr->xs[i] = xs[i];
        pr->ws[i] = ws[i];
        pr->ys[i] = ys[i];
    }
    pr->N = N; pr->C = C; pr->H = H; pr->W = W; pr->K = K; pr->R = R; pr->S = S;
    pr->pt = pt; pr->pb = pb; pr->pl = pl; pr->pr = prt;
    pr->u = u; pr->v = v; pr->dh = dh; pr->dw = dw;
    pr->alpha = alpha; pr->beta = beta; pr->relu = relu;
    pr->P = oracle_out_extent(H, pt, pb, R, dh, u);
    pr->Q = oracle_out_extent(W, pl, prt, S, dw, v);
    if (pr->P <= 0 || pr->Q <= 0)
        return 2;
    return 0;
}

/*
 * Full forward convolution.  Strides are in elements: xs = {n,c,h,w},
 * ws = {k,c,r,s}, ys = {n,k,p,q} (y, bound and y_in share ys).
 * Returns 0 on success, 1 on a bad argument, 2 when the output is empty.
 */
int oracle_conv2d_fprop(const double *x, const i64 *xs, const double *w, const i64 *ws,
                        double *y, const i64 *ys, double *bound,
                        int N, int C, int H, int W, int K, int R, int S,
                        int pad_top, int pad_bottom, int pad_left, int pad_right,
                        int u, int v, int dil_h, int dil_w,
                        double alpha, double beta, const double *y_in, const double *bias,
                        int relu, int nthreads)
{
    oracle_problem pr;
    int rc = oracle_fill(&pr, x, xs, w, ws, y, ys, bound, N, C, H, W, K, R, S,
                         pad_top, pad_bottom, pad_left, pad_right, u, v, dil_h, dil_w,
                         alpha, beta, y_in, bias, relu);
    if (rc)
        return rc;
    if (!y)
        return 1;
    i64 pairs = (i64)N * K;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if ((i64)nthreads > pairs)
        nthreads = (int)(pairs > 0 ? pairs : 1);
    pthread_t tid[256];
    oracle_slice sl[256];
    int started[256];
    for (int t = 0; t < nthreads; ++t) {
        sl[t].pr = &pr;
        sl[t].first = pairs * t / nthreads;
        sl[t].last = pairs * (t + 1) / nthreads;
        started[t] = 0;
    }
    for (int t = 1; t < nthreads; ++t)
        started[t] = pthread_create(&tid[t], NULL, oracle_worker, &sl[t]) == 0;
    oracle_worker(&sl[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (started[t])
            pthread_join(tid[t], NULL);
        else
            oracle_worker(&sl[t]);   /* thread could not start: do its share here */
    }
    return 0;
}

/*
 * The same definition at a list of output coordinates pts[i] = (n,k,p,q),
 * i < npts.  out[i] gets the epilogued value, bound_out[i] (if not NULL)
 * gets sum |x*w|.  y_in (if beta != 0) is read with strides ys.
 * Returns 0, 1 on a bad argument or coordinate, 2 when the output is empty.
 */
int oracle_conv2d_fprop_points(const double *x, const i64 *xs, const double *w, const i64 *ws,
                               const i64 *ys, int N, int C, int H, int W, int K, int R, int S,
                               int pad_top, int pad_bottom, int pad_left, int pad_right,
                               int u, int v, int dil_h, int dil_w,
                               double alpha, double beta, const double *y_in, const double *bias,
                               int relu, const i64 *pts, i64 npts, double *out, double *bound_out)
{
    oracle_problem pr;
    i64 zero_strides[4] = {0, 0, 0, 0};
    int rc = oracle_fill(&pr, x, xs, w, ws, NULL, ys ? ys : zero_strides, NULL,
                         N, C, H, W, K, R, S, pad_top, pad_bottom, pad_left, pad_right,
                         u, v, dil_h, dil_w, alpha, beta, y_in, bias, relu);
    if (rc)
        return rc;
    if (!pts || !out)
        return 1;
    for (i64 i = 0; i < npts; ++i) {
        i64 n = pts[4 * i], k = pts[4 * i + 1], p = pts[4 * i + 2], q = pts[4 * i + 3];
        if (n < 0 || n >= N || k < 0 || k >= K || p < 0 || p >= pr.P || q < 0 || q >= pr.Q)
            return 1;
        double val, bnd;
        oracle_one(&pr, n, k, p, q, &val, &bnd);
        out[i] = val;
        if (bound_out)
            bound_out[i] = bnd;
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Backward passes (the data and filter gradients).
 *
 * "cuDNN: Efficient Primitives for Deep Learning", method section: the
 * library offers, beside the forward convolution, routines for the gradients
 * with respect to the data and to the filters.  Both are the plain
 * derivatives of the forward sum above (alpha = 1, no epilogue):
 *
 *   dx[n,c,h,w]  = sum over k, r, s and over the outputs (p, q) that read
 *                  input pixel (h, w) through tap (r, s), i.e.
 *                  p*u + r*dh - pad_top = h and q*v + s*dw - pad_left = w,
 *                  0 <= p < P, 0 <= q < Q, of dy[n,k,p,q] * w[k,c,r,s];
 *   dw[k,c,r,s]  = sum_{n, p<P, q<Q} dy[n,k,p,q]
 *                      * X(n, c, p*u + r*dh - pad_top, q*v + s*dw - pad_left),
 *                  with X = 0 outside the image.
 *
 * Each returns alongside the sum of |products| (the same tolerance scale as
 * the forward bound).  FP64, loop orders (n,c,h,w,k,r,s) and (k,c,r,s,n,p,q),
 * pthreads over (n,c) and (k,c) pairs.
 * ------------------------------------------------------------------------ */

typedef struct {
    const double *dy;  i64 dys[4];   /* n, k, p, q */
    const double *w;   i64 ws[4];    /* k, c, r, s */
    const double *x;   i64 xs[4];    /* n, c, h, w (wgrad input) */
    double *out;       i64 os[4];    /* dx: n, c, h, w  -- dw: k, c, r, s */
    double *bound;                   /* same strides as out; may be NULL */
    int N, C, H, W, K, R, S;
    int pt, pl, u, v, dh, dw;
    i64 P, Q;
    int wgrad;
} grad_problem;

typedef struct {
    const grad_problem *gp;
    i64 first, last;
} grad_slice;

/* dx at (n, c, h, w) */
static void dgrad_one(const grad_problem *g, i64 n, i64 c, i64 h, i64 wi, double *val, double *bnd)
{
    double acc = 0.0, b = 0.0;
    for (i64 k = 0; k < g->K; ++k) {
        for (i64 r = 0; r < g->R; ++r) {
            i64 tp = h + g->pt - r * g->dh;          /* = p*u for a reading output */
            if (tp < 0 || tp % g->u != 0)
                continue;
            i64 p = tp / g->u;
            if (p >= g->P)
                continue;
            for (i64 s = 0; s < g->S; ++s) {
                i64 tq = wi + g->pl - s * g->dw;     /* = q*v for a reading output */
                if (tq < 0 || tq % g->v != 0)
                    continue;
                i64 q = tq / g->v;
                if (q >= g->Q)
                    continue;
                double dv = g->dy[n * g->dys[0] + k * g->dys[1] + p * g->dys[2] + q * g->dys[3]];
                double wv = g->w[k * g->ws[0] + c * g->ws[1] + r * g->ws[2] + s * g->ws[3]];
                acc += dv * wv;
                b += fabs(dv * wv);
            }
        }
    }
    *val = acc;
    *bnd = b;
}

/* dw at (k, c, r, s) */
static void wgrad_one(const grad_problem *g, i64 k, i64 c, i64 r, i64 s, double *val, double *bnd)
{
    double acc = 0.0, b = 0.0;
    for (i64 n = 0; n < g->N; ++n) {
        for (i64 p = 0; p < g->P; ++p) {
            i64 h = p * g->u + r * g->dh - g->pt;
            if (h < 0 || h >= g->H)
                continue;                            /* zero padding row */
            for (i64 q = 0; q < g->Q; ++q) {
                i64 wi = q * g->v + s * g->dw - g->pl;
                if (wi < 0 || wi >= g->W)
                    continue;                        /* zero padding column */
                double dv = g->dy[n * g->dys[0] + k * g->dys[1] + p * g->dys[2] + q * g->dys[3]];
                double xv = g->x[n * g->xs[0] + c * g->xs[1] + h * g->xs[2] + wi * g->xs[3]];
                acc += dv * xv;
                b += fabs(dv * xv);
            }
        }
    }
    *val = acc;
    *bnd = b;
}

static void *grad_worker(void *arg)
{
    const grad_slice *sl = (const grad_slice *)arg;
    const grad_problem *g = sl->gp;
    for (i64 pair = sl->first; pair < sl->last; ++pair) {
        i64 a = pair / g->C, c = pair % g->C;      /* a = n (dgrad) or k (wgrad) */
        i64 e2 = g->wgrad ? g->R : g->H, e3 = g->wgrad ? g->S : g->W;
        for (i64 i2 = 0; i2 < e2; ++i2) {
            for (i64 i3 = 0; i3 < e3; ++i3) {
                double val, bnd;
                if (g->wgrad)
                    wgrad_one(g, a, c, i2, i3, &val, &bnd);
                else
                    dgrad_one(g, a, c, i2, i3, &val, &bnd);
                i64 off = a * g->os[0] + c * g->os[1] + i2 * g->os[2] + i3 * g->os[3];
                g->out[off] = val;
                if (g->bound)
                    g->bound[off] = bnd;
            }
        }
    }
    return NULL;
}

static int grad_run(grad_problem *g, int nthreads)
{
    i64 pairs = (i64)(g->wgrad ? g->K : g->N) * g->C;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if ((i64)nthreads > pairs)
        nthreads = (int)(pairs > 0 ? pairs : 1);
    pthread_t tid[256];
    grad_slice sl[256];
    int started[256];
    for (int t = 0; t < nthreads; ++t) {
        sl[t].gp = g;
        sl[t].first = pairs * t / nthreads;
        sl[t].last = pairs * (t + 1) / nthreads;
        started[t] = 0;
    }
    for (int t = 1; t < nthreads; ++t)
        started[t] = pthread_create(&tid[t], NULL, grad_worker, &sl[t]) == 0;
    grad_worker(&sl[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (started[t])
            pthread_join(tid[t], NULL);
        else
            grad_worker(&sl[t]);
    }
    return 0;
}

static int grad_fill(grad_problem *g, int N, int C, int H, int W, int K, int R, int S,
                     int pad_top, int pad_bottom, int pad_left, int pad_right,
                     int u, int v, int dil_h, int dil_w)
{
    if (N <= 0 || C <= 0 || H <= 0 || W <= 0 || K <= 0 || R <= 0 || S <= 0)
        return 1;
    g->N = N; g->C = C; g->H = H; g->W = W; g->K = K; g->R = R; g->S = S;
    g->pt = pad_top; g->pl = pad_left; g->u = u; g->v = v; g->dh = dil_h; g->dw = dil_w;
    g->P = oracle_out_extent(H, pad_top, pad_bottom, R, dil_h, u);
    g->Q = oracle_out_extent(W, pad_left, pad_right, S, dil_w, v);
    if (g->P < 0 || g->Q < 0)
        return 1;
    if (g->P == 0 || g->Q == 0)
        return 2;
    return 0;
}

/* dx (strides dxs = {n,c,h,w}) from dy (dys = {n,k,p,q}) and w (ws = {k,c,r,s}).
 * Returns 0, 1 on a bad argument, 2 when the forward output is empty. */
int oracle_conv2d_dgrad(const double *dy, const i64 *dys, const double *w, const i64 *ws,
                        double *dx, const i64 *dxs, double *bound,
                        int N, int C, int H, int W, int K, int R, int S,
                        int pad_top, int pad_bottom, int pad_left, int pad_right,
                        int u, int v, int dil_h, int dil_w, int nthreads)
{
    if (!dy || !dys || !w || !ws || !dx || !dxs)
        return 1;
    grad_problem g;
    int rc = grad_fill(&g, N, C, H, W, K, R, S, pad_top, pad_bottom, pad_left, pad_right,
                       u, v, dil_h, dil_w);
    if (rc)
        return rc;
    g.dy = dy; g.w = w; g.x = NULL; g.out = dx; g.bound = bound; g.wgrad = 0;
    for (int i = 0; i < 4; ++i) {
        g.dys[i] = dys[i]; g.ws[i] = ws[i]; g.xs[i] = 0; g.os[i] = dxs[i];
    }
    return grad_run(&g, nthreads);
}

/* dw (strides dws = {k,c,r,s}) from x (xs = {n,c,h,w}) and dy (dys = {n,k,p,q}).
 * Returns 0, 1 on a bad argument, 2 when the forward output is empty. */
int oracle_conv2d_wgrad(const double *x, const i64 *xs, const double *dy, const i64 *dys,
                        double *dw, const i64 *dws, double *bound,
                        int N, int C, int H, int W, int K, int R, int S,
                        int pad_top, int pad_bottom, int pad_left, int pad_right,
                        int u, int v, int dil_h, int dil_w, int nthreads)
{
    if (!x || !xs || !dy || !dys || !dw || !dws)
        return 1;
    grad_problem g;
    int rc = grad_fill(&g, N, C, H, W, K, R, S, pad_top, pad_bottom, pad_left, pad_right,
                       u, v, dil_h, dil_w);
    if (rc)
        return rc;
    g.dy = dy; g.w = NULL; g.x = x; g.out = dw; g.bound = bound; g.wgrad = 1;
    for (int i = 0; i < 4; ++i) {
        g.dys[i] = dys[i]; g.ws[i] = 0; g.xs[i] = xs[i]; g.os[i] = dws[i];
    }
    return grad_run(&g, nthreads);
}

/* The same gradients at a list of coordinates pts[i] (n,c,h,w for dx;
 * k,c,r,s for dw), i < npts: out[i] gets the sum, bound_out[i] (if not NULL)
 * the sum of |products|.  Returns 0, 1 on a bad argument or coordinate, 2
 * when the forward output is empty. */
static int grad_points(grad_problem *g, const i64 *pts, i64 npts, double *out, double *bound_out)
{
    if (!pts || !out)
        return 1;
    for (i64 i = 0; i < npts; ++i) {
        i64 a = pts[4 * i], c = pts[4 * i + 1], i2 = pts[4 * i + 2], i3 = pts[4 * i + 3];
        i64 e0 = g->wgrad ? g->K : g->N, e2 = g->wgrad ? g->R : g->H, e3 = g->wgrad ? g->S : g->W;
        if (a < 0 || a >= e0 || c < 0 || c >= g->C || i2 < 0 || i2 >= e2 || i3 < 0 || i3 >= e3)
            return 1;
        double val, bnd;
        if (g->wgrad)
            wgrad_one(g, a, c, i2, i3, &val, &bnd);
        else
            dgrad_one(g, a, c, i2, i3, &val, &bnd);
        out[i] = val;
        if (bound_out)
            bound_out[i] = bnd;
    }
    return 0;
}

int oracle_conv2d_dgrad_points(const double *dy, const i64 *dys, const double *w, const i64 *ws,
                               int N, int C, int H, int W, int K, int R, int S,
                               int pad_top, int pad_bottom, int pad_left, int pad_right,
                               int u, int v, int dil_h, int dil_w,
                               const i64 *pts, i64 npts, double *out, double *bound_out)
{
    if (!dy || !dys || !w || !ws)
        return 1;
    grad_problem g;
    int rc = grad_fill(&g, N, C, H, W, K, R, S, pad_top, pad_bottom, pad_left, pad_right,
                       u, v, dil_h, dil_w);
    if (rc)
        return rc;
    g.dy = dy; g.w = w; g.x = NULL; g.out = NULL; g.bound = NULL; g.wgrad = 0;
    for (int i = 0; i < 4; ++i) {
        g.dys[i] = dys[i]; g.ws[i] = ws[i]; g.xs[i] = 0; g.os[i] = 0;
    }
    return grad_points(&g, pts, npts, out, bound_out);
}

int oracle_conv2d_wgrad_points(const double *x, const i64 *xs, const double *dy, const i64 *dys,
                               int N, int C, int H, int W, int K, int R, int S,
                               int pad_top, int pad_bottom, int pad_left, int pad_right,
                               int u, int v, int dil_h, int dil_w,
                               const i64 *pts, i64 npts, double *out, double *bound_out)
{
    if (!x || !xs || !dy || !dys)
        return 1;
    grad_problem g;
    int rc = grad_fill(&g, N, C, H, W, K, R, S, pad_top, pad_bottom, pad_left, pad_right,
                       u, v, dil_h, dil_w);
    if (rc)
        return rc;
    g.dy = dy; g.w = NULL; g.x = x; g.out = NULL; g.bound = NULL; g.wgrad = 1;
    for (int i = 0; i < 4; ++i) {
        g.dys[i] = dys[i]; g.ws[i] = 0; g.xs[i] = xs[i]; g.os[i] = 0;
    }
    return grad_points(&g, pts, npts, out, bound_out);
}

/* ------------------------------------------------------------------------
 * Pooling and activation forward (the cuDNN page's one-line summary and
 * method section: pooling and activation functions are the library's other
 * primitives, beside convolution).
 *
 *   pooling:    y[n,c,p,q] = alpha * POOL over the window rows
 *               h = p*u - pad_top + i (i < R) and columns w = q*v - pad_left + j
 *               (j < S) that lie inside the image of x[n,c,h,w]
 *               + beta * y_in[n,c,p,q]
 *     POOL = the largest value (mode 0), the sum divided by R*S (mode 1:
 *     padding counted as zeros) or by the number of in-image elements (mode
 *     2: padding excluded).  Output extent as the convolution's (floor), with
 *     every pad smaller than the window so that no window is empty.
 *   activation: y = alpha * f(x) + beta * y_in elementwise, f one of
 *     identity (0), max(0, x) (1), 1 / (1 + e^-x) (2), tanh x (3),
 *     min(max(0, x), coef) (4).
 * FP64 throughout; strided addressing as above.
 * ------------------------------------------------------------------------ */

int oracle_pool2d_fprop(const double *x, const i64 *xs, double *y, const i64 *ys,
                        int N, int C, int H, int W, int R, int S,
                        int pad_top, int pad_bottom, int pad_left, int pad_right, int u, int v,
                        int mode, double alpha, double beta, const double *y_in)
{
    if (!x || !xs || !y || !ys || N <= 0 || C <= 0 || H <= 0 || W <= 0 || R <= 0 || S <= 0)
        return 1;
    if (mode < 0 || mode > 2 || pad_top >= R || pad_bottom >= R || pad_left >= S || pad_right >= S)
        return 1;
    i64 P = oracle_out_extent(H, pad_top, pad_bottom, R, 1, u);
    i64 Q = oracle_out_extent(W, pad_left, pad_right, S, 1, v);
    if (P <= 0 || Q <= 0)
        return 2;
    for (i64 n = 0; n < N; ++n)
        for (i64 c = 0; c < C; ++c)
            for (i64 p = 0; p < P; ++p)
                for (i64 q = 0; q < Q; ++q) {
                    double acc = 0.0;
                    i64 count = 0;
                    int first = 1;
                    for (i64 i = 0; i < R; ++i) {
                        i64 h = p * u - pad_top + i;
                        if (h < 0 || h >= H)
                            continue;
                        for (i64 j = 0; j < S; ++j) {
                            i64 wi = q * v - pad_left + j;
                            if (wi < 0 || wi >= W)
                                continue;
                            double xv = x[n * xs[0] + c * xs[1] + h * xs[2] + wi * xs[3]];
                            if (mode == 0) {
                                if (first || xv > acc)
                                    acc = xv;
                                first = 0;
                            } else {
                                acc += xv;
                            }
                            ++count;
                        }
                    }
                    if (mode == 1)
                        acc /= (double)(R * S);
                    else if (mode == 2)
                        acc /= (double)count;
                    i64 yo = n * ys[0] + c * ys[1] + p * ys[2] + q * ys[3];
                    double val = alpha * acc;
                    if (beta != 0.0 && y_in)
                        val += beta * y_in[yo];
                    y[yo] = val;
                }
    return 0;
}

static double oracle_act(int mode, double xv, double coef)
{
    switch (mode) {
        case 0: return xv;
        case 1: return xv > 0.0 ? xv : 0.0;
        case 2: return 1.0 / (1.0 + exp(-xv));
        case 3: return tanh(xv);
        case 4: return xv < 0.0 ? 0.0 : (xv > coef ? coef : xv);
    }
    return 0.0;
}

int oracle_activation_fprop(const double *x, const i64 *xs, double *y, const i64 *ys,
                            int N, int C, int H, int W, int mode, double coef,
                            double alpha, double beta, const double *y_in)
{
    if (!x || !xs || !y || !ys || N <= 0 || C <= 0 || H <= 0 || W <= 0 || mode < 0 || mode > 4)
        return 1;
    for (i64 n = 0; n < N; ++n)
        for (i64 c = 0; c < C; ++c)
            for (i64 h = 0; h < H; ++h)
                for (i64 wi = 0; wi < W; ++wi) {
                    double xv = x[n * xs[0] + c * xs[1] + h * xs[2] + wi * xs[3]];
                    i64 yo = n * ys[0] + c * ys[1] + h * ys[2] + wi * ys[3];
                    double val = alpha * oracle_act(mode, xv, coef);
                    if (beta != 0.0 && y_in)
                        val += beta * y_in[yo];
                    y[yo] = val;
                }
    return 0;
}
