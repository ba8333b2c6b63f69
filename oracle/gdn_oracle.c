/*
 * gdn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64 CPU reference for draft-tree verification and
 * accepted-path commit of one Gated DeltaNet (GDN) layer.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg load this
 * library; the product path never does.  It shares no code, header or
 * constant with the CUDA library.
 *
 * What it computes is the plain definition, not the fast method:
 *
 *   For every sequence b, head h and draft node t, start from the committed
 *   state S = S0[b,h] (d_v x d_k) and walk the node's root-to-node path
 *   j_0 (root), j_1, ..., j_m = t, applying the gated delta rule
 *
 *       S <- alpha_j S (I - beta_j k_j k_j^T) + beta_j v_j k_j^T
 *
 *   (SpecLA review, pith.science 7ERME3HB, "Load-bearing premise" and
 *   "What would settle it": each node must see exactly the sequential GDN
 *   recurrence along its ancestor path and nothing from its siblings; the
 *   recurrence itself is the GDN delta rule of "Gated Delta Networks:
 *   Improving Mamba2 with Delta Rule", cited there).  The node's output is
 *   o_t = S q_t after its own update.
 *
 *   Besides o_t it reports, per node, the quantities a verifier hands to the
 *   commit: the delta-rule innovation
 *       delta_t = beta_t (v_t - alpha_t S_parent k_t)
 *   (so that the update reads S_t = alpha_t S_parent + delta_t k_t^T) and the
 *   cumulative log gate g_t = sum of log alpha_j over the root-to-t path.
 *
 *   The commit walks the accepted root-first path the same way and returns
 *   the state after its last node (the state unchanged when the path is
 *   empty).
 *
 * Arithmetic is fp64 with a fixed order; build with -ffp-contract=off so the
 * results are the same on every host.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_TREE (-2)
#define ORACLE_BAD_PATH (-3)
#define ORACLE_BAD_ARG (-1)

/* ------------------------------------------------------------------ */
/* topology                                                            */
/* ------------------------------------------------------------------ */

/* parent[t] must be -1 (child of the committed state) or an earlier node. */
static int tree_is_valid(const int32_t* parent, int N)
{
    for (int t = 0; t < N; ++t)
        if (parent[t] < -1 || parent[t] >= t) return 0;
    return 1;
}

/* Root-first node list ending at t; returns its length. */
static int path_to(const int32_t* parent, int t, int* out)
{
    int len = 0;
    for (int j = t; j >= 0; j = parent[j]) out[len++] = j;
    for (int i = 0; i < len / 2; ++i) {
        int tmp = out[i];
        out[i] = out[len - 1 - i];
        out[len - 1 - i] = tmp;
    }
    return len;
}

/*
 * Strict-ancestor bitmask and depth of every node (N <= 64): bit j of
 * mask[b*N+t] is set iff node j lies on the path from the root to t, t
 * excluded.  Roots have depth 0.
 */
int oracle_tree_meta(int B, int N, const int32_t* parent, uint64_t* mask, int32_t* depth)
{
    if (B < 0 || N < 1 || N > 64) return ORACLE_BAD_ARG;
    for (int b = 0; b < B; ++b) {
        const int32_t* par = parent + (size_t)b * N;
        if (!tree_is_valid(par, N)) return ORACLE_BAD_TREE;
        for (int t = 0; t < N; ++t) {
            uint64_t m = 0;
            int d = 0;
            for (int j = par[t]; j >= 0; j = par[j]) {
                m |= (uint64_t)1 << j;
                ++d;
            }
            mask[(size_t)b * N + t] = m;
            depth[(size_t)b * N + t] = d;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* one gated delta-rule step on a d_v x d_k row-major state             */
/* ------------------------------------------------------------------ */

/*
 * S <- a * S (I - b k k^T) + b v k^T, written out as
 * S <- a * (S - b (S k) k^T) + b v k^T.  Sk receives S k before the update.
 */
static void delta_step(double* S, int dv, int dk, const double* k, const double* v,
                       double a, double b, double* Sk)
{
    for (int i = 0; i < dv; ++i) {
        double s = 0.0;
        const double* row = S + (size_t)i * dk;
        for (int c = 0; c < dk; ++c) s += row[c] * k[c];
        Sk[i] = s;
    }
    for (int i = 0; i < dv; ++i) {
        double* row = S + (size_t)i * dk;
        for (int c = 0; c < dk; ++c) row[c] = a * (row[c] - b * Sk[i] * k[c]) + b * v[i] * k[c];
    }
}

/* ------------------------------------------------------------------ */
/* threading over (b, h) work items                                     */
/* ------------------------------------------------------------------ */

typedef struct {
    int B, N, H, dk, dv;
    const double *q, *k, *v, *alpha, *beta, *S0;
    const int32_t* parent;
    const uint8_t* want;   /* [B,N] or NULL: nodes to evaluate */
    double *out, *delta, *g;
    const int32_t* path;   /* commit only: [B, Lmax] */
    int Lmax;
    double* S_new;
    int nthreads;
    int tid;
} job_t;

static double* row_qkv(const double* base, const job_t* J, int b, int t, int h, int d)
{
    return (double*)base + (((size_t)b * J->N + t) * J->H + h) * d;
}

static void* verify_worker(void* arg)
{
    const job_t* J = (const job_t*)arg;
    const int N = J->N, H = J->H, dk = J->dk, dv = J->dv;
    double* S = (double*)malloc(sizeof(double) * (size_t)dv * dk);
    double* Sk = (double*)malloc(sizeof(double) * (size_t)dv);
    int* path = (int*)malloc(sizeof(int) * (size_t)N);
    for (int item = J->tid; item < J->B * H; item += J->nthreads) {
        const int b = item / H, h = item % H;
        const int32_t* par = J->parent + (size_t)b * N;
        const double* S0 = J->S0 + (size_t)(b * H + h) * dv * dk;
        for (int t = 0; t < N; ++t) {
            if (J->want && !J->want[(size_t)b * N + t]) continue;
            const int len = path_to(par, t, path);
            memcpy(S, S0, sizeof(double) * (size_t)dv * dk);
            double gsum = 0.0;
            for (int s = 0; s < len; ++s) {
                const int j = path[s];
                const size_t gi = ((size_t)b * N + j) * H + h;
                const double a = J->alpha[gi], be = J->beta[gi];
                const double* kj = row_qkv(J->k, J, b, j, h, dk);
                const double* vj = row_qkv(J->v, J, b, j, h, dv);
                delta_step(S, dv, dk, kj, vj, a, be, Sk);
                gsum += log(a);
                if (s == len - 1 && J->delta) {
                    /* delta_t = beta_t (v_t - alpha_t S_parent k_t); Sk holds S_parent k_t. */
                    double* dl = J->delta + (((size_t)b * H + h) * N + t) * dv;
                    for (int i = 0; i < dv; ++i) dl[i] = be * (vj[i] - a * Sk[i]);
                }
            }
            if (J->g) J->g[((size_t)b * H + h) * N + t] = gsum;
            /* o_t = S_t q_t */
            const double* qt = row_qkv(J->q, J, b, t, h, dk);
            double* o = J->out + (((size_t)b * N + t) * H + h) * dv;
            for (int i = 0; i < dv; ++i) {
                double s = 0.0;
                const double* row = S + (size_t)i * dk;
                for (int c = 0; c < dk; ++c) s += row[c] * qt[c];
                o[i] = s;
            }
        }
    }
    free(S);
    free(Sk);
    free(path);
    return NULL;
}

static void run_threads(job_t* proto, void* (*fn)(void*))
{
    int nt = proto->nthreads < 1 ? 1 : proto->nthreads;
    if (nt == 1) {
        proto->tid = 0;
        proto->nthreads = 1;
        fn(proto);
        return;
    }
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
    job_t* jobs = (job_t*)malloc(sizeof(job_t) * (size_t)nt);
    for (int i = 0; i < nt; ++i) {
        jobs[i] = *proto;
        jobs[i].tid = i;
        jobs[i].nthreads = nt;
        pthread_create(&th[i], NULL, fn, &jobs[i]);
    }
    for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
    free(th);
    free(jobs);
}

/*
 * Verify every draft node (or those with want[b*N+t] != 0) of B trees.
 *   q, k  [B,N,H,dk]   v [B,N,H,dv]   alpha, beta [B,N,H]   parent [B,N]
 *   S0    [B,H,dv,dk]
 * Outputs: out [B,N,H,dv]; delta [B,H,N,dv] and g [B,H,N] when non-NULL.
 */
int oracle_tree_verify(int B, int N, int H, int dk, int dv, const double* q, const double* k,
                       const double* v, const double* alpha, const double* beta,
                       const int32_t* parent, const double* S0, const uint8_t* want, double* out,
                       double* delta, double* g, int nthreads)
{
    if (B < 0 || N < 1 || H < 1 || dk < 1 || dv < 1) return ORACLE_BAD_ARG;
    for (int b = 0; b < B; ++b)
        if (!tree_is_valid(parent + (size_t)b * N, N)) return ORACLE_BAD_TREE;
    job_t J;
    memset(&J, 0, sizeof J);
    J.B = B; J.N = N; J.H = H; J.dk = dk; J.dv = dv;
    J.q = q; J.k = k; J.v = v; J.alpha = alpha; J.beta = beta; J.S0 = S0;
    J.parent = parent; J.want = want; J.out = out; J.delta = delta; J.g = g;
    J.nthreads = nthreads;
    run_threads(&J, verify_worker);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* accepted-path commit                                                 */
/* ------------------------------------------------------------------ */

/* Number of accepted nodes in a root-first, -1 padded path, or -1 if invalid. */
static int path_length(const int32_t* par, int N, const int32_t* path, int Lmax)
{
    int L = 0;
    while (L < Lmax && path[L] >= 0) ++L;
    for (int i = L; i < Lmax; ++i)
        if (path[i] != -1) return -1;
    for (int i = 0; i < L; ++i) {
        if (path[i] >= N) return -1;
        const int want_parent = i == 0 ? -1 : path[i - 1];
        if (par[path[i]] != want_parent) return -1;
    }
    return L;
}

static void* commit_worker(void* arg)
{
    const job_t* J = (const job_t*)arg;
    const int N = J->N, H = J->H, dk = J->dk, dv = J->dv;
    double* Sk = (double*)malloc(sizeof(double) * (size_t)dv);
    for (int item = J->tid; item < J->B * H; item += J->nthreads) {
        const int b = item / H, h = item % H;
        const int32_t* par = J->parent + (size_t)b * N;
        const int32_t* path = J->path + (size_t)b * J->Lmax;
        const int L = path_length(par, N, path, J->Lmax);
        double* S = J->S_new + (size_t)(b * H + h) * dv * dk;
        memcpy(S, J->S0 + (size_t)(b * H + h) * dv * dk, sizeof(double) * (size_t)dv * dk);
        for (int s = 0; s < L; ++s) {
            const int j = path[s];
            const size_t gi = ((size_t)b * N + j) * H + h;
            delta_step(S, dv, dk, row_qkv(J->k, J, b, j, h, dk), row_qkv(J->v, J, b, j, h, dv),
                       J->alpha[gi], J->beta[gi], Sk);
        }
    }
    free(Sk);
    return NULL;
}

/*
 * State after the accepted path: S_new[b,h] = S0[b,h] walked through
 * path[b, 0..L-1] (root first, -1 padded; L = 0 leaves S0 unchanged).
 * path[b,0] must be a root and path[b,i] a child of path[b,i-1].
 */
int oracle_commit(int B, int N, int H, int dk, int dv, const double* k, const double* v,
                  const double* alpha, const double* beta, const int32_t* parent,
                  const double* S0, const int32_t* path, int Lmax, double* S_new, int nthreads)
{
    if (B < 0 || N < 1 || H < 1 || dk < 1 || dv < 1 || Lmax < 1) return ORACLE_BAD_ARG;
    for (int b = 0; b < B; ++b) {
        if (!tree_is_valid(parent + (size_t)b * N, N)) return ORACLE_BAD_TREE;
        if (path_length(parent + (size_t)b * N, N, path + (size_t)b * Lmax, Lmax) < 0)
            return ORACLE_BAD_PATH;
    }
    job_t J;
    memset(&J, 0, sizeof J);
    J.B = B; J.N = N; J.H = H; J.dk = dk; J.dv = dv;
    J.k = k; J.v = v; J.alpha = alpha; J.beta = beta; J.S0 = S0; J.parent = parent;
    J.path = path; J.Lmax = Lmax; J.S_new = S_new;
    J.nthreads = nthreads;
    run_threads(&J, commit_worker);
    return ORACLE_OK;
}
