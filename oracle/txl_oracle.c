/*
 * Plain fp64 CPU oracle for Transformer-XL relative attention over a
 * recurrence memory.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check
 * and the CPU-baseline leg of the benchmark load it; the product path never
 * does.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes is the plain definition, written out with one loop per
 * (query i, key j) pair and no blocking, fusion or reordering:
 *
 *   keys j = 0 .. M+L-1; rows j < M are the memory, rows j >= M the current
 *   segment ("Transformer-XL" notes, zty624, section "Batched Tensor
 *   Contract": Q has L rows, K and V have M+L rows);
 *
 *   allow(i, j)  <=>  j <= M + i
 *     (same notes, section "Causal Mask With Memory": with key position
 *      p = j - M, memory keys p < 0 are all visible and current keys are
 *      visible when p <= i);
 *
 *   with same_length (source-reading notes, MemTransformerLM._forward: every
 *   query attends over the same number of keys), the mask adds the lower
 *   triangle tril(ones, -mask_shift_len) to triu(ones, 1+mlen), where
 *   mask_len = klen - mem_len and mask_shift_len = qlen - mask_len when
 *   mask_len > 0, else qlen; so additionally
 *     allow(i, j)  requires  j - i > -mask_shift_len;
 *
 *   dist(i, j) = M + i - j, the relative distance query minus key, and the
 *   position row used is r_k[M+L-1-dist] because the position sequence runs
 *   from M+L-1 down to 0 ("Transformer-XL模型 核心源码阅读笔记", section
 *   "Build the model", MemTransformerLM._forward: pos_seq);
 *
 *   score(i, j) = scale * (a + b + c + d) with the four terms of the same
 *   notes' section "Relative Positional Encoding":
 *       a = q_i . k_j      (content-content)
 *       b = q_i . R_dist   (content-position)
 *       c = u   . k_j      (global content bias)
 *       d = v   . R_dist   (global position bias);
 *
 *   masked pairs get probability exactly 0 (the -inf fill of
 *   RelPartialLearnableMultiHeadAttn.forward in the source-reading notes),
 *   then softmax over keys and the probability-weighted sum of V rows.
 *
 * Layouts (all contiguous, row-major, fp64):
 *   q   [B, H, L, dh]      k, v [B, H, M+L, dh]
 *   r_k [M+L, H, dh]       u, vb [H, dh]
 *   out [B, H, L, dh]      scores (optional) [B, H, L, M+L], -inf if masked
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdlib.h>
#include <unistd.h>

typedef struct {
    const double *q, *k, *v, *r, *u, *vb;
    int B, H, L, M, dh;
    int same_length;
    int mask_shift_len; /* used when same_length */
    double scale;
    double *out;
    double *scores;
    const int *pairs; /* flat (b*H + h) indices to compute; NULL = all */
    int npairs;
    int next;
    int failed;
    pthread_mutex_t mu;
} oracle_job;

static double dot(const double *x, const double *y, int n) {
    double s = 0.0;
    for (int t = 0; t < n; ++t) s += x[t] * y[t];
    return s;
}

/* One (batch row, head) pair: every query row, every key, four terms. */
static int attn_pair(const oracle_job *J, int bh) {
    const int H = J->H, L = J->L, M = J->M, dh = J->dh, K = M + L;
    const int h = bh % H;
    const double *Q = J->q + (size_t)bh * L * dh;
    const double *Kp = J->k + (size_t)bh * K * dh;
    const double *Vp = J->v + (size_t)bh * K * dh;
    const double *u = J->u + (size_t)h * dh;
    const double *vb = J->vb + (size_t)h * dh;
    double *s = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    if (!s) return -1;
    for (int i = 0; i < L; ++i) {
        const double *qi = Q + (size_t)i * dh;
        double m = -INFINITY;
        for (int j = 0; j < K; ++j) {
            int allow = (j - i <= M);
            if (J->same_length && !(j - i > -J->mask_shift_len)) allow = 0;
            if (!allow) {
                s[j] = -INFINITY;
                continue;
            }
            int dist = M + i - j;
            const double *R = J->r + ((size_t)(K - 1 - dist) * H + h) * dh;
            const double *kj = Kp + (size_t)j * dh;
            double a = dot(qi, kj, dh);
            double b = dot(qi, R, dh);
            double c = dot(u, kj, dh);
            double d = dot(vb, R, dh);
            s[j] = J->scale * (a + b + c + d);
            if (s[j] > m) m = s[j];
        }
        double denom = 0.0;
        for (int j = 0; j < K; ++j) {
            double p = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
            denom += p;
        }
        double *o = J->out + ((size_t)bh * L + i) * dh;
        for (int t = 0; t < dh; ++t) o[t] = 0.0;
        for (int j = 0; j < K; ++j) {
            if (s[j] == -INFINITY) continue;
            double p = exp(s[j] - m) / denom;
            const double *vj = Vp + (size_t)j * dh;
            for (int t = 0; t < dh; ++t) o[t] += p * vj[t];
        }
        if (J->scores) {
            double *srow = J->scores + ((size_t)bh * L + i) * K;
            for (int j = 0; j < K; ++j) srow[j] = s[j];
        }
    }
    free(s);
    return 0;
}

static void *worker(void *arg) {
    oracle_job *J = (oracle_job *)arg;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int idx = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (idx >= J->npairs) break;
        int bh = J->pairs ? J->pairs[idx] : idx;
        if (attn_pair(J, bh) != 0) {
            pthread_mutex_lock(&J->mu);
            J->failed = 1;
            pthread_mutex_unlock(&J->mu);
        }
    }
    return NULL;
}

int oracle_num_cores(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Relative attention forward.  pairs/npairs select (b*H+h) pairs (for a
 * bounded sample of a large workload); pairs == NULL computes all B*H.
 * Rows of out/scores belonging to pairs not selected are left untouched.
 * nthreads <= 0 uses every online core.  Returns the thread count used,
 * or a negative value on bad arguments / allocation failure.
 */
int oracle_attn_f64_ex(const double *q, const double *k, const double *v,
                       const double *r_k, const double *u, const double *vb,
                       int B, int H, int L, int M, int dh, double scale,
                       int same_length, int mem_len,
                       double *out, double *scores, const int *pairs, int npairs,
                       int nthreads) {
    if (B <= 0 || H <= 0 || L <= 0 || M < 0 || dh <= 0) return -1;
    if (!q || !k || !v || !r_k || !u || !vb || !out) return -1;
    if (same_length && mem_len < 0) return -1;
    oracle_job J;
    {
        const int klen = M + L, mask_len = klen - mem_len;
        J.same_length = same_length != 0;
        J.mask_shift_len = mask_len > 0 ? L - mask_len : L;
    }
    J.q = q; J.k = k; J.v = v; J.r = r_k; J.u = u; J.vb = vb;
    J.B = B; J.H = H; J.L = L; J.M = M; J.dh = dh;
    J.scale = scale; J.out = out; J.scores = scores;
    J.pairs = pairs;
    J.npairs = pairs ? npairs : B * H;
    J.next = 0;
    J.failed = 0;
    pthread_mutex_init(&J.mu, NULL);
    int nt = nthreads > 0 ? nthreads : oracle_num_cores();
    if (nt > J.npairs) nt = J.npairs > 0 ? J.npairs : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    if (!th) return -2;
    int started = 0;
    for (int t = 0; t < nt; ++t) {
        if (pthread_create(&th[t], NULL, worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) worker(&J);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&J.mu);
    return J.failed ? -2 : (started ? started : 1);
}

/* The plain causal mask (same_length off). */
int oracle_attn_f64(const double *q, const double *k, const double *v,
                    const double *r_k, const double *u, const double *vb,
                    int B, int H, int L, int M, int dh, double scale,
                    double *out, double *scores, const int *pairs, int npairs,
                    int nthreads) {
    return oracle_attn_f64_ex(q, k, v, r_k, u, vb, B, H, L, M, dh, scale, 0, 0, out, scores,
                              pairs, npairs, nthreads);
}
