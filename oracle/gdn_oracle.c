/*
 * gdn_oracle.c -- plain fp64 CPU oracle for the chunked Gated DeltaNet prefill.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (per sequence i and state head h), following
 *   - "GDN 与 Chunked Prefill" (weigao.cc), sections "GDN 是什么",
 *     "块内 state 和块间 final state" and the 4-token expansion table;
 *   - "FlashInfer GDN Prefill 完全指南" (gitcode blog), the API table of
 *     chunk_gated_delta_rule and the sections on the state pool and on
 *     intermediate-state checkpoints:
 *
 *   S <- S0 (pool row state_indices[i], or row i, or zero)      S is V x K
 *   for each token t of the sequence, local position p = 1..L:
 *       S <- alpha_t * S * (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *       o_t <- scale * S q_t                (read AFTER the update)
 *       if n > 0 and p % n == 0: checkpoint[cu_starts[i] + p/n - 1] <- S
 *   final_state[state_indices ? state_indices[i] : i] <- S
 *
 * Two independent evaluations are provided:
 *   oracle_gdn_sequential -- the per-token recurrence above, literally.
 *   oracle_gdn_chunked    -- the chunk form: gate cumulative sums in log space,
 *       the strictly-lower decay matrix A, T = (I + A)^-1 by forward
 *       substitution, W = T diag(beta*gamma) K, U = T diag(beta) V,
 *       Delta = U - W S^T, O = scale*(diag(gamma) Q S^T + (causal decayed
 *       Q K^T) Delta), S <- gamma_last S + (decayed Delta)^T K.
 *       ("GDN 与 Chunked Prefill", sections "为什么要切成 64-token chunk" and
 *       "递推公式如何展开成块内计算"; "GDN与线性注意力GPU并行实现" section 3.3,
 *       the O_init = Q_b S_b product plus a triangular-masked product.)
 * plus oracle_chunk_map, the flat chunk -> (sequence, chunk) table
 * ("GDN 与 Chunked Prefill", section "chunked prefill 有两层含义").
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes): g is alpha in linear space (0 < alpha <= 1) and NULL means ones;
 * beta NULL means ones; the in-kernel L2 norm is x / sqrt(sum x^2 + 1e-6)
 * evaluated exactly in fp64; state head h reads q head h/(H/hq), k head
 * h/(H/hk), v head h/(H/hv) with H = max(hq, hv); g and beta are indexed by
 * the state head; zero-length sequences pass their initial state through.
 *
 * Arithmetic is fp64 throughout.  Work is spread over (sequence, head) units
 * with POSIX threads; every unit is computed by exactly the code above.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t T;
    int32_t N;
    const int64_t *cu_seqlens;    /* [N+1] */
    int32_t hq, hk, hv, D;        /* head counts, head size (K = V = D) */
    const double *q, *k, *v;      /* [T, hq|hk|hv, D] */
    const double *g, *beta;       /* [T, H] or NULL (= all ones) */
    double scale;
    int32_t l2norm;
    const double *initial_state;  /* NULL or [rows, H, D, D] (rows = N or pool) */
    const int64_t *state_indices; /* NULL or [N] */
    double *output;               /* [T, H, D] */
    double *final_state;          /* NULL or [rows, H, D, D]; may alias initial_state */
    int32_t ckpt_n;               /* 0 = no checkpoints */
    const int64_t *ckpt_cu_starts;/* [N+1] */
    double *checkpoints;          /* [total, H, D, D] */
    int32_t chunk;                /* chunked form only: chunk length C */
    double *dump_g;               /* chunked only, optional: [n_flat_chunks, H, C] */
    double *dump_w;               /* chunked only, optional: [n_flat_chunks, H, C, D] */
    double *dump_u;               /* chunked only, optional: [n_flat_chunks, H, C, D] */
    int32_t threads;
} oracle_args;

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_NO_MEMORY = 2 };

static int32_t num_state_heads(const oracle_args *a) { return a->hq > a->hv ? a->hq : a->hv; }

/* x <- x / sqrt(sum x^2 + 1e-6), in fp64 (the pages give eps = 1e-6). */
static void l2_normalise(double *x, int32_t n)
{
    double ss = 0.0;
    for (int32_t c = 0; c < n; ++c) ss += x[c] * x[c];
    double inv = 1.0 / sqrt(ss + 1e-6);
    for (int32_t c = 0; c < n; ++c) x[c] *= inv;
}

/* Load the q, k, v vectors of token t for state head h (head mapping reading). */
static void load_token(const oracle_args *a, int64_t t, int32_t h, double *qt, double *kt, double *vt)
{
    const int32_t H = num_state_heads(a), D = a->D;
    const int32_t hq_i = h / (H / a->hq), hk_i = h / (H / a->hk), hv_i = h / (H / a->hv);
    memcpy(qt, a->q + ((size_t)t * a->hq + hq_i) * D, sizeof(double) * D);
    memcpy(kt, a->k + ((size_t)t * a->hk + hk_i) * D, sizeof(double) * D);
    memcpy(vt, a->v + ((size_t)t * a->hv + hv_i) * D, sizeof(double) * D);
    if (a->l2norm) {
        l2_normalise(qt, D);
        l2_normalise(kt, D);
    }
}

static double gate_alpha(const oracle_args *a, int64_t t, int32_t h)
{
    return a->g ? a->g[(size_t)t * num_state_heads(a) + h] : 1.0;
}

static double gate_beta(const oracle_args *a, int64_t t, int32_t h)
{
    return a->beta ? a->beta[(size_t)t * num_state_heads(a) + h] : 1.0;
}

/* S <- initial state of unit (i, h), or zeros. */
static void load_initial(const oracle_args *a, int32_t i, int32_t h, double *S)
{
    const int32_t H = num_state_heads(a), D = a->D;
    if (!a->initial_state) {
        memset(S, 0, sizeof(double) * D * D);
        return;
    }
    int64_t row = a->state_indices ? a->state_indices[i] : i;
    memcpy(S, a->initial_state + ((size_t)row * H + h) * D * D, sizeof(double) * D * D);
}

static void store_final(const oracle_args *a, int32_t i, int32_t h, const double *S)
{
    const int32_t H = num_state_heads(a), D = a->D;
    if (!a->final_state) return;
    int64_t row = a->state_indices ? a->state_indices[i] : i;
    memcpy(a->final_state + ((size_t)row * H + h) * D * D, S, sizeof(double) * D * D);
}

/* Checkpoint after local position p (1-based) when p is a multiple of n. */
static void maybe_checkpoint(const oracle_args *a, int32_t i, int32_t h, int64_t p, const double *S)
{
    const int32_t H = num_state_heads(a), D = a->D;
    if (a->ckpt_n <= 0 || !a->checkpoints || p % a->ckpt_n != 0) return;
    int64_t slot = a->ckpt_cu_starts[i] + p / a->ckpt_n - 1;
    memcpy(a->checkpoints + ((size_t)slot * H + h) * D * D, S, sizeof(double) * D * D);
}

/* ---------------------------------------------------------------------------
 * Sequential form: one token at a time, exactly the recurrence.
 * ------------------------------------------------------------------------- */
static void unit_sequential(const oracle_args *a, int32_t i, int32_t h, double *work)
{
    const int32_t H = num_state_heads(a), D = a->D;
    double *S = work, *qt = S + D * D, *kt = qt + D, *vt = kt + D, *Sk = vt + D;
    load_initial(a, i, h, S);
    const int64_t t0 = a->cu_seqlens[i], L = a->cu_seqlens[i + 1] - t0;
    for (int64_t p = 1; p <= L; ++p) {
        const int64_t t = t0 + p - 1;
        load_token(a, t, h, qt, kt, vt);
        const double al = gate_alpha(a, t, h), be = gate_beta(a, t, h);
        /* S (I - be k k^T) = S - be (S k) k^T */
        for (int32_t r = 0; r < D; ++r) {
            double acc = 0.0;
            for (int32_t c = 0; c < D; ++c) acc += S[r * D + c] * kt[c];
            Sk[r] = acc;
        }
        for (int32_t r = 0; r < D; ++r)
            for (int32_t c = 0; c < D; ++c)
                S[r * D + c] = al * (S[r * D + c] - be * Sk[r] * kt[c]) + be * vt[r] * kt[c];
        double *o = a->output + ((size_t)t * H + h) * D;
        for (int32_t r = 0; r < D; ++r) {
            double acc = 0.0;
            for (int32_t c = 0; c < D; ++c) acc += S[r * D + c] * qt[c];
            o[r] = a->scale * acc;
        }
        maybe_checkpoint(a, i, h, p, S);
    }
    store_final(a, i, h, S);
}

/* ---------------------------------------------------------------------------
 * Chunked form.
 * ------------------------------------------------------------------------- */
static int64_t chunks_before(const oracle_args *a, int32_t i)
{
    const int64_t C = a->chunk;
    int64_t n = 0;
    for (int32_t s = 0; s < i; ++s) n += (a->cu_seqlens[s + 1] - a->cu_seqlens[s] + C - 1) / C;
    return n;
}

static void unit_chunked(const oracle_args *a, int32_t i, int32_t h, double *work)
{
    const int32_t H = num_state_heads(a), D = a->D, C = a->chunk;
    double *S = work;                  /* D*D */
    double *Q = S + D * D;             /* C*D */
    double *K = Q + C * D;             /* C*D */
    double *V = K + C * D;             /* C*D */
    double *G = V + C * D;             /* C   */
    double *B = G + C;                 /* C   */
    double *A = B + C;                 /* C*C */
    double *Tm = A + C * C;            /* C*C */
    double *W = Tm + C * C;            /* C*D */
    double *U = W + C * D;             /* C*D */
    double *Dl = U + C * D;            /* C*D  Delta */
    double *Snew = Dl + C * D;         /* D*D */

    load_initial(a, i, h, S);
    const int64_t t0 = a->cu_seqlens[i], L = a->cu_seqlens[i + 1] - t0;
    const int64_t nchunks = (L + C - 1) / C;
    const int64_t flat0 = chunks_before(a, i);

    for (int64_t c = 0; c < nchunks; ++c) {
        const int64_t start = c * C;
        const int64_t Lc = (L - start < C) ? (L - start) : C;
        /* Rows past the end of the sequence: q = k = v = 0, alpha = 1, beta = 0. */
        double run = 0.0;
        for (int32_t r = 0; r < C; ++r) {
            if (r < Lc) {
                const int64_t t = t0 + start + r;
                load_token(a, t, h, Q + r * D, K + r * D, V + r * D);
                run += log(gate_alpha(a, t, h));
                B[r] = gate_beta(a, t, h);
            } else {
                memset(Q + r * D, 0, sizeof(double) * D);
                memset(K + r * D, 0, sizeof(double) * D);
                memset(V + r * D, 0, sizeof(double) * D);
                B[r] = 0.0;
            }
            G[r] = run; /* G_r = sum_{m <= r} log alpha_m */
        }
        /* A_rj = beta_r exp(G_r - G_j) (k_r . k_j) for j < r, else 0. */
        for (int32_t r = 0; r < C; ++r)
            for (int32_t j = 0; j < C; ++j) {
                double val = 0.0;
                if (j < r) {
                    double kk = 0.0;
                    for (int32_t d = 0; d < D; ++d) kk += K[r * D + d] * K[j * D + d];
                    val = B[r] * exp(G[r] - G[j]) * kk;
                }
                A[r * C + j] = val;
            }
        /* T = (I + A)^-1 by forward substitution, row by row. */
        for (int32_t r = 0; r < C; ++r)
            for (int32_t j = 0; j < C; ++j) {
                double val = (r == j) ? 1.0 : 0.0;
                for (int32_t m = 0; m < r; ++m) val -= A[r * C + m] * Tm[m * C + j];
                Tm[r * C + j] = val;
            }
        /* W = T diag(beta * gamma) K,  U = T diag(beta) V. */
        for (int32_t r = 0; r < C; ++r)
            for (int32_t d = 0; d < D; ++d) {
                double w = 0.0, u = 0.0;
                for (int32_t j = 0; j < C; ++j) {
                    w += Tm[r * C + j] * B[j] * exp(G[j]) * K[j * D + d];
                    u += Tm[r * C + j] * B[j] * V[j * D + d];
                }
                W[r * D + d] = w;
                U[r * D + d] = u;
            }
        if (a->dump_g || a->dump_w || a->dump_u) {
            const size_t base = (size_t)(flat0 + c) * H + h;
            if (a->dump_g) memcpy(a->dump_g + base * C, G, sizeof(double) * C);
            if (a->dump_w) memcpy(a->dump_w + base * C * D, W, sizeof(double) * C * D);
            if (a->dump_u) memcpy(a->dump_u + base * C * D, U, sizeof(double) * C * D);
        }
        /* Delta = U - W S^T   (Delta[r][v] = U[r][v] - sum_k W[r][k] S[v][k]). */
        for (int32_t r = 0; r < C; ++r)
            for (int32_t vv = 0; vv < D; ++vv) {
                double acc = 0.0;
                for (int32_t kk = 0; kk < D; ++kk) acc += W[r * D + kk] * S[vv * D + kk];
                Dl[r * D + vv] = U[r * D + vv] - acc;
            }
        /* O_r = scale * (gamma_r S q_r + sum_{j <= r} exp(G_r - G_j) (q_r . k_j) Delta_j). */
        for (int32_t r = 0; r < Lc; ++r) {
            double *o = a->output + ((size_t)(t0 + start + r) * H + h) * D;
            const double gam = exp(G[r]);
            for (int32_t vv = 0; vv < D; ++vv) {
                double acc = 0.0;
                for (int32_t kk = 0; kk < D; ++kk) acc += S[vv * D + kk] * Q[r * D + kk];
                o[vv] = gam * acc;
            }
            for (int32_t j = 0; j <= r; ++j) {
                double qk = 0.0;
                for (int32_t d = 0; d < D; ++d) qk += Q[r * D + d] * K[j * D + d];
                const double wgt = exp(G[r] - G[j]) * qk;
                for (int32_t vv = 0; vv < D; ++vv) o[vv] += wgt * Dl[j * D + vv];
            }
            for (int32_t vv = 0; vv < D; ++vv) o[vv] *= a->scale;
        }
        /* S <- gamma_last S + sum_j exp(G_last - G_j) Delta_j k_j^T. */
        const double glast = G[C - 1];
        for (int32_t vv = 0; vv < D; ++vv)
            for (int32_t kk = 0; kk < D; ++kk) {
                double acc = exp(glast) * S[vv * D + kk];
                for (int32_t j = 0; j < C; ++j) acc += exp(glast - G[j]) * Dl[j * D + vv] * K[j * D + kk];
                Snew[vv * D + kk] = acc;
            }
        memcpy(S, Snew, sizeof(double) * D * D);
        if (start + C <= L) maybe_checkpoint(a, i, h, start + C, S);
    }
    store_final(a, i, h, S);
}

/* ---------------------------------------------------------------------------
 * Thread pool over (sequence, head) units.
 * ------------------------------------------------------------------------- */
typedef struct {
    const oracle_args *a;
    int chunked;
    int64_t next;
    pthread_mutex_t lock;
    size_t work_doubles;
    int failed;
} pool_t;

static void *worker(void *arg)
{
    pool_t *p = (pool_t *)arg;
    const int32_t H = num_state_heads(p->a);
    const int64_t units = (int64_t)p->a->N * H;
    double *work = (double *)malloc(sizeof(double) * p->work_doubles);
    if (!work) {
        pthread_mutex_lock(&p->lock);
        p->failed = 1;
        pthread_mutex_unlock(&p->lock);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&p->lock);
        int64_t u = p->next++;
        pthread_mutex_unlock(&p->lock);
        if (u >= units) break;
        const int32_t i = (int32_t)(u / H), h = (int32_t)(u % H);
        if (p->chunked) unit_chunked(p->a, i, h, work);
        else unit_sequential(p->a, i, h, work);
    }
    free(work);
    return NULL;
}

static int check_args(const oracle_args *a, int chunked)
{
    if (!a || a->N < 0 || a->D <= 0 || a->hq <= 0 || a->hk <= 0 || a->hv <= 0) return ORACLE_BAD_ARG;
    const int32_t H = num_state_heads(a);
    if (H % a->hq || H % a->hk || H % a->hv) return ORACLE_BAD_ARG;
    if (!a->cu_seqlens || !a->q || !a->k || !a->v || !a->output) return ORACLE_BAD_ARG;
    if (a->ckpt_n > 0 && (!a->ckpt_cu_starts || !a->checkpoints)) return ORACLE_BAD_ARG;
    if (chunked && a->chunk <= 0) return ORACLE_BAD_ARG;
    for (int32_t i = 0; i < a->N; ++i)
        if (a->cu_seqlens[i + 1] < a->cu_seqlens[i]) return ORACLE_BAD_ARG;
    return ORACLE_OK;
}

static int run_pool(const oracle_args *a, int chunked)
{
    int rc = check_args(a, chunked);
    if (rc) return rc;
    pool_t p;
    p.a = a;
    p.chunked = chunked;
    p.next = 0;
    p.failed = 0;
    pthread_mutex_init(&p.lock, NULL);
    const size_t D = (size_t)a->D, C = (size_t)(chunked ? a->chunk : 1);
    p.work_doubles = chunked ? (2 * D * D + 6 * C * D + 2 * C * C + 2 * C) : (D * D + 4 * D);
    int nt = a->threads > 0 ? a->threads : 1;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * nt);
    if (!tid) return ORACLE_NO_MEMORY;
    int started = 0;
    for (int t = 0; t < nt; ++t)
        if (pthread_create(&tid[t], NULL, worker, &p) == 0) ++started;
    if (started == 0) worker(&p);
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    free(tid);
    pthread_mutex_destroy(&p.lock);
    return p.failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

int oracle_gdn_sequential(const oracle_args *a) { return run_pool(a, 0); }

int oracle_gdn_chunked(const oracle_args *a) { return run_pool(a, 1); }

/*
 * Flat chunk table: sequence i owns ceil(L_i / C) chunks (zero-length
 * sequences own none); flat chunk f = offsets[i] + c maps to (i, c).
 * offsets is [N+1] (exclusive prefix sum), map is [map_rows, 2], rows past
 * the last chunk are filled with -1.  Returns the number of chunks, or -1 if
 * map_rows is too small or cu_seqlens decreases.
 */
int64_t oracle_chunk_map(int32_t N, const int64_t *cu_seqlens, int32_t C, int32_t *offsets, int32_t *map,
                         int64_t map_rows)
{
    int64_t total = 0;
    for (int32_t i = 0; i < N; ++i) {
        const int64_t L = cu_seqlens[i + 1] - cu_seqlens[i];
        if (L < 0) return -1;
        offsets[i] = (int32_t)total;
        total += (L + C - 1) / C;
    }
    offsets[N] = (int32_t)total;
    if (total > map_rows) return -1;
    for (int64_t f = 0; f < map_rows; ++f) map[2 * f] = map[2 * f + 1] = -1;
    for (int32_t i = 0; i < N; ++i)
        for (int32_t c = 0; offsets[i] + c < offsets[i + 1]; ++c) {
            map[2 * (offsets[i] + c)] = i;
            map[2 * (offsets[i] + c) + 1] = c;
        }
    return total;
}
