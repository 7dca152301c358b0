/*
 * Float64 CPU oracle of the multi-adapter LoRA linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this code; the product path never calls it.  It
 * shares no code, header, table or helper with the CUDA library.
 *
 * What it computes, for every requested row m and every output column n:
 *
 *     y[m,n] = sum_k W[n,k] x[m,k]                                 (base)
 *            + (alpha_i / r_i) * sum_j B_i[n,j] * (sum_k A_i[j,k] x[m,k])
 *
 * where i = row_adapter[m]; the second line is absent when i == -1.  This is
 * the scaled LoRA form "W' = W + (alpha/r) B A" applied additively, without
 * merging ("Your LoRA Adapters Are Thrashing Your GPUs", §02 "The full
 * decomposition with scaling factor" and "Weight merging vs. keeping adapters
 * separate"), evaluated per row as in the adapted_linear sketch of "Adapter
 * Residency When One Replica Serves Many Fine-Tunes", §"What the forward pass
 * has to do differently": dense base projection first, then the rank-r
 * bottleneck v = A x, then B v times the adapter's own scale added to the
 * row.  Shapes: W is d x k (here N x K), A is r x k, B is d x r (the shapes
 * govern where the pages' role labels for A and B disagree).
 *
 * Arithmetic: every input is a float32 value (exact for bf16 and fp32
 * inputs) widened to double; sums run over k (resp. j) in ascending order in
 * double; the scale is (double)alpha / (double)r.  No reassociation, no
 * blocking, no fused operations beyond what the C compiler does for a plain
 * multiply-add written as such (build with -ffp-contract=off).
 *
 * Threads: rows are independent, so rows are split statically over POSIX
 * threads; each thread writes only its own output rows.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int n_rows;
    const int32_t *rows; /* which input rows to compute; NULL = 0..n_rows-1 */
    int K, N;
    const float *x;          /* [*, K] */
    const float *W;          /* [N, K] */
    const int32_t *row_adapter; /* indexed by input row */
    int num_adapters;
    const int32_t *ranks;    /* [num_adapters] */
    const double *alphas;    /* [num_adapters] */
    const float *const *A;   /* A[i] -> [r_i, K] row-major */
    const float *const *B;   /* B[i] -> [N, r_i] row-major */
    double *y;               /* [n_rows, N] */
    int n_threads;
    int thread_index;
    int status;
} oracle_job;

/* One output row: base dot products, then the adapter's correction. */
static int oracle_row(const oracle_job *J, int out_index, double *v_scratch)
{
    const int m = J->rows ? J->rows[out_index] : out_index;
    const float *xr = J->x + (size_t)m * (size_t)J->K;
    double *yr = J->y + (size_t)out_index * (size_t)J->N;

    for (int n = 0; n < J->N; ++n) {
        const float *wr = J->W + (size_t)n * (size_t)J->K;
        double acc = 0.0;
        for (int k = 0; k < J->K; ++k)
            acc += (double)wr[k] * (double)xr[k];
        yr[n] = acc;
    }

    const int i = J->row_adapter[m];
    if (i == -1)
        return 0;
    if (i < -1 || i >= J->num_adapters)
        return 1;
    const int r = J->ranks[i];
    if (r <= 0)
        return 2;
    const double s = J->alphas[i] / (double)r;
    const float *Ai = J->A[i];
    const float *Bi = J->B[i];

    /* rank-r bottleneck v = A_i x */
    for (int j = 0; j < r; ++j) {
        const float *ar = Ai + (size_t)j * (size_t)J->K;
        double t = 0.0;
        for (int k = 0; k < J->K; ++k)
            t += (double)ar[k] * (double)xr[k];
        v_scratch[j] = t;
    }
    /* y += s * B_i v */
    for (int n = 0; n < J->N; ++n) {
        const float *br = Bi + (size_t)n * (size_t)r;
        double t = 0.0;
        for (int j = 0; j < r; ++j)
            t += (double)br[j] * v_scratch[j];
        yr[n] += s * t;
    }
    return 0;
}

static void *oracle_worker(void *arg)
{
    oracle_job *J = (oracle_job *)arg;
    int max_r = 1;
    for (int i = 0; i < J->num_adapters; ++i)
        if (J->ranks[i] > max_r)
            max_r = J->ranks[i];
    double *v = (double *)malloc(sizeof(double) * (size_t)max_r);
    if (!v) {
        J->status = 3;
        return NULL;
    }
    for (int o = J->thread_index; o < J->n_rows; o += J->n_threads) {
        int st = oracle_row(J, o, v);
        if (st) {
            J->status = st;
            break;
        }
    }
    free(v);
    return NULL;
}

/*
 * Compute y for n_rows rows of x (rows[] lists the input row of each output
 * row; NULL means rows 0..n_rows-1).  Returns 0 on success, nonzero on a bad
 * adapter id or rank.
 */
int lora_oracle_forward(int n_rows, const int32_t *rows, int K, int N,
                        const float *x, const float *W,
                        const int32_t *row_adapter, int num_adapters,
                        const int32_t *ranks, const double *alphas,
                        const float *const *A, const float *const *B,
                        double *y, int n_threads)
{
    if (n_rows < 0 || K < 0 || N < 0)
        return 4;
    if (n_rows == 0 || N == 0)
        return 0;
    if (n_threads < 1)
        n_threads = 1;
    if (n_threads > n_rows)
        n_threads = n_rows;

    oracle_job *jobs = (oracle_job *)calloc((size_t)n_threads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return 3;
    }
    for (int t = 0; t < n_threads; ++t) {
        oracle_job *J = &jobs[t];
        J->n_rows = n_rows; J->rows = rows; J->K = K; J->N = N;
        J->x = x; J->W = W; J->row_adapter = row_adapter;
        J->num_adapters = num_adapters; J->ranks = ranks; J->alphas = alphas;
        J->A = A; J->B = B; J->y = y;
        J->n_threads = n_threads; J->thread_index = t; J->status = 0;
    }
    int started = 0;
    for (int t = 1; t < n_threads; ++t) {
        if (pthread_create(&tids[t], NULL, oracle_worker, &jobs[t]) != 0)
            break;
        started = t;
    }
    /* threads that could not be started: run their share here */
    oracle_worker(&jobs[0]);
    for (int t = started + 1; t < n_threads; ++t)
        oracle_worker(&jobs[t]);
    for (int t = 1; t <= started; ++t)
        pthread_join(tids[t], NULL);

    int status = 0;
    for (int t = 0; t < n_threads; ++t)
        if (jobs[t].status)
            status = jobs[t].status;
    free(jobs);
    free(tids);
    return status;
}
