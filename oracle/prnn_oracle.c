/*
 * prnn_oracle.c -- plain, slow, fp64 CPU oracle for the forward recurrence of a
 * vanilla ReLU RNN layer.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check
 * and the benchmark's CPU-baseline leg call it; the CUDA library never does,
 * and the two share no code.
 *
 * What it computes (the basic, non-LSTM RNN layer of the persistent-rnn library
 * page, gitmyhub.com/pineking/persistent-rnn, "Important Constraints"; the
 * single-layer stage of "Optimizing Performance of Recurrent Neural Networks
 * on GPUs", Abstract):
 *
 *     h_{-1} = h0 (zeros when h0 is NULL)
 *     for t = 0 .. T-1, for every batch column b and hidden row r:
 *         s        = bias[r] + sum_c Wx[r,c] x[t,b,c] + sum_c Wh[r,c] h_{t-1}[b,c]
 *         h_t[b,r] = s > 0 ? s : 0                                      (ReLU)
 *         y[t,b,r] = h_t[b,r]
 *
 * The sparse form takes Wh as k (value, column) pairs per row (the row-balanced
 * layout of "Sparse Persistent RNNs: Squeezing Large Recurrent Networks
 * On-Chip", measured-effects table, load-balanced pruning rows) and sums over
 * the listed columns in the order given.  Persistence, sparsity tricks and
 * timestamps change how fast the result is reached, never the result, so the
 * oracle is the definition written out: one double accumulator per output,
 * terms added in the order above, no blocking or reordering.
 *
 * Layouts (all row-major, time-major sequences):
 *   x [T][B][I], Wx [H][I], Wh [H][H], vals/cols [H][k], bias [H],
 *   h0 [B][H] or NULL, y [T][B][H].
 * Return: 0 on success, -1 on bad sizes or NULL pointers.
 */
#define _POSIX_C_SOURCE 200809L
#include <pthread.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

static double relu(double s) { return s > 0.0 ? s : 0.0; }

/* One output element of one step, dense Wh.  x_t is [I], h_prev is [H]. */
double oracle_rnn_cell_dense(long H, long I, long r, const double* x_t,
                             const double* Wx, const double* Wh,
                             const double* bias, const double* h_prev) {
    double s = bias[r];
    for (long c = 0; c < I; ++c) s += Wx[r * I + c] * x_t[c];
    for (long c = 0; c < H; ++c) s += Wh[r * H + c] * h_prev[c];
    return relu(s);
}

/* One output element of one step, row-balanced sparse Wh (k entries per row). */
double oracle_rnn_cell_sparse(long H, long I, long k, long r, const double* x_t,
                              const double* Wx, const double* vals,
                              const long* cols, const double* bias,
                              const double* h_prev) {
    (void)H;
    double s = bias[r];
    for (long c = 0; c < I; ++c) s += Wx[r * I + c] * x_t[c];
    for (long j = 0; j < k; ++j) s += vals[r * k + j] * h_prev[cols[r * k + j]];
    return relu(s);
}

/* Shared driver of the time loop.  Only the cell differs between the forms. */
static int forward(long T, long B, long H, long I, long k, const double* x,
                   const double* Wx, const double* Wh, const double* vals,
                   const long* cols, const double* bias, const double* h0,
                   double* y) {
    if (T < 0 || B < 0 || H <= 0 || I <= 0) return -1;
    if (!x || !Wx || !bias || !y) return -1;
    if (!Wh && (!vals || !cols || k <= 0)) return -1;
    if (T == 0 || B == 0) return 0;
    double* zeros = NULL;
    if (!h0) {
        zeros = (double*)calloc((size_t)(B * H), sizeof(double));
        if (!zeros) return -1;
        h0 = zeros;
    }
    for (long t = 0; t < T; ++t) {
        for (long b = 0; b < B; ++b) {
            const double* x_t = x + (t * B + b) * I;
            /* h_{t-1}: the previous step's output, or h0 at t = 0 */
            const double* h_prev = (t == 0) ? h0 + b * H : y + ((t - 1) * B + b) * H;
            double* out = y + (t * B + b) * H;
            for (long r = 0; r < H; ++r) {
                out[r] = Wh ? oracle_rnn_cell_dense(H, I, r, x_t, Wx, Wh, bias, h_prev)
                            : oracle_rnn_cell_sparse(H, I, k, r, x_t, Wx, vals, cols,
                                                     bias, h_prev);
            }
        }
    }
    free(zeros);
    return 0;
}

int oracle_rnn_forward_dense(long T, long B, long H, long I, const double* x,
                             const double* Wx, const double* Wh,
                             const double* bias, const double* h0, double* y) {
    if (!Wh) return -1;
    return forward(T, B, H, I, 0, x, Wx, Wh, NULL, NULL, bias, h0, y);
}

int oracle_rnn_forward_sparse(long T, long B, long H, long I, long k,
                              const double* x, const double* Wx,
                              const double* vals, const long* cols,
                              const double* bias, const double* h0, double* y) {
    if (!vals || !cols || k <= 0 || k > H) return -1;
    for (long i = 0; i < H * k; ++i)
        if (cols[i] < 0 || cols[i] >= H) return -1;
    return forward(T, B, H, I, k, x, Wx, NULL, vals, cols, bias, h0, y);
}

/*
 * The same time loop run by a team of POSIX threads, for timing the oracle on
 * every host core.  Each step's B*H outputs are split into contiguous runs of
 * (b, r), one per thread, and a barrier separates the steps (step t reads all
 * of h_{t-1}).  Every output is computed by the same cell function as the
 * one-thread driver above, from the same inputs, so y is bit-identical to it;
 * only the order in which outputs are produced differs.  Wh != NULL selects the
 * dense form, else the row-balanced sparse form (k, vals, cols).
 */
typedef struct {
    long T, B, H, I, k;
    const double *x, *Wx, *Wh, *vals, *bias, *h0;
    const long* cols;
    double* y;
    pthread_mutex_t gate_m;
    pthread_cond_t gate_c;
    int started;
    long nlive; /* threads that take part, set before the gate opens */
    pthread_barrier_t step;
} team_t;

typedef struct {
    team_t* team;
    long id;
} member_t;

static void team_work(team_t* tm, long id) {
    pthread_mutex_lock(&tm->gate_m);
    while (!tm->started) pthread_cond_wait(&tm->gate_c, &tm->gate_m);
    pthread_mutex_unlock(&tm->gate_m);
    const long n = tm->B * tm->H;
    const long i0 = n * id / tm->nlive, i1 = n * (id + 1) / tm->nlive;
    for (long t = 0; t < tm->T; ++t) {
        for (long i = i0; i < i1; ++i) {
            const long b = i / tm->H, r = i % tm->H;
            const double* x_t = tm->x + (t * tm->B + b) * tm->I;
            const double* h_prev =
                (t == 0) ? tm->h0 + b * tm->H : tm->y + ((t - 1) * tm->B + b) * tm->H;
            tm->y[(t * tm->B + b) * tm->H + r] =
                tm->Wh ? oracle_rnn_cell_dense(tm->H, tm->I, r, x_t, tm->Wx, tm->Wh, tm->bias,
                                               h_prev)
                       : oracle_rnn_cell_sparse(tm->H, tm->I, tm->k, r, x_t, tm->Wx, tm->vals,
                                                tm->cols, tm->bias, h_prev);
        }
        pthread_barrier_wait(&tm->step);
    }
}

static void* team_member(void* arg) {
    member_t* m = (member_t*)arg;
    team_work(m->team, m->id);
    return NULL;
}

int oracle_rnn_forward_threads(long T, long B, long H, long I, long k, const double* x,
                               const double* Wx, const double* Wh, const double* vals,
                               const long* cols, const double* bias, const double* h0,
                               double* y, long nthreads) {
    if (T < 0 || B < 0 || H <= 0 || I <= 0 || nthreads < 1 || nthreads > 1024) return -1;
    if (!x || !Wx || !bias || !y) return -1;
    if (!Wh) {
        if (!vals || !cols || k <= 0 || k > H) return -1;
        for (long i = 0; i < H * k; ++i)
            if (cols[i] < 0 || cols[i] >= H) return -1;
    }
    if (T == 0 || B == 0) return 0;
    double* zeros = NULL;
    if (!h0) {
        zeros = (double*)calloc((size_t)(B * H), sizeof(double));
        if (!zeros) return -1;
        h0 = zeros;
    }
    pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    member_t* members = (member_t*)calloc((size_t)nthreads, sizeof(member_t));
    if (!tids || !members) {
        free(tids);
        free(members);
        free(zeros);
        return -1;
    }
    team_t tm = {.T = T, .B = B, .H = H, .I = I, .k = k, .x = x, .Wx = Wx, .Wh = Wh,
                 .vals = vals, .bias = bias, .h0 = h0, .cols = cols, .y = y};
    pthread_mutex_init(&tm.gate_m, NULL);
    pthread_cond_init(&tm.gate_c, NULL);
    tm.started = 0;
    /* the calling thread is member 0; members 1.. are started until one fails */
    long nlive = 1;
    for (long id = 1; id < nthreads; ++id) {
        members[id].team = &tm;
        members[id].id = id;
        if (pthread_create(&tids[id], NULL, team_member, &members[id]) != 0) break;
        ++nlive;
    }
    tm.nlive = nlive;
    pthread_barrier_init(&tm.step, NULL, (unsigned)nlive);
    pthread_mutex_lock(&tm.gate_m);
    tm.started = 1;
    pthread_cond_broadcast(&tm.gate_c);
    pthread_mutex_unlock(&tm.gate_m);
    team_work(&tm, 0);
    for (long id = 1; id < nlive; ++id) pthread_join(tids[id], NULL);
    pthread_barrier_destroy(&tm.step);
    pthread_cond_destroy(&tm.gate_c);
    pthread_mutex_destroy(&tm.gate_m);
    free(tids);
    free(members);
    free(zeros);
    return 0;
}

/*
 * Unbalanced sparse Wh in compressed-row form: row r holds the entries
 * row_ptr[r] .. row_ptr[r+1]-1 of (vals, cols), summed in the order given.
 * This is the matrix straightforward (global, not per-row) magnitude pruning
 * leaves behind -- rows of unequal length -- the comparison point of the
 * load-balanced pruning rows of "Sparse Persistent RNNs: Squeezing Large
 * Recurrent Networks On-Chip" (measured-effects table).
 */
double oracle_rnn_cell_csr(long H, long I, long r, const double* x_t, const double* Wx,
                           const long* row_ptr, const double* vals, const long* cols,
                           const double* bias, const double* h_prev) {
    (void)H;
    double s = bias[r];
    for (long c = 0; c < I; ++c) s += Wx[r * I + c] * x_t[c];
    for (long j = row_ptr[r]; j < row_ptr[r + 1]; ++j) s += vals[j] * h_prev[cols[j]];
    return relu(s);
}

int oracle_rnn_forward_csr(long T, long B, long H, long I, const double* x,
                           const double* Wx, const long* row_ptr, const double* vals,
                           const long* cols, const double* bias, const double* h0,
                           double* y) {
    if (T < 0 || B < 0 || H <= 0 || I <= 0) return -1;
    if (!x || !Wx || !row_ptr || !bias || !y) return -1;
    if (row_ptr[0] != 0) return -1;
    for (long r = 0; r < H; ++r)
        if (row_ptr[r + 1] < row_ptr[r]) return -1;
    for (long j = 0; j < row_ptr[H]; ++j)
        if (!vals || !cols || cols[j] < 0 || cols[j] >= H) return -1;
    if (T == 0 || B == 0) return 0;
    double* zeros = NULL;
    if (!h0) {
        zeros = (double*)calloc((size_t)(B * H), sizeof(double));
        if (!zeros) return -1;
        h0 = zeros;
    }
    for (long t = 0; t < T; ++t)
        for (long b = 0; b < B; ++b) {
            const double* x_t = x + (t * B + b) * I;
            const double* h_prev = (t == 0) ? h0 + b * H : y + ((t - 1) * B + b) * H;
            double* out = y + (t * B + b) * H;
            for (long r = 0; r < H; ++r)
                out[r] = oracle_rnn_cell_csr(H, I, r, x_t, Wx, row_ptr, vals, cols, bias,
                                             h_prev);
        }
    free(zeros);
    return 0;
}

/*
 * The input projection on its own, P[t,b,r] = bias[r] + sum_c Wx[r,c] x[t,b,c]:
 * the part of every step that does not depend on h_{t-1} and so can be done for
 * all steps at once (work that does not depend on the previous step is batched
 * across steps: Abstract of "Optimizing Performance of Recurrent Neural
 * Networks on GPUs").
 */
int oracle_rnn_input_projection(long T, long B, long H, long I, const double* x,
                                const double* Wx, const double* bias, double* P) {
    if (T < 0 || B < 0 || H <= 0 || I <= 0 || !x || !Wx || !bias || !P) return -1;
    for (long m = 0; m < T * B; ++m)
        for (long r = 0; r < H; ++r) {
            double s = bias[r];
            for (long c = 0; c < I; ++c) s += Wx[r * I + c] * x[m * I + c];
            P[m * H + r] = s;
        }
    return 0;
}

/*
 * Backward pass (backpropagation through time) of the same layer, for the
 * scalar objective L = sum_{t,b,r} dy[t,b,r] * y[t,b,r] -- dy is the gradient
 * of the training loss with respect to every output.  Training is what the
 * persistent kernels are built for ("Optimizing Performance of Recurrent
 * Neural Networks on GPUs", Abstract: training recurrent networks); the
 * steps are those of the chain rule applied to the forward definition above:
 *
 *   delta_T = 0
 *   for t = T-1 .. 0:   g = dy_t + Wh^T delta_{t+1}
 *                       delta_t[r] = y_t[r] > 0 ? g[r] : 0      (ReLU'(a) = [a > 0])
 *   db[r]     = sum_{t,b} delta_t[b,r]
 *   dWh[r,c]  = sum_{t,b} delta_t[b,r] * h_{t-1}[b,c]          (h_{-1} = h0)
 *   dWx[r,c]  = sum_{t,b} delta_t[b,r] * x_t[b,c]
 *   dx_t[b,c] = sum_r Wx[r,c] * delta_t[b,r]
 *   dh0[b,c]  = sum_r Wh[r,c] * delta_0[b,r]
 *
 * y is the oracle's own forward output (this function runs the forward
 * first).  delta [T][B][H] is returned too.  Any output pointer may be NULL.
 * Returns 0, or -1 on bad arguments.
 */
/* One element of the reverse recurrence, given delta_{t+1} ([H], NULL = 0). */
double oracle_rnn_delta_cell_dense(long H, long r, const double* Wh, const double* dy_t,
                                   const double* y_t, const double* delta_next) {
    double g = dy_t[r];
    if (delta_next)
        for (long c = 0; c < H; ++c) g += Wh[c * H + r] * delta_next[c];
    return y_t[r] > 0.0 ? g : 0.0;
}

int oracle_rnn_backward_dense(long T, long B, long H, long I, const double* x, const double* Wx,
                              const double* Wh, const double* bias, const double* h0,
                              const double* dy, double* delta, double* dx, double* dh0,
                              double* dWx, double* dWh, double* db) {
    if (T < 0 || B < 0 || H <= 0 || I <= 0 || !x || !Wx || !Wh || !bias || !dy) return -1;
    double* y = (double*)calloc((size_t)(T * B * H) + 1, sizeof(double));
    double* d = delta ? delta : (double*)calloc((size_t)(T * B * H) + 1, sizeof(double));
    if (!y || !d) { free(y); if (!delta) free(d); return -1; }
    if (oracle_rnn_forward_dense(T, B, H, I, x, Wx, Wh, bias, h0, y) != 0) {
        free(y); if (!delta) free(d); return -1;
    }
    for (long t = T - 1; t >= 0; --t)
        for (long b = 0; b < B; ++b) {
            const double* next = (t == T - 1) ? NULL : d + ((t + 1) * B + b) * H;
            for (long r = 0; r < H; ++r)
                d[(t * B + b) * H + r] = oracle_rnn_delta_cell_dense(
                    H, r, Wh, dy + (t * B + b) * H, y + (t * B + b) * H, next);
        }
    if (db)
        for (long r = 0; r < H; ++r) {
            double s = 0.0;
            for (long t = 0; t < T; ++t)
                for (long b = 0; b < B; ++b) s += d[(t * B + b) * H + r];
            db[r] = s;
        }
    if (dWh)
        for (long r = 0; r < H; ++r)
            for (long c = 0; c < H; ++c) {
                double s = 0.0;
                for (long t = 0; t < T; ++t)
                    for (long b = 0; b < B; ++b) {
                        const double hp = (t == 0) ? (h0 ? h0[b * H + c] : 0.0)
                                                   : y[((t - 1) * B + b) * H + c];
                        s += d[(t * B + b) * H + r] * hp;
                    }
                dWh[r * H + c] = s;
            }
    if (dWx)
        for (long r = 0; r < H; ++r)
            for (long c = 0; c < I; ++c) {
                double s = 0.0;
                for (long t = 0; t < T; ++t)
                    for (long b = 0; b < B; ++b)
                        s += d[(t * B + b) * H + r] * x[(t * B + b) * I + c];
                dWx[r * I + c] = s;
            }
    if (dx)
        for (long t = 0; t < T; ++t)
            for (long b = 0; b < B; ++b)
                for (long c = 0; c < I; ++c) {
                    double s = 0.0;
                    for (long r = 0; r < H; ++r) s += Wx[r * I + c] * d[(t * B + b) * H + r];
                    dx[(t * B + b) * I + c] = s;
                }
    if (dh0)
        for (long b = 0; b < B; ++b)
            for (long c = 0; c < H; ++c) {
                double s = 0.0;
                if (T > 0)
                    for (long r = 0; r < H; ++r) s += Wh[r * H + c] * d[b * H + r];
                dh0[b * H + c] = s;
            }
    free(y);
    if (!delta) free(d);
    return 0;
}
