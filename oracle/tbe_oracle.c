/*
 * TBE oracle: a plain, slow, obviously correct CPU statement of what the
 * table-batched embedding operator computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark use this file.  It shares no code, header or
 * constant with the CUDA library, and the library never calls it.
 *
 * Sources (three web pages on FBTriton table-batched embeddings):
 *  - "Optimizing Recommendation Systems with FBTriton Table Batched
 *    Embeddings", section "Implementation Guide: Integrating TBE": the call
 *    takes tables, a flat index list and an offsets list that cuts it into
 *    bags (CSR layout).
 *  - "FBTriton Rewrites Table Batched Embedding", section "Responsibilities of
 *    the forward and backward passes": forward gathers rows by index and
 *    aggregates them per sample; backward scatters the upstream gradient back
 *    to the looked-up rows and accumulates when one row is hit several times.
 *  - kimbodo "What Happened": one launch pools across tables; per-sample
 *    weights; higher-precision accumulation; backward groups updates by
 *    (table, row) so that each row receives one optimizer update.
 *  - kimbodo "Kimbodo Engineering Perspective": the backward steps are
 *    transpose, sort and run-length encoding.
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes of the repository):
 *  - offsets has T*B+1 entries, table-major: bag (t,b) is flat bag t*B+b.
 *  - an index outside [0, rows_t) is skipped: it contributes nothing and
 *    updates nothing; the count of such lookups is reported.
 *  - output is fp32 [B, sum_t D_t]; table t owns columns [Doff_t, Doff_t+D_t).
 *  - mean pooling divides the (weighted) sum by the bag length L (the CSR
 *    length, skipped lookups included); an empty bag pools to 0.
 *  - the scale of lookup i is s_i = w_i (or 1 without weights), times 1/L
 *    for mean pooling; the backward pass uses the same s_i.
 *  - SGD: w <- w - lr*g.  Row-wise Adagrad (fp32 per-row state m, m0 = 0):
 *    m <- m + mean_j g_j^2, w_j <- w_j - lr*g_j/(sqrt(m)+eps), new m used.
 *  - all sums and updates run in double; each stored value is rounded once,
 *    to nearest even, to its storage type (fp32, fp16 or bf16).
 *  - sort key of lookup i is rowbase_t + idx_i (rowbase_t = sum of rows of
 *    the tables before t); a skipped lookup gets the key sum_t rows_t.  The
 *    sort is stable (equal keys keep ascending position).
 *  - the per-sample weights are trainable inputs: their gradient is the dot
 *    product of the looked-up row (as stored, before this step's update)
 *    with the bag's slice of the upstream gradient, times 1/L for mean
 *    pooling; a skipped lookup's weight gets gradient 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_F32 0
#define OR_F16 1
#define OR_BF16 2

#define OR_OK 0
#define OR_BAD_ARG -1
#define OR_BAD_OFFSETS -2
#define OR_NO_MEMORY -3

/* Threads of the parallel loops in the timing build (compiled with OpenMP);
 * returns the count in effect.  The plain build runs on one thread. */
int oracle_set_threads(int32_t n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* ---------------------------------------------------------------- storage */

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double f16_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25); /* (1 + f/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

/* Round a double, to nearest even, to a binary format with `ebits` exponent
 * bits (bias 2^(ebits-1)-1, all-ones exponent = inf/nan) and `mbits` fraction
 * bits, with subnormals; returns the encoded bits (sign in bit ebits+mbits). */
static uint32_t round_to_small_float(double x, int mbits, int ebits) {
    const int bias = (1 << (ebits - 1)) - 1;
    const uint32_t sign = signbit(x) ? (1u << (ebits + mbits)) : 0u;
    const uint32_t inf = ((1u << ebits) - 1u) << mbits;
    double a = fabs(x);
    if (isnan(x)) return sign | inf | (1u << (mbits - 1));
    if (isinf(x)) return sign | inf;
    const int emin = 1 - bias; /* smallest normal exponent */
    if (a < ldexp(1.0, emin)) {
        /* subnormal range: quantum 2^(emin - mbits); rint rounds to nearest
         * even; a result of 2^mbits lands exactly on the smallest normal. */
        double q = rint(ldexp(a, mbits - emin));
        return sign | (uint32_t)q;
    }
    int e2;
    frexp(a, &e2); /* a in [2^(e2-1), 2^e2) */
    int E = e2 - 1;
    double q = rint(ldexp(a, mbits - E)); /* in [2^mbits, 2^(mbits+1)] */
    if (q == ldexp(1.0, mbits + 1)) {
        q = ldexp(1.0, mbits);
        E += 1;
    }
    if (E > bias) return sign | inf; /* overflow rounds to infinity */
    return sign | ((uint32_t)(E + bias) << mbits) | ((uint32_t)q - (1u << mbits));
}

static uint16_t double_to_f16_bits(double x) { return (uint16_t)round_to_small_float(x, 10, 5); }
static uint16_t double_to_bf16_bits(double x) { return (uint16_t)round_to_small_float(x, 7, 8); }

static double load_elem(const void* base, int dtype, int64_t k) {
    switch (dtype) {
        case OR_F32: return (double)((const float*)base)[k];
        case OR_F16: return f16_bits_to_double(((const uint16_t*)base)[k]);
        default: return bf16_bits_to_double(((const uint16_t*)base)[k]);
    }
}

static void store_elem(void* base, int dtype, int64_t k, double v) {
    switch (dtype) {
        case OR_F32: ((float*)base)[k] = (float)v; break; /* C rounds to nearest */
        case OR_F16: ((uint16_t*)base)[k] = double_to_f16_bits(v); break;
        default: ((uint16_t*)base)[k] = double_to_bf16_bits(v); break;
    }
}

/* Exposed so the tests can pin the rounding against library conversions. */
void oracle_round(int32_t dtype, const double* x, int64_t n, void* out) {
    for (int64_t i = 0; i < n; ++i) store_elem(out, dtype, i, x[i]);
}

void oracle_decode(int32_t dtype, const void* x, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = load_elem(x, dtype, i);
}

/* ------------------------------------------------------------ CSR helpers */

static int64_t load_index(const void* p, int is64, int64_t k) {
    return is64 ? ((const int64_t*)p)[k] : (int64_t)((const int32_t*)p)[k];
}

/* offsets must start at 0, never decrease and end at N. */
static int check_offsets(const void* offsets, int is64, int64_t nbags, int64_t N) {
    if (load_index(offsets, is64, 0) != 0) return OR_BAD_OFFSETS;
    for (int64_t k = 0; k < nbags; ++k)
        if (load_index(offsets, is64, k + 1) < load_index(offsets, is64, k)) return OR_BAD_OFFSETS;
    if (load_index(offsets, is64, nbags) != N) return OR_BAD_OFFSETS;
    return OR_OK;
}

/* ----------------------------------------------------------------- forward */

/* out[b, Doff_t + j] = (1/L if mean) * sum_{i in bag(t,b)} s_i * W_t[idx_i, j]
 * tables[t] points at a row-major rows[t] x dims[t] array of dtypes[t]. */
int oracle_forward(int32_t T, const int64_t* rows, const int32_t* dims, const int32_t* dtypes,
                   const void* const* tables, int32_t B, int32_t index_is64,
                   const void* indices, const void* offsets, int64_t N,
                   const float* weights, int32_t mean_pooling, float* out, int64_t* n_skipped) {
    if (T <= 0 || B < 0 || N < 0) return OR_BAD_ARG;
    int rc = check_offsets(offsets, index_is64, (int64_t)T * B, N);
    if (rc) return rc;
    int64_t total_d = 0, maxd = 1;
    int64_t* doffs = (int64_t*)malloc(sizeof(int64_t) * (size_t)T);
    if (!doffs) return OR_NO_MEMORY;
    for (int t = 0; t < T; ++t) {
        doffs[t] = total_d;
        total_d += dims[t];
        if (dims[t] > maxd) maxd = dims[t];
    }
    int64_t skipped = 0;
    int nomem = 0;
    /* bags are independent: the timing build runs them on all host cores
     * (OpenMP); every bag's sum is the same sequence of additions either way */
#pragma omp parallel reduction(+ : skipped, nomem)
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)maxd);
        if (!acc) nomem = 1;
#pragma omp for schedule(static)
        for (int64_t bag = 0; bag < (int64_t)T * B; ++bag) {
            if (!acc) continue;
            const int t = (int)(bag / B);
            const int64_t b = bag - (int64_t)t * B;
            const int D = dims[t];
            const int64_t start = load_index(offsets, index_is64, bag);
            const int64_t end = load_index(offsets, index_is64, bag + 1);
            for (int j = 0; j < D; ++j) acc[j] = 0.0;
            for (int64_t i = start; i < end; ++i) {
                const int64_t r = load_index(indices, index_is64, i);
                if (r < 0 || r >= rows[t]) {
                    ++skipped;
                    continue;
                }
                const double s = weights ? (double)weights[i] : 1.0;
                for (int j = 0; j < D; ++j) acc[j] += s * load_elem(tables[t], dtypes[t], r * D + j);
            }
            const int64_t L = end - start;
            for (int j = 0; j < D; ++j) {
                double v = acc[j];
                if (mean_pooling && L > 0) v = v / (double)L;
                out[b * total_d + doffs[t] + j] = (float)v;
            }
        }
        free(acc);
    }
    free(doffs);
    if (nomem) return OR_NO_MEMORY;
    if (n_skipped) *n_skipped = skipped;
    return OR_OK;
}

/* Gradient of the loss with respect to each lookup's per-sample weight
 * (kimbodo "What Happened": per-sample weights), given the upstream gradient
 * G = dL/dout:  out[b, Doff_t + j] = sum_i s_i W_t[idx_i, j] with
 * s_i = w_i (times 1/L for mean pooling), so
 * dL/dw_i = sum_j G[b, Doff_t + j] W_t[idx_i, j]   (times 1/L for mean).
 * A skipped lookup (index out of range) gets 0.  Sums in double, one
 * rounding to float. */
int oracle_weight_grad(int32_t T, const int64_t* rows, const int32_t* dims, const int32_t* dtypes,
                       const void* const* tables, int32_t B, int32_t index_is64,
                       const void* indices, const void* offsets, int64_t N, int32_t mean_pooling,
                       const float* grad_out, float* wgrad) {
    if (T <= 0 || B < 0 || N < 0) return OR_BAD_ARG;
    int rc = check_offsets(offsets, index_is64, (int64_t)T * B, N);
    if (rc) return rc;
    int64_t total_d = 0;
    for (int t = 0; t < T; ++t) total_d += dims[t];
    int64_t doff = 0;
    for (int t = 0; t < T; ++t) {
        const int D = dims[t];
        for (int b = 0; b < B; ++b) {
            const int64_t bag = (int64_t)t * B + b;
            const int64_t start = load_index(offsets, index_is64, bag);
            const int64_t end = load_index(offsets, index_is64, bag + 1);
            const int64_t L = end - start;
            const float* g = grad_out + (int64_t)b * total_d + doff;
            for (int64_t i = start; i < end; ++i) {
                const int64_t r = load_index(indices, index_is64, i);
                if (r < 0 || r >= rows[t]) {
                    wgrad[i] = 0.0f;
                    continue;
                }
                double dot = 0.0;
                for (int j = 0; j < D; ++j) dot += (double)g[j] * load_elem(tables[t], dtypes[t], r * D + j);
                if (mean_pooling && L > 0) dot /= (double)L;
                wgrad[i] = (float)dot;
            }
        }
        doff += D;
    }
    return OR_OK;
}

/* -------------------------------------------- transpose, sort, run-length */

/* key_i = rowbase_t + idx_i; a skipped lookup gets key = sum of all rows. */
int oracle_make_keys(int32_t T, const int64_t* rows, int32_t B, int32_t index_is64,
                     const void* indices, const void* offsets, int64_t N,
                     int64_t* keys, int64_t* bag_of) {
    if (T <= 0 || B < 0 || N < 0) return OR_BAD_ARG;
    int rc = check_offsets(offsets, index_is64, (int64_t)T * B, N);
    if (rc) return rc;
    int64_t total_rows = 0;
    for (int t = 0; t < T; ++t) total_rows += rows[t];
    int64_t rowbase = 0;
    for (int t = 0; t < T; ++t) {
        for (int b = 0; b < B; ++b) {
            const int64_t bag = (int64_t)t * B + b;
            const int64_t start = load_index(offsets, index_is64, bag);
            const int64_t end = load_index(offsets, index_is64, bag + 1);
            for (int64_t i = start; i < end; ++i) {
                const int64_t r = load_index(indices, index_is64, i);
                keys[i] = (r < 0 || r >= rows[t]) ? total_rows : rowbase + r;
                if (bag_of) bag_of[i] = bag;
            }
        }
        rowbase += rows[t];
    }
    return OR_OK;
}

typedef struct {
    int64_t key;
    int64_t pos;
} key_pos;

/* (key, pos) ascending: since positions are distinct this is exactly a
 * stable sort by key. */
static int cmp_key_pos(const void* a, const void* b) {
    const key_pos* x = (const key_pos*)a;
    const key_pos* y = (const key_pos*)b;
    if (x->key != y->key) return x->key < y->key ? -1 : 1;
    return (x->pos > y->pos) - (x->pos < y->pos);
}

/* Stable sort of keys[0..N) (values = positions), then run-length encoding:
 * uniq[u] is the u-th distinct key, runstart[u] its first sorted slot,
 * runlen[u] its count.  Returns U (>= 0) or an error. */
int64_t oracle_sort_rle(const int64_t* keys, int64_t N, int64_t* sorted_keys, int64_t* sorted_pos,
                        int64_t* uniq, int64_t* runstart, int64_t* runlen) {
    if (N < 0) return OR_BAD_ARG;
    key_pos* kp = (key_pos*)malloc(sizeof(key_pos) * (size_t)(N > 0 ? N : 1));
    if (!kp) return OR_NO_MEMORY;
    for (int64_t i = 0; i < N; ++i) {
        kp[i].key = keys[i];
        kp[i].pos = i;
    }
    qsort(kp, (size_t)N, sizeof(key_pos), cmp_key_pos);
    int64_t U = 0;
    for (int64_t i = 0; i < N; ++i) {
        if (sorted_keys) sorted_keys[i] = kp[i].key;
        if (sorted_pos) sorted_pos[i] = kp[i].pos;
        if (i == 0 || kp[i].key != kp[i - 1].key) {
            if (uniq) uniq[U] = kp[i].key;
            if (runstart) runstart[U] = i;
            if (runlen) runlen[U] = 0;
            ++U;
        }
        if (runlen) runlen[U - 1] += 1;
    }
    free(kp);
    return U;
}

/* ---------------------------------------------------------------- backward */

#define OPT_NONE 0
#define OPT_SGD 1
#define OPT_ROWWISE_ADAGRAD 2

/*
 * Backward + optimizer.  Groups the lookups by (table, row) through the
 * stable sort above, sums s_i * G[bag_i, Doff_t : Doff_t+D_t] over each group
 * in double, then applies exactly one optimizer step to that row.  Tables are
 * updated in place; `state` (fp32, one entry per row of every table, laid out
 * at rowbase_t + r) is updated for row-wise Adagrad.
 *
 * If row_grads is non-null it receives, for each distinct valid key u (in key
 * order), the gradient row g (double, padded to max_dim columns), and
 * row_keys[u] its key; *n_rows receives the number of such rows.
 */
int oracle_backward(int32_t T, const int64_t* rows, const int32_t* dims, const int32_t* dtypes,
                    void* const* tables, int32_t B, int32_t index_is64, const void* indices,
                    const void* offsets, int64_t N, const float* weights, int32_t mean_pooling,
                    const float* grad_out, int32_t optimizer, float lr, float eps, float* state,
                    double* row_grads, int64_t* row_keys, int64_t* n_rows) {
    if (T <= 0 || B < 0 || N < 0) return OR_BAD_ARG;
    int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)(N > 0 ? N : 1));
    int64_t* bag_of = (int64_t*)malloc(sizeof(int64_t) * (size_t)(N > 0 ? N : 1));
    int64_t* skeys = (int64_t*)malloc(sizeof(int64_t) * (size_t)(N > 0 ? N : 1));
    int64_t* spos = (int64_t*)malloc(sizeof(int64_t) * (size_t)(N > 0 ? N : 1));
    int64_t* rowbase = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T + 1));
    int64_t* doff = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T + 1));
    int maxd = 1;
    for (int t = 0; t < T; ++t)
        if (dims[t] > maxd) maxd = dims[t];
    int64_t* rstart = (int64_t*)malloc(sizeof(int64_t) * (size_t)(N + 1));
    int rc = OR_OK;
    if (!keys || !bag_of || !skeys || !spos || !rowbase || !doff || !rstart) {
        rc = OR_NO_MEMORY;
        goto done;
    }
    rowbase[0] = 0;
    doff[0] = 0;
    for (int t = 0; t < T; ++t) {
        rowbase[t + 1] = rowbase[t] + rows[t];
        doff[t + 1] = doff[t] + dims[t];
    }
    const int64_t total_rows = rowbase[T], total_d = doff[T];

    /* transpose: one (table,row) key per lookup */
    rc = oracle_make_keys(T, rows, B, index_is64, indices, offsets, N, keys, bag_of);
    if (rc) goto done;
    /* sort: group equal keys, positions ascending inside a group */
    if (oracle_sort_rle(keys, N, skeys, spos, NULL, NULL, NULL) < 0) {
        rc = OR_NO_MEMORY;
        goto done;
    }

    /* run-length: the runs of equal keys (first sorted slot of each) */
    int64_t nruns = 0;
    for (int64_t i = 0; i < N; ++i)
        if (i == 0 || skeys[i] != skeys[i - 1]) rstart[nruns++] = i;
    rstart[nruns] = N;
    /* the key of skipped lookups (sum of rows) is the largest, so every run
     * before it is a valid row; runs update distinct rows and state entries,
     * so the timing build runs them on all host cores (OpenMP) */
    const int64_t nr = (nruns > 0 && skeys[rstart[nruns - 1]] >= total_rows) ? nruns - 1 : nruns;
    int nomem = 0;
#pragma omp parallel reduction(+ : nomem)
    {
        double* g = (double*)malloc(sizeof(double) * (size_t)maxd);
        if (!g) nomem = 1;
#pragma omp for schedule(dynamic, 64)
        for (int64_t u = 0; u < nr; ++u) {
            if (!g) continue;
            const int64_t i = rstart[u], e = rstart[u + 1];
            const int64_t key = skeys[i];
            int t = 0;
            while (rowbase[t + 1] <= key) ++t;
            const int64_t r = key - rowbase[t];
            const int D = dims[t];
            for (int j = 0; j < D; ++j) g[j] = 0.0;
            for (int64_t k = i; k < e; ++k) {
                const int64_t pos = spos[k];
                const int64_t bag = bag_of[pos];
                double s = weights ? (double)weights[pos] : 1.0;
                if (mean_pooling) {
                    const int64_t L = load_index(offsets, index_is64, bag + 1) -
                                      load_index(offsets, index_is64, bag);
                    s = s / (double)L;
                }
                const int64_t b = bag - (int64_t)t * B;
                const float* grow = grad_out + b * total_d + doff[t];
                for (int j = 0; j < D; ++j) g[j] += s * (double)grow[j];
            }
            if (row_grads) {
                for (int j = 0; j < maxd; ++j) row_grads[u * maxd + j] = j < D ? g[j] : 0.0;
                row_keys[u] = key;
            }
            /* one optimizer step for this row */
            if (optimizer == OPT_SGD) {
                for (int j = 0; j < D; ++j) {
                    const double w = load_elem(tables[t], dtypes[t], r * D + j);
                    store_elem(tables[t], dtypes[t], r * D + j, w - (double)lr * g[j]);
                }
            } else if (optimizer == OPT_ROWWISE_ADAGRAD) {
                double sq = 0.0;
                for (int j = 0; j < D; ++j) sq += g[j] * g[j];
                const double m = (double)state[key] + sq / (double)D;
                state[key] = (float)m;
                const double denom = sqrt(m) + (double)eps;
                for (int j = 0; j < D; ++j) {
                    const double w = load_elem(tables[t], dtypes[t], r * D + j);
                    store_elem(tables[t], dtypes[t], r * D + j, w - (double)lr * g[j] / denom);
                }
            }
        }
        free(g);
    }
    if (nomem) {
        rc = OR_NO_MEMORY;
        goto done;
    }
    if (n_rows) *n_rows = nr;

done:
    free(keys);
    free(bag_of);
    free(skeys);
    free(spos);
    free(rowbase);
    free(doff);
    free(rstart);
    return rc;
}
