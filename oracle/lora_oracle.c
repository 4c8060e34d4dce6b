/*
 * lora_oracle.c -- plain CPU fp64 oracle for the mixed-adapter LoRA linear layer.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg load this library.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * What it computes (fp64, from the exact values of the given inputs):
 *
 *   y[i,n] = sum_k x[i,k] W[k,n]
 *          + [slot_i != -1] * (alpha_s / r_s) * sum_{j<r_s} (sum_k x[i,k] A_s[k,j]) B_s[j,n],
 *            with s = slot_i.
 *
 * Sources:
 *  - "Serving multiple LoRAs: segmented matrix multiplies and adapter scheduling",
 *    section "Not merging the weights, computing in batches": y = xW + s*(xA)B with
 *    A in R^{d x r}, B in R^{r x d'}; the base product is shared, the low-rank part is
 *    computed per request; BGMV gathers per token, SGMV groups same-adapter tokens.
 *  - "LoRAX, in depth", section "Computing a batch that mixes adapters": s = alpha / r,
 *    segments given by boundaries of length n_segments + 1, an owner per segment,
 *    "None" meaning base only.
 *  - "Multi-LoRA Serving 与 Adapter 隔离" (llm-glossary), sections on adapter ownership
 *    in one continuous batch and the runnable grouped-batch experiment:
 *    group rows by adapter, compute each group, scatter back to row order; each group
 *    also equals x times the merged weight W + (alpha/r) A B.
 *  - "Serving LoRA adapters: from the model name to the wrapped layer" (vLLM),
 *    Step 5: a token without an adapter maps to slot -1.
 *
 * Three independent evaluators of the same definition are provided:
 *   oracle_forward_rows    -- row by row, the naive per-request loop;
 *   oracle_forward_grouped -- one shared base product, then one small product per
 *                             segment of rows sorted by slot, scattered back;
 *   oracle_forward_merged  -- x times W' = W + (alpha/r) A B per adapter.
 * and the reference segment builder oracle_segments (a stable sort of the adapted
 * rows by slot, written as the definition: for each slot in ascending order, list
 * its rows in their original order).
 *
 * Layouts (all row-major, C order):
 *   x      [T][K]        W [K][N]
 *   A      [S][K][R]     adapter s uses columns j < rank[s]; the rest is ignored
 *   B      [S][R][N]     adapter s uses rows    j < rank[s]; the rest is ignored
 *   rank   [S] (int32, 1..R), alpha [S] (double), slot [T] (int32, -1 = base only)
 * Rows whose slot is outside [-1, S) are counted as bad and treated as base only.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

static int slot_is_adapted(int32_t s, int S) { return s >= 0 && s < S; }

/*
 * Segment builder: the adapted rows (slot in [0, S)) sorted stably by slot.
 * perm[0..T_a) lists row indices; seg_offsets[0..n_seg] are boundaries into perm;
 * seg_slot[g] is the slot owning segment g; slots with no rows get no segment.
 * Returns the number of rows whose slot id lies outside [-1, S).
 */
int oracle_segments(int T, const int32_t* slot, int S,
                    int32_t* perm, int32_t* seg_offsets, int32_t* seg_slot,
                    int32_t* n_seg_out)
{
    int bad = 0;
    for (int i = 0; i < T; i++)
        if (slot[i] < -1 || slot[i] >= S) bad++;

    int p = 0, g = 0;
    seg_offsets[0] = 0;
    for (int s = 0; s < S; s++) {
        int count = 0;
        for (int i = 0; i < T; i++) {
            if (slot[i] == s) {
                perm[p++] = i;
                count++;
            }
        }
        if (count > 0) {
            seg_slot[g] = s;
            g++;
            seg_offsets[g] = p;
        }
    }
    *n_seg_out = g;
    return bad;
}

/*
 * Evaluator 1, row by row.  Computes the requested rows only: y[q][:] is row rows[q].
 */
void oracle_forward_rows(int T, int K, int N, int S, int R,
                         const double* x, const double* W,
                         const double* A, const double* B,
                         const int32_t* rank, const double* alpha,
                         const int32_t* slot,
                         int nrows, const int64_t* rows, double* y)
{
    (void)T;
#pragma omp parallel
    {
        double* v = (double*)malloc(sizeof(double) * (size_t)(R > 0 ? R : 1));
#pragma omp for schedule(dynamic, 1)
        for (int q = 0; q < nrows; q++) {
            const int64_t i = rows[q];
            const double* xi = x + (size_t)i * K;
            double* yi = y + (size_t)q * N;

            /* base term: sum_k x[i,k] W[k,n] */
            for (int n = 0; n < N; n++) yi[n] = 0.0;
            for (int k = 0; k < K; k++) {
                const double xk = xi[k];
                const double* Wk = W + (size_t)k * N;
                for (int n = 0; n < N; n++) yi[n] += xk * Wk[n];
            }

            const int32_t s = slot[i];
            if (!slot_is_adapted(s, S)) continue;
            const int r = rank[s];
            const double scale = alpha[s] / (double)r;
            const double* As = A + (size_t)s * K * R;
            const double* Bs = B + (size_t)s * R * N;

            /* shrink: v_j = sum_k x[i,k] A_s[k,j] */
            for (int j = 0; j < r; j++) {
                double acc = 0.0;
                for (int k = 0; k < K; k++) acc += xi[k] * As[(size_t)k * R + j];
                v[j] = acc;
            }
            /* expand: y[i,n] += scale * sum_j v_j B_s[j,n] */
            for (int n = 0; n < N; n++) {
                double d = 0.0;
                for (int j = 0; j < r; j++) d += v[j] * Bs[(size_t)j * N + n];
                yi[n] += scale * d;
            }
        }
        free(v);
    }
}

/*
 * Evaluator 2, grouped: one base product over all rows, then per segment of rows
 * sharing a slot: gather the rows, V = X_g A_s, D = scale * V B_s, scatter-add D.
 * Writes all T rows of y.  Returns the bad-id count of the segment builder.
 */
int oracle_forward_grouped(int T, int K, int N, int S, int R,
                           const double* x, const double* W,
                           const double* A, const double* B,
                           const int32_t* rank, const double* alpha,
                           const int32_t* slot, double* y)
{
    /* shared base product Y = X W */
#pragma omp parallel for schedule(static)
    for (int i = 0; i < T; i++) {
        double* yi = y + (size_t)i * N;
        const double* xi = x + (size_t)i * K;
        for (int n = 0; n < N; n++) yi[n] = 0.0;
        for (int k = 0; k < K; k++) {
            const double xk = xi[k];
            const double* Wk = W + (size_t)k * N;
            for (int n = 0; n < N; n++) yi[n] += xk * Wk[n];
        }
    }

    int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    int32_t* offs = (int32_t*)malloc(sizeof(int32_t) * (size_t)(S + 1));
    int32_t* sslot = (int32_t*)malloc(sizeof(int32_t) * (size_t)(S > 0 ? S : 1));
    int32_t n_seg = 0;
    const int bad = oracle_segments(T, slot, S, perm, offs, sslot, &n_seg);

    for (int g = 0; g < n_seg; g++) {
        const int s = sslot[g];
        const int lo = offs[g], hi = offs[g + 1], m = hi - lo;
        const int r = rank[s];
        const double scale = alpha[s] / (double)r;
        const double* As = A + (size_t)s * K * R;
        const double* Bs = B + (size_t)s * R * N;

        /* gather X_g [m][K] */
        double* Xg = (double*)malloc(sizeof(double) * (size_t)m * K);
        for (int p = 0; p < m; p++)
            memcpy(Xg + (size_t)p * K, x + (size_t)perm[lo + p] * K, sizeof(double) * (size_t)K);

        /* V = X_g A_s  [m][r] */
        double* V = (double*)calloc((size_t)m * r, sizeof(double));
#pragma omp parallel for schedule(static)
        for (int p = 0; p < m; p++)
            for (int k = 0; k < K; k++) {
                const double xv = Xg[(size_t)p * K + k];
                for (int j = 0; j < r; j++) V[(size_t)p * r + j] += xv * As[(size_t)k * R + j];
            }

        /* D = scale * V B_s, scattered back to the original rows */
#pragma omp parallel for schedule(static)
        for (int p = 0; p < m; p++) {
            double* yi = y + (size_t)perm[lo + p] * N;
            for (int n = 0; n < N; n++) {
                double d = 0.0;
                for (int j = 0; j < r; j++) d += V[(size_t)p * r + j] * Bs[(size_t)j * N + n];
                yi[n] += scale * d;
            }
        }
        free(V);
        free(Xg);
    }
    free(sslot);
    free(offs);
    free(perm);
    return bad;
}

/*
 * Evaluator 3, merged weight: for each slot that owns rows, W' = W + (alpha/r) A_s B_s,
 * then y_i = x_i W'.  Base-only rows use W.  Writes all T rows of y.
 */
void oracle_forward_merged(int T, int K, int N, int S, int R,
                           const double* x, const double* W,
                           const double* A, const double* B,
                           const int32_t* rank, const double* alpha,
                           const int32_t* slot, double* y)
{
    double* Wm = (double*)malloc(sizeof(double) * (size_t)K * N);
    /* slot index -1 stands for the base weight itself */
    for (int s = -1; s < S; s++) {
        int used = 0;
        for (int i = 0; i < T; i++) {
            const int32_t si = slot_is_adapted(slot[i], S) ? slot[i] : -1;
            if (si == s) { used = 1; break; }
        }
        if (!used) continue;

        if (s < 0) {
            memcpy(Wm, W, sizeof(double) * (size_t)K * N);
        } else {
            const int r = rank[s];
            const double scale = alpha[s] / (double)r;
            const double* As = A + (size_t)s * K * R;
            const double* Bs = B + (size_t)s * R * N;
#pragma omp parallel for schedule(static)
            for (int k = 0; k < K; k++)
                for (int n = 0; n < N; n++) {
                    double ab = 0.0;
                    for (int j = 0; j < r; j++) ab += As[(size_t)k * R + j] * Bs[(size_t)j * N + n];
                    Wm[(size_t)k * N + n] = W[(size_t)k * N + n] + scale * ab;
                }
        }

#pragma omp parallel for schedule(static)
        for (int i = 0; i < T; i++) {
            const int32_t si = slot_is_adapted(slot[i], S) ? slot[i] : -1;
            if (si != s) continue;
            double* yi = y + (size_t)i * N;
            const double* xi = x + (size_t)i * K;
            for (int n = 0; n < N; n++) yi[n] = 0.0;
            for (int k = 0; k < K; k++) {
                const double xk = xi[k];
                const double* Wk = Wm + (size_t)k * N;
                for (int n = 0; n < N; n++) yi[n] += xk * Wk[n];
            }
        }
    }
    free(Wm);
}
