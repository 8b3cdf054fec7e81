/*
 * CPU oracle for the fused cross-entropy loss -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline /
 * reference legs may load this file's library.  It shares no code with the CUDA
 * path and is deliberately plain: float64 throughout, one row at a time, sums in
 * ascending column order, no blocking, no fusion.
 *
 * What it computes (the FOAK pages name the kernel -- "Fast Cross Entropy Triton
 * Kernels" on the fms-acceleration-foak 0.7.4 page, FastCrossEntropyLoss in
 * fms-acceleration PR #79 "Allow Kernels for Full FT and Non-Quantized PEFT" --
 * but never write out its formula; the reading taken here is the textbook
 * softmax cross-entropy with mean reduction over rows whose label is not
 * ignore_index, which is the loss that kernel replaces in a causal-LM head):
 *
 *   row i, label y_i:   ignored if y_i == ignore_index; invalid (reported, and
 *                       then treated like an ignored row) if y_i is outside [0,V)
 *   m_i   = max_j x_ij
 *   S_i   = sum_j exp(x_ij - m_i)
 *   lse_i = m_i + ln S_i
 *   l_i   = lse_i - x_i,y_i
 *   loss  = (sum over valid i of l_i) / D,   D = denom if denom > 0 else n_valid
 *   dx_ij = (g / D) * (exp(x_ij - lse_i) - [j == y_i])   for valid rows, 0 else
 *
 * n_valid == 0 with no denom gives loss = 0/0 = NaN and an all-zero gradient.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { OR_F32 = 0, OR_BF16 = 1, OR_F64 = 2 };
enum { OR_IGNORED = 0, OR_VALID = 1, OR_BAD_LABEL = 2 };

/* Element j of row r, widened exactly to double. */
static double elem(const void* x, int dtype, int64_t ld, int64_t r, int64_t j) {
    int64_t k = r * ld + j;
    if (dtype == OR_F32) return (double)((const float*)x)[k];
    if (dtype == OR_F64) return ((const double*)x)[k];
    uint32_t bits = (uint32_t)((const uint16_t*)x)[k] << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

static int row_state(int64_t y, int64_t V, int64_t ignore_index) {
    if (y == ignore_index) return OR_IGNORED;
    if (y < 0 || y >= V) return OR_BAD_LABEL;
    return OR_VALID;
}

/* Count rows with a usable label, and rows whose label is out of range. */
void oracle_ce_count(const int64_t* labels, int64_t N, int64_t V, int64_t ignore_index,
                     int64_t* n_valid, int64_t* n_bad) {
    int64_t nv = 0, nb = 0;
    for (int64_t i = 0; i < N; ++i) {
        int s = row_state(labels[i], V, ignore_index);
        nv += s == OR_VALID;
        nb += s == OR_BAD_LABEL;
    }
    *n_valid = nv;
    *n_bad = nb;
}

/*
 * Rows [r0, r1): per-row state, lse and loss term; and, when grad != NULL, the
 * gradient rows scaled by `scale` (= g / D), written densely as (r1-r0) x V.
 * x points at row 0 of the whole matrix (row stride ld elements).
 * Ignored and bad-label rows get lse = 0, loss term = 0 and a zero gradient row.
 */
void oracle_ce_rows(const void* x, int dtype, int64_t ld, const int64_t* labels, int64_t r0,
                    int64_t r1, int64_t V, int64_t ignore_index, double scale, double* lse,
                    double* row_loss, int8_t* state, double* grad) {
    for (int64_t r = r0; r < r1; ++r) {
        int64_t o = r - r0;
        int s = row_state(labels[r], V, ignore_index);
        state[o] = (int8_t)s;
        double* gr = grad ? grad + o * V : NULL;
        if (s != OR_VALID) {
            lse[o] = 0.0;
            row_loss[o] = 0.0;
            if (gr)
                for (int64_t j = 0; j < V; ++j) gr[j] = 0.0;
            continue;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < V; ++j) {
            double v = elem(x, dtype, ld, r, j);
            if (v > m) m = v;
        }
        double S = 0.0;
        for (int64_t j = 0; j < V; ++j) S += exp(elem(x, dtype, ld, r, j) - m);
        double l = m + log(S);
        int64_t y = labels[r];
        lse[o] = l;
        row_loss[o] = l - elem(x, dtype, ld, r, y);
        if (gr) {
            for (int64_t j = 0; j < V; ++j) {
                double p = exp(elem(x, dtype, ld, r, j) - l);
                gr[j] = scale * (p - (j == y ? 1.0 : 0.0));
            }
        }
    }
}

/* Mean of the valid rows' loss terms over D (denom if > 0, else n_valid), summed in row order. */
double oracle_ce_mean(const double* row_loss, const int8_t* state, int64_t N, double denom) {
    double sum = 0.0;
    int64_t nv = 0;
    for (int64_t i = 0; i < N; ++i) {
        if (state[i] == OR_VALID) {
            sum += row_loss[i];
            nv += 1;
        }
    }
    double D = denom > 0.0 ? denom : (double)nv;
    return sum / D;
}
