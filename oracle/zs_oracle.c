/*
 * CPU fp64 oracle for the GIE zonal scatter.  TEST INFRASTRUCTURE.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this file's library.  It shares no source with the CUDA path.
 *
 * What it computes follows the deepmd-kit pull request "fused Triton zonal
 * scatter for the GIE head (DP_GIE_SCATTER_INFER)":
 *   - section "What", forward bullet: a destination CSR in stable edge order
 *     is walked per node and the per-edge message is summed into the padded
 *     (N, D, C) node layout whose scalar row 0 is zero;
 *   - section "What", backward bullet: per edge, the coupling gradient
 *     (E, D-1) and the radial gradient (E, lmax, C);
 *   - section "Boundary and layout contract": the lmax = 3 ladder packs the
 *     15 zonal rows as contiguous degree groups of 3, 5 and 7 rows.
 *
 * The ladder of degree lmax has D = (lmax+1)^2 node rows: the scalar row and
 * D - 1 zonal rows packed as contiguous degree groups of 2l+1 rows for
 * l = 1..lmax, so row r belongs to degree l for r in [l^2 - 1, (l+1)^2 - 1)
 * (degree 1: rows 0..2, degree 2: rows 3..7, degree 3: rows 8..14, ...); the
 * radial slot of degree l is l - 1.  lmax = 3 is the pages' operator; other
 * lmax (1..5) extend it the same way.
 *
 * Message, forward and backward (plain definition, accumulated in fp64):
 *   msg[e,r,c]    = coup[e,r] * rad[e, slot(r), c]
 *   out[n,0,c]    = 0
 *   out[n,1+r,c]  = sum over CSR positions j of n, in order, of msg[perm[j],r,c]
 *   d_coup[e,r]   = sum_c g[dst[e],1+r,c] * rad[e,slot(r),c]
 *   d_rad[e,s,c]  = sum_{r: slot(r)=s} g[dst[e],1+r,c] * coup[e,r]
 *
 * Readings where the pages are silent: a destination outside [0, N) belongs
 * to no node; the CSR places such edges after all valid ones, in edge order,
 * and counts them; the backward gives such edges zero gradients.
 *
 * Alongside every value the oracle returns the sum of |terms| that formed
 * it, the denominator of the normalised error used to assess fp32 results.
 */
#include <math.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* degree group of zonal row r, as a radial slot index (degree - 1): the
 * degree l of row r is the one whose group [l^2 - 1, (l+1)^2 - 1) holds r */
static int slot_of_row(int r) {
    int l = 1;
    while ((l + 1) * (l + 1) - 1 <= r) ++l;
    return l - 1;
}

/*
 * Stable destination CSR by counting sort with a sequential cursor.
 * row_ptr has N+1 entries, perm has E.  Edges with dst outside [0, N) follow
 * all valid edges in perm, in edge order.  Returns the number of such edges.
 */
int64_t oracle_build_csr(const int32_t* dst, int64_t E, int32_t N,
                         int32_t* row_ptr, int32_t* perm) {
    int64_t* count = (int64_t*)calloc((size_t)N + 1, sizeof(int64_t));
    int64_t bad = 0;
    for (int64_t e = 0; e < E; ++e) {
        int32_t d = dst[e];
        if (d >= 0 && d < N) count[d] += 1; else bad += 1;
    }
    int64_t run = 0;
    for (int32_t n = 0; n < N; ++n) {
        row_ptr[n] = (int32_t)run;
        run += count[n];
    }
    row_ptr[N] = (int32_t)run;
    /* cursor per node, starting at its segment; bad edges start at run */
    int64_t* cursor = count;
    for (int32_t n = 0; n < N; ++n) cursor[n] = row_ptr[n];
    int64_t bad_cursor = run;
    for (int64_t e = 0; e < E; ++e) {
        int32_t d = dst[e];
        if (d >= 0 && d < N) perm[cursor[d]++] = (int32_t)e;
        else perm[bad_cursor++] = (int32_t)e;
    }
    free(count);
    return bad;
}

/*
 * Forward for the nodes listed in `nodes` (or all N nodes when nodes == NULL,
 * in which case n_nodes is ignored).  coup is (E, D-1), rad (E, lmax, C);
 * out and absum are (n_out, D, C) fp64, one block per listed node, in list
 * order.
 */
void oracle_forward(const float* coup, const float* rad,
                    const int32_t* row_ptr, const int32_t* perm,
                    int32_t N, int32_t C, int32_t lmax,
                    const int32_t* nodes, int64_t n_nodes,
                    double* out, double* absum) {
    const int D = (lmax + 1) * (lmax + 1), R = D - 1, S = lmax;
    int64_t n_out = nodes ? n_nodes : (int64_t)N;
    size_t block = (size_t)D * (size_t)C;
    memset(out, 0, sizeof(double) * block * (size_t)n_out);
    if (absum) memset(absum, 0, sizeof(double) * block * (size_t)n_out);
    /* nodes are independent: each is summed by one thread in CSR order */
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 16)
#endif
    for (int64_t k = 0; k < n_out; ++k) {
        int32_t n = nodes ? nodes[k] : (int32_t)k;
        double* o = out + block * (size_t)k;
        double* a = absum ? absum + block * (size_t)k : NULL;
        for (int32_t j = row_ptr[n]; j < row_ptr[n + 1]; ++j) {
            int64_t e = perm[j];
            const float* cp = coup + (size_t)e * R;
            const float* rp = rad + (size_t)e * S * (size_t)C;
            for (int r = 0; r < R; ++r) {
                double cv = (double)cp[r];
                const float* rs = rp + (size_t)slot_of_row(r) * (size_t)C;
                double* orow = o + (size_t)(1 + r) * (size_t)C;
                double* arow = a ? a + (size_t)(1 + r) * (size_t)C : NULL;
                for (int32_t c = 0; c < C; ++c) {
                    double t = cv * (double)rs[c];
                    orow[c] += t;
                    if (arow) arow[c] += fabs(t);
                }
            }
        }
    }
}

/*
 * Backward for the edges listed in `edges` (or all E edges when
 * edges == NULL).  d_coup / abs_dcoup are (n_out, D-1), d_rad / abs_drad are
 * (n_out, lmax, C), fp64, one block per listed edge in list order.  g is the
 * (N, D, C) output cotangent; its row 0 is never read.
 */
void oracle_backward(const float* g, const float* coup, const float* rad,
                     const int32_t* dst, int64_t E, int32_t N, int32_t C, int32_t lmax,
                     const int64_t* edges, int64_t n_edges,
                     double* d_coup, double* d_rad,
                     double* abs_dcoup, double* abs_drad) {
    const int D = (lmax + 1) * (lmax + 1), R = D - 1, S = lmax;
    int64_t n_out = edges ? n_edges : E;
    /* edges are independent: each one's gradients by one thread */
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t k = 0; k < n_out; ++k) {
        int64_t e = edges ? edges[k] : k;
        double* dc = d_coup + (size_t)k * R;
        double* dr = d_rad + (size_t)k * S * (size_t)C;
        double* adc = abs_dcoup ? abs_dcoup + (size_t)k * R : NULL;
        double* adr = abs_drad ? abs_drad + (size_t)k * S * (size_t)C : NULL;
        for (int r = 0; r < R; ++r) { dc[r] = 0.0; if (adc) adc[r] = 0.0; }
        for (size_t i = 0; i < (size_t)S * (size_t)C; ++i) { dr[i] = 0.0; if (adr) adr[i] = 0.0; }
        int32_t d = dst[e];
        if (d < 0 || d >= N) continue;
        const float* cp = coup + (size_t)e * R;
        const float* rp = rad + (size_t)e * S * (size_t)C;
        const float* gn = g + (size_t)d * D * (size_t)C;
        for (int r = 0; r < R; ++r) {
            int s = slot_of_row(r);
            const float* grow = gn + (size_t)(1 + r) * (size_t)C;
            const float* rs = rp + (size_t)s * (size_t)C;
            double cv = (double)cp[r];
            for (int32_t c = 0; c < C; ++c) {
                double gv = (double)grow[c];
                double tc = gv * (double)rs[c];
                dc[r] += tc;
                if (adc) adc[r] += fabs(tc);
                double tr = gv * cv;
                dr[(size_t)s * (size_t)C + c] += tr;
                if (adr) adr[(size_t)s * (size_t)C + c] += fabs(tr);
            }
        }
    }
}

/* Row-to-slot map as the oracle uses it, for the tests' cross-checks. */
int oracle_slot_of_row(int r) { return slot_of_row(r); }

/* Threads the forward and backward loops may use (1 unless raised); the
 * arithmetic of every node and edge is the same whatever the count. */
void oracle_set_threads(int n) {
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : 1);
#else
    (void)n;
#endif
}
