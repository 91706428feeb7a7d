/*
 * pk_oracle.c -- plain, slow, single-threaded CPU oracle for the Jacobi
 * 5-point Laplace/Poisson solver.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline / reference arm may load this library.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * Sources (page title -- section):
 *   [P1] "Persistent Kernels: Bridging GPU-CPU Execution"
 *        -- "The problem (another PDE solver)": Poisson's equation on the
 *           unit square, central differences, the update
 *           u_ij <- 1/4 (u_{i+1,j} + u_{i-1,j} + u_{i,j+1} + u_{i,j-1} - D^2 f_ij)
 *        -- "Implementation details and correctness": Jacobi computes every
 *           point from the previous iteration's values into a separate
 *           result matrix; convergence measured by the change between
 *           iterations.
 *   [P2] "Grid-Wide Barriers and Persistent Work Queues"
 *        -- "What the barrier buys": the convergence check is a reduction
 *           whose result every block reads after the barrier; the solver
 *           stops early without a host round trip.
 *   [P3] "CUDA persist kernel" (finaltheory) -- "Ping-Pong Buffer":
 *           two buffers alternate between iterations.
 *
 * Readings taken where the pages are silent (each is stated again where it
 * is used):
 *   - the field is (ny+2) x (nx+2) fp32, row-major, packed, the outer ring
 *     holds the Dirichlet values and is never written;
 *   - h = 1/(nx+1); h2 = (float)(1.0 / ((double)(nx+1)^2)), the double
 *     quotient rounded once to float; g = fl32(h2 * f);
 *   - summation order (W+E)+(S+N), then - g, then * 0.25f; every operation
 *     is one IEEE binary32 operation, rounded to nearest even, no FMA
 *     contraction (build with -ffp-contract=off), no flush to zero;
 *   - residual of iterate U: r = fl32(t - 4*C) with t the same value the
 *     sweep computes before the 1/4 (so for Poisson t already has -g);
 *     its L2 norm accumulates (double)r*(double)r with Neumaier-compensated
 *     summation in row-major order; max|r| is also reported;
 *   - with checks on, iterate k is checked when k % check_every == 0; the
 *     run stops at the first checked k > 0 with res_k < tol * res_0 and
 *     returns U_k, or at k == n and returns U_n.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared [-fopenmp].  With
 * threads > 1 the row loop of a sweep is split across OpenMP threads; every
 * cell's arithmetic is unchanged, so the result is the same bit for bit.
 * The residual is always summed by one thread in row-major order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int64_t sweeps_done;  /* index k of the iterate returned */
    double res0;          /* ||r(U_0)||_2, 0 when checks are off */
    double res_last;      /* ||r(U_k)||_2 at the last check */
    float rmax_last;      /* max |r(U_k)| at the last check */
    int32_t n_checks;     /* number of residual evaluations */
} oracle_info;

/* Row-major index into the packed (ny+2) x (nx+2) field. */
#define AT(u, nx, j, i) ((u)[(size_t)(j) * (size_t)((nx) + 2) + (size_t)(i)])

/* h^2 with h = 1/(nx+1): double quotient, rounded once to float. */
float oracle_h2(int nx)
{
    double np1 = (double)nx + 1.0;
    return (float)(1.0 / (np1 * np1));
}

/* g = fl32(h2 * f) over the ny x nx interior (row-major, packed). */
void oracle_scale_source(int nx, int ny, float h2, const float *f, float *g)
{
    size_t count = (size_t)nx * (size_t)ny;
    for (size_t q = 0; q < count; ++q) {
        float prod = h2 * f[q];
        g[q] = prod;
    }
}

/* The pre-quarter value t of the update at interior cell (j, i) of u:
 * t = ((W + E) + (S + N)) [- g].  [P1] "The problem": the update rule. */
static float stencil_t(int nx, const float *u, const float *g, int j, int i)
{
    float w = AT(u, nx, j, i - 1);
    float e = AT(u, nx, j, i + 1);
    float s = AT(u, nx, j - 1, i);
    float n = AT(u, nx, j + 1, i);
    float we = w + e;
    float sn = s + n;
    float t = we + sn;
    if (g) {
        float gv = g[(size_t)(j - 1) * (size_t)nx + (size_t)(i - 1)];
        t = t - gv;
    }
    return t;
}

/* One Jacobi sweep [P1] "Implementation details": every interior cell of
 * dst is computed from src only; the ring of dst is copied from src. */
void oracle_sweep(int nx, int ny, const float *src, float *dst, const float *g,
                  int threads)
{
    /* Ring: rows 0 and ny+1 whole, columns 0 and nx+1 of the other rows. */
    memcpy(&AT(dst, nx, 0, 0), &AT(src, nx, 0, 0), sizeof(float) * (size_t)(nx + 2));
    memcpy(&AT(dst, nx, ny + 1, 0), &AT(src, nx, ny + 1, 0),
           sizeof(float) * (size_t)(nx + 2));
    for (int j = 1; j <= ny; ++j) {
        AT(dst, nx, j, 0) = AT(src, nx, j, 0);
        AT(dst, nx, j, nx + 1) = AT(src, nx, j, nx + 1);
    }
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : 1) if (threads > 1)
#endif
    for (int j = 1; j <= ny; ++j) {
        for (int i = 1; i <= nx; ++i) {
            float t = stencil_t(nx, src, g, j, i);
            AT(dst, nx, j, i) = 0.25f * t;
        }
    }
    (void)threads;
}

/* Residual of iterate u: r = fl32(t - 4C); returns sqrt of the
 * Neumaier-compensated row-major sum of (double)r^2 and max|r|. */
void oracle_residual(int nx, int ny, const float *u, const float *g, double *res_out,
                     float *rmax_out)
{
    double sum = 0.0, comp = 0.0;
    float rmax = 0.0f;
    for (int j = 1; j <= ny; ++j) {
        for (int i = 1; i <= nx; ++i) {
            float t = stencil_t(nx, u, g, j, i);
            float c4 = 4.0f * AT(u, nx, j, i);
            float r = t - c4;
            double sq = (double)r * (double)r;
            double s_new = sum + sq;
            if (fabs(sum) >= fabs(sq))
                comp += (sum - s_new) + sq;
            else
                comp += (sq - s_new) + sum;
            sum = s_new;
            float ar = fabsf(r);
            if (ar > rmax) rmax = ar;
        }
    }
    *res_out = sqrt(sum + comp);
    *rmax_out = rmax;
}

/* Full run: copies u0 into two buffers (ping-pong, [P3] "Ping-Pong
 * Buffer"), sweeps, checks the residual ([P2] "What the barrier buys") and
 * writes the returned iterate to out.  f may be NULL (Laplace).  Checks are
 * off when tol <= 0 or check_every <= 0.  Returns 0, or -1 on bad sizes or
 * allocation failure. */
int oracle_jacobi_run(int nx, int ny, float h2, const float *u0, const float *f, int64_t n,
                      float tol, int check_every, int threads, float *out,
                      oracle_info *info)
{
    if (nx <= 0 || ny <= 0 || n < 0) return -1;
    size_t cells = (size_t)(nx + 2) * (size_t)(ny + 2);
    float *buf[2];
    buf[0] = (float *)malloc(sizeof(float) * cells);
    buf[1] = (float *)malloc(sizeof(float) * cells);
    float *g = NULL;
    if (f) g = (float *)malloc(sizeof(float) * (size_t)nx * (size_t)ny);
    if (!buf[0] || !buf[1] || (f && !g)) {
        free(buf[0]);
        free(buf[1]);
        free(g);
        return -1;
    }
    memcpy(buf[0], u0, sizeof(float) * cells);
    memcpy(buf[1], u0, sizeof(float) * cells);
    if (f) oracle_scale_source(nx, ny, h2, f, g);

    int checks = (tol > 0.0f && check_every > 0);
    double res0 = 0.0, res_last = 0.0;
    float rmax_last = 0.0f;
    int32_t n_checks = 0;
    int64_t k = 0;
    for (;;) {
        const float *cur = buf[k & 1];
        if (checks && (k % check_every) == 0) {
            double res;
            float rmax;
            oracle_residual(nx, ny, cur, g, &res, &rmax);
            ++n_checks;
            res_last = res;
            rmax_last = rmax;
            if (k == 0) {
                res0 = res;
            } else if (res < (double)tol * res0) {
                break;
            }
        }
        if (k == n) break;
        oracle_sweep(nx, ny, cur, buf[(k + 1) & 1], g, threads);
        ++k;
    }
    memcpy(out, buf[k & 1], sizeof(float) * cells);
    if (info) {
        info->sweeps_done = k;
        info->res0 = res0;
        info->res_last = res_last;
        info->rmax_last = rmax_last;
        info->n_checks = n_checks;
    }
    free(buf[0]);
    free(buf[1]);
    free(g);
    return 0;
}

/* ---- red-black Gauss-Seidel -------------------------------------------
 * [P1] "Implementation details and correctness": first update every point
 * whose i and j have the same parity (red), then every other point (black);
 * a half-sweep reads only the other colour, so the update is in place and
 * the black half-sweep sees the new red values.  Each point uses the same
 * arithmetic as the Jacobi update. */
void oracle_rb_half_sweep(int nx, int ny, float *u, const float *g, int colour)
{
    for (int j = 1; j <= ny; ++j) {
        for (int i = 1; i <= nx; ++i) {
            if (((i + j) & 1) != colour) continue;
            float t = stencil_t(nx, u, g, j, i);
            AT(u, nx, j, i) = 0.25f * t;
        }
    }
}

/* Full red-black run: iteration k = red half-sweep then black half-sweep.
 * Checks, exit rule and returned iterate as oracle_jacobi_run (the residual
 * of U_k is taken before iteration k). */
int oracle_rb_run(int nx, int ny, float h2, const float *u0, const float *f, int64_t n, float tol,
                  int check_every, float *out, oracle_info *info)
{
    if (nx <= 0 || ny <= 0 || n < 0) return -1;
    size_t cells = (size_t)(nx + 2) * (size_t)(ny + 2);
    float *g = NULL;
    if (f) {
        g = (float *)malloc(sizeof(float) * (size_t)nx * (size_t)ny);
        if (!g) return -1;
        oracle_scale_source(nx, ny, h2, f, g);
    }
    memcpy(out, u0, sizeof(float) * cells);
    int checks = (tol > 0.0f && check_every > 0);
    double res0 = 0.0, res_last = 0.0;
    float rmax_last = 0.0f;
    int32_t n_checks = 0;
    int64_t k = 0;
    for (;;) {
        if (checks && (k % check_every) == 0) {
            double res;
            float rmax;
            oracle_residual(nx, ny, out, g, &res, &rmax);
            ++n_checks;
            res_last = res;
            rmax_last = rmax;
            if (k == 0) {
                res0 = res;
            } else if (res < (double)tol * res0) {
                break;
            }
        }
        if (k == n) break;
        oracle_rb_half_sweep(nx, ny, out, g, 0);
        oracle_rb_half_sweep(nx, ny, out, g, 1);
        ++k;
    }
    if (info) {
        info->sweeps_done = k;
        info->res0 = res0;
        info->res_last = res_last;
        info->rmax_last = rmax_last;
        info->n_checks = n_checks;
    }
    free(g);
    return 0;
}

/* y <- fl32(fl32(a * x) + y), element by element. */
void oracle_axpy(int64_t len, float a, const float *x, float *y)
{
    for (int64_t q = 0; q < len; ++q) {
        float ax = a * x[q];
        y[q] = ax + y[q];
    }
}

/* Host-driven task sequence: task t = 0 .. n_tasks-1; even t is one Jacobi
 * sweep (Laplace) of the (ny+2) x (nx+2) field, odd t is y <- a*x + y.
 * field is updated in place with the returned iterate. */
int oracle_task_sequence(int nx, int ny, float *field, int64_t len, float a, const float *x,
                         float *y, int64_t n_tasks)
{
    size_t cells = (size_t)(nx + 2) * (size_t)(ny + 2);
    float *other = (float *)malloc(sizeof(float) * cells);
    if (!other) return -1;
    memcpy(other, field, sizeof(float) * cells);
    float *cur = field, *nxt = other;
    for (int64_t t = 0; t < n_tasks; ++t) {
        if ((t & 1) == 0) {
            oracle_sweep(nx, ny, cur, nxt, NULL, 1);
            float *tmp = cur;
            cur = nxt;
            nxt = tmp;
        } else {
            oracle_axpy(len, a, x, y);
        }
    }
    if (cur != field) memcpy(field, cur, sizeof(float) * cells);
    free(other);
    return 0;
}

/* ---- grid-barrier stress: expected observations ----------------------
 * The stress kernel runs `rounds` rounds over `nblocks` CTAs.  In round r
 * CTA b writes `words` 32-bit stamps w = 0..words-1, each the low 32 bits of
 * mix64(((r * nblocks + b) * words + w) + 1), where mix64 is the SplitMix64
 * output function (Steele, Lea, Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014).  After the barrier CTA b reads every word of
 * the CTAs (b+1), (b + nblocks/2) and (b + r + 1), all mod nblocks, and adds
 * each value (as uint64) into a wrapping 64-bit checksum.  The oracle gives
 * each CTA's checksum after all rounds. */
static uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static uint32_t stamp(uint64_t r, uint64_t nblocks, uint64_t b, uint64_t words, uint64_t w)
{
    return (uint32_t)mix64(((r * nblocks + b) * words + w) + 1ull);
}

void oracle_barrier_stress(int nblocks, int rounds, int words, uint64_t *checksums)
{
    for (int b = 0; b < nblocks; ++b) {
        uint64_t acc = 0;
        for (int r = 0; r < rounds; ++r) {
            int peers[3];
            peers[0] = (b + 1) % nblocks;
            peers[1] = (b + nblocks / 2) % nblocks;
            peers[2] = (int)(((int64_t)b + r + 1) % nblocks);
            for (int p = 0; p < 3; ++p)
                for (int w = 0; w < words; ++w)
                    acc += (uint64_t)stamp((uint64_t)r, (uint64_t)nblocks, (uint64_t)peers[p],
                                           (uint64_t)words, (uint64_t)w);
        }
        checksums[b] = acc;
    }
}

int oracle_has_openmp(void)
{
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}
