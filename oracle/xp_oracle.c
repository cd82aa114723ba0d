/*
 * xp_oracle.c -- plain CPU oracle for one XPress Jacobi draft pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load this library.  The CUDA
 * product path never links, imports or calls it, and it shares no code, header
 * or constant with the CUDA sources.
 *
 * It is slow and obviously correct: every floating-point sum accumulates in
 * double, and values are rounded to bf16 exactly where the method rounds them.
 * Source of each definition (vLLM docs, module
 * "vllm.v1.worker.gpu.spec_decode.xpress.kernels", the PR 61746 build [p1] and
 * the PR 66547 build [p2]):
 *
 *   module docstring (both builds): the pass is
 *       latent   u = causal_mix(hcache + embed(prev) @ W_lat), x = u + SwiGLU(u)
 *       readout  logits = base + x @ W2
 *       argmax   blk = argmax_v logits
 *   _xpress_add_argmax_partial_kernel / _reduce_to_blk_kernel: the sum is
 *       rounded to the input dtype (bf16) before it is compared; ties go to
 *       the lowest vocab index; row r = n*(B-1)+b writes blk[n, 1+b].
 *   _xpress_latent_kernel: slot b gathers the embedding of blk[n, b-1]
 *       (slot 0 gathers am1[n]); u[b] = sum_{j<=b} L[b,j,:] * x[j];
 *       ub = bf16(u); m = bf16(silu(ub@Wg) * (ub@Wu)); y = u + m@Wd (residual
 *       on the unrounded u); lat_out[n, b-1] = bf16(y) for b = 1..B-1.
 *   xpress_latent_pass with do_mlp False (the GEMM schedule): the kernel
 *       stops after the mixer and hands back bf16(u); the caller then runs
 *       gu = u @ wgu_t (a bf16 matmul, [Wg | Wu] side by side),
 *       m = silu_and_mul(gu) and u.addmm_(m, wd_t) on the bf16 u.
 *   fused_topc_argmax_to_blk: the top-C variant over gathered candidates.
 *
 * Readings where the pages leave a step open (each is listed in the design
 * notes of the repository):
 *   - the readout bias is rounded to bf16 once (the caller's matmul returns a
 *     bf16 tensor), then added to base and rounded again;
 *   - -0 and +0 compare equal;
 *   - the mixer sums j <= b only (the pages' formula);
 *   - the embedding is E[V, D] and W_lat is [D, R] (D == R is the pages' case).
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC xp_oracle.c -o libxp_oracle.so -lm
 * (OpenMP is optional; without it everything runs on one thread).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_ARG -1
#define ORC_ERR_TOKEN -2
#define ORC_ERR_NONFINITE -3

/* ------------------------------------------------------------------------ */
/* bf16 helpers                                                              */
/* ------------------------------------------------------------------------ */

/* bf16 bits -> the float (and double) value they encode: the top 16 bits of
 * an IEEE binary32. */
static double bf(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round a double to the nearest bf16, ties to even, by arithmetic on the
 * value (not on its bits): find the bf16 spacing at the value's binade and
 * round the scaled value with nearbyint (the default rounding mode is
 * round-to-nearest-even).  Exact: dividing by a power of two is exact and the
 * quotient has at most 53 significant bits. */
static uint16_t bf16_from_double(double d) {
    if (isnan(d)) return (uint16_t)0x7fc0;
    uint16_t sign = signbit(d) ? (uint16_t)0x8000 : (uint16_t)0;
    double a = fabs(d);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7f80);
    int e;
    (void)frexp(a, &e);          /* a = m * 2^e, m in [0.5, 1) */
    int E = e - 1;               /* a in [2^E, 2^(E+1)) */
    if (E < -126) E = -126;      /* subnormal range keeps the smallest spacing */
    double ulp = ldexp(1.0, E - 7);   /* 7 stored fraction bits */
    double q = nearbyint(a / ulp);
    double r = q * ulp;
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7f80);
    float f = (float)r;          /* exact: r is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

/* Round a float to bf16, ties to even, on the bit pattern (add half an ulp
 * minus one, plus the kept lsb, then truncate).  NaNs stay NaN (quiet bit
 * set).  Exported so the tests can check it against the arithmetic rounding
 * above over every float. */
static uint16_t bf16_from_float_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

uint16_t orc_bf16_from_double(double d) { return bf16_from_double(d); }
uint16_t orc_bf16_from_float(float f) { return bf16_from_float_bits(f); }
double orc_double_from_bf16(uint16_t h) { return bf(h); }

void orc_bf16_from_float_array(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_from_float_bits(in[i]);
}
void orc_bf16_from_double_array(const double* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_from_double(in[i]);
}

/* The bf16 sum of two bf16 values, correctly rounded: the double sum of two
 * bf16 values is exact unless their exponents differ by more than 53, and in
 * that case the smaller is far below half a bf16 spacing of the larger and
 * cannot change the rounding. */
static uint16_t bf16_add(uint16_t a, uint16_t b) { return bf16_from_double(bf(a) + bf(b)); }
uint16_t orc_bf16_add(uint16_t a, uint16_t b) { return bf16_add(a, b); }

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int all_finite_bf16(const uint16_t* p, int64_t rows, int64_t cols, int64_t ld) {
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            if ((p[r * ld + c] & 0x7f80u) == 0x7f80u) return 0;
    return 1;
}

/* ------------------------------------------------------------------------ */
/* add-argmax: blk[n, 1+b] = argmax_v bf16(base[r,v] + bias[r,v]),          */
/* r = n*(B-1) + b, lowest index on ties; slot 0 is never written.          */
/* ------------------------------------------------------------------------ */

/* One row: scan v ascending with a strict '>' so the first maximal index
 * wins.  Returns the index; *best_out receives the maximal value. */
static int64_t row_argmax(const uint16_t* base, const uint16_t* bias, int64_t V, double* best_out) {
    double best = -INFINITY;
    int64_t idx = 0;
    for (int64_t v = 0; v < V; ++v) {
        double s = bf(bf16_add(base[v], bias[v]));
        if (s > best) {
            best = s;
            idx = v;
        }
    }
    if (best_out) *best_out = best;
    return idx;
}

int orc_add_argmax(const uint16_t* base, int64_t ld_base, const uint16_t* bias, int64_t ld_bias,
                   int64_t rows, int64_t V, int64_t* blk, int64_t N, int64_t B) {
    if (!base || !bias || !blk || V <= 0 || N < 1 || B < 2 || rows != N * (B - 1)) return ORC_ERR_ARG;
    if (ld_base < V || ld_bias < V) return ORC_ERR_ARG;
    if (!all_finite_bf16(base, rows, V, ld_base) || !all_finite_bf16(bias, rows, V, ld_bias))
        return ORC_ERR_NONFINITE;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        int64_t idx = row_argmax(base + r * ld_base, bias + r * ld_bias, V, NULL);
        int64_t n = r / (B - 1), b = r % (B - 1);
        blk[n * B + 1 + b] = idx;
    }
    return ORC_OK;
}

/* Top-C variant (fused_topc_argmax_to_blk): per row, the argmax over C
 * candidates of bf16(base_c + bias_c), lowest candidate position on ties,
 * mapped back to a vocab id through cand and written to blk[n, 1+b]. */
int orc_topc_argmax(const uint16_t* base_c, const uint16_t* bias_c, const int64_t* cand,
                    int64_t rows, int64_t C, int64_t* blk, int64_t N, int64_t B) {
    if (!base_c || !bias_c || !cand || !blk || C <= 0 || N < 1 || B < 2 || rows != N * (B - 1))
        return ORC_ERR_ARG;
    if (!all_finite_bf16(base_c, rows, C, C) || !all_finite_bf16(bias_c, rows, C, C))
        return ORC_ERR_NONFINITE;
    for (int64_t r = 0; r < rows; ++r) {
        int64_t pos = row_argmax(base_c + r * C, bias_c + r * C, C, NULL);
        int64_t n = r / (B - 1), b = r % (B - 1);
        blk[n * B + 1 + b] = cand[r * C + pos];
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* latent stage (_xpress_latent_kernel), general D.                          */
/* ------------------------------------------------------------------------ */

static double silu_times(double g, double v) { return g * (1.0 / (1.0 + exp(-g))) * v; }

/* One block n.  x, u: B*R doubles of scratch; ub: R; m: H.  Writes
 * lat_out[n, 0..B-2, :] and, when u_out is given, u_out[n, :, :] (the mixer
 * output, before the MLP).  do_mlp selects the MLP schedule: 1 the in-kernel
 * MLP (fp32 g, v and residual), 0 the GEMM schedule (bf16 g, v and residual). */
static int latent_block(int64_t n, const int64_t* blk, const int64_t* am1, const uint16_t* hcache,
                        const uint16_t* E, const uint16_t* W_lat, const float* L, const uint16_t* Wg,
                        const uint16_t* Wu, const uint16_t* Wd, uint16_t* lat_out, int64_t B,
                        int64_t V, int64_t D, int64_t R, int64_t H, int do_mlp, double* u_out, double* x,
                        double* u, double* ubd, double* m) {
    /* gather + projection + hidden cache */
    for (int64_t b = 0; b < B; ++b) {
        int64_t p = (b == 0) ? am1[n] : blk[n * B + b - 1];
        if (p < 0 || p >= V) return ORC_ERR_TOKEN;
        const uint16_t* e = E + p * D;
        double* xb = x + b * R;
        for (int64_t r = 0; r < R; ++r) xb[r] = bf(hcache[(n * B + b) * R + r]);
        for (int64_t k = 0; k < D; ++k) {
            double ek = bf(e[k]);
            const uint16_t* w = W_lat + k * R;
            for (int64_t r = 0; r < R; ++r) xb[r] += ek * bf(w[r]);
        }
    }
    /* causal mixer: u[b] = sum_{j<=b} L[b,j,:] * x[j] */
    for (int64_t b = 0; b < B; ++b) {
        double* ub = u + b * R;
        for (int64_t r = 0; r < R; ++r) ub[r] = 0.0;
        for (int64_t j = 0; j <= b; ++j) {
            const float* l = L + (b * B + j) * R;
            const double* xj = x + j * R;
            for (int64_t r = 0; r < R; ++r) ub[r] += (double)l[r] * xj[r];
        }
        if (u_out)
            for (int64_t r = 0; r < R; ++r) u_out[(n * B + b) * R + r] = ub[r];
    }
    /* SwiGLU MLP with the residual on u, slots 1..B-1 only (slot 0's latent is
     * never read out). */
    for (int64_t b = 1; b < B; ++b) {
        const double* ub = u + b * R;
        for (int64_t r = 0; r < R; ++r) ubd[r] = bf(bf16_from_double(ub[r]));
        if (!do_mlp) {
            /* GEMM schedule: the latent kernel's output is bf16(u) = ubd.
             * gu = bf16(ubd @ [Wg | Wu]): each half rounded to bf16 (the
             * matmul returns a bf16 tensor); silu_and_mul: m = bf16(silu(g) * v)
             * from the bf16 g and v; addmm_ into the bf16 u: the product is
             * added to ubd and the sum rounded to bf16 once. */
            for (int64_t h = 0; h < H; ++h) {
                double g = 0.0, v = 0.0;
                for (int64_t r = 0; r < R; ++r) {
                    g += ubd[r] * bf(Wg[r * H + h]);
                    v += ubd[r] * bf(Wu[r * H + h]);
                }
                m[h] = bf(bf16_from_double(silu_times(bf(bf16_from_double(g)), bf(bf16_from_double(v)))));
            }
            uint16_t* out = lat_out + (n * (B - 1) + (b - 1)) * R;
            for (int64_t r = 0; r < R; ++r) {
                double y = ubd[r];
                for (int64_t h = 0; h < H; ++h) y += m[h] * bf(Wd[h * R + r]);
                out[r] = bf16_from_double(y);
            }
            continue;
        }
        for (int64_t h = 0; h < H; ++h) {
            double g = 0.0, v = 0.0;
            for (int64_t r = 0; r < R; ++r) {
                g += ubd[r] * bf(Wg[r * H + h]);
                v += ubd[r] * bf(Wu[r * H + h]);
            }
            m[h] = bf(bf16_from_double(silu_times(g, v)));
        }
        uint16_t* out = lat_out + (n * (B - 1) + (b - 1)) * R;
        for (int64_t r = 0; r < R; ++r) {
            double y = ub[r];
            for (int64_t h = 0; h < H; ++h) y += m[h] * bf(Wd[h * R + r]);
            out[r] = bf16_from_double(y);
        }
    }
    return ORC_OK;
}

/* Latent for blocks [n_lo, n_hi).  lat_out is the full [N, B-1, R] buffer;
 * u_out (nullable) the full [N, B, R] buffer of mixer outputs in double;
 * do_mlp as in latent_block. */
int orc_latent_ex(const int64_t* blk, const int64_t* am1, const uint16_t* hcache, const uint16_t* E,
                  const uint16_t* W_lat, const float* L, const uint16_t* Wg, const uint16_t* Wu,
                  const uint16_t* Wd, uint16_t* lat_out, int64_t N, int64_t B, int64_t V, int64_t D,
                  int64_t R, int64_t H, int64_t do_mlp, double* u_out, int64_t n_lo, int64_t n_hi) {
    if (!blk || !am1 || !hcache || !E || !W_lat || !L || !Wg || !Wu || !Wd || !lat_out) return ORC_ERR_ARG;
    if (N < 1 || B < 2 || V < 1 || D < 1 || R < 1 || H < 1) return ORC_ERR_ARG;
    if (n_lo < 0 || n_hi > N || n_lo > n_hi) return ORC_ERR_ARG;
    int status = ORC_OK;
#pragma omp parallel
    {
        double* x = (double*)malloc(sizeof(double) * (size_t)(B * R));
        double* u = (double*)malloc(sizeof(double) * (size_t)(B * R));
        double* ubd = (double*)malloc(sizeof(double) * (size_t)R);
        double* m = (double*)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
        for (int64_t n = n_lo; n < n_hi; ++n) {
            int st = latent_block(n, blk, am1, hcache, E, W_lat, L, Wg, Wu, Wd, lat_out, B, V, D, R, H,
                                  do_mlp != 0, u_out, x, u, ubd, m);
            if (st != ORC_OK) {
#pragma omp critical
                status = st;
            }
        }
        free(x);
        free(u);
        free(ubd);
        free(m);
    }
    return status;
}

/* The in-kernel MLP schedule. */
int orc_latent(const int64_t* blk, const int64_t* am1, const uint16_t* hcache, const uint16_t* E,
               const uint16_t* W_lat, const float* L, const uint16_t* Wg, const uint16_t* Wu,
               const uint16_t* Wd, uint16_t* lat_out, int64_t N, int64_t B, int64_t V, int64_t D,
               int64_t R, int64_t H, double* u_out, int64_t n_lo, int64_t n_hi) {
    return orc_latent_ex(blk, am1, hcache, E, W_lat, L, Wg, Wu, Wd, lat_out, N, B, V, D, R, H, 1, u_out, n_lo,
                         n_hi);
}

/* ------------------------------------------------------------------------ */
/* readout: bias[r, v] = bf16(sum_k lat[r,k] * W2[k,v]), never stored by the */
/* fused pass; here computed per row.                                        */
/* ------------------------------------------------------------------------ */

#define VCHUNK 2048

/* The logits of one row, s[v] = bf16(base[v] + bf16(lat . W2[:, v])), as
 * doubles.  Parallel over vocab chunks. */
int orc_row_logits(const uint16_t* lat_row, const uint16_t* W2, const uint16_t* base_row, int64_t R,
                   int64_t V, double* s_out) {
    if (!lat_row || !W2 || !base_row || !s_out || R < 1 || V < 1) return ORC_ERR_ARG;
    int64_t nchunks = (V + VCHUNK - 1) / VCHUNK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t c = 0; c < nchunks; ++c) {
        double acc[VCHUNK];
        int64_t v0 = c * VCHUNK, w = (V - v0 < VCHUNK) ? V - v0 : VCHUNK;
        for (int64_t i = 0; i < w; ++i) acc[i] = 0.0;
        for (int64_t k = 0; k < R; ++k) {
            double a = bf(lat_row[k]);
            const uint16_t* wk = W2 + k * V + v0;
            for (int64_t i = 0; i < w; ++i) acc[i] += a * bf(wk[i]);
        }
        for (int64_t i = 0; i < w; ++i)
            s_out[v0 + i] = bf(bf16_add(base_row[v0 + i], bf16_from_double(acc[i])));
    }
    return ORC_OK;
}

/* bias = bf16(lat @ W2) for rows x V, written as bf16 bits. */
int orc_readout_bias(const uint16_t* lat, const uint16_t* W2, int64_t rows, int64_t R, int64_t V,
                     uint16_t* bias_out) {
    if (!lat || !W2 || !bias_out || rows < 1 || R < 1 || V < 1) return ORC_ERR_ARG;
    int64_t nchunks = (V + VCHUNK - 1) / VCHUNK;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < nchunks; ++c) {
            double acc[VCHUNK];
            int64_t v0 = c * VCHUNK, w = (V - v0 < VCHUNK) ? V - v0 : VCHUNK;
            for (int64_t i = 0; i < w; ++i) acc[i] = 0.0;
            for (int64_t k = 0; k < R; ++k) {
                double a = bf(lat[r * R + k]);
                const uint16_t* wk = W2 + k * V + v0;
                for (int64_t i = 0; i < w; ++i) acc[i] += a * bf(wk[i]);
            }
            for (int64_t i = 0; i < w; ++i) bias_out[r * V + v0 + i] = bf16_from_double(acc[i]);
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* one Jacobi pass: latent -> readout -> add-argmax into blk (in place).    */
/* *changed (nullable) receives the number of slots whose token changed.    */
/* ------------------------------------------------------------------------ */

int orc_jacobi_pass_ex(int64_t* blk, const int64_t* am1, const uint16_t* hcache, const uint16_t* E,
                       const uint16_t* W_lat, const float* L, const uint16_t* Wg, const uint16_t* Wu,
                       const uint16_t* Wd, const uint16_t* W2, const uint16_t* base, int64_t ld_base,
                       int64_t N, int64_t B, int64_t V, int64_t D, int64_t R, int64_t H, int64_t do_mlp,
                       int64_t* changed) {
    if (!blk || !W2 || !base || ld_base < V) return ORC_ERR_ARG;
    int64_t rows = N * (B - 1);
    if (!all_finite_bf16(base, rows, V, ld_base)) return ORC_ERR_NONFINITE;
    uint16_t* lat = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(rows * R));
    uint16_t* bias = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(rows * V));
    int64_t* fresh = (int64_t*)malloc(sizeof(int64_t) * (size_t)rows);
    if (!lat || !bias || !fresh) {
        free(lat);
        free(bias);
        free(fresh);
        return ORC_ERR_ARG;
    }
    int st = orc_latent_ex(blk, am1, hcache, E, W_lat, L, Wg, Wu, Wd, lat, N, B, V, D, R, H, do_mlp, NULL, 0, N);
    if (st == ORC_OK) st = orc_readout_bias(lat, W2, rows, R, V, bias);
    if (st == ORC_OK) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t r = 0; r < rows; ++r) fresh[r] = row_argmax(base + r * ld_base, bias + r * V, V, NULL);
        int64_t nchanged = 0;
        for (int64_t r = 0; r < rows; ++r) {
            int64_t n = r / (B - 1), b = r % (B - 1);
            if (blk[n * B + 1 + b] != fresh[r]) ++nchanged;
            blk[n * B + 1 + b] = fresh[r];
        }
        if (changed) *changed = nchanged;
    }
    free(lat);
    free(bias);
    free(fresh);
    return st;
}

int orc_jacobi_pass(int64_t* blk, const int64_t* am1, const uint16_t* hcache, const uint16_t* E,
                    const uint16_t* W_lat, const float* L, const uint16_t* Wg, const uint16_t* Wu,
                    const uint16_t* Wd, const uint16_t* W2, const uint16_t* base, int64_t ld_base,
                    int64_t N, int64_t B, int64_t V, int64_t D, int64_t R, int64_t H, int64_t* changed) {
    return orc_jacobi_pass_ex(blk, am1, hcache, E, W_lat, L, Wg, Wu, Wd, W2, base, ld_base, N, B, V, D, R, H, 1,
                              changed);
}
