/*
 * Exhaustive checks of the oracle's bf16 rounding (loaded with dlopen):
 *   1. for every 32-bit pattern f, the bit-pattern rounding
 *      orc_bf16_from_float_array(f) equals the value-arithmetic rounding
 *      orc_bf16_from_double_array((double)f) (NaNs: both must be NaN);
 *   2. for every pair of finite bf16 values (a, b), rounding the fp32 sum
 *      (what a GPU does with an fp32 add and a round-to-nearest-even convert)
 *      equals orc_bf16_add(a, b), the correctly rounded sum.
 * Prints "OK <counts>" or the first mismatches, exit status 0 on success.
 */
#include <dlfcn.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

typedef void (*f2b_t)(const float*, uint16_t*, int64_t);
typedef void (*d2b_t)(const double*, uint16_t*, int64_t);
typedef uint16_t (*add_t)(uint16_t, uint16_t);

static int is_nan_bits16(uint16_t h) { return (h & 0x7f80u) == 0x7f80u && (h & 0x7fu) != 0; }

int main(int argc, char** argv) {
    if (argc < 2) return 2;
    void* h = dlopen(argv[1], RTLD_NOW);
    if (!h) { fprintf(stderr, "dlopen: %s\n", dlerror()); return 2; }
    f2b_t f2b = (f2b_t)dlsym(h, "orc_bf16_from_float_array");
    d2b_t d2b = (d2b_t)dlsym(h, "orc_bf16_from_double_array");
    add_t add = (add_t)dlsym(h, "orc_bf16_add");
    if (!f2b || !d2b || !add) return 2;
    const int64_t CH = 1 << 20;
    long long bad1 = 0, bad2 = 0, n2 = 0;
#pragma omp parallel reduction(+ : bad1)
    {
        float* f = malloc(sizeof(float) * CH);
        double* d = malloc(sizeof(double) * CH);
        uint16_t* o1 = malloc(2 * CH);
        uint16_t* o2 = malloc(2 * CH);
#pragma omp for schedule(dynamic, 16)
        for (int64_t c = 0; c < (1LL << 32) / CH; ++c) {
            for (int64_t i = 0; i < CH; ++i) {
                uint32_t u = (uint32_t)(c * CH + i);
                memcpy(&f[i], &u, 4);
                d[i] = (double)f[i];
            }
            f2b(f, o1, CH);
            d2b(d, o2, CH);
            for (int64_t i = 0; i < CH; ++i) {
                int ok = is_nan_bits16(o1[i]) ? is_nan_bits16(o2[i]) : (o1[i] == o2[i]);
                if (!ok) {
                    if (bad1 < 5) {
                        uint32_t u; memcpy(&u, &f[i], 4);
#pragma omp critical
                        fprintf(stderr, "round mismatch f=%08x bits=%04x arith=%04x\n", u, o1[i], o2[i]);
                    }
                    ++bad1;
                }
            }
        }
        free(f); free(d); free(o1); free(o2);
    }
#pragma omp parallel for reduction(+ : bad2, n2) schedule(dynamic, 64)
    for (int a = 0; a < 65536; ++a) {
        if (((uint16_t)a & 0x7f80u) == 0x7f80u) continue;
        float fa; uint32_t ua = (uint32_t)a << 16; memcpy(&fa, &ua, 4);
        for (int b = 0; b < 65536; ++b) {
            if (((uint16_t)b & 0x7f80u) == 0x7f80u) continue;
            float fb; uint32_t ub = (uint32_t)b << 16; memcpy(&fb, &ub, 4);
            float s = fa + fb;
            uint16_t viaf;
            f2b(&s, &viaf, 1);
            uint16_t exact = add((uint16_t)a, (uint16_t)b);
            ++n2;
            if (viaf != exact) {
                if (bad2 < 5) {
#pragma omp critical
                    fprintf(stderr, "add mismatch a=%04x b=%04x f32=%04x exact=%04x\n", a, b, viaf, exact);
                }
                ++bad2;
            }
        }
    }
    if (bad1 || bad2) { printf("FAIL %lld %lld\n", bad1, bad2); return 1; }
    printf("OK %lld %lld\n", 1LL << 32, n2);
    return 0;
}
