/*
 * round_check.c -- exhaustive pin of the oracle's binary32 -> bf16 rounding.
 *
 * For every binary32 pattern in [start, end) it derives the expected bf16
 * result a second, independent way -- by comparing the exact distances from
 * the value to its two bf16 neighbours (computed in binary64, where both
 * differences are exact) -- and compares it with orc_f32_to_bf16.
 * IEEE-754 roundTiesToEven: the nearer neighbour wins; on a tie the one with
 * an even last mantissa bit; a magnitude at or beyond the midpoint between the
 * largest finite bf16 and 2^128 rounds to infinity.  NaN -> 0x7FC0.
 *
 * Usage: round_check START END   (hex or decimal, END exclusive, <= 2^32)
 * Prints "mismatches=<k> first=<pattern>" and exits 0 iff k == 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

uint16_t orc_f32_to_bf16(float f);

static float as_float(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

static uint16_t expected(uint32_t u)
{
    float f = as_float(u);
    if (isnan(f))
        return 0x7FC0u;
    uint32_t lo_u = u & 0xFFFF0000u;         /* neighbour toward zero */
    if (lo_u == u)
        return (uint16_t)(u >> 16);
    uint32_t hi_u = lo_u + 0x10000u;          /* neighbour away from zero */
    double x = (double)f;
    double lo = (double)as_float(lo_u);
    double hi;
    if ((hi_u & 0x7F800000u) == 0x7F800000u)  /* past the largest finite */
        hi = (u >> 31) ? -ldexp(1.0, 128) : ldexp(1.0, 128);
    else
        hi = (double)as_float(hi_u);
    double dlo = fabs(x - lo), dhi = fabs(hi - x);
    if (dlo < dhi)
        return (uint16_t)(lo_u >> 16);
    if (dhi < dlo)
        return (uint16_t)(hi_u >> 16);
    return ((lo_u >> 16) & 1u) ? (uint16_t)(hi_u >> 16) : (uint16_t)(lo_u >> 16);
}

int main(int argc, char **argv)
{
    if (argc != 3)
        return 2;
    uint64_t start = strtoull(argv[1], NULL, 0), end = strtoull(argv[2], NULL, 0);
    uint64_t bad = 0, first = 0;
    for (uint64_t v = start; v < end; ++v) {
        uint32_t u = (uint32_t)v;
        if (orc_f32_to_bf16(as_float(u)) != expected(u)) {
            if (bad == 0)
                first = v;
            ++bad;
        }
    }
    printf("mismatches=%llu first=0x%08llx\n", (unsigned long long)bad,
           (unsigned long long)first);
    return bad == 0 ? 0 : 1;
}
