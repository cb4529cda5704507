/*
 * oracle.c -- plain CPU oracle for the collective datapath.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h): used by the tests, the smoke check
 * and the benchmark's CPU-baseline leg, never by the product path.  Plain
 * loops, one element at a time, no blocking, no fusion, no reordering.
 *
 * Build: gcc -std=c99 -O2 -fPIC -shared -ffp-contract=off -fno-fast-math
 */
#include "oracle.h"

#include <string.h>

/* ---- scalar arithmetic ------------------------------------------------ */

float orc_bf16_to_f32(uint16_t b)
{
    /* The bf16 pattern is the top 16 bits of a binary32 pattern. */
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t exponent = (u >> 23) & 0xFFu;
    uint32_t mantissa = u & 0x7FFFFFu;
    if (exponent == 0xFFu && mantissa != 0u)
        return (uint16_t)0x7FC0u; /* any NaN -> the quiet NaN */
    /* Keep the high 16 bits; look at the 16 discarded ones.  Above half an
     * ulp of the kept part rounds away from zero, below rounds toward zero,
     * exactly half rounds to the neighbour whose last kept bit is 0.  A carry
     * out of the kept mantissa moves into the exponent, which is exactly the
     * next representable magnitude (or +-Inf past the largest finite). */
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u) != 0u))
        kept += 1u;
    return (uint16_t)kept;
}

uint16_t orc_fold(const uint16_t *const *x, int n, size_t i)
{
    float acc = orc_bf16_to_f32(x[0][i]);
    for (int p = 1; p < n; ++p)
        acc = acc + orc_bf16_to_f32(x[p][i]);
    return orc_f32_to_bf16(acc);
}

uint16_t orc_fold_zero_start(const uint16_t *const *x, int n, size_t i)
{
    float acc = 0.0f;
    for (int p = 0; p < n; ++p)
        acc = acc + orc_bf16_to_f32(x[p][i]);
    return orc_f32_to_bf16(acc);
}

/* ---- partition geometry ----------------------------------------------- */

size_t orc_shard_elems(size_t count, int n)
{
    if (n <= 0)
        return 0;
    size_t per = (count + (size_t)n - 1) / (size_t)n; /* ceil(count / n) */
    return (per + 7u) / 8u * 8u;                       /* round up to 8 */
}

size_t orc_shard_begin(size_t count, int n, int r)
{
    size_t m = orc_shard_elems(count, n);
    size_t b = (size_t)r * m;
    return b < count ? b : count;
}

size_t orc_shard_len(size_t count, int n, int r)
{
    size_t m = orc_shard_elems(count, n);
    size_t b = orc_shard_begin(count, n, r);
    size_t e = b + m;
    if (e > count)
        e = count;
    return e - b;
}

/* ---- collectives ------------------------------------------------------ */

static int bad_args(int n, const void *in, const void *out)
{
    return n < 1 || in == NULL || out == NULL;
}

int orc_allreduce(int n, size_t count, const uint16_t *const *in,
                  uint16_t *const *out)
{
    if (bad_args(n, in, out))
        return -1;
    for (int d = 0; d < n; ++d)
        for (size_t i = 0; i < count; ++i)
            out[d][i] = orc_fold(in, n, i);
    return 0;
}

int orc_reduce_scatter(int n, size_t count, const uint16_t *const *in,
                       uint16_t *const *out)
{
    if (bad_args(n, in, out))
        return -1;
    for (int r = 0; r < n; ++r) {
        size_t b = orc_shard_begin(count, n, r);
        size_t len = orc_shard_len(count, n, r);
        for (size_t j = 0; j < len; ++j)
            out[r][j] = orc_fold(in, n, b + j);
    }
    return 0;
}

int orc_all_gather(int n, size_t count, const uint16_t *const *in,
                   uint16_t *const *out)
{
    if (bad_args(n, in, out))
        return -1;
    for (int d = 0; d < n; ++d)
        for (int p = 0; p < n; ++p) {
            size_t b = orc_shard_begin(count, n, p);
            size_t len = orc_shard_len(count, n, p);
            for (size_t j = 0; j < len; ++j)
                out[d][b + j] = in[p][j];
        }
    return 0;
}

int orc_all_to_all(int n, size_t count, const uint16_t *const *in,
                   uint16_t *const *out)
{
    if (bad_args(n, in, out))
        return -1;
    /* The exchange needs equal partitions: partition d of source p lands in
     * slot p of destination d, so all slots must have one length. */
    size_t m = orc_shard_elems(count, n);
    if (m * (size_t)n != count)
        return -1;
    for (int d = 0; d < n; ++d)
        for (int p = 0; p < n; ++p)
            for (size_t j = 0; j < m; ++j)
                out[d][(size_t)p * m + j] = in[p][(size_t)d * m + j];
    return 0;
}

int orc_reduce_scatter_v(int n, const size_t *len, const uint16_t *const *in,
                         uint16_t *const *out)
{
    if (bad_args(n, in, out) || len == NULL)
        return -1;
    size_t off = 0;
    for (int r = 0; r < n; ++r) {
        for (size_t j = 0; j < len[r]; ++j)
            out[r][j] = orc_fold(in, n, off + j);
        off += len[r];
    }
    return 0;
}

int orc_all_gather_v(int n, const size_t *len, const uint16_t *const *in,
                     uint16_t *const *out)
{
    if (bad_args(n, in, out) || len == NULL)
        return -1;
    for (int d = 0; d < n; ++d) {
        size_t off = 0;
        for (int p = 0; p < n; ++p) {
            for (size_t j = 0; j < len[p]; ++j)
                out[d][off + j] = in[p][j];
            off += len[p];
        }
    }
    return 0;
}

int orc_all_to_all_v(int n, const size_t *len, const uint16_t *const *in,
                     uint16_t *const *out)
{
    if (bad_args(n, in, out) || len == NULL)
        return -1;
    for (int d = 0; d < n; ++d) {
        size_t dst = 0;
        for (int p = 0; p < n; ++p) {
            size_t src = 0;
            for (int k = 0; k < d; ++k)
                src += len[(size_t)p * n + k];
            for (size_t j = 0; j < len[(size_t)p * n + d]; ++j)
                out[d][dst + j] = in[p][src + j];
            dst += len[(size_t)p * n + d];
        }
    }
    return 0;
}

int orc_allreduce_composed(int n, size_t count, const uint16_t *const *in,
                           uint16_t *const *out, uint16_t *const *tmp)
{
    if (bad_args(n, in, out) || tmp == NULL)
        return -1;
    if (orc_reduce_scatter(n, count, in, tmp) != 0)
        return -1;
    return orc_all_gather(n, count, (const uint16_t *const *)tmp, out);
}

int orc_moe_dispatch(int n, int tokens, int hidden, int k, int experts,
                     const int32_t *const *topk, const uint16_t *const *in,
                     uint16_t *const *out, int32_t *counts, int64_t *out_rows)
{
    if (n < 1 || tokens < 0 || hidden < 0 || k < 0 || experts < n ||
        experts % n != 0 || topk == NULL || in == NULL || counts == NULL ||
        out_rows == NULL)
        return -1;
    int el = experts / n;
    for (int i = 0; i < experts * n; ++i)
        counts[i] = 0;
    for (int p = 0; p < n; ++p)
        for (int t = 0; t < tokens; ++t)
            for (int j = 0; j < k; ++j) {
                int e = topk[p][(size_t)t * (size_t)k + (size_t)j];
                if (e < 0 || e >= experts)
                    return -1;
                counts[e * n + p] += 1; /* e*n + p == (d*EL + le)*n + p */
            }
    for (int d = 0; d < n; ++d) {
        int64_t row = 0;
        for (int le = 0; le < el; ++le) {
            int e = d * el + le;
            for (int p = 0; p < n; ++p)
                for (int t = 0; t < tokens; ++t) {
                    int routed = 0;
                    for (int j = 0; j < k; ++j)
                        if (topk[p][(size_t)t * (size_t)k + (size_t)j] == e)
                            routed = 1;
                    if (!routed)
                        continue;
                    if (out != NULL && out[d] != NULL)
                        memcpy(out[d] + (size_t)row * (size_t)hidden,
                               in[p] + (size_t)t * (size_t)hidden,
                               (size_t)hidden * sizeof(uint16_t));
                    row += 1;
                }
        }
        out_rows[d] = row;
    }
    return 0;
}

int64_t orc_moe_row_sources(int n, int tokens, int k, int experts,
                            const int32_t *const *topk, int d, int32_t *src_rank,
                            int32_t *src_token)
{
    if (n < 1 || experts < n || experts % n != 0 || d < 0 || d >= n ||
        topk == NULL || src_rank == NULL || src_token == NULL)
        return -1;
    int el = experts / n;
    int64_t row = 0;
    for (int le = 0; le < el; ++le) {
        int e = d * el + le;
        for (int p = 0; p < n; ++p)
            for (int t = 0; t < tokens; ++t)
                for (int j = 0; j < k; ++j)
                    if (topk[p][(size_t)t * (size_t)k + (size_t)j] == e) {
                        src_rank[row] = p;
                        src_token[row] = t;
                        row += 1;
                    }
    }
    return row;
}

/* ---- readiness encodings ---------------------------------------------- */

size_t orc_ll8_lines(size_t elems) { return (elems + 1u) / 2u; }

void orc_ll8_encode(const uint16_t *in, size_t elems, uint64_t epoch,
                    uint64_t *lines)
{
    size_t nl = orc_ll8_lines(elems);
    for (size_t j = 0; j < nl; ++j) {
        uint64_t lo = in[2 * j];
        uint64_t hi = 2 * j + 1 < elems ? in[2 * j + 1] : 0u;
        uint64_t flag = (uint32_t)epoch;
        lines[j] = lo | (hi << 16) | (flag << 32);
    }
}

size_t orc_ll8_decode(const uint64_t *lines, size_t elems, uint64_t epoch,
                      uint16_t *out)
{
    size_t nl = orc_ll8_lines(elems);
    size_t rejected = 0;
    for (size_t j = 0; j < nl; ++j) {
        uint64_t line = lines[j];
        if ((uint32_t)(line >> 32) != (uint32_t)epoch) {
            rejected += 1;
            continue;
        }
        out[2 * j] = (uint16_t)(line & 0xFFFFu);
        if (2 * j + 1 < elems)
            out[2 * j + 1] = (uint16_t)((line >> 16) & 0xFFFFu);
    }
    return rejected;
}

size_t orc_ll128_lines(size_t elems) { return (elems + 59u) / 60u; }

void orc_ll128_encode(const uint16_t *in, size_t elems, uint64_t epoch,
                      uint8_t *lines)
{
    size_t nl = orc_ll128_lines(elems);
    for (size_t j = 0; j < nl; ++j) {
        uint8_t *line = lines + j * 128u;
        for (size_t q = 0; q < 60; ++q) {
            size_t idx = j * 60u + q;
            uint16_t v = idx < elems ? in[idx] : 0u;
            line[2 * q] = (uint8_t)(v & 0xFFu);
            line[2 * q + 1] = (uint8_t)(v >> 8);
        }
        for (int b = 0; b < 8; ++b)
            line[120 + b] = (uint8_t)((epoch >> (8 * b)) & 0xFFu);
    }
}

size_t orc_ll128_decode(const uint8_t *lines, size_t elems, uint64_t epoch,
                        uint16_t *out)
{
    size_t nl = orc_ll128_lines(elems);
    size_t rejected = 0;
    for (size_t j = 0; j < nl; ++j) {
        const uint8_t *line = lines + j * 128u;
        uint64_t seq = 0;
        for (int b = 0; b < 8; ++b)
            seq |= (uint64_t)line[120 + b] << (8 * b);
        if (seq != epoch) {
            rejected += 1;
            continue;
        }
        for (size_t q = 0; q < 60; ++q) {
            size_t idx = j * 60u + q;
            if (idx < elems)
                out[idx] = (uint16_t)(line[2 * q] | (line[2 * q + 1] << 8));
        }
    }
    return rejected;
}

uint16_t orc_sent_sanitize(uint16_t x)
{
    if (x == ORC_SENT_BF16)
        return (uint16_t)ORC_CANONICAL_NAN;
    return x;
}

void orc_sent_sanitize_buf(const uint16_t *in, size_t elems, uint16_t *out)
{
    for (size_t i = 0; i < elems; ++i)
        out[i] = orc_sent_sanitize(in[i]);
}

size_t orc_sent_packs(size_t elems) { return (elems + 3u) / 4u; }

void orc_sent_encode(const uint16_t *in, size_t elems, uint64_t *packs)
{
    size_t np = orc_sent_packs(elems);
    for (size_t j = 0; j < np; ++j) {
        uint64_t pack = 0;
        for (size_t q = 0; q < 4; ++q) {
            size_t idx = 4 * j + q;
            uint64_t v = idx < elems ? orc_sent_sanitize(in[idx]) : 0u;
            pack |= v << (16 * q);
        }
        packs[j] = pack;
    }
}

size_t orc_sent_decode(const uint64_t *packs, size_t elems, uint16_t *out)
{
    size_t np = orc_sent_packs(elems);
    size_t skipped = 0;
    for (size_t j = 0; j < np; ++j) {
        uint64_t pack = packs[j];
        if (pack == ~(uint64_t)0) {
            skipped += 1;
            continue;
        }
        for (size_t q = 0; q < 4; ++q) {
            size_t idx = 4 * j + q;
            if (idx < elems)
                out[idx] = (uint16_t)((pack >> (16 * q)) & 0xFFFFu);
        }
    }
    return skipped;
}

/* ---- fp32 tensors -------------------------------------------------------- */

static float f32_of(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t bits_of(float f)
{
    uint32_t u;
    if (f != f)
        return 0x7FC00000u; /* any NaN: the canonical quiet NaN */
    memcpy(&u, &f, sizeof u);
    return u;
}

uint32_t orc_fold_f32(const uint32_t *const *x, int n, size_t i)
{
    float acc = f32_of(x[0][i]);
    for (int p = 1; p < n; ++p)
        acc = acc + f32_of(x[p][i]);
    return bits_of(acc);
}

static int bad_args_f32(int n, const uint32_t *const *in, uint32_t *const *out)
{
    if (n < 1 || in == NULL || out == NULL)
        return 1;
    for (int p = 0; p < n; ++p)
        if (in[p] == NULL || out[p] == NULL)
            return 1;
    return 0;
}

int orc_allreduce_f32(int n, size_t count, const uint32_t *const *in,
                      uint32_t *const *out)
{
    if (bad_args_f32(n, in, out))
        return -1;
    for (int d = 0; d < n; ++d)
        for (size_t i = 0; i < count; ++i)
            out[d][i] = orc_fold_f32(in, n, i);
    return 0;
}

int orc_reduce_scatter_f32(int n, size_t count, const uint32_t *const *in,
                           uint32_t *const *out)
{
    if (bad_args_f32(n, in, out))
        return -1;
    for (int r = 0; r < n; ++r) {
        size_t b = orc_shard_begin(count, n, r);
        size_t len = orc_shard_len(count, n, r);
        for (size_t j = 0; j < len; ++j)
            out[r][j] = orc_fold_f32(in, n, b + j);
    }
    return 0;
}

uint32_t orc_sent_sanitize_f32(uint32_t x)
{
    if (x == 0xFFFFFFFFu)
        return 0x7FC00000u;
    return x;
}

void orc_sent_encode_f32(const uint32_t *in, size_t elems, uint64_t *packs)
{
    size_t np = (elems + 1u) / 2u;
    for (size_t j = 0; j < np; ++j) {
        uint64_t lo = orc_sent_sanitize_f32(in[2 * j]);
        uint64_t hi = 2 * j + 1 < elems ? orc_sent_sanitize_f32(in[2 * j + 1]) : 0u;
        packs[j] = lo | (hi << 32);
    }
}

size_t orc_sent_decode_f32(const uint64_t *packs, size_t elems, uint32_t *out)
{
    size_t np = (elems + 1u) / 2u;
    size_t skipped = 0;
    for (size_t j = 0; j < np; ++j) {
        uint64_t pack = packs[j];
        if (pack == 0xFFFFFFFFFFFFFFFFull) { /* not yet published */
            skipped += 1;
            continue;
        }
        out[2 * j] = (uint32_t)(pack & 0xFFFFFFFFu);
        if (2 * j + 1 < elems)
            out[2 * j + 1] = (uint32_t)(pack >> 32);
    }
    return skipped;
}

void orc_one_sided_copy(const uint8_t *src, size_t bytes, uint8_t *dst)
{
    for (size_t i = 0; i < bytes; ++i)
        dst[i] = src[i];
}
