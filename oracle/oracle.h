/*
 * oracle.h -- plain, slow, single-threaded CPU oracle for the collective
 * datapath (staging as self-synchronizing LL lines, validation, fixed
 * rank-order reduction, layout-derived copies).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link
 * or call this code: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA path (collective_datapath_gb300/csrc), and neither side includes
 * the other.
 *
 * Every function states the plain definition it computes and the passage of
 * the pages it follows:
 *   [Purlin]  "Purlin: Separating Orchestration from the Datapath of
 *             Collectives"
 *   [flash]   "flash-comm: Self-Synchronizing Collective Communication for
 *             LLM Decoding"
 *   [SiFAR]   "SiFAR: Synchronization-Free All-Reduce for Low-Latency LLM
 *             Inference"
 *
 * Data: bf16 values are carried as their raw 16-bit patterns (uint16_t).
 * Arithmetic is IEEE-754 binary32 with round-to-nearest-even; the file must
 * be compiled without fast-math and without FMA contraction (only additions
 * occur, so contraction cannot change a result, but the flag is set anyway).
 *
 * Parity pins: every function here is pinned by tests/test_oracle_*.py
 * against values fixed by the pages or by mathematics (closed forms,
 * exhaustive checks, brute force with exact rational arithmetic, the worked
 * layout example of [Purlin] Figure 4).  None is "parity unpinned".
 */
#ifndef COLL_ORACLE_H
#define COLL_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- scalar arithmetic ------------------------------------------------ */

/* bf16 -> binary32 widening: the bf16 pattern is the high half of the
 * binary32 pattern, so the conversion is exact.  [Purlin] §3.3 "convert each
 * x_p[i] from type E to FP32". */
float orc_bf16_to_f32(uint16_t b);

/* binary32 -> bf16, roundTiesToEven on the 16 discarded bits (IEEE-754
 * §4.3.1).  Overflow rounds to +-Inf, subnormals are kept (no flush to
 * zero), any NaN becomes the quiet NaN 0x7FC0.  [Purlin] §3.3 "convert y[i]
 * to E after the sum completes" (one rounding). */
uint16_t orc_f32_to_bf16(float f);

/* Fixed-order fold of n contributions at index i, then one rounding:
 *   acc = f32(x_0[i]); for p = 1..n-1: acc = acc + f32(x_p[i]);
 *   return bf16(acc).
 * [Purlin] §3.3 Eq. (2) (ascending rank order, fp32 accumulate, convert
 * once) and [flash] §3.3 (every replica folds rank 0 through N-1).
 * Reading of the pages: the sum starts from rank 0's value rather than from
 * +0.0; the two differ only when x_0[i] is -0.0 (see orc_fold_zero_start). */
uint16_t orc_fold(const uint16_t *const *x, int n, size_t i);

/* The literal "start from zero" form of Eq. (2): acc = +0.0, then add ranks
 * 0..n-1.  Kept only to show that it differs from orc_fold solely on -0.0. */
uint16_t orc_fold_zero_start(const uint16_t *const *x, int n, size_t i);

/* ---- partition geometry ----------------------------------------------- */

/* Shard (partition) geometry of a scattered buffer of `count` elements over
 * n ranks.  [Purlin] §3.1: a scattered buffer holds contiguous partitions
 * indexed by rank.  The pages use equal partitions; for a count that does
 * not split evenly they are silent.  Reading: every partition holds
 *   M = roundup(ceil(count / n), 8)
 * elements (8 bf16 = 16 bytes, the admission alignment of [flash] §4.1),
 * partition r covers [r*M, min(count, (r+1)*M)), so trailing partitions may
 * be shorter or empty.  When 8n divides count this is count/n. */
size_t orc_shard_elems(size_t count, int n);
size_t orc_shard_begin(size_t count, int n, int r);
size_t orc_shard_len(size_t count, int n, int r);

/* ---- collectives (plain definitions) ---------------------------------- */
/* All return 0 on success, -1 on invalid arguments.  `count` is always the
 * element count of the SCATTERED buffer of the collective (AR: input and
 * output; RS: input; AG: output; A2A: input and output), the per-rank
 * message size convention of [Purlin] §5 "Microbenchmarks". */

/* All-reduce: out_d[i] = orc_fold(in, n, i) for every rank d.
 * [Purlin] §2.1 (AllReduce leaves the complete reduced result at every
 * rank), §3.3 Eq. (2); [flash] §3.3. */
int orc_allreduce(int n, size_t count, const uint16_t *const *in,
                  uint16_t *const *out);

/* Reduce-scatter: out_r[j] = orc_fold over p of in_p[begin(r) + j],
 * j < len(r).  [Purlin] §2.1 (rank r receives the r-th reduced slice),
 * §3.1 Figure 4 top (scattered -> packed). */
int orc_reduce_scatter(int n, size_t count, const uint16_t *const *in,
                       uint16_t *const *out);

/* All-gather: out_d[begin(p) + j] = in_p[j], j < len(p).  [Purlin] §2.1
 * (concatenation in rank order), §3.1 Figure 4 (packed -> scattered). */
int orc_all_gather(int n, size_t count, const uint16_t *const *in,
                   uint16_t *const *out);

/* All-to-all: out_d[p*M + j] = in_p[d*M + j], j < M = count / n.  The
 * exchange needs equal partitions; a count that does not split into n equal
 * partitions of a multiple of 8 elements returns -1.  [Purlin] §2.1 (rank r
 * gets the r-th partition of every participant), §3.1 "transposed" layout
 * and Figure 4 bottom. */
int orc_all_to_all(int n, size_t count, const uint16_t *const *in,
                   uint16_t *const *out);

/* Variable-length (V) collectives ([Purlin] §3.1: the V variants keep the
 * layouts' relations but take partition sizes at runtime; §2.1 contracts).
 * len[] are element counts; offsets are their prefix sums.
 * RSV: every rank holds sum(len) elements partitioned by len;
 *      out_r[j] = fold over p of in_p[off_r + j], j < len[r].
 * AGV: rank p contributes len[p] elements; out_d = in_0 | in_1 | ... in rank
 *      order (sum(len) elements).
 * A2AV: len[p*n + d] = elements source p sends to destination d; source p's
 *      buffer holds its partitions in destination order; out_d = partition d
 *      of source 0 | of source 1 | ... in source-rank order. */
int orc_reduce_scatter_v(int n, const size_t *len, const uint16_t *const *in,
                         uint16_t *const *out);
int orc_all_gather_v(int n, const size_t *len, const uint16_t *const *in,
                     uint16_t *const *out);
int orc_all_to_all_v(int n, const size_t *len, const uint16_t *const *in,
                     uint16_t *const *out);

/* Twoshot all-reduce written as the composition of [Purlin] §3.1
 * "Composing transformations": reduce-scatter into a packed intermediate,
 * then all-gather of that intermediate.  `tmp` holds n intermediates of
 * orc_shard_elems(count, n) elements each. */
int orc_allreduce_composed(int n, size_t count, const uint16_t *const *in,
                           uint16_t *const *out, uint16_t *const *tmp);

/* MoE dispatch all-to-all (scatteredV -> transposedV copy).  Source rank p
 * holds `tokens` rows of `hidden` bf16 and topk_p[t*k + j] = expert of its
 * j-th choice for token t (experts 0..experts-1, distinct per token).
 * Expert e lives on destination d = e / (experts/n) as local expert
 * le = e % (experts/n).
 * counts[(d*EL + le)*n + p] = number of tokens of source p routed to expert
 * d*EL + le  (EL = experts / n).
 * Output rows of destination d are ordered by (le ascending, p ascending,
 * t ascending): out_d[row] = in_p[t] (hidden elements).
 * out_rows[d] = total rows at destination d.  out may be NULL (counts only);
 * otherwise out[d] must hold tokens * n * min(k, EL) rows of `hidden`.
 * [Purlin] §3.1 (transposed layout: source-rank order within a
 * destination; V variants take sizes at runtime), §2.1 Table 2 (expert
 * parallel dispatch).  The order within a destination (expert, then source
 * rank, then token) is a reading: the pages fix only source-rank order. */
int orc_moe_dispatch(int n, int tokens, int hidden, int k, int experts,
                     const int32_t *const *topk, const uint16_t *const *in,
                     uint16_t *const *out, int32_t *counts, int64_t *out_rows);

/* Source of every output row of destination d under the same definition as
 * orc_moe_dispatch: src_rank[row], src_token[row] for row < rows (the
 * return value), in the (local expert, source rank, token) order.  Lets a
 * test check a full-size dispatch row by row without materialising it.
 * Returns -1 on invalid arguments. */
int64_t orc_moe_row_sources(int n, int tokens, int k, int experts,
                            const int32_t *const *topk, int d, int32_t *src_rank,
                            int32_t *src_token);

/* ---- readiness encodings ---------------------------------------------- */
/* LL8 line (8 bytes, a little-endian uint64):
 *   bits  0..15 = element 2j, bits 16..31 = element 2j+1 (0 past the end),
 *   bits 32..63 = (uint32) epoch.
 * [Purlin] §3.2 "Specializing for latency" (payload packed with a flag that
 * carries the epoch, §4.2), [flash] §4.3 (a 16-byte unit carries 8 payload
 * bytes and two copies of the sequence number: two LL8 lines side by side).
 * Byte order within the line is a reading (the pages do not fix it). */
size_t orc_ll8_lines(size_t elems);
void orc_ll8_encode(const uint16_t *in, size_t elems, uint64_t epoch,
                    uint64_t *lines);
/* Decode lines whose flag equals (uint32) epoch; a line with another flag is
 * stale and is rejected (its payload is not written).  Returns the number of
 * rejected lines.  [flash] §3.1 (accept only data carrying the current
 * call's evidence). */
size_t orc_ll8_decode(const uint64_t *lines, size_t elems, uint64_t epoch,
                      uint16_t *out);

/* LL128 line (128 bytes): bytes 0..119 hold elements 60j..60j+59 as
 * little-endian uint16 (0 past the end), bytes 120..127 hold the epoch as a
 * little-endian uint64 sequence number.  [flash] §3.1 "Sequence-number
 * readiness" (data and the call's sequence number in one transfer unit,
 * accepted only when the number matches); the 120+8 split is the 128-byte
 * line of the workload; the position of the number is a reading. */
size_t orc_ll128_lines(size_t elems);
void orc_ll128_encode(const uint16_t *in, size_t elems, uint64_t epoch,
                      uint8_t *lines);
size_t orc_ll128_decode(const uint8_t *lines, size_t elems, uint64_t epoch,
                        uint16_t *out);

/* Sentinel readiness: [flash] §3.1 "Sentinel readiness".  Receive storage is
 * pre-filled with a reserved bit pattern; a producer publishes a pack by
 * overwriting it, so a pack that differs from the sentinel has arrived, and
 * no flag travels with the payload.  A value that equals the reserved
 * pattern is replaced by the canonical quiet NaN before publication, so it
 * can never look unready.
 * Readings (the pages fix neither): the reserved bf16 pattern is 0xFFFF (a
 * NaN, so only a NaN input changes, and it stays a NaN); the canonical
 * quiet NaN is 0x7FC0 (the NaN the fold's rounding produces); a pack is 8
 * bytes = 4 elements, little-endian (element 4j in bits 0..15), 0 past the
 * end; the sentinel pack is all ones (four sentinel elements). */
#define ORC_SENT_BF16 0xFFFFu
#define ORC_CANONICAL_NAN 0x7FC0u
uint16_t orc_sent_sanitize(uint16_t x);
void orc_sent_sanitize_buf(const uint16_t *in, size_t elems, uint16_t *out);
size_t orc_sent_packs(size_t elems);
void orc_sent_encode(const uint16_t *in, size_t elems, uint64_t *packs);
/* Decode packs that are not the sentinel pack; a sentinel pack has not
 * arrived and is skipped (its elements are not written).  Returns the number
 * of packs skipped. */
size_t orc_sent_decode(const uint64_t *packs, size_t elems, uint16_t *out);

/* ---- fp32 tensors -------------------------------------------------------
 * [flash] §4.1 admits bf16 and fp32 tensors.  For fp32 the fold is the same
 * left fold in rank order, in binary32 with round-to-nearest-even, and there
 * is no final narrowing: acc = x_0; acc = acc + x_p for p = 1..N-1.
 * Readings: elements are uint32 bit patterns; a NaN result is written as the
 * canonical quiet NaN 0x7FC00000 (the pages fix no NaN payload; this is the
 * binary32 counterpart of the bf16 rule, whose 0x7FC0 is its upper half).
 * Partitions are counted in fp32 elements with the same rule as bf16.
 * Copies (all-gather, all-to-all and their V forms) move bytes and need no
 * fp32 form: they are the bf16 ones on the same bytes. */
uint32_t orc_fold_f32(const uint32_t *const *x, int n, size_t i);
int orc_allreduce_f32(int n, size_t count, const uint32_t *const *in,
                      uint32_t *const *out);
int orc_reduce_scatter_f32(int n, size_t count, const uint32_t *const *in,
                           uint32_t *const *out);

/* Sentinel packs of fp32: 8 bytes = 2 elements (element 2j in the low
 * word), the reserved pattern 0xFFFFFFFF (a NaN), published as 0x7FC00000;
 * the unready pack is all ones. */
uint32_t orc_sent_sanitize_f32(uint32_t x);
void orc_sent_encode_f32(const uint32_t *in, size_t elems, uint64_t *packs);
size_t orc_sent_decode_f32(const uint64_t *packs, size_t elems, uint32_t *out);

/* One-sided copy -- Purlin §3.3 (Atom::copy): dst[i] = src[i] for every
 * byte i < bytes.  Pipeline depth, stage size and CTA count change how the
 * bytes move, never which bytes arrive, so none of them is a parameter. */
void orc_one_sided_copy(const uint8_t *src, size_t bytes, uint8_t *dst);

#ifdef __cplusplus
}
#endif
#endif /* COLL_ORACLE_H */
