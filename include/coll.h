/*
 * coll.h -- C ABI of the single-GPU collective datapath for GB300 (sm_103a).
 *
 * What it computes.  N emulated ranks live in one GPU's HBM.  Each rank's
 * bf16 buffer is staged as self-synchronizing lines that carry their own
 * readiness evidence (a flag or sequence word equal to the current epoch);
 * consumers poll the lines they need, reject stale ones, unpack them, and
 * either copy them into the output layout or fold the N contributions in
 * fixed rank order (fp32 accumulate, one rounding to bf16).  A collective is
 * named by (input layout, output layout, copy-or-reduce), as in
 *   "Purlin: Separating Orchestration from the Datapath of Collectives",
 *   §3.1 Listing 1 (collective declarations) and Figure 4;
 * staging and consumption follow its Stage-Notify-Consume protocol (§3.2,
 * Listing 2), with the notification carried inside the data as in its
 * latency path (§3.2 "Specializing for latency") and in
 *   "flash-comm: Self-Synchronizing Collective Communication for LLM
 *   Decoding", §3.1 (self-synchronizing transfers, sequence-number
 *   readiness), §3.3 (rank-order reduction), §4.2 (device-side call counter
 *   selects the buffer slot).
 *
 * Supported (in, out, op) triples and the meaning of `count` (always the
 * element count of the scattered buffer of the collective, the per-rank size
 * convention of Purlin §5 "Microbenchmarks"):
 *   (SCATTERED,   SCATTERED,   REDUCE)  all-reduce      in = out = count
 *   (SCATTERED,   PACKED,      REDUCE)  reduce-scatter  in = count, out = len(r)
 *   (PACKED,      SCATTERED,   COPY)    all-gather      in = len(p), out = count
 *   (SCATTERED,   TRANSPOSED,  COPY)    all-to-all      in = out = count
 *   (SCATTERED_V, PACKED_V,    REDUCE)  reduce-scatter V  in = count, out = vcounts[r]
 *   (PACKED_V,    SCATTERED_V, COPY)    all-gather V      in = vcounts[p], out = count
 *   (SCATTERED_V, TRANSPOSED_V,COPY)    all-to-all V      sizes from vcounts[p][d];
 *                                       MoE dispatch      when experts > 0 (rows
 *                                       routed by top-k)
 * V variants keep the layouts' relations with runtime sizes (Purlin §3.1).
 * Partition r of a scattered buffer covers [r*M, min(count, (r+1)*M)) with
 * M = roundup(ceil(count / nranks), 8) elements (equal partitions when
 * 8*nranks divides count).  Every other triple returns COLL_ERR_UNSUPPORTED.
 *
 * Ownership.  The caller owns every device buffer: inputs, outputs and the
 * workspace (obtain its size from coll_workspace_bytes, allocate it however
 * it likes, hand it over with coll_bind).  The library allocates no device
 * memory and frees nothing of the caller's.  A spec holds host state only;
 * it is not thread-safe and must be used from one stream at a time.
 *
 * Asynchrony.  coll_bind, coll_stage and coll_run only enqueue work on the
 * given stream (coll_set_routing records a pointer on the host).  coll_stage
 * and coll_run may be captured in a CUDA graph and replayed: the epoch that
 * selects the staging slot and the readiness value lives in the workspace,
 * on the device, and advances on the device.  coll_bind copies the spec's
 * work lists from host memory and is made once, outside any capture.
 *
 * Errors.  Host-side argument errors return a status immediately and enqueue
 * nothing.  Device-side errors (a wait that exceeded its time bound) are
 * latched in the workspace; coll_query_status reports and clears them.
 * Kernels never trap and never wait without a bound.
 *
 * Streams are passed as `coll_stream_t` (a cudaStream_t; NULL = the legacy
 * default stream).
 */
#ifndef COLL_H
#define COLL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define COLL_VERSION 1
#define COLL_MAX_RANKS 8

typedef void *coll_stream_t;

/* Layouts of Purlin §3.1: packed = one contiguous contribution; scattered =
 * rank-indexed contiguous partitions; transposed = partition r of every
 * source, in source-rank order.  _V variants take sizes at runtime. */
typedef enum {
    COLL_PACKED = 0,
    COLL_SCATTERED = 1,
    COLL_TRANSPOSED = 2,
    COLL_PACKED_V = 3,
    COLL_SCATTERED_V = 4,
    COLL_TRANSPOSED_V = 5
} coll_layout_t;

/* Consume operation of Purlin Listing 1: copy into distinct output regions,
 * or reduce corresponding elements. */
typedef enum { COLL_COPY = 0, COLL_REDUCE = 1 } coll_op_t;

typedef enum { COLL_BF16 = 0, COLL_F32 = 1 } coll_dtype_t;
/* COLL_F32 (flash-comm §4.1 admits bf16 and fp32 tensors): the fold is the
 * same left fold in rank order in binary32 with no final narrowing; a NaN
 * result is written as 0x7FC00000.  `count`, `vcounts` and the element
 * counts of coll_buffer_elems are fp32 elements; every count is still a
 * multiple of 8.  Lines carry the same bytes as for bf16 (an LL8 line one
 * fp32, an LL128 line 30, a sentinel pack 2, whose reserved pattern is
 * 0xFFFFFFFF, published as 0x7FC00000).  MoE dispatch copies fp32 rows
 * byte for byte (`hidden` fp32 elements per row, at most 24,576). */

typedef enum {
    COLL_OK = 0,
    COLL_ERR_INVALID = 1,     /* bad argument (null pointer, rank range...) */
    COLL_ERR_UNSUPPORTED = 2, /* triple, dtype, rank count or option */
    COLL_ERR_ALIGN = 3,       /* pointer or count not 16-byte aligned */
    COLL_ERR_NOMEM = 4,       /* bound workspace smaller than required */
    COLL_ERR_CUDA = 5,        /* a CUDA runtime call failed */
    COLL_ERR_TIMEOUT = 6,     /* a device wait exceeded its bound */
    COLL_ERR_STATE = 7        /* call out of sequence (e.g. run before bind) */
} coll_status_t;

/* Readiness encodings.
 * COLL_LL8: 8-byte line = 4 bytes of data (two bf16) + 4-byte flag = the
 *   epoch's low 32 bits; two lines per 16-byte store.  Purlin §3.2 packet,
 *   flash-comm §4.3 sequence-numbered packet.
 * COLL_LL128: 128-byte line = 120 bytes of data (60 bf16) + 8-byte sequence
 *   number = the epoch (bytes 120..127).  flash-comm §3.1 sequence-number
 *   readiness, at 128-byte granularity.
 * COLL_SENT: 8-byte pack = four bf16 and nothing else.  flash-comm §3.1
 *   sentinel readiness: staging holds the all-ones pattern until a producer
 *   overwrites it, so no byte beyond the payload moves.  An input element
 *   equal to 0xFFFF (a NaN) is delivered as the canonical quiet NaN 0x7FC0;
 *   all other bit patterns pass unchanged, and reductions are unaffected
 *   (NaN in, NaN out).  Consumed packs must be re-armed: any reset mode but
 *   COLL_RESET_NONE (which gets COLL_ERR_UNSUPPORTED). */
enum { COLL_LL8 = 0, COLL_LL128 = 1, COLL_SENT = 2, COLL_ENC_AUTO = 3 };
/* COLL_ENC_AUTO: for an all-reduce whose algorithm and path are AUTO too,
 * encoding, algorithm and path come from a policy table calibrated on GB300
 * per group size and bytes per rank (flash-comm §3.2 cost-guided selection,
 * §4.1 table lookup; the table is csrc/policy_table.h, written by tune.py).
 * Otherwise sentinel packs up to 1 MiB per rank (LL8 when the reset mode is
 * COLL_RESET_NONE) and LL128 lines above. */

/* All-reduce algorithm: oneshot (every rank folds all N inputs), twoshot
 * (reduce-scatter to an owner per partition, which publishes its reduced
 * partition, then all-gather).  Purlin §3.1 compose<reduceScatter,
 * allGather>; SiFAR §3.1; flash-comm §4.3 (one-hop / sharded two-hop). */
enum { COLL_ALGO_AUTO = 0, COLL_ONESHOT = 1, COLL_TWOSHOT = 2 };

/* Re-arm (LL8 and sentinel; LL128 sequence numbers need none, flash-comm
 * §3.1 Table 2): after every reader of a line consumed it, its LL8 flag word
 * is set back to 0, or a sentinel pack back to the pattern --
 *   FUSED:    by the last reader, counted per tile inside the consume kernel;
 *   KERNEL:   by a separate kernel at the end of the run;
 *   DEFERRED: (default) by the owning rank during the next epoch, in the slot
 *             that epoch does not use: the completed previous run is the
 *             evidence that every reader consumed it (the dual-buffering
 *             argument of SiFAR §3.3), so no counter or barrier is needed;
 *   NONE:     never (LL8 flags are epoch values, so a stale line never
 *             matches; not allowed with COLL_SENT).
 */
enum { COLL_RESET_FUSED = 0, COLL_RESET_KERNEL = 1, COLL_RESET_NONE = 2,
       COLL_RESET_DEFERRED = 3 };

/* Launch path: FUSED = stage and consume inside one cooperative kernel
 * (all CTAs co-resident; a CTA serves one emulated rank).  STREAMED =
 * separate stage and consume kernels ordered by the stream.  COMPOSED (LL128
 * only: the twoshot all-reduce, reduce-scatter, all-gather, all-to-all and
 * their V forms) = one cooperative launch by columns: a column is one chunk
 * of one partition, and one CTA runs its stage, fold (+ publish) and gather
 * or copy phases back to back, so the chunk's lines stay in L2 between
 * their producer and their reader and no CTA waits for another (Purlin
 * §3.2, Algorithm 1, Figure 5, with the chunk counter inside a CTA).  A
 * short run (fewer columns than co-resident CTAs) launches one CTA per
 * 16-line column; a longer one staggers each CTA's first column and ends
 * on 16-line columns.
 * Dependent launches: FUSED and COMPOSED runs up to 512 KiB per rank (input
 * or output, whichever is larger), STREAMED runs up to 128 KiB, carry
 * programmatic stream serialization, so their CTAs can be placed while the
 * previous kernel in the stream finishes; they wait for that kernel to
 * complete, with its writes visible, before reading the workspace or any
 * input (griddepcontrol.wait).  Each of the library's kernels allows the
 * next dependent launch to be placed once it has read the epoch; a caller's
 * kernel launched that way must wait the same way before it reads the
 * outputs.
 * AUTO picks FUSED for LL8 and sentinel packs up to 256 KiB per rank,
 * COMPOSED for LL128 (the all-to-all and all-to-all V from 4 MiB per rank),
 * STREAMED otherwise, and, for the all-reduce, ONESHOT up to 512 KiB per rank
 * (boundaries on measured GB300 points); with COLL_ENC_AUTO the all-reduce
 * takes the calibrated table. */
enum { COLL_PATH_AUTO = 0, COLL_PATH_FUSED = 1, COLL_PATH_STREAMED = 2,
       COLL_PATH_COMPOSED = 3 };

typedef struct {
    int encoding;        /* COLL_LL8 | COLL_LL128 | COLL_SENT | COLL_ENC_AUTO
                            (default LL8) */
    int algorithm;       /* COLL_ALGO_AUTO | COLL_ONESHOT | COLL_TWOSHOT */
    int reset_mode;      /* COLL_RESET_* (default DEFERRED) */
    int path;            /* COLL_PATH_* (default AUTO) */
    int ctas;            /* CTAs of the consume grid, 0 = auto */
    int tile_lines;      /* lines per work item, 0 = auto */
    uint64_t timeout_ns; /* bound on every device wait, 0 = 200 ms */
    /* MoE dispatch (SCATTERED_V -> TRANSPOSED_V) only: */
    int tokens;          /* rows per source rank */
    int hidden;          /* elements per row (of the dtype; a multiple of 8,
                            at most 49,152 bf16 or 24,576 fp32) */
    int topk;            /* experts per token */
    int experts;         /* total experts, a multiple of nranks (<= 1024) */
    int max_rows;        /* output rows each destination can hold, 0 = the
                            worst case tokens * nranks * min(topk, experts/nranks) */
    /* Variable-length collectives (V layouts, MoE dispatch excepted): element
     * counts, each a multiple of 8, copied at coll_spec_create.
     *   reduce-scatter V: nranks entries, the output of each rank (their sum
     *     is every rank's input, `count` of the spec);
     *   all-gather V: nranks entries, the contribution of each rank (their sum
     *     is every rank's output, `count`);
     *   all-to-all V: nranks * nranks entries, [p * nranks + d] = elements
     *     source p sends to destination d (count is ignored). */
    const uint64_t *vcounts;
    int nvcounts;
    int slots;           /* staging slots used in turn by consecutive runs:
                            2 (default, 0 means 2) or 4 (flash-comm §4.2
                            rotating slots; twice the staging memory) */
    uint64_t staging_bytes; /* capacity of each rank's staging image per
                            slot, in bytes; 0 (default) = the whole message.
                            Purlin §4.1: when the staging a collective needs
                            exceeds the capacity, chunks cycle through a
                            fixed number of chunk slots (in the launch by
                            columns, each CTA owns one).  A capacity below
                            the message requires the composed launch (the
                            LL128 twoshot all-reduce, reduce-scatter,
                            all-to-all and their V forms; path AUTO selects
                            it) and must hold
                            at least 4096 * nranks bytes (two chunk slots of
                            the smallest chunk), else COLL_ERR_UNSUPPORTED /
                            COLL_ERR_INVALID.  Such a spec runs only through
                            coll_run with inputs (and coll_run_host):
                            coll_stage, coll_run without inputs,
                            coll_stage_withheld, coll_run_late and
                            coll_staging_layout return COLL_ERR_UNSUPPORTED.
                            Staged lines of chunk c carry epoch + c, and a
                            run advances the epoch by its chunk count
                            rounded up to an odd number (Purlin §4.2), so
                            consecutive runs still alternate slots. */
} coll_options_t;

typedef struct coll_spec coll_spec_t;

/* Fill *opt with the defaults above. */
void coll_options_default(coll_options_t *opt);

/* Validate a collective and derive its schedule (host only, no CUDA call).
 * Purlin §3.1 Listing 1: the triple names the collective; §3.2 Listing 2:
 * the layouts decide who notifies whom and whether consumers copy or reduce.
 * nranks in [1, 8]; count % 8 == 0 (16-byte length alignment, flash-comm
 * §4.1 admission); count may be 0 (an empty call still advances the epoch,
 * flash-comm §4.2).  For MoE dispatch `count` is ignored and tokens, hidden
 * (a multiple of 8), topk and experts come from *opt.
 * Returns COLL_OK and a new spec in *spec, or an error and *spec = NULL. */
coll_status_t coll_spec_create(coll_layout_t in_layout, coll_layout_t out_layout,
                               coll_op_t op, coll_dtype_t dtype, int nranks,
                               size_t count, const coll_options_t *opt,
                               coll_spec_t **spec);

/* Bytes of device workspace the spec needs (header, work lists, reader
 * counters, two staging slots per rank, and for twoshot the two slots of the
 * reduced-partition region).  Purlin §4.1: two staging buffers alternate. */
coll_status_t coll_workspace_bytes(const coll_spec_t *spec, size_t *bytes);

/* Element counts of rank `rank`'s input and output buffers. */
coll_status_t coll_buffer_elems(const coll_spec_t *spec, int rank,
                                size_t *in_elems, size_t *out_elems);

/* Hand the caller-allocated workspace (device memory, 256-byte aligned) to
 * the spec and initialise it on `stream`: every readiness word = 0 (sentinel
 * staging: the all-ones pattern), epoch = 1, status clear, work lists
 * uploaded from host memory (not capturable in a CUDA graph).  Purlin §4
 * "Initialization": buffers are given once and reused for every call.
 * COLL_ERR_NOMEM if bytes is smaller than coll_workspace_bytes. */
coll_status_t coll_bind(coll_spec_t *spec, void *dev_workspace, size_t bytes,
                        coll_stream_t stream);

/* MoE dispatch only: give source rank `rank`'s routing, dev_topk[tokens*topk]
 * (int32 expert ids, distinct per token; the array must stay valid and
 * unchanged until the run that uses it completes).  Counting, the prefix
 * sums and the row placement run on the device at the next coll_stage /
 * coll_run.  Output of destination d: its rows in the order (local expert,
 * source rank, token), each the source's token row; an expert id outside
 * [0, experts) latches COLL_ERR_INVALID and the row is dropped; more rows
 * than max_rows latch COLL_ERR_NOMEM and the excess rows are dropped. */
coll_status_t coll_set_routing(coll_spec_t *spec, int rank,
                               const int32_t *dev_topk, coll_stream_t stream);

/* Stage rank `rank`'s input for the current epoch e: encode it as lines with
 * readiness value e into staging slot e mod slots (2 or 4) of that rank.  The store of a
 * line is its notification (no separate notify step): Purlin §3.2 latency
 * path, flash-comm §3.1.  All ranks must be staged before coll_run(ins=NULL)
 * of the same epoch, in stream order. */
coll_status_t coll_stage(coll_spec_t *spec, int rank, const void *dev_in,
                         coll_stream_t stream);

/* Run the collective for the current epoch, then advance the epoch (by 1;
 * with bounded staging by the run's column count rounded up to odd).
 * dev_ins == NULL: every rank was staged by coll_stage; the consume kernels
 * validate and consume.  dev_ins != NULL (nranks input pointers): staging is
 * done here too -- inside the same cooperative kernel on the FUSED path, as
 * the stage phase of each column of the one launch on the COMPOSED path.
 * dev_outs: nranks output pointers (16-byte aligned).  Consumers reduce in
 * rank order 0..N-1 whatever order lines become ready in (flash-comm §3.3). */
coll_status_t coll_run(coll_spec_t *spec, const void *const *dev_ins,
                       void *const *dev_outs, coll_stream_t stream);

/* End to end from host memory: copy each rank's input from (pinned) host
 * memory into dev_ins[r], run the collective, copy each output back into
 * host_outs[r].  One cudaMemcpyAsync per buffer, all on `stream`. */
coll_status_t coll_run_host(coll_spec_t *spec, const void *const *host_ins,
                            void *const *dev_ins, void *const *dev_outs,
                            void *const *host_outs, coll_stream_t stream);

/* MoE dispatch only: copy counts[dest][local expert][source] (int32,
 * nranks * experts entries) and, after them, the rows of each destination
 * (nranks int32) of the last run into dev_counts (stream-ordered). */
coll_status_t coll_get_counts(const coll_spec_t *spec, int32_t *dev_counts,
                              coll_stream_t stream);

/* Synchronize `stream`, report the latched device error (COLL_OK if none)
 * with the rank and line it concerns, and clear it. */
coll_status_t coll_query_status(coll_spec_t *spec, coll_stream_t stream,
                                int *code, int *rank, int64_t *line);

/* Synchronize `stream` and read the device epoch. */
coll_status_t coll_get_epoch(coll_spec_t *spec, coll_stream_t stream,
                             uint64_t *epoch);

/* Staging geometry, for inspection: region 0 = the rank images written by
 * coll_stage, region 1 = the reduced partitions published by twoshot owners.
 * Returns the byte offset (from the workspace base) of segment `seg` of rank
 * `rank` in slot `slot` (0 .. slots-1; run e uses slot e mod slots), its line
 * count and the line size in bytes. */
coll_status_t coll_staging_layout(const coll_spec_t *spec, int region, int slot,
                                  int rank, int seg, uint64_t *byte_offset,
                                  uint64_t *lines, int *line_bytes);

/* Fault-injection support for the stale-line tests (host-made failures, no
 * GPU fault).  coll_stage_withheld stages rank `rank` like coll_stage but
 * leaves the listed lines stale: their readiness word holds the previous
 * epoch (kind 0), the slot's previous occupant e-2 (kind 1) or zero
 * (kind 2), and their payload a poison pattern.  Line indices are global
 * line numbers of the rank image (segments in order, as given by
 * coll_staging_layout).  All arrays are device arrays of n entries. */
coll_status_t coll_stage_withheld(coll_spec_t *spec, int rank, const void *dev_in,
                                  const int64_t *dev_lines, const int32_t *dev_kind,
                                  const uint16_t *dev_poison, int64_t n,
                                  coll_stream_t stream);

/* Run (inputs already staged, some lines withheld) with late producers in
 * the same cooperative launch: for each rank r, dev_order[r] lists its
 * withheld lines in the order a producer CTA of rank r publishes them after
 * the consumers have started polling; n_late[r] (host array) is the count.
 * dev_ins gives the producers the data to publish. */
coll_status_t coll_run_late(coll_spec_t *spec, const void *const *dev_ins,
                            void *const *dev_outs,
                            const int64_t *const *dev_order,
                            const int64_t *n_late, coll_stream_t stream);

/* Number of stale lines the consumers of the last runs observed and rejected
 * (a diagnostic counter, reset by coll_bind).  Synchronizes `stream`, then
 * reads the counter from the workspace into *rejections (host memory).
 * COLL_ERR_INVALID for a NULL argument, COLL_ERR_STATE before coll_bind,
 * COLL_ERR_CUDA if the synchronization or the copy fails. */
coll_status_t coll_get_rejections(coll_spec_t *spec, coll_stream_t stream,
                                  uint64_t *rejections);

/* Inspection of the derived schedule (host only, no CUDA call).  which = 0:
 * staging items, 1: first consume phase, 2: second consume phase (twoshot
 * all-gather), 3: the exchange pieces of a composed all-to-all (V).  Each
 * item is written as 10 int64 values:
 *   consume: kind (0 fold, 1 copy), flags (1 publish, 2 sole-reader re-arm,
 *            4 counted re-arm), dst rank, src rank, readers, lines, elements,
 *            first source line, output offset (element, or line when
 *            publishing), counter index;
 *   staging: rank, 0, 0, 0, 0, lines, elements, first image line, first
 *            input element, 0;
 *   exchange: source rank p, destination rank x, first line of partition x
 *            in p's image, elements, first input element in p, first output
 *            element in x, 0, 0, 0, 0 (an empty list for other plans).
 * *n receives the number of items; at most cap items are written. */
coll_status_t coll_debug_items(const coll_spec_t *spec, int which, int64_t *buf,
                               size_t cap, size_t *n);

/* Summary of the derived plan: all-reduce algorithm (COLL_ONESHOT /
 * COLL_TWOSHOT, 0 for other collectives), launch path used when inputs are
 * given to coll_run (COLL_PATH_*), CTAs per rank of the fused path, the
 * encoding, and whether the run's kernels are dependent launches (1:
 * launched with programmatic stream serialization; see COLL_PATH_FUSED and
 * COLL_PATH_STREAMED).  Any output pointer may be NULL. */
coll_status_t coll_debug_plan(const coll_spec_t *spec, int *algorithm, int *path,
                              int *ctas_per_rank, int *encoding, int *dependent_launch);

/* Per-launch timing: when set, every following coll_run records events[0]
 * on its stream before its first launch and events[k] after its k-th launch
 * (k = 1 .. n-1; launches beyond n-1 record nothing).  `events` are
 * cudaEvent_t handles owned by the caller; n = 0 turns recording off.  The
 * array is copied, so the caller may reuse its own storage. */
coll_status_t coll_set_profile_events(coll_spec_t *spec, void *const *events, int n);

/* Number of kernel launches the last coll_run issued (host state, no CUDA
 * call; 0 before the first run).  COLL_ERR_INVALID for a NULL argument. */
coll_status_t coll_last_launches(const coll_spec_t *spec, int *launches);

/* Launch floor, for measurement.  flash-comm (Appendix A, Table 8) calibrates
 * an empty-kernel floor inside CUDA graphs, and its cost model (§3.2,
 * Eq. (1)) carries a fixed per-operation term.  This enqueues one empty
 * kernel on `stream` in exactly the launch configuration coll_run(spec, ins,
 * outs) uses on the one-launch paths, the fused kernel or the composed
 * launch by columns: the same grid and block size, the cooperative
 * attribute, and programmatic stream serialization when the spec's runs are
 * dependent launches (the kernel then makes the same dependent-launch
 * handshake as a run's prologue).  It reads and writes no memory and leaves
 * the spec's device state (epoch, staging) untouched, so it may be timed
 * between or instead of runs, eagerly or in a graph.  Returns
 * COLL_ERR_UNSUPPORTED for specs whose runs take neither path (or the
 * composed queue schedule), COLL_ERR_STATE for a composed spec not yet
 * bound, COLL_ERR_CUDA if the launch fails. */
coll_status_t coll_launch_floor(coll_spec_t *spec, coll_stream_t stream);

/* All-reduce without any allocation.  The pages have no counterpart: this is
 * an entry point for callers that cannot allocate device memory when they
 * need the collective -- code running under a stream capture that must not
 * allocate, inside an allocator's own callback, or in a process whose device
 * memory another runtime has fully reserved -- and so cannot provide the
 * workspace that coll_bind takes.
 * It runs the oneshot LL8 all-reduce (stage, validate, fold in rank order
 * 0..nranks-1 in fp32, one rounding to bf16) of nranks buffers of `count`
 * bf16 each into nranks outputs, like coll_run on an (SCATTERED, SCATTERED,
 * REDUCE) spec with COLL_LL8 and COLL_ONESHOT, and gives the same bytes.
 * Its scratch is a fixed array inside the library (8 MiB + 4 KiB), held by
 * every GPU that loads the library until the process exits:
 *   - nranks * count must not exceed 1,048,576 elements: larger requests
 *     return COLL_ERR_NOMEM and enqueue nothing; count % 8 != 0 returns
 *     COLL_ERR_ALIGN; count == 0 does nothing;
 *   - the first call on a device sets that device up (looks up the scratch
 *     address, clears its header, sets the first epoch) with blocking CUDA
 *     calls, so make it before any stream capture that includes this call;
 *   - every call on a device shares the one scratch array, which keeps the
 *     previous call's contents; calls that overlap on the GPU (other streams,
 *     other host threads) race and give undefined outputs;
 *   - a device-side wait that exceeds its bound (200 ms) leaves that call's
 *     outputs undefined.  Such a timeout is not reported: this entry point
 *     returns only host-side errors, and every call first clears the scratch's
 *     status and abort words in stream order (a cudaMemsetAsync ahead of its
 *     launch), so a timeout in one call never affects a later call, and its
 *     status is dropped.  Callers that need device-side error reports use a
 *     bound spec and coll_query_status.
 * It calls no cudaMalloc, cudaFree or other allocating routine. */
coll_status_t coll_allreduce_static(int nranks, size_t count, const void *const *dev_ins,
                                    void *const *dev_outs, coll_stream_t stream);

/* One-sided copy with an explicit pipeline depth -- Purlin §3.3, Eq. (3):
 * `ctas` transfer CTAs (C), each with `stages` pipeline stages (S) of
 * `stage_bytes` bytes (B_stage), keep at most Q_cap = C * S * B_stage bytes
 * of loads in flight; §5.2 (Figure 9) ablates S at fixed C and message size.
 * dev_dst[0 .. bytes) <- dev_src[0 .. bytes), byte for byte.  Both pointers
 * are device addresses of this GPU, 16-byte aligned; the ranges must not
 * overlap.  Chunk c (stage_bytes each, the last one shorter) is copied by
 * CTA c mod C.  Engines:
 *   COLL_ATOM_BULK: one thread per CTA drives S shared-memory stages with
 *     TMA bulk loads (mbarrier completion) and TMA bulk stores;
 *   COLL_ATOM_LSU: 256 threads per CTA keep S stages of cp.async granules in
 *     flight and store them from registers.
 * Arguments: stages 1..8; stage_bytes a positive multiple of 16 with
 * stages * stage_bytes <= 196,608 (shared memory per CTA); ctas 0..65535,
 * 0 = one per SM; bytes a multiple of 16, 0 = nothing to do.  Out-of-range
 * arguments, null pointers or overlapping ranges return COLL_ERR_INVALID,
 * misaligned pointers, sizes or stage_bytes COLL_ERR_ALIGN, and in each case
 * nothing is enqueued.  The copy is asynchronous on `stream`.
 * dev_status (a device int32, may be NULL) is set to COLL_ERR_TIMEOUT if a
 * stage waits longer than one second for its load (the CTA then drains its
 * copies and stops); it is never cleared by the library. */
typedef enum { COLL_ATOM_BULK = 0, COLL_ATOM_LSU = 1 } coll_atom_engine_t;

coll_status_t coll_atom_copy(void *dev_dst, const void *dev_src, size_t bytes, int engine,
                             int ctas, int stages, int stage_bytes, int32_t *dev_status,
                             coll_stream_t stream);

/* Copy ceiling probe, for measurement: `passes` full copies of
 * dev_src[0 .. bytes) into dev_dst in ONE launch, with `ctas` CTAs of 256
 * threads (0 = eight per SM) moving 16-byte granules grid-stride; loads are
 * cached in L2 only.  With both buffers small enough to stay in L2 it gives
 * the SM <-> L2 copy throughput this GPU reaches (read + write bytes =
 * 2 * bytes * passes over the launch's time) without the launch gaps a loop
 * of short copies would measure.  Both pointers are device addresses of this
 * GPU, 16-byte aligned, not overlapping; bytes a multiple of 16 (0 = no
 * launch).  Out-of-range arguments or overlapping ranges return
 * COLL_ERR_INVALID, misalignment COLL_ERR_ALIGN; asynchronous on `stream`. */
coll_status_t coll_copy_passes(void *dev_dst, const void *dev_src, size_t bytes, int passes,
                               int ctas, coll_stream_t stream);

/* Release the spec's host state (never the caller's device memory). */
coll_status_t coll_destroy(coll_spec_t *spec);

/* A short English description of a status code (a static string, never
 * NULL; "unknown status" for a value outside coll_status_t). */
const char *coll_status_string(coll_status_t status);

#ifdef __cplusplus
}
#endif
#endif /* COLL_H */
