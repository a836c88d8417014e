/*
 * seg_reduce.h -- C ABI of libsegreduce, a segmented reduction over
 * offset-delimited (CSR indptr) segments for NVIDIA GB300 (sm_103a).
 *
 * The operation.  GPUSegmentedReduction (luma.gl API reference), sections
 * "What is an offset-delimited segment?" and "Contract": segment s owns the
 * half-open row range [offsets[s], offsets[s+1]); S segments take S+1
 * offsets; repeated offsets are empty segments and an empty segment produces
 * zero; offsets[0] may be non-zero and rows outside [offsets[0], offsets[S])
 * are ignored.  graph-reduce README (HF kernels hub), sections "API",
 * "Method" and "Correctness": values may be a row tensor [N, F] reduced
 * over dimension 0 (one result per segment and column); min and max also
 * report the source row, with ties going to the lower row; mean is the
 * segment sum divided by the segment length and is 0 for an empty segment;
 * the arg of an empty segment is -1.
 *
 * Numerics.  uint32 / sint32 sums wrap modulo 2^32.  uint32 compares
 * unsigned, sint32 signed, float32 by IEEE '<' / '>' (-0.0 ties with +0.0,
 * so the lower row and its bits win; NaN inputs give unspecified results).
 * float32 sums are not in row order, but the order is a pure function of
 * (num_values, F, S, offsets) and the GPU's SM count, so repeated calls are
 * bitwise identical; the error is below 1e-5 * sum(|x|) + 1e-6 per output.
 * mean = (float)sum / (float)length, rounded to nearest.
 *
 * Memory.  Every pointer argument except `out_arg` may be NULL only when
 * num_segments == 0.  All data pointers are device pointers owned by the
 * caller, on the device that is current for the calling host thread; the
 * library keeps no reference after the call returns.  Scratch space is owned
 * by the library: one small buffer per (device, stream), allocated on first
 * use (stream-ordered), grown when needed and kept until process exit.
 * Outputs must not overlap inputs.
 *
 * Asynchrony.  seg_reduce enqueues work on `stream` and returns without
 * synchronising and without reading any device memory on the host.  Errors
 * that the host can see (argument checks, launch failures) are returned
 * before or at launch; a device-side error (a bounded wait that ran out)
 * is recorded in a per-device status word that seg_reduce_device_status
 * reads.
 */
#ifndef SEG_REDUCE_H
#define SEG_REDUCE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as the CUDA runtime's cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *seg_stream_t;

typedef enum { SEG_U32 = 0, SEG_S32 = 1, SEG_F32 = 2 } seg_dtype_t;
typedef enum { SEG_OFF_U32 = 0, SEG_OFF_I64 = 1 } seg_offset_dtype_t;
typedef enum { SEG_SUM = 0, SEG_MIN = 1, SEG_MAX = 2, SEG_MEAN = 3 } seg_op_t;

typedef enum {
    SEG_OK = 0,
    SEG_ERR_INVALID_ARGUMENT = 1, /* a null pointer, a bad enum, a negative size, misaligned data */
    SEG_ERR_UNSUPPORTED = 2,      /* mean on integer values, F above SEG_MAX_FEATURES */
    SEG_ERR_OUT_OF_MEMORY = 3,    /* the scratch buffer could not be allocated */
    SEG_ERR_CUDA = 4,             /* a CUDA runtime call or a launch failed */
    SEG_ERR_DEVICE_TIMEOUT = 5,   /* a device-side bounded wait ran out (see seg_reduce_device_status) */
    SEG_ERR_SCRATCH_LIMIT = 6     /* seg_reduce_noalloc: the call needs more than SEG_NOALLOC_SCRATCH_BYTES */
} seg_status_t;

/* Largest F (columns per row) that seg_reduce accepts. */
#define SEG_MAX_FEATURES 2048

/*
 * seg_reduce -- out[s, f] = op over rows r in [offsets[s], offsets[s+1]) of values[r, f].
 *
 *   values        device, [num_values, F] row-major, element type `dtype`,
 *                 aligned to 4 bytes (16 bytes enables the vectorised
 *                 row path when F is a multiple of 4).
 *   dtype         SEG_U32, SEG_S32 or SEG_F32.
 *   F             columns per row, 1 <= F <= SEG_MAX_FEATURES; F == 1 is the
 *                 scalar vector case.
 *   num_values    rows in `values` (N >= 0).  Offsets are clamped to [0, N]
 *                 on the device, so malformed offsets never read out of bounds.
 *   offsets       device, [num_segments + 1], SEG_OFF_U32 (uint32) or
 *                 SEG_OFF_I64 (int64), aligned to its element size.
 *                 Precondition (not checked, as in the luma contract):
 *                 nondecreasing and within [0, N].  If it does not hold the
 *                 results are unspecified but no memory outside the
 *                 arguments is touched.
 *   num_segments  S >= 0.  S == 0 returns SEG_OK and launches nothing.
 *   op            SEG_SUM, SEG_MIN, SEG_MAX, or SEG_MEAN (float32 only,
 *                 otherwise SEG_ERR_UNSUPPORTED).
 *   out           device, [S, F], element type `dtype`, aligned to 4 bytes.
 *   out_arg       device, [S, F] int64, or NULL.  For SEG_MIN / SEG_MAX it
 *                 receives the absolute row index of the extreme (lowest
 *                 row on ties), -1 for an empty segment.  It must be NULL
 *                 for SEG_SUM / SEG_MEAN (SEG_ERR_INVALID_ARGUMENT otherwise).
 *   stream        CUDA stream the work is ordered on.
 *
 * Returns SEG_OK when the work was enqueued.
 */
seg_status_t seg_reduce(const void *values, seg_dtype_t dtype, int64_t F,
                        int64_t num_values, const void *offsets,
                        seg_offset_dtype_t offsets_dtype,
                        int64_t num_segments, seg_op_t op, void *out,
                        int64_t *out_arg, seg_stream_t stream);

/* Static, human-readable text for a status code (never NULL). */
const char *seg_reduce_strerror(seg_status_t status);

/*
 * Synchronises `stream`, then reads and clears the device status word of
 * the current device.  Returns SEG_OK if no call on this device has
 * recorded a device-side error since the last read, SEG_ERR_DEVICE_TIMEOUT
 * if a bounded wait inside a kernel ran out (that call's outputs are then
 * incomplete), or SEG_ERR_CUDA if synchronising failed.
 */
seg_status_t seg_reduce_device_status(seg_stream_t stream);

/*
 * The launch the library would make, computed on the host only (no CUDA
 * call, no device memory touched), so that it can be inspected and tested
 * without a GPU.  `values_addr` is the address `values` would have (only
 * its alignment matters) and `sm_count` the device's multiprocessor count.
 */
typedef struct {
    int32_t grid;            /* CTAs launched (at most one per SM)                         */
    int32_t block;           /* threads per CTA (one work unit per warp)                   */
    int32_t slot_threads;    /* lanes that work on one row (scalar kernel: 1)              */
    int32_t items_per_slot;  /* scalar: rows per lane per tile; rows: rows in flight       */
    int32_t vec;             /* 32-bit elements per load                                   */
    int32_t vecs_per_thread; /* column slices a row is cut into (scalar kernel: 1)         */
    int32_t max_ends;        /* scalar: segment ends per tile at most; rows: 0             */
    int32_t kernel_variant;  /* index of the compiled kernel shape                         */
    int64_t smem_bytes;      /* dynamic shared memory per CTA                              */
    int64_t workspace_bytes; /* library-owned scratch the launch uses                      */
} seg_plan_t;

seg_status_t seg_reduce_plan(seg_dtype_t dtype, int64_t F, int64_t num_values,
                             seg_offset_dtype_t offsets_dtype,
                             int64_t num_segments, seg_op_t op,
                             uint64_t values_addr, int32_t sm_count,
                             seg_plan_t *plan);

/*
 * seg_reduce_noalloc -- seg_reduce without any allocation.
 *
 * The reduction pages have no counterpart of this call: it exists for
 * callers that may not allocate device memory at the moment they reduce,
 * for example a runtime whose device memory is all reserved ahead of time by
 * its own arena, or a latency-critical loop that must not touch the
 * stream-ordered allocator pool (growing or trimming that pool can add
 * synchronisation and jitter).  It computes exactly what seg_reduce computes
 * for the same arguments (same kernels, same launch shape, same summation
 * order, so results are bitwise equal to seg_reduce's), but the scratch it
 * needs (ticket words and cross-unit partials) lives in a fixed array of
 * SEG_NOALLOC_SCRATCH_BYTES bytes of static device memory inside the library,
 * one per device, and no call to cudaMalloc, cudaMallocAsync, cudaFree or any
 * other allocating routine is made.
 *
 * Arguments are those of seg_reduce plus:
 *   status_word   device, caller-owned, 4-byte aligned, or NULL.  A kernel
 *                 whose bounded wait runs out ORs a nonzero code into it
 *                 (the call's outputs are then incomplete); the library never
 *                 clears it.  NULL sends such codes to a word inside the
 *                 library that nothing reads.  seg_reduce_device_status does
 *                 not see errors of this call.
 *
 * Limit.  The scratch a launch needs grows with the grid: (ticket words:
 * SM count * 128 bytes rounded up to 256) + (partials: 2 * grid * 16 * 16
 * bytes for F == 1; 2 * grid * 8 * 32 * vec * (4, or 12 for min / max)
 * bytes for F > 1, grid and vec being seg_reduce_plan's).  On a 152-SM GPU
 * every F == 1 call, every sum and mean, and min / max on rows loaded at
 * most two columns at a time fit.  The planner loads four columns at a time
 * whenever F > 64, F % 4 == 0 and the rows are 16-byte aligned; min / max on
 * such rows need 24 KiB per CTA and fit while the grid is at most 84 CTAs
 * (for F = 96, up to about 86,000 weighted rows; seg_reduce_plan reports
 * workspace_bytes).  A call that would need more returns
 * SEG_ERR_SCRATCH_LIMIT before launching anything; use seg_reduce for it.
 *
 * Set-up.  The first call on each device looks up the array's address
 * (cudaGetSymbolAddress, with that device current), clears its ticket words
 * (a stream-ordered memset on `stream`) and waits for `stream` to finish
 * that; the first call of each kernel shape on a device also sets the
 * kernel's shared-memory attribute.  Make one call of each shape you will
 * use before any stream capture.  After that a call only enqueues one
 * memset every 2^32 - 1 calls (when the generation tag of the ticket words
 * wraps) plus the kernel launch.
 *
 * What must start at zero: only the ticket words (the first
 * SM count * 128 bytes of the array); the library zeroes them itself as
 * described above.  Partials are always written before they are read.
 *
 * Concurrency.  All calls on one device share the one array.  Two calls
 * whose kernels can overlap in time (different streams without an ordering
 * between them, or different host threads) race on it and give wrong
 * results; order them on one stream, or synchronise between them.
 */
#define SEG_NOALLOC_SCRATCH_BYTES (2u << 20)

seg_status_t seg_reduce_noalloc(const void *values, seg_dtype_t dtype, int64_t F,
                                int64_t num_values, const void *offsets,
                                seg_offset_dtype_t offsets_dtype,
                                int64_t num_segments, seg_op_t op, void *out,
                                int64_t *out_arg, unsigned int *status_word,
                                seg_stream_t stream);

/*
 * seg_scan -- segmented scan over the same offsets.
 *
 * The pages name a segmented scan (GPUSegmentedScan, beside GPUScan on the
 * luma.gl GPURunLengthEncode page) without defining it; the segments are
 * GPUSegmentedReduction's ("What is an offset-delimited segment?").  For
 * every row r of segment s (offsets[s] <= r < offsets[s+1]):
 *   inclusive: out[r] = op(values[offsets[s]], ..., values[r]);
 *   exclusive (SEG_SUM only): out[r] = sum(values[offsets[s] .. r - 1]),
 *     0 at the segment's first row;
 * and out[r] = 0 for a row in no segment (before offsets[0] or from
 * offsets[S] on).  Integer sums wrap modulo 2^32; uint32 compares unsigned,
 * sint32 signed, float32 by IEEE '<' / '>'.  float32 sums are not in row
 * order; the order is a pure function of (num_values, offsets, the SM count)
 * and the error stays below 1e-5 * sum(|x| over the row's prefix) + 1e-6.
 *
 *   values         device, [num_values] of `dtype`, aligned to 4 bytes (16
 *                  bytes, with out 16-byte aligned, enables 128-bit loads).
 *   num_values     N >= 0; N == 0 returns SEG_OK and launches nothing.
 *   offsets, offsets_dtype, num_segments: as for seg_reduce (S >= 0; with
 *                  S == 0 every row is in no segment).
 *   op             SEG_SUM, SEG_MIN or SEG_MAX.
 *   exclusive      0 or 1 (1 only with SEG_SUM, else SEG_ERR_UNSUPPORTED).
 *   out            device, [num_values] of `dtype`, aligned to 4 bytes; must
 *                  not overlap values.
 *
 * Scratch (a start bitmap of N / 8 bytes and 36 KiB of per-CTA words) comes
 * from the library's per-(device, stream) buffer.  Enqueues four kernel
 * launches and returns without synchronising.
 */
seg_status_t seg_scan(const void *values, seg_dtype_t dtype, int64_t num_values,
                      const void *offsets, seg_offset_dtype_t offsets_dtype,
                      int64_t num_segments, seg_op_t op, int32_t exclusive, void *out,
                      seg_stream_t stream);

/*
 * seg_scatter -- the unsorted scatter path: row r of src goes to output row
 * index[r].
 *
 * graph-reduce README (HF kernels hub), "API": scatter_sum / scatter_add,
 * scatter_mean (an output that receives no row is 0), scatter_max /
 * scatter_min returning (values, arg); index is [N] int64.  "Method": one
 * atomic per element; for max / min the value and its row settle inside one
 * 64-bit atomic, with ties to the lower row.  Here max / min first read the
 * output's current word and skip the atomic when the element cannot win
 * (the word only moves one way, so a stale read only costs an atomic); the
 * results are those of one atomic per element.
 *
 *   src        device, [num_rows, F] row-major, element type `dtype`, aligned
 *              to 4 bytes (16 bytes, with out 16-byte aligned and F % 4 == 0,
 *              enables 128-bit float32 vector reductions).
 *   dtype      SEG_U32, SEG_S32 or SEG_F32.
 *   F          columns, 1 <= F <= SEG_MAX_FEATURES.
 *   num_rows   N, 0 <= N < 2^32 - 1 (rows are packed into 32 bits), and
 *              N * F <= 2^40 (else SEG_ERR_UNSUPPORTED).
 *   index      device, [N] int64, aligned to 8 bytes.  A row whose index is
 *              outside [0, dim_size) goes nowhere.
 *   dim_size   D >= 0 output rows; D == 0 returns SEG_OK and launches nothing.
 *   op         SEG_SUM, SEG_MIN, SEG_MAX, or SEG_MEAN (float32 only).
 *   out        device, [D, F], element type `dtype`, aligned to 4 bytes.  An
 *              output that receives no row is 0.
 *   out_arg    device, [D, F] int64, or NULL: for SEG_MIN / SEG_MAX the row
 *              holding the extreme (the lowest such row; -1 when none).  It
 *              must be NULL for SEG_SUM / SEG_MEAN.
 *
 * Numerics as for seg_reduce (integer sums wrap modulo 2^32; -0.0 and +0.0
 * tie), except that float32 sums and means are not reproducible bit for
 * bit: the order in which the atomics land varies from run to run (the
 * error stays below 1e-5 * sum(|x|) + 1e-6 per output).  Integer sums and
 * max / min are deterministic.  Scratch (D * F * 8 bytes for max / min, D * 4
 * for mean) comes from the library's per-(device, stream) buffer.  Enqueues
 * two or three kernel launches and returns without synchronising.
 */
seg_status_t seg_scatter(const void *src, seg_dtype_t dtype, int64_t F, int64_t num_rows,
                         const int64_t *index, int64_t dim_size, seg_op_t op, void *out,
                         int64_t *out_arg, seg_stream_t stream);

/*
 * seg_scatter_sorted -- the scatter path made deterministic: the same
 * results as seg_scatter (same arguments, same readings), but float32 sums
 * and means are bitwise reproducible.
 *
 * graph-reduce README (HF kernels hub), "Correctness": the atomic scatter's
 * order is not fixed, the CSR path's is; and "Usage": rows sorted by
 * destination, with the pointer built from the destination counts, go
 * through the CSR path.  This call does that on the device: a stable radix
 * sort of the rows by destination (an index outside [0, dim_size) sorts
 * last and is left out), the offsets of each destination's rows, a gather
 * of the rows in sorted order, seg_reduce over them, and the args of
 * max / min mapped back to src's rows.  Within a destination the rows keep
 * their order, so the result equals, bit for bit, seg_reduce over all of
 * src's rows stably sorted by destination (an index outside [0, dim_size)
 * taken as dim_size) with the offsets of the destinations' counts.
 *
 * Arguments as for seg_scatter; num_rows and dim_size below 2^32 - 1.
 * Scratch: a buffer of its own per (device, stream) of about 16 bytes per row
 * plus num_rows * F * 4 bytes for the gathered rows plus 8 bytes per output
 * row; seg_reduce uses its own.  Enqueues the sort (three launches per 8 bits
 * of dim_size), three more launches and seg_reduce's, and returns without
 * synchronising.
 */
seg_status_t seg_scatter_sorted(const void *src, seg_dtype_t dtype, int64_t F, int64_t num_rows,
                                const int64_t *index, int64_t dim_size, seg_op_t op, void *out,
                                int64_t *out_arg, seg_stream_t stream);

/*
 * seg_reduce_sequential -- the input-order float32 mode of the sum and mean.
 *
 * graph-reduce README (HF kernels hub), "Correctness": its CSR path is
 * bitwise equal to torch.segment_reduce because the summation order is
 * fixed.  Here that order is the input order: out[s, f] starts at 0.0f and
 * adds values[r, f] for r = offsets[s], ..., offsets[s+1] - 1, each
 * addition rounded to float32 (round to nearest even); SEG_MEAN divides that
 * sum by the length as a float32 (one more rounding); an empty segment gives
 * 0.  The result is a pure function of the inputs, so any machine that adds
 * in that order reproduces it bit for bit.  seg_reduce's float sums use a
 * different (also fixed) order and are faster: this call is one chain of
 * dependent additions per (segment, column), so its time grows with the
 * longest segment (about one float32 addition latency per row).  min and
 * max do not depend on the order: use seg_reduce.
 *
 *   values, F, num_values, offsets, offsets_dtype, num_segments, out:
 *            as for seg_reduce, with float32 values and out.
 *   op       SEG_SUM or SEG_MEAN (SEG_ERR_INVALID_ARGUMENT otherwise).
 *   stream   CUDA stream the work is ordered on.
 *
 * Enqueues one kernel launch (none when num_segments == 0), uses no
 * scratch, and returns without synchronising.  Argument errors as for
 * seg_reduce.
 */
seg_status_t seg_reduce_sequential(const float *values, int64_t F, int64_t num_values,
                                   const void *offsets, seg_offset_dtype_t offsets_dtype,
                                   int64_t num_segments, seg_op_t op, float *out,
                                   seg_stream_t stream);

/*
 * seg_rle -- run-length encoding of an ordered uint32 vector: the producer
 * of offsets that groups equal adjacent keys.
 *
 * GPURunLengthEncode and GPUUnique (luma.gl API reference), sections "What
 * is run-length encoding?" and "Contract": every maximal run of adjacent
 * equal keys becomes one run; runs keep first-occurrence order; equal keys
 * that are not adjacent start separate runs; an empty input gives zero
 * runs.  Run r has value values[r], length lengths[r] and starts at
 * offsets[r]; offsets[count] = n, so offsets delimit the runs as CSR
 * offsets (lengths [3,2,4] go with offsets [0,3,5,9], the page's "Why RLE
 * matters for GPU grouping") and can be passed to seg_reduce as they are.
 * GPUUnique is this call with only `values` requested.
 *
 *   keys     device, [n] uint32, aligned to 4 bytes (16 bytes enables
 *            128-bit loads).  May be NULL only when n == 0.
 *   n        0 <= n <= UINT32_MAX (lengths are uint32).
 *   values   device, room for n uint32, aligned to 4 bytes, or NULL.
 *   lengths  device, room for n uint32, aligned to 4 bytes, or NULL.
 *   offsets  device, room for n + 1 int64, aligned to 8 bytes, or NULL.
 *   count    device, one int64, aligned to 8 bytes: receives the number of
 *            runs.  Required.
 *   stream   CUDA stream the work is ordered on.
 *
 * Only the first count (values, lengths) or count + 1 (offsets) entries are
 * written.  Inputs and outputs must not overlap.  Scratch is the library's
 * per-(device, stream) buffer described above; these calls grow it to hold
 * a start bitmap (n / 8 bytes) and 12 bytes per 16,384 elements.  The call
 * enqueues two kernel launches (one when n == 0) and returns without
 * synchronising; the count stays on the device.  Returns
 * SEG_ERR_INVALID_ARGUMENT for a NULL keys with n > 0, a NULL count, a
 * negative or too large n, or a misaligned pointer.
 */
seg_status_t seg_rle(const uint32_t *keys, int64_t n, uint32_t *values, uint32_t *lengths,
                     int64_t *offsets, int64_t *count, seg_stream_t stream);

/*
 * seg_flags_to_offsets -- offsets from segment-start flags.
 *
 * GPUSegmentedLayout as GPUSegmentedReduction's "What is an offset-delimited
 * segment?" names it: it materialises offsets from segment-start flags.
 * Every index i with flags[i] != 0 starts a segment; the offsets list those
 * indices in increasing order followed by n.  Rows before the first flag
 * belong to no segment (the reduction allows offsets[0] > 0).
 *
 *   flags    device, [n] bytes (any non-zero byte is a start).  May be NULL
 *            only when n == 0.  16-byte alignment enables 128-bit loads.
 *   n        n >= 0.
 *   offsets  device, room for n + 1 int64, aligned to 8 bytes.  Required.
 *   count    device, one int64, aligned to 8 bytes: receives the number of
 *            segments.  Required.
 *   stream   CUDA stream the work is ordered on.
 *
 * Enqueues two kernel launches (one when n == 0; scratch as for seg_rle)
 * and returns without synchronising.  Returns SEG_ERR_INVALID_ARGUMENT for a
 * NULL flags with n > 0, a NULL offsets or count, a negative n, or a
 * misaligned pointer; SEG_ERR_UNSUPPORTED when n needs more than 2^31 - 1
 * tiles of 16,384 flags.
 */
seg_status_t seg_flags_to_offsets(const uint8_t *flags, int64_t n, int64_t *offsets,
                                  int64_t *count, seg_stream_t stream);

/*
 * seg_selftest_wait_timeout -- exercise the failure path of the bounded
 * waits without a fault.  The kernels wait on mbarriers for their bulk
 * copies with a time limit (2 s); a wait that runs out records
 * SEG_ERR_DEVICE_TIMEOUT in the device status word (read by
 * seg_reduce_device_status) and the kernel returns, so the context stays
 * usable.  This call launches one thread that runs the same bounded wait on
 * an mbarrier phase that nothing completes, with a limit of `limit_ms`
 * milliseconds (1 .. 10000): after it, seg_reduce_device_status reports
 * SEG_ERR_DEVICE_TIMEOUT once and the device keeps working.  The pages have
 * no counterpart of this call; it exists for tests.
 */
seg_status_t seg_selftest_wait_timeout(uint32_t limit_ms, seg_stream_t stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t seg_reduce_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SEG_REDUCE_H */
