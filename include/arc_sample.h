/*
 * arc_sample.h -- on-device logits sampling for GB300 (sm_103a).
 *
 * Turns a decode step's [B, V] logits into next-token ids i32[B] entirely on
 * the GPU, in one launch on the caller's stream, with no host round trip.
 *
 * The operation is the one the Arc pull requests describe:
 *   - Arc PR #222, "ARC_SAMPLE_ON_DEVICE", section 2: at B > 1 the whole
 *     [B, 1, vocab] logits tensor (256 x 129,280 x 2 B = 66.2 MB/step) was
 *     copied to the host for a CPU sampler; this library keeps it on device.
 *   - the same page, section 3(b): the sampler's filters are top-k
 *     ("zero-rest"), the top-p walk and the min-p scan, in that order, and
 *     the server defaults (top_k=-1, top_p=1.0, min_p=0.0) must go straight
 *     to the multinomial draw.
 *   - Arc PR #217, "device decode loop", section "What this does": the
 *     device sampler writes the token to an i32[batch] device buffer that is
 *     never copied down; its greedy argmax is bit-exact with the host's.
 *   - the hybrid-nucleus commit quoted on Arc PR #194: the generator's state
 *     must live in device memory (a by-value argument baked by graph capture
 *     gave 1 distinct token over 64 replays); the device generator is
 *     Splitmix64.
 *
 * Per row r, with z the row's logits as fp32 (bf16 widens exactly):
 *   1. penalties for ids in the row's history, each an fp32 round-to-nearest
 *      operation, count c > 0:  z = z > 0 ? z / rep : z * rep;
 *      z -= fl(c * freq);  z -= pres
 *   2. greedy when temperature == 0 or top_k == 1: smallest index of max z
 *   3. w_i = exp((z_i - max z) / T)
 *   4. top-k (1 < top_k < V): the first top_k ids by (z desc, id asc)
 *   5. top-p (top_p < 1) over the top-k survivors: the largest cutoff tau
 *      with mass{w >= tau} >= top_p * (top-k mass); every entry tied at the
 *      cutoff survives
 *   6. min-p (min_p > 0): w >= min_p
 *   7. u = (splitmix64(seed ^ (row << 32) ^ step) >> 11) * 2^-53, where
 *      splitmix64(x) adds 0x9E3779B97F4A7C15 to x and mixes once
 *   8. the smallest surviving id, in ascending id order, whose running mass
 *      exceeds u * (surviving mass)
 * Greedy tokens and top-k survivor sets are exact.  Weights, masses and the
 * draw use fp32 exponentials with exact fixed-point (integer) sums, so the
 * top-p / min-p cutoffs and the drawn token agree with an fp64 evaluation
 * except where that evaluation lies within about 1e-6 (relative) of a cutoff
 * or of u; results are deterministic and independent of the launch geometry.
 *
 * Threading and memory: all pointers named "device" are caller-owned device
 * memory.  The library allocates nothing and never synchronises; each call
 * enqueues its kernels (arc_sample_batch: a streaming scan, then a per-row
 * finish) on `stream` and returns.  Calls are safe inside CUDA stream capture
 * once the first call for the device has returned (the first call sets
 * per-kernel shared-memory attributes).
 *
 * Workspace: arc_sample_batch needs a caller-owned device workspace of
 * arc_sample_workspace_bytes() bytes, 16-byte aligned.  It carries one small
 * summary per row slice (1,664 bytes) from the scan kernel to the finish
 * kernel of the same call; every byte the finish kernel uses is written earlier in that call, so
 * the workspace needs no initial contents and keeps nothing between calls.
 * Calls that share a workspace must be ordered (same stream, or events);
 * calls that overlap on the GPU and share a workspace race.
 */
#ifndef ARC_SAMPLE_H
#define ARC_SAMPLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 3: arc_commit_record (arc_decode.h) stamps each of its three words;
 *    arc_sample_batch_commit; arc_sample_geometry.finish_ctas; ARC_F16 */
#define ARC_SAMPLE_ABI_VERSION 3

/* logits element types */
#define ARC_F32 0
#define ARC_BF16 1
#define ARC_F16 2

/* host-side return codes: nothing was enqueued when a call returns < 0 */
#define ARC_OK 0
#define ARC_E_NULL (-1)        /* a required pointer is NULL */
#define ARC_E_SHAPE (-2)       /* B <= 0, V <= 0, V > 2^31-1 or ld < V */
#define ARC_E_DTYPE (-3)       /* dtype is not ARC_F32 / ARC_BF16 / ARC_F16 */
#define ARC_E_ALIGN (-4)       /* logits not aligned to the element size */
#define ARC_E_UNSUPPORTED (-5) /* a row does not fit on chip (see arc_sample_plan) */
#define ARC_E_OPTION (-6)      /* bad field in arc_sample_options */
#define ARC_E_CUDA (-7)        /* CUDA error while configuring or launching */
#define ARC_E_WORKSPACE (-8)   /* workspace NULL or smaller than arc_sample_workspace_bytes() */

/* device-side per-row error bits, ORed into *err_word and arc_row_debug.err */
#define ARC_ERR_PARAM 0x1u      /* invalid row parameters: out[row] = -1 */
#define ARC_ERR_HIST_ID 0x2u    /* history id outside [0, V): out[row] = -1 */
#define ARC_ERR_NAN 0x4u        /* NaN logit seen; it counts as -inf */
#define ARC_ERR_DEGENERATE 0x8u /* every logit is -inf or NaN: out[row] = 0 */
#define ARC_ERR_HIST_CAP 0x10u  /* history longer than max_hist_len: out[row] = -1 */
#define ARC_ERR_TIMEOUT 0x20u   /* a bounded on-chip wait gave up: out[row] = -1 */
#define ARC_ERR_INTERNAL 0x40u  /* an exact-arithmetic search failed (a library bug) */

/*
 * Per-row sampling parameters, one per row, in DEVICE memory (48 bytes).
 * Rows are independent; every field is read on the device at each call, so
 * a captured CUDA graph sees the current values on every replay.
 *   temperature       0 => greedy; must be finite and >= 0
 *   top_k             <= 0 or >= V => off; 1 => greedy
 *   top_p             (0, 1]; 1 => off
 *   min_p             [0, 1]; 0 => off
 *   repetition_penalty > 0; 1 => off
 *   frequency_penalty finite; 0 => off
 *   presence_penalty  finite; 0 => off
 *   flags             reserved, must be 0
 *   seed, step        generator inputs: u depends on (seed, row, step)
 * A row with an invalid field gets out[row] = -1 and ARC_ERR_PARAM; the rest
 * of the batch is unaffected.
 */
typedef struct arc_row_params {
    float temperature;
    int32_t top_k;
    float top_p;
    float min_p;
    float repetition_penalty;
    float frequency_penalty;
    float presence_penalty;
    uint32_t flags;
    uint64_t seed;
    uint64_t step;
} arc_row_params;

/*
 * Optional per-row diagnostics (DEVICE memory, [B]), written when
 * arc_sample_options.debug is not NULL.  Survivor sets are described by a
 * threshold on the order-preserving key of the penalised fp32 logit,
 *     key(z) = sign(z) ? ~bits(z) : bits(z) | 0x80000000   (with -0 read as +0),
 * and an id bound: id survives iff key > kappa || (key == kappa && id < iota).
 * kappa = 0, iota = V means "every id".
 */
typedef struct arc_row_debug {
    int32_t mode;       /* -1 invalid, 0 greedy, 1 inert, 2 filtered */
    uint32_t err;       /* ARC_ERR_* bits of this row */
    int32_t token;      /* the value written to out[row] */
    int32_t passes;     /* 1: greedy, default or direct selection; >= 2: threshold
                           bisection ran, one more per pass over the row */
    uint32_t kappa_k;   /* top-k survivor set */
    int32_t iota_k;
    uint32_t kappa_r;   /* final survivor set (top-k, then top-p, then min-p) */
    int32_t iota_r;
    float max_z;        /* max penalised logit */
    int32_t frac_bits;  /* F: masses are integers in units of 2^-F (max w = 1) */
    uint64_t rbits;     /* splitmix64(...) >> 11, so u = rbits * 2^-53 */
    uint64_t mass_k;    /* surviving mass after top-k (0 when not computed) */
    uint64_t mass_r;    /* final surviving mass S_R */
    uint64_t target;    /* floor(u * S_R): token is the first id whose running mass exceeds it */
} arc_row_debug;

/* arc_sample_options.flags */
#define ARC_OPT_STEP_AUTOINC 0x1u /* after reading params[row].step, store step + 1 */
/* filtered rows skip the direct selection (exact enumeration of the few ids
 * above a provable floor) and take the threshold bisection over the whole
 * row; both are exact, so tokens and survivor sets do not change -- a switch
 * for cross-checking the two (arc_row_debug.passes tells which ran) */
#define ARC_OPT_FORCE_BISECTION 0x2u

/*
 * Top-n log-probabilities, one record per listed id (DEVICE memory, [B][top_n]).
 * Arc PR #222, section 3(b): the top-n log-probability output reads the
 * sampler's sort.  Row r lists the top_n ids first in (z desc, id asc) order
 * of its penalised logits -- the top-k filter's order -- with
 *     logprob = (z - max z) / T - ln(sum over every id of exp((z' - max z) / T))
 * at the row's sampling temperature (T = 1 for a greedy row, T == 0), before
 * the top-k / top-p / min-p filters.  -inf logits list logprob -inf; when the
 * max is +inf the +inf ids share the mass; entries past V, and every entry of
 * a row with invalid parameters, are (id -1, logprob -inf).
 */
typedef struct arc_top_logprob {
    int32_t id;
    float logprob;
} arc_top_logprob;

#define ARC_MAX_TOP_N 64

/* Host struct; pass NULL for defaults. */
typedef struct arc_sample_options {
    uint32_t flags;
    int32_t ctas_per_row;  /* slices (scan CTAs) per row: 0 = automatic, else 1..128 */
    int32_t max_hist_len;  /* upper bound on any row's history length; 0 = 1024 */
    int32_t top_n;         /* 0: off; 1..ARC_MAX_TOP_N: write top_logprobs */
    arc_row_debug* debug;  /* device [B] or NULL */
    arc_top_logprob* top_logprobs;  /* device [B][top_n]; required when top_n > 0 */
} arc_sample_options;

/*
 * Sample one token per row.
 *   logits        device, [B rows][ld elements], ARC_F32, ARC_BF16 or ARC_F16, aligned
 *                 to its element size (16-byte aligned rows use 16-byte loads)
 *   B, V, ld      rows, vocabulary, row stride in elements (ld >= V)
 *   params        device [B]; written only under ARC_OPT_STEP_AUTOINC
 *   hist_offsets  device [B + 1] or NULL: row r's history is
 *                 hist_ids[hist_offsets[r] .. hist_offsets[r+1]); ids repeat
 *                 to count occurrences.  NULL means no row has a history.
 *   hist_ids      device, required when hist_offsets is not NULL
 *   out           device [B]: the token ids
 *   err_word      device uint32 or NULL: ARC_ERR_* bits ORed in (sticky:
 *                 the library never clears it)
 *   workspace     device, workspace_bytes >= arc_sample_workspace_bytes(B, V,
 *                 dtype, hist_offsets != NULL, opts); see "Workspace" above
 *   opts          host pointer or NULL
 *   stream        cudaStream_t (NULL = legacy default stream)
 * Returns ARC_OK after enqueueing, or a negative ARC_E_* code with nothing
 * enqueued.  Host checks run before any CUDA call.
 */
int arc_sample_batch(const void* logits, int64_t B, int64_t V, int64_t ld, int32_t dtype,
                     arc_row_params* params, const int32_t* hist_offsets,
                     const int32_t* hist_ids, int32_t* out, uint32_t* err_word,
                     void* workspace, size_t workspace_bytes,
                     const arc_sample_options* opts, void* stream);

/*
 * Workspace bytes arc_sample_batch needs for this shape (host only, no CUDA
 * calls); 0 for arguments arc_sample_batch would reject.  The size covers
 * every automatic launch geometry, so it does not depend on the device.
 */
size_t arc_sample_workspace_bytes(int64_t B, int64_t V, int32_t dtype, int32_t has_history,
                                  const arc_sample_options* opts);

/*
 * Greedy only: out[r] = smallest index of max logits[r, :] (NaN ignored, all
 * -inf/NaN => 0 with ARC_ERR_DEGENERATE).  A streaming kernel: no parameters,
 * no penalties, nothing staged on chip.  Arc PR #217 ("device decode loop",
 * section "What this does"): argmax on device into an i32[batch] buffer.
 */
int arc_sample_greedy(const void* logits, int64_t B, int64_t V, int64_t ld, int32_t dtype,
                      int32_t* out, uint32_t* err_word, void* stream);

/* Launch geometry arc_sample_batch would use (host only, no CUDA calls,
 * assuming a 152-SM GB300 for the automatic choice). */
typedef struct arc_sample_geometry {
    int32_t ctas_per_row;    /* CTAs sharing one row */
    int32_t threads;         /* threads per CTA */
    int32_t slice_elems;     /* logits per CTA */
    int32_t smem_bytes;      /* dynamic shared memory per CTA */
    int64_t grid_ctas;       /* total CTAs */
    int32_t frac_bits;       /* fixed-point fraction bits of the masses */
    int32_t launches;        /* 1: one cluster kernel (a thread-block cluster of
                                ctas_per_row CTAs per row, summaries combined in
                                distributed shared memory); 2: scan + finish */
    int64_t workspace_bytes; /* workspace this geometry uses (0 with one launch) */
    int32_t finish_ctas;     /* two launches: finish CTAs per row (a cluster
                                when > 1: small batches split a row's
                                threshold bisection over it); 1 otherwise */
    int32_t reserved;        /* 0 */
} arc_sample_geometry;

int arc_sample_plan(int64_t B, int64_t V, int32_t dtype, int32_t has_history,
                    const arc_sample_options* opts, arc_sample_geometry* geom);

/*
 * arc_sample_batch without a caller-provided workspace: the entry point for
 * callers that cannot allocate device memory on their sampling path -- a
 * host program that links only this library and the CUDA runtime and owns
 * no allocator, or a serving loop held to a fixed device-memory budget that
 * must not allocate per call.  (The pages have no counterpart: their
 * samplers leave scratch memory to the engine around them.)
 *
 * Arguments, results and error codes are those of arc_sample_batch.  The
 * per-slice summaries go to a scratch array of ARC_STATIC_WORKSPACE_BYTES
 * compiled into the library (a static device array, one per device context,
 * created when the CUDA runtime loads the library's kernels); the library
 * never calls an allocator.  Every call looks the array's address up in the
 * current context (cudaGetSymbolAddress, a host-side lookup), so a device
 * reset or another context never sees a stale address.  The first call on a
 * device sets the kernels' attributes: make it before any stream capture
 * that contains a call.
 *
 * Limit: a shape whose workspace on this device (arc_sample_plan
 * workspace_bytes = B x slices-per-row x 1,664 bytes) exceeds
 * ARC_STATIC_WORKSPACE_BYTES returns ARC_E_WORKSPACE with nothing enqueued.
 * At V = 129,280 a row has 16 slices in bf16 or fp16 and 32 in fp32, so B up
 * to 630 (bf16, fp16) or 315 (fp32) is accepted.  Nothing in the array needs to start at
 * zero: each call writes every byte it later uses.  Every call on a device
 * shares the one array, so calls that may overlap on the GPU (different
 * streams without an ordering between them, or concurrent host threads)
 * race: the caller must serialise them.
 */
#define ARC_STATIC_WORKSPACE_BYTES (16u << 20)

int arc_sample_batch_static(const void* logits, int64_t B, int64_t V, int64_t ld, int32_t dtype,
                            arc_row_params* params, const int32_t* hist_offsets,
                            const int32_t* hist_ids, int32_t* out, uint32_t* err_word,
                            const arc_sample_options* opts, void* stream);

/* Text for an ARC_E_* code (static storage). */
const char* arc_sample_strerror(int code);

/* ARC_SAMPLE_ABI_VERSION of the built library. */
int arc_sample_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* ARC_SAMPLE_H */
