/*
 * arc_decode.h -- the decode-loop commit that follows on-device sampling.
 *
 * Arc PR #217, "device decode loop", sections "What this does" and "Fault
 * detection replaces the sync rather than dropping it": per decode step, on
 * one stream and with no host in the middle, the captured forward runs, the
 * device sampler writes token ids to an i32[batch] device buffer, and a
 * commit kernel range-checks each token and position before it writes
 * anything, scatters the token into the buffer the next forward reads,
 * advances the device position and publishes the token into a pinned,
 * device-mapped host ring; a sticky fault word records what it refused.  The
 * host drains the ring with plain loads -- no CUDA call, no stream sync --
 * and tells "not yet" from "never" with a non-blocking stream query: a stream
 * that has retired every step while fewer records than steps have landed did
 * not do what it was asked.  A bound on polls is a last-resort backstop, not
 * the detector.
 * Arc PR #220 (parked burst tokens no longer outlive their sequence): a
 * token must never be taken by another sequence as its own, so every ring
 * record carries its row's owner tag.
 * The pages give no code for either; the record layout and the calls below
 * are this library's own.
 *
 * The commit runs either as its own kernel after the sampler
 * (arc_decode_commit) or inside the sampler's per-row finish
 * (arc_sample_batch_commit), with the same checks, record and ordering.
 *
 * Publication: a record is three 8-byte words -- (token, stamp), (position,
 * stamp), (owner, stamp) -- each written with one system-scope 64-bit store,
 * and a host read of an aligned 8-byte word sees one store or another, never
 * a mix.  The host accepts a slot as record i only when all three words carry
 * stamp i + 1: a slot caught while a later lap rewrites it shows a later
 * stamp in some word (an overrun), a slot not yet written an earlier one (not
 * yet), so no copy mixes two records and the writer needs no fence.  Every
 * argument is a pointer or a size and the ring index lives in device memory
 * (*head), so a commit captured into a CUDA graph publishes fresh records on
 * every replay.  Stamps are 32-bit: a host that falls 2^32 records behind a
 * slot could take a record 2^32 laps old for the one it waits for.
 */
#ifndef ARC_DECODE_H
#define ARC_DECODE_H

#include <stddef.h>
#include <stdint.h>

#include "arc_sample.h"

#ifdef __cplusplus
extern "C" {
#endif

/* One published row-step: three 8-byte words, each with the record's stamp
 * (record index + 1) mod 2^32 in its high half.  24 bytes. */
typedef struct arc_commit_record {
    int32_t token;        /* the committed id, or -1 when the row was refused */
    uint32_t stamp;
    int32_t position;     /* the row's position before this commit */
    uint32_t stamp_pos;   /* == stamp in a complete record */
    uint32_t owner;       /* owners[row] when the commit ran (0 when owners is NULL) */
    uint32_t stamp_owner; /* == stamp in a complete record */
} arc_commit_record;

/* fault bits ORed into *fault_word (sticky: the library never clears it) */
#define ARC_COMMIT_BAD_TOKEN 0x1u    /* a token outside [0, V): the row is refused */
#define ARC_COMMIT_BAD_POSITION 0x2u /* a position outside [0, max_position): refused */

/* return codes of the calls below besides the ARC_E_* codes of arc_sample.h */
#define ARC_E_RING_OVERRUN (-9) /* the ring was overwritten before it was drained */

/* the largest ring (records) */
#define ARC_RING_MAX_CAPACITY (1u << 30)

/*
 * Commit one step: row r of tokens[0 .. B) becomes record number *head + r.
 *   tokens        device [B]: the step's ids (arc_sample_batch's `out`)
 *   B, V          rows; vocabulary size (a committed id lies in [0, V))
 *   next_ids      device or mapped [B]: next_ids[r] = tokens[r] when row r
 *                 commits (the input buffer the next forward reads)
 *   positions     device [B]: row r commits only when 0 <= positions[r] <
 *                 max_position, and then positions[r] += 1
 *   max_position  > 0
 *   owners        device [B] or NULL: owner tags copied into the records
 *   ring          device-visible address of `capacity` records in pinned,
 *                 mapped host memory, 8-byte aligned (arc_ring_alloc gives
 *                 both addresses)
 *   capacity      records in the ring, >= B and <= 2^30
 *   head          device uint64: records published by all earlier commits;
 *                 this call publishes records *head .. *head + B - 1, record
 *                 i at ring[i % capacity], and adds B
 *   fault_word    device or mapped uint32, or NULL: ARC_COMMIT_* bits
 *   stream        cudaStream_t
 * A refused row writes nothing but its record (token -1) and its fault bit.
 * Returns ARC_OK after enqueueing, or a negative ARC_E_* code (arc_sample.h)
 * with nothing enqueued (ARC_E_ALIGN: ring or head not 8-byte aligned); host
 * checks run before any CUDA call.
 */
int arc_decode_commit(const int32_t* tokens, int64_t B, int32_t V, int32_t* next_ids,
                      int32_t* positions, int32_t max_position, const uint32_t* owners,
                      arc_commit_record* ring, uint32_t capacity, uint64_t* head,
                      uint32_t* fault_word, void* stream);

/* The commit's arguments for arc_sample_batch_commit (56 bytes). */
typedef struct arc_commit_target {
    int32_t* next_ids;          /* as in arc_decode_commit */
    int32_t* positions;         /* as in arc_decode_commit */
    const uint32_t* owners;     /* as in arc_decode_commit (NULL: owner 0) */
    arc_commit_record* ring;    /* as in arc_decode_commit */
    uint64_t* head;             /* device, TWO words: head[0] as arc_decode_commit's
                                   *head; head[1] the rows of the running call that
                                   have committed: 0 before the first call, and
                                   every call leaves it 0 */
    uint32_t* fault_word;       /* as in arc_decode_commit (NULL: none) */
    int32_t max_position;       /* as in arc_decode_commit */
    uint32_t capacity;          /* as in arc_decode_commit */
} arc_commit_target;

/*
 * arc_sample_batch followed by arc_decode_commit, without the commit's own
 * launch: the CTA that finishes row r commits row r right after it writes
 * out[r] (same checks, same record, same publication); head[0] is read by
 * every row early in the call and advanced by B once all have read it.  Sampling arguments, results
 * and return codes are arc_sample_batch's; tokens = out, B and V are the
 * sampler's.  Afterwards out, next_ids, positions, the ring, head[0] and the
 * fault word hold exactly what arc_sample_batch then arc_decode_commit on the
 * same stream would leave.  Calls that share a head must not overlap (as for
 * arc_decode_commit).  Extra host checks, before any CUDA call: commit,
 * next_ids, positions, ring and head non-NULL (ARC_E_NULL), ring and head
 * 8-byte aligned (ARC_E_ALIGN), max_position > 0 and B <= capacity <=
 * ARC_RING_MAX_CAPACITY (ARC_E_SHAPE).
 */
int arc_sample_batch_commit(const void* logits, int64_t B, int64_t V, int64_t ld, int32_t dtype,
                            arc_row_params* params, const int32_t* hist_offsets, const int32_t* hist_ids,
                            int32_t* out, uint32_t* err_word, void* workspace, size_t workspace_bytes,
                            const arc_sample_options* opts, const arc_commit_target* commit, void* stream);

/*
 * Host only, no CUDA call: copy records first .. first + count - 1 of `ring`
 * (the host address of the pinned array) to out[0 .. count), in order, each
 * once all three of its stamps are (index + 1) mod 2^32.  Polls a missing record at most
 * max_spins times before giving up.  Returns how many records were copied
 * (fewer than count when one did not land in time), or ARC_E_RING_OVERRUN
 * when a slot holds (part of) a later record, or ARC_E_NULL / ARC_E_SHAPE for
 * bad arguments.
 */
int64_t arc_ring_drain(const arc_commit_record* ring, uint32_t capacity, uint64_t first, int64_t count,
                       arc_commit_record* out, uint64_t max_spins);

/*
 * Non-blocking: 1 when every piece of work enqueued on `stream` has retired,
 * 0 while some has not, or a negative ARC_E_CUDA when the query reports an
 * error (which may come from an earlier, asynchronous launch).
 */
int arc_stream_idle(void* stream);

/*
 * A pinned host array of `bytes` bytes, zero-filled and mapped into the
 * device's address space: *host for the host's reads, *device for kernels.
 * The only allocating calls of the library, kept apart from the sampling
 * path.  Returns ARC_OK, ARC_E_NULL or ARC_E_CUDA.
 */
int arc_ring_alloc(size_t bytes, void** host, void** device);
int arc_ring_free(void* host);

#ifdef __cplusplus
}
#endif
#endif /* ARC_DECODE_H */
