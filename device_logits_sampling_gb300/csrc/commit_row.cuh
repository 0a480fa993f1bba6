// The decode-loop commit of one row (arc_decode.h), shared by the standalone
// commit kernel and the finish kernels that commit their own row.
//
// Arc PR #217 "device decode loop", section "What this does" (step 3: the
// token goes into the buffer the next forward reads, the device position
// advances, the token is published into a pinned host ring) and section
// "Fault detection replaces the sync rather than dropping it" (range checks
// before any write, a sticky fault word); Arc PR #220 (records carry the
// row's owner, so a token never reaches another sequence).
#pragma once

#include <cstdint>

#include "arc_decode.h"

namespace arc {

// System-scope release store of a record's stamp: the record's other fields,
// stored before it by this thread, are visible to a host that reads the
// stamp with acquire semantics.
__device__ __forceinline__ void store_release_sys(uint32_t* p, uint32_t v) {
    asm volatile("st.release.sys.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void store_relaxed_sys(uint32_t* p, uint32_t v) {
    asm volatile("st.relaxed.sys.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Orders this thread's earlier stores before its later ones for every
// observer, the host included.
__device__ __forceinline__ void fence_acq_rel_sys() { asm volatile("fence.acq_rel.sys;" ::: "memory"); }

// Row r's commit as record number idx: checks token and position before any
// write, then (when both pass) next_ids[r] = tok and positions[r] += 1, then
// the record.  Returns the row's ARC_COMMIT_* bits.  A slot being rewritten
// first carries a "writing" stamp two laps behind the new record (it matches
// no record a reader waits for and reads as behind, not as an overrun), so a
// host copy taken while the fields change fails its second stamp read.
__device__ __forceinline__ uint32_t commit_row(int32_t tok, int64_t r, uint64_t idx, int32_t V, int32_t* next_ids,
                                               int32_t* positions, int32_t max_position, const uint32_t* owners,
                                               arc_commit_record* ring, uint32_t capacity) {
    const int32_t pos = positions[r];
    uint32_t bad = 0;
    if (tok < 0 || tok >= V) bad |= ARC_COMMIT_BAD_TOKEN;
    if (pos < 0 || pos >= max_position) bad |= ARC_COMMIT_BAD_POSITION;
    if (bad == 0) {
        next_ids[r] = tok;
        positions[r] = pos + 1;
    }
    arc_commit_record* rec = ring + (idx % capacity);
    store_relaxed_sys(&rec->stamp, static_cast<uint32_t>(idx + 1 - 2 * static_cast<uint64_t>(capacity)));
    fence_acq_rel_sys();
    rec->token = bad ? -1 : tok;
    rec->position = pos;
    rec->owner = owners ? owners[r] : 0u;
    store_release_sys(&rec->stamp, static_cast<uint32_t>(idx + 1));
    return bad;
}

}  // namespace arc
