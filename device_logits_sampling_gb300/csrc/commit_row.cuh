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

// One 8-byte word of a record, (value, stamp), by one system-scope store: a
// host read of the aligned word sees all of it or none of it.
__device__ __forceinline__ void store_word_sys(void* p, uint32_t value, uint32_t stamp) {
    const unsigned long long w = (static_cast<unsigned long long>(stamp) << 32) | value;
    asm volatile("st.relaxed.sys.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

// Row r's commit as record number idx, its position `pos` and owner tag
// already read: checks token and position before any write, then (when both
// pass) next_ids[r] = tok and positions[r] = pos + 1, then the record's three
// words, each carrying the stamp idx + 1.  Returns the row's ARC_COMMIT_*
// bits.  No fence: a host accepts the slot only once all three words show the
// same stamp, so their order does not matter.
__device__ __forceinline__ uint32_t commit_row_read(int32_t tok, int32_t pos, uint32_t owner, int64_t r, uint64_t idx,
                                                    int32_t V, int32_t* next_ids, int32_t* positions,
                                                    int32_t max_position, arc_commit_record* ring,
                                                    uint32_t capacity) {
    uint32_t bad = 0;
    if (tok < 0 || tok >= V) bad |= ARC_COMMIT_BAD_TOKEN;
    if (pos < 0 || pos >= max_position) bad |= ARC_COMMIT_BAD_POSITION;
    if (bad == 0) {
        next_ids[r] = tok;
        positions[r] = pos + 1;
    }
    arc_commit_record* rec = ring + (idx % capacity);
    const uint32_t stamp = static_cast<uint32_t>(idx + 1);
    store_word_sys(&rec->token, static_cast<uint32_t>(bad ? -1 : tok), stamp);
    store_word_sys(&rec->position, static_cast<uint32_t>(pos), stamp);
    store_word_sys(&rec->owner, owner, stamp);
    return bad;
}

// The same, reading the row's position and owner tag first.
__device__ __forceinline__ uint32_t commit_row(int32_t tok, int64_t r, uint64_t idx, int32_t V, int32_t* next_ids,
                                               int32_t* positions, int32_t max_position, const uint32_t* owners,
                                               arc_commit_record* ring, uint32_t capacity) {
    return commit_row_read(tok, positions[r], owners ? owners[r] : 0u, r, idx, V, next_ids, positions, max_position,
                           ring, capacity);
}

}  // namespace arc
