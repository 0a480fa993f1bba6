// The decode-loop commit (arc_decode.h): one small kernel after the sampler,
// and the host side of the ring it publishes into.
#include <cuda_runtime.h>

#include <cstdint>

#include "arc_decode.h"
#include "arc_sample.h"
#include "commit_row.cuh"

namespace {

constexpr int kCommitThreads = 1024;

struct CommitArgs {
    const int32_t* tokens;
    int64_t B;
    int32_t V;
    int32_t* next_ids;
    int32_t* positions;
    int32_t max_position;
    const uint32_t* owners;
    arc_commit_record* ring;
    uint32_t capacity;
    uint64_t* head;
    uint32_t* fault_word;
};

// One CTA: every row of the step, then the ring head.  The range checks come
// before any write of the row; a refused row publishes a record with token -1.
__global__ void __launch_bounds__(kCommitThreads) commit_kernel(const __grid_constant__ CommitArgs a) {
    const uint64_t head = *a.head;  // read by every thread before thread 0 advances it
    uint32_t faults = 0;
    for (int64_t r = threadIdx.x; r < a.B; r += kCommitThreads)
        faults |= arc::commit_row(a.tokens[r], r, head + static_cast<uint64_t>(r), a.V, a.next_ids, a.positions,
                                  a.max_position, a.owners, a.ring, a.capacity);
    if (faults && a.fault_word) atomicOr(a.fault_word, faults);
    __syncthreads();  // every thread has read *head
    if (threadIdx.x == 0) *a.head = head + static_cast<uint64_t>(a.B);
}

}  // namespace

extern "C" {

int arc_decode_commit(const int32_t* tokens, int64_t B, int32_t V, int32_t* next_ids,
                      int32_t* positions, int32_t max_position, const uint32_t* owners,
                      arc_commit_record* ring, uint32_t capacity, uint64_t* head,
                      uint32_t* fault_word, void* stream) {
    if (tokens == nullptr || next_ids == nullptr || positions == nullptr || ring == nullptr ||
        head == nullptr)
        return ARC_E_NULL;
    if (B <= 0 || V <= 0 || max_position <= 0 || capacity == 0 || static_cast<uint64_t>(B) > capacity ||
        capacity > ARC_RING_MAX_CAPACITY)
        return ARC_E_SHAPE;
    if (reinterpret_cast<uintptr_t>(ring) % 8 != 0 || reinterpret_cast<uintptr_t>(head) % 8 != 0) return ARC_E_ALIGN;
    CommitArgs a{tokens, B, V, next_ids, positions, max_position, owners, ring, capacity, head, fault_word};
    commit_kernel<<<1, kCommitThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
    return cudaGetLastError() == cudaSuccess ? ARC_OK : ARC_E_CUDA;
}

int64_t arc_ring_drain(const arc_commit_record* ring, uint32_t capacity, uint64_t first, int64_t count,
                       arc_commit_record* out, uint64_t max_spins) {
    if (ring == nullptr || out == nullptr) return ARC_E_NULL;
    if (capacity == 0 || count < 0) return ARC_E_SHAPE;
    for (int64_t i = 0; i < count; ++i) {
        const uint64_t idx = first + static_cast<uint64_t>(i);
        const uint64_t* w = reinterpret_cast<const uint64_t*>(ring + (idx % capacity));
        const uint32_t want = static_cast<uint32_t>(idx + 1);
        uint64_t spins = 0;
        uint64_t v[3];
        while (true) {
            // each word is one device store; all three with the wanted stamp
            // are one record
            bool all = true, overrun = false;
            for (int k = 0; k < 3; ++k) {
                v[k] = __atomic_load_n(w + k, __ATOMIC_ACQUIRE);
                const uint32_t stamp = static_cast<uint32_t>(v[k] >> 32);
                all = all && stamp == want;
                // a stamp ahead of the wanted one (modulo 2^32) is a later lap
                // of the ring: the wanted record was (or is being) overwritten
                const uint32_t ahead = stamp - want;
                overrun = overrun || (stamp != 0 && ahead != 0 && ahead < 0x80000000u);
            }
            if (all) break;
            if (overrun) return ARC_E_RING_OVERRUN;
            if (++spins > max_spins) return i;
        }
        out[i].token = static_cast<int32_t>(static_cast<uint32_t>(v[0]));
        out[i].stamp = want;
        out[i].position = static_cast<int32_t>(static_cast<uint32_t>(v[1]));
        out[i].stamp_pos = want;
        out[i].owner = static_cast<uint32_t>(v[2]);
        out[i].stamp_owner = want;
    }
    return count;
}

int arc_stream_idle(void* stream) {
    const cudaError_t e = cudaStreamQuery(static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) return 1;
    if (e == cudaErrorNotReady) return 0;
    return ARC_E_CUDA;
}

int arc_ring_alloc(size_t bytes, void** host, void** device) {
    if (host == nullptr || device == nullptr || bytes == 0) return ARC_E_NULL;
    *host = nullptr;
    *device = nullptr;
    void* h = nullptr;
    if (cudaHostAlloc(&h, bytes, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) return ARC_E_CUDA;
    void* d = nullptr;
    if (cudaHostGetDevicePointer(&d, h, 0) != cudaSuccess) {
        cudaFreeHost(h);
        return ARC_E_CUDA;
    }
    for (size_t i = 0; i < bytes; ++i) static_cast<volatile unsigned char*>(h)[i] = 0;
    *host = h;
    *device = d;
    return ARC_OK;
}

int arc_ring_free(void* host) {
    if (host == nullptr) return ARC_E_NULL;
    return cudaFreeHost(host) == cudaSuccess ? ARC_OK : ARC_E_CUDA;
}

}  // extern "C"
