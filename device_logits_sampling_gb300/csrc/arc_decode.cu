// The decode-loop commit (arc_decode.h): one small kernel after the sampler,
// and the host side of the ring it publishes into.
#include <cuda_runtime.h>

#include <atomic>
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
        const arc_commit_record* rec = ring + (idx % capacity);
        const uint32_t want = static_cast<uint32_t>(idx + 1);
        uint64_t spins = 0;
        uint32_t stamp;
        while (true) {
            stamp = __atomic_load_n(&rec->stamp, __ATOMIC_ACQUIRE);
            if (stamp == want) break;
            // a stamp ahead of the wanted one (modulo 2^32) is a later lap of
            // the ring: the wanted record was overwritten
            const uint32_t ahead = stamp - want;
            if (stamp != 0 && ahead != 0 && ahead < 0x80000000u) return ARC_E_RING_OVERRUN;
            if (++spins > max_spins) return i;
        }
        out[i].token = __atomic_load_n(&rec->token, __ATOMIC_RELAXED);
        out[i].position = __atomic_load_n(&rec->position, __ATOMIC_RELAXED);
        out[i].owner = __atomic_load_n(&rec->owner, __ATOMIC_RELAXED);
        out[i].stamp = stamp;
        // the slot may be rewritten by a later lap while being read: a writer
        // replaces the stamp before it touches the fields (see commit_kernel),
        // so the stamp read again after the fields confirms the copy
        std::atomic_thread_fence(std::memory_order_acquire);
        if (__atomic_load_n(&rec->stamp, __ATOMIC_RELAXED) != want) return ARC_E_RING_OVERRUN;
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
