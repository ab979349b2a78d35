// dsa_prefetch_l2: stage a read-only range (a layer's weights) in L2 ahead of its
// use. A decode step's top-k and gather stages are latency-bound and leave HBM
// mostly idle; a prefetch issued beside them (another stream, or a parallel branch
// of a graph) moves the first part of the o_absorb stream out of the projection's
// critical path.
//
// The staged lines carry the evict_last priority so that the latent rows gathered
// in between do not push them out. The projection that reads them puts them back to
// normal priority (applypriority) once consumed: the library remembers the last
// staged range per device, and a projection whose o_absorb overlaps it demotes the
// overlap. Lines left at evict_last would otherwise outlive the step and hold L2
// against everything after it.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "dsa.h"

namespace dsa {
namespace {

constexpr unsigned kChunk = 16 * 1024;  // bytes per bulk prefetch

// Each lane issues whole chunks, grid-stride; the tail chunk is shorter. Nothing is
// written and nothing waits: the bulk prefetch is a hint the memory system may drop.
__global__ void __launch_bounds__(32) prefetch_l2_kernel(const char* p, unsigned long long bytes) {
    // evict_last: the staged lines should outlive the gather traffic that passes
    // through L2 before the projection reads them
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(policy));
    const unsigned long long n = (bytes + kChunk - 1) / kChunk;
    for (unsigned long long i = blockIdx.x * 32ull + threadIdx.x; i < n;
         i += (unsigned long long)gridDim.x * 32ull) {
        const unsigned long long off = i * kChunk;
        const unsigned long long left = bytes - off;
        const unsigned sz = left < kChunk ? (unsigned)left : kChunk;
        asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p + off),
                     "r"(sz), "l"(policy)
                     : "memory");
    }
}

struct Staged {
    const char* p = nullptr;
    size_t bytes = 0;
};
std::mutex g_staged_mu;
Staged g_staged[64];

}  // namespace

size_t l2_staged_overlap(const void* p, size_t bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lk(g_staged_mu);
    const Staged& s = g_staged[dev];
    const char* q = static_cast<const char*>(p);
    if (!s.p || q < s.p || q >= s.p + s.bytes) return 0;
    return std::min(bytes, (size_t)(s.p + s.bytes - q));
}

}  // namespace dsa

using namespace dsa;

extern "C" int dsa_prefetch_l2(const void* ptr, size_t bytes, void* stream) {
    if (bytes == 0) return DSA_OK;
    if (!ptr) return fail(DSA_ERR_INVALID_ARG, "dsa_prefetch_l2: NULL pointer");
    if (((uintptr_t)ptr) & 15)
        return fail(DSA_ERR_INVALID_ARG, "dsa_prefetch_l2: pointer not 16-byte aligned");
    bytes &= ~(size_t)15;  // the bulk prefetch moves whole 16-byte units
    if (bytes == 0) return DSA_OK;
    const unsigned long long chunks = (bytes + kChunk - 1) / kChunk;
    const int blocks = (int)std::min<unsigned long long>((chunks + 31) / 32, (unsigned long long)sm_count());
    prefetch_l2_kernel<<<blocks, 32, 0, (cudaStream_t)stream>>>((const char*)ptr,
                                                                 (unsigned long long)bytes);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "dsa_prefetch_l2 launch");
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
        std::lock_guard<std::mutex> lk(g_staged_mu);
        g_staged[dev].p = static_cast<const char*>(ptr);
        g_staged[dev].bytes = bytes;
    }
    return DSA_OK;
}
