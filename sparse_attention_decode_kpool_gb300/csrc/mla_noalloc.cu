// dsa_sparse_mla_decode_noalloc: dsa_sparse_mla_decode with its scratch in a fixed
// device array of this library instead of a caller-provided workspace.
//
// Some callers cannot hand us a workspace: a host framework that owns every device
// allocation and gives plug-in code no allocator, or a latency-critical loop that
// must never call cudaMalloc/cudaFree (both may synchronise the device). For them
// the scratch is a file-scope static __device__ array, sized once at build time and
// held by every GPU that loads this code until the process exits.
//
// Set-up: the first call on each device, with that device current, looks up the
// array's device address with cudaGetSymbolAddress and caches it; later calls on
// that device reuse it. Make that first call before any stream capture begins (if
// the lookup fails, the call returns DSA_ERR_CUDA and a later call looks again).
//
// Sharing: every call uses the same array, which keeps the previous call's
// contents. Nothing in it needs to start at zero (each call writes every scratch
// value it reads), but two calls whose GPU work overlaps in time -- on different
// streams, or from different host threads -- race on the array and corrupt each
// other's results. Serialise them.
#include <mutex>

#include "common.cuh"

constexpr size_t kNoAllocScratchBytes = DSA_NOALLOC_SCRATCH_BYTES;

// The scratch itself: one copy per device that loads this code.
static __device__ __align__(256) uint8_t g_scratch[kNoAllocScratchBytes];

namespace dsa {
namespace {

// Device address of g_scratch per device, filled by the first call on that device
// whose lookup succeeds. A failed lookup (for instance a first call made during a
// stream capture) is not remembered: the next call tries again.
std::mutex g_mu;
void* g_ptr[64] = {};

int scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_mla_decode_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= 64)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_sparse_mla_decode_noalloc: device %d >= 64", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_ptr[dev]) {
        // Host code sees g_scratch only as a stand-in symbol; the device address of
        // this device's copy comes from the runtime.
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess) {
            cudaGetLastError();  // leave no sticky launch error behind
            return cuda_fail(e, "dsa_sparse_mla_decode_noalloc: cudaGetSymbolAddress");
        }
        g_ptr[dev] = p;
    }
    *out = g_ptr[dev];
    return DSA_OK;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" int dsa_sparse_mla_decode_noalloc(const dsa_bf16* qlat, int rows, int heads,
                                             int kv_lora_rank, const int32_t* row_seq,
                                             const dsa_bf16* ckv, const dsa_paging* pg,
                                             const int32_t* token_ids, int out_width,
                                             float softmax_scale, const dsa_bf16* o_absorb,
                                             int hidden, dsa_bf16* y, float* olat,
                                             int32_t* status, void* stream) {
    size_t need = 0;
    int rc = dsa_sparse_mla_decode_workspace(rows, heads, kv_lora_rank, out_width, hidden,
                                             o_absorb != nullptr, &need);
    if (rc) return rc;
    if (need > kNoAllocScratchBytes)
        return fail(DSA_ERR_UNSUPPORTED,
                    "dsa_sparse_mla_decode_noalloc: this problem needs %zu B of scratch, more than "
                    "the fixed %zu B array; use dsa_sparse_mla_decode with a workspace",
                    need, kNoAllocScratchBytes);
    void* ws = nullptr;
    rc = scratch_for_current_device(&ws);
    if (rc) return rc;
    return dsa_sparse_mla_decode(qlat, rows, heads, kv_lora_rank, row_seq, ckv, pg, token_ids,
                                 out_width, softmax_scale, o_absorb, hidden, y, olat, status, ws,
                                 kNoAllocScratchBytes, stream);
}
