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
// that device reuse it. Make that first call before any stream capture begins.
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

struct DevScratch {
    std::once_flag once;
    void* ptr = nullptr;
    cudaError_t err = cudaSuccess;
};
DevScratch g_dev[64];

int scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_mla_decode_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= 64)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_sparse_mla_decode_noalloc: device %d >= 64", dev);
    DevScratch& d = g_dev[dev];
    std::call_once(d.once, [&d]() {
        // Host code sees g_scratch only as a stand-in symbol; the device address of
        // this device's copy comes from the runtime.
        d.err = cudaGetSymbolAddress(&d.ptr, g_scratch);
    });
    if (d.err != cudaSuccess)
        return cuda_fail(d.err, "dsa_sparse_mla_decode_noalloc: cudaGetSymbolAddress");
    *out = d.ptr;
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
