// Decode-time append and the geometry derived from the live sequence lengths.
//
// Page: metrale_model_arch/glm5next_dsa/mod.rs, Glm5NextDsaKernels (`indexer_store`,
// `write_geom`). The new token's indexer row is placed at a position the device
// reads (the live length), flagged valid, and the selector's per-row geometry is
// recomputed on the device from the lengths: no host value changes between steps,
// which is what lets one captured graph serve every step.
//
// dsa_indexer_store: one CTA per sequence. The position is the sequence's current
// length, read on the device; the rows go there through the cache layout, the
// token is marked valid, and the length grows by one. Nothing on the host depends
// on the length, so a graph holding this launch appends one token per replay.
//
// dsa_write_geom: row r's context length is its sequence's current length.
#include "common.cuh"
#include "store.cuh"

namespace dsa {
namespace {

constexpr int kStoreThreads = 128;

struct StoreArgs {
    const uint16_t* k_new;
    const uint16_t* gate_new;
    const uint16_t* ckv_new;  // nullable (with ckv)
    uint16_t* k_raw;
    uint16_t* gate;
    uint8_t* valid;
    uint16_t* ckv;
    int32_t* seq_lens;  // the paging descriptor's lengths, advanced here
    int32_t* status;
    Paging pg;
    int ihd;
    int kvl;
};

__global__ void __launch_bounds__(kStoreThreads) indexer_store_kernel(StoreArgs a) {
    pdl_wait();
    __shared__ long long s_row;
    __shared__ int s_t;
    const int b = blockIdx.x;
    if (threadIdx.x == 0) s_row = next_token_row(a.pg, a.seq_lens, b, &s_t, a.status);
    __syncthreads();
    const long long row = s_row;
    if (row < 0) return;
    store_token_rows(a.k_new, a.gate_new, a.ckv_new, a.k_raw, a.gate, a.valid, a.ckv, b, row,
                     a.ihd, a.kvl);
    __syncthreads();  // every thread has used s_t's position before the length moves
    if (threadIdx.x == 0) a.seq_lens[b] = s_t + 1;
}

__global__ void write_geom_kernel(const int32_t* __restrict__ seq_lens, int batch,
                                  const int32_t* __restrict__ row_seq, int rows,
                                  int32_t* __restrict__ row_ctx, int32_t* status) {
    pdl_wait();
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += gridDim.x * blockDim.x) {
        const int b = row_seq ? row_seq[r] : r;
        int L = 0;
        if (b < 0 || b >= batch)
            flag_status(status, DSA_STATUS_BAD_TOKEN);
        else
            L = seq_lens[b];
        row_ctx[r] = L;
    }
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" int dsa_indexer_store(const dsa_bf16* k_new, const dsa_bf16* gate_new,
                                 const dsa_bf16* ckv_new, int ihd, int kv_lora_rank,
                                 const dsa_paging* pg, int32_t* seq_lens, dsa_bf16* k_raw,
                                 dsa_bf16* gate, uint8_t* token_valid, dsa_bf16* ckv,
                                 int32_t* status, void* stream) {
    if (ihd != 64 && ihd != 128)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_indexer_store: index_head_dim %d not in {64, 128}",
                    ihd);
    if ((ckv == nullptr) != (ckv_new == nullptr))
        return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_store: ckv and ckv_new go together");
    if (ckv && (kv_lora_rank < 8 || kv_lora_rank % 8 != 0))
        return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_store: kv_lora_rank %d not a multiple of 8",
                    kv_lora_rank);
    Paging P;
    int rc = check_paging(pg, 0, &P);
    if (rc) return rc;
    if (!seq_lens || seq_lens != pg->seq_lens)
        return fail(DSA_ERR_INVALID_ARG,
                    "dsa_indexer_store: seq_lens must be the descriptor's (writable) lengths");
    if (!k_new || !gate_new || !k_raw || !gate || !token_valid)
        return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_store: NULL tensor");
    if ((((uintptr_t)k_new) | ((uintptr_t)gate_new) | ((uintptr_t)ckv_new) | ((uintptr_t)k_raw) |
         ((uintptr_t)gate) | ((uintptr_t)ckv)) & 15)
        return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_store: rows must be 16-byte aligned");
    StoreArgs a;
    a.k_new = k_new;
    a.gate_new = gate_new;
    a.ckv_new = ckv_new;
    a.k_raw = k_raw;
    a.gate = gate;
    a.valid = token_valid;
    a.ckv = ckv;
    a.seq_lens = seq_lens;
    a.status = status;
    a.pg = P;
    a.ihd = ihd;
    a.kvl = kv_lora_rank;
    cudaError_t e = launch_pdl(indexer_store_kernel, dim3((unsigned)P.batch), dim3(kStoreThreads),
                               0, (cudaStream_t)stream, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "dsa_indexer_store launch");
    return DSA_OK;
}

extern "C" int dsa_write_geom(const int32_t* seq_lens, int batch, const int32_t* row_seq,
                              int rows, int32_t* row_ctx, int32_t* status, void* stream) {
    if (batch < 1 || rows < 0)
        return fail(DSA_ERR_INVALID_ARG, "dsa_write_geom: batch %d, rows %d", batch, rows);
    if (rows == 0) return DSA_OK;
    if (!seq_lens || !row_ctx) return fail(DSA_ERR_INVALID_ARG, "dsa_write_geom: NULL tensor");
    const int threads = 128;
    const int blocks = (rows + threads - 1) / threads;
    cudaError_t e = launch_pdl(write_geom_kernel, dim3((unsigned)blocks), dim3(threads), 0,
                               (cudaStream_t)stream, seq_lens, batch, row_seq, rows, row_ctx,
                               status);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "dsa_write_geom launch");
    return DSA_OK;
}
