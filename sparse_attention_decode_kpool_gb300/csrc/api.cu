// Host-side core of libdsa: error reporting, geometry rules, paging checks, and
// dsa_expand (expand_selection).
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>
#include <set>
#include <utility>

#include "common.cuh"

namespace dsa {

static thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(DSA_ERR_CUDA, "%s: CUDA error %d (%s)", what, (int)e, cudaGetErrorString(e));
}

int sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) {
        int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

int set_max_smem(const void* kernel, int bytes) {
    static std::mutex mu;
    static std::set<std::pair<int, std::pair<const void*, int>>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(mu);
    auto key = std::make_pair(dev, std::make_pair(kernel, bytes));
    if (done.count(key)) return DSA_OK;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    done.insert(key);
    return DSA_OK;
}

// Process-wide launch options (dsa_set_option); read by the launch code, never from
// the environment.
static std::atomic<int> g_opt_pdl{1};
static std::atomic<int> g_opt_mla_kernel{DSA_MLA_KERNEL_AUTO};
static std::atomic<int> g_opt_select_kernel{DSA_SELECT_KERNEL_MERGE};
static std::atomic<int> g_opt_project_kernel{DSA_PROJECT_KERNEL_AUTO};
static std::atomic<int> g_opt_inject_stall{0};

bool pdl_enabled() { return g_opt_pdl.load(std::memory_order_relaxed) != 0; }

int mla_kernel_choice() { return g_opt_mla_kernel.load(std::memory_order_relaxed); }

int select_kernel_choice() { return g_opt_select_kernel.load(std::memory_order_relaxed); }

int project_kernel_choice() { return g_opt_project_kernel.load(std::memory_order_relaxed); }

int take_inject_stall() { return g_opt_inject_stall.exchange(0, std::memory_order_relaxed); }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                 uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                 CUtensorMapSwizzle swizzle) {
    static std::once_flag once;
    static EncodeTiledFn encode = nullptr;
    std::call_once(once, []() {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    if (!encode) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return DSA_OK;
}

int check_paging(const dsa_paging* pg, int kpool, Paging* out) {
    if (!pg) return fail(DSA_ERR_INVALID_ARG, "paging descriptor is NULL");
    if (pg->batch < 1) return fail(DSA_ERR_INVALID_ARG, "paging: batch %d < 1", pg->batch);
    if (pg->max_seq_len < 0)
        return fail(DSA_ERR_INVALID_ARG, "paging: max_seq_len %d < 0", pg->max_seq_len);
    if (!pg->seq_lens) return fail(DSA_ERR_INVALID_ARG, "paging: seq_lens is NULL");
    if (pg->block_table) {
        if (pg->block_size < 1 || pg->max_blocks < 1 || pg->num_blocks < 1)
            return fail(DSA_ERR_INVALID_ARG,
                        "paging: block_size %d, max_blocks %d, num_blocks %lld must be >= 1",
                        pg->block_size, pg->max_blocks, (long long)pg->num_blocks);
        if ((long long)pg->max_blocks * pg->block_size < pg->max_seq_len)
            return fail(DSA_ERR_INVALID_ARG,
                        "paging: max_blocks*block_size %lld < max_seq_len %d",
                        (long long)pg->max_blocks * pg->block_size, pg->max_seq_len);
        if (kpool > 0 && pg->block_size % kpool != 0)
            return fail(DSA_ERR_UNSUPPORTED, "paging: block_size %d is not a multiple of kpool %d",
                        pg->block_size, kpool);
    }
    out->seq_lens = pg->seq_lens;
    out->block_table = pg->block_table;
    out->num_blocks = pg->num_blocks;
    out->batch = pg->batch;
    out->max_seq_len = pg->max_seq_len;
    out->max_blocks = pg->max_blocks;
    out->block_size = pg->block_size;
    return DSA_OK;
}

// ---------------------------------------------------------------------------
// dsa_expand / dsa_expand_tail: one thread per output slot; each slot written
// exactly once. With row_ctx, positions tail_at + i hold the row's trailing
// partial-pool tokens [t0, L), t0 = first_key + kpool * floor((L - first_key) / kpool).

__global__ void expand_kernel(const int32_t* __restrict__ pool_ids, int rows, int sk,
                              int first_key, int kpool, int out_width,
                              const int32_t* __restrict__ row_ctx, int tail_at,
                              int32_t* __restrict__ token_ids) {
    pdl_wait();
    long long n = (long long)rows * out_width;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        int r = (int)(i / out_width);
        int j = (int)(i % out_width);
        int slot = j / kpool;
        int v = -1;
        if (slot < sk) {
            int p = __ldg(pool_ids + (long long)r * sk + slot);
            if (p >= 0) v = first_key + p * kpool + (j - slot * kpool);
        } else if (row_ctx && j >= tail_at) {
            const int L = __ldg(row_ctx + r);
            const int t0 = first_key + (L > first_key ? (L - first_key) / kpool * kpool : 0);
            const int t = t0 + (j - tail_at);
            if (t < L) v = t;
        }
        token_ids[i] = v;
    }
}

int expand_launch(const int32_t* pool_ids, int rows, int sk, int first_key, int kpool,
                  int out_width, const int32_t* row_ctx, int tail_at, int32_t* token_ids,
                  void* stream, const char* name) {
    long long n = (long long)rows * out_width;
    int threads = 256;
    long long blocks = (n + threads - 1) / threads;
    int cap = sm_count() * 8;
    if (cap < 1) cap = 1024;
    if (blocks > cap) blocks = cap;
    cudaError_t e = launch_pdl(expand_kernel, dim3((unsigned)blocks), dim3(threads), 0,
                               (cudaStream_t)stream, pool_ids, rows, sk, first_key, kpool,
                               out_width, row_ctx, tail_at, token_ids);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, name);
    return DSA_OK;
}

}  // namespace dsa

using namespace dsa;

extern "C" {

const char* dsa_last_error(void) { return g_err; }

int dsa_abi_version(void) { return DSA_ABI_VERSION; }

int dsa_set_option(int option, int value) {
    switch (option) {
        case DSA_OPT_PDL:
            if (value != 0 && value != 1)
                return fail(DSA_ERR_INVALID_ARG, "dsa_set_option: DSA_OPT_PDL takes 0 or 1, not %d",
                            value);
            g_opt_pdl.store(value, std::memory_order_relaxed);
            return DSA_OK;
        case DSA_OPT_MLA_KERNEL:
            if (value != DSA_MLA_KERNEL_AUTO && value != DSA_MLA_KERNEL_TCGEN05 &&
                value != DSA_MLA_KERNEL_MMA && value != DSA_MLA_KERNEL_CLUSTER)
                return fail(DSA_ERR_INVALID_ARG,
                            "dsa_set_option: DSA_OPT_MLA_KERNEL takes 0 to 3, not %d", value);
            g_opt_mla_kernel.store(value, std::memory_order_relaxed);
            return DSA_OK;
        case DSA_OPT_SELECT_KERNEL:
            if (value != DSA_SELECT_KERNEL_MERGE && value != DSA_SELECT_KERNEL_RADIX)
                return fail(DSA_ERR_INVALID_ARG,
                            "dsa_set_option: DSA_OPT_SELECT_KERNEL takes 0 or 1, not %d", value);
            g_opt_select_kernel.store(value, std::memory_order_relaxed);
            return DSA_OK;
        case DSA_OPT_PROJECT_KERNEL:
            if (value != DSA_PROJECT_KERNEL_AUTO && value != DSA_PROJECT_KERNEL_TCGEN05 &&
                value != DSA_PROJECT_KERNEL_MMA)
                return fail(DSA_ERR_INVALID_ARG,
                            "dsa_set_option: DSA_OPT_PROJECT_KERNEL takes 0, 1 or 2, not %d", value);
            g_opt_project_kernel.store(value, std::memory_order_relaxed);
            return DSA_OK;
        case DSA_OPT_INJECT_STALL:
            if (value != 0 && value != 1)
                return fail(DSA_ERR_INVALID_ARG,
                            "dsa_set_option: DSA_OPT_INJECT_STALL takes 0 or 1, not %d", value);
            g_opt_inject_stall.store(value, std::memory_order_relaxed);
            return DSA_OK;
        default:
            return fail(DSA_ERR_INVALID_ARG, "dsa_set_option: unknown option %d", option);
    }
}

int dsa_get_option(int option) {
    switch (option) {
        case DSA_OPT_PDL: return g_opt_pdl.load(std::memory_order_relaxed);
        case DSA_OPT_MLA_KERNEL: return g_opt_mla_kernel.load(std::memory_order_relaxed);
        case DSA_OPT_SELECT_KERNEL: return g_opt_select_kernel.load(std::memory_order_relaxed);
        case DSA_OPT_PROJECT_KERNEL: return g_opt_project_kernel.load(std::memory_order_relaxed);
        case DSA_OPT_INJECT_STALL: return g_opt_inject_stall.load(std::memory_order_relaxed);
        default: return -1;
    }
}

int dsa_validate_config(int index_kpool, int index_topk, int kv_lora_rank, int local_heads) {
    if (index_kpool <= 0 || index_topk <= 0)
        return fail(DSA_ERR_CONFIG, "DSA needs index_kpool > 0 and index_topk > 0 (got %d, %d)",
                    index_kpool, index_topk);
    if (index_topk % index_kpool != 0)
        return fail(DSA_ERR_CONFIG,
                    "index_topk %d is not a multiple of index_kpool %d: the pool budget is "
                    "index_topk / index_kpool",
                    index_topk, index_kpool);
    if (index_kpool > DSA_MAX_KPOOL)
        return fail(DSA_ERR_UNSUPPORTED,
                    "index_kpool %d exceeds the %d slots dsa_compress pools; refused instead of "
                    "pooling only the first slots",
                    index_kpool, DSA_MAX_KPOOL);
    if (kv_lora_rank == 0) return fail(DSA_ERR_CONFIG, "MLA needs kv_lora_rank > 0");
    if (kv_lora_rank != DSA_KV_LORA_RANK)
        return fail(DSA_ERR_UNSUPPORTED,
                    "kv_lora_rank %d: the attention kernels are built for a %d-wide latent",
                    kv_lora_rank, DSA_KV_LORA_RANK);
    if (local_heads <= 0) return fail(DSA_ERR_CONFIG, "zero attention heads (local_heads %d)",
                                      local_heads);
    return DSA_OK;
}

int dsa_select_k(int index_topk, int kpool, int n_pools) {
    if (index_topk <= 0 || kpool <= 0 || n_pools < 0) return -1;
    int k = index_topk / kpool;
    return k < n_pools ? k : n_pools;
}

int dsa_expand(const int32_t* pool_ids, int rows, int sk, int first_key, int kpool,
               int out_width, int32_t* token_ids, void* stream) {
    if (rows < 0 || sk < 0 || first_key < 0 || kpool < 1 || out_width < 0)
        return fail(DSA_ERR_INVALID_ARG,
                    "dsa_expand: rows %d, sk %d, first_key %d, kpool %d, out_width %d", rows, sk,
                    first_key, kpool, out_width);
    if ((long long)sk * kpool > out_width)
        return fail(DSA_ERR_INVALID_ARG, "dsa_expand: out_width %d < sk*kpool %lld", out_width,
                    (long long)sk * kpool);
    if (rows == 0 || out_width == 0) return DSA_OK;
    if (!token_ids || (sk > 0 && !pool_ids))
        return fail(DSA_ERR_INVALID_ARG, "dsa_expand: NULL tensor");
    return expand_launch(pool_ids, rows, sk, first_key, kpool, out_width, nullptr, out_width,
                         token_ids, stream, "dsa_expand launch");
}

int dsa_expand_tail(const int32_t* pool_ids, int rows, int sk, int first_key, int kpool,
                    int index_topk, const int32_t* row_ctx, int out_width, int32_t* token_ids,
                    void* stream) {
    if (rows < 0 || sk < 0 || first_key < 0 || kpool < 1 || index_topk < 0 || out_width < 0)
        return fail(DSA_ERR_INVALID_ARG,
                    "dsa_expand_tail: rows %d, sk %d, first_key %d, kpool %d, index_topk %d, "
                    "out_width %d",
                    rows, sk, first_key, kpool, index_topk, out_width);
    if ((long long)sk * kpool > index_topk)
        return fail(DSA_ERR_INVALID_ARG, "dsa_expand_tail: sk*kpool %lld > index_topk %d",
                    (long long)sk * kpool, index_topk);
    if ((long long)index_topk + kpool - 1 > out_width)
        return fail(DSA_ERR_INVALID_ARG,
                    "dsa_expand_tail: out_width %d < index_topk + kpool - 1 = %lld", out_width,
                    (long long)index_topk + kpool - 1);
    if (rows == 0 || out_width == 0) return DSA_OK;
    if (!token_ids || !row_ctx || (sk > 0 && !pool_ids))
        return fail(DSA_ERR_INVALID_ARG, "dsa_expand_tail: NULL tensor");
    return expand_launch(pool_ids, rows, sk, first_key, kpool, out_width, row_ctx, index_topk,
                         token_ids, stream, "dsa_expand_tail launch");
}

}  // extern "C"
