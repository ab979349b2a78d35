// Shared device and host helpers of libdsa (sm_103a).
#pragma once

#include <cuda.h>  // CUtensorMap (types only; the encoder is fetched at run time)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "dsa.h"

namespace dsa {

// ---------------------------------------------------------------------------
// Host side: error state and launch bookkeeping (defined in api.cu).

int fail(int code, const char* fmt, ...);  // records the message, returns code
int cuda_fail(cudaError_t e, const char* what);
int sm_count();                            // SMs of the current device (cached)
int set_max_smem(const void* kernel, int bytes);  // once per (device, kernel)

// Programmatic dependent launch. Every kernel of the library is launched as a
// programmatic dependent of the work before it on the stream, and waits for that
// work (pdl_wait) before it reads anything that work may have written; the only
// earlier reads are of weights (the projection's first ring of o_absorb boxes).
// Two kernels let their dependents start early (pdl_trigger): the split combine, so
// that the projection fetches o_absorb meanwhile, and the front-end norm kernel,
// ahead of the q GEMM. Elsewhere, dependent blocks waiting beside a running grid
// slowed it. dsa_set_option(DSA_OPT_PDL, 0) turns the attribute off (the wait then
// returns at once).
// Bytes of [p, p + bytes), from p on, that the last dsa_prefetch_l2 on this device
// staged in L2 at evict_last priority (0 if p is outside that range).
size_t l2_staged_overlap(const void* p, size_t bytes);
bool pdl_enabled();
int mla_kernel_choice();     // DSA_OPT_MLA_KERNEL
int select_kernel_choice();  // DSA_OPT_SELECT_KERNEL
int project_kernel_choice();  // DSA_OPT_PROJECT_KERNEL
int take_inject_stall();      // DSA_OPT_INJECT_STALL, reset to 0 by the taking
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Kernel-side copy of dsa_paging.
struct Paging {
    const int32_t* seq_lens;
    const int32_t* block_table;
    long long num_blocks;
    int batch;
    int max_seq_len;
    int max_blocks;
    int block_size;
};

int check_paging(const dsa_paging* pg, int kpool, Paging* out);

// 2-D tiled tensor map over a row-major [outer, inner] array (zero fill out of
// bounds), boxes of box_inner x box_outer elements, stored in shared memory with the
// given swizzle (128-byte swizzle: box_inner x element size must be 128 bytes).
int make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                 uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                 CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE);

// The o_absorb projection (project.cu), a skinny GEMM: y[r] = bf16(A . x[r]), x bf16 or
// f32, A [hidden, K] bf16. With yf the sums are stored as f32 there instead of y; with
// y2, output columns from `split` (a multiple of 64) on go to y2 [rows, hidden - split]
// and y is [rows, split].
bool project_supported(int K, int hidden);
// The tensor-core form (project_tc.cu): hidden a multiple of 128, K of 512.
bool project_tc_supported(int K, int hidden);
// f32 x is rounded to bf16 into the workspace first (project_tc_convert_bytes).
size_t project_tc_convert_bytes(int rows, int K);
int project_tc_launch(const void* x, bool x_f32, int rows, int K, const uint16_t* A, int hidden,
                      uint16_t* y, int32_t* status, void* ws, size_t ws_bytes, cudaStream_t st,
                      float* yf, uint16_t* y2, int split);
size_t project_workspace_bytes(int rows, int K, int hidden, int sms);
int project_launch(const void* x, bool x_f32, int rows, int K, const uint16_t* A, int hidden,
                   uint16_t* y, int32_t* status, void* ws, size_t ws_bytes, cudaStream_t st,
                   float* yf = nullptr, uint16_t* y2 = nullptr, int split = 0);

// Sparse latent attention on the tensor cores (mla_tc.cu): the split kernel of
// dsa_sparse_mla_decode for 64 heads (large batches, or forced by DSA_OPT_MLA_KERNEL). Writes the splits' partials
// (ns > 1) or olat / its bf16 copy (ns == 1) in the same layout as the mma.sync split
// kernel.
struct MlaTcParams {
    const uint16_t* qlat;
    const int32_t* row_seq;
    const uint16_t* ckv;
    const uint8_t* ckv8;     // non-null: the FP8 cache (E4M3 codes [.., 512]) is read instead
    const float* ckv_scale;  // ... with its power-of-two scales [.., 4]
    const int32_t* token_ids;
    float* part_o;
    float* part_ml;
    float* olat;
    uint16_t* xbf;
    int32_t* status;
    Paging pg;
    int rows;
    int ow;
    int ns;
    int tps;
    float sl2;  // softmax_scale * log2(e)
};
bool mla_tc_supported(int heads, int kv_lora_rank);
int mla_tc_chunk();  // tokens per chunk: split sizes are rounded to it
int mla_tc_launch(const MlaTcParams& a, long long ckv_rows, cudaStream_t st);
// The decode kernel (mla_dec.cu): 64 heads, a row's selected tokens spread over CTAs
// (mla_dec_plan: CTAs per row, tokens per CTA, and whether the row's CTAs form a
// cluster that merges its partials into olat / xbf; otherwise the partials in
// part_o / part_ml go to the combine kernel).
bool mla_dec_supported(int heads, int kv_lora_rank, int ow);
void mla_dec_plan(int ow, int* cs, int* tps, bool* merge);  // merge: in the kernel
int mla_dec_launch(const MlaTcParams& a, long long ckv_rows, cudaStream_t st);

// ---------------------------------------------------------------------------
// Device side.

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float round_bf16(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint4 ldg16(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

// 16-byte load that bypasses L1 allocation: for data streamed exactly once.
__device__ __forceinline__ uint4 ldg16_stream(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// D += A * B, m16n8k16, bf16 inputs, f32 accumulate (warp-wide).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// 16-byte async copy global -> shared; src_bytes == 0 zero-fills without reading.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
// L2 eviction-priority policy for the cache_hint copy forms below: data read once
// per call (the o_absorb stream) is loaded evict_first, so it does not push out
// lines staged in L2 for later use.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
    return p;
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ---- programmatic dependent launch -------------------------------------------

// Blocks until the grids this one depends on have completed and their memory is
// visible (returns at once when launched without the attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
// Lets the next kernel on the stream (a programmatic dependent) start its blocks now;
// it still waits in pdl_wait() until this grid has completed.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// ---- mbarrier + bulk async copy (TMA engine, non-tensor form) ----------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// As mbar_try_wait, but a thread whose phase is not complete is suspended in
// hardware until it completes or about hint_ns nanoseconds pass, instead of
// returning at once (a waiting warp then takes no issue slots).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity,
                                                    uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase of `bar` with the given parity; gives up after ~1 s and
// returns false (the caller flags DSA_STATUS_TIMEOUT and winds down).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0u && global_ns() - t0 > 1000000000ull) return false;
    }
}
// Bulk copy global -> this CTA's shared memory, completing `bytes` on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// Tiled 2-D tensor copy global -> this CTA's shared memory (box at inner coordinate
// x, outer coordinate y), completing its bytes on `bar`. x * element size must be a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
// tma_load_2d with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ uint4 lds16(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr));
    return r;
}

__device__ __forceinline__ void flag_status(int32_t* status, int bits) {
    if (status) atomicOr(status, bits);
}

// Physical row of token t of sequence b in a token cache (-1: bad block entry).
__device__ __forceinline__ long long token_row(const Paging& pg, int b, int t) {
    if (pg.block_table == nullptr) return (long long)b * pg.max_seq_len + t;
    int blk = __ldg(pg.block_table + (long long)b * pg.max_blocks + t / pg.block_size);
    if (blk < 0 || blk >= pg.num_blocks) return -1;
    return (long long)blk * pg.block_size + t % pg.block_size;
}

// Physical row of pool p of sequence b in a pooled-key cache (-1: bad block entry).
__device__ __forceinline__ long long pool_row(const Paging& pg, int b, int p, int kpool) {
    if (pg.block_table == nullptr) return (long long)b * (pg.max_seq_len / kpool) + p;
    int ppb = pg.block_size / kpool;
    int blk = __ldg(pg.block_table + (long long)b * pg.max_blocks + p / ppb);
    if (blk < 0 || blk >= pg.num_blocks) return -1;
    return (long long)blk * ppb + p % ppb;
}

// Tokens a sequence can hold in its cache.
__device__ __forceinline__ int seq_capacity(const Paging& pg) {
    return pg.block_table == nullptr ? pg.max_seq_len : pg.max_blocks * pg.block_size;
}

}  // namespace dsa
