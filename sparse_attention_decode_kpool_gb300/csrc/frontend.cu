// dsa_frontend: the layer's step inputs from the hidden state.
//
// Page: metrale_model_arch/glm5next_dsa/build.rs, the tensor table of DsaTpPlan::new
// and build_dsa_weights (q_a_proj, q_a_layernorm, q_absorb = q_b_proj through
// kv_b_proj's K half, kv_a_proj_with_mqa, kv_a_layernorm, indexer.wq_b, indexer.wk,
// indexer.weights_proj scaled by index_heads^-0.5, the compress gate). Per row:
//
//   [q_a | kv_a | k | gate | w] = W_x . x        (one skinny GEMM over the x weights,
//                                                 f32 results)
//   q_lora = bf16(rms(q_a) * q_a_norm)           ckv = bf16(rms(kv_a) * kv_a_norm)
//   [qlat | qidx] = bf16(w_q . q_lora)            (w_q = [q_absorb ; wq_b], one GEMM)
//   k_new  = bf16(k),  gate_new = bf16(gate),    w (f32)
//
// with rms(v) = v / sqrt(mean(v^2) + eps). At decode sizes each GEMM streams its
// weights once for all rows (the projection kernel's TMA ring, stream-K split and
// ordered partial sums); the norms and casts run in one small kernel between them.
#include "common.cuh"

namespace dsa {
namespace {

constexpr int kNormThreads = 256;

struct NormArgs {
    const float* y1;  // [R, n_x]
    int n_x, ql, kvl, ihd, hi;
    const uint16_t* q_norm;
    const uint16_t* kv_norm;
    float eps;
    uint16_t* q_lora;  // [R, ql]
    uint16_t* ckv_new;
    uint16_t* k_new;
    uint16_t* gate_new;
    float* w;
};

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();  // red is reused by consecutive calls
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < kNormThreads / 32; ++i) t += red[i];
    return t;
}

__global__ void __launch_bounds__(kNormThreads) frontend_norm_kernel(NormArgs a) {
    // The q GEMM after this kernel streams weights it can fetch before q_lora
    // exists: let its blocks start now (they wait for this grid before reading it).
    pdl_trigger();
    pdl_wait();
    __shared__ float red[kNormThreads / 32];
    const int r = blockIdx.x;
    const float* y = a.y1 + (long long)r * a.n_x;
    float sq = 0.f, skv = 0.f;
    for (int c = threadIdx.x; c < a.ql; c += kNormThreads) sq = fmaf(y[c], y[c], sq);
    for (int c = threadIdx.x; c < a.kvl; c += kNormThreads) {
        const float v = y[a.ql + c];
        skv = fmaf(v, v, skv);
    }
    const float rq = rsqrtf(block_sum(sq, red) / (float)a.ql + a.eps);
    const float rkv = rsqrtf(block_sum(skv, red) / (float)a.kvl + a.eps);
    for (int c = threadIdx.x; c < a.ql; c += kNormThreads)
        a.q_lora[(long long)r * a.ql + c] =
            __bfloat16_as_ushort(__float2bfloat16_rn(y[c] * rq * bf16_lo(a.q_norm[c])));
    for (int c = threadIdx.x; c < a.kvl; c += kNormThreads)
        a.ckv_new[(long long)r * a.kvl + c] =
            __bfloat16_as_ushort(__float2bfloat16_rn(y[a.ql + c] * rkv * bf16_lo(a.kv_norm[c])));
    const float* yk = y + a.ql + a.kvl;
    for (int c = threadIdx.x; c < a.ihd; c += kNormThreads) {
        a.k_new[(long long)r * a.ihd + c] = __bfloat16_as_ushort(__float2bfloat16_rn(yk[c]));
        a.gate_new[(long long)r * a.ihd + c] =
            __bfloat16_as_ushort(__float2bfloat16_rn(yk[a.ihd + c]));
    }
    for (int c = threadIdx.x; c < a.hi; c += kNormThreads)
        a.w[(long long)r * a.hi + c] = yk[2 * a.ihd + c];
}

struct FrontPlan {
    size_t off_y1, off_qlora, off_part, bytes;
};

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

FrontPlan front_plan(int rows, int hidden, int n_x, int ql, int nq, int sms) {
    FrontPlan p;
    p.off_y1 = 0;
    p.off_qlora = al256((size_t)rows * n_x * 4);
    p.off_part = p.off_qlora + al256((size_t)rows * ql * 2);
    size_t part = project_workspace_bytes(rows, hidden, n_x, sms);
    const size_t b = project_workspace_bytes(rows, ql, nq, sms);
    if (b > part) part = b;
    p.bytes = p.off_part + al256(part);
    return p;
}

int check_front(int rows, int hidden, int n_x, int ql, int kvl, int ihd, int hi, int heads) {
    if (rows < 0 || rows > 65535 || hidden < 1 || ql < 1 || kvl < 1 || ihd < 1 || hi < 1 ||
        heads < 1)
        return fail(DSA_ERR_INVALID_ARG,
                    "dsa_frontend: rows %d, hidden %d, q_lora_rank %d, kv_lora_rank %d, ihd %d, "
                    "index_heads %d, heads %d",
                    rows, hidden, ql, kvl, ihd, hi, heads);
    if ((long long)ql + kvl + 2LL * ihd + hi > n_x)
        return fail(DSA_ERR_INVALID_ARG, "dsa_frontend: n_x %d < q_lora + kv_lora + 2*ihd + heads",
                    n_x);
    if (!project_supported(hidden, n_x) || !project_supported(ql, heads * kvl) ||
        !project_supported(ql, hi * ihd) || !project_supported(ql, heads * kvl + hi * ihd))
        return fail(DSA_ERR_UNSUPPORTED,
                    "dsa_frontend: hidden and q_lora_rank must be multiples of 256; n_x, "
                    "heads*kv_lora_rank and index_heads*ihd multiples of 64");
    if (ihd % 8 != 0 || kvl % 8 != 0)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_frontend: ihd and kv_lora_rank multiples of 8");
    return DSA_OK;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" int dsa_frontend_workspace(int rows, int hidden, int n_x, int q_lora_rank,
                                      int kv_lora_rank, int ihd, int index_heads, int heads,
                                      size_t* bytes) {
    if (!bytes) return fail(DSA_ERR_INVALID_ARG, "dsa_frontend_workspace: bytes is NULL");
    int rc = check_front(rows, hidden, n_x, q_lora_rank, kv_lora_rank, ihd, index_heads, heads);
    if (rc) return rc;
    const int sms = sm_count();
    if (sms <= 0) return fail(DSA_ERR_CUDA, "dsa_frontend_workspace: no CUDA device");
    *bytes = front_plan(rows, hidden, n_x, q_lora_rank, heads * kv_lora_rank + index_heads * ihd,
                        sms)
                 .bytes;
    return DSA_OK;
}

extern "C" int dsa_frontend(const dsa_bf16* x, int rows, int hidden, const dsa_bf16* w_x, int n_x,
                            int q_lora_rank, int kv_lora_rank, int ihd, int index_heads,
                            const dsa_bf16* q_a_norm, const dsa_bf16* kv_a_norm, float eps,
                            const dsa_bf16* w_q, int heads, dsa_bf16* qlat, dsa_bf16* qidx,
                            float* w, dsa_bf16* k_new, dsa_bf16* gate_new, dsa_bf16* ckv_new,
                            int32_t* status,
                            void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_front(rows, hidden, n_x, q_lora_rank, kv_lora_rank, ihd, index_heads, heads);
    if (rc) return rc;
    if (!(eps >= 0.f)) return fail(DSA_ERR_INVALID_ARG, "dsa_frontend: eps must be >= 0");
    if (rows == 0) return DSA_OK;
    if (!x || !w_x || !q_a_norm || !kv_a_norm || !w_q || !qlat || !qidx || !w ||
        !k_new || !gate_new || !ckv_new)
        return fail(DSA_ERR_INVALID_ARG, "dsa_frontend: NULL tensor");
    if ((((uintptr_t)x) | ((uintptr_t)w_x) | ((uintptr_t)w_q) | ((uintptr_t)qlat) |
         ((uintptr_t)qidx) | ((uintptr_t)workspace)) & 15)
        return fail(DSA_ERR_INVALID_ARG, "dsa_frontend: tensors must be 16-byte aligned");
    const int sms = sm_count();
    if (sms <= 0) return fail(DSA_ERR_CUDA, "dsa_frontend: no CUDA device");
    const int nq = heads * kv_lora_rank + index_heads * ihd;
    const FrontPlan p = front_plan(rows, hidden, n_x, q_lora_rank, nq, sms);
    if (!workspace || workspace_bytes < p.bytes)
        return fail(DSA_ERR_INVALID_ARG, "dsa_frontend: workspace %zu B < %zu B needed",
                    workspace_bytes, p.bytes);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* y1 = reinterpret_cast<float*>(ws + p.off_y1);
    uint16_t* q_lora = reinterpret_cast<uint16_t*>(ws + p.off_qlora);
    void* part = ws + p.off_part;
    const size_t part_bytes = workspace_bytes - p.off_part;
    cudaStream_t st = (cudaStream_t)stream;

    rc = project_launch(x, false, rows, hidden, w_x, n_x, nullptr, status, part, part_bytes, st,
                        y1);
    if (rc) return rc;
    NormArgs na;
    na.y1 = y1;
    na.n_x = n_x;
    na.ql = q_lora_rank;
    na.kvl = kv_lora_rank;
    na.ihd = ihd;
    na.hi = index_heads;
    na.q_norm = q_a_norm;
    na.kv_norm = kv_a_norm;
    na.eps = eps;
    na.q_lora = q_lora;
    na.ckv_new = ckv_new;
    na.k_new = k_new;
    na.gate_new = gate_new;
    na.w = w;
    cudaError_t e = launch_pdl(frontend_norm_kernel, dim3((unsigned)rows), dim3(kNormThreads), 0,
                               st, na);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "dsa_frontend norm launch");
    return project_launch(q_lora, false, rows, q_lora_rank, w_q, nq, qlat, status, part,
                          part_bytes, st, nullptr, qidx, heads * kv_lora_rank);
}
