// dsa_quantize_latent: the FP8 latent cache's encoder.
//
// Format (the layer's stated choice; mod.rs names the FP8 decode kernel,
// glm5next_dsa_mla_decode_fp8, and nothing of its format): OCP E4M3 codes with one
// power-of-two scale 2^k per token and 128-channel group, k the smallest integer with
// amax <= 448 * 2^k (not below -126; 0 for an all-zero group). Dividing by 2^k is
// exact, so the only rounding is the E4M3 conversion (nearest, ties to even), and a
// decoded value (code times 2^k) is exact in bf16.
//
// One warp per latent row; for each 128-channel group every lane takes 4 channels,
// the group's largest magnitude comes from a warp max, and the scale exponent from
// its float bits (fp8.cuh).
#include "fp8.cuh"

namespace dsa {
namespace {

constexpr int kQuantWarps = 8;

__global__ void __launch_bounds__(kQuantWarps * 32) quantize_latent_kernel(
    const uint16_t* __restrict__ x, long long rows, int kvl, uint8_t* __restrict__ codes,
    float* __restrict__ scales) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long r = (long long)blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
    if (r >= rows) return;
    const int G = kvl / 128;
    for (int gi = 0; gi < G; ++gi)
        fp8_encode_group(x + r * kvl + gi * 128, codes + r * kvl + gi * 128, scales + r * G + gi, lane);
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" int dsa_quantize_latent(const dsa_bf16* x, long long rows, int kv_lora_rank,
                                   uint8_t* codes, float* scales, void* stream) {
    if (rows < 0 || kv_lora_rank < 128 || kv_lora_rank % 128 != 0)
        return fail(DSA_ERR_INVALID_ARG, "dsa_quantize_latent: rows %lld, kv_lora_rank %d",
                    rows, kv_lora_rank);
    if (rows == 0) return DSA_OK;
    if (!x || !codes || !scales) return fail(DSA_ERR_INVALID_ARG, "dsa_quantize_latent: NULL tensor");
    if ((((uintptr_t)x) | ((uintptr_t)codes) | ((uintptr_t)scales)) & 15)
        return fail(DSA_ERR_INVALID_ARG, "dsa_quantize_latent: tensors must be 16-byte aligned");
    const long long blocks = (rows + kQuantWarps - 1) / kQuantWarps;
    if (blocks > 0x7fffffffLL) return fail(DSA_ERR_UNSUPPORTED, "dsa_quantize_latent: too many rows");
    cudaError_t e = launch_pdl(quantize_latent_kernel, dim3((unsigned)blocks), dim3(kQuantWarps * 32),
                               0, (cudaStream_t)stream, (const uint16_t*)x, rows, kv_lora_rank,
                               codes, scales);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "dsa_quantize_latent launch");
    return DSA_OK;
}
