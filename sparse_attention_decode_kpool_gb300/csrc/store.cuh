// One staged token's rows copied into the token caches (the decode-time append).
#pragma once

#include "common.cuh"

namespace dsa {

// Copies sequence b's staged key, gate and (optional) latent rows into cache row
// `row` with 16-byte vectors spread over the block's threads, and marks the token
// valid. ihd and kvl are multiples of 8.
__device__ __forceinline__ void store_token_rows(const uint16_t* k_new, const uint16_t* gate_new,
                                                 const uint16_t* ckv_new, uint16_t* k_raw,
                                                 uint16_t* gate, uint8_t* valid, uint16_t* ckv,
                                                 int b, long long row, int ihd, int kvl) {
    const int nk = ihd / 8, nl = ckv ? kvl / 8 : 0;
    for (int i = threadIdx.x; i < 2 * nk + nl; i += blockDim.x) {
        if (i < nk) {
            *reinterpret_cast<uint4*>(k_raw + row * ihd + 8 * i) =
                ldg16(k_new + (long long)b * ihd + 8 * i);
        } else if (i < 2 * nk) {
            const int j = i - nk;
            *reinterpret_cast<uint4*>(gate + row * ihd + 8 * j) =
                ldg16(gate_new + (long long)b * ihd + 8 * j);
        } else {
            const int j = i - 2 * nk;
            *reinterpret_cast<uint4*>(ckv + row * kvl + 8 * j) =
                ldg16(ckv_new + (long long)b * kvl + 8 * j);
        }
    }
    if (threadIdx.x == 0) valid[row] = 1;
}

// Thread 0 only: the cache row of sequence b's next token, or -1 (with the status
// bit set) when the cache is full or the block table entry is bad.
__device__ __forceinline__ long long next_token_row(const Paging& pg, const int32_t* seq_lens,
                                                    int b, int* t_out, int32_t* status) {
    const int t = seq_lens[b];
    *t_out = t;
    if (t < 0 || t >= seq_capacity(pg)) {
        flag_status(status, DSA_STATUS_CACHE_FULL);
        return -1;
    }
    const long long row = token_row(pg, b, t);
    if (row < 0) flag_status(status, DSA_STATUS_BAD_BLOCK);
    return row;
}

}  // namespace dsa
