// dsa_sparse_mla_decode: NoPE MLA over the selected tokens, in the 512-wide latent
// space, followed by the absorbed output projection.
//
// Pages: metrale_model_arch/glm5next_dsa/mod.rs, "Shape of the pipeline" (last stage:
// NoPE MLA restricted to the expanded token ids, -1 = invalid) and build.rs, module
// doc, transforms 1 and 3 (Q absorbed through kv_b_proj's K half, o_proj through its
// V half: the latent row is both key and value, and the decode output
// [heads, kv_lora_rank] maps back to hidden through o_absorb).
//
// Three kernels (four with a split combine):
//
// 1. mla_split_kernel -- one CTA per (split of the token list, query row, group of up
//    to 64 heads). All heads share the latent rows (like MQA), so every gathered
//    1 KiB row is read once per query row and used by all heads. Rows are gathered
//    64 tokens at a time with cp.async into a double-buffered, XOR-swizzled
//    shared-memory tile while the previous chunk computes. S = Q K^T and O += P V run
//    on m16n8k16 bf16 MMAs (f32 accumulate) with ldmatrix operands; softmax is online
//    in the log2 domain. Output: unnormalised partial O and (max, sum) per head, or,
//    with a single split, the normalised olat directly.
// 2. mla_combine_kernel -- merges the splits of a row (log-sum-exp weights).
// 3. oabs_gemv_kernel -- y_part = olat_bf16 @ o_absorb^T over a k-range, streaming
//    o_absorb from HBM once per step straight into MMA A-fragments (same permuted-k
//    trick as the score kernel), query rows on the MMA N axis.
// 4. ysum_kernel -- adds the k-range partials and rounds y to bf16.
#include "common.cuh"
#include "fp8.cuh"

namespace dsa {
namespace {

constexpr int KVL = DSA_KV_LORA_RANK;  // 512
constexpr int CH = 64;                 // tokens per gathered chunk
constexpr int kMaxSplits = 64;         // token splits per row (make_plan's bound)
constexpr int ROWB = KVL * 2;          // bytes per latent row
constexpr int kF8Groups = KVL / 128;   // FP8 cache: one scale per 128 channels
constexpr int ROW8 = KVL + kF8Groups * 4;  // FP8 cache: codes + scales of one token (528 B)
constexpr float kLog2e = 1.4426950408889634f;

struct MlaArgs {
    const uint16_t* qlat;
    const int32_t* row_seq;
    const uint16_t* ckv;
    const uint8_t* ckv8;     // FP8 cache: E4M3 codes [.., KVL]
    const float* ckv_scale;  // FP8 cache: power-of-two scales [.., KVL / 128]
    const int32_t* token_ids;
    float* part_o;
    float* part_ml;
    float* olat;
    uint16_t* xbf;
    int32_t* status;
    Paging pg;
    int rows;
    int heads;
    int ow;
    int ns;
    int tps;
    float sl2;  // softmax_scale * log2(e)
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) {  // byte offset in a 1 KiB-row tile
    return (uint32_t)(row * ROWB + ((chunk ^ (row & 7)) << 4));
}

template <int MT, bool F8>
constexpr int split_smem_bytes() {
    return MT * 16 * ROWB                 // Q
           + (F8 ? 1 : 2) * CH * ROWB     // latent rows as bf16: double buffered, or one
                                          // tile converted from the FP8 stage
           + (F8 ? 2 * CH * ROW8 : 0)     // FP8 codes + scales, double buffered
           + MT * 16 * CH * 2             // P (bf16)
           + 4 * MT * 16 * 4              // cross-warp max/sum exchange
           + 2 * CH;                      // token validity
}

template <int MT, bool F8>
__global__ void __launch_bounds__(MT * 64, 1) mla_split_kernel(MlaArgs a) {
    pdl_wait();
    constexpr int NW = 2 * MT;
    constexpr int NTH = NW * 32;
    constexpr int HP = 16 * MT;
    constexpr int RPW = CH / NW;  // gathered rows per warp

    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* Qs = smem;
    uint8_t* KV = Qs + HP * ROWB;
    uint8_t* stage = KV + (F8 ? 1 : 2) * CH * ROWB;  // FP8 only
    uint8_t* Ps = stage + (F8 ? 2 * CH * ROW8 : 0);
    float* red = reinterpret_cast<float*>(Ps + HP * CH * 2);  // [max|sum][half][HP]
    uint8_t* vmask = reinterpret_cast<uint8_t*>(red + 4 * HP);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int g = lane >> 2;
    const int q = lane & 3;
    const int mt = warp % MT;
    const int half = warp / MT;  // token half in QK, dim half in PV
    const int split = blockIdx.x;
    const int r = blockIdx.y;
    const int head0 = blockIdx.z * HP;
    const int nh = min(HP, a.heads - head0);

    int seq = a.row_seq ? __ldg(a.row_seq + r) : r;
    int L = 0;
    if (seq >= 0 && seq < a.pg.batch) {
        L = min(__ldg(a.pg.seq_lens + seq), seq_capacity(a.pg));
    } else {
        if (tid == 0 && split == 0 && blockIdx.z == 0) flag_status(a.status, DSA_STATUS_BAD_TOKEN);
        seq = 0;
    }
    const int t_begin = split * a.tps;
    const int t_end = min(t_begin + a.tps, a.ow);
    const int nch = t_end > t_begin ? (t_end - t_begin + CH - 1) / CH : 0;

    // Q rows -> shared (zero rows past the last head).
    {
        const uint16_t* qbase = a.qlat + ((long long)r * a.heads + head0) * KVL;
        for (int i = tid; i < HP * 64; i += NTH) {
            const int row = i >> 6, c = i & 63;
            const bool ok = row < nh;
            cp_async16(smem_u32(Qs + swz(row, c)), ok ? (const void*)(qbase + row * KVL + c * 8)
                                                      : (const void*)a.qlat,
                       ok ? 16 : 0);
        }
    }

    auto gather = [&](int c, int buf) {
        const int base = t_begin + c * CH;
        long long prow = -1;
        if (lane < RPW) {
            const int j = warp * RPW + lane;
            const int pos = base + j;
            if (pos < t_end) {
                const int t = __ldg(a.token_ids + (long long)r * a.ow + pos);
                if (t >= 0) {
                    if (t >= L) {
                        flag_status(a.status, DSA_STATUS_BAD_TOKEN);
                    } else {
                        prow = token_row(a.pg, seq, t);
                        if (prow < 0) flag_status(a.status, DSA_STATUS_BAD_BLOCK);
                    }
                } else if (t < -1) {
                    flag_status(a.status, DSA_STATUS_BAD_TOKEN);
                }
            }
            vmask[buf * CH + j] = prow >= 0 ? 1 : 0;
        }
        if constexpr (F8) {
            // codes (32 lanes x 16 B) and the row's scales (16 B) into the stage
            uint8_t* dst = stage + buf * CH * ROW8;
#pragma unroll 4
            for (int jj = 0; jj < RPW; ++jj) {
                const long long pr = __shfl_sync(0xffffffffu, prow, jj);
                const int row = warp * RPW + jj;
                const int nb = pr >= 0 ? 16 : 0;
                const uint8_t* src = pr >= 0 ? a.ckv8 + pr * KVL : a.ckv8;
                cp_async16(smem_u32(dst + row * ROW8 + lane * 16), src + lane * 16, nb);
                if (lane == 0)
                    cp_async16(smem_u32(dst + row * ROW8 + KVL),
                               pr >= 0 ? (const void*)(a.ckv_scale + pr * kF8Groups)
                                       : (const void*)a.ckv_scale,
                               nb);
            }
        } else {
            uint8_t* dst = KV + buf * CH * ROWB;
#pragma unroll 4
            for (int jj = 0; jj < RPW; ++jj) {
                const long long pr = __shfl_sync(0xffffffffu, prow, jj);
                const int row = warp * RPW + jj;
                const uint16_t* src = pr >= 0 ? a.ckv + pr * KVL : a.ckv;
                const int nb = pr >= 0 ? 16 : 0;
                cp_async16(smem_u32(dst + swz(row, lane)), src + lane * 8, nb);
                cp_async16(smem_u32(dst + swz(row, lane + 32)), src + (lane + 32) * 8, nb);
            }
        }
    };

    if (nch > 0) gather(0, 0);
    cp_async_commit();

    float m0 = -INFINITY, m1 = -INFINITY;  // running max (log2 domain), rows g, g+8
    float l0 = 0.f, l1 = 0.f;              // running sum
    float oacc[32][4];
#pragma unroll
    for (int i = 0; i < 32; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;

    const int hrow0 = mt * 16 + g;  // head rows of this thread within the CTA tile
    const int hrow1 = hrow0 + 8;

    for (int c = 0; c < nch; ++c) {
        const int buf = c & 1;
        if (c + 1 < nch) {
            gather(c + 1, buf ^ 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if constexpr (F8) {
            // Stage -> bf16 tile: each thread converts 8 codes into one 16-byte chunk
            // (a quarter warp covers 8 consecutive chunks of a row: no bank conflicts).
            const uint8_t* sb = stage + buf * CH * ROW8;
            for (int u = tid; u < CH * 64; u += NTH) {
                const int row = u >> 6, j = u & 63;
                const uint2 cw = *reinterpret_cast<const uint2*>(sb + row * ROW8 + j * 8);
                const float sc = *reinterpret_cast<const float*>(sb + row * ROW8 + KVL + (j >> 4) * 4);
                uint4 o;
                o.x = e4m3x2_to_bf16x2(cw.x, sc);
                o.y = e4m3x2_to_bf16x2(cw.x >> 16, sc);
                o.z = e4m3x2_to_bf16x2(cw.y, sc);
                o.w = e4m3x2_to_bf16x2(cw.y >> 16, sc);
                *reinterpret_cast<uint4*>(KV + swz(row, j)) = o;
            }
            __syncthreads();
        }
        const uint8_t* Kb = KV + (F8 ? 0 : buf) * CH * ROWB;

        // ---- S = Q K^T for 16 heads x 32 tokens
        float sacc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
        {
            const int arow = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int mi = lane >> 3;
#pragma unroll 8
            for (int kk = 0; kk < KVL / 16; ++kk) {
                uint32_t af[4];
                ldsm_x4(af, smem_u32(Qs + swz(arow, 2 * kk + (lane >> 4))));
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    const int tok = half * 32 + np * 16 + (mi >> 1) * 8 + (lane & 7);
                    uint32_t bf[4];
                    ldsm_x4(bf, smem_u32(Kb + swz(tok, 2 * kk + (mi & 1))));
                    mma_16816(sacc[2 * np], af[0], af[1], af[2], af[3], bf[0], bf[1]);
                    mma_16816(sacc[2 * np + 1], af[0], af[1], af[2], af[3], bf[2], bf[3]);
                }
            }
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int tok = half * 32 + nt * 8 + 2 * q + j;
                const bool ok = vmask[buf * CH + tok] != 0;
                sacc[nt][j] = ok ? sacc[nt][j] * a.sl2 : -INFINITY;
                sacc[nt][2 + j] = ok ? sacc[nt][2 + j] * a.sl2 : -INFINITY;
                mx0 = fmaxf(mx0, sacc[nt][j]);
                mx1 = fmaxf(mx1, sacc[nt][2 + j]);
            }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        if (q == 0) {
            red[half * HP + hrow0] = mx0;
            red[half * HP + hrow1] = mx1;
        }
        __syncthreads();
        const float cm0 = fmaxf(red[hrow0], red[HP + hrow0]);
        const float cm1 = fmaxf(red[hrow1], red[HP + hrow1]);
        const float mn0 = fmaxf(m0, cm0), mn1 = fmaxf(m1, cm1);
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
        const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = exp2f(m0 - mu0), al1 = exp2f(m1 - mu1);
        float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const float p00 = round_bf16(exp2f(sacc[nt][0] - mu0));
            const float p01 = round_bf16(exp2f(sacc[nt][1] - mu0));
            const float p10 = round_bf16(exp2f(sacc[nt][2] - mu1));
            const float p11 = round_bf16(exp2f(sacc[nt][3] - mu1));
            ls0 += p00 + p01;
            ls1 += p10 + p11;
            const int chunk = half * 4 + nt;
            *reinterpret_cast<uint32_t*>(Ps + hrow0 * (CH * 2) + ((chunk ^ (hrow0 & 7)) << 4) +
                                         4 * q) = pack_bf16x2(p00, p01);
            *reinterpret_cast<uint32_t*>(Ps + hrow1 * (CH * 2) + ((chunk ^ (hrow1 & 7)) << 4) +
                                         4 * q) = pack_bf16x2(p10, p11);
        }
        ls0 += __shfl_xor_sync(0xffffffffu, ls0, 1);
        ls1 += __shfl_xor_sync(0xffffffffu, ls1, 1);
        ls0 += __shfl_xor_sync(0xffffffffu, ls0, 2);
        ls1 += __shfl_xor_sync(0xffffffffu, ls1, 2);
        if (q == 0) {
            red[2 * HP + half * HP + hrow0] = ls0;
            red[2 * HP + half * HP + hrow1] = ls1;
        }
        __syncthreads();
        l0 = l0 * al0 + red[2 * HP + hrow0] + red[3 * HP + hrow0];
        l1 = l1 * al1 + red[2 * HP + hrow1] + red[3 * HP + hrow1];
        m0 = mn0;
        m1 = mn1;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            oacc[i][0] *= al0;
            oacc[i][1] *= al0;
            oacc[i][2] *= al1;
            oacc[i][3] *= al1;
        }

        // ---- O += P V for 16 heads x 256 latent dims
        {
            const int arow = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int mi = lane >> 3;
#pragma unroll
            for (int kk = 0; kk < CH / 16; ++kk) {
                uint32_t af[4];
                const int pch = 2 * kk + (lane >> 4);
                ldsm_x4(af, smem_u32(Ps + arow * (CH * 2) + ((pch ^ (arow & 7)) << 4)));
                const int tok = kk * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
                for (int dp = 0; dp < 16; ++dp) {
                    uint32_t bf[4];
                    ldsm_x4_t(bf, smem_u32(Kb + swz(tok, half * 32 + 2 * dp + (mi >> 1))));
                    mma_16816(oacc[2 * dp], af[0], af[1], af[2], af[3], bf[0], bf[1]);
                    mma_16816(oacc[2 * dp + 1], af[0], af[1], af[2], af[3], bf[2], bf[3]);
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    // ---- write out
    const bool ok0 = hrow0 < nh, ok1 = hrow1 < nh;
    const int dim0 = half * 256 + 2 * q;
    if (a.ns == 1) {
        const float i0 = l0 > 0.f ? 1.f / l0 : 0.f;
        const float i1 = l1 > 0.f ? 1.f / l1 : 0.f;
        const long long o0 = ((long long)r * a.heads + head0 + hrow0) * KVL;
        const long long o1 = ((long long)r * a.heads + head0 + hrow1) * KVL;
#pragma unroll
        for (int nt = 0; nt < 32; ++nt) {
            const int d = dim0 + nt * 8;
            if (ok0) {
                const float x0 = oacc[nt][0] * i0, x1 = oacc[nt][1] * i0;
                if (a.olat) *reinterpret_cast<float2*>(a.olat + o0 + d) = make_float2(x0, x1);
                if (a.xbf) *reinterpret_cast<uint32_t*>(a.xbf + o0 + d) = pack_bf16x2(x0, x1);
            }
            if (ok1) {
                const float x0 = oacc[nt][2] * i1, x1 = oacc[nt][3] * i1;
                if (a.olat) *reinterpret_cast<float2*>(a.olat + o1 + d) = make_float2(x0, x1);
                if (a.xbf) *reinterpret_cast<uint32_t*>(a.xbf + o1 + d) = pack_bf16x2(x0, x1);
            }
        }
    } else {
        const long long base = ((long long)r * a.ns + split) * a.heads + head0;
#pragma unroll
        for (int nt = 0; nt < 32; ++nt) {
            const int d = dim0 + nt * 8;
            if (ok0)
                *reinterpret_cast<float2*>(a.part_o + (base + hrow0) * KVL + d) =
                    make_float2(oacc[nt][0], oacc[nt][1]);
            if (ok1)
                *reinterpret_cast<float2*>(a.part_o + (base + hrow1) * KVL + d) =
                    make_float2(oacc[nt][2], oacc[nt][3]);
        }
        if (half == 0 && q == 0) {
            if (ok0) *reinterpret_cast<float2*>(a.part_ml + (base + hrow0) * 2) = make_float2(m0, l0);
            if (ok1) *reinterpret_cast<float2*>(a.part_ml + (base + hrow1) * 2) = make_float2(m1, l1);
        }
    }
}

// One CTA per (head, row): merge the splits with log-sum-exp weights. The splits'
// (m, l) pairs are read once into shared memory as weights 2^(m_s - M); the partial
// outputs are then summed in split order, eight independent 16-byte loads in flight
// per thread.
__global__ void __launch_bounds__(128) mla_combine_kernel(const float* __restrict__ part_o,
                                                          const float* __restrict__ part_ml,
                                                          int heads, int ns, float* olat,
                                                          uint16_t* xbf) {
    // The projection that follows streams weights it can fetch before olat exists:
    // let its blocks start now (they wait for this grid before reading olat).
    pdl_trigger();
    pdl_wait();
    __shared__ float wsh[kMaxSplits];
    __shared__ float lsum;
    const int h = blockIdx.x, r = blockIdx.y, t = threadIdx.x;
    const long long stride = (long long)heads * (KVL / 4);  // float4s between splits
    const float4* po = reinterpret_cast<const float4*>(part_o) +
                       ((long long)r * ns * heads + h) * (KVL / 4) + t;
    // The first 16 splits' partials are requested before the weights are known, so
    // the two round trips to L2 overlap.
    constexpr int kEarly = 16;
    float4 oe[kEarly];
#pragma unroll
    for (int j = 0; j < kEarly; ++j)
        oe[j] = j < ns ? __ldg(po + j * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < 32) {
        float m[2], l[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int s = t + 32 * k;
            m[k] = -INFINITY;
            l[k] = 0.f;
            if (s < ns) {
                const float2 ml = __ldg(reinterpret_cast<const float2*>(part_ml) +
                                        ((long long)r * ns + s) * heads + h);
                m[k] = ml.x;
                l[k] = ml.y;
            }
        }
        float M = fmaxf(m[0], m[1]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float L = 0.f;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float wgt = m[k] == -INFINITY ? 0.f : exp2f(m[k] - M);
            L += wgt * l[k];
            if (t + 32 * k < ns) wsh[t + 32 * k] = wgt;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
        if (t == 0) lsum = L;
    }
    __syncthreads();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kEarly; ++j) {
        if (j < ns) {
            const float wgt = wsh[j];
            acc.x += wgt * oe[j].x;
            acc.y += wgt * oe[j].y;
            acc.z += wgt * oe[j].z;
            acc.w += wgt * oe[j].w;
        }
    }
    for (int s0 = kEarly; s0 < ns; s0 += 8) {
        float4 o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            o[j] = s0 + j < ns ? __ldg(po + (s0 + j) * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (s0 + j < ns) {
                const float wgt = wsh[s0 + j];
                acc.x += wgt * o[j].x;
                acc.y += wgt * o[j].y;
                acc.z += wgt * o[j].z;
                acc.w += wgt * o[j].w;
            }
        }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    const long long o = ((long long)r * heads + h) * KVL + 4 * t;
    if (olat) *reinterpret_cast<float4*>(olat + o) = acc;
    if (xbf) {
        uint2 v;
        v.x = pack_bf16x2(acc.x, acc.y);
        v.y = pack_bf16x2(acc.z, acc.w);
        *reinterpret_cast<uint2*>(xbf + o) = v;
    }
}

// ---------------------------------------------------------------------------
// y_part[ks, n, i] = sum_{k in range ks} A[i, k] * X[n, k]    (A = o_absorb, X = olat)

struct GemvArgs {
    const uint16_t* A;
    const uint16_t* X;
    float* ypart;
    int R;       // query rows in X (total)
    int n0;      // first query row of this launch
    int nrows;   // query rows of this launch (<= 8 * NT)
    int hidden;
    int K;
    int KS;
    int n_mg;
};

constexpr int kGemvWarps = 4;
constexpr int kGemvMT = 2;

template <int NT>
__device__ __forceinline__ void gemv_step(float (&acc)[kGemvMT][NT][4],
                                          const uint4 (&av)[kGemvMT][2][4],
                                          const uint16_t* const (&xrow)[NT],
                                          const bool (&xok)[NT], int kc) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        uint4 xv[4];
#pragma unroll
        for (int v = 0; v < 4; ++v)
            xv[v] = xok[nt] ? ldg16(xrow[nt] + kc * 128 + 32 * v) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint32_t xb[4] = {xv[v].x, xv[v].y, xv[v].z, xv[v].w};
#pragma unroll
            for (int m = 0; m < kGemvMT; ++m) {
                const uint32_t ra[4] = {av[m][0][v].x, av[m][0][v].y, av[m][0][v].z, av[m][0][v].w};
                const uint32_t rb[4] = {av[m][1][v].x, av[m][1][v].y, av[m][1][v].z, av[m][1][v].w};
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2)
                    mma_16816(acc[m][nt], ra[2 * h2], rb[2 * h2], ra[2 * h2 + 1], rb[2 * h2 + 1],
                              xb[2 * h2], xb[2 * h2 + 1]);
            }
        }
    }
}

template <int NT>
__global__ void __launch_bounds__(kGemvWarps * 32) oabs_gemv_kernel(GemvArgs a) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int unit = blockIdx.x * kGemvWarps + warp;
    if (unit >= a.n_mg * a.KS) return;
    const int mg = unit % a.n_mg;
    const int ks = unit / a.n_mg;
    const int KC = a.K / 128;
    const int kc0 = (int)((long long)ks * KC / a.KS);
    const int kc1 = (int)((long long)(ks + 1) * KC / a.KS);
    const int row0 = mg * 16 * kGemvMT;

    const uint16_t* arow[kGemvMT][2];
#pragma unroll
    for (int m = 0; m < kGemvMT; ++m)
#pragma unroll
        for (int h = 0; h < 2; ++h)
            arow[m][h] = a.A + (long long)(row0 + m * 16 + g + 8 * h) * a.K + 8 * q;
    const uint16_t* xrow[NT];
    bool xok[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int n = nt * 8 + g;
        xok[nt] = n < a.nrows;
        xrow[nt] = a.X + (long long)(a.n0 + (xok[nt] ? n : 0)) * a.K + 8 * q;
    }

    float acc[kGemvMT][NT][4];
#pragma unroll
    for (int m = 0; m < kGemvMT; ++m)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[m][nt][0] = acc[m][nt][1] = acc[m][nt][2] = acc[m][nt][3] = 0.f;

    uint4 av0[kGemvMT][2][4], av1[kGemvMT][2][4];
    auto load = [&](uint4(&av)[kGemvMT][2][4], int kc) {
#pragma unroll
        for (int m = 0; m < kGemvMT; ++m)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int v = 0; v < 4; ++v) av[m][h][v] = ldg16_stream(arow[m][h] + kc * 128 + 32 * v);
    };
    if (kc0 < kc1) load(av0, kc0);
    for (int kc = kc0; kc < kc1; kc += 2) {
        if (kc + 1 < kc1) load(av1, kc + 1);
        gemv_step<NT>(acc, av0, xrow, xok, kc);
        if (kc + 2 < kc1) load(av0, kc + 2);
        if (kc + 1 < kc1) gemv_step<NT>(acc, av1, xrow, xok, kc + 1);
    }

#pragma unroll
    for (int m = 0; m < kGemvMT; ++m)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int n = nt * 8 + 2 * q + j;
                if (n < a.nrows) {
                    float* yp = a.ypart + ((long long)ks * a.R + a.n0 + n) * a.hidden + row0 + m * 16 + g;
                    yp[0] = acc[m][nt][j];
                    yp[8] = acc[m][nt][2 + j];
                }
            }
}

__global__ void ysum_kernel(const float* __restrict__ ypart, int KS, long long n,
                            uint16_t* __restrict__ y) {
    pdl_wait();
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int k = 0; k < KS; ++k) s += __ldg(ypart + k * n + i);
        y[i] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
    }
}

// ---------------------------------------------------------------------------
// Launch plan (shared by the workspace query and the call).

struct Plan {
    bool tc;   // the persistent tensor-core split kernel (mla_tc.cu): 64 heads, large batches
    bool dec;        // the decode kernel (mla_dec.cu): 64 heads, decode batches
    bool dec_merge;  // ... whose row clusters merge their partials themselves
    int mt;
    int hgroups;
    int ns;
    int tps;
    int gemv_nt;
    int KS;
    int n_mg;
    bool tma_proj;  // the TMA-pipelined projection (project.cu) handles o_absorb
    size_t off_part_o, off_part_ml, off_xbf, off_ypart, bytes;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

Plan make_plan(int rows, int heads, int ow, int hidden, bool with_oabs, int sms,
               bool fp8 = false) {
    Plan p;
    // 64 heads: the persistent tensor-core kernel when the batch holds at least 4 of
    // its 128-token chunks per SM (64 rows of 2,048 tokens, a prefill chunk), the
    // cluster decode kernel below that (decode batches of a few rows); other head
    // counts and the FP8 cache: the mma.sync kernel. DSA_OPT_MLA_KERNEL forces one.
    const int choice = mla_kernel_choice();
    const long long tc_chunks = (long long)rows * ((ow + mla_tc_chunk() - 1) / mla_tc_chunk());
    const bool tc_ok = mla_tc_supported(heads, KVL);  // bf16 or FP8 cache
    const bool dec_ok = !fp8 && mla_dec_supported(heads, KVL, ow);
    if (choice == DSA_MLA_KERNEL_TCGEN05) {
        p.tc = tc_ok;
    } else if (choice == DSA_MLA_KERNEL_CLUSTER) {
        p.tc = false;
    } else if (choice == DSA_MLA_KERNEL_MMA) {
        p.tc = false;
    } else {
        p.tc = tc_ok && tc_chunks >= 4LL * sms;
    }
    // The tcgen05 decode kernel runs when forced: at 8 rows of 2,048 tokens it takes
    // 19.1 us (one chunk per CTA, combine kernel after it) against 16.8 us for the
    // mma.sync split kernel (cold-cache launch list), so by size the latter stays.
    p.dec = !p.tc && dec_ok && choice == DSA_MLA_KERNEL_CLUSTER;
    p.mt = heads <= 16 ? 1 : heads <= 32 ? 2 : 4;
    p.hgroups = p.tc ? 1 : (heads + 16 * p.mt - 1) / (16 * p.mt);
    const int chunk = p.tc ? mla_tc_chunk() : CH;
    const long long base = (long long)rows * p.hgroups;
    const int max_ns = ow > 0 ? (ow + chunk - 1) / chunk : 1;
    // one CTA per SM: at most sms / base splits keeps the grid to one wave
    long long ns = base > 0 ? sms / base : 1;
    if (ns < 1) ns = 1;
    if (ns > max_ns) ns = max_ns;
    if (ns > kMaxSplits) ns = kMaxSplits;
    const int per = ow > 0 ? (int)((ow + ns - 1) / ns) : 0;
    p.tps = per > 0 ? ((per + chunk - 1) / chunk) * chunk : chunk;
    p.ns = ow > 0 ? (ow + p.tps - 1) / p.tps : 1;
    p.dec_merge = false;
    if (p.dec) {
        mla_dec_plan(ow, &p.ns, &p.tps, &p.dec_merge);
        p.hgroups = 1;
    } else if (p.tc && ow > 0) {
        // Persistent grid: the busiest CTA walks ceil(units / sms) units of
        // ceil(chunks per row / ns) chunks, plus about a chunk's time per unit (Q,
        // the epilogue, the partials); take the split count that makes this smallest
        // (the fewest splits on ties: less to combine).
        const long long cpr = (ow + chunk - 1) / chunk;
        long long best = -1;
        for (long long t = 1; t <= cpr && t <= kMaxSplits; ++t) {
            const long long tps = ((cpr + t - 1) / t) * chunk;
            const long long nst = (ow + tps - 1) / tps;
            const long long cost =
                ((long long)rows * nst + sms - 1) / sms * ((cpr + nst - 1) / nst + 1);
            if (best < 0 || cost < best) {
                best = cost;
                p.tps = (int)tps;
                p.ns = (int)nst;
            }
        }
    }

    const int nr = rows < 64 ? rows : 64;
    p.gemv_nt = nr <= 8 ? 1 : nr <= 16 ? 2 : nr <= 32 ? 4 : 8;
    p.n_mg = hidden / (16 * kGemvMT);
    const int KC = heads * KVL / 128;
    const long long target = (long long)sms * (p.gemv_nt <= 2 ? 12 : 8);
    long long ks = p.n_mg > 0 ? (target + p.n_mg / 2) / p.n_mg : 1;
    if (ks < 1) ks = 1;
    if (ks > KC) ks = KC;
    p.KS = (int)ks;

    // partials: the split kernels' when a row has several splits; the decode kernel
    // always stores its CTAs' partials and merges them itself
    const bool parts = p.ns > 1 || p.dec;
    size_t off = 0;
    p.off_part_o = off;
    if (parts) off += align256((size_t)rows * p.ns * heads * KVL * 4);
    p.off_part_ml = off;
    if (parts) off += align256((size_t)rows * p.ns * heads * 2 * 4);
    p.off_xbf = off;
    if (with_oabs) off += align256((size_t)rows * heads * KVL * 2);
    p.off_ypart = off;
    p.tma_proj = with_oabs && project_supported(heads * KVL, hidden);
    if (p.tma_proj)
        off += align256(project_workspace_bytes(rows, heads * KVL, hidden, sms));
    else if (with_oabs)
        off += align256((size_t)p.KS * rows * hidden * 4);
    p.bytes = off;
    return p;
}

int check_common(int rows, int heads, int kv_lora_rank, int out_width, int hidden,
                 bool with_oabs) {
    if (rows < 0 || heads < 1 || out_width < 0)
        return fail(DSA_ERR_INVALID_ARG, "dsa_sparse_mla_decode: rows %d, heads %d, out_width %d",
                    rows, heads, out_width);
    if (kv_lora_rank != KVL)
        return fail(kv_lora_rank == 0 ? DSA_ERR_CONFIG : DSA_ERR_UNSUPPORTED,
                    "dsa_sparse_mla_decode: kv_lora_rank %d, kernels are built for %d",
                    kv_lora_rank, KVL);
    if (with_oabs && (hidden < 32 || hidden % 32 != 0))
        return fail(DSA_ERR_UNSUPPORTED,
                    "dsa_sparse_mla_decode: hidden %d must be a positive multiple of 32", hidden);
    if (rows > 65535) return fail(DSA_ERR_UNSUPPORTED, "dsa_sparse_mla_decode: rows %d > 65535", rows);
    return DSA_OK;
}

template <int MT, bool F8>
int launch_split(const MlaArgs& a, const Plan& p, cudaStream_t st) {
    constexpr int smem = split_smem_bytes<MT, F8>();
    static_assert(smem <= 227 * 1024, "split kernel shared memory");
    int rc = set_max_smem((const void*)mla_split_kernel<MT, F8>, smem);
    if (rc) return rc;
    dim3 grid(p.ns, a.rows, p.hgroups);
    cudaError_t e = launch_pdl(mla_split_kernel<MT, F8>, grid, dim3(MT * 64), smem, st, a);
    if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_mla_decode split launch");
    return DSA_OK;
}

template <int NT>
void launch_gemv(GemvArgs g, cudaStream_t st) {
    const int units = g.n_mg * g.KS;
    launch_pdl(oabs_gemv_kernel<NT>, dim3((units + kGemvWarps - 1) / kGemvWarps),
               dim3(kGemvWarps * 32), 0, st, g);
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" int dsa_sparse_mla_decode_workspace(int rows, int heads, int kv_lora_rank,
                                               int out_width, int hidden, int with_o_absorb,
                                               size_t* bytes) {
    if (!bytes) return fail(DSA_ERR_INVALID_ARG, "dsa_sparse_mla_decode_workspace: bytes is NULL");
    int rc = check_common(rows, heads, kv_lora_rank, out_width, hidden, with_o_absorb != 0);
    if (rc) return rc;
    const int sms = sm_count();
    if (sms <= 0) return fail(DSA_ERR_CUDA, "dsa_sparse_mla_decode_workspace: no CUDA device");
    // Enough for either cache format (the FP8 path never takes the tensor-core plan).
    const size_t b16 = make_plan(rows, heads, out_width, hidden, with_o_absorb != 0, sms).bytes;
    const size_t b8 = make_plan(rows, heads, out_width, hidden, with_o_absorb != 0, sms, true).bytes;
    *bytes = b16 > b8 ? b16 : b8;
    return DSA_OK;
}

namespace {
// dsa_sparse_mla_decode (ckv) and dsa_sparse_mla_decode_fp8 (ckv8 + ckv_scale).
int mla_decode_impl(const dsa_bf16* qlat, int rows, int heads, int kv_lora_rank,
                    const int32_t* row_seq, const dsa_bf16* ckv, const uint8_t* ckv8,
                    const float* ckv_scale, const dsa_paging* pg, const int32_t* token_ids,
                    int out_width, float softmax_scale, const dsa_bf16* o_absorb, int hidden,
                    dsa_bf16* y, float* olat, int32_t* status, void* workspace,
                    size_t workspace_bytes, void* stream) {
    const bool with_oabs = o_absorb != nullptr;
    const bool fp8 = ckv8 != nullptr;
    int rc = check_common(rows, heads, kv_lora_rank, out_width, hidden, with_oabs);
    if (rc) return rc;
    if (with_oabs != (y != nullptr))
        return fail(DSA_ERR_INVALID_ARG,
                    "dsa_sparse_mla_decode: o_absorb and y must be both given or both NULL");
    Paging P;
    rc = check_paging(pg, 0, &P);
    if (rc) return rc;
    if (rows == 0) return DSA_OK;
    if (!qlat || (fp8 ? !ckv_scale : !ckv) || (out_width > 0 && !token_ids))
        return fail(DSA_ERR_INVALID_ARG, "dsa_sparse_mla_decode: NULL tensor");
    if ((((uintptr_t)qlat) | ((uintptr_t)ckv) | ((uintptr_t)ckv8) | ((uintptr_t)ckv_scale) |
         ((uintptr_t)o_absorb) | ((uintptr_t)olat) | ((uintptr_t)y) | ((uintptr_t)workspace)) & 15)
        return fail(DSA_ERR_INVALID_ARG, "dsa_sparse_mla_decode: tensors must be 16-byte aligned");
    const int sms = sm_count();
    if (sms <= 0) return fail(DSA_ERR_CUDA, "dsa_sparse_mla_decode: no CUDA device");
    const Plan p = make_plan(rows, heads, out_width, hidden, with_oabs, sms, fp8);
    if (p.bytes > 0 && (!workspace || workspace_bytes < p.bytes))
        return fail(DSA_ERR_INVALID_ARG, "dsa_sparse_mla_decode: workspace %zu B < %zu B needed",
                    workspace_bytes, p.bytes);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t st = (cudaStream_t)stream;

    MlaArgs a;
    a.qlat = qlat;
    a.row_seq = row_seq;
    a.ckv = ckv;
    a.ckv8 = ckv8;
    a.ckv_scale = ckv_scale;
    a.token_ids = token_ids;
    const bool parts = p.ns > 1 || p.dec;
    a.part_o = parts ? reinterpret_cast<float*>(ws + p.off_part_o) : nullptr;
    a.part_ml = parts ? reinterpret_cast<float*>(ws + p.off_part_ml) : nullptr;
    a.olat = olat;
    a.xbf = with_oabs ? reinterpret_cast<uint16_t*>(ws + p.off_xbf) : nullptr;
    a.status = status;
    a.pg = P;
    a.rows = rows;
    a.heads = heads;
    a.ow = out_width;
    a.ns = p.ns;
    a.tps = p.tps;
    a.sl2 = softmax_scale * kLog2e;

    if (!olat && !with_oabs) return DSA_OK;  // nothing requested
    if (p.tc || p.dec) {
        MlaTcParams t;
        t.qlat = qlat;
        t.row_seq = row_seq;
        t.ckv = ckv;
        t.ckv8 = ckv8;
        t.ckv_scale = ckv_scale;
        t.token_ids = token_ids;
        t.part_o = a.part_o;
        t.part_ml = a.part_ml;
        t.olat = olat;
        t.xbf = a.xbf;
        t.status = status;
        t.pg = P;
        t.rows = rows;
        t.ow = out_width;
        t.ns = p.ns;
        t.tps = p.tps;
        t.sl2 = a.sl2;
        const long long ckv_rows = P.block_table ? (long long)P.num_blocks * P.block_size
                                                 : (long long)P.batch * P.max_seq_len;
        rc = p.dec ? mla_dec_launch(t, ckv_rows, st) : mla_tc_launch(t, ckv_rows, st);
    } else {
        switch (p.mt * 2 + (fp8 ? 1 : 0)) {
            case 2: rc = launch_split<1, false>(a, p, st); break;
            case 3: rc = launch_split<1, true>(a, p, st); break;
            case 4: rc = launch_split<2, false>(a, p, st); break;
            case 5: rc = launch_split<2, true>(a, p, st); break;
            case 9: rc = launch_split<4, true>(a, p, st); break;
            default: rc = launch_split<4, false>(a, p, st); break;
        }
    }
    if (rc) return rc;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_mla_decode split launch");
    if ((p.ns > 1 && !p.dec) || (p.dec && !p.dec_merge)) {
        e = launch_pdl(mla_combine_kernel, dim3(heads, rows), dim3(128), 0, st,
                       (const float*)a.part_o, (const float*)a.part_ml, heads, p.ns, olat, a.xbf);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_mla_decode combine launch");
    }
    if (p.tma_proj) {
        return project_launch(a.xbf, false, rows, heads * KVL, o_absorb, hidden, y, status,
                              ws + p.off_ypart, workspace_bytes - p.off_ypart, st);
    }
    if (with_oabs) {
        GemvArgs g;
        g.A = o_absorb;
        g.X = a.xbf;
        g.ypart = reinterpret_cast<float*>(ws + p.off_ypart);
        g.R = rows;
        g.hidden = hidden;
        g.K = heads * KVL;
        g.KS = p.KS;
        g.n_mg = p.n_mg;
        for (int n0 = 0; n0 < rows; n0 += 64) {
            g.n0 = n0;
            g.nrows = rows - n0 < 64 ? rows - n0 : 64;
            switch (p.gemv_nt) {
                case 1: launch_gemv<1>(g, st); break;
                case 2: launch_gemv<2>(g, st); break;
                case 4: launch_gemv<4>(g, st); break;
                default: launch_gemv<8>(g, st); break;
            }
        }
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_mla_decode gemv launch");
        const long long n = (long long)rows * hidden;
        long long blocks = (n + 255) / 256;
        if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
        e = launch_pdl(ysum_kernel, dim3((unsigned)blocks), dim3(256), 0, st,
                       (const float*)g.ypart, p.KS, n, (uint16_t*)y);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_mla_decode ysum launch");
    }
    return DSA_OK;
}
}  // namespace

extern "C" int dsa_sparse_mla_decode(const dsa_bf16* qlat, int rows, int heads, int kv_lora_rank,
                                     const int32_t* row_seq, const dsa_bf16* ckv,
                                     const dsa_paging* pg, const int32_t* token_ids,
                                     int out_width, float softmax_scale,
                                     const dsa_bf16* o_absorb, int hidden, dsa_bf16* y,
                                     float* olat, int32_t* status, void* workspace,
                                     size_t workspace_bytes, void* stream) {
    return mla_decode_impl(qlat, rows, heads, kv_lora_rank, row_seq, ckv, nullptr, nullptr, pg,
                           token_ids, out_width, softmax_scale, o_absorb, hidden, y, olat, status,
                           workspace, workspace_bytes, stream);
}

extern "C" int dsa_sparse_mla_decode_fp8(const dsa_bf16* qlat, int rows, int heads,
                                         int kv_lora_rank, const int32_t* row_seq,
                                         const uint8_t* ckv_codes, const float* ckv_scales,
                                         const dsa_paging* pg, const int32_t* token_ids,
                                         int out_width, float softmax_scale,
                                         const dsa_bf16* o_absorb, int hidden, dsa_bf16* y,
                                         float* olat, int32_t* status, void* workspace,
                                         size_t workspace_bytes, void* stream) {
    if (!ckv_codes) return fail(DSA_ERR_INVALID_ARG, "dsa_sparse_mla_decode_fp8: NULL codes");
    return mla_decode_impl(qlat, rows, heads, kv_lora_rank, row_seq, nullptr, ckv_codes,
                           ckv_scales, pg, token_ids, out_width, softmax_scale, o_absorb, hidden,
                           y, olat, status, workspace, workspace_bytes, stream);
}
