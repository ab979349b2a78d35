// Sparse latent attention on the tensor cores (tcgen05) for 64 heads: the split
// kernel of dsa_sparse_mla_decode when heads == 64.
//
// Page: metrale_model_arch/glm5next_dsa/mod.rs, "Shape of the pipeline" (last stage)
// and build.rs module doc, transforms 1 and 3 (absorbed Q; each latent row is both
// key and value). Per row r, head h, over the selected tokens t of a split:
//   s[t,h] = softmax_scale * <ckv[t,:], qlat[r,h,:]>;  O[h,:] = sum_t p[t,h] ckv[t,:]
// with p = 2^(s*log2e - m_h) against a running per-head maximum m_h.
//
// A CTA takes one (split, row) and walks its tokens in chunks of 128:
//   - warp 0 resolves the chunk's token rows, and it and the four softmax warps
//     gather the 128 latent rows with cp.async (512 contiguous bytes per warp
//     instruction) into eight 128-byte-swizzled atoms of 64 latent columns
//     ([atom][token][64 c]); the row's Q (64 heads x 512) is loaded once by TMA;
//   - warp 1 owns the tensor memory and issues the MMAs:
//       S^T = K Q^T   M = 128 tokens, N = 64 heads, K = 512 (the atoms are K-major);
//       O^T += V^T P^T  M = 512 latent (4 tiles of 128), N = 64 heads, K = 128 tokens,
//     where the same atoms are read MN-major for V^T and P^T is written by the
//     softmax warps as [token][64 heads] (MN-major);
//   - warps 2..5 (one tensor-memory lane per token) take S^T, find each head's chunk
//     maximum (warp max, then across the four warps through shared memory), update
//     the running maximum only when it grows by more than 2^8 (then O^T and the
//     partial sums are rescaled), write P^T in bf16, keep per-thread partial sums,
//     and at the end write the split's partial (or, with one split, olat).
// All waits are bounded; a timeout sets DSA_STATUS_TIMEOUT, every role leaves its
// loop, copies and MMAs in flight are drained, and the tensor memory is released.
#include <stdlib.h>

#include "common.cuh"
#include "tc.cuh"

namespace dsa {
namespace {

constexpr int kT = 128;                        // tokens per chunk
constexpr int kH = 64;                         // heads
constexpr int kKVL = 512;                      // latent width
constexpr int kAtoms = kKVL / 64;              // 128-byte atoms per latent row
constexpr uint32_t kLatAtom = kT * 128;        // one atom of the token tile
constexpr uint32_t kQAtom = kH * 128;          // one atom of the Q tile
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffLat = kOffQ + kAtoms * kQAtom;
constexpr uint32_t kOffP = kOffLat + kAtoms * kLatAtom;
constexpr uint32_t kOffRed = kOffP + kT * 128;          // [2][4 warps][kH] f32
constexpr uint32_t kOffM = kOffRed + 2 * 4 * kH * 4;    // [2][kH] running maxima
constexpr uint32_t kOffRows = kOffM + 2 * kH * 4;       // [kT] cache row per token
constexpr uint32_t kOffMask = kOffRows + kT * 4;        // [kT] token valid
constexpr uint32_t kOffBar = kOffMask + kT;
constexpr int kBars = 11;
constexpr uint32_t kOffMisc = kOffBar + kBars * 8;
constexpr uint32_t kBytes = kOffMisc + 16;
constexpr uint32_t kDyn = kBytes + 1024;
constexpr uint32_t kTmemCols = 512;  // S^T: columns [0, 64); O^T tile i: [64 + 64 i, +64)
constexpr int kThreads = 192;
constexpr int kGatherWarps = 5;  // warp 0 and the four softmax warps
constexpr float kLazy = 8.f;     // log2 units the running max may lag behind

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;\n" ::: "memory");
}

// Rows j of the chunk with j % kGatherWarps == gw: two warp instructions of 512
// contiguous bytes per token row, into the row's place in each 128-byte atom.
__device__ __forceinline__ void gather_rows(uint8_t* sLat, const int* rows, const uint16_t* ckv,
                                            int gw, int lane) {
    const uint32_t lat = smem_u32(sLat);
    for (int j = gw; j < kT; j += kGatherWarps) {
        const long long row = rows[j];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int at = 4 * half + (lane >> 3), q = lane & 7;
            const uint16_t* src = ckv + row * kKVL + at * 64 + q * 8;
            const uint32_t dst = lat + at * kLatAtom + j * 128 + ((q ^ (j & 7)) << 4);
            cp_async16(dst, src, 16);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_tc_kernel(const __grid_constant__ CUtensorMap tmQ, MlaTcParams a) {
    pdl_wait();
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sQ = smem + kOffQ;
    uint8_t* sLat = smem + kOffLat;
    uint8_t* sP = smem + kOffP;
    float* red = reinterpret_cast<float*>(smem + kOffRed);
    int* rows = reinterpret_cast<int*>(smem + kOffRows);
    float* msm = reinterpret_cast<float*>(smem + kOffM);
    uint8_t* mask = smem + kOffMask;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint64_t* q_full = bars + 0;
    uint64_t* lat_full = bars + 1;
    uint64_t* lat_empty = bars + 2;
    uint64_t* s_full = bars + 3;
    uint64_t* p_full = bars + 4;
    uint64_t* o_done = bars + 5;
    uint64_t* red_bar = bars + 6;  // [2]
    uint64_t* sum_bar = bars + 8;
    uint64_t* drain = bars + 9;
    uint64_t* rows_ready = bars + 10;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, r = blockIdx.y;
    int seq = a.row_seq ? __ldg(a.row_seq + r) : r;
    int L = 0;
    if (seq >= 0 && seq < a.pg.batch) {
        L = min(__ldg(a.pg.seq_lens + seq), seq_capacity(a.pg));
    } else {
        if (threadIdx.x == 0 && split == 0) flag_status(a.status, DSA_STATUS_BAD_TOKEN);
        seq = 0;
    }
    const int t_begin = split * a.tps;
    const int t_end = min(t_begin + a.tps, a.ow);
    const int nch = t_end > t_begin ? (t_end - t_begin + kT - 1) / kT : 0;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(lat_full, kGatherWarps);
        mbar_init(lat_empty, 1);
        mbar_init(s_full, 1);
        mbar_init(p_full, 4);
        mbar_init(o_done, 1);
        mbar_init(red_bar + 0, 4);
        mbar_init(red_bar + 1, 4);
        mbar_init(sum_bar, 4);
        mbar_init(drain, 1);
        mbar_init(rows_ready, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (threadIdx.x < kH) msm[threadIdx.x] = __int_as_float(0xff800000);
    if (warp == 1) tc_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // one lane waits, the warp follows its verdict
    auto bwait = [&](uint64_t* bar, uint32_t parity) -> bool {
        int got = 1;
        if (lane == 0) got = wait_or_abort(bar, parity, abort_flag, a.status);
        return __shfl_sync(0xffffffffu, got, 0) != 0;
    };
    // this warp's share of chunk c's gather, then its arrival on lat_full
    auto gather_and_arrive = [&](int gw) {
        gather_rows(sLat, rows, a.ckv, gw, lane);
        cp_async_wait_all();
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(lat_full);
    };

    if (warp == 0) {
        // ---- Q once (TMA), then per chunk: token rows, rows_ready, a share of the gather
        if (lane == 0 && nch > 0) {
            mbar_arrive_expect_tx(q_full, kAtoms * kQAtom);
            for (int at = 0; at < kAtoms; ++at)
                tma_load_2d(smem_u32(sQ + at * kQAtom), &tmQ, 64 * at, r * kH, q_full);
        }
        for (int c = 0; c < nch; ++c) {
            if (!bwait(lat_empty, (uint32_t)(c & 1) ^ 1u)) break;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int j = 4 * lane + k;
                const int pos = t_begin + c * kT + j;
                long long prow = -1;
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
                mask[j] = prow >= 0 ? 1 : 0;
                rows[j] = prow >= 0 ? (int)prow : 0;  // a real row; masked in the softmax
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(rows_ready);
            gather_and_arrive(0);
        }
        if (lane == 0 && nch > 0) mbar_wait(q_full, 0);  // drain the Q copy
    } else if (warp == 1) {
        // ---- MMA issuer ----
        if (lane == 0) {
            constexpr uint32_t IDESC_QK = idesc_bf16(kT, kH);
            constexpr uint32_t IDESC_PV = idesc_bf16(128, kH) | (1u << 15) | (1u << 16);
            bool ok = nch == 0 || wait_or_abort(q_full, 0, abort_flag, a.status);
            const uint32_t q0 = smem_u32(sQ), l0 = smem_u32(sLat), p0 = smem_u32(sP);
            for (int c = 0; c < nch && ok; ++c) {
                if (!wait_or_abort(lat_full, (uint32_t)(c & 1), abort_flag, a.status)) break;
                tc_fence_after();
#pragma unroll 1
                for (int at = 0; at < kAtoms; ++at)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma(tmem, sw128_desc(l0 + at * kLatAtom + 32 * kk),
                               sw128_desc(q0 + at * kQAtom + 32 * kk), IDESC_QK,
                               (at | kk) != 0 ? 1u : 0u);
                tc_commit(s_full);
                if (!wait_or_abort(p_full, (uint32_t)(c & 1), abort_flag, a.status)) break;
                tc_fence_after();
#pragma unroll 1
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int kk = 0; kk < kT / 16; ++kk)
                        tc_mma(tmem + 64 + 64 * i,
                               sw128_desc_mn(l0 + 2 * i * kLatAtom + kk * 2048, kLatAtom, 1024),
                               sw128_desc_mn(p0 + kk * 2048, kQAtom, 1024), IDESC_PV,
                               (c > 0 || kk > 0) ? 1u : 0u);
                tc_commit(lat_empty);
                tc_commit(o_done);
            }
            // Drain: every MMA issued has completed before tensor memory is released.
            tc_commit(drain);
            mbar_wait(drain, 0);
        }
    } else {
        // ---- softmax and epilogue: thread j owns token j of a chunk (tensor lane j) ----
        const int qd = warp & 3;
        const int j = 32 * qd + lane;
        const uint32_t lrow = (uint32_t)(32 * qd) << 16;
        const float NEG_INF = __int_as_float(0xff800000);
        // Running maxima (identical in every thread) live in msm[c & 1] during chunk c;
        // the chunk's new ones go to msm[(c + 1) & 1].
        float lacc[kH];
#pragma unroll
        for (int h = 0; h < kH; ++h) lacc[h] = 0.f;
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            // a share of this chunk's gather
            if (!bwait(rows_ready, (uint32_t)(c & 1))) {
                ok = false;
                break;
            }
            gather_and_arrive(1 + (warp - 2));
            if (!bwait(s_full, (uint32_t)(c & 1))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const bool valid = mask[j] != 0;
            // chunk maximum per head: over the warp, then over the four warps
            const int b = c & 1;
            float* rb = red + b * 4 * kH;
            {
                uint32_t sv[2][32];
                tc_ld32(sv[0], tmem + lrow);
                tc_ld32(sv[1], tmem + lrow + 32);
                tc_wait_ld(sv[0]);
                tc_tie(sv[1]);
                float4* dst = reinterpret_cast<float4*>(rb + qd * kH);
#pragma unroll
                for (int i = 0; i < kH / 4; ++i) {
                    float4 m4;
                    m4.x = warp_max(valid ? __uint_as_float(sv[i >> 3][(4 * i) & 31]) * a.sl2 : NEG_INF);
                    m4.y = warp_max(valid ? __uint_as_float(sv[i >> 3][(4 * i + 1) & 31]) * a.sl2
                                          : NEG_INF);
                    m4.z = warp_max(valid ? __uint_as_float(sv[i >> 3][(4 * i + 2) & 31]) * a.sl2
                                          : NEG_INF);
                    m4.w = warp_max(valid ? __uint_as_float(sv[i >> 3][(4 * i + 3) & 31]) * a.sl2
                                          : NEG_INF);
                    if (lane == 0) dst[i] = m4;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(red_bar + b);
            if (!bwait(red_bar + b, (uint32_t)((c >> 1) & 1))) {
                ok = false;
                break;
            }
            // new running maxima (lagging by at most kLazy) into cm
            float cm[kH];
            {
                const float4* r4 = reinterpret_cast<const float4*>(rb);
#pragma unroll
                for (int i = 0; i < kH / 4; ++i) {
                    const float4 w0 = r4[i], w1 = r4[kH / 4 + i], w2 = r4[2 * (kH / 4) + i],
                                 w3 = r4[3 * (kH / 4) + i];
                    cm[4 * i] = fmaxf(fmaxf(w0.x, w1.x), fmaxf(w2.x, w3.x));
                    cm[4 * i + 1] = fmaxf(fmaxf(w0.y, w1.y), fmaxf(w2.y, w3.y));
                    cm[4 * i + 2] = fmaxf(fmaxf(w0.z, w1.z), fmaxf(w2.z, w3.z));
                    cm[4 * i + 3] = fmaxf(fmaxf(w0.w, w1.w), fmaxf(w2.w, w3.w));
                }
            }
            const float* mold = msm + b * kH;
            bool resc = false;
#pragma unroll
            for (int h = 0; h < kH; ++h) {
                const float mo = mold[h];
                const bool up = mo != NEG_INF && cm[h] > mo + kLazy;
                resc = resc || up;
                cm[h] = (mo == NEG_INF || up) ? cm[h] : mo;
            }
            if (resc) {
                // O^T through the previous chunk is complete before it is rescaled
                if (!bwait(o_done, (uint32_t)((c - 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int i = 0; i < 4; ++i) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t v[32];
                        const uint32_t addr = tmem + lrow + 64 + 64 * i + 32 * hh;
                        tc_ld32(v, addr);
                        tc_wait_ld(v);
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            const int h = 32 * hh + k;
                            const float f = mold[h] == NEG_INF ? 1.f : exp2f(mold[h] - cm[h]);
                            v[k] = __float_as_uint(__uint_as_float(v[k]) * f);
                        }
                        tc_st32(addr, v);
                    }
                }
                tc_wait_st();
            }
#pragma unroll
            for (int h = 0; h < kH; ++h)
                if (mold[h] != NEG_INF && cm[h] != mold[h]) lacc[h] *= exp2f(mold[h] - cm[h]);
            if (lane == 0) {  // every warp writes the same values
                float4* mn4 = reinterpret_cast<float4*>(msm + (b ^ 1) * kH);
#pragma unroll
                for (int i = 0; i < kH / 4; ++i)
                    mn4[i] = make_float4(cm[4 * i], cm[4 * i + 1], cm[4 * i + 2], cm[4 * i + 3]);
            }
            // probabilities (scores read again from tensor memory) as P^T row j in bf16
            {
                uint32_t sv[2][32];
                tc_ld32(sv[0], tmem + lrow);
                tc_ld32(sv[1], tmem + lrow + 32);
                tc_wait_ld(sv[0]);
                tc_tie(sv[1]);
                uint4* prow = reinterpret_cast<uint4*>(sP + j * 128);
#pragma unroll
                for (int q = 0; q < 8; ++q) {  // heads 8q .. 8q+7 -> one 16-byte chunk
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int h = 8 * q + 2 * e;
                        const float x0 = __uint_as_float(sv[h >> 5][h & 31]) * a.sl2;
                        const float x1 = __uint_as_float(sv[(h + 1) >> 5][(h + 1) & 31]) * a.sl2;
                        const float p0 = (valid && cm[h] != NEG_INF) ? exp2f(x0 - cm[h]) : 0.f;
                        const float p1 =
                            (valid && cm[h + 1] != NEG_INF) ? exp2f(x1 - cm[h + 1]) : 0.f;
                        lacc[h] += p0;
                        lacc[h + 1] += p1;
                        pk[e] = pack_bf16x2(p0, p1);
                    }
                    prow[q ^ (j & 7)] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }

        // ---- epilogue ----
        if (ok && nch > 0 && !bwait(o_done, (uint32_t)((nch - 1) & 1))) ok = false;
        // head sums: reduce-scatter over the warp (lane l ends with heads 2l, 2l+1),
        // then over the four warps through shared memory
        float v64[kH];
#pragma unroll
        for (int h = 0; h < kH; ++h) v64[h] = lacc[h];
#pragma unroll
        for (int w = kH / 2, m = 16; m >= 1; w >>= 1, m >>= 1) {
#pragma unroll
            for (int i = 0; i < w; ++i) {
                const bool hi = (lane & m) != 0;
                const float send = hi ? v64[i] : v64[w + i];
                const float recv = __shfl_xor_sync(0xffffffffu, send, m);
                v64[i] = (hi ? v64[w + i] : v64[i]) + recv;
            }
        }
        // [4 warps][kH] in the buffer the last chunk did not use: every warp finished
        // its reads of that one before the last chunk's scores existed
        float* sums = red + (nch & 1) * 4 * kH;
        sums[qd * kH + 2 * lane] = v64[0];
        sums[qd * kH + 2 * lane + 1] = v64[1];
        __syncwarp();
        if (lane == 0) mbar_arrive(sum_bar);
        if (!bwait(sum_bar, 0)) ok = false;
        if (ok) {
            if (a.ns > 1 && j < kH) {  // thread j writes head j's (m, l)
                const float mj = msm[(nch & 1) * kH + j];  // the last chunk's new maxima
                const float ls = (sums[j] + sums[kH + j]) + (sums[2 * kH + j] + sums[3 * kH + j]);
                *reinterpret_cast<float2*>(a.part_ml + (((long long)r * a.ns + split) * kH + j) * 2) =
                    make_float2(mj, ls);
            }
            const long long pbase = ((long long)r * a.ns + split) * kH;
            if (nch > 0) tc_fence_after();
#pragma unroll 1
            for (int i = 0; i < 4; ++i) {
                const int cidx = 128 * i + j;  // latent column = tensor lane of tile i
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t v[32];
                    if (nch > 0) {
                        tc_ld32(v, tmem + lrow + 64 + 64 * i + 32 * hh);
                        tc_wait_ld(v);
                    } else {
#pragma unroll
                        for (int k = 0; k < 32; ++k) v[k] = 0u;
                    }
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const int h = 32 * hh + k;
                        const float o = __uint_as_float(v[k]);
                        if (a.ns > 1) {
                            a.part_o[(pbase + h) * kKVL + cidx] = o;
                        } else {
                            const float ls = (sums[h] + sums[kH + h]) +
                                             (sums[2 * kH + h] + sums[3 * kH + h]);
                            const float val = ls > 0.f ? o / ls : 0.f;
                            const long long oi = ((long long)r * kH + h) * kKVL + cidx;
                            if (a.olat) a.olat[oi] = val;
                            if (a.xbf)
                                a.xbf[oi] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tc_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

// Opt-in (DSA_MLA_TC=1): at the sizes measured so far it is not faster than the
// mma.sync split kernel. At decode size each CTA runs its single chunk once and
// waits on instruction fetch; at prefill size its gather, QK, softmax and PV of a
// chunk run back to back (one latent buffer fits next to Q).
bool mla_tc_supported(int heads, int kv_lora_rank) {
    if (heads != kH || kv_lora_rank != kKVL) return false;
    const char* v = getenv("DSA_MLA_TC");
    return v && v[0] == '1';
}

int mla_tc_chunk() { return kT; }

int mla_tc_launch(const MlaTcParams& a, long long ckv_rows, cudaStream_t st) {
    if (ckv_rows < 1 || ckv_rows > 0x7fffffffLL)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_sparse_mla_decode: latent cache rows %lld",
                    ckv_rows);
    if ((long long)a.rows * kH > 0x7fffffffLL)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_sparse_mla_decode: too many rows");
    CUtensorMap tmQ;
    int rc = make_tmap_2d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.qlat, kKVL,
                          (uint64_t)a.rows * kH, kKVL * 2, 64, kH, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    rc = set_max_smem((const void*)mla_tc_kernel, (int)kDyn);
    if (rc) return rc;
    cudaError_t e = launch_pdl(mla_tc_kernel, dim3((unsigned)a.ns, (unsigned)a.rows), dim3(kThreads),
                               kDyn, st, tmQ, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_mla_decode tensor-core launch");
    return DSA_OK;
}

}  // namespace dsa
