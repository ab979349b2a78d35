// Sparse latent attention for decode batches on the tensor cores (tcgen05), 64 heads:
// one thread-block cluster per query row, each CTA attending a contiguous share of the
// row's selected tokens, the shares merged inside the cluster.
//
// Page: metrale_model_arch/glm5next_dsa/mod.rs, "Shape of the pipeline" (last stage)
// and build.rs module doc, transforms 1 and 3 (absorbed Q; each latent row is both key
// and value). Per row r, head h, over the selected tokens t of the CTA's share:
//   s[t,h] = softmax_scale * <ckv[t,:], qlat[r,h,:]>;  O[h,:] = sum_t p[t,h] ckv[t,:]
// with p = 2^(s*log2e - m_h) against a running per-head maximum m_h.
//
// A decode batch has few rows, so a persistent grid would leave most SMs without a
// full chunk; here the CS CTAs of a row's cluster each take 128-token chunks of their
// share (one or two at 2,048 selected tokens over 8 CTAs), and the cluster merges the
// shares itself: every CTA stores its unnormalised partial O and (m, l) per head,
// a cluster barrier (release / acquire) makes them visible, and CTA s then merges
// heads [64 s / CS, 64 (s + 1) / CS) over the CS partials in rank order and writes
// olat. No second launch, and the merge runs on every CTA of the cluster at once.
//
// Shared memory: Q (64 heads x 512, 64 KB), one 128-token latent tile (128 KB), P^T
// (16 KB), token rows of the whole share. Twenty warps:
//   - warp 0 (one lane) loads Q by TMA and issues the MMAs, accumulators in tensor
//     memory: S^T = K Q^T (M = 128 tokens, N = 64 heads, K = 512) quarter by quarter
//     as the tile lands; O^T += V^T P^T (M = 512 latent in four tiles, tile i = quarter
//     i of the token tile read MN-major, N = 64 heads, K = 128 tokens), each tile's
//     completion freeing its quarter for the next chunk;
//   - warps 1-19 resolve the share's token ids to cache rows, then gather the first
//     chunk with cp.async into the 128-byte-swizzled atoms (each thread's copies
//     complete on the quarter's mbarrier); warps 1-3 gather later chunks as quarters
//     free up, and so do the softmax warps, right after their softmax of the chunk
//     before;
//   - warps 4-19 (one tensor-memory lane, i.e. one token, and 16 of the heads per
//     thread: four warps per lane quarter) take S^T, keep a running maximum per head
//     (moved, and O^T rescaled, only when a chunk raises it by more than 2^8), write
//     P^T in bf16 and accumulate the row sums; at the end they store the partial.
// All mbarrier waits are bounded: a timeout sets DSA_STATUS_TIMEOUT, the roles leave
// their loops, copies and MMAs in flight are drained, and tensor memory is released.
#include "common.cuh"
#include "tc.cuh"

namespace dsa {
namespace {

constexpr int kT = 128;                          // tokens per chunk
constexpr int kH = 64;                           // heads
constexpr int kKVL = 512;                        // latent width
constexpr int kAtoms = kKVL / 64;                // 128-byte atoms per latent row
constexpr int kQuarters = 4;                     // two atoms each
constexpr int kMaxTok = 1024;                    // tokens per CTA (eight chunks)
constexpr int kMaxSplit = 32;                    // CTAs per row
constexpr uint32_t kLatAtom = kT * 128;          // one atom of the token tile
constexpr uint32_t kQAtom = kH * 128;            // one atom of the Q tile
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffLat = kOffQ + kAtoms * kQAtom;
constexpr uint32_t kOffP = kOffLat + kAtoms * kLatAtom;
constexpr uint32_t kOffRed = kOffP + kT * 128;         // [4 lane quarters][kH] chunk maxima
constexpr uint32_t kOffSums = kOffRed + 4 * kH * 4;    // [4 lane quarters][kH] row sums
constexpr uint32_t kOffRows = kOffSums + 4 * kH * 4;   // [kMaxTok] cache row per token
constexpr uint32_t kOffMask = kOffRows + kMaxTok * 4;  // [kMaxTok] token valid
constexpr uint32_t kOffW = kOffMask + kMaxTok;         // merge weights [CS][kH]
constexpr uint32_t kOffL = kOffW + 8 * kH * 4;         // merge sums [kH]
constexpr uint32_t kOffMold = kOffL + kH * 4;          // running maxima before a chunk [kH]
constexpr uint32_t kOffBar = kOffMold + kH * 4;
// mbarriers
constexpr int Q_FULL = 0;
constexpr int LAT_FULL = 1;   // [4] a quarter gathered (the gather threads' copies)
constexpr int LAT_EMPTY = 5;  // [4] a quarter's PV tile done (commit)
constexpr int S_FULL = 9;     // S^T of a chunk complete (commit)
constexpr int P_FULL = 10;    // P^T written, S^T read (the softmax warps)
constexpr int O_DONE = 11;    // the last PV done (commit)
constexpr int DRAIN = 12;     // every MMA issued has completed
constexpr int kBars = 13;
constexpr uint32_t kOffMisc = kOffBar + kBars * 8;
constexpr uint32_t kBytes = kOffMisc + 16;
constexpr uint32_t kDyn = kBytes + 1024;  // room to align the base to 1024 bytes
constexpr uint32_t kTmemCols = 512;        // S^T: columns [0, 64); O^T tile i: [64 + 64 i, +64)
constexpr int kSoftWarps = 16;                     // four per tensor-memory lane quarter
constexpr int kWarps = 4 + kSoftWarps;
constexpr int kThreads = kWarps * 32;
constexpr int kGatherThreads = (kWarps - 1) * 32;  // warps 1-19
constexpr int kHPW = kH / 4;                       // heads per softmax thread
constexpr float kLazy = 8.f;  // log2 units the running maximum may lag behind
static_assert(kDyn <= 227 * 1024, "decode attention shared memory");
static_assert(kOffBar % 8 == 0, "mbarrier alignment");
static_assert(kGatherThreads % 16 == 0, "gather threads");

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ float4 ldcg4(const float* p) {
    return __ldcg(reinterpret_cast<const float4*>(p));
}
// 16 consecutive f32 columns of this thread's tensor-memory lane, and the matching
// store; each wait ties the registers so that no use is scheduled before it.
__device__ __forceinline__ void tc_ld16(uint32_t (&v)[16], uint32_t taddr) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];\n"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld16(uint32_t (&v)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;\n"
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                   "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                   "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15])
                 :
                 : "memory");
}
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};\n" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
        : "memory");
}

// Quarter q of a chunk (atoms 2q, 2q+1: latent columns 128q .. 128q+127 of every
// token): 2048 copies of 16 bytes. Gather thread g keeps one (atom, 16-byte chunk)
// pair, g & 15, and steps over the chunk's tokens g / 16, + kGatherThreads / 16, ...
__device__ __forceinline__ void gather_quarter(uint32_t lat, const int* rows, const uint16_t* ckv,
                                               int q, int g) {
    const int c = g & 7, at = 2 * q + ((g >> 3) & 1);
    const uint32_t dst0 = lat + at * kLatAtom;
    const uint16_t* src0 = ckv + at * 64 + c * 8;
    constexpr int kStep = kGatherThreads / 16;
    const int j0 = g >> 4;
#pragma unroll
    for (int m = 0; m < (kT + kStep - 1) / kStep; ++m) {
        const int j = j0 + kStep * m;
        if (j < kT)
            cp_async16(dst0 + j * 128 + ((c ^ (j & 7)) << 4), src0 + (long long)rows[j] * kKVL, 16);
    }
}

struct DecArgs {
    const int32_t* row_seq;
    const uint16_t* ckv;
    const int32_t* token_ids;
    float* part_o;   // [rows, CS, kH, kKVL]
    float* part_ml;  // [rows, CS, kH, 2]
    float* olat;     // nullable
    uint16_t* xbf;   // nullable: bf16 copy of olat
    int32_t* status;
    Paging pg;
    int ow;
    int cs;     // CTAs per row
    int tps;    // tokens per CTA (a multiple of kT)
    int merge;  // 1: a row's CTAs form a cluster and merge their partials into olat
    float sl2;
};

__global__ void __launch_bounds__(kThreads, 1)
    mla_dec_kernel(const __grid_constant__ CUtensorMap tmQ, DecArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sQ = smem + kOffQ;
    uint8_t* sLat = smem + kOffLat;
    uint8_t* sP = smem + kOffP;
    float* red = reinterpret_cast<float*>(smem + kOffRed);
    float* sums = reinterpret_cast<float*>(smem + kOffSums);
    int* rows = reinterpret_cast<int*>(smem + kOffRows);
    uint8_t* mask = smem + kOffMask;
    float* wsm = reinterpret_cast<float*>(smem + kOffW);
    float* lsm = reinterpret_cast<float*>(smem + kOffL);
    float* mold = reinterpret_cast<float*>(smem + kOffMold);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int CS = a.cs;
    const int r = blockIdx.x / CS;
    const int split = blockIdx.x - r * CS;  // the CTA's rank in its (one-dimensional) cluster
    const int t_begin = split * a.tps;
    const int t_end = min(t_begin + a.tps, a.ow);
    const int ntok = max(0, t_end - t_begin);
    const int nch = (ntok + kT - 1) / kT;

    if (threadIdx.x == 0) {
        mbar_init(bars + Q_FULL, 1);
        for (int q = 0; q < kQuarters; ++q) {
            mbar_init(bars + LAT_FULL + q, kGatherThreads);
            mbar_init(bars + LAT_EMPTY + q, 1);
        }
        mbar_init(bars + S_FULL, 1);
        mbar_init(bars + P_FULL, kSoftWarps);
        mbar_init(bars + O_DONE, 1);
        mbar_init(bars + DRAIN, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tc_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // token ids, qlat and the caches come from the kernels before this one
    pdl_wait();
    if (threadIdx.x == 0 && nch > 0) {
        mbar_arrive_expect_tx(bars + Q_FULL, kAtoms * kQAtom);
        for (int at = 0; at < kAtoms; ++at)
            tma_load_2d(smem_u32(sQ + at * kQAtom), &tmQ, 64 * at, r * kH, bars + Q_FULL);
    }

    // ---- the share's token ids -> cache rows (bounds against the cache's capacity
    // first, so the gather can start; the sequence length masks afterwards)
    int seq = a.row_seq ? __ldg(a.row_seq + r) : r;
    const bool seq_ok = seq >= 0 && seq < a.pg.batch;
    if (!seq_ok) {
        if (threadIdx.x == 0 && split == 0) flag_status(a.status, DSA_STATUS_BAD_TOKEN);
        seq = 0;
    }
    const int cap = seq_capacity(a.pg);
    for (int j = threadIdx.x; j < nch * kT; j += kThreads) {
        const int pos = t_begin + j;
        long long prow = -1;
        if (pos < t_end && seq_ok) {
            const int t = __ldg(a.token_ids + (long long)r * a.ow + pos);
            if (t >= 0 && t < cap) {
                prow = token_row(a.pg, seq, t);
                if (prow < 0) flag_status(a.status, DSA_STATUS_BAD_BLOCK);
                const int L = min(__ldg(a.pg.seq_lens + seq), cap);
                if (t >= L) {
                    flag_status(a.status, DSA_STATUS_BAD_TOKEN);
                    mask[j] = 0;  // gathered (in range of the cache) but not attended
                } else {
                    mask[j] = prow >= 0 ? 1 : 0;
                }
            } else {
                if (t < -1 || t >= cap) flag_status(a.status, DSA_STATUS_BAD_TOKEN);
                mask[j] = 0;
            }
        } else {
            mask[j] = 0;
        }
        rows[j] = prow >= 0 ? (int)prow : 0;  // a real row; masked tokens are not attended
    }
    __syncthreads();

    const uint32_t lat = smem_u32(sLat);
    bool ok = true;
    if (warp == 0) {
        // ---------------- MMA issuer ----------------
        if (lane == 0 && nch > 0) {
            constexpr uint32_t IDESC_QK = idesc_bf16(kT, kH);
            constexpr uint32_t IDESC_PV = idesc_bf16(128, kH) | (1u << 15) | (1u << 16);
            const uint32_t q0 = smem_u32(sQ), p0 = smem_u32(sP);
            if (wait_or_abort(bars + Q_FULL, 0, abort_flag, a.status)) {
                for (int c = 0; c < nch && ok; ++c) {
                    for (int q = 0; q < kQuarters && ok; ++q) {
                        if (!wait_or_abort(bars + LAT_FULL + q, (uint32_t)(c & 1), abort_flag,
                                           a.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int at = 2 * q + h;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                tc_mma(tmem, sw128_desc(lat + at * kLatAtom + 32 * kk),
                                       sw128_desc(q0 + at * kQAtom + 32 * kk), IDESC_QK,
                                       (at | kk) != 0 ? 1u : 0u);
                        }
                    }
                    if (!ok) break;
                    tc_commit(bars + S_FULL);
                    if (!wait_or_abort(bars + P_FULL, (uint32_t)(c & 1), abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int i = 0; i < kQuarters; ++i) {
#pragma unroll
                        for (int kk = 0; kk < kT / 16; ++kk)
                            tc_mma(tmem + 64 + 64 * i,
                                   sw128_desc_mn(lat + 2 * i * kLatAtom + kk * 2048, kLatAtom, 1024),
                                   sw128_desc_mn(p0 + kk * 2048, kQAtom, 1024), IDESC_PV,
                                   (c > 0 || kk > 0) ? 1u : 0u);
                        tc_commit(bars + LAT_EMPTY + i);
                    }
                    if (c == nch - 1) tc_commit(bars + O_DONE);
                }
            }
            // every MMA issued has completed before tensor memory is read or released
            tc_commit(bars + DRAIN);
            mbar_wait(bars + DRAIN, 0);
        }
    } else {
        // ---------------- gather of the first chunk (warps 1-19) ----------------
        const int g = threadIdx.x - 32;
        if (nch > 0) {
            for (int q = 0; q < kQuarters; ++q) {
                gather_quarter(lat, rows, a.ckv, q, g);
                cp_async_arrive_noinc(bars + LAT_FULL + q);
            }
        }
        if (warp < 4) {
            // ---- later chunks: quarters as the PV of the chunk before frees them ----
            for (int c = 1; c < nch && ok; ++c) {
                for (int q = 0; q < kQuarters; ++q) {
                    int got = 1;
                    if (lane == 0)
                        got = wait_or_abort(bars + LAT_EMPTY + q, (uint32_t)((c - 1) & 1), abort_flag,
                                            a.status);
                    if (!__shfl_sync(0xffffffffu, got, 0)) {
                        ok = false;
                        break;
                    }
                    gather_quarter(lat, rows + c * kT, a.ckv, q, g);
                    cp_async_arrive_noinc(bars + LAT_FULL + q);
                }
            }
        } else {
            // ---- softmax (warps 4-19): thread = token lane 32 qd + lane, heads
            // h0 .. h0 + 15 (head quarter hq; four warps, one per lane quarter, per hq)
            const int qd = warp & 3;
            const int hq = (warp - 4) >> 2;
            const int h0 = kHPW * hq;
            const int j = 32 * qd + lane;
            const uint32_t lrow = (uint32_t)(32 * qd) << 16;
            const float NEG_INF = __int_as_float(0xff800000);
            float m_run[kHPW], lacc[kHPW];
#pragma unroll
            for (int h = 0; h < kHPW; ++h) {
                m_run[h] = NEG_INF;
                lacc[h] = 0.f;
            }
            auto bwait = [&](int bar, uint32_t parity) -> bool {
                int got = 1;
                if (lane == 0) got = wait_or_abort(bars + bar, parity, abort_flag, a.status);
                return __shfl_sync(0xffffffffu, got, 0) != 0;
            };
            // Every warp of a head quarter passes the same named barriers in the same
            // order whatever its waits return (a wait that gave up only skips work), so
            // an aborted wait never leaves a partner warp at a barrier.
            for (int c = 0; c < nch; ++c) {
                if (ok && !bwait(S_FULL, (uint32_t)(c & 1))) ok = false;
                uint32_t sv[kHPW];
                bool valid = false;
                if (ok) {
                    tc_fence_after();
                    tc_ld16(sv, tmem + lrow + h0);
                    tc_wait_ld16(sv);
                    valid = mask[c * kT + j] != 0;
                    // the running maxima before this chunk (identical in the four warps
                    // of a head quarter), kept for a rescale
                    if (qd == 0 && lane == 0) {
                        float4* mo4 = reinterpret_cast<float4*>(mold + h0);
#pragma unroll
                        for (int i = 0; i < kHPW / 4; ++i)
                            mo4[i] = make_float4(m_run[4 * i], m_run[4 * i + 1], m_run[4 * i + 2],
                                                 m_run[4 * i + 3]);
                    }
                    // chunk maxima of this warp's 32 tokens
                    float4* dst = reinterpret_cast<float4*>(red + qd * kH + h0);
#pragma unroll
                    for (int i = 0; i < kHPW / 4; ++i) {
                        float4 m4;
                        m4.x = warp_max(valid ? __uint_as_float(sv[4 * i]) * a.sl2 : NEG_INF);
                        m4.y = warp_max(valid ? __uint_as_float(sv[4 * i + 1]) * a.sl2 : NEG_INF);
                        m4.z = warp_max(valid ? __uint_as_float(sv[4 * i + 2]) * a.sl2 : NEG_INF);
                        m4.w = warp_max(valid ? __uint_as_float(sv[4 * i + 3]) * a.sl2 : NEG_INF);
                        if (lane == 0) dst[i] = m4;
                    }
                }
                named_sync(1 + hq, 128);  // the four lane quarters of this head quarter
                bool resc = false;
                if (ok) {
#pragma unroll
                    for (int i = 0; i < kHPW / 4; ++i) {
                        float4 w4 = reinterpret_cast<const float4*>(red + h0)[i];
#pragma unroll
                        for (int q = 1; q < 4; ++q) {
                            const float4 v4 = reinterpret_cast<const float4*>(red + q * kH + h0)[i];
                            w4.x = fmaxf(w4.x, v4.x);
                            w4.y = fmaxf(w4.y, v4.y);
                            w4.z = fmaxf(w4.z, v4.z);
                            w4.w = fmaxf(w4.w, v4.w);
                        }
                        const float cm4[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int h = 4 * i + e;
                            const float mo = m_run[h];
                            // move the running maximum only when it lags by more than kLazy
                            const bool up =
                                cm4[e] != NEG_INF && (mo == NEG_INF || cm4[e] > mo + kLazy);
                            resc = resc || (up && mo != NEG_INF);
                            m_run[h] = up ? cm4[e] : mo;
                        }
                    }
                }
                // the maxima of this chunk are read: the next chunk may overwrite them
                named_sync(1 + hq, 128);
                if (!ok) continue;
                if (resc) {
                    // O^T through the previous chunk is complete: S_FULL of this chunk
                    // was committed after that chunk's PV. Factor 2^(m_old - m_new) per
                    // head (1 where the maximum did not move).
#pragma unroll 1
                    for (int i = 0; i < kQuarters; ++i) {
                        uint32_t v[kHPW];
                        const uint32_t addr = tmem + lrow + 64 + 64 * i + h0;
                        tc_ld16(v, addr);
                        tc_wait_ld16(v);
#pragma unroll
                        for (int kk = 0; kk < kHPW; ++kk) {
                            const float mo = mold[h0 + kk];
                            const float f =
                                (mo == NEG_INF || mo == m_run[kk]) ? 1.f : exp2f(mo - m_run[kk]);
                            v[kk] = __float_as_uint(__uint_as_float(v[kk]) * f);
                        }
                        tc_st16(addr, v);
                    }
                    tc_wait_st();
#pragma unroll
                    for (int h = 0; h < kHPW; ++h) {
                        const float mo = mold[h0 + h];
                        if (mo != NEG_INF && mo != m_run[h]) lacc[h] *= exp2f(mo - m_run[h]);
                    }
                }
                // probabilities into row j of P^T (bf16), and the row sums of what the
                // MMA will use
                {
                    uint4* prow = reinterpret_cast<uint4*>(sP + j * 128);
#pragma unroll
                    for (int q = 0; q < kHPW / 8; ++q) {  // heads h0 + 8q .. +7 -> one 16-byte chunk
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int h = 8 * q + 2 * e;
                            const float x0 = __uint_as_float(sv[h]) * a.sl2;
                            const float x1 = __uint_as_float(sv[h + 1]) * a.sl2;
                            const float p0 =
                                (valid && m_run[h] != NEG_INF) ? ex2_sfu(x0 - m_run[h]) : 0.f;
                            const float p1 =
                                (valid && m_run[h + 1] != NEG_INF) ? ex2_sfu(x1 - m_run[h + 1]) : 0.f;
                            pk[e] = pack_bf16x2(p0, p1);
                            lacc[h] += bf16_lo(pk[e]);
                            lacc[h + 1] += bf16_hi(pk[e]);
                        }
                        prow[((h0 >> 3) + q) ^ (j & 7)] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars + P_FULL);
                // this warp's share of the next chunk's gather, quarter by quarter as
                // this chunk's PV frees them
                if (c + 1 < nch) {
                    for (int q = 0; q < kQuarters; ++q) {
                        if (!bwait(LAT_EMPTY + q, (uint32_t)(c & 1))) {
                            ok = false;
                            break;
                        }
                        gather_quarter(lat, rows + (c + 1) * kT, a.ckv, q, g);
                        cp_async_arrive_noinc(bars + LAT_FULL + q);
                    }
                }
            }

            // ---- the CTA's partial: (m, l) per head and unnormalised O ----
            const long long pbase = ((long long)r * CS + split) * kH;
            const bool have = ok && nch > 0 && bwait(O_DONE, 0);
            if (have) {
                tc_fence_after();
                // the final running maxima, for the (m, l) pairs below
                if (qd == 0 && lane == 0) {
                    float4* mo4 = reinterpret_cast<float4*>(mold + h0);
#pragma unroll
                    for (int i = 0; i < kHPW / 4; ++i)
                        mo4[i] = make_float4(m_run[4 * i], m_run[4 * i + 1], m_run[4 * i + 2],
                                             m_run[4 * i + 3]);
                }
                // row sums over the warp's 32 tokens: fold the two half-warps, then a
                // reduce-scatter over 16 lanes (lane l < 16 ends with head h0 + l)
                float v16[kHPW];
#pragma unroll
                for (int h = 0; h < kHPW; ++h) v16[h] = lacc[h] + __shfl_xor_sync(0xffffffffu, lacc[h], 16);
#pragma unroll
                for (int ww = 8, m = 8; m >= 1; ww >>= 1, m >>= 1) {
#pragma unroll
                    for (int i = 0; i < ww; ++i) {
                        const bool hi = (lane & m) != 0;
                        const float send = hi ? v16[i] : v16[ww + i];
                        const float recv = __shfl_xor_sync(0xffffffffu, send, m);
                        v16[i] = (hi ? v16[ww + i] : v16[i]) + recv;
                    }
                }
                if (lane < kHPW) sums[qd * kH + h0 + lane] = v16[0];
            }
            named_sync(1 + hq, 128);  // every lane quarter's sums are in place
            if (qd == 0 && lane < kHPW) {
                // (m, l) per head; no tokens (or a wait that gave up): an empty share,
                // weight 0 in the merge
                const int hd = h0 + lane;
                float2 ml = make_float2(NEG_INF, 0.f);
                if (have)
                    ml = make_float2(mold[hd], (sums[hd] + sums[kH + hd]) +
                                                   (sums[2 * kH + hd] + sums[3 * kH + hd]));
                *reinterpret_cast<float2*>(a.part_ml + (pbase + hd) * 2) = ml;
            }
            if (have) {
#pragma unroll 1
                for (int i = 0; i < kQuarters; ++i) {
                    const int cidx = 128 * i + j;  // latent column = tensor lane of tile i
                    uint32_t v[kHPW];
                    tc_ld16(v, tmem + lrow + 64 + 64 * i + h0);
                    tc_wait_ld16(v);
#pragma unroll
                    for (int kk = 0; kk < kHPW; ++kk)
                        a.part_o[(pbase + h0 + kk) * kKVL + cidx] = __uint_as_float(v[kk]);
                }
            }
        }
        cp_async_wait_all();  // drain this thread's copies
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tc_dealloc(tmem, kTmemCols);
    }

    if (!a.merge) return;  // the partials go to the combine kernel

    // ---- merge the row's CS partials: this CTA takes heads [hA, hB) ----
    const float NEG_INF_F = __int_as_float(0xff800000);
    cluster_sync_all();  // every CTA's partial is written and visible
    const int hA = split * kH / CS, hB = (split + 1) * kH / CS;
    const long long rbase = (long long)r * CS * kH;
    const int nitems = (hB - hA) * 8;
    for (int i0 = 0; i0 < nitems; i0 += kThreads) {
        // (head, split) weights 2^(m_s - M) and the merged sum L; lanes 8k .. 8k+7 of
        // a warp hold the eight splits of one head (the whole warp shuffles)
        const int i = i0 + threadIdx.x;
        const int hl = i >> 3, s = i & 7;
        const int h = hA + hl;
        const bool act = i < nitems;
        float m = NEG_INF_F, l = 0.f;
        if (act && s < CS) {
            const float2 ml =
                __ldcg(reinterpret_cast<const float2*>(a.part_ml) + rbase + (long long)s * kH + h);
            m = ml.x;
            l = ml.y;
        }
        float M = m;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float w = m == NEG_INF_F ? 0.f : exp2f(m - M);
        float L = w * l;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (act && s < CS) wsm[s * kH + h] = w;
        if (act && s == 0) lsm[h] = L;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < (hB - hA) * (kKVL / 4); i += kThreads) {
        const int h = hA + i / (kKVL / 4);
        const int c4 = i % (kKVL / 4);
        // all splits' values requested before any is used
        float4 v[8];
#pragma unroll
        for (int s = 0; s < 8; ++s)
            v[s] = (s < CS && wsm[s * kH + h] != 0.f)
                       ? ldcg4(a.part_o + ((rbase + (long long)s * kH + h) * kKVL) + 4 * c4)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const float w = s < CS ? wsm[s * kH + h] : 0.f;
            if (w != 0.f) {
                acc.x += w * v[s].x;
                acc.y += w * v[s].y;
                acc.z += w * v[s].z;
                acc.w += w * v[s].w;
            }
        }
        const float L = lsm[h];
        const float inv = L > 0.f ? 1.f / L : 0.f;
        acc.x *= inv;
        acc.y *= inv;
        acc.z *= inv;
        acc.w *= inv;
        const long long o = ((long long)r * kH + h) * kKVL + 4 * c4;
        if (a.olat) *reinterpret_cast<float4*>(a.olat + o) = acc;
        if (a.xbf) {
            uint2 v;
            v.x = pack_bf16x2(acc.x, acc.y);
            v.y = pack_bf16x2(acc.z, acc.w);
            *reinterpret_cast<uint2*>(a.xbf + o) = v;
        }
    }
}

}  // namespace

bool mla_dec_supported(int heads, int kv_lora_rank, int ow) {
    return heads == kH && kv_lora_rank == kKVL && ow > 0 && ow <= kMaxSplit * kMaxTok;
}

// CTAs per row and tokens per CTA. Up to 8 chunks of 128 tokens a row is one cluster
// with a chunk per CTA, merged in the kernel; longer rows take one chunk per CTA
// without a cluster (the combine kernel merges), up to kMaxSplit CTAs per row.
void mla_dec_plan(int ow, int* cs, int* tps, bool* merge) {
    const int chunks = (ow + kT - 1) / kT;
    const int c0 = chunks < kMaxSplit ? chunks : kMaxSplit;
    const int per = (chunks + c0 - 1) / c0;
    *tps = per * kT;
    *cs = (ow + *tps - 1) / *tps;
    *merge = *cs <= 8;
}

int mla_dec_launch(const MlaTcParams& p, long long ckv_rows, cudaStream_t st) {
    if (ckv_rows < 1 || ckv_rows > 0x7fffffffLL)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_sparse_mla_decode: latent cache rows %lld", ckv_rows);
    int cs = 0, tps = 0;
    bool merge = false;
    mla_dec_plan(p.ow, &cs, &tps, &merge);
    if (cs != p.ns || tps != p.tps)
        return fail(DSA_ERR_INVALID_ARG, "dsa_sparse_mla_decode: decode plan mismatch");
    if ((long long)p.rows * cs > 0x7fffffffLL)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_sparse_mla_decode: too many rows");
    CUtensorMap tmQ;
    int rc = make_tmap_2d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.qlat, kKVL,
                          (uint64_t)p.rows * kH, kKVL * 2, 64, kH, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    rc = set_max_smem((const void*)mla_dec_kernel, (int)kDyn);
    if (rc) return rc;
    DecArgs a;
    a.row_seq = p.row_seq;
    a.ckv = p.ckv;
    a.token_ids = p.token_ids;
    a.part_o = p.part_o;
    a.part_ml = p.part_ml;
    a.olat = p.olat;
    a.xbf = p.xbf;
    a.status = p.status;
    a.pg = p.pg;
    a.ow = p.ow;
    a.cs = cs;
    a.tps = tps;
    a.merge = merge ? 1 : 0;
    a.sl2 = p.sl2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.rows * cs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kDyn;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = merge ? (unsigned)cs : 1u;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, mla_dec_kernel, tmQ, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_mla_decode decode launch");
    return DSA_OK;
}

}  // namespace dsa
