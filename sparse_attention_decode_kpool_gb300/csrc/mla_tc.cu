// Sparse latent attention on the tensor cores (tcgen05) for 64 heads: the split
// kernel of dsa_sparse_mla_decode when heads == 64 and the batch holds enough
// 128-token chunks to keep a persistent grid busy (prefill chunks).
//
// Page: metrale_model_arch/glm5next_dsa/mod.rs, "Shape of the pipeline" (last stage)
// and build.rs module doc, transforms 1 and 3 (absorbed Q; each latent row is both
// key and value). Per row r, head h, over the selected tokens t of a split:
//   s[t,h] = softmax_scale * <ckv[t,:], qlat[r,h,:]>;  O[h,:] = sum_t p[t,h] ckv[t,:]
// with p = 2^(s*log2e - m_h) against a running per-head maximum m_h.
//
// The grid is persistent: CTA b takes the (row, split) units b, b + G, b + 2G, ...
// and walks each unit's tokens in chunks of 128. Shared memory holds the unit's Q
// (64 heads x 512, 64 KB), one 128-token latent tile (128 KB) and P^T (16 KB); there
// is no room for a second tile, so the tile is refilled a quarter (two 64-column
// atoms, the rows of one O^T tile) at a time, as soon as the MMAs of the previous
// chunk are done with that quarter. Roles (sixteen warps, four warpgroups):
//   - warp 0 resolves each chunk's token ids to cache rows, two chunks ahead, into a
//     double buffer, and loads each unit's Q by TMA once the last unit's QK is done;
//   - warps 2-3 and 12-15 gather, and so do the softmax warps (each chunk's share
//     right after their softmax of the chunk before): per quarter, 128 tokens x 256
//     bytes with cp.async into the 128-byte-swizzled atoms, each thread's copies
//     completing on the quarter's mbarrier (cp.async.mbarrier.arrive.noinc);
//   - warp 1 (one lane) issues the MMAs, accumulators in tensor memory:
//       S^T = K Q^T   M = 128 tokens, N = 64 heads, K = 512, quarter by quarter;
//       O^T += V^T P^T  M = 512 latent (four tiles of 128, tile i = quarter i read
//       MN-major), N = 64 heads, K = 128 tokens; each tile's completion frees its
//       quarter for the next chunk's gather;
//   - warps 4-11 (one tensor-memory lane, i.e. one token, and half of the heads per
//     thread: two warps per lane quarter) take S^T and keep a lazy running maximum
//     per head: a warp vote asks whether any score moves a maximum by more than 2^8
//     (or there is none yet); only such warps publish chunk maxima (redux.sync, then
//     shared memory), and only then are the maxima moved and O^T and the partial sums
//     rescaled. They write P^T in bf16 (ex2 on the special-function unit) and, at the
//     end of a unit, its partial (or, with one split, olat), then free O^T.
// All waits are bounded; a timeout sets DSA_STATUS_TIMEOUT, every role leaves its
// loops, copies and MMAs in flight are drained, and the tensor memory is released.
#include "common.cuh"
#include "fp8.cuh"
#include "tc.cuh"

namespace dsa {
namespace {

constexpr int kT = 128;                        // tokens per chunk
constexpr int kH = 64;                         // heads
constexpr int kKVL = 512;                      // latent width
constexpr int kAtoms = kKVL / 64;              // 128-byte atoms per latent row
constexpr int kQuarters = 4;                   // two atoms each
constexpr uint32_t kLatAtom = kT * 128;        // one atom of the token tile
constexpr uint32_t kQAtom = kH * 128;          // one atom of the Q tile
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffLat = kOffQ + kAtoms * kQAtom;
constexpr uint32_t kOffP = kOffLat + kAtoms * kLatAtom;
constexpr uint32_t kOffRed = kOffP + kT * 128;          // [2][4 warps][kH] f32 chunk maxima
constexpr uint32_t kOffSums = kOffRed + 2 * 4 * kH * 4; // [4 warps][kH] f32 head sums
constexpr uint32_t kOffM = kOffSums + 4 * kH * 4;       // [2][kH] running maxima
constexpr uint32_t kOffRows = kOffM + 2 * kH * 4;       // [2][kT] cache row per token
constexpr uint32_t kOffMask = kOffRows + 2 * kT * 4;    // [2][kT] token valid
constexpr uint32_t kOffFlag = kOffMask + 2 * kT;      // [2][8 softmax warps] maxima written
constexpr uint32_t kOffBar = kOffFlag + 2 * 8 * 4;
// mbarriers
constexpr int Q_FULL = 0;         // Q landed (TMA bytes)
constexpr int Q_EMPTY = 1;        // the unit's last QK is done with Q (commit)
constexpr int ROWS_FULL = 2;      // [2] token rows of a chunk resolved (warp 0)
constexpr int ROWS_EMPTY = 4;     // [2] rows and mask read (2 gather + 4 softmax warps)
constexpr int LAT_FULL = 6;       // [4] a quarter gathered (64 gather threads' copies)
constexpr int LAT_EMPTY = 10;     // [4] a quarter's PV tile done (commit)
constexpr int S_FULL = 14;        // S^T of a chunk complete (commit)
constexpr int P_FULL = 15;        // P^T written, S^T read (4 softmax warps)
constexpr int O_DONE = 16;        // the unit's last PV done (commit)
constexpr int O_FREE = 17;        // the unit's O^T read out (4 softmax warps)
constexpr int RED = 18;           // [2] chunk maxima of all four warps in place
constexpr int SUM_IN = 20;        // head sums of all four warps in place
constexpr int SUM_OUT = 21;       // head sums read by all four warps
constexpr int DRAIN = 22;         // every MMA issued has completed
constexpr int kBars = 23;
constexpr uint32_t kOffMisc = kOffBar + kBars * 8;
constexpr uint32_t kBytes = kOffMisc + 16;
constexpr uint32_t kDyn = kBytes + 1024;
constexpr uint32_t kTmemCols = 512;  // S^T: columns [0, 64); O^T tile i: [64 + 64 i, +64)
// Four warpgroups. 0: warp 0 token rows and Q, warp 1 MMA issue, warps 2-3 gather;
// 1 and 2: softmax (warps 4-11, two per tensor-memory lane quarter); 3: gather
// (warps 12-15). Launched at 128 registers a thread; the softmax warpgroups raise
// theirs to 176 and the others lower theirs to 80 (setmaxnreg), which adds up to
// the launch's 512 x 128 exactly, in every SM sub-partition too (one warp of each
// warpgroup per sub-partition).
constexpr int kSoftWarps = 8;
constexpr int kGatherWarps = 6;
constexpr int kThreads = 16 * 32;
constexpr int kGatherThreads = kGatherWarps * 32;
// The softmax warps gather too: each chunk's share right after their softmax of the
// chunk before, while the PV that frees the tile runs.
constexpr int kCopyThreads = (kGatherWarps + kSoftWarps) * 32;
constexpr int kRegLow = 80, kRegHigh = 176;
static_assert(2 * kRegLow + 2 * kRegHigh == 4 * 128, "register split");
constexpr float kLazy = 8.f;         // log2 units the running max may lag behind
static_assert(kDyn <= 227 * 1024, "tcgen05 attention shared memory");
static_assert(kOffBar % 8 == 0, "mbarrier alignment");

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;\n" ::: "memory");
}
// Arrive on bar once every cp.async this thread issued so far has landed (the
// arrival counts against the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar))
                 : "memory");
}

// Token range of a unit: split `split` of its row, in chunks of kT.
struct Unit {
    int r, split, t_begin, t_end, nch;
};
__device__ __forceinline__ Unit unit_of(const MlaTcParams& a, int u) {
    Unit w;
    w.r = u / a.ns;
    w.split = u - w.r * a.ns;
    w.t_begin = w.split * a.tps;
    w.t_end = min(w.t_begin + a.tps, a.ow);
    w.nch = w.t_end > w.t_begin ? (w.t_end - w.t_begin + kT - 1) / kT : 0;
    return w;
}

// Quarter q of a chunk (atoms 2q, 2q+1: latent columns 128q .. 128q+127 of every
// token): 2048 copies of 16 bytes. The gather threads' count is a multiple of 16, so
// thread g keeps one (atom, 16-byte chunk) pair, g & 15, and steps over the tokens
// g / 16, + kGatherThreads / 16, ...; a warp's 32 copies are two tokens' 256
// contiguous bytes.
static_assert(kCopyThreads % 16 == 0, "gather threads");
__device__ __forceinline__ void gather_quarter(uint32_t lat, const int* rows, const uint16_t* ckv,
                                               int q, int g) {
    const int c = g & 7, at = 2 * q + ((g >> 3) & 1);
    const uint32_t dst0 = lat + at * kLatAtom;
    const uint16_t* src0 = ckv + at * 64 + c * 8;
    constexpr int kStep = kCopyThreads / 16;
    const int j0 = g >> 4;
#pragma unroll
    for (int m = 0; m < (kT + kStep - 1) / kStep; ++m) {
        const int j = j0 + kStep * m;
        if (j < kT)
            cp_async16(dst0 + j * 128 + ((c ^ (j & 7)) << 4), src0 + (long long)rows[j] * kKVL, 16);
    }
}

// FP8 cache: quarter q of a chunk decoded into the swizzled bf16 atoms by the six
// gather warps. Unit u = (token u >> 3, 16-column group u & 7 of the quarter's 128
// columns); gather thread g takes units g, g + kGatherThreads, ...: its 16 E4M3 codes
// and the token's scale for this quarter (one 128-channel group) are loaded into
// registers first (f8_load), and once the quarter is free decoded (exact: an E4M3
// value times 2^k fits bf16) and stored as two 16-byte chunks of the atom (f8_store).
constexpr int kF8Units = (kT * 8 + kGatherThreads - 1) / kGatherThreads;
struct F8Quarter {
    uint4 c[kF8Units];
    float sc[kF8Units];
};
__device__ __forceinline__ void f8_load(F8Quarter& L, const int* rows, const uint8_t* ckv8,
                                        const float* scl, int q, int g) {
#pragma unroll
    for (int m = 0; m < kF8Units; ++m) {
        const int u = g + m * kGatherThreads;
        if (u < kT * 8) {
            const long long r = rows[u >> 3];
            L.c[m] = __ldg(reinterpret_cast<const uint4*>(ckv8 + r * kKVL + q * 128 + (u & 7) * 16));
            L.sc[m] = __ldg(scl + r * (kKVL / 128) + q);
        }
    }
}
__device__ __forceinline__ void f8_store(const F8Quarter& L, uint32_t lat, int q, int g) {
#pragma unroll
    for (int m = 0; m < kF8Units; ++m) {
        const int u = g + m * kGatherThreads;
        if (u < kT * 8) {
            const int j = u >> 3, grp = u & 7;
            const int c0 = 2 * (grp & 3);
            const uint32_t row = lat + (2 * q + (grp >> 2)) * kLatAtom + j * 128;
            const float sc = L.sc[m];
            const uint4 c = L.c[m];
            const uint4 lo = make_uint4(e4m3x2_to_bf16x2(c.x, sc), e4m3x2_to_bf16x2(c.x >> 16, sc),
                                        e4m3x2_to_bf16x2(c.y, sc), e4m3x2_to_bf16x2(c.y >> 16, sc));
            const uint4 hi = make_uint4(e4m3x2_to_bf16x2(c.z, sc), e4m3x2_to_bf16x2(c.z >> 16, sc),
                                        e4m3x2_to_bf16x2(c.w, sc), e4m3x2_to_bf16x2(c.w >> 16, sc));
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"r"(row + ((c0 ^ (j & 7)) << 4)),
                         "r"(lo.x), "r"(lo.y), "r"(lo.z), "r"(lo.w)
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"r"(row + (((c0 + 1) ^ (j & 7)) << 4)),
                         "r"(hi.x), "r"(hi.y), "r"(hi.z), "r"(hi.w)
                         : "memory");
        }
    }
}

template <bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    mla_tc_kernel(const __grid_constant__ CUtensorMap tmQ, MlaTcParams a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sQ = smem + kOffQ;
    uint8_t* sLat = smem + kOffLat;
    uint8_t* sP = smem + kOffP;
    float* red = reinterpret_cast<float*>(smem + kOffRed);
    float* sums = reinterpret_cast<float*>(smem + kOffSums);
    uint32_t* wflag = reinterpret_cast<uint32_t*>(smem + kOffFlag);
    float* msm = reinterpret_cast<float*>(smem + kOffM);
    int* rows = reinterpret_cast<int*>(smem + kOffRows);
    uint8_t* mask = smem + kOffMask;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int units = a.rows * a.ns;
    constexpr bool f8 = F8;  // the FP8 cache: only the gather warps decode it

    if (threadIdx.x == 0) {
        mbar_init(bars + Q_FULL, 1);
        mbar_init(bars + Q_EMPTY, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bars + ROWS_FULL + b, 1);
            mbar_init(bars + ROWS_EMPTY + b, kGatherWarps + kSoftWarps);
            mbar_init(bars + RED + b, kSoftWarps);
        }
        for (int q = 0; q < kQuarters; ++q) {
            mbar_init(bars + LAT_FULL + q, f8 ? kGatherThreads : kCopyThreads);
            mbar_init(bars + LAT_EMPTY + q, 1);
        }
        mbar_init(bars + S_FULL, 1);
        mbar_init(bars + P_FULL, kSoftWarps);
        mbar_init(bars + O_DONE, 1);
        mbar_init(bars + O_FREE, kSoftWarps);
        mbar_init(bars + SUM_IN, kSoftWarps);
        mbar_init(bars + SUM_OUT, kSoftWarps);
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

    // one lane waits, the warp follows its verdict
    auto bwait = [&](int bar, uint32_t parity) -> bool {
        int got = 1;
        if (lane == 0) got = wait_or_abort(bars + bar, parity, abort_flag, a.status);
        return __shfl_sync(0xffffffffu, got, 0) != 0;
    };

    // Register split by warpgroup: the softmax warpgroups (warps 4-11) raise their
    // registers, the other two lower theirs; each instruction is executed by whole
    // warpgroups.
    if (warp >= 4 && warp < 12) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kRegHigh));
        // ---- softmax and epilogue: thread j owns token j of a chunk (tensor lane j)
        // and one half of the heads (h0 .. h0 + 31); two warps share each lane quarter ----
        const int qd = warp & 3;
        const int h0 = 32 * ((warp - 4) >> 2);
        const int j = 32 * qd + lane;
        const uint32_t lrow = (uint32_t)(32 * qd) << 16;
        const float NEG_INF = __int_as_float(0xff800000);
        int n = 0, k = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const Unit w = unit_of(a, u);
            const long long pbase = ((long long)w.r * a.ns + w.split) * kH;
            if (w.nch == 0) {
                // no tokens: zero output, (m, l) = (-inf, 0)
                if (a.ns > 1 && qd == 0)
                    *reinterpret_cast<float2*>(a.part_ml + (pbase + h0 + lane) * 2) =
                        make_float2(NEG_INF, 0.f);
                for (int h = h0; h < h0 + 32; ++h)
                    for (int i = 0; i < kQuarters; ++i) {
                        const int cidx = 128 * i + j;
                        if (a.ns > 1) {
                            a.part_o[(pbase + h) * kKVL + cidx] = 0.f;
                        } else {
                            const long long oi = ((long long)w.r * kH + h) * kKVL + cidx;
                            if (a.olat) a.olat[oi] = 0.f;
                            if (a.xbf) a.xbf[oi] = 0;
                        }
                    }
                continue;
            }
            // Running maxima (identical in every thread) live in msm[n & 1] during
            // chunk n; the chunk's new ones go to msm[(n + 1) & 1].
            float lacc[32];
#pragma unroll
            for (int h = 0; h < 32; ++h) lacc[h] = 0.f;
            for (int c = 0; c < w.nch; ++c, ++n) {
                const int b = n & 1;
                if (!bwait(ROWS_FULL + b, (uint32_t)((n >> 1) & 1))) {
                    ok = false;
                    break;
                }
                const bool valid = mask[b * kT + j] != 0;
                // this warp's share of the chunk's gather, quarter by quarter as the
                // previous chunk's PV frees them (the bf16 cache only)
                for (int q = 0; q < kQuarters && ok && !f8; ++q) {
                    if (!bwait(LAT_EMPTY + q, (uint32_t)(n & 1) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    gather_quarter(smem_u32(sLat), rows + b * kT, a.ckv, q,
                                   kGatherThreads + (warp - 4) * 32 + lane);
                    cp_async_arrive_noinc(bars + LAT_FULL + q);
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(bars + ROWS_EMPTY + b);
                if (!bwait(S_FULL, (uint32_t)(n & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sv[32];  // this token's scores for heads h0 .. h0 + 31
                tc_ld32(sv, tmem + lrow + h0);
                tc_wait_ld(sv);
                const float* mold = msm + b * kH + h0;  // running maxima (read when c > 0)
                // Does any score of this warp move a running maximum (lag above kLazy,
                // or none yet)? Only such warps publish their chunk maxima: a warp with
                // no such score cannot change the new maximum of any head.
                bool mine = c == 0;
                if (!mine && valid) {
#pragma unroll
                    for (int h = 0; h < 32; ++h) {
                        const float mo = mold[h];
                        mine = mine || mo == NEG_INF || __uint_as_float(sv[h]) * a.sl2 > mo + kLazy;
                    }
                }
                const bool pub = __any_sync(0xffffffffu, mine);
                float* rb = red + b * 4 * kH;
                const int sw = warp - 4;  // softmax warp 0..7: lane quarter sw & 3, half sw >> 2
                if (pub) {
                    float4* dst = reinterpret_cast<float4*>(rb + qd * kH + h0);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float4 m4;
                        m4.x = warp_max(valid ? __uint_as_float(sv[4 * i]) * a.sl2 : NEG_INF);
                        m4.y = warp_max(valid ? __uint_as_float(sv[4 * i + 1]) * a.sl2 : NEG_INF);
                        m4.z = warp_max(valid ? __uint_as_float(sv[4 * i + 2]) * a.sl2 : NEG_INF);
                        m4.w = warp_max(valid ? __uint_as_float(sv[4 * i + 3]) * a.sl2 : NEG_INF);
                        if (lane == 0) dst[i] = m4;
                    }
                }
                if (lane == 0) wflag[b * 8 + sw] = pub ? 1u : 0u;
                __syncwarp();
                if (lane == 0) mbar_arrive(bars + RED + b);
                if (!bwait(RED + b, (uint32_t)((n >> 1) & 1))) {
                    ok = false;
                    break;
                }
                // new running maxima of this half (lagging by at most kLazy) into cm,
                // from the lane quarters that published
                const int hw = (sw >> 2) * 4;
                const bool any = (wflag[b * 8 + hw] | wflag[b * 8 + hw + 1] | wflag[b * 8 + hw + 2] |
                                  wflag[b * 8 + hw + 3]) != 0u;
                float cm[32];
                bool resc = false;
                if (!any) {
#pragma unroll
                    for (int h = 0; h < 32; ++h) cm[h] = mold[h];  // c > 0 here
                } else {
#pragma unroll
                    for (int h = 0; h < 32; ++h) cm[h] = NEG_INF;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (wflag[b * 8 + hw + q] == 0u) continue;
                        const float4* r4 = reinterpret_cast<const float4*>(rb + q * kH + h0);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float4 w4 = r4[i];
                            cm[4 * i] = fmaxf(cm[4 * i], w4.x);
                            cm[4 * i + 1] = fmaxf(cm[4 * i + 1], w4.y);
                            cm[4 * i + 2] = fmaxf(cm[4 * i + 2], w4.z);
                            cm[4 * i + 3] = fmaxf(cm[4 * i + 3], w4.w);
                        }
                    }
#pragma unroll
                    for (int h = 0; h < 32; ++h) {
                        const float mo = c > 0 ? mold[h] : NEG_INF;
                        const bool up = mo != NEG_INF && cm[h] > mo + kLazy;
                        resc = resc || up;
                        cm[h] = (mo == NEG_INF || up) ? cm[h] : mo;
                    }
                }
                if (resc) {
                    // O^T through the previous chunk is complete: S_FULL of this chunk
                    // was committed after that chunk's PV.
#pragma unroll 1
                    for (int i = 0; i < kQuarters; ++i) {
                        uint32_t v[32];
                        const uint32_t addr = tmem + lrow + 64 + 64 * i + h0;
                        tc_ld32(v, addr);
                        tc_wait_ld(v);
#pragma unroll
                        for (int kk = 0; kk < 32; ++kk) {
                            const float f = mold[kk] == NEG_INF ? 1.f : exp2f(mold[kk] - cm[kk]);
                            v[kk] = __float_as_uint(__uint_as_float(v[kk]) * f);
                        }
                        tc_st32(addr, v);
                    }
                    tc_wait_st();
                }
                if (any && c > 0) {
#pragma unroll
                    for (int h = 0; h < 32; ++h)
                        if (mold[h] != NEG_INF && cm[h] != mold[h]) lacc[h] *= exp2f(mold[h] - cm[h]);
                }
                if (lane == 0) {  // both warps of a half write the same values
                    float4* mn4 = reinterpret_cast<float4*>(msm + (b ^ 1) * kH + h0);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        mn4[i] = make_float4(cm[4 * i], cm[4 * i + 1], cm[4 * i + 2], cm[4 * i + 3]);
                }
                // probabilities into row j of P^T (bf16)
                {
                    uint4* prow = reinterpret_cast<uint4*>(sP + j * 128);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {  // heads h0 + 8q .. +7 -> one 16-byte chunk
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int h = 8 * q + 2 * e;
                            const float x0 = __uint_as_float(sv[h]) * a.sl2;
                            const float x1 = __uint_as_float(sv[h + 1]) * a.sl2;
                            const float p0 = (valid && cm[h] != NEG_INF) ? ex2_sfu(x0 - cm[h]) : 0.f;
                            const float p1 =
                                (valid && cm[h + 1] != NEG_INF) ? ex2_sfu(x1 - cm[h + 1]) : 0.f;
                            lacc[h] += p0;
                            lacc[h + 1] += p1;
                            pk[e] = pack_bf16x2(p0, p1);
                        }
                        prow[((h0 >> 3) + q) ^ (j & 7)] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars + P_FULL);
            }
            if (!ok) break;

            // ---- epilogue of the unit ----
            if (!bwait(O_DONE, (uint32_t)(k & 1))) {
                ok = false;
                break;
            }
            tc_fence_after();
            // head sums: reduce-scatter over the warp (lane l ends with head h0 + l),
            // then over the four lane quarters through shared memory
            float v32[32];
#pragma unroll
            for (int h = 0; h < 32; ++h) v32[h] = lacc[h];
#pragma unroll
            for (int ww = 16, m = 16; m >= 1; ww >>= 1, m >>= 1) {
#pragma unroll
                for (int i = 0; i < ww; ++i) {
                    const bool hi = (lane & m) != 0;
                    const float send = hi ? v32[i] : v32[ww + i];
                    const float recv = __shfl_xor_sync(0xffffffffu, send, m);
                    v32[i] = (hi ? v32[ww + i] : v32[i]) + recv;
                }
            }
            // the sums buffer is free once every warp has read the last unit's sums
            if (k > 0 && !bwait(SUM_OUT, (uint32_t)((k - 1) & 1))) {
                ok = false;
                break;
            }
            sums[qd * kH + h0 + lane] = v32[0];
            __syncwarp();
            if (lane == 0) mbar_arrive(bars + SUM_IN);
            if (!bwait(SUM_IN, (uint32_t)(k & 1))) {
                ok = false;
                break;
            }
            if (a.ns > 1 && qd == 0) {  // lane l writes head h0 + l's (m, l)
                const int hd = h0 + lane;
                const float mj = msm[(n & 1) * kH + hd];  // the last chunk's new maxima
                const float ls = (sums[hd] + sums[kH + hd]) + (sums[2 * kH + hd] + sums[3 * kH + hd]);
                *reinterpret_cast<float2*>(a.part_ml + (pbase + hd) * 2) = make_float2(mj, ls);
            }
#pragma unroll 1
            for (int i = 0; i < kQuarters; ++i) {
                const int cidx = 128 * i + j;  // latent column = tensor lane of tile i
                uint32_t v[32];
                tc_ld32(v, tmem + lrow + 64 + 64 * i + h0);
                tc_wait_ld(v);
#pragma unroll
                for (int kk = 0; kk < 32; ++kk) {
                    const int h = h0 + kk;
                    const float o = __uint_as_float(v[kk]);
                    if (a.ns > 1) {
                        a.part_o[(pbase + h) * kKVL + cidx] = o;
                    } else {
                        const float ls =
                            (sums[h] + sums[kH + h]) + (sums[2 * kH + h] + sums[3 * kH + h]);
                        const float val = ls > 0.f ? o / ls : 0.f;
                        const long long oi = ((long long)w.r * kH + h) * kKVL + cidx;
                        if (a.olat) a.olat[oi] = val;
                        if (a.xbf) a.xbf[oi] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
                    }
                }
            }
            // O^T is read: the next unit's first PV may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bars + O_FREE);
                mbar_arrive(bars + SUM_OUT);
            }
            ++k;
        }
        cp_async_wait_all();  // drain this warp's copies
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegLow));
        if (warp == 0) {
        // ---- token rows (two chunks ahead) and each unit's Q ----
        int n = 0, k = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const Unit w = unit_of(a, u);
            if (w.nch == 0) continue;
            int seq = a.row_seq ? __ldg(a.row_seq + w.r) : w.r;
            int L = 0;
            if (seq >= 0 && seq < a.pg.batch) {
                L = min(__ldg(a.pg.seq_lens + seq), seq_capacity(a.pg));
            } else {
                if (lane == 0 && w.split == 0) flag_status(a.status, DSA_STATUS_BAD_TOKEN);
                seq = 0;
            }
            for (int c = 0; c < w.nch; ++c, ++n) {
                const int b = n & 1;
                if (!bwait(ROWS_EMPTY + b, (uint32_t)((n >> 1) & 1) ^ 1u)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const int j = 4 * lane + kk;
                    const int pos = w.t_begin + c * kT + j;
                    long long prow = -1;
                    if (pos < w.t_end) {
                        const int t = __ldg(a.token_ids + (long long)w.r * a.ow + pos);
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
                    mask[b * kT + j] = prow >= 0 ? 1 : 0;
                    rows[b * kT + j] = prow >= 0 ? (int)prow : 0;  // a real row; masked later
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bars + ROWS_FULL + b);
                if (c == 0) {
                    // Q of this unit, once the last unit's QK is done with the buffer
                    int got = 1;
                    if (lane == 0) {
                        got = k == 0 || wait_or_abort(bars + Q_EMPTY, (uint32_t)((k - 1) & 1),
                                                      abort_flag, a.status);
                        if (got) {
                            mbar_arrive_expect_tx(bars + Q_FULL, kAtoms * kQAtom);
                            for (int at = 0; at < kAtoms; ++at)
                                tma_load_2d(smem_u32(sQ + at * kQAtom), &tmQ, 64 * at, w.r * kH,
                                            bars + Q_FULL);
                        }
                    }
                    if (!__shfl_sync(0xffffffffu, got, 0)) {
                        ok = false;
                        ++n;
                        break;
                    }
                    ++k;
                }
            }
        }
        // drain: the last Q copy issued has landed before the CTA may exit
        if (lane == 0 && k > 0) mbar_wait(bars + Q_FULL, (uint32_t)((k - 1) & 1));
        } else if (warp == 1) {
        // ---- MMA issuer ----
        if (lane == 0) {
            constexpr uint32_t IDESC_QK = idesc_bf16(kT, kH);
            constexpr uint32_t IDESC_PV = idesc_bf16(128, kH) | (1u << 15) | (1u << 16);
            const uint32_t q0 = smem_u32(sQ), l0 = smem_u32(sLat), p0 = smem_u32(sP);
            int n = 0, k = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                const Unit w = unit_of(a, u);
                if (w.nch == 0) continue;
                if (!wait_or_abort(bars + Q_FULL, (uint32_t)(k & 1), abort_flag, a.status)) break;
                for (int c = 0; c < w.nch; ++c, ++n) {
                    // S^T = K Q^T, quarter by quarter as the gather lands
                    for (int q = 0; q < kQuarters && ok; ++q) {
                        if (!wait_or_abort(bars + LAT_FULL + q, (uint32_t)(n & 1), abort_flag,
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
                                tc_mma(tmem, sw128_desc(l0 + at * kLatAtom + 32 * kk),
                                       sw128_desc(q0 + at * kQAtom + 32 * kk), IDESC_QK,
                                       (at | kk) != 0 ? 1u : 0u);
                        }
                    }
                    if (!ok) break;
                    if (c == w.nch - 1) tc_commit(bars + Q_EMPTY);
                    tc_commit(bars + S_FULL);
                    if (!wait_or_abort(bars + P_FULL, (uint32_t)(n & 1), abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    if (c == 0 && k > 0 &&
                        !wait_or_abort(bars + O_FREE, (uint32_t)((k - 1) & 1), abort_flag,
                                       a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // O^T += V^T P^T, tile by tile; each frees its quarter
                    for (int i = 0; i < kQuarters; ++i) {
#pragma unroll
                        for (int kk = 0; kk < kT / 16; ++kk)
                            tc_mma(tmem + 64 + 64 * i,
                                   sw128_desc_mn(l0 + 2 * i * kLatAtom + kk * 2048, kLatAtom, 1024),
                                   sw128_desc_mn(p0 + kk * 2048, kQAtom, 1024), IDESC_PV,
                                   (c > 0 || kk > 0) ? 1u : 0u);
                        tc_commit(bars + LAT_EMPTY + i);
                    }
                    if (c == w.nch - 1) tc_commit(bars + O_DONE);
                }
                ++k;
            }
            // Drain: every MMA issued has completed before tensor memory is released.
            tc_commit(bars + DRAIN);
            mbar_wait(bars + DRAIN, 0);
        }
        } else {
        // ---- gather: quarters of each chunk as the previous chunk's PV frees them ----
        const int g = (warp < 4 ? warp - 2 : warp - 10) * 32 + lane;
        const uint32_t lat = smem_u32(sLat);
        int n = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const Unit w = unit_of(a, u);
            for (int c = 0; c < w.nch; ++c, ++n) {
                const int b = n & 1;
                if (!bwait(ROWS_FULL + b, (uint32_t)((n >> 1) & 1))) {
                    ok = false;
                    break;
                }
                if constexpr (F8) {
                    // quarter q + 1's codes are requested while quarter q is decoded
                    F8Quarter L;
                    f8_load(L, rows + b * kT, a.ckv8, a.ckv_scale, 0, g);
                    for (int q = 0; q < kQuarters && ok; ++q) {
                        if (!bwait(LAT_EMPTY + q, (uint32_t)(n & 1) ^ 1u)) {
                            ok = false;
                            break;
                        }
                        f8_store(L, lat, q, g);
                        fence_async_smem();  // the tile's bytes are visible to the MMAs
                        mbar_arrive(bars + LAT_FULL + q);
                        if (q + 1 < kQuarters) f8_load(L, rows + b * kT, a.ckv8, a.ckv_scale, q + 1, g);
                    }
                }
                for (int q = 0; q < kQuarters && ok && !f8; ++q) {
                    if (!bwait(LAT_EMPTY + q, (uint32_t)(n & 1) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    gather_quarter(lat, rows + b * kT, a.ckv, q, g);
                    cp_async_arrive_noinc(bars + LAT_FULL + q);
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(bars + ROWS_EMPTY + b);
            }
        }
        cp_async_wait_all();  // drain
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

// The tensor-core kernel serves 64 heads of a 512-wide latent. It is chosen for
// batches with at least 4 of its 128-token chunks per SM (see make_plan): 64 paged
// rows of 2,048 tokens (two splits per row) and prefill chunks of thousands of rows
// run faster on it than on the mma.sync kernel; with one chunk per CTA (decode
// batches of a few rows) the mma.sync kernel is faster.
bool mla_tc_supported(int heads, int kv_lora_rank) { return heads == kH && kv_lora_rank == kKVL; }

int mla_tc_chunk() { return kT; }

int mla_tc_launch(const MlaTcParams& a, long long ckv_rows, cudaStream_t st) {
    if (ckv_rows < 1 || ckv_rows > 0x7fffffffLL)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_sparse_mla_decode: latent cache rows %lld",
                    ckv_rows);
    if ((long long)a.rows * kH > 0x7fffffffLL || (long long)a.rows * a.ns > 0x7fffffffLL)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_sparse_mla_decode: too many rows");
    const int sms = sm_count();
    if (sms <= 0) return fail(DSA_ERR_CUDA, "dsa_sparse_mla_decode: no CUDA device");
    const long long units = (long long)a.rows * a.ns;
    if (units == 0) return DSA_OK;
    const int grid = (int)(units < sms ? units : sms);
    CUtensorMap tmQ;
    int rc = make_tmap_2d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.qlat, kKVL,
                          (uint64_t)a.rows * kH, kKVL * 2, 64, kH, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    auto kernel = a.ckv8 ? mla_tc_kernel<true> : mla_tc_kernel<false>;
    rc = set_max_smem((const void*)kernel, (int)kDyn);
    if (rc) return rc;
    cudaError_t e = launch_pdl(kernel, dim3((unsigned)grid), dim3(kThreads), kDyn, st, tmQ, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_mla_decode tensor-core launch");
    return DSA_OK;
}

}  // namespace dsa
