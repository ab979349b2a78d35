// dsa_score_prefill: index scores of many query rows of one sequence (chunked
// prefill) as a dense contraction on the tensor cores.
//
// Page: metrale_model_arch/glm5next_dsa/tp.rs, "Why the indexer is replicated"
// (score[q, p] = sum_h w[q,h] * relu(scale * <qidx[q,h,:], kpool[p,:]>)); the dense
// [Q * index_heads, ihd] x [ihd, P] form is the chunked-prefill case of the same
// equation, with the candidate rule of dsa_score (pool flag set, last slot before the
// row's context length).
//
// Tile: D[p, (q,h)] = sign(scale) * <kpool[p,:], qidx[q,h,:]> for 128 pools (the
// MMA's M, one tensor-memory lane each) by 256 (query, head) columns (N), K = ihd,
// bf16 operands (the sign applied by the MMA's negate-A bit), f32 accumulation in
// tensor memory. A pool's row of D holds every head of the tile's queries, so the
// head sum stays in one thread:
//   score[q, p] = sum_h (w[q,h] * |scale|) * relu(D[p, (q,h)]).
//
// Roles (one CTA per SM, persistent over work units of one query tile x 32 pool
// tiles):
//   warp 0      TMA producer: the unit's query tile once, pool tiles through a ring
//               of shared-memory stages (128-byte swizzled K-major boxes);
//   warp 1      owns the 512 tensor-memory columns (two 256-column accumulators) and
//               issues tcgen05.mma from one thread;
//   warps 2..   epilogue (16 warps, or 8 at 128 heads): tcgen05.ld of their lane
//               quarter and column slice, the relu-weighted head sum (packed f32x2
//               FMAs), masking, and the f32 score stores.
// Every wait is bounded: a wait that runs out sets DSA_STATUS_TIMEOUT and a CTA-wide
// abort flag, every role then leaves its loop, copies and MMAs in flight are drained,
// and tensor memory is released.
#include <algorithm>

#include "common.cuh"
#include "tc.cuh"

namespace dsa {
namespace {

constexpr int kTileP = 128;        // pools per tile
constexpr int kTileN = 256;        // (query, head) columns per tile
constexpr int kTilesPerUnit = 32;  // pool tiles per work unit
constexpr int kWTab = 1024;        // floats of per-warp weight tables, all warps together

// Epilogue warps: four per tensor-memory lane quarter (64 columns each) when a
// query's heads fit in 64 columns, else two (128 columns each).
__host__ __device__ constexpr int epi_warps(int heads) { return heads <= 64 ? 16 : 8; }
__host__ __device__ constexpr int block_threads(int heads) { return 64 + 32 * epi_warps(heads); }
constexpr uint32_t kTmemCols = 2 * kTileN;

struct PrefillArgs {
    const float* w;
    const int32_t* row_ctx;
    const int32_t* seq_lens;
    const uint8_t* pv;  // this sequence's pool flags
    float* scores;
    int32_t* status;
    int rows;
    int p_stride;
    int first_key;
    int kpool;
    int seq;
    int cap;   // token capacity of a sequence
    int pcap;  // pool capacity of a sequence
    long long prow0;  // this sequence's first pool row in the pooled-key tensor
    int qtiles, ptiles, pchunks;
    float wscale;  // |scale|
    int neg;       // scale < 0
};

// Per chunk c of NCH 32-column chunks: sum_i w[c][i] * relu(x[c][i]), the weights
// read from shared memory at byte address waddr + 128 c. The chunks are interleaved,
// four packed f32x2 FMA chains each, so that their work overlaps.
template <int NCH>
__device__ __forceinline__ void chunk_sums(const uint32_t (&x)[NCH][32], uint32_t waddr,
                                           float (&out)[NCH]) {
    float2 s[NCH][4];
#pragma unroll
    for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int k = 0; k < 4; ++k) s[c][k] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const float4 wa = lds_f4(waddr + 128u * c + 16u * i);
            const float4 wb = lds_f4(waddr + 128u * c + 16u * (i + 1));
            float r[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) r[j] = fmaxf(__uint_as_float(x[c][4 * i + j]), 0.f);
            s[c][0] = __ffma2_rn(make_float2(r[0], r[1]), make_float2(wa.x, wa.y), s[c][0]);
            s[c][1] = __ffma2_rn(make_float2(r[2], r[3]), make_float2(wa.z, wa.w), s[c][1]);
            s[c][2] = __ffma2_rn(make_float2(r[4], r[5]), make_float2(wb.x, wb.y), s[c][2]);
            s[c][3] = __ffma2_rn(make_float2(r[6], r[7]), make_float2(wb.z, wb.w), s[c][3]);
        }
    }
#pragma unroll
    for (int c = 0; c < NCH; ++c)
        out[c] = ((s[c][0].x + s[c][0].y) + (s[c][1].x + s[c][1].y)) +
                 ((s[c][2].x + s[c][2].y) + (s[c][3].x + s[c][3].y));
}

template <int KA>
struct Layout {
    static constexpr int kStages = KA == 2 ? 4 : 8;
    static constexpr uint32_t kRowBytes = 128;                      // one swizzle row
    static constexpr uint32_t kABox = kTileP * kRowBytes;           // one K atom of a pool tile
    static constexpr uint32_t kBBox = kTileN * kRowBytes;           // one K atom of a query tile
    static constexpr uint32_t kABytes = KA * kABox;                 // a stage
    static constexpr uint32_t kBBytes = KA * kBBox;
    static constexpr uint32_t kOffA = kBBytes;
    static constexpr uint32_t kOffW = kOffA + kStages * kABytes;    // per-warp weights, f32
    static constexpr uint32_t kOffN = kOffW + kWTab * 4;            // [warp][8] i32
    static constexpr uint32_t kOffBar = kOffN + 16 * 8 * 4;
    static constexpr int kBars = 2 * kStages + 2 + 4 + 1;
    static constexpr uint32_t kOffMisc = kOffBar + kBars * 8;
    static constexpr uint32_t kBytes = kOffMisc + 16;
    static constexpr uint32_t kDynBytes = kBytes + 1024;  // room to align the base to 1024
};

template <int KA, int HI>
__global__ void __launch_bounds__(block_threads(HI), 1)
    prefill_score_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB, PrefillArgs a) {
    using L = Layout<KA>;
    constexpr int S = L::kStages;
    constexpr int EPW = epi_warps(HI);
    constexpr int SLICES = EPW / 4;     // column slices per lane quarter
    constexpr int CW = kTileN / SLICES; // columns per epilogue warp
    constexpr int NCH = CW / 32;        // 32-column chunks per epilogue warp
    constexpr int QPT = kTileN / HI;    // queries per tile
    constexpr int QPW = CW / HI;        // queries per epilogue warp
    constexpr int KSTEPS = KA * 4;      // MMAs of K = 16 per tile
    // A negative scale negates the pooled keys inside the MMA (exact for bf16), so
    // D = sign(scale) * <kpool, qidx> and the epilogue applies relu and |scale| only.
    const uint32_t IDESC = idesc_bf16(kTileP, kTileN) | (a.neg ? (1u << 13) : 0u);
    static_assert(HI % 32 == 0 && QPT >= 2 && QPW >= 1 && EPW * CW == kWTab,
                  "index heads must be 32, 64 or 128");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sB = smem;
    uint8_t* sA = smem + L::kOffA;
    float* wtab_all = reinterpret_cast<float*>(smem + L::kOffW);
    int* ntab_all = reinterpret_cast<int*>(smem + L::kOffN);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
    uint64_t* full = bars;
    uint64_t* empty = bars + S;
    uint64_t* bfull = bars + 2 * S;
    uint64_t* bempty = bfull + 1;
    uint64_t* accfull = bempty + 1;   // [2]
    uint64_t* accempty = accfull + 2; // [2]
    uint64_t* drain = accempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(bfull, 1);
        mbar_init(bempty, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(accfull + b, 1);
            mbar_init(accempty + b, EPW);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                smem_u32(tmem_slot)),
            "r"(kTmemCols)
            : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const long long units = (long long)a.qtiles * a.pchunks;

    if (warp == 0) {
        // ---- TMA producer ----
        // Per unit: the first pool tiles (as many as there are stages), then the query
        // tile once the previous unit's MMAs have released it, then the rest; so the
        // reload of the query tile overlaps pool tiles already in flight.
        if (lane == 0) {
            int stage = 0;
            uint32_t sphase = 0;
            bool armed[S];
            uint32_t apar[S];
            for (int s = 0; s < S; ++s) armed[s] = false, apar[s] = 0;
            bool barmed = false;
            uint32_t bpar = 0;
            int uc = 0;
            bool ok = true;
            for (long long u = blockIdx.x; u < units && ok; u += gridDim.x, ++uc) {
                const int qt = (int)(u / a.pchunks), pc = (int)(u % a.pchunks);
                const int t0 = pc * kTilesPerUnit, t1 = min(a.ptiles, t0 + kTilesPerUnit);
                const int tb = min(t1, t0 + S);  // the query tile is loaded before tile tb
                for (int t = t0; t <= t1 && ok; ++t) {
                    if (t == tb) {
                        if (!wait_or_abort(bempty, (uint32_t)(uc & 1) ^ 1u, abort_flag,
                                           a.status)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(bfull, L::kBBytes);
                        for (int ka = 0; ka < KA; ++ka)
                            tma_load_2d(smem_u32(sB + ka * L::kBBox), &tmB, ka * 64,
                                        qt * kTileN, bfull);
                        barmed = true;
                        bpar = (uint32_t)(uc & 1);
                    }
                    if (t == t1) break;
                    if (!wait_or_abort(empty + stage, sphase ^ 1u, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full + stage, L::kABytes);
                    const int y = (int)(a.prow0 + (long long)t * kTileP);
                    for (int ka = 0; ka < KA; ++ka)
                        tma_load_2d(smem_u32(sA + stage * L::kABytes + ka * L::kABox), &tmA,
                                    ka * 64, y, full + stage);
                    armed[stage] = true;
                    apar[stage] = sphase;
                    if (++stage == S) stage = 0, sphase ^= 1u;
                }
            }
            // Drain: every copy this thread issued has landed before the CTA ends.
            for (int s = 0; s < S; ++s)
                if (armed[s]) mbar_wait(full + s, apar[s]);
            if (barmed) mbar_wait(bfull, bpar);
        }
    } else if (warp == 1) {
        // ---- MMA issuer ----
        if (lane == 0) {
            int stage = 0;
            uint32_t sphase = 0;
            int tc = 0, uc = 0;
            bool ok = true;
            for (long long u = blockIdx.x; u < units && ok; u += gridDim.x, ++uc) {
                const int pc = (int)(u % a.pchunks);
                const int t0 = pc * kTilesPerUnit, t1 = min(a.ptiles, t0 + kTilesPerUnit);
                if (!wait_or_abort(bfull, (uint32_t)(uc & 1), abort_flag, a.status)) break;
                tc_fence_after();
                for (int t = t0; t < t1; ++t, ++tc) {
                    const int buf = tc & 1;
                    if (!wait_or_abort(accempty + buf, (uint32_t)((tc >> 1) & 1) ^ 1u, abort_flag,
                                       a.status) ||
                        !wait_or_abort(full + stage, sphase, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)(buf * kTileN);
                    const uint32_t a0 = smem_u32(sA + stage * L::kABytes);
                    const uint32_t b0 = smem_u32(sB);
#pragma unroll
                    for (int k = 0; k < KSTEPS; ++k) {
                        const uint32_t off = (uint32_t)(k & 3) * 32u;  // K = 16 bf16 = 32 B
                        const uint64_t ad = sw128_desc(a0 + (uint32_t)(k >> 2) * L::kABox + off);
                        const uint64_t bd = sw128_desc(b0 + (uint32_t)(k >> 2) * L::kBBox + off);
                        tc_mma(d, ad, bd, IDESC, k > 0 ? 1u : 0u);
                    }
                    tc_commit(empty + stage);
                    tc_commit(accfull + buf);
                    if (++stage == S) stage = 0, sphase ^= 1u;
                }
                if (ok) tc_commit(bempty);
            }
            // Drain: every MMA issued has completed before tensor memory is released.
            tc_commit(drain);
            mbar_wait(drain, 0);
        }
    } else {
        // ---- epilogue ----
        const int e = warp - 2;
        const int quarter = warp & 3;  // tensor-memory lanes 32*quarter .. +31
        const int slice = e >> 2;      // columns CW*slice .. +CW-1
        float* wtab = wtab_all + e * CW;
        int* ntab = ntab_all + e * 8;
        const uint32_t wtab_s = smem_u32(wtab), ntab_s = smem_u32(ntab);
        const float NEG_INF = __int_as_float(0xff800000);
        const int Lseq = min(__ldg(a.seq_lens + a.seq), a.cap);
        int tc = 0;
        bool ok = true;
        for (long long u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const int qt = (int)(u / a.pchunks), pc = (int)(u % a.pchunks);
            const int t0 = pc * kTilesPerUnit, t1 = min(a.ptiles, t0 + kTilesPerUnit);
            // This warp's weights (w * |scale|) and visible-pool counts for the unit.
            const long long wbase = (long long)qt * kTileN + slice * CW;
            const long long wlim = (long long)a.rows * HI;
#pragma unroll
            for (int i = 0; i < NCH; ++i) {
                const long long idx = wbase + lane + 32 * i;
                wtab[lane + 32 * i] = idx < wlim ? __ldg(a.w + idx) * a.wscale : 0.f;
            }
            if (lane < QPW) {
                const int r = qt * QPT + slice * QPW + lane;
                int nv = 0;
                if (r < a.rows) {
                    const int ctx = a.row_ctx ? min(__ldg(a.row_ctx + r), Lseq) : Lseq;
                    nv = ctx > a.first_key ? (ctx - a.first_key) / a.kpool : 0;
                }
                ntab[lane] = nv;
            }
            __syncwarp();
            // Pool flags are fetched one tile ahead, so their latency hides behind a
            // tile of work.
            const int prow = 32 * quarter + lane;
            auto load_flag = [&](int t) -> int {
                const int p = t * kTileP + prow;
                return (t < t1 && p < a.pcap) ? (int)__ldg(a.pv + p) : 0;
            };
            int flag_next = load_flag(t0);
            for (int t = t0; t < t1; ++t, ++tc) {
                const int buf = tc & 1;
                const int p = t * kTileP + prow;
                const bool flag = flag_next != 0;
                flag_next = load_flag(t + 1);
                // One lane waits and the warp follows its verdict, so the warp-wide
                // tensor-memory loads below are always reached by all lanes together.
                int got = 1;
                if (lane == 0)
                    got = wait_or_abort(accfull + buf, (uint32_t)((tc >> 1) & 1), abort_flag,
                                        a.status);
                if (!__shfl_sync(0xffffffffu, got, 0)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tb = tmem + ((uint32_t)(32 * quarter) << 16) +
                                    (uint32_t)(buf * kTileN + slice * CW);
                uint32_t v[NCH][32];
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) tc_ld32(v[ch], tb + 32u * ch);
                tc_wait_ld(v[0]);
#pragma unroll
                for (int ch = 1; ch < NCH; ++ch) tc_tie(v[ch]);
                float cs[NCH];
                chunk_sums<NCH>(v, wtab_s, cs);
                float acc = 0.f;
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    acc += cs[ch];
                    if ((32 * (ch + 1)) % HI == 0) {  // the chunk ends a query
                        const int jl = (32 * ch) / HI;  // query within this warp's slice
                        const int r = qt * QPT + slice * QPW + jl;
                        if (r < a.rows && p < a.p_stride)
                            a.scores[(long long)r * a.p_stride + p] =
                                (flag && p < lds_s32(ntab_s + 4u * jl)) ? acc : NEG_INF;
                        acc = 0.f;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(accempty + buf);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

__global__ void fill_neg_inf_kernel(float* scores, long long n) {
    pdl_wait();
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        scores[i] = __int_as_float(0xff800000);
}

template <int KA, int HI>
int launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const PrefillArgs& a, int grid,
           cudaStream_t st) {
    constexpr uint32_t bytes = Layout<KA>::kDynBytes;
    int rc = set_max_smem((const void*)prefill_score_kernel<KA, HI>, (int)bytes);
    if (rc) return rc;
    cudaError_t e = launch_pdl(prefill_score_kernel<KA, HI>, dim3(grid), dim3(block_threads(HI)),
                               bytes, st, tmA, tmB, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "dsa_score_prefill launch");
    return DSA_OK;
}

template <int KA>
int launch_heads(int heads, const CUtensorMap& tmA, const CUtensorMap& tmB,
                 const PrefillArgs& a, int grid, cudaStream_t st) {
    switch (heads) {
        case 32: return launch<KA, 32>(tmA, tmB, a, grid, st);
        case 64: return launch<KA, 64>(tmA, tmB, a, grid, st);
        default: return launch<KA, 128>(tmA, tmB, a, grid, st);
    }
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" int dsa_score_prefill(const dsa_bf16* qidx, const float* w, int rows,
                                 int index_heads, int ihd, int seq, const int32_t* row_ctx,
                                 const dsa_bf16* kpool, const uint8_t* pool_valid,
                                 const dsa_paging* pg, int first_key, int kpool_size,
                                 float scale, float* scores, int p_stride, int32_t* status,
                                 void* stream) {
    if (rows < 0 || p_stride < 0 || first_key < 0)
        return fail(DSA_ERR_INVALID_ARG, "dsa_score_prefill: rows %d, p_stride %d, first_key %d",
                    rows, p_stride, first_key);
    if (kpool_size < 1 || kpool_size > DSA_MAX_KPOOL)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_score_prefill: kpool %d outside [1, %d]",
                    kpool_size, DSA_MAX_KPOOL);
    if (ihd != 64 && ihd != 128)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_score_prefill: index_head_dim %d not in {64, 128}",
                    ihd);
    if (index_heads != 32 && index_heads != 64 && index_heads != 128)
        return fail(DSA_ERR_UNSUPPORTED,
                    "dsa_score_prefill: index_heads %d not in {32, 64, 128}; dsa_score takes "
                    "any head count",
                    index_heads);
    Paging P;
    int rc = check_paging(pg, kpool_size, &P);
    if (rc) return rc;
    if (P.block_table)
        return fail(DSA_ERR_UNSUPPORTED,
                    "dsa_score_prefill: contiguous caches only; dsa_score takes paged caches");
    if (seq < 0 || seq >= P.batch)
        return fail(DSA_ERR_INVALID_ARG, "dsa_score_prefill: seq %d outside [0, %d)", seq,
                    P.batch);
    if (rows == 0 || p_stride == 0) return DSA_OK;
    if (!qidx || !w || !kpool || !pool_valid || !scores)
        return fail(DSA_ERR_INVALID_ARG, "dsa_score_prefill: NULL tensor");
    if ((((uintptr_t)qidx) | ((uintptr_t)kpool)) & 15)
        return fail(DSA_ERR_INVALID_ARG,
                    "dsa_score_prefill: qidx and kpool must be 16-byte aligned");
    if ((long long)rows * index_heads > 0x7fffffffLL)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_score_prefill: rows x index_heads too large");
    cudaStream_t st = (cudaStream_t)stream;
    const int pcap = P.max_seq_len / kpool_size;
    if (pcap == 0) {  // no pool fits a sequence: every score is -inf
        const long long n = (long long)rows * p_stride;
        cudaError_t e = launch_pdl(fill_neg_inf_kernel,
                                   dim3((unsigned)std::min<long long>((n + 255) / 256, 4096)),
                                   dim3(256), 0, st, scores, n);
        if (e == cudaSuccess) e = cudaGetLastError();
        return e == cudaSuccess ? DSA_OK : cuda_fail(e, "dsa_score_prefill launch");
    }
    const long long prows = (long long)P.batch * pcap;
    if (prows + kTileP * 2LL > 0x7fffffffLL)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_score_prefill: pooled-key tensor too large");

    PrefillArgs a;
    a.w = w;
    a.row_ctx = row_ctx;
    a.seq_lens = P.seq_lens;
    a.pv = pool_valid + (long long)seq * pcap;
    a.scores = scores;
    a.status = status;
    a.rows = rows;
    a.p_stride = p_stride;
    a.first_key = first_key;
    a.kpool = kpool_size;
    a.seq = seq;
    a.cap = P.max_seq_len;
    a.pcap = pcap;
    a.prow0 = (long long)seq * pcap;
    const int qpt = kTileN / index_heads;
    a.qtiles = (rows + qpt - 1) / qpt;
    a.ptiles = (p_stride + kTileP - 1) / kTileP;
    a.pchunks = (a.ptiles + kTilesPerUnit - 1) / kTilesPerUnit;
    a.wscale = fabsf(scale);
    a.neg = scale < 0.f ? 1 : 0;
    const long long units = (long long)a.qtiles * a.pchunks;
    if (a.prow0 + (long long)a.ptiles * kTileP > 0x7fffffffLL)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_score_prefill: pool coordinates exceed int32");
    if (units > 0x7fffffffLL)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_score_prefill: too many tiles");

    CUtensorMap tmA, tmB;
    rc = make_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kpool, (uint64_t)ihd,
                      (uint64_t)prows, (uint64_t)ihd * 2, 64, kTileP,
                      CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    rc = make_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, qidx, (uint64_t)ihd,
                      (uint64_t)rows * index_heads, (uint64_t)ihd * 2, 64, kTileN,
                      CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    const int sms = sm_count() > 0 ? sm_count() : 148;
    const int grid = (int)std::min<long long>(units, sms);
    return ihd == 128 ? launch_heads<2>(index_heads, tmA, tmB, a, grid, st)
                      : launch_heads<1>(index_heads, tmA, tmB, a, grid, st);
}
