// dsa_compress: indexer k_norm (LayerNorm with bias) fused with k-pool compression.
//
// Page: metrale_model_arch/glm5next_dsa/mod.rs, "Checkpoint and kernel facts the code
// depends on" (k_norm is a LayerNorm with a bias; the pool softmax runs over the slot
// axis per channel; pooling starts at first_key; a pool counts only if every slot is
// valid) and build.rs, transform 4 (ape is f32).
//
// Layout of the work: a pool of KP tokens x IHD channels is handled by IHD/8 lanes,
// each lane owning 8 consecutive channels (one 16-byte vector per token row). All
// KP rows of keys and gate logits are issued as 16-byte streaming loads before any
// arithmetic, so a warp keeps 2 * KP * 512 bytes in flight. The per-token LayerNorm
// reduces over the pool's lane group with xor shuffles (two passes: mean, then the
// centred second moment); the normalised key is rounded to bf16 in registers, the
// storage point of the unfused pipeline, and pooled with the slot softmax in f32.
// The softmax uses exp2 of log2(e)-scaled logits, the LayerNorm rsqrt and the final
// ratio a fast divide: each is within a few f32 ulp, far below the bf16 rounding of
// the stored key.
#include <algorithm>

#include "common.cuh"
#include "fp8.cuh"
#include "store.cuh"

namespace dsa {
namespace {

struct CompressArgs {
    const uint16_t* k_raw;
    const uint16_t* gate;
    const uint8_t* valid;
    const float* ape;
    const uint16_t* ln_w;
    const uint16_t* ln_b;
    uint16_t* kout;
    uint8_t* pvalid;
    int32_t* pidx;
    int32_t* status;
    Paging pg;
    float eps;
    int first_key;
    int kpool;
    int append;  // > 0: only the pools completed by the last `append` tokens
    int tiles;   // units of PPC pools per sequence
};

constexpr int kThreads = 256;

// Pools whole among the first n tokens.
__device__ __forceinline__ int whole_pools(int n, int first_key, int kpool) {
    return n > first_key ? (n - first_key) / kpool : 0;
}

// 2^x on the special-function unit (x <= 0 here: softmax weights in (0, 1]).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The pooled key of one pool for the 8 channels [c0, c0 + 8) this lane owns, from
// its kpool rows of raw keys and gate logits (kr(s), gr(s): 16-byte vectors of slot
// s): LayerNorm per slot (the pool's IHD/8 lanes reduce together, so every lane of
// the warp must call this), bf16 rounding of the normalised key, and the slot softmax
// in the log2 domain. Channels are processed in pairs with packed f32x2 arithmetic.
// Returns the packed bf16 result (to be stored only for a valid pool).
template <int IHD, int KPMAX, class KR, class GR>
__device__ __forceinline__ uint4 pool_lane(KR kr, GR gr, int KP, const float* __restrict__ ape,
                                           const uint16_t* __restrict__ ln_w,
                                           const uint16_t* __restrict__ ln_b, float eps, int c0) {
    constexpr int LPP = IHD / 8;
    constexpr float kLog2e = 1.4426950408889634f;
    auto pair = [](uint32_t u) { return make_float2(bf16_lo(u), bf16_hi(u)); };
    float2 lw[4], lb[4];
    {
        const uint4 w4 = ldg16(ln_w + c0);
        const uint4 b4 = ldg16(ln_b + c0);
        const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
        const uint32_t bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lw[i] = pair(wv[i]);
            lb[i] = pair(bv[i]);
        }
    }
    auto logits = [&](int s, float2 (&l)[4]) {  // gate + ape of slot s
        const float4 ap0 = __ldg(reinterpret_cast<const float4*>(ape + s * IHD + c0));
        const float4 ap1 = __ldg(reinterpret_cast<const float4*>(ape + s * IHD + c0 + 4));
        const float2 ap[4] = {make_float2(ap0.x, ap0.y), make_float2(ap0.z, ap0.w),
                              make_float2(ap1.x, ap1.y), make_float2(ap1.z, ap1.w)};
        const uint4 g4 = gr(s);
        const uint32_t gv[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) l[i] = __fadd2_rn(pair(gv[i]), ap[i]);
    };

    // Pass 1: the slot logits (kept in registers when kpool <= 4) and their
    // per-channel max.
    constexpr int KC = KPMAX <= 4 ? KPMAX : 1;  // cached slots
    float2 lg[KC][4];
    float2 mx[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) mx[i] = make_float2(-INFINITY, -INFINITY);
#pragma unroll
    for (int s = 0; s < KPMAX; ++s) {
        if (s < KP) {
            float2 l[4];
            logits(s, l);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (s < KC) lg[s < KC ? s : 0][i] = l[i];
                mx[i] = make_float2(fmaxf(mx[i].x, l[i].x), fmaxf(mx[i].y, l[i].y));
            }
        }
    }
    // softmax weights as 2^(l*log2e - max*log2e)
    const float2 log2e2 = make_float2(kLog2e, kLog2e);
    float2 nmxs[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __fmul2_rn(mx[i], log2e2);
        nmxs[i] = make_float2(-t.x, -t.y);
    }

    // Pass 2: LayerNorm each slot, round to bf16, accumulate the softmax-weighted sum.
    float2 num[4], den[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) num[i] = den[i] = make_float2(0.f, 0.f);
#pragma unroll
    for (int s = 0; s < KPMAX; ++s) {
        if (s < KP) {  // KP is warp-uniform: the shuffles below see the whole warp
            const uint4 k4 = kr(s);
            const uint32_t kv[4] = {k4.x, k4.y, k4.z, k4.w};
            float2 x[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i] = pair(kv[i]);
            float2 s2 = __fadd2_rn(__fadd2_rn(x[0], x[1]), __fadd2_rn(x[2], x[3]));
            float sum = s2.x + s2.y;
#pragma unroll
            for (int off = LPP / 2; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            const float nm = -sum * (1.0f / IHD);
            const float2 nm2 = make_float2(nm, nm);
            float2 q2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                x[i] = __fadd2_rn(x[i], nm2);
                q2 = __ffma2_rn(x[i], x[i], q2);
            }
            float sq = q2.x + q2.y;
#pragma unroll
            for (int off = LPP / 2; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
            const float rstd = rsqrtf(fmaf(sq, 1.0f / IHD, eps));
            const float2 r2 = make_float2(rstd, rstd);

            float2 l[4];
            if (s < KC) {
#pragma unroll
                for (int i = 0; i < 4; ++i) l[i] = lg[s < KC ? s : 0][i];
            } else {
                logits(s, l);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 kn2 = __ffma2_rn(__fmul2_rn(x[i], r2), lw[i], lb[i]);
                const uint32_t kb = pack_bf16x2(kn2.x, kn2.y);  // the bf16 storage point
                const float2 kn = pair(kb);
                const float2 a = __ffma2_rn(l[i], log2e2, nmxs[i]);
                const float2 e = make_float2(ex2(a.x), ex2(a.y));
                den[i] = __fadd2_rn(den[i], e);
                num[i] = __ffma2_rn(e, kn, num[i]);
            }
        }
    }

    uint4 o;
    o.x = pack_bf16x2(__fdividef(num[0].x, den[0].x), __fdividef(num[0].y, den[0].y));
    o.y = pack_bf16x2(__fdividef(num[1].x, den[1].x), __fdividef(num[1].y, den[1].y));
    o.z = pack_bf16x2(__fdividef(num[2].x, den[2].x), __fdividef(num[2].y, den[2].y));
    o.w = pack_bf16x2(__fdividef(num[3].x, den[3].x), __fdividef(num[3].y, den[3].y));
    return o;
}

template <int IHD, int KPMAX>
__device__ __forceinline__ void compress_unit(const CompressArgs& a, int b, int tile);

template <int IHD, int KPMAX>
__global__ void __launch_bounds__(kThreads) compress_kernel(CompressArgs a) {
    pdl_wait();
    // A persistent grid: CTA units (sequence b, PPC consecutive pools) are taken in
    // turn, so the per-CTA start-up is paid once per CTA, not once per 16 pools.
    for (long long u = blockIdx.x; u < (long long)a.tiles * a.pg.batch; u += gridDim.x)
        compress_unit<IHD, KPMAX>(a, (int)(u / a.tiles), (int)(u % a.tiles));
}

template <int IHD, int KPMAX>
__device__ __forceinline__ void compress_unit(const CompressArgs& a, int b, int tile) {
    constexpr int LPP = IHD / 8;     // lanes per pool
    constexpr int PPW = 32 / LPP;    // pools per warp
    constexpr int PPC = PPW * (kThreads / 32);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int sub = lane % LPP;
    const int c0 = sub * 8;
    const int KP = a.kpool;

    int L = __ldg(a.pg.seq_lens + b);
    L = min(L, seq_capacity(a.pg));
    const int P = whole_pools(L, a.first_key, KP);
    const int p0 = a.append > 0 ? whole_pools(max(L - a.append, 0), a.first_key, KP) : 0;
    const int p = p0 + tile * PPC + warp * PPW + lane / LPP;
    bool active = p < P;
    const int t0 = a.first_key + p * KP;
    long long trow = -1, orow = -1;
    if (active) {
        trow = token_row(a.pg, b, t0);  // all slots of a pool share one block
        orow = pool_row(a.pg, b, p, KP);
        if (trow < 0 || orow < 0) {
            if (sub == 0) flag_status(a.status, DSA_STATUS_BAD_BLOCK);
            active = false;
        }
    }

    uint4 kr[KPMAX], gr[KPMAX];
    bool ok = true;
#pragma unroll
    for (int s = 0; s < KPMAX; ++s) {
        kr[s] = make_uint4(0, 0, 0, 0);
        gr[s] = make_uint4(0, 0, 0, 0);
        if (s < KP && active) {
            const long long row = trow + s;
            kr[s] = ldg16_stream(a.k_raw + row * IHD + c0);
            gr[s] = ldg16_stream(a.gate + row * IHD + c0);
            ok = ok && (__ldg(a.valid + row) != 0);
        }
    }

    const uint4 pooled = pool_lane<IHD, KPMAX>([&](int q) { return kr[q]; },
                                               [&](int q) { return gr[q]; }, KP, a.ape, a.ln_w,
                                               a.ln_b, a.eps, c0);
    if (!active) return;
    const bool pv = ok;
    *reinterpret_cast<uint4*>(a.kout + orow * IHD + c0) = pv ? pooled : make_uint4(0, 0, 0, 0);
    if (sub == 0) {
        a.pvalid[orow] = pv ? 1 : 0;
        if (a.pidx) {
            for (int s = 0; s < KP; ++s) a.pidx[orow * KP + s] = t0 + s;
        }
    }
}

// dsa_decode_append: one CTA per sequence stores the staged token at the live
// length, advances the length, writes the row context, and (warp 0) pools the pool
// that token completed, with the same pool_lane arithmetic as compress_kernel.
struct AppendArgs {
    const uint16_t* k_new;
    const uint16_t* gate_new;
    const uint16_t* ckv_new;
    uint16_t* k_raw;
    uint16_t* gate;
    uint8_t* valid;
    uint16_t* ckv;
    uint8_t* ckv8;      // nullable: the FP8 latent cache's codes ...
    float* ckv_scale;   // ... and scales, written from ckv_new
    int32_t* seq_lens;
    int32_t* row_ctx;
    int32_t* status;
    const float* ape;
    const uint16_t* ln_w;
    const uint16_t* ln_b;
    uint16_t* kout;
    uint8_t* pvalid;
    int32_t* pidx;
    Paging pg;
    float eps;
    int first_key;
    int kpool;
    int kvl;
};

constexpr int kAppendThreads = 128;

template <int IHD, int KPMAX>
__global__ void __launch_bounds__(kAppendThreads) decode_append_kernel(AppendArgs a) {
    pdl_wait();
    constexpr int LPP = IHD / 8;
    __shared__ long long s_row;
    __shared__ int s_t;
    const int b = blockIdx.x;
    if (threadIdx.x == 0) s_row = next_token_row(a.pg, a.seq_lens, b, &s_t, a.status);
    __syncthreads();
    const long long row = s_row;
    const int t = s_t;
    if (row >= 0) {
        store_token_rows(a.k_new, a.gate_new, a.ckv_new, a.k_raw, a.gate, a.valid, a.ckv, b, row,
                         IHD, a.kvl);
        if (a.ckv8) {
            // the FP8 cache: warp w encodes 128-channel groups w, w + 4, ... of the
            // staged latent row, with the same codec as dsa_quantize_latent
            const int G = a.kvl / 128;
            for (int gi = threadIdx.x >> 5; gi < G; gi += kAppendThreads / 32)
                fp8_encode_group(a.ckv_new + (long long)b * a.kvl + gi * 128,
                                 a.ckv8 + row * a.kvl + gi * 128, a.ckv_scale + row * G + gi,
                                 threadIdx.x & 31);
        }
    }
    __syncthreads();  // the stored rows are visible to the whole block from here on
    const int L = row >= 0 ? t + 1 : t;
    if (threadIdx.x == 0) {
        if (row >= 0) a.seq_lens[b] = L;
        if (a.row_ctx) a.row_ctx[b] = L;
    }
    const int KP = a.kpool;
    const int Lc = min(L, seq_capacity(a.pg));
    const int P = whole_pools(Lc, a.first_key, KP);
    const int p = whole_pools(max(Lc - 1, 0), a.first_key, KP);  // the pool the token completed
    if (p >= P || threadIdx.x >= 32) return;  // block-uniform, then warp 0 only

    const int lane = threadIdx.x;
    const int c0 = (lane % LPP) * 8;
    bool active = lane < LPP;  // lanes past the pool's width join the shuffles with zeros
    const int t0 = a.first_key + p * KP;
    long long trow = -1, orow = -1;
    if (active) {
        trow = token_row(a.pg, b, t0);
        orow = pool_row(a.pg, b, p, KP);
        if (trow < 0 || orow < 0) {
            if (lane == 0) flag_status(a.status, DSA_STATUS_BAD_BLOCK);
            active = false;
        }
    }
    uint4 kr[KPMAX], gr[KPMAX];
    bool ok = true;
#pragma unroll
    for (int s = 0; s < KPMAX; ++s) {
        kr[s] = make_uint4(0, 0, 0, 0);
        gr[s] = make_uint4(0, 0, 0, 0);
        if (s < KP && active) {
            // Plain (coherent) loads: this block wrote the newest row.
            const long long r = trow + s;
            kr[s] = *reinterpret_cast<const uint4*>(a.k_raw + r * IHD + c0);
            gr[s] = *reinterpret_cast<const uint4*>(a.gate + r * IHD + c0);
            ok = ok && (a.valid[r] != 0);
        }
    }
    const uint4 pooled = pool_lane<IHD, KPMAX>([&](int q) { return kr[q]; },
                                               [&](int q) { return gr[q]; }, KP, a.ape, a.ln_w,
                                               a.ln_b, a.eps, c0);
    if (!active) return;
    *reinterpret_cast<uint4*>(a.kout + orow * IHD + c0) = ok ? pooled : make_uint4(0, 0, 0, 0);
    if (lane == 0) {
        a.pvalid[orow] = ok ? 1 : 0;
        if (a.pidx)
            for (int s = 0; s < KP; ++s) a.pidx[orow * KP + s] = t0 + s;
    }
}

template <int IHD, int KPMAX>
int launch(CompressArgs a, int pmax, cudaStream_t st) {
    constexpr int PPC = (32 / (IHD / 8)) * (kThreads / 32);
    a.tiles = (pmax + PPC - 1) / PPC;
    const long long units = (long long)a.tiles * a.pg.batch;
    if (units == 0) return DSA_OK;
    const int sms = sm_count() > 0 ? sm_count() : 148;
    const long long grid = units < 2LL * sms ? units : 2LL * sms;  // two CTAs fit per SM
    cudaError_t le = launch_pdl(compress_kernel<IHD, KPMAX>, dim3((unsigned)grid), dim3(kThreads),
                                0, st, a);
    if (le != cudaSuccess) return cuda_fail(le, "dsa_compress launch");
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "dsa_compress launch");
    return DSA_OK;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

namespace {
int compress_impl(const char* name, const dsa_bf16* k_raw, const dsa_bf16* gate,
                  const uint8_t* token_valid, const float* ape, const dsa_bf16* ln_w,
                  const dsa_bf16* ln_b, float eps, const dsa_paging* pg, int first_key, int kpool,
                  int ihd, int append, dsa_bf16* kpool_out, uint8_t* pool_valid,
                  int32_t* pool_idx, int32_t* status, void* stream) {
    if (kpool < 1 || kpool > DSA_MAX_KPOOL)
        return fail(DSA_ERR_UNSUPPORTED, "%s: kpool %d outside [1, %d]", name, kpool,
                    DSA_MAX_KPOOL);
    if (ihd != 64 && ihd != 128)
        return fail(DSA_ERR_UNSUPPORTED, "%s: index_head_dim %d not in {64, 128}", name, ihd);
    if (first_key < 0) return fail(DSA_ERR_INVALID_ARG, "%s: first_key %d < 0", name, first_key);
    if (!(eps >= 0.f)) return fail(DSA_ERR_INVALID_ARG, "%s: eps must be >= 0", name);
    Paging P;
    int rc = check_paging(pg, kpool, &P);
    if (rc) return rc;
    if (P.block_table && first_key % kpool != 0)
        return fail(DSA_ERR_UNSUPPORTED,
                    "%s: paged layout needs first_key %% kpool == 0 (got %d, %d)", name,
                    first_key, kpool);
    if (!k_raw || !gate || !token_valid || !ape || !ln_w || !ln_b || !kpool_out || !pool_valid)
        return fail(DSA_ERR_INVALID_ARG, "%s: NULL tensor", name);
    if ((((uintptr_t)k_raw) | ((uintptr_t)gate) | ((uintptr_t)kpool_out) | ((uintptr_t)ape) |
         ((uintptr_t)ln_w) | ((uintptr_t)ln_b)) & 15)
        return fail(DSA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", name);
    const int full = P.max_seq_len > first_key ? (P.max_seq_len - first_key) / kpool : 0;
    // At most ceil(append / kpool) pools become whole over `append` tokens.
    const int pmax = append > 0 ? (int)std::min<long long>(full, (append + (long long)kpool - 1) / kpool)
                                : full;
    CompressArgs a;
    a.k_raw = k_raw;
    a.gate = gate;
    a.valid = token_valid;
    a.ape = ape;
    a.ln_w = ln_w;
    a.ln_b = ln_b;
    a.kout = kpool_out;
    a.pvalid = pool_valid;
    a.pidx = pool_idx;
    a.status = status;
    a.pg = P;
    a.eps = eps;
    a.first_key = first_key;
    a.kpool = kpool;
    a.append = append;
    cudaStream_t st = (cudaStream_t)stream;
    if (ihd == 128) return kpool <= 4 ? launch<128, 4>(a, pmax, st) : launch<128, 16>(a, pmax, st);
    return kpool <= 4 ? launch<64, 4>(a, pmax, st) : launch<64, 16>(a, pmax, st);
}
}  // namespace

extern "C" int dsa_compress(const dsa_bf16* k_raw, const dsa_bf16* gate,
                            const uint8_t* token_valid, const float* ape, const dsa_bf16* ln_w,
                            const dsa_bf16* ln_b, float eps, const dsa_paging* pg,
                            int first_key, int kpool, int ihd, dsa_bf16* kpool_out,
                            uint8_t* pool_valid, int32_t* pool_idx, int32_t* status,
                            void* stream) {
    return compress_impl("dsa_compress", k_raw, gate, token_valid, ape, ln_w, ln_b, eps, pg,
                         first_key, kpool, ihd, 0, kpool_out, pool_valid, pool_idx, status,
                         stream);
}

extern "C" int dsa_compress_append(const dsa_bf16* k_raw, const dsa_bf16* gate,
                                   const uint8_t* token_valid, const float* ape,
                                   const dsa_bf16* ln_w, const dsa_bf16* ln_b, float eps,
                                   const dsa_paging* pg, int first_key, int kpool, int ihd,
                                   int new_tokens, dsa_bf16* kpool_out, uint8_t* pool_valid,
                                   int32_t* pool_idx, int32_t* status, void* stream) {
    if (new_tokens < 1)
        return fail(DSA_ERR_INVALID_ARG, "dsa_compress_append: new_tokens %d < 1", new_tokens);
    return compress_impl("dsa_compress_append", k_raw, gate, token_valid, ape, ln_w, ln_b, eps,
                         pg, first_key, kpool, ihd, new_tokens, kpool_out, pool_valid, pool_idx,
                         status, stream);
}

namespace {
// dsa_decode_append and dsa_decode_append_fp8 (ckv8 / ckv_scale set).
int decode_append_impl(const char* name, const dsa_bf16* k_new, const dsa_bf16* gate_new,
                       const dsa_bf16* ckv_new, const float* ape, const dsa_bf16* ln_w,
                       const dsa_bf16* ln_b, float eps, const dsa_paging* pg, int32_t* seq_lens,
                       int first_key, int kpool, int ihd, int kv_lora_rank, dsa_bf16* k_raw,
                       dsa_bf16* gate, uint8_t* token_valid, dsa_bf16* ckv, uint8_t* ckv8,
                       float* ckv_scale, dsa_bf16* kpool_out, uint8_t* pool_valid,
                       int32_t* pool_idx, int32_t* row_ctx, int32_t* status, void* stream) {
    if (kpool < 1 || kpool > DSA_MAX_KPOOL)
        return fail(DSA_ERR_UNSUPPORTED, "%s: kpool %d outside [1, %d]", name, kpool,
                    DSA_MAX_KPOOL);
    if (ihd != 64 && ihd != 128)
        return fail(DSA_ERR_UNSUPPORTED, "%s: index_head_dim %d not in {64, 128}", name, ihd);
    if (first_key < 0) return fail(DSA_ERR_INVALID_ARG, "%s: first_key %d < 0", name, first_key);
    if (!(eps >= 0.f)) return fail(DSA_ERR_INVALID_ARG, "%s: eps must be >= 0", name);
    const bool fp8 = ckv8 != nullptr;
    if (fp8 != (ckv_scale != nullptr))
        return fail(DSA_ERR_INVALID_ARG, "%s: ckv_codes and ckv_scales go together", name);
    if (fp8 ? !ckv_new : (ckv == nullptr) != (ckv_new == nullptr))
        return fail(DSA_ERR_INVALID_ARG, "%s: ckv_new and the latent cache go together", name);
    if (ckv_new && (kv_lora_rank < 8 || kv_lora_rank % 8 != 0))
        return fail(DSA_ERR_INVALID_ARG, "%s: kv_lora_rank %d not a multiple of 8", name,
                    kv_lora_rank);
    if (fp8 && kv_lora_rank % 128 != 0)
        return fail(DSA_ERR_INVALID_ARG, "%s: kv_lora_rank %d not a multiple of 128", name,
                    kv_lora_rank);
    Paging P;
    int rc = check_paging(pg, kpool, &P);
    if (rc) return rc;
    if (P.block_table && first_key % kpool != 0)
        return fail(DSA_ERR_UNSUPPORTED,
                    "%s: paged layout needs first_key %% kpool == 0 (got %d, %d)", name,
                    first_key, kpool);
    if (!seq_lens || seq_lens != pg->seq_lens)
        return fail(DSA_ERR_INVALID_ARG, "%s: seq_lens must be the descriptor's (writable) lengths",
                    name);
    if (!k_new || !gate_new || !k_raw || !gate || !token_valid || !ape || !ln_w || !ln_b ||
        !kpool_out || !pool_valid)
        return fail(DSA_ERR_INVALID_ARG, "%s: NULL tensor", name);
    if ((((uintptr_t)k_new) | ((uintptr_t)gate_new) | ((uintptr_t)ckv_new) | ((uintptr_t)k_raw) |
         ((uintptr_t)gate) | ((uintptr_t)ckv) | ((uintptr_t)kpool_out) | ((uintptr_t)ape) |
         ((uintptr_t)ln_w) | ((uintptr_t)ln_b) | ((uintptr_t)ckv8) | ((uintptr_t)ckv_scale)) & 15)
        return fail(DSA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", name);
    AppendArgs a;
    a.k_new = k_new;
    a.gate_new = gate_new;
    a.ckv_new = ckv_new;
    a.k_raw = k_raw;
    a.gate = gate;
    a.valid = token_valid;
    a.ckv = ckv;
    a.ckv8 = ckv8;
    a.ckv_scale = ckv_scale;
    a.seq_lens = seq_lens;
    a.row_ctx = row_ctx;
    a.status = status;
    a.ape = ape;
    a.ln_w = ln_w;
    a.ln_b = ln_b;
    a.kout = kpool_out;
    a.pvalid = pool_valid;
    a.pidx = pool_idx;
    a.pg = P;
    a.eps = eps;
    a.first_key = first_key;
    a.kpool = kpool;
    a.kvl = kv_lora_rank;
    const dim3 grid((unsigned)P.batch), block(kAppendThreads);
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e;
    if (ihd == 128)
        e = kpool <= 4 ? launch_pdl(decode_append_kernel<128, 4>, grid, block, 0, st, a)
                       : launch_pdl(decode_append_kernel<128, 16>, grid, block, 0, st, a);
    else
        e = kpool <= 4 ? launch_pdl(decode_append_kernel<64, 4>, grid, block, 0, st, a)
                       : launch_pdl(decode_append_kernel<64, 16>, grid, block, 0, st, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "dsa_decode_append launch");
    return DSA_OK;
}
}  // namespace

extern "C" int dsa_decode_append(const dsa_bf16* k_new, const dsa_bf16* gate_new,
                                 const dsa_bf16* ckv_new, const float* ape, const dsa_bf16* ln_w,
                                 const dsa_bf16* ln_b, float eps, const dsa_paging* pg,
                                 int32_t* seq_lens, int first_key, int kpool, int ihd,
                                 int kv_lora_rank, dsa_bf16* k_raw, dsa_bf16* gate,
                                 uint8_t* token_valid, dsa_bf16* ckv, dsa_bf16* kpool_out,
                                 uint8_t* pool_valid, int32_t* pool_idx, int32_t* row_ctx,
                                 int32_t* status, void* stream) {
    return decode_append_impl("dsa_decode_append", k_new, gate_new, ckv_new, ape, ln_w, ln_b, eps,
                              pg, seq_lens, first_key, kpool, ihd, kv_lora_rank, k_raw, gate,
                              token_valid, ckv, nullptr, nullptr, kpool_out, pool_valid, pool_idx,
                              row_ctx, status, stream);
}

extern "C" int dsa_decode_append_fp8(const dsa_bf16* k_new, const dsa_bf16* gate_new,
                                     const dsa_bf16* ckv_new, const float* ape,
                                     const dsa_bf16* ln_w, const dsa_bf16* ln_b, float eps,
                                     const dsa_paging* pg, int32_t* seq_lens, int first_key,
                                     int kpool, int ihd, int kv_lora_rank, dsa_bf16* k_raw,
                                     dsa_bf16* gate, uint8_t* token_valid, dsa_bf16* ckv,
                                     uint8_t* ckv_codes, float* ckv_scales, dsa_bf16* kpool_out,
                                     uint8_t* pool_valid, int32_t* pool_idx, int32_t* row_ctx,
                                     int32_t* status, void* stream) {
    if (!ckv_codes || !ckv_scales)
        return fail(DSA_ERR_INVALID_ARG, "dsa_decode_append_fp8: NULL FP8 cache");
    return decode_append_impl("dsa_decode_append_fp8", k_new, gate_new, ckv_new, ape, ln_w, ln_b,
                              eps, pg, seq_lens, first_key, kpool, ihd, kv_lora_rank, k_raw, gate,
                              token_valid, ckv, ckv_codes, ckv_scales, kpool_out, pool_valid,
                              pool_idx, row_ctx, status, stream);
}
