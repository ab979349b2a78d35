// dsa_select: per-row top-k pool selection (dsa_topk_pools).
//
// Page: metrale_model_arch/glm5next_dsa/mod.rs, "Shape of the pipeline" ([Q, P] scores
// -> [Q, select_k] pool ids) and Glm5NextDsaConfig::select_k.
//
// Order: score descending, ties to the lower pool id; -0.0 == +0.0; -inf is never
// chosen. The chosen ids are written in ascending order and padded with -1.
//
// Each row is split over a thread-block cluster of C CTAs (C in {1,2,4,8}); each CTA
// keeps its slice of the row in shared memory as order-preserving u32 keys (0 for
// -inf). An exact radix select finds the k'-th largest key T in four 8-bit passes:
// every pass builds per-CTA histograms of the next digit among keys that match the
// prefix found so far (warp-aggregated with match.any), merges them across the
// cluster through distributed shared memory, and picks the digit where the running
// count from the top reaches the remaining rank. Then every key > T is selected,
// plus the first (in pool order) keys == T needed to reach k'. Positions come from
// a cluster prefix over the CTAs' counts and warp-ballot prefixes inside each
// CTA, so ids are written already in ascending order with no sort.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxChunk = 49152;  // keys per CTA (192 KiB of shared memory)
constexpr int kMaxCluster = 8;

struct SelectArgs {
    const float* scores;
    int32_t* pool_ids;
    int rows;
    int p_stride;
    int sk;
    int chunk;
};

__device__ __forceinline__ uint32_t score_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) == 0u) u = 0u;  // -0.0 == +0.0
    if (u == 0xff800000u) return 0u;      // -inf: not a candidate
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kThreads, 1) select_kernel(SelectArgs a) {
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int crank = (int)cluster.block_rank();
    const int r = blockIdx.x / C;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;

    extern __shared__ uint32_t keys[];
    __shared__ uint32_t hist[256];
    __shared__ uint32_t tot[256];
    __shared__ int s_gt[kWarps], s_eq[kWarps], s_eqb[kWarps], s_selb[kWarps];
    __shared__ int s_cta[2];
    __shared__ int s_pick[3];

    const int begin = crank * a.chunk;
    const int n = max(0, min(a.chunk, a.p_stride - begin));
    const int n32 = (n + 31) & ~31;
    const float* srow = a.scores + (long long)r * a.p_stride + begin;
    for (int i = threadIdx.x; i < n; i += kThreads) keys[i] = score_key(__ldg(srow + i));

    uint32_t prefix = 0u, pmask = 0u;
    int krem = 0, kk = 0;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        if (threadIdx.x < 256) hist[threadIdx.x] = 0u;
        __syncthreads();
        for (int i = threadIdx.x; i < n32; i += kThreads) {
            const uint32_t k = i < n ? keys[i] : 0u;
            const bool take = k != 0u && (k & pmask) == prefix;
            const unsigned act = __ballot_sync(0xffffffffu, take);
            if (take) {
                const uint32_t bin = (k >> shift) & 255u;
                const unsigned peers = __match_any_sync(act, bin);
                if ((__ffs(peers) - 1) == lane) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
            }
        }
        cluster.sync();
        if (threadIdx.x < 256) {
            uint32_t s = 0u;
            for (int c = 0; c < C; ++c) s += cluster.map_shared_rank(hist, c)[threadIdx.x];
            tot[threadIdx.x] = s;
        }
        __syncthreads();
        if (warp == 0) {
            // lane l covers bins 8*(31-l) .. 8*(31-l)+7, scanned from the top.
            uint32_t cnt[8];
            uint32_t local = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                cnt[j] = tot[8 * (31 - lane) + 7 - j];
                local += cnt[j];
            }
            uint32_t incl = local;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            const uint32_t excl = incl - local;
            int want = krem;
            if (pass == 0) {
                const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
                want = min(a.sk, (int)total);
                if (lane == 0) s_pick[2] = want;
            }
            if (want > 0 && excl < (uint32_t)want && (uint32_t)want <= incl) {
                uint32_t above = excl;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (above + cnt[j] >= (uint32_t)want) {
                        s_pick[0] = 8 * (31 - lane) + 7 - j;
                        s_pick[1] = (int)above;
                        break;
                    }
                    above += cnt[j];
                }
            }
        }
        __syncthreads();
        if (pass == 0) {
            kk = s_pick[2];
            krem = kk;
        }
        if (kk == 0) break;  // uniform across the cluster: same merged counts everywhere
        krem -= s_pick[1];
        prefix |= (uint32_t)s_pick[0] << shift;
        pmask |= 255u << shift;
        cluster.sync();  // all remote reads of hist done before it is cleared
    }

    int32_t* out = a.pool_ids + (long long)r * a.sk;
    if (kk > 0) {
        const uint32_t T = prefix;
        const int need_eq = krem;  // keys equal to T still to take, lowest ids first
        const int seg = (((n + kWarps - 1) / kWarps) + 31) & ~31;
        const int w0 = warp * seg;
        const int w1 = min(n, w0 + seg);
        int gt = 0, eq = 0;
        for (int i = w0 + lane; i < w0 + seg; i += 32) {
            const uint32_t k = i < w1 ? keys[i] : 0u;
            gt += __popc(__ballot_sync(0xffffffffu, k > T));
            eq += __popc(__ballot_sync(0xffffffffu, k == T));
        }
        if (lane == 0) {
            s_gt[warp] = gt;
            s_eq[warp] = eq;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int cg_ = 0, ce = 0;
            for (int w = 0; w < kWarps; ++w) {
                cg_ += s_gt[w];
                ce += s_eq[w];
            }
            s_cta[0] = cg_;
            s_cta[1] = ce;
        }
        cluster.sync();
        if (threadIdx.x == 0) {
            int eqb = 0, selb = 0;
            for (int c = 0; c < crank; ++c) {
                const int* rc = cluster.map_shared_rank(s_cta, c);
                const int e = rc[1];
                selb += rc[0] + max(0, min(need_eq - eqb, e));
                eqb += e;
            }
            for (int w = 0; w < kWarps; ++w) {
                s_eqb[w] = eqb;
                s_selb[w] = selb;
                selb += s_gt[w] + max(0, min(need_eq - eqb, s_eq[w]));
                eqb += s_eq[w];
            }
        }
        __syncthreads();
        int eqr = s_eqb[warp], pos = s_selb[warp];
        const unsigned lt = (1u << lane) - 1u;
        for (int i = w0 + lane; i < w0 + seg; i += 32) {
            const uint32_t k = i < w1 ? keys[i] : 0u;
            const unsigned beq = __ballot_sync(0xffffffffu, k == T);
            const bool sel = k > T || (k == T && eqr + __popc(beq & lt) < need_eq);
            const unsigned bsel = __ballot_sync(0xffffffffu, sel);
            const int at = pos + __popc(bsel & lt);
            if (sel && at < kk) out[at] = begin + i;
            eqr += __popc(beq);
            pos += __popc(bsel);
        }
    }
    if (crank == 0)
        for (int j = kk + threadIdx.x; j < a.sk; j += kThreads) out[j] = -1;
    cluster.sync();  // keep this CTA's shared memory alive for remote readers
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" int dsa_select(const float* scores, int rows, int p_stride, int index_topk, int kpool,
                          int32_t* pool_ids, void* stream) {
    if (rows < 0 || p_stride < 0)
        return fail(DSA_ERR_INVALID_ARG, "dsa_select: rows %d, p_stride %d", rows, p_stride);
    if (index_topk < 1 || kpool < 1)
        return fail(DSA_ERR_CONFIG, "dsa_select: index_topk %d and kpool %d must be > 0",
                    index_topk, kpool);
    const int sk = dsa_select_k(index_topk, kpool, p_stride);
    if (rows == 0 || sk == 0) return DSA_OK;
    if (!scores || !pool_ids) return fail(DSA_ERR_INVALID_ARG, "dsa_select: NULL tensor");
    if ((long long)p_stride > (long long)kMaxChunk * kMaxCluster)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_select: p_stride %d > %d", p_stride,
                    kMaxChunk * kMaxCluster);
    const int sms = sm_count() > 0 ? sm_count() : 148;
    int C = 1;
    while (C < kMaxCluster) {
        const int chunk = (p_stride + C - 1) / C;
        const bool too_big = chunk > kMaxChunk;
        const bool underfilled = (long long)rows * C < 2LL * sms && chunk > 2048;
        if (!too_big && !underfilled) break;
        C *= 2;
    }
    SelectArgs a;
    a.scores = scores;
    a.pool_ids = pool_ids;
    a.rows = rows;
    a.p_stride = p_stride;
    a.sk = sk;
    a.chunk = (p_stride + C - 1) / C;
    const int smem = a.chunk * (int)sizeof(uint32_t);
    int rc = set_max_smem((const void*)select_kernel, kMaxChunk * (int)sizeof(uint32_t));
    if (rc) return rc;
    if ((long long)rows * C > 0x7fffffffLL) return fail(DSA_ERR_UNSUPPORTED, "dsa_select: too many rows");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(rows * C));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, select_kernel, a);
    if (e != cudaSuccess) return cuda_fail(e, "dsa_select launch");
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "dsa_select launch");
    return DSA_OK;
}
