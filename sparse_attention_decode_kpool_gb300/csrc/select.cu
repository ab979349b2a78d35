// dsa_select: per-row top-k pool selection (dsa_topk_pools).
//
// Page: metrale_model_arch/glm5next_dsa/mod.rs, "Shape of the pipeline" ([Q, P] scores
// -> [Q, select_k] pool ids) and Glm5NextDsaConfig::select_k.
//
// Order: score descending, ties to the lower pool id; -0.0 == +0.0; -inf is never
// chosen. The chosen ids are written in ascending order and padded with -1.
//
// A row is split over a thread-block cluster of C CTAs (C in {1,2,4,8}, chosen so
// that rows x C covers the GPU). Scores become order-preserving u32 keys (0 for
// -inf) in shared memory. Each CTA finds the exact threshold of its slice's top-k:
// the key range [kmin, kmax] gives a monotone 4096-bin index (kmax - key) >> shift; a
// histogram locates the bin holding the k-th key; only that bin's keys are
// collected, and a radix select over the bits that vary inside it (per-warp
// shared-memory histograms) resolves the exact key and how many equal keys to take.
// A ballot-prefix pass then emits the chosen positions in ascending order.
//
// With the radix option, rows split over a cluster (C > 1) take select_radix_kernel:
// the CTAs first share their slices' key bounds, then find the row's k-th key digit by digit (9-bit digits
// of kmax - key, from the top of the row's key range). Each CTA histograms the
// next digit of its slice's keys that match the digits fixed so far and sends the
// histogram to every other CTA of the cluster (bulk copies into the same place of each
// peer's shared memory, completing on that peer's mbarrier); every CTA sums the C
// histograms and walks them from the top to the bin holding the k-th key, so all CTAs
// reach the same bin. Keys in higher bins are chosen. As soon as the bin holds few
// enough keys, each CTA sends its keys of the bin to every peer, and every CTA ranks
// the gathered keys (radix passes in shared memory): the k-th key T and how many keys
// equal to T are taken (the lowest pool ids first, i.e. lower CTA ranks first, then
// lower positions). Once every bit is fixed the bin holds one key value and nothing
// is gathered. Every CTA then knows how many keys each CTA takes, hence its own offset in
// the output row, and emits its chosen positions there in ascending order.
//
// The default form for clustered rows merges instead: every CTA stages its slice's
// top-kt (key, id) pairs, kt = min(k, 2 ceil(k / C)), in its own slot of a merge area
// (unused entries get key 0) and moves the slot to the same place in CTA 0 with bulk
// copies that complete on an mbarrier there; CTA 0 then selects the row's top-k among
// the C x kt candidates, slot order keeping the ids ascending. That is exact when each
// slice that left keys out has its threshold below the candidates' k-th key; when one
// does not (the row's top keys crowd into few slices), CTA 0 tells the other CTAs and
// the exchange is repeated with every slice's full top-k, whose union always holds the
// row's top-k.
#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxChunk = 40960;      // keys per CTA slice
constexpr int kMaxCluster = 8;
constexpr int kMaxSmem = 200 * 1024;  // dynamic shared memory per CTA
constexpr int kBins = 4096;
constexpr int kRankMax = 128;        // threshold bins up to this size are ranked directly

struct SelectArgs {
    const float* scores;
    int32_t* pool_ids;
    int rows;
    int p_stride;
    int sk;
    int chunk;
    int merge_off;  // byte offsets in dynamic shared memory: merge keys, then ids
    int tbuf_off;   // the threshold bin's scratch list
    int tcap;       // its capacity (keys)
    int32_t* tok;   // nullable: token ids [rows, ow] (dsa_select_expand)
    int first_key;
    int kpool;
    int ow;
    const int32_t* row_ctx;  // nullable: rows' context lengths, for the tail tokens
    int tail_at;             // token-id position of the first tail slot (ow: no tail)
};

// Orders this thread's shared-memory writes before later bulk (async proxy) copies.
__device__ __forceinline__ void fence_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
// Cluster barrier halves (every thread of every CTA of the cluster arrives).
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// bytes (a multiple of 16) from this CTA's shared memory at src to dst in CTA
// `rank`'s shared memory (same offsets), completing on that CTA's mbarrier bar.
__device__ __forceinline__ void bulk_to_peer(const void* src, const void* dst, uint32_t bytes,
                                             const uint64_t* bar, uint32_t rank) {
    uint32_t d, b;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(d) : "r"(smem_u32(dst)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(b) : "r"(smem_u32(bar)), "r"(rank));
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];\n" ::"r"(d),
        "r"(smem_u32(src)), "r"(bytes), "r"(b)
        : "memory");
}

__device__ __forceinline__ uint32_t score_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) == 0u) u = 0u;  // -0.0 == +0.0
    if (u == 0xff800000u) return 0u;      // -inf: not a candidate
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct BlockScratch {
    uint32_t hist[kBins];  // 4096-bin histogram, or 16 per-warp 256-bin histograms
    uint32_t tot[256];
    int pick[4];
    uint32_t wmax[kWarps], wmin[kWarps];
    int wcnt[kWarps];
    int tcount;
};

// Chosen keys: every key > T plus the first need_eq keys == T in position order;
// kk keys in all.
struct Thr {
    uint32_t T;
    int need_eq;
    int kk;
};

struct MinMax {
    uint32_t kmin, kmax;
    int count;
};

// Combine per-thread (min, max, count) of nonzero keys over the block.
__device__ __noinline__ MinMax block_minmax(uint32_t mn, uint32_t mx, int cnt, BlockScratch& sc) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, off));
        cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
    }
    if (lane == 0) {
        sc.wmax[warp] = mx;
        sc.wmin[warp] = mn;
        sc.wcnt[warp] = cnt;
    }
    __syncthreads();
    MinMax r{0xffffffffu, 0u, 0};
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        r.kmax = max(r.kmax, sc.wmax[w]);
        r.kmin = min(r.kmin, sc.wmin[w]);
        r.count += sc.wcnt[w];
    }
    __syncthreads();  // w* arrays are reused by the caller
    return r;
}

// Exact k-th largest key of the nonzero keys in keys[0..n), whose min, max and
// count are mm. Radix passes of 8 bits over v = key - kmin, only over the bits
// v can have. With allow_all, k >= count means "take every nonzero key".
__device__ __noinline__ Thr radix_threshold(const uint32_t* keys, int n, int k, MinMax mm,
                                            BlockScratch& sc, bool allow_all) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (mm.count == 0) return Thr{0xffffffffu, 0, 0};
    const int kk = min(k, mm.count);
    if (allow_all && mm.count <= k) return Thr{0u, 0, kk};
    if (mm.kmin == mm.kmax) return Thr{mm.kmax, kk, kk};
    const uint32_t range = mm.kmax - mm.kmin;
    const int bits = 32 - __clz(range);
    const int passes = (bits + 7) >> 3;
    uint32_t prefix = 0u;  // over v, bits above the current digit
    int krem = kk;
    for (int p = passes - 1; p >= 0; --p) {
        const int shift = 8 * p;
        const uint32_t hmask = (shift + 8 >= 32) ? 0u : ~((1u << (shift + 8)) - 1u);
        for (int b = threadIdx.x; b < kBins; b += kThreads) sc.hist[b] = 0u;
        __syncthreads();
        uint32_t* wh = sc.hist + warp * 256;
        for (int i = threadIdx.x; i < n; i += kThreads) {
            const uint32_t key = keys[i];
            if (key) {
                const uint32_t v = key - mm.kmin;
                if ((v & hmask) == prefix) atomicAdd(&wh[(v >> shift) & 255u], 1u);
            }
        }
        __syncthreads();
        if (threadIdx.x < 256) {
            uint32_t t = 0u;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) t += sc.hist[w * 256 + threadIdx.x];
            sc.tot[threadIdx.x] = t;
        }
        __syncthreads();
        if (warp == 0) {
            // lane l covers bins 8*(31-l) .. 8*(31-l)+7, scanned from the top.
            uint32_t cnt[8];
            uint32_t local = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                cnt[j] = sc.tot[8 * (31 - lane) + 7 - j];
                local += cnt[j];
            }
            uint32_t incl = local;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            const uint32_t excl = incl - local;
            if (excl < (uint32_t)krem && (uint32_t)krem <= incl) {
                uint32_t above = excl;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (above + cnt[j] >= (uint32_t)krem) {
                        sc.pick[0] = 8 * (31 - lane) + 7 - j;
                        sc.pick[1] = (int)above;
                        break;
                    }
                    above += cnt[j];
                }
            }
        }
        __syncthreads();
        krem -= sc.pick[1];
        prefix |= (uint32_t)sc.pick[0] << shift;
        __syncthreads();  // pick[] and hist are rewritten by the next pass
    }
    return Thr{prefix + mm.kmin, krem, kk};
}

// Exact threshold of the top-k of keys[0..n) whose nonzero keys have min, max and
// count mm (see the file comment). The k-th key's bin usually holds a handful of
// keys: up to 64 are ranked by one warp with shuffles; more go through radix passes.
__device__ __noinline__ Thr bin_threshold(const uint32_t* keys, int n, int k, MinMax mm,
                                          BlockScratch& sc, uint32_t* tbuf, int tcap) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (mm.count == 0) return Thr{0xffffffffu, 0, 0};
    const int kk = min(k, mm.count);
    if (mm.count <= k) return Thr{0u, 0, kk};          // every nonzero key is chosen
    if (mm.kmax == mm.kmin) return Thr{mm.kmax, kk, kk};  // all equal: lowest positions
    const uint32_t range = mm.kmax - mm.kmin;
    const int bits = 32 - __clz(range);
    const int shift = bits > 12 ? bits - 12 : 0;

    for (int b = threadIdx.x; b < kBins; b += kThreads) sc.hist[b] = 0u;
    if (threadIdx.x == 0) sc.tcount = 0;
    __syncthreads();
    {
        // four independent loads per step (the pass is bound by their latency)
        int i = threadIdx.x;
        for (; i + 3 * kThreads < n; i += 4 * kThreads) {
            uint32_t k4[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) k4[t] = keys[i + t * kThreads];
#pragma unroll
            for (int t = 0; t < 4; ++t)
                if (k4[t]) atomicAdd(&sc.hist[(mm.kmax - k4[t]) >> shift], 1u);
        }
        for (; i < n; i += kThreads) {
            const uint32_t key = keys[i];
            if (key) atomicAdd(&sc.hist[(mm.kmax - key) >> shift], 1u);
        }
    }
    __syncthreads();
    // Thread t owns bins 8t .. 8t+7 (bin 0 holds the largest keys).
    constexpr int BPT = kBins / kThreads;
    uint32_t c[BPT];
    uint32_t local = 0u;
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
        c[j] = sc.hist[BPT * threadIdx.x + j];
        local += c[j];
    }
    uint32_t incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) sc.wcnt[warp] = (int)incl;
    __syncthreads();
    uint32_t wbase = 0u;
    for (int w = 0; w < warp; ++w) wbase += (uint32_t)sc.wcnt[w];
    const uint32_t excl = wbase + incl - local;
    if (excl < (uint32_t)kk && (uint32_t)kk <= excl + local) {
        uint32_t before = excl;
#pragma unroll
        for (int j = 0; j < BPT; ++j) {
            if (before + c[j] >= (uint32_t)kk) {
                sc.pick[0] = BPT * threadIdx.x + j;
                sc.pick[1] = (int)before;
                break;
            }
            before += c[j];
        }
    }
    __syncthreads();
    const uint32_t bstar = (uint32_t)sc.pick[0];
    const int need = kk - sc.pick[1];  // 1 <= need <= nb
    const int nb = (int)sc.hist[bstar];
    if (nb > tcap) {
        __syncthreads();
        return radix_threshold(keys, n, k, mm, sc, true);
    }
    // Collect the bin's keys (order is irrelevant to ranking). Exactly nb keys match,
    // so the slot index stays below nb <= tcap.
    uint32_t bmx = 0u, bmn = 0xffffffffu;
    auto collect = [&](uint32_t key) {
        if (key != 0u && ((mm.kmax - key) >> shift) == bstar) {
            const int at = atomicAdd(&sc.tcount, 1);
            if (at < tcap) tbuf[at] = key;
            bmx = max(bmx, key);
            bmn = min(bmn, key);
        }
    };
    {
        int i = threadIdx.x;
        for (; i + 3 * kThreads < n; i += 4 * kThreads) {
            uint32_t k4[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) k4[t] = keys[i + t * kThreads];
#pragma unroll
            for (int t = 0; t < 4; ++t) collect(k4[t]);
        }
        for (; i < n; i += kThreads) collect(keys[i]);
    }
    if (nb > kRankMax) {
        const MinMax bm = block_minmax(bmn, bmx, 0, sc);  // syncs: tbuf complete after it
        const Thr t = radix_threshold(tbuf, nb, need, MinMax{bm.kmin, bm.kmax, nb}, sc, false);
        return Thr{t.T, t.need_eq, kk};
    }
    __syncthreads();  // tbuf complete
    if (threadIdx.x < nb) {
        // Rank this thread's key against the bin by broadcast reads: the need-th
        // largest is T, and need - (#greater) of the keys equal to T are taken.
        const uint32_t mine = tbuf[threadIdx.x];
        int gt = 0, eq = 0;
        for (int j = 0; j < nb; ++j) {
            const uint32_t a = tbuf[j];
            gt += a > mine;
            eq += a == mine;
        }
        if (gt < need && need <= gt + eq) {  // equal keys write equal values
            sc.pick[2] = (int)mine;
            sc.pick[3] = need - gt;
        }
    }
    __syncthreads();
    return Thr{(uint32_t)sc.pick[2], sc.pick[3], kk};
}

// Where the chosen positions go (one code path for all three uses keeps the kernel
// small: it runs once per CTA, so instruction fetch matters).
struct EmitTo {
    int mode;               // 0: out[rank] = base + pos
                            // 1: rkeys[rank] = keys[pos], rids[rank] = base + pos
                            // 2: out[rank] = ids[pos]
    int base;
    int32_t* out;
    uint32_t* rkeys;
    uint32_t* rids;
    const uint32_t* ids;
    int32_t* tok;  // nullable: also write the pool's token ids at rank*kpool (modes 0, 2)
    int first_key;
    int kpool;
};

__device__ __forceinline__ void emit_one(const EmitTo& e, const uint32_t* keys, int at, int i) {
    if (e.mode == 1) {
        e.rkeys[at] = keys[i];
        e.rids[at] = (uint32_t)(e.base + i);
        return;
    }
    const int p = e.mode == 0 ? e.base + i : (int)e.ids[i];
    e.out[at] = p;
    if (e.tok) {
        const int t0 = e.first_key + p * e.kpool;
        int32_t* dst = e.tok + at * e.kpool;
        if (e.kpool == 4 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0u) {
            *reinterpret_cast<int4*>(dst) = make_int4(t0, t0 + 1, t0 + 2, t0 + 3);
        } else {
            for (int s = 0; s < e.kpool; ++s) dst[s] = t0 + s;
        }
    }
}

// The emit loop of ordered_emit for mode 0, with the per-key work written so that it
// needs no branch: a warp's threads rarely agree on which of their four keys are
// chosen, and a divergent branch per key makes the pass issue-bound. KIND 0: pool
// ids; KIND 2: pool ids and four token ids per pool, 16-byte stores (kpool 4, an
// aligned token row). Used by the kernel that walks single-CTA rows, where the
// pass repeats per row; elsewhere the generic loop below runs (there each CTA runs
// the emit once, and a second loop's instructions cost more to fetch than they save
// under the step's concurrent L2 prefetch).
template <int KIND>
__device__ __forceinline__ void emit_runs(const uint32_t* keys, int i0, int i1, uint32_t T,
                                          int need_eq, int kk, int pos, int eqr, const EmitTo& e) {
    for (int i = i0; i < i1 && pos < kk; i += 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(keys + i);
        const uint32_t k4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t key = i + j < i1 ? k4[j] : 0u;
            const bool eq = key == T;
            const bool sel = (key > T || (eq && eqr < need_eq)) && pos < kk;
            eqr += eq ? 1 : 0;
            const int at = pos;
            pos += sel ? 1 : 0;
            if (sel) {
                const int p = e.base + i + j;
                e.out[at] = p;
                if (KIND == 2) {
                    const int t0 = e.first_key + 4 * p;
                    *reinterpret_cast<int4*>(e.tok + 4 * at) = make_int4(t0, t0 + 1, t0 + 2, t0 + 3);
                }
            }
        }
    }
}

// -1 over the pool ids from rank kk on, and over the token ids from kk*kpool on,
// except that token-id positions tail_at + i hold t0 + i while that is below tend
// (the tokens of the row's trailing partial pool, with always_select_tail).
__device__ __forceinline__ void fill_tail(int32_t* out, int sk, int32_t* tok, int ow, int kpool,
                                          int kk, int tail_at, int t0, int tend) {
    for (int j = kk + threadIdx.x; j < sk; j += blockDim.x) out[j] = -1;
    if (tok)
        for (int j = kk * kpool + threadIdx.x; j < ow; j += blockDim.x) {
            const int t = t0 + (j - tail_at);
            tok[j] = (j >= tail_at && t < tend) ? t : -1;
        }
}

// The trailing partial pool of a row that sees the first L tokens: [t0, L) with
// t0 = first_key + kpool * floor((L - first_key) / kpool); empty when L <= first_key.
__device__ __forceinline__ void tail_range(const SelectArgs& a, int r, int* t0, int* tend) {
    *t0 = 0;
    *tend = 0;
    if (a.row_ctx && a.tok) {
        const int L = __ldg(a.row_ctx + r);
        *t0 = a.first_key + (L > a.first_key ? (L - a.first_key) / a.kpool * a.kpool : 0);
        *tend = L;
    }
}

// Emits every chosen position, ranks ascending with position. Thread t owns the
// contiguous run [t*per, (t+1)*per), per = 4 x an odd number so that the 16-byte
// loads of a quarter warp hit distinct banks; one block scan of its (#greater,
// #equal) counts, packed in 16-bit halves (n <= 65535), gives the rank of its first
// chosen key.
template <bool RUNS>
__device__ __noinline__ void ordered_emit(const uint32_t* keys, int n, Thr t, BlockScratch& sc,
                                          EmitTo e) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t T = t.T;
    const int per = 4 * (((n + 4 * kThreads - 1) / (4 * kThreads)) | 1);
    const int i0 = threadIdx.x * per;
    const int i1 = min(n, i0 + per);
    uint32_t gt = 0u, eq = 0u;
#pragma unroll 4
    for (int i = i0; i < i1; i += 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(keys + i);
        const uint32_t k4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t key = i + j < i1 ? k4[j] : 0u;
            gt += key > T;
            eq += key == T;
        }
    }
    const uint32_t packed = (eq << 16) | gt;
    uint32_t incl = packed;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) sc.wcnt[warp] = (int)incl;
    __syncthreads();
    uint32_t excl = incl - packed;
    for (int w = 0; w < warp; ++w) excl += (uint32_t)sc.wcnt[w];
    int eqr = (int)(excl >> 16);
    int pos = (int)(excl & 0xffffu) + min(eqr, t.need_eq);
    if (RUNS && e.mode == 0 && !e.tok) {
        emit_runs<0>(keys, i0, i1, T, t.need_eq, t.kk, pos, eqr, e);
    } else if (RUNS && e.mode == 0 && e.kpool == 4 &&
               (reinterpret_cast<uintptr_t>(e.tok) & 15u) == 0u) {
        emit_runs<2>(keys, i0, i1, T, t.need_eq, t.kk, pos, eqr, e);
    } else {
        for (int i = i0; i < i1 && pos < t.kk; i += 4) {
            const uint4 v = *reinterpret_cast<const uint4*>(keys + i);
            const uint32_t k4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t key = i + j < i1 ? k4[j] : 0u;
                bool sel = key > T;
                if (key == T) sel = eqr++ < t.need_eq;
                if (sel && pos < t.kk) emit_one(e, keys, pos++, i + j);
            }
        }
    }
    __syncthreads();
}

// Exact top-k of keys[0..n) (key desc, position asc; key 0 never chosen) whose
// nonzero keys have min, max and count mm (bounds may be loose): emits the chosen
// positions ascending and returns how many, min(k, #nonzero keys); *thr gets the
// threshold (every chosen key is >= thr->T).
template <bool RUNS>
__device__ __noinline__ int block_topk(const uint32_t* keys, int n, int k, MinMax mm,
                                       BlockScratch& sc, uint32_t* tbuf, int tcap, EmitTo e,
                                       Thr* thr) {
    const Thr t = bin_threshold(keys, n, k, mm, sc, tbuf, tcap);
    *thr = t;
    if (t.kk == 0) return 0;
    ordered_emit<RUNS>(keys, n, t, sc, e);
    return t.kk;
}

template <bool RUNS>
__device__ __forceinline__ void select_row(const SelectArgs& a, cg::cluster_group& cluster,
                                           int r, uint32_t* keys, BlockScratch& sc);

// ROWS: single-CTA rows (C == 1) taken in turn by a grid of at most one CTA per SM,
// so the start-up of a CTA is paid once per SM rather than once per row. Otherwise
// one row per CTA or cluster.
template <bool ROWS>
__global__ void __launch_bounds__(kThreads, 1) select_kernel(SelectArgs a) {
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    extern __shared__ __align__(16) uint32_t keys[];
    __shared__ BlockScratch sc;
    pdl_wait();
    if (!ROWS) {
        select_row<false>(a, cluster, (int)blockIdx.x / C, keys, sc);
        return;
    }
    for (int r = blockIdx.x; r < a.rows; r += gridDim.x) {
        // this CTA's next row streams into L2 while this one is selected
        const int rn = r + (int)gridDim.x;
        if (threadIdx.x == 0 && rn < a.rows) {
            const float* nxt = a.scores + (long long)rn * a.p_stride;
            const uintptr_t lo = ((uintptr_t)nxt + 15u) & ~(uintptr_t)15u;
            const uintptr_t hi = ((uintptr_t)(nxt + a.p_stride)) & ~(uintptr_t)15u;
            if (hi > lo)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(lo),
                             "r"((uint32_t)(hi - lo))
                             : "memory");
        }
        select_row<true>(a, cluster, r, keys, sc);
        __syncthreads();  // the next row reuses keys[] and the scratch
    }
}

template <bool RUNS>
__device__ __forceinline__ void select_row(const SelectArgs& a, cg::cluster_group& cluster,
                                           int r, uint32_t* keys, BlockScratch& sc) {
    const int C = (int)cluster.num_blocks();
    const int crank = (int)cluster.block_rank();
    uint8_t* dyn = reinterpret_cast<uint8_t*>(keys);
    uint32_t* tbuf = reinterpret_cast<uint32_t*>(dyn + a.tbuf_off);
    const int begin = crank * a.chunk;
    const int n = max(0, min(a.chunk, a.p_stride - begin));
    const float* srow = a.scores + (long long)r * a.p_stride + begin;
    // Merge area (used in CTA 0; the other CTAs stage their own slot there first):
    // keys [C][sk4], ids [C][sk4], bounds [C][4], then the mbarrier the pushes
    // complete on. sk4 = select_k rounded up to whole 16-byte rows.
    const int sk4 = (a.sk + 3) & ~3;
    uint32_t* mloc = reinterpret_cast<uint32_t*>(dyn + a.merge_off);
    uint64_t* mbar = reinterpret_cast<uint64_t*>(mloc + 2 * C * sk4 + 4 * C);
    if (C > 1) {
        if (crank == 0 && threadIdx.x == 0) {
            mbar_init(mbar, 1);
            fence_mbar_init();
        }
        cluster_arrive();  // phase 1: CTA 0's mbarrier exists (waited on before the push)
    }
    uint32_t kmx = 0u, kmn = 0xffffffffu;
    int kcnt = 0;
    auto put = [&](int i, float f) {
        const uint32_t key = score_key(f);
        keys[i] = key;
        if (key) {
            kmx = max(kmx, key);
            kmn = min(kmn, key);
            ++kcnt;
        }
    };
    if ((reinterpret_cast<uintptr_t>(srow) & 15u) == 0u) {
        // 16-byte loads, eight per thread in flight before any is converted.
        const float4* s4 = reinterpret_cast<const float4*>(srow);
        const int nv = n >> 2;
        for (int base = 0; base < nv; base += 8 * kThreads) {
            float4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = base + j * kThreads + threadIdx.x;
                v[j] = i < nv ? __ldg(s4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = base + j * kThreads + threadIdx.x;
                if (i < nv) {
                    put(4 * i, v[j].x);
                    put(4 * i + 1, v[j].y);
                    put(4 * i + 2, v[j].z);
                    put(4 * i + 3, v[j].w);
                }
            }
        }
        for (int i = (nv << 2) + threadIdx.x; i < n; i += kThreads) put(i, __ldg(srow + i));
    } else {
        for (int i = threadIdx.x; i < n; i += kThreads) put(i, __ldg(srow + i));
    }
    const MinMax mm = block_minmax(kmn, kmx, kcnt, sc);  // also publishes keys[]

    int32_t* out = a.pool_ids + (long long)r * a.sk;
    int32_t* tok = a.tok ? a.tok + (long long)r * a.ow : nullptr;
    EmitTo e;
    e.base = begin;
    e.out = out;
    e.rkeys = e.rids = nullptr;
    e.ids = nullptr;
    e.tok = tok;
    e.first_key = a.first_key;
    e.kpool = a.kpool;
    Thr t;
    if (C == 1) {
        e.mode = 0;
        const int kk = block_topk<RUNS>(keys, n, a.sk, mm, sc, tbuf, a.tcap, e, &t);
        int t0, tend;
        tail_range(a, r, &t0, &tend);
        fill_tail(out, a.sk, tok, a.ow, a.kpool, kk, a.tail_at, t0, tend);
        return;
    }

    // Exchange 0: this slice's top-kt, kt = min(k, 2 ceil(k / C)) (twice a slice's share
    // of the row's top-k), staged in slot crank of this CTA's merge area with bounds
    // (chosen keys are >= the slice threshold and <= the slice maximum), count and
    // whether keys were left out; one bulk copy per part moves the slot to the same
    // place in CTA 0, which finds the top-k threshold T of the C x kt candidates. The
    // candidates hold the row's top-k whenever every slice that left keys out has a
    // threshold below T: each left-out key is then below T, so every key >= T is a
    // candidate, and slot order keeps equal keys in id order. Otherwise (a row whose
    // top keys crowd into one slice) exchange 1 repeats it with every slice's
    // full top-k, whose union always holds the row's top-k.
    const int kt = min(a.sk, 2 * ((a.sk + C - 1) / C));
    const bool trim = kt < a.sk;
    uint32_t* st = mloc + 2 * C * sk4;
    uint32_t* again_flag = reinterpret_cast<uint32_t*>(mbar + 1);  // written by CTA 0
    for (int xg = 0;; ++xg) {
        const int kr = xg == 0 ? kt : a.sk;
        const int w = (kr + 3) & ~3;  // slot stride (keys)
        e.mode = 1;
        e.base = begin;
        e.rkeys = mloc + crank * w;
        e.rids = mloc + C * w + crank * w;
        const int kc = block_topk<false>(keys, n, kr, mm, sc, tbuf, a.tcap, e, &t);
        for (int j = kc + threadIdx.x; j < w; j += kThreads) e.rkeys[j] = 0u;
        if (threadIdx.x == 0) {
            st[4 * crank] = kc > 0 ? t.T : 0xffffffffu;
            st[4 * crank + 1] = kc > 0 ? mm.kmax : 0u;
            st[4 * crank + 2] = (uint32_t)kc;
            st[4 * crank + 3] = mm.count > kr ? 1u : 0u;
        }
        // phase 1 (long complete: CTA 0 arrived before its slice work)
        if (xg == 0) cluster_wait();
        const uint32_t slot = (uint32_t)w * 4u;
        if (crank != 0) {
            fence_async_shared();  // the staged slot, written by this CTA's threads ...
            __syncthreads();       // ... is visible to the bulk copies
            if (threadIdx.x == 0) {
                bulk_to_peer(e.rkeys, e.rkeys, slot, mbar, 0);
                bulk_to_peer(e.rids, e.rids, slot, mbar, 0);
                bulk_to_peer(st + 4 * crank, st + 4 * crank, 16, mbar, 0);
            }
            // phase 2 (3 in exchange 1): CTA 0 arrives once every push has landed, so
            // this CTA's shared memory is no longer read when it goes on; in exchange 0
            // it has written again_flag here before it arrives
            cluster_arrive();
            cluster_wait();
            if (xg == 1 || *reinterpret_cast<volatile uint32_t*>(again_flag) == 0u) return;
            continue;
        }
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(mbar, (uint32_t)(C - 1) * (2u * slot + 16u));
            // bounded: a push that never lands leaves the row unselected (all -1)
            sc.pick[0] = mbar_wait(mbar, (uint32_t)xg) ? 1 : 0;
        }
        __syncthreads();
        const bool landed = sc.pick[0] != 0;
        __syncthreads();  // pick[] is scratch of the threshold below
        const uint32_t* mkeys = mloc;
        MinMax mg{0xffffffffu, 0u, 0};
        bool again = false;
        Thr tm{0xffffffffu, 0, 0};
        if (landed) {
            for (int c = 0; c < C; ++c) {
                mg.kmin = min(mg.kmin, st[4 * c]);
                mg.kmax = max(mg.kmax, st[4 * c + 1]);
                mg.count += (int)st[4 * c + 2];
            }
            tm = bin_threshold(mkeys, C * w, a.sk, mg, sc, tbuf, a.tcap);
            if (xg == 0 && trim)
                for (int c = 0; c < C; ++c) again |= st[4 * c + 3] != 0u && !(st[4 * c] < tm.T);
        }
        if (xg == 0 && threadIdx.x > 0 && threadIdx.x < C) {
            uint32_t d;
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n"
                         : "=r"(d)
                         : "r"(smem_u32(again_flag)), "r"((uint32_t)threadIdx.x));
            asm volatile("st.shared::cluster.u32 [%0], %1;\n" ::"r"(d), "r"(again ? 1u : 0u)
                         : "memory");
        }
        // phase 2 (3 in exchange 1): the pushed slots are in; the other CTAs may go on
        __syncwarp();
        cluster_arrive();
        if (!again) {
            int kk = 0;
            if (landed && tm.kk > 0) {
                e.mode = 2;
                e.base = 0;
                e.ids = mkeys + C * w;
                ordered_emit<false>(mkeys, C * w, tm, sc, e);
                kk = tm.kk;
            }
            int t0, tend;
            tail_range(a, r, &t0, &tend);
            fill_tail(out, a.sk, tok, a.ow, a.kpool, kk, a.tail_at, t0, tend);
            cluster_wait();
            return;
        }
        cluster_wait();  // phase 2 (complete) before exchange 1's arrive
    }
}

// ---------------------------------------------------------------------------
// Cluster top-k by radix digits (see the file comment).

constexpr int kDigitBits = 9;
constexpr int kDigitBins = 1 << kDigitBits;
constexpr int kRounds = 6;  // bounds, up to four digits, one key gather

struct RadixLayout {
    int hist_off;  // byte offsets in dynamic shared memory: histograms [2][C][kDigitBins]
    int mm_off;    // slice bounds [C][4]: min key, max key, nonzero keys, 0
    int list_off;  // the gathered keys of the final bin
    int list_cap;  // its capacity (keys)
    int bar_off;   // kRounds mbarriers
};

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}
// Returns once every bulk copy this thread committed has finished reading its source.
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}

// Thread 0 sends bytes (a multiple of 16) at src to the same offset in every other CTA
// of the cluster and waits until `expect` bytes from the peers have landed here on
// bar. Returns false (in every thread) if that wait gave up.
__device__ __noinline__ bool exchange(const void* src, uint32_t bytes, uint64_t* bar,
                                      uint32_t expect, int C, int crank, BlockScratch& sc) {
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(bar, expect);
        if (bytes) {
            for (int p = 0; p < C; ++p)
                if (p != crank) bulk_to_peer(src, src, bytes, bar, (uint32_t)p);
            bulk_commit();
        }
        sc.pick[0] = mbar_wait(bar, 0) ? 1 : 0;
    }
    __syncthreads();
    const bool ok = sc.pick[0] != 0;
    __syncthreads();  // pick[] is scratch again
    return ok;
}

// Digits are taken over v = kmax - key (0 for the row's largest key), the row's key
// range split into 9-bit digits from the top: the first digit's bins are spread over
// the keys the row actually holds.
__global__ void __launch_bounds__(kThreads, 1) select_radix_kernel(SelectArgs a, RadixLayout L) {
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int crank = (int)cluster.block_rank();
    const int r = (int)blockIdx.x / C;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    extern __shared__ __align__(16) uint32_t keys[];
    __shared__ BlockScratch sc;
    __shared__ int above_c[kMaxCluster];  // per CTA: its keys above the current bin
    __shared__ int bin_c[kMaxCluster];    // per CTA: its keys in the current bin
    __shared__ int gt_c[kMaxCluster], eq_c[kMaxCluster];
    __shared__ int res[8];
    uint8_t* dyn = reinterpret_cast<uint8_t*>(keys);
    uint32_t* hist0 = reinterpret_cast<uint32_t*>(dyn + L.hist_off);
    uint32_t* mmv = reinterpret_cast<uint32_t*>(dyn + L.mm_off);
    uint32_t* list = reinterpret_cast<uint32_t*>(dyn + L.list_off);
    uint64_t* bars = reinterpret_cast<uint64_t*>(dyn + L.bar_off);

    const int begin = crank * a.chunk;
    const int n = max(0, min(a.chunk, a.p_stride - begin));
    const int k = a.sk;
    int32_t* out = a.pool_ids + (long long)r * a.sk;
    int32_t* tok = a.tok ? a.tok + (long long)r * a.ow : nullptr;

    if (tid == 0) {
        for (int i = 0; i < kRounds; ++i) mbar_init(bars + i, 1);
        fence_mbar_init();
    }
    if (tid < kMaxCluster) above_c[tid] = 0;
    cluster_arrive();  // the mbarriers exist before any peer's first copy
    pdl_wait();

    // ---- slice -> order-preserving keys, with their bounds
    const float* srow = a.scores + (long long)r * a.p_stride + begin;
    uint32_t kmx = 0u, kmn = 0xffffffffu;
    int kcnt = 0;
    auto put = [&](int i, float f) {
        const uint32_t key = score_key(f);
        keys[i] = key;
        if (key) {
            kmx = max(kmx, key);
            kmn = min(kmn, key);
            ++kcnt;
        }
    };
    if ((reinterpret_cast<uintptr_t>(srow) & 15u) == 0u) {
        const float4* s4 = reinterpret_cast<const float4*>(srow);
        const int nv = n >> 2;
        for (int base = 0; base < nv; base += 8 * kThreads) {
            float4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = base + j * kThreads + tid;
                v[j] = i < nv ? __ldg(s4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = base + j * kThreads + tid;
                if (i < nv) {
                    put(4 * i, v[j].x);
                    put(4 * i + 1, v[j].y);
                    put(4 * i + 2, v[j].z);
                    put(4 * i + 3, v[j].w);
                }
            }
        }
        for (int i = (nv << 2) + tid; i < n; i += kThreads) put(i, __ldg(srow + i));
    } else {
        for (int i = tid; i < n; i += kThreads) put(i, __ldg(srow + i));
    }
    const MinMax sm = block_minmax(kmn, kmx, kcnt, sc);  // also publishes keys[]
    if (tid == 0) {
        mmv[4 * crank] = sm.kmin;
        mmv[4 * crank + 1] = sm.kmax;
        mmv[4 * crank + 2] = (uint32_t)sm.count;
        mmv[4 * crank + 3] = 0u;
        fence_async_shared();
    }
    __syncthreads();
    cluster_wait();

    // ---- the row's bounds
    bool ok = exchange(mmv + 4 * crank, 16u, bars + 0, (uint32_t)(C - 1) * 16u, C, crank, sc);
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    int total = 0;
    for (int c = 0; c < C; ++c) {
        if (mmv[4 * c + 2] == 0u) continue;
        kmin = min(kmin, mmv[4 * c]);
        kmax = max(kmax, mmv[4 * c + 1]);
        total += (int)mmv[4 * c + 2];
    }
    const bool take_all = total <= k;  // every finite score is chosen

    // ---- digits of v = kmax - key, from the top, down to the bin of the k-th key
    int A = 0;            // keys of the row above the current bin
    uint32_t prefix = 0u; // v >> hi of the keys in the current bin
    int hi = kmax > kmin ? 32 - __clz(kmax - kmin) : 0;  // low bits of v still open
    int nB = total;
    if (ok && !take_all && hi > 0) {
        for (int level = 0;; ++level) {
            const int d = min(kDigitBits, hi);
            const int lo = hi - d;
            const int nbins = 1 << d;
            uint32_t* hist = hist0 + (level & 1) * C * kDigitBins;
            uint32_t* myh = hist + crank * kDigitBins;
            // This buffer was last read two levels ago: every peer has finished that
            // level (it needed this CTA's histogram of the level in between), and this
            // CTA's own copies out of it are done once bulk_wait_read returns.
            if (tid == 0) bulk_wait_read();
            for (int b = tid; b < nbins; b += kThreads) myh[b] = 0u;
            __syncthreads();
            for (int i = tid; i < n; i += kThreads) {
                const uint32_t key = keys[i];
                const uint32_t v = kmax - key;
                if (key != 0u && (hi >= 32 ? 0u : v >> hi) == prefix)
                    atomicAdd(&myh[(v >> lo) & (uint32_t)(nbins - 1)], 1u);
            }
            fence_async_shared();
            __syncthreads();
            if (!exchange(myh, (uint32_t)nbins * 4u, bars + 1 + level, (uint32_t)(C - 1) * nbins * 4u,
                          C, crank, sc)) {
                ok = false;
                break;
            }
            // thread t owns bin t (bin 0: the largest keys)
            uint32_t g = 0u;
            if (tid < nbins)
                for (int c = 0; c < C; ++c) g += hist[c * kDigitBins + tid];
            uint32_t incl = g;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t x = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += x;
            }
            if (lane == 31) sc.wcnt[warp] = (int)incl;
            __syncthreads();
            uint32_t wbase = 0u;
            for (int w = 0; w < warp; ++w) wbase += (uint32_t)sc.wcnt[w];
            const uint32_t need = (uint32_t)(k - A);
            const uint32_t excl = wbase + incl - g;
            if (tid < nbins && excl < need && need <= excl + g) {
                res[0] = tid;
                res[1] = (int)excl;
                res[2] = (int)g;
            }
            __syncthreads();
            const int B = res[0];
            A += res[1];
            nB = res[2];
            // each CTA's keys above the bin and in it (warp c sums CTA c's bins)
            if (warp < C) {
                uint32_t s = 0u;
                for (int b = lane; b < B; b += 32) s += hist[warp * kDigitBins + b];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
                if (lane == 0) {
                    above_c[warp] += (int)s;
                    bin_c[warp] = (int)hist[warp * kDigitBins + B];
                }
            }
            prefix = (prefix << d) | (uint32_t)B;
            hi = lo;
            __syncthreads();  // res[], sc.wcnt, above_c, bin_c
            if (hi == 0 || nB + 3 * C <= L.list_cap) break;
        }
    } else if (ok && !take_all) {
        // one key value (kmin == kmax): it is T, and every CTA's keys are equal to it
        if (tid < C) bin_c[tid] = (int)mmv[4 * tid + 2];
        __syncthreads();
    }

    Thr t{0u, 0, 0};  // this CTA's threshold, its quota of keys equal to T, its count
    int off = 0, K = 0;
    if (ok && take_all) {
        // each CTA takes all of its finite keys; T = 0 takes every nonzero key
        if (tid == 0) {
            int o = 0;
            for (int c = 0; c < C; ++c) {
                if (c == crank) {
                    res[3] = o;
                    res[4] = (int)mmv[4 * c + 2];
                }
                o += (int)mmv[4 * c + 2];
            }
            res[5] = o;
        }
        __syncthreads();
        off = res[3];
        t = Thr{0u, 0, res[4]};
        K = res[5];
    } else if (ok) {
        const int need = k - A;  // keys still to take from the bin: 1 <= need <= nB
        uint32_t T = 0u;
        int need_eq = 0;
        if (hi == 0) {
            // the bin is a single key value
            T = kmax - prefix;
            need_eq = need;
            if (tid < C) {
                gt_c[tid] = 0;
                eq_c[tid] = bin_c[tid];
            }
        } else {
            // gather the bin's keys: CTA c's at list offset sum_{c' < c} pad4(bin_c')
            int loff = 0, ltot = 0;
            for (int c = 0; c < C; ++c) {
                const int padded = (bin_c[c] + 3) & ~3;
                if (c < crank) loff += padded;
                ltot += padded;
            }
            const int mine = (bin_c[crank] + 3) & ~3;
            if (tid == 0) sc.tcount = 0;
            __syncthreads();
            for (int i = tid; i < n; i += kThreads) {
                const uint32_t key = keys[i];
                if (key != 0u && ((kmax - key) >> hi) == prefix) {
                    const int at = atomicAdd(&sc.tcount, 1);
                    if (at < mine) list[loff + at] = key;
                }
            }
            if (tid < mine - bin_c[crank]) list[loff + bin_c[crank] + tid] = 0u;  // padding
            fence_async_shared();
            __syncthreads();
            if (!exchange(list + loff, (uint32_t)mine * 4u, bars + kRounds - 1,
                          (uint32_t)(ltot - mine) * 4u, C, crank, sc)) {
                ok = false;
            } else {
                uint32_t mx = 0u, mn = 0xffffffffu;
                int cnt = 0;
                for (int i = tid; i < ltot; i += kThreads) {
                    const uint32_t key = list[i];
                    if (key) {
                        mx = max(mx, key);
                        mn = min(mn, key);
                        ++cnt;
                    }
                }
                const MinMax mm = block_minmax(mn, mx, cnt, sc);
                const Thr th = radix_threshold(list, ltot, need, mm, sc, false);
                T = th.T;
                need_eq = th.need_eq;
                // each CTA's keys of the bin above T and equal to T
                if (warp < C) {
                    int lo = 0;
                    for (int c = 0; c < warp; ++c) lo += (bin_c[c] + 3) & ~3;
                    int gt = 0, eq = 0;
                    for (int i = lo + lane; i < lo + bin_c[warp]; i += 32) {
                        const uint32_t key = list[i];
                        gt += key > T;
                        eq += key == T;
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        gt += __shfl_xor_sync(0xffffffffu, gt, o);
                        eq += __shfl_xor_sync(0xffffffffu, eq, o);
                    }
                    if (lane == 0) {
                        gt_c[warp] = gt;
                        eq_c[warp] = eq;
                    }
                }
            }
        }
        __syncthreads();
        if (ok) {
            // quotas of T-keys go to the lowest CTA ranks first; offsets follow
            if (tid == 0) {
                int eqp = 0, o = 0;
                for (int c = 0; c < C; ++c) {
                    const int q = min(eq_c[c], max(0, need_eq - eqp));
                    eqp += eq_c[c];
                    const int sel = above_c[c] + gt_c[c] + q;
                    if (c == crank) {
                        res[3] = o;
                        res[4] = sel;
                        res[5] = q;
                    }
                    o += sel;
                }
                res[6] = o;
            }
            __syncthreads();
            off = res[3];
            t = Thr{T, res[5], res[4]};
            K = res[6];
        }
    }

    int t0, tend;
    tail_range(a, r, &t0, &tend);
    if (!ok) {
        // a copy that never landed: this row is left unselected
        fill_tail(out, a.sk, tok, a.ow, a.kpool, 0, a.tail_at, t0, tend);
    } else {
        if (t.kk > 0) {
            EmitTo e;
            e.mode = 0;
            e.base = begin;
            e.out = out + off;
            e.rkeys = e.rids = nullptr;
            e.ids = nullptr;
            e.tok = tok ? tok + (long long)off * a.kpool : nullptr;
            e.first_key = a.first_key;
            e.kpool = a.kpool;
            ordered_emit<false>(keys, n, t, sc, e);
        }
        if (crank == 0) fill_tail(out, a.sk, tok, a.ow, a.kpool, K, a.tail_at, t0, tend);
    }
    if (tid == 0) bulk_wait_read();  // this CTA's outgoing copies have read their sources
    __syncthreads();
    // no CTA leaves while a peer may still copy into it
    cluster_arrive();
    cluster_wait();
}

// Shared memory of select_radix_kernel for slices of `chunk` keys (a list_cap below
// the minimum when it does not fit).
RadixLayout radix_layout(int chunk, int C, long long* bytes) {
    RadixLayout L;
    long long off = ((long long)chunk * 4 + 15) & ~15LL;
    L.hist_off = (int)off;
    off += 2LL * C * kDigitBins * 4;
    L.mm_off = (int)off;
    off += 16LL * kMaxCluster;
    L.bar_off = (int)off;
    off += kRounds * 8;
    L.list_off = (int)((off + 15) & ~15LL);
    off = L.list_off;
    const long long room = (kMaxSmem - off) / 4;
    L.list_cap = (int)(room > 16384 ? 16384 : room);
    *bytes = off + 4LL * (L.list_cap > 0 ? L.list_cap : 0);
    return L;
}

// Dynamic shared memory: the slice's keys (4 B each); with C > 1 the merge area
// (C x sk4 keys and ids, 4 words of bounds per slice and an mbarrier; sk4 = select_k
// rounded up to a multiple of 4); the threshold bin's list.
struct SmemPlan {
    long long merge_off, tbuf_off, tcap, bytes;
};
SmemPlan smem_plan(int p_stride, int sk, int C) {
    const long long chunk = (p_stride + C - 1) / C;
    SmemPlan p;
    p.merge_off = (chunk * 4 + 15) & ~15LL;
    const long long sk4 = (sk + 3) & ~3LL;
    p.tbuf_off = p.merge_off + (C > 1 ? (long long)C * sk4 * 8 + 16LL * C + 16 : 0);
    const long long room = (kMaxSmem - p.tbuf_off) / 4;
    p.tcap = room > 2048 ? 2048 : room;
    p.bytes = p.tbuf_off + 4 * (p.tcap > 0 ? p.tcap : 0);
    return p;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

namespace {
int select_launch(const float* scores, int rows, int p_stride, int sk, int32_t* pool_ids,
                  int32_t* tok, int first_key, int kpool, int ow, const int32_t* row_ctx,
                  int tail_at, void* stream) {
    if ((long long)p_stride > (long long)kMaxChunk * kMaxCluster)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_select: p_stride %d > %d", p_stride,
                    kMaxChunk * kMaxCluster);
    const int sms = sm_count() > 0 ? sm_count() : 148;
    auto fits = [&](int C) {
        const SmemPlan sp = smem_plan(p_stride, sk, C);
        return (p_stride + C - 1) / C <= kMaxChunk && sp.tcap >= 256 && sp.bytes <= kMaxSmem;
    };
    int C = 1;
    while (C < kMaxCluster) {
        const long long chunk = (p_stride + C - 1) / C;
        // A slice of about 8,192 keys per CTA: a CTA's passes over its keys cost about
        // the same up to there, while each further CTA of a cluster adds k keys to
        // the merge (64 rows of 16,384 pools: two CTAs per row take 20.8 us, eight
        // take 43.4 us; 8 rows of 65,536 pools: eight per row 20.8, four 22.9).
        const bool underfilled = (long long)rows * C < 2LL * sms && chunk > 8192;
        if (fits(C) && !underfilled) break;
        if (fits(C) && !fits(2 * C)) break;
        C *= 2;
    }
    if (!fits(C))
        return fail(DSA_ERR_UNSUPPORTED, "dsa_select: p_stride %d with select_k %d does not fit",
                    p_stride, sk);
    const SmemPlan sp = smem_plan(p_stride, sk, C);
    SelectArgs a;
    a.scores = scores;
    a.pool_ids = pool_ids;
    a.rows = rows;
    a.p_stride = p_stride;
    a.sk = sk;
    a.chunk = (p_stride + C - 1) / C;
    a.merge_off = (int)sp.merge_off;
    a.tbuf_off = (int)sp.tbuf_off;
    a.tcap = (int)sp.tcap;
    a.tok = tok;
    a.first_key = first_key;
    a.kpool = kpool;
    a.ow = ow;
    a.row_ctx = row_ctx;
    a.tail_at = row_ctx ? tail_at : ow;
    const bool by_rows = C == 1 && rows > sms;
    // Clustered rows take the radix kernel when its histograms fit beside the slice.
    long long rbytes = 0;
    const RadixLayout rl = radix_layout(a.chunk, C, &rbytes);
    const bool radix = C > 1 && rl.list_cap >= 1024 && select_kernel_choice() == DSA_SELECT_KERNEL_RADIX;
    if ((long long)rows * C > 0x7fffffffLL) return fail(DSA_ERR_UNSUPPORTED, "dsa_select: too many rows");
    cudaLaunchConfig_t cfg = {};
    // single-CTA rows: a grid of at most one CTA per SM walks the rows
    cfg.gridDim = dim3((unsigned)(by_rows ? sms : rows * C));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = radix ? (size_t)rbytes : (size_t)sp.bytes;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    cudaError_t e;
    if (radix) {
        int rc = set_max_smem((const void*)select_radix_kernel, kMaxSmem);
        if (rc) return rc;
        e = cudaLaunchKernelEx(&cfg, select_radix_kernel, a, rl);
    } else {
        auto kernel = by_rows ? select_kernel<true> : select_kernel<false>;
        int rc = set_max_smem((const void*)kernel, kMaxSmem);
        if (rc) return rc;
        e = cudaLaunchKernelEx(&cfg, kernel, a);
    }
    if (e != cudaSuccess) return cuda_fail(e, "dsa_select launch");
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "dsa_select launch");
    return DSA_OK;
}
}  // namespace

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
    return select_launch(scores, rows, p_stride, sk, pool_ids, nullptr, 0, kpool, 0, nullptr, 0,
                         stream);
}

namespace {
// dsa_select_expand and dsa_select_expand_tail (row_ctx != nullptr).
int select_expand_impl(const char* name, const float* scores, int rows, int p_stride,
                       int index_topk, int kpool, int first_key, const int32_t* row_ctx,
                       int out_width, int32_t* pool_ids, int32_t* token_ids, void* stream) {
    if (rows < 0 || p_stride < 0 || first_key < 0 || out_width < 0)
        return fail(DSA_ERR_INVALID_ARG, "%s: rows %d, p_stride %d, first_key %d, out_width %d",
                    name, rows, p_stride, first_key, out_width);
    if (index_topk < 1 || kpool < 1)
        return fail(DSA_ERR_CONFIG, "%s: index_topk %d and kpool %d must be > 0", name,
                    index_topk, kpool);
    if (kpool > DSA_MAX_KPOOL)
        return fail(DSA_ERR_UNSUPPORTED, "%s: kpool %d > %d", name, kpool, DSA_MAX_KPOOL);
    const int sk = dsa_select_k(index_topk, kpool, p_stride);
    if ((long long)sk * kpool > out_width)
        return fail(DSA_ERR_INVALID_ARG, "%s: out_width %d < sk*kpool %lld", name, out_width,
                    (long long)sk * kpool);
    if (row_ctx && (long long)index_topk + kpool - 1 > out_width)
        return fail(DSA_ERR_INVALID_ARG, "%s: out_width %d < index_topk + kpool - 1 = %lld",
                    name, out_width, (long long)index_topk + kpool - 1);
    if (rows == 0) return DSA_OK;
    if (sk == 0) {  // nothing to select: token slots are -1 but for the tail
        if (row_ctx)
            return dsa_expand_tail(nullptr, rows, 0, first_key, kpool, index_topk, row_ctx,
                                   out_width, token_ids, stream);
        return dsa_expand(nullptr, rows, 0, first_key, kpool, out_width, token_ids, stream);
    }
    if (!scores || !pool_ids || (out_width > 0 && !token_ids))
        return fail(DSA_ERR_INVALID_ARG, "%s: NULL tensor", name);
    return select_launch(scores, rows, p_stride, sk, pool_ids, token_ids, first_key, kpool,
                         out_width, row_ctx, index_topk, stream);
}
}  // namespace

extern "C" int dsa_select_expand(const float* scores, int rows, int p_stride, int index_topk,
                                 int kpool, int first_key, int out_width, int32_t* pool_ids,
                                 int32_t* token_ids, void* stream) {
    return select_expand_impl("dsa_select_expand", scores, rows, p_stride, index_topk, kpool,
                              first_key, nullptr, out_width, pool_ids, token_ids, stream);
}

extern "C" int dsa_select_expand_tail(const float* scores, int rows, int p_stride,
                                      int index_topk, int kpool, int first_key,
                                      const int32_t* row_ctx, int out_width, int32_t* pool_ids,
                                      int32_t* token_ids, void* stream) {
    if (!row_ctx && rows > 0)
        return fail(DSA_ERR_INVALID_ARG, "dsa_select_expand_tail: NULL row_ctx");
    return select_expand_impl("dsa_select_expand_tail", scores, rows, p_stride, index_topk,
                              kpool, first_key, row_ctx, out_width, pool_ids, token_ids, stream);
}
