// dsa_score: index scores of query rows against their sequence's pooled keys.
//
// Page: metrale_model_arch/glm5next_dsa/tp.rs, "Why the indexer is replicated":
//   score[r, p] = sum_h w[r, h] * max(0, scale * <qidx[r, h, :], kpool[p, :]>)
// for every (query row, pool). build.rs, transform 2: w already carries the
// index_heads^-0.5 factor.
//
// Per pooled key (ihd bf16 = 256 B at ihd 128) the row does index_heads * ihd MACs:
// 16 MAC per byte at 32 x 128, more than the f32 pipes sustain at HBM speed. So the
// contraction [16 pools x ihd] x [ihd x 8 heads] runs on the tensor cores as
// m16n8k16 bf16 MMAs with f32 accumulation, and the head reduction
// sum_h w[h] * relu(scale * acc) happens in the accumulator registers: each thread
// holds 2 pools x 2 heads per 8-head tile, so the sum over heads is a local sum plus
// two xor shuffles inside the lane quad.
//
// Keys are streamed straight from HBM into the MMA A-fragments, without shared
// memory. The dot product does not depend on the order of the ihd axis, so the
// same permutation of that axis is applied to keys and queries: lane quad q owns
// physical elements [32v + 8q, 32v + 8q + 8) of each row, loaded as one 16-byte
// vector per v, which makes every warp load 8 rows x 64 contiguous bytes.
#include "common.cuh"

namespace dsa {
namespace {

struct ScoreArgs {
    const uint16_t* qidx;
    const float* w;
    const int32_t* row_seq;
    const int32_t* row_ctx;
    const uint16_t* kp;
    const uint8_t* pv;
    float* scores;
    int32_t* status;
    Paging pg;
    int rows;
    int heads;
    int first_key;
    int kpool;
    int p_stride;
    int tiles_per_warp;
    int flags_tma;  // pool flags arrive with the keys (alignment allows 16-byte copies)
    float scale;
};

constexpr int kWarps = 4;

template <int IHD, int NT>
__global__ void __launch_bounds__(kWarps * 32) score_kernel(ScoreArgs a) {
    constexpr int NV = IHD / 32;  // 16-byte vectors per row per lane
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = lane >> 2;
    const int q = lane & 3;
    const int r = blockIdx.y;
    const int ntiles = (a.p_stride + 15) >> 4;
    const int t_begin = (blockIdx.x * kWarps + warp) * a.tiles_per_warp;
    if (t_begin >= ntiles) return;
    const int t_end = min(ntiles, t_begin + a.tiles_per_warp);
    float* srow = a.scores + (long long)r * a.p_stride;

    int seq = a.row_seq ? __ldg(a.row_seq + r) : r;
    int nvis = 0;
    if (seq >= 0 && seq < a.pg.batch) {
        int L = min(__ldg(a.pg.seq_lens + seq), seq_capacity(a.pg));
        int ctx = a.row_ctx ? min(__ldg(a.row_ctx + r), L) : L;
        nvis = ctx > a.first_key ? (ctx - a.first_key) / a.kpool : 0;
    } else if (lane == 0 && blockIdx.x == 0 && warp == 0) {
        flag_status(a.status, DSA_STATUS_BAD_TOKEN);
    }

    // Query fragments (B operand): head 8*nt + g, this quad's permuted elements.
    uint32_t bq[NT][NV][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int h = nt * 8 + g;
        const uint16_t* qp = a.qidx + ((long long)r * a.heads + h) * IHD + 8 * q;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            uint4 x = make_uint4(0, 0, 0, 0);
            if (h < a.heads) x = ldg16(qp + 32 * v);
            bq[nt][v][0] = x.x;
            bq[nt][v][1] = x.y;
            bq[nt][v][2] = x.z;
            bq[nt][v][3] = x.w;
        }
    }
    float wv[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int h = nt * 8 + 2 * q + j;
            wv[nt][j] = h < a.heads ? __ldg(a.w + (long long)r * a.heads + h) : 0.f;
        }

    for (int t = t_begin; t < t_end; t += 2) {
        const bool two = (t + 1) < t_end;
        if ((t << 4) >= nvis) {  // nothing visible from here on in this warp's range
            const int p0 = t << 4;
            const int p1 = min(a.p_stride, (t_end << 4));
            for (int p = p0 + lane; p < p1; p += 32) srow[p] = -INFINITY;
            break;
        }
        // This thread's 4 pools: tile t rows g, g+8; tile t+1 rows g, g+8.
        int pool[4];
        pool[0] = (t << 4) + g;
        pool[1] = pool[0] + 8;
        pool[2] = pool[0] + 16;
        pool[3] = pool[0] + 24;
        long long prow[4];
        bool cand[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            prow[i] = -1;
            if (pool[i] < nvis && (i < 2 || two)) {
                prow[i] = pool_row(a.pg, seq, pool[i], a.kpool);
                if (prow[i] < 0) flag_status(a.status, DSA_STATUS_BAD_BLOCK);
            }
        }
        uint4 kr[4][NV];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                kr[i][v] = make_uint4(0, 0, 0, 0);
                if (prow[i] >= 0) kr[i][v] = ldg16_stream(a.kp + prow[i] * IHD + 8 * q + 32 * v);
            }
#pragma unroll
        for (int i = 0; i < 4; ++i) cand[i] = prow[i] >= 0 && __ldg(a.pv + prow[i]) != 0;

#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
            if (tt == 1 && !two) break;
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const uint32_t ra[4] = {kr[2 * tt][v].x, kr[2 * tt][v].y, kr[2 * tt][v].z,
                                        kr[2 * tt][v].w};
                const uint32_t rb[4] = {kr[2 * tt + 1][v].x, kr[2 * tt + 1][v].y,
                                        kr[2 * tt + 1][v].z, kr[2 * tt + 1][v].w};
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_16816(acc[nt], ra[2 * h2], rb[2 * h2], ra[2 * h2 + 1], rb[2 * h2 + 1],
                                  bq[nt][v][2 * h2], bq[nt][v][2 * h2 + 1]);
            }
            float s0 = 0.f, s1 = 0.f;  // rows g and g+8 of this tile
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                s0 += wv[nt][0] * fmaxf(a.scale * acc[nt][0], 0.f) +
                      wv[nt][1] * fmaxf(a.scale * acc[nt][1], 0.f);
                s1 += wv[nt][0] * fmaxf(a.scale * acc[nt][2], 0.f) +
                      wv[nt][1] * fmaxf(a.scale * acc[nt][3], 0.f);
            }
            s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
            s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
            s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
            s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
            if (q < 2) {
                const int p = (t << 4) + g + 8 * (2 * tt + q);
                const bool c = q == 0 ? cand[2 * tt] : cand[2 * tt + 1];
                if (p < a.p_stride) srow[p] = c ? (q == 0 ? s0 : s1) : -INFINITY;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// TMA-fed variant: one producer warp streams runs of 64 pooled keys (16 KiB at
// ihd 128) per stage with bulk async copies into an 8-stage shared-memory ring;
// four consumer warps each turn one 16-pool tile of the stage into MMAs and the
// head reduction. Work units are (row, 64-pool stage) pairs split evenly over one
// CTA per SM. Pool flags are read by the consumers while the keys are in flight.

constexpr int kStagePools = 64;
constexpr int kStages = 3;  // deeper rings measured slower (less L1 beside them)
constexpr int kCtasPerSm = 3;  // 12 consumer warps per SM hide the MMA and shuffle latency
constexpr int kTmaThreads = 5 * 32;
// Paged caches with up to this many rows: the units are the rows' visible stages only,
// split evenly over the CTAs (a CTA finds its first unit by a scan over the rows), and
// the pools past a row's visible stages are filled with -inf afterwards by every CTA.
// A batch of unequal lengths would otherwise leave the CTAs that cover long rows with
// all the copies. (A contiguous cache keeps every stage of every row a unit: its rows
// are usually equal, and the scan would delay the first copy.)
constexpr int kBalRows = 256;

struct RowInfo {
    int seq;
    int nvis;
};

__device__ __forceinline__ RowInfo row_info(const ScoreArgs& a, int r) {
    RowInfo ri;
    ri.seq = a.row_seq ? __ldg(a.row_seq + r) : r;
    ri.nvis = 0;
    if (ri.seq >= 0 && ri.seq < a.pg.batch) {
        const int L = min(__ldg(a.pg.seq_lens + ri.seq), seq_capacity(a.pg));
        const int ctx = a.row_ctx ? min(__ldg(a.row_ctx + r), L) : L;
        ri.nvis = ctx > a.first_key ? (ctx - a.first_key) / a.kpool : 0;
    } else {
        ri.seq = -1;
    }
    return ri;
}

// 64-pool stages of a row that hold visible pools.
__device__ __forceinline__ int vis_stages(const RowInfo& ri, int spr) {
    return ri.seq < 0 ? 0 : min(spr, (ri.nvis + kStagePools - 1) / kStagePools);
}

// Moves (r, st) to the unit to process next and refreshes the row's info when the row
// changes (returns true then). Balanced: rows' stages from their visible count on are
// skipped; otherwise every stage of every row is a unit.
template <bool BAL>
__device__ __forceinline__ bool next_unit(const ScoreArgs& a, int spr, int& r, int& st, int& cur_r,
                                          RowInfo& ri, int& vs) {
    bool changed = false;
    if (BAL) {
        if (r != cur_r) {
            ri = row_info(a, r);
            vs = vis_stages(ri, spr);
            cur_r = r;
            changed = true;
        }
        while (st >= vs && r + 1 < a.rows) {
            ++r;
            st = 0;
            ri = row_info(a, r);
            vs = vis_stages(ri, spr);
            cur_r = r;
            changed = true;
        }
    } else {
        if (st == spr) {
            st = 0;
            ++r;
        }
        if (r != cur_r) {
            ri = row_info(a, r);
            cur_r = r;
            changed = true;
        }
    }
    return changed;
}

template <int IHD, int NT, bool BAL>
__global__ void __launch_bounds__(kTmaThreads, kCtasPerSm) score_tma_kernel(ScoreArgs a) {
    constexpr int NV = IHD / 32;
    constexpr int ROWB = IHD * 2;                    // bytes per pooled key
    constexpr int STAGE = kStagePools * ROWB;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* flags = smem + kStages * STAGE;                                  // [stage][64]
    unsigned long long* bad = reinterpret_cast<unsigned long long*>(flags + kStages * kStagePools);
    uint64_t* full = reinterpret_cast<uint64_t*>(bad + kStages);
    uint64_t* empty = full + kStages;
    long long* s_unit = reinterpret_cast<long long*>(empty + kStages);  // BAL: [u0, u1)
    int* s_first = reinterpret_cast<int*>(s_unit + 2);                  // and u0's (row, stage)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int spr = (a.p_stride + kStagePools - 1) / kStagePools;  // stages per row
    const long long U = (long long)a.rows * spr;
    const long long G = gridDim.x;
    pdl_wait();
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 4);
        }
        fence_mbar_init();
    }
    if (BAL && warp == 0) {
        // visible stages of rows 32k + lane, their total, and the row holding unit u0
        int vsl[kBalRows / 32];
        long long tot = 0;
#pragma unroll
        for (int k = 0; k < kBalRows / 32; ++k) {
            const int rr = 32 * k + lane;
            vsl[k] = rr < a.rows ? vis_stages(row_info(a, rr), spr) : 0;
            tot += vsl[k];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
        const long long b0 = blockIdx.x * tot / G, b1 = (blockIdx.x + 1) * tot / G;
        long long base = 0;
        int r0 = 0, st0 = 0;
        bool found = false;
#pragma unroll
        for (int k = 0; k < kBalRows / 32; ++k) {
            int incl = vsl[k];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            const long long end = base + incl;  // units up to the end of row 32k + lane
            const unsigned m = __ballot_sync(0xffffffffu, !found && end > b0);
            if (m != 0u) {
                const int l = __ffs(m) - 1;
                const long long endl = __shfl_sync(0xffffffffu, end, l);
                const int vl = __shfl_sync(0xffffffffu, vsl[k], l);
                r0 = 32 * k + l;
                st0 = (int)(b0 - (endl - vl));
                found = true;
            }
            base += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            s_unit[0] = b0;
            s_unit[1] = b1;
            s_first[0] = r0;
            s_first[1] = st0;
        }
    }
    __syncthreads();
    const long long u0 = BAL ? s_unit[0] : blockIdx.x * U / G;
    const long long u1 = BAL ? s_unit[1] : (blockIdx.x + 1) * U / G;
    const int r_first = BAL ? s_first[0] : (int)(u0 / spr);
    const int st_first = BAL ? s_first[1] : (int)(u0 % spr);

    if (warp == 4) {
        // ---------------- producer (lane 0 owns the ring; on a paged cache the whole
        // warp resolves the stage's block-table entries, one block per lane, ahead of
        // the slot wait, and each lane copies its block's run of pools)
        const bool paged = a.pg.block_table != nullptr;
        const int ppb = paged ? a.pg.block_size / a.kpool : 1;
        int cur_r = -1, vs = 0;
        RowInfo ri{};
        long long i = 0;
        bool ok = true;
        int r = r_first, st = st_first;
        for (long long u = u0; u < u1; ++u, ++i) {
            const int s = (int)(i % kStages);
            const uint32_t ph = (uint32_t)((i / kStages) & 1);
            if (next_unit<BAL>(a, spr, r, st, cur_r, ri, vs) && lane == 0 && ri.seq < 0 && u == u0)
                flag_status(a.status, DSA_STATUS_BAD_TOKEN);
            const int p0 = st++ * kStagePools;
            const int nvalid = ri.seq < 0 ? 0 : max(0, min(kStagePools, ri.nvis - p0));
            // blocks b0 .. b0 + nb - 1 hold the stage's pools; lane j looks up j and j + 32
            const int b0 = p0 / ppb;
            const int nb = paged && nvalid > 0 ? (p0 + nvalid - 1) / ppb - b0 + 1 : 0;
            long long brow[2] = {-1, -1};  // first pool row of the lane's blocks, -1: bad
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int j = lane + 32 * t;
                if (j < nb) {
                    const int blk = __ldg(a.pg.block_table + (long long)ri.seq * a.pg.max_blocks + b0 + j);
                    brow[t] = blk >= 0 && blk < a.pg.num_blocks ? (long long)blk * ppb : -1;
                }
            }
            int got = 1;
            if (lane == 0) got = mbar_wait(&empty[s], ph ^ 1u) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, got, 0)) {
                ok = false;
                break;
            }
            const uint32_t dst = smem_u32(smem + s * STAGE);
            const uint32_t fdst = smem_u32(flags + s * kStagePools);
            if (!paged) {
                if (lane == 0) {
                    const long long prow0 = (long long)ri.seq * (a.pg.max_seq_len / a.kpool) + p0;
                    const uint32_t kbytes = (uint32_t)(nvalid * ROWB);
                    const uint32_t fbytes = a.flags_tma ? (uint32_t)((nvalid + 15) & ~15) : 0u;
                    bad[s] = 0ull;
                    mbar_arrive_expect_tx(&full[s], kbytes + fbytes);
                    if (kbytes) bulk_g2s(dst, a.kp + prow0 * IHD, kbytes, &full[s]);
                    if (fbytes) bulk_g2s(fdst, a.pv + prow0, fbytes, &full[s]);
                }
                continue;
            }
            // Pools of one block are contiguous: one copy per block run.
            uint32_t bytes = 0;
            unsigned long long badm = 0ull;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int j = lane + 32 * t;
                if (j >= nb) continue;
                const int pb = (b0 + j) * ppb;
                const int ps = max(p0, pb), run = min(p0 + nvalid, pb + ppb) - ps;
                if (brow[t] >= 0) {
                    bytes += (uint32_t)(run * ROWB);
                    if (a.flags_tma) bytes += (uint32_t)((run + 15) & ~15);
                } else {
                    badm |= ((run >= 64) ? ~0ull : ((1ull << run) - 1ull)) << (ps - p0);
                    flag_status(a.status, DSA_STATUS_BAD_BLOCK);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
                badm |= __shfl_xor_sync(0xffffffffu, badm, o);
            }
            if (lane == 0) {
                bad[s] = badm;
                mbar_arrive_expect_tx(&full[s], bytes);
            }
            __syncwarp();  // the stage's bytes are expected before any copy lands
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int j = lane + 32 * t;
                if (j >= nb || brow[t] < 0) continue;
                const int pb = (b0 + j) * ppb;
                const int ps = max(p0, pb), run = min(p0 + nvalid, pb + ppb) - ps;
                const long long row = brow[t] + (ps - pb);
                bulk_g2s(dst + (ps - p0) * ROWB, a.kp + row * IHD, (uint32_t)(run * ROWB), &full[s]);
                if (a.flags_tma)
                    bulk_g2s(fdst + (ps - p0), a.pv + row, (uint32_t)((run + 15) & ~15), &full[s]);
            }
        }
        if (lane == 0) {
            if (!ok) flag_status(a.status, DSA_STATUS_TIMEOUT);
            // the copies issued have landed before the CTA leaves
            const long long first = i > kStages ? i - kStages : 0;
            for (long long j = first; j < i; ++j)
                if (!mbar_wait(&full[j % kStages], (uint32_t)((j / kStages) & 1))) break;
        }
        return;
    }

    // ---------------- consumers: warp w takes pools p0 + 16w .. +15 of each stage
    const int g = lane >> 2, q = lane & 3;
    uint32_t bq[NT][NV][4];
    float wv[NT][2];
    int cur_r = -1, vs = 0;
    RowInfo ri{};
    long long i = 0;
    int r = r_first, st = st_first;
    for (long long u = u0; u < u1; ++u, ++i) {
        const int s = (int)(i % kStages);
        const uint32_t ph = (uint32_t)((i / kStages) & 1);
        const bool new_row = next_unit<BAL>(a, spr, r, st, cur_r, ri, vs);
        const int p0 = st++ * kStagePools + 16 * warp;
        if (new_row) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int h = nt * 8 + g;
                const uint16_t* qp = a.qidx + ((long long)r * a.heads + h) * IHD + 8 * q;
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    uint4 x = make_uint4(0, 0, 0, 0);
                    if (h < a.heads) x = ldg16(qp + 32 * v);
                    bq[nt][v][0] = x.x;
                    bq[nt][v][1] = x.y;
                    bq[nt][v][2] = x.z;
                    bq[nt][v][3] = x.w;
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int hh = nt * 8 + 2 * q + j;
                    wv[nt][j] = hh < a.heads ? __ldg(a.w + (long long)r * a.heads + hh) : 0.f;
                }
            }
        }
        const int pA = p0 + g, pB = pA + 8;
        bool cA = false, cB = false;
        if (!a.flags_tma && ri.seq >= 0) {  // flags not copied with the keys: load them
            if (pA < ri.nvis) {
                const long long rw = pool_row(a.pg, ri.seq, pA, a.kpool);
                cA = rw >= 0 && __ldg(a.pv + rw) != 0;
            }
            if (pB < ri.nvis) {
                const long long rw = pool_row(a.pg, ri.seq, pB, a.kpool);
                cB = rw >= 0 && __ldg(a.pv + rw) != 0;
            }
        }
        if (!mbar_wait(&full[s], ph)) {
            if (lane == 0) flag_status(a.status, DSA_STATUS_TIMEOUT);
            break;
        }
        if (a.flags_tma && ri.seq >= 0) {
            const uint8_t* fl = flags + s * kStagePools + 16 * warp;
            const unsigned long long bm = bad[s] >> (16 * warp);
            cA = pA < ri.nvis && !((bm >> g) & 1ull) && fl[g] != 0;
            cB = pB < ri.nvis && !((bm >> (g + 8)) & 1ull) && fl[g + 8] != 0;
        }
        float sA = 0.f, sB = 0.f;
        if (p0 < ri.nvis) {  // warp-uniform: the tile has visible pools
            const uint32_t base = smem_u32(smem + s * STAGE) + (16 * warp) * ROWB;
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const uint4 ra = lds16(base + g * ROWB + 64 * v + 16 * q);
                const uint4 rb = lds16(base + (g + 8) * ROWB + 64 * v + 16 * q);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mma_16816(acc[nt], ra.x, rb.x, ra.y, rb.y, bq[nt][v][0], bq[nt][v][1]);
                    mma_16816(acc[nt], ra.z, rb.z, ra.w, rb.w, bq[nt][v][2], bq[nt][v][3]);
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                sA += wv[nt][0] * fmaxf(a.scale * acc[nt][0], 0.f) +
                      wv[nt][1] * fmaxf(a.scale * acc[nt][1], 0.f);
                sB += wv[nt][0] * fmaxf(a.scale * acc[nt][2], 0.f) +
                      wv[nt][1] * fmaxf(a.scale * acc[nt][3], 0.f);
            }
            sA += __shfl_xor_sync(0xffffffffu, sA, 1);
            sB += __shfl_xor_sync(0xffffffffu, sB, 1);
            sA += __shfl_xor_sync(0xffffffffu, sA, 2);
            sB += __shfl_xor_sync(0xffffffffu, sB, 2);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        float* srow = a.scores + (long long)r * a.p_stride;
        if (q == 0 && pA < a.p_stride) srow[pA] = cA ? sA : -INFINITY;
        if (q == 1 && pB < a.p_stride) srow[pB] = cB ? sB : -INFINITY;
    }
    if (BAL) {
        // -inf over each row's pools past its visible stages (no unit covers them):
        // CTA b writes the b-th of G equal runs of that tail, thread t rows t, t + 128, ...
        for (int rr = tid; rr < a.rows; rr += 4 * 32) {
            const RowInfo rj = row_info(a, rr);
            if (rj.seq < 0 && blockIdx.x == 0) flag_status(a.status, DSA_STATUS_BAD_TOKEN);
            const long long t0 = (long long)vis_stages(rj, spr) * kStagePools;
            const long long len = (long long)a.p_stride - t0;
            if (len <= 0) continue;
            const long long per = (len + G - 1) / G;
            const long long lo = t0 + (long long)blockIdx.x * per;
            const long long hi = min(lo + per, (long long)a.p_stride);
            float* srow = a.scores + (long long)rr * a.p_stride;
            for (long long p = lo; p < hi; ++p) srow[p] = -INFINITY;
        }
    }
}

template <int IHD, int NT>
int launch_tma(const ScoreArgs& a0, cudaStream_t st) {
    // ring, flags, bad masks, full and empty barriers, the balanced split's unit range
    constexpr int smem =
        kStages * kStagePools * IHD * 2 + kStages * kStagePools + 3 * kStages * 8 + 32;
    ScoreArgs a = a0;
    // 16-byte flag copies need 16-byte aligned runs: whole 16-pool groups per row.
    const bool al = (reinterpret_cast<uintptr_t>(a.pv) & 15u) == 0u;
    a.flags_tma = al && (a.pg.block_table == nullptr
                             ? (a.pg.max_seq_len / a.kpool) % 16 == 0
                             : (a.pg.block_size / a.kpool) % 16 == 0);
    const bool bal = a.pg.block_table != nullptr && a.rows <= kBalRows;
    auto kernel = bal ? score_tma_kernel<IHD, NT, true> : score_tma_kernel<IHD, NT, false>;
    int rc = set_max_smem((const void*)kernel, smem);
    if (rc) return rc;
    const int spr = (a.p_stride + kStagePools - 1) / kStagePools;
    const long long U = (long long)a.rows * spr;
    const long long slots = (long long)sm_count() * kCtasPerSm;
    const int G = (int)(U < slots ? U : slots);
    cudaError_t e = launch_pdl(kernel, dim3(G), dim3(kTmaThreads), smem, st, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "dsa_score launch");
    return DSA_OK;
}

template <int IHD, int NT>
int launch(const ScoreArgs& a0, cudaStream_t st) {
    ScoreArgs a = a0;
    const int ntiles = (a.p_stride + 15) / 16;
    // Enough warps to cover the GPU a few times over; at least 2 tiles per warp.
    const long long want_warps = (long long)sm_count() * 48;
    long long per = ((long long)ntiles * a.rows + want_warps - 1) / want_warps;
    if (per < 2) per = 2;
    if (per > 64) per = 64;
    a.tiles_per_warp = (int)((per + 1) & ~1LL);
    const long long warps_per_row = (ntiles + a.tiles_per_warp - 1) / a.tiles_per_warp;
    dim3 grid((unsigned)((warps_per_row + kWarps - 1) / kWarps), a.rows);
    if (grid.y > 65535u) return fail(DSA_ERR_UNSUPPORTED, "dsa_score: rows %d > 65535", a.rows);
    cudaError_t e = launch_pdl(score_kernel<IHD, NT>, grid, dim3(kWarps * 32), 0, st, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "dsa_score launch");
    return DSA_OK;
}

template <int IHD>
int dispatch_heads(const ScoreArgs& a, cudaStream_t st) {
    const int nt = (a.heads + 7) / 8;
    // Paged caches need whole 16-byte runs per block (always true for kpool | block).
    switch (nt) {
        case 1: return launch_tma<IHD, 1>(a, st);
        case 2: return launch_tma<IHD, 2>(a, st);
        case 3:
        case 4: return launch_tma<IHD, 4>(a, st);
        default: return launch<IHD, 8>(a, st);
    }
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" int dsa_score(const dsa_bf16* qidx, const float* w, int rows, int index_heads,
                         int ihd, const int32_t* row_seq, const int32_t* row_ctx,
                         const dsa_bf16* kpool, const uint8_t* pool_valid, const dsa_paging* pg,
                         int first_key, int kpool_size, float scale, float* scores,
                         int p_stride, int32_t* status, void* stream) {
    if (rows < 0 || p_stride < 0 || first_key < 0)
        return fail(DSA_ERR_INVALID_ARG, "dsa_score: rows %d, p_stride %d, first_key %d", rows,
                    p_stride, first_key);
    if (kpool_size < 1 || kpool_size > DSA_MAX_KPOOL)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_score: kpool %d outside [1, %d]", kpool_size,
                    DSA_MAX_KPOOL);
    if (ihd != 64 && ihd != 128)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_score: index_head_dim %d not in {64, 128}", ihd);
    if (index_heads < 1 || index_heads > 64)
        return fail(DSA_ERR_UNSUPPORTED, "dsa_score: index_heads %d outside [1, 64]", index_heads);
    Paging P;
    int rc = check_paging(pg, kpool_size, &P);
    if (rc) return rc;
    if (rows == 0 || p_stride == 0) return DSA_OK;
    if (!qidx || !w || !kpool || !pool_valid || !scores)
        return fail(DSA_ERR_INVALID_ARG, "dsa_score: NULL tensor");
    if ((((uintptr_t)qidx) | ((uintptr_t)kpool)) & 15)
        return fail(DSA_ERR_INVALID_ARG, "dsa_score: qidx and kpool must be 16-byte aligned");
    ScoreArgs a;
    a.qidx = qidx;
    a.w = w;
    a.row_seq = row_seq;
    a.row_ctx = row_ctx;
    a.kp = kpool;
    a.pv = pool_valid;
    a.scores = scores;
    a.status = status;
    a.pg = P;
    a.rows = rows;
    a.heads = index_heads;
    a.first_key = first_key;
    a.kpool = kpool_size;
    a.p_stride = p_stride;
    a.tiles_per_warp = 2;
    a.scale = scale;
    cudaStream_t st = (cudaStream_t)stream;
    return ihd == 128 ? dispatch_heads<128>(a, st) : dispatch_heads<64>(a, st);
}
