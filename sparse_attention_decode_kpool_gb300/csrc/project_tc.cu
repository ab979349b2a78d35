// The o_absorb projection on the tensor cores (tcgen05): y = x . A^T with A =
// o_absorb [hidden, K] bf16 and x [rows, K] (the bf16 copy of olat, or olat f32 rounded
// to bf16 first).
//
// Page: metrale_model_arch/glm5next_dsa/build.rs, module doc, transform 3 and
// absorb_o: the decode output [heads, kv_lora_rank] maps back to hidden through
// o_absorb [hidden, heads * kv_lora_rank].
//
// Every element of A is used by the step's few query rows only, so the projection is
// a stream of A (268 MB at 4096 x 64 x 512). Here the tensor core reads A straight
// from shared memory: D^T [128 A rows x N] += A_tile [128 x 64] . X_tile^T, with the
// query rows as the MMA's N (16, 32 or 64; rows past the last are zero) and f32
// accumulators in tensor memory. A CTA streams one 128-row tile of A over a 1/KS share
// of K through a ring of TMA stages (128-byte swizzle; the bf16 x box of the same K
// range rides with each stage; f32 x is rounded to bf16 once, before the kernel). The
// ring is sized so that about 160 KB of A is in flight per SM: that, not the tensor
// core, is what holds the stream at HBM speed. The KS
// CTAs that share a row tile form a thread-block cluster and add their partials
// through distributed shared memory in rank order, so the sums are deterministic and
// no reduction kernel follows.
//
// Roles (four warps): warp 0 (one lane) issues the TMA copies, warp 1 allocates tensor
// memory and (one lane) issues the MMAs; all four warps then read the accumulators
// (one tensor-memory lane each) and
// take part in the cluster's sum. Every mbarrier wait is bounded (about 1 s); a wait
// that gives up sets DSA_STATUS_TIMEOUT, the roles skip their remaining work, and the
// cluster barriers are still passed by every thread.
#include "common.cuh"
#include "tc.cuh"

namespace dsa {
namespace {

constexpr int BM = 128;         // A rows per MMA tile (tensor-memory lanes)
constexpr int BK = 64;          // K per stage: one 128-byte swizzle atom of bf16
constexpr int kThreads = 128;
constexpr uint32_t kABytes = BM * BK * 2;  // 16 KB

// MT 128-row tiles of A per CTA share each stage's x tile (MT = 2 halves the x bytes
// per byte of A, which matters once there are tens of query rows).
constexpr int kMaxStages = 8;
template <int N, int MT, int KS>
struct PL {  // shared-memory layout of one CTA (offsets from a 1024-aligned base)
    static constexpr uint32_t AB = MT * kABytes;                // A boxes of a stage
    static constexpr uint32_t XB = N * BK * 2;                  // bf16 x tile
    static constexpr uint32_t STAGE = AB + XB;                  // multiple of 1 KB
    // Bytes of A in flight are what keep the stream at HBM speed (about 160 KB per
    // SM): two CTAs per SM with 16 query rows, one otherwise.
    static constexpr int CTAS_PER_SM = (MT == 1 && N <= 16) ? 2 : 1;
    static constexpr int S_FIT = (int)(((CTAS_PER_SM == 2 ? 220u : 200u) * 1024u / CTAS_PER_SM) / STAGE);
    static constexpr int S = S_FIT > kMaxStages ? kMaxStages : S_FIT;  // ring stages
    static constexpr uint32_t RED = MT * BM * N * 4;            // the partial, f32 [MT*BM][N]
    static constexpr uint32_t RING = S * STAGE;
    static constexpr uint32_t BODY = RING > RED ? RING : RED;
    static constexpr uint32_t BARS = BODY;                      // mbarriers after the body
    static constexpr uint32_t BYTES = BARS + 8 * (2 * kMaxStages + 1) + 16;
    static constexpr uint32_t DYN = BYTES + 1024;
    static_assert(STAGE % 1024 == 0, "stage alignment");
    static_assert(S >= 2, "ring");
};

// Bounded wait that polls (the pipeline's hand-offs are short; a suspended wait wakes
// up late enough to starve the ring). Gives up after about 2^31 cycles (~1 s), or at
// once when another role already gave up; either way it returns false and the first
// to give up flags DSA_STATUS_TIMEOUT.
__device__ __forceinline__ bool poll_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 1023u) == 0u) {
            if (*abort_flag) return false;
            if (clock64() - t0 > (1ll << 31)) {
                *abort_flag = 1;
                flag_status(status, DSA_STATUS_TIMEOUT);
                return false;
            }
        }
    }
}

// Four f32 at the same offset of cluster CTA `rank`'s shared memory. Volatile (kept
// after the cluster barrier, in order) but without a memory clobber, so the loads of
// all ranks are issued back to back and are in flight together.
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t local_addr, uint32_t rank) {
    uint32_t ra;
    float4 v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(ra) : "r"(local_addr), "r"(rank));
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];\n"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "r"(ra));
    return v;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

struct TcProjArgs {
    int32_t* status;
    uint16_t* y;    // bf16 [R, split] (or [R, hidden] when y2 is NULL)
    float* yf;      // f32 [R, hidden] instead of y, when set
    uint16_t* y2;   // bf16 [R, hidden - split] for columns from `split` on
    int split;
    int hidden;
    int R;          // query rows in x (all chunks)
    int n0;         // first query row of this launch
    int nrows;      // query rows of this launch (<= N)
    int kper;       // K per CTA (a multiple of BK)
    const uint8_t* A;  // o_absorb, for the demotion below
    int demote_rows;   // A rows [0, demote_rows) were staged in L2 at evict_last
    int stall_at;      // >= 0: the copies stop before this stage (DSA_OPT_INJECT_STALL)
};

template <int N, int MT, int KS>
__global__ void __launch_bounds__(kThreads, 1)
    project_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmX,
                      TcProjArgs a) {
    using L = PL<N, MT, KS>;
    constexpr int kKS = KS;
    constexpr int kStages = L::S;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BARS);
    uint64_t* empty = full + kMaxStages;
    uint64_t* done = empty + kMaxStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)(blockIdx.x % kKS);  // the CTA's share of K (its cluster rank)
    const int mt = (int)(blockIdx.x / kKS);    // its MT*128 rows of A
    const int nst = a.kper / BK;
    const int k0 = rank * a.kper;

    // Staged rows of A (see the demotion warp below): how many of this CTA's.
    const int row0 = mt * MT * BM;
    const int nstaged = max(0, min(MT * BM, a.demote_rows - row0));
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, nstaged > 0 ? 2 : 1);  // + the demotion warp
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    constexpr uint32_t kCols = MT * N < 32 ? 32 : MT * N;  // MMA tile i: columns [i N, +N)
    if (warp == 1) tc_alloc(tmem_slot, kCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            const uint32_t bytes = L::STAGE;  // A boxes and the x box (zero fill counts too)
            // A (o_absorb) is not written by the kernels before this one: the first
            // ring's A boxes are requested before waiting for them; x follows the wait.
            // A is read once per call: evict_first, so that the stream does not push
            // out A lines a prefetch staged in L2 before the other CTAs reach them.
            const uint64_t ef = l2_evict_first();
            int pre = nst < kStages ? nst : kStages;
            if (a.stall_at >= 0 && a.stall_at < pre) pre = a.stall_at;
            for (int i = 0; i < pre; ++i) {
                mbar_arrive_expect_tx(full + i, bytes);
#pragma unroll
                for (int t = 0; t < MT; ++t)
                    tma_load_2d_hint(smem_u32(smem + i * L::STAGE + t * kABytes), &tmA,
                                     k0 + i * BK, (mt * MT + t) * BM, full + i, ef);
            }
            pdl_wait();
            for (int i = 0; i < pre; ++i)
                tma_load_2d(smem_u32(smem + i * L::STAGE + L::AB), &tmX, k0 + i * BK, a.n0, full + i);
            int i = pre;
            for (; i < nst; ++i) {
                if (i == a.stall_at) break;  // injected stall: nothing more is copied
                const int s = i % kStages;
                if (!poll_wait(empty + s, (uint32_t)(((i / kStages) & 1) ^ 1), abort_flag,
                                   a.status))
                    break;
                mbar_arrive_expect_tx(full + s, bytes);
                const uint32_t dst = smem_u32(smem + s * L::STAGE);
#pragma unroll
                for (int t = 0; t < MT; ++t)
                    tma_load_2d_hint(dst + t * kABytes, &tmA, k0 + i * BK, (mt * MT + t) * BM,
                                     full + s, ef);
                tma_load_2d(dst + L::AB, &tmX, k0 + i * BK, a.n0, full + s);
            }
            // the copies issued have landed before the CTA may reuse or leave its memory
            const int first = i > kStages ? i - kStages : 0;
            for (int j = first; j < i; ++j)
                if (!poll_wait(full + (j % kStages), (uint32_t)((j / kStages) & 1), abort_flag, a.status))
                    break;
        } else {
            pdl_wait();
        }
    } else if (warp == 1) {
        pdl_wait();
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_bf16(BM, N);
            bool ok = true;
            for (int i = 0; i < nst && ok; ++i) {
                const int s = i % kStages;
                const uint32_t par = (uint32_t)((i / kStages) & 1);
                if (!poll_wait(full + s, par, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + s * L::STAGE);
                const uint32_t sx = sa + L::AB;
#pragma unroll
                for (int t = 0; t < MT; ++t)
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        tc_mma(tmem + t * N, sw128_desc(sa + t * kABytes + 32 * kk),
                               sw128_desc(sx + 32 * kk), IDESC, (i | kk) != 0 ? 1u : 0u);
                tc_commit(empty + s);
            }
            tc_commit(done);  // every MMA issued (all of them, or those before an abort)
        }
    } else if (warp == 2 && nstaged > 0) {
        // ---------------- demotion of staged A lines ----------------
        // Rows of A that dsa_prefetch_l2 staged at evict_last go back to normal L2
        // priority as soon as their box has landed in shared memory: one 128-byte
        // line per row and stage. The warp is the second arrival on each empty
        // barrier, so the ring never runs a phase ahead of it.
        const long long rb = (long long)a.kper * kKS * 2;  // bytes per A row
        for (int i = 0; i < nst; ++i) {
            const int s = i % kStages;
            int ok = 1;
            if (lane == 0) ok = poll_wait(full + s, (uint32_t)((i / kStages) & 1), abort_flag, a.status);
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            const uint8_t* col = a.A + ((long long)k0 + (long long)i * BK) * 2;
            for (int r = lane; r < nstaged; r += 32)
                asm volatile("applypriority.global.L2::evict_normal [%0], 128;" ::"l"(col + (row0 + r) * rb)
                             : "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + s);
        }
        pdl_wait();
    } else {
        pdl_wait();
    }

    // ---------------- the partial: tensor memory -> shared memory [BM][N] ----------------
    __syncwarp();
    int got = 1;
    if (lane == 0) got = poll_wait(done, 0, abort_flag, a.status);
    got = __shfl_sync(0xffffffffu, got, 0);
    __syncthreads();  // every role is done with the ring: it becomes the partial's buffer
    float* red = reinterpret_cast<float*>(smem);
    if (got) {
        tc_fence_after();
        const uint32_t lrow = (uint32_t)(32 * warp) << 16;
#pragma unroll 1
        for (int mtile = 0; mtile < MT; ++mtile) {
            const int t = mtile * BM + threadIdx.x;  // A row of the CTA = tensor-memory lane
            const uint32_t cbase = tmem + lrow + mtile * N;
            if constexpr (N == 16) {
                uint32_t w[16];
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"
                    "%12,%13,%14,%15}, [%16];\n"
                    : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                      "=r"(w[6]), "=r"(w[7]), "=r"(w[8]), "=r"(w[9]), "=r"(w[10]), "=r"(w[11]),
                      "=r"(w[12]), "=r"(w[13]), "=r"(w[14]), "=r"(w[15])
                    : "r"(cbase));
                asm volatile("tcgen05.wait::ld.sync.aligned;\n"
                             : "+r"(w[0]), "+r"(w[1]), "+r"(w[2]), "+r"(w[3]), "+r"(w[4]),
                               "+r"(w[5]), "+r"(w[6]), "+r"(w[7]), "+r"(w[8]), "+r"(w[9]),
                               "+r"(w[10]), "+r"(w[11]), "+r"(w[12]), "+r"(w[13]), "+r"(w[14]),
                               "+r"(w[15])
                             :
                             : "memory");
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    *reinterpret_cast<float4*>(red + t * N + j) =
                        make_float4(__uint_as_float(w[j]), __uint_as_float(w[j + 1]),
                                    __uint_as_float(w[j + 2]), __uint_as_float(w[j + 3]));
            } else {
#pragma unroll 1
                for (int c0 = 0; c0 < N; c0 += 32) {
                    uint32_t v[32];
                    tc_ld32(v, cbase + c0);
                    tc_wait_ld(v);
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(red + t * N + c0 + j) =
                            make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                        __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tc_dealloc(tmem, kCols);
    }

    // ---------------- the cluster's sum: this CTA adds rows [kRows rank, +kRows) ----------
    cluster_sync_all();  // every CTA's partial is in its shared memory
    constexpr int kRows = MT * BM / kKS;
    const uint32_t red_s = smem_u32(red);
    // thread o: A row t (consecutive threads, consecutive rows), query rows 4 q4 .. +3
    for (int o = threadIdx.x; o < kRows * (N / 4); o += kThreads) {
        const int q4 = o / kRows, tl = o % kRows;
        const int t = rank * kRows + tl;
        const uint32_t off = red_s + (uint32_t)(t * N + 4 * q4) * 4u;
        float4 v[kKS];
#pragma unroll
        for (int k = 0; k < kKS; ++k) v[k] = ld_cluster_f32x4(off, (uint32_t)k);
        float4 sum = v[0];
#pragma unroll
        for (int k = 1; k < kKS; ++k) {  // rank order: deterministic
            sum.x += v[k].x;
            sum.y += v[k].y;
            sum.z += v[k].z;
            sum.w += v[k].w;
        }
        if (!got) continue;
        const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
        const int col = mt * MT * BM + t;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = 4 * q4 + j;
            if (n >= a.nrows) break;
            const int r = a.n0 + n;
            if (a.yf) {
                a.yf[(long long)r * a.hidden + col] = sv[j];
            } else {
                const uint16_t b = __bfloat16_as_ushort(__float2bfloat16_rn(sv[j]));
                if (col < a.split)
                    a.y[(long long)r * a.split + col] = b;
                else
                    a.y2[(long long)r * (a.hidden - a.split) + (col - a.split)] = b;
            }
        }
    }
    cluster_sync_all();  // no CTA leaves while a peer may still read its partial
}

template <int N, int MT, int KS>
int launch_tc(const uint16_t* x, int R, int K, const uint16_t* A, int hidden, const TcProjArgs& a0,
              cudaStream_t st) {
    using L = PL<N, MT, KS>;
    constexpr int kKS = KS;
    TcProjArgs a = a0;
    a.kper = K / KS;
    if (a.stall_at >= 0) a.stall_at = a.kper / BK - 1;  // before the last stage
    int rc = set_max_smem((const void*)project_tc_kernel<N, MT, KS>, (int)L::DYN);
    if (rc) return rc;
    CUtensorMap tmA, tmX;
    rc = make_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, (uint64_t)K, (uint64_t)hidden,
                      (uint64_t)K * 2, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    rc = make_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)K, (uint64_t)R,
                      (uint64_t)K * 2, BK, N, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((hidden / (MT * BM)) * kKS));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::DYN;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kKS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, project_tc_kernel<N, MT, KS>, tmA, tmX, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "projection (tensor cores) launch");
    return DSA_OK;
}

// K shares per 128-row tile: the most (up to `most`) that keep the grid within one wave
// of `slots` CTAs and give each share at least eight 64-wide stages.
int pick_ks(int tiles, int K, int slots, int most) {
    int ks = most;
    while (ks > 1 && ((long long)tiles * ks > slots || K / ks < 8 * BK || K % (ks * BK) != 0))
        ks >>= 1;
    return ks;
}

int dispatch_tc(const uint16_t* x, int R, int K, const uint16_t* A, int hidden, const TcProjArgs& a,
                int n, cudaStream_t st) {
    // Up to 16 query rows: two CTAs per SM, clusters of up to 8 K shares. More rows: a
    // larger ring per CTA (one per SM) and clusters of up to 4 K shares, so that the
    // grid of 128-row tiles stays one wave of clusters (eight-CTA clusters of one-CTA
    // SMs do not all fit). Many tiles (a tall weight with a short K, such as the
    // front-end's q projection) take fewer shares: each CTA then streams a longer run.
    const int tiles = hidden / BM;
    const int sms = sm_count() > 0 ? sm_count() : 148;
    if (n <= 16) {
        switch (pick_ks(tiles, K, 2 * sms, 8)) {
            case 8: return launch_tc<16, 1, 8>(x, R, K, A, hidden, a, st);
            case 4: return launch_tc<16, 1, 4>(x, R, K, A, hidden, a, st);
            case 2: return launch_tc<16, 1, 2>(x, R, K, A, hidden, a, st);
            default: return launch_tc<16, 1, 1>(x, R, K, A, hidden, a, st);
        }
    }
    const int ks = pick_ks(tiles, K, sms, 4);
    if (n <= 32) {
        switch (ks) {
            case 4: return launch_tc<32, 1, 4>(x, R, K, A, hidden, a, st);
            case 2: return launch_tc<32, 1, 2>(x, R, K, A, hidden, a, st);
            default: return launch_tc<32, 1, 1>(x, R, K, A, hidden, a, st);
        }
    }
    switch (ks) {
        case 4: return launch_tc<64, 1, 4>(x, R, K, A, hidden, a, st);
        case 2: return launch_tc<64, 1, 2>(x, R, K, A, hidden, a, st);
        default: return launch_tc<64, 1, 1>(x, R, K, A, hidden, a, st);
    }
}

// x f32 -> bf16 (round to nearest even), for the projection's bf16 x tiles.
__global__ void to_bf16_kernel(const float* __restrict__ x, long long n4, uint16_t* __restrict__ xb) {
    pdl_wait();
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
         i += (long long)gridDim.x * blockDim.x) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(x) + i);
        uint2 o;
        o.x = pack_bf16x2(v.x, v.y);
        o.y = pack_bf16x2(v.z, v.w);
        reinterpret_cast<uint2*>(xb)[i] = o;
    }
}

}  // namespace

bool project_tc_supported(int K, int hidden) {
    return hidden > 0 && hidden % BM == 0 && K > 0 && K % (8 * BK) == 0;
}

size_t project_tc_convert_bytes(int rows, int K) { return (size_t)rows * K * 2; }

int project_tc_launch(const void* x, bool x_f32, int rows, int K, const uint16_t* A, int hidden,
                      uint16_t* y, int32_t* status, void* ws, size_t ws_bytes, cudaStream_t st,
                      float* yf, uint16_t* y2, int split) {
    if (!project_tc_supported(K, hidden))
        return fail(DSA_ERR_UNSUPPORTED, "projection (tensor cores): K %d, hidden %d", K, hidden);
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    if (x_f32) {
        // f32 x: one rounding pass into the workspace first
        if (!ws || ws_bytes < project_tc_convert_bytes(rows, K))
            return fail(DSA_ERR_INVALID_ARG, "projection: workspace too small for the bf16 copy of x");
        const long long n4 = (long long)rows * K / 4;
        long long blocks = (n4 + 255) / 256;
        const int sms = sm_count();
        if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
        cudaError_t e = launch_pdl(to_bf16_kernel, dim3((unsigned)blocks), dim3(256), 0, st,
                                   static_cast<const float*>(x), n4, static_cast<uint16_t*>(ws));
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "projection: x rounding launch");
        xb = static_cast<const uint16_t*>(ws);
    }
    TcProjArgs a;
    a.status = status;
    a.y = y;
    a.yf = yf;
    a.y2 = y2;
    a.split = y2 ? split : hidden;
    a.hidden = hidden;
    a.R = rows;
    a.kper = 0;  // set per launch form
    a.A = reinterpret_cast<const uint8_t*>(A);
    // o_absorb rows staged in L2 by dsa_prefetch_l2 (the last launch demotes them)
    const size_t row_bytes = (size_t)K * 2;
    // (applypriority acts on whole 128-byte lines: only for a line-aligned o_absorb)
    const size_t staged = (reinterpret_cast<uintptr_t>(A) & 127u)
                              ? 0
                              : l2_staged_overlap(A, (size_t)hidden * row_bytes);
    const int staged_rows = (int)((staged + row_bytes - 1) / row_bytes);
    const bool stall = take_inject_stall() != 0;
    for (int n0 = 0; n0 < rows; n0 += 64) {
        a.stall_at = stall && n0 == 0 ? 0 : -1;
        a.n0 = n0;
        a.nrows = rows - n0 < 64 ? rows - n0 : 64;
        a.demote_rows = n0 + 64 >= rows ? staged_rows : 0;
        int rc = dispatch_tc(xb, rows, K, A, hidden, a, a.nrows, st);
        if (rc) return rc;
    }
    return DSA_OK;
}

}  // namespace dsa
