// The absorbed output projection y = o_absorb . olat (dsa_latent_project, and the last
// step of dsa_sparse_mla_decode).
//
// Page: metrale_model_arch/glm5next_dsa/build.rs, module doc, transform 3 and
// absorb_o: o_proj is multiplied through kv_b_proj's V half at load, so the decode
// kernel's latent output [heads, kv_lora_rank] maps back to hidden through
// o_absorb [hidden, heads * kv_lora_rank].
//
// At decode sizes this is a skinny GEMM: every element of o_absorb (268 MB at
// 4096 x 64 x 512) is used by only the few query rows of the step, so the kernel is
// an HBM stream. It is built so the number of bytes in flight does not depend on
// registers: one producer lane per CTA issues 2-D tensor copies (a 256 x 64 box of
// o_absorb and the matching 256 x 8 box of the queries per stage) into a ring of
// shared-memory stages guarded by mbarriers; four consumer warps turn each stage into
// m16n8k16 MMAs (o_absorb rows on M, query rows on N, f32 accumulation). The grid is
// two CTAs per SM at decode sizes and the (row block, k block) units are split evenly
// over the CTAs in row-block-major order ("stream-K"), so every SM streams the same
// number of bytes;
// a CTA whose range crosses a row block writes one partial per row block, and a
// small reduction adds the partials of each row block in a fixed order.
//
// All waits are bounded (about 1 s); a wait that gives up sets DSA_STATUS_TIMEOUT in
// the status word and the CTA winds down after its own copies have landed.
#include "common.cuh"

namespace dsa {
namespace {

constexpr int KT = 256;               // k per stage (one 512-byte box row of o_absorb)
constexpr int MROWS = 64;             // o_absorb rows per CTA tile: 4 consumer warps x 16
constexpr int kConsumers = 4;
constexpr int kThreads = (kConsumers + 1) * 32;

// CTAs per SM: two for the decode sizes (<= 16 query rows), so that every scheduler
// has two consumer warps; one with the larger query-row tiles.
__host__ __device__ constexpr int ctas_per_sm(int nt) { return nt <= 2 ? 2 : 1; }

template <int NT, bool XF32>
struct Cfg {
    static constexpr int XB = XF32 ? 4 : 2;
    static constexpr int A_BYTES = MROWS * KT * 2;        // one 256 x 64 box
    static constexpr int X_BYTES = 8 * NT * KT * XB;      // one 256 x (8*NT) box
    static constexpr int STAGE = A_BYTES + X_BYTES;       // multiple of 1 KiB
    static constexpr int S_FIT = (200 * 1024) / ctas_per_sm(NT) / STAGE;
    static constexpr int S = S_FIT > 6 ? 6 : (S_FIT < 2 ? 2 : S_FIT);
    static constexpr int SMEM = S * STAGE + 2 * S * 8;
};

struct ProjArgs {
    const uint16_t* A;  // [hidden, K] bf16
    const void* X;      // [R, K] bf16 or f32
    float* ypart;       // [G, J, R, 64]
    int32_t* status;
    long long U;        // units = (hidden / 64) * KB
    int K;
    int KB;             // K / KT
    int R;
    int n0;
    int nrows;
    int J;
};

__host__ __device__ inline long long unit_begin(long long c, long long U, long long G) {
    return c * U / G;
}

template <int NT, bool XF32>
__global__ void __launch_bounds__(kThreads, ctas_per_sm(NT))
    project_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmX,
                   ProjArgs a) {
    using C = Cfg<NT, XF32>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::S * C::STAGE);
    uint64_t* empty = full + C::S;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const long long G = gridDim.x;
    const long long u0 = unit_begin(blockIdx.x, a.U, G);
    const long long u1 = unit_begin(blockIdx.x + 1, a.U, G);

    if (tid == 0) {
        for (int s = 0; s < C::S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumers);
        }
        fence_mbar_init();
    }
    if ((smem_u32(smem) & 127u) != 0u) {  // tensor copies need an aligned destination
        if (tid == 0) flag_status(a.status, DSA_STATUS_TIMEOUT);
        pdl_wait();
        return;
    }
    __syncthreads();

    if (warp == kConsumers) {
        // ---------------- producer warp: one elected lane issues two tensor copies per stage
        const uint32_t bytes = (uint32_t)C::STAGE;  // full boxes (zero fill counts too)
        long long i = 0;
        bool ok = true;
        // o_absorb is not written by the kernels before this one: the first ring's
        // worth of its boxes is requested before waiting for them, so it streams in
        // while the preceding kernel finishes; the X (olat) boxes follow the wait.
        const long long pre = (u1 - u0) < C::S ? (u1 - u0) : C::S;
        if (lane == 0) {
            for (long long j = 0; j < pre; ++j) {
                const long long u = u0 + j;
                mbar_arrive_expect_tx(&full[j], bytes);
                tma_load_2d(smem_u32(smem + j * C::STAGE), &tmA, (int)(u % a.KB) * KT,
                            (int)(u / a.KB) * MROWS, &full[j]);
            }
        }
        pdl_wait();
        if (lane == 0) {
            for (long long j = 0; j < pre; ++j) {
                const long long u = u0 + j;
                tma_load_2d(smem_u32(smem + j * C::STAGE) + C::A_BYTES, &tmX, (int)(u % a.KB) * KT,
                            a.n0, &full[j]);
            }
            i = pre;
            for (long long u = u0 + pre; u < u1; ++u, ++i) {
                const int s = (int)(i % C::S);
                const uint32_t ph = (uint32_t)((i / C::S) & 1);
                if (!mbar_wait(&empty[s], ph ^ 1u)) {
                    ok = false;
                    break;
                }
                const int mb = (int)(u / a.KB);
                const int kb = (int)(u % a.KB);
                mbar_arrive_expect_tx(&full[s], bytes);
                const uint32_t dst = smem_u32(smem + s * C::STAGE);
                tma_load_2d(dst, &tmA, kb * KT, mb * MROWS, &full[s]);
                tma_load_2d(dst + C::A_BYTES, &tmX, kb * KT, a.n0, &full[s]);
            }
        }
        if (lane == 0) {
            if (!ok) flag_status(a.status, DSA_STATUS_TIMEOUT);
            // Let the copies already issued land before the CTA may exit.
            const long long first = i > C::S ? i - C::S : 0;
            for (long long j = first; j < i; ++j)
                if (!mbar_wait(&full[j % C::S], (uint32_t)((j / C::S) & 1))) break;
        }
        return;
    }

    // ---------------- consumer warps: rows 16*warp .. +15 of the 64-row tile
    pdl_wait();
    const int g = lane >> 2, q = lane & 3;
    const int rA = 16 * warp + g;
    float acc[NT][4];
    long long cur_mb = -1;
    const int J = a.J;
    auto flush = [&](long long mb) {
        const int j = (int)(mb - u0 / a.KB);
        float* base = a.ypart + (((long long)blockIdx.x * J + j) * a.R + a.n0) * MROWS;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int n = nt * 8 + 2 * q + jj;
                if (n < a.nrows) {
                    base[(long long)n * MROWS + rA] = acc[nt][jj];
                    base[(long long)n * MROWS + rA + 8] = acc[nt][2 + jj];
                }
            }
    };
    long long i = 0;
    for (long long u = u0; u < u1; ++u, ++i) {
        const int s = (int)(i % C::S);
        const uint32_t ph = (uint32_t)((i / C::S) & 1);
        const long long mb = u / a.KB;
        if (mb != cur_mb) {
            if (cur_mb >= 0) flush(cur_mb);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
            cur_mb = mb;
        }
        if (!mbar_wait(&full[s], ph)) {
            if (lane == 0) flag_status(a.status, DSA_STATUS_TIMEOUT);
            break;
        }
        const uint32_t sa = smem_u32(smem + s * C::STAGE);
        const uint32_t sx = sa + C::A_BYTES;
#pragma unroll
        for (int kc = 0; kc < KT / 128; ++kc) {
            uint4 ra0[4], ra1[4];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int e = kc * 128 + 32 * v + 8 * q;
                ra0[v] = lds16(sa + rA * (KT * 2) + e * 2);
                ra1[v] = lds16(sa + (rA + 8) * (KT * 2) + e * 2);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int n = nt * 8 + g;
                uint4 xv[4];
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int e = kc * 128 + 32 * v + 8 * q;
                    if (XF32) {
                        const uint32_t ad = sx + n * (KT * 4) + e * 4;
                        const uint4 f0 = lds16(ad), f1 = lds16(ad + 16);
                        xv[v].x = pack_bf16x2(__uint_as_float(f0.x), __uint_as_float(f0.y));
                        xv[v].y = pack_bf16x2(__uint_as_float(f0.z), __uint_as_float(f0.w));
                        xv[v].z = pack_bf16x2(__uint_as_float(f1.x), __uint_as_float(f1.y));
                        xv[v].w = pack_bf16x2(__uint_as_float(f1.z), __uint_as_float(f1.w));
                    } else {
                        xv[v] = lds16(sx + n * (KT * 2) + e * 2);
                    }
                }
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    mma_16816(acc[nt], ra0[v].x, ra1[v].x, ra0[v].y, ra1[v].y, xv[v].x, xv[v].y);
                    mma_16816(acc[nt], ra0[v].z, ra1[v].z, ra0[v].w, ra1[v].w, xv[v].z, xv[v].w);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (cur_mb >= 0) flush(cur_mb);
}

// y[r, col] = bf16(sum over the CTAs that covered row block col/64 of their partial),
// the CTAs in ascending order. One thread per 4 columns; the contributing CTAs are
// read four at a time so their loads overlap.
// Where the sums go: f32 into yf [R, hidden] when it is set; else bf16, columns
// below `split` into y [R, split] and the rest into y2 [R, hidden - split] (split is
// hidden when y2 is NULL, and a multiple of 64).
struct ProjOut {
    uint16_t* y;
    float* yf;
    uint16_t* y2;
    int split;
};

__device__ __forceinline__ void store_sum(const ProjOut& o, int r, int hidden, int col, float4 v) {
    if (o.yf) {
        *reinterpret_cast<float4*>(o.yf + (long long)r * hidden + col) = v;
        return;
    }
    uint2 b;
    b.x = pack_bf16x2(v.x, v.y);
    b.y = pack_bf16x2(v.z, v.w);
    if (col < o.split)
        *reinterpret_cast<uint2*>(o.y + (long long)r * o.split + col) = b;
    else
        *reinterpret_cast<uint2*>(o.y2 + (long long)r * (hidden - o.split) + (col - o.split)) = b;
}

__global__ void project_reduce_kernel(const float* __restrict__ ypart, long long U, int KB, int G,
                                      int J, int R, int hidden, ProjOut out) {
    pdl_wait();
    const long long n4 = (long long)R * hidden / 4;
    for (long long i4 = blockIdx.x * (long long)blockDim.x + threadIdx.x; i4 < n4;
         i4 += (long long)gridDim.x * blockDim.x) {
        const long long i = 4 * i4;
        const int r = (int)(i / hidden);
        const int col = (int)(i % hidden);
        const long long mb = col / MROWS;
        const long long lo = mb * KB, hi = lo + KB;
        long long c = lo * G / U;
        while (c > 0 && unit_begin(c, U, G) > lo) --c;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (; c < G; c += 4) {
            float4 v[4];
            bool use[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const long long cc = c + k;
                const long long b0 = unit_begin(cc, U, G), b1 = unit_begin(cc + 1, U, G);
                use[k] = cc < G && b0 < hi && b1 > lo && b1 > b0;
                v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (use[k]) {
                    const int j = (int)(mb - b0 / KB);
                    v[k] = __ldg(reinterpret_cast<const float4*>(
                        ypart + ((cc * J + j) * R + r) * MROWS + (col % MROWS)));
                }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (use[k]) {
                    s.x += v[k].x;
                    s.y += v[k].y;
                    s.z += v[k].z;
                    s.w += v[k].w;
                }
            }
            if (c + 4 >= G || unit_begin(c + 4, U, G) >= hi) break;
        }
        store_sum(out, r, hidden, col, s);
    }
}

// Row-block form of the same sum: one CTA per 64-row block of y and up to 128 of
// its (row, 4-column) outputs. The first warp finds the CTAs whose unit ranges meet
// the block (consecutive, at most 32: checked on the host) and stores their partial
// offsets in shared memory; every thread then sums its output over them in CTA
// order with all its loads issued together (eight at a time).
__global__ void __launch_bounds__(128) project_reduce_rows_kernel(
    const float* __restrict__ ypart, long long U, int KB, int G, int J, int R, int hidden,
    ProjOut out) {
    pdl_wait();
    __shared__ long long soff[32];
    __shared__ int scount;
    const int tid = threadIdx.x;
    const long long mb = blockIdx.x;
    if (tid < 32) {
        const long long lo = mb * KB, hi = lo + KB;
        long long c0 = lo * G / U;
        while (c0 > 0 && unit_begin(c0, U, G) > lo) --c0;
        while (c0 + 1 < G && unit_begin(c0 + 1, U, G) <= lo) ++c0;
        const long long c = c0 + tid;
        bool contrib = false;
        if (c < G) {
            const long long b0 = unit_begin(c, U, G), b1 = unit_begin(c + 1, U, G);
            contrib = b0 < hi && b1 > lo && b1 > b0;
            if (contrib) soff[tid] = ((c * J + (mb - b0 / KB)) * R) * MROWS;
        }
        const int n = __popc(__ballot_sync(0xffffffffu, contrib));
        if (tid == 0) scount = n;
    }
    __syncthreads();
    const int n = scount;
    const int o = blockIdx.y * 128 + tid;
    if (o >= R * (MROWS / 4)) return;
    const int r = o / (MROWS / 4), c4 = o % (MROWS / 4);
    const long long ro = (long long)r * MROWS + 4 * c4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < n; k += 8) {
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = k + i < n ? __ldg(reinterpret_cast<const float4*>(ypart + soff[k + i] + ro))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (k + i < n) {
                acc.x += v[i].x;
                acc.y += v[i].y;
                acc.z += v[i].z;
                acc.w += v[i].w;
            }
        }
    }
    store_sum(out, r, hidden, (int)(mb * MROWS) + 4 * c4, acc);
}

struct ProjPlan {
    long long U;
    int KB, G, J, nt;
    size_t bytes;
};

ProjPlan plan_for(int rows, int K, int hidden, int sms) {
    ProjPlan p;
    const int nr = rows < 64 ? rows : 64;
    p.nt = nr <= 8 ? 1 : nr <= 16 ? 2 : nr <= 32 ? 4 : 8;
    p.KB = K / KT;
    p.U = (long long)(hidden / MROWS) * p.KB;
    const long long slots = (long long)sms * ctas_per_sm(p.nt);
    p.G = (int)(p.U < slots ? p.U : slots);
    if (p.G < 1) p.G = 1;
    const long long per = (p.U + p.G - 1) / p.G;
    p.J = (int)((per + p.KB - 1) / p.KB) + 1;
    p.bytes = (size_t)p.G * p.J * rows * MROWS * sizeof(float);
    return p;
}

template <int NT, bool XF32>
int launch_proj(const ProjArgs& a, int G, cudaStream_t st) {
    using C = Cfg<NT, XF32>;
    int rc = set_max_smem((const void*)project_kernel<NT, XF32>, C::SMEM);
    if (rc) return rc;
    CUtensorMap tmA, tmX;
    rc = make_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.A, (uint64_t)a.K,
                      (uint64_t)(a.U / a.KB) * MROWS, (uint64_t)a.K * 2, KT, MROWS);
    if (rc) return rc;
    rc = make_tmap_2d(&tmX, XF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      a.X, (uint64_t)a.K, (uint64_t)a.R, (uint64_t)a.K * C::XB, KT, 8 * NT);
    if (rc) return rc;
    cudaError_t e = launch_pdl(project_kernel<NT, XF32>, dim3(G), dim3(kThreads), C::SMEM, st,
                               tmA, tmX, a);
    if (e != cudaSuccess) return cuda_fail(e, "projection launch");
    return DSA_OK;
}

template <bool XF32>
int dispatch(const ProjArgs& a, int nt, int G, cudaStream_t st) {
    switch (nt) {
        case 1: return launch_proj<1, XF32>(a, G, st);
        case 2: return launch_proj<2, XF32>(a, G, st);
        case 4: return launch_proj<4, XF32>(a, G, st);
        default: return launch_proj<8, XF32>(a, G, st);
    }
}

}  // namespace

bool project_supported(int K, int hidden) { return hidden > 0 && hidden % MROWS == 0 && K % KT == 0; }

size_t project_workspace_bytes(int rows, int K, int hidden, int sms) {
    // the stream-K partials, or the tensor-core form's bf16 copy of an f32 x
    const size_t part = plan_for(rows, K, hidden, sms).bytes;
    const size_t conv = project_tc_supported(K, hidden) ? project_tc_convert_bytes(rows, K) : 0;
    return part > conv ? part : conv;
}

int project_launch(const void* x, bool x_f32, int rows, int K, const uint16_t* A, int hidden,
                   uint16_t* y, int32_t* status, void* ws, size_t ws_bytes, cudaStream_t st,
                   float* yf, uint16_t* y2, int split) {
    ProjOut out;
    out.y = y;
    out.yf = yf;
    out.y2 = y2;
    out.split = y2 ? split : hidden;
    const int sms = sm_count();
    if (sms <= 0) return fail(DSA_ERR_CUDA, "projection: no CUDA device");
    // The tensor-core form where the shape allows it (128-row tiles of A, K in eight
    // equal shares of 64-column stages); no reduction launch follows it.
    if (project_kernel_choice() != DSA_PROJECT_KERNEL_MMA && project_tc_supported(K, hidden))
        return project_tc_launch(x, x_f32, rows, K, A, hidden, y, status, ws, ws_bytes, st, yf, y2,
                                 split);
    const ProjPlan p = plan_for(rows, K, hidden, sms);
    if (ws_bytes < p.bytes) return fail(DSA_ERR_INVALID_ARG, "projection: workspace too small");
    ProjArgs a;
    a.A = A;
    a.X = x;
    a.ypart = static_cast<float*>(ws);
    a.status = status;
    a.U = p.U;
    a.K = K;
    a.KB = p.KB;
    a.R = rows;
    a.J = p.J;
    for (int n0 = 0; n0 < rows; n0 += 64) {
        a.n0 = n0;
        a.nrows = rows - n0 < 64 ? rows - n0 : 64;
        int rc = x_f32 ? dispatch<true>(a, p.nt, p.G, st) : dispatch<false>(a, p.nt, p.G, st);
        if (rc) return rc;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "projection launch");
    // Most CTAs meeting one row block: the row-block reduce takes up to 32.
    int most = 0;
    for (long long mb = 0; mb < hidden / MROWS; ++mb) {
        const long long lo = mb * p.KB, hi = lo + p.KB;
        long long c = lo * p.G / p.U;
        while (c > 0 && unit_begin(c, p.U, p.G) > lo) --c;
        int cnt = 0;
        for (; c < p.G && unit_begin(c, p.U, p.G) < hi; ++c)
            if (unit_begin(c + 1, p.U, p.G) > lo) ++cnt;
        if (cnt > most) most = cnt;
    }
    if (most <= 32) {
        const long long nmb = hidden / MROWS;
        const unsigned yb = (unsigned)((rows * (MROWS / 4) + 127) / 128);
        e = launch_pdl(project_reduce_rows_kernel, dim3((unsigned)nmb, yb), dim3(128), 0, st,
                       (const float*)ws, p.U, p.KB, p.G, p.J, rows, hidden, out);
    } else {
        const long long n4 = (long long)rows * hidden / 4;
        long long blocks = (n4 + 255) / 256;
        if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
        e = launch_pdl(project_reduce_kernel, dim3((unsigned)blocks), dim3(256), 0, st,
                       (const float*)ws, p.U, p.KB, p.G, p.J, rows, hidden, out);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "projection reduce launch");
    return DSA_OK;
}

}  // namespace dsa

using namespace dsa;

extern "C" int dsa_latent_project_workspace(int rows, int heads, int kv_lora_rank, int hidden,
                                            size_t* bytes) {
    if (!bytes) return fail(DSA_ERR_INVALID_ARG, "dsa_latent_project_workspace: bytes is NULL");
    if (rows < 0 || heads < 1) return fail(DSA_ERR_INVALID_ARG, "dsa_latent_project: rows/heads");
    if (kv_lora_rank != DSA_KV_LORA_RANK)
        return fail(kv_lora_rank == 0 ? DSA_ERR_CONFIG : DSA_ERR_UNSUPPORTED,
                    "dsa_latent_project: kv_lora_rank %d, built for %d", kv_lora_rank,
                    DSA_KV_LORA_RANK);
    if (!project_supported(heads * kv_lora_rank, hidden))
        return fail(DSA_ERR_UNSUPPORTED, "dsa_latent_project: hidden %d must be a multiple of 64",
                    hidden);
    const int sms = sm_count();
    if (sms <= 0) return fail(DSA_ERR_CUDA, "dsa_latent_project_workspace: no CUDA device");
    *bytes = project_workspace_bytes(rows, heads * kv_lora_rank, hidden, sms);
    return DSA_OK;
}

extern "C" int dsa_latent_project(const float* olat, int rows, int heads, int kv_lora_rank,
                                  const dsa_bf16* o_absorb, int hidden, dsa_bf16* y,
                                  int32_t* status, void* workspace, size_t workspace_bytes,
                                  void* stream) {
    if (rows < 0 || heads < 1) return fail(DSA_ERR_INVALID_ARG, "dsa_latent_project: rows/heads");
    if (kv_lora_rank != DSA_KV_LORA_RANK)
        return fail(kv_lora_rank == 0 ? DSA_ERR_CONFIG : DSA_ERR_UNSUPPORTED,
                    "dsa_latent_project: kv_lora_rank %d, built for %d", kv_lora_rank,
                    DSA_KV_LORA_RANK);
    if (!project_supported(heads * kv_lora_rank, hidden))
        return fail(DSA_ERR_UNSUPPORTED, "dsa_latent_project: hidden %d must be a multiple of 64",
                    hidden);
    if (rows == 0) return DSA_OK;
    if (!olat || !o_absorb || !y) return fail(DSA_ERR_INVALID_ARG, "dsa_latent_project: NULL tensor");
    if ((((uintptr_t)olat) | ((uintptr_t)o_absorb) | ((uintptr_t)y) | ((uintptr_t)workspace)) & 15)
        return fail(DSA_ERR_INVALID_ARG, "dsa_latent_project: tensors must be 16-byte aligned");
    return project_launch(olat, true, rows, heads * kv_lora_rank, o_absorb, hidden, y, status,
                          workspace, workspace_bytes, (cudaStream_t)stream);
}
