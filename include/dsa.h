/*
 * dsa.h -- C ABI of the GB300 (sm_103a) DSA decode library, libdsa.so.
 *
 * One DeepSeek-Sparse-Attention decode step of a GLM-5.3-style layer, in the
 * order of the pipeline in metrale_model_arch/glm5next_dsa/mod.rs, "Shape of the
 * pipeline":
 *
 *   k, gate, valid, ape -> dsa_compress          -> pooled keys / pool flags
 *                        -> dsa_score             -> [rows, p_stride] f32 scores
 *                        -> dsa_select            -> [rows, select_k] pool ids
 *                        -> dsa_expand            -> [rows, out_width] token ids
 *                        -> dsa_sparse_mla_decode -> [rows, hidden] bf16 output
 *
 * Conventions shared by every entry point:
 *
 *  - Pointers to tensors are DEVICE pointers owned by the caller; the library
 *    never frees or retains them past the call's stream work. Pointers to
 *    dsa_paging structs and to size_t results are HOST pointers, read during
 *    the call only.
 *  - Tensors are dense row-major. bf16 values are passed as their 16-bit
 *    patterns (dsa_bf16); the library rounds every bf16 it stores to nearest,
 *    ties to even.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Every call only
 *    enqueues work on it: no host synchronisation, no allocation. Calls that
 *    need scratch take a caller-owned device `workspace` of at least the size
 *    the matching *_workspace query reports.
 *  - Return value: DSA_OK, or an error code with a message from
 *    dsa_last_error(). Argument errors are found on the host before anything
 *    is enqueued; nothing is launched then.
 *  - `status` (nullable): a device int32 word the kernels OR DSA_STATUS_* bits
 *    into when they meet an out-of-range token id or block-table entry. Such
 *    entries are skipped (treated as absent); kernels never trap. The caller
 *    clears the word and reads it after synchronising.
 *  - Device-side values the host cannot see (sequence lengths, block-table
 *    entries, token ids) are range-checked on the device against the sizes
 *    given here.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_OK 0
#define DSA_ERR_INVALID_ARG 1 /* null, negative, inconsistent or mis-sized argument */
#define DSA_ERR_UNSUPPORTED 2 /* a size outside what the kernels are built for     */
#define DSA_ERR_CONFIG 3      /* a layer-geometry rule of the pages is violated     */
#define DSA_ERR_CUDA 4        /* a CUDA runtime error while enqueueing              */

#define DSA_STATUS_BAD_TOKEN 1 /* token id < -1, or >= its sequence's length  */
#define DSA_STATUS_BAD_BLOCK 2 /* block-table entry outside [0, num_blocks)    */
#define DSA_STATUS_TIMEOUT 4   /* a pipeline wait gave up after ~1 s (results invalid) */
#define DSA_STATUS_CACHE_FULL 8 /* dsa_indexer_store: a sequence's cache was full (not stored) */

#define DSA_KV_LORA_RANK 512 /* latent width the attention kernels are built for */
#define DSA_MAX_KPOOL 16     /* most slots per pool dsa_compress handles         */

typedef uint16_t dsa_bf16;

/*
 * Where a sequence's tokens (and pooled keys) live.
 *
 * Contiguous (block_table == NULL): a token cache is [batch, max_seq_len, D]
 * and a pooled-key cache is [batch, max_seq_len / kpool, D]; pool p of
 * sequence b is row b * (max_seq_len / kpool) + p.
 *
 * Paged (block_table != NULL): a token cache is [num_blocks, block_size, D];
 * token t of sequence b is slot t % block_size of physical block
 * block_table[b * max_blocks + t / block_size]. The pooled-key cache is
 * [num_blocks, block_size / kpool, D] through the same table: pool p of
 * sequence b is slot p % (block_size / kpool) of block
 * block_table[b * max_blocks + p / (block_size / kpool)].
 *
 * seq_lens[b] (device) is the number of tokens sequence b holds; it must not
 * exceed max_seq_len (contiguous) or max_blocks * block_size (paged).
 * max_seq_len is a host-side upper bound used to size grids.
 */
typedef struct dsa_paging {
    int32_t batch;
    int32_t max_seq_len;
    const int32_t* seq_lens;    /* device [batch]                          */
    const int32_t* block_table; /* device [batch, max_blocks], or NULL     */
    int32_t max_blocks;
    int32_t block_size;
    int64_t num_blocks;
} dsa_paging;

/* Message for the last error returned on this host thread ("" if none). */
const char* dsa_last_error(void);

/* ABI version of this header (bumped on any signature change). */
int dsa_abi_version(void);
#define DSA_ABI_VERSION 8

/*
 * Process-wide launch options (no counterpart on the pages: they choose between
 * equivalent launch forms, for profiling and for tests that pin one kernel). They
 * are plain values read at each call; the library reads no environment variable.
 * Set them before enqueueing work that depends on them, and keep
 * DSA_OPT_MLA_KERNEL fixed between a *_workspace query and the calls that use
 * that workspace (the kernel choice sizes the workspace).
 *
 *   DSA_OPT_PDL         1 (default): every kernel is launched as a programmatic
 *                       dependent of the work before it on the stream (it still
 *                       waits for that work before reading its outputs);
 *                       0: ordinary stream-ordered launches.
 *   DSA_OPT_MLA_KERNEL  which kernel the sparse latent attention uses:
 *                       DSA_MLA_KERNEL_AUTO (default, chosen by size),
 *                       DSA_MLA_KERNEL_TCGEN05 (the persistent tensor-core split
 *                       kernel wherever it supports the shape),
 *                       DSA_MLA_KERNEL_MMA (the mma.sync split kernel),
 *                       DSA_MLA_KERNEL_CLUSTER (the tensor-core decode kernel:
 *                       a chunk of 128 selected tokens per CTA; a row's CTAs merge
 *                       their partials inside a thread-block cluster when they are
 *                       at most 8, else the combine kernel merges them).
 *   DSA_OPT_SELECT_KERNEL  how rows split over a thread-block cluster are selected:
 *                       DSA_SELECT_KERNEL_MERGE (default: each CTA's slice
 *                       candidates merged in CTA 0; a slice first sends its top
 *                       2 ceil(k / C) and all slices send their full top-k only
 *                       when those cannot hold the row's top-k) or
 *                       DSA_SELECT_KERNEL_RADIX (the row's
 *                       k-th key found digit by digit from histograms shared across
 *                       the cluster). Both give the same ids.
 *   DSA_OPT_PROJECT_KERNEL  the o_absorb projection (and the front-end GEMMs):
 *                       DSA_PROJECT_KERNEL_AUTO (default: the tensor-core form
 *                       wherever the shape allows it, i.e. hidden a multiple of 128
 *                       and K of 512), DSA_PROJECT_KERNEL_TCGEN05 (the same),
 *                       DSA_PROJECT_KERNEL_MMA (the mma.sync stream-K form with
 *                       its partial-sum reduction).
 *   DSA_OPT_INJECT_STALL  fault injection for tests of the bounded pipeline waits
 *                       (default 0, off). 1 arms it for the next launch of the
 *                       tensor-core projection: that launch's copy warp stops before
 *                       its last stage, so the MMA warp's bounded wait gives up after
 *                       about 1 s; the launch ORs DSA_STATUS_TIMEOUT into its status
 *                       word, winds down (the copies it issued have landed, its
 *                       tensor memory is freed, every cluster barrier is passed) and
 *                       leaves y invalid. The launch that takes it resets it to 0.
 *
 * dsa_set_option returns DSA_ERR_INVALID_ARG for an unknown option or value;
 * dsa_get_option returns the current value, or -1 for an unknown option.
 */
#define DSA_OPT_PDL 0
#define DSA_OPT_MLA_KERNEL 1
#define DSA_MLA_KERNEL_AUTO 0
#define DSA_MLA_KERNEL_TCGEN05 1
#define DSA_MLA_KERNEL_MMA 2
#define DSA_MLA_KERNEL_CLUSTER 3
#define DSA_OPT_SELECT_KERNEL 2
#define DSA_SELECT_KERNEL_MERGE 0
#define DSA_SELECT_KERNEL_RADIX 1
#define DSA_OPT_PROJECT_KERNEL 3
#define DSA_PROJECT_KERNEL_AUTO 0
#define DSA_PROJECT_KERNEL_TCGEN05 1
#define DSA_PROJECT_KERNEL_MMA 2
#define DSA_OPT_INJECT_STALL 4
int dsa_set_option(int option, int value);
int dsa_get_option(int option);

/*
 * dsa_prefetch_l2 -- ask the memory system to bring the device range
 * [ptr, ptr + bytes) into L2 (bulk prefetch, 16 KB per request; the tail below 16
 * bytes is ignored). Meant for read-only data needed soon, such as o_absorb, issued
 * on a second stream or graph branch beside latency-bound stages so that the
 * projection finds part of its weights in L2. A hint: nothing is written, nothing
 * waits for it, and results never depend on it. ptr must be 16-byte aligned;
 * bytes == 0 is a no-op. The range should stay well below the L2's 126 MB.
 */
int dsa_prefetch_l2(const void* ptr, size_t bytes, void* stream);

/*
 * Layer-geometry rules (mod.rs, Glm5NextDsaConfig::validate): index_kpool and
 * index_topk positive (DSA_ERR_CONFIG), index_topk a multiple of index_kpool
 * (DSA_ERR_CONFIG), index_kpool <= DSA_MAX_KPOOL (DSA_ERR_UNSUPPORTED; the
 * pages' 8-slot register bound is replaced by ours, refused rather than
 * truncated), kv_lora_rank == DSA_KV_LORA_RANK (0: DSA_ERR_CONFIG; other:
 * DSA_ERR_UNSUPPORTED), local_heads > 0 (DSA_ERR_CONFIG).
 */
int dsa_validate_config(int index_kpool, int index_topk, int kv_lora_rank, int local_heads);

/* Pools selected per row: min(index_topk / kpool, n_pools)
 * (mod.rs, Glm5NextDsaConfig::select_k). Returns -1 on invalid input. */
int dsa_select_k(int index_topk, int kpool, int n_pools);

/*
 * dsa_compress -- indexer k_norm fused with dsa_kpool_compress.
 * mod.rs, "Checkpoint and kernel facts": k_norm is a LayerNorm with a bias; the
 * pool softmax runs over the slot axis, per channel; pooling starts at
 * first_key; a pool counts only if all its slots are valid, so a trailing
 * partial pool is not a pool. build.rs transform 4: ape is f32.
 *
 *   kn[t, c]       = bf16((k[t,c] - mean_t) / sqrt(var_t + eps) * ln_w[c] + ln_b[c])
 *   logit_s[c]     = gate[t_s, c] + ape[s, c],   t_s = first_key + p*kpool + s
 *   kpool_out[p,c] = bf16(sum_s softmax_s(logit[c]) * kn[t_s, c])
 *   pool_valid[p]  = all_s token_valid[t_s] != 0   (invalid pools: zero keys)
 *   pool_idx[p,s]  = t_s                            (optional)
 *
 * k_raw, gate: token caches of width ihd (bf16); token_valid: token cache of
 * width 1 (u8); ape [kpool, ihd] f32; ln_w, ln_b [ihd] bf16. Outputs are
 * pooled-key caches (see dsa_paging): kpool_out width ihd (bf16), pool_valid
 * width 1 (u8), pool_idx width kpool (i32, nullable). For each sequence b the
 * pools p < floor((seq_lens[b] - first_key) / kpool) are written; other rows
 * are not touched.
 * Limits: ihd in {64, 128}; 1 <= kpool <= DSA_MAX_KPOOL; first_key >= 0.
 * Paged: block_size % kpool == 0 and first_key % kpool == 0.
 */
int dsa_compress(const dsa_bf16* k_raw, const dsa_bf16* gate, const uint8_t* token_valid,
                 const float* ape, const dsa_bf16* ln_w, const dsa_bf16* ln_b, float eps,
                 const dsa_paging* pg, int first_key, int kpool, int ihd,
                 dsa_bf16* kpool_out, uint8_t* pool_valid, int32_t* pool_idx,
                 int32_t* status, void* stream);

/*
 * dsa_compress_append -- dsa_compress for the pools that the last new_tokens
 * tokens of each sequence completed (the decode-time form: only the newly whole
 * pool is pooled). With L = seq_lens[b] read on the device and
 * whole(n) = floor((n - first_key) / kpool) for n > first_key, else 0, the pools
 * p in [whole(max(L - new_tokens, 0)), whole(L)) are written exactly as
 * dsa_compress writes them (bit-identical); every other row is not touched.
 * new_tokens >= 1 is a host constant, so a captured graph stays valid as the
 * lengths grow. Arguments, limits and errors otherwise as dsa_compress.
 */
int dsa_compress_append(const dsa_bf16* k_raw, const dsa_bf16* gate, const uint8_t* token_valid,
                        const float* ape, const dsa_bf16* ln_w, const dsa_bf16* ln_b, float eps,
                        const dsa_paging* pg, int first_key, int kpool, int ihd, int new_tokens,
                        dsa_bf16* kpool_out, uint8_t* pool_valid, int32_t* pool_idx,
                        int32_t* status, void* stream);

/*
 * dsa_indexer_store -- the decode-time append (mod.rs, Glm5NextDsaKernels,
 * indexer_store): the staged row lands at the position the device holds for the
 * sequence and is flagged valid. For each sequence b, with t = seq_lens[b] read
 * on the device:
 *
 *   k_raw[b, t, :] = k_new[b, :]     gate[b, t, :] = gate_new[b, :]
 *   token_valid[b, t] = 1            ckv[b, t, :] = ckv_new[b, :]  (when given)
 *   seq_lens[b] = t + 1
 *
 * through pg's layout (for a paged cache the block table must already map block
 * t / block_size). The latent row (ckv, ckv_new) is optional and has no
 * counterpart on the pages: it is the layer's own cache append for the same
 * token, done in the same launch. t at or past the capacity (max_seq_len, or
 * max_blocks * block_size when paged) sets DSA_STATUS_CACHE_FULL and stores
 * nothing; a bad block-table entry sets DSA_STATUS_BAD_BLOCK and stores nothing;
 * in both cases seq_lens[b] is left as it was.
 *
 * k_new, gate_new [batch, ihd] bf16; ckv_new [batch, kv_lora_rank] bf16
 * (nullable, with ckv); seq_lens must be pg->seq_lens, writable. k_raw, gate,
 * ckv: token caches (bf16) of widths ihd, ihd, kv_lora_rank; token_valid: token
 * cache of width 1 (u8). No host value depends on the lengths, so a captured
 * graph appends one token per sequence per replay.
 * Limits: ihd in {64, 128}; kv_lora_rank % 8 == 0; rows 16-byte aligned.
 */
int dsa_indexer_store(const dsa_bf16* k_new, const dsa_bf16* gate_new, const dsa_bf16* ckv_new,
                      int ihd, int kv_lora_rank, const dsa_paging* pg, int32_t* seq_lens,
                      dsa_bf16* k_raw, dsa_bf16* gate, uint8_t* token_valid, dsa_bf16* ckv,
                      int32_t* status, void* stream);

/*
 * dsa_write_geom -- mod.rs, Glm5NextDsaKernels, write_geom: the selector's
 * per-row geometry is recomputed on the device from the current lengths, which
 * keeps one captured graph valid as the sequences grow. A decode row sees its
 * whole sequence:
 *
 *   row_ctx[r] = seq_lens[row_seq[r]]   (row_seq NULL: seq_lens[r])
 *
 * The other kernels take their candidate pools, tails and bounds from row_ctx
 * (or seq_lens) on the device. A row_seq entry outside [0, batch) gives
 * row_ctx[r] = 0 and sets DSA_STATUS_BAD_TOKEN.
 * seq_lens [batch] i32, row_seq [rows] i32, row_ctx [rows] i32 (device).
 */
int dsa_write_geom(const int32_t* seq_lens, int batch, const int32_t* row_seq, int rows,
                   int32_t* row_ctx, int32_t* status, void* stream);

/*
 * dsa_decode_append -- dsa_indexer_store, then dsa_write_geom (row_seq NULL,
 * rows = batch: one decode row per sequence), then dsa_compress_append with
 * new_tokens = 1, in one launch: every output (caches, lengths, row_ctx, pooled
 * keys, flags, pool_idx, status bits) is bit-identical to the three calls in
 * sequence. One CTA per sequence stores the staged rows, advances the length and
 * writes row_ctx[b]; when the stored token completes a pool, one warp of the same
 * CTA pools it. No counterpart on the pages beyond the steps it joins.
 *
 * Arguments as in the three calls; row_ctx [batch] i32 (device, nullable).
 * Limits: those of dsa_indexer_store and dsa_compress.
 */
int dsa_decode_append(const dsa_bf16* k_new, const dsa_bf16* gate_new, const dsa_bf16* ckv_new,
                      const float* ape, const dsa_bf16* ln_w, const dsa_bf16* ln_b, float eps,
                      const dsa_paging* pg, int32_t* seq_lens, int first_key, int kpool, int ihd,
                      int kv_lora_rank, dsa_bf16* k_raw, dsa_bf16* gate, uint8_t* token_valid,
                      dsa_bf16* ckv, dsa_bf16* kpool_out, uint8_t* pool_valid, int32_t* pool_idx,
                      int32_t* row_ctx, int32_t* status, void* stream);

/*
 * dsa_decode_append_fp8 -- dsa_decode_append for a layer with the FP8 latent cache
 * (see dsa_quantize_latent): the staged latent row ckv_new is also encoded into
 * ckv_codes [.., kv_lora_rank] u8 and ckv_scales [.., kv_lora_rank / 128] f32 at the
 * token's cache row, with the same codec, so the bytes equal what
 * dsa_quantize_latent makes of that row. ckv (the bf16 latent cache) is nullable
 * here; ckv_new is required. Limits: those of dsa_decode_append, kv_lora_rank % 128
 * == 0, FP8 caches 16-byte aligned. No counterpart on the pages (their FP8 kernel's
 * format is not given; this library's is stated at dsa_quantize_latent).
 */
int dsa_decode_append_fp8(const dsa_bf16* k_new, const dsa_bf16* gate_new,
                          const dsa_bf16* ckv_new, const float* ape, const dsa_bf16* ln_w,
                          const dsa_bf16* ln_b, float eps, const dsa_paging* pg, int32_t* seq_lens,
                          int first_key, int kpool, int ihd, int kv_lora_rank, dsa_bf16* k_raw,
                          dsa_bf16* gate, uint8_t* token_valid, dsa_bf16* ckv, uint8_t* ckv_codes,
                          float* ckv_scales, dsa_bf16* kpool_out, uint8_t* pool_valid,
                          int32_t* pool_idx, int32_t* row_ctx, int32_t* status, void* stream);

/*
 * dsa_score -- dsa_index_scores (tp.rs, "Why the indexer is replicated": a sum
 * over the indexer heads of weighted, rectified, scaled dot products; build.rs
 * transform 2: w arrives already multiplied by index_heads^-0.5).
 *
 *   scores[r, p] = sum_h w[r,h] * relu(scale * <qidx[r,h,:], kpool[p,:]>)
 *
 * when pool p of row r's sequence is a candidate: pool_valid[p] != 0 and its
 * last slot first_key + (p+1)*kpool - 1 < row_ctx[r]; every other entry of the
 * p_stride-wide row, up to p_stride, is -inf.
 *
 * qidx [rows, index_heads, ihd] bf16; w [rows, index_heads] f32; row_seq [rows]
 * i32 (device, nullable: row r -> sequence r); row_ctx [rows] i32 (device,
 * nullable: seq_lens[row_seq[r]]); kpool / pool_valid: pooled-key caches laid
 * out as pg says; scores [rows, p_stride] f32.
 * Limits: ihd in {64, 128}; 1 <= index_heads <= 64; p_stride >= 0.
 */
int dsa_score(const dsa_bf16* qidx, const float* w, int rows, int index_heads, int ihd,
              const int32_t* row_seq, const int32_t* row_ctx,
              const dsa_bf16* kpool, const uint8_t* pool_valid, const dsa_paging* pg,
              int first_key, int kpool_size, float scale,
              float* scores, int p_stride, int32_t* status, void* stream);

/*
 * dsa_score_prefill -- dsa_index_scores for a chunk of query rows of ONE sequence
 * (chunked prefill), as a dense [rows * index_heads, ihd] x [ihd, P] contraction on
 * the tensor cores (tcgen05, accumulators in tensor memory). Same equation and
 * candidate rule as dsa_score (tp.rs, "Why the indexer is replicated"), with every
 * row reading sequence `seq`:
 *
 *   scores[r, p] = sum_h w[r,h] * relu(scale * <qidx[r,h,:], kpool[seq, p, :]>)
 *
 * when pool_valid[seq, p] != 0 and first_key + (p+1)*kpool - 1 < min(row_ctx[r],
 * seq_lens[seq]); every other entry up to p_stride is -inf. The products are bf16 x
 * bf16 accumulated in f32; the head sum is f32 and takes w[r,h] * |scale| once.
 *
 * qidx [rows, index_heads, ihd] bf16 (16-byte aligned); w [rows, index_heads] f32;
 * row_ctx [rows] i32 (device, nullable: seq_lens[seq]); kpool / pool_valid: the
 * contiguous pooled-key caches [batch, max_seq_len / kpool, ihd] and
 * [batch, max_seq_len / kpool] (pg->block_table must be NULL; dsa_score takes paged
 * caches); seq in [0, pg->batch) (host value); scores [rows, p_stride] f32.
 * Limits: ihd in {64, 128}; index_heads in {32, 64, 128}; 1 <= kpool <= 16.
 * Errors: DSA_ERR_UNSUPPORTED outside the limits or for a paged cache;
 * DSA_ERR_INVALID_ARG for a bad seq, NULL or misaligned tensors. `status` gets
 * DSA_STATUS_TIMEOUT if a pipeline wait inside the kernel gives up (about 1 s); the
 * scores are then incomplete.
 */
int dsa_score_prefill(const dsa_bf16* qidx, const float* w, int rows, int index_heads, int ihd,
                      int seq, const int32_t* row_ctx,
                      const dsa_bf16* kpool, const uint8_t* pool_valid, const dsa_paging* pg,
                      int first_key, int kpool_size, float scale,
                      float* scores, int p_stride, int32_t* status, void* stream);

/*
 * dsa_select -- dsa_topk_pools. mod.rs "Shape of the pipeline": [Q, P] scores
 * -> [Q, select_k] pool ids, select_k = min(index_topk / kpool, p_stride).
 * Per row, k' = min(select_k, number of finite scores); the k' pools first in
 * the order (score descending, pool id ascending; -0.0 equals +0.0) are
 * written in ascending pool id, then -1 up to select_k. -inf is never chosen.
 * NaN scores give unspecified (but in-bounds) results.
 *
 * scores [rows, p_stride] f32; pool_ids [rows, select_k] i32.
 * Limits: p_stride <= 327,680.
 */
int dsa_select(const float* scores, int rows, int p_stride, int index_topk, int kpool,
               int32_t* pool_ids, void* stream);

/*
 * dsa_expand -- dsa_expand_selection. mod.rs, "Checkpoint and kernel facts":
 * the whole index row is -1 except the expanded tokens, so every slot is
 * written: token_ids[r, j*kpool + s] = first_key + pool_ids[r, j]*kpool + s for
 * pool_ids[r, j] >= 0, else -1; positions >= sk*kpool are -1.
 *
 * pool_ids [rows, sk] i32; token_ids [rows, out_width] i32; out_width >= sk*kpool.
 */
int dsa_expand(const int32_t* pool_ids, int rows, int sk, int first_key, int kpool,
               int out_width, int32_t* token_ids, void* stream);

/*
 * dsa_select_expand -- dsa_select then dsa_expand in one launch (the top-k kernel
 * writes each chosen pool's token ids as it writes the pool id): pool_ids and
 * token_ids are bit-identical to the two calls in sequence. No counterpart on the
 * pages beyond the two steps it fuses (mod.rs "Shape of the pipeline", top-k and
 * expand).
 *
 * scores [rows, p_stride] f32; pool_ids [rows, select_k] i32; token_ids
 * [rows, out_width] i32 with out_width >= select_k * kpool.
 * Limits: p_stride <= 327,680; 1 <= kpool <= 16; first_key >= 0.
 */
int dsa_select_expand(const float* scores, int rows, int p_stride, int index_topk, int kpool,
                      int first_key, int out_width, int32_t* pool_ids, int32_t* token_ids,
                      void* stream);

/*
 * dsa_expand_tail -- dsa_expand_selection with always_select_tail set.
 * Glm5NextDsaConfig::out_width (mod.rs) widens the index row by kpool - 1 slots
 * for this flag; mod.rs "Checkpoint and kernel facts" says pooling starts at
 * first_key and a trailing partial pool is not a pool. Reading implemented: the
 * pools expand as in dsa_expand into positions [0, index_topk); from position
 * index_topk on, row r holds the tokens of its trailing partial pool,
 *   [first_key + kpool * floor((L_r - first_key) / kpool), L_r)   (L_r = row_ctx[r]),
 * ascending, by position alone (token validity only gates pool candidacy), and
 * every other slot is -1. Rows with L_r <= first_key have no tail.
 *
 * pool_ids [rows, sk] i32 with sk*kpool <= index_topk; row_ctx [rows] i32
 * (device); token_ids [rows, out_width] i32, out_width >= index_topk + kpool - 1.
 */
int dsa_expand_tail(const int32_t* pool_ids, int rows, int sk, int first_key, int kpool,
                    int index_topk, const int32_t* row_ctx, int out_width, int32_t* token_ids,
                    void* stream);

/*
 * dsa_select_expand_tail -- dsa_select then dsa_expand_tail in one launch:
 * pool_ids and token_ids are bit-identical to the two calls in sequence.
 *
 * scores [rows, p_stride] f32; row_ctx [rows] i32 (device, not NULL); pool_ids
 * [rows, select_k] i32; token_ids [rows, out_width] i32 with
 * out_width >= index_topk + kpool - 1. Limits as dsa_select_expand.
 */
int dsa_select_expand_tail(const float* scores, int rows, int p_stride, int index_topk,
                           int kpool, int first_key, const int32_t* row_ctx, int out_width,
                           int32_t* pool_ids, int32_t* token_ids, void* stream);

/*
 * dsa_sparse_mla_decode -- NoPE MLA restricted to the selected tokens, in the
 * latent space (mod.rs "Shape of the pipeline", last stage; build.rs module
 * doc, transforms 1 and 3: Q is absorbed through kv_b_proj's K half, o_proj
 * through its V half, so each latent row is both key and value).
 *
 *   logit[r,h,t] = softmax_scale * <qlat[r,h,:], ckv[t,:]>, t in token_ids[r] (>= 0)
 *   olat[r,h,:]  = sum_t softmax_t(logit[r,h]) * ckv[t,:]   (0 if no token)
 *   y[r,i]       = bf16(sum_{h,c} o_absorb[i, h*kv_lora_rank + c] * olat[r,h,c])
 *
 * qlat [rows, heads, kv_lora_rank] bf16; row_seq [rows] (device, nullable:
 * row r -> sequence r); ckv: token cache of width kv_lora_rank (bf16) laid out
 * as pg says; token_ids [rows, out_width] i32 (-1 = empty; ids must be below
 * seq_lens of the row's sequence); o_absorb [hidden, heads*kv_lora_rank] bf16
 * (nullable: then y must be NULL and only olat is produced); y [rows, hidden]
 * bf16; olat [rows, heads, kv_lora_rank] f32 (nullable).
 * Limits: kv_lora_rank == 512; hidden % 32 == 0; heads >= 1; qlat, ckv, o_absorb,
 * y, olat and workspace 16-byte aligned (DSA_ERR_INVALID_ARG otherwise). y may be
 * pinned host memory (its sums are then stored straight into it).
 * Projection: with hidden % 128 == 0 the tensor-core form (see dsa_latent_project)
 * takes the bf16 copy of olat this call makes; else the mma.sync stream-K form.
 * Kernels: with 64 heads and at least 4 chunks of 128 tokens per SM
 * (rows * ceil(out_width / 128) >= 4 * SMs: 64 rows of 2,048 tokens) a persistent
 * tensor-core (tcgen05) kernel runs; otherwise a split kernel on mma.sync and a
 * combine. Each is deterministic; their results agree within rounding, not bit for
 * bit. The option DSA_OPT_MLA_KERNEL (dsa_set_option) forces one or the other.
 */
int dsa_sparse_mla_decode_workspace(int rows, int heads, int kv_lora_rank, int out_width,
                                    int hidden, int with_o_absorb, size_t* bytes);

int dsa_sparse_mla_decode(const dsa_bf16* qlat, int rows, int heads, int kv_lora_rank,
                          const int32_t* row_seq, const dsa_bf16* ckv, const dsa_paging* pg,
                          const int32_t* token_ids, int out_width, float softmax_scale,
                          const dsa_bf16* o_absorb, int hidden, dsa_bf16* y, float* olat,
                          int32_t* status, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * dsa_quantize_latent -- encoder of the FP8 latent cache. mod.rs names the serve's
 * FP8 decode kernel (glm5next_dsa_mla_decode_fp8) and nothing of its format; the
 * format here is this library's stated choice: OCP FP8 E4M3 codes (largest finite
 * 448, nearest rounding with ties to even) and one power-of-two scale per token and
 * 128-channel group,
 *
 *   k = the smallest integer with amax_g <= 448 * 2^k, not below -126 (0 if amax_g = 0)
 *   scales[r, g] = 2^k,   codes[r, c] = E4M3(x[r, c] / 2^k)   for c in group g
 *
 * so decoding (code value times 2^k) is exact in bf16.
 * x [rows, kv_lora_rank] bf16 (any token cache viewed as rows); codes [rows,
 * kv_lora_rank] u8; scales [rows, kv_lora_rank / 128] f32.
 * Limits: kv_lora_rank a positive multiple of 128; 16-byte aligned tensors.
 */
int dsa_quantize_latent(const dsa_bf16* x, long long rows, int kv_lora_rank, uint8_t* codes,
                        float* scales, void* stream);

/*
 * dsa_sparse_mla_decode_fp8 -- dsa_sparse_mla_decode over an FP8 latent cache
 * (mod.rs: the serve's decode kernel glm5next_dsa_mla_decode_fp8 reads the selected
 * tokens through the block table). The latent row of token t is the decoded
 * E4M3 code times its group's scale (dsa_quantize_latent); everything else, the
 * equations included, is dsa_sparse_mla_decode's. Each gathered row is 528 bytes
 * (512 codes + 4 scales) instead of 1,024.
 *
 * ckv_codes: token cache of width kv_lora_rank (u8); ckv_scales: token cache of
 * width kv_lora_rank / 128 (f32), both laid out as pg says. The workspace size is
 * dsa_sparse_mla_decode_workspace's. Limits as dsa_sparse_mla_decode.
 */
int dsa_sparse_mla_decode_fp8(const dsa_bf16* qlat, int rows, int heads, int kv_lora_rank,
                              const int32_t* row_seq, const uint8_t* ckv_codes,
                              const float* ckv_scales, const dsa_paging* pg,
                              const int32_t* token_ids, int out_width, float softmax_scale,
                              const dsa_bf16* o_absorb, int hidden, dsa_bf16* y, float* olat,
                              int32_t* status, void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * dsa_frontend -- the decode step's inputs from the hidden state x. build.rs lists
 * the weights and their shapes (DsaTpPlan::new tensor table, build_dsa_weights);
 * the computation is the plain reading of those shapes, with the two a-norms read
 * as RMSNorm (a weight and no bias: the pages single out k_norm as the one norm
 * with a bias):
 *
 *   [q_a | kv_a | k | g | wv] = w_x . x[r]                    (f32 sums)
 *   q_lora   = bf16(q_a / sqrt(mean(q_a^2) + eps) * q_a_norm)
 *   ckv_new  = bf16(kv_a / sqrt(mean(kv_a^2) + eps) * kv_a_norm)
 *   [qlat | qidx] = bf16(w_q . q_lora)
 *   k_new    = bf16(k)    gate_new = bf16(g)    w = wv (f32)
 *
 * w_x [n_x, hidden] bf16 is the load-time row concatenation of q_a_proj
 * [q_lora_rank], kv_a_proj_with_mqa [kv_lora_rank], indexer.wk [ihd], the compress
 * gate [ihd] and indexer.weights_proj [index_heads] (already scaled by
 * index_heads^-0.5, build.rs transform 2), then zero rows up to n_x, so the hidden
 * state is streamed once for all five. w_q [heads * kv_lora_rank + index_heads *
 * ihd, q_lora_rank] bf16 is likewise q_absorb (build.rs absorb_q) with indexer.wq_b
 * below it. q_a_norm [q_lora_rank], kv_a_norm [kv_lora_rank] bf16. x [rows, hidden]
 * bf16.
 * Outputs (row-major, one row per query): qlat [rows, heads, kv_lora_rank] bf16,
 * qidx [rows, index_heads, ihd] bf16, w [rows, index_heads] f32, and the token's
 * staged rows for dsa_indexer_store / dsa_decode_append: k_new, gate_new
 * [rows, ihd] bf16, ckv_new [rows, kv_lora_rank] bf16.
 * Limits: hidden and q_lora_rank multiples of 256; n_x, heads * kv_lora_rank and
 * index_heads * ihd multiples of 64; rows <= 65535; 16-byte aligned x, weights,
 * qlat, qidx and workspace. The weights may be read before the kernel just before
 * this call on the stream has finished, so that kernel must not write them.
 */
int dsa_frontend_workspace(int rows, int hidden, int n_x, int q_lora_rank, int kv_lora_rank,
                           int ihd, int index_heads, int heads, size_t* bytes);

int dsa_frontend(const dsa_bf16* x, int rows, int hidden, const dsa_bf16* w_x, int n_x,
                 int q_lora_rank, int kv_lora_rank, int ihd, int index_heads,
                 const dsa_bf16* q_a_norm, const dsa_bf16* kv_a_norm, float eps,
                 const dsa_bf16* w_q, int heads, dsa_bf16* qlat,
                 dsa_bf16* qidx, float* w, dsa_bf16* k_new, dsa_bf16* gate_new,
                 dsa_bf16* ckv_new, int32_t* status, void* workspace, size_t workspace_bytes,
                 void* stream);

/*
 * dsa_latent_project -- the absorbed output projection on its own (build.rs,
 * module doc, transform 3 and absorb_o: o_proj is multiplied through kv_b_proj's V
 * half, so the decode output [heads, kv_lora_rank] maps back to hidden):
 *
 *   y[r, i] = bf16(sum_k o_absorb[i, k] * bf16(olat[r, k])),  k < heads*kv_lora_rank
 *
 * This is the last step of dsa_sparse_mla_decode, callable separately so that the
 * attention (o_absorb = NULL, olat output) and the projection can be scheduled and
 * timed apart; the two-call form gives results identical to the one-call form.
 * olat [rows, heads*kv_lora_rank] f32 (rounded to bf16 as the MMA operand);
 * Kernel: with hidden % 128 == 0 (and DSA_OPT_PROJECT_KERNEL not forcing mma.sync)
 * olat is first rounded to a bf16 copy in the workspace, then 128-row tiles of
 * o_absorb stream through a TMA ring into tcgen05 MMAs (query rows as N, 16 to 64 per
 * launch), K split over the CTAs of a thread-block cluster whose partials are added
 * through distributed shared memory in rank order; else the mma.sync stream-K kernel
 * and its partial-sum reduction. Both are deterministic; they agree within rounding.
 * o_absorb [hidden, heads*kv_lora_rank] bf16; y [rows, hidden] bf16; status as
 * above (DSA_STATUS_TIMEOUT only). Limits: kv_lora_rank == 512; hidden % 64 == 0;
 * olat, o_absorb, y and workspace 16-byte aligned (DSA_ERR_INVALID_ARG otherwise).
 * Ordering: the kernel may start reading o_absorb (weights) before the kernel just
 * before it on the stream has finished (programmatic dependent launch), so that
 * kernel must not write o_absorb; olat is read only after it has finished.
 * y may be pinned host memory (under unified addressing its address is valid on
 * the device): the final sums are then stored straight into it, with no copy.
 */
int dsa_latent_project_workspace(int rows, int heads, int kv_lora_rank, int hidden,
                                 size_t* bytes);
int dsa_latent_project(const float* olat, int rows, int heads, int kv_lora_rank,
                       const dsa_bf16* o_absorb, int hidden, dsa_bf16* y, int32_t* status,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * dsa_sparse_mla_decode_noalloc -- dsa_sparse_mla_decode for callers that cannot
 * allocate device memory. The pages have no counterpart: this is an interface
 * convenience of this library, not a step of the method.
 *
 * Who needs it: code hosted inside a framework that owns every device
 * allocation and gives plug-ins no allocator, or a latency-critical loop that
 * must never call cudaMalloc/cudaFree (both can synchronise the whole device).
 * Such a caller still passes its inputs and outputs, but no workspace.
 *
 * Arguments, results and errors are those of dsa_sparse_mla_decode, without the
 * workspace pair. The scratch is a fixed array of DSA_NOALLOC_SCRATCH_BYTES
 * compiled into the library; every GPU that loads the library holds one copy
 * until the process exits. A problem whose workspace (as reported by
 * dsa_sparse_mla_decode_workspace) exceeds it is refused with
 * DSA_ERR_UNSUPPORTED before anything is enqueued. No allocation of any kind
 * happens in the call.
 *
 * The first call on each device (with that device current) looks up the
 * array's device address and caches it; make that first call before any stream
 * capture. All calls share the one array and it keeps the last call's
 * contents; nothing in it needs clearing, but calls whose GPU work overlaps in
 * time (other streams, other host threads) race on it: serialise them.
 */
#define DSA_NOALLOC_SCRATCH_BYTES ((size_t)48 << 20)
int dsa_sparse_mla_decode_noalloc(const dsa_bf16* qlat, int rows, int heads, int kv_lora_rank,
                                  const int32_t* row_seq, const dsa_bf16* ckv,
                                  const dsa_paging* pg, const int32_t* token_ids, int out_width,
                                  float softmax_scale, const dsa_bf16* o_absorb, int hidden,
                                  dsa_bf16* y, float* olat, int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
