/*
 * dsa.h -- C ABI of libdsa_gb300.so: the DeepSeek / GLM-5.x sparse-attention
 * hot path (DSA indexer -> per-query top-k -> sparse absorbed-MLA attention)
 * as hand-written CUDA kernels for sm_103a (GB300).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or reads device memory on the host, and never
 *     synchronises the stream.  The only global state is a sticky device error
 *     word (dsa_device_status) and per-kernel launch attributes set once.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every call is asynchronous and ordered on that stream.
 *   - bf16 tensors are raw IEEE bfloat16 bit patterns, row-major, contiguous,
 *     with the base 16-byte aligned.
 *   - Errors are return codes; nothing is thrown across the ABI and the process
 *     is never aborted.  Argument errors are found on the host before any
 *     launch.  Inside kernels, an index outside the cache or a wait that runs
 *     past its limit is recorded in the device status word and the access is
 *     skipped (no trap).
 *   - The model constants are fixed to the GLM-5.x layer traced on the pages
 *     (SlimServe "GLM52_PIPELINE_TRACE.md", Config line; exo PR #2539,
 *     section Prefill): 32 indexer heads of width 128, 64 attention heads,
 *     576-wide absorbed query/key ([512 latent | 64 rope]), 512-wide latent V,
 *     256-wide per-head value after the wv_b up-projection.
 *     Other shapes are DSA_ERR_UNSUPPORTED_SHAPE: there is no fallback path.
 */
#ifndef DSA_GB300_H
#define DSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_ABI_VERSION 5  /* 2: paged-cache entry points; 3: value up-projection, indexer layer schedule;
                              4: attention output element type (out_dtype); 5: wait-timeout self-test */

#define DSA_INDEXER_HEADS 32
#define DSA_INDEXER_DIM 128
#define DSA_HEADS 64
#define DSA_QK_DIM 576
#define DSA_V_DIM 512
#define DSA_V_HEAD_DIM 256
#define DSA_MAX_TOPK 2048

typedef int32_t dsa_status_t;

enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1,         /* null pointer, non-positive size, bad stride */
    DSA_ERR_UNSUPPORTED_SHAPE = 2,   /* head count / width / top_k outside what is built */
    DSA_ERR_MISALIGNED = 3,          /* base pointer or row stride not 16-byte aligned */
    DSA_ERR_WORKSPACE_TOO_SMALL = 4, /* ws_bytes below the matching *_workspace_size() */
    DSA_ERR_CUDA = 5,                /* a CUDA runtime call or launch failed */
    DSA_ERR_DEVICE_TIMEOUT = 6,      /* (device word) an in-kernel wait hit its limit */
    DSA_ERR_DEVICE_BOUNDS = 7,       /* (device word) an index outside the cache was met */
    DSA_ERR_UNSUPPORTED_DEVICE = 8,  /* current device is not compute capability 10.3 */
    DSA_ERR_SCRATCH_TOO_SMALL = 9    /* request does not fit the library's fixed device scratch */
};

/*
 * Element type of an attention output buffer (the out_dtype argument of the
 * mla_sparse_attn_* calls).  The pages fix the softmax in float32 (exo PR
 * #2539, section "Prefill") but not the type of the attention output; in the
 * llama.cpp graph on the SlimServe page ("GLM52_PIPELINE_TRACE.md", section 6)
 * the output kqv = mul_mat(v, kq) is a float32 product that feeds the wv_b
 * up-projection.  DSA_OUT_F32 returns that float32 result.  DSA_OUT_BF16
 * returns the same float32 result rounded to nearest even, for a bf16
 * consumer (such as mla_value_up_proj); the rounding alone moves each element
 * by up to 2^-9 of its magnitude.
 */
#define DSA_OUT_F32 0
#define DSA_OUT_BF16 1

/* Text for a status code (static storage, never NULL). */
const char *dsa_status_string(dsa_status_t status);

/* DSA_ABI_VERSION of the loaded library. */
int dsa_abi_version(void);

/*
 * dsa_indexer_scores -- DSA indexer scores, float32, causal mask applied.
 * Defined on exo PR #2539 (GLM-5.2/5.3 attention), section "Prefill", bullet
 * "Indexer scores in float32, in one kernel": a key's score is relu(q_h . k)
 * times head h's weight, summed over the 32 indexer heads in float32 in one
 * pass with the mask applied (no per-head [L, N] tensors).
 *
 *   scores[b, i, j] = sum_{h<32} w[b,i,h] * relu( sum_{d<128} q_idx[b,i,h,d] * k_idx[b,j,d] )
 *                     for j <= min(q_pos0[b] + i, kv_len[b] - 1)
 *   scores[b, i, j] = -inf for the other j < Nmax          (columns >= Nmax untouched)
 *
 *   q_idx   bf16 [B, L, 32, 128]   indexer queries (post-RoPE)
 *   k_idx   bf16 [B, Nmax, 128]    indexer keys (post-RoPE)
 *   w       f32  [B, L, 32]        per-head weights (any scale folded in)
 *   q_pos0  int32 [B] (device)     position of query 0 of batch b; query i sits at q_pos0[b]+i
 *   kv_len  int32 [B] (device)     keys present in batch b's cache (<= Nmax)
 *   scores  f32  [B, L, ld]        output; ld >= Nmax, ld % 4 == 0
 * Prefill is B = 1 with L queries; batched decode is L = 1 with B sequences.
 * Products are exact bf16 x bf16 in the tensor core, accumulated in float32.
 */
dsa_status_t dsa_indexer_scores(const void *q_idx, const void *k_idx, const float *w,
                                const int32_t *q_pos0, const int32_t *kv_len, int B, int L,
                                int Nmax, float *scores, int64_t ld, void *stream);

/*
 * dsa_topk -- per-query selection of the top_k best-scored causal keys.
 * Defined on exo PR #2539, section "Prefill": each query keeps its top_k
 * (index_topk = 2048) keys; "The first 2048 queries attend causally": a query
 * whose causal key count n = min(q_pos0[b] + i + 1, kv_len[b]) is <= top_k
 * selects every key 0..n-1.  Readings of points the pages leave open:
 * equal scores rank the lower key index first; -0.0 equals +0.0; the chosen
 * indices are written in ascending order; unused slots hold -1.
 *
 *   scores  f32 [B, L, ld] (as written by dsa_indexer_scores; only j < n is read)
 *   idx     int32 [B, L, top_k] output, ascending, -1 padded
 *   1 <= top_k <= 2048; ld >= Nmax, ld % 4 == 0.  Scores must be finite or -inf.
 * Needs no workspace (dsa_topk_workspace_size returns 0; pass NULL, 0).
 */
size_t dsa_topk_workspace_size(int B, int L, int Nmax, int top_k);
dsa_status_t dsa_topk(const float *scores, int64_t ld, const int32_t *q_pos0,
                      const int32_t *kv_len, int B, int L, int Nmax, int top_k, int32_t *idx,
                      void *workspace, size_t ws_bytes, void *stream);

/*
 * mla_sparse_attn_prefill -- absorbed-MLA attention of L queries over their
 * selected keys of one latent cache.
 * Defined on SlimServe "GLM52_PIPELINE_TRACE.md", section 6 "Attention core
 * (absorbed MLA)": Q = [q_nope . wk_b (512) | q_pe (64)], K = [kv_cmpr (512) |
 * k_pe (64)], V = kv_cmpr; scores K.Q times kq_scale, softmax, then V.softmax.
 * exo PR #2539, section "Prefill": each query gathers only its selected keys;
 * scaling, masking and the float32 softmax are fused.
 *
 *   out[i, h, :] = sum_t softmax_t(scale * q[i,h,:] . kv[idx[i,t], :]) * kv[idx[i,t], 0:512]
 * over the entries t with idx[i,t] >= 0 (negative entries are skipped).
 *   q    bf16 [L, 64, 576]     absorbed queries
 *   kv   bf16 [N, 576]         latent cache rows [kv_cmpr | k_pe]
 *   idx  int32 [L, top_k]      selected keys (from dsa_topk); entries >= N are
 *                              recorded as DSA_ERR_DEVICE_BOUNDS and skipped
 *   out  [L, 64, 512]          output: float32 (out_dtype DSA_OUT_F32) or bf16
 *                              (DSA_OUT_BF16, the float32 result rounded to nearest even)
 *   lse  f32 [L, 64] or NULL   natural-log sum of exp of the scaled scores
 * The scores, the softmax and both sums are float32; the probabilities enter the
 * value product as bf16 (the tensor-core operand type of the latent rows).
 * A row with no selected key writes zeros and lse = -inf.
 * scale is the softmax scale (1/sqrt(192 + 64) = 1/16 for GLM-5.x).
 * Needs no workspace for prefill (pass NULL, 0).
 * Errors: DSA_ERR_INVALID_ARG for a null pointer, L < 1, N < 1, a scale that
 * is not a positive finite number or an out_dtype other than DSA_OUT_F32 /
 * DSA_OUT_BF16; DSA_ERR_UNSUPPORTED_SHAPE for top_k outside 1..2048;
 * DSA_ERR_MISALIGNED for q, kv or out not 16-byte aligned.
 */
dsa_status_t mla_sparse_attn_prefill(const void *q, const void *kv, const int32_t *idx, int L,
                                     int N, int top_k, float scale, void *out, int out_dtype,
                                     float *lse, void *workspace, size_t ws_bytes, void *stream);

/*
 * mla_sparse_attn_decode -- the same attention for one new token in each of B
 * independent sequences (exo PR #2539, section "Decode", bullet "Decode
 * attention as GEMMs": the 64 heads of a token share its selected latent
 * keys, so scores and values are two products over those keys).  The selected
 * keys of a sequence are split across CTAs and the partial results merged by a
 * second kernel, through the caller's workspace.
 *
 *   q       bf16 [B, 64, 576]; kv bf16 [B, Nmax, 576]; kv_len int32 [B] (device)
 *   idx     int32 [B, top_k]   (entries >= kv_len[b] recorded as bounds errors, skipped)
 *   out     [B, 64, 512] float32 or bf16 (out_dtype, as for prefill); lse f32 [B, 64] or NULL
 *   workspace  device buffer of at least mla_sparse_attn_workspace_size(B, 1, top_k, 1)
 *              bytes, 16-byte aligned; its contents need no initialisation.
 */
size_t mla_sparse_attn_workspace_size(int B, int L, int top_k, int is_decode);
dsa_status_t mla_sparse_attn_decode(const void *q, const void *kv, const int32_t *kv_len,
                                    const int32_t *idx, int B, int Nmax, int top_k, float scale,
                                    void *out, int out_dtype, float *lse, void *workspace,
                                    size_t ws_bytes, void *stream);

/*
 * mla_sparse_attn_decode_noalloc -- mla_sparse_attn_decode for callers that
 * cannot allocate device memory.  No counterpart in the paper: this is an
 * integration aid, not part of the method.
 *
 * Some callers are not allowed to call cudaMalloc: plugins hosted inside an
 * engine that owns every byte of device memory through its own pool, or
 * latency-critical decode loops where a device allocation (which may
 * synchronise the whole device) is forbidden.  Such callers cannot provide the
 * split-partials workspace that mla_sparse_attn_decode needs.  This variant
 * keeps those partials in a fixed scratch array that lives inside the library
 * (DSA_NOALLOC_SCRATCH_BYTES = 8 MiB on every GPU that loads the library, held
 * until the process exits).  The caller still passes q, kv, kv_len, idx, out
 * and lse exactly as for mla_sparse_attn_decode; arguments and results are the
 * same (the keys of a sequence may be split over fewer CTAs, which changes
 * only float32 rounding).
 *
 *   - B * splits * 64 * 513 * 4 bytes must fit the scratch; this holds for any
 *     B <= DSA_NOALLOC_MAX_BATCH (63) and top_k <= 2048.  Larger B returns
 *     DSA_ERR_SCRATCH_TOO_SMALL without launching anything.
 *   - The first call on a device looks up the scratch's device address (a
 *     runtime symbol query, no allocation); make that first call before any
 *     stream capture.
 *   - Every call on a device shares the one scratch array and it keeps the last
 *     call's contents (nothing in it needs to start at zero).  Calls whose
 *     kernels overlap on the GPU (different streams, or different host threads
 *     without ordering) race on it and give wrong results: serialise them.
 *   - Allocates nothing: no cudaMalloc / cudaFree and no allocating library call.
 */
#define DSA_NOALLOC_SCRATCH_BYTES (8u << 20)
#define DSA_NOALLOC_MAX_BATCH 63
dsa_status_t mla_sparse_attn_decode_noalloc(const void *q, const void *kv, const int32_t *kv_len,
                                            const int32_t *idx, int B, int Nmax, int top_k,
                                            float scale, void *out, int out_dtype, float *lse,
                                            void *stream);

/*
 * Paged caches.  Serving engines keep each sequence's cache rows in fixed-size
 * pages of one shared pool instead of a dense [B, Nmax, ...] block (exo PR
 * #2539 batches decode through per-sequence "batch caches", section "Decode";
 * the page table is this library's layout for them).  The two calls below read
 * the keys through a page table; everything else (positions, kv_len, the
 * top-k, the results) is exactly as in dsa_indexer_scores and
 * mla_sparse_attn_decode with the dense cache
 *
 *   k[b, j, :] = pool[block_table[b * bt_stride + j / page_size] * page_size + j % page_size, :]
 *
 * for every key j < kv_len[b].  So dsa_topk runs unchanged on the scores and
 * the selected indices stay logical key positions.
 *
 *   block_table  int32 [B, bt_stride] (device): pool page of each logical page.
 *                Entries of pages that hold a key j < kv_len[b] must lie in
 *                [0, num_pages); an entry outside that range is recorded as
 *                DSA_ERR_DEVICE_BOUNDS and its rows are read as zeros.  Entries
 *                of later pages are never read.
 *   page_size    rows per page: a power of two, 16 <= page_size <= 65536.
 *   num_pages    pages in the pool; num_pages * page_size <= 2^31 - 1.
 *   Nmax         the largest kv_len (a bound, as for the dense calls);
 *                Nmax <= bt_stride * page_size.
 *   k_pool       bf16 [num_pages * page_size, 128]   indexer keys
 *   kv_pool      bf16 [num_pages * page_size, 576]   latent cache rows
 * Any L works for the indexer (chunked prefill over a paged cache as well as
 * decode); attention has a decode call (one query per sequence) and a prefill
 * call (a chunk of one sequence's queries).
 */
dsa_status_t dsa_indexer_scores_paged(const void *q_idx, const void *k_pool, const float *w,
                                      const int32_t *q_pos0, const int32_t *kv_len,
                                      const int32_t *block_table, int bt_stride, int page_size,
                                      int num_pages, int B, int L, int Nmax, float *scores,
                                      int64_t ld, void *stream);
dsa_status_t mla_sparse_attn_decode_paged(const void *q, const void *kv_pool, const int32_t *kv_len,
                                          const int32_t *block_table, int bt_stride, int page_size,
                                          int num_pages, const int32_t *idx, int B, int Nmax,
                                          int top_k, float scale, void *out, int out_dtype,
                                          float *lse, void *workspace, size_t ws_bytes,
                                          void *stream);
/* Prefill (a chunk of L queries of one sequence) over that sequence's paged
 * cache: mla_sparse_attn_prefill with kv[j] = kv_pool[block_table[j / page_size]
 * * page_size + j % page_size] for the N keys j < N (block_table holds
 * ceil(N / page_size) entries).  Chunked prefill writes a chunk's keys into the
 * pool, runs dsa_indexer_scores_paged and dsa_topk for the chunk's queries, then
 * this call.  Needs no workspace (pass NULL, 0). */
dsa_status_t mla_sparse_attn_prefill_paged(const void *q, const void *kv_pool,
                                           const int32_t *block_table, int page_size, int num_pages,
                                           const int32_t *idx, int L, int N, int top_k, float scale,
                                           void *out, int out_dtype, float *lse, void *workspace,
                                           size_t ws_bytes, void *stream);

/*
 * mla_value_up_proj -- the value up-projection (wv_b) after the attention.
 * Defined on SlimServe "GLM52_PIPELINE_TRACE.md", section 6 "Attention core
 * (absorbed MLA)": the attention's output lives in the 512-wide latent space
 * and the product with wv_b decompresses it to each head's value ("MQA ->
 * MHA"); Config line: kv_lora_rank 512, v_head_dim 256, 64 heads.  exo PR
 * #2539, section "Prefill": the value up-projection runs once for all queries.
 *
 *   v[r, h, e] = sum_{d<512} o[r, h, d] * wv_b[h, e, d]     for e < 256
 *
 *   o     bf16 [R, 64, 512]    attention output (mla_sparse_attn_prefill / _decode)
 *   wv_b  bf16 [64, 256, 512]  per head, one 512-wide row per value feature
 *                              (the row-major layout of a per-head [256 x 512] weight)
 *   v     bf16 [R, 64, 256]    output (round to nearest even from float32)
 * bf16 x bf16 products accumulated in float32 by the tensor cores.  R >= 1 rows
 * (a prefill chunk's queries, or one row per sequence in decode).  All three
 * pointers are caller-owned device memory, 16-byte aligned; o and v must not
 * overlap.  Needs no workspace.
 * Errors (host, before any launch): DSA_ERR_INVALID_ARG for a null pointer or
 * R < 1, DSA_ERR_UNSUPPORTED_SHAPE when R * 64 exceeds 2^31 - 1,
 * DSA_ERR_MISALIGNED, DSA_ERR_UNSUPPORTED_DEVICE, DSA_ERR_CUDA when the launch
 * fails.  An in-kernel wait that runs past its limit sets
 * DSA_ERR_DEVICE_TIMEOUT in the device status word.
 */
dsa_status_t mla_value_up_proj(const void *o, const void *wv_b, int R, void *v, void *stream);

/*
 * dsa_indexer_source_layer -- which layer's top-k selection a layer attends
 * with, when the indexer is shared across layers.
 * SlimServe "GLM52_PIPELINE_TRACE.md", Config line: index_topk_freq and
 * index_skip_topk_offset (4 and 3 for GLM-5.x); exo PR #2539, section
 * "Correctness" (weights bullet): of the first 8 layers, layers 0, 1, 2 and 6
 * run the indexer and layers 3, 4, 5 and 7 reuse a selection.  Reading (the
 * pages give only these values and that example): every layer below
 * skip_offset runs the indexer; from skip_offset on, layer l runs it when
 * (l - skip_offset + 1) is a multiple of topk_freq, and otherwise reuses the
 * selection of the nearest earlier layer that ran it.
 *
 * Returns `layer` itself when the layer runs the indexer, the earlier layer it
 * reuses otherwise, or -1 for invalid arguments (layer < 0, topk_freq < 1,
 * skip_offset < 1).  Host-only, pure function.
 */
int dsa_indexer_source_layer(int layer, int topk_freq, int skip_offset);

/*
 * dsa_selftest_wait_timeout -- failure-detection self-test of the kernels'
 * bounded waits.  Launches one CTA on `stream` whose first thread waits, with
 * the same wait routine the kernels use (spin = 0: the suspending try_wait
 * form of the worker warps; spin = 1: the polling test_wait form of the MMA
 * issuers and loaders), on a fresh mbarrier that nothing arrives on.  The wait
 * gives up after `limit_ns` nanoseconds of the global timer, records
 * DSA_ERR_DEVICE_TIMEOUT in the device status word (dsa_device_status reads
 * it) and the kernel returns; the context stays usable.  Nothing faults,
 * traps or hangs.
 * Errors (host, before any launch): DSA_ERR_INVALID_ARG unless spin is 0 or 1
 * and 0 < limit_ns <= 1e9; DSA_ERR_UNSUPPORTED_DEVICE; DSA_ERR_CUDA when the
 * launch fails.
 */
dsa_status_t dsa_selftest_wait_timeout(int spin, uint64_t limit_ns, void *stream);

/*
 * dsa_device_status -- synchronise `stream`, then read (and if `reset` is
 * non-zero, clear) the sticky device error word.  *code_out receives DSA_OK,
 * DSA_ERR_DEVICE_TIMEOUT or DSA_ERR_DEVICE_BOUNDS (timeout wins if both).
 */
dsa_status_t dsa_device_status(void *stream, int32_t *code_out, int reset);

#ifdef __cplusplus
}
#endif

#endif /* DSA_GB300_H */
