/*
 * paged_attn.h -- C ABI of the GB300 (sm_103a) ubatch-aligned paged attention
 * library (libpagedattn.so).
 *
 * The method: "面向多并发长上下文的 llama.cpp 分页式 KV Cache 与计算加速优化"
 * (gitlink IFwnjPgFSU/mxzntdncglxtsjysx), section 作品简介.  The KV cache keeps,
 * per sequence, a page mapping and a true KV length; at graph build both are
 * expanded per ubatch token in token order; the attention operator then reads,
 * for each query, only the valid pages of that query's own sequence -- never
 * the free cells or padding of a unified span.  The companion write of new K/V
 * rows into their pages is the "reshape-and-cache" kernel of the CacheFlow page
 * (section 核心架构 3).
 *
 * Entry points
 * ------------
 *  the path:   paged_expand_ubatch, paged_kv_append, paged_attn_plan,
 *              paged_attn_prefill, paged_attn_decode, paged_attn_decode_append,
 *              paged_attn_run, paged_attn_forward, paged_attn_forward_noalloc
 *  around it:  paged_attn_workspace_size, paged_attn_validate,
 *              paged_attn_read_error, paged_attn_strerror, paged_attn_version,
 *              paged_attn_set_prefill_min_run, paged_attn_set_decode_wait_limit,
 *              pa_pool_* (host page pool)
 *  beyond it:  paged_attn_plan_decode, paged_attn_plan_prefill;
 *              paged_attn_masked_decode and paged_attn_masked_prefill (the
 *              unified-span baseline that paging replaces); paged_kv_append_fp8,
 *              paged_attn_decode_fp8, paged_attn_prefill_fp8 and
 *              paged_attn_forward_fp8 (FP8 pages); paged_copy_pages and
 *              pa_pool_fork (copy-on-write forks of shared pages)
 *
 * Conventions shared by every call
 * --------------------------------
 *  - f16 data are IEEE binary16 values passed as uint16_t bit patterns.
 *  - KV pool: k_pages and v_pages, each [num_pages][Hkv][P][d], contiguous.
 *    Sequence position p lives in page tok_page_table[t][p / P] at in-page
 *    offset p % P.  One (page, KV head) tile is contiguous.
 *  - q and out: [T][Hq][d]; new K/V rows k and v: [T][Hkv][d]; contiguous.
 *  - Query head h reads KV head h / (Hq / Hkv) (contiguous GQA grouping).
 *  - tok_kv_len[t] is the number of keys token t attends to: keys 0 ..
 *    tok_kv_len[t]-1 of its sequence (causal prefill: position + 1).  A value of
 *    0 gives an all-zero output row.
 *  - tok_page_table rows are padded with -1 past the sequence's pages.  Tokens
 *    whose rows are byte-identical may share tensor-core tiles; pad rows
 *    canonically (the same way for every token of a sequence).
 *  - Supported shapes: d in {64, 128}; P in {16, 32, 64, 128}; Hq % Hkv == 0
 *    with Hq / Hkv in {1, 2, 4, 8}; T >= 0.  Others return PA_EUNSUPPORTED.
 *  - All pointers except `stream` are DEVICE pointers unless stated.  Device
 *    buffers must be 16-byte aligned.  The caller owns every buffer; the
 *    library allocates no device memory.  Calls are asynchronous on `stream`
 *    (a cudaStream_t; NULL = legacy default stream) and never synchronise,
 *    except paged_attn_read_error.
 *  - Errors: host-side argument checks return a negative status before any
 *    launch.  Device-side problems (a page id outside [0, num_pages), a
 *    kv_len beyond the row's capacity, a bounded wait that timed out) never
 *    trap: the kernel skips the bad access, records a PA_ERR_* bit in the
 *    workspace error word, and paged_attn_read_error returns it.
 *  - Tracing: every call that launches kernels opens an NVTX range named after
 *    itself for its duration on the host, so a profiler's timeline shows which
 *    call launched which kernels.  Without a tool attached it costs nothing.
 */
#ifndef PAGED_ATTN_H
#define PAGED_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define PA_OK 0
#define PA_EINVAL (-1)        /* null pointer, negative size, inconsistent shapes */
#define PA_EUNSUPPORTED (-2)  /* shape outside the supported set */
#define PA_EWORKSPACE (-3)    /* workspace missing or smaller than required */
#define PA_ELAUNCH (-4)       /* a CUDA launch or runtime call failed */
#define PA_EDEVICE (-5)       /* the device error word is non-zero (see PA_ERR_*) */
#define PA_EALIGN (-6)        /* a device pointer is not 16-byte aligned */

/* Bits of the device error word. */
#define PA_ERR_PAGE_RANGE 0x1   /* a page id needed by some token is outside [0, num_pages) */
#define PA_ERR_KV_RANGE 0x2     /* tok_kv_len[t] < 0 or > max_pages * P */
#define PA_ERR_SLOT_RANGE 0x4   /* slot_mapping[t] >= num_pages * P */
#define PA_ERR_TIMEOUT 0x8      /* a bounded device-side wait gave up */
#define PA_ERR_SEQ_RANGE 0x10   /* expansion: tok_seq[t] >= n_seq or position beyond the row */

/* Human-readable text of a status code (static storage). */
const char *paged_attn_strerror(int status);

/* ABI version of this library (major * 100 + minor). */
int paged_attn_version(void);

/*
 * Per-token expansion of the page table and the true KV length (page section
 * 作品简介: "依据 ubatch 中各 token 的序列归属将页表和真实 KV 长度按 token 顺序展开").
 *
 *   seq_page_table [n_seq][max_pages] int32  per-sequence physical page ids, -1 padded
 *   tok_seq [T] int32     sequence of each ubatch token; < 0 marks a padding token
 *   tok_pos [T] int32     position of the token in its sequence
 *   tok_page_table [T][max_pages] int32 (out)  copy of the token's sequence row
 *   tok_kv_len [T] int32 (out)                 tok_pos + 1 (0 for padding)
 *   slot_mapping [T] int64 (out)               page * P + tok_pos % P, with
 *       page = row[tok_pos / P]; -1 for padding or an unallocated page
 *   err (device, optional, may be NULL): PA_ERR_SEQ_RANGE is OR-ed in when a
 *       token names a sequence >= n_seq or a position beyond its row; such a
 *       token is expanded as padding.
 * One launch.  Returns PA_OK or a negative status.
 */
int paged_expand_ubatch(const int32_t *seq_page_table, int n_seq, int max_pages,
                        const int32_t *tok_seq, const int32_t *tok_pos, int T, int P,
                        int32_t *tok_page_table, int32_t *tok_kv_len, int64_t *slot_mapping,
                        int *err, void *stream);

/*
 * reshape-and-cache (CacheFlow page, section 核心架构 3): write the new K and V
 * rows of each ubatch token into their slots.
 *
 *   k, v [T][Hkv][d] binary16      new rows
 *   slot_mapping [T] int64          slot = page * P + offset; < 0 = skip token
 *   k_pages, v_pages [num_pages][Hkv][P][d] binary16 (in/out)
 *   err (device, optional): PA_ERR_SLOT_RANGE is OR-ed in for a slot beyond the
 *       pool; that token is skipped.
 * Bit copy: the pool after the call differs from before only in the written
 * rows.  One launch.
 */
int paged_kv_append(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping, int T,
                    uint16_t *k_pages, uint16_t *v_pages, int num_pages, int Hkv, int P, int d,
                    int *err, void *stream);

/*
 * Bytes of device workspace that paged_attn_plan / _prefill / _decode /
 * _forward need for a ubatch of T tokens (current device's SM count is used).
 * Returns 0 for unsupported shapes.
 */
size_t paged_attn_workspace_size(int T, int Hq, int Hkv, int d);

/*
 * Plan a ubatch (device-side, no host round trip, graph-capturable).  Finds
 * runs of consecutive tokens whose page-table rows are byte-identical; runs of
 * at least the prefill threshold (paged_attn_set_prefill_min_run) become
 * tensor-core tiles of up to 128 tokens; the remaining tokens become decode
 * work, split along the KV axis over all SMs.  Also clears the workspace error
 * word.  The plan stays valid for any number of later _prefill / _decode /
 * _run calls with the same tok_page_table / tok_kv_len contents (for example
 * once per layer).
 */
int paged_attn_plan(const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len,
                    int T, int Hq, int Hkv, int P, int d,
                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * Prefill part of the attention: every planned tile computes
 *   out[t][h] = softmax_j(scale * q[t][h] . K_t[j]) V_t[j],  j < tok_kv_len[t],
 * with K_t/V_t read through the tile's page-table row, on tcgen05 tensor cores
 * (f16 inputs, f32 accumulation, f16 output).  Writes only the rows of tile
 * tokens.  Requires a preceding paged_attn_plan on the same workspace.
 */
int paged_attn_prefill(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                       const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len,
                       int T, int Hq, int Hkv, int P, int d, int num_pages, float scale,
                       uint16_t *out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Decode part: split-KV attention for the planned decode tokens (GQA-grouped,
 * each KV block read once per KV head), then the log-sum-exp reduce of the
 * splits (CacheFlow page, section 核心架构 3: partition + reduce for long
 * contexts).  Writes only the rows of decode tokens.  Requires a preceding
 * paged_attn_plan on the same workspace.
 */
int paged_attn_decode(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                      const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len,
                      int T, int Hq, int Hkv, int P, int d, int num_pages, float scale,
                      uint16_t *out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * paged_attn_decode with the decode step's append fused in: the launch also writes
 * the new K and V rows of the planned decode tokens (reshape-and-cache, CacheFlow
 * page, section 核心架构 3), so a decode layer is one launch instead of two.
 *   k_new, v_new [T][Hkv][d] binary16 (16-byte aligned); slot_mapping [T] int64, as
 *   paged_kv_append; k_pages, v_pages are written.  Other arguments as
 *   paged_attn_decode (a preceding plan on the same workspace).
 * Each decode token's new row must be its last key (slot of position kv_len - 1), as
 * in a decode step, and a sequence may have at most one decode token in the ubatch:
 * the row is written by the CTA that reads it, just before it reads it.  A token with
 * slot < 0 is not written; a slot other than its last key's sets PA_ERR_SLOT_RANGE and
 * is not written.  Rows of tokens on the prefill path are not written (append them
 * with paged_kv_append).  The result equals paged_kv_append then paged_attn_decode.
 */
int paged_attn_decode_append(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                             const int64_t *slot_mapping, uint16_t *k_pages, uint16_t *v_pages,
                             const int32_t *tok_page_table, int max_pages,
                             const int32_t *tok_kv_len, int T, int Hq, int Hkv, int P, int d,
                             int num_pages, float scale, uint16_t *out, void *workspace,
                             size_t workspace_bytes, void *stream);

/* paged_attn_prefill followed by paged_attn_decode (a planned ubatch). */
int paged_attn_run(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                   const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len,
                   int T, int Hq, int Hkv, int P, int d, int num_pages, float scale,
                   uint16_t *out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * The whole attention for one ubatch: paged_attn_plan then paged_attn_run.
 * out[t][h] for every token t and query head h.  workspace_bytes must be at
 * least paged_attn_workspace_size(T, Hq, Hkv, d).
 */
int paged_attn_forward(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                       const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len,
                       int T, int Hq, int Hkv, int P, int d, int num_pages, float scale,
                       uint16_t *out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * paged_attn_forward without a caller-provided workspace, for callers that
 * cannot allocate device memory (a host framework that owns all device memory,
 * a fixed up-front memory budget, a latency-critical path where an allocation
 * could synchronise the device).  The pages have no counterpart of this call;
 * it exists only for such callers.
 *
 * Same arguments and result as paged_attn_forward, minus workspace.  The
 * scratch is one fixed 64 MiB array in device memory inside this library,
 * held by every GPU that loads the library until the process exits; the call
 * allocates nothing.  A ubatch whose paged_attn_workspace_size(T, Hq, Hkv, d)
 * exceeds 64 MiB is rejected with PA_EWORKSPACE (about 4000 tokens at 32/8
 * heads, d 128, on 152 SMs).  The first call on each device looks up the array's device
 * address; make that first call before any stream capture.  Every call shares
 * the array and it keeps the last call's contents (each call clears what it
 * needs); calls that overlap on the GPU race and must be serialised.  The
 * device error word of these calls is not exposed, so a bad page id or kv_len
 * goes unreported (the bad access is still skipped, never made): check the
 * tables with paged_attn_validate first.  Every input gets the status that
 * paged_attn_forward would return for it (the same checks, in the same order).
 */
int paged_attn_forward_noalloc(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                               const int32_t *tok_page_table, int max_pages,
                               const int32_t *tok_kv_len, int T, int Hq, int Hkv, int P, int d,
                               int num_pages, float scale, uint16_t *out, void *stream);

/*
 * Check the tables without trapping: every page id a token needs
 * (row[0 .. ceil(kv_len/P)-1]) must lie in [0, num_pages) and 0 <= kv_len <=
 * max_pages * P.  OR-s PA_ERR_PAGE_RANGE / PA_ERR_KV_RANGE into *err (device).
 */
int paged_attn_validate(const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len,
                        int T, int P, int num_pages, int *err, void *stream);

/*
 * paged_attn_plan with every token routed to the split-KV path (none to the
 * tensor-core tiles): the plan that paged_attn_masked_decode and
 * paged_attn_decode_fp8 run on.  Arguments as paged_attn_plan.
 */
int paged_attn_plan_decode(const int32_t *tok_page_table, int max_pages,
                           const int32_t *tok_kv_len, int T, int Hq, int Hkv, int P, int d,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * Unified-span baseline (UA-PagedAttention page, section 作品简介: the original
 * llama.cpp cache is one span of cells shared by all sequences, and attention
 * reads the whole span under a mask that keeps each query's own sequence).
 * Split-KV decode attention of every token over the keys its table row names,
 * keeping only key j whose slot s = page * P + j % P holds a cell of the token's
 * own sequence at a position up to its own:
 *     cell_seq[s] == tok_seq[t]  and  cell_pos[s] <= tok_pos[t].
 * Point every token's row at all pages of a span, with kv_len = the span length,
 * and this is the unified-cache attention that paging replaces: same kernel
 * engine as paged_attn_decode, but each token streams the whole span.
 *   cell_seq, cell_pos [num_pages * P] int32 (device, 16-byte aligned): the
 *       sequence (-1 = free) and position of the cell in each slot
 *   tok_seq, tok_pos [T] int32 (device): each token's sequence and position
 *   other arguments as paged_attn_forward.  Runs on the workspace's plan, which
 *   must come from paged_attn_plan_decode (every token on the split-KV path) for
 *   the same tables; writes out for every token.  A token whose mask keeps no
 *   key gets a zero row.
 */
int paged_attn_masked_decode(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                             const int32_t *tok_page_table, int max_pages,
                             const int32_t *tok_kv_len, int T, int Hq, int Hkv, int P, int d,
                             int num_pages, float scale, const int32_t *cell_seq,
                             const int32_t *cell_pos, const int32_t *tok_seq,
                             const int32_t *tok_pos, uint16_t *out, void *workspace,
                             size_t workspace_bytes, void *stream);

/*
 * paged_attn_plan with every token routed to the tensor-core tiles (none to the
 * split-KV path): the plan that paged_attn_masked_prefill runs on.  Arguments as
 * paged_attn_plan.
 */
int paged_attn_plan_prefill(const int32_t *tok_page_table, int max_pages,
                            const int32_t *tok_kv_len, int T, int Hq, int Hkv, int P, int d,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * Unified-span baseline for prefill (UA-PagedAttention page, section 作品简介: the
 * original cache is one span of cells shared by all sequences, read whole under a
 * mask; section 关键性能数据 measures the prefill of 16K prompts x 8 against it).
 * The same computation as paged_attn_masked_decode, on the tcgen05 prefill tiles:
 * every token attends to the keys its table row names, keeping only key j whose slot
 * s = page * P + j % P holds a cell of the token's own sequence at a position up to
 * its own (cell_seq[s] == tok_seq[t] and cell_pos[s] <= tok_pos[t]).  With every row
 * naming the whole span and kv_len = the span length, consecutive tokens share a tile
 * whatever their sequence, and each tile streams the whole span.
 *   Arguments as paged_attn_masked_decode.  Runs on the workspace's plan, which must
 *   come from paged_attn_plan_prefill (every token in a tile) for the same tables;
 *   writes out for every token.  A cell with cell_seq >= 0 must hold written (finite)
 *   K/V; the V rows of free cells (cell_seq < 0) are zeroed in shared memory, so their
 *   contents never matter.  A token whose mask keeps no key gets a zero row.
 */
int paged_attn_masked_prefill(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                              const int32_t *tok_page_table, int max_pages,
                              const int32_t *tok_kv_len, int T, int Hq, int Hkv, int P, int d,
                              int num_pages, float scale, const int32_t *cell_seq,
                              const int32_t *cell_pos, const int32_t *tok_seq,
                              const int32_t *tok_pos, uint16_t *out, void *workspace,
                              size_t workspace_bytes, void *stream);

/*
 * Reduced-precision KV pages: FP8 E4M3 codes with one binary32 scale per cached
 * row (token, KV head) -- the adaptive KV quantisation the
 * "面向边缘智能体推理的 llama.cpp KV Cache 共享与复用优化" page names; on the
 * UA-PagedAttention page the KV cache is binary16.  Decode streams half the bytes.
 *
 * Quantising reshape-and-cache: for each token with slot >= 0 and each KV head,
 * scale = amax(row) / 448 in binary32 (1 for an all-zero row) and
 * code_i = E4M3(x_i / scale) (nearest, ties to even, saturating at +-448).
 *   k, v [T][Hkv][d] binary16; slot_mapping [T] int64 (as paged_kv_append)
 *   k8_pages  [num_pages][Hkv][P][d] uint8   K codes, one row per cached token
 *   v8t_pages [num_pages][Hkv][d][P] uint8   V codes, transposed in each block
 *   k_scale, v_scale [num_pages][Hkv][P] float
 *   err (device, optional): PA_ERR_SLOT_RANGE for a slot beyond the pool.
 * d must be a multiple of 32, at most 128.  Bit-exact against the reference
 * quantiser.  One launch.
 */
int paged_kv_append_fp8(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping, int T,
                        uint8_t *k8_pages, uint8_t *v8t_pages, float *k_scale, float *v_scale,
                        int num_pages, int Hkv, int P, int d, int *err, void *stream);

/*
 * Split-KV decode attention over FP8 pages (layout above; page size 128, d 128,
 * scale arrays 16-byte aligned): K_t[j] = E4M3(k8) * k_scale, V_t[j] likewise.
 * Runs on the workspace's plan for the same tables (one plan serves every layer):
 * from paged_attn_plan_decode it writes out for every token; from paged_attn_plan,
 * for the tokens the plan leaves to the decode kernel (as paged_attn_decode).  Other
 * arguments as paged_attn_forward.  PA_EUNSUPPORTED for another page size or head
 * dimension.
 */
int paged_attn_decode_fp8(const uint16_t *q, const uint8_t *k8_pages, const uint8_t *v8t_pages,
                          const float *k_scale, const float *v_scale,
                          const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len,
                          int T, int Hq, int Hkv, int P, int d, int num_pages, float scale,
                          uint16_t *out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Tensor-core prefill tiles over FP8 pages: the tokens of the workspace's plan's
 * tiles (from paged_attn_plan or paged_attn_plan_prefill for the same tables), as
 * paged_attn_prefill.  Layout, page size, head dimension and scale arrays as
 * paged_attn_decode_fp8.  Each key block's codes are widened in shared memory: K to
 * binary16(code * scale), the value a binary16 cache of the dequantised rows would
 * hold; V to the exact code values, with each key's V scale carried by the
 * probabilities (binary16(p * scale)), as in paged_attn_decode_fp8.  The tile then runs
 * the binary16 MMAs of paged_attn_prefill.  Keys past a tile's longest kv_len get
 * cleared V codes and a zero scale, so unwritten cells (NaN codes included) never
 * reach the output.  A K scale below the binary16 range (2^-24) widens to zero.
 * PA_ERR_PAGE_RANGE as paged_attn_forward.  One launch.
 */
int paged_attn_prefill_fp8(const uint16_t *q, const uint8_t *k8_pages, const uint8_t *v8t_pages,
                           const float *k_scale, const float *v_scale,
                           const int32_t *tok_page_table, int max_pages,
                           const int32_t *tok_kv_len, int T, int Hq, int Hkv, int P, int d,
                           int num_pages, float scale, uint16_t *out, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * paged_attn_forward over FP8 pages: paged_attn_plan, then paged_attn_prefill_fp8
 * and paged_attn_decode_fp8 on that plan.  A whole mixed ubatch (prefill runs and
 * decode tokens) in three launches plus the plan's two.
 */
int paged_attn_forward_fp8(const uint16_t *q, const uint8_t *k8_pages, const uint8_t *v8t_pages,
                           const float *k_scale, const float *v_scale,
                           const int32_t *tok_page_table, int max_pages,
                           const int32_t *tok_kv_len, int T, int Hq, int Hkv, int P, int d,
                           int num_pages, float scale, uint16_t *out, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * Page copy for copy-on-write forks (CacheFlow page, section 核心架构 2: blocks
 * shared by reference count; 核心架构 3: a block-copy kernel).  A forked sequence
 * shares every full page of its parent and gets a private copy of the partly
 * filled last page before it appends to it (see pa_pool_fork).
 *
 * Copies whole pages, every KV head, K and V: page dst[i] <- page src[i], i < n.
 *   src, dst [n] int32 (device)     page ids
 *   k_pages, v_pages [num_pages][Hkv][P][d] binary16 (in/out, 16-byte aligned)
 *   err (device, optional, may be NULL): PA_ERR_PAGE_RANGE is OR-ed in for a
 *       pair with an id outside [0, num_pages); that pair is skipped.
 * The dst ids must be distinct and none may be among the src ids: the pairs are
 * copied in parallel.  Bit copy in 16-byte units.  One launch; PA_EUNSUPPORTED
 * if Hkv * P * d is not a multiple of 8.
 */
int paged_copy_pages(const int32_t *src, const int32_t *dst, int n, uint16_t *k_pages,
                     uint16_t *v_pages, int num_pages, int Hkv, int P, int d, int *err,
                     void *stream);

/*
 * Synchronise `stream` and copy the workspace error word to *err_host (host
 * pointer).  Returns PA_OK if it is zero, PA_EDEVICE otherwise.
 */
int paged_attn_read_error(const void *workspace, int *err_host, void *stream);

/*
 * Tuning knob: the shortest run of consecutive same-row tokens that is sent
 * to the tensor-core prefill path (default 16; 1 sends every token there,
 * a huge value sends every token to the decode path).  Process-wide; affects
 * plans made after the call.  Returns the previous value.
 */
int paged_attn_set_prefill_min_run(int min_run);

/*
 * Limit, in nanoseconds, of every bounded device-side wait of the split-KV decode
 * kernel (paged_attn_decode, paged_attn_masked_decode, paged_attn_decode_fp8 and the
 * decode part of paged_attn_run / _forward); default 2 s.  0 restores the default;
 * values below 1000 become 1000.  Process-wide; affects launches made after the call.
 * Returns the previous value.  A wait that gives up sets PA_ERR_TIMEOUT in the
 * workspace error word; every role of the CTA then stops, the copies it already
 * issued land (their own, unshortened bound) and the launch returns with the rows it
 * did not finish unwritten.  After such a launch, plan again before the next run (the
 * plan's arrival counters may be left mid-count).  The other kernels keep the fixed
 * 2 s limit.  Meant for tests of the timeout path and for callers that prefer an
 * early error to a long stall.
 */
unsigned long long paged_attn_set_decode_wait_limit(unsigned long long ns);

/*
 * Host-side page pool (the per-sequence page mapping of 作品简介; CacheFlow
 * section 核心架构 2: fixed-size blocks with a block table, blocks shared by
 * reference count).  Pure host code; no CUDA call.  Page ids are handed out
 * lowest-first from a free list; a page returns to the free list when its
 * reference count drops to zero.
 */
typedef struct pa_page_pool pa_page_pool;

/* New pool of num_pages pages, all free.  NULL on bad size or allocation failure. */
pa_page_pool *pa_pool_create(int num_pages);
void pa_pool_destroy(pa_page_pool *pool);
/* Number of free pages. */
int pa_pool_num_free(const pa_page_pool *pool);
/* Take n free pages (refcount 1) into out_pages (host array of n).  Returns n,
 * or PA_EINVAL / -7 (PA_ENOSPACE) without taking any when fewer than n are free. */
#define PA_ENOSPACE (-7)
int pa_pool_alloc(pa_page_pool *pool, int n, int32_t *out_pages);
/* Add one reference to each of the n pages (sharing, e.g. a common prefix). */
int pa_pool_share(pa_page_pool *pool, const int32_t *pages, int n);
/* Drop one reference from each of the n pages; pages reaching zero are freed. */
int pa_pool_release(pa_page_pool *pool, const int32_t *pages, int n);
/* Reference count of one page (0 = free), or PA_EINVAL. */
int pa_pool_refcount(const pa_page_pool *pool, int32_t page);
/*
 * Copy-on-write fork of a sequence that holds n_tokens tokens in pages[0 ..
 * ceil(n_tokens / P)) (host arrays).  The child shares the full pages (one more
 * reference each).  If the last page is partly filled, the child gets a fresh
 * page in its place and (*copy_src, *copy_dst) receive (parent's last page,
 * fresh page): copy it with paged_copy_pages before either side appends into
 * it.  out_pages (host, ceil(n_tokens / P) entries) receives the child's list.
 * Returns the number of pages to copy (0 or 1), PA_EINVAL (bad arguments or a
 * page not in use), or PA_ENOSPACE; on error nothing changes.
 */
int pa_pool_fork(pa_page_pool *pool, const int32_t *pages, int n_tokens, int P,
                 int32_t *out_pages, int32_t *copy_src, int32_t *copy_dst);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_ATTN_H */
