/*
 * cpmla.h -- C ABI of libcpmla.so: context-parallel (PCP) prefill attention
 * over MLA latent KV on one GB300 (sm_103a).
 *
 * The path (one call each, in this order):
 *   1. pcp_dualchunk_partition   host: DualChunkSwap split into P virtual shards
 *   2. mla_partial_attn_dense /  device: per-shard partial attention (O, LSE)
 *      mla_partial_attn_sparse           over the full latent KV, no sink
 *   3. lse_merge_with_sink       device: global LSE merge, sink applied once,
 *                                         output written in global token order
 *
 * Conventions shared by every entry point
 *   - Return value: CPMLA_OK (0) or a negative CPMLA_ERR_* code.  On error the
 *     calling thread's message is available from cpmla_last_error().  Nothing
 *     is launched when argument checks fail.
 *   - Ownership: every pointer is owned by the caller; the library never
 *     allocates, frees or retains memory.  "host" pointers are read/written
 *     during the call only; "device" pointers must be valid on the current
 *     CUDA device until the work queued on `stream` has finished.
 *   - Device entry points are asynchronous on `stream` (a cudaStream_t passed
 *     as void*, NULL = legacy default stream).  Launch errors are reported
 *     immediately as CPMLA_ERR_CUDA.  Faults detected inside a kernel (an index
 *     outside its row's causal prefix, a bounded wait that ran out) are
 *     recorded in a per-device status word read with cpmla_device_status().
 *   - Element types: bf16 = IEEE bfloat16 stored as uint16; fp8 = OCP E4M3
 *     stored as uint8; LSE values are natural-log fp32, -inf for a row with no
 *     key.
 *   - Head dims are fixed by the model family: D_qk = 576 (512 latent + 64
 *     rope, absorbed), D_v = 512 (the latent, which is also the value).
 */
#ifndef CPMLA_H
#define CPMLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  CPMLA_OK = 0,
  CPMLA_ERR_ARG = -1,         /* bad argument (null, size, alignment, range) */
  CPMLA_ERR_CUDA = -2,        /* a CUDA runtime call or launch failed */
  CPMLA_ERR_UNSUPPORTED = -3, /* valid request the library does not implement */
  CPMLA_ERR_TIMEOUT = -4,     /* status word: a bounded device wait ran out */
  CPMLA_ERR_INDEX = -5        /* status word: an index outside its row's range */
};

/* KV cache layouts. */
enum {
  /* kv: bf16 [S_kv, 576], row stride 576 elements, 16-byte aligned. */
  CPMLA_KV_BF16 = 0,
  /* kv_fp8: E4M3 latent [S_kv, 512]; kv_scale: fp32 [S_kv, 4], one scale per
   * 128 latent channels (value = e4m3 * scale); kv_rope: bf16 [S_kv, 64].
   * The pages name an fp8 MLA cache ("fp8_ds_mla") without a layout; this
   * one is the library's own.  The sparse kernel multiplies the E4M3 codes
   * (exactly as fp16) with the latent part of q rounded once to fp16: exact
   * for 2^-14 <= |q| < 65504, absolute error <= 2^-25 below that range; q
   * must stay below 65504 in magnitude.  The rope part is exact (bf16). */
  CPMLA_KV_FP8_E4M3_G128 = 1
};

#define CPMLA_DQK 576
#define CPMLA_DV 512
#define CPMLA_DROPE 64

/* Thread-local message for the last error returned on this thread ("" if none). */
const char *cpmla_last_error(void);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int cpmla_version(void);

/*
 * Reads (and, if clear != 0, resets) the device-side status word of the
 * current device: CPMLA_OK, CPMLA_ERR_INDEX or CPMLA_ERR_TIMEOUT (the first
 * fault recorded since the last reset).  Synchronises the current device.
 */
int cpmla_device_status(int *status, int clear);

/*
 * Support entry point with no counterpart on the pages: exercises the bounded
 * waits every kernel uses.  Launches one CTA on `stream` whose pipeline wait
 * is on a barrier that nothing arrives at; after limit_ms (1..2000) it gives
 * up, records CPMLA_ERR_TIMEOUT in the status word and exits normally (no
 * trap, no fault), so the CUDA context stays usable.  Read the result with
 * cpmla_device_status().  Errors: CPMLA_ERR_ARG, CPMLA_ERR_CUDA.
 */
int cpmla_selftest_wait_timeout(unsigned int limit_ms, void *stream);

/* --------------------------------------------------------------------------
 * 1. DualChunkSwap partition (host)
 *
 * "[Core] Add MRV2 virtual-batch PCP for MLA", sections "PCP algorithm" and
 * "DualChunkSwap partitioning" (PCP=4 diagram): each prefill request is cut
 * into 2P contiguous chunks and virtual shard r takes chunks r and 2P-1-r;
 * each prefill is partitioned on its own; decode rows are replicated on every
 * shard.  Where the page is silent: chunk c of an S-token request has
 * floor(S/2P) tokens plus one when c < S mod 2P; inside a shard the rows go by
 * request in input order, then chunk r before chunk 2P-1-r, ascending; a
 * replicated decode row is owned by shard 0.
 *
 * Inputs (host):
 *   P             number of virtual shards, 1..1024
 *   B             number of requests, >= 0
 *   cu_seqlens    [B+1] non-decreasing global token offsets, cu_seqlens[0]=0
 *   q_start_pos   [B] position of each request's first scheduled token
 *                 (0 for a fresh prefill; context length - 1 for a decode)
 *   is_decode     [B] 1 = decode request (replicated on all shards), else 0
 * Outputs (host, caller-allocated; sizes from pcp_partition_size):
 *   shard_offsets [P+1] shard r owns rows [shard_offsets[r], shard_offsets[r+1])
 *   rows, pos, req [n_rows_total] global token id, request-local position and
 *                 request index of each shard row (all shards concatenated)
 *   owner_shard, owner_row [T = cu_seqlens[B]] for every global token the
 *                 shard and the concatenated row index whose result is kept
 * Errors: CPMLA_ERR_ARG (null pointer, P out of range, decreasing offsets,
 * negative position, sizes beyond int32).
 * ------------------------------------------------------------------------ */
int pcp_partition_size(int P, int B, const int32_t *cu_seqlens, const uint8_t *is_decode,
                       int64_t *n_rows_total);

int pcp_dualchunk_partition(int P, int B, const int32_t *cu_seqlens, const int32_t *q_start_pos,
                            const uint8_t *is_decode, int32_t *shard_offsets, int32_t *rows,
                            int32_t *pos, int32_t *req, int32_t *owner_shard,
                            int32_t *owner_row);

/* --------------------------------------------------------------------------
 * 1b. Ratio-2 compressor linkage across chunks (host) and the gather of the
 *     linked rows (device)
 *
 * "[Feature][PCP] Add DeepSeek-V4.1-Flash support", "Overview" and
 * "Implementation": ratio-2 groups are compressed on each rank's local token
 * rows; a pair split across two PCP chunks is closed with the preceding
 * chunk's last row, and only the last (fp32) row of each local chunk is
 * gathered.  "Rank-local Compressor Revision" names the cases: PCP2/4 linkage,
 * replicated short prefills, empty ranks, request isolation and the newest
 * open ring rows.  Readings where the page is silent: a ratio-2 group is the
 * pair of request positions (2m, 2m+1); chunks are those of
 * pcp_dualchunk_partition; decode requests have no chunks and no entries.
 * The compressor's combining arithmetic is not on the pages and not here.
 *
 * pcp_ratio2_linkage_size: n_links = 2 * P * (number of prefill requests).
 * pcp_ratio2_linkage (host; inputs as for pcp_dualchunk_partition): one entry
 * per (shard r, prefill request in input order, local chunk h), shard-major,
 * h = 0 for chunk r and h = 1 for chunk 2P-1-r.  For a chunk holding request
 * positions p0 .. p1, global tokens first .. last (all [n_links], int32):
 *   first, last  the chunk's first and last global token, -1 when empty
 *   pred         global token at position p0-1 when p0 is odd and that
 *                position is in this batch (the last token of the nearest
 *                earlier non-empty chunk of the same request), else -1
 *   pred_shard   the shard holding pred, else -1
 *   flags        bit 0: p0 is odd (the pair (p0-1, p0) straddles the start);
 *                bit 1: ... and p0-1 was scheduled in an earlier step (the
 *                request's open ring row); bit 2: p1 is even (the pair (p1,
 *                p1+1) is open at the end); bit 3: ... and p1 is the
 *                request's last scheduled token (its newest open ring row)
 * Errors: CPMLA_ERR_ARG (null pointer, P outside 1..1024, decreasing offsets,
 * negative position).
 *
 * pcp_gather_rows_f32 (device): out[i, 0:D] = src[idx[i], 0:D] for
 * i < n, zeros where idx[i] == -1 -- with idx = pred, each chunk's
 * predecessor row out of the rows all shards share on one GPU (the gathered
 * last rows; with idx = last, the gathered buffer itself).
 *   src    fp32 [n_src, src_row_stride], out fp32 [n, out_row_stride]; both
 *          16-byte aligned, strides (elements) >= D and multiples of 4
 *   D      row width, a positive multiple of 4
 *   idx    int32 [n]; an index outside [-1, n_src) zeroes its row and is
 *          recorded as CPMLA_ERR_INDEX in the status word
 * Errors: CPMLA_ERR_ARG, CPMLA_ERR_CUDA.  Asynchronous on `stream`.
 * ------------------------------------------------------------------------ */
int pcp_ratio2_linkage_size(int P, int B, const int32_t *cu_seqlens, const uint8_t *is_decode,
                            int64_t *n_links);

int pcp_ratio2_linkage(int P, int B, const int32_t *cu_seqlens, const int32_t *q_start_pos,
                       const uint8_t *is_decode, int32_t *first, int32_t *last, int32_t *pred,
                       int32_t *pred_shard, int32_t *flags);

int pcp_gather_rows_f32(const float *src, int64_t src_row_stride, int64_t n_src, int D, int n,
                        const int32_t *idx, float *out, int64_t out_row_stride, void *stream);

/* --------------------------------------------------------------------------
 * 2. Per-shard partial MLA attention (device)
 *
 * "[DeepSeekV4][PCP] Enable context-parallel prefill for hybrid KV and
 * MegaMoE", "Implementation summary": each PCP rank computes local partial
 * attention and hands (output, LSE) to a global merge; "[Core] Add MRV2
 * virtual-batch PCP for MLA", "DualChunkSwap partitioning": the latent KV is
 * all-gathered so every shard sees the full KV.  No sink is applied here.
 *
 * For shard row i (global token g = rows[i], position t = pos[i], request
 * b = req[i]) and head h, with key set J_i:
 *   s_j    = softmax_scale * q[g,h,:] . kv[kv_start[b] + j, :]   (576 wide)
 *   lse    = ln sum_{j in J_i} exp(s_j)
 *   o_part = sum_{j in J_i} exp(s_j - lse) * kv[kv_start[b] + j, 0:512]
 * J_i = {0..t} (dense) or the entries >= 0 of topk_idx[g, 0..k-1] (sparse),
 * intersected with [kv_lo[i], kv_hi[i]] when those arrays are given.
 *
 * Arguments (device unless noted):
 *   q            bf16 [T, H, 576]; token g's head h starts at
 *                q + g*q_token_stride + h*576 (elements); 16-byte aligned
 *   q_token_stride  elements between tokens, >= H*576, multiple of 8 (host)
 *   H            heads, 1..128; if H > 64 it must be a multiple of 64; sparse
 *                over the fp8 cache: at most 16, or a multiple of 16 (a CTA
 *                takes 16 heads of a token); otherwise CPMLA_ERR_UNSUPPORTED
 *                (host)
 *   kv_format    CPMLA_KV_* (host).  Dense accepts CPMLA_KV_BF16 only.
 *   kv / kv_fp8, kv_scale, kv_rope   per kv_format (unused ones may be NULL);
 *                each 16-byte aligned
 *   s_kv         KV rows (host); every key read lies in [0, s_kv).  Every
 *                KV row must be finite: the sparse kernel reads row 0 in
 *                place of an empty or skipped top-k slot (weight exactly 0)
 *   kv_start     int64 [B] KV row of request b's position 0
 *   rows, pos, req  int32 [n_rows] as produced by pcp_dualchunk_partition;
 *                every rows[i] must index a token of q (and of topk_idx)
 *   n_rows       shard rows to compute (host); 0 is a no-op
 *   kv_lo, kv_hi int32 [n_rows] or NULL: inclusive position range a row may use
 *   topk_idx     int32 [T, k] (sparse) request-local key positions by global
 *                token, -1 = empty slot; an entry outside 0..t is skipped and
 *                recorded as CPMLA_ERR_INDEX in the status word
 *   k            top-k width (host), 1..65536
 *   softmax_scale  (host), finite and > 0
 *   o_part       fp32 [n_rows, H, 512] output; lse_part fp32 [n_rows, H] output
 * Errors: CPMLA_ERR_ARG, CPMLA_ERR_UNSUPPORTED, CPMLA_ERR_CUDA.
 * ------------------------------------------------------------------------ */
int mla_partial_attn_dense(const void *q, int64_t q_token_stride, int H, int kv_format,
                           const void *kv, const void *kv_fp8, const float *kv_scale,
                           const void *kv_rope, int64_t s_kv, const int64_t *kv_start,
                           const int32_t *rows, const int32_t *pos, const int32_t *req,
                           int n_rows, const int32_t *kv_lo, const int32_t *kv_hi,
                           float softmax_scale, float *o_part, float *lse_part, void *stream);

int mla_partial_attn_sparse(const void *q, int64_t q_token_stride, int H, int kv_format,
                            const void *kv, const void *kv_fp8, const float *kv_scale,
                            const void *kv_rope, int64_t s_kv, const int64_t *kv_start,
                            const int32_t *rows, const int32_t *pos, const int32_t *req,
                            int n_rows, const int32_t *kv_lo, const int32_t *kv_hi,
                            const int32_t *topk_idx, int k, float softmax_scale, float *o_part,
                            float *lse_part, void *stream);

/* --------------------------------------------------------------------------
 * 2b. Partial attention with the merge folded in (query-partitioned path)
 *
 * The pages merge per-shard partials globally, apply the sink once and
 * restore global order ("[DeepSeekV4][PCP] ...", "Implementation summary";
 * "[Core] Add MRV2 virtual-batch PCP for MLA", "DualChunkSwap partitioning").
 * When every global token has exactly one partial -- its owner shard row, as
 * after pcp_dualchunk_partition -- that merge is the identity on O and LSE, so
 * these entry points (the library's own fusion; the pages have no
 * counterpart) run the partial-attention kernels of section 2 and let the
 * owner row write the final result directly:
 *   lse_out[g,h] = LSE of the row (natural log, without the sink)
 *   o_out[g,h,:] = bf16( (O_row[h,:]) * 1 / (1 + exp(sink[h] - LSE)) )
 * with the same fp32 operations, in the same order, as the partial
 * attention followed by lse_merge_with_sink; an empty row gives O = 0,
 * LSE = -inf.  Replica rows that do not own their token (decode rows in
 * shards other than their owner) compute and write nothing, so a replicated
 * decode row is computed once; a caller that sets owner_row[g] = -1 leaves
 * token g to another call (e.g. mla_attn_split_kv).
 *
 * Arguments as in section 2, without o_part / lse_part, plus (device unless
 * noted):
 *   owner_row  int32 [T]: the shard row that owns global token g (the
 *              partition's owner_row); rows[i] = g is written only when
 *              owner_row[g] == i
 *   T          global tokens (host)
 *   sink       fp32 [H] or NULL
 *   o_out      bf16 [T, H, 512] output, 16-byte aligned (each owned token's
 *              rows are written by bulk copies); lse_out fp32 [T, H] output
 * Errors: as section 2.  A shard row whose token lies outside [0, T) is
 * skipped and recorded as CPMLA_ERR_INDEX in the status word.
 * ------------------------------------------------------------------------ */
int mla_attn_dense_merged(const void *q, int64_t q_token_stride, int H, int kv_format,
                          const void *kv, const void *kv_fp8, const float *kv_scale,
                          const void *kv_rope, int64_t s_kv, const int64_t *kv_start,
                          const int32_t *rows, const int32_t *pos, const int32_t *req,
                          int n_rows, const int32_t *kv_lo, const int32_t *kv_hi,
                          float softmax_scale, const int32_t *owner_row, int T, const float *sink,
                          void *o_out, float *lse_out, void *stream);

int mla_attn_sparse_merged(const void *q, int64_t q_token_stride, int H, int kv_format,
                           const void *kv, const void *kv_fp8, const float *kv_scale,
                           const void *kv_rope, int64_t s_kv, const int64_t *kv_start,
                           const int32_t *rows, const int32_t *pos, const int32_t *req,
                           int n_rows, const int32_t *kv_lo, const int32_t *kv_hi,
                           const int32_t *topk_idx, int k, float softmax_scale,
                           const int32_t *owner_row, int T, const float *sink, void *o_out,
                           float *lse_out, void *stream);

/* --------------------------------------------------------------------------
 * 2c. Latent KV-cache insertion (device)
 *
 * "[Core] Add MRV2 virtual-batch PCP for MLA", Summary (sparse MLA cache
 * insertion) and "DualChunkSwap partitioning" (every rank holds the
 * all-gathered latent KV it inserts into the cache); the fp8_ds_mla cache
 * dtype of "[Feature][PCP] Add DeepSeek-V4.1-Flash support".  Token t's row
 * kv[t] (bf16, 512 latent + 64 rope) goes to cache row slot_mapping[t]; a
 * slot of -1 skips the token.  The pages give no quantisation rule; this is
 * the library's own:
 *   CPMLA_KV_BF16          cache[s, :] = kv[t, :]
 *   CPMLA_KV_FP8_E4M3_G128 per 128-channel latent group g:
 *                          amax = max |kv[t, 128g .. 128g+127]|,
 *                          scale = amax / 448 in binary32 (1 if amax == 0),
 *                          cache_fp8[s, c] = E4M3(kv[t, c] / scale), the
 *                          quotient in binary32, round to nearest even,
 *                          saturating at +-448 (NaN stays NaN);
 *                          cache_scale[s, g] = scale; cache_rope[s, :] =
 *                          kv[t, 512:576]
 * so that the fp8 attention's value kv_fp8 * kv_scale is within half an E4M3
 * step of the bf16 input.
 *
 * Arguments (device unless noted):
 *   kv             bf16 [n, 576], token t at kv + t * kv_token_stride
 *                  (elements, host, >= 576, multiple of 8); 16-byte aligned
 *   n              tokens (host); 0 is a no-op
 *   slot_mapping   int64 [n]: cache row of each token, or -1
 *   kv_format      CPMLA_KV_* (host)
 *   cache          bf16 [s_cache, 576] (bf16 format), 16-byte aligned
 *   cache_fp8      uint8 [s_cache, 512], cache_scale fp32 [s_cache, 4],
 *                  cache_rope bf16 [s_cache, 64] (fp8 format); the first and
 *                  last 16-byte aligned
 *   s_cache        cache rows (host)
 * Slots must be distinct (two tokens writing one row race).  A slot outside
 * [-1, s_cache) is skipped and recorded as CPMLA_ERR_INDEX in the status word.
 * Errors: CPMLA_ERR_ARG, CPMLA_ERR_CUDA.
 * ------------------------------------------------------------------------ */
int mla_kv_cache_insert(const void *kv, int64_t kv_token_stride, int n,
                        const int64_t *slot_mapping, int kv_format, void *cache, void *cache_fp8,
                        float *cache_scale, void *cache_rope, int64_t s_cache, void *stream);

/* --------------------------------------------------------------------------
 * 2d. Top-k selection of the indexer's logits (device)
 *
 * "[Feat][NVIDIA] DeepSeek-V4.1: Prefill support CP with multistream forward
 * prepare (4/N)": the sparse attention's key lists come from the indexer,
 * whose mqa_logits step scores each query token against its request's keys
 * and whose topk_v2 step keeps the best k.  The pages give no formula for
 * either; the scores need trained indexer weights, so they are an input here
 * and this call is the selection.  For row i with m = row_len[i] candidates
 * logits[i, 0 .. m-1]:
 *   m <= k : topk_idx[i, :] = 0, 1, .., m-1, then -1
 *   m >  k : the k columns of the largest values, ordered by the IEEE total
 *            order of binary32 (-0 below +0), ties to the smaller column,
 *            written in ascending column order
 * For a request's query at position t, row_len = t + 1 gives the causal
 * prefix, and the result is the request-local topk_idx row the sparse
 * attention (2., 2b.) reads.
 *
 * Arguments (device unless noted):
 *   logits        fp32 [n_rows, logits_row_stride] (the whole extent
 *                 allocated), 16-byte aligned; never read for rows with
 *                 row_len <= k.  NaN logits leave the selection unspecified
 *                 (still k distinct in-range columns).
 *   logits_row_stride  elements between rows (host), >= max_row_len, a
 *                 multiple of 4
 *   n_rows        rows (host); 0 is a no-op
 *   row_len       int32 [n_rows], each in 0 .. max_row_len
 *   max_row_len   bound on row_len (host), 0 .. CPMLA_TOPK_MAX_ROW
 *   k             (host), 1 .. CPMLA_TOPK_MAX
 *   topk_idx      int32 [n_rows, k] output
 * A row_len outside 0 .. max_row_len writes an all -1 row and is recorded as
 * CPMLA_ERR_INDEX in the status word.  Errors: CPMLA_ERR_ARG, CPMLA_ERR_CUDA.
 * ------------------------------------------------------------------------ */
#define CPMLA_TOPK_MAX 65536
#define CPMLA_TOPK_MAX_ROW (1 << 20)
int mla_topk_select(const float *logits, int64_t logits_row_stride, int n_rows,
                    const int32_t *row_len, int max_row_len, int k, int32_t *topk_idx,
                    void *stream);

/* --------------------------------------------------------------------------
 * 2e. Split-KV attention of a list of tokens (device)
 *
 * "[Core] Add MRV2 virtual-batch PCP for MLA", "PCP algorithm": decode rows
 * are replicated on every PCP rank; "[DeepSeekV4][PCP] ...", "Implementation
 * summary": partial (output, LSE) pairs are merged by LSE and the sink is
 * applied once.  A decode row (one query over a long context or top-k list)
 * is one work item in sections 2 / 2b; here each listed token's keys are cut
 * into n_split parts, one work item each -- as if each replica of the row took
 * one part -- and the parts are merged with the sink once (the library's own
 * split; the pages give none):
 *   dense  (topk_idx == NULL): part s of a token at position t takes positions
 *          floor((t+1) s / n_split) .. floor((t+1)(s+1) / n_split) - 1
 *   sparse: part s takes entries s*ke .. (s+1)*ke - 1 of the token's top-k
 *          list, ke = ceil(k / n_split)
 * Result for token tokens[i] (natural-log LSE without the sink, as in 2b):
 *   lse_out[tokens[i], h] = ln sum over its keys of exp(s_j)
 *   o_out[tokens[i], h, :] = bf16( O * 1 / (1 + exp(sink[h] - LSE)) )
 * Nothing else of o_out / lse_out is written.
 *
 * Arguments (device unless noted): q, q_token_stride, H, kv_format, kv,
 * kv_fp8, kv_scale, kv_rope, s_kv, kv_start, softmax_scale as in section 2;
 *   tokens, pos, req  int32 [n_tokens]: global token, position in its request
 *                and request index of each listed token (e.g. the decode rows
 *                of a batch, pos = context length - 1)
 *   n_tokens     (host) >= 0; 0 is a no-op
 *   topk_idx, k  as in section 2 (indexed by global token), or NULL / 0 for
 *                dense causal attention
 *   n_split      (host) 1..64
 *   sink         fp32 [H] or NULL; T (host) tokens of o_out / lse_out
 *   o_out        bf16 [T, H, 512], lse_out fp32 [T, H] outputs (16-byte
 *                aligned); a token outside [0, T) is skipped and recorded as
 *                CPMLA_ERR_INDEX in the status word
 *   workspace    device scratch of at least
 *                mla_attn_split_kv_workspace_size(H, n_tokens, n_split) bytes,
 *                256-byte aligned, owned by the caller; it holds the parts'
 *                row arrays and their fp32 partial O and LSE (about 2 KB per
 *                part and head), and must not be in use by other work until
 *                this call's work on `stream` is done
 * Errors: CPMLA_ERR_ARG (incl. a workspace that is too small or misaligned),
 * CPMLA_ERR_UNSUPPORTED, CPMLA_ERR_CUDA.  Three launches on `stream`.
 * mla_attn_split_kv_workspace_size returns 0 for invalid sizes.
 * ------------------------------------------------------------------------ */
size_t mla_attn_split_kv_workspace_size(int H, int n_tokens, int n_split);

int mla_attn_split_kv(const void *q, int64_t q_token_stride, int H, int kv_format, const void *kv,
                      const void *kv_fp8, const float *kv_scale, const void *kv_rope, int64_t s_kv,
                      const int64_t *kv_start, const int32_t *tokens, const int32_t *pos,
                      const int32_t *req, int n_tokens, const int32_t *topk_idx, int k,
                      int n_split, float softmax_scale, const float *sink, int T, void *o_out,
                      float *lse_out, void *workspace, size_t workspace_bytes, void *stream);

/* --------------------------------------------------------------------------
 * 2f. Split-KV attention without a caller workspace (device)
 *
 * No counterpart on the pages: a convenience of this library.  The same
 * computation, arguments, results and errors as mla_attn_split_kv (2e),
 * without workspace / workspace_bytes: the parts' partial results go to a
 * fixed array of the library's own device memory, so the call allocates
 * nothing (no cudaMalloc, cudaFree or allocating library routine).  It is for
 * callers that cannot allocate device scratch -- code hosted inside a
 * framework that owns all device memory and gives it only inputs and
 * outputs, or a serving loop whose memory is fixed at start-up.
 *   - The array holds CPMLA_SPLIT_KV_STATIC_BYTES on every GPU that loads the
 *     library, until the process exits.  A call needing more scratch than
 *     that, mla_attn_split_kv_workspace_size(H, n_tokens, n_split) bytes,
 *     fails with CPMLA_ERR_ARG and says so (fewer tokens or parts per call,
 *     or use mla_attn_split_kv).
 *   - The first call on a device looks up the array's device address on that
 *     device (cudaGetSymbolAddress, with the device current); make that
 *     first call before any stream capture.
 *   - Every call on a device shares the array, which keeps the last call's
 *     contents; nothing in it has to start at zero, but calls whose work can
 *     overlap on the GPU (other streams, other host threads) race on it --
 *     order them on one stream.
 * ------------------------------------------------------------------------ */
#define CPMLA_SPLIT_KV_STATIC_BYTES (32u << 20)
int mla_attn_split_kv_noalloc(const void *q, int64_t q_token_stride, int H, int kv_format,
                              const void *kv, const void *kv_fp8, const float *kv_scale,
                              const void *kv_rope, int64_t s_kv, const int64_t *kv_start,
                              const int32_t *tokens, const int32_t *pos, const int32_t *req,
                              int n_tokens, const int32_t *topk_idx, int k, int n_split,
                              float softmax_scale, const float *sink, int T, void *o_out,
                              float *lse_out, void *stream);

/* --------------------------------------------------------------------------
 * 3. Global LSE merge + attention sink once + restore to global order (device)
 *
 * "[DeepSeekV4][PCP] ...", "Implementation summary" (merge LSE/output
 * globally, apply attn_sink only once) and "Main challenges" (attn_sink must
 * not be applied on each rank); "[Core] Add MRV2 virtual-batch PCP for MLA",
 * "DualChunkSwap partitioning" (restore to global scheduled-token order).
 * The sink is read as one extra logit per head with a zero value vector.
 *
 * For global token g and head h, with partial rows c in C_g:
 *   L   = ln sum_c exp(lse_part[c,h])
 *   O   = sum_c exp(lse_part[c,h] - L) * o_part[c,h,:]
 *   O  *= 1 / (1 + exp(sink[h] - L))          (skipped when sink == NULL)
 *   o_out[g,h,:] = bf16(O),  lse_out[g,h] = L (the sink is not folded in)
 * A token whose partials are all empty (lse = -inf) gets O = 0, L = -inf.
 *
 * Arguments (device unless noted):
 *   o_part fp32 [n_part, H, 512], 16-byte aligned; lse_part fp32 [n_part, H]
 *   n_part, H, T  sizes (host); H 1..1024
 *   contrib_off  int32 [T+1] CSR offsets into contrib_rows, or NULL meaning
 *                exactly one partial per token: C_g = {contrib_rows[g]}
 *   contrib_rows int32 partial-row indices in [0, n_part)
 *   sink         fp32 [H] or NULL
 *   o_out        bf16 [T, H, 512] output (16-byte aligned); lse_out fp32 [T, H]
 * Errors: CPMLA_ERR_ARG, CPMLA_ERR_CUDA.  A contrib row outside [0, n_part)
 * is skipped and recorded as CPMLA_ERR_INDEX in the status word.
 * ------------------------------------------------------------------------ */
int lse_merge_with_sink(const float *o_part, const float *lse_part, int64_t n_part, int H,
                        const int32_t *contrib_off, const int32_t *contrib_rows, int T,
                        const float *sink, void *o_out, float *lse_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* CPMLA_H */
