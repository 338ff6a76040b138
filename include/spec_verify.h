/*
 * spec_verify.h -- C ABI of the target-verify step of speculative decoding
 * on one GB300 GPU (sm_103a).
 *
 * Two operations make up the step:
 *
 *   spec_verify_attention  multi-query paged GQA attention of each request's
 *                          verify block over its cached KV (bf16 or FP8-E4M3
 *                          with fp16 scales), split over the KV and merged by
 *                          log-sum-exp;
 *   spec_greedy_accept     per-row vocabulary argmax compared with the drafts,
 *                          giving the accepted prefix length and the bonus
 *                          token.
 *
 * Conventions shared by every entry point:
 *   - Every pointer argument except `desc`, the host-side outputs of
 *     spec_verify_status, and the returned strings is a DEVICE pointer of the
 *     current CUDA device.  The caller owns every buffer, including the
 *     workspaces; the library allocates no device memory and keeps no state
 *     between calls besides a per-device cache of the SM count (and the
 *     fixed scratch array of spec_verify_attention_noalloc, which the CUDA
 *     runtime reserves when it loads the library's GPU code on a device).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *     enqueue kernels on it: no host synchronisation, no host<->device copy
 *     (spec_verify_status excepted).  The result is visible to later work on
 *     the same stream.
 *   - Return value 0 = success.  Negative codes are detected on the host
 *     before anything is enqueued, except SPEC_ERR_CUDA, which reports a
 *     failed launch.  After a nonzero return, spec_last_error() describes it.
 *   - Argument errors never reach the GPU: a call that returns a negative
 *     code has enqueued nothing.
 */
#ifndef SPEC_VERIFY_H_
#define SPEC_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_OK 0
#define SPEC_ERR_ARG (-1)         /* null pointer, bad size or shape */
#define SPEC_ERR_ALIGN (-2)       /* pointer not aligned as documented */
#define SPEC_ERR_WORKSPACE (-3)   /* workspace missing or too small */
#define SPEC_ERR_UNSUPPORTED (-4) /* valid request this library does not run */
#define SPEC_ERR_CUDA (-5)        /* CUDA runtime error (no device, launch) */

/* Device-side status bits (see spec_verify_status). */
#define SPEC_STATUS_BAD_PAGE 1u   /* a page id outside [0, num_pages) */
#define SPEC_STATUS_TIMEOUT 2u    /* a kernel wait ran past its bound (a bug,
                                     not a data condition); output invalid */
#define SPEC_STATUS_NO_SLOT 4u    /* spec_prepare_next_block: a next-block
                                     row has no reserved cache slot */

typedef enum {
  SPEC_KV_BF16 = 0,     /* K/V elements are bf16 */
  SPEC_KV_FP8_E4M3 = 1  /* K/V elements are OCP E4M3 bytes, fp16 scales */
} spec_kv_dtype;

/* desc.flags */
#define SPEC_FLAG_CHECKED 1u  /* zero the status word, then report bad page
                                 ids through it (adds one memset) */

/*
 * Shape of a verify-attention call.
 *   batch            requests B (>= 0; 0 is a no-op)
 *   q_len            verify block rows per request, 1 + k drafts, 1..16
 *   num_q_heads      Hq; num_kv_heads Hkv; Hq % Hkv == 0.  Query head h
 *                    reads KV head h / (Hq / Hkv) (contiguous groups).
 *                    q_len * Hq / Hkv must be <= 128.
 *   head_dim         D, must be 256
 *   page_size        tokens per page, a power of two, 1..4096
 *   num_pages        pages in the pool (page ids are 0..num_pages-1)
 *   max_pages_per_seq  columns of page_table
 *   kv_dtype         spec_kv_dtype
 *   flags            SPEC_FLAG_* bits
 *   q_lens           optional DEVICE pointer, int32 [B], 4-byte aligned:
 *                    the rows request b verifies this step, its block
 *                    padded to q_len rows ("Qwen3.8-27B-FP8" page: adaptive
 *                    MTP K and the EWMA-driven DFlash2 verify width; "DFlash
 *                    to dLLM self-spec, part 1", section 1.7.2: the verify
 *                    length as a per-request scheduling decision).  Values
 *                    are clamped to [0, q_len].  Block row i < q_lens[b] is
 *                    token seq_lens[b] - q_lens[b] + i; rows past q_lens[b]
 *                    are never read, output zeros and are not appended.
 *                    NULL: every request verifies q_len rows.  Read on the
 *                    device, so it may change between graph replays.
 */
typedef struct {
  int32_t batch, q_len, num_q_heads, num_kv_heads, head_dim;
  int32_t page_size, num_pages, max_pages_per_seq;
  int32_t kv_dtype;
  uint32_t flags;
  const int32_t* q_lens;
} spec_attn_desc;

/*
 * Bytes of device workspace spec_verify_attention needs for `desc` on the
 * current device (the split count depends on the SM count).  The workspace
 * holds the split partials: per split and block row an fp32 output row and
 * an fp32 log-sum-exp, plus a 256-byte header whose first 32-bit word is
 * the status word.  Returns 0 and sets spec_last_error() on a bad desc or
 * when no CUDA device is usable.
 */
size_t spec_verify_workspace_size(const spec_attn_desc* desc);

/*
 * Verify attention.
 *
 * The verify block of request b is the last q_len tokens of its cache
 * ([boundary, d1 .. dk]); their K/V are already written to the pool.  Block
 * row i (0-based) attends causally to the first seq_lens[b] - q_len + i + 1
 * cached tokens, i.e. the committed prefix and the block up to and including
 * itself ("MTP and DFlash2 at long context on XPU", Part II "Why the target
 * output stayed the same", and Part III "Reducing an eight-query verify with
 * a severe shape cliff": each verify position is an independent query row
 * with its own cache length; "DFlash to dLLM self-spec, part 1", section
 * 1.1: verify is a short causal extend over the existing prefix KV).
 *
 *   out[b,i,h,:] = sum_t softmax_t(scale * <q[b,i,h,:], K[b,t,g,:]>) V[b,t,g,:]
 *   over t < seq_lens[b] - q_b + i + 1, g = h / (Hq/Hkv), for block rows
 *   i < q_b (q_b = desc->q_lens[b] when given, else q_len); rows i >= q_b
 *   output zeros.
 *
 * Token t of request b lives in page page_table[b, t / page_size], slot
 * t % page_size.  Pool layout [num_pages, Hkv, page_size, D] (a page holds a
 * contiguous run of page_size*D elements per KV head).
 *
 *   q         bf16 [B, q_len, Hq, D], 16-byte aligned
 *   k_pages, v_pages  bf16 or E4M3 bytes [num_pages, Hkv, page_size, D],
 *             16-byte aligned
 *   k_scales, v_scales  fp16 [num_pages, Hkv, page_size, D/64] for
 *             SPEC_KV_FP8_E4M3 (element c of a cached row is
 *             e4m3(byte_c) * scale[c/64]: "Qwen3.8-27B-FP8" page,
 *             "Implemented execution path"), 16-byte aligned; NULL for
 *             bf16.  FP8 KV is computed in fp16: dequantised K/V and Q must
 *             lie within the fp16 range (|x| <= 65504); needs page_size >= 8
 *   page_table int32 [B, max_pages_per_seq]; only the first
 *             ceil(seq_lens[b]/page_size) entries of row b are read
 *   seq_lens  int32 [B]: cached tokens of each request INCLUDING the
 *             block; values are clamped to [0, max_pages_per_seq*page_size].
 *             A row whose causal window is empty outputs zeros.
 *   scale     softmax scale (1/sqrt(D) for the pages' model), finite, > 0
 *   out       bf16 [B, q_len, Hq, D], 16-byte aligned
 *   workspace device scratch of >= spec_verify_workspace_size(desc) bytes,
 *             256-byte aligned; contents need no initialisation
 *
 * Page ids outside [0, num_pages) are never dereferenced; the rows that
 * would read them get unspecified output, and with SPEC_FLAG_CHECKED the
 * status word records SPEC_STATUS_BAD_PAGE.  The KV is split into contiguous runs of 64-token
 * tiles, one run per CTA of a fixed grid; runs that cover part of a
 * (request, KV head) produce fp32 partials (o, lse) that a second kernel
 * merges ("Qwen3.8-27B-FP8" page, "Implemented execution path": split-context
 * decode with compact online-softmax partials and a merge).
 */
int spec_verify_attention(const spec_attn_desc* desc, const void* q,
                          const void* k_pages, const void* v_pages,
                          const void* k_scales, const void* v_scales,
                          const int32_t* page_table, const int32_t* seq_lens,
                          float scale, void* out, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * Test hook for the failure path: the main-loop bound, in SM clock cycles,
 * of every mbarrier wait of the split kernels in calls made with
 * SPEC_FLAG_CHECKED.  0 (the default) restores the normal bound of about
 * two seconds (4e9 cycles), the largest value accepted.  Calls without
 * SPEC_FLAG_CHECKED always use the normal bound.
 *
 * A wait that runs past its bound is a bug, not a data condition: the CTA
 * records SPEC_STATUS_TIMEOUT in the status word, makes its other waits
 * return at once, stops issuing loads, then waits (with the normal bound)
 * for the loads, bulk stores and MMAs it already issued, frees its tensor
 * memory and exits.  The output of that call is invalid; the device and the
 * stream stay usable.  A short bound therefore lets a test make the waits
 * run out on purpose and check the status without hanging the GPU.  The
 * setting is process-wide; returns SPEC_ERR_ARG outside [0, 4e9].
 */
int spec_verify_set_wait_limit(int64_t cycles);

/*
 * Read (and optionally clear) the status word of a verify workspace.
 * Synchronises `stream`, copies 4 bytes to *status_out (host pointer).
 * Meaningful for calls made with SPEC_FLAG_CHECKED.
 */
int spec_verify_status(const void* workspace, uint32_t* status_out,
                       int32_t clear, void* stream);

/*
 * Bytes of device workspace spec_greedy_accept needs for `rows` = batch *
 * q_len logits rows of `vocab` entries (per-row, per-vocabulary-chunk
 * argmax partials, and a per-request count of finished CTAs that the call
 * zeroes itself).  Returns 0 on bad sizes.
 */
size_t spec_accept_workspace_size(int32_t rows, int32_t vocab);

/*
 * Greedy acceptance with bonus token.
 *
 * Row (b, j) of `logits` holds the target's scores for the token that
 * follows block position j.  t[b,j] = argmax over the vocabulary, lowest id
 * on ties, NaN above every number (first NaN wins), -0 == +0.  Column 0 of
 * draft_ids is the boundary token and is not compared; draft j (1..k) is
 * accepted while draft_ids[b,j] == t[b,j-1] for every earlier j
 * ("DFlash to dLLM self-spec, part 1", section 1.1, verify comparison
 * table; "MTP and DFlash2 at long context on XPU", Part II "Why the target
 * output stayed the same").
 *
 *   logits     fp32 [batch*q_len, vocab], row stride vocab, 4-byte aligned
 *              (16-byte aligned with vocab % 4 == 0 takes the vector path)
 *   draft_ids  int32 [batch, q_len]
 *   q_len      1..16;  vocab >= 1
 *   accept_len int32 [batch]: a in [0, q_len-1]
 *   next_token int32 [batch]: t[b, a], the bonus token; the request commits
 *              a + 1 tokens ("DFlash to dLLM self-spec, part 1", section
 *              1.6.1: commit_lens = accept_len + 1)
 *   out_tokens optional int32 [batch, q_len]: d1..da, next, then -1
 *   workspace  >= spec_accept_workspace_size(batch*q_len, vocab) bytes,
 *              16-byte aligned; contents need no initialisation
 */
int spec_greedy_accept(const float* logits, const int32_t* draft_ids,
                       int32_t batch, int32_t q_len, int32_t vocab,
                       int32_t* accept_len, int32_t* next_token,
                       int32_t* out_tokens, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * Greedy acceptance with per-request block widths and the cache length
 * after the commit, in the same single launch as spec_greedy_accept ("DFlash
 * to dLLM self-spec, part 1", section 1.3.3: accept, bonus and new sequence
 * lengths from one kernel; section 1.3.2: the GPU-side lengths advance
 * without a copy to the host).
 *
 * Arguments as spec_greedy_accept, with q_len the padded block width, plus:
 *   q_lens       optional int32 [batch]: rows request b verified, clamped
 *                to [0, q_len] (NULL: q_len).  Only rows j < q_b are read
 *                from `logits` (rows past it are skipped unread) and only
 *                drafts 1..q_b-1 are compared, so accept_len <= q_b - 1.
 *                A request with q_b = 0 is idle: accept_len 0, next_token
 *                -1, out_tokens all -1, new_seq_len = seq_len.
 *   seq_lens     optional int32 [batch]: cache lengths of this verify step,
 *                block included (as for spec_verify_attention)
 *   new_seq_lens optional int32 [batch], given together with seq_lens:
 *                seq_len - q_b + accept_len + 1, the cache length once the
 *                boundary token and d1..da are committed.  The bonus token
 *                is not in the cache yet: it opens the next block at that
 *                position.
 * All pointers are device pointers; nothing is copied to the host.
 */
int spec_greedy_accept_commit(const float* logits, const int32_t* draft_ids,
                              const int32_t* q_lens, int32_t batch,
                              int32_t q_len, int32_t vocab,
                              const int32_t* seq_lens, int32_t* new_seq_lens,
                              int32_t* accept_len, int32_t* next_token,
                              int32_t* out_tokens, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * Bytes of workspace spec_stochastic_accept needs (per row and 8192-entry
 * vocabulary chunk: the chunk's maximum and exponential sum; per request
 * and chunk: a draw weight).  Returns 0 on bad sizes.
 */
size_t spec_stochastic_workspace_size(int32_t batch, int32_t q_len,
                                      int32_t vocab);

/*
 * Stochastic verify: acceptance by rejection sampling against target and
 * draft probabilities ("MTP and DFlash2 at long context on XPU", Part II:
 * sampling requires rejection sampling against target and draft
 * probabilities; the rule is speculative sampling, Leviathan et al. 2023,
 * "Fast Inference from Transformers via Speculative Decoding", and Chen et
 * al. 2023).
 *
 * p_j = softmax(logits[b, j] / temperature[b]) is the target's distribution
 * for the token after block position j; q_j the distribution draft j was
 * drawn from.  For j = 1 .. q_b-1 in order, draft j is accepted iff
 *     u_accept[b, j-1] * q_j(d_j) < p_{j-1}(d_j);
 * at the first rejection the next token is drawn from the normalised
 * residual max(0, p_{j-1} - q_j) (from p_{j-1} itself when that residual is
 * zero everywhere); when every draft is accepted it is drawn from
 * p_{q_b-1}.  A draw from weights w with the uniform u = u_sample[b] is the
 * smallest token v with w(v) > 0 whose running sum w(0) + .. + w(v)
 * exceeds u * sum(w).  The committed tokens then follow the target's
 * distribution whatever the drafts.
 *
 * Arithmetic is float32 (the probabilities through exp2 of the scaled
 * logit differences, the sums over 8192-token chunks); a decision whose
 * two sides lie within float32 rounding of each other may come out
 * differently from an exact evaluation.
 *
 *   logits       fp32 [batch * q_len, vocab], finite or -inf, at least one
 *                finite entry per row that is read; vocab <= 1,048,576
 *   draft_ids    int32 [batch, q_len], column 0 the boundary token
 *   draft_probs  optional fp32 [batch, q_len - 1, vocab]: row j-1 is q_j
 *                (non-negative); NULL means greedy drafts (q_j one-hot at
 *                d_j)
 *   q_lens       optional int32 [batch] rows per request, as in
 *                spec_greedy_accept_commit (rows past q_b are not read)
 *   temperature  fp32 [batch], > 0 (a request whose temperature is not
 *                > 0 is treated as idle)
 *   u_accept     fp32 [batch, q_len - 1] uniforms in [0, 1) (may be NULL
 *                when q_len == 1); u_sample fp32 [batch] uniforms in [0, 1)
 *   seq_lens / new_seq_lens, accept_len, next_token, out_tokens  as in
 *                spec_greedy_accept_commit
 *   workspace    >= spec_stochastic_workspace_size(batch, q_len, vocab)
 *                bytes, 16-byte aligned; contents need no initialisation
 * All pointers are device pointers, 4-byte aligned; three launches on
 * `stream`, nothing copied to the host.
 */
int spec_stochastic_accept(const float* logits, const int32_t* draft_ids,
                           const float* draft_probs, const int32_t* q_lens,
                           int32_t batch, int32_t q_len, int32_t vocab,
                           const float* temperature, const float* u_accept,
                           const float* u_sample, const int32_t* seq_lens,
                           int32_t* new_seq_lens, int32_t* accept_len,
                           int32_t* next_token, int32_t* out_tokens,
                           void* workspace, size_t workspace_bytes,
                           void* stream);

/* Walks of the DFlash2 candidate selector (spec_select_desc.mode). */
#define SPEC_SELECT_GREEDY 0  /* best successor of the token already chosen */
#define SPEC_SELECT_MAP 1     /* the chain with the best total score */

/*
 * Shape of a DFlash2 candidate selection.
 *   batch      requests B
 *   positions  P: draft block rows, position 0 the verified boundary token,
 *              positions 1 .. P-1 drafted (2..16; 8 for the pages' model)
 *   vocab      V <= 262,144
 *   top        K candidates per position (1..16; 16 for the pages' model)
 *   rank       R of the codebooks, a multiple of 8 up to 256 (256 on the
 *              pages)
 *   dim        D of the draft hidden state, a multiple of 16
 *   mode       SPEC_SELECT_GREEDY or SPEC_SELECT_MAP
 */
typedef struct {
  int32_t batch, positions, vocab, top, rank, dim, mode;
} spec_select_desc;

/* Workspace bytes for spec_dflash2_select (0 on a bad desc). */
size_t spec_select_workspace_size(const spec_select_desc* desc);

/*
 * DFlash2 candidate selection: choose one draft chain from the top-K
 * candidates of every draft position through learned transition scores
 * ("MTP and DFlash2 at long context on XPU", "The part that makes DFlash2
 * different": top 16 per position, S_t(a, b) = U_t(b) + dot(A(a) * H(h_t),
 * B(b)) at rank 256, a short causal walk choosing the best successor of the
 * candidate already chosen; "Selector and recurrent math": 16 x 16 tables
 * for adjacent positions; "Qwen3.8-27B-FP8" page: an exact MAP over the
 * chain as an option).
 *
 * Position t = 1 .. P-1 keeps the K best entries of cand_logits[b, t-1]
 * (larger first, lower token id on ties).  With U_t(c) that candidate's
 * logit, H_t = W_H h_t (h_t = hidden[b, t-1]) and A, B the predecessor and
 * successor codebooks indexed by token id,
 *     S_t(a, c) = U_t(c) + sum_r A[tok(a), r] H_t[r] B[tok(c), r],
 * where a ranges over the candidates of t-1, or is the boundary token at
 * t = 1.  Greedy: c_0 = boundary, c_t = argmax_c S_t(c_{t-1}, c).  MAP: the
 * chain maximising sum_t S_t(c_{t-1}, c_t).  Ties go to the lower
 * candidate rank.  Arithmetic is float32 (bf16 inputs); a decision whose
 * best and runner-up scores lie within float32 rounding of each other may
 * come out differently from an exact evaluation.
 *
 *   cand_logits  fp32 [B, P-1, V], finite or -inf (the target head's
 *                candidate logits for each drafted position)
 *   boundary     int32 [B] token ids
 *   hidden       bf16 [B, P-1, D]; w_h bf16 [R, D] (4-byte aligned)
 *   code_a, code_b  bf16 [V, R]
 *   draft_ids    int32 [B, P] out: [boundary, c_1, .., c_{P-1}], the
 *                draft_ids layout of spec_greedy_accept
 *   cand_ids     optional int32 [B, P-1, K] out: candidate token ids in
 *                rank order (-1 past the finite entries)
 *   cand_logit   optional fp32 [B, P-1, K] out: their logits
 *   trans        optional fp32 [B, P-1, K, K] out: trans[b, t-1, a, c] =
 *                S_t(a, c); at t = 1 only a = 0 (the boundary) is defined,
 *                rows a >= 1 are -inf
 *   workspace    >= spec_select_workspace_size(desc) bytes, 256-byte
 *                aligned; contents need no initialisation
 * A counter reset and three launches on `stream`; nothing is copied to the
 * host.
 */
int spec_dflash2_select(const spec_select_desc* desc, const float* cand_logits,
                        const int32_t* boundary, const void* hidden,
                        const void* w_h, const void* code_a, const void* code_b,
                        int32_t* draft_ids, int32_t* cand_ids,
                        float* cand_logit, float* trans, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Verify width policies (spec_width_policy.policy). */
#define SPEC_WIDTH_FIXED 0     /* always q_max rows */
#define SPEC_WIDTH_EWMA 1      /* EWMA of the accepted count + offset */
#define SPEC_WIDTH_DOUBLING 2  /* K doubles on full acceptance, else halves */

/*
 * How spec_prepare_next_block picks each request's next verify width w
 * (rows, boundary included) from the accept count a of a block of q_b rows:
 *
 *   SPEC_WIDTH_FIXED     w = q_max.
 *   SPEC_WIDTH_EWMA      ("Qwen3.8-27B-FP8" page: DFlash2 adaptive width
 *                        tracks an EWMA of the accepted count and verifies
 *                        ewma + 1.5 rows with a floor of two)
 *                        e = (1 - alpha) * e + alpha * a, every operation
 *                        rounded to float32 (no fused multiply-add);
 *                        w = ceil(e + offset) clamped to [min_width, q_max].
 *                        state[b] holds e; start it at q_max - 1 for a full
 *                        first block.  Rounding up lets a fully accepted
 *                        narrow block grow again.
 *   SPEC_WIDTH_DOUBLING  ("Qwen3.8-27B-FP8" page: adaptive MTP starts at
 *                        K = 1, doubles K after full acceptance and backs
 *                        off after rejection)
 *                        K = 2K if a == q_b - 1 else K / 2 (integer),
 *                        clamped to [1, max(1, q_max - 1)]; w = min(K + 1,
 *                        q_max).  state[b] holds K as a float; start it at 1.
 */
typedef struct {
  int32_t policy;     /* SPEC_WIDTH_* */
  int32_t q_max;      /* padded block width, 1..16 */
  int32_t min_width;  /* EWMA floor, 1..q_max (2 on the page) */
  int32_t mask_id;    /* token id written into the next block's draft rows */
  float alpha;        /* EWMA weight of the newest accept count, in [0, 1] */
  float offset;       /* EWMA rows beyond the average (1.5 on the page) */
} spec_width_policy;

/*
 * After spec_greedy_accept_commit: the next verify width of every request
 * and its next block's layout, on the device ("DFlash to dLLM self-spec,
 * part 1", section 1.3.3: block ids, positions and cache loc from one
 * kernel; section 1.3.2: slots reserved ahead by KV over-allocation).
 *
 *   pol          host pointer to the policy
 *   q_lens       optional int32 [B]: rows verified this step (NULL: q_max)
 *   accept_len, next_token, new_seq_lens  int32 [B], as produced by
 *                spec_greedy_accept_commit
 *   state        float [B], read and updated (EWMA value or K); may be NULL
 *                for SPEC_WIDTH_FIXED
 *   page_table   int32 [B, max_pages_per_seq]: the request's reserved pages
 *   next_q_lens  int32 [B] out: w (0 for an idle request, q_b = 0)
 *   next_seq_lens int32 [B] out: new_seq_len + w, the seq_lens of the next
 *                verify step
 *   block_ids    optional int32 [B, q_max] out: [next_token, mask_id x
 *                (w - 1), -1 ...]
 *   positions    optional int32 [B, q_max] out: new_seq_len + i for i < w,
 *                else -1
 *   cache_loc    optional int64 [B, q_max] out: page * page_size + slot of
 *                position new_seq_len + i, or -1 for i >= w and for a slot
 *                that is not reserved (past the table, page id outside the
 *                pool)
 *   status       optional device uint32: SPEC_STATUS_NO_SLOT is OR-ed in
 *                when a row i < w has no reserved slot (never cleared here;
 *                read it with spec_verify_status)
 * int32 / float buffers 4-byte aligned, cache_loc 8-byte aligned.  Host
 * checks return SPEC_ERR_ARG / SPEC_ERR_ALIGN before anything is enqueued.
 */
int spec_prepare_next_block(const spec_width_policy* pol, int32_t batch,
                            const int32_t* q_lens, const int32_t* accept_len,
                            const int32_t* next_token,
                            const int32_t* new_seq_lens, float* state,
                            const int32_t* page_table,
                            int32_t max_pages_per_seq, int32_t page_size,
                            int32_t num_pages, int32_t* next_q_lens,
                            int32_t* next_seq_lens, int32_t* block_ids,
                            int32_t* positions, int64_t* cache_loc,
                            uint32_t* status, void* stream);

/*
 * Verify attention without a caller workspace, for callers that cannot
 * allocate device memory (no cudaMalloc and no pool of their own: e.g. code
 * handed only the input and output buffers of an engine that owns all device
 * memory).  The pages have no counterpart of this entry point; it is an
 * addition of this library.
 *
 * Arguments, layouts, results and errors are those of spec_verify_attention,
 * minus the workspace.  The split partials live instead in a fixed device
 * array of SPEC_NOALLOC_SCRATCH_BYTES inside the library, reserved on every
 * GPU that loads the library until the process exits; the call allocates
 * nothing.
 *   - A shape whose workspace (spec_verify_workspace_size) exceeds
 *     SPEC_NOALLOC_SCRATCH_BYTES is rejected with SPEC_ERR_WORKSPACE.
 *   - SPEC_FLAG_CHECKED is rejected with SPEC_ERR_UNSUPPORTED (its status
 *     word lives in a caller workspace).
 *   - The array's device address is looked up (cudaGetSymbolAddress) on
 *     the first call in each CUDA context and cached under that context's
 *     process-unique id, so a caller that runs in a driver context of its
 *     own, and the new primary context after a device reset, each get their
 *     own lookup, never a stale address.  The first call in a context may
 *     load the library's GPU code there; make it before any stream capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; nothing in it needs to start at zero.  Calls whose kernels
 *     overlap on the GPU (on different streams, or from different threads)
 *     race on it: order them on one stream, or give each its own workspace
 *     through spec_verify_attention.
 */
#define SPEC_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int spec_verify_attention_noalloc(const spec_attn_desc* desc, const void* q,
                                  const void* k_pages, const void* v_pages,
                                  const void* k_scales, const void* v_scales,
                                  const int32_t* page_table,
                                  const int32_t* seq_lens, float scale,
                                  void* out, void* stream);

/*
 * Append each request's verify block to its paged KV cache.
 *
 * Block row i < q_b of request b is token t = seq_lens[b] - q_b + i
 * (seq_lens includes the block, as for spec_verify_attention; q_b =
 * desc->q_lens[b] when given, else q_len); its K and V rows of
 * every KV head go to page page_table[b, t / page_size], slot
 * t % page_size.  The pages' serving stacks reserve those slots ahead of
 * the verify pass and hand the kernels the block's positions and cache
 * locations ("DFlash to dLLM self-spec, part 1", section 1.3.2 "KV
 * over-allocation", and section 1.3.3: one kernel producing block ids,
 * positions and cache loc); this call writes the rows and those two index
 * arrays in one launch.
 *
 * bf16 pool (desc->kv_dtype == SPEC_KV_BF16): the rows are copied.
 * FP8 pool: each 64-channel block of a row is quantised on write ("Qwen3.8-
 * 27B-FP8" page, "Implemented execution path": E4M3 cache with per-token /
 * per-KV-head FP16 scales over 64-channel blocks), with this library's rule
 * (the pages fix only the format):
 *   amax  = max |x| over the block (x the bf16 input, as fp32)
 *   scale = fp16_rn(amax / 448), the division in fp32 round-to-nearest;
 *           1 if that rounds to zero
 *   byte  = E4M3 of fp32 x / scale, round-to-nearest-even, saturated to
 *           +-448 (inputs must be finite)
 *
 *   k_new, v_new  bf16 [B, q_len, Hkv, D], 16-byte aligned
 *   k_pages, v_pages, k_scales, v_scales  the pool, as in
 *                 spec_verify_attention (scales only for FP8)
 *   page_table, seq_lens  as in spec_verify_attention
 *   positions     optional int32 [B, q_len]: t (or -1 where t < 0 or
 *                 i >= q_b)
 *   cache_loc     optional int64 [B, q_len]: page * page_size + slot, the
 *                 flat token slot in the pool (or -1 where the token has no
 *                 slot: i >= q_b, t < 0, t beyond the table, or a page id outside the
 *                 pool; such rows are not written, and SPEC_FLAG_CHECKED
 *                 reports a bad page id through spec_verify_status on
 *                 `workspace`)
 *   workspace     only used with SPEC_FLAG_CHECKED (its status word);
 *                 NULL otherwise
 */
int spec_kv_append(const spec_attn_desc* desc, const void* k_new,
                   const void* v_new, void* k_pages, void* v_pages,
                   void* k_scales, void* v_scales, const int32_t* page_table,
                   const int32_t* seq_lens, int32_t* positions,
                   int64_t* cache_loc, void* workspace, void* stream);

/* Message for the last nonzero return on this thread ("" if none). */
const char* spec_last_error(void);

/* Library version string. */
const char* spec_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H_ */
