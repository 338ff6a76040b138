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
#define SPEC_ERR_UNSUPPORTED (-4) /* valid request this build does not run */
#define SPEC_ERR_CUDA (-5)        /* CUDA runtime error (no device, launch) */

/* Device-side status bits (see spec_verify_status). */
#define SPEC_STATUS_BAD_PAGE 1u   /* a page id outside [0, num_pages) */
#define SPEC_STATUS_TIMEOUT 2u    /* a kernel wait ran past its bound (a bug,
                                     not a data condition); output invalid */

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
 */
typedef struct {
  int32_t batch, q_len, num_q_heads, num_kv_heads, head_dim;
  int32_t page_size, num_pages, max_pages_per_seq;
  int32_t kv_dtype;
  uint32_t flags;
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
 *   over t < seq_lens[b] - q_len + i + 1, g = h / (Hq/Hkv).
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
 * Read (and optionally clear) the status word of a verify workspace.
 * Synchronises `stream`, copies 4 bytes to *status_out (host pointer).
 * Meaningful for calls made with SPEC_FLAG_CHECKED.
 */
int spec_verify_status(const void* workspace, uint32_t* status_out,
                       int32_t clear, void* stream);

/*
 * Bytes of device workspace spec_greedy_accept needs for `rows` = batch *
 * q_len logits rows of `vocab` entries (per-row, per-vocabulary-chunk
 * argmax partials).  Returns 0 on bad sizes.
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
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, which may load the library's GPU code on that
 *     device); make that first call before any stream capture.
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
 * Block row i of request b is token t = seq_lens[b] - q_len + i (seq_lens
 * includes the block, as for spec_verify_attention); its K and V rows of
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
 *   positions     optional int32 [B, q_len]: t (or -1 where t < 0)
 *   cache_loc     optional int64 [B, q_len]: page * page_size + slot, the
 *                 flat token slot in the pool (or -1 where the token has no
 *                 slot: t < 0, t beyond the table, or a page id outside the
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
