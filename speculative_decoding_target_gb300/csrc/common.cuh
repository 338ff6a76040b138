// Internal definitions shared by the verify-attention kernels and the C ABI.
//
// Work plan of the split-KV verify attention.  The KV of every (request b,
// KV head g) pair -- a "segment" -- is cut into 64-token units.  Segments are
// laid end to end in (b, g) order, giving U units in total; CTA c of the
// fixed grid of P CTAs takes the contiguous unit range ("chunk")
// [floor(c*U/P), floor((c+1)*U/P)), where P is the launched grid capped so
// that no chunk is empty.  A segment touched by several chunks is "split":
// each touching chunk writes an fp32 partial (normalised output row and
// base-2 log-sum-exp per block row) into its own slot and the merge kernel
// combines them ("Qwen3.8-27B-FP8" page, "Implemented execution path":
// split-context decode with compact online-softmax partials and a merge).
// A segment inside one chunk is written straight to the output.  Every
// kernel derives the same plan from seq_lens on the device, so the grid
// never depends on host-side lengths and the launch is graph-capturable.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace specv {

constexpr int kHeadDim = 256;
constexpr int kUnit = 64;        // tokens per plan unit
constexpr int kMaxRows = 128;    // q_len * group rows of one KV head
constexpr int kMaxBatch = 1024;  // requests per call (shared-memory prefix)
constexpr int kWsHeader = 256;   // bytes; word 0 = status

struct AttnParams {
  const __nv_bfloat16* q;
  const void* k_pages;
  const void* v_pages;
  const __half* k_scales;
  const __half* v_scales;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* q_lens;  // optional [B]: rows of each block (<= q_len)
  __nv_bfloat16* out;
  float* part_o;      // [nslots, rows, 256]
  float* part_lse;    // [nslots, rows] (base 2)
  uint32_t* status;   // workspace word 0
  int batch, q_len, hq, hkv, group, rows;
  int page_size, log2_ps, num_pages, max_pages;
  int max_tokens;     // max_pages * page_size: seq_lens clamp
  int grid;           // P: CTAs of the split kernel
  int piece_cost;     // plan units charged per segment (<= kMaxPieceCost)
  int box_rows;       // TMA box height (tcgen05 kernel): min(page_size, 64)
  float scale_log2;   // softmax scale * log2(e)
  // clock cycles a main-loop wait of the split kernels may last before the
  // CTA gives up (sets SPEC_STATUS_TIMEOUT and drains); the teardown's
  // drain of copies and MMAs already issued always uses kDrainWaitCycles
  long long wait_cycles;
};
constexpr long long kDrainWaitCycles = 4000000000LL;  // about two seconds

__device__ __forceinline__ int clamp_len(int len, int cap) {
  return len < 0 ? 0 : (len > cap ? cap : len);
}

// Rows of request b's verify block: q_lens[b] clamped to [0, q_len], or
// q_len.  Block row i < rows is token seq_len - rows + i; the rows past it
// do not exist and get an empty causal window (zero output).
__device__ __forceinline__ int block_rows(const AttnParams& p, int b) {
  return p.q_lens ? clamp_len(p.q_lens[b], p.q_len) : p.q_len;
}

// Keys visible to block row i of a request with len cached tokens and qb
// block rows.
__device__ __forceinline__ int causal_limit(int len, int qb, int i) {
  return i < qb ? len - qb + i + 1 : 0;
}

__device__ __forceinline__ int units_of(int len) {
  return (len + kUnit - 1) / kUnit;
}

// The plan runs on virtual units: every (request, KV head) segment is
// charged piece_cost units in front of its real ones, the fixed cost of a
// piece (loading Q, the pipeline's fill and drain, the epilogue) in 64-token
// units of that kernel's streaming time.  Every CTA pays for its first
// piece; a CTA that crosses into a new segment pays for one more, and the
// charge at the segment's start bills exactly those.  CTAs split the virtual
// units evenly and process the real units in their range, so a CTA that
// starts a segment owns fewer real units.  In virtual units segment (b, g)
// starts at hkv s_pre[b] + g nt'_b and its real units at piece_cost beyond
// that, nt'_b = s_pre[b+1] - s_pre[b].  Each kernel's cost was measured as
// the time a piece boundary adds (clock64 timelines, and calls on equal
// total KV cut into more or fewer segments).
constexpr int kMaxPieceCost = 16;
constexpr int kTcPieceCost = 3;     // bf16/FP8 tcgen05 kernel, Q in TMEM
constexpr int kFp8tPieceCost = 10;  // FP8 kernel with K and V^T in TMEM
constexpr int kMmaPieceCost = 3;    // mma.sync kernel (bf16, small pages)

struct Plan {
  long long U;  // virtual units
  int P;        // chunks = CTAs that run
};

// First unit of chunk c (0 <= c <= P).
__device__ __forceinline__ long long chunk_start(const Plan& pl, int c) {
  return (long long)c * pl.U / pl.P;
}

// Chunk whose range holds unit u (0 <= u < U).
__device__ __forceinline__ int chunk_of(const Plan& pl, long long u) {
  return (int)(((u + 1) * (long long)pl.P - 1) / pl.U);
}

// Number of chunks that touch a segment starting at unit s0 with nt units.
__device__ __forceinline__ int seg_splits(const Plan& pl, long long s0, int nt) {
  if (nt <= 0) return 0;
  return chunk_of(pl, s0 + nt - 1) - chunk_of(pl, s0) + 1;
}

// Exclusive prefix of virtual units per request (real units + piece_cost)
// into s_pre[0..batch] (s_pre[0] = 0).  Called by the whole block; ends
// with __syncthreads().
__device__ __forceinline__ void plan_prefix(const AttnParams& p, int* s_pre) {
  const int tid = threadIdx.x;
  if (tid < 32) {
    int carry = 0;
    const int lane = tid;
    for (int base = 0; base < p.batch; base += 32) {
      int b = base + lane;
      int v = b < p.batch
                  ? units_of(clamp_len(p.seq_lens[b], p.max_tokens)) + p.piece_cost
                  : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
      }
      if (b < p.batch) s_pre[b + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) s_pre[0] = 0;
  }
  __syncthreads();
}

// Effective grid: the launched grid, capped so that every CTA owns at least
// kMinUnitsPerCta units (a small workload cut finer would write more split
// partials than it saves in parallel reads).  Every CTA below it owns at
// least one unit, so consecutive CTAs of a segment have consecutive ids.
constexpr int kMinUnitsPerCta = 3;
__device__ __forceinline__ int effective_grid(int grid, long long U) {
  const long long want = (U + kMinUnitsPerCta - 1) / kMinUnitsPerCta;
  return want < grid ? (int)want : grid;
}

__device__ __forceinline__ Plan make_plan(const AttnParams& p, long long U) {
  Plan pl;
  pl.U = U;
  pl.P = effective_grid(p.grid, U);
  return pl;
}

// Partial slot of segment k's piece in chunk ch: ch + k.  Chunks are
// monotone along the unit line and segment k + 1 lies after segment k, so
// a later segment never touches an earlier chunk: two (segment, chunk)
// pairs with the same sum would need k1 < k2 and ch1 > ch2, which cannot
// both touch.  The slots are distinct, those of one segment consecutive
// (from chunk_of(its first unit) + k), and all below chunks + segments.
__device__ __forceinline__ int partial_slot(int chunk, int k) {
  return chunk + k;
}

// Request owning unit u: the largest b with hkv * s_pre[b] <= u.
__device__ __forceinline__ int find_request(const int* s_pre, int batch,
                                            int hkv, long long u) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if ((long long)hkv * s_pre[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Programmatic dependent launch: a primary grid lets its dependent grid be
// scheduled; the dependent waits until the primary grid has completed and
// its memory operations are visible.
__device__ __forceinline__ void tc_grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void tc_grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launch configuration of a programmatic dependent launch: the grid may be
// scheduled while the kernel before it on the stream runs (once that one
// has executed griddepcontrol.launch_dependents in every CTA, or exited),
// and waits for it with griddepcontrol.wait before touching memory that
// kernel writes or reads.  `attr` must outlive the launch call.
inline cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t s, cudaLaunchAttribute* attr) {
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Record an error message for spec_last_error() and return `code`.
int set_error(int code, const char* fmt, ...);

// Launchers (defined in the kernel translation units).
cudaError_t launch_verify_split_bf16(const AttnParams& p, cudaStream_t s);
cudaError_t launch_verify_merge(const AttnParams& p, cudaStream_t s);
int verify_split_bf16_ctas_per_sm(int rows);
cudaError_t launch_verify_split_tc(const AttnParams& p, const CUtensorMap& tm_k,
                                   const CUtensorMap& tm_v, cudaStream_t s);
int verify_split_tc_ctas_per_sm(bool fp8);
int verify_split_tc_box_rows(int page_size);
// FP8 KV with at most kFp8tMaxRows block rows per KV head: the kernel with
// K and V^T as tensor-memory operands (tensor maps over the byte pools with
// boxes of 128 bytes x box_rows rows).
constexpr int kFp8tMaxRows = 64;
cudaError_t launch_verify_split_fp8t(const AttnParams& p,
                                     const CUtensorMap& tm_k,
                                     const CUtensorMap& tm_v, cudaStream_t s);
int verify_split_fp8t_ctas_per_sm();
// The tcgen05 kernel loads whole 8-row swizzle groups (and, for FP8 KV,
// 16-byte multiples of the scales) per page run, so it needs pages of at
// least 8 tokens; smaller bf16 pages take the mma.sync kernel.
constexpr int kTcMinPageSize = 8;

}  // namespace specv
