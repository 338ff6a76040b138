// Next verify width per request and the next block's layout, on the device
// ("DFlash to dLLM self-spec, part 1", section 1.3.3: one kernel produces the
// block's ids, positions and cache locations; section 1.3.2: the GPU-side
// lengths advance without a copy to the host.  "Qwen3.8-27B-FP8" page: the
// EWMA-driven DFlash2 verify width and the doubling MTP K).
//
// One warp per request.  Lane 0 applies the width policy to the request's
// accept count (the float32 steps rounded one at a time, as stated in
// spec_verify.h); lanes 0 .. q_max-1 then write one block row each.
#include "common.cuh"
#include "next_block.cuh"
#include "spec_verify.h"

namespace specv {
namespace {

constexpr int kWarps = 4;

__device__ int next_width(const NextBlockParams& p, int b, int qb, int a) {
  if (qb == 0) return 0;  // an idle request stays idle
  if (p.policy == SPEC_WIDTH_FIXED) return p.q_max;
  if (p.policy == SPEC_WIDTH_EWMA) {
    const float keep = __fsub_rn(1.0f, p.alpha);
    const float e = __fadd_rn(__fmul_rn(keep, p.state[b]),
                              __fmul_rn(p.alpha, (float)a));
    p.state[b] = e;
    const float wf = ceilf(__fadd_rn(e, p.offset));
    int w;
    if (!(wf < (float)p.q_max)) w = p.q_max;  // also NaN
    else if (wf < (float)p.min_width) w = p.min_width;
    else w = (int)wf;
    return min(max(w, 1), p.q_max);
  }
  // doubling K: x2 after a fully accepted block, /2 after a rejection
  const int kmax = max(p.q_max - 1, 1);
  int k = (int)p.state[b];
  k = a == qb - 1 ? 2 * k : k / 2;
  k = min(max(k, 1), kmax);
  p.state[b] = (float)k;
  return min(k + 1, p.q_max);
}

__global__ void __launch_bounds__(kWarps * 32)
    prepare_next_block_kernel(const NextBlockParams p) {
  // the attention call that follows may be scheduled now (it waits for
  // this grid before touching memory)
  specv::tc_grid_launch_dependents();
  const int b = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= p.batch) return;  // uniform per warp
  int w = 0;
  if (lane == 0) {
    const int qb = p.q_lens ? min(max(p.q_lens[b], 0), p.q_max) : p.q_max;
    w = next_width(p, b, qb, p.accept_len[b]);
    p.next_q_lens[b] = w;
    p.next_seq_lens[b] = p.new_seq_lens[b] + w;
  }
  w = __shfl_sync(0xffffffffu, w, 0);
  const long long pos0 = p.new_seq_lens[b];
  bool no_slot = false;
  if (lane < p.q_max) {
    const long long o = (long long)b * p.q_max + lane;
    int id = -1, pos = -1;
    long long loc = -1;
    if (lane < w) {
      const long long t = pos0 + lane;
      id = lane == 0 ? p.next_token[b] : p.mask_id;
      pos = (int)t;
      if (t >= 0 && t / p.page_size < p.max_pages) {
        const int page =
            p.page_table[(long long)b * p.max_pages + t / p.page_size];
        if (page >= 0 && page < p.num_pages)
          loc = (long long)page * p.page_size + t % p.page_size;
      }
      no_slot = loc < 0;
    }
    if (p.block_ids) p.block_ids[o] = id;
    if (p.positions) p.positions[o] = pos;
    if (p.cache_loc) p.cache_loc[o] = loc;
  }
  if (__any_sync(0xffffffffu, no_slot) && lane == 0 && p.status)
    atomicOr(p.status, SPEC_STATUS_NO_SLOT);
}

}  // namespace

cudaError_t launch_prepare_next_block(const NextBlockParams& p,
                                      cudaStream_t s) {
  if (p.batch == 0) return cudaSuccess;
  prepare_next_block_kernel<<<(p.batch + kWarps - 1) / kWarps, kWarps * 32, 0,
                              s>>>(p);
  return cudaGetLastError();
}

}  // namespace specv
