// Split-KV paged GQA verify attention, bf16 KV, warp-level tensor-core MMA
// (mma.sync m16n8k16) path, and the log-sum-exp merge kernel.
//
// One CTA walks a contiguous run of 64-token units (see common.cuh).  For a
// (request b, KV head g) piece it packs all q_len x group query rows that
// share KV head g into one tile ("MTP and DFlash2 at long context on XPU",
// Part III: folding query positions into heads, so each KV byte is read
// once), streams the piece's K/V through a cp.async double buffer gathered
// page by page from the pool, and keeps a flash-style online softmax per row
// (running max m, running sum l, rescaled output accumulator) in base 2.
// Warp w owns query rows 16w..16w+15: QK^T and PV run on mma.sync with the
// score accumulator re-packed in registers as the PV A operand.
//
// Shared-memory rows are 512 B (256 bf16); 16-byte chunk c of row r sits at
// chunk c ^ (r & 7) so that ldmatrix's eight row addresses hit distinct
// bank groups.
#include "common.cuh"

namespace specv {
namespace {

constexpr int kTile = 32;     // tokens per pipeline stage
constexpr int kStages = 2;
constexpr int kPreBytes = ((kMaxBatch + 1) * 4 + 127) / 128 * 128;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ int swz(int row, int chunk) {
  return row * 512 + ((chunk ^ (row & 7)) << 4);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src,
                                           bool valid) {
  int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zeroed
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst),
               "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi), packed in pairs.
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi,
                                           uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __low2float(h),
                                                 x1 - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

template <int kWarps>
struct Cfg {
  static constexpr int kThreads = (kWarps < 4 ? 4 : kWarps) * 32;
  static constexpr int kQRows = kWarps * 16;
  static constexpr int kSmem =
      kPreBytes + kQRows * 512 + kStages * 2 * kTile * 512;
};

// Gather one KV tile (K and V, tokens [t0, t0 + kTile) clipped to tok_end)
// of request b, KV head g into stage st.  Missing tokens and tokens on a
// page id outside the pool are zero-filled.
template <int kThreads>
__device__ __forceinline__ void load_kv_tile(const AttnParams& p, uint8_t* kv_s,
                                             int st, int b, int g, int t0,
                                             int tok_end) {
  const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(p.k_pages);
  const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(p.v_pages);
  const int ps_mask = p.page_size - 1;
#pragma unroll 4
  for (int idx = threadIdx.x; idx < 2 * kTile * 32; idx += kThreads) {
    const int is_v = idx >= kTile * 32;
    const int rem = idx - is_v * kTile * 32;
    const int row = rem >> 5, cc = rem & 31;
    const int t = t0 + row;
    bool valid = t < tok_end;
    int page = 0;
    if (valid) {
      page = __ldg(p.page_table + (long long)b * p.max_pages + (t >> p.log2_ps));
      if (page < 0 || page >= p.num_pages) {
        valid = false;
        page = 0;
        if (p.status && cc == 0) atomicOr(p.status, 1u);
      }
    }
    const long long elem =
        ((((long long)page * p.hkv + g) << p.log2_ps) + (t & ps_mask)) *
            kHeadDim + cc * 8;
    const __nv_bfloat16* src = (is_v ? vp : kp) + (valid ? elem : 0);
    uint8_t* dst = kv_s + (st * 2 + is_v) * (kTile * 512) + swz(row, cc);
    cp_async16(smem_addr(dst), src, valid);
  }
}

template <int kWarps>
__global__ void __launch_bounds__(Cfg<kWarps>::kThreads, 1)
    verify_split_bf16_kernel(const AttnParams p) {
  using C = Cfg<kWarps>;
  extern __shared__ __align__(128) uint8_t smem[];
  int* s_pre = reinterpret_cast<int*>(smem);
  uint8_t* q_s = smem + kPreBytes;
  uint8_t* kv_s = q_s + C::kQRows * 512;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mi = lane >> 3, lr = lane & 7;
  tc_grid_launch_dependents();  // the merge kernel may be scheduled now
  const int g4 = lane >> 2, t4 = lane & 3;
  // a programmatic dependent of the kernel before it on the stream: inputs
  // and outputs are touched only once that grid is complete
  tc_grid_dependency_wait();

  plan_prefix(p, s_pre);
  const Plan pl = make_plan(p, (long long)p.hkv * s_pre[p.batch]);
  const int c = blockIdx.x;  // this kernel runs static plans only
  if (c >= pl.P) return;     // uniform over the CTA
  long long u = chunk_start(pl, c);
  const long long u_end = chunk_start(pl, c + 1);

  while (u < u_end) {
    const int b = find_request(s_pre, p.batch, p.hkv, u);
    const int ntv = s_pre[b + 1] - s_pre[b];  // virtual units
    const long long rb = (long long)p.hkv * s_pre[b];
    const int g = (int)((u - rb) / ntv);
    const long long vs = rb + (long long)g * ntv;
    const int j0v = (int)(u - vs);
    const int j1v = (int)(u_end - vs < ntv ? u_end - vs : ntv);
    u = vs + j1v;
    // real units of the piece; a range of phantom units only does nothing
    const int j0 = max(j0v - p.piece_cost, 0), j1 = max(j1v - p.piece_cost, 0);
    if (j1 <= j0) continue;  // uniform over the CTA
    const int nt = ntv - p.piece_cost;
    const long long s0 = vs + p.piece_cost;  // the segment's first real unit

    const int len = clamp_len(p.seq_lens[b], p.max_tokens);
    const int qb = block_rows(p, b);
    const int tok_begin = j0 * kUnit;
    const int tok_end = min(j1 * kUnit, len);
    const int n_tiles = (tok_end - tok_begin + kTile - 1) / kTile;

    // Q rows r = i * group + j of KV head g: q[b, i, g * group + j, :]
    for (int idx = tid; idx < C::kQRows * 32; idx += C::kThreads) {
      const int r = idx >> 5, cc = idx & 31;
      const bool in_tile = r < p.rows;
      const int i = in_tile ? r / p.group : 0;
      const int h = g * p.group + (in_tile ? r - i * p.group : 0);
      const bool valid = in_tile && i < qb;   // zero-fill rows past the block
      const __nv_bfloat16* src =
          p.q + ((((long long)b * p.q_len + i) * p.hq + h) * kHeadDim + cc * 8);
      cp_async16(smem_addr(q_s + swz(r, cc)), valid ? src : p.q, valid);
    }
    load_kv_tile<C::kThreads>(p, kv_s, 0, b, g, tok_begin, tok_end);
    cp_async_commit();

    float o_acc[32][4];
#pragma unroll
    for (int n = 0; n < 32; ++n)
      o_acc[n][0] = o_acc[n][1] = o_acc[n][2] = o_acc[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const int r0 = warp * 16 + g4, r1 = r0 + 8;
    const int lim0 = causal_limit(len, qb, r0 / p.group);
    const int lim1 = causal_limit(len, qb, r1 / p.group);
    // smallest limit over the piece's rows: 0 once a row lies past the block
    const int lim_min = qb < p.q_len ? 0 : len - qb + 1;

    for (int it = 0; it < n_tiles; ++it) {
      const int t0 = tok_begin + it * kTile;
      if (it + 1 < n_tiles) {
        load_kv_tile<C::kThreads>(p, kv_s, (it + 1) & 1, b, g, t0 + kTile,
                                  tok_end);
        cp_async_commit();
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();

      if (warp < kWarps) {
        const uint8_t* k_st = kv_s + ((it & 1) * 2) * (kTile * 512);
        const uint8_t* v_st = k_st + kTile * 512;
        float s_acc[kTile / 8][4];
#pragma unroll
        for (int n = 0; n < kTile / 8; ++n)
          s_acc[n][0] = s_acc[n][1] = s_acc[n][2] = s_acc[n][3] = 0.f;
        // S = Q K^T over the 256 channels
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          uint32_t a[4];
          ldsm_x4(smem_addr(q_s + swz(warp * 16 + (mi & 1) * 8 + lr,
                                      2 * kk + (mi >> 1))), a);
#pragma unroll
          for (int np = 0; np < kTile / 16; ++np) {
            uint32_t bb[4];
            ldsm_x4(smem_addr(k_st + swz(np * 16 + (mi >> 1) * 8 + lr,
                                         2 * kk + (mi & 1))), bb);
            mma_bf16(s_acc[2 * np], a, bb[0], bb[1]);
            mma_bf16(s_acc[2 * np + 1], a, bb[2], bb[3]);
          }
        }
        // scale to base 2, causal / length mask on the block tail
        const bool need_mask = t0 + kTile > lim_min;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int n = 0; n < kTile / 8; ++n) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int tok = t0 + n * 8 + 2 * t4 + e;
            float x0 = s_acc[n][e] * p.scale_log2;
            float x1 = s_acc[n][2 + e] * p.scale_log2;
            if (need_mask) {
              if (tok >= lim0) x0 = -INFINITY;
              if (tok >= lim1) x1 = -INFINITY;
            }
            s_acc[n][e] = x0;
            s_acc[n][2 + e] = x1;
            mx0 = fmaxf(mx0, x0);
            mx1 = fmaxf(mx1, x1);
          }
        }
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float ms0 = mn0 == -INFINITY ? 0.f : mn0;
        const float ms1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = exp2f(m0 - ms0), al1 = exp2f(m1 - ms1);
        m0 = mn0;
        m1 = mn1;
        float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
        for (int n = 0; n < kTile / 8; ++n) {
          s_acc[n][0] = exp2f(s_acc[n][0] - ms0);
          s_acc[n][1] = exp2f(s_acc[n][1] - ms0);
          s_acc[n][2] = exp2f(s_acc[n][2] - ms1);
          s_acc[n][3] = exp2f(s_acc[n][3] - ms1);
          sum0 += s_acc[n][0] + s_acc[n][1];
          sum1 += s_acc[n][2] + s_acc[n][3];
        }
        l0 = l0 * al0 + sum0;
        l1 = l1 * al1 + sum1;
#pragma unroll
        for (int n = 0; n < 32; ++n) {
          o_acc[n][0] *= al0;
          o_acc[n][1] *= al0;
          o_acc[n][2] *= al1;
          o_acc[n][3] *= al1;
        }
        // O += P V with P = P_hi + P_lo, both bf16: a single bf16 P would
        // carry a 2^-9 relative error per weight, which over a few visible
        // keys is an absolute error of order 2^-9 |v| in the output.
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          uint32_t a_hi[4], a_lo[4];
          split_bf16(s_acc[2 * kk][0], s_acc[2 * kk][1], a_hi[0], a_lo[0]);
          split_bf16(s_acc[2 * kk][2], s_acc[2 * kk][3], a_hi[1], a_lo[1]);
          split_bf16(s_acc[2 * kk + 1][0], s_acc[2 * kk + 1][1], a_hi[2],
                     a_lo[2]);
          split_bf16(s_acc[2 * kk + 1][2], s_acc[2 * kk + 1][3], a_hi[3],
                     a_lo[3]);
#pragma unroll
          for (int cp = 0; cp < 16; ++cp) {
            uint32_t bb[4];
            ldsm_x4_t(smem_addr(v_st + swz(kk * 16 + (mi & 1) * 8 + lr,
                                           2 * cp + (mi >> 1))), bb);
            mma_bf16(o_acc[2 * cp], a_hi, bb[0], bb[1]);
            mma_bf16(o_acc[2 * cp + 1], a_hi, bb[2], bb[3]);
            mma_bf16(o_acc[2 * cp], a_lo, bb[0], bb[1]);
            mma_bf16(o_acc[2 * cp + 1], a_lo, bb[2], bb[3]);
          }
        }
      }
      __syncthreads();
    }

    // epilogue: direct bf16 output, or an fp32 partial for the merge
    if (warp < kWarps) {
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
      }
      const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
      const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
      const int S = seg_splits(pl, s0, nt);
      if (S == 1) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int r = half ? r1 : r0;
          if (r < p.rows) {
            const int i = r / p.group, h = g * p.group + (r - i * p.group);
            __nv_bfloat16* dst =
                p.out + (((long long)b * p.q_len + i) * p.hq + h) * kHeadDim;
            const float inv = half ? inv1 : inv0;
#pragma unroll
            for (int n = 0; n < 32; ++n) {
              __nv_bfloat162 v = __floats2bfloat162_rn(
                  o_acc[n][2 * half] * inv, o_acc[n][2 * half + 1] * inv);
              *reinterpret_cast<__nv_bfloat162*>(dst + n * 8 + 2 * t4) = v;
            }
          }
        }
      } else {
        const int k = b * p.hkv + g;
        const int slot = partial_slot(c, k);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int r = half ? r1 : r0;
          if (r < p.rows) {
            const float inv = half ? inv1 : inv0;
            float* dst = p.part_o + ((long long)slot * p.rows + r) * kHeadDim;
#pragma unroll
            for (int n = 0; n < 32; ++n) {
              float2 v = make_float2(o_acc[n][2 * half] * inv,
                                     o_acc[n][2 * half + 1] * inv);
              *reinterpret_cast<float2*>(dst + n * 8 + 2 * t4) = v;
            }
            if (t4 == 0) {
              const float l = half ? l1 : l0, m = half ? m1 : m0;
              p.part_lse[(long long)slot * p.rows + r] =
                  l > 0.f ? m + log2f(l) : -INFINITY;
            }
          }
        }
      }
    }
    // the next piece reuses q_s and the stages: every warp is done here
    __syncthreads();
  }
}

// out = sum_s 2^(lse_s - lse) o_s over the splits of a segment; segments
// with no cached token get zero rows.  Two warps per block row take
// alternate batches of kBatch splits, every load of a batch (the partial
// rows and their log-sum-exps) issued before any is used, and keep a
// running maximum over their batches (rescaling their sums when it grows),
// so no pass over the log-sum-exps has to come first: up to 2 kBatch splits
// cost one round of dependent loads.  The odd warp hands its maximum and
// sums to the even one through shared memory.  kBatch = 8 keeps the kernel
// at ~100 registers for calls with many segments and few splits each;
// kBatch = 12 (~140 registers) and 20 (~210) serve calls with few, long
// segments, whose rows are few and whose splits are many.
constexpr int kMergeRowsPerBlock = 4;
template <int kBatch>
__global__ void __launch_bounds__(256) verify_merge_kernel(const AttnParams p) {
  __shared__ int s_pre[kMaxBatch + 1];
  // a following attention call's split kernel may be scheduled now
  tc_grid_launch_dependents();
  __shared__ float s_acc[kMergeRowsPerBlock][32][10];  // the odd warp's sums
  plan_prefix(p, s_pre);
  const long long U = (long long)p.hkv * s_pre[p.batch];
  const int k = blockIdx.y, b = k / p.hkv, g = k - b * p.hkv;
  const int ntv = s_pre[b + 1] - s_pre[b];  // virtual units
  const int nt = ntv - p.piece_cost;           // real units
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pr = warp >> 1, odd = warp & 1;  // row of the block, half
  const int r = blockIdx.x * kMergeRowsPerBlock + pr;
  if (r >= p.rows) return;  // both warps of the pair
  const int i = r / p.group, h = g * p.group + (r - i * p.group);
  __nv_bfloat16* dst =
      p.out + (((long long)b * p.q_len + i) * p.hq + h) * kHeadDim + lane * 8;
  if (nt == 0) {
    if (!odd) *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    return;
  }
  const Plan pl = make_plan(p, U);
  const long long s0 =
      (long long)p.hkv * s_pre[b] + (long long)g * ntv + p.piece_cost;
  const int S = seg_splits(pl, s0, nt);
  if (S <= 1) return;
  const int base = partial_slot(chunk_of(pl, s0), k);
  // launched as a programmatic dependent of the split kernel: everything
  // above overlapped its tail; the partials are read only once it is done
  tc_grid_dependency_wait();
  const float* lse = p.part_lse + (long long)base * p.rows + r;
  const float* o = p.part_o + ((long long)base * p.rows + r) * kHeadDim + lane * 8;
  const long long stride = (long long)p.rows * kHeadDim;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float den = 0.f, mx = -INFINITY;
  for (int sb = kBatch * odd; sb < S; sb += 2 * kBatch) {
    float lv[kBatch];
    float4 x0[kBatch], x1[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int s = sb + j;
      if (s < S) {
        lv[j] = lse[(long long)s * p.rows];
        x0[j] = *reinterpret_cast<const float4*>(o + s * stride);
        x1[j] = *reinterpret_cast<const float4*>(o + s * stride + 4);
      } else {
        lv[j] = -INFINITY;
        x0[j] = x1[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float bm = lv[0];
#pragma unroll
    for (int j = 1; j < kBatch; ++j) bm = fmaxf(bm, lv[j]);
    if (bm == -INFINITY) continue;  // no split of this batch saw a key
    if (bm > mx) {  // the running maximum grows: rescale what is summed
      const float c = exp2f(mx - bm);  // 0 while nothing was summed
      den *= c;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] *= c;
      mx = bm;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const float w = exp2f(lv[j] - mx);  // 0 for an empty split
      den += w;
      acc[0] += w * x0[j].x; acc[1] += w * x0[j].y; acc[2] += w * x0[j].z;
      acc[3] += w * x0[j].w; acc[4] += w * x1[j].x; acc[5] += w * x1[j].y;
      acc[6] += w * x1[j].z; acc[7] += w * x1[j].w;
    }
  }
  // the odd warp hands its maximum and sums to the even one (named barrier
  // of the pair)
  if (odd) {
#pragma unroll
    for (int e = 0; e < 8; ++e) s_acc[pr][lane][e] = acc[e];
    s_acc[pr][lane][8] = den;
    s_acc[pr][lane][9] = mx;
  }
  asm volatile("bar.sync %0, 64;" ::"r"(1 + pr) : "memory");
  if (odd) return;
  const float m1 = s_acc[pr][lane][9];
  const float M = fmaxf(mx, m1);
  if (M != -INFINITY) {
    const float c0 = exp2f(mx - M), c1 = exp2f(m1 - M);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = acc[e] * c0 + s_acc[pr][lane][e] * c1;
    den = den * c0 + s_acc[pr][lane][8] * c1;
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint4 v;
  v.x = pack_bf16(acc[0] * inv, acc[1] * inv);
  v.y = pack_bf16(acc[2] * inv, acc[3] * inv);
  v.z = pack_bf16(acc[4] * inv, acc[5] * inv);
  v.w = pack_bf16(acc[6] * inv, acc[7] * inv);
  *reinterpret_cast<uint4*>(dst) = v;
}

template <int kWarps>
cudaError_t launch_split(const AttnParams& p, cudaStream_t s) {
  using C = Cfg<kWarps>;
  cudaError_t e = cudaFuncSetAttribute(verify_split_bf16_kernel<kWarps>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg =
      pdl_config(dim3(p.grid), dim3(C::kThreads), C::kSmem, s, attr);
  return cudaLaunchKernelEx(&cfg, verify_split_bf16_kernel<kWarps>, p);
}

template <int kWarps>
int occupancy() {
  using C = Cfg<kWarps>;
  if (cudaFuncSetAttribute(verify_split_bf16_kernel<kWarps>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kSmem) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &n, verify_split_bf16_kernel<kWarps>, C::kThreads, C::kSmem) !=
      cudaSuccess)
    return 0;
  return n;
}

}  // namespace

cudaError_t launch_verify_split_bf16(const AttnParams& p, cudaStream_t s) {
  switch ((p.rows + 15) / 16) {
    case 1: return launch_split<1>(p, s);
    case 2: return launch_split<2>(p, s);
    case 3: return launch_split<3>(p, s);
    case 4: return launch_split<4>(p, s);
    case 5: return launch_split<5>(p, s);
    case 6: return launch_split<6>(p, s);
    case 7: return launch_split<7>(p, s);
    case 8: return launch_split<8>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

int verify_split_bf16_ctas_per_sm(int rows) {
  switch ((rows + 15) / 16) {
    case 1: return occupancy<1>();
    case 2: return occupancy<2>();
    case 3: return occupancy<3>();
    case 4: return occupancy<4>();
    case 5: return occupancy<5>();
    case 6: return occupancy<6>();
    case 7: return occupancy<7>();
    case 8: return occupancy<8>();
    default: return 0;
  }
}

cudaError_t launch_verify_merge(const AttnParams& p, cudaStream_t s) {
  // a programmatic dependent launch: the merge grid may start once every
  // split CTA has begun, and waits for the split grid before its reads
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.rows + kMergeRowsPerBlock - 1) / kMergeRowsPerBlock,
                     p.batch * p.hkv);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // few (request, KV head) segments over the whole grid: each is split many
  // ways, and fewer, larger merge blocks suit it
  if ((long long)p.batch * p.hkv * 38 <= p.grid)
    return cudaLaunchKernelEx(&cfg, verify_merge_kernel<20>, p);
  if ((long long)p.batch * p.hkv * 19 <= p.grid)
    return cudaLaunchKernelEx(&cfg, verify_merge_kernel<12>, p);
  return cudaLaunchKernelEx(&cfg, verify_merge_kernel<8>, p);
}

}  // namespace specv
