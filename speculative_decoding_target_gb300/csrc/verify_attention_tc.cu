// Split-KV paged GQA verify attention on the 5th-generation tensor cores
// (tcgen05 MMA with TMEM accumulators, TMA tile loads), bf16 KV.
//
// One CTA per SM walks its contiguous run of 64-token units (the plan in
// common.cuh).  For every (request b, KV head g) piece of the run, all
// q_len x group query rows that read KV head g form the M = 128 rows of one
// MMA tile ("MTP and DFlash2 at long context on XPU", Part III: the query
// positions of a verify block folded into the head dimension, so every KV
// byte is read once).  Query row r sits at TMEM lane 32*(r / R) + r % R,
// R = ceil(rows / 4), which spreads the rows over the four TMEM lane
// quarters; the other lanes carry zero rows.
//
// Warp roles (192 threads):
//   warp 0      TMA producer (all 32 lanes): gathers each 64-token K and V
//               tile of the piece page by page from the pool (one 2-D box of
//               64 channels x min(page_size, 64) tokens per column block,
//               lane i issuing box i) into a 2-stage ring.
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//               S buffers and O += P_j V_j into the TMEM O accumulator, each
//               issued as soon as its inputs are ready.
//   warps 2..5  softmax: one thread per TMEM lane (query row).  Load S_j,
//               mask the block's causal tail, keep a running max m and sum l
//               in base 2, and write P_j = 2^(s - m) back over S_j as bf16
//               hi + lo parts (the PV MMA takes P from TMEM and runs once per
//               part, so the bf16 rounding of P does not reach the output);
//               rescale O in TMEM only when the running max grows by more
//               than 2^8; finally read O, divide by l and write the bf16
//               output or an fp32 partial.
//
// The tile width is set by the MMA issue rate: QK^T costs 16 instructions
// per tile whatever its width, so 64-token tiles halve the instructions per
// KV byte of 32-token tiles.
//
// Every wait is bounded (about two seconds of clock); a wait that runs out
// sets SPEC_STATUS_TIMEOUT in the status word (checked mode) and makes every
// later wait of the CTA return at once, so the kernel always finishes.
#include "common.cuh"
#include "spec_verify.h"
#include "tc_ptx.cuh"

namespace specv {
namespace {

constexpr int kT = 64;                        // tokens per tile
constexpr int kStages = 2;
constexpr int kThreads = 192;
constexpr int kQBytes = 4 * 128 * 128;        // Q: 4 column blocks x 128 rows
constexpr int kHalfBytes = 4 * kT * 128;      // K (or V) of one stage
constexpr int kStageBytes = 2 * kHalfBytes;
constexpr int kOffKV = kQBytes;
constexpr int kOffPre = kOffKV + kStages * kStageBytes;
constexpr int kPreBytes = ((kMaxBatch + 1) * 4 + 127) / 128 * 128;
constexpr int kSmemBytes = kOffPre + kPreBytes + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 256;               // S/P buffers: columns 256, 320
constexpr long long kWaitCycles = 4000000000LL;
constexpr float kRescaleLog2 = 8.0f;          // rescale O when m grows > 2^8

constexpr uint32_t kIdescQK = tc::idesc_bf16(128, kT, 0);
constexpr uint32_t kIdescPV = tc::idesc_bf16(128, 256, 1);

struct Bars {
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t drain;
};

struct Ctx {
  Bars* bars;
  volatile int* abort;
  const AttnParams* p;
};

// Bounded wait on phase `parity` of an mbarrier.  Returns false (and flags
// the CTA) when the bound runs out or another wait of the CTA already did.
__device__ __noinline__ bool wait_slow(uint32_t a, uint32_t parity,
                                       volatile int* abort, uint32_t* status,
                                       bool ignore_abort) {
  if (!ignore_abort && *abort) return false;
  const long long t0 = clock64();
  while (true) {
    if (tc::bar_try_wait(a, parity)) return true;
    if (!ignore_abort && *abort) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort = 1;
      if (status) atomicOr(status, SPEC_STATUS_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_bar(const Ctx& cx, uint64_t* bar,
                                         uint32_t parity,
                                         bool ignore_abort = false) {
  const uint32_t a = tc::smem_u32(bar);
  if (tc::bar_try_wait(a, parity)) return true;
  return wait_slow(a, parity, cx.abort, cx.p->status, ignore_abort);
}

struct Piece {
  int b, g, nt, len, tok_begin, tok_end, n_tiles;
  long long s0;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

// ---- warp 0: TMA loads of the piece's K/V tiles ----------------------------
// Lane i owns box i of a tile (a run of min(page_size, 64) tokens of one
// page); its page id for the next tile is loaded while the current tile
// waits for a free stage, so the page-table latency stays off the pipeline.
__device__ __forceinline__ int box_page(const AttnParams& p, const Piece& pc,
                                        int jt, int lane) {
  const int t = pc.tok_begin + jt * kT + lane * p.box_rows;
  if (jt >= pc.n_tiles || t >= pc.tok_end || lane * p.box_rows >= kT) return 0;
  int page = __ldg(p.page_table + (long long)pc.b * p.max_pages +
                   (t >> p.log2_ps));
  if (page < 0 || page >= p.num_pages) {
    if (p.status) atomicOr(p.status, SPEC_STATUS_BAD_PAGE);
    page = 0;  // in bounds; the affected rows are unspecified
  }
  return page;
}

__device__ void produce(const Ctx& cx, const Piece& pc, int gj0, uint8_t* kv,
                        const CUtensorMap* tm_k, const CUtensorMap* tm_v) {
  const AttnParams& p = *cx.p;
  const int lane = threadIdx.x & 31;
  const int rpb = p.box_rows;
  int page = box_page(p, pc, 0, lane);
  for (int jt = 0; jt < pc.n_tiles; ++jt) {
    const int next_page = box_page(p, pc, jt + 1, lane);
    const int gj = gj0 + jt, st = gj % kStages;
    if (gj >= kStages)
      wait_bar(cx, &cx.bars->kv_empty[st], ((gj / kStages) - 1) & 1);
    const int t0 = pc.tok_begin + jt * kT;
    const int ntok = min(kT, pc.tok_end - t0);
    const int nbox = (ntok + rpb - 1) / rpb;
    const uint32_t full = tc::smem_u32(&cx.bars->kv_full[st]);
    if (lane == 0)
      tc::bar_arrive_expect_tx(full, (uint32_t)(nbox * rpb * 128 * 4 * 2));
    __syncwarp();
    if (lane < nbox) {
      const uint32_t kdst = tc::smem_u32(kv + st * kStageBytes);
      const uint32_t vdst = kdst + kHalfBytes;
      const int t = t0 + lane * rpb;
      const int y = ((page * p.hkv + pc.g) << p.log2_ps) + (t & (p.page_size - 1));
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        const uint32_t off = cb * (kT * 128) + lane * rpb * 128;
        tc::tma_load_2d(kdst + off, tm_k, full, cb * 64, y);
        tc::tma_load_2d(vdst + off, tm_v, full, cb * 64, y);
      }
    }
    page = next_page;
  }
}

// ---- warp 1, one thread: MMA issue -------------------------------------------
// S_j = Q K_j^T and O += P_j V_j are issued as soon as their inputs are
// ready, whichever comes first: a PV never waits behind the next tile's TMA.
__device__ __forceinline__ void issue_qk(const Ctx& cx, int gj, uint32_t tmem,
                                         uint8_t* smem) {
  const int st = gj % kStages;
  const uint32_t qbase = tc::smem_u32(smem);
  const uint32_t kbase = tc::smem_u32(smem + kOffKV + st * kStageBytes);
  const uint32_t d = tmem + kColS + (gj & 1) * kT;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint64_t ad = tc::desc_sw128(qbase + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024);
    const uint64_t bd = tc::desc_sw128(kbase + (k >> 2) * (kT * 128) + (k & 3) * 32, 16, 1024);
    tc::mma_bf16(d, ad, bd, kIdescQK, k > 0 ? 1u : 0u);
  }
  tc::commit(tc::smem_u32(&cx.bars->s_full[gj & 1]));
}

__device__ __forceinline__ void issue_pv(const Ctx& cx, int gj, bool first,
                                         uint32_t tmem, uint8_t* smem) {
  const int st = gj % kStages;
  const uint32_t vbase = tc::smem_u32(smem + kOffKV + st * kStageBytes) + kHalfBytes;
  const uint32_t p_hi = tmem + kColS + (gj & 1) * kT;  // 32 columns: bf16 pairs
  const uint32_t p_lo = p_hi + kT / 2;
#pragma unroll
  for (int kk = 0; kk < kT / 16; ++kk) {
    const uint64_t bd = tc::desc_sw128(vbase + kk * 2048, kT * 128, 1024);
    tc::mma_bf16_ta(tmem, p_hi + kk * 8, bd, kIdescPV,
                    (first && kk == 0) ? 0u : 1u);
    tc::mma_bf16_ta(tmem, p_lo + kk * 8, bd, kIdescPV, 1u);
  }
  tc::commit(tc::smem_u32(&cx.bars->kv_empty[st]));
  tc::commit(tc::smem_u32(&cx.bars->pv_done[gj & 1]));
}

__device__ void mma_piece(const Ctx& cx, const Piece& pc, int gj0, uint32_t tmem,
                          uint8_t* smem) {
  int qk = 0, pv = 0;
  long long last = clock64();
  while (pv < pc.n_tiles) {
    bool did = false;
    if (qk < pc.n_tiles) {
      const int gj = gj0 + qk;
      if (tc::bar_try_wait(tc::smem_u32(&cx.bars->kv_full[gj % kStages]),
                           (gj / kStages) & 1) &&
          (gj < 2 || tc::bar_try_wait(tc::smem_u32(&cx.bars->pv_done[gj & 1]),
                                      ((gj >> 1) - 1) & 1))) {
        tc::fence_after();
        issue_qk(cx, gj, tmem, smem);
        ++qk;
        did = true;
      }
    }
    if (pv < qk) {
      const int gj = gj0 + pv;
      if (tc::bar_try_wait(tc::smem_u32(&cx.bars->p_full[gj & 1]),
                           (gj >> 1) & 1)) {
        tc::fence_after();
        issue_pv(cx, gj, pv == 0, tmem, smem);
        ++pv;
        did = true;
      }
    }
    if (did) {
      last = clock64();
    } else if (*cx.abort) {
      break;
    } else if (clock64() - last > kWaitCycles) {
      *cx.abort = 1;
      if (cx.p->status) atomicOr(cx.p->status, SPEC_STATUS_TIMEOUT);
      break;
    }
  }
}

// ---- warps 2..5: softmax and epilogue ----------------------------------------
__device__ void softmax_piece(const Ctx& cx, const Piece& pc, int gj0,
                              uint32_t tmem, uint8_t* smem, const int* s_pre,
                              long long U, int P, int c) {
  const AttnParams& p = *cx.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w4 = warp & 3, pos = 32 * w4 + lane;
  const int R = (p.rows + 3) >> 2;
  const int r = w4 * R + lane;
  const bool valid = lane < R && r < p.rows;
  const int i = valid ? r / p.group : 0;
  const int lim = pc.len - p.q_len + i + 1;
  const uint32_t lane_base = tmem + ((uint32_t)(32 * w4) << 16);
  const float sl2 = p.scale_log2;

  float m = -INFINITY, l = 0.f;
  for (int jt = 0; jt < pc.n_tiles; ++jt) {
    const int gj = gj0 + jt;
    const uint32_t sbuf = lane_base + kColS + (gj & 1) * kT;
    wait_bar(cx, &cx.bars->s_full[gj & 1], (gj >> 1) & 1);
    tc::fence_after();
    float s[kT];
    tc::tmem_ld32(sbuf, s);
    tc::tmem_ld32(sbuf + 32, s + 32);

    const int t0 = pc.tok_begin + jt * kT;
    if (t0 + kT > lim) {  // the causal tail of the block reaches this tile
#pragma unroll
      for (int k = 0; k < kT; ++k)
        if (t0 + k >= lim) s[k] = -INFINITY;
    }
    float mx4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
    for (int k = 4; k < kT; ++k) mx4[k & 3] = fmaxf(mx4[k & 3], s[k]);
    // scale > 0, so the max of the raw scores gives the max of the scaled
    const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * sl2;
    bool need = false;
    float alpha = 1.f;
    if (jt == 0) {
      m = mx;
    } else if (m != -INFINITY) {
      const float mn = fmaxf(m, mx);
      if (mn > m + kRescaleLog2) {
        need = true;
        alpha = exp2f(m - mn);
        m = mn;
      }
    }
    if (__any_sync(0xffffffffu, need)) {
      // O must be final for tile gj-1 before it is rescaled
      wait_bar(cx, &cx.bars->pv_done[(gj - 1) & 1], ((gj - 1) >> 1) & 1);
      tc::fence_after();
#pragma unroll 1
      for (int cb = 0; cb < 8; ++cb) {
        float o[32];
        tc::tmem_ld32(lane_base + cb * 32, o);
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] *= alpha;
        tc::tmem_st32(lane_base + cb * 32, o);
      }
      tc::tmem_wait_st();
      l *= alpha;
    }
    const float mu = m == -INFINITY ? 0.f : m;
    float sum4[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t hi[kT / 2], lo[kT / 2];
#pragma unroll
    for (int k = 0; k < kT; k += 2) {
      const float x0 = exp2f(fmaf(s[k], sl2, -mu));
      const float x1 = exp2f(fmaf(s[k + 1], sl2, -mu));
      sum4[k & 3] += x0;
      sum4[(k & 3) + 1] += x1;
      const __nv_bfloat162 hh = __floats2bfloat162_rn(x0, x1);
      const __nv_bfloat162 ll =
          __floats2bfloat162_rn(x0 - __low2float(hh), x1 - __high2float(hh));
      hi[k >> 1] = *reinterpret_cast<const uint32_t*>(&hh);
      lo[k >> 1] = *reinterpret_cast<const uint32_t*>(&ll);
    }
    l += (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
    // V rows past the piece's last token must be zero (0 * NaN poisons PV)
    if (t0 + kT > pc.tok_end) {
      const int st = gj % kStages;
      wait_bar(cx, &cx.bars->kv_full[st], (gj / kStages) & 1);
      uint8_t* v = smem + kOffKV + st * kStageBytes + kHalfBytes;
      const int z0 = pc.tok_end - t0;
      const int n = (kT - z0) * 4 * 8;  // rows x column blocks x chunks
      for (int e = threadIdx.x - 64; e < n; e += 128) {
        const int row = z0 + e / 32, rem = e % 32, cb = rem >> 3, ch = rem & 7;
        *reinterpret_cast<uint4*>(v + cb * (kT * 128) + row * 128 + (ch << 4)) =
            make_uint4(0, 0, 0, 0);
      }
      tc::fence_proxy_async_smem();
    }
    // P_j over S_j: hi in the first 32 columns, lo in the next 32
    tc::tmem_st32(sbuf, reinterpret_cast<const float*>(hi));
    tc::tmem_st32(sbuf + kT / 2, reinterpret_cast<const float*>(lo));
    tc::tmem_wait_st();
    tc::fence_before();
    __syncwarp();
    if (lane == 0) tc::bar_arrive(tc::smem_u32(&cx.bars->p_full[gj & 1]));
  }

  // epilogue: O / l
  const int gl = gj0 + pc.n_tiles - 1;
  wait_bar(cx, &cx.bars->pv_done[gl & 1], (gl >> 1) & 1);
  tc::fence_after();
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const float mu = m == -INFINITY ? 0.f : m;
  const int S = seg_splits(pc.s0, pc.nt, U, P);
  const int head = pc.g * p.group + (r - i * p.group);
  if (S == 1) {
    __nv_bfloat16* dst =
        p.out + (((long long)pc.b * p.q_len + i) * p.hq + head) * kHeadDim;
#pragma unroll 1
    for (int cb = 0; cb < 8; ++cb) {
      float o[32];
      tc::tmem_ld32(lane_base + cb * 32, o);
      if (valid) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint4 v;
          __nv_bfloat162 t;
          t = __floats2bfloat162_rn(o[8 * k] * inv, o[8 * k + 1] * inv);
          v.x = *reinterpret_cast<uint32_t*>(&t);
          t = __floats2bfloat162_rn(o[8 * k + 2] * inv, o[8 * k + 3] * inv);
          v.y = *reinterpret_cast<uint32_t*>(&t);
          t = __floats2bfloat162_rn(o[8 * k + 4] * inv, o[8 * k + 5] * inv);
          v.z = *reinterpret_cast<uint32_t*>(&t);
          t = __floats2bfloat162_rn(o[8 * k + 6] * inv, o[8 * k + 7] * inv);
          v.w = *reinterpret_cast<uint32_t*>(&t);
          *reinterpret_cast<uint4*>(dst + cb * 32 + 8 * k) = v;
        }
      }
    }
  } else {
    const int k = pc.b * p.hkv + pc.g;
    const int slot = slot_base_warp(p, s_pre, k, U, P) + (c - cta_of(pc.s0, U, P));
    float* dst = p.part_o + ((long long)slot * p.rows + r) * kHeadDim;
#pragma unroll 1
    for (int cb = 0; cb < 8; ++cb) {
      float o[32];
      tc::tmem_ld32(lane_base + cb * 32, o);
      if (valid) {
#pragma unroll
        for (int k4 = 0; k4 < 8; ++k4)
          *reinterpret_cast<float4*>(dst + cb * 32 + 4 * k4) =
              make_float4(o[4 * k4] * inv, o[4 * k4 + 1] * inv,
                          o[4 * k4 + 2] * inv, o[4 * k4 + 3] * inv);
      }
    }
    if (valid)
      p.part_lse[(long long)slot * p.rows + r] =
          l > 0.f ? mu + log2f(l) : -INFINITY;
  }
}

// Softmax threads write their Q row of piece (b, g) into the swizzled tile.
__device__ __forceinline__ void load_q_row(const AttnParams& p, const Piece& pc,
                                           uint8_t* q_s) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w4 = warp & 3, pos = 32 * w4 + lane;
  const int R = (p.rows + 3) >> 2;
  const int r = w4 * R + lane;
  if (!(lane < R && r < p.rows)) return;
  const int i = r / p.group, h = pc.g * p.group + (r - i * p.group);
  const uint4* src = reinterpret_cast<const uint4*>(
      p.q + (((long long)pc.b * p.q_len + i) * p.hq + h) * kHeadDim);
#pragma unroll 8
  for (int cidx = 0; cidx < 32; ++cidx) {
    const uint4 v = __ldg(src + cidx);
    const int blk = cidx >> 3, ch = cidx & 7;
    *reinterpret_cast<uint4*>(q_s + blk * 16384 + pos * 128 +
                              ((ch ^ (pos & 7)) << 4)) = v;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    verify_split_tc_kernel(const AttnParams p,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  int* s_pre = reinterpret_cast<int*>(smem + kOffPre);
  __shared__ __align__(8) Bars bars;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  plan_prefix(p, s_pre);
  const long long U = (long long)p.hkv * s_pre[p.batch];
  const int P = effective_grid(p.grid, U);
  const int c = blockIdx.x;
  if (c >= P) return;  // uniform over the CTA, before any TMEM or barrier use

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::bar_init(tc::smem_u32(&bars.kv_full[s]), 1);
      tc::bar_init(tc::smem_u32(&bars.kv_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::bar_init(tc::smem_u32(&bars.s_full[s]), 1);
      tc::bar_init(tc::smem_u32(&bars.p_full[s]), 4);
      tc::bar_init(tc::smem_u32(&bars.pv_done[s]), 1);
    }
    tc::bar_init(tc::smem_u32(&bars.drain), 1);
    s_abort = 0;
    tc::bar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(&s_tmem), kTmemCols);
  if (warp >= 2) {  // zero every Q row once; valid rows are rewritten per piece
    const int pos = 32 * (warp & 3) + lane;
#pragma unroll
    for (int blk = 0; blk < 4; ++blk)
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        *reinterpret_cast<uint4*>(smem + blk * 16384 + pos * 128 + ch * 16) =
            make_uint4(0, 0, 0, 0);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = s_tmem;
  Ctx cx{&bars, &s_abort, &p};

  long long u = cta_start(c, U, P);
  const long long u_end = cta_start(c + 1, U, P);
  int gj0 = 0;
  int last_loaded = -1;  // last tile index the producer loaded
  while (u < u_end) {
    Piece pc;
    pc.b = find_request(s_pre, p.batch, p.hkv, u);
    pc.nt = s_pre[pc.b + 1] - s_pre[pc.b];
    const long long rb = (long long)p.hkv * s_pre[pc.b];
    pc.g = (int)((u - rb) / pc.nt);
    pc.s0 = rb + (long long)pc.g * pc.nt;
    const int j0 = (int)(u - pc.s0);
    const int j1 = (int)(u_end - pc.s0 < pc.nt ? u_end - pc.s0 : pc.nt);
    u = pc.s0 + j1;
    pc.len = clamp_len(p.seq_lens[pc.b], p.max_tokens);
    pc.tok_begin = j0 * kUnit;
    pc.tok_end = min(j1 * kUnit, pc.len);
    pc.n_tiles = (pc.tok_end - pc.tok_begin + kT - 1) / kT;

    if (warp >= 2) {
      load_q_row(p, pc, smem);
      tc::fence_proxy_async_smem();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) {
      // the whole warp: lanes issue the boxes of their pages
      produce(cx, pc, gj0, smem + kOffKV, &tm_k, &tm_v);
      last_loaded = gj0 + pc.n_tiles - 1;
      __syncwarp();
    } else if (warp == 1) {
      if (lane == 0) mma_piece(cx, pc, gj0, tmem, smem);
      __syncwarp();
    } else {
      softmax_piece(cx, pc, gj0, tmem, smem, s_pre, U, P, c);
    }
    gj0 += pc.n_tiles;
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
  }

  // teardown: no TMA copy or MMA may still be in flight
  if (warp == 0 && lane == 0) {
    for (int gj = max(0, last_loaded - kStages + 1); gj <= last_loaded; ++gj)
      wait_bar(cx, &bars.kv_full[gj % kStages], (gj / kStages) & 1, true);
  }
  if (warp == 1 && lane == 0) {
    tc::commit(tc::smem_u32(&bars.drain));
    wait_bar(cx, &bars.drain, 0, true);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_verify_split_tc(const AttnParams& p, const CUtensorMap& tm_k,
                                   const CUtensorMap& tm_v, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(
      verify_split_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      kSmemBytes);
  if (e != cudaSuccess) return e;
  verify_split_tc_kernel<<<p.grid, kThreads, kSmemBytes, s>>>(p, tm_k, tm_v);
  return cudaGetLastError();
}

int verify_split_tc_ctas_per_sm() {
  if (cudaFuncSetAttribute(verify_split_tc_kernel,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &n, verify_split_tc_kernel, kThreads, kSmemBytes) != cudaSuccess)
    return 0;
  return n < 1 ? 0 : 1;  // TMEM: one 512-column allocation per SM
}

int verify_split_tc_box_rows(int page_size) { return page_size < kT ? page_size : kT; }

}  // namespace specv
