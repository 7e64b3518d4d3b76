// Decode path (rows <= 4): the whole FFN block in one persistent launch.
//
// docs.rs "hf2q 0.1.3 .../deepseek4/ffn_forward.rs", forward_ffn_rows, every stage in order:
// rms_norm_no_scale_f32 + raw_matmul "HC FFN function" + dispatch_hc_split_sinkhorn (mix roles),
// dispatch_hc_pre + rms_norm + raw_matmul "MoE gate" + dispatch_deepseek_moe_{score,hash}_route +
// dispatch_deepseek_moe_sanitize_indices (router roles), expert_matmul "routed gate"/"routed up" +
// raw_matmul "shared gate"/"shared up" + dispatch_deepseek_moe_swiglu (phase A), expert_matmul
// "routed down" + raw_matmul "shared down" (phase B), dispatch_deepseek_moe_weighted_reduce +
// dispatch_hc_post (phase C).
//
// At 1-4 tokens every expert weight byte feeds 1-4 multiply-adds, so the block is bound by HBM
// bandwidth once the weights stream, and by latency before that.  One launch holds all of it, so
// no kernel boundary sits on the critical path and HBM never idles between the stages:
//
//   roles    the first CTAs to arrive take the prelude by a CTA ticket: `nm` mix CTAs (a column
//            chunk of the flattened state each; the last one forms pre/post, publishes them and
//            then forms the Sinkhorn comb), then `nr` router CTAs (a 64-wide chunk of hidden each:
//            ffn_input, its RMS partial and the partial logits; the last one reduces, routes
//            every row and groups the (row, slot) pairs by expert).  Router CTAs load their
//            router-weight chunk before the mix is done.
//   phase A  gate/up rows, group-major with the shared expert first (its tickets need no
//            routing, so they start as soon as the normalised input is known):
//            act[g, r, i] = silu(x_r . G[i]) * (x_r . U[i]); each row bumps its group's counter;
//   phase B  down rows, group-major; a group's rows wait (bounded) until its gate/up rows are all
//            published, then y[g, r, d] = act[g, r, :] . Dn[d, :]; each ticket bumps its d-block;
//   phase C  per 32-wide d-block, once every group's rows of it are in: ffn_out = sum_g w * y and
//            the hc_post output of that block.
//
// Work is handed out by device-wide tickets, so only running CTAs ever hold work, and every wait
// is for work that running CTAs hold: every wait ends whatever the number of co-resident CTAs.
// Waits still give up after 1 s (device timeout bit).  The serial tails run once per call, out of
// an instruction cache that streaming hundreds of MB through L2 leaves cold, so a few CTAs that
// would otherwise idle first run them on scratch data ("dry" runs) to pull the code into L2.  The last CTA to leave resets the counters, so
// the next launch (or a graph replay) starts from zero without a separate clearing step.
#include <math.h>
#include <stddef.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

struct DecodeArgs {
  // inputs
  const float *state;              // [rows, hc, hidden]
  const uint16_t *hc_fn;           // [M, hc * hidden] bf16
  const float *hc_scale, *hc_base;  // [3], [M]
  const float *norm_w;             // [hidden]
  const uint16_t *gate;            // [experts, hidden] router, bf16
  RouteParams rp;                  // routing source and the idx / rw / safe outputs
  const uint16_t *gate_exps, *up_exps, *down_exps, *gate_sh, *up_sh, *down_sh;
  // MXFP8 experts (the MX instances): E4M3 codes in the bf16 matrices' layouts, and E8M0 scales,
  // one per 32 consecutive elements of a row
  const uint8_t *gate_q, *up_q, *down_q, *gate_sh_q, *up_sh_q, *down_sh_q;
  const uint8_t *gate_s, *up_s, *down_s, *gate_sh_s, *up_sh_s, *down_sh_s;
  // scratch
  float *mix_part;   // [nm, rows, M + 1] mix partial sums (the last entry: sum of squares)
  float *mixes, *pre, *post, *comb;
  float *xw;         // [rows, hidden] ffn_input * ffn_norm weight (the RMS scale applied later)
  float *ss_part;    // [nr, rows] partial sums of ffn_input^2
  float *lg_part;    // [nr, rows, experts] partial logits (before the RMS scale)
  float *row_rs;     // [rows] rsqrt(mean(ffn_input^2) + eps)
  float *ffn_norm;   // [rows, hidden] stage tap, written by CTA 0
  float *logits;     // [rows, experts]
  int *ngroups, *group_e, *group_mask;
  float *group_w;    // [groups, 4]
  float *act;        // [groups, 4, inter]
  float *y;          // [groups, 4, hidden]
  float *ffn_out, *out_state;
  unsigned *counters;  // kDecCnt* layout below, zero at launch, zeroed again by the last CTA out
  int n_counters;
  int *status;
  int rows, hidden, inter, experts, hc, M, iters, nm, nr, mix_chunk;
  float eps;
};

// counter slots.  The prelude flags share one 128-byte line; each work-ticket counter, the group
// counters and the d-block counters get lines of their own, so that the atomics of one phase do
// not queue behind another's at the same L2 line.
constexpr int kCntRole = 0, kCntMixDone = 1, kCntRtDone = 3, kCntRoute = 5,
              kCntComb = 6, kCntExit = 7, kCntAbort = 8;
constexpr int kCntTickA = 32, kCntTickB = 64, kCntTickC = 96, kCntGroups = 128;
constexpr int kCntDBlocks = kCntGroups + 64;  // after the group counters, on a fresh line
static_assert(kDecodeGroupsMax <= 64, "group counters fit before the d-block counters");

constexpr uint64_t kSpinLimitNs = 1000000000ull;
constexpr int kRouterChunk = 64;  // hidden columns per router CTA
constexpr int kMixCols = 512;     // flattened-state columns per mix CTA (a multiple of 128)
constexpr int kWarmCtas = 16;     // streaming-only CTAs that pre-run the prelude tails' code
constexpr int kRowsPerTicketA = 1;  // gate/up rows per ticket
constexpr int kRowsPerTicketB = 4;  // down rows per ticket (a 32-row d-block holds 8 tickets)

// Shared memory of the prelude roles (static; the streaming phases use the dynamic x buffer).
// The arrays read or written as float4 come first, each 16-byte aligned (checked below).
struct PreludeSmem {
  alignas(16) float st[kDecodeRows][kMixCols];        // mix: state chunk; router: [rows][hc][64]
  alignas(16) float xw[kDecodeRows][kRouterChunk];    // router: ffn_input * norm weight chunk
  alignas(16) float lg[kDecodeRows][kExpertsMax];     // router tail: logits
  alignas(16) float sc[kDecodeRows][kExpertsMax];     // router tail: selection scores
  alignas(16) float bias[kExpertsMax];                // router: selection bias (score layers)
  float sums[kDecodeRows][kMixMax + 1];               // mix tail: reduced sums
  float nw[kRouterChunk];                             // router: norm weight chunk
  float pre[kDecodeRows][kHcMax];
  float hc_scale[3], hc_base[kMixMax];                // mix: split parameters
  float red[8][kDecodeRows];
  float rs[kDecodeRows];
  int hash_e[kDecodeRows][kTopKMax];                  // router: tid2eid rows (hash layers)
  int tok_ok[kDecodeRows];                            // router: token id in range (hash layers)
  int sel[kDecodeRows][kTopKMax];
  float w[kDecodeRows][kTopKMax];
  int flag;
};
static_assert(offsetof(PreludeSmem, st) % 16 == 0 && offsetof(PreludeSmem, xw) % 16 == 0 &&
                  offsetof(PreludeSmem, lg) % 16 == 0 && offsetof(PreludeSmem, sc) % 16 == 0 &&
                  (kMixCols * 4) % 16 == 0 && (kRouterChunk * 4) % 16 == 0 && (kExpertsMax * 4) % 16 == 0,
              "float4 accesses of the prelude shared memory need 16-byte aligned rows");

__device__ __forceinline__ uint4 ld_weight(const uint16_t *p) { return ld_stream(p); }

// act is written during this kernel, so it is read through L1 (ld.global.ca) only after the
// reading warp has acquired its group's completion counter: no line of it can be cached earlier.
__device__ __forceinline__ float4 ld_ca4(const float *p) {
  float4 v;
  asm volatile("ld.global.ca.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// Adds n to a completion counter with release semantics: this thread's earlier writes (and those
// ordered before them by a fence) are visible to whoever acquires the new value.
__device__ __forceinline__ void publish(unsigned *counter, unsigned n) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(counter), "r"(n) : "memory");
}

// Polls (one thread) until *counter >= target, with a bounded wait.  False on timeout; once any
// wait of this launch has timed out (`abort`, a counter slot of the launch), every later wait of
// the launch fails at once, so that a failed launch still ends quickly.
// `nap`: sleep briefly between polls (waits that may last, with many waiters); without it the
// poll spins, for the short waits at the end of the launch where latency is all that counts.
__device__ bool poll_at_least(const unsigned *counter, unsigned target, int *status, unsigned *abort,
                              bool nap = true) {
  if (ld_acquire_u32(counter) >= target) return true;
  const uint64_t w0 = global_timer_ns();
  while (ld_acquire_u32(counter) < target) {
    if (*reinterpret_cast<volatile unsigned *>(abort) != 0u || global_timer_ns() - w0 > kSpinLimitNs) {
      atomicOr(status, kDevTimeout);
      atomicExch(abort, 1u);
      return false;
    }
    if (nap) __nanosleep(64);
  }
  return true;
}

// Warp-wide bounded wait: lane 0 polls, then every lane acquires the counter so that its later
// reads see what the producers published.
__device__ bool wait_at_least(const unsigned *counter, unsigned target, int *status, unsigned *abort,
                              bool nap = true) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = poll_at_least(counter, target, status, abort, nap) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) (void)ld_acquire_u32(counter);
  return ok != 0;
}

// CTA-wide bounded wait (every thread of the CTA calls it).
__device__ bool cta_wait_at_least(const unsigned *counter, unsigned target, int *status, unsigned *abort,
                                  int *s_flag) {
  if (threadIdx.x == 0) *s_flag = poll_at_least(counter, target, status, abort) ? 1 : 0;
  __syncthreads();
  const bool ok = *s_flag != 0;
  if (ok) (void)ld_acquire_u32(counter);
  __syncthreads();
  return ok;
}

// Next work ticket of a phase: lane 0 draws it, the warp shares it.
__device__ __forceinline__ int draw_ticket(unsigned *tick) {
  int c = 0;
  if ((threadIdx.x & 31) == 0) c = (int)atomicAdd(tick, 1u);
  return __shfl_sync(0xffffffffu, c, 0);
}

// True in exactly one CTA: the last of `total` to finish its share of a role (all earlier global
// writes of every thread of the CTA are fenced before the count).
__device__ bool cta_arrive_last(unsigned *count, unsigned total, int *s_flag) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *s_flag = atomicAdd(count, 1u) == total - 1 ? 1 : 0;
  __syncthreads();
  const bool last = *s_flag != 0;
  if (last) __threadfence();
  return last;
}

// One lane's share of the mix partial sums of item `it` (row r, output m; it = r * (M + 1) + m):
// chunks `lane` and `lane + 32` (at most 64 mix CTAs).  Every reduction of an item adds these two
// and then sums over the warp, so the result has the same bits wherever it is formed.
__device__ __forceinline__ float mix_item_partial(const DecodeArgs &a, int items, int it, int lane) {
  const float *p = a.mix_part + it;  // [chunk][row][m] = it + chunk * items
  float x = 0.f;
  if (lane < a.nm) x = __ldcg(p + (size_t)lane * items);
  if (lane + 32 < a.nm) x += __ldcg(p + (size_t)(lane + 32) * items);
  return x;
}

// RMS scale of the flattened state from its sum of squares, and a stream gate
// sigmoid(sum * rs * scale + base) (pre; post is twice the same form).
__device__ __forceinline__ float mix_rs(float ss, int hcd, float eps) { return rsqrtf(ss / (float)hcd + eps); }
__device__ __forceinline__ float hc_gate(float sum, float rs, float scale, float base) {
  return sigmoidf_(fmaf(sum * rs, scale, base));
}

// ---------------------------------------------------------------------------------------------
// Mix role (rms_norm_no_scale_f32 + raw_matmul "HC FFN function" + dispatch_hc_split_sinkhorn).
// Per row: ss = sum x^2 and dot_m = sum x * hc_fn[m] over the flattened hc*hidden state;
// mixes = dot * rsqrt(ss / (hc*hidden) + eps) (the RMS scale factors out of the dot product).
// ---------------------------------------------------------------------------------------------

// Tail of the mix role, run by the last mix CTA, off the critical path (the router CTAs form pre
// themselves from the same partials): the mixes, pre and post of every row, then the comb
// (Sinkhorn), which only the final hc_post needs, published.
template <int ROWS>
__device__ __noinline__ void mix_tail(const DecodeArgs &a, PreludeSmem &sm, unsigned *cnt) {
  constexpr int rows = ROWS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, M = a.M, hc = a.hc;
  const int items = rows * (M + 1);
  // warp w reduces items w, w + 8, ...; every load is issued before the first sum
  constexpr int kItemsPerWarp = (ROWS * (kMixMax + 1) + 7) / 8;
  float v[kItemsPerWarp];
#pragma unroll
  for (int k = 0; k < kItemsPerWarp; ++k) {
    const int it = warp + 8 * k;
    v[k] = it < items ? mix_item_partial(a, items, it, lane) : 0.f;
  }
#pragma unroll
  for (int k = 0; k < kItemsPerWarp; ++k) {
    const int it = warp + 8 * k;
    const float x = warp_sum(v[k]);
    if (lane == 0 && it < items) sm.sums[it / (M + 1)][it % (M + 1)] = x;
  }
  __syncthreads();
  if (tid < rows) {
    const float rs = mix_rs(sm.sums[tid][M], hc * a.hidden, a.eps);
    for (int h = 0; h < hc; ++h) {
      a.pre[tid * hc + h] = hc_gate(sm.sums[tid][h], rs, sm.hc_scale[0], sm.hc_base[h]);
      a.post[tid * hc + h] = 2.0f * hc_gate(sm.sums[tid][hc + h], rs, sm.hc_scale[1], sm.hc_base[hc + h]);
    }
    for (int m = 0; m < M; ++m) a.mixes[tid * M + m] = sm.sums[tid][m] * rs;
  }
  __syncthreads();
  if (warp < rows) sinkhorn_comb_warp(a.mixes + warp * M, sm.hc_scale, sm.hc_base, hc, a.iters, a.comb + warp * hc * hc);
  __threadfence();
  __syncthreads();
  if (tid == 0) publish(&cnt[kCntComb], 1u);
}

// Mix CTA j: flattened-state columns [j * kMixCols, +kMixCols) (the last chunk may be shorter, a
// multiple of 128).  Warp w forms outputs w, w + 8, w + 16; lane l covers columns 4l + 128p of the
// chunk, so the shared-memory state reads are conflict-free and the hc_fn reads coalesced.
template <int ROWS>
__device__ void mix_role(const DecodeArgs &a, int j, PreludeSmem &sm, unsigned *cnt) {
  constexpr int rows = ROWS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hcd = a.hc * a.hidden, M = a.M;
  const int c0 = j * kMixCols, width = min(kMixCols, hcd - c0);
  // hc_fn does not come from the previous kernel: load it before waiting for that kernel
  uint2 hw[3][4];
#pragma unroll
  for (int q = 0; q < 3; ++q)
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int m = warp + 8 * q, c = 4 * lane + 128 * p;
      hw[q][p] = (m < M && c < width) ? __ldg(reinterpret_cast<const uint2 *>(a.hc_fn + (size_t)m * hcd + c0 + c))
                                      : make_uint2(0u, 0u);
    }
  if (tid < 3) sm.hc_scale[tid] = a.hc_scale[tid];
  if (tid < M) sm.hc_base[tid] = a.hc_base[tid];
  pdl_wait();
  // the state chunk (one float4 per thread and row)
  static_assert(kMixCols / 4 <= 256, "one float4 of each row per thread");
  float4 sv[kDecodeRows];
#pragma unroll
  for (int r = 0; r < kDecodeRows; ++r)
    sv[r] = (r < rows && tid < width / 4) ? __ldcg(reinterpret_cast<const float4 *>(a.state + (size_t)r * hcd + c0 + tid * 4))
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
  float ss[kDecodeRows];
#pragma unroll
  for (int r = 0; r < kDecodeRows; ++r) {
    const float4 v = sv[r];
    if (tid < width / 4) *reinterpret_cast<float4 *>(&sm.st[r][tid * 4]) = v;
    ss[r] = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  __syncthreads();
  float acc[3][kDecodeRows];
#pragma unroll
  for (int q = 0; q < 3; ++q)
#pragma unroll
    for (int r = 0; r < kDecodeRows; ++r) acc[q][r] = 0.f;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const int c = 4 * lane + 128 * p;
    if (c < width) {
#pragma unroll
      for (int r = 0; r < kDecodeRows; ++r) {
        if (r < rows) {
          const float4 x = *reinterpret_cast<const float4 *>(&sm.st[r][c]);
#pragma unroll
          for (int q = 0; q < 3; ++q)
            acc[q][r] += bf_lo(hw[q][p].x) * x.x + bf_hi(hw[q][p].x) * x.y + bf_lo(hw[q][p].y) * x.z +
                         bf_hi(hw[q][p].y) * x.w;
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kDecodeRows; ++r) {
    if (r < rows) {
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const float v = warp_sum(acc[q][r]);
        const int m = warp + 8 * q;
        if (lane == 0 && m < M) a.mix_part[((size_t)j * rows + r) * (M + 1) + m] = v;
      }
      const float s = warp_sum(ss[r]);
      if (lane == 0) sm.red[warp][r] = s;
    }
  }
  __syncthreads();
  if (tid < rows) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += sm.red[w][tid];
    a.mix_part[((size_t)j * rows + tid) * (M + 1) + M] = s;
  }
  if (cta_arrive_last(&cnt[kCntMixDone], (unsigned)a.nm, &sm.flag)) mix_tail<ROWS>(a, sm, cnt);
}

// ---------------------------------------------------------------------------------------------
// Router role (dispatch_hc_pre + rms_norm + raw_matmul "MoE gate" + the route and sanitize
// dispatches).  ffn_input v = sum_h pre[h] * state[h]; logits = rs * sum_d (v_d * w_d) * gate[e, d]
// with rs = rsqrt(mean(v^2) + eps): the RMS scale factors out of the dot product, so each router
// CTA works on its own chunk of hidden and only the last one needs the whole row.
// ---------------------------------------------------------------------------------------------

// RMS scale of row r from the router CTAs' partial sums of squares, by one warp (lane l: router
// CTAs l, l + 32, ...; then a warp sum).  The router tail and every streaming CTA form it this
// way, so all of them get the same bits.
__device__ __forceinline__ float row_rs_from_partials(const DecodeArgs &a, int rows, int r, int nsum) {
  const int lane = threadIdx.x & 31;
  float x = 0.f;
  for (int c = lane; c < nsum; c += 32) x += __ldcg(a.ss_part + c * rows + r);
  x = warp_sum(x);
  return rsqrtf(x / (float)a.hidden + a.eps);
}

// Routing of row r by one warp.  Score layers: top_k on the selection scores sigmoid(logit) + bias
// (formed beforehand in sm.sc, in f32; ties to the lower expert index), weights = the chosen
// unbiased scores / their sum.  Hash layers: the tid2eid row in table order, weights =
// sigmoid(logit) normalised over the valid slots.
__device__ void route_row(const DecodeArgs &a, PreludeSmem &sm, int r, bool live) {
  const RouteParams &p = a.rp;
  const int lane = threadIdx.x & 31, E = p.experts, K = p.top_k;
  int my_sel = -1;
  if (!p.hash) {
    uint32_t taken = 0;  // bit j: expert lane + 32 j already chosen
#pragma unroll 1
    for (int k = 0; k < K; ++k) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll 1
      for (int j = 0, e = lane; e < E; ++j, e += 32) {
        const float x = sm.sc[r][e];
        if (!((taken >> j) & 1u) && (x > bv || be == 0x7fffffff)) {
          bv = x;
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      if (lane == k) my_sel = be;
    }
  } else {
    const bool tok_ok = sm.tok_ok[r] != 0;
    if (!tok_ok && lane == 0 && live) atomicOr(p.status, kDevTokenRange);
    if (lane < K) my_sel = sm.hash_e[r][lane];
    const bool bad_entry = tok_ok && lane < K && !(my_sel >= 0 && my_sel < E);
    if (__any_sync(0xffffffffu, bad_entry) && lane == 0 && live) atomicOr(p.status, kDevRouteRange);
  }
  const bool valid = lane < K && my_sel >= 0 && my_sel < E;
  const float sc = valid ? sigmoidf_(sm.lg[r][my_sel]) : 0.f;
  const float tot = warp_sum(sc);
  if (lane < K) {
    const float w = tot > 0.f ? sc / tot : 0.f;
    if (live) {
      p.idx[r * K + lane] = my_sel;
      p.rw[r * K + lane] = w;
      p.safe[r * K + lane] = valid ? (unsigned)my_sel : 0u;
    }
    sm.sel[r][lane] = my_sel;
    sm.w[r][lane] = w;
  }
}

// Groups the (row, slot) pairs by expert, one pair per lane of one warp (rows * top_k <= 32).
// Group 0 is the shared expert (weight 1 for every row); then the distinct routed experts in order
// of first appearance, each with the mask of rows using it and their summed route weights.
template <int ROWS>
__device__ void group_rows(const DecodeArgs &a, PreludeSmem &sm, bool live) {
  constexpr int rows = ROWS;
  const int lane = threadIdx.x & 31, K = a.rp.top_k, E = a.experts;
  int e = -1;
  if (lane < rows * K) e = sm.sel[lane / K][lane % K];
  const bool valid = lane < rows * K && e >= 0 && e < E;
  const unsigned same = __match_any_sync(0xffffffffu, valid ? e : E + 1 + lane);
  const unsigned below = (1u << lane) - 1u;
  const bool leader = valid && (same & below) == 0u;
  const unsigned leaders = __ballot_sync(0xffffffffu, leader);
  if (leader && live) {
    const int g = 1 + __popc(leaders & below);
    int mask = 0;
    float w0 = 0.f, w1 = 0.f, w2 = 0.f, w3 = 0.f;
    for (unsigned m = same; m != 0u; m &= m - 1u) {
      const int b = __ffs(m) - 1, rb = b / K;
      const float wb = sm.w[rb][b - rb * K];
      mask |= 1 << rb;
      if (rb == 0) w0 += wb;
      else if (rb == 1) w1 += wb;
      else if (rb == 2) w2 += wb;
      else w3 += wb;
    }
    a.group_e[g] = e;
    a.group_mask[g] = mask;
    *reinterpret_cast<float4 *>(a.group_w + g * 4) = make_float4(w0, w1, w2, w3);
  }
  if (lane == 0 && live) {
    a.group_e[0] = E;
    a.group_mask[0] = (1 << rows) - 1;
    *reinterpret_cast<float4 *>(a.group_w) =
        make_float4(1.f, rows > 1 ? 1.f : 0.f, rows > 2 ? 1.f : 0.f, rows > 3 ? 1.f : 0.f);
    *a.ngroups = 1 + __popc(leaders);
  }
}

// Tail of the router role, run by the last router CTA: the RMS scale of every row, the logits
// reduced in a fixed order, the selection scores (every thread a share), routing (one
// warp per row) and grouping (published).  `live` false: the same code
// with one partial and no global write or publication, run by idle CTAs to bring it into L2.
template <int ROWS>
__device__ __noinline__ void router_tail(const DecodeArgs &a, PreludeSmem &sm, unsigned *cnt, bool live) {
  constexpr int rows = ROWS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.experts;
  const int nsum = live ? a.nr : 1;
  // RMS scales (the streaming CTAs form the same values themselves)
  if (warp < rows) {
    const float rs = row_rs_from_partials(a, rows, warp, nsum);
    if (lane == 0) {
      sm.rs[warp] = rs;
      if (live) a.row_rs[warp] = rs;
    }
  }
  __syncthreads();
  // logits: four quarters of the router CTAs per (row, 4 experts); each thread issues its quarter's
  // loads back to back, then the quarters are added in a fixed order
  const int E4 = E / 4, units = rows * E4, q4 = (nsum + 3) / 4;
  for (int u0 = 0; u0 < units * 4; u0 += blockDim.x) {
    const int u = u0 + tid;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (u < units * 4) {
      const int item = u >> 2, quarter = u & 3;
      const int r = item / E4, e = (item - r * E4) * 4;
      const float *p = a.lg_part + (size_t)r * E + e;
      const int c0 = quarter * q4, c1 = min(nsum, c0 + q4);
#pragma unroll 8
      for (int c = c0; c < c1; ++c) {
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(p + (size_t)c * rows * E));
        s.x += v.x;
        s.y += v.y;
        s.z += v.z;
        s.w += v.w;
      }
    }
    // the four quarters of an item sit in four neighbouring lanes
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      s.x += __shfl_xor_sync(0xffffffffu, s.x, o);
      s.y += __shfl_xor_sync(0xffffffffu, s.y, o);
      s.z += __shfl_xor_sync(0xffffffffu, s.z, o);
      s.w += __shfl_xor_sync(0xffffffffu, s.w, o);
    }
    if (u < units * 4 && (u & 3) == 0) {
      const int item = u >> 2, r = item / E4, e = (item - r * E4) * 4;
      const float rs = sm.rs[r];
      const float4 l = make_float4(s.x * rs, s.y * rs, s.z * rs, s.w * rs);
      *reinterpret_cast<float4 *>(&sm.lg[r][e]) = l;
      if (live) *reinterpret_cast<float4 *>(a.logits + (size_t)r * E + e) = l;
    }
  }
  if (tid == 0) sm.flag = 0;
  __syncthreads();
  // selection scores sigmoid(logit) + bias (score layers), a non-finite logit flagged
  if (!a.rp.hash) {
    bool bad = false;
    for (int i = tid; i < rows * E; i += blockDim.x) {
      const int r = i / E, e = i - r * E;
      const float l = sm.lg[r][e];
      bad |= !isfinite(l);
      const float x = sigmoidf_(l) + sm.bias[e];
      sm.sc[r][e] = isnan(x) ? -INFINITY : x;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) sm.flag = 1;
  }
  __syncthreads();
  if (tid == 0 && sm.flag && live) atomicOr(a.rp.status, kDevNonFinite);
  if (warp < rows) route_row(a, sm, warp, live);
  __syncthreads();
  if (warp == 0) group_rows<ROWS>(a, sm, live);
  if (live) __threadfence();
  __syncthreads();
  if (tid == 0 && live) publish(&cnt[kCntRoute], 1u);
}

// Router CTA j: hidden columns [64 j, 64 j + 64).  Thread e holds expert e's 64 router weights of
// the chunk in registers (experts beyond the block size are read when needed).  pre is formed
// here from the mix CTAs' partial sums, as soon as all of them are in.
template <int ROWS>
__device__ void router_role(const DecodeArgs &a, int j, PreludeSmem &sm, unsigned *cnt) {
  constexpr int rows = ROWS;
  const RouteParams &p = a.rp;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.experts, D = a.hidden, hc = a.hc, K = p.top_k, M = a.M;
  const int d0 = j * kRouterChunk;
  // weights do not come from the previous kernel: load them before waiting for it
  uint4 gw[8];
#pragma unroll
  for (int q = 0; q < 8; ++q)
    gw[q] = tid < E ? __ldg(reinterpret_cast<const uint4 *>(a.gate + (size_t)tid * D + d0 + 8 * q))
                    : make_uint4(0u, 0u, 0u, 0u);
  if (tid < kRouterChunk) sm.nw[tid] = a.norm_w[d0 + tid];
  for (int e = tid; e < E; e += blockDim.x) sm.bias[e] = p.hash ? 0.f : p.bias[e];
  if (tid == 0) sm.hc_scale[0] = a.hc_scale[0];
  if (tid < hc) sm.hc_base[tid] = a.hc_base[tid];
  pdl_wait();
  float(&st)[kDecodeRows][kHcMax][kRouterChunk] =
      *reinterpret_cast<float(*)[kDecodeRows][kHcMax][kRouterChunk]>(&sm.st[0][0]);
  for (int i = tid; i < rows * hc * (kRouterChunk / 4); i += blockDim.x) {
    const int rh = i / (kRouterChunk / 4), c = (i - rh * (kRouterChunk / 4)) * 4;
    const int r = rh / hc, h = rh - r * hc;
    *reinterpret_cast<float4 *>(&st[r][h][c]) =
        __ldcg(reinterpret_cast<const float4 *>(a.state + ((size_t)r * hc + h) * D + d0 + c));
  }
  if (p.hash && tid < rows * K) {
    const int r = tid / K, k = tid - r * K;
    const int tok = p.token_ids[r];
    const bool ok = tok >= 0 && tok < p.vocab;
    sm.hash_e[r][k] = ok ? p.tid2eid[(size_t)tok * K + k] : -1;
    if (k == 0) sm.tok_ok[r] = ok ? 1 : 0;
  }
  // pre from the mix partials, once every mix CTA has written its own (bounded wait; on timeout
  // the status says so and the values below are not meaningful, but every CTA still finishes)
  (void)cta_wait_at_least(&cnt[kCntMixDone], (unsigned)a.nm, a.status, &cnt[kCntAbort], &sm.flag);
  {
    // items (r, h < hc) and (r, M): warp w reduces items w and w + 8, ...
    const int per = hc + 1, items = rows * per;
    for (int k = warp; k < items; k += 8) {
      const int r = k / per, h = k - r * per;
      const int m = h < hc ? h : M;
      const float x = warp_sum(mix_item_partial(a, rows * (M + 1), r * (M + 1) + m, lane));
      if (lane == 0) sm.sums[r][h] = x;
    }
  }
  __syncthreads();
  if (tid < rows * hc) {
    const int r = tid / hc, h = tid - r * hc;
    sm.pre[r][h] = hc_gate(sm.sums[r][h], mix_rs(sm.sums[r][hc], hc * D, a.eps), sm.hc_scale[0], sm.hc_base[h]);
  }
  __syncthreads();
  float ssq = 0.f;
  if (tid < rows * kRouterChunk) {
    const int r = tid / kRouterChunk, d = tid - r * kRouterChunk;
    float v = 0.f;
    for (int h = 0; h < hc; ++h) v += sm.pre[r][h] * st[r][h][d];
    const float xw = v * sm.nw[d];
    sm.xw[r][d] = xw;
    a.xw[(size_t)r * D + d0 + d] = xw;
    ssq = v * v;
  }
  ssq = warp_sum(ssq);
  if (lane == 0) sm.red[warp][0] = ssq;
  __syncthreads();
  static_assert(kRouterChunk == 64, "two warps per row below");
  if (tid < rows) a.ss_part[j * rows + tid] = sm.red[2 * tid][0] + sm.red[2 * tid + 1][0];
  auto partial_logits = [&](int e, const uint4(&w)[8]) {
#pragma unroll
    for (int r = 0; r < rows; ++r) {
      float l = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        l += dot8(w[q], *reinterpret_cast<const float4 *>(&sm.xw[r][8 * q]),
                  *reinterpret_cast<const float4 *>(&sm.xw[r][8 * q + 4]));
      a.lg_part[((size_t)j * rows + r) * E + e] = l;
    }
  };
  if (tid < E) partial_logits(tid, gw);
  for (int e = tid + blockDim.x; e < E; e += blockDim.x) {
    uint4 w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) w[q] = __ldg(reinterpret_cast<const uint4 *>(a.gate + (size_t)e * D + d0 + 8 * q));
    partial_logits(e, w);
  }
  if (cta_arrive_last(&cnt[kCntRtDone], (unsigned)a.nr, &sm.flag)) router_tail<ROWS>(a, sm, cnt, true);
}

// ---------------------------------------------------------------------------------------------
// Streaming phases
// ---------------------------------------------------------------------------------------------

template <int ROWS, bool MX>
__global__ void __launch_bounds__(256, 2) decode_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) float xs[];  // [rows, hidden]: x = ffn_norm(ffn_input)
  __shared__ __align__(16) PreludeSmem sm;
  constexpr int rows = ROWS;  // every row loop is unrolled exactly, without run-time guards
  unsigned *cnt = a.counters;
  const int tid = threadIdx.x, lane = tid & 31;
  const int D = a.hidden, I = a.inter, E = a.experts;
  if (tid == 0) sm.flag = (int)atomicAdd(&cnt[kCntRole], 1u);
  __syncthreads();
  const int role = sm.flag;
  __syncthreads();
  if (role < a.nm) {
    mix_role<ROWS>(a, role, sm, cnt);
  } else if (role < a.nm + a.nr) {
    router_role<ROWS>(a, role - a.nm, sm, cnt);
  } else {
    // streaming only, idle until the prelude is done: the first few CTAs run the router tail on
    // scratch data, which brings its code into L2 before the live tail needs it
    if (role < a.nm + a.nr + kWarmCtas) router_tail<ROWS>(a, sm, cnt, false);
  }
  pdl_wait();  // the state (read by phase C) comes from the previous kernel

  // ---- x = (ffn_input * norm weight) * rs, once every router CTA has written its share of xw and
  // of the sums of squares: each CTA forms rs itself, so the shared expert, which needs no
  // routing, streams while the router tail still routes ----
  (void)cta_wait_at_least(&cnt[kCntRtDone], (unsigned)a.nr, a.status, &cnt[kCntAbort], &sm.flag);
  if ((tid >> 5) < rows) {
    const float rs = row_rs_from_partials(a, rows, tid >> 5, a.nr);
    if (lane == 0) sm.rs[tid >> 5] = rs;
  }
  __syncthreads();
  for (int i = tid * 4; i < rows * D; i += blockDim.x * 4) {
    const int r = i / D;
    const float rs = sm.rs[r];
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.xw + i));
    const float4 x = make_float4(v.x * rs, v.y * rs, v.z * rs, v.w * rs);
    *reinterpret_cast<float4 *>(&xs[i]) = x;
    if (blockIdx.x == 0) *reinterpret_cast<float4 *>(a.ffn_norm + i) = x;
  }
  __syncthreads();
  unsigned *group_done = cnt + kCntGroups;
  unsigned *dblock_done = cnt + kCntDBlocks;
  const int nblk = D / kDecodeDBlock;
  const int all_rows = (1 << rows) - 1;

  // ---- phase A: gate/up rows, tickets in group-major order (the shared expert first) ----
  // A row's gate and up elements stream in batches of UA 16-byte loads per lane and matrix, all
  // of a batch in flight at once (fewer for 3-4 rows, whose FMAs take longer).  Group 0 (the
  // shared expert) needs no routing; the first ticket past it waits for the routing.
  constexpr int UA = ROWS >= 3 ? 4 : 8;
  constexpr int UQA = 4;  // MX: 16-byte loads per lane and matrix in flight (2048 codes a trip)
  const int perg = I / kRowsPerTicketA;
  int ng = -1;
  // the group table, once routed, in registers: lane l holds groups l and l + 32 (group 0, the
  // shared expert, is known without routing)
  int gt_e0 = E, gt_e1 = E, gt_m0 = all_rows, gt_m1 = 0;
  float gt_w0[rows], gt_w1[rows];  // route weights of groups lane and lane + 32, per row
#pragma unroll
  for (int r = 0; r < rows; ++r) gt_w0[r] = gt_w1[r] = 0.f;
  auto group_of = [&](int g, int &e, int &mask) {
    const int src = g & 31;
    const int e0 = __shfl_sync(0xffffffffu, gt_e0, src), e1 = __shfl_sync(0xffffffffu, gt_e1, src);
    const int m0 = __shfl_sync(0xffffffffu, gt_m0, src), m1 = __shfl_sync(0xffffffffu, gt_m1, src);
    e = g < 32 ? e0 : e1;
    mask = g < 32 ? m0 : m1;
  };
  for (int c = draw_ticket(&cnt[kCntTickA]);;) {
    if (ng < 0 && c >= perg) {
      if (wait_at_least(&cnt[kCntRoute], 1u, a.status, &cnt[kCntAbort])) {
        ng = __ldcg(a.ngroups);
        if (lane < ng) {
          gt_e0 = __ldcg(a.group_e + lane);
          gt_m0 = __ldcg(a.group_mask + lane);
#pragma unroll
          for (int r = 0; r < rows; ++r) gt_w0[r] = __ldcg(a.group_w + lane * kDecodeRows + r);
        }
        if (lane + 32 < ng) {
          gt_e1 = __ldcg(a.group_e + lane + 32);
          gt_m1 = __ldcg(a.group_mask + lane + 32);
#pragma unroll
          for (int r = 0; r < rows; ++r) gt_w1[r] = __ldcg(a.group_w + (lane + 32) * kDecodeRows + r);
        }
      } else {
        ng = 1;
      }
    }
    if (ng >= 0 && c >= ng * perg) break;
    int next = 0;
    if (lane == 0) next = (int)atomicAdd(&cnt[kCntTickA], 1u);  // consumed after this ticket: latency hidden
    const int g = c / perg, i0 = (c - g * perg) * kRowsPerTicketA;
    int e, mask;
    group_of(g, e, mask);
    const bool routed = e < E;
    for (int i = i0; i < i0 + kRowsPerTicketA; ++i) {
      float ga[kDecodeRows] = {0.f, 0.f, 0.f, 0.f}, ua[kDecodeRows] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (MX) {
        // 16 codes per lane and 16-byte load, all of a batch in flight; each 16-code piece lies in
        // one 32-element scale block, so its partial dot takes the block's scale once
        const size_t ro = routed ? (size_t)e * I + i : (size_t)i;
        const uint8_t *gq = (routed ? a.gate_q : a.gate_sh_q) + ro * D;
        const uint8_t *uq = (routed ? a.up_q : a.up_sh_q) + ro * D;
        const uint8_t *gsc = (routed ? a.gate_s : a.gate_sh_s) + ro * (D / 32);
        const uint8_t *usc = (routed ? a.up_s : a.up_sh_s) + ro * (D / 32);
        // the loop runs the same trips on every lane (its shuffles need the whole warp); lanes past
        // the row's end only skip the loads and the arithmetic.  Each trip covers 512 * UQA codes
        // (up to 128 scale blocks); lane l loads scale word k0 / 128 + l of the row (four blocks)
        // with the codes, and a code piece takes its block's byte from the lane that holds it.
        const unsigned *gsw = reinterpret_cast<const unsigned *>(gsc), *usw = reinterpret_cast<const unsigned *>(usc);
        for (int k0 = 0; k0 < D; k0 += 512 * UQA) {
          uint4 gv[UQA], uv[UQA];
          const bool wl = k0 / 128 + lane < D / 128;
          const unsigned gword = wl ? __ldg(gsw + k0 / 128 + lane) : 0u, uword = wl ? __ldg(usw + k0 / 128 + lane) : 0u;
#pragma unroll
          for (int u = 0; u < UQA; ++u) {
            const int cc = k0 + u * 512 + lane * 16;
            if (cc < D) {
              gv[u] = ld_stream(gq + cc);
              uv[u] = ld_stream(uq + cc);
            }
          }
#pragma unroll
          for (int u = 0; u < UQA; ++u) {
            const int cc = k0 + u * 512 + lane * 16;
            // block cc / 32 is block 16u + lane / 2 of this trip: byte (lane / 2) % 4 of the trip's
            // word 4u + lane / 8
            const int src = 4 * u + lane / 8, sh = ((lane >> 1) & 3) * 8;
            const unsigned gw = __shfl_sync(0xffffffffu, gword, src);
            const unsigned uw = __shfl_sync(0xffffffffu, uword, src);
            if (cc < D) {
              // both matrices decoded, so each row's x is read from shared memory once for both
              float fg[16], fu[16];
              e4m3x16_to_float_scaled(gv[u], fg);
              e4m3x16_to_float_scaled(uv[u], fu);
              const float sg = e8m0_value((gw >> sh) & 0xFFu), su = e8m0_value((uw >> sh) & 0xFFu);
#pragma unroll
              for (int r = 0; r < kDecodeRows; ++r) {
                if ((mask >> r) & 1) {
                  const float4 *xp = reinterpret_cast<const float4 *>(&xs[r * D + cc]);
                  const float4 x0 = xp[0], x1 = xp[1], x2 = xp[2], x3 = xp[3];
                  ga[r] = fmaf(sg, dot16(fg, x0, x1, x2, x3) * kE4m3Unscale, ga[r]);
                  ua[r] = fmaf(su, dot16(fu, x0, x1, x2, x3) * kE4m3Unscale, ua[r]);
                }
              }
            }
          }
        }
      } else {
      const uint16_t *gw = routed ? a.gate_exps + ((size_t)e * I + i) * D : a.gate_sh + (size_t)i * D;
      const uint16_t *uw = routed ? a.up_exps + ((size_t)e * I + i) * D : a.up_sh + (size_t)i * D;
      for (int base = lane * 8; base < D; base += 256 * UA) {
        uint4 gv[UA], uv[UA];
#pragma unroll
        for (int u = 0; u < UA; ++u) {
          const int cc = base + u * 256;
          if (cc < D) {
            gv[u] = ld_weight(gw + cc);
            uv[u] = ld_weight(uw + cc);
          }
        }
#pragma unroll
        for (int u = 0; u < UA; ++u) {
          const int cc = base + u * 256;
          if (cc < D) {
#pragma unroll
            for (int r = 0; r < kDecodeRows; ++r) {
              if ((mask >> r) & 1) {  // rows this expert does not serve cost nothing
                const float4 x0 = *reinterpret_cast<const float4 *>(&xs[r * D + cc]);
                const float4 x1 = *reinterpret_cast<const float4 *>(&xs[r * D + cc + 4]);
                ga[r] += dot8(gv[u], x0, x1);
                ua[r] += dot8(uv[u], x0, x1);
              }
            }
          }
        }
      }
      }
#pragma unroll
      for (int r = 0; r < kDecodeRows; ++r) {
        if ((mask >> r) & 1) {
          const float gs = warp_sum(ga[r]);
          const float us = warp_sum(ua[r]);
          if (lane == 0) a.act[((size_t)g * kDecodeRows + r) * I + i] = gs * sigmoidf_(gs) * us;
        }
      }
    }
    if (lane == 0) publish(&group_done[g], (unsigned)kRowsPerTicketA);  // one release per ticket
    c = __shfl_sync(0xffffffffu, next, 0);
  }
  if (ng < 0) ng = 1;

  // ---- phase B: down rows, tickets in group-major order; a ticket's rows share one group and one
  // d-block.  A group's rows wait (bounded) until all of its gate/up rows are published.
  constexpr int UB = ROWS >= 3 ? 4 : 8;
  constexpr int UQB = 4;  // MX: 16-byte loads per lane and down row in flight (4 x 512 codes: inter 2048)
  const int nB = ng * D / kRowsPerTicketB;
  int cur = -1;
  bool ready = false;
  for (int c = draw_ticket(&cnt[kCntTickB]); c < nB;) {
    int next = 0;
    if (lane == 0) next = (int)atomicAdd(&cnt[kCntTickB], 1u);
    const int t0 = c * kRowsPerTicketB;
    const int g = t0 / D, d0 = t0 - g * D;
    if (g != cur) {
      cur = g;
      ready = wait_at_least(&group_done[g], (unsigned)I, a.status, &cnt[kCntAbort]);
    }
    int e, mask;
    group_of(g, e, mask);
    const bool routed = e < E;
    if (ready) {
      const float *act = a.act + (size_t)g * kDecodeRows * I;
#pragma unroll 1
      for (int q = 0; q < kRowsPerTicketB; q += 2) {
        // two down rows in flight together
        const int dd = d0 + q;
        float acc0[kDecodeRows] = {0.f, 0.f, 0.f, 0.f}, acc1[kDecodeRows] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (MX) {
          const size_t ro = routed ? (size_t)e * D + dd : (size_t)dd;
          const uint8_t *dq0 = (routed ? a.down_q : a.down_sh_q) + ro * I, *dq1 = dq0 + I;
          const uint8_t *ds0 = (routed ? a.down_s : a.down_sh_s) + ro * (I / 32), *ds1 = ds0 + I / 32;
          // scale words as in phase A: lane l loads word k0 / 128 + l of each row with the codes
          const unsigned *d0w = reinterpret_cast<const unsigned *>(ds0), *d1w = reinterpret_cast<const unsigned *>(ds1);
          for (int k0 = 0; k0 < I; k0 += 512 * UQB) {  // warp-uniform trips, as in phase A
            uint4 w0[UQB], w1[UQB];
            const bool wl = k0 / 128 + lane < I / 128;
            const unsigned word0 = wl ? __ldg(d0w + k0 / 128 + lane) : 0u, word1 = wl ? __ldg(d1w + k0 / 128 + lane) : 0u;
#pragma unroll
            for (int u = 0; u < UQB; ++u) {
              const int cc = k0 + u * 512 + lane * 16;
              if (cc < I) {
                w0[u] = ld_stream(dq0 + cc);
                w1[u] = ld_stream(dq1 + cc);
              }
            }
#pragma unroll
            for (int u = 0; u < UQB; ++u) {
              const int cc = k0 + u * 512 + lane * 16;
              const int src = 4 * u + lane / 8, sh = ((lane >> 1) & 3) * 8;
              const unsigned sw0 = __shfl_sync(0xffffffffu, word0, src);
              const unsigned sw1 = __shfl_sync(0xffffffffu, word1, src);
              if (cc < I) {
                float f0[16], f1[16];
                e4m3x16_to_float_scaled(w0[u], f0);
                e4m3x16_to_float_scaled(w1[u], f1);
                const float sc0 = e8m0_value((sw0 >> sh) & 0xFFu), sc1 = e8m0_value((sw1 >> sh) & 0xFFu);
#pragma unroll
                for (int r = 0; r < kDecodeRows; ++r) {
                  if ((mask >> r) & 1) {
                    const float *ar = act + (size_t)r * I + cc;
                    const float4 x0 = ld_ca4(ar), x1 = ld_ca4(ar + 4), x2 = ld_ca4(ar + 8), x3 = ld_ca4(ar + 12);
                    acc0[r] = fmaf(sc0, dot16(f0, x0, x1, x2, x3) * kE4m3Unscale, acc0[r]);
                    acc1[r] = fmaf(sc1, dot16(f1, x0, x1, x2, x3) * kE4m3Unscale, acc1[r]);
                  }
                }
              }
            }
          }
        } else {
        const uint16_t *dw0 = routed ? a.down_exps + ((size_t)e * D + dd) * I : a.down_sh + (size_t)dd * I;
        const uint16_t *dw1 = dw0 + I;
        for (int base = lane * 8; base < I; base += 256 * UB) {
          uint4 w0[UB], w1[UB];
#pragma unroll
          for (int u = 0; u < UB; ++u) {
            if (base + u * 256 < I) {
              w0[u] = ld_weight(dw0 + base + u * 256);
              w1[u] = ld_weight(dw1 + base + u * 256);
            }
          }
#pragma unroll
          for (int u = 0; u < UB; ++u) {
            const int cc = base + u * 256;
            if (cc < I) {
#pragma unroll
              for (int r = 0; r < kDecodeRows; ++r) {
                if ((mask >> r) & 1) {
                  const float4 x0 = ld_ca4(act + (size_t)r * I + cc);
                  const float4 x1 = ld_ca4(act + (size_t)r * I + cc + 4);
                  acc0[r] += dot8(w0[u], x0, x1);
                  acc1[r] += dot8(w1[u], x0, x1);
                }
              }
            }
          }
        }
        }
#pragma unroll
        for (int r = 0; r < kDecodeRows; ++r) {
          if (r < rows) {
            const float s0 = warp_sum(acc0[r]);
            const float s1 = warp_sum(acc1[r]);
            if (lane == 0) {  // zeros for rows this group does not serve
              const bool use = (mask >> r) & 1;
              a.y[((size_t)g * kDecodeRows + r) * D + dd] = use ? s0 : 0.f;
              a.y[((size_t)g * kDecodeRows + r) * D + dd + 1] = use ? s1 : 0.f;
            }
          }
        }
      }
    }
    if (lane == 0) publish(&dblock_done[d0 / kDecodeDBlock], (unsigned)kRowsPerTicketB);
    c = __shfl_sync(0xffffffffu, next, 0);
  }

  // ---- phase C: per 32-wide d-block, once every group's rows of it are in: ffn_out = sum_g w * y
  // and the hc_post output out_i = post_i * ffn_out + sum_j comb[i, j] * state_j.  The comb term
  // needs no y, so it is formed before the block's wait; the wait then spins (it is short, at the
  // end of the launch) and only the sum over groups follows it.
  const int hc = a.hc;
  const bool comb_ok = wait_at_least(&cnt[kCntComb], 1u, a.status, &cnt[kCntAbort]);
  for (int c = draw_ticket(&cnt[kCntTickC]); c < nblk && comb_ok; c = draw_ticket(&cnt[kCntTickC])) {
    const int d = c * kDecodeDBlock + lane;
    float po[rows][kHcMax], t[rows][kHcMax];
#pragma unroll
    for (int r = 0; r < rows; ++r) {
      float sj[kHcMax];
#pragma unroll
      for (int j = 0; j < kHcMax; ++j) sj[j] = j < hc ? a.state[((size_t)r * hc + j) * D + d] : 0.f;
#pragma unroll
      for (int o = 0; o < kHcMax; ++o) {
        po[r][o] = o < hc ? __ldcg(a.post + r * hc + o) : 0.f;
        float v = 0.f;
#pragma unroll
        for (int j = 0; j < kHcMax; ++j)
          if (o < hc && j < hc) v += __ldcg(a.comb + (r * hc + o) * hc + j) * sj[j];
        t[r][o] = v;
      }
    }
    // Two passes over the same instructions: the first, before the wait and without stores, only
    // brings this code into the instruction cache, so that the second runs warm right after it.
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      const bool live = pass == 1;
      if (live && !wait_at_least(&dblock_done[c], (unsigned)(ng * kDecodeDBlock), a.status, &cnt[kCntAbort], false))
        break;
#pragma unroll
      for (int r = 0; r < rows; ++r) {
        float f = 0.f;
#pragma unroll 8
        for (int g = 0; g < ng; ++g) {
          const float w = __shfl_sync(0xffffffffu, g < 32 ? gt_w0[r] : gt_w1[r], g & 31);
          f += w * __ldcg(a.y + ((size_t)g * kDecodeRows + r) * D + d);
        }
        if (live) a.ffn_out[(size_t)r * D + d] = f;
#pragma unroll
        for (int o = 0; o < kHcMax; ++o)
          if (live && o < hc) a.out_state[((size_t)r * hc + o) * D + d] = po[r][o] * f + t[r][o];
      }
    }
  }

  // ---- the last CTA out resets the counters for the next launch ----
  __threadfence();
  __syncthreads();
  if (tid == 0) sm.flag = atomicAdd(&cnt[kCntExit], 1u) == gridDim.x - 1 ? 1 : 0;
  __syncthreads();
  if (sm.flag) {
    __threadfence();
    for (int i = tid; i < a.n_counters; i += blockDim.x) cnt[i] = 0u;
    // performed before this CTA retires: a decode launch that follows directly (programmatic
    // dependent launch) draws its role ticket before its griddepcontrol.wait
    __threadfence();
  }
}

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------

int decode_mix_ctas(int hc, int hidden) { return (hc * hidden + kMixCols - 1) / kMixCols; }
int decode_router_ctas(int hidden) { return hidden / kRouterChunk; }
int decode_counter_count(const Dims &d) { return kCntDBlocks + d.hidden / kDecodeDBlock; }

using DecodeKernel = void (*)(DecodeArgs);
static DecodeKernel decode_kernel_for(int rows, bool mx) {
  if (mx)
    return rows == 1   ? decode_kernel<1, true>
           : rows == 2 ? decode_kernel<2, true>
           : rows == 3 ? decode_kernel<3, true>
                       : decode_kernel<4, true>;
  return rows == 1   ? decode_kernel<1, false>
         : rows == 2 ? decode_kernel<2, false>
         : rows == 3 ? decode_kernel<3, false>
                     : decode_kernel<4, false>;
}

cudaError_t decode_configure(int hidden) {
  for (int mx = 0; mx < 2; ++mx)
    for (int r = 1; r <= kDecodeRows; ++r) {
      const cudaError_t e = cudaFuncSetAttribute(decode_kernel_for(r, mx != 0),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 r * hidden * (int)sizeof(float));
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

int decode_resident_ctas(int hidden, int rows, int num_sms, bool mx) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel_for(rows, mx), 256,
                                                    (size_t)rows * hidden * sizeof(float)) != cudaSuccess)
    return 0;
  return per_sm * num_sms;
}

void launch_decode(const Dims &d, const Scratch &s, const LayerDev &w, const float *state, const int32_t *token_ids,
                   int rows, bool hash, float *out_state, cudaStream_t st, StageTimer *tm) {
  DecodeArgs a;
  a.state = state;
  a.hc_fn = w.hc_fn;
  a.hc_scale = w.hc_scale;
  a.hc_base = w.hc_base;
  a.norm_w = w.ffn_norm;
  a.gate = w.gate;
  a.rp = make_route(d, s, w, token_ids, hash, nullptr);
  a.gate_exps = w.gate_exps;
  a.up_exps = w.up_exps;
  a.down_exps = w.down_exps;
  a.gate_sh = w.gate_sh;
  a.up_sh = w.up_sh;
  a.down_sh = w.down_sh;
  a.gate_q = w.gate_q;
  a.up_q = w.up_q;
  a.down_q = w.down_q;
  a.gate_sh_q = w.gate_sh_q;
  a.up_sh_q = w.up_sh_q;
  a.down_sh_q = w.down_sh_q;
  a.gate_s = w.gate_s;
  a.up_s = w.up_s;
  a.down_s = w.down_s;
  a.gate_sh_s = w.gate_sh_s;
  a.up_sh_s = w.up_sh_s;
  a.down_sh_s = w.down_sh_s;
  a.nm = decode_mix_ctas(d.hc, d.hidden);
  a.nr = decode_router_ctas(d.hidden);
  a.mix_part = s.mix_partial;
  a.mixes = s.mixes;
  a.pre = s.pre;
  a.post = s.post;
  a.comb = s.comb;
  a.xw = s.ffn_input;
  a.ss_part = s.dec_part;
  a.lg_part = s.dec_part + (size_t)a.nr * kDecodeRows;
  a.row_rs = s.row_rs;
  a.ffn_norm = s.ffn_norm;
  a.logits = s.logits;
  a.ngroups = s.ngroups;
  a.group_e = s.group_e;
  a.group_mask = s.group_mask;
  a.group_w = s.group_w;
  a.act = s.act_dec;
  a.y = s.y_dec;
  a.ffn_out = s.ffn_out;
  a.out_state = out_state;
  a.counters = s.dec_counters;
  a.n_counters = decode_counter_count(d);
  a.status = s.status;
  a.rows = rows;
  a.hidden = d.hidden;
  a.inter = d.inter;
  a.experts = d.experts;
  a.hc = d.hc;
  a.M = d.mix();
  a.iters = d.iters;
  a.mix_chunk = kMixCols;
  a.eps = d.eps;
  const size_t xs_bytes = (size_t)rows * d.hidden * sizeof(float);
  launch_pdl(decode_kernel_for(rows, w.mx), dim3(w.mx ? s.decode_ctas_mx[rows] : s.decode_ctas_by_rows[rows]), dim3(256),
             xs_bytes, st, a);
  stage(tm, "decode", st);
}

}  // namespace moe
