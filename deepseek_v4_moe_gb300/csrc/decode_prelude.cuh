// The decode kernels' shared device code: their arguments and counters, the shared-memory block
// of the prelude, the mix role (HC RMSNorm + mix GEMV + split + Sinkhorn), x formation (hc_pre +
// ffn_norm) in every CTA, the router role (the gate GEMV) and the routing (score or hash top-k and
// the expert groups), as decode.cu describes them.  Included by decode.cu (the CUDA-core kernel)
// and decode_tc.cu (the tensor-core kernel).
#pragma once
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
  float *x;          // [rows, hidden] ffn_norm(ffn_input), written by router CTA 0 (also the stage tap)
  float *sel;        // [4, experts] sigmoid(logit) of each row and expert; all-ones bits until written
                     // in this launch (the last CTA out writes that pattern back)
  float *logits;     // [rows, experts]
  float *act;        // [groups, 4, inter]
  float *y;          // [groups, 4, hidden]
  float *ffn_out, *out_state;
  unsigned *counters;  // kCnt* layout below, zero at launch, zeroed again by the last CTA out
  int n_counters;
  int *status;
  int rows, hidden, inter, experts, hc, M, iters, nm, nr, epc;
  float eps;
  uint64_t wait_ns;  // bound of every wait
  int inject;        // test hook: 1 = phase C first waits for a count that is never reached
};

// counter slots.  The prelude flags share one 128-byte line; the ticket counters, the group
// counters and the d-block counters get lines of their own.
constexpr int kCntRole = 0, kCntMixDone = 1, kCntComb = 6, kCntExit = 7, kCntAbort = 8;
constexpr unsigned kUnwritten = 0xFFFFFFFFu;  // an NaN pattern no arithmetic produces (CUDA's NaN is 0x7FFFFFFF)
constexpr int kCntTick = 32, kCntTickC = 64, kCntGroups = 128;
constexpr int kCntDBlocks = kCntGroups + 64;  // after the group counters, on a fresh line
static_assert(kDecodeGroupsMax <= 64, "group counters fit before the d-block counters");

constexpr uint64_t kSpinLimitNs = 1000000000ull;  // default bound of every wait
constexpr int kWorkerWarps = 8, kWorkers = 32 * kWorkerWarps, kDecThreads = kWorkers + 64;
constexpr int kProducerWarp = kWorkerWarps, kPublisherWarp = kWorkerWarps + 1;
constexpr int kPublishBatch = 16;  // slots a publisher may hold before it publishes their counts
constexpr int kMixCols = 512;     // flattened-state columns per mix CTA (a multiple of 128)
constexpr int kChunk = 4;         // tickets claimed by one atomic of a producer (consecutive slots)
// kind A: each worker thread owns 16 columns of a row (hidden <= 16 x 256 = 4096); kind B: 8
// columns of a down row (inter <= 8 x 256 = 2048); moe_ffn_init enforces both limits
constexpr int kMaxEpc = 4;        // experts per router CTA (64 CTAs up to 256 experts, 128 for 512)

template <bool MX>
struct Ring {
  // bf16: one gate + up row pair (4 hidden bytes) or four down rows (8 inter bytes), 16 KB at most,
  // six slots.  MXFP8 (whose codes take more decoding per byte): two row pairs (4 hidden bytes of
  // codes) or eight down rows (8 inter bytes) and their scales, each scale run copied as the
  // 16-byte-aligned span that holds it, five slots.  Two CTAs per SM: 2 x (96 or 85 KB) of slots.
  static constexpr int kRowsA = MX ? 2 : 1;  // gate/up row pairs per kind-A slot
  static constexpr int kRowsB = MX ? 8 : 4;  // down rows per kind-B slot
  static constexpr int kSlots = MX ? 5 : 6;
  static constexpr int kSlotBytes = MX ? 17408 : 16384;
  static constexpr int kRed = 4 * kRowsB;  // partial sums per warp and slot (4 rows x the down rows at most)
  static constexpr size_t kSmem = (size_t)kSlots * kSlotBytes + (size_t)kSlots * kWorkerWarps * kRed * 4;
};

enum : int { kKindA = 0, kKindB = 1, kKindEnd = 2 };
struct SlotMeta {
  int kind, g, row, e, mask, s0, s1;  // row: i (kind A) or the first of four down rows (kind B)
};

// Shared memory outside the ring (static).
struct DecSmem {
  union {
    alignas(16) float st[kDecodeRows][kMixCols];  // mix role: the state columns
    alignas(16) float sel[kDecodeRows * kExpertsMax];  // routing: the score table as the bulk copy left it
  };
  float bias[kExpertsMax];                        // routing (score layers): exp_probs_b
  int hsel[kDecodeRows][kTopKMax], hbad[kDecodeRows];  // routing (hash layers): tid2eid rows, token out of range
  float sums[kDecodeRows][kMixMax + 1];
  float mixes[kDecodeRows][kMixMax];  // the last mix CTA's mixes, for its publisher's Sinkhorn
  int comb_todo;                      // mix CTAs: 1 = the last one (its publisher forms the comb), 2 = not
  float hc_scale[3], hc_base[kMixMax];
  float red[kWorkerWarps][32];
  float pre[kDecodeRows][kHcMax];
  float rs[kDecodeRows];
  // ring bookkeeping
  SlotMeta meta[8];
  // the producer's (row, slot) pairs while it groups them, then the group table
  float rtw[32];
  int ng;
  int ge[kDecodeGroupsMax], gm[kDecodeGroupsMax];
  float gw[kDecodeGroupsMax][kDecodeRows];
  int flag, abort;
};

__device__ __forceinline__ void workers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kWorkers) : "memory"); }

// Adds n to a completion counter with release semantics: this thread's earlier writes (and those
// ordered before them by a fence) are visible to whoever acquires the new value.
__device__ __forceinline__ void publish(unsigned *counter, unsigned n) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(counter), "r"(n) : "memory");
}
// The same add without ordering of its own (after a fence, it publishes what the fence ordered).
__device__ __forceinline__ void add_relaxed(unsigned *counter, unsigned n) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(counter), "r"(n) : "memory");
}

// Polls (one thread) until *counter >= target, with a bounded wait.  False on timeout; once any
// wait of this launch has timed out (the launch's abort counter), every later wait of the launch
// fails at once, so that a failed launch still ends quickly.
static __device__ bool poll_at_least(const unsigned *counter, unsigned target, const DecodeArgs &a, bool nap = true) {
  if (ld_acquire_u32(counter) >= target) return true;
  unsigned *abort = a.counters + kCntAbort;
  const uint64_t w0 = global_timer_ns();
  while (ld_acquire_u32(counter) < target) {
    if (*reinterpret_cast<volatile unsigned *>(abort) != 0u || global_timer_ns() - w0 > a.wait_ns) {
      atomicOr(a.status, kDevTimeout);
      atomicExch(abort, 1u);
      return false;
    }
    if (nap) __nanosleep(64);
  }
  return true;
}

// Warp-wide bounded wait: lane 0 polls, then every lane acquires the counter so that its later
// reads see what the producers published.
static __device__ bool wait_at_least(const unsigned *counter, unsigned target, const DecodeArgs &a, bool nap = true) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = poll_at_least(counter, target, a, nap) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) (void)ld_acquire_u32(counter);
  return ok != 0;
}

// Worker-wide bounded wait (every worker thread calls it).
static __device__ bool workers_wait_at_least(const unsigned *counter, unsigned target, const DecodeArgs &a, int *s_flag) {
  if (threadIdx.x == 0) *s_flag = poll_at_least(counter, target, a) ? 1 : 0;
  workers_sync();
  const bool ok = *s_flag != 0;
  if (ok) (void)ld_acquire_u32(counter);
  workers_sync();
  return ok;
}

// True in exactly one CTA: the last of `total` to finish its share of a role (all earlier global
// writes of every worker thread of the CTA are fenced before the count).
static __device__ bool workers_arrive_last(unsigned *count, unsigned total, int *s_flag) {
  __threadfence();
  workers_sync();
  if (threadIdx.x == 0) *s_flag = atomicAdd(count, 1u) == total - 1 ? 1 : 0;
  workers_sync();
  const bool last = *s_flag != 0;
  if (last) __threadfence();
  return last;
}

// Next phase-C ticket: lane 0 draws it, the warp shares it.
__device__ __forceinline__ int draw_ticket(unsigned *tick) {
  int c = 0;
  if ((threadIdx.x & 31) == 0) c = (int)atomicAdd(tick, 1u);
  return __shfl_sync(0xffffffffu, c, 0);
}

// The producer and publisher wait with a short sleep between tests, so that their spinning takes
// few issue slots from the worker warps of the SM.
constexpr unsigned kBackoffNs = 64;

// mbar_wait_bounded with a sleep between tests.
__device__ __forceinline__ bool mbar_wait_backoff(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                                  int *dev_status, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    __nanosleep(kBackoffNs);
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicOr(dev_status, kDevTimeout);
      return false;
    }
  }
}

// Warp-wide bounded mbarrier wait: every lane tests the phase; unless all saw it complete, lane 0
// waits (bounded) and the warp follows its verdict.  A timeout also raises the launch's abort flag.
static __device__ bool warp_mbar_wait(uint64_t *bar, uint32_t parity, DecSmem &sm, const DecodeArgs &a) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  int ok = 0;
  if ((threadIdx.x & 31) == 0) {
    ok = mbar_wait_bounded(bar, parity, &sm.abort, a.status, a.wait_ns) ? 1 : 0;
    if (!ok) atomicExch(&a.counters[kCntAbort], 1u);
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
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

// Sum over the warp of V values per lane (V a power of two, at most 32), scattered: afterwards lane
// l holds the warp total of value l % V (V - 1 shuffles halve the live values, then the remaining
// lanes are summed).
template <int V>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[V]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = V / 2; s >= 1; s >>= 1) {
    const bool hi = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = hi ? v[i] : v[i + s];
      const float keep = hi ? v[i + s] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  float x = v[0];
#pragma unroll
  for (int o = V; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__host__ __device__ constexpr int pow2_at_least(int n) { return n <= 1 ? 1 : n <= 2 ? 2 : n <= 4 ? 4 : n <= 8 ? 8 : n <= 16 ? 16 : 32; }

// ---------------------------------------------------------------------------------------------
// Mix role (rms_norm_no_scale_f32 + raw_matmul "HC FFN function" + dispatch_hc_split_sinkhorn).
// Per row: ss = sum x^2 and dot_m = sum x * hc_fn[m] over the flattened hc*hidden state;
// mixes = dot * rsqrt(ss / (hc*hidden) + eps) (the RMS scale factors out of the dot product).
// ---------------------------------------------------------------------------------------------

// Tail of the mix role, run by the last mix CTA's workers: the mixes, pre and post of every row
// (the router and stream CTAs form pre themselves from the same partials).  The comb (Sinkhorn),
// which only the final hc_post needs, is left to the CTA's publisher warp, idle until the first
// slot is full, so that the workers go on to form x at once.
template <int ROWS>
__device__ __noinline__ void mix_tail(const DecodeArgs &a, DecSmem &sm) {
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
  workers_sync();
  if (tid < rows) {
    const float rs = mix_rs(sm.sums[tid][M], hc * a.hidden, a.eps);
    for (int h = 0; h < hc; ++h) {
      a.pre[tid * hc + h] = hc_gate(sm.sums[tid][h], rs, sm.hc_scale[0], sm.hc_base[h]);
      a.post[tid * hc + h] = 2.0f * hc_gate(sm.sums[tid][hc + h], rs, sm.hc_scale[1], sm.hc_base[hc + h]);
    }
    for (int m = 0; m < M; ++m) {
      const float mx = sm.sums[tid][m] * rs;
      a.mixes[tid * M + m] = mx;
      sm.mixes[tid][m] = mx;
    }
  }
  workers_sync();
}

// The comb of every row (split + Sinkhorn) by the last mix CTA's publisher warp, published for
// phase C.
template <int ROWS>
__device__ __noinline__ void mix_comb(const DecodeArgs &a, DecSmem &sm, unsigned *cnt) {
  for (int r = 0; r < ROWS; ++r) sinkhorn_comb_warp(&sm.mixes[r][0], sm.hc_scale, sm.hc_base, a.hc, a.iters, a.comb + r * a.hc * a.hc);
  __threadfence();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) publish(&cnt[kCntComb], 1u);
}

// Mix CTA j: flattened-state columns [j * kMixCols, +kMixCols) (the last chunk may be shorter, a
// multiple of 128).  Warp w forms outputs w, w + 8, w + 16; lane l covers columns 4l + 128p of the
// chunk, so the shared-memory state reads are conflict-free and the hc_fn reads coalesced.
template <int ROWS>
static __device__ void mix_role(const DecodeArgs &a, int j, DecSmem &sm, unsigned *cnt) {
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
  static_assert(kMixCols / 4 <= kWorkers, "one float4 of each row per thread");
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
  workers_sync();
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
  workers_sync();
  if (tid < rows) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWorkerWarps; ++w) s += sm.red[w][tid];
    a.mix_part[((size_t)j * rows + tid) * (M + 1) + M] = s;
  }
  const bool last = workers_arrive_last(&cnt[kCntMixDone], (unsigned)a.nm, &sm.flag);
  if (last) mix_tail<ROWS>(a, sm);
  if (tid == 0) {  // after mix_tail's shared-memory writes
    __threadfence_block();
    *reinterpret_cast<volatile int *>(&sm.comb_todo) = last ? 1 : 2;
  }
}

// ---------------------------------------------------------------------------------------------
// x in every CTA (dispatch_hc_pre + rms_norm), and the router role (raw_matmul "MoE gate" for a
// share of the experts).  Each worker thread owns 16 columns of hidden: bf16 experts, 8t .. 8t + 7
// and 2048 + 8t .. 2048 + 8t + 7 (conflict-free 16-byte reads of a shared-memory weight row);
// MXFP8 experts, 16t .. 16t + 15 (one 16-byte load of codes).  Every CTA forms x on its own
// columns from the mix partials and the state (in L2 by then), with the RMS over the CTA, so no CTA
// waits for another to publish x; router CTA j then adds the logits of experts [j epc, (j + 1)
// epc) over the CTA and publishes their selection scores sigmoid(logit) + bias (f32).
// ---------------------------------------------------------------------------------------------
template <bool MX>
__device__ __forceinline__ int own_col(int tid, int h) { return MX ? 16 * tid + 8 * h : 8 * tid + 2048 * h; }

// The state of row r, streams h < hc, on the own column group g (8 columns), into v[h][0..1].
template <bool MX>
__device__ __forceinline__ void load_state_group(const DecodeArgs &a, int r, int g, float4 (&v)[kHcMax][2]) {
  const int c = own_col<MX>(threadIdx.x, g);
#pragma unroll
  for (int h = 0; h < kHcMax; ++h) {
    const bool in = h < a.hc && c < a.hidden;
    const float4 *sp = reinterpret_cast<const float4 *>(a.state + ((size_t)r * a.hc + h) * a.hidden + c);
    v[h][0] = in ? __ldcg(sp) : make_float4(0.f, 0.f, 0.f, 0.f);
    v[h][1] = in ? __ldcg(sp + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

template <int ROWS, bool MX>
__device__ __forceinline__ void form_x(const DecodeArgs &a, DecSmem &sm, unsigned *cnt, float4 (&xr)[ROWS][4]) {
  constexpr int rows = ROWS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int D = a.hidden, hc = a.hc, M = a.M;
  float4 nw[4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = own_col<MX>(tid, h);
    const float4 *np = reinterpret_cast<const float4 *>(a.norm_w + c);
    nw[2 * h] = c < D ? __ldg(np) : make_float4(0.f, 0.f, 0.f, 0.f);
    nw[2 * h + 1] = c < D ? __ldg(np + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (tid == 0) sm.hc_scale[0] = a.hc_scale[0];
  if (tid < hc) sm.hc_base[tid] = a.hc_base[tid];
  pdl_wait();
  // the state loads of a row and column group go out together (one L2 round trip each); at one or
  // two rows (registers to spare) row 0's first group goes out before the mix partials are read
  constexpr bool kEarly = ROWS <= 2;
  float4 sv0[kHcMax][2];
  if (kEarly) load_state_group<MX>(a, 0, 0, sv0);
  // pre from the mix partials, once every mix CTA has written its own (bounded wait; on timeout
  // the status says so and the values below are not meaningful, but every CTA still finishes)
  (void)workers_wait_at_least(&cnt[kCntMixDone], (unsigned)a.nm, a, &sm.flag);
  {
    // items (r, h < hc) and (r, M): warp w reduces items w and w + 8, ...
    const int per = hc + 1, items = rows * per;
    for (int k = warp; k < items; k += kWorkerWarps) {
      const int r = k / per, h = k - r * per;
      const int m = h < hc ? h : M;
      const float x = warp_sum(mix_item_partial(a, rows * (M + 1), r * (M + 1) + m, lane));
      if (lane == 0) sm.sums[r][h] = x;
    }
  }
  workers_sync();
  if (tid < rows * hc) {
    const int r = tid / hc, h = tid - r * hc;
    sm.pre[r][h] = hc_gate(sm.sums[r][h], mix_rs(sm.sums[r][hc], hc * D, a.eps), sm.hc_scale[0], sm.hc_base[h]);
  }
  workers_sync();
  // ffn_input = sum_h pre[h] * state[h] on the own columns, and its sum of squares per row
  float ssq[kDecodeRows] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int r = 0; r < rows; ++r) {
#pragma unroll
    for (int i = 0; i < 4; ++i) xr[r][i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      float4 sv[kHcMax][2];
      if (kEarly && r == 0 && g == 0) {
#pragma unroll
        for (int h = 0; h < kHcMax; ++h) {
          sv[h][0] = sv0[h][0];
          sv[h][1] = sv0[h][1];
        }
      } else {
        load_state_group<MX>(a, r, g, sv);
      }
      // streams in order h = 0, 1, ... (absent streams add zeros)
#pragma unroll
      for (int h = 0; h < kHcMax; ++h) {
        const float ph = h < hc ? sm.pre[r][h] : 0.f;
        const float4 s0 = sv[h][0], s1 = sv[h][1];
        xr[r][2 * g] = make_float4(xr[r][2 * g].x + ph * s0.x, xr[r][2 * g].y + ph * s0.y, xr[r][2 * g].z + ph * s0.z,
                                   xr[r][2 * g].w + ph * s0.w);
        xr[r][2 * g + 1] = make_float4(xr[r][2 * g + 1].x + ph * s1.x, xr[r][2 * g + 1].y + ph * s1.y,
                                       xr[r][2 * g + 1].z + ph * s1.z, xr[r][2 * g + 1].w + ph * s1.w);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
      ssq[r] += xr[r][i].x * xr[r][i].x + xr[r][i].y * xr[r][i].y + xr[r][i].z * xr[r][i].z + xr[r][i].w * xr[r][i].w;
  }
  {
    float t4[4] = {ssq[0], ssq[1], ssq[2], ssq[3]};
    const float s = warp_reduce_scatter<4>(t4);  // lane l: the warp total of row l % 4
    if (lane < 4) sm.red[warp][lane] = s;
  }
  workers_sync();
  // x = ffn_input * rs * norm weight, rs = rsqrt(mean(ffn_input^2) + eps) over the CTA's columns
  // (all of hidden); CTA 0 also writes x out (the ffn_norm stage tap)
#pragma unroll
  for (int r = 0; r < rows; ++r) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kWorkerWarps; ++w) tot += sm.red[w][r];
    const float rs = rsqrtf(tot / (float)D + a.eps);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      xr[r][i] = make_float4(xr[r][i].x * rs * nw[i].x, xr[r][i].y * rs * nw[i].y, xr[r][i].z * rs * nw[i].z,
                             xr[r][i].w * rs * nw[i].w);
    if (blockIdx.x == 0) {
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const int c = own_col<MX>(tid, g);
        if (c < D) {
          float4 *xp = reinterpret_cast<float4 *>(a.x + (size_t)r * D + c);
          xp[0] = xr[r][2 * g];
          xp[1] = xr[r][2 * g + 1];
        }
      }
    }
  }
  workers_sync();  // sm.red is free again
}

// Router CTA j: its experts' rows of the router matrix go to L2 at launch (they do not depend on
// the previous kernel), and are read on the own columns once x is formed.
__device__ __forceinline__ void router_prefetch(const DecodeArgs &a, int j) {
  const int e0 = j * a.epc, ne = min(a.epc, a.experts - e0);
  if ((int)threadIdx.x < ne) prefetch_l2(a.gate + (size_t)(e0 + threadIdx.x) * a.hidden, (uint32_t)(a.hidden * 2), make_policy_evict_last());
}

template <int ROWS, bool MX>
__device__ __forceinline__ void router_logits(const DecodeArgs &a, DecSmem &sm, unsigned *cnt, int j,
                                           const float4 (&xr)[ROWS][4]) {
  constexpr int rows = ROWS;
  const RouteParams &p = a.rp;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.experts, D = a.hidden;
  const int e0 = j * a.epc, ne = min(a.epc, E - e0);
  uint4 gw[kMaxEpc][2];
#pragma unroll
  for (int q = 0; q < kMaxEpc; ++q)
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const int c = own_col<MX>(tid, g);
      gw[q][g] = q < ne && c < D ? __ldg(reinterpret_cast<const uint4 *>(a.gate + (size_t)(e0 + q) * D + c))
                                 : make_uint4(0u, 0u, 0u, 0u);
    }
  // item q * ROWS + r: expert e0 + q, row r; summed over the CTA (lane l of each warp holds the
  // warp total of item l, then warp 0 adds the warps' totals)
  constexpr int V = pow2_at_least(kMaxEpc * ROWS);
  float lp[V];
#pragma unroll
  for (int i = 0; i < V; ++i) lp[i] = 0.f;
#pragma unroll
  for (int q = 0; q < kMaxEpc; ++q)
#pragma unroll
    for (int r = 0; r < rows; ++r)
      lp[q * ROWS + r] = dot8(gw[q][0], xr[r][0], xr[r][1]) + dot8(gw[q][1], xr[r][2], xr[r][3]);
  const float wt = warp_reduce_scatter<V>(lp);
  if (lane < V) sm.red[warp][lane] = wt;
  workers_sync();
  if (warp == 0) {
    bool bad = false;
    if (lane < ne * ROWS) {
      float l = 0.f;
#pragma unroll
      for (int w = 0; w < kWorkerWarps; ++w) l += sm.red[w][lane];
      const int q = lane / ROWS, r = lane - q * ROWS, e = e0 + q;
      bad = !isfinite(l);
      a.logits[(size_t)r * E + e] = l;  // the stage tap
      // one 4-byte store, the NaN made canonical so that it never reads as the unwritten pattern
      // (no fence or counter: the producers copy the table until no entry holds that pattern)
      const float sg = sigmoidf_(l);
      a.sel[(size_t)r * E + e] = isnan(sg) ? __uint_as_float(0x7FFFFFFFu) : sg;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, kDevNonFinite);
  }
  workers_sync();  // sm.red is free again
}

// ---------------------------------------------------------------------------------------------
// Routing, by each CTA's producer warp once the router CTAs have written every score: the top_k
// of each row on sigmoid(logit) + bias (f32; ties to the lower expert index; slots in descending
// order), or the tid2eid row of its token (hash layers); weights = the chosen sigmoid(logit)
// normalised over the valid slots.  Then the (row, slot) pairs are grouped by expert: group 0 is
// the shared expert (weight 1 for every row), then the distinct routed experts in order of first
// appearance, each with the mask of rows using it and their summed route weights.  CTA 0 also
// writes the idx / weight / safe-index outputs and the status bits.
//
// The producer never blocks on the scores while it still has weight rows to fill: it keeps one
// bulk copy of the rows' sigmoid(logit) table (rows x experts f32) in flight into shared memory and
// looks at it between fills; a copy that still holds the unwritten pattern anywhere is issued
// again.  The bias and the hash rows (which do not depend on the scores) are read at launch.
// ---------------------------------------------------------------------------------------------

// Non-blocking look at an mbarrier phase.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// At launch (producer warp): the bias into shared memory (score layers), or each row's tid2eid
// entries (hash layers; -1 for a token out of range, whose status bit CTA 0 raises).
template <int ROWS>
__device__ __forceinline__ void route_setup(const DecodeArgs &a, DecSmem &sm) {
  const RouteParams &p = a.rp;
  const int lane = threadIdx.x & 31, E = a.experts, K = p.top_k;
  if (!p.hash) {
    for (int e = lane; e < E; e += 32) sm.bias[e] = p.bias[e];
  } else {
    pdl_wait();  // the token ids come from the previous kernel
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      const int tok = p.token_ids[r];
      const bool tok_ok = tok >= 0 && tok < p.vocab;
      if (!tok_ok && lane == 0 && blockIdx.x == 0) atomicOr(p.status, kDevTokenRange);
      if (lane < K) sm.hsel[r][lane] = tok_ok ? p.tid2eid[(size_t)tok * K + lane] : -1;
      if (lane == 0) sm.hbad[r] = tok_ok ? 0 : 1;
    }
  }
  __syncwarp();
}

// The group table from the score table in shared memory (sm.sel, row stride experts).  `dry`:
// the same instructions on whatever shared memory holds, without any global write, run once at
// launch so that the code is in L2 when the scores arrive (the weight stream and the L2 flush of
// a benchmark evict it between launches; code that runs once per launch otherwise pays the
// instruction-fetch latency line by line).  Its table is overwritten by the live run.
template <int ROWS, int J2>  // J2: candidates per lane, experts / 32 rounded up to 8 or 16
__device__ __noinline__ void route_compute(const DecodeArgs &a, DecSmem &sm, bool dry) {
  constexpr int rows = ROWS;
  const RouteParams &p = a.rp;
  const int lane = threadIdx.x & 31, E = a.experts, K = p.top_k;
  const bool live = blockIdx.x == 0 && !dry;
  int sel[rows];
  float wgt[rows];
#pragma unroll
  for (int r = 0; r < rows; ++r) {
    const float *s_row = sm.sel + r * E;
    int my_sel = -1;
    if (!p.hash) {
      float v[J2];
#pragma unroll
      for (int jj = 0; jj < J2; ++jj) {
        const int e = lane + 32 * jj;
        const float key = e < E ? s_row[e] + sm.bias[e] : -INFINITY;
        v[jj] = isnan(key) ? -INFINITY : key;
      }
      uint32_t taken = 0;
#pragma unroll 1
      for (int k = 0; k < K; ++k) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int jj = 0; jj < J2; ++jj) {
          const int e = lane + 32 * jj;
          if (e < E && !((taken >> jj) & 1u) && (v[jj] > bv || be == 0x7fffffff)) {
            bv = v[jj];
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
      if (lane < K) my_sel = sm.hsel[r][lane];
      const bool bad_entry = !sm.hbad[r] && lane < K && !(my_sel >= 0 && my_sel < E);
      if (__any_sync(0xffffffffu, bad_entry) && lane == 0 && live) atomicOr(p.status, kDevRouteRange);
    }
    const bool valid = lane < K && my_sel >= 0 && my_sel < E;
    const float sc = valid ? s_row[my_sel] : 0.f;  // sigmoid(logit) as the router CTA formed it
    const float tot = warp_sum(sc);
    const float w = lane < K && tot > 0.f ? sc / tot : 0.f;
    if (lane < K && live) {
      p.idx[r * K + lane] = my_sel;
      p.rw[r * K + lane] = w;
      p.safe[r * K + lane] = valid ? (unsigned)my_sel : 0u;
    }
    sel[r] = my_sel;
    wgt[r] = w;
  }
  // lane rr * K + k takes slot k of row rr (rows * top_k <= 32)
  const int rr = lane / K, kk = lane - rr * K;
  int e = -1;
  float wl = 0.f;
#pragma unroll
  for (int r = 0; r < rows; ++r) {
    const int se = __shfl_sync(0xffffffffu, sel[r], kk & 31);
    const float sw = __shfl_sync(0xffffffffu, wgt[r], kk & 31);
    if (rr == r) {
      e = se;
      wl = sw;
    }
  }
  const bool valid = lane < rows * K && e >= 0 && e < E;
  sm.rtw[lane] = wl;
  __syncwarp();
  const unsigned same = __match_any_sync(0xffffffffu, valid ? e : E + 1 + lane);
  const unsigned below = (1u << lane) - 1u;
  const bool leader = valid && (same & below) == 0u;
  const unsigned leaders = __ballot_sync(0xffffffffu, leader);
  if (leader) {
    const int g = 1 + __popc(leaders & below);
    int mask = 0;
    float w0 = 0.f, w1 = 0.f, w2 = 0.f, w3 = 0.f;
    for (unsigned m = same; m != 0u; m &= m - 1u) {
      const int b = __ffs(m) - 1, rb = b / K;
      const float wb = sm.rtw[b];
      mask |= 1 << rb;
      if (rb == 0) w0 += wb;
      else if (rb == 1) w1 += wb;
      else if (rb == 2) w2 += wb;
      else w3 += wb;
    }
    sm.ge[g] = e;
    sm.gm[g] = mask;
    sm.gw[g][0] = w0;
    sm.gw[g][1] = w1;
    sm.gw[g][2] = w2;
    sm.gw[g][3] = w3;
  }
  if (lane == 0) {
    sm.ge[0] = E;
    sm.gm[0] = (1 << rows) - 1;
    for (int r = 0; r < kDecodeRows; ++r) sm.gw[0][r] = r < rows ? 1.f : 0.f;
    sm.ng = 1 + __popc(leaders);
  }
  __syncwarp();
}

template <int ROWS>
__device__ __forceinline__ void route_compute(const DecodeArgs &a, DecSmem &sm, bool dry) {
  if (a.experts <= 256) route_compute<ROWS, 8>(a, sm, dry);
  else route_compute<ROWS, 16>(a, sm, dry);
}

// The producer's view of the score table: one bulk copy of it in flight at a time.
struct ScorePoll {
  uint64_t *bar;
  uint32_t phase;    // parity of the copy in flight
  bool in_flight;
  bool routed;       // the group table is the live one
  uint64_t t0;       // first issue (bound of the wait)
};

__device__ __forceinline__ void score_copy_issue(const DecodeArgs &a, DecSmem &sm, ScorePoll &q, int rows) {
  if ((threadIdx.x & 31) == 0) {
    const uint32_t bytes = (uint32_t)(rows * a.experts * 4);  // experts % 16 == 0: a multiple of 16
    mbar_arrive_expect_tx(q.bar, bytes);
    tma_bulk_g2s(sm.sel, a.sel, bytes, q.bar);
  }
  q.in_flight = true;
}

// Looks at the copy in flight (blocking: until the table is complete, bounded); when it has landed
// and every entry is written, forms the group table.  Returns q.routed.  Warp-uniform.
template <int ROWS>
static __device__ bool score_poll(const DecodeArgs &a, DecSmem &sm, unsigned *cnt, ScorePoll &q, bool block) {
  const int lane = threadIdx.x & 31;
  if (q.routed) return true;
  for (;;) {
    int landed = 0;
    if (lane == 0) landed = mbar_test_wait(q.bar, q.phase) ? 1 : 0;
    if (__shfl_sync(0xffffffffu, landed, 0)) {
      q.phase ^= 1u;
      q.in_flight = false;
      bool pending = false;
      for (int i = lane; i < ROWS * a.experts; i += 32) pending |= __float_as_uint(sm.sel[i]) == kUnwritten;
      if (!__any_sync(0xffffffffu, pending)) {
        route_compute<ROWS>(a, sm, false);
        q.routed = true;
        return true;
      }
      // the reads above come before the next copy's writes to the same bytes
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      score_copy_issue(a, sm, q, ROWS);
    }
    if (!block) return false;
    if (global_timer_ns() - q.t0 > a.wait_ns || *reinterpret_cast<volatile unsigned *>(&cnt[kCntAbort]) != 0u ||
        *reinterpret_cast<volatile int *>(&sm.abort) != 0) {
      if (lane == 0) {
        atomicOr(a.status, kDevTimeout);
        atomicExch(&cnt[kCntAbort], 1u);
      }
      // give up: a table of the shared expert only, so that the stream and phase C end at once
      if (lane == 0) {
        sm.ge[0] = a.experts;
        sm.gm[0] = (1 << ROWS) - 1;
        for (int r = 0; r < kDecodeRows; ++r) sm.gw[0][r] = r < ROWS ? 1.f : 0.f;
        sm.ng = 1;
      }
      __syncwarp();
      q.routed = true;
      return true;
    }
    __nanosleep(64);
  }
}

}  // namespace moe
