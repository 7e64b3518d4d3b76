// Grouped expert GEMMs of the rows > 4 path on the 5th-generation tensor cores (tcgen05, TMEM,
// TMA), sm_103a.
//
// docs.rs "hf2q 0.1.3 .../deepseek4/ffn_forward.rs", forward_ffn_rows: expert_matmul "routed
// gate"/"routed up" + raw_matmul "shared gate"/"shared up" + dispatch_deepseek_moe_swiglu (fused
// into the gate/up epilogue), and expert_matmul "routed down" + raw_matmul "shared down" +
// dispatch_deepseek_moe_weighted_reduce (fused into the down epilogue: each token's output column,
// times its route weight, is added into the row's FFN output).
//
// The reduce: a row's top_k + 1 contributions come from different expert tiles, finished by
// different CTAs in no fixed order.  Each contribution is rounded to f32 (y * w, as an f32 reduce
// would take it) and added in f64 at the L2 (red.global.add.f64) into a zeroed f64 row.  The sum
// of at most 9 f32 values is exact in f64 whenever their magnitudes lie within a factor 2^25 of
// each other, so the result, rounded to f32 once by hc_post, does not depend on the order the
// tiles finish in; only a contribution below 2^-25 of a larger one can leave a last-bit difference
// between runs.
//
// Layout ("swap AB"): the expert's weight rows are the MMA's M = 128 side (operand A), the
// expert's tokens the N side (operand B, N = 16..128 by tile), K = hidden (gate/up) or inter
// (down), 64 per pipeline stage.  Every tile holds two A operands against the same B: the gate and
// the up rows of one 128-row block (gate/up), or two adjacent 128-row blocks of the down matrix
// (down).
//
// Pipeline: the weights (A, from DRAM) and the activation planes (B, mostly from L2) sit in two
// rings of 32 KB slots, four for A and three for B.  Step j (one 64-wide k-block of some tile) uses
// A slot j % 4 and B slot j % 3 and completes on full barrier j % 4, which takes two arrivals: the
// A copies of step j are issued one step before its B copies, so three weight slots (96 KB) are in
// flight while the MMAs read the fourth, with the B planes of a 128-token tile still fitting.  So a weight tile is read from HBM once per 128 tokens of its
// expert however few tokens that is, and the B planes are loaded with a box of the tile's own
// N rows (one tensor map per multiple of 16), not 128.  The shared expert is group `experts` (every row), so one
// persistent launch covers routed and shared work.
//
// Precision: the weights are the caller's bf16 matrices, read by TMA as they are.  The activations
// (the normalised input for gate/up, the SwiGLU output for down) are f32 values held as two bf16
// planes, hi = rn(x) and lo = rn(x - hi), so |x - hi - lo| <= 2^-16 |x|; two MMAs per k-step (hi
// and lo against the same weight tile) accumulate in f32 in TMEM, and bf16 x bf16 products are
// exact there.
//
// Roles per CTA (320 threads, one CTA per SM, persistent over a device-built tile list):
//   warp 0     TMA producer: claims tiles (one claim ahead), hands each tile number to the other
//              roles through a small shared-memory queue, and loads A (gate and up, or down) and
//              the two B planes into the rings.  The list has a heavy part (groups of several token
//              blocks: MMA-bound, their weight tiles mostly from L2) and a light part (one token
//              block: bound by the weight bytes).  Even CTAs claim from the heavy part first, odd
//              ones from the light part, each turning to the other part when its own runs out,
//              so the tensor pipes and DRAM are busy together; a device-wide counter per part
//              keeps every SM loaded whatever each tile costs
//   warp 1     TMEM allocator and MMA issuer (one thread), commits free smem stages / TMEM
//   warps 2-9  epilogue: tcgen05.ld of the accumulator (double buffered in TMEM, so the next
//              tile's MMAs run under this tile's epilogue); SwiGLU and the hi/lo split of its
//              output (gate/up), or route-weight scaling and the reduction into the FFN output (down);
//              two warps per TMEM lane quarter, each every other 16-column chunk
// Every mbarrier wait is bounded (2 s unless a test sets a shorter limit); on expiry the CTA raises
// the device timeout bit and all roles leave their loops; before the kernel returns, the producer
// waits (bounded) for its own copies still in flight, the MMA issuer for its MMAs, and TMEM is
// freed.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int BM = 128, BN = 128, BK = 64, UMMA_K = 16;
constexpr int kTileBytes = BM * BK * 2;  // 16 KB: one 128 x 64 bf16 tile (A and B planes alike)

template <bool GATEUP>
struct GemmCfg {
  static constexpr int kSA = 4, kSB = 3;           // A (weight) and B (activation) ring slots
  static constexpr int kLag = kSA - kSB;           // steps by which a step's B copies follow its A copies
  static constexpr int kSlotBytes = 2 * kTileBytes;  // A: the two weight tiles; B: the hi and lo planes
  static constexpr int kAccCols = 2 * BN;                // the two A operands' accumulators side by side
  static constexpr int kTmemCols = 2 * kAccCols;         // two accumulator buffers
  static constexpr size_t kSmem = (size_t)(kSA + kSB) * kSlotBytes + 1024;
  static_assert(kSmem <= 227 * 1024, "shared memory of one CTA");
};

struct GemmArgs {
  const int4 *tiles;   // (group, m-block, n-block, valid tokens); a down m-block is 256 rows
  const int *n_tiles;  // [0] gate/up, [1] down
  int *tile_ctr;       // [2 which], [2 which + 1]: heavy and light tile claim counters, zero on entry
  const int *offsets;  // first list position of each group
  const int2 *list;    // (row, slot) per position
  const float *list_w;
  uint16_t *act2;      // [2 * plane_rows, inter] bf16: SwiGLU output hi plane, then lo plane
  double *ffn_acc;     // [rows, hidden], zero on entry to the down GEMM
  int *status;
  int inter, hidden, k_blocks, a_rows_per_group, which, experts, plane_rows;
  uint64_t wait_ns;  // bound of every wait
  int inject;        // test hook: 2 = CTA 0's MMA issuer of the gate/up GEMM first waits on a barrier nothing arrives at
};

constexpr int kEpiWarps = 8, kGemmThreads = 32 * (2 + kEpiWarps);
constexpr int kTQ = 4;  // tile queue entries (the producer runs at most about two tiles ahead)

template <bool GATEUP>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                        const __grid_constant__ CUtensorMap tmS0, const __grid_constant__ CUtensorMap tmS1,
                        const CUtensorMap *__restrict__ tmB, GemmArgs a) {
  using C = GemmCfg<GATEUP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[C::kSA], emptyA_bar[C::kSA], emptyB_bar[C::kSB], tfull_bar[2], tempty_bar[2];
  __shared__ __align__(8) uint64_t mma_done_bar, never_bar, tq_full[kTQ], tq_empty[kTQ];
  __shared__ int tq[kTQ];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const uint64_t kWaitLimitNs = a.wait_ns;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kSA; ++s) {
      mbar_init(&full_bar[s], 2);  // the A copies' arrival and the B copies' arrival
      mbar_init(&emptyA_bar[s], 1);
    }
    for (int s = 0; s < C::kSB; ++s) mbar_init(&emptyB_bar[s], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], kEpiWarps);
    }
    mbar_init(&mma_done_bar, 1);
    mbar_init(&never_bar, 1);
    for (int i = 0; i < kTQ; ++i) {
      mbar_init(&tq_full[i], 1);              // the producer has written the entry
      mbar_init(&tq_empty[i], 1 + kEpiWarps);  // the MMA issuer and every epilogue warp have read it
    }
    abort_flag = 0;
    fence_mbar_init();
    tmap_prefetch(&tmA0);
    tmap_prefetch(&tmS0);
    tmap_prefetch(&tmA1);
    tmap_prefetch(&tmS1);
    for (int i = 0; i < BN / 16; ++i) tmap_prefetch(&tmB[i]);
  }
  if (warp == 1) tmem_alloc(&tmem_base, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const int ntiles = a.n_tiles[a.which];
  volatile int *abort_p = &abort_flag;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    uint8_t *ringA = smem, *ringB = smem + (size_t)C::kSA * C::kSlotBytes;
    int j = 0;   // steps whose A copies are issued
    int jb = 0;  // steps whose B copies are issued (jb <= j)
    // the B side of the last kLag steps: (activation row, tensor map) of each
    int hist_row[C::kLag > 0 ? C::kLag : 1];
    const CUtensorMap *hist_map[C::kLag > 0 ? C::kLag : 1];
    // B copies of step jb: wait until its slot is free, then both planes onto step jb's full barrier
    auto issue_b = [&](int b_row, const CUtensorMap *mb, int kb) -> bool {
      const int sb = jb % C::kSB;
      if (!mbar_wait_bounded(&emptyB_bar[sb], (uint32_t)((jb / C::kSB) & 1) ^ 1u, abort_p, a.status, kWaitLimitNs))
        return false;
      const int nrows = (int)(mb - tmB) + 1;  // B box height in 16-row groups
      uint64_t *fb = &full_bar[jb % C::kSA];
      mbar_arrive_expect_tx(fb, 2u * (uint32_t)nrows * 16u * BK * 2u);
      uint8_t *bp = ringB + (size_t)sb * C::kSlotBytes;
      tma_load_2d(bp, mb, fb, kb * BK, b_row);
      tma_load_2d(bp + kTileBytes, mb, fb, kb * BK, a.plane_rows + b_row);
      ++jb;
      return true;
    };
    int hist_kb[C::kLag > 0 ? C::kLag : 1];
    bool ok = true;
    const int n_heavy = a.n_tiles[2 + a.which];
    int *ctr_h = a.tile_ctr + 2 * a.which, *ctr_l = ctr_h + 1;
    bool heavy_done = false, light_done = false;
    const bool heavy_first = (blockIdx.x & 1) == 0;
    auto claim = [&]() -> int {  // the next tile, or ntiles once both parts are used up
      for (int pass = 0; pass < 2; ++pass) {
        const bool h = (pass == 0) == heavy_first;
        if (h && !heavy_done) {
          const int t = atomicAdd(ctr_h, 1);
          if (t < n_heavy) return t;
          heavy_done = true;
        }
        if (!h && !light_done) {
          const int t = n_heavy + atomicAdd(ctr_l, 1);
          if (t < ntiles) return t;
          light_done = true;
        }
      }
      return ntiles;
    };
    int next = claim();
    for (int i = 0; ok && !*abort_p; ++i) {
      // hand tile `next` (or the end mark, a number past the list) to the other roles
      const int t = next;
      const int q = i % kTQ;
      if (!mbar_wait_bounded(&tq_empty[q], (uint32_t)((i / kTQ) & 1) ^ 1u, abort_p, a.status, kWaitLimitNs)) break;
      tq[q] = t;
      mbar_arrive(&tq_full[q]);
      if (t >= ntiles) break;
      next = claim();  // used at the next tile: its latency hides under this one
      const int4 tl = a.tiles[t];
      const bool shared = tl.x == a.experts;  // the shared expert's matrices are separate tensors
      const CUtensorMap *m0 = shared ? &tmS0 : &tmA0;
      const CUtensorMap *m1 = shared ? &tmS1 : &tmA1;
      // gate/up: the gate and up rows of block tl.y; down: blocks 2 tl.y and 2 tl.y + 1 (rows past
      // the matrix read as zeros, or as the next expert's rows, whose products are not stored)
      const int a_row = (shared ? 0 : tl.x * a.a_rows_per_group) + tl.y * (GATEUP ? BM : 2 * BM);
      const int b_row = a.offsets[tl.x] + tl.z * BN;
      const int nb = (tl.w + 15) >> 4;  // B box: the tile's tokens in whole 16-row groups
      const CUtensorMap *mb = &tmB[nb - 1];
      for (int kb = 0; kb < a.k_blocks; ++kb) {
        const int sa = j % C::kSA;
        if (!mbar_wait_bounded(&emptyA_bar[sa], (uint32_t)((j / C::kSA) & 1) ^ 1u, abort_p, a.status, kWaitLimitNs)) {
          ok = false;
          break;
        }
        uint64_t *fb = &full_bar[sa];
        mbar_arrive_expect_tx(fb, 2u * kTileBytes);
        uint8_t *ap = ringA + (size_t)sa * C::kSlotBytes;
        tma_load_2d(ap, m0, fb, kb * BK, a_row);
        tma_load_2d(ap + kTileBytes, m1, fb, kb * BK, GATEUP ? a_row : a_row + BM);
        if (C::kLag > 0) {
          if (j >= C::kLag) {  // the B copies of step j - kLag
            const int h = jb % C::kLag;
            if (!issue_b(hist_row[h], hist_map[h], hist_kb[h])) {
              ok = false;
              ++j;
              break;
            }
          }
          hist_row[j % C::kLag] = b_row;
          hist_map[j % C::kLag] = mb;
          hist_kb[j % C::kLag] = kb;
          ++j;
        } else {
          ++j;
          if (!issue_b(b_row, mb, kb)) {
            ok = false;
            break;
          }
        }
      }
    }
    // the B copies of the last steps
    while (ok && jb < j && !*abort_p) {
      const int h = jb % C::kLag;
      if (!issue_b(hist_row[h], hist_map[h], hist_kb[h])) break;
    }
    // after an abort: the B arrival of every step still missing one, so that each full barrier
    // completes once its A copies have landed
    for (; jb < j; ++jb) mbar_arrive(&full_bar[jb % C::kSA]);
    // copies still in flight after an abort land before the CTA may leave: wait (bounded) for the
    // last phase asked of every full barrier (in a normal run each has completed long ago)
    int no_abort = 0;
    for (int s = 0; s < C::kSA; ++s) {
      const int n = j / C::kSA + (s < j % C::kSA ? 1 : 0);
      if (n > 0) (void)mbar_wait_bounded(&full_bar[s], (uint32_t)((n - 1) & 1), &no_abort, a.status, kWaitLimitNs);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    int j = 0;  // step
    int it = 0;
    if (GATEUP && a.inject == 2 && blockIdx.x == 0)  // test hook: a wait that runs out
      (void)mbar_wait_bounded(&never_bar, 0u, abort_p, a.status, kWaitLimitNs);
    for (;; ++it) {
      const int q = it % kTQ;
      if (!mbar_wait_bounded(&tq_full[q], (uint32_t)((it / kTQ) & 1), abort_p, a.status, kWaitLimitNs)) break;
      const int t = tq[q];
      mbar_arrive(&tq_empty[q]);
      if (t >= ntiles || *abort_p) break;
      const int4 tl = a.tiles[t];
      const int n_mma = (tl.w + 15) & ~15;
      const int acc = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      if (!mbar_wait_bounded(&tempty_bar[acc], acc_phase ^ 1u, abort_p, a.status, kWaitLimitNs)) break;
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(BM, n_mma);
      const uint32_t d0 = tmem + (uint32_t)(acc * C::kAccCols);
      bool ok = true;
      for (int kb = 0; kb < a.k_blocks; ++kb, ++j) {
        const int slot_a = j % C::kSA, slot_b = j % C::kSB;
        if (!mbar_wait_bounded(&full_bar[slot_a], (uint32_t)((j / C::kSA) & 1), abort_p, a.status, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + (size_t)slot_a * C::kSlotBytes);
        const uint32_t sb = smem_u32(smem + (size_t)(C::kSA + slot_b) * C::kSlotBytes);
#pragma unroll
        for (int k = 0; k < BK / UMMA_K; ++k) {
          const uint32_t accum = (kb > 0 || k > 0) ? 1u : 0u;
          const uint64_t bhi = smem_desc_sw128(sb + k * UMMA_K * 2);
          const uint64_t blo = smem_desc_sw128(sb + kTileBytes + k * UMMA_K * 2);
          const uint64_t a0 = smem_desc_sw128(sa + k * UMMA_K * 2);
          const uint64_t a1 = smem_desc_sw128(sa + kTileBytes + k * UMMA_K * 2);
          tc_mma_f16(d0, a0, bhi, idesc, accum);
          tc_mma_f16(d0, a0, blo, idesc, 1u);
          tc_mma_f16(d0 + BN, a1, bhi, idesc, accum);
          tc_mma_f16(d0 + BN, a1, blo, idesc, 1u);
        }
        tc_commit(&emptyA_bar[slot_a]);  // both slots are free once these MMAs have read them
        tc_commit(&emptyB_bar[slot_b]);
      }
      if (!ok) break;
      tc_commit(&tfull_bar[acc]);
    }
    // every MMA this thread issued completes before TMEM is freed (immediate in a normal run)
    tc_commit(&mma_done_bar);
    int no_abort = 0;
    (void)mbar_wait_bounded(&mma_done_bar, 0u, &no_abort, a.status, kWaitLimitNs);
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // which 16-column chunks of the quarter's rows
    const int row = q * 32 + lane;
    bool nonfinite = false;
    int it = 0;
    for (;; ++it) {
      // the next tile number from the queue (lane 0 reads it, the warp follows)
      const int qe = it % kTQ;
      int t = 0, got = 0;
      if (lane == 0) {
        got = mbar_wait_bounded(&tq_full[qe], (uint32_t)((it / kTQ) & 1), abort_p, a.status, kWaitLimitNs) ? 1 : 0;
        if (got) {
          t = tq[qe];
          mbar_arrive(&tq_empty[qe]);
        }
      }
      got = __shfl_sync(0xffffffffu, got, 0);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (!got || t >= ntiles) break;
      const int4 tl = a.tiles[t];
      const int acc = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      // One lane waits and the warp follows its verdict, so the warp-collective TMEM loads below
      // always run on the full warp.
      int ready = 0;
      if (lane == 0) ready = mbar_wait_bounded(&tfull_bar[acc], acc_phase, abort_p, a.status, kWaitLimitNs) ? 1 : 0;
      ready = __shfl_sync(0xffffffffu, ready, 0);
      if (!ready) break;
      tc_fence_after();
      const int pos0 = a.offsets[tl.x] + tl.z * BN;
      const int n_valid = tl.w;
      // this lane's weight row: a column of inter (gate/up), or of hidden (down: m and m + 128)
      const int m = tl.y * (GATEUP ? BM : 2 * BM) + row;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C::kAccCols);
      for (int c0 = half * 16; c0 < n_valid; c0 += 32) {
        if (GATEUP) {
          float gv[16], uv[16];
          tmem_ld16(tbase + c0, gv);
          tmem_ld16(tbase + BN + c0, uv);
          uint16_t *dst = a.act2 + (size_t)(pos0 + c0) * a.inter + m;
          const size_t lo_off = (size_t)a.plane_rows * a.inter;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < n_valid) {
              const float g = gv[j];
              const float v = g * sigmoidf_(g) * uv[j];
              nonfinite |= !isfinite(v);
              const float hi = round_bf16(v);
              const float lo = round_bf16(v - hi);
              dst[(size_t)j * a.inter] = (uint16_t)(__float_as_uint(hi) >> 16);
              dst[lo_off + (size_t)j * a.inter] = (uint16_t)(__float_as_uint(lo) >> 16);
            }
          }
        } else {
          float yv[16], yv1[16];
          tmem_ld16(tbase + c0, yv);
          tmem_ld16(tbase + BN + c0, yv1);
          const bool second = m + BM < a.hidden;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < n_valid) {
              const int p = pos0 + c0 + j;
              const int2 rk = a.list[p];
              const float w = a.list_w[p];
              const float v = yv[j] * w, v1 = yv1[j] * w;
              nonfinite |= !isfinite(v) || (second && !isfinite(v1));
              double *dst = a.ffn_acc + (size_t)rk.x * a.hidden + m;
              red_add_f64(dst, (double)v);
              if (second) red_add_f64(dst + BM, (double)v1);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[acc]);
    }
    if (__any_sync(0xffffffffu, nonfinite) && lane == 0) atomicOr(a.status, kDevNonFinite);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

size_t gemm_smem_bytes(bool gateup) { return gateup ? GemmCfg<true>::kSmem : GemmCfg<false>::kSmem; }

cudaError_t gemm_configure() {
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)GemmCfg<true>::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(grouped_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)GemmCfg<false>::kSmem);
}

void launch_grouped_gemms(const Dims &d, const Scratch &s, const LayerDev &w, const CUtensorMap *tm_x2,
                          const CUtensorMap *tm_act2, int num_sms, cudaStream_t st, StageTimer *tm,
                          const DebugOpts &dbg) {
  GemmArgs a;
  a.tiles = s.tiles_gu;
  a.n_tiles = s.n_tiles;
  a.tile_ctr = s.n_tiles + 4;
  a.offsets = s.offsets;
  a.list = s.list;
  a.list_w = s.list_w;
  a.act2 = s.act2;
  a.ffn_acc = s.ffn_acc;
  a.status = s.status;
  a.inter = d.inter;
  a.hidden = d.hidden;
  a.k_blocks = d.hidden / BK;
  a.a_rows_per_group = d.inter;
  a.which = 0;
  a.experts = d.experts;
  a.plane_rows = s.max_positions;
  a.wait_ns = dbg.wait_ns ? dbg.wait_ns : 2000000000ull;
  a.inject = dbg.inject;
  const int grid_gu = num_sms < s.max_tiles_gu ? num_sms : s.max_tiles_gu;
  grouped_gemm_kernel<true><<<grid_gu, kGemmThreads, GemmCfg<true>::kSmem, st>>>(w.tm_gate, w.tm_up, w.tm_gate_sh,
                                                                                  w.tm_up_sh, tm_x2, a);
  stage(tm, "gemm_gateup", st);
  a.tiles = s.tiles_dn;
  a.k_blocks = d.inter / BK;
  a.a_rows_per_group = d.hidden;
  a.which = 1;
  const int grid_dn = num_sms < s.max_tiles_dn ? num_sms : s.max_tiles_dn;
  grouped_gemm_kernel<false><<<grid_dn, kGemmThreads, GemmCfg<false>::kSmem, st>>>(
      w.tm_down, w.tm_down, w.tm_down_sh, w.tm_down_sh, tm_act2, a);
  stage(tm, "gemm_down", st);
}

// MXFP8 (E4M3 codes q[n], E8M0 scales s[n / 32]) to bf16, the operand format of the tensor-core
// path: each code's value times 2^(s - 127), formed exactly in f32, has at most four significant
// bits, so clearing the low 16 bits gives it exactly as bf16 (for products above 2^-133).
__global__ void mxfp8_to_bf16_kernel(const uint8_t *__restrict__ q, const uint8_t *__restrict__ sc,
                                     uint16_t *__restrict__ dst, size_t n) {
  const size_t stride = (size_t)gridDim.x * blockDim.x * 16;
  for (size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 16; i < n; i += stride) {
    float f[16];
    e4m3x16_to_float(*reinterpret_cast<const uint4 *>(q + i), f);
    const float x = e8m0_value(sc[i / 32]);
    uint32_t packed[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) packed[k] = pack_bf16_pair(f[2 * k] * x, f[2 * k + 1] * x);
    *reinterpret_cast<uint4 *>(dst + i) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    *reinterpret_cast<uint4 *>(dst + i + 8) = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  }
}
void launch_mxfp8_to_bf16(const uint8_t *q, const uint8_t *s, uint16_t *dst, size_t n, cudaStream_t st) {
  mxfp8_to_bf16_kernel<<<1024, 256, 0, st>>>(q, s, dst, n);
}

// Sets *flag when one of the n E4M3 codes (n a multiple of 16) is a NaN (S.1111.111): a byte whose
// low seven bits are all ones carries into its top bit when 1 is added to them.
__global__ void e4m3_nan_scan_kernel(const uint8_t *__restrict__ q, size_t n, int *flag) {
  const size_t stride = (size_t)gridDim.x * blockDim.x * 16;
  unsigned any = 0u;
  for (size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 16; i < n; i += stride) {
    const uint4 w = *reinterpret_cast<const uint4 *>(q + i);
    any |= ((w.x & 0x7F7F7F7Fu) + 0x01010101u) | ((w.y & 0x7F7F7F7Fu) + 0x01010101u) |
           ((w.z & 0x7F7F7F7Fu) + 0x01010101u) | ((w.w & 0x7F7F7F7Fu) + 0x01010101u);
  }
  if (__any_sync(0xffffffffu, (any & 0x80808080u) != 0u) && (threadIdx.x & 31) == 0) atomicOr(flag, 1);
}
void launch_e4m3_nan_scan(const uint8_t *q, size_t n, int *flag, cudaStream_t st) {
  e4m3_nan_scan_kernel<<<1024, 256, 0, st>>>(q, n, flag);
}

// The smallest and the largest of n E8M0 scale codes (n a multiple of 16) into mm[0] and mm[1]
// (atomic min / max; mm[0] starts at 255 and mm[1] at 0).
__global__ void e8m0_range_kernel(const uint8_t *__restrict__ sc, size_t n, unsigned *mm) {
  const size_t stride = (size_t)gridDim.x * blockDim.x * 16;
  unsigned lo = 0xFFFFFFFFu, hi = 0u;  // four byte lanes each
  for (size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 16; i < n; i += stride) {
    const uint4 w = *reinterpret_cast<const uint4 *>(sc + i);
    lo = __vminu4(__vminu4(lo, w.x), __vminu4(w.y, __vminu4(w.z, w.w)));
    hi = __vmaxu4(__vmaxu4(hi, w.x), __vmaxu4(w.y, __vmaxu4(w.z, w.w)));
  }
  unsigned l = min(min(lo & 0xFFu, (lo >> 8) & 0xFFu), min((lo >> 16) & 0xFFu, lo >> 24));
  unsigned h = max(max(hi & 0xFFu, (hi >> 8) & 0xFFu), max((hi >> 16) & 0xFFu, hi >> 24));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    l = min(l, __shfl_xor_sync(0xffffffffu, l, o));
    h = max(h, __shfl_xor_sync(0xffffffffu, h, o));
  }
  if ((threadIdx.x & 31) == 0) {
    atomicMin(&mm[0], l);
    atomicMax(&mm[1], h);
  }
}
void launch_e8m0_range(const uint8_t *sc, size_t n, unsigned *mm, cudaStream_t st) {
  e8m0_range_kernel<<<512, 256, 0, st>>>(sc, n, mm);
}

}  // namespace moe
