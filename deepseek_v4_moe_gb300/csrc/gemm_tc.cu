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
// (down), so each stage carries 32 KB of weights and three stages keep 96 KB of them in flight.  So a weight tile is read from HBM once per 128 tokens of its
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
//   warp 0     TMA producer: A (gate and up, or down) and the two B planes into a multi-stage ring
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
  static constexpr int kStages = 3;
  static constexpr int kATiles = 2;
  static constexpr int kStageBytes = (kATiles + 2) * kTileBytes;  // A tiles, then B hi and B lo
  static constexpr int kAccCols = 2 * BN;                // the two A operands' accumulators side by side
  static constexpr int kTmemCols = 2 * kAccCols;         // two accumulator buffers
  static constexpr size_t kSmem = (size_t)kStages * kStageBytes + 1024;
  static_assert(kSmem <= 227 * 1024, "shared memory of one CTA");
};

struct GemmArgs {
  const int4 *tiles;   // (group, m-block, n-block, valid tokens); a down m-block is 256 rows
  const int *n_tiles;  // [0] gate/up, [1] down
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

template <bool GATEUP>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                        const __grid_constant__ CUtensorMap tmS0, const __grid_constant__ CUtensorMap tmS1,
                        const CUtensorMap *__restrict__ tmB, GemmArgs a) {
  using C = GemmCfg<GATEUP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[C::kStages], empty_bar[C::kStages], tfull_bar[2], tempty_bar[2];
  __shared__ __align__(8) uint64_t mma_done_bar, never_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const uint64_t kWaitLimitNs = a.wait_ns;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], kEpiWarps);
    }
    mbar_init(&mma_done_bar, 1);
    mbar_init(&never_bar, 1);
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
    int stage = 0;
    uint32_t phase = 0;
    int issued = 0;  // stages handed to TMA
    for (int t = blockIdx.x; t < ntiles && !*abort_p; t += gridDim.x) {
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
      const uint32_t bytes = C::kATiles * kTileBytes + 2u * (uint32_t)nb * 16u * BK * 2u;
      for (int kb = 0; kb < a.k_blocks; ++kb) {
        if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, abort_p, a.status, kWaitLimitNs)) break;
        mbar_arrive_expect_tx(&full_bar[stage], bytes);
        uint8_t *base = smem + (size_t)stage * C::kStageBytes;
        tma_load_2d(base, m0, &full_bar[stage], kb * BK, a_row);
        tma_load_2d(base + kTileBytes, m1, &full_bar[stage], kb * BK, GATEUP ? a_row : a_row + BM);
        uint8_t *bp = base + C::kATiles * kTileBytes;
        tma_load_2d(bp, mb, &full_bar[stage], kb * BK, b_row);
        tma_load_2d(bp + kTileBytes, mb, &full_bar[stage], kb * BK, a.plane_rows + b_row);
        ++issued;
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // copies still in flight after an abort land before the CTA may leave: wait (bounded) for the
    // last phase asked of every stage (in a normal run each has completed long ago)
    int no_abort = 0;
    for (int s = 0; s < C::kStages; ++s) {
      const int n = issued / C::kStages + (s < issued % C::kStages ? 1 : 0);
      if (n > 0) (void)mbar_wait_bounded(&full_bar[s], (uint32_t)((n - 1) & 1), &no_abort, a.status, kWaitLimitNs);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    if (GATEUP && a.inject == 2 && blockIdx.x == 0)  // test hook: a wait that runs out
      (void)mbar_wait_bounded(&never_bar, 0u, abort_p, a.status, kWaitLimitNs);
    for (int t = blockIdx.x; t < ntiles && !*abort_p; t += gridDim.x, ++it) {
      const int4 tl = a.tiles[t];
      const int n_mma = (tl.w + 15) & ~15;
      const int acc = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      if (!mbar_wait_bounded(&tempty_bar[acc], acc_phase ^ 1u, abort_p, a.status, kWaitLimitNs)) break;
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(BM, n_mma);
      const uint32_t d0 = tmem + (uint32_t)(acc * C::kAccCols);
      bool ok = true;
      for (int kb = 0; kb < a.k_blocks; ++kb) {
        if (!mbar_wait_bounded(&full_bar[stage], phase, abort_p, a.status, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + (size_t)stage * C::kStageBytes);
        const uint32_t sb = sa + C::kATiles * kTileBytes;
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
        tc_commit(&empty_bar[stage]);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
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
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
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

}  // namespace moe
