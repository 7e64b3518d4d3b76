// Grouped expert GEMMs of the rows > 4 path on the 5th-generation tensor cores (tcgen05, TMEM,
// TMA), sm_103a.
//
// docs.rs "hf2q 0.1.3 .../deepseek4/ffn_forward.rs", forward_ffn_rows: expert_matmul "routed
// gate"/"routed up" + raw_matmul "shared gate"/"shared up" + dispatch_deepseek_moe_swiglu (fused
// into the gate/up epilogue), and expert_matmul "routed down" + raw_matmul "shared down" with the
// route weight of dispatch_deepseek_moe_weighted_reduce applied in the down epilogue.
//
// Layout ("swap AB"): the expert's weight rows are the MMA's M = 128 side (operand A), the
// expert's tokens the N side (operand B, N = 16..128 by tile), K = hidden (gate/up) or inter
// (down), 64 per pipeline stage.  So a weight tile is read from HBM once per 128 tokens of its
// expert however few tokens that is.  The shared expert is group `experts` (every row), so one
// persistent launch covers routed and shared work.  Operands are fp16 (the weights' bf16 values
// are exact in fp16 above 2^-14; activations get an 11-bit significand), accumulation is f32 in
// TMEM.
//
// Roles per CTA (320 threads, one CTA per SM, persistent over a device-built tile list):
//   warp 0     TMA producer: A (gate and up, or down) and B tiles into a multi-stage smem ring
//   warp 1     TMEM allocator and MMA issuer (one thread), commits free smem stages / TMEM
//   warps 2-9  epilogue: tcgen05.ld of the accumulator (double buffered in TMEM, so the next
//              tile's MMAs run under this tile's epilogue), SwiGLU or route-weight scaling; two
//              warps per TMEM lane quarter, each every other 16-column chunk, so that the
//              epilogue keeps up with the MMAs
// Every mbarrier wait is bounded (2 s); on expiry the CTA raises the device timeout bit, all roles
// leave their loops, and TMEM is freed before the kernel returns.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int BM = 128, BN = 128, BK = 64, UMMA_K = 16;
constexpr int kTileBytes = BM * BK * 2;  // 16 KB: one 128 x 64 fp16 tile (A and B alike)
constexpr uint64_t kWaitLimitNs = 2000000000ull;

template <bool GATEUP>
struct GemmCfg {
  static constexpr int kStages = GATEUP ? 4 : 6;
  static constexpr int kATiles = GATEUP ? 2 : 1;
  static constexpr int kStageBytes = (kATiles + 1) * kTileBytes;
  static constexpr int kAccCols = GATEUP ? 2 * BN : BN;  // gate and up accumulators side by side
  static constexpr int kTmemCols = 2 * kAccCols;         // two accumulator buffers
  static constexpr size_t kSmem = (size_t)kStages * kStageBytes + 1024;
};

struct GemmArgs {
  const int4 *tiles;   // (group, m-block, n-block, valid tokens)
  const int *n_tiles;  // [0] gate/up, [1] down
  const int *offsets;  // first list position of each group
  const int2 *list;    // (row, slot) per position
  const float *list_w;
  __half *act16;       // [positions, inter]
  float *y_slot;       // [rows, top_k + 1, hidden]
  int *status;
  int inter, hidden, top_k, k_blocks, a_rows_per_group, which;
};

constexpr int kEpiWarps = 8, kGemmThreads = 32 * (2 + kEpiWarps);

template <bool GATEUP>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                        const __grid_constant__ CUtensorMap tmB, GemmArgs a) {
  using C = GemmCfg<GATEUP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[C::kStages], empty_bar[C::kStages], tfull_bar[2], tempty_bar[2];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

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
    abort_flag = 0;
    fence_mbar_init();
    tmap_prefetch(&tmA0);
    if (GATEUP) tmap_prefetch(&tmA1);
    tmap_prefetch(&tmB);
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
    for (int t = blockIdx.x; t < ntiles && !*abort_p; t += gridDim.x) {
      const int4 tl = a.tiles[t];
      const int a_row = tl.x * a.a_rows_per_group + tl.y * BM;
      const int b_row = a.offsets[tl.x] + tl.z * BN;
      for (int kb = 0; kb < a.k_blocks; ++kb) {
        if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, abort_p, a.status, kWaitLimitNs)) break;
        mbar_arrive_expect_tx(&full_bar[stage], C::kStageBytes);
        uint8_t *base = smem + (size_t)stage * C::kStageBytes;
        tma_load_2d(base, &tmA0, &full_bar[stage], kb * BK, a_row);
        if (GATEUP) tma_load_2d(base + kTileBytes, &tmA1, &full_bar[stage], kb * BK, a_row);
        tma_load_2d(base + C::kATiles * kTileBytes, &tmB, &full_bar[stage], kb * BK, b_row);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    for (int t = blockIdx.x; t < ntiles && !*abort_p; t += gridDim.x, ++it) {
      const int4 tl = a.tiles[t];
      const int n_mma = (tl.w + 15) & ~15;
      const int acc = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      if (!mbar_wait_bounded(&tempty_bar[acc], acc_phase ^ 1u, abort_p, a.status, kWaitLimitNs)) break;
      tc_fence_after();
      const uint32_t idesc = idesc_f16_f32(BM, n_mma);
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
          const uint64_t bdesc = smem_desc_sw128(sb + k * UMMA_K * 2);
          tc_mma_f16(d0, smem_desc_sw128(sa + k * UMMA_K * 2), bdesc, idesc, accum);
          if (GATEUP) tc_mma_f16(d0 + BN, smem_desc_sw128(sa + kTileBytes + k * UMMA_K * 2), bdesc, idesc, accum);
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
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // which 16-column chunks of the quarter's rows
    const int row = q * 32 + lane;
    const int K1 = a.top_k + 1;
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
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C::kAccCols);
      for (int c0 = half * 16; c0 < n_valid; c0 += 32) {
        if (GATEUP) {
          float gv[16], uv[16];
          tmem_ld16(tbase + c0, gv);
          tmem_ld16(tbase + BN + c0, uv);
          __half *dst = a.act16 + (size_t)(pos0 + c0) * a.inter + tl.y * BM + row;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < n_valid) {
              const float g = gv[j];
              dst[(size_t)j * a.inter] = __float2half_rn(g * sigmoidf_(g) * uv[j]);
            }
          }
        } else {
          float yv[16];
          tmem_ld16(tbase + c0, yv);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < n_valid) {
              const int p = pos0 + c0 + j;
              const int2 rk = a.list[p];
              const float w = a.list_w[p];
              a.y_slot[((size_t)rk.x * K1 + rk.y) * a.hidden + tl.y * BM + row] = yv[j] * w;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[acc]);
    }
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

void launch_grouped_gemms(const Dims &d, const Scratch &s, const LayerDev &w, const CUtensorMap &tm_x16,
                          const CUtensorMap &tm_act16, int num_sms, cudaStream_t st, StageTimer *tm) {
  GemmArgs a;
  a.tiles = s.tiles_gu;
  a.n_tiles = s.n_tiles;
  a.offsets = s.offsets;
  a.list = s.list;
  a.list_w = s.list_w;
  a.act16 = s.act16;
  a.y_slot = s.y_slot;
  a.status = s.status;
  a.inter = d.inter;
  a.hidden = d.hidden;
  a.top_k = d.top_k;
  a.k_blocks = d.hidden / BK;
  a.a_rows_per_group = d.inter;
  a.which = 0;
  const int grid_gu = num_sms < s.max_tiles_gu ? num_sms : s.max_tiles_gu;
  grouped_gemm_kernel<true><<<grid_gu, kGemmThreads, GemmCfg<true>::kSmem, st>>>(w.tm_gate, w.tm_up, tm_x16, a);
  stage(tm, "gemm_gateup", st);
  a.tiles = s.tiles_dn;
  a.k_blocks = d.inter / BK;
  a.a_rows_per_group = d.hidden;
  a.which = 1;
  const int grid_dn = num_sms < s.max_tiles_dn ? num_sms : s.max_tiles_dn;
  grouped_gemm_kernel<false><<<grid_dn, kGemmThreads, GemmCfg<false>::kSmem, st>>>(w.tm_down, w.tm_down, tm_act16, a);
  stage(tm, "gemm_down", st);
}

// bf16 -> fp16 copy of the expert weights for the tensor-core path (init only).
__global__ void bf16_to_f16_kernel(const uint16_t *__restrict__ src, __half *__restrict__ dst, size_t n) {
  const size_t stride = (size_t)gridDim.x * blockDim.x * 8;
  for (size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 8; i < n; i += stride) {
    const uint4 v = *reinterpret_cast<const uint4 *>(src + i);
    __half2 h[4];
    h[0] = __floats2half2_rn(bf_lo(v.x), bf_hi(v.x));
    h[1] = __floats2half2_rn(bf_lo(v.y), bf_hi(v.y));
    h[2] = __floats2half2_rn(bf_lo(v.z), bf_hi(v.z));
    h[3] = __floats2half2_rn(bf_lo(v.w), bf_hi(v.w));
    *reinterpret_cast<uint4 *>(dst + i) = *reinterpret_cast<uint4 *>(h);
  }
}

void launch_bf16_to_f16(const uint16_t *src, __half *dst, size_t n, cudaStream_t st) {
  bf16_to_f16_kernel<<<1024, 256, 0, st>>>(src, dst, n);
}

// MXFP8 (E4M3 codes q[n], E8M0 scales s[n / 32]) to fp16 for the tensor-core operands: each 16-code
// piece of a 32-element block decoded exactly in f32 (code value times 2^(s - 127)), then rounded to
// f16, which is exact whenever the product is an f16 value (scales 2^-15 .. 2^7).
__global__ void mxfp8_to_f16_kernel(const uint8_t *__restrict__ q, const uint8_t *__restrict__ sc,
                                    __half *__restrict__ dst, size_t n) {
  const size_t stride = (size_t)gridDim.x * blockDim.x * 16;
  for (size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 16; i < n; i += stride) {
    float f[16];
    e4m3x16_to_float(*reinterpret_cast<const uint4 *>(q + i), f);
    const float x = e8m0_value(sc[i / 32]);
    __half2 h[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) h[k] = __floats2half2_rn(f[2 * k] * x, f[2 * k + 1] * x);
    *reinterpret_cast<uint4 *>(dst + i) = *reinterpret_cast<uint4 *>(h);
    *reinterpret_cast<uint4 *>(dst + i + 8) = *reinterpret_cast<uint4 *>(h + 4);
  }
}
void launch_mxfp8_to_f16(const uint8_t *q, const uint8_t *s, __half *dst, size_t n, cudaStream_t st) {
  mxfp8_to_f16_kernel<<<1024, 256, 0, st>>>(q, s, dst, n);
}

}  // namespace moe
