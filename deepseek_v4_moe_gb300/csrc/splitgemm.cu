// f32 activations times fp16 weights on the tensor cores (tcgen05, TMEM, TMA), sm_103a: the
// prefill HC mix and router projections.
//
// docs.rs "hf2q 0.1.3 .../deepseek4/ffn_forward.rs", forward_ffn_rows: raw_matmul "HC FFN function"
// (with the sum of squares of rms_norm_no_scale_f32) and raw_matmul "MoE gate".
//
// Both are f32 GEMMs whose results decide integers later (the top-k) or feed a Sinkhorn, so they
// must be about as exact as f32 arithmetic.  Each activation is split x = hi + lo into two fp16
// values (hi = rn(x), lo = rn(x - hi), so |x - hi - lo| <= 2^-22 |x|), the weights are fp16
// copies of the bf16 ones (exact above 2^-14), fp16 x fp16 products are exact in the f32
// accumulator, and two MMAs per k-step (hi and lo) give f32-level dot products at tensor-core
// rate.
//
//   C_part[s, r, n] = sum over k in split s of X[r, k] * W[n, k]
//   ss_part[s, r]   = sum over k in split s of X[r, k]^2           (when asked for)
//
// Layout: A = the 128 activation rows of the tile (M = 128), converted in shared memory by eight
// warps into two 128 x 64 fp16 planes per k-stage in the 128-byte-swizzled K-major layout the MMA
// reads; B = BN weight rows (N = BN), loaded by TMA.  Roles (320 threads, one CTA per SM):
//   warps 0-7  converters: f32 loads (next stage in flight while this one converts), split,
//              swizzled shared stores, sums of squares; then the epilogue (TMEM -> global)
//   warp 8     TMEM allocator and TMA producer of B (one thread)
//   warp 9     MMA issuer (one thread)
// Every mbarrier wait is bounded (2 s); on expiry the device timeout bit is raised, every role
// leaves its loop and TMEM is freed before the kernel returns.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace sg {
constexpr int BM = 128, BK = 64, UMMA_K = 16;
constexpr int kPlaneBytes = BM * BK * 2;  // one 128 x 64 fp16 plane: 16 KB
constexpr int kConvWarps = 8, kThreads = 32 * (kConvWarps + 2);
constexpr uint64_t kWaitNs = 2000000000ull;

template <int BN, int STAGES>
struct Cfg {
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kStageBytes = 2 * kPlaneBytes + kBBytes;
  static constexpr size_t kSmem = (size_t)STAGES * kStageBytes + 1024;
  static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;  // two accumulators
};
}  // namespace sg

struct SplitGemmArgs {
  const float *X;     // [R, K] row-major
  float *c_part;      // [splits, R, ldc]
  float *ss_part;     // [splits, R] or nullptr
  int *status;
  int R, K, N, ldc, kb_per_split, splits, n_tiles;
};

// The 16-byte chunk `c` (0..7) of row `r` of a 128 x 64 fp16 K-major tile in the 128-byte
// swizzled layout: rows of 128 B, 8-row groups 1024 B apart, chunk index XOR-ed with r % 8.
__device__ __forceinline__ uint32_t sw128_chunk(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_half2(__half a, __half b) {
  return (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(sg::kThreads, 1)
    splitgemm_kernel(const __grid_constant__ CUtensorMap tmW, SplitGemmArgs a) {
  using C = sg::Cfg<BN, STAGES>;
  using namespace sg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES], tfull_bar[2], tempty_bar[2];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // work items (row tile, K split, weight tile), this CTA's items b, b + grid, ...
  const int m_tiles = (a.R + BM - 1) / BM, nkb = a.kb_per_split;
  const int n_items = m_tiles * a.splits * a.n_tiles;
  const int my_items = blockIdx.x < n_items ? (n_items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  auto item_of = [&](int i, int &r0, int &split, int &n0) {
    const int it = blockIdx.x + i * gridDim.x;
    r0 = (it % m_tiles) * BM;
    split = (it / m_tiles) % a.splits;
    n0 = (it / (m_tiles * a.splits)) * BN;
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], kConvWarps + 1);  // eight converter warps + the producer's expect_tx
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], kConvWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
    tmap_prefetch(&tmW);
  }
  if (warp == kConvWarps) tmem_alloc(&tmem_base, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  volatile int *abort_p = &abort_flag;

  if (warp < kConvWarps) {
    // ---------------- converters, and the epilogue of the previous item ----------------
    // thread t: row t / 2 of the tile, k half t % 2 (32 values = 8 float4 = 4 chunks per plane)
    const int t = threadIdx.x, row = t >> 1, half = t & 1;
    const int total = my_items * nkb;  // k-blocks this CTA converts, over all of its items
    auto x_at = [&](int g) -> const float * {
      int r0, split, n0;
      item_of(g / nkb, r0, split, n0);
      if (r0 + row >= a.R) return nullptr;
      return a.X + (size_t)(r0 + row) * a.K + (size_t)(split * nkb + g % nkb) * BK + half * 32;
    };
    // drains the accumulator of item i to the global partials
    auto drain = [&](int i) -> bool {
      int ready = 0;
      if (lane == 0) ready = mbar_wait_bounded(&tfull_bar[i & 1], (uint32_t)(i >> 1) & 1u, abort_p, a.status, kWaitNs) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ready, 0)) return false;
      tc_fence_after();
      int r0, split, n0;
      item_of(i, r0, split, n0);
      static_assert(BN % 32 == 0, "each epilogue warp of a lane quarter takes half the columns");
      const int q = warp & 3, er = q * 32 + lane;
      const int cbeg = (warp >> 2) * (BN / 2), cend = cbeg + BN / 2;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)((i & 1) * BN);
      float *dst = a.c_part + ((size_t)split * a.R + r0 + er) * a.ldc + n0;
      for (int c0 = cbeg; c0 < cend; c0 += 16) {
        float v[16];
        tmem_ld16(tbase + c0, v);
        if (r0 + er < a.R) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (n0 + c0 + j < a.N) dst[c0 + j] = v[j];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[i & 1]);
      return true;
    };
    float ss = 0.f;
    float4 cur[8], nxt[8];
    {
      const float *x0 = total > 0 ? x_at(0) : nullptr;
#pragma unroll
      for (int j = 0; j < 8; ++j) cur[j] = x0 ? __ldcs(reinterpret_cast<const float4 *>(x0) + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int g = 0; g < total && ok; ++g) {
      if (g + 1 < total) {
        const float *xn = x_at(g + 1);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          nxt[j] = xn ? __ldcs(reinterpret_cast<const float4 *>(xn) + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      int w_ok = 1;
      if (lane == 0) w_ok = mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, abort_p, a.status, kWaitNs) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
        ok = false;
        break;
      }
      uint8_t *hi_p = smem + (size_t)stage * C::kStageBytes;
      uint8_t *lo_p = hi_p + kPlaneBytes;
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // chunk c of this half: float4 2c and 2c + 1
        uint32_t h[4], l[4];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float4 v = cur[2 * c + q];
          ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
          const __half hx = __float2half_rn(v.x), hy = __float2half_rn(v.y), hz = __float2half_rn(v.z),
                       hw = __float2half_rn(v.w);
          h[2 * q] = pack_half2(hx, hy);
          h[2 * q + 1] = pack_half2(hz, hw);
          l[2 * q] = pack_half2(__float2half_rn(v.x - __half2float(hx)), __float2half_rn(v.y - __half2float(hy)));
          l[2 * q + 1] = pack_half2(__float2half_rn(v.z - __half2float(hz)), __float2half_rn(v.w - __half2float(hw)));
        }
        const uint32_t off = sw128_chunk(row, half * 4 + c);
        *reinterpret_cast<uint4 *>(hi_p + off) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4 *>(lo_p + off) = make_uint4(l[0], l[1], l[2], l[3]);
      }
      // the generic-proxy stores must be visible to the tensor core's async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&full_bar[stage]);
#pragma unroll
      for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
      if (g % nkb == nkb - 1) {  // the last k-block of item i: its sums of squares, then drain item i - 1
        const int i = g / nkb;
        if (a.ss_part) {
          const float s2 = ss + __shfl_xor_sync(0xffffffffu, ss, 1);  // the two halves of the row
          int r0, split, n0;
          item_of(i, r0, split, n0);
          if (half == 0 && r0 + row < a.R && n0 == 0) a.ss_part[(size_t)split * a.R + r0 + row] = s2;
        }
        ss = 0.f;
        if (i > 0 && !drain(i - 1)) ok = false;
      }
    }
    if (ok && my_items > 0) (void)drain(my_items - 1);
  } else if (warp == kConvWarps && lane == 0) {
    // ---------------- TMA producer of the weights ----------------
    int stage = 0;
    uint32_t phase = 0;
    for (int g = 0; g < my_items * nkb && !*abort_p; ++g) {
      int r0, split, n0;
      item_of(g / nkb, r0, split, n0);
      if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, abort_p, a.status, kWaitNs)) break;
      mbar_arrive_expect_tx(&full_bar[stage], C::kBBytes);
      tma_load_2d(smem + (size_t)stage * C::kStageBytes + 2 * kPlaneBytes, &tmW, &full_bar[stage],
                  (split * nkb + g % nkb) * BK, n0);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  } else if (warp == kConvWarps + 1 && lane == 0) {
    // ---------------- MMA issuer: item i accumulates in TMEM buffer i % 2 ----------------
    const uint32_t idesc = idesc_f16_f32(BM, BN);
    int stage = 0;
    uint32_t phase = 0;
    for (int i = 0; i < my_items && !*abort_p; ++i) {
      if (!mbar_wait_bounded(&tempty_bar[i & 1], ((uint32_t)(i >> 1) & 1u) ^ 1u, abort_p, a.status, kWaitNs)) break;
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)((i & 1) * BN);
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait_bounded(&full_bar[stage], phase, abort_p, a.status, kWaitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t shi = smem_u32(smem + (size_t)stage * C::kStageBytes);
        const uint32_t slo = shi + kPlaneBytes, sb = shi + 2 * kPlaneBytes;
#pragma unroll
        for (int k = 0; k < BK / UMMA_K; ++k) {
          const uint64_t bdesc = smem_desc_sw128(sb + k * UMMA_K * 2);
          tc_mma_f16(acc, smem_desc_sw128(shi + k * UMMA_K * 2), bdesc, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          tc_mma_f16(acc, smem_desc_sw128(slo + k * UMMA_K * 2), bdesc, idesc, 1u);
        }
        tc_commit(&empty_bar[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      tc_commit(&tfull_bar[i & 1]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kConvWarps) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------------
// Host side and the mix finish
// ---------------------------------------------------------------------------------------------

constexpr int kMixBN = 32, kMixStages = 5;       // mix: up to 24 outputs, a light B tile
constexpr int kRouterBN = 256, kRouterStages = 3;

cudaError_t splitgemm_configure() {
  cudaError_t e = cudaFuncSetAttribute(splitgemm_kernel<kMixBN, kMixStages>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sg::Cfg<kMixBN, kMixStages>::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(splitgemm_kernel<kRouterBN, kRouterStages>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sg::Cfg<kRouterBN, kRouterStages>::kSmem);
}

// Splits of K.  The tensor cores' f32 accumulation does not round every addition to nearest, so
// its error grows with the number of MMAs accumulated in place; every split therefore sums at most
// kMaxKbPerSplit k-blocks (8 x 2 MMAs of K = 16 each), and the splits are added on the CUDA cores
// in a fixed order.
constexpr int kMaxKbPerSplit = 8;
int splitgemm_splits(int k) {
  const int kb = k / sg::BK;
  int per = kMaxKbPerSplit;
  while (per > 1 && kb % per) per >>= 1;
  return kb / per;
}

// One CTA per SM at most, each with the same number of work items (the last ones possibly one less).
static int persistent_grid(int rows, int splits, int n_tiles, int num_sms) {
  const int items = (rows + sg::BM - 1) / sg::BM * splits * n_tiles;
  const int per = (items + num_sms - 1) / num_sms;
  return (items + per - 1) / per;
}

int mix_tc_part_floats(int max_rows, int hcd) { return splitgemm_splits(hcd) * max_rows * (kMixBN + 1); }

// Per row (one warp): the split partials summed in a fixed order (lane l takes splits l, l + 32,
// ..., then a transpose reduction over the warp gives lane m the sum of output m), then
// mixes = dot * rsqrt(ss / (hc*hidden) + eps), pre = sigmoid, post = 2 sigmoid, and the comb
// (Sinkhorn, the warp-parallel form) of the row.
__global__ void __launch_bounds__(256) mix_finish_kernel(const float *__restrict__ part, const float *__restrict__ ss_part,
                                                         int splits, int rows, int hcd, int M, int hc,
                                                         const float *__restrict__ scale, const float *__restrict__ base,
                                                         int iters, float eps, float *mixes, float *pre, float *post,
                                                         float *comb) {
  const int lane = threadIdx.x & 31, r = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= rows) return;
  static_assert(kMixBN == 32, "one partial row per lane and split");
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = 0.f;
  float ss = 0.f;
  for (int sp = lane; sp < splits; sp += 32) {
    const float4 *p = reinterpret_cast<const float4 *>(part + ((size_t)sp * rows + r) * kMixBN);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 x = __ldcg(p + q);
      v[4 * q] += x.x;
      v[4 * q + 1] += x.y;
      v[4 * q + 2] += x.z;
      v[4 * q + 3] += x.w;
    }
    ss += __ldcg(ss_part + (size_t)sp * rows + r);
  }
  const float dot = transpose_reduce32(v);  // lane m: sum of output m
  ss = warp_sum(ss);
  const float rs = rsqrtf(ss / (float)hcd + eps);
  const float mix = dot * rs;
  if (lane < M) mixes[(size_t)r * M + lane] = mix;
  if (lane < hc) pre[(size_t)r * hc + lane] = sigmoidf_(mix * scale[0] + base[lane]);
  const float mpost = __shfl_sync(0xffffffffu, mix, (hc + lane) & 31);
  if (lane < hc) post[(size_t)r * hc + lane] = 2.0f * sigmoidf_(mpost * scale[1] + base[hc + lane]);
  __syncwarp();
  sinkhorn_comb_warp(mixes + (size_t)r * M, scale, base, hc, iters, comb + (size_t)r * hc * hc);
}

void launch_prefill_mix(const Dims &d, const Scratch &s, const LayerDev &w, const float *state, int rows, int num_sms,
                        cudaStream_t st, StageTimer *tm) {
  const int hcd = d.hc * d.hidden;
  const int splits = splitgemm_splits(hcd);
  SplitGemmArgs a;
  a.X = state;
  a.c_part = s.mix_tc_part;
  a.ss_part = s.mix_tc_part + (size_t)splits * rows * kMixBN;
  a.status = s.status;
  a.R = rows;
  a.K = hcd;
  a.N = d.mix();
  a.ldc = kMixBN;
  a.kb_per_split = hcd / sg::BK / splits;
  a.splits = splits;
  a.n_tiles = 1;
  splitgemm_kernel<kMixBN, kMixStages>
      <<<persistent_grid(rows, splits, 1, num_sms), sg::kThreads, sg::Cfg<kMixBN, kMixStages>::kSmem, st>>>(w.tm_hcfn, a);
  stage(tm, "mix_gemm", st);
  mix_finish_kernel<<<(rows + 7) / 8, 256, 0, st>>>(s.mix_tc_part, a.ss_part, splits, rows, hcd, d.mix(), d.hc,
                                                        w.hc_scale, w.hc_base, d.iters, d.eps, s.mixes, s.pre, s.post,
                                                        s.comb);
  stage(tm, "mix_finish", st);
}

// Router logits of the rows > 4 path: partials [splits, rows, experts] for route_rows_kernel, which
// sums them in a fixed order.  Returns the number of splits.
int launch_router_tc(const Dims &d, const Scratch &s, const LayerDev &w, int rows, int num_sms, cudaStream_t st) {
  const int n_tiles = (d.experts + kRouterBN - 1) / kRouterBN;
  const int splits = splitgemm_splits(d.hidden);  // at most 16 for hidden <= 8192
  SplitGemmArgs a;
  a.X = s.ffn_norm;
  a.c_part = s.router_part;
  a.ss_part = nullptr;
  a.status = s.status;
  a.R = rows;
  a.K = d.hidden;
  a.N = d.experts;
  a.ldc = d.experts;
  a.kb_per_split = d.hidden / sg::BK / splits;
  a.splits = splits;
  a.n_tiles = n_tiles;
  splitgemm_kernel<kRouterBN, kRouterStages>
      <<<persistent_grid(rows, splits, n_tiles, num_sms), sg::kThreads, sg::Cfg<kRouterBN, kRouterStages>::kSmem, st>>>(
          w.tm_router, a);
  return splits;
}

}  // namespace moe
