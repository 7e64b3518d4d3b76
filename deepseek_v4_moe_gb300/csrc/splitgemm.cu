// f32 activations times bf16 weights on the tensor cores (tcgen05, TMEM, TMA), sm_103a: the
// prefill HC mix and router projections.
//
// docs.rs "hf2q 0.1.3 .../deepseek4/ffn_forward.rs", forward_ffn_rows: raw_matmul "HC FFN function"
// (with the sum of squares of rms_norm_no_scale_f32) and raw_matmul "MoE gate".
//
// Both are f32 GEMMs whose results decide integers later (the top-k) or feed a Sinkhorn, so they
// must be about as exact as f32 arithmetic.  The weights are the caller's bf16 matrices, read by
// TMA as they are (no copy).  Each f32 activation is split into three bf16 planes by truncation,
// x = hi + mid + lo + r with hi = trunc(x), mid = trunc(x - hi), lo = trunc(x - hi - mid) (each
// subtraction exact in f32), so |r| < 2^-21 |x| over the whole f32 range; bf16 x bf16 products are
// exact in the f32 accumulator, and three MMAs per k-step (hi, mid, lo against the same weight
// tile) give f32-level dot products at tensor-core rate.
//
//   C_part[s, r, n] = sum over k in split s of X[r, k] * W[n, k]
//   ss_part[s, r]   = sum over k in split s of X[r, k]^2           (when asked for)
//
// Layout: A = the 128 activation rows of a tile (M = 128), converted in shared memory into three
// 128 x 64 bf16 planes per k-stage in the 128-byte-swizzled K-major layout the MMA reads; B = BN
// weight rows (N = BN), loaded by TMA (rows past the matrix arrive as zeros).  Persistent: one CTA
// per SM walks (row tile, K split, weight tile) items.  Roles:
//   next warp  TMEM allocator and activation producer: one 128 x 64 f32 TMA box per k-stage into
//              a ring of f32 slots (the bytes in flight cost no registers)
//   converters (kConvWarps): f32 from shared memory, split, swizzled stores, sums of squares; then
//              the epilogue of the previous item (TMEM -> global), so that it overlaps the next
//              item's MMAs (two TMEM accumulators)
//   next warp  MMA issuer (one thread)
//   last warp  weight producer (one thread, TMA)
// Every wait is bounded (2 s); after a timeout every role leaves its loop, the producers wait
// (bounded) for their own copies in flight and the MMA issuer for its MMAs, then TMEM is freed.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace sg {
constexpr int BM = 128, BK = 64, UMMA_K = 16;
constexpr int kPlaneBytes = BM * BK * 2;  // one 128 x 64 bf16 plane: 16 KB
constexpr int kPlanes = 3;                // hi, mid, lo
constexpr int kXBytes = BM * BK * 4;      // one 128 x 64 f32 activation tile: 32 KB
constexpr int kConvWarps = 8, kThreads = 32 * (kConvWarps + 3);
constexpr int kConvSteps = BM / kConvWarps / 2;  // two tile rows per converter-warp step
constexpr uint64_t kWaitNs = 2000000000ull;

// XS slots of staged f32 activations (bulk copies, so the bytes in flight cost no registers) and
// CS slots of converted bf16 planes with their weight tile
template <int BN, int XS, int CS>
struct Cfg {
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kCBytes = kPlanes * kPlaneBytes + kBBytes;
  static constexpr size_t kSmem = (size_t)XS * kXBytes + (size_t)CS * kCBytes + 1024;
  static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;  // two accumulators
  // converter warps draining an accumulator: groups of four (one per TMEM lane quarter), each
  // group a share of the columns in whole 16-column loads
  static constexpr int kDrainGroups = kConvWarps / 4 < BN / 16 ? kConvWarps / 4 : BN / 16;
  static_assert(kSmem <= 227 * 1024, "shared memory of one CTA");
};
}  // namespace sg

struct SplitGemmArgs {
  const float *X;     // [R, K] row-major
  float *c_part;      // [splits, R, ldc]
  float *ss_part;     // [splits, R] or nullptr
  int *status;
  int R, K, N, ldc, kb_per_split, splits, n_tiles;
};

// The 16-byte chunk `c` (0..7) of row `r` of a 128 x 64 bf16 K-major tile in the 128-byte
// swizzled layout: rows of 128 B, 8-row groups 1024 B apart, chunk index XOR-ed with r % 8.
__device__ __forceinline__ uint32_t sw128_chunk(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// x truncated to bf16 (the low 16 bits cleared), still an f32: x - trunc_bf16(x) is exact in f32.
__device__ __forceinline__ float trunc_bf16(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFF0000u); }

// Four activations as three bf16 planes: hi = trunc(x), mid = trunc(x - hi), lo = trunc(x - hi - mid).
__device__ __forceinline__ void split3(const float4 v, uint2 &hi, uint2 &mid, uint2 &lo) {
  const float x[4] = {v.x, v.y, v.z, v.w};
  float h[4], m[4], l[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    h[k] = trunc_bf16(x[k]);
    const float r1 = x[k] - h[k];
    m[k] = trunc_bf16(r1);
    l[k] = trunc_bf16(r1 - m[k]);
  }
  hi = make_uint2(pack_bf16_pair(h[0], h[1]), pack_bf16_pair(h[2], h[3]));
  mid = make_uint2(pack_bf16_pair(m[0], m[1]), pack_bf16_pair(m[2], m[3]));
  lo = make_uint2(pack_bf16_pair(l[0], l[1]), pack_bf16_pair(l[2], l[3]));
}

template <int BN, int XS, int CS>
__global__ void __launch_bounds__(sg::kThreads, 1)
    splitgemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                     SplitGemmArgs a) {
  using C = sg::Cfg<BN, XS, CS>;
  using namespace sg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *xring = smem, *cring = smem + (size_t)XS * kXBytes;
  __shared__ __align__(8) uint64_t xfull[XS], xempty[XS], cfull[CS], wfull[CS], cempty[CS], tfull[2], tempty[2];
  __shared__ __align__(8) uint64_t mma_done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // work items (row tile, K split, weight tile), this CTA's items b, b + grid, ...
  const int m_tiles = (a.R + BM - 1) / BM, nkb = a.kb_per_split;
  const int n_items = m_tiles * a.splits * a.n_tiles;
  const int my_items = blockIdx.x < n_items ? (n_items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int total = my_items * nkb;  // k-blocks of this CTA over all of its items
  auto item_of = [&](int i, int &r0, int &split, int &n0) {
    const int it = blockIdx.x + i * gridDim.x;
    r0 = (it % m_tiles) * BM;
    split = (it / m_tiles) % a.splits;
    n0 = (it / (m_tiles * a.splits)) * BN;
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < XS; ++s) {
      mbar_init(&xfull[s], 1);            // the producer's expect_tx
      mbar_init(&xempty[s], kConvWarps);  // every converter warp has read the slot
    }
    for (int s = 0; s < CS; ++s) {
      mbar_init(&cfull[s], kConvWarps);  // every converter warp has written its rows
      mbar_init(&wfull[s], 1);           // the weight producer's expect_tx
      mbar_init(&cempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4 * C::kDrainGroups);
    }
    mbar_init(&mma_done, 1);
    abort_flag = 0;
    fence_mbar_init();
    tmap_prefetch(&tmW);
    tmap_prefetch(&tmX);
  }
  if (warp == kConvWarps) tmem_alloc(&tmem_base, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  volatile int *abort_p = &abort_flag;
  // warp-wide bounded wait: lane 0 waits, the warp follows its verdict
  auto warp_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
    int ok = 0;
    if (lane == 0) ok = mbar_wait_bounded(bar, parity, abort_p, a.status, kWaitNs) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
  };

  if (warp < kConvWarps) {
    // ---------------- converters, and the epilogue of the previous item ----------------
    // Warp w converts 2 kConvSteps rows of each tile, two rows per step: lane l takes float4
    // l % 16 of row 2 kConvSteps w + 2j + l / 16 (a conflict-free 512-byte read) and writes its
    // 4 bf16 of each plane as 8 bytes of the row's swizzled 128-byte line.
    auto drain = [&](int i) -> bool {
      if ((warp >> 2) >= C::kDrainGroups) return true;  // not a draining warp
      if (!warp_wait(&tfull[i & 1], (uint32_t)(i >> 1) & 1u)) return false;
      tc_fence_after();
      int r0, split, n0;
      item_of(i, r0, split, n0);
      static_assert(BN % (16 * C::kDrainGroups) == 0, "whole 16-column loads per drain group");
      const int q = warp & 3, er = q * 32 + lane;
      const int cbeg = (warp >> 2) * (BN / C::kDrainGroups), cend = cbeg + BN / C::kDrainGroups;
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
      if (lane == 0) mbar_arrive(&tempty[i & 1]);
      return true;
    };
    const int f4 = lane & 15, sub = lane >> 4;
    float ss[kConvSteps];
#pragma unroll
    for (int j = 0; j < kConvSteps; ++j) ss[j] = 0.f;
    bool ok = true;
    for (int g = 0; g < total && ok; ++g) {
      const int xs = g % XS, cs = g % CS;
      const int i = g / nkb;
      int r0, split, n0;
      item_of(i, r0, split, n0);
      if (!warp_wait(&xfull[xs], (uint32_t)(g / XS) & 1u) || !warp_wait(&cempty[cs], ((uint32_t)(g / CS) & 1u) ^ 1u)) {
        ok = false;
        break;
      }
      const uint8_t *xp = xring + (size_t)xs * kXBytes;
      uint8_t *hi_p = cring + (size_t)cs * C::kCBytes;
      uint8_t *mid_p = hi_p + kPlaneBytes, *lo_p = hi_p + 2 * kPlaneBytes;
#pragma unroll
      for (int j = 0; j < kConvSteps; ++j) {
        const int row = warp * 2 * kConvSteps + 2 * j + sub;
        float4 v = *reinterpret_cast<const float4 *>(xp + row * 256 + f4 * 16);
        if (r0 + row >= a.R) v = make_float4(0.f, 0.f, 0.f, 0.f);  // past this call's rows
        ss[j] += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        uint2 hi, mid, lo;
        split3(v, hi, mid, lo);
        const uint32_t off = sw128_chunk(row, f4 >> 1) + (uint32_t)((f4 & 1) * 8);
        *reinterpret_cast<uint2 *>(hi_p + off) = hi;
        *reinterpret_cast<uint2 *>(mid_p + off) = mid;
        *reinterpret_cast<uint2 *>(lo_p + off) = lo;
      }
      // the generic-proxy stores must be visible to the tensor core's async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&cfull[cs]);
        mbar_arrive(&xempty[xs]);
      }
      if (g % nkb == nkb - 1) {  // the last k-block of item i: its sums of squares, then drain item i - 1
        if (a.ss_part) {
#pragma unroll
          for (int j = 0; j < kConvSteps; ++j) {
            float t = ss[j];
            t += __shfl_xor_sync(0xffffffffu, t, 1);
            t += __shfl_xor_sync(0xffffffffu, t, 2);
            t += __shfl_xor_sync(0xffffffffu, t, 4);
            t += __shfl_xor_sync(0xffffffffu, t, 8);
            const int row = warp * 2 * kConvSteps + 2 * j + sub;
            if (f4 == 0 && r0 + row < a.R && n0 == 0) a.ss_part[(size_t)split * a.R + r0 + row] = t;
          }
        }
#pragma unroll
        for (int j = 0; j < kConvSteps; ++j) ss[j] = 0.f;
        if (i > 0 && !drain(i - 1)) ok = false;
      }
    }
    if (ok && my_items > 0) (void)drain(my_items - 1);
  } else if (warp == kConvWarps && lane == 0) {
    // ---------------- activation producer: one 128 x 64 f32 TMA box per k-stage ----------------
    // (rows past the end of X arrive as zeros)
    int g = 0;
    for (; g < total && !*abort_p; ++g) {
      const int xs = g % XS;
      int r0, split, n0;
      item_of(g / nkb, r0, split, n0);
      if (!mbar_wait_bounded(&xempty[xs], ((uint32_t)(g / XS) & 1u) ^ 1u, abort_p, a.status, kWaitNs)) break;
      mbar_arrive_expect_tx(&xfull[xs], kXBytes);
      tma_load_2d(xring + (size_t)xs * kXBytes, &tmX, &xfull[xs], (split * nkb + g % nkb) * BK, r0);
    }
    // copies still in flight after an abort land before the CTA may leave (bounded; immediate in
    // a normal run)
    int no_abort = 0;
    for (int s = 0; s < XS; ++s) {
      const int n = g / XS + (s < g % XS ? 1 : 0);
      if (n > 0) (void)mbar_wait_bounded(&xfull[s], (uint32_t)((n - 1) & 1), &no_abort, a.status, kWaitNs);
    }
  } else if (warp == kConvWarps + 1 && lane == 0) {
    // ---------------- MMA issuer: item i accumulates in TMEM buffer i % 2 ----------------
    const uint32_t idesc = idesc_bf16_f32(BM, BN);
    int g = 0;
    for (int i = 0; i < my_items && !*abort_p; ++i) {
      if (!mbar_wait_bounded(&tempty[i & 1], ((uint32_t)(i >> 1) & 1u) ^ 1u, abort_p, a.status, kWaitNs)) break;
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)((i & 1) * BN);
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb, ++g) {
        const int cs = g % CS;
        if (!mbar_wait_bounded(&cfull[cs], (uint32_t)(g / CS) & 1u, abort_p, a.status, kWaitNs) ||
            !mbar_wait_bounded(&wfull[cs], (uint32_t)(g / CS) & 1u, abort_p, a.status, kWaitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t shi = smem_u32(cring + (size_t)cs * C::kCBytes);
        const uint32_t sb = shi + kPlanes * kPlaneBytes;
#pragma unroll
        for (int k = 0; k < BK / UMMA_K; ++k) {
          const uint64_t bdesc = smem_desc_sw128(sb + k * UMMA_K * 2);
#pragma unroll
          for (int pl = 0; pl < kPlanes; ++pl)
            tc_mma_f16(acc, smem_desc_sw128(shi + pl * kPlaneBytes + k * UMMA_K * 2), bdesc, idesc,
                       (kb > 0 || k > 0 || pl > 0) ? 1u : 0u);
        }
        tc_commit(&cempty[cs]);
      }
      if (!ok) break;
      tc_commit(&tfull[i & 1]);
    }
    // every MMA issued here completes before TMEM is freed (immediate in a normal run)
    tc_commit(&mma_done);
    int no_abort = 0;
    (void)mbar_wait_bounded(&mma_done, 0u, &no_abort, a.status, kWaitNs);
  } else if (warp == kConvWarps + 2 && lane == 0) {
    // ---------------- weight producer ----------------
    int g = 0;
    for (; g < total && !*abort_p; ++g) {
      const int cs = g % CS;
      int r0, split, n0;
      item_of(g / nkb, r0, split, n0);
      if (!mbar_wait_bounded(&cempty[cs], ((uint32_t)(g / CS) & 1u) ^ 1u, abort_p, a.status, kWaitNs)) break;
      mbar_arrive_expect_tx(&wfull[cs], C::kBBytes);
      tma_load_2d(cring + (size_t)cs * C::kCBytes + kPlanes * kPlaneBytes, &tmW, &wfull[cs], (split * nkb + g % nkb) * BK, n0);
    }
    int no_abort = 0;  // copies in flight land before the CTA may leave, as above
    for (int s = 0; s < CS; ++s) {
      const int n = g / CS + (s < g % CS ? 1 : 0);
      if (n > 0) (void)mbar_wait_bounded(&wfull[s], (uint32_t)((n - 1) & 1), &no_abort, a.status, kWaitNs);
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

constexpr int kMixBN = 32, kMixXS = 3, kMixCS = 2;           // mix: up to 24 outputs, a light B tile
constexpr int kRouterBN = 256, kRouterXS = 2, kRouterCS = 2;

cudaError_t splitgemm_configure() {
  cudaError_t e = cudaFuncSetAttribute(splitgemm_kernel<kMixBN, kMixXS, kMixCS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sg::Cfg<kMixBN, kMixXS, kMixCS>::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(splitgemm_kernel<kRouterBN, kRouterXS, kRouterCS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sg::Cfg<kRouterBN, kRouterXS, kRouterCS>::kSmem);
}

// Splits of K.  The tensor cores' f32 accumulation does not round every addition to nearest, so
// its error grows with the number of MMAs accumulated in place; every split therefore sums at most
// kMaxKbPerSplit k-blocks (8 x 4 k-steps x 3 planes of K = 16 each), and the splits are added on
// the CUDA cores in a fixed order.
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

void launch_prefill_mix(const Dims &d, const Scratch &s, const LayerDev &w, const float *state,
                        const CUtensorMap &tm_state, int rows, int num_sms, cudaStream_t st, StageTimer *tm) {
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
  splitgemm_kernel<kMixBN, kMixXS, kMixCS>
      <<<persistent_grid(rows, splits, 1, num_sms), sg::kThreads, sg::Cfg<kMixBN, kMixXS, kMixCS>::kSmem, st>>>(w.tm_hcfn, tm_state, a);
  stage(tm, "mix_gemm", st);
  mix_finish_kernel<<<(rows + 7) / 8, 256, 0, st>>>(s.mix_tc_part, a.ss_part, splits, rows, hcd, d.mix(), d.hc,
                                                        w.hc_scale, w.hc_base, d.iters, d.eps, s.mixes, s.pre, s.post,
                                                        s.comb);
  stage(tm, "mix_finish", st);
}

// Router logits of the rows > 4 path: partials [splits, rows, experts] for route_rows_kernel, which
// sums them in a fixed order.  Returns the number of splits.
int launch_router_tc(const Dims &d, const Scratch &s, const LayerDev &w, const CUtensorMap &tm_x, int rows, int num_sms,
                     cudaStream_t st) {
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
  splitgemm_kernel<kRouterBN, kRouterXS, kRouterCS>
      <<<persistent_grid(rows, splits, n_tiles, num_sms), sg::kThreads, sg::Cfg<kRouterBN, kRouterXS, kRouterCS>::kSmem, st>>>(
          w.tm_router, tm_x, a);
  return splits;
}

}  // namespace moe
