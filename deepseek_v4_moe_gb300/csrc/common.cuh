// Device helpers shared by the MoE-FFN kernels (sm_103a).
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kHcMax = 4;        // hyper-connection streams supported
constexpr int kMixMax = 24;      // (2 + hc) * hc for hc <= 4
constexpr int kTopKMax = 8;
constexpr int kDecodeRows = 4;   // rows handled by the weight-streaming decode path
constexpr int kExpertsMax = 512;

// Device status bits (mirror MOE_FFN_DEV_* in moe_ffn.h).
constexpr int kDevTokenRange = 0x1;
constexpr int kDevRouteRange = 0x2;
constexpr int kDevNonFinite = 0x4;
constexpr int kDevTimeout = 0x8;

// bf16 pair packed in a 32-bit word: element 2j in the low half, 2j+1 in the high half.
__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// 16-byte read of data used once (weights): non-coherent path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// dot of 8 bf16 (one uint4) with 8 floats
__device__ __forceinline__ float dot8(const uint4 w, const float4 a, const float4 b) {
  float s = bf_lo(w.x) * a.x;
  s = fmaf(bf_hi(w.x), a.y, s);
  s = fmaf(bf_lo(w.y), a.z, s);
  s = fmaf(bf_hi(w.y), a.w, s);
  s = fmaf(bf_lo(w.z), b.x, s);
  s = fmaf(bf_hi(w.z), b.y, s);
  s = fmaf(bf_lo(w.w), b.z, s);
  s = fmaf(bf_hi(w.w), b.w, s);
  return s;
}

// 16-byte streaming read with an L2 eviction-priority policy (see make_policy_*).
// ---- MXFP8 (OCP Microscaling, E4M3 elements, one E8M0 scale per 32 elements) -----------------
// E8M0 scale code -> 2^(s - 127): the code is the float's exponent field (0: 2^-127, a subnormal;
// 255: NaN).
__device__ __forceinline__ float e8m0_value(unsigned s) {
  return __uint_as_float(s == 0u ? 0x00400000u : s == 255u ? 0x7FC00000u : s << 23);
}

// two floats as one 64-bit operand of the packed f32x2 instructions (lo in the low half)
__device__ __forceinline__ unsigned long long pack_f32x2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

// The 16 E4M3 codes of w (element k in byte k) as floats: the hardware converts pairs to f16
// (exact: every E4M3 value is an f16 value), then to f32.
__device__ __forceinline__ void e4m3x16_to_float(const uint4 w, float (&f)[16]) {
  const unsigned words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    unsigned h0, h1;
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n cvt.rn.f16x2.e4m3x2 %1, hi;\n}"
        : "=r"(h0), "=r"(h1)
        : "r"(words[q]));
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&h0));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&h1));
    f[4 * q] = a.x;
    f[4 * q + 1] = a.y;
    f[4 * q + 2] = b.x;
    f[4 * q + 3] = b.y;
  }
}


__device__ __forceinline__ uint4 ld_stream_hint(const void *p, uint64_t policy) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p), "l"(policy));
  return r;
}

__device__ __forceinline__ uint64_t make_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t make_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t make_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Asynchronous prefetch of [p, p + bytes) into L2 (bytes a multiple of 16, p 16-byte aligned).
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes, uint64_t policy) {
  asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p), "r"(bytes), "l"(policy)
               : "memory");
}

// Programmatic dependent launch: wait for the preceding kernel's results / let the next kernel start.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

// Comb of one row from its RMS-scaled mixes (split + Sinkhorn, docs.rs "hf2q 0.1.3
// .../deepseek4/ffn_forward.rs", dispatch_hc_split_sinkhorn), by a whole warp: a[i][j] =
// mix[2hc + i*hc + j] * scale[2] + base[2hc + i*hc + j]; start exp(a - rowmax); `iters` sweeps,
// each normalising every row then every column (multiplying by the correctly rounded reciprocal
// of the sum).  Lane 4i + j (lanes 0-15; 16-31 mirror them) holds entry (i, j).  Row sums pair
// entries as (c0 + c1) + (c2 + c3) through xor shuffles 1 and 2, column sums through xor 4 and 8,
// so every kernel that forms a comb with it gets the same bits.  Lanes 0..hc*hc-1 by (i, j) < hc
// store.  Every lane of the warp must call it.
__device__ inline void sinkhorn_comb_warp(const float *mix, const float *scale, const float *base, int hc, int iters,
                                          float *comb) {
  const int lane = threadIdx.x & 31, i = (lane >> 2) & 3, j = lane & 3;
  const bool in = i < hc && j < hc;
  float c = in ? mix[2 * hc + i * hc + j] * scale[2] + base[2 * hc + i * hc + j] : 0.f;
  float mx = in ? c : -INFINITY;
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  c = in ? expf(c - mx) : 0.f;
#pragma unroll 1
  for (int it = 0; it < iters; ++it) {
    const float r1 = c + __shfl_xor_sync(0xffffffffu, c, 1);
    const float rsum = r1 + __shfl_xor_sync(0xffffffffu, r1, 2);
    c *= i < hc ? __frcp_rn(rsum) : 0.f;
    const float c1 = c + __shfl_xor_sync(0xffffffffu, c, 4);
    const float csum = c1 + __shfl_xor_sync(0xffffffffu, c1, 8);
    c *= j < hc ? __frcp_rn(csum) : 0.f;
  }
  if (lane < 16 && in) comb[i * hc + j] = c;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier / TMA / tcgen05 wrappers (PTX ISA 8.6+, sm_100 family) ------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: returns false (and raises the abort flag and the device timeout bit) when the
// phase has not completed within `limit_ns`, or when another role of the CTA already aborted.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                                  int *dev_status, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicOr(dev_status, kDevTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(void *smem_dst, const void *tmap, uint64_t *bar, int c_inner,
                                            int c_outer) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::
          "r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(smem_u32(bar)), "r"(c_inner), "r"(c_outer)
      : "memory");
}

// 1-D bulk copy global -> shared memory, completion counted on `bar` (bytes: multiple of 16; both
// addresses 16-byte aligned).
__device__ __forceinline__ void tma_bulk_g2s(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(smem_dst)),
               "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ uint4 lds128(const void *p) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(smem_u32(p)));
  return r;
}

// Sum over the warp of 32 values per lane: afterwards lane l holds the sum of every lane's v[l]
// (a butterfly that halves the live values at each of 5 steps: 31 shuffles for 32 sums).
__device__ __forceinline__ float transpose_reduce32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool hi = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = hi ? v[i] : v[i + s];
      const float keep = hi ? v[i + s] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  return v[0];
}

__device__ __forceinline__ void tmap_prefetch(const void *tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// K-major operand tile in shared memory, 128-byte rows, SWIZZLE_128B, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);          // start address
  d |= (uint64_t)1u << 16;                           // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024u >> 4) << 32;                 // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1u << 46;                           // descriptor version (sm_100 family)
  d |= (uint64_t)2u << 61;                           // swizzle mode: 128B
  return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (K-major), f32 accumulator, shape M x N.
__device__ __forceinline__ uint32_t idesc_f16_f32(int M, int N) {
  uint32_t d = 0;
  d |= 1u << 4;                                      // D format: f32
  d |= 0u << 7;                                      // A format: f16
  d |= 0u << 10;                                     // B format: f16
  d |= (uint32_t)(N >> 3) << 17;
  d |= (uint32_t)(M >> 4) << 24;
  return d;
}

// Instruction descriptor, kind::f16 with bf16 A and B (K-major), f32 accumulator, shape M x N.
__device__ __forceinline__ uint32_t idesc_bf16_f32(int M, int N) {
  uint32_t d = 0;
  d |= 1u << 4;                                      // D format: f32
  d |= 1u << 7;                                      // A format: bf16
  d |= 1u << 10;                                     // B format: bf16
  d |= (uint32_t)(N >> 3) << 17;
  d |= (uint32_t)(M >> 4) << 24;
  return d;
}

// x rounded to bf16 (nearest, ties to even), kept as an f32 whose low 16 bits are zero.  Integer
// operations only; a NaN is returned as it is (the rounding add would carry a NaN with a full
// mantissa into the sign bit), and its high half is a bf16 NaN.  For finite x the difference
// x - round_bf16(x) is exact in f32.
__device__ __forceinline__ float round_bf16(float x) {
  uint32_t u = __float_as_uint(x);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return x != x ? x : __uint_as_float(u & 0xFFFF0000u);
}

// Two bf16-valued floats (low 16 bits zero) packed as a bf16 pair: a in the low half, b in the high.
__device__ __forceinline__ uint32_t pack_bf16_pair(float a, float b) {
  return __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x7632);
}

// Fire-and-forget f64 add in global memory (performed at the L2; no return value).
__device__ __forceinline__ void red_add_f64(double *p, double v) {
  asm volatile("red.global.add.f64 [%0], %1;" ::"l"(p), "d"(v) : "memory");
}

__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives on `bar` once all previously issued tcgen05.mma of this thread have completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t *smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 32 lanes x 32-bit, 16 consecutive columns: thread i of the warp gets lane (base + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace moe
