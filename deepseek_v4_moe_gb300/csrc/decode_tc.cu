// Decode path (rows <= 4) on the tensor cores: the whole FFN block in one persistent launch, one
// CTA per SM, for bf16 experts and for MXFP8 experts.
//
// docs.rs "hf2q 0.1.3 .../deepseek4/ffn_forward.rs", forward_ffn_rows, every stage in order, as in
// decode.cu: the prelude (mix CTAs, x in every CTA, router CTAs, routing by every producer) is the
// same code.  What differs is the expert stream: instead of CUDA-core dot products, the weight
// tiles go by TMA into a shared-memory ring and tcgen05.mma multiplies them, in TMEM, against the
// batch rows held in shared memory as bf16 hi and lo planes (x = hi + lo with |x - hi - lo| <=
// 2^-16 |x|, the same split as the rows > 4 path).
//
// Layout of one MMA ("swap AB"): A = 128 weight rows x 64 k (a 16 KB tile, 128-byte swizzled, as
// TMA leaves it); B = 16 rows x 64 k: rows 0-3 the hi planes of batch rows 0-3, rows 4-7 their lo
// planes (rows 8-15 are never read back); D = 128 x 16 f32 in TMEM, column r + column 4 + r being
// the dot of weight row i with batch row r.
//
// Work units, claimed from per-split queues so that every CTA keeps its own K range:
//   kind A  (group g, 128-row block of inter, K split s of hidden): the gate and the up tiles of
//           each 64-wide k-step (32 KB a step) against the CTA's slice of x, which its worker
//           threads wrote into shared memory once x was formed.  The partial dots are added in
//           f64 at the L2 (red.add.f64: the sum of the few f32 partials is exact, so it does not
//           depend on their order); the last of the splits of a (g, block, lane quarter) forms
//           SwiGLU, stores act as bf16 hi/lo planes, and publishes the group's progress.
//   kind B  (group g, two 128-row blocks of hidden, K split s of inter): two down tiles a step
//           against the group's act planes, loaded by TMA once the group's act is complete.  The
//           epilogue scales each batch row by its route weight and adds it in f64 into the FFN
//           output; each 32-row block of hidden counts the units that have landed.
// Every CTA draws all of its kind A units before its first kind B unit, and a kind B unit waits only
// for kind A work, which running CTAs hold: every wait ends.
//
// MXFP8 experts: the producer streams the E4M3 code tiles by TMA (64-byte swizzle) into a code ring and
// copies each unit's E8M0 scales with cp.async; warps 4-7 turn every k-step's codes into exact f16
// weights (see e4m3x16_scaled_f16) and store them into an A slot in TMEM, which the MMAs read in
// place of a shared-memory A tile (so the widened weights never pass through shared memory).  The
// batch rows are then three f16 planes (split3_f16) instead of the bf16 hi / lo pair, in B rows
// r, 4 + r and 8 + r, and the MMAs run kind::f16 with f16 operands.
//
// Roles: warps 0-7 run the prelude, then the epilogue (two groups of four alternating units, one TMEM
// lane quarter per warp; MXFP8: warps 0-3 take every unit and warps 4-7 convert);
// warp 8 is the producer (routing, unit claims, TMA), warp 9 the MMA issuer and TMEM owner.  Phase C
// (per 32-wide block of hidden: ffn_out and hc_post) is shared by all warps at the end.  Waits are
// bounded (1 s); after a timeout every later wait fails at once, the producer waits (bounded) for
// its copies in flight and the MMA issuer for its MMAs, and TMEM is freed.  The last CTA out resets
// the counters and the score table; the f64 accumulators are left zero by the roles that read them.
#include "common.cuh"
#include "decode_prelude.cuh"
#include "kernels.h"

namespace moe {

namespace dtc {
constexpr int kStages = 5;                 // bf16 experts: A ring slots of 32 KB, filled by TMA
constexpr int kStagesMx = 4;               // MXFP8 experts: A slots in TMEM (64 columns: two tiles of f16
                                           // pairs) the converter warps fill
constexpr int kCodeStages = 8;             // MXFP8 experts: code slots (two 128 x 64 code tiles) filled by TMA
constexpr int kCodeTile = 128 * 64;        // one code tile, 8 KB
constexpr int kCodeSlot = 2 * kCodeTile;   // 16 KB
constexpr int kScaleSlot = 2 * 128 * 16;   // one unit's scales: [tile][row][16 bytes], one byte per 32 k
constexpr int kTile = 128 * 64 * 2;        // one A tile, 16 KB
constexpr int kSlotBytes = 2 * kTile;      // gate + up tile, or two down tiles
constexpr int kBTile = 16 * 64 * 2;        // one B tile (16 rows x 64 k), 2 KB
constexpr int kMaxChunks = 8;              // 64-wide k-chunks of one unit
constexpr int kBSlice = kMaxChunks * kBTile;  // 16 KB: x slice, or one act slice
constexpr int kEpiWarps = 4;
constexpr int kConvWarps = 4;              // MXFP8 experts: warps 4-7 convert, warps 0-3 run the epilogue
constexpr int kMmaWarp = 9;
constexpr int kTQ = 4;                     // unit queue entries
constexpr int kTmemCols = 64;              // two accumulator buffers of 32 columns
constexpr int kTmemColsMx = 512;           // MXFP8: the accumulators, then the A slots from column 64
constexpr size_t kSmem = (size_t)kStages * kSlotBytes + 3 * kBSlice + 1024;
constexpr size_t kSmemMx = (size_t)kCodeStages * kCodeSlot + 2 * kScaleSlot + 3 * kBSlice + 1024;
static_assert(kTmemCols + kStagesMx * 64 <= kTmemColsMx, "TMEM of the MXFP8 instance");
static_assert(kSmem <= 227 * 1024 - sizeof(DecSmem) - 512, "shared memory of one CTA");
static_assert(kSmemMx <= 227 * 1024 - sizeof(DecSmem) - 512, "shared memory of one CTA (MXFP8 experts)");
static_assert(kEpiWarps + kConvWarps == kWorkerWarps, "the worker warps split into epilogue and converters");
enum : int { kUnitA = 0, kUnitB = 1, kUnitEnd = 2 };
}  // namespace dtc

// Tensor maps of one launch (grid constants): the layer's bf16 expert matrices (boxes of 64 k x 128
// rows), the act planes (boxes of 64 k x 16 rows), and for MXFP8 layers the E4M3 code matrices
// (boxes of 64 codes x 128 rows).
struct DecodeTcMaps {
  CUtensorMap gate, up, down, gate_sh, up_sh, down_sh, act2;
  CUtensorMap gate_q, up_q, down_q, gate_sh_q, up_sh_q, down_sh_q;
};

// Where the tensor-core kernel keeps its f64 partial sums and act planes, and how its K range is
// split (host-computed).
struct DecodeTcArgs {
  double *acc_gu;   // [groups, 2, 4, inter]: gate and up partial sums (zero between launches)
  double *acc_y;    // [4, hidden]: route-weighted FFN output (zero between launches)
  uint16_t *act2;   // [groups, 16, inter]: bf16 experts, rows 0-3 the bf16 hi planes of act, rows 4-7
                    // the lo planes; MXFP8 experts, rows 0-3 / 4-7 / 8-11 its three f16 planes
  int sa, ca;       // kind A: K splits of hidden and 64-wide chunks per split
  int sb, cb;       // kind B: K splits of inter and chunks per split
  int cnt_tick_a, cnt_tick_b, cnt_units;  // counter slots: per-split tickets, SwiGLU unit counts
  int n_acc_gu, n_acc_y;                  // element counts of the two accumulators
  int mx_c;                               // MXFP8 experts: the f16 weights are code x 2^(S - 127 + mx_c)
  float mx_unscale;                       // 2^-mx_c
};

// Counter slots of the tensor-core kernel past the d-block counters: the kind A and kind B tickets
// of each K split (a 128-byte line each, up to 64 splits), then the SwiGLU unit counts per (group,
// 128-row block of inter, lane quarter).
constexpr int kMaxSplits = 64;
static int tc_counter_base(const Dims &d) { return kCntDBlocks + d.hidden / kDecodeDBlock; }
int decode_tc_counter_count(const Dims &d) {
  return tc_counter_base(d) + 2 * kMaxSplits * 32 + kDecodeGroupsMax * (d.inter / 128) * 4;
}

__device__ __forceinline__ void tma_load_2d_hint(void *smem_dst, const void *tmap, uint64_t *bar, int c_inner,
                                                 int c_outer, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
      "%4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(smem_u32(bar)), "r"(c_inner), "r"(c_outer), "l"(policy)
      : "memory");
}

// Byte offset of element (row n, k) in a 16-row x 64-k bf16 tile with the 128-byte swizzle that TMA
// writes and the MMA descriptors expect: 16-byte chunk k / 8 of row n lands at chunk (k / 8) ^ (n % 8).
__device__ __forceinline__ uint32_t btile_offset(int n, int k) {
  return (uint32_t)(n * 128 + ((((k >> 3) ^ (n & 7)) & 7) << 4) + (k & 7) * 2);
}

// hi = rn(x), lo = rn(x - hi) of 8 values, packed as bf16.
__device__ __forceinline__ void split8(const float4 a, const float4 b, uint4 &hi, uint4 &lo) {
  const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float h[8], l[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    h[j] = round_bf16(v[j]);
    l[j] = round_bf16(v[j] - h[j]);
  }
  hi = make_uint4(pack_bf16_pair(h[0], h[1]), pack_bf16_pair(h[2], h[3]), pack_bf16_pair(h[4], h[5]),
                  pack_bf16_pair(h[6], h[7]));
  lo = make_uint4(pack_bf16_pair(l[0], l[1]), pack_bf16_pair(l[2], l[3]), pack_bf16_pair(l[4], l[5]),
                  pack_bf16_pair(l[6], l[7]));
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned *p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ double ld_cg_f64(const double *p) {
  double v;
  asm volatile("ld.global.cg.f64 %0, [%1];" : "=d"(v) : "l"(p) : "memory");
  return v;
}

// ---- MXFP8 experts on the f16 tensor path ----
// A layer whose E8M0 scales all lie within 22 binades of its largest, Smax, streams its weights as
// A' = code x 2^(S - 127 + c) in f16, c = 134 - Smax: the largest |A'| is 448 x 2^7 < 65504, and the
// smallest nonzero one, 2^-9 x 2^(S - Smax + 7) >= 2^-24, is still a multiple of f16's finest step;
// with at most 4 significant bits a code, every A' is exact.  The batch rows are f16 planes too
// (split3_f16), and the epilogue multiplies by 2^-c.  Layers outside that range, or with a NaN code
// or scale, decode on the CUDA-core kernel.

// f16 bits of 2^k (k in [-24, 15]) in both halves
__device__ __forceinline__ uint32_t f16x2_pow2(int k) {
  const uint32_t h = k >= -14 ? (uint32_t)(k + 15) << 10 : 1u << (k + 24);
  return h * 0x00010001u;
}
// 16 E4M3 codes (element k in byte k) times 2^k (fac = f16x2_pow2(k)), as 16 f16 (elements 0-7 in o0,
// 8-15 in o1): the hardware turns each code pair into an f16 pair, exactly, and one f16 multiply by
// the power of two scales it, exactly (by the range argument above).
__device__ __forceinline__ void e4m3x16_scaled_f16(const uint4 q, uint32_t fac, uint4 &o0, uint4 &o1) {
  const unsigned words[4] = {q.x, q.y, q.z, q.w};
  uint32_t p[8];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    unsigned h0, h1;
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n cvt.rn.f16x2.e4m3x2 %1, hi;\n}"
        : "=r"(h0), "=r"(h1)
        : "r"(words[w]));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(p[2 * w]) : "r"(h0), "r"(fac));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(p[2 * w + 1]) : "r"(h1), "r"(fac));
  }
  o0 = make_uint4(p[0], p[1], p[2], p[3]);
  o1 = make_uint4(p[4], p[5], p[6], p[7]);
}

// 32 consecutive TMEM columns of this thread's lane (32x32b shape: lane 32 (warp % 4) + laneid)
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
// D (+)= A B^T with A (128 rows x 16 k, f16) in TMEM at column a_tmem, B from shared memory
__device__ __forceinline__ void tc_mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// x as three f16 planes, x ~ 2^16 p0 + 2^5 p1 + 2^-6 p2, each plane the f16 rounding of what the
// planes before it left (the residuals are exact in f32).  For |x| < 2^32 every plane is in range and
// |x - sum| <= 2^-33 |x| + 2^-31; beyond, p0 is infinite.  The epilogue weighs the three column
// groups of the MMA output the same way (mx_planes).
__device__ __forceinline__ void split3_f16(float x, uint16_t &p0, uint16_t &p1, uint16_t &p2) {
  const __half h0 = __float2half_rn(x * 0x1p-16f);
  const float r0 = x - __half2float(h0) * 0x1p16f;
  const __half h1 = __float2half_rn(r0 * 0x1p-5f);
  const float r1 = r0 - __half2float(h1) * 0x1p5f;
  const __half h2 = __float2half_rn(r1 * 0x1p6f);
  p0 = __half_as_ushort(h0);
  p1 = __half_as_ushort(h1);
  p2 = __half_as_ushort(h2);
}
__device__ __forceinline__ uint32_t pack_u16(uint16_t lo, uint16_t hi) { return (uint32_t)lo | ((uint32_t)hi << 16); }
__device__ __forceinline__ void split3_f16x8(const float4 a, const float4 b, uint4 &q0, uint4 &q1, uint4 &q2) {
  const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint16_t h[3][8];
#pragma unroll
  for (int j = 0; j < 8; ++j) split3_f16(v[j], h[0][j], h[1][j], h[2][j]);
  q0 = make_uint4(pack_u16(h[0][0], h[0][1]), pack_u16(h[0][2], h[0][3]), pack_u16(h[0][4], h[0][5]),
                  pack_u16(h[0][6], h[0][7]));
  q1 = make_uint4(pack_u16(h[1][0], h[1][1]), pack_u16(h[1][2], h[1][3]), pack_u16(h[1][4], h[1][5]),
                  pack_u16(h[1][6], h[1][7]));
  q2 = make_uint4(pack_u16(h[2][0], h[2][1]), pack_u16(h[2][2], h[2][3]), pack_u16(h[2][4], h[2][5]),
                  pack_u16(h[2][6], h[2][7]));
}
// batch row r's dot from a row of MMA output: bf16 experts, columns r (hi) + 4 + r (lo); MXFP8 experts,
// the three planes' columns r, 4 + r, 8 + r, weighed as split3_f16 split them, times 2^-c
template <bool MX>
__device__ __forceinline__ float plane_sum(const float (&v)[16], int r, float unscale) {
  if (MX) return unscale * (v[r] * 0x1p16f + v[4 + r] * 0x1p5f + v[8 + r] * 0x1p-6f);
  return v[r] + v[4 + r];
}

// One unit's E8M0 scales into a scale slot ([tile][row][16 bytes]; byte b of a row is the scale of
// the unit's 32-wide k-block b): for each of the two tiles, `rows` rows from src[t] on, `stride`
// bytes apart, `nbytes` (<= 16) bytes a row.  The producer warp's lanes copy them with cp.async
// where every row start is 4-byte aligned, with plain loads otherwise; each lane then arrives once
// on `bar` (32 arrivals), the cp.async ones when the copies have landed.
__device__ __forceinline__ void scale_copy(uint8_t *dst, const uint8_t *src0, const uint8_t *src1, int rows0,
                                           int rows1, int stride, int nbytes, uint64_t *bar, int lane) {
  const uint8_t *src[2] = {src0, src1};
  const int rows[2] = {rows0, rows1};
  const uintptr_t al = reinterpret_cast<uintptr_t>(src0) | reinterpret_cast<uintptr_t>(src1) |
                       (uintptr_t)stride | (uintptr_t)nbytes;
  const int w = (al & 15) == 0 ? 16 : (al & 7) == 0 ? 8 : (al & 3) == 0 ? 4 : 0;
  if (w) {
#pragma unroll
    for (int t = 0; t < 2; ++t)
      for (int n = lane; n < rows[t]; n += 32)
        for (int b = 0; b < nbytes; b += w) {
          const uint32_t d = smem_u32(dst + t * 2048 + n * 16 + b);
          const uint8_t *sp = src[t] + (size_t)n * stride + b;
          if (w == 16)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(sp) : "memory");
          else if (w == 8)
            asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(d), "l"(sp) : "memory");
          else
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(sp) : "memory");
        }
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
  } else {
#pragma unroll
    for (int t = 0; t < 2; ++t)
      for (int n = lane; n < rows[t]; n += 32)
        for (int b = 0; b < nbytes; ++b) dst[t * 2048 + n * 16 + b] = __ldg(src[t] + (size_t)n * stride + b);
    mbar_arrive(bar);
  }
}

template <int ROWS, bool MX>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_tc_kernel(const __grid_constant__ DecodeTcMaps tm, DecodeArgs a, DecodeTcArgs t) {
  using namespace dtc;
  constexpr int rows = ROWS;
  constexpr int NA = MX ? kStagesMx : kStages;  // A slots (bf16: shared memory; MXFP8: TMEM)
  constexpr int kCols = MX ? kTmemColsMx : kTmemCols;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *codes = ring + (MX ? 0 : (size_t)NA * kSlotBytes);     // MXFP8: the code ring
  uint8_t *scales = codes + (MX ? (size_t)kCodeStages * kCodeSlot : 0);  // MXFP8: two scale slots
  uint8_t *xs = scales + (MX ? 2 * kScaleSlot : 0);  // this CTA's slice of x as B tiles
  uint8_t *as = xs + kBSlice;                          // two act slices
  __shared__ __align__(16) DecSmem sm;
  __shared__ __align__(8) uint64_t full_bar[NA], empty_bar[NA], tfull[2], tempty[2], afull[2], aempty[2];
  __shared__ __align__(8) uint64_t xready, score_bar, tq_full[kTQ], tq_empty[kTQ], mma_done;
  // MXFP8: code slots (TMA in, converters out) and scale slots (producer in, converters out)
  __shared__ __align__(8) uint64_t code_full[MX ? kCodeStages : 1], code_empty[MX ? kCodeStages : 1];
  __shared__ __align__(8) uint64_t scale_full[2], scale_empty[2];
  __shared__ int4 tq[kTQ];
  __shared__ uint32_t tmem_base;
  unsigned *cnt = a.counters;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int D = a.hidden, I = a.inter, E = a.experts;
  if (tid == 0) {
    for (int s = 0; s < NA; ++s) {
      mbar_init(&full_bar[s], MX ? kConvWarps : 1);  // MXFP8: each converter warp's share of the slot
      mbar_init(&empty_bar[s], 1);
    }
    if (MX) {
      for (int s = 0; s < kCodeStages; ++s) {
        mbar_init(&code_full[s], 1);
        mbar_init(&code_empty[s], kConvWarps);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(&scale_full[b], 32);  // one arrival per producer lane
        mbar_init(&scale_empty[b], kConvWarps);
      }
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kEpiWarps);
      mbar_init(&afull[b], 1);
      mbar_init(&aempty[b], 1);
    }
    mbar_init(&xready, 1);
    mbar_init(&score_bar, 1);
    for (int q = 0; q < kTQ; ++q) {
      mbar_init(&tq_full[q], 1);
      mbar_init(&tq_empty[q], 1 + kWorkerWarps);  // the MMA issuer and the eight worker warps
    }
    mbar_init(&mma_done, 1);
    sm.abort = 0;
    sm.comb_todo = 0;
    sm.flag = (int)atomicAdd(&cnt[kCntRole], 1u);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&tmem_base, kCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int role = sm.flag;
  const uint32_t tmem = tmem_base;
  __syncthreads();

  unsigned *group_done = cnt + kCntGroups;
  unsigned *dblock_done = cnt + kCntDBlocks;
  const int ka = (int)blockIdx.x % t.sa, kbs = (int)blockIdx.x % t.sb;  // this CTA's K splits
  const int rba = I / 128, rbb = (D + 255) / 256;  // kind A row blocks, kind B row-block pairs

  if (warp < kWorkerWarps) {
    // ================= prelude (every worker warp), then the epilogue (warps 0-3) =================
    const bool router = role >= a.nm && role < a.nm + a.nr;
    if (router) router_prefetch(a, role - a.nm);
    if (role < a.nm) mix_role<ROWS>(a, role, sm, cnt);
    float4 xr[rows][4];
    form_x<ROWS, false>(a, sm, cnt, xr);  // (x and the logits do not depend on the expert format)
    if (router) router_logits<ROWS, false>(a, sm, cnt, role - a.nm, xr);
    // this CTA's K slice of x as B tiles: batch row r's hi plane in tile row r, its lo plane in row 4 + r
    const int k0 = ka * t.ca * 64, k1 = k0 + t.ca * 64;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = own_col<false>(tid, h);
      if (c >= k0 && c < k1 && c < D) {
        const int kk = c - k0;
        uint8_t *tile = xs + (size_t)(kk >> 6) * kBTile;
#pragma unroll
        for (int r = 0; r < rows; ++r) {
          if (MX) {  // three f16 planes in rows r, 4 + r, 8 + r
            uint4 q0, q1, q2;
            split3_f16x8(xr[r][2 * h], xr[r][2 * h + 1], q0, q1, q2);
            *reinterpret_cast<uint4 *>(tile + btile_offset(r, kk & 63)) = q0;
            *reinterpret_cast<uint4 *>(tile + btile_offset(4 + r, kk & 63)) = q1;
            *reinterpret_cast<uint4 *>(tile + btile_offset(8 + r, kk & 63)) = q2;
          } else {
            uint4 hi, lo;
            split8(xr[r][2 * h], xr[r][2 * h + 1], hi, lo);
            *reinterpret_cast<uint4 *>(tile + btile_offset(r, kk & 63)) = hi;
            *reinterpret_cast<uint4 *>(tile + btile_offset(4 + r, kk & 63)) = lo;
          }
        }
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the MMAs read them through the async proxy
    workers_sync();
    if (tid == 0) mbar_arrive(&xready);
    if (warp == kEpiWarps && role < a.nm) {
      // the last mix CTA's warp 4 forms the comb before it joins the epilogue
      int todo = 0;
      const uint64_t t0 = global_timer_ns();
      while ((todo = *reinterpret_cast<volatile int *>(&sm.comb_todo)) == 0) {
        if (global_timer_ns() - t0 > a.wait_ns) {
          if (lane == 0) {
            atomicOr(a.status, kDevTimeout);
            atomicExch(&cnt[kCntAbort], 1u);
          }
          break;
        }
        __nanosleep(32);
      }
      __threadfence_block();
      __syncwarp();
      if (todo == 1) mix_comb<ROWS>(a, sm, cnt);
    }
    if (MX && warp >= kEpiWarps) {
      // ---------------- converters (MXFP8 experts): each k-step's two 128 x 64 code tiles times
      // their scales, as f16 weights into an A slot in TMEM, where the MMAs read them (row i of a
      // tile in TMEM lane i, f16 pair (2c, 2c + 1) in column c of its 32).  Warp w converts rows
      // 32 (w - 4) .. + 31, its own TMEM lane quarter, one row a thread; TMA leaves the code tiles
      // with the 64-byte swizzle, so that the 16-byte chunk c of row n sits at chunk c ^ ((n / 2) % 4)
      // and a warp's reads of one chunk from 32 rows are conflict-free. ----------------
      const int cw = warp - kEpiWarps, n = cw * 32 + lane;
      const uint32_t tq_lane = tmem + ((uint32_t)(cw * 32) << 16);
      int j = 0;  // k-steps converted
      for (int u = 0;; ++u) {
        const int q = u % kTQ;
        int4 e = make_int4(kUnitEnd, 0, 0, 0);
        int ok = 0;
        if (lane == 0) {
          ok = mbar_wait_bounded(&tq_full[q], (uint32_t)((u / kTQ) & 1), &sm.abort, a.status, a.wait_ns) ? 1 : 0;
          if (ok) {
            e = tq[q];
            mbar_arrive(&tq_empty[q]);
          } else {
            atomicExch(&cnt[kCntAbort], 1u);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        const int kind = __shfl_sync(0xffffffffu, e.x, 0) & 15;
        if (kind == kUnitEnd) break;
        // every lane tests each phase itself once the warp's verdict is in (its own acquire of the
        // copies; a phase that has completed cannot complete again while this warp holds the slot)
        if (!warp_mbar_wait(&scale_full[u & 1], (uint32_t)((u >> 1) & 1), sm, a)) break;
        (void)mbar_try_wait(&scale_full[u & 1], (uint32_t)((u >> 1) & 1));
        const uint8_t *sc = scales + (size_t)(u & 1) * kScaleSlot;
        const int nc = kind == kUnitA ? t.ca : t.cb;
        bool good = true;
        for (int c = 0; c < nc; ++c, ++j) {
          const int cs = j % kCodeStages, s = j % NA;
          const uint32_t pc = (uint32_t)((j / kCodeStages) & 1), pa = (uint32_t)((j / NA) & 1) ^ 1u;
          if (!warp_mbar_wait(&code_full[cs], pc, sm, a) || !warp_mbar_wait(&empty_bar[s], pa, sm, a)) {
            good = false;
            break;
          }
          (void)mbar_try_wait(&code_full[cs], pc);
          tc_fence_after();  // the MMAs that read this A slot before are complete
          const uint8_t *src = codes + (size_t)cs * kCodeSlot + n * 64;
          // the row's codes (both tiles) and scales first, so that the conversions overlap
          uint4 qv[8];
          unsigned sv[4];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            qv[i] = *reinterpret_cast<const uint4 *>(src + (i >> 2) * kCodeTile + (((i & 3) ^ ((n >> 1) & 3)) << 4));
#pragma unroll
          for (int i = 0; i < 4; ++i) sv[i] = sc[(i >> 1) * 2048 + n * 16 + 2 * c + (i & 1)];
#pragma unroll
          for (int tt = 0; tt < 2; ++tt) {
            uint32_t v[32];
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
              uint4 o0, o1;
              e4m3x16_scaled_f16(qv[tt * 4 + ch], f16x2_pow2((int)sv[tt * 2 + (ch >> 1)] - 127 + t.mx_c), o0, o1);
              v[ch * 8 + 0] = o0.x, v[ch * 8 + 1] = o0.y, v[ch * 8 + 2] = o0.z, v[ch * 8 + 3] = o0.w;
              v[ch * 8 + 4] = o1.x, v[ch * 8 + 5] = o1.y, v[ch * 8 + 6] = o1.z, v[ch * 8 + 7] = o1.w;
            }
            tmem_st32(tq_lane + (uint32_t)(kTmemCols + s * 64 + tt * 32), v);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          tc_fence_before();  // the MMA issuer reads the slot after the barrier
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&full_bar[s]);
            mbar_arrive(&code_empty[cs]);
          }
        }
        if (!good) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&scale_empty[u & 1]);
      }
    } else {
    // ---------------- epilogue: warps 0-3 take the even units, warps 4-7 the odd ones (accumulator
    // buffer u & 1), each warp its TMEM lane quarter, so each has two units' time for its
    // reductions; with MXFP8 experts warps 0-3 take every unit ----------------
    const int quarter = warp & 3, group = warp >> 2;
    bool nonfinite = false;
    for (int u = 0;; ++u) {
      const int q = u % kTQ;
      int4 e = make_int4(kUnitEnd, 0, 0, 0);
      int ok = 0;
      const bool mine = MX || (u & 1) == group;
      if (lane == 0) {
        ok = mbar_wait_bounded(&tq_full[q], (uint32_t)((u / kTQ) & 1), &sm.abort, a.status, a.wait_ns) ? 1 : 0;
        if (ok) {
          e = tq[q];
          mbar_arrive(&tq_empty[q]);
          ok = (e.x & 15) == kUnitEnd || !mine ||
               mbar_wait_bounded(&tfull[u & 1], (uint32_t)((u >> 1) & 1), &sm.abort, a.status, a.wait_ns);
        }
        if (!ok) atomicExch(&cnt[kCntAbort], 1u);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      const int kind = __shfl_sync(0xffffffffu, e.x, 0) & 15;
      if (!ok || kind == kUnitEnd) break;
      if (!mine) continue;
      const int g = __shfl_sync(0xffffffffu, e.y, 0), blk = __shfl_sync(0xffffffffu, e.z, 0);
      tc_fence_after();
      float v0[16], v1[16];
      const uint32_t tb = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)((u & 1) * 32);
      tmem_ld16(tb, v0);
      tmem_ld16(tb + 16, v1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[u & 1]);  // the accumulator buffer is free for the next unit
      if (kind == kUnitA) {
        const int i = blk * 128 + quarter * 32 + lane;  // this lane's row of inter
        double *acc = t.acc_gu + (size_t)g * 2 * 4 * I + i;
#pragma unroll
        for (int r = 0; r < rows; ++r) {
          red_add_f64(acc + (size_t)r * I, (double)plane_sum<MX>(v0, r, t.mx_unscale));        // gate
          red_add_f64(acc + (size_t)(4 + r) * I, (double)plane_sum<MX>(v1, r, t.mx_unscale));  // up
        }
        // the count is an acquire-release add: it publishes the warp's adds (ordered before it by the
        // warp barrier) and, in the last split, makes every other split's adds visible
        __syncwarp();
        int last = 0;
        if (lane == 0)
          last = atom_add_acq_rel(&cnt[t.cnt_units + (g * rba + blk) * 4 + quarter], 1u) == (unsigned)(t.sa - 1);
        __syncwarp();  // lane 0's acquire is ordered before every lane's reads below
        if (__shfl_sync(0xffffffffu, last, 0)) {
          // every split of this (group, block, quarter) is in: SwiGLU, as bf16 hi / lo planes
          asm volatile("fence.acq_rel.gpu;" ::: "memory");
#pragma unroll
          for (int r = 0; r < rows; ++r) {
            const float gv = (float)ld_cg_f64(acc + (size_t)r * I), uv = (float)ld_cg_f64(acc + (size_t)(4 + r) * I);
            acc[(size_t)r * I] = 0.0;  // zero again for the next launch
            acc[(size_t)(4 + r) * I] = 0.0;
            const float v = gv * sigmoidf_(gv) * uv;
            nonfinite |= !isfinite(v);
            if (MX) {  // three f16 planes in rows r, 4 + r, 8 + r
              uint16_t p0, p1, p2;
              split3_f16(v, p0, p1, p2);
              t.act2[((size_t)g * 16 + r) * I + i] = p0;
              t.act2[((size_t)g * 16 + 4 + r) * I + i] = p1;
              t.act2[((size_t)g * 16 + 8 + r) * I + i] = p2;
            } else {
              const float hi = round_bf16(v), lo = round_bf16(v - hi);
              t.act2[((size_t)g * 16 + r) * I + i] = (uint16_t)(__float_as_uint(hi) >> 16);
              t.act2[((size_t)g * 16 + 4 + r) * I + i] = (uint16_t)(__float_as_uint(lo) >> 16);
            }
          }
          asm volatile("fence.proxy.async.global;" ::: "memory");  // read back by TMA
          __syncwarp();
          if (lane == 0) publish(&group_done[g], 32u);
        }
      } else {
        // kind B: rows d0 (first block of the pair) and d0 + 128 of hidden, scaled by the route weights
        const int d0 = blk * 256 + quarter * 32 + lane, d1 = d0 + 128;
        const int mask = sm.gm[g];
#pragma unroll
        for (int r = 0; r < rows; ++r) {
          if ((mask >> r) & 1) {
            const float w = sm.gw[g][r];
            const float y0 = w * plane_sum<MX>(v0, r, t.mx_unscale), y1 = w * plane_sum<MX>(v1, r, t.mx_unscale);
            nonfinite |= !isfinite(y0);
            red_add_f64(t.acc_y + (size_t)r * D + d0, (double)y0);
            if (d1 < D) {
              nonfinite |= !isfinite(y1);
              red_add_f64(t.acc_y + (size_t)r * D + d1, (double)y1);
            }
          }
        }
        __syncwarp();
        if (lane == 0) {  // release adds: the warp's reductions before the counts
          publish(&dblock_done[(blk * 256 + quarter * 32) / kDecodeDBlock], 1u);
          if (blk * 256 + 128 < D) publish(&dblock_done[(blk * 256 + 128 + quarter * 32) / kDecodeDBlock], 1u);
        }
      }
    }
    if (__any_sync(0xffffffffu, nonfinite) && lane == 0) atomicOr(a.status, kDevNonFinite);
    }
  } else if (warp == kProducerWarp) {
    // ================= producer: routing, unit claims, TMA =================
    route_setup<ROWS>(a, sm);
    route_compute<ROWS>(a, sm, true);
    ScorePoll sp{&score_bar, 0u, false, false, 0};
    // the stream starts once the mix CTAs have read the state (the prelude's loads are latency-bound
    // chains that must not queue behind it)
    (void)wait_at_least(&cnt[kCntMixDone], (unsigned)a.nm, a);
    sp.t0 = global_timer_ns();
    score_copy_issue(a, sm, sp, ROWS);
    const uint64_t pol = make_policy_evict_first();  // every weight byte is read once
    int j = 0;    // A ring steps issued
    int nab = 0;  // act slices issued
    int u = 0;    // units handed to the MMA issuer and the epilogue
    int ng = -1;
    bool ok = true;
    // a unit into the queue (lane 0 writes, the warp follows its verdict)
    auto hand = [&](int kind, int g, int blk, int e) -> bool {
      const int q = u % kTQ;
      int r = 0;
      if (lane == 0) {
        r = mbar_wait_backoff(&tq_empty[q], (uint32_t)((u / kTQ) & 1) ^ 1u, &sm.abort, a.status, a.wait_ns) ? 1 : 0;
        if (r) {
          tq[q] = make_int4(kind, g, blk, e);
          mbar_arrive(&tq_full[q]);
        } else {
          atomicExch(&cnt[kCntAbort], 1u);
        }
      }
      ++u;
      return __shfl_sync(0xffffffffu, r, 0) != 0;
    };
    // the next free ring slot (lane 0 waits, the warp follows)
    // (bf16 experts: the A ring; MXFP8 experts: the code ring)
    constexpr int NF = MX ? kCodeStages : NA;
    uint64_t *fill_full = MX ? code_full : full_bar, *fill_empty = MX ? code_empty : empty_bar;
    auto slot = [&]() -> int {
      const int s = j % NF;
      int r = 1;
      if (lane == 0) {
        r = mbar_wait_backoff(&fill_empty[s], (uint32_t)((j / NF) & 1) ^ 1u, &sm.abort, a.status, a.wait_ns) ? 1 : 0;
        if (!r) atomicExch(&cnt[kCntAbort], 1u);
      }
      return __shfl_sync(0xffffffffu, r, 0) ? s : -1;
    };
    // one k-step's two tiles into slot s: tile 0 from m0 at (kc, r0), tile 1 from m1 at (kc, r1)
    auto fill = [&](int s, const CUtensorMap *m0, const CUtensorMap *m1, int kc, int r0, int r1) {
      if (lane == 0) {
        const int tb = MX ? kCodeTile : kTile;
        uint8_t *dst = MX ? codes + (size_t)s * kCodeSlot : ring + (size_t)s * kSlotBytes;
        mbar_arrive_expect_tx(&fill_full[s], 2u * tb);
        tma_load_2d_hint(dst, m0, &fill_full[s], kc, r0, pol);
        tma_load_2d_hint(dst + tb, m1, &fill_full[s], kc, r1, pol);
      }
      __syncwarp();
    };
    // MXFP8: the scales of the unit just handed into its scale slot, once the converters are done
    // with the unit two before it
    auto unit_scales = [&](const uint8_t *s0, const uint8_t *s1, int rows0, int rows1, int stride,
                           int nbytes) -> bool {
      const int us = u - 1;
      int r = 1;
      if (lane == 0) {
        r = mbar_wait_backoff(&scale_empty[us & 1], (uint32_t)((us >> 1) & 1) ^ 1u, &sm.abort, a.status, a.wait_ns)
                ? 1
                : 0;
        if (!r) atomicExch(&cnt[kCntAbort], 1u);
      }
      if (!__shfl_sync(0xffffffffu, r, 0)) return false;
      scale_copy(scales + (size_t)(us & 1) * kScaleSlot, s0, s1, rows0, rows1, stride, nbytes, &scale_full[us & 1],
                 lane);
      return true;
    };
    // The units of this CTA's two K splits, from two queues in group order: kind A (group, 128-row
    // block of inter), then, once that queue is used up, kind B (group, pair of 128-row blocks of
    // hidden).  (Taking kind B units of groups whose act was complete between kind A units, and
    // holding the fills until the CTA's own prelude was done, both measured slower.)
    unsigned *tick_a = cnt + t.cnt_tick_a + 32 * ka, *tick_b = cnt + t.cnt_tick_b + 32 * kbs;
    bool a_done = false;
    while (ok) {
      if (!sp.routed) (void)score_poll<ROWS>(a, sm, cnt, sp, false);
      if (a_done) {
        // ---- a kind B unit: this CTA's split of inter, two 128-row blocks of hidden ----
        int tk = 0;
        if (lane == 0) tk = (int)atomicAdd(tick_b, 1u);
        tk = __shfl_sync(0xffffffffu, tk, 0);
        const int g = tk / rbb, blk = tk - g * rbb;
        if (g >= ng) break;
        const int e = sm.ge[g];
        // the group's act planes, once every 128-row block of inter has published them
        if (!wait_at_least(&group_done[g], (unsigned)I, a)) {
          ok = false;
          break;
        }
        const int ab = nab & 1;
        int r = 1;
        if (lane == 0) {
          r = mbar_wait_backoff(&aempty[ab], (uint32_t)((nab >> 1) & 1) ^ 1u, &sm.abort, a.status, a.wait_ns) ? 1 : 0;
          if (r) {
            // written by other CTAs' generic stores, read here by TMA
            asm volatile("fence.proxy.async.global;" ::: "memory");
            mbar_arrive_expect_tx(&afull[ab], (uint32_t)(t.cb * kBTile));
            for (int c = 0; c < t.cb; ++c)
              tma_load_2d(as + (size_t)ab * kBSlice + (size_t)c * kBTile, &tm.act2, &afull[ab],
                          (kbs * t.cb + c) * 64, g * 16);
          } else {
            atomicExch(&cnt[kCntAbort], 1u);
          }
        }
        if (!__shfl_sync(0xffffffffu, r, 0)) {
          ok = false;
          break;
        }
        ++nab;
        if (!hand(kUnitB | (ab << 4), g, blk, e)) {
          ok = false;
          break;
        }
        const CUtensorMap *md = MX ? (g == 0 ? &tm.down_sh_q : &tm.down_q) : (g == 0 ? &tm.down_sh : &tm.down);
        const int row = (g == 0 ? 0 : e * D) + blk * 256;
        if (MX) {
          const int st = I / 32;
          const uint8_t *s0 = (g == 0 ? a.down_sh_s : a.down_s) + (size_t)row * st + kbs * t.cb * 2;
          if (!unit_scales(s0, s0 + (size_t)128 * st, min(128, D - blk * 256), max(0, min(128, D - blk * 256 - 128)),
                           st, 2 * t.cb)) {
            ok = false;
            break;
          }
        }
        for (int c = 0; c < t.cb; ++c, ++j) {
          const int s = slot();
          if (s < 0) {
            ok = false;
            break;
          }
          fill(s, md, md, (kbs * t.cb + c) * 64, row, row + 128);
        }
        continue;
      }
      // ---- a kind A unit: this CTA's split of hidden, a 128-row block of inter ----
      int tk = 0;
      if (lane == 0) tk = (int)atomicAdd(tick_a, 1u);
      tk = __shfl_sync(0xffffffffu, tk, 0);
      const int g = tk / rba, blk = tk - g * rba;
      if (g > 0 && ng < 0) {  // the first routed unit: the group table
        (void)score_poll<ROWS>(a, sm, cnt, sp, true);
        ng = sm.ng;
      }
      if (g > 0 && g >= ng) {  // every kind A unit of this split is claimed
        a_done = true;
        continue;
      }
      const int e = g == 0 ? E : sm.ge[g];
      if (!hand(kUnitA, g, blk, e)) {
        ok = false;
        break;
      }
      const CUtensorMap *mg = MX ? (g == 0 ? &tm.gate_sh_q : &tm.gate_q) : (g == 0 ? &tm.gate_sh : &tm.gate);
      const CUtensorMap *mu = MX ? (g == 0 ? &tm.up_sh_q : &tm.up_q) : (g == 0 ? &tm.up_sh : &tm.up);
      const int row = (g == 0 ? 0 : e * I) + blk * 128;
      if (MX) {
        const int st = D / 32;
        const size_t off = (size_t)row * st + ka * t.ca * 2;
        if (!unit_scales((g == 0 ? a.gate_sh_s : a.gate_s) + off, (g == 0 ? a.up_sh_s : a.up_s) + off, 128, 128, st,
                         2 * t.ca)) {
          ok = false;
          break;
        }
      }
      for (int c = 0; c < t.ca; ++c, ++j) {
        const int s = slot();
        if (s < 0) {
          ok = false;
          break;
        }
        fill(s, mg, mu, (ka * t.ca + c) * 64, row, row);
      }
    }
    (void)hand(kUnitEnd, 0, 0, 0);
    // phase C needs the group table even where no routed unit was drawn
    (void)score_poll<ROWS>(a, sm, cnt, sp, true);
    // copies still in flight (after a timeout) land before the CTA may leave
    if (lane == 0) {
      int no_abort = 0;
      for (int s = 0; s < NF; ++s) {
        const int n = j / NF + (s < j % NF ? 1 : 0);
        if (n > 0) (void)mbar_wait_bounded(&fill_full[s], (uint32_t)((n - 1) & 1), &no_abort, a.status, a.wait_ns);
      }
      for (int b = 0; b < 2; ++b) {
        const int n = nab / 2 + (b < nab % 2 ? 1 : 0);
        if (n > 0) (void)mbar_wait_bounded(&afull[b], (uint32_t)((n - 1) & 1), &no_abort, a.status, a.wait_ns);
      }
      if (sp.in_flight) (void)mbar_wait_bounded(&score_bar, sp.phase, &no_abort, a.status, a.wait_ns);
    }
    if (MX) asm volatile("cp.async.wait_all;" ::: "memory");  // this lane's scale copies
    __syncwarp();
  } else if (warp == kMmaWarp && lane == 0) {
    // ================= MMA issuer =================
    int ok = mbar_wait_bounded(&xready, 0u, &sm.abort, a.status, a.wait_ns) ? 1 : 0;
    const uint32_t idesc = MX ? idesc_f16_f32(128, 16) : idesc_bf16_f32(128, 16);
    int j = 0, na = 0;
    for (int u = 0; ok; ++u) {
      const int q = u % kTQ;
      if (!mbar_wait_bounded(&tq_full[q], (uint32_t)((u / kTQ) & 1), &sm.abort, a.status, a.wait_ns)) break;
      const int4 e = tq[q];
      mbar_arrive(&tq_empty[q]);
      const int kind = e.x & 15;
      if (kind == kUnitEnd) break;
      const int b = u & 1;
      if (!mbar_wait_bounded(&tempty[b], (uint32_t)((u >> 1) & 1) ^ 1u, &sm.abort, a.status, a.wait_ns)) break;
      tc_fence_after();
      const uint32_t d0 = tmem + (uint32_t)(b * 32), d1 = d0 + 16;
      const int ab = (e.x >> 4) & 1;
      if (kind == kUnitB &&
          !mbar_wait_bounded(&afull[ab], (uint32_t)((na >> 1) & 1), &sm.abort, a.status, a.wait_ns))
        break;
      const int nc = kind == kUnitA ? t.ca : t.cb;
      const uint32_t bbase = smem_u32(kind == kUnitA ? xs : as + (size_t)ab * kBSlice);
      for (int c = 0; c < nc; ++c, ++j) {
        const int s = j % NA;
        if (!mbar_wait_bounded(&full_bar[s], (uint32_t)((j / NA) & 1), &sm.abort, a.status, a.wait_ns)) {
          ok = 0;
          break;
        }
        tc_fence_after();
        const uint32_t sb = bbase + (uint32_t)(c * kBTile);
        if (MX) {  // A from TMEM: slot s, 8 columns (16 k) an MMA
          const uint32_t ta = tmem + (uint32_t)(kTmemCols + s * 64);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t accum = (c > 0 || k > 0) ? 1u : 0u;
            const uint64_t bd = smem_desc_sw128(sb + k * 32);
            tc_mma_f16_tmem_a(d0, ta + k * 8, bd, idesc, accum);
            tc_mma_f16_tmem_a(d1, ta + 32 + k * 8, bd, idesc, accum);
          }
        } else {
          const uint32_t sa = smem_u32(ring + (size_t)s * kSlotBytes);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t accum = (c > 0 || k > 0) ? 1u : 0u;
            const uint64_t bd = smem_desc_sw128(sb + k * 32);
            tc_mma_f16(d0, smem_desc_sw128(sa + k * 32), bd, idesc, accum);
            tc_mma_f16(d1, smem_desc_sw128(sa + kTile + k * 32), bd, idesc, accum);
          }
        }
        tc_commit(&empty_bar[s]);  // the slot is free once these MMAs have read it
      }
      if (!ok) break;
      if (kind == kUnitB) {
        tc_commit(&aempty[ab]);
        ++na;
      }
      tc_commit(&tfull[b]);
    }
    // every MMA issued completes before TMEM is freed (immediate in a normal run)
    tc_commit(&mma_done);
    int no_abort = 0;
    (void)mbar_wait_bounded(&mma_done, 0u, &no_abort, a.status, a.wait_ns);
  }
  __syncthreads();  // the group table is complete for phase C; no unit is in flight
  pdl_wait();       // phase C reads the state, which comes from the previous kernel

  // ---- phase C: per 32-wide block of hidden, once every group's kind B units of it are in: ffn_out
  // (the f64 sum, rounded once) and the hc_post output out_i = post_i * ffn_out + sum_j comb[i, j] *
  // state_j.  The comb term needs no FFN output, so it is formed before the block's wait.
  const int hc = a.hc, ng = sm.ng, nblk = D / kDecodeDBlock;
  const bool comb_ok = wait_at_least(&cnt[kCntComb], a.inject == 1 ? 2u : 1u, a);
  for (int c = draw_ticket(&cnt[kCntTickC]); c < nblk && comb_ok; c = draw_ticket(&cnt[kCntTickC])) {
    const int d = c * kDecodeDBlock + lane;
    float po[rows][kHcMax], tt[rows][kHcMax];
#pragma unroll
    for (int r = 0; r < rows; ++r) {
      float sj[kHcMax];
#pragma unroll
      for (int q = 0; q < kHcMax; ++q) sj[q] = q < hc ? a.state[((size_t)r * hc + q) * D + d] : 0.f;
#pragma unroll
      for (int o = 0; o < kHcMax; ++o) {
        po[r][o] = o < hc ? __ldcg(a.post + r * hc + o) : 0.f;
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < kHcMax; ++q)
          if (o < hc && q < hc) v += __ldcg(a.comb + (r * hc + o) * hc + q) * sj[q];
        tt[r][o] = v;
      }
    }
    if (!wait_at_least(&dblock_done[c], (unsigned)(ng * t.sb), a, false)) break;
#pragma unroll
    for (int r = 0; r < rows; ++r) {
      double *src = t.acc_y + (size_t)r * D + d;
      const float f = (float)ld_cg_f64(src);
      *src = 0.0;  // zero again for the next launch
      a.ffn_out[(size_t)r * D + d] = f;
#pragma unroll
      for (int o = 0; o < kHcMax; ++o)
        if (o < hc) a.out_state[((size_t)r * hc + o) * D + d] = po[r][o] * f + tt[r][o];
    }
  }

  // ---- the last CTA out resets the counters and the score table for the next launch ----
  __threadfence();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
  if (tid == 0) sm.flag = atomicAdd(&cnt[kCntExit], 1u) == gridDim.x - 1 ? 1 : 0;
  __syncthreads();
  if (sm.flag) {
    __threadfence();
    // a launch that gave up somewhere may have left partial sums that their readers never took:
    // zero both accumulators (every CTA has left its loops and fenced its adds)
    if (*reinterpret_cast<volatile unsigned *>(&cnt[kCntAbort]) != 0u) {
      for (int i = tid; i < t.n_acc_gu; i += blockDim.x) t.acc_gu[i] = 0.0;
      for (int i = tid; i < t.n_acc_y; i += blockDim.x) t.acc_y[i] = 0.0;
    }
    __syncthreads();
    for (int i = tid; i < a.n_counters; i += blockDim.x) cnt[i] = 0u;
    for (int i = tid; i < kDecodeRows * E; i += blockDim.x) a.sel[i] = __uint_as_float(kUnwritten);
    __threadfence();
  }
}

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------

using DecodeTcKernel = void (*)(DecodeTcMaps, DecodeArgs, DecodeTcArgs);
static DecodeTcKernel decode_tc_kernel_for(int rows, bool mx) {
  if (mx)
    return rows == 1 ? decode_tc_kernel<1, true>
           : rows == 2 ? decode_tc_kernel<2, true>
           : rows == 3 ? decode_tc_kernel<3, true>
                       : decode_tc_kernel<4, true>;
  return rows == 1 ? decode_tc_kernel<1, false>
         : rows == 2 ? decode_tc_kernel<2, false>
         : rows == 3 ? decode_tc_kernel<3, false>
                     : decode_tc_kernel<4, false>;
}
static size_t decode_tc_smem(bool mx) { return mx ? dtc::kSmemMx : dtc::kSmem; }

cudaError_t decode_tc_configure() {
  for (int mx = 0; mx < 2; ++mx)
    for (int r = 1; r <= kDecodeRows; ++r) {
      const cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel_for(r, mx != 0),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)decode_tc_smem(mx != 0));
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

int decode_tc_resident_ctas(int rows, int num_sms, bool mx) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_tc_kernel_for(rows, mx), kDecThreads,
                                                    decode_tc_smem(mx)) != cudaSuccess)
    return 0;
  return per_sm * num_sms;
}

// The fewest K splits of `chunks` 64-wide chunks that leave at most kMaxChunks chunks to a split.
static void tc_split(int chunks, int &splits, int &per) {
  for (splits = 1; splits < chunks; ++splits)
    if (chunks % splits == 0 && chunks / splits <= dtc::kMaxChunks) break;
  per = chunks / splits;
}

bool decode_tc_fits(const Dims &d, int grid) {
  int sa, ca, sb, cb;
  tc_split(d.hidden / 64, sa, ca);
  tc_split(d.inter / 64, sb, cb);
  return ca <= dtc::kMaxChunks && cb <= dtc::kMaxChunks && sa <= kMaxSplits && sb <= kMaxSplits && grid >= sa &&
         grid >= sb;
}

void launch_decode_tc(const DecodeArgs &a, const Dims &d, const Scratch &s, const LayerDev &w, int rows, int grid,
                      cudaStream_t st) {
  DecodeTcMaps m;
  m.gate = w.tm_gate;
  m.up = w.tm_up;
  m.down = w.tm_down;
  m.gate_sh = w.tm_gate_sh;
  m.up_sh = w.tm_up_sh;
  m.down_sh = w.tm_down_sh;
  m.act2 = s.tm_dtc_act2;
  m.gate_q = w.tm_gate_q;
  m.up_q = w.tm_up_q;
  m.down_q = w.tm_down_q;
  m.gate_sh_q = w.tm_gate_sh_q;
  m.up_sh_q = w.tm_up_sh_q;
  m.down_sh_q = w.tm_down_sh_q;
  DecodeTcArgs t;
  t.acc_gu = s.dtc_acc_gu;
  t.acc_y = s.dtc_acc_y;
  t.act2 = s.dtc_act2;
  tc_split(d.hidden / 64, t.sa, t.ca);
  tc_split(d.inter / 64, t.sb, t.cb);
  t.cnt_tick_a = tc_counter_base(d);
  t.cnt_tick_b = t.cnt_tick_a + kMaxSplits * 32;
  t.cnt_units = t.cnt_tick_b + kMaxSplits * 32;
  t.n_acc_gu = (d.top_k * kDecodeRows + 1) * 2 * 4 * d.inter;
  t.n_acc_y = 4 * d.hidden;
  t.mx_c = w.mx_c;
  t.mx_unscale = ldexpf(1.f, -w.mx_c);
  launch_pdl(decode_tc_kernel_for(rows, w.mx), dim3(grid), dim3(kDecThreads), decode_tc_smem(w.mx), st, m, a, t);
}

}  // namespace moe
