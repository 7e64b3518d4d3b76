// Decode path (rows <= 4) on the CUDA cores: the whole FFN block in one persistent launch, two CTAs
// per SM.  It serves layers whose experts are MXFP8 (the codes are decoded in the dot products),
// and bf16 layers where the tensor-core kernel (decode_tc.cu) does not fit the configuration.
//
// docs.rs "hf2q 0.1.3 .../deepseek4/ffn_forward.rs", forward_ffn_rows, every stage in order:
// rms_norm_no_scale_f32 + raw_matmul "HC FFN function" + dispatch_hc_split_sinkhorn (mix CTAs),
// dispatch_hc_pre + rms_norm (every CTA), raw_matmul "MoE gate" (router CTAs) +
// dispatch_deepseek_moe_{score,hash}_route + dispatch_deepseek_moe_sanitize_indices (every CTA's
// producer), expert_matmul "routed gate"/"routed up" + raw_matmul "shared gate"/"shared up" +
// dispatch_deepseek_moe_swiglu (stream, kind A), expert_matmul "routed down" + raw_matmul "shared
// down" (stream, kind B), dispatch_deepseek_moe_weighted_reduce + dispatch_hc_post (phase C).
//
// At 1-4 tokens every expert weight byte feeds 1-4 multiply-adds: the block is bound by HBM
// bandwidth once the weights stream, and by latency before that.  Each CTA has 8 worker warps, one
// producer warp and one publisher warp:
//
//   workers   (a) prelude: the first CTAs to arrive (a CTA ticket) are `nm` mix CTAs (a column chunk
//             of the flattened state each: the partial mixes and sum of squares; the last one forms
//             mixes, pre and post) and `nr` router CTAs.  Every CTA then forms x = ffn_norm(hc_pre)
//             itself, on the 16 hidden columns each worker thread owns, from the mix partials and
//             the state (in L2 by then), with the RMS over the CTA: x lands in the registers the
//             stream needs and no CTA waits for another to publish it.  Router CTA j adds the
//             logits of experts [j epc, (j + 1) epc) over the CTA and writes each sigmoid(logit)
//             with one 4-byte store into a table that starts all-ones.
//             (b) the stream: every slot is consumed by all 8 warps at once (split K, x or the
//             group's SwiGLU output in registers), each leaving its partial sums in shared memory:
//               kind A: a gate row and an up row of one expert group;
//               kind B: four down rows of one group, once its act is complete.
//             (c) phase C: per 32-wide d-block, once every group's rows of it are in: ffn_out =
//             sum_g w * y and the hc_post output of that block.
//   producer  draws work tickets from a device-wide counter (in chunks of four consecutive numbers,
//             two claims ahead) and moves each ticket's weight rows into a ring of shared-memory
//             slots with bulk asynchronous copies (TMA, completion on the slot's mbarrier), so the
//             bytes in flight cost no registers.  The shared expert needs no routing: its rows
//             stream as soon as the mix CTAs have read the state.  Between fills it keeps one bulk
//             copy of the sigmoid table in flight into shared memory; once a copy holds no
//             all-ones entry it routes the batch itself: the top_k by warp-shuffle argmax rounds,
//             the same code on the same values in every CTA.
//   publisher takes the slots in order: adds the 8 warps' partial sums, applies SwiGLU (kind A),
//             stores act or y, frees the slot for the producer, and publishes completion counts
//             in batches (one fence, then relaxed adds): a release fence waits microseconds under
//             load, and no worker warp, which every slot needs, may stall on one.  It publishes
//             whenever it has waited 2 us, so a batch never holds back work some CTA waits for.
//             The last mix CTA's publisher also forms the comb (Sinkhorn) for phase C.
//
// Code that runs once per launch runs out of an instruction cache that the weight stream (and a
// benchmark's L2 flush) leaves cold; the producer therefore runs its routing code once on scratch
// data at launch, so that the code is in L2 when the scores arrive.
//
// Tickets are drawn in order (all kind-A tickets before any kind-B ticket), a CTA consumes its
// slots in ticket order, and a kind-B slot waits only for kind-A work, which running CTAs hold
// ahead of it: every wait ends whatever the number of co-resident CTAs.  Waits still give up after
// 1 s (device timeout bit), and a CTA that gives up first waits (bounded) for its own copies in
// flight.  The last CTA to leave resets the counters and the score entries, so the next launch
// (or a graph replay) starts clean without a separate clearing step.
#include <math.h>
#include <stddef.h>

#include "common.cuh"
#include "decode_prelude.cuh"
#include "kernels.h"

namespace moe {

// ---------------------------------------------------------------------------------------------
// The stream
// ---------------------------------------------------------------------------------------------

// The 8 E4M3 codes of a uint2 as floats: the hardware converts pairs to f16 (exact), then to f32
// (the same conversion as e4m3x16_to_float; it measured faster than decoding the fields with
// integer operations).
__device__ __forceinline__ void e4m3x8_to_float_cvt(const uint2 w, float (&f)[8]) {
  const unsigned words[2] = {w.x, w.y};
#pragma unroll
  for (int q = 0; q < 2; ++q) {
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

// Packed f32 pairs (sm_100 and later: one fma.rn.f32x2 does two FMAs).
__device__ __forceinline__ void fma_f32x2(unsigned long long &acc, unsigned long long a, unsigned long long b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
__device__ __forceinline__ float sum_f32x2(unsigned long long v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo + hi;
}
// sum_k f[k] x[k] over 16 elements as two interleaved partial sums (even and odd k)
__device__ __forceinline__ float dot16x2(const float (&f)[16], const float4 x0, const float4 x1, const float4 x2,
                                         const float4 x3) {
  unsigned long long acc = 0ull;
  fma_f32x2(acc, pack_f32x2(f[0], f[1]), pack_f32x2(x0.x, x0.y));
  fma_f32x2(acc, pack_f32x2(f[2], f[3]), pack_f32x2(x0.z, x0.w));
  fma_f32x2(acc, pack_f32x2(f[4], f[5]), pack_f32x2(x1.x, x1.y));
  fma_f32x2(acc, pack_f32x2(f[6], f[7]), pack_f32x2(x1.z, x1.w));
  fma_f32x2(acc, pack_f32x2(f[8], f[9]), pack_f32x2(x2.x, x2.y));
  fma_f32x2(acc, pack_f32x2(f[10], f[11]), pack_f32x2(x2.z, x2.w));
  fma_f32x2(acc, pack_f32x2(f[12], f[13]), pack_f32x2(x3.x, x3.y));
  fma_f32x2(acc, pack_f32x2(f[14], f[15]), pack_f32x2(x3.z, x3.w));
  return sum_f32x2(acc);
}
__device__ __forceinline__ float dot8fx2(const float (&f)[8], const float4 x0, const float4 x1) {
  unsigned long long acc = 0ull;
  fma_f32x2(acc, pack_f32x2(f[0], f[1]), pack_f32x2(x0.x, x0.y));
  fma_f32x2(acc, pack_f32x2(f[2], f[3]), pack_f32x2(x0.z, x0.w));
  fma_f32x2(acc, pack_f32x2(f[4], f[5]), pack_f32x2(x1.x, x1.y));
  fma_f32x2(acc, pack_f32x2(f[6], f[7]), pack_f32x2(x1.z, x1.w));
  return sum_f32x2(acc);
}

__device__ __forceinline__ uint2 lds64(const void *p) {
  uint2 r;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(smem_u32(p)));
  return r;
}

// 1-D bulk copy global -> shared memory with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

template <int ROWS, bool MX>
__global__ void __launch_bounds__(kDecThreads, 2) decode_kernel(DecodeArgs a) {
  using RG = Ring<MX>;
  constexpr int S = RG::kSlots;
  constexpr int rows = ROWS;  // every row loop is unrolled exactly, without run-time guards
  extern __shared__ __align__(128) uint8_t dsm[];
  uint8_t *ring = dsm;
  float *red = reinterpret_cast<float *>(dsm + (size_t)S * RG::kSlotBytes);  // [S][8 warps][kRed]
  __shared__ __align__(16) DecSmem sm;
  __shared__ __align__(8) uint64_t full_bar[S], empty_bar[S], red_bar[S], score_bar;
  unsigned *cnt = a.counters;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int D = a.hidden, I = a.inter, E = a.experts;
  const int all_rows = (1 << rows) - 1;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);             // the publisher has taken the slot's partial sums
      mbar_init(&red_bar[s], kWorkerWarps);    // every worker warp has left its partial sums
    }
    mbar_init(&score_bar, 1);                  // a copy of the score table has landed
    sm.abort = 0;
    sm.comb_todo = 0;
    sm.flag = (int)atomicAdd(&cnt[kCntRole], 1u);
    fence_mbar_init();
  }
  __syncthreads();
  const int role = sm.flag;
  __syncthreads();

  unsigned *group_done = cnt + kCntGroups;
  unsigned *dblock_done = cnt + kCntDBlocks;
  // a kind-A slot: the gate and up rows i, i + 1 of group g; a kind-B slot: down rows d0 .. d0 + 7
  const int perg = I / RG::kRowsA, nb_per_g = D / RG::kRowsB;

  if (warp == kProducerWarp) {
    // ================= producer =================
    // every weight row is read once (evict first), so that none crowds the kernel's own code or the
    // prelude's data out of L2 (the shared expert's rows prefetched to L2 are the newest lines, read
    // again within microseconds)
    const uint64_t pol_first = make_policy_evict_first(), pol_last = pol_first;
    const int span = MX ? (((RG::kRowsA * D / 32 + 32) + 15) & ~15) : 0;  // bytes per MX scale run of a kind-A slot
    route_setup<ROWS>(a, sm);
    route_compute<ROWS>(a, sm, true);
    ScorePoll sp{&score_bar, 0u, false, false, 0};
    // the prelude's loads are latency-bound chains: the stream starts once the mix CTAs have read
    // the state (later prelude reads hit L2), so that they do not queue behind it.  Then the shared
    // expert's gate/up rows that the first ring fills do not cover go to L2 (they are read again by
    // whichever CTA draws their tickets).
    (void)wait_at_least(&cnt[kCntMixDone], (unsigned)a.nm, a);
    // the mix role's reads of the shared-memory rows the score table overlays are done (mix CTAs
    // arrive on that count after them)
    sp.t0 = global_timer_ns();
    score_copy_issue(a, sm, sp, ROWS);
    {
      const int first = gridDim.x * S * RG::kRowsA;  // rows of the first fills
      const int rest = I - first;
      if (rest > 0) {
        const int per = (rest + gridDim.x - 1) / gridDim.x;
        for (int i = first + blockIdx.x * per + lane; i < min(I, first + (blockIdx.x + 1) * per); i += 32) {
          if (MX) {
            prefetch_l2(a.gate_sh_q + (size_t)i * D, (uint32_t)D, pol_last);
            prefetch_l2(a.up_sh_q + (size_t)i * D, (uint32_t)D, pol_last);
          } else {
            prefetch_l2(a.gate_sh + (size_t)i * D, (uint32_t)(2 * D), pol_last);
            prefetch_l2(a.up_sh + (size_t)i * D, (uint32_t)(2 * D), pol_last);
          }
        }
      }
    }
    int ng = -1;
    // tickets come in chunks of kChunk consecutive numbers; two chunk claims are in flight ahead of
    // the slots, so the atomic's round trip (microseconds under load) never stalls the ring
    int c0 = 0, c1 = 0, c2 = 0;  // the current chunk and the two claimed after it (lane 0)
    if (lane == 0) {
      c0 = (int)atomicAdd(&cnt[kCntTick], (unsigned)kChunk);
      c1 = (int)atomicAdd(&cnt[kCntTick], (unsigned)kChunk);
      c2 = (int)atomicAdd(&cnt[kCntTick], (unsigned)kChunk);
    }
    int phases[S];  // completions asked of each slot's full barrier (fills and end marks)
#pragma unroll
    for (int s = 0; s < S; ++s) phases[s] = 0;
    for (int k = 0;; ++k) {
      const int s = k % S;
      const int t = __shfl_sync(0xffffffffu, c0, 0) + k % kChunk;
      if (!sp.routed) (void)score_poll<ROWS>(a, sm, cnt, sp, false);
      SlotMeta m;
      m.s0 = m.s1 = 0;
      if (t < perg) {
        m.kind = kKindA;
        m.g = 0;
        m.row = t * RG::kRowsA;
        m.e = E;
        m.mask = all_rows;
      } else {
        if (ng < 0) {
          (void)score_poll<ROWS>(a, sm, cnt, sp, true);
          ng = sm.ng;
        }
        const int nA = ng * perg, nB = ng * nb_per_g;
        if (t < nA) {
          m.kind = kKindA;
          m.g = t / perg;
          m.row = (t - m.g * perg) * RG::kRowsA;
        } else if (t < nA + nB) {
          m.kind = kKindB;
          m.g = (t - nA) / nb_per_g;
          m.row = (t - nA - m.g * nb_per_g) * RG::kRowsB;
        } else {
          m.kind = kKindEnd;
          m.g = 0;
          m.row = 0;
        }
        m.e = sm.ge[m.g];
        m.mask = sm.gm[m.g];
      }
      // the slot is free once every worker warp has read its previous contents
      int got = 1;
      if (lane == 0) {
        got = mbar_wait_backoff(&empty_bar[s], ((uint32_t)(k / S) & 1u) ^ 1u, &sm.abort, a.status, a.wait_ns) ? 1 : 0;
        if (!got) atomicExch(&cnt[kCntAbort], 1u);
      }
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) m.kind = kKindEnd;  // give up: the workers stop at this slot
      if (lane == 0) {
        uint8_t *dst = ring + (size_t)s * RG::kSlotBytes;
        const bool routed = m.e < E;
        const uint64_t pol = routed ? pol_first : pol_last;
        // the slot's metadata is written before the barrier arrive that releases it to the workers
        if (m.kind == kKindA) {
          const size_t ro = routed ? (size_t)m.e * I + m.row : (size_t)m.row;
          if (MX) {
            const uint8_t *gs = (routed ? a.gate_s : a.gate_sh_s), *us = (routed ? a.up_s : a.up_sh_s);
            const size_t so = ro * (D / 32), a0 = so & ~(size_t)15;
            const size_t a1 = (so + RG::kRowsA * D / 32 + 15) & ~(size_t)15;
            m.s0 = m.s1 = (int)(so - a0);
            const uint32_t sb = (uint32_t)(a1 - a0);
            sm.meta[s] = m;
            mbar_arrive_expect_tx(&full_bar[s], (uint32_t)(2 * RG::kRowsA * D) + 2 * sb);
            bulk_g2s(dst, (routed ? a.gate_q : a.gate_sh_q) + ro * D, (uint32_t)(RG::kRowsA * D), &full_bar[s], pol);
            bulk_g2s(dst + RG::kRowsA * D, (routed ? a.up_q : a.up_sh_q) + ro * D, (uint32_t)(RG::kRowsA * D), &full_bar[s], pol);
            bulk_g2s(dst + 2 * RG::kRowsA * D, gs + a0, sb, &full_bar[s], pol);
            bulk_g2s(dst + 2 * RG::kRowsA * D + span, us + a0, sb, &full_bar[s], pol);
          } else {
            sm.meta[s] = m;
            mbar_arrive_expect_tx(&full_bar[s], (uint32_t)(4 * RG::kRowsA * D));
            bulk_g2s(dst, (routed ? a.gate_exps : a.gate_sh) + ro * D, (uint32_t)(2 * RG::kRowsA * D), &full_bar[s], pol);
            bulk_g2s(dst + 2 * RG::kRowsA * D, (routed ? a.up_exps : a.up_sh) + ro * D, (uint32_t)(2 * RG::kRowsA * D), &full_bar[s],
                     pol);
          }
        } else if (m.kind == kKindB) {
          const size_t ro = routed ? (size_t)m.e * D + m.row : (size_t)m.row;
          sm.meta[s] = m;
          if (MX) {
            mbar_arrive_expect_tx(&full_bar[s], (uint32_t)(RG::kRowsB * I + RG::kRowsB * (I / 32)));
            bulk_g2s(dst, (routed ? a.down_q : a.down_sh_q) + ro * I, (uint32_t)(RG::kRowsB * I), &full_bar[s], pol);
            bulk_g2s(dst + RG::kRowsB * I, (routed ? a.down_s : a.down_sh_s) + ro * (I / 32), (uint32_t)(RG::kRowsB * (I / 32)),
                     &full_bar[s], pol);
          } else {
            mbar_arrive_expect_tx(&full_bar[s], (uint32_t)(RG::kRowsB * I * 2));
            bulk_g2s(dst, (routed ? a.down_exps : a.down_sh) + ro * I, (uint32_t)(RG::kRowsB * I * 2), &full_bar[s], pol);
          }
        } else {
          sm.meta[s] = m;
          mbar_arrive(&full_bar[s]);  // metadata only: the workers stop here
        }
        ++phases[s];
      }
      __syncwarp();
      if (m.kind == kKindEnd) break;
      if (k % kChunk == kChunk - 1 && lane == 0) {  // the chunk is used up: claim one more ahead
        c0 = c1;
        c1 = c2;
        c2 = (int)atomicAdd(&cnt[kCntTick], (unsigned)kChunk);
      }
    }
    // copies still in flight (after a timeout) complete before the CTA may leave: wait (bounded)
    // for the last completion asked of every slot (in a normal run every one has completed)
    if (lane == 0) {
      int no_abort = 0;
#pragma unroll
      for (int s = 0; s < S; ++s)
        if (phases[s] > 0)
          (void)mbar_wait_bounded(&full_bar[s], (uint32_t)((phases[s] - 1) & 1), &no_abort, a.status, a.wait_ns);
    }
    __syncwarp();
    // phase C needs the group table even where no routed ticket was drawn
    (void)score_poll<ROWS>(a, sm, cnt, sp, true);
    if (sp.in_flight && lane == 0) {  // after a timeout: the copy lands before the CTA may leave
      int no_abort = 0;
      (void)mbar_wait_bounded(&score_bar, sp.phase, &no_abort, a.status, a.wait_ns);
    }
    __syncwarp();
  } else if (warp == kPublisherWarp) {
    // ================= publisher =================
    if (role < a.nm) {  // a mix CTA: the last one's publisher forms the comb
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
    // unpublished counts: up to 8 counters (a group's rows, kind A; a d-block's rows, kind B)
    int keys[8], cnts[8], nkeys = 0, held = 0;
    auto flush = [&]() {
      if (held > 0) {
        __threadfence();  // every lane's act / y stores reach the device before the counts do
        __syncwarp();
        if (lane == 0)
          for (int i = 0; i < nkeys; ++i)
            add_relaxed(keys[i] < 1024 ? &group_done[keys[i]] : &dblock_done[keys[i] - 1024], (unsigned)cnts[i]);
      }
      nkeys = held = 0;
    };
    // a bounded wait that publishes what is held once it has waited 2 us: the counts are held back
    // only while slots keep coming
    auto idle_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      int ready = 0;
      if (lane == 0) ready = mbar_try_wait(bar, parity) ? 1 : 0;
      if (__shfl_sync(0xffffffffu, ready, 0)) return true;
      const uint64_t t0 = global_timer_ns();
      bool flushed = false;
      while (true) {
        __nanosleep(kBackoffNs);
        if (lane == 0) ready = mbar_try_wait(bar, parity) ? 1 : 0;
        if (__shfl_sync(0xffffffffu, ready, 0)) return true;
        const uint64_t el = global_timer_ns() - t0;
        if (!flushed && el > 2000u) {
          flush();
          flushed = true;
        }
        int give_up = 0;
        if (lane == 0 && (*reinterpret_cast<volatile int *>(&sm.abort) != 0 || el > a.wait_ns)) {
          give_up = 1;
          sm.abort = 1;
          atomicOr(a.status, kDevTimeout);
          atomicExch(&cnt[kCntAbort], 1u);
        }
        if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
      }
    };
    for (int k = 0;; ++k) {
      const int s = k % S;
      const uint32_t par = (uint32_t)(k / S) & 1u;
      if (!idle_wait(&full_bar[s], par)) break;
      const SlotMeta m = sm.meta[s];
      if (m.kind == kKindEnd) break;
      if (!idle_wait(&red_bar[s], par)) break;
      const float *rb = red + (size_t)s * kWorkerWarps * RG::kRed;
      const int nv = m.kind == kKindA ? 2 * RG::kRowsA * ROWS : RG::kRowsB * ROWS;
      float tot = 0.f;
      if (lane < nv) {
#pragma unroll
        for (int w = 0; w < kWorkerWarps; ++w) tot += rb[w * RG::kRed + lane];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);  // the slot is free for the producer
      int key, n;
      if (m.kind == kKindA) {
        // item (ii * ROWS + r) is gate row m.row + ii of batch row r; RG::kRowsA * ROWS later, its up row
        const float u = __shfl_sync(0xffffffffu, tot, (lane + RG::kRowsA * ROWS) & 31);
        const int ii = lane / ROWS, r = lane - ii * ROWS;
        if (lane < RG::kRowsA * ROWS && ((m.mask >> r) & 1))
          a.act[((size_t)m.g * kDecodeRows + r) * I + m.row + ii] = tot * sigmoidf_(tot) * u;
        key = m.g;
        n = RG::kRowsA;
      } else {
        if (lane < RG::kRowsB * ROWS) {  // zeros for rows this group does not serve
          const int q = lane / ROWS, r = lane - q * ROWS;
          a.y[((size_t)m.g * kDecodeRows + r) * D + m.row + q] = ((m.mask >> r) & 1) ? tot : 0.f;
        }
        key = 1024 + m.row / kDecodeDBlock;
        n = RG::kRowsB;
      }
      int i = 0;
      while (i < nkeys && keys[i] != key) ++i;
      if (i == nkeys) {
        if (nkeys == 8) {
          flush();
          i = 0;
        }
        keys[nkeys] = key;
        cnts[nkeys] = 0;
        ++nkeys;
      }
      cnts[i] += n;
      if (++held >= kPublishBatch) flush();
    }
    flush();
  } else {
    // ================= workers =================
    const bool router = role >= a.nm && role < a.nm + a.nr;
    if (router) router_prefetch(a, role - a.nm);
    if (role < a.nm) mix_role<ROWS>(a, role, sm, cnt);
    // x in registers on the own columns (every CTA forms it), then the router CTAs' logits
    float4 xr[rows][4];
    form_x<ROWS, MX>(a, sm, cnt, xr);
    if (router) router_logits<ROWS, MX>(a, sm, cnt, role - a.nm, xr);
    pdl_wait();  // the state (read by phase C) comes from the previous kernel
    constexpr int VA = pow2_at_least(2 * RG::kRowsA * ROWS), VB = pow2_at_least(RG::kRowsB * ROWS);
    static_assert(VB <= RG::kRed && VA <= RG::kRed, "partial sums per warp and slot");
    const int span = MX ? (((RG::kRowsA * D / 32 + 32) + 15) & ~15) : 0;
    // A CTA draws all of its kind-A tickets before its first kind-B one, so the slots come as a run
    // of kind A, then a run of kind B: two loops, so that x and the SwiGLU slice are never held in
    // registers at the same time
    int k = 0;
    bool stop = false;
    for (;; ++k) {
      const int s = k % S;
      const uint32_t par = (uint32_t)(k / S) & 1u;
      if (!warp_mbar_wait(&full_bar[s], par, sm, a)) {
        stop = true;
        break;
      }
      const SlotMeta m = sm.meta[s];
      if (m.kind != kKindA) {
        stop = m.kind != kKindB;
        break;
      }
      const uint8_t *src = ring + (size_t)s * RG::kSlotBytes;
      float *rp = red + ((size_t)s * kWorkerWarps + warp) * RG::kRed;
      float pv[VA];
#pragma unroll
      for (int i = 0; i < VA; ++i) pv[i] = 0.f;
      // item (ii * ROWS + r): gate row m.row + ii, batch row r; RG::kRowsA * ROWS later, its up row
#pragma unroll
      for (int ii = 0; ii < RG::kRowsA; ++ii) {
        if constexpr (MX) {
          if (16 * tid < D) {
            const uint4 gq = lds128(src + ii * D + 16 * tid), uq = lds128(src + (RG::kRowsA + ii) * D + 16 * tid);
            const float sg = e8m0_value(src[2 * RG::kRowsA * D + m.s0 + ii * (D / 32) + tid / 2]);
            const float su = e8m0_value(src[2 * RG::kRowsA * D + span + m.s1 + ii * (D / 32) + tid / 2]);
            float fg[16], fu[16];
            e4m3x16_to_float(gq, fg);
            e4m3x16_to_float(uq, fu);
#pragma unroll
            for (int r = 0; r < rows; ++r) {
              if ((m.mask >> r) & 1) {
                pv[ii * ROWS + r] = sg * (dot16x2(fg, xr[r][0], xr[r][1], xr[r][2], xr[r][3]));
                pv[(RG::kRowsA + ii) * ROWS + r] = su * (dot16x2(fu, xr[r][0], xr[r][1], xr[r][2], xr[r][3]));
              }
            }
          }
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int c = 8 * tid + 2048 * h;
            if (c < D) {
              const uint4 gv = lds128(src + 2 * (ii * D + c)), uv = lds128(src + 2 * ((RG::kRowsA + ii) * D + c));
#pragma unroll
              for (int r = 0; r < rows; ++r) {
                if ((m.mask >> r) & 1) {
                  pv[ii * ROWS + r] += dot8(gv, xr[r][2 * h], xr[r][2 * h + 1]);
                  pv[(RG::kRowsA + ii) * ROWS + r] += dot8(uv, xr[r][2 * h], xr[r][2 * h + 1]);
                }
              }
            }
          }
        }
      }
      const float wt = warp_reduce_scatter<VA>(pv);
      if (lane < VA) rp[lane] = wt;
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_bar[s]);  // after this warp's reads of the slot and its partial sums
    }
    // the group's SwiGLU output (kind B): thread t owns columns 8t .. 8t + 7
    float4 ar[rows][2];
    int cur_g = -1;
    bool act_ok = false;
    for (; !stop; ++k) {  // from the first kind-B slot on (waiting again on its completed phase returns at once)
      const int s = k % S;
      const uint32_t par = (uint32_t)(k / S) & 1u;
      if (!warp_mbar_wait(&full_bar[s], par, sm, a)) break;
      const SlotMeta m = sm.meta[s];
      if (m.kind != kKindB) break;
      const uint8_t *src = ring + (size_t)s * RG::kSlotBytes;
      float *rp = red + ((size_t)s * kWorkerWarps + warp) * RG::kRed;
      if (m.g != cur_g) {  // the group's SwiGLU output, once its every gate/up row is published
        cur_g = m.g;
        act_ok = wait_at_least(&group_done[m.g], (unsigned)I, a);
#pragma unroll
        for (int r = 0; r < rows; ++r) {
          const bool in = act_ok && 8 * tid < I && ((m.mask >> r) & 1);
          const float4 *ap = reinterpret_cast<const float4 *>(a.act + ((size_t)m.g * kDecodeRows + r) * I + 8 * tid);
          ar[r][0] = in ? __ldcg(ap) : make_float4(0.f, 0.f, 0.f, 0.f);
          ar[r][1] = in ? __ldcg(ap + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float pv[VB];
#pragma unroll
      for (int i = 0; i < VB; ++i) pv[i] = 0.f;
      if (8 * tid < I) {
#pragma unroll
        for (int q = 0; q < RG::kRowsB; ++q) {
          float f[8];
          float sc = 1.f;
          uint4 wv = make_uint4(0u, 0u, 0u, 0u);
          if constexpr (MX) {
            e4m3x8_to_float_cvt(lds64(src + (size_t)q * I + 8 * tid), f);
            sc = e8m0_value(src[RG::kRowsB * I + q * (I / 32) + tid / 4]);
          } else {
            wv = lds128(src + (size_t)q * I * 2 + 16 * tid);
          }
#pragma unroll
          for (int r = 0; r < rows; ++r) {
            if ((m.mask >> r) & 1) {
              if constexpr (MX) pv[q * ROWS + r] = sc * (dot8fx2(f, ar[r][0], ar[r][1]));
              else pv[q * ROWS + r] = dot8(wv, ar[r][0], ar[r][1]);
            }
          }
        }
      }
      const float wt = warp_reduce_scatter<VB>(pv);
      if (lane < VB) rp[lane] = wt;
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_bar[s]);
    }
  }
  __syncthreads();  // the producer's group table is complete for phase C

  // ---- phase C: per 32-wide d-block, once every group's rows of it are in: ffn_out = sum_g w * y
  // and the hc_post output out_i = post_i * ffn_out + sum_j comb[i, j] * state_j.  The comb term
  // needs no y, so it is formed before the block's wait.
  const int hc = a.hc, ng = sm.ng, nblk = D / kDecodeDBlock;
  // (test hook 1: a count that is never reached, so that this wait runs out)
  const bool comb_ok = wait_at_least(&cnt[kCntComb], a.inject == 1 ? 2u : 1u, a);
  bool nonfinite = false;  // an FFN output element (a sum of expert outputs) that is NaN or infinite
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
    if (!wait_at_least(&dblock_done[c], (unsigned)(ng * kDecodeDBlock), a, false)) break;
#pragma unroll
    for (int r = 0; r < rows; ++r) {
      float f = 0.f;
#pragma unroll 4
      for (int g = 0; g < ng; ++g) f += sm.gw[g][r] * __ldcg(a.y + ((size_t)g * kDecodeRows + r) * D + d);
      nonfinite |= !isfinite(f);
      a.ffn_out[(size_t)r * D + d] = f;
#pragma unroll
      for (int o = 0; o < kHcMax; ++o)
        if (o < hc) a.out_state[((size_t)r * hc + o) * D + d] = po[r][o] * f + t[r][o];
    }
  }

  if (__any_sync(0xffffffffu, nonfinite) && lane == 0) atomicOr(a.status, kDevNonFinite);

  // ---- the last CTA out resets the counters for the next launch ----
  __threadfence();
  __syncthreads();
  if (tid == 0) sm.flag = atomicAdd(&cnt[kCntExit], 1u) == gridDim.x - 1 ? 1 : 0;
  __syncthreads();
  if (sm.flag) {
    __threadfence();
    for (int i = tid; i < a.n_counters; i += blockDim.x) cnt[i] = 0u;
    // every row's entries, whatever the next launch's row count
    for (int i = tid; i < kDecodeRows * E; i += blockDim.x) a.sel[i] = __uint_as_float(kUnwritten);
    // performed before this CTA retires: a decode launch that follows directly (programmatic
    // dependent launch) starts only after every CTA of this one has left
    __threadfence();
  }
}

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------

int decode_mix_ctas(int hc, int hidden) { return (hc * hidden + kMixCols - 1) / kMixCols; }
int decode_router_epc(int experts) { return (experts + 63) / 64 < kMaxEpc ? (experts + 63) / 64 : kMaxEpc; }
int decode_router_ctas(int experts) {
  const int epc = decode_router_epc(experts);
  return (experts + epc - 1) / epc;
}
// the tensor-core kernel's counters extend the CUDA-core kernel's
int decode_counter_count(const Dims &d) { return decode_tc_counter_count(d); }

struct DecodeTcMaps;
void launch_decode_tc(const DecodeArgs &a, const Dims &d, const Scratch &s, const LayerDev &w, int rows, int grid,
                      cudaStream_t st);

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
static size_t decode_smem(bool mx) { return mx ? Ring<true>::kSmem : Ring<false>::kSmem; }

cudaError_t decode_configure(int hidden) {
  (void)hidden;
  for (int mx = 0; mx < 2; ++mx)
    for (int r = 1; r <= kDecodeRows; ++r) {
      const cudaError_t e = cudaFuncSetAttribute(decode_kernel_for(r, mx != 0),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)decode_smem(mx != 0));
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

int decode_resident_ctas(int hidden, int rows, int num_sms, bool mx) {
  (void)hidden;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel_for(rows, mx), kDecThreads,
                                                    decode_smem(mx)) != cudaSuccess)
    return 0;
  return per_sm * num_sms;
}

void launch_decode(const Dims &d, const Scratch &s, const LayerDev &w, const float *state, const int32_t *token_ids,
                   int rows, bool hash, float *out_state, cudaStream_t st, StageTimer *tm, const DebugOpts &dbg) {
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
  a.epc = decode_router_epc(d.experts);
  a.nr = decode_router_ctas(d.experts);
  a.mix_part = s.mix_partial;
  a.mixes = s.mixes;
  a.pre = s.pre;
  a.post = s.post;
  a.comb = s.comb;
  a.x = s.ffn_norm;
  a.sel = s.dec_part;
  a.logits = s.logits;
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
  a.eps = d.eps;
  a.wait_ns = dbg.wait_ns ? dbg.wait_ns : kSpinLimitNs;
  a.inject = dbg.inject;
  // the tensor-core kernel; MXFP8 layers take it at four rows only (on the 4096 x 2048, 256-expert
  // shapes it measured 229 us against this kernel's 296 us at four rows, but 184 / 136 / 83 us
  // against 172 / 109 / 72 us at three / two / one rows)
  if (w.mx ? s.dtc_mx && w.mx_tc && rows == kDecodeRows : s.dtc)
    launch_decode_tc(a, d, s, w, rows, w.mx ? s.decode_ctas_mx[rows] : s.decode_ctas_by_rows[rows], st);
  else
    launch_pdl(decode_kernel_for(rows, w.mx), dim3(w.mx ? s.decode_ctas_mx_cc[rows] : s.decode_ctas_by_rows[rows]),
               dim3(kDecThreads), decode_smem(w.mx), st, a);
  stage(tm, "decode", st);
}

}  // namespace moe
