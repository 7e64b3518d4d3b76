// Decode path (rows <= 4) of the routed + shared experts: one persistent weight-streaming kernel.
//
// docs.rs "hf2q 0.1.3 .../deepseek4/ffn_forward.rs", forward_ffn_rows: expert_matmul "routed
// gate"/"routed up", raw_matmul "shared gate"/"shared up", dispatch_deepseek_moe_swiglu,
// expert_matmul "routed down", raw_matmul "shared down", dispatch_deepseek_moe_weighted_reduce,
// dispatch_hc_post.
//
// At 1-4 tokens every expert weight byte feeds 1-4 multiply-adds, so the work is bound by HBM
// bandwidth.  The router groups the batch's (row, slot) pairs by expert (group 0 = the shared
// expert); each weight row is streamed once by one warp with 16-byte loads, whatever the number of
// batch rows that use it.  Activations stay f32.
//
// One launch covers all of it, so HBM never idles between the gate/up and down projections.  Work
// is handed out by device-wide tickets (warps that stream faster take more), in three phases:
//   phase A  gate/up rows, group-major with the shared expert first, so groups complete in turn:
//            act[g, r, i] = silu(x_r . G[i]) * (x_r . U[i]); each row bumps its group's counter;
//   phase B  down rows, group-major; a group's rows wait (bounded) until its gate/up rows are all
//            published, then y[g, r, d] = act[g, r, :] . Dn[d, :]; each ticket bumps its d-block;
//   phase C  per 32-wide d-block, once every group's rows of it are in: ffn_out = sum_g w * y and
//            the hc_post output of that block.
// The grid is exactly the number of co-resident CTAs, every ticket of a phase is claimed before
// any warp moves to the next phase, and phase-A work never waits: so every wait ends.  Waits still
// give up after 1 s (device timeout bit).
#include "common.cuh"
#include "kernels.h"

namespace moe {

struct DecodeArgs {
  const int *ngroups, *group_e, *group_mask;
  const float *group_w;
  const float *ffn_input, *row_rs, *norm_w;  // x = ffn_input * row_rs * norm_w (= ffn_norm)
  float *ffn_norm;                           // written by CTA 0 (stage tap)
  const float *mixes, *hc_scale, *hc_base;   // for the comb, formed here off the critical path
  int iters;
  const uint16_t *gate_exps, *up_exps, *down_exps, *gate_sh, *up_sh, *down_sh;
  float *act;      // [groups, 4, inter]
  float *y;        // [groups, 4, hidden]
  unsigned *counters;  // [kDecodeGroupsMax] rows done per group, then [hidden / 64] d-block arrivals
  const float *state, *post;
  float *comb;
  float *ffn_out, *out_state;
  int *status;
  int rows, hidden, inter, experts, hc;
};

constexpr uint64_t kSpinLimitNs = 1000000000ull;

__device__ __forceinline__ uint4 ld_weight(const uint16_t *p, bool routed, uint64_t pol) {
  (void)routed;
  (void)pol;
  return ld_stream(p);
}

// Final reduce + hc_post of d-block `blk` (32 d, one per lane) by one warp, once its y rows and the
// comb are published.  y holds zeros for the rows a group does not serve, so the sum over groups
// is unconditional and its loads are batched.  s_pre holds this lane's state values, loaded before
// the wait.
__device__ void combine_dblock(const DecodeArgs &a, int blk, int ng, const float (&s_pre)[kDecodeRows][kHcMax]) {
  const int lane = threadIdx.x & 31, D = a.hidden, hc = a.hc;
  const int d = blk * kDecodeDBlock + lane;
#pragma unroll
  for (int r = 0; r < kDecodeRows; ++r) {
    if (r >= a.rows) break;
    float f = 0.f;
#pragma unroll 8
    for (int g = 0; g < ng; ++g)
      f += __ldcg(a.group_w + g * kDecodeRows + r) * __ldcg(a.y + ((size_t)g * kDecodeRows + r) * D + d);
    a.ffn_out[(size_t)r * D + d] = f;
#pragma unroll
    for (int o = 0; o < kHcMax; ++o) {
      if (o < hc) {
        float v = __ldcg(a.post + r * hc + o) * f;
#pragma unroll
        for (int j = 0; j < kHcMax; ++j)
          if (j < hc) v += __ldcg(a.comb + (r * hc + o) * hc + j) * s_pre[r][j];
        a.out_state[((size_t)r * hc + o) * D + d] = v;
      }
    }
  }
}

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

// Adds n to a completion counter with release semantics: this thread's earlier writes are visible
// to whoever acquires the new value.  No value is returned, so the warp does not wait for it.
__device__ __forceinline__ void publish(unsigned *counter, unsigned n) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(counter), "r"(n) : "memory");
}

// Bounded wait (lane 0 polls, the warp follows) until *counter >= target; every lane then acquires
// the counter so its later reads see what the producers published.  False on timeout.
__device__ bool wait_at_least(const unsigned *counter, unsigned target, int *status) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0 && ld_acquire_u32(counter) < target) {
    const uint64_t w0 = global_timer_ns();
    while (ld_acquire_u32(counter) < target) {
      if (global_timer_ns() - w0 > kSpinLimitNs) {
        atomicOr(status, kDevTimeout);
        ok = 0;
        break;
      }
      __nanosleep(128);
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) (void)ld_acquire_u32(counter);
  return ok != 0;
}

// Next work ticket of a phase: lane 0 draws it, the warp shares it.
__device__ __forceinline__ int draw_ticket(unsigned *tick) {
  int c = 0;
  if ((threadIdx.x & 31) == 0) c = (int)atomicAdd(tick, 1u);
  return __shfl_sync(0xffffffffu, c, 0);
}

constexpr int kRowsPerTicketA = 2;  // gate/up rows per ticket
constexpr int kRowsPerTicketB = 4;  // down rows per ticket (a 64-row d-block holds 16 tickets)

__global__ void __launch_bounds__(256, 2) decode_experts_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) float xs[];  // [rows, hidden]
  pdl_wait();
  const int D = a.hidden, I = a.inter, rows = a.rows, E = a.experts;
  for (int i = threadIdx.x * 4; i < rows * D; i += blockDim.x * 4) {
    const int r = i / D;
    const float rs = __ldcg(a.row_rs + r);
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.ffn_input + i));
    const float4 w = *reinterpret_cast<const float4 *>(a.norm_w + (i - r * D));
    const float4 x = make_float4(v.x * rs * w.x, v.y * rs * w.y, v.z * rs * w.z, v.w * rs * w.w);
    *reinterpret_cast<float4 *>(&xs[i]) = x;
    if (blockIdx.x == 0) *reinterpret_cast<float4 *>(a.ffn_norm + i) = x;
  }
  __syncthreads();
  const uint64_t pol = make_policy_evict_first();
  const int lane = threadIdx.x & 31;
  const int gwarp = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int last_warp = gridDim.x * (blockDim.x >> 5) - 1;
  const int ng = *a.ngroups;
  const int nblk = D / kDecodeDBlock;
  unsigned *group_done = a.counters;
  unsigned *dblock_done = a.counters + kDecodeGroupsMax;
  unsigned *comb_ready = dblock_done + nblk;
  unsigned *tick = comb_ready + 1;  // [3]
  if (gwarp == last_warp) {
    // The hc x hc comb (Sinkhorn) is only needed by the final hc_post: form it here, one thread
    // per row, while the other warps stream the expert weights.
    if (lane < rows)
      sinkhorn_comb_row(a.mixes + (size_t)lane * ((2 + a.hc) * a.hc), a.hc_scale, a.hc_base, a.hc, a.iters,
                        a.comb + (size_t)lane * a.hc * a.hc);
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      publish(comb_ready, 1u);
    }
    return;
  }

  // ---- phase A: gate/up rows, tickets in group-major order (the shared expert first) ----
  // Every row's 2 x hidden bf16 are in flight at once (UA loads per lane per matrix).
  constexpr int UA = 8;
  const int TA = ng * I, nA = (TA + kRowsPerTicketA - 1) / kRowsPerTicketA;
  for (int c = draw_ticket(&tick[0]); c < nA;) {
    int next = 0;
    if (lane == 0) next = (int)atomicAdd(&tick[0], 1u);  // consumed after this chunk: latency hidden
    const int t_end = min(TA, (c + 1) * kRowsPerTicketA);
    for (int t = c * kRowsPerTicketA; t < t_end; ++t) {
      const int g = t / I, i = t - g * I;
      const int e = a.group_e[g];
      const int mask = a.group_mask[g];
      const bool routed = e < E;
      const uint16_t *gw = routed ? a.gate_exps + ((size_t)e * I + i) * D : a.gate_sh + (size_t)i * D;
      const uint16_t *uw = routed ? a.up_exps + ((size_t)e * I + i) * D : a.up_sh + (size_t)i * D;
      float ga[kDecodeRows] = {0.f, 0.f, 0.f, 0.f}, ua[kDecodeRows] = {0.f, 0.f, 0.f, 0.f};
      for (int base = lane * 8; base < D; base += 256 * UA) {
        uint4 gv[UA], uv[UA];
#pragma unroll
        for (int u = 0; u < UA; ++u) {
          const int cc = base + u * 256;
          if (cc < D) {
            gv[u] = ld_weight(gw + cc, routed, pol);
            uv[u] = ld_weight(uw + cc, routed, pol);
          }
        }
#pragma unroll
        for (int u = 0; u < UA; ++u) {
          const int cc = base + u * 256;
          if (cc < D) {
#pragma unroll
            for (int r = 0; r < kDecodeRows; ++r) {
              if (r < rows) {
                const float4 x0 = *reinterpret_cast<const float4 *>(&xs[r * D + cc]);
                const float4 x1 = *reinterpret_cast<const float4 *>(&xs[r * D + cc + 4]);
                ga[r] += dot8(gv[u], x0, x1);
                ua[r] += dot8(uv[u], x0, x1);
              }
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kDecodeRows; ++r) {
        if (r < rows) {
          const float gs = warp_sum(ga[r]);
          const float us = warp_sum(ua[r]);
          if (lane == 0 && ((mask >> r) & 1)) a.act[((size_t)g * kDecodeRows + r) * I + i] = gs * sigmoidf_(gs) * us;
        }
      }
      if (lane == 0) publish(&group_done[g], 1u);
    }
    c = __shfl_sync(0xffffffffu, next, 0);
  }

  // ---- phase B: down rows, tickets in group-major order; a ticket's rows share one group and one
  // d-block.  A group's rows wait (bounded) until all of its gate/up rows are published.
  constexpr int UB = 8;
  const int TB = ng * D, nB = TB / kRowsPerTicketB;
  int cur = -1;
  bool ready = false;
  for (int c = draw_ticket(&tick[1]); c < nB;) {
    int next = 0;
    if (lane == 0) next = (int)atomicAdd(&tick[1], 1u);
    const int t0 = c * kRowsPerTicketB;
    const int g = t0 / D, d0 = t0 - g * D;
    if (g != cur) {
      cur = g;
      ready = wait_at_least(&group_done[g], (unsigned)I, a.status);
    }
    const int e = a.group_e[g];
    const int mask = a.group_mask[g];
    const bool routed = e < E;
    if (ready) {
      const float *act = a.act + (size_t)g * kDecodeRows * I;
#pragma unroll 1
      for (int q = 0; q < kRowsPerTicketB; q += 2) {
        // two down rows in flight together
        const int dd = d0 + q;
        const uint16_t *dw0 = routed ? a.down_exps + ((size_t)e * D + dd) * I : a.down_sh + (size_t)dd * I;
        const uint16_t *dw1 = dw0 + I;
        float acc0[kDecodeRows] = {0.f, 0.f, 0.f, 0.f}, acc1[kDecodeRows] = {0.f, 0.f, 0.f, 0.f};
        for (int base = lane * 8; base < I; base += 256 * UB) {
          uint4 w0[UB], w1[UB];
#pragma unroll
          for (int u = 0; u < UB; ++u) {
            if (base + u * 256 < I) {
              w0[u] = ld_weight(dw0 + base + u * 256, routed, pol);
              w1[u] = ld_weight(dw1 + base + u * 256, routed, pol);
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

  // ---- phase C: per d-block, once all groups' rows of it are in, ffn_out and hc_post ----
  for (int c = draw_ticket(&tick[2]); c < nblk; c = draw_ticket(&tick[2])) {
    float s_pre[kDecodeRows][kHcMax];
    const int d = c * kDecodeDBlock + lane;
#pragma unroll
    for (int r = 0; r < kDecodeRows; ++r)
#pragma unroll
      for (int j = 0; j < kHcMax; ++j)
        s_pre[r][j] = (r < rows && j < a.hc) ? a.state[((size_t)r * a.hc + j) * D + d] : 0.f;
    if (wait_at_least(&dblock_done[c], (unsigned)(ng * kDecodeDBlock), a.status) &&
        wait_at_least(comb_ready, 1u, a.status))
      combine_dblock(a, c, ng, s_pre);
  }
}

cudaError_t decode_configure(int hidden) {
  return cudaFuncSetAttribute(decode_experts_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kDecodeRows * hidden * (int)sizeof(float));
}

int decode_resident_ctas(int hidden, int rows, int num_sms) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_experts_kernel, 256,
                                                    (size_t)rows * hidden * sizeof(float)) != cudaSuccess)
    return 0;
  return per_sm * num_sms;
}

void launch_decode_experts(const Dims &d, const Scratch &s, const LayerDev &w, const float *state, int rows,
                           float *out_state, int num_sms, cudaStream_t st, StageTimer *tm) {
  (void)num_sms;
  DecodeArgs a;
  a.ngroups = s.ngroups;
  a.group_e = s.group_e;
  a.group_mask = s.group_mask;
  a.group_w = s.group_w;
  a.ffn_input = s.ffn_input;
  a.row_rs = s.row_rs;
  a.norm_w = w.ffn_norm;
  a.ffn_norm = s.ffn_norm;
  a.mixes = s.mixes;
  a.hc_scale = w.hc_scale;
  a.hc_base = w.hc_base;
  a.iters = d.iters;
  a.gate_exps = w.gate_exps;
  a.up_exps = w.up_exps;
  a.down_exps = w.down_exps;
  a.gate_sh = w.gate_sh;
  a.up_sh = w.up_sh;
  a.down_sh = w.down_sh;
  a.act = s.act_dec;
  a.y = s.y_dec;
  a.counters = s.dec_counters;
  a.state = state;
  a.post = s.post;
  a.comb = s.comb;
  a.ffn_out = s.ffn_out;
  a.out_state = out_state;
  a.status = s.status;
  a.rows = rows;
  a.hidden = d.hidden;
  a.inter = d.inter;
  a.experts = d.experts;
  a.hc = d.hc;
  const size_t xs_bytes = (size_t)rows * d.hidden * sizeof(float);
  launch_pdl(decode_experts_kernel, dim3(s.decode_ctas_by_rows[rows]), dim3(256), xs_bytes, st, a);
  stage(tm, "decode_experts", st);
}

}  // namespace moe
