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
// One launch covers all of it, so HBM never idles between the gate/up and down projections:
//   phase A  warps take gate/up rows (group-major, shared expert first) and write
//            act[g, r, i] = silu(x_r . G[i]) * (x_r . U[i]); each finished row bumps its group's
//            counter;
//   phase B  warps take down rows (group-major); a row of group g waits (bounded) until all of
//            g's gate/up rows are done, then writes y[g, r, d] = act[g, r, :] . Dn[d, :]; the last
//            writer of a 64-wide d-block (a device-scope counter) forms ffn_out = sum_g w * y and
//            the hc_post output for that block.
// The grid is exactly the number of co-resident CTAs, and a phase-B wait only depends on phase-A
// rows, which never wait; so every wait ends.  Waits still give up after 1 s (device timeout bit).
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
  return routed ? ld_stream_hint(p, pol) : ld_stream(p);
}

// Final reduce + hc_post of d-block `blk` by one warp (after the comb is published).
__device__ void combine_dblock(const DecodeArgs &a, int blk, int ng, const unsigned *comb_ready) {
  const int lane = threadIdx.x & 31, D = a.hidden, hc = a.hc;
  int ok = 1;
  if (lane == 0 && ld_acquire_u32(comb_ready) == 0u) {
    const uint64_t w0 = global_timer_ns();
    while (ld_acquire_u32(comb_ready) == 0u) {
      if (global_timer_ns() - w0 > 1000000000ull) {
        atomicOr(a.status, kDevTimeout);
        ok = 0;
        break;
      }
      __nanosleep(100);
    }
  }
  if (!__shfl_sync(0xffffffffu, ok, 0)) return;
  (void)ld_acquire_u32(comb_ready);
  for (int d = blk * kDecodeDBlock + lane; d < (blk + 1) * kDecodeDBlock; d += 32) {
    for (int r = 0; r < a.rows; ++r) {
      float f = 0.f;
#pragma unroll 8
      for (int g = 0; g < ng; ++g) {
        if ((a.group_mask[g] >> r) & 1)
          f += a.group_w[g * kDecodeRows + r] * __ldcg(a.y + ((size_t)g * kDecodeRows + r) * D + d);
      }
      a.ffn_out[(size_t)r * D + d] = f;
      float s[kHcMax];
#pragma unroll
      for (int j = 0; j < kHcMax; ++j) s[j] = j < hc ? a.state[((size_t)r * hc + j) * D + d] : 0.f;
#pragma unroll
      for (int o = 0; o < kHcMax; ++o) {
        if (o < hc) {
          float v = a.post[r * hc + o] * f;
#pragma unroll
          for (int j = 0; j < kHcMax; ++j)
            if (j < hc) v += __ldcg(a.comb + (r * hc + o) * hc + j) * s[j];
          a.out_state[((size_t)r * hc + o) * D + d] = v;
        }
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

// Publishes `n` finished rows on a counter: the writes before it become visible first.
__device__ __forceinline__ unsigned publish(unsigned *counter, unsigned n) {
  __threadfence();
  return atomicAdd(counter, n);
}

__global__ void __launch_bounds__(256, 3) decode_experts_kernel(DecodeArgs a) {
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
  const int nwarps = gridDim.x * (blockDim.x >> 5) - 1;  // the grid's last warp forms the comb
  const int ng = *a.ngroups;
  unsigned *group_done = a.counters;
  unsigned *dblock_done = a.counters + kDecodeGroupsMax;
  unsigned *comb_ready = a.counters + kDecodeGroupsMax + D / kDecodeDBlock;
  if (gwarp == nwarps) {
    // The hc x hc comb (Sinkhorn) is only needed by the final hc_post: form it here, one thread
    // per row, while the other warps stream the expert weights.
    if (lane < rows)
      sinkhorn_comb_row(a.mixes + (size_t)lane * ((2 + a.hc) * a.hc), a.hc_scale, a.hc_base, a.hc, a.iters,
                        a.comb + (size_t)lane * a.hc * a.hc);
    __syncwarp();
    if (lane == 0) publish(comb_ready, 1u);
    return;
  }

  // ---- phase A: a contiguous range of gate/up rows per warp (group-major, shared expert first) ----
  constexpr int UA = 4;
  {
    const long long TA = (long long)ng * I;
    const int t0 = (int)(TA * gwarp / nwarps), t1 = (int)(TA * (gwarp + 1) / nwarps);
    int cur = -1, e = 0, mask = 0;
    bool routed = false;
    unsigned cnt = 0;
    for (int t = t0; t < t1; ++t) {
      const int g = t / I, i = t - g * I;
      if (g != cur) {
        if (cnt && lane == 0) publish(&group_done[cur], cnt);
        cur = g;
        cnt = 0;
        e = a.group_e[g];
        mask = a.group_mask[g];
        routed = e < E;
      }
      const uint16_t *gw = routed ? a.gate_exps + ((size_t)e * I + i) * D : a.gate_sh + (size_t)i * D;
      const uint16_t *uw = routed ? a.up_exps + ((size_t)e * I + i) * D : a.up_sh + (size_t)i * D;
      float ga[kDecodeRows] = {0.f, 0.f, 0.f, 0.f}, ua[kDecodeRows] = {0.f, 0.f, 0.f, 0.f};
      for (int base = lane * 8; base < D; base += 256 * UA) {
        uint4 gv[UA], uv[UA];
#pragma unroll
        for (int u = 0; u < UA; ++u) {
          const int c = base + u * 256;
          if (c < D) {
            gv[u] = ld_weight(gw + c, routed, pol);
            uv[u] = ld_weight(uw + c, routed, pol);
          }
        }
#pragma unroll
        for (int u = 0; u < UA; ++u) {
          const int c = base + u * 256;
          if (c < D) {
#pragma unroll
            for (int r = 0; r < kDecodeRows; ++r) {
              if (r < rows) {
                const float4 x0 = *reinterpret_cast<const float4 *>(&xs[r * D + c]);
                const float4 x1 = *reinterpret_cast<const float4 *>(&xs[r * D + c + 4]);
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
      ++cnt;
    }
    if (cnt && lane == 0) publish(&group_done[cur], cnt);
  }

  // ---- phase B: a contiguous range of down rows per warp; per completed d-block, reduce + hc_post ----
  constexpr int UB = 8;
  {
    const unsigned dblock_total = (unsigned)(ng * kDecodeDBlock);
    const long long TB = (long long)ng * D;
    const int t0 = (int)(TB * gwarp / nwarps), t1 = (int)(TB * (gwarp + 1) / nwarps);
    int cur = -1, e = 0, mask = 0, blk = -1;
    bool routed = false, ready = false;
    unsigned cnt = 0;
    auto flush_block = [&]() {
      unsigned prev = 0;
      if (lane == 0) prev = publish(&dblock_done[blk], cnt);
      prev = __shfl_sync(0xffffffffu, prev, 0);
      if (prev + cnt == dblock_total) {
        __threadfence();
        combine_dblock(a, blk, ng, comb_ready);
      }
    };
    for (int t = t0; t < t1; ++t) {
      const int g = t / D, dd = t - g * D;
      if (dd / kDecodeDBlock != blk || g != cur) {
        if (cnt) flush_block();
        blk = dd / kDecodeDBlock;
        cnt = 0;
      }
      if (g != cur) {
        cur = g;
        e = a.group_e[g];
        mask = a.group_mask[g];
        routed = e < E;
        int ok = 1;
        if (lane == 0 && ld_acquire_u32(&group_done[g]) < (unsigned)I) {
          const uint64_t w0 = global_timer_ns();
          while (ld_acquire_u32(&group_done[g]) < (unsigned)I) {
            if (global_timer_ns() - w0 > kSpinLimitNs) {
              atomicOr(a.status, kDevTimeout);
              ok = 0;
              break;
            }
            __nanosleep(100);
          }
        }
        ready = __shfl_sync(0xffffffffu, ok, 0) != 0;
        (void)ld_acquire_u32(&group_done[g]);  // each lane orders its act reads after the counter
      }
      if (ready) {
        const uint16_t *dw = routed ? a.down_exps + ((size_t)e * D + dd) * I : a.down_sh + (size_t)dd * I;
        const float *act = a.act + (size_t)g * kDecodeRows * I;
        float acc[kDecodeRows] = {0.f, 0.f, 0.f, 0.f};
        for (int base = lane * 8; base < I; base += 256 * UB) {
          uint4 wv[UB];
#pragma unroll
          for (int u = 0; u < UB; ++u)
            if (base + u * 256 < I) wv[u] = ld_weight(dw + base + u * 256, routed, pol);
#pragma unroll
          for (int u = 0; u < UB; ++u) {
            const int c = base + u * 256;
            if (c < I) {
#pragma unroll
              for (int r = 0; r < kDecodeRows; ++r) {
                if ((mask >> r) & 1) {
                  const float4 x0 = ld_ca4(act + (size_t)r * I + c);
                  const float4 x1 = ld_ca4(act + (size_t)r * I + c + 4);
                  acc[r] += dot8(wv[u], x0, x1);
                }
              }
            }
          }
        }
#pragma unroll
        for (int r = 0; r < kDecodeRows; ++r) {
          if (r < rows) {
            const float s = warp_sum(acc[r]);
            if (lane == 0 && ((mask >> r) & 1)) a.y[((size_t)g * kDecodeRows + r) * D + dd] = s;
          }
        }
      }
      ++cnt;
    }
    if (cnt) flush_block();
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
