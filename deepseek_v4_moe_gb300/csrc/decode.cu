// Decode path (rows <= 4) of the routed + shared experts: weight-streaming GEMVs.
//
// docs.rs "hf2q 0.1.3 .../deepseek4/ffn_forward.rs", forward_ffn_rows: expert_matmul "routed
// gate"/"routed up", raw_matmul "shared gate"/"shared up", dispatch_deepseek_moe_swiglu,
// expert_matmul "routed down", raw_matmul "shared down", dispatch_deepseek_moe_weighted_reduce,
// dispatch_hc_post.
//
// At 1-4 tokens every expert weight byte is used for 1-4 multiply-adds, so the kernels are bound
// by HBM bandwidth: each weight row is streamed once with 16-byte loads by one warp, whatever
// the number of rows of the batch that use the expert (the router groups slots by expert).
// Activations stay f32 (they are tiny), which keeps the GEMVs exact to f32 accumulation.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kGroupsMax = kDecodeRows * kTopKMax + 1;

struct DecodeArgs {
  const int *ngroups, *group_e, *group_mask;
  const float *group_w;
  const float *x;  // ffn_norm [rows, hidden]
  const uint16_t *gate_exps, *up_exps, *down_exps, *gate_sh, *up_sh, *down_sh;
  float *act;      // [groups, 4, inter]
  float *y;        // [groups, 4, hidden]
  const float *state, *post, *comb;
  float *ffn_out, *out_state;
  int rows, hidden, inter, experts, hc;
};

// Tasks (group, inter row i): act[g, r, i] = silu(x_r . G_e[i]) * (x_r . U_e[i]).
template <int UNROLL>
__global__ void __launch_bounds__(256) decode_gateup_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) float xs[];  // [rows, hidden]
  const int D = a.hidden, I = a.inter, rows = a.rows;
  for (int i = threadIdx.x * 4; i < rows * D; i += blockDim.x * 4)
    *reinterpret_cast<float4 *>(&xs[i]) = *reinterpret_cast<const float4 *>(a.x + i);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int total = *a.ngroups * I;
  for (int t = warp; t < total; t += nwarps) {
    const int g = t / I, i = t - g * I;
    const int e = a.group_e[g];
    const uint16_t *gw = e < a.experts ? a.gate_exps + ((size_t)e * I + i) * D : a.gate_sh + (size_t)i * D;
    const uint16_t *uw = e < a.experts ? a.up_exps + ((size_t)e * I + i) * D : a.up_sh + (size_t)i * D;
    float ga[kDecodeRows] = {0.f, 0.f, 0.f, 0.f}, ua[kDecodeRows] = {0.f, 0.f, 0.f, 0.f};
    for (int base = lane * 8; base < D; base += 256 * UNROLL) {
      uint4 gv[UNROLL], uv[UNROLL];
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int c = base + u * 256;
        if (c < D) {
          gv[u] = ld_stream(gw + c);
          uv[u] = ld_stream(uw + c);
        }
      }
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
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
    const int mask = a.group_mask[g];
#pragma unroll
    for (int r = 0; r < kDecodeRows; ++r) {
      if (r < rows) {
        const float gs = warp_sum(ga[r]);
        const float us = warp_sum(ua[r]);
        if (lane == 0 && ((mask >> r) & 1)) a.act[((size_t)g * kDecodeRows + r) * I + i] = gs * sigmoidf_(gs) * us;
      }
    }
  }
}

// Tasks (group, output d): y[g, r, d] = act[g, r, :] . Dn_e[d, :].
template <int UNROLL>
__global__ void __launch_bounds__(256) decode_down_kernel(DecodeArgs a) {
  const int D = a.hidden, I = a.inter, rows = a.rows;
  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int total = *a.ngroups * D;
  for (int t = warp; t < total; t += nwarps) {
    const int g = t / D, dd = t - g * D;
    const int e = a.group_e[g];
    const int mask = a.group_mask[g];
    const uint16_t *dw = e < a.experts ? a.down_exps + ((size_t)e * D + dd) * I : a.down_sh + (size_t)dd * I;
    const float *act = a.act + (size_t)g * kDecodeRows * I;
    float acc[kDecodeRows] = {0.f, 0.f, 0.f, 0.f};
    for (int base = lane * 8; base < I; base += 256 * UNROLL) {
      uint4 wv[UNROLL];
#pragma unroll
      for (int u = 0; u < UNROLL; ++u)
        if (base + u * 256 < I) wv[u] = ld_stream(dw + base + u * 256);
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int c = base + u * 256;
        if (c < I) {
#pragma unroll
          for (int r = 0; r < kDecodeRows; ++r) {
            if ((mask >> r) & 1) {
              const float4 x0 = __ldg(reinterpret_cast<const float4 *>(act + (size_t)r * I + c));
              const float4 x1 = __ldg(reinterpret_cast<const float4 *>(act + (size_t)r * I + c + 4));
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
}

// ffn_out[r, d] = sum_g w[g, r] * y[g, r, d] over the groups row r uses (shared weight 1);
// out[r, i, d] = post[r, i] * ffn_out[r, d] + sum_j comb[r, i, j] * state[r, j, d].
__global__ void __launch_bounds__(256) decode_combine_kernel(DecodeArgs a) {
  const int D = a.hidden, hc = a.hc;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.rows * D) return;
  const int r = i / D, d = i - r * D;
  const int ng = *a.ngroups;
  float f = 0.f;
  for (int g = 0; g < ng; ++g)
    if ((a.group_mask[g] >> r) & 1) f += a.group_w[g * kDecodeRows + r] * a.y[((size_t)g * kDecodeRows + r) * D + d];
  a.ffn_out[i] = f;
  float s[kHcMax];
  for (int j = 0; j < hc; ++j) s[j] = a.state[((size_t)r * hc + j) * D + d];
  for (int o = 0; o < hc; ++o) {
    float v = a.post[r * hc + o] * f;
    for (int j = 0; j < hc; ++j) v += a.comb[(r * hc + o) * hc + j] * s[j];
    a.out_state[((size_t)r * hc + o) * D + d] = v;
  }
}

cudaError_t decode_configure(int hidden) {
  return cudaFuncSetAttribute(decode_gateup_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kDecodeRows * hidden * (int)sizeof(float));
}

void launch_decode_experts(const Dims &d, const Scratch &s, const LayerDev &w, const float *state, int rows,
                           float *out_state, int num_sms, cudaStream_t st, StageTimer *tm) {
  DecodeArgs a;
  a.ngroups = s.ngroups;
  a.group_e = s.group_e;
  a.group_mask = s.group_mask;
  a.group_w = s.group_w;
  a.x = s.ffn_norm;
  a.gate_exps = w.gate_exps;
  a.up_exps = w.up_exps;
  a.down_exps = w.down_exps;
  a.gate_sh = w.gate_sh;
  a.up_sh = w.up_sh;
  a.down_sh = w.down_sh;
  a.act = s.act_dec;
  a.y = s.y_dec;
  a.state = state;
  a.post = s.post;
  a.comb = s.comb;
  a.ffn_out = s.ffn_out;
  a.out_state = out_state;
  a.rows = rows;
  a.hidden = d.hidden;
  a.inter = d.inter;
  a.experts = d.experts;
  a.hc = d.hc;
  const size_t xs_bytes = (size_t)rows * d.hidden * sizeof(float);
  decode_gateup_kernel<4><<<num_sms * 2, 256, xs_bytes, st>>>(a);
  stage(tm, "decode_gateup", st);
  decode_down_kernel<4><<<num_sms * 2, 256, 0, st>>>(a);
  stage(tm, "decode_down", st);
  decode_combine_kernel<<<(rows * d.hidden + 255) / 256, 256, 0, st>>>(a);
  stage(tm, "decode_combine", st);
}

}  // namespace moe
