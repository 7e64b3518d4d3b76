// Hyper-connection prelude and router of the MoE-FFN block (docs.rs "hf2q 0.1.3
// .../deepseek4/ffn_forward.rs", forward_ffn_rows: rms_norm_no_scale_f32, raw_matmul "HC FFN
// function", dispatch_hc_split_sinkhorn, dispatch_hc_pre, rms_norm, raw_matmul "MoE gate",
// dispatch_deepseek_moe_{score,hash}_route, dispatch_deepseek_moe_sanitize_indices).
//
// All of it is f32 CUDA-core arithmetic: the router's top-k must agree exactly with an f64
// reference whenever the selection margin exceeds 1e-5, which bf16/fp16 tensor-core inputs would
// not guarantee.  The work is small (0.8 MB hc_fn + 2 MB router per decode call) and latency
// bound, so it is spread over many CTAs with split-K partial sums; the CTA that finishes last
// (a device-scope ticket) reduces the partials in a fixed order and runs the serial tail.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

// ---------------------------------------------------------------------------------------------
// HC mix: per row, ss = sum x^2 and dot_m = sum x * hc_fn[m] over the flattened hc*hidden state;
// mixes = dot * rsqrt(ss / (hc*hidden) + eps) (the RMS scale factors out of the dot product).
// Grid (chunks, row groups of RB); the last CTA of a row group splits the mixes into pre, post
// and the Sinkhorn-balanced comb.
// ---------------------------------------------------------------------------------------------
struct MixArgs {
  const float *state;
  const uint16_t *hc_fn;
  const float *hc_scale, *hc_base;
  float *partial;
  unsigned *tickets;
  float *mixes, *pre, *post, *comb;
  int rows, hcd, M, hc, chunk, iters;
  float eps;
};

__device__ void split_sinkhorn_row(const float *sums, const MixArgs &a, int r) {
  const int hc = a.hc, M = a.M;
  const float rs = rsqrtf(sums[M] / (float)a.hcd + a.eps);
  float mix[kMixMax];
  for (int m = 0; m < M; ++m) {
    mix[m] = sums[m] * rs;
    a.mixes[(size_t)r * M + m] = mix[m];
  }
  const float s0 = a.hc_scale[0], s1 = a.hc_scale[1], s2 = a.hc_scale[2];
  for (int h = 0; h < hc; ++h) {
    a.pre[(size_t)r * hc + h] = sigmoidf_(mix[h] * s0 + a.hc_base[h]);
    a.post[(size_t)r * hc + h] = 2.0f * sigmoidf_(mix[hc + h] * s1 + a.hc_base[hc + h]);
  }
  float c[kHcMax][kHcMax];
  for (int i = 0; i < hc; ++i) {
    float mx = -INFINITY;
    for (int j = 0; j < hc; ++j) {
      c[i][j] = mix[2 * hc + i * hc + j] * s2 + a.hc_base[2 * hc + i * hc + j];
      mx = fmaxf(mx, c[i][j]);
    }
    for (int j = 0; j < hc; ++j) c[i][j] = expf(c[i][j] - mx);
  }
  for (int it = 0; it < a.iters; ++it) {
    for (int i = 0; i < hc; ++i) {
      float s = 0.f;
      for (int j = 0; j < hc; ++j) s += c[i][j];
      for (int j = 0; j < hc; ++j) c[i][j] = c[i][j] / s;
    }
    for (int j = 0; j < hc; ++j) {
      float s = 0.f;
      for (int i = 0; i < hc; ++i) s += c[i][j];
      for (int i = 0; i < hc; ++i) c[i][j] = c[i][j] / s;
    }
  }
  for (int i = 0; i < hc; ++i)
    for (int j = 0; j < hc; ++j) a.comb[((size_t)r * hc + i) * hc + j] = c[i][j];
}

template <int RB>
__global__ void __launch_bounds__(256) hc_mix_kernel(MixArgs a) {
  const int nch = gridDim.x;
  const int c0 = blockIdx.x * a.chunk;
  const int r0 = blockIdx.y * RB;
  const int nr = min(RB, a.rows - r0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = a.M;
  float acc[RB][3], ss[RB];
#pragma unroll
  for (int r = 0; r < RB; ++r) {
    ss[r] = 0.f;
#pragma unroll
    for (int q = 0; q < 3; ++q) acc[r][q] = 0.f;
  }
  for (int c = c0 + lane * 4; c < c0 + a.chunk; c += 128) {
    float4 x[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r)
      x[r] = (r < nr) ? *reinterpret_cast<const float4 *>(a.state + (size_t)(r0 + r) * a.hcd + c)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < RB; ++r) ss[r] += x[r].x * x[r].x + x[r].y * x[r].y + x[r].z * x[r].z + x[r].w * x[r].w;
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const int m = warp + 8 * q;
      if (m < M) {
        const uint2 wv = __ldg(reinterpret_cast<const uint2 *>(a.hc_fn + (size_t)m * a.hcd + c));
        const float w0 = bf_lo(wv.x), w1 = bf_hi(wv.x), w2 = bf_lo(wv.y), w3 = bf_hi(wv.y);
#pragma unroll
        for (int r = 0; r < RB; ++r) acc[r][q] += x[r].x * w0 + x[r].y * w1 + x[r].z * w2 + x[r].w * w3;
      }
    }
  }
#pragma unroll
  for (int r = 0; r < RB; ++r) {
    ss[r] = warp_sum(ss[r]);
#pragma unroll
    for (int q = 0; q < 3; ++q) acc[r][q] = warp_sum(acc[r][q]);
  }
  if (lane == 0) {
    for (int r = 0; r < nr; ++r) {
      float *p = a.partial + ((size_t)(r0 + r) * nch + blockIdx.x) * (M + 1);
#pragma unroll
      for (int q = 0; q < 3; ++q)
        if (warp + 8 * q < M) p[warp + 8 * q] = acc[r][q];
      if (warp == 0) p[M] = ss[r];
    }
  }
  __threadfence();
  __syncthreads();
  __shared__ int is_last;
  if (threadIdx.x == 0) is_last = (atomicAdd(&a.tickets[blockIdx.y], 1u) == (unsigned)(nch - 1));
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  __shared__ float sums[RB][kMixMax + 1];
  for (int i = threadIdx.x; i < nr * (M + 1); i += blockDim.x) {
    const int r = i / (M + 1), v = i - r * (M + 1);
    const float *p = a.partial + (size_t)(r0 + r) * nch * (M + 1) + v;
    float s = 0.f;
    for (int ch = 0; ch < nch; ++ch) s += __ldcg(p + (size_t)ch * (M + 1));
    sums[r][v] = s;
  }
  __syncthreads();
  if (threadIdx.x < nr) split_sinkhorn_row(sums[threadIdx.x], a, r0 + threadIdx.x);
  if (threadIdx.x == 0) a.tickets[blockIdx.y] = 0u;
}

void launch_hc_mix(const Dims &d, const Scratch &s, const LayerDev &w, const float *state, int rows,
                   cudaStream_t st, StageTimer *tm) {
  MixArgs a;
  a.state = state;
  a.hc_fn = w.hc_fn;
  a.hc_scale = w.hc_scale;
  a.hc_base = w.hc_base;
  a.partial = s.mix_partial;
  a.tickets = s.tickets;
  a.mixes = s.mixes;
  a.pre = s.pre;
  a.post = s.post;
  a.comb = s.comb;
  a.rows = rows;
  a.hcd = d.hc * d.hidden;
  a.M = d.mix();
  a.hc = d.hc;
  a.iters = d.iters;
  a.eps = d.eps;
  // Decode: 128-column chunks so that the 0.8 MB hc_fn read spreads over ~128 CTAs.
  // Prefill: 4 chunks per row group of 4 rows.
  const int nch = rows <= kDecodeRows ? a.hcd / 128 : (a.hcd % 512 == 0 ? 4 : a.hcd / 128);
  a.chunk = a.hcd / nch;
  dim3 grid(nch, (rows + 3) / 4);
  hc_mix_kernel<4><<<grid, 256, 0, st>>>(a);
  stage(tm, "hc_mix", st);
}

// Same kernel with caller-chosen scratch (the allocation-free entry point's fixed array).
int hc_mix_chunks(int rows, int hcd) {
  return rows <= kDecodeRows ? hcd / 128 : (hcd % 512 == 0 ? 4 : hcd / 128);
}

void launch_hc_mix_raw(const float *state, const uint16_t *hc_fn, const float *hc_scale, const float *hc_base,
                       int rows, int hc, int hidden, int iters, float eps, float *partial, unsigned *tickets,
                       float *mixes, float *pre, float *post, float *comb, cudaStream_t st) {
  MixArgs a;
  a.state = state;
  a.hc_fn = hc_fn;
  a.hc_scale = hc_scale;
  a.hc_base = hc_base;
  a.partial = partial;
  a.tickets = tickets;
  a.mixes = mixes;
  a.pre = pre;
  a.post = post;
  a.comb = comb;
  a.rows = rows;
  a.hcd = hc * hidden;
  a.M = (2 + hc) * hc;
  a.hc = hc;
  a.iters = iters;
  a.eps = eps;
  const int nch = hc_mix_chunks(rows, a.hcd);
  a.chunk = a.hcd / nch;
  dim3 grid(nch, (rows + 3) / 4);
  hc_mix_kernel<4><<<grid, 256, 0, st>>>(a);
}

// ---------------------------------------------------------------------------------------------
// Routing of one row by one warp.  Score layers: sigmoid scores, top_k on score + bias in f32
// (ties to the lower expert index), weights = chosen unbiased scores / their sum.  Hash layers:
// tid2eid[token] in table order, weights = sigmoid(logit) normalised over valid slots.
// ---------------------------------------------------------------------------------------------
struct RouteParams {
  int experts, top_k, vocab;
  bool hash;
  const float *bias;
  const int32_t *tid2eid;
  const int32_t *token_ids;
  int *idx;
  float *rw;
  unsigned *safe;
  int *status;
  int *counts;  // optional per-expert histogram (rows > 4 path)
};

__device__ void route_row_warp(const float *logits, int r, const RouteParams &p) {
  const int lane = threadIdx.x & 31;
  const int E = p.experts, K = p.top_k;
  int sel[kTopKMax];
  float sc[kTopKMax];
  bool valid[kTopKMax];
  if (!p.hash) {
    constexpr int J = kExpertsMax / 32;
    float val[J];
    bool bad = false;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int e = lane + 32 * j;
      val[j] = -INFINITY;
      if (e < E) {
        const float l = logits[e];
        bad |= !isfinite(l);
        const float v = sigmoidf_(l) + p.bias[e];
        val[j] = isnan(v) ? -INFINITY : v;
      }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, kDevNonFinite);
    uint32_t taken = 0;
    for (int k = 0; k < K; ++k) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        if (e < E && !((taken >> j) & 1u)) {
          if (val[j] > bv || be == 0x7fffffff) {
            bv = val[j];
            be = e;
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      sel[k] = be;
      valid[k] = true;
    }
  } else {
    const int tok = p.token_ids[r];
    const bool tok_ok = tok >= 0 && tok < p.vocab;
    if (!tok_ok && lane == 0) atomicOr(p.status, kDevTokenRange);
    for (int k = 0; k < K; ++k) {
      const int e = tok_ok ? p.tid2eid[(size_t)tok * K + k] : -1;
      sel[k] = e;
      valid[k] = e >= 0 && e < E;
      if (tok_ok && !valid[k] && lane == 0) atomicOr(p.status, kDevRouteRange);
    }
  }
  float tot = 0.f;
  for (int k = 0; k < K; ++k) {
    sc[k] = valid[k] ? sigmoidf_(logits[sel[k]]) : 0.f;
    tot += sc[k];
  }
  if (lane == 0) {
    for (int k = 0; k < K; ++k) {
      p.idx[(size_t)r * K + k] = sel[k];
      p.rw[(size_t)r * K + k] = tot > 0.f ? sc[k] / tot : 0.f;
      p.safe[(size_t)r * K + k] = valid[k] ? (unsigned)sel[k] : 0u;
      if (p.counts && valid[k]) atomicAdd(&p.counts[sel[k]], 1);
    }
  }
}

// ---------------------------------------------------------------------------------------------
// Decode router (rows <= 4).  Grid: hidden/128 chunks of d.  Each CTA forms ffn_input =
// sum_h pre[h] * state[h] on its chunk, partial sum of squares, and partial logits
// sum_d ffn_input[d] * w[d] * gate[e, d] for every expert (the RMS scale factors out).  The last
// CTA reduces, writes logits and ffn_norm, routes each row and groups the (row, slot) pairs by
// expert for the expert kernels (the shared expert is the last group, weight 1).
// ---------------------------------------------------------------------------------------------
struct DecodeRouterArgs {
  const float *state, *pre, *norm_w;
  const uint16_t *gate;
  float *ffn_input, *ffn_norm, *partial, *logits;
  unsigned *ticket;
  int *ngroups, *group_e, *group_mask;
  float *group_w;
  int rows, hidden, hc;
  float eps;
  RouteParams rp;
};

constexpr int kRouterChunk = 128;

__global__ void __launch_bounds__(256) decode_router_kernel(DecodeRouterArgs a) {
  const int nch = gridDim.x;
  const int d0 = blockIdx.x * kRouterChunk;
  const int E = a.rp.experts, rows = a.rows, tid = threadIdx.x;
  __shared__ __align__(16) float xw[kDecodeRows][kRouterChunk];
  __shared__ float red[8][kDecodeRows];
  __shared__ float rs_s[kDecodeRows];
  __shared__ int is_last;

  float ssl[kDecodeRows];
#pragma unroll
  for (int r = 0; r < kDecodeRows; ++r) {
    ssl[r] = 0.f;
    if (r < rows && tid < kRouterChunk) {
      const int d = d0 + tid;
      float v = 0.f;
      for (int h = 0; h < a.hc; ++h) v += a.pre[r * a.hc + h] * a.state[((size_t)r * a.hc + h) * a.hidden + d];
      a.ffn_input[(size_t)r * a.hidden + d] = v;
      xw[r][tid] = v * a.norm_w[d];
      ssl[r] = v * v;
    }
  }
#pragma unroll
  for (int r = 0; r < kDecodeRows; ++r) {
    const float v = warp_sum(ssl[r]);
    if ((tid & 31) == 0) red[tid >> 5][r] = v;
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    float acc[kDecodeRows] = {0.f, 0.f, 0.f, 0.f};
    const uint16_t *g = a.gate + (size_t)e * a.hidden + d0;
#pragma unroll 4
    for (int dd = 0; dd < kRouterChunk; dd += 8) {
      const uint4 wv = __ldg(reinterpret_cast<const uint4 *>(g + dd));
#pragma unroll
      for (int r = 0; r < kDecodeRows; ++r)
        if (r < rows)
          acc[r] += dot8(wv, *reinterpret_cast<const float4 *>(&xw[r][dd]),
                         *reinterpret_cast<const float4 *>(&xw[r][dd + 4]));
    }
    for (int r = 0; r < rows; ++r) a.partial[((size_t)r * nch + blockIdx.x) * (E + 1) + e] = acc[r];
  }
  if (tid < rows) {
    float s = 0.f;
    for (int w = 0; w < 8; ++w) s += red[w][tid];
    a.partial[((size_t)tid * nch + blockIdx.x) * (E + 1) + E] = s;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = (atomicAdd(a.ticket, 1u) == (unsigned)(nch - 1));
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  __shared__ float lg[kDecodeRows][kExpertsMax];
  if (tid < rows) {
    float s = 0.f;
    for (int ch = 0; ch < nch; ++ch) s += __ldcg(a.partial + ((size_t)tid * nch + ch) * (E + 1) + E);
    rs_s[tid] = rsqrtf(s / (float)a.hidden + a.eps);
  }
  __syncthreads();
  for (int i = tid; i < rows * E; i += blockDim.x) {
    const int r = i / E, e = i - r * E;
    float s = 0.f;
    for (int ch = 0; ch < nch; ++ch) s += __ldcg(a.partial + ((size_t)r * nch + ch) * (E + 1) + e);
    const float l = s * rs_s[r];
    lg[r][e] = l;
    a.logits[(size_t)r * E + e] = l;
  }
  for (int i = tid; i < rows * a.hidden; i += blockDim.x) {
    const int r = i / a.hidden, d = i - r * a.hidden;
    a.ffn_norm[i] = __ldcg(a.ffn_input + i) * rs_s[r] * a.norm_w[d];
  }
  __syncthreads();
  const int warp = tid >> 5;
  if (warp < rows) route_row_warp(lg[warp], warp, a.rp);
  __syncthreads();
  if (tid == 0) {
    const int K = a.rp.top_k;
    int ng = 0;
    for (int r = 0; r < rows; ++r)
      for (int k = 0; k < K; ++k) {
        const int e = a.rp.idx[r * K + k];
        if (e < 0 || e >= E) continue;
        int g = 0;
        while (g < ng && a.group_e[g] != e) ++g;
        if (g == ng) {
          a.group_e[g] = e;
          a.group_mask[g] = 0;
          for (int q = 0; q < kDecodeRows; ++q) a.group_w[g * kDecodeRows + q] = 0.f;
          ++ng;
        }
        a.group_mask[g] |= 1 << r;
        a.group_w[g * kDecodeRows + r] += a.rp.rw[r * K + k];
      }
    a.group_e[ng] = E;  // shared expert
    a.group_mask[ng] = (1 << rows) - 1;
    for (int q = 0; q < kDecodeRows; ++q) a.group_w[ng * kDecodeRows + q] = q < rows ? 1.f : 0.f;
    *a.ngroups = ng + 1;
    *a.ticket = 0u;
  }
}

static RouteParams make_route(const Dims &d, const Scratch &s, const LayerDev &w, const int32_t *token_ids,
                              bool hash, int *counts) {
  RouteParams p;
  p.experts = d.experts;
  p.top_k = d.top_k;
  p.vocab = d.vocab;
  p.hash = hash;
  p.bias = w.exp_probs_b;
  p.tid2eid = w.tid2eid;
  p.token_ids = token_ids;
  p.idx = s.idx;
  p.rw = s.rw;
  p.safe = s.safe;
  p.status = s.status;
  p.counts = counts;
  return p;
}

void launch_decode_router(const Dims &d, const Scratch &s, const LayerDev &w, const float *state,
                          const int32_t *token_ids, int rows, bool hash, cudaStream_t st, StageTimer *tm) {
  DecodeRouterArgs a;
  a.state = state;
  a.pre = s.pre;
  a.norm_w = w.ffn_norm;
  a.gate = w.gate;
  a.ffn_input = s.ffn_input;
  a.ffn_norm = s.ffn_norm;
  a.partial = s.router_partial;
  a.logits = s.logits;
  a.ticket = s.tickets + (s.max_rows / 4 + 1);
  a.ngroups = s.ngroups;
  a.group_e = s.group_e;
  a.group_mask = s.group_mask;
  a.group_w = s.group_w;
  a.rows = rows;
  a.hidden = d.hidden;
  a.hc = d.hc;
  a.eps = d.eps;
  a.rp = make_route(d, s, w, token_ids, hash, nullptr);
  decode_router_kernel<<<d.hidden / kRouterChunk, 256, 0, st>>>(a);
  stage(tm, "decode_router", st);
}

// ---------------------------------------------------------------------------------------------
// Rows > 4: per-row hc_pre + ffn_norm, a tiled f32 router GEMM, then one warp per row routes
// and counts slots per expert for the dispatch.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) prefill_prenorm_kernel(const float *__restrict__ state,
                                                              const float *__restrict__ pre,
                                                              const float *__restrict__ norm_w, int hidden, int hc,
                                                              float eps, float *__restrict__ ffn_input,
                                                              float *__restrict__ ffn_norm) {
  extern __shared__ __align__(16) float xin[];
  __shared__ float red[8];
  const int r = blockIdx.x, tid = threadIdx.x;
  float p[kHcMax];
  for (int h = 0; h < kHcMax; ++h) p[h] = h < hc ? pre[(size_t)r * hc + h] : 0.f;
  float ss = 0.f;
  for (int dd = tid * 4; dd < hidden; dd += blockDim.x * 4) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int h = 0; h < hc; ++h) {
      const float4 x = *reinterpret_cast<const float4 *>(state + ((size_t)r * hc + h) * hidden + dd);
      v.x += p[h] * x.x;
      v.y += p[h] * x.y;
      v.z += p[h] * x.z;
      v.w += p[h] * x.w;
    }
    *reinterpret_cast<float4 *>(&xin[dd]) = v;
    *reinterpret_cast<float4 *>(ffn_input + (size_t)r * hidden + dd) = v;
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
  const float rs = rsqrtf(tot / (float)hidden + eps);
  for (int dd = tid * 4; dd < hidden; dd += blockDim.x * 4) {
    const float4 v = *reinterpret_cast<const float4 *>(&xin[dd]);
    const float4 g = *reinterpret_cast<const float4 *>(norm_w + dd);
    *reinterpret_cast<float4 *>(ffn_norm + (size_t)r * hidden + dd) =
        make_float4(v.x * rs * g.x, v.y * rs * g.y, v.z * rs * g.z, v.w * rs * g.w);
  }
}

// logits[R, E] = X[R, D] . G[E, D]^T, X f32, G bf16; 64x64 tile, 4x4 per thread.
__global__ void __launch_bounds__(256) router_gemm_kernel(const float *__restrict__ X, const uint16_t *__restrict__ G,
                                                          int R, int E, int D, float *__restrict__ out) {
  __shared__ float Xs[32][68];
  __shared__ float Gs[32][68];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int r0 = blockIdx.y * 64, e0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < D; k0 += 32) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int id = tid + i * 256, row = id >> 3, kq = (id & 7) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r0 + row < R) v = *reinterpret_cast<const float4 *>(X + (size_t)(r0 + row) * D + k0 + kq);
      Xs[kq + 0][row] = v.x;
      Xs[kq + 1][row] = v.y;
      Xs[kq + 2][row] = v.z;
      Xs[kq + 3][row] = v.w;
    }
    {
      const int e = tid >> 2, kq = (tid & 3) * 8;
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (e0 + e < E) w = __ldg(reinterpret_cast<const uint4 *>(G + (size_t)(e0 + e) * D + k0 + kq));
      Gs[kq + 0][e] = bf_lo(w.x);
      Gs[kq + 1][e] = bf_hi(w.x);
      Gs[kq + 2][e] = bf_lo(w.y);
      Gs[kq + 3][e] = bf_hi(w.y);
      Gs[kq + 4][e] = bf_lo(w.z);
      Gs[kq + 5][e] = bf_hi(w.z);
      Gs[kq + 6][e] = bf_lo(w.w);
      Gs[kq + 7][e] = bf_hi(w.w);
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = Xs[k][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Gs[k][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + ty * 4 + i;
    if (r >= R) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) out[(size_t)r * E + e] = acc[i][j];
    }
  }
}

__global__ void __launch_bounds__(256) route_rows_kernel(const float *__restrict__ logits, int rows, RouteParams p) {
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= rows) return;
  route_row_warp(logits + (size_t)r * p.experts, r, p);
}

void launch_prefill_router(const Dims &d, const Scratch &s, const LayerDev &w, const float *state,
                           const int32_t *token_ids, int rows, bool hash, cudaStream_t st, StageTimer *tm) {
  prefill_prenorm_kernel<<<rows, 256, d.hidden * sizeof(float), st>>>(state, s.pre, w.ffn_norm, d.hidden, d.hc,
                                                                       d.eps, s.ffn_input, s.ffn_norm);
  stage(tm, "prenorm", st);
  dim3 g((d.experts + 63) / 64, (rows + 63) / 64);
  router_gemm_kernel<<<g, 256, 0, st>>>(s.ffn_norm, w.gate, rows, d.experts, d.hidden, s.logits);
  stage(tm, "router_gemm", st);
  RouteParams p = make_route(d, s, w, token_ids, hash, s.counts);
  route_rows_kernel<<<(rows + 7) / 8, 256, 0, st>>>(s.logits, rows, p);
  stage(tm, "route", st);
}

}  // namespace moe
