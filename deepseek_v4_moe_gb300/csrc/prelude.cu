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
  float *partial;   // [rows, M + 1, chunks]
  unsigned *tickets;
  float *mixes, *pre, *post, *comb;
  const float *norm_w;  // with x_norm: the last CTA also forms x_norm = RMSNorm(hc_pre(state, pre)) * norm_w
  float *x_norm;        // [rows, hidden], or null
  int rows, hcd, M, hc, chunk, iters;
  float eps;
};

// hc_pre and the sublayer's RMSNorm for rows r0..r0+nr-1 by the last 128 threads of the mix's
// last CTA (warps 4-7; the first four run the Sinkhorn meanwhile), synchronised by named barrier 1.
// A row's x waits in shared memory (hidden <= 8192 = kPrenormSlots x 128 threads x 4 columns)
// for its RMS; the state loads go out four slots (16 float4) at a time, so a row of hidden 4096
// costs two round trips to L2, where the mix CTAs just left the state.  The loops stay rolled:
// this code runs once per call, mostly out of a cold instruction cache.
constexpr int kPrenormThreads = 128, kPrenormSlots = 16, kPrenormBatch = 4;
__device__ __forceinline__ void prenorm_barrier() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ void prenorm_rows(const MixArgs &a, int r0, int nr, int t, const float *sums, const float *scale,
                             const float *base) {
  __shared__ float red[kPrenormThreads / 32];
  __shared__ float4 xs[kPrenormSlots * kPrenormThreads];  // slot k of thread t at k * 128 + t
  const int hc = a.hc, hidden = a.hcd / hc;
  const int w = t >> 5, lane = t & 31;
  for (int r = r0; r < r0 + nr; ++r) {
    // pre of row r from its reduced sums (row r - r0 of sums, stride kMixMax + 1), exactly as the
    // split forms it
    const float *sm = sums + (size_t)(r - r0) * (kMixMax + 1);
    const float rs = rsqrtf(sm[a.M] / (float)a.hcd + a.eps);
    float p[kHcMax];
#pragma unroll
    for (int h = 0; h < kHcMax; ++h) p[h] = h < hc ? sigmoidf_(sm[h] * rs * scale[0] + base[h]) : 0.f;
    float ss = 0.f;
#pragma unroll 1
    for (int k0 = 0; k0 < kPrenormSlots; k0 += kPrenormBatch) {
      if (k0 * kPrenormThreads * 4 >= hidden) break;  // uniform: no slot of this batch is in range
      float4 v[kPrenormBatch][kHcMax];
#pragma unroll
      for (int k = 0; k < kPrenormBatch; ++k) {
        const int d = ((k0 + k) * kPrenormThreads + t) * 4;
#pragma unroll
        for (int h = 0; h < kHcMax; ++h)
          v[k][h] = (d < hidden && h < hc)
                        ? __ldcg(reinterpret_cast<const float4 *>(a.state + ((size_t)r * hc + h) * hidden + d))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < kPrenormBatch; ++k) {
        float4 xv = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int h = 0; h < kHcMax; ++h) {
          xv.x += p[h] * v[k][h].x;
          xv.y += p[h] * v[k][h].y;
          xv.z += p[h] * v[k][h].z;
          xv.w += p[h] * v[k][h].w;
        }
        xs[(k0 + k) * kPrenormThreads + t] = xv;
        ss += xv.x * xv.x + xv.y * xv.y + xv.z * xv.z + xv.w * xv.w;
      }
    }
    ss = warp_sum(ss);
    if (lane == 0) red[w] = ss;
    prenorm_barrier();
    float tot = 0.f;
#pragma unroll
    for (int q = 0; q < kPrenormThreads / 32; ++q) tot += red[q];
    const float xrs = rsqrtf(tot / (float)hidden + a.eps);
#pragma unroll 4
    for (int k = 0; k < kPrenormSlots; ++k) {
      const int d = (k * kPrenormThreads + t) * 4;
      if (d < hidden) {
        const float4 g = *reinterpret_cast<const float4 *>(a.norm_w + d);
        const float4 x = xs[k * kPrenormThreads + t];
        *reinterpret_cast<float4 *>(a.x_norm + (size_t)r * hidden + d) =
            make_float4(x.x * xrs * g.x, x.y * xrs * g.y, x.z * xrs * g.z, x.w * xrs * g.w);
      }
    }
    prenorm_barrier();  // red is reused by the next row
  }
}

int hc_mix_chunks(int rows, int hcd) {
  if (rows <= kDecodeRows) return hcd / 128;
  return hcd % 512 == 0 ? 2 : hcd / 128;
}

template <int RB>
__global__ void __launch_bounds__(256, 2) hc_mix_kernel(MixArgs a) {
  pdl_trigger();
  const int nch = gridDim.x;
  const int c0 = blockIdx.x * a.chunk;
  const int r0 = blockIdx.y * RB;
  const int nr = min(RB, a.rows - r0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = a.M;
  __shared__ float s_scale[3], s_base[kMixMax];
  if (threadIdx.x < 3) s_scale[threadIdx.x] = a.hc_scale[threadIdx.x];
  if (threadIdx.x < M) s_base[threadIdx.x] = a.hc_base[threadIdx.x];
  pdl_wait();
  float acc[RB][3], ss[RB];
#pragma unroll
  for (int r = 0; r < RB; ++r) {
    ss[r] = 0.f;
#pragma unroll
    for (int q = 0; q < 3; ++q) acc[r][q] = 0.f;
  }
  // Each lane walks its 4-column slots of the chunk; the next slot's loads are issued before the
  // current slot's FMAs, so two global round trips are always in flight.
  auto load_slot = [&](int c, float4 (&x)[RB], uint2 (&w)[3]) {
#pragma unroll
    for (int r = 0; r < RB; ++r)
      x[r] = (r < nr) ? *reinterpret_cast<const float4 *>(a.state + (size_t)(r0 + r) * a.hcd + c)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const int m = warp + 8 * q;
      w[q] = m < M ? __ldg(reinterpret_cast<const uint2 *>(a.hc_fn + (size_t)m * a.hcd + c)) : make_uint2(0u, 0u);
    }
  };
  auto fma_slot = [&](const float4 (&x)[RB], const uint2 (&w)[3]) {
#pragma unroll
    for (int r = 0; r < RB; ++r) ss[r] += x[r].x * x[r].x + x[r].y * x[r].y + x[r].z * x[r].z + x[r].w * x[r].w;
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const float w0 = bf_lo(w[q].x), w1 = bf_hi(w[q].x), w2 = bf_lo(w[q].y), w3 = bf_hi(w[q].y);
#pragma unroll
      for (int r = 0; r < RB; ++r) acc[r][q] += x[r].x * w0 + x[r].y * w1 + x[r].z * w2 + x[r].w * w3;
    }
  };
  {
    const int slots = a.chunk / 128;
    float4 xa[RB], xb[RB];
    uint2 wa[3], wb[3];
    int c = c0 + lane * 4;
    load_slot(c, xa, wa);
    for (int k = 0; k < slots; k += 2) {
      if (k + 1 < slots) load_slot(c + 128, xb, wb);
      fma_slot(xa, wa);
      if (k + 1 >= slots) break;
      if (k + 2 < slots) load_slot(c + 256, xa, wa);
      fma_slot(xb, wb);
      c += 256;
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
      float *p = a.partial + (size_t)(r0 + r) * (M + 1) * nch + blockIdx.x;
#pragma unroll
      for (int q = 0; q < 3; ++q)
        if (warp + 8 * q < M) p[(size_t)(warp + 8 * q) * nch] = acc[r][q];
      if (warp == 0) p[(size_t)M * nch] = ss[r];
    }
  }
  __threadfence();
  __syncthreads();
  __shared__ int is_last;
  if (threadIdx.x == 0) is_last = (atomicAdd(&a.tickets[blockIdx.y], 1u) == (unsigned)(nch - 1));
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // Reduce the chunk partials: tpi threads per (row, value), each over a strided share of the
  // chunks with independent loads, then a shuffle tree; fixed order, so deterministic.
  __shared__ float sums[RB][kMixMax + 1];
  const int items = nr * (M + 1);
  int tpi = 32;
  while (tpi > 1 && items * tpi > (int)blockDim.x) tpi >>= 1;
  for (int i = threadIdx.x; i < ((items * tpi + 31) / 32) * 32; i += blockDim.x) {
    const int item = i / tpi, part = i % tpi;
    float s = 0.f;
    if (item < items) {
      const float *p = a.partial + (size_t)(r0 * (M + 1) + item) * nch;
#pragma unroll 16
      for (int ch = part; ch < nch; ch += tpi) s += __ldcg(p + ch);
    }
    for (int o = tpi >> 1; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (part == 0 && item < items) sums[item / (M + 1)][item % (M + 1)] = s;
  }
  __syncthreads();
  // warps 0-3, one row each: the split, lane-parallel (mixes = sums * rs; pre and post from the
  // first 2hc), then the comb (warp Sinkhorn).  Warps 4-7 meanwhile: x_norm, forming pre
  // themselves from the same sums by the same expression (x_norm needs pre, not the comb).
  __shared__ float s_mix[RB][kMixMax];
  if (warp < nr) {
    const int r = r0 + warp, hc = a.hc;
    const float rs = rsqrtf(sums[warp][M] / (float)a.hcd + a.eps);
    if (lane < M) {
      const float mx = sums[warp][lane] * rs;
      s_mix[warp][lane] = mx;
      a.mixes[(size_t)r * M + lane] = mx;
      if (lane < hc)
        a.pre[(size_t)r * hc + lane] = sigmoidf_(mx * s_scale[0] + s_base[lane]);
      else if (lane < 2 * hc)
        a.post[(size_t)r * hc + lane - hc] = 2.0f * sigmoidf_(mx * s_scale[1] + s_base[lane]);
    }
    __syncwarp();
    sinkhorn_comb_warp(s_mix[warp], s_scale, s_base, hc, a.iters, a.comb + (size_t)r * hc * hc);
  } else if (a.x_norm && threadIdx.x >= 256 - kPrenormThreads) {
    prenorm_rows(a, r0, nr, threadIdx.x - (256 - kPrenormThreads), &sums[0][0], s_scale, s_base);
  }
  if (threadIdx.x == 0) a.tickets[blockIdx.y] = 0u;
}

// Same kernel with caller-chosen scratch (the allocation-free entry point's fixed array).
void launch_hc_mix_raw(const float *state, const uint16_t *hc_fn, const float *hc_scale, const float *hc_base,
                       int rows, int hc, int hidden, int iters, float eps, float *partial, unsigned *tickets,
                       float *mixes, float *pre, float *post, float *comb, cudaStream_t st, const float *norm_w,
                       float *x_norm) {
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
  a.norm_w = norm_w;
  a.x_norm = x_norm;
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

// Routes row r with one warp.  `logits` is the row's logits (shared or global memory), `v` a
// shared buffer of `experts` floats for the row's selection scores.  The code stays compact (the
// serial tail runs once per forward, mostly out of a cold instruction cache): candidates are
// scanned with a rolled loop, and slot k of the result lives in lane k.
__device__ void route_row_warp(const float *logits, int r, const RouteParams &p, float *v, int *s_idx = nullptr,
                               float *s_w = nullptr) {
  const int lane = threadIdx.x & 31;
  const int E = p.experts, K = p.top_k;
  int my_sel = -1;
  if (!p.hash) {
    bool bad = false;
    for (int e = lane; e < E; e += 32) {
      const float l = logits[e];
      bad |= !isfinite(l);
      const float x = sigmoidf_(l) + p.bias[e];
      v[e] = isnan(x) ? -INFINITY : x;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, kDevNonFinite);
    __syncwarp();
    uint32_t taken = 0;
#pragma unroll 1
    for (int k = 0; k < K; ++k) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll 1
      for (int j = 0, e = lane; e < E; ++j, e += 32) {
        const float x = v[e];
        if (!((taken >> j) & 1u) && (x > bv || be == 0x7fffffff)) {
          bv = x;
          be = e;
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
      if (lane == k) my_sel = be;
    }
  } else {
    const int tok = p.token_ids[r];
    const bool tok_ok = tok >= 0 && tok < p.vocab;
    if (!tok_ok && lane == 0) atomicOr(p.status, kDevTokenRange);
    if (lane < K) my_sel = tok_ok ? p.tid2eid[(size_t)tok * K + lane] : -1;
    const bool bad_entry = tok_ok && lane < K && !(my_sel >= 0 && my_sel < E);
    if (__any_sync(0xffffffffu, bad_entry) && lane == 0) atomicOr(p.status, kDevRouteRange);
  }
  const bool valid = lane < K && my_sel >= 0 && my_sel < E;
  const float sc = valid ? sigmoidf_(logits[my_sel]) : 0.f;
  const float tot = warp_sum(sc);
  if (lane < K) {
    const float w = tot > 0.f ? sc / tot : 0.f;
    p.idx[(size_t)r * K + lane] = my_sel;
    p.rw[(size_t)r * K + lane] = w;
    p.safe[(size_t)r * K + lane] = valid ? (unsigned)my_sel : 0u;
    if (p.counts && valid) atomicAdd(&p.counts[my_sel], 1);
    if (s_idx) {
      s_idx[lane] = my_sel;
      s_w[lane] = w;
    }
  }
}

RouteParams make_route(const Dims &d, const Scratch &s, const LayerDev &w, const int32_t *token_ids,
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

// ---------------------------------------------------------------------------------------------
// Rows > 4: per-row hc_pre + ffn_norm, a tiled f32 router GEMM, then one warp per row routes
// and counts slots per expert for the dispatch.
// ---------------------------------------------------------------------------------------------
// One CTA per row: ffn_input = sum_h pre[h] * state[h] (in shared memory), then ffn_norm =
// ffn_input * rsqrt(mean(ffn_input^2) + eps) * w.  With zero_acc set, also clears that row of the
// f64 FFN output, which the down GEMM's epilogue accumulates into.
__global__ void __launch_bounds__(256) prefill_prenorm_kernel(const float *__restrict__ state,
                                                              const float *__restrict__ pre,
                                                              const float *__restrict__ norm_w, int hidden, int hc,
                                                              float eps, float *__restrict__ ffn_norm,
                                                              double *__restrict__ zero_acc) {
  extern __shared__ __align__(16) float xin[];
  __shared__ float red[8];
  const int r = blockIdx.x, tid = threadIdx.x;
  float p[kHcMax];
#pragma unroll
  for (int h = 0; h < kHcMax; ++h) p[h] = h < hc ? pre[(size_t)r * hc + h] : 0.f;
  float ss = 0.f;
  for (int dd = tid * 4; dd < hidden; dd += blockDim.x * 4) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int h = 0; h < kHcMax; ++h) {
      if (h >= hc) break;
      const float4 x = *reinterpret_cast<const float4 *>(state + ((size_t)r * hc + h) * hidden + dd);
      v.x += p[h] * x.x;
      v.y += p[h] * x.y;
      v.z += p[h] * x.z;
      v.w += p[h] * x.w;
    }
    *reinterpret_cast<float4 *>(&xin[dd]) = v;
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
    if (zero_acc) {
      double2 *z = reinterpret_cast<double2 *>(zero_acc + (size_t)r * hidden + dd);
      z[0] = make_double2(0.0, 0.0);
      z[1] = make_double2(0.0, 0.0);
    }
  }
}

__global__ void __launch_bounds__(256) route_rows_kernel(const float *__restrict__ part, int nsplit, float *logits,
                                                         int rows, RouteParams p) {
  __shared__ float sv[8][kExpertsMax];
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const int E = p.experts;
  float *lr = logits + (size_t)r * E;
  for (int e = threadIdx.x & 31; e < E; e += 32) {
    float l = 0.f;
    for (int z = 0; z < nsplit; ++z) l += part[((size_t)z * rows + r) * E + e];
    lr[e] = l;
  }
  __syncwarp();
  route_row_warp(lr, r, p, sv[threadIdx.x >> 5]);
}

void launch_prefill_router(const Dims &d, const Scratch &s, const LayerDev &w, const float *state,
                           const int32_t *token_ids, const CUtensorMap &tm_ffn_norm, int rows, bool hash, int num_sms,
                           cudaStream_t st, StageTimer *tm) {
  prefill_prenorm_kernel<<<rows, 256, d.hidden * sizeof(float), st>>>(state, s.pre, w.ffn_norm, d.hidden, d.hc,
                                                                       d.eps, s.ffn_norm, s.ffn_acc);
  stage(tm, "prenorm", st);
  // logits on the tensor cores (splitgemm.cu), split over K so that the grid fills the GPU
  const int nsplit = launch_router_tc(d, s, w, tm_ffn_norm, rows, num_sms, st);
  stage(tm, "router_gemm", st);
  RouteParams p = make_route(d, s, w, token_ids, hash, s.counts);
  route_rows_kernel<<<(rows + 7) / 8, 256, 0, st>>>(s.router_part, nsplit, s.logits, rows, p);
  stage(tm, "route", st);
}

// The HC prelude of a sublayer on its own (the attention sublayer, or the FFN's without its
// body): pre/post/comb into the caller's buffers, then hc_pre + the sublayer's RMSNorm into x_norm.
// Rows <= 4 take the split-K CUDA-core mix; more rows the tensor-core split GEMM (tm_state set).
void launch_hc_pre(const Dims &d, const Scratch &s, const LayerDev &w, const float *state, const CUtensorMap *tm_state,
                   int rows, int num_sms, float *x_norm, float *pre, float *post, float *comb, cudaStream_t st) {
  if (rows <= kDecodeRows) {  // one launch: the mix's last CTA also forms x_norm
    launch_hc_mix_raw(state, w.hc_fn, w.hc_scale, w.hc_base, rows, d.hc, d.hidden, d.iters, d.eps, s.mix_partial,
                      s.tickets, s.mixes, pre, post, comb, st, w.ffn_norm, x_norm);
    return;
  }
  Scratch s2 = s;
  s2.pre = pre;
  s2.post = post;
  s2.comb = comb;
  launch_prefill_mix(d, s2, w, state, *tm_state, rows, num_sms, st, nullptr);
  prefill_prenorm_kernel<<<rows, 256, d.hidden * sizeof(float), st>>>(state, pre, w.ffn_norm, d.hidden, d.hc, d.eps,
                                                                       x_norm, nullptr);
}

}  // namespace moe
