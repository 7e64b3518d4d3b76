// Token -> expert dispatch of the rows > 4 path, and the hc_post kernel that closes it.
//
// The pages' mm_id path (expert_matmul with IdMmScratch in forward_ffn_rows, docs.rs "hf2q 0.1.3
// .../deepseek4/ffn_forward.rs") groups routed rows by expert; here that is a histogram (counted by
// the router), an exclusive scan, a tile list for the persistent grouped GEMMs, and a scatter of
// (row, slot) pairs with their activation rows (as bf16 hi and lo planes) into expert-sorted
// order.  The shared expert is the last group and holds every row.  The order of rows inside a
// group comes from atomics and does not affect the GEMMs' results: each token's output column is
// computed alone.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// Inclusive scan of one value per thread over a 1024-thread block (warp shuffles, then the warp
// totals); `tmp` holds 32 floats of scratch.
__device__ int block_scan_incl(int v, int *tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) tmp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int t = tmp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += n;
    }
    tmp[lane] = t;
  }
  __syncthreads();
  const int res = v + (warp > 0 ? tmp[warp - 1] : 0);
  __syncthreads();
  return res;
}

// Groups 0..E-1 are the routed experts (counts from the router), group E the shared expert (every
// row).  Exclusive scans give each group's first list position.  The gate/up and down tile lists are
// (group, weight block, token block, valid tokens) in two parts: first the tiles of the heavy groups
// (more than one token block, so each weight tile is multiplied several times: MMA-bound), then those
// of the light groups (one token block: bound by the weight bytes).  Within a part, group-major then
// weight-block-major, so the token blocks of one weight tile run side by side.  The GEMMs take tiles
// from both parts at once, which keeps the tensor pipes and DRAM busy together.  Resets the counts
// for the next forward and the GEMMs' claim counters.
__global__ void __launch_bounds__(1024) build_tiles_kernel(int *__restrict__ counts, int E, int rows, int mb_gu,
                                                           int mb_dn, int *__restrict__ offsets,
                                                           int *__restrict__ cursor, int4 *__restrict__ tiles_gu,
                                                           int4 *__restrict__ tiles_dn, int *__restrict__ n_tiles) {
  __shared__ int cnt[kExpertsMax + 1], nb[kExpertsMax + 1], toff[kExpertsMax + 2], poff[kExpertsMax + 1];
  __shared__ int tmp[32], parts[2];
  const int G = E + 1, g = threadIdx.x;
  const int c = g < G ? (g < E ? counts[g] : rows) : 0;
  const int n = (c + 127) / 128;
  const bool heavy = n >= 2;
  if (g < G) {
    cnt[g] = c;
    nb[g] = n;
    if (g < E) counts[g] = 0;
    cursor[g] = 0;
  }
  const int off_incl = block_scan_incl(c, tmp);
  const int tb_incl = block_scan_incl(n, tmp);
  const int hb_incl = block_scan_incl(heavy ? n : 0, tmp);  // token blocks of heavy groups
  const int lb_incl = block_scan_incl(heavy ? 0 : n, tmp);  // and of light ones
  if (g < G) {
    offsets[g] = off_incl - c;
    toff[g] = tb_incl - n;
    poff[g] = heavy ? hb_incl - n : lb_incl - n;  // first token block of the group within its part
  }
  if (g == G - 1) {
    offsets[G] = off_incl;
    toff[G] = tb_incl;
    parts[0] = hb_incl;  // heavy token blocks
    n_tiles[0] = tb_incl * mb_gu;
    n_tiles[1] = tb_incl * mb_dn;
    n_tiles[2] = hb_incl * mb_gu;
    n_tiles[3] = hb_incl * mb_dn;
    for (int i = 4; i < 8; ++i) n_tiles[i] = 0;
  }
  __syncthreads();
  const int total_b = toff[G], heavy_b = parts[0];
  // every (group, token block) pair, found by binary search over the group tile offsets
  for (int t = threadIdx.x; t < total_b * (mb_gu > mb_dn ? mb_gu : mb_dn); t += blockDim.x) {
    const int mb_max = mb_gu > mb_dn ? mb_gu : mb_dn;
    const int bt = t / mb_max, m = t - bt * mb_max;
    int lo = 0, hi = G - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (toff[mid] <= bt) lo = mid;
      else hi = mid - 1;
    }
    const int gg = lo, b = bt - toff[gg], nbg = nb[gg];
    const int base = nbg >= 2 ? poff[gg] : heavy_b + poff[gg];  // the group's first block in the list
    const int4 tile = make_int4(gg, m, b, min(128, cnt[gg] - b * 128));
    if (m < mb_gu) tiles_gu[base * mb_gu + m * nbg + b] = tile;
    if (m < mb_dn) tiles_dn[base * mb_dn + m * nbg + b] = tile;
  }
}

// One warp per (row, slot), slot top_k being the shared expert: claims the pair's position in its
// group, then writes the row's normalised input as two bf16 planes, hi = rn(x) at row pos of x2
// and lo = rn(x - hi) at row plane_rows + pos.
__global__ void __launch_bounds__(256) scatter_kernel(const int *__restrict__ idx, const float *__restrict__ rw,
                                                      const float *__restrict__ x, int rows, int K, int E, int D,
                                                      const int *__restrict__ offsets, int *__restrict__ cursor,
                                                      int2 *__restrict__ list, float *__restrict__ list_w,
                                                      uint16_t *__restrict__ x2, int plane_rows) {
  const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= rows * (K + 1)) return;
  const int r = w / (K + 1), k = w - r * (K + 1);
  int g;
  float wt;
  if (k < K) {
    const int e = idx[(size_t)r * K + k];
    if (e < 0 || e >= E) return;
    g = e;
    wt = rw[(size_t)r * K + k];
  } else {
    g = E;
    wt = 1.f;
  }
  int pos = 0;
  if (lane == 0) {
    pos = offsets[g] + atomicAdd(&cursor[g], 1);
    list[pos] = make_int2(r, k);
    list_w[pos] = wt;
  }
  pos = __shfl_sync(0xffffffffu, pos, 0);
  const float *src = x + (size_t)r * D;
  uint16_t *dhi = x2 + (size_t)pos * D, *dlo = x2 + ((size_t)plane_rows + pos) * D;
  for (int c = lane * 8; c < D; c += 256) {
    const float4 a = *reinterpret_cast<const float4 *>(src + c);
    const float4 b = *reinterpret_cast<const float4 *>(src + c + 4);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float h[8], l[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      h[j] = round_bf16(v[j]);
      l[j] = round_bf16(v[j] - h[j]);
    }
    *reinterpret_cast<uint4 *>(dhi + c) = make_uint4(pack_bf16_pair(h[0], h[1]), pack_bf16_pair(h[2], h[3]),
                                                     pack_bf16_pair(h[4], h[5]), pack_bf16_pair(h[6], h[7]));
    *reinterpret_cast<uint4 *>(dlo + c) = make_uint4(pack_bf16_pair(l[0], l[1]), pack_bf16_pair(l[2], l[3]),
                                                     pack_bf16_pair(l[4], l[5]), pack_bf16_pair(l[6], l[7]));
  }
}

void launch_dispatch(const Dims &d, const Scratch &s, int rows, cudaStream_t st, StageTimer *tm) {
  // down tiles cover two 128-row blocks of hidden each
  build_tiles_kernel<<<1, 1024, 0, st>>>(s.counts, d.experts, rows, d.inter / 128, (d.hidden + 255) / 256, s.offsets,
                                         s.cursor, s.tiles_gu, s.tiles_dn, s.n_tiles);
  stage(tm, "build_tiles", st);
  const int warps = rows * (d.top_k + 1);
  scatter_kernel<<<(warps + 7) / 8, 256, 0, st>>>(s.idx, s.rw, s.ffn_norm, rows, d.top_k, d.experts, d.hidden,
                                                  s.offsets, s.cursor, s.list, s.list_w, s.x2, s.max_positions);
  stage(tm, "scatter", st);
}

// hc_post of a sublayer whose output f is given (the FFN's ffn_out on the rows > 4 path, the
// attention sublayer's output projection, or any body): out[r, i, d] = post[r, i] * f[r, d] +
// sum_j comb[r, i, j] * state[r, j, d].  One thread per (row, 4 columns), a row's post and comb
// staged once per CTA.  Every byte is read or written once, so loads and stores take the streaming
// (evict-first) path.
constexpr int kHcPostThreads = 128;

__device__ __forceinline__ float4 ld_f4_stream(const float *p) { return __ldcs(reinterpret_cast<const float4 *>(p)); }
__device__ __forceinline__ float4 ld_f4_stream(const double *p) {
  const double2 a = __ldcs(reinterpret_cast<const double2 *>(p)), b = __ldcs(reinterpret_cast<const double2 *>(p) + 1);
  return make_float4((float)a.x, (float)a.y, (float)b.x, (float)b.y);  // the f64 FFN output rounded to f32 once
}

template <typename F>
__global__ void __launch_bounds__(kHcPostThreads) hc_post_kernel(const F *__restrict__ f,
                                                                  const float *__restrict__ state,
                                                                  const float *__restrict__ post,
                                                                  const float *__restrict__ comb, int D, int hc,
                                                                  int blocks_per_row, float *__restrict__ out) {
  const int r = blockIdx.x / blocks_per_row;
  const int d = ((blockIdx.x - r * blocks_per_row) * kHcPostThreads + threadIdx.x) * 4;
  __shared__ float pc[kHcMax + kHcMax * kHcMax];
  if (threadIdx.x < hc) pc[threadIdx.x] = post[(size_t)r * hc + threadIdx.x];
  if (threadIdx.x < hc * hc) pc[kHcMax + threadIdx.x] = comb[(size_t)r * hc * hc + threadIdx.x];
  __syncthreads();
  if (d >= D) return;
  const float4 fv = ld_f4_stream(f + (size_t)r * D + d);
  float4 sv[kHcMax];
#pragma unroll
  for (int j = 0; j < kHcMax; ++j)
    sv[j] = j < hc ? __ldcs(reinterpret_cast<const float4 *>(state + ((size_t)r * hc + j) * D + d))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int o = 0; o < kHcMax; ++o) {
    if (o >= hc) break;
    const float p = pc[o];
    float4 v = make_float4(p * fv.x, p * fv.y, p * fv.z, p * fv.w);
#pragma unroll
    for (int j = 0; j < kHcMax; ++j) {
      if (j >= hc) break;
      const float c = pc[kHcMax + o * hc + j];
      v.x += c * sv[j].x;
      v.y += c * sv[j].y;
      v.z += c * sv[j].z;
      v.w += c * sv[j].w;
    }
    __stcs(reinterpret_cast<float4 *>(out + ((size_t)r * hc + o) * D + d), v);
  }
}

template <typename F>
static void hc_post_launch(const Dims &d, const F *f, const float *state, const float *post, const float *comb,
                           int rows, float *out_state, cudaStream_t st) {
  const int per_row = (d.hidden / 4 + kHcPostThreads - 1) / kHcPostThreads;
  hc_post_kernel<F><<<(unsigned)rows * per_row, kHcPostThreads, 0, st>>>(f, state, post, comb, d.hidden, d.hc, per_row,
                                                                        out_state);
}

void launch_hc_post(const Dims &d, const float *f, const float *state, const float *post, const float *comb,
                    int rows, float *out_state, cudaStream_t st) {
  hc_post_launch(d, f, state, post, comb, rows, out_state, st);
}

void launch_hc_post(const Dims &d, const double *f, const float *state, const float *post, const float *comb,
                    int rows, float *out_state, cudaStream_t st) {
  hc_post_launch(d, f, state, post, comb, rows, out_state, st);
}

}  // namespace moe
