// C ABI of the MoE-FFN block: validation, scratch ownership, and the order of kernel launches.
// The argument checks mirror the guards of forward_ffn_rows (docs.rs "hf2q 0.1.3
// .../deepseek4/ffn_forward.rs"): layer range, at least one row, rows*top_k overflow, routing
// source present, output distinct from the input state.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "moe_ffn.h"

using moe::Dims;
using moe::LayerDev;
using moe::Scratch;

struct moe_ffn_handle {
  moe_ffn_config cfg;
  Dims dims;
  int device = 0, num_sms = 0;
  std::vector<LayerDev> layers;
  std::vector<LayerDev> attn;  // the attention sublayer's HC weights (hc fields and ffn_norm = attn_norm only)
  Scratch s;
  CUtensorMap tm_ffn_norm;
  CUtensorMap *tm_b = nullptr;  // device: [2][8] maps over x2 and act2, boxes of 16 .. 128 rows
  float *host_in = nullptr, *host_out = nullptr;  // device staging of moe_ffn_forward_host
  int32_t *host_tok = nullptr;
  std::vector<void *> allocs;
  cudaStream_t last_stream = nullptr;
  int last_rows = 0;
  moe::StageTimer timer;
  moe::DebugOpts dbg;  // test hooks (moe_ffn_set_fault_injection); defaults in normal use
  std::string err;
  // moe_ffn_forward_layers: captured chains (most recent use last) and the intermediate state
  struct Chain {
    const void *state, *tok, *out;
    int rows, first, n;
    cudaGraphExec_t exec;
  };
  std::vector<Chain> chains;
  cudaStream_t capture = nullptr;
  float *chain_state = nullptr;  // [max_rows, hc, hidden]
};

static constexpr size_t kMaxChains = 8;

// Message of the last failure without a handle, one per host thread: several threads may fail
// validation at the same time, and each reads back its own text.
static thread_local std::string g_init_err;

namespace moe {
void set_global_error(const char *msg) { g_init_err = msg; }
}  // namespace moe

static int fail(moe_ffn_handle *h, int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (h)
    h->err = buf;
  else
    g_init_err = buf;
  return code;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int check_config(const moe_ffn_config *c) {
  if (c->hc < 1 || c->hc > moe::kHcMax) return fail(nullptr, MOE_FFN_ERR_BAD_CONFIG, "hc must be in 1..4");
  if (c->hidden < 128 || c->hidden % 128 || c->hidden > 4096)
    return fail(nullptr, MOE_FFN_ERR_BAD_CONFIG, "hidden must be a multiple of 128 in 128..4096");
  if (c->inter < 128 || c->inter % 128 || c->inter > 2048)
    return fail(nullptr, MOE_FFN_ERR_BAD_CONFIG, "inter must be a multiple of 128 in 128..2048");
  if (c->shared_inter != c->inter) return fail(nullptr, MOE_FFN_ERR_BAD_CONFIG, "shared_inter must equal inter");
  if (c->experts < 16 || c->experts > moe::kExpertsMax || c->experts % 16)
    return fail(nullptr, MOE_FFN_ERR_BAD_CONFIG, "experts must be a multiple of 16 in 16..512");
  if (c->top_k < 1 || c->top_k > moe::kTopKMax || c->top_k > c->experts)
    return fail(nullptr, MOE_FFN_ERR_BAD_CONFIG, "top_k must be in 1..min(8, experts)");
  if (c->n_layers < 1 || c->hash_layer_count < 0 || c->hash_layer_count > c->n_layers)
    return fail(nullptr, MOE_FFN_ERR_BAD_CONFIG, "need n_layers >= 1 and 0 <= hash_layer_count <= n_layers");
  if (c->max_rows < 1 || c->max_rows > 65536) return fail(nullptr, MOE_FFN_ERR_BAD_CONFIG, "max_rows must be in 1..65536");
  if (c->vocab < 1) return fail(nullptr, MOE_FFN_ERR_BAD_CONFIG, "vocab must be positive");
  if (c->sinkhorn_iters < 0 || c->sinkhorn_iters > 100000)
    return fail(nullptr, MOE_FFN_ERR_BAD_CONFIG, "sinkhorn_iters out of range");
  if (!(c->rms_eps >= 0.f)) return fail(nullptr, MOE_FFN_ERR_BAD_CONFIG, "rms_eps must be >= 0");
  return MOE_FFN_OK;
}

static int check_layer(const moe_ffn_config *c, int l, const moe_ffn_layer_weights *w, bool *has, bool *experts) {
  const void *core[] = {w->hc_fn, w->hc_base, w->hc_scale, w->ffn_norm, w->gate};
  const void *exps[] = {w->gate_exps, w->up_exps, w->down_exps, w->gate_sh, w->up_sh, w->down_sh};
  int n_core = 0, n_exps = 0;
  for (const void *p : core) n_core += p != nullptr;
  for (const void *p : exps) n_exps += p != nullptr;
  *has = *experts = false;
  if (n_core == 0 && n_exps == 0 && !w->exp_probs_b && !w->tid2eid) return MOE_FFN_OK;
  if (n_core != (int)(sizeof core / sizeof core[0]))
    return fail(nullptr, MOE_FFN_ERR_NULL_PTR, "layer %d: some weight pointers are NULL", l);
  if (n_exps != 0 && n_exps != (int)(sizeof exps / sizeof exps[0]))
    return fail(nullptr, MOE_FFN_ERR_NULL_PTR,
                "layer %d: some expert pointers are NULL (give all six, or none and register MXFP8 experts)", l);
  const bool hash = l < c->hash_layer_count;
  if (hash && !w->tid2eid) return fail(nullptr, MOE_FFN_ERR_NO_ROUTING_SOURCE, "layer %d has no routing source (tid2eid)", l);
  if (!hash && !w->exp_probs_b)
    return fail(nullptr, MOE_FFN_ERR_NO_ROUTING_SOURCE, "layer %d has no routing source (exp_probs_b)", l);
  for (const void *p : core)
    if (!aligned16(p)) return fail(nullptr, MOE_FFN_ERR_ALIGNMENT, "layer %d: weight pointer not 16-byte aligned", l);
  for (const void *p : exps)
    if (p && !aligned16(p)) return fail(nullptr, MOE_FFN_ERR_ALIGNMENT, "layer %d: weight pointer not 16-byte aligned", l);
  *has = true;
  *experts = n_exps != 0;
  return MOE_FFN_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D f32 matrix [outer, inner], row-major; boxes of 128 rows x 64 columns, unswizzled (the
// tensor-core mix/router GEMMs convert them in shared memory); rows past `outer` read as zeros.
static bool make_tmap_f32(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 4};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 matrix [outer, inner], row-major; boxes of `box_rows` rows x 64 columns, 128-byte
// swizzle (the K-major operand layout of the tensor-core GEMMs); rows past `outer` read as zeros.
static bool make_tmap_bf16(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint32_t box_rows = 128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte matrix [outer, inner] (E4M3 codes), row-major; boxes of 128 rows x 64 bytes with the
// 64-byte swizzle (16-byte chunk c of box row n lands at chunk c ^ ((n / 2) % 4), so that the
// converter warps of the tensor-core decode, one row a thread, read them without bank conflicts);
// rows past `outer` read as zeros.
static bool make_tmap_u8(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T>
static bool dalloc(moe_ffn_handle *h, T **p, size_t count) {
  void *q = nullptr;
  const size_t bytes = count * sizeof(T) > 0 ? count * sizeof(T) : 16;
  if (cudaMalloc(&q, bytes) != cudaSuccess) return false;
  h->allocs.push_back(q);
  *p = static_cast<T *>(q);
  return true;
}

static void free_all(moe_ffn_handle *h) {
  for (void *p : h->allocs) cudaFree(p);
  h->allocs.clear();
}

// Tensor maps of a layer's expert matrices for the rows > 4 path: routed gate/up [experts * inter,
// hidden], routed down [experts * hidden, inter], and the shared expert's three matrices.
static bool expert_tmaps(const moe_ffn_handle *h, LayerDev &L, const uint16_t *g, const uint16_t *u, const uint16_t *dn,
                         const uint16_t *gs, const uint16_t *us, const uint16_t *ds) {
  const uint64_t E = h->dims.experts, I = h->dims.inter, D = h->dims.hidden;
  return make_tmap_bf16(&L.tm_gate, g, D, E * I) && make_tmap_bf16(&L.tm_up, u, D, E * I) &&
         make_tmap_bf16(&L.tm_down, dn, I, E * D) && make_tmap_bf16(&L.tm_gate_sh, gs, D, I) &&
         make_tmap_bf16(&L.tm_up_sh, us, D, I) && make_tmap_bf16(&L.tm_down_sh, ds, I, D);
}

extern "C" int moe_ffn_init(const moe_ffn_config *cfg, const moe_ffn_layer_weights *layers, moe_ffn_handle **out) {
  if (!out) return fail(nullptr, MOE_FFN_ERR_NULL_PTR, "out is NULL");
  *out = nullptr;
  if (!cfg || !layers) return fail(nullptr, MOE_FFN_ERR_NULL_PTR, "cfg or layers is NULL");
  int rc = check_config(cfg);
  if (rc) return rc;
  std::vector<bool> has(cfg->n_layers), has_exps(cfg->n_layers);
  for (int l = 0; l < cfg->n_layers; ++l) {
    bool hl = false, he = false;
    rc = check_layer(cfg, l, &layers[l], &hl, &he);
    if (rc) return rc;
    has[l] = hl;
    has_exps[l] = he;
  }
  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
    return fail(nullptr, MOE_FFN_ERR_CUDA, "no CUDA device");
  if (prop.major != 10 || prop.minor != 3)
    return fail(nullptr, MOE_FFN_ERR_UNSUPPORTED, "needs an sm_103 device, found sm_%d%d", prop.major, prop.minor);

  moe_ffn_handle *h = new moe_ffn_handle();
  h->cfg = *cfg;
  h->device = dev;
  h->num_sms = prop.multiProcessorCount;
  Dims &d = h->dims;
  d.hidden = cfg->hidden;
  d.hc = cfg->hc;
  d.experts = cfg->experts;
  d.top_k = cfg->top_k;
  d.inter = cfg->inter;
  d.vocab = cfg->vocab;
  d.iters = cfg->sinkhorn_iters;
  d.eps = cfg->rms_eps;
  const size_t R = cfg->max_rows, D = d.hidden, E = d.experts, K = d.top_k, I = d.inter, HC = d.hc, M = d.mix();
  const size_t hcd = HC * D;
  Scratch &s = h->s;
  s.max_rows = (int)R;
  s.mix_chunks = (int)(hcd / 128);
  s.router_chunks = (int)(D / 128);
  const size_t mix_part = std::max((size_t)4 * (hcd / 128), R * (size_t)moe::hc_mix_chunks((int)R, (int)hcd)) * (M + 1);
  const size_t G = moe::kDecodeRows * K + 1;
  bool ok = dalloc(h, &s.status, 1) && dalloc(h, &s.mix_partial, mix_part) && dalloc(h, &s.tickets, R / 4 + 2) &&
            dalloc(h, &s.mixes, R * M) && dalloc(h, &s.pre, R * HC) && dalloc(h, &s.post, R * HC) &&
            dalloc(h, &s.comb, R * HC * HC) && dalloc(h, &s.ffn_input, R * D) && dalloc(h, &s.ffn_norm, R * D) &&
            dalloc(h, &s.row_rs, R) &&
            dalloc(h, &s.dec_part, (size_t)moe::kDecodeRows * E * 2) &&
            dalloc(h, &s.logits, R * E) &&
            dalloc(h, &s.idx, R * K) && dalloc(h, &s.rw, R * K) && dalloc(h, &s.safe, R * K) &&
            dalloc(h, &s.ffn_out, R * D) && dalloc(h, &s.ngroups, 1) && dalloc(h, &s.group_e, G) &&
            dalloc(h, &s.group_mask, G) && dalloc(h, &s.group_w, G * 4) && dalloc(h, &s.act_dec, G * 4 * I) &&
            dalloc(h, &s.y_dec, G * 4 * D) && dalloc(h, &s.dec_counters, (size_t)moe::decode_counter_count(d)) &&
            dalloc(h, &s.dtc_acc_gu, G * 2 * 4 * I) && dalloc(h, &s.dtc_acc_y, 4 * D) &&
            dalloc(h, &s.dtc_act2, G * 16 * I) &&
            dalloc(h, &h->host_in, R * hcd) &&
            dalloc(h, &h->host_out, R * hcd) && dalloc(h, &h->host_tok, R);
  const bool prefill = R > (size_t)moe::kDecodeRows;
  s.max_positions = (int)(R * K + R);
  const size_t P = prefill ? s.max_positions : 0;
  s.max_tiles_gu = (int)((P / 128 + E + 1) * (I / 128));
  s.max_tiles_dn = (int)((P / 128 + E + 1) * ((D + 255) / 256));
  if (ok && prefill)
    ok = dalloc(h, &s.counts, E) && dalloc(h, &s.offsets, E + 2) && dalloc(h, &s.cursor, E + 1) &&
         dalloc(h, &s.router_part, (size_t)moe::splitgemm_splits((int)D) * R * E) &&
         dalloc(h, &s.tiles_gu, (size_t)s.max_tiles_gu) && dalloc(h, &s.tiles_dn, (size_t)s.max_tiles_dn) &&
         dalloc(h, &s.n_tiles, 8) && dalloc(h, &s.list, P) && dalloc(h, &s.list_w, P) &&
         dalloc(h, &s.x2, 2 * P * D) && dalloc(h, &s.act2, 2 * P * I) && dalloc(h, &s.ffn_acc, R * D) &&
         dalloc(h, &s.mix_tc_part, (size_t)moe::mix_tc_part_floats((int)R, (int)hcd));
  if (!ok) {
    free_all(h);
    delete h;
    return fail(nullptr, MOE_FFN_ERR_NO_MEMORY, "device allocation of the scratch failed");
  }
  cudaMemset(s.status, 0, sizeof(int));
  cudaMemset(s.dec_counters, 0, (size_t)moe::decode_counter_count(d) * sizeof(unsigned));
  cudaMemset(s.dec_part, 0xFF, (size_t)moe::kDecodeRows * E * 2 * sizeof(float));  // "not written yet"
  cudaMemset(s.dtc_acc_gu, 0, G * 2 * 4 * I * sizeof(double));
  cudaMemset(s.dtc_acc_y, 0, 4 * D * sizeof(double));
  cudaMemset(s.dtc_act2, 0, G * 16 * I * sizeof(uint16_t));
  if (!make_tmap_bf16(&s.tm_dtc_act2, s.dtc_act2, I, G * 16, 16)) {
    free_all(h);
    delete h;
    return fail(nullptr, MOE_FFN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the decode act planes");
  }
  cudaMemset(s.tickets, 0, (R / 4 + 2) * sizeof(unsigned));
  if (prefill) {
    cudaMemset(s.counts, 0, E * sizeof(int));
    CUtensorMap maps[16];
    bool enc = make_tmap_f32(&h->tm_ffn_norm, s.ffn_norm, D, R);
    for (int i = 0; i < 8 && enc; ++i)
      enc = make_tmap_bf16(&maps[i], s.x2, D, 2 * P, 16u * (i + 1)) &&
            make_tmap_bf16(&maps[8 + i], s.act2, I, 2 * P, 16u * (i + 1));
    if (enc) enc = dalloc(h, &h->tm_b, 16) && cudaMemcpy(h->tm_b, maps, sizeof maps, cudaMemcpyHostToDevice) == cudaSuccess;
    if (!enc) {
      free_all(h);
      delete h;
      return fail(nullptr, MOE_FFN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the activation buffers");
    }
  }
  if (moe::gemm_configure() != cudaSuccess || moe::decode_configure(d.hidden) != cudaSuccess ||
      moe::decode_tc_configure() != cudaSuccess || moe::splitgemm_configure() != cudaSuccess) {
    free_all(h);
    delete h;
    return fail(nullptr, MOE_FFN_ERR_CUDA, "kernel attribute setup failed");
  }
  for (int mx = 0; mx < 2; ++mx)
    for (int r = 1; r <= moe::kDecodeRows; ++r) {
      int &n = mx ? s.decode_ctas_mx[r] : s.decode_ctas_by_rows[r];
      // the tensor-core decode (one CTA per SM) where its K splits fit the grid; the CUDA-core
      // kernel's count is kept for MXFP8 layers, which use it at one to three rows
      const int tc = moe::decode_tc_resident_ctas(r, h->num_sms, mx != 0);
      bool &fits = mx ? s.dtc_mx : s.dtc;
      fits = tc > 0 && moe::decode_tc_fits(d, tc);
      const int cc = moe::decode_resident_ctas(d.hidden, r, h->num_sms, mx != 0);
      n = fits ? tc : cc;
      if (mx) s.decode_ctas_mx_cc[r] = cc;
      if (n <= 0 || cc <= 0) {
        free_all(h);
        delete h;
        return fail(nullptr, MOE_FFN_ERR_CUDA, "the decode kernel does not fit on an SM");
      }
      // its prelude roles are claimed by the first CTAs to arrive; at least one CTA must be left
      if ((n < cc ? n : cc) <= moe::decode_mix_ctas(d.hc, d.hidden) + moe::decode_router_ctas(d.experts)) {
        free_all(h);
        delete h;
        return fail(nullptr, MOE_FFN_ERR_CUDA, "too few co-resident CTAs (%d) for the decode kernel's roles", n);
      }
    }
  s.decode_ctas_by_rows[0] = s.decode_ctas_mx[0] = s.decode_ctas_mx_cc[0] = 0;
  h->layers.resize(cfg->n_layers);
  h->attn.resize(cfg->n_layers);
  for (LayerDev &A : h->attn) std::memset(&A, 0, sizeof A);
  for (int l = 0; l < cfg->n_layers; ++l) {
    LayerDev &L = h->layers[l];
    std::memset(&L, 0, sizeof L);
    L.has_weights = has[l];
    L.has_experts = has_exps[l];
    if (!has[l]) continue;
    const moe_ffn_layer_weights &w = layers[l];
    L.hc_fn = w.hc_fn;
    L.hc_base = w.hc_base;
    L.hc_scale = w.hc_scale;
    L.ffn_norm = w.ffn_norm;
    L.gate = w.gate;
    L.exp_probs_b = w.exp_probs_b;
    L.tid2eid = w.tid2eid;
    L.gate_exps = w.gate_exps;
    L.up_exps = w.up_exps;
    L.down_exps = w.down_exps;
    L.gate_sh = w.gate_sh;
    L.up_sh = w.up_sh;
    L.down_sh = w.down_sh;
    // the tensor-core paths read the caller's bf16 expert matrices through tensor maps (both
    // paths); the rows > 4 path also hc_fn in boxes of 32 rows (the mix's MMA width; rows past
    // (2+hc)*hc read as zeros) and the router in boxes of 256
    if ((L.has_experts && !expert_tmaps(h, L, w.gate_exps, w.up_exps, w.down_exps, w.gate_sh, w.up_sh, w.down_sh)) ||
        (prefill && (!make_tmap_bf16(&L.tm_hcfn, w.hc_fn, hcd, M, 32) ||
                     !make_tmap_bf16(&L.tm_router, w.gate, D, E, 256)))) {
      free_all(h);
      delete h;
      return fail(nullptr, MOE_FFN_ERR_CUDA, "cuTensorMapEncodeTiled failed for layer %d", l);
    }
  }
  const cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    const std::string msg = cudaGetErrorString(e);
    free_all(h);
    delete h;
    return fail(nullptr, MOE_FFN_ERR_CUDA, "init: %s", msg.c_str());
  }
  *out = h;
  return MOE_FFN_OK;
}

// The forward's host-side checks (the guards of forward_ffn_rows, plus pointers and alignment).
static int check_forward(moe_ffn_handle *h, const float *state, const int32_t *token_ids, int32_t rows, int32_t layer,
                         const float *out_state) {
  const moe_ffn_config &c = h->cfg;
  if (layer < 0 || layer >= c.n_layers)
    return fail(h, MOE_FFN_ERR_LAYER_RANGE, "FFN layer index %d is outside 0..%d", layer, c.n_layers);
  if (rows == 0) return fail(h, MOE_FFN_ERR_ROWS_ZERO, "the FFN requires at least one token row");
  if (rows < 0 || rows > c.max_rows)
    return fail(h, MOE_FFN_ERR_ROWS_RANGE, "rows %d outside 1..max_rows (%d)", rows, c.max_rows);
  if (!state || !out_state) return fail(h, MOE_FFN_ERR_NULL_PTR, "state or out_state is NULL");
  if (!h->layers[layer].has_weights) return fail(h, MOE_FFN_ERR_NO_WEIGHTS, "layer %d has no weights", layer);
  if (!h->layers[layer].has_experts)
    return fail(h, MOE_FFN_ERR_NO_WEIGHTS, "layer %d has no expert weights (bf16 at init, or MXFP8)", layer);
  if (layer < c.hash_layer_count && !token_ids)
    return fail(h, MOE_FFN_ERR_NULL_PTR, "hash layer %d needs token_ids", layer);
  if (!aligned16(state) || !aligned16(out_state))
    return fail(h, MOE_FFN_ERR_ALIGNMENT, "state and out_state must be 16-byte aligned");
  const size_t bytes = (size_t)rows * c.hc * c.hidden * sizeof(float);
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(state), b0 = reinterpret_cast<uintptr_t>(out_state);
  if (a0 < b0 + bytes && b0 < a0 + bytes) return fail(h, MOE_FFN_ERR_ALIAS, "out_state overlaps state");
  return MOE_FFN_OK;
}

// Enqueues one layer's block (arguments already checked).
static int enqueue_forward(moe_ffn_handle *h, const float *state, const int32_t *token_ids, int32_t rows,
                           int32_t layer, float *out_state, cudaStream_t st, moe::StageTimer *tm) {
  const moe_ffn_config &c = h->cfg;
  const LayerDev &L = h->layers[layer];
  const bool hash = layer < c.hash_layer_count;
  if (rows <= moe::kDecodeRows) {
    moe::launch_decode(h->dims, h->s, L, state, token_ids, rows, hash, out_state, st, tm, h->dbg);
  } else {
    // the state changes with every call: its tensor map is encoded here (host only, no GPU work)
    CUtensorMap tm_state;
    if (!make_tmap_f32(&tm_state, state, (uint64_t)c.hc * c.hidden, (uint64_t)rows))
      return fail(h, MOE_FFN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the state");
    moe::launch_prefill_mix(h->dims, h->s, L, state, tm_state, rows, h->num_sms, st, tm);
    moe::launch_prefill_router(h->dims, h->s, L, state, token_ids, h->tm_ffn_norm, rows, hash, h->num_sms, st, tm);
    moe::launch_dispatch(h->dims, h->s, rows, st, tm);
    moe::launch_grouped_gemms(h->dims, h->s, L, h->tm_b, h->tm_b + 8, h->num_sms, st, tm, h->dbg);
    moe::launch_hc_post(h->dims, h->s.ffn_acc, state, h->s.post, h->s.comb, rows, out_state, st);
    moe::stage(tm, "post", st);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(h, MOE_FFN_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
  return MOE_FFN_OK;
}

extern "C" int moe_ffn_forward(moe_ffn_handle *h, const float *state, const int32_t *token_ids, int32_t rows,
                               int32_t layer, float *out_state, void *stream) {
  if (!h) return fail(nullptr, MOE_FFN_ERR_NULL_PTR, "handle is NULL");
  int rc = check_forward(h, state, token_ids, rows, layer, out_state);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  moe::StageTimer *tm = h->timer.on ? &h->timer : nullptr;
  if (tm) tm->begin(st);
  rc = enqueue_forward(h, state, token_ids, rows, layer, out_state, st, tm);
  if (rc) return rc;
  h->last_stream = st;
  h->last_rows = rows;
  return MOE_FFN_OK;
}

extern "C" int moe_ffn_forward_layers(moe_ffn_handle *h, const float *state, const int32_t *token_ids, int32_t rows,
                                      int32_t first_layer, int32_t n_layers, float *out_state, void *stream) {
  if (!h) return fail(nullptr, MOE_FFN_ERR_NULL_PTR, "handle is NULL");
  const moe_ffn_config &c = h->cfg;
  if (n_layers < 1 || first_layer < 0 || first_layer > c.n_layers - n_layers)
    return fail(h, MOE_FFN_ERR_LAYER_RANGE, "layers %d..%d are outside 0..%d", first_layer, first_layer + n_layers - 1,
                c.n_layers - 1);
  for (int l = first_layer; l < first_layer + n_layers; ++l) {
    const int rc = check_forward(h, state, token_ids, rows, l, out_state);
    if (rc) return rc;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (n_layers == 1) return moe_ffn_forward(h, state, token_ids, rows, first_layer, out_state, stream);
  if (!h->chain_state && !dalloc(h, &h->chain_state, (size_t)c.max_rows * c.hc * c.hidden))
    return fail(h, MOE_FFN_ERR_NO_MEMORY, "device allocation of the chain's intermediate state failed");
  size_t k = 0;
  for (; k < h->chains.size(); ++k) {
    const moe_ffn_handle::Chain &ch = h->chains[k];
    if (ch.state == state && ch.tok == token_ids && ch.out == out_state && ch.rows == rows &&
        ch.first == first_layer && ch.n == n_layers)
      break;
  }
  if (k == h->chains.size()) {
    // capture the chain on the handle's own stream: layer i writes out_state when n_layers - 1 - i
    // is even, else the intermediate buffer, so the last layer lands in out_state and no layer
    // reads the buffer it writes
    if (!h->capture && cudaStreamCreateWithFlags(&h->capture, cudaStreamNonBlocking) != cudaSuccess)
      return fail(h, MOE_FFN_ERR_CUDA, "cudaStreamCreate failed");
    cudaError_t e = cudaStreamBeginCapture(h->capture, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return fail(h, MOE_FFN_ERR_CUDA, "begin capture: %s", cudaGetErrorString(e));
    int rc = MOE_FFN_OK;
    const float *in = state;
    for (int i = 0; i < n_layers && rc == MOE_FFN_OK; ++i) {
      float *o = (n_layers - 1 - i) % 2 == 0 ? out_state : h->chain_state;
      rc = enqueue_forward(h, in, token_ids, rows, first_layer + i, o, h->capture, nullptr);
      in = o;
    }
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(h->capture, &g);
    if (rc != MOE_FFN_OK || e != cudaSuccess) {
      if (g) cudaGraphDestroy(g);
      return rc != MOE_FFN_OK ? rc : fail(h, MOE_FFN_ERR_CUDA, "end capture: %s", cudaGetErrorString(e));
    }
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return fail(h, MOE_FFN_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(e));
    if (h->chains.size() == kMaxChains) {  // the least recently used goes (freed once it has run)
      cudaGraphExecDestroy(h->chains.front().exec);
      h->chains.erase(h->chains.begin());
    }
    h->chains.push_back({state, token_ids, out_state, rows, first_layer, n_layers, exec});
    k = h->chains.size() - 1;
  } else if (k + 1 != h->chains.size()) {
    const moe_ffn_handle::Chain ch = h->chains[k];
    h->chains.erase(h->chains.begin() + (long)k);
    h->chains.push_back(ch);
    k = h->chains.size() - 1;
  }
  const cudaError_t e = cudaGraphLaunch(h->chains[k].exec, st);
  if (e != cudaSuccess) return fail(h, MOE_FFN_ERR_CUDA, "graph launch: %s", cudaGetErrorString(e));
  h->last_stream = st;
  h->last_rows = rows;
  return MOE_FFN_OK;
}

extern "C" int moe_ffn_forward_host(moe_ffn_handle *h, const float *state, const int32_t *token_ids, int32_t rows,
                                    int32_t layer, float *out_state, void *stream) {
  if (!h) return fail(nullptr, MOE_FFN_ERR_NULL_PTR, "handle is NULL");
  if (rows <= 0 || rows > h->cfg.max_rows || !state || !out_state)  // the same checks, on the staging buffers
    return moe_ffn_forward(h, state, token_ids, rows, layer, out_state, stream);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)rows * h->cfg.hc * h->cfg.hidden * sizeof(float);
  cudaError_t e = cudaMemcpyAsync(h->host_in, state, bytes, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess && token_ids)
    e = cudaMemcpyAsync(h->host_tok, token_ids, (size_t)rows * sizeof(int32_t), cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return fail(h, MOE_FFN_ERR_CUDA, "host-to-device copy: %s", cudaGetErrorString(e));
  const int rc = moe_ffn_forward(h, h->host_in, token_ids ? h->host_tok : nullptr, rows, layer, h->host_out, stream);
  if (rc != MOE_FFN_OK) return rc;
  e = cudaMemcpyAsync(out_state, h->host_out, bytes, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail(h, MOE_FFN_ERR_CUDA, "device-to-host copy: %s", cudaGetErrorString(e));
  return MOE_FFN_OK;
}

static bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return a && b && x < y + nb && y < x + na;
}

static int check_rows(moe_ffn_handle *h, int32_t rows) {
  if (rows == 0) return fail(h, MOE_FFN_ERR_ROWS_ZERO, "at least one token row is required");
  if (rows < 0 || rows > h->cfg.max_rows)
    return fail(h, MOE_FFN_ERR_ROWS_RANGE, "rows %d outside 1..max_rows (%d)", rows, h->cfg.max_rows);
  return MOE_FFN_OK;
}

extern "C" int moe_ffn_set_attn_hc(moe_ffn_handle *h, int32_t layer, const moe_ffn_hc_weights *w) {
  if (!h) return fail(nullptr, MOE_FFN_ERR_NULL_PTR, "handle is NULL");
  const moe_ffn_config &c = h->cfg;
  if (layer < 0 || layer >= c.n_layers)
    return fail(h, MOE_FFN_ERR_LAYER_RANGE, "layer index %d is outside 0..%d", layer, c.n_layers);
  if (!w || !w->hc_fn || !w->hc_base || !w->hc_scale || !w->norm)
    return fail(h, MOE_FFN_ERR_NULL_PTR, "attention HC weights of layer %d: a pointer is NULL", layer);
  if (!aligned16(w->hc_fn) || !aligned16(w->hc_base) || !aligned16(w->hc_scale) || !aligned16(w->norm))
    return fail(h, MOE_FFN_ERR_ALIGNMENT, "attention HC weights of layer %d must be 16-byte aligned", layer);
  LayerDev &A = h->attn[layer];
  A.hc_fn = w->hc_fn;
  A.hc_base = w->hc_base;
  A.hc_scale = w->hc_scale;
  A.ffn_norm = w->norm;
  if (c.max_rows > moe::kDecodeRows &&
      !make_tmap_bf16(&A.tm_hcfn, w->hc_fn, (uint64_t)c.hc * c.hidden, (uint64_t)h->dims.mix(), 32)) {
    A.has_weights = false;
    return fail(h, MOE_FFN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the attention hc_fn of layer %d", layer);
  }
  const cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    A.has_weights = false;
    return fail(h, MOE_FFN_ERR_CUDA, "set_attn_hc: %s", cudaGetErrorString(e));
  }
  A.has_weights = true;
  return MOE_FFN_OK;
}

extern "C" int moe_ffn_hc_pre(moe_ffn_handle *h, int32_t layer, int32_t sublayer, const float *state, int32_t rows,
                              float *x_norm, float *pre, float *post, float *comb, void *stream) {
  if (!h) return fail(nullptr, MOE_FFN_ERR_NULL_PTR, "handle is NULL");
  const moe_ffn_config &c = h->cfg;
  if (layer < 0 || layer >= c.n_layers)
    return fail(h, MOE_FFN_ERR_LAYER_RANGE, "layer index %d is outside 0..%d", layer, c.n_layers);
  if (sublayer != MOE_FFN_SUBLAYER_ATTN && sublayer != MOE_FFN_SUBLAYER_FFN)
    return fail(h, MOE_FFN_ERR_BAD_CONFIG, "unknown sublayer %d", sublayer);
  int rc = check_rows(h, rows);
  if (rc) return rc;
  if (!state || !x_norm || !post || !comb) return fail(h, MOE_FFN_ERR_NULL_PTR, "state, x_norm, post or comb is NULL");
  if (!aligned16(state) || !aligned16(x_norm))
    return fail(h, MOE_FFN_ERR_ALIGNMENT, "state and x_norm must be 16-byte aligned");
  const LayerDev &L = sublayer == MOE_FFN_SUBLAYER_ATTN ? h->attn[layer] : h->layers[layer];
  if (!L.has_weights)
    return fail(h, MOE_FFN_ERR_NO_WEIGHTS, "layer %d has no %s HC weights", layer,
                sublayer == MOE_FFN_SUBLAYER_ATTN ? "attention" : "FFN");
  const size_t R = rows, HC = c.hc, D = c.hidden, sb = R * HC * D * 4;
  if (overlaps(state, sb, x_norm, R * D * 4) || overlaps(state, sb, pre, R * HC * 4) ||
      overlaps(state, sb, post, R * HC * 4) || overlaps(state, sb, comb, R * HC * HC * 4))
    return fail(h, MOE_FFN_ERR_ALIAS, "an output overlaps state");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUtensorMap tm_state;
  if (rows > moe::kDecodeRows && !make_tmap_f32(&tm_state, state, (uint64_t)HC * D, (uint64_t)rows))
    return fail(h, MOE_FFN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the state");
  moe::launch_hc_pre(h->dims, h->s, L, state, &tm_state, rows, h->num_sms, x_norm, pre ? pre : h->s.pre, post, comb,
                     st);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(h, MOE_FFN_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
  h->last_stream = st;
  return MOE_FFN_OK;
}

extern "C" int moe_ffn_hc_post(moe_ffn_handle *h, const float *f, const float *state, const float *post,
                               const float *comb, int32_t rows, float *out_state, void *stream) {
  if (!h) return fail(nullptr, MOE_FFN_ERR_NULL_PTR, "handle is NULL");
  int rc = check_rows(h, rows);
  if (rc) return rc;
  if (!f || !state || !post || !comb || !out_state)
    return fail(h, MOE_FFN_ERR_NULL_PTR, "f, state, post, comb or out_state is NULL");
  if (!aligned16(f) || !aligned16(state) || !aligned16(out_state))
    return fail(h, MOE_FFN_ERR_ALIGNMENT, "f, state and out_state must be 16-byte aligned");
  const size_t R = rows, HC = h->cfg.hc, D = h->cfg.hidden, sb = R * HC * D * 4;
  if (overlaps(out_state, sb, state, sb) || overlaps(out_state, sb, f, R * D * 4) ||
      overlaps(out_state, sb, post, R * HC * 4) || overlaps(out_state, sb, comb, R * HC * HC * 4))
    return fail(h, MOE_FFN_ERR_ALIAS, "out_state overlaps an input");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  moe::launch_hc_post(h->dims, f, state, post, comb, rows, out_state, st);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(h, MOE_FFN_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
  h->last_stream = st;
  return MOE_FFN_OK;
}

extern "C" int moe_ffn_set_mxfp8_experts(moe_ffn_handle *h, int32_t layer, const moe_ffn_mxfp8_experts *w) {
  if (!h) return fail(nullptr, MOE_FFN_ERR_NULL_PTR, "handle is NULL");
  const moe_ffn_config &c = h->cfg;
  if (layer < 0 || layer >= c.n_layers)
    return fail(h, MOE_FFN_ERR_LAYER_RANGE, "layer index %d is outside 0..%d", layer, c.n_layers);
  LayerDev &L = h->layers[layer];
  if (!L.has_weights) return fail(h, MOE_FFN_ERR_NO_WEIGHTS, "layer %d has no weights (moe_ffn_init)", layer);
  if (!w) return fail(h, MOE_FFN_ERR_NULL_PTR, "MXFP8 experts of layer %d: NULL", layer);
  const uint8_t *p[] = {w->gate_exps, w->gate_exps_scale, w->up_exps, w->up_exps_scale, w->down_exps,
                        w->down_exps_scale, w->gate_sh, w->gate_sh_scale, w->up_sh, w->up_sh_scale,
                        w->down_sh, w->down_sh_scale};
  for (const uint8_t *q : p) {
    if (!q) return fail(h, MOE_FFN_ERR_NULL_PTR, "MXFP8 experts of layer %d: a pointer is NULL", layer);
    if (!aligned16(q)) return fail(h, MOE_FFN_ERR_ALIGNMENT, "MXFP8 experts of layer %d must be 16-byte aligned", layer);
  }
  L.gate_q = w->gate_exps;
  L.gate_s = w->gate_exps_scale;
  L.up_q = w->up_exps;
  L.up_s = w->up_exps_scale;
  L.down_q = w->down_exps;
  L.down_s = w->down_exps_scale;
  L.gate_sh_q = w->gate_sh;
  L.gate_sh_s = w->gate_sh_scale;
  L.up_sh_q = w->up_sh;
  L.up_sh_s = w->up_sh_scale;
  L.down_sh_q = w->down_sh;
  L.down_sh_s = w->down_sh_scale;
  {
    // the tensor-core decode streams the weights as f16 (code x 2^(S - 127 + c)); that is exact when
    // no code or scale is NaN and every scale lies within 22 binades of the largest
    unsigned *scan = nullptr;  // [0] NaN code found, [1] smallest scale, [2] largest scale
    unsigned host[3] = {0u, 255u, 0u};
    const size_t n_exp = (size_t)c.experts * c.inter * c.hidden, n_sh = (size_t)c.inter * c.hidden;
    cudaError_t e = cudaMalloc(&scan, sizeof host);
    if (e == cudaSuccess) e = cudaMemcpy(scan, host, sizeof host, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) {
      const uint8_t *q[6] = {L.gate_q, L.up_q, L.down_q, L.gate_sh_q, L.up_sh_q, L.down_sh_q};
      const uint8_t *sc[6] = {L.gate_s, L.up_s, L.down_s, L.gate_sh_s, L.up_sh_s, L.down_sh_s};
      for (int i = 0; i < 6; ++i) {
        const size_t n = i < 3 ? n_exp : n_sh;
        moe::launch_e4m3_nan_scan(q[i], n, reinterpret_cast<int *>(scan), 0);
        moe::launch_e8m0_range(sc[i], n / 32, scan + 1, 0);
      }
      e = cudaMemcpy(host, scan, sizeof host, cudaMemcpyDeviceToHost);
    }
    if (scan) cudaFree(scan);
    if (e != cudaSuccess) return fail(h, MOE_FFN_ERR_CUDA, "set_mxfp8_experts: %s", cudaGetErrorString(e));
    L.mx_tc = host[0] == 0u && host[2] != 255u && host[2] - host[1] <= 22u;
    L.mx_c = 134 - (int)host[2];
  }
  {
    const uint64_t E = h->dims.experts, I = h->dims.inter, D = h->dims.hidden;
    if (!make_tmap_u8(&L.tm_gate_q, L.gate_q, D, E * I) || !make_tmap_u8(&L.tm_up_q, L.up_q, D, E * I) ||
        !make_tmap_u8(&L.tm_down_q, L.down_q, I, E * D) || !make_tmap_u8(&L.tm_gate_sh_q, L.gate_sh_q, D, I) ||
        !make_tmap_u8(&L.tm_up_sh_q, L.up_sh_q, D, I) || !make_tmap_u8(&L.tm_down_sh_q, L.down_sh_q, I, D))
      return fail(h, MOE_FFN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the MXFP8 codes of layer %d", layer);
  }
  if (c.max_rows > moe::kDecodeRows) {  // the tensor-core path reads an exact bf16 expansion
    const size_t E = c.experts, I = c.inter, D = c.hidden, n_exp = E * I * D, n_sh = I * D;
    if (!L.mx_bf16 && !dalloc(h, &L.mx_bf16, 3 * (n_exp + n_sh)))
      return fail(h, MOE_FFN_ERR_NO_MEMORY, "device allocation of the bf16 expansion of layer %d failed", layer);
    uint16_t *g = L.mx_bf16, *u = g + n_exp, *dn = u + n_exp, *gs = dn + n_exp, *us = gs + n_sh, *ds = us + n_sh;
    moe::launch_mxfp8_to_bf16(L.gate_q, L.gate_s, g, n_exp, 0);
    moe::launch_mxfp8_to_bf16(L.up_q, L.up_s, u, n_exp, 0);
    moe::launch_mxfp8_to_bf16(L.down_q, L.down_s, dn, n_exp, 0);
    moe::launch_mxfp8_to_bf16(L.gate_sh_q, L.gate_sh_s, gs, n_sh, 0);
    moe::launch_mxfp8_to_bf16(L.up_sh_q, L.up_sh_s, us, n_sh, 0);
    moe::launch_mxfp8_to_bf16(L.down_sh_q, L.down_sh_s, ds, n_sh, 0);
    if (!expert_tmaps(h, L, g, u, dn, gs, us, ds))
      return fail(h, MOE_FFN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the MXFP8 experts of layer %d", layer);
  }
  const cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(h, MOE_FFN_ERR_CUDA, "set_mxfp8_experts: %s", cudaGetErrorString(e));
  L.mx = true;
  L.has_experts = true;
  return MOE_FFN_OK;
}

extern "C" int moe_ffn_status(moe_ffn_handle *h) {
  if (!h) return fail(nullptr, MOE_FFN_ERR_NULL_PTR, "handle is NULL");
  int v = 0;
  cudaError_t e = cudaStreamSynchronize(h->last_stream);
  if (e == cudaSuccess) e = cudaMemcpy(&v, h->s.status, sizeof v, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(h->s.status, 0, sizeof v);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(h, MOE_FFN_ERR_CUDA, "status: %s", cudaGetErrorString(e));
  return v;
}

extern "C" int moe_ffn_debug_copy(moe_ffn_handle *h, int32_t which, void *host_dst, size_t bytes) {
  if (!h || !host_dst) return fail(h, MOE_FFN_ERR_NULL_PTR, "handle or destination is NULL");
  const size_t R = h->last_rows, D = h->dims.hidden, HC = h->dims.hc, E = h->dims.experts, K = h->dims.top_k;
  const void *src = nullptr;
  size_t n = 0;
  switch (which) {
    case 0: src = h->s.pre; n = R * HC * 4; break;
    case 1: src = h->s.post; n = R * HC * 4; break;
    case 2: src = h->s.comb; n = R * HC * HC * 4; break;
    case 3: src = h->s.ffn_norm; n = R * D * 4; break;
    case 4: src = h->s.logits; n = R * E * 4; break;
    case 5: src = h->s.idx; n = R * K * 4; break;
    case 6: src = h->s.rw; n = R * K * 4; break;
    case 7: src = h->s.safe; n = R * K * 4; break;
    case 8: src = h->s.ffn_out; n = R * D * 4; break;
    default: return fail(h, MOE_FFN_ERR_BAD_CONFIG, "unknown debug buffer %d", which);
  }
  if (bytes != n) return fail(h, MOE_FFN_ERR_BAD_CONFIG, "debug buffer %d holds %zu bytes, not %zu", which, n, bytes);
  cudaError_t e = cudaStreamSynchronize(h->last_stream);
  if (which == 8 && R > (size_t)moe::kDecodeRows) {
    // the rows > 4 path accumulates the FFN output in f64; it is rounded to f32 as hc_post reads it
    std::vector<double> tmp(R * D);
    if (e == cudaSuccess) e = cudaMemcpy(tmp.data(), h->s.ffn_acc, R * D * sizeof(double), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess)
      for (size_t i = 0; i < R * D; ++i) static_cast<float *>(host_dst)[i] = (float)tmp[i];
  } else if (e == cudaSuccess) {
    e = cudaMemcpy(host_dst, src, n, cudaMemcpyDeviceToHost);
  }
  if (e != cudaSuccess) return fail(h, MOE_FFN_ERR_CUDA, "debug copy: %s", cudaGetErrorString(e));
  return MOE_FFN_OK;
}

extern "C" int moe_ffn_set_stage_timing(moe_ffn_handle *h, int32_t enable) {
  if (!h) return fail(nullptr, MOE_FFN_ERR_NULL_PTR, "handle is NULL");
  moe::StageTimer &t = h->timer;
  if (enable && !t.created) {
    for (int i = 0; i <= moe::StageTimer::kMax; ++i)
      if (cudaEventCreate(&t.ev[i]) != cudaSuccess) return fail(h, MOE_FFN_ERR_CUDA, "cudaEventCreate failed");
    t.created = true;
  }
  t.on = enable != 0;
  t.n = 0;
  return MOE_FFN_OK;
}

extern "C" int moe_ffn_stage_times(moe_ffn_handle *h, float *ms, const char **names, int32_t max_stages) {
  if (!h || !ms) return fail(h, MOE_FFN_ERR_NULL_PTR, "handle or output is NULL");
  moe::StageTimer &t = h->timer;
  if (!t.created || t.n == 0) return 0;
  if (cudaEventSynchronize(t.ev[t.n]) != cudaSuccess) return fail(h, MOE_FFN_ERR_CUDA, "event wait failed");
  const int n = t.n < max_stages ? t.n : max_stages;
  for (int i = 0; i < n; ++i) {
    if (cudaEventElapsedTime(&ms[i], t.ev[i], t.ev[i + 1]) != cudaSuccess)
      return fail(h, MOE_FFN_ERR_CUDA, "cudaEventElapsedTime failed");
    if (names) names[i] = t.name[i];
  }
  return n;
}

extern "C" int moe_ffn_set_fault_injection(moe_ffn_handle *h, int32_t which, uint32_t wait_limit_us) {
  if (!h) return fail(nullptr, MOE_FFN_ERR_NULL_PTR, "handle is NULL");
  if (which < MOE_FFN_INJECT_NONE || which > MOE_FFN_INJECT_GEMM_WAIT)
    return fail(h, MOE_FFN_ERR_BAD_CONFIG, "unknown fault injection %d", which);
  h->dbg.inject = which;
  h->dbg.wait_ns = (uint64_t)wait_limit_us * 1000ull;
  return MOE_FFN_OK;
}

extern "C" const char *moe_ffn_last_error(const moe_ffn_handle *h) { return h ? h->err.c_str() : g_init_err.c_str(); }

extern "C" void moe_ffn_destroy(moe_ffn_handle *h) {
  if (!h) return;
  cudaDeviceSynchronize();
  if (h->timer.created)
    for (int i = 0; i <= moe::StageTimer::kMax; ++i) cudaEventDestroy(h->timer.ev[i]);
  for (const moe_ffn_handle::Chain &ch : h->chains) cudaGraphExecDestroy(ch.exec);
  if (h->capture) cudaStreamDestroy(h->capture);
  free_all(h);
  delete h;
}
