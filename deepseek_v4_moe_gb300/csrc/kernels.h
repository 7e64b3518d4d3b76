// Host-side launchers of the MoE-FFN kernels, shared between the translation units.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Launch with programmatic stream serialisation: the kernel may start while the previous kernel on
// the stream finishes; it must call griddepcontrol.wait before reading that kernel's results.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Routing source and outputs of one layer (device pointers): score layers use `bias`
// (exp_probs_b), hash layers `tid2eid` and the token ids.
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

struct Dims {
  int hidden, hc, experts, top_k, inter, vocab, iters;
  float eps;
  int mix() const { return (2 + hc) * hc; }
};

// Scratch owned by the handle, sized for max_rows at init.
struct Scratch {
  int *status;            // [1] device status bits
  float *mix_partial;     // [max_rows, mix_chunks, mix+1]
  unsigned *tickets;      // [max(max_rows/4+1, 1) + 1] zero between launches
  float *mixes, *pre, *post, *comb;  // [rows, mix] [rows, hc] [rows, hc] [rows, hc, hc]
  float *ffn_input, *ffn_norm;       // [rows, hidden]
  float *row_rs;          // [rows] rsqrt(mean(ffn_input^2) + eps) (decode)
  float *dec_part;        // decode: [4, experts] (selection score, logit) pairs the router CTAs write
  float *logits;          // [rows, experts]
  float *router_part;     // [splits, rows, experts] split-K partial logits (rows > 4)
  int *idx;               // [rows, top_k]
  float *rw;              // [rows, top_k]
  unsigned *safe;         // [rows, top_k]
  float *ffn_out;         // [rows, hidden] (decode path)
  double *ffn_acc;        // [rows, hidden] the rows > 4 path's FFN output, accumulated by the down GEMM
  // decode path
  int *ngroups, *group_e, *group_mask;  // groups of (expert, rows using it); shared expert last
  float *group_w;         // [groups, 4]
  float *act_dec;         // [groups, 4, inter]
  float *y_dec;           // [groups, 4, hidden]
  unsigned *dec_counters; // the decode kernel's tickets and completion counters (zero between launches)
  int decode_ctas_by_rows[5];  // co-resident CTAs of the persistent decode kernel, per row count
  int decode_ctas_mx[5];       // the same for its MXFP8-expert instances
  int decode_ctas_mx_cc[5];    // the CUDA-core kernel's MXFP8 instances (one to three rows, and layers
                               // whose codes the tensor-core instance cannot widen exactly)
  // decode on the tensor cores
  double *dtc_acc_gu;          // [groups, 2, 4, inter] gate and up partial sums (zero between launches)
  double *dtc_acc_y;           // [4, hidden] the FFN output (zero between launches)
  uint16_t *dtc_act2;          // [groups, 16, inter]: act as bf16 hi (rows 0-3) and lo (rows 4-7) planes,
                               // or (MXFP8 experts) as three f16 planes (rows 0-3, 4-7, 8-11)
  CUtensorMap tm_dtc_act2;     // over dtc_act2, boxes of 64 x 16 rows
  bool dtc;                    // the tensor-core decode kernel fits this configuration (bf16 experts)
  bool dtc_mx;                 // ... and its MXFP8 instance
  // rows > 4 path
  int *counts;            // [experts] routed slots per expert (zero between launches)
  int *offsets;           // [experts + 2]
  int *cursor;            // [experts + 1]
  int4 *tiles_gu, *tiles_dn;  // (group, m-block, n-block, valid columns)
  int *n_tiles;           // [8]: gate/up tiles, down tiles, the heavy ones of each (listed first),
                          // then claim counters: gate/up heavy and light, down heavy and light
  int2 *list;             // [positions] (row, slot) in expert-sorted order; slot top_k = shared expert
  float *list_w;          // [positions] route weight of that slot (1 for the shared expert)
  uint16_t *x2;           // [2 * max_positions, hidden] bf16: ffn_norm rows in expert-sorted order,
                          // hi plane (rows 0..P-1) then lo plane (rows P..2P-1)
  uint16_t *act2;         // [2 * max_positions, inter] bf16: SwiGLU output in the same order, hi then lo
  float *mix_tc_part;     // [splits, rows, 32] mix partials, then [splits, rows] sums of squares
  int max_rows, mix_chunks, router_chunks, max_positions, max_tiles_gu, max_tiles_dn;
};

// Optional per-kernel timing: an event after each kernel launch of a forward.
struct StageTimer {
  static constexpr int kMax = 16;
  cudaEvent_t ev[kMax + 1];
  const char *name[kMax];
  int n = 0;
  bool on = false, created = false;
  void begin(cudaStream_t st) {
    n = 0;
    cudaEventRecord(ev[0], st);
  }
  void mark(const char *nm, cudaStream_t st) {
    if (n < kMax) {
      name[n] = nm;
      cudaEventRecord(ev[n + 1], st);
      ++n;
    }
  }
};

// Test hooks (moe_ffn_set_fault_injection): the bound of every in-kernel wait, and which kernel, if
// any, waits on a barrier or counter that nothing completes.
struct DebugOpts {
  uint64_t wait_ns = 0;  // 0: the kernels' defaults
  int inject = 0;        // 1: the decode kernel; 2: the gate/up GEMM
};

inline void stage(StageTimer *t, const char *nm, cudaStream_t st) {
  if (t) t->mark(nm, st);
}

struct LayerDev {
  const uint16_t *hc_fn;
  const float *hc_base, *hc_scale, *ffn_norm, *exp_probs_b;
  const uint16_t *gate;
  const int32_t *tid2eid;
  const uint16_t *gate_exps, *up_exps, *down_exps, *gate_sh, *up_sh, *down_sh;
  // tensor maps of the rows > 4 path over the caller's bf16 matrices (routed experts, the shared
  // expert, hc_fn in boxes of 32 rows, the router in boxes of 256 rows; rows past a matrix read as 0)
  CUtensorMap tm_gate, tm_up, tm_down, tm_gate_sh, tm_up_sh, tm_down_sh, tm_hcfn, tm_router;
  uint16_t *mx_bf16;  // bf16 expansion of MXFP8 experts for the rows > 4 path: gate, up, down (routed),
                      // then the shared gate, up, down; null for bf16 layers
  // MXFP8 experts (moe_ffn_set_mxfp8_experts): E4M3 codes in the bf16 layouts, E8M0 scales [rows, K/32]
  const uint8_t *gate_q, *up_q, *down_q, *gate_sh_q, *up_sh_q, *down_sh_q;
  const uint8_t *gate_s, *up_s, *down_s, *gate_sh_s, *up_sh_s, *down_sh_s;
  // tensor maps over the code matrices for the tensor-core decode (boxes of 128 rows x 64 codes)
  CUtensorMap tm_gate_q, tm_up_q, tm_down_q, tm_gate_sh_q, tm_up_sh_q, tm_down_sh_q;
  bool mx_tc;         // MXFP8: no NaN code or scale and every scale within 22 binades of the largest,
                      // so the tensor-core decode's f16 weights are exact (else the CUDA-core kernel)
  int mx_c;           // MXFP8: 134 - the largest scale code (the f16 weights are code x 2^(S - 127 + mx_c))
  bool mx;            // the experts are the MXFP8 ones (decode streams them; prefill their bf16 expansion)
  bool has_experts;   // some expert weights are registered (bf16 at init, or MXFP8 later)
  bool has_weights;
};

// prelude.cu
void launch_prefill_router(const Dims &d, const Scratch &s, const LayerDev &w, const float *state,
                           const int32_t *token_ids, const CUtensorMap &tm_ffn_norm, int rows, bool hash, int num_sms,
                           cudaStream_t st, StageTimer *tm);
int hc_mix_chunks(int rows, int hcd);
void launch_hc_pre(const Dims &d, const Scratch &s, const LayerDev &w, const float *state, const CUtensorMap *tm_state,
                   int rows, int num_sms, float *x_norm, float *pre, float *post, float *comb, cudaStream_t st);
void launch_hc_mix_raw(const float *state, const uint16_t *hc_fn, const float *hc_scale, const float *hc_base,
                       int rows, int hc, int hidden, int iters, float eps, float *partial, unsigned *tickets,
                       float *mixes, float *pre, float *post, float *comb, cudaStream_t st,
                       const float *norm_w = nullptr, float *x_norm = nullptr);
RouteParams make_route(const Dims &d, const Scratch &s, const LayerDev &w, const int32_t *token_ids, bool hash,
                       int *counts);
// moe_ffn.cu
void set_global_error(const char *msg);
// decode.cu
constexpr int kDecodeGroupsMax = 4 * 8 + 1;  // rows x top_k distinct experts + the shared one
constexpr int kDecodeDBlock = 32;            // d-block of the decode reduce + hc_post (one d per lane)
int decode_counter_count(const Dims &d);
int decode_mix_ctas(int hc, int hidden);     // CTAs of the decode kernel's mix role
int decode_router_ctas(int experts);         // CTAs of its router role
void launch_decode(const Dims &d, const Scratch &s, const LayerDev &w, const float *state, const int32_t *token_ids,
                   int rows, bool hash, float *out_state, cudaStream_t st, StageTimer *tm, const DebugOpts &dbg);
cudaError_t decode_configure(int hidden);
int decode_resident_ctas(int hidden, int rows, int num_sms, bool mx);
// decode_tc.cu
int decode_tc_counter_count(const Dims &d);
cudaError_t decode_tc_configure();
int decode_tc_resident_ctas(int rows, int num_sms, bool mx);
bool decode_tc_fits(const Dims &d, int grid);
void launch_mxfp8_to_bf16(const uint8_t *q, const uint8_t *s, uint16_t *dst, size_t n, cudaStream_t st);
void launch_e4m3_nan_scan(const uint8_t *q, size_t n, int *flag, cudaStream_t st);
void launch_e8m0_range(const uint8_t *sc, size_t n, unsigned *mm, cudaStream_t st);
// dispatch.cu
void launch_dispatch(const Dims &d, const Scratch &s, int rows, cudaStream_t st, StageTimer *tm);
void launch_hc_post(const Dims &d, const float *f, const float *state, const float *post, const float *comb,
                    int rows, float *out_state, cudaStream_t st);
void launch_hc_post(const Dims &d, const double *f, const float *state, const float *post, const float *comb,
                    int rows, float *out_state, cudaStream_t st);
// splitgemm.cu
void launch_prefill_mix(const Dims &d, const Scratch &s, const LayerDev &w, const float *state,
                        const CUtensorMap &tm_state, int rows, int num_sms, cudaStream_t st, StageTimer *tm);
int launch_router_tc(const Dims &d, const Scratch &s, const LayerDev &w, const CUtensorMap &tm_x, int rows, int num_sms,
                     cudaStream_t st);
int mix_tc_part_floats(int max_rows, int hcd);
int splitgemm_splits(int k);  // K splits of the tensor-core mix / router GEMMs
cudaError_t splitgemm_configure();
// gemm_tc.cu
// tm_x2, tm_act2: device arrays of 8 tensor maps each over the activation planes, with boxes of
// 16, 32, ..., 128 rows
void launch_grouped_gemms(const Dims &d, const Scratch &s, const LayerDev &w, const CUtensorMap *tm_x2,
                          const CUtensorMap *tm_act2, int num_sms, cudaStream_t st, StageTimer *tm,
                          const DebugOpts &dbg);
size_t gemm_smem_bytes(bool gateup);
cudaError_t gemm_configure();

}  // namespace moe
