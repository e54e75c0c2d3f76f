// Internal declarations shared by the translation units of libsbp.so.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/sbp.h"

namespace sbp {

// Width (in vocabulary columns) of one row-statistics tile: each (row, tile) pair gets
// one partial (max, sum of exp) and one gradient scale.
constexpr int kStatW = 128;

// Guard zones of the checked build (compiled with SBP_CHECKED): every workspace region is
// followed by kGuardBytes holding a known pattern, written by the call before its first
// kernel and verified after its last one; a mismatch (a kernel wrote past its region)
// sets SBP_ERR_WORKSPACE_OVERRUN.  The release build has no guard zones.
#ifdef SBP_CHECKED
constexpr size_t kGuardBytes = 256;
#else
constexpr size_t kGuardBytes = 0;
#endif
constexpr int kMaxGuards = 24;
struct Guards {
  int n = 0;
  size_t off[kMaxGuards] = {};
};

// The next workspace region of `bytes` at offset o (256-byte aligned); o moves past the
// region and, in the checked build, past the region's guard zone.
inline size_t take_region(size_t& o, size_t bytes, Guards& g) {
  const size_t at = o;
  o = (o + bytes + 255) & ~size_t(255);
  if (kGuardBytes && g.n < kMaxGuards) {
    g.off[g.n++] = o;
    o += kGuardBytes;
  }
  return at;
}

// NVTX ranges around each call and its phases in the NVTX build (SBP_NVTX); nothing in
// the others.  The ranges mark the host's enqueueing; a timeline tool pairs them with
// the launches they contain.
#ifdef SBP_NVTX
#include <nvtx3/nvToolsExt.h>
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
#else
struct NvtxRange {
  explicit NvtxRange(const char*) {}
};
#endif

// Workspace carve-up.  Every region starts on a 256-byte boundary.
struct Layout {
  int64_t T = 0, d = 0, V = 0, chunk = 0;  // chunk = rows of the largest chunk (<= T)
  int dtype = 0, mode = 0;
  int64_t ldv = 0;      // row stride (elements) of the chunk logit/gradient buffer
  int nbuf = 1;         // chunk buffers: 2 lets chunk c's gradient form inside chunk c+1's forward
  int64_t ntiles = 0;   // row-statistics tiles per row = ceil(V / kStatW)
  int splits = 1;       // dH split-K factor (tensor-core path)
  size_t esize = 0;     // bytes per element of the chunk buffer
  size_t off_zg = 0, off_part = 0, off_zy = 0, off_rowv = 0, off_dhp = 0;
  size_t off_zg2 = 0, off_part2 = 0, off_rowv2 = 0;   // second buffer set (nbuf = 2)
  size_t off_tokloss = 0, off_logp = 0, off_seqw = 0, off_scal = 0, off_cnt = 0;
  int64_t n_chunks = 0, max_seq = 0;
  // streaming host buffers (sbp_lmhead_sft_host): device slots for three chunks of H rows
  // and two of dH rows, the labels [T] int32, and the loss / N scalars
  bool host = false;
  size_t off_hs = 0, off_dhs = 0, off_y = 0, off_hscal = 0;
  size_t total = 0;
  Guards guards;   // checked build only
};

// Fills `L`; returns false for arguments no call can accept.
bool make_layout(int64_t T, int64_t d, int64_t V, int64_t chunk, int dtype, int mode, Layout* L,
                 int nbuf = 0,    // 0: the entry points' default (2 for bf16 gradients, else 1)
                 bool host = false);

// dH split-K factor of the tensor-core backward kernel for a chunk of `rows` rows.
int choose_splits(int64_t rows, int64_t d, int64_t V, int num_sms);
int num_sms();

// ----- launchers (enqueue only; return cudaError_t of the launch) -----

// tensor-core kernels (bf16 operands), sbp_tc.cu
struct TcFwdArgs {
  const void* H; const void* W; int64_t T, d, V;
  int64_t r0; int rows;
  const int32_t* labels;   // labels of the chunk (already offset by r0)
  int32_t ignore_index;
  void* E; int64_t lde;    // fp16 exp(z - tile max), [rows, lde]; nullptr: statistics only
  float2* part; float* zy;
  int32_t* status;
  // optional: the previous chunk's logit gradient, formed in place by this launch's
  // epilogue warps between tiles (G = e * scale, w expm1(logp) at the label; fp16 -> bf16)
  void* gprev = nullptr; const float2* part_prev = nullptr; const float* w_prev = nullptr;
  const int32_t* y_prev = nullptr; int rows_prev = 0;
};
cudaError_t tc_forward(const TcFwdArgs& a, cudaStream_t s);

struct TcBwdArgs {
  const void* G; int64_t ldg;   // bf16 [rows, ldg]
  const void* H; const void* W; int64_t T, d, V;
  int64_t r0; int rows;
  int splits;
  float* dh_part;               // [splits, rows, d] fp32
  float* dW; int dw_accumulate;
  uint32_t* counter;            // zero before launch
  int32_t* status;
  int dw_only = 0;              // 1: only the dW units (no dH)
  // a batch of problems stacked along the rows of every operand (attention heads): the
  // maps span all of them; problem z starts at row z * zr_* of G, W, H and dW, and its
  // dH partials at plane (split * batch + z)
  int batch = 1;
  int zr_g = 0, zr_w = 0, zr_h = 0, zr_dw = 0;
  // row extents of the maps (0: rows for G, T for H, V for W and dW)
  int64_t g_rows = 0, w_rows = 0, h_rows = 0, dw_rows = 0;
};
cudaError_t tc_backward(const TcBwdArgs& a, cudaStream_t s);

// SwiGLU-MLP pair GEMMs, sbp_mlp.cu.  da = false: g | u = x_c [Wg; Wu]^T with the
// activation epilogue (B = packed Wgu [2f, d]); da = true: da = dY_c Wd with the
// activation-backward epilogue (B = Wd [d, f]), in place over g | u.
struct TcMlpArgs {
  const void* Arows; int64_t T, d, f;  // x or dY [T, d] bf16
  const void* B;                       // Wgu [2f, d] or Wd [d, f], bf16
  int64_t r0; int rows;
  void* Aout;                          // a = silu(g) u [rows, f] bf16 (da = false)
  void* GU;                            // [rows, 2f] bf16
  int32_t* status;
};
cudaError_t tc_mlp(const TcMlpArgs& a, bool da, cudaStream_t s);

// Causal-attention pair GEMMs, sbp_attn.cu, batched over heads.  ds = false: P = softmax
// row of S = Q_c K^T (lse given) into P; ds = true: dS = s P (dO_c V^T - D) into dS.
struct TcAttnArgs {
  const void* A; const void* B;   // Q / K (ds = false) or dO / V (ds = true), [H * T, hd] bf16
  int64_t T, hd; int H;
  int64_t c0; int rows;           // queries [c0, c0 + rows), keys [0, c0 + rows)
  float scale;
  const float* lse; const float* D;   // [H, T]
  void* P; void* dS;              // [H, Cmax, Lp] bf16
  int64_t Cmax, Lp;
  int32_t* status;
};
cudaError_t tc_attn(const TcAttnArgs& a, bool ds, cudaStream_t s);

// Fused causal-attention backward at head dimension 128, sbp_attn_fused.cu: per chunk
// of queries [c0, c1), k_attn_kv adds dV and s dK of keys [0, c1) into the fp32 outputs
// and k_attn_q writes dQ of the chunk's rows (bf16); P and dS never leave the chip.
// The tensor maps are built once per call (init) and serve every chunk.
struct AttnFusedPlan {
  int64_t T = 0, H = 0, Hkv = 0;   // query heads H = Hkv x group (grouped-query attention)
  CUtensorMap K128, V128, Q64, O64, Q128, O128, K64, V64, dK, dV;
  bool init(const void* Q, const void* K, const void* V, const void* dO, float* dK, float* dV, int64_t T,
            int64_t H, int64_t Hkv);
};
cudaError_t attn_fused_kv(const AttnFusedPlan& plan, int64_t c0, int64_t c1, float scale, const float* lse,
                          const float* D, int32_t* status, cudaStream_t s);
cudaError_t attn_fused_q(const AttnFusedPlan& plan, int64_t c0, int64_t c1, float scale, const float* lse,
                         const float* D, void* dQ, int32_t* status, cudaStream_t s);

// SIMT fp32 kernels (fp32 operands), sbp_simt.cu
cudaError_t simt_forward(const float* H, const float* W, int64_t d, int64_t V, int64_t r0, int rows,
                         const int32_t* labels, int32_t ign, float* E, int64_t lde, float2* part,
                         float* zy, bool store_e, cudaStream_t s);
cudaError_t simt_backward(const float* G, int64_t ldg, const float* H, const float* W, int64_t d,
                          int64_t V, int64_t r0, int rows, float* dh_part, float* dW,
                          int dw_accumulate, cudaStream_t s);

}  // namespace sbp
