// C ABI of libsbp.so and the host-side chunk scheduler.
//
// One call = label scan, then for each chunk of `chunk` rows (the chunk loop of the
// StreamBP LM head: ziziman.com article, LM-head paragraphs):
//   forward GEMM + row-statistics epilogue -> combine (lse, logp, weight) ->
//   logit gradient (in place over the chunk buffer) -> dH / dW GEMMs -> dH reduce,
// and finally the deterministic loss reduction.  Everything is enqueued on the
// caller's stream; nothing here synchronises the host or allocates device memory.
#include <cfloat>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "sbp_internal.h"

namespace sbp {

static thread_local int g_launches = 0;

// ---- optional per-kernel-class timing (CUDA events on the call's stream) ----
namespace prof {
constexpr int kClasses = 4;
struct Pair { cudaEvent_t a, b; int cls; };
static thread_local bool g_on = false;
static thread_local std::vector<Pair>* g_pairs = nullptr;   // recorded, not yet read
static thread_local std::vector<cudaEvent_t>* g_pool = nullptr;

static cudaEvent_t get_event() {
  if (!g_pool) g_pool = new std::vector<cudaEvent_t>();
  if (!g_pool->empty()) {
    cudaEvent_t e = g_pool->back();
    g_pool->pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}
struct Scope {
  cudaEvent_t a = nullptr, b = nullptr;
  int cls;
  cudaStream_t s;
  Scope(int c, cudaStream_t st) : cls(c), s(st) {
    if (!g_on) return;
    a = get_event();
    b = get_event();
    if (a && b) cudaEventRecord(a, s);
  }
  ~Scope() {
    if (!g_on || !a || !b) return;
    cudaEventRecord(b, s);
    if (!g_pairs) g_pairs = new std::vector<Pair>();
    g_pairs->push_back({a, b, cls});
  }
};
}  // namespace prof

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

// Split-K factor for dH: the backward kernel schedules the dH units (K = V, long)
// before the dW units (K = rows, short) from one dynamic queue.  One dH unit should
// stay below a quarter of the average per-SM work so the short dW units can even
// out the finish times.
int choose_splits(int64_t rows, int64_t d, int64_t V, int sms) {
  // units are 256-row tiles computed by SM pairs
  const int64_t mt_c = (rows + 255) / 256, nt_d = (d + 255) / 256, kb_v = (V + 63) / 64;
  const int64_t mt_v = (V + 255) / 256, kb_c = (rows + 63) / 64;
  const double total = double(mt_c * nt_d * kb_v + mt_v * nt_d * kb_c);
  const double per_sm = total / double(sms > 1 ? sms / 2 : 74);
  int s = (int)std::ceil(4.0 * double(kb_v) / (per_sm > 1.0 ? per_sm : 1.0));
  if (s < 1) s = 1;
  if (s > 16) s = 16;
  if (s > kb_v) s = (int)kb_v;
  return s;
}

bool make_layout(int64_t T, int64_t d, int64_t V, int64_t chunk, int dtype, int mode, Layout* L, int nbuf,
                 bool host) {
  if (T < 0 || d < 1 || V < 1 || chunk < 1 || chunk > 65535) return false;
  if (dtype != SBP_BF16 && dtype != SBP_FP32) return false;
  if (mode < SBP_MODE_SFT || mode > SBP_MODE_DPO2) return false;
  Layout l;
  l.T = T; l.d = d; l.V = V; l.dtype = dtype; l.mode = mode;
  l.chunk = T > 0 ? (chunk < T ? chunk : T) : 1;
  l.esize = dtype == SBP_BF16 ? 2 : 4;
  l.ldv = dtype == SBP_BF16 ? ((V + 63) / 64) * 64 : ((V + 3) / 4) * 4;
  l.ntiles = (V + kStatW - 1) / kStatW;
  l.splits = dtype == SBP_BF16 ? choose_splits(l.chunk, d, V, num_sms()) : 1;
  l.n_chunks = T > 0 ? (T + l.chunk - 1) / l.chunk : 0;
  l.max_seq = T + 64;
  if (nbuf == 0) nbuf = (dtype == SBP_BF16 && mode != SBP_MODE_DPO1 && l.n_chunks > 1) ? 2 : 1;
  l.nbuf = nbuf;
  size_t o = 0;
  Guards& g = l.guards;
  l.off_zg = take_region(o, (size_t)l.chunk * l.ldv * l.esize, g);
  l.off_part = take_region(o, (size_t)l.chunk * l.ntiles * sizeof(float2), g);
  l.off_zy = take_region(o, (size_t)l.chunk * sizeof(float), g);
  l.off_rowv = take_region(o, (size_t)l.chunk * sizeof(float), g);
  if (nbuf == 2) {
    l.off_zg2 = take_region(o, (size_t)l.chunk * l.ldv * l.esize, g);
    l.off_part2 = take_region(o, (size_t)l.chunk * l.ntiles * sizeof(float2), g);
    l.off_rowv2 = take_region(o, (size_t)l.chunk * sizeof(float), g);
  }
  l.off_dhp = take_region(o, (size_t)l.splits * l.chunk * d * sizeof(float), g);
  l.off_tokloss = take_region(o, (size_t)(T + 1) * sizeof(float), g);
  l.off_logp = take_region(o, (size_t)(T + 1) * sizeof(float), g);
  l.off_seqw = take_region(o, (size_t)l.max_seq * sizeof(float), g);
  l.off_scal = take_region(o, 64, g);  // [0] int64 N
  l.off_cnt = take_region(o, (size_t)(l.n_chunks + 1) * sizeof(uint32_t), g);
  if (host) {
    const size_t slot = (size_t)l.chunk * d * l.esize;
    l.host = true;
    l.off_hs = take_region(o, 3 * slot, g);
    l.off_dhs = take_region(o, 2 * slot, g);
    l.off_y = take_region(o, (size_t)(T + 1) * sizeof(int32_t), g);
    l.off_hscal = take_region(o, 64, g);  // [0] fp32 loss, [8] int64 N
  }
  l.total = o;
  *L = l;
  return true;
}

namespace {

__device__ __forceinline__ void set_status(int32_t* st, int32_t code) {
  if (st) atomicCAS(st, 0, code);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Label scan (one block): N = #{t : y_t != ign}; labels outside [0, V) other than
// ign raise SBP_ERR_LABEL_RANGE; zeroes the per-chunk scheduler counters.
__global__ void __launch_bounds__(1024) k_prep(const int32_t* __restrict__ y, int64_t T, int64_t V, int32_t ign,
                                               long long* __restrict__ nvalid, uint32_t* __restrict__ counters,
                                               int64_t n_counters, int32_t* status) {
  __shared__ long long red[32];
  long long c = 0;
  bool bad = false;
  for (int64_t t = threadIdx.x; t < T; t += blockDim.x) {
    const int32_t v = y[t];
    if (v != ign) {
      ++c;
      if (v < 0 || (int64_t)v >= V) bad = true;
    }
  }
  for (int64_t i = threadIdx.x; i < n_counters; i += blockDim.x) counters[i] = 0u;
  if (bad) set_status(status, SBP_ERR_LABEL_RANGE);
#pragma unroll
  for (int o = 16; o; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    long long s = 0;
    for (int i = 0; i < (int)(blockDim.x / 32); ++i) s += red[i];
    *nvalid = s;
  }
}

struct CombineArgs {
  const float2* part; int64_t ntiles;
  const float* zy;
  const int32_t* labels;   // chunk-offset
  int rows; int64_t r0; int64_t V; int32_t ign;
  const long long* nvalid;
  float* w_row;            // [rows] weight of the row's logit gradient
  float* logp;             // [T]
  float* tokloss;          // [T] loss contribution of the token
  // GRPO
  const float* adv; const float* logp_old; float clip_lo, clip_hi;
  // DPO pass 2; GRPO per-sequence mean (seqw = each sequence's share of the mean)
  const int32_t* cu; int n_seq; const float* seqw;
  // GRPO KL penalty
  const float* ref_logp; float kl_coef;
};

// Index of the sequence holding token t (cu non-decreasing), or -1 outside all.
__device__ __forceinline__ int seq_of(const int32_t* cu, int n_seq, int64_t t) {
  if (n_seq <= 0 || t < cu[0] || t >= cu[n_seq]) return -1;
  int lo = 0, hi = n_seq - 1;  // last i with cu[i] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// One warp per row over the row's tile partials (m_i, r_i), where r_i = sum of
// exp(z - m_i) over the tile's columns less the one at the tile's maximum (whose term is
// exactly 1).  With M = max_i m_i, the sum of exp(z - M) over the whole row is 1 + R,
//   R = sum_{i: m_i < M} (1 + r_i) exp(m_i - M) + sum_{i: m_i = M} r_i + (#{i: m_i = M} - 1),
// a sum of non-negative terms, so lse = M + log1p(R) and logp = (z_y - M) - log1p(R) keep
// their relative precision when the label holds almost all the probability mass (R -> 0,
// the confident-token regime), where 1 + R itself would round to 1.  Then the
// objective's weight w and loss term.  The tile maxima are replaced in place by the
// gradient scales w exp(m_i - lse), so that the gradient kernel needs one multiply per
// element, G = e * scale; the label's own entry, w (p_y - 1) = w expm1(logp), is written
// into the second field of the label's tile partial, so that it does not come from the
// cancelling difference e_y * scale - w.
template <int MODE>
__global__ void __launch_bounds__(256) k_combine(CombineArgs a) {
  const int lane = threadIdx.x % 32;
  const int row = blockIdx.x * 8 + threadIdx.x / 32;
  if (row >= a.rows) return;
  float2* p = const_cast<float2*>(a.part) + (int64_t)row * a.ntiles;
  float m = -FLT_MAX;
  for (int64_t i = lane; i < a.ntiles; i += 32) m = fmaxf(m, p[i].x);
  m = warp_max(m);
  float rest = 0.f, ties = 0.f;
  for (int64_t i = lane; i < a.ntiles; i += 32) {
    const float2 q = p[i];
    if (q.x == m) {
      rest += q.y;
      ties += 1.f;
    } else {
      rest += (1.f + q.y) * expf(q.x - m);
    }
  }
  rest = warp_sum(rest) + (warp_sum(ties) - 1.f);
  const float l1 = log1pf(rest);
  const int32_t y = a.labels[row];
  const bool valid = y != a.ign && y >= 0 && (int64_t)y < a.V;
  const float logp = valid ? (a.zy[row] - m) - l1 : 0.f;
  const long long N = *a.nvalid;
  const float invN = N > 0 ? (float)(1.0 / (double)N) : 0.f;
  float w = 0.f, tl = 0.f;
  const int64_t t = a.r0 + row;
  if (MODE == SBP_MODE_SFT) {
    w = valid ? invN : 0.f;
    tl = valid ? -logp * invN : 0.f;
  } else if (MODE == SBP_MODE_GRPO) {
    if (valid) {
      const float A = a.adv[t];
      const float r = expf(logp - a.logp_old[t]);
      const float rc = fminf(fmaxf(r, a.clip_lo), a.clip_hi);
      const float o = fminf(r * A, rc * A);
      const bool g = (A >= 0.f) ? (r <= a.clip_hi) : (r >= a.clip_lo);
      float fac = invN;  // the token's share of the mean
      if (a.cu) {
        const int sq = seq_of(a.cu, a.n_seq, t);
        fac = sq >= 0 ? a.seqw[sq] : 0.f;
      }
      float kl = 0.f, dkl = 0.f;  // k3 KL to the reference and its logp-derivative
      if (a.ref_logp && a.kl_coef != 0.f) {
        const float q = a.ref_logp[t] - logp;
        const float eq = expf(q);
        kl = eq - q - 1.f;
        dkl = 1.f - eq;
      }
      w = fac * ((g ? A * r : 0.f) - a.kl_coef * dkl);
      tl = fac * (-o + a.kl_coef * kl);
    }
  } else if (MODE == SBP_MODE_DPO2) {
    const int sq = valid ? seq_of(a.cu, a.n_seq, t) : -1;
    if (sq >= 0) w = a.seqw[sq];
  }
  const int64_t ty = valid ? (int64_t)y / kStatW : -1;
  const float gy = w * expm1f(logp);
  for (int64_t i = lane; i < a.ntiles; i += 32) p[i] = make_float2(w * expf((p[i].x - m) - l1), i == ty ? gy : 0.f);
  if (lane == 0) {
    a.w_row[row] = w;
    a.logp[t] = logp;
    a.tokloss[t] = tl;
  }
}

__device__ __forceinline__ void load8(const __half* p, float* f) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = __half22float2(h[i]);
    f[2 * i] = x.x; f[2 * i + 1] = x.y;
  }
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float* f) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void load8(const float* p, float* f) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
__device__ __forceinline__ void store8(float* p, const float* f) {
  reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}
__device__ __forceinline__ float ld1(const __half* p) { return __half2float(*p); }
__device__ __forceinline__ float ld1(const float* p) { return *p; }
__device__ __forceinline__ void st1(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ void st1(float* p, float v) { *p = v; }

// Logit gradient of one chunk, in place over the chunk buffer:
//   G[r, v] = e[r, v] * scale[r, tile(v)] for v != y_r, and w_r expm1(logp_r) at the
//   label (both from the combine step), i.e. w_r (softmax - onehot).
// TE -> TG: fp16 -> bf16 (tensor-core path) or fp32 -> fp32 (SIMT path).
template <typename TE, typename TG>
__global__ void __launch_bounds__(256) k_grad(void* buf, int64_t ld, int64_t V, const float2* __restrict__ part,
                                              int64_t ntiles, const float* __restrict__ w_row,
                                              const int32_t* __restrict__ labels) {
  static_assert(sizeof(TE) == sizeof(TG), "in-place conversion needs equal element sizes");
  const int64_t row = blockIdx.y;
  const float w = w_row[row];
  const int32_t y = labels[row];
  TE* e = reinterpret_cast<TE*>(buf) + row * ld;
  TG* g = reinterpret_cast<TG*>(buf) + row * ld;
  const float2* sc = part + row * ntiles;
  for (int64_t v0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8; v0 < V;
       v0 += (int64_t)gridDim.x * blockDim.x * 8) {
    float f[8];
    if (v0 + 8 <= V) {
      if (w == 0.f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = 0.f;
      } else {
        load8(e + v0, f);
        const float2 s = sc[v0 / kStatW];
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = v0 + i == (int64_t)y ? s.y : f[i] * s.x;
      }
      store8(g + v0, f);
    } else {
      for (int64_t v = v0; v < V; ++v) {
        const float2 s = sc[v / kStatW];
        const float x = w == 0.f ? 0.f : (v == y ? s.y : ld1(e + v) * s.x);
        st1(g + v, x);
      }
    }
  }
}

// dH rows of the chunk = sum over the split-K partials, converted to the output dtype.
template <typename TO>
__global__ void __launch_bounds__(256) k_dh_reduce(const float* __restrict__ part, int splits, int64_t n,
                                                   int64_t plane, TO* __restrict__ out) {
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; i < n;
       i += (int64_t)gridDim.x * blockDim.x * 4) {
    if (i + 4 <= n) {
      float4 acc = *reinterpret_cast<const float4*>(part + i);
      for (int s = 1; s < splits; ++s) {
        const float4 q = *reinterpret_cast<const float4*>(part + s * plane + i);
        acc.x += q.x; acc.y += q.y; acc.z += q.z; acc.w += q.w;
      }
      st1(out + i, acc.x); st1(out + i + 1, acc.y); st1(out + i + 2, acc.z); st1(out + i + 3, acc.w);
    } else {
      for (int64_t j = i; j < n; ++j) {
        float acc = part[j];
        for (int s = 1; s < splits; ++s) acc += part[s * plane + j];
        st1(out + j, acc);
      }
    }
  }
}

// Deterministic loss reduction (one block, fp64, fixed order).
__global__ void __launch_bounds__(1024) k_loss_final(const float* __restrict__ tokloss, int64_t T,
                                                     const long long* __restrict__ nvalid_ws, float* loss,
                                                     int64_t* n_valid_out) {
  __shared__ double red[1024];
  double acc = 0.0;
  for (int64_t t = threadIdx.x; t < T; t += blockDim.x) acc += (double)tokloss[t];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int s = blockDim.x / 2; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    if (loss) *loss = (float)red[0];
    if (n_valid_out) *n_valid_out = (int64_t)*nvalid_ws;
  }
}

// DPO pass 1: S_i = sum of logp over [cu[i], cu[i+1]) (one block per sequence, fp64).
__global__ void __launch_bounds__(256) k_seq_sums(const float* __restrict__ logp, const int32_t* __restrict__ cu,
                                                  double* __restrict__ seq_logp) {
  __shared__ double red[256];
  const int i = blockIdx.x;
  const int64_t b = cu[i], e = cu[i + 1];
  double acc = 0.0;
  for (int64_t t = b + threadIdx.x; t < e; t += blockDim.x) acc += (double)logp[t];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) seq_logp[i] = red[0];
}

// GRPO per-sequence mean: each sequence's share 1 / (n_seq * N_i) of the mean, N_i its
// number of non-ignored tokens (0 when N_i = 0).  One block per sequence.
__global__ void __launch_bounds__(256) k_seq_share(const int32_t* __restrict__ y, const int32_t* __restrict__ cu,
                                                   int n_seq, int32_t ign, float* __restrict__ share) {
  __shared__ int red[256];
  const int i = blockIdx.x;
  int c = 0;
  for (int64_t t = cu[i] + threadIdx.x; t < cu[i + 1]; t += blockDim.x) c += y[t] != ign;
  red[threadIdx.x] = c;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) share[i] = red[0] > 0 ? (float)(1.0 / ((double)n_seq * (double)red[0])) : 0.f;
}

__device__ __forceinline__ double softplus_d(double x) {
  return (x > 0 ? x : 0.0) + log1p(exp(-fabs(x)));
}
__device__ __forceinline__ double sigmoid_d(double x) {
  if (x >= 0) return 1.0 / (1.0 + exp(-x));
  const double e = exp(x);
  return e / (1.0 + e);
}

// DPO pass 2 prologue (one thread): margins, loss and per-sequence weights.
__global__ void k_dpo_scales(const double* __restrict__ S, const double* __restrict__ R, int n_seq, double beta,
                             float* loss, double* margins, float* seqw) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  const int P = n_seq / 2;
  double L = 0.0;
  for (int i = 0; i < P; ++i) {
    const double m = beta * ((S[i] - R[i]) - (S[i + P] - R[i + P]));
    L += softplus_d(-m);
    const double w = beta * sigmoid_d(-m) / (double)P;
    seqw[i] = (float)w;
    seqw[i + P] = (float)(-w);
    if (margins) margins[i] = m;
  }
  if (loss) *loss = P > 0 ? (float)(L / (double)P) : 0.f;
}

#ifdef SBP_CHECKED
// Guard zone z holds the words 0x5BADF00D ^ (z << 16) ^ i; `skew` (the SBP_FAULT_GUARD
// test knob) plants a wrong first word in the last zone, standing in for an overrun.
__global__ void __launch_bounds__(64) k_guard(unsigned char* ws, Guards g, int check, uint32_t skew,
                                              int32_t* status) {
  const int z = blockIdx.x;
  if (z >= g.n) return;
  uint32_t* p = reinterpret_cast<uint32_t*>(ws + g.off[z]);
  for (int i = threadIdx.x; i < (int)(kGuardBytes / 4); i += blockDim.x) {
    const uint32_t want = 0x5BADF00Du ^ ((uint32_t)z << 16) ^ (uint32_t)i;
    if (!check)
      p[i] = want + ((z == g.n - 1 && i == 0) ? skew : 0u);
    else if (p[i] != want)
      set_status(status, SBP_ERR_WORKSPACE_OVERRUN);
  }
}
#endif

// Fills (check = 0) or verifies (check = 1) a workspace's guard zones on stream s; nothing
// in the release build, whose layouts have no guard zones.
int guard_zones(void* ws, const Guards& g, int check, int32_t* status, cudaStream_t s, int* launches) {
#ifdef SBP_CHECKED
  if (g.n == 0) return SBP_OK;
  uint32_t skew = 0;
  if (!check) {
    const char* e = std::getenv("SBP_FAULT_GUARD");
    skew = (e && e[0] == '1') ? 1u : 0u;
  }
  k_guard<<<g.n, 64, 0, s>>>(static_cast<unsigned char*>(ws), g, check, skew, status);
  ++*launches;
  return cudaGetLastError() == cudaSuccess ? SBP_OK : SBP_ERR_CUDA;
#else
  (void)ws; (void)g; (void)check; (void)status; (void)s; (void)launches;
  return SBP_OK;
#endif
}

__global__ void k_zero_f32(float* p, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    p[i] = 0.f;
}

inline unsigned grid_for(int64_t work, int threads, int64_t cap = 4096) {
  int64_t g = (work + threads - 1) / threads;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return (unsigned)g;
}

// A second stream per device, for the work of one call that may run beside the caller's
// stream: forked from it after an event and joined back into it before the call returns,
// so the caller sees one ordered call on its own stream.  The lock is held while a call
// enqueues its fork .. join, so concurrent calls never mix their events.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  cudaEvent_t ev[8] = {};   // handoffs inside a call (the LM head's host-buffer pipeline)
  std::mutex mu;
};
static SideStream g_side[64];
static std::mutex g_side_init;

SideStream* side_stream() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_side_init);
  SideStream& ss = g_side[dev];
  if (!ss.s) {
    cudaStream_t st = nullptr;
    cudaEvent_t a = nullptr, b = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&a, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&b, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    for (cudaEvent_t& e : ss.ev)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
      }
    ss.s = st;
    ss.fork = a;
    ss.join = b;
  }
  return &ss;
}

// Host side of a streaming call: H [T, d] and the labels are read from host memory and
// dH [T, d], the loss and N written to it; only a few chunks of rows are ever on the device.
struct HostIO {
  const void* H; const int32_t* labels; void* dH; float* loss; int64_t* n_valid;
};

struct Call {
  int mode;
  const void* H; const void* W; const int32_t* labels;
  int64_t T, d, V, chunk; int32_t ign; int dtype;
  // SFT / GRPO / DPO2 outputs
  float* loss; int64_t* n_valid; float* logp_out;
  void* dH; float* dW; int accumulate_dW;
  // GRPO
  const float* adv; const float* logp_old; float clip_lo, clip_hi;
  const float* ref_logp; float kl_coef;
  // DPO
  const int32_t* cu; int n_seq; double* seq_logp; const double* seq_in; const double* ref_in;
  float beta; double* margins;
  void* ws; size_t ws_bytes; int32_t* dev_status; cudaStream_t stream;
  int nbuf = 0;   // chunk buffer sets (0: default of make_layout)
  const HostIO* host = nullptr;   // non-null: H, labels, dH, loss and N live in host memory
};

#define SBP_CUDA(x)                        \
  do {                                     \
    cudaError_t e_ = (x);                  \
    if (e_ != cudaSuccess) return SBP_ERR_CUDA; \
  } while (0)

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int validate(const Call& c, Layout* L) {
  const bool host = c.host != nullptr;
  if (!make_layout(c.T, c.d, c.V, c.chunk, c.dtype, c.mode, L, c.nbuf, host)) return SBP_ERR_INVALID_ARG;
  // a workspace too small for the default two chunk buffers but large enough for one
  // selects the one-buffer schedule (the logit gradient as its own pass per chunk)
  if (c.nbuf == 0 && L->nbuf == 2 && c.ws_bytes < L->total) {
    Layout lean;
    if (make_layout(c.T, c.d, c.V, c.chunk, c.dtype, c.mode, &lean, 1, host) && c.ws_bytes >= lean.total)
      *L = lean;
  }
  if (host) {
    if (c.mode != SBP_MODE_SFT || !c.host->loss) return SBP_ERR_INVALID_ARG;
    if (c.T > 0 && (!c.host->H || !c.host->labels || !c.host->dH)) return SBP_ERR_INVALID_ARG;
  } else if (c.T > 0 && (!c.H || !c.labels)) {
    return SBP_ERR_INVALID_ARG;
  }
  if (!c.W || !c.dev_status) return SBP_ERR_INVALID_ARG;
  if (c.T > (int64_t)INT32_MAX) return SBP_ERR_UNSUPPORTED;
  const bool grad = c.mode != SBP_MODE_DPO1;
  if (grad && !c.dW) return SBP_ERR_INVALID_ARG;
  if (grad && c.T > 0 && !c.dH && !host) return SBP_ERR_INVALID_ARG;
  if (c.mode == SBP_MODE_GRPO && c.T > 0 && (!c.adv || !c.logp_old)) return SBP_ERR_INVALID_ARG;
  if (c.mode == SBP_MODE_GRPO && !(c.clip_lo <= c.clip_hi)) return SBP_ERR_INVALID_ARG;
  if (c.mode == SBP_MODE_GRPO && c.kl_coef != 0.f && c.T > 0 && !c.ref_logp) return SBP_ERR_INVALID_ARG;
  if (c.mode == SBP_MODE_GRPO && c.cu && (c.n_seq < 1 || c.n_seq > L->max_seq)) return SBP_ERR_INVALID_ARG;
  if (c.mode == SBP_MODE_DPO1 || c.mode == SBP_MODE_DPO2) {
    if (c.n_seq < 0 || c.n_seq > L->max_seq || (c.n_seq > 0 && !c.cu)) return SBP_ERR_INVALID_ARG;
    if (c.mode == SBP_MODE_DPO1 && c.n_seq > 0 && !c.seq_logp) return SBP_ERR_INVALID_ARG;
    if (c.mode == SBP_MODE_DPO2 && (c.n_seq % 2 != 0 || (c.n_seq > 0 && (!c.seq_in || !c.ref_in))))
      return SBP_ERR_INVALID_ARG;
  }
  if (c.dtype == SBP_BF16 && (c.d % 8 != 0 || c.V % 8 != 0)) return SBP_ERR_UNSUPPORTED;
  if ((c.H && !al16(c.H)) || !al16(c.W) || (c.dH && !al16(c.dH)) || (c.dW && !al16(c.dW)))
    return SBP_ERR_ALIGNMENT;
  // (fp32 dH rows are written 4 at a time only when d % 4 == 0; other d take the scalar
  // tail path, which needs no alignment beyond the element size.)
  if (!c.ws || (reinterpret_cast<uintptr_t>(c.ws) & 255u) || c.ws_bytes < L->total) return SBP_ERR_WORKSPACE;
  return SBP_OK;
}

int run(const Call& cin) {
  Layout L;
  int st = validate(cin, &L);
  if (st != SBP_OK) return st;
  cudaStream_t s = cin.stream;
  char* ws = static_cast<char*>(cin.ws);
  void* zg = ws + L.off_zg;
  float2* part = reinterpret_cast<float2*>(ws + L.off_part);
  float* zy = reinterpret_cast<float*>(ws + L.off_zy);
  float* w_row = reinterpret_cast<float*>(ws + L.off_rowv);
  float* dhp = reinterpret_cast<float*>(ws + L.off_dhp);
  float* tokloss = reinterpret_cast<float*>(ws + L.off_tokloss);
  float* logp = reinterpret_cast<float*>(ws + L.off_logp);
  float* seqw = reinterpret_cast<float*>(ws + L.off_seqw);
  long long* nvalid = reinterpret_cast<long long*>(ws + L.off_scal);
  uint32_t* counters = reinterpret_cast<uint32_t*>(ws + L.off_cnt);
  int launches = 0;

  // Streaming host buffers: the labels, the loss and N go through the workspace, and the
  // rows of H and dH through slots there, one chunk at a time, on the side stream:
  // chunk j's H rows enter slot j % 3 ahead of its forward GEMM (at most three chunks
  // ahead: a slot is refilled once its chunk's backward GEMMs are done), and its dH rows
  // leave slot j % 2 for the host while later chunks compute.
  const HostIO* hio = cin.host;
  Call c = cin;
  SideStream* ss = nullptr;
  std::unique_lock<std::mutex> side_lock;
  const size_t row_bytes = (size_t)c.d * L.esize;
  if (hio) {
    c.labels = reinterpret_cast<const int32_t*>(ws + L.off_y);
    c.loss = reinterpret_cast<float*>(ws + L.off_hscal);
    c.n_valid = reinterpret_cast<int64_t*>(ws + L.off_hscal + 8);
    ss = side_stream();
    if (!ss) return SBP_ERR_CUDA;
    side_lock = std::unique_lock<std::mutex>(ss->mu);
  }
  cudaEvent_t* ev_hready = hio ? ss->ev : nullptr;      // [3] chunk's H rows in their slot
  cudaEvent_t* ev_bdone = hio ? ss->ev + 3 : nullptr;   // [2] chunk's backward done
  cudaEvent_t* ev_dhfree = hio ? ss->ev + 5 : nullptr;  // [2] dH slot copied out
  auto h_slot = [&](int64_t ci) { return ws + L.off_hs + (size_t)(ci % 3) * L.chunk * row_bytes; };
  auto dh_slot = [&](int64_t ci) { return ws + L.off_dhs + (size_t)(ci % 2) * L.chunk * row_bytes; };

  NvtxRange nv_call("sbp_lmhead");
  SBP_CUDA(cudaMemsetAsync(c.dev_status, 0, sizeof(int32_t), s));
  st = guard_zones(ws, L.guards, 0, c.dev_status, s, &launches);
  if (st != SBP_OK) return st;
  if (hio && c.T > 0)
    SBP_CUDA(cudaMemcpyAsync(const_cast<int32_t*>(c.labels), hio->labels, (size_t)c.T * sizeof(int32_t),
                             cudaMemcpyHostToDevice, s));
  {
    prof::Scope ps(3, s);
    k_prep<<<1, 1024, 0, s>>>(c.labels, c.T, c.V, c.ign, nvalid, counters, L.n_chunks + 1, c.dev_status);
  }
  ++launches;
  SBP_CUDA(cudaGetLastError());

  const bool grad = c.mode != SBP_MODE_DPO1;
  if (c.mode == SBP_MODE_GRPO && c.cu) {
    prof::Scope ps(3, s);
    k_seq_share<<<c.n_seq, 256, 0, s>>>(c.labels, c.cu, c.n_seq, c.ign, seqw);
    ++launches;
    SBP_CUDA(cudaGetLastError());
  }
  if (c.mode == SBP_MODE_DPO2) {
    k_dpo_scales<<<1, 32, 0, s>>>(c.seq_in, c.ref_in, c.n_seq, (double)c.beta, c.loss, c.margins, seqw);
    ++launches;
    SBP_CUDA(cudaGetLastError());
  }
  if (grad && c.T == 0 && !c.accumulate_dW) {
    k_zero_f32<<<grid_for(c.V * c.d, 256), 256, 0, s>>>(c.dW, c.V * c.d);
    ++launches;
    SBP_CUDA(cudaGetLastError());
  }

  const bool bf16 = c.dtype == SBP_BF16;
  // buffer set b: the chunk's e / G values, tile partials (then scales), row weights
  void* zgb[2] = {zg, L.nbuf == 2 ? ws + L.off_zg2 : zg};
  float2* partb[2] = {part, L.nbuf == 2 ? reinterpret_cast<float2*>(ws + L.off_part2) : part};
  float* wb[2] = {w_row, L.nbuf == 2 ? reinterpret_cast<float*>(ws + L.off_rowv2) : w_row};
  auto r0_of = [&](int64_t ci) { return ci * L.chunk; };
  auto rows_of = [&](int64_t ci) {
    const int64_t r0 = r0_of(ci);
    return (int)((r0 + L.chunk <= c.T) ? L.chunk : c.T - r0);
  };
  // where the GEMMs find chunk ci's H rows: the caller's H at row r0, or the chunk's slot
  auto h_rows = [&](int64_t ci, const void** base, int64_t* T_map, int64_t* r0) {
    if (hio) {
      *base = h_slot(ci); *T_map = rows_of(ci); *r0 = 0;
    } else {
      *base = c.H; *T_map = c.T; *r0 = r0_of(ci);
    }
  };
  // side stream: chunk j's H rows from the host into their slot
  auto h_in = [&](int64_t j) -> int {
    SBP_CUDA(cudaMemcpyAsync(h_slot(j), static_cast<const char*>(hio->H) + (size_t)r0_of(j) * row_bytes,
                             (size_t)rows_of(j) * row_bytes, cudaMemcpyHostToDevice, ss->s));
    SBP_CUDA(cudaEventRecord(ev_hready[j % 3], ss->s));
    return SBP_OK;
  };

  // forward GEMM + row statistics of chunk ci into buffer set b; on the tensor-core path it
  // also forms chunk `prev`'s gradient (buffer set pb) between its tiles when prev >= 0
  auto forward = [&](int64_t ci, int b, int64_t prev, int pb) -> int {
    NvtxRange nv("forward");
    const int64_t r0 = r0_of(ci);
    const int rows = rows_of(ci);
    const void* hb; int64_t hT, hr0;
    h_rows(ci, &hb, &hT, &hr0);
    if (hio) SBP_CUDA(cudaStreamWaitEvent(s, ev_hready[ci % 3], 0));
    if (bf16) {
      TcFwdArgs a{};
      a.H = hb; a.W = c.W; a.T = hT; a.d = c.d; a.V = c.V; a.r0 = hr0; a.rows = rows;
      a.labels = c.labels + r0; a.ignore_index = c.ign;
      a.E = grad ? zgb[b] : nullptr; a.lde = L.ldv; a.part = partb[b]; a.zy = zy; a.status = c.dev_status;
      if (prev >= 0) {
        a.gprev = zgb[pb]; a.part_prev = partb[pb]; a.w_prev = wb[pb];
        a.y_prev = c.labels + r0_of(prev); a.rows_prev = rows_of(prev);
      }
      prof::Scope ps(0, s);
      SBP_CUDA(tc_forward(a, s));
      ++launches;
    } else {
      prof::Scope ps(0, s);
      SBP_CUDA(simt_forward(static_cast<const float*>(hb), static_cast<const float*>(c.W), c.d, c.V, hr0, rows,
                            c.labels + r0, c.ign, static_cast<float*>(zgb[b]), L.ldv, partb[b], zy, grad, s));
      launches += 2;
    }
    return SBP_OK;
  };
  // lse, logp, weights, loss terms; the tile maxima become gradient scales
  auto combine = [&](int64_t ci, int b) -> int {
    NvtxRange nv("combine");
    const int64_t r0 = r0_of(ci);
    const int rows = rows_of(ci);
    CombineArgs ca{};
    ca.part = partb[b]; ca.ntiles = L.ntiles; ca.zy = zy; ca.labels = c.labels + r0; ca.rows = rows; ca.r0 = r0;
    ca.V = c.V; ca.ign = c.ign; ca.nvalid = nvalid; ca.w_row = wb[b]; ca.logp = logp; ca.tokloss = tokloss;
    ca.adv = c.adv; ca.logp_old = c.logp_old; ca.clip_lo = c.clip_lo; ca.clip_hi = c.clip_hi;
    ca.cu = c.cu; ca.n_seq = c.n_seq; ca.seqw = seqw;
    ca.ref_logp = c.ref_logp; ca.kl_coef = c.kl_coef;
    const unsigned gc = (unsigned)((rows + 7) / 8);
    prof::Scope ps(3, s);
    switch (c.mode) {
      case SBP_MODE_SFT: k_combine<SBP_MODE_SFT><<<gc, 256, 0, s>>>(ca); break;
      case SBP_MODE_GRPO: k_combine<SBP_MODE_GRPO><<<gc, 256, 0, s>>>(ca); break;
      case SBP_MODE_DPO1: k_combine<SBP_MODE_DPO1><<<gc, 256, 0, s>>>(ca); break;
      default: k_combine<SBP_MODE_DPO2><<<gc, 256, 0, s>>>(ca); break;
    }
    ++launches;
    SBP_CUDA(cudaGetLastError());
    return SBP_OK;
  };
  // standalone logit gradient, in place
  auto gradient = [&](int64_t ci, int b) -> int {
    NvtxRange nv("gradient");
    const int64_t vec = (c.V + 7) / 8;
    dim3 g((unsigned)((vec + 255) / 256), (unsigned)rows_of(ci));
    prof::Scope ps(2, s);
    if (bf16)
      k_grad<__half, __nv_bfloat16><<<g, 256, 0, s>>>(zgb[b], L.ldv, c.V, partb[b], L.ntiles, wb[b],
                                                       c.labels + r0_of(ci));
    else
      k_grad<float, float><<<g, 256, 0, s>>>(zgb[b], L.ldv, c.V, partb[b], L.ntiles, wb[b], c.labels + r0_of(ci));
    ++launches;
    SBP_CUDA(cudaGetLastError());
    return SBP_OK;
  };
  // dH_c = G_c W and dW (+)= G_c^T H_c, then dH_c's split partials -> dH rows
  auto backward = [&](int64_t ci, int b) -> int {
    NvtxRange nv("backward");
    const int64_t r0 = r0_of(ci);
    const int rows = rows_of(ci);
    const int dw_acc = (ci > 0 || c.accumulate_dW) ? 1 : 0;
    const void* hb; int64_t hT, hr0;
    h_rows(ci, &hb, &hT, &hr0);
    // the dH slot's previous chunk must have left for the host
    if (hio && ci >= 2) SBP_CUDA(cudaStreamWaitEvent(s, ev_dhfree[ci % 2], 0));
    int splits = 1;
    if (bf16) {
      TcBwdArgs bw{};
      bw.G = zgb[b]; bw.ldg = L.ldv; bw.H = hb; bw.W = c.W; bw.T = hT; bw.d = c.d; bw.V = c.V;
      bw.r0 = hr0; bw.rows = rows;
      splits = std::min(choose_splits(rows, c.d, c.V, num_sms()), L.splits);
      bw.splits = splits; bw.dh_part = dhp; bw.dW = c.dW; bw.dw_accumulate = dw_acc;
      bw.counter = counters + ci; bw.status = c.dev_status;
      prof::Scope ps(1, s);
      SBP_CUDA(tc_backward(bw, s));
      ++launches;
    } else {
      prof::Scope ps(1, s);
      SBP_CUDA(simt_backward(static_cast<const float*>(zgb[b]), L.ldv, static_cast<const float*>(hb),
                             static_cast<const float*>(c.W), c.d, c.V, hr0, rows, dhp, c.dW, dw_acc, s));
      launches += 2;
    }
    const int64_t n = (int64_t)rows * c.d;
    void* dst = hio ? static_cast<void*>(dh_slot(ci)) : static_cast<char*>(c.dH) + (size_t)r0 * row_bytes;
    {
      prof::Scope ps(3, s);
      if (bf16)
        k_dh_reduce<__nv_bfloat16><<<grid_for(n / 4 + 1, 256), 256, 0, s>>>(
            dhp, splits, n, n, static_cast<__nv_bfloat16*>(dst));
      else
        k_dh_reduce<float><<<grid_for(n / 4 + 1, 256), 256, 0, s>>>(dhp, splits, n, n, static_cast<float*>(dst));
      ++launches;
      SBP_CUDA(cudaGetLastError());
    }
    if (hio) {
      // side stream: dH rows out to the host, then the freed H slot takes chunk ci + 3
      SBP_CUDA(cudaEventRecord(ev_bdone[ci % 2], s));
      SBP_CUDA(cudaStreamWaitEvent(ss->s, ev_bdone[ci % 2], 0));
      SBP_CUDA(cudaMemcpyAsync(static_cast<char*>(hio->dH) + (size_t)r0 * row_bytes, dst, (size_t)n * L.esize,
                               cudaMemcpyDeviceToHost, ss->s));
      SBP_CUDA(cudaEventRecord(ev_dhfree[ci % 2], ss->s));
      if (ci + 3 < L.n_chunks) {
        const int hs = h_in(ci + 3);
        if (hs != SBP_OK) return hs;
      }
    }
    return SBP_OK;
  };

#define SBP_TRY(x)                      \
  do {                                  \
    const int st_ = (x);                \
    if (st_ != SBP_OK) return st_;      \
  } while (0)

  auto schedule = [&]() -> int {
    if (hio) {
      SBP_CUDA(cudaEventRecord(ss->fork, s));
      SBP_CUDA(cudaStreamWaitEvent(ss->s, ss->fork, 0));
      for (int64_t j = 0; j < std::min<int64_t>(3, L.n_chunks); ++j) SBP_TRY(h_in(j));
    }
    if (!grad) {
      for (int64_t ci = 0; ci < L.n_chunks; ++ci) {
        SBP_TRY(forward(ci, 0, -1, 0));
        SBP_TRY(combine(ci, 0));
      }
    } else if (L.nbuf == 2 && bf16) {
      // chunk ci's gradient forms inside chunk ci+1's forward (two buffer sets):
      //   F0 C0 | F1(+G0) C1 B0 | F2(+G1) C2 B1 | ... | G_last B_last
      SBP_TRY(forward(0, 0, -1, 0));
      SBP_TRY(combine(0, 0));
      for (int64_t ci = 1; ci < L.n_chunks; ++ci) {
        const int b = (int)(ci & 1), pb = b ^ 1;
        SBP_TRY(forward(ci, b, ci - 1, pb));
        SBP_TRY(combine(ci, b));
        SBP_TRY(backward(ci - 1, pb));
      }
      const int64_t last = L.n_chunks - 1;
      if (last >= 0) {
        SBP_TRY(gradient(last, (int)(last & 1)));
        SBP_TRY(backward(last, (int)(last & 1)));
      }
    } else {
      for (int64_t ci = 0; ci < L.n_chunks; ++ci) {
        SBP_TRY(forward(ci, 0, -1, 0));
        SBP_TRY(combine(ci, 0));
        SBP_TRY(gradient(ci, 0));
        SBP_TRY(backward(ci, 0));
      }
    }

    if (c.mode == SBP_MODE_SFT || c.mode == SBP_MODE_GRPO) {
      k_loss_final<<<1, 1024, 0, s>>>(tokloss, c.T, nvalid, c.loss, c.n_valid);
      ++launches;
    } else if (c.mode == SBP_MODE_DPO1) {
      if (c.n_seq > 0) {
        k_seq_sums<<<c.n_seq, 256, 0, s>>>(logp, c.cu, c.seq_logp);
        ++launches;
      }
      if (c.n_valid) {
        k_loss_final<<<1, 1024, 0, s>>>(tokloss, 0, nvalid, nullptr, c.n_valid);
        ++launches;
      }
    }
    SBP_CUDA(cudaGetLastError());
    return SBP_OK;
  };
#undef SBP_TRY

  st = schedule();
  if (hio) {
    // join the side stream back into the caller's stream whatever happened above, so
    // that nothing of this call runs past it
    const cudaError_t e1 = cudaEventRecord(ss->join, ss->s);
    const cudaError_t e2 = cudaStreamWaitEvent(s, ss->join, 0);
    if (st == SBP_OK && (e1 != cudaSuccess || e2 != cudaSuccess)) st = SBP_ERR_CUDA;
    if (st == SBP_OK) st = guard_zones(ws, L.guards, 1, c.dev_status, s, &launches);
    if (st == SBP_OK) {
      SBP_CUDA(cudaMemcpyAsync(hio->loss, c.loss, sizeof(float), cudaMemcpyDeviceToHost, s));
      if (hio->n_valid)
        SBP_CUDA(cudaMemcpyAsync(hio->n_valid, c.n_valid, sizeof(int64_t), cudaMemcpyDeviceToHost, s));
    }
  }
  if (st != SBP_OK) return st;
  if (!hio) {
    st = guard_zones(ws, L.guards, 1, c.dev_status, s, &launches);
    if (st != SBP_OK) return st;
  }
  if (c.logp_out && c.T > 0)
    SBP_CUDA(cudaMemcpyAsync(c.logp_out, logp, (size_t)c.T * sizeof(float), cudaMemcpyDeviceToDevice, s));
  g_launches = launches;
  return SBP_OK;
}

// ------------------------------------------------------------------------- MLP sublayer

struct MlpLayout {
  int64_t chunk = 0, n_chunks = 0;
  int splits = 1;
  size_t off_gu = 0, off_a = 0, off_dhp = 0, off_cnt = 0, total = 0;
  Guards guards;   // checked build only
};

bool mlp_layout(int64_t T, int64_t d, int64_t f, int64_t chunk, MlpLayout* L) {
  if (T < 0 || d < 64 || f < 256 || d % 64 || f % 256 || chunk < 1 || chunk > 65535) return false;
  MlpLayout l;
  l.chunk = T > 0 ? (chunk < T ? chunk : T) : 1;
  l.n_chunks = T > 0 ? (T + l.chunk - 1) / l.chunk : 0;
  l.splits = choose_splits(l.chunk, d, 2 * f, num_sms());
  size_t o = 0;
  l.off_gu = take_region(o, (size_t)l.chunk * 2 * f * 2, l.guards);
  l.off_a = take_region(o, (size_t)l.chunk * f * 2, l.guards);
  l.off_dhp = take_region(o, (size_t)l.splits * l.chunk * d * sizeof(float), l.guards);
  l.off_cnt = take_region(o, (size_t)(2 * l.n_chunks + 1) * sizeof(uint32_t), l.guards);
  l.total = o;
  *L = l;
  return true;
}


int run_mlp(const void* X, const void* Wgu, const void* Wd, const void* dY, int64_t T, int64_t d, int64_t f,
            int64_t chunk, void* dX, float* dWgu, float* dWd, int accumulate, void* ws, size_t ws_bytes,
            int32_t* dev_status, cudaStream_t s) {
  MlpLayout L;
  if (!mlp_layout(T, d, f, chunk, &L)) return SBP_ERR_INVALID_ARG;
  if (!Wgu || !Wd || !dWgu || !dWd || !dev_status) return SBP_ERR_INVALID_ARG;
  if (T > 0 && (!X || !dY || !dX)) return SBP_ERR_INVALID_ARG;
  if (T > (int64_t)INT32_MAX) return SBP_ERR_UNSUPPORTED;
  for (const void* q : {X, Wgu, Wd, dY, (const void*)dX, (const void*)dWgu, (const void*)dWd})
    if (q && !al16(q)) return SBP_ERR_ALIGNMENT;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < L.total) return SBP_ERR_WORKSPACE;
  char* w = static_cast<char*>(ws);
  void* gu = w + L.off_gu;
  void* abuf = w + L.off_a;
  float* dhp = reinterpret_cast<float*>(w + L.off_dhp);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(w + L.off_cnt);
  int launches = 0;
  NvtxRange nv_call("sbp_mlp");
  SBP_CUDA(cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s));
  {
    const int gs = guard_zones(ws, L.guards, 0, dev_status, s, &launches);
    if (gs != SBP_OK) return gs;
  }
  SBP_CUDA(cudaMemsetAsync(cnt, 0, (size_t)(2 * L.n_chunks + 1) * sizeof(uint32_t), s));
  if (T == 0 && !accumulate) {
    k_zero_f32<<<grid_for(2 * f * d, 256), 256, 0, s>>>(dWgu, 2 * f * d);
    k_zero_f32<<<grid_for(d * f, 256), 256, 0, s>>>(dWd, d * f);
    launches += 2;
    SBP_CUDA(cudaGetLastError());
  }
  // dWd (+)= dY_c^T a_c needs only the chunk's a: it runs on the side stream beside the
  // chunk's da and dX GEMMs (fork after a is formed, join before the next chunk overwrites
  // a); the dWd launches stay in chunk order on that stream, so the sums keep their order
  SideStream* ss = T > 0 ? side_stream() : nullptr;
  std::unique_lock<std::mutex> lk;
  if (ss) lk = std::unique_lock<std::mutex>(ss->mu);
  cudaStream_t se = ss ? ss->s : s;
  int rc = SBP_OK;
#define MLP_CUDA(x)                                  \
  do {                                               \
    if ((x) != cudaSuccess) { rc = SBP_ERR_CUDA; break; } \
  } while (0)
  for (int64_t ci = 0; ci < L.n_chunks && rc == SBP_OK; ++ci) {
    const int64_t r0 = ci * L.chunk;
    const int rows = (int)((r0 + L.chunk <= T) ? L.chunk : T - r0);
    const int acc = (ci > 0 || accumulate) ? 1 : 0;
    if (ss && ci > 0 && cudaStreamWaitEvent(s, ss->join, 0) != cudaSuccess) { rc = SBP_ERR_CUDA; break; }
    {
      // recompute g, u and a = silu(g) u for the chunk, then dg | du in place
      prof::Scope ps(0, s);
      TcMlpArgs m{};
      m.Arows = X; m.T = T; m.d = d; m.f = f; m.B = Wgu; m.r0 = r0; m.rows = rows; m.Aout = abuf; m.GU = gu;
      m.status = dev_status;
      if (tc_mlp(m, false, s) != cudaSuccess) { rc = SBP_ERR_CUDA; break; }
      if (ss && (cudaEventRecord(ss->fork, s) != cudaSuccess || cudaStreamWaitEvent(se, ss->fork, 0) != cudaSuccess)) {
        rc = SBP_ERR_CUDA;
        break;
      }
      m.Arows = dY; m.B = Wd;
      if (tc_mlp(m, true, s) != cudaSuccess) { rc = SBP_ERR_CUDA; break; }
      launches += 2;
    }
    const int splits = std::min(choose_splits(rows, d, 2 * f, num_sms()), L.splits);
    {
      // dX_c = [dg du] [Wg; Wu] and [dWg; dWu] (+)= [dg du]^T x_c
      prof::Scope ps(1, s);
      TcBwdArgs b{};
      b.G = gu; b.ldg = 2 * f; b.H = X; b.W = Wgu; b.T = T; b.d = d; b.V = 2 * f; b.r0 = r0; b.rows = rows;
      b.splits = splits; b.dh_part = dhp; b.dW = dWgu; b.dw_accumulate = acc; b.counter = cnt + 2 * ci;
      b.status = dev_status;
      if (tc_backward(b, s) != cudaSuccess) { rc = SBP_ERR_CUDA; break; }
      ++launches;
    }
    {
      // dWd (+)= dY_c^T a_c : the dW units only, with M over d and N over f
      prof::Scope ps(1, se);
      TcBwdArgs e{};
      e.G = static_cast<const __nv_bfloat16*>(dY) + r0 * d; e.ldg = d; e.H = abuf; e.W = Wd; e.T = rows;
      e.d = f; e.V = d; e.r0 = 0; e.rows = rows; e.splits = 1; e.dh_part = dhp; e.dW = dWd;
      e.dw_accumulate = acc; e.counter = cnt + 2 * ci + 1; e.status = dev_status; e.dw_only = 1;
      if (tc_backward(e, se) != cudaSuccess) { rc = SBP_ERR_CUDA; break; }
      if (ss && cudaEventRecord(ss->join, se) != cudaSuccess) { rc = SBP_ERR_CUDA; break; }
      ++launches;
    }
    {
      prof::Scope ps(3, s);
      const int64_t n = (int64_t)rows * d;
      k_dh_reduce<__nv_bfloat16><<<grid_for(n / 4 + 1, 256), 256, 0, s>>>(
          dhp, splits, n, n, static_cast<__nv_bfloat16*>(dX) + r0 * d);
      ++launches;
      MLP_CUDA(cudaGetLastError());
    }
  }
#undef MLP_CUDA
  // join: the caller's stream waits for the last dWd (the side stream has waited on it for
  // every fork, so nothing of this call is left behind even after an error)
  if (ss && L.n_chunks > 0) {
    if (cudaEventRecord(ss->join, se) != cudaSuccess || cudaStreamWaitEvent(s, ss->join, 0) != cudaSuccess)
      rc = SBP_ERR_CUDA;
  }
  if (rc == SBP_OK) rc = guard_zones(ws, L.guards, 1, dev_status, s, &launches);
  if (rc != SBP_OK) return rc;
  g_launches = launches;
  return SBP_OK;
}

// ------------------------------------------------------------------ causal attention

// D[z, t] = dO[z, t, :] . O[z, t, :] (one warp per row)
__global__ void __launch_bounds__(256) k_attn_D(const __nv_bfloat16* __restrict__ O,
                                                const __nv_bfloat16* __restrict__ dO, int64_t rows, int64_t hd,
                                                float* __restrict__ D) {
  const int64_t r = (int64_t)blockIdx.x * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (r >= rows) return;
  float acc = 0.f;
  for (int64_t k = lane; k < hd; k += 32)
    acc += __bfloat162float(O[r * hd + k]) * __bfloat162float(dO[r * hd + k]);
  acc = warp_sum(acc);
  if (lane == 0) D[r] = acc;
}

// dQ rows of a chunk for every head: sum over the split-K partials [splits][H][rows][hd]
__global__ void __launch_bounds__(256) k_dq_reduce(const float* __restrict__ part, int splits, int H, int rows,
                                                   int64_t hd, int64_t T, int64_t c0, __nv_bfloat16* __restrict__ dQ) {
  const int z = blockIdx.y;
  const int64_t plane = (int64_t)rows * hd;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < plane; i += (int64_t)gridDim.x * blockDim.x) {
    float acc = 0.f;
    for (int s2 = 0; s2 < splits; ++s2) acc += part[((int64_t)s2 * H + z) * plane + i];
    dQ[((int64_t)z * T + c0) * hd + i] = __float2bfloat16_rn(acc);
  }
}

struct AttnLayout {
  int64_t chunk = 0, n_chunks = 0, Cmax = 0, Lp = 0;
  int splits = 1;
  bool fused = false;   // hd = 128: P and dS stay on chip, the workspace holds D only
  size_t off_p = 0, off_ds = 0, off_d = 0, off_dqp = 0, off_cnt = 0, total = 0;
  Guards guards;   // checked build only
};

int attn_splits(int64_t rows, int64_t hd, int64_t L, int H) {
  // dQ units are few (H x row pairs) but long (K = L); split them so that one stays below
  // a quarter of a pair's share of the launch
  const int64_t mt_c = (rows + 255) / 256, kb_v = (L + 63) / 64, mt_v = (L + 255) / 256, kb_c = (rows + 63) / 64;
  const double total = double(H) * double(mt_c * kb_v + mt_v * kb_c);
  const double per_pair = total / double(std::max(1, num_sms() / 2));
  int s = (int)std::ceil(4.0 * double(kb_v) / std::max(per_pair, 1.0));
  s = std::max(1, std::min(s, 8));
  return (int)std::min<int64_t>(s, kb_v);
}

bool attn_layout(int64_t H, int64_t T, int64_t hd, int64_t chunk, AttnLayout* L) {
  if (H < 1 || T < 0 || hd < 64 || hd > 256 || hd % 64 || chunk < 1 || chunk > 65535) return false;
  AttnLayout l;
  l.chunk = T > 0 ? std::min(chunk, T) : 1;
  l.n_chunks = T > 0 ? (T + l.chunk - 1) / l.chunk : 0;
  l.Cmax = ((l.chunk + 255) / 256) * 256;
  l.Lp = ((std::max<int64_t>(T, 1) + 255) / 256) * 256;
  l.splits = attn_splits(l.chunk, hd, std::max<int64_t>(T, 1), (int)H);
  l.fused = hd == 128;
  size_t o = 0;
  if (l.fused) {
    l.off_d = take_region(o, (size_t)H * std::max<int64_t>(T, 1) * sizeof(float), l.guards);
    l.total = o;
    *L = l;
    return true;
  }
  l.off_p = take_region(o, (size_t)H * l.Cmax * l.Lp * 2, l.guards);
  l.off_ds = take_region(o, (size_t)H * l.Cmax * l.Lp * 2, l.guards);
  l.off_d = take_region(o, (size_t)H * std::max<int64_t>(T, 1) * sizeof(float), l.guards);
  l.off_dqp = take_region(o, (size_t)l.splits * H * l.Cmax * hd * sizeof(float), l.guards);
  l.off_cnt = take_region(o, (size_t)(2 * l.n_chunks + 1) * sizeof(uint32_t), l.guards);
  l.total = o;
  *L = l;
  return true;
}

// hd = 128: per chunk, k_attn_kv (dK, dV of keys [0, c1)) on the caller's stream and
// k_attn_q (dQ of the chunk) on the side stream: the two families write disjoint outputs,
// so they may overlap (each fills the other's last, partly occupied wave); each family
// stays in chunk order on its own stream, so the results do not depend on the overlap
int run_attn_fused(const void* Q, const void* K, const void* Vv, const void* O, const void* dO, const float* lse,
                   int64_t H, int64_t Hkv, int64_t T, float scale, const AttnLayout& L, void* dQ, float* dK,
                   float* dV, int accumulate, char* w, int32_t* dev_status, cudaStream_t s) {
  const int64_t hd = 128;
  float* D = reinterpret_cast<float*>(w + L.off_d);
  int launches = 0;
  SBP_CUDA(cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s));
  if (!accumulate) {
    SBP_CUDA(cudaMemsetAsync(dK, 0, (size_t)Hkv * T * hd * sizeof(float), s));
    SBP_CUDA(cudaMemsetAsync(dV, 0, (size_t)Hkv * T * hd * sizeof(float), s));
  }
  if (T == 0) {
    g_launches = 0;
    return SBP_OK;
  }
  AttnFusedPlan plan;
  if (!plan.init(Q, K, Vv, dO, dK, dV, T, H, Hkv)) return SBP_ERR_CUDA;
  {
    prof::Scope ps(3, s);
    k_attn_D<<<(unsigned)((H * T + 7) / 8), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(O),
                                                       static_cast<const __nv_bfloat16*>(dO), H * T, hd, D);
    ++launches;
    SBP_CUDA(cudaGetLastError());
  }
  SideStream* ss = side_stream();
  std::unique_lock<std::mutex> lk;
  cudaStream_t sq = s;
  if (ss) {
    lk = std::unique_lock<std::mutex>(ss->mu);
    SBP_CUDA(cudaEventRecord(ss->fork, s));
    SBP_CUDA(cudaStreamWaitEvent(ss->s, ss->fork, 0));
    sq = ss->s;
  }
  // With one key / value head per query head, one k_attn_kv launch may cover a run of
  // consecutive chunks (up to kKvSpan queries): nothing of size (queries x keys) is stored
  // on this path, so the span changes no memory, and a unit (one head, 256 keys) then
  // walks more query blocks for each K / V load and dK / dV write-back.  A run is taken
  // only if its launch still has at least 4 units per SM pair.  Measured: merging 4
  // chunks of 1024 gave +2% with 32 heads at T = 8192; with grouped heads (units 4 times
  // longer and fewer) it lost 5% at T = 8192 and 3.5% at T = 32768, so grouped heads keep
  // one launch per chunk.  k_attn_q keeps the caller's chunks.  Both schedules are fixed
  // by the arguments, so the results stay bitwise repeatable.
  constexpr int64_t kKvSpan = 4096;
  const int64_t kv_max = Hkv == H ? std::max<int64_t>(1, kKvSpan / L.chunk) : 1;
  const int64_t min_units = 4 * std::max(1, num_sms() / 2);
  auto kv_units = [&](int64_t c1) { return ((c1 + 255) / 256) * Hkv; };
  int64_t kv_next = 0;   // first chunk no k_attn_kv launch has covered yet
  int rc = SBP_OK;
  for (int64_t ci = 0; ci < L.n_chunks && rc == SBP_OK; ++ci) {
    const int64_t c0 = ci * L.chunk, c1 = std::min(T, c0 + L.chunk);
    if (ci == kv_next) {
      int64_t e = ci + 1;   // this launch covers chunks [ci, e)
      for (int64_t f = std::min(L.n_chunks, ci + kv_max); f > ci + 1; --f)
        if (kv_units(std::min(T, f * L.chunk)) >= min_units) {
          e = f;
          break;
        }
      kv_next = e;
      prof::Scope ps(0, s);
      if (attn_fused_kv(plan, c0, std::min(T, e * L.chunk), scale, lse, D, dev_status, s) != cudaSuccess)
        rc = SBP_ERR_CUDA;
      ++launches;
    }
    if (rc != SBP_OK) break;
    {
      prof::Scope ps(1, sq);
      if (attn_fused_q(plan, c0, c1, scale, lse, D, dQ, dev_status, sq) != cudaSuccess) rc = SBP_ERR_CUDA;
      ++launches;
    }
  }
  if (ss) {   // join even after an error, so the caller's stream is never left behind
    if (cudaEventRecord(ss->join, sq) != cudaSuccess || cudaStreamWaitEvent(s, ss->join, 0) != cudaSuccess)
      rc = SBP_ERR_CUDA;
  }
  if (rc != SBP_OK) return rc;
  g_launches = launches;
  return SBP_OK;
}

int run_attn_chunks(const void* Q, const void* K, const void* Vv, const void* O, const void* dO, const float* lse,
                    int64_t H, int64_t T, int64_t hd, float scale, const AttnLayout& L, void* dQ, float* dK,
                    float* dV, int accumulate, char* w, int32_t* dev_status, cudaStream_t s);

int run_attn(const void* Q, const void* K, const void* Vv, const void* O, const void* dO, const float* lse,
             int64_t H, int64_t Hkv, int64_t T, int64_t hd, float scale, int64_t chunk, void* dQ, float* dK,
             float* dV, int accumulate, void* ws, size_t ws_bytes, int32_t* dev_status, cudaStream_t s) {
  AttnLayout L;
  if (!attn_layout(H, T, hd, chunk, &L)) return SBP_ERR_INVALID_ARG;
  if (Hkv < 1 || Hkv > H || H % Hkv != 0) return SBP_ERR_INVALID_ARG;
  if (Hkv != H && !L.fused) return SBP_ERR_UNSUPPORTED;   // grouped heads: head dimension 128 only
  if (!dev_status || !dK || !dV) return SBP_ERR_INVALID_ARG;
  if (T > 0 && (!Q || !K || !Vv || !O || !dO || !lse || !dQ)) return SBP_ERR_INVALID_ARG;
  if (H * T > (int64_t)INT32_MAX) return SBP_ERR_UNSUPPORTED;
  for (const void* q : {Q, K, Vv, O, dO, (const void*)lse, (const void*)dQ, (const void*)dK, (const void*)dV})
    if (q && !al16(q)) return SBP_ERR_ALIGNMENT;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < L.total) return SBP_ERR_WORKSPACE;
  char* w = static_cast<char*>(ws);
  NvtxRange nv_call("sbp_attn");
  int gl = 0;
  int rc = guard_zones(w, L.guards, 0, dev_status, s, &gl);
  if (rc != SBP_OK) return rc;
  rc = L.fused ? run_attn_fused(Q, K, Vv, O, dO, lse, H, Hkv, T, scale, L, dQ, dK, dV, accumulate, w, dev_status, s)
               : run_attn_chunks(Q, K, Vv, O, dO, lse, H, T, hd, scale, L, dQ, dK, dV, accumulate, w, dev_status, s);
  if (rc == SBP_OK) rc = guard_zones(w, L.guards, 1, dev_status, s, &gl);
  if (rc == SBP_OK) g_launches += gl;
  return rc;
}

// other head widths: per chunk, P and dS through chunk buffers in the workspace
int run_attn_chunks(const void* Q, const void* K, const void* Vv, const void* O, const void* dO, const float* lse,
                    int64_t H, int64_t T, int64_t hd, float scale, const AttnLayout& L, void* dQ, float* dK,
                    float* dV, int accumulate, char* w, int32_t* dev_status, cudaStream_t s) {
  void* pbuf = w + L.off_p;
  void* dsbuf = w + L.off_ds;
  float* D = reinterpret_cast<float*>(w + L.off_d);
  float* dqp = reinterpret_cast<float*>(w + L.off_dqp);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(w + L.off_cnt);
  int launches = 0;
  SBP_CUDA(cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s));
  SBP_CUDA(cudaMemsetAsync(cnt, 0, (size_t)(2 * L.n_chunks + 1) * sizeof(uint32_t), s));
  if (!accumulate) {   // every chunk adds into dK and dV rows [0, L)
    SBP_CUDA(cudaMemsetAsync(dK, 0, (size_t)H * T * hd * sizeof(float), s));
    SBP_CUDA(cudaMemsetAsync(dV, 0, (size_t)H * T * hd * sizeof(float), s));
  }
  if (T == 0) {
    g_launches = 0;
    return SBP_OK;
  }
  {
    prof::Scope ps(3, s);
    k_attn_D<<<(unsigned)((H * T + 7) / 8), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(O),
                                                       static_cast<const __nv_bfloat16*>(dO), H * T, hd, D);
    ++launches;
    SBP_CUDA(cudaGetLastError());
  }
  for (int64_t ci = 0; ci < L.n_chunks; ++ci) {
    const int64_t c0 = ci * L.chunk;
    const int rows = (int)((c0 + L.chunk <= T) ? L.chunk : T - c0);
    const int64_t Lk = c0 + rows;   // keys of this chunk's queries
    {
      prof::Scope ps(0, s);
      TcAttnArgs a{};
      a.A = Q; a.B = K; a.T = T; a.hd = hd; a.H = (int)H; a.c0 = c0; a.rows = rows; a.scale = scale;
      a.lse = lse; a.D = D; a.P = pbuf; a.dS = dsbuf; a.Cmax = L.Cmax; a.Lp = L.Lp; a.status = dev_status;
      SBP_CUDA(tc_attn(a, false, s));
      a.A = dO; a.B = Vv;
      SBP_CUDA(tc_attn(a, true, s));
      launches += 2;
    }
    const int splits = std::min(attn_splits(rows, hd, Lk, (int)H), L.splits);
    {
      prof::Scope ps(1, s);
      // dQ_c = dS K (dH units) and dK[:Lk] += dS^T Q_c (dW units), every head
      TcBwdArgs b{};
      b.G = dsbuf; b.ldg = L.Lp; b.g_rows = H * L.Cmax; b.zr_g = (int)L.Cmax;
      b.W = K; b.w_rows = H * T; b.zr_w = (int)T;
      b.H = Q; b.h_rows = H * T; b.zr_h = (int)T; b.T = T; b.r0 = c0;
      b.dW = dK; b.dw_rows = H * T; b.zr_dw = (int)T;
      b.d = hd; b.V = Lk; b.rows = rows; b.batch = (int)H;
      b.splits = splits; b.dh_part = dqp; b.dw_accumulate = 1; b.counter = cnt + 2 * ci; b.status = dev_status;
      SBP_CUDA(tc_backward(b, s));
      // dV[:Lk] += P^T dO_c (dW units only)
      TcBwdArgs e = b;
      e.G = pbuf; e.H = dO; e.dW = dV; e.dw_only = 1; e.counter = cnt + 2 * ci + 1;
      SBP_CUDA(tc_backward(e, s));
      launches += 2;
    }
    {
      prof::Scope ps(3, s);
      dim3 g((unsigned)std::min<int64_t>(((int64_t)rows * hd + 255) / 256, 1024), (unsigned)H);
      k_dq_reduce<<<g, 256, 0, s>>>(dqp, splits, (int)H, rows, hd, T, c0, static_cast<__nv_bfloat16*>(dQ));
      ++launches;
      SBP_CUDA(cudaGetLastError());
    }
  }
  g_launches = launches;
  return SBP_OK;
}

}  // namespace

// Scratch of sbp_lmhead_sft_noalloc: a fixed device array in this module, so that
// callers without an allocator can still run the chunked LM head.  Every GPU that
// loads the library holds it until the process exits; all calls share it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SBP_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once per
// device (cudaGetSymbolAddress, with that device current) and cached.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SBP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SBP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SBP_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return SBP_OK;
}
}  // namespace
}  // namespace sbp

using namespace sbp;

extern "C" {

size_t sbp_lmhead_workspace_bytes(int64_t T, int64_t d, int64_t V, int64_t chunk, int dtype, int mode) {
  Layout L;
  if (!make_layout(T, d, V, chunk, dtype, mode, &L)) return 0;
  return L.total;
}

size_t sbp_lmhead_workspace_bytes_lean(int64_t T, int64_t d, int64_t V, int64_t chunk, int dtype, int mode) {
  Layout L;
  if (!make_layout(T, d, V, chunk, dtype, mode, &L, 1)) return 0;
  return L.total;
}

int sbp_lmhead_sft(const void* H, const void* W, const int32_t* labels, int64_t T, int64_t d, int64_t V,
                   int64_t chunk, int32_t ignore_index, int dtype, float* loss, int64_t* n_valid,
                   float* logp_out, void* dH, float* dW, int accumulate_dW, void* workspace, size_t ws_bytes,
                   int32_t* dev_status, void* stream) {
  if (!loss) return SBP_ERR_INVALID_ARG;
  Call c{};
  c.mode = SBP_MODE_SFT; c.H = H; c.W = W; c.labels = labels; c.T = T; c.d = d; c.V = V; c.chunk = chunk;
  c.ign = ignore_index; c.dtype = dtype; c.loss = loss; c.n_valid = n_valid; c.logp_out = logp_out;
  c.dH = dH; c.dW = dW; c.accumulate_dW = accumulate_dW; c.ws = workspace; c.ws_bytes = ws_bytes;
  c.dev_status = dev_status; c.stream = static_cast<cudaStream_t>(stream);
  return run(c);
}

int sbp_lmhead_grpo(const void* H, const void* W, const int32_t* labels, const float* advantages,
                    const float* logp_old, float clip_lo, float clip_hi, int64_t T, int64_t d, int64_t V,
                    int64_t chunk, int32_t ignore_index, int dtype, float* loss, int64_t* n_valid,
                    float* logp_out, void* dH, float* dW, int accumulate_dW, void* workspace, size_t ws_bytes,
                    int32_t* dev_status, void* stream) {
  if (!loss) return SBP_ERR_INVALID_ARG;
  Call c{};
  c.mode = SBP_MODE_GRPO; c.H = H; c.W = W; c.labels = labels; c.T = T; c.d = d; c.V = V; c.chunk = chunk;
  c.ign = ignore_index; c.dtype = dtype; c.loss = loss; c.n_valid = n_valid; c.logp_out = logp_out;
  c.dH = dH; c.dW = dW; c.accumulate_dW = accumulate_dW; c.adv = advantages; c.logp_old = logp_old;
  c.clip_lo = clip_lo; c.clip_hi = clip_hi; c.ws = workspace; c.ws_bytes = ws_bytes;
  c.dev_status = dev_status; c.stream = static_cast<cudaStream_t>(stream);
  return run(c);
}

int sbp_lmhead_grpo_ext(const void* H, const void* W, const int32_t* labels, const float* advantages,
                        const float* logp_old, float clip_lo, float clip_hi, const float* ref_logp, float kl_coef,
                        const int32_t* cu_seqlens, int32_t n_seq, int64_t T, int64_t d, int64_t V, int64_t chunk,
                        int32_t ignore_index, int dtype, float* loss, int64_t* n_valid, float* logp_out, void* dH,
                        float* dW, int accumulate_dW, void* workspace, size_t ws_bytes, int32_t* dev_status,
                        void* stream) {
  if (!loss) return SBP_ERR_INVALID_ARG;
  Call c{};
  c.mode = SBP_MODE_GRPO; c.H = H; c.W = W; c.labels = labels; c.T = T; c.d = d; c.V = V; c.chunk = chunk;
  c.ign = ignore_index; c.dtype = dtype; c.loss = loss; c.n_valid = n_valid; c.logp_out = logp_out;
  c.dH = dH; c.dW = dW; c.accumulate_dW = accumulate_dW; c.adv = advantages; c.logp_old = logp_old;
  c.clip_lo = clip_lo; c.clip_hi = clip_hi; c.ref_logp = ref_logp; c.kl_coef = kl_coef;
  c.cu = cu_seqlens; c.n_seq = cu_seqlens ? n_seq : 0;
  c.ws = workspace; c.ws_bytes = ws_bytes; c.dev_status = dev_status; c.stream = static_cast<cudaStream_t>(stream);
  return run(c);
}

int sbp_lmhead_dpo_pass1(const void* H, const void* W, const int32_t* labels, const int32_t* cu_seqlens,
                         int32_t n_seq, int64_t T, int64_t d, int64_t V, int64_t chunk, int32_t ignore_index,
                         int dtype, double* seq_logp, float* logp_out, int64_t* n_valid, void* workspace,
                         size_t ws_bytes, int32_t* dev_status, void* stream) {
  Call c{};
  c.mode = SBP_MODE_DPO1; c.H = H; c.W = W; c.labels = labels; c.T = T; c.d = d; c.V = V; c.chunk = chunk;
  c.ign = ignore_index; c.dtype = dtype; c.cu = cu_seqlens; c.n_seq = n_seq; c.seq_logp = seq_logp;
  c.logp_out = logp_out; c.n_valid = n_valid; c.ws = workspace; c.ws_bytes = ws_bytes;
  c.dev_status = dev_status; c.stream = static_cast<cudaStream_t>(stream);
  return run(c);
}

int sbp_lmhead_dpo_pass2(const void* H, const void* W, const int32_t* labels, const int32_t* cu_seqlens,
                         int32_t n_seq, const double* seq_logp, const double* ref_seq_logp, float beta,
                         int64_t T, int64_t d, int64_t V, int64_t chunk, int32_t ignore_index, int dtype,
                         float* loss, double* margins, void* dH, float* dW, int accumulate_dW,
                         void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream) {
  if (!loss) return SBP_ERR_INVALID_ARG;
  Call c{};
  c.mode = SBP_MODE_DPO2; c.H = H; c.W = W; c.labels = labels; c.T = T; c.d = d; c.V = V; c.chunk = chunk;
  c.ign = ignore_index; c.dtype = dtype; c.cu = cu_seqlens; c.n_seq = n_seq; c.seq_in = seq_logp;
  c.ref_in = ref_seq_logp; c.beta = beta; c.loss = loss; c.margins = margins; c.dH = dH; c.dW = dW;
  c.accumulate_dW = accumulate_dW; c.ws = workspace; c.ws_bytes = ws_bytes; c.dev_status = dev_status;
  c.stream = static_cast<cudaStream_t>(stream);
  return run(c);
}

int sbp_lmhead_sft_noalloc(const void* H, const void* W, const int32_t* labels, int64_t T, int64_t d, int64_t V,
                           int64_t chunk, int32_t ignore_index, int dtype, float* loss, int64_t* n_valid,
                           float* logp_out, void* dH, float* dW, int accumulate_dW, int32_t* dev_status,
                           void* stream) {
  if (!loss) return SBP_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(T, d, V, chunk, dtype, SBP_MODE_SFT, &L, 1)) return SBP_ERR_INVALID_ARG;
  if (L.total > (size_t)SBP_NOALLOC_SCRATCH_BYTES) return SBP_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const int st = noalloc_scratch(&scratch);
  if (st != SBP_OK) return st;
  Call c{};
  c.mode = SBP_MODE_SFT; c.H = H; c.W = W; c.labels = labels; c.T = T; c.d = d; c.V = V; c.chunk = chunk;
  c.ign = ignore_index; c.dtype = dtype; c.loss = loss; c.n_valid = n_valid; c.logp_out = logp_out;
  c.dH = dH; c.dW = dW; c.accumulate_dW = accumulate_dW; c.ws = scratch;
  c.ws_bytes = (size_t)SBP_NOALLOC_SCRATCH_BYTES; c.dev_status = dev_status;
  c.stream = static_cast<cudaStream_t>(stream);
  c.nbuf = 1;   // one buffer set: the gradient of each chunk runs as its own pass
  return run(c);
}

size_t sbp_lmhead_sft_host_workspace_bytes(int64_t T, int64_t d, int64_t V, int64_t chunk, int dtype) {
  Layout L;
  if (!make_layout(T, d, V, chunk, dtype, SBP_MODE_SFT, &L, 0, true)) return 0;
  return L.total;
}

int sbp_lmhead_sft_host(const void* H_host, const void* W, const int32_t* labels_host, int64_t T, int64_t d,
                        int64_t V, int64_t chunk, int32_t ignore_index, int dtype, float* loss_host,
                        int64_t* n_valid_host, void* dH_host, float* dW, int accumulate_dW, void* workspace,
                        size_t ws_bytes, int32_t* dev_status, void* stream) {
  const HostIO io{H_host, labels_host, dH_host, loss_host, n_valid_host};
  Call c{};
  c.mode = SBP_MODE_SFT; c.W = W; c.T = T; c.d = d; c.V = V; c.chunk = chunk; c.ign = ignore_index;
  c.dtype = dtype; c.dW = dW; c.accumulate_dW = accumulate_dW; c.ws = workspace; c.ws_bytes = ws_bytes;
  c.dev_status = dev_status; c.stream = static_cast<cudaStream_t>(stream); c.host = &io;
  return run(c);
}

size_t sbp_mlp_workspace_bytes(int64_t T, int64_t d, int64_t f, int64_t chunk) {
  MlpLayout L;
  if (!mlp_layout(T, d, f, chunk, &L)) return 0;
  return L.total;
}

int sbp_mlp_swiglu_backward(const void* X, const void* Wgu, const void* Wd, const void* dY, int64_t T, int64_t d,
                            int64_t f, int64_t chunk, void* dX, float* dWgu, float* dWd, int accumulate,
                            void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream) {
  return run_mlp(X, Wgu, Wd, dY, T, d, f, chunk, dX, dWgu, dWd, accumulate, workspace, ws_bytes, dev_status,
                 static_cast<cudaStream_t>(stream));
}

size_t sbp_attn_workspace_bytes(int64_t H, int64_t T, int64_t hd, int64_t chunk) {
  AttnLayout L;
  if (!attn_layout(H, T, hd, chunk, &L)) return 0;
  return L.total;
}

int sbp_attn_causal_backward(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                             const float* lse, int64_t H, int64_t T, int64_t hd, float scale, int64_t chunk,
                             void* dQ, float* dK, float* dV, int accumulate, void* workspace, size_t ws_bytes,
                             int32_t* dev_status, void* stream) {
  return run_attn(Q, K, V, O, dO, lse, H, H, T, hd, scale, chunk, dQ, dK, dV, accumulate, workspace, ws_bytes,
                  dev_status, static_cast<cudaStream_t>(stream));
}

int sbp_attn_causal_backward_gqa(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                                 const float* lse, int64_t H, int64_t Hkv, int64_t T, int64_t hd, float scale,
                                 int64_t chunk, void* dQ, float* dK, float* dV, int accumulate, void* workspace,
                                 size_t ws_bytes, int32_t* dev_status, void* stream) {
  return run_attn(Q, K, V, O, dO, lse, H, Hkv, T, hd, scale, chunk, dQ, dK, dV, accumulate, workspace, ws_bytes,
                  dev_status, static_cast<cudaStream_t>(stream));
}

const char* sbp_status_string(int status) {
  switch (status) {
    case SBP_OK: return "SBP_OK";
    case SBP_ERR_INVALID_ARG: return "SBP_ERR_INVALID_ARG";
    case SBP_ERR_ALIGNMENT: return "SBP_ERR_ALIGNMENT";
    case SBP_ERR_WORKSPACE: return "SBP_ERR_WORKSPACE";
    case SBP_ERR_LABEL_RANGE: return "SBP_ERR_LABEL_RANGE";
    case SBP_ERR_TIMEOUT: return "SBP_ERR_TIMEOUT";
    case SBP_ERR_CUDA: return "SBP_ERR_CUDA";
    case SBP_ERR_UNSUPPORTED: return "SBP_ERR_UNSUPPORTED";
    case SBP_ERR_SCRATCH_LIMIT: return "SBP_ERR_SCRATCH_LIMIT";
    case SBP_ERR_WORKSPACE_OVERRUN: return "SBP_ERR_WORKSPACE_OVERRUN";
    default: return "SBP_ERR_UNKNOWN";
  }
}

int sbp_last_launch_count(void) { return g_launches; }

int sbp_profile_enable(int on) {
  prof::g_on = on != 0;
  return SBP_OK;
}

int sbp_profile_read(double* ms, int64_t* launches, int n) {
  if (!prof::g_pairs) return 0;
  int cnt = 0;
  int err = 0;
  for (auto& p : *prof::g_pairs) {
    float t = 0.f;
    if (cudaEventSynchronize(p.b) != cudaSuccess || cudaEventElapsedTime(&t, p.a, p.b) != cudaSuccess) err = 1;
    if (p.cls < n && p.cls < prof::kClasses) {
      if (ms) ms[p.cls] += (double)t;
      if (launches) launches[p.cls] += 1;
    }
    if (!prof::g_pool) prof::g_pool = new std::vector<cudaEvent_t>();
    prof::g_pool->push_back(p.a);
    prof::g_pool->push_back(p.b);
    ++cnt;
  }
  prof::g_pairs->clear();
  return err ? -SBP_ERR_CUDA : cnt;
}

}  // extern "C"
