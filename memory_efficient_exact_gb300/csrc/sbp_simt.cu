// fp32 path of the LM head: SIMT FMA kernels (no TF32: fp32 inputs are held to
// fp32 accuracy).  Used for SBP_FP32 calls; the bf16 path runs on tcgen05.
#include <cfloat>
#include <cuda_runtime.h>

#include "sbp_internal.h"

namespace sbp {
namespace {

constexpr int GBM = 64, GBN = 64, GBK = 16;

// C[m, n] (+)= sum_k A(m, k) B(n, k), arbitrary element strides; 64x64 tile per block,
// 4x4 outputs per thread, fp32 accumulation.
__global__ void __launch_bounds__(256) k_gemm_f32(int64_t M, int64_t N, int64_t K,
                                                  const float* __restrict__ A, int64_t sam, int64_t sak,
                                                  const float* __restrict__ B, int64_t sbn, int64_t sbk,
                                                  float* __restrict__ C, int64_t ldc, int accumulate) {
  __shared__ float As[GBK][GBM + 4];
  __shared__ float Bs[GBK][GBN + 4];
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  const int64_t m0 = (int64_t)blockIdx.y * GBM, n0 = (int64_t)blockIdx.x * GBN;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int64_t k0 = 0; k0 < K; k0 += GBK) {
    for (int i = tid; i < GBM * GBK; i += 256) {
      int mm, kk;
      if (sak == 1) { kk = i % GBK; mm = i / GBK; } else { mm = i % GBM; kk = i / GBM; }
      const int64_t gm = m0 + mm, gk = k0 + kk;
      As[kk][mm] = (gm < M && gk < K) ? A[gm * sam + gk * sak] : 0.f;
    }
    for (int i = tid; i < GBN * GBK; i += 256) {
      int nn, kk;
      if (sbk == 1) { kk = i % GBK; nn = i / GBK; } else { nn = i % GBN; kk = i / GBN; }
      const int64_t gn = n0 + nn, gk = k0 + kk;
      Bs[kk][nn] = (gn < N && gk < K) ? B[gn * sbn + gk * sbk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < GBK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t gn = n0 + tx * 4 + j;
      if (gn >= N) continue;
      float* c = C + gm * ldc + gn;
      *c = accumulate ? *c + acc[i][j] : acc[i][j];
    }
  }
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

// One block of kStatW threads per (tile, row): the tile's max m, e = exp(z - m) written
// over z, s = sum e less the maximum's own term 1, and the label's logit gathered when
// it falls in the tile.
__global__ void __launch_bounds__(kStatW) k_tile_stats_f32(float* __restrict__ E, int64_t lde, int64_t V,
                                                           int64_t ntiles, const int32_t* __restrict__ labels,
                                                           float2* __restrict__ part, float* __restrict__ zy) {
  __shared__ float red[kStatW / 32], cnt[kStatW / 32];
  const int64_t row = blockIdx.y, tile = blockIdx.x;
  const int64_t col = tile * kStatW + threadIdx.x;
  const int lane = threadIdx.x % 32, wid = threadIdx.x / 32;
  float* e = E + row * lde;
  const float z = col < V ? e[col] : -FLT_MAX;
  float m = warp_max(z);
  if (lane == 0) red[wid] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int i = 1; i < kStatW / 32; ++i) m = fmaxf(m, red[i]);
  __syncthreads();
  const float x = col < V ? expf(z - m) : 0.f;
  if (col < V) e[col] = x;
  // the tile's sum less the term of one maximum (exactly 1); the other maxima count 1
  const bool top = col < V && z == m;
  float s = warp_sum(top ? 0.f : x);
  float c = warp_sum(top ? 1.f : 0.f);
  if (lane == 0) {
    red[wid] = s;
    cnt[wid] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    s = 0.f;
    c = -1.f;
#pragma unroll
    for (int i = 0; i < kStatW / 32; ++i) {
      s += red[i];
      c += cnt[i];
    }
    part[row * ntiles + tile] = make_float2(m, s + c);
  }
  if (col < V && labels[row] == (int32_t)col) zy[row] = z;
}

}  // namespace

cudaError_t simt_forward(const float* H, const float* W, int64_t d, int64_t V, int64_t r0, int rows,
                         const int32_t* labels, int32_t /*ign*/, float* E, int64_t lde, float2* part,
                         float* zy, bool /*store_e*/, cudaStream_t s) {
  dim3 g1((unsigned)((V + GBN - 1) / GBN), (unsigned)((rows + GBM - 1) / GBM));
  k_gemm_f32<<<g1, 256, 0, s>>>(rows, V, d, H + r0 * d, d, 1, W, d, 1, E, lde, 0);
  const int64_t ntiles = (V + kStatW - 1) / kStatW;
  dim3 g2((unsigned)ntiles, (unsigned)rows);
  k_tile_stats_f32<<<g2, kStatW, 0, s>>>(E, lde, V, ntiles, labels, part, zy);
  return cudaGetLastError();
}

cudaError_t simt_backward(const float* G, int64_t ldg, const float* H, const float* W, int64_t d,
                          int64_t V, int64_t r0, int rows, float* dh_part, float* dW,
                          int dw_accumulate, cudaStream_t s) {
  // dH_c = G_c W : M = rows, N = d, K = V
  dim3 g1((unsigned)((d + GBN - 1) / GBN), (unsigned)((rows + GBM - 1) / GBM));
  k_gemm_f32<<<g1, 256, 0, s>>>(rows, d, V, G, ldg, 1, W, 1, d, dh_part, d, 0);
  // dW (+)= G_c^T H_c : M = V, N = d, K = rows
  dim3 g2((unsigned)((d + GBN - 1) / GBN), (unsigned)((V + GBM - 1) / GBM));
  k_gemm_f32<<<g2, 256, 0, s>>>(V, d, rows, G, 1, ldg, H + r0 * d, 1, d, dW, d, dw_accumulate);
  return cudaGetLastError();
}

}  // namespace sbp
