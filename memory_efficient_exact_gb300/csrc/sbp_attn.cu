// Tensor-core kernels of the chunked causal-attention backward (bf16, sm_103a).
//
// For a chunk of queries [c0, c0 + rows) the keys [0, L), L = c0 + rows, are all it
// touches (the causal structure StreamBP uses).  Two pair GEMMs per chunk, batched over
// the heads (problem z = head; rows of head z start at z * T in Q, K, V, O, dO):
//   k_attn<false>  S = Q_c K^T;  epilogue P = exp(s S - lse_t) for keys j <= t, else 0
//   k_attn<true>   dP = dO_c V^T; epilogue dS = s P (dP - D_t), D_t = dO_t . O_t
// Both write bf16 [H, Cmax, Lp] chunk buffers (zero in the rows past the chunk, which
// the weight-gradient GEMMs read); dQ, dK and dV then come from k_bwd.  Same pair
// protocol, warp roles and bounded waits as the other tensor-core kernels.
#include "sbp_tc_common.cuh"

namespace sbp {
namespace tc {

struct AttnP {
  int64_t T; int H;
  int64_t c0; int rows; int64_t L;
  int mt, ntn, kb;
  float scale;
  const float* lse;        // [H, T]
  const float* D;          // [H, T]
  __nv_bfloat16* P;        // [H, Cmax, Lp]
  __nv_bfloat16* dS;       // [H, Cmax, Lp]
  int64_t Cmax, Lp;
  int32_t* status; uint64_t limit_ns;
};

// P and dS leave through one 32 x 64 bf16 staging block per epilogue warp and TMA stores
// (k_attn<true> reads P back the same way, by TMA loads completing on a per-warp
// mbarrier): row-per-thread global accesses were measured to starve the operand loads.
constexpr uint32_t STG_ATTN = 32 * 64 * 2;
constexpr size_t SMEM_ATTN =
    STAGES * STAGE_BYTES + NUM_EPI_WARPS * STG_ATTN + sizeof(Ctrl) + NUM_EPI_WARPS * sizeof(uint64_t) + 1024;
static_assert(SMEM_ATTN <= 232448, "shared memory budget of one CTA");
constexpr uint32_t IDESC_ATTN = idesc_bf16(256, 256, false, false);

template <bool DS>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    k_attn(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
           const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmDS, const AttnP p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stg_base = base + STAGES * STAGE_BYTES;
  Ctrl* c = reinterpret_cast<Ctrl*>(stg_base + NUM_EPI_WARPS * STG_ATTN);
  uint64_t* lbar = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(c) + sizeof(Ctrl));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = ctarank();
  prologue(c, warp);
  const uint32_t tmem = c->tmem_base;
  const int per_head = p.mt * p.ntn;
  const int total = per_head * p.H;
  const int pid = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_map(&tmA);
      prefetch_map(&tmB);
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_phase[STAGES] = {0, 0, 0, 0, 0, 0};
      bool ok = true;
      for (int tile = pid; tile < total && ok; tile += npairs) {
        const int z = tile / per_head, rem = tile % per_head;
        const int mp = rem % p.mt, nb = rem / p.mt;
        const int arow = (int)(z * p.T + p.c0 + (int64_t)mp * 256 + rank * 128);
        const int brow = (int)(z * p.T + (int64_t)nb * BN + rank * 128);
        for (int kb = 0; kb < p.kb; ++kb) {
          if (!wait_bounded(&c->empty[stage], phase ^ 1u, &c->abort, p.limit_ns)) { ok = false; break; }
          const uint32_t sa = saddr(base + stage * STAGE_BYTES), sb = sa + A_BYTES;
          const uint32_t fb = mapa(saddr(&c->full[stage]), 0);
          if (rank == 0) mbar_expect_tx(&c->full[stage], PAIR_TX);
          tma_load_2d_pair(sa, &tmA, fb, kb * BK, arow);
          tma_load_2d_pair(sb, &tmB, fb, kb * BK, brow);
          issued |= 1u << stage;
          last_phase[stage] = phase;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        fail(c, p.status);
        if (rank == 0) drain_copies(c, last_phase, issued);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      int stage = 0, local = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = pid; tile < total && ok; tile += npairs, ++local) {
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!wait_cluster(&c->tempty[buf], (use & 1u) ^ 1u, &c->abort, p.limit_ns)) { ok = false; break; }
        tc_fence_after();
        const uint32_t dt = tmem + (uint32_t)(buf * BN);
        for (int kb = 0; kb < p.kb; ++kb) {
          if (!wait_bounded(&c->full[stage], phase, &c->abort, p.limit_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = saddr(base + stage * STAGE_BYTES), sb = sa + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma2_bf16(dt, sw128_desc(sa + k * 32, 16, 1024), sw128_desc(sb + k * 32, 16, 1024), IDESC_ATTN,
                      (kb | k) != 0);
          commit2_mc(&c->empty[stage], 3);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        commit2_mc(&c->tfull[buf], 3);
      }
      if (!ok) fail(c, p.status);
      commit2_mc(&c->mdone, 1);
      wait_bounded(&c->mdone, 0, nullptr, 200000000ull);
    }
    __syncwarp();
  } else {
    const int q = warp & 3, h = (warp - 2) >> 2;
    const int lrow = q * 32 + lane;
    const float sl2 = p.scale * L2E;
    const uint32_t stg = saddr(stg_base + (warp - 2) * STG_ATTN);
    uint64_t* bar = lbar + (warp - 2);
    uint32_t lphase = 0;
    if (DS) {
      if (lane == 0) {
        mbar_init(bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      }
      __syncwarp();
    }
    int local = 0;
    bool ok = true;
    for (int tile = pid; tile < total && ok; tile += npairs, ++local) {
      const int z = tile / per_head, rem = tile % per_head;
      const int mp = rem % p.mt, nb = rem / p.mt;
      const int buf = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      const int row = mp * 256 + (int)rank * 128 + lrow;   // within the chunk (< Cmax)
      if (!warp_wait_cluster(&c->tfull[buf], use & 1u, c, p.limit_ns)) {
        fail(c, p.status);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + h * 128);
      __syncwarp();
      const int64_t j0 = (int64_t)nb * BN + h * 128;        // first key of this thread's 128
      const int yrow = (int)(z * p.Cmax) + mp * 256 + (int)rank * 128 + q * 32;   // the warp's first row
      const bool vrow = row < p.rows;                        // padding rows are written as zero
      const int64_t t = p.c0 + row;                          // query position
      const float lz = (!DS && vrow) ? p.lse[z * p.T + t] * L2E : 0.f;
      const float Dt = (DS && vrow) ? p.D[z * p.T + t] : 0.f;
#pragma unroll
      for (int bx = 0; bx < 2; ++bx) {   // two 64-key blocks of the warp's 128
        uint32_t r[2][32];
        tmem_ld32(tb + 64 * bx, r[0]);
        tmem_ld32(tb + 64 * bx + 32, r[1]);
        tmem_ld_wait();
        if (bx == 1) release_tmem(c, buf, lane);
        stage_free(lane);
        uint32_t pin[32];
        if (DS) {
          if (!stage_load(&tmP, stg, STG_ATTN, bar, lphase, lane, (int)(j0 + 64 * bx), yrow, c, p.limit_ns)) {
            fail(c, p.status);
            ok = false;
            break;
          }
          stage_read_row(stg, lane, pin);
          __syncwarp();
        }
#pragma unroll
        for (int gg = 0; gg < 2; ++gg) {
          const int g = 2 * bx + gg;
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float v0 = 0.f, v1 = 0.f;
            if (vrow) {
              if (!DS) {
                const int64_t key = j0 + g * 32 + j;
                v0 = key <= t ? ex2(fmaf(__uint_as_float(r[gg][j]), sl2, -lz)) : 0.f;
                v1 = key + 1 <= t ? ex2(fmaf(__uint_as_float(r[gg][j + 1]), sl2, -lz)) : 0.f;
              } else {
                const __nv_bfloat162 pb = *reinterpret_cast<const __nv_bfloat162*>(&pin[16 * gg + j / 2]);
                const float2 pp = __bfloat1622float2(pb);
                v0 = p.scale * pp.x * (__uint_as_float(r[gg][j]) - Dt);
                v1 = p.scale * pp.y * (__uint_as_float(r[gg][j + 1]) - Dt);
              }
            }
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(v0, v1);
            pk[j / 2] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          stage4(stg, lane, 4 * gg, pk);
        }
        stage_store(DS ? &tmDS : &tmP, stg, lane, (int)(j0 + 64 * bx), yrow);
      }
    }
    if (lane == 0) bulk_wait_all();   // every block has left shared memory and landed
    __syncwarp();
  }
  teardown(c, warp);
}

}  // namespace tc

cudaError_t tc_attn(const TcAttnArgs& a, bool ds, cudaStream_t s) {
  using namespace tc;
  static int attr_state[64] = {};
  static std::mutex mu;
  if (!once_per_device(attr_state, mu, [] {
        return cudaFuncSetAttribute(k_attn<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ATTN) ==
                   cudaSuccess &&
               cudaFuncSetAttribute(k_attn<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ATTN) ==
                   cudaSuccess;
      }))
    return cudaErrorInvalidConfiguration;
  // A: Q or dO, B: K or V, all [H * T, hd] row-major; boxes of 64 (hd) x 128 rows
  CUtensorMap mA, mB;
  const uint64_t rows_all = (uint64_t)a.H * (uint64_t)a.T;
  if (!make_map(&mA, a.A, (uint64_t)a.hd, rows_all, (uint64_t)a.hd, BK, 128)) return cudaErrorInvalidValue;
  if (!make_map(&mB, a.B, (uint64_t)a.hd, rows_all, (uint64_t)a.hd, BK, 128)) return cudaErrorInvalidValue;
  AttnP p;
  p.T = a.T; p.H = a.H; p.c0 = a.c0; p.rows = a.rows; p.L = a.c0 + a.rows;
  p.mt = (a.rows + 255) / 256;
  p.ntn = (int)((p.L + BN - 1) / BN);
  p.kb = (int)((a.hd + BK - 1) / BK);
  p.scale = a.scale;
  p.lse = a.lse; p.D = a.D;
  p.P = static_cast<__nv_bfloat16*>(a.P); p.dS = static_cast<__nv_bfloat16*>(a.dS);
  p.Cmax = a.Cmax; p.Lp = a.Lp;
  p.status = a.status; p.limit_ns = wait_limit_ns();
  const int total = p.mt * p.ntn * p.H;
  // P and dS: [H * Cmax, Lp] bf16, 64 x 32 blocks
  CUtensorMap mP, mDS;
  const uint64_t prow = (uint64_t)a.H * (uint64_t)a.Cmax;
  if (!make_map(&mP, a.P, (uint64_t)a.Lp, prow, (uint64_t)a.Lp, 64, 32)) return cudaErrorInvalidValue;
  if (!make_map(&mDS, a.dS, (uint64_t)a.Lp, prow, (uint64_t)a.Lp, 64, 32)) return cudaErrorInvalidValue;
  const void* kern = ds ? (const void*)k_attn<true> : (const void*)k_attn<false>;
  int pairs = max_pairs(kern, SMEM_ATTN);
  if (pairs > total) pairs = total;
  if (ds) k_attn<true><<<2 * pairs, NUM_THREADS, SMEM_ATTN, s>>>(mA, mB, mP, mDS, p);
  else k_attn<false><<<2 * pairs, NUM_THREADS, SMEM_ATTN, s>>>(mA, mB, mP, mDS, p);
  return cudaGetLastError();
}

}  // namespace sbp
