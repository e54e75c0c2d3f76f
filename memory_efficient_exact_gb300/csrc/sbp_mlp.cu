// Tensor-core kernels of the chunked SwiGLU-MLP backward (bf16, sm_103a).
//
// The position-wise MLP sublayer y = a Wd^T, a = silu(x Wg^T) * (x Wu^T), splits over row
// chunks exactly as the LM head does: each chunk recomputes its activations and adds its
// share of the weight gradients.  Two pair GEMMs are specific to it (the rest reuses
// k_bwd):
//   k_mlp<false>  gu = x_c [Wg; Wu]^T for one 128-wide block of f at a time: CTA 0 of the
//                 pair stages gate rows, CTA 1 the matching up rows of the packed Wgu
//                 [2f, d], so one 256-column accumulator tile holds g | u of the same f;
//                 epilogue: a = silu(g) u (bf16), and g, u kept (bf16) for the backward.
//   k_mlp<true>   da = dY_c Wd (B = Wd [d, f], MN-major); epilogue: dg = da u silu'(g),
//                 du = da silu(g), written in place over g | u.
// Same pair protocol, warp roles and bounded waits as the LM-head kernels.
#include "sbp_tc_common.cuh"

namespace sbp {
namespace tc {

struct MlpP {
  int64_t r0; int rows; int64_t f;
  int mt, ntn, kb;
  __nv_bfloat16* A;    // [rows, f]   a = silu(g) u                (k_mlp<false>)
  __nv_bfloat16* GU;   // [rows, 2f]  g | u, then dg | du in place
  int32_t* status; uint64_t limit_ns;
};

// The epilogue's bf16 outputs leave through one 32 x 64 staging block (4 KB, 128-byte
// swizzle) per warp and TMA stores, and k_mlp<true> reads g and u through the same block
// with TMA loads (completing on one mbarrier per warp): row-per-thread global accesses
// (32 L2 sectors per request) were measured to starve the operand loads.
constexpr uint32_t STG_MLP = 32 * 64 * 2;
constexpr size_t SMEM_MLP =
    STAGES * STAGE_BYTES + NUM_EPI_WARPS * STG_MLP + sizeof(Ctrl) + NUM_EPI_WARPS * sizeof(uint64_t) + 1024;
static_assert(SMEM_MLP <= 232448, "shared memory budget of one CTA");

template <bool DA>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    k_mlp(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
          const __grid_constant__ CUtensorMap tmAo, const __grid_constant__ CUtensorMap tmGU, const MlpP p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stg_base = base + STAGES * STAGE_BYTES;
  Ctrl* c = reinterpret_cast<Ctrl*>(stg_base + NUM_EPI_WARPS * STG_MLP);
  uint64_t* lbar = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(c) + sizeof(Ctrl));   // per epilogue warp
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = ctarank();
  prologue(c, warp);
  const uint32_t tmem = c->tmem_base;
  const int total = p.mt * p.ntn;
  const int pid = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_map(&tmA);
      prefetch_map(&tmB);
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_phase[STAGES] = {0, 0, 0, 0, 0, 0};
      bool ok = true;
      for (int tile = pid; tile < total && ok; tile += npairs) {
        const int mp = tile % p.mt, nb = tile / p.mt;
        const int arow = (int)(p.r0 + (int64_t)mp * 256 + rank * 128);
        for (int kb = 0; kb < p.kb; ++kb) {
          if (!wait_bounded(&c->empty[stage], phase ^ 1u, &c->abort, p.limit_ns)) { ok = false; break; }
          const uint32_t sa = saddr(base + stage * STAGE_BYTES), sb = sa + A_BYTES;
          const uint32_t fb = mapa(saddr(&c->full[stage]), 0);
          if (rank == 0) mbar_expect_tx(&c->full[stage], PAIR_TX);
          tma_load_2d_pair(sa, &tmA, fb, kb * BK, arow);
          if (!DA) {
            // gate rows [128 nb, +128) in CTA 0, up rows [f + 128 nb, +128) in CTA 1
            tma_load_2d_pair(sb, &tmB, fb, kb * BK, (int)((rank ? p.f : 0) + (int64_t)nb * 128));
          } else {
#pragma unroll
            for (int j = 0; j < 2; ++j)
              tma_load_2d_pair(sb + j * BOX_BYTES, &tmB, fb, nb * BN + (int)rank * 128 + j * 64, kb * BK);
          }
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
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t bdesc =
                DA ? sw128_desc(sb + k * 2048, BOX_BYTES, 1024) : sw128_desc(sb + k * 32, 16, 1024);
            mma2_bf16(dt, sw128_desc(sa + k * 32, 16, 1024), bdesc, DA ? IDESC_KM : IDESC_KK, (kb | k) != 0);
          }
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
    uint64_t* bar = lbar + (warp - 2);
    uint32_t lphase = 0;
    if (DA) {
      if (lane == 0) {
        mbar_init(bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      }
      __syncwarp();
    }
    int local = 0;
    for (int tile = pid; tile < total; tile += npairs, ++local) {
      const int mp = tile % p.mt, nb = tile / p.mt;
      const int buf = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      if (!warp_wait_cluster(&c->tfull[buf], use & 1u, c, p.limit_ns)) {
        fail(c, p.status);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
      const uint32_t stg = saddr(stg_base + (warp - 2) * STG_MLP);
      const int yrow = mp * 256 + (int)rank * 128 + q * 32;   // this warp's first row
      __syncwarp();
      if (!DA) {
        // g in accumulator columns [64h, 64h+64), u in [128 + 64h, 128 + 64h + 64)
        uint32_t r[4][32];
        tmem_ld32(tb + 64 * h, r[0]);
        tmem_ld32(tb + 64 * h + 32, r[1]);
        tmem_ld32(tb + 128 + 64 * h, r[2]);
        tmem_ld32(tb + 128 + 64 * h + 32, r[3]);
        tmem_ld_wait();
        release_tmem(c, buf, lane);
        const int f0 = nb * 128 + 64 * h;
        // a = silu(g) u, then g, then u: one 32 x 64 block each (rows past the chunk are
        // clipped by the tensor maps)
        stage_free(lane);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          uint32_t av[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float g0 = __uint_as_float(r[g][j]), g1 = __uint_as_float(r[g][j + 1]);
            const float u0 = __uint_as_float(r[2 + g][j]), u1 = __uint_as_float(r[2 + g][j + 1]);
            av[j / 2] = pack_bf16(g0 * sigmoid_fast(g0) * u0, g1 * sigmoid_fast(g1) * u1);
          }
          stage4(stg, lane, 4 * g, av);
        }
        stage_store(&tmAo, stg, lane, f0, yrow);
#pragma unroll
        for (int t = 0; t < 2; ++t) {   // t = 0: g, t = 1: u
          stage_free(lane);
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            uint32_t v[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2)
              v[j / 2] = pack_bf16(__uint_as_float(r[2 * t + g][j]), __uint_as_float(r[2 * t + g][j + 1]));
            stage4(stg, lane, 4 * g, v);
          }
          stage_store(&tmGU, stg, lane, (t ? p.f : 0) + f0, yrow);
        }
      } else {
        // this half tile's 128 columns of da in two 64-column blocks; g and u come in by TMA
        // loads through the staging block, dg and du go out by TMA stores in their place
        bool lok = true;
#pragma unroll 1
        for (int bx = 0; bx < 2 && lok; ++bx) {
          uint32_t r[2][32];
          tmem_ld32(tb + 128 * h + 64 * bx, r[0]);
          tmem_ld32(tb + 128 * h + 64 * bx + 32, r[1]);
          tmem_ld_wait();
          if (bx == 1) release_tmem(c, buf, lane);
          const int f0 = nb * BN + 128 * h + 64 * bx;
          uint32_t gw[32], uw[32];
          stage_free(lane);
          lok = stage_load(&tmGU, stg, STG_MLP, bar, lphase, lane, f0, yrow, c, p.limit_ns);
          stage_read_row(stg, lane, gw);
          lok = lok && stage_load(&tmGU, stg, STG_MLP, bar, lphase, lane, (int)p.f + f0, yrow, c, p.limit_ns);
          stage_read_row(stg, lane, uw);
          if (!lok) break;
          __syncwarp();
#pragma unroll
          for (int w = 0; w < 32; ++w) {   // dg replaces g, du replaces u (word by word)
            const float2 gg = unpack_bf16(gw[w]), uu = unpack_bf16(uw[w]);
            const float a0 = __uint_as_float(r[w >> 4][(2 * w) & 31]), a1 = __uint_as_float(r[w >> 4][(2 * w + 1) & 31]);
            const float s0 = sigmoid_fast(gg.x), s1 = sigmoid_fast(gg.y);
            // dg = da u silu'(g), silu'(g) = s (1 + g (1 - s));  du = da silu(g)
            gw[w] = pack_bf16(a0 * uu.x * s0 * (1.f + gg.x * (1.f - s0)), a1 * uu.y * s1 * (1.f + gg.y * (1.f - s1)));
            uw[w] = pack_bf16(a0 * gg.x * s0, a1 * gg.y * s1);
          }
          // the staging block holds u (read by every lane above): dg replaces it
          stage4(stg, lane, 0, gw);
          stage4(stg, lane, 4, gw + 16);
          stage_store(&tmGU, stg, lane, f0, yrow);
          stage_free(lane);
          stage4(stg, lane, 0, uw);
          stage4(stg, lane, 4, uw + 16);
          stage_store(&tmGU, stg, lane, (int)p.f + f0, yrow);
        }
        if (!lok) {
          fail(c, p.status);
          break;
        }
      }
    }
    if (lane == 0) bulk_wait_all();   // every output block has left shared memory and landed
    __syncwarp();
  }
  teardown(c, warp);
}

}  // namespace tc

cudaError_t tc_mlp(const TcMlpArgs& a, bool da, cudaStream_t s) {
  using namespace tc;
  static int attr_state[64] = {};
  static std::mutex mu;
  if (!once_per_device(attr_state, mu, [] {
        return cudaFuncSetAttribute(k_mlp<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_MLP) ==
                   cudaSuccess &&
               cudaFuncSetAttribute(k_mlp<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_MLP) ==
                   cudaSuccess;
      }))
    return cudaErrorInvalidConfiguration;
  CUtensorMap mA, mB;
  // A: x or dY rows [T, d], boxes of 64 (K) x 128 rows
  if (!make_map(&mA, a.Arows, (uint64_t)a.d, (uint64_t)a.T, (uint64_t)a.d, BK, 128)) return cudaErrorInvalidValue;
  if (!da) {
    // B: the packed [Wg; Wu] = [2f, d], K-major boxes of 64 x 128 rows
    if (!make_map(&mB, a.B, (uint64_t)a.d, (uint64_t)(2 * a.f), (uint64_t)a.d, BK, 128)) return cudaErrorInvalidValue;
  } else {
    // B: Wd [d, f] read MN-major: boxes of 64 f-columns x 64 d-rows
    if (!make_map(&mB, a.B, (uint64_t)a.f, (uint64_t)a.d, (uint64_t)a.f, 64, 64)) return cudaErrorInvalidValue;
  }
  // outputs of the chunk: a [rows, f] and g | u [rows, 2f], bf16, stored in 64 x 32 blocks
  CUtensorMap mAo, mGU;
  if (!make_map(&mGU, a.GU, (uint64_t)(2 * a.f), (uint64_t)a.rows, (uint64_t)(2 * a.f), 64, 32))
    return cudaErrorInvalidValue;
  if (!da) {
    if (!make_map(&mAo, a.Aout, (uint64_t)a.f, (uint64_t)a.rows, (uint64_t)a.f, 64, 32)) return cudaErrorInvalidValue;
  } else {
    mAo = mGU;
  }
  MlpP p;
  p.r0 = a.r0; p.rows = a.rows; p.f = a.f;
  p.mt = (a.rows + 255) / 256;
  p.ntn = da ? (int)(a.f / BN) : (int)(a.f / 128);
  p.kb = (int)((a.d + BK - 1) / BK);
  p.A = static_cast<__nv_bfloat16*>(a.Aout);
  p.GU = static_cast<__nv_bfloat16*>(a.GU);
  p.status = a.status; p.limit_ns = wait_limit_ns();
  const int total = p.mt * p.ntn;
  const void* kern = da ? (const void*)k_mlp<true> : (const void*)k_mlp<false>;
  int pairs = max_pairs(kern, SMEM_MLP);
  if (pairs > total) pairs = total;
  if (da) k_mlp<true><<<2 * pairs, NUM_THREADS, SMEM_MLP, s>>>(mA, mB, mAo, mGU, p);
  else k_mlp<false><<<2 * pairs, NUM_THREADS, SMEM_MLP, s>>>(mA, mB, mAo, mGU, p);
  return cudaGetLastError();
}

}  // namespace sbp
