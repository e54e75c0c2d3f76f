// Tensor-core (tcgen05 / TMEM / TMA) kernels of the bf16 LM-head path, sm_103a.
//
// Both kernels are persistent, warp-specialised GEMMs run by clusters of two CTAs on two
// SMs ("pairs").  A pair computes one 256x256 fp32 tile with tcgen05.mma.cta_group::2:
// CTA r of the pair stages rows [128r, 128r+128) of A and rows [128r, 128r+128) of B's N
// extent through a 6-stage TMA -> shared-memory ring (32 KB per 64-deep k-block), the
// leader (r = 0) issues the MMAs, and each CTA's tensor memory receives its own 128
// accumulator rows x 256 columns (two buffers, 512 columns).  Per SM this moves a third
// less data through shared memory and L2 than a 1-SM 128x256 tile, whose operand
// traffic exceeds what the SM's shared memory delivers.  Roles per CTA:
//   warp 0      TMA producer (one lane)
//   warp 1      TMEM allocator; in the leader, the MMA issuer (one lane)
//   warps 2..9  epilogue: warp w reads TMEM lanes 32*(w%4).. (one accumulator row per
//               thread) and columns [128*h, 128*h+128) of the tile, h = (w-2)/4.
//
// k_fwd  : Z_c = H_c W^T  (A = H rows, B = W rows, both K-major), epilogue = row
//          statistics per 128-column tile: max m, e = exp(z - m) stored as fp16,
//          s = sum e less the maximum's own term 1, and the label logit z_y (the chunk
//          forward of the StreamBP LM head).
// k_bwd  : one dynamic queue of units of two kinds, dH first:
//          dH_c = G_c W    (A = G rows, K-major; B = W, MN-major), split along V,
//          dW  += G_c^T H_c (A = G columns, MN-major; B = H_c, MN-major).
//
// Every mbarrier wait is bounded in time: past the limit the kernel records
// SBP_ERR_TIMEOUT in the status word, stops issuing work, waits (bounded) for its own
// copies and MMAs in flight, frees its tensor memory and returns.



#include "sbp_tc_common.cuh"

namespace sbp {
namespace tc {

// ==================================================================================== forward

struct FwdP {
  int64_t r0; int rows; int64_t V;
  int mt, ntn, kb;
  const int32_t* labels;
  __half* E; int64_t lde;
  float2* part; int64_t ntiles; float* zy;
  int32_t* status; uint64_t limit_ns;
  int stall;   // failure-detection test: the MMA thread first waits on a barrier nothing arrives on
  // The previous chunk's logit gradient, formed by the epilogue warps in the time they
  // do not need for this chunk's tiles: G = e * scale, and at the label the entry
  // w expm1(logp) that the combine step left beside the label tile's scale; fp16 -> bf16
  // in place.
  __half* gprev;              // nullptr: no previous chunk to convert
  const float2* part_prev;    // its tile scales
  const float* w_prev;        // its row weights
  const int32_t* y_prev;      // its labels
  int rows_prev;
};

// A slice of the previous chunk's gradient conversion: this CTA owns a contiguous range of
// its rows; epilogue thread t takes the 8-column vectors t, t + 256, ... of that range
// (consecutive threads touch consecutive 16-byte vectors).
struct SideJob {
  int64_t rbeg, nvec, next, end;   // vector cursor of this thread, flat index over [rbeg, rend) x nvec
};

__device__ __forceinline__ void side_vector(const FwdP& p, int64_t r, int64_t v0) {
  __half* e = p.gprev + r * p.lde;
  __nv_bfloat16* g = reinterpret_cast<__nv_bfloat16*>(e);
  const float w = p.w_prev[r];
  const int32_t y = p.y_prev[r];
  if (v0 + 8 <= p.V) {
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (w != 0.f) {
      const uint4 in = *reinterpret_cast<const uint4*>(e + v0);
      const float2 s = p.part_prev[r * p.ntiles + v0 / kStatW];
      const __half2* hin = reinterpret_cast<const __half2*>(&in);
      float f[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 x = __half22float2(hin[i]);
        f[2 * i] = x.x * s.x;
        f[2 * i + 1] = x.y * s.x;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (v0 + i == (int64_t)y) f[i] = s.y;
      __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&out);
#pragma unroll
      for (int i = 0; i < 4; ++i) ob[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    }
    *reinterpret_cast<uint4*>(g + v0) = out;
  } else {
    for (int64_t v = v0; v < p.V; ++v) {
      const float2 s = p.part_prev[r * p.ntiles + v / kStatW];
      const float x = w == 0.f ? 0.f : (v == y ? s.y : __half2float(e[v]) * s.x);
      g[v] = __float2bfloat16_rn(x);
    }
  }
}

__device__ __forceinline__ void side_run(const FwdP& p, SideJob& j, int64_t quota) {
  for (int64_t k = 0; k < quota && j.next < j.end; ++k, j.next += NUM_EPI_WARPS * 32) {
    const int64_t r = j.rbeg + j.next / j.nvec;
    side_vector(p, r, (j.next % j.nvec) * 8);
  }
}

// =================================================================================== backward

struct BwdP {
  int rows; int64_t r0; int64_t V, d;
  int mt_c, nt_d, kb_v, splits, mt_v, kb_c;
  int n_dh, n_total;
  float* dh_part; int64_t plane;
  float* dW; int dw_acc;
  uint32_t* counter;
  int32_t* status; uint64_t limit_ns;
  // a batch of independent problems (attention heads) stacked along the rows of every
  // operand: problem z reads G rows from z * zr_g, W rows from z * zr_w, H rows from
  // z * zr_h and writes dW rows from z * zr_dw (all 0 when batch = 1)
  int batch, n_dh_b, n_dw_b;
  int zr_g, zr_w, zr_h, zr_dw;
  // 1: the MN-major map of G / W / H is the three-dimensional one that loads 128 columns
  // in one copy (make_map_mn2); 0: the two-dimensional 64 x 64 one, two copies
  int mn2_g, mn2_w, mn2_h;
};

// k_bwd stages its dW output through shared memory: one 32x32 fp32 block (4 KB, 128-byte
// swizzle) per epilogue warp, handed to the TMA unit for an asynchronous, coalesced
// reduce-add (or store, first chunk) into dW.
constexpr uint32_t STG_BYTES = 32 * 32 * 4;
// k_fwd stages its fp16 exp tile the same way: 32 rows x 64 columns (4 KB, 128-byte
// swizzle) per epilogue warp at a time, written out by TMA stores.  Row-per-thread global
// stores (32 L2 sectors per request) were measured to starve the operand loads.
constexpr size_t SMEM_FWD = STAGES * STAGE_BYTES + NUM_EPI_WARPS * STG_BYTES + sizeof(Ctrl) + 1024;
static_assert(SMEM_FWD <= 232448, "shared memory budget of one CTA");
constexpr size_t SMEM_BWD = STAGES * STAGE_BYTES + NUM_EPI_WARPS * STG_BYTES + sizeof(Ctrl) + 1024;
static_assert(SMEM_BWD <= 232448, "shared memory budget of one CTA");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    k_fwd(const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmW,
          const __grid_constant__ CUtensorMap tmE, const FwdP p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stg_base = base + STAGES * STAGE_BYTES;
  Ctrl* c = reinterpret_cast<Ctrl*>(stg_base + NUM_EPI_WARPS * STG_BYTES);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = ctarank();
  prologue(c, warp);
  const uint32_t tmem = c->tmem_base;
  const int mtp = (p.rows + 255) / 256;
  const int total = mtp * p.ntn;
  const int pid = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_map(&tmH);
      prefetch_map(&tmW);
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_phase[STAGES] = {0, 0, 0, 0, 0, 0};
      bool ok = true;
      for (int tile = pid; tile < total && ok; tile += npairs) {
        const int mp = tile % mtp, nb = tile / mtp;
        const int arow = (int)(p.r0 + (int64_t)mp * 256 + rank * 128);
        const int brow = nb * BN + (int)rank * 128;
        for (int kb = 0; kb < p.kb; ++kb) {
          if (!wait_bounded(&c->empty[stage], phase ^ 1u, &c->abort, p.limit_ns)) { ok = false; break; }
          const uint32_t sa = saddr(base + stage * STAGE_BYTES), sb = sa + A_BYTES;
          const uint32_t fb = mapa(saddr(&c->full[stage]), 0);
          if (rank == 0) mbar_expect_tx(&c->full[stage], PAIR_TX);
          tma_load_2d_pair(sa, &tmH, fb, kb * BK, arow);
          tma_load_2d_pair(sb, &tmW, fb, kb * BK, brow);
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
      // injected stall: mdone completes only after the commit below, so this wait runs
      // out, and every role of the pair takes the bounded-abort path
      bool ok = !p.stall || wait_bounded(&c->mdone, 0, &c->abort, p.limit_ns);
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
            mma2_bf16(dt, sw128_desc(sa + k * 32, 16, 1024), sw128_desc(sb + k * 32, 16, 1024), IDESC_FWD,
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
    // this thread's share of the previous chunk's gradient conversion, spread evenly over
    // the tiles this CTA's epilogue handles
    SideJob sj{0, 1, 0, 0};
    int64_t quota = 0;
    if (p.gprev) {
      const int64_t rbeg = (int64_t)blockIdx.x * p.rows_prev / gridDim.x;
      const int64_t rend = (int64_t)(blockIdx.x + 1) * p.rows_prev / gridDim.x;
      sj.rbeg = rbeg;
      sj.nvec = (p.V + 7) / 8;
      sj.next = (warp - 2) * 32 + lane;
      sj.end = (rend - rbeg) * sj.nvec;
      const int64_t mine = sj.end > sj.next ? (sj.end - sj.next + NUM_EPI_WARPS * 32 - 1) / (NUM_EPI_WARPS * 32) : 0;
      const int64_t ntiles_here = pid < total ? (total - pid + npairs - 1) / npairs : 0;
      quota = ntiles_here > 0 ? (mine + ntiles_here - 1) / ntiles_here : mine;
    }
    int local = 0;
    for (int tile = pid; tile < total; tile += npairs, ++local) {
      const int mp = tile % mtp, nb = tile / mtp;
      const int buf = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      const int row = mp * 256 + (int)rank * 128 + lrow;
      const bool vrow = row < p.rows;
      const int32_t y = vrow ? p.labels[row] : INT_MIN;
      if (!warp_wait_cluster(&c->tfull[buf], use & 1u, c, p.limit_ns)) {
        fail(c, p.status);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + h * 128);
      const int64_t c0 = (int64_t)nb * BN + h * 128;
      // the row's 128 accumulator columns of this half tile, then the buffer goes back
      // to the MMA at once: the statistics below run while the next tile accumulates
      uint32_t r[4][32];
      __syncwarp();
#pragma unroll
      for (int g = 0; g < 4; ++g) tmem_ld32(tb + g * 32, r[g]);
      tmem_ld_wait();
      release_tmem(c, buf, lane);
      const int64_t nv = p.V - c0;                  // valid columns of this half tile
      const int ncol = nv >= 128 ? 128 : (nv > 0 ? (int)nv : 0);
      float m = -INFINITY;
      if (ncol == 128) {
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
          for (int j = 0; j < 32; ++j) m = fmaxf(m, __uint_as_float(r[g][j]));
      } else {
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (g * 32 + j < ncol) m = fmaxf(m, __uint_as_float(r[g][j]));
      }
      const int64_t jy = (int64_t)y - c0;           // the label's column within the half tile
      const bool has_y = vrow && jy >= 0 && jy < ncol;
      float zyv = 0.f;
      if (has_y) {
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (g * 32 + j == (int)jy) zyv = __uint_as_float(r[g][j]);
      }
      // s = sum of exp(z - m) over the tile less the term of one maximum (exactly 1): the
      // other maxima count 1 each; kept apart so that the confident regime, where the
      // rest is far below 1, does not round it away
      const float mb2 = m * L2E;
      float s = 0.f, nmax = -1.f;
      const uint32_t stg = saddr(stg_base + (warp - 2) * STG_BYTES);
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        if (g * 32 >= ncol) break;
        if (p.E && (g & 1) == 0) {   // the staging block's previous contents have left
          if (lane == 0) bulk_wait_read();
          __syncwarp();
        }
        uint32_t hv[16];
        if (ncol == 128) {
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float z0 = __uint_as_float(r[g][j]), z1 = __uint_as_float(r[g][j + 1]);
            const float e0 = ex2(fmaf(z0, L2E, -mb2));
            const float e1 = ex2(fmaf(z1, L2E, -mb2));
            s += (z0 == m ? 0.f : e0) + (z1 == m ? 0.f : e1);
            nmax += (z0 == m ? 1.f : 0.f) + (z1 == m ? 1.f : 0.f);
            const __half2 hh = __floats2half2_rn(e0, e1);
            hv[j / 2] = *reinterpret_cast<const uint32_t*>(&hh);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float z0 = __uint_as_float(r[g][j]), z1 = __uint_as_float(r[g][j + 1]);
            const bool in0 = g * 32 + j < ncol, in1 = g * 32 + j + 1 < ncol;
            const float e0 = in0 ? ex2(fmaf(z0, L2E, -mb2)) : 0.f;
            const float e1 = in1 ? ex2(fmaf(z1, L2E, -mb2)) : 0.f;
            s += (in0 && z0 == m ? 0.f : e0) + (in1 && z1 == m ? 0.f : e1);
            nmax += (in0 && z0 == m ? 1.f : 0.f) + (in1 && z1 == m ? 1.f : 0.f);
            const __half2 hh = __floats2half2_rn(e0, e1);
            hv[j / 2] = *reinterpret_cast<const uint32_t*>(&hh);
          }
        }
        if (p.E) {
          // row `lane` of the warp's 32 x 64 block, 16-byte chunk k at chunk k ^ (lane % 8)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            sts128(stg + lane * 128 + ((((g & 1) * 4 + k) ^ (lane & 7)) << 4), hv[4 * k], hv[4 * k + 1],
                   hv[4 * k + 2], hv[4 * k + 3]);
          if ((g & 1) == 1 || (g + 1) * 32 >= ncol) {
            // the block goes out by TMA; rows past the chunk and columns past V are clipped
            // by the tensor map (the columns a half-filled block leaves are past V)
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmE, stg, (int)(c0 + (g >> 1) * 64), mp * 256 + (int)rank * 128 + q * 32);
              bulk_commit();
            }
          }
        }
      }
      const int64_t tix = (int64_t)nb * 2 + h;
      if (vrow && tix < p.ntiles) p.part[(int64_t)row * p.ntiles + tix] = make_float2(m, s + nmax);
      if (vrow && has_y) p.zy[row] = zyv;
      if (p.gprev) side_run(p, sj, quota);
    }
    if (p.gprev && !c->abort) side_run(p, sj, INT64_MAX);   // what rounding left over
    if (lane == 0) bulk_wait_all();   // every exp block has left shared memory and landed
    __syncwarp();
  }
  teardown(c, warp);
}

// Backward, pair version.  Units are decoded from the same atomic queue as the 1-CTA
// kernel, but M tiles are 256 rows (a pair) and the leader's producer takes each unit
// from the queue and hands it to the peer through distributed shared memory.
struct Unit {
  int kind, mp, nb, split, kb0, kb1;
  int z;   // problem of the batch
};

// dH units of one split run in bands of kDhBand row tiles: a band's units cover its row
// tiles for every column tile of d, row tiles fastest.  A wave of 76 SM pairs then holds
// about 8 row tiles x 9.5 column tiles, so G's k-blocks (one per row tile) and W's (one per
// column tile) are each fetched about twice per wave, instead of G about 3.4 times and W
// once when all 16 row tiles of a 4096-row chunk come first.  Measured on the profile case
// (chunk 4096, d 4096, V 32768): 5.4% less DRAM traffic per k_bwd launch and 1.5% more
// tokens per MHz on the bench workload.  Only the order changes: the partials of each
// split are summed in a fixed order, so the results are the same bits.
constexpr int kDhBand = 8;

__device__ __forceinline__ Unit decode(const BwdP& p, int u) {
  Unit w;
  if (u < p.n_dh) {
    w.kind = 0;
    w.z = u / p.n_dh_b;
    u -= w.z * p.n_dh_b;
    const int per = p.mt_c * p.nt_d;
    w.split = u / per;
    const int t = u - w.split * per;
    const int R = p.mt_c < kDhBand ? p.mt_c : kDhBand;
    const int band = t / (R * p.nt_d);
    const int t2 = t - band * R * p.nt_d;
    const int rk = p.mt_c - band * R < R ? p.mt_c - band * R : R;   // row tiles in this band
    w.mp = band * R + t2 % rk;
    w.nb = t2 / rk;
    w.kb0 = (int)((int64_t)w.split * p.kb_v / p.splits);
    w.kb1 = (int)((int64_t)(w.split + 1) * p.kb_v / p.splits);
  } else {
    u -= p.n_dh;
    w.kind = 1;
    w.z = u / p.n_dw_b;
    u -= w.z * p.n_dw_b;
    w.nb = u % p.nt_d;
    w.mp = u / p.nt_d;
    w.split = 0;
    w.kb0 = 0;
    w.kb1 = p.kb_c;
  }
  return w;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    k_bwd(const __grid_constant__ CUtensorMap tmGk, const __grid_constant__ CUtensorMap tmGmn,
          const __grid_constant__ CUtensorMap tmWmn, const __grid_constant__ CUtensorMap tmHmn,
          const __grid_constant__ CUtensorMap tmDW, const __grid_constant__ CUtensorMap tmDH, const BwdP p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stg_base = base + STAGES * STAGE_BYTES;
  Ctrl* c = reinterpret_cast<Ctrl*>(stg_base + NUM_EPI_WARPS * STG_BYTES);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = ctarank();
  prologue(c, warp);
  const uint32_t tmem = c->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_map(&tmGk);
      prefetch_map(&tmGmn);
      prefetch_map(&tmWmn);
      prefetch_map(&tmHmn);
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_phase[STAGES] = {0, 0, 0, 0, 0, 0};
      bool ok = true;
      // the leader takes units one ahead, so the atomic's latency overlaps the loads
      // of the unit in hand instead of stalling the ring at every unit boundary
      int next_u = rank == 0 ? (int)atomicAdd(p.counter, 1u) : -1;
      for (int i = 0; ok; ++i) {
        const int slot = i % RING;
        const uint32_t rph = (uint32_t)((i / RING) & 1);
        int u;
        if (rank == 0) {
          if (!wait_cluster(&c->rempty[slot], rph ^ 1u, &c->abort, p.limit_ns)) { ok = false; break; }
          u = next_u < p.n_total ? next_u : -1;
          if (u >= 0) next_u = (int)atomicAdd(p.counter, 1u);
          c->ring[slot] = u;
          asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(mapa(saddr(&c->ring[slot]), 1)), "r"(u) : "memory");
          mbar_arrive(&c->rfull[slot]);
          arrive_cluster(mapa(saddr(&c->rfull[slot]), 1));
        } else {
          if (!wait_cluster(&c->rfull[slot], rph, &c->abort, p.limit_ns)) { ok = false; break; }
          u = *(volatile int*)&c->ring[slot];
          arrive_cluster(mapa(saddr(&c->rempty[slot]), 0));
        }
        if (u < 0) break;
        const Unit w = decode(p, u);
        const int mrow = w.mp * 256 + (int)rank * 128;      // this CTA's first M row (or V row)
        const int ncol = w.nb * BN + (int)rank * 128;       // this CTA's first N column of d
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!wait_bounded(&c->empty[stage], phase ^ 1u, &c->abort, p.limit_ns)) { ok = false; break; }
          const uint32_t sa = saddr(base + stage * STAGE_BYTES), sb = sa + A_BYTES;
          const uint32_t fb = mapa(saddr(&c->full[stage]), 0);
          if (rank == 0) mbar_expect_tx(&c->full[stage], PAIR_TX);
          if (w.kind == 0) {
            tma_load_2d_pair(sa, &tmGk, fb, kb * BK, w.z * p.zr_g + mrow);
            const int wr = w.z * p.zr_w + kb * BK;
            if (p.mn2_w) {
              tma_load_3d_pair(sb, &tmWmn, fb, 0, wr, ncol / 64);
            } else {
#pragma unroll
              for (int j = 0; j < 2; ++j) tma_load_2d_pair(sb + j * BOX_BYTES, &tmWmn, fb, ncol + j * 64, wr);
            }
          } else {
            const int gr = w.z * p.zr_g + kb * BK;
            if (p.mn2_g) {
              tma_load_3d_pair(sa, &tmGmn, fb, 0, gr, mrow / 64);
            } else {
#pragma unroll
              for (int j = 0; j < 2; ++j) tma_load_2d_pair(sa + j * BOX_BYTES, &tmGmn, fb, mrow + j * 64, gr);
            }
            const int hr = (int)(w.z * (int64_t)p.zr_h + p.r0 + (int64_t)kb * BK);
            if (p.mn2_h) {
              tma_load_3d_pair(sb, &tmHmn, fb, 0, hr, ncol / 64);
            } else {
#pragma unroll
              for (int j = 0; j < 2; ++j) tma_load_2d_pair(sb + j * BOX_BYTES, &tmHmn, fb, ncol + j * 64, hr);
            }
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
      for (int i = 0; ok; ++i, ++local) {
        const int slot = i % RING;
        const uint32_t rph = (uint32_t)((i / RING) & 1);
        if (!wait_cluster(&c->rfull[slot], rph, &c->abort, p.limit_ns)) { ok = false; break; }
        const int u = *(volatile int*)&c->ring[slot];
        mbar_arrive(&c->rempty[slot]);
        if (u < 0) break;
        const Unit w = decode(p, u);
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!wait_cluster(&c->tempty[buf], (use & 1u) ^ 1u, &c->abort, p.limit_ns)) { ok = false; break; }
        tc_fence_after();
        const uint32_t dt = tmem + (uint32_t)(buf * BN);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!wait_bounded(&c->full[stage], phase, &c->abort, p.limit_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = saddr(base + stage * STAGE_BYTES), sb = sa + A_BYTES;
          const uint32_t acc0 = kb != w.kb0 ? 1u : 0u;
          if (w.kind == 0) {
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              mma2_bf16(dt, sw128_desc(sa + k * 32, 16, 1024), sw128_desc(sb + k * 2048, BOX_BYTES, 1024), IDESC_DH,
                        acc0 | (k != 0));
          } else {
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              mma2_bf16(dt, sw128_desc(sa + k * 2048, BOX_BYTES, 1024), sw128_desc(sb + k * 2048, BOX_BYTES, 1024),
                        IDESC_DW, acc0 | (k != 0));
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
    int local = 0;
    for (int i = 0;; ++i, ++local) {
      const int slot = i % RING;
      const uint32_t rph = (uint32_t)((i / RING) & 1);
      if (!warp_wait_cluster(&c->rfull[slot], rph, c, p.limit_ns)) {
        fail(c, p.status);
        break;
      }
      const int u = *(volatile int*)&c->ring[slot];
      __syncwarp();
      if (lane == 0) arrive_cluster(mapa(saddr(&c->rempty[slot]), 0));
      if (u < 0) break;
      const Unit w = decode(p, u);
      const int buf = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      if (!warp_wait_cluster(&c->tfull[buf], use & 1u, c, p.limit_ns)) {
        fail(c, p.status);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + h * 128);
      const int64_t c0 = (int64_t)w.nb * BN + h * 128;
      uint32_t r[4][32];
      __syncwarp();
#pragma unroll
      for (int g = 0; g < 4; ++g) tmem_ld32(tb + g * 32, r[g]);
      tmem_ld_wait();
      release_tmem(c, buf, lane);
      if (w.kind == 1) {
        // dW rows [y0, y0+32) x columns [cg, cg+32): through the warp's staging block.
        // Each dW element receives one add per launch (one unit owns each tile), so the
        // TMA reduce-add is deterministic.  Rows past V and columns past d are clipped
        // by the tensor map.
        const uint32_t stg = saddr(stg_base + (warp - 2) * STG_BYTES);
        const int y0 = w.mp * 256 + (int)rank * 128 + q * 32;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int64_t cg = c0 + g * 32;
          if (cg >= p.d) break;
          if (lane == 0) bulk_wait_read();   // the previous block has left the staging buffer
          __syncwarp();
          // row `lane`, 16-byte chunk k stored at chunk k ^ (lane % 8): the 128-byte swizzle
          // the tensor map reads, and conflict-free for the 32 lanes
#pragma unroll
          for (int k = 0; k < 8; ++k)
            sts128(stg + lane * 128 + ((k ^ (lane & 7)) << 4), r[g][4 * k], r[g][4 * k + 1], r[g][4 * k + 2],
                   r[g][4 * k + 3]);
          fence_proxy_async();
          __syncwarp();
          if (lane == 0 && y0 < p.V) {
            const int yz = w.z * p.zr_dw + y0;
            if (p.dw_acc) tma_reduce_add_2d(&tmDW, stg, (int)cg, yz);
            else tma_store_2d(&tmDW, stg, (int)cg, yz);
            bulk_commit();
          }
        }
        continue;
      }
      {
        // dH split-K partial rows [y0, y0+32) x columns [cg, cg+32) of plane split * batch + z,
        // through the same staging block and a TMA store (rows past the chunk and columns
        // past d are clipped by the three-dimensional map)
        const uint32_t stg = saddr(stg_base + (warp - 2) * STG_BYTES);
        const int y0 = w.mp * 256 + (int)rank * 128 + q * 32;
        const int zpl = w.split * p.batch + w.z;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int64_t cg = c0 + g * 32;
          if (cg >= p.d) break;
          if (lane == 0) bulk_wait_read();
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            sts128(stg + lane * 128 + ((k ^ (lane & 7)) << 4), r[g][4 * k], r[g][4 * k + 1], r[g][4 * k + 2],
                   r[g][4 * k + 3]);
          fence_proxy_async();
          __syncwarp();
          if (lane == 0 && y0 < p.rows) {
            tma_store_3d(&tmDH, stg, (int)cg, y0, zpl);
            bulk_commit();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_all();   // every dW block has left shared memory and landed
    __syncwarp();
  }
  teardown(c, warp);
}

// ======================================================================================= host

bool set_smem_attr() {
  static int attr_state[64] = {};
  static std::mutex mu;
  return once_per_device(attr_state, mu, [] {
    return cudaFuncSetAttribute(k_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_FWD) == cudaSuccess &&
           cudaFuncSetAttribute(k_bwd, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BWD) == cudaSuccess;
  });
}

}  // namespace tc

cudaError_t tc_forward(const TcFwdArgs& a, cudaStream_t s) {
  using namespace tc;
  if (!set_smem_attr()) return cudaErrorInvalidConfiguration;
  // boxes of 64 (K) x 128 rows: each CTA of a pair stages 128 rows of H and 128 of W
  CUtensorMap mH, mW, mE;
  if (!make_map(&mH, a.H, (uint64_t)a.d, (uint64_t)a.T, (uint64_t)a.d, BK, 128)) return cudaErrorInvalidValue;
  if (!make_map(&mW, a.W, (uint64_t)a.d, (uint64_t)a.V, (uint64_t)a.d, BK, 128)) return cudaErrorInvalidValue;
  // fp16 exp tile [rows, V] with row stride lde, stored in 64 x 32 blocks (a 16-bit map:
  // the store copies the bits); statistics-only launches pass no E and use the H map
  if (a.E) {
    if (!make_map(&mE, a.E, (uint64_t)a.V, (uint64_t)a.rows, (uint64_t)a.lde, 64, 32)) return cudaErrorInvalidValue;
  } else {
    mE = mH;
  }
  FwdP p;
  p.r0 = a.r0; p.rows = a.rows; p.V = a.V;
  p.mt = (a.rows + 255) / 256;
  p.ntn = (int)((a.V + BN - 1) / BN);
  p.kb = (int)((a.d + BK - 1) / BK);
  p.labels = a.labels;
  p.E = static_cast<__half*>(a.E); p.lde = a.lde;
  p.part = a.part; p.ntiles = (a.V + kStatW - 1) / kStatW; p.zy = a.zy;
  p.status = a.status; p.limit_ns = wait_limit_ns();
  p.stall = fault_stall_requested();
  p.gprev = static_cast<__half*>(a.gprev); p.part_prev = a.part_prev; p.w_prev = a.w_prev;
  p.y_prev = a.y_prev; p.rows_prev = a.rows_prev;
  const int total = p.mt * p.ntn;
  int pairs = max_pairs((const void*)k_fwd, SMEM_FWD);
  if (pairs > total) pairs = total;
  k_fwd<<<2 * pairs, NUM_THREADS, SMEM_FWD, s>>>(mH, mW, mE, p);
  return cudaGetLastError();
}

cudaError_t tc_backward(const TcBwdArgs& a, cudaStream_t s) {
  using namespace tc;
  if (!set_smem_attr()) return cudaErrorInvalidConfiguration;
  CUtensorMap mGk, mGmn, mWmn, mHmn;
  // G: [rows, V] with row stride ldg; rows past the chunk read as zero.
  const uint64_t g_rows = a.g_rows ? (uint64_t)a.g_rows : (uint64_t)a.rows;
  const uint64_t w_rows = a.w_rows ? (uint64_t)a.w_rows : (uint64_t)a.V;
  const uint64_t h_rows = a.h_rows ? (uint64_t)a.h_rows : (uint64_t)a.T;
  const uint64_t dw_rows = a.dw_rows ? (uint64_t)a.dw_rows : (uint64_t)a.V;
  if (!make_map(&mGk, a.G, (uint64_t)a.V, g_rows, (uint64_t)a.ldg, BK, 128)) return cudaErrorInvalidValue;
  // MN-major operands: one copy of 128 columns where the row length allows it (multiples of
  // 64 elements), else two 64 x 64 boxes
  const int mn2_g = make_map_mn2(&mGmn, a.G, g_rows, (uint64_t)a.ldg) ? 1 : 0;
  if (!mn2_g && !make_map(&mGmn, a.G, (uint64_t)a.V, g_rows, (uint64_t)a.ldg, 64, 64)) return cudaErrorInvalidValue;
  const int mn2_w = make_map_mn2(&mWmn, a.W, w_rows, (uint64_t)a.d) ? 1 : 0;
  if (!mn2_w && !make_map(&mWmn, a.W, (uint64_t)a.d, w_rows, (uint64_t)a.d, 64, 64)) return cudaErrorInvalidValue;
  const int mn2_h = make_map_mn2(&mHmn, a.H, h_rows, (uint64_t)a.d) ? 1 : 0;
  if (!mn2_h && !make_map(&mHmn, a.H, (uint64_t)a.d, h_rows, (uint64_t)a.d, 64, 64)) return cudaErrorInvalidValue;
  CUtensorMap mDW, mDH;
  if (!make_map_f32(&mDW, a.dW, (uint64_t)a.d, dw_rows)) return cudaErrorInvalidValue;
  // dH partials [splits * batch planes][rows][d] fp32: a 3-D map, so that stores clip at
  // the chunk's last row of each plane
  if (!a.dw_only && a.dh_part) {
    if (!make_map3_f32(&mDH, a.dh_part, (uint64_t)a.d, (uint64_t)a.rows,
                       (uint64_t)a.splits * (uint64_t)(a.batch > 0 ? a.batch : 1)))
      return cudaErrorInvalidValue;
  } else {
    mDH = mDW;
  }
  BwdP p;
  p.rows = a.rows; p.r0 = a.r0; p.V = a.V; p.d = a.d;
  p.mt_c = (a.rows + 255) / 256;
  p.nt_d = (int)((a.d + BN - 1) / BN);
  p.kb_v = (int)((a.V + BK - 1) / BK);
  p.splits = a.splits;
  p.mt_v = (int)((a.V + 255) / 256);
  p.kb_c = (a.rows + BK - 1) / BK;
  p.batch = a.batch > 0 ? a.batch : 1;
  p.n_dh_b = a.dw_only ? 0 : p.mt_c * p.nt_d * p.splits;
  p.n_dw_b = p.mt_v * p.nt_d;
  p.n_dh = p.n_dh_b * p.batch;
  p.n_total = p.n_dh + p.n_dw_b * p.batch;
  p.zr_g = a.zr_g; p.zr_w = a.zr_w; p.zr_h = a.zr_h; p.zr_dw = a.zr_dw;
  p.mn2_g = mn2_g; p.mn2_w = mn2_w; p.mn2_h = mn2_h;
  p.dh_part = a.dh_part; p.plane = (int64_t)a.rows * a.d;
  p.dW = a.dW; p.dw_acc = a.dw_accumulate;
  p.counter = a.counter; p.status = a.status; p.limit_ns = wait_limit_ns();
  int pairs = max_pairs((const void*)k_bwd, SMEM_BWD);
  if (pairs > p.n_total) pairs = p.n_total;
  k_bwd<<<2 * pairs, NUM_THREADS, SMEM_BWD, s>>>(mGk, mGmn, mWmn, mHmn, mDW, mDH, p);
  return cudaGetLastError();
}

}  // namespace sbp
