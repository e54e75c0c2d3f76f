// Fused tensor-core kernels of the chunked causal-attention backward at head dimension
// 128 (bf16 operands, fp32 accumulation, sm_103a).
//
// Per chunk of queries [c0, c1), which reads keys [0, c1) only (the causal structure
// StreamBP uses), two SM-pair kernels keep the chunk's probabilities and score gradients
// on chip: nothing of size (queries x keys) goes through HBM.
//
//   k_attn_kv  unit = (head, 256 keys).  dV and dK of those keys stay in tensor memory
//              while the unit walks the chunk's query blocks of 128:
//                S^T = K Q^T,  dP^T = V dO^T                      (tensor memory)
//                P^T = exp(s S^T - lse),  dS^T = P^T (dP^T - D)   (epilogue -> shared memory)
//                dV += P^T dO,  dK += dS^T Q                      (tensor memory)
//              then adds dV and s dK into the fp32 outputs (TMA reduce-add).
//   k_attn_q   unit = (head, 256 queries of the chunk).  dQ stays in tensor memory while
//              the unit walks the key blocks of 128 up to its last query:
//                S = Q K^T,  dP = dO V^T,  dS = P (dP - D),  dQ += dS K
//              then stores s dQ in bf16.
// S and dP are formed in both kernels, so that no accumulator is shared between units:
// every output element is written by one unit in a fixed order (deterministic, no
// floating-point atomics).
//
// Pair protocol as in the other tensor-core kernels: the leader CTA's thread issues
// tcgen05.mma cta_group::2 with M = 256 (128 rows in each CTA) and N = 128 (each CTA
// supplies half of B); TMA copies of both CTAs complete on the leader's barriers; the
// commits are multicast to both CTAs; every wait is bounded in time.
#include "sbp_tc_common.cuh"

namespace sbp {
namespace tc {
namespace fa {

// Warps: 0 TMA producers, 1 MMA issuer, then the epilogue warps (lane quadrant warp % 4),
// then (k_attn_kv) one warp that stages lse and D per block, and one forwarder warp.  The
// epilogue warps arrive on CTA-local barriers; the forwarder turns each completed local
// phase into one arrival at the leader, which keeps the remote arrival's latency off the
// epilogue's critical path.
// k_attn_q: sixteen epilogue warps of 32 of the 128 columns each (19 warps, 85 registers
// a thread, no spills; eight warps of 64 columns measured the same).
constexpr int Q_EPI = 16;
// k_attn_kv: eight epilogue warps of 64 columns each (12 warps in all, so 168 registers a
// thread): its epilogue measured 1490 cycles per block this way against 2350 for sixteen
// warps of 32 columns held to 96 registers, the same work spilling.
constexpr int KV_EPI = 8;
constexpr int KV_LD_WARP = 2 + KV_EPI, KV_FWD_WARP = KV_LD_WARP + 1, Q_FWD_WARP = 2 + Q_EPI;
constexpr int KV_THREADS = 32 * (KV_FWD_WARP + 1);
constexpr int Q_THREADS = 32 * (Q_FWD_WARP + 1);
constexpr uint32_t IDESC_KK = idesc_bf16(256, 128, false, false);  // A, B K-major
constexpr uint32_t IDESC_KM = idesc_bf16(256, 128, false, true);   // A K-major, B MN-major

// Shared memory of k_attn_kv, bytes from the 1024-aligned base.  Tiles are 128-byte
// swizzled: [64-element block][rows][128 B].
constexpr uint32_t KV_K = 0;          // K rows of the unit (this CTA's 128 keys x 128)
constexpr uint32_t KV_V = 32768;      // V rows
constexpr uint32_t KV_A = 65536;      // 2 stages: Q then dO of the block, this CTA's 64 queries x 128
constexpr uint32_t KV_A_STAGE = 32768;
constexpr uint32_t KV_B = 131072;     // Q then dO of the block, 128 queries x this CTA's 64 of hd
constexpr uint32_t KV_PT = 163840;    // P^T  [2 query halves][128 keys][128 B]
constexpr uint32_t KV_DST = 196608;   // dS^T [2 query halves][128 keys][128 B]
constexpr uint32_t KV_LD = 229376;    // lse * log2(e) [128], then D [128], of the block's queries
constexpr uint32_t KV_CTRL = 230400;

// Shared memory of k_attn_q.
constexpr uint32_t Q_Q = 0;           // Q rows of the unit (this CTA's 128 queries x 128)
constexpr uint32_t Q_DO = 32768;      // dO rows
constexpr uint32_t Q_X = 65536;       // 2 stages: K then V of the key block, this CTA's 64 keys x 128
constexpr uint32_t Q_X_STAGE = 32768;
constexpr uint32_t Q_Y = 131072;      // 2 stages: K of the key block, 128 keys x this CTA's 64 of hd
constexpr uint32_t Q_Y_STAGE = 16384;
constexpr uint32_t Q_CTRL = 163840;
// Tensor memory of k_attn_q: S [0, 128), dP [128, 256), dQ [256, 384), and two bf16 dS
// buffers of 64 columns (128 keys) at Q_TDS and Q_TDS + 64: the A operand of dQ += dS K.
constexpr uint32_t Q_TDS = 384;

struct CtrlF {
  uint64_t afull[2], aempty[2];  // ring of the S / dP B operands
  uint64_t bfull[2], bempty[2];  // ring of the B operands of the accumulating GEMMs
  uint64_t rfull, rempty;        // the unit's resident A operands
  uint64_t tfull, tempty;        // S and dP accumulators (tempty: leader, one arrival per CTA)
  uint64_t oready, ofree;        // P^T, dS^T (or dS) in shared memory (oready: leader, one per CTA)
  uint64_t tempty_l, oready_l;   // the CTA's epilogue warps, forwarded to tempty / oready
  uint64_t dsfree[2];            // k_attn_q: the dQ GEMM has read dS buffer 0 / 1 (tensor memory)
  uint64_t accempty;             // the unit's accumulators have been read out
  uint64_t lfull, lempty;        // lse / D of the block (k_attn_kv)
  uint64_t sfree;                // the dV / dK staging has left shared memory (k_attn_kv)
  uint64_t mdone;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t SMEM_KV = KV_CTRL + sizeof(CtrlF) + 1024;
constexpr size_t SMEM_Q = Q_CTRL + sizeof(CtrlF) + 1024;
static_assert(SMEM_KV <= 232448, "k_attn_kv shared memory");

__device__ __forceinline__ void prologue_f(CtrlF* c, int warp, int epi) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->afull[i], 1);
      mbar_init(&c->aempty[i], 1);
      mbar_init(&c->bfull[i], 1);
      mbar_init(&c->bempty[i], 1);
    }
    mbar_init(&c->rfull, 1);
    mbar_init(&c->rempty, 1);
    mbar_init(&c->tfull, 1);
    mbar_init(&c->tempty, 2);
    mbar_init(&c->oready, 2);
    mbar_init(&c->tempty_l, epi);
    mbar_init(&c->oready_l, epi);
    mbar_init(&c->ofree, 1);
    mbar_init(&c->dsfree[0], 1);
    mbar_init(&c->dsfree[1], 1);
    mbar_init(&c->accempty, 2 * epi);
    mbar_init(&c->lfull, 1);
    mbar_init(&c->lempty, epi);
    mbar_init(&c->sfree, epi);
    mbar_init(&c->mdone, 1);
    c->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&c->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
}

__device__ __forceinline__ void teardown_f(CtrlF* c, int warp) {
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(c->tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
}

__device__ __forceinline__ void fail_f(CtrlF* c, int32_t* status) {
  *(volatile int*)&c->abort = 1;
  if (status) atomicCAS(status, 0, SBP_ERR_TIMEOUT);
}

// Waits until barrier b has completed `need` phases; `seen` counts the phases this
// thread already waited for.  Bounded like every other wait.
__device__ __forceinline__ bool wait_n(uint64_t* b, uint32_t& seen, uint32_t need, CtrlF* c, uint64_t limit) {
  while (seen < need) {
    if (!wait_inl<true>(b, seen & 1u, &c->abort, limit)) return false;
    ++seen;
  }
  return true;
}
// The same for a whole warp (seen and need are warp-uniform).
__device__ __forceinline__ bool warp_wait_n(uint64_t* b, uint32_t& seen, uint32_t need, CtrlF* c, uint64_t limit) {
  while (seen < need) {
    if (!__all_sync(0xffffffffu, wait_inl<true>(b, seen & 1u, &c->abort, limit))) return false;
    ++seen;
  }
  return true;
}

// The forwarder: for block g, waits for the CTA's 8 epilogue warps on tempty_l, then on
// oready_l, and passes each on to the leader's barrier.
__device__ __forceinline__ bool forward_block(CtrlF* c, uint32_t g, uint32_t& te_seen, uint32_t& or_seen,
                                              uint64_t limit) {
  if (!wait_n(&c->tempty_l, te_seen, g + 1, c, limit)) return false;
  arrive_remote(mapa(saddr(&c->tempty), 0));
  if (!wait_n(&c->oready_l, or_seen, g + 1, c, limit)) return false;
  arrive_remote(mapa(saddr(&c->oready), 0));
  return true;
}

__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z), "r"(src)
               : "memory");
}

// 2^a and 2^b (fp32 special-function unit; measured faster here than the packed
// half-precision form, whose conversions cost more than the halved exp count saves).
__device__ __forceinline__ float2 exp2_pair(float a, float b) { return make_float2(ex2(a), ex2(b)); }

// Descriptor d advanced by `bytes` (a multiple of 16 that keeps the start address inside
// its 14-bit field): one 32-bit add on the low word instead of rebuilding the descriptor
// for every operand and k-step.
__device__ __forceinline__ uint64_t dplus(uint64_t d, uint32_t bytes) {
  return (d & 0xFFFFFFFF00000000ull) | (uint64_t)((uint32_t)d + (bytes >> 4));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Half `half` (64 B = 32 bf16) of row `row` of a 128-byte-swizzled K-major tile: 16-byte
// chunk k of the row sits at chunk k ^ (row % 8), the layout TMA writes and tcgen05.mma
// reads.
__device__ __forceinline__ void store_half_row(uint32_t tile, int row, int half, const uint32_t (&w)[16]) {
  const uint32_t r = tile + (uint32_t)row * 128u;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    sts128(r + ((uint32_t)((4 * half + k) ^ (row & 7)) << 4), w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
}

// tcgen05.mma with A in tensor memory (each CTA's 128 rows in its lanes, two bf16 of
// consecutive K per 32-bit column, the lower K in the low half) and B in shared memory.
__device__ __forceinline__ void mma2_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                             uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// ================================================================ k_attn_kv (dK, dV)

// One round of k_attn_kv's epilogue: 16 queries (columns j0 .. j0+15 of the thread's
// 32-column group) of this thread's key row.  P^T = 2^(s S^T - lse log2 e) and
// dS^T = P^T (dP^T - D), packed to bf16 pairs.  MASK: the round holds queries before the
// key or past the chunk's end (a diagonal block or the ragged tail), which get P = 0; the
// other rounds skip the per-element test (the mask costs more than the math it guards).
template <bool MASK>
__device__ __forceinline__ void kv_round(const uint32_t (&rs)[32], const uint32_t (&rd)[32], int j0,
                                         const float* lds, float sl2, int qg, int key, int c1, uint32_t* pw,
                                         uint32_t* dw) {
  const float4* l4 = reinterpret_cast<const float4*>(lds);
  const float4* d4 = reinterpret_cast<const float4*>(lds + 128);
#pragma unroll
  for (int j4 = 0; j4 < 4; ++j4) {
    const float4 L = l4[j4], Dv = d4[j4];
    const float lz[4] = {L.x, L.y, L.z, L.w}, dz[4] = {Dv.x, Dv.y, Dv.z, Dv.w};
    float pv[4], sv[4];
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      const int j = j0 + 4 * j4 + e;
      const float2 pp = exp2_pair(fmaf(__uint_as_float(rs[j]), sl2, -lz[e]),
                                  fmaf(__uint_as_float(rs[j + 1]), sl2, -lz[e + 1]));
      pv[e] = pp.x;
      pv[e + 1] = pp.y;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = 4 * j4 + e;
      if (MASK && (qg + j < key || qg + j >= c1)) pv[e] = 0.f;
      sv[e] = pv[e] * (__uint_as_float(rd[j0 + j]) - dz[e]);
    }
    pw[2 * j4] = pack_bf16(pv[0], pv[1]);
    pw[2 * j4 + 1] = pack_bf16(pv[2], pv[3]);
    dw[2 * j4] = pack_bf16(sv[0], sv[1]);
    dw[2 * j4 + 1] = pack_bf16(sv[2], sv[3]);
  }
}

struct KvP {
  int H, T, c0, c1, nb, n_units;
  int Hkv, group;    // key / value heads; query heads per key / value head (H = Hkv * group)
  float scale;
  const float* lse;  // [H, T]
  const float* D;    // [H, T]
  int32_t* status;
  uint64_t limit_ns;
};

// Unit u: key / value head zk, keys [256 kp, 256 kp + 256); query blocks b0 .. nb-1 of the
// chunk hold at least one query at or after the unit's first key.  The unit walks those
// blocks for each query head of zk's group (nblk blocks in all), accumulating dV and dK
// of the shared head.  Key pairs in ascending order, so the longest units start first.
__device__ __forceinline__ void kv_unit(const KvP& p, int u, int& zk, int& kp, int& b0, int& nblk) {
  kp = u / p.Hkv;
  zk = u - kp * p.Hkv;
  const int num = 256 * kp - p.c0 - 127;
  b0 = num <= 0 ? 0 : (num + 127) / 128;
  nblk = p.group * (p.nb - b0);
}
// Block n of a unit: query head z of the group, query block b of the chunk.
__device__ __forceinline__ void kv_block(const KvP& p, int zk, int b0, int n, int& z, int& b) {
  const int nbl = p.nb - b0;
  const int gh = n / nbl;
  z = zk * p.group + gh;
  b = b0 + (n - gh * nbl);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(KV_THREADS, 1)
    k_attn_kv(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const __grid_constant__ CUtensorMap tmQa, const __grid_constant__ CUtensorMap tmOa,
              const __grid_constant__ CUtensorMap tmQb, const __grid_constant__ CUtensorMap tmOb,
              const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV, const KvP p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  CtrlF* c = reinterpret_cast<CtrlF*>(base + KV_CTRL);
  const uint32_t sb = saddr(base);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = ctarank();
  prologue_f(c, warp, KV_EPI);
  const uint32_t tmem = c->tmem_base;
  const int pid = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == 0) {
    if (lane == 0) {
      // the unit's K and V, then ring A: Q and dO of each block (this CTA's 64 queries)
      prefetch_map(&tmK);
      prefetch_map(&tmV);
      prefetch_map(&tmQa);
      prefetch_map(&tmOa);
      int sa = 0;
      uint32_t pha = 0, phr = 0, iss = 0, lph_a[2] = {0, 0}, lph_r = 0;
      bool ok = true;
      for (int u = pid; u < p.n_units && ok; u += npairs) {
        int zk, kp, b0, nblk;
        kv_unit(p, u, zk, kp, b0, nblk);
        if (!wait_inl<false>(&c->rempty, phr ^ 1u, &c->abort, p.limit_ns)) { ok = false; break; }
        const uint32_t fr = mapa(saddr(&c->rfull), 0);
        if (rank == 0) mbar_expect_tx(&c->rfull, 4u * 32768u);
        const int krow = 256 * kp + 128 * (int)rank;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          tma_load_3d_pair(sb + KV_K + hb * 16384, &tmK, fr, 64 * hb, krow, zk);
          tma_load_3d_pair(sb + KV_V + hb * 16384, &tmV, fr, 64 * hb, krow, zk);
        }
        iss |= 4u;
        lph_r = phr;
        phr ^= 1u;
        for (int n = 0; n < nblk; ++n) {
          int z, b;
          kv_block(p, zk, b0, n, z, b);
          if (!wait_inl<false>(&c->aempty[sa], pha ^ 1u, &c->abort, p.limit_ns)) { ok = false; break; }
          const uint32_t fa = mapa(saddr(&c->afull[sa]), 0);
          if (rank == 0) mbar_expect_tx(&c->afull[sa], 2u * KV_A_STAGE);
          const uint32_t st = sb + KV_A + sa * KV_A_STAGE;
          const int qrow = p.c0 + 128 * b + 64 * (int)rank;
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            tma_load_3d_pair(st + hb * 8192, &tmQa, fa, 64 * hb, qrow, z);
            tma_load_3d_pair(st + 16384 + hb * 8192, &tmOa, fa, 64 * hb, qrow, z);
          }
          iss |= 1u << sa;
          lph_a[sa] = pha;
          if (++sa == 2) { sa = 0; pha ^= 1u; }
        }
      }
      if (!ok) {
        fail_f(c, p.status);
        if (rank == 0) {
          if (iss & 4u) wait_inl<false>(&c->rfull, lph_r, nullptr, 200000000ull);
          for (int s = 0; s < 2; ++s)
            if (iss & (1u << s)) wait_inl<false>(&c->afull[s], lph_a[s], nullptr, 200000000ull);
        }
      }
    } else if (lane == 16) {
      // ring B (one stage): Q and dO of the block, 128 queries x this CTA's half of hd
      prefetch_map(&tmQb);
      prefetch_map(&tmOb);
      uint32_t phb = 0, lph = 0;
      bool ok = true, any = false;
      for (int u = pid; u < p.n_units && ok; u += npairs) {
        int zk, kp, b0, nblk;
        kv_unit(p, u, zk, kp, b0, nblk);
        for (int n = 0; n < nblk; ++n) {
          int z, b;
          kv_block(p, zk, b0, n, z, b);
          if (!wait_inl<false>(&c->bempty[0], phb ^ 1u, &c->abort, p.limit_ns)) { ok = false; break; }
          const uint32_t fb = mapa(saddr(&c->bfull[0]), 0);
          if (rank == 0) mbar_expect_tx(&c->bfull[0], 4u * 16384u);
          const int qrow = p.c0 + 128 * b;
          tma_load_3d_pair(sb + KV_B, &tmQb, fb, 64 * (int)rank, qrow, z);
          tma_load_3d_pair(sb + KV_B + 16384, &tmOb, fb, 64 * (int)rank, qrow, z);
          any = true;
          lph = phb;
          phb ^= 1u;
        }
      }
      if (!ok) {
        fail_f(c, p.status);
        if (rank == 0 && any) wait_inl<false>(&c->bfull[0], lph, nullptr, 200000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      int sa = 0, lu = 0;
      uint32_t pha = 0, phb = 0, phr = 0, tempty_seen = 0, oready_seen = 0, acc_seen = 0, g = 0;
      bool ok = true;
      const uint64_t dK = sw128_desc(sb + KV_K, 16, 1024), dV = sw128_desc(sb + KV_V, 16, 1024),
                     dA = sw128_desc(sb + KV_A, 16, 1024), dPT = sw128_desc(sb + KV_PT, 16, 1024),
                     dDST = sw128_desc(sb + KV_DST, 16, 1024), dBm = sw128_desc(sb + KV_B, 16384, 1024);
      // dV += P^T dO and dK += dS^T Q for global block gg (the first of its unit overwrites)
      auto accumulate = [&](uint32_t gg, bool first) -> bool {
        if (!wait_n(&c->oready, oready_seen, gg + 1, c, p.limit_ns)) return false;
        if (!wait_inl<false>(&c->bfull[0], phb, &c->abort, p.limit_ns)) return false;
        phb ^= 1u;
        if (first && !wait_n(&c->accempty, acc_seen, (uint32_t)lu, c, p.limit_ns)) return false;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma2_bf16(tmem + 256, dplus(dPT, (k >> 2) * 16384 + (k & 3) * 32), dplus(dBm, 16384 + k * 2048), IDESC_KM,
                    (!first || k) ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma2_bf16(tmem + 384, dplus(dDST, (k >> 2) * 16384 + (k & 3) * 32), dplus(dBm, k * 2048), IDESC_KM,
                    (!first || k) ? 1u : 0u);
        commit2_mc(&c->bempty[0], 3);
        commit2_mc(&c->ofree, 3);
        return true;
      };
      for (int u = pid; u < p.n_units && ok; u += npairs, ++lu) {
        int zk, kp, b0, nbl;
        kv_unit(p, u, zk, kp, b0, nbl);
        if (!wait_inl<false>(&c->rfull, phr, &c->abort, p.limit_ns)) { ok = false; break; }
        phr ^= 1u;
        tc_fence_after();
        for (int n = 0; n < nbl; ++n, ++g) {
          // S^T and dP^T of block g; the previous block's accumulation follows, so the
          // epilogue's work on block g overlaps it
          if (!wait_n(&c->tempty, tempty_seen, g, c, p.limit_ns)) { ok = false; break; }
          if (!wait_inl<false>(&c->afull[sa], pha, &c->abort, p.limit_ns)) { ok = false; break; }
          tc_fence_after();
          const uint64_t dst = dplus(dA, sa * KV_A_STAGE);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma2_bf16(tmem, dplus(dK, (k >> 2) * 16384 + (k & 3) * 32), dplus(dst, (k >> 2) * 8192 + (k & 3) * 32),
                      IDESC_KK, k ? 1u : 0u);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma2_bf16(tmem + 128, dplus(dV, (k >> 2) * 16384 + (k & 3) * 32),
                      dplus(dst, 16384 + (k >> 2) * 8192 + (k & 3) * 32), IDESC_KK, k ? 1u : 0u);
          commit2_mc(&c->aempty[sa], 3);
          commit2_mc(&c->tfull, 3);
          if (n == nbl - 1) commit2_mc(&c->rempty, 3);
          if (++sa == 2) { sa = 0; pha ^= 1u; }
          if (n >= 1 && !accumulate(g - 1, n == 1)) { ok = false; break; }
        }
        if (!ok) break;
        if (!accumulate(g - 1, nbl == 1)) { ok = false; break; }
      }
      if (!ok) fail_f(c, p.status);
      commit2_mc(&c->mdone, 1);
      wait_inl<false>(&c->mdone, 0, nullptr, 200000000ull);
    }
    __syncwarp();
  } else if (warp == KV_FWD_WARP) {
    if (lane == 0) {
      uint32_t te_seen = 0, or_seen = 0, g = 0;
      bool ok = true;
      for (int u = pid; u < p.n_units && ok; u += npairs) {
        int zk, kp, b0, nblk;
        kv_unit(p, u, zk, kp, b0, nblk);
        for (int n = 0; n < nblk; ++n, ++g)
          if (!forward_block(c, g, te_seen, or_seen, p.limit_ns)) { ok = false; break; }
      }
      if (!ok) fail_f(c, p.status);
    }
    __syncwarp();
  } else if (warp == KV_LD_WARP) {
    // lse * log2(e) and D of each block's 128 queries into shared memory (one buffer,
    // refilled once the epilogue warps have read it); loads issued a block ahead
    float* ld = reinterpret_cast<float*>(base + KV_LD);
    uint32_t lempty_seen = 0, g = 0;
    for (int u = pid; u < p.n_units; u += npairs) {
      int zk, kp, b0, nblk;
      kv_unit(p, u, zk, kp, b0, nblk);
      bool ok = true;
      for (int n = 0; n < nblk; ++n, ++g) {
        int z, b;
        kv_block(p, zk, b0, n, z, b);
        float lv[4], dv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int q = p.c0 + 128 * b + lane + 32 * i;
          const bool v = q < p.c1;
          const int64_t o = (int64_t)z * p.T + q;
          lv[i] = v ? p.lse[o] * L2E : 0.f;
          dv[i] = v ? p.D[o] : 0.f;
        }
        if (!warp_wait_n(&c->lempty, lempty_seen, g, c, p.limit_ns)) { ok = false; break; }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ld[lane + 32 * i] = lv[i];
          ld[128 + lane + 32 * i] = dv[i];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&c->lfull);
      }
      if (!ok) {
        fail_f(c, p.status);
        break;
      }
    }
  } else {
    const int q = warp & 3, ch = (warp - 2) >> 2;   // lane quadrant; 64-column half of the block
    const int lrow = q * 32 + lane;
    const uint32_t trow = (uint32_t)(q * 32) << 16;
    const float sl2 = p.scale * L2E;
    const float* ld = reinterpret_cast<const float*>(base + KV_LD);
    uint32_t tfull_seen = 0, ofree_seen = 0, lfull_seen = 0, sfree_seen = 0, g = 0;
    int lu = 0;
    bool ok = true;
    for (int u = pid; u < p.n_units && ok; u += npairs, ++lu) {
      int zk, kp, b0, nblk;
      kv_unit(p, u, zk, kp, b0, nblk);
      const int kw = 256 * kp + 128 * (int)rank + 32 * q;   // this warp's first key
      const int key = kw + lane;
      for (int n = 0; n < nblk; ++n, ++g) {
        int z, b;
        kv_block(p, zk, b0, n, z, b);
        (void)z;
        if (!warp_wait_n(&c->tfull, tfull_seen, g + 1, c, p.limit_ns) ||
            !warp_wait_n(&c->lfull, lfull_seen, g + 1, c, p.limit_ns)) { ok = false; break; }
        tc_fence_after();
        uint32_t pw[2][16], dw[2][16];   // bf16 pairs of P^T and dS^T over this thread's 64 queries
#pragma unroll
        for (int h = 0; h < 2; ++h) {   // the half's two 32-column groups, one after the other
          const int cg = 2 * ch + h;
          uint32_t rs[32], rd[32];
          tmem_ld32(tmem + trow + (uint32_t)(32 * cg), rs);
          tmem_ld32(tmem + trow + (uint32_t)(128 + 32 * cg), rd);
          tmem_ld_wait();
          if (h == 1) {   // S^T and dP^T are all in registers: the next block's may be formed
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&c->tempty_l);
          }
#pragma unroll
          for (int r = 0; r < 2; ++r) {   // two rounds of 16 queries
            const int qg = p.c0 + 128 * b + 32 * cg + 16 * r;   // first query of the round
            const bool none = qg + 15 < kw || qg >= p.c1;
            const bool all = qg >= kw + 31 && qg + 15 < p.c1;
            if (none) {
#pragma unroll
              for (int j = 0; j < 8; ++j) pw[h][8 * r + j] = dw[h][8 * r + j] = 0u;
            } else if (all) {
              kv_round<false>(rs, rd, 16 * r, ld + 32 * cg + 16 * r, sl2, qg, key, p.c1, &pw[h][8 * r], &dw[h][8 * r]);
            } else {
              kv_round<true>(rs, rd, 16 * r, ld + 32 * cg + 16 * r, sl2, qg, key, p.c1, &pw[h][8 * r], &dw[h][8 * r]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&c->lempty);
        // the previous block's accumulation has read P^T and dS^T; at a unit's first
        // block, also the previous unit's dV / dK staging has left this area
        if (!warp_wait_n(&c->ofree, ofree_seen, g, c, p.limit_ns) ||
            (n == 0 && !warp_wait_n(&c->sfree, sfree_seen, (uint32_t)lu, c, p.limit_ns))) { ok = false; break; }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          store_half_row(sb + KV_PT + ch * 16384, lrow, h, pw[h]);
          store_half_row(sb + KV_DST + ch * 16384, lrow, h, dw[h]);
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c->oready_l);
      }
      if (!ok) break;
      // the unit's dV and dK: out of tensor memory, through this warp's 8 KB of the
      // P^T / dS^T area (one 4 KB block per 32 columns), added into the fp32 outputs.
      // Each output element receives one add per launch; rows past T are clipped by the
      // tensor map, rows in [c1, T) add 0.
      if (!warp_wait_n(&c->ofree, ofree_seen, g, c, p.limit_ns)) { ok = false; break; }
      tc_fence_after();
      const uint32_t stg = sb + KV_PT + (uint32_t)(warp - 2) * 8192u;
#pragma unroll 1
      for (int t = 0; t < 2; ++t) {   // t = 0: dV, t = 1: s dK
        uint32_t ra[2][32];
        tmem_ld32(tmem + trow + (uint32_t)((t ? 384 : 256) + 64 * ch), ra[0]);
        tmem_ld32(tmem + trow + (uint32_t)((t ? 384 : 256) + 64 * ch + 32), ra[1]);
        tmem_ld_wait();
        if (t == 1) {   // both accumulators are in registers: the next unit may overwrite them
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_remote(mapa(saddr(&c->accempty), 0));
        }
        if (kw >= p.c1) continue;
        if (t == 1) {
          if (lane == 0) bulk_wait_read();
          __syncwarp();
        }
        const float f = t ? p.scale : 1.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t buf = stg + (uint32_t)h * 4096u + (uint32_t)lane * 128u;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            sts128(buf + ((uint32_t)(k ^ (lane & 7)) << 4), __float_as_uint(__uint_as_float(ra[h][4 * k]) * f),
                   __float_as_uint(__uint_as_float(ra[h][4 * k + 1]) * f),
                   __float_as_uint(__uint_as_float(ra[h][4 * k + 2]) * f),
                   __float_as_uint(__uint_as_float(ra[h][4 * k + 3]) * f));
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(t ? &tmdK : &tmdV, stg, 64 * ch, kw, zk);
          tma_reduce_add_3d(t ? &tmdK : &tmdV, stg + 4096u, 64 * ch + 32, kw, zk);
          bulk_commit();
        }
      }
      if (lane == 0) bulk_wait_read();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c->sfree);
    }
    if (!ok) fail_f(c, p.status);
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  teardown_f(c, warp);
}

// ===================================================================== k_attn_q (dQ)

// One round of k_attn_q's epilogue: 16 keys of this thread's query row.  P = 2^(s S -
// lse log2 e), dS = P (dP - D), packed to bf16 pairs.  MASK: the round holds keys after
// the query (the diagonal block) or the row is past the chunk's end; the other rounds
// skip the per-element test.
template <bool MASK>
__device__ __forceinline__ void q_round(const uint32_t (&rs)[16], const uint32_t (&rd)[16], float sl2, float lz,
                                        float Dq, int kg, int qr, bool vrow, uint32_t* dw) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 pp = exp2_pair(fmaf(__uint_as_float(rs[2 * i]), sl2, -lz),
                                fmaf(__uint_as_float(rs[2 * i + 1]), sl2, -lz));
    float pv[2] = {pp.x, pp.y}, sv[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int jj = 2 * i + e;
      if (MASK && (kg + jj > qr || !vrow)) pv[e] = 0.f;
      sv[e] = pv[e] * (__uint_as_float(rd[jj]) - Dq);
    }
    dw[i] = pack_bf16(sv[0], sv[1]);
  }
}

struct QP {
  int H, T, c0, c1, n_qp, n_units;
  int group;         // query heads per key / value head
  float scale;
  const float* lse;
  const float* D;
  __nv_bfloat16* dQ;  // [H, T, 128]
  int32_t* status;
  uint64_t limit_ns;
};

// Unit u: head z, queries [c0 + 256 qp, +256) of the chunk, key blocks 0 .. nj-1 (128
// keys each) up to the unit's last query.  Later query pairs (more keys) first.
__device__ __forceinline__ void q_unit(const QP& p, int u, int& z, int& qp, int& nj) {
  const int i = u / p.H;
  z = u - i * p.H;
  qp = p.n_qp - 1 - i;
  const int qend = min(p.c0 + 256 * qp + 256, p.c1);
  nj = (qend + 127) / 128;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Q_THREADS, 1)
    k_attn_q(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO,
             const __grid_constant__ CUtensorMap tmKa, const __grid_constant__ CUtensorMap tmVa,
             const __grid_constant__ CUtensorMap tmKb, const QP p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  CtrlF* c = reinterpret_cast<CtrlF*>(base + Q_CTRL);
  const uint32_t sb = saddr(base);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = ctarank();
  prologue_f(c, warp, Q_EPI);
  const uint32_t tmem = c->tmem_base;
  const int pid = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == 0) {
    if (lane == 0) {
      // the unit's Q and dO, then ring X: K and V of each key block (this CTA's 64 keys)
      prefetch_map(&tmQ);
      prefetch_map(&tmO);
      prefetch_map(&tmKa);
      prefetch_map(&tmVa);
      int sa = 0;
      uint32_t pha = 0, phr = 0, iss = 0, lph_a[2] = {0, 0}, lph_r = 0;
      bool ok = true;
      for (int u = pid; u < p.n_units && ok; u += npairs) {
        int z, qp, nj;
        q_unit(p, u, z, qp, nj);
        if (!wait_inl<false>(&c->rempty, phr ^ 1u, &c->abort, p.limit_ns)) { ok = false; break; }
        const uint32_t fr = mapa(saddr(&c->rfull), 0);
        if (rank == 0) mbar_expect_tx(&c->rfull, 4u * 32768u);
        const int qrow = p.c0 + 256 * qp + 128 * (int)rank;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          tma_load_3d_pair(sb + Q_Q + hb * 16384, &tmQ, fr, 64 * hb, qrow, z);
          tma_load_3d_pair(sb + Q_DO + hb * 16384, &tmO, fr, 64 * hb, qrow, z);
        }
        iss |= 4u;
        lph_r = phr;
        phr ^= 1u;
        for (int j = 0; j < nj; ++j) {
          if (!wait_inl<false>(&c->aempty[sa], pha ^ 1u, &c->abort, p.limit_ns)) { ok = false; break; }
          const uint32_t fa = mapa(saddr(&c->afull[sa]), 0);
          if (rank == 0) mbar_expect_tx(&c->afull[sa], 2u * Q_X_STAGE);
          const uint32_t st = sb + Q_X + sa * Q_X_STAGE;
          const int krow = 128 * j + 64 * (int)rank;
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            tma_load_3d_pair(st + hb * 8192, &tmKa, fa, 64 * hb, krow, z / p.group);
            tma_load_3d_pair(st + 16384 + hb * 8192, &tmVa, fa, 64 * hb, krow, z / p.group);
          }
          iss |= 1u << sa;
          lph_a[sa] = pha;
          if (++sa == 2) { sa = 0; pha ^= 1u; }
        }
      }
      if (!ok) {
        fail_f(c, p.status);
        if (rank == 0) {
          if (iss & 4u) wait_inl<false>(&c->rfull, lph_r, nullptr, 200000000ull);
          for (int s = 0; s < 2; ++s)
            if (iss & (1u << s)) wait_inl<false>(&c->afull[s], lph_a[s], nullptr, 200000000ull);
        }
      }
    } else if (lane == 16) {
      // ring Y: K of each key block, 128 keys x this CTA's half of hd (B of dQ += dS K)
      prefetch_map(&tmKb);
      int sy = 0;
      uint32_t phy = 0, iss = 0, lph[2] = {0, 0};
      bool ok = true;
      for (int u = pid; u < p.n_units && ok; u += npairs) {
        int z, qp, nj;
        q_unit(p, u, z, qp, nj);
        for (int j = 0; j < nj; ++j) {
          if (!wait_inl<false>(&c->bempty[sy], phy ^ 1u, &c->abort, p.limit_ns)) { ok = false; break; }
          const uint32_t fb = mapa(saddr(&c->bfull[sy]), 0);
          if (rank == 0) mbar_expect_tx(&c->bfull[sy], 2u * Q_Y_STAGE);
          tma_load_3d_pair(sb + Q_Y + sy * Q_Y_STAGE, &tmKb, fb, 64 * (int)rank, 128 * j, z / p.group);
          iss |= 1u << sy;
          lph[sy] = phy;
          if (++sy == 2) { sy = 0; phy ^= 1u; }
        }
      }
      if (!ok) {
        fail_f(c, p.status);
        if (rank == 0)
          for (int s = 0; s < 2; ++s)
            if (iss & (1u << s)) wait_inl<false>(&c->bfull[s], lph[s], nullptr, 200000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      int sa = 0, sy = 0, lu = 0;
      uint32_t pha = 0, phy = 0, phr = 0, tempty_seen = 0, oready_seen = 0, acc_seen = 0, g = 0;
      bool ok = true;
      const uint64_t dQd = sw128_desc(sb + Q_Q, 16, 1024), dOd = sw128_desc(sb + Q_DO, 16, 1024),
                     dX = sw128_desc(sb + Q_X, 16, 1024), dY = sw128_desc(sb + Q_Y, 16384, 1024);
      // dQ += dS K for global key block gg (the first of its unit overwrites)
      auto accumulate = [&](uint32_t gg, bool first) -> bool {
        if (!wait_n(&c->oready, oready_seen, gg + 1, c, p.limit_ns)) return false;
        if (!wait_inl<false>(&c->bfull[sy], phy, &c->abort, p.limit_ns)) return false;
        if (first && !wait_n(&c->accempty, acc_seen, (uint32_t)lu, c, p.limit_ns)) return false;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma2_bf16_ts(tmem + 256, tmem + Q_TDS + 64 * (gg & 1) + 8 * k,
                       dplus(dY, sy * Q_Y_STAGE + k * 2048), IDESC_KM,
                       (!first || k) ? 1u : 0u);
        commit2_mc(&c->bempty[sy], 3);
        commit2_mc(&c->dsfree[gg & 1], 3);
        if (++sy == 2) { sy = 0; phy ^= 1u; }
        return true;
      };
      for (int u = pid; u < p.n_units && ok; u += npairs, ++lu) {
        int z, qp, nj;
        q_unit(p, u, z, qp, nj);
        if (!wait_inl<false>(&c->rfull, phr, &c->abort, p.limit_ns)) { ok = false; break; }
        phr ^= 1u;
        tc_fence_after();
        for (int n = 0; n < nj; ++n, ++g) {
          if (!wait_n(&c->tempty, tempty_seen, g, c, p.limit_ns)) { ok = false; break; }
          if (!wait_inl<false>(&c->afull[sa], pha, &c->abort, p.limit_ns)) { ok = false; break; }
          tc_fence_after();
          const uint64_t dst = dplus(dX, sa * Q_X_STAGE);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma2_bf16(tmem, dplus(dQd, (k >> 2) * 16384 + (k & 3) * 32), dplus(dst, (k >> 2) * 8192 + (k & 3) * 32),
                      IDESC_KK, k ? 1u : 0u);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma2_bf16(tmem + 128, dplus(dOd, (k >> 2) * 16384 + (k & 3) * 32),
                      dplus(dst, 16384 + (k >> 2) * 8192 + (k & 3) * 32), IDESC_KK, k ? 1u : 0u);
          commit2_mc(&c->aempty[sa], 3);
          commit2_mc(&c->tfull, 3);
          if (n == nj - 1) commit2_mc(&c->rempty, 3);
          if (++sa == 2) { sa = 0; pha ^= 1u; }
          if (n >= 1 && !accumulate(g - 1, n == 1)) { ok = false; break; }
        }
        if (!ok) break;
        if (!accumulate(g - 1, nj == 1)) { ok = false; break; }
      }
      if (!ok) fail_f(c, p.status);
      commit2_mc(&c->mdone, 1);
      wait_inl<false>(&c->mdone, 0, nullptr, 200000000ull);
    }
    __syncwarp();
  } else if (warp == Q_FWD_WARP) {
    if (lane == 0) {
      uint32_t te_seen = 0, or_seen = 0, g = 0;
      bool ok = true;
      for (int u = pid; u < p.n_units && ok; u += npairs) {
        int z, qp, nj;
        q_unit(p, u, z, qp, nj);
        for (int j = 0; j < nj; ++j, ++g)
          if (!forward_block(c, g, te_seen, or_seen, p.limit_ns)) { ok = false; break; }
      }
      if (!ok) fail_f(c, p.status);
    }
    __syncwarp();
  } else {
    const int q = warp & 3, cg = (warp - 2) >> 2;   // lane quadrant, 32-column group
    const uint32_t trow = (uint32_t)(q * 32) << 16;
    const float sl2 = p.scale * L2E;
    uint32_t tfull_seen = 0, g = 0;
    uint32_t ds_seen0 = 0, ds_seen1 = 0, ds_uses0 = 0, ds_uses1 = 0;   // per dS buffer: completions waited, blocks written
    bool ok = true;
    for (int u = pid; u < p.n_units && ok; u += npairs) {
      int z, qp, nj;
      q_unit(p, u, z, qp, nj);
      const int qw = p.c0 + 256 * qp + 128 * (int)rank + 32 * q;   // this warp's first query
      const int qr = qw + lane;                                     // this thread's query
      const bool vrow = qr < p.c1;
      const int64_t ro = (int64_t)z * p.T + qr;
      const float lz = vrow ? p.lse[ro] * L2E : 0.f;
      const float Dq = vrow ? p.D[ro] : 0.f;
      for (int j = 0; j < nj; ++j, ++g) {
        if (!warp_wait_n(&c->tfull, tfull_seen, g + 1, c, p.limit_ns)) { ok = false; break; }
        tc_fence_after();
        uint32_t dw[16];   // bf16 pairs of dS over this thread's 32 keys
#pragma unroll
        for (int r = 0; r < 2; ++r) {   // two rounds of 16 keys
          uint32_t rs[16], rd[16];
          tmem_ld16(tmem + trow + (uint32_t)(32 * cg + 16 * r), rs);
          tmem_ld16(tmem + trow + (uint32_t)(128 + 32 * cg + 16 * r), rd);
          tmem_ld_wait();
          if (r == 1) {   // S and dP are in registers: the next block's may be formed
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&c->tempty_l);
          }
          const int kg = 128 * j + 32 * cg + 16 * r;   // first key of the round
          const bool none = kg > qw + 31 || qw >= p.c1;
          const bool all = kg + 15 <= qw && qw + 31 < p.c1;
          if (none) {
#pragma unroll
            for (int i = 0; i < 8; ++i) dw[8 * r + i] = 0u;
          } else if (all) {
            q_round<false>(rs, rd, sl2, lz, Dq, kg, qr, vrow, &dw[8 * r]);
          } else {
            q_round<true>(rs, rd, sl2, lz, Dq, kg, qr, vrow, &dw[8 * r]);
          }
        }
        // dS into tensor-memory buffer g % 2 once the dQ GEMM of its previous block has read it
        const int bf = (int)(g & 1u);
        if (!(bf ? warp_wait_n(&c->dsfree[1], ds_seen1, ds_uses1, c, p.limit_ns)
                 : warp_wait_n(&c->dsfree[0], ds_seen0, ds_uses0, c, p.limit_ns))) { ok = false; break; }
        tmem_st16(tmem + trow + (uint32_t)(Q_TDS + 64 * bf + 16 * cg), dw);
        tmem_st_wait();
        if (bf) ++ds_uses1; else ++ds_uses0;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c->oready_l);
      }
      if (!ok) break;
      // dQ of the unit's queries: s * accumulator, bf16, this thread's row and 32 of hd (the
      // commit after the last dQ GEMM covers all earlier ones)
      if (!(((g - 1u) & 1u) ? warp_wait_n(&c->dsfree[1], ds_seen1, ds_uses1, c, p.limit_ns)
                            : warp_wait_n(&c->dsfree[0], ds_seen0, ds_uses0, c, p.limit_ns))) { ok = false; break; }
      tc_fence_after();
      uint32_t ra[32];
      tmem_ld32(tmem + trow + (uint32_t)(256 + 32 * cg), ra);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_remote(mapa(saddr(&c->accempty), 0));
      if (vrow) {
        uint4* o = reinterpret_cast<uint4*>(p.dQ + ro * 128 + 32 * cg);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t* v = &ra[8 * k];
          o[k] = make_uint4(pack_bf16(__uint_as_float(v[0]) * p.scale, __uint_as_float(v[1]) * p.scale),
                            pack_bf16(__uint_as_float(v[2]) * p.scale, __uint_as_float(v[3]) * p.scale),
                            pack_bf16(__uint_as_float(v[4]) * p.scale, __uint_as_float(v[5]) * p.scale),
                            pack_bf16(__uint_as_float(v[6]) * p.scale, __uint_as_float(v[7]) * p.scale));
        }
      }
    }
    if (!ok) fail_f(c, p.status);
  }
  teardown_f(c, warp);
}

}  // namespace fa
}  // namespace tc

// ========================================================================== host side

namespace {

// 3-D bf16 map over [H, T, 128] (dims hd, T, H): boxes of 64 x rows x 1, 128-byte swizzle,
// zero fill past T in each head.
bool map3_bf16(CUtensorMap* m, const void* ptr, int64_t T, int64_t H, uint32_t rows) {
  auto enc = tc::encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)T, (cuuint64_t)H};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)T * 128 * 2};
  cuuint32_t box[3] = {64, rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D fp32 map over [H, T, 128] for the dK / dV reduce-adds: 32 x 32 x 1 boxes.
bool map3_f32(CUtensorMap* m, void* ptr, int64_t T, int64_t H) {
  auto enc = tc::encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)T, (cuuint64_t)H};
  cuuint64_t strides[2] = {128 * 4, (cuuint64_t)T * 128 * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool fused_attrs() {
  static int attr_state[64] = {};
  static std::mutex mu;
  return tc::once_per_device(attr_state, mu, [] {
    return cudaFuncSetAttribute(tc::fa::k_attn_kv, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)tc::fa::SMEM_KV) == cudaSuccess &&
           cudaFuncSetAttribute(tc::fa::k_attn_q, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)tc::fa::SMEM_Q) == cudaSuccess;
  });
}

}  // namespace

bool AttnFusedPlan::init(const void* Q, const void* K, const void* V, const void* dO, float* dK_, float* dV_,
                         int64_t T_, int64_t H_, int64_t Hkv_) {
  T = T_;
  H = H_;
  Hkv = Hkv_;
  // query-side operands over H heads, key / value side (and dK, dV) over Hkv heads
  return map3_bf16(&K128, K, T, Hkv, 128) && map3_bf16(&V128, V, T, Hkv, 128) && map3_bf16(&Q64, Q, T, H, 64) &&
         map3_bf16(&O64, dO, T, H, 64) && map3_bf16(&Q128, Q, T, H, 128) && map3_bf16(&O128, dO, T, H, 128) &&
         map3_bf16(&K64, K, T, Hkv, 64) && map3_bf16(&V64, V, T, Hkv, 64) && map3_f32(&dK, dK_, T, Hkv) &&
         map3_f32(&dV, dV_, T, Hkv);
}

cudaError_t attn_fused_kv(const AttnFusedPlan& plan, int64_t c0, int64_t c1, float scale, const float* lse,
                          const float* D, int32_t* status, cudaStream_t s) {
  using namespace tc;
  using namespace tc::fa;
  if (!fused_attrs()) return cudaErrorInvalidConfiguration;
  KvP p;
  p.H = (int)plan.H; p.T = (int)plan.T; p.c0 = (int)c0; p.c1 = (int)c1;
  p.nb = (int)((c1 - c0 + 127) / 128);
  p.Hkv = (int)plan.Hkv;
  p.group = (int)(plan.H / plan.Hkv);
  p.n_units = (int)((c1 + 255) / 256) * p.Hkv;
  p.scale = scale; p.lse = lse; p.D = D; p.status = status; p.limit_ns = wait_limit_ns();
  int pairs = max_pairs((const void*)k_attn_kv, SMEM_KV, KV_THREADS);
  if (pairs > p.n_units) pairs = p.n_units;
  k_attn_kv<<<2 * pairs, KV_THREADS, SMEM_KV, s>>>(plan.K128, plan.V128, plan.Q64, plan.O64, plan.Q128, plan.O128,
                                                   plan.dK, plan.dV, p);
  return cudaGetLastError();
}

cudaError_t attn_fused_q(const AttnFusedPlan& plan, int64_t c0, int64_t c1, float scale, const float* lse,
                         const float* D, void* dQ, int32_t* status, cudaStream_t s) {
  using namespace tc;
  using namespace tc::fa;
  if (!fused_attrs()) return cudaErrorInvalidConfiguration;
  QP p;
  p.H = (int)plan.H; p.T = (int)plan.T; p.c0 = (int)c0; p.c1 = (int)c1;
  p.n_qp = (int)((c1 - c0 + 255) / 256);
  p.n_units = p.n_qp * p.H;
  p.group = (int)(plan.H / plan.Hkv);
  p.scale = scale; p.lse = lse; p.D = D; p.dQ = static_cast<__nv_bfloat16*>(dQ);
  p.status = status; p.limit_ns = wait_limit_ns();
  int pairs = max_pairs((const void*)k_attn_q, SMEM_Q, Q_THREADS);
  if (pairs > p.n_units) pairs = p.n_units;
  k_attn_q<<<2 * pairs, Q_THREADS, SMEM_Q, s>>>(plan.Q128, plan.O128, plan.K64, plan.V64, plan.K128, p);
  return cudaGetLastError();
}

}  // namespace sbp
