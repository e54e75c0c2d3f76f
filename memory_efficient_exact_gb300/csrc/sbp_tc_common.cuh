// Shared machinery of the tcgen05 kernels (sm_103a): PTX wrappers for mbarriers,
// TMA, tensor memory and tcgen05.mma, the SM-pair (cta_group::2) protocol, and the
// host-side tensor-map builders.  Included by the translation units that define
// pair GEMM kernels; every wait in here is bounded in time.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <climits>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include "sbp_internal.h"

namespace sbp {
namespace tc {

constexpr int BN = 256, BK = 64;
constexpr uint32_t BOX_BYTES = 64 * 64 * 2; // one 64x64 bf16 box (MN-major operands)
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_THREADS = 64 + NUM_EPI_WARPS * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr int RING = 4;
constexpr float L2E = 1.4426950408889634f;

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9, 10-12 = 1), A / B major-ness (bit 15 / 16: 0 = K-major, 1 = MN-major),
// N >> 3 at bit 17, M >> 4 at bit 24.
constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(saddr(b)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(saddr(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(saddr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Waits for the phase of parity `parity` of barrier b.  Returns false when the time
// limit passes or (if abort_flag is given) another role of the CTA has aborted.
static __device__ __noinline__ bool wait_slow(uint64_t* b, uint32_t parity, const volatile int* abort_flag,
                                       uint64_t limit_ns) {
  const uint64_t t0 = gtimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(b, parity)) return true;
    if ((i & 15u) == 0) {
      if (abort_flag && *abort_flag) return false;
      if (gtimer() - t0 > limit_ns) return false;
    }
  }
}
__device__ __forceinline__ bool wait_bounded(uint64_t* b, uint32_t parity, const volatile int* abort_flag,
                                             uint64_t limit_ns) {
  if (mbar_try(b, parity)) return true;
  return wait_slow(b, parity, abort_flag, limit_ns);
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }


// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2), version 1 (bit 46).
// K-major tiles: rows of 128 B, 8-row groups 1024 B apart (SBO); LBO unused.
// MN-major tiles: K rows of 128 B (64 MN elements), 8-row K groups 1024 B apart (SBO),
// consecutive 64-element MN blocks LBO bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}


__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ============================================================================ pair protocol
//   full[s]   (leader only) completes when both CTAs' TMA copies of stage s landed: the
//             leader expects 64 KB, the peer's copies complete on it across the pair
//   empty[s]  (both) the leader's MMA commit, multicast to the pair, frees stage s
//   tfull[b]  (both) the leader's commit, multicast: accumulator b is ready
//   tempty[b] (leader) all 16 epilogue warps of the pair drained accumulator b
//   rfull/rempty  the work queue of k_bwd: the leader takes a unit and writes it into
//             both CTAs' rings (distributed shared memory)

constexpr int STAGES = 6;
constexpr uint32_t A_BYTES = 128 * BK * 2;   // 16 KB: this CTA's 128 rows of A
constexpr uint32_t B_BYTES = 128 * BK * 2;   // 16 KB: this CTA's 128 rows of B
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t PAIR_TX = 2 * STAGE_BYTES;  // bytes that complete one leader full barrier
constexpr uint32_t IDESC_FWD = idesc_bf16(256, 256, false, false);
constexpr uint32_t IDESC_DH = idesc_bf16(256, 256, false, true);
constexpr uint32_t IDESC_DW = idesc_bf16(256, 256, true, true);

struct Ctrl {
  uint64_t full[STAGES], empty[STAGES];
  uint64_t tfull[2], tempty[2];
  uint64_t rfull[RING], rempty[RING];
  uint64_t mdone;
  int ring[RING];
  uint32_t tmem_base;
  int abort;
};
__device__ __forceinline__ uint32_t ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Arrival on a barrier of the pair with the instruction's default semantics (release at
// CTA scope), about 500 cycles against about 1300 for the cluster-scope release above
// (measured on GB300).  Used where the arriving thread has already acquired what it
// passes on (a forwarder) or where the protected data is tensor memory that has been
// read out (tcgen05.wait::ld done before the arrival).
__device__ __forceinline__ void arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool try_cluster(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(saddr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait with cluster-scope acquire (barriers that remote CTAs arrive on).
static __device__ __noinline__ bool wait_cluster_slow(uint64_t* b, uint32_t parity, const volatile int* abort_flag,
                                               uint64_t limit_ns) {
  const uint64_t t0 = gtimer();
  for (uint32_t i = 1;; ++i) {
    if (try_cluster(b, parity)) return true;
    if ((i & 15u) == 0) {
      if (abort_flag && *abort_flag) return false;
      if (gtimer() - t0 > limit_ns) return false;
    }
  }
}
__device__ __forceinline__ bool wait_cluster(uint64_t* b, uint32_t parity, const volatile int* abort_flag,
                                             uint64_t limit_ns) {
  if (try_cluster(b, parity)) return true;
  return wait_cluster_slow(b, parity, abort_flag, limit_ns);
}
// The same two waits with the spin loop inlined instead of called: no call-site register
// saves (the fused attention kernels use these: k_attn_q then needs no local memory, and
// the pair ran about 1% faster).  A register split between warpgroups (setmaxnreg) also
// requires it, since a call would run under the kernel-wide register count.
template <bool CLUSTER>
__device__ __forceinline__ bool wait_inl(uint64_t* b, uint32_t parity, const volatile int* abort_flag,
                                         uint64_t limit_ns) {
  if (CLUSTER ? try_cluster(b, parity) : mbar_try(b, parity)) return true;
  const uint64_t t0 = gtimer();
  for (uint32_t i = 1;; ++i) {
    if (CLUSTER ? try_cluster(b, parity) : mbar_try(b, parity)) return true;
    if ((i & 15u) == 0) {
      if (abort_flag && *abort_flag) return false;
      if (gtimer() - t0 > limit_ns) return false;
    }
  }
}
__device__ __forceinline__ bool warp_wait_cluster(uint64_t* b, uint32_t parity, Ctrl* c, uint64_t limit) {
  const bool ok = wait_cluster(b, parity, &c->abort, limit);
  return __all_sync(0xffffffffu, ok);
}

// TMA load into this CTA's shared memory whose completion is counted on an mbarrier
// that may live in the peer CTA (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t mbar_cluster, int x,
                                                 int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar_cluster)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t mbar_cluster, int x,
                                                 int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(mbar_cluster)
      : "memory");
}
__device__ __forceinline__ void mma2_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// Arrive (once the MMAs issued so far complete) on the barrier at this offset in every
// CTA of `mask`.
__device__ __forceinline__ void commit2_mc(uint64_t* bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   saddr(bar)),
               "h"(mask)
               : "memory");
}

__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void fail(Ctrl* c, int32_t* status) {
  *(volatile int*)&c->abort = 1;
  if (status) atomicCAS(status, 0, SBP_ERR_TIMEOUT);
}

__device__ __forceinline__ void prologue(Ctrl* c, int warp) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&c->full[i], 1);
      mbar_init(&c->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->tfull[i], 1);
      mbar_init(&c->tempty[i], 2 * NUM_EPI_WARPS);
    }
    for (int i = 0; i < RING; ++i) {
      mbar_init(&c->rfull[i], 1);
      // leader: its MMA thread and epilogue warps, the peer's producer and epilogue warps
      mbar_init(&c->rempty[i], 2 + 2 * NUM_EPI_WARPS);
    }
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

__device__ __forceinline__ void drain_copies(Ctrl* c, const uint32_t* last_phase, uint32_t issued_mask) {
  for (int s = 0; s < STAGES; ++s)
    if (issued_mask & (1u << s)) wait_bounded(&c->full[s], last_phase[s], nullptr, 200000000ull);
}

__device__ __forceinline__ void teardown(Ctrl* c, int warp) {
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(c->tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
}

// Epilogue arrival on the leader's tempty[buf]: one per warp.
__device__ __forceinline__ void release_tmem(Ctrl* c, int buf, int lane) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) arrive_cluster(mapa(saddr(&c->tempty[buf]), 0));
}


// ------------------------------------------------- per-warp staging blocks (epilogues)
// A warp's staging block is 32 rows of 128 bytes with the 128-byte swizzle TMA uses:
// row `lane` is the lane's row, its 16-byte chunk k at chunk k ^ (lane % 8).

// Row `lane` of a warp's staging block: 16-byte chunks k0 .. k0+3 from w (chunk k at
// chunk k ^ (lane % 8)).
__device__ __forceinline__ void stage4(uint32_t stg, int lane, int k0, const uint32_t* w) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
    sts128(stg + lane * 128 + (((k0 + k) ^ (lane & 7)) << 4), w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
}
// Hands the staging block to TMA (store at column x, row y of `map`) once the previous
// contents have been read out; the next write must wait for this one to be read.
__device__ __forceinline__ void stage_store(const CUtensorMap* map, uint32_t stg, int lane, int x, int y) {
  fence_proxy_async();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, stg, x, y);
    bulk_commit();
  }
}
__device__ __forceinline__ void stage_free(int lane) {
  if (lane == 0) bulk_wait_read();
  __syncwarp();
}
// TMA load of a 32 x 64 block of `map` at column x, row y into this warp's staging block,
// completing on the warp's mbarrier; waits for it (bounded) and returns whether it came.
// The block's previous readers are this warp's lanes: their generic-proxy reads are
// ordered before the asynchronous write by the proxy fence and the warp barrier.
__device__ __forceinline__ bool stage_load(const CUtensorMap* map, uint32_t stg, uint32_t bytes, uint64_t* bar,
                                           uint32_t& phase, int lane, int x, int y, Ctrl* c, uint64_t limit) {
  fence_proxy_async();
  __syncwarp();
  if (lane == 0) {
    mbar_expect_tx(bar, bytes);
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            stg),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(saddr(bar))
        : "memory");
  }
  const bool ok = __all_sync(0xffffffffu, wait_bounded(bar, phase, &c->abort, limit));
  phase ^= 1u;
  return ok;
}
// Row `lane` of the warp's staging block (64 bf16 as 32 words), undoing the swizzle.
__device__ __forceinline__ void stage_read_row(uint32_t stg, int lane, uint32_t (&w)[32]) {
#pragma unroll
  for (int k = 0; k < 8; ++k)
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[4 * k]), "=r"(w[4 * k + 1]), "=r"(w[4 * k + 2]), "=r"(w[4 * k + 3])
                 : "r"(stg + lane * 128 + ((k ^ (lane & 7)) << 4))
                 : "memory");
}
constexpr uint32_t IDESC_KK = idesc_bf16(256, 256, false, false);
constexpr uint32_t IDESC_KM = idesc_bf16(256, 256, false, true);

__device__ __forceinline__ float sigmoid_fast(float t) { return __fdividef(1.f, 1.f + ex2(-t * L2E)); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
}


// ================================================================================ host side

inline PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D bf16 tensor map over a row-major [outer, inner] array with a row stride of
// row_elems elements, 128-byte swizzle, zero fill outside the array.
// 2-D fp32 tensor map for the dW output: [outer, inner] row-major, 32x32 boxes of
// 128-byte rows, 128-byte swizzle.
inline bool make_map_f32(CUtensorMap* m, void* ptr, uint64_t inner, uint64_t outer) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D fp32 tensor map over [planes, outer, inner] (contiguous), 32x32x1 boxes of 128-byte
// rows, 128-byte swizzle.
inline bool make_map3_f32(CUtensorMap* m, void* ptr, uint64_t inner, uint64_t outer, uint64_t planes) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {inner, outer, planes};
  cuuint64_t strides[2] = {inner * 4, inner * outer * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t row_elems, uint32_t box_in,
              uint32_t box_out) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_elems * 2};
  cuuint32_t box[2] = {box_in, box_out};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MN-major bf16 operand map that loads 128 columns in one copy: the [outer, row_elems]
// matrix (row_elems a multiple of 64) seen as [row_elems / 64][outer][64], box 64 x 64 x 2.
// The two 64-column blocks land 8 KB apart in shared memory with the 128-byte swizzle,
// exactly where two 64 x 64 boxes of the two-dimensional map would.  Columns of the last
// block are real memory of the row (row_elems is the row stride), so nothing past the
// allocation is read; columns past the matrix's logical width hold what the buffer holds
// there, which only reaches outputs that the stores clip.
inline bool make_map_mn2(CUtensorMap* m, const void* ptr, uint64_t outer, uint64_t row_elems) {
  if (row_elems % 64 != 0) return false;
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {64, outer, row_elems / 64};
  cuuint64_t strides[2] = {row_elems * 2, 128};
  cuuint32_t box[3] = {64, 64, 2};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Failure-detection test hook: SBP_FAULT_STALL=1 makes the next forward kernels stall
// on purpose (read at every launch, so a test can switch it off again).  Together with a
// short SBP_WAIT_LIMIT_MS it exercises the bounded-wait abort path: status
// SBP_ERR_TIMEOUT, copies drained, tensor memory freed, the context still usable.
inline int fault_stall_requested() {
  const char* e = std::getenv("SBP_FAULT_STALL");
  return (e && e[0] == '1') ? 1 : 0;
}

inline uint64_t wait_limit_ns() {
  static uint64_t v = [] {
    const char* e = std::getenv("SBP_WAIT_LIMIT_MS");
    long long ms = e ? std::atoll(e) : 0;
    if (ms <= 0) ms = 2000;
    return (uint64_t)ms * 1000000ull;
  }();
  return v;
}

// Runs `set` (the cudaFuncSetAttribute calls of one kernel family) once for the current
// device: function attributes are per device, so a process driving several GPUs sets
// them on each.  Returns whether they are set.
template <class F>
inline bool once_per_device(int (&state)[64], std::mutex& mu, F set) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lk(mu);
  if (state[dev] == 0) state[dev] = set() ? 1 : -1;
  return state[dev] == 1;
}

// Clusters of two (SM pairs) of `kernel` that can be resident at once, cached per
// device and kernel.
inline int max_pairs(const void* kernel, size_t smem_bytes, int threads = NUM_THREADS) {
  struct Entry { const void* k; int dev; int n; };
  static Entry cache[32] = {};
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(mu);
  for (auto& e : cache)
    if (e.k == kernel && e.dev == dev && e.n > 0) return e.n;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 76, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = num_sms() / 2;
  }
  for (auto& e : cache)
    if (e.k == nullptr) {
      e = {kernel, dev, n};
      break;
    }
  return n;
}

}  // namespace tc
}  // namespace sbp
