// 5th-generation tensor core (tcgen05) building blocks for sm_103a, as inline PTX.
//
// Operands live in shared memory in the K-major layout with 128-byte swizzle, as TMA
// writes it: a [128][kD] fp16 tile is two k-blocks of 64 channels, each [128 rows][128 B]
// (16 KB, 1024-byte aligned); inside each 1024-byte group of 8 rows, 16-byte chunk c of row
// r sits at chunk c ^ (r % 8).  The MMA descriptor names that layout (type 2), the 8-row
// group stride (1024 B), and a start address that advances 32 B per 16-channel K step
// inside a k-block.  Accumulators live in tensor memory (TMEM): for M = 128 with one CTA,
// row i of D is TMEM lane i and column n is column base + n, fp32.  One thread issues the
// MMAs; completion is signalled on an mbarrier by tcgen05.commit; every wait on an
// mbarrier is bounded.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"

namespace mikv {
namespace tc {

constexpr int kTileRows = 128;                 // M = N = 128 rows per operand tile
constexpr int kTileBytes = kTileRows * kD * 2; // 32 KB fp16
constexpr uint32_t kKBlock = kTileRows * 128;  // one 64-channel k-block of a tile (16 KB)

// Byte offset of element (r, k) of a [128][kD] fp16 tile in the swizzled layout.
__host__ __device__ __forceinline__ uint32_t tile_off(int r, int k) {
  return static_cast<uint32_t>((k >> 6) * kKBlock + r * 128 + ((((k & 63) >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}

// Shared-memory matrix descriptor for the swizzled K-major layout: start address, the
// (unused) leading offset, 8-row group stride 1024 B, descriptor version of this
// architecture (bits 46-47 = 1), layout type 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;                  // leading offset (16 B, unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;          // 8-row group stride
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;                  // 128-byte swizzle
  return d;
}

// Instruction descriptor for kind::f16: D fp32, A and B fp16, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A . B^T over K = 16 (one fp16 MMA step).
__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1u : 0u));
}

// D = A . B^T for two [128][kD] tiles at sa / sb (8 MMA steps along K: 4 per k-block).
__device__ __forceinline__ void mma_tile(uint32_t tmem_d, uint32_t sa, uint32_t sb, uint32_t idesc) {
#pragma unroll
  for (int ks = 0; ks < kD / 16; ++ks) {
    const uint32_t off = (ks >> 2) * kKBlock + (ks & 3) * 32;
    mma_f16(tmem_d, smem_desc(sa + off), smem_desc(sb + off), idesc, ks > 0);
  }
}

// The mbarrier at `mbar` completes when every tcgen05 op this thread issued so far is done.
__device__ __forceinline__ void commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(mbar)
               : "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(mbar), "r"(count));
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

// Wait-status bits (mikv_wait_status): the kernel in which a bounded mbarrier wait gave up.
constexpr unsigned kGiveupRowLse = 1u;   // K3 pass 1, row_lse_tc_kernel
constexpr unsigned kGiveupColSum = 2u;   // K3 pass 2, col_sum_tc_kernel
constexpr unsigned kGiveupVwo = 4u;      // K6, vwo_norm_tc_kernel
constexpr unsigned kGiveupPerturb = 8u;  // K9, perturb_tc_kernel
constexpr unsigned kGiveupProbe = 16u;   // wait_probe_kernel (mikv_wait_probe)

// The wait-status word of the translation unit that includes this header (internal
// linkage: one word per source file, each read by that file's wait_giveups()).
static __device__ unsigned g_wait_giveups = 0;

// Called by a thread whose bounded wait gave up: records `bit` in the status word.
__device__ __forceinline__ void report_giveup(unsigned bit) { atomicOr(&g_wait_giveups, bit); }

// Host side: this source file's status word, cleared if `clear`.  Synchronous copies.
static inline int wait_giveups(unsigned* out, bool clear) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_wait_giveups, sizeof(v));
  if (e == cudaSuccess && clear && v) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_wait_giveups, &zero, sizeof(zero));
  }
  if (e != cudaSuccess) return fail(MIKV_ECUDA, "wait_status: %s", cudaGetErrorString(e));
  *out |= v;
  return MIKV_OK;
}

// Wait for phase `parity` of the mbarrier, giving up after `limit` polls; true if it completed.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, long limit) {
  uint32_t done = 0;
  for (long it = 0; it < limit && !done; ++it) {
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(mbar), "r"(parity)
        : "memory");
  }
  return done != 0;
}

constexpr long kWaitPolls = 1L << 22;              // polls before a wait gives up
constexpr long kWaitPollsAfterGiveup = 1L << 10;   // polls of each later wait of that thread

// One thread's waits.  After its first give-up (`ok` false) the thread issues no further
// copies or MMAs (the producers test `ok` before each) and its remaining waits poll briefly,
// so that a stuck pipeline still ends in a bounded time; the kernel then marks its outputs
// and sets its status bit.
struct Waits {
  bool ok = true;
  long polls = kWaitPolls;
  __device__ __forceinline__ bool operator()(uint32_t mbar, uint32_t parity) {
    const bool done = mbar_wait(mbar, parity, ok ? polls : kWaitPollsAfterGiveup);
    ok = ok && done;
    return done;
  }
};

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// Shared-memory writes of the generic proxy (cp.async, st.shared) visible to the tensor core.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// TMEM allocation by one full warp: writes the base address to `slot` (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(slot), "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(base), "r"(ncols));
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes 32*(w%4)..).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// One thread: expect `bytes` of asynchronous copies on the mbarrier (one arrival).
__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(mbar), "r"(bytes) : "memory");
}
// One arrival on the mbarrier.
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(mbar) : "memory");
}

// One thread: TMA-load rows [row0, row0 + 128) of a [rows][kD] fp16 matrix described by the
// 2-D tensor map `tmap` (box 64 channels x 128 rows, 128-byte swizzle) into the tile at `s`
// (1024-byte aligned): two boxes, one per k-block (x = 0 and 64).  Rows past the end of the
// matrix are zero-filled.  Completes 32 KB on the mbarrier.
__device__ __forceinline__ void tma_tile(uint32_t s, const void* tmap, int row0, uint32_t mbar) {
#pragma unroll
  for (int j = 0; j < kD / 64; ++j)
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(s + j * kKBlock),
        "l"(tmap), "r"(j * 64), "r"(row0), "r"(mbar)
        : "memory");
}

// One thread: bulk-copy `bytes` (multiple of 16, both addresses 16-byte aligned) into
// shared memory, completing on the mbarrier.
__device__ __forceinline__ void bulk_copy(uint32_t s, const void* g, uint32_t bytes, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(s),
      "l"(g), "r"(bytes), "r"(mbar)
      : "memory");
}

// ---------------------------------------------------------------------------------
// CTA scaffolding of the warp-specialised tile pipelines: one producer lane (TMA + MMA
// issue) and `consumers` threads that read the accumulators.
struct Bars {
  uint64_t load[2];   // operand buffer b filled (TMA bytes)
  uint64_t mma[2];    // accumulator b written (tcgen05.commit)
  uint64_t freed[2];  // accumulator b read by all consumer threads
  uint64_t fixed;     // the resident operand tile filled
};

// mbarriers and the TMEM allocation (`cols` columns); returns the TMEM base.  Every thread
// of the CTA calls it (it holds a barrier).
__device__ __forceinline__ uint32_t cta_setup(Bars& bar, uint32_t* tslot, int consumers, uint32_t cols) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar.load[i]), 1);
      mbar_init(smem_u32(&bar.mma[i]), 1);
      mbar_init(smem_u32(&bar.freed[i]), consumers);
    }
    mbar_init(smem_u32(&bar.fixed), 1);
    mbar_init_fence();
  }
  if (threadIdx.x < 32) tmem_alloc(smem_u32(tslot), cols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  return *tslot;
}
// ---------------------------------------------------------------------------------
// Ring pipeline of the warp-specialised kernels: resident operand tiles plus a stream of
// operand tiles through R shared-memory buffers, and NACC TMEM accumulators.  One producer
// lane issues the TMA copies and the MMAs; step s reads buffer s % R and writes accumulator
// s % NACC; consumer threads read each accumulator and release it.
//   full[b]   buffer b landed (TMA transaction bytes)
//   empty[b]  the MMAs that read buffer b are done (tcgen05.commit)
//   mma[a]    accumulator a written (tcgen05.commit)
//   freed[a]  accumulator a read by its consumers (`consumers` arrivals)
//   fixed     the resident tiles landed
template <int R, int NACC>
struct Ring {
  uint64_t full[R], empty[R], mma[NACC], freed[NACC], fixed;
};

// mbarriers and the TMEM allocation (`cols` columns); returns the TMEM base.  Every thread
// of the CTA calls it (it holds a barrier).
template <int R, int NACC>
__device__ __forceinline__ uint32_t ring_setup(Ring<R, NACC>& r, uint32_t* tslot, int consumers, uint32_t cols) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < R; ++i) {
      mbar_init(smem_u32(&r.full[i]), 1);
      mbar_init(smem_u32(&r.empty[i]), 1);
    }
    for (int i = 0; i < NACC; ++i) {
      mbar_init(smem_u32(&r.mma[i]), 1);
      mbar_init(smem_u32(&r.freed[i]), consumers);
    }
    mbar_init(smem_u32(&r.fixed), 1);
    mbar_init_fence();
  }
  if (threadIdx.x < 32) tmem_alloc(smem_u32(tslot), cols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  return *tslot;
}

// Consumer side of step s: wait for its accumulator; release it after the last tcgen05.ld.
template <int R, int NACC>
__device__ __forceinline__ void ring_acquire(Ring<R, NACC>& r, int s, Waits& w) {
  w(smem_u32(&r.mma[s % NACC]), (s / NACC) & 1);
  fence_after_sync();
}
template <int R, int NACC>
__device__ __forceinline__ void ring_release(Ring<R, NACC>& r, int s) {
  fence_before_sync();
  mbar_arrive(smem_u32(&r.freed[s % NACC]));
}

// Consumer-only barrier (named barrier 1; the producer warp does not take part).
template <int N>
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;\n" ::"n"(N) : "memory");
}

// Every thread of the CTA calls it after its last TMEM access.
__device__ __forceinline__ void cta_teardown(uint32_t tbase, uint32_t cols) {
  fence_before_sync();
  __syncthreads();
  if (threadIdx.x < 32) tmem_dealloc(tbase, cols);
}
// 1024-byte aligned base of the dynamic shared memory (swizzled TMA destinations).
__device__ __forceinline__ uint32_t smem_base(uint8_t* sm) { return (smem_u32(sm) + 1023u) & ~1023u; }

// ---------------------------------------------------------------------------------
// Host: 2-D tensor map of a row-major [rows][cols] fp16 matrix (cols a multiple of 64)
// with a 64-column x box_rows box (128 by default) and 128-byte swizzle, through the driver's encoder
// (looked up once).  `what` names the caller in the error message.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    (void)cudaGetLastError();
  });
  return fn;
}
inline int encode_rows(CUtensorMap* map, const void* base, long rows, const char* what, long cols = kD,
                       int box_rows = kTileRows) {
  const auto enc = tensor_map_encoder();
  if (!enc) return fail(MIKV_ECUDA, "%s: cuTensorMapEncodeTiled unavailable", what);
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides,
                         box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MIKV_ECUDA, "%s: tensor map (error %d)", what, static_cast<int>(r));
  return MIKV_OK;
}

}  // namespace tc
}  // namespace mikv
