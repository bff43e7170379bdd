// K1: channel balancer b = sqrt(max|q| / max|k|) over the prompt.
//
// Source: "No Token Left Behind" reading notes (velog), "Key contributions, 2)
// Outlier-aware handling", balancer equation; paperlayer summary of arXiv
// 2402.18096v1, section 3.2 (balancer computed once at prefill).
//
// One HBM pass over the prompt's Q and K.  Grid (B*Hkv, nsplit): each CTA scans a
// slice of the (rep*T) query rows and T key rows of one (batch, key head) with
// 16-byte loads (16 threads cover one 256-byte row), keeps per-channel |x| maxima
// in half precision (max of fp16 values is exact), reduces them in shared memory
// and folds them into the workspace with an integer atomicMax on the float bits
// (non-negative floats order like their bit patterns, so the result does not
// depend on the order).  A second kernel forms b in fp32, RN division then RN
// square root.
#include <algorithm>

#include "common.cuh"

namespace mikv {
namespace {

constexpr int kBalThreads = 256;
constexpr int kRowsPerIter = kBalThreads / 16;  // 16 rows of 256 B per CTA iteration

__device__ __forceinline__ void absmax8(uint4 v, __half2 (&m)[4]) {
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = __hmax2(m[i], __habs2(h[i]));
}

__device__ void scan_rows(const uint4* base, long rows, long r0, long r1, float* ws_out,
                          float (*red)[kD]) {
  const int tid = threadIdx.x;
  const int col = tid & 15;          // 16-byte chunk of the row: channels 8*col..8*col+7
  const int rsub = tid >> 4;         // row within an iteration
  __half2 m[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = __float2half2_rn(0.f);
  long r = r0 + rsub;
  // 4 independent loads in flight per thread
  for (; r + 3 * kRowsPerIter < r1; r += 4 * kRowsPerIter) {
    uint4 v0 = __ldg(base + (r)*16 + col);
    uint4 v1 = __ldg(base + (r + kRowsPerIter) * 16 + col);
    uint4 v2 = __ldg(base + (r + 2 * kRowsPerIter) * 16 + col);
    uint4 v3 = __ldg(base + (r + 3 * kRowsPerIter) * 16 + col);
    absmax8(v0, m);
    absmax8(v1, m);
    absmax8(v2, m);
    absmax8(v3, m);
  }
  for (; r < r1; r += kRowsPerIter) absmax8(__ldg(base + r * 16 + col), m);
  (void)rows;
  // CTA reduction over the 16 row lanes of each channel
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __half22float2(m[i]);
    red[rsub][col * 8 + 2 * i] = f.x;
    red[rsub][col * 8 + 2 * i + 1] = f.y;
  }
  __syncthreads();
  if (tid < kD) {
    float mx = 0.f;
#pragma unroll
    for (int j = 0; j < kRowsPerIter; ++j) mx = fmaxf(mx, red[j][tid]);
    atomic_max_nonneg(ws_out + tid, mx);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kBalThreads) balance_max_kernel(
    const uint4* __restrict__ q, const uint4* __restrict__ k, int Hq, int Hkv, int T, int nsplit,
    float* __restrict__ ws_q, float* __restrict__ ws_k) {
  __shared__ float red[kRowsPerIter][kD];
  const int unit = blockIdx.x;  // b*Hkv + g
  const int split = blockIdx.y;
  const int b = unit / Hkv, g = unit % Hkv;
  const int rep = Hq / Hkv;
  // query rows of the group's heads are contiguous: [b][g*rep .. g*rep+rep)[T]
  const long qrows = static_cast<long>(rep) * T;
  const uint4* qb = q + (static_cast<long>(b) * Hq + static_cast<long>(g) * rep) * T * 16;
  const long qs0 = qrows * split / nsplit, qs1 = qrows * (split + 1) / nsplit;
  scan_rows(qb, qrows, qs0, qs1, ws_q + static_cast<long>(unit) * kD, red);
  const uint4* kb = k + static_cast<long>(unit) * T * 16;
  const long ks0 = static_cast<long>(T) * split / nsplit;
  const long ks1 = static_cast<long>(T) * (split + 1) / nsplit;
  scan_rows(kb, T, ks0, ks1, ws_k + static_cast<long>(unit) * kD, red);
}

__global__ void balance_finalize_kernel(const float* __restrict__ ws_q,
                                        const float* __restrict__ ws_k, float* __restrict__ b,
                                        int n) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float mq = ws_q[i], mk = ws_k[i];
  b[i] = (mq == 0.f || mk == 0.f) ? 1.f : __fsqrt_rn(__fdiv_rn(mq, mk));
}

}  // namespace
}  // namespace mikv

using namespace mikv;

extern "C" size_t mikv_balance_workspace_bytes(int B, int Hkv, int D) {
  if (B <= 0 || Hkv <= 0 || D <= 0) return 0;
  return 2 * align_up(static_cast<size_t>(B) * Hkv * D * sizeof(float), 256);
}

extern "C" int mikv_balance_prefill(const uint16_t* q, const uint16_t* k, int B, int Hq, int Hkv,
                                    int T, int D, float* b_out, void* ws, size_t ws_bytes,
                                    void* stream) {
  clear_error();
  if (!q || !k || !b_out || !ws) return fail(MIKV_EINVAL, "balance_prefill: null pointer");
  if (D != kD) return fail(MIKV_EUNSUPPORTED, "balance_prefill: D=%d (only %d)", D, kD);
  if (B < 1 || Hkv < 1 || Hq < Hkv || Hq % Hkv || Hq / Hkv > 8 || T < 1)
    return fail(MIKV_ESHAPE, "balance_prefill: bad shape B=%d Hq=%d Hkv=%d T=%d", B, Hq, Hkv, T);
  if (!aligned16(q) || !aligned16(k) || !aligned16(ws))
    return fail(MIKV_EALIGN, "balance_prefill: q, k and ws must be 16-byte aligned");
  const size_t need = mikv_balance_workspace_bytes(B, Hkv, D);
  if (ws_bytes < need) return fail(MIKV_ESHAPE, "balance_prefill: workspace %zu < %zu", ws_bytes, need);
  cudaStream_t s = as_stream(stream);
  const size_t half = need / 2;
  float* ws_q = static_cast<float*>(ws);
  float* ws_k = reinterpret_cast<float*>(static_cast<char*>(ws) + half);
  if (cudaMemsetAsync(ws, 0, need, s) != cudaSuccess) return check_launch("balance_prefill memset");
  const int units = B * Hkv;
  // enough CTAs for ~4 per SM, each scanning at least 64 query rows
  const long qrows = static_cast<long>(Hq / Hkv) * T;
  int nsplit = (4 * kNumSMs + units - 1) / units;
  nsplit = static_cast<int>(std::min<long>(nsplit, std::max<long>(1, qrows / 64)));
  dim3 grid(units, nsplit);
  balance_max_kernel<<<grid, kBalThreads, 0, s>>>(reinterpret_cast<const uint4*>(q),
                                                  reinterpret_cast<const uint4*>(k), Hq, Hkv, T,
                                                  nsplit, ws_q, ws_k);
  if (int e = check_launch("balance_max_kernel")) return e;
  const int n = units * D;
  balance_finalize_kernel<<<(n + 255) / 256, 256, 0, s>>>(ws_q, ws_k, b_out, n);
  return check_launch("balance_finalize_kernel");
}

// ---------------------------------------------------------------------------------
// Allocation-free variant of mikv_balance_prefill.
//
// Some callers cannot allocate device memory for the workspace: a plugin that a host
// framework hands only its input and output buffers, or a serving loop that must never
// reach the allocator (cudaMalloc and cudaFree synchronise the device and can fail under
// memory pressure).  This entry point keeps its scratch (the per-channel query and key
// maxima) in a fixed static device array instead.  The array is sized for
// kNoAllocMaxUnits (batch x key heads) units of 128 channels, 1 MiB in total, and every
// device that loads the library holds it until the process exits.
namespace mikv {
namespace {

constexpr int kNoAllocMaxUnits = 1024;
constexpr int kNoAllocFloats = 2 * kNoAllocMaxUnits * kD;  // Mq then Mk
static __device__ __align__(256) float g_balance_scratch[kNoAllocFloats];

// Device address of g_balance_scratch in the context current on this thread, looked up on
// every call.  (In host code the symbol is only a host-side stand-in, never a device
// address.)  The lookup is not cached: after cudaDeviceReset, or under another context on
// the same device, the array lives at a different address, and a cached one would point at
// memory that no longer belongs to it.  The lookup allocates nothing.
int scratch_for_current_context(float** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_balance_scratch);
  if (e != cudaSuccess || !p)
    return fail(MIKV_ECUDA, "balance_prefill_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
  *out = static_cast<float*>(p);
  return MIKV_OK;
}

}  // namespace
}  // namespace mikv

extern "C" int mikv_balance_prefill_noalloc(const uint16_t* q, const uint16_t* k, int B, int Hq,
                                            int Hkv, int T, int D, float* b_out, void* stream) {
  clear_error();
  if (!q || !k || !b_out) return fail(MIKV_EINVAL, "balance_prefill_noalloc: null pointer");
  if (D != kD) return fail(MIKV_EUNSUPPORTED, "balance_prefill_noalloc: D=%d (only %d)", D, kD);
  if (B < 1 || Hkv < 1 || Hq < Hkv || Hq % Hkv || Hq / Hkv > 8 || T < 1)
    return fail(MIKV_ESHAPE, "balance_prefill_noalloc: bad shape B=%d Hq=%d Hkv=%d T=%d", B, Hq, Hkv, T);
  if (static_cast<long>(B) * Hkv > kNoAllocMaxUnits)
    return fail(MIKV_ESHAPE,
                "balance_prefill_noalloc: B*Hkv=%ld exceeds the static scratch limit of %d "
                "(batch x key heads); use mikv_balance_prefill with a workspace",
                static_cast<long>(B) * Hkv, kNoAllocMaxUnits);
  if (!aligned16(q) || !aligned16(k))
    return fail(MIKV_EALIGN, "balance_prefill_noalloc: q and k must be 16-byte aligned");
  float* scratch = nullptr;
  if (int e = scratch_for_current_context(&scratch)) return e;
  cudaStream_t s = as_stream(stream);
  const int units = B * Hkv;
  float* ws_q = scratch;
  float* ws_k = scratch + static_cast<long>(units) * kD;
  // the maxima are folded in with atomicMax, so the used part must start at zero
  if (cudaMemsetAsync(scratch, 0, 2 * static_cast<size_t>(units) * kD * sizeof(float), s) != cudaSuccess)
    return check_launch("balance_prefill_noalloc memset");
  const long qrows = static_cast<long>(Hq / Hkv) * T;
  int nsplit = (4 * kNumSMs + units - 1) / units;
  nsplit = static_cast<int>(std::min<long>(nsplit, std::max<long>(1, qrows / 64)));
  balance_max_kernel<<<dim3(units, nsplit), kBalThreads, 0, s>>>(
      reinterpret_cast<const uint4*>(q), reinterpret_cast<const uint4*>(k), Hq, Hkv, T, nsplit, ws_q, ws_k);
  if (int e = check_launch("balance_max_kernel (noalloc)")) return e;
  const int n = units * D;
  balance_finalize_kernel<<<(n + 255) / 256, 256, 0, s>>>(ws_q, ws_k, b_out, n);
  return check_launch("balance_finalize_kernel (noalloc)");
}
