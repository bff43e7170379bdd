// K5 + K6: token selection (H2O top-k with a recent window, CriticalKV two-stage
// selection, the per-step demotion victim) and the projected-value L1 norms.
//
// Sources: "No Token Left Behind" reading notes (velog), "Key contributions 1)"
// (H2O decides the important tokens; the rest are kept in low precision);
// paperlayer summary, section 5 (local tokens and heavy hitters); CriticalKV
// summary (gist.science), "Algorithm: perturbation-constrained selection"
// (b' = alpha*b by attention weight, the remaining b'' by A_i * ||V_i W_O||_1)
// and "Theoretical framework" (projected value state V W_O).
//
// Selection is exact integer work on the float bit patterns: one CTA per
// (batch, key head) runs an MSB-first radix select (digits of 12, 10 and 10
// bits) over order-preserving 32-bit keys to find the b-th best value, takes
// every candidate above it and, among candidates equal to it, the lowest
// positions (block-wide prefix count in position order), then writes the kept
// and evicted positions in ascending order with a block scan.  Rows of up to
// 8192 positions take 512 threads, each holding the states of 16 consecutive
// positions as bit masks, so after the first digit (whose bin keeps a few
// percent of a row of logits or scores) only the threads still holding a
// candidate read keys again.  Longer rows take 1024 threads with a flag byte
// per position, the first digit's candidates compacted into a shared-memory
// list when they fit.  The result is unique, so it is bit-exact against any
// correct implementation given the same scores.
//
// K6, N[b][h][i] = || v_i . W_O[h*D:(h+1)*D, :] ||_1, is a dense GEMM
// (L x 128) x (128 x hidden) per query head on the tcgen05 tensor cores (fp16
// operands, fp32 accumulate in tensor memory) whose output is never stored:
// the epilogue sums |.| per row.
#include <algorithm>
#include <cmath>
#include <type_traits>

#include "common.cuh"
#include "tcgen05.cuh"

namespace mikv {
int validate_cache_public(const mikv_cache* c, const char* who);

namespace {

constexpr int kSelThreads = 1024;
constexpr int kMaxSelectL = 131072;

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t b = __float_as_uint(x);
  if ((b & 0x7fffffffu) == 0) b = 0;  // -0 == +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Block-wide exclusive scan of one int per thread; returns the exclusive prefix, sets total.
__device__ int block_exclusive_scan(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = (lane < (blockDim.x >> 5)) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;  // inclusive warp prefix
  }
  __syncthreads();
  const int before = (warp > 0) ? warp_sums[warp - 1] : 0;
  total = warp_sums[(blockDim.x >> 5) - 1];
  __syncthreads();
  return before + x - v;
}

// Order keys of a row, read from global memory (converted on each read) or from a staged
// shared-memory copy.
struct GlobalKeys {
  const float* k;
  __device__ __forceinline__ uint32_t operator()(int i) const { return order_key(k[i]); }
};
struct SharedKeys {
  const uint32_t* k;
  __device__ __forceinline__ uint32_t operator()(int i) const { return k[i]; }
};

// Radix digits of the 32-bit order key, high to low: 12 bits (sign, exponent and three
// mantissa bits, which already splits a row of logits or scores finely), then 10 and 10.
constexpr int kSelBins1 = 4096;
constexpr int kSelBins = 1024;

// The digit d where the count of candidates in bins above d first reaches `remaining`
// (scanning nb - 1 -> 0), into scratch[0], and what is left to take inside bin d, into
// scratch[1]; if every bin together holds fewer than `remaining`, d = 0 with the count above
// it.  Thread t of the NT owns the NB / NT bins from NB - 1 - t * (NB / NT) down.  The caller
// synchronises before reading scratch; scratch[0..1] are written only after every thread has
// passed the barriers of the block scan, so a result read before the next search is safe.
template <int NB, int NT>
__device__ __forceinline__ void digit_search(const unsigned* hist, int remaining, int* scratch) {
  constexpr int per = NB / NT;
  const int top = NB - 1 - static_cast<int>(threadIdx.x) * per;
  int sum = 0;
#pragma unroll
  for (int j = 0; j < per; ++j) sum += static_cast<int>(hist[top - j]);
  int total;
  int above = block_exclusive_scan(sum, scratch + 2, total);
  if (above < remaining && remaining <= above + sum) {
    int d = top;
    for (int j = 0; j < per; ++j) {
      d = top - j;
      const int c = static_cast<int>(hist[d]);
      if (above + c >= remaining) break;
      above += c;
    }
    scratch[0] = d;
    scratch[1] = remaining - above;
  } else if (threadIdx.x == NT - 1 && above + sum < remaining) {
    scratch[0] = 0;
    scratch[1] = remaining - (above + sum - static_cast<int>(hist[0]));
  }
}

// Histogram of the digit (u >> shift) & dmask over the candidates (flag == 0) of the whole row
// whose key u matches `prefix` under `mask`.
template <class Keys>
__device__ __forceinline__ void hist_row(Keys key, int L, const uint8_t* flag, unsigned* hist, int shift,
                                         uint32_t dmask, uint32_t mask, uint32_t prefix) {
  const int tid = threadIdx.x;
  int i0 = 0;
  if constexpr (std::is_same<Keys, SharedKeys>::value) {
    // staged rows: four keys and their four flags per load (the flags start L * 4 bytes
    // after the keys, so both are 16- and 4-byte aligned)
    const uint4* k4 = reinterpret_cast<const uint4*>(key.k);
    const uint32_t* f4 = reinterpret_cast<const uint32_t*>(flag);
    for (int q = tid; q < (L >> 2); q += blockDim.x) {
      const uint32_t fl = f4[q];
      if (fl == 0x01010101u * (fl & 0xffu) && (fl & 0xffu) != 0) continue;  // all four taken
      const uint4 u4 = k4[q];
      const uint32_t uu[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (((fl >> (8 * e)) & 0xffu) == 0 && (uu[e] & mask) == prefix)
          atomicAdd(&hist[(uu[e] >> shift) & dmask], 1u);
    }
    i0 = L & ~3;
  }
  for (int i = i0 + tid; i < L; i += blockDim.x) {
    if (flag[i] != 0) continue;
    const uint32_t u = key(i);
    if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & dmask], 1u);
  }
}

// Mark (flag = 1) the `take` best candidates (flag == 0) by key, ties to lower positions.
// hA holds kSelBins1 counters, hB kSelBins.  After the first digit the candidates left in its
// bin are copied, in position order, to the list ckey / cpos when they fit in `cap` entries,
// and the last two digits and the final marking visit only that list; otherwise they visit
// the whole row.
template <class Keys>
__device__ void topk_mark(Keys key, int L, int take, uint8_t* flag, unsigned* hA, unsigned* hB, int* scratch,
                          uint32_t* ckey, uint16_t* cpos, int cap) {
  if (take <= 0) return;
  const int tid = threadIdx.x;
  for (int i = tid; i < kSelBins1; i += blockDim.x) hA[i] = 0;
  for (int i = tid; i < kSelBins; i += blockDim.x) hB[i] = 0;
  __syncthreads();
  hist_row(key, L, flag, hA, 20, kSelBins1 - 1, 0u, 0u);
  __syncthreads();
  digit_search<kSelBins1, kSelThreads>(hA, take, scratch);
  __syncthreads();
  const uint32_t d1 = static_cast<uint32_t>(scratch[0]);
  uint32_t prefix = d1 << 20, mask = 0xfff00000u;
  int remaining = scratch[1];
  const int n1 = static_cast<int>(hA[d1]);
  __syncthreads();
  for (int i = tid; i < kSelBins; i += blockDim.x) hA[i] = 0;  // the third digit's counters

  if (cap > 0 && n1 <= cap) {
    // candidates above bin d1 are taken now; those in it go to the list, in position order
    // (each thread a contiguous run of at most 64 positions, placed by a block scan)
    const int per = ((L + static_cast<int>(blockDim.x) - 1) / static_cast<int>(blockDim.x) + 3) & ~3;
    const int lo = min(L, tid * per), hi = min(L, lo + per);
    uint64_t cm = 0;
    int cnt = 0;
    auto visit = [&](int i, uint32_t u) {
      const uint32_t t = u >> 20;
      if (t > d1) {
        flag[i] = 1;
      } else if (t == d1) {
        cm |= 1ull << (i - lo);
        ++cnt;
      }
    };
    int i = lo;
    if constexpr (std::is_same<Keys, SharedKeys>::value) {
      for (; i + 4 <= hi; i += 4) {  // lo is a multiple of 4: aligned uint4 keys, uint32 flags
        const uint32_t fl = *reinterpret_cast<const uint32_t*>(flag + i);
        if (fl == 0x01010101u * (fl & 0xffu) && (fl & 0xffu) != 0) continue;
        const uint4 u4 = *reinterpret_cast<const uint4*>(key.k + i);
        const uint32_t uu[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (((fl >> (8 * e)) & 0xffu) == 0) visit(i + e, uu[e]);
      }
    }
    for (; i < hi; ++i)
      if (flag[i] == 0) visit(i, key(i));
    int total;
    int at = block_exclusive_scan(cnt, scratch + 2, total);
    while (cm) {
      const int i = lo + __ffsll(static_cast<long long>(cm)) - 1;
      cm &= cm - 1;
      ckey[at] = key(i);
      cpos[at] = static_cast<uint16_t>(i);
      ++at;
    }
    __syncthreads();
    for (int shift = 10; shift >= 0; shift -= 10) {
      unsigned* h = shift ? hB : hA;
      for (int j = tid; j < n1; j += blockDim.x) {
        const uint32_t u = ckey[j];
        if ((u & mask) == prefix) atomicAdd(&h[(u >> shift) & (kSelBins - 1)], 1u);
      }
      __syncthreads();
      digit_search<kSelBins, kSelThreads>(h, remaining, scratch);
      __syncthreads();
      prefix |= static_cast<uint32_t>(scratch[0]) << shift;
      mask |= static_cast<uint32_t>(kSelBins - 1) << shift;
      remaining = scratch[1];
      __syncthreads();
    }
    // list entries above prefix are taken; `remaining` of those equal to it, first in the list
    const int pc = (n1 + static_cast<int>(blockDim.x) - 1) / static_cast<int>(blockDim.x);
    const int clo = min(n1, tid * pc), chi = min(n1, clo + pc);
    int ties = 0;
    for (int j = clo; j < chi; ++j) ties += ckey[j] == prefix;
    int rank = block_exclusive_scan(ties, scratch + 2, total);
    for (int j = clo; j < chi; ++j) {
      const uint32_t u = ckey[j];
      if (u > prefix) flag[cpos[j]] = 1;
      else if (u == prefix) {
        if (rank < remaining) flag[cpos[j]] = 1;
        ++rank;
      }
    }
    __syncthreads();
    return;
  }

  for (int shift = 10; shift >= 0; shift -= 10) {
    unsigned* h = shift ? hB : hA;
    hist_row(key, L, flag, h, shift, kSelBins - 1, mask, prefix);
    __syncthreads();
    digit_search<kSelBins, kSelThreads>(h, remaining, scratch);
    __syncthreads();
    prefix |= static_cast<uint32_t>(scratch[0]) << shift;
    mask |= static_cast<uint32_t>(kSelBins - 1) << shift;
    remaining = scratch[1];
    __syncthreads();
  }
  // every candidate > prefix is taken; `remaining` of those == prefix, lowest positions first
  const int per = (L + blockDim.x - 1) / blockDim.x;
  const int lo = min(L, tid * per), hi = min(L, lo + per);
  int ties = 0;
  for (int i = lo; i < hi; ++i)
    if (flag[i] == 0 && key(i) == prefix) ++ties;
  int total;
  int rank = block_exclusive_scan(ties, scratch + 2, total);
  for (int i = lo; i < hi; ++i) {
    if (flag[i] != 0) continue;
    const uint32_t u = key(i);
    if (u > prefix) flag[i] = 1;
    else if (u == prefix) {
      if (rank < remaining) flag[i] = 1;
      ++rank;
    }
  }
  __syncthreads();
}

// skey[i] = order_key(row[i]), i < L, by the NT threads of the block: kBatch coalesced loads
// in flight per thread (at fixed offsets from one address) before the stores.
template <int kBatch, int NT>
__device__ __forceinline__ void stage_row(const float* __restrict__ row, int L, uint32_t* skey) {
  for (int base = threadIdx.x; base < L; base += kBatch * NT) {
    const float* r = row + base;
    float v[kBatch];
    if (base + (kBatch - 1) * NT < L) {
#pragma unroll
      for (int j = 0; j < kBatch; ++j) v[j] = __ldg(r + j * NT);
#pragma unroll
      for (int j = 0; j < kBatch; ++j) skey[base + j * NT] = order_key(v[j]);
    } else {
#pragma unroll
      for (int j = 0; j < kBatch; ++j) v[j] = base + j * NT < L ? __ldg(r + j * NT) : 0.f;
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (base + j * NT < L) skey[base + j * NT] = order_key(v[j]);
    }
  }
}

// One CTA per (batch, key head).  flag: 0 evicted, 1 taken by a stage, 2 recent window.
// key1 rows are `stride1` floats apart (L for the score arrays, the slot capacity for logits).
// STAGE: the row's order keys are read once into shared memory (L x 4 bytes before the L
// flag bytes) and every pass of each stage reads them there.  After the flags, from byte
// `list_off`, the candidate list: `cap` keys, then `cap` 16-bit positions.
template <bool STAGE>
__global__ void __launch_bounds__(kSelThreads, 2) select_kernel(
    const float* __restrict__ key1, long stride1, const float* __restrict__ key2, int L, int window,
    int take1, int take2, int n_keep, int32_t* __restrict__ keep_pos, int32_t* __restrict__ evict_pos,
    float* __restrict__ keep_scores, int list_off, int cap) {
  extern __shared__ __align__(16) uint8_t sel_smem[];
  uint32_t* skey = reinterpret_cast<uint32_t*>(sel_smem);
  uint8_t* flag = STAGE ? sel_smem + static_cast<size_t>(L) * 4 : sel_smem;
  uint32_t* ckey = reinterpret_cast<uint32_t*>(sel_smem + list_off);
  uint16_t* cpos = reinterpret_cast<uint16_t*>(ckey + cap);
  __shared__ unsigned hA[kSelBins1], hB[kSelBins];
  __shared__ int scratch[2 + 32];
  const long unit = blockIdx.x;
  const float* k1 = key1 + unit * stride1;
  const int w = min(window, L);
  if (STAGE) {
    stage_row<4, kSelThreads>(k1, L, skey);
  }
  for (int i = threadIdx.x; i < L; i += blockDim.x) flag[i] = (i >= L - w) ? 2 : 0;
  __syncthreads();
  if (STAGE) topk_mark(SharedKeys{skey}, L, take1, flag, hA, hB, scratch, ckey, cpos, cap);
  else topk_mark(GlobalKeys{k1}, L, take1, flag, hA, hB, scratch, ckey, cpos, cap);
  if (key2) {
    if (STAGE) {
      stage_row<4, kSelThreads>(key2 + unit * L, L, skey);
      __syncthreads();
      topk_mark(SharedKeys{skey}, L, take2, flag, hA, hB, scratch, ckey, cpos, cap);
    } else {
      topk_mark(GlobalKeys{key2 + unit * L}, L, take2, flag, hA, hB, scratch, ckey, cpos, cap);
    }
  }
  // compaction in position order
  const int per = (L + blockDim.x - 1) / blockDim.x;
  const int lo = min(L, static_cast<int>(threadIdx.x) * per), hi = min(L, lo + per);
  int kept = 0;
  for (int i = lo; i < hi; ++i) kept += flag[i] != 0;
  int total;
  int kp = block_exclusive_scan(kept, scratch + 2, total);
  int ep = lo - kp;
  int32_t* kout = keep_pos + unit * n_keep;
  int32_t* eout = evict_pos ? evict_pos + unit * (L - n_keep) : nullptr;  // null: not wanted
  float* sout = keep_scores ? keep_scores + unit * n_keep : nullptr;
  for (int i = lo; i < hi; ++i) {
    if (flag[i] != 0) {
      if (kp < n_keep) {
        kout[kp] = i;
        if (sout) sout[kp] = k1[i];
      }
      ++kp;
    } else {
      if (eout && ep < L - n_keep) eout[ep] = i;
      ++ep;
    }
  }
}

// Rows of up to kMaskRow positions: thread t of kMaskThreads owns the kMaskKeys consecutive
// positions from t * kMaskKeys, and keeps their taken / window / candidate states as bit masks
// in registers; the staged keys are read back from shared memory (16 bytes at a time) only by
// the loops that need them, and after the first digit only by the threads that still hold a
// candidate.  With many keys per thread the fixed cost of a row (histogram clears, block scans,
// barriers) is shared by fewer threads.  Same result as select_kernel.
constexpr int kMaskKeys = 16;
constexpr int kMaskRow = 8192;
constexpr int kMaskThreads = kMaskRow / kMaskKeys;
constexpr int kMaskMinBlocks = kMaskThreads >= 1024 ? 2 : 4;

// Bits j < kMaskKeys of the positions p0 + j in [lo, hi).
__device__ __forceinline__ uint32_t span_bits(int p0, int lo, int hi) {
  const int a = max(lo - p0, 0), b = min(hi - p0, kMaskKeys);
  return a < b ? static_cast<uint32_t>(((1ull << b) - 1ull) & ~((1ull << a) - 1ull)) : 0u;
}

__device__ __forceinline__ void clear_hists(unsigned* hA, unsigned* hB) {
  for (int i = threadIdx.x; i < kSelBins1; i += kMaskThreads) hA[i] = 0;
  for (int i = threadIdx.x; i < kSelBins; i += kMaskThreads) hB[i] = 0;
}

// The eight staged keys of positions p .. p + 7, p a multiple of 8 (past L: 0, never a candidate).
__device__ __forceinline__ void keys8(const uint32_t* skey, int L, int p, uint32_t (&u)[8]) {
  if (p + 8 <= L) {
    const uint4 a = *reinterpret_cast<const uint4*>(skey + p);
    const uint4 b = *reinterpret_cast<const uint4*>(skey + p + 4);
    u[0] = a.x; u[1] = a.y; u[2] = a.z; u[3] = a.w;
    u[4] = b.x; u[5] = b.y; u[6] = b.z; u[7] = b.w;
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) u[j] = p + j < L ? skey[p + j] : 0u;
  }
}

// Set in `taken` the bits of the `take` best candidates of the block (bits of `cand`), by key,
// ties to lower positions: digits of 12, 10 and 10 bits; after each digit the candidates in the
// chosen bin stay in `eq`, those above it are taken.  hA and hB are zero on entry (cleared
// before the barrier that ends the row's staging).
__device__ __forceinline__ void mask_mark(const uint32_t* skey, int L, uint32_t cand, int take, uint32_t& taken,
                                          unsigned* hA, unsigned* hB, int* scratch) {
  if (take <= 0) return;
  const int tid = threadIdx.x, p0 = tid * kMaskKeys;
#pragma unroll
  for (int c = 0; c < kMaskKeys / 8; ++c) {
    const uint32_t m = (cand >> (8 * c)) & 0xffu;
    if (!m) continue;
    uint32_t u[8];
    keys8(skey, L, p0 + 8 * c, u);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if ((m >> j) & 1u) atomicAdd(&hA[u[j] >> 20], 1u);
  }
  __syncthreads();
  digit_search<kSelBins1, kMaskThreads>(hA, take, scratch);
  __syncthreads();
  uint32_t d = static_cast<uint32_t>(scratch[0]);
  int remaining = scratch[1];
  // hA is read no more in this digit: clear the part the third digit counts in
  for (int i = tid; i < kSelBins; i += kMaskThreads) hA[i] = 0;
  uint32_t eq = 0;
#pragma unroll
  for (int c = 0; c < kMaskKeys / 8; ++c) {
    const uint32_t m = (cand >> (8 * c)) & 0xffu;
    if (!m) continue;
    uint32_t u[8];
    keys8(skey, L, p0 + 8 * c, u);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t t = u[j] >> 20;
      if ((m >> j) & 1u) {
        if (t > d) taken |= 1u << (8 * c + j);
        else if (t == d) eq |= 1u << (8 * c + j);
      }
    }
  }
  for (int shift = 10; shift >= 0; shift -= 10) {
    unsigned* h = shift ? hB : hA;
#pragma unroll
    for (int c = 0; c < kMaskKeys / 8; ++c) {
      const uint32_t m = (eq >> (8 * c)) & 0xffu;
      if (!m) continue;
      uint32_t u[8];
      keys8(skey, L, p0 + 8 * c, u);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if ((m >> j) & 1u) atomicAdd(&h[(u[j] >> shift) & (kSelBins - 1)], 1u);
    }
    __syncthreads();
    digit_search<kSelBins, kMaskThreads>(h, remaining, scratch);
    __syncthreads();
    d = static_cast<uint32_t>(scratch[0]);
    remaining = scratch[1];
#pragma unroll
    for (int c = 0; c < kMaskKeys / 8; ++c) {
      const uint32_t m = (eq >> (8 * c)) & 0xffu;
      if (!m) continue;
      uint32_t u[8];
      keys8(skey, L, p0 + 8 * c, u);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t t = (u[j] >> shift) & (kSelBins - 1);
        if ((m >> j) & 1u) {
          if (t > d) taken |= 1u << (8 * c + j);
          if (t != d) eq &= ~(1u << (8 * c + j));
        }
      }
    }
  }
  // eq: the candidates equal to the threshold key; the first `remaining` in position order
  int total;
  int rank = block_exclusive_scan(__popc(eq), scratch + 2, total);
  for (uint32_t m = eq; m; m &= m - 1) {
    if (rank < remaining) taken |= m & (0u - m);
    ++rank;
  }
}

__global__ void __launch_bounds__(kMaskThreads, kMaskMinBlocks) select_mask_kernel(
    const float* __restrict__ key1, long stride1, const float* __restrict__ key2, int L, int window,
    int take1, int take2, int n_keep, int32_t* __restrict__ keep_pos, int32_t* __restrict__ evict_pos,
    float* __restrict__ keep_scores) {
  extern __shared__ __align__(16) uint8_t sel_smem[];
  uint32_t* skey = reinterpret_cast<uint32_t*>(sel_smem);  // L keys
  __shared__ unsigned hA[kSelBins1], hB[kSelBins];
  __shared__ int scratch[2 + 32];
  const long unit = blockIdx.x;
  const float* k1 = key1 + unit * stride1;
  const int w = min(window, L);
  const int p0 = threadIdx.x * kMaskKeys;
  uint32_t taken = 0;
  clear_hists(hA, hB);
  stage_row<16, kMaskThreads>(k1, L, skey);
  __syncthreads();
  mask_mark(skey, L, span_bits(p0, 0, L - w), take1, taken, hA, hB, scratch);
  if (key2) {
    __syncthreads();  // every read of the first row's keys and of the histograms is done
    clear_hists(hA, hB);
    stage_row<16, kMaskThreads>(key2 + unit * L, L, skey);
    __syncthreads();
    mask_mark(skey, L, span_bits(p0, 0, L - w) & ~taken, take2, taken, hA, hB, scratch);
  }
  // compaction in position order.  Kept positions alone: each thread stores its own.  With
  // scores or evicted positions: the kept positions, then the evicted, into shared memory (over
  // the keys, read no more), then copied out with coalesced stores.
  const uint32_t valid = span_bits(p0, 0, L);
  const uint32_t kept = taken | span_bits(p0, L - w, L);
  int total;
  int kp = block_exclusive_scan(__popc(kept), scratch + 2, total);
  if (!keep_scores && !evict_pos) {
    int32_t* kout = keep_pos + unit * n_keep;
    for (uint32_t m = kept; m; m &= m - 1, ++kp)
      if (kp < n_keep) kout[kp] = p0 + __ffs(m) - 1;
    return;
  }
  int ep = total + min(p0, L) - kp;
  int32_t* pos = reinterpret_cast<int32_t*>(skey);
  for (uint32_t m = kept; m; m &= m - 1) pos[kp++] = p0 + __ffs(m) - 1;
  for (uint32_t m = valid & ~kept; m; m &= m - 1) pos[ep++] = p0 + __ffs(m) - 1;
  __syncthreads();
  const int nk = min(n_keep, total);
  int32_t* kout = keep_pos + unit * n_keep;
  for (int j = threadIdx.x; j < nk; j += kMaskThreads) kout[j] = pos[j];
  if (keep_scores) {
    float* sout = keep_scores + unit * n_keep;
#pragma unroll 1
    for (int j = threadIdx.x; j < nk; j += kMaskThreads) sout[j] = k1[pos[j]];
  }
  if (evict_pos) {  // null: not wanted
    const int ne = min(L - n_keep, L - total);
    int32_t* eout = evict_pos + unit * (L - n_keep);
    for (int j = threadIdx.x; j < ne; j += kMaskThreads) eout[j] = pos[total + j];
  }
}

// Rows of up to kSelStageMax / 5 keys are staged in shared memory (4 bytes of key and one of
// flag per position); longer rows are read from global memory in every pass.  The candidate
// list takes up to L / 8 entries of 6 bytes in what is left (none beyond 65536 positions).
constexpr int kSelStageMax = 200 * 1024;
int launch_select(int units, const float* key1, long stride1, const float* key2, int L, int window, int take1,
                  int take2, int n_keep, int32_t* keep_pos, int32_t* evict_pos, float* keep_scores,
                  cudaStream_t s) {
  if (L <= kMaskRow) {
    const int smem = (L * 4 + 15) & ~15;
    if (cudaFuncSetAttribute(select_mask_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return check_launch("select_mask_kernel attribute");
    select_mask_kernel<<<units, kMaskThreads, smem, s>>>(key1, stride1, key2, L, window, take1, take2, n_keep,
                                                         keep_pos, evict_pos, keep_scores);
    return check_launch("select_mask_kernel");
  }
  const bool stage = static_cast<long>(L) * 5 <= kSelStageMax;
  const int list_off = ((stage ? L * 5 : L) + 15) & ~15;
  const int cap = L <= 65536 ? std::max(0, std::min(L / 8 + 32, (kSelStageMax - list_off) / 6)) : 0;
  const int smem = list_off + cap * 6;
  auto kern = stage ? select_kernel<true> : select_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return check_launch("select_kernel attribute");
  kern<<<units, kSelThreads, smem, s>>>(key1, stride1, key2, L, window, take1, take2, n_keep, keep_pos,
                                               evict_pos, keep_scores, list_off, cap);
  return check_launch("select_kernel");
}

// Demotion victim: among slots j < n_hi with pos < L - window, the minimum of
// (score ascending, position descending).  One CTA per (batch, key head).
__global__ void __launch_bounds__(256) demote_select_kernel(const float* __restrict__ scores,
                                                            const int32_t* __restrict__ pos,
                                                            int cap, int n_hi, int limit,
                                                            int32_t* __restrict__ victim) {
  __shared__ float ss[256];
  __shared__ int sp[256], sj[256];
  const long unit = blockIdx.x;
  float bs = INFINITY;
  int bp = -1, bj = -1;
  for (int j = threadIdx.x; j < n_hi; j += blockDim.x) {
    const int p = pos[unit * cap + j];
    if (p >= limit) continue;
    const float s = scores[unit * cap + j];
    if (bj < 0 || s < bs || (s == bs && p > bp)) {
      bs = s;
      bp = p;
      bj = j;
    }
  }
  ss[threadIdx.x] = bs;
  sp[threadIdx.x] = bp;
  sj[threadIdx.x] = bj;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (threadIdx.x < o) {
      const int t = threadIdx.x + o;
      const bool better = sj[t] >= 0 &&
                          (sj[threadIdx.x] < 0 || ss[t] < ss[threadIdx.x] ||
                           (ss[t] == ss[threadIdx.x] && sp[t] > sp[threadIdx.x]));
      if (better) {
        ss[threadIdx.x] = ss[t];
        sp[threadIdx.x] = sp[t];
        sj[threadIdx.x] = sj[t];
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) victim[unit] = sj[0];
}

// C[b][g][i] = sum_{h in group, ascending} fl(S^h_i * N_{h,i}), fp32 without fusion.
__global__ void ckey_kernel(const float* __restrict__ s_head, const float* __restrict__ n,
                            int Hq, int Hkv, int L, float* __restrict__ ckey) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int unit = blockIdx.y, b = unit / Hkv, g = unit % Hkv;
  if (i >= L) return;
  const int rep = Hq / Hkv;
  float c = 0.f;
  for (int r = 0; r < rep; ++r) {
    const long row = (static_cast<long>(b) * Hq + g * rep + r) * L + i;
    c = __fadd_rn(c, __fmul_rn(s_head[row], n[row]));
  }
  ckey[static_cast<long>(unit) * L + i] = c;
}

// ---------------------------------------------------------------------------------
// K6: projected-value L1 norms on the 5th-generation tensor cores.
// N[b][h][i] = sum_col | v_i^g . W_O[hD:(h+1)D, col] |.  W_O [Hq*D][hidden] is first
// transposed into the workspace, so both operands are K-major (channels contiguous): per CTA
// the V tile of 128 tokens of one (b, key head) stays resident; for each query head of the
// group the 128-column blocks of W_O^T stream through TMA into two buffers, C = V . W^T
// (128 x 128, fp32 in TMEM) by tcgen05.mma, and the consumers (two threads per token, 64
// columns each) add |C|.  The same producer / consumer pipeline as the prefill scores.
constexpr int kVwoThreads = 256;                        // consumers
constexpr int kVwoBlock = kVwoThreads + 64;             // + the copy and MMA warps
constexpr int kVwoCopyThread = kVwoThreads, kVwoMmaThread = kVwoThreads + 32;
constexpr int kVwoN = tc::kTileRows;                    // hidden columns per tile
constexpr int kVwoCols = 2 * kVwoN;                     // two TMEM accumulators
constexpr int kVwoSmem = 3 * tc::kTileBytes + 1024;
constexpr uint32_t kVwoIdesc = tc::idesc_f16(tc::kTileRows, kVwoN);

// W^T[c][r] = W[r][c] for a [rows][cols] fp16 matrix, 32 x 32 tiles through shared memory.
__global__ void __launch_bounds__(256) transpose_kernel(const __half* __restrict__ w, int rows, int cols,
                                                        __half* __restrict__ wt) {
  __shared__ __half tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int j = ty; j < 32; j += 8)
    if (r0 + j < rows && c0 + tx < cols) tile[j][tx] = w[static_cast<long>(r0 + j) * cols + c0 + tx];
  __syncthreads();
  for (int j = ty; j < 32; j += 8)
    if (c0 + j < cols && r0 + tx < rows) wt[static_cast<long>(c0 + j) * rows + r0 + tx] = tile[tx][j];
}

__global__ void __launch_bounds__(kVwoBlock, 2) vwo_norm_tc_kernel(const __grid_constant__ CUtensorMap tv,
                                                                   const __grid_constant__ CUtensorMap twt,
                                                                   int Hq, int Hkv, int L, int hidden,
                                                                   float* __restrict__ out) {
  extern __shared__ __align__(128) uint8_t sm[];  // V tile, 2 W tiles
  __shared__ __align__(8) tc::Bars bar;
  __shared__ uint32_t tslot;
  __shared__ float xs[tc::kTileRows];
  __shared__ int bad;
  const int unit = blockIdx.y, b = unit / Hkv, g = unit % Hkv;
  const int rep = Hq / Hkv;
  const int i0 = blockIdx.x * tc::kTileRows;
  const int tid = threadIdx.x, warp = tid >> 5, row = tid & 127, half = (tid >> 7) & 1;
  const uint32_t sv = tc::smem_base(sm), sw0 = sv + tc::kTileBytes;
  const int per = hidden / kVwoN;  // column blocks per head
  const int ntile = rep * per;     // tiles of this CTA, head-major
  if (tid == 0) bad = 0;
  const uint32_t tbase = tc::cta_setup(bar, &tslot, kVwoThreads, kVwoCols);
  tc::Waits w;
  const int i = i0 + row;  // a consumer's token
  if (tid == kVwoCopyThread) {
    // copies.  Tile n: head g*rep + n / per, columns (n % per) * 128 ..: rows of W^T, the
    // head's 128 channels at x = h * 128
    auto load_w = [&](int n) {
      const int h = g * rep + n / per, cb = n % per;
      const uint32_t mb = smem_u32(&bar.load[n & 1]);
      tc::mbar_expect_tx(mb, tc::kTileBytes);
#pragma unroll
      for (int j = 0; j < kD / 64; ++j)
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(sw0 + (n & 1) * tc::kTileBytes + j * tc::kKBlock),
            "l"(&twt), "r"(h * kD + j * 64), "r"(cb * kVwoN), "r"(mb)
            : "memory");
    };
    tc::mbar_expect_tx(smem_u32(&bar.fixed), tc::kTileBytes);
    tc::tma_tile(sv, &tv, unit * L + i0, smem_u32(&bar.fixed));
    load_w(0);
    if (ntile > 1) load_w(1);
    for (int n = 0; n + 2 < ntile; ++n) {  // W buffer n & 1 is free once MMA n is done
      w(smem_u32(&bar.mma[n & 1]), (n >> 1) & 1);
      if (w.ok) load_w(n + 2);  // after a give-up nothing more is issued
    }
  } else if (tid == kVwoMmaThread) {
    // MMAs: tile n as soon as its W tile is in and accumulator n & 1 was read (tile n - 2)
    w(smem_u32(&bar.fixed), 0);
    for (int n = 0; n < ntile; ++n) {
      const int buf = n & 1;
      w(smem_u32(&bar.load[buf]), (n >> 1) & 1);
      if (n >= 2) w(smem_u32(&bar.freed[buf]), ((n - 2) >> 1) & 1);
      tc::fence_after_sync();
      if (w.ok) {
        tc::mma_tile(tbase + buf * kVwoN, sv, sw0 + buf * tc::kTileBytes, kVwoIdesc);
        tc::commit(smem_u32(&bar.mma[buf]));
      }
    }
  } else if (tid < kVwoThreads) {
    float run = 0.f, comp = 0.f;
    for (int n = 0; n < ntile; ++n) {
      const int buf = n & 1;
      w(smem_u32(&bar.mma[buf]), (n >> 1) & 1);
      tc::fence_after_sync();
      float c0[32], c1[32];
      const uint32_t lane_addr =
          tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16) + buf * kVwoN + half * (kVwoN / 2);
      tc::tmem_ld32(lane_addr, c0);
      tc::tmem_ld32(lane_addr + 32, c1);
      tc::fence_before_sync();
      tc::mbar_arrive(smem_u32(&bar.freed[buf]));  // accumulator read
      float p8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 32; ++e) p8[e & 7] += fabsf(c0[e]);
#pragma unroll
      for (int e = 0; e < 32; ++e) p8[e & 7] += fabsf(c1[e]);
      const float part = ((p8[0] + p8[1]) + (p8[2] + p8[3])) + ((p8[4] + p8[5]) + (p8[6] + p8[7]));
      const float y = part - comp;
      const float t = run + y;
      comp = (t - run) - y;
      run = t;
      if (n % per == per - 1) {  // head done: the two column halves of each token
        if (half == 1) xs[row] = run - comp;
        asm volatile("bar.sync 1, %0;\n" ::"n"(kVwoThreads));  // consumers only
        if (half == 0 && i < L) {
          const int h = g * rep + n / per;
          out[(static_cast<long>(b) * Hq + h) * L + i] = (run - comp) + xs[row];
        }
        run = comp = 0.f;
        asm volatile("bar.sync 1, %0;\n" ::"n"(kVwoThreads));  // xs may be rewritten
      }
    }
  }
  if (!w.ok) {
    atomicExch(&bad, 1);
    tc::report_giveup(tc::kGiveupVwo);
  }
  tc::cta_teardown(tbase, kVwoCols);
  if (bad && tid < tc::kTileRows && i < L)  // a wait gave up: mark the unit's rows
    for (int hr = 0; hr < rep; ++hr) out[(static_cast<long>(b) * Hq + g * rep + hr) * L + i] = __int_as_float(0x7fc00000);
}

// ---------------------------------------------------------------------------------
// Post-attention top-k over the full cache (MiKV reading notes, "1-4) Quantitative
// analysis": the oracle-eviction simulation computes the attention map over the full cache
// first and applies top-k sparsity after it, an upper-bound proxy).  Reading: per query head
// the k = max(1, floor(p * L / 100)) largest logits (ties to the lower slot) are kept and the
// output is attention over them alone, the softmax renormalised over the kept set.
// topk_attend_kernel: one CTA per (batch, query head): the max of the kept logits, then the
// kept tokens in chunks (weights exp(l - m) and slot indices in shared memory).  Sixteen
// threads share a V row, eight channels (16 bytes) each, so the CTA's 512 threads take 32 rows
// at a time, rows j = slot (mod 32), several 16-byte loads in flight per thread; the 32 slots'
// sums are then added in slot order.
constexpr int kTkChunk = 1024;
constexpr int kTkThreads = 512;
constexpr int kTkRowThreads = kD / 8;                      // threads per V row
constexpr int kTkSlots = kTkThreads / kTkRowThreads;       // rows taken at a time

__global__ void __launch_bounds__(kTkThreads) topk_attend_kernel(const float* __restrict__ logits, int cap,
                                                                const int32_t* __restrict__ keep, int k,
                                                                const __half* __restrict__ v, int Hq, int Hkv,
                                                                float* __restrict__ out, float* __restrict__ lse) {
  __shared__ float w[kTkChunk];
  __shared__ int idx[kTkChunk];
  __shared__ float red[kTkThreads / 32];
  __shared__ float part[kTkSlots][kD];
  const int bh = blockIdx.x, b = bh / Hq, h = bh % Hq, g = h / (Hq / Hkv);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = tid / kTkRowThreads, c8 = (tid % kTkRowThreads) * 8;
  const float* lg = logits + static_cast<long>(bh) * cap;
  const int32_t* kp = keep + static_cast<long>(bh) * k;
  const __half* vb = v + static_cast<long>(b * Hkv + g) * cap * kD + c8;
  float m = -INFINITY;
  for (int j = tid; j < k; j += kTkThreads) m = fmaxf(m, lg[kp[j]]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int i = 1; i < kTkThreads / 32; ++i) m = fmaxf(m, red[i]);
  __syncthreads();
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float tsum = 0.f;
  for (int c0 = 0; c0 < k; c0 += kTkChunk) {
    const int n = min(kTkChunk, k - c0);
    for (int j = tid; j < n; j += kTkThreads) {
      const int i = kp[c0 + j];
      const float e = expf(lg[i] - m);
      w[j] = e;
      idx[j] = i;
      tsum += e;
    }
    __syncthreads();
#pragma unroll 4
    for (int j = slot; j < n; j += kTkSlots) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(vb + static_cast<long>(idx[j]) * kD));
      const float wj = w[j];
      const __half2* hv = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __half22float2(hv[q]);
        acc[2 * q] = fmaf(wj, f.x, acc[2 * q]);
        acc[2 * q + 1] = fmaf(wj, f.y, acc[2 * q + 1]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) tsum += __shfl_xor_sync(0xffffffffu, tsum, off);
  if (lane == 0) red[warp] = tsum;
#pragma unroll
  for (int q = 0; q < 8; ++q) part[slot][c8 + q] = acc[q];
  __syncthreads();
  if (tid < kD) {
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < kTkThreads / 32; ++i) tot += red[i];
    float o = 0.f;
    for (int r = 0; r < kTkSlots; ++r) o += part[r][tid];
    out[static_cast<long>(bh) * kD + tid] = o / tot;
    if (tid == 0 && lse) lse[bh] = m + logf(tot);
  }
}

int topk_count(int L, int budget_pct) { return std::max(1, static_cast<int>(static_cast<long>(budget_pct) * L / 100)); }

struct TopkWs {
  size_t dec, out, lse, logits, keep, total;
};
TopkWs topk_ws_layout(const mikv_cache* c, int k) {
  const size_t bh = static_cast<size_t>(c->B) * c->Hq;
  TopkWs t;
  t.dec = 0;
  t.out = align_up(mikv_decode_workspace_bytes(c), 256);
  t.lse = t.out + align_up(bh * kD * sizeof(float), 256);
  t.logits = t.lse + align_up(bh * sizeof(float), 256);
  t.keep = t.logits + align_up(bh * c->cap_hi * sizeof(float), 256);
  t.total = t.keep + align_up(bh * k * sizeof(int32_t), 256);
  return t;
}

}  // namespace
}  // namespace mikv

using namespace mikv;

static int n_keep_of(int L, int pct, int window) {
  const long p = static_cast<long>(pct) * L / 100;
  return static_cast<int>(std::min<long>(L, std::max<long>(window, p)));
}

extern "C" size_t mikv_select_workspace_bytes(int policy, int B, int Hkv, int Hq, int L, int hidden) {
  if (policy != MIKV_CRITICALKV || B < 1 || Hkv < 1 || L < 1) return 0;
  // the stage-2 keys, then the transpose of W_O (when hidden > 0)
  return align_up(static_cast<size_t>(B) * Hkv * L * sizeof(float), 256) +
         align_up(static_cast<size_t>(std::max(hidden, 0)) * std::max(Hq, 0) * kD * 2, 256);
}

extern "C" int mikv_select(int policy, const mikv_cache* c, int L, int budget_pct, int window,
                           float alpha, const float* scores, const float* scores_head,
                           const uint16_t* v, const uint16_t* w_o, int hidden, float* vwo_norm,
                           int32_t* keep_pos, int32_t* evict_pos, float* keep_scores, void* ws,
                           size_t ws_bytes, void* stream) {
  clear_error();
  if (!c) return fail(MIKV_EINVAL, "select: null cache");
  if (c->B < 1 || c->Hkv < 1 || c->Hq < c->Hkv || c->Hq % c->Hkv || c->Hq / c->Hkv > 8)
    return fail(MIKV_ESHAPE, "select: bad heads");
  if (L < 1 || window < 0) return fail(MIKV_ESHAPE, "select: L=%d window=%d", L, window);
  cudaStream_t s = as_stream(stream);
  const int units = c->B * c->Hkv;
  if (policy == MIKV_DEMOTE) {
    if (int e = validate_cache_public(c, "select(DEMOTE)")) return e;
    if (!evict_pos || !c->scores || !c->pos_hi) return fail(MIKV_EINVAL, "select(DEMOTE): null pointer");
    if (c->n_hi <= window)
      return fail(MIKV_ESHAPE, "select(DEMOTE): n_hi=%d must exceed window=%d", c->n_hi, window);
    demote_select_kernel<<<units, 256, 0, s>>>(c->scores, c->pos_hi, c->cap_hi, c->n_hi,
                                               L - window, evict_pos);
    return check_launch("demote_select_kernel");
  }
  if (policy != MIKV_H2O && policy != MIKV_CRITICALKV) return fail(MIKV_EINVAL, "select: policy %d", policy);
  if (budget_pct < 0 || budget_pct > 100) return fail(MIKV_ESHAPE, "select: budget_pct=%d", budget_pct);
  if (L > kMaxSelectL) return fail(MIKV_ESHAPE, "select: L=%d above %d", L, kMaxSelectL);
  const int n_keep = n_keep_of(L, budget_pct, window);
  if (!scores || (!keep_pos && n_keep > 0) || (!evict_pos && L - n_keep > 0))
    return fail(MIKV_EINVAL, "select: null pointer");
  const int w = std::min(window, L);
  const int bud = n_keep - w;
  int take1 = bud, take2 = 0;
  const float* key2 = nullptr;
  if (policy == MIKV_CRITICALKV) {
    if (!(alpha >= 0.f && alpha <= 1.f)) return fail(MIKV_EINVAL, "select: alpha=%g", alpha);
    if (!scores_head || !vwo_norm || !ws) return fail(MIKV_EINVAL, "select(CRITICALKV): null pointer");
    const size_t need = mikv_select_workspace_bytes(policy, c->B, c->Hkv, c->Hq, L, hidden);
    if (ws_bytes < need) return fail(MIKV_ESHAPE, "select: workspace %zu < %zu", ws_bytes, need);
    if (!aligned16(ws)) return fail(MIKV_EALIGN, "select: workspace alignment");
    take1 = static_cast<int>(std::floor(static_cast<double>(alpha) * bud));
    take2 = bud - take1;
    if (w_o) {
      if (!v) return fail(MIKV_EINVAL, "select(CRITICALKV): null v");
      if (c->D != kD) return fail(MIKV_EUNSUPPORTED, "select: D=%d", c->D);
      if (hidden < kVwoN || hidden % kVwoN) return fail(MIKV_ESHAPE, "select: hidden=%d (multiple of %d)", hidden, kVwoN);
      if (static_cast<long>(c->B) * c->Hkv * L > (1L << 31) - 1) return fail(MIKV_ESHAPE, "select: B*Hkv*L too large");
      if (!aligned16(v) || !aligned16(w_o)) return fail(MIKV_EALIGN, "select: v/w_o alignment");
      // W_O^T into the workspace after the stage-2 keys
      __half* wt = reinterpret_cast<__half*>(static_cast<char*>(ws) +
                                             align_up(static_cast<size_t>(c->B) * c->Hkv * L * sizeof(float), 256));
      const int wrows = c->Hq * kD;
      transpose_kernel<<<dim3((hidden + 31) / 32, (wrows + 31) / 32), 256, 0, s>>>(
          reinterpret_cast<const __half*>(w_o), wrows, hidden, wt);
      if (int e = check_launch("transpose_kernel")) return e;
      CUtensorMap tv, twt;
      if (int e = tc::encode_rows(&tv, v, static_cast<long>(c->B) * c->Hkv * L, "select: v")) return e;
      if (int e = tc::encode_rows(&twt, wt, hidden, "select: w_o^T", wrows)) return e;
      if (cudaFuncSetAttribute(vwo_norm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kVwoSmem) != cudaSuccess)
        return check_launch("vwo_norm_tc_kernel attribute");
      vwo_norm_tc_kernel<<<dim3((L + tc::kTileRows - 1) / tc::kTileRows, units), kVwoBlock, kVwoSmem, s>>>(
          tv, twt, c->Hq, c->Hkv, L, hidden, vwo_norm);
      if (int e = check_launch("vwo_norm_tc_kernel")) return e;
    }
    float* ckey = static_cast<float*>(ws);
    ckey_kernel<<<dim3((L + 255) / 256, units), 256, 0, s>>>(scores_head, vwo_norm, c->Hq, c->Hkv, L, ckey);
    if (int e = check_launch("ckey_kernel")) return e;
    key2 = ckey;
  }
  return launch_select(units, scores, L, key2, L, window, take1, take2, n_keep, keep_pos, evict_pos,
                       keep_scores, s);
}

extern "C" size_t mikv_topk_attention_workspace_bytes(const mikv_cache* c, int budget_pct) {
  if (!c || c->n_hi < 1 || c->B < 1 || c->Hq < 1 || budget_pct < 0 || budget_pct > 100) return 0;
  return topk_ws_layout(c, topk_count(c->n_hi, budget_pct)).total;
}

extern "C" int mikv_topk_attention(const uint16_t* q, const mikv_cache* c, int budget_pct, float* out, float* lse,
                                   int32_t* keep_idx, void* ws, size_t ws_bytes, void* stream) {
  clear_error();
  if (!c) return fail(MIKV_EINVAL, "topk_attention: null cache");
  if (!q || !out || !ws) return fail(MIKV_EINVAL, "topk_attention: null pointer");
  if (c->hi_bits != 16 || c->n_lo != 0)
    return fail(MIKV_EUNSUPPORTED, "topk_attention: needs the full FP16 cache (hi_bits=%d, n_lo=%d)", c->hi_bits, c->n_lo);
  if (budget_pct < 0 || budget_pct > 100) return fail(MIKV_ESHAPE, "topk_attention: budget_pct=%d", budget_pct);
  const int L = c->n_hi;
  if (L < 1 || L > kMaxSelectL) return fail(MIKV_ESHAPE, "topk_attention: n_hi=%d (1..%d)", L, kMaxSelectL);
  if (c->B < 1 || c->Hkv < 1 || c->Hq < c->Hkv || c->Hq % c->Hkv) return fail(MIKV_ESHAPE, "topk_attention: bad heads");
  const int k = topk_count(L, budget_pct);
  const TopkWs t = topk_ws_layout(c, k);
  if (ws_bytes < t.total) return fail(MIKV_ESHAPE, "topk_attention: workspace %zu < %zu", ws_bytes, t.total);
  char* w = static_cast<char*>(ws);
  float* full_out = reinterpret_cast<float*>(w + t.out);
  float* full_lse = reinterpret_cast<float*>(w + t.lse);
  float* logits = reinterpret_cast<float*>(w + t.logits);
  int32_t* keep = keep_idx ? keep_idx : reinterpret_cast<int32_t*>(w + t.keep);
  // 1. the full attention map: every logit of the cache (and the full-cache output)
  if (int e = mikv_decode_attention(q, c, full_out, full_lse, logits, w + t.dec, t.out, stream)) return e;
  cudaStream_t s = as_stream(stream);
  const int units = c->B * c->Hq;
  // 2. per query head, the k largest logits (ties to the lower slot), slots ascending
  if (int e = launch_select(units, logits, c->cap_hi, nullptr, L, 0, k, 0, k, keep, nullptr, nullptr, s)) return e;
  // 3. attention over the kept tokens alone
  topk_attend_kernel<<<units, kTkThreads, 0, s>>>(logits, c->cap_hi, keep, k, reinterpret_cast<const __half*>(c->v_hi),
                                          c->Hq, c->Hkv, out, lse);
  return check_launch("topk_attend_kernel");
}

namespace mikv {
// This file's wait-status word (see tc::wait_giveups), for mikv_wait_status.
int select_wait_giveups(unsigned* out, bool clear) { return tc::wait_giveups(out, clear); }
}  // namespace mikv
