// K3 + K4: H2O accumulated-attention importance.
//
// Sources: "No Token Left Behind" reading notes (velog), "Observation 1-4" and
// "Key contributions 1)" (H2O, heavy hitters by accumulated attention); the
// pages name H2O without its formula, so the plain definition is used:
//   prefill  S^h_i = sum_{t >= i} softmax_t(q_t . k / sqrt(D))_i  (causal rows)
//            S_i   = sum over the key head's query heads, h ascending, fp32
//   decode   S_j  += sum_h exp(logit_{h,j} - lse_h) for important-tier slots.
//
// K3 is a dense causal QK^T: two tensor-core passes (tcgen05, fp16 in, fp32 accumulate)
// over 128x128 tiles:
//   pass 1  per (b, h, 128 query rows): online row max/sum -> lse_t (base 2),
//   pass 2  per (b, key head, 128 keys): for every query head of the group and
//           every query tile at or below the diagonal, exp2(s - lse_t) summed
//           over the queries -> S^h_i, then S_i in head order.
// Work is triangular, so CTAs are numbered heaviest first.
#include <algorithm>

#include "common.cuh"
#include "tcgen05.cuh"

namespace mikv {
int validate_cache_public(const mikv_cache* c, const char* who);

namespace {

// log2(e)/sqrt(128): logits in base 2, one rounding shared by both passes
constexpr float kC = 0.12751743082459868f;

// 2^x in one MUFU instruction (ex2.approx.ftz: relative error ~2^-22, exp2(-inf) = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction (exact, like two fmaxf).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ---------------------------------------------------------------------------------
// The two passes on the 5th-generation tensor cores.  128 x 128 tiles, S = A . B^T by
// tcgen05.mma (fp16 in, fp32 accumulate in TMEM), two TMEM accumulators so the next tile's
// MMA runs while the CTA exponentiates the current one.  A ninth warp is the producer: its
// lane 0 streams the operand tiles with TMA (two shared-memory buffers) and issues the
// MMAs; every hand-off is an mbarrier (tile loaded, MMA done, accumulator consumed by all
// 256 consumer threads), so no thread waits at a CTA barrier inside the loop.  Row r of S (TMEM lane r) belongs to
// threads r and r + 128, which take columns 0..63 and 64..127 and keep their own running
// state, combined once at the end.  Per CTA: 3 tiles of 32 KB plus 2 KB of lse rows and
// 256 TMEM columns, so two CTAs share an SM.
constexpr int kTcTile = tc::kTileRows;
constexpr int kTcThreads = 256;                                        // consumers
constexpr int kTcBlock = kTcThreads + 32;                              // + the producer warp
constexpr int kTcHalf = kTcTile / 2;                                    // columns per thread
constexpr int kTcCols = 2 * kTcTile;                                    // two accumulators
constexpr int kTcLseRing = 8;                                           // lse rows in flight
constexpr int kTcSmem = 3 * tc::kTileBytes + kTcLseRing * kTcTile * 4 + 1024;  // + alignment
constexpr uint32_t kTcIdesc = tc::idesc_f16(kTcTile, kTcTile);

// lse rows are padded to whole tiles so one tile's 128 values are one aligned bulk copy.
__host__ __device__ __forceinline__ int lse_stride(int T) { return (T + kTcTile - 1) / kTcTile * kTcTile; }

// Pass 1 on tcgen05: nlse2[b][h][t] = -lse_t in base 2 (row stride lse_stride(T)) for 128
// query rows (negated, so pass 2 forms s * kC - lse_t with one fma).
__global__ void __launch_bounds__(kTcBlock, 2) row_lse_tc_kernel(const __grid_constant__ CUtensorMap tq,
                                                                 const __grid_constant__ CUtensorMap tk,
                                                                 int Hq, int Hkv, int T,
                                                                 float* __restrict__ nlse2) {
  extern __shared__ __align__(128) uint8_t sm[];  // Q tile, 2 K tiles
  __shared__ __align__(8) tc::Bars bar;
  __shared__ uint32_t tslot;
  __shared__ float xm[kTcTile], xl[kTcTile];
  __shared__ int bad;
  const int nblk = (T + kTcTile - 1) / kTcTile;
  const int rb = nblk - 1 - blockIdx.x;  // heaviest (last) row block first
  const int bh = blockIdx.y, b = bh / Hq, h = bh % Hq;
  const int g = h / (Hq / Hkv);
  const int tid = threadIdx.x, warp = tid >> 5, row = tid & 127, half = (tid >> 7) & 1;
  const int qrow0 = bh * T, krow0 = (b * Hkv + g) * T;  // first rows of this head in the maps
  const uint32_t sq = tc::smem_base(sm), sk0 = sq + tc::kTileBytes;
  const int t0 = rb * kTcTile;
  if (tid == 0) bad = 0;
  const uint32_t tbase = tc::cta_setup(bar, &tslot, kTcThreads, kTcCols);
  tc::Waits w;
  float m = -INFINITY, l = 0.f, lc = 0.f;
  const int t = t0 + row;  // a consumer's query row
  if (tid == kTcThreads) {
    // producer: Q once; K tiles through two buffers.  MMA kt as soon as its K tile is in
    // and its accumulator's previous tile was read; K tile kt + 2 once MMA kt is done.
    tc::mbar_expect_tx(smem_u32(&bar.fixed), tc::kTileBytes);
    tc::tma_tile(sq, &tq, qrow0 + t0, smem_u32(&bar.fixed));
    for (int j = 0; j < 2 && j <= rb; ++j) {
      tc::mbar_expect_tx(smem_u32(&bar.load[j]), tc::kTileBytes);
      tc::tma_tile(sk0 + j * tc::kTileBytes, &tk, krow0 + j * kTcTile, smem_u32(&bar.load[j]));
    }
    w(smem_u32(&bar.fixed), 0);
    for (int kt = 0; kt <= rb; ++kt) {
      const int buf = kt & 1;
      w(smem_u32(&bar.load[buf]), (kt >> 1) & 1);
      if (kt >= 2) w(smem_u32(&bar.freed[buf]), ((kt - 2) >> 1) & 1);
      tc::fence_after_sync();
      if (w.ok) {  // after a give-up nothing more is issued
        tc::mma_tile(tbase + buf * kTcTile, sq, sk0 + buf * tc::kTileBytes, kTcIdesc);
        tc::commit(smem_u32(&bar.mma[buf]));
      }
      if (kt + 2 <= rb) {
        w(smem_u32(&bar.mma[buf]), (kt >> 1) & 1);
        if (w.ok) {
          tc::mbar_expect_tx(smem_u32(&bar.load[buf]), tc::kTileBytes);
          tc::tma_tile(sk0 + buf * tc::kTileBytes, &tk, krow0 + (kt + 2) * kTcTile, smem_u32(&bar.load[buf]));
        }
      }
    }
  } else if (tid < kTcThreads) {
    for (int kt = 0; kt <= rb; ++kt) {
      const int buf = kt & 1;
      w(smem_u32(&bar.mma[buf]), (kt >> 1) & 1);
      tc::fence_after_sync();
      // this thread's 64 raw dot products: row t, keys kt*128 + half*64 ..
      float s[kTcHalf];
      const uint32_t lane_addr =
          tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16) + buf * kTcTile + half * kTcHalf;
      tc::tmem_ld32(lane_addr, *reinterpret_cast<float(*)[32]>(s));
      tc::tmem_ld32(lane_addr + 32, *reinterpret_cast<float(*)[32]>(s + 32));
      tc::fence_before_sync();
      tc::mbar_arrive(smem_u32(&bar.freed[buf]));  // accumulator read: the MMA may reuse it
      const int i0 = kt * kTcTile + half * kTcHalf;
      const int lim = min(t - i0, T - 1 - i0);  // columns 0..lim are causal and in range
      // 8 independent max / sum chains (chain c % 8); masks only on the diagonal or last
      // tile.  Unmasked tiles take three-input max and packed f32x2 fma / add: the same
      // chains, in the same order, in fewer instructions.
      const bool full = lim >= kTcHalf - 1;
      float mx8[8];
      if (full) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float x = max3(s[j], s[8 + j], s[16 + j]);
          x = max3(x, s[24 + j], s[32 + j]);
          x = max3(x, s[40 + j], s[48 + j]);
          mx8[j] = fmaxf(x, s[56 + j]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) mx8[j] = -INFINITY;
#pragma unroll
        for (int c = 0; c < kTcHalf; ++c)
          if (c <= lim) mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
      }
      const float mxr = fmaxf(max3(mx8[0], mx8[1], mx8[2]), max3(max3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
      const float mn = fmaxf(m, mxr * kC);  // kC > 0: the max commutes with the scaling
      if (mn != -INFINITY) {
        float2 sm4[4];  // chains 2j, 2j + 1
#pragma unroll
        for (int j = 0; j < 4; ++j) sm4[j] = make_float2(0.f, 0.f);
        if (full) {
          const float2 k2 = make_float2(kC, kC), nm = make_float2(-mn, -mn);
#pragma unroll
          for (int c = 0; c < kTcHalf; c += 2) {
            const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), k2, nm);
            sm4[(c >> 1) & 3] = __fadd2_rn(sm4[(c >> 1) & 3], make_float2(fast_exp2(x.x), fast_exp2(x.y)));
          }
        } else {
#pragma unroll
          for (int c = 0; c < kTcHalf; ++c)
            if (c <= lim) {
              const float e = fast_exp2(fmaf(s[c], kC, -mn));
              if (c & 1) sm4[(c >> 1) & 3].y += e;
              else sm4[(c >> 1) & 3].x += e;
            }
        }
        const float sum = ((sm4[0].x + sm4[0].y) + (sm4[1].x + sm4[1].y)) + ((sm4[2].x + sm4[2].y) + (sm4[3].x + sm4[3].y));
        const float alpha = fast_exp2(m - mn);
        l = __fmul_rn(l, alpha);
        lc = __fmul_rn(lc, alpha);
        const float y = sum - lc;
        const float tt = l + y;
        lc = (tt - l) - y;
        l = tt;
        m = mn;
      }
    }
    // the two halves of each row: half 1 hands its (m, l) to half 0
    if (half == 1) {
      xm[row] = m;
      xl[row] = l - lc;
    }
  }
  if (!w.ok) {
    atomicExch(&bad, 1);
    tc::report_giveup(tc::kGiveupRowLse);
  }
  tc::cta_teardown(tbase, kTcCols);  // (its barrier also publishes xm / xl / bad)
  if (tid < kTcTile && t < T) {
    const float m1 = xm[row], l1 = xl[row], l0 = l - lc;
    const float M = fmaxf(m, m1);
    const float L = (m == -INFINITY ? 0.f : l0 * fast_exp2(m - M)) + (m1 == -INFINITY ? 0.f : l1 * fast_exp2(m1 - M));
    nlse2[static_cast<long>(bh) * lse_stride(T) + t] = bad ? __int_as_float(0x7fc00000) : -(M + log2f(L));
  }
}

// Pass 2 on tcgen05: S^h_i (and S_i) for 128 keys of one (b, key head).  S^T = K . Q^T per
// query tile: TMEM lane = key, column = query; thread i and i + 128 take the query halves.
__global__ void __launch_bounds__(kTcBlock, 2) col_sum_tc_kernel(const __grid_constant__ CUtensorMap tq,
                                                                 const __grid_constant__ CUtensorMap tk,
                                                                 const float* __restrict__ nlse2, int Hq,
                                                                 int Hkv, int T, float* __restrict__ s_full,
                                                                 float* __restrict__ s_head) {
  extern __shared__ __align__(128) uint8_t sm[];  // K tile, 2 Q tiles, lse ring
  __shared__ __align__(8) tc::Bars bar;
  __shared__ uint32_t tslot;
  __shared__ float xs[kTcTile];
  __shared__ int bad;
  const int nblk = (T + kTcTile - 1) / kTcTile;
  const int ls = lse_stride(T);
  const int kbi = blockIdx.x;  // key block 0 (heaviest) first
  const int unit = blockIdx.y, b = unit / Hkv, g = unit % Hkv;
  const int rep = Hq / Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, row = tid & 127, half = (tid >> 7) & 1;
  const uint32_t sk = tc::smem_base(sm), sq0 = sk + tc::kTileBytes, sl0 = sk + 3 * tc::kTileBytes;
  const float* sl = reinterpret_cast<const float*>(sm + (sl0 - smem_u32(sm)));
  const int i0 = kbi * kTcTile;
  const int per = nblk - kbi;   // query tiles per head
  const int ntile = rep * per;  // tiles of this CTA, head-major
  if (tid == 0) bad = 0;
  const uint32_t tbase = tc::cta_setup(bar, &tslot, kTcThreads, kTcCols);
  tc::Waits w;
  const int i = i0 + row;  // a consumer's key
  float tot = 0.f;
  if (tid == kTcThreads) {
    // producer.  Tile n: head hr = n / per, query tile qt = kbi + n % per; Q into buffer
    // n & 1 and its lse row into ring slot n % kTcLseRing, one transaction on load[n & 1].
    // When tile n + 2 is loaded (after MMA n), every consumer is at tile n - 2 or later, so
    // the slots of tiles n - 2 .. n + 1 may still be read and slot (n + 2) % 8 is not one.
    auto load_q = [&](int n) {
      const int hr = n / per, qt = kbi + n % per;
      const long bh = static_cast<long>(b) * Hq + g * rep + hr;
      const uint32_t mb = smem_u32(&bar.load[n & 1]);
      tc::mbar_expect_tx(mb, tc::kTileBytes + kTcTile * 4);
      tc::tma_tile(sq0 + (n & 1) * tc::kTileBytes, &tq, static_cast<int>(bh * T) + qt * kTcTile, mb);
      tc::bulk_copy(sl0 + (n % kTcLseRing) * kTcTile * 4, nlse2 + bh * ls + qt * kTcTile, kTcTile * 4, mb);
    };
    tc::mbar_expect_tx(smem_u32(&bar.fixed), tc::kTileBytes);
    tc::tma_tile(sk, &tk, unit * T + i0, smem_u32(&bar.fixed));
    load_q(0);
    if (ntile > 1) load_q(1);
    w(smem_u32(&bar.fixed), 0);
    for (int n = 0; n < ntile; ++n) {
      const int buf = n & 1;
      w(smem_u32(&bar.load[buf]), (n >> 1) & 1);
      // accumulator buf is free once every consumer has read tile n - 2 from TMEM
      if (n >= 2) w(smem_u32(&bar.freed[buf]), ((n - 2) >> 1) & 1);
      tc::fence_after_sync();
      if (w.ok) {  // after a give-up nothing more is issued
        tc::mma_tile(tbase + buf * kTcTile, sk, sq0 + buf * tc::kTileBytes, kTcIdesc);
        tc::commit(smem_u32(&bar.mma[buf]));
      }
      if (n + 2 < ntile) {  // Q buffer buf is free once MMA n is done
        w(smem_u32(&bar.mma[buf]), (n >> 1) & 1);
        if (w.ok) load_q(n + 2);
      }
    }
  } else if (tid < kTcThreads) {
    float col = 0.f, colc = 0.f;
    for (int n = 0; n < ntile; ++n) {
      const int buf = n & 1;
      w(smem_u32(&bar.mma[buf]), (n >> 1) & 1);
      tc::fence_after_sync();
      const int qt = kbi + n % per;
      const int cq = qt * kTcTile + half * kTcHalf;  // query of this thread's column 0
      const int c0 = max(i - cq, 0);                  // first causal column (query >= key)
      const int c1 = min(kTcHalf, T - cq);            // columns past T are padding
      const float* lt = sl + (n % kTcLseRing) * kTcTile + half * kTcHalf;  // -lse of the columns
      float2 p4[4];  // independent chains e % 8 = 2j, 2j + 1
#pragma unroll
      for (int j = 0; j < 4; ++j) p4[j] = make_float2(0.f, 0.f);
      const bool full = c0 == 0 && c1 == kTcHalf;
      const uint32_t lane_addr =
          tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16) + buf * kTcTile + half * kTcHalf;
      float s0[32], s1[32];
      tc::tmem_ld32(lane_addr, s0);
      tc::tmem_ld32(lane_addr + 32, s1);
      // accumulator read: the MMA may reuse it.  Its lse slot stays valid: tile n + 2's row
      // (slot (n + 2) % 8) is loaded only after MMA n, and tiles n - 2 .. n + 1 hold the
      // slots that consumers may still be reading.
      tc::fence_before_sync();
      tc::mbar_arrive(smem_u32(&bar.freed[buf]));
      if (full) {  // packed f32x2 fma / add, -lse read four at a time
        const float4* l4 = reinterpret_cast<const float4*>(lt);
        const float2 k2 = make_float2(kC, kC);
#pragma unroll
        for (int e = 0; e < 64; e += 4) {
          const float4 a = l4[e >> 2];
          const float* sv = e < 32 ? s0 + e : s1 + (e - 32);
          const float2 x0 = __ffma2_rn(make_float2(sv[0], sv[1]), k2, make_float2(a.x, a.y));
          const float2 x1 = __ffma2_rn(make_float2(sv[2], sv[3]), k2, make_float2(a.z, a.w));
          p4[(e >> 1) & 3] = __fadd2_rn(p4[(e >> 1) & 3], make_float2(fast_exp2(x0.x), fast_exp2(x0.y)));
          p4[((e >> 1) + 1) & 3] =
              __fadd2_rn(p4[((e >> 1) + 1) & 3], make_float2(fast_exp2(x1.x), fast_exp2(x1.y)));
        }
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (e >= c0 && e < c1) {
            const float x = fast_exp2(fmaf(e < 32 ? s0[e] : s1[e - 32], kC, lt[e]));
            if (e & 1) p4[(e >> 1) & 3].y += x;
            else p4[(e >> 1) & 3].x += x;
          }
      }
      const float part = ((p4[0].x + p4[0].y) + (p4[1].x + p4[1].y)) + ((p4[2].x + p4[2].y) + (p4[3].x + p4[3].y));
      const float y = part - colc;
      const float tt = col + y;
      colc = (tt - col) - y;
      col = tt;
      if (n % per == per - 1) {  // head done: the two query halves of each key, then the group
        if (half == 1) xs[row] = col - colc;
        asm volatile("bar.sync 1, %0;\n" ::"n"(kTcThreads));  // consumers only
        if (half == 0) {
          const int hr = n / per;
          const float sh = (col - colc) + xs[row];
          const long bh = static_cast<long>(b) * Hq + g * rep + hr;
          if (i < T && s_head) s_head[bh * T + i] = sh;
          tot = __fadd_rn(tot, sh);  // group sum in head order
        }
        col = colc = 0.f;
        asm volatile("bar.sync 1, %0;\n" ::"n"(kTcThreads));  // xs may be rewritten
      }
    }
  }
  if (!w.ok) {
    atomicExch(&bad, 1);
    tc::report_giveup(tc::kGiveupColSum);
  }
  tc::cta_teardown(tbase, kTcCols);
  if (tid < kTcTile && i < T) s_full[static_cast<long>(unit) * T + i] = bad ? __int_as_float(0x7fc00000) : tot;
}

// K4: S[b][g][j] += sum_h exp(logit[b][h][j] - lse[b][h]) for j < n_hi.
__global__ void score_decode_kernel(const float* __restrict__ logits, const float* __restrict__ lse,
                                    float* __restrict__ scores, int Hq, int Hkv, int cap, int n) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const int unit = blockIdx.y, b = unit / Hkv, g = unit % Hkv;
  if (j >= n) return;
  const int rep = Hq / Hkv;
  float add = 0.f;
  for (int r = 0; r < rep; ++r) {
    const long bh = static_cast<long>(b) * Hq + g * rep + r;
    add += expf(logits[bh * cap + j] - lse[bh]);
  }
  scores[static_cast<long>(unit) * cap + j] += add;
}

}  // namespace
}  // namespace mikv

namespace mikv {
namespace {
}  // namespace
}  // namespace mikv

using namespace mikv;

extern "C" size_t mikv_score_workspace_bytes(int B, int Hq, int T) {
  if (B < 1 || Hq < 1 || T < 1) return 0;
  return align_up(static_cast<size_t>(B) * Hq * lse_stride(T) * sizeof(float), 256);
}

extern "C" int mikv_score_update(int mode, const uint16_t* q, const uint16_t* k, int T,
                                 const float* hi_logits, const float* lse, mikv_cache* c,
                                 float* scores_full, float* scores_head, void* ws, size_t ws_bytes,
                                 void* stream) {
  clear_error();
  if (!c) return fail(MIKV_EINVAL, "score_update: null cache");
  if (c->D != kD) return fail(MIKV_EUNSUPPORTED, "score_update: D=%d (only %d)", c->D, kD);
  if (c->B < 1 || c->Hkv < 1 || c->Hq < c->Hkv || c->Hq % c->Hkv || c->Hq / c->Hkv > 8)
    return fail(MIKV_ESHAPE, "score_update: bad heads");
  cudaStream_t s = as_stream(stream);
  if (mode == MIKV_PREFILL) {
    if (!q || !k || !scores_full || !ws) return fail(MIKV_EINVAL, "score_update: null pointer");
    if (T < 1) return fail(MIKV_ESHAPE, "score_update: T=%d", T);
    if (static_cast<long>(c->B) * c->Hq * T > (1L << 31) - 1) return fail(MIKV_ESHAPE, "score_update: B*Hq*T too large");
    if (!aligned16(q) || !aligned16(k)) return fail(MIKV_EALIGN, "score_update: q/k alignment");
    const size_t need = mikv_score_workspace_bytes(c->B, c->Hq, T);
    if (ws_bytes < need) return fail(MIKV_ESHAPE, "score_update: workspace %zu < %zu", ws_bytes, need);
    float* nlse2 = static_cast<float*>(ws);
    const int nblk = (T + kTcTile - 1) / kTcTile;
    CUtensorMap tq, tk;
    if (int e = tc::encode_rows(&tq, q, static_cast<long>(c->B) * c->Hq * T, "score_update: q")) return e;
    if (int e = tc::encode_rows(&tk, k, static_cast<long>(c->B) * c->Hkv * T, "score_update: k")) return e;
    if (cudaFuncSetAttribute(row_lse_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem) != cudaSuccess ||
        cudaFuncSetAttribute(col_sum_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem) != cudaSuccess)
      return check_launch("score kernels attribute");
    row_lse_tc_kernel<<<dim3(nblk, c->B * c->Hq), kTcBlock, kTcSmem, s>>>(tq, tk, c->Hq, c->Hkv, T, nlse2);
    if (int e = check_launch("row_lse_tc_kernel")) return e;
    col_sum_tc_kernel<<<dim3(nblk, c->B * c->Hkv), kTcBlock, kTcSmem, s>>>(tq, tk, nlse2, c->Hq, c->Hkv, T,
                                                                             scores_full, scores_head);
    return check_launch("col_sum_tc_kernel");
  }
  if (mode == MIKV_DECODE) {
    if (int e = validate_cache_public(c, "score_update")) return e;
    if (!hi_logits || !lse || !c->scores) return fail(MIKV_EINVAL, "score_update: null pointer");
    if (c->n_hi == 0) return MIKV_OK;
    dim3 grid((c->n_hi + 255) / 256, c->B * c->Hkv);
    score_decode_kernel<<<grid, 256, 0, s>>>(hi_logits, lse, c->scores, c->Hq, c->Hkv, c->cap_hi,
                                             c->n_hi);
    return check_launch("score_decode_kernel");
  }
  return fail(MIKV_EINVAL, "score_update: bad mode %d", mode);
}

namespace mikv {
// This file's wait-status word (see tc::wait_giveups), for mikv_wait_status.
int scores_wait_giveups(unsigned* out, bool clear) { return tc::wait_giveups(out, clear); }
}  // namespace mikv
