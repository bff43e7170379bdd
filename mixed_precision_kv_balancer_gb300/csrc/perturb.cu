// K9: the step after attention -- the output projection y = o . W_O and the per-head output
// perturbation of CriticalKV.
//
// Sources: CriticalKV summary (gist.science, arXiv 2502.03805), "Theoretical framework":
// replacing the full cache by a subset perturbs the attention output, L = ||o - o^||_1, and
// the bound on it runs through the value states projected by the output projection W_O;
// "Experimental results": the perturbation is reported per attention head.  Reading: head h
// reaches the hidden state through rows h*D .. h*D + D - 1 of W_O [Hq*D][hidden], so
//   y[b]      = sum_h o[b][h] . W_O^(h)                     (hidden values)
//   L[b][h]   = || (o[b][h] - o^[b][h]) . W_O^(h) ||_1       (sum over hidden)
// and without W_O, L[b][h] = || o[b][h] - o^[b][h] ||_1 over D.
//
// Layout: the projection comes as nn.Linear stores it, w_o_t = W_O^T [hidden][Hq*D], which is
// already K-major (channels contiguous) for the tensor core.  A prep kernel writes, per head
// and block of 32 batch rows, one 128-row fp16 operand tile: rows 0..63 hold o, rows 64..127
// hold d = o - o^, each row scaled by a power of two (max magnitude in [2^13, 2^14)) and
// written as two fp16 rows (hi = fp16(x), lo = fp16(x - hi): ~22 bits, so the products stay
// near fp32 accuracy for differences of any size).  The main kernel (one CTA per 64 hidden columns
// and batch block) streams, head by head, that tile and the head's 64 x 128 block of W_O^T
// through a four-stage TMA ring (48 KB a stage: three stages in flight hide the L2 / DRAM
// latency), multiplies them with tcgen05.mma (M 128, N 64, K 128, fp32
// in TMEM), and the consumers add hi + lo, accumulate y over the heads in registers and sum
// |z| of the d rows per head.  A last kernel adds the per-head partial sums in a fixed order.
#include <algorithm>

#include "common.cuh"
#include "tcgen05.cuh"

namespace mikv {
namespace {

constexpr int kPtRows = tc::kTileRows;           // operand rows per batch block
constexpr int kPtBatch = 32;                     // batch rows per block (hi, lo) x (o, d)
constexpr int kPtN = 64;                         // hidden columns per CTA
constexpr int kPtThreads = 256;                  // consumers
constexpr int kPtBlock = kPtThreads + 32;        // + the producer warp
constexpr int kPtABytes = kPtRows * kD * 2;      // 32 KB
constexpr int kPtWBytes = kPtN * kD * 2;         // 16 KB
constexpr int kPtStage = kPtABytes + kPtWBytes;  // 48 KB
constexpr int kPtRing = 4;                       // stages in flight
constexpr int kPtAcc = 4;                        // 64-column TMEM accumulators
constexpr int kPtSmem = kPtRing * kPtStage + 1024;  // + the row scales of the block (Hq * 64 floats)
constexpr int kPtMaxHq = 128;
using PtRing = tc::Ring<kPtRing, kPtAcc>;
constexpr uint32_t kPtIdesc = tc::idesc_f16(kPtRows, kPtN);

__host__ __device__ constexpr int pt_blocks(int B) { return (B + kPtBatch - 1) / kPtBatch; }

// One warp per (head h, batch row b < 32 * nbb): the four operand rows of (b, h) in the tile
// of (h, b / 32): r = (b % 32) * 2 + {0: hi, 1: lo} for o, the same + 64 for d = o - o_hat.
// Each row (b, h, o | d) is first scaled by a power of two that brings its largest magnitude
// into [2^13, 2^14), exactly, so that neither part falls into fp16's subnormal range;
// invs[(h * 32 * nbb + b) * 2 + {0: o, 1: d}] receives the inverse.  Rows b >= B are zero.
__global__ void perturb_prep_kernel(const float* __restrict__ o, const float* __restrict__ o_hat, int B, int Hq,
                                    __half* __restrict__ a, float* __restrict__ invs) {
  const int nbb = pt_blocks(B), Bp = nbb * kPtBatch;
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (w >= Hq * Bp) return;
  const int h = w / Bp, b = w % Bp, bb = b / kPtBatch;
  float xo[4] = {0.f, 0.f, 0.f, 0.f}, xd[4] = {0.f, 0.f, 0.f, 0.f};  // channels 4 * lane ..
  if (b < B) {
    const long src = (static_cast<long>(b) * Hq + h) * kD + 4 * lane;
    const float4 v = *reinterpret_cast<const float4*>(o + src);
    xo[0] = v.x, xo[1] = v.y, xo[2] = v.z, xo[3] = v.w;
    if (o_hat) {
      const float4 u = *reinterpret_cast<const float4*>(o_hat + src);
      xd[0] = v.x - u.x, xd[1] = v.y - u.y, xd[2] = v.z - u.z, xd[3] = v.w - u.w;
    }
  }
  float mo = fmaxf(fmaxf(fabsf(xo[0]), fabsf(xo[1])), fmaxf(fabsf(xo[2]), fabsf(xo[3])));
  float md = fmaxf(fmaxf(fabsf(xd[0]), fabsf(xd[1])), fmaxf(fabsf(xd[2]), fabsf(xd[3])));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    mo = fmaxf(mo, __shfl_xor_sync(0xffffffffu, mo, off));
    md = fmaxf(md, __shfl_xor_sync(0xffffffffu, md, off));
  }
  auto scale_exp = [](float m) {  // e with m * 2^e in [2^13, 2^14); 0 for m == 0
    if (!(m > 0.f)) return 0;
    int E;
    frexpf(m, &E);  // m = f * 2^E, f in [0.5, 1)
    return min(max(14 - E, -100), 100);
  };
  const int eo = scale_exp(mo), ed = scale_exp(md);
  __half* tile = a + static_cast<long>(h * nbb + bb) * kPtRows * kD;
  const int r0 = (b % kPtBatch) * 2;
#pragma unroll
  for (int part = 0; part < 2; ++part) {
    const float* x = part ? xd : xo;
    const int e = part ? ed : eo;
    float hi[4], lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float xs = ldexpf(x[j], e);  // exact
      hi[j] = __half2float(__float2half_rn(xs));
      lo[j] = xs - hi[j];
    }
    __half2* rh = reinterpret_cast<__half2*>(tile + (part * 64 + r0) * kD + 4 * lane);
    __half2* rl = reinterpret_cast<__half2*>(tile + (part * 64 + r0 + 1) * kD + 4 * lane);
    rh[0] = __floats2half2_rn(hi[0], hi[1]);
    rh[1] = __floats2half2_rn(hi[2], hi[3]);
    rl[0] = __floats2half2_rn(lo[0], lo[1]);
    rl[1] = __floats2half2_rn(lo[2], lo[3]);
  }
  if (lane == 0) {
    invs[(static_cast<long>(h) * Bp + b) * 2] = ldexpf(1.f, -eo);
    invs[(static_cast<long>(h) * Bp + b) * 2 + 1] = ldexpf(1.f, -ed);
  }
}

// D (TMEM, 128 x 64) = A (128 x kD, 32 KB tile) . W^T (64 x kD, 16 KB tile): 8 K steps; the
// W tile's k-blocks are 8 KB apart.
__device__ __forceinline__ void mma_a_w(uint32_t tmem_d, uint32_t sa, uint32_t sw) {
#pragma unroll
  for (int ks = 0; ks < kD / 16; ++ks) {
    const uint32_t a_off = (ks >> 2) * tc::kKBlock + (ks & 3) * 32;
    const uint32_t w_off = (ks >> 2) * (kPtN * 128) + (ks & 3) * 32;
    tc::mma_f16(tmem_d, tc::smem_desc(sa + a_off), tc::smem_desc(sw + w_off), kPtIdesc, ks > 0);
  }
}

__global__ void __launch_bounds__(kPtBlock, 1) perturb_tc_kernel(const __grid_constant__ CUtensorMap ta,
                                                                 const __grid_constant__ CUtensorMap tw, int B,
                                                                 int Hq, int hidden,
                                                                 const float* __restrict__ invs,
                                                                 float* __restrict__ y, float* __restrict__ part) {
  extern __shared__ __align__(128) uint8_t sm[];  // kPtRing stages of (A tile, W tile), row scales
  __shared__ __align__(8) PtRing ring;
  __shared__ uint32_t tslot;
  __shared__ int bad;
  const int cb = blockIdx.x, bb = blockIdx.y, nbb = gridDim.y, Bp = nbb * kPtBatch;
  const int ncb = hidden / kPtN;
  const int tid = threadIdx.x, warp = tid >> 5, row = tid & 127, half = (tid >> 7) & 1;
  const int b = bb * kPtBatch + ((row & 63) >> 1);
  const bool drow = row >= 64, hirow = (row & 1) == 0;
  const uint32_t s0 = tc::smem_base(sm);
  // inverse row scales of this batch block for every head, [h][64] (read each step)
  float* sinv = reinterpret_cast<float*>(sm + (s0 - smem_u32(sm)) + kPtRing * kPtStage);
  for (int j = tid; j < Hq * 2 * kPtBatch; j += kPtBlock)
    sinv[j] = invs[(static_cast<long>(j / (2 * kPtBatch)) * Bp + bb * kPtBatch) * 2 + j % (2 * kPtBatch)];
  if (tid == 0) bad = 0;
  const uint32_t tbase = tc::ring_setup(ring, &tslot, kPtThreads, kPtAcc * kPtN);  // (its barrier publishes sinv)
  bool ok = true;
  if (tid == kPtThreads) {
    // producer.  Step s takes head h = (s + cb) % Hq: the operand tile of (h, bb) and the
    // 64 x 128 block of W^T at rows cb*64, channels h*128; nothing is resident.  The head
    // order is rotated per column block so that the CTAs running at one time read different
    // operand tiles (all reading the same tile at once concentrates them on a few L2 slices).
    tc::mbar_arrive(smem_u32(&ring.fixed));
    ok = tc::ring_produce(
        ring, Hq,
        [&](int s, int st, uint32_t mb) {
          const int h = (s + cb) % Hq;
          const uint32_t sa = s0 + st * kPtStage;
          tc::mbar_expect_tx(mb, kPtStage);
          tc::tma_tile(sa, &ta, (h * nbb + bb) * kPtRows, mb);
#pragma unroll
          for (int j = 0; j < kD / 64; ++j)
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(sa + kPtABytes + j * (kPtN * 128)),
                "l"(&tw), "r"(h * kD + j * 64), "r"(cb * kPtN), "r"(mb)
                : "memory");
        },
        [&](int, int st, int acc) {
          const uint32_t sa = s0 + st * kPtStage;
          mma_a_w(tbase + acc * kPtN, sa, sa + kPtABytes);
        });
  } else if (tid < kPtThreads) {
    float yacc[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) yacc[e] = 0.f;
    for (int st = 0; st < Hq; ++st) {
      const int h = (st + cb) % Hq;
      ok = tc::ring_acquire(ring, st) && ok;
      float v[32];
      tc::tmem_ld32(tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16) + (st % kPtAcc) * kPtN + half * 32, v);
      tc::ring_release(ring, st);  // accumulator read
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] += __shfl_xor_sync(0xffffffffu, v[e], 1);  // hi + lo row
      if (hirow && b < B) {
        const float is = sinv[h * 2 * kPtBatch + (b - bb * kPtBatch) * 2 + (drow ? 1 : 0)];  // undo the row scale
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] *= is;
        if (!drow) {
#pragma unroll
          for (int e = 0; e < 32; ++e) yacc[e] += v[e];
        } else {
          float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int e = 0; e < 32; ++e) s4[e & 3] += fabsf(v[e]);
          part[(static_cast<long>(b) * Hq + h) * (2 * ncb) + 2 * cb + half] = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        }
      }
    }
    if (y && hirow && !drow && b < B) {
      float4* dst = reinterpret_cast<float4*>(y + static_cast<long>(b) * hidden + cb * kPtN + half * 32);
#pragma unroll
      for (int e = 0; e < 8; ++e) dst[e] = make_float4(yacc[4 * e], yacc[4 * e + 1], yacc[4 * e + 2], yacc[4 * e + 3]);
    }
  }
  if (!ok) atomicExch(&bad, 1);
  tc::cta_teardown(tbase, kPtAcc * kPtN);
  if (bad && tid < kPtThreads && hirow && b < B) {  // a wait gave up: mark this CTA's outputs
    if (y && !drow)
      for (int e = 0; e < 32; ++e) y[static_cast<long>(b) * hidden + cb * kPtN + half * 32 + e] = __int_as_float(0x7fc00000);
    if (drow)
      for (int h = 0; h < Hq; ++h) part[(static_cast<long>(b) * Hq + h) * (2 * ncb) + 2 * cb + half] = __int_as_float(0x7fc00000);
  }
}

// pert[b][h] = sum of the 2 * ncb partial sums, in column order.  One warp per (b, h).
__global__ void perturb_reduce_kernel(const float* __restrict__ part, int n, int nparts, float* __restrict__ pert) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (w >= n) return;
  float s = 0.f;
  for (int j = lane; j < nparts; j += 32) s += part[static_cast<long>(w) * nparts + j];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) pert[w] = s;
}

// Without W_O: pert[b][h] = sum_k |o - o_hat| over D.  One warp per (b, h).
__global__ void perturb_raw_kernel(const float* __restrict__ o, const float* __restrict__ o_hat, int n,
                                   float* __restrict__ pert) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (w >= n) return;
  float s = 0.f;
  for (int k = lane; k < kD; k += 32) s += fabsf(o[static_cast<long>(w) * kD + k] - o_hat[static_cast<long>(w) * kD + k]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) pert[w] = s;
}

size_t a_bytes(int B, int Hq) { return align_up(static_cast<size_t>(Hq) * pt_blocks(B) * kPtABytes, 256); }
size_t invs_bytes(int B, int Hq) {
  return align_up(static_cast<size_t>(Hq) * pt_blocks(B) * kPtBatch * 2 * sizeof(float), 256);
}

}  // namespace
}  // namespace mikv

using namespace mikv;

extern "C" size_t mikv_output_perturbation_workspace_bytes(int B, int Hq, int hidden) {
  if (B < 1 || Hq < 1 || hidden < kPtN) return 0;
  return a_bytes(B, Hq) + invs_bytes(B, Hq) +
         align_up(static_cast<size_t>(B) * Hq * 2 * (hidden / kPtN) * sizeof(float), 256);
}

extern "C" int mikv_output_perturbation(const float* o, const float* o_hat, const uint16_t* w_o_t, int B, int Hq,
                                        int D, int hidden, float* y, float* pert, void* ws, size_t ws_bytes,
                                        void* stream) {
  clear_error();
  if (!o) return fail(MIKV_EINVAL, "output_perturbation: null o");
  if (D != kD) return fail(MIKV_EUNSUPPORTED, "output_perturbation: D=%d (only %d)", D, kD);
  if (B < 1 || Hq < 1 || Hq > kPtMaxHq) return fail(MIKV_ESHAPE, "output_perturbation: B=%d Hq=%d", B, Hq);
  if (pert && !o_hat) return fail(MIKV_EINVAL, "output_perturbation: pert needs o_hat");
  if (!y && !pert) return MIKV_OK;
  cudaStream_t s = as_stream(stream);
  if (!w_o_t) {
    if (y) return fail(MIKV_EINVAL, "output_perturbation: y needs w_o_t");
    const int n = B * Hq;
    perturb_raw_kernel<<<(n + 7) / 8, 256, 0, s>>>(o, o_hat, n, pert);
    return check_launch("perturb_raw_kernel");
  }
  if (hidden < kPtN || hidden % kPtN)
    return fail(MIKV_ESHAPE, "output_perturbation: hidden=%d (multiple of %d)", hidden, kPtN);
  if (static_cast<long>(Hq) * pt_blocks(B) * kPtRows > (1L << 31) - 1 || static_cast<long>(Hq) * kD > (1L << 31) - 1)
    return fail(MIKV_ESHAPE, "output_perturbation: too large");
  if (!ws) return fail(MIKV_EINVAL, "output_perturbation: null workspace");
  const size_t need = mikv_output_perturbation_workspace_bytes(B, Hq, hidden);
  if (ws_bytes < need) return fail(MIKV_ESHAPE, "output_perturbation: workspace %zu < %zu", ws_bytes, need);
  if (!aligned16(o) || (o_hat && !aligned16(o_hat)) || !aligned16(w_o_t) || !aligned16(ws) || (y && !aligned16(y)))
    return fail(MIKV_EALIGN, "output_perturbation: o / o_hat / w_o_t / ws / y alignment");
  const int nbb = pt_blocks(B), ncb = hidden / kPtN;
  __half* a = static_cast<__half*>(ws);
  float* invs = reinterpret_cast<float*>(static_cast<char*>(ws) + a_bytes(B, Hq));
  float* part = reinterpret_cast<float*>(static_cast<char*>(ws) + a_bytes(B, Hq) + invs_bytes(B, Hq));
  const int nwarp = Hq * nbb * kPtBatch;
  perturb_prep_kernel<<<(nwarp + 7) / 8, 256, 0, s>>>(o, o_hat, B, Hq, a, invs);
  if (int e = check_launch("perturb_prep_kernel")) return e;
  CUtensorMap ta, tw;
  if (int e = tc::encode_rows(&ta, a, static_cast<long>(Hq) * nbb * kPtRows, "output_perturbation: operand")) return e;
  if (int e = tc::encode_rows(&tw, w_o_t, hidden, "output_perturbation: w_o_t", static_cast<long>(Hq) * kD, kPtN))
    return e;
  const int smem = kPtSmem + Hq * 2 * kPtBatch * static_cast<int>(sizeof(float));
  if (cudaFuncSetAttribute(perturb_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return check_launch("perturb_tc_kernel attribute");
  perturb_tc_kernel<<<dim3(ncb, nbb), kPtBlock, smem, s>>>(ta, tw, B, Hq, hidden, invs, y, part);
  if (int e = check_launch("perturb_tc_kernel")) return e;
  if (!pert) return MIKV_OK;
  const int n = B * Hq;
  perturb_reduce_kernel<<<(n + 7) / 8, 256, 0, s>>>(part, n, 2 * ncb, pert);
  return check_launch("perturb_reduce_kernel");
}
