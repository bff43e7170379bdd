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
// and block of 64 batch rows, one 256-row fp16 operand tile: four rows per batch row, o and
// d = o - o^ each scaled by a power of two (max magnitude in [2^13, 2^14)) and split into two
// fp16 rows (hi = fp16(x), lo = fp16(x - hi): ~22 bits, so the products stay near fp32
// accuracy for differences of any size).  The product kernel (one CTA per 128 hidden columns,
// chunk of heads and batch block) streams, head by head, the head's 128 x 128 block of W_O^T
// (the MMA's M operand) and the operand tile (N = 256) as 64-channel k-blocks through a
// four-stage TMA ring (one thread issues the copies, another the MMAs, so neither waits on
// the other's barriers), multiplies them with tcgen05.mma into one of two TMEM accumulators, and
// the consumers add hi + lo, accumulate y over the chunk's heads in registers and sum |z| of
// the d rows per (batch row, head).  One small kernel adds the chunks' y and the column
// blocks' sums in a fixed order.  The three launches are chained with programmatic dependent
// launch: each is placed while its predecessor runs and waits for it before reading what the
// predecessor writes (the product kernel requests its first W_O^T k-blocks before that wait).
#include <algorithm>

#include "common.cuh"
#include "tcgen05.cuh"

namespace mikv {
namespace {

constexpr int kPtM = tc::kTileRows;              // hidden columns per CTA (the MMA's M)
constexpr int kPtBatch = 64;                     // batch rows per block
constexpr int kPtN = 4 * kPtBatch;               // operand rows: (o, d) x (hi, lo) per batch row
constexpr int kPtThreads = 256;                  // consumers
constexpr int kPtBlock = kPtThreads + 64;        // + the copy warp and the MMA warp
constexpr int kPtCopyThread = kPtThreads, kPtMmaThread = kPtThreads + 32;
constexpr int kPtWBytes = kPtM * 64 * 2;         // one 64-channel k-block of the W^T block: 16 KB
constexpr int kPtOBytes = kPtN * 64 * 2;         // one k-block of the operand tile: 32 KB
constexpr int kPtStage = kPtWBytes + kPtOBytes;  // 48 KB
constexpr long kPtOTile = static_cast<long>(kPtN) * kD * 2;  // a whole operand tile in global memory: 64 KB
constexpr int kPtRing = 4;                       // stages: two per head, three in flight
constexpr int kPtSmem = kPtRing * kPtStage + 1024;  // + the chunk's row scales
constexpr int kPtMaxHq = 128;
constexpr uint32_t kPtIdesc = tc::idesc_f16(kPtM, kPtN);
using PtRing = tc::Ring<kPtRing, 2>;

__host__ __device__ constexpr int pt_blocks(int B) { return (B + kPtBatch - 1) / kPtBatch; }
// Head chunks per (column block, batch block): as many as fill one wave of CTAs (one per SM of
// the current device), at most one head each, and enough that a chunk's row scales (512 B a
// head) fit beside the ring in shared memory (at most kPtMaxChunkHeads heads).
constexpr int kPtMaxChunkHeads = 48;  // 24 KB of row scales beside the 193 KB ring
inline int pt_chunks(int Hq, int ncb, int nbb) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 148;
  const int fill = std::max(1, std::min(Hq, sms / std::max(1, ncb * nbb)));
  return std::max(fill, (Hq + kPtMaxChunkHeads - 1) / kPtMaxChunkHeads);
}
__host__ __device__ inline int pt_chunk_begin(int Hq, int nch, int c) { return static_cast<int>(static_cast<long>(Hq) * c / nch); }

// One warp per (head h, batch row b < 64 * nbb): the four operand rows of (b, h) in the tile
// of (h, b / 64): r = 4 * (b % 64) + 2 * {0: o, 1: d} + {0: hi, 1: lo}, d = o - o_hat.  Each
// row (b, h, o | d) is first scaled by a power of two that brings its largest magnitude into
// [2^13, 2^14), exactly, so that neither part falls into fp16's subnormal range;
// invs[(h * 64 * nbb + b) * 2 + {0: o, 1: d}] receives the inverse.  Rows b >= B are zero.
__global__ void perturb_prep_kernel(const float* __restrict__ o, const float* __restrict__ o_hat, int B, int Hq,
                                    __half* __restrict__ a, float* __restrict__ invs) {
  pdl_trigger();
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
  __half* tile = a + static_cast<long>(h * nbb + bb) * kPtN * kD;
  const int r0 = 4 * (b % kPtBatch);
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
    __half2* rh = reinterpret_cast<__half2*>(tile + (r0 + 2 * part) * kD + 4 * lane);
    __half2* rl = reinterpret_cast<__half2*>(tile + (r0 + 2 * part + 1) * kD + 4 * lane);
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

// D (TMEM, 128 hidden columns x 256 operand rows) (+)= one 64-channel k-block: the W^T
// k-block (128 rows x 128 B) times the operand k-block (256 rows x 128 B), 4 K steps of 16.
__device__ __forceinline__ void mma_w_o_kblock(uint32_t tmem_d, uint32_t sw, uint32_t so, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    tc::mma_f16(tmem_d, tc::smem_desc(sw + kk * 32), tc::smem_desc(so + kk * 32), kPtIdesc, accumulate || kk > 0);
}

// Lane l of the warp ends with the sum over the 32 lanes of v[l] (butterfly reduce-scatter:
// at offset r each lane keeps the half of its values selected by bit r of its index).
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int r = 16, n = 16; r >= 1; r >>= 1, n >>= 1) {
    const bool up = (lane & r) != 0;
#pragma unroll
    for (int j = 0; j < n; ++j) {
      const float send = up ? v[j] : v[j + n];
      const float keep = up ? v[j + n] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, r);
    }
  }
  return v[0];
}

// CTA (column block cb of 128 hidden columns, head chunk hc, batch block bb).  For each head
// h of the chunk, its two 64-channel k-blocks of the W^T block (rows cb*128) and of the operand
// tile of (h, bb) go through a four-stage TMA ring (48 KB a stage); tcgen05.mma accumulates
// them into one of two 256-column TMEM accumulators (TMEM lane = hidden column, column =
// operand row).
// Consumer thread (lane = hidden column c, half) reads the 128 columns of batch rows
// 32 * half .. + 32: y[b] += (o_hi + o_lo) * 2^-eo for the chunk's heads (written once as the
// chunk's partial), |z| = |d_hi + d_lo| * 2^-ed summed over the 128 columns per (b, h) by a
// warp reduce-scatter and a shared-memory add over the four lane quarters.
__global__ void __launch_bounds__(kPtBlock, 1) perturb_tc_kernel(const __grid_constant__ CUtensorMap tw,
                                                                 const __grid_constant__ CUtensorMap to, int B,
                                                                 int Hq, int hidden,
                                                                 const float* __restrict__ invs,
                                                                 float* __restrict__ ypart, float* __restrict__ part) {
  extern __shared__ __align__(128) uint8_t sm[];  // kPtRing stages of (W tile, operand tile), row scales
  __shared__ __align__(8) PtRing ring;
  __shared__ uint32_t tslot;
  __shared__ float red[2][8][32];
  __shared__ int bad;
  pdl_trigger();
  const int cb = blockIdx.x, hc = blockIdx.y, bb = blockIdx.z, nbb = gridDim.z, Bp = nbb * kPtBatch;
  const int ncb = hidden / kPtM;
  const int nch = gridDim.y;
  const int h0 = pt_chunk_begin(Hq, nch, hc), nh = pt_chunk_begin(Hq, nch, hc + 1) - h0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, half = (tid >> 7) & 1;
  const int col = cb * kPtM + (warp & 3) * 32 + lane;  // a consumer's hidden column
  const uint32_t s0 = tc::smem_base(sm);
  float* sinv = reinterpret_cast<float*>(sm + (s0 - smem_u32(sm)) + kPtRing * kPtStage);  // [nh][64][2]
  if (tid == 0) bad = 0;
  const uint32_t tbase = tc::ring_setup(ring, &tslot, kPtThreads, 2 * kPtN);
  tc::Waits w;
  // Step s = k-block s % 2 of head h0 + s / 2: the W^T k-block at rows cb*128, channels
  // h*128 + 64*(s % 2), and the operand tile's k-block, into stage s % kPtRing (one
  // transaction count on full[stage] for both copies).
  const int nsteps = 2 * nh;
  auto load_w = [&](int s, int st) {
    const int h = h0 + s / 2, kb = s % 2;
    const uint32_t sw = s0 + st * kPtStage, mb = smem_u32(&ring.full[st]);
    tc::mbar_expect_tx(mb, kPtStage);
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(sw), "l"(&tw), "r"(h * kD + kb * 64), "r"(cb * kPtM), "r"(mb)
        : "memory");
  };
  auto load_o = [&](int s, int st) {
    const int h = h0 + s / 2, kb = s % 2;
    const uint32_t so = s0 + st * kPtStage + kPtWBytes, mb = smem_u32(&ring.full[st]);
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(so), "l"(&to), "r"(kb * 64), "r"((h * nbb + bb) * kPtN), "r"(mb)
        : "memory");
  };
  // W_O^T is an input of the call, complete before the prep kernel (a normal launch) started,
  // and this kernel starts only after that: its first k-blocks are requested before waiting
  // for the prep kernel's operand tiles and row scales.
  if (tid == kPtCopyThread)
    for (int st = 0; st < nsteps && st < kPtRing; ++st) load_w(st, st);
  pdl_wait();
  for (int j = tid; j < nh * 2 * kPtBatch; j += kPtBlock)
    sinv[j] = invs[(static_cast<long>(h0 + j / (2 * kPtBatch)) * Bp + bb * kPtBatch) * 2 + j % (2 * kPtBatch)];
  __syncthreads();  // publishes sinv
  if (tid == kPtCopyThread) {
    // copies: step st into stage st % kPtRing once the MMAs of step st - kPtRing are done
    for (int st = 0; st < nsteps && st < kPtRing; ++st) load_o(st, st);
    for (int st = kPtRing; st < nsteps; ++st) {
      const int b = st % kPtRing;
      w(smem_u32(&ring.empty[b]), (st / kPtRing - 1) & 1);
      if (w.ok) {  // after a give-up nothing more is issued
        load_w(st, b);
        load_o(st, b);
      }
    }
    for (int st = nsteps > kPtRing ? nsteps - kPtRing : 0; st < nsteps; ++st)  // the last commits landed
      w(smem_u32(&ring.empty[st % kPtRing]), (st / kPtRing) & 1);
  } else if (tid == kPtMmaThread) {
    // MMAs: step st as soon as its stage landed; the head's accumulator (h & 1) is committed
    // after its second k-block, and the first waits until head h - 2 was read from it
    for (int st = 0; st < nsteps; ++st) {
      const int b = st % kPtRing, hl = st / 2, a = hl & 1;
      w(smem_u32(&ring.full[b]), (st / kPtRing) & 1);
      if (st % 2 == 0 && hl >= 2) w(smem_u32(&ring.freed[a]), ((hl - 2) / 2) & 1);
      tc::fence_after_sync();
      const uint32_t sw = s0 + b * kPtStage;
      if (w.ok) {  // after a give-up nothing more is issued
        mma_w_o_kblock(tbase + a * kPtN, sw, sw + kPtWBytes, st % 2 == 1);
        tc::commit(smem_u32(&ring.empty[b]));
        if (st % 2 == 1) tc::commit(smem_u32(&ring.mma[a]));
      }
    }
  } else if (tid < kPtThreads) {
    float y[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) y[i] = 0.f;
    for (int s = 0; s < nh; ++s) {
      tc::ring_acquire(ring, s, w);
      const float* si = sinv + s * 2 * kPtBatch + half * 64;  // (b_local, o | d) of this half
      float za[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // 8 batch rows per 32 columns
        float v[32];
        tc::tmem_ld32(tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16) + (s & 1) * kPtN + half * 128 + q * 32, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int bi = q * 8 + i;
          y[bi] = fmaf(v[4 * i] + v[4 * i + 1], si[2 * bi], y[bi]);
          za[bi] = fabsf((v[4 * i + 2] + v[4 * i + 3]) * si[2 * bi + 1]);
        }
      }
      tc::ring_release(ring, s);  // accumulator read
      const float zs = reduce_scatter32(za, lane);  // lane l: batch row 32 * half + l
      red[s & 1][warp][lane] = zs;
      tc::consumer_sync<kPtThreads>();
      if (tid < 64) {  // (half, l) = (tid / 32, tid % 32): add the four lane quarters
        const int hf = tid >> 5, l = tid & 31;
        const float t = (red[s & 1][4 * hf][l] + red[s & 1][4 * hf + 1][l]) +
                        (red[s & 1][4 * hf + 2][l] + red[s & 1][4 * hf + 3][l]);
        const int b = bb * kPtBatch + 32 * hf + l;
        if (b < B) part[(static_cast<long>(b) * Hq + h0 + s) * ncb + cb] = t;
      }
    }
    if (ypart) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int b = bb * kPtBatch + 32 * half + i;
        if (b < B) ypart[(static_cast<long>(hc) * B + b) * hidden + col] = y[i];
      }
    }
  }
  if (!w.ok) {
    atomicExch(&bad, 1);
    tc::report_giveup(tc::kGiveupPerturb);
  }
  tc::cta_teardown(tbase, 2 * kPtN);
  if (bad && tid < 64) {  // a wait gave up: mark this CTA's perturbation outputs
    const int b = bb * kPtBatch + tid;
    if (b < B)
      for (int s = 0; s < nh; ++s) part[(static_cast<long>(b) * Hq + h0 + s) * ncb + cb] = __int_as_float(0x7fc00000);
  }
  if (bad && ypart && tid < kPtThreads)
    for (int i = 0; i < 32; ++i) {
      const int b = bb * kPtBatch + 32 * half + i;
      if (b < B) ypart[(static_cast<long>(hc) * B + b) * hidden + col] = __int_as_float(0x7fc00000);
    }
}

// Both ordered reductions in one launch.  Blocks [0, yblocks): y[b][c] = the sum of the head
// chunks' partials, in chunk order (grid-stride over the ny elements).  The other blocks:
// pert[b][h] = the sum of the ncb column-block partial sums, in column order, one warp per
// (b, h) (lane j adds parts j, j + 32, ..., then a butterfly over the lanes).
__global__ void perturb_reduce_kernel(const float* __restrict__ ypart, int nchunk, long ny, float* __restrict__ y,
                                      int yblocks, const float* __restrict__ part, int n, int nparts,
                                      float* __restrict__ pert) {
  pdl_wait();
  if (static_cast<int>(blockIdx.x) < yblocks) {
    for (long i = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; i < ny;
         i += static_cast<long>(yblocks) * blockDim.x) {
      float t = 0.f;
      for (int c = 0; c < nchunk; ++c) t += ypart[c * ny + i];
      y[i] = t;
    }
    return;
  }
  const int w = ((blockIdx.x - yblocks) * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
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

struct PtWs {
  size_t a, invs, part, ypart, total;
};
PtWs pt_ws_layout(int B, int Hq, int hidden) {  // y partials sized for one chunk per head (the most)
  const int nbb = pt_blocks(B);
  PtWs w;
  w.a = 0;
  w.invs = align_up(static_cast<size_t>(Hq) * nbb * kPtOTile, 256);
  w.part = w.invs + align_up(static_cast<size_t>(Hq) * nbb * kPtBatch * 2 * sizeof(float), 256);
  w.ypart = w.part + align_up(static_cast<size_t>(B) * Hq * (hidden / kPtM) * sizeof(float), 256);
  w.total = w.ypart + align_up(static_cast<size_t>(Hq) * B * hidden * sizeof(float), 256);
  return w;
}

}  // namespace
}  // namespace mikv

using namespace mikv;

extern "C" size_t mikv_output_perturbation_workspace_bytes(int B, int Hq, int hidden) {
  if (B < 1 || Hq < 1 || hidden < kPtM) return 0;
  return pt_ws_layout(B, Hq, hidden).total;
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
  if (hidden < kPtM || hidden % kPtM)
    return fail(MIKV_ESHAPE, "output_perturbation: hidden=%d (multiple of %d)", hidden, kPtM);
  if (static_cast<long>(Hq) * pt_blocks(B) * kPtN > (1L << 31) - 1 || static_cast<long>(B) * hidden * Hq > (1L << 31) - 1)
    return fail(MIKV_ESHAPE, "output_perturbation: too large");
  if (!ws) return fail(MIKV_EINVAL, "output_perturbation: null workspace");
  const PtWs L = pt_ws_layout(B, Hq, hidden);
  if (ws_bytes < L.total) return fail(MIKV_ESHAPE, "output_perturbation: workspace %zu < %zu", ws_bytes, L.total);
  if (!aligned16(o) || (o_hat && !aligned16(o_hat)) || !aligned16(w_o_t) || !aligned16(ws))
    return fail(MIKV_EALIGN, "output_perturbation: o / o_hat / w_o_t / ws alignment");
  const int nbb = pt_blocks(B), ncb = hidden / kPtM, nch = pt_chunks(Hq, ncb, nbb);
  char* w = static_cast<char*>(ws);
  __half* a = reinterpret_cast<__half*>(w + L.a);
  float* invs = reinterpret_cast<float*>(w + L.invs);
  float* part = reinterpret_cast<float*>(w + L.part);
  float* ypart = y ? reinterpret_cast<float*>(w + L.ypart) : nullptr;
  const int nwarp = Hq * nbb * kPtBatch;
  perturb_prep_kernel<<<(nwarp + 7) / 8, 256, 0, s>>>(o, o_hat, B, Hq, a, invs);
  if (int e = check_launch("perturb_prep_kernel")) return e;
  CUtensorMap tw, to;
  if (int e = tc::encode_rows(&tw, w_o_t, hidden, "output_perturbation: w_o_t", static_cast<long>(Hq) * kD)) return e;
  if (int e = tc::encode_rows(&to, a, static_cast<long>(Hq) * nbb * kPtN, "output_perturbation: operand", kD, kPtN))
    return e;
  const int hmax = (Hq + nch - 1) / nch;  // heads of the largest chunk
  const int smem = kPtSmem + hmax * 2 * kPtBatch * static_cast<int>(sizeof(float));
  if (cudaFuncSetAttribute(perturb_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return check_launch("perturb_tc_kernel attribute");
  if (int e = check_launch_after(launch_after(perturb_tc_kernel, dim3(ncb, nch, nbb), dim3(kPtBlock), smem, s, tw, to,
                                              B, Hq, hidden, invs, ypart, part),
                                 "perturb_tc_kernel"))
    return e;
  const long ny = y ? static_cast<long>(B) * hidden : 0;
  const int yblocks = static_cast<int>(std::min<long>((ny + 255) / 256, 152L * 8));
  const int n = pert ? B * Hq : 0;
  return check_launch_after(launch_after(perturb_reduce_kernel, dim3(yblocks + (n + 7) / 8), dim3(256), 0, s, ypart,
                                         nch, ny, y, yblocks, part, n, ncb, pert),
                            "perturb_reduce_kernel");
}

namespace mikv {
// This file's wait-status word (see tc::wait_giveups), for mikv_wait_status.
int perturb_wait_giveups(unsigned* out, bool clear) { return tc::wait_giveups(out, clear); }
}  // namespace mikv
