// W4 group-quantized verification projection for small M (1..64 rows), with
// two epilogues: store y (vq_linear) or a fused greedy arg max over the
// output columns (vq_vocab_argmax).
//
// What is computed (dflash-mlx #7 "perf: tune DFlash2 M=8 verification for
// M1 and M2", PR description: VerifyQuantizedLinear over 4-bit weights;
// ds4 #778 "dspark: fold first-token forward into verify ...", commit 1: one
// pass over the weights serves every row of the verify block):
//
//   y[m][n] = sum_g ( scale[n][g] * A_g[m][n] + bias[n][g] * X_g[m] )
//   A_g[m][n] = sum_{k in group g} code(n,k) * x[m][k]      (exact products)
//   X_g[m]    = sum_{k in group g} x[m][k]
//
// which is the definition sum_k x[m][k] * (scale*code + bias) regrouped per
// 64-wide group. Codes are integers 0..15, exact in bf16 / f16, so every
// product inside the tensor-core MMA is exact and the group sum A_g is an
// fp32 accumulation; the scale is applied once per group in fp32.
//
// Block structure (one CTA per SM, persistent over work units):
//   consumers   8*KH warps. Warp w owns weight rows 16*(w%8) .. +15 of the
//               128-row unit and, when KH = 2, one half of every stage's 8
//               groups (the two halves are summed at the end of the unit).
//               Per 64-wide group it reads its codes from shared memory,
//               turns nibbles into bf16/f16 integers in registers and issues
//               mma.sync m16n8k16 with the weights as the 16-row A operand
//               and the M activation rows as the n8 operand(s), then folds
//               the group into fp32 totals.
//   producer    one lane streams each stage (128 rows x 512 k of packed
//               codes, their scales and biases, and the matching x[M][512])
//               from HBM with cp.async.bulk.tensor (TMA) into a D-deep ring
//               of shared-memory stages, completion tracked by mbarriers.
//   helper      one warp computes X_g[m] for the 8 groups of each stage once
//               per CTA and rewrites the stage's 16-bit x in place into the
//               MMA's B-fragment order, so consumers load fragments directly.
// Every weight byte crosses HBM exactly once per call, for all M rows.
//
// MMA row i (0..7) of a warp maps to weight row 2i and MMA row i+8 to weight
// row 2i+1: with the 128-byte TMA swizzle this puts the four rows read by a
// half-warp on four different bank quarters.
//
// Code layout inside a group: thread (g, t) of a warp (g = lane/4,
// t = lane%4) reads the two 32-bit words 2t, 2t+1 of its rows' 8-word group,
// i.e. codes k = 16t .. 16t+15. Nibble pair (i, i+4) of a word lands in one
// bf16x2 register with a single AND/OR against the exponent pattern of
// 128.0 (bf16) or 1024.0 (f16), i.e. as the exact integers 128+q / 1024+q;
// the offset is removed in the fold (bias - 128*scale multiplies X_g). The
// MMA's k order within the group is permuted to match the pairs, and x is
// stored in the same permuted order, so no shuffles of weights are needed.
// fp32 activations (W4A32) are split into three bf16 terms whose sum is x
// exactly; there the codes are made exact (offset subtracted) before the MMA.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "vq_common.cuh"

namespace vq {

constexpr int kBN = 128;             // weight rows per work unit
constexpr int kBK = 512;             // k per pipeline stage: 8 groups of 64
constexpr int kRowTiles = kBN / 16;  // 16-row MMA tiles per unit
constexpr int kMaxStages = 8;
constexpr int kWeightBoxBytes = kBN * 128;   // 128 rows x 32 words
constexpr int kSmemLimit = 232448;           // 227 KiB opt-in per block
// misc area after the stage ring: 3 x 8 mbarriers, flags, arg max scratch
constexpr int kMiscBytes = 256 + 2 * kRowTiles * 64 * 4;

// K-halves per stage (consumer warps = 8 * KH): two for the small-M variants,
// which are latency-bound, one for the large-M variants, which are bound by
// MMA issue and need the registers.
__host__ __device__ constexpr int kh_for(int MT) { return MT <= 2 ? 2 : 1; }
__host__ __device__ constexpr int threads_for(int MT) { return (kRowTiles * kh_for(MT) + 2) * 32; }
// bytes of the end-of-unit reduction of the two K-halves
__host__ __device__ constexpr int red_bytes_for(int MT) { return kh_for(MT) == 2 ? kBN * 8 * MT * 4 : 0; }

struct GemmParams {
  int M, K, N;
  int KT;           // stages along the full K
  int S;            // K splits per row block (1 = no split)
  int n_units;      // row blocks * S
  int D;            // pipeline depth (stages in the shared-memory ring)
  int stage_bytes;
  int off_x, off_s, off_b, off_xs;   // offsets inside a stage (codes at 0)
  int xbox_bytes;   // shared-memory stride between the x boxes of a stage
  uint32_t tx_bytes;
  void* y;
  float* part;                 // split-K partials [S][M][N]
  uint32_t* cnt;               // split-K arrival counters [row blocks]
  unsigned long long* keys;    // arg max keys [M]
  uint32_t* done;              // arg max block counter
  int32_t* argmax;
  float* maxval;
  int32_t* err;
};

struct GemmLaunch {
  GemmParams p;
  CUtensorMap tm_w, tm_s, tm_b, tm_x;
  int grid;
  int MT;
  bool argmax;
  size_t smem;
  cudaStream_t stream;
};

int launch_gemm_bf16(const GemmLaunch& L);
int launch_gemm_f16(const GemmLaunch& L);
int launch_gemm_f32(const GemmLaunch& L);

#ifdef __CUDACC__

// A wait that also gives up when another warp of the block already gave up.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, int32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
      *abort_flag = 1;
      atomicOr(err, kErrWaitTimeout);
      return false;
    }
  }
}

// A wait that ignores the abort flag (used to let issued copies land).
__device__ __forceinline__ void wait_bounded(uint32_t bar, uint32_t parity, int32_t* err) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
      atomicOr(err, kErrWaitTimeout);
      return;
    }
  }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Codes (i, i+4) of a word as a bf16x2 / f16x2 pair. With kExact the pair is
// (q_i, q_{i+4}); otherwise it is (M + q_i, M + q_{i+4}) with M = 128 (bf16)
// or 1024 (f16), one AND/OR and no arithmetic.
template <bool kF16, bool kExact>
__device__ __forceinline__ uint32_t code_pair(uint32_t word, int i) {
  constexpr uint32_t kMagic = kF16 ? 0x64006400u : 0x43004300u;   // 1024.0 / 128.0
  const uint32_t v = lop3_and_or(word >> (4 * i), 0x000F000Fu, kMagic);
  if constexpr (!kExact) {
    return v;
  } else if constexpr (kF16) {
    const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&v),
                              *reinterpret_cast<const __half2*>(&kMagic));
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 h = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v),
                                     *reinterpret_cast<const __nv_bfloat162*>(&kMagic));
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

// Element j (0..3) of four packed bf16 values, widened exactly to fp32.
__device__ __forceinline__ float bf16_at(const uint2& v, int j) {
  const uint32_t w = (j >> 1) ? v.y : v.x;
  return __uint_as_float((j & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

// fp32 x as the exact sum of three bf16 terms, packed as (a, b) pairs.
__device__ __forceinline__ void split3(float a, float b, uint32_t& hi, uint32_t& mid,
                                       uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float ra = a - __low2float(h), rb = b - __high2float(h);
  const __nv_bfloat162 m = __floats2bfloat162_rn(ra, rb);
  const float la = ra - __low2float(m), lb = rb - __high2float(m);
  const __nv_bfloat162 l = __floats2bfloat162_rn(la, lb);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  mid = *reinterpret_cast<const uint32_t*>(&m);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

template <int ACT>
__device__ __forceinline__ void store_out(void* y, size_t i, float v) {
  if constexpr (ACT == VQ_BF16) {
    reinterpret_cast<__nv_bfloat16*>(y)[i] = __float2bfloat16_rn(v);
  } else if constexpr (ACT == VQ_F16) {
    reinterpret_cast<__half*>(y)[i] = __float2half_rn(v);
  } else {
    reinterpret_cast<float*>(y)[i] = v;
  }
}

// Order-preserving 32-bit image of a (non-NaN) float; -0 is folded into +0
// by the caller so that equal values compare equal.
__device__ __forceinline__ uint32_t float_order(float v) {
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float float_from_order(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// (v, n) beats (bv, bn): larger value, or equal value and lower index.
__device__ __forceinline__ bool better(float v, uint32_t n, bool has, float bv, uint32_t bn,
                                       bool bhas) {
  if (!has) return false;
  if (!bhas) return true;
  return v > bv || (v == bv && n < bn);
}

// Four groups (4kh .. 4kh+3) of one 512-wide stage for this thread's weight
// rows r0, r0+1: totals += scale * A_g + bias * X_g per group.
template <int ACT, int MT>
__device__ __forceinline__ void consume_stage(const uint8_t* st, const GemmParams& p, int rt,
                                              int kh, int g, int t, float (&tot)[MT][4]) {
  constexpr bool kF16 = (ACT == VQ_F16);
  constexpr bool kF32 = (ACT == VQ_F32);
  constexpr int MP = 8 * MT;
  // codes enter the MMA as (offset + q) except for fp32 activations
  constexpr float kOffset = kF32 ? 0.f : (kF16 ? 1024.f : 128.f);
  const int r0 = 16 * rt + 2 * g;   // weight rows r0 (MMA row g) and r0+1 (MMA row g+8)
  const uint2 sv0 = *reinterpret_cast<const uint2*>(st + p.off_s + r0 * 16 + kh * 8);
  const uint2 sv1 = *reinterpret_cast<const uint2*>(st + p.off_s + (r0 + 1) * 16 + kh * 8);
  const uint2 bv0 = *reinterpret_cast<const uint2*>(st + p.off_b + r0 * 16 + kh * 8);
  const uint2 bv1 = *reinterpret_cast<const uint2*>(st + p.off_b + (r0 + 1) * 16 + kh * 8);
  const float* xs = reinterpret_cast<const float*>(st + p.off_xs);
  const uint8_t* wbox = st + kh * kWeightBoxBytes;   // groups 4kh .. 4kh+3
  const int sw0 = r0 & 7, sw1 = (r0 + 1) & 7;        // 128-byte swizzle of the two rows

#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const int j = 4 * kh + jj;
    const int cw = 2 * jj + (t >> 1);                 // 16-byte chunk of words 2t, 2t+1
    const uint2 wa = *reinterpret_cast<const uint2*>(wbox + r0 * 128 + ((cw ^ sw0) << 4) +
                                                     ((t & 1) << 3));
    const uint2 wb = *reinterpret_cast<const uint2*>(wbox + (r0 + 1) * 128 + ((cw ^ sw1) << 4) +
                                                     ((t & 1) << 3));
    float acc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t qa = h ? wa.y : wa.x;
      const uint32_t qb = h ? wb.y : wb.x;
      if constexpr (!kF32) {
        // x[m][64j + 16t + 8h + i], stored by the helper as the fragment
        // pairs (x0,x4) (x1,x5) (x2,x6) (x3,x7)
        uint4 xv[MT];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int m = 8 * mt + g;
          xv[mt] = make_uint4(0u, 0u, 0u, 0u);
          if (m < p.M)
            xv[mt] = *reinterpret_cast<const uint4*>(st + p.off_x + j * p.xbox_bytes + m * 128 +
                                                     (((2 * t + h) ^ g) << 4));
        }
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
          uint32_t a[4];
          a[0] = code_pair<kF16, false>(qa, 2 * s2);
          a[1] = code_pair<kF16, false>(qb, 2 * s2);
          a[2] = code_pair<kF16, false>(qa, 2 * s2 + 1);
          a[3] = code_pair<kF16, false>(qb, 2 * s2 + 1);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
            mma_16816<kF16>(acc[mt], a, s2 ? xv[mt].z : xv[mt].x, s2 ? xv[mt].w : xv[mt].y);
        }
      } else {
        // fp32 x: half-group boxes of 32 values; this thread's 8 values are
        // chunks c, c+1 of line m in box 2j + t/2
        float4 x0[MT], x1[MT];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int m = 8 * mt + g;
          const int c = 4 * (t & 1) + 2 * h;
          x0[mt] = x1[mt] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (m < p.M) {
            const uint8_t* line = st + p.off_x + (2 * j + (t >> 1)) * p.xbox_bytes + m * 128;
            x0[mt] = *reinterpret_cast<const float4*>(line + ((c ^ g) << 4));
            x1[mt] = *reinterpret_cast<const float4*>(line + (((c + 1) ^ g) << 4));
          }
        }
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
          uint32_t a[4];
          a[0] = code_pair<false, true>(qa, 2 * s2);
          a[1] = code_pair<false, true>(qb, 2 * s2);
          a[2] = code_pair<false, true>(qa, 2 * s2 + 1);
          a[3] = code_pair<false, true>(qb, 2 * s2 + 1);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const float e0 = s2 ? x0[mt].z : x0[mt].x;   // x_{2s'}
            const float e4 = s2 ? x1[mt].z : x1[mt].x;   // x_{2s'+4}
            const float e1 = s2 ? x0[mt].w : x0[mt].y;   // x_{2s'+1}
            const float e5 = s2 ? x1[mt].w : x1[mt].y;   // x_{2s'+5}
            uint32_t b0h, b0m, b0l, b1h, b1m, b1l;
            split3(e0, e4, b0h, b0m, b0l);
            split3(e1, e5, b1h, b1m, b1l);
            mma_16816<false>(acc[mt], a, b0h, b1h);
            mma_16816<false>(acc[mt], a, b0m, b1m);
            mma_16816<false>(acc[mt], a, b0l, b1l);
          }
        }
      }
    }

    // fold group j: scale the code sums; the bias term (less the code
    // offset) multiplies the group sum of x
    const float s_a = bf16_at(sv0, jj), s_b = bf16_at(sv1, jj);
    const float c_a = fmaf(-kOffset, s_a, bf16_at(bv0, jj));
    const float c_b = fmaf(-kOffset, s_b, bf16_at(bv1, jj));
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const float2 xsum = *reinterpret_cast<const float2*>(xs + j * MP + 8 * mt + 2 * t);
      tot[mt][0] = fmaf(s_a, acc[mt][0], fmaf(c_a, xsum.x, tot[mt][0]));
      tot[mt][1] = fmaf(s_a, acc[mt][1], fmaf(c_a, xsum.y, tot[mt][1]));
      tot[mt][2] = fmaf(s_b, acc[mt][2], fmaf(c_b, xsum.x, tot[mt][2]));
      tot[mt][3] = fmaf(s_b, acc[mt][3], fmaf(c_b, xsum.y, tot[mt][3]));
    }
  }
}

// Helper work on one landed stage: X_g[m] for every group and row, and (for
// 16-bit x) each 16-byte chunk of x rewritten in place as the fragment pairs
// (x0,x4) (x1,x5) (x2,x6) (x3,x7).
template <int ACT, int MT>
__device__ __forceinline__ void prepare_stage(uint8_t* st, const GemmParams& p, int lane) {
  constexpr int MP = 8 * MT;
  float* xs = reinterpret_cast<float*>(st + p.off_xs);
  for (int idx = lane; idx < 8 * MP; idx += 32) {
    const int j = idx / MP, m = idx - (idx / MP) * MP;
    float s = 0.f;
    if (m < p.M) {
      if constexpr (ACT == VQ_F32) {
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          const uint8_t* line = st + p.off_x + (2 * j + hb) * p.xbox_bytes + m * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 v = *reinterpret_cast<const float4*>(line + ((c ^ (m & 7)) << 4));
            s += v.x;
            s += v.y;
            s += v.z;
            s += v.w;
          }
        }
      } else {
        uint8_t* line = st + p.off_x + j * p.xbox_bytes + m * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4* ptr = reinterpret_cast<uint4*>(line + ((c ^ (m & 7)) << 4));
          const uint4 v = *ptr;
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if constexpr (ACT == VQ_F16) {
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
              s += f.x;
              s += f.y;
            } else {
              s += __uint_as_float(w[e] << 16);
              s += __uint_as_float(w[e] & 0xFFFF0000u);
            }
          }
          *ptr = make_uint4(prmt(v.x, v.z, 0x5410u), prmt(v.x, v.z, 0x7632u),
                            prmt(v.y, v.w, 0x5410u), prmt(v.y, v.w, 0x7632u));
        }
      }
    }
    xs[idx] = s;
  }
  // the slot is refilled by TMA (async proxy) after these generic writes
  fence_proxy_async_smem();
}

template <int ACT, int MT, bool ARGMAX>
__global__ void __launch_bounds__(threads_for(MT), 1)
    vq_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s,
                   const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_x,
                   const GemmParams p) {
  constexpr int MP = 8 * MT;
  constexpr int KH = kh_for(MT);
  constexpr int kConsumers = kRowTiles * KH;          // consumer warps
  constexpr int kProducerWarp = kConsumers;
  constexpr int kHelperWarp = kConsumers + 1;
  constexpr int kXBoxes = (ACT == VQ_F32) ? 16 : 8;
  constexpr int kXBoxElems = kBK / kXBoxes;
  constexpr uint32_t kEpiThreads = kRowTiles * 32;     // the K-half-0 consumers

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - raw);
  uint8_t* const misc = sbase + p.D * p.stage_bytes;
  const uint32_t misc_a = base + p.D * p.stage_bytes;
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(misc + 192);
  volatile int* const epi_flag = reinterpret_cast<volatile int*>(misc + 196);
  float* const red_v = reinterpret_cast<float*>(misc + 256);
  uint32_t* const red_i = reinterpret_cast<uint32_t*>(misc + 256 + kRowTiles * 64 * 4);
  float* const red_k = reinterpret_cast<float*>(misc + kMiscBytes);   // K-half partials
  auto full_bar = [&](int s) { return misc_a + 8u * s; };
  auto empty_bar = [&](int s) { return misc_a + 64u + 8u * s; };
  auto xsum_bar = [&](int s) { return misc_a + 128u + 8u * s; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.D; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kConsumers + 1);
      mbar_init(xsum_bar(s), 32);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tm_w);
      prefetch_tensormap(&tm_s);
      prefetch_tensormap(&tm_b);
      prefetch_tensormap(&tm_x);
      int q = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
        const int rb = u / p.S, sp = u - rb * p.S;
        const int kt0 = sp * p.KT / p.S, kt1 = (sp + 1) * p.KT / p.S;
        for (int kt = kt0; kt < kt1; ++kt) {
          const int slot = q % p.D;
          const uint32_t ph = (uint32_t)(q / p.D) & 1u;
          if (!wait_or_abort(empty_bar(slot), ph ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t sb = base + slot * p.stage_bytes;
          const uint32_t fb = full_bar(slot);
          mbar_arrive_expect_tx(fb, p.tx_bytes);
          tma_load_2d(sb, &tm_w, kt * (kBK / 8), rb * kBN, fb);
          tma_load_2d(sb + kWeightBoxBytes, &tm_w, kt * (kBK / 8) + 32, rb * kBN, fb);
          tma_load_2d(sb + p.off_s, &tm_s, kt * (kBK / 64), rb * kBN, fb);
          tma_load_2d(sb + p.off_b, &tm_b, kt * (kBK / 64), rb * kBN, fb);
#pragma unroll
          for (int j = 0; j < kXBoxes; ++j)
            tma_load_2d(sb + p.off_x + j * p.xbox_bytes, &tm_x, kt * kBK + j * kXBoxElems, 0, fb);
          ++q;
        }
      }
      if (!ok) {
        // let the copies already issued land before the block can exit
        for (int r = (q > p.D ? q - p.D : 0); r < q; ++r)
          wait_bounded(full_bar(r % p.D), (uint32_t)(r / p.D) & 1u, p.err);
      }
    }
    return;
  }

  if (warp == kHelperWarp) {
    // ------------------------------------------------------------ helper
    int q = 0;
    for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
      const int sp = u - (u / p.S) * p.S;
      const int kt0 = sp * p.KT / p.S, kt1 = (sp + 1) * p.KT / p.S;
      for (int kt = kt0; kt < kt1; ++kt, ++q) {
        const int slot = q % p.D;
        const uint32_t ph = (uint32_t)(q / p.D) & 1u;
        if (wait_or_abort(full_bar(slot), ph, abort_flag, p.err))
          prepare_stage<ACT, MT>(sbase + slot * p.stage_bytes, p, lane);
        mbar_arrive(xsum_bar(slot));
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(slot));
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  const int rt = warp % kRowTiles, kh = warp / kRowTiles;
  const int r0 = 16 * rt + 2 * g;
  float best_v[MT][2];
  uint32_t best_n[MT][2];
  bool best_has[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      best_v[mt][c] = 0.f;
      best_n[mt][c] = 0u;
      best_has[mt][c] = false;
    }

  int q = 0;
  bool aborted = false;
  for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
    const int rb = u / p.S, sp = u - rb * p.S;
    const int kt0 = sp * p.KT / p.S, kt1 = (sp + 1) * p.KT / p.S;
    float tot[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) tot[mt][0] = tot[mt][1] = tot[mt][2] = tot[mt][3] = 0.f;

    for (int kt = kt0; kt < kt1; ++kt, ++q) {
      const int slot = q % p.D;
      const uint32_t ph = (uint32_t)(q / p.D) & 1u;
      const bool ok = !aborted && wait_or_abort(full_bar(slot), ph, abort_flag, p.err) &&
                      wait_or_abort(xsum_bar(slot), ph, abort_flag, p.err);
      if (ok) {
        consume_stage<ACT, MT>(sbase + slot * p.stage_bytes, p, rt, kh, g, t, tot);
        if constexpr (KH == 1)   // one warp per row tile covers both halves
          consume_stage<ACT, MT>(sbase + slot * p.stage_bytes, p, rt, 1, g, t, tot);
      } else {
        aborted = true;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(slot));
    }

    if constexpr (KH == 2) {
      // add the second K-half into the first; red_k is [128 rows][MP]
      if (kh == 1) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            red_k[(r0 + (e >> 1)) * MP + 8 * mt + 2 * t + (e & 1)] = tot[mt][e];
      }
      named_bar_sync(1, kConsumers * 32);
      if (kh == 0) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            tot[mt][e] += red_k[(r0 + (e >> 1)) * MP + 8 * mt + 2 * t + (e & 1)];
      }
      named_bar_sync(1, kConsumers * 32);
      if (kh == 1) continue;
    }

    const int n0 = rb * kBN + r0;   // this thread's rows n0 (e < 2) and n0 + 1
    if constexpr (!ARGMAX) {
      if (p.S == 1) {
        if (!aborted) {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int n = n0 + (e >> 1), m = 8 * mt + 2 * t + (e & 1);
              if (n < p.N && m < p.M) store_out<ACT>(p.y, (size_t)m * p.N + n, tot[mt][e]);
            }
        }
      } else {
        // split K: publish this slice, the last slice to arrive reduces all
        // slices in slice order (deterministic) and stores y
        float* part = p.part + (size_t)sp * p.M * p.N;
        if (!aborted) {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int n = n0 + (e >> 1), m = 8 * mt + 2 * t + (e & 1);
              if (n < p.N && m < p.M) __stcg(part + (size_t)m * p.N + n, tot[mt][e]);
            }
        }
        __threadfence();
        named_bar_sync(2, kEpiThreads);
        if (threadIdx.x == 0) *epi_flag = (atomicAdd(p.cnt + rb, 1u) == (uint32_t)(p.S - 1));
        named_bar_sync(2, kEpiThreads);
        if (*epi_flag) {
          __threadfence();
          if (!aborted) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int n = n0 + (e >> 1), m = 8 * mt + 2 * t + (e & 1);
                if (n < p.N && m < p.M) {
                  float s = 0.f;
                  for (int k = 0; k < p.S; ++k)
                    s += __ldcg(p.part + ((size_t)k * p.M + m) * p.N + n);
                  store_out<ACT>(p.y, (size_t)m * p.N + n, s);
                }
              }
          }
          if (threadIdx.x == 0) p.cnt[rb] = 0u;
        }
        named_bar_sync(2, kEpiThreads);
      }
    } else {
      // running arg max per output row m over this thread's columns n
      // (n grows monotonically for a thread, so strict '>' keeps the lowest)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int n = n0 + (e >> 1), c = e & 1;
          const float v = tot[mt][e] + 0.0f;   // -0 -> +0
          if (!aborted && n < p.N && !(v != v)) {
            if (!best_has[mt][c] || v > best_v[mt][c]) {
              best_v[mt][c] = v;
              best_n[mt][c] = (uint32_t)n;
              best_has[mt][c] = true;
            }
          }
        }
    }
  }

  if constexpr (ARGMAX) {
    if (KH == 2 && kh == 1) return;
    // reduce over the 8 row-lanes g of the warp, then over the 8 row tiles
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float v = best_v[mt][c];
        uint32_t n = best_n[mt][c];
        bool h = best_has[mt][c];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, v, off);
          const uint32_t on = __shfl_xor_sync(0xffffffffu, n, off);
          const bool oh = __shfl_xor_sync(0xffffffffu, (int)h, off) != 0;
          if (better(ov, on, oh, v, n, h)) {
            v = ov;
            n = on;
            h = true;
          }
        }
        if (g == 0) {
          const int m = 8 * mt + 2 * t + c;
          red_v[rt * 64 + m] = v;
          red_i[rt * 64 + m] = h ? n : 0xFFFFFFFFu;
        }
      }
    named_bar_sync(2, kEpiThreads);
    if (threadIdx.x < MP) {
      const int m = threadIdx.x;
      float v = 0.f;
      uint32_t n = 0u;
      bool h = false;
      for (int w = 0; w < kRowTiles; ++w) {
        const uint32_t on = red_i[w * 64 + m];
        const float ov = red_v[w * 64 + m];
        if (better(ov, on, on != 0xFFFFFFFFu, v, n, h)) {
          v = ov;
          n = on;
          h = true;
        }
      }
      if (h && m < p.M && !aborted) {
        const unsigned long long key =
            ((unsigned long long)float_order(v) << 32) | (unsigned long long)(0xFFFFFFFFu - n);
        atomicMax(p.keys + m, key);
      }
    }
    __threadfence();
    named_bar_sync(2, kEpiThreads);
    if (threadIdx.x == 0) *epi_flag = (atomicAdd(p.done, 1u) == gridDim.x - 1);
    named_bar_sync(2, kEpiThreads);
    if (*epi_flag) {
      __threadfence();
      if (threadIdx.x < p.M) {
        const int m = threadIdx.x;
        const unsigned long long key = atomicExch(p.keys + m, 0ull);
        if (key == 0ull) {
          p.argmax[m] = 0;
          if (p.maxval) p.maxval[m] = __uint_as_float(0x7FC00000u);
        } else {
          p.argmax[m] = (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
          if (p.maxval) p.maxval[m] = float_from_order((uint32_t)(key >> 32));
        }
      }
      if (threadIdx.x == 0) *p.done = 0u;
    }
  }
}

template <int ACT, int MT, bool AM>
int launch_one(const GemmLaunch& L) {
  auto k = vq_gemm_kernel<ACT, MT, AM>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem) !=
      cudaSuccess)
    return VQ_ECUDA;
  k<<<L.grid, threads_for(MT), L.smem, L.stream>>>(L.tm_w, L.tm_s, L.tm_b, L.tm_x, L.p);
  return cudaGetLastError() == cudaSuccess ? VQ_OK : VQ_ECUDA;
}

template <int ACT>
int launch_gemm_act(const GemmLaunch& L) {
#define VQ_CASE(mt)                                                      \
  case mt:                                                               \
    return L.argmax ? launch_one<ACT, mt, true>(L) : launch_one<ACT, mt, false>(L);
  if constexpr (ACT == VQ_F32) {
    switch (L.MT) {
      VQ_CASE(1)
      VQ_CASE(2)
      VQ_CASE(4)
      default:
        return VQ_EUNSUPPORTED;
    }
  } else {
    switch (L.MT) {
      VQ_CASE(1)
      VQ_CASE(2)
      VQ_CASE(4)
      VQ_CASE(8)
      default:
        return VQ_EUNSUPPORTED;
    }
  }
#undef VQ_CASE
}

#endif  // __CUDACC__

}  // namespace vq
