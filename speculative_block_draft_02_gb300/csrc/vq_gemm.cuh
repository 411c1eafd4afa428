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
//   consumers   TEAMS teams of warps; team i takes the stages q with
//               q % TEAMS == i, so one team's stage boundary overlaps the
//               other team's work. Within a team each warp owns RT 16-row MMA
//               tiles of the 128-row unit and a K-slice of GPW groups of its
//               stages (all partial sums of a row tile are added at the end
//               of the unit). Per 64-wide group a warp reads its codes from
//               shared memory, turns nibbles into bf16/f16 integers in
//               registers and issues mma.sync m16n8k16 with the weights as
//               the 16-row A operand and the M activation rows as the n8
//               operand(s), then folds the group into fp32 totals.
//   x           comes one of three ways: (a) vq_linear with 16-bit x and
//               M <= 8: per-stage slices of scaled fp16 fragments, group sums
//               and -U terms, prepared once per call by vq_prep_kernel and
//               copied in next to each stage's weights; (b) the arg max with
//               16-bit x, M <= 8 and several row blocks per block: a per-block
//               fp16 table of all of x; (c) otherwise x per stage by TMA and
//               X_g[m] for every group of K computed once per block from
//               global x while the first stages are in flight.
//   producer    one lane streams each stage (128 rows x 512 k of packed
//               codes, their scales and biases, and the stage's x) from HBM
//               with cp.async.bulk.tensor (TMA) into a D-deep ring of
//               shared-memory stages, completion tracked by mbarriers. The
//               first stages' weights are requested before griddepcontrol.wait,
//               so a call overlaps the tail of the kernel before it.
// Every weight byte crosses HBM exactly once per call, for all M rows. (16-bit
// x with M > 16 runs on the tcgen05 kernel in vq_tc.cuh instead.)
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
// MMA's k order within the group is permuted to match the pairs, and the x
// fragments are permuted the same way with byte permutes, so the weights are
// never shuffled.
// fp32 activations (W4A32) are split into three bf16 terms whose sum is x
// exactly; there the codes are made exact (offset subtracted) before the MMA.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "vq_common.cuh"

namespace vq {

constexpr int kBN = 128;             // weight rows per work unit
constexpr int kBK = 512;             // k per pipeline stage: 8 groups of 64
constexpr int kMaxStages = 8;
constexpr int kWeightBoxBytes = kBN * 128;   // 128 rows x 32 words
constexpr int kSmemLimit = 232448;           // 227 KiB opt-in per block
// misc area after the stage ring: 3 x 8 mbarriers and one more, flags, arg
// max scratch
constexpr int kBarBytes = 320;
constexpr int kMiscBytes = kBarBytes + 3 * 8 * 64 * 4;
// bytes of the misc region: the arg max's cross-warp buffers only with ARGMAX
__host__ __device__ constexpr int misc_bytes(bool argmax) { return argmax ? kMiscBytes : kBarBytes; }

// Work split of the consumers by the number MT of n8 tiles (M <= 8*MT):
// TEAMS teams taking alternate stages, RT 16-row tiles per warp (the tiles
// share the x fragments), KQ K-slices per stage within a team, GPW = 8/KQ
// groups per warp and stage. WIDE != 0 (no K split): half the warps, so that
// with 9 warps a block each has up to 168 registers (17 warps cap them at
// 96). WIDE == 2 (prepared slices): each warp two row tiles over all 8 groups
// of a stage; measured per call at K=5120, N=17408: M=8 10.6 us (four tiles
// over four groups 10.8, two tiles over four groups with 17 warps 12.0), M=16
// 15.2 us (four tiles over four groups spilled its accumulators: 17.0).
// WIDE == 1 (x per stage by TMA: fp32 x, arg max): four row tiles over four
// groups (two tiles over all eight measured 24.8 vs 22.8 us at fp32 M=8).
// With a K split, whose units are one or two stages, the narrower split
// stays faster.
template <int MT, int WIDE = 0>
struct Cfg {
  static constexpr int TEAMS = MT <= 2 ? 2 : 1;   // a power of two
  static constexpr int RT = (MT <= 2 && WIDE == 1) ? 4 : (MT <= 2 ? 2 : 1);
  static constexpr int KQ = (MT <= 2 && WIDE != 2) ? 2 : 1;
  static constexpr int GPW = 8 / KQ;
  static constexpr int RW = 8 / RT;                 // warps along the rows
  static constexpr int WPT = RW * KQ;               // warps per team
  static constexpr int WARPS = WPT * TEAMS;         // consumer warps
  static constexpr int THREADS = (WARPS + 1) * 32;  // + the producer warp
  static constexpr int SLICES = TEAMS * KQ;         // partial sums per row
  static constexpr int RED = (SLICES - 1) * kBN * 8 * MT * 4;
};

// Stage layout in shared memory (bytes from the 1 KiB-aligned stage start):
// codes [2][128 rows][128 B] (two 128-byte TMA boxes, 128-byte swizzle),
// x [groups][8*MT rows][128 B] (swizzled), scales [128][16 B], biases [128][16 B].
__host__ __device__ constexpr int x_boxes(int act) { return act == VQ_F32 ? 16 : 8; }
__host__ __device__ constexpr int stage_off_x() { return 2 * kWeightBoxBytes; }
__host__ __device__ constexpr int stage_off_s(int act, int MT) {
  return stage_off_x() + x_boxes(act) * 128 * 8 * MT;
}
__host__ __device__ constexpr int stage_off_b(int act, int MT) {
  return stage_off_s(act, MT) + kBN * 16;
}
__host__ __device__ constexpr int stage_bytes(int act, int MT) {
  return (stage_off_b(act, MT) + kBN * 16 + 1023) / 1024 * 1024;
}

// x-table variant (16-bit x, M <= 8): the stage holds codes, scales and
// biases only; x lives in a per-block table converted once at block start.
__host__ __device__ constexpr int xt_stage_off_s() { return 2 * kWeightBoxBytes; }
__host__ __device__ constexpr int xt_stage_bytes() {
  return (xt_stage_off_s() + 2 * kBN * 16 + 1023) / 1024 * 1024;
}
// Prepared x slices (vq_linear, 16-bit x, M <= 8): one slice per 512-wide
// stage, [8 groups][8 rows][128 B] fp16 fragments, T [8 groups][8 rows] fp32
// (f * group sums), -U [8 groups][4][4] fp32 (U = 1024 * the group sum of the
// fp16 values, laid out as the MMA accumulator quad (row 2t, 2t+1, 2t, 2t+1)
// of thread t), and 1/f [8 rows] fp32, with f a power of two per (stage,
// row); the slice rides in the stage next to its weights.
constexpr int kSliceT = 8 * 1024;
constexpr int kSliceU = kSliceT + 8 * 8 * 4;
constexpr int kSliceInv = kSliceU + 8 * 4 * 16;
constexpr int kSliceBytes = kSliceInv + 8 * 4;
// With M <= 16 (two n8 tiles) a stage holds one slice per tile, tile mt's
// at xs_stage_off_x() + mt * kSliceBytes (slice-local rows 0..7 = x rows
// 8mt .. 8mt + 7).
__host__ __device__ constexpr int xs_stage_off_x() { return 2 * kWeightBoxBytes + 2 * kBN * 16; }
__host__ __device__ constexpr int xs_stage_bytes(int MT = 1) {
  return (xs_stage_off_x() + MT * kSliceBytes + 1023) / 1024 * 1024;
}

// x table [K/64 groups][8 rows][128 B] fp16, then T [K/64][8] fp32 and 1/f [8]
// fp32 (this much is what a prepared table holds), then the build's scratch:
// [K/64][8] fp32 and the row maxima [8] u32.
__host__ __device__ constexpr int xt_prepared_bytes(int K) { return (K / 64) * 1024 + (K / 64) * 32 + 32; }
__host__ __device__ constexpr int xt_table_bytes(int K) { return xt_prepared_bytes(K) + (K / 64) * 32 + 32; }
constexpr int kMaxXtBytes = 96 * 1024;

// Bytes of the per-block table of group sums X_g[m]: [K/64][8*MT] fp32 (the
// caller passes K rounded up to whole stages; the groups past K are zero).
__host__ __device__ constexpr int xsum_bytes(int K, int MT) { return (K / 64) * 8 * MT * 4; }
constexpr int kMaxXsumBytes = 32 * 1024;

struct GemmParams {
  const void* x;    // activations in global memory (for the group sums)
  int M, K, N;
  int KT;           // stages along K (the last one partial when K % 512 != 0)
  int S;            // K splits per row block (1 = no split)
  int n_units;      // row blocks * S
  int D;            // pipeline depth (stages in the shared-memory ring)
  int pre;          // stages whose weights are requested before griddepcontrol.wait
  // SM clock cycles between those requests while the kernel before this one
  // is still running (0: all at once)
  int pace;
  int red_alias;    // 1: the K-slice partials live in the stage ring (one unit per block)
  int stage_bytes;
  int off_x, off_s, off_b;   // offsets inside a stage (codes at 0)
  int xm;           // x source: 0 per-stage TMA, 1 per-block table, 2 prepared slices,
                    // 3 per-stage TMA for the tensor-core (tcgen05) kernel
  int xs_stage;     // tcgen05 kernel: 1 = group row sums per stage from the x tile,
                    // 0 = a table for all of K
  const void* xprep;  // prepared slices [KT] (xm == 2), written by vq_prep_kernel
  int tab_bytes;    // bytes of the table region after the stage ring (1 KiB multiple)
  int x3d;          // 1: x arrives as one 3-D box per stage, 0: one box per group
                    // (same shared-memory layout either way: [group][8*MT rows][128 B],
                    // rows >= M zero-filled by the copy)
  uint32_t tx_bytes;
  // K not a multiple of 512 (x per stage by TMA only): the rows of scales and
  // biases are not 16-byte multiples, which a TMA tensor map needs, so the
  // producer warp's lanes load each stage's scales and biases themselves
  int sb_plain;
  const uint16_t* scales;   // [N][K/64] bf16 bits
  const uint16_t* biases;
  void* y;
  float* part;                 // split-K partials [S][M][N]
  uint32_t* cnt;               // split-K arrival counters [row blocks]
  unsigned long long* keys;    // arg max keys [M]
  uint32_t* done;              // arg max block counter
  int32_t* argmax;
  float* maxval;
  float* second;               // runner-up logit [M] (top-2 arg max), or null
  uint4* cand;                 // per-block (best, index, runner-up) [grid][M], or null
  int32_t* err;
  // extents (elements) of the buffers the kernels store to, for the checks of
  // bounds-checked builds: y, the split-K partials, the per-block arg max
  // candidates
  size_t y_elems, part_elems, cand_elems;
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

// Scales and biases of one stage (128 rows x 8 groups from row block rb,
// stage kt) with plain loads by the 32 lanes of a warp, rows past N and
// groups past K as zeros, in the layout the TMA box would leave ([row][8]
// bf16, 16 B a row); lane l takes rows l + 32i. For K % 512 != 0, whose rows
// of K/32 bytes no tensor map can describe.
template <typename Params>
__device__ __forceinline__ void load_stage_sb(const Params& p, uint8_t* s_dst, uint8_t* b_dst,
                                              int kt, int rb, int lane) {
  const int G = p.K / 64;
  uint4 vs[4], vb[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const long long n = (long long)rb * 128 + lane + 32 * i;
    uint32_t ws[4] = {0u, 0u, 0u, 0u}, wb[4] = {0u, 0u, 0u, 0u};
    if (n < p.N) {
      const unsigned short* ps = reinterpret_cast<const unsigned short*>(p.scales) + n * G;
      const unsigned short* pb = reinterpret_cast<const unsigned short*>(p.biases) + n * G;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int gi = kt * 8 + j;
        if (gi < G) {
          ws[j >> 1] |= (uint32_t)__ldg(ps + gi) << (16 * (j & 1));
          wb[j >> 1] |= (uint32_t)__ldg(pb + gi) << (16 * (j & 1));
        }
      }
    }
    vs[i] = make_uint4(ws[0], ws[1], ws[2], ws[3]);
    vb[i] = make_uint4(wb[0], wb[1], wb[2], wb[3]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    *reinterpret_cast<uint4*>(s_dst + (lane + 32 * i) * 16) = vs[i];
    *reinterpret_cast<uint4*>(b_dst + (lane + 32 * i) * 16) = vb[i];
  }
}

// A wait that also gives up when another warp of the block already gave up.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, int32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*abort_flag) return false;
      if (clock64() - t0 > kWaitTimeoutCycles) {
        *abort_flag = 1;
        atomicOr(err, kErrWaitTimeout);
        return false;
      }
    }
  }
}

// A wait that ignores the abort flag (used to let issued copies land).
__device__ __forceinline__ void wait_bounded(uint32_t bar, uint32_t parity, int32_t* err) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitTimeoutCycles) {
      atomicOr(err, kErrWaitTimeout);
      return;
    }
  }
}

// Codes (i, i+4) of a word as a bf16x2 / f16x2 pair. With kExact the pair is
// (q_i, q_{i+4}); otherwise it is (B + q_i, B + q_{i+4}) with B = 128 (bf16)
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

// GPW consecutive bf16 values (4, 8 or 16 bytes) as packed words.
template <int GPW>
struct Packed {
  uint32_t w[GPW / 2];
};
template <int GPW>
__device__ __forceinline__ Packed<GPW> lds_packed(const uint8_t* ptr) {
  Packed<GPW> r;
  if constexpr (GPW == 2) {
    r.w[0] = *reinterpret_cast<const uint32_t*>(ptr);
  } else if constexpr (GPW == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(ptr);
    r.w[0] = v.x;
    r.w[1] = v.y;
  } else {
    const uint4 v = *reinterpret_cast<const uint4*>(ptr);
    r.w[0] = v.x;
    r.w[1] = v.y;
    r.w[2] = v.z;
    r.w[3] = v.w;
  }
  return r;
}
template <int GPW>
__device__ __forceinline__ float bf16_of(const Packed<GPW>& p, int jj) {
  const uint32_t w = p.w[jj >> 1];
  return __uint_as_float((jj & 1) ? (w & 0xFFFF0000u) : (w << 16));
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

// Two adjacent 16-bit outputs (index i even) as one 4-byte store.
template <int ACT>
__device__ __forceinline__ void store_out2(void* y, size_t i, float a, float b) {
  if constexpr (ACT == VQ_BF16) {
    *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(y) + i) =
        __floats2bfloat162_rn(a, b);
  } else if constexpr (ACT == VQ_F16) {
    *reinterpret_cast<__half2*>(reinterpret_cast<__half*>(y) + i) = __floats2half2_rn(a, b);
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

// Merges candidate (ov, on, oh, os) into (v, n, h, s): the best by value, ties
// to the lower index, and as runner-up the largest of the other values
// (-inf when there is none). A candidate without a value (oh false) only
// contributes its runner-up, which is then -inf too.
__device__ __forceinline__ void top2_merge(float& v, uint32_t& n, bool& h, float& s, float ov,
                                           uint32_t on, bool oh, float os) {
  if (better(ov, on, oh, v, n, h)) {
    s = fmaxf(os, h ? v : -INFINITY);
    v = ov;
    n = on;
    h = true;
  } else {
    s = fmaxf(s, fmaxf(os, oh ? ov : -INFINITY));
  }
}

// The last block's decode of row m: arg max and maximum from the packed key,
// and (top-2 calls) the runner-up from every block's candidate: the block
// that holds the winning index gives its own runner-up, every other block
// its best.
__device__ __forceinline__ void argmax_decode(const GemmParams& p, int m, unsigned long long key,
                                              int nblocks) {
  const uint32_t n1 = key == 0ull ? 0xFFFFFFFFu : 0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull);
  if (!in_bounds((size_t)m, (size_t)p.M, p.err)) return;
  if (key == 0ull) {
    p.argmax[m] = 0;
    if (p.maxval) p.maxval[m] = __uint_as_float(0x7FC00000u);
  } else {
    p.argmax[m] = (int32_t)n1;
    if (p.maxval) p.maxval[m] = float_from_order((uint32_t)(key >> 32));
  }
  if (p.second) {
    float sec = -INFINITY;
    for (int c = 0; c < nblocks; ++c) {
      const uint4 e = __ldcg(p.cand + (size_t)c * p.M + m);
      if (e.y == 0xFFFFFFFFu) continue;   // no value of row m in that block
      sec = fmaxf(sec, e.y == n1 ? __uint_as_float(e.z) : __uint_as_float(e.x));
    }
    p.second[m] = sec;
  }
}

// Per-thread constants of a consumer: 32-bit shared-memory offsets that do
// not change from stage to stage (the rest of each address is an immediate).
template <int ACT, int MT>
struct LaneOffsets {
  uint32_t w_even, w_odd;   // codes of this thread's even / odd weight row, tile 0
  uint32_t g3x32;           // (g % 4) * 32: the row-dependent part of the swizzle
  uint32_t x_h0, x_h1;      // x: the chunk of row g, first group of the slice, for
                            // k-halves h = 0, 1 (16-bit x); line and chunk (fp32 x)
  uint32_t sc;              // scales of the even row of tile 0 for this K-slice
  uint32_t xs;              // (first group of the slice, row 2t) in the group-sum table, bytes
};

template <int ACT, int MT, int WIDE>
__device__ __forceinline__ LaneOffsets<ACT, MT> lane_offsets(int rw, int kq, int g, int t) {
  using C = Cfg<MT, WIDE>;
  constexpr int MP = 8 * MT;
  LaneOffsets<ACT, MT> o;
  const int row = 16 * (C::RT * rw) + 2 * g;               // even row of tile 0
  const int box = (C::GPW == 4) ? kq * kWeightBoxBytes : 0;
  o.w_even = box + row * 128 + ((t >> 1) << 4) + ((t & 1) << 3);
  o.w_odd = box + (row + 1) * 128 + (((t >> 1) ^ 1) << 4) + ((t & 1) << 3);
  o.g3x32 = (uint32_t)(g & 3) << 5;
  if constexpr (ACT == VQ_F32) {
    // line (half-group 2j + t/2, row g) and the swizzled chunk 4(t&1) ^ g
    const int hg0 = 2 * (kq * C::GPW) + (t >> 1);
    o.x_h0 = stage_off_x() + (hg0 * MP + g) * 128;
    o.x_h1 = (uint32_t)((4 * (t & 1)) ^ g) << 4;
  } else {
    const int j0 = kq * C::GPW;
    o.x_h0 = stage_off_x() + (j0 * MP + g) * 128 + (((2 * t) ^ g) << 4);
    o.x_h1 = stage_off_x() + (j0 * MP + g) * 128 + (((2 * t + 1) ^ g) << 4);
  }
  o.sc = stage_off_s(ACT, MT) + row * 16 + kq * C::GPW * 2;
  o.xs = (uint32_t)((kq * C::GPW * MP + 2 * t) * 4);
  return o;
}

template <int GPW, int kOff>
__device__ __forceinline__ Packed<GPW> lds_packed_at(uint32_t a) {
  Packed<GPW> r;
  if constexpr (GPW == 4) {
    const uint2 v = lds64<kOff>(a);
    r.w[0] = v.x;
    r.w[1] = v.y;
  } else {
    const uint4 v = lds128<kOff>(a);
    r.w[0] = v.x;
    r.w[1] = v.y;
    r.w[2] = v.z;
    r.w[3] = v.w;
  }
  return r;
}

// This warp's share of one stage: groups kq*GPW .. kq*GPW+GPW-1 for its RT
// row tiles. MMA row i of tile r is weight row 16r + 2i, MMA row i+8 is
// weight row 16r + 2i + 1. sb is the stage's shared address, xsb the group-sum
// table's shared address for the stage's first group. All per-tile, per-group
// and per-row offsets are load immediates.
template <int ACT, int MT, int WIDE>
__device__ __forceinline__ void consume_stage(uint32_t sb, uint32_t xsb,
                                              const LaneOffsets<ACT, MT>& o,
                                              float (&tot)[Cfg<MT, WIDE>::RT][MT][4]) {
  using C = Cfg<MT, WIDE>;
  constexpr int RT = C::RT, GPW = C::GPW, MP = 8 * MT;
  constexpr bool kF16 = (ACT == VQ_F16);
  constexpr bool kF32 = (ACT == VQ_F32);
  constexpr int kBiasOff = kBN * 16;   // biases follow the scales
  static_assert(GPW == 4 || GPW == 8, "K-slices of 4 or 8 groups");
  // codes enter the MMA as (offset + q) except for fp32 activations
  constexpr float kOffset = kF32 ? 0.f : (kF16 ? 1024.f : 128.f);

  Packed<GPW> sc0[RT], sc1[RT], bi0[RT], bi1[RT];
  const uint32_t sa = sb + o.sc;
  static_for<RT>([&](auto rc) {
    constexpr int r = decltype(rc)::value;
    sc0[r] = lds_packed_at<GPW, 256 * r>(sa);
    sc1[r] = lds_packed_at<GPW, 256 * r + 16>(sa);
    bi0[r] = lds_packed_at<GPW, 256 * r + kBiasOff>(sa);
    bi1[r] = lds_packed_at<GPW, 256 * r + kBiasOff + 16>(sa);
  });
  const uint32_t we = sb + o.w_even, wo = sb + o.w_odd;
  const uint32_t xa0 = sb + o.x_h0, xa1 = sb + o.x_h1;

  static_for<GPW>([&](auto jc) {
    constexpr int jj = decltype(jc)::value;
    // codes: 16-byte chunk (2*(j%4) + t/2) of the row, XOR-swizzled by row % 8;
    // tile r is 16 rows (2 KiB) further, groups 4..7 (GPW = 8) in box 1
    constexpr int kBox = (GPW == 8 && jj >= 4) ? kWeightBoxBytes : 0;
    const uint32_t sw = ((uint32_t)((jj & 3) << 5)) ^ o.g3x32;
    const uint32_t ae = we + sw, ao = wo + sw;
    uint2 wa[RT], wb[RT];
    static_for<RT>([&](auto rc) {
      constexpr int r = decltype(rc)::value;
      wa[r] = lds64<kBox + 2048 * r>(ae);
      wb[r] = lds64<kBox + 2048 * r>(ao);
    });
    float acc[RT][MT][4];

    static_for<2>([&](auto hc) {
      constexpr int h = decltype(hc)::value;
      // B fragments of rows m = 8mt + g for k = 16t + 8h + (0..7):
      // bx[mt][s'][0..1] = (x_{2s'}, x_{2s'+4}), (x_{2s'+1}, x_{2s'+5})
      uint32_t bx[MT][2][2];
      [[maybe_unused]] uint32_t bxm[MT][2][2], bxl[MT][2][2];   // fp32 only: middle / low terms
      static_for<MT>([&](auto mc) {
        constexpr int mt = decltype(mc)::value;
        if constexpr (!kF32) {
          const uint4 v = lds128<(jj * MP + 8 * mt) * 128>(h ? xa1 : xa0);
          bx[mt][0][0] = prmt(v.x, v.z, 0x5410u);
          bx[mt][0][1] = prmt(v.x, v.z, 0x7632u);
          bx[mt][1][0] = prmt(v.y, v.w, 0x5410u);
          bx[mt][1][1] = prmt(v.y, v.w, 0x7632u);
        } else {
          // chunks 4(t&1) + 2h and that + 1 of line (half-group, row): x_h0
          // holds the line, x_h1 the swizzled chunk (4(t&1) ^ g) << 4
          const uint32_t c0 = xa0 + (o.x_h1 ^ (32u * h));
          const uint4 u0 = lds128<(2 * jj * MP + 8 * mt) * 128>(c0);
          const uint4 u1 = lds128<(2 * jj * MP + 8 * mt) * 128>(xa0 + ((o.x_h1 ^ (32u * h)) ^ 16u));
          split3(__uint_as_float(u0.x), __uint_as_float(u1.x), bx[mt][0][0], bxm[mt][0][0], bxl[mt][0][0]);
          split3(__uint_as_float(u0.y), __uint_as_float(u1.y), bx[mt][0][1], bxm[mt][0][1], bxl[mt][0][1]);
          split3(__uint_as_float(u0.z), __uint_as_float(u1.z), bx[mt][1][0], bxm[mt][1][0], bxl[mt][1][0]);
          split3(__uint_as_float(u0.w), __uint_as_float(u1.w), bx[mt][1][1], bxm[mt][1][1], bxl[mt][1][1]);
        }
      });
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        const bool first = (h == 0 && s2 == 0);
#pragma unroll
        for (int r = 0; r < RT; ++r) {
          const uint32_t qa = h ? wa[r].y : wa[r].x;
          const uint32_t qb = h ? wb[r].y : wb[r].x;
          uint32_t a[4];
          a[0] = code_pair<kF16, kF32>(qa, 2 * s2);
          a[1] = code_pair<kF16, kF32>(qb, 2 * s2);
          a[2] = code_pair<kF16, kF32>(qa, 2 * s2 + 1);
          a[3] = code_pair<kF16, kF32>(qb, 2 * s2 + 1);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            if (first)
              mma_16816_zc<kF16>(acc[r][mt], a, bx[mt][s2][0], bx[mt][s2][1]);
            else
              mma_16816<kF16>(acc[r][mt], a, bx[mt][s2][0], bx[mt][s2][1]);
            if constexpr (kF32) {
              mma_16816<false>(acc[r][mt], a, bxm[mt][s2][0], bxm[mt][s2][1]);
              mma_16816<false>(acc[r][mt], a, bxl[mt][s2][0], bxl[mt][s2][1]);
            }
          }
        }
      }
    });

    // fold group jj: scale the code sums; the bias term (less the code
    // offset) multiplies the group sum of x, rows 8mt+2t and 8mt+2t+1
    float2 xs[MT];
    static_for<MT>([&](auto mc) {
      constexpr int mt = decltype(mc)::value;
      const uint2 v = lds64<(jj * MP + 8 * mt) * 4>(xsb);
      xs[mt] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
    });
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      const float s_a = bf16_of(sc0[r], jj), s_b = bf16_of(sc1[r], jj);
      const float c_a = fmaf(-kOffset, s_a, bf16_of(bi0[r], jj));
      const float c_b = fmaf(-kOffset, s_b, bf16_of(bi1[r], jj));
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        // tot = s*acc + (c*xs + tot), two lanes per instruction
        fma2(tot[r][mt][0], tot[r][mt][1], c_a, c_a, xs[mt].x, xs[mt].y);
        fma2(tot[r][mt][0], tot[r][mt][1], s_a, s_a, acc[r][mt][0], acc[r][mt][1]);
        fma2(tot[r][mt][2], tot[r][mt][3], c_b, c_b, xs[mt].x, xs[mt].y);
        fma2(tot[r][mt][2], tot[r][mt][3], s_b, s_b, acc[r][mt][2], acc[r][mt][3]);
      }
    }
  });
}

// The block's table of group sums X_g[m] = sum of x[m][64g .. 64g+63] for all
// K/64 groups, laid out [K/64][8*MT] (rows m >= M are 0). Every 16-byte chunk
// of x is read once, eight loads in flight per thread; the chunks of one
// group are summed across lanes.
template <int ACT>
__device__ __forceinline__ float chunk_sum(const uint4& v) {
  if constexpr (ACT == VQ_F32) {
    return (__uint_as_float(v.x) + __uint_as_float(v.y)) +
           (__uint_as_float(v.z) + __uint_as_float(v.w));
  } else {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float a[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if constexpr (ACT == VQ_F16) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
        a[e] = f.x + f.y;
      } else {
        a[e] = __uint_as_float(w[e] << 16) + __uint_as_float(w[e] & 0xFFFF0000u);
      }
    }
    return (a[0] + a[1]) + (a[2] + a[3]);
  }
}

template <int ACT, int MT>
__device__ __forceinline__ void build_xsum(float* xsum, const GemmParams& p, int warp, int lane,
                                           int n_warps) {
  constexpr int MP = 8 * MT;
  constexpr int CPG = (ACT == VQ_F32) ? 16 : 8;   // 16-byte chunks per group
  constexpr int PPW = 32 / CPG;                   // (group, row) pairs per warp step
  constexpr int kBatch = 8;                       // loads in flight per thread
  const int KG = p.K / 64;
  const int pairs = p.KT * 8 * MP;   // whole stages: groups past K are summed as 0
  const int chunk = lane % CPG;
  const int step = n_warps * PPW;
  const size_t eb = (ACT == VQ_F32) ? 4 : 2;
  for (int base = warp * PPW; base < pairs; base += step * kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int pair = base + b * step + lane / CPG;
      const int gi = pair / MP, m = pair - (pair / MP) * MP;
      v[b] = make_uint4(0u, 0u, 0u, 0u);
      if (pair < pairs && m < p.M && gi < KG)
        v[b] = __ldg(reinterpret_cast<const uint4*>(
            static_cast<const uint8_t*>(p.x) + ((size_t)m * p.K + (size_t)gi * 64) * eb +
            chunk * 16));
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int pair = base + b * step + lane / CPG;
      float s = chunk_sum<ACT>(v[b]);
#pragma unroll
      for (int off = CPG / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (chunk == 0 && pair < pairs) xsum[pair] = s;
    }
  }
}

// ---------------------------------------------------------------- x table
// For 16-bit x and M <= 8 the block converts x once, while its first stages
// are in flight, into an fp16 table laid out as MMA B fragments:
//   line (group gi, row m) = 128 bytes = 8 chunks; chunk c (holding k =
//   64gi + 8c .. +7) sits at position c ^ m and stores the fp16 pairs
//   (x'0,x'4) (x'1,x'5) (x'2,x'6) (x'3,x'7), where x'_i = x_i * f_m * phi_i,
//   phi_i = 1 for even i and 1/16 for odd i, and f_m = 2^(13 - floor(log2
//   max|x_m|)) so that every |x'| < 2^14 (no fp16 overflow, whatever the
//   scale of the activations).
// Codes enter the MMA as the exact fp16 values q (even i) and 16q (odd i),
// taken from nibble positions 0-3 and 4-7 of each byte pair (one AND/OR with
// the pattern of 1024.0 and one fp16 subtraction), so each product is q x'
// and the group folds as  tot += s * acc_g + b * T_g,  T_g = f_m * sum_g x,
// with y = tot / f_m at the end.
struct XTab {
  uint32_t lines;   // shared address of the fp16 table
  float* T;         // [K/64][8] group sums f_m * sum x
  float* U;         // [K/64][8] scratch of the table build
  float* inv_f;     // [8]
  uint32_t* rmax;   // [8] float bits of max |x_m|
};

template <int ACT>
__device__ __forceinline__ float x_at(const uint4& v, int i) {
  const uint32_t w = (i >> 1) == 0 ? v.x : (i >> 1) == 1 ? v.y : (i >> 1) == 2 ? v.z : v.w;
  if constexpr (ACT == VQ_F16) {
    const __half2 h = *reinterpret_cast<const __half2*>(&w);
    return (i & 1) ? __high2float(h) : __low2float(h);
  } else {
    return __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
}

__device__ __forceinline__ float row_scale(uint32_t rmax_bits) {
  // 2^(13 - floor(log2 max)); 1 for an all-zero row
  if (rmax_bits == 0u) return 1.f;
  const int e = (int)(rmax_bits >> 23);
  const int fe = 267 - e;   // biased exponent of the scale
  return __uint_as_float((uint32_t)(fe > 254 ? 254 : fe) << 23);
}

template <int ACT>
__device__ __forceinline__ void build_xtab(uint8_t* tab_gen, const XTab& X, const GemmParams& p,
                                           int tid, int n_threads, uint32_t bar_threads) {
  // x is already in place (raw 16-bit values, lines swizzled) from the TMA
  const int KG = p.K / 64;
  const int chunks = KG * 64;   // 8 rows x 8 chunks per group
  // pass A: per-(group,row) even / odd sums and the row maxima
  for (int base = tid; base - tid < chunks; base += n_threads) {
    const int ci = base;
    const int m = (ci >> 3) & 7, gi = ci >> 6, c = ci & 7;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (ci < chunks) v = *reinterpret_cast<const uint4*>(tab_gen + (gi * 8 + m) * 128 + ((c ^ m) << 4));
    float se = 0.f, so = 0.f, mx = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float xv = x_at<ACT>(v, i);
      if (i & 1) so += xv; else se += xv;
      mx = fmaxf(mx, fabsf(xv));
    }
    // the 8 chunks of a (group, row) line are 8 consecutive lanes
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) {
      se += __shfl_xor_sync(0xffffffffu, se, off);
      so += __shfl_xor_sync(0xffffffffu, so, off);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    }
    if (ci < chunks && c == 0) {
      X.T[gi * 8 + m] = se;
      X.U[gi * 8 + m] = so;
      atomicMax(X.rmax + m, __float_as_uint(mx));
    }
  }
  named_bar_sync(1, bar_threads);
  // pass B: scale and convert in place; turn the sums into T
  for (int ci = tid; ci < chunks; ci += n_threads) {
    const int m = (ci >> 3) & 7, gi = ci >> 6, c = ci & 7;
    const float f = row_scale(X.rmax[m]);
    uint4* ptr = reinterpret_cast<uint4*>(tab_gen + (gi * 8 + m) * 128 + ((c ^ m) << 4));
    const uint4 v = *ptr;
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float ph = (i & 1) ? 0.0625f : 1.f;
      const __half2 hp = __floats2half2_rn(x_at<ACT>(v, i) * f * ph, x_at<ACT>(v, i + 4) * f * ph);
      o[i] = *reinterpret_cast<const uint32_t*>(&hp);
    }
    *ptr = make_uint4(o[0], o[1], o[2], o[3]);
    if (c == 0) {
      const float se = X.T[gi * 8 + m], so = X.U[gi * 8 + m];
      X.T[gi * 8 + m] = f * (se + so);
    }
  }
  if (tid < 8) X.inv_f[tid] = 1.f / row_scale(X.rmax[tid]);
  named_bar_sync(1, bar_threads);
}

// Per-thread constants of the x-table consumer.
struct XtLane {
  uint32_t w_even, w_odd;   // codes of the even / odd weight row of tile 0
  uint32_t g3x32;           // (g % 4) * 32
  uint32_t x_h0, x_h1;      // table chunk (group 0 of the slice, row g) for h = 0, 1
  uint32_t sc;              // scales of the even row of tile 0 for the slice
  uint32_t ts;              // byte offset of (first group of the slice, row 2t) in T / U
};

template <int MT>
__device__ __forceinline__ XtLane xt_lane(uint32_t lines, int rw, int kq, int g, int t) {
  using C = Cfg<MT>;
  XtLane o;
  const int row = 16 * (C::RT * rw) + 2 * g;
  const int box = (C::GPW == 4) ? kq * kWeightBoxBytes : 0;
  o.w_even = box + row * 128 + ((t >> 1) << 4) + ((t & 1) << 3);
  o.w_odd = box + (row + 1) * 128 + (((t >> 1) ^ 1) << 4) + ((t & 1) << 3);
  o.g3x32 = (uint32_t)(g & 3) << 5;
  const int j0 = kq * C::GPW;
  o.x_h0 = lines + (j0 * 8 + g) * 128 + (((2 * t) ^ g) << 4);
  o.x_h1 = lines + (j0 * 8 + g) * 128 + (((2 * t + 1) ^ g) << 4);
  o.sc = xt_stage_off_s() + row * 16 + kq * C::GPW * 2;
  o.ts = (uint32_t)((j0 * 8 + 2 * t) * 4);
  return o;
}

// Nibbles of a word under `mask` (bits 0-3 or 4-7 of each 16-bit half) as an
// exact fp16 pair: q, or 16q for the upper nibble position.
__device__ __forceinline__ uint32_t xt_code(uint32_t w, uint32_t mask) {
  constexpr uint32_t kMagic = 0x64006400u;   // fp16 1024.0 in both halves
  const uint32_t v = lop3_and_or(w, mask, kMagic);
  const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&v),
                            *reinterpret_cast<const __half2*>(&kMagic));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// One stage of the x-table variant (MT = 1): groups kq*GPW .. +GPW-1 of
// stage kt for the warp's RT row tiles.
template <int ACT>
__device__ __forceinline__ void consume_stage_xt(uint32_t sb, int kt, uint32_t T_a,
                                                 const XtLane& o,
                                                 float (&tot)[Cfg<1>::RT][1][4]) {
  using C = Cfg<1>;
  constexpr int RT = C::RT, GPW = C::GPW;
  constexpr int kBiasOff = kBN * 16;
  static_assert(GPW == 4 || GPW == 8, "K-slices of 4 or 8 groups");

  Packed<GPW> sc0[RT], sc1[RT], bi0[RT], bi1[RT];
  const uint32_t sa = sb + o.sc;
  static_for<RT>([&](auto rc) {
    constexpr int r = decltype(rc)::value;
    sc0[r] = lds_packed_at<GPW, 256 * r>(sa);
    sc1[r] = lds_packed_at<GPW, 256 * r + 16>(sa);
    bi0[r] = lds_packed_at<GPW, 256 * r + kBiasOff>(sa);
    bi1[r] = lds_packed_at<GPW, 256 * r + kBiasOff + 16>(sa);
  });
  const uint32_t we = sb + o.w_even, wo = sb + o.w_odd;
  const uint32_t xg = (uint32_t)kt * 8 * 1024;   // the stage's first group in the x table
  const uint32_t xa0 = o.x_h0 + xg, xa1 = o.x_h1 + xg;
  const uint32_t ta = T_a + (uint32_t)kt * 8 * 32;

  static_for<GPW>([&](auto jc) {
    constexpr int jj = decltype(jc)::value;
    constexpr int kBox = (GPW == 8 && jj >= 4) ? kWeightBoxBytes : 0;
    const uint32_t sw = ((uint32_t)((jj & 3) << 5)) ^ o.g3x32;
    const uint32_t ae = we + sw, ao = wo + sw;
    uint2 wa[RT], wb[RT];
    static_for<RT>([&](auto rc) {
      constexpr int r = decltype(rc)::value;
      wa[r] = lds64<kBox + 2048 * r>(ae);
      wb[r] = lds64<kBox + 2048 * r>(ao);
    });
    float acc[RT][4];
    static_for<2>([&](auto hc) {
      constexpr int h = decltype(hc)::value;
      const uint4 bx = lds128<jj * 1024>(h ? xa1 : xa0);
#pragma unroll
      for (int r = 0; r < RT; ++r) {
        const uint32_t qa = h ? wa[r].y : wa[r].x;
        const uint32_t qb = h ? wb[r].y : wb[r].x;
        const uint32_t qa8 = qa >> 8, qb8 = qb >> 8;
        // step s' = 0: pairs (c0,c4) and (c1,c5); s' = 1: (c2,c6) and (c3,c7);
        // made exact (q or 16q) by one fp16 subtraction on the FMA pipe
        const uint32_t a0[4] = {xt_code(qa, 0x000F000Fu), xt_code(qb, 0x000F000Fu),
                                xt_code(qa, 0x00F000F0u), xt_code(qb, 0x00F000F0u)};
        const uint32_t a1[4] = {xt_code(qa8, 0x000F000Fu), xt_code(qb8, 0x000F000Fu),
                                xt_code(qa8, 0x00F000F0u), xt_code(qb8, 0x00F000F0u)};
        float (&d)[4] = acc[r];
        if (h == 0)
          mma_16816_zc<true>(d, a0, bx.x, bx.y);
        else
          mma_16816<true>(d, a0, bx.x, bx.y);
        mma_16816<true>(d, a1, bx.z, bx.w);
      }
    });
    // fold: tot += s * acc + b * T, rows 2t and 2t+1 of the block
    const uint2 tv = lds64<jj * 32>(ta);
    const float T0 = __uint_as_float(tv.x), T1 = __uint_as_float(tv.y);
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      const float s_a = bf16_of(sc0[r], jj), s_b = bf16_of(sc1[r], jj);
      const float b_a = bf16_of(bi0[r], jj), b_b = bf16_of(bi1[r], jj);
      fma2(tot[r][0][0], tot[r][0][1], b_a, b_a, T0, T1);
      fma2(tot[r][0][0], tot[r][0][1], s_a, s_a, acc[r][0], acc[r][1]);
      fma2(tot[r][0][2], tot[r][0][3], b_b, b_b, T0, T1);
      fma2(tot[r][0][2], tot[r][0][3], s_b, s_b, acc[r][2], acc[r][3]);
    }
  });
}

// The x slice of stage kt, row m, written by one warp: it reads the row's 512
// values, picks the power-of-two scale f that brings their largest magnitude
// into [2^13, 2^14) (no fp16 overflow whatever the activations' scale), and
// writes the scaled fp16 fragments (odd nibble positions also divided by 16),
// the f-scaled group sums T, -U and 1/f. Each slice is prepared once per call.
template <int ACT>
__device__ __forceinline__ void prep_slice_row(const void* __restrict__ x, int M, int K, int kt,
                                               int xm_row, int lane, uint8_t* __restrict__ slice) {
  const int m = xm_row & 7;   // the row within the slice
  uint4 v[2];
  float mx = 0.f, gs[2];
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const int ci = lane + 32 * b;   // chunk of 8 values: group ci/8, position ci%8
    v[b] = make_uint4(0u, 0u, 0u, 0u);
    if (xm_row < M)
      v[b] = __ldg(reinterpret_cast<const uint4*>(
          static_cast<const uint8_t*>(x) + ((size_t)xm_row * K + (size_t)kt * kBK + ci * 8) * 2));
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float xv = x_at<ACT>(v[b], i);
      s += xv;
      mx = fmaxf(mx, fabsf(xv));
    }
    gs[b] = s;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  const float f = row_scale(__float_as_uint(mx));
  float* T = reinterpret_cast<float*>(slice + kSliceT);
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const int ci = lane + 32 * b, j = ci >> 3, c = ci & 7;
    uint32_t o4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float ph = (i & 1) ? 0.0625f : 1.f;
      const __half2 hp =
          __floats2half2_rn(x_at<ACT>(v[b], i) * f * ph, x_at<ACT>(v[b], i + 4) * f * ph);
      o4[i] = *reinterpret_cast<const uint32_t*>(&hp);
    }
    *reinterpret_cast<uint4*>(slice + (j * 8 + m) * 128 + ((c ^ m) << 4)) =
        make_uint4(o4[0], o4[1], o4[2], o4[3]);
    // the fp16 values exactly as the MMA will see them
    float u = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&o4[i]));
      u += h.x + h.y;
    }
    float s = gs[b];
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) {
      s += __shfl_xor_sync(0xffffffffu, s, off);
      u += __shfl_xor_sync(0xffffffffu, u, off);
    }
    if (c == 0) {
      T[j * 8 + m] = f * s;
      float* nu = reinterpret_cast<float*>(slice + kSliceU) + j * 16 + (m >> 1) * 4 + (m & 1);
      nu[0] = -1024.f * u;
      nu[2] = -1024.f * u;
    }
  }
  if (lane == 0) reinterpret_cast<float*>(slice + kSliceInv)[m] = 1.f / f;
}

// The slices of one call, [KT stages][MT tiles]: block b prepares stage
// b / MT, tile b % MT, one row per warp. It is launched so that it may start
// while the kernel before it in the stream is finishing, and waits for that
// kernel before it reads x or overwrites the slices; the projection after it
// waits for it in the same way.
constexpr int kPrepThreads = 256;   // 8 warps: the 8 rows of a tile

template <int ACT>
__global__ void __launch_bounds__(kPrepThreads)
    vq_prep_kernel(const void* __restrict__ x, int M, int K, int MT, uint8_t* __restrict__ out) {
  grid_launch_dependents();
  grid_wait_prerequisites();
  const int kt = blockIdx.x / MT, mt = blockIdx.x - (blockIdx.x / MT) * MT;
  prep_slice_row<ACT>(x, M, K, kt, 8 * mt + (threadIdx.x >> 5), threadIdx.x & 31,
                      out + (size_t)blockIdx.x * kSliceBytes);
}

// Per-thread constants of the prepared-slice consumer (offsets in a stage).
struct XsLane {
  uint32_t w_even, w_odd;   // codes of the even / odd weight row of tile 0
  uint32_t g3x32;           // (g % 4) * 32
  uint32_t x_h0, x_h1;      // slice chunk of row g, first group of the K-slice, h = 0, 1
  uint32_t sc;              // scales of the even row of tile 0 for the K-slice
  uint32_t ts;              // T of (first group of the K-slice, row 2t)
  uint32_t nu;              // -U quad of (first group of the K-slice, thread t)
  uint32_t inv;             // 1/f of rows 2t, 2t+1
};

template <int MT, int WIDE>
__device__ __forceinline__ XsLane xs_lane(int rw, int kq, int g, int t) {
  using C = Cfg<MT, WIDE>;
  XsLane o;
  const int row = 16 * (C::RT * rw) + 2 * g;
  const int box = (C::GPW == 4) ? kq * kWeightBoxBytes : 0;
  o.w_even = box + row * 128 + ((t >> 1) << 4) + ((t & 1) << 3);
  o.w_odd = box + (row + 1) * 128 + (((t >> 1) ^ 1) << 4) + ((t & 1) << 3);
  o.g3x32 = (uint32_t)(g & 3) << 5;
  const int j0 = kq * C::GPW;
  o.x_h0 = xs_stage_off_x() + (j0 * 8 + g) * 128 + (((2 * t) ^ g) << 4);
  o.x_h1 = xs_stage_off_x() + (j0 * 8 + g) * 128 + (((2 * t + 1) ^ g) << 4);
  o.sc = xt_stage_off_s() + row * 16 + kq * C::GPW * 2;
  o.ts = xs_stage_off_x() + kSliceT + (j0 * 8 + 2 * t) * 4;
  o.nu = xs_stage_off_x() + kSliceU + (j0 * 4 + t) * 16;
  o.inv = xs_stage_off_x() + kSliceInv + 2 * t * 4;
  return o;
}

// One stage of the prepared-slice variant (MT n8 tiles, one slice each):
// the warp's K-slice of groups for its RT row tiles, folded in each slice's
// scaled units and then brought back with the slice's 1/f. The codes are
// unpacked once per row tile and serve every n8 tile.
template <int ACT, int MT, int WIDE>
__device__ __forceinline__ void consume_stage_xs(uint32_t sb, const XsLane& o,
                                                 float (&tot)[Cfg<MT, WIDE>::RT][MT][4]) {
  using C = Cfg<MT, WIDE>;
  constexpr int RT = C::RT, GPW = C::GPW;
  constexpr int kBiasOff = kBN * 16;
  constexpr uint32_t kMagic16 = 0x64006400u;   // fp16 1024.0 in both halves
  static_assert(GPW == 4 || GPW == 8, "K-slices of 4 or 8 groups");
  static_assert(MT == 1 || MT == 2, "one or two n8 tiles");

  Packed<GPW> sc0[RT], sc1[RT], bi0[RT], bi1[RT];
  const uint32_t sa = sb + o.sc;
  static_for<RT>([&](auto rc) {
    constexpr int r = decltype(rc)::value;
    sc0[r] = lds_packed_at<GPW, 256 * r>(sa);
    sc1[r] = lds_packed_at<GPW, 256 * r + 16>(sa);
    bi0[r] = lds_packed_at<GPW, 256 * r + kBiasOff>(sa);
    bi1[r] = lds_packed_at<GPW, 256 * r + kBiasOff + 16>(sa);
  });
  const uint32_t we = sb + o.w_even, wo = sb + o.w_odd;
  const uint32_t xa0 = sb + o.x_h0, xa1 = sb + o.x_h1;
  const uint32_t ta = sb + o.ts;
  float part[RT][MT][4];
#pragma unroll
  for (int r = 0; r < RT; ++r)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) part[r][mt][0] = part[r][mt][1] = part[r][mt][2] = part[r][mt][3] = 0.f;

  static_for<GPW>([&](auto jc) {
    constexpr int jj = decltype(jc)::value;
    constexpr int kBox = (GPW == 8 && jj >= 4) ? kWeightBoxBytes : 0;
    const uint32_t sw = ((uint32_t)((jj & 3) << 5)) ^ o.g3x32;
    const uint32_t ae = we + sw, ao = wo + sw;
    uint2 wa[RT], wb[RT];
    static_for<RT>([&](auto rc) {
      constexpr int r = decltype(rc)::value;
      wa[r] = lds64<kBox + 2048 * r>(ae);
      wb[r] = lds64<kBox + 2048 * r>(ao);
    });
    float4 nu[MT];
    static_for<MT>([&](auto mc) {
      constexpr int mt = decltype(mc)::value;
      const uint4 nuv = lds128<jj * 64 + mt * kSliceBytes>(sb + o.nu);
      nu[mt] = make_float4(__uint_as_float(nuv.x), __uint_as_float(nuv.y), __uint_as_float(nuv.z),
                           __uint_as_float(nuv.w));
    });
    float acc[RT][MT][4];
    static_for<2>([&](auto hc) {
      constexpr int h = decltype(hc)::value;
      uint4 bx[MT];
      static_for<MT>([&](auto mc) {
        constexpr int mt = decltype(mc)::value;
        bx[mt] = lds128<jj * 1024 + mt * kSliceBytes>(h ? xa1 : xa0);
      });
#pragma unroll
      for (int r = 0; r < RT; ++r) {
        const uint32_t qa = h ? wa[r].y : wa[r].x;
        const uint32_t qb = h ? wb[r].y : wb[r].x;
        const uint32_t qa8 = qa >> 8, qb8 = qb >> 8;
        // codes as fp16 1024 + q (or 1024 + 16q): one AND/OR each; the
        // accumulator starts at -U, which cancels the 1024s
        const uint32_t a0[4] = {lop3_and_or(qa, 0x000F000Fu, kMagic16), lop3_and_or(qb, 0x000F000Fu, kMagic16),
                                lop3_and_or(qa, 0x00F000F0u, kMagic16), lop3_and_or(qb, 0x00F000F0u, kMagic16)};
        const uint32_t a1[4] = {lop3_and_or(qa8, 0x000F000Fu, kMagic16), lop3_and_or(qb8, 0x000F000Fu, kMagic16),
                                lop3_and_or(qa8, 0x00F000F0u, kMagic16), lop3_and_or(qb8, 0x00F000F0u, kMagic16)};
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          float (&d)[4] = acc[r][mt];
          if (h == 0)
            mma_16816_c<true>(d, a0, bx[mt].x, bx[mt].y, nu[mt]);
          else
            mma_16816<true>(d, a0, bx[mt].x, bx[mt].y);
          mma_16816<true>(d, a1, bx[mt].z, bx[mt].w);
        }
      }
    });
    static_for<MT>([&](auto mc) {
      constexpr int mt = decltype(mc)::value;
      const uint2 tv = lds64<jj * 32 + mt * kSliceBytes>(ta);
      const float T0 = __uint_as_float(tv.x), T1 = __uint_as_float(tv.y);
#pragma unroll
      for (int r = 0; r < RT; ++r) {
        const float s_a = bf16_of(sc0[r], jj), s_b = bf16_of(sc1[r], jj);
        const float b_a = bf16_of(bi0[r], jj), b_b = bf16_of(bi1[r], jj);
        fma2(part[r][mt][0], part[r][mt][1], b_a, b_a, T0, T1);
        fma2(part[r][mt][0], part[r][mt][1], s_a, s_a, acc[r][mt][0], acc[r][mt][1]);
        fma2(part[r][mt][2], part[r][mt][3], b_b, b_b, T0, T1);
        fma2(part[r][mt][2], part[r][mt][3], s_b, s_b, acc[r][mt][2], acc[r][mt][3]);
      }
    });
  });
  static_for<MT>([&](auto mc) {
    constexpr int mt = decltype(mc)::value;
    const uint2 iv = lds64<mt * kSliceBytes>(sb + o.inv);
    const float i0 = __uint_as_float(iv.x), i1 = __uint_as_float(iv.y);
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      fma2(tot[r][mt][0], tot[r][mt][1], i0, i1, part[r][mt][0], part[r][mt][1]);
      fma2(tot[r][mt][2], tot[r][mt][3], i0, i1, part[r][mt][2], part[r][mt][3]);
    }
  });
}

template <int ACT, int MT, bool ARGMAX, int XM, int WIDE = 0>
__global__ void __launch_bounds__(Cfg<MT, WIDE>::THREADS, 1)
    vq_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s,
                   const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_x,
                   const GemmParams p) {
  using C = Cfg<MT, WIDE>;
  constexpr int MP = 8 * MT;
  constexpr int RT = C::RT, KQ = C::KQ, RW = C::RW, TEAMS = C::TEAMS, SLICES = C::SLICES;
  constexpr bool XT = (XM == 1);   // x table built in the block
  constexpr bool XS = (XM == 2);   // prepared x slices in the stages
  constexpr int kConsumers = C::WARPS;
  constexpr int kProducerWarp = kConsumers;
  constexpr int kXBoxes = (ACT == VQ_F32) ? 16 : 8;   // per-group boxes (x3d == 0)
  constexpr int kXBoxElems = kBK / kXBoxes;
  constexpr uint32_t kEpiThreads = RW * 32;            // the K-slice-0 consumers

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - raw);
  // [D stages][tables: x table (x-table variant) or group sums][misc][K-slice partials]
  uint8_t* const tabs = sbase + p.D * p.stage_bytes;
  uint8_t* const misc = tabs + p.tab_bytes;
  const uint32_t misc_a = base + p.D * p.stage_bytes + p.tab_bytes;
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(misc + 264);
  volatile int* const epi_flag = reinterpret_cast<volatile int*>(misc + 268);
  // set once the consumers' griddepcontrol.wait has returned
  volatile int* const dep_flag = reinterpret_cast<volatile int*>(misc + 272);
  float* const red_v = reinterpret_cast<float*>(misc + kBarBytes);
  uint32_t* const red_i = reinterpret_cast<uint32_t*>(misc + kBarBytes + 8 * 64 * 4);
  float* const red_s = reinterpret_cast<float*>(misc + kBarBytes + 2 * 8 * 64 * 4);
  float* const red_k = p.red_alias ? reinterpret_cast<float*>(sbase)   // [SLICES-1][128][MP]
                                   : reinterpret_cast<float*>(misc + misc_bytes(ARGMAX));
  float* const xsum = reinterpret_cast<float*>(tabs);   // [K/64][MP]
  const int KG = p.K / 64;
  XTab X;
  X.lines = smem_addr(tabs);
  X.T = reinterpret_cast<float*>(tabs + KG * 1024);
  X.inv_f = X.T + KG * 8;
  X.U = X.inv_f + 8;
  X.rmax = reinterpret_cast<uint32_t*>(X.U + KG * 8);
  auto full_bar = [&](int s) { return misc_a + 8u * s; };
  auto empty_bar = [&](int s) { return misc_a + 64u + 8u * s; };
  // scales and biases loaded by the producer lanes landed (sb_plain)
  auto sbfull_bar = [&](int s) { return misc_a + 136u + 8u * s; };
  const bool sbp = (XM == 0) && p.sb_plain;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the next kernel in the stream may be scheduled as soon as SMs free up
  grid_launch_dependents();
  const uint32_t x_bar = misc_a + 128u;   // x table landed (x-table variant)
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.D; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), C::WPT);   // one team consumes each stage
      if (sbp) mbar_init(sbfull_bar(s), 32);   // every producer lane
    }
    mbar_init(x_bar, 1);
    *abort_flag = 0;
    *dep_flag = 0;
    if constexpr (XT) {
      for (int i = 0; i < 8; ++i) X.rmax[i] = 0u;
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // lane 0 issues the TMA copies; with sb_plain all 32 lanes also load the
    // stage's scales and biases (weights too: they may be read before the wait)
    if (lane == 0 || sbp) {
      if (lane == 0) {
        prefetch_tensormap(&tm_w);
        if (!sbp) {
          prefetch_tensormap(&tm_s);
          prefetch_tensormap(&tm_b);
        }
        if (!XS) prefetch_tensormap(&tm_x);   // prepared slices: x is not read by TMA
      }
      // Weights are constants of the model: the first stages' weights are
      // requested before waiting for the kernel before this one in the stream
      // (programmatic dependent launch), so the weight stream overlaps that
      // kernel's tail. x, which that kernel may write, is requested only after
      // the wait.
      const uint64_t w_policy = l2_evict_first_policy();
      auto load_sb = [&](int slot, int kt, int rb) {
        uint8_t* const st = sbase + slot * p.stage_bytes;
        load_stage_sb(p, st + p.off_s, st + p.off_b, kt, rb, lane);
        mbar_arrive(sbfull_bar(slot));
      };
      auto issue_w = [&](int slot, int kt, int rb) {
        const uint32_t sb = base + slot * p.stage_bytes;
        const uint32_t fb = full_bar(slot);
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, p.tx_bytes);
          tma_load_2d_hint(sb, &tm_w, kt * (kBK / 8), rb * kBN, fb, w_policy);
          tma_load_2d_hint(sb + kWeightBoxBytes, &tm_w, kt * (kBK / 8) + 32, rb * kBN, fb,
                           w_policy);
          if (!sbp) {
            tma_load_2d_hint(sb + p.off_s, &tm_s, kt * (kBK / 64), rb * kBN, fb, w_policy);
            tma_load_2d_hint(sb + p.off_b, &tm_b, kt * (kBK / 64), rb * kBN, fb, w_policy);
          }
        }
        if (sbp) load_sb(slot, kt, rb);
      };
      auto issue_x = [&](int slot, int kt) {
        if (lane != 0) return;
        const uint32_t sb = base + slot * p.stage_bytes;
        const uint32_t fb = full_bar(slot);
        if constexpr (XS) {
          bulk_load(sb + p.off_x,
                    static_cast<const uint8_t*>(p.xprep) + (size_t)kt * MT * kSliceBytes,
                    MT * kSliceBytes, fb);
        } else if constexpr (XT) {
          // x comes from the block's table
        } else if (p.x3d) {
          tma_load_3d(sb + p.off_x, &tm_x, 0, 0, kt * kXBoxes, fb);
        } else {
#pragma unroll
          for (int j = 0; j < kXBoxes; ++j)
            tma_load_2d(sb + p.off_x + j * MP * 128, &tm_x, kt * kBK + j * kXBoxElems, 0, fb);
        }
      };
      int pre = 0;   // stages whose weights were issued before the wait
      int kt_first = 0;
      if (blockIdx.x < p.n_units) {
        const int u0 = blockIdx.x;
        const int rb = u0 / p.S, sp = u0 - rb * p.S;
        const int kt0 = sp * p.KT / p.S, kt1 = (sp + 1) * p.KT / p.S;
        kt_first = kt0;
        // The requests are spaced while the kernel before this one runs: the
        // memory system then holds a short queue of weight requests rather
        // than megabytes of them, and the small reads that come right after
        // the wait (that kernel's successor reading x, this kernel's slices)
        // are not stuck behind it. The spacing stops once the consumers have
        // seen the wait return, so a call with nothing before it is not slowed.
        const long long t_pace = clock64();
        for (int r = 0; r < p.pre && r < p.D && kt0 + r < kt1; ++r) {
          if (r > 0)
            while (!*dep_flag && clock64() - t_pace < (long long)r * p.pace) {
            }
          issue_w(r, kt0 + r, rb);
          ++pre;
        }
      }
      grid_wait_prerequisites();
      bool ok = true;
      if (XT && lane == 0) {
        // the block's x, all K/64 groups of 8 rows, first of all
        mbar_arrive_expect_tx(x_bar, (uint32_t)KG * 1024u);
        if (p.x3d) {
          tma_load_3d(X.lines, &tm_x, 0, 0, 0, x_bar);
        } else {
          for (int gi = 0; gi < KG; ++gi) tma_load_2d(X.lines + gi * 1024, &tm_x, gi * 64, 0, x_bar);
        }
      }
      int q = 0;
      for (int r = 0; r < pre; ++r) issue_x(r, kt_first + r);
      for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
        const int rb = u / p.S, sp = u - rb * p.S;
        const int kt0 = sp * p.KT / p.S, kt1 = (sp + 1) * p.KT / p.S;
        for (int kt = kt0; kt < kt1; ++kt) {
          if (pre > 0) {   // weights issued before the wait, x just after it
            --pre;
            ++q;
            continue;
          }
          const int slot = q % p.D;
          const uint32_t ph = (uint32_t)(q / p.D) & 1u;
          if (!wait_or_abort(empty_bar(slot), ph ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          issue_w(slot, kt, rb);
          issue_x(slot, kt);
          ++q;
        }
      }
      if (!ok && lane == 0) {
        // let the copies already issued land before the block can exit
        for (int r = (q > p.D ? q - p.D : 0); r < q; ++r)
          wait_bounded(full_bar(r % p.D), (uint32_t)(r / p.D) & 1u, p.err);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  const int team = warp / C::WPT, wt = warp - (warp / C::WPT) * C::WPT;
  const int rw = wt % RW, kq = wt / RW;
  const int slice = team * KQ + kq;   // which partial sum of its rows this warp holds
  float best_v[MT][2];
  uint32_t best_n[MT][2];
  bool best_has[MT][2];
  float best_s[MT][2];   // runner-up value (-inf: none yet)
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      best_v[mt][c] = 0.f;
      best_n[mt][c] = 0u;
      best_has[mt][c] = false;
      best_s[mt][c] = -INFINITY;
    }

  bool aborted = false;
  // x and every output may belong to the kernel before this one in the stream
  grid_wait_prerequisites();
  if (threadIdx.x == 0) *dep_flag = 1;
  // group sums of x (or the whole x table) for all of K, while the first
  // stages are in flight
  LaneOffsets<ACT, MT> lo;
  XtLane xl;
  uint32_t xsum_a = 0, T_a = 0;
  XsLane xsl;
  if constexpr (XS) {
    xsl = xs_lane<MT, WIDE>(rw, kq, g, t);
  } else if constexpr (XT) {
    if (!wait_or_abort(x_bar, 0u, abort_flag, p.err)) aborted = true;
    build_xtab<ACT>(tabs, X, p, threadIdx.x, kConsumers * 32, kConsumers * 32);
    xl = xt_lane<MT>(X.lines, rw, kq, g, t);
    T_a = smem_addr(X.T) + xl.ts;
  } else {
    build_xsum<ACT, MT>(xsum, p, warp, lane, kConsumers);
    named_bar_sync(1, kConsumers * 32);
    lo = lane_offsets<ACT, MT, WIDE>(rw, kq, g, t);
    xsum_a = smem_addr(xsum) + lo.xs;
  }

  // stage counter q, and (slot, phase) of this team's next stage, advanced
  // incrementally (no division in the loop)
  int q = 0;
  int slot = team, phase = 0;
  while (slot >= p.D) {
    slot -= p.D;
    phase ^= 1;
  }
  for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
    const int rb = u / p.S, sp = u - rb * p.S;
    const int kt0 = sp * p.KT / p.S, kt1 = (sp + 1) * p.KT / p.S;
    float tot[RT][MT][4];
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) tot[r][mt][0] = tot[r][mt][1] = tot[r][mt][2] = tot[r][mt][3] = 0.f;

    for (int kt = kt0; kt < kt1; ++kt, ++q) {
      if (TEAMS > 1 && (q & (TEAMS - 1)) != team) continue;   // the other team's stage
      const uint32_t ph = (uint32_t)phase;
      bool ok = !aborted && wait_or_abort(full_bar(slot), ph, abort_flag, p.err);
      if (sbp) ok = ok && wait_or_abort(sbfull_bar(slot), ph, abort_flag, p.err);
      if (ok) {
        if constexpr (XS)
          consume_stage_xs<ACT, MT, WIDE>(base + slot * p.stage_bytes, xsl, tot);
        else if constexpr (XT)
          consume_stage_xt<ACT>(base + slot * p.stage_bytes, kt, T_a, xl, tot);
        else
          consume_stage<ACT, MT, WIDE>(base + slot * p.stage_bytes, xsum_a + kt * (8 * MP * 4), lo,
                                       tot);
      } else {
        aborted = true;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(slot));
      slot += TEAMS;
      if (slot >= p.D) {
        slot -= p.D;
        phase ^= 1;
      }
    }

    if constexpr (SLICES > 1) {
      // partials in the stage ring: every team must be done with its stages
      if (p.red_alias) named_bar_sync(1, kConsumers * 32);
      // slices 1.. publish their partial sums, slice 0 adds them in order
      if (slice > 0) {
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int row = 16 * (RT * rw + r) + 2 * g + (e >> 1);
              red_k[((slice - 1) * kBN + row) * MP + 8 * mt + 2 * t + (e & 1)] = tot[r][mt][e];
            }
      }
      named_bar_sync(1, kConsumers * 32);
      if (slice == 0) {
#pragma unroll
        for (int k = 1; k < SLICES; ++k)
#pragma unroll
          for (int r = 0; r < RT; ++r)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int row = 16 * (RT * rw + r) + 2 * g + (e >> 1);
                tot[r][mt][e] += red_k[((k - 1) * kBN + row) * MP + 8 * mt + 2 * t + (e & 1)];
              }
      }
      named_bar_sync(1, kConsumers * 32);
      if (slice > 0) continue;
    }
    if constexpr (XT) {
      // back from the x table's per-row scale f_m to y
#pragma unroll
      for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int e = 0; e < 4; ++e) tot[r][0][e] *= X.inv_f[2 * t + (e & 1)];
    }

    if constexpr (!ARGMAX) {
      // (the WIDE layout is only launched without a K split)
      if (WIDE != 0 || p.S == 1) {
        if (!aborted) {
          // a lane holds columns n, n + 1 of rows m: with 16-bit y and an even
          // N they go out as one 4-byte store, so that the eight lanes of a
          // row fill whole 32-byte sectors (this matters when y is host memory)
          const bool pair = ACT != VQ_F32 && (p.N & 1) == 0;
#pragma unroll
          for (int r = 0; r < RT; ++r)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int n = rb * kBN + 16 * (RT * rw + r) + 2 * g;
                const int m = 8 * mt + 2 * t + h;
                if (m >= p.M) continue;
                const size_t i = (size_t)m * p.N + n;
                if (pair && n + 1 < p.N) {
                  if (in_bounds(i + 1, p.y_elems, p.err))
                    store_out2<ACT>(p.y, i, tot[r][mt][h], tot[r][mt][h + 2]);
                } else {
                  if (n < p.N && in_bounds(i, p.y_elems, p.err))
                    store_out<ACT>(p.y, i, tot[r][mt][h]);
                  if (n + 1 < p.N && in_bounds(i + 1, p.y_elems, p.err))
                    store_out<ACT>(p.y, i + 1, tot[r][mt][h + 2]);
                }
              }
        }
      } else {
        // split K: publish this slice, the last slice to arrive reduces all
        // slices in slice order (deterministic) and stores y
        float* part = p.part + (size_t)sp * p.M * p.N;
        if (!aborted) {
#pragma unroll
          for (int r = 0; r < RT; ++r)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int n = rb * kBN + 16 * (RT * rw + r) + 2 * g + (e >> 1);
                const int m = 8 * mt + 2 * t + (e & 1);
                if (n < p.N && m < p.M &&
                    in_bounds((size_t)sp * p.M * p.N + (size_t)m * p.N + n, p.part_elems, p.err))
                  __stcg(part + (size_t)m * p.N + n, tot[r][mt][e]);
              }
        }
        __threadfence();
        named_bar_sync(2, kEpiThreads);
        if (threadIdx.x == 0) *epi_flag = (atomicAdd(p.cnt + rb, 1u) == (uint32_t)(p.S - 1));
        named_bar_sync(2, kEpiThreads);
        if (*epi_flag) {
          __threadfence();
          if (!aborted) {
            // the slices are added in slice order (deterministic). Every load
            // of a round (all elements of the thread, KB slices) is issued
            // before any is used: the addresses of elements outside y and of
            // slices past S are clamped to valid ones and their values
            // dropped, so no load sits behind a branch and the sum costs
            // ceil(S / KB) L2 round trips rather than one per element.
            constexpr int KB = (RT * MT <= 2) ? 4 : 2;
            const size_t slice_stride = (size_t)p.M * p.N;
            float acc[RT][MT][4];
#pragma unroll
            for (int r = 0; r < RT; ++r)
#pragma unroll
              for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[r][mt][e] = 0.f;
            for (int k0 = 0; k0 < p.S; k0 += KB) {
              float v[RT][MT][4][KB];
#pragma unroll
              for (int i = 0; i < KB; ++i) {
                const float* sl = p.part + (size_t)(k0 + i < p.S ? k0 + i : p.S - 1) * slice_stride;
#pragma unroll
                for (int r = 0; r < RT; ++r)
#pragma unroll
                  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                      const int n = rb * kBN + 16 * (RT * rw + r) + 2 * g + (e >> 1);
                      const int m = 8 * mt + 2 * t + (e & 1);
                      const bool in = n < p.N && m < p.M;
                      v[r][mt][e][i] = __ldcg(sl + (in ? (size_t)m * p.N + n : 0));
                    }
              }
#pragma unroll
              for (int i = 0; i < KB; ++i)
                if (k0 + i < p.S) {
#pragma unroll
                  for (int r = 0; r < RT; ++r)
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                      for (int e = 0; e < 4; ++e) acc[r][mt][e] += v[r][mt][e][i];
                }
            }
#pragma unroll
            for (int r = 0; r < RT; ++r)
#pragma unroll
              for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int n = rb * kBN + 16 * (RT * rw + r) + 2 * g + (e >> 1);
                  const int m = 8 * mt + 2 * t + (e & 1);
                  if (n < p.N && m < p.M && in_bounds((size_t)m * p.N + n, p.y_elems, p.err))
                    store_out<ACT>(p.y, (size_t)m * p.N + n, acc[r][mt][e]);
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
      for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int n = rb * kBN + 16 * (RT * rw + r) + 2 * g + (e >> 1), c = e & 1;
            const float v = tot[r][mt][e] + 0.0f;   // -0 -> +0
            if (!aborted && n < p.N && !(v != v)) {
              if (!best_has[mt][c] || v > best_v[mt][c]) {
                if (best_has[mt][c]) best_s[mt][c] = fmaxf(best_s[mt][c], best_v[mt][c]);
                best_v[mt][c] = v;
                best_n[mt][c] = (uint32_t)n;
                best_has[mt][c] = true;
              } else {
                best_s[mt][c] = fmaxf(best_s[mt][c], v);
              }
            }
          }
    }
  }

  if constexpr (ARGMAX) {
    if (slice > 0) return;
    // reduce over the 8 row-lanes g of the warp, then over the row warps
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float v = best_v[mt][c];
        uint32_t n = best_n[mt][c];
        bool h = best_has[mt][c];
        float sv = best_s[mt][c];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, v, off);
          const uint32_t on = __shfl_xor_sync(0xffffffffu, n, off);
          const bool oh = __shfl_xor_sync(0xffffffffu, (int)h, off) != 0;
          const float os = __shfl_xor_sync(0xffffffffu, sv, off);
          top2_merge(v, n, h, sv, ov, on, oh, os);
        }
        if (g == 0) {
          const int m = 8 * mt + 2 * t + c;
          red_v[rw * 64 + m] = v;
          red_i[rw * 64 + m] = h ? n : 0xFFFFFFFFu;
          red_s[rw * 64 + m] = sv;
        }
      }
    named_bar_sync(2, kEpiThreads);
    if (threadIdx.x < MP) {
      const int m = threadIdx.x;
      float v = 0.f, sv = -INFINITY;
      uint32_t n = 0u;
      bool h = false;
      for (int w = 0; w < RW; ++w) {
        const uint32_t on = red_i[w * 64 + m];
        top2_merge(v, n, h, sv, red_v[w * 64 + m], on, on != 0xFFFFFFFFu, red_s[w * 64 + m]);
      }
      if (h && m < p.M && !aborted) {
        const unsigned long long key =
            ((unsigned long long)float_order(v) << 32) | (unsigned long long)(0xFFFFFFFFu - n);
        if (in_bounds((size_t)m, (size_t)p.M, p.err)) atomicMax(p.keys + m, key);
      }
      if (p.cand && m < p.M && in_bounds((size_t)blockIdx.x * p.M + m, p.cand_elems, p.err))
        p.cand[(size_t)blockIdx.x * p.M + m] =
            make_uint4(__float_as_uint(v), (h && !aborted) ? n : 0xFFFFFFFFu,
                       __float_as_uint(sv), 0u);
    }
    __threadfence();
    named_bar_sync(2, kEpiThreads);
    if (threadIdx.x == 0) *epi_flag = (atomicAdd(p.done, 1u) == gridDim.x - 1);
    named_bar_sync(2, kEpiThreads);
    if (*epi_flag) {
      __threadfence();
      if (threadIdx.x < p.M)
        argmax_decode(p, threadIdx.x, atomicExch(p.keys + threadIdx.x, 0ull), gridDim.x);
      if (threadIdx.x == 0) *p.done = 0u;
    }
  }
}

// Every kernel of the projection is launched with programmatic stream
// serialization: it may be scheduled while the kernel before it in the stream
// is finishing, and waits for that kernel (griddepcontrol.wait) before it
// touches anything the kernel may have written.
template <typename Kern, typename... Args>
int launch_pdl(Kern k, dim3 grid, int threads, size_t smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...) == cudaSuccess ? VQ_OK : VQ_ECUDA;
}

template <int ACT, int MT, bool AM, int XM = 0, int WIDE = 0>
int launch_one(const GemmLaunch& L) {
  auto k = vq_gemm_kernel<ACT, MT, AM, XM, WIDE>;
  if (ensure_smem<vq_gemm_kernel<ACT, MT, AM, XM, WIDE>>(L.smem) != VQ_OK) return VQ_ECUDA;
  if constexpr (XM == 2 && ACT != VQ_F32) {
    // the slices first; the projection may start before they are done
    const int rc = launch_pdl(vq_prep_kernel<ACT>, dim3(L.p.KT * MT), kPrepThreads, 0, L.stream,
                              L.p.x, L.p.M, L.p.K, MT, (uint8_t*)L.p.xprep);
    if (rc != VQ_OK) return rc;
  }
  return launch_pdl(k, dim3(L.grid), Cfg<MT, WIDE>::THREADS, L.smem, L.stream, L.tm_w, L.tm_s, L.tm_b,
                    L.tm_x, L.p);
}

// The tensor-core (tcgen05) kernel for 16-bit x with M > 16 (vq_tc.cuh).
template <int ACT, int MP, bool AM>
int launch_tc(const GemmLaunch& L);

template <int ACT>
int launch_gemm_act(const GemmLaunch& L) {
#define VQ_CASE(mt)                                                      \
  case mt:                                                               \
    if (mt <= 2 && L.p.S == 1)                                           \
      return L.argmax ? launch_one<ACT, mt, true, 0, (mt <= 2)>(L)        \
                      : launch_one<ACT, mt, false, 0, (mt <= 2)>(L);      \
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
    if (L.p.xm == 1) {
      if (L.MT != 1 || !L.argmax) return VQ_EUNSUPPORTED;
      return launch_one<ACT, 1, true, 1>(L);
    }
    if (L.p.xm == 2) {
      if (L.MT > 2 || L.argmax) return VQ_EUNSUPPORTED;
      if (L.MT == 2)
        return L.p.S == 1 ? launch_one<ACT, 2, false, 2, 2>(L) : launch_one<ACT, 2, false, 2>(L);
      return L.p.S == 1 ? launch_one<ACT, 1, false, 2, 2>(L) : launch_one<ACT, 1, false, 2>(L);
    }
    if (L.p.xm == 3) {
      switch (L.MT) {
        case 4:
          return L.argmax ? launch_tc<ACT, 32, true>(L) : launch_tc<ACT, 32, false>(L);
        case 8:
          return L.argmax ? launch_tc<ACT, 64, true>(L) : launch_tc<ACT, 64, false>(L);
        default:
          return VQ_EUNSUPPORTED;
      }
    }
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
