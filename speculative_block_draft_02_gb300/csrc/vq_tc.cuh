// Tensor-core (tcgen05) variant of the W4 projection for 16-bit x with
// 16 < M <= 64 rows, where the product is a real dense contraction: a 128-row
// weight tile times 32 or 64 activation rows per 16-wide k step.
//
// Same definition as the mma.sync kernel (dflash-mlx #7, PR description:
// VerifyQuantizedLinear over 4-bit weights; ds4 #778, commit 1: one pass over
// the weights for every row of the verify block):
//
//   y[m][n] = sum_g ( scale[n][g] * A_g[n][m] + (bias[n][g] - c0*scale[n][g]) * X_g[m] )
//   A_g[n][m] = sum_{k in g} (c0 + code(n,k)) * x[m][k]
//   X_g[m]    = sum_{k in g} x[m][k]
//
// with c0 = 128 (bf16) or 1024 (f16): the codes enter the MMA as the exact
// integers c0+q, made from a nibble pair with one byte permute and one
// AND/OR, and every product is exact in the fp32 accumulator. (The f16 arg
// max subtracts the 1024 before the MMA, c0 = 0, to keep its fp32 maximum
// free of the offset's cancellation.)
//
// Roles in a block (one per SM, persistent over 128-row units):
//   producer (1 lane)  TMA: per 512-wide stage the unit's packed codes (2 x
//                      16 KiB), scales and biases (2 KiB each) and x as
//                      [8 groups][MP rows][128 B] 128B-swizzled tiles, into a
//                      D-deep ring; completion on mbarriers.
//   unpack (8 warps)   per 64-wide group (warps 0-3 even groups, 4-7 odd),
//                      row n = lane of the warp's TMEM lane quarter: 64 codes
//                      -> 32 columns of bf16/f16 pairs, written to the A
//                      buffer (4 buffers) with tcgen05.st.
//   MMA (2 lanes)      one thread per group parity; per group 4 x
//                      tcgen05.mma kind::f16, M=128, N=MP,
//                      K=16, A from TMEM, B (x) from shared memory, into one
//                      of 4 fp32 accumulators in TMEM; tcgen05.commit.
//   fold (16 warps, 8 at MP = 32)
//                      per group, tcgen05.ld of its accumulator (a row per
//                      lane, a quarter (half) of the MP columns per warp) and
//                      the fp32 fold with scale, bias and X_g, two columns per
//                      packed multiply-add; then the epilogue (store y, or
//                      the running arg max).
// X_g: a table for all of K in shared memory, written once per call by a
// small kernel into the workspace and copied in (vq_linear), or summed by the
// fold warps from each stage's x tile during the block's first unit (arg max,
// whose blocks take many units); when the table would leave room for fewer
// than two stages (long K at M > 32), the fold warps sum each stage's groups
// from its x tile into a double-buffered area instead, and K is not limited.
#pragma once

#include "vq_gemm.cuh"

namespace vq {

#ifdef __CUDACC__

constexpr int kTcUnpackWarps = 8;
constexpr int kTcMmaWarps = 2;
// Warp roles of a block: unpack warps 0-7, then the fold warps, the producer
// and the two MMA warps. Sixteen fold warps (each a lane quarter and a quarter
// of the MP accumulator columns) at MP = 64, eight (half the columns each) at
// MP = 32 — measured: the projection at M = 32, K = 5120, N = 17408 27.7 ->
// 25.8 us with eight, the arg max at M = 32, K = 2560, N = 151936 104.4 ->
// 100.7 us; at MP = 64 sixteen stay faster (projection 32.3 against 34.7 us,
// arg max 143 against 170 us).
template <int MP, bool ARGMAX>
struct TcRoles {
  static constexpr int kFold = MP == 32 ? 8 : 16;
  static constexpr int kProducer = kTcUnpackWarps + kFold;
  static constexpr int kMma = kProducer + 1;
  static constexpr int kThreads = (kMma + kTcMmaWarps) * 32;   // 864 (608 with 8 fold warps)
};
constexpr int kTcBufs = 4;              // A buffers and accumulators in flight
constexpr uint32_t kTcTmemCols = 512;   // A: 4 x 32 columns, D: 4 x MP (<= 64) columns
constexpr uint32_t kTcDCol = 32 * kTcBufs;   // first accumulator column

// ------------------------------------------------------------ tcgen05 PTX
__device__ __forceinline__ void tc_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[tmem] * B[smem descriptor]^T, kind::f16, fp32 accumulate.
__device__ __forceinline__ void tc_mma(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives on the mbarrier once every MMA this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),
      "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),
      "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tc_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Columns [taddr, taddr + N) of this warp's 32 TMEM lanes, one lane per thread.
template <int N>
__device__ __forceinline__ void tc_ld(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 4) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr)
                 : "memory");
  } else if constexpr (N == 8) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
  } else if constexpr (N == 16) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
  } else {
    static_assert(N == 32, "4, 8, 16 or 32 columns");
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
  }
}
__device__ __forceinline__ uint32_t lds32_at(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 lds128_at(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Shared-memory descriptor of a K-major operand whose rows are 128 bytes in
// the 128-byte swizzle (8-row atoms of 1 KiB, the TMA SWIZZLE_128B image):
// start address, leading offset (unused for this layout), stride between
// 8-row atoms, descriptor version 1, layout 128B swizzle.
__device__ __forceinline__ uint64_t tc_sdesc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: fp32 D, A and B both bf16 (or both f16),
// both K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t tc_idesc(bool bf16, int n) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// Codes 2p and 2p+1 of a word as the pair (c0 + q_2p, c0 + q_2p+1): byte p of
// w (low nibble = code 2p) and byte p of w >> 4 (low nibble = code 2p+1) go
// to the two halves, the AND/OR keeps the nibbles under the exponent of c0.
template <int P>
__device__ __forceinline__ uint32_t tc_pair(uint32_t w, uint32_t w4, uint32_t magic) {
  constexpr uint32_t sel = (uint32_t)P | ((uint32_t)P << 4) | ((uint32_t)(4 + P) << 8) |
                           ((uint32_t)(4 + P) << 12);
  return lop3_and_or(prmt(w, w4, sel), 0x000F000Fu, magic);
}

// X_g[m] (fp32, [K/64][MP], rows m >= M zero) in a fixed summation order.
template <int ACT>
__device__ __forceinline__ float tc_group_sum(const void* x, int K, int m, int g) {
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(x) +
                                                    ((size_t)m * K + (size_t)g * 64) * 2);
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 v = __ldg(src + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (ACT == VQ_F16) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        s += f.x;
        s += f.y;
      } else {
        s += __uint_as_float(w[i] << 16);
        s += __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
  }
  return s;
}

// X_g[m] from a stage's x tile in shared memory: group j's row m is 128 bytes
// at tile + (j*MP + m)*128, its 16-byte chunks 128B-swizzled (chunk c at
// (c ^ (m & 7)) << 4). Rows past M arrive zero-filled. Fixed summation order.
template <int ACT, int MP>
__device__ __forceinline__ float tc_group_sum_smem(uint32_t tile, int j, int m) {
  const uint32_t row = tile + (uint32_t)((j * MP + m) * 128);
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 v = lds128_at(row + (((uint32_t)c ^ (uint32_t)(m & 7)) << 4));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (ACT == VQ_F16) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        s += f.x;
        s += f.y;
      } else {
        s += __uint_as_float(w[i] << 16);
        s += __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
  }
  return s;
}

// X_g for the projection, once per call: thread e -> (g, m) = (e / MP, e % MP),
// for the groups of KT whole stages (those past K are 0).
template <int ACT>
__global__ void __launch_bounds__(256)
    vq_tc_xsum_kernel(const void* __restrict__ x, int M, int K, int KT, int MP,
                      float* __restrict__ out) {
  grid_launch_dependents();
  // x and the table may still be in use by the kernel before this one
  grid_wait_prerequisites();
  const int e = blockIdx.x * 256 + threadIdx.x;
  if (e >= KT * 8 * MP) return;
  const int g = e / MP, m = e - g * MP;
  out[e] = (m < M && g < K / 64) ? tc_group_sum<ACT>(x, K, m, g) : 0.f;
}

// Stage layout: [codes 2 x 16 KiB][scales 128 x 16 B][biases 128 x 16 B][x 8 x MP x 128 B]
constexpr int kTcOffS = 2 * kWeightBoxBytes;
constexpr int kTcOffB = kTcOffS + kBN * 16;
constexpr int kTcOffX = kTcOffB + kBN * 16;   // 36864: 1 KiB aligned
__host__ __device__ constexpr int tc_stage_bytes(int MP) { return kTcOffX + 8 * MP * 128; }
__host__ __device__ constexpr int tc_xs_bytes(int K, int MP) { return (K / 64) * MP * 4; }
// misc: mbarriers and flags (320 B), arg max scratch [4][64] value, index, runner-up
constexpr int kTcBarBytes = 320;
constexpr int kTcMiscBytes = kTcBarBytes + 3 * 4 * 64 * 4;

// Best row, its value and the runner-up value over the warp's 32 rows for each
// of its HC columns, by halving: at offset o (16, 8, ...) a lane keeps the
// half of its current columns selected by its lane bit o and merges in the
// partner's values for them; once one column is left, the remaining offsets
// merge whole. Lane l ends with column l / (32 / HC). Index 0xFFFFFFFF = no value.
template <int HC>
__device__ __forceinline__ void warp_top2_columns(float (&v)[HC], uint32_t (&n)[HC],
                                                  float (&s)[HC], int lane) {
  int o = 16;
#pragma unroll
  for (int cur = HC; cur > 1; cur >>= 1, o >>= 1) {
    const bool hi = (lane & o) != 0;
    const int half = cur >> 1;
#pragma unroll
    for (int j = 0; j < half; ++j) {
      const float rv = __shfl_xor_sync(0xffffffffu, hi ? v[j] : v[j + half], o);
      const uint32_t rn = __shfl_xor_sync(0xffffffffu, hi ? n[j] : n[j + half], o);
      const float rs = __shfl_xor_sync(0xffffffffu, hi ? s[j] : s[j + half], o);
      float kv = hi ? v[j + half] : v[j];
      uint32_t kn = hi ? n[j + half] : n[j];
      float ks = hi ? s[j + half] : s[j];
      bool kh = kn != 0xFFFFFFFFu;
      top2_merge(kv, kn, kh, ks, rv, rn, rn != 0xFFFFFFFFu, rs);
      v[j] = kv;
      n[j] = kh ? kn : 0xFFFFFFFFu;
      s[j] = ks;
    }
  }
#pragma unroll
  for (; o >= 1; o >>= 1) {
    const float rv = __shfl_xor_sync(0xffffffffu, v[0], o);
    const uint32_t rn = __shfl_xor_sync(0xffffffffu, n[0], o);
    const float rs = __shfl_xor_sync(0xffffffffu, s[0], o);
    bool kh = n[0] != 0xFFFFFFFFu;
    top2_merge(v[0], n[0], kh, s[0], rv, rn, rn != 0xFFFFFFFFu, rs);
    if (!kh) n[0] = 0xFFFFFFFFu;
  }
}

template <int ACT, int MP, bool ARGMAX>
__global__ void __launch_bounds__(TcRoles<MP, ARGMAX>::kThreads, 1)
    vq_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s,
                 const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_x,
                 const GemmParams p) {
  constexpr bool kF16 = ACT == VQ_F16;
  constexpr uint32_t kMagic = kF16 ? 0x64006400u : 0x43004300u;   // 1024 / 128
  // The arg max also returns the fp32 maximum, which the f16 offset (1024,
  // 137x the mean code) would blur through cancellation: there the codes are
  // made exact (one fp16 subtraction per pair) and c0 = 0.
  constexpr bool kExact = ARGMAX && kF16;
  constexpr float kC0 = kExact ? 0.f : kF16 ? 1024.f : 128.f;
  constexpr int kTcFoldWarps = TcRoles<MP, ARGMAX>::kFold;
  constexpr int kTcProducerWarp = TcRoles<MP, ARGMAX>::kProducer;
  constexpr int kTcMmaWarp = TcRoles<MP, ARGMAX>::kMma;
  constexpr int HC = MP / (kTcFoldWarps / 4);   // accumulator columns per fold warp
  constexpr uint32_t kIdesc = tc_idesc(!kF16, MP);
  static_assert(MP == 32 || MP == 64, "MP");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - raw);
  // [D stages][X_g table][misc]
  float* const xs_tab = reinterpret_cast<float*>(sbase + p.D * p.stage_bytes);
  uint8_t* const misc = sbase + p.D * p.stage_bytes + p.tab_bytes;
  const uint32_t misc_a = base + p.D * p.stage_bytes + p.tab_bytes;
  auto full_bar = [&](int s) { return misc_a + 8u * s; };
  auto empty_bar = [&](int s) { return misc_a + 64u + 8u * s; };
  auto afull_bar = [&](int b) { return misc_a + 128u + 8u * b; };    // A buffer written
  auto mdone_bar = [&](int b) { return misc_a + 160u + 8u * b; };    // MMAs of the group done
  auto dempty_bar = [&](int b) { return misc_a + 192u + 8u * b; };   // accumulator read
  const uint32_t xs_bar = misc_a + 224u;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(misc + 232);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(misc + 240);
  volatile int* const epi_flag = reinterpret_cast<volatile int*>(misc + 244);
  // scales and biases loaded by the producer lanes landed (sb_plain)
  auto sbfull_bar = [&](int s) { return misc_a + 256u + 8u * s; };
  float* const red_v = reinterpret_cast<float*>(misc + kTcBarBytes);
  uint32_t* const red_i = reinterpret_cast<uint32_t*>(misc + kTcBarBytes + 4 * 64 * 4);
  float* const red_s = reinterpret_cast<float*>(misc + kTcBarBytes + 2 * 4 * 64 * 4);
  const bool sbp = p.sb_plain != 0;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the next kernel in the stream may be scheduled as soon as SMs free up
  grid_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.D; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kTcFoldWarps);
      if (sbp) mbar_init(sbfull_bar(s), 32);   // every producer lane
    }
    for (int b = 0; b < kTcBufs; ++b) {
      mbar_init(afull_bar(b), kTcUnpackWarps / 2);
      mbar_init(mdone_bar(b), 1);
      mbar_init(dempty_bar(b), kTcFoldWarps);
    }
    mbar_init(xs_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kTcMmaWarp) {
    tc_alloc(smem_addr(tmem_slot), kTcTmemCols);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kTcProducerWarp) {
    // ------------------------------------------------------------ producer
    // lane 0 issues the TMA copies; with sb_plain (K % 512 != 0) all 32 lanes
    // also load the stage's scales and biases
    if (lane == 0 || sbp) {
      if (lane == 0) {
        prefetch_tensormap(&tm_w);
        if (!sbp) {
          prefetch_tensormap(&tm_s);
          prefetch_tensormap(&tm_b);
        }
        prefetch_tensormap(&tm_x);
      }
      // weights (constants of the model) before the wait for the kernel
      // before this one in the stream; x and X_g only after it
      const uint64_t w_policy = l2_evict_first_policy();
      auto issue_w = [&](int slot, int kt, int rb) {
        const uint32_t sb = base + slot * p.stage_bytes;
        const uint32_t fb = full_bar(slot);
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, p.tx_bytes);
          tma_load_2d_hint(sb, &tm_w, kt * (kBK / 8), rb * kBN, fb, w_policy);
          tma_load_2d_hint(sb + kWeightBoxBytes, &tm_w, kt * (kBK / 8) + 32, rb * kBN, fb,
                           w_policy);
          if (!sbp) {
            tma_load_2d_hint(sb + kTcOffS, &tm_s, kt * (kBK / 64), rb * kBN, fb, w_policy);
            tma_load_2d_hint(sb + kTcOffB, &tm_b, kt * (kBK / 64), rb * kBN, fb, w_policy);
          }
        }
        if (sbp) {
          load_stage_sb(p, sbase + slot * p.stage_bytes + kTcOffS,
                        sbase + slot * p.stage_bytes + kTcOffB, kt, rb, lane);
          mbar_arrive(sbfull_bar(slot));
        }
      };
      auto issue_x = [&](int slot, int kt) {
        if (lane != 0) return;
        const uint32_t sb = base + slot * p.stage_bytes;
        const uint32_t fb = full_bar(slot);
        if (p.x3d) {
          tma_load_3d(sb + kTcOffX, &tm_x, 0, 0, kt * 8, fb);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            tma_load_2d(sb + kTcOffX + j * MP * 128, &tm_x, kt * kBK + j * 64, 0, fb);
        }
      };
      int pre = 0;
      if ((int)blockIdx.x < p.n_units)
        for (int r = 0; r < p.pre && r < p.D && r < p.KT; ++r) {
          issue_w(r, r, blockIdx.x);
          ++pre;
        }
      grid_wait_prerequisites();
      if (!ARGMAX && !p.xs_stage && lane == 0) {
        const uint32_t xs_bytes = (uint32_t)tc_xs_bytes(p.KT * kBK, MP);
        mbar_arrive_expect_tx(xs_bar, xs_bytes);
        bulk_load(smem_addr(xs_tab), p.xprep, xs_bytes, xs_bar);
      }
      for (int r = 0; r < pre; ++r) issue_x(r, r);
      int q = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
        for (int kt = 0; kt < p.KT; ++kt) {
          if (pre > 0) {
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
          issue_w(slot, kt, u);
          issue_x(slot, kt);
          ++q;
        }
      }
      // let every copy issued land before the block can exit
      if (lane == 0) {
        for (int r = (q > p.D ? q - p.D : 0); r < q; ++r)
          wait_bounded(full_bar(r % p.D), (uint32_t)(r / p.D) & 1u, p.err);
        if (!ARGMAX && !p.xs_stage) wait_bounded(xs_bar, 0u, p.err);
      }
    }
  } else if (warp >= kTcMmaWarp) {
    // ------------------------------------------------------------- MMA issue
    // two issuing threads, one per group parity: each keeps its own two
    // accumulators and barriers busy while the other waits or commits
    if (lane == 0) {
      const int par = warp - kTcMmaWarp;
      bool aborted = false;
      int committed = -1;
      int q = 0;
      for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
        for (int kt = 0; kt < p.KT; ++kt, ++q) {
          const int slot = q % p.D;
          if (!aborted &&
              !wait_or_abort(full_bar(slot), (uint32_t)(q / p.D) & 1u, abort_flag, p.err))
            aborted = true;
          // descriptor of the stage's x tile; the group and k offsets only
          // add to its start-address field
          const uint64_t xdesc = tc_sdesc(base + slot * p.stage_bytes + kTcOffX);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int j = 2 * jj + par;
            const int G = 8 * q + j;
            const int b = j & 3;   // = G % kTcBufs
            const uint32_t ph = (uint32_t)(G / kTcBufs) & 1u;
            if (!aborted && !wait_or_abort(afull_bar(b), ph, abort_flag, p.err)) aborted = true;
            if (!aborted && G >= kTcBufs &&
                !wait_or_abort(dempty_bar(b), ph ^ 1u, abort_flag, p.err))
              aborted = true;
            if (aborted) continue;
            tc_fence_after();
            const uint32_t d = tmem + kTcDCol + (uint32_t)(MP * b);
            const uint32_t a = tmem + (uint32_t)(32 * b);
            const uint64_t gdesc = xdesc + (uint64_t)((j * MP * 128) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma(d, a + 8u * kk, gdesc + (uint64_t)(2 * kk), kIdesc, kk > 0 ? 1u : 0u);
            tc_commit(mdone_bar(b));
            committed = G;
          }
        }
      }
      // every MMA this thread issued has completed before TMEM is released
      if (committed >= 0)
        wait_bounded(mdone_bar(committed % kTcBufs), (uint32_t)(committed / kTcBufs) & 1u, p.err);
    }
  } else if (warp < kTcUnpackWarps) {
    // ---------------------------------------------------------------- unpack
    // warps 0-3 take the even groups, 4-7 the odd ones; each writes all 32
    // columns of its lane quarter's rows
    const int qd = warp & 3, par = warp >> 2;
    const int nl = 32 * qd + lane;   // row of the unit = TMEM lane
    const uint32_t tl = (uint32_t)(32 * qd) << 16;
    const uint32_t row_off = (uint32_t)nl * 128u;
    const uint32_t sw = (uint32_t)(nl & 7);
    bool aborted = false;
    int q = 0;
    for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
      for (int kt = 0; kt < p.KT; ++kt, ++q) {
        const int slot = q % p.D;
        if (!aborted &&
            !wait_or_abort(full_bar(slot), (uint32_t)(q / p.D) & 1u, abort_flag, p.err))
          aborted = true;
        const uint32_t sb = base + slot * p.stage_bytes;
        // unrolled only by two (the projection at M = 64 14 % faster than
        // fully unrolled: less code to fetch among the roles; the arg max,
        // with its fold loop unrolled by four, 1 % faster)
#pragma unroll(2)
        for (int jj = 0; jj < 4; ++jj) {
          const int j = 2 * jj + par;
          const int G = 8 * q + j;
          const int b = j & 3;
          const uint32_t ph = (uint32_t)(G / kTcBufs) & 1u;
          // the A buffer is free once the MMAs of its previous group are done
          if (!aborted && G >= kTcBufs &&
              !wait_or_abort(mdone_bar(b), ph ^ 1u, abort_flag, p.err))
            aborted = true;
          if (!aborted) {
            tc_fence_after();
            // the group's 8 words: 16-byte chunks (j%4)*2 and (j%4)*2+1 of the box j/4 row
            const uint32_t rb = sb + (uint32_t)(j >> 2) * kWeightBoxBytes + row_off;
            const uint32_t c0 = (uint32_t)((j & 3) * 2);
            const uint4 w0 = lds128_at(rb + ((c0 ^ sw) << 4));
            const uint4 w1 = lds128_at(rb + (((c0 + 1u) ^ sw) << 4));
            const uint32_t wd[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            uint32_t r[32];
#pragma unroll
            for (int wi = 0; wi < 8; ++wi) {
              const uint32_t w4 = wd[wi] >> 4;
              r[4 * wi + 0] = tc_pair<0>(wd[wi], w4, kMagic);
              r[4 * wi + 1] = tc_pair<1>(wd[wi], w4, kMagic);
              r[4 * wi + 2] = tc_pair<2>(wd[wi], w4, kMagic);
              r[4 * wi + 3] = tc_pair<3>(wd[wi], w4, kMagic);
            }
            if constexpr (kExact) {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&r[i]),
                                          __half2(__half(1024.f), __half(1024.f)));
                r[i] = *reinterpret_cast<const uint32_t*>(&v);
              }
            }
            tc_st32(tmem + tl + (uint32_t)(32 * b), r);
            tc_wait_st();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(afull_bar(b));
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ fold
    const int f = warp - kTcUnpackWarps;
    const int qd = f & 3, ch = f >> 2;   // lane quarter, column chunk
    const int nl = 32 * qd + lane;
    const uint32_t tl = (uint32_t)(32 * qd) << 16;
    const int ft = f * 32 + lane;   // 0 .. 32 * kTcFoldWarps - 1 over the fold warps
    bool aborted = false;
    // x and every output may belong to the kernel before this one
    grid_wait_prerequisites();
    if (!ARGMAX && !p.xs_stage) {
      if (!wait_or_abort(xs_bar, 0u, abort_flag, p.err)) aborted = true;
    }
    float run_v = 0.f, run_s = -INFINITY;
    uint32_t run_n = 0u;
    bool run_h = false;
    int q = 0;
    for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
      float tot[HC];
#pragma unroll
      for (int i = 0; i < HC; ++i) tot[i] = 0.f;
      for (int kt = 0; kt < p.KT; ++kt, ++q) {
        const int slot = q % p.D;
        if (!aborted &&
            !wait_or_abort(full_bar(slot), (uint32_t)(q / p.D) & 1u, abort_flag, p.err))
          aborted = true;
        const uint32_t sb = base + slot * p.stage_bytes;
        // X_g of this stage's groups: from the table, or summed here from the
        // stage's x tile (one (group, row) pair per fold thread) into a
        // double-buffered area (per-stage mode, or the arg max's first unit,
        // which fills the table for the units after it)
        const float* xs_base = xs_tab + kt * 8 * MP;
        if (p.xs_stage || (ARGMAX && u == (int)blockIdx.x)) {
          float* dst = p.xs_stage ? xs_tab + (q & 1) * 8 * MP : xs_tab + kt * 8 * MP;
          if (!aborted)
            for (int e = ft; e < 8 * MP; e += kTcFoldWarps * 32) {
              const int j = e / MP, m = e - j * MP;
              dst[j * MP + m] = tc_group_sum_smem<ACT, MP>(sb + kTcOffX, j, m);
            }
          named_bar_sync(1, kTcFoldWarps * 32);
          xs_base = dst;
        }
        uint4 sv = make_uint4(0u, 0u, 0u, 0u), bv = sv;
        if (sbp && !aborted &&
            !wait_or_abort(sbfull_bar(slot), (uint32_t)(q / p.D) & 1u, abort_flag, p.err))
          aborted = true;
        if (!aborted) {
          sv = lds128_at(sb + kTcOffS + (uint32_t)nl * 16u);
          bv = lds128_at(sb + kTcOffB + (uint32_t)nl * 16u);
        }
        const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
        const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
        // one group per step (buffer j & 3): its accumulator is read, the
        // buffer released, then folded (one group's HC registers at a time
        // keeps the fold warps within their register budget). The projection
        // unrolls this loop fully; the arg max, whose larger epilogue shares
        // the instruction cache, by four (measured with the packed
        // multiply-adds, per call: rolled 142.9 us, by two 137.8, by four
        // 130.3, fully 138.1).
#pragma unroll(ARGMAX ? 4 : 8)
        for (int j = 0; j < 8; ++j) {
          const int G = 8 * q + j;
          const int b = j & 3;
          const uint32_t ph = (uint32_t)(G / kTcBufs) & 1u;
          if (!aborted && !wait_or_abort(mdone_bar(b), ph, abort_flag, p.err)) aborted = true;
          uint32_t acc[HC];
          if (!aborted) {
            tc_fence_after();
            tc_ld<HC>(tmem + tl + kTcDCol + (uint32_t)(MP * b + HC * ch), acc);
            tc_wait_ld();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dempty_bar(b));
          if (!aborted) {
            uint32_t s2, b2;
            if constexpr (ARGMAX) {   // from shared memory (fewer live registers)
              s2 = lds32_at(sb + kTcOffS + (uint32_t)nl * 16u + (uint32_t)(j >> 1) * 4u);
              b2 = lds32_at(sb + kTcOffB + (uint32_t)nl * 16u + (uint32_t)(j >> 1) * 4u);
            } else {
              s2 = sw[j >> 1];
              b2 = bw[j >> 1];
            }
            const bool h = (j & 1) != 0;
            const float s = __uint_as_float(h ? (s2 & 0xFFFF0000u) : (s2 << 16));
            const float bb = __uint_as_float(h ? (b2 & 0xFFFF0000u) : (b2 << 16));
            const float c = fmaf(-kC0, s, bb);   // exact: bias - c0*scale
            const float4* xs4 = reinterpret_cast<const float4*>(xs_base + j * MP + HC * ch);
#pragma unroll
            for (int i4 = 0; i4 < HC / 4; ++i4) {
              // tot = s*acc + (c*X_g + tot), two columns per instruction
              const float4 xs = xs4[i4];
              fma2(tot[4 * i4 + 0], tot[4 * i4 + 1], c, c, xs.x, xs.y);
              fma2(tot[4 * i4 + 0], tot[4 * i4 + 1], s, s, __uint_as_float(acc[4 * i4 + 0]),
                   __uint_as_float(acc[4 * i4 + 1]));
              fma2(tot[4 * i4 + 2], tot[4 * i4 + 3], c, c, xs.z, xs.w);
              fma2(tot[4 * i4 + 2], tot[4 * i4 + 3], s, s, __uint_as_float(acc[4 * i4 + 2]),
                   __uint_as_float(acc[4 * i4 + 3]));
            }
          }
        }
        // every reader of the stage is done with it after its last group
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(slot));
      }
      const int n = u * kBN + nl;
      if constexpr (!ARGMAX) {
        if (!aborted && n < p.N) {
#pragma unroll
          for (int i = 0; i < HC; ++i) {
            const int m = HC * ch + i;
            if (m < p.M && in_bounds((size_t)m * p.N + n, p.y_elems, p.err))
              store_out<ACT>(p.y, (size_t)m * p.N + n, tot[i]);
          }
        }
      } else {
        // best row of this unit, its value and the runner-up for each of the
        // warp's columns; lane l keeps the running ones of column
        // HC*ch + l / (32 / HC) (rows grow with the unit, so ties keep the
        // lowest row)
        uint32_t cn[HC];
        float cs[HC];
#pragma unroll
        for (int i = 0; i < HC; ++i) {
          tot[i] += 0.0f;   // -0 -> +0
          cn[i] = (!aborted && n < p.N && !(tot[i] != tot[i])) ? (uint32_t)n : 0xFFFFFFFFu;
          cs[i] = -INFINITY;
        }
        warp_top2_columns<HC>(tot, cn, cs, lane);
        top2_merge(run_v, run_n, run_h, run_s, tot[0], cn[0], cn[0] != 0xFFFFFFFFu, cs[0]);
      }
    }
    if constexpr (ARGMAX) {
      if (lane % (32 / HC) == 0) {
        const int col = HC * ch + lane / (32 / HC);
        red_v[qd * 64 + col] = run_v;
        red_i[qd * 64 + col] = run_h ? run_n : 0xFFFFFFFFu;
        red_s[qd * 64 + col] = run_s;
      }
      named_bar_sync(1, kTcFoldWarps * 32);
      if (ft < MP) {
        float v = 0.f, vs = -INFINITY;
        uint32_t vn = 0u;
        bool vh = false;
        for (int w = 0; w < 4; ++w) {
          const uint32_t on = red_i[w * 64 + ft];
          top2_merge(v, vn, vh, vs, red_v[w * 64 + ft], on, on != 0xFFFFFFFFu, red_s[w * 64 + ft]);
        }
        if (vh && ft < p.M && !aborted) {
          const unsigned long long key =
              ((unsigned long long)float_order(v) << 32) | (unsigned long long)(0xFFFFFFFFu - vn);
          if (in_bounds((size_t)ft, (size_t)p.M, p.err)) atomicMax(p.keys + ft, key);
        }
        if (p.cand && ft < p.M && in_bounds((size_t)blockIdx.x * p.M + ft, p.cand_elems, p.err))
          p.cand[(size_t)blockIdx.x * p.M + ft] =
              make_uint4(__float_as_uint(v), (vh && !aborted) ? vn : 0xFFFFFFFFu,
                         __float_as_uint(vs), 0u);
      }
      __threadfence();
      named_bar_sync(1, kTcFoldWarps * 32);
      if (ft == 0) *epi_flag = (atomicAdd(p.done, 1u) == gridDim.x - 1);
      named_bar_sync(1, kTcFoldWarps * 32);
      if (*epi_flag) {
        __threadfence();
        if (ft < p.M) argmax_decode(p, ft, atomicExch(p.keys + ft, 0ull), gridDim.x);
        if (ft == 0) *p.done = 0u;
      }
    }
  }

  // every role is done with TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    tc_fence_after();
    tc_dealloc(tmem, kTcTmemCols);
  }
}

template <int ACT, int MP, bool AM>
int launch_tc(const GemmLaunch& L) {
  auto k = vq_tc_kernel<ACT, MP, AM>;
  if (ensure_smem<vq_tc_kernel<ACT, MP, AM>>(L.smem) != VQ_OK) return VQ_ECUDA;
  if (!AM && !L.p.xs_stage) {
    const int n = L.p.KT * 8 * MP;
    const int rc = launch_pdl(vq_tc_xsum_kernel<ACT>, dim3((n + 255) / 256), 256, 0, L.stream,
                              L.p.x, L.p.M, L.p.K, L.p.KT, MP, (float*)L.p.xprep);
    if (rc != VQ_OK) return rc;
  }
  return launch_pdl(k, dim3(L.grid), TcRoles<MP, AM>::kThreads, L.smem, L.stream, L.tm_w, L.tm_s, L.tm_b, L.tm_x,
                    L.p);
}

#endif  // __CUDACC__

}  // namespace vq
