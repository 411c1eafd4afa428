// Verify-block attention over the per-row KV cache (verify_attention).
//
// mlxcel #2865 "perf(speculative): commit per-row accepts in batched DFlash",
// Summary and commit message: once every batch row keeps its own accept count,
// the target rotates the verify block at each row's logical positions and
// masks, for every query, the stale gap between the row's valid prefix and the
// verify slots the rectangular cache shares across rows.
//
// Three kernels per call:
//   verify_attn_rope_kernel  one block per (query, key or value head, block
//       position j, batch row), one thread per rotation pair: rotates the
//       block's queries and keys at the logical position P + j and rounds them
//       to the storage type; the queries go to the workspace, the keys and the
//       values to cache slot S + j.
//   verify_attn_partial_kernel  one block per (chunk of 64 keys, KV head, group
//       of 64 query rows, batch row). It stages the group's rotated queries, the
//       chunk's keys (prefix slots, then the block's slots) and its values
//       (transposed) in shared memory, every load requested before any is waited
//       for, then four warps of 16 query rows each run S = Q K^T and O = P V on
//       mma.sync m16n8k16 with the softmax in fp32. P is split into a 16-bit high
//       part and a 16-bit remainder so that the probabilities keep about 16
//       significant bits through the tensor cores. It writes the chunk's
//       unnormalised output and its (max, sum) per row to the workspace.
//   verify_attn_combine_kernel  merges the chunks of every query row and writes
//       the 16-bit output.
// The second and third are launched with programmatic stream serialization and
// wait (griddepcontrol.wait) for the kernel before them; small blocks (52 KB of
// shared memory, at most 128 registers a thread) let four of them share an SM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "vq_common.cuh"

namespace vq {
namespace {

constexpr int kAttnThreads = 128;  // four warps of 16 query rows
constexpr int kAttnRows = 64;      // query rows per block
constexpr int kChunk = 64;         // keys per block
constexpr int kMaxRotPairs = 64;   // rotary_dim / 2 for D <= 128
constexpr int kMaxBlock = 64;      // largest verify block L
constexpr int kMaxCap = 1 << 24;   // positions stay exact in fp32

static_assert(kAttnThreads == 2 * kChunk, "the value tile is staged two threads per key");
static_assert(kChunk == 8 * 8, "the score tile is eight mma n-tiles of 8 keys");

struct AttnParams {
  const uint16_t* q;
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint16_t* k_cache;
  uint16_t* v_cache;
  const int32_t* prefix_len;
  const int32_t* src_off;
  uint16_t* out;
  int32_t* status;
  float* part_o;    // [B][Hkv][RG][NC][64][D]   unnormalised chunk outputs
  float2* part_ml;  // [B][Hkv][RG][NC][64]      (max in log2 units, sum)
  uint16_t* q_rot;  // [B][L][Hq][D]              rotated, rounded queries
  int L, Hq, Hkv, G, R, RG, NC, S_cap, rot_half;
  float scale_log2;                  // scale * log2(e)
  float2 inv_freq[kMaxRotPairs];     // (hi, lo): hi + lo = theta^(-2i / rotary_dim)
};

template <bool kF16>
__device__ __forceinline__ float h2f(uint16_t h) {
  if constexpr (kF16) {
    return __half2float(__ushort_as_half(h));
  } else {
    return __bfloat162float(__ushort_as_bfloat16(h));
  }
}

// Round to nearest even into the storage type.
template <bool kF16>
__device__ __forceinline__ uint16_t f2h(float v) {
  if constexpr (kF16) {
    return __half_as_ushort(__float2half_rn(v));
  } else {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
}

// (a, b) as a 16-bit pair hi, and what rounding left behind as a second pair lo.
template <bool kF16>
__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
  const uint16_t ha = f2h<kF16>(a), hb = f2h<kF16>(b);
  hi = (uint32_t)ha | ((uint32_t)hb << 16);
  lo = (uint32_t)f2h<kF16>(a - h2f<kF16>(ha)) | ((uint32_t)f2h<kF16>(b - h2f<kF16>(hb)) << 16);
}

// 16 bytes global -> shared without a register round trip; zeros when !valid
// (nothing is read then).
__device__ __forceinline__ void cp_async_16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ uint32_t ld_u32(const uint16_t* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

__device__ __forceinline__ bool row_in_range(int P, int S, int L, int S_cap) {
  return P >= 0 && S >= P && (long long)S + L <= (long long)S_cap;
}

// (cos, sin) of pos * f for f = hi + lo: the angle is formed as a + err with
// a = fl(pos * hi) and err the rest of pos * (hi + lo), then turned to first
// order: sin(a + err) ~ sin a + err cos a (|err| < 1e-3 rad).
__device__ __forceinline__ float2 rope_cos_sin(float pos, float2 f) {
  const float a = pos * f.x;
  const float err = fmaf(pos, f.x, -a) + pos * f.y;
  float s, c;
  sincosf(a, &s, &c);
  return make_float2(c - err * s, s + err * c);
}

// Row r of blockIdx.x: query heads 0..Hq-1, then key heads, then value heads.
// Thread e < rot_half turns the pair (e, e + rot_half); the others copy two of
// the dimensions rotary_dim..D-1 (value rows: two dimensions per thread).
template <bool kF16, int D>
__global__ void __launch_bounds__(D / 2)
    verify_attn_rope_kernel(const __grid_constant__ AttnParams p) {
  const int r = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int e = threadIdx.x;
  grid_launch_dependents();
  const int P = p.prefix_len[b], S = p.src_off[b];
  if (!row_in_range(P, S, p.L, p.S_cap)) return;   // flagged by the combine kernel
  const int rh = p.rot_half;
  const uint16_t* src;
  uint16_t* dst;
  if (r < p.Hq) {
    src = p.q + (((size_t)b * p.L + j) * p.Hq + r) * D;
    dst = p.q_rot + (((size_t)b * p.L + j) * p.Hq + r) * D;
  } else if (r < p.Hq + p.Hkv) {
    const int h = r - p.Hq;
    src = p.k_new + (((size_t)b * p.L + j) * p.Hkv + h) * D;
    dst = p.k_cache + (((size_t)b * p.Hkv + h) * p.S_cap + (S + j)) * D;
  } else {
    const int h = r - p.Hq - p.Hkv;
    const uint32_t v = reinterpret_cast<const uint32_t*>(
        p.v_new + (((size_t)b * p.L + j) * p.Hkv + h) * D)[e];
    reinterpret_cast<uint32_t*>(p.v_cache + (((size_t)b * p.Hkv + h) * p.S_cap + (S + j)) * D)[e] = v;
    return;
  }
  if (e < rh) {
    const float2 cs = rope_cos_sin((float)(P + j), p.inv_freq[e]);
    const float x1 = h2f<kF16>(src[e]), x2 = h2f<kF16>(src[e + rh]);
    dst[e] = f2h<kF16>(x1 * cs.x - x2 * cs.y);
    dst[e + rh] = f2h<kF16>(x2 * cs.x + x1 * cs.y);
  } else {
    const int d = 2 * rh + 2 * (e - rh);
    dst[d] = src[d];
    dst[d + 1] = src[d + 1];
  }
}

template <bool kF16, int D>
__global__ void __launch_bounds__(kAttnThreads, 4)
    verify_attn_partial_kernel(const __grid_constant__ AttnParams p) {
  constexpr int QS = D + 8;        // row stride of the query and key tiles (16-bit elements)
  constexpr int VS = kChunk + 8;   // row stride of the transposed value tile
  constexpr int DC = D / 8;        // 16-byte pieces per row
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem);   // [64][QS]
  uint16_t* Ks = Qs + kAttnRows * QS;                  // [kChunk][QS]
  uint16_t* Vt = Ks + kChunk * QS;                     // [D][VS]: Vt[d][key]

  const int chunk = blockIdx.x;
  const int hk = blockIdx.y / p.RG, rg = blockIdx.y % p.RG;
  const int b = blockIdx.z;
  grid_launch_dependents();
  const int P = p.prefix_len[b], S = p.src_off[b];
  if (!row_in_range(P, S, p.L, p.S_cap)) return;   // flagged by the combine kernel
  const int T = P + p.L;                            // visible keys of the last query
  const int c0 = chunk * kChunk;
  if (c0 >= T) return;
  const int tid = threadIdx.x;
  // the rotated queries and the block's cache slots come from the kernel before
  grid_wait_prerequisites();

  // Visible key t (t < T) sits in cache slot t below P, in slot S + (t - P) above.
  const uint16_t* kbase = p.k_cache + ((size_t)b * p.Hkv + hk) * p.S_cap * D;
  const uint16_t* vbase = p.v_cache + ((size_t)b * p.Hkv + hk) * p.S_cap * D;
  // Query rows of this group: row r = j * G + (hq - hk * G).
  for (int i = tid; i < kAttnRows * DC; i += kAttnThreads) {
    const int r = i / DC, dc = i - r * DC;
    const int rr = rg * kAttnRows + r;
    const uint16_t* src = p.q_rot;
    if (rr < p.R) {
      const int j = rr / p.G, hq = hk * p.G + (rr - j * p.G);
      src = p.q_rot + (((size_t)b * p.L + j) * p.Hq + hq) * D + dc * 8;
    }
    cp_async_16(Qs + r * QS + dc * 8, src, rr < p.R);
  }
  for (int i = tid; i < kChunk * DC; i += kAttnThreads) {
    const int tl = i / DC, dc = i - tl * DC;
    const int t = c0 + tl;
    const int slot = t < P ? t : S + (t - P);
    cp_async_16(Ks + tl * QS + dc * 8, t < T ? kbase + (size_t)slot * D + dc * 8 : p.k_cache,
                t < T);
  }
  // Values: threads tid and tid + 64 share key c0 + (tid & 63), half of D each.
  {
    const int tl = tid & (kChunk - 1), half = tid / kChunk;
    const int t = c0 + tl;
    const int slot = t < P ? t : S + (t - P);
    const uint16_t* src = t < T ? vbase + (size_t)slot * D + half * (D / 2) : nullptr;
    uint4 vv[DC / 2];
#pragma unroll
    for (int dc = 0; dc < DC / 2; ++dc)
      vv[dc] = src ? __ldcg(reinterpret_cast<const uint4*>(src) + dc) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int dc = 0; dc < DC / 2; ++dc) {
      const uint32_t w[4] = {vv[dc].x, vv[dc].y, vv[dc].z, vv[dc].w};
      uint16_t* col = Vt + (half * (D / 2) + dc * 8) * VS + tl;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        col[(2 * e) * VS] = (uint16_t)(w[e] & 0xFFFFu);
        col[(2 * e + 1) * VS] = (uint16_t)(w[e] >> 16);
      }
    }
  }
  cp_async_wait_all();
  __syncthreads();

  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, tq = lane & 3;
  const int row0 = warp * 16;
  const int rA = rg * kAttnRows + row0 + g, rB = rA + 8;   // rows of c0/c1 and c2/c3
  if (rg * kAttnRows + row0 >= p.R) return;               // no barrier follows
  const bool okA = rA < p.R, okB = rB < p.R;
  const int jA = rA / p.G, jB = rB / p.G;

  float sc[8][4];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint16_t* q0 = Qs + (row0 + g) * QS + ks * 16 + 2 * tq;
    const uint32_t qa[4] = {ld_u32(q0), ld_u32(q0 + 8 * QS), ld_u32(q0 + 8),
                            ld_u32(q0 + 8 * QS + 8)};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const uint16_t* k0 = Ks + (nt * 8 + g) * QS + ks * 16 + 2 * tq;
      mma_16816<kF16>(sc[nt], qa, ld_u32(k0), ld_u32(k0 + 8));
    }
  }
  // mask (prefix for all, block keys causally, nothing past T), scale, row max
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int t = c0 + nt * 8 + 2 * tq + (e & 1);
      const int hh = e >> 1;
      const bool vis = (hh ? okB : okA) && t < T && (t < P || t - P <= (hh ? jB : jA));
      const float v = vis ? sc[nt][e] * p.scale_log2 : -INFINITY;
      sc[nt][e] = v;
      mx[hh] = fmaxf(mx[hh], v);
    }
  }
  float mu[2], l[2] = {0.f, 0.f};
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 1));
    mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 2));
    mu[hh] = mx[hh] == -INFINITY ? 0.f : mx[hh];   // no visible key: every p is 0
  }
  float o[D / 8][4];
#pragma unroll
  for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < kChunk / 16; ++kk) {
    uint32_t ah[4], al[4];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int nt = 2 * kk + half;
      const float p0 = exp2f(sc[nt][0] - mu[0]), p1 = exp2f(sc[nt][1] - mu[0]);
      const float p2 = exp2f(sc[nt][2] - mu[1]), p3 = exp2f(sc[nt][3] - mu[1]);
      l[0] += p0 + p1;
      l[1] += p2 + p3;
      split_pair<kF16>(p0, p1, ah[2 * half], al[2 * half]);
      split_pair<kF16>(p2, p3, ah[2 * half + 1], al[2 * half + 1]);
    }
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      const uint16_t* v0 = Vt + (nd * 8 + g) * VS + kk * 16 + 2 * tq;
      const uint32_t b0 = ld_u32(v0), b1 = ld_u32(v0 + 8);
      mma_16816<kF16>(o[nd], ah, b0, b1);
      mma_16816<kF16>(o[nd], al, b0, b1);
    }
  }

#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    l[hh] += __shfl_xor_sync(0xffffffffu, l[hh], 1);
    l[hh] += __shfl_xor_sync(0xffffffffu, l[hh], 2);
  }
  const size_t part = (((size_t)b * p.Hkv + hk) * p.RG + rg) * p.NC + chunk;
  float* po = p.part_o + part * kAttnRows * D;
  float2* pml = p.part_ml + part * kAttnRows;
  const int lA = row0 + g, lB = lA + 8;
  if (okA) {
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd)
      *reinterpret_cast<float2*>(po + lA * D + nd * 8 + 2 * tq) = make_float2(o[nd][0], o[nd][1]);
    if (tq == 0) pml[lA] = make_float2(mx[0], l[0]);
  }
  if (okB) {
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd)
      *reinterpret_cast<float2*>(po + lB * D + nd * 8 + 2 * tq) = make_float2(o[nd][2], o[nd][3]);
    if (tq == 0) pml[lB] = make_float2(mx[1], l[1]);
  }
}

// One block per (block position j, query head), one thread per dimension.
template <bool kF16, int D>
__global__ void __launch_bounds__(D) verify_attn_combine_kernel(const __grid_constant__ AttnParams p) {
  const int jh = blockIdx.x, b = blockIdx.y;
  const int j = jh / p.Hq, hq = jh - j * p.Hq;
  const int d = threadIdx.x;
  grid_wait_prerequisites();   // launched early (programmatic serialization)
  uint16_t* dst = p.out + (((size_t)b * p.L + j) * p.Hq + hq) * D;
  const int P = p.prefix_len[b], S = p.src_off[b];
  if (!row_in_range(P, S, p.L, p.S_cap)) {
    dst[d] = 0;
    if (jh == 0 && d == 0 && p.status) atomicOr(p.status, 1);
    return;
  }
  const int nc = (P + p.L + kChunk - 1) / kChunk;
  const int hk = hq / p.G, rr = j * p.G + (hq - hk * p.G);
  const int rg = rr / kAttnRows, lr = rr - rg * kAttnRows;
  const size_t part0 = (((size_t)b * p.Hkv + hk) * p.RG + rg) * p.NC;
  // every query sees its own key, so some chunk has a finite maximum
  float mmax = -INFINITY;
#pragma unroll 8
  for (int c = 0; c < nc; ++c) mmax = fmaxf(mmax, p.part_ml[(part0 + c) * kAttnRows + lr].x);
  float acc = 0.f, den = 0.f;
#pragma unroll 8
  for (int c = 0; c < nc; ++c) {
    const float2 ml = p.part_ml[(part0 + c) * kAttnRows + lr];
    const float w = exp2f(ml.x - mmax);
    den += w * ml.y;
    acc += w * p.part_o[((part0 + c) * kAttnRows + lr) * D + d];
  }
  dst[d] = f2h<kF16>(acc / den);
}

int attn_check(const void* q, const void* k_new, const void* v_new, const void* k_cache,
               const void* v_cache, const int32_t* prefix_len, const int32_t* src_off,
               const void* out, int B, int L, int Hq, int Hkv, int D, int S_cap, int rotary_dim,
               double theta, double scale, int dtype, const int32_t* status) {
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !prefix_len || !src_off || !out)
    return VQ_EINVAL;
  if (B < 1 || L < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 1 || S_cap < L)
    return VQ_EINVAL;
  if (dtype != VQ_BF16 && dtype != VQ_F16) return VQ_EINVAL;
  if (rotary_dim < 0 || rotary_dim > D || rotary_dim % 2 != 0) return VQ_EINVAL;
  if (rotary_dim > 0 && !(theta > 0.0 && std::isfinite(theta))) return VQ_EINVAL;
  if (!std::isfinite(scale)) return VQ_EINVAL;
  if (D != 64 && D != 128) return VQ_EUNSUPPORTED;
  if (L > kMaxBlock || S_cap > kMaxCap) return VQ_EUNSUPPORTED;
  // grid limits: (chunks, Hkv x row groups, B) and (L x Hq, B)
  const long long row_groups = ((long long)L * (Hq / Hkv) + kAttnRows - 1) / kAttnRows;
  if ((long long)Hkv * row_groups > 65535 || B > 65535 || (long long)L * Hq > 0x7fffffffll ||
      (long long)Hq + 2ll * Hkv > 0x7fffffffll)
    return VQ_EUNSUPPORTED;
  const uintptr_t a16 = (uintptr_t)q | (uintptr_t)k_new | (uintptr_t)v_new |
                        (uintptr_t)k_cache | (uintptr_t)v_cache;
  if ((a16 & 15u) || ((uintptr_t)out & 1u) ||
      (((uintptr_t)prefix_len | (uintptr_t)src_off | (uintptr_t)status) & 3u))
    return VQ_EALIGN;
  return VQ_OK;
}

struct AttnShape {
  int G, R, RG, NC;
};

AttnShape attn_shape(int L, int Hq, int Hkv, int S_cap) {
  AttnShape s;
  s.G = Hq / Hkv;
  s.R = L * s.G;
  s.RG = (s.R + kAttnRows - 1) / kAttnRows;
  s.NC = (S_cap + kChunk - 1) / kChunk;
  return s;
}

size_t attn_part_count(int B, int Hkv, const AttnShape& s) {
  return (size_t)B * Hkv * s.RG * s.NC * kAttnRows;
}

// A launch that may start while the kernel before it in the stream finishes;
// the kernel itself waits (griddepcontrol.wait) before reading that kernel's
// results.
template <typename Kern>
int launch_overlapped(Kern k, dim3 grid, int threads, size_t smem, cudaStream_t stream,
                      const AttnParams& p) {
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
  return cudaLaunchKernelEx(&cfg, k, p) == cudaSuccess ? VQ_OK : VQ_ECUDA;
}

template <bool kF16, int D>
int attn_launch(const AttnParams& p, int B, cudaStream_t stream) {
  const size_t smem = (size_t)(kAttnRows + kChunk) * (D + 8) * 2 + (size_t)D * (kChunk + 8) * 2;
  auto* partial = verify_attn_partial_kernel<kF16, D>;
  if (cudaFuncSetAttribute(partial, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return VQ_ECUDA;
  // the rope kernel runs after everything before it in the stream (a plain launch)
  verify_attn_rope_kernel<kF16, D><<<dim3(p.Hq + 2 * p.Hkv, p.L, B), D / 2, 0, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return VQ_ECUDA;
  int rc = launch_overlapped(partial, dim3(p.NC, p.Hkv * p.RG, B), kAttnThreads, smem, stream, p);
  if (rc) return rc;
  return launch_overlapped(verify_attn_combine_kernel<kF16, D>, dim3(p.L * p.Hq, B), D, 0, stream,
                           p);
}

}  // namespace
}  // namespace vq

using namespace vq;

extern "C" size_t verify_attention_workspace_bytes(int B, int L, int Hq, int Hkv, int D,
                                                   int S_cap) {
  if (B < 1 || L < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 1 || S_cap < 1) return 0;
  const AttnShape s = attn_shape(L, Hq, Hkv, S_cap);
  const size_t rows = attn_part_count(B, Hkv, s);
  return rows * (size_t)D * sizeof(float) + rows * sizeof(float2) +
         (size_t)B * L * Hq * D * sizeof(uint16_t);
}

extern "C" int verify_attention(const void* q, const void* k_new, const void* v_new,
                                void* k_cache, void* v_cache, const int32_t* prefix_len,
                                const int32_t* src_off, void* out, int B, int L, int Hq, int Hkv,
                                int D, int S_cap, int rotary_dim, double theta, double scale,
                                int dtype, int32_t* status, void* workspace,
                                size_t workspace_bytes, void* stream) {
  int rc = attn_check(q, k_new, v_new, k_cache, v_cache, prefix_len, src_off, out, B, L, Hq, Hkv,
                      D, S_cap, rotary_dim, theta, scale, dtype, status);
  if (rc) return rc;
  const size_t need = verify_attention_workspace_bytes(B, L, Hq, Hkv, D, S_cap);
  if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 15u)) return VQ_EWORKSPACE;
  rc = num_sms_current_device(nullptr);   // a usable current device
  if (rc) return rc;

  const AttnShape s = attn_shape(L, Hq, Hkv, S_cap);
  AttnParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.k_cache = static_cast<uint16_t*>(k_cache);
  p.v_cache = static_cast<uint16_t*>(v_cache);
  p.prefix_len = prefix_len;
  p.src_off = src_off;
  p.out = static_cast<uint16_t*>(out);
  p.status = status;
  const size_t rows = attn_part_count(B, Hkv, s);
  p.part_o = static_cast<float*>(workspace);
  p.part_ml = reinterpret_cast<float2*>(static_cast<char*>(workspace) +
                                        rows * (size_t)D * sizeof(float));
  p.q_rot = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) +
                                        rows * ((size_t)D * sizeof(float) + sizeof(float2)));
  p.L = L;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = s.G;
  p.R = s.R;
  p.RG = s.RG;
  p.NC = s.NC;
  p.S_cap = S_cap;
  p.rot_half = rotary_dim / 2;
  p.scale_log2 = (float)(scale * 1.4426950408889634);   // log2(e)
  for (int i = 0; i < p.rot_half; ++i) {
    const double f = pow(theta, -2.0 * i / (double)rotary_dim);
    const float hi = (float)f;
    p.inv_freq[i] = make_float2(hi, (float)(f - (double)hi));
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == VQ_F16) return D == 64 ? attn_launch<true, 64>(p, B, st) : attn_launch<true, 128>(p, B, st);
  return D == 64 ? attn_launch<false, 64>(p, B, st) : attn_launch<false, 128>(p, B, st);
}
