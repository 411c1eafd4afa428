// Verify-block attention over the per-row KV cache (verify_attention).
//
// mlxcel #2865 "perf(speculative): commit per-row accepts in batched DFlash",
// Summary and commit message: once every batch row keeps its own accept count,
// the rotary embedding and the attention of the verify block use every row's
// own logical positions, and no query sees the stale gap between its row's
// valid prefix and the verify slots the rectangular cache shares across rows.
//
// Two kernels per call:
//   verify_attn_partial_kernel  one block per (key chunk of 128, KV head, group
//       of 64 query rows, batch row). It stages the group's rotated queries and
//       the chunk's keys (prefix slots read from the cache; the block's own keys
//       rotated at their logical positions, rounded to the storage type and
//       appended to the cache) and values in shared memory, then four warps of
//       16 query rows each run S = Q K^T and O += P V on mma.sync m16n8k16 with
//       an online softmax in fp32. P is split into a 16-bit high part and a
//       16-bit remainder so that the probabilities keep about 16 significant
//       bits through the tensor cores. It writes the chunk's unnormalised
//       output and its (max, sum) per row to the workspace.
//   verify_attn_combine_kernel  merges the chunks of every query row and writes
//       the 16-bit output.
// The chunks are small (at most 64 KB of K and V per block) and every block
// reads its own slice once, so the staging is 16-byte pieces, all requested
// before any is waited for: cp.async for the query rows and keys, register
// loads for the values (transposed into shared memory). The merge is launched
// with programmatic stream serialization and waits for the partial kernel.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "vq_common.cuh"

namespace vq {
namespace {

constexpr int kAttnThreads = 128;  // four warps of 16 query rows
constexpr int kAttnRows = 64;      // query rows per block
constexpr int kChunk = 128;        // keys per block (one per thread when staging V)
constexpr int kSub = 64;           // keys per softmax step
constexpr int kMaxRotPairs = 64;   // rotary_dim / 2 for D <= 128
constexpr int kMaxBlock = 64;      // largest verify block L
constexpr int kMaxCap = 1 << 24;   // positions stay exact in fp32

static_assert(kChunk == kAttnThreads, "the value tile is staged one key per thread");
static_assert(kChunk % kSub == 0 && kSub % 16 == 0, "softmax steps cover whole mma k-steps");

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

// Turns the pair (x[e], x[e + h]) of a 16-bit row in shared memory by the angle
// whose (cos, sin) is cs, rounding the results to the storage type.
template <bool kF16>
__device__ __forceinline__ void rotate_pair(uint16_t* row, int e, int h, float2 cs) {
  const float x1 = h2f<kF16>(row[e]), x2 = h2f<kF16>(row[e + h]);
  row[e] = f2h<kF16>(x1 * cs.x - x2 * cs.y);
  row[e + h] = f2h<kF16>(x2 * cs.x + x1 * cs.y);
}

template <bool kF16, int D>
__global__ void __launch_bounds__(kAttnThreads)
    verify_attn_partial_kernel(const __grid_constant__ AttnParams p) {
  constexpr int QS = D + 8;        // row stride of the query and key tiles (16-bit elements)
  constexpr int VS = kChunk + 8;   // row stride of the transposed value tile
  constexpr int DC = D / 8;        // 16-byte pieces per row
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem);   // [64][QS]
  uint16_t* Ks = Qs + kAttnRows * QS;                  // [kChunk][QS]
  uint16_t* Vt = Ks + kChunk * QS;                     // [D][VS]: Vt[d][key]
  float2* cs = reinterpret_cast<float2*>(Vt + D * VS); // [L][rot_half] (cos, sin)

  const int chunk = blockIdx.x;
  const int hk = blockIdx.y / p.RG, rg = blockIdx.y % p.RG;
  const int b = blockIdx.z;
  const int P = p.prefix_len[b], S = p.src_off[b];
  if (!row_in_range(P, S, p.L, p.S_cap)) return;   // flagged by the combine kernel
  const int T = P + p.L;                            // visible keys of the last query
  const int c0 = chunk * kChunk;
  if (c0 >= T) return;
  const int tid = threadIdx.x;
  const int rh = p.rot_half;
  grid_launch_dependents();

  // Every load of the stage is issued before any of them is waited for: the
  // query rows and the keys go global -> shared asynchronously, the values
  // (transposed on the way) through registers.
  // Query rows of this group: row r = j * G + (hq - hk * G).
  for (int i = tid; i < kAttnRows * DC; i += kAttnThreads) {
    const int r = i / DC, dc = i - r * DC;
    const int rr = rg * kAttnRows + r;
    const uint16_t* src = p.q;
    if (rr < p.R) {
      const int j = rr / p.G, hq = hk * p.G + (rr - j * p.G);
      src = p.q + (((size_t)b * p.L + j) * p.Hq + hq) * D + dc * 8;
    }
    cp_async_16(Qs + r * QS + dc * 8, src, rr < p.R);
  }
  // Keys: prefix slots from the cache, the block's keys (rotated below), zeros past T.
  for (int i = tid; i < kChunk * DC; i += kAttnThreads) {
    const int tl = i / DC, dc = i - tl * DC;
    const int t = c0 + tl;
    const uint16_t* src = p.k_cache;
    if (t < P) {
      src = p.k_cache + (((size_t)b * p.Hkv + hk) * p.S_cap + t) * D + dc * 8;
    } else if (t < T) {
      src = p.k_new + (((size_t)b * p.L + (t - P)) * p.Hkv + hk) * D + dc * 8;
    }
    cp_async_16(Ks + tl * QS + dc * 8, src, t < T);
  }
  // Values: thread tid owns key c0 + tid.
  uint4 vv[DC];
  {
    const int t = c0 + tid;
    const uint16_t* src = nullptr;
    if (t < P) {
      src = p.v_cache + (((size_t)b * p.Hkv + hk) * p.S_cap + t) * D;
    } else if (t < T) {
      src = p.v_new + (((size_t)b * p.L + (t - P)) * p.Hkv + hk) * D;
    }
#pragma unroll
    for (int dc = 0; dc < DC; ++dc)
      vv[dc] = src ? __ldg(reinterpret_cast<const uint4*>(src) + dc) : make_uint4(0u, 0u, 0u, 0u);
  }

  // (cos, sin) of every block position's angles, while the loads are in flight.
  // The angle pos * f is formed as a + err with a = fl(pos * hi) and err the rest
  // of pos * (hi + lo), then turned to first order: sin(a + err) ~ sin a + err cos a
  // (|err| < 1e-3 rad).
  for (int i = tid; i < p.L * rh; i += kAttnThreads) {
    const int j = i / rh, e = i - j * rh;
    const float pos = (float)(P + j);
    const float2 f = p.inv_freq[e];
    const float a = pos * f.x;
    const float err = fmaf(pos, f.x, -a) + pos * f.y;
    float s, c;
    sincosf(a, &s, &c);
    cs[i] = make_float2(c - err * s, s + err * c);
  }

#pragma unroll
  for (int dc = 0; dc < DC; ++dc) {
    const uint32_t w[4] = {vv[dc].x, vv[dc].y, vv[dc].z, vv[dc].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      Vt[(dc * 8 + 2 * e) * VS + tid] = (uint16_t)(w[e] & 0xFFFFu);
      Vt[(dc * 8 + 2 * e + 1) * VS + tid] = (uint16_t)(w[e] >> 16);
    }
  }
  cp_async_wait_all();
  __syncthreads();

  // Rotate the queries and the block's keys at their logical positions P + j.
  for (int i = tid; i < kAttnRows * rh; i += kAttnThreads) {
    const int r = i / rh, e = i - r * rh;
    const int rr = rg * kAttnRows + r;
    if (rr < p.R) rotate_pair<kF16>(Qs + r * QS, e, rh, cs[(rr / p.G) * rh + e]);
  }
  const int tb0 = max(c0, P) - c0;               // first block key in this chunk
  const int nb = min(c0 + kChunk, T) - c0 - tb0;  // block keys in this chunk (may be <= 0)
  for (int i = tid; i < max(nb, 0) * rh; i += kAttnThreads) {
    const int k = i / rh, e = i - k * rh;
    const int tl = tb0 + k;
    rotate_pair<kF16>(Ks + tl * QS, e, rh, cs[(c0 + tl - P) * rh + e]);
  }
  __syncthreads();

  // Append the block's keys and values at slots S + j (one row group writes).
  if (rg == 0) {
    for (int i = tid; i < max(nb, 0) * DC; i += kAttnThreads) {
      const int k = i / DC, dc = i - k * DC;
      const int tl = tb0 + k;
      const int j = c0 + tl - P;
      const size_t slot = (((size_t)b * p.Hkv + hk) * p.S_cap + (S + j)) * D;
      reinterpret_cast<uint4*>(p.k_cache + slot)[dc] =
          *reinterpret_cast<const uint4*>(Ks + tl * QS + dc * 8);
      reinterpret_cast<uint4*>(p.v_cache + slot)[dc] = __ldg(
          reinterpret_cast<const uint4*>(p.v_new + (((size_t)b * p.L + j) * p.Hkv + hk) * D) + dc);
    }
  }

  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, tq = lane & 3;
  const int row0 = warp * 16;
  const int rA = rg * kAttnRows + row0 + g, rB = rA + 8;   // rows of c0/c1 and c2/c3
  if (rg * kAttnRows + row0 >= p.R) return;               // no barrier follows
  const bool okA = rA < p.R, okB = rB < p.R;
  const int jA = rA / p.G, jB = rB / p.G;

  uint32_t qa[D / 16][4];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint16_t* q0 = Qs + (row0 + g) * QS + ks * 16 + 2 * tq;
    qa[ks][0] = ld_u32(q0);
    qa[ks][1] = ld_u32(q0 + 8 * QS);
    qa[ks][2] = ld_u32(q0 + 8);
    qa[ks][3] = ld_u32(q0 + 8 * QS + 8);
  }
  float o[D / 8][4];
#pragma unroll
  for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

#pragma unroll 1
  for (int st = 0; st < kChunk / kSub; ++st) {
    const int kb = c0 + st * kSub;
    if (kb >= T) break;
    float sc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const uint16_t* k0 = Ks + (st * kSub + nt * 8 + g) * QS + ks * 16 + 2 * tq;
        mma_16816<kF16>(sc[nt], qa[ks], ld_u32(k0), ld_u32(k0 + 8));
      }
    }
    // mask (prefix for all, block keys causally, nothing past T), scale, row max
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = kb + nt * 8 + 2 * tq + (e & 1);
        const int hh = e >> 1;
        const bool vis = (hh ? okB : okA) && t < T && (t < P || t - P <= (hh ? jB : jA));
        const float v = vis ? sc[nt][e] * p.scale_log2 : -INFINITY;
        sc[nt][e] = v;
        mx[hh] = fmaxf(mx[hh], v);
      }
    }
    float mu[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 1));
      mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 2));
      const float mn = fmaxf(m[hh], mx[hh]);
      mu[hh] = mn == -INFINITY ? 0.f : mn;        // no visible key yet: nothing to scale
      const float alpha = exp2f(m[hh] - mu[hh]);
      m[hh] = mn;
      l[hh] *= alpha;
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) {
        o[nd][2 * hh] *= alpha;
        o[nd][2 * hh + 1] *= alpha;
      }
    }
#pragma unroll
    for (int kk = 0; kk < kSub / 16; ++kk) {
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
        const uint16_t* v0 = Vt + (nd * 8 + g) * VS + st * kSub + kk * 16 + 2 * tq;
        const uint32_t b0 = ld_u32(v0), b1 = ld_u32(v0 + 8);
        mma_16816<kF16>(o[nd], ah, b0, b1);
        mma_16816<kF16>(o[nd], al, b0, b1);
      }
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
    if (tq == 0) pml[lA] = make_float2(m[0], l[0]);
  }
  if (okB) {
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd)
      *reinterpret_cast<float2*>(po + lB * D + nd * 8 + 2 * tq) = make_float2(o[nd][2], o[nd][3]);
    if (tq == 0) pml[lB] = make_float2(m[1], l[1]);
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
  for (int c = 0; c < nc; ++c) mmax = fmaxf(mmax, p.part_ml[(part0 + c) * kAttnRows + lr].x);
  float acc = 0.f, den = 0.f;
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
  if ((long long)Hkv * row_groups > 65535 || B > 65535 || (long long)L * Hq > 0x7fffffffll)
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

template <bool kF16, int D>
int attn_launch(const AttnParams& p, int B, cudaStream_t stream) {
  const size_t smem = (size_t)(kAttnRows + kChunk) * (D + 8) * 2 + (size_t)D * (kChunk + 8) * 2 +
                      (size_t)p.L * p.rot_half * sizeof(float2);
  auto* partial = verify_attn_partial_kernel<kF16, D>;
  if (ensure_smem<verify_attn_partial_kernel<kF16, D>>(smem) != VQ_OK) return VQ_ECUDA;
  partial<<<dim3(p.NC, p.Hkv * p.RG, B), kAttnThreads, smem, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return VQ_ECUDA;
  // the merge may be scheduled while the partial kernel runs; it waits for it
  // (griddepcontrol.wait) before reading anything
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.L * p.Hq, B);
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, verify_attn_combine_kernel<kF16, D>, p) != cudaSuccess)
    return VQ_ECUDA;
  return VQ_OK;
}

}  // namespace
}  // namespace vq

using namespace vq;

extern "C" size_t verify_attention_workspace_bytes(int B, int L, int Hq, int Hkv, int D,
                                                   int S_cap) {
  if (B < 1 || L < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 1 || S_cap < 1) return 0;
  const AttnShape s = attn_shape(L, Hq, Hkv, S_cap);
  const size_t rows = attn_part_count(B, Hkv, s);
  return rows * (size_t)D * sizeof(float) + rows * sizeof(float2);
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
