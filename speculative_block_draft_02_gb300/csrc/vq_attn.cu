// Verify-block attention over the per-row KV cache (verify_attention).
//
// mlxcel #2865 "perf(speculative): commit per-row accepts in batched DFlash",
// Summary and commit message: once every batch row keeps its own accept count,
// the rotary embedding and the attention of the verify block use every row's
// own logical positions, and no query sees the stale gap between its row's
// valid prefix and the verify slots the rectangular cache shares across rows.
//
// Three kernels per call:
//   verify_attn_rope_kernel  one block per (block position j, batch row): the
//       (cos, sin) of the row's logical position P + j once, then the position's
//       queries rotated and rounded to the storage type into the workspace, its
//       keys rotated into cache slot S + j and its values copied to slot S + j.
//   verify_attn_partial_kernel  one block per (key chunk of 64, KV head, group
//       of 64 query rows, batch row). It stages the group's rotated queries and
//       the chunk's keys and values (prefix slots, then the block's slots) in
//       shared memory, every load requested before any is waited for, then four
//       warps of 16 query rows each run S = Q K^T and O = P V on mma.sync
//       m16n8k16 with the softmax in fp32. For bf16, P is split into a 16-bit
//       high part and a 16-bit remainder so that the probabilities keep about
//       16 significant bits through the tensor cores. It writes the chunk's
//       unnormalised output and its (max, sum) per row to the workspace.
//   verify_attn_combine_kernel  merges the chunks of every query row and writes
//       the 16-bit output.
// 52 KB of shared memory and at most 128 registers a thread let four partial
// blocks share an SM. The partial and the merge kernels are launched with
// programmatic stream serialization: each may be scheduled while the kernel
// before it runs and waits for it (griddepcontrol.wait) before reading what it
// wrote; the partial kernel requests the prefix keys and values, which the
// rotation kernel does not write, before that wait.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "vq_common.cuh"

namespace vq {
namespace {

constexpr int kAttnThreads = 128;  // four warps of 16 query rows
constexpr int kAttnRows = 64;      // query rows per block
constexpr int kChunk = 64;         // keys per block (two threads per key when staging V)
constexpr int kMaxRotPairs = 64;   // rotary_dim / 2 for D <= 128
constexpr int kMaxBlock = 64;      // largest verify block L
constexpr int kMaxCap = 1 << 24;   // positions stay exact in fp32

constexpr int kRopeThreads = 256;
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
  int32_t* err;     // the library's status word (a wait that gave up)
  float* part_o;    // [B][Hkv][RG][NC][64][D]   unnormalised chunk outputs
  float2* part_ml;  // [B][Hkv][RG][NC][64]      (max in log2 units, sum)
  uint16_t* q_rot;  // [B][Hkv][RG][64][D] rotated, rounded queries, one swizzled tile
                    // per (row, KV head, group of 64 query rows) (sw_off layout)
  size_t cache_elems, out_elems, part_rows, qrot_bytes;   // extents (bounds-checked builds)
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

// 16 bytes global -> shared (at a shared-space address) without a register
// round trip; zeros when !valid (nothing is read then).
__device__ __forceinline__ void cp_async_16s(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}

__device__ __forceinline__ void sts128_zero(uint32_t addr) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Byte offset of element (row, col) of a [64 rows][D] 16-bit tile kept as D/64
// segments of [64 rows][128 B] in the 128-byte swizzle (the layout a 2-D TMA
// box of 64 x 64 values with SWIZZLE_128B lands in): 16-byte piece c of a
// segment's row r sits at piece c ^ (r % 8). col is a multiple of 8.
__device__ __forceinline__ uint32_t sw_off(int row, int col) {
  return (uint32_t)((col >> 6) * 8192 + row * 128 + ((((col >> 3) & 7) ^ (row & 7)) << 4));
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

// One block per (block position j, batch row). Rows of the position: the Hq
// query heads (rotated into the workspace), the Hkv key heads (rotated into
// cache slot S + j) and the Hkv value heads (copied to slot S + j); dimensions
// past rotary_dim are copied unchanged. Up to 64 rows at a time go through
// shared memory: all of their 16-byte loads are requested together, the
// pairs are turned in place, then the rows are stored in 16-byte pieces.
template <bool kF16, int D>
__global__ void __launch_bounds__(kRopeThreads)
    verify_attn_rope_kernel(const __grid_constant__ AttnParams p) {
  constexpr int RP = 64;       // rows per pass
  constexpr int DC = D / 8;    // 16-byte pieces per row
  __shared__ float2 cs[kMaxRotPairs];
  __shared__ __align__(16) uint16_t tile[RP * D];
  grid_launch_dependents();    // the partial kernel may be scheduled; it waits for this one
  const int j = blockIdx.x, b = blockIdx.y;
  const int P = p.prefix_len[b], S = p.src_off[b];
  if (!row_in_range(P, S, p.L, p.S_cap)) return;   // flagged by the combine kernel
  const int rh = p.rot_half;
  const int tid = threadIdx.x;
  // row r of the position: where it comes from and where it goes
  auto row_src = [&](int r) -> const uint16_t* {
    if (r < p.Hq) return p.q + (((size_t)b * p.L + j) * p.Hq + r) * D;
    if (r < p.Hq + p.Hkv) return p.k_new + (((size_t)b * p.L + j) * p.Hkv + (r - p.Hq)) * D;
    return p.v_new + (((size_t)b * p.L + j) * p.Hkv + (r - p.Hq - p.Hkv)) * D;
  };
  // key and value rows go to cache slot S + j; query head hq to row
  // rr = j * G + (hq - hk * G) of its group's tile
  auto row_dst = [&](int r) -> uint16_t* {
    const int h = r < p.Hq + p.Hkv ? r - p.Hq : r - p.Hq - p.Hkv;
    uint16_t* cache = r < p.Hq + p.Hkv ? p.k_cache : p.v_cache;
    return cache + (((size_t)b * p.Hkv + h) * p.S_cap + (S + j)) * D;
  };
  const int rows = p.Hq + 2 * p.Hkv, n_rot = p.Hq + p.Hkv;
  for (int r0 = 0; r0 < rows; r0 += RP) {
    const int nr = min(RP, rows - r0);
    if (r0 > 0) __syncthreads();   // the previous pass has stored its rows
#pragma unroll 4
    for (int i = tid; i < nr * DC; i += kRopeThreads) {
      const int rl = i / DC, c = i - rl * DC;
      *reinterpret_cast<uint4*>(tile + rl * D + c * 8) =
          __ldg(reinterpret_cast<const uint4*>(row_src(r0 + rl)) + c);
    }
    // the angles of the position, while the first rows are in flight
    if (r0 == 0)
      for (int e = tid; e < rh; e += kRopeThreads) cs[e] = rope_cos_sin((float)(P + j), p.inv_freq[e]);
    __syncthreads();
    const int nrot = max(0, min(nr, n_rot - r0));   // rows of this pass that turn
    for (int i = tid; i < nrot * rh; i += kRopeThreads) {
      const int rl = i / rh, e = i - rl * rh;
      uint16_t* row = tile + rl * D;
      const float x1 = h2f<kF16>(row[e]), x2 = h2f<kF16>(row[e + rh]);
      row[e] = f2h<kF16>(x1 * cs[e].x - x2 * cs[e].y);
      row[e + rh] = f2h<kF16>(x2 * cs[e].x + x1 * cs[e].y);
    }
    __syncthreads();
    for (int i = tid; i < nr * DC; i += kRopeThreads) {
      const int rl = i / DC, c = i - rl * DC;
      const int r = r0 + rl;
      const uint4 v = *reinterpret_cast<const uint4*>(tile + rl * D + c * 8);
      if (r < p.Hq) {
        const int hk = r / p.G, rr = j * p.G + (r - hk * p.G);
        const int rg = rr / kAttnRows, row = rr - rg * kAttnRows;
        const size_t off = (((size_t)b * p.Hkv + hk) * p.RG + rg) * (size_t)(kAttnRows * D * 2) +
                           sw_off(row, c * 8);
        if (in_bounds(off, p.qrot_bytes, p.err))
          *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.q_rot) + off) = v;
      } else {
        uint16_t* d = row_dst(r) + c * 8;
        if (in_bounds((size_t)(d - (r < p.Hq + p.Hkv ? p.k_cache : p.v_cache)), p.cache_elems, p.err))
          *reinterpret_cast<uint4*>(d) = v;
      }
    }
  }
}

// A bounded wait on phase 0 of an mbarrier: false after about a second.
__device__ __forceinline__ bool attn_wait(uint32_t bar) {
  if (mbar_try_wait(bar, 0u)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, 0u))
    if (clock64() - t0 > kWaitTimeoutCycles) return false;
  return true;
}

template <bool kF16, int D>
__global__ void __launch_bounds__(kAttnThreads, 4)
    verify_attn_partial_kernel(const __grid_constant__ CUtensorMap tm_k,
                               const __grid_constant__ CUtensorMap tm_v,
                               const __grid_constant__ AttnParams p) {
  constexpr uint32_t TILE = kAttnRows * D * 2;   // bytes of a 64-row tile
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t Qs = (raw + 1023u) & ~1023u;   // the swizzle wants 1 KiB-aligned tiles
  const uint32_t Ks = Qs + TILE, Vs = Qs + 2 * TILE;
  const uint32_t bar_pre = Qs + 3 * TILE, bar_rest = bar_pre + 8u;

  const int chunk = blockIdx.x;
  const int hk = blockIdx.y / p.RG, rg = blockIdx.y % p.RG;
  const int b = blockIdx.z;
  const int P = p.prefix_len[b], S = p.src_off[b];
  if (!row_in_range(P, S, p.L, p.S_cap)) return;   // flagged by the combine kernel
  const int T = P + p.L;                            // visible keys of the last query
  const int c0 = chunk * kChunk;
  if (c0 >= T) return;
  const int tid = threadIdx.x;
  grid_launch_dependents();   // the merge may be scheduled; it waits for this kernel
  if (tid == 0) {
    mbar_init(bar_pre, 1);
    mbar_init(bar_rest, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Key tl of the chunk (t = c0 + tl) sits in cache slot t below P and in slot
  // S + (t - P) from P on. The chunk's rows from slot c0 on arrive as 2-D TMA
  // boxes of 64 rows x 64 values (two per tile at D = 128), requested before
  // the wait for the rotation kernel (which writes only slots S.. and the
  // rotated queries; everything before it in the stream had completed when it
  // started); that is the whole chunk when it lies in the prefix. In a chunk
  // that reaches the block, the rows from P on are then replaced, once the
  // boxes have landed: the block's keys and values (slots S..) 16 bytes at a
  // time into the same swizzled layout, zeros past T. The group's rotated
  // queries are one tile of the workspace: one bulk copy after the wait.
  const bool whole = c0 + kChunk <= P;
  const int n_pre = max(0, min(P - c0, kChunk));   // prefix rows: tl < n_pre
  const int n_vis = min(T - c0, kChunk);           // visible rows: tl < n_vis
  const size_t head = ((size_t)b * p.Hkv + hk) * p.S_cap;
  if (tid == 0) {
    if (n_pre > 0) {
      mbar_arrive_expect_tx(bar_pre, 2u * TILE);
#pragma unroll
      for (int sg = 0; sg < D / 64; ++sg) {
        tma_load_2d(Ks + sg * 8192, &tm_k, sg * 64, (int)(head + c0), bar_pre);
        tma_load_2d(Vs + sg * 8192, &tm_v, sg * 64, (int)(head + c0), bar_pre);
      }
    } else {
      mbar_arrive(bar_pre);
    }
  }
  grid_wait_prerequisites();
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_rest, TILE);
    bulk_load(Qs,
              reinterpret_cast<const uint8_t*>(p.q_rot) +
                  (((size_t)b * p.Hkv + hk) * p.RG + rg) * (size_t)TILE,
              TILE, bar_rest);
  }
  bool ok = true;
  if (!whole) {
    ok = attn_wait(bar_pre);   // the boxes' rows past n_pre are replaced next
    if (ok) {
      for (int i = tid; i < (n_vis - n_pre) * (D / 8); i += kAttnThreads) {
        const int tl = n_pre + i / (D / 8), c = i % (D / 8);
        const size_t slot = head + (size_t)(S + (c0 + tl - P));
        const uint32_t o = sw_off(tl, c * 8);
        const bool in = in_bounds(slot * D + c * 8, p.cache_elems, p.err);
        cp_async_16s(Ks + o, p.k_cache + (in ? slot * D + c * 8 : 0), in);
        cp_async_16s(Vs + o, p.v_cache + (in ? slot * D + c * 8 : 0), in);
      }
      for (int i = tid; i < (kChunk - n_vis) * (D / 8); i += kAttnThreads) {
        const int tl = n_vis + i / (D / 8), c = i % (D / 8);
        const uint32_t o = sw_off(tl, c * 8);
        sts128_zero(Ks + o);
        sts128_zero(Vs + o);
      }
      cp_async_wait_all();
    }
  }
  if (!ok || !attn_wait(bar_pre) || !attn_wait(bar_rest)) {
    // give up: report it, let the copies already issued land, and leave
    if (tid == 0) atomicOr(p.err, kErrWaitTimeout);
    attn_wait(bar_pre);
    attn_wait(bar_rest);
    return;
  }
  __syncthreads();   // the gathered rows too

  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, tq = lane & 3;
  const int row0 = warp * 16;
  const int rA = rg * kAttnRows + row0 + g, rB = rA + 8;   // rows of c0/c1 and c2/c3
  if (rg * kAttnRows + row0 >= p.R) return;               // no barrier follows
  const bool okA = rA < p.R, okB = rB < p.R;
  const int jA = rA / p.G, jB = rB / p.G;

  // S = Q K^T: A fragments of the warp's 16 query rows, B fragments of two
  // 8-key tiles per ldmatrix.x4
  float sc[8][4];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
  const int qa_row = row0 + (lane & 15), qa_col = (lane >> 4) * 8;
  const int kb_row = (lane & 7) + ((lane >> 4) << 3), kb_col = ((lane >> 3) & 1) * 8;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    uint32_t qa[4];
    ldsm_x4(qa, Qs + sw_off(qa_row, ks * 16 + qa_col));
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      uint32_t kb[4];
      ldsm_x4(kb, Ks + sw_off(np * 16 + kb_row, ks * 16 + kb_col));
      mma_16816<kF16>(sc[2 * np], qa, kb[0], kb[1]);
      mma_16816<kF16>(sc[2 * np + 1], qa, kb[2], kb[3]);
    }
  }
  // mask (prefix for all, block keys causally, nothing past T), scale, row max;
  // a chunk wholly in the prefix is visible to every row
  float m[2] = {-INFINITY, -INFINITY};
  if (c0 + kChunk <= P) {
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sc[nt][e] *= p.scale_log2;
        m[e >> 1] = fmaxf(m[e >> 1], sc[nt][e]);
      }
  } else {
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = c0 + nt * 8 + 2 * tq + (e & 1);
        const int hh = e >> 1;
        const bool vis = (hh ? okB : okA) && t < T && (t < P || t - P <= (hh ? jB : jA));
        const float v = vis ? sc[nt][e] * p.scale_log2 : -INFINITY;
        sc[nt][e] = v;
        m[hh] = fmaxf(m[hh], v);
      }
    }
  }
  float mu[2], l[2] = {0.f, 0.f};
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    m[hh] = fmaxf(m[hh], __shfl_xor_sync(0xffffffffu, m[hh], 1));
    m[hh] = fmaxf(m[hh], __shfl_xor_sync(0xffffffffu, m[hh], 2));
    mu[hh] = m[hh] == -INFINITY ? 0.f : m[hh];   // no visible key in the chunk: every p is 0
  }
  float o[D / 8][4];
#pragma unroll
  for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  // O = P V: P as 16-bit MMA operands. bf16 keeps 8 significant bits, which
  // would move the outputs by up to 2^-9 relative, so there P is split into a
  // high part and the remainder (two MMAs, about 16 bits); fp16's 11 bits
  // suffice alone. B fragments of two 8-dimension tiles per ldmatrix.x4.trans.
  const int vb_row = (lane & 7) + ((lane >> 3) & 1) * 8, vb_col = (lane >> 4) * 8;
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
      if constexpr (kF16) {
        ah[2 * half] = (uint32_t)f2h<true>(p0) | ((uint32_t)f2h<true>(p1) << 16);
        ah[2 * half + 1] = (uint32_t)f2h<true>(p2) | ((uint32_t)f2h<true>(p3) << 16);
      } else {
        split_pair<false>(p0, p1, ah[2 * half], al[2 * half]);
        split_pair<false>(p2, p3, ah[2 * half + 1], al[2 * half + 1]);
      }
    }
#pragma unroll
    for (int np = 0; np < D / 16; ++np) {
      uint32_t vb[4];
      ldsm_x4_t(vb, Vs + sw_off(kk * 16 + vb_row, np * 16 + vb_col));
      mma_16816<kF16>(o[2 * np], ah, vb[0], vb[1]);
      mma_16816<kF16>(o[2 * np + 1], ah, vb[2], vb[3]);
      if constexpr (!kF16) {
        mma_16816<kF16>(o[2 * np], al, vb[0], vb[1]);
        mma_16816<kF16>(o[2 * np + 1], al, vb[2], vb[3]);
      }
    }
  }
  for (int hh = 0; hh < 2; ++hh) {
    l[hh] += __shfl_xor_sync(0xffffffffu, l[hh], 1);
    l[hh] += __shfl_xor_sync(0xffffffffu, l[hh], 2);
  }
  const size_t part = (((size_t)b * p.Hkv + hk) * p.RG + rg) * p.NC + chunk;
  float* po = p.part_o + part * kAttnRows * D;
  float2* pml = p.part_ml + part * kAttnRows;
  const int lA = row0 + g, lB = lA + 8;
  const bool stA = okA && in_bounds(part * kAttnRows + lA, p.part_rows, p.err);
  const bool stB = okB && in_bounds(part * kAttnRows + lB, p.part_rows, p.err);
  if (stA) {
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd)
      *reinterpret_cast<float2*>(po + lA * D + nd * 8 + 2 * tq) = make_float2(o[nd][0], o[nd][1]);
    if (tq == 0) pml[lA] = make_float2(m[0], l[0]);
  }
  if (stB) {
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd)
      *reinterpret_cast<float2*>(po + lB * D + nd * 8 + 2 * tq) = make_float2(o[nd][2], o[nd][3]);
    if (tq == 0) pml[lB] = make_float2(m[1], l[1]);
  }
}

// One block per (block position j, query head, batch row), D threads. Lane l of
// every warp covers dimensions VEC*l .. VEC*l + VEC-1; warp w takes chunks w,
// w + NW, ... so that all of a row's chunks are requested at once; the warps'
// sums are then added in warp order (a fixed order: the result does not depend
// on timing).
template <bool kF16, int D>
__global__ void __launch_bounds__(D) verify_attn_combine_kernel(const __grid_constant__ AttnParams p) {
  constexpr int NW = D / 32, VEC = D / 32;
  const int jh = blockIdx.x, b = blockIdx.y;
  const int j = jh / p.Hq, hq = jh - j * p.Hq;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  grid_wait_prerequisites();   // launched early (programmatic serialization)
  const size_t dst_off = (((size_t)b * p.L + j) * p.Hq + hq) * D;
  if (!in_bounds(dst_off + D - 1, p.out_elems, p.err)) return;
  uint16_t* dst = p.out + dst_off;
  const int P = p.prefix_len[b], S = p.src_off[b];
  if (!row_in_range(P, S, p.L, p.S_cap)) {
    dst[tid] = 0;
    if (jh == 0 && tid == 0 && p.status) atomicOr(p.status, 1);
    return;
  }
  const int nc = (P + p.L + kChunk - 1) / kChunk;
  const int hk = hq / p.G, rr = j * p.G + (hq - hk * p.G);
  const int rg = rr / kAttnRows, lr = rr - rg * kAttnRows;
  const size_t part0 = (((size_t)b * p.Hkv + hk) * p.RG + rg) * p.NC;
  const float2* ml = p.part_ml + part0 * kAttnRows + lr;                    // chunk c at ml[c * 64]
  const float* po = p.part_o + (part0 * kAttnRows + lr) * D + VEC * lane;   // at po[c * 64 * D]
  // the chunks' maxima: strided over the threads, then over the block; every
  // query sees its own key, so some chunk has a finite maximum
  __shared__ float red_m[NW];
  __shared__ float red_s[NW][VEC * 32 + 1];   // each warp's sums, then its denominator
  float mx = -INFINITY;
  for (int c = tid; c < nc; c += D) mx = fmaxf(mx, ml[(size_t)c * kAttnRows].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red_m[w] = mx;
  __syncthreads();
  float mmax = red_m[0];
#pragma unroll
  for (int i = 1; i < NW; ++i) mmax = fmaxf(mmax, red_m[i]);
  float acc[VEC], den = 0.f;
#pragma unroll
  for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
#pragma unroll 4
  for (int c = w; c < nc; c += NW) {
    const float2 mc = ml[(size_t)c * kAttnRows];
    const float* src = po + (size_t)c * kAttnRows * D;
    float x[VEC];
    if constexpr (VEC == 4) {
      const float4 t = *reinterpret_cast<const float4*>(src);
      x[0] = t.x;
      x[1] = t.y;
      x[2] = t.z;
      x[3] = t.w;
    } else {
      const float2 t = *reinterpret_cast<const float2*>(src);
      x[0] = t.x;
      x[1] = t.y;
    }
    const float wt = exp2f(mc.x - mmax);
    den += wt * mc.y;
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[v] += wt * x[v];
  }
#pragma unroll
  for (int v = 0; v < VEC; ++v) red_s[w][VEC * lane + v] = acc[v];
  if (lane == 0) red_s[w][VEC * 32] = den;
  __syncthreads();
  // thread tid writes dimension tid: the warps' sums in warp order
  float o = red_s[0][tid], dsum = red_s[0][VEC * 32];
#pragma unroll
  for (int i = 1; i < NW; ++i) {
    o += red_s[i][tid];
    dsum += red_s[i][VEC * 32];
  }
  dst[tid] = f2h<kF16>(o / dsum);
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
  // (the cache rows are addressed by 32-bit TMA coordinates)
  if ((long long)Hkv * row_groups > 65535 || B > 65535 || (long long)L * Hq > 0x7fffffffll ||
      (long long)B * Hkv * S_cap > 0x7fffffffll)
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

// Byte offset of the rotated queries in the workspace (rows: partial-result rows).
size_t attn_qrot_offset(size_t rows, int D) {
  return (rows * (size_t)D * sizeof(float) + rows * sizeof(float2) + 15) / 16 * 16;
}

template <bool kF16, int D>
int attn_launch(const AttnParams& p, int B, cudaStream_t stream, const CUtensorMap& tm_k,
                const CUtensorMap& tm_v) {
  // three swizzled tiles (1 KiB-aligned) and two mbarriers
  const size_t smem = 1024 + (size_t)3 * kAttnRows * D * 2 + 16;
  auto* partial = verify_attn_partial_kernel<kF16, D>;
  if (ensure_smem<verify_attn_partial_kernel<kF16, D>>(smem) != VQ_OK) return VQ_ECUDA;
  // the rotation runs after everything before it in the stream; the partial
  // kernel may be scheduled while it runs and waits for it on the GPU
  verify_attn_rope_kernel<kF16, D><<<dim3(p.L, B), kRopeThreads, 0, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return VQ_ECUDA;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.NC, p.Hkv * p.RG, B);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, partial, tm_k, tm_v, p) != cudaSuccess) return VQ_ECUDA;
  }
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
  // [partial outputs][partial (max, sum)][rotated queries], each 16-byte aligned
  return attn_qrot_offset(rows, D) + (size_t)B * Hkv * s.RG * kAttnRows * D * sizeof(uint16_t);
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
  int32_t* err = nullptr;   // the device's status word (a usable current device)
  rc = device_error_word(&err);
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
  p.err = err;
  const size_t rows = attn_part_count(B, Hkv, s);
  p.part_o = static_cast<float*>(workspace);
  p.part_ml = reinterpret_cast<float2*>(static_cast<char*>(workspace) +
                                        rows * (size_t)D * sizeof(float));
  p.q_rot = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + attn_qrot_offset(rows, D));
  p.cache_elems = (size_t)B * Hkv * S_cap * D;
  p.out_elems = (size_t)B * L * Hq * D;
  p.part_rows = rows;
  p.qrot_bytes = (size_t)B * Hkv * s.RG * kAttnRows * D * sizeof(uint16_t);
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
  // the caches as rows of D values, boxes of 64 rows x 64 values (cached per
  // host thread, so a call on the same caches encodes nothing)
  CUtensorMap tm_k, tm_v;
  const uint64_t kv_rows = (uint64_t)B * Hkv * S_cap;
  if (encode_rows_sw128(&tm_k, k_cache, (uint64_t)D, kv_rows, kChunk) != VQ_OK ||
      encode_rows_sw128(&tm_v, v_cache, (uint64_t)D, kv_rows, kChunk) != VQ_OK)
    return VQ_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == VQ_F16)
    return D == 64 ? attn_launch<true, 64>(p, B, st, tm_k, tm_v)
                   : attn_launch<true, 128>(p, B, st, tm_k, tm_v);
  return D == 64 ? attn_launch<false, 64>(p, B, st, tm_k, tm_v)
                 : attn_launch<false, 128>(p, B, st, tm_k, tm_v);
}
