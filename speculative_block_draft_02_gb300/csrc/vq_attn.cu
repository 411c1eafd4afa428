// Verify-block attention over the per-row KV cache (verify_attention).
//
// mlxcel #2865 "perf(speculative): commit per-row accepts in batched DFlash",
// Summary and commit message: once every batch row keeps its own accept count,
// the rotary embedding and the attention of the verify block use every row's
// own logical positions, and no query sees the stale gap between its row's
// valid prefix and the verify slots the rectangular cache shares across rows.
//
// One kernel per call, launched in clusters of kCluster blocks: one cluster per
// (batch row b, KV head hk, group of 64 query rows). Query row rr of a group is
// (block position j, query head hq) with rr = j * G + (hq - hk * G).
//   - Logical key t of the row is cache slot t below P and the block's key
//     t - P from P on (slot S + t - P once appended). Block r of the cluster
//     takes the row's chunks of 64 keys r, r + kCluster, ...: the prefix rows
//     of a chunk arrive as 2-D TMA boxes in a two-deep ring, both stages
//     requested before anything else is done. The block's keys span at most
//     two consecutive chunks, so each block owns at most one of them: it
//     prefetches those rows of k_new and v_new at the start (up to 16 of
//     them), rotates the keys at P + j and, in row group 0, appends keys and
//     values to slots S + j of the caches there and then, and places them in
//     the chunk's tile when that chunk comes (more than 16 rows: loaded,
//     rotated and appended in the tile when the chunk comes).
//   - Meanwhile the block loads the group's queries, rotates them at P + j and
//     rounds them to the storage type (the (cos, sin) of up to 16 positions at
//     a time in a shared table, the frequencies staged in shared memory).
//   - Four warps of 16 query rows run S = Q K^T and O = P V on mma.sync
//     m16n8k16 over each chunk, with an online softmax in fp32. For bf16, P is
//     split into a 16-bit high part and the remainder, so that the
//     probabilities keep about 16 significant bits through the tensor cores.
//   - Each block leaves its (max, sum, unnormalised output) per query row in
//     its shared memory. After a cluster barrier, block r merges rows
//     8r .. 8r + 7 over the cluster's blocks in rank order (a fixed order),
//     reading its peers' shared memory, and writes the 16-bit output; a second
//     cluster barrier keeps every block resident until its peers have read it.
// No workspace. The launch is ordered after everything before it in the
// stream (the caches' prefixes may have been written just before).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "vq_common.cuh"

namespace vq {
namespace {

constexpr int kAttnThreads = 128;  // four warps of 16 query rows
constexpr int kAttnRows = 64;      // query rows per cluster
constexpr int kChunk = 64;         // keys per chunk
constexpr int kCluster = 8;        // blocks per cluster (portable size)
constexpr int kMergeRows = kAttnRows / kCluster;
constexpr int kAppRows = 16;       // block rows a block prefetches for its boundary chunk
constexpr int kMaxRotPairs = 64;   // rotary_dim / 2 for D <= 128
constexpr int kTabPos = 16;        // positions per (cos, sin) table pass
constexpr int kMaxBlock = 64;      // largest verify block L
constexpr int kMaxCap = 1 << 24;   // positions stay exact in fp32
static_assert(kMergeRows * 16 == kAttnThreads, "sixteen threads per merged row");
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
  int32_t* err;                      // the library's status word (a wait that gave up)
  size_t cache_elems, out_elems;     // extents (bounds-checked builds)
  int L, Hq, Hkv, G, R, RG, S_cap, rot_half;
  int out_vec;                       // out is 16-byte aligned: vector stores
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

__device__ __forceinline__ void sts64f(uint32_t a, float x, float y) {
  asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(x), "f"(y) : "memory");
}

__device__ __forceinline__ float2 lds64f(uint32_t a) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ uint16_t lds16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ void sts16(uint32_t a, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"(v) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a)
               : "memory");
  return v;
}

// 16 bytes global -> shared without a register round trip; zeros when !valid
// (nothing is read then). Completed by cp_async_wait_all.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Orders this thread's generic-proxy accesses of shared memory before later
// async-proxy (TMA) writes to it.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every block of the cluster: shared-memory writes before it
// are visible to the whole cluster after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// The two halves of a cluster barrier: an arrival that orders nothing, and a
// wait (with acquire) for every thread of the cluster to have arrived.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// The address of the same shared-memory location in block `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_peer_v4(uint32_t a, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_peer_f2(uint32_t a, float x, float y) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(x), "f"(y) : "memory");
}

// Byte offset of element (row, col) of a [64 rows][D] 16-bit tile kept as D/64
// segments of [64 rows][128 B] in the 128-byte swizzle (the layout a 2-D TMA
// box of 64 x 64 values with SWIZZLE_128B lands in): 16-byte piece c of a
// segment's row r sits at piece c ^ (r % 8). col is a multiple of 8.
__device__ __forceinline__ uint32_t sw_off(int row, int col) {
  return (uint32_t)((col >> 6) * 8192 + row * 128 + ((((col >> 3) & 7) ^ (row & 7)) << 4));
}

// The same for any column (one 16-bit element).
__device__ __forceinline__ uint32_t el_off(int row, int col) {
  return sw_off(row, col & ~7) + (uint32_t)(col & 7) * 2u;
}

__device__ __forceinline__ bool row_in_range(int P, int S, int L, int S_cap) {
  return P >= 0 && S >= P && (long long)S + L <= (long long)S_cap;
}

// (cos, sin) of pos * f for f = hi + lo: the angle is formed as a + err with
// a = fl(pos * hi) and err the rest of pos * (hi + lo), then turned to first
// order: sin(a + err) ~ sin a + err cos a (|err| < 1e-3 rad). Every rounding
// is spelled out, so that the same position gives the same bits everywhere.
__device__ __forceinline__ float2 rope_cos_sin(float pos, float2 f) {
  const float a = __fmul_rn(pos, f.x);
  const float err = __fadd_rn(__fmaf_rn(pos, f.x, -a), __fmul_rn(pos, f.y));
  float s, c;
  sincosf(a, &s, &c);
  return make_float2(__fmaf_rn(-err, s, c), __fmaf_rn(err, c, s));
}

// The pair (x1, x2) turned by the angle of cs = (cos, sin), each result with
// one rounded product and one fused multiply-add, spelled out so that every
// place that rotates a key gets the same bits.
__device__ __forceinline__ void rot_pair(float x1, float x2, float2 cs, float& r1, float& r2) {
  r1 = __fmaf_rn(x1, cs.x, -__fmul_rn(x2, cs.y));
  r2 = __fmaf_rn(x2, cs.x, __fmul_rn(x1, cs.y));
}

__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Eight consecutive pairs of a row: dimensions e0 .. e0 + 7 (16 bytes at
// shared address a1) with their partners e0 + rh .. (16 bytes at a2), turned
// by cs[k] = (cos, sin) of pair e0 + k and rounded to the storage type in place.
// Two 16-bit values (low, high) as floats, and two floats rounded into one word.
template <bool kF16>
__device__ __forceinline__ float2 h2f2(uint32_t w) {
  if constexpr (kF16) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  } else {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  }
}

template <bool kF16>
__device__ __forceinline__ uint32_t f2h2(float lo, float hi) {
  if constexpr (kF16) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

// Eight consecutive pairs of a row: dimensions e0 .. e0 + 7 (16 bytes at
// shared address a1) with their partners e0 + rh .. (16 bytes at a2), turned
// by cs[k] = (cos, sin) of pair e0 + k and rounded to the storage type in place.
template <bool kF16>
__device__ __forceinline__ void rot8(uint32_t a1, uint32_t a2, const float2 (&cs)[8]) {
  const uint4 x1 = lds128(a1), x2 = lds128(a2);
  const uint32_t w1[4] = {x1.x, x1.y, x1.z, x1.w}, w2[4] = {x2.x, x2.y, x2.z, x2.w};
  uint32_t o1[4], o2[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 u = h2f2<kF16>(w1[k]), v = h2f2<kF16>(w2[k]);
    float r1a, r2a, r1b, r2b;
    rot_pair(u.x, v.x, cs[2 * k], r1a, r2a);
    rot_pair(u.y, v.y, cs[2 * k + 1], r1b, r2b);
    o1[k] = f2h2<kF16>(r1a, r1b);
    o2[k] = f2h2<kF16>(r2a, r2b);
  }
  sts128(a1, make_uint4(o1[0], o1[1], o1[2], o1[3]));
  sts128(a2, make_uint4(o2[0], o2[1], o2[2], o2[3]));
}

// A bounded wait on an mbarrier phase: false after about a second.
__device__ __forceinline__ bool attn_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitTimeoutCycles) return false;
  return true;
}

// Shared memory of a block (offsets from a 1 KiB-aligned base; TILE = 64 rows
// of D 16-bit values): the rotated queries, then the ring's two stages of
// (keys, values), the (cos, sin) table of the prefetched block keys, those
// block rows of this block's boundary chunk (keys, then values, as given),
// the rotation frequencies, the (cos, sin) table of this block's query rows'
// positions and two mbarriers. Once every block of the cluster is done with its
// chunks, the ring receives the partial results the cluster's blocks send for
// this block's eight query rows, at [sender][row]: the unnormalised outputs
// [8][8][D + 4] fp32 (rows padded against bank conflicts), then (max, sum) [8][8].
template <int D>
struct AttnSmem {
  static constexpr uint32_t TILE = kAttnRows * D * 2;
  static constexpr uint32_t Q = 0, RING = TILE, TAB = 5 * TILE;
  static constexpr uint32_t APP = TAB + kTabPos * kMaxRotPairs * 8;
  static constexpr uint32_t FREQ = APP + 2 * kAppRows * D * 2;
  static constexpr uint32_t TABQ = FREQ + kMaxRotPairs * 8;
  static constexpr uint32_t BARS = TABQ + kMergeRows * kMaxRotPairs * 8;
  static constexpr uint32_t BYTES = BARS + 16;
  static constexpr uint32_t O_STRIDE = (D + 4) * 4;
  static constexpr uint32_t OM = RING, ML = RING + kAttnRows * O_STRIDE;
  static_assert(kAttnRows * O_STRIDE + kAttnRows * 8 <= 4 * TILE, "partials fit in the ring");
};

template <bool kF16, int D>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kAttnThreads, 2)
    verify_attn_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ AttnParams p) {
  using SM = AttnSmem<D>;
  constexpr uint32_t TILE = SM::TILE;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;   // the swizzle wants 1 KiB
  const uint32_t Qs = base + SM::Q, tab = base + SM::TAB, app = base + SM::APP;
  const uint32_t freq = base + SM::FREQ, tabq = base + SM::TABQ, bars = base + SM::BARS;

  const int tid = threadIdx.x;
  const uint32_t rank = cluster_rank();
  const int hk = blockIdx.y / p.RG, rg = blockIdx.y - hk * p.RG;
  const int b = blockIdx.z;
  const int rr0 = rg * kAttnRows;
  const int P = p.prefix_len[b], S = p.src_off[b];
  if (!row_in_range(P, S, p.L, p.S_cap)) {
    // the whole cluster leaves here (no barrier follows): zero output, flagged
    for (int i = tid; i < kMergeRows * D; i += kAttnThreads) {
      const int rr = rr0 + (int)rank * kMergeRows + i / D, d = i % D;
      if (rr < p.R) {
        const int j = rr / p.G, hq = hk * p.G + (rr - j * p.G);
        const size_t o = (((size_t)b * p.L + j) * p.Hq + hq) * D + d;
        if (in_bounds(o, p.out_elems, p.err)) p.out[o] = 0;
      }
    }
    if (rank == 0 && blockIdx.y == 0 && tid == 0 && p.status) atomicOr(p.status, 1);
    return;
  }
  const int T = P + p.L;   // visible keys of the last query
  const int n_chunks = (T + kChunk - 1) / kChunk;
  const int n_mine = (int)rank < n_chunks ? (n_chunks - 1 - (int)rank) / kCluster + 1 : 0;
  const size_t head = ((size_t)b * p.Hkv + hk) * p.S_cap;   // cache row of slot 0
  const int rh = p.rot_half;

  if (tid == 0) {
    mbar_init(bars, 1);
    mbar_init(bars + 8, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // thread 0: the prefix rows of chunk i of this block into stage i % 2 (the
  // whole box; rows from P on are replaced once it has landed)
  auto issue = [&](int i) {
    const int c0 = ((int)rank + i * kCluster) * kChunk;
    const uint32_t bar = bars + 8u * (uint32_t)(i & 1);
    const uint32_t Ks = base + SM::RING + (uint32_t)(i & 1) * 2u * TILE, Vs = Ks + TILE;
    if (c0 < P) {
      mbar_arrive_expect_tx(bar, 2u * TILE);
#pragma unroll
      for (int sg = 0; sg < D / 64; ++sg) {
        tma_load_2d(Ks + sg * 8192, &tm_k, sg * 64, (int)(head + c0), bar);
        tma_load_2d(Vs + sg * 8192, &tm_v, sg * 64, (int)(head + c0), bar);
      }
    } else {
      mbar_arrive(bar);
    }
  };
  if (tid == 0) {
    if (n_mine > 0) issue(0);
    if (n_mine > 1) issue(1);
  }

  // every block of the cluster has started once this barrier completes (before
  // the first write into a peer's shared memory)
  cluster_arrive_relaxed();
  // this block's eight query rows of the group (zeros past R)
  const int q0 = (int)rank * kMergeRows;   // local rows q0 .. q0 + 7
  for (int i = tid; i < kMergeRows * (D / 8); i += kAttnThreads) {
    const int lr = q0 + i / (D / 8), c = i % (D / 8);
    const int rr = rr0 + lr;
    const bool valid = rr < p.R;
    const int j = valid ? rr / p.G : 0, hq = valid ? hk * p.G + (rr - j * p.G) : 0;
    cp_async_16(Qs + sw_off(lr, c * 8), p.q + (((size_t)b * p.L + j) * p.Hq + hq) * D + c * 8,
                valid);
  }
  // the block rows jb0 .. jb1 - 1 of this block's boundary chunk (the block
  // keys span at most two consecutive chunks, so a block owns at most one),
  // prefetched when they fit
  int jb0 = 0, jb1 = 0;
  for (int ci = P / kChunk; ci * kChunk < T; ++ci)
    if (ci % kCluster == (int)rank) {
      jb0 = max(ci * kChunk, P) - P;
      jb1 = min(ci * kChunk + kChunk, T) - P;
    }
  const bool staged = jb1 - jb0 <= kAppRows;
  if (staged)
    for (int i = tid; i < (jb1 - jb0) * 2 * (D / 8); i += kAttnThreads) {
      const int a = i / (2 * (D / 8)), rem = i - a * (2 * (D / 8));
      const int kv = rem / (D / 8), c = rem - kv * (D / 8);
      cp_async_16(app + (uint32_t)((kv * kAppRows + a) * D * 2 + c * 16),
                  (kv ? p.v_new : p.k_new) + (((size_t)b * p.L + jb0 + a) * p.Hkv + hk) * D + c * 8,
                  true);
    }
  // while the copies land: the frequencies into shared memory, the (cos, sin)
  // of this block's query positions P + jq0 .. (at most eight) and of the
  // prefetched keys' positions P + jb0 ..; each thread keeps one frequency
  // (one read of the parameter array each)
  const bool vec8 = (rh & 7) == 0;
  const int npc = vec8 ? rh / 8 : rh;   // rotation steps per row
  const int tab_lo = jb0, tab_n = staged ? jb1 - jb0 : 0;
  const int q_end = min(p.R, rr0 + q0 + kMergeRows);   // this block's query rows: .. q_end - 1
  const int jq0 = (rr0 + q0) / p.G, nq = q_end > rr0 + q0 ? (q_end - 1) / p.G - jq0 + 1 : 0;
  const int tpe = rh > 0 ? kAttnThreads / rh : 0;   // threads per frequency (rh <= 64)
  if (tid < tpe * rh) {
    const int e = tid % rh, j0 = tid / rh;
    const float2 fq = p.inv_freq[e];
    if (j0 == 0) sts64f(freq + (uint32_t)e * 8u, fq.x, fq.y);
    for (int jj = j0; jj < nq; jj += tpe) {
      const float2 cs = rope_cos_sin((float)(P + jq0 + jj), fq);
      sts64f(tabq + (uint32_t)(jj * kMaxRotPairs + e) * 8u, cs.x, cs.y);
    }
    for (int jj = j0; jj < tab_n; jj += tpe) {
      const float2 cs = rope_cos_sin((float)(P + tab_lo + jj), fq);
      sts64f(tab + (uint32_t)(jj * kMaxRotPairs + e) * 8u, cs.x, cs.y);
    }
  }
  cp_async_wait_all();
  __syncthreads();
  // the eight rows rotated at P + j in place (eight pairs per step when rh is
  // a multiple of 8, else one), and after them the prefetched block keys at
  // P + jb0 + a in the staging rows (so that the chunk holding them only
  // copies them into its tile)
  const int nq_items = max(q_end - rr0 - q0, 0) * npc, nk_items = staged ? (jb1 - jb0) * npc : 0;
  if (rh > 0)
    for (int i = tid; i < nq_items + nk_items; i += kAttnThreads) {
      if (i >= nq_items) {
        const int a = (i - nq_items) / npc, u = (i - nq_items) - a * npc;
        const uint32_t row = app + (uint32_t)(a * D * 2);
        const uint32_t cs_row = tab + (uint32_t)(a * kMaxRotPairs) * 8u;
        if (vec8) {
          float2 cs[8];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint4 w = lds128(cs_row + (uint32_t)(8 * u + 2 * m) * 8u);
            cs[2 * m] = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
            cs[2 * m + 1] = make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
          }
          rot8<kF16>(row + 16u * (uint32_t)u, row + 2u * (uint32_t)(8 * u + rh), cs);
        } else {
          const uint32_t a1 = row + 2u * (uint32_t)u, a2 = row + 2u * (uint32_t)(u + rh);
          float r1, r2;
          rot_pair(h2f<kF16>(lds16(a1)), h2f<kF16>(lds16(a2)), lds64f(cs_row + (uint32_t)u * 8u),
                   r1, r2);
          sts16(a1, f2h<kF16>(r1));
          sts16(a2, f2h<kF16>(r2));
        }
        continue;
      }
      const int k = i / npc, u = i - k * npc;
      const int lr = q0 + k;
      const uint32_t cs_row = tabq + (uint32_t)(((rr0 + lr) / p.G - jq0) * kMaxRotPairs) * 8u;
      if (vec8) {
        float2 cs[8];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const uint4 w = lds128(cs_row + (uint32_t)(8 * u + 2 * m) * 8u);
          cs[2 * m] = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
          cs[2 * m + 1] = make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
        }
        rot8<kF16>(Qs + sw_off(lr, 8 * u), Qs + sw_off(lr, 8 * u + rh), cs);
      } else {
        const uint32_t a1 = Qs + el_off(lr, u), a2 = Qs + el_off(lr, u + rh);
        float r1, r2;
        rot_pair(h2f<kF16>(lds16(a1)), h2f<kF16>(lds16(a2)), lds64f(cs_row + (uint32_t)u * 8u), r1,
                 r2);
        sts16(a1, f2h<kF16>(r1));
        sts16(a2, f2h<kF16>(r2));
      }
    }
  __syncthreads();
  // row group 0 appends the prefetched block keys (rotated) and values to
  // slots S + jb0 .. of the caches: nothing in this call reads them back (the
  // chunk that holds those keys takes them from the staging rows; a box that
  // covers the slots is overwritten there)
  if (staged && rg == 0)
    for (int e = tid; e < (jb1 - jb0) * 2 * (D / 8); e += kAttnThreads) {
      const int a = e / (2 * (D / 8)), rem = e - a * (2 * (D / 8));
      const int kv = rem / (D / 8), c = rem - kv * (D / 8);
      const uint4 v = lds128(app + (uint32_t)((kv * kAppRows + a) * D * 2 + c * 16));
      const size_t dst = (head + (size_t)(S + jb0 + a)) * D + c * 8;
      if (in_bounds(dst + 7, p.cache_elems, p.err))
        *reinterpret_cast<uint4*>((kv ? p.v_cache : p.k_cache) + dst) = v;
    }
  // the eight rows into every other block's query tile (the same offsets)
  cluster_wait();
  for (int i = tid; i < (kCluster - 1) * kMergeRows * (D / 8); i += kAttnThreads) {
    const int c = i % (D / 8), lr = q0 + (i / (D / 8)) % kMergeRows;
    const uint32_t peer = ((uint32_t)(i / (kMergeRows * (D / 8))) + rank + 1u) % kCluster;
    const uint32_t off = Qs + sw_off(lr, c * 8);
    st_peer_v4(peer_addr(off, peer), lds128(off));
  }
  // (cos, sin) of pairs at block position j (position P + j): from the table
  // when it holds the position (the same bits as computing it)
  auto cs_one = [&](int j, int e) -> float2 {
    const int jj = j - tab_lo;
    if (jj >= 0 && jj < tab_n) return lds64f(tab + (uint32_t)(jj * kMaxRotPairs + e) * 8u);
    return rope_cos_sin((float)(P + j), lds64f(freq + (uint32_t)e * 8u));
  };
  auto cs_eight = [&](int j, int e0, float2 (&cs)[8]) {
    const int jj = j - tab_lo;
    if (jj >= 0 && jj < tab_n) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 w = lds128(tab + (uint32_t)(jj * kMaxRotPairs + e0 + 2 * k) * 8u);
        cs[2 * k] = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
        cs[2 * k + 1] = make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        cs[k] = rope_cos_sin((float)(P + j), lds64f(freq + (uint32_t)(e0 + k) * 8u));
    }
  };
  // block key row at shared address row (16-bit values, dimension d at
  // row_at(d)) of block position j: step u of its rotation
  auto rot_key_step = [&](int j, int u, uint32_t a_lo, uint32_t a_hi) {
    if (vec8) {
      float2 cs[8];
      cs_eight(j, 8 * u, cs);
      rot8<kF16>(a_lo, a_hi, cs);
    } else {
      float r1, r2;
      rot_pair(h2f<kF16>(lds16(a_lo)), h2f<kF16>(lds16(a_hi)), cs_one(j, u), r1, r2);
      sts16(a_lo, f2h<kF16>(r1));
      sts16(a_hi, f2h<kF16>(r2));
    }
  };

  cluster_sync_all();   // every block's query tile is complete

  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, tq = lane & 3;
  const int row0 = warp * 16;
  const int rA = rr0 + row0 + g, rB = rA + 8;   // rows of c0/c1 and c2/c3
  const bool live = rr0 + row0 < p.R;           // the warp has query rows
  // the last visible key of each of the thread's two rows (-1: past R)
  const int limA = rA < p.R ? P + rA / p.G : -1, limB = rB < p.R ? P + rB / p.G : -1;
  const int qa_row = row0 + (lane & 15), qa_col = (lane >> 4) * 8;
  const int kb_row = (lane & 7) + ((lane >> 4) << 3), kb_col = ((lane >> 3) & 1) * 8;
  const int vb_row = (lane & 7) + ((lane >> 3) & 1) * 8, vb_col = (lane >> 4) * 8;

  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[D / 8][4];
#pragma unroll
  for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;

  bool ok = true;
  int done = 0;   // chunks consumed
  for (; done < n_mine; ++done) {
    const int i = done;
    const uint32_t Ks = base + SM::RING + (uint32_t)(i & 1) * 2u * TILE, Vs = Ks + TILE;
    const int c0 = ((int)rank + i * kCluster) * kChunk;
    const int n_pre = max(0, min(P - c0, kChunk));   // prefix rows: tl < n_pre
    const int n_vis = min(T - c0, kChunk);           // visible rows: tl < n_vis
    const bool got = attn_wait(bars + 8u * (uint32_t)(i & 1), (uint32_t)(i >> 1) & 1u);
    if (c0 + kChunk > P) {
      // the chunk reaches the block: its keys and values from P on (block rows
      // jb0 ..), zeros past T; then the keys rotated, and row group 0 appends
      // them with the values to slots S + jb0 ..
      if (staged) {
        for (int e = tid; e < (kChunk - n_pre) * (D / 8); e += kAttnThreads) {
          const int tl = n_pre + e / (D / 8), c = e % (D / 8);
          uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
          if (tl < n_vis) {
            const int a = c0 + tl - P - jb0;
            kv = lds128(app + (uint32_t)((a * D + c * 8) * 2));
            vv = lds128(app + (uint32_t)(((kAppRows + a) * D + c * 8) * 2));
          }
          sts128(Ks + sw_off(tl, c * 8), kv);
          sts128(Vs + sw_off(tl, c * 8), vv);
        }
      } else {
        for (int e = tid; e < (kChunk - n_pre) * (D / 8); e += kAttnThreads) {
          const int tl = n_pre + e / (D / 8), c = e % (D / 8);
          const bool valid = tl < n_vis;
          const size_t src =
              valid ? (((size_t)b * p.L + (c0 + tl - P)) * p.Hkv + hk) * D + c * 8 : 0;
          cp_async_16(Ks + sw_off(tl, c * 8), p.k_new + src, valid);
          cp_async_16(Vs + sw_off(tl, c * 8), p.v_new + src, valid);
        }
        cp_async_wait_all();
      }
      __syncthreads();   // block-uniform branch: the rows are in place
      // (staged rows were rotated and appended at the start)
      if (rh > 0 && !staged) {
        for (int e = tid; e < (n_vis - n_pre) * npc; e += kAttnThreads) {
          const int tl = n_pre + e / npc, u = e - (e / npc) * npc;
          if (vec8)
            rot_key_step(c0 + tl - P, u, Ks + sw_off(tl, 8 * u), Ks + sw_off(tl, 8 * u + rh));
          else
            rot_key_step(c0 + tl - P, u, Ks + el_off(tl, u), Ks + el_off(tl, u + rh));
        }
        __syncthreads();
      }
      if (rg == 0 && !staged)
        for (int e = tid; e < (n_vis - n_pre) * 2 * (D / 8); e += kAttnThreads) {
          const int tl = n_pre + e / (2 * (D / 8)), rem = e % (2 * (D / 8));
          const int kv = rem / (D / 8), c = rem - kv * (D / 8);
          const uint4 v = lds128((kv ? Vs : Ks) + sw_off(tl, c * 8));
          const size_t dst = (head + (size_t)(S + c0 + tl - P)) * D + c * 8;
          if (in_bounds(dst + 7, p.cache_elems, p.err))
            *reinterpret_cast<uint4*>((kv ? p.v_cache : p.k_cache) + dst) = v;
        }
    }
    ok = __syncthreads_and(got) != 0;   // the whole tile, and one decision for the block
    if (!ok) break;

    if (live) {
      // S = Q K^T: A fragments of the warp's 16 query rows, B fragments of two
      // 8-key tiles per ldmatrix.x4
      float sc[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
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
      // mask, scale and the chunk's row maxima: key t is visible to query row
      // (j) iff t <= P + j (the prefix, then the block causally; never past
      // T); rows past R see nothing (lim -1)
      float mc[2] = {-INFINITY, -INFINITY};
      const int tb = c0 + 2 * tq;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int hh = e >> 1;
          const float v =
              tb + nt * 8 + (e & 1) <= (hh ? limB : limA) ? sc[nt][e] * p.scale_log2 : -INFINITY;
          sc[nt][e] = v;
          mc[hh] = fmaxf(mc[hh], v);
        }
      // online softmax: the running sums and outputs move to the new maximum
      float mu[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        mc[hh] = fmaxf(mc[hh], __shfl_xor_sync(0xffffffffu, mc[hh], 1));
        mc[hh] = fmaxf(mc[hh], __shfl_xor_sync(0xffffffffu, mc[hh], 2));
        const float mn = fmaxf(m_run[hh], mc[hh]);
        mu[hh] = mn == -INFINITY ? 0.f : mn;   // nothing visible yet: every p is 0
        const float alpha = exp2f(m_run[hh] - mu[hh]);
        m_run[hh] = mn;
        l_run[hh] *= alpha;
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd) {
          o[nd][2 * hh] *= alpha;
          o[nd][2 * hh + 1] *= alpha;
        }
      }
      // O += P V: P as 16-bit MMA operands (bf16: high part and remainder),
      // B fragments of two 8-dimension tiles per ldmatrix.x4.trans
#pragma unroll
      for (int kk = 0; kk < kChunk / 16; ++kk) {
        uint32_t ah[4], al[4];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int nt = 2 * kk + half;
          const float p0 = exp2f(sc[nt][0] - mu[0]), p1 = exp2f(sc[nt][1] - mu[0]);
          const float p2 = exp2f(sc[nt][2] - mu[1]), p3 = exp2f(sc[nt][3] - mu[1]);
          l_run[0] += p0 + p1;
          l_run[1] += p2 + p3;
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
    }
    // this stage's reads and writes before the TMA reuses it (never after a
    // chunk that reaches the block: that is the block's last)
    if (i + 2 < n_mine) fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0 && i + 2 < n_mine) issue(i + 2);
  }
  if (!ok) {
    // gave up on a stage: report it and let the copies already issued land
    if (tid == 0) atomicOr(p.err, kErrWaitTimeout);
    for (int i = done; i < n_mine && i < done + 2; ++i)
      attn_wait(bars + 8u * (uint32_t)(i & 1), (uint32_t)(i >> 1) & 1u);
    __syncthreads();
  }

#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 1);
    l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 2);
  }
  // every block is done with its ring (and every copy into it has landed):
  // the partial results of row r go to block r / 8, into its ring at
  // [this block][r % 8] (posted stores)
  cluster_sync_all();
  {
    const int rowA = row0 + g, rowB = rowA + 8;   // owners rowA / 8 and rowB / 8
    const uint32_t slot = (uint32_t)((int)rank * kMergeRows + g);
    // the two threads tq, tq ^ 1 trade halves so that each holds four
    // consecutive dimensions: the even one those of 8-column tile 2k, the odd
    // one those of tile 2k + 1 (one shuffle per value, half the stores)
    const bool odd = (tq & 1) != 0;
    const uint32_t oa = base + SM::OM + slot * SM::O_STRIDE +
                        (uint32_t)((odd ? 8 + 2 * (tq - 1) : 2 * tq) * 4);
    const uint32_t dA = peer_addr(oa, (uint32_t)(rowA / kMergeRows));
    const uint32_t dB = peer_addr(oa, (uint32_t)(rowB / kMergeRows));
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      float t[4], keep[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        // the half the partner takes goes over, the other half stays
        t[e] = __shfl_xor_sync(0xffffffffu, odd ? o[2 * k][e] : o[2 * k + 1][e], 1);
        keep[e] = odd ? o[2 * k + 1][e] : o[2 * k][e];
      }
      float4 va, vb;
      if (odd) {
        va = make_float4(t[0], t[1], keep[0], keep[1]);
        vb = make_float4(t[2], t[3], keep[2], keep[3]);
      } else {
        va = make_float4(keep[0], keep[1], t[0], t[1]);
        vb = make_float4(keep[2], keep[3], t[2], t[3]);
      }
      st_peer_v4(dA + k * 64, make_uint4(__float_as_uint(va.x), __float_as_uint(va.y),
                                         __float_as_uint(va.z), __float_as_uint(va.w)));
      st_peer_v4(dB + k * 64, make_uint4(__float_as_uint(vb.x), __float_as_uint(vb.y),
                                         __float_as_uint(vb.z), __float_as_uint(vb.w)));
    }
    if (tq == 0) {
      const uint32_t ma = base + SM::ML + slot * 8u;
      st_peer_f2(peer_addr(ma, (uint32_t)(rowA / kMergeRows)), m_run[0], l_run[0]);
      st_peer_f2(peer_addr(ma, (uint32_t)(rowB / kMergeRows)), m_run[1], l_run[1]);
    }
  }
  cluster_sync_all();   // every block's partial results have landed

  // merge rows q0 .. q0 + 7 over the cluster's blocks in rank order: sixteen
  // threads per row; thread q of a row takes the float4s q, q + 16, ... of it
  // (dimensions 4q .. 4q + 3, ...)
  constexpr int NV = D / 64;   // float4s per thread
  constexpr int VEC = 4 * NV;
  const int r8 = tid / 16, q16 = tid % 16;
  float2 ml[kCluster];
  float4 ov[kCluster][NV];
#pragma unroll
  for (int c = 0; c < kCluster; ++c) {
    const uint32_t slot = (uint32_t)(c * kMergeRows + r8);
    ml[c] = lds64f(base + SM::ML + slot * 8u);
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const uint4 w = lds128(base + SM::OM + slot * SM::O_STRIDE + (uint32_t)(q16 + 16 * v) * 16u);
      ov[c][v] = make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                             __uint_as_float(w.w));
    }
  }
  float mx = -INFINITY;
#pragma unroll
  for (int c = 0; c < kCluster; ++c)
    if (ml[c].y > 0.f) mx = fmaxf(mx, ml[c].x);
  float acc[VEC], den = 0.f;
#pragma unroll
  for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
#pragma unroll
  for (int c = 0; c < kCluster; ++c) {
    // a block that saw no visible key of this row adds nothing
    const float w = ml[c].y > 0.f ? exp2f(ml[c].x - mx) : 0.f;
    den += w * ml[c].y;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      acc[4 * v] += w * ov[c][v].x;
      acc[4 * v + 1] += w * ov[c][v].y;
      acc[4 * v + 2] += w * ov[c][v].z;
      acc[4 * v + 3] += w * ov[c][v].w;
    }
  }

  const int rr = rr0 + q0 + r8;
  if (rr < p.R) {
    const int j = rr / p.G, hq = hk * p.G + (rr - j * p.G);
    const size_t row = (((size_t)b * p.L + j) * p.Hq + hq) * D;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const size_t dst = row + 4 * (q16 + 16 * v);
      if (!in_bounds(dst + 3, p.out_elems, p.err)) continue;
      uint16_t h[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) h[k] = f2h<kF16>(acc[4 * v + k] / den);
      if (p.out_vec) {
        *reinterpret_cast<uint2*>(p.out + dst) =
            make_uint2((uint32_t)h[0] | ((uint32_t)h[1] << 16), (uint32_t)h[2] | ((uint32_t)h[3] << 16));
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) p.out[dst + k] = h[k];
      }
    }
  }
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
  // grid limits: (cluster, Hkv x row groups, B); the cache rows are addressed
  // by 32-bit TMA coordinates
  const long long row_groups = ((long long)L * (Hq / Hkv) + kAttnRows - 1) / kAttnRows;
  if ((long long)Hkv * row_groups > 65535 || B > 65535 || (long long)B * Hkv * S_cap > 0x7fffffffll)
    return VQ_EUNSUPPORTED;
  const uintptr_t a16 = (uintptr_t)q | (uintptr_t)k_new | (uintptr_t)v_new |
                        (uintptr_t)k_cache | (uintptr_t)v_cache;
  if ((a16 & 15u) || ((uintptr_t)out & 1u) ||
      (((uintptr_t)prefix_len | (uintptr_t)src_off | (uintptr_t)status) & 3u))
    return VQ_EALIGN;
  return VQ_OK;
}

struct AttnShape {
  int G, R, RG;
};

AttnShape attn_shape(int L, int Hq, int Hkv) {
  AttnShape s;
  s.G = Hq / Hkv;
  s.R = L * s.G;
  s.RG = (s.R + kAttnRows - 1) / kAttnRows;
  return s;
}

template <bool kF16, int D>
int attn_launch(const AttnParams& p, int B, cudaStream_t stream, const CUtensorMap& tm_k,
                const CUtensorMap& tm_v) {
  const size_t smem = 1024 + AttnSmem<D>::BYTES;   // + the 1 KiB alignment of the base
  if (ensure_smem<verify_attn_kernel<kF16, D>>(smem) != VQ_OK) return VQ_ECUDA;
  // clusters of kCluster blocks along x (the kernel's compile-time cluster shape)
  verify_attn_kernel<kF16, D>
      <<<dim3(kCluster, p.Hkv * p.RG, B), kAttnThreads, smem, stream>>>(tm_k, tm_v, p);
  return cudaGetLastError() == cudaSuccess ? VQ_OK : VQ_ECUDA;
}

}  // namespace
}  // namespace vq

using namespace vq;

extern "C" size_t verify_attention_workspace_bytes(int, int, int, int, int, int) {
  return 0;   // the kernel keeps its partial results in the cluster's shared memory
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
  (void)workspace;   // none needed
  (void)workspace_bytes;
  int32_t* err = nullptr;   // the device's status word (a usable current device)
  rc = device_error_word(&err);
  if (rc) return rc;

  const AttnShape s = attn_shape(L, Hq, Hkv);
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
  p.cache_elems = (size_t)B * Hkv * S_cap * D;
  p.out_elems = (size_t)B * L * Hq * D;
  p.out_vec = ((uintptr_t)out & 15u) == 0;
  p.L = L;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = s.G;
  p.R = s.R;
  p.RG = s.RG;
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
