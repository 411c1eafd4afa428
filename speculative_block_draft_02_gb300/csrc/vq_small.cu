// The two integer / byte steps of a verify round: the per-row accept walk and
// the per-row KV commit (mlxcel #2865 "perf(speculative): commit per-row
// accepts in batched DFlash", Summary and commit message).
#include <mutex>

#include "vq_common.cuh"

namespace vq {

// One warp per batch row: the first mismatch among 32 positions at a time is
// found with a ballot, so the walk costs ceil(L/32) coalesced loads per row.
__global__ void accept_walk_kernel(const int32_t* __restrict__ draft,
                                   const int32_t* __restrict__ target, int B, int L,
                                   int32_t* __restrict__ accept) {
  const int row = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= B) return;
  const int32_t* d = draft + (size_t)row * L;
  const int32_t* t = target + (size_t)row * L;
  int a = L;
  for (int j0 = 0; j0 < L; j0 += 32) {
    const int j = j0 + lane;
    const bool miss = j < L && d[j] != t[j];
    const unsigned mask = __ballot_sync(0xffffffffu, miss);
    if (mask) {
      a = j0 + __ffs(mask) - 1;
      break;
    }
  }
  if (lane == 0) accept[row] = a;
}

constexpr int kMaxKvTensors = 64;
struct KvTensors {
  void* p[kMaxKvTensors];
};

// One block per (tensor, row b, head h): the kept slots are read into shared
// memory in full before any is written, so overlapping source and
// destination ranges are safe. 16-byte vector copies throughout.
__global__ void kv_compact_kernel(KvTensors tp, int B, int H, int S_cap, int vec_per_slot,
                                  const int32_t* __restrict__ prefix_len,
                                  const int32_t* __restrict__ src_off,
                                  const int32_t* __restrict__ keep, int max_keep,
                                  int32_t* __restrict__ new_len, int32_t* __restrict__ status) {
  extern __shared__ uint4 kv_buf[];
  const int h = blockIdx.x % H;
  const int b = (blockIdx.x / H) % B;
  const int t = blockIdx.x / (H * B);
  const int p = prefix_len[b], s = src_off[b], c = keep[b];
  const bool ok = c >= 0 && c <= max_keep && p >= 0 && s >= 0 && p <= S_cap - c && s <= S_cap - c;
  if (t == 0 && h == 0 && threadIdx.x == 0) {
    new_len[b] = ok ? p + c : -1;
    if (!ok && status) atomicOr(status, 1);
  }
  if (!ok || c == 0 || p == s) return;
  uint4* row = reinterpret_cast<uint4*>(tp.p[t]) + ((size_t)b * H + h) * (size_t)S_cap * vec_per_slot;
  const int n = c * vec_per_slot;
  const uint4* src = row + (size_t)s * vec_per_slot;
  uint4* dst = row + (size_t)p * vec_per_slot;
  for (int i = threadIdx.x; i < n; i += blockDim.x) kv_buf[i] = src[i];
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = kv_buf[i];
}

}  // namespace vq

using namespace vq;

extern "C" int verify_accept_walk(const int32_t* draft, const int32_t* target, int B, int L,
                                  int32_t* accept, void* stream) {
  if (!draft || !target || !accept || B < 1 || L < 1) return VQ_EINVAL;
  if (((uintptr_t)draft | (uintptr_t)target | (uintptr_t)accept) & 3u) return VQ_EALIGN;
  const int threads = 128;
  const long long blocks = ((long long)B * 32 + threads - 1) / threads;
  if (blocks > 0x7fffffffLL) return VQ_EINVAL;
  accept_walk_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(draft, target, B, L,
                                                                           accept);
  return cudaGetLastError() == cudaSuccess ? VQ_OK : VQ_ECUDA;
}

extern "C" int kv_compact_per_row(void* const* tensors, int n_tensors, int B, int H, int S_cap,
                                  int D, int elem_bytes, const int32_t* prefix_len,
                                  const int32_t* src_off, const int32_t* keep, int max_keep,
                                  int32_t* new_len, int32_t* status, void* stream) {
  if (!tensors || n_tensors < 1 || n_tensors > kMaxKvTensors) return VQ_EINVAL;
  if (B < 1 || H < 1 || S_cap < 1 || D < 1 || elem_bytes < 1 || max_keep < 0) return VQ_EINVAL;
  if (!prefix_len || !src_off || !keep || !new_len) return VQ_EINVAL;
  const long long slot_bytes = (long long)D * elem_bytes;
  if (slot_bytes % 16 != 0) return VQ_EALIGN;
  const long long buf_bytes = (long long)max_keep * slot_bytes;
  if (buf_bytes > 160 * 1024) return VQ_EUNSUPPORTED;
  const long long blocks = (long long)n_tensors * B * H;
  if (blocks > 0x7fffffffLL) return VQ_EINVAL;
  KvTensors tp;
  for (int i = 0; i < kMaxKvTensors; ++i) tp.p[i] = nullptr;
  for (int i = 0; i < n_tensors; ++i) {
    if (!tensors[i]) return VQ_EINVAL;
    if ((uintptr_t)tensors[i] & 15u) return VQ_EALIGN;
    tp.p[i] = tensors[i];
  }
  if (((uintptr_t)prefix_len | (uintptr_t)src_off | (uintptr_t)keep | (uintptr_t)new_len |
       (uintptr_t)status) & 3u)
    return VQ_EALIGN;
  const size_t smem = (size_t)(buf_bytes > 0 ? buf_bytes : 16);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(kv_compact_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return VQ_ECUDA;
  }
  kv_compact_kernel<<<(unsigned)blocks, 256, smem, (cudaStream_t)stream>>>(
      tp, B, H, S_cap, (int)(slot_bytes / 16), prefix_len, src_off, keep, max_keep, new_len,
      status);
  return cudaGetLastError() == cudaSuccess ? VQ_OK : VQ_ECUDA;
}
