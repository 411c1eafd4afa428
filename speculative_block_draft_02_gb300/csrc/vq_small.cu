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

// Fold layout (ds4 #778, PR description: the committed token is verified as
// row 0 of the verify block): tokens[b][0] is row b's committed token,
// tokens[b][1..L-1] its drafts, and target[b][j] the greedy token the target
// predicts after position j. Draft j+1 is accepted while it equals
// target[b][j]: accept[b] in 0..L-1, bonus[b] = target[b][accept[b]] (the
// next block's committed token), keep[b] = accept[b] + 1 KV slots (the
// committed token's and the accepted drafts').
__global__ void fold_accept_kernel(const int32_t* __restrict__ tokens,
                                   const int32_t* __restrict__ target, int B, int L,
                                   int32_t* __restrict__ accept, int32_t* __restrict__ bonus,
                                   int32_t* __restrict__ keep) {
  const int row = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= B) return;
  const int32_t* d = tokens + (size_t)row * L + 1;
  const int32_t* t = target + (size_t)row * L;
  int a = L - 1;
  for (int j0 = 0; j0 < L - 1; j0 += 32) {
    const int j = j0 + lane;
    const bool miss = j < L - 1 && d[j] != t[j];
    const unsigned mask = __ballot_sync(0xffffffffu, miss);
    if (mask) {
      a = j0 + __ffs(mask) - 1;
      break;
    }
  }
  if (lane == 0) {
    accept[row] = a;
    bonus[row] = t[a];
    keep[row] = a + 1;
  }
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
                                  int32_t* __restrict__ new_len, int32_t* __restrict__ status,
                                  int32_t* __restrict__ err) {
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
  // Bounds-checked builds test each vector index against the tensor's B*H*S_cap slots.
  const size_t base = ((size_t)b * H + h) * (size_t)S_cap * vec_per_slot;
  const size_t extent = (size_t)B * H * (size_t)S_cap * vec_per_slot;
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    if (in_bounds(base + (size_t)s * vec_per_slot + i, extent, err)) kv_buf[i] = src[i];
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    if (in_bounds(base + (size_t)p * vec_per_slot + i, extent, err)) dst[i] = kv_buf[i];
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

namespace {
// Host checks of a KV commit; fills the tensor table.
int kv_check(void* const* tensors, int n_tensors, int B, int H, int S_cap, int D, int elem_bytes,
             const int32_t* prefix_len, const int32_t* src_off, const int32_t* keep,
             int max_keep, int32_t* new_len, int32_t* status, KvTensors* tp) {
  if (!tensors || n_tensors < 1 || n_tensors > kMaxKvTensors) return VQ_EINVAL;
  if (B < 1 || H < 1 || S_cap < 1 || D < 1 || elem_bytes < 1 || max_keep < 0) return VQ_EINVAL;
  if (!prefix_len || !src_off || !keep || !new_len) return VQ_EINVAL;
  const long long slot_bytes = (long long)D * elem_bytes;
  if (slot_bytes % 16 != 0) return VQ_EALIGN;
  if ((long long)max_keep * slot_bytes > 160 * 1024) return VQ_EUNSUPPORTED;
  if ((long long)n_tensors * B * H > 0x7fffffffLL) return VQ_EINVAL;
  for (int i = 0; i < kMaxKvTensors; ++i) tp->p[i] = nullptr;
  for (int i = 0; i < n_tensors; ++i) {
    if (!tensors[i]) return VQ_EINVAL;
    if ((uintptr_t)tensors[i] & 15u) return VQ_EALIGN;
    tp->p[i] = tensors[i];
  }
  if (((uintptr_t)prefix_len | (uintptr_t)src_off | (uintptr_t)keep | (uintptr_t)new_len |
       (uintptr_t)status) & 3u)
    return VQ_EALIGN;
  return VQ_OK;
}
}  // namespace

extern "C" int kv_compact_per_row(void* const* tensors, int n_tensors, int B, int H, int S_cap,
                                  int D, int elem_bytes, const int32_t* prefix_len,
                                  const int32_t* src_off, const int32_t* keep, int max_keep,
                                  int32_t* new_len, int32_t* status, void* stream) {
  KvTensors tp;
  const int rc = kv_check(tensors, n_tensors, B, H, S_cap, D, elem_bytes, prefix_len, src_off,
                          keep, max_keep, new_len, status, &tp);
  if (rc) return rc;
  const long long slot_bytes = (long long)D * elem_bytes;
  const long long buf_bytes = (long long)max_keep * slot_bytes;
  const long long blocks = (long long)n_tensors * B * H;
  const size_t smem = (size_t)(buf_bytes > 0 ? buf_bytes : 16);
  if (smem > 48 * 1024 && ensure_smem<kv_compact_kernel>(smem) != VQ_OK) return VQ_ECUDA;
  int32_t* err = nullptr;
  if (device_error_word(&err) != VQ_OK) return VQ_ECUDA;
  kv_compact_kernel<<<(unsigned)blocks, 256, smem, (cudaStream_t)stream>>>(
      tp, B, H, S_cap, (int)(slot_bytes / 16), prefix_len, src_off, keep, max_keep, new_len,
      status, err);
  return cudaGetLastError() == cudaSuccess ? VQ_OK : VQ_ECUDA;
}

extern "C" size_t vq_vocab_argmax_workspace_bytes(int M);
extern "C" int vq_vocab_argmax(const void* x, int M, int K, int N, const uint32_t* qw,
                               const uint16_t* scales, const uint16_t* biases, int act_dtype,
                               int32_t* argmax, float* maxval, void* workspace,
                               size_t workspace_bytes, void* stream);

extern "C" size_t verify_round_workspace_bytes(int B, int L) {
  if (B < 1 || L < 1 || (long long)B * L > 64) return 0;
  return vq_vocab_argmax_workspace_bytes(B * L) + (((size_t)B * 4 + 15) & ~(size_t)15);
}

extern "C" int verify_round_multi(const void* h, int B, int L, int K, int N, const uint32_t* qw,
                                  const uint16_t* scales, const uint16_t* biases, int act_dtype,
                                  const int32_t* tokens, int32_t* target, int32_t* accept,
                                  int32_t* bonus, const vq_kv_set* sets, int n_sets,
                                  int32_t* status, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  if (B < 1 || L < 1 || (long long)B * L > 64) return VQ_EINVAL;
  if (!tokens || !target || !accept || !bonus) return VQ_EINVAL;
  if (n_sets < 0 || (n_sets > 0 && !sets)) return VQ_EINVAL;
  if (((uintptr_t)tokens | (uintptr_t)target | (uintptr_t)accept | (uintptr_t)bonus) & 3u)
    return VQ_EALIGN;
  const size_t need = verify_round_workspace_bytes(B, L);
  if (!workspace || workspace_bytes < need) return VQ_EWORKSPACE;
  if ((uintptr_t)workspace & 15u) return VQ_EALIGN;
  const size_t wa = vq_vocab_argmax_workspace_bytes(B * L);
  int32_t* keep = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + wa);
  // every argument of every set is checked before the first launch
  for (int i = 0; i < n_sets; ++i) {
    const vq_kv_set& c = sets[i];
    KvTensors tp;
    const int rc = kv_check(c.tensors, c.n_tensors, B, c.H, c.S_cap, c.D, c.elem_bytes,
                            c.prefix_len, c.src_off, keep, L, c.new_len, status, &tp);
    if (rc) return rc;
  }
  int rc = vq_vocab_argmax(h, B * L, K, N, qw, scales, biases, act_dtype, target, nullptr,
                           workspace, wa, stream);
  if (rc) return rc;
  const int threads = 128;
  const unsigned blocks = (unsigned)(((long long)B * 32 + threads - 1) / threads);
  fold_accept_kernel<<<blocks, threads, 0, (cudaStream_t)stream>>>(tokens, target, B, L, accept,
                                                                   bonus, keep);
  if (cudaGetLastError() != cudaSuccess) return VQ_ECUDA;
  for (int i = 0; i < n_sets; ++i) {
    const vq_kv_set& c = sets[i];
    rc = kv_compact_per_row(c.tensors, c.n_tensors, B, c.H, c.S_cap, c.D, c.elem_bytes,
                            c.prefix_len, c.src_off, keep, L, c.new_len, status, stream);
    if (rc) return rc;
  }
  return VQ_OK;
}

extern "C" int verify_round(const void* h, int B, int L, int K, int N, const uint32_t* qw,
                            const uint16_t* scales, const uint16_t* biases, int act_dtype,
                            const int32_t* tokens, int32_t* target, int32_t* accept,
                            int32_t* bonus, void* const* kv_tensors, int n_tensors, int H,
                            int S_cap, int D, int elem_bytes, const int32_t* prefix_len,
                            const int32_t* src_off, int32_t* new_len, int32_t* status,
                            void* workspace, size_t workspace_bytes, void* stream) {
  vq_kv_set set;
  set.tensors = kv_tensors;
  set.n_tensors = n_tensors;
  set.H = H;
  set.S_cap = S_cap;
  set.D = D;
  set.elem_bytes = elem_bytes;
  set.prefix_len = prefix_len;
  set.src_off = src_off;
  set.new_len = new_len;
  return verify_round_multi(h, B, L, K, N, qw, scales, biases, act_dtype, tokens, target, accept,
                            bonus, &set, n_tensors > 0 ? 1 : 0, status, workspace,
                            workspace_bytes, stream);
}
