/*
 * vq.h -- C ABI of the GB300 (sm_103a) block-verification hot path.
 *
 * Four operations make up one verify round of DFlash-style block speculative
 * decoding once the target has produced its hidden states (verify_round
 * chains the last three in one call):
 *
 *   vq_linear            the small-M verification projection over 4-bit
 *                        group-quantized weights
 *   vq_vocab_argmax      the vocabulary projection with the greedy arg max
 *                        fused in (no logits are written)
 *   verify_accept_walk   the per-row accept walk
 *   kv_compact_per_row   the per-row KV commit
 *
 * verify_attention is the attention of the verify block inside the target's
 * forward pass, over the same per-row cache the KV commit maintains.
 *
 * Common rules
 *   - Every tensor pointer is caller-owned DEVICE memory unless a parameter
 *     says otherwise. The library allocates nothing.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). Every call only enqueues work on it and returns without
 *     synchronizing; results are ready when the stream reaches that point.
 *   - Calls return VQ_OK (0) or a negative VQ_E* code. Argument errors are
 *     found on the host before anything is enqueued. Failures found on the
 *     device never trap: they are OR-ed into a status word that
 *     vq_device_error() reads, or into a caller-provided status.
 *   - Row-major layouts throughout; sizes are in elements unless noted.
 *   - A workspace may be shared by successive calls on one stream, never by
 *     calls that can run at the same time.
 *   - Set-up: the first call of any projection entry point (vq_linear,
 *     vq_vocab_argmax and their variants, verify_round*) on a device, with
 *     that device current, looks up the library's device symbols and the
 *     driver's tensor-map encoder; make that first call before any stream
 *     capture on that device.
 *   - vq_linear, vq_vocab_argmax and vq_vocab_argmax_noalloc launch their
 *     kernels with programmatic stream serialization, so that back-to-back
 *     projections overlap: a kernel may start while the kernel before it in
 *     the stream is finishing. It requests its first weight stages (qw,
 *     scales, biases) right away, and reads x and writes its outputs and
 *     workspace only after that kernel has completed (griddepcontrol.wait).
 *     So the weights must not be written by the kernel launched immediately
 *     before the call on the same stream; weights written at load time are
 *     fine, as is any write followed by another operation on the stream.
 */
#ifndef VQ_H_
#define VQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define VQ_OK 0
#define VQ_EINVAL (-1)        /* a shape, size or enum argument is out of range */
#define VQ_EALIGN (-2)        /* a pointer is not aligned as required */
#define VQ_ECUDA (-3)         /* the CUDA runtime reported an error */
#define VQ_EUNSUPPORTED (-4)  /* valid, but outside the variants compiled here */
#define VQ_EWORKSPACE (-5)    /* workspace missing or smaller than required */

/* Activation dtypes. The output of vq_linear has the activation dtype. */
#define VQ_BF16 0
#define VQ_F16 1
#define VQ_F32 2

/*
 * Verification projection over W4 group-quantized weights.
 *
 * Source: dflash-mlx #7 "perf: tune DFlash2 M=8 verification for M1 and M2",
 * PR description -- VerifyQuantizedLinear runs the M rows of a verify block
 * (M = 8 for DFlash2's eight-token block, "Why") through 4-bit weights; the
 * W4A32 path takes fp32 activations. ds4 #778 "dspark: fold first-token
 * forward into verify ...", commit 1 message -- row tiles so that a verify
 * block reads every weight once, not once per row.
 *
 *   y[m][n] = sum_k x[m][k] * w(n,k),   0 <= m < M, 0 <= n < N
 *   w(n,k)  = scale[n][k/64] * code(n,k) + bias[n][k/64]
 *   code(n,k) = (qw[n][k/8] >> (4*(k%8))) & 15     (lowest nibble first)
 *
 * x        [M][K] activations, dtype act_dtype (bf16 / f16 bits or fp32),
 *          16-byte aligned.
 * qw       [N][K/8] uint32, eight 4-bit codes per word along K, 16-byte aligned.
 * scales   [N][K/64] bf16 bits, 16-byte aligned.
 * biases   [N][K/64] bf16 bits, 16-byte aligned.
 * y        [M][N] output in act_dtype (round to nearest even from the fp32
 *          accumulator; fp32 output for VQ_F32), 4-byte aligned.
 * workspace / workspace_bytes
 *          scratch for (a) x converted once per call into per-stage slices of
 *          scaled fp16 MMA fragments (16-bit x with M <= 16 and K a multiple
 *          of 512: about 17.6*K bytes per 8 rows), (b) the group row sums of x
 *          (16-bit x, M > 16), and (c) the split-K reduction used when N is
 *          too narrow to fill the GPU. vq_linear_workspace_bytes() gives the size needed (0
 *          when neither is used; then workspace may be NULL). The workspace
 *          must be zero-filled before its first use; every call leaves the
 *          part that must start at zero zero-filled again. 16-byte aligned.
 *          With the slices, the call enqueues two kernels: the slices, then
 *          the projection, which may start before the slices are done and
 *          waits for them.
 * Sizes    1 <= M <= 64 (M <= 32 for VQ_F32), K a positive multiple of 64,
 *          N >= 1. K that is not a multiple of 512 runs on the per-stage x
 *          kernels with a last, partial stage (the scales and biases are then
 *          read without a tensor map, whose rows must be 16-byte multiples).
 *          Shapes whose shared-memory plan does not fit return
 *          VQ_EUNSUPPORTED: K > 32768 with fp32 x and 8 < M <= 16, or with
 *          K not a multiple of 512 and 8 < M <= 16; with fp32 x and M > 16,
 *          K > 12800; with 16-bit x, M > 16 and an N narrow enough that K is
 *          split (N < 9728 on 152 SMs), K > 16384 for M <= 32 and K > 6144
 *          above. vq_plan() tells whether a shape runs.
 * Accumulation is fp32; each 64-wide group is accumulated from exact integer
 * codes and scaled once, so the only roundings are the fp32 sums and the
 * final cast.
 */
size_t vq_linear_workspace_bytes(int M, int K, int N, int act_dtype);
int vq_linear(const void* x, int M, int K, int N, const uint32_t* qw, const uint16_t* scales,
              const uint16_t* biases, void* y, int act_dtype, void* workspace,
              size_t workspace_bytes, void* stream);

/*
 * vq_linear for activations and outputs in host memory: enqueues on `stream`
 * the copy of x_host into x_dev, vq_linear(x_dev -> y_dev) and the copy of
 * y_dev into y_host, and returns (nothing is waited for; the caller
 * synchronizes the stream before reading y_host). For the step a serving
 * loop makes when the activations arrive from and the logits go back to the
 * host.
 *
 * x_host   [M][K] in act_dtype, host memory (page-locked for the copies to
 *          be asynchronous). y_host [M][N] in act_dtype, host memory.
 * x_dev, y_dev  device buffers of the same shapes, with vq_linear's
 *          alignment (16 bytes for x_dev, 4 for y_dev); owned by the caller.
 * Other arguments as vq_linear. Errors in the shape, the device buffers and
 * the workspace are returned before anything is enqueued; an error in the
 * weights' arguments (as vq_linear returns it) may come after the copy of x
 * has been enqueued; VQ_ECUDA if a copy cannot be enqueued. Where the device
 * can address page-locked host buffers directly (cudaPointerGetAttributes;
 * with unified addressing, as on GB300), the plans that read x only in their
 * slice kernel read it from x_host and, without a K split, write y straight
 * into y_host; x_dev and y_dev are then not touched.
 */
int vq_linear_host(const void* x_host, int M, int K, int N, const uint32_t* qw,
                   const uint16_t* scales, const uint16_t* biases, void* y_host, int act_dtype,
                   void* x_dev, void* y_dev, void* workspace, size_t workspace_bytes,
                   void* stream);

/*
 * Vocabulary projection with a fused greedy arg max.
 *
 * Source: dflash-mlx #7, PR description (the W4A32 vocabulary projection of
 * the verify path); ds4 #778, commit 1 message (a fused matvec + arg max
 * kernel; greedy decoding at temperature 0).
 *
 *   logits[m][n] = the vq_linear result, kept in fp32 and never stored
 *   argmax[m]    = the n with the largest logits[m][n]; ties go to the
 *                  lowest n; NaN logits never win (a row with no non-NaN
 *                  logit gives 0)
 *   maxval[m]    = logits[m][argmax[m]] in fp32 (optional, may be NULL)
 *
 * Arguments as in vq_linear; argmax is int32 [M], maxval float [M].
 * workspace: vq_vocab_argmax_workspace_bytes(M) bytes, required, 16-byte
 *          aligned, zero-filled before its first use; every call leaves it
 *          zero-filled again.
 * Sizes    1 <= M <= 64 (M <= 32 for VQ_F32), K a positive multiple of 64,
 *          1 <= N < 2^31; as vq_linear, K > 32768 with 8 < M <= 16 and
 *          K > 9728 with fp32 x and M > 16 return VQ_EUNSUPPORTED.
 */
size_t vq_vocab_argmax_workspace_bytes(int M);
int vq_vocab_argmax(const void* x, int M, int K, int N, const uint32_t* qw,
                    const uint16_t* scales, const uint16_t* biases, int act_dtype,
                    int32_t* argmax, float* maxval, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * Vocabulary projection with the fused arg max and the runner-up logit.
 *
 * Source: ds4 #778 "dspark: fold first-token forward into verify ...", PR
 * description (the margin gate: the drafter does not propose where the
 * target's top-1/top-2 logit margin shows that the target is hesitating).
 *
 * The same operation, arguments and results as vq_vocab_argmax, plus
 *   second[m] = the largest logits[m][n] over n != argmax[m] in fp32 (NaN
 *               logits skipped; -inf when the row has no other non-NaN
 *               logit); an exact tie for the maximum gives second = maxval.
 * so that maxval[m] - second[m] is the top-1/top-2 margin.
 * second     float [M] on the device, required.
 * workspace  vq_vocab_argmax_top2_workspace_bytes(M) bytes (528 + 4096*M at
 *            most), 16-byte aligned, zero-filled before its first use; the
 *            part that must start at zero is left zero-filled by every call.
 */
size_t vq_vocab_argmax_top2_workspace_bytes(int M);
int vq_vocab_argmax_top2(const void* x, int M, int K, int N, const uint32_t* qw,
                         const uint16_t* scales, const uint16_t* biases, int act_dtype,
                         int32_t* argmax, float* maxval, float* second, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * vq_vocab_argmax without a workspace: the same operation, arguments and
 * results as vq_vocab_argmax, but its scratch memory (M*8 + 4 bytes, rounded
 * up to 16) lives in a fixed 1 KiB array inside this library, so the call
 * allocates nothing. The pages have no counterpart of this entry point; it is
 * there for callers that cannot call cudaMalloc or have a buffer made for
 * them: serving runtimes that forbid device allocation once they are running
 * (an allocation can block, fragment memory or fail at a bad moment), and
 * plug-ins embedded in a host application that owns all device memory and
 * hands out none for scratch.
 *
 * Limit: 1 <= M <= 64 (the array's size); a larger M returns VQ_EINVAL.
 * Set-up: the first call on a device (with that device current) also looks
 * up the array's device address (see the common set-up rule above).
 * The array is held by every GPU that loads the library until the process
 * exits. Each call clears the part it uses on `stream` before the kernel
 * (a completed call leaves it zeroed already; only a call that gave up on a
 * bounded wait leaves keys behind).
 * Calls share the one array: calls that can overlap on the GPU (different
 * streams, or different host threads) race and must not be made.
 */
int vq_vocab_argmax_noalloc(const void* x, int M, int K, int N, const uint32_t* qw,
                            const uint16_t* scales, const uint16_t* biases, int act_dtype,
                            int32_t* argmax, float* maxval, void* stream);

/*
 * Per-row accept walk.
 *
 * Source: mlxcel #2865 "perf(speculative): commit per-row accepts in batched
 * DFlash", Summary and commit message -- each batch row commits its own walk
 * count instead of the shortest row's.
 *
 *   accept[b] = the number of leading positions j with
 *               draft[b][j] == target[b][j]  (L when all L match)
 *
 * draft, target  int32 [B][L]; target[b][j] is the greedy token of verify
 *                row j of batch row b, aligned with draft[b][j].
 * accept         int32 [B].
 * Sizes          B >= 1, L >= 1.
 */
int verify_accept_walk(const int32_t* draft, const int32_t* target, int B, int L,
                       int32_t* accept, void* stream);

/*
 * Per-row KV commit (compaction to a contiguous valid prefix).
 *
 * Source: mlxcel #2865, Summary -- after each round the target's attention
 * cache is packed again so that every row's valid tokens form one unbroken
 * run from slot 0, which lets each row keep its own accept count in a
 * rectangular cache.
 *
 * For each of the n_tensors tensors (e.g. K and V of every layer), each row b
 * and head h: slots src_off[b] .. src_off[b]+keep[b]-1, as they were before
 * the call, are copied to slots prefix_len[b] .. prefix_len[b]+keep[b]-1
 * (the ranges may overlap), and new_len[b] = prefix_len[b] + keep[b].
 * Slots below prefix_len[b] are untouched.
 *
 * tensors     HOST array of n_tensors DEVICE pointers, each a
 *             [B][H][S_cap][D] tensor of elem_bytes-byte elements,
 *             16-byte aligned; 1 <= n_tensors <= 64.
 * prefix_len, src_off, keep   int32 [B] on the device (keep may come straight
 *             from verify_accept_walk, so no host round trip is needed).
 * max_keep    host bound on keep[b]; D*elem_bytes must be a multiple of 16
 *             and max_keep*D*elem_bytes at most 160 KiB.
 * new_len     int32 [B] on the device.
 * status      optional int32 on the device: a row whose keep is outside
 *             0..max_keep, or whose source or destination range leaves
 *             0..S_cap, is left untouched, gets new_len[b] = -1, and bit 0
 *             is OR-ed into *status. The call never clears *status.
 */
int kv_compact_per_row(void* const* tensors, int n_tensors, int B, int H, int S_cap, int D,
                       int elem_bytes, const int32_t* prefix_len, const int32_t* src_off,
                       const int32_t* keep, int max_keep, int32_t* new_len, int32_t* status,
                       void* stream);

/*
 * One verify round in one call, in the fold layout: vocabulary arg max over
 * the verify block, accept walk, and per-row KV commit, enqueued back to back
 * on `stream` with no host round trip (the call can be captured in a CUDA
 * graph as it is).
 *
 * Source: ds4 #778 "dspark: fold first-token forward into verify ...", PR
 * description and commit 1 (the committed token is verified as row 0 of the
 * verify block, so one batched pass covers it and the drafts); mlxcel #2865,
 * Summary (per-row accepts and the per-row KV commit).
 *
 *   tokens[b][0]      row b's committed token; tokens[b][1..L-1] its drafts
 *   target[b][j]      = arg max of logits of verify row (b, j), as
 *                       vq_vocab_argmax with M = B*L rows ordered (b, j)
 *   accept[b]         = number of leading j in 0..L-2 with
 *                       tokens[b][j+1] == target[b][j]   (0..L-1)
 *   bonus[b]          = target[b][accept[b]]: the next block's committed token
 *   KV commit         as kv_compact_per_row with keep[b] = accept[b] + 1 (the
 *                     committed token's slot and the accepted drafts'),
 *                     max_keep = L; skipped when n_tensors == 0.
 *
 * h          [B*L][K] hidden states of the verify block (act_dtype), the
 *            vocabulary projection's x; qw, scales, biases as vq_vocab_argmax.
 * tokens     int32 [B][L]; target int32 [B][L]; accept, bonus int32 [B].
 * kv_tensors ... status: as kv_compact_per_row (HOST array of device
 *            pointers); all ignored when n_tensors == 0.
 * workspace  verify_round_workspace_bytes(B, L) bytes, 16-byte aligned,
 *            zero-filled before its first use; left zero-filled where needed.
 * Sizes      1 <= B*L <= 64, K a positive multiple of 64, N >= 1. Every
 *            argument is checked before the first launch.
 */
size_t verify_round_workspace_bytes(int B, int L);
int verify_round(const void* h, int B, int L, int K, int N, const uint32_t* qw,
                 const uint16_t* scales, const uint16_t* biases, int act_dtype,
                 const int32_t* tokens, int32_t* target, int32_t* accept, int32_t* bonus,
                 void* const* kv_tensors, int n_tensors, int H, int S_cap, int D, int elem_bytes,
                 const int32_t* prefix_len, const int32_t* src_off, int32_t* new_len,
                 int32_t* status, void* workspace, size_t workspace_bytes, void* stream);

/*
 * One verify round committing several caches, each with its own geometry.
 *
 * Source: mlxcel #2865 "perf(speculative): commit per-row accepts in batched
 * DFlash", Summary -- besides the target's attention cache, the drafter's
 * context is still one rectangular prefix shared by the batch, which keeps
 * the drafter's walk short; the follow-up it records is to give the drafter a
 * per-row context as well. That is the same per-row commit applied to the
 * drafter's cache, whose layer count, head count, head size, capacity and
 * prefix lengths are its own.
 *
 * The same operation as verify_round (arg max, fold accept, bonus), then, for
 * every set i of sets[0..n_sets-1], the per-row commit of kv_compact_per_row
 * on that set's tensors with its own H, S_cap, D, elem_bytes, prefix_len,
 * src_off and new_len, and with keep[b] = accept[b] + 1 for every set (the
 * committed token's slot and the accepted drafts'), max_keep = L.
 *
 * sets     HOST array of n_sets descriptors (0 <= n_sets; NULL when 0); each
 *          descriptor's fields are as kv_compact_per_row's arguments of the
 *          same names (tensors is a HOST array of DEVICE pointers).
 * status   optional int32 on the device, shared by every set: bit 0 is OR-ed
 *          in for any row any set leaves untouched (never cleared).
 * Other arguments, sizes and the workspace as verify_round. Every argument of
 * every set is checked before the first launch.
 */
typedef struct {
  void* const* tensors;
  int32_t n_tensors;
  int32_t H, S_cap, D, elem_bytes;
  const int32_t* prefix_len;
  const int32_t* src_off;
  int32_t* new_len;
} vq_kv_set;
int verify_round_multi(const void* h, int B, int L, int K, int N, const uint32_t* qw,
                       const uint16_t* scales, const uint16_t* biases, int act_dtype,
                       const int32_t* tokens, int32_t* target, int32_t* accept, int32_t* bonus,
                       const vq_kv_set* sets, int n_sets, int32_t* status, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * Attention of the verify block over the per-row KV cache, one layer.
 *
 * Source: mlxcel #2865 "perf(speculative): commit per-row accepts in batched
 * DFlash", Summary and commit message -- with per-row accept counts, the
 * rotary embedding and the attention of the verify block use every row's own
 * logical positions, and each query is kept from seeing the stale gap between
 * its row's valid prefix and the verify slots the rectangular cache shares
 * across rows.
 *
 * For each batch row b (P = prefix_len[b], S = src_off[b]) and block position
 * j = 0..L-1, at logical position P + j:
 *   1. the block's key k_new[b][j][h] is rotated at P + j, rounded to the
 *      storage type and written to slot S + j of k_cache; v_new[b][j][h] is
 *      copied to slot S + j of v_cache;
 *   2. the query q[b][j][hq] is rotated at P + j and rounded to the storage
 *      type; it reads KV head hq / (Hq / Hkv);
 *   3. out[b][j][hq] = softmax over the visible slots of scale * (q . k),
 *      applied to v, where the visible slots are 0..P-1 (the row's valid
 *      prefix) and S..S+j (the block, causally). Slots P..S-1 (the stale gap)
 *      and everything after S + j are masked.
 * Rotation: within the first rotary_dim dimensions, dimension i < rotary_dim/2
 * pairs with i + rotary_dim/2 and turns by pos * theta^(-2i/rotary_dim)
 * (y_i = x_i cos - x_{i+h} sin, y_{i+h} = x_{i+h} cos + x_i sin); dimensions
 * from rotary_dim on are not rotated. The softmax and its sums are fp32.
 *
 * q, out        [B][L][Hq][D]; k_new, v_new [B][L][Hkv][D];
 * k_cache, v_cache  [B][Hkv][S_cap][D], keys stored rotated. All 16-bit of
 *               `dtype` (VQ_BF16 or VQ_F16); q, k_new, v_new and the caches
 *               16-byte aligned, out 2-byte aligned; no tensor overlaps
 *               another.
 * prefix_len, src_off  int32 [B] on the device.
 * status        optional int32 on the device: a row with P < 0, S < P or
 *               S + L > S_cap is left untouched in the caches, gets zero
 *               output, and bit 0 is OR-ed into *status (never cleared).
 * workspace     not used (verify_attention_workspace_bytes returns 0 for
 *               every shape); any pointer and size, null and 0 included.
 * Sizes         B >= 1, 1 <= L <= 64, Hq a multiple of Hkv, D 64 or 128
 *               (VQ_EUNSUPPORTED otherwise), L <= S_cap <= 2^24, rotary_dim
 *               even in 0..D, theta > 0 when rotary_dim > 0.
 * One kernel, in clusters of 8 blocks: a cluster per (batch row, KV head,
 * group of 64 query rows). Each block rotates the group's queries, takes
 * every 8th chunk of 64 keys with an online softmax, and the cluster merges
 * its blocks' partial results through distributed shared memory; the
 * clusters of the first query group also append the block to the caches.
 */
size_t verify_attention_workspace_bytes(int B, int L, int Hq, int Hkv, int D, int S_cap);
int verify_attention(const void* q, const void* k_new, const void* v_new, void* k_cache,
                     void* v_cache, const int32_t* prefix_len, const int32_t* src_off,
                     void* out, int B, int L, int Hq, int Hkv, int D, int S_cap, int rotary_dim,
                     double theta, double scale, int dtype, int32_t* status, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * The launch plan a projection or arg max call would use, computed on the
 * host for a device with `sm_count` SMs (no device is touched): which kernel,
 * how deep its shared-memory ring is, how K is split, the grid, and the
 * shared memory and workspace it needs. For capacity planning and tests; the
 * calls themselves use the current device's SM count. The pages have no
 * counterpart: this reports how this library maps a shape onto the GPU.
 * Returns VQ_OK and fills *out, or the code the call itself would return for
 * this shape (VQ_EINVAL, VQ_EUNSUPPORTED); out must be a host pointer.
 */
typedef struct {
  int32_t kernel;       /* 0 mma.sync, x per stage; 1 mma.sync, per-block x table;
                           2 mma.sync, prepared x slices; 3 tcgen05 */
  int32_t rows_padded;  /* M rounded up to the kernel's row tile (8, 16, 32 or 64) */
  int32_t stages;       /* depth of the shared-memory stage ring (512 k per stage) */
  int32_t prefetch;     /* stages whose weights are requested before the wait */
  int32_t k_splits;     /* K splits per 128-row block (1 = none) */
  int32_t units;        /* 128-row blocks x K splits */
  int32_t grid;         /* blocks launched (persistent over units) */
  int32_t launches;     /* kernels per call */
  int64_t smem_bytes;   /* dynamic shared memory per block */
  int64_t workspace_bytes;
} vq_plan_t;
int vq_plan(int M, int K, int N, int act_dtype, int argmax, int sm_count, vq_plan_t* out);

/* A short description of a VQ_* code. Never NULL. */
const char* vq_strerror(int code);

/*
 * Reads the library's device status word of the current device into *out
 * (host pointer): bit 0 = a kernel gave up waiting on one of its own
 * pipeline barriers and returned early, so its outputs are not valid.
 * Synchronizes `stream`. If clear != 0 the word is reset to 0 afterwards.
 */
int vq_device_error(int32_t* out, int clear, void* stream);

/*
 * Self-test of the bounded waits the pipelined kernels rely on: one block
 * waits, with the kernels' own wait helpers, on an mbarrier that completes and
 * on one that nothing ever arrives at. The stuck waits give up after the
 * kernels' wait limit (2^31 SM cycles, about a second each; the call runs for
 * about two seconds) and flag their status word instead of hanging. The pages
 * have no counterpart: this checks that a stuck pipeline in this library ends
 * with an error status.
 *
 * status  int32[2] on the device, zero before the call: bit 0 of status[0] is
 *         set by the aborting waits, bit 0 of status[1] by the teardown wait.
 * report  int64[8] on the device: [0] completed-barrier wait succeeded (1),
 *         [1] its SM cycles, [2] stuck wait succeeded (0), [3] its cycles,
 *         [4] the block's abort flag afterwards (1), [5] a second warp's wait
 *         on the stuck barrier succeeded (0), [6] its cycles (short: it sees
 *         the abort flag), [7] cycles of the teardown wait on it.
 * The library's own status word (vq_device_error) is not touched.
 */
int vq_wait_selftest(int32_t* status, int64_t* report, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VQ_H_ */
