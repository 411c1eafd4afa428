// C-ABI entry points of the W4 projections (vq_linear, vq_vocab_argmax),
// their host-side planning and tensor-map encoding, and the status calls.
#include <cstring>
#include <mutex>

#include "vq_gemm.cuh"
#include "vq_tc.cuh"

namespace vq {

// Status word of the device kernels (see vq_device_error).
__device__ int32_t g_vq_device_error = 0;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices];
int32_t* g_err_ptr[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) return VQ_ECUDA;
  if (*dev < 0 || *dev >= kMaxDevices) return VQ_EUNSUPPORTED;
  return VQ_OK;
}

int device_state(int* sms, int32_t** err) {
  int dev;
  int rc = current_device(&dev);
  if (rc) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      return VQ_ECUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_vq_device_error) != cudaSuccess) return VQ_ECUDA;
    g_err_ptr[dev] = static_cast<int32_t*>(p);
    g_sms[dev] = n;
  }
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return VQ_ECUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  if (sms) *sms = g_sms[dev];
  if (err) *err = g_err_ptr[dev];
  return VQ_OK;
}

// Encoded tensor maps, cached per host thread: a verify step calls the same
// projections on the same weights every time, and cuTensorMapEncodeTiled is a
// driver call per map, four per call. A map depends only on what the key
// holds (address, type, sizes, strides, box, swizzle), never on the contents,
// so a buffer freed and allocated again at the same address reuses its map.
struct TmKey {
  const void* ptr;
  int32_t dev, dt, rank, sw, l2, pad;
  uint64_t dims[3], strides[2];
  uint32_t box[3];
};
struct TmEntry {
  TmKey key;
  CUtensorMap map;
};
constexpr int kTmCache = 64;
thread_local TmEntry t_tm[kTmCache];
thread_local int t_tm_used = 0, t_tm_next = 0;

int encode(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, int rank,
           const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
           CUtensorMapSwizzle sw, CUtensorMapL2promotion l2) {
  TmKey k;
  memset(&k, 0, sizeof k);   // the padding takes part in the comparison
  k.ptr = ptr;
  if (cudaGetDevice(&k.dev) != cudaSuccess) return VQ_ECUDA;
  k.dt = (int32_t)dt;
  k.rank = rank;
  k.sw = (int32_t)sw;
  k.l2 = (int32_t)l2;
  for (int i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) k.strides[i] = strides[i];
  for (int i = 0; i < t_tm_used; ++i) {
    // the address first: a lookup scans up to kTmCache entries on every call
    if (t_tm[i].key.ptr == ptr && memcmp(&t_tm[i].key, &k, sizeof k) == 0) {
      *m = t_tm[i].map;
      return VQ_OK;
    }
  }
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(m, dt, (cuuint32_t)rank, const_cast<void*>(ptr), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, l2,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return VQ_ECUDA;
  TmEntry& e = t_tm[t_tm_next];
  e.key = k;
  e.map = *m;
  t_tm_next = (t_tm_next + 1) % kTmCache;
  if (t_tm_used < kTmCache) ++t_tm_used;
  return VQ_OK;
}

int encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
              uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle sw, CUtensorMapL2promotion l2) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  return encode(m, dt, ptr, 2, dims, strides, box, sw, l2);
}

// x viewed as [K/inner][M][inner] (group-major), so one box brings a stage's
// x for all M rows as [group][row][128 bytes]. The strides are not
// increasing; if the driver rejects that view the caller falls back to one
// 2-D box per group.
int encode_x3d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, int M, int K,
               int elem_bytes, int box_rows, int box_groups) {
  const uint64_t inner = 128 / elem_bytes;
  const cuuint64_t dims[3] = {inner, (cuuint64_t)M, (cuuint64_t)K / inner};
  const cuuint64_t strides[2] = {(cuuint64_t)K * elem_bytes, 128};
  const cuuint32_t box[3] = {(cuuint32_t)inner, (cuuint32_t)box_rows, (cuuint32_t)box_groups};
  return encode(m, dt, ptr, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int red_bytes(int MT) {
  switch (MT) {
    case 1:
      return Cfg<1>::RED;
    case 2:
      return Cfg<2>::RED;
    case 4:
      return Cfg<4>::RED;
    default:
      return Cfg<8>::RED;
  }
}

// Shape of one launch: everything but the pointers.
struct Plan {
  int MT, MP, D, pre, pace, KT, RB, S, n_units, grid;
  bool sb_plain;    // K % 512 != 0: scales and biases by plain loads (see GemmParams)
  bool red_alias;   // K-slice partials in the stage ring (one unit per block)
  int stage_bytes, off_x, off_s, off_b, xbox_bytes, xm, tab_bytes, xs_stage;
  uint32_t tx_bytes;
  size_t smem;
  size_t ws_xp_bytes;    // prepared x table (start of the workspace), 0 if none
  size_t ws_cnt_bytes, ws_bytes;
};

int check_shape(int M, int K, int N, int act) {
  if (act != VQ_BF16 && act != VQ_F16 && act != VQ_F32) return VQ_EINVAL;
  if (M < 1 || M > 64 || K < 64 || N < 1 || K % 64 != 0) return VQ_EINVAL;
  if (act == VQ_F32 && M > 32) return VQ_EUNSUPPORTED;
  return VQ_OK;
}

int make_plan(int M, int K, int N, int act, bool argmax, int sms, Plan* pl) {
  int rc = check_shape(M, K, N, act);
  if (rc) return rc;
  Plan p{};
  p.MT = M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8;
  p.MP = 8 * p.MT;
  const bool f32 = act == VQ_F32;
  const int n_xbox = f32 ? 16 : 8;
  // Where x comes from:
  //  xm = 2 (vq_linear, 16-bit x, M <= 16): slices of scaled fp16
  //         fragments prepared by a small kernel before the projection, one
  //         per stage and n8 tile, copied into the stage next to its weights;
  //  xm = 1 (arg max, 16-bit x, M <= 8, several row blocks per block): the
  //         block converts all of x once into a table (the conversion costs
  //         about what two row blocks of the main loop save);
  //  xm = 0 otherwise: x for the stage by TMA, [group][8*MT rows][128 B] with
  //         rows >= M zero-filled, and a table of group sums per block.
  // K not a multiple of 512: a last, partial stage whose groups past K arrive
  // zero-filled, and scales and biases by plain loads (their rows are then
  // not the 16-byte multiples a TMA tensor map needs) on the per-stage x
  // kernels (xm = 0, xm = 3); the x-table and prepared-slice variants take
  // whole stages only
  p.KT = (K + kBK - 1) / kBK;
  p.sb_plain = K % kBK != 0;
  p.RB = (int)(((long long)N + kBN - 1) / kBN);
  p.S = 1;
  if (!argmax && 2 * p.RB < sms) {
    // The projection is bound by HBM bandwidth, which half the SMs already
    // saturate, so K is split only when the row blocks alone would leave
    // more than half the SMs idle (a narrow N); the split then fills the
    // SMs in one wave. Each extra slice adds 2*M*N*4 bytes of partials.
    p.S = sms / p.RB;
    if (p.S > p.KT) p.S = p.KT;
    if (p.S < 1) p.S = 1;
  }
  p.n_units = p.RB * p.S;
  p.grid = p.n_units < sms ? p.n_units : sms;
  //  xm = 3 (16-bit x, M > 16, no K split): the tensor-core (tcgen05)
  //         kernel; x for the stage by TMA as for xm = 0, X_g from a small
  //         kernel (vq_linear) or summed per block (arg max). Measured at
  //         K=5120, N=17408: M=24..64 it beats the mma.sync kernel (27.6 vs
  //         33.1 us at M=24, 33.8 vs 59.2 us at M=64); at M=16 it does not
  //         (25.7 vs 20.6 us), its per-group MMA issue and handoffs cost more
  //         than the 16-row mma.sync work they replace.
  if (!f32 && p.MT >= 4 && p.S == 1) {
    // a table of X_g for all of K if it leaves room for two stages, else
    // X_g per stage from the x tile (two stages' worth, double-buffered)
    const int sb = tc_stage_bytes(p.MP);
    int tab_tc = (int)round_up((size_t)tc_xs_bytes(p.KT * kBK, p.MP), 1024);
    p.xs_stage = 0;
    if ((kSmemLimit - 1024 - kTcMiscBytes - tab_tc) / sb < 2) {
      p.xs_stage = 1;
      tab_tc = (int)round_up((size_t)2 * 8 * p.MP * 4, 1024);
    }
    int D = (kSmemLimit - 1024 - kTcMiscBytes - tab_tc) / sb;
    if (D > kMaxStages) D = kMaxStages;
    if (D >= 2) {
      p.xm = 3;
      p.D = D;
      p.pre = D < 3 ? D : 3;
      p.stage_bytes = sb;
      p.off_x = kTcOffX;
      p.off_s = kTcOffS;
      p.off_b = kTcOffB;
      p.xbox_bytes = 128 * p.MP;
      p.tx_bytes = (uint32_t)(2 * kWeightBoxBytes + (p.sb_plain ? 0 : 2 * kBN * 16) +
                              8 * 128 * p.MP);
      p.tab_bytes = tab_tc;
      p.red_alias = false;
      p.smem = 1024 + (size_t)D * sb + tab_tc + kTcMiscBytes;
      p.ws_cnt_bytes = 0;
      if (argmax) {
        p.ws_xp_bytes = 0;
        p.ws_bytes = round_up((size_t)M * 8 + 4, 16);
      } else {
        p.ws_xp_bytes = p.xs_stage ? 0 : round_up((size_t)tc_xs_bytes(p.KT * kBK, p.MP), 256);
        p.ws_bytes = p.ws_xp_bytes;
      }
      *pl = p;
      return VQ_OK;
    }
  }
  // The K-slice partial sums are only needed after a unit's last stage: with
  // one unit per block they can share the stage ring instead of taking
  // shared memory of their own.
  p.red_alias = p.n_units <= p.grid && red_bytes(p.MT) > 0;
  const int red = p.red_alias ? 0 : red_bytes(p.MT);
  const long long rb_total = ((long long)N + kBN - 1) / kBN;
  const long long per_block = (rb_total + sms - 1) / sms;
  const bool mt1_16 = !f32 && p.MT == 1 && !p.sb_plain;
  if (!f32 && p.MT <= 2 && !p.sb_plain && !argmax)
    p.xm = 2;
  else if (mt1_16 && argmax && xt_table_bytes(K) <= kMaxXtBytes && per_block >= 3)
    p.xm = 1;
  else
    p.xm = 0;
  p.ws_xp_bytes = (p.xm == 2) ? round_up((size_t)p.KT * p.MT * kSliceBytes, 256) : 0;
  int tab;
  int x_bytes;   // x bytes a stage receives
  if (p.xm == 2) {
    p.xbox_bytes = 0;
    p.off_x = xs_stage_off_x();
    p.off_s = xt_stage_off_s();
    p.off_b = xt_stage_off_s() + kBN * 16;
    p.stage_bytes = xs_stage_bytes(p.MT);
    tab = 0;
    x_bytes = p.MT * kSliceBytes;
  } else if (p.xm == 1) {
    p.xbox_bytes = 0;
    p.off_x = 0;
    p.off_s = xt_stage_off_s();
    p.off_b = xt_stage_off_s() + kBN * 16;
    p.stage_bytes = xt_stage_bytes();
    tab = xt_table_bytes(K);
    x_bytes = 0;
  } else {
    p.xbox_bytes = 128 * p.MP;
    p.off_x = stage_off_x();
    p.off_s = stage_off_s(act, p.MT);
    p.off_b = stage_off_b(act, p.MT);
    p.stage_bytes = stage_bytes(act, p.MT);
    tab = xsum_bytes(p.KT * kBK, p.MT);
    if (tab > kMaxXsumBytes) return VQ_EUNSUPPORTED;
    x_bytes = n_xbox * p.xbox_bytes;
  }
  tab = (int)round_up((size_t)tab, 1024);
  p.D = (kSmemLimit - 1024 - misc_bytes(argmax) - red - tab) / p.stage_bytes;
  if (p.D > kMaxStages) p.D = kMaxStages;
  if (p.D < 2) return VQ_EUNSUPPORTED;
  // stages whose weights a block requests before it waits for the kernel
  // before it in the stream. Three measured best for the projection: the
  // first stages' x then queues behind fewer weight bytes.
  p.pre = p.D < 3 ? p.D : 3;
  // With prepared slices the kernel spaces those requests; measured at M=8,
  // K=5120, N=17408 in a stream of calls: 1500 cycles 10.93 us per call,
  // 800 cycles 11.06, none 11.35, 2500 cycles 11.74.
  p.pace = p.xm == 2 ? 1500 : 0;
  p.tx_bytes = (uint32_t)(2 * kWeightBoxBytes + (p.sb_plain ? 0 : 2 * kBN * 16) + x_bytes);
  p.tab_bytes = tab;
  p.smem = 1024 + (size_t)p.D * p.stage_bytes + misc_bytes(argmax) + red + tab;
  // workspace: [prepared x table][split-K counters][split-K partials]
  if (argmax) {
    p.ws_cnt_bytes = 0;
    p.ws_bytes = round_up((size_t)M * 8 + 4, 16);
  } else if (p.S > 1) {
    p.ws_cnt_bytes = round_up((size_t)p.RB * 4, 16);
    p.ws_bytes = p.ws_xp_bytes + p.ws_cnt_bytes + (size_t)p.S * M * N * 4;
  } else {
    p.ws_cnt_bytes = 0;
    p.ws_bytes = p.ws_xp_bytes;
  }
  *pl = p;
  return VQ_OK;
}

// Blocks whose top-2 candidates the workspace of vq_vocab_argmax_top2 holds;
// the arg max grid is capped to it (it is persistent over row blocks).
constexpr int kMaxTop2Blocks = 256;

int run_gemm(const void* x, int M, int K, int N, const uint32_t* qw, const uint16_t* scales,
             const uint16_t* biases, int act, bool argmax, void* y, int32_t* amax, float* maxval,
             void* ws, size_t ws_bytes, void* stream, float* second = nullptr) {
  int rc = check_shape(M, K, N, act);
  if (rc) return rc;
  if (!x || !qw || !scales || !biases) return VQ_EINVAL;
  if (argmax ? !amax : !y) return VQ_EINVAL;
  if (((uintptr_t)x | (uintptr_t)qw | (uintptr_t)scales | (uintptr_t)biases) & 15u)
    return VQ_EALIGN;
  if (((uintptr_t)y | (uintptr_t)amax | (uintptr_t)maxval | (uintptr_t)second) & 3u)
    return VQ_EALIGN;
  int sms;
  int32_t* err;
  if ((rc = device_state(&sms, &err))) return rc;
  Plan pl;
  if ((rc = make_plan(M, K, N, act, argmax, sms, &pl))) return rc;
  size_t need = pl.ws_bytes;
  if (second) {
    if (pl.grid > kMaxTop2Blocks) pl.grid = kMaxTop2Blocks;
    need = round_up((size_t)M * 8 + 4, 16) + (size_t)kMaxTop2Blocks * M * 16;
  }
  if (need) {
    if (!ws || ws_bytes < need) return VQ_EWORKSPACE;
    if ((uintptr_t)ws & 15u) return VQ_EALIGN;
  }

  GemmLaunch L;
  GemmParams& p = L.p;
  p = GemmParams{};
  p.x = x;
  p.M = M;
  p.K = K;
  p.N = N;
  p.KT = pl.KT;
  p.S = pl.S;
  p.n_units = pl.n_units;
  p.D = pl.D;
  p.pre = pl.pre;
  p.pace = pl.pace;
  p.red_alias = pl.red_alias ? 1 : 0;
  p.stage_bytes = pl.stage_bytes;
  p.off_x = pl.off_x;
  p.off_s = pl.off_s;
  p.off_b = pl.off_b;

  p.tx_bytes = pl.tx_bytes;
  p.sb_plain = pl.sb_plain ? 1 : 0;
  p.scales = scales;
  p.biases = biases;
  p.xm = pl.xm;
  p.xs_stage = pl.xs_stage;
  p.tab_bytes = pl.tab_bytes;
  p.y = y;
  p.err = err;
  // extents for bounds-checked builds, from the sizes of the call and of the
  // workspace the caller passed (not from the plan's own counts)
  p.y_elems = (size_t)M * N;
  if (argmax) {
    p.keys = static_cast<unsigned long long*>(ws);
    p.done = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + (size_t)M * 8);
    p.argmax = amax;
    p.maxval = maxval;
    if (second) {
      p.second = second;
      const size_t off = round_up((size_t)M * 8 + 4, 16);
      p.cand = reinterpret_cast<uint4*>(static_cast<char*>(ws) + off);
      p.cand_elems = ws_bytes > off ? (ws_bytes - off) / 16 : 0;
    }
  } else {
    if (pl.ws_xp_bytes) p.xprep = ws;
    if (pl.S > 1) {
      p.cnt = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + pl.ws_xp_bytes);
      p.part = reinterpret_cast<float*>(static_cast<char*>(ws) + pl.ws_xp_bytes + pl.ws_cnt_bytes);
      const size_t off = pl.ws_xp_bytes + pl.ws_cnt_bytes;
      p.part_elems = ws_bytes > off ? (ws_bytes - off) / 4 : 0;
    }
  }

  const bool f32 = act == VQ_F32;
  const CUtensorMapDataType xdt = act == VQ_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                  : act == VQ_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  if ((rc = encode_2d(&L.tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT32, qw, (uint64_t)K / 8, (uint64_t)N,
                      (uint64_t)K / 2, 32, kBN, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B)))
    return rc;
  if (pl.sb_plain) {
    // rows of K/32 bytes: no tensor map can describe them; the kernel loads
    // scales and biases itself and never reads these maps
    memset(&L.tm_s, 0, sizeof L.tm_s);
    memset(&L.tm_b, 0, sizeof L.tm_b);
  } else {
    if ((rc = encode_2d(&L.tm_s, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, (uint64_t)K / 64,
                        (uint64_t)N, (uint64_t)K / 32, 8, kBN, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B)))
      return rc;
    if ((rc = encode_2d(&L.tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT16, biases, (uint64_t)K / 64,
                        (uint64_t)N, (uint64_t)K / 32, 8, kBN, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B)))
      return rc;
  }
  const int eb = f32 ? 4 : 2;
  // box rows = 8*MT >= M: the rows past M are out of range and arrive zeroed;
  // the x-table variant takes every group of K in one box. The prepared-slice
  // plan reads x only in the slice kernel (plain loads): no map.
  if (pl.xm == 2) {
    memset(&L.tm_x, 0, sizeof L.tm_x);
    p.x3d = 0;
  } else if (encode_x3d(&L.tm_x, xdt, x, M, K, eb, pl.MP, pl.xm == 1 ? K / 64 : kBK / (128 / eb)) == VQ_OK) {
    p.x3d = 1;
  } else {
    if ((rc = encode_2d(&L.tm_x, xdt, x, (uint64_t)K, (uint64_t)M, (uint64_t)K * eb, 128 / eb,
                        (uint32_t)pl.MP, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B)))
      return rc;
    p.x3d = 0;
  }

  L.grid = pl.grid;
  L.MT = pl.MT;
  L.argmax = argmax;
  L.smem = pl.smem;
  L.stream = static_cast<cudaStream_t>(stream);
  switch (act) {
    case VQ_BF16:
      return launch_gemm_bf16(L);
    case VQ_F16:
      return launch_gemm_f16(L);
    default:
      return launch_gemm_f32(L);
  }
}

}  // namespace

int num_sms_current_device(int* out) { return device_state(out, nullptr); }
int device_error_word(int32_t** out) { return device_state(nullptr, out); }
int encode_rows_sw128(CUtensorMap* m, const void* ptr, uint64_t row_elems, uint64_t rows,
                      uint32_t box_rows) {
  return encode_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, ptr, row_elems, rows, row_elems * 2, 64,
                   box_rows, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
}

}  // namespace vq

using namespace vq;

extern "C" size_t vq_linear_workspace_bytes(int M, int K, int N, int act_dtype) {
  int sms;
  if (device_state(&sms, nullptr)) return 0;
  Plan pl;
  if (make_plan(M, K, N, act_dtype, false, sms, &pl)) return 0;
  return pl.ws_bytes;
}

extern "C" int vq_linear(const void* x, int M, int K, int N, const uint32_t* qw,
                         const uint16_t* scales, const uint16_t* biases, void* y, int act_dtype,
                         void* workspace, size_t workspace_bytes, void* stream) {
  return run_gemm(x, M, K, N, qw, scales, biases, act_dtype, false, y, nullptr, nullptr,
                  workspace, workspace_bytes, stream);
}

namespace {
// The device address of page-locked host memory that the current device can
// address (false for anything else; the error a failed query leaves is cleared).
bool device_view(const void* h, void** d) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer) return false;
  *d = a.devicePointer;
  return true;
}
}  // namespace

extern "C" int vq_linear_host(const void* x_host, int M, int K, int N, const uint32_t* qw,
                              const uint16_t* scales, const uint16_t* biases, void* y_host,
                              int act_dtype, void* x_dev, void* y_dev, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (!x_host || !y_host || !x_dev || !y_dev) return VQ_EINVAL;
  if (M < 1 || K < 1 || N < 1) return VQ_EINVAL;
  if (act_dtype != VQ_BF16 && act_dtype != VQ_F16 && act_dtype != VQ_F32) return VQ_EINVAL;
  const size_t eb = act_dtype == VQ_F32 ? 4 : 2;
  const size_t x_bytes = (size_t)M * K * eb, y_bytes = (size_t)M * N * eb;
  // the shape, the device buffers and the workspace are checked before
  // anything is enqueued (the weights' arguments by vq_linear itself)
  int sms = 0;
  int rc = device_state(&sms, nullptr);
  if (rc) return rc;
  Plan pl;
  if ((rc = make_plan(M, K, N, act_dtype, false, sms, &pl))) return rc;
  if (((uintptr_t)x_dev & 15u) || ((uintptr_t)y_dev & 3u)) return VQ_EALIGN;
  const size_t need = pl.ws_bytes;
  if (need && (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 15u)))
    return VQ_EWORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Where the device can address the page-locked host buffers (unified
  // addressing; on a coherent CPU-GPU link as on GB300 at full link speed),
  // the prepared-slice plan's slice kernel reads x from them directly and,
  // without a K split, the projection writes y into them directly; otherwise
  // (and for every other plan) the buffers are copied through x_dev and y_dev.
  const void* xs = x_dev;
  void* yd = y_dev;
  void* xv = nullptr;
  void* yv = nullptr;
  const bool zx = pl.xm == 2 && device_view(x_host, &xv) && !((uintptr_t)xv & 15u);
  const bool zy = pl.xm == 2 && pl.S == 1 && device_view(y_host, &yv) && !((uintptr_t)yv & 3u);
  if (zx) {
    xs = xv;
  } else if (cudaMemcpyAsync(x_dev, x_host, x_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) {
    return VQ_ECUDA;
  }
  if (zy) yd = yv;
  rc = run_gemm(xs, M, K, N, qw, scales, biases, act_dtype, false, yd, nullptr, nullptr, workspace,
                workspace_bytes, stream);
  if (rc || zy) return rc;
  return cudaMemcpyAsync(y_host, y_dev, y_bytes, cudaMemcpyDeviceToHost, st) == cudaSuccess
             ? VQ_OK
             : VQ_ECUDA;
}

extern "C" size_t vq_vocab_argmax_workspace_bytes(int M) {
  if (M < 1 || M > 64) return 0;
  return round_up((size_t)M * 8 + 4, 16);
}

extern "C" int vq_vocab_argmax(const void* x, int M, int K, int N, const uint32_t* qw,
                               const uint16_t* scales, const uint16_t* biases, int act_dtype,
                               int32_t* argmax, float* maxval, void* workspace,
                               size_t workspace_bytes, void* stream) {
  return run_gemm(x, M, K, N, qw, scales, biases, act_dtype, true, nullptr, argmax, maxval,
                  workspace, workspace_bytes, stream);
}

extern "C" int vq_plan(int M, int K, int N, int act_dtype, int argmax, int sm_count,
                       vq_plan_t* out) {
  if (!out || sm_count < 1) return VQ_EINVAL;
  Plan pl;
  const int rc = make_plan(M, K, N, act_dtype, argmax != 0, sm_count, &pl);
  if (rc) return rc;
  out->kernel = pl.xm;
  out->rows_padded = pl.MP;
  out->stages = pl.D;
  out->prefetch = pl.pre;
  out->k_splits = pl.S;
  out->units = pl.n_units;
  out->grid = pl.grid;
  out->launches = (pl.xm == 2 || (pl.xm == 3 && !argmax && !pl.xs_stage)) ? 2 : 1;
  out->smem_bytes = (int64_t)pl.smem;
  out->workspace_bytes = (int64_t)pl.ws_bytes;
  return VQ_OK;
}

extern "C" size_t vq_vocab_argmax_top2_workspace_bytes(int M) {
  if (M < 1 || M > 64) return 0;
  return round_up((size_t)M * 8 + 4, 16) + (size_t)kMaxTop2Blocks * M * 16;
}

extern "C" int vq_vocab_argmax_top2(const void* x, int M, int K, int N, const uint32_t* qw,
                                    const uint16_t* scales, const uint16_t* biases, int act_dtype,
                                    int32_t* argmax, float* maxval, float* second,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (!second) return VQ_EINVAL;
  return run_gemm(x, M, K, N, qw, scales, biases, act_dtype, true, nullptr, argmax, maxval,
                  workspace, workspace_bytes, stream, second);
}

// ---------------------------------------------------------------- no-alloc arg max
// Scratch of vq_vocab_argmax_noalloc: one file-scope device array instead of
// a caller-provided workspace. It holds the arg max workspace of every valid
// M (M * 8 + 4 bytes rounded up to 16, at most 528 bytes for M = 64). Every
// GPU that loads this library holds it until the process exits, and every
// call on that GPU shares it.
namespace vq {
namespace {
constexpr size_t kNoAllocScratchBytes = 1024;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
void* g_noalloc_ptr[kMaxDevices];   // device address of the array, per device
}  // namespace
}  // namespace vq

extern "C" int vq_vocab_argmax_noalloc(const void* x, int M, int K, int N, const uint32_t* qw,
                                       const uint16_t* scales, const uint16_t* biases,
                                       int act_dtype, int32_t* argmax, float* maxval,
                                       void* stream) {
  if (M < 1 || M > 64) return VQ_EINVAL;
  const size_t need = vq_vocab_argmax_workspace_bytes(M);
  if (need == 0 || need > kNoAllocScratchBytes) return VQ_EWORKSPACE;
  int dev;
  int rc = current_device(&dev);
  if (rc) return rc;
  void* scratch;
  {
    // set-up, once per device with that device current: the host-side name
    // of the array is not a device address, so look the address up
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_noalloc_ptr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return VQ_ECUDA;
      g_noalloc_ptr[dev] = p;
    }
    scratch = g_noalloc_ptr[dev];
  }
  // the array keeps whatever the last call left: clear the keys and the
  // block counter, which must start at zero, on the call's stream
  if (cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return VQ_ECUDA;
  return run_gemm(x, M, K, N, qw, scales, biases, act_dtype, true, nullptr, argmax, maxval,
                  scratch, need, stream);
}

extern "C" const char* vq_strerror(int code) {
  switch (code) {
    case VQ_OK:
      return "ok";
    case VQ_EINVAL:
      return "invalid argument (shape, size or enum out of range)";
    case VQ_EALIGN:
      return "pointer not aligned as required";
    case VQ_ECUDA:
      return "CUDA runtime error";
    case VQ_EUNSUPPORTED:
      return "valid but outside the compiled variants";
    case VQ_EWORKSPACE:
      return "workspace missing or too small";
    default:
      return "unknown status";
  }
}

extern "C" int vq_device_error(int32_t* out, int clear, void* stream) {
  if (!out) return VQ_EINVAL;
  int rc = device_state(nullptr, nullptr);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_vq_device_error, sizeof v, 0, cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return VQ_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return VQ_ECUDA;
  if (clear) {
    const int32_t zero = 0;
    if (cudaMemcpyToSymbolAsync(g_vq_device_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice,
                                s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return VQ_ECUDA;
  }
  *out = v;
  return VQ_OK;
}
