// Host side of the fused, chunked top-K KL loss: argument checks, workspace carving,
// tensor-map encoding, the chunk loop and the kernel launches behind include/fckl.h.
//
// Forward, per chunk of positions ("Fused, chunked KL loss": project the chunk, fold it
// into the running loss, drop it):
//   preprocess -> fwd_logits_lse (tcgen05, online max/sum-exp + top-K gather) -> combine
// then one fixed-order sum of the per-position losses.
// Backward, per chunk (the chunk's logits are recomputed):
//   preprocess -> bwd_logit_grad (tcgen05, G to a bf16 chunk x V slab)
//              -> dH = G W (tcgen05, split over V, fp32 partials) -> dH reduce
//              -> dW (+)= G^T H_chunk (tcgen05, TMA store on the first chunk, TMA
//                 reduce-add afterwards)
// fckl_forward_backward runs both per chunk (lse of a position depends on its own row only),
// ordering the chunk's cache slots once.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/fckl.h"
#include "simt.cuh"
#include "tc_gemm.cuh"

namespace fckl {
namespace {

enum Kind {
  KIND_PREPROCESS = 0,
  KIND_FWD_LOGITS,
  KIND_FWD_COMBINE,
  KIND_LOSS_REDUCE,
  KIND_BWD_GRAD,
  KIND_BWD_DH,
  KIND_BWD_DH_REDUCE,
  KIND_BWD_DW,
  KIND_CVT,
  KIND_SELFTEST,
  KIND_TOPK_LOGITS,
  KIND_TOPK_THRESHOLD,
  KIND_TOPK_COLLECT,
  KIND_TOPK_SELECT,
  KIND_FWD_LOGITS_KEEP,
  KIND_BWD_GRAD_KEPT,
  KIND_TOPK_LOGITS_KEEP,
  KIND_TOPK_COLLECT_KEPT,
  KIND_BWD_GRAD_KEPT_SIDE,      // the instances launched on the second stream beside a product
  KIND_TOPK_COLLECT_KEPT_SIDE,
  KIND_TOPK_SELECT_SIDE,
  KIND_COUNT
};
const char* const kKindNames[KIND_COUNT] = {"preprocess",     "fwd_logits_lse", "fwd_combine",
                                            "loss_reduce",    "bwd_logit_grad", "bwd_dH_gemm",
                                            "bwd_dH_reduce",  "bwd_dW_gemm",    "cvt_inputs",
                                            "wait_timeout_selftest", "topk_logits_stats", "topk_threshold",
                                            "topk_collect",           "topk_select",
                                            "fwd_logits_keep",        "bwd_grad_from_logits",
                                            "topk_logits_keep",       "topk_collect_from_logits",
                                            "bwd_grad_from_logits_side", "topk_collect_from_logits_side",
                                            "topk_select_side"};

// ------------------------------------------------------------------ process state
std::mutex g_mu;
std::mutex g_setup_mu;  // serialises one-time per-device kernel set-up
char g_last_error[512] = "";
long long g_launches = 0;
bool g_prof = false;
struct ProfRec {
  int kind;
  cudaEvent_t a, b;
};
std::vector<ProfRec> g_prof_recs;
std::vector<cudaEvent_t> g_event_pool;

void set_error(const char* what, cudaError_t e) {
  std::lock_guard<std::mutex> lk(g_mu);
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s", what, cudaGetErrorString(e));
}
void set_error_text(const char* what) {
  std::lock_guard<std::mutex> lk(g_mu);
  snprintf(g_last_error, sizeof(g_last_error), "%s", what);
}

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Runs `launch` (which enqueues one kernel on `s`), counts it, optionally brackets it
// with events, and converts a launch error into FCKL_ERR_CUDA.
template <class F>
int launch(int kind, cudaStream_t s, const char* what, F&& fn) {
  cudaEvent_t a = nullptr, b = nullptr;
  bool prof;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    prof = g_prof;
    if (prof) {
      a = take_event();
      b = take_event();
    }
  }
  if (prof) cudaEventRecord(a, s);
  fn();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error(what, e);
    if (prof) {
      std::lock_guard<std::mutex> lk(g_mu);
      g_event_pool.push_back(a);
      g_event_pool.push_back(b);
    }
    return FCKL_ERR_CUDA;
  }
  if (prof) cudaEventRecord(b, s);
  std::lock_guard<std::mutex> lk(g_mu);
  ++g_launches;
  if (prof) g_prof_recs.push_back({kind, a, b});
  return FCKL_OK;
}

// ------------------------------------------------------------------ device info
struct DevInfo {
  bool init = false;
  int id = 0, sms = 0, major = 0, minor = 0;
  bool pre_attr_done = false;
};
DevInfo g_dev[64];

int device_info(DevInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error("cudaGetDevice", e);
    return FCKL_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) return FCKL_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& d = g_dev[dev];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      snprintf(g_last_error, sizeof(g_last_error), "cudaDeviceGetAttribute failed");
      return FCKL_ERR_CUDA;
    }
    d.id = dev;
    d.init = true;
  }
  *out = &d;
  if (d.major != 10 || d.minor != 3) return FCKL_ERR_UNSUPPORTED;
  return FCKL_OK;
}

// ------------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D map over a row-major [dim1][dim0] array with row pitch `pitch_bytes`, zero fill
// outside the array; 128-byte swizzle unless asked otherwise.
int make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t dim0, uint64_t dim1,
             uint64_t pitch_bytes, uint32_t box0, uint32_t box1,
             CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto enc = encode_fn();
  if (!enc) {
    set_error_text("cuTensorMapEncodeTiled entry point not found");
    return FCKL_ERR_CUDA;
  }
  cuuint64_t gdim[2] = {dim0, dim1};
  cuuint64_t gstride[1] = {pitch_bytes};
  cuuint32_t box[2] = {box0, box1};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), gdim, gstride, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::lock_guard<std::mutex> lk(g_mu);
    snprintf(g_last_error, sizeof(g_last_error),
             "cuTensorMapEncodeTiled failed (%d): dims %llu x %llu pitch %llu box %u x %u", static_cast<int>(r),
             static_cast<unsigned long long>(dim0), static_cast<unsigned long long>(dim1),
             static_cast<unsigned long long>(pitch_bytes), box0, box1);
    return FCKL_ERR_CUDA;
  }
  return FCKL_OK;
}

// ------------------------------------------------------------------ plan / workspace
constexpr int MAX_SPLITS = 4;    // K-splits of the dH product

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t rup(int64_t a, int64_t b) { return cdiv(a, b) * b; }

struct Plan {
  int64_t N;
  int d, V, K, chunk, dt;
  int rows_alloc;  // chunk rounded up to 256 rows (the tile of an SM pair)
  int tiles_v;     // vocabulary tiles of 256
  int ldG;         // row pitch (elements) of the bf16 gradient slab
  int bn_d;        // N-tile of the dH / dW products
  size_t off_status, off_sidx, off_sp, off_S, off_T, off_pm, off_pl, off_pc, off_rowloss, off_G, off_dhp,
      off_Hb, off_Wb, off_Ht, off_Wt, total;
  // A second set of the per-chunk buffers (ordered slots, S, T, tile statistics, gradient slab,
  // bf16 H copy), after everything above; present when there is more than one chunk. With it
  // (a workspace of total_overlap bytes) the one call forms chunk c's G on a second stream
  // while chunk c+1's forward runs.
  size_t alt_sidx, alt_sp, alt_S, alt_T, alt_pm, alt_pl, alt_pc, alt_G, alt_Hb, total_overlap;
};

// The plan as seen by a chunk in buffer set 1: the same layout with the second set's offsets.
Plan second_set(const Plan& p) {
  Plan q = p;
  q.off_sidx = p.alt_sidx;
  q.off_sp = p.alt_sp;
  q.off_S = p.alt_S;
  q.off_T = p.alt_T;
  q.off_pm = p.alt_pm;
  q.off_pl = p.alt_pl;
  q.off_pc = p.alt_pc;
  q.off_G = p.alt_G;
  q.off_Hb = p.alt_Hb;
  return q;
}

// N-tile of the dH and dW products (over d). 256 columns: an SM pair stages 128 each, two
// 64-wide swizzle blocks; a d that is not a multiple of 256 ends in a ragged tile.
int choose_bn(int) { return 256; }

int check_shape(int64_t N, int d, int V, int K, int chunk, int dt) {
  if (N < 1 || d < 1 || V < 1 || K < 1 || chunk < 1) return FCKL_ERR_ARG;
  if (dt != FCKL_BF16 && dt != FCKL_F32) return FCKL_ERR_ARG;
  if (K > V || K > K_LIMIT) return FCKL_ERR_UNSUPPORTED;
  if (d % 8 != 0) return FCKL_ERR_UNSUPPORTED;
  if (N > (int64_t(1) << 40) || V > (1 << 30) || d > (1 << 20)) return FCKL_ERR_UNSUPPORTED;
  // The rows of one chunk are counted in int (rounded up to 256) and multiply V and d in the
  // workspace layout; 2^24 rows keeps every product far from overflow (and any workspace of
  // such a chunk would exceed device memory anyway).
  if (std::min<int64_t>(chunk, N) > (int64_t(1) << 24)) return FCKL_ERR_UNSUPPORTED;
  return FCKL_OK;
}

Plan make_plan(int64_t N, int d, int V, int K, int chunk, int dt) {
  Plan p{};
  p.N = N;
  p.d = d;
  p.V = V;
  p.K = K;
  p.chunk = static_cast<int>(std::min<int64_t>(chunk, N));
  p.dt = dt;
  p.rows_alloc = static_cast<int>(rup(p.chunk, 256));
  p.tiles_v = static_cast<int>(cdiv(V, VOCAB_TILE));
  p.ldG = static_cast<int>(rup(V, 8));
  p.bn_d = choose_bn(d);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t r = o;
    o = static_cast<size_t>(rup(static_cast<int64_t>(o + bytes), 1024));
    return r;
  };
  const size_t R = p.rows_alloc;
  p.off_status = take(256);
  p.off_sidx = take(R * K * 4);
  p.off_sp = take(R * K * 4);
  p.off_S = take(R * 4);
  p.off_T = take(R * 4);
  p.off_pm = take(static_cast<size_t>(p.tiles_v) * R * 4);
  p.off_pl = take(static_cast<size_t>(p.tiles_v) * R * 4);
  p.off_pc = take(static_cast<size_t>(p.tiles_v) * R * 4);
  p.off_rowloss = take(static_cast<size_t>(N) * 4);
  p.off_G = take(R * p.ldG * 2);
  p.off_dhp = take(static_cast<size_t>(MAX_SPLITS) * R * d * 4);
  p.off_Hb = dt == FCKL_F32 ? take(R * d * 2) : o;
  p.off_Wb = dt == FCKL_F32 ? take(static_cast<size_t>(V) * d * 2) : o;
  p.off_Ht = dt == FCKL_F32 ? take(R * d * 4) : o;
  p.off_Wt = dt == FCKL_F32 ? take(static_cast<size_t>(V) * d * 4) : o;
  p.total = o;
  if (N > p.chunk) {
    p.alt_sidx = take(R * K * 4);
    p.alt_sp = take(R * K * 4);
    p.alt_S = take(R * 4);
    p.alt_T = take(R * 4);
    p.alt_pm = take(static_cast<size_t>(p.tiles_v) * R * 4);
    p.alt_pl = take(static_cast<size_t>(p.tiles_v) * R * 4);
    p.alt_pc = take(static_cast<size_t>(p.tiles_v) * R * 4);
    p.alt_G = take(R * p.ldG * 2);
    p.alt_Hb = dt == FCKL_F32 ? take(R * d * 2) : o;
  }
  p.total_overlap = o;
  return p;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ------------------------------------------------------------------ kernel launchers
#ifndef FCKL_CG
#define FCKL_CG 2  // CTAs per MMA in the four products: 2 = SM pairs (cta_group::2)
#endif
constexpr int CG = FCKL_CG;
constexpr int TILE_M = BM * CG;  // rows of one MMA tile

// Operand maps of the bf16 products, whose ring stages hold kps K-blocks (64 bf16 of K each):
// two in the logits products (both operands K-major), one in dH and dW. 3-D maps fetch a whole
// stage of an operand in one copy, laid out in shared memory as the engine expects; where the
// needed dimension is not a multiple of 64 (or a K-major stage is one K-block) the 2-D map is
// used and the engine issues one copy per K-block (K-major) or per 64-wide block (MN-major).
int encode3(CUtensorMap* m, const void* base, const cuuint64_t (&gdim)[3], const cuuint64_t (&gstride)[2],
            const cuuint32_t (&box)[3]) {
  auto enc = encode_fn();
  if (!enc) {
    set_error_text("cuTensorMapEncodeTiled entry point not found");
    return FCKL_ERR_CUDA;
  }
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstride, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::lock_guard<std::mutex> lk(g_mu);
    snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled (3-D) failed (%d): %llu x %llu x %llu",
             static_cast<int>(r), static_cast<unsigned long long>(gdim[0]), static_cast<unsigned long long>(gdim[1]),
             static_cast<unsigned long long>(gdim[2]));
    return FCKL_ERR_CUDA;
  }
  return FCKL_OK;
}

// K-major operand, a row-major bf16 [rows][K] array read box_rows rows at a time. With two
// K-blocks per stage and K % 64 == 0: 3-D (64 K-values, rows, K / 64 blocks), a box of
// 64 x box_rows x 2 is a stage's two K-blocks, each rows x 128 bytes.
int map_kmajor(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint64_t pitch_bytes, uint32_t box_rows,
               int kps, int* is3d) {
  *is3d = CG == 2 && kps == 2 && K % 64 == 0;
  if (*is3d) return encode3(m, base, {64, rows, K / 64}, {pitch_bytes, 128}, {64, box_rows, 2});
  return make_map(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, rows, pitch_bytes, BK, box_rows);
}

// MN-major operand, a row-major bf16 [K][MN] array (MN contiguous). 3-D (64 MN-values, K rows,
// MN / 64 blocks) when MN % 64 == 0: a box of 64 x (kps * 64) x 2 is a stage of two 64-wide MN
// blocks, kps * 8 KB apart; else 2-D boxes of 64 x (kps * 64), one per MN block.
int map_mnmajor(CUtensorMap* m, const void* base, uint64_t MN, uint64_t K, uint64_t pitch_bytes, int kps,
                int* is3d) {
  *is3d = CG == 2 && MN % 64 == 0;
  const uint32_t krows = static_cast<uint32_t>(kps * BK);
  if (*is3d) return encode3(m, base, {64, K, MN / 64}, {pitch_bytes, 128}, {64, krows, 2});
  return make_map(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, MN, K, pitch_bytes, 64, krows);
}
constexpr int KPS_LOGITS = 2;  // K-blocks per stage of the bf16 logits products
constexpr int KPS_GRAD = 1;    // of dH and dW


// Launch configuration of one engine instantiation: one CTA (pair) per SM (pair), as many
// clusters as can be resident at once. The first call on a device sets the shared-memory limit
// and asks the occupancy calculator; *clusters receives the resident cluster count.
template <int BN, bool AMN, bool BMN, int EPI, bool TF32 = false>
int tc_setup(DevInfo* di, cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int* clusters) {
  auto k = tc_gemm_kernel<CG, BN, AMN, BMN, EPI, TF32>;
  constexpr uint32_t smem = TcSmem<CG, BN, (TF32 || AMN || BMN) ? 1 : 2>::DYN_BYTES;
  static_assert(smem <= 232448, "shared memory budget");
  static bool attr_done[64] = {};  // one flag per device for this instantiation
  static int max_clusters[64] = {};
  const int dev = di->id;
  *cfg = cudaLaunchConfig_t{};
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg->blockDim = dim3(NUM_THREADS);
  cfg->dynamicSmemBytes = smem;
  cfg->attrs = attr;
  cfg->numAttrs = CG > 1 ? 1 : 0;
  {
    std::lock_guard<std::mutex> lk(g_setup_mu);  // one-time per-device set-up, any host thread
    if (!attr_done[dev]) {
      cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) {
        set_error("cudaFuncSetAttribute", e);
        return FCKL_ERR_CUDA;
      }
      int n = di->sms / CG;
      if (CG > 1) {
        cfg->gridDim = dim3(static_cast<unsigned>(CG * n));
        int m = 0;
        if (cudaOccupancyMaxActiveClusters(&m, k, cfg) == cudaSuccess && m > 0) n = std::min(n, m);
        cudaGetLastError();
      }
      max_clusters[dev] = n;
      attr_done[dev] = true;
    }
  }
  *clusters = max_clusters[dev];
  return FCKL_OK;
}

// Persistent launch: as many clusters as can be resident, capped by the number of work units.
template <int BN, bool AMN, bool BMN, int EPI, bool TF32 = false>
int launch_tc(int kind, DevInfo* di, const TcParams& p, cudaStream_t s, const char* what) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  int max_clusters = 0;
  int st = tc_setup<BN, AMN, BMN, EPI, TF32>(di, &cfg, attr, &max_clusters);
  if (st) return st;
  const int clusters = static_cast<int>(std::min<int64_t>(p.num_units, max_clusters));
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * CG));
  cfg.stream = s;
  auto k = tc_gemm_kernel<CG, BN, AMN, BMN, EPI, TF32>;
  return launch(kind, s, what, [&] { cudaLaunchKernelEx(&cfg, k, p); });
}

// Copies of fp32 inputs: tf32-rounded into t32 (for the logits products) and/or bf16 into b16
// (for the dH and dW products); either may be null.
int launch_cvt(const float* src, void* t32, void* b16, int64_t n, DevInfo* di, cudaStream_t s) {
  const int grid = static_cast<int>(std::min<int64_t>(cdiv(n / 4, 256), int64_t(di->sms) * 8));
  return launch(KIND_CVT, s, "cvt_inputs", [&] {
    cvt_inputs_kernel<<<std::max(grid, 1), 256, 0, s>>>(src, static_cast<float*>(t32),
                                                        static_cast<__nv_bfloat16*>(b16), n);
  });
}

int launch_preprocess(const Plan& pl, const int32_t* idx, const float* logp, int rows, uint8_t* w, unsigned* status,
                      DevInfo* di, cudaStream_t s) {
  const int blocks = static_cast<int>(cdiv(rows, PRE_WARPS));
  const size_t smem = static_cast<size_t>(PRE_WARPS) * pl.K * 8;
  if (smem > 48 * 1024) {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!di->pre_attr_done) {
      cudaError_t e = cudaFuncSetAttribute(preprocess_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(PRE_WARPS * K_LIMIT * 8));
      if (e != cudaSuccess) {
        set_error("cudaFuncSetAttribute(preprocess)", e);
        return FCKL_ERR_CUDA;
      }
      di->pre_attr_done = true;
    }
  }
  return launch(KIND_PREPROCESS, s, "preprocess", [&] {
    preprocess_kernel<<<blocks, 32 * PRE_WARPS, smem, s>>>(
        idx, logp, rows, pl.K, pl.V, reinterpret_cast<int*>(w + pl.off_sidx), reinterpret_cast<float*>(w + pl.off_sp),
        reinterpret_cast<float*>(w + pl.off_S), reinterpret_cast<float*>(w + pl.off_T), status);
  });
}

int common_checks(const void* H, const void* W, int dt, const int32_t* idx, const float* logp, int64_t N, int d,
                  int V, int K, int chunk, void* ws, size_t ws_bytes, Plan* pl, DevInfo** di) {
  int st = check_shape(N, d, V, K, chunk, dt);
  if (st) return st;
  if (!H || !W || !idx || !logp || !ws) return FCKL_ERR_ARG;
  if (!aligned(H, 16) || !aligned(W, 16) || !aligned(ws, 256) || !aligned(idx, 4) || !aligned(logp, 4))
    return FCKL_ERR_ARG;
  *pl = make_plan(N, d, V, K, chunk, dt);
  if (ws_bytes < pl->total) return FCKL_ERR_WORKSPACE;
  return device_info(di);
}

// Everything one call needs to run the per-chunk steps.
struct Run {
  Plan pl;   // buffer set 0
  Plan pl1;  // buffer set 1 (second_set(pl)), used by the overlapped one call
  const Plan& plan(int set) const { return set ? pl1 : pl; }
  DevInfo* di = nullptr;
  cudaStream_t s = nullptr;
  uint8_t* w = nullptr;  // workspace
  unsigned* status = nullptr;
  const void* H = nullptr;
  const void* Wraw = nullptr;  // the caller's W (bf16, or fp32 read as tf32 by the logits products)
  const void* Wb = nullptr;  // W as bf16 (the caller's W, or its bf16 copy for the dH product)
  int dtype = FCKL_BF16;
  const int32_t* idx = nullptr;
  const float* logp = nullptr;
  const float* weight = nullptr;  // [N] or null
  float* lse = nullptr;           // [N]
  float* rl = nullptr;            // [N] per-position loss
  float grad_scale = 1.f;
  void* dH = nullptr;
  float* dW = nullptr;
  int splits = 1;  // K-splits of the dH product
  CUtensorMap tmW_k, tmW_mn, tmDW, tmDWp;
  int w_k_3d = 0, w_mn_3d = 0;  // tmW_k / tmW_mn are 3-D maps
};

// Clears the status word, rounds fp32 W to bf16 when needed and encodes the maps over W
// (and dW) shared by every chunk.
int run_begin(Run& r, bool backward) {
  const Plan& pl = r.pl;
  cudaError_t e = cudaMemsetAsync(r.status, 0, sizeof(unsigned), r.s);
  if (e != cudaSuccess) {
    set_error("cudaMemsetAsync", e);
    return FCKL_ERR_CUDA;
  }
  int st;
  if (r.dtype == FCKL_F32) {  // tf32 copy for the logits products, bf16 copy for the dH product
    if ((st = launch_cvt(static_cast<const float*>(r.Wraw), r.w + pl.off_Wt, backward ? r.w + pl.off_Wb : nullptr,
                         int64_t(pl.V) * pl.d, r.di, r.s)))
      return st;
    r.Wraw = r.w + pl.off_Wt;
    if (backward) r.Wb = r.w + pl.off_Wb;
  }
  const int d = pl.d, V = pl.V;
  // The logits products read W K-major: bf16, or the tf32-rounded copy of an fp32 W (32
  // values per 128-byte stage row).
  if (r.dtype == FCKL_F32) {
    if ((st = make_map(&r.tmW_k, r.Wraw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, d, V, uint64_t(d) * 4, BK / 2,
                       VOCAB_TILE / CG)))
      return st;
  } else if ((st = map_kmajor(&r.tmW_k, r.Wb, d, V, uint64_t(d) * 2, VOCAB_TILE / CG, KPS_LOGITS, &r.w_k_3d))) {
    return st;
  }
  if (!backward) return FCKL_OK;
  if ((st = map_mnmajor(&r.tmW_mn, r.Wb, d, V, uint64_t(d) * 2, KPS_GRAD, &r.w_mn_3d))) return st;
  if ((st = make_map(&r.tmDW, r.dW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, d, V, uint64_t(d) * 4, 32, 32))) return st;
  if ((st = make_map(&r.tmDWp, r.dW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, d, V, uint64_t(d) * 4, 256, BM,
                     CU_TENSOR_MAP_SWIZZLE_NONE)))
    return st;
  // K-splits of dH = G W (K = V): the count that best fills the SM pairs.
  const int kb_v = static_cast<int>(cdiv(V, BK));
  const int tiles = static_cast<int>(cdiv(pl.chunk, TILE_M) * cdiv(d, pl.bn_d));
  double best = -1.0;
  for (int sp = 1; sp <= MAX_SPLITS && sp <= kb_v; ++sp) {
    const int kbps = static_cast<int>(cdiv(kb_v, sp));
    if (cdiv(kb_v, kbps) != sp) continue;
    const int64_t units = int64_t(tiles) * sp;
    const int64_t slots = r.di->sms / CG;
    const double eff = double(units) / double(cdiv(units, slots) * slots);
    if (eff > best + 0.02) {
      best = eff;
      r.splits = sp;
    }
  }
  // FCKL_SPLITS (environment, 1..MAX_SPLITS) overrides the count for tuning; a count whose
  // K-blocks would leave a split empty is ignored. Results then differ from the default only
  // by the fp32 summation order of the partials.
  if (const char* env = std::getenv("FCKL_SPLITS")) {
    const int sp = std::atoi(env);
    if (sp >= 1 && sp <= MAX_SPLITS && sp <= kb_v && cdiv(kb_v, cdiv(kb_v, sp)) == sp) r.splits = sp;
  }
  return FCKL_OK;
}

// Orders the chunk's cache slots; returns the chunk's H rows as the logits products read them
// (*Hl: bf16, or for fp32 inputs a tf32-rounded copy) and as the dW product reads them (*Hc:
// bf16; for fp32 inputs a bf16 copy, made only when `backward`).
int chunk_prepare(Run& r, int set, int64_t r0, int rows, const void** Hl, const void** Hc, bool backward) {
  const Plan& pl = r.plan(set);
  int st = launch_preprocess(pl, r.idx + r0 * pl.K, r.logp + r0 * pl.K, rows, r.w, r.status, r.di, r.s);
  if (st) return st;
  const size_t esz = r.dtype == FCKL_F32 ? 4 : 2;
  *Hl = static_cast<const uint8_t*>(r.H) + static_cast<size_t>(r0) * pl.d * esz;
  *Hc = *Hl;
  if (r.dtype == FCKL_F32) {
    if ((st = launch_cvt(static_cast<const float*>(*Hl), r.w + pl.off_Ht, backward ? r.w + pl.off_Hb : nullptr,
                         int64_t(rows) * pl.d, r.di, r.s)))
      return st;
    *Hl = r.w + pl.off_Ht;
    *Hc = r.w + pl.off_Hb;
  }
  return FCKL_OK;
}

// Map of a chunk's hidden states as the logits products read them (K-major, 128 rows a box).
int map_logits_A(const Run& r, CUtensorMap* m, const void* Hl, int rows, int* is3d) {
  const int d = r.pl.d;
  if (r.dtype == FCKL_F32) {
    *is3d = 0;
    return make_map(m, Hl, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, d, rows, uint64_t(d) * 4, BK / 2, BM);
  }
  return map_kmajor(m, Hl, d, rows, uint64_t(d) * 2, BM, KPS_LOGITS, is3d);
}
// K-blocks of the logits products: 64 bf16 or 32 fp32 values of d per stage.
int logits_kblocks(const Run& r) { return static_cast<int>(cdiv(r.pl.d, r.dtype == FCKL_F32 ? BK / 2 : BK)); }

// Forward of one chunk: logits tiles -> per-tile (max, sum-exp, gathered sum) -> lse and loss.
// With keep, exp(z - tile max) is also stored (fp16) into the gradient slab for the chunk's
// backward.
int chunk_forward(Run& r, int set, int64_t r0, int rows, const void* Hl, bool keep = false) {
  const Plan& pl = r.plan(set);
  uint8_t* w = r.w;
  int st;
  TcParams p;
  memset(&p, 0, sizeof(p));
  if ((st = map_logits_A(r, &p.tmA, Hl, rows, &p.a_3d))) return st;
  p.tmB = r.tmW_k;
  p.b_3d = r.w_k_3d;
  const int kbl = logits_kblocks(r);
  p.sch = {static_cast<int>(cdiv(rows, TILE_M)), pl.tiles_v, kbl, 1, kbl, 1};
  p.num_units = p.sch.m_blocks * p.sch.n_blocks;
  p.status = r.status;
  p.rows_valid = rows;
  p.V = pl.V;
  p.K = pl.K;
  p.sidx = reinterpret_cast<const int*>(w + pl.off_sidx);
  p.sp = reinterpret_cast<const float*>(w + pl.off_sp);
  p.S = reinterpret_cast<const float*>(w + pl.off_S);
  p.pm = reinterpret_cast<float*>(w + pl.off_pm);
  p.pl = reinterpret_cast<float*>(w + pl.off_pl);
  p.pc = reinterpret_cast<float*>(w + pl.off_pc);
  p.ld_part = pl.rows_alloc;
  if (keep) {
    if ((st = make_map(&p.tmC, w + pl.off_G, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, pl.V, rows, uint64_t(pl.ldG) * 2, 64,
                       32)))
      return st;
    p.c_xlim = pl.V;
    p.c_ylim = rows;
    st = r.dtype == FCKL_F32
             ? launch_tc<VOCAB_TILE, false, false, EPI_FWD_KEEP, true>(KIND_FWD_LOGITS_KEEP, r.di, p, r.s,
                                                                       "fwd_logits_keep")
             : launch_tc<VOCAB_TILE, false, false, EPI_FWD_KEEP>(KIND_FWD_LOGITS_KEEP, r.di, p, r.s, "fwd_logits_keep");
  } else {
    st = r.dtype == FCKL_F32
             ? launch_tc<VOCAB_TILE, false, false, EPI_FWD_STATS, true>(KIND_FWD_LOGITS, r.di, p, r.s,
                                                                        "fwd_logits_lse")
             : launch_tc<VOCAB_TILE, false, false, EPI_FWD_STATS>(KIND_FWD_LOGITS, r.di, p, r.s, "fwd_logits_lse");
  }
  if (st) return st;
  const int cblocks = static_cast<int>(cdiv(rows, 32));
  const float* wc = r.weight ? r.weight + r0 : nullptr;
  cudaStream_t s = r.s;
  float* lse = r.lse + r0;
  float* rl = r.rl + r0;
  return launch(KIND_FWD_COMBINE, s, "fwd_combine", [&] {
    combine_kernel<<<cblocks, 32 * COMBINE_WARPS, 0, s>>>(p.pm, p.pl, p.pc, pl.rows_alloc, pl.tiles_v, rows, p.S,
                                           reinterpret_cast<const float*>(w + pl.off_T), wc, lse, rl);
  });
}

// G = scale * w_n * (S softmax(z) - p_sparse) of one chunk, from its recomputed logits.
int grad_recompute(Run& r, int set, int64_t r0, int rows, const void* Hl) {
  const Plan& pl = r.plan(set);
  const int V = pl.V;
  uint8_t* w = r.w;
  cudaStream_t s = r.s;
  void* G = w + pl.off_G;
  const int mbr = static_cast<int>(cdiv(rows, TILE_M));
  int st;
  TcParams pg;
  memset(&pg, 0, sizeof(pg));
  if ((st = map_logits_A(r, &pg.tmA, Hl, rows, &pg.a_3d))) return st;
  pg.tmB = r.tmW_k;
  pg.b_3d = r.w_k_3d;
  if ((st = make_map(&pg.tmC, G, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, V, rows, uint64_t(pl.ldG) * 2, 64, 32)))
    return st;
  const int kbl = logits_kblocks(r);
  pg.sch = {mbr, pl.tiles_v, kbl, 1, kbl, 1};
  pg.num_units = mbr * pl.tiles_v;
  pg.status = r.status;
  pg.rows_valid = rows;
  pg.V = V;
  pg.K = pl.K;
  pg.sidx = reinterpret_cast<const int*>(w + pl.off_sidx);
  pg.sp = reinterpret_cast<const float*>(w + pl.off_sp);
  pg.S = reinterpret_cast<const float*>(w + pl.off_S);
  pg.lse = r.lse + r0;
  pg.wrow = r.weight ? r.weight + r0 : nullptr;
  pg.gscale = r.grad_scale;
  pg.c_xlim = V;
  pg.c_ylim = rows;
  if (r.dtype == FCKL_F32)
    return launch_tc<VOCAB_TILE, false, false, EPI_LOGIT_GRAD, true>(KIND_BWD_GRAD, r.di, pg, s, "bwd_logit_grad");
  return launch_tc<VOCAB_TILE, false, false, EPI_LOGIT_GRAD>(KIND_BWD_GRAD, r.di, pg, s, "bwd_logit_grad");
}

constexpr int GRAD_BLOCKS_PER_SM = 8;  // blocks per SM of the G pass when it runs alone

// The same G formed in place from what the chunk's forward kept in the slab (fp16
// exp(z - tile max), with the tile maxima in pm), on stream s: alone (GRAD_BLOCKS_PER_SM blocks
// per SM) or, with beside, one block per SM next to a tensor-core product.
int grad_from_kept(Run& r, int set, int64_t r0, int rows, cudaStream_t s, bool beside) {
  const Plan& pl = r.plan(set);
  const int V = pl.V;
  uint8_t* w = r.w;
  const int64_t units = int64_t(rows) * cdiv(V, KG_SEG);
  const int grid =
      static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(units, int64_t(r.di->sms) * (beside ? 1 : GRAD_BLOCKS_PER_SM))));
  __nv_bfloat16* G = reinterpret_cast<__nv_bfloat16*>(w + pl.off_G);
  const int* sidx = reinterpret_cast<const int*>(w + pl.off_sidx);
  const float* spp = reinterpret_cast<const float*>(w + pl.off_sp);
  const float* S = reinterpret_cast<const float*>(w + pl.off_S);
  const float* pm = reinterpret_cast<const float*>(w + pl.off_pm);
  const float* lse = r.lse + r0;
  const float* wr = r.weight ? r.weight + r0 : nullptr;
  const float gsc = r.grad_scale;
  const int K = pl.K, ldp = pl.rows_alloc;
  const int64_t ld = pl.ldG;
  if (beside) {
    static bool done[64] = {};
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!done[r.di->id]) {
      cudaError_t e = cudaFuncSetAttribute(logit_grad_kernel<true>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                           cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) {
        set_error("cudaFuncSetAttribute(logit_grad_kernel)", e);
        return FCKL_ERR_CUDA;
      }
      done[r.di->id] = true;
    }
  }
  return launch(beside ? KIND_BWD_GRAD_KEPT_SIDE : KIND_BWD_GRAD_KEPT, s, "bwd_grad_from_logits", [&] {
    if (beside)
      logit_grad_kernel<true><<<grid, GRAD_THREADS, 0, s>>>(G, ld, rows, V, K, sidx, spp, S, lse, wr, gsc, pm, ldp);
    else
      logit_grad_kernel<false><<<grid, GRAD_THREADS, 0, s>>>(G, ld, rows, V, K, sidx, spp, S, lse, wr, gsc, pm, ldp);
  });
}

// The gradient products of one chunk whose G is in its slab: dH_chunk = G W and
// dW (+)= G^T H_chunk.
int chunk_products(Run& r, int set, int64_t r0, int rows, const void* Hc) {
  const Plan& pl = r.plan(set);
  const int d = pl.d, V = pl.V;
  uint8_t* w = r.w;
  cudaStream_t s = r.s;
  void* G = w + pl.off_G;
  float* dhp = reinterpret_cast<float*>(w + pl.off_dhp);
  const int mbr = static_cast<int>(cdiv(rows, TILE_M));
  const int kb_v = static_cast<int>(cdiv(V, BK));
  int st;

  // --- dH_chunk = G W, split over the vocabulary into fp32 partials, then summed
  const int nbd = static_cast<int>(cdiv(d, pl.bn_d));
  const int splits = r.splits;
  TcParams ph;
  memset(&ph, 0, sizeof(ph));
  if ((st = map_kmajor(&ph.tmA, G, V, rows, uint64_t(pl.ldG) * 2, BM, KPS_GRAD, &ph.a_3d))) return st;
  ph.tmB = r.tmW_mn;
  ph.b_3d = r.w_mn_3d;
  if ((st = make_map(&ph.tmC, dhp, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, d, uint64_t(splits) * pl.rows_alloc,
                     uint64_t(d) * 4, 32, 32)))
    return st;
  const int kbps = static_cast<int>(cdiv(kb_v, splits));
  ph.sch = {mbr, nbd, kb_v, splits, kbps, 1};
  ph.num_units = mbr * nbd * splits;
  ph.status = r.status;
  ph.c_split_rows = pl.rows_alloc;
  ph.c_reduce = 0;
  ph.c_xlim = d;
  ph.c_ylim = splits * pl.rows_alloc;
  if ((st = launch_tc<256, false, true, EPI_STORE_F32>(KIND_BWD_DH, r.di, ph, s, "bwd_dH_gemm"))) return st;
  {
    const int64_t n4 = int64_t(rows) * d / 4;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(cdiv(n4, 256), int64_t(r.di->sms) * 8)));
    const int64_t stride = int64_t(pl.rows_alloc) * d;
    if (r.dtype == FCKL_F32) {
      float* out = static_cast<float*>(r.dH) + static_cast<size_t>(r0) * d;
      st = launch(KIND_BWD_DH_REDUCE, s, "bwd_dH_reduce",
                  [&] { dh_reduce_kernel<float><<<grid, 256, 0, s>>>(dhp, splits, stride, rows, d, out); });
    } else {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(r.dH) + static_cast<size_t>(r0) * d;
      st = launch(KIND_BWD_DH_REDUCE, s, "bwd_dH_reduce", [&] {
        dh_reduce_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(dhp, splits, stride, rows, d, out);
      });
    }
    if (st) return st;
  }

  // --- dW (+)= G^T H_chunk: the first chunk stores, later chunks reduce-add
  TcParams pw;
  memset(&pw, 0, sizeof(pw));
  if ((st = map_mnmajor(&pw.tmA, G, V, rows, uint64_t(pl.ldG) * 2, KPS_GRAD, &pw.a_3d))) return st;
  if ((st = map_mnmajor(&pw.tmB, Hc, d, rows, uint64_t(d) * 2, KPS_GRAD, &pw.b_3d))) return st;
  pw.tmC = r.tmDW;
  pw.tmP = r.tmDWp;
  const int kb_r = static_cast<int>(cdiv(rows, BK));
  pw.sch = {static_cast<int>(cdiv(V, TILE_M)), nbd, kb_r, 1, kb_r, 0};
  pw.num_units = pw.sch.m_blocks * nbd;
  pw.status = r.status;
  pw.c_split_rows = 0;
  pw.c_reduce = r0 > 0 ? 1 : 0;
  pw.c_prefetch = pw.c_reduce;
  pw.c_xlim = d;
  pw.c_ylim = V;
  return launch_tc<256, true, true, EPI_STORE_F32>(KIND_BWD_DW, r.di, pw, s, "bwd_dW_gemm");
}

// Backward of one chunk: G = scale * w_n * (S softmax(z) - p_sparse) from recomputed logits
// (or, with keep, from what the chunk's forward kept in the slab), then the gradient products.
int chunk_backward(Run& r, int set, int64_t r0, int rows, const void* Hl, const void* Hc, bool keep = false) {
  int st = keep ? grad_from_kept(r, set, r0, rows, r.s, false) : grad_recompute(r, set, r0, rows, Hl);
  if (st) return st;
  return chunk_products(r, set, r0, rows, Hc);
}

// Id of the current CUDA context, unique within the process (a device reset, or another
// context of the device, gets a new one); 0 if it cannot be read.
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS)
    return id;
  return 0;
}

// Second stream of the one call and its fork/join events, one set per host thread and device
// (calls from different host threads never share them), created on first use and kept for the
// context they were made in: under a new context of the device (after a device reset) a new
// set is made (the old handles belong to the destroyed context and are not touched).
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  cudaEvent_t join_set[2] = {nullptr, nullptr};  // the side work of each buffer set (top-K builder)
  unsigned long long ctx = 0;
};
thread_local SideStream t_side[64];

int side_stream(int dev, SideStream** out) {
  SideStream& x = t_side[dev];
  const unsigned long long id = current_context_id();
  if (!x.s || (id != 0 && id != x.ctx)) {
    SideStream n;
    cudaError_t e = cudaStreamCreateWithFlags(&n.s, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&n.join, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&n.join_set[0], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&n.join_set[1], cudaEventDisableTiming);
    if (e != cudaSuccess) {
      set_error("side stream set-up", e);
      for (cudaEvent_t ev : n.join_set)
        if (ev) cudaEventDestroy(ev);
      if (n.join) cudaEventDestroy(n.join);
      if (n.fork) cudaEventDestroy(n.fork);
      if (n.s) cudaStreamDestroy(n.s);
      return FCKL_ERR_CUDA;
    }
    n.ctx = current_context_id();  // read after the creation, which makes the context current
    x = n;
  }
  *out = &x;
  return FCKL_OK;
}

// Whether overlapping a chunk's side work with the next chunk's tensor-core pass pays. The side
// kernels run one block per SM beside the product, so they take longer than alone; the product
// must be long enough to cover them and the per-chunk fork and join. Measured on the one call
// (V = 128256, chunk 2048): d = 3072 and 2048 gain 1-1.5%, d = 1536 and 2560 are even, d = 1024
// loses 5%; at V = 32000, d = 2048 loses 2% and d = 1024 10%. Rule: a chunk's projection of at
// least 5e11 FLOPs and, where the side pass scales with V like the projection (the G pass), d of
// at least 2048. FCKL_OVERLAP (environment) forces it on (1) or off (0) when the workspace allows.
bool overlap_pays(int64_t rows, int d, int V, bool side_scales_with_v) {
  if (const char* env = std::getenv("FCKL_OVERLAP")) {
    if (env[0] == '0' && env[1] == '\0') return false;
    if (env[0] == '1' && env[1] == '\0') return true;
  }
  const double flops = 2.0 * double(rows) * double(d) * double(V);
  return flops >= 5e11 && (!side_scales_with_v || d >= 2048);
}

// Makes stream s wait for event ev (stream order only, no host wait).
int wait_event(cudaStream_t s, cudaEvent_t ev) {
  const cudaError_t e = cudaStreamWaitEvent(s, ev, 0);
  if (e != cudaSuccess) {
    set_error("join from the side stream", e);
    return FCKL_ERR_CUDA;
  }
  return FCKL_OK;
}

// The one call over chunks c = 0, 1, ... with chunk c in buffer set c % 2: after chunk c's
// forward and chunk c+1's preprocessing, chunk c's G is formed on the second stream (one
// block per SM, which fits beside a tensor-core product's CTA) while chunk c+1's forward runs
// on the caller's stream; the caller's stream then waits for G before chunk c's gradient
// products. The last chunk's G runs on the caller's stream. Every kernel computes what it
// does in the sequential order from the same inputs, so the results are bitwise the same.
// The HBM-bound G pass thus runs under a tensor-bound product instead of between two.
int run_overlapped(Run& r, SideStream* side) {
  const int64_t N = r.pl.N, C = r.pl.chunk;
  int64_t r0 = 0;
  int rows = static_cast<int>(std::min<int64_t>(C, N));
  const void *Hl = nullptr, *Hc = nullptr;
  int st;
  if ((st = chunk_prepare(r, 0, r0, rows, &Hl, &Hc, true))) return st;
  if ((st = chunk_forward(r, 0, r0, rows, Hl, true))) return st;
  for (int set = 0;; set ^= 1) {
    const int64_t n0 = r0 + C;
    if (n0 >= N) {
      if ((st = grad_from_kept(r, set, r0, rows, r.s, false))) return st;
      return chunk_products(r, set, r0, rows, Hc);
    }
    const int nrows = static_cast<int>(std::min<int64_t>(C, N - n0));
    const void *nHl = nullptr, *nHc = nullptr;
    // G waits for the next chunk's preprocessing too, so that it is released together with
    // that chunk's forward rather than ahead of it
    if ((st = chunk_prepare(r, set ^ 1, n0, nrows, &nHl, &nHc, true))) return st;
    cudaError_t e = cudaEventRecord(side->fork, r.s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side->s, side->fork, 0);
    if (e != cudaSuccess) {
      set_error("fork to the side stream", e);
      return FCKL_ERR_CUDA;
    }
    st = grad_from_kept(r, set, r0, rows, side->s, true);
    // the join is recorded and waited for even after a failed launch, so that nothing of
    // this call is left running outside the caller's stream
    e = cudaEventRecord(side->join, side->s);
    if (!st) st = chunk_forward(r, set ^ 1, n0, nrows, nHl, true);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(r.s, side->join, 0);
    if (e != cudaSuccess) {
      set_error("join from the side stream", e);
      return FCKL_ERR_CUDA;
    }
    if (st) return st;
    if ((st = chunk_products(r, set, r0, rows, Hc))) return st;
    r0 = n0;
    rows = nrows;
    Hl = nHl;
    Hc = nHc;
  }
}

int run_loss(Run& r, float* loss) {
  const float* rl = r.rl;
  const int64_t N = r.pl.N;
  cudaStream_t s = r.s;
  return launch(KIND_LOSS_REDUCE, s, "loss_reduce", [&] { loss_reduce_kernel<<<1, 1024, 0, s>>>(rl, N, loss); });
}

int run_setup(Run& r, const void* H, const void* W, int dtype, const int32_t* idx, const float* logp,
              const float* weight, int64_t N, int d, int V, int K, int chunk, void* ws, size_t ws_bytes,
              void* stream) {
  int st = common_checks(H, W, dtype, idx, logp, N, d, V, K, chunk, ws, ws_bytes, &r.pl, &r.di);
  if (st) return st;
  if (!aligned(weight, 4)) return FCKL_ERR_ARG;
  r.s = static_cast<cudaStream_t>(stream);
  r.w = static_cast<uint8_t*>(ws);
  r.status = reinterpret_cast<unsigned*>(r.w + r.pl.off_status);
  r.H = H;
  r.Wraw = W;
  r.Wb = W;
  r.dtype = dtype;
  r.idx = idx;
  r.logp = logp;
  r.weight = weight;
  return FCKL_OK;
}

// ------------------------------------------------------------------ teacher top-K cache builder
constexpr int TOPK_CAND_MAX = 2048;  // candidate slots per position when K <= vocabulary tiles
constexpr size_t TOPK_THR_SMEM = 160 * 1024;  // shared-memory budget of the threshold kernel

struct TopkPlan {
  int chunk, rows_alloc, tiles_v, cmax;
  int thr_rows, thr_stride;  // threshold kernel: positions per block, shared-memory row pitch
  int ldz;  // row pitch (elements) of the kept logits
  size_t off_status, off_pm, off_pl, off_pc, off_lse, off_thr, off_cnt, off_cv, off_cz, off_Ht, off_Wt, total;
  // the chunk's fp32 logits from pass 1, read by the collect step, and per position the list
  // of tiles whose maximum reaches the threshold
  size_t off_Z, off_live, off_live_cnt, total_keep;
  // A second set of what pass 2 and the selection of a chunk use (lse, threshold, counts,
  // candidates, kept logits, live-tile lists), after everything above when there is more than
  // one chunk: with it (total_overlap bytes) chunk c's collect and select run on a second
  // stream beside chunk c+1's pass 1.
  size_t alt_lse, alt_thr, alt_cnt, alt_cv, alt_cz, alt_Z, alt_live, alt_live_cnt, total_overlap;
};

TopkPlan make_topk_plan(int64_t N, int d, int V, int K, int chunk, int dt) {
  TopkPlan p{};
  p.chunk = static_cast<int>(std::min<int64_t>(chunk, N));
  p.rows_alloc = static_cast<int>(rup(p.chunk, 256));
  p.tiles_v = static_cast<int>(cdiv(V, VOCAB_TILE));
  // With fewer vocabulary tiles than K the threshold is -inf and every token is a candidate.
  p.cmax = K > p.tiles_v ? V : std::min(V, TOPK_CAND_MAX);
  p.thr_stride = p.tiles_v | 1;  // odd pitch: the lanes of a warp hit distinct banks
  p.thr_rows = 8;  // 8 positions per block: one per warp in the search, many blocks per chunk
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t r = o;
    o = static_cast<size_t>(rup(static_cast<int64_t>(o + bytes), 1024));
    return r;
  };
  const size_t R = p.rows_alloc;
  p.off_status = take(256);
  p.off_pm = take(static_cast<size_t>(p.tiles_v) * R * 4);
  p.off_pl = take(static_cast<size_t>(p.tiles_v) * R * 4);
  p.off_pc = take(static_cast<size_t>(p.tiles_v) * R * 4);
  p.off_lse = take(R * 4);
  p.off_thr = take(R * 4);
  p.off_cnt = take(R * 4);
  p.off_cv = take(R * p.cmax * 4);
  p.off_cz = take(R * p.cmax * 4);
  p.off_Ht = dt == FCKL_F32 ? take(R * d * 4) : o;
  p.off_Wt = dt == FCKL_F32 ? take(static_cast<size_t>(V) * d * 4) : o;
  p.total = o;
  p.ldz = static_cast<int>(rup(V, 8));
  p.off_Z = take(R * p.ldz * 4);
  p.off_live = take(R * static_cast<size_t>(p.tiles_v) * 4);
  p.off_live_cnt = take(R * 4);
  p.total_keep = o;
  if (N > p.chunk) {
    p.alt_lse = take(R * 4);
    p.alt_thr = take(R * 4);
    p.alt_cnt = take(R * 4);
    p.alt_cv = take(R * p.cmax * 4);
    p.alt_cz = take(R * p.cmax * 4);
    p.alt_Z = take(R * p.ldz * 4);
    p.alt_live = take(R * static_cast<size_t>(p.tiles_v) * 4);
    p.alt_live_cnt = take(R * 4);
  }
  p.total_overlap = o;
  return p;
}

}  // namespace
}  // namespace fckl

using namespace fckl;

extern "C" {

size_t fckl_workspace_bytes(int64_t N, int d, int V, int K, int chunk, int dtype) {
  if (check_shape(N, d, V, K, chunk, dtype) != FCKL_OK) return 0;
  return make_plan(N, d, V, K, chunk, dtype).total;
}

size_t fckl_overlap_workspace_bytes(int64_t N, int d, int V, int K, int chunk, int dtype) {
  if (check_shape(N, d, V, K, chunk, dtype) != FCKL_OK) return 0;
  return make_plan(N, d, V, K, chunk, dtype).total_overlap;
}


int fckl_forward(const void* H, const void* W, int dtype, const int32_t* idx, const float* logp,
                 const float* weight, int64_t N, int d, int V, int K, int chunk, float* loss, float* lse,
                 float* row_loss, void* ws, size_t ws_bytes, void* stream) {
  Run r;
  int st = run_setup(r, H, W, dtype, idx, logp, weight, N, d, V, K, chunk, ws, ws_bytes, stream);
  if (st) return st;
  if (!loss || !lse || !aligned(loss, 4) || !aligned(lse, 4) || !aligned(row_loss, 4)) return FCKL_ERR_ARG;
  r.lse = lse;
  r.rl = row_loss ? row_loss : reinterpret_cast<float*>(r.w + r.pl.off_rowloss);
  if ((st = run_begin(r, false))) return st;
  for (int64_t r0 = 0; r0 < N; r0 += r.pl.chunk) {
    const int rows = static_cast<int>(std::min<int64_t>(r.pl.chunk, N - r0));
    const void *Hl = nullptr, *Hc = nullptr;
    if ((st = chunk_prepare(r, 0, r0, rows, &Hl, &Hc, false))) return st;
    if ((st = chunk_forward(r, 0, r0, rows, Hl))) return st;
  }
  return run_loss(r, loss);
}

int fckl_backward(const void* H, const void* W, int dtype, const int32_t* idx, const float* logp,
                  const float* weight, const float* lse, int64_t N, int d, int V, int K, int chunk,
                  float grad_scale, void* dH, float* dW, void* ws, size_t ws_bytes, void* stream) {
  Run r;
  int st = run_setup(r, H, W, dtype, idx, logp, weight, N, d, V, K, chunk, ws, ws_bytes, stream);
  if (st) return st;
  if (!lse || !dH || !dW || !aligned(lse, 4) || !aligned(dH, 16) || !aligned(dW, 16)) return FCKL_ERR_ARG;
  r.lse = const_cast<float*>(lse);
  r.grad_scale = grad_scale;
  r.dH = dH;
  r.dW = dW;
  if ((st = run_begin(r, true))) return st;
  for (int64_t r0 = 0; r0 < N; r0 += r.pl.chunk) {
    const int rows = static_cast<int>(std::min<int64_t>(r.pl.chunk, N - r0));
    const void *Hl = nullptr, *Hc = nullptr;
    if ((st = chunk_prepare(r, 0, r0, rows, &Hl, &Hc, true))) return st;
    if ((st = chunk_backward(r, 0, r0, rows, Hl, Hc))) return st;
  }
  return FCKL_OK;
}

int fckl_forward_backward(const void* H, const void* W, int dtype, const int32_t* idx, const float* logp,
                          const float* weight, int64_t N, int d, int V, int K, int chunk, float grad_scale,
                          float* loss, float* lse, float* row_loss, void* dH, float* dW, void* ws, size_t ws_bytes,
                          void* stream) {
  Run r;
  int st = run_setup(r, H, W, dtype, idx, logp, weight, N, d, V, K, chunk, ws, ws_bytes, stream);
  if (st) return st;
  if (!loss || !lse || !dH || !dW || !aligned(loss, 4) || !aligned(lse, 4) || !aligned(row_loss, 4) ||
      !aligned(dH, 16) || !aligned(dW, 16))
    return FCKL_ERR_ARG;
  r.lse = lse;
  r.rl = row_loss ? row_loss : reinterpret_cast<float*>(r.w + r.pl.off_rowloss);
  r.grad_scale = grad_scale;
  r.dH = dH;
  r.dW = dW;
  // With the second buffer set in the workspace, G of each chunk overlaps the next forward.
  const bool overlap =
      N > r.pl.chunk && ws_bytes >= r.pl.total_overlap && overlap_pays(r.pl.chunk, d, V, true);
  SideStream* side = nullptr;
  if (overlap) {
    r.pl1 = second_set(r.pl);
    if ((st = side_stream(r.di->id, &side))) return st;
  }
  if ((st = run_begin(r, true))) return st;
  if (overlap) {
    if ((st = run_overlapped(r, side))) return st;
    return run_loss(r, loss);
  }
  for (int64_t r0 = 0; r0 < N; r0 += r.pl.chunk) {
    const int rows = static_cast<int>(std::min<int64_t>(r.pl.chunk, N - r0));
    const void *Hl = nullptr, *Hc = nullptr;
    if ((st = chunk_prepare(r, 0, r0, rows, &Hl, &Hc, true))) return st;
    if ((st = chunk_forward(r, 0, r0, rows, Hl, true))) return st;
    if ((st = chunk_backward(r, 0, r0, rows, Hl, Hc, true))) return st;
  }
  return run_loss(r, loss);
}

int fckl_selftest_wait_timeout(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || !aligned(ws, 256) || ws_bytes < 256) return FCKL_ERR_ARG;
  DevInfo* di = nullptr;
  int st = device_info(&di);
  if (st) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned* status = static_cast<unsigned*>(ws);
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) {
    set_error("cudaMemsetAsync", e);
    return FCKL_ERR_CUDA;
  }
  return launch(KIND_SELFTEST, s, "wait_timeout_selftest",
                [&] { wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(status, 50000000ull); });
}

size_t fckl_topk_workspace_bytes(int64_t N, int d, int V, int K, int chunk, int dtype) {
  if (check_shape(N, d, V, K, chunk, dtype) != FCKL_OK) return 0;
  return make_topk_plan(N, d, V, K, chunk, dtype).total;
}

size_t fckl_topk_kept_logits_workspace_bytes(int64_t N, int d, int V, int K, int chunk, int dtype) {
  if (check_shape(N, d, V, K, chunk, dtype) != FCKL_OK) return 0;
  return make_topk_plan(N, d, V, K, chunk, dtype).total_keep;
}

size_t fckl_topk_overlap_workspace_bytes(int64_t N, int d, int V, int K, int chunk, int dtype) {
  if (check_shape(N, d, V, K, chunk, dtype) != FCKL_OK) return 0;
  return make_topk_plan(N, d, V, K, chunk, dtype).total_overlap;
}

int fckl_teacher_topk(const void* Ht, const void* Wt, int dtype, int64_t N, int d, int V, int K, int chunk,
                      int32_t* idx, float* logp, void* ws, size_t ws_bytes, void* stream) {
  int st = check_shape(N, d, V, K, chunk, dtype);
  if (st) return st;
  if (!Ht || !Wt || !idx || !logp || !ws) return FCKL_ERR_ARG;
  if (!aligned(Ht, 16) || !aligned(Wt, 16) || !aligned(ws, 256) || !aligned(idx, 4) || !aligned(logp, 4))
    return FCKL_ERR_ARG;
  const TopkPlan tp = make_topk_plan(N, d, V, K, chunk, dtype);
  if (static_cast<size_t>(tp.thr_rows) * tp.thr_stride * 4 > TOPK_THR_SMEM) return FCKL_ERR_UNSUPPORTED;
  if (ws_bytes < tp.total) return FCKL_ERR_WORKSPACE;
  const bool keep = ws_bytes >= tp.total_keep;
  DevInfo* di = nullptr;
  if ((st = device_info(&di))) return st;
  {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    static bool thr_attr[64] = {};
    if (!thr_attr[di->id]) {
      cudaError_t e = cudaFuncSetAttribute(topk_threshold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(TOPK_THR_SMEM));
      if (e != cudaSuccess) {
        set_error("cudaFuncSetAttribute(topk_threshold)", e);
        return FCKL_ERR_CUDA;
      }
      thr_attr[di->id] = true;
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  unsigned* status = reinterpret_cast<unsigned*>(w + tp.off_status);
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) {
    set_error("cudaMemsetAsync", e);
    return FCKL_ERR_CUDA;
  }
  // Both passes are logits products: bf16 operands, or tf32-rounded copies of fp32 ones.
  const bool f32 = dtype == FCKL_F32;
  const CUtensorMapDataType mdt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint32_t ke = f32 ? BK / 2 : BK;  // K values per 128-byte stage row
  const size_t esz = f32 ? 4 : 2;
  const void* Wl = Wt;
  if (f32) {
    if ((st = launch_cvt(static_cast<const float*>(Wt), w + tp.off_Wt, nullptr, int64_t(V) * d, di, s))) return st;
    Wl = w + tp.off_Wt;
  }
  CUtensorMap tmW;
  int w3d = 0;
  if (f32) {
    if ((st = make_map(&tmW, Wl, mdt, d, V, uint64_t(d) * esz, ke, VOCAB_TILE / CG))) return st;
  } else if ((st = map_kmajor(&tmW, Wl, d, V, uint64_t(d) * 2, VOCAB_TILE / CG, KPS_LOGITS, &w3d))) {
    return st;
  }
  float* pm = reinterpret_cast<float*>(w + tp.off_pm);
  float* pl = reinterpret_cast<float*>(w + tp.off_pl);
  // Buffers of the chunk's pass 2 and selection, per buffer set (chunk c uses set c % 2 when
  // the workspace holds the second set; then chunk c's collect and select run on the side
  // stream beside chunk c+1's pass 1).
  struct Set {
    float *lse, *thr, *cz, *Z;
    int *cnt, *cv, *live, *live_cnt;
  } sets[2];
  auto set_at = [&](size_t olse, size_t othr, size_t ocnt, size_t ocv, size_t ocz, size_t oZ, size_t olive,
                    size_t olc) {
    return Set{reinterpret_cast<float*>(w + olse), reinterpret_cast<float*>(w + othr),
               reinterpret_cast<float*>(w + ocz),  reinterpret_cast<float*>(w + oZ),
               reinterpret_cast<int*>(w + ocnt),   reinterpret_cast<int*>(w + ocv),
               reinterpret_cast<int*>(w + olive),  reinterpret_cast<int*>(w + olc)};
  };
  sets[0] = set_at(tp.off_lse, tp.off_thr, tp.off_cnt, tp.off_cv, tp.off_cz, tp.off_Z, tp.off_live, tp.off_live_cnt);
  const bool overlap =
      keep && N > tp.chunk && ws_bytes >= tp.total_overlap && overlap_pays(tp.chunk, d, V, false);
  SideStream* side = nullptr;
  if (overlap) {
    sets[1] = set_at(tp.alt_lse, tp.alt_thr, tp.alt_cnt, tp.alt_cv, tp.alt_cz, tp.alt_Z, tp.alt_live,
                     tp.alt_live_cnt);
    if ((st = side_stream(di->id, &side))) return st;
    std::lock_guard<std::mutex> lk(g_setup_mu);
    static bool carve[64] = {};
    if (!carve[di->id]) {
      cudaError_t ce = cudaFuncSetAttribute(topk_collect_kernel<true>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                            cudaSharedmemCarveoutMaxShared);
      if (ce == cudaSuccess)
        ce = cudaFuncSetAttribute(topk_select_kernel<true>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared);
      if (ce != cudaSuccess) {
        set_error("cudaFuncSetAttribute(top-K side kernels)", ce);
        return FCKL_ERR_CUDA;
      }
      carve[di->id] = true;
    }
  }
  const int kbl = static_cast<int>(cdiv(d, ke));
  // One chunk: pass 1 and the threshold on the caller's stream; pass 2 and the selection
  // there too, or on the side stream.
  auto topk_chunk = [&](int64_t r0, const Set& B, SideStream* side, int c) -> int {
    int st = FCKL_OK;
    float* lse = B.lse;
    float* thr = B.thr;
    int* cnt = B.cnt;
    int* cv = B.cv;
    float* cz = B.cz;
    const int rows = static_cast<int>(std::min<int64_t>(tp.chunk, N - r0));
    const void* Hc = static_cast<const uint8_t*>(Ht) + static_cast<size_t>(r0) * d * esz;
    if (f32) {
      if ((st = launch_cvt(static_cast<const float*>(Hc), w + tp.off_Ht, nullptr, int64_t(rows) * d, di, s)))
        return st;
      Hc = w + tp.off_Ht;
    }
    // pass 1: per (row, vocabulary tile) max and sum-exp
    TcParams p;
    memset(&p, 0, sizeof(p));
    if (f32) {
      if ((st = make_map(&p.tmA, Hc, mdt, d, rows, uint64_t(d) * esz, ke, BM))) return st;
    } else if ((st = map_kmajor(&p.tmA, Hc, d, rows, uint64_t(d) * 2, BM, KPS_LOGITS, &p.a_3d))) {
      return st;
    }
    p.tmB = tmW;
    p.b_3d = w3d;
    p.sch = {static_cast<int>(cdiv(rows, TILE_M)), tp.tiles_v, kbl, 1, kbl, 1};
    p.num_units = p.sch.m_blocks * p.sch.n_blocks;
    p.status = status;
    p.rows_valid = rows;
    p.V = V;
    p.K = 0;  // no cached teacher slots to gather
    p.pm = pm;
    p.pl = pl;
    p.pc = reinterpret_cast<float*>(w + tp.off_pc);
    p.ld_part = tp.rows_alloc;
    float* Z = B.Z;
    if (keep) {  // pass 1 also stores the logits for the collect step
      if ((st = make_map(&p.tmC, Z, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, V, rows, uint64_t(tp.ldz) * 4, 32, 32)))
        return st;
      p.c_xlim = V;
      p.c_ylim = rows;
      st = f32 ? launch_tc<VOCAB_TILE, false, false, EPI_FWD_Z, true>(KIND_TOPK_LOGITS_KEEP, di, p, s,
                                                                      "topk_logits_keep")
               : launch_tc<VOCAB_TILE, false, false, EPI_FWD_Z>(KIND_TOPK_LOGITS_KEEP, di, p, s, "topk_logits_keep");
    } else {
      st = f32 ? launch_tc<VOCAB_TILE, false, false, EPI_FWD_STATS, true>(KIND_TOPK_LOGITS, di, p, s,
                                                                          "topk_logits_stats")
               : launch_tc<VOCAB_TILE, false, false, EPI_FWD_STATS>(KIND_TOPK_LOGITS, di, p, s, "topk_logits_stats");
    }
    if (st) return st;
    const int wblocks = static_cast<int>(cdiv(rows, 4));
    const int ld = tp.rows_alloc, tiles = tp.tiles_v;
    const int tR = tp.thr_rows, tstride = tp.thr_stride;
    const int tblocks = static_cast<int>(cdiv(rows, tR));
    const size_t tsmem = static_cast<size_t>(tR) * tstride * 4;
    int* live = keep ? B.live : nullptr;
    int* live_cnt = keep ? B.live_cnt : nullptr;
    if ((st = launch(KIND_TOPK_THRESHOLD, s, "topk_threshold", [&] {
           topk_threshold_kernel<<<tblocks, 256, tsmem, s>>>(pm, pl, ld, tiles, rows, tR, tstride, K, lse, thr,
                                                             cnt, live, live_cnt);
         })))
      return st;
    // pass 2: every logit at or above the threshold becomes a candidate (logits kept from
    // pass 1, or recomputed), then the selection. With a side stream both run there, released
    // together with the next chunk's pass 1 (one block per SM beside its CTAs), and the buffer
    // set's join event is recorded after them.
    const int cmax = tp.cmax;
    cudaStream_t ps = s;
    if (side) {
      cudaError_t e = cudaEventRecord(side->fork, s);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(side->s, side->fork, 0);
      if (e != cudaSuccess) {
        set_error("fork to the side stream", e);
        return FCKL_ERR_CUDA;
      }
      ps = side->s;
    }
    if (keep) {
      const int grid = std::max(1, std::min(rows, di->sms * (side ? 1 : 8)));
      const int64_t ldz = tp.ldz;
      st = launch(side ? KIND_TOPK_COLLECT_KEPT_SIDE : KIND_TOPK_COLLECT_KEPT, ps, "topk_collect_from_logits", [&] {
        if (side)
          topk_collect_kernel<true><<<grid, 256, 0, ps>>>(Z, ldz, rows, V, tiles, thr, live, live_cnt, cnt, cv, cz,
                                                          cmax);
        else
          topk_collect_kernel<false><<<grid, 256, 0, ps>>>(Z, ldz, rows, V, tiles, thr, live, live_cnt, cnt, cv,
                                                           cz, cmax);
      });
    } else {
      p.thr = thr;
      p.cnt = cnt;
      p.cand_v = cv;
      p.cand_z = cz;
      p.cmax = cmax;
      st = f32 ? launch_tc<VOCAB_TILE, false, false, EPI_TOPK_COLLECT, true>(KIND_TOPK_COLLECT, di, p, s,
                                                                             "topk_collect")
               : launch_tc<VOCAB_TILE, false, false, EPI_TOPK_COLLECT>(KIND_TOPK_COLLECT, di, p, s, "topk_collect");
    }
    if (!st) {
      int32_t* io = idx + r0 * K;
      float* lo = logp + r0 * K;
      st = launch(side ? KIND_TOPK_SELECT_SIDE : KIND_TOPK_SELECT, ps, "topk_select", [&] {
        if (side)
          topk_select_kernel<true><<<wblocks, 128, 0, ps>>>(cv, cz, cnt, cmax, rows, K, lse, io, lo, status);
        else
          topk_select_kernel<false><<<wblocks, 128, 0, ps>>>(cv, cz, cnt, cmax, rows, K, lse, io, lo, status);
      });
    }
    if (side) {  // recorded whatever failed: the caller's stream waits for it before returning
      const cudaError_t e = cudaEventRecord(side->join_set[c & 1], side->s);
      if (e != cudaSuccess && !st) {
        set_error("join from the side stream", e);
        st = FCKL_ERR_CUDA;
      }
    }
    return st;
  };
  int c = 0;
  for (int64_t r0 = 0; r0 < N; r0 += tp.chunk, ++c) {
    const Set& B = sets[overlap ? (c & 1) : 0];
    // the side work of chunk c-2 (same buffer set) is done before pass 1 overwrites its logits
    if (overlap && c >= 2 && (st = wait_event(s, side->join_set[c & 1]))) break;
    if ((st = topk_chunk(r0, B, overlap ? side : nullptr, c))) break;
  }
  if (overlap) {  // nothing of this call stays outside the caller's stream order, error or not
    // (an event not recorded by this call is already complete, or orders after earlier work)
    for (cudaEvent_t ev : side->join_set) {
      const int sj = wait_event(s, ev);
      if (!st) st = sj;
    }
  }
  return st;
}

int fckl_check(void* ws, void* stream) {
  if (!ws) return FCKL_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned word = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(unsigned), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    set_error("fckl_check", e);
    return FCKL_ERR_CUDA;
  }
  if (word & ST_TIMEOUT) return FCKL_ERR_TIMEOUT;
  if (word & ST_BAD_INDEX) return FCKL_ERR_INDEX;
  if (word & ST_CAPACITY) return FCKL_ERR_CAPACITY;
  return FCKL_OK;
}

const char* fckl_status_string(int status) {
  switch (status) {
    case FCKL_OK: return "ok";
    case FCKL_ERR_ARG: return "invalid argument (size, null or misaligned pointer)";
    case FCKL_ERR_INDEX: return "teacher id outside [0, V)";
    case FCKL_ERR_CUDA: return "CUDA error (see fckl_last_error)";
    case FCKL_ERR_TIMEOUT: return "a bounded device wait ran out";
    case FCKL_ERR_WORKSPACE: return "workspace smaller than fckl_workspace_bytes()";
    case FCKL_ERR_UNSUPPORTED: return "unsupported shape or device (needs sm_103, d % 8 == 0, K <= min(V, 1024))";
    case FCKL_ERR_CAPACITY: return "a position had more top-K candidates than the candidate buffer holds";
    default: return "unknown status";
  }
}

const char* fckl_last_error(void) { return g_last_error; }

int64_t fckl_launch_count(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  return g_launches;
}

int fckl_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_prof = on != 0;
  return FCKL_OK;
}

int fckl_profile_read(double* ms, int64_t* launches, int n_kinds) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    set_error("cudaDeviceSynchronize", e);
    return FCKL_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  for (const ProfRec& r : g_prof_recs) {
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) == cudaSuccess && r.kind < n_kinds) {
      if (ms) ms[r.kind] += t;
      if (launches) launches[r.kind] += 1;
    }
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  g_prof_recs.clear();
  return FCKL_OK;
}

const char* fckl_kernel_name(int kind) {
  if (kind < 0 || kind >= KIND_COUNT) return nullptr;
  return kKindNames[kind];
}

}  // extern "C"

// ------------------------------------------------------------------ forward with library-owned scratch
// For callers that cannot allocate device memory themselves (see fckl_forward_static in
// include/fckl.h). The scratch is one file-scope device array, reserved on every GPU where
// this library is loaded until the process exits, and shared by every call on that GPU.
static __device__ __align__(256) uint8_t g_fckl_static_scratch[FCKL_STATIC_SCRATCH_BYTES];

namespace fckl {
namespace {

void* g_static_scratch_addr[64] = {};

// Device address of g_fckl_static_scratch in the current context. The host-side name of the
// array is only a stand-in, never a device address, so the address is looked up with the
// device current. Outside stream capture it is looked up again on every call (a table lookup
// in the runtime), so it stays right after a device reset or under another context of the
// same device; while `s` is being captured, the address found by the last uncaptured call on
// this device is used, and a first call on a device made during capture is refused.
int static_scratch_address(int dev, cudaStream_t s, void** out) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const bool capturing = cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone;
  cudaGetLastError();  // a refused query must not surface as the next launch's error
  std::lock_guard<std::mutex> lk(g_mu);
  if (!capturing) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_fckl_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      snprintf(g_last_error, sizeof(g_last_error), "cudaGetSymbolAddress(static scratch): %s",
               cudaGetErrorString(e));
      return FCKL_ERR_CUDA;
    }
    g_static_scratch_addr[dev] = p;
  } else if (!g_static_scratch_addr[dev]) {
    snprintf(g_last_error, sizeof(g_last_error),
             "fckl_forward_static: the first call on a device must come before any stream capture");
    return FCKL_ERR_CUDA;
  }
  *out = g_static_scratch_addr[dev];
  return FCKL_OK;
}

}  // namespace
}  // namespace fckl

extern "C" int fckl_forward_static(const void* H, const void* W, int dtype, const int32_t* idx, const float* logp,
                                   int64_t N, int d, int V, int K, int chunk, float* loss, float* lse,
                                   float* row_loss, uint32_t* status, void* stream) {
  int st = check_shape(N, d, V, K, chunk, dtype);
  if (st) return st;
  if (dtype != FCKL_BF16) {
    set_error_text("fckl_forward_static takes bf16 H and W only");
    return FCKL_ERR_UNSUPPORTED;
  }
  if (!H || !W || !idx || !logp || !loss || !lse || !row_loss || !status) return FCKL_ERR_ARG;
  if (!aligned(H, 16) || !aligned(W, 16) || !aligned(idx, 4) || !aligned(logp, 4) || !aligned(loss, 4) ||
      !aligned(lse, 4) || !aligned(row_loss, 4) || !aligned(status, 4))
    return FCKL_ERR_ARG;

  // Forward-only layout inside the static array: status word, ordered cache slots, S, T and
  // the per-vocabulary-tile statistics of one chunk. The per-position losses go straight
  // to the caller's row_loss, so nothing here grows with N.
  Plan pl = make_plan(N, d, V, K, chunk, dtype);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t r = o;
    o = static_cast<size_t>(rup(static_cast<int64_t>(o + bytes), 1024));
    return r;
  };
  const size_t R = pl.rows_alloc;
  pl.off_status = take(256);
  pl.off_sidx = take(R * K * 4);
  pl.off_sp = take(R * K * 4);
  pl.off_S = take(R * 4);
  pl.off_T = take(R * 4);
  pl.off_pm = take(static_cast<size_t>(pl.tiles_v) * R * 4);
  pl.off_pl = take(static_cast<size_t>(pl.tiles_v) * R * 4);
  pl.off_pc = take(static_cast<size_t>(pl.tiles_v) * R * 4);
  if (o > FCKL_STATIC_SCRATCH_BYTES) {
    std::lock_guard<std::mutex> lk(g_mu);
    snprintf(g_last_error, sizeof(g_last_error),
             "fckl_forward_static: this shape needs %zu bytes of scratch, above the %zu-byte maximum; "
             "use a smaller chunk or fckl_forward with a workspace",
             o, static_cast<size_t>(FCKL_STATIC_SCRATCH_BYTES));
    return FCKL_ERR_WORKSPACE;
  }
  DevInfo* di = nullptr;
  if ((st = device_info(&di))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* base = nullptr;
  if ((st = static_scratch_address(di->id, s, &base))) return st;

  uint8_t* w = static_cast<uint8_t*>(base);
  unsigned* dstatus = reinterpret_cast<unsigned*>(w + pl.off_status);
  // The array keeps whatever the previous call left; only the status word must start at 0
  // (every other region is written before it is read).
  cudaError_t e = cudaMemsetAsync(dstatus, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) {
    set_error("cudaMemsetAsync", e);
    return FCKL_ERR_CUDA;
  }
  CUtensorMap tmW;
  int w3d = 0;
  if ((st = map_kmajor(&tmW, W, d, V, uint64_t(d) * 2, VOCAB_TILE / CG, KPS_LOGITS, &w3d))) return st;
  for (int64_t r0 = 0; r0 < N; r0 += pl.chunk) {
    const int rows = static_cast<int>(std::min<int64_t>(pl.chunk, N - r0));
    if ((st = launch_preprocess(pl, idx + r0 * K, logp + r0 * K, rows, w, dstatus, di, s))) return st;
    const void* Hc = static_cast<const uint8_t*>(H) + static_cast<size_t>(r0) * d * 2;
    TcParams p;
    memset(&p, 0, sizeof(p));
    if ((st = map_kmajor(&p.tmA, Hc, d, rows, uint64_t(d) * 2, BM, KPS_LOGITS, &p.a_3d))) return st;
    p.tmB = tmW;
    p.b_3d = w3d;
    p.sch = {static_cast<int>(cdiv(rows, TILE_M)), pl.tiles_v, static_cast<int>(cdiv(d, BK)), 1,
             static_cast<int>(cdiv(d, BK)), 1};
    p.num_units = p.sch.m_blocks * p.sch.n_blocks;
    p.status = dstatus;
    p.rows_valid = rows;
    p.V = V;
    p.K = K;
    p.sidx = reinterpret_cast<const int*>(w + pl.off_sidx);
    p.sp = reinterpret_cast<const float*>(w + pl.off_sp);
    p.S = reinterpret_cast<const float*>(w + pl.off_S);
    p.pm = reinterpret_cast<float*>(w + pl.off_pm);
    p.pl = reinterpret_cast<float*>(w + pl.off_pl);
    p.pc = reinterpret_cast<float*>(w + pl.off_pc);
    p.ld_part = pl.rows_alloc;
    if ((st = launch_tc<VOCAB_TILE, false, false, EPI_FWD_STATS>(KIND_FWD_LOGITS, di, p, s, "fwd_logits_lse")))
      return st;
    const int cblocks = static_cast<int>(cdiv(rows, 32));
    if ((st = launch(KIND_FWD_COMBINE, s, "fwd_combine", [&] {
           combine_kernel<<<cblocks, 32 * COMBINE_WARPS, 0, s>>>(p.pm, p.pl, p.pc, pl.rows_alloc, pl.tiles_v, rows, p.S,
                                                  reinterpret_cast<const float*>(w + pl.off_T), nullptr,
                                                  lse + r0, row_loss + r0);
         })))
      return st;
  }
  if ((st = launch(KIND_LOSS_REDUCE, s, "loss_reduce",
                   [&] { loss_reduce_kernel<<<1, 1024, 0, s>>>(row_loss, N, loss); })))
    return st;
  e = cudaMemcpyAsync(status, dstatus, sizeof(unsigned), cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) {
    set_error("cudaMemcpyAsync(status)", e);
    return FCKL_ERR_CUDA;
  }
  return FCKL_OK;
}
