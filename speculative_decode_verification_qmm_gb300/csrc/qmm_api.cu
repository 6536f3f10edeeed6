// qmm_api.cu -- the C ABI (include/qmm.h): handles, validation, the launch
// planner, device repack at create time, and the asynchronous verify call.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <unordered_set>

#include "qmm.h"
#include "qmm_kernels.h"

using namespace qmm;

namespace {

constexpr uint64_t HANDLE_MAGIC = 0x514D4D5645524946ull;  // "QMMVERIF"
constexpr uint64_t DEFAULT_WAIT_LIMIT_NS = 2000000000ull;  // 2 s
constexpr size_t GREEDY_STATE_BYTES = MAX_M * sizeof(unsigned long long) + 16;

// Planner constants (they only rank candidate plans; see make_plan()): HBM
// copy bandwidth of the part; tcgen05 kernel: what one CTA with its pipeline
// full sustains and the cluster reduction; mma.sync kernels: one stage's time
// for a CTA alone on its SM and for each of two CTAs sharing one (measured at
// M <= 8), the fixed cost of a call (first bytes, epilogue) and of the split-K
// fix-up by the last split to arrive.
constexpr double PLAN_HBM_BPS = 6.8e12;
constexpr double PLAN_CTA_BPS = 30e9;
constexpr double PLAN_CLUSTER_REDUCE_S = 0.4e-6;
// a CTA alone on its SM streams ~0.67 us per stage over a long range (Q8_0 and
// FP8, 17408 x 5120: 40 stages in 26.7 us), so a grid of one CTA per SM only
// wins when the stages per CTA are few
constexpr double PLAN_STAGE_1_S = 0.65e-6;
constexpr double PLAN_STAGE_2_S = 0.50e-6;
constexpr double PLAN_FIXED_S = 1.5e-6;
constexpr double PLAN_FIXUP_S = 0.8e-6;

struct Plan {
  int n_tiles = 0, S = 1, spc = 1, stage_k = 0, stage_bytes = 0, depth = 0;
  int64_t nst = 0;  // stages per row tile before padding
  bool tc = false;  // tcgen05 kernel and its weight layout
};

}  // namespace

struct qmm_handle {
  uint64_t magic = 0;
  int device = 0;
  int sm_count = 0;
  int fmt = 0;
  uint32_t flags = 0;
  int64_t N = 0, K = 0;
  Plan plan;
  uint8_t* wdev = nullptr;
  size_t wdev_bytes = 0;
  float* f8_scale = nullptr;      // FP8: [n_tiles][S * spc] tile scales
  uint16_t* act_scratch = nullptr;  // f16 paths: [MAX_M][act_ld]
  int64_t act_ld = 0;
  size_t act_bytes = 0;
  float* out_scale = nullptr;  // [MAX_M][S]
  float* ws = nullptr;         // mma.sync kernels, S > 1: split partials
  int* counters = nullptr;     // mma.sync kernels, S > 1: [n_tiles] arrivals
  int* status = nullptr;       // device error word
  // greedy acceptance state: [MAX_M] running maxima, then the finished-tile
  // count (zero between calls)
  unsigned long long* greedy = nullptr;
  uint16_t* stage_act = nullptr;  // host-buffer path: [MAX_M][act_pitch]
  int64_t stage_act_pitch = 0;
  float* stage_out = nullptr;     // [MAX_M][N]
  uint64_t wait_limit_ns = DEFAULT_WAIT_LIMIT_NS;
  int last_cuda_error = 0;
  // qmm_debug_set_trace (builds with QMM_TRACE): the caller's stamp buffer,
  // its slot count and the verify calls made since it was set
  unsigned long long* trace = nullptr;
  int64_t trace_slots = 0;
  int64_t trace_calls = 0;
  // Tensor maps over the activation rows of recent calls, keyed by what they
  // encode (a graph captures the map by value, so an entry can be reused or
  // replaced freely).
  struct MapEntry {
    const void* ptr = nullptr;
    int64_t lda = -1;
    int M = -1, box_r = 0, box_k = 0;
    bool f16 = false;
    CUtensorMap map;
  };
  static constexpr int MAP_CACHE = 8;
  MapEntry maps[MAP_CACHE];
  int map_next = 0;
};

namespace {

std::mutex g_mu;
std::unordered_set<qmm_handle*>& live_handles() {
  static std::unordered_set<qmm_handle*> s;
  return s;
}
std::atomic<int> g_fail_allocs{0};
std::atomic<int> g_last_error{0};

bool is_live(qmm_handle* h) {
  if (!h) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  return live_handles().count(h) != 0 && h->magic == HANDLE_MAGIC;
}

// g_fail_allocs > 0 counts down the allocations until the one that fails.
cudaError_t dev_alloc(void** p, size_t bytes) {
  *p = nullptr;
  int n = g_fail_allocs.load();
  while (n > 0) {
    if (g_fail_allocs.compare_exchange_weak(n, n - 1)) {
      if (n == 1) return cudaErrorMemoryAllocation;
      break;
    }
  }
  if (bytes == 0) bytes = 16;
  return cudaMalloc(p, bytes);
}

int cuda_fail(qmm_handle* h, cudaError_t e) {
  if (h) h->last_cuda_error = (int)e;
  g_last_error.store((int)e);
  return QMM_ERR_CUDA;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

constexpr uint32_t ROTATION_FLAGS = QMM_FLAG_HADAMARD32 | QMM_FLAG_HADAMARD64 | QMM_FLAG_HADAMARD128;

// Rotation block size of a flag set: 0 (none), 32, 64 or 128; -1 for more than one.
int rotation_block(uint32_t flags) {
  switch (flags & ROTATION_FLAGS) {
    case 0: return 0;
    case QMM_FLAG_HADAMARD32: return 32;
    case QMM_FLAG_HADAMARD64: return 64;
    case QMM_FLAG_HADAMARD128: return 128;
    default: return -1;
  }
}

// Choose the K split count S.  With S > 1 every CTA stays resident in one
// wave (two CTAs per SM; tcgen05: as many clusters of S as the device holds at
// once).  tcgen05: score = time to stream the padded bytes at min(HBM
// bandwidth, CTAs x per-CTA rate) plus the cluster reduction.  mma.sync:
// score = max(stream time of the padded bytes, stages per CTA x stage time)
// plus the fixed cost and the fix-up; near-ties go to the plan with more CTAs.
Plan make_plan(int fmt, bool tc, int64_t N, int64_t K, int sm_count, int forced_splits) {
  Plan p;
  p.tc = tc;
  p.stage_k = fmt == 0 ? Q4_STAGE_K : (fmt == 2 ? Q8_STAGE_K : F8_STAGE_K);
  p.stage_bytes = fmt == 0 ? Q4_STAGE_BYTES : (fmt == 2 ? Q8_STAGE_BYTES : F8_STAGE_BYTES);
  p.depth = tc ? tc_pipeline_depth()
               : (fmt == 0 ? q4_pipeline_depth() : (fmt == 2 ? q8_pipeline_depth() : fp8_pipeline_depth()));
  p.n_tiles = (int)ceil_div(N, TILE_N);
  p.nst = ceil_div(K, p.stage_k);
  auto fix = [&](int S) {
    int64_t spc = ceil_div(p.nst, S);
    p.spc = (int)spc;
    p.S = (int)ceil_div(p.nst, spc);
  };
  if (forced_splits > 0) {
    int S = forced_splits < MAX_SPLITS ? forced_splits : MAX_SPLITS;
    fix((int)(S < p.nst ? S : p.nst));
    return p;
  }
  const int64_t max_ctas = 2ll * sm_count;
  double best = 1e30;
  int best_s = 1;
  int64_t best_ctas = 0;
  for (int S = 1; S <= MAX_SPLITS && S <= p.nst; ++S) {
    const int64_t spc = ceil_div(p.nst, S);
    if (ceil_div(p.nst, spc) != S) continue;
    const int64_t ctas = (int64_t)p.n_tiles * S;
    if (S > 1 && ctas > max_ctas) break;
    const double bytes = (double)ctas * spc * p.stage_bytes;
    double t;
    if (tc) {
      if (S > 1) {
        const int clusters = tc_max_active_clusters(S);
        if (clusters > 0 && p.n_tiles > clusters) continue;
      }
      double rate = (double)ctas * PLAN_CTA_BPS;
      if (rate > PLAN_HBM_BPS) rate = PLAN_HBM_BPS;
      t = bytes / rate + (S > 1 ? PLAN_CLUSTER_REDUCE_S : 0.0);
    } else {
      const int64_t waves = ceil_div(ctas, max_ctas);
      const double stage = ctas > sm_count ? PLAN_STAGE_2_S : PLAN_STAGE_1_S;
      const double compute = (double)waves * spc * stage;
      const double stream = bytes / PLAN_HBM_BPS;
      t = (compute > stream ? compute : stream) + PLAN_FIXED_S + (S > 1 ? PLAN_FIXUP_S : 0.0);
    }
    if (t < best * 0.99 || (t <= best * 1.01 && ctas > best_ctas)) {
      if (t < best) best = t;
      best_s = S;
      best_ctas = ctas;
    }
  }
  fix(best_s);
  return p;
}

void free_handle(qmm_handle* h) {
  if (!h) return;
  int old = -1;
  cudaGetDevice(&old);
  if (old != h->device) cudaSetDevice(h->device);
  cudaFree(h->wdev);
  cudaFree(h->f8_scale);
  cudaFree(h->act_scratch);
  cudaFree(h->out_scale);
  cudaFree(h->ws);
  cudaFree(h->counters);
  cudaFree(h->status);
  cudaFree(h->greedy);
  cudaFree(h->stage_act);
  cudaFree(h->stage_out);
  if (old >= 0 && old != h->device) cudaSetDevice(old);
  h->magic = 0;
  delete h;
}

int check_device(int* dev, int* sms) {
  if (cudaGetDevice(dev) != cudaSuccess) return QMM_ERR_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess)
    return QMM_ERR_DEVICE;
  if (major != 10 || minor != 3) return QMM_ERR_DEVICE;
  return QMM_OK;
}

// cuTensorMapEncodeTiled from the driver (looked up once through the runtime).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D view of M activation rows: dim 0 = 8 consecutive 16-bit values, dim 1 =
// rows (stride lda), dim 2 = 8-column groups (stride 16 bytes).  A box of
// 8 x box_r x box_k lands as [group][row][8 values] (the canonical no-swizzle
// K-major layout), with rows >= M and columns >= K read as zeros.
cudaError_t encode_act_map(CUtensorMap* map, const void* base, int64_t lda, int M, int64_t K, bool f16,
                           int box_r, int box_k) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {8, (cuuint64_t)M, (cuuint64_t)((K + 7) / 8)};
  cuuint64_t strides[2] = {(cuuint64_t)lda * 2, 16};
  cuuint32_t box[3] = {8, (cuuint32_t)box_r, (cuuint32_t)box_k};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 2-D view of M activation rows for the mma.sync kernels: dim 0 = K, dim 1 =
// rows (stride lda); boxes of box_k columns x box_r rows land row after row
// with the swizzle as wide as a box row (2 x box_k bytes: 128 or 64).
cudaError_t encode_act_map_2d(CUtensorMap* map, const void* base, int64_t lda, int M, int64_t K,
                              bool f16, int box_r, int box_k) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  cuuint64_t strides[1] = {(cuuint64_t)lda * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_k, (cuuint32_t)box_r};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = box_k * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   sw, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The tensor map over `rows` (M rows of 16-bit values, stride lda) with the
// box the handle's kernel loads: the tcgen05 kernel takes a 3-D view, 16 rows
// x one stage; the mma.sync kernels a 2-D view, R = 8 or 16 rows x one chunk.
cudaError_t act_map_for(qmm_handle* h, const void* rows, int64_t lda, int M, bool f16,
                        const CUtensorMap** out) {
  const int box_r = h->plan.tc ? 16 : (M > 8 ? 16 : 8);
  const int box_k = h->plan.tc ? Q4_STAGE_K / 8 : h->plan.stage_k / STAGE_CHUNKS;
  for (auto& m : h->maps)
    if (m.ptr == rows && m.lda == lda && m.M == M && m.f16 == f16 && m.box_r == box_r &&
        m.box_k == box_k) {
      *out = &m.map;
      return cudaSuccess;
    }
  qmm_handle::MapEntry& m = h->maps[h->map_next];
  h->map_next = (h->map_next + 1) % qmm_handle::MAP_CACHE;
  m.ptr = nullptr;
  cudaError_t e = h->plan.tc ? encode_act_map(&m.map, rows, lda, M, h->K, f16, box_r, box_k)
                             : encode_act_map_2d(&m.map, rows, lda, M, h->K, f16, box_r, box_k);
  if (e != cudaSuccess) return e;
  m.ptr = rows;
  m.lda = lda;
  m.M = M;
  m.f16 = f16;
  m.box_r = box_r;
  m.box_k = box_k;
  *out = &m.map;
  return cudaSuccess;
}

// The tensor map over the prefill pre-pass's f16 rows [M][K]: 2-D, boxes of
// 64 columns x prefill_tile_rows() rows, 128-byte swizzle.
cudaError_t prefill_map_for(qmm_handle* h, const void* rows, int M, const CUtensorMap** out) {
  const int box_r = prefill_tile_rows(), box_k = 64;
  for (auto& m : h->maps)
    if (m.ptr == rows && m.lda == h->K && m.M == M && m.f16 && m.box_r == box_r && m.box_k == box_k) {
      *out = &m.map;
      return cudaSuccess;
    }
  qmm_handle::MapEntry& m = h->maps[h->map_next];
  h->map_next = (h->map_next + 1) % qmm_handle::MAP_CACHE;
  m.ptr = nullptr;
  cudaError_t e = encode_act_map_2d(&m.map, rows, h->K, M, h->K, true, box_r, box_k);
  if (e != cudaSuccess) return e;
  m.ptr = rows;
  m.lda = h->K;
  m.M = M;
  m.f16 = true;
  m.box_r = box_r;
  m.box_k = box_k;
  *out = &m.map;
  return cudaSuccess;
}

// Prefill workspace: f16 rows [M][K], then the rows' multipliers [M] fp32.
int64_t prefill_rows_bytes(const qmm_handle* h, int64_t M) { return (M * h->K * 2 + 255) & ~(int64_t)255; }
int64_t prefill_ws_bytes(const qmm_handle* h, int64_t M) { return prefill_rows_bytes(h, M) + M * 4; }

// The verify kernel of the handle's plan, reading M activation rows of 16-bit
// values at `rows` (the caller's bf16 rows, or the pre-pass's f16 scratch).
cudaError_t launch_verify_kernel(qmm_handle* h, const VerifyParams& vp, const VerifyLaunch& vl,
                                 const void* rows, int64_t lda, int M, bool f16) {
  const CUtensorMap* map = nullptr;
  cudaError_t e = act_map_for(h, rows, lda, M, f16, &map);
  if (e != cudaSuccess) return e;
  if (h->plan.tc) return launch_verify_tc(vp, map, false, vl.ctas, vl.stream);
  if (h->fmt == 0) return launch_verify_q4(vp, vl, map);
  return h->fmt == 2 ? launch_verify_q8(vp, vl, map) : launch_verify_fp8(vp, vl, map);
}

}  // namespace

extern "C" {

const char* qmm_strerror(int code) {
  switch (code) {
    case QMM_OK: return "QMM_OK";
    case QMM_ERR_INVALID_ARG: return "QMM_ERR_INVALID_ARG";
    case QMM_ERR_SHAPE: return "QMM_ERR_SHAPE";
    case QMM_ERR_M_RANGE: return "QMM_ERR_M_RANGE";
    case QMM_ERR_ALIGN: return "QMM_ERR_ALIGN";
    case QMM_ERR_CUDA: return "QMM_ERR_CUDA";
    case QMM_ERR_TIMEOUT: return "QMM_ERR_TIMEOUT";
    case QMM_ERR_STATE: return "QMM_ERR_STATE";
    case QMM_ERR_DEVICE: return "QMM_ERR_DEVICE";
    default: return "QMM_ERR_UNKNOWN";
  }
}

int qmm_debug_fail_allocs(int n) {
  if (n < 0) return QMM_ERR_INVALID_ARG;
  g_fail_allocs.store(n);
  return QMM_OK;
}

int qmm_create(qmm_t* out, const qmm_desc* d, void* stream) {
  if (!out) return QMM_ERR_INVALID_ARG;
  *out = nullptr;
  if (!d || d->struct_size != sizeof(qmm_desc) || !d->weights) return QMM_ERR_INVALID_ARG;
  if (d->format != QMM_FMT_Q4_0 && d->format != QMM_FMT_FP8_E4M3_B128 && d->format != QMM_FMT_Q8_0)
    return QMM_ERR_INVALID_ARG;
  if (d->flags & ~(uint32_t)(ROTATION_FLAGS | QMM_FLAG_SIMT | QMM_FLAG_TCGEN05))
    return QMM_ERR_INVALID_ARG;
  const int rb = rotation_block(d->flags);
  if (rb < 0) return QMM_ERR_INVALID_ARG;
  if (d->k_splits < 0) return QMM_ERR_INVALID_ARG;
  const int fmt = (int)d->format;
  if (fmt == 1 && !d->scales) return QMM_ERR_INVALID_ARG;
  if (fmt != 0 && (d->flags & QMM_FLAG_SIMT)) return QMM_ERR_INVALID_ARG;
  // the tcgen05 kernel serves bf16 Q4_0 only: no rotation, not the CUDA-core baseline
  if ((d->flags & QMM_FLAG_TCGEN05) &&
      (fmt != 0 || (d->flags & (ROTATION_FLAGS | QMM_FLAG_SIMT))))
    return QMM_ERR_INVALID_ARG;
  if (d->N < 1 || d->K < 1) return QMM_ERR_SHAPE;
  if ((fmt == 0 || fmt == 2) && d->K % 32) return QMM_ERR_SHAPE;
  if (fmt == 1 && (d->N % 128 || d->K % 128)) return QMM_ERR_SHAPE;
  if (rb > 0 && d->K % rb) return QMM_ERR_SHAPE;
  if (d->N > (1ll << 31) || d->K > (1ll << 31)) return QMM_ERR_SHAPE;
  int dev = 0, sms = 0;
  int rc = check_device(&dev, &sms);
  if (rc != QMM_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;

  qmm_handle* h = new qmm_handle();
  h->device = dev;
  h->sm_count = sms;
  h->fmt = fmt;
  h->flags = d->flags;
  h->N = d->N;
  h->K = d->K;
  // The mma.sync kernels serve every path; QMM_FLAG_TCGEN05 selects the
  // tcgen05 kernel for bf16 Q4_0 (checked above).
  const bool tc = (d->flags & QMM_FLAG_TCGEN05) != 0;
  cudaError_t e = tc ? prepare_tc_attributes()
                     : (fmt == 0 ? prepare_q4_attributes()
                                 : (fmt == 2 ? prepare_q8_attributes() : prepare_fp8_attributes()));
  if (e == cudaSuccess && fmt == 1) e = prepare_prefill_attributes();
  if (e != cudaSuccess) {
    free_handle(h);
    return cuda_fail(nullptr, e);
  }
  h->plan = make_plan(fmt, tc, d->N, d->K, sms, d->k_splits);
  const Plan& p = h->plan;
  const int64_t stages_total = (int64_t)p.S * p.spc;
  h->wdev_bytes = (size_t)p.n_tiles * stages_total * p.stage_bytes;
  h->act_ld = stages_total * p.stage_k;
  h->act_bytes = (size_t)MAX_M * h->act_ld * sizeof(uint16_t);
  h->stage_act_pitch = ceil_div(d->K, 8) * 8;
  void* tmp_w = nullptr;
  void* tmp_s = nullptr;
#define QMM_ALLOC(ptr, bytes)                                   \
  do {                                                          \
    void* _p = nullptr;                                         \
    cudaError_t _e = dev_alloc(&_p, (bytes));                   \
    if (_e != cudaSuccess) {                                    \
      cudaGetLastError();                                       \
      cudaFree(tmp_w);                                          \
      cudaFree(tmp_s);                                          \
      free_handle(h);                                           \
      return cuda_fail(nullptr, _e);                            \
    }                                                           \
    ptr = reinterpret_cast<decltype(ptr)>(_p);                  \
  } while (0)
  QMM_ALLOC(h->wdev, h->wdev_bytes);
  if (fmt == 1) QMM_ALLOC(h->f8_scale, (size_t)p.n_tiles * stages_total * sizeof(float));
  QMM_ALLOC(h->act_scratch, h->act_bytes);
  QMM_ALLOC(h->out_scale, (size_t)MAX_M * p.S * sizeof(float));
  if (!p.tc && p.S > 1) {
    QMM_ALLOC(h->ws, (size_t)p.n_tiles * p.S * MAX_M * TILE_N * sizeof(float));
    QMM_ALLOC(h->counters, (size_t)p.n_tiles * sizeof(int));
  }
  QMM_ALLOC(h->status, sizeof(int));
  QMM_ALLOC(h->greedy, GREEDY_STATE_BYTES);
  QMM_ALLOC(h->stage_act, (size_t)MAX_M * h->stage_act_pitch * sizeof(uint16_t));
  QMM_ALLOC(h->stage_out, (size_t)MAX_M * d->N * sizeof(float));

  const uint8_t* wsrc = reinterpret_cast<const uint8_t*>(d->weights);
  const float* ssrc = d->scales;
  const size_t wbytes = fmt == 0   ? (size_t)d->N * (d->K / 32) * 18
                        : fmt == 2 ? (size_t)d->N * (d->K / 32) * 34
                                   : (size_t)d->N * d->K;
  const size_t sbytes = fmt == 1 ? (size_t)(d->N / 128) * (d->K / 128) * sizeof(float) : 0;
  if (!d->weights_on_device) {
    QMM_ALLOC(tmp_w, wbytes);
    if ((e = cudaMemcpyAsync(tmp_w, d->weights, wbytes, cudaMemcpyHostToDevice, st)) != cudaSuccess)
      goto fail;
    wsrc = reinterpret_cast<const uint8_t*>(tmp_w);
    if (fmt == 1) {
      QMM_ALLOC(tmp_s, sbytes);
      if ((e = cudaMemcpyAsync(tmp_s, d->scales, sbytes, cudaMemcpyHostToDevice, st)) != cudaSuccess)
        goto fail;
      ssrc = reinterpret_cast<const float*>(tmp_s);
    }
  }
#undef QMM_ALLOC
  e = p.tc ? launch_repack_tc(wsrc, d->N, d->K, p.n_tiles, p.S, p.spc, h->wdev, st)
           : launch_repack(fmt, wsrc, ssrc, d->N, d->K, p.n_tiles, p.S, p.spc, h->wdev, h->f8_scale,
                           st);
  if (e != cudaSuccess) goto fail;
  if ((e = cudaMemsetAsync(h->act_scratch, 0, h->act_bytes, st)) != cudaSuccess) goto fail;
  if ((e = cudaMemsetAsync(h->status, 0, sizeof(int), st)) != cudaSuccess) goto fail;
  if ((e = cudaMemsetAsync(h->greedy, 0, GREEDY_STATE_BYTES, st)) != cudaSuccess) goto fail;
  if (h->counters &&
      (e = cudaMemsetAsync(h->counters, 0, (size_t)p.n_tiles * sizeof(int), st)) != cudaSuccess)
    goto fail;
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) goto fail;
  cudaFree(tmp_w);
  cudaFree(tmp_s);
  h->magic = HANDLE_MAGIC;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    live_handles().insert(h);
  }
  *out = h;
  return QMM_OK;
fail:
  cudaFree(tmp_w);
  cudaFree(tmp_s);
  free_handle(h);
  return cuda_fail(nullptr, e);
}

int qmm_create_rows(qmm_t* out, const qmm_desc* d, int64_t n_begin, int64_t n_end, void* stream) {
  if (!out) return QMM_ERR_INVALID_ARG;
  *out = nullptr;
  if (!d || d->struct_size != sizeof(qmm_desc) || !d->weights) return QMM_ERR_INVALID_ARG;
  if (d->format != QMM_FMT_Q4_0 && d->format != QMM_FMT_FP8_E4M3_B128 && d->format != QMM_FMT_Q8_0)
    return QMM_ERR_INVALID_ARG;
  if (n_begin < 0 || n_end > d->N || n_begin >= n_end) return QMM_ERR_SHAPE;
  const int fmt = (int)d->format;
  if (fmt == QMM_FMT_FP8_E4M3_B128 && ((n_begin % 128) || (n_end % 128))) return QMM_ERR_SHAPE;
  if ((fmt == QMM_FMT_Q4_0 || fmt == QMM_FMT_Q8_0) && d->K % 32) return QMM_ERR_SHAPE;
  if (fmt == QMM_FMT_FP8_E4M3_B128 && (d->K % 128 || d->N % 128)) return QMM_ERR_SHAPE;
  // The rows of every format are stored one after another, so the shard is a
  // sub-range of the caller's buffers (host or device alike).
  qmm_desc sub = *d;
  sub.N = n_end - n_begin;
  const uint8_t* w = reinterpret_cast<const uint8_t*>(d->weights);
  if (fmt == QMM_FMT_Q4_0) {
    sub.weights = w + (size_t)n_begin * (size_t)(d->K / 32) * 18;
  } else if (fmt == QMM_FMT_Q8_0) {
    sub.weights = w + (size_t)n_begin * (size_t)(d->K / 32) * 34;
  } else {
    sub.weights = w + (size_t)n_begin * (size_t)d->K;
    if (d->scales) sub.scales = d->scales + (size_t)(n_begin / 128) * (size_t)(d->K / 128);
  }
  return qmm_create(out, &sub, stream);
}

int qmm_destroy(qmm_t h) {
  if (!h) return QMM_OK;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!live_handles().count(h)) return QMM_ERR_STATE;
    live_handles().erase(h);
  }
  free_handle(h);
  return QMM_OK;
}

}  // extern "C"

namespace {

struct GreedyArgs {
  const int32_t* tokens;
  int32_t* argmax;
  int32_t* accept;
};

// The working memory of one verify call: the pre-pass's f16 rows and their
// per-(row, split) factors (f16 paths only), the split-K partials and the
// per-tile arrival counts (S > 1 only; the counts are zero on entry).
struct VerifyScratch {
  uint16_t* act = nullptr;
  float* out_scale = nullptr;
  float* ws = nullptr;
  int* counters = nullptr;
};

VerifyScratch handle_scratch(const qmm_handle* h) {
  VerifyScratch sc;
  sc.act = h->act_scratch;
  sc.out_scale = h->out_scale;
  sc.ws = h->ws;
  sc.counters = h->counters;
  return sc;
}

// Argument checks shared by every verify entry point.
int check_verify_args(qmm_t h, const uint16_t* act, int64_t lda, const float* out, int64_t ldo,
                      int M) {
  if (!is_live(h)) return QMM_ERR_STATE;
  if (M < 1 || M > MAX_M) return QMM_ERR_M_RANGE;
  if (!act || !out) return QMM_ERR_INVALID_ARG;
  if (((uintptr_t)act & 15) || ((uintptr_t)out & 15) || lda < h->K || (lda & 7) || ldo < h->N)
    return QMM_ERR_ALIGN;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return QMM_ERR_DEVICE;
  return QMM_OK;
}

// qmm_verify, and qmm_verify_greedy when `g` is not NULL, with the working
// memory `sc` (the handle's own, or the fixed array of qmm_verify_noalloc).
int verify_impl(qmm_t h, const uint16_t* act, int64_t lda, float* out, int64_t ldo, int M,
                void* stream, const GreedyArgs* g, const VerifyScratch& sc) {
  cudaStream_t st = (cudaStream_t)stream;
  const Plan& p = h->plan;
  const int hb = rotation_block(h->flags);
  const bool had = hb > 0;
  const bool f16 = had || h->fmt != 0;
  // bf16 operands read the caller's rows directly; the f16 paths (Hadamard
  // rotation, FP8) go through the activation pre-pass and its scratch.
  cudaError_t e = cudaSuccess;
  if (f16) {
    PrepParams pp;
    pp.act = act;
    pp.lda = lda;
    pp.out = sc.act;
    pp.ld_out = h->act_ld;
    pp.out_scale = sc.out_scale;
    pp.K = h->K;
    pp.M = M;
    pp.S = p.S;
    pp.spc = p.spc;
    pp.stage_k = p.stage_k;
    e = launch_act_prep(pp, f16, hb, st);
    if (e != cudaSuccess) return cuda_fail(h, e);
  }

  VerifyParams vp;
  vp.wdev = h->wdev;
  vp.f8_scale = h->f8_scale;
  vp.K = h->K;
  vp.out_scale = f16 ? sc.out_scale : nullptr;
  vp.out = out;
  vp.status = h->status;
  vp.ldo = ldo;
  vp.N = h->N;
  vp.M = M;
  vp.S = p.S;
  vp.spc = p.spc;
  vp.ws = sc.ws;
  vp.counters = sc.counters;
  vp.wait_limit_ns = h->wait_limit_ns;
  vp.best = nullptr;
  vp.tiles_done = nullptr;
  vp.tokens = nullptr;
  vp.argmax_out = nullptr;
  vp.accept_out = nullptr;
  vp.n_tiles = p.n_tiles;
  vp.trace = nullptr;
  if (h->trace) {
    const int64_t slot = (int64_t)p.n_tiles * p.S * QMM_TRACE_FIELDS;
    vp.trace = h->trace + (h->trace_calls++ % h->trace_slots) * slot;
  }
  if (g) {
    vp.best = h->greedy;
    vp.tiles_done = reinterpret_cast<int*>(h->greedy + MAX_M);
    vp.tokens = g->tokens;
    vp.argmax_out = g->argmax;
    vp.accept_out = g->accept;
  }
  VerifyLaunch vl;
  vl.fmt = h->fmt;
  vl.f16_ops = f16;
  vl.simt = (h->flags & QMM_FLAG_SIMT) != 0;
  vl.ctas = p.n_tiles * p.S;
  vl.stream = st;
  e = f16 ? launch_verify_kernel(h, vp, vl, sc.act, h->act_ld, M, true)
          : launch_verify_kernel(h, vp, vl, act, lda, M, false);
  if (e != cudaSuccess) return cuda_fail(h, e);
  return QMM_OK;
}

}  // namespace

extern "C" {

int qmm_verify(qmm_t h, const uint16_t* act, int64_t lda, float* out, int64_t ldo, int M,
               void* stream) {
  const int rc = check_verify_args(h, act, lda, out, ldo, M);
  if (rc != QMM_OK) return rc;
  return verify_impl(h, act, lda, out, ldo, M, stream, nullptr, handle_scratch(h));
}

int qmm_verify_greedy(qmm_t h, const uint16_t* act, int64_t lda, float* out, int64_t ldo, int M,
                      const int32_t* tokens, int32_t* argmax, int32_t* accept, void* stream) {
  if (!is_live(h)) return QMM_ERR_STATE;
  if (M < 1 || M > MAX_M) return QMM_ERR_M_RANGE;
  if (!tokens || !argmax || !accept || h->plan.tc) return QMM_ERR_INVALID_ARG;
  if (((uintptr_t)tokens | (uintptr_t)argmax | (uintptr_t)accept) & 3) return QMM_ERR_ALIGN;
  const int rc = check_verify_args(h, act, lda, out, ldo, M);
  if (rc != QMM_OK) return rc;
  GreedyArgs g{tokens, argmax, accept};
  return verify_impl(h, act, lda, out, ldo, M, stream, &g, handle_scratch(h));
}

int qmm_prefill_workspace(qmm_t h, int64_t M, int64_t* bytes) {
  if (!bytes) return QMM_ERR_INVALID_ARG;
  *bytes = 0;
  if (!is_live(h)) return QMM_ERR_STATE;
  if (h->fmt != QMM_FMT_FP8_E4M3_B128) return QMM_ERR_INVALID_ARG;
  if (M < 1 || M > QMM_PREFILL_MAX_M) return QMM_ERR_M_RANGE;
  *bytes = prefill_ws_bytes(h, M);
  return QMM_OK;
}

int qmm_prefill(qmm_t h, const uint16_t* act, int64_t lda, float* out, int64_t ldo, int64_t M,
                void* workspace, int64_t workspace_bytes, void* stream) {
  if (!is_live(h)) return QMM_ERR_STATE;
  if (h->fmt != QMM_FMT_FP8_E4M3_B128) return QMM_ERR_INVALID_ARG;
  if (M < 1 || M > QMM_PREFILL_MAX_M) return QMM_ERR_M_RANGE;
  if (!act || !out || !workspace) return QMM_ERR_INVALID_ARG;
  if (workspace_bytes < prefill_ws_bytes(h, M)) return QMM_ERR_INVALID_ARG;
  if (((uintptr_t)act & 15) || ((uintptr_t)out & 15) || ((uintptr_t)workspace & 255) || lda < h->K ||
      (lda & 7) || ldo < h->N)
    return QMM_ERR_ALIGN;
  // the kernel counts tiles and 128-column stages in 32-bit integers
  const int64_t pf_tiles = (int64_t)h->plan.n_tiles * ceil_div(M, prefill_tile_rows());
  if (pf_tiles * (h->K / 128) > INT32_MAX) return QMM_ERR_SHAPE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return QMM_ERR_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  uint16_t* rows = static_cast<uint16_t*>(workspace);
  float* row_scale = reinterpret_cast<float*>(static_cast<char*>(workspace) + prefill_rows_bytes(h, M));
  cudaError_t e = launch_prefill_prep(act, lda, rows, row_scale, M, h->K, rotation_block(h->flags), st);
  if (e != cudaSuccess) return cuda_fail(h, e);
  const CUtensorMap* map = nullptr;
  e = prefill_map_for(h, rows, (int)M, &map);
  if (e != cudaSuccess) return cuda_fail(h, e);
  PrefillLaunch pl;
  pl.wdev = h->wdev;
  pl.f8_scale = h->f8_scale;
  pl.row_scale = row_scale;
  pl.out = out;
  pl.status = h->status;
  pl.ldo = ldo;
  pl.M = (int)M;
  pl.n_tiles = h->plan.n_tiles;
  pl.spt = h->plan.S * h->plan.spc;
  pl.kb_count = (int)(h->K / 128);
  pl.sm_count = h->sm_count;
  pl.wait_limit_ns = h->wait_limit_ns;
  e = launch_prefill_fp8(pl, map, st);
  if (e != cudaSuccess) return cuda_fail(h, e);
  return QMM_OK;
}

int qmm_verify_host(qmm_t h, const uint16_t* act_host, int64_t lda, float* out_host, int64_t ldo,
                    int M, void* stream) {
  if (!is_live(h)) return QMM_ERR_STATE;
  if (M < 1 || M > MAX_M) return QMM_ERR_M_RANGE;
  if (!act_host || !out_host) return QMM_ERR_INVALID_ARG;
  if (lda < h->K || ldo < h->N) return QMM_ERR_ALIGN;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return QMM_ERR_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpy2DAsync(h->stage_act, (size_t)h->stage_act_pitch * 2, act_host,
                                    (size_t)lda * 2, (size_t)h->K * 2, (size_t)M,
                                    cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(h, e);
  int rc = qmm_verify(h, h->stage_act, h->stage_act_pitch, h->stage_out, h->N, M, stream);
  if (rc != QMM_OK) return rc;
  e = cudaMemcpy2DAsync(out_host, (size_t)ldo * 4, h->stage_out, (size_t)h->N * 4, (size_t)h->N * 4,
                        (size_t)M, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(h, e);
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(h, e);
  return QMM_OK;
}

int qmm_sync_status(qmm_t h, void* stream) {
  if (!is_live(h)) return QMM_ERR_STATE;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(h, e);
  int word = 0;
  e = cudaMemcpy(&word, h->status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(h, e);
  if (word != 0) {
    // A kernel gave up: clear the word on the handle's stream so the handle
    // can be used again (other streams of the device are not waited for).
    e = cudaMemsetAsync(h->status, 0, sizeof(int), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(h, e);
    return QMM_ERR_TIMEOUT;
  }
  return QMM_OK;
}

int qmm_last_cuda_error(qmm_t h) {
  if (!h) return g_last_error.load();
  if (!is_live(h)) return QMM_ERR_STATE;
  return h->last_cuda_error;
}

int qmm_get_info(qmm_t h, qmm_info* info) {
  if (!is_live(h)) return QMM_ERR_STATE;
  if (!info || info->struct_size != sizeof(qmm_info)) return QMM_ERR_INVALID_ARG;
  const Plan& p = h->plan;
  info->format = (uint32_t)h->fmt;
  info->flags = h->flags;
  info->N = h->N;
  info->K = h->K;
  info->weight_bytes = h->fmt == 0   ? h->N * h->K / 32 * 18
                       : h->fmt == 2 ? h->N * h->K / 32 * 34
                                     : h->N * h->K + 4 * (h->N / 128) * (h->K / 128);
  info->device_weight_bytes = (int64_t)h->wdev_bytes;
  info->scratch_bytes = (int64_t)(h->act_bytes + MAX_M * p.S * sizeof(float) + sizeof(int)) +
                        (h->ws ? (int64_t)p.n_tiles * p.S * MAX_M * TILE_N * 4 + (int64_t)p.n_tiles * 4 : 0);
  info->n_tiles = p.n_tiles;
  info->k_splits = p.S;
  info->ctas = p.n_tiles * p.S;
  info->stages_per_cta = p.spc;
  info->stage_bytes = p.stage_bytes;
  info->pipeline_depth = p.depth;
  info->device = h->device;
  info->sm_count = h->sm_count;
  return QMM_OK;
}

int qmm_dequantize(qmm_t h, float* w_out, void* stream) {
  if (!is_live(h)) return QMM_ERR_STATE;
  if (!w_out) return QMM_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return QMM_ERR_DEVICE;
  const Plan& p = h->plan;
  cudaError_t e = p.tc ? launch_dequant_tc(h->wdev, h->N, h->K, p.n_tiles, p.S, p.spc, w_out,
                                           (cudaStream_t)stream)
                       : launch_dequant(h->fmt, h->wdev, h->f8_scale, h->N, h->K, p.n_tiles, p.S,
                                        p.spc, w_out,
                                        (cudaStream_t)stream);
  return e == cudaSuccess ? QMM_OK : cuda_fail(h, e);
}

int qmm_hadamard(const uint16_t* act, int64_t lda, float* act_out, int M, int64_t K, int block,
                 void* stream) {
  if (!act || !act_out) return QMM_ERR_INVALID_ARG;
  if (block != 32 && block != 64 && block != 128) return QMM_ERR_INVALID_ARG;
  if (M < 1) return QMM_ERR_M_RANGE;
  if (K < block || K % block) return QMM_ERR_SHAPE;
  if (((uintptr_t)act & 15) || ((uintptr_t)act_out & 15) || lda < K || (lda & 7)) return QMM_ERR_ALIGN;
  int dev = 0, sms = 0;
  int rc = check_device(&dev, &sms);
  if (rc != QMM_OK) return rc;
  cudaError_t e = launch_hadamard(act, lda, act_out, M, K, block, sms, (cudaStream_t)stream);
  return e == cudaSuccess ? QMM_OK : cuda_fail(nullptr, e);
}

int qmm_hadamard32(const uint16_t* act, int64_t lda, float* act_out, int M, int64_t K, void* stream) {
  return qmm_hadamard(act, lda, act_out, M, K, 32, stream);
}

}  // extern "C"

namespace {

// The weights w rotated in rb-blocks (64 or 128) and divided by rb, in a
// temporary buffer allocated and freed in stream order; the plain quantizer
// `quant` then reads it.
template <typename F>
cudaError_t quantize_rotated(const float* w, int64_t N, int64_t K, int rb, cudaStream_t st, F quant) {
  void* tmp = nullptr;
  cudaError_t e = cudaMallocAsync(&tmp, (size_t)N * (size_t)K * sizeof(float), st);
  if (e != cudaSuccess) return e;
  e = launch_rotate_weights(w, N, K, rb, reinterpret_cast<float*>(tmp), st);
  if (e == cudaSuccess) e = quant(reinterpret_cast<const float*>(tmp));
  const cudaError_t f = cudaFreeAsync(tmp, st);
  return e != cudaSuccess ? e : f;
}

}  // namespace

extern "C" {

int qmm_quantize_q4_0(const float* w, int64_t N, int64_t K, uint32_t flags, uint8_t* blocks,
                      void* stream) {
  if (!w || !blocks) return QMM_ERR_INVALID_ARG;
  if (flags & ~ROTATION_FLAGS) return QMM_ERR_INVALID_ARG;
  const int rb = rotation_block(flags);
  if (rb < 0) return QMM_ERR_INVALID_ARG;
  if (N < 1 || K < 32 || K % 32 || (rb > 0 && K % rb)) return QMM_ERR_SHAPE;
  if ((uintptr_t)w & 15) return QMM_ERR_ALIGN;
  int dev = 0, sms = 0;
  int rc = check_device(&dev, &sms);
  if (rc != QMM_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e;
  if (rb > 32)
    e = quantize_rotated(w, N, K, rb, st, [&](const float* r) {
      return launch_quantize_q4(r, N, K, 0, blocks, st);
    });
  else
    e = launch_quantize_q4(w, N, K, rb == 32 ? 1 : 0, blocks, st);
  return e == cudaSuccess ? QMM_OK : cuda_fail(nullptr, e);
}

int qmm_quantize_q8_0(const float* w, int64_t N, int64_t K, uint32_t flags, uint8_t* blocks,
                      void* stream) {
  if (!w || !blocks) return QMM_ERR_INVALID_ARG;
  if (flags & ~ROTATION_FLAGS) return QMM_ERR_INVALID_ARG;
  const int rb = rotation_block(flags);
  if (rb < 0) return QMM_ERR_INVALID_ARG;
  if (N < 1 || K < 32 || K % 32 || (rb > 0 && K % rb)) return QMM_ERR_SHAPE;
  if ((uintptr_t)w & 15) return QMM_ERR_ALIGN;
  int dev = 0, sms = 0;
  int rc = check_device(&dev, &sms);
  if (rc != QMM_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e;
  if (rb > 0)
    e = quantize_rotated(w, N, K, rb, st, [&](const float* r) { return launch_quantize_q8(r, N, K, blocks, st); });
  else
    e = launch_quantize_q8(w, N, K, blocks, st);
  return e == cudaSuccess ? QMM_OK : cuda_fail(nullptr, e);
}

int qmm_quantize_fp8(const float* w, int64_t N, int64_t K, uint32_t flags, uint8_t* codes,
                     float* scales, void* stream) {
  if (!w || !codes || !scales) return QMM_ERR_INVALID_ARG;
  if (flags & ~ROTATION_FLAGS) return QMM_ERR_INVALID_ARG;
  const int rb = rotation_block(flags);
  if (rb < 0) return QMM_ERR_INVALID_ARG;
  if (N < 128 || K < 128 || N % 128 || K % 128) return QMM_ERR_SHAPE;
  if (((uintptr_t)w & 15) || ((uintptr_t)codes & 15)) return QMM_ERR_ALIGN;
  int dev = 0, sms = 0;
  int rc = check_device(&dev, &sms);
  if (rc != QMM_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e;
  if (rb > 32)
    e = quantize_rotated(w, N, K, rb, st, [&](const float* r) {
      return launch_quantize_fp8(r, N, K, 0, codes, scales, st);
    });
  else
    e = launch_quantize_fp8(w, N, K, rb == 32 ? 1 : 0, codes, scales, st);
  return e == cudaSuccess ? QMM_OK : cuda_fail(nullptr, e);
}

int qmm_debug_set_wait_limit(qmm_t h, int64_t ns) {
  if (!is_live(h)) return QMM_ERR_STATE;
  if (ns < 0) return QMM_ERR_INVALID_ARG;
  h->wait_limit_ns = (uint64_t)ns;
  return QMM_OK;
}

int qmm_debug_set_trace(qmm_t h, uint64_t* buf, int64_t n_words) {
#ifndef QMM_TRACE
  (void)buf;
  (void)n_words;
  return QMM_ERR_STATE;  // the stamps are compiled out of this build
#else
  if (!is_live(h)) return QMM_ERR_STATE;
  if (h->plan.tc) return QMM_ERR_SHAPE;
  h->trace = nullptr;
  h->trace_slots = 0;
  h->trace_calls = 0;
  if (!buf) return QMM_OK;
  const int64_t slot = (int64_t)h->plan.n_tiles * h->plan.S * QMM_TRACE_FIELDS;
  if (n_words < slot) return QMM_ERR_INVALID_ARG;
  h->trace = reinterpret_cast<unsigned long long*>(buf);
  h->trace_slots = n_words / slot;
  return QMM_OK;
#endif
}

}  // extern "C"

// ---------------------------------------------------------------------------
// qmm_verify_noalloc: the verify product with its working memory taken from a
// fixed array that lives in this library, instead of from the handle.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t STATIC_SCRATCH_BYTES = QMM_NOALLOC_SCRATCH_BYTES;

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[STATIC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_static_mu;
void* g_static_addr[MAX_DEVICES] = {};

// Device address of the array on `dev`, looked up once per device with that
// device current.  Host code must not use the array's name as an address.
cudaError_t static_scratch_addr(int dev, unsigned char** out) {
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_static_addr[dev] = p;
  }
  *out = reinterpret_cast<unsigned char*>(g_static_addr[dev]);
  return cudaSuccess;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

extern "C" int qmm_verify_noalloc(qmm_t h, const uint16_t* act, int64_t lda, float* out,
                                  int64_t ldo, int M, void* stream) {
  const int rc = check_verify_args(h, act, lda, out, ldo, M);
  if (rc != QMM_OK) return rc;
  const Plan& p = h->plan;
  const bool f16 = rotation_block(h->flags) > 0 || h->fmt != 0;
  // Carve the array: [f16 rows | per-(row, split) factors] on the f16 paths,
  // then [split partials | per-tile arrival counts] when the plan splits K.
  // The pre-pass writes the first two in full and the kernel writes every
  // partial before it is read, so only the counts have to start at zero:
  // they are cleared on the stream before the kernel runs.
  size_t off = 0;
  const size_t act_off = off;
  if (f16) off = align256(off + h->act_bytes);
  const size_t scale_off = off;
  if (f16) off = align256(off + (size_t)MAX_M * p.S * sizeof(float));
  const bool split = !p.tc && p.S > 1;
  const size_t ws_off = off;
  if (split) off = align256(off + (size_t)p.n_tiles * p.S * MAX_M * TILE_N * sizeof(float));
  const size_t cnt_off = off;
  if (split) off = align256(off + (size_t)p.n_tiles * sizeof(int));
  if (off > STATIC_SCRATCH_BYTES) return QMM_ERR_SHAPE;
  int dev = -1;
  cudaGetDevice(&dev);
  unsigned char* base = nullptr;
  cudaError_t e = static_scratch_addr(dev, &base);
  if (e != cudaSuccess) return cuda_fail(h, e);
  VerifyScratch sc;
  if (f16) {
    sc.act = reinterpret_cast<uint16_t*>(base + act_off);
    sc.out_scale = reinterpret_cast<float*>(base + scale_off);
  }
  if (split) {
    sc.ws = reinterpret_cast<float*>(base + ws_off);
    sc.counters = reinterpret_cast<int*>(base + cnt_off);
    e = cudaMemsetAsync(sc.counters, 0, (size_t)p.n_tiles * sizeof(int), (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(h, e);
  }
  // (the tcgen05 kernel serves the bf16 path and reduces its splits inside a
  // thread-block cluster: it needs none of the array)
  return verify_impl(h, act, lda, out, ldo, M, stream, nullptr, sc);
}
