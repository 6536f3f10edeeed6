// qmm_prefill.cu -- the prefill-shaped block-scaled FP8 GEMM: out[M][N] =
// act[M][K] * W[N][K]^T for any number of activation rows M, on the
// 5th-generation tensor cores, with W the FP8 E4M3 codes of a verify handle
// and one fp32 scale per 128 x 128 tile ["r9k: a from-scratch inference
// engine for Qwen3.8-27B on two Radeon AI PRO R9700", opening section: the
// prompt is processed by a block-scaled FP8 GEMM over weights in 128 x 128
// scale blocks; its list of planned work names block-scaled FP8 GEMMs for
// prefill again, and its correctness notes a BF16-activation prefill].
//
// Pre-pass (prefill_prep_kernel).  One warp per activation row: the row
// (rotated in B-blocks for the Hadamard variants) is multiplied by 2^e, with e
// chosen so that its largest magnitude lands in [2^14, 2^15), rounded to f16
// and written to the workspace; 2^-e is the row's output multiplier.
//
// GEMM (prefill_fp8_kernel), persistent, one CTA per SM.  A tile is 128
// weight rows (one scale row) x 192 activation rows; tiles are visited in
// groups of weight tiles, weight tiles fastest within a group, so that the
// CTAs in flight share each activation tile and the group's codes stay in L2
// while the activation tiles stream past (the group size is chosen by the
// host, see launch_prefill_fp8).  Per 128-column stage (one scale column):
//   warp 0      producer: one bulk copy of the stage's 16 KB of codes (the
//               verify layout: units of 16 rows x 32 columns in mma.sync
//               fragment order) and two 2-D tensor copies of the activation
//               tile, 192 rows x 64 columns each, 128-byte swizzled;
//   warp 1      allocates tensor memory; one thread issues eight
//               tcgen05.mma (M = 128 weight rows, N = 192 activation rows,
//               K = 16; A = f16 weights in tensor memory, B = f16 activations
//               in shared memory) into a fresh fp32 accumulator;
//   warps 2-5   convert: warp q reads the units of rows 32q .. 32q + 31,
//               converts E4M3 to f16 exactly (one cvt per pair) and stores
//               them with tcgen05.st.16x128b, whose lane pattern is the
//               fragment order of the units;
//   warps 6-17  promote: warp (q, h) reads its 32 weight rows x 64 activation
//               columns of the stage's accumulator (tcgen05.ld, 16 columns at
//               a time) and adds scale * partial into fp32 registers (packed
//               FMAs); after the last stage of a tile it writes
//               out[m][n] = sum * 2^-e(m), 32 consecutive n per store.
// Tensor memory (512 columns) holds two 192-column accumulators (columns
// 0-383) and two A operands (384-511), so the MMAs of one stage overlap the
// conversion of the next and the promotion of the last.  The ring's three
// 64 KB stages are each held until their MMAs complete and a stage lands
// ~2 us after it is requested, so the rate is set by the work per stage: the
// widest activation tile the accumulators and the promotion registers allow.
// Every wait is bounded; on a timeout the CTA records it in the status word,
// stops, drains its own copies and MMAs in flight and frees tensor memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include "qmm_common.cuh"
#include "qmm_kernels.h"
#include "qmm_tc.cuh"

namespace qmm {

constexpr int PF_BM = 192;  // activation rows per tile (the MMA's N)
constexpr int PF_BK = 128;  // columns per stage: one scale column
constexpr int PF_NS = 3;    // stages in the shared-memory ring
constexpr int PF_NA = 2;    // f16 weight (A operand) buffers in tensor memory
constexpr int PF_ND = 2;    // fp32 accumulators in tensor memory
constexpr int PF_WARPS = 18;
constexpr int PF_THREADS = PF_WARPS * 32;
constexpr int PF_CV_WARP0 = 2, PF_CV_WARPS = 4;
constexpr int PF_EP_WARP0 = 6, PF_EP_WARPS = 12;  // 4 lane quarters x 3 column blocks
static_assert(PF_CV_WARP0 + PF_CV_WARPS == PF_EP_WARP0 && PF_EP_WARP0 + PF_EP_WARPS == PF_WARPS, "warp roles");
constexpr int PF_ACT_BYTES = PF_BM * PF_BK * 2;  // 48 KB: two 64-column swizzled halves
constexpr int PF_TMEM_COLS = 512;
constexpr int PF_D_COL = 0;    // accumulator b: columns b * PF_BM + [0, PF_BM)
constexpr int PF_A_COL = PF_ND * PF_BM;  // A operand a: columns PF_A_COL + a * 64 + [0, 64)
static_assert(PF_A_COL + PF_NA * (PF_BK / 2) <= PF_TMEM_COLS, "tensor memory budget");
// Raster groups (weight tiles visited together; see launch_prefill_fp8): the
// size for activation rows that stay in L2 beside a group, and the L2 budget
// of a group's codes when they do not.
constexpr int PF_GROUP_MIN = 16;
constexpr int64_t PF_ACT_L2_BYTES = 32ll << 20;
constexpr int64_t PF_GROUP_L2_BYTES = 30ll << 20;

struct PfSmem {
  static constexpr int ACT_OFF = 0;
  static constexpr int W_OFF = ACT_OFF + PF_NS * PF_ACT_BYTES;
  static constexpr int BAR_OFF = W_OFF + PF_NS * F8_STAGE_BYTES;
  // full[NS], empty[NS], afull[NA], aempty[NA], dfull[ND], dempty[ND]
  static constexpr int SLOT_OFF = BAR_OFF + (2 * PF_NS + 2 * PF_NA + 2 * PF_ND) * 8;
  static constexpr int FLAG_OFF = SLOT_OFF + 16;
  static constexpr int BYTES = FLAG_OFF + 16;
  static_assert(PF_ACT_BYTES % 1024 == 0 && W_OFF % 1024 == 0, "swizzled tiles need 1024-byte alignment");
};

struct PrefillParams {
  const uint8_t* wdev;     // FP8 stage stream: weight tile t's stage kb at (t * spt + kb) * 16 KB
  const float* f8_scale;   // [n_tiles][spt]
  const float* row_scale;  // [M] output multiplier of each activation row
  float* out;
  int* status;
  int64_t ldo;
  int M;
  int n_tiles;
  int m_tiles;
  int spt;       // stages per weight tile in the stream
  int kb_count;  // stages that hold columns < K (K / 128)
  int group;     // weight tiles per raster group
  uint64_t wait_limit_ns;
};

// Tile t -> (weight tile nt, activation tile mt): groups of `group` weight
// tiles (the last one shorter), weight tiles fastest within a group.
__device__ __forceinline__ void pf_tile(int t, int n_tiles, int m_tiles, int group, int& nt,
                                        int& mt) {
  const int per_group = group * m_tiles;
  const int g = t / per_group, r = t - g * per_group;
  const int left = n_tiles - g * group;
  const int gn = left < group ? left : group;
  nt = g * group + r % gn;
  mt = r / gn;
}

// Every lane waits; the warp continues only if all of them saw the phase.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t lim) {
  const bool ok = mbar_wait_bounded(bar, parity, lim);
  return __all_sync(0xFFFFFFFFu, ok);
}

__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_fp8_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap amap) {
  using L = PfSmem;
  constexpr int NS = PF_NS;
  constexpr uint32_t IDESC = tc_idesc_n(0u, PF_BM);  // f16 x f16 -> fp32, M = 128, N = 192
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  const uint32_t s_base = smem_u32(smem);
  const uint32_t s_act = s_base + L::ACT_OFF;
  const uint32_t s_w = s_base + L::W_OFF;
  const uint32_t s_full = s_base + L::BAR_OFF;
  const uint32_t s_empty = s_full + NS * 8;
  const uint32_t s_afull = s_empty + NS * 8;
  const uint32_t s_aempty = s_afull + PF_NA * 8;
  const uint32_t s_dfull = s_aempty + PF_NA * 8;
  const uint32_t s_dempty = s_dfull + PF_ND * 8;
  // [0] abort, [1] stages committed by the MMA thread, [2] stages issued by the producer
  volatile int* s_flag = reinterpret_cast<volatile int*>(smem + L::FLAG_OFF);

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(s_full + 8 * i, 1);
      mbar_init(s_empty + 8 * i, PF_CV_WARPS + 1);  // the converters and the MMA commit
    }
    for (int a = 0; a < PF_NA; ++a) {
      mbar_init(s_afull + 8 * a, PF_CV_WARPS);
      mbar_init(s_aempty + 8 * a, 1);
    }
    for (int b = 0; b < PF_ND; ++b) {
      mbar_init(s_dfull + 8 * b, 1);
      mbar_init(s_dempty + 8 * b, PF_EP_WARPS);
    }
    s_flag[0] = 0;
    s_flag[1] = 0;
    s_flag[2] = 0;
    if (s_base & 1023u) {
      atomicOr(p.status, DEV_ERR_SMEM_ALIGN);
      s_flag[0] = 1;
    }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(s_base + L::SLOT_OFF, PF_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::SLOT_OFF);

  const uint64_t lim = p.wait_limit_ns;
  const int tiles = p.n_tiles * p.m_tiles;
  const int kbs = p.kb_count;
  auto fail = [&](int code) {
    atomicOr(p.status, code);
    s_flag[0] = 1;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int u = 0;
      bool ok = s_flag[0] == 0;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        int nt, mt;
        pf_tile(t, p.n_tiles, p.m_tiles, p.group, nt, mt);
        const uint8_t* wt = p.wdev + (size_t)nt * p.spt * F8_STAGE_BYTES;
        for (int kb = 0; kb < kbs; ++kb) {
          const int slot = u % NS;
          if (u >= NS && !mbar_wait_bounded(s_empty + 8 * slot, ((u / NS) - 1) & 1, lim)) {
            fail(DEV_ERR_TIMEOUT_EMPTY);
            ok = false;
            break;
          }
          if (s_flag[0]) {
            ok = false;
            break;
          }
          const uint32_t bar = s_full + 8 * slot;
          const uint32_t a_dst = s_act + slot * PF_ACT_BYTES;
          mbar_arrive_expect_tx(bar, F8_STAGE_BYTES + PF_ACT_BYTES);
          bulk_g2s(s_w + slot * F8_STAGE_BYTES, wt + (size_t)kb * F8_STAGE_BYTES, F8_STAGE_BYTES, bar);
          tma_load_2d(a_dst, &amap, kb * PF_BK, mt * PF_BM, bar);
          tma_load_2d(a_dst + PF_ACT_BYTES / 2, &amap, kb * PF_BK + 64, mt * PF_BM, bar);
          ++u;
          s_flag[2] = u;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      int u = 0;
      bool ok = s_flag[0] == 0;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        for (int kb = 0; kb < kbs; ++kb) {
          const int slot = u % NS, b = u % PF_ND, a = u % PF_NA;
          if (!mbar_wait_bounded(s_full + 8 * slot, (u / NS) & 1, lim) ||
              !mbar_wait_bounded(s_afull + 8 * a, (u / PF_NA) & 1, lim) ||
              (u >= PF_ND && !mbar_wait_bounded(s_dempty + 8 * b, ((u / PF_ND) - 1) & 1, lim))) {
            fail(DEV_ERR_TIMEOUT_FULL);
            ok = false;
            break;
          }
          if (s_flag[0]) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t act = s_act + slot * PF_ACT_BYTES;
          const uint32_t d_t = tmem + PF_D_COL + b * PF_BM;
          const uint32_t a_t = tmem + PF_A_COL + a * (PF_BK / 2);
#pragma unroll
          for (int kk = 0; kk < PF_BK / 16; ++kk) {
            const uint64_t bdesc =
                smem_desc_sw128(act + (uint32_t)(kk >> 2) * (PF_ACT_BYTES / 2) + (uint32_t)(kk & 3) * 32u);
            tc_mma(d_t, a_t + kk * 8, bdesc, IDESC, kk > 0 ? 1u : 0u);
          }
          tc_commit(s_empty + 8 * slot);
          tc_commit(s_aempty + 8 * a);
          tc_commit(s_dfull + 8 * b);
          ++u;
          s_flag[1] = u;
        }
      }
    }
  } else if (warp < PF_EP_WARP0) {
    // ------------------------------------------------------------ convert
    const int q = warp & 3;
    int u = 0;
    bool ok = __all_sync(0xFFFFFFFFu, s_flag[0] == 0);
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
      for (int kb = 0; kb < kbs; ++kb) {
        const int slot = u % NS, a = u % PF_NA;
        if (!warp_wait(s_full + 8 * slot, (u / NS) & 1, lim) ||
            (u >= PF_NA && !warp_wait(s_aempty + 8 * a, ((u / PF_NA) - 1) & 1, lim))) {
          if (lane == 0) fail(DEV_ERR_TIMEOUT_FULL);
          ok = false;
          break;
        }
        if (__any_sync(0xFFFFFFFFu, s_flag[0] != 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t wst = s_w + slot * F8_STAGE_BYTES;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // units (c, r = 2q + h), c = 0..3: rows 32q + 16h + [0, 16), columns 32c + [0, 32)
          uint4 c4[4];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            c4[c] = lds128(wst + (uint32_t)((c * 8 + 2 * q + h) * F8_UNIT_BYTES + 16 * lane));
          uint32_t r[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t w4[4] = {c4[c].x, c4[c].y, c4[c].z, c4[c].w};
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              // word v: bytes 0-1 row g, bytes 2-3 row g + 8, column pair 16c + 4v + t
              r[2 * (4 * c + v)] = e4m3x2_to_f16x2(w4[v] & 0xFFFFu);
              r[2 * (4 * c + v) + 1] = e4m3x2_to_f16x2(w4[v] >> 16);
            }
          }
          tmem_st_16x128b_x16(tmem + ((uint32_t)(32 * q + 16 * h) << 16) + PF_A_COL + a * (PF_BK / 2), r);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(s_afull + 8 * a);
          mbar_arrive(s_empty + 8 * slot);
        }
        ++u;
      }
    }
  } else {
    // ------------------------------------------------------------ promote and store
    const int q = warp & 3, h = (warp - PF_EP_WARP0) >> 2;
    const uint32_t tl = (uint32_t)(32 * q) << 16;
    int u = 0;
    bool ok = __all_sync(0xFFFFFFFFu, s_flag[0] == 0);
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
      int nt, mt;
      pf_tile(t, p.n_tiles, p.m_tiles, p.group, nt, mt);
      float acc[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0.f;
      const float* wsc = p.f8_scale + (size_t)nt * p.spt;
      for (int kb = 0; kb < kbs; ++kb) {
        const int b = u % PF_ND;
        const float s = __ldg(wsc + kb);
        if (!warp_wait(s_dfull + 8 * b, (u / PF_ND) & 1, lim)) {
          if (lane == 0) fail(DEV_ERR_TIMEOUT_FULL);
          ok = false;
          break;
        }
        tc_fence_after();
        // 16 columns per load: 32 at a time spills the running sums at 18 warps
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          uint32_t v[16];
          tmem_ld16(tmem + tl + PF_D_COL + b * PF_BM + h * 64 + qq * 16, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; j += 2)
            ffma2(acc[qq * 16 + j], acc[qq * 16 + j + 1], s, __uint_as_float(v[j]),
                  __uint_as_float(v[j + 1]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_dempty + 8 * b);
        ++u;
      }
      if (!ok) break;
      // out[m][n]: lane = weight row n, register j = activation row m
      const int64_t n = (int64_t)nt * TILE_N + 32 * q + lane;
      const int m0 = mt * PF_BM + h * 64;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const int m = m0 + j;
        if (m < p.M) p.out[(int64_t)m * p.ldo + n] = acc[j] * __ldg(p.row_scale + m);
      }
    }
  }

  __syncthreads();
  if (s_flag[0]) {
    // Nothing may still land in shared or tensor memory once the CTA exits:
    // wait for the copies and the MMAs this CTA issued.
    if (warp == 0 && lane == 0) {
      const int issued = s_flag[2];
      for (int i = issued - NS < 0 ? 0 : issued - NS; i < issued; ++i)
        if (!mbar_wait_bounded(s_full + 8 * (i % NS), (i / NS) & 1, 1000000000ull))
          atomicOr(p.status, DEV_ERR_TIMEOUT_DRAIN);
    }
    if (warp == 1 && lane == 0) {
      const int c = s_flag[1];
      if (c > 0 &&
          !mbar_wait_bounded(s_dfull + 8 * ((c - 1) % PF_ND), ((c - 1) / PF_ND) & 1, 1000000000ull))
        atomicOr(p.status, DEV_ERR_TIMEOUT_DRAIN);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, PF_TMEM_COLS);
  }
}

// ---------------------------------------------------------------- pre-pass
// One warp per activation row (K % 128 == 0, so every lane runs the same
// number of 128-column steps and the rotation's shuffles stay converged).
template <int HB>
__global__ void __launch_bounds__(256)
    prefill_prep_kernel(const uint16_t* __restrict__ act, int64_t lda, uint16_t* __restrict__ out,
                        float* __restrict__ row_scale, int64_t M, int64_t K) {
  const int lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (m >= M) return;
  const uint16_t* src = act + m * lda;
  float amax = 0.f;
  for (int64_t k = lane * 4; k < K; k += 128) {
    float v[4];
    load4_bf16(src + k, v);
    if constexpr (HB != 0) fwht_lanes<HB>(v, lane);
#pragma unroll
    for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(v[e]));
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, d));
  int sh = 0;
  if (amax > 0.f && isfinite(amax)) {
    int E;
    frexpf(amax, &E);  // amax = f * 2^E, f in [0.5, 1)
    sh = 15 - E;       // amax * 2^sh in [2^14, 2^15)
    sh = sh > 100 ? 100 : (sh < -100 ? -100 : sh);
  }
  const float mul = ldexpf(1.0f, sh);
  if (lane == 0) row_scale[m] = ldexpf(1.0f, -sh);
  uint16_t* dst = out + m * K;
  for (int64_t k = lane * 4; k < K; k += 128) {
    float v[4];
    load4_bf16(src + k, v);
    if constexpr (HB != 0) fwht_lanes<HB>(v, lane);
    const __half2 h01 = __floats2half2_rn(v[0] * mul, v[1] * mul);
    const __half2 h23 = __floats2half2_rn(v[2] * mul, v[3] * mul);
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t*>(&h01);
    o.y = *reinterpret_cast<const uint32_t*>(&h23);
    *reinterpret_cast<uint2*>(dst + k) = o;
  }
}

// ---------------------------------------------------------------- host side
cudaError_t prepare_prefill_attributes() {
  return cudaFuncSetAttribute(prefill_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PfSmem::BYTES);
}

cudaError_t launch_prefill_prep(const uint16_t* act, int64_t lda, uint16_t* out, float* row_scale, int64_t M,
                                int64_t K, int hb, cudaStream_t st) {
  const unsigned blocks = (unsigned)((M + 7) / 8);
  switch (hb) {
    case 32: prefill_prep_kernel<32><<<blocks, 256, 0, st>>>(act, lda, out, row_scale, M, K); break;
    case 64: prefill_prep_kernel<64><<<blocks, 256, 0, st>>>(act, lda, out, row_scale, M, K); break;
    case 128: prefill_prep_kernel<128><<<blocks, 256, 0, st>>>(act, lda, out, row_scale, M, K); break;
    default: prefill_prep_kernel<0><<<blocks, 256, 0, st>>>(act, lda, out, row_scale, M, K); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_prefill_fp8(const PrefillLaunch& pl, const void* act_map, cudaStream_t st) {
  PrefillParams p;
  p.wdev = pl.wdev;
  p.f8_scale = pl.f8_scale;
  p.row_scale = pl.row_scale;
  p.out = pl.out;
  p.status = pl.status;
  p.ldo = pl.ldo;
  p.M = pl.M;
  p.n_tiles = pl.n_tiles;
  p.m_tiles = (int)((pl.M + PF_BM - 1) / PF_BM);
  p.spt = pl.spt;
  p.kb_count = pl.kb_count;
  p.wait_limit_ns = pl.wait_limit_ns;
  // Raster groups.  The activation rows are read once per group: from L2
  // when they fit there beside the group (then the least L2-hungry group
  // size is kept), from HBM otherwise, and then the fewest groups whose
  // codes fit the L2 budget cut those re-reads (measured on 17408 x 5120 at
  // M = 8192: 3 groups move 886 MB, 16-tile groups 1381 MB, and the call is
  // 3 % shorter; at M = 2048, whose 21 MB of rows stay in L2, 16-tile groups
  // are 2 % faster).
  p.group = PF_GROUP_MIN;
  const int64_t act_bytes = (int64_t)pl.M * p.kb_count * F8_STAGE_K * 2;
  if (act_bytes > PF_ACT_L2_BYTES) {
    const int64_t tile_bytes = (int64_t)TILE_N * p.kb_count * F8_STAGE_K;
    const int64_t groups = ((int64_t)p.n_tiles * tile_bytes + PF_GROUP_L2_BYTES - 1) / PF_GROUP_L2_BYTES;
    const int64_t g = (p.n_tiles + groups - 1) / groups;
    if (g > p.group) p.group = (int)g;
  }
  const int tiles = p.n_tiles * p.m_tiles;
  const int ctas = tiles < pl.sm_count ? tiles : pl.sm_count;
  const CUtensorMap& map = *reinterpret_cast<const CUtensorMap*>(act_map);
  prefill_fp8_kernel<<<(unsigned)ctas, PF_THREADS, PfSmem::BYTES, st>>>(p, map);
  return cudaGetLastError();
}

int prefill_tile_rows() { return PF_BM; }

}  // namespace qmm
