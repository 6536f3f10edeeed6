// qmm_verify_tc.cu -- the tcgen05 verify kernel for Q4_0 (5th-generation tensor
// cores, accumulators in tensor memory), its weight layout, repack and exact
// dequantization.
//
// Weight layout ("tc" layout).  Same stage grid as the mma.sync layout (row
// tiles of 128 rows, stages of 256 columns, CTA (tile, split) streams stages
// [split*spc, (split+1)*spc) as contiguous 18,432-byte ranges), but inside a
// stage:
//   codes  [block b = 0..7][row 0..127][16 bytes]  (16,384 B)
//   scales [row 0..127][block 0..7] fp16           ( 2,048 B)
// The 16 code bytes of (row, block) are four 32-bit words; word w holds the
// 8 columns 32 b + 8 w .. + 7, element 2p in nibble p and element 2p + 1 in
// nibble p + 4 (p = 0..3), so that one magic-number step per nibble pair gives
// the (low, high) 16-bit pair of one tensor-memory column.
//
// CTA roles (14 warps):
//   warp 0      producer: per stage one bulk copy of the weights and one 3-D
//               tensor copy of the 16 activation rows, landing in the UMMA
//               canonical K-major layout ([8-column group][16 rows][8 values]),
//               rows >= M and columns >= K zero-filled by the copy engine;
//   warp 1      allocates tensor memory and issues the MMAs (one thread);
//   warps 2-9   dequantize: thread = weight row = tensor-memory lane; they
//               write (q - 8) as bf16/f16 pairs into a two-buffer A ring in
//               tensor memory (tcgen05.st);
//   warps 10-13 scale: read each 32-block's 128 x 16 fp32 accumulator from
//               tensor memory (tcgen05.ld) and add d[row][block] * partial into
//               registers with packed fp32 FMAs.
// Per 32-block the MMA thread issues two tcgen05.mma (M = 128, N = 16, K = 16,
// A from tensor memory, B from shared memory) into a fresh accumulator, four
// blocks per commit.  The epilogue is the mma.sync kernel's: one split writes
// `out`; K splits form a cluster and add their partials over DSMEM in order.
#include <cuda.h>
#include <cuda_runtime.h>

#include "qmm_kernels.h"
#include "qmm_tc.cuh"
#include "qmm_verify.cuh"

namespace qmm {

constexpr int TC_WARPS = 14;
constexpr int TC_THREADS = TC_WARPS * 32;
constexpr int TC_DQ_WARP0 = 2, TC_DQ_WARPS = 8;
constexpr int TC_EP_WARP0 = 10, TC_EP_WARPS = 4;
constexpr int TC_ACT_STAGE_BYTES = MAX_M * Q4_STAGE_K * 2;  // 8 KB
constexpr int TC_TMEM_COLS = 256;  // buffer u: A columns u*128 + [0, 64), D columns u*128 + [64, 128)
constexpr int TC_NS = 4;

template <int NS>
struct TcSmem {
  static constexpr int W_OFF = 0;
  static constexpr int A_OFF = NS * Q4_STAGE_BYTES;
  static constexpr int BAR_OFF = A_OFF + NS * TC_ACT_STAGE_BYTES;
  // full[NS], empty[NS], afull[2], mmadone[2], dfree[2]
  static constexpr int SLOT_OFF = BAR_OFF + (2 * NS + 6) * 8;
  static constexpr int FLAG_OFF = SLOT_OFF + 16;
  static constexpr int BYTES = FLAG_OFF + 16;
  static constexpr int CP_PITCH = MAX_M + 1;
  static_assert(A_OFF % 1024 == 0, "activation ring alignment");
  static_assert(TILE_N * CP_PITCH * 4 <= NS * Q4_STAGE_BYTES, "cluster partial fits in the ring");
};

struct TcParams {
  const uint8_t* wdev;
  float* out;
  int* status;
  const float* out_scale;  // [MAX_M][S] or NULL
  int64_t ldo;
  int64_t N;
  int M;
  int S;
  int spc;
  uint64_t wait_limit_ns;
};

// 8 nibbles (element 2p in nibble p, 2p + 1 in nibble p + 4) -> 4 registers of
// (q - 8) pairs in element order.
template <typename Op>
__device__ __forceinline__ void dequant8(uint32_t w, uint32_t* r) {
  uint32_t t[4];
  Op::dequant_word(w, t);
  r[0] = t[0];
  r[1] = t[1];
  r[2] = t[2];
  r[3] = t[3];
}

// ---------------------------------------------------------------- the kernel
template <typename Op>
__global__ void __launch_bounds__(TC_THREADS, 2)
    verify_tc_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap amap) {
  using L = TcSmem<TC_NS>;
  constexpr int NS = TC_NS;
  constexpr uint32_t IDESC = tc_idesc(std::is_same<Op, Bf16Op>::value ? 1u : 0u);
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x / p.S;
  const int split = blockIdx.x % p.S;
  const int M = p.M;
  const int nst = p.spc;

  const uint32_t s_base = smem_u32(smem);
  const uint32_t s_w = s_base + L::W_OFF;
  const uint32_t s_a = s_base + L::A_OFF;
  const uint32_t s_full = s_base + L::BAR_OFF;
  const uint32_t s_empty = s_full + NS * 8;
  const uint32_t s_afull = s_empty + NS * 8;
  const uint32_t s_mdone = s_afull + 2 * 8;
  const uint32_t s_dfree = s_mdone + 2 * 8;
  const uint32_t s_slot = s_base + L::SLOT_OFF;
  // [0] abort, [1] commits issued by the MMA thread, [2] stages issued by the producer
  volatile int* s_flag = reinterpret_cast<volatile int*>(smem + L::FLAG_OFF);

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(s_full + 8 * i, 1);
      mbar_init(s_empty + 8 * i, TC_DQ_WARPS + TC_EP_WARPS);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_afull + 8 * b, TC_DQ_WARPS);
      mbar_init(s_mdone + 8 * b, 1);
      mbar_init(s_dfree + 8 * b, TC_EP_WARPS);
    }
    s_flag[0] = 0;
    s_flag[1] = 0;
    s_flag[2] = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(s_slot, TC_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::SLOT_OFF);
  pdl_trigger();

  const uint8_t* wsrc = p.wdev + ((size_t)tile * p.S + split) * nst * Q4_STAGE_BYTES;
  const int kg_base = split * nst * (Q4_STAGE_K / 8);  // first 8-column group of this CTA
  const uint64_t lim = p.wait_limit_ns;
  auto fail = [&](int code) {
    atomicOr(p.status, code);
    s_flag[0] = 1;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const int pre = nst < NS ? nst : NS;
      for (int i = 0; i < pre; ++i) {
        mbar_expect_tx(s_full + 8 * i, Q4_STAGE_BYTES);
        bulk_g2s_hint(s_w + i * Q4_STAGE_BYTES, wsrc + (size_t)i * Q4_STAGE_BYTES, Q4_STAGE_BYTES,
                      s_full + 8 * i, pol);
      }
      pdl_wait();  // the activations may be written by the previous kernel
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(s_full + 8 * i, TC_ACT_STAGE_BYTES);
        tma_load_3d(s_a + i * TC_ACT_STAGE_BYTES, &amap, 0, 0, kg_base + i * (Q4_STAGE_K / 8),
                    s_full + 8 * i);
      }
      int issued = pre;
      for (int i = NS; i < nst; ++i) {
        const int slot = i % NS;
        if (!mbar_wait_bounded(s_empty + 8 * slot, ((i / NS) - 1) & 1, lim)) {
          fail(DEV_ERR_TIMEOUT_EMPTY);
          break;
        }
        if (s_flag[0]) break;
        mbar_arrive_expect_tx(s_full + 8 * slot, Q4_STAGE_BYTES + TC_ACT_STAGE_BYTES);
        bulk_g2s_hint(s_w + slot * Q4_STAGE_BYTES, wsrc + (size_t)i * Q4_STAGE_BYTES, Q4_STAGE_BYTES,
                      s_full + 8 * slot, pol);
        tma_load_3d(s_a + slot * TC_ACT_STAGE_BYTES, &amap, 0, 0, kg_base + i * (Q4_STAGE_K / 8),
                    s_full + 8 * slot);
        issued = i + 1;
      }
      s_flag[2] = issued;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      int commits = 0;
      for (int i = 0; i < nst && !s_flag[0]; ++i) {
        const int slot = i % NS;
        if (!mbar_wait_bounded(s_full + 8 * slot, (i / NS) & 1, lim)) {
          fail(DEV_ERR_TIMEOUT_FULL);
          break;
        }
        const uint32_t act = s_a + slot * TC_ACT_STAGE_BYTES;
        bool ok = true;
        for (int h = 0; h < 2; ++h) {
          const int u = 2 * i + h, buf = u & 1;
          if (!mbar_wait_bounded(s_afull + 8 * buf, (u >> 1) & 1, lim) ||
              (u >= 2 && !mbar_wait_bounded(s_dfree + 8 * buf, ((u >> 1) - 1) & 1, lim))) {
            fail(DEV_ERR_TIMEOUT_FULL);
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            const int blk = 4 * h + bb;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const uint64_t bdesc = smem_desc(act + (uint32_t)(blk * 4 + hh * 2) * 256u, 256u, 128u);
              tc_mma(tmem + buf * 128 + 64 + bb * 16, tmem + buf * 128 + bb * 16 + hh * 8, bdesc,
                     IDESC, (uint32_t)hh);
            }
          }
          tc_commit(s_mdone + 8 * buf);
          ++commits;
        }
        if (!ok) break;
      }
      s_flag[1] = commits;
    }
  } else if (warp < TC_EP_WARP0) {
    // ------------------------------------------------------------ dequantize
    const int q = warp & 3, pi = (warp - TC_DQ_WARP0) >> 2;
    const int row = q * 32 + lane;
    const uint32_t tlane = (uint32_t)(q * 32) << 16;
    for (int i = 0; i < nst && !s_flag[0]; ++i) {
      const int slot = i % NS;
      if (!mbar_wait_bounded(s_full + 8 * slot, (i / NS) & 1, lim)) {
        fail(DEV_ERR_TIMEOUT_FULL);
        break;
      }
      const uint32_t wst = s_w + slot * Q4_STAGE_BYTES;
      bool ok = true;
      for (int h = 0; h < 2; ++h) {
        const int u = 2 * i + h, buf = u & 1;
        if (u >= 2 && !mbar_wait_bounded(s_mdone + 8 * buf, ((u >> 1) - 1) & 1, lim)) {
          fail(DEV_ERR_TIMEOUT_FULL);
          ok = false;
          break;
        }
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const int sb = 2 * pi + bb;        // block within the sub-stage
          const int blk = 4 * h + sb;        // block within the stage
          const uint4 c = lds128(wst + (uint32_t)(blk * 2048 + row * 16));
          uint32_t r[16];
          dequant8<Op>(c.x, r + 0);
          dequant8<Op>(c.y, r + 4);
          dequant8<Op>(c.z, r + 8);
          dequant8<Op>(c.w, r + 12);
          tmem_st16(tmem + tlane + buf * 128 + sb * 16, r);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_afull + 8 * buf);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty + 8 * slot);
      if (!ok) break;
    }
  }

  // ------------------------------------------------------------ scale warps
  float acc[MAX_M];
#pragma unroll
  for (int m = 0; m < MAX_M; ++m) acc[m] = 0.f;
  if (warp >= TC_EP_WARP0) {
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t tlane = (uint32_t)(q * 32) << 16;
    for (int i = 0; i < nst && !s_flag[0]; ++i) {
      const int slot = i % NS;
      if (!mbar_wait_bounded(s_full + 8 * slot, (i / NS) & 1, lim)) {
        fail(DEV_ERR_TIMEOUT_FULL);
        break;
      }
      const uint4 sc = lds128(s_w + slot * Q4_STAGE_BYTES + 16384u + (uint32_t)row * 16u);
      const uint32_t dw[4] = {sc.x, sc.y, sc.z, sc.w};
      bool ok = true;
      for (int h = 0; h < 2; ++h) {
        const int u = 2 * i + h, buf = u & 1;
        if (!mbar_wait_bounded(s_mdone + 8 * buf, (u >> 1) & 1, lim)) {
          fail(DEV_ERR_TIMEOUT_FULL);
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          uint32_t v0[16], v1[16];
          tmem_ld16(tmem + tlane + buf * 128 + 64 + (2 * pr) * 16, v0);
          tmem_ld16(tmem + tlane + buf * 128 + 64 + (2 * pr + 1) * 16, v1);
          tmem_wait_ld();
          const uint32_t dpair = dw[2 * h + pr];  // fp16 d of blocks 4h + 2pr, 4h + 2pr + 1
          const float d0 = __half2float(__ushort_as_half((unsigned short)(dpair & 0xFFFF)));
          const float d1 = __half2float(__ushort_as_half((unsigned short)(dpair >> 16)));
#pragma unroll
          for (int m = 0; m < MAX_M; m += 2)
            ffma2(acc[m], acc[m + 1], d0, __uint_as_float(v0[m]), __uint_as_float(v0[m + 1]));
#pragma unroll
          for (int m = 0; m < MAX_M; m += 2)
            ffma2(acc[m], acc[m + 1], d1, __uint_as_float(v1[m]), __uint_as_float(v1[m + 1]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_dfree + 8 * buf);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty + 8 * slot);
      if (!ok) break;
    }
  }

  __syncthreads();
  const bool aborted = s_flag[0] != 0;
  if (aborted) {
    // Nothing may still be landing in shared memory or tensor memory when the
    // CTA exits: wait for this CTA's copies in flight and its last commit.
    if (warp == 0 && lane == 0) {
      const int issued = s_flag[2];
      for (int i = issued - NS < 0 ? 0 : issued - NS; i < issued; ++i)
        if (!mbar_wait_bounded(s_full + 8 * (i % NS), (i / NS) & 1, 1000000000ull))
          atomicOr(p.status, DEV_ERR_TIMEOUT_DRAIN);
    }
    if (warp == 1 && lane == 0) {
      const int commits = s_flag[1];
      for (int c = commits - 2 < 0 ? 0 : commits - 2; c < commits; ++c)
        if (!mbar_wait_bounded(s_mdone + 8 * (c & 1), (c >> 1) & 1, 1000000000ull))
          atomicOr(p.status, DEV_ERR_TIMEOUT_DRAIN);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TC_TMEM_COLS);
  }

  // ------------------------------------------------------------ epilogue
  pdl_wait();
  float* cpart = reinterpret_cast<float*>(smem + L::W_OFF);
  constexpr int CP = L::CP_PITCH;
  if (warp >= TC_EP_WARP0 && !aborted) {
    const int row = (warp & 3) * 32 + lane;
    const int64_t n = (int64_t)tile * TILE_N + row;
    for (int m = 0; m < M; ++m) {
      float v = acc[m];
      if (p.out_scale) v *= p.out_scale[m * p.S + split];
      if (p.S == 1) {
        if (n < p.N) p.out[(int64_t)m * p.ldo + n] = v;
      } else {
        cpart[row * CP + m] = v;
      }
    }
  }
  if (p.S == 1) return;
  cluster_sync_all();
  if (!aborted) {
    const int r0 = (split * TILE_N) / p.S, r1 = ((split + 1) * TILE_N) / p.S;
    const int nr = r1 - r0;
    const uint32_t cbase = smem_u32(cpart);
    for (int idx = tid; idx < nr * M; idx += TC_THREADS) {
      const int m = idx / nr, row = r0 + idx % nr;
      const uint32_t la = cbase + (uint32_t)(row * CP + m) * 4u;
      float x[MAX_SPLITS];
#pragma unroll
      for (int s = 0; s < MAX_SPLITS; ++s)
        if (s < p.S) x[s] = ld_dsmem_f32(dsmem_map(la, (uint32_t)s));
      float v = x[0];
#pragma unroll
      for (int s = 1; s < MAX_SPLITS; ++s)
        if (s < p.S) v += x[s];
      const int64_t n = (int64_t)tile * TILE_N + row;
      if (n < p.N) p.out[(int64_t)m * p.ldo + n] = v;
    }
  }
  cluster_sync_all();
}

// ---------------------------------------------------------------- layout kernels
__device__ __forceinline__ uint32_t tc_q4_code(const uint8_t* blocks, int64_t N, int64_t K, int64_t n,
                                               int64_t k) {
  if (n >= N || k >= K) return 8u;
  const uint8_t* blk = blocks + (n * (K / 32) + k / 32) * 18;
  const int e = (int)(k % 32);
  const uint8_t byte = blk[2 + (e & 15)];
  return (e < 16) ? (byte & 15u) : (byte >> 4);
}

// One thread per (stage, block, row): 16 code bytes; block-0 threads also
// write the row's 8 scales.
__global__ void repack_tc_q4_kernel(const uint8_t* __restrict__ blocks, int64_t N, int64_t K, int S,
                                    int spc, int64_t total, uint8_t* __restrict__ wdev) {
  const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gt >= total) return;
  const int row = (int)(gt % TILE_N);
  const int blk = (int)((gt / TILE_N) % 8);
  int64_t u = gt / (TILE_N * 8);  // ((tile * S + split) * spc + i)
  const int64_t stage_global = u;
  const int i = (int)(u % spc);
  u /= spc;
  const int split = (int)(u % S);
  const int64_t tile = u / S;
  const int64_t n = tile * TILE_N + row;
  const int64_t k0 = ((int64_t)split * spc + i) * Q4_STAGE_K + 32 * blk;
  uint32_t words[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t x = 0;
#pragma unroll
    for (int pn = 0; pn < 8; ++pn) {
      const int e = (pn < 4) ? 2 * pn : 2 * (pn - 4) + 1;  // element within the 8 columns
      x |= tc_q4_code(blocks, N, K, n, k0 + 8 * w + e) << (4 * pn);
    }
    words[w] = x;
  }
  uint8_t* stage = wdev + stage_global * Q4_STAGE_BYTES;
  *reinterpret_cast<uint4*>(stage + blk * 2048 + row * 16) = make_uint4(words[0], words[1], words[2], words[3]);
  if (blk == 0) {
    uint16_t d[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int64_t kb = ((int64_t)split * spc + i) * Q4_STAGE_K + 32 * b;
      d[b] = 0;
      if (n < N && kb < K) {
        const uint8_t* q = blocks + (n * (K / 32) + kb / 32) * 18;
        d[b] = (uint16_t)(q[0] | (q[1] << 8));
      }
    }
    uint4 v;
    v.x = d[0] | ((uint32_t)d[1] << 16);
    v.y = d[2] | ((uint32_t)d[3] << 16);
    v.z = d[4] | ((uint32_t)d[5] << 16);
    v.w = d[6] | ((uint32_t)d[7] << 16);
    *reinterpret_cast<uint4*>(stage + 16384 + row * 16) = v;
  }
}

__global__ void dequant_tc_q4_kernel(const uint8_t* __restrict__ wdev, int64_t N, int64_t K, int S, int spc,
                                     int64_t total, float* __restrict__ out) {
  const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gt >= total) return;
  const int row = (int)(gt % TILE_N);
  const int blk = (int)((gt / TILE_N) % 8);
  int64_t u = gt / (TILE_N * 8);
  const int64_t stage_global = u;
  const int i = (int)(u % spc);
  u /= spc;
  const int split = (int)(u % S);
  const int64_t tile = u / S;
  const int64_t n = tile * TILE_N + row;
  const int64_t k0 = ((int64_t)split * spc + i) * Q4_STAGE_K + 32 * blk;
  if (n >= N || k0 >= K) return;
  const uint8_t* stage = wdev + stage_global * Q4_STAGE_BYTES;
  const uint4 c = *reinterpret_cast<const uint4*>(stage + blk * 2048 + row * 16);
  const uint16_t dbits = *reinterpret_cast<const uint16_t*>(stage + 16384 + row * 16 + blk * 2);
  const float d = __half2float(__ushort_as_half(dbits));
  const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int w = 0; w < 4; ++w)
#pragma unroll
    for (int pn = 0; pn < 8; ++pn) {
      const int e = (pn < 4) ? 2 * pn : 2 * (pn - 4) + 1;
      const int q = (int)((words[w] >> (4 * pn)) & 15u);
      out[n * K + k0 + 8 * w + e] = d * (float)(q - 8);
    }
}

// ---------------------------------------------------------------- host side
namespace {
template <typename Op>
cudaError_t set_tc_attr() {
  cudaError_t e = cudaFuncSetAttribute(verify_tc_kernel<Op>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TcSmem<TC_NS>::BYTES);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(verify_tc_kernel<Op>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}
}  // namespace

cudaError_t prepare_tc_attributes() {
  cudaError_t e = set_tc_attr<Bf16Op>();
  if (e != cudaSuccess) return e;
  return set_tc_attr<F16Op>();
}

int tc_max_active_clusters(int S) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)S, 1, 1);
  cfg.blockDim = dim3(TC_THREADS, 1, 1);
  cfg.dynamicSmemBytes = TcSmem<TC_NS>::BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, verify_tc_kernel<Bf16Op>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return n;
}

int tc_pipeline_depth() { return TC_NS; }

cudaError_t launch_verify_tc(const VerifyParams& vp, const void* act_map, bool f16_ops, int ctas,
                             cudaStream_t st) {
  TcParams p;
  p.wdev = vp.wdev;
  p.out = vp.out;
  p.status = vp.status;
  p.out_scale = vp.out_scale;
  p.ldo = vp.ldo;
  p.N = vp.N;
  p.M = vp.M;
  p.S = vp.S;
  p.spc = vp.spc;
  p.wait_limit_ns = vp.wait_limit_ns;
  const CUtensorMap& map = *reinterpret_cast<const CUtensorMap*>(act_map);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas, 1, 1);
  cfg.blockDim = dim3(TC_THREADS, 1, 1);
  cfg.dynamicSmemBytes = TcSmem<TC_NS>::BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)vp.S;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = vp.S > 1 ? 2 : 1;
  if (f16_ops) return cudaLaunchKernelEx(&cfg, verify_tc_kernel<F16Op>, p, map);
  return cudaLaunchKernelEx(&cfg, verify_tc_kernel<Bf16Op>, p, map);
}

cudaError_t launch_repack_tc(const uint8_t* blocks, int64_t N, int64_t K, int n_tiles, int S, int spc,
                             uint8_t* wdev, cudaStream_t st) {
  const int64_t total = (int64_t)n_tiles * S * spc * 8 * TILE_N;
  repack_tc_q4_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(blocks, N, K, S, spc, total, wdev);
  return cudaGetLastError();
}

cudaError_t launch_dequant_tc(const uint8_t* wdev, int64_t N, int64_t K, int n_tiles, int S, int spc,
                              float* out, cudaStream_t st) {
  const int64_t total = (int64_t)n_tiles * S * spc * 8 * TILE_N;
  dequant_tc_q4_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(wdev, N, K, S, spc, total, out);
  return cudaGetLastError();
}

}  // namespace qmm
