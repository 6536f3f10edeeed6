// qmm_verify.cuh -- the weight-streaming verify kernel.
//
// One CTA = one row tile of W (128 rows) x one K split.  A producer warp
// streams the CTA's stages (weights: one bulk copy; activations of the drafted
// rows: one bulk copy) through an NS-deep shared-memory ring guarded by
// mbarriers.  Four consumer warps each own one quarter of every stage's K
// range for all 128 rows: they dequantize codes in registers straight into
// mma.sync A fragments (weights are the MMA's M dimension, the drafted rows
// its N = 8 or 16 dimension, "swap AB"), keep fp32 accumulators in registers
// across the whole K range, and apply the per-block (Q4_0) or per-tile (FP8)
// scale with packed fp32 FMAs.  The epilogue sums the four warps in a fixed
// order through shared memory, multiplies by the activation pre-pass's
// per-(row, split) power-of-two factor and either writes `out` (one split) or
// writes a partial and lets the last-arriving split of the tile add all
// partials in split order (deterministic, no spinning).
//
// The summation order of every output element is fixed by (N, K, plan) and
// never depends on M, so row m of the result is bit-identical for M = 1..16.
#pragma once

#include <type_traits>

#include "qmm_common.cuh"

namespace qmm {

template <int FMT>
struct FmtTraits;

template <>
struct FmtTraits<0> {  // Q4_0
  static constexpr int STAGE_K = Q4_STAGE_K;
  static constexpr int STAGE_BYTES = Q4_STAGE_BYTES;
  static constexpr int UNIT_BYTES = Q4_UNIT_BYTES;
  static constexpr int CHUNK_K = STAGE_K / CONSUMER_WARPS;  // 64
};

template <>
struct FmtTraits<1> {  // FP8 E4M3, 128x128 scales
  static constexpr int STAGE_K = F8_STAGE_K;
  static constexpr int STAGE_BYTES = F8_STAGE_BYTES;
  static constexpr int UNIT_BYTES = F8_UNIT_BYTES;
  static constexpr int CHUNK_K = STAGE_K / CONSUMER_WARPS;  // 32
};

template <int FMT, int NS>
struct SmemLayout {
  using F = FmtTraits<FMT>;
  static constexpr int W_OFF = 0;
  static constexpr int A_OFF = NS * F::STAGE_BYTES;
  static constexpr int BAR_OFF = A_OFF + NS * act_stage_bytes(F::STAGE_K);
  static constexpr int FLAG_OFF = BAR_OFF + 2 * NS * 8;
  static constexpr int BYTES = FLAG_OFF + 16;
  // epilogue reduction area (reuses the weight ring)
  static constexpr int RED_PITCH = MAX_M + 2;  // floats per row
  static constexpr int RED_BYTES = CONSUMER_WARPS * TILE_N * RED_PITCH * 4;
  static_assert(RED_BYTES <= NS * F::STAGE_BYTES, "reduction area must fit in the ring");
};

// e4m3 pair (16 bits) -> f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v16) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(r)
      : "r"(v16));
  return r;
}

// ---------------------------------------------------------------------------
// Consumer compute for one stage.  acc[r][j][0..3] is the C fragment of row
// subtile r (16 rows) and draft-row tile j (8 columns).
// ---------------------------------------------------------------------------
template <typename Op, int NT8>
__device__ __forceinline__ void q4_stage_mma(uint32_t wunit0, uint32_t abase, int lane,
                                             float (&acc)[8][2][4]) {
  const int g = lane >> 2;
  // B fragments for the warp's 64 columns: 4 k16 steps x (b0, b1) x NT8 tiles.
  uint32_t b[4][4];
  {
    const int row = (lane & 7) + ((lane >> 4) << 3);
    const int koff = ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const uint32_t addr = abase + (uint32_t)(row * act_pitch(Q4_STAGE_K) + s * 16 + koff) * 2u;
      ldmatrix_x4(addr, b[s][0], b[s][1], b[s][2], b[s][3]);
    }
  }
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const uint32_t unit = wunit0 + (uint32_t)(r * Q4_UNIT_BYTES);
    const uint4 codes = lds128(unit + 16u * lane);
    const uint2 sc = lds64(unit + 512u + 8u * g);
    const uint32_t words[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      uint32_t a0[4], a1[4];
      Op::dequant_word(words[2 * blk + 0], a0);
      Op::dequant_word(words[2 * blk + 1], a1);
      const uint32_t dpair = blk ? sc.y : sc.x;  // (d[g], d[g+8]) of this block
      const float dg = __half2float(__ushort_as_half((unsigned short)(dpair & 0xFFFF)));
      const float dg8 = __half2float(__ushort_as_half((unsigned short)(dpair >> 16)));
#pragma unroll
      for (int j = 0; j < NT8; ++j) {
        float p[4];
        Op::mma(p, a0[0], a0[1], a0[2], a0[3], b[2 * blk][2 * j], b[2 * blk][2 * j + 1], zero);
        Op::mma(p, a1[0], a1[1], a1[2], a1[3], b[2 * blk + 1][2 * j], b[2 * blk + 1][2 * j + 1], p);
        ffma2(acc[r][j][0], acc[r][j][1], dg, p[0], p[1]);
        ffma2(acc[r][j][2], acc[r][j][3], dg8, p[2], p[3]);
      }
    }
  }
}

template <int NT8>
__device__ __forceinline__ void f8_stage_mma(uint32_t wunit0, uint32_t abase, float s, int lane,
                                             float (&acc)[8][2][4]) {
  uint32_t b[2][4];
  {
    const int row = (lane & 7) + ((lane >> 4) << 3);
    const int koff = ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int st = 0; st < 2; ++st) {
      const uint32_t addr = abase + (uint32_t)(row * act_pitch(F8_STAGE_K) + st * 16 + koff) * 2u;
      ldmatrix_x4(addr, b[st][0], b[st][1], b[st][2], b[st][3]);
    }
  }
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const uint4 codes = lds128(wunit0 + (uint32_t)(r * F8_UNIT_BYTES) + 16u * lane);
    // word v: step j = v / 2, half h = v % 2 -> A registers (a0, a1) or (a2, a3)
    const uint32_t a00 = e4m3x2_to_f16x2(codes.x & 0xFFFFu), a01 = e4m3x2_to_f16x2(codes.x >> 16);
    const uint32_t a02 = e4m3x2_to_f16x2(codes.y & 0xFFFFu), a03 = e4m3x2_to_f16x2(codes.y >> 16);
    const uint32_t a10 = e4m3x2_to_f16x2(codes.z & 0xFFFFu), a11 = e4m3x2_to_f16x2(codes.z >> 16);
    const uint32_t a12 = e4m3x2_to_f16x2(codes.w & 0xFFFFu), a13 = e4m3x2_to_f16x2(codes.w >> 16);
#pragma unroll
    for (int j = 0; j < NT8; ++j) {
      float p[4];
      F16Op::mma(p, a00, a01, a02, a03, b[0][2 * j], b[0][2 * j + 1], zero);
      F16Op::mma(p, a10, a11, a12, a13, b[1][2 * j], b[1][2 * j + 1], p);
      ffma2(acc[r][j][0], acc[r][j][1], s, p[0], p[1]);
      ffma2(acc[r][j][2], acc[r][j][3], s, p[2], p[3]);
    }
  }
}

// CUDA-core baseline for Q4_0: fp32 dequantization and one FFMA per weight and
// drafted row; each lane accumulates its own columns and the four lanes of a
// group are added with warp shuffles at the end (split K inside the warp).
// Here warps own row subtiles {2w, 2w+1} over all four chunks of the stage.
template <typename T, int NT8>
__device__ __forceinline__ void q4_stage_simt(uint32_t wstage, uint32_t abase, int warp, int lane,
                                              int M, float (&acc)[2][2][MAX_M]) {
  const int g = lane >> 2, t = lane & 3;
  constexpr int MR = 8 * NT8;
#pragma unroll 1
  for (int c = 0; c < CONSUMER_WARPS; ++c) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int r = 2 * warp + rr;
      const uint32_t unit = wstage + (uint32_t)((c * 8 + r) * Q4_UNIT_BYTES);
      const uint4 codes = lds128(unit + 16u * lane);
      const uint2 sc = lds64(unit + 512u + 8u * g);
      const uint32_t words[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const uint32_t dpair = blk ? sc.y : sc.x;
        const float d[2] = {__half2float(__ushort_as_half((unsigned short)(dpair & 0xFFFF))),
                            __half2float(__ushort_as_half((unsigned short)(dpair >> 16)))};
        float part[2][MR];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int m = 0; m < MR; ++m) part[h][m] = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint32_t w = words[2 * blk + j];
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            const int pair = p & 3, half = p >> 2;
            const int h = pair & 1;  // row g or g + 8
            const int k = c * 64 + 32 * blk + 16 * j + 2 * t + half + 8 * (pair >> 1);
            const float q = __int_as_float(0x4B000000 | ((w >> (4 * p)) & 15u)) - 8388616.0f;
#pragma unroll
            for (int m = 0; m < MR; ++m) {
              if (m < M) {
                const uint32_t bits = lds_u16(abase + (uint32_t)(m * act_pitch(Q4_STAGE_K) + k) * 2u);
                float a;
                if constexpr (std::is_same<T, __nv_bfloat16>::value)
                  a = __uint_as_float(bits << 16);
                else
                  a = __half2float(__ushort_as_half((unsigned short)bits));
                part[h][m] = fmaf(q, a, part[h][m]);
              }
            }
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int m = 0; m < MR; ++m) acc[rr][h][m] = fmaf(d[h], part[h][m], acc[rr][h][m]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// The kernel.
//   FMT  0 = Q4_0, 1 = FP8
//   Op   Bf16Op or F16Op (FP8 always F16Op)
//   NT8  1 for M <= 8, 2 for M <= 16
//   SIMT true: CUDA-core baseline compute (Q4_0 only)
//   NS   pipeline depth
// ---------------------------------------------------------------------------
template <int FMT, typename Op, int NT8, bool SIMT, int NS>
__global__ void __launch_bounds__(THREADS, 2) verify_kernel(const __grid_constant__ VerifyParams p) {
  using F = FmtTraits<FMT>;
  using L = SmemLayout<FMT, NS>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x / p.S;
  const int split = blockIdx.x % p.S;
  const int M = p.M;

  const uint32_t s_base = smem_u32(smem);
  const uint32_t s_w = s_base + L::W_OFF;
  const uint32_t s_a = s_base + L::A_OFF;
  const uint32_t s_full = s_base + L::BAR_OFF;
  const uint32_t s_empty = s_full + NS * 8;
  // [0] abort, [1] this CTA adds the split partials, [2] stages issued by the producer
  volatile int* s_flag = reinterpret_cast<volatile int*>(smem + L::FLAG_OFF);

  // Rows >= M of every activation slot are never written by the copies: zero them.
  {
    constexpr int ROW_BYTES = act_pitch(F::STAGE_K) * 2;
    const int zbytes = (MAX_M - M) * ROW_BYTES;
    for (int slot = 0; slot < NS; ++slot) {
      uint8_t* base = smem + L::A_OFF + slot * act_stage_bytes(F::STAGE_K) + M * ROW_BYTES;
      for (int i = tid * 16; i < zbytes; i += THREADS * 16)
        *reinterpret_cast<uint4*>(base + i) = make_uint4(0, 0, 0, 0);
    }
  }
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(s_full + 8 * i, 1);
      mbar_init(s_empty + 8 * i, CONSUMER_WARPS);
    }
    s_flag[0] = 0;
    s_flag[1] = 0;
    s_flag[2] = 0;
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  __syncthreads();
  // Let the next kernel in the stream start its prologue (weight prefetch).
  pdl_trigger();

  const int nst = p.spc;
  const uint8_t* wsrc = p.wdev + (size_t)(tile * p.S + split) * nst * F::STAGE_BYTES;
  const uint8_t* asrc = p.act + (size_t)split * nst * act_stage_bytes(F::STAGE_K);
  const uint32_t abytes = (uint32_t)(M * act_pitch(F::STAGE_K) * 2);

  if (warp == CONSUMER_WARPS) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const int pre = nst < NS ? nst : NS;
      // Weights never depend on earlier kernels: fetch the first stages now.
      for (int i = 0; i < pre; ++i) {
        mbar_expect_tx(s_full + 8 * i, F::STAGE_BYTES);
        bulk_g2s_hint(s_w + i * F::STAGE_BYTES, wsrc + (size_t)i * F::STAGE_BYTES, F::STAGE_BYTES,
                      s_full + 8 * i, pol);
      }
      // Activations come from the pre-pass: wait for it.
      pdl_wait();
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(s_full + 8 * i, abytes);
        bulk_g2s(s_a + i * act_stage_bytes(F::STAGE_K),
                 asrc + (size_t)i * act_stage_bytes(F::STAGE_K), abytes, s_full + 8 * i);
      }
      int issued = pre;
      for (int i = NS; i < nst; ++i) {
        const int slot = i % NS;
        if (!mbar_wait_bounded(s_empty + 8 * slot, ((i / NS) - 1) & 1, p.wait_limit_ns)) {
          atomicOr(p.status, DEV_ERR_TIMEOUT_EMPTY);
          s_flag[0] = 1;
          break;
        }
        if (s_flag[0]) break;
        issued = i + 1;
        mbar_arrive_expect_tx(s_full + 8 * slot, F::STAGE_BYTES + abytes);
        bulk_g2s_hint(s_w + slot * F::STAGE_BYTES, wsrc + (size_t)i * F::STAGE_BYTES,
                      F::STAGE_BYTES, s_full + 8 * slot, pol);
        bulk_g2s(s_a + slot * act_stage_bytes(F::STAGE_K),
                 asrc + (size_t)i * act_stage_bytes(F::STAGE_K), abytes, s_full + 8 * slot);
      }
      s_flag[2] = issued;
    }
  }

  // Accumulators (registers) of the consumer warps.
  float acc[8][2][4];
  float accs[2][2][MAX_M];
  if constexpr (!SIMT) {
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[r][j][e] = 0.f;
  } else {
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int m = 0; m < MAX_M; ++m) accs[a][b][m] = 0.f;
  }

  if (warp < CONSUMER_WARPS) {
    // ------------------------------------------------------------ consumers
    for (int i = 0; i < nst; ++i) {
      const int slot = i % NS;
      if (!mbar_wait_bounded(s_full + 8 * slot, (i / NS) & 1, p.wait_limit_ns)) {
        if (lane == 0) atomicOr(p.status, DEV_ERR_TIMEOUT_FULL);
        s_flag[0] = 1;
        break;
      }
      const uint32_t wst = s_w + slot * F::STAGE_BYTES;
      const uint32_t ast = s_a + slot * act_stage_bytes(F::STAGE_K);
      if constexpr (FMT == 0) {
        if constexpr (SIMT) {
          q4_stage_simt<typename std::conditional<std::is_same<Op, Bf16Op>::value, __nv_bfloat16,
                                                  __half>::type,
                        NT8>(wst, ast, warp, lane, M, accs);
        } else {
          q4_stage_mma<Op, NT8>(wst + warp * 8 * Q4_UNIT_BYTES, ast + warp * F::CHUNK_K * 2, lane,
                                acc);
        }
      } else {
        const float s = lds_f32(wst + (F::STAGE_BYTES - 16));
        f8_stage_mma<NT8>(wst + warp * 8 * F8_UNIT_BYTES, ast + warp * F::CHUNK_K * 2, s, lane, acc);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty + 8 * slot);
      if (s_flag[0]) break;
    }
  }
  __syncthreads();
  if (s_flag[0]) {
    // Give up: no copy issued by this CTA may still be landing in shared memory
    // when the CTA exits.  Only the last NS issued stages can be in flight, and
    // each of them is the latest phase armed on its slot; its phase completes
    // when its bytes land, whether or not a consumer waited for it.
    if (warp == CONSUMER_WARPS && lane == 0) {
      const int issued = s_flag[2];
      for (int i = issued - NS < 0 ? 0 : issued - NS; i < issued; ++i) {
        if (!mbar_wait_bounded(s_full + 8 * (i % NS), (i / NS) & 1, 1000000000ull))
          atomicOr(p.status, DEV_ERR_TIMEOUT_DRAIN);
      }
    }
    __syncthreads();
    return;
  }

  // ------------------------------------------------------------ epilogue
  pdl_wait();  // order our writes after every earlier kernel's
  float* red = reinterpret_cast<float*>(smem + L::W_OFF);
  constexpr int RP = L::RED_PITCH;
  if (warp < CONSUMER_WARPS) {
    const int g = lane >> 2, t = lane & 3;
    if constexpr (!SIMT) {
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int j = 0; j < NT8; ++j) {
          const int row = 16 * r + g, col = 8 * j + 2 * t;
          float* d0 = red + (warp * TILE_N + row) * RP + col;
          float* d1 = red + (warp * TILE_N + row + 8) * RP + col;
          *reinterpret_cast<float2*>(d0) = make_float2(acc[r][j][0], acc[r][j][1]);
          *reinterpret_cast<float2*>(d1) = make_float2(acc[r][j][2], acc[r][j][3]);
        }
    } else {
      // add the four lanes of each group (their column subsets of K)
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int m = 0; m < MAX_M; ++m) {
            float v = accs[rr][h][m];
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
            accs[rr][h][m] = v;
          }
      // the SIMT warps own distinct rows: reduction slot 0 holds every row
      if (t == 0) {
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int row = 16 * (2 * warp + rr) + g + 8 * h;
#pragma unroll
            for (int m = 0; m < MAX_M; ++m) red[row * RP + m] = accs[rr][h][m];
          }
      }
    }
  }
  __syncthreads();

  const int64_t n = (int64_t)tile * TILE_N + tid;
  if (tid < TILE_N) {
    for (int m = 0; m < M; ++m) {
      constexpr int NRED = SIMT ? 1 : CONSUMER_WARPS;
      float v = red[tid * RP + m];
#pragma unroll
      for (int w = 1; w < NRED; ++w) v += red[(w * TILE_N + tid) * RP + m];
      v *= p.out_scale[m * p.S + split];
      if (p.S == 1) {
        if (n < p.N) p.out[(int64_t)m * p.ldo + n] = v;
      } else {
        p.partial[(((size_t)tile * p.S + split) * MAX_M + m) * TILE_N + tid] = v;
      }
    }
  }
  if (p.S == 1) return;

  // Split-K: the last split of this tile to arrive adds all partials in split order.
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&p.counters[tile], 1);
    s_flag[1] = (prev == p.S - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!s_flag[1]) return;
  __threadfence();
  if (tid < TILE_N) {
    for (int m = 0; m < M; ++m) {
      float v = 0.f;
      for (int s = 0; s < p.S; ++s) {
        const float x = __ldcg(&p.partial[(((size_t)tile * p.S + s) * MAX_M + m) * TILE_N + tid]);
        v = (s == 0) ? x : v + x;
      }
      if (n < p.N) p.out[(int64_t)m * p.ldo + n] = v;
    }
  }
  if (tid == 0) p.counters[tile] = 0;
}

}  // namespace qmm
