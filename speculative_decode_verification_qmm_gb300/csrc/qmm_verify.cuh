// qmm_verify.cuh -- the weight-streaming verify kernel.
//
// One CTA = one row tile of W (128 rows) x one K split; it streams its stages
// through an NS-deep shared-memory ring.  A stage is four column chunks and
// each chunk has its own full mbarrier: one bulk copy of the chunk's repacked
// weights and one tensor-map box of the activations (R = 8 or 16 drafted rows
// x the chunk's columns) complete it.  There is no producer warp: thread 0
// requests the first NS stages, and afterwards the last warp to finish with a
// chunk (a shared-memory counter picks it, nobody waits) requests the same
// chunk of the stage NS ahead into the slot it just freed.  Eight compute
// warps (chunk x half of the tile's rows) wait for their own chunk only, dequantize their codes in registers straight into
// mma.sync A fragments (weights are the MMA's M dimension, drafted rows its
// N = 8 or 16 dimension, "swap AB"), keep fp32 accumulators in registers
// across the CTA's K range, and apply the per-block (Q4_0) or per-tile (FP8)
// scale with packed fp32 FMAs.  The epilogue adds the four chunk partials in a
// fixed order through shared memory, multiplies by the pre-pass's per-(row,
// split) power-of-two factor, and either writes `out` (one split) or, when the
// K range is split, writes its partial to the handle's workspace and bumps the
// tile's arrival count: the last of the S splits to arrive adds the S partials
// in split order and writes the tile (deterministic; no split waits for
// another, so they need not be resident at the same time).
//
// The summation order of every output element is fixed by (N, K, plan) and
// never depends on M, so row m of the result is bit-identical for M = 1..16.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "qmm_common.cuh"

namespace qmm {

template <int FMT>
struct FmtTraits;

template <>
struct FmtTraits<0> {  // Q4_0
  static constexpr int STAGE_K = Q4_STAGE_K;
  static constexpr int STAGE_BYTES = Q4_STAGE_BYTES;
  static constexpr int CHUNK_BYTES = Q4_CHUNK_BYTES;
  static constexpr int UNIT_BYTES = Q4_UNIT_BYTES;
  static constexpr int CHUNK_K = STAGE_K / STAGE_CHUNKS;  // 64
};

template <>
struct FmtTraits<1> {  // FP8 E4M3, 128x128 scales
  static constexpr int STAGE_K = F8_STAGE_K;
  static constexpr int STAGE_BYTES = F8_STAGE_BYTES;
  static constexpr int CHUNK_BYTES = F8_CHUNK_BYTES;
  static constexpr int UNIT_BYTES = F8_UNIT_BYTES;
  static constexpr int CHUNK_K = STAGE_K / STAGE_CHUNKS;  // 32
};

template <>
struct FmtTraits<2> {  // Q8_0
  static constexpr int STAGE_K = Q8_STAGE_K;
  static constexpr int STAGE_BYTES = Q8_STAGE_BYTES;
  static constexpr int CHUNK_BYTES = Q8_CHUNK_BYTES;
  static constexpr int UNIT_BYTES = Q8_UNIT_BYTES;
  static constexpr int CHUNK_K = STAGE_K / STAGE_CHUNKS;  // 32: one Q8_0 block
};

// Row subtiles (16 rows) per compute warp: the 8 subtiles of a tile are split
// into two halves.
constexpr int WARP_SUBTILES = 8 * STAGE_CHUNKS / COMPUTE_WARPS;  // 4
static_assert(WARP_SUBTILES * 2 == 8, "two row halves per chunk");

// R = activation rows staged per chunk (8 for M <= 8, else 16).  Offsets are
// from the dynamic shared memory base rounded up to 1024 bytes (BYTES
// includes that slack), the period of the tensor map's swizzle.
template <int FMT, int NS, int R>
struct SmemLayout {
  using F = FmtTraits<FMT>;
  static constexpr int W_OFF = 0;
  static constexpr int A_OFF = NS * F::STAGE_BYTES;
  static constexpr int A_CHUNK = F::CHUNK_K * R * 2;  // one tensor-map box: R rows x CHUNK_K
  static constexpr int A_STAGE = STAGE_CHUNKS * A_CHUNK;
  static constexpr int A_BYTES = NS * A_STAGE;
  // full[NS][4] mbarriers, then per (slot, chunk) {finished-warp count, last stage requested}
  static constexpr int BAR_OFF = A_OFF + A_BYTES;
  static constexpr int FLAG_OFF = BAR_OFF + 2 * NS * STAGE_CHUNKS * 8;
  static constexpr int BYTES = FLAG_OFF + 16 + 1024;
  // epilogue areas (reuse the weight ring): chunk partials [chunk][row][RED_PITCH],
  // (the split partials go to the workspace in global memory)
  static constexpr int RED_PITCH = MAX_M + 2;  // floats per row
  static constexpr int RED_BYTES = STAGE_CHUNKS * TILE_N * RED_PITCH * 4;
  // then the finished tile [m][row] for the greedy epilogue
  static constexpr int FIN_OFF = RED_BYTES;
  static constexpr int FIN_BYTES = MAX_M * TILE_N * 4;
  static_assert(FIN_OFF + FIN_BYTES <= NS * F::STAGE_BYTES, "the epilogue areas must fit in the ring");
  static_assert(A_OFF % 1024 == 0 && A_CHUNK % (F::CHUNK_K * 2 * 8) == 0,
                "every box starts on a swizzle period");
  static_assert(F::CHUNK_BYTES % 16 == 0 && BAR_OFF % 8 == 0, "alignment");
};

// Shared-memory address of the 8 values k = 8 kc .. 8 kc + 7 of activation
// row `row` in a chunk box: rows of RB = 2 x CHUNK_K bytes, and the tensor
// map's RB-byte swizzle moves 16-byte piece kc of row r to kc ^ (r & 7)
// (128-byte rows) or kc ^ ((r >> 1) & 3) (64-byte rows).  Box bases are
// aligned to the swizzle period, so row r's pattern depends on r alone.
template <int RB>
__device__ __forceinline__ uint32_t act_piece(uint32_t abase, int row, int kc) {
  static_assert(RB == 128 || RB == 64, "swizzle width");
  const int sw = RB == 128 ? (row & 7) : ((row >> 1) & 3);
  return abase + (uint32_t)(row * RB + ((kc ^ sw) << 4));
}

// B fragments for the NSTEP k16 steps of the activation chunk at `abase` (R
// rows of RB bytes): b[s][0..1] serve draft rows 0..7, b[s][2..3] rows 8..15
// (R = 16 only).
template <int NSTEP, int R, int RB>
__device__ __forceinline__ void load_b_frags(uint32_t abase, int lane, uint32_t (&b)[NSTEP][4]) {
  static_assert(NSTEP % 2 == 0, "pairs of k16 steps");
  if constexpr (R == 16) {
    // matrices: rows 0-7 / 8-15 x columns 0-7 / 8-15 of step s
    const int row = (lane & 7) + ((lane >> 4) << 3);
    const int kh = (lane >> 3) & 1;
#pragma unroll
    for (int s = 0; s < NSTEP; ++s)
      ldmatrix_x4(act_piece<RB>(abase, row, 2 * s + kh), b[s][0], b[s][1], b[s][2], b[s][3]);
  } else {
    // matrices: columns 0-7 / 8-15 of steps s and s + 1
    const int row = lane & 7;
    const int kq = lane >> 3;
#pragma unroll
    for (int s = 0; s < NSTEP; s += 2) {
      ldmatrix_x4(act_piece<RB>(abase, row, 2 * s + kq), b[s][0], b[s][1], b[s + 1][0], b[s + 1][1]);
      b[s][2] = b[s][3] = b[s + 1][2] = b[s + 1][3] = 0u;
    }
  }
}

// ---------------------------------------------------------------------------
// Compute for one stage and one warp.  acc[r][j][0..3] is the C fragment of
// the warp's row subtile r (16 rows) and draft-row tile j (8 columns).
// ---------------------------------------------------------------------------
template <typename Op, int NT8>
__device__ __forceinline__ void q4_stage_mma(uint32_t wunit0, uint32_t abase, int lane,
                                             float (&acc)[WARP_SUBTILES][2][4]) {
  const int g = lane >> 2;
  uint32_t b[4][4];
  load_b_frags<4, 8 * NT8, 2 * Q4_STAGE_K / STAGE_CHUNKS>(abase, lane, b);
  // The weights enter the MMA as the exact values q - 8 (bf16 or f16), so a
  // block's partial is the sum of exact products and never the difference of
  // two large sums: a block of zero weights gives exactly zero whatever the
  // activations are.
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int r = 0; r < WARP_SUBTILES; ++r) {
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
        float pp[4];
        Op::mma(pp, a0[0], a0[1], a0[2], a0[3], b[2 * blk][2 * j], b[2 * blk][2 * j + 1], zero);
        Op::mma(pp, a1[0], a1[1], a1[2], a1[3], b[2 * blk + 1][2 * j], b[2 * blk + 1][2 * j + 1], pp);
        ffma2(acc[r][j][0], acc[r][j][1], dg, pp[0], pp[1]);
        ffma2(acc[r][j][2], acc[r][j][3], dg8, pp[2], pp[3]);
      }
    }
  }
}

// Q8_0 codes stored as u = q + 128, two bytes -> f16x2 (q, exact): one byte
// permute gives (b_lo, 0x64, b_hi, 0x64) = 1024 + u = 1152 + q, and one packed
// subtraction of 1152 leaves q (every integer below 2048 is an f16 value).
__device__ __forceinline__ uint32_t u8x2_to_f16x2(uint32_t w, uint32_t sel) {
  uint32_t x, r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(x) : "r"(w), "r"(0x64646464u), "r"(sel));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(0x64806480u));
  return r;
}

// Q8_0: the chunk's 32 columns are one block per row.  The weights enter the
// MMA as the exact codes q (f16), so each block's partial is a sum of exact
// products; the block scale d (per row) is then applied with packed fp32
// FMAs, as for Q4_0.
template <int NT8>
__device__ __forceinline__ void q8_stage_mma(uint32_t wunit0, uint32_t abase, int lane,
                                             float (&acc)[WARP_SUBTILES][2][4]) {
  const int g = lane >> 2;
  uint32_t b[2][4];
  load_b_frags<2, 8 * NT8, 2 * Q8_STAGE_K / STAGE_CHUNKS>(abase, lane, b);
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int r = 0; r < WARP_SUBTILES; ++r) {
    const uint32_t unit = wunit0 + (uint32_t)(r * Q8_UNIT_BYTES);
    const uint4 codes = lds128(unit + 16u * lane);
    const uint32_t dpair = lds32(unit + 512u + 4u * g);  // (d[g], d[g + 8])
    // word v: k16 step v / 2, half v % 2 -> A registers (a0, a1) or (a2, a3)
    const uint32_t a00 = u8x2_to_f16x2(codes.x, 0x4140u), a01 = u8x2_to_f16x2(codes.x, 0x4342u);
    const uint32_t a02 = u8x2_to_f16x2(codes.y, 0x4140u), a03 = u8x2_to_f16x2(codes.y, 0x4342u);
    const uint32_t a10 = u8x2_to_f16x2(codes.z, 0x4140u), a11 = u8x2_to_f16x2(codes.z, 0x4342u);
    const uint32_t a12 = u8x2_to_f16x2(codes.w, 0x4140u), a13 = u8x2_to_f16x2(codes.w, 0x4342u);
    const float dg = __half2float(__ushort_as_half((unsigned short)(dpair & 0xFFFF)));
    const float dg8 = __half2float(__ushort_as_half((unsigned short)(dpair >> 16)));
#pragma unroll
    for (int j = 0; j < NT8; ++j) {
      float pp[4];
      F16Op::mma(pp, a00, a01, a02, a03, b[0][2 * j], b[0][2 * j + 1], zero);
      F16Op::mma(pp, a10, a11, a12, a13, b[1][2 * j], b[1][2 * j + 1], pp);
      ffma2(acc[r][j][0], acc[r][j][1], dg, pp[0], pp[1]);
      ffma2(acc[r][j][2], acc[r][j][3], dg8, pp[2], pp[3]);
    }
  }
}

template <int NT8>
__device__ __forceinline__ void f8_stage_mma(uint32_t wunit0, uint32_t abase, float s, int lane,
                                             float (&acc)[WARP_SUBTILES][2][4]) {
  uint32_t b[2][4];
  load_b_frags<2, 8 * NT8, 2 * F8_STAGE_K / STAGE_CHUNKS>(abase, lane, b);
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int r = 0; r < WARP_SUBTILES; ++r) {
    const uint4 codes = lds128(wunit0 + (uint32_t)(r * F8_UNIT_BYTES) + 16u * lane);
    // word v: k16 step v / 2, half v % 2 -> A registers (a0, a1) or (a2, a3)
    const uint32_t a00 = e4m3x2_to_f16x2(codes.x & 0xFFFFu), a01 = e4m3x2_to_f16x2(codes.x >> 16);
    const uint32_t a02 = e4m3x2_to_f16x2(codes.y & 0xFFFFu), a03 = e4m3x2_to_f16x2(codes.y >> 16);
    const uint32_t a10 = e4m3x2_to_f16x2(codes.z & 0xFFFFu), a11 = e4m3x2_to_f16x2(codes.z >> 16);
    const uint32_t a12 = e4m3x2_to_f16x2(codes.w & 0xFFFFu), a13 = e4m3x2_to_f16x2(codes.w >> 16);
#pragma unroll
    for (int j = 0; j < NT8; ++j) {
      float pp[4];
      F16Op::mma(pp, a00, a01, a02, a03, b[0][2 * j], b[0][2 * j + 1], zero);
      F16Op::mma(pp, a10, a11, a12, a13, b[1][2 * j], b[1][2 * j + 1], pp);
      ffma2(acc[r][j][0], acc[r][j][1], s, pp[0], pp[1]);
      ffma2(acc[r][j][2], acc[r][j][3], s, pp[2], pp[3]);
    }
  }
}

// CUDA-core baseline for Q4_0: fp32 dequantization and one FMA per weight and
// drafted row; each lane accumulates its own columns and the four lanes of a
// group are added with warp shuffles at the end (split K inside the warp).
// Warp w owns row subtile w over all four chunks of every stage; this is one
// chunk (its unit at `unit`, the chunk's activation box at `achunk`).
template <typename T, int NT8>
__device__ __forceinline__ void q4_chunk_simt(uint32_t unit, uint32_t achunk, int lane, int M,
                                              float (&acc)[2][MAX_M]) {
  const int g = lane >> 2, t = lane & 3;
  constexpr int MR = 8 * NT8;
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
      for (int pn = 0; pn < 8; ++pn) {
        const int pair = pn & 3, half = pn >> 2;
        const int h = pair & 1;  // row g or g + 8
        const int k = 32 * blk + 16 * j + 2 * t + half + 8 * (pair >> 1);  // column in the chunk
        const float qv = __int_as_float(0x4B000000 | ((w >> (4 * pn)) & 15u)) - 8388616.0f;
#pragma unroll
        for (int m = 0; m < MR; ++m) {
          if (m < M) {
            const uint32_t bits = lds_u16(act_piece<128>(achunk, m, k >> 3) + (uint32_t)(k & 7) * 2u);
            float a;
            if constexpr (std::is_same<T, __nv_bfloat16>::value)
              a = __uint_as_float(bits << 16);
            else
              a = __half2float(__ushort_as_half((unsigned short)bits));
            part[h][m] = fmaf(qv, a, part[h][m]);
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int m = 0; m < MR; ++m) acc[h][m] = fmaf(d[h], part[h][m], acc[h][m]);
  }
}

// ---------------------------------------------------------------------------
// Greedy acceptance, the step after the verify product: the target's greedy
// token at every block position is the argmax of its row of scores, and the
// drafts are accepted while they agree with it (see qmm_verify_greedy in
// qmm.h).  Called by the CTA that finished row tile `tile` (its scores, times
// the pre-pass multipliers, in fin[m][row]) with every thread.  For each
// drafted row m the tile's best (score, row) pair joins the call-wide maximum
// through one 64-bit atomicMax on a key that orders scores as floats and
// equal scores by the lower row (so the result is the first index of the
// maximum whatever order the tiles finish in; a NaN counts as the largest).
// The last tile of the call to finish writes argmax_out, accept_out and clears
// the state for the next call.  `valid` false (the CTA gave up on a wait): the
// tile only counts its arrival.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long greedy_key(float v, int64_t row) {
  uint32_t u = __float_as_uint(v + 0.0f);      // -0 -> +0
  if (v != v) u = 0x7FC00000u;                 // every NaN as one positive NaN
  const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)o << 32) | (uint32_t)~(uint32_t)row;
}

static __device__ __noinline__ void greedy_tile(const VerifyParams& p, const float* fin, int tile, int M,
                                         bool valid, int tid, volatile int* flag) {
  const int warp = tid >> 5, lane = tid & 31;
  if (valid) {
    // warp w: drafted rows w and w + 8; lane l: tile rows l, l + 32, l + 64, l + 96
    for (int m = warp; m < M; m += THREADS / 32) {
      unsigned long long best = 0;
#pragma unroll
      for (int r = 0; r < TILE_N / 32; ++r) {
        const int row = lane + 32 * r;
        const int64_t n = (int64_t)tile * TILE_N + row;
        if (n < p.N) {
          const unsigned long long k = greedy_key(fin[m * TILE_N + row], n);
          best = k > best ? k : best;
        }
      }
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, best, d);
        best = o > best ? o : best;
      }
      if (lane == 0 && best) atomicMax(p.best + m, best);
    }
  }
  // One GPU-scope acquire-release add after the CTA barrier: it releases the
  // maxima of this tile and, for the last tile, acquires every other tile's.
  __syncthreads();
  if (tid == 0) {
    int prev;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;"
                 : "=r"(prev)
                 : "l"(p.tiles_done)
                 : "memory");
    flag[3] = prev == p.n_tiles - 1 ? 1 : 0;
  }
  __syncthreads();
  if (flag[3] && tid == 0) {
    *p.tiles_done = 0;
    int32_t y[MAX_M];
    for (int m = 0; m < M; ++m) {
      const unsigned long long k = __ldcg(p.best + m);
      y[m] = (int32_t)~(uint32_t)(k & 0xFFFFFFFFull);
      p.argmax_out[m] = y[m];
    }
    int k = 0;
    while (k < M - 1 && y[k] == p.tokens[k + 1]) ++k;
    p.accept_out[0] = k;
    p.accept_out[1] = y[k];
    for (int m = 0; m < MAX_M; ++m) p.best[m] = 0ull;
  }
}

// ---------------------------------------------------------------------------
// The kernel.
//   FMT  0 = Q4_0, 1 = FP8, 2 = Q8_0
//   Op   Bf16Op or F16Op (FP8 always F16Op)
//   NT8  1 for M <= 8, 2 for M <= 16 (R = 8 * NT8 activation rows staged)
//   SIMT true: CUDA-core baseline compute (Q4_0 only)
//   NS   pipeline depth in stages
//   GREEDY  also the greedy acceptance step (p.best and the rest set)
// `amap` is a 2-D tensor map over the 16-bit activation rows (see
// qmm_common.cuh) whose boxes are CHUNK_K columns x R rows, swizzled by
// 2 x CHUNK_K bytes.
// ---------------------------------------------------------------------------
// Two CTAs per SM: 16 warps, four per SM sub-partition, up to 128 registers.
template <int FMT, typename Op, int NT8, bool SIMT, int NS, bool GREEDY>
__global__ void __launch_bounds__(THREADS, 2)
    verify_kernel(const __grid_constant__ VerifyParams p, const __grid_constant__ CUtensorMap amap) {
  using F = FmtTraits<FMT>;
  constexpr int R = 8 * NT8;
  using L = SmemLayout<FMT, NS, R>;
  constexpr int NCH = STAGE_CHUNKS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x / p.S;
  const int split = blockIdx.x % p.S;
  const int M = p.M;

  const uint32_t s_raw = smem_u32(smem_raw);
  const uint32_t s_base = (s_raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (s_base - s_raw);
  const uint32_t s_w = s_base + L::W_OFF;
  const uint32_t s_a = s_base + L::A_OFF;
  const uint32_t s_full = s_base + L::BAR_OFF;        // [slot][chunk]
  auto full_bar = [&](int slot, int c) { return s_full + (uint32_t)(slot * NCH + c) * 8u; };
  // [slot][chunk][0]: warps done with the chunk's current stage; [1]: last stage requested
  int* s_chunk = reinterpret_cast<int*>(smem + L::BAR_OFF + NS * NCH * 8);
  // MMA warps: two per chunk; CUDA-core warps: every warp reads every chunk
  constexpr int READERS = SIMT ? COMPUTE_WARPS : COMPUTE_WARPS / NCH;
  // [0] abort
  volatile int* s_flag = reinterpret_cast<volatile int*>(smem + L::FLAG_OFF);

  if (tid == 0) {
    for (int i = 0; i < NS * NCH; ++i) {
      mbar_init(s_full + 8 * i, 1);
      s_chunk[2 * i] = 0;
      s_chunk[2 * i + 1] = -1;
    }
    s_flag[0] = 0;
    s_flag[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    QMM_STAMP(p, QMM_TR_ENTRY, global_timer_ns());
    QMM_STAMP(p, QMM_TR_SMID, sm_id());
  }
  // Let the next kernel in the stream start its prologue (weight prefetch).
  pdl_trigger();

  const int nst = p.spc;
  const int64_t gstage0 = (int64_t)split * nst;  // global index of this CTA's first stage
  const uint8_t* wsrc = p.wdev + ((size_t)tile * p.S + split) * nst * F::STAGE_BYTES;
  const int k0 = (int)(gstage0 * F::STAGE_K);  // first column of this CTA (a multiple of 8)
  constexpr uint32_t CHUNK_TX = F::CHUNK_BYTES + L::A_CHUNK;

  const uint64_t pol = policy_evict_first();
  // Request chunk c of stage i into ring slot i % NS (weights, then activations).
  auto request = [&](int i, int c, bool weights, bool act) {
    const int slot = i % NS;
    if (weights) {
      mbar_arrive_expect_tx(full_bar(slot, c), CHUNK_TX);
      bulk_g2s_hint(s_w + slot * F::STAGE_BYTES + c * F::CHUNK_BYTES,
                    wsrc + (size_t)i * F::STAGE_BYTES + c * F::CHUNK_BYTES, F::CHUNK_BYTES,
                    full_bar(slot, c), pol);
      s_chunk[2 * (slot * NCH + c) + 1] = i;
    }
    if (act)
      tma_load_2d(s_a + slot * L::A_STAGE + c * L::A_CHUNK, &amap,
                  k0 + i * F::STAGE_K + c * F::CHUNK_K, 0, full_bar(slot, c));
  };
  // The last of the READERS warps done with chunk c of stage i (ring slot
  // i % NS) requests the same chunk of stage i + NS into that slot.  Called
  // by lane 0 after the warp's reads of the chunk.
  auto release = [&](int i, int c) {
    const int slot = i % NS;
    int* cnt = s_chunk + 2 * (slot * NCH + c);
    // acquire-release: this warp's reads of the chunk (ordered before the
    // add by __syncwarp) come before whatever the last reader issues next
    int done;
    asm volatile("atom.add.acq_rel.cta.shared::cta.s32 %0, [%1], 1;"
                 : "=r"(done)
                 : "r"(smem_u32(cnt))
                 : "memory");
    ++done;
    if (done == READERS) {
      *cnt = 0;
      if (i + NS < nst && !s_flag[0]) {
        fence_proxy_async_smem();  // the readers' loads come before the copy's writes
        request(i + NS, c, true, true);
      }
    }
  };

  if (tid == 0) {
    const int pre = nst < NS ? nst : NS;
    // Weights never depend on earlier kernels: fetch the first stages now.
    for (int i = 0; i < pre; ++i)
      for (int c = 0; c < NCH; ++c) request(i, c, true, false);
    // Activations may be written by the previous kernel: wait for it.
    pdl_wait();
    QMM_STAMP(p, QMM_TR_PDL, global_timer_ns());
    for (int i = 0; i < pre; ++i)
      for (int c = 0; c < NCH; ++c) request(i, c, false, true);
  }
  __syncwarp();

  // Accumulators (registers) of the compute warps.
  float acc[WARP_SUBTILES][2][4];
  float accs[2][MAX_M];
  if constexpr (!SIMT) {
#pragma unroll
    for (int r = 0; r < WARP_SUBTILES; ++r)
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[r][j][e] = 0.f;
  } else {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int m = 0; m < MAX_M; ++m) accs[h][m] = 0.f;
  }

  const int chunk = warp & (NCH - 1);
  const int sub0 = (warp / NCH) * WARP_SUBTILES;  // first row subtile of this warp
  if (warp < COMPUTE_WARPS) {
    // ------------------------------------------------------------ compute
    if constexpr (!SIMT) {
      const float* f8s = FMT == 1 ? p.f8_scale + (size_t)tile * p.S * nst + gstage0 : nullptr;
      for (int i = 0; i < nst; ++i) {
        const int slot = i % NS;
        float fs = 0.f;
        if constexpr (FMT == 1) fs = __ldg(f8s + i);  // lands while the chunk is awaited
        if (!mbar_wait_bounded(full_bar(slot, chunk), (i / NS) & 1, p.wait_limit_ns)) {
          if (lane == 0) atomicOr(p.status, DEV_ERR_TIMEOUT_FULL);
          s_flag[0] = 1;
          break;
        }
        if (i == 0 && warp == 0 && lane == 0) QMM_STAMP(p, QMM_TR_DATA, global_timer_ns());
        const uint32_t wch = s_w + slot * F::STAGE_BYTES + chunk * F::CHUNK_BYTES +
                             sub0 * F::UNIT_BYTES;
        const uint32_t ach = s_a + slot * L::A_STAGE + chunk * L::A_CHUNK;
        if constexpr (FMT == 0)
          q4_stage_mma<Op, NT8>(wch, ach, lane, acc);
        else if constexpr (FMT == 1)
          f8_stage_mma<NT8>(wch, ach, fs, lane, acc);
        else
          q8_stage_mma<NT8>(wch, ach, lane, acc);
        __syncwarp();
        if (lane == 0) release(i, chunk);
        __syncwarp();
        if (s_flag[0]) break;
      }
      if (warp == 0 && lane == 0) QMM_STAMP(p, QMM_TR_LOOP, global_timer_ns());
    } else {
      using T = typename std::conditional<std::is_same<Op, Bf16Op>::value, __nv_bfloat16,
                                          __half>::type;
      bool ok = true;
      for (int i = 0; i < nst && ok; ++i) {
        const int slot = i % NS;
#pragma unroll 1
        for (int c = 0; c < NCH; ++c) {
          if (!mbar_wait_bounded(full_bar(slot, c), (i / NS) & 1, p.wait_limit_ns)) {
            if (lane == 0) atomicOr(p.status, DEV_ERR_TIMEOUT_FULL);
            s_flag[0] = 1;
            ok = false;
            break;
          }
          q4_chunk_simt<T, NT8>(s_w + slot * F::STAGE_BYTES + c * F::CHUNK_BYTES +
                                    warp * F::UNIT_BYTES,
                                s_a + slot * L::A_STAGE + c * L::A_CHUNK, lane, M, accs);
          __syncwarp();
          if (lane == 0) release(i, c);
          __syncwarp();
        }
        if (s_flag[0]) ok = false;
      }
    }
  }
  __syncthreads();
  if (tid == 0) QMM_STAMP(p, QMM_TR_EPI, global_timer_ns());
  const bool aborted = s_flag[0] != 0;
  if (aborted) {
    // Give up: no copy requested by this CTA may still be landing in shared
    // memory when the CTA exits.  The last stage requested into each (slot,
    // chunk) is the latest phase armed on its barrier; that phase completes
    // when its bytes land, whether or not a compute warp waited for it.
    if (tid == 0) {
      for (int x = 0; x < NS * NCH; ++x) {
        const int i = s_chunk[2 * x + 1];
        if (i >= 0 && !mbar_wait_bounded(s_full + 8u * x, (i / NS) & 1, 1000000000ull))
          atomicOr(p.status, DEV_ERR_TIMEOUT_DRAIN);
      }
    }
    __syncthreads();
    // An aborted CTA writes nothing but still counts its arrival, so that the
    // tile's count returns to zero for the next call.
  }

  // ------------------------------------------------------------ epilogue
  pdl_wait();  // order our writes after every earlier kernel's
  float* red = reinterpret_cast<float*>(smem + L::W_OFF);
  constexpr int RP = L::RED_PITCH;
  if (warp < COMPUTE_WARPS && !aborted) {
    const int g = lane >> 2, t = lane & 3;
    if constexpr (!SIMT) {
#pragma unroll
      for (int r = 0; r < WARP_SUBTILES; ++r)
#pragma unroll
        for (int j = 0; j < NT8; ++j) {
          const int row = 16 * (sub0 + r) + g, col = 8 * j + 2 * t;
          float* d0 = red + (chunk * TILE_N + row) * RP + col;
          float* d1 = red + (chunk * TILE_N + row + 8) * RP + col;
          *reinterpret_cast<float2*>(d0) = make_float2(acc[r][j][0], acc[r][j][1]);
          *reinterpret_cast<float2*>(d1) = make_float2(acc[r][j][2], acc[r][j][3]);
        }
    } else {
      // add the four lanes of each group (their column subsets of K)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int m = 0; m < MAX_M; ++m) {
          float v = accs[h][m];
          v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
          v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
          accs[h][m] = v;
        }
      if (t == 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = 16 * warp + g + 8 * h;
#pragma unroll
          for (int m = 0; m < MAX_M; ++m) red[row * RP + m] = accs[h][m];
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0) QMM_STAMP(p, QMM_TR_RED, global_timer_ns());

  // The CTA's partial: the chunk partials added in chunk order, times the
  // pre-pass's factor of this (row, split).  With one split it is the result;
  // otherwise it goes to the handle's workspace, [tile][split][m][row].
  float* mine = p.ws + ((int64_t)tile * p.S + split) * (MAX_M * TILE_N);
  float* fin = reinterpret_cast<float*>(smem + L::W_OFF + L::FIN_OFF);  // [m][row], greedy only
  if (tid < TILE_N && !aborted) {
    constexpr int NRED = SIMT ? 1 : STAGE_CHUNKS;
    const int64_t n = (int64_t)tile * TILE_N + tid;
    for (int m = 0; m < M; ++m) {
      float v = red[tid * RP + m];
#pragma unroll
      for (int c = 1; c < NRED; ++c) v += red[(c * TILE_N + tid) * RP + m];
      if (p.out_scale) v *= p.out_scale[m * p.S + split];
      if (p.S == 1) {
        if (n < p.N) p.out[(int64_t)m * p.ldo + n] = v;
        if constexpr (GREEDY) fin[m * TILE_N + tid] = v;
      } else {
        mine[m * TILE_N + tid] = v;
      }
    }
  }
  if (p.S == 1) {
    if (tid == 0) QMM_STAMP(p, QMM_TR_PART, global_timer_ns());
    if constexpr (GREEDY) {
      __syncthreads();  // fin complete
      greedy_tile(p, fin, tile, M, !aborted, tid, s_flag);
    }
    if (tid == 0) QMM_STAMP(p, QMM_TR_EXIT, global_timer_ns());
    return;
  }

  // Split K: the last of the tile's S CTAs to arrive adds the S partials in
  // split order (the count goes back to zero for the next call).  Nobody
  // waits for anybody, so the splits need not be resident together.
  // One GPU-scope acquire-release add by thread 0 after the CTA barrier:
  // it releases every thread's partial (ordered before it by the barrier)
  // and, for the last arrival, acquires the other splits' partials for the
  // threads ordered after it by the second barrier.
  __syncthreads();
  if (tid == 0) {
    QMM_STAMP(p, QMM_TR_PART, global_timer_ns());
    int prev;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;"
                 : "=r"(prev)
                 : "l"(p.counters + tile)
                 : "memory");
    const bool last = prev == p.S - 1;
    if (last) p.counters[tile] = 0;
    s_flag[1] = last ? 1 : 0;
    QMM_STAMP(p, QMM_TR_ARRIVE, global_timer_ns());
    QMM_STAMP(p, QMM_TR_LAST, last ? 1ull : 0ull);
  }
  __syncthreads();
  if (s_flag[1] && !aborted) {
    const float* base = p.ws + (int64_t)tile * p.S * (MAX_M * TILE_N);
    // float4 piece q: drafted row q / 32, rows 4 (q % 32) .. + 3
    for (int q = tid; q < M * (TILE_N / 4); q += THREADS) {
      const int m = q / (TILE_N / 4), row = 4 * (q % (TILE_N / 4));
      float4 v;
      if (NT8 == 2 && p.S <= 8) {
        // 9-16 drafted rows: every split's piece is requested before the
        // first add (one round trip to L2), then added in split order, as
        // below.  (At 8 rows and fewer the plain loop measured faster on
        // 5120 x 5120; here it saves 4 % of a down call at 16 rows.)
        float4 x[8];
#pragma unroll
        for (int sp = 0; sp < 8; ++sp)
          if (sp < p.S)
            x[sp] = __ldcg(reinterpret_cast<const float4*>(base + ((int64_t)sp * MAX_M + m) * TILE_N + row));
        v = x[0];
#pragma unroll
        for (int sp = 1; sp < 8; ++sp)
          if (sp < p.S) {
            v.x += x[sp].x;
            v.y += x[sp].y;
            v.z += x[sp].z;
            v.w += x[sp].w;
          }
      } else {
        v = __ldcg(reinterpret_cast<const float4*>(base + m * TILE_N + row));
        for (int sp = 1; sp < p.S; ++sp) {
          const float4 x =
              __ldcg(reinterpret_cast<const float4*>(base + ((int64_t)sp * MAX_M + m) * TILE_N + row));
          v.x += x.x;
          v.y += x.y;
          v.z += x.z;
          v.w += x.w;
        }
      }
      const float vals[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int64_t n = (int64_t)tile * TILE_N + row + r;
        if (n < p.N) p.out[(int64_t)m * p.ldo + n] = vals[r];
      }
      if constexpr (GREEDY) *reinterpret_cast<float4*>(fin + m * TILE_N + row) = v;
    }
  }
  // the tile is finished by its last split
  if constexpr (GREEDY) {
    if (s_flag[1]) {
      __syncthreads();
      greedy_tile(p, fin, tile, M, !aborted, tid, s_flag);
    }
  }
  if (tid == 0) QMM_STAMP(p, QMM_TR_EXIT, global_timer_ns());
}

}  // namespace qmm
