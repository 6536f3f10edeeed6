// qmm_aux.cu -- activation pre-pass, Walsh-Hadamard rotation, weight repack,
// exact dequantization hook and the device quantizers (the offline tools that
// write Q4_0 / FP8 weight files, including the rotated "-H32" variant).
#include <cuda_runtime.h>

#include "qmm_common.cuh"
#include "qmm_kernels.h"

namespace qmm {

// ---------------------------------------------------------------------------
// Activation pre-pass.  CTA (s, m) converts row m's K range of split s into the
// stage-ordered 16-bit scratch read by the verify kernel.
//   OUT_F16 = false: bf16 copied unchanged (exact); multiplier 1.
//   OUT_F16 = true : values (rotated in HB-blocks when HB != 0) are multiplied by 2^e with e
//                    chosen so that the largest magnitude of the range lands
//                    in [2^14, 2^15), rounded to f16, and 2^-e is recorded as
//                    the multiplier of this (row, split)'s partial sums.
// Elements past K are written as zeros.
// ---------------------------------------------------------------------------
template <bool OUT_F16, int HB>
__global__ void __launch_bounds__(256) act_prep_kernel(const __grid_constant__ PrepParams p) {
  constexpr bool HAD = HB != 0;
  pdl_trigger();
  const int s = blockIdx.x, m = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t k0 = (int64_t)s * p.spc * p.stage_k;
  const int64_t kr = (int64_t)p.spc * p.stage_k;  // elements of this split
  const uint16_t* src = p.act + (int64_t)m * p.lda;
  // Earlier kernels may still read the scratch this writes.
  pdl_wait();

  auto dst_index = [&](int64_t kl) -> int64_t { return (int64_t)m * p.ld_out + k0 + kl; };

  if constexpr (!OUT_F16) {
    for (int64_t kl = (int64_t)tid * 4; kl < kr; kl += 256 * 4) {
      const int64_t k = k0 + kl;
      uint2 v = make_uint2(0, 0);
      if (k < p.K) v = *reinterpret_cast<const uint2*>(src + k);  // K % 32 == 0: whole group in range
      *reinterpret_cast<uint2*>(p.out + dst_index(kl)) = v;
    }
    if (tid == 0) p.out_scale[m * p.S + s] = 1.0f;
    return;
  } else {
    __shared__ float s_max[8];
    __shared__ float s_mul;
    const int warp = tid >> 5;
    // Splits of up to IT x 1024 elements keep the thread's values in
    // registers: every load is issued before any is used (one memory round
    // trip for the whole split) and the values are rotated once.
    constexpr int IT = 8;
    const int64_t nit = (kr + 1023) / 1024;
    const bool resident = nit <= IT;
    float v[IT][4];
    float amax = 0.f;
    if (resident) {
#pragma unroll
      for (int it = 0; it < IT; ++it) {
        v[it][0] = v[it][1] = v[it][2] = v[it][3] = 0.f;
        const int64_t kl = (int64_t)it * 1024 + warp * 128 + lane * 4;
        if (it < nit && kl < kr && k0 + kl < p.K) load4_bf16(src + k0 + kl, v[it]);
      }
#pragma unroll
      for (int it = 0; it < IT; ++it) {
        if (it < nit) {  // uniform over the block
          if constexpr (HAD) fwht_lanes<HB>(v[it], lane);
#pragma unroll
          for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(v[it][e]));
        }
      }
    } else {
      // pass 1 over a long split: largest magnitude of the (rotated) values
      for (int64_t base = (int64_t)warp * 128; base < kr; base += 256 * 4) {
        const int64_t kl = base + lane * 4;
        const int64_t k = k0 + kl;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (k < p.K) load4_bf16(src + k, x);
        if constexpr (HAD) fwht_lanes<HB>(x, lane);
#pragma unroll
        for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(x[e]));
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, d));
    if (lane == 0) s_max[warp] = amax;
    __syncthreads();
    if (tid == 0) {
      float a = s_max[0];
      for (int w = 1; w < 8; ++w) a = fmaxf(a, s_max[w]);
      int sh = 0;
      if (a > 0.f && isfinite(a)) {
        int E;
        frexpf(a, &E);  // a = f * 2^E, f in [0.5, 1)
        sh = 15 - E;    // a * 2^sh in [2^14, 2^15)
        sh = sh > 100 ? 100 : (sh < -100 ? -100 : sh);
      }
      s_mul = ldexpf(1.0f, sh);
      p.out_scale[m * p.S + s] = ldexpf(1.0f, -sh);
    }
    __syncthreads();
    const float mul = s_mul;
    auto store4 = [&](int64_t kl, const float (&x)[4]) {
      const __half2 h01 = __floats2half2_rn(x[0] * mul, x[1] * mul);
      const __half2 h23 = __floats2half2_rn(x[2] * mul, x[3] * mul);
      uint2 o;
      o.x = *reinterpret_cast<const uint32_t*>(&h01);
      o.y = *reinterpret_cast<const uint32_t*>(&h23);
      *reinterpret_cast<uint2*>(p.out + dst_index(kl)) = o;
    };
    // pass 2: scale (exact power of two), round to f16, store
    if (resident) {
#pragma unroll
      for (int it = 0; it < IT; ++it) {
        const int64_t kl = (int64_t)it * 1024 + warp * 128 + lane * 4;
        if (it < nit && kl < kr) store4(kl, v[it]);
      }
    } else {
      for (int64_t base = (int64_t)warp * 128; base < kr; base += 256 * 4) {
        const int64_t kl = base + lane * 4;
        const int64_t k = k0 + kl;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (k < p.K) load4_bf16(src + k, x);
        if constexpr (HAD) fwht_lanes<HB>(x, lane);
        store4(kl, x);
      }
    }
  }
}

// Standalone rotation: fp32 output [M][K], each warp rotates 128 / HB blocks at a time.
template <int HB>
__global__ void __launch_bounds__(256) hadamard_kernel(const uint16_t* __restrict__ act, int64_t lda,
                                                       float* __restrict__ out, int M, int64_t K) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * 8;
  const int64_t per_row = K / 128 + ((K % 128) ? 1 : 0);  // 128-element groups per row
  for (int64_t wid = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); wid < per_row * M; wid += warps) {
    const int m = (int)(wid / per_row);
    const int64_t k = (wid % per_row) * 128 + lane * 4;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    const bool ok = k < K;  // K % HB == 0: a block's lanes are all in or all out
    if (ok) load4_bf16(act + (int64_t)m * lda + k, v);
    fwht_lanes<HB>(v, lane);
    if (ok) *reinterpret_cast<float4*>(out + (int64_t)m * K + k) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

// ---------------------------------------------------------------------------
// Repack: canonical Q4_0 blocks -> tile-major stage stream (see qmm_common.cuh).
// One thread per (unit, lane).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t q4_code(const uint8_t* blocks, int64_t N, int64_t K, int64_t n,
                                            int64_t k) {
  if (n >= N || k >= K) return 8u;
  const uint8_t* blk = blocks + (n * (K / 32) + k / 32) * 18;
  const int e = (int)(k % 32);
  const uint8_t byte = blk[2 + (e & 15)];
  return (e < 16) ? (byte & 15u) : (byte >> 4);
}

__device__ __forceinline__ uint16_t q4_scale_bits(const uint8_t* blocks, int64_t N, int64_t K,
                                                  int64_t n, int64_t b) {
  if (n >= N || b * 32 >= K) return 0;
  const uint8_t* blk = blocks + (n * (K / 32) + b) * 18;
  return (uint16_t)(blk[0] | (blk[1] << 8));
}

__global__ void repack_q4_kernel(const uint8_t* __restrict__ blocks, int64_t N, int64_t K, int S,
                                 int spc, int64_t total_units, uint8_t* __restrict__ wdev) {
  const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gt >= total_units * 32) return;
  const int lane = (int)(gt & 31);
  int64_t u = gt >> 5;
  const int r = (int)(u % 8); u /= 8;
  const int c = (int)(u % STAGE_CHUNKS); u /= STAGE_CHUNKS;
  const int64_t stage_global = u;  // ((tile * S + split) * spc + i)
  const int i = (int)(u % spc); u /= spc;
  const int split = (int)(u % S);
  const int64_t tile = u / S;
  const int g = lane >> 2, t = lane & 3;
  const int64_t kstage = ((int64_t)split * spc + i) * Q4_STAGE_K + 64 * c;
  uint32_t words[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const int blk = v >> 1, j = v & 1;
    uint32_t w = 0;
#pragma unroll
    for (int pn = 0; pn < 8; ++pn) {
      const int pair = pn & 3, half = pn >> 2;
      const int64_t n = tile * TILE_N + 16 * r + g + 8 * (pair & 1);
      const int64_t k = kstage + 32 * blk + 16 * j + 2 * t + half + 8 * (pair >> 1);
      w |= q4_code(blocks, N, K, n, k) << (4 * pn);
    }
    words[v] = w;
  }
  uint8_t* unit = wdev + stage_global * Q4_STAGE_BYTES + (int64_t)(c * 8 + r) * Q4_UNIT_BYTES;
  *reinterpret_cast<uint4*>(unit + 16 * lane) = make_uint4(words[0], words[1], words[2], words[3]);
  if (t == 0) {
    const int64_t n = tile * TILE_N + 16 * r + g;
    const int64_t b0 = kstage / 32;
    uint2 sc;
    sc.x = (uint32_t)q4_scale_bits(blocks, N, K, n, b0) |
           ((uint32_t)q4_scale_bits(blocks, N, K, n + 8, b0) << 16);
    sc.y = (uint32_t)q4_scale_bits(blocks, N, K, n, b0 + 1) |
           ((uint32_t)q4_scale_bits(blocks, N, K, n + 8, b0 + 1) << 16);
    *reinterpret_cast<uint2*>(unit + 512 + 8 * g) = sc;
  }
}

__global__ void repack_fp8_kernel(const uint8_t* __restrict__ codes, const float* __restrict__ scales,
                                  int64_t N, int64_t K, int S, int spc, int64_t total_units,
                                  uint8_t* __restrict__ wdev, float* __restrict__ f8_scale) {
  const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gt >= total_units * 32) return;
  const int lane = (int)(gt & 31);
  int64_t u = gt >> 5;
  const int r = (int)(u % 8); u /= 8;
  const int c = (int)(u % STAGE_CHUNKS); u /= STAGE_CHUNKS;
  const int64_t stage_global = u;
  const int i = (int)(u % spc); u /= spc;
  const int split = (int)(u % S);
  const int64_t tile = u / S;
  const int g = lane >> 2, t = lane & 3;
  const int64_t kt = (int64_t)split * spc + i;  // 128-column tile index
  const int64_t kbase = kt * F8_STAGE_K + 32 * c;
  uint32_t words[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const int j = v >> 1, h = v & 1;
    uint32_t w = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int a = 2 * h + (e >> 1);
      const int64_t n = tile * TILE_N + 16 * r + g + 8 * (a & 1);
      const int64_t k = kbase + 16 * j + 2 * t + (e & 1) + 8 * (a >> 1);
      const uint32_t code = (n < N && k < K) ? codes[n * K + k] : 0u;
      w |= code << (8 * e);
    }
    words[v] = w;
  }
  uint8_t* stage = wdev + stage_global * F8_STAGE_BYTES;
  uint8_t* unit = stage + (int64_t)(c * 8 + r) * F8_UNIT_BYTES;
  *reinterpret_cast<uint4*>(unit + 16 * lane) = make_uint4(words[0], words[1], words[2], words[3]);
  if (c == 0 && r == 0 && lane == 0) {
    // one stage = one 128x128 tile; its scale, indexed [tile][S * spc]
    const int64_t tk_n = K / 128;
    float s = 0.f;
    if (tile * TILE_N < N && kt * 128 < K) s = scales[tile * tk_n + kt];
    f8_scale[stage_global] = s;
  }
}

// Q8_0 canonical blocks (34 bytes: fp16 d, 32 int8 codes) -> stage units:
// the codes in the FP8 unit's order, stored as q + 128; lanes 0..7 also store
// the (d[g], d[g + 8]) pair of rows g, g + 8 of the unit.  Padding rows and
// columns hold code 0 (stored 128) and scale 0.
__global__ void repack_q8_kernel(const uint8_t* __restrict__ blocks, int64_t N, int64_t K, int S,
                                 int spc, int64_t total_units, uint8_t* __restrict__ wdev) {
  const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gt >= total_units * 32) return;
  const int lane = (int)(gt & 31);
  int64_t u = gt >> 5;
  const int r = (int)(u % 8); u /= 8;
  const int c = (int)(u % STAGE_CHUNKS); u /= STAGE_CHUNKS;
  const int64_t stage_global = u;
  const int i = (int)(u % spc); u /= spc;
  const int split = (int)(u % S);
  const int64_t tile = u / S;
  const int g = lane >> 2, t = lane & 3;
  const int64_t nb = K / 32;
  const int64_t kbase = ((int64_t)split * spc + i) * Q8_STAGE_K + 32 * c;
  uint32_t words[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const int j = v >> 1, h = v & 1;
    uint32_t w = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int a = 2 * h + (e >> 1);
      const int64_t n = tile * TILE_N + 16 * r + g + 8 * (a & 1);
      const int64_t k = kbase + 16 * j + 2 * t + (e & 1) + 8 * (a >> 1);
      const uint32_t code = (n < N && k < K) ? blocks[(n * nb + k / 32) * 34 + 2 + k % 32] : 0u;
      w |= (code ^ 0x80u) << (8 * e);
    }
    words[v] = w;
  }
  uint8_t* unit = wdev + stage_global * Q8_STAGE_BYTES + (int64_t)(c * 8 + r) * Q8_UNIT_BYTES;
  *reinterpret_cast<uint4*>(unit + 16 * lane) = make_uint4(words[0], words[1], words[2], words[3]);
  if (lane < 8) {
    uint32_t pair = 0;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int64_t n = tile * TILE_N + 16 * r + lane + 8 * hh;
      uint32_t d = 0;
      if (n < N && kbase < K) {
        const uint8_t* blk = blocks + (n * nb + kbase / 32) * 34;
        d = (uint32_t)blk[0] | ((uint32_t)blk[1] << 8);
      }
      pair |= d << (16 * hh);
    }
    *reinterpret_cast<uint32_t*>(unit + 512 + 4 * lane) = pair;
  }
}

// ---------------------------------------------------------------------------
// Exact dequantization from the repacked stream (test hook): one thread per
// (unit, lane) decodes its 16 bytes back to (n, k) positions.
// ---------------------------------------------------------------------------
__global__ void dequant_q4_kernel(const uint8_t* __restrict__ wdev, int64_t N, int64_t K, int S, int spc,
                                  int64_t total_units, float* __restrict__ out) {
  const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gt >= total_units * 32) return;
  const int lane = (int)(gt & 31);
  int64_t u = gt >> 5;
  const int r = (int)(u % 8); u /= 8;
  const int c = (int)(u % STAGE_CHUNKS); u /= STAGE_CHUNKS;
  const int64_t stage_global = u;
  const int i = (int)(u % spc); u /= spc;
  const int split = (int)(u % S);
  const int64_t tile = u / S;
  const int g = lane >> 2, t = lane & 3;
  const int64_t kstage = ((int64_t)split * spc + i) * Q4_STAGE_K + 64 * c;
  const uint8_t* unit = wdev + stage_global * Q4_STAGE_BYTES + (int64_t)(c * 8 + r) * Q4_UNIT_BYTES;
  const uint4 cw = *reinterpret_cast<const uint4*>(unit + 16 * lane);
  const uint2 sc = *reinterpret_cast<const uint2*>(unit + 512 + 8 * g);
  const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const int blk = v >> 1, j = v & 1;
    const uint32_t dp = blk ? sc.y : sc.x;
#pragma unroll
    for (int pn = 0; pn < 8; ++pn) {
      const int pair = pn & 3, half = pn >> 2;
      const int64_t n = tile * TILE_N + 16 * r + g + 8 * (pair & 1);
      const int64_t k = kstage + 32 * blk + 16 * j + 2 * t + half + 8 * (pair >> 1);
      if (n < N && k < K) {
        const uint16_t dbits = (uint16_t)((pair & 1) ? (dp >> 16) : (dp & 0xFFFF));
        const int q = (int)((words[v] >> (4 * pn)) & 15u);
        out[n * K + k] = __half2float(__ushort_as_half(dbits)) * (float)(q - 8);
      }
    }
  }
}

__global__ void dequant_q8_kernel(const uint8_t* __restrict__ wdev, int64_t N, int64_t K, int S, int spc,
                                  int64_t total_units, float* __restrict__ out) {
  const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gt >= total_units * 32) return;
  const int lane = (int)(gt & 31);
  int64_t u = gt >> 5;
  const int r = (int)(u % 8); u /= 8;
  const int c = (int)(u % STAGE_CHUNKS); u /= STAGE_CHUNKS;
  const int64_t stage_global = u;
  const int i = (int)(u % spc); u /= spc;
  const int split = (int)(u % S);
  const int64_t tile = u / S;
  const int g = lane >> 2, t = lane & 3;
  const int64_t kbase = ((int64_t)split * spc + i) * Q8_STAGE_K + 32 * c;
  const uint8_t* unit = wdev + stage_global * Q8_STAGE_BYTES + (int64_t)(c * 8 + r) * Q8_UNIT_BYTES;
  const uint4 cw = *reinterpret_cast<const uint4*>(unit + 16 * lane);
  const uint32_t dpair = *reinterpret_cast<const uint32_t*>(unit + 512 + 4 * g);
  const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const int j = v >> 1, h = v & 1;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int a = 2 * h + (e >> 1);
      const int64_t n = tile * TILE_N + 16 * r + g + 8 * (a & 1);
      const int64_t k = kbase + 16 * j + 2 * t + (e & 1) + 8 * (a >> 1);
      if (n < N && k < K) {
        const uint16_t dbits = (uint16_t)((a & 1) ? (dpair >> 16) : (dpair & 0xFFFF));
        const int q = (int)((words[v] >> (8 * e)) & 0xFFu) - 128;
        out[n * K + k] = __half2float(__ushort_as_half(dbits)) * (float)q;
      }
    }
  }
}

__global__ void dequant_fp8_kernel(const uint8_t* __restrict__ wdev, const float* __restrict__ f8_scale,
                                   int64_t N, int64_t K, int S, int spc, int64_t total_units,
                                   float* __restrict__ out) {
  const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gt >= total_units * 32) return;
  const int lane = (int)(gt & 31);
  int64_t u = gt >> 5;
  const int r = (int)(u % 8); u /= 8;
  const int c = (int)(u % STAGE_CHUNKS); u /= STAGE_CHUNKS;
  const int64_t stage_global = u;
  const int i = (int)(u % spc); u /= spc;
  const int split = (int)(u % S);
  const int64_t tile = u / S;
  const int g = lane >> 2, t = lane & 3;
  const int64_t kbase = ((int64_t)split * spc + i) * F8_STAGE_K + 32 * c;
  const uint8_t* stage = wdev + stage_global * F8_STAGE_BYTES;
  const uint8_t* unit = stage + (int64_t)(c * 8 + r) * F8_UNIT_BYTES;
  const float s = f8_scale[stage_global];
  const uint4 cw = *reinterpret_cast<const uint4*>(unit + 16 * lane);
  const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const int j = v >> 1, h = v & 1;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int a = 2 * h + (e >> 1);
      const int64_t n = tile * TILE_N + 16 * r + g + 8 * (a & 1);
      const int64_t k = kbase + 16 * j + 2 * t + (e & 1) + 8 * (a >> 1);
      if (n < N && k < K) {
        const uint32_t code = (words[v] >> (8 * e)) & 0xFFu;
        const uint32_t h2 = e4m3x2_to_f16x2(code);
        const float w = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFF)));
        out[n * K + k] = __fmul_rn(w, s);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Quantizers (offline tools).
// ---------------------------------------------------------------------------
// The offline weight rotation ahead of the plain quantizers (the 64- and
// 128-point variants, and every rotation of Q8_0): every HB-block of a row of w [N][K] fp32 rotated with
// fwht_lanes and multiplied by 1/HB (a power of two, exact) into out.
template <int HB>
__global__ void __launch_bounds__(256) rotate_weights_kernel(const float* __restrict__ w, int64_t N,
                                                             int64_t K, float* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * 8;
  const int64_t per_row = K / 128 + ((K % 128) ? 1 : 0);
  for (int64_t wid = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); wid < per_row * N; wid += warps) {
    const int64_t n = wid / per_row;
    const int64_t k = (wid % per_row) * 128 + lane * 4;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    const bool ok = k < K;  // K % HB == 0: a block's lanes are all in or all out
    if (ok) {
      const float4 f = *reinterpret_cast<const float4*>(w + n * K + k);
      v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    }
    fwht_lanes<HB>(v, lane);
    constexpr float inv = 1.0f / (float)HB;
    if (ok)
      *reinterpret_cast<float4*>(out + n * K + k) =
          make_float4(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv), __fmul_rn(v[2], inv),
                      __fmul_rn(v[3], inv));
  }
}

// Rotate a 32-block held by one thread (same stage order as fwht32_lanes).
__device__ __forceinline__ void fwht32_thread(float (&v)[32]) {
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i & h) continue;
      const float x = v[i], y = v[i + h];
      v[i] = __fadd_rn(x, y);
      v[i + h] = __fsub_rn(x, y);
    }
  }
}

// Round half away from zero, from the definition: t = r + f with r = trunc(t)
// and f = t - r exact (|t| < 2^23); step away from zero when |f| >= 1/2.
__device__ __forceinline__ int round_half_away(float t) {
  const float r = truncf(t);
  const float f = __fsub_rn(t, r);
  int q = (int)r;
  if (fabsf(f) >= 0.5f) q += (t < 0.f) ? -1 : 1;
  return q;
}

__global__ void quantize_q4_kernel(const float* __restrict__ w, int64_t N, int64_t K, int had,
                                   uint8_t* __restrict__ blocks) {
  const int64_t nb = K / 32;
  const int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (id >= N * nb) return;
  const int64_t n = id / nb, b = id % nb;
  float x[32];
  const float4* src = reinterpret_cast<const float4*>(w + n * K + 32 * b);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 f = src[i];
    x[4 * i] = f.x; x[4 * i + 1] = f.y; x[4 * i + 2] = f.z; x[4 * i + 3] = f.w;
  }
  if (had) {
    fwht32_thread(x);
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = __fmul_rn(x[i], 0.03125f);
  }
  float amax = 0.f, amax_s = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float a = fabsf(x[i]);
    if (a > amax) { amax = a; amax_s = x[i]; }
  }
  const float d32 = __fdiv_rn(amax_s, -8.0f);
  const float inv = (d32 != 0.f) ? __fdiv_rn(1.0f, d32) : 0.f;
  uint8_t q[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    int qi = round_half_away(__fmul_rn(x[i], inv)) + 8;
    qi = qi < 0 ? 0 : (qi > 15 ? 15 : qi);
    q[i] = (uint8_t)qi;
  }
  const unsigned short d16 = __half_as_ushort(__float2half_rn(d32));
  // 18-byte blocks start on even addresses: write nine aligned 16-bit words
  // (little endian: fp16 d, then code bytes 2j and 2j+1 of the block).
  unsigned short* dst = reinterpret_cast<unsigned short*>(blocks + id * 18);
  dst[0] = d16;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const unsigned int lo = (unsigned int)q[2 * j] | ((unsigned int)q[2 * j + 16] << 4);
    const unsigned int hi = (unsigned int)q[2 * j + 1] | ((unsigned int)q[2 * j + 17] << 4);
    dst[1 + j] = (unsigned short)(lo | (hi << 8));
  }
}

// Q8_0: one thread per 32-block.  amax = largest |x|, d32 = amax / 127,
// inv = 1 / d32 (0 for an all-zero block), q = clamp(round half away from zero
// of x * inv, -127, 127), stored d = fp16_rne(d32); 34-byte blocks start on
// even addresses, so the block is written as 17 aligned 16-bit words.
__global__ void quantize_q8_kernel(const float* __restrict__ w, int64_t N, int64_t K,
                                   uint8_t* __restrict__ blocks) {
  const int64_t nb = K / 32;
  const int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (id >= N * nb) return;
  const int64_t n = id / nb, b = id % nb;
  float x[32];
  const float4* src = reinterpret_cast<const float4*>(w + n * K + 32 * b);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 f = src[i];
    x[4 * i] = f.x; x[4 * i + 1] = f.y; x[4 * i + 2] = f.z; x[4 * i + 3] = f.w;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const float d32 = __fdiv_rn(amax, 127.0f);
  const float inv = (d32 != 0.f) ? __fdiv_rn(1.0f, d32) : 0.f;
  unsigned short* dst = reinterpret_cast<unsigned short*>(blocks + id * 34);
  dst[0] = __half_as_ushort(__float2half_rn(d32));
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    int q0 = round_half_away(__fmul_rn(x[2 * j], inv));
    int q1 = round_half_away(__fmul_rn(x[2 * j + 1], inv));
    q0 = q0 < -127 ? -127 : (q0 > 127 ? 127 : q0);
    q1 = q1 < -127 ? -127 : (q1 > 127 ? 127 : q1);
    dst[1 + j] = (unsigned short)(((unsigned)q0 & 0xFFu) | (((unsigned)q1 & 0xFFu) << 8));
  }
}

// One CTA per 128x128 tile.  Pass 1: max |value| (after the optional rotation);
// pass 2: codes.  Each thread owns whole 32-blocks (row n, block b).
__global__ void __launch_bounds__(256) quantize_fp8_kernel(const float* __restrict__ w, int64_t N, int64_t K,
                                                           int had, uint8_t* __restrict__ codes,
                                                           float* __restrict__ scales) {
  const int64_t tn = blockIdx.y, tk = blockIdx.x;
  const int tid = threadIdx.x;
  __shared__ float s_red[8];
  __shared__ float s_s;
  auto load_block = [&](int idx, float (&x)[32]) {
    const int64_t n = tn * 128 + idx / 4;
    const int64_t k = tk * 128 + 32 * (idx % 4);
    const float4* src = reinterpret_cast<const float4*>(w + n * K + k);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 f = src[i];
      x[4 * i] = f.x; x[4 * i + 1] = f.y; x[4 * i + 2] = f.z; x[4 * i + 3] = f.w;
    }
    if (had) {
      fwht32_thread(x);
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = __fmul_rn(x[i], 0.03125f);
    }
  };
  float amax = 0.f;
  for (int idx = tid; idx < 512; idx += 256) {
    float x[32];
    load_block(idx, x);
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, d));
  if ((tid & 31) == 0) s_red[tid >> 5] = amax;
  __syncthreads();
  if (tid == 0) {
    float a = s_red[0];
    for (int i = 1; i < 8; ++i) a = fmaxf(a, s_red[i]);
    const float s = __fdiv_rn(a, 448.0f);
    s_s = s;
    scales[tn * (K / 128) + tk] = s;
  }
  __syncthreads();
  const float s = s_s;
  for (int idx = tid; idx < 512; idx += 256) {
    float x[32];
    load_block(idx, x);
    const int64_t n = tn * 128 + idx / 4;
    const int64_t k = tk * 128 + 32 * (idx % 4);
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        uint16_t pr = 0;
        if (s != 0.f) {
          const float lo = __fdiv_rn(x[4 * i + e], s), hi = __fdiv_rn(x[4 * i + e + 1], s);
          asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pr) : "f"(hi), "f"(lo));
        }
        word |= (uint32_t)pr << (8 * e);
      }
      out[i] = word;
    }
    uint4* dst = reinterpret_cast<uint4*>(codes + n * K + k);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
  }
}

// ---------------------------------------------------------------------------
// Host launchers.
// ---------------------------------------------------------------------------
cudaError_t launch_act_prep(const PrepParams& p, bool out_f16, int hb, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.S, (unsigned)p.M, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!out_f16) return cudaLaunchKernelEx(&cfg, act_prep_kernel<false, 0>, p);
  switch (hb) {
    case 32: return cudaLaunchKernelEx(&cfg, act_prep_kernel<true, 32>, p);
    case 64: return cudaLaunchKernelEx(&cfg, act_prep_kernel<true, 64>, p);
    case 128: return cudaLaunchKernelEx(&cfg, act_prep_kernel<true, 128>, p);
    default: return cudaLaunchKernelEx(&cfg, act_prep_kernel<true, 0>, p);
  }
}

cudaError_t launch_hadamard(const uint16_t* act, int64_t lda, float* out, int M, int64_t K, int hb,
                            int sm_count, cudaStream_t st) {
  const int64_t work = (K / 128 + 1) * M;
  int64_t blocks = (work + 7) / 8;
  const int64_t cap = (int64_t)sm_count * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (hb == 128)
    hadamard_kernel<128><<<(unsigned)blocks, 256, 0, st>>>(act, lda, out, M, K);
  else if (hb == 64)
    hadamard_kernel<64><<<(unsigned)blocks, 256, 0, st>>>(act, lda, out, M, K);
  else
    hadamard_kernel<32><<<(unsigned)blocks, 256, 0, st>>>(act, lda, out, M, K);
  return cudaGetLastError();
}

// w rotated in hb-blocks (hb = 32, 64 or 128) and times 1/hb into out (fp32 [N][K]).
cudaError_t launch_rotate_weights(const float* w, int64_t N, int64_t K, int hb, float* out,
                                  cudaStream_t st) {
  const int64_t work = (K / 128 + 1) * N;
  int64_t blocks = (work + 7) / 8;
  if (blocks > 65535ll * 8) blocks = 65535ll * 8;
  if (blocks < 1) blocks = 1;
  if (hb == 128)
    rotate_weights_kernel<128><<<(unsigned)blocks, 256, 0, st>>>(w, N, K, out);
  else if (hb == 64)
    rotate_weights_kernel<64><<<(unsigned)blocks, 256, 0, st>>>(w, N, K, out);
  else
    rotate_weights_kernel<32><<<(unsigned)blocks, 256, 0, st>>>(w, N, K, out);
  return cudaGetLastError();
}

cudaError_t launch_repack(int fmt, const uint8_t* wsrc, const float* scales, int64_t N, int64_t K,
                          int n_tiles, int S, int spc, uint8_t* wdev, float* f8_scale,
                          cudaStream_t st) {
  const int64_t units = (int64_t)n_tiles * S * spc * STAGE_CHUNKS * 8;
  const int64_t threads = units * 32;
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  if (fmt == 0)
    repack_q4_kernel<<<blocks, 256, 0, st>>>(wsrc, N, K, S, spc, units, wdev);
  else if (fmt == 2)
    repack_q8_kernel<<<blocks, 256, 0, st>>>(wsrc, N, K, S, spc, units, wdev);
  else
    repack_fp8_kernel<<<blocks, 256, 0, st>>>(wsrc, scales, N, K, S, spc, units, wdev, f8_scale);
  return cudaGetLastError();
}

cudaError_t launch_dequant(int fmt, const uint8_t* wdev, const float* f8_scale, int64_t N, int64_t K,
                           int n_tiles, int S, int spc, float* out, cudaStream_t st) {
  const int64_t units = (int64_t)n_tiles * S * spc * STAGE_CHUNKS * 8;
  const int64_t threads = units * 32;
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  if (fmt == 0)
    dequant_q4_kernel<<<blocks, 256, 0, st>>>(wdev, N, K, S, spc, units, out);
  else if (fmt == 2)
    dequant_q8_kernel<<<blocks, 256, 0, st>>>(wdev, N, K, S, spc, units, out);
  else
    dequant_fp8_kernel<<<blocks, 256, 0, st>>>(wdev, f8_scale, N, K, S, spc, units, out);
  return cudaGetLastError();
}

cudaError_t launch_quantize_q4(const float* w, int64_t N, int64_t K, int had, uint8_t* blocks,
                               cudaStream_t st) {
  const int64_t n = N * (K / 32);
  if (n == 0) return cudaSuccess;
  quantize_q4_kernel<<<(unsigned)((n + 127) / 128), 128, 0, st>>>(w, N, K, had, blocks);
  return cudaGetLastError();
}

cudaError_t launch_quantize_q8(const float* w, int64_t N, int64_t K, uint8_t* blocks, cudaStream_t st) {
  const int64_t n = N * (K / 32);
  if (n == 0) return cudaSuccess;
  quantize_q8_kernel<<<(unsigned)((n + 127) / 128), 128, 0, st>>>(w, N, K, blocks);
  return cudaGetLastError();
}

cudaError_t launch_quantize_fp8(const float* w, int64_t N, int64_t K, int had, uint8_t* codes,
                                float* scales, cudaStream_t st) {
  dim3 grid((unsigned)(K / 128), (unsigned)(N / 128), 1);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  quantize_fp8_kernel<<<grid, 256, 0, st>>>(w, N, K, had, codes, scales);
  return cudaGetLastError();
}

}  // namespace qmm
