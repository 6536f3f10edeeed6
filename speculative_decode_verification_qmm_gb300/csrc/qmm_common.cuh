// qmm_common.cuh -- layouts, launch parameters and inline-PTX helpers shared by
// the verify kernels, the activation pre-pass and the tool kernels.
//
// Device layout of a repacked weight matrix ("tile-major stage stream").
//   The N rows are cut into row tiles of TILE_N = 128 rows (zero-padded at the
//   end) and the K axis into pipeline stages of STAGE_K elements (zero-padded).
//   The stages of row tile `tile` are split into `S` contiguous K ranges (the
//   K splits); CTA (tile, s) streams stages [s*spc, (s+1)*spc) where spc is the
//   number of stages per CTA.  Every stage of every CTA is one contiguous byte
//   range, so one bulk copy moves it into shared memory:
//       wdev + ((tile * S + s) * spc + i) * stage_bytes
//   Inside a stage the bytes are ordered [chunk c][row subtile r][unit]: the
//   four column chunks are contiguous and each is moved by its own bulk copy.
//   A unit is what one warp needs for 16 rows x (STAGE_K / 4) columns,
//   already permuted into mma.sync m16n8k16 A-fragment order: lane l (group
//   g = l / 4, thread t = l % 4) finds its 16 bytes at unit + 16 l.
//
//   Q4_0 (STAGE_K = 256, chunk = 64 columns = two 32-blocks):
//     unit = 512 B codes + 64 B scales = 576 B.  Lane word v (0..3) covers
//     block b = v / 2 and k16 step j = v % 2; its nibble p (0..7), with
//     pair = p & 3 and half = p >> 2, is the element
//       row = g + 8 * (pair & 1),   k = 32 b + 16 j + 2 t + half + 8 * (pair >> 1)
//     (pairs 0..3 are the A registers a0..a3).  Nibble pair (p, p + 4) sits in the
//     low nibbles of the two 16-bit lanes after a right shift by 4 p, which is
//     exactly the (low, high) element order of one bf16x2 / f16x2 A register.
//     Scales: for g = 0..7, 8 bytes = fp16 d[g][b0], d[g+8][b0], d[g][b1], d[g+8][b1].
//   FP8 (STAGE_K = 128, chunk = 32 columns):
//     unit = 512 B codes; lane word v covers k16 step j = v / 2, half h = v % 2;
//     byte e (0..3) is element row = g + 8 * ((2h + e/2) & 1),
//     k = 16 j + 2 t + (e & 1) + 8 * ((2h + e/2) >> 1).  A stage is exactly one
//     128x128 weight tile; its fp32 scale lives in a separate array
//     [tile][stage] next to the stream.
//
// Activations reach shared memory through a 2-D tensor map over the 16-bit
// rows (dim 0: K, dim 1: the M rows).  One box per chunk, CHUNK_K columns x
// R = 8 or 16 rows, lands as R rows of 2 x CHUNK_K bytes with the map's
// swizzle of that width, which spreads the eight 16-byte rows of every
// ldmatrix 8x8 matrix over distinct banks; rows >= M and columns >= K read
// as zeros.  The f16 paths read the pre-pass's scratch [MAX_M][Kp] the same
// way.  (The tcgen05 kernel uses a 3-D view instead; see its source.)
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "qmm.h"

namespace qmm {

constexpr int TILE_N = 128;           // rows of W per CTA tile
constexpr int STAGE_CHUNKS = 4;       // column chunks per stage in the layout
constexpr int COMPUTE_WARPS = 8;      // warps that compute: chunk x half of the tile's rows
// No separate producer warp: the compute warps also issue the copies, so two
// CTAs (16 warps) keep exactly four warps per SM sub-partition.
constexpr int THREADS = COMPUTE_WARPS * 32;
constexpr int MAX_M = 16;

// Q4_0
constexpr int Q4_STAGE_K = 256;
constexpr int Q4_UNIT_BYTES = 576;
constexpr int Q4_CHUNK_BYTES = 8 * Q4_UNIT_BYTES;                 // 4608
constexpr int Q4_STAGE_BYTES = STAGE_CHUNKS * Q4_CHUNK_BYTES;      // 18432
// FP8
constexpr int F8_STAGE_K = 128;
constexpr int F8_UNIT_BYTES = 512;
constexpr int F8_CHUNK_BYTES = 8 * F8_UNIT_BYTES;                  // 4096
constexpr int F8_STAGE_BYTES = STAGE_CHUNKS * F8_CHUNK_BYTES;      // 16384
// Q8_0: a unit is 16 rows x 32 columns (one block per row): 512 code bytes in
// the FP8 unit's order, stored as q + 128, then 8 x (d[g], d[g + 8]) fp16 pairs
constexpr int Q8_STAGE_K = 128;
constexpr int Q8_UNIT_BYTES = 544;
constexpr int Q8_CHUNK_BYTES = 8 * Q8_UNIT_BYTES;                  // 4352
constexpr int Q8_STAGE_BYTES = STAGE_CHUNKS * Q8_CHUNK_BYTES;      // 17408

// Device error word bits (OR-ed into the handle's status word).
constexpr int DEV_ERR_TIMEOUT_FULL = 1;   // consumer gave up waiting for a stage
constexpr int DEV_ERR_TIMEOUT_EMPTY = 2;  // producer gave up waiting for a free slot
constexpr int DEV_ERR_TIMEOUT_DRAIN = 4;  // copies in flight did not land in time
constexpr int DEV_ERR_SMEM_ALIGN = 8;     // dynamic shared memory not 1024-byte aligned

struct VerifyParams {
  const uint8_t* wdev;       // repacked weights
  const float* f8_scale;     // FP8: [n_tiles][S * spc] fp32 scale of each stage's tile
  int64_t K;                 // true K
  const float* out_scale;    // [MAX_M][S]: multiplier of split s's partial for row m, or NULL
  float* out;                // [M][ldo]
  int* status;               // device error word
  int64_t ldo;
  int64_t N;
  int M;
  int S;                     // K splits per row tile (tcgen05 kernel: CTAs per cluster)
  int spc;                   // stages per CTA
  float* ws;                 // mma.sync kernels, S > 1: [n_tiles][S][MAX_M][TILE_N] partials
  int* counters;             // mma.sync kernels, S > 1: [n_tiles] arrivals, zero between calls
  uint64_t wait_limit_ns;    // bounded waits give up after this (0: at once)
  // Greedy acceptance (mma.sync kernels; best == NULL: plain verify).
  unsigned long long* best;  // [MAX_M] largest (score key << 32 | ~row) so far, zero between calls
  int* tiles_done;           // row tiles of the call finished, zero between calls
  const int32_t* tokens;     // [M] the block's input tokens (tokens[0]: last committed)
  int32_t* argmax_out;       // [M] first row of the largest score of each drafted row
  int32_t* accept_out;       // [2] accepted drafts k, then argmax_out[k]
  int n_tiles;               // row tiles of the call
  // Builds with QMM_TRACE: per-CTA timeline of this call, [CTA][QMM_TRACE_FIELDS]
  // global-timer stamps (NULL: none).  The product build compiles the stamps out.
  unsigned long long* trace;
};

struct PrepParams {
  const uint16_t* act;       // caller's bf16 rows
  int64_t lda;
  uint16_t* out;             // activation scratch [MAX_M][ld_out], 16-bit values
  int64_t ld_out;            // = S * spc * stage_k
  float* out_scale;          // [MAX_M][S]
  int64_t K;                 // true K
  int M;
  int S;
  int spc;
  int stage_k;
};

// Per-CTA timeline stamp (builds with QMM_TRACE only; the field indices are
// QMM_TR_* of qmm.h).
#ifdef QMM_TRACE
#define QMM_STAMP(p, field, value)                                                   \
  do {                                                                               \
    if ((p).trace) (p).trace[(size_t)blockIdx.x * QMM_TRACE_FIELDS + (field)] = (value); \
  } while (0)
#else
#define QMM_STAMP(p, field, value) \
  do {                             \
  } while (0)
#endif

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint32_t sm_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of parity `parity` of barrier `bar`; give up after about
// `limit_ns` nanoseconds (limit 0: give up at once).  Returns true on success.
// The deadline is kept in SM clock cycles (clock64 is cheap to read, unlike the
// global timer) at 2 cycles per nanosecond, so at clocks below 2 GHz the wait
// lasts proportionally longer before it gives up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (limit_ns == 0) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  const long long limit = (long long)(limit_ns < (1ull << 40) ? limit_ns : (1ull << 40)) * 2;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > limit) return false;
  }
}

// One-dimensional bulk copy global -> shared, completing on `bar`'s tx count.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Same with an L2 eviction-priority hint (weights stream once: evict first).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Tiled tensor copies global -> shared of one box of a 2-D or 3-D tensor map
// (coordinates innermost first).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4}], [%5];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Thread-block clusters: barrier over every thread of every CTA of the
// cluster (release/acquire), and loads from another CTA's shared memory.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t dsmem_map(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t cluster_addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
  return v;
}

// Programmatic dependent launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// Operand-type traits: mma.sync m16n8k16 with fp32 accumulation, and the
// exact conversion of a 4-bit code pair (two nibbles in the low nibbles of the
// two 16-bit lanes) to (q - 8) in that type.
struct Bf16Op {
  __device__ __forceinline__ static void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1,
                                             const float (&c)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
  }
  // 4 pairs of q - 8 from one 32-bit word of 8 nibbles, pair p from nibbles
  // (p, p + 4): bf16 128.0 = 0x4300 has a 7-bit mantissa whose low 4 bits
  // take q exactly (one lop3), and subtracting 136 = 0x4308 leaves q - 8.
  __device__ __forceinline__ static void dequant_word(uint32_t w, uint32_t (&r)[4]) {
    const uint32_t magic = 0x43004300u, bias = 0x43084308u;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      uint32_t x;
      asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(x) : "r"(w >> (4 * p)), "r"(0x000F000Fu), "r"(magic));
      asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r[p]) : "r"(x), "r"(bias));
    }
  }
};

struct F16Op {
  __device__ __forceinline__ static void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1,
                                             const float (&c)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
  }
  // f16 1024.0 = 0x6400 has a 10-bit mantissa: nibbles at bit offsets 0 and 4
  // of each lane are taken in place (1024 + q and 1024 + 16 q), the other two
  // after one shift by 8.  (1024 + q) - 1032 and (1024 + 16 q) / 16 - 72 are
  // both q - 8, exactly.
  __device__ __forceinline__ static void dequant_word(uint32_t w, uint32_t (&r)[4]) {
    const uint32_t magic = 0x64006400u;
    const uint32_t bias_lo = 0x64086408u;   // 1032
    const uint32_t sixteenth = 0x2C002C00u; // 1/16
    const uint32_t bias_hi = 0xD480D480u;   // -72
    const uint32_t w8 = w >> 8;
    uint32_t x0, x1, x2, x3;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(x0) : "r"(w), "r"(0x000F000Fu), "r"(magic));
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(x1) : "r"(w), "r"(0x00F000F0u), "r"(magic));
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(x2) : "r"(w8), "r"(0x000F000Fu), "r"(magic));
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(x3) : "r"(w8), "r"(0x00F000F0u), "r"(magic));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r[0]) : "r"(x0), "r"(bias_lo));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r[1]) : "r"(x1), "r"(sixteenth), "r"(bias_hi));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r[2]) : "r"(x2), "r"(bias_lo));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r[3]) : "r"(x3), "r"(sixteenth), "r"(bias_hi));
  }
};

// e4m3 pair (16 bits, first value in the low byte) -> f16x2 (first value in
// the low half), exact: every E4M3 value is an f16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v16) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(r)
      : "r"(v16));
  return r;
}

// acc[0..1] += d * p[0..1] as one packed fp32x2 FMA (two IEEE fma.rn).
__device__ __forceinline__ void ffma2(float& a0, float& a1, float d, float p0, float p1) {
  float2 r = __ffma2_rn(make_float2(d, d), make_float2(p0, p1), make_float2(a0, a1));
  a0 = r.x;
  a1 = r.y;
}

// ---------------------------------------------------------------------------
// B-point Walsh-Hadamard rotation (B = 32, 64 or 128) across B/4 lanes holding
// 4 consecutive values each: strides 1 and 2 inside the lane, then strides
// 4, 8, ..., B/2 with lane shuffles (partner lane = lane ^ 1, ^ 2, ..., ^ B/8).
// Every stage maps the pair (x at the lower index, y at the upper) to
// (x + y, x - y) in fp32, the stage order and arithmetic of the unnormalised
// transform ["Qwen3.8-27B at 45.7 tok/s: DFlash2 in 1bit serve, and 4-bit
// activations with a Hadamard rotation", section "Prompt processing: 4-bit
// activations, rotated first": two in-register butterfly steps and three lane
// shuffles for B = 32; the larger rotations that the page names as the next
// step keep the stride-ascending order].  All 32 lanes of the warp must call
// it (a warp holds 128 values: 128 / B blocks).
// ---------------------------------------------------------------------------
template <int B>
__device__ __forceinline__ void fwht_lanes(float (&v)[4], int lane) {
  static_assert(B == 32 || B == 64 || B == 128, "rotation size");
  float x, y;
  // stride 1: (0,1), (2,3)
  x = v[0]; y = v[1]; v[0] = __fadd_rn(x, y); v[1] = __fsub_rn(x, y);
  x = v[2]; y = v[3]; v[2] = __fadd_rn(x, y); v[3] = __fsub_rn(x, y);
  // stride 2: (0,2), (1,3)
  x = v[0]; y = v[2]; v[0] = __fadd_rn(x, y); v[2] = __fsub_rn(x, y);
  x = v[1]; y = v[3]; v[1] = __fadd_rn(x, y); v[3] = __fsub_rn(x, y);
  // strides 4 .. B/2 across lanes
#pragma unroll
  for (int d = 1; d < B / 4; d <<= 1) {
    const bool upper = (lane & d) != 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float other = __shfl_xor_sync(0xFFFFFFFFu, v[e], d);
      v[e] = upper ? __fsub_rn(other, v[e]) : __fadd_rn(v[e], other);
    }
  }
}

__device__ __forceinline__ void load4_bf16(const uint16_t* p, float (&v)[4]) {
  const uint2 raw = *reinterpret_cast<const uint2*>(p);
  v[0] = __uint_as_float((raw.x & 0xFFFFu) << 16);
  v[1] = __uint_as_float(raw.x & 0xFFFF0000u);
  v[2] = __uint_as_float((raw.y & 0xFFFFu) << 16);
  v[3] = __uint_as_float(raw.y & 0xFFFF0000u);
}

}  // namespace qmm
