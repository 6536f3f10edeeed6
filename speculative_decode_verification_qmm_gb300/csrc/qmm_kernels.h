// qmm_kernels.h -- host launchers of the library's kernels (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "qmm_common.cuh"

namespace qmm {

// Verify kernel configuration chosen by the host for one launch.
struct VerifyLaunch {
  int fmt;        // 0 Q4_0, 1 FP8
  bool f16_ops;   // Q4_0: f16 operands (Hadamard path) instead of bf16
  bool simt;      // CUDA-core baseline (Q4_0 only)
  int ctas;
  cudaStream_t stream;
};

// Pipeline depth (stages in flight per CTA), dynamic shared memory, and the
// kernels' shared-memory attribute (set on the current device).
int q4_pipeline_depth();
int fp8_pipeline_depth();
int q8_pipeline_depth();
size_t q8_smem_bytes();
cudaError_t prepare_q8_attributes();
size_t q4_smem_bytes();
size_t fp8_smem_bytes();
cudaError_t prepare_q4_attributes();
cudaError_t prepare_fp8_attributes();
constexpr int MAX_SPLITS = 16;  // K splits per row tile (tcgen05: = cluster size, 16 is non-portable)

// tcgen05 kernel (Q4_0): its weight layout, repack, dequantization and launch.
// act_map points to a CUtensorMap over the activation rows (3-D view
// [K/8 groups][M rows][8 values], boxes of 32 x 16 x 8).
cudaError_t prepare_tc_attributes();
int tc_max_active_clusters(int S);
int tc_pipeline_depth();
cudaError_t launch_verify_tc(const VerifyParams& vp, const void* act_map, bool f16_ops, int ctas,
                             cudaStream_t st);
cudaError_t launch_repack_tc(const uint8_t* blocks, int64_t N, int64_t K, int n_tiles, int S, int spc,
                             uint8_t* wdev, cudaStream_t st);
cudaError_t launch_dequant_tc(const uint8_t* wdev, int64_t N, int64_t K, int n_tiles, int S, int spc,
                              float* out, cudaStream_t st);

// act_map points to a CUtensorMap over the activation rows (see qmm_common.cuh)
// with boxes of 8 values x R rows x chunk columns / 8, R = 8 for M <= 8, else 16.
cudaError_t launch_verify_q4(const VerifyParams& p, const VerifyLaunch& l, const void* act_map);
cudaError_t launch_verify_fp8(const VerifyParams& p, const VerifyLaunch& l, const void* act_map);
cudaError_t launch_verify_q8(const VerifyParams& p, const VerifyLaunch& l, const void* act_map);

// The activation pre-pass of the f16 operand paths; hb = rotation block size
// (0 none, 32, 64, 128).
cudaError_t launch_act_prep(const PrepParams& p, bool out_f16, int hb, cudaStream_t st);
// Rotation of activation rows in hb-blocks (32, 64, 128) to fp32.
cudaError_t launch_hadamard(const uint16_t* act, int64_t lda, float* out, int M, int64_t K, int hb,
                            int sm_count, cudaStream_t st);
// Offline weight rotation in hb-blocks (32, 64, 128), times 1/hb.
cudaError_t launch_rotate_weights(const float* w, int64_t N, int64_t K, int hb, float* out,
                                  cudaStream_t st);
cudaError_t launch_repack(int fmt, const uint8_t* wsrc, const float* scales, int64_t N, int64_t K,
                          int n_tiles, int S, int spc, uint8_t* wdev, float* f8_scale,
                          cudaStream_t st);
cudaError_t launch_dequant(int fmt, const uint8_t* wdev, const float* f8_scale, int64_t N, int64_t K,
                           int n_tiles, int S, int spc, float* out, cudaStream_t st);
cudaError_t launch_quantize_q4(const float* w, int64_t N, int64_t K, int had, uint8_t* blocks,
                               cudaStream_t st);
cudaError_t launch_quantize_q8(const float* w, int64_t N, int64_t K, uint8_t* blocks, cudaStream_t st);
cudaError_t launch_quantize_fp8(const float* w, int64_t N, int64_t K, int had, uint8_t* codes,
                                float* scales, cudaStream_t st);

// Prefill GEMM (FP8 handles): out[M][N] = act[M][K] * W^T for any M, on the
// verify layout's stage stream.  act_map points to a CUtensorMap over the
// pre-pass's f16 rows (2-D, boxes of 64 columns x prefill_tile_rows() rows,
// 128-byte swizzle).
struct PrefillLaunch {
  const uint8_t* wdev;
  const float* f8_scale;
  const float* row_scale;
  float* out;
  int* status;
  int64_t ldo;
  int M;
  int n_tiles;
  int spt;       // stages per weight tile in the stream (S * spc)
  int kb_count;  // K / 128
  int sm_count;
  uint64_t wait_limit_ns;
};
cudaError_t prepare_prefill_attributes();
int prefill_tile_rows();
// bf16 rows -> f16 rows times 2^e (row_scale[m] = 2^-e), rotated in hb-blocks when hb != 0.
cudaError_t launch_prefill_prep(const uint16_t* act, int64_t lda, uint16_t* out, float* row_scale, int64_t M,
                                int64_t K, int hb, cudaStream_t st);
cudaError_t launch_prefill_fp8(const PrefillLaunch& pl, const void* act_map, cudaStream_t st);

}  // namespace qmm
