// qmm_verify_fp8.cu -- FP8 E4M3 instantiations of the verify kernel and their launcher.
#include "qmm_kernels.h"
#include "qmm_verify.cuh"

namespace qmm {

namespace {
constexpr int NS_F8 = 5;

template <int NT8, bool GREEDY>
cudaError_t launch_one(const VerifyParams& p, const VerifyLaunch& l, const CUtensorMap& amap) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)l.ctas, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = SmemLayout<1, NS_F8, 8 * NT8>::BYTES;
  cfg.stream = l.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_kernel<1, F16Op, NT8, false, NS_F8, GREEDY>, p, amap);
}

template <int NT8, bool GREEDY>
cudaError_t set_attr_one() {
  return cudaFuncSetAttribute(verify_kernel<1, F16Op, NT8, false, NS_F8, GREEDY>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              SmemLayout<1, NS_F8, 8 * NT8>::BYTES);
}

template <int NT8>
cudaError_t set_attr() {
  cudaError_t e = set_attr_one<NT8, false>();
  return e != cudaSuccess ? e : set_attr_one<NT8, true>();
}

template <int NT8>
cudaError_t launch_sel(const VerifyParams& p, const VerifyLaunch& l, const CUtensorMap& amap) {
  return p.best ? launch_one<NT8, true>(p, l, amap) : launch_one<NT8, false>(p, l, amap);
}
}  // namespace

cudaError_t prepare_fp8_attributes() {
  cudaError_t e = set_attr<1>();
  if (e != cudaSuccess) return e;
  return set_attr<2>();
}

size_t fp8_smem_bytes() { return SmemLayout<1, NS_F8, 16>::BYTES; }

int fp8_pipeline_depth() { return NS_F8; }

cudaError_t launch_verify_fp8(const VerifyParams& p, const VerifyLaunch& l, const void* act_map) {
  const CUtensorMap& m = *reinterpret_cast<const CUtensorMap*>(act_map);
  return p.M > 8 ? launch_sel<2>(p, l, m) : launch_sel<1>(p, l, m);
}

}  // namespace qmm
