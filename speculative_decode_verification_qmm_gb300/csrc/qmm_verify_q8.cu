// qmm_verify_q8.cu -- Q8_0 instantiations of the verify kernel and their launcher
// (f16 operands: the activations always go through the pre-pass).
#include "qmm_kernels.h"
#include "qmm_verify.cuh"

namespace qmm {

namespace {
constexpr int NS_Q8 = 5;

template <int NT8, bool GREEDY>
cudaError_t launch_one(const VerifyParams& p, const VerifyLaunch& l, const CUtensorMap& amap) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)l.ctas, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = SmemLayout<2, NS_Q8, 8 * NT8>::BYTES;
  cfg.stream = l.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_kernel<2, F16Op, NT8, false, NS_Q8, GREEDY>, p, amap);
}

template <int NT8, bool GREEDY>
cudaError_t set_attr_one() {
  return cudaFuncSetAttribute(verify_kernel<2, F16Op, NT8, false, NS_Q8, GREEDY>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              SmemLayout<2, NS_Q8, 8 * NT8>::BYTES);
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

cudaError_t prepare_q8_attributes() {
  cudaError_t e = set_attr<1>();
  if (e != cudaSuccess) return e;
  return set_attr<2>();
}

size_t q8_smem_bytes() { return SmemLayout<2, NS_Q8, 16>::BYTES; }

int q8_pipeline_depth() { return NS_Q8; }

cudaError_t launch_verify_q8(const VerifyParams& p, const VerifyLaunch& l, const void* act_map) {
  const CUtensorMap& m = *reinterpret_cast<const CUtensorMap*>(act_map);
  return p.M > 8 ? launch_sel<2>(p, l, m) : launch_sel<1>(p, l, m);
}

}  // namespace qmm
