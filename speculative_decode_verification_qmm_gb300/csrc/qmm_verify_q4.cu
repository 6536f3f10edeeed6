// qmm_verify_q4.cu -- Q4_0 instantiations of the verify kernel and their launcher.
#include "qmm_kernels.h"
#include "qmm_verify.cuh"

namespace qmm {

namespace {
constexpr int NS_Q4 = 4;

template <typename Op, int NT8, bool SIMT, bool GREEDY>
cudaError_t launch_one(const VerifyParams& p, const VerifyLaunch& l, const CUtensorMap& amap) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)l.ctas, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = SmemLayout<0, NS_Q4, 8 * NT8>::BYTES;
  cfg.stream = l.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_kernel<0, Op, NT8, SIMT, NS_Q4, GREEDY>, p, amap);
}

template <typename Op, int NT8, bool SIMT, bool GREEDY>
cudaError_t set_attr_one() {
  cudaError_t e = cudaFuncSetAttribute(verify_kernel<0, Op, NT8, SIMT, NS_Q4, GREEDY>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SmemLayout<0, NS_Q4, 8 * NT8>::BYTES);
  return e;
}
template <typename Op, int NT8, bool SIMT>
cudaError_t set_attr() {
  cudaError_t e = set_attr_one<Op, NT8, SIMT, false>();
  return e != cudaSuccess ? e : set_attr_one<Op, NT8, SIMT, true>();
}

template <typename Op, int NT8, bool SIMT>
cudaError_t launch_sel(const VerifyParams& p, const VerifyLaunch& l, const CUtensorMap& amap) {
  return p.best ? launch_one<Op, NT8, SIMT, true>(p, l, amap) : launch_one<Op, NT8, SIMT, false>(p, l, amap);
}
}  // namespace

cudaError_t prepare_q4_attributes() {
  cudaError_t e;
  if ((e = set_attr<Bf16Op, 1, false>()) != cudaSuccess) return e;
  if ((e = set_attr<Bf16Op, 2, false>()) != cudaSuccess) return e;
  if ((e = set_attr<F16Op, 1, false>()) != cudaSuccess) return e;
  if ((e = set_attr<F16Op, 2, false>()) != cudaSuccess) return e;
  if ((e = set_attr<Bf16Op, 1, true>()) != cudaSuccess) return e;
  if ((e = set_attr<Bf16Op, 2, true>()) != cudaSuccess) return e;
  if ((e = set_attr<F16Op, 1, true>()) != cudaSuccess) return e;
  return set_attr<F16Op, 2, true>();
}

size_t q4_smem_bytes() { return SmemLayout<0, NS_Q4, 16>::BYTES; }

int q4_pipeline_depth() { return NS_Q4; }

cudaError_t launch_verify_q4(const VerifyParams& p, const VerifyLaunch& l, const void* act_map) {
  const CUtensorMap& m = *reinterpret_cast<const CUtensorMap*>(act_map);
  const bool nt2 = p.M > 8;
  if (l.simt) {
    if (l.f16_ops) return nt2 ? launch_sel<F16Op, 2, true>(p, l, m) : launch_sel<F16Op, 1, true>(p, l, m);
    return nt2 ? launch_sel<Bf16Op, 2, true>(p, l, m) : launch_sel<Bf16Op, 1, true>(p, l, m);
  }
  if (l.f16_ops) return nt2 ? launch_sel<F16Op, 2, false>(p, l, m) : launch_sel<F16Op, 1, false>(p, l, m);
  return nt2 ? launch_sel<Bf16Op, 2, false>(p, l, m) : launch_sel<Bf16Op, 1, false>(p, l, m);
}

}  // namespace qmm
