// aquant.cu -- per-token absmax activation_quant with the optional fused
// prologues (ReLU^2 gating and RMSNorm).  One CTA per token row; the row
// routine (quant_row.cuh) states the arithmetic and its sources.
#include "quant_row.cuh"

namespace bitlinear {
namespace {

constexpr int kActThreadsMany = 256;   // many rows: several CTAs per SM
constexpr int kActThreadsFew = 1024;   // few rows: one wide CTA per row for latency

// Dynamic shared memory: the K fp32 values of h for this row.
__global__ void __launch_bounds__(kActThreadsFew, 1)
act_quant_kernel(const float* __restrict__ x, const float* __restrict__ mul, int K,
                 const float* __restrict__ gamma, double eps, int8_t* __restrict__ xq,
                 float* __restrict__ sx) {
  extern __shared__ float4 hs[];
  __shared__ RowQuantScratch sc;
  // Let a dependent forward kernel start streaming its weights now.
  pdl_release_dependents();
  // With programmatic launch, x (and mul) come from the previous kernel, which
  // may also still be reading xq.
  pdl_wait_primary();
  const int64_t row = blockIdx.x;
  const float s = quantize_row(x + row * (int64_t)K, mul ? mul + row * (int64_t)K : nullptr, gamma, eps, K,
                               hs, sc, xq + row * (int64_t)K);
  if (threadIdx.x == 0) sx[row] = s;
}

}  // namespace

cudaError_t launch_act_quant(const float* x, const float* mul, int64_t M, int64_t K,
                             const float* gamma, double eps, int8_t* xq, float* sx,
                             const DeviceInfo& dev, cudaStream_t stream, bool pdl) {
  const size_t smem = (size_t)K * sizeof(float);
  static thread_local int configured_device = -1;
  static thread_local size_t configured_smem = 0;
  if (configured_device != dev.device || configured_smem < smem) {
    cudaError_t err = cudaFuncSetAttribute(act_quant_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)(dev.smem_optin - 4096));
    if (err != cudaSuccess) return err;
    configured_device = dev.device;
    configured_smem = dev.smem_optin - 4096;
  }
  const int threads = M < dev.num_sms ? kActThreadsFew : kActThreadsMany;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)M, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, act_quant_kernel, x, mul, (int)K, gamma, eps, xq, sx);
}

}  // namespace bitlinear
