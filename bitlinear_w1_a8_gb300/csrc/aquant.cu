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

// The FFN gating of a gate / up pair: y0 = (r * r) * y1 with r = max(y0, 0),
// the fp32 steps of the gating prologue.
constexpr int kGateThreads = 256;
__global__ void __launch_bounds__(kGateThreads) gate_kernel(float* __restrict__ y0, const float* __restrict__ y1,
                                                            int64_t n) {
  pdl_release_dependents();
  pdl_wait_primary();  // y0 and y1 come from the kernel before
  const int64_t n4 = n >> 2;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  float4* g4 = reinterpret_cast<float4*>(y0);
  const float4* u4 = reinterpret_cast<const float4*>(y1);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 g = g4[i];
    const float4 u = u4[i];
    float r;
    r = fmaxf(g.x, 0.0f); g.x = __fmul_rn(__fmul_rn(r, r), u.x);
    r = fmaxf(g.y, 0.0f); g.y = __fmul_rn(__fmul_rn(r, r), u.y);
    r = fmaxf(g.z, 0.0f); g.z = __fmul_rn(__fmul_rn(r, r), u.z);
    r = fmaxf(g.w, 0.0f); g.w = __fmul_rn(__fmul_rn(r, r), u.w);
    g4[i] = g;
  }
  for (int64_t i = (n4 << 2) + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float r = fmaxf(y0[i], 0.0f);
    y0[i] = __fmul_rn(__fmul_rn(r, r), y1[i]);
  }
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

cudaError_t launch_gate(float* y0, const float* y1, int64_t n, bool pdl, const DeviceInfo& dev,
                        cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int64_t want = ((n >> 2) + kGateThreads - 1) / kGateThreads;
  const int64_t cap = (int64_t)dev.num_sms * 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(want < 1 ? 1 : (want < cap ? want : cap)), 1, 1);
  cfg.blockDim = dim3(kGateThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gate_kernel, y0, y1, n);
}

}  // namespace bitlinear
