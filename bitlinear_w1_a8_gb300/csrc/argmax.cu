// argmax.cu -- greedy token choice on the GPU after the LM head.
//
// index[m] = the smallest n with y[m, n] = max_n y[m, n]  (the LM head is a
// BitLinear too, "Hesper.Models.BitNet" page, section "Performance (BitNet-3B
// on A100)": LM head 13 ms of the 883 ms per token; greedy decoding takes the
// argmax of its logits, so only 4 bytes per token go back to the host).
//
// One CTA per token row: every thread scans a strided share of the row with
// 16-byte loads, keeping (value, index) with ties to the smaller index; the
// pairs meet through warp shuffles and shared memory under the same rule, so
// the answer does not depend on the launch shape.
#include "common.cuh"

namespace bitlinear {
namespace {

constexpr int kArgThreads = 512;

// (v, i) beats (bv, bi) when larger, or equal and earlier.
__device__ __forceinline__ void better(float v, int64_t i, float& bv, int64_t& bi) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

__global__ void __launch_bounds__(kArgThreads) argmax_kernel(const float* __restrict__ y, int64_t N,
                                                             int32_t* __restrict__ out) {
  pdl_release_dependents();
  __shared__ float sv[kArgThreads / 32];
  __shared__ int64_t si[kArgThreads / 32];
  const float* row = y + (int64_t)blockIdx.x * N;
  float bv = -INFINITY;
  int64_t bi = N;  // loses to every real element
  const int t = threadIdx.x;
  if ((N & 3) == 0 && ((reinterpret_cast<uintptr_t>(row) & 15u) == 0)) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const int64_t n4 = N >> 2;
    for (int64_t i = t; i < n4; i += kArgThreads) {
      const float4 v = r4[i];
      better(v.x, 4 * i, bv, bi);
      better(v.y, 4 * i + 1, bv, bi);
      better(v.z, 4 * i + 2, bv, bi);
      better(v.w, 4 * i + 3, bv, bi);
    }
  } else {
    for (int64_t i = t; i < N; i += kArgThreads) better(row[i], i, bv, bi);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(kFullMask, bv, o);
    const int64_t oi = __shfl_xor_sync(kFullMask, bi, o);
    better(ov, oi, bv, bi);
  }
  const int warp = t >> 5, lane = t & 31;
  if (lane == 0) {
    sv[warp] = bv;
    si[warp] = bi;
  }
  __syncthreads();
  if (warp == 0) {
    bv = lane < kArgThreads / 32 ? sv[lane] : -INFINITY;
    bi = lane < kArgThreads / 32 ? si[lane] : N;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(kFullMask, bv, o);
      const int64_t oi = __shfl_xor_sync(kFullMask, bi, o);
      better(ov, oi, bv, bi);
    }
    // A row of -inf (or NaN) only: index 0, like the host reference.
    if (lane == 0) out[blockIdx.x] = (int32_t)(bi < N ? bi : 0);
  }
}

}  // namespace

cudaError_t launch_argmax(const float* y, int64_t M, int64_t N, int32_t* out, cudaStream_t stream) {
  for (int64_t m0 = 0; m0 < M; m0 += 65535) {
    const int64_t rows = M - m0 < 65535 ? M - m0 : 65535;
    argmax_kernel<<<(unsigned)rows, kArgThreads, 0, stream>>>(y + m0 * N, N, out + m0);
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace bitlinear
