// wquant.cu -- absmean weight_quant and the 2-bit pack (offline, once per matrix).
//
// BitLinear weight_quant (BitNet b1.58, named in the Candle BitNet PR's list of
// changes): sw = 1 / max(mean|W|, 1e-5), Wq = clamp(round_half_even(W*sw), -1, 1),
// stored as 2-bit codes Wq+1 (0.25 byte per weight, the figure the pages'
// memory tables use, "Transformer Block" page, section "Memory Layout").
//
// Three kernels on the caller's stream:
//   1. wq_bucket_sums: exact sum of |W| into 256 per-exponent uint64 buckets in
//      the workspace (shared-memory buckets per CTA, warp-aggregated).
//   2. wq_finalize (one warp): fold the buckets, round once to fp64,
//      mean = fp32(S / (N*K)) in fp64, sw = 1 / max(mean, 1e-5) in fp32.
//   3. wq_pack: one thread per 32-bit output word (16 weights).
#include "common.cuh"

namespace bitlinear {
namespace {

constexpr int kReduceThreads = 256;
constexpr int kPackThreads = 256;

__global__ void __launch_bounds__(kReduceThreads)
wq_bucket_sums(const float4* __restrict__ W4, int64_t n4, unsigned long long* __restrict__ gbuckets) {
  __shared__ unsigned long long sb[kBuckets];
  for (int i = threadIdx.x; i < kBuckets; i += blockDim.x) sb[i] = 0ull;
  __syncthreads();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  // Warp-uniform trip count: all lanes take part in the warp aggregation.
  const int64_t warp_base = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31);
  for (int64_t base = warp_base; base < n4; base += stride) {
    const int64_t i = base + (threadIdx.x & 31);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < n4) v = W4[i];
    const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      int b;
      uint32_t m;
      fp32_bucket(f[c], &b, &m);
      warp_bucket_add(sb, b, (unsigned long long)m);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kBuckets; i += blockDim.x) {
    if (sb[i]) atomicAdd(&gbuckets[i], sb[i]);
  }
}

__global__ void __launch_bounds__(32)
wq_finalize(const unsigned long long* __restrict__ gbuckets, double count, float* __restrict__ w_scale,
            float* __restrict__ mean_out) {
  __shared__ unsigned long long sb[kBuckets];
  __shared__ unsigned long long digits[kSumDigits];
  for (int i = threadIdx.x; i < kBuckets; i += 32) sb[i] = gbuckets[i];
  __syncwarp();
  const double S = warp_fold_buckets(sb, 1, -149, digits);
  if (threadIdx.x == 0) {
    const float mean = __double2float_rn(__ddiv_rn(S, count));
    const float sw = __fdiv_rn(1.0f, fmaxf(mean, 1e-5f));
    *w_scale = sw;
    *mean_out = mean;
  }
}

// Thread t writes word w = t % 4 of chunk (kb, n) with n = (t / 4) % N and
// kb = t / (4N): the 16 weights W[n, 64kb + 16w .. 64kb + 16w + 15].
__global__ void __launch_bounds__(kPackThreads)
wq_pack(const float* __restrict__ W, int64_t N, int64_t K, const float* __restrict__ w_scale,
        uint32_t* __restrict__ packed_words) {
  const int64_t KB = K / 64;
  const int64_t total = N * KB * 4;
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= total) return;
  const float sw = *w_scale;
  const int64_t w = t & 3;
  const int64_t n = (t >> 2) % N;
  const int64_t kb = (t >> 2) / N;
  const float4* src = reinterpret_cast<const float4*>(W + n * K + kb * 64 + w * 16);
  uint32_t word = 0;
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    const float4 v = src[q4];
    const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = 4 * q4 + c;  // k % 16
      int q = __float2int_rn(__fmul_rn(f[c], sw));
      q = q < -1 ? -1 : (q > 1 ? 1 : q);
      word |= (uint32_t)(q + 1) << (8 * (i & 3) + 2 * (i >> 2));
    }
  }
  packed_words[t] = word;
}

}  // namespace

cudaError_t launch_weight_quant(const float* W, int64_t N, int64_t K, uint8_t* packed,
                                float* w_scale, unsigned long long* buckets,
                                const DeviceInfo& dev, cudaStream_t stream) {
  // workspace: buckets[256] then a float holding mean|W| (debug read-back)
  cudaError_t err = cudaMemsetAsync(buckets, 0, kBuckets * sizeof(unsigned long long) + 64, stream);
  if (err != cudaSuccess) return err;
  const int64_t n4 = N * K / 4;
  int64_t blocks = (n4 + kReduceThreads - 1) / kReduceThreads;
  const int64_t cap = (int64_t)dev.num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  wq_bucket_sums<<<(unsigned)blocks, kReduceThreads, 0, stream>>>(
      reinterpret_cast<const float4*>(W), n4, buckets);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  wq_finalize<<<1, 32, 0, stream>>>(buckets, (double)(N * K), w_scale,
                                    reinterpret_cast<float*>(buckets + kBuckets));
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int64_t words = N * (K / 64) * 4;
  const int64_t pblocks = (words + kPackThreads - 1) / kPackThreads;
  wq_pack<<<(unsigned)pblocks, kPackThreads, 0, stream>>>(W, N, K, w_scale,
                                                         reinterpret_cast<uint32_t*>(packed));
  return cudaGetLastError();
}

}  // namespace bitlinear
