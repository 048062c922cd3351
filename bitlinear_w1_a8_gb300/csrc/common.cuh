// common.cuh -- device helpers shared by the BitLinear kernels (sm_103a).
//
// Contents:
//  * small PTX wrappers (programmatic dependent launch, streaming loads);
//  * the exact "sum of floats" used for mean|W| and for the RMSNorm sum of
//    squares: every term is an integer mantissa times a power of two, so the
//    kernels add mantissas (or squared mantissas) into one 64-bit bucket per
//    fp32 exponent with integer atomics (exact, order independent), and one
//    warp folds the 254 buckets into a wide integer and rounds it once to
//    fp64, ties to even.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "bitlinear.h"

namespace bitlinear {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kBuckets = 256;       // one per fp32 biased exponent
constexpr int kSumDigits = 24;      // 32-bit digits of the folded sum (768 bits)

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Both are no-ops when the kernel was not
// launched with the programmatic-serialization attribute.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_release_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 16-byte load that bypasses L1 (the packed weights are touched once per call).
__device__ __forceinline__ uint4 ld_stream_u4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// Exact sums.
// A finite fp32 value |v| equals mant * 2^(e - 150) with e its biased exponent
// and mant its 24-bit significand (subnormals: e treated as 1, no hidden bit).
// Bucket e (1..254) of a sum of |v| holds the integer sum of mant; bucket e of a
// sum of v^2 holds the integer sum of mant^2.  Bucket 0 is never used and
// bucket 255 (Inf/NaN) is ignored.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void fp32_bucket(float v, int* bucket, uint32_t* mant) {
  uint32_t u = __float_as_uint(v) & 0x7fffffffu;
  uint32_t e = u >> 23;
  *mant = (u & 0x7fffffu) | (e ? 0x800000u : 0u);
  *bucket = e ? (int)e : 1;
}

// Adds `value` (< 2^48) to smem bucket `b` after summing it over the lanes of
// the warp that target the same bucket.  Every lane of the warp must call it
// (pass value 0 for lanes without data).
__device__ __forceinline__ void warp_bucket_add(unsigned long long* buckets, int b,
                                                unsigned long long value) {
  unsigned peers = __match_any_sync(kFullMask, b);
  uint32_t hi = (uint32_t)(value >> 24);          // < 2^24
  uint32_t lo = (uint32_t)(value & 0xffffffu);    // < 2^24
  uint32_t shi = __reduce_add_sync(peers, hi);     // <= 32 * 2^24 < 2^29
  uint32_t slo = __reduce_add_sync(peers, lo);
  int leader = __ffs(peers) - 1;
  if ((int)(threadIdx.x & 31) == leader && (shi | slo) != 0u) {
    atomicAdd(&buckets[b], ((unsigned long long)shi << 24) + (unsigned long long)slo);
  }
}

// One warp folds value = sum_{e=1}^{254} B[e] * 2^(shift*(e-1) + unit_exp2)
// (shift 1 for sums of |v| with unit 2^-149, shift 2 for sums of v^2 with
// unit 2^-298) and returns it rounded to the nearest double, ties to even.
// `digits` is kSumDigits words of scratch shared memory.  B[e] < 2^64 and the
// eight buckets a lane folds must stay below 2^81 in total (true for both
// uses: |v| buckets < 2^51, square buckets < 2^64 with shift 2).
// All 32 lanes must call; every lane gets the result.
__device__ inline double warp_fold_buckets(const unsigned long long* B, int shift, int unit_exp2,
                                    unsigned long long* digits) {
  const int lane = threadIdx.x & 31;
  for (int i = lane; i < kSumDigits; i += 32) digits[i] = 0ull;
  __syncwarp();
  // Lane l folds exponent offsets f = e - 1 in [8l, 8l + 8) into a local
  // 128-bit integer placed at bit shift*8*l of the total.
  unsigned __int128 local = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    int e = 8 * lane + j + 1;
    if (e <= 254) local += ((unsigned __int128)B[e]) << (shift * j);
  }
  const int off = shift * 8 * lane;
  const int d0 = off >> 5;
  const unsigned __int128 sh = local << (off & 31);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    unsigned long long part = (unsigned long long)(sh >> (32 * i)) & 0xffffffffull;
    if (part) atomicAdd(&digits[d0 + i], part);
  }
  __syncwarp();
  double result = 0.0;
  if (lane == 0) {
    unsigned long long carry = 0;
    int top = -1;
    for (int i = 0; i < kSumDigits; ++i) {
      unsigned long long v = digits[i] + carry;
      digits[i] = v & 0xffffffffull;
      carry = v >> 32;
      if (digits[i]) top = i;
    }
    if (top >= 0) {
      const int P = 32 * top + 31 - __clz((unsigned)digits[top]);  // top bit index
      unsigned long long mant;
      bool round_bit = false, sticky = false;
      if (P <= 52) {
        unsigned long long v = digits[0] | (top >= 1 ? digits[1] << 32 : 0ull);
        mant = v << (52 - P);
      } else {
        // 64-bit window of bits [P-63, P] (bits below 0 read as zero)
        const int lo = P - 63;
        unsigned long long win;
        if (lo >= 0) {
          const int di = lo >> 5, ds = lo & 31;
          unsigned __int128 w = (unsigned __int128)digits[di];
          if (di + 1 < kSumDigits) w |= (unsigned __int128)digits[di + 1] << 32;
          if (di + 2 < kSumDigits) w |= (unsigned __int128)digits[di + 2] << 64;
          win = (unsigned long long)(w >> ds);
          if (ds && (digits[di] & ((1ull << ds) - 1ull))) sticky = true;
          for (int i = 0; i < di && !sticky; ++i) sticky = digits[i] != 0ull;
        } else {
          unsigned long long v = digits[0] | (digits[1] << 32);
          win = v << (-lo);
        }
        mant = win >> 11;
        round_bit = (win >> 10) & 1ull;
        sticky = sticky || (win & 0x3ffull) != 0ull;
      }
      int E = P + unit_exp2;
      if (round_bit && (sticky || (mant & 1ull))) {
        mant += 1ull;
        if (mant == (1ull << 53)) { mant >>= 1; E += 1; }
      }
      unsigned long long bits =
          ((unsigned long long)(E + 1023) << 52) | (mant & ((1ull << 52) - 1ull));
      result = __longlong_as_double((long long)bits);
    }
  }
  return __shfl_sync(kFullMask, result, 0);
}

// ---------------------------------------------------------------------------
// Host-side launchers (one per kernel family), defined in the .cu files.
// ---------------------------------------------------------------------------
struct DeviceInfo {
  int device;
  int num_sms;
  int cc_major, cc_minor;
  size_t smem_optin;
  size_t smem_per_sm;  // shared memory of one SM (all its resident CTAs together)
  int* status;  // device address of the per-device status word
};

cudaError_t launch_weight_quant(const float* W, int64_t N, int64_t K, uint8_t* packed,
                                float* w_scale, unsigned long long* buckets,
                                const DeviceInfo& dev, cudaStream_t stream);

// pdl: launched with programmatic dependent launch (waits for the previous
// kernel on the stream before it reads x or writes xq).
cudaError_t launch_act_quant(const float* x, const float* mul, int64_t M, int64_t K,
                             const float* gamma, double eps, int8_t* xq, float* sx,
                             const DeviceInfo& dev, cudaStream_t stream, bool pdl = false);

cudaError_t launch_prefill(const int8_t* xq, const float* sx, int64_t M, const uint8_t* packed,
                           const float* sw, int64_t N, int64_t K, float* y, int32_t* acc,
                           bool pdl, const DeviceInfo& dev, cudaStream_t stream);

cudaError_t launch_wait_selftest(int64_t limit_ns, const DeviceInfo& dev, cudaStream_t stream);

// One weight matrix of a decode launch (several matrices may share one input).
constexpr int kMaxDecodeMats = 4;
struct DecodeMatrix {
  const uint8_t* packed;
  const float* w_scale;
  int64_t N;
  float* y;
  int32_t* acc;
};

// Tokens a decode CTA takes (a token group: gridDim.y is ceil(M / group)),
// whether its dots run on the warp-level MMA, and over how many CTAs of a
// cluster K is split (1: none).
int decode_token_group(int64_t M, int64_t K, bool* mma, int* ks);

// gated: nmats == 2 with equal N (gate, up); every CTA takes the same rows of
// both and mats[0].y receives (r * r) * u with r = max(gate, 0), mats[1].y u.
cudaError_t launch_decode(const int8_t* xq, const float* sx, int64_t M, const DecodeMatrix* mats, int nmats,
                          int64_t K, bool gated, bool pdl, const DeviceInfo& dev, cudaStream_t stream);

// M = 1 only: every CTA quantises x (with the optional gating / RMSNorm
// prologue) itself; CTA 0 writes xq_out / sx_out when they are not NULL.
cudaError_t launch_decode_fused(const float* x, const float* mul, const float* gamma, double eps, int64_t K,
                                const DecodeMatrix* mats, int nmats, int8_t* xq_out, float* sx_out,
                                bool gated, bool pdl, const DeviceInfo& dev, cudaStream_t stream);

// M = 2 token rows without prologues: every CTA quantises the rows itself
// from registers (decode_rows_fit: K <= 3072); CTA 0 writes xq_out / sx_out
// when they are not NULL.
bool decode_rows_fit(int64_t M, int64_t K);
cudaError_t launch_decode_rows(const float* x, int64_t M, int64_t K, const DecodeMatrix* mats, int nmats,
                               int8_t* xq_out, float* sx_out, bool gated, bool pdl, const DeviceInfo& dev,
                               cudaStream_t stream);

// y0[i] = (r * r) * y1[i] with r = max(y0[i], 0) for i < n (the FFN gating of
// a gate / up pair computed by another kernel); waits for the previous kernel
// on the stream when launched with programmatic dependent launch.
cudaError_t launch_gate(float* y0, const float* y1, int64_t n, bool pdl, const DeviceInfo& dev,
                        cudaStream_t stream);

}  // namespace bitlinear
