// quant_row.cuh -- block-cooperative activation_quant of one token row, shared
// by the act_quant kernel and the fused decode kernel.
//
// activation_quant (BitNet b1.58, named in the Candle BitNet PR's list of
// changes): sx = 127 / max(max_k |h|, 1e-5), xq = clamp(rne(h*sx), -128, 127).
// Prologues, in this order when both are requested:
//   gating   h = (r*r)*u, r = max(g, 0)   ("Transformer Block" page, section
//            "Feed-Forward Network": hidden = ReLU^2(gate) x up)
//   RMSNorm  inv = fp32(1 / sqrt(S/K + eps)) in fp64 with S the exact sum of
//            h^2, then h = (h*inv)*gamma in fp32 (an RMSNorm before every
//            BitLinear, Candle BitNet PR, list of changes; the FFN sub-norm of
//            the "Transformer Block" layer structure).
// Every product and the division are single IEEE fp32 operations (no FMA), so
// the int8 codes do not depend on the launch shape.
#pragma once

#include "common.cuh"

namespace bitlinear {

struct RowQuantScratch {
  unsigned long long buckets[kBuckets];
  unsigned long long digits[kSumDigits];
  unsigned long long wlo[32], whi[32];  // per-warp 128-bit partial sums
  float red[32];
  int ired[32];
  float inv;
};

// Exact sum of squares of the K values in hs (shared memory), rounded once to
// the nearest double (ties to even).  Every thread of the block calls it.
// v^2 = m^2 * 2^(2e - 300) (m the 24-bit significand, e the biased exponent,
// subnormals e = 1).  Fast path: with E the largest exponent of the row,
// every square of exponent e >= E - 32 is added as the integer m^2 << 2(e - E
// + 32) < 2^112 into a 128-bit fixed-point sum (at most 2^15 values: < 2^127),
// which is rounded to double directly.  If any nonzero value lies below that
// window (|v| < max|v| / 2^32), the whole sum is taken again with one integer
// bucket per exponent (warp_bucket_add / warp_fold_buckets, exact for every
// input).  Both give the exact sum rounded once.
static __device__ double block_sq_sum_exact(const float4* hs, int K4, RowQuantScratch& sc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = (int)(blockDim.x >> 5);
  int emax = 0;
  for (int i = threadIdx.x; i < K4; i += blockDim.x) {
    const float4 h = hs[i];
    const uint32_t u[4] = {__float_as_uint(h.x), __float_as_uint(h.y), __float_as_uint(h.z), __float_as_uint(h.w)};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t a = u[c] & 0x7fffffffu;
      const int e = a ? max((int)(a >> 23), 1) : 0;
      emax = max(emax, e);
    }
  }
  emax = __reduce_max_sync(kFullMask, emax);
  if (lane == 0) sc.ired[warp] = emax;
  __syncthreads();
  emax = 0;
  for (int w = 0; w < nwarps; ++w) emax = max(emax, sc.ired[w]);
  if (emax == 0) return 0.0;  // every value is zero (the same on every thread)
  const int eb = max(emax - 32, 1);
  unsigned __int128 acc = 0;
  int slow = 0;
  for (int i = threadIdx.x; i < K4; i += blockDim.x) {
    const float4 h = hs[i];
    const uint32_t u[4] = {__float_as_uint(h.x), __float_as_uint(h.y), __float_as_uint(h.z), __float_as_uint(h.w)};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t a = u[c] & 0x7fffffffu;
      if (!a) continue;
      const int e = max((int)(a >> 23), 1);
      const uint64_t m = (a & 0x7fffffu) | ((a >> 23) ? 0x800000u : 0u);
      if (e < eb) slow = 1;
      else acc += ((unsigned __int128)(m * m)) << (2 * (e - eb));
    }
  }
  uint64_t lo = (uint64_t)acc, hi = (uint64_t)(acc >> 64);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t olo = __shfl_xor_sync(kFullMask, lo, o), ohi = __shfl_xor_sync(kFullMask, hi, o);
    lo += olo;
    hi += ohi + (lo < olo ? 1u : 0u);
  }
  if (lane == 0) {
    sc.wlo[warp] = lo;
    sc.whi[warp] = hi;
  }
  slow = __syncthreads_or(slow);
  if (slow) {
    // exact for every input: one integer bucket per exponent
    for (int i = threadIdx.x; i < kBuckets; i += blockDim.x) sc.buckets[i] = 0ull;
    __syncthreads();
    for (int base = (threadIdx.x & ~31); base < K4; base += blockDim.x) {
      const int i = base + lane;
      const float4 h = i < K4 ? hs[i] : make_float4(0.f, 0.f, 0.f, 0.f);
      const float f[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        int b;
        uint32_t m;
        fp32_bucket(f[c], &b, &m);
        warp_bucket_add(sc.buckets, b, (unsigned long long)m * (unsigned long long)m);
      }
    }
    __syncthreads();
    double S = 0.0;
    if (warp == 0) S = warp_fold_buckets(sc.buckets, 2, -298, sc.digits);
    if (threadIdx.x == 0) sc.digits[0] = (unsigned long long)__double_as_longlong(S);
    __syncthreads();
    const double r = __longlong_as_double((long long)sc.digits[0]);
    __syncthreads();
    return r;
  }
  // every thread folds the per-warp sums (the same result everywhere)
  lo = 0;
  hi = 0;
  for (int w = 0; w < nwarps; ++w) {
    const uint64_t a = sc.wlo[w];
    lo += a;
    hi += sc.whi[w] + (lo < a ? 1u : 0u);
  }
  __syncthreads();  // sc.wlo / whi / ired may be reused after this
  // value = (hi:lo) * 2^(2 eb - 300), rounded to 53 bits, ties to even
  const int P = hi ? 127 - __clzll((long long)hi) : 63 - __clzll((long long)lo);  // top bit (lo != 0 here)
  const unsigned __int128 W = ((unsigned __int128)hi << 64) | lo;
  uint64_t mant;
  int E = P + 2 * eb - 300;
  if (P <= 52) {
    mant = (uint64_t)(W << (52 - P));
  } else {
    const int sh = P - 52;
    mant = (uint64_t)(W >> sh);
    const unsigned __int128 rem = W & ((((unsigned __int128)1) << sh) - 1);
    const unsigned __int128 half = ((unsigned __int128)1) << (sh - 1);
    if (rem > half || (rem == half && (mant & 1ull))) {
      mant += 1ull;
      if (mant == (1ull << 53)) {
        mant >>= 1;
        E += 1;
      }
    }
  }
  return __longlong_as_double((long long)(((uint64_t)(E + 1023) << 52) | (mant & ((1ull << 52) - 1ull))));
}

// h = x, or h = (r*r)*u with r = max(x, 0) when the gating input u is given.
__device__ __forceinline__ float4 gated4(const float4* __restrict__ xr, const float4* __restrict__ ur, int i) {
  const float4 g = xr[i];
  if (!ur) return g;
  const float4 u = ur[i];
  float4 h;
  float r;
  r = fmaxf(g.x, 0.0f); h.x = __fmul_rn(__fmul_rn(r, r), u.x);
  r = fmaxf(g.y, 0.0f); h.y = __fmul_rn(__fmul_rn(r, r), u.y);
  r = fmaxf(g.z, 0.0f); h.z = __fmul_rn(__fmul_rn(r, r), u.z);
  r = fmaxf(g.w, 0.0f); h.w = __fmul_rn(__fmul_rn(r, r), u.w);
  return h;
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, o));
    if (lane == 0) red[0] = v;
  }
  __syncthreads();
  const float r = red[0];
  __syncthreads();
  return r;
}

// Quantises one row of K values (K % 64 == 0).  Every thread of the block
// must call it.  hs: K floats of shared scratch; out: where the K int8 codes
// go (shared or global memory, 4-byte aligned).  Returns sx.
static __device__ __forceinline__ float quantize_row(const float* __restrict__ x, const float* __restrict__ mul,
                                           const float* __restrict__ gamma, double eps, int K, float4* hs,
                                           RowQuantScratch& sc, int8_t* out) {
  const int K4 = K >> 2;
  const float4* xr = reinterpret_cast<const float4*>(x);
  const float4* ur = reinterpret_cast<const float4*>(mul);
  const bool norm = gamma != nullptr;
  float amax = 0.0f;
  if (norm) {
    for (int i = threadIdx.x; i < K4; i += blockDim.x) hs[i] = gated4(xr, ur, i);
    __syncthreads();
    const double S = block_sq_sum_exact(hs, K4, sc);
    if (threadIdx.x == 0) {
      const double ms = __dadd_rn(__ddiv_rn(S, (double)K), eps);
      sc.inv = __double2float_rn(__ddiv_rn(1.0, __dsqrt_rn(ms)));
    }
    __syncthreads();
    const float inv = sc.inv;
    const float4* g4 = reinterpret_cast<const float4*>(gamma);
    for (int i = threadIdx.x; i < K4; i += blockDim.x) {
      float4 h = hs[i];
      const float4 gm = g4[i];
      h.x = __fmul_rn(__fmul_rn(h.x, inv), gm.x);
      h.y = __fmul_rn(__fmul_rn(h.y, inv), gm.y);
      h.z = __fmul_rn(__fmul_rn(h.z, inv), gm.z);
      h.w = __fmul_rn(__fmul_rn(h.w, inv), gm.w);
      hs[i] = h;
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(h.x), fabsf(h.y)), fmaxf(fabsf(h.z), fabsf(h.w))));
    }
  } else {
#pragma unroll 4
    for (int i = threadIdx.x; i < K4; i += blockDim.x) {
      const float4 h = gated4(xr, ur, i);
      hs[i] = h;
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(h.x), fabsf(h.y)), fmaxf(fabsf(h.z), fabsf(h.w))));
    }
  }
  amax = block_max(amax, sc.red);
  const float s = __fdiv_rn(127.0f, fmaxf(amax, 1e-5f));
  int* o = reinterpret_cast<int*>(out);
  for (int i = threadIdx.x; i < K4; i += blockDim.x) {
    const float4 h = hs[i];
    const float f[4] = {h.x, h.y, h.z, h.w};
    uint32_t word = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      int q = __float2int_rn(__fmul_rn(f[c], s));
      q = q < -128 ? -128 : (q > 127 ? 127 : q);
      word |= ((uint32_t)q & 0xffu) << (8 * c);
    }
    o[i] = (int)word;
  }
  return s;
}

// 16-byte global -> shared copy that bypasses the registers; completes at the
// issuing thread's cp.async.wait_all.
__device__ __forceinline__ void cp_async16_row(void* dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst_smem)),
               "l"(src)
               : "memory");
}

// quantize_row in two parts for the fused decode kernel: the row, the gating
// input and gamma are first staged in shared memory with cp.async -- every
// thread issues all of its copies before waiting, so the row costs one memory
// round trip, and the kernel can queue its weight loads behind them -- and the
// arithmetic then runs from shared memory, element by element the same
// operations as quantize_row.  hs, us, gs: K floats of shared memory each (us
// only with mul, gs only with gamma).  *sumx (shared, zero on entry) receives
// sum_k xq[k].  Returns sx.
// Part 1: issue this thread's copies of the row (and mul, gamma) into shared
// memory.  Part 2 (quantize_row_staged) waits for them.
static __device__ __forceinline__ void stage_row(const float* __restrict__ x, const float* __restrict__ mul,
                                                 const float* __restrict__ gamma, int K, float4* hs, float4* us,
                                                 float4* gs) {
  const int K4 = K >> 2;
  const float4* xr = reinterpret_cast<const float4*>(x);
  const float4* ur = reinterpret_cast<const float4*>(mul);
  const float4* gr = reinterpret_cast<const float4*>(gamma);
  // Every CTA of a decode launch stages the same row: each starts at its own
  // 128-byte line (rotated by CTA), so the CTAs' first requests spread over
  // the L2 slices instead of all hitting the row's first lines at once.
  const int rot = (int)((blockIdx.x * 296u) % (unsigned)K4) & ~7;
  for (int j = threadIdx.x; j < K4; j += blockDim.x) {
    int i = j + rot;
    if (i >= K4) i -= K4;
    cp_async16_row(hs + i, xr + i);
    if (ur) cp_async16_row(us + i, ur + i);
    if (gr) cp_async16_row(gs + i, gr + i);
  }
}
static __device__ __forceinline__ float quantize_row_staged(bool gated, bool norm, double eps, int K, float4* hs,
                                                  const float4* us, const float4* gs, RowQuantScratch& sc,
                                                  int8_t* out, int* sumx) {
  const int K4 = K >> 2;
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  const float4* hsc = hs;
  const float4* usc = gated ? us : nullptr;
  float amax = 0.0f;
  if (norm) {
    if (usc) {
      for (int i = threadIdx.x; i < K4; i += blockDim.x) hs[i] = gated4(hsc, usc, i);
      __syncthreads();
    }
    const double S = block_sq_sum_exact(hs, K4, sc);
    if (threadIdx.x == 0) {
      const double ms = __dadd_rn(__ddiv_rn(S, (double)K), eps);
      sc.inv = __double2float_rn(__ddiv_rn(1.0, __dsqrt_rn(ms)));
    }
    __syncthreads();
    const float inv = sc.inv;
    for (int i = threadIdx.x; i < K4; i += blockDim.x) {
      float4 h = hs[i];
      const float4 gm = gs[i];
      h.x = __fmul_rn(__fmul_rn(h.x, inv), gm.x);
      h.y = __fmul_rn(__fmul_rn(h.y, inv), gm.y);
      h.z = __fmul_rn(__fmul_rn(h.z, inv), gm.z);
      h.w = __fmul_rn(__fmul_rn(h.w, inv), gm.w);
      hs[i] = h;
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(h.x), fabsf(h.y)), fmaxf(fabsf(h.z), fabsf(h.w))));
    }
  } else {
    for (int i = threadIdx.x; i < K4; i += blockDim.x) {
      const float4 h = gated4(hsc, usc, i);
      if (usc) hs[i] = h;
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(h.x), fabsf(h.y)), fmaxf(fabsf(h.z), fabsf(h.w))));
    }
  }
  amax = block_max(amax, sc.red);
  const float s = __fdiv_rn(127.0f, fmaxf(amax, 1e-5f));
  int* o = reinterpret_cast<int*>(out);
  int qsum = 0;
  for (int i = threadIdx.x; i < K4; i += blockDim.x) {
    const float4 h = hs[i];
    const float f[4] = {h.x, h.y, h.z, h.w};
    uint32_t word = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      int q = __float2int_rn(__fmul_rn(f[c], s));
      q = q < -128 ? -128 : (q > 127 ? 127 : q);
      qsum += q;
      word |= ((uint32_t)q & 0xffu) << (8 * c);
    }
    o[i] = (int)word;
  }
  qsum = __reduce_add_sync(kFullMask, qsum);
  if ((threadIdx.x & 31) == 0 && qsum != 0) atomicAdd(sumx, qsum);
  return s;
}

}  // namespace bitlinear
