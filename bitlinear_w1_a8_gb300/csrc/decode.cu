// decode.cu -- BitLinear contraction for few tokens (decode, M small).
//
// y[m, n] = (sum_k xq[m, k] * Wq[n, k]) / (sx[m] * sw)      (BitNet b1.58 BitLinear;
// the per-token BitLinear calls of the decode loop, "Hesper.Models.BitNet"
// page, section "Performance (BitNet-3B on A100)": 870 of 883 ms per token go
// to the 32 layers, i.e. to streaming the 2-bit weights once per token).
//
// At M = 1 the kernel is bound by HBM: every packed byte is read exactly once
// and does 4 weights of work.  Design:
//  * grid: G CTAs (a multiple of the SM count) times ceil(M / MT) token
//    groups; CTA c of a matrix owns rows [c*N/G, (c+1)*N/G), so every SM
//    streams the same number of bytes; several matrices that share one input
//    (q, k, v or gate, up) share one grid;
//  * thread t takes row r = t % R and k-blocks j, j+J, ... (j = t / R,
//    J = 512 / R): consecutive threads read consecutive 16-byte chunks of one
//    k-block plane (coalesced); G is chosen so that every thread holds at most
//    kChunks chunks, and all of them are requested before
//    griddepcontrol.wait -- the packed weights never come from the previous
//    kernel, so under programmatic dependent launch they stream while the
//    previous kernel finishes.  512-thread CTAs of at most 64 registers fit two
//    per SM, so consecutive kernels overlap;
//  * after the wait, the token group's int8 activations are staged in shared
//    memory (or, in the fused mode, quantised there from fp32 by every CTA);
//  * a chunk holds 64 codes c = Wq+1; with w one 32-bit word,
//    w & (0x03030303 << 2s) holds the codes of k = 16w'+4s .. +3 scaled by
//    4^s, so one mask and one dp4a (unsigned x signed) add 4^s * sum c*x; the
//    four partial sums are combined with exact shifts, and subtracting the
//    row sum of x gives sum Wq*x (the ternary add/sub) exactly;
//  * partial sums of a row meet in shared memory (int32 atomics, exact in
//    any order), then one thread per row rescales.
#include "quant_row.cuh"

namespace bitlinear {
namespace {

constexpr int kDecThreads = 512;
constexpr unsigned long long kWaitNs = 2000000000ull;

struct DecodeMat {
  const uint8_t* packed;
  const float* sw;
  float* y;
  int32_t* acc;
  int N;
  int G;   // CTAs of this matrix
  int g0;  // first CTA of this matrix
};

struct DecodeParams {
  // int8 input (fused == 0): xq_in, sx_in.  fp32 input (fused == 1, M == 1):
  // x, mul, gamma, eps; every CTA quantises the row itself and CTA 0 writes
  // xq_out, sx_out when they are given.
  const int8_t* xq_in;
  const float* sx_in;
  const float* x;
  const float* mul;
  const float* gamma;
  double eps;
  int8_t* xq_out;
  float* sx_out;
  int fused;
  int* status;
  int M, K, KB;
  int rows_max;  // max rows of a CTA over all matrices: sizes the shared-memory carve-up
  int nmats;
  DecodeMat mats[kMaxDecodeMats];
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void bar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ bool bar_try(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for phase 0 of a single-use barrier.
__device__ __noinline__ bool bar_wait(unsigned long long* bar, int* status,
                                      unsigned long long limit_ns = kWaitNs) {
  if (bar_try(bar, 0)) return true;
  const unsigned long long t0 = now_ns();
  for (uint32_t i = 1;; ++i) {
    if (bar_try(bar, 0)) return true;
    if ((i & 63u) == 0u && now_ns() - t0 > limit_ns) {
      atomicExch(status, (int)BITLINEAR_ERR_TIMEOUT);
      return false;
    }
  }
}
// sum over 4 bytes of (unsigned a_i) * (signed b_i), plus c
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

constexpr int kChunks = 6;  // 16-byte weight chunks a thread holds in registers

// Dynamic shared memory: xs[MT][K] int8 activations, red[MT][rows_max] int32
// partial sums, and (fused mode) hs[K] fp32 scratch of the row quantiser.
template <int MT, bool FUSED>
__global__ void __launch_bounds__(kDecThreads, MT <= 2 ? 2 : 1) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t dsmem[];
  __shared__ int sumx[MT];
  __shared__ float den[MT];
  __shared__ RowQuantScratch qsc;

  // Let the next kernel on the stream start (and request its own weights) on
  // the SM resources this grid leaves free; it still waits for our results.
  pdl_release_dependents();

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int c = blockIdx.x;
  int mi = 0;
#pragma unroll
  for (int i = 1; i < kMaxDecodeMats; ++i)
    if (i < p.nmats && c >= p.mats[i].g0) mi = i;
  const DecodeMat& mat = p.mats[mi];
  const int cl = c - mat.g0;
  const int m0 = blockIdx.y * MT;
  const int mcount = min(MT, p.M - m0);
  const int r0 = (int)(((int64_t)cl * mat.N) / mat.G);
  const int r1 = (int)(((int64_t)(cl + 1) * mat.N) / mat.G);
  const int R = r1 - r0;
  const int KB = p.KB;
  const size_t red_off = (size_t)MT * p.K;
  const size_t hs_off = (red_off + (size_t)MT * p.rows_max * 4 + 15) & ~(size_t)15;
  int8_t* xs = reinterpret_cast<int8_t*>(dsmem);
  int* red = reinterpret_cast<int*>(dsmem + red_off);
  float4* hs = reinterpret_cast<float4*>(dsmem + hs_off);

  const int J = kDecThreads / R;
  const int r = t % R, j = t / R;
  const bool active = j < J;
  const uint4* wcol = reinterpret_cast<const uint4*>(mat.packed) + (r0 + r);

  // First batch of weight chunks, requested before the dependency wait.
  uint4 w[kChunks];
#pragma unroll
  for (int u = 0; u < kChunks; ++u) {
    const int kb = j + u * J;
    w[u] = (active && kb < KB) ? ld_stream_u4(wcol + (int64_t)kb * mat.N) : make_uint4(0, 0, 0, 0);
  }

  pdl_wait_primary();

  if constexpr (FUSED) {
    // One token row (MT == 1): quantised here exactly as the act_quant kernel does.
    const float s = quantize_row(p.x + (int64_t)m0 * p.K, p.mul ? p.mul + (int64_t)m0 * p.K : nullptr, p.gamma,
                                 p.eps, p.K, hs, qsc, xs);
    if (t == 0) {
      sumx[0] = 0;
      den[0] = __fmul_rn(s, *mat.sw);
      if (c == 0 && p.sx_out) p.sx_out[m0] = s;
    }
  } else {
    const int4* src = reinterpret_cast<const int4*>(p.xq_in + (int64_t)m0 * p.K);
    int4* dst = reinterpret_cast<int4*>(xs);
    for (int i = t; i < mcount * (p.K >> 4); i += kDecThreads) dst[i] = src[i];
    if (t < MT) {
      sumx[t] = 0;
      den[t] = t < mcount ? __fmul_rn(p.sx_in[m0 + t], *mat.sw) : 1.0f;
    }
  }
  for (int i = t; i < MT * p.rows_max; i += kDecThreads) red[i] = 0;
  __syncthreads();
  if (FUSED && c == 0 && p.xq_out) {
    const int4* src4 = reinterpret_cast<const int4*>(xs);
    int4* dst4 = reinterpret_cast<int4*>(p.xq_out + (int64_t)m0 * p.K);
    for (int i = t; i < (p.K >> 4); i += kDecThreads) dst4[i] = src4[i];
  }

  // Row sums of the activations (the bias of the biased codes c = Wq + 1).
  const int K16 = p.K >> 4;
  for (int m = warp; m < mcount; m += kDecThreads / 32) {
    const int4* row = reinterpret_cast<const int4*>(xs + (size_t)m * p.K);
    int s = 0;
    for (int i = lane; i < K16; i += 32) {
      const int4 v = row[i];
      s = __dp4a(v.x, 0x01010101, s);
      s = __dp4a(v.y, 0x01010101, s);
      s = __dp4a(v.z, 0x01010101, s);
      s = __dp4a(v.w, 0x01010101, s);
    }
    s = __reduce_add_sync(kFullMask, s);
    if (lane == 0) sumx[m] = s;
  }

  if (active) {
    int a0[MT], a1[MT], a2[MT], a3[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) a0[m] = a1[m] = a2[m] = a3[m] = 0;
    for (int kb0 = j; kb0 < KB; kb0 += kChunks * J) {
      if (kb0 != j) {
#pragma unroll
        for (int u = 0; u < kChunks; ++u) {
          const int kb = kb0 + u * J;
          w[u] = kb < KB ? ld_stream_u4(wcol + (int64_t)kb * mat.N) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int u = 0; u < kChunks; ++u) {
        const int kb = kb0 + u * J;
        if (kb < KB) {
          const uint32_t cw[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            const uint32_t q0 = cw[wi] & 0x03030303u, q1 = cw[wi] & 0x0C0C0C0Cu;
            const uint32_t q2 = cw[wi] & 0x30303030u, q3 = cw[wi] & 0xC0C0C0C0u;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              if (m < mcount) {
                const int4 xv = reinterpret_cast<const int4*>(xs + (size_t)m * p.K)[kb * 4 + wi];
                a0[m] = dp4a_us(q0, xv.x, a0[m]);
                a1[m] = dp4a_us(q1, xv.y, a1[m]);
                a2[m] = dp4a_us(q2, xv.z, a2[m]);
                a3[m] = dp4a_us(q3, xv.w, a3[m]);
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m < mcount) {
        // a_s is an exact multiple of 4^s: the shifts are exact
        const int total = a0[m] + (a1[m] >> 2) + (a2[m] >> 4) + (a3[m] >> 6);
        atomicAdd(&red[m * p.rows_max + r], total);
      }
    }
  }
  __syncthreads();
  if (t < R) {
    const int n = r0 + t;
    for (int m = 0; m < mcount; ++m) {
      const int total = red[m * p.rows_max + t] - sumx[m];
      mat.y[(int64_t)(m0 + m) * mat.N + n] = __fdiv_rn(__int2float_rn(total), den[m]);
      if (mat.acc) mat.acc[(int64_t)(m0 + m) * mat.N + n] = total;
    }
  }
}

// Self-test of the bounded wait: one warp waits on an mbarrier that nothing
// ever arrives on; the wait gives up after limit_ns and records the timeout.
__global__ void __launch_bounds__(32) wait_timeout_selftest(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) unsigned long long bar;
  if (threadIdx.x == 0) {
    bar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  if (threadIdx.x == 0) bar_wait(&bar, status, limit_ns);
}

size_t decode_smem_bytes(const DecodeParams& p, int mt) {
  size_t smem = (size_t)mt * p.K + (size_t)mt * p.rows_max * sizeof(int);
  if (p.fused) smem = ((smem + 15) & ~(size_t)15) + (size_t)p.K * sizeof(float);
  return smem;
}

template <int MT, bool FUSED>
cudaError_t launch_mt(const DecodeParams& p, int grid_x, bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  const size_t smem = decode_smem_bytes(p, MT);
  const size_t limit = dev.smem_optin - sizeof(RowQuantScratch) - 1024;
  if (smem > limit) return cudaErrorInvalidValue;
  if (smem > 48 * 1024) {
    static thread_local int configured_device = -1;
    if (configured_device != dev.device) {
      cudaError_t err =
          cudaFuncSetAttribute(decode_kernel<MT, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)limit);
      if (err != cudaSuccess) return err;
      configured_device = dev.device;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid_x, (unsigned)((p.M + MT - 1) / MT), 1);
  cfg.blockDim = dim3(kDecThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, decode_kernel<MT, FUSED>, p);
}

// Splits every matrix into CTAs whose threads hold at most kChunks weight
// chunks each (rows per CTA <= kChunks * 512 / KB, and <= 512), rounded up to a
// multiple of the SM count (balanced waves) but never more CTAs than rows.
// Returns the total CTA count.
int plan_decode(DecodeParams& p, const DecodeMatrix* mats, int nmats, int64_t K, const DeviceInfo& dev) {
  p.K = (int)K;
  p.KB = (int)(K / 64);
  p.nmats = nmats;
  int64_t rows_cap = (int64_t)kChunks * kDecThreads / p.KB;
  if (rows_cap < 1) rows_cap = 1;
  if (rows_cap > kDecThreads) rows_cap = kDecThreads;
  int total = 0, rows_max = 1;
  for (int i = 0; i < nmats; ++i) {
    const int64_t N = mats[i].N;
    int64_t G = (N + rows_cap - 1) / rows_cap;
    G = ((G + dev.num_sms - 1) / dev.num_sms) * dev.num_sms;
    if (G > N) G = N;
    DecodeMat& m = p.mats[i];
    m.packed = mats[i].packed;
    m.sw = mats[i].w_scale;
    m.y = mats[i].y;
    m.acc = mats[i].acc;
    m.N = (int)N;
    m.G = (int)G;
    m.g0 = total;
    total += (int)G;
    const int rm = (int)((N + G - 1) / G);
    if (rm > rows_max) rows_max = rm;
  }
  p.rows_max = rows_max;
  return total;
}

}  // namespace

cudaError_t launch_decode(const int8_t* xq, const float* sx, int64_t M, const DecodeMatrix* mats, int nmats,
                          int64_t K, bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  DecodeParams p = {};
  p.xq_in = xq;
  p.sx_in = sx;
  p.fused = 0;
  p.status = dev.status;
  p.M = (int)M;
  const int grid = plan_decode(p, mats, nmats, K, dev);
  // Token group: up to 8 tokens whose activations (MT * K bytes) fit in 64 KB.
  int mt = M <= 1 ? 1 : (M <= 2 ? 2 : (M <= 4 ? 4 : 8));
  while (mt > 1 && (int64_t)mt * K > 65536) mt >>= 1;
  switch (mt) {
    case 1: return launch_mt<1, false>(p, grid, pdl, dev, stream);
    case 2: return launch_mt<2, false>(p, grid, pdl, dev, stream);
    case 4: return launch_mt<4, false>(p, grid, pdl, dev, stream);
    default: return launch_mt<8, false>(p, grid, pdl, dev, stream);
  }
}

cudaError_t launch_decode_fused(const float* x, const float* mul, const float* gamma, double eps, int64_t K,
                                const DecodeMatrix* mats, int nmats, int8_t* xq_out, float* sx_out, bool pdl,
                                const DeviceInfo& dev, cudaStream_t stream) {
  DecodeParams p = {};
  p.x = x;
  p.mul = mul;
  p.gamma = gamma;
  p.eps = eps;
  p.xq_out = xq_out;
  p.sx_out = sx_out;
  p.fused = 1;
  p.status = dev.status;
  p.M = 1;
  const int grid = plan_decode(p, mats, nmats, K, dev);
  return launch_mt<1, true>(p, grid, pdl, dev, stream);
}

cudaError_t launch_wait_selftest(int64_t limit_ns, const DeviceInfo& dev, cudaStream_t stream) {
  wait_timeout_selftest<<<1, 32, 0, stream>>>(dev.status, (unsigned long long)limit_ns);
  return cudaGetLastError();
}

}  // namespace bitlinear
