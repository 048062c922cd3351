// decode.cu -- BitLinear contraction for few tokens (decode, M small).
//
// y[m, n] = (sum_k xq[m, k] * Wq[n, k]) / (sx[m] * sw)      (BitNet b1.58 BitLinear;
// the per-token BitLinear calls of the decode loop, "Hesper.Models.BitNet"
// page, section "Performance (BitNet-3B on A100)": 870 of 883 ms per token go
// to the 32 layers, i.e. to streaming the 2-bit weights once per token).
//
// At M = 1 the kernel is bound by HBM: every packed byte is read exactly once
// and does 4 weights of work.  Design:
//  * grid: about one CTA per SM per launch (CTA c of a matrix owns rows
//    [c*N/G, (c+1)*N/G); the matrices of one launch -- q, k, v or gate, up,
//    which share one input -- split the SMs in proportion to their bytes), and
//    each CTA uses at most half of an SM (512 threads of <= 64 registers, about
//    100 KB of shared memory), so under programmatic dependent launch the
//    next launch's CTAs become resident while this one runs;
//  * first thing, before griddepcontrol.wait, a CTA bulk-copies all of its
//    weights (one copy per k-block plane: its rows are contiguous there) into
//    shared memory -- the packed weights never come from the previous kernel,
//    so they stream from HBM while the previous kernel finishes, through the
//    copy engine rather than the load/store path;
//  * after the wait, the token group's int8 activations are staged in shared
//    memory (or, in the fused mode, the fp32 row is staged and quantised there
//    by every CTA), one memory round trip;
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
  uint32_t w_off;  // byte offset of the weight planes in dynamic shared memory
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

constexpr int kMaxWeightBytes = 96 * 1024;  // weight planes a CTA holds in shared memory

__device__ __forceinline__ void expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_copy(void* dst_smem, const void* src, uint32_t bytes, unsigned long long* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst_smem)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// Dynamic shared memory: xs[MT][K] int8 activations, red[MT][rows_max] int32
// partial sums, (fused mode) the staged fp32 row, gating input and gamma, and
// at w_off the CTA's weight planes: plane kb holds rows r0 .. r1 as R
// consecutive 16-byte chunks.
template <int MT, bool FUSED>
__global__ void __launch_bounds__(kDecThreads, 2) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t dsmem[];
  __shared__ int sumx[MT];
  __shared__ float den[MT];
  __shared__ __align__(8) unsigned long long wbar;
  __shared__ RowQuantScratch qsc;

  const int t = threadIdx.x, lane = t & 31;
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
  float4* hs = reinterpret_cast<float4*>(dsmem + hs_off);      // fused: staged row
  float4* us = hs + (p.K >> 2);                                 // fused: staged gating input
  float4* gs = us + (p.mul ? (p.K >> 2) : 0);                   // fused: staged gamma
  uint4* wsm = reinterpret_cast<uint4*>(dsmem + p.w_off);

  // The weights: one bulk copy per k-block plane into shared memory, issued
  // before the dependency wait (warp 0; the byte count is registered first).
  if (t < 32) {
    if (t == 0) {
      bar_init(&wbar, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      expect_tx(&wbar, (uint32_t)R * (uint32_t)KB * 16u);
    }
    __syncwarp();
    const uint4* src = reinterpret_cast<const uint4*>(mat.packed) + r0;
    for (int kb = lane; kb < KB; kb += 32)
      bulk_copy(wsm + (size_t)kb * R, src + (int64_t)kb * mat.N, (uint32_t)R * 16u, &wbar);
  }
  // Let the next kernel on the stream start (and request its own weights) on
  // the SM resources this grid leaves free; it still waits for our results.
  pdl_release_dependents();
  if (t < MT) sumx[t] = 0;
  for (int i = t; i < MT * p.rows_max; i += kDecThreads) red[i] = 0;

  pdl_wait_primary();

  if constexpr (FUSED) {
    // One token row (MT == 1): quantised here exactly as the act_quant kernel
    // does; the quantiser also leaves sum_k xq[k] in sumx[0].
    stage_row(p.x + (int64_t)m0 * p.K, p.mul ? p.mul + (int64_t)m0 * p.K : nullptr, p.gamma, p.K, hs, us, gs);
    const float s = quantize_row_staged(p.mul != nullptr, p.gamma != nullptr, p.eps, p.K, hs, us, gs, qsc, xs,
                                        &sumx[0]);
    if (t == 0) {
      den[0] = __fmul_rn(s, *mat.sw);
      if (c == 0 && p.sx_out) p.sx_out[m0] = s;
    }
  } else {
    // int8 rows -> shared memory in one round trip (cp.async bypasses the registers)
    const int4* src = reinterpret_cast<const int4*>(p.xq_in + (int64_t)m0 * p.K);
    int4* dst = reinterpret_cast<int4*>(xs);
    for (int i = t; i < mcount * (p.K >> 4); i += kDecThreads) cp_async16_row(dst + i, src + i);
    if (t < MT) den[t] = t < mcount ? __fmul_rn(p.sx_in[m0 + t], *mat.sw) : 1.0f;
    asm volatile("cp.async.wait_all;" ::: "memory");
  }
  __syncthreads();
  if (FUSED && c == 0 && p.xq_out) {
    const int4* src4 = reinterpret_cast<const int4*>(xs);
    int4* dst4 = reinterpret_cast<int4*>(p.xq_out + (int64_t)m0 * p.K);
    for (int i = t; i < (p.K >> 4); i += kDecThreads) dst4[i] = src4[i];
  }

  // Row sums of the activations (the bias of the biased codes c = Wq + 1):
  // every warp sums a slice of each row, the slices meet in shared memory
  // (exact in any order); they are read after the barrier that ends the dots.
  if constexpr (!FUSED) {
    const int K16 = p.K >> 4;
    for (int m = 0; m < mcount; ++m) {
      const int4* row = reinterpret_cast<const int4*>(xs + (size_t)m * p.K);
      int s = 0;
      for (int i = t; i < K16; i += kDecThreads) {
        const int4 v = row[i];
        s = __dp4a(v.x, 0x01010101, s);
        s = __dp4a(v.y, 0x01010101, s);
        s = __dp4a(v.z, 0x01010101, s);
        s = __dp4a(v.w, 0x01010101, s);
      }
      s = __reduce_add_sync(kFullMask, s);
      if (lane == 0 && s != 0) atomicAdd(&sumx[m], s);
    }
  }

  // The weights have landed (bounded wait; on timeout the status word says so
  // and the outputs are not written).
  const bool have_w = bar_wait(&wbar, p.status);

  // Thread t: row r = t % R, planes kb = j, j + J, ... (j = t / R, J = 512 / R).
  const int J = kDecThreads / R;
  const int r = t % R, j = t / R;
  if (have_w && j < J) {
    int a0[MT], a1[MT], a2[MT], a3[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) a0[m] = a1[m] = a2[m] = a3[m] = 0;
#pragma unroll 2
    for (int kb = j; kb < KB; kb += J) {
      const uint4 wv = wsm[(size_t)kb * R + r];
      const uint32_t cw[4] = {wv.x, wv.y, wv.z, wv.w};
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
  if (have_w && t < R) {
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

// Activations, partial sums and staging first; the weight planes after them.
size_t decode_front_bytes(const DecodeParams& p, int mt) {
  size_t smem = (size_t)mt * p.K + (size_t)mt * p.rows_max * sizeof(int);
  if (p.fused) {
    const int rows = 1 + (p.mul ? 1 : 0) + (p.gamma ? 1 : 0);  // staged x, mul, gamma
    smem = ((smem + 15) & ~(size_t)15) + (size_t)rows * p.K * sizeof(float);
  }
  return (smem + 127) & ~(size_t)127;
}

template <int MT, bool FUSED>
cudaError_t launch_mt(const DecodeParams& p, int grid_x, bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  DecodeParams q = p;
  q.w_off = (uint32_t)decode_front_bytes(p, MT);
  const size_t smem = (size_t)q.w_off + (size_t)p.rows_max * p.KB * 16;
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
  return cudaLaunchKernelEx(&cfg, decode_kernel<MT, FUSED>, q);
}

// Splits the launch's matrices over about one CTA per SM, in proportion to
// their bytes, with at most kMaxWeightBytes of weights and at most 512 rows a
// CTA (more CTAs, in further waves, where a matrix needs it).  Returns the
// total CTA count.
int plan_decode(DecodeParams& p, const DecodeMatrix* mats, int nmats, int64_t K, int mt, const DeviceInfo& dev) {
  p.K = (int)K;
  p.KB = (int)(K / 64);
  p.nmats = nmats;
  int64_t all_rows = 0;
  for (int i = 0; i < nmats; ++i) all_rows += mats[i].N;
  const int64_t row_bytes = (int64_t)p.KB * 16;
  // Shared memory left for weights next to the activations, partial sums
  // (sized for the 512-row maximum here) and staging.
  p.rows_max = kDecThreads;
  const int64_t room = (int64_t)dev.smem_optin - (int64_t)sizeof(RowQuantScratch) - 1024 -
                       (int64_t)decode_front_bytes(p, mt);
  int64_t rows_cap = (room < kMaxWeightBytes ? room : kMaxWeightBytes) / row_bytes;
  if (rows_cap < 1) rows_cap = 1;
  if (rows_cap > kDecThreads) rows_cap = kDecThreads;
  int total = 0, rows_max = 1;
  for (int i = 0; i < nmats; ++i) {
    const int64_t N = mats[i].N;
    int64_t G = (dev.num_sms * N + all_rows / 2) / all_rows;  // this matrix's share of the SMs
    if (G < 1) G = 1;
    if ((N + G - 1) / G > rows_cap) G = (N + rows_cap - 1) / rows_cap;
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
  // Token group: up to 8 tokens whose activations (MT * K bytes) fit in 64 KB.
  int mt = M <= 1 ? 1 : (M <= 2 ? 2 : (M <= 4 ? 4 : 8));
  while (mt > 1 && (int64_t)mt * K > 65536) mt >>= 1;
  const int grid = plan_decode(p, mats, nmats, K, mt, dev);
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
  const int grid = plan_decode(p, mats, nmats, K, 1, dev);
  return launch_mt<1, true>(p, grid, pdl, dev, stream);
}

cudaError_t launch_wait_selftest(int64_t limit_ns, const DeviceInfo& dev, cudaStream_t stream) {
  wait_timeout_selftest<<<1, 32, 0, stream>>>(dev.status, (unsigned long long)limit_ns);
  return cudaGetLastError();
}

}  // namespace bitlinear
