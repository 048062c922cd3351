// decode.cu -- BitLinear contraction for few tokens (decode, M small).
//
// y[m, n] = (sum_k xq[m, k] * Wq[n, k]) / (sx[m] * sw)      (BitNet b1.58 BitLinear;
// the per-token BitLinear calls of the decode loop, "Hesper.Models.BitNet"
// page, section "Performance (BitNet-3B on A100)": 870 of 883 ms per token go
// to the 32 layers, i.e. to streaming the 2-bit weights once per token).
//
// At M = 1 the kernel is bound by HBM: every packed byte is read exactly once
// and does 4 weights of work.  Design:
//  * grid = one CTA per SM (x) times ceil(M / MT) token groups (y); CTA c owns
//    rows [c*N/G, (c+1)*N/G) so every SM streams the same number of bytes;
//  * thread t of a CTA owning R rows takes row r = t % R and k-blocks
//    j, j+J, j+2J, ... with j = t / R, J = blockDim / R; consecutive threads
//    read consecutive 16-byte chunks of one k-block plane (fully coalesced);
//  * the first batch of weight loads is issued before griddepcontrol.wait (the
//    packed weights never come from the previous kernel), then the token
//    group's int8 activations, their row sums and sx*sw are staged in shared
//    memory in a single pass, so each CTA waits on memory about twice: once
//    for HBM (weights, overlapping the previous kernel under PDL) and once
//    for L2 (activations);
//  * each 16-byte chunk holds 64 two-bit codes c = Wq+1; (word >> 2s) &
//    0x03030303 lines four codes up with four int8 activations and one dp4a
//    adds c*x for all four; the sum of c*x minus the row sum of x equals the
//    sum of Wq*x (the ternary add/sub) exactly;
//  * partial sums of the J threads of a row meet in shared memory (int32
//    atomics, exact in any order), then one thread per row rescales.
#include "common.cuh"

namespace bitlinear {
namespace {

struct DecodeParams {
  const int8_t* xq;
  const float* sx;
  const uint4* packed;
  const float* sw;
  float* y;
  int32_t* acc;
  int M, N, K, KB;
  int rows_tile;  // rows per pass of a CTA (<= blockDim.x)
};

constexpr int kUnroll = 4;

// Dynamic shared memory: xs[MT][K] int8 activations of the token group, then
// red[MT][rows_tile] int32 partial sums.
template <int MT>
__global__ void __launch_bounds__(MT <= 2 ? 1024 : 512, 1) decode_kernel(const DecodeParams p) {
  extern __shared__ int4 dsmem[];
  __shared__ int sumx[MT];
  __shared__ float den[MT];
  int8_t* xs = reinterpret_cast<int8_t*>(dsmem);
  int* red = reinterpret_cast<int*>(xs + (size_t)MT * p.K);

  // Let the next kernel on the stream (normally the next BitLinear call) start
  // its weight loads on SMs this grid frees; it still waits for our results.
  pdl_release_dependents();

  const int G = gridDim.x;
  const int c = blockIdx.x;
  const int m0 = blockIdx.y * MT;
  const int mcount = min(MT, p.M - m0);
  const int r0 = (int)(((int64_t)c * p.N) / G);
  const int r1 = (int)(((int64_t)(c + 1) * p.N) / G);
  const int T = blockDim.x;
  const int t = threadIdx.x;
  const int warp = t >> 5, lane = t & 31;
  const int K16 = p.K >> 4;

  // First tile geometry and its first batch of weight loads: issued before the
  // wait because the packed weights do not come from the previous kernel.
  int rt0 = r0;
  int R = min(p.rows_tile, r1 - rt0);
  int J = T / R;
  int r = t % R, j = t / R;
  uint4 w[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int kb = j + u * J;
    w[u] = (j < J && kb < p.KB) ? ld_stream_u4(p.packed + (int64_t)kb * p.N + rt0 + r)
                                : make_uint4(0, 0, 0, 0);
  }

  pdl_wait_primary();

  // Stage the token group's activations (one pass over L2) and the scales.
  if (t < MT) {
    sumx[t] = 0;
    den[t] = t < mcount ? __fmul_rn(p.sx[m0 + t], *p.sw) : 1.0f;
  }
  {
    const int4* src = reinterpret_cast<const int4*>(p.xq + (int64_t)m0 * p.K);
    int4* dst = reinterpret_cast<int4*>(xs);
    for (int i = t; i < mcount * K16; i += T) dst[i] = src[i];
  }
  __syncthreads();
  // Row sums of the activations (the bias of the biased codes c = Wq + 1).
  for (int m = warp; m < mcount; m += T / 32) {
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

  bool first = true;
  for (; rt0 < r1; rt0 += p.rows_tile) {
    if (!first) {
      R = min(p.rows_tile, r1 - rt0);
      J = T / R;
      r = t % R;
      j = t / R;
    }
    for (int i = t; i < MT * p.rows_tile; i += T) red[i] = 0;
    __syncthreads();

    int acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0;

    if (j < J) {
      const uint4* wcol = p.packed + (rt0 + r);
      for (int kb0 = j; kb0 < p.KB; kb0 += kUnroll * J) {
        if (!first) {
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int kb = kb0 + u * J;
            w[u] = kb < p.KB ? ld_stream_u4(wcol + (int64_t)kb * p.N) : make_uint4(0, 0, 0, 0);
          }
        }
        first = false;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int kb = kb0 + u * J;
          if (kb < p.KB) {
            const uint32_t cw[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
              const int c0 = (int)(cw[wi] & 0x03030303u);
              const int c1 = (int)((cw[wi] >> 2) & 0x03030303u);
              const int c2 = (int)((cw[wi] >> 4) & 0x03030303u);
              const int c3 = (int)((cw[wi] >> 6) & 0x03030303u);
#pragma unroll
              for (int m = 0; m < MT; ++m) {
                if (m < mcount) {
                  const int4 xv = reinterpret_cast<const int4*>(xs + (size_t)m * p.K)[kb * 4 + wi];
                  int a = acc[m];
                  a = __dp4a(c0, xv.x, a);
                  a = __dp4a(c1, xv.y, a);
                  a = __dp4a(c2, xv.z, a);
                  a = __dp4a(c3, xv.w, a);
                  acc[m] = a;
                }
              }
            }
          }
        }
      }
#pragma unroll
      for (int m = 0; m < MT; ++m)
        if (m < mcount) atomicAdd(&red[m * p.rows_tile + r], acc[m]);
    }
    first = false;
    __syncthreads();
    if (t < R) {
      const int n = rt0 + t;
      for (int m = 0; m < mcount; ++m) {
        const int total = red[m * p.rows_tile + t] - sumx[m];
        p.y[(int64_t)(m0 + m) * p.N + n] = __fdiv_rn(__int2float_rn(total), den[m]);
        if (p.acc) p.acc[(int64_t)(m0 + m) * p.N + n] = total;
      }
    }
    __syncthreads();
  }
}

template <int MT>
cudaError_t launch_mt(const DecodeParams& p, int grid_x, int threads, bool pdl, const DeviceInfo& dev,
                      cudaStream_t stream) {
  const size_t smem = (size_t)MT * p.K + (size_t)MT * p.rows_tile * sizeof(int);
  if (smem > 48 * 1024) {
    static thread_local int configured_device = -1;
    if (configured_device != dev.device) {
      cudaError_t err = cudaFuncSetAttribute(decode_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(dev.smem_optin - 2048));
      if (err != cudaSuccess) return err;
      configured_device = dev.device;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid_x, (unsigned)((p.M + MT - 1) / MT), 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, decode_kernel<MT>, p);
}

}  // namespace

cudaError_t launch_decode(const int8_t* xq, const float* sx, int64_t M, const uint8_t* packed,
                          const float* sw, int64_t N, int64_t K, float* y, int32_t* acc,
                          bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  DecodeParams p;
  p.xq = xq;
  p.sx = sx;
  p.packed = reinterpret_cast<const uint4*>(packed);
  p.sw = sw;
  p.y = y;
  p.acc = acc;
  p.M = (int)M;
  p.N = (int)N;
  p.K = (int)K;
  p.KB = (int)(K / 64);
  // Token group size: up to 8 tokens, with the group's activations (MT * K
  // bytes) held in at most 64 KB of shared memory.
  int mt = M <= 1 ? 1 : (M <= 2 ? 2 : (M <= 4 ? 4 : 8));
  while (mt > 1 && (int64_t)mt * K > 65536) mt >>= 1;
  const int tmax = mt <= 2 ? 1024 : 512;
  const int G = (int)(N < dev.num_sms ? N : dev.num_sms);
  const int rmax = (int)((N + G - 1) / G);
  p.rows_tile = rmax < tmax ? rmax : tmax;
  const int threads = p.rows_tile * (tmax / p.rows_tile);
  switch (mt) {
    case 1: return launch_mt<1>(p, G, threads, pdl, dev, stream);
    case 2: return launch_mt<2>(p, G, threads, pdl, dev, stream);
    case 4: return launch_mt<4>(p, G, threads, pdl, dev, stream);
    default: return launch_mt<8>(p, G, threads, pdl, dev, stream);
  }
}

}  // namespace bitlinear
