// decode.cu -- BitLinear contraction for few tokens (decode, M small).
//
// y[m, n] = (sum_k xq[m, k] * Wq[n, k]) / (sx[m] * sw)      (BitNet b1.58 BitLinear;
// the per-token BitLinear calls of the decode loop, "Hesper.Models.BitNet"
// page, section "Performance (BitNet-3B on A100)": 870 of 883 ms per token go
// to the 32 layers, i.e. to streaming the 2-bit weights once per token).
//
// At M = 1 every packed byte is read exactly once and does 4 weights of work;
// calls run back to back, each waiting for the previous one's output.  Design:
//  * grid: about one CTA per SM per launch (CTA c of a matrix owns rows
//    [c*N/G, (c+1)*N/G); the matrices of one launch -- q, k, v or gate, up,
//    which share one input -- split the SMs in proportion to their rows, or,
//    for a gated gate / up pair, every CTA holds the same rows of both), and
//    each CTA uses at most half of an SM (512 threads of <= 64 registers,
//    <= ~110 KB of shared memory; for one or two tokens, whose launches
//    follow one another directly), so under programmatic dependent launch the
//    next launch's CTAs are resident while this one runs;
//  * first thing, before griddepcontrol.wait, warp 0 bulk-copies the RMSNorm
//    gamma when there is one (on its own mbarrier) and all of the CTA's
//    weights (one copy per k-block plane: its rows are contiguous there) into
//    shared memory, and the weight scales are loaded -- they never come from
//    the previous kernel, so they stream from HBM while it finishes;
//  * after the wait (fused mode: M = 1, or two tokens without prologues)
//    every thread loads its share of the fp32 rows straight into registers
//    -- one memory round trip -- applies the optional gating and RMSNorm
//    there, and the rows are quantised with block barriers (the absmax, then
//    the codes in shared memory); with int8 input (M tokens) the token rows
//    are staged with cp.async;
//  * dots: the CTA's (k-block, row) chunks are dealt out to the 512 threads
//    flat, in the order of the weight planes (chunk c = kb * R + r), so every
//    thread gets the same number of chunks and a warp reads 32 consecutive
//    16-byte chunks of one plane while its lanes share the activation slice
//    (a shared-memory broadcast).  Per 32-bit code word w, the masks
//    w & (0x03030303 << 2s) (s = 0..3) hold four codes scaled by 4^s, so one
//    dp4a (unsigned x signed) per mask adds 4^s * sum c*x; the four sums are
//    combined with exact shifts and subtracting the row sum of x gives
//    sum Wq*x (the ternary add/sub) exactly.  On GB300 the dp4a pipe accepts
//    about 32 per clock per SM, which bounds this phase;
//  * dots for 8 or 16 tokens (int8 input): the warp-level fp16 MMA
//    (m16n8k16, fp32 sums; ~950 multiply-adds per clock per SM on GB300
//    against dp4a's ~128, while its int8 form runs at a quarter of that).
//    The masked code words are the A fragments as they are (fp16 subnormals
//    c * 2^-24, exact), each warp works through a contiguous piece of the
//    CTA's (16-row tile group, k-block) space, and every 8 tokens are one
//    column tile; see the dot phase for the k matching and the exactness;
//  * each chunk's or piece's sum meets its row's others in shared memory (an
//    int32 atomic, exact in any order), then one thread per row rescales
//    (and, for a gated pair, writes ReLU^2(gate) * up).
#include "quant_row.cuh"

namespace bitlinear {
namespace {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr unsigned long long kWaitNs = 2000000000ull;
// Static shared memory of a decode CTA (the row-quantisation scratch, the
// barriers and the per-token scalars: 4 KB by ptxas for every instance), for
// the two-CTAs-per-SM budget below.
constexpr int kDecStaticSmem = 4352;
constexpr int kMaxNJ = 8;                   // fused mode: K <= kDecThreads * 4 * kMaxNJ

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
  // int8 input (not fused): xq_in, sx_in.  fp32 input (fused, M == 1): x,
  // mul, gamma, eps; every CTA quantises the row itself and CTA 0 writes
  // xq_out, sx_out when they are given.
  const int8_t* xq_in;
  const float* sx_in;
  const float* x;
  const float* mul;
  const float* gamma;
  double eps;
  int8_t* xq_out;
  float* sx_out;
  int* status;
  int M, K, KB;
  int ksplit;       // CTAs of a thread-block cluster, each taking one K range of the same rows
  int XS;           // bytes from one token row of xs to the next (the CTA's K range, + 64 for the MMA dots)
  int rows_max;     // max rows of a CTA over all matrices
  uint32_t off_xs;  // byte offsets in dynamic shared memory: int8 activations,
  uint32_t off_red; //   int32 row sums,
  uint32_t off_gs;  //   gamma (fused RMSNorm); the weight planes start at 0
  int nmats;
  // Gated pair (nmats == 2, equal N): every CTA takes rows r0 .. r1 - 1 of
  // both matrices (gate, then up) and writes mats[0].y = (r * r) * u with
  // r = max(gate, 0), mats[1].y = u.
  int gated;
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
// Bounded wait for phase 0 of a single-use barrier (the first test inline:
// a call costs several times the test).
__device__ __noinline__ bool bar_wait_slow(unsigned long long* bar, int* status, unsigned long long limit_ns) {
  const unsigned long long t0 = now_ns();
  for (uint32_t i = 1;; ++i) {
    if (bar_try(bar, 0)) return true;
    if ((i & 63u) == 0u && now_ns() - t0 > limit_ns) {
      atomicExch(status, (int)BITLINEAR_ERR_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ bool bar_wait(unsigned long long* bar, int* status, unsigned long long limit_ns = kWaitNs) {
  return bar_try(bar, 0) || bar_wait_slow(bar, status, limit_ns);
}
// sum over 4 bytes of (unsigned a_i) * (signed b_i), plus c
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ void expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_copy(void* dst_smem, const void* src, uint32_t bytes, unsigned long long* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst_smem)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}
// Thread-block clusters (the K split): this CTA's rank, the split halves of
// the all-thread cluster barrier, and an atomic add into the shared memory
// of another CTA of the cluster.
__device__ __forceinline__ int cluster_rank_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return (int)r;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t shared_of_rank(uint32_t addr, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void red_add_cluster(uint32_t cluster_addr, int v) {
  asm volatile("red.relaxed.cluster.shared::cluster.add.s32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// 16-byte load through L2 only (the row was written by the previous kernel).
__device__ __forceinline__ float4 ld_cg4(const float4* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}
// sum_k c_k x_k over one 16-byte chunk (64 codes) and its 64 activations
__device__ __forceinline__ int chunk_dot(const uint4 wv, const int4* xp) {
  int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
  const uint32_t cw[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    const int4 xv = xp[wi];
    a0 = dp4a_us(cw[wi] & 0x03030303u, xv.x, a0);
    a1 = dp4a_us(cw[wi] & 0x0C0C0C0Cu, xv.y, a1);
    a2 = dp4a_us(cw[wi] & 0x30303030u, xv.z, a2);
    a3 = dp4a_us(cw[wi] & 0xC0C0C0C0u, xv.w, a3);
  }
  // a_s is an exact multiple of 4^s: the shifts are exact
  return a0 + (a1 >> 2) + (a2 >> 4) + (a3 >> 6);
}

// D += A * B for one 16 x 8 x 16 fp16 tile with fp32 accumulation (the warp-level MMA)
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Four int8 activations (bytes 0..3 of X) as two fp16 pairs (bytes 0, 2) and
// (bytes 1, 3), exactly: with u = X ^ 0x80 per byte (the value + 128), the half
// with bits 0x64uu is 1024 + u, and subtracting 1152 leaves the value.
__device__ __forceinline__ void int8x4_to_f16x2x2(uint32_t X, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = X ^ 0x80808080u;
  const uint32_t e = __byte_perm(u, 0x64646464u, 0x4240);
  const uint32_t o = __byte_perm(u, 0x64646464u, 0x4341);
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(e), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(o), "r"(0x64806480u));
}

// Fused-mode quantisation of one token row held in registers: thread t owns
// the float4 elements e = t + 512 j (j < NJ, e < K/4) of the row, taken in a
// CTA-dependent rotation (by whole 128-byte lines) so that the CTAs' first
// requests spread over the L2 slices.  Writes the int8 codes to xs (shared)
// and, when out is not NULL, to out (global); adds sum_k xq[k] to *sumx.
// Returns sx; *have_g is false when gamma's copy (completing on gbar) did not
// arrive in time.  Every thread of the block calls it.
template <int NJ, bool NORM>
__device__ float quantize_row_regs(const float* __restrict__ x, const float* __restrict__ mul,
                                   const float4* gs, double eps, int K, unsigned long long* gbar, int* status,
                                   RowQuantScratch& sc, int8_t* xs, int8_t* out, int* sumx, bool* have_g) {
  const int t = threadIdx.x, lane = t & 31;
  const int K4 = K >> 2;
  const int rot = (int)((blockIdx.x * 296u) % (unsigned)K4) & ~7;
  int idx[NJ];
  bool ok[NJ];
  float4 h[NJ];
  const float4* x4 = reinterpret_cast<const float4*>(x);
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = t + j * kDecThreads;
    ok[j] = e < K4;
    int i = e + rot;
    if (i >= K4) i -= K4;
    idx[j] = ok[j] ? i : 0;
    h[j] = ok[j] ? ld_cg4(x4 + idx[j]) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // 1/K for the RMSNorm scale, by the thread that takes it, while the row's
  // loads are in flight (parked in shared memory, not a register)
  if (NORM && t == 0) sc.rcp_k = __drcp_rn((double)K);
  if (mul) {
    // h = (r*r)*u with r = max(g, 0): the ReLU^2 gating of the FFN
    const float4* u4 = reinterpret_cast<const float4*>(mul);
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (!ok[j]) continue;
      const float4 u = ld_cg4(u4 + idx[j]);
      float r;
      r = fmaxf(h[j].x, 0.0f); h[j].x = __fmul_rn(__fmul_rn(r, r), u.x);
      r = fmaxf(h[j].y, 0.0f); h[j].y = __fmul_rn(__fmul_rn(r, r), u.y);
      r = fmaxf(h[j].z, 0.0f); h[j].z = __fmul_rn(__fmul_rn(r, r), u.z);
      r = fmaxf(h[j].w, 0.0f); h[j].w = __fmul_rn(__fmul_rn(r, r), u.w);
    }
  }
  if constexpr (NORM) {
    // RMSNorm: inv = fp32(1 / sqrt(S/K + eps)) in fp64 from the exact sum S
    int e = 0, lo = 255;
#pragma unroll
    for (int j = 0; j < NJ; ++j)
      if (ok[j]) {
        exponent_range_add(__float_as_uint(h[j].x), e, lo);
        exponent_range_add(__float_as_uint(h[j].y), e, lo);
        exponent_range_add(__float_as_uint(h[j].z), e, lo);
        exponent_range_add(__float_as_uint(h[j].w), e, lo);
      }
    int emax, emin;
    block_exponent_range(e, lo, sc, &emax, &emin);
    double S = 0.0;
    bool done = emax == 0;
    if (!done && emax - emin <= 31) {
      U128 W = {0, 0};
      int far = 0;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        if (!ok[j]) continue;
        sq_window0_add(__float_as_uint(h[j].x), emax, W, far);
        sq_window0_add(__float_as_uint(h[j].y), emax, W, far);
        sq_window0_add(__float_as_uint(h[j].z), emax, W, far);
        sq_window0_add(__float_as_uint(h[j].w), emax, W, far);
      }
      done = block_window0(W, far, emax, sc, &S);
    }
    if (!done && emax - emin <= 95) {
      U128 A[3] = {{0, 0}, {0, 0}, {0, 0}};
      int slow = 0;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        if (!ok[j]) continue;
        sq_window_add(__float_as_uint(h[j].x), emax, A, slow);
        sq_window_add(__float_as_uint(h[j].y), emax, A, slow);
        sq_window_add(__float_as_uint(h[j].z), emax, A, slow);
        sq_window_add(__float_as_uint(h[j].w), emax, A, slow);
      }
      done = block_windows(A, slow, emax, sc, &S);
    }
    if (!done) {
      zero_buckets(sc);
      __syncthreads();
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const float4 v = ok[j] ? h[j] : make_float4(0.f, 0.f, 0.f, 0.f);
        bucket_sq_add(v.x, sc);
        bucket_sq_add(v.y, sc);
        bucket_sq_add(v.z, sc);
        bucket_sq_add(v.w, sc);
      }
      S = bucket_fold(sc);
    }
    // one thread takes the fp64 steps (fp64 is slow on this GPU), the block
    // picks the result up after a barrier
    if (t == 0) sc.inv = rms_inv(S, K, sc.rcp_k, eps);
    __syncthreads();
    const float inv = sc.inv;
    // gamma's own copy, issued ahead of the weights (bounded wait; on timeout
    // the status word says so and the outputs are not written)
    *have_g = bar_wait(gbar, status);
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (!ok[j]) continue;
      const float4 g = gs[idx[j]];
      h[j].x = __fmul_rn(__fmul_rn(h[j].x, inv), g.x);
      h[j].y = __fmul_rn(__fmul_rn(h[j].y, inv), g.y);
      h[j].z = __fmul_rn(__fmul_rn(h[j].z, inv), g.z);
      h[j].w = __fmul_rn(__fmul_rn(h[j].w, inv), g.w);
    }
  }
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < NJ; ++j)
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(h[j].x), fabsf(h[j].y)), fmaxf(fabsf(h[j].z), fabsf(h[j].w))));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, o));
  if (lane == 0) sc.red[t >> 5] = amax;
  __syncthreads();
  amax = sc.red[0];
#pragma unroll
  for (int w = 1; w < kDecWarps; ++w) amax = fmaxf(amax, sc.red[w]);
  const float s = __fdiv_rn(127.0f, fmaxf(amax, 1e-5f));
  int qsum = 0;
  int* xs32 = reinterpret_cast<int*>(xs);
  int* xo32 = reinterpret_cast<int*>(out);
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    if (!ok[j]) continue;
    const float f[4] = {h[j].x, h[j].y, h[j].z, h[j].w};
    uint32_t word = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      int v = __float2int_rn(__fmul_rn(f[q], s));
      v = v < -128 ? -128 : (v > 127 ? 127 : v);
      qsum += v;
      word |= ((uint32_t)v & 0xffu) << (8 * q);
    }
    xs32[idx[j]] = (int)word;
    if (out) xo32[idx[j]] = (int)word;
  }
  qsum = __reduce_add_sync(kFullMask, qsum);
  if (lane == 0 && qsum != 0) atomicAdd(sumx, qsum);
  return s;
}

// Fused-mode quantisation of a group's mcount (<= MT <= 8) token rows held in
// registers, without prologues: thread t owns the float4 elements
// f = t + 512 j (j < NJ) of the rows laid end to end (row f / K4), so every
// load is issued before the first use.  Per element group a warp reduces
// first and adds to its row in shared memory (amx: the row's absmax as
// integer bits, which order like the non-negative floats; sumx: the row's sum
// of codes); thread m < mcount leaves row m's sx in sxs[m].  Writes the int8
// codes to xs (shared) and, when out is not NULL, to out (global).  amx must
// be zero and sumx zero before the call; every thread of the block calls it.
template <int MT, int NJ>
__device__ __forceinline__ void quantize_rows_regs(const float* __restrict__ x, int K, int mcount, int* amx,
                                                   float* sxs, int8_t* xs, int8_t* out, int* sumx) {
  static_assert(MT <= 8 && NJ <= 10, "row indices are packed 3 bits each into one word");
  const int t = threadIdx.x, lane = t & 31;
  const int K4 = K >> 2;
  const int total = mcount * K4;
  const int nvalid = total > t ? (total - t + kDecThreads - 1) / kDecThreads : 0;  // elements f < total
  const float4* x4 = reinterpret_cast<const float4*>(x);
  float4 h[NJ];
  uint32_t rows = 0;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int f = t + j * kDecThreads;
    const bool ok = j < nvalid;
    h[j] = ok ? ld_cg4(x4 + f) : make_float4(0.f, 0.f, 0.f, 0.f);
    rows |= (uint32_t)(ok ? f / K4 : 0) << (3 * j);
  }
  __syncthreads();  // amx and sumx were zeroed before the call
  // A warp whose valid lanes share one row reduces first; otherwise each lane adds.
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const bool ok = j < nvalid;
    const int rj = (int)((rows >> (3 * j)) & 7u);
    float a = ok ? fmaxf(fmaxf(fabsf(h[j].x), fabsf(h[j].y)), fmaxf(fabsf(h[j].z), fabsf(h[j].w))) : 0.0f;
    const int r0 = __shfl_sync(kFullMask, rj, 0);
    if (__all_sync(kFullMask, !ok || rj == r0)) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(kFullMask, a, o));
      if (lane == 0 && a > 0.0f) atomicMax(&amx[r0], __float_as_int(a));
    } else if (ok && a > 0.0f) {
      atomicMax(&amx[rj], __float_as_int(a));
    }
  }
  __syncthreads();
  if (t < mcount) sxs[t] = __fdiv_rn(127.0f, fmaxf(__int_as_float(amx[t]), 1e-5f));
  __syncthreads();
  int* xs32 = reinterpret_cast<int*>(xs);
  int* xo32 = reinterpret_cast<int*>(out);
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const bool ok = j < nvalid;
    const int rj = (int)((rows >> (3 * j)) & 7u);
    int q4 = 0;
    if (ok) {
      const float sj = sxs[rj];
      const float f4[4] = {h[j].x, h[j].y, h[j].z, h[j].w};
      uint32_t word = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        int v = __float2int_rn(__fmul_rn(f4[q], sj));
        v = v < -128 ? -128 : (v > 127 ? 127 : v);
        q4 += v;
        word |= ((uint32_t)v & 0xffu) << (8 * q);
      }
      const int f = t + j * kDecThreads;
      xs32[f] = (int)word;
      if (out) xo32[f] = (int)word;
    }
    const int r0 = __shfl_sync(kFullMask, rj, 0);
    if (__all_sync(kFullMask, !ok || rj == r0)) {
      const int q = __reduce_add_sync(kFullMask, q4);
      if (lane == 0 && q != 0) atomicAdd(&sumx[r0], q);
    } else if (ok && q4 != 0) {
      atomicAdd(&sumx[rj], q4);
    }
  }
}

// Dynamic shared memory: the CTA's weight planes at 0 (plane kb holds rows
// r0 .. r1-1 as R consecutive 16-byte chunks), xs[MT][XS] int8 activations at
// off_xs, red[MT][R] int32 row sums at off_red, (fused RMSNorm) gamma at off_gs.
// MMA: the dots run on the warp-level fp16 MMA instead of dp4a (int8 input).
template <int MT, bool FUSED, bool NORM, int NJ, bool MMA = false>
__global__ void __launch_bounds__(kDecThreads, 2) decode_kernel(const __grid_constant__ DecodeParams p) {
  static_assert(!(MMA && FUSED), "the MMA dots take int8 token rows");
  static_assert(MT <= kDecWarps, "the activation row sums take at least one warp a token row");
  extern __shared__ __align__(128) uint8_t dsmem[];
  __shared__ int sumx[MT];
  __shared__ float den[2][MT];  // sx * sw of each token, for mats[mi] and (gated) mats[1]
  __shared__ __align__(8) unsigned long long wbar;
  __shared__ __align__(8) unsigned long long gbar;
  __shared__ RowQuantScratch qsc;

  const int t = threadIdx.x, lane = t & 31;
  // With a K split, the ks CTAs of a cluster take the same rows, each one
  // range of the k-blocks; rank 0 adds up the ranges and writes the outputs.
  const int ks = MMA ? p.ksplit : 1;  // only the MMA dots take a split
  const int rank = ks > 1 ? cluster_rank_id() : 0;
  const int c = ks > 1 ? (int)blockIdx.x / ks : (int)blockIdx.x;
  const bool gated = p.gated != 0;
  int mi = 0;
#pragma unroll
  for (int i = 1; i < kMaxDecodeMats; ++i)
    if (!gated && i < p.nmats && c >= p.mats[i].g0) mi = i;
  const DecodeMat& mat = p.mats[mi];
  const int cl = c - mat.g0;
  const int m0 = blockIdx.y * MT;
  const int mcount = min(MT, p.M - m0);
  const int r0 = (int)(((int64_t)cl * mat.N) / mat.G);
  const int r1 = (int)(((int64_t)(cl + 1) * mat.N) / mat.G);
  const int R = r1 - r0;
  const int RR = gated ? 2 * R : R;  // rows held: R of mats[mi], then (gated) the same R of mats[1]
  const int kb_lo = ks > 1 ? rank * p.KB / ks : 0;
  const int KB = (ks > 1 ? (rank + 1) * p.KB / ks : p.KB) - kb_lo, K = p.K;  // this CTA's k-blocks
  const uint4* wsm = reinterpret_cast<const uint4*>(dsmem);
  int8_t* xs = reinterpret_cast<int8_t*>(dsmem + p.off_xs);
  int* red = reinterpret_cast<int*>(dsmem + p.off_red);
  float4* gs = reinterpret_cast<float4*>(dsmem + p.off_gs);
  constexpr bool norm = FUSED && NORM;  // the host launches NORM exactly when gamma is given

  // The weights and gamma: bulk copies into shared memory, issued before the
  // dependency wait by warp 0 (the byte counts are registered first).  Gamma
  // goes first and completes on its own barrier: the row's scaling needs it
  // long before the last weight plane lands.
  if (t < 32) {
    if (t == 0) {
      bar_init(&wbar, 1);
      if (norm) bar_init(&gbar, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      if (norm) expect_tx(&gbar, (uint32_t)K * 4u);
      expect_tx(&wbar, (uint32_t)RR * (uint32_t)KB * 16u);
    }
    __syncwarp();
    if (norm && lane == 0) bulk_copy(gs, p.gamma, (uint32_t)K * 4u, &gbar);
    const uint4* src = reinterpret_cast<const uint4*>(mat.packed) + (int64_t)kb_lo * mat.N + r0;
    for (int kb = lane; kb < KB; kb += 32)
      bulk_copy((void*)(wsm + (size_t)kb * RR), src + (int64_t)kb * mat.N, (uint32_t)R * 16u, &wbar);
    if (gated) {
      const uint4* src1 = reinterpret_cast<const uint4*>(p.mats[1].packed) + (int64_t)kb_lo * mat.N + r0;
      for (int kb = lane; kb < KB; kb += 32)
        bulk_copy((void*)(wsm + (size_t)kb * RR + R), src1 + (int64_t)kb * mat.N, (uint32_t)R * 16u, &wbar);
    }
  }
  // Let the next kernel on the stream start (and request its own weights) on
  // the SM resources this grid leaves free; it still waits for our results.
  pdl_release_dependents();
  if (t < MT) sumx[t] = 0;
  for (int i = t; i < MT * RR; i += kDecThreads) red[i] = 0;
  // K split: the zeroed row sums are released to the other ranks, whose
  // additions into rank 0's come after the matching wait.
  if (ks > 1) cluster_arrive();
  // The weight scales, like the weights, do not come from the kernel before
  // (the rule of FLAG_PDL): their loads are off the path after the wait.
  const float sw = t < MT ? *mat.sw : 0.0f;
  const float sw1 = gated && t < MT ? *p.mats[1].sw : 0.0f;

  pdl_wait_primary();

  bool have_g = true;
  if constexpr (FUSED && MT > 1) {
    static_assert(!NORM, "the RMSNorm prologue is fused for one token only");
    // a few token rows, no prologue: every CTA quantises the group itself
    __shared__ int amx[MT];
    __shared__ float sxs[MT];
    if (t < MT) amx[t] = 0;
    quantize_rows_regs<MT, NJ>(p.x + (int64_t)m0 * K, K, mcount, amx, sxs, xs,
                               c == 0 && p.xq_out ? p.xq_out + (int64_t)m0 * K : nullptr, &sumx[0]);
    if (t < MT) {
      den[0][t] = t < mcount ? __fmul_rn(sxs[t], sw) : 1.0f;
      den[1][t] = t < mcount ? __fmul_rn(sxs[t], sw1) : 1.0f;
      if (c == 0 && p.sx_out && t < mcount) p.sx_out[m0 + t] = sxs[t];
    }
    __syncthreads();
  } else if constexpr (FUSED) {
    const float s = quantize_row_regs<NJ, norm>(p.x + (int64_t)m0 * K, p.mul ? p.mul + (int64_t)m0 * K : nullptr,
                                                gs, p.eps, K, &gbar, p.status, qsc, xs,
                                          c == 0 ? p.xq_out + (p.xq_out ? (int64_t)m0 * K : 0) : nullptr,
                                          &sumx[0], &have_g);
    if (t == 0) {
      den[0][0] = __fmul_rn(s, sw);
      den[1][0] = __fmul_rn(s, sw1);
      if (c == 0 && p.sx_out) p.sx_out[m0] = s;
    }
    __syncthreads();
  } else {
    // int8 rows -> shared memory in one round trip (cp.async bypasses the registers)
    // this CTA's k range of each token row
    const int4* src = reinterpret_cast<const int4*>(p.xq_in + (int64_t)m0 * K) + kb_lo * 4;
    const int K16 = K >> 4, R16 = KB * 4, XS16 = p.XS >> 4;
    int4* dst = reinterpret_cast<int4*>(xs);
    int m = t / R16, j = t - m * R16;  // element t + 512 i of the ranges laid end to end
    for (int i = t; i < mcount * R16; i += kDecThreads) {
      cp_async16_row(dst + (m * XS16 + j), src + ((int64_t)m * K16 + j));
      j += kDecThreads;
      while (j >= R16) {
        j -= R16;
        ++m;
      }
    }
    if (t < MT) {
      den[0][t] = t < mcount ? __fmul_rn(p.sx_in[m0 + t], sw) : 1.0f;
      den[1][t] = t < mcount ? __fmul_rn(p.sx_in[m0 + t], sw1) : 1.0f;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    // Row sums of the activations (the bias of the biased codes c = Wq + 1);
    // read after the barrier that ends the dots.  The warps split the rows
    // (kDecWarps / mcount warps a row), so the rows are summed side by side.
    {
      const int wpr = kDecWarps / mcount, warp = t >> 5;
      const int m = warp / wpr;
      if (m < mcount) {
        const int4* row = reinterpret_cast<const int4*>(xs + (size_t)m * p.XS);
        int s = 0;
        for (int i = (warp - m * wpr) * 32 + lane; i < R16; i += wpr * 32) {
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
  }

  // The weights have landed (bounded wait; on timeout the status word says so
  // and the outputs are not written).
  const bool have_w = bar_wait(&wbar, p.status) && have_g;
  if (MMA && have_w) {
    // Warp-level MMA, 16 weight rows x 8 tokens x 16 k a step, fp32 sums.
    // Thread (g = lane / 4, q = lane % 4) of a warp takes, in every 64-k
    // block, code word q of rows g and g + 8 and the 16 activations
    // 16q .. 16q + 15 of token g: the MMA sums over its 16 k in any order, so
    // the k of the fragments are matched up rather than laid out in order.
    // A code word w (code of k = 16q + i at bit 8 (i % 4) + 2 (i / 4)) gives,
    // per 16-bit half, w & 0x0003 -> c and w & 0x000C -> 4c: the fp16 with
    // those bits is the subnormal c * 2^-24 or 4c * 2^-24, exact, and so is
    // every product with an int8 activation.  The fp32 sums stay exact integer
    // multiples of 2^-24 (of 2^-22 for the 4c terms, kept in their own
    // accumulator) below 2^24 of those units for K <= 131072, and scale back
    // to int32 exactly.  The activations are widened per use (two byte
    // permutes and an fp16 subtract per pair).
    constexpr int NT = MT >= 8 ? MT / 8 : 1;  // 8-token column tiles
    constexpr int TT = NT == 1 ? 2 : 1;       // 16-row tiles of a unit (register budget)
    constexpr uint32_t M0 = 0x00030003u, M1 = 0x000C000Cu;
    const int warp = t >> 5, g = lane >> 2, q = lane & 3;
    const int NG = (((RR + 15) >> 4) + TT - 1) / TT;  // row-tile groups
    const uint32_t* w32 = reinterpret_cast<const uint32_t*>(dsmem);
    int xrow[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) xrow[nt] = min(nt * 8 + g, MT - 1) * p.XS + 16 * q;
    // The (group, k-block) space in group-major order, cut into one piece a
    // warp; a piece that crosses into the next group flushes its sums there.
    const int total = NG * KB;
    int pos = (int)((int64_t)warp * total / kDecWarps);
    const int end = (int)((int64_t)(warp + 1) * total / kDecWarps);
    while (pos < end) {
      const int gi = pos / KB, kb0 = pos - gi * KB;
      const int kb1 = min(KB, kb0 + (end - pos));
      pos += kb1 - kb0;
      float acc[TT][NT][2][4];
#pragma unroll
      for (int ti = 0; ti < TT; ++ti)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[ti][nt][0][i] = acc[ti][nt][1][i] = 0.0f;
      const int rbase = gi * TT * 16 + g;  // rows past RR read a valid row; their sums are dropped
      for (int kb = kb0; kb < kb1; ++kb) {
        uint32_t bf[NT][4][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xs + xrow[nt] + kb * 64);
          int8x4_to_f16x2x2(xv.x, bf[nt][0][0], bf[nt][0][1]);
          int8x4_to_f16x2x2(xv.y, bf[nt][1][0], bf[nt][1][1]);
          int8x4_to_f16x2x2(xv.z, bf[nt][2][0], bf[nt][2][1]);
          int8x4_to_f16x2x2(xv.w, bf[nt][3][0], bf[nt][3][1]);
        }
        const uint32_t* wp = w32 + (size_t)kb * RR * 4;
#pragma unroll
        for (int ti = 0; ti < TT; ++ti) {
          // word s of the activations holds k = 16q + 4s + (0, 1, 2, 3); the
          // code pairs (4s, 4s + 2) and (4s + 1, 4s + 3) match its halves
          const uint32_t wa = wp[min(rbase + ti * 16, RR - 1) * 4 + q];
          const uint32_t wb = wp[min(rbase + ti * 16 + 8, RR - 1) * 4 + q];
          const uint32_t wa4 = wa >> 4, wb4 = wb >> 4, wa8 = wa >> 8, wb8 = wb >> 8;
          const uint32_t wa12 = wa >> 12, wb12 = wb >> 12;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_f16(acc[ti][nt][0], wa & M0, wb & M0, wa8 & M0, wb8 & M0, bf[nt][0][0], bf[nt][0][1]);
            mma_f16(acc[ti][nt][1], wa & M1, wb & M1, wa8 & M1, wb8 & M1, bf[nt][1][0], bf[nt][1][1]);
            mma_f16(acc[ti][nt][0], wa4 & M0, wb4 & M0, wa12 & M0, wb12 & M0, bf[nt][2][0], bf[nt][2][1]);
            mma_f16(acc[ti][nt][1], wa4 & M1, wb4 & M1, wa12 & M1, wb12 & M1, bf[nt][3][0], bf[nt][3][1]);
          }
        }
      }
      // C fragment: (row g, tokens 2q, 2q + 1), then (row g + 8, the same tokens)
#pragma unroll
      for (int ti = 0; ti < TT; ++ti)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int row = (gi * TT + ti) * 16 + g + (i >= 2 ? 8 : 0);
            const int m = nt * 8 + 2 * q + (i & 1);
            const int v = __float2int_rn(acc[ti][nt][0][i] * 16777216.0f) +
                          __float2int_rn(acc[ti][nt][1][i] * 4194304.0f);
            if (row < RR && m < mcount && v != 0) atomicAdd(&red[m * RR + row], v);
          }
    }
  } else if (have_w) {
    // chunk cc = kb * R + r, dealt out flat: thread t takes t, t + 512, ...
    const int4* xs4 = reinterpret_cast<const int4*>(xs);
    const int XS16 = p.XS >> 4;
    const int C = RR * KB;
    const int dq = kDecThreads / RR, dr = kDecThreads - dq * RR;
    int kb = t / RR, r = t - kb * RR;
#pragma unroll 2
    for (int cc = t; cc < C; cc += kDecThreads) {
      const uint4 wv = wsm[cc];
#pragma unroll
      for (int m = 0; m < MT; ++m)
        if (m < mcount) atomicAdd(&red[m * RR + r], chunk_dot(wv, xs4 + m * XS16 + kb * 4));
      kb += dq;
      r += dr;
      if (r >= RR) {
        r -= RR;
        ++kb;
      }
    }
  }
  __syncthreads();
  bool write_out = have_w;
  if (ks > 1) {
    // Ranks 1 .. ks-1 add their sums, each less its own range's activation
    // sums, into rank 0's (after rank 0's row sums were zeroed: the wait);
    // the second barrier makes them visible to rank 0 and keeps rank 0's
    // shared memory alive until the last of them.  A rank that timed out has
    // set the status word, and then rank 0 writes nothing.
    cluster_wait();
    if (rank != 0 && have_w) {
      const uint32_t red0 = shared_of_rank(smem_addr(red), 0);
      for (int i = t; i < mcount * RR; i += kDecThreads) {
        const int v = red[i] - sumx[i / RR];
        if (v != 0) red_add_cluster(red0 + 4u * (uint32_t)i, v);
      }
    }
    cluster_arrive();
    cluster_wait();
    write_out = have_w && rank == 0 && *reinterpret_cast<volatile int*>(p.status) == 0;
  }
  if (write_out) {
    for (int i = t; i < mcount * R; i += kDecThreads) {
      const int m = i / R, rr = i - m * R;
      const int64_t o = (int64_t)(m0 + m) * mat.N + r0 + rr;
      const int total = red[m * RR + rr] - sumx[m];
      const float y0 = __fdiv_rn(__int2float_rn(total), den[0][m]);
      if (mat.acc) mat.acc[o] = total;
      if (gated) {
        // the FFN gating, in the same fp32 steps as the activation prologue
        const int total1 = red[m * RR + R + rr] - sumx[m];
        const float u = __fdiv_rn(__int2float_rn(total1), den[1][m]);
        const float rp = fmaxf(y0, 0.0f);
        mat.y[o] = __fmul_rn(__fmul_rn(rp, rp), u);
        p.mats[1].y[o] = u;
        if (p.mats[1].acc) p.mats[1].acc[o] = total1;
      } else {
        mat.y[o] = y0;
      }
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

// Bytes from one token row of xs to the next: K, or for the MMA dots K
// rounded to an odd multiple of 64, so that the 8 token rows of a warp's
// 16-byte activation loads fall on distinct shared-memory banks.
int64_t decode_xs_stride(int64_t K, bool mma) { return mma && K % 128 == 0 ? K + 64 : K; }

// Bytes of dynamic shared memory besides the weight planes.
size_t decode_front_bytes(int64_t K, int64_t xs_stride, int mt, int rows_max, bool norm) {
  size_t b = (size_t)mt * xs_stride;                       // xs
  b = ((b + 15) & ~(size_t)15) + (size_t)mt * rows_max * 4;  // red
  b = (b + 15) & ~(size_t)15;
  if (norm) b += (size_t)K * 4;                            // gamma
  return (b + 127) & ~(size_t)127;
}

// k-blocks of the widest K range of a split into ks ranges.
int split_kblocks(int KB, int ks) { return (KB + ks - 1) / ks; }

template <int MT, bool FUSED, bool NORM, int NJ, bool MMA = false>
cudaError_t launch_mt(DecodeParams p, int grid_x, bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  const int ks = p.ksplit;
  if (ks < 1 || ks > 8 || (ks > 1 && (!MMA || ks > p.KB))) return cudaErrorInvalidValue;
  const int kbn = split_kblocks(p.KB, ks);
  if (p.XS != decode_xs_stride((int64_t)kbn * 64, MMA)) return cudaErrorInvalidValue;
  const size_t wbytes = ((size_t)p.rows_max * kbn * 16 + 127) & ~(size_t)127;
  p.off_xs = (uint32_t)wbytes;
  p.off_red = (uint32_t)(((wbytes + (size_t)MT * p.XS) + 15) & ~(size_t)15);
  p.off_gs = (uint32_t)((p.off_red + (size_t)MT * p.rows_max * 4 + 15) & ~(size_t)15);
  const size_t smem = wbytes + decode_front_bytes(p.K, p.XS, MT, p.rows_max, NORM);
  const size_t limit = dev.smem_optin - sizeof(RowQuantScratch) - 1024;
  if (smem > limit) return cudaErrorInvalidValue;
  if (smem > 48 * 1024) {
    static thread_local int configured_device = -1;
    if (configured_device != dev.device) {
      cudaError_t err =
          cudaFuncSetAttribute(decode_kernel<MT, FUSED, NORM, NJ, MMA>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)limit);
      if (err != cudaSuccess) return err;
      configured_device = dev.device;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(grid_x * ks), (unsigned)((p.M + MT - 1) / MT), 1);
  cfg.blockDim = dim3(kDecThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (ks > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)ks;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = na ? attr : nullptr;
  cfg.numAttrs = (unsigned)na;
  return cudaLaunchKernelEx(&cfg, decode_kernel<MT, FUSED, NORM, NJ, MMA>, p);
}

// Splits the launch's matrices over about one CTA per SM, in proportion to
// their rows, with at most 512 rows a CTA and, for one or two tokens, no more
// weights than leave room for two CTAs on an SM -- this launch's and the next
// one's, or two of a tall matrix's (more CTAs, in further waves, where a
// matrix needs it).  A gated pair
// (two matrices of equal N) splits as one matrix whose rows weigh double:
// every CTA holds the same rows of both.  With a K split (ks > 1) the unit is
// a row group of ks CTAs, one K range each.  Returns the total row-group count.
int plan_decode(DecodeParams& p, const DecodeMatrix* mats, int nmats, int64_t K, int mt, bool norm, bool gated,
                const DeviceInfo& dev, bool mma = false, int ks = 1) {
  p.K = (int)K;
  p.KB = (int)(K / 64);
  p.ksplit = ks;
  const int kbn = split_kblocks(p.KB, ks);  // a CTA's k-blocks (the widest range)
  p.XS = (int)decode_xs_stride((int64_t)kbn * 64, mma);
  p.nmats = nmats;
  p.gated = gated ? 1 : 0;
  const int per = gated ? 2 : 1;  // weight rows a CTA holds per output row
  int64_t all_rows = 0;
  for (int i = 0; i < (gated ? 1 : nmats); ++i) all_rows += mats[i].N;
  // Shared memory a CTA row costs: its weights and its row sums (one int32 a
  // token); besides them the activations and gamma, and a little for the
  // alignment of each part.
  const int64_t row_bytes = ((int64_t)kbn * 16 + (int64_t)mt * 4) * per;
  const int64_t fixed = (int64_t)decode_front_bytes(K, p.XS, mt, 0, norm) + 384;
  const int64_t room = (int64_t)dev.smem_optin - (int64_t)sizeof(RowQuantScratch) - 1024 - fixed;
  const int64_t pair = (int64_t)dev.smem_per_sm / 2 - 1024 - kDecStaticSmem - fixed;  // two CTAs an SM
  // Groups of 4 tokens or more come after an act_quant launch, during which
  // the next decode launch becomes resident anyway: their CTAs may fill an SM
  // (BitNet-3B token step at M = 16: 1846 -> 1718 us, gate || up's paired
  // rows no longer cut into 209 CTAs; M = 4 and 8 unchanged).
  int64_t rows_cap = (mt >= 4 ? room : (room < pair ? room : pair)) / row_bytes;
  if (rows_cap < 1) rows_cap = 1;
  if (rows_cap * per > kDecThreads) rows_cap = kDecThreads / per;
  // Each matrix's share of the SMs in proportion to its rows, rounded down and
  // the SMs left over given to the largest remainders, so that the shares add
  // up to the SM count: one CTA more than there are SMs waits for a free slot
  // behind the co-resident previous launch and delays the whole grid.
  // (Every matrix has one CTA first; the rest of the SMs are shared out.)
  const int nshare = gated ? 1 : nmats;
  const int64_t groups = dev.num_sms / ks;  // row groups of ks CTAs
  const int64_t pool = groups > nshare ? groups - nshare : 0;
  int64_t share[kMaxDecodeMats];
  int64_t left = pool;
  for (int i = 0; i < nshare; ++i) {
    share[i] = pool * mats[i].N / all_rows;
    left -= share[i];
  }
  for (; left > 0; --left) {
    int best = 0;
    int64_t best_rem = -1;
    for (int i = 0; i < nshare; ++i) {
      const int64_t rem = pool * mats[i].N - share[i] * all_rows;
      if (rem > best_rem) {
        best_rem = rem;
        best = i;
      }
    }
    ++share[best];
  }
  int total = 0, rows_max = 1;
  for (int i = 0; i < nmats; ++i) {
    const int64_t N = mats[i].N;
    int64_t G;
    if (gated && i == 1) {
      G = p.mats[0].G;  // the pair shares one split
    } else {
      G = 1 + share[i];
      if ((N + G - 1) / G > rows_cap) G = (N + rows_cap - 1) / rows_cap;
      if (G > N) G = N;
    }
    DecodeMat& m = p.mats[i];
    m.packed = mats[i].packed;
    m.sw = mats[i].w_scale;
    m.y = mats[i].y;
    m.acc = mats[i].acc;
    m.N = (int)N;
    m.G = (int)G;
    m.g0 = gated ? 0 : total;
    if (!(gated && i == 1)) total += (int)G;
    const int rm = (int)((N + G - 1) / G) * per;
    if (rm > rows_max) rows_max = rm;
  }
  p.rows_max = rows_max;
  return total;
}

// The fused launch for nj float4 elements of the row per thread; the RMSNorm
// prologue is a template argument, so the kernel without it carries none of
// its code.
template <bool NORM>
cudaError_t launch_fused(const DecodeParams& p, int grid, int nj, bool pdl, const DeviceInfo& dev,
                         cudaStream_t stream) {
  switch (nj) {
    case 1: return launch_mt<1, true, NORM, 1>(p, grid, pdl, dev, stream);
    case 2: return launch_mt<1, true, NORM, 2>(p, grid, pdl, dev, stream);
    case 3: return launch_mt<1, true, NORM, 3>(p, grid, pdl, dev, stream);
    case 4: return launch_mt<1, true, NORM, 4>(p, grid, pdl, dev, stream);
    case 5: return launch_mt<1, true, NORM, 5>(p, grid, pdl, dev, stream);
    case 6: return launch_mt<1, true, NORM, 6>(p, grid, pdl, dev, stream);
    default: return launch_mt<1, true, NORM, kMaxNJ>(p, grid, pdl, dev, stream);
  }
}

}  // namespace

// Token groups of up to 16 tokens whose activations stay within 64 KB.  A
// group of 8 or 16 (one or two 8-token column tiles of the warp-level MMA)
// takes the MMA dots; a smaller one dp4a, which at 3-4 tokens beats MMAs
// whose column tiles would be half empty (and at K = 10240, where 8 tokens
// of activations do not fit, 4-token dp4a groups beat 8-token MMA groups
// with fewer weight rows a CTA: 12.4 vs 14.6 us a call at M = 8).
int decode_token_group(int64_t M, int64_t K, bool* mma, int* ks) {
  const int want = M <= 2 ? (int)(M < 1 ? 1 : M) : (M <= 4 ? 4 : (M <= 8 ? 8 : 16));
  int mt = want;
  *ks = 1;
  while (mt > 8 && (int64_t)mt * decode_xs_stride(K, true) > 65536) mt >>= 1;
  *mma = mt >= 8 && (int64_t)mt * decode_xs_stride(K, true) <= 65536;
  if (want >= 8 && !*mma) {
    // Long K: all the tokens (up to 16) in one group, K split over a
    // cluster of 2, 4 or 8 CTAs so that a CTA's range of activations fits
    // (BitNet-3B down, 2560 x 10240: 12.6 -> 8.3 us a call at M = 8, where
    // 4-token dp4a groups ran before; 14.4 on the batched kernel at M = 16
    // -> 14.0).
    const int KB = (int)(K / 64);
    for (int s = 2; s <= 8 && s <= KB; s *= 2)
      if ((int64_t)want * decode_xs_stride((int64_t)split_kblocks(KB, s) * 64, true) <= 65536) {
        *ks = s;
        *mma = true;
        return want;
      }
  }
  while (!*mma && mt > 1 && (int64_t)mt * K > 65536) mt >>= 1;
  return mt;
}

cudaError_t launch_decode(const int8_t* xq, const float* sx, int64_t M, const DecodeMatrix* mats, int nmats,
                          int64_t K, bool gated, bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  DecodeParams p = {};
  p.xq_in = xq;
  p.sx_in = sx;
  p.status = dev.status;
  p.M = (int)M;
  bool mma = false;
  int ks = 1;
  const int mt = decode_token_group(M, K, &mma, &ks);
  const int grid = plan_decode(p, mats, nmats, K, mt, false, gated, dev, mma, ks);
  switch (mt) {
    case 1: return launch_mt<1, false, false, 1>(p, grid, pdl, dev, stream);
    case 2: return launch_mt<2, false, false, 1>(p, grid, pdl, dev, stream);
    case 4: return launch_mt<4, false, false, 1>(p, grid, pdl, dev, stream);
    case 8: return mma ? launch_mt<8, false, false, 1, true>(p, grid, pdl, dev, stream)
                       : launch_mt<8, false, false, 1>(p, grid, pdl, dev, stream);
    default: return launch_mt<16, false, false, 1, true>(p, grid, pdl, dev, stream);
  }
}

// Two tokens only: the 4- and 8-token instances (58 and 64 registers a
// thread) were faster on each projection alone but slower inside a block's
// chain of calls (BitNet-3B, eight layers: 42.0 -> 43.9 us a layer at M = 4,
// 63.9 -> 71.5 at M = 8, against 29.8 -> 28.6 at M = 2): beside them the next
// launch's CTAs no longer fit on the SM early.
bool decode_rows_fit(int64_t M, int64_t K) {
  return M == 2 && K > 0 && M * (K / 4) <= 3 * kDecThreads;  // 3 float4 a thread
}

cudaError_t launch_decode_rows(const float* x, int64_t M, int64_t K, const DecodeMatrix* mats, int nmats,
                               int8_t* xq_out, float* sx_out, bool gated, bool pdl, const DeviceInfo& dev,
                               cudaStream_t stream) {
  if (!decode_rows_fit(M, K)) return cudaErrorInvalidValue;
  DecodeParams p = {};
  p.x = x;
  p.xq_out = xq_out;
  p.sx_out = sx_out;
  p.status = dev.status;
  p.M = (int)M;
  const int grid = plan_decode(p, mats, nmats, K, 2, false, gated, dev);
  return launch_mt<2, true, false, 3>(p, grid, pdl, dev, stream);
}

cudaError_t launch_decode_fused(const float* x, const float* mul, const float* gamma, double eps, int64_t K,
                                const DecodeMatrix* mats, int nmats, int8_t* xq_out, float* sx_out,
                                bool gated, bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  if (K > (int64_t)kDecThreads * 4 * kMaxNJ) return cudaErrorInvalidValue;
  DecodeParams p = {};
  p.x = x;
  p.mul = mul;
  p.gamma = gamma;
  p.eps = eps;
  p.xq_out = xq_out;
  p.sx_out = sx_out;
  p.status = dev.status;
  p.M = 1;
  const bool norm = gamma != nullptr;
  const int grid = plan_decode(p, mats, nmats, K, 1, norm, gated, dev);
  // float4 elements of the row a thread owns (the kernel keeps them in registers)
  const int nj = (int)((K / 4 + kDecThreads - 1) / kDecThreads);
  return norm ? launch_fused<true>(p, grid, nj, pdl, dev, stream) : launch_fused<false>(p, grid, nj, pdl, dev, stream);
}

cudaError_t launch_wait_selftest(int64_t limit_ns, const DeviceInfo& dev, cudaStream_t stream) {
  wait_timeout_selftest<<<1, 32, 0, stream>>>(dev.status, (unsigned long long)limit_ns);
  return cudaGetLastError();
}

}  // namespace bitlinear
