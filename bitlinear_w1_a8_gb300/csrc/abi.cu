// abi.cu -- the extern "C" entry points: argument checks, device discovery and
// dispatch to the kernel launchers.  Nothing here allocates device memory.
#include <mutex>

#include "common.cuh"

namespace bitlinear {
// argmax.cu: index[m] = first n of the largest y[m, n], M rows of N floats.
cudaError_t launch_argmax(const float* y, int64_t M, int64_t N, int32_t* index, cudaStream_t stream);
// prefill.cu, 1 <= M <= 128: weight rows on the MMA's M side, tokens on its N side.
cudaError_t launch_batched(const int8_t* xq, const float* sx, int64_t M, const uint8_t* packed,
                           const float* sw, int64_t N, int64_t K, float* y, int32_t* acc,
                           bool pdl, const DeviceInfo& dev, cudaStream_t stream);
// prefill.cu: several matrices sharing xq (and K) in one launch of either kernel.
cudaError_t launch_prefill_mats(const int8_t* xq, const float* sx, int64_t M, const DecodeMatrix* mats, int nmats,
                                int64_t K, bool pdl, const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_batched_mats(const int8_t* xq, const float* sx, int64_t M, const DecodeMatrix* mats, int nmats,
                                int64_t K, bool pdl, const DeviceInfo& dev, cudaStream_t stream);
// wide.cu: activations widened once into `workspace`, 128 weight rows x up to
// 192 tokens per tile.
size_t wide_workspace_bytes(int64_t M, int64_t K);
cudaError_t launch_wide(const int8_t* xq, const float* sx, int64_t M, const uint8_t* packed, const float* sw,
                        int64_t N, int64_t K, float* y, int32_t* acc, void* workspace, bool widen, bool pdl,
                        const DeviceInfo& dev, cudaStream_t stream);
}  // namespace bitlinear

namespace bitlinear {
namespace {

// One status word per device: kernels record a timed-out bounded wait here.
__device__ int g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
DeviceInfo g_devs[kMaxDevices];
bool g_dev_ready[kMaxDevices] = {};

bitlinear_status current_device(DeviceInfo* out) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return BITLINEAR_ERR_CUDA;
  if (d < 0 || d >= kMaxDevices) return BITLINEAR_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (!g_dev_ready[d]) {
    DeviceInfo info = {};
    info.device = d;
    int smem = 0, smem_sm = 0;
    if (cudaDeviceGetAttribute(&info.num_sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&info.cc_major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&info.cc_minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, d) != cudaSuccess) {
      return BITLINEAR_ERR_CUDA;
    }
    info.smem_optin = (size_t)smem;
    info.smem_per_sm = (size_t)smem_sm;
    // The kernels are built for sm_103a only.
    if (info.cc_major != 10 || info.cc_minor != 3) return BITLINEAR_ERR_UNSUPPORTED;
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return BITLINEAR_ERR_CUDA;
    info.status = static_cast<int*>(addr);
    g_devs[d] = info;
    g_dev_ready[d] = true;
  }
  *out = g_devs[d];
  return BITLINEAR_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bitlinear_status from_cuda(cudaError_t e) { return e == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA; }

constexpr int64_t kMaxDim = (int64_t)1 << 30;
// Decode kernel: activations of a token group are staged in shared memory.
constexpr int64_t kDecodeMaxK = 65536;
// Tensor-core kernel: the fp32 accumulator is exact while 127 * K < 2^24.
constexpr int64_t kPrefillMaxK = 131072;
// AUTO, from timings on GB300 over the BitNet-3B shapes (back-to-back calls
// and a layer's chain of calls):
//  * the decode kernel for up to 16 tokens (K <= 32768; up to 8 tokens at
//    longer K): dp4a in token groups of up to 4, the warp-level MMA in groups
//    of 8 or 16 (K split over a cluster where a group's activations would
//    exceed 64 KB);
//  * the batched tensor-core kernel (weight rows on the MMA's M side, all
//    tokens in one tile) for outputs up to 8192 rows up to M = 128;
//  * the tensor-core kernel with 128-token tiles otherwise (both tensor-core
//    kernels split K over the CTAs of a cluster when their tiles fill less
//    than half the SMs).
int auto_algo(int64_t M, int64_t N, int64_t K) {
  if (M <= 4 && K <= 65536) return BITLINEAR_ALGO_DECODE;
  // Measured on GB300 (BitNet-3B projections, back-to-back calls, us a call,
  // decode / batched / 128-token tiles): from 5 tokens the decode kernel runs
  // its dots on the warp-level MMA in 8- or 16-token groups (at long K split
  // over a cluster) and wins up to 16 tokens, the very wide LM head included
  // (10240 x 2560 at M = 16: 7.8 / 20.4 / 22.2; 2560 x 10240: 14.0 / 14.4 /
  // 22.1; 50000 x 2560 at M = 12 / 16: 31.7 / 32.9 against 45.9 / 44.5 on
  // 128-token tiles; eight BitNet-3B layers of calls at M = 12 / 16: 55.9 /
  // 57.4 -> 54.1 / 56.2 us a layer with the long-K calls on decode too).
  // Beyond, the batched tensor-core kernel
  // (weight rows on the MMA's M side, K split inside a cluster) wins up to 64
  // column tiles, and the 128-token-tile kernel on wider outputs (M = 32:
  // q||k||v 13.0 vs 18.8, o 8.4 vs 12.3, down 15.3 vs 22.3; 10240 x 2560
  // 19.6 vs 20.5 batched, 14.8 decode -- slower inside a layer's chain).
  if (M <= 16 && K <= 32768) return BITLINEAR_ALGO_DECODE;
  if (N >= 32768 || K > 131072) return BITLINEAR_ALGO_PREFILL;
  if (M <= 8 && K <= 65536) return BITLINEAR_ALGO_DECODE;
  if (M <= 128 && N <= 8192) return BITLINEAR_ALGO_BATCHED;
  return BITLINEAR_ALGO_PREFILL;
}

// With a workspace, AUTO takes the WIDE kernel for narrow outputs at medium
// token counts above the batched kernel's range, where it measured faster on
// GB300 than the 128-token-tile kernel (pre-pass included, back to back; us
// per call, 128-token tiles / WIDE):
//   N = 2048, K = 8192:   M = 256 37.2 / 20.1, M = 512 38.1 / 33.2, M = 1024 48.3 / 52.7
//   N = 2560, K = 10240:  M = 256 32.9 / 34.5, M = 512 49.3 / 41.4, M = 1024 61.2 / 65.0
//   N = K = 2560:         M = 256 17.6 / 17.5, M = 512 19.2 / 23.3
//   N = 1000, K = 4096, M = 200: 14.4 / 12.7;  N = K = 4096, M = 384: 28.8 / 29.4
// and for wide outputs (N = 8192, 10240) and at M = 2048 the other kernels
// measured faster.  Up to M = 128 the batched kernel (K split inside a
// cluster) is within a few per cent of WIDE without the pre-pass launch
// (BitNet-3B o / down at M = 64: 10.1 / 17.4 us against 10.7 / 17.9).  In a
// layer's chain of calls WIDE pays only at long K: with q, k, v and o
// (K = 2560) on it too, eight BitNet-3B layers took 126.0 / 133.3 / 155.7 us
// a layer at M = 160 / 192 / 256, and 111.6 / 113.4 / 126.7 with down alone
// on it (unchanged at M = 384 / 512, where only down qualified).  So: up to
// 512 tokens at K >= 8192.
bool wide_wins(int64_t M, int64_t N, int64_t K) {
  if (N > 4096 || M <= 128) return false;
  return K >= 8192 && M <= 512;
}

// bitlinear_linear's single-launch path: the row quantiser keeps K fp32 values
// in shared memory next to the weights.
constexpr int64_t kFusedMaxK = 16384;

// The decode grid's height (token groups) stays within the launch limit.
bool decode_grid_ok(int64_t M, int64_t K) {
  bool mma = false;
  int ks = 1;
  const int64_t group = decode_token_group(M, K, &mma, &ks);
  return (M + group - 1) / group <= 65535;
}

bitlinear_status check_nk(int64_t N, int64_t K) {
  if (N <= 0 || K <= 0 || N > kMaxDim || K > kMaxDim) return BITLINEAR_ERR_SHAPE;
  if (K % 64 != 0) return BITLINEAR_ERR_SHAPE;
  if (N * K >= ((int64_t)1 << 40)) return BITLINEAR_ERR_SHAPE;
  return BITLINEAR_OK;
}

}  // namespace
}  // namespace bitlinear

using namespace bitlinear;

extern "C" {

int bitlinear_abi_version(void) { return 1; }

const char* bitlinear_status_string(bitlinear_status s) {
  switch (s) {
    case BITLINEAR_OK: return "BITLINEAR_OK";
    case BITLINEAR_ERR_NULL: return "BITLINEAR_ERR_NULL: a required pointer is NULL";
    case BITLINEAR_ERR_SHAPE: return "BITLINEAR_ERR_SHAPE: invalid M, N or K";
    case BITLINEAR_ERR_ALIGN: return "BITLINEAR_ERR_ALIGN: a pointer is not 16-byte aligned";
    case BITLINEAR_ERR_UNSUPPORTED: return "BITLINEAR_ERR_UNSUPPORTED: unsupported device, algorithm or flag";
    case BITLINEAR_ERR_CUDA: return "BITLINEAR_ERR_CUDA: a CUDA call failed";
    case BITLINEAR_ERR_TIMEOUT: return "BITLINEAR_ERR_TIMEOUT: a bounded wait in a kernel ran out";
    case BITLINEAR_ERR_WORKSPACE: return "BITLINEAR_ERR_WORKSPACE: workspace missing or too small";
    default: return "BITLINEAR_ERR_UNKNOWN";
  }
}

size_t bitlinear_packed_bytes(int64_t N, int64_t K) {
  if (N <= 0 || K <= 0) return 0;
  return (size_t)N * (size_t)((K + 63) / 64) * 16u;
}

size_t bitlinear_quantize_weights_workspace(int64_t N, int64_t K) {
  (void)N;
  (void)K;
  return 4096;
}

bitlinear_status bitlinear_quantize_weights(const float* W, int64_t N, int64_t K, uint8_t* packed,
                                            float* w_scale, void* workspace, size_t workspace_bytes,
                                            void* stream) {
  if (!W || !packed || !w_scale) return BITLINEAR_ERR_NULL;
  bitlinear_status st = check_nk(N, K);
  if (st != BITLINEAR_OK) return st;
  if (!workspace || workspace_bytes < bitlinear_quantize_weights_workspace(N, K))
    return BITLINEAR_ERR_WORKSPACE;
  if (!aligned16(W) || !aligned16(packed) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(w_scale) & 3u))
    return BITLINEAR_ERR_ALIGN;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != BITLINEAR_OK) return st;
  return from_cuda(launch_weight_quant(W, N, K, packed, w_scale,
                                       static_cast<unsigned long long*>(workspace), dev,
                                       static_cast<cudaStream_t>(stream)));
}

bitlinear_status bitlinear_quant_act(const float* x, const float* mul, int64_t M, int64_t K,
                                     const float* rms_weight, double rms_eps, int8_t* xq,
                                     float* x_scale, void* stream) {
  if (M < 0 || M > kMaxDim || K <= 0 || K % 64 != 0 || K > 32768) return BITLINEAR_ERR_SHAPE;
  if (rms_weight && !(rms_eps >= 0.0)) return BITLINEAR_ERR_SHAPE;
  if (M == 0) return BITLINEAR_OK;  // empty batch: the M-sized buffers may be NULL
  if (!x || !xq || !x_scale) return BITLINEAR_ERR_NULL;
  if (!aligned16(x) || !aligned16(xq) || (mul && !aligned16(mul)) ||
      (rms_weight && !aligned16(rms_weight)) || (reinterpret_cast<uintptr_t>(x_scale) & 3u))
    return BITLINEAR_ERR_ALIGN;
  DeviceInfo dev;
  bitlinear_status st = current_device(&dev);
  if (st != BITLINEAR_OK) return st;
  return from_cuda(launch_act_quant(x, mul, M, K, rms_weight, rms_eps, xq, x_scale, dev,
                                    static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

bitlinear_status forward_impl(const int8_t* xq, const float* x_scale, int64_t M, const uint8_t* packed,
                              const float* w_scale, int64_t N, int64_t K, float* y, int32_t* acc, int algo,
                              int flags, void* workspace, size_t workspace_bytes, void* stream) {
  if (!packed || !w_scale) return BITLINEAR_ERR_NULL;
  bitlinear_status st = check_nk(N, K);
  if (st != BITLINEAR_OK) return st;
  if (M < 0 || M > kMaxDim) return BITLINEAR_ERR_SHAPE;
  // y holds M * N floats; below 2^40 every tile and work-unit count of the
  // kernels fits in 32 bits.
  if (M * N >= ((int64_t)1 << 40)) return BITLINEAR_ERR_SHAPE;
  if (flags & ~BITLINEAR_FLAG_PDL) return BITLINEAR_ERR_UNSUPPORTED;
  if (algo != BITLINEAR_ALGO_AUTO && algo != BITLINEAR_ALGO_DECODE && algo != BITLINEAR_ALGO_PREFILL &&
      algo != BITLINEAR_ALGO_BATCHED && algo != BITLINEAR_ALGO_WIDE)
    return BITLINEAR_ERR_UNSUPPORTED;
  // the WIDE pre-pass indexes the 16-byte chunks of a k-block plane (8 per row) in 32 bits
  if (algo == BITLINEAR_ALGO_WIDE && (M + 15) / 16 * 16 * 8 > (int64_t)0x7fffffff) return BITLINEAR_ERR_UNSUPPORTED;
  if (M == 0) return BITLINEAR_OK;  // empty batch: the M-sized buffers may be NULL
  if (!xq || !x_scale || !y) return BITLINEAR_ERR_NULL;
  if (!aligned16(xq) || !aligned16(packed) || !aligned16(y) || (acc && !aligned16(acc)) ||
      (reinterpret_cast<uintptr_t>(x_scale) & 3u) || (reinterpret_cast<uintptr_t>(w_scale) & 3u))
    return BITLINEAR_ERR_ALIGN;
  const bool have_ws = workspace && workspace_bytes >= wide_workspace_bytes(M, K);
  if (algo == BITLINEAR_ALGO_WIDE && !have_ws) return BITLINEAR_ERR_WORKSPACE;
  if (have_ws && !aligned16(workspace)) return BITLINEAR_ERR_ALIGN;
  int use = algo;
  if (use == BITLINEAR_ALGO_AUTO) {
    use = auto_algo(M, N, K);
    if (use != BITLINEAR_ALGO_DECODE && have_ws && K <= kPrefillMaxK && wide_wins(M, N, K)) use = BITLINEAR_ALGO_WIDE;
  }
  if (use == BITLINEAR_ALGO_DECODE && (K > kDecodeMaxK || !decode_grid_ok(M, K)))
    return BITLINEAR_ERR_UNSUPPORTED;
  if ((use == BITLINEAR_ALGO_PREFILL || use == BITLINEAR_ALGO_WIDE) && K > kPrefillMaxK)
    return BITLINEAR_ERR_UNSUPPORTED;
  if (use == BITLINEAR_ALGO_BATCHED && (K > kPrefillMaxK || M > 128)) return BITLINEAR_ERR_UNSUPPORTED;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != BITLINEAR_OK) return st;
  const bool pdl = (flags & BITLINEAR_FLAG_PDL) != 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (use == BITLINEAR_ALGO_WIDE)
    return from_cuda(launch_wide(xq, x_scale, M, packed, w_scale, N, K, y, acc, workspace, true, pdl, dev, s));
  if (use == BITLINEAR_ALGO_BATCHED)
    return from_cuda(launch_batched(xq, x_scale, M, packed, w_scale, N, K, y, acc, pdl, dev, s));
  if (use == BITLINEAR_ALGO_DECODE) {
    const DecodeMatrix mat = {packed, w_scale, N, y, acc};
    return from_cuda(launch_decode(xq, x_scale, M, &mat, 1, K, false, pdl, dev, s));
  }
  return from_cuda(launch_prefill(xq, x_scale, M, packed, w_scale, N, K, y, acc, pdl, dev, s));
}

}  // namespace

extern "C" {

bitlinear_status bitlinear_forward_ex(const int8_t* xq, const float* x_scale, int64_t M,
                                      const uint8_t* packed, const float* w_scale, int64_t N,
                                      int64_t K, float* y, int32_t* acc, int algo, int flags,
                                      void* stream) {
  return forward_impl(xq, x_scale, M, packed, w_scale, N, K, y, acc, algo, flags, nullptr, 0, stream);
}

size_t bitlinear_forward_workspace(int64_t M, int64_t K) {
  if (M <= 0 || K <= 0 || M > kMaxDim || K > kMaxDim) return 0;
  return wide_workspace_bytes(M, K);
}

bitlinear_status bitlinear_forward_ws(const int8_t* xq, const float* x_scale, int64_t M,
                                      const uint8_t* packed, const float* w_scale, int64_t N,
                                      int64_t K, float* y, int32_t* acc, int algo, int flags,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  return forward_impl(xq, x_scale, M, packed, w_scale, N, K, y, acc, algo, flags, workspace, workspace_bytes,
                      stream);
}

}  // extern "C"

namespace {

bitlinear_status linear_impl(const float* x, const float* mul, int64_t M, int64_t K, const float* rms_weight,
                             double rms_eps, const bitlinear_weight* weights, int num_weights, int8_t* xq,
                             float* x_scale, int flags, void* workspace, size_t workspace_bytes, void* stream) {
  if (!weights) return BITLINEAR_ERR_NULL;
  if (num_weights < 1 || num_weights > kMaxDecodeMats) return BITLINEAR_ERR_SHAPE;
  if (M < 0 || M > kMaxDim || K <= 0 || K % 64 != 0 || K > 32768) return BITLINEAR_ERR_SHAPE;
  if (rms_weight && !(rms_eps >= 0.0)) return BITLINEAR_ERR_SHAPE;
  if (flags & ~(BITLINEAR_FLAG_PDL | BITLINEAR_FLAG_GATED)) return BITLINEAR_ERR_UNSUPPORTED;
  const bool gated = (flags & BITLINEAR_FLAG_GATED) != 0;
  if (gated && (num_weights != 2 || weights[0].N != weights[1].N)) return BITLINEAR_ERR_SHAPE;
  for (int i = 0; i < num_weights; ++i) {
    const bitlinear_weight& w = weights[i];
    if (!w.packed || !w.w_scale) return BITLINEAR_ERR_NULL;
    const bitlinear_status st = check_nk(w.N, K);
    if (st != BITLINEAR_OK) return st;
    if (M * w.N >= ((int64_t)1 << 40)) return BITLINEAR_ERR_SHAPE;  // as bitlinear_forward
    if (!aligned16(w.packed) || (reinterpret_cast<uintptr_t>(w.w_scale) & 3u)) return BITLINEAR_ERR_ALIGN;
  }
  if (M == 0) return BITLINEAR_OK;  // empty batch: the M-sized buffers may be NULL
  if (!x || !xq || !x_scale) return BITLINEAR_ERR_NULL;
  if (!aligned16(x) || !aligned16(xq) || (mul && !aligned16(mul)) || (rms_weight && !aligned16(rms_weight)) ||
      (reinterpret_cast<uintptr_t>(x_scale) & 3u))
    return BITLINEAR_ERR_ALIGN;
  for (int i = 0; i < num_weights; ++i) {
    if (!weights[i].y) return BITLINEAR_ERR_NULL;
    if (!aligned16(weights[i].y) || (weights[i].acc && !aligned16(weights[i].acc))) return BITLINEAR_ERR_ALIGN;
  }
  if (workspace && workspace_bytes < wide_workspace_bytes(M, K)) return BITLINEAR_ERR_WORKSPACE;
  if (workspace && !aligned16(workspace)) return BITLINEAR_ERR_ALIGN;
  const bool have_ws = workspace != nullptr && (M + 15) / 16 * 16 * 8 <= (int64_t)0x7fffffff;
  DeviceInfo dev;
  bitlinear_status st = current_device(&dev);
  if (st != BITLINEAR_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool pdl = (flags & BITLINEAR_FLAG_PDL) != 0;
  DecodeMatrix mats[kMaxDecodeMats];
  for (int i = 0; i < num_weights; ++i)
    mats[i] = DecodeMatrix{weights[i].packed, weights[i].w_scale, weights[i].N, weights[i].y, weights[i].acc};
  if (M == 1 && K <= kFusedMaxK) {
    // one launch: every CTA quantises the token itself
    return from_cuda(launch_decode_fused(x, mul, rms_weight, rms_eps, K, mats, num_weights, xq, x_scale, gated,
                                         pdl, dev, s));
  }
  if (!mul && !rms_weight && decode_rows_fit(M, K)) {
    // Two tokens without a prologue, every matrix on the decode kernel: one
    // launch again, every CTA quantising the token rows itself -- when each
    // CTA's weight rows (about all rows / SMs) outnumber 4 M, i.e. its dots
    // outweigh loading the fp32 rows
    bool all_decode = true;
    int64_t rows = 0;
    for (int i = 0; i < num_weights; ++i) {
      all_decode = all_decode && auto_algo(M, mats[i].N, K) == BITLINEAR_ALGO_DECODE;
      rows += mats[i].N;
    }
    if (all_decode && rows >= 4 * M * dev.num_sms)
      return from_cuda(launch_decode_rows(x, M, K, mats, num_weights, xq, x_scale, gated, pdl, dev, s));
  }
  cudaError_t err = launch_act_quant(x, mul, M, K, rms_weight, rms_eps, xq, x_scale, dev, s, pdl);
  if (err != cudaSuccess) return BITLINEAR_ERR_CUDA;
  // The matrices that take the same kernel share one launch of it (WIDE, with
  // its per-matrix pre-pass bookkeeping, takes one launch each).
  DecodeMatrix dec[kMaxDecodeMats], bat[kMaxDecodeMats], pre[kMaxDecodeMats];
  int ndec = 0, nbat = 0, npre = 0;
  bool widened = false;  // the workspace holds this call's xq once a WIDE launch has widened it
  for (int i = 0; i < num_weights; ++i) {
    const int algo = auto_algo(M, mats[i].N, K);
    if (algo == BITLINEAR_ALGO_DECODE) {
      dec[ndec++] = mats[i];
    } else if (have_ws && wide_wins(M, mats[i].N, K)) {
      err = launch_wide(xq, x_scale, M, mats[i].packed, mats[i].w_scale, mats[i].N, K, mats[i].y, mats[i].acc,
                        workspace, !widened, pdl, dev, s);
      if (err != cudaSuccess) return BITLINEAR_ERR_CUDA;
      widened = true;
    } else if (algo == BITLINEAR_ALGO_BATCHED) {
      bat[nbat++] = mats[i];
    } else {
      pre[npre++] = mats[i];
    }
  }
  // A gated pair that the decode kernel takes is gated in its epilogue; on
  // any other kernel one elementwise launch follows.
  const bool gate_in_decode = gated && ndec == 2;
  if (ndec > 0) {
    if (!decode_grid_ok(M, K)) return BITLINEAR_ERR_UNSUPPORTED;
    err = launch_decode(xq, x_scale, M, dec, ndec, K, gate_in_decode, pdl, dev, s);
    if (err != cudaSuccess) return BITLINEAR_ERR_CUDA;
  }
  if (nbat > 0) {
    err = launch_batched_mats(xq, x_scale, M, bat, nbat, K, pdl, dev, s);
    if (err != cudaSuccess) return BITLINEAR_ERR_CUDA;
  }
  if (npre > 0) {
    err = launch_prefill_mats(xq, x_scale, M, pre, npre, K, pdl, dev, s);
    if (err != cudaSuccess) return BITLINEAR_ERR_CUDA;
  }
  if (gated && !gate_in_decode) {
    err = launch_gate(mats[0].y, mats[1].y, M * mats[0].N, pdl, dev, s);
    if (err != cudaSuccess) return BITLINEAR_ERR_CUDA;
  }
  return BITLINEAR_OK;
}

}  // namespace

extern "C" {

bitlinear_status bitlinear_linear(const float* x, const float* mul, int64_t M, int64_t K,
                                  const float* rms_weight, double rms_eps, const bitlinear_weight* weights,
                                  int num_weights, int8_t* xq, float* x_scale, int flags, void* stream) {
  return linear_impl(x, mul, M, K, rms_weight, rms_eps, weights, num_weights, xq, x_scale, flags, nullptr, 0,
                     stream);
}

bitlinear_status bitlinear_linear_ws(const float* x, const float* mul, int64_t M, int64_t K,
                                     const float* rms_weight, double rms_eps, const bitlinear_weight* weights,
                                     int num_weights, int8_t* xq, float* x_scale, int flags, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  return linear_impl(x, mul, M, K, rms_weight, rms_eps, weights, num_weights, xq, x_scale, flags, workspace,
                     workspace_bytes, stream);
}



bitlinear_status bitlinear_argmax(const float* y, int64_t M, int64_t N, int32_t* index, void* stream) {
  if (M < 0 || M > kMaxDim || N <= 0 || N > 0x7fffffffLL) return BITLINEAR_ERR_SHAPE;
  if (M == 0) return BITLINEAR_OK;
  if (!y || !index) return BITLINEAR_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(y) & 3u) || (reinterpret_cast<uintptr_t>(index) & 3u)) return BITLINEAR_ERR_ALIGN;
  DeviceInfo dev;
  const bitlinear_status st = current_device(&dev);
  if (st != BITLINEAR_OK) return st;
  return from_cuda(launch_argmax(y, M, N, index, static_cast<cudaStream_t>(stream)));
}

bitlinear_status bitlinear_forward(const int8_t* xq, const float* x_scale, int64_t M,
                                   const uint8_t* packed, const float* w_scale, int64_t N,
                                   int64_t K, float* y, int32_t* acc, void* stream) {
  return bitlinear_forward_ex(xq, x_scale, M, packed, w_scale, N, K, y, acc,
                              BITLINEAR_ALGO_AUTO, 0, stream);
}

// ---------------------------------------------------------------------------
// bitlinear_quantize_weights_noalloc: the weight_quant scratch (bucket sums)
// lives in this file-scope device array instead of a caller workspace.  Host
// code may not pass the symbol itself to a kernel (on the host it names a
// shadow, not device memory): its device address is looked up once per device
// with cudaGetSymbolAddress and that pointer is passed on.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[BITLINEAR_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

bitlinear_status noalloc_scratch(int device, void** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[device]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return BITLINEAR_ERR_CUDA;
    g_noalloc_ptr[device] = ptr;
  }
  *out = g_noalloc_ptr[device];
  return BITLINEAR_OK;
}
}  // namespace

bitlinear_status bitlinear_quantize_weights_noalloc(const float* W, int64_t N, int64_t K, uint8_t* packed,
                                                    float* w_scale, void* stream) {
  if (!W || !packed || !w_scale) return BITLINEAR_ERR_NULL;
  bitlinear_status st = check_nk(N, K);
  if (st != BITLINEAR_OK) return st;
  if (bitlinear_quantize_weights_workspace(N, K) > sizeof(g_noalloc_scratch)) return BITLINEAR_ERR_WORKSPACE;
  if (!aligned16(W) || !aligned16(packed) || (reinterpret_cast<uintptr_t>(w_scale) & 3u))
    return BITLINEAR_ERR_ALIGN;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != BITLINEAR_OK) return st;
  void* scratch = nullptr;
  st = noalloc_scratch(dev.device, &scratch);
  if (st != BITLINEAR_OK) return st;
  return from_cuda(launch_weight_quant(W, N, K, packed, w_scale, static_cast<unsigned long long*>(scratch),
                                       dev, static_cast<cudaStream_t>(stream)));
}

bitlinear_status bitlinear_selftest_wait_timeout(int64_t limit_ns, void* stream) {
  if (limit_ns <= 0 || limit_ns > 1000000000ll) return BITLINEAR_ERR_SHAPE;
  DeviceInfo dev;
  bitlinear_status st = current_device(&dev);
  if (st != BITLINEAR_OK) return st;
  return from_cuda(launch_wait_selftest(limit_ns, dev, static_cast<cudaStream_t>(stream)));
}

bitlinear_status bitlinear_device_status(void* stream, int clear) {
  DeviceInfo dev;
  bitlinear_status st = current_device(&dev);
  if (st != BITLINEAR_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return BITLINEAR_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, dev.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return BITLINEAR_ERR_CUDA;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpy(dev.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return BITLINEAR_ERR_CUDA;
  }
  return word != 0 ? BITLINEAR_ERR_TIMEOUT : BITLINEAR_OK;
}

}  // extern "C"
