/*
 * bitlinear.h -- C ABI of the GB300 (sm_103a) BitLinear W1.58A8 library.
 *
 * BitLinear is the layer that replaces every nn.Linear of a BitNet b1.58
 * transformer (q, k, v, o and the FFN gate, up, down projections; "Add
 * Support for BitNet Architecture Inference", Candle PR, list of changes made:
 * "Replace Linear with BitLinear in MLP and Attention", with an RMSNorm before
 * each BitLinear and the activation_quant / weight_quant pair of the BitNet
 * paper).  The layer computes
 *
 *   weight_quant (absmean, once per matrix, offline):
 *       sw = 1 / max(mean|W|, 1e-5),   Wq = clamp(round_half_even(W*sw), -1, 1)
 *   activation_quant (absmax, per token row):
 *       sx = 127 / max(max_k |x|, 1e-5), xq = clamp(round_half_even(x*sx), -128, 127)
 *   contraction and rescale:
 *       acc[m,n] = sum_k xq[m,k] * Wq[n,k]   (exact int32)
 *       y[m,n]   = acc[m,n] / (sx[m] * sw)   (fp32: one product, one division)
 *
 * Shapes: W is [N, K] fp32 row-major (out features x in features), x is
 * [M, K] fp32 row-major (M tokens), y is [M, N] fp32 row-major.
 *
 * Conventions shared by every entry point:
 *  - All pointers named "device" are CUDA device pointers on the current
 *    device; the caller allocates and owns every buffer.  No entry point keeps
 *    a pointer after it returns.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *    only enqueues work: results are ready when the stream reaches them.
 *  - Argument errors are reported synchronously, before anything is enqueued:
 *    a NULL required pointer, a non-positive N or K, a negative M, K not a
 *    multiple of 64, M * N >= 2^40 or N * K >= 2^40, a pointer not aligned to
 *    16 bytes, or a too small workspace.  M == 0 is a valid empty batch and enqueues nothing.
 *  - A failed launch returns BITLINEAR_ERR_CUDA.  Every wait inside a kernel
 *    is bounded; a wait that runs out records BITLINEAR_ERR_TIMEOUT in a
 *    per-device status word that bitlinear_device_status() reports, and that
 *    launch's outputs are unspecified.  While that word is set, a
 *    decode launch whose K is split over a thread-block cluster writes no
 *    outputs at all (its CTAs learn of a peer's timeout through the word), so
 *    clear it before relying on results again.
 *  - Non-finite inputs (Inf, NaN) give unspecified outputs.
 *  - Rounding: every quantisation decision is taken in IEEE fp32 with
 *    round-to-nearest-even and no fused multiply-add; the sums that feed the
 *    scales (sum|W| and the RMSNorm sum of squares) are exact, then rounded
 *    once to fp64, so results do not depend on launch shape or timing.
 *
 * Packed weight layout (this library's own 2-bit format; 0.25 byte per
 * weight, the figure of the pages' memory tables):
 *  - code = Wq + 1 in {0, 1, 2}; code 3 never occurs; weights past K (none
 *    while K % 64 == 0) would hold code 1.
 *  - The 16-byte chunk of row n and k-block kb = k / 64 starts at byte
 *    (kb * N + n) * 16, so one k-block of all rows is contiguous.
 *  - Inside a chunk, little-endian 32-bit word w = (k % 64) / 16 holds
 *    i = k % 16 at bit 8*(i%4) + 2*(i/4): (word >> 2j) & 0x03030303 gives the
 *    codes of k = 16w+4j .. 16w+4j+3 in bytes 0..3.
 */
#ifndef BITLINEAR_H
#define BITLINEAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int bitlinear_status;

enum {
  BITLINEAR_OK = 0,
  BITLINEAR_ERR_NULL = -1,        /* a required pointer is NULL */
  BITLINEAR_ERR_SHAPE = -2,       /* N or K <= 0, M < 0, K % 64 != 0, size overflow */
  BITLINEAR_ERR_ALIGN = -3,       /* a pointer is not 16-byte aligned */
  BITLINEAR_ERR_UNSUPPORTED = -4, /* no sm_103 device, or an unknown algorithm / flag */
  BITLINEAR_ERR_CUDA = -5,        /* a CUDA runtime call or a launch failed */
  BITLINEAR_ERR_TIMEOUT = -6,     /* a bounded wait inside a kernel ran out */
  BITLINEAR_ERR_WORKSPACE = -7    /* workspace NULL or smaller than required */
};

/* Version of this ABI (increments on any incompatible change). */
int bitlinear_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* bitlinear_status_string(bitlinear_status status);

/* Bytes of the packed layout for an [N, K] matrix: N * ceil(K/64) * 16
 * (0 if N or K is not positive). */
size_t bitlinear_packed_bytes(int64_t N, int64_t K);

/* Workspace bytes bitlinear_quantize_weights needs (a constant 4096 today:
 * 256 per-exponent bucket sums of 8 bytes, plus room). */
size_t bitlinear_quantize_weights_workspace(int64_t N, int64_t K);

/*
 * weight_quant + pack (absmean ternary quantiser; one fp32 scale per matrix).
 * The weight_quant of the BitNet paper that the Candle PR ("Add Support for
 * BitNet Architecture Inference", the answer listing the changes made) names
 * for every BitLinear; the 2-bit codes give the 0.25 byte per weight of the
 * per-layer weight table ("Transformer Block" page, section "Memory Layout")
 * and of the model footprint ("Hesper.Models.BitNet" page, section "Memory
 * Footprint (BitNet-3B with TQ2_0)").
 *   W          device, fp32 [N, K] row-major, read only.
 *   N, K       N > 0, K > 0, K % 64 == 0, N*K < 2^40.
 *   packed     device, bitlinear_packed_bytes(N, K) bytes, written.
 *   w_scale    device, 1 fp32, receives sw = 1 / max(mean|W|, 1e-5).
 *   workspace  device, >= bitlinear_quantize_weights_workspace(N, K) bytes,
 *              16-byte aligned; its contents on entry do not matter and are
 *              overwritten (it is cleared on the stream first).
 * Three kernels: an exact per-exponent sum of |W|, a one-warp finalisation of
 * mean and sw, and the quantise-and-pack pass.
 */
bitlinear_status bitlinear_quantize_weights(const float* W, int64_t N, int64_t K,
                                            uint8_t* packed, float* w_scale,
                                            void* workspace, size_t workspace_bytes,
                                            void* stream);

/*
 * activation_quant with optional fused prologues, one kernel, one CTA per row.
 * The activation_quant of the BitNet paper named in the Candle PR's list of
 * changes (per-token absmax to int8), after the RMSNorm that sits before
 * every BitLinear there.
 * rms_eps is a double: the norm's mean square S/K + eps is formed in fp64
 * from the exact sum of squares, and a double keeps the caller's epsilon
 * exactly as given (1e-6 is not a float value; a float parameter would add
 * its rounding to every call).
 *   x           device, fp32 [M, K] row-major.
 *   mul         device fp32 [M, K] or NULL.  When given, the row fed to the
 *               quantiser is h = (r*r)*mul with r = max(x, 0) (the ReLU^2
 *               gating of the BitNet FFN, "Transformer Block" page, section
 *               "Feed-Forward Network"); x is then the gate projection.
 *   rms_weight  device fp32 [K] (gamma) or NULL.  When given, h is first
 *               normalised: inv = 1/sqrt(sum_k h_k^2 / K + rms_eps) computed in
 *               fp64 from the exact sum, rounded to fp32, then
 *               h_k = (h_k * inv) * gamma_k in fp32 (an RMSNorm before the
 *               BitLinear; the gating, when present, comes first).
 *   rms_eps     the RMSNorm epsilon (ignored without rms_weight), >= 0.
 *   xq          device, int8 [M, K] row-major, written.
 *   x_scale     device, fp32 [M], receives sx per row.
 * K % 64 == 0 and K <= 32768 (the row is staged in shared memory as fp32).
 */
bitlinear_status bitlinear_quant_act(const float* x, const float* mul, int64_t M, int64_t K,
                                     const float* rms_weight, double rms_eps,
                                     int8_t* xq, float* x_scale, void* stream);

/*
 * Contraction + rescale: y = (xq . Wq^T) / (sx * sw).
 * The BitLinear matmul that replaces every Linear of the attention and the
 * MLP (Candle PR "Add Support for BitNet Architecture Inference", the answer
 * listing the changes made): int8 activations times ternary weights with
 * exact integer accumulation, then one rescale by both quantisation scales.
 * At M = 1 it is the per-token work that dominates decoding ("Hesper.Models.
 * BitNet" page, section "Performance (BitNet-3B on A100)": the 32 layers take
 * 870 of 883 ms per token).
 *   xq, x_scale   device, from bitlinear_quant_act (int8 [M, K], fp32 [M]).
 *   packed, w_scale  device, from bitlinear_quantize_weights for [N, K].
 *   y             device, fp32 [M, N] row-major, written.
 *   acc           device int32 [M, N] or NULL; when given it receives the raw
 *                 integer accumulators (for checking and debugging).
 * The kernel is chosen from M, N and K (BITLINEAR_ALGO_AUTO): the decode
 * kernel (packed weights bulk-copied into shared memory; K <= 65536; dp4a on
 * the 2-bit codes for token groups of up to 4, the warp-level fp16 MMA for
 * groups of 8 or 16 tokens, with K split over a cluster of 2-8 CTAs when the
 * group's activations would exceed 64 KB of shared memory) for M <= 16 when
 * K <= 32768, and for M <= 8 when N < 32768; the
 * batched tcgen05 kernel (128 weight rows per tile on the
 * MMA's M side, all tokens on its N side) for N <= 8192 and M <= 128; the
 * tcgen05 kernel with 128-token tiles (K <= 131072) otherwise.  Both
 * tensor-core kernels split K over up to 8 CTAs when their tiles fill less
 * than half of the SMs; the CTAs of a tile form one thread-block cluster and
 * add their partial sums through distributed shared memory (one launch).
 */
bitlinear_status bitlinear_forward(const int8_t* xq, const float* x_scale, int64_t M,
                                   const uint8_t* packed, const float* w_scale,
                                   int64_t N, int64_t K, float* y, int32_t* acc,
                                   void* stream);

enum {
  BITLINEAR_ALGO_AUTO = 0,
  BITLINEAR_ALGO_DECODE = 1,   /* the decode kernel (dp4a; the warp-level MMA for
                                  8- or 16-token groups), K <= 65536, at most
                                  65535 token groups (16 tokens a group, fewer
                                  where 16 tokens of activations do not fit) */
  BITLINEAR_ALGO_PREFILL = 2,  /* tcgen05 kernel, any M: 128-token tiles */
  BITLINEAR_ALGO_BATCHED = 3,  /* tcgen05 kernel, 1 <= M <= 128: 128-row weight
                                  tiles with every token in one tile */
  BITLINEAR_ALGO_WIDE = 4      /* tcgen05 kernel, any M, bitlinear_forward_ws only:
                                  the activations widened once to fp16 in the
                                  workspace, 128-row weight tiles x up to 192
                                  tokens */
};

enum {
  /* Launch with programmatic dependent launch: the kernel starts streaming
   * the packed weights while the previous kernel on the stream (normally the
   * bitlinear_quant_act that produced xq) is still running, and waits for it
   * before touching xq / x_scale and before writing y / acc.  Every kernel of
   * this library lets the next one start this way as soon as all of its CTAs
   * are running, so in a chain of calls with this flag several launches can
   * be copying weights at once.  Only valid when `packed` and `w_scale` were
   * written before the chain began: not by the kernel immediately before on
   * the stream, nor by any kernel between it and the last launch made
   * without this flag. */
  BITLINEAR_FLAG_PDL = 1,
  /* bitlinear_linear / bitlinear_linear_ws only: the two matrices are an FFN
   * gate and up projection of equal N ("Hesper.Layers.TransformerBlock" page,
   * section "Forward Pass", FFN sub-layer: hidden = ReLU^2(gate) x up, which
   * the page's fused gate / up / ReLU kernel computes).  weights[0].y receives
   * h = (r * r) * u with r = max(g, 0), g and u the gate and up outputs (the
   * fp32 steps of the gating prologue, so a following call on h without mul
   * gives bit for bit the results of one on g with mul = u); weights[1].y
   * receives u.  The decode kernel computes h in its epilogue, every CTA
   * holding the same rows of both matrices; the tensor-core kernels are
   * followed by one elementwise launch. */
  BITLINEAR_FLAG_GATED = 2
};

/* bitlinear_forward with an explicit algorithm and flags (see above).
 * Errors: as bitlinear_forward; BITLINEAR_ERR_UNSUPPORTED for an unknown
 * algorithm or flag bit, or a shape outside the chosen kernel's limits. */
bitlinear_status bitlinear_forward_ex(const int8_t* xq, const float* x_scale, int64_t M,
                                      const uint8_t* packed, const float* w_scale,
                                      int64_t N, int64_t K, float* y, int32_t* acc,
                                      int algo, int flags, void* stream);

/*
 * Workspace of bitlinear_forward_ws: 2 * K * (M rounded up to 16) bytes (0 for
 * M <= 0 or K <= 0).
 */
size_t bitlinear_forward_workspace(int64_t M, int64_t K);

/*
 * bitlinear_forward_ex with a caller-provided device workspace (16-byte
 * aligned, at least bitlinear_forward_workspace(M, K) bytes; its contents
 * are scratch, overwritten on the stream).  It enables BITLINEAR_ALGO_WIDE,
 * the tensor-core path for many tokens ("Hesper.Models.BitNet" page, section
 * "Architecture": a full-sequence forward runs every BitLinear on all tokens
 * at once): a pre-pass widens xq once to fp16 in the workspace, laid out as
 * the MMA's shared-memory operand, so the contraction kernel only widens the
 * 2-bit weight codes (into tensor memory) and bulk-copies the token tiles.
 * Results are bit-identical to every other algorithm.  BITLINEAR_ALGO_AUTO
 * follows bitlinear_forward's rule, except that it takes WIDE for narrow
 * outputs of long K at medium token counts -- N <= 4096, K >= 8192 and
 * 128 < M <= 512 -- where it measured faster on GB300 (BitNet-3B and
 * BitNet-1.3B down shapes, alone and inside a layer's chain of calls); for
 * shorter K (faster alone for some shapes, slower in the chain), wide outputs,
 * more tokens and below 129 tokens the other kernels measured faster or
 * within a few per cent.  The other algorithms ignore the workspace.
 * Errors: as bitlinear_forward_ex; BITLINEAR_ERR_WORKSPACE when
 * BITLINEAR_ALGO_WIDE is asked for without a large enough workspace;
 * BITLINEAR_ERR_ALIGN for a misaligned workspace.
 */
bitlinear_status bitlinear_forward_ws(const int8_t* xq, const float* x_scale, int64_t M,
                                      const uint8_t* packed, const float* w_scale,
                                      int64_t N, int64_t K, float* y, int32_t* acc,
                                      int algo, int flags, void* workspace, size_t workspace_bytes,
                                      void* stream);

/* One weight matrix of a bitlinear_linear call. */
typedef struct bitlinear_weight {
  const uint8_t* packed;  /* device, bitlinear_packed_bytes(N, K) bytes */
  const float* w_scale;   /* device, 1 fp32 (sw) */
  int64_t N;              /* output features, > 0 */
  float* y;               /* device fp32 [M, N] row-major, written */
  int32_t* acc;           /* device int32 [M, N] or NULL (raw accumulators) */
} bitlinear_weight;

/*
 * A whole BitLinear call: activation_quant (with the optional gating and
 * RMSNorm prologues) and the contraction + rescale for 1..4 weight matrices
 * that share the input (q, k, v; gate, up; or a single projection).  The
 * results are exactly those of bitlinear_quant_act(x, mul, M, K, rms_weight,
 * rms_eps, xq, x_scale) followed by bitlinear_forward for each matrix; xq and
 * x_scale receive the quantised activations.
 * With M == 1 and K <= 16384 this is one kernel launch: every CTA streams its
 * share of the packed weights while it quantises the token itself (CTA 0
 * writes xq, x_scale), which keeps a separate act_quant kernel and its
 * latency off the decode critical path; the matrices' CTAs share one grid.
 * So is a call of M = 2 tokens without mul and rms_weight whose matrices
 * all take the decode kernel, when K <= 3072 (the rows fit the kernel's
 * registers) and the matrices have at least 8 * (SM count) rows together
 * (each CTA's dots outweigh its loading the two rows).
 * Otherwise it runs bitlinear_quant_act, then one launch per kernel that
 * bitlinear_forward's AUTO rule picks for some matrix: the matrices given to
 * the same kernel (decode, batched or 128-token-tile) share one grid, whose
 * tiles span all of them.
 * Constraints: K % 64 == 0, K <= 32768, every matrix with the same K;
 * BITLINEAR_FLAG_PDL as for bitlinear_forward_ex (the packed weights and
 * scales must not come from the kernel immediately before on the stream);
 * BITLINEAR_FLAG_GATED (see above) needs num_weights == 2 and equal N, else
 * BITLINEAR_ERR_SHAPE.  Other flag bits: BITLINEAR_ERR_UNSUPPORTED.
 */
bitlinear_status bitlinear_linear(const float* x, const float* mul, int64_t M, int64_t K,
                                  const float* rms_weight, double rms_eps,
                                  const bitlinear_weight* weights, int num_weights,
                                  int8_t* xq, float* x_scale, int flags, void* stream);

/*
 * bitlinear_linear with an optional device workspace (NULL: exactly
 * bitlinear_linear; otherwise 16-byte aligned and at least
 * bitlinear_forward_workspace(M, K) bytes, else BITLINEAR_ERR_WORKSPACE).
 * Matrices that bitlinear_forward_ws's AUTO rule gives to the WIDE kernel use
 * it, one launch each; the activations are widened into the workspace once per call, shared by
 * those matrices.  Results are bit-identical to bitlinear_linear.
 */
bitlinear_status bitlinear_linear_ws(const float* x, const float* mul, int64_t M, int64_t K,
                                     const float* rms_weight, double rms_eps,
                                     const bitlinear_weight* weights, int num_weights,
                                     int8_t* xq, float* x_scale, int flags,
                                     void* workspace, size_t workspace_bytes, void* stream);

/* Size of the library's own device scratch array used by
 * bitlinear_quantize_weights_noalloc. */
#define BITLINEAR_NOALLOC_SCRATCH_BYTES 4096

/*
 * bitlinear_quantize_weights without a caller-provided workspace.
 * (No counterpart on the pages: this is an interface convenience of this
 * library, not part of the BitLinear method.)
 *
 * Some callers cannot allocate device memory at the point where they quantise
 * weights: a runtime that fixes its memory budget at start-up and forbids
 * later allocations, a plugin whose host gives it kernels and streams but no
 * allocator, or code that must not touch the allocator at all.  This entry
 * point takes the same inputs and outputs as bitlinear_quantize_weights and
 * gives bit-identical results, but its scratch space (the per-exponent
 * bucket sums) lives in a 4096-byte array inside this library
 * (BITLINEAR_NOALLOC_SCRATCH_BYTES), held on every GPU that loads the library
 * until the process exits.  It calls no cudaMalloc/cudaFree and no allocating
 * library routine.
 *  - The first call on a device looks up that array's device address (once
 *    per device, with the device current); make that first call before any
 *    stream capture begins.
 *  - Every call on a device shares the one array and clears it on the stream
 *    before use, so calls whose kernels overlap on the GPU (different streams
 *    without ordering between them) race and give wrong results; order them.
 *  - A matrix whose scratch need would exceed the array is rejected with
 *    BITLINEAR_ERR_WORKSPACE (never the case today: the need is 4096 bytes for
 *    every N, K that the shape checks accept).
 * Other arguments, errors and results: as bitlinear_quantize_weights.
 */
bitlinear_status bitlinear_quantize_weights_noalloc(const float* W, int64_t N, int64_t K,
                                                    uint8_t* packed, float* w_scale, void* stream);

/* Greedy token choice after the LM head (which is a BitLinear too,
 * "Hesper.Models.BitNet" page, section "Performance (BitNet-3B on A100)"):
 * index[m] = the smallest n with y[m, n] == max over n of y[m, n], so that
 * only 4 bytes per token need to reach the host.
 *   y      device, fp32 [M, N] row-major (e.g. bitlinear_forward's output).
 *   M      rows (tokens), M >= 0; M == 0 enqueues nothing.
 *   N      1 <= N < 2^31.
 *   index  device int32 [M], written.
 * Ties go to the smaller index; -0.0 and +0.0 are equal.  Rows holding NaN
 * give an unspecified index (like every non-finite input here).
 * Errors: BITLINEAR_ERR_NULL, BITLINEAR_ERR_SHAPE, BITLINEAR_ERR_ALIGN (y not
 * 4-byte aligned), BITLINEAR_ERR_CUDA. */
bitlinear_status bitlinear_argmax(const float* y, int64_t M, int64_t N, int32_t* index, void* stream);

/* Exercises the failure-detection path without faulting anything: launches a
 * one-warp kernel that waits on an mbarrier nothing ever arrives on, with the
 * same bounded wait the kernels use, giving up after limit_ns (0 < limit_ns
 * <= 1 s).  The expired wait records BITLINEAR_ERR_TIMEOUT in the device
 * status word (read it with bitlinear_device_status); the CUDA context stays
 * usable. */
bitlinear_status bitlinear_selftest_wait_timeout(int64_t limit_ns, void* stream);

/* Synchronises `stream`, then returns BITLINEAR_ERR_TIMEOUT if any kernel of
 * this library recorded a timed-out wait on the current device since the last
 * call with clear != 0, BITLINEAR_ERR_CUDA if the stream reports an error,
 * else BITLINEAR_OK.  With clear != 0 the status word is reset. */
bitlinear_status bitlinear_device_status(void* stream, int clear);

#ifdef __cplusplus
}
#endif

#endif /* BITLINEAR_H */
