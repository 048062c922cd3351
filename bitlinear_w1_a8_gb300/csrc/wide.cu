// wide.cu -- BitLinear contraction for many tokens on the tcgen05 tensor
// cores, with the activations widened once per call.
//
// y[m, n] = acc[m, n] / (sx[m] * sw),  acc = xq . Wq^T  (BitNet b1.58 BitLinear
// over a whole sequence: every projection runs on [batch*seq, dim] tokens,
// "Hesper.Models.BitNet" page, section "Architecture", and "Transformer Block"
// page, section "Forward Pass").
//
// sm_103a has no integer tcgen05 MMA, so both operands enter kind::f16 MMAs as
// fp16: int8 activations and ternary weights are exact in fp16, every product
// is an exact integer and the fp32 accumulator is exact while |acc| < 2^24
// (|acc| <= 127 K, K <= 131072).
//
// The kernel with 128-token tiles (prefill.cu) widens each activation again
// for every tile of output columns (54 times at N = 10240) and its converter
// warps' instruction issue sets its pace.  Here a pre-pass widens the int8
// activations ONCE into a workspace laid out as the MMA's shared-memory
// operand wants it, and the contraction kernel
//   * puts 128 weight rows on the MMA's M side: converter warps widen the
//     2-bit codes straight into TMEM (tcgen05.st, one weight row per lane),
//   * puts up to 192 tokens on the MMA's N side: ONE bulk copy per k-step
//     brings their fp16 tile from the workspace into shared memory, already
//     in the 128-byte-swizzled K-major layout, with no conversion at all.
// Per 128 x 192 x 64 k-step that is 2 KB of codes widened (instead of 8 KB of
// activations and 12 KB of codes), 26 KB copied from L2 and 24 KB read by the
// MMA from shared memory.
//
// Workspace layout (written by widen_tokens): for k-block kb (k = 64 kb ..
// 64 kb + 63) and token row m < Mp (M rounded up to 16; rows >= M are zero),
// the 128 bytes at ((kb * Mp) + m) * 128 hold that row's 64 fp16 values as 8
// 16-byte chunks; chunk c (k = 64 kb + 8c .. 8c + 7, inside each group of four
// in the order (0, 2, 1, 3), the order in which the weight codes are widened)
// sits at chunk position c ^ (m % 8).  A token tile that starts at a multiple
// of 8 rows is therefore, byte for byte, the 128-byte-swizzled K-major tile.
//
// CTA roles (one persistent CTA per SM, 23 warps):
//   warps 0-3    epilogue: TMEM -> registers -> y = acc/(sx*sw) -> global
//   warps 4-19   converters, four groups of four: group g widens the codes of
//                every fourth k-step into TMEM weight stage f % 4
//   warps 20-21  loaders (even / odd k-steps): per k-step, one
//                arrive.expect_tx and two bulk copies (token tile, packed
//                codes) into an 8-slot shared-memory ring
//   warp 22      allocates TMEM; one lane issues tcgen05.mma and one
//                tcgen05.commit per k-step, which frees both the ring slot and
//                the TMEM weight stage
// TMEM: two 128 x 192 fp32 accumulators (the epilogue of one tile overlaps
// the MMAs of the next) and four 128 x 64 fp16 weight stages.  When tiles are
// few, K is split over the CTAs of a thread-block cluster that add their
// partial sums through distributed shared memory.  Every wait is
// bounded by the global timer; on timeout the kernel records BITLINEAR_ERR_TIMEOUT, every role
// leaves its loop, the loaders wait (bounded) for their own copies, the MMA
// warp for its own MMAs, and TMEM is freed before the kernel returns.
#include "common.cuh"
#include "tc_util.cuh"

namespace bitlinear {
namespace {

using namespace tc;

constexpr int kRing = 8;                           // shared-memory slots (token tile + codes)
constexpr int kRows = 128;                         // weight rows per tile = MMA M = TMEM lanes
constexpr int kMaxTok = 192;                       // token rows per tile = MMA N (multiple of 16)
// TMEM (512 columns): kAccBufs accumulators of kMaxTok columns, then as many
// 32-column weight stages as fit.  Two accumulators (the epilogue of one tile
// overlaps the MMAs of the next) and four stages measured faster than one
// accumulator and ten stages: the k-step is bounded by the token ring's
// round trip (MMA complete -> commit -> loader -> bulk copy -> converter ->
// MMA, ~2.5 us, against 8 slots of ~0.2 us of MMA work each), not by the
// stages.
constexpr int kAccBufs = 2;
constexpr int kWStages = (512 - kAccBufs * kMaxTok) / 32;  // 4
constexpr int kDoneRing = 16;                      // kstep_done barriers: k-step f uses f % 16
constexpr int kKStep = 64;                         // K per k-step (128 bytes of fp16)
constexpr int kTokBytes = kMaxTok * 128;           // 24 KB fp16 token tile
constexpr int kCodeBytes = kRows * 16;             // 2 KB packed codes
constexpr int kSlotBytes = kTokBytes + kCodeBytes;  // 26 KB
constexpr int kSmemBytes = kRing * kSlotBytes;
constexpr int kEpiWarps = 4;
constexpr int kGroupWarps = 4;
constexpr int kGroupThreads = kGroupWarps * 32;    // 128: one weight row each
constexpr int kConvGroups = 4;                     // group g converts the k-steps f with f % 4 == g
constexpr int kConvWarps = kConvGroups * kGroupWarps;  // 16
constexpr int kLoadWarp0 = kEpiWarps + kConvWarps;  // 20
constexpr int kLoadWarps = 2;                       // a second issuing warp doubles the copy issue rate
constexpr int kMmaWarp = kLoadWarp0 + kLoadWarps;   // 22
constexpr int kThreads = (kMmaWarp + 1) * 32;       // 736
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemW = kAccBufs * kMaxTok;    // weight stages follow the accumulators
constexpr uint32_t kTmemWStageCols = kKStep / 2;   // 64 fp16 of a row = 32 columns
static_assert(kGroupThreads == kRows, "one weight row (TMEM lane) per converter thread");
static_assert(kEpiWarps % 4 == 0, "converter warp w reaches TMEM lanes 32 (w % 4) ..");
static_assert(kTmemW + kWStages * kTmemWStageCols <= kTmemCols, "TMEM budget");
static_assert(kSlotBytes % 1024 == 0, "token tiles 1024-byte aligned for the swizzle");
static_assert(kSmemBytes + 1024 <= 232448, "shared memory per CTA");
static_assert((kRing & (kRing - 1)) == 0 && kRing % kLoadWarps == 0, "ring indexing");
static_assert((kDoneRing & (kDoneRing - 1)) == 0 && kDoneRing > kWStages && kDoneRing >= kRing,
              "a kstep_done barrier is reused only after its waiters are past");
constexpr int kEpiBar = 1 + kWStages;              // the epilogue warps' named barrier
constexpr int kMaxSplits = 8;                      // K ranges of a tile: a portable cluster
static_assert(kEpiBar < 16, "named barriers 1 .. kWStages, kEpiBar");
static_assert(kSmemBytes >= kMaxTok * kRows * 4, "split-K partial sums fit over the ring");

struct WideParams {
  const uint8_t* xw;      // widened tokens (layout above)
  const float* sx;
  const uint8_t* packed;
  const float* sw;
  float* y;
  int32_t* acc;
  int* status;
  int M, Mp, N;
  int KB;                 // k-steps per work unit (K / 64 / splits)
  int tn;                 // token rows per tile, multiple of 16, <= kMaxTok
  int tiles_w, tiles_t;   // weight tiles (128 rows), token tiles (tn rows)
  int splits;             // K ranges per tile
  int num_units;          // tiles_w * tiles_t * splits
};

struct WideCtl {
  unsigned long long ring_full[kRing];     // token tile + codes of k-step f landed (transaction bytes)
  unsigned long long kstep_done[kDoneRing];  // the MMAs of k-step f are complete: slot f % kRing and
                                            // TMEM weight stage f % kWStages are free again
  unsigned long long acc_full[kAccBufs];
  unsigned long long acc_empty[kAccBufs];
  unsigned long long mma_done;
  unsigned long long parts_ready;           // split K: one arrival per other rank of the cluster
  uint32_t tmem_base;
  int abort_flag;
};

// Work unit -> first weight row, first token row, first k-block, token rows.
// Weight tiles vary fastest, so the CTAs running at once share token tiles.
__device__ __forceinline__ void unit_coords(const WideParams& p, int unit, int& n0, int& m0, int& kb0, int& rows_t) {
  const int tile = unit / p.splits;
  kb0 = (unit - tile * p.splits) * p.KB;
  const int tt = tile / p.tiles_w;
  n0 = (tile - tt * p.tiles_w) * kRows;
  m0 = tt * p.tn;
  rows_t = p.Mp - m0 < p.tn ? p.Mp - m0 : p.tn;
}

// int8 activations [M, K] -> the fp16 workspace.  Block (x, kb): one thread per
// 16-byte chunk of k-block kb; rows M .. Mp-1 are written as zeros.
__global__ void __launch_bounds__(256) widen_tokens(const int8_t* __restrict__ xq, int M, int Mp, int K,
                                                    uint4* __restrict__ xw) {
  pdl_release_dependents();
  pdl_wait_primary();  // xq comes from the previous kernel on the stream
  const int kb = blockIdx.y;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;  // chunk within the k-block plane
  if (i >= Mp * 8) return;
  const int m = i >> 3, c = i & 7;
  uint4 o = make_uint4(0u, 0u, 0u, 0u);
  if (m < M) {
    const uint2 v = *reinterpret_cast<const uint2*>(xq + (int64_t)m * K + (int64_t)kb * kKStep + c * 8);
    i8x4_to_f16x4(v.x, o.x, o.y);
    i8x4_to_f16x4(v.y, o.z, o.w);
  }
  xw[((int64_t)kb * Mp + m) * 8 + (c ^ (m & 7))] = o;
}

// At most 80 registers a thread: the 23 warps are spread over the SM's four
// schedulers (6 on the busiest), each with 16384 registers.  The converters
// keep a k-step's 32 widened words in registers across a wait.
static_assert((kThreads / 32 + 3) / 4 * 32 * 80 <= 16384, "register budget per scheduler");
__global__ void __maxnreg__(80) wide_kernel(const __grid_constant__ WideParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ WideCtl ctl;
  __shared__ float den_s[kEpiWarps][kMaxTok];  // epilogue warp w: sx[t] * sw of the tile's tokens
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t ring_base = (smem_u32(smem_raw) + 1023u) & ~1023u;  // the swizzle follows address bits

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRing; ++s) mbar_init(&ctl.ring_full[s], 1);
    for (int s = 0; s < kDoneRing; ++s) mbar_init(&ctl.kstep_done[s], 1);
    for (int s = 0; s < kAccBufs; ++s) {
      mbar_init(&ctl.acc_full[s], 1);
      mbar_init(&ctl.acc_empty[s], kEpiWarps);
    }
    mbar_init(&ctl.mma_done, 1);
    mbar_init(&ctl.parts_ready, p.splits > 1 ? (uint32_t)(p.splits - 1) : 1u);
    ctl.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) tmem_alloc(&ctl.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Split K: the ranks' barriers are initialised before another rank arrives on them.
  if (p.splits > 1) cluster_sync_all();
  const uint32_t tmem_base = ctl.tmem_base;

  // The workspace is written by the pre-pass just before on the stream.
  pdl_release_dependents();
  pdl_wait_primary();

  const int my_units = (int)blockIdx.x < p.num_units ? (p.num_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int total = my_units * p.KB;  // flat k-steps of this CTA, unit-major

  if (warp >= kLoadWarp0 && warp < kMmaWarp) {
    // ------------------------------------------------------------------ loaders
    // Loader li takes the k-steps f = li, li + 2, ... (slot f % kRing): lane 0
    // waits until the MMAs of k-step f - kRing are complete, arms the slot's
    // barrier with the bytes of both copies, then lane 0 copies the token tile
    // and lane 1 the codes.
    const int li = warp - kLoadWarp0;
    int unit = blockIdx.x, ks = li;
    while (ks >= p.KB) {
      ks -= p.KB;
      unit += gridDim.x;
    }
    int cur = -1, n0 = 0, m0 = 0, kb0 = 0, rows_t = 0;
    uint32_t tok_bytes = 0, code_bytes = 0;
    int last = -1;
    for (int f = li; f < total; f += kLoadWarps) {
      if (unit != cur) {
        unit_coords(p, unit, n0, m0, kb0, rows_t);
        tok_bytes = (uint32_t)rows_t * 128u;
        code_bytes = (uint32_t)(p.N - n0 < kRows ? p.N - n0 : kRows) * 16u;  // rows past N are not read
        cur = unit;
      }
      const int slot = f & (kRing - 1);
      bool ok = true;
      if (lane == 0 && f >= kRing) {
        const int prev = f - kRing;  // the slot's previous k-step
        ok = mbar_wait(&ctl.kstep_done[prev & (kDoneRing - 1)], (uint32_t)((prev / kDoneRing) & 1), &ctl.abort_flag,
                       p.status);
      }
      if (__shfl_sync(kFullMask, ok ? 1 : 0, 0) == 0) break;
      const uint32_t dst = ring_base + (uint32_t)slot * kSlotBytes;
      const int64_t kb = kb0 + ks;
      if (lane == 0) mbar_arrive_expect_tx(&ctl.ring_full[slot], tok_bytes + code_bytes);
      __syncwarp();
      if (lane == 0) bulk_copy_g2s(dst, p.xw + (kb * p.Mp + m0) * 128, tok_bytes, &ctl.ring_full[slot]);
      if (lane == 1) bulk_copy_g2s(dst + kTokBytes, p.packed + (kb * p.N + n0) * 16, code_bytes, &ctl.ring_full[slot]);
      last = f;
      ks += kLoadWarps;
      while (ks >= p.KB) {
        ks -= p.KB;
        unit += gridDim.x;
      }
    }
    // No copy may outlive the CTA: wait (bounded, abort or not) for the last
    // fill of every slot this loader armed.
    if (lane == 0) {
      for (int f = last; f >= 0 && f > last - kRing; f -= kLoadWarps)
        mbar_drain(&ctl.ring_full[f & (kRing - 1)], (uint32_t)((f / kRing) & 1), p.status);
    }
    __syncwarp();
  } else if (warp >= kEpiWarps && warp < kLoadWarp0) {
    // ------------------------------------------------------------------ converters
    // Group g widens the codes of k-steps f = g, g + 4, ... into TMEM weight
    // stage f % kWStages; thread u takes weight row u of the tile (TMEM lane u).  Codes of
    // rows past N are whatever the slot held: they only reach accumulator rows
    // that the epilogue skips.
    // Every k-step f the group owns ends with its arrival on named barrier
    // 1 + f % kWStages (one barrier per TMEM stage), after an abort too
    // (without the work), and never before the MMAs of k-step f - kWStages,
    // the stage's previous user, were committed (a wait that ignores the
    // abort flag; the MMA warp keeps committing after an abort).  The MMA warp
    // syncs that barrier for k-step f - kWStages before it commits it, so each
    // phase of a barrier holds one k-step's converters and the MMA warp's sync
    // of that k-step, and the MMA warp's syncs, which cannot time out, always
    // complete.
    const int cw = warp - kEpiWarps;
    const int grp = cw / kGroupWarps;
    const int u = (cw % kGroupWarps) * 32 + lane;
    const uint32_t t_lane = tmem_base + ((uint32_t)((u >> 5) * 32) << 16) + kTmemW;
    bool live = true;
    for (int f = grp; f < total; f += kConvGroups) {
      const int slot = f & (kRing - 1);
      // Widen the codes into registers as soon as they have landed, and only
      // then wait for the stage: the MMAs of k-step f - kWStages (the last
      // reader of this stage) must be complete before the TMEM stores.
      live = live && mbar_wait(&ctl.ring_full[slot], (uint32_t)((f / kRing) & 1), &ctl.abort_flag, p.status);
      uint32_t lo[16], hi[16];
      if (live) {
        const uint4 wv = ld_shared_v4(ring_base + (uint32_t)slot * kSlotBytes + kTokBytes + (uint32_t)(u * 16));
        codes_to_f16x8(wv.x, lo);
        codes_to_f16x8(wv.y, lo + 8);
        codes_to_f16x8(wv.z, hi);
        codes_to_f16x8(wv.w, hi + 8);
      }
      const int prev = f - kWStages;
      const bool stage_free =
          prev < 0 || mbar_wait_lockstep(&ctl.kstep_done[prev & (kDoneRing - 1)], (uint32_t)((prev / kDoneRing) & 1),
                                         &ctl.abort_flag, p.status);
      live = live && stage_free;
      if (live) {
        tc_fence_after();  // the MMAs that read this stage are complete
        const uint32_t t_addr = t_lane + (uint32_t)(f % kWStages) * kTmemWStageCols;
        tmem_st16(t_addr, lo);
        tmem_st16(t_addr + 16u, hi);
        tmem_st_wait();
        tc_fence_before();
      }
      named_bar_arrive(1 + f % kWStages, kGroupThreads + 32);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp takes each stage's named barrier (an mbarrier wait by the
    // issuing thread would wait for its in-flight MMAs to drain); lane 0 issues
    // four 128 x rows_t x 16 MMAs and one commit.  After an
    // abort the warp still syncs and commits every k-step (issuing nothing), so
    // the converters, which wait for those commits, stay in step with it.
    bool aborted = false;
    int f = 0, it = 0;
    for (int unit = blockIdx.x; unit < p.num_units; unit += gridDim.x, ++it) {
      int n0, m0, kb0, rows_t;
      unit_coords(p, unit, n0, m0, kb0, rows_t);
      const uint32_t idesc = make_idesc(kRows, rows_t);
      const int aslot = it % kAccBufs;
      const uint32_t use = (uint32_t)(it / kAccBufs);  // earlier tiles in this accumulator
      // lane 0 decides for the warp
      bool ab = aborted || *reinterpret_cast<volatile int*>(&ctl.abort_flag) != 0;
      if (!ab && lane == 0) ab = !mbar_wait(&ctl.acc_empty[aslot], (use & 1u) ^ 1u, &ctl.abort_flag, p.status);
      aborted = __shfl_sync(kFullMask, ab ? 1 : 0, 0) != 0;
      const uint32_t d_tmem = tmem_base + (uint32_t)(aslot * kMaxTok);
      for (int ks = 0; ks < p.KB; ++ks, ++f) {
        const int stage = f % kWStages;
        const int slot = f & (kRing - 1);
        named_bar_sync(1 + stage, kGroupThreads + 32);
        if (lane == 0) {
          if (!aborted) {
            tc_fence_after();
            const uint32_t a_tmem = tmem_base + kTmemW + (uint32_t)stage * kTmemWStageCols;
            const uint64_t b_desc = smem_desc_sw128(ring_base + (uint32_t)slot * kSlotBytes);
#pragma unroll
            for (int kk = 0; kk < kKStep / 16; ++kk) {
              // 16 fp16 along K: 8 TMEM columns of A, 32 bytes inside B's swizzle atom
              mma_f16_ta(d_tmem, a_tmem + (uint32_t)(kk * 8), b_desc + (uint64_t)(kk * 2), idesc,
                         (ks | kk) != 0 ? 1u : 0u);
            }
          }
          mma_commit(&ctl.kstep_done[f & (kDoneRing - 1)]);
        }
        __syncwarp();
      }
      if (lane == 0) mma_commit(&ctl.acc_full[aslot]);
    }
    if (lane == 0) {
      // All MMAs this thread issued must be complete before TMEM is freed.
      mma_commit(&ctl.mma_done);
      mbar_drain(&ctl.mma_done, 0u, p.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue
    // TMEM lane = weight row n, column j = token m0 + j: a warp writes 32
    // consecutive n of one token row.  Before waiting for a tile's
    // accumulator, each warp stages the tile's denominators sx[t] * sw in its
    // own shared-memory row with one batch of independent loads (loaded per
    // 16-token chunk they cost a dependent round trip each, serialised with
    // the MMAs of the next tile).
    const int row = warp * 32 + lane;
    const float sw = *p.sw;
    float* dw = den_s[warp];
    int it = 0;
    for (int unit = blockIdx.x; unit < p.num_units; unit += gridDim.x, ++it) {
      int n0, m0, kb0, rows_t;
      unit_coords(p, unit, n0, m0, kb0, rows_t);
      const int aslot = it % kAccBufs;
      __syncwarp();  // the previous tile's reads of dw are done
      for (int j = lane; j < rows_t; j += 32) {
        const int t = m0 + j;
        dw[j] = t < p.M ? __fmul_rn(__ldg(p.sx + t), sw) : 1.0f;
      }
      __syncwarp();
      if (!mbar_wait(&ctl.acc_full[aslot], (uint32_t)((it / kAccBufs) & 1), &ctl.abort_flag, p.status)) break;
      tc_fence_after();
      const int n = n0 + row;
      const bool n_ok = n < p.N;
      const uint32_t t_row = tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)(aslot * kMaxTok);
      for (int c = 0; c < rows_t; c += 16) {
        uint32_t r[16];
        tmem_ld16(t_row + (uint32_t)c, r);
        if (p.splits > 1) {
          // Split K (one unit per CTA; the units of a tile are one cluster,
          // rank = K range): this rank's exact partial sums go to its own
          // shared memory, [token column][128 weight rows], over the ring,
          // which no copy or MMA uses any more.  (Kept inside this loop and
          // ahead of the row test: the unsplit epilogue measured ~8% slower
          // at 2048 tokens with the split stores in a loop of their own or
          // after the row test.)
#pragma unroll
          for (int j = 0; j < 16; ++j)
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(ring_base + (uint32_t)(((c + j) * kRows + row) * 4)),
                         "r"(__float2int_rn(__uint_as_float(r[j])))
                         : "memory");
          continue;
        }
        if (!n_ok) continue;
        float* yc = p.y + (int64_t)(m0 + c) * p.N + n;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (m0 + c + j < p.M) yc[(int64_t)j * p.N] = __fdiv_rn(__uint_as_float(r[j]), dw[c + j]);  // r[j]: an exact integer
        if (p.acc) {
          int32_t* ac = p.acc + (int64_t)(m0 + c) * p.N + n;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (m0 + c + j < p.M) ac[(int64_t)j * p.N] = __float2int_rn(__uint_as_float(r[j]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.acc_empty[aslot]);  // one arrival per warp
      if (p.splits > 1) break;
    }
    if (p.splits > 1 && (int)blockIdx.x < p.num_units) {
      // Every rank adds one share of the tile's token columns over all ranks'
      // partial sums (distributed shared memory) and writes those outputs.
      // Every rank takes part whatever happened before, so the others' waits
      // end early.
      named_bar_sync(kEpiBar, kEpiWarps * 32);  // this rank's partial sums are written
      const uint32_t rank = cluster_rank();
      if (warp == 0 && lane < p.splits && lane != (int)rank)
        mbar_arrive_remote(map_shared(smem_u32(&ctl.parts_ready), (uint32_t)lane));
      if (mbar_wait_cluster(&ctl.parts_ready, 0u, &ctl.abort_flag, p.status) &&
          *reinterpret_cast<volatile int*>(&ctl.abort_flag) == 0) {
        int n0, m0, kb0, rows_t;
        unit_coords(p, blockIdx.x, n0, m0, kb0, rows_t);
        const int c0 = (int)rank * rows_t / p.splits, c1 = ((int)rank + 1) * rows_t / p.splits;
        // item: token column c, weight rows l4 .. l4 + 3
        for (int it2 = c0 * (kRows / 4) + warp * 32 + lane; it2 < c1 * (kRows / 4); it2 += kEpiWarps * 32) {
          const int c = it2 / (kRows / 4), l4 = (it2 % (kRows / 4)) * 4;
          const uint32_t off = ring_base + (uint32_t)((c * kRows + l4) * 4);
          uint4 part[kMaxSplits];
#pragma unroll
          for (int k = 0; k < kMaxSplits; ++k)  // every load issued before the sum
            part[k] = k < p.splits ? ld_cluster_v4(map_shared(off, (uint32_t)k)) : make_uint4(0u, 0u, 0u, 0u);
          uint4 tot = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int k = 0; k < kMaxSplits; ++k) {
            tot.x += part[k].x;
            tot.y += part[k].y;
            tot.z += part[k].z;
            tot.w += part[k].w;
          }
          const int t = m0 + c;
          if (t >= p.M) continue;
          const float den = __fmul_rn(p.sx[t], sw);
          const int av[4] = {(int)tot.x, (int)tot.y, (int)tot.z, (int)tot.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int n = n0 + l4 + e;
            if (n < p.N) {
              p.y[(int64_t)t * p.N + n] = __fdiv_rn(__int2float_rn(av[e]), den);
              if (p.acc) p.acc[(int64_t)t * p.N + n] = av[e];
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  // Split K: every rank has read the others' shared memory before any exits.
  if (p.splits > 1) cluster_sync_all();
}

cudaLaunchConfig_t launch_config(dim3 grid, dim3 block, size_t smem, bool pdl, int cluster, cudaStream_t stream,
                                 cudaLaunchAttribute (&attr)[2]) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  int na = 0;
  if (cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)cluster;
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
  return cfg;
}

cudaError_t launch_pdl(const void* func, dim3 grid, dim3 block, size_t smem, bool pdl, cudaStream_t stream,
                       void** args, int cluster = 1) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_config(grid, block, smem, pdl, cluster, stream, attr);
  return cudaLaunchKernelExC(&cfg, func, args);
}

// Clusters of `size` WIDE CTAs that fit on the GPU at once (0 on error);
// cached per device and size.  Needs the kernel's shared-memory attribute set.
int max_clusters(int size, const DeviceInfo& dev) {
  static thread_local int cache_dev = -1;
  static thread_local int cache[kMaxSplits + 1];
  if (cache_dev != dev.device) {
    for (int i = 0; i <= kMaxSplits; ++i) cache[i] = -1;
    cache_dev = dev.device;
  }
  if (cache[size] < 0) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg =
        launch_config(dim3((unsigned)size, 1, 1), dim3(kThreads, 1, 1), (size_t)kSmemBytes + 1024, false, size, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, wide_kernel, &cfg) != cudaSuccess) n = 0;
    cache[size] = n;
  }
  return cache[size];
}

// Estimated time of one k-step of a 128 x tn tile, in ns: the MMAs take about
// 1.1 tn ns per SM; below that the loader's ~250 ns per k-step (one mbarrier
// wait, one arm, two bulk copies) sets the pace.
int64_t kstep_ns(int tn) {
  const int64_t mma = (int64_t)tn * 11 / 10;
  return (mma > 250 ? mma : 250) + 20;
}

}  // namespace


size_t wide_workspace_bytes(int64_t M, int64_t K) {
  return (size_t)((M + 15) / 16 * 16) * (size_t)K * 2u;
}

// widen = false: the workspace already holds this xq (an earlier launch on the
// stream widened it), so only the contraction kernel is launched.
cudaError_t launch_wide(const int8_t* xq, const float* sx, int64_t M, const uint8_t* packed, const float* sw,
                        int64_t N, int64_t K, float* y, int32_t* acc, void* workspace, bool widen, bool pdl,
                        const DeviceInfo& dev, cudaStream_t stream) {
  if (M < 1 || N < 1 || K < kKStep || K % kKStep) return cudaErrorInvalidValue;
  const int64_t Mp = (M + 15) / 16 * 16;
  const int KB = (int)(K / kKStep);
  WideParams p;
  p.xw = static_cast<const uint8_t*>(workspace);
  p.sx = sx;
  p.packed = packed;
  p.sw = sw;
  p.y = y;
  p.acc = acc;
  p.status = dev.status;
  p.M = (int)M;
  p.Mp = (int)Mp;
  p.N = (int)N;
  p.tiles_w = (int)((N + kRows - 1) / kRows);
  {
    const size_t smem = (size_t)kSmemBytes + 1024;
    static thread_local int configured = -1;
    if (configured != dev.device) {
      cudaError_t err = cudaFuncSetAttribute(wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (err != cudaSuccess) return err;
      configured = dev.device;
    }
  }
  // Token-tile width and K split: the least estimated time of the busiest
  // CTA.  A split (only while the tiles fill at most half of the SMs) divides
  // K into at most 8 ranges of at least 8 k-steps; the ranges of a tile run as
  // one thread-block cluster that adds the partial sums through distributed
  // shared memory (~1 us), so all of the launch's clusters must fit at once.
  {
    int64_t best = -1;
    for (int tn = 16; tn <= kMaxTok; tn += 16) {
      const int tn_eff = tn < Mp ? tn : (int)Mp;
      const int64_t tiles = (int64_t)p.tiles_w * ((Mp + tn_eff - 1) / tn_eff);
      for (int sp = 1; sp <= kMaxSplits && sp <= KB; ++sp) {
        if (KB % sp) continue;
        if (sp > 1 && (2 * tiles > dev.num_sms || tiles * sp > dev.num_sms || KB / sp < 8)) continue;
        if (sp > 1 && tiles > max_clusters(sp, dev)) continue;
        const int64_t waves = (tiles * sp + dev.num_sms - 1) / dev.num_sms;
        const int64_t cost = waves * (KB / sp) * kstep_ns(tn_eff) + (sp > 1 ? 1000 : 0);
        if (best < 0 || cost < best) {
          best = cost;
          p.tn = tn_eff;
          p.splits = sp;
        }
      }
      if (tn >= Mp) break;
    }
  }
  p.tiles_t = (int)((Mp + p.tn - 1) / p.tn);
  p.KB = KB / p.splits;
  p.num_units = p.tiles_w * p.tiles_t * p.splits;

  cudaError_t err;
  if (widen) {
    const int m32 = (int)M, mp32 = (int)Mp, k32 = (int)K;
    uint4* xw = static_cast<uint4*>(workspace);
    void* args[] = {(void*)&xq, (void*)&m32, (void*)&mp32, (void*)&k32, (void*)&xw};
    err = launch_pdl((const void*)widen_tokens, dim3((unsigned)((Mp * 8 + 255) / 256), (unsigned)KB, 1), dim3(256, 1, 1),
                     0, pdl, stream, args);
    if (err != cudaSuccess) return err;
  }
  const int grid = p.splits > 1 ? p.num_units : (p.num_units < dev.num_sms ? p.num_units : dev.num_sms);
  void* args[] = {(void*)&p};
  return launch_pdl((const void*)wide_kernel, dim3((unsigned)grid, 1, 1), dim3(kThreads, 1, 1),
                    (size_t)kSmemBytes + 1024, true, stream, args, p.splits);
}

}  // namespace bitlinear
