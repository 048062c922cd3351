// prefill.cu -- BitLinear contraction for many tokens on the 5th-generation
// tensor cores (tcgen05, sm_103a).
//
// y[m, n] = acc[m, n] / (sx[m] * sw),  acc = xq . Wq^T  (BitNet b1.58 BitLinear;
// a full-sequence forward runs every projection on [batch*seq, dim] tokens,
// "Hesper.Models.BitNet" page, section "Architecture", and "Transformer Block"
// page, section "Forward Pass").  At M = 2048 tokens this is a dense
// contraction, so it runs on the tensor cores.
//
// sm_103a has no integer tcgen05 MMA (ptxas rejects kind::i8 for this
// target), so the operands are widened to fp16 on chip: int8
// activations (|xq| <= 127) and ternary weights are exact in fp16, every
// product is an exact integer, and the fp32 accumulator holds every partial
// sum exactly while |acc| < 2^24 (|acc| <= 127*K, K <= 131072 here).  The
// int32 result is therefore bit-exact.
//
// CTA roles (one persistent CTA per SM, 25 warps):
//   warps 0-3   epilogue: TMEM -> registers -> y = acc/(sx*sw) -> global
//   warps 4-19  converters, four groups of four: group g widens the raw
//               tiles of every fourth k-step to fp16 in stage g -- the
//               activations into TMEM (one row per lane), the weights into
//               shared memory in the 128-byte-swizzled K-major layout
//   warps 20-23 loaders of the shared-memory ring: per k-step one
//               thread of warp 20 issues the TMA tensor copy of the 128 x 64
//               int8 activation tile (64-byte swizzle) and one thread of warp
//               21 the bulk copy of the packed codes, both completing on the
//               slot's barrier; warps 22-23 only reach the final barrier
//               (16-byte cp.async from 128 loader threads had bounded the
//               192-wide k-step: 130.7 -> 121.3 us at M = 2048, K = 2560 ->
//               N = 10240)
//   warp 24     allocates TMEM; one lane issues tcgen05.mma
// Every hand-off between roles is one mbarrier arrival per warp (raw slot
// full: the two loaders' arrive.expect_tx plus the copies' transaction bytes),
// except "stage full" (converters -> MMA warp), a named barrier per stage.
// The MMA takes A (activations) from TMEM and B (weights) from shared memory,
// so the widened activations never pass through shared memory, whose
// bandwidth the weight stores, the raw copies and the MMA's reads of B share.
// Shared memory holds kStages fp16 weight stages (n_tile x 64) and a ring of
// raw stages (A 128x64 int8, B n_tile x 16 B packed); TMEM holds two
// 128 x n_tile fp32 accumulators, so the epilogue of one tile overlaps the
// MMAs of the next, and kStages 128 x 64 fp16 activation stages -- or, with
// 320-wide tiles (one per CTA), one accumulator (Shape<true>).  When tiles are
// few, K is split over the CTAs of a thread-block cluster that add their
// partial sums through distributed shared memory.  Every mbarrier wait is
// bounded by the global timer: on timeout the kernel records
// BITLINEAR_ERR_TIMEOUT in the status word, every role leaves its loop, the
// MMA warp waits (bounded) for its own MMAs, frees TMEM and the kernel
// returns.
#include <cuda.h>

#include "common.cuh"
#include "tc_util.cuh"

namespace bitlinear {
namespace {

using namespace tc;

constexpr int kStages = 4;                       // fp16 operand stages read by the MMA
constexpr int kRawStages = 8;                    // raw int8 / packed k-steps in the ring (192-wide tiles)
constexpr int kRawStagesBig = 4;                 // the same for 320-wide tiles (the stages take the room)
constexpr int kTileM = 128;
constexpr int kMaxTileN = 192;                   // multiple of 16; TMEM holds 2 x 192 + 4 x 32 columns
constexpr int kMaxTileNBig = 320;                // one accumulator: TMEM holds 320 + 4 x 32 columns
constexpr int kKStep = 64;                       // K elements per stage (128 B of fp16)
constexpr int kMaxSplits = 8;                    // K ranges of a tile: a portable cluster
constexpr int kRawABytes = kTileM * kKStep;      // 8 KB of int8 activations
constexpr int kEpiWarps = 4;
constexpr int kConvGroups = kStages;                // group g converts the k-steps f with f % kStages == g
constexpr int kGroupWarps = 4;
constexpr int kGroupThreads = kGroupWarps * 32;     // 128
constexpr int kConvWarps = kConvGroups * kGroupWarps;  // 16
constexpr int kLoadWarps = 4;                       // warps 20, 21 load; 22-23 keep the warp layout
constexpr int kLoadWarp0 = kEpiWarps + kConvWarps;  // 20
constexpr int kMmaWarp = kLoadWarp0 + kLoadWarps;   // 24
constexpr int kThreads = (kMmaWarp + 1) * 32;       // 800
static_assert(kGroupThreads == kTileM, "one activation row (TMEM lane) per converter thread");
static_assert(kThreads * 80 <= 65536, "80 registers a thread for one CTA per SM");
constexpr int kEpiBar = 1 + kStages;  // the epilogue warps' named barrier
static_assert(kEpiBar < 16, "named barriers 1 .. kStages, kEpiBar");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemAStageCols = kKStep / 2;   // 64 fp16 of a row = 32 columns

// Tile geometry.  Normal: output tiles up to 192 wide with two TMEM
// accumulators, so the epilogue of one tile overlaps the MMAs of the next.
// BIG: one tile up to 320 wide per CTA (two MMAs per K slice beyond 256
// columns) with one accumulator: the activations of a k-step are widened once
// for 320 weight rows instead of 192, which pays when the tiles fit in one
// wave (the epilogue then overlaps nothing anyway).
template <bool BIG>
struct Shape {
  static constexpr int kTileNMax = BIG ? kMaxTileNBig : kMaxTileN;
  static constexpr int kAccBufs = BIG ? 1 : 2;
  static constexpr int kRing = BIG ? kRawStagesBig : kRawStages;
  static constexpr int kStageBytes = kTileNMax * 128;  // fp16 weights of a stage (activations live in TMEM)
  static constexpr int kRawStageBytes = kRawABytes + kTileNMax * 16;
  static constexpr int kSmemBytes = kStages * kStageBytes + kRing * kRawStageBytes;
  static constexpr uint32_t kTmemACol = (uint32_t)(kAccBufs * kTileNMax);  // activation stages follow
  static constexpr int kHalvesPerThread = (2 * kTileNMax + kGroupThreads - 1) / kGroupThreads;
  static_assert(kTmemACol + kStages * kTmemAStageCols <= kTmemCols, "TMEM budget");
  static_assert(kStageBytes % 1024 == 0 && kRawStageBytes % 16 == 0, "stage alignment");
  static_assert(kStages * kStageBytes >= kTileNMax * kTileM * 4, "split-K partial sums fit over the operand stages");
  static_assert(kSmemBytes + 1024 <= 227 * 1024, "shared memory");
};

// One weight matrix of a launch: the matrices share the activations, each has
// its own codes, scale, output and row count; its column tiles are the global
// column tiles tn0 .. tn0 + tiles_n - 1.
struct PrefillMat {
  const uint4* packed;
  const float* sw;
  float* y;
  int32_t* acc;
  int N;
  int tn0;
};

struct PrefillParams {
  CUtensorMap tmap_a;  // xq [M, K] int8: 64 x 128 boxes, 64-byte swizzle (the raw ring's layout)
  const int8_t* xq;
  const float* sx;
  int* status;
  int M, K, KB;
  int n_tile;      // multiple of 16, <= 192 (BIG: 320; SWAP: 128 weight rows a tile)
  int mma_n;       // MMA N = the rows of the shared-memory operand: n_tile, or (SWAP) tokens rounded up to 16
  int mma_n1;      // BIG, n_tile > 256: the first MMA of a K slice covers rows 0 .. mma_n1 - 1, the second the rest
  int tiles_m, tiles_n;  // tiles_n: column tiles of all matrices together
  int splits;      // K is split into this many ranges of KB k-steps (1 otherwise)
  int num_tiles;   // work units: tiles_m * tiles_n * splits
  int nmats;
  PrefillMat mats[kMaxDecodeMats];
};

struct SharedCtl {
  unsigned long long empty[kStages];  // stage s consumed (tcgen05.commit); "full" is named barrier 1 + s
  unsigned long long raw_full[kRawStages];
  unsigned long long raw_empty[kRawStages];
  unsigned long long tmem_full[2];
  unsigned long long tmem_empty[2];
  unsigned long long mma_done;
  unsigned long long parts_ready;  // split K: one arrival per other rank of the cluster
  uint32_t tmem_base;
  int abort_flag;
};

// Half of a packed chunk (words 2*half, 2*half+1: k = 32*half .. 32*half+31)
// -> fp16 chunks 4*half .. 4*half+3 of weight row r.
__device__ __forceinline__ void store_weight_half(uint32_t row_addr, int r, int half, const uint2 v) {
  uint32_t q[16];
  codes_to_f16x8(v.x, q);
  codes_to_f16x8(v.y, q + 8);
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    const int c = 4 * half + cc;
    st_shared_v4(row_addr + ((uint32_t)((c ^ (r & 7)) << 4)), q[4 * cc], q[4 * cc + 1], q[4 * cc + 2], q[4 * cc + 3]);
  }
}

// Work unit -> first token row, matrix, first weight row of that matrix and
// first k-block.
__device__ __forceinline__ void tile_coords(const PrefillParams& p, int unit, int& m0, int& mi, int& n0, int& kb0) {
  const int tile = unit / p.splits;
  kb0 = (unit - tile * p.splits) * p.KB;
  const int tm = tile % p.tiles_m;
  const int tn = tile / p.tiles_m;
  mi = 0;
#pragma unroll
  for (int i = 1; i < kMaxDecodeMats; ++i)
    if (i < p.nmats && tn >= p.mats[i].tn0) mi = i;
  m0 = tm * kTileM;
  n0 = (tn - p.mats[mi].tn0) * p.n_tile;
}

// SWAP = false: A (TMEM) = 128 token rows, B (shared) = n_tile weight rows.
// SWAP = true (few tokens): A = 128 weight rows, B = every token (M <= 128),
// so the weights pass through the tensor cores once.  The loader is the same
// (token rows 0 .. 127 of the activations, weight rows n0 .. n0 + 127).
template <bool SWAP, bool BIG>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillParams p) {
  using S = Shape<BIG>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ SharedCtl ctl;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // 1024-byte aligned stage buffers (the swizzle pattern follows address bits)
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t stage_base = (raw_addr + 1023u) & ~1023u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl.empty[s], 1);
    }
    for (int s = 0; s < S::kRing; ++s) {
      mbar_init(&ctl.raw_full[s], 2);  // the activation and the code loader
      mbar_init(&ctl.raw_empty[s], kGroupWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctl.tmem_full[s], 1);
      mbar_init(&ctl.tmem_empty[s], kEpiWarps);
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

  // Let the next kernel on the stream start as SM resources free up; it still
  // waits for this grid's results.
  pdl_release_dependents();

  const uint32_t raw_base = stage_base + (uint32_t)kStages * S::kStageBytes;
  const int my_tiles = (int)blockIdx.x < p.num_tiles ? (p.num_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int total = my_tiles * p.KB;  // flat k-steps of this CTA, tile-major

  if (warp >= kLoadWarp0 && warp < kMmaWarp) {
    // ------------------------------------------------------------------ loaders
    // Per k-step one TMA tensor copy of the 128 x 64 int8 activation tile
    // (64-byte swizzle: piece q of row r at q ^ ((r / 2) % 4); rows past M read
    // as zeros), issued by warp 20, and one bulk copy of the packed codes of the
    // tile's rows, issued by warp 21.  Each issuing thread arms the slot's
    // barrier with its own bytes (two arrivals a phase): one thread issuing
    // both copies took about 0.1 us a copy, which bounded the k-step.
    // The packed codes do not come from the previous kernel on the stream:
    // only the activation loader waits for it (the codes of the first ring
    // slots are requested while that kernel finishes).
    if (warp == kLoadWarp0) pdl_wait_primary();
    if ((warp == kLoadWarp0 || warp == kLoadWarp0 + 1) && lane == 0) {
      const bool codes = warp != kLoadWarp0;
      int ks = 0, tile = blockIdx.x;
      int m0 = 0, mi = 0, n0 = 0, kb0 = 0;
      uint32_t code_bytes = 0;
      auto start_tile = [&]() {
        tile_coords(p, tile, m0, mi, n0, kb0);
        const int Nm = p.mats[mi].N;
        const int rows = Nm - n0 < p.n_tile ? Nm - n0 : p.n_tile;  // rows past N are not read
        code_bytes = (uint32_t)rows * 16u;
      };
      if (total > 0) start_tile();
      int last = -1;
      for (int f = 0; f < total; ++f) {
        const int slot = f % S::kRing;
        const uint32_t use = (uint32_t)(f / S::kRing);
        if (!mbar_wait(&ctl.raw_empty[slot], (use & 1u) ^ 1u, &ctl.abort_flag, p.status)) break;
        const uint32_t raw = raw_base + (uint32_t)slot * S::kRawStageBytes;
        if (codes) {
          mbar_arrive_expect_tx(&ctl.raw_full[slot], code_bytes);
          bulk_copy_g2s(raw + kRawABytes, p.mats[mi].packed + ((int64_t)(kb0 + ks) * p.mats[mi].N + n0), code_bytes,
                        &ctl.raw_full[slot]);
        } else {
          mbar_arrive_expect_tx(&ctl.raw_full[slot], (uint32_t)kRawABytes);
          const int kx = (kb0 + ks) * kKStep;  // a multiple of 64 bytes
          asm volatile(
              "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
              ::"r"(raw), "l"(reinterpret_cast<uint64_t>(&p.tmap_a)), "r"(kx), "r"(m0),
                "r"(smem_u32(&ctl.raw_full[slot]))
              : "memory");
        }
        last = f;
        if (++ks == p.KB) {
          ks = 0;
          tile += gridDim.x;
          if (f + 1 < total) start_tile();
        }
      }
      // No copy may outlive the CTA: wait (bounded) for the last fills.
      for (int f = last; f >= 0 && f > last - S::kRing; --f)
        mbar_drain(&ctl.raw_full[f % S::kRing], (uint32_t)((f / S::kRing) & 1), p.status);
    }
    __syncwarp();
  } else if (warp >= kEpiWarps && warp < kLoadWarp0) {
    // ------------------------------------------------------------------ converters
    // Group g (4 warps) converts the flat k-steps f = g, g + kStages, ... into
    // stage g, so the groups work on different k-steps at once.  Thread u of a
    // group widens activation row u (its warp's TMEM lanes are rows 32(u/32)
    // ..) and weight half-rows u + 128j (half h of row r: k = 32h .. 32h+31 of
    // the row's packed chunk).
    const int cw = warp - kEpiWarps;
    const int grp = cw / kGroupWarps;
    const int u = (cw % kGroupWarps) * 32 + lane;  // 0 .. 127
    const int nh = 2 * p.n_tile;                   // weight half-rows, <= 512
    const int npieces = p.mma_n * 4;               // SWAP: 16-byte token pieces
    int cks = grp, ctile = blockIdx.x;             // k-step f as (tile, k-step in tile)
    while (cks >= p.KB) { cks -= p.KB; ctile += gridDim.x; }
    int cm0, cmi, n0, ckb0;
    tile_coords(p, ctile, cm0, cmi, n0, ckb0);
    int Nm = p.mats[cmi].N;
    // Every k-step this group owns ends with its arrival on the stage's named
    // barrier, after an abort too (without the work), and never before the
    // stage's previous MMAs were committed (a wait that ignores the abort flag;
    // the MMA warp keeps committing after an abort): so each phase of the
    // barrier holds one k-step's converters and the MMA warp's sync of that
    // k-step, and the MMA warp's syncs, which cannot time out, always complete.
    bool live = true;
    for (int f = grp; f < total; f += kConvGroups) {
      const int slot = f % S::kRing;
      const uint32_t use = (uint32_t)(f / S::kRing);
      const uint32_t fill = (uint32_t)(f / kConvGroups);  // earlier fills of this stage
      const bool stage_free = mbar_wait_lockstep(&ctl.empty[grp], (fill & 1u) ^ 1u, &ctl.abort_flag, p.status);
      live = live && stage_free && mbar_wait(&ctl.raw_full[slot], use & 1u, &ctl.abort_flag, p.status);
      if (!live) {
        named_bar_arrive(1 + grp, kGroupThreads + 32);
        continue;
      }
      const uint32_t raw = raw_base + (uint32_t)slot * S::kRawStageBytes;
      tc_fence_after();  // the MMAs that read this stage are complete
      const uint32_t b_tile = stage_base + (uint32_t)grp * S::kStageBytes;
      if constexpr (SWAP) {
        // Weights: row u of the tile (its 64 codes of this k-block) -> TMEM lane u;
        // rows past N (not copied) are zeros.
        const uint4 wv = n0 + u < Nm ? ld_shared_v4(raw + kRawABytes + (uint32_t)(u * 16))
                                     : make_uint4(0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u);
        const uint32_t t_addr = tmem_base + ((uint32_t)((u >> 5) * 32) << 16) + S::kTmemACol +
                                (uint32_t)grp * kTmemAStageCols;
        uint32_t cols[16];
        codes_to_f16x8(wv.x, cols);
        codes_to_f16x8(wv.y, cols + 8);
        tmem_st16(t_addr, cols);
        codes_to_f16x8(wv.z, cols);
        codes_to_f16x8(wv.w, cols + 8);
        tmem_st16(t_addr + 16u, cols);
        // Tokens: piece q of token row r (16 int8) -> fp16 chunks 2q, 2q+1 of row r.
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int pc = u + j * kGroupThreads;
          if (pc >= npieces) continue;
          const int row = pc >> 2, q = pc & 3;
          const uint4 av = ld_shared_v4(raw + (uint32_t)(row * kKStep + ((q ^ ((row >> 1) & 3)) << 4)));
          const uint32_t row_addr = b_tile + (uint32_t)row * 128u;
          const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t l0, h0, l1, h1;
            i8x4_to_f16x4(aw[2 * half], l0, h0);
            i8x4_to_f16x4(aw[2 * half + 1], l1, h1);
            const int c = 2 * q + half;
            st_shared_v4(row_addr + ((uint32_t)((c ^ (row & 7)) << 4)), l0, h0, l1, h1);
          }
        }
      } else {
        // Activations: row u of the tile -> TMEM lane u, columns of stage grp;
        // weight half-rows h = u + 128 j.  Every shared-memory read of the
        // k-step is issued before the first conversion (the wrappers are
        // volatile, so program order is issue order), so their latencies
        // overlap instead of adding up.
        const uint32_t row_raw = raw + (uint32_t)(u * kKStep);
        const uint32_t sw = (uint32_t)((u >> 1) & 3);
        const uint32_t t_addr = tmem_base + ((uint32_t)((u >> 5) * 32) << 16) + S::kTmemACol +
                                (uint32_t)grp * kTmemAStageCols;
        uint4 av[4];
#pragma unroll
        for (int piece = 0; piece < 4; ++piece) av[piece] = ld_shared_v4(row_raw + (((uint32_t)piece ^ sw) << 4));
        uint2 wv[S::kHalvesPerThread];
#pragma unroll
        for (int j = 0; j < S::kHalvesPerThread; ++j) {
          const int h = u + j * kGroupThreads;
          wv[j] = (h < nh && n0 + (h >> 1) < Nm) ? ld_shared_v2(raw + kRawABytes + (uint32_t)(h * 8)) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int hpair = 0; hpair < 2; ++hpair) {  // pieces 2h, 2h+1 -> columns 16h .. 16h+15
          uint32_t cols[16];
#pragma unroll
          for (int pi = 0; pi < 2; ++pi) {
            const uint4 a = av[2 * hpair + pi];
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) i8x4_to_f16x4(aw[j], cols[8 * pi + 2 * j], cols[8 * pi + 2 * j + 1]);
          }
          tmem_st16(t_addr + (uint32_t)(16 * hpair), cols);
        }
#pragma unroll
        for (int j = 0; j < S::kHalvesPerThread; ++j) {
          const int h = u + j * kGroupThreads;
          if (h >= nh) continue;
          const int row = h >> 1, half = h & 1;
          const uint32_t row_addr = b_tile + (uint32_t)row * 128u;
          if (n0 + row < Nm) {
            store_weight_half(row_addr, row, half, wv[j]);
          } else {  // rows past N are zeros
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) st_shared_v4(row_addr + (uint32_t)((4 * half + cc) << 4), 0u, 0u, 0u, 0u);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.raw_empty[slot]);  // one arrival per warp
      named_bar_arrive(1 + grp, kGroupThreads + 32);
      cks += kConvGroups;
      if (cks >= p.KB) {
        while (cks >= p.KB) { cks -= p.KB; ctile += gridDim.x; }
        tile_coords(p, ctile, cm0, cmi, n0, ckb0);
        Nm = p.mats[cmi].N;
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp takes each stage's named barrier; lane 0 issues.  (An
    // mbarrier wait or any shared-memory load by the issuing thread returned
    // only after its in-flight MMAs had drained, which idled the tensor pipe
    // between k-steps; a named barrier does not.)  After an abort the warp
    // still syncs and commits every k-step (issuing nothing), so the
    // converters, which wait for those commits, stay in step with it.
    {
      // BIG tiles wider than 256 take two MMAs a K slice (rows 0 .. mma_n1 - 1,
      // then the rest: B 128 bytes a row further, D mma_n1 columns further).
      const bool two = BIG && p.mma_n1 > 0;
      const int n1 = two ? p.mma_n1 : p.mma_n;
      const uint32_t idesc = make_idesc(kTileM, n1);
      const uint32_t idesc2 = make_idesc(kTileM, two ? p.mma_n - n1 : 16);
      int stage = 0;
      bool aborted = false;
      int it = 0;
      for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
        const int slot = it % S::kAccBufs;
        const uint32_t use = (uint32_t)(it / S::kAccBufs);
        // lane 0 decides for the warp
        bool ab = aborted || *reinterpret_cast<volatile int*>(&ctl.abort_flag) != 0;
        if (!ab && lane == 0) ab = !mbar_wait(&ctl.tmem_empty[slot], (use & 1u) ^ 1u, &ctl.abort_flag, p.status);
        aborted = __shfl_sync(0xffffffffu, ab ? 1 : 0, 0) != 0;
        const uint32_t d_tmem = tmem_base + (uint32_t)(slot * S::kTileNMax);
        for (int ks = 0; ks < p.KB; ++ks) {
          named_bar_sync(1 + stage, kGroupThreads + 32);
          if (lane == 0) {
            if (!aborted) {
              tc_fence_after();
              const uint32_t a_tmem = tmem_base + S::kTmemACol + (uint32_t)stage * kTmemAStageCols;
              const uint64_t b_desc = smem_desc_sw128(stage_base + (uint32_t)stage * S::kStageBytes);
#pragma unroll
              for (int kk = 0; kk < kKStep / 16; ++kk) {
                // 16 fp16 along K: 8 TMEM columns of A, 32 bytes inside B's swizzle atom
                mma_f16_ta(d_tmem, a_tmem + (uint32_t)(kk * 8), b_desc + (uint64_t)(kk * 2), idesc,
                           (ks | kk) != 0 ? 1u : 0u);
                if (two)  // rows n1 ..: 8-row swizzle atoms of 1024 bytes further (n1 is a multiple of 16)
                  mma_f16_ta(d_tmem + (uint32_t)n1, a_tmem + (uint32_t)(kk * 8),
                             b_desc + (uint64_t)(n1 * 8 + kk * 2), idesc2, (ks | kk) != 0 ? 1u : 0u);
              }
            }
            mma_commit(&ctl.empty[stage]);
          }
          __syncwarp();
          if (++stage == kStages) stage = 0;
        }
        if (lane == 0) mma_commit(&ctl.tmem_full[slot]);
      }
    }
    if (lane == 0) {
      // All MMAs this thread issued must be complete before TMEM is freed.
      mma_commit(&ctl.mma_done);
      mbar_drain(&ctl.mma_done, 0u, p.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue
    pdl_wait_primary();  // sx comes from the previous kernel, which may still read y
    const int row = warp * 32 + lane;  // TMEM lane = row of the tile
    int it = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
      int m0, mi, n0, kb0;
      tile_coords(p, tile, m0, mi, n0, kb0);
      const PrefillMat& mat = p.mats[mi];
      const float sw = *mat.sw;
      const int N = mat.N;
      const int slot = it % S::kAccBufs;
      const uint32_t use = (uint32_t)(it / S::kAccBufs);
      if (!mbar_wait(&ctl.tmem_full[slot], use & 1u, &ctl.abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)(slot * S::kTileNMax);
      if (p.splits > 1) {
        // Split K (one unit per CTA; the units of a tile are one cluster, rank
        // = K range): this rank's exact partial sums go to its own shared
        // memory, column-major by TMEM lane ([column][128]), over the operand
        // stages, which no MMA reads any more.
        const int ncols = SWAP ? p.mma_n : p.n_tile;
        for (int c = 0; c < ncols; c += 16) {
          uint32_t r[16];
          tmem_ld16(t_row + (uint32_t)c, r);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(stage_base + (uint32_t)(((c + j) * kTileM + row) * 4)),
                         "r"(__float2int_rn(__uint_as_float(r[j])))
                         : "memory");
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.tmem_empty[slot]);
        break;
      }
      if constexpr (SWAP) {
        // TMEM lane = weight row n, column t = token t: y[t, n] for t < M
        // (a warp writes 32 consecutive n of one token).
        const int n = n0 + row;
        const bool n_ok = n < N;
        for (int c = 0; c < p.mma_n; c += 16) {
          uint32_t r[16];
          tmem_ld16(t_row + (uint32_t)c, r);
          if (!n_ok) continue;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = c + j;
            if (t < p.M) {
              const float a = __uint_as_float(r[j]);  // an exact integer
              mat.y[(int64_t)t * N + n] = __fdiv_rn(a, __fmul_rn(p.sx[t], sw));
              if (mat.acc) mat.acc[(int64_t)t * N + n] = __float2int_rn(a);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.tmem_empty[slot]);  // one arrival per warp
        continue;
      }
      const int m = m0 + row;
      const bool row_ok = m < p.M;
      const float den = row_ok ? __fmul_rn(p.sx[m], sw) : 1.0f;
      float* yrow = mat.y + (int64_t)(row_ok ? m : 0) * N;
      int32_t* arow = mat.acc ? mat.acc + (int64_t)(row_ok ? m : 0) * N : nullptr;
      for (int c = 0; c < p.n_tile; c += 16) {
        uint32_t r[16];
        tmem_ld16(t_row + (uint32_t)c, r);
        const int n = n0 + c;
        if (!row_ok || n >= N) continue;
        float yv[16];
        int av[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float a = __uint_as_float(r[j]);  // an exact integer
          yv[j] = __fdiv_rn(a, den);
          av[j] = __float2int_rn(a);
        }
        if (n + 16 <= N && ((((uintptr_t)(yrow + n)) & 15u) == 0)) {
          float4* dst = reinterpret_cast<float4*>(yrow + n);
#pragma unroll
          for (int j = 0; j < 4; ++j) dst[j] = make_float4(yv[4 * j], yv[4 * j + 1], yv[4 * j + 2], yv[4 * j + 3]);
          if (arow) {
            int4* ad = reinterpret_cast<int4*>(arow + n);
#pragma unroll
            for (int j = 0; j < 4; ++j) ad[j] = make_int4(av[4 * j], av[4 * j + 1], av[4 * j + 2], av[4 * j + 3]);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (n + j < N) {
              yrow[n + j] = yv[j];
              if (arow) arow[n + j] = av[j];
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.tmem_empty[slot]);  // one arrival per warp
    }
    if (p.splits > 1 && (int)blockIdx.x < p.num_tiles) {
      // Every rank adds one share of the tile's columns over all ranks'
      // partial sums (distributed shared memory) and writes those outputs.
      // Every rank takes part whatever happened before, so the others' waits
      // end early.
      named_bar_sync(kEpiBar, kEpiWarps * 32);  // this rank's partial sums are written
      const uint32_t rank = cluster_rank();
      if (warp == 0 && lane < p.splits && lane != (int)rank)
        mbar_arrive_remote(map_shared(smem_u32(&ctl.parts_ready), (uint32_t)lane));
      if (mbar_wait_cluster(&ctl.parts_ready, 0u, &ctl.abort_flag, p.status) &&
          *reinterpret_cast<volatile int*>(&ctl.abort_flag) == 0) {
        int m0, mi, n0, kb0;
        tile_coords(p, blockIdx.x, m0, mi, n0, kb0);
        const PrefillMat& mat = p.mats[mi];
        const float sw = *mat.sw;
        const int N = mat.N;
        const int ncols = SWAP ? p.mma_n : p.n_tile;
        const int c0 = (int)rank * ncols / p.splits, c1 = ((int)rank + 1) * ncols / p.splits;
        // item: column c, TMEM lanes l4 .. l4 + 3
        for (int it = c0 * (kTileM / 4) + warp * 32 + lane; it < c1 * (kTileM / 4); it += kEpiWarps * 32) {
          const int c = it / (kTileM / 4), l4 = (it % (kTileM / 4)) * 4;
          const uint32_t off = stage_base + (uint32_t)((c * kTileM + l4) * 4);
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
          const int av[4] = {(int)tot.x, (int)tot.y, (int)tot.z, (int)tot.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            // SWAP: lane = weight row, column = token; else lane = token, column = weight row
            const int t = SWAP ? c : m0 + l4 + e;
            const int n = SWAP ? n0 + l4 + e : n0 + c;
            if (t < p.M && n < N) {
              mat.y[(int64_t)t * N + n] = __fdiv_rn(__int2float_rn(av[e]), __fmul_rn(p.sx[t], sw));
              if (mat.acc) mat.acc[(int64_t)t * N + n] = av[e];
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



}  // namespace

namespace {

template <bool SWAP, bool BIG>
cudaError_t configure(const DeviceInfo& dev) {
  static thread_local int configured = -1;
  if (configured != dev.device) {
    cudaError_t err = cudaFuncSetAttribute(prefill_kernel<SWAP, BIG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           Shape<BIG>::kSmemBytes + 1024);
    if (err != cudaSuccess) return err;
    configured = dev.device;
  }
  return cudaSuccess;
}

template <bool BIG>
cudaLaunchConfig_t launch_config(int grid, int cluster, bool pdl, cudaStream_t stream, cudaLaunchAttribute (&attr)[2]) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)Shape<BIG>::kSmemBytes + 1024;
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

// Clusters of `size` CTAs of this kernel that fit on the GPU at once (0 on
// error); cached per device and size.
template <bool SWAP, bool BIG>
int max_clusters(int size, const DeviceInfo& dev) {
  static thread_local int cache_dev = -1;
  static thread_local int cache[kMaxSplits + 1];
  if (cache_dev != dev.device) {
    for (int i = 0; i <= kMaxSplits; ++i) cache[i] = -1;
    cache_dev = dev.device;
  }
  if (cache[size] < 0) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = launch_config<BIG>(size, size, false, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, prefill_kernel<SWAP, BIG>, &cfg) != cudaSuccess) n = 0;
    cache[size] = n;
  }
  return cache[size];
}

template <bool SWAP, bool BIG>
cudaError_t launch_impl(const PrefillParams& p, bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  cudaError_t err = configure<SWAP, BIG>(dev);
  if (err != cudaSuccess) return err;
  const int grid = p.splits > 1 ? p.num_tiles : (p.num_tiles < dev.num_sms ? p.num_tiles : dev.num_sms);
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_config<BIG>(grid, p.splits, pdl, stream, attr);
  return cudaLaunchKernelEx(&cfg, prefill_kernel<SWAP, BIG>, p);
}

// Split K (into a divisor of the k-block count, at most kMaxSplits: a portable
// cluster) when there are too few tiles to fill the SMs: minimise the k-steps
// of the busiest CTA.  The units of a tile run as one thread-block cluster;
// each rank adds a share of the tile's columns over all ranks' partial sums
// (distributed shared memory), so every cluster must be resident at once (at
// most `clusters[sp]` of them).
int best_split(int64_t tiles, int KB, int num_sms, int64_t* cost_out, const int* clusters = nullptr) {
  int best_s = 1;
  int64_t best_cost = -1;
  // A split keeps every unit in one wave and at least 8 k-steps long (each
  // unit pays a pipeline fill and the reduction).
  for (int sp = 1; sp <= kMaxSplits && sp <= KB && (sp == 1 || 2 * tiles <= num_sms); ++sp) {
    if (KB % sp) continue;
    if (sp > 1 && (tiles * sp > num_sms || KB / sp < 8)) continue;
    if (sp > 1 && clusters && tiles > clusters[sp]) continue;
    const int64_t units = tiles * sp;
    const int64_t waves = (units + num_sms - 1) / num_sms;
    const int64_t cost = waves * (KB / sp) + (sp > 1 ? 2 : 0);  // + the reduction
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_s = sp;
    }
  }
  if (cost_out) *cost_out = best_cost;
  return best_s;
}

template <bool SWAP, bool BIG>
cudaError_t launch_split(PrefillParams& p, bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  cudaError_t err = configure<SWAP, BIG>(dev);
  if (err != cudaSuccess) return err;
  const int KB = p.KB;
  const int64_t tiles = (int64_t)p.tiles_m * p.tiles_n;
  int clusters[kMaxSplits + 1] = {0};
  if (2 * tiles <= dev.num_sms)
    for (int sp = 2; sp <= kMaxSplits; ++sp) clusters[sp] = max_clusters<SWAP, BIG>(sp, dev);
  const int best_s = best_split(tiles, KB, dev.num_sms, nullptr, clusters);
  p.splits = best_s;
  p.KB = KB / best_s;
  p.num_tiles = (int)(tiles * best_s);
  return launch_impl<SWAP, BIG>(p, pdl, dev, stream);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

PrefillParams common_params(const int8_t* xq, const float* sx, int64_t M, const DecodeMatrix* mats, int nmats,
                            int64_t K, const DeviceInfo& dev) {
  PrefillParams p;
  p.KB = 0;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K};
    const cuuint32_t box[2] = {(cuuint32_t)kKStep, (cuuint32_t)kTileM};
    const cuuint32_t estr[2] = {1, 1};
    EncodeTiledFn fn = encode_fn();
    if (!fn || fn(&p.tmap_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(xq), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      p.KB = -1;  // reported by the launchers
  }
  p.xq = xq;
  p.sx = sx;
  p.status = dev.status;
  p.M = (int)M;
  p.K = (int)K;
  p.nmats = nmats;
  for (int i = 0; i < kMaxDecodeMats; ++i) {
    PrefillMat& m = p.mats[i];
    if (i < nmats) {
      m.packed = reinterpret_cast<const uint4*>(mats[i].packed);
      m.sw = mats[i].w_scale;
      m.y = mats[i].y;
      m.acc = mats[i].acc;
      m.N = (int)mats[i].N;
    } else {
      m = PrefillMat{nullptr, nullptr, nullptr, nullptr, 0, 1 << 30};
    }
  }
  if (p.KB != -1) p.KB = (int)(K / kKStep);
  return p;
}

// Column tiles of n_tile rows: each matrix starts a new tile.
int64_t column_tiles(const DecodeMatrix* mats, int nmats, int64_t n_tile) {
  int64_t t = 0;
  for (int i = 0; i < nmats; ++i) t += (mats[i].N + n_tile - 1) / n_tile;
  return t;
}

void assign_tiles(PrefillParams& p, const DecodeMatrix* mats, int nmats) {
  int tn = 0;
  for (int i = 0; i < nmats; ++i) {
    p.mats[i].tn0 = tn;
    tn += (int)((mats[i].N + p.n_tile - 1) / p.n_tile);
  }
  p.tiles_n = tn;
}

}  // namespace


// The matrices share xq and K; one launch covers all of their tiles.
cudaError_t launch_prefill_mats(const int8_t* xq, const float* sx, int64_t M, const DecodeMatrix* mats, int nmats,
                                int64_t K, bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  if (nmats < 1 || nmats > kMaxDecodeMats) return cudaErrorInvalidValue;
  PrefillParams p = common_params(xq, sx, M, mats, nmats, K, dev);
  if (p.KB < 0) return cudaErrorNotSupported;
  // Tile width and K split together: the fewest (k-steps of the busiest CTA)
  // x (tile width + 64), the +64 being the activation widening of a k-step;
  // a split also pays its fill and its partial-sum exchange, which grows with
  // the tile width (128 x width fp32 per rank): 1024 + 16 x width.  (With a
  // flat 1024 the planner split 320-wide tiles four ways where plain 80-wide
  // tiles run twice as fast: 10240 x 2560 at M = 32 took 39.6 us against
  // 20.1, 256 x 2560 x 2560 21.8 against 17.5, 1024 x 2048 x 8192 68.2 against
  // 48.2, on GB300.)
  // 320-wide single-accumulator tiles only when every CTA has one tile: a
  // CTA with more would run each tile's epilogue with no MMAs beside it (the
  // up shape at M = 2048 took 144 us that way against 108).
  const int64_t tiles_m = (M + kTileM - 1) / kTileM;
  int64_t best = -1;
  bool big = false;
  p.n_tile = kMaxTileN;
  for (int nt = kMaxTileNBig; nt >= 64; nt -= 16) {
    int64_t ksteps = 0;
    const int64_t tiles = tiles_m * column_tiles(mats, nmats, nt);
    const bool is_big = nt > kMaxTileN;
    if (is_big && tiles > dev.num_sms) continue;
    const int sp = best_split(tiles, p.KB, dev.num_sms, &ksteps);
    const int64_t cost = ksteps * (nt + 64) + (sp > 1 ? 4 * 256 + 16 * nt : 0);
    if (best < 0 || cost < best) {
      best = cost;
      p.n_tile = nt;
      big = is_big;
    }
  }
  p.mma_n = p.n_tile;
  // two MMAs a K slice beyond 256 columns: halves rounded to 16 rows
  p.mma_n1 = p.n_tile > 256 ? (p.n_tile / 2 + 15) / 16 * 16 : 0;
  p.tiles_m = (int)tiles_m;
  assign_tiles(p, mats, nmats);
  return big ? launch_split<false, true>(p, pdl, dev, stream) : launch_split<false, false>(p, pdl, dev, stream);
}

cudaError_t launch_prefill(const int8_t* xq, const float* sx, int64_t M, const uint8_t* packed,
                           const float* sw, int64_t N, int64_t K, float* y, int32_t* acc,
                           bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  const DecodeMatrix m = {packed, sw, N, y, acc};
  return launch_prefill_mats(xq, sx, M, &m, 1, K, pdl, dev, stream);
}

// 1 <= M <= 128: 128-row weight tiles on the M side of the MMA, all tokens on
// its N side (rounded up to 16; token rows past M are zeros).
cudaError_t launch_batched_mats(const int8_t* xq, const float* sx, int64_t M, const DecodeMatrix* mats, int nmats,
                                int64_t K, bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  if (M < 1 || M > kTileM || nmats < 1 || nmats > kMaxDecodeMats) return cudaErrorInvalidValue;
  PrefillParams p = common_params(xq, sx, M, mats, nmats, K, dev);
  if (p.KB < 0) return cudaErrorNotSupported;
  p.n_tile = kTileM;
  p.mma_n = (int)((M + 15) / 16 * 16);
  p.tiles_m = 1;
  assign_tiles(p, mats, nmats);
  p.mma_n1 = 0;
  return launch_split<true, false>(p, pdl, dev, stream);
}

cudaError_t launch_batched(const int8_t* xq, const float* sx, int64_t M, const uint8_t* packed,
                           const float* sw, int64_t N, int64_t K, float* y, int32_t* acc,
                           bool pdl, const DeviceInfo& dev, cudaStream_t stream) {
  const DecodeMatrix m = {packed, sw, N, y, acc};
  return launch_batched_mats(xq, sx, M, &m, 1, K, pdl, dev, stream);
}

}  // namespace bitlinear
