// tc_gemm.cu -- persistent, warp-specialised TMA + tcgen05 GEMM with a fused epilogue (sm_103a).
//
// One CTA per SM walks output tiles of BM x BN = 128 x 256 in grouped-M order (tile_order.h), or,
// in the CTA-pair form (PAIR), one 2-CTA cluster per SM pair walks 256 x 256 tiles: each CTA
// stages its own 128 rows of A and half (128 columns) of B, the even CTA issues
// tcgen05.mma.cta_group::2 (M = 256) for both, and each CTA's TMEM receives its 128 rows.  The pair
// halves the B bytes each SM fetches per MMA.  fp16 / bf16 operands use kind::f16, fp8 e4m3
// operands kind::f8f6f4; one "K row" of a stage is 128 bytes of K per operand row either way.
//   warp 0      TMA producer: per stage, A as KSUB boxes of 128 rows x one K row (K-major) and
//               B as 128-byte-wide boxes of KSUB K rows (N-major), into a shared-memory ring as
//               deep as the epilogue's buffers allow (three 64 KB stages with two K rows on pairs,
//               else up to six of 32 KB); completion counted in bytes on full[s] (with fp8
//               operands and staged Y, a full barrier per K row of the stage, B then copied one
//               K row at a time, so the first row's MMAs start while the second lands; the fp8
//               column pieces of the last round on pairs, 64 columns per CTA, take B as
//               64-byte-wide boxes with 64-byte swizzle); out-of-range
//               rows / columns / K are zero-filled by TMA, which is the M/N/K tail mask of
//               "I3. Fuse a GEMM epilogue and change tile scheduling" ("Tiles and grouped
//               ownership": A's M/K edges, B's K/N edges).
//   warp 1      MMA issuer (one thread): fp32 accumulate in tensor memory, 128 x 256 accumulator
//               per CTA, double-buffered (2 x 256 of the 512 TMEM columns) so the epilogue of tile
//               i overlaps the main loop of tile i + 1.  The MMA's N is the work item's width: 256,
//               or less for the pieces of the last partial round and for the last column of tiles
//               (narrowed to the columns left of N).  tcgen05.commit releases each smem stage
//               (empty[s]) and hands a finished accumulator over (acc_full[b]).
//   warps 2-9   epilogue, two warpgroups splitting the tile's columns (or warps 2-17, four
//               warpgroups of 64 columns, as an option for single CTAs with staged Y): each warp
//               owns the 32 TMEM lanes (rows) its warp id allows, reads its bias with one coalesced load
//               per work item (shuffled to the granules), and per 64-column chunk:
//               tcgen05.ld -> + bias[j] -> ReLU (fmaxf), the gate fma(x, y, x), the residual, or
//               the fp8 scale-and-clamp -> one round-to-nearest conversion -> 128-byte-swizzled
//               staging buffer -> one TMA store, which clips rows >= M and columns >= N (the store
//               mask).  The bias is added after the reduction ("Triton: Fused Matmul + Bias + ReLU
//               (Epilogue Fusion)", "Pitfalls": after the K loop, masked with j < N), or, with the
//               bias-initialised accumulator ("Optimizing GEMM + Activation on CDNA4 with TLX",
//               V4; the default for short K loops), written into the free TMEM buffer before its
//               tile's first MMA, or set there by one extra MMA (a 128 x 16 tile of ones times a
//               16-row tile whose first K row is the bias row, staged by TMA).  For the gate (and the residual add, "Variants") the second
//               M x N operand is prefetched by TMA into the epilogue's own buffers while the main
//               loop runs (a whole 8 KB block per warp a work item ahead, or one 4 KB chunk at a
//               time on long K loops), and the result is written over it and stored from there;
//               with fp32 outputs it is loaded straight into registers ahead of the TMEM read.
// The accumulator goes from TMEM to registers to the single store; it never touches HBM.
#include <atomic>
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_order.h"

namespace fgemm {
namespace tc {

constexpr int BM = 128, BN = 256;  // per-CTA rows, tile columns
// Epilogue warps: EW = 8 (two warpgroups, each owning half (128) of a tile's columns) or 16 (four
// warpgroups of 64 columns each; single CTAs with a staged Y block per warp).  Threads per CTA:
__host__ __device__ constexpr int threads_for(int ew) { return 64 + 32 * ew; }
constexpr int THREADS = threads_for(8);  // the pair kernels
// One K row of a stage is one 128-byte swizzle row per operand row: 64 16-bit or 128 fp8 elements.
constexpr uint32_t A_ROW_BYTES = BM * 128;       // 16 KB: A's 128 rows x one K row
constexpr uint32_t B_ROW_BYTES = 128 * 128;      // 16 KB: one K row of B for 128 columns
constexpr uint32_t EPI_BUF_BYTES = 32 * 128;     // 32 rows x 128 bytes
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SMEM_LIMIT = 232448;          // dynamic shared memory per CTA
constexpr int MAX_STAGES = 6;

// YS: the gate's Y is staged through shared memory by TMA (16-bit outputs), which costs one ring
// stage of shared memory for a 64 KB Y / output block.  YB = 2 (CTA pairs, short K loops) keeps two
// such blocks per epilogue warp, so that Y is fetched two tiles ahead, in exchange for three stages
// of the ring: with few K blocks per tile the epilogue's streams of Y and out, not the main loop,
// set the pace.
// KSUB: K rows per stage (1 or 2).  A stage holds KSUB x 128 bytes of K for every operand row,
// so two K rows halve the number of stage hand-offs (TMA completion -> MMA -> release -> reload)
// per byte, at the price of half as many, twice as large stages in the same shared memory.
// The ring takes whatever the epilogue's buffers leave, up to MAX_STAGES stages.
// MB: room for the bias-initialised accumulator set by one extra MMA ("Optimizing GEMM +
// Activation on CDNA4 with TLX", V4: the accumulator starts at the bias): a 128 x 16 tile of ones
// (A, K-major, no swizzle) and a 16-row tile of B whose first K row is the bias of the work item's
// columns and whose other rows are zero (B's own MN-major, 128-byte-swizzled layout, 16 K rows per
// 64-column box).  ones x that tile = the bias in every row, exactly (16-bit bias, products by 1).
constexpr uint32_t ONES_BYTES = 4096;             // 128 rows x 16 K of 16-bit ones
constexpr uint32_t BIAS_BOX_BYTES = 16 * 128;     // 16 K rows x 64 columns of 16-bit values
template <bool PAIR, bool YS = false, int YB = 1, int KSUB = 1, bool MB = false, int EW = 8>
struct Cfg {
  static constexpr int EPI_WARPS = EW;
  static constexpr int COLS_W = BN / (EW / 4);  // tile columns per epilogue warp
  static_assert(YB == 1 || (YB == 2 && YS) || (YB == 0 && PAIR && YS),
                "Y staging variants: staged Y (chunk at a time on CTA pairs only)");
  static_assert(KSUB == 1 || KSUB == 2, "one or two K rows per stage");
  static constexpr uint32_t A_STAGE_BYTES = KSUB * A_ROW_BYTES;
  static constexpr uint32_t B_STAGE_BYTES = KSUB * (PAIR ? 1 : 2) * B_ROW_BYTES;  // this CTA's columns
  static constexpr uint32_t STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
  static constexpr int TILE_M = PAIR ? 2 * BM : BM;
  // per epilogue warp: its 32 x 128 block of Y and results (YS), or one 32-row staging buffer
  static constexpr uint32_t Y_BLOCK_BYTES = (COLS_W / 64) * EPI_BUF_BYTES;  // a warp's block of Y
  // YB = 0 (staged Y): one 32 x 64 chunk of Y at a time per warp
  static constexpr uint32_t EPI_WARP_BYTES = YS ? (YB == 0 ? EPI_BUF_BYTES : YB * Y_BLOCK_BYTES) : EPI_BUF_BYTES;
  static constexpr uint32_t MB_BYTES = MB ? ONES_BYTES + (PAIR ? 2u : 4u) * BIAS_BOX_BYTES : 0u;
  static constexpr uint32_t RING_BUDGET =
      SMEM_LIMIT - 512 - 1024 - EPI_WARPS * EPI_WARP_BYTES - MB_BYTES;
  static constexpr int STAGES =
      RING_BUDGET / STAGE_BYTES > MAX_STAGES ? MAX_STAGES : static_cast<int>(RING_BUDGET / STAGE_BYTES);
  static_assert(STAGES >= 2, "at least two stages in the ring");
  static_assert(STAGES * KSUB <= MAX_STAGES, "one full barrier per stage and K row");
  static constexpr uint32_t SMEM_A = 0;
  static constexpr uint32_t SMEM_B = SMEM_A + STAGES * A_STAGE_BYTES;
  static constexpr uint32_t SMEM_EPI = SMEM_B + STAGES * B_STAGE_BYTES;
  static constexpr uint32_t SMEM_MB = SMEM_EPI + EPI_WARPS * EPI_WARP_BYTES;  // ones, then bias
  static constexpr uint32_t SMEM_BAR = SMEM_MB + MB_BYTES;
  static constexpr uint32_t SMEM_BYTES = SMEM_BAR + 512 + 1024;  // + barriers + 1024-B alignment slack
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
};

// barrier slots (uint64 each) inside the SMEM_BAR area; full barriers BAR_FULL + stage * KSUB +
// (row with per-row barriers, else 0), empty barriers per stage
constexpr int BAR_FULL = 0;
constexpr int BAR_EMPTY = MAX_STAGES;
constexpr int BAR_ACC_FULL = 2 * MAX_STAGES;
constexpr int BAR_ACC_EMPTY = 2 * MAX_STAGES + 2;
constexpr int BAR_MMA_DONE = 2 * MAX_STAGES + 4;
constexpr int BAR_Y = 2 * MAX_STAGES + 5;  // one per epilogue warp and Y block (staged Y)
constexpr int BAR_BIAS_FULL = 2 * MAX_STAGES + 5 + 2 * 16;  // the staged bias row landed (MB)
constexpr int BAR_BIAS_EMPTY = BAR_BIAS_FULL + 1;          // the bias MMA has read it
constexpr uint32_t OFF_TMEM_SLOT = 8 * (BAR_BIAS_EMPTY + 1);
constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 8;
static_assert(OFF_ABORT + 4 <= 512, "barrier area");

// wait sites recorded with a timeout
enum { SITE_PROD_EMPTY = 1, SITE_MMA_ACC_EMPTY, SITE_MMA_FULL, SITE_EPI_ACC_FULL, SITE_DRAIN,
       SITE_EPI_Y };

// Bounded wait that ignores the abort flag: used only to drain copies / MMAs already in flight.
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                           int* err) {
  volatile int never = 0;
  return mbar_wait(bar, parity, &never, timeout_ns, err, SITE_DRAIN);
}

// One unit of work of the persistent loop: a whole 256-column tile, or a piece of a tail tile.
struct Work {
  int tm, tn;   // tile coordinates
  int col0;     // first output column of the piece
  int width;    // columns in the piece (256, 128 or 64)
};
__device__ __forceinline__ Work work_of(const TcParams& p, int item) {
  Work w;
  int tile = item, piece = 0, split = 1;
  if (item >= p.full_tiles) {
    const int j = item - p.full_tiles;
    split = p.tail_split;
    tile = p.full_tiles + j / split;
    piece = j % split;
  }
  if (p.raster_n)  // the same grouped order with the roles of M and N exchanged
    tile_of(tile, p.tiles_n, p.tiles_m, p.group, w.tn, w.tm);
  else
    tile_of(tile, p.tiles_m, p.tiles_n, p.group, w.tm, w.tn);
  w.width = BN / split;
  w.col0 = w.tn * BN + piece * w.width;
  if (w.tn == p.tiles_n - 1) {  // ragged last column of tiles: only as wide as N needs
    const int left = p.last_width - piece * w.width;
    if (left < w.width) w.width = left > 0 ? left : p.gran;
  }
  return w;
}

// Bias of the 128 columns [col, col + 128) that one epilogue warpgroup owns: lane l holds columns
// col + 4l .. col + 4l + 3 as fp32 (zeros past N; N is a multiple of 8 here).  One coalesced load
// per warp and work item, issued before the accumulator wait so that its latency is hidden.
__device__ __forceinline__ void load_bias_quad(const TcParams& p, int col, float (&b)[4]) {
  const int c = col + 4 * static_cast<int>(threadIdx.x & 31);
  b[0] = b[1] = b[2] = b[3] = 0.f;
  if (c >= p.N) return;
  if (p.bias_type == ELEM_F32) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.bias) + c));
    b[0] = f.x; b[1] = f.y; b[2] = f.z; b[3] = f.w;
  } else {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.bias) + c));
    const bool bf = p.bias_type == ELEM_BF16;
    const float2 f0 = unpack2(u.x, bf), f1 = unpack2(u.y, bf);
    b[0] = f0.x; b[1] = f0.y; b[2] = f1.x; b[3] = f1.y;
  }
}

// Bias of the G columns j0 .. j0 + G - 1 (warpgroup-local, j0 a multiple of 4) broadcast to every
// lane from the lanes of load_bias_quad that hold them.  Called by all 32 lanes.
template <int G>
__device__ __forceinline__ void bias_granule(const float (&b)[4], int j0, float (&out)[G]) {
#pragma unroll
  for (int e = 0; e < G; ++e) out[e] = __shfl_sync(0xffffffffu, b[e & 3], (j0 >> 2) + (e >> 2));
}

template <int EPI, int OUT_BYTES, bool PAIR, bool F8 = false, int YB = 1, int KSUB = 1,
          bool MB = false, int EW = 8>
__global__ void __launch_bounds__(threads_for(EW), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmY,
                   const __grid_constant__ CUtensorMap tmBias,
                   const __grid_constant__ CUtensorMap tmB64, const TcParams p) {
  constexpr int CH = 128 / OUT_BYTES;  // output columns per 128-byte staging row
  constexpr int G = 16 / OUT_BYTES;    // columns per 16-byte granule
  constexpr int NG = CH / G;           // granules per chunk (8)
  // the gate's Y and the residual R are staged the same way (16-bit outputs)
  constexpr bool YS = (EPI == EPI_GATE || EPI == EPI_RESID) && (OUT_BYTES == 2);
  using C = Cfg<PAIR, YS, YB, KSUB, MB, EW>;
  constexpr int EPI_WARPS = EW;
  static_assert(EW == 8 || (EW == 16 && !PAIR && YS && YB == 1), "16 epilogue warps: single CTAs with one staged Y block");
  static_assert(!MB || !F8, "the bias MMA is a kind::f16 MMA");
  // Operand element size: one K row of a stage is one 128-byte swizzle row per A row (64 16-bit or
  // 128 fp8 elements); A arrives as KSUB boxes of 128 rows x one K row, B as boxes of (128 bytes
  // of N) x (KSUB K rows); the stage byte counts and the ring are the same for both types.
  constexpr int EB = F8 ? 1 : 2;
  constexpr int KROW = 128 / EB;                          // K elements per K row
  constexpr int KB_ELEMS = KSUB * KROW;                   // K per stage
  constexpr int BOXC = 128 / EB;                          // B box columns
  constexpr uint32_t BBOX = static_cast<uint32_t>(KB_ELEMS * BOXC * EB);  // KSUB x 8 KB / 16 KB
  // With p.row_bars (two K rows per stage) each K row of a stage completes on its own full barrier,
  // so that the MMAs on the first row start while the second is still landing; B's column boxes
  // are then copied one K row at a time (BBOX_ROW bytes each, stacked at the 1024-byte-aligned
  // offsets one two-row box would fill: the same swizzled layout).  Measured on GB300: fp8
  // operands 4096^3 49.3 -> 48.4 us, GLU block K = 4096 120.0 -> 118.4 us; on 16-bit operands
  // without staged Y 4096^3 equal and FFN 8192 x 14336 x 4096 543 -> 548 us, so the host enables
  // it for fp8 operands and staged Y only.
  constexpr uint32_t BBOX_ROW = BBOX / KSUB;
  const bool rowbar = KSUB > 1 && p.row_bars != 0;
  const int nfb = rowbar ? KSUB : 1;  // full barriers per stage
  constexpr int KSTEP = F8 ? 32 : 16;                     // K per MMA instruction
  constexpr int KPR = KROW / KSTEP;                       // MMAs per K row (4)
  constexpr uint32_t B_KADV = static_cast<uint32_t>(KSTEP) * 128u;  // MN-major B bytes per MMA
  constexpr uint32_t A_STAGE_BYTES = C::A_STAGE_BYTES;
  constexpr int STAGES = C::STAGES;
  constexpr int CG = PAIR ? 2 : 1;
  constexpr uint32_t SMEM_A = C::SMEM_A, SMEM_B = C::SMEM_B, SMEM_EPI = C::SMEM_EPI,
                     SMEM_BAR = C::SMEM_BAR;
  constexpr uint32_t SMEM_ONES = C::SMEM_MB, SMEM_BIAS = C::SMEM_MB + ONES_BYTES;
  // the bias-initialised accumulator: set by the extra MMA (MB) or written by the epilogue
  const bool bias_mma = MB && p.bias_init;
  const bool bias_tmem = p.bias_init && !bias_mma;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + SMEM_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SMEM_BAR + OFF_TMEM_SLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SMEM_BAR + OFF_ABORT);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;     // 0 = the MMA-issuing CTA
  const bool leader = rank == 0;
  const int unit = PAIR ? static_cast<int>(blockIdx.x / 2) : static_cast<int>(blockIdx.x);
  const int units = PAIR ? static_cast<int>(gridDim.x / 2) : static_cast<int>(gridDim.x);
  // barriers of the even CTA as seen from anywhere in the cluster
  auto lead_bar = [&](int i) { return PAIR ? map_shared_rank(bar(i), 0) : bar(i); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      for (int r = 0; r < KSUB; ++r) mbar_init(bar(BAR_FULL + s * KSUB + r), 1);
      mbar_init(bar(BAR_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(BAR_ACC_FULL + b), 1);
      mbar_init(bar(BAR_ACC_EMPTY + b), (PAIR ? 2 : 1) * EPI_WARPS);
    }
    mbar_init(bar(BAR_MMA_DONE), 1);
    for (int w = 0; w < (YB == 0 ? 1 : YB) * EPI_WARPS; ++w) mbar_init(bar(BAR_Y + w), 1);
    if (MB) {
      mbar_init(bar(BAR_BIAS_FULL), 1);
      mbar_init(bar(BAR_BIAS_EMPTY), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (F8 && PAIR && p.tail_split > 1) tma_prefetch_desc(&tmB64);
    tma_prefetch_desc(&tmOut);
    if (YS) tma_prefetch_desc(&tmY);
  }
  if (warp == 1) {
    tmem_alloc_cg<CG>(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish_cg<CG>();
  }
  if constexpr (MB) {
    // the ones tile (every 16-bit element 1.0) and the bias tile's zero rows, written once; the
    // bias row of each work item is then copied over the first K row of each box by TMA
    if (warp >= 2) {
      const uint32_t one = p.ab_bf16 ? 0x3F803F80u : 0x3C003C00u;
      uint32_t* w = reinterpret_cast<uint32_t*>(smem + SMEM_ONES);
      for (int i = static_cast<int>(threadIdx.x) - 64; i < static_cast<int>(C::MB_BYTES / 4);
           i += 32 * EPI_WARPS)
        w[i] = i < static_cast<int>(ONES_BYTES / 4) ? one : 0u;
      fence_proxy_async_smem();  // generic-proxy writes, read by the MMA (async proxy)
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // the peer signals the even CTA's barriers: both must be initialised
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_kb = (p.K + KB_ELEMS - 1) / KB_ELEMS;
  // Up to here only this CTA's shared and tensor memory were touched; with programmatic
  // dependent launch that set-up overlaps the previous kernel in the stream, and global memory is
  // read only after it has completed.  Single CTAs prefetch their first work item into L2 before
  // that -- the first ring stages' operands (up to two rings' worth) and the warps' first Y --
  // in the time the previous kernel's last CTAs leave: a prefetch only moves lines into L2, which
  // stays coherent with whatever that kernel still writes.  Measured on one GB300 (graph replay,
  // alternating builds): GLU block M = 1024, N = 21568, K = 256 / 512 (single CTAs) 25.6 -> 25.1,
  // 35.0 -> 34.1 us; on CTA pairs it measured slower (K = 1024 42.4 -> 43.6 us, 4096^3 80.9 ->
  // 81.5 us), so pairs do not prefetch.
  if (!PAIR && p.pdl && unit < p.num_items) {
    const Work w0 = work_of(p, unit);
    if (warp == 0 && lane == 0) {
      const int m0 = w0.tm * C::TILE_M + static_cast<int>(rank) * BM;
      const int cols = PAIR ? w0.width / 2 : w0.width;
      const int nb0 = w0.col0 + static_cast<int>(rank) * cols;
      const int boxes = (cols + BOXC - 1) / BOXC;
      const int nkb = num_kb < 2 * STAGES ? num_kb : 2 * STAGES;
      for (int kb = 0; kb < nkb; ++kb)
        for (int r = 0; r < KSUB; ++r) {
          const int kx = kb * KB_ELEMS + r * KROW;
          tma_prefetch_2d(&tmA, kx, m0);
          if (rowbar || r == 0)
            for (int c = 0; c < boxes; ++c) tma_prefetch_2d(&tmB, nb0 + BOXC * c, kx);
        }
    }
    if (YS && warp >= 2 && warp < 2 + EPI_WARPS && lane == 0) {
      const int cb = ((warp - 2) >> 2) * C::COLS_W;
      const int r0 = w0.tm * C::TILE_M + static_cast<int>(rank) * BM + 32 * (warp & 3);
      if (r0 < p.M)
        for (int c = cb; c < cb + C::COLS_W && c < w0.width; c += 64)
          if (w0.col0 + c < p.N) tma_prefetch_2d(&tmY, w0.col0 + c, r0);
    }
  }
  grid_dependency_wait();

  const uint64_t tmo = p.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // L2 hints: A (a few MB, read by every column of tiles) is kept; B's boxes are read by the
      // M-tiles of one band in quick succession and then not again, so they go first (measured:
      // 4096^3 83.7 -> 82.4 us, GLU block K = 4096 120.1 -> 118.7 us).
      const uint64_t pol_a = policy_evict_last();
      const uint64_t pol_b = policy_evict_first();
      uint32_t stage = 0, phase = 0;
      uint32_t issued = 0, issued_parity = 0;
      uint32_t bias_items = 0;  // bias rows copied (bias MMA)
      bool ok = true;
      for (int t = unit; ok && t < p.num_items; t += units) {
        // This CTA's last work item: the next kernel in the stream may launch (its CTAs become
        // resident as this kernel's CTAs exit and prefetch their first data while the others
        // finish; it reads global memory only after this kernel has completed).
        if (t + units >= p.num_items) grid_dependents_launch();
        const Work wk = work_of(p, t);
        const int m0 = wk.tm * C::TILE_M + static_cast<int>(rank) * BM;
        // each CTA of a pair stages half of the piece's columns
        const int cols = PAIR ? wk.width / 2 : wk.width;
        const int nb0 = wk.col0 + static_cast<int>(rank) * cols;
        const int boxes = (cols + BOXC - 1) / BOXC;
        // This work item's bias row (bias MMA), once the previous item's bias MMA has read the
        // tile: one 128-byte row per 64-column box, zero-filled past N (the bias mask).  Copied
        // after the item's first stage: by then the MMA warp has begun the previous item (its
        // stages are being consumed), so its bias MMA has been issued and the wait is short,
        // while the producer itself never waits here ahead of the ring.
        auto load_bias = [&]() -> bool {
          if (!mbar_wait(bar(BAR_BIAS_EMPTY), (bias_items & 1u) ^ 1u, abort_flag, tmo, p.err,
                         SITE_PROD_EMPTY))
            return false;
          const uint32_t bfull = lead_bar(BAR_BIAS_FULL);
          if (leader)
            mbar_arrive_expect_tx(bar(BAR_BIAS_FULL),
                                  (PAIR ? 2u : 1u) * static_cast<uint32_t>(boxes) * 128u);
          for (int c = 0; c < boxes; ++c) {
            const uint32_t dst = sbase + SMEM_BIAS + static_cast<uint32_t>(c) * BIAS_BOX_BYTES;
            if constexpr (PAIR)
              tma_load_2d_pair(dst, &tmBias, bfull, nb0 + BOXC * c, 0, pol_a);
            else
              tma_load_2d(dst, &tmBias, bfull, nb0 + BOXC * c, 0, pol_a);
          }
          ++bias_items;
          return true;
        };
        // fp8 operands on pairs, a column piece (64 columns per CTA): B as one 64-byte-wide box
        // per K row set with 64-byte swizzle (tmB64), half a 128-byte box's bytes
        const bool b64 = F8 && PAIR && cols == 64;
        const uint32_t b_bytes = b64 ? BBOX_ROW / 2 : static_cast<uint32_t>(boxes) * BBOX_ROW;
        // bytes per full barrier: one K row, or the whole stage (both CTAs of a pair)
        const uint32_t tx = (PAIR ? 2u : 1u) * (A_ROW_BYTES + b_bytes) * static_cast<uint32_t>(KSUB / nfb);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(bar(BAR_EMPTY + stage), phase ^ 1u, abort_flag, tmo, p.err,
                         SITE_PROD_EMPTY)) {
            ok = false;
            break;
          }
          const uint32_t a_dst = sbase + SMEM_A + stage * A_STAGE_BYTES;
          const uint32_t b_dst = sbase + SMEM_B + stage * C::B_STAGE_BYTES;
          // diagnostic stall: announce the stage's bytes but never load them
          const bool stall = p.inject_stall && blockIdx.x == 0 && t == unit && kb == 0;
          // the even CTA's full barriers count both CTAs' bytes
          if (leader)
            for (int f = 0; f < nfb; ++f) mbar_arrive_expect_tx(bar(BAR_FULL + stage * KSUB + f), tx);
#pragma unroll
          for (int r = 0; r < KSUB; ++r) {
            const int fi = BAR_FULL + static_cast<int>(stage) * KSUB + (rowbar ? r : 0);
            const int kx = kb * KB_ELEMS + r * KROW;
            // B: per K row with row barriers, else the whole stage's rows with the first A row
            const bool b_now = rowbar || r == 0;
            const uint32_t b_off = rowbar ? r * BBOX_ROW : 0u;
            if (stall) {
            } else if constexpr (PAIR) {
              const uint32_t lfb = lead_bar(fi);
              tma_load_2d_pair(a_dst + r * A_ROW_BYTES, &tmA, lfb, kx, m0, pol_a);
              if (b_now) {
                if (b64)  // K rows of 64 bytes: a K row set of the stage every BBOX_ROW / 2
                  tma_load_2d_pair(b_dst + b_off / 2, &tmB64, lfb, nb0, kx, pol_b);
                else
                  for (int c = 0; c < boxes; ++c)
                    tma_load_2d_pair(b_dst + c * BBOX + b_off, &tmB, lfb, nb0 + BOXC * c, kx, pol_b);
              }
            } else {
              tma_load_2d(a_dst + r * A_ROW_BYTES, &tmA, bar(fi), kx, m0, pol_a);
              if (b_now)
                for (int c = 0; c < boxes; ++c)
                  tma_load_2d(b_dst + c * BBOX + b_off, &tmB, bar(fi), nb0 + BOXC * c, kx, pol_b);
            }
          }
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if (MB && bias_mma && kb == 0 && !load_bias()) {
            ok = false;
            break;
          }
        }
        if (MB && bias_mma && num_kb == 0 && ok && !load_bias()) ok = false;
      }
      // Every load issued must land before the CTA may exit (also after an abort).  In a pair the
      // even CTA's full barriers count the peer's bytes too; the closing cluster barrier keeps the
      // peer resident until then.
      if (leader) {
        for (int s = 0; s < STAGES; ++s)
          if ((issued >> s) & 1u)
            for (int f = 0; f < nfb; ++f)
              drain_wait(bar(BAR_FULL + s * KSUB + f), (issued_parity >> s) & 1u, tmo, p.err);
        if (MB && bias_items > 0) drain_wait(bar(BAR_BIAS_FULL), (bias_items - 1u) & 1u, tmo, p.err);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      constexpr uint16_t kPair = 0x3;
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = unit; ok && t < p.num_items; t += units, ++it) {
        // MMA N = the piece's width (all tiles but the tail pieces: 256)
        const int width = work_of(p, t).width;
        // fp8 pairs' column pieces: B in 64-byte-swizzled K rows (8 rows x 64 bytes per atom)
        const bool b64 = F8 && PAIR && width == 128;
        const uint32_t idesc = (p.idesc & ~(0x3Fu << 17)) | (static_cast<uint32_t>(width >> 3) << 17);
        const int b = it & 1;
        const uint32_t acc_phase = (static_cast<uint32_t>(it) >> 1) & 1u;
        // Buffer b is free once the epilogue has read its previous tile; with the bias written by
        // the epilogue, the epilogue has also written this tile's bias row into it (one more phase).
        const uint32_t want = bias_tmem ? acc_phase : (acc_phase ^ 1u);
        if (!mbar_wait(bar(BAR_ACC_EMPTY + b), want, abort_flag, tmo, p.err, SITE_MMA_ACC_EMPTY))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
        if (MB && bias_mma) {
          // D = ones (128 x 16) x [bias row; 15 zero rows]: every row of the accumulator starts at
          // the bias of its column; the K loop then accumulates onto it
          if (!mbar_wait(bar(BAR_BIAS_FULL), static_cast<uint32_t>(it) & 1u, abort_flag, tmo, p.err,
                         SITE_MMA_FULL))
            break;
          tc_fence_after();
          // ones: K-major without swizzle, 8-row x 16-byte core matrices, 128 B apart along K and
          // 256 B apart along M (the whole 4 KB tile is ones, so only the extent matters)
          const uint64_t ad = sdesc_none(sbase + SMEM_ONES, 128u, 256u);
          const uint64_t bd = sdesc_sw128(sbase + SMEM_BIAS, BIAS_BOX_BYTES, 1024u);
          umma_f16_cg<CG>(d_tmem, ad, bd, idesc, 0u);
          umma_commit_cg<CG>(bar(BAR_BIAS_EMPTY), kPair);  // bias tile free (both CTAs) once read
        }
        for (int kb = 0; kb < num_kb; ++kb) {
          const uint32_t a_addr = sbase + SMEM_A + stage * A_STAGE_BYTES;
          const uint32_t b_addr = sbase + SMEM_B + stage * C::B_STAGE_BYTES;
#pragma unroll
          for (int r = 0; r < KSUB; ++r) {  // with row barriers each K row as soon as it has landed
            if (r == 0 || rowbar) {
              if (!mbar_wait(bar(BAR_FULL + static_cast<int>(stage) * KSUB + (rowbar ? r : 0)), phase,
                             abort_flag, tmo, p.err, SITE_MMA_FULL)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
#pragma unroll
            for (int k = r * KPR; k < (r + 1) * KPR; ++k) {  // 32 bytes of K per MMA
              const uint64_t ad =
                  sdesc_sw128(a_addr + (k / KPR) * A_ROW_BYTES + 32u * (k % KPR), 16u, 1024u);
              // MN-major B: one column box (BBOX bytes) apart along N, 1 KB per 8 K rows (or, for
              // the 64-byte-wide boxes, one atom along N and 512 bytes per 8 K rows)
              const uint64_t bd = b64 ? sdesc_sw64(b_addr + (B_KADV / 2) * k, BBOX, 512u)
                                      : sdesc_sw128(b_addr + B_KADV * k, BBOX, 1024u);
              const uint32_t acc = (p.bias_init | kb | k) != 0 ? 1u : 0u;  // bias: already in D
              if constexpr (F8)
                umma_f8_cg<CG>(d_tmem, ad, bd, idesc, acc);
              else
                umma_f16_cg<CG>(d_tmem, ad, bd, idesc, acc);
            }
          }
          if (!ok) break;
          umma_commit_cg<CG>(bar(BAR_EMPTY + stage), kPair);  // stage free (both CTAs) once read
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_cg<CG>(bar(BAR_ACC_FULL + b), kPair);  // accumulator complete (both CTAs)
      }
      // All MMAs issued by this thread must finish before TMEM is released.
      umma_commit_cg<CG>(bar(BAR_MMA_DONE), 0x1);
      drain_wait(bar(BAR_MMA_DONE), 0, tmo, p.err);
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int ew = warp - 2;
    const int cbeg = (ew >> 2) * C::COLS_W;  // first column (within the tile) of this warpgroup
    const uint32_t ebuf = sbase + SMEM_EPI + static_cast<uint32_t>(ew) * C::EPI_WARP_BYTES;
    const bool out_bf = p.out_type == ELEM_BF16;
    const bool y_bf = p.y_bf16 != 0;  // the gate's Y / the residual's R
    const uint64_t pol_out = policy_evict_first();
    const bool add_bias = !p.bias_init;  // else the accumulator already holds the bias
    // Bias-initialised accumulator ("Optimizing GEMM + Activation on CDNA4 with TLX", V4: the
    // accumulator starts at the bias instead of zero): this warp writes bias[col] into every lane
    // (row) of its quarter and every column it owns of buffer bb for work item t, then hands
    // the buffer to the MMA warp, whose first MMA of the tile accumulates onto it.
    auto release_acc = [&](int t, int bb) {
      if (bias_tmem && t < p.num_items) {
        const Work w = work_of(p, t);
        const uint32_t ta =
            tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(bb * BN);
        float bq[4];
        load_bias_quad(p, w.col0 + cbeg, bq);
#pragma unroll 1
        for (int c = cbeg; c < cbeg + C::COLS_W && c < w.width; c += 16) {
          float b16[16];
          bias_granule<16>(bq, c - cbeg, b16);
          uint32_t r[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(b16[e]);
          __syncwarp();  // tcgen05.st is warp-collective
          tmem_st16(ta + static_cast<uint32_t>(c), r);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR)
          mbar_arrive_cluster(lead_bar(BAR_ACC_EMPTY + bb));  // the even CTA's MMA waits on it
        else
          mbar_arrive(bar(BAR_ACC_EMPTY + bb));
      }
    };
    if (bias_tmem) {  // first use of both buffers
      release_acc(unit, 0);
      release_acc(unit + units, 1);
    }
    int it = 0;
    if constexpr (YS) {
      // Gate with Y staged by TMA: the warp's 32 x 128 block of Y lands in one of its NYB 8 KB
      // blocks (two 128-byte-swizzled 32 x 64 chunks) while earlier tiles are still computed; the
      // epilogue reads y from there, writes the result over it, and stores each chunk with one TMA
      // store.  Work item number `it` of this CTA uses block it % NYB.
      // YB = 0 (long K loops): one 4 KB chunk buffer per warp; the tile's first chunk of Y is
      // prefetched a work item ahead, the second is loaded once the first chunk's store has read
      // the buffer (the epilogue has the whole next main loop to do it), which leaves the ring
      // room for three two-row stages.
      constexpr bool YHALF = YB == 0;
      constexpr int NYB = YHALF ? 1 : YB;  // prefetched Y blocks per warp
      auto ybar = [&](int yb) { return bar(BAR_Y + yb * EPI_WARPS + ew); };
      uint32_t y_par = 0, y_issued = 0;  // bit yb: parity to wait for / a load is in flight
      auto issue_y = [&](int t, int yb) -> bool {  // warp-uniform result
        const Work w = work_of(p, t);
        const int r0 = w.tm * C::TILE_M + static_cast<int>(rank) * BM + 32 * q;
        if (r0 >= p.M) return false;
        int nchunks = 0;
        for (int c = cbeg; c < cbeg + C::COLS_W && c < w.width; c += CH)
          if (w.col0 + c < p.N) ++nchunks;
        if (nchunks == 0) return false;
        if (YHALF) nchunks = 1;
        if (lane == 0) {
          bulk_wait_read<0>();  // the stores that last read this region are done with it
          const uint32_t yblk = ebuf + static_cast<uint32_t>(yb) * C::Y_BLOCK_BYTES;
          mbar_arrive_expect_tx(ybar(yb), static_cast<uint32_t>(nchunks) * EPI_BUF_BYTES);
          for (int j = 0; j < nchunks; ++j)
            tma_load_2d(yblk + j * EPI_BUF_BYTES, &tmY, ybar(yb), w.col0 + cbeg + j * CH, r0, pol_out);
        }
        return true;
      };
      for (int j = 0; j < NYB; ++j)
        if (unit + j * units < p.num_items && issue_y(unit + j * units, j)) y_issued |= 1u << j;
      for (int t = unit; t < p.num_items; t += units, ++it) {
        const Work wk = work_of(p, t);
        const int m0 = wk.tm * C::TILE_M + static_cast<int>(rank) * BM, n0 = wk.col0;
        const int nch = wk.width / CH;
        const int b = it & 1;
        const uint32_t acc_phase = (static_cast<uint32_t>(it) >> 1) & 1u;
        const int row0 = m0 + 32 * q;
        const bool rows_live = row0 < p.M;  // warp-uniform
        float bq[4];
        if (add_bias) load_bias_quad(p, n0 + cbeg, bq);

        if (!mbar_wait_sleepy(bar(BAR_ACC_FULL + b), acc_phase, abort_flag, tmo, p.err, SITE_EPI_ACC_FULL))
          break;
        tc_fence_after();
        const int yb = NYB == 1 ? 0 : (it & 1);
        if ((y_issued >> yb) & 1u) {
          if (!mbar_wait(ybar(yb), (y_par >> yb) & 1u, abort_flag, tmo, p.err, SITE_EPI_Y)) break;
          y_par ^= 1u << yb;
          y_issued &= ~(1u << yb);
        }
        const uint32_t taddr =
            tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(b * BN);
        bool aborted = false;
#pragma unroll 1
        for (int c = cbeg / CH; c < nch && c < (cbeg + C::COLS_W) / CH; ++c) {
          const int col0 = n0 + c * CH;
          if (!rows_live || col0 >= p.N) break;  // warp-uniform; columns only grow with c
          if constexpr (YHALF) {
            if (c != cbeg / CH) {  // later chunks: Y into the buffer the last store has read
              if (lane == 0) {
                bulk_wait_read<0>();
                mbar_arrive_expect_tx(ybar(0), EPI_BUF_BYTES);
                tma_load_2d(ebuf, &tmY, ybar(0), col0, row0, pol_out);
              }
              y_issued |= 1u;
              if (!mbar_wait(ybar(0), y_par & 1u, abort_flag, tmo, p.err, SITE_EPI_Y)) {
                aborted = true;
                break;
              }
              y_par ^= 1u;
              y_issued &= ~1u;
            }
          }
          uint32_t acc[CH];
          __syncwarp();  // tcgen05.ld is warp-collective
          {
            uint32_t(&a0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&acc[0]);
            uint32_t(&a1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&acc[32]);
            tmem_ld32(taddr, a0, c * CH);
            tmem_ld32(taddr, a1, c * CH + 32);
            tmem_ld_wait();
          }
          const uint32_t sb = YHALF ? ebuf
                                    : ebuf + static_cast<uint32_t>(yb) * C::Y_BLOCK_BYTES +
                                          static_cast<uint32_t>(c - cbeg / CH) * EPI_BUF_BYTES;
          // Y and out share the 16-bit operand type here: the chunk is compiled for fp16 and for
          // bf16 and one of the two is taken (a warp-uniform branch), so that no conversion
          // carries a run-time type test.
          auto chunk = [&](auto bf_tag) {
          constexpr bool BF = decltype(bf_tag)::value;
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            // 128-byte swizzle: granule g of row `lane` sits at slot g ^ (lane & 7)
            const uint32_t addr = sb + static_cast<uint32_t>(lane) * 128u +
                                  (static_cast<uint32_t>(g ^ (lane & 7)) << 4);
            uint32_t y[4];
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(y[0]), "=r"(y[1]), "=r"(y[2]), "=r"(y[3])
                         : "r"(addr)
                         : "memory");
            float bv[G];
            if (add_bias) {
              bias_granule<G>(bq, c * CH + g * G - cbeg, bv);
            } else {
#pragma unroll
              for (int e = 0; e < G; ++e) bv[e] = 0.f;
            }
            uint32_t packed[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 y2 = unpack2(y[e], BF);
              float x0 = __uint_as_float(acc[g * G + 2 * e]) + bv[2 * e];  // bias once
              float x1 = __uint_as_float(acc[g * G + 2 * e + 1]) + bv[2 * e + 1];
              if constexpr (EPI == EPI_GATE) {
                x0 = fmaf(x0, y2.x, x0);  // X + X * Y
                x1 = fmaf(x1, y2.y, x1);
              } else {                    // residual before the activation
                x0 = fmaxf(x0 + y2.x, 0.0f);
                x1 = fmaxf(x1 + y2.y, 0.0f);
              }
              packed[e] = pack2(x0, x1, BF);
            }
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(packed[0]),
                         "r"(packed[1]), "r"(packed[2]), "r"(packed[3])
                         : "memory");
          }
          };
          if (y_bf)
            chunk(std::true_type{});
          else
            chunk(std::false_type{});
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmOut, sb, col0, row0, pol_out);
            if (YHALF) bulk_commit();  // the next chunk's Y load waits for this store's read
          }
        }
        if (aborted) break;
        if (lane == 0) bulk_commit();
        // This warp has finished reading accumulator b: release it to the MMA warp.
        release_acc(t + 2 * units, b);
        // Prefetch into this block the Y of the work item NYB items ahead (main loops run
        // meanwhile).
        if (t + NYB * units < p.num_items && issue_y(t + NYB * units, yb)) y_issued |= 1u << yb;
      }
      // After an abort a prefetched Y block may still be landing: wait for it (bounded).
      for (int j = 0; j < NYB; ++j)
        if ((y_issued >> j) & 1u) drain_wait(ybar(j), (y_par >> j) & 1u, tmo, p.err);
    } else {
    for (int t = unit; t < p.num_items; t += units, ++it) {
      const Work wk = work_of(p, t);
      const int m0 = wk.tm * C::TILE_M + static_cast<int>(rank) * BM, n0 = wk.col0;
      const int nch = wk.width / CH;
      const int b = it & 1;
      const uint32_t acc_phase = (static_cast<uint32_t>(it) >> 1) & 1u;
      const int row0 = m0 + 32 * q;
      const int row = row0 + lane;
      const bool rows_live = row0 < p.M;  // warp-uniform
      const bool use_bias = EPI != EPI_NONE && add_bias;
      float bq[4];
      if (use_bias) load_bias_quad(p, n0 + cbeg, bq);

      if (!mbar_wait_sleepy(bar(BAR_ACC_FULL + b), acc_phase, abort_flag, tmo, p.err, SITE_EPI_ACC_FULL))
        break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(b * BN);

#pragma unroll 1
      for (int c = cbeg / CH; c < nch && c < (cbeg + C::COLS_W) / CH; ++c) {
        const int col0 = n0 + c * CH;
        if (!rows_live || col0 >= p.N) break;  // warp-uniform; columns only grow with c

        if constexpr (OUT_BYTES == 1) {
          // fp8 output: one 128-byte staging row holds 128 columns; work on them 64 at a time.
          const uint32_t sb = ebuf;
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            uint32_t acc[64];
            __syncwarp();  // tcgen05.ld is warp-collective
            {
              uint32_t(&a0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&acc[0]);
              uint32_t(&a1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&acc[32]);
              tmem_ld32(taddr, a0, c * CH + 64 * h);
              tmem_ld32(taddr, a1, c * CH + 64 * h + 32);
              tmem_ld_wait();
            }
#pragma unroll
            for (int gi = 0; gi < 4; ++gi) {
              const int g = 4 * h + gi;  // 16-column granule within the 128-column row
              float bv[16];
              if (add_bias) {
                bias_granule<16>(bq, c * CH + g * 16 - cbeg, bv);
              } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) bv[e] = 0.f;
              }
              uint32_t packed[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float x[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const int j = 16 * gi + 4 * e + k;
                  float v = fmaxf(__uint_as_float(acc[j]) + bv[4 * e + k], 0.0f);  // bias, ReLU
                  v = fminf(fmaxf(v * p.out_scale, -448.0f), 448.0f);              // scale, clamp
                  x[k] = v;
                }
                packed[e] = pack2_e4m3(x[0], x[1]) | (pack2_e4m3(x[2], x[3]) << 16);
              }
              const uint32_t dst = sb + static_cast<uint32_t>(lane) * 128u +
                                   (static_cast<uint32_t>(g ^ (lane & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(packed[0]),
                           "r"(packed[1]), "r"(packed[2]), "r"(packed[3])
                           : "memory");
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmOut, sb, col0, row0, pol_out);
            bulk_commit();
          }
          continue;
        } else {
        // Gate: this thread's row of Y for the chunk, loaded before the TMEM read.
        constexpr bool HAS_Y = EPI == EPI_GATE || EPI == EPI_RESID;
        uint4 yv[HAS_Y ? NG * G / 8 : 1];
        if constexpr (HAS_Y) {
          const uint16_t* yrow = static_cast<const uint16_t*>(p.Y) + static_cast<int64_t>(row) * p.N;
#pragma unroll
          for (int v = 0; v < NG * G / 8; ++v) {
            const int col = col0 + 8 * v;
            if (row < p.M && col < p.N)
              yv[v] = __ldcs(reinterpret_cast<const uint4*>(yrow + col));
            else
              yv[v] = make_uint4(0, 0, 0, 0);
          }
        }

        uint32_t acc[CH];
        __syncwarp();  // tcgen05.ld is warp-collective
        {
          uint32_t(&a0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&acc[0]);
          tmem_ld32(taddr, a0, c * CH);
          if constexpr (CH == 64) {
            uint32_t(&a1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&acc[32]);
            tmem_ld32(taddr, a1, c * CH + 32);
          }
          tmem_ld_wait();
        }

        // Staging buffer: wait until the store that last read it has finished reading.
        const uint32_t sb = ebuf;
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();

        // compiled for both 16-bit types (of out, or of Y with fp32 outputs); a warp-uniform
        // branch picks one, so that no conversion carries a run-time type test
        auto chunk = [&](auto bf_tag) {
        constexpr bool BF = decltype(bf_tag)::value;
        (void)BF;  // unused when neither out nor Y is 16-bit
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          float bv[G];
          if (use_bias) bias_granule<G>(bq, c * CH + g * G - cbeg, bv);
          float v[G];
#pragma unroll
          for (int e = 0; e < G; ++e) {
            v[e] = __uint_as_float(acc[g * G + e]);
            if (use_bias) v[e] += bv[e];  // bias once, after the full sum
          }
          if constexpr (EPI == EPI_RELU) {
#pragma unroll
            for (int e = 0; e < G; ++e) v[e] = fmaxf(v[e], 0.0f);  // branchless clamp
          }
          if constexpr (HAS_Y) {
            // 16-bit Y (or R): granule g covers columns g*G .. g*G+G-1 of the chunk
#pragma unroll
            for (int e = 0; e < G; e += 2) {
              const int idx = g * G + e;  // column within the chunk
              const uint4 u = yv[idx / 8];
              const uint32_t w = (idx % 8 < 2) ? u.x : (idx % 8 < 4) ? u.y : (idx % 8 < 6) ? u.z : u.w;
              const float2 y2 = unpack2(w, BF);
              if constexpr (EPI == EPI_GATE) {
                v[e] = fmaf(v[e], y2.x, v[e]);          // X + X * Y
                v[e + 1] = fmaf(v[e + 1], y2.y, v[e + 1]);
              } else {                                  // residual before the activation
                v[e] = fmaxf(v[e] + y2.x, 0.0f);
                v[e + 1] = fmaxf(v[e + 1] + y2.y, 0.0f);
              }
            }
          }
          uint4 packed;
          if constexpr (OUT_BYTES == 2) {
            packed.x = pack2(v[0], v[1], BF);
            packed.y = pack2(v[2], v[3], BF);
            packed.z = pack2(v[4 % G], v[5 % G], BF);
            packed.w = pack2(v[6 % G], v[7 % G], BF);
          } else {
            packed.x = __float_as_uint(v[0]);
            packed.y = __float_as_uint(v[1]);
            packed.z = __float_as_uint(v[2 % G]);
            packed.w = __float_as_uint(v[3 % G]);
          }
          // 128-byte swizzle: granule g of row `lane` sits at slot g ^ (lane & 7)
          const uint32_t dst = sb + static_cast<uint32_t>(lane) * 128u +
                               (static_cast<uint32_t>(g ^ (lane & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(packed.x),
                       "r"(packed.y), "r"(packed.z), "r"(packed.w)
                       : "memory");
        }
        };
        if ((OUT_BYTES == 2) ? out_bf : y_bf)
          chunk(std::true_type{});
        else
          chunk(std::false_type{});
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmOut, sb, col0, row0, pol_out);
          bulk_commit();
        }
        }  // OUT_BYTES != 1
      }
      // This warp has finished reading accumulator b: release it to the MMA warp.
      release_acc(t + 2 * units, b);
    }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  // ------------------------------------------------------------ teardown
  // The next kernel may launch: the producer allowed it when this CTA began its last work item;
  // a CTA without work items allows it here.
  grid_dependents_launch();
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // the even CTA's MMAs and both epilogues are done with TMEM
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_cg<CG>(tmem_base, TMEM_COLS);
  }
}

template <int EPI, int OUT_BYTES, bool PAIR, bool F8 = false, int YB = 1, int KSUB = 1,
          bool MB = false, int EW = 8>
cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                       const CUtensorMap& y, const CUtensorMap& bm, const CUtensorMap& b64,
                       const TcParams& p, int grid, cudaStream_t s) {
  auto k = tc_gemm_kernel<EPI, OUT_BYTES, PAIR, F8, YB, KSUB, MB, EW>;
  constexpr uint32_t smem =
      Cfg<PAIR, (EPI == EPI_GATE || EPI == EPI_RESID) && OUT_BYTES == 2, YB, KSUB, MB, EW>::SMEM_BYTES;
  // Per device: the shared-memory opt-in is set once.  Host threads may race on a first call;
  // setting the attribute twice is harmless, and the flag is atomic.
  static std::atomic<bool> opted_in[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!opted_in[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    opted_in[dev].store(true, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(threads_for(EW)));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k, a, b, o, y, bm, b64, p);
}

// A persistent grid must be co-resident: clusters of two need two free SMs in one GPC, so the
// number of pairs that fit at once can be below SMs / 2.
template <int EPI, int OUT_BYTES>
int max_pairs() {
  // Per device (0 = not yet known).  Host threads may race on a first call: each computes the
  // same count, and the slot is atomic.
  static std::atomic<int> cached_dev[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::atomic<int>& slot = cached_dev[dev];
  int cached = slot.load(std::memory_order_acquire);
  if (cached == 0) {
    auto k = tc_gemm_kernel<EPI, OUT_BYTES, true>;
    constexpr uint32_t smem =
        Cfg<true, (EPI == EPI_GATE || EPI == EPI_RESID) && OUT_BYTES == 2>::SMEM_BYTES;
    int n = 0;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(2);
      cfg.blockDim = dim3(THREADS);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    cached = n > 0 ? n : -1;
    slot.store(cached, std::memory_order_release);
  }
  return cached;
}

template <int EPI, int OUT_BYTES, bool F8 = false>
cudaError_t launch_pair_or_not(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                               const CUtensorMap& y, const CUtensorMap& bm, const CUtensorMap& b64,
                               const TcParams& p, int grid, bool pair, cudaStream_t s) {
  if constexpr ((EPI == EPI_GATE || EPI == EPI_RESID) && OUT_BYTES == 2) {
    if (p.y_blocks == 2)
      return pair ? launch_one<EPI, OUT_BYTES, true, F8, 2>(a, b, o, y, bm, b64, p, grid, s)
                  : launch_one<EPI, OUT_BYTES, false, F8, 2>(a, b, o, y, bm, b64, p, grid, s);
    if (pair && p.y_blocks == 0)  // one 4 KB chunk of Y per warp
      return p.k_rows == 2 ? launch_one<EPI, OUT_BYTES, true, F8, 0, 2>(a, b, o, y, bm, b64, p, grid, s)
                           : launch_one<EPI, OUT_BYTES, true, F8, 0, 1>(a, b, o, y, bm, b64, p, grid, s);
    // sixteen epilogue warps on single CTAs (one staged Y block each, 64 columns)
    if (!pair && p.epi_warps == 16) {
      if constexpr (!F8)
        if (p.bias_init && p.bias_mma)
          return launch_one<EPI, OUT_BYTES, false, false, 1, 1, true, 16>(a, b, o, y, bm, b64, p, grid, s);
      return launch_one<EPI, OUT_BYTES, false, F8, 1, 1, false, 16>(a, b, o, y, bm, b64, p, grid, s);
    }
    // the bias-initialised accumulator set by an extra MMA (room for its tiles in shared memory)
    if constexpr (!F8)
      if (p.bias_init && p.bias_mma && p.k_rows != 2)
        return pair ? launch_one<EPI, OUT_BYTES, true, false, 1, 1, true>(a, b, o, y, bm, b64, p, grid, s)
                    : launch_one<EPI, OUT_BYTES, false, false, 1, 1, true>(a, b, o, y, bm, b64, p, grid, s);
  }
  if (pair && p.k_rows == 2) return launch_one<EPI, OUT_BYTES, true, F8, 1, 2>(a, b, o, y, bm, b64, p, grid, s);
  return pair ? launch_one<EPI, OUT_BYTES, true, F8>(a, b, o, y, bm, b64, p, grid, s)
              : launch_one<EPI, OUT_BYTES, false, F8>(a, b, o, y, bm, b64, p, grid, s);
}

}  // namespace tc

int tc_max_active_pairs(int epi, int out_type) {
  const bool f32 = out_type == ELEM_F32;
  if (epi == EPI_QUANT) return tc::max_pairs<EPI_QUANT, 1>();
  switch (epi) {
    case EPI_RELU: return f32 ? tc::max_pairs<EPI_RELU, 4>() : tc::max_pairs<EPI_RELU, 2>();
    case EPI_GATE: return f32 ? tc::max_pairs<EPI_GATE, 4>() : tc::max_pairs<EPI_GATE, 2>();
    case EPI_RESID: return f32 ? tc::max_pairs<EPI_RESID, 4>() : tc::max_pairs<EPI_RESID, 2>();
    default: return f32 ? tc::max_pairs<EPI_NONE, 4>() : tc::max_pairs<EPI_NONE, 2>();
  }
}

int tc_block_m() { return tc::BM; }
int tc_block_n() { return tc::BN; }

cudaError_t launch_tc(int epi, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                      const CUtensorMap& y, const CUtensorMap& bm, const CUtensorMap& b64,
                      const TcParams& p, int grid, bool pair, cudaStream_t s) {
  const bool f32 = p.out_type == ELEM_F32;
  if (p.ab_f8) {  // fp8 operands: bias + ReLU, the gate and the residual (16-bit / fp32 out),
                  // and the quantized epilogue
    if (epi == EPI_QUANT) return tc::launch_pair_or_not<EPI_QUANT, 1, true>(a, b, o, y, bm, b64, p, grid, pair, s);
    switch (epi) {
      case EPI_RELU: return f32 ? tc::launch_pair_or_not<EPI_RELU, 4, true>(a, b, o, y, bm, b64, p, grid, pair, s)
                                : tc::launch_pair_or_not<EPI_RELU, 2, true>(a, b, o, y, bm, b64, p, grid, pair, s);
      case EPI_GATE: return f32 ? tc::launch_pair_or_not<EPI_GATE, 4, true>(a, b, o, y, bm, b64, p, grid, pair, s)
                                : tc::launch_pair_or_not<EPI_GATE, 2, true>(a, b, o, y, bm, b64, p, grid, pair, s);
      case EPI_RESID: return f32 ? tc::launch_pair_or_not<EPI_RESID, 4, true>(a, b, o, y, bm, b64, p, grid, pair, s)
                                 : tc::launch_pair_or_not<EPI_RESID, 2, true>(a, b, o, y, bm, b64, p, grid, pair, s);
      default: return cudaErrorNotSupported;
    }
  }
  if (epi == EPI_QUANT) return tc::launch_pair_or_not<EPI_QUANT, 1>(a, b, o, y, bm, b64, p, grid, pair, s);
  switch (epi) {
    case EPI_RELU: return f32 ? tc::launch_pair_or_not<EPI_RELU, 4>(a, b, o, y, bm, b64, p, grid, pair, s)
                              : tc::launch_pair_or_not<EPI_RELU, 2>(a, b, o, y, bm, b64, p, grid, pair, s);
    case EPI_GATE: return f32 ? tc::launch_pair_or_not<EPI_GATE, 4>(a, b, o, y, bm, b64, p, grid, pair, s)
                              : tc::launch_pair_or_not<EPI_GATE, 2>(a, b, o, y, bm, b64, p, grid, pair, s);
    case EPI_RESID: return f32 ? tc::launch_pair_or_not<EPI_RESID, 4>(a, b, o, y, bm, b64, p, grid, pair, s)
                               : tc::launch_pair_or_not<EPI_RESID, 2>(a, b, o, y, bm, b64, p, grid, pair, s);
    default: return f32 ? tc::launch_pair_or_not<EPI_NONE, 4>(a, b, o, y, bm, b64, p, grid, pair, s)
                        : tc::launch_pair_or_not<EPI_NONE, 2>(a, b, o, y, bm, b64, p, grid, pair, s);
  }
}

}  // namespace fgemm
