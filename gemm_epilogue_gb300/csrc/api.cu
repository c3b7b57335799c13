// api.cu -- the C ABI (include/fgemm.h): argument validation, path choice, TMA descriptor
// encoding and launches on the caller's stream.  Host code only, apart from the error word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "fgemm.h"
#include "kernels.h"
#include "ptx.cuh"
#include "tile_order.h"

namespace fgemm {

// The device error word (one per device that loads the library).
__device__ int g_error_word;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  std::once_flag once;
  int ok = 0;  // 1 = usable (compute capability 10.3)
  int num_sms = 0;
  int* err = nullptr;  // device address of g_error_word
};
DeviceInfo g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

// Current device, checked once: must be compute capability 10.3 (the library is built for
// sm_103a only).  Also resolves the address of this device's error word.
DeviceInfo* current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  DeviceInfo& d = g_dev[dev];
  std::call_once(d.once, [&] {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    if (major != 10 || minor != 3) return;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    d.err = static_cast<int*>(p);
    d.num_sms = sms;
    d.ok = 1;
  });
  return d.ok ? &d : nullptr;
}

struct Types {
  int ab, bias, out;  // Elem codes
  int y;              // Elem code of the gate's Y / the residual R (the operand type by default)
};

// fp8_out: the entry produces fp8 e4m3 (FGEMM_OUT_E4M3 required); otherwise it is refused.
// fp8 operands (FGEMM_E4M3) take an explicit bias type (fp32 / bf16) and output type.
// second: the entry takes a second M x N operand (the gate's Y, the residual's R), whose type
// may be given (FGEMM_Y_*); other entries refuse those bits.
int parse_dtype(int dtype, Types* t, bool fp8_out = false, bool second = false) {
  const int ab = dtype & 0xF, bias = dtype & 0xF0, out = dtype & 0xF00, y = dtype & 0xF000;
  if ((dtype & ~0xFFFF) != 0) return FGEMM_ERR_UNSUPPORTED_DTYPE;
  if (y != FGEMM_Y_SAME && y != FGEMM_Y_F16 && y != FGEMM_Y_BF16) return FGEMM_ERR_UNSUPPORTED_DTYPE;
  if (y != FGEMM_Y_SAME && !second) return FGEMM_ERR_UNSUPPORTED_DTYPE;
  if (ab != FGEMM_F16 && ab != FGEMM_BF16 && ab != FGEMM_E4M3) return FGEMM_ERR_UNSUPPORTED_DTYPE;
  if (bias != FGEMM_BIAS_SAME && bias != FGEMM_BIAS_F32 && bias != FGEMM_BIAS_BF16)
    return FGEMM_ERR_UNSUPPORTED_DTYPE;
  if (fp8_out ? (out != FGEMM_OUT_E4M3)
              : (out != FGEMM_OUT_SAME && out != FGEMM_OUT_F32 && out != FGEMM_OUT_BF16 &&
                 out != FGEMM_OUT_F16))
    return FGEMM_ERR_UNSUPPORTED_DTYPE;
  const bool f8 = ab == FGEMM_E4M3;
  if (f8 && (bias == FGEMM_BIAS_SAME || out == FGEMM_OUT_SAME)) return FGEMM_ERR_UNSUPPORTED_DTYPE;
  t->ab = f8 ? ELEM_E4M3 : ((ab == FGEMM_BF16) ? ELEM_BF16 : ELEM_F16);
  t->bias = (bias == FGEMM_BIAS_F32) ? ELEM_F32 : (bias == FGEMM_BIAS_BF16 ? ELEM_BF16 : t->ab);
  t->out = (out == FGEMM_OUT_F32)    ? ELEM_F32
           : (out == FGEMM_OUT_E4M3) ? ELEM_E4M3
           : (out == FGEMM_OUT_BF16) ? ELEM_BF16
           : (out == FGEMM_OUT_F16)  ? ELEM_F16
                                     : t->ab;
  t->y = (y == FGEMM_Y_F16) ? ELEM_F16 : (y == FGEMM_Y_BF16) ? ELEM_BF16 : t->ab;
  return FGEMM_OK;
}

// The gate's Y / the residual's R: a 16-bit type (explicit with fp8 operands), and with a 16-bit
// output the output has Y's type (the tensor-core epilogue writes the result over the staged Y).
int check_second_operand(const Types& t) {
  if (t.y != ELEM_F16 && t.y != ELEM_BF16) return FGEMM_ERR_UNSUPPORTED_DTYPE;
  if ((t.out == ELEM_F16 || t.out == ELEM_BF16) && t.out != t.y) return FGEMM_ERR_UNSUPPORTED_DTYPE;
  if (t.out == ELEM_E4M3) return FGEMM_ERR_UNSUPPORTED_DTYPE;
  return FGEMM_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

CUtensorMapDataType tma_type(int e) {
  switch (e) {
    case ELEM_F32: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    case ELEM_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    case ELEM_E4M3: return CU_TENSOR_MAP_DATA_TYPE_UINT8;  // stored bytes; no TMA conversion
    default: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  }
}

// Row-major matrix of `rows` x `cols` elements; box of box_rows x box_cols, 128-byte swizzle.
bool encode_2d(CUtensorMap* m, int elem, const void* base, int64_t rows, int64_t cols,
               uint32_t box_rows, uint32_t box_cols,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * elem_bytes(elem)};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, tma_type(elem), 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Call {
  const void *A, *B, *bias, *Y;
  void* out;
  int64_t M, N, K;
  Types t;
  int epi;  // Epi
  cudaStream_t stream;
  const fgemm_opts* opts;
  float out_scale = 1.0f;  // quantized epilogue only
};

int status_of(cudaError_t e) {
  if (e == cudaSuccess) return FGEMM_OK;
  cudaGetLastError();
  return FGEMM_ERR_LAUNCH;
}

// Checks shared by the fused and unfused entries.  Returns FGEMM_OK or an error; sets *nothing
// to true when M or N is zero.
int validate(const Call& c, bool* nothing) {
  *nothing = false;
  if (c.M < 0 || c.N < 0 || c.K < 0 || c.M > 0x7fffffffLL || c.N > 0x7fffffffLL ||
      c.K > 0x7fffffffLL)
    return FGEMM_ERR_INVALID_VALUE;
  if (c.M == 0 || c.N == 0) {
    *nothing = true;
    return FGEMM_OK;
  }
  if (!c.out || (c.epi != EPI_NONE && !c.bias) ||
      ((c.epi == EPI_GATE || c.epi == EPI_RESID) && !c.Y))
    return FGEMM_ERR_INVALID_VALUE;
  if (c.K > 0 && (!c.A || !c.B)) return FGEMM_ERR_INVALID_VALUE;
  const size_t eab = elem_bytes(c.t.ab);
  if ((c.A && !aligned(c.A, eab)) || (c.B && !aligned(c.B, eab)) ||
      (c.Y && !aligned(c.Y, eab)) || (c.bias && !aligned(c.bias, elem_bytes(c.t.bias))) ||
      !aligned(c.out, elem_bytes(c.t.out)))
    return FGEMM_ERR_MISALIGNED;
  if (c.opts) {
    const fgemm_opts& o = *c.opts;
    if (o.group_m < 0 || o.path < 0 || o.path > FGEMM_PATH_KZERO || o.split_k < 0 ||
        o.split_k > 8 || o.max_ctas < 0 || o.timeout_ms < 0 || o.cta_pair < 0 || o.cta_pair > 2 ||
        o.tail_split < 0 || o.tail_split > 1 || o.skinny_tiles < 0 || o.skinny_tiles > 2 || o.stages < 0 || o.stages > 8 ||
        o.inject_stall < 0 || o.inject_stall > 1 || o.bias_init < 0 || o.bias_init > 2 ||
        o.full_last_n < 0 || o.full_last_n > 1 || o.y_blocks < 0 || o.y_blocks > 3 ||
        o.k_rows < 0 || o.k_rows > 2 || o.bias_mma < 0 || o.bias_mma > 2 || o.pdl < 0 ||
        o.pdl > 2 || o.raster < 0 || o.raster > 1 ||
        (o.epi_warps != 0 && o.epi_warps != 8 && o.epi_warps != 16))
      return FGEMM_ERR_INVALID_VALUE;
  }
  return FGEMM_OK;
}

bool tc_eligible(const Call& c) {
  if (c.K % 8 != 0 || c.N % 8 != 0) return false;  // 16-byte row strides for TMA
  if (c.t.ab == ELEM_E4M3 && (c.K % 16 != 0 || c.N % 16 != 0)) return false;  // 1-byte operands
  if (c.t.out == ELEM_E4M3 && c.N % 16 != 0) return false;  // 1-byte outputs: N bytes per row
  return aligned(c.A, 16) && aligned(c.B, 16) && aligned(c.out, 16) &&
         (c.bias == nullptr || aligned(c.bias, 16)) && (c.Y == nullptr || aligned(c.Y, 16));
}

// ---------------------------------------------------------------- launch plans
struct TcPlan {
  bool pair;
  int tiles_m, tiles_n, num_tiles;
  int units;       // persistent CTAs (or CTA pairs)
  int resident;    // pairs that can be resident at once (pair mode), else 0
  int tail_split, full_tiles, num_items;
  int last_width, gran;  // width of the last column of tiles, and the width it is rounded up to
  int y_blocks;          // staged Y blocks per epilogue warp (gate / residual, 16-bit out)
  int k_rows;            // 128-byte K rows per ring stage
  bool row_bars;         // a full barrier per K row of a stage
  bool bias_init;        // the accumulator starts at the bias
  bool bias_mma;         // ... set by an extra MMA from the staged bias row
  int epi_warps;         // epilogue warps per CTA (8, or 16 on single CTAs with a staged Y block)
};

// What the planners need to know about the device: its SM count and how many CTA pairs of the
// tensor-core kernel can be resident at once (< 0: ask the device when pairs are planned).
struct DevShape {
  int num_sms;
  int resident_pairs;
};
DevShape shape_of(const DeviceInfo* d) { return DevShape{d->num_sms, -1}; }

TcPlan plan_tc(const Call& c, const DevShape& d) {
  TcPlan t{};
  const int mode = c.opts ? c.opts->cta_pair : 0;
  // Pairs halve the B bytes each SM stages per MMA, which pays when the main loop is long; with
  // at most 8 K blocks per tile (K <= 512) the per-tile hand-offs dominate and single CTAs are as
  // fast or faster (measured on the GLU block, M = 1024, N = 21568: K = 256 29.9 vs 34.0 us,
  // K = 512 36.9 vs 37.2 us, K = 1024 54.4 vs 45.3 us).
  t.pair = (mode == 2) || (mode == 0 && c.M > 128 && c.K > 512 && d.num_sms >= 2);
  const int TILE_M = t.pair ? 2 * tc_block_m() : tc_block_m(), BN = tc_block_n();
  t.tiles_m = static_cast<int>((c.M + TILE_M - 1) / TILE_M);
  t.tiles_n = static_cast<int>((c.N + BN - 1) / BN);
  const int64_t tiles = static_cast<int64_t>(t.tiles_m) * t.tiles_n;
  t.num_tiles = tiles > 0x7fffffffLL ? -1 : static_cast<int>(tiles);
  if (t.num_tiles < 0) return t;
  // persistent grid: one CTA (or CTA pair) per SM (pair of SMs) that can be resident at once,
  // never more than the tiles
  const int per_unit = t.pair ? 2 : 1;
  int units = d.num_sms / per_unit;
  if (t.pair) {
    t.resident = d.resident_pairs >= 0 ? d.resident_pairs : tc_max_active_pairs(c.epi, c.t.out);
    if (t.resident > 0 && t.resident < units) units = t.resident;
  }
  if (c.opts && c.opts->max_ctas > 0 && c.opts->max_ctas / per_unit < units)
    units = c.opts->max_ctas / per_unit;
  if (units < 1) units = 1;
  if (units > t.num_tiles) units = t.num_tiles;
  t.units = units;
  // Tail: the tiles of the last, partial round are cut along N into pieces so that the round's
  // pieces still fit on the grid (pairs need >= 64 columns per CTA: at most 2 pieces).
  const int rem = t.num_tiles % units;
  int split = 1;
  const bool allow = !(c.opts && c.opts->tail_split == 1);
  if (allow && rem > 0 && t.num_tiles > units) {
    // fp8 outputs are stored 128 columns at a time: pieces stay >= 128 columns wide; fp8
    // operands stage B in 128-column boxes per CTA, so single CTAs keep pieces of >= 128
    // columns, and pairs' 128-column pieces (64 per CTA) take B as 64-byte-swizzled boxes
    int max_split = (t.pair || c.t.out == ELEM_E4M3) ? 2 : 4;
    if (c.t.ab == ELEM_E4M3 && !t.pair) max_split = 2;
    while (split * 2 <= max_split && rem * split * 2 <= units) split *= 2;
  }
  t.tail_split = split;
  t.full_tiles = t.num_tiles - (split > 1 ? rem : 0);
  t.num_items = t.full_tiles + (t.num_tiles - t.full_tiles) * split;
  // Non-power-of-two last tile ("Optimizing GEMM + Activation on CDNA4 with TLX", "Future Work":
  // N = 21568 = 84 x 256 + 64 leaves a ragged last tile): the MMA's N can be any multiple of 16, so
  // the last column of tiles is cut down to the columns left, rounded up to the smallest width
  // that still fills whole 128-byte B boxes on each CTA and whole output staging rows.
  const int box_cols = 128 / static_cast<int>(elem_bytes(c.t.ab));
  const int out_cols = 128 / static_cast<int>(elem_bytes(c.t.out));
  t.gran = (t.pair ? 2 : 1) * box_cols;
  if (t.gran < out_cols) t.gran = out_cols;
  const int left = static_cast<int>(c.N - static_cast<int64_t>(t.tiles_n - 1) * BN);
  t.last_width = (left + t.gran - 1) / t.gran * t.gran;
  if (t.last_width > BN || (c.opts && c.opts->full_last_n)) t.last_width = BN;
  // Gate / residual with 16-bit outputs on CTA pairs (the Y of the second operand staged per
  // epilogue warp; internal y_blocks: 1 = the tile's 8 KB block, 2 = two blocks, 0 = one 4 KB
  // chunk at a time).  K > 1024: chunk at a time, which leaves the ring three two-row stages
  // (the epilogue has a whole main loop of slack); K <= 256: two blocks (Y two tiles ahead);
  // else one block.
  t.y_blocks = 1;
  const bool staged_y = (c.epi == EPI_GATE || c.epi == EPI_RESID) && elem_bytes(c.t.out) == 2;
  if (t.pair && staged_y) {
    const int want = c.opts ? c.opts->y_blocks : 0;
    if (want == 3)
      t.y_blocks = 0;
    else if (want)
      t.y_blocks = want;
    else
      t.y_blocks = c.K > 1024 ? 0 : (c.K <= 256 ? 2 : 1);
  } else if (staged_y) {
    // single CTAs: one block per warp, or two (Y two work items ahead, for a two-stage ring)
    const int want = c.opts ? c.opts->y_blocks : 0;
    t.y_blocks = want == 2 ? 2 : 1;
  }
  // Two K rows per stage on CTA pairs (half the stage hand-offs; 3 stages of 64 KB instead of 6
  // of 32 KB), unless a whole staged Y block per warp leaves room for two stages only.
  t.k_rows = 1;
  if (t.pair) {
    const int want = c.opts ? c.opts->k_rows : 0;
    t.k_rows = want ? want : ((staged_y && t.y_blocks > 0) ? 1 : 2);
    if (t.y_blocks == 2) t.k_rows = 1;
  }
  // Each K row of a two-row stage on its own full barrier: measured faster with fp8 operands and
  // with staged Y, slower on the plain 16-bit FFN shape, equal on 4096^3.
  t.row_bars = t.k_rows > 1 && (c.t.ab == ELEM_E4M3 || staged_y);
  // Bias-initialised accumulator: on by default for short K loops (K <= 1024), where the epilogue
  // sets the pace and moving the bias out of it pays (GLU block, M = 1024, N = 21568, on vs off,
  // each timed after an idle second: K = 256 / 512 / 1024 24.9 vs 26.4, 34.5 vs 35.1, 41.8 vs
  // 42.0 us); with long K loops it does not (4096^3 80.9 vs 80.3 us).
  const int bi = c.opts ? c.opts->bias_init : 0;
  t.bias_init = c.epi != EPI_NONE && (bi == 1 || (bi == 0 && c.K <= 1024));
  // Set by one extra MMA (ones x the staged bias row) instead of by the epilogue warps, where the
  // bias has the 16-bit operand type and the kernel instance has shared memory for the two small
  // tiles it needs (staged second operand; single CTAs, or CTA pairs with one-row stages, where
  // the tiles cost a ring stage).  Automatic for single CTAs with K <= 256 only: measured on the
  // GLU block (M = 1024, N = 21568), alternating on one GB300, K = 256 26.3 vs 26.9 us; K = 512
  // 37.8 vs 35.9 us; CTA pairs at K = 1024 48.9 vs 44.1 us.
  // Sixteen epilogue warps (64 columns each) for single CTAs with one staged Y block per warp.
  t.epi_warps = (!t.pair && staged_y && t.y_blocks == 1 && c.opts && c.opts->epi_warps == 16) ? 16 : 8;
  const int bm = c.opts ? c.opts->bias_mma : 0;
  t.bias_mma = t.bias_init && staged_y && c.t.bias == c.t.ab && c.t.ab != ELEM_F32 &&
               t.y_blocks == 1 && t.k_rows == 1 &&
               (bm == 2 || (bm == 0 && !t.pair && c.K <= 256));
  return t;
}

struct SkPlan {
  int mpad, nt, tmem_cols, tiles_n, groups, split, stages;
};

SkPlan plan_skinny(const Call& c, const DevShape& d) {
  // Default shape of the grid (measured on GB300 for N = K = 8192, M = 1 .. 128): every CTA must
  // be resident at once, two per SM, so the ring is at most 4 stages and small enough that two
  // CTAs fit on an SM, and K is split until the clusters cover 2 x SMs.  One 128-column tile per
  // CTA: sharing A between two tiles halves A's L2 re-reads but measured slower.
  SkPlan s{};
  s.mpad = static_cast<int>((c.M + 15) / 16 * 16);
  s.tiles_n = static_cast<int>((c.N + skinny_block_n() - 1) / skinny_block_n());
  const int kelems = c.t.ab == ELEM_E4M3 ? 128 : 64;  // K per stage: one 128-byte row of A
  const int kb = static_cast<int>((c.K + kelems - 1) / kelems);
  const int want_stages = c.opts ? c.opts->stages : 0;
  int nt = (c.opts && c.opts->skinny_tiles > 0) ? c.opts->skinny_tiles : 1;
  for (;; --nt) {
    s.nt = nt;
    s.groups = (s.tiles_n + nt - 1) / nt;
    int split = (c.opts && c.opts->split_k > 0) ? c.opts->split_k : 0;
    if (split == 0) {
      split = (2 * d.num_sms) / (s.groups > 0 ? s.groups : 1);
      if (split > kb / 4) split = kb / 4;
      if (split > 8) split = 8;
      if (split < 1) split = 1;
    }
    s.split = split;
    int stages = want_stages;
    if (stages == 0) {  // deepest ring (at most 4) with which two CTAs still fit on one SM
      stages = 4;
      while (stages > 2 && skinny_smem_bytes(s.mpad, nt, split, stages) > 113 * 1024) --stages;
    }
    s.stages = stages;
    if (nt == 1 || skinny_fits(s.mpad, nt, split, stages)) break;
  }
  s.tmem_cols = 32;
  while (s.tmem_cols < s.nt * s.mpad) s.tmem_cols *= 2;
  return s;
}

// Programmatic dependent launch (fgemm_opts.pdl), on by default on both paths: the launch gap
// and set-up between consecutive kernels (about 1.5 us) overlap the previous kernel's last CTAs.
// Measured on one GB300, CUDA-graph replay of back-to-back calls, each variant timed after a
// second of idle GPU: GLU block M = 1024, N = 21568, K = 256 / 512 / 1024 25.5 -> 24.9,
// 35.3 -> 34.5, 43.2 -> 41.8 us; 4096^3 80.3 -> 79.6 us, fp8 4096^3 48.0 -> 46.7 us, fp8 GLU block
// K = 4096 67.8 -> 66.4 us, FFN 8192 x 14336 x 4096 551.6 -> 547.5 us; skinny N = K = 8192,
// M = 1 / 128 24.5 -> 24.0, 29.4 -> 28.6 us.
int pdl_of(const Call& c) {
  const int want = c.opts ? c.opts->pdl : 0;
  return want == 2 ? 0 : 1;
}

int run_tc(const Call& c, DeviceInfo* d) {
  const TcPlan t = plan_tc(c, shape_of(d));
  if (t.num_tiles < 0) return FGEMM_ERR_INVALID_VALUE;
  const int BM = tc_block_m(), BN = tc_block_n();
  const int TILE_M = t.pair ? 2 * BM : BM;
  CUtensorMap tmA, tmB, tmO, tmY;
  const uint32_t out_box_cols = 128u / static_cast<uint32_t>(elem_bytes(c.t.out));
  const uint32_t kb_elems = 128u / static_cast<uint32_t>(elem_bytes(c.t.ab));  // one 128-B row
  if (!encode_2d(&tmA, c.t.ab, c.A, c.M, c.K, BM, kb_elems) ||
      !encode_2d(&tmB, c.t.ab, c.B, c.K, c.N,
                 kb_elems * static_cast<uint32_t>(t.row_bars ? 1 : t.k_rows), kb_elems) ||
      !encode_2d(&tmO, c.t.out, c.out, c.M, c.N, 32, out_box_cols))
    return FGEMM_ERR_LAUNCH;
  if ((c.epi == EPI_GATE || c.epi == EPI_RESID) && c.t.out != ELEM_F32) {
    if (!encode_2d(&tmY, c.t.y, c.Y, c.M, c.N, 32, 64)) return FGEMM_ERR_LAUNCH;
  } else {
    tmY = tmO;  // unused
  }
  CUtensorMap tmBias = tmO;  // unused unless the bias MMA runs
  if (t.bias_mma && !encode_2d(&tmBias, c.t.bias, c.bias, 1, c.N, 1, 64)) return FGEMM_ERR_LAUNCH;
  CUtensorMap tmB64 = tmB;  // fp8 pairs' column pieces: 64-column, 64-byte-swizzled B boxes
  if (t.pair && c.t.ab == ELEM_E4M3 && t.tail_split > 1 &&
      !encode_2d(&tmB64, c.t.ab, c.B, c.K, c.N,
                 kb_elems * static_cast<uint32_t>(t.row_bars ? 1 : t.k_rows), 64,
                 CU_TENSOR_MAP_SWIZZLE_64B))
    return FGEMM_ERR_LAUNCH;
  TcParams p{};
  p.M = static_cast<int>(c.M);
  p.N = static_cast<int>(c.N);
  p.K = static_cast<int>(c.K);
  p.tiles_m = t.tiles_m;
  p.tiles_n = t.tiles_n;
  p.num_tiles = t.num_tiles;
  p.full_tiles = t.full_tiles;
  p.tail_split = t.tail_split;
  p.num_items = t.num_items;
  p.last_width = t.last_width;
  p.gran = t.gran;
  p.bias_init = t.bias_init ? 1 : 0;
  p.bias_mma = t.bias_mma ? 1 : 0;
  p.y_blocks = t.y_blocks;
  p.epi_warps = t.epi_warps;
  p.k_rows = t.k_rows;
  p.row_bars = t.row_bars ? 1 : 0;
  // 16 M-tiles per band: measured best on the 8192-row FFN (577-583 vs 595-605 us for 8); the
  // square and GLU shapes have at most 16 tile rows, so every value from there up is the same order
  p.group = (c.opts && c.opts->group_m > 0) ? c.opts->group_m : 16;
  p.raster_n = (c.opts && c.opts->raster == 1) ? 1 : 0;
  p.ab_bf16 = c.t.ab == ELEM_BF16;
  p.ab_f8 = c.t.ab == ELEM_E4M3;
  p.y_bf16 = c.t.y == ELEM_BF16;
  p.bias_type = c.t.bias;
  p.out_type = c.t.out;
  p.bias = c.bias;
  p.Y = c.Y;
  p.out_scale = c.out_scale;
  p.idesc = idesc_f16_f32acc(p.ab_bf16 != 0, TILE_M, BN, /*a_mn=*/false, /*b_mn=*/true);
  const int tmo_ms = (c.opts && c.opts->timeout_ms > 0) ? c.opts->timeout_ms : 1000;
  p.timeout_ns = static_cast<uint64_t>(tmo_ms) * 1000000ull;
  p.err = d->err;
  p.inject_stall = (c.opts && c.opts->inject_stall) ? 1 : 0;
  p.pdl = pdl_of(c);
  return status_of(
      launch_tc(c.epi, tmA, tmB, tmO, tmY, tmBias, tmB64, p, t.units * (t.pair ? 2 : 1), t.pair,
                c.stream));
}

int run_skinny(const Call& c, DeviceInfo* d) {
  const SkPlan s = plan_skinny(c, shape_of(d));
  CUtensorMap tmB, tmA;
  // one 128-byte row of K per stage: B as 64 x 64 boxes (16-bit) or one 128 x 128 box (fp8)
  const uint32_t kelems = c.t.ab == ELEM_E4M3 ? 128u : 64u;
  if (!encode_2d(&tmB, c.t.ab, c.B, c.K, c.N, kelems, kelems) ||
      !encode_2d(&tmA, c.t.ab, c.A, c.M, c.K, static_cast<uint32_t>(s.mpad), kelems))
    return FGEMM_ERR_LAUNCH;
  SkParams p{};
  p.M = static_cast<int>(c.M);
  p.N = static_cast<int>(c.N);
  p.K = static_cast<int>(c.K);
  p.mpad = s.mpad;
  p.nt = s.nt;
  p.tmem_cols = s.tmem_cols;
  p.split = s.split;
  p.stages = s.stages;
  p.ab_type = c.t.ab;
  p.y_type = c.t.y;
  p.bias_type = c.t.bias;
  p.out_type = c.t.out;
  p.bias = c.bias;
  p.Y = c.Y;
  p.out = c.out;
  p.out_scale = c.out_scale;
  p.idesc = idesc_f16_f32acc(c.t.ab == ELEM_BF16, skinny_block_n(), s.mpad, /*a_mn=*/true,
                             /*b_mn=*/false);
  const int tmo_ms = (c.opts && c.opts->timeout_ms > 0) ? c.opts->timeout_ms : 1000;
  p.timeout_ns = static_cast<uint64_t>(tmo_ms) * 1000000ull;
  p.err = d->err;
  p.inject_stall = (c.opts && c.opts->inject_stall) ? 1 : 0;
  p.pdl = pdl_of(c);
  if (!skinny_fits(s.mpad, s.nt, s.split, s.stages)) return FGEMM_ERR_INVALID_VALUE;
  return status_of(launch_skinny(c.epi, tmB, tmA, p, s.groups * s.split, c.stream));
}

SimtParams simt_params(const Call& c) {
  SimtParams p{};
  p.A = c.A;
  p.B = c.B;
  p.bias = c.bias;
  p.Y = c.Y;
  p.out = c.out;
  p.M = static_cast<int>(c.M);
  p.N = static_cast<int>(c.N);
  p.K = static_cast<int>(c.K);
  p.ab_type = c.t.ab;
  p.y_type = c.t.y;
  p.bias_type = c.t.bias;
  p.out_type = c.t.out;
  p.out_scale = c.out_scale;
  return p;
}

// Choose the path for a validated, non-empty call.
int choose_path(const Call& c, int* out_path) {
  const int forced = c.opts ? c.opts->path : FGEMM_PATH_AUTO;
  int path;
  if (forced == FGEMM_PATH_AUTO) {
    if (c.K == 0)
      path = (c.epi == EPI_NONE) ? FGEMM_PATH_GENERIC : FGEMM_PATH_KZERO;
    else if (!tc_eligible(c))
      path = FGEMM_PATH_GENERIC;
    else
      path = c.M <= skinny_max_m() ? FGEMM_PATH_SKINNY : FGEMM_PATH_TC;
  } else {
    path = forced;
    if (path == FGEMM_PATH_TC && (c.K == 0 || !tc_eligible(c))) return FGEMM_ERR_INVALID_VALUE;
    if (path == FGEMM_PATH_SKINNY && (c.K == 0 || !tc_eligible(c) || c.M > skinny_max_m()))
      return FGEMM_ERR_INVALID_VALUE;
    if (path == FGEMM_PATH_KZERO && (c.K != 0 || c.epi == EPI_NONE)) return FGEMM_ERR_INVALID_VALUE;
  }
  *out_path = path;
  return FGEMM_OK;
}

// Choose and run a path for a validated, non-empty call.
int dispatch(const Call& c, DeviceInfo* d, int* path_taken) {
  int path = 0;
  const int st = choose_path(c, &path);
  if (st != FGEMM_OK) return st;
  if (path_taken) *path_taken = path;
  switch (path) {
    case FGEMM_PATH_TC: return run_tc(c, d);
    case FGEMM_PATH_SKINNY: return run_skinny(c, d);
    case FGEMM_PATH_KZERO: return status_of(launch_kzero(c.epi, simt_params(c), d->num_sms, c.stream));
    default: return status_of(launch_generic(c.epi, simt_params(c), c.stream));
  }
}

int fused(const Call& c, int* path_taken) {
  if (path_taken) *path_taken = FGEMM_PATH_NONE;
  bool nothing = false;
  int st = validate(c, &nothing);
  if (st != FGEMM_OK || nothing) return st;
  DeviceInfo* d = current_device();
  if (!d) return FGEMM_ERR_NO_DEVICE;
  return dispatch(c, d, path_taken);
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace
}  // namespace fgemm

using namespace fgemm;

extern "C" {

int fgemm_bias_relu_ex(const void* A, const void* B, const void* bias, void* out, int64_t M,
                       int64_t N, int64_t K, int dtype, void* stream, const fgemm_opts* opts,
                       int* path_taken) {
  Call c{A, B, bias, nullptr, out, M, N, K, {}, EPI_RELU, static_cast<cudaStream_t>(stream), opts};
  const int st = parse_dtype(dtype, &c.t);
  if (st != FGEMM_OK) return st;
  return fused(c, path_taken);
}

int fgemm_addmm_gate_ex(const void* A, const void* B, const void* bias, const void* Y, void* out,
                        int64_t M, int64_t N, int64_t K, int dtype, void* stream,
                        const fgemm_opts* opts, int* path_taken) {
  Call c{A, B, bias, Y, out, M, N, K, {}, EPI_GATE, static_cast<cudaStream_t>(stream), opts};
  int st = parse_dtype(dtype, &c.t, false, true);
  if (st == FGEMM_OK) st = check_second_operand(c.t);
  if (st != FGEMM_OK) return st;
  return fused(c, path_taken);
}

int fgemm_bias_residual_relu_ex(const void* A, const void* B, const void* bias, const void* R,
                                void* out, int64_t M, int64_t N, int64_t K, int dtype,
                                void* stream, const fgemm_opts* opts, int* path_taken) {
  Call c{A, B, bias, R, out, M, N, K, {}, EPI_RESID, static_cast<cudaStream_t>(stream), opts};
  int st = parse_dtype(dtype, &c.t, false, true);
  if (st == FGEMM_OK) st = check_second_operand(c.t);
  if (st != FGEMM_OK) return st;
  return fused(c, path_taken);
}

int fgemm_bias_residual_relu(const void* A, const void* B, const void* bias, const void* R,
                             void* out, int64_t M, int64_t N, int64_t K, int dtype, void* stream) {
  return fgemm_bias_residual_relu_ex(A, B, bias, R, out, M, N, K, dtype, stream, nullptr, nullptr);
}

int fgemm_bias_relu_quant_ex(const void* A, const void* B, const void* bias, void* out, int64_t M,
                             int64_t N, int64_t K, int dtype, float scale, void* stream,
                             const fgemm_opts* opts, int* path_taken) {
  Call c{A, B, bias, nullptr, out, M, N, K, {}, EPI_QUANT, static_cast<cudaStream_t>(stream), opts};
  c.out_scale = scale;
  const int st = parse_dtype(dtype, &c.t, /*fp8_out=*/true);
  if (st != FGEMM_OK) return st;
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return FGEMM_ERR_INVALID_VALUE;
  return fused(c, path_taken);
}

int fgemm_bias_relu_quant(const void* A, const void* B, const void* bias, void* out, int64_t M,
                          int64_t N, int64_t K, int dtype, float scale, void* stream) {
  return fgemm_bias_relu_quant_ex(A, B, bias, out, M, N, K, dtype, scale, stream, nullptr, nullptr);
}

int fgemm_bias_relu(const void* A, const void* B, const void* bias, void* out, int64_t M,
                    int64_t N, int64_t K, int dtype, void* stream) {
  return fgemm_bias_relu_ex(A, B, bias, out, M, N, K, dtype, stream, nullptr, nullptr);
}

int fgemm_addmm_gate(const void* A, const void* B, const void* bias, const void* Y, void* out,
                     int64_t M, int64_t N, int64_t K, int dtype, void* stream) {
  return fgemm_addmm_gate_ex(A, B, bias, Y, out, M, N, K, dtype, stream, nullptr, nullptr);
}

size_t fgemm_unfused_workspace_bytes(int64_t M, int64_t N, int dtype, int inter_f32) {
  Types t{};
  if (parse_dtype(dtype, &t, false, true) != FGEMM_OK || M < 0 || N < 0) return 0;
  const size_t e = inter_f32 ? 4 : static_cast<size_t>(elem_bytes(t.out));
  return round_up(static_cast<size_t>(M) * static_cast<size_t>(N) * e, 256);
}

static int unfused(const void* A, const void* B, const void* bias, const void* Y, void* out,
                   int64_t M, int64_t N, int64_t K, int dtype, void* workspace,
                   size_t workspace_bytes, int inter_f32, void* stream, int epi) {
  Call fin{A, B, bias, Y, out, M, N, K, {}, epi, static_cast<cudaStream_t>(stream), nullptr};
  int st = parse_dtype(dtype, &fin.t, false, epi == EPI_GATE);
  if (st == FGEMM_OK && epi == EPI_GATE) st = check_second_operand(fin.t);
  if (st != FGEMM_OK) return st;
  if (fin.t.ab == ELEM_E4M3) return FGEMM_ERR_UNSUPPORTED_DTYPE;
  bool nothing = false;
  st = validate(fin, &nothing);
  if (st != FGEMM_OK || nothing) return st;
  const size_t need = fgemm_unfused_workspace_bytes(M, N, dtype, inter_f32);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return FGEMM_ERR_WORKSPACE;
  DeviceInfo* d = current_device();
  if (!d) return FGEMM_ERR_NO_DEVICE;
  const int inter = inter_f32 ? ELEM_F32 : fin.t.out;
  // step 1: plain GEMM, I = A @ B (rounded once to the intermediate type)
  Call g = fin;
  g.epi = EPI_NONE;
  g.bias = nullptr;
  g.Y = nullptr;
  g.out = workspace;
  g.t.out = inter;
  st = dispatch(g, d, nullptr);
  if (st != FGEMM_OK) return st;
  const int m = static_cast<int>(M), n = static_cast<int>(N);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (epi == EPI_RELU) {
    // step 2: I = I + bias (read + write I); step 3: out = ReLU(I) (read I, write out)
    st = status_of(launch_ew_bias_inplace(workspace, inter, bias, fin.t.bias, m, n, d->num_sms, s));
    if (st != FGEMM_OK) return st;
    return status_of(launch_ew_relu(workspace, inter, out, fin.t.out, m, n, d->num_sms, s));
  }
  // step 2: out = (I + bias) + (I + bias) * Y
  return status_of(launch_ew_bias_gate(workspace, inter, bias, fin.t.bias, Y, fin.t.y, out,
                                       fin.t.out, m, n, d->num_sms, s));
}

int fgemm_unfused_bias_relu(const void* A, const void* B, const void* bias, void* out, int64_t M,
                            int64_t N, int64_t K, int dtype, void* workspace,
                            size_t workspace_bytes, int inter_f32, void* stream) {
  return unfused(A, B, bias, nullptr, out, M, N, K, dtype, workspace, workspace_bytes, inter_f32,
                 stream, EPI_RELU);
}

int fgemm_unfused_addmm_gate(const void* A, const void* B, const void* bias, const void* Y,
                             void* out, int64_t M, int64_t N, int64_t K, int dtype,
                             void* workspace, size_t workspace_bytes, int inter_f32,
                             void* stream) {
  return unfused(A, B, bias, Y, out, M, N, K, dtype, workspace, workspace_bytes, inter_f32, stream,
                 EPI_GATE);
}

int fgemm_device_status(void* stream, int* code) {
  if (!code) return FGEMM_ERR_INVALID_VALUE;
  *code = 0;
  if (!current_device()) return FGEMM_ERR_NO_DEVICE;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return FGEMM_ERR_LAUNCH;
  }
  int v = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return FGEMM_ERR_LAUNCH;
  }
  *code = v;
  return FGEMM_OK;
}

const char* fgemm_status_string(int s) {
  switch (s) {
    case FGEMM_OK: return "FGEMM_OK";
    case FGEMM_ERR_INVALID_VALUE: return "FGEMM_ERR_INVALID_VALUE";
    case FGEMM_ERR_UNSUPPORTED_DTYPE: return "FGEMM_ERR_UNSUPPORTED_DTYPE";
    case FGEMM_ERR_MISALIGNED: return "FGEMM_ERR_MISALIGNED";
    case FGEMM_ERR_NO_DEVICE: return "FGEMM_ERR_NO_DEVICE";
    case FGEMM_ERR_LAUNCH: return "FGEMM_ERR_LAUNCH";
    case FGEMM_ERR_TIMEOUT: return "FGEMM_ERR_TIMEOUT";
    case FGEMM_ERR_WORKSPACE: return "FGEMM_ERR_WORKSPACE";
    default: return "FGEMM_ERR_UNKNOWN";
  }
}

}  // extern "C"

namespace {

// fgemm_plan / fgemm_plan_on: the plan for the device `shape` (nullptr: the current device).
int plan_info(const void* A, const void* B, const void* bias, const void* Y, const void* out,
              int64_t M, int64_t N, int64_t K, int dtype, int epilogue, const fgemm_opts* opts,
              const DevShape* shape, fgemm_plan_info* info) {
  if (!info) return FGEMM_ERR_INVALID_VALUE;
  *info = fgemm_plan_info{};
  info->path = FGEMM_PATH_NONE;
  if (epilogue < FGEMM_EPI_RELU || epilogue > FGEMM_EPI_RELU_QUANT) return FGEMM_ERR_INVALID_VALUE;
  const int epi = epilogue == FGEMM_EPI_GATE ? EPI_GATE
                : epilogue == FGEMM_EPI_RESIDUAL_RELU ? EPI_RESID
                : epilogue == FGEMM_EPI_RELU_QUANT ? EPI_QUANT : EPI_RELU;
  Call c{A, B, bias, (epi == EPI_GATE || epi == EPI_RESID) ? Y : nullptr, const_cast<void*>(out),
         M, N, K, {}, epi, nullptr, opts};
  const bool second = epi == EPI_GATE || epi == EPI_RESID;
  int st = parse_dtype(dtype, &c.t, epi == EPI_QUANT, second);
  if (st == FGEMM_OK && second) st = check_second_operand(c.t);
  if (st != FGEMM_OK) return st;
  bool nothing = false;
  st = validate(c, &nothing);
  if (st != FGEMM_OK || nothing) return st;
  DevShape dev{};
  if (shape) {
    dev = *shape;
  } else {
    DeviceInfo* d = current_device();
    if (!d) return FGEMM_ERR_NO_DEVICE;
    dev = shape_of(d);
  }
  int path = 0;
  st = choose_path(c, &path);
  if (st != FGEMM_OK) return st;
  info->path = path;
  info->cluster = 1;
  info->tail_split = 1;
  if (path == FGEMM_PATH_TC) {
    const TcPlan t = plan_tc(c, dev);
    if (t.num_tiles < 0) return FGEMM_ERR_INVALID_VALUE;
    info->cluster = t.pair ? 2 : 1;
    info->grid = t.units * info->cluster;
    info->tiles = t.num_tiles;
    info->work_items = t.num_items;
    info->tail_split = t.tail_split;
    info->last_tile_n = t.last_width;
    info->y_blocks = t.y_blocks == 0 ? 3 : t.y_blocks;
    info->k_rows = t.k_rows;
    info->resident_pairs = t.resident;
    info->row_barriers = t.row_bars ? 1 : 0;
    info->bias_init = t.bias_init ? (t.bias_mma ? 2 : 1) : 0;
    info->epi_warps = t.epi_warps;
  } else if (path == FGEMM_PATH_SKINNY) {
    const SkPlan s = plan_skinny(c, dev);
    info->cluster = s.split;
    info->grid = s.groups * s.split;
    info->tiles = s.tiles_n;
    info->work_items = s.groups * s.split;
    info->tail_split = s.nt;  // reused: 128-column tiles per CTA on the skinny path
  }
  return FGEMM_OK;
}

}  // namespace

extern "C" {

int fgemm_plan(const void* A, const void* B, const void* bias, const void* Y, const void* out,
               int64_t M, int64_t N, int64_t K, int dtype, int epilogue, const fgemm_opts* opts,
               fgemm_plan_info* info) {
  return plan_info(A, B, bias, Y, out, M, N, K, dtype, epilogue, opts, nullptr, info);
}

int fgemm_plan_on(const void* A, const void* B, const void* bias, const void* Y, const void* out,
                  int64_t M, int64_t N, int64_t K, int dtype, int epilogue, const fgemm_opts* opts,
                  int num_sms, int resident_pairs, fgemm_plan_info* info) {
  if (num_sms < 1 || resident_pairs < 0) {
    if (info) {
      *info = fgemm_plan_info{};
      info->path = FGEMM_PATH_NONE;
    }
    return FGEMM_ERR_INVALID_VALUE;
  }
  const DevShape shape{num_sms, resident_pairs};
  return plan_info(A, B, bias, Y, out, M, N, K, dtype, epilogue, opts, &shape, info);
}

int fgemm_tile_of(int64_t t, int64_t tiles_m, int64_t tiles_n, int group, int64_t* m_tile,
                  int64_t* n_tile) {
  if (!m_tile || !n_tile || tiles_m <= 0 || tiles_n <= 0 || group <= 0 || t < 0 ||
      tiles_m > 0x7fffffffLL || tiles_n > 0x7fffffffLL || t >= tiles_m * tiles_n)
    return FGEMM_ERR_INVALID_VALUE;
  int m = 0, n = 0;
  tile_of(t, static_cast<int>(tiles_m), static_cast<int>(tiles_n), group, m, n);
  *m_tile = m;
  *n_tile = n;
  return FGEMM_OK;
}

}  // extern "C"
