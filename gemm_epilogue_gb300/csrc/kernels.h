// kernels.h -- internal launch interface between the C ABI (api.cu) and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fgemm {

// EPI_RESID: out = ReLU(acc + bias + R) with R (M x N, operand type) passed where the gate's Y is.
// EPI_QUANT: out = e4m3(clamp(out_scale * ReLU(acc + bias), -448, 448)), fp8 output.
enum Epi : int { EPI_RELU = 0, EPI_GATE = 1, EPI_NONE = 2, EPI_RESID = 3, EPI_QUANT = 4 };
enum Elem : int { ELEM_F16 = 0, ELEM_BF16 = 1, ELEM_F32 = 2, ELEM_E4M3 = 3 };

inline int elem_bytes(int e) { return e == ELEM_F32 ? 4 : (e == ELEM_E4M3 ? 1 : 2); }

// Arguments of the persistent tensor-core kernel (tensor maps travel separately as
// __grid_constant__ parameters).
struct TcParams {
  int M, N, K;
  int tiles_m, tiles_n, num_tiles, group;
  int raster_n;    // 1: the grouped order runs over N (bands of `group` N-tiles, N fastest inside)
  // Work items: items 0 .. full_tiles-1 are whole tiles; the remaining num_tiles - full_tiles tiles
  // (the last, partial round of the persistent grid) are each cut into `tail_split` pieces along N
  // (256 / tail_split columns each) so that the last round takes a fraction of a tile's time.
  int full_tiles, tail_split, num_items;
  // The last column of tiles is narrowed to `last_width` columns (the columns left of N, rounded up
  // to `gran`, the smallest width one CTA (pair) can stage and store); pieces of it that start at
  // or past that width are `gran` wide and store nothing.
  int last_width, gran;
  int bias_init;   // 1: the accumulator starts at the bias
  int bias_mma;    // with bias_init: 1 = set by an extra MMA from the staged bias row (16-bit bias of
                   // the operand type, instances with room for it), 0 = written into TMEM
  int y_blocks;    // gate / residual with 16-bit out on CTA pairs: Y blocks per epilogue warp (1, 2)
  int epi_warps;   // epilogue warps: 8, or 16 (single CTAs with one staged Y block per warp)
  int k_rows;      // CTA pairs: 128-byte K rows per ring stage (1, 2)
  int row_bars;    // k_rows 2: a full barrier per K row of a stage (B copied one K row at a time)
  int ab_bf16;     // operand (and Y) type: 0 = f16, 1 = bf16
  int ab_f8;       // 1: A and B are fp8 e4m3 (kind::f8f6f4 MMAs, 128-element K blocks)
  int y_bf16;      // the gate's Y / the residual's R: 0 = f16, 1 = bf16
  int bias_type;   // Elem of the bias
  int out_type;    // Elem of out
  const void* bias;
  const void* Y;   // gate only, M x N operand type
  float out_scale; // quantized epilogue only
  uint32_t idesc;  // tcgen05 instruction descriptor
  uint64_t timeout_ns;
  int* err;        // device error word
  int inject_stall;  // diagnostic: CTA 0 skips the loads of its first stage (see fgemm_opts)
  int pdl;           // launched with programmatic stream serialization (see fgemm_opts)
};

// Generic CUDA-core kernel and elementwise kernels: plain pointers.
struct SimtParams {
  const void* A;
  const void* B;
  const void* bias;  // may be NULL for EPI_NONE
  const void* Y;
  void* out;
  int M, N, K;
  int ab_type;    // Elem
  int y_type;     // Elem of Y / R
  int bias_type;  // Elem
  int out_type;   // Elem
  float out_scale;  // quantized epilogue only
};

// pair = true: 2-CTA clusters (grid even), 256 x 256 tiles, tiles_m counted in 256-row tiles.
// tmY: the gate's Y (M x N, operand type, 32 x 64 boxes, 128-byte swizzle); any map otherwise.
// tmBias: the bias as a 1 x N tensor (64-column boxes, 128-byte swizzle) for the bias MMA; any
// map otherwise.
// tmB64: fp8 operands on CTA pairs, B as 64-column boxes with 64-byte swizzle (the column pieces
// of the last round, 64 columns per CTA); any map otherwise.
cudaError_t launch_tc(int epi, const CUtensorMap& tmA, const CUtensorMap& tmB,
                      const CUtensorMap& tmOut, const CUtensorMap& tmY, const CUtensorMap& tmBias,
                      const CUtensorMap& tmB64, const TcParams& p, int grid, bool pair,
                      cudaStream_t s);
// How many CTA pairs of the pair-mode kernel can be resident at once (clusters need two free SMs
// in one GPC); cached per process.
int tc_max_active_pairs(int epi, int out_type);
int tc_block_m();
int tc_block_n();

// Small-M kernel (swap-AB, split-K over a cluster, reduction through distributed shared memory).
struct SkParams {
  int M, N, K;
  int mpad;       // M rounded up to a multiple of 16 (the MMA's N), <= 128
  int nt;         // 128-column tiles per CTA (1 or 2), sharing each staged block of A
  int tmem_cols;  // power of two >= 32 and >= nt * mpad
  int split;      // CTAs per cluster splitting K (1..8)
  int stages;     // ring depth requested (0 = default)
  int ab_type, bias_type, out_type;  // Elem
  int y_type;     // Elem of Y / R
  const void* bias;
  const void* Y;
  void* out;
  float out_scale;  // quantized epilogue only
  uint32_t idesc;
  uint64_t timeout_ns;
  int* err;
  int inject_stall;  // diagnostic: CTA 0 skips the loads of its first stage (see fgemm_opts)
  int pdl;           // launched with programmatic stream serialization (see fgemm_opts)
};
cudaError_t launch_skinny(int epi, const CUtensorMap& tmB, const CUtensorMap& tmA,
                          const SkParams& p, int ctas, cudaStream_t s);
int skinny_block_n();
int skinny_max_m();
// Whether the stage ring and the cluster-reduction buffer fit in shared memory.
bool skinny_fits(int mpad, int nt, int split, int stages);
uint32_t skinny_smem_bytes(int mpad, int nt, int split, int stages);

cudaError_t launch_generic(int epi, const SimtParams& p, cudaStream_t s);

// K == 0: out[i,j] = epilogue(0 + bias[j], Y[i,j])
cudaError_t launch_kzero(int epi, const SimtParams& p, int num_sms, cudaStream_t s);

// Unfused chain pieces.  I is M x N of type inter_type.
cudaError_t launch_ew_bias_inplace(void* I, int inter_type, const void* bias, int bias_type, int M,
                                   int N, int num_sms, cudaStream_t s);
cudaError_t launch_ew_relu(const void* I, int inter_type, void* out, int out_type, int M, int N,
                           int num_sms, cudaStream_t s);
cudaError_t launch_ew_bias_gate(const void* I, int inter_type, const void* bias, int bias_type,
                                const void* Y, int y_type, void* out, int out_type, int M, int N,
                                int num_sms, cudaStream_t s);

}  // namespace fgemm
