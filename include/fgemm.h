/*
 * fgemm.h -- C ABI of the fused GEMM + epilogue library for NVIDIA GB300 (sm_103a).
 *
 * Fused operations, each one kernel launch in which the fp32 accumulator never leaves the chip
 * (tensor memory) between the end of the K reduction and the single store:
 *
 *   fgemm_bias_relu   out[i,j] = max(0, sum_k A[i,k] B[k,j] + bias[j])
 *       "Triton: Fused Matmul + Bias + ReLU (Epilogue Fusion)", the defining equation: the bias is
 *       per column, broadcast over rows, added once after the K loop; "Epilogue concept", "Where
 *       the accumulator is finally correct": bias and activation run on the complete sum.
 *
 *   fgemm_addmm_gate  X = A @ B + bias;  out = X + X * Y
 *       "Optimizing GEMM + Activation on CDNA4 with TLX", "The GLU Block" (the projection, then
 *       the elementwise gate with a second tensor Y of the output's shape), evaluated as
 *       fma(X, Y, X) as in that page's "Version 4: Making the Epilogue Nearly Free".
 *
 *   fgemm_bias_residual_relu  out = max(0, A @ B + bias + R)      ("Variants": residual add)
 *   fgemm_bias_relu_quant     out = e4m3(clamp(scale * max(0, A @ B + bias), +-448))
 *                                                        ("Variants": quantized output)
 *
 * Rounding: products are accumulated in fp32; the epilogue runs in fp32; the result is rounded
 * once (round to nearest even) to the output type at the store ("I3. Fuse a GEMM epilogue and
 * change tile scheduling", opening paragraph and "Why the baseline uses FP32").  On the tensor-core
 * path with K <= 1024 the fp32 sum starts at the bias instead of taking it last (the same value up
 * to the rounding order; fgemm_opts.bias_init selects either order).
 *
 * K = 0 is valid: the zero accumulator still passes through the epilogue, so bias+ReLU gives
 * ReLU(bias) on every row ("I3 ...", "Implement in stages", stage 2); the gate gives
 * bias + bias * Y.  A and B may then be NULL.
 *
 * Conventions shared by every entry point
 *   Layout     dense row-major, no leading-dimension arguments: A is M x K, B is K x N, Y and out
 *              are M x N, bias has N elements.
 *   Pointers   device pointers owned by the caller.  The library allocates nothing per call.
 *   Stream     `stream` is a cudaStream_t (NULL = legacy default stream).  Calls return after
 *              enqueueing the work; in-kernel failures are read with fgemm_device_status().
 *   Aliasing   out must not overlap A, B, bias or Y (undefined behaviour).
 *   Sizes      M, N, K >= 0 and each below 2^31; M == 0 or N == 0 returns FGEMM_OK without a launch.
 *   Alignment  every pointer must be aligned to its element size (else FGEMM_ERR_MISALIGNED).
 *              The tensor-core path additionally needs 16-byte aligned base pointers and row
 *              strides (K and N multiples of 8); other shapes run on the generic CUDA-core path,
 *              which is not an error.
 *   Threading  no per-call global state: per device, the library keeps the error word, cached
 *              launch attributes (set once, idempotent) and, for fgemm_unfused_bias_relu_noalloc
 *              only, its scratch array.
 */
#ifndef FGEMM_H
#define FGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FGEMM_OK = 0,
  FGEMM_ERR_INVALID_VALUE = 1,     /* negative size, NULL pointer where data is needed, bad option */
  FGEMM_ERR_UNSUPPORTED_DTYPE = 2, /* unknown dtype word */
  FGEMM_ERR_MISALIGNED = 3,        /* a pointer not aligned to its element size */
  FGEMM_ERR_NO_DEVICE = 4,         /* no current CUDA device, or not compute capability 10.3 */
  FGEMM_ERR_LAUNCH = 5,            /* a CUDA call or kernel launch failed */
  FGEMM_ERR_TIMEOUT = 6,           /* a device-side wait exceeded its bound (see fgemm_opts) */
  FGEMM_ERR_WORKSPACE = 7          /* workspace NULL or smaller than required */
} fgemm_status;

/* dtype word = operand type | bias type | output type [| Y type].  The gate's Y (and the residual's
   R) has the operand type unless a Y type is given. */
#define FGEMM_F16 0x1        /* A, B (and Y) are IEEE binary16 */
#define FGEMM_BF16 0x2       /* A, B (and Y) are bfloat16 */
#define FGEMM_E4M3 0x3       /* A, B are fp8 e4m3 (the bias and output types must then be given
                                explicitly, and for the gate and the residual the Y type as well;
                                tensor-core path for K, N multiples of 16, CUDA-core path
                                otherwise) */
#define FGEMM_BIAS_SAME 0x00 /* bias has the operand type (16-bit operands) */
#define FGEMM_BIAS_F32 0x10  /* bias is fp32 */
#define FGEMM_BIAS_BF16 0x20 /* bias is bfloat16 */
#define FGEMM_OUT_SAME 0x000 /* out has the operand type (16-bit operands) */
#define FGEMM_OUT_F32 0x100  /* out is fp32 */
#define FGEMM_OUT_E4M3 0x200 /* out is fp8 e4m3 (fgemm_bias_relu_quant only) */
#define FGEMM_OUT_BF16 0x300 /* out is bfloat16 */
#define FGEMM_OUT_F16 0x400  /* out is IEEE binary16 */
#define FGEMM_Y_SAME 0x0000  /* Y (or R) has the operand type (16-bit operands) */
#define FGEMM_Y_F16 0x1000   /* Y (or R) is IEEE binary16 (fgemm_addmm_gate, fgemm_bias_residual_relu) */
#define FGEMM_Y_BF16 0x2000  /* Y (or R) is bfloat16 (fgemm_addmm_gate, fgemm_bias_residual_relu) */

/* Epilogue codes (fgemm_plan). */
#define FGEMM_EPI_RELU 0          /* fgemm_bias_relu */
#define FGEMM_EPI_GATE 1          /* fgemm_addmm_gate */
#define FGEMM_EPI_RESIDUAL_RELU 2 /* fgemm_bias_residual_relu */
#define FGEMM_EPI_RELU_QUANT 3    /* fgemm_bias_relu_quant */

/* Kernel paths (fgemm_opts.path, and *path_taken of the _ex entries). */
#define FGEMM_PATH_AUTO 0    /* library choice */
#define FGEMM_PATH_TC 1      /* persistent TMA + tcgen05 kernel, grouped-M tile order */
#define FGEMM_PATH_SKINNY 2  /* M <= 128: swap-AB kernel, K split over a cluster, DSMEM reduction */
#define FGEMM_PATH_GENERIC 3 /* CUDA-core tiled kernel: any shape and alignment */
#define FGEMM_PATH_KZERO 4   /* K == 0: epilogue over the zero accumulator, no MMA */
#define FGEMM_PATH_NONE 5    /* M == 0 or N == 0: nothing launched */

/* Per-call options of the _ex entry points.  Zero-initialised fields mean "default". */
typedef struct {
  int group_m;    /* M-tiles per band of the grouped tile order (default 16; 1 = row-major) */
  int path;       /* FGEMM_PATH_*; forcing a path the shape cannot take -> INVALID_VALUE */
  int split_k;    /* skinny path: K splits (1..8, one CTA each in a cluster); 0 = automatic */
  int max_ctas;   /* persistent grid cap (default: one CTA per SM) */
  int timeout_ms; /* bound on every device-side barrier wait (default 1000 ms) */
  int cta_pair;   /* tensor-core path: 0 = automatic, 1 = one CTA per 128 x 256 tile,
                     2 = CTA pairs (2-SM clusters, tcgen05 cta_group::2) on 256 x 256 tiles */
  int tail_split; /* tensor-core path: 0 = cut the tiles of the last partial round of the
                     persistent grid into 128- or 64-column pieces, 1 = keep whole tiles */
  int skinny_tiles; /* skinny path: 128-column tiles per CTA sharing each A block (1 or 2);
                       0 = automatic */
  int stages;     /* skinny path: TMA ring depth 2..8 (capped by shared memory); 0 = default */
  int inject_stall; /* diagnostic for testing the bounded waits: 1 = the first CTA's producer
                       announces its first stage but issues none of its loads, so the MMA's wait
                       on that stage can never complete; it expires after timeout_ms, the kernel
                       drains and exits, and fgemm_device_status reports FGEMM_ERR_TIMEOUT.
                       The output of that call is undefined.  Tensor-core and skinny paths. */
  int bias_init;  /* tensor-core path: start each tile's accumulator at the bias (written into
                     tensor memory before the K loop) instead of adding it after the reduction;
                     same result up to the rounding order ("Optimizing GEMM + Activation on CDNA4
                     with TLX", V4).  0 = automatic (on when K <= 1024), 1 = on, 2 = off.
                     Ignored by the other paths and by the plain GEMM. */
  int full_last_n; /* tensor-core path, diagnostic: 1 = run the last column of tiles at the full
                      256-column width instead of narrowing it to the columns left of N */
  int y_blocks;   /* tensor-core path, gate and residual with 16-bit outputs: how each epilogue
                     warp stages its share of the second M x N operand: 0 = automatic (on CTA
                     pairs 3 when K > 1024, 2 when K <= 256, else 1; on single CTAs 1), 1 = the
                     tile's 32 x 128 block, one work item ahead, 2 = two such blocks, two items
                     ahead (a 3-stage ring on pairs, 2 stages on single CTAs), 3 = one 32 x 64
                     chunk at a time (4 KB; leaves room for two-row ring stages; CTA pairs only,
                     else as 1).  Ignored elsewhere. */
  int k_rows;     /* tensor-core path on CTA pairs: 128-byte K rows (64 16-bit or 128 fp8
                     elements) per stage of the operand ring; 0 = automatic (2, or 1 for the
                     gate and residual with 16-bit outputs), 1 = six stages of 32 KB per SM,
                     2 = three stages of 64 KB.  Ignored elsewhere. */
  int bias_mma;   /* tensor-core path, bias-initialised accumulator: how the bias gets into it.
                     1 = written into tensor memory by the epilogue warps; 2 = set by one extra MMA
                     (a tile of ones times the bias row staged by TMA), where the bias has the
                     16-bit operand type and the kernel has room for the two small tiles (gate and
                     residual with 16-bit outputs on single CTAs, or on CTA pairs with one-row
                     stages), else as 1; 0 = automatic: 2 on single CTAs with K <= 256, else 1 */
  int pdl;        /* tensor-core and skinny paths: launch with programmatic stream serialization:
                     the kernel's set-up (barriers, tensor memory) may run while the previous
                     kernel in the stream is finishing, and the kernel waits for that kernel to
                     complete (griddepcontrol.wait) before it copies or stores any global data, so
                     a dependency between the two stays safe (before the wait it may prefetch its
                     first inputs into L2, which stays coherent with that kernel's writes).
                     0 = automatic (on), 1 = on, 2 = off */
  int raster;     /* tensor-core path: 0 = the grouped order over M ("I3. Fuse a GEMM epilogue and
                     change tile scheduling": bands of group_m M-tiles walking N); 1 = the same
                     order with M and N exchanged (bands of group_m N-tiles walking M), which keeps
                     a band of B instead of A in L2 */
  int epi_warps;  /* tensor-core path: epilogue warps per CTA: 0 = automatic (8), 8, or 16 (single
                     CTAs with the gate or residual's Y staged one block per warp: four warps per
                     TMEM lane quadrant, 64 columns each; else 8) */
} fgemm_opts;

/*
 * out = ReLU(A @ B + bias).  dtype: FGEMM_F16|FGEMM_BF16, optionally | FGEMM_BIAS_F32 and/or
 * | FGEMM_OUT_F32.  Returns an fgemm_status.
 */
int fgemm_bias_relu(const void* A, const void* B, const void* bias, void* out, int64_t M,
                    int64_t N, int64_t K, int dtype, void* stream);

/*
 * X = A @ B + bias; out = X + X * Y (Y: M x N, 16-bit: the operand type, or the FGEMM_Y_* type).
 * With fp8 e4m3 operands the projection A @ B runs on fp8 while Y stays 16-bit ("Optimizing GEMM +
 * Activation on CDNA4 with TLX", "Future Work": FP8 precision); e.g. dtype = FGEMM_E4M3 |
 * FGEMM_BIAS_F32 | FGEMM_OUT_F16 | FGEMM_Y_F16.  A 16-bit output has Y's type (else
 * FGEMM_ERR_UNSUPPORTED_DTYPE); an fp32 output takes any 16-bit Y.  Returns an fgemm_status.
 */
int fgemm_addmm_gate(const void* A, const void* B, const void* bias, const void* Y, void* out,
                     int64_t M, int64_t N, int64_t K, int dtype, void* stream);

/*
 * out = ReLU(A @ B + bias + R), R: M x N, 16-bit (the operand type, or the FGEMM_Y_* type, with
 * the same rules as the gate's Y), added after the K loop and before the activation ("Triton: Fused Matmul + Bias + ReLU (Epilogue Fusion)", "Variants": matmul +
 * residual add).  Same conventions as fgemm_bias_relu.  Returns an fgemm_status.
 */
int fgemm_bias_residual_relu(const void* A, const void* B, const void* bias, const void* R,
                             void* out, int64_t M, int64_t N, int64_t K, int dtype, void* stream);

/*
 * Quantized output: out = e4m3(clamp(scale * ReLU(A @ B + bias), -448, 448)), one byte per element
 * (fp8 e4m3, round to nearest even).  "Triton: Fused Matmul + Bias + ReLU (Epilogue Fusion)",
 * "Variants": matmul + quantized output -- a scale and a clamp applied to the accumulator, then
 * the cast before the store.  dtype = operand type | bias type | FGEMM_OUT_E4M3.  scale must be
 * finite (else FGEMM_ERR_INVALID_VALUE).  The tensor-core path needs N to be a multiple of 16.
 */
int fgemm_bias_relu_quant(const void* A, const void* B, const void* bias, void* out, int64_t M,
                          int64_t N, int64_t K, int dtype, float scale, void* stream);

/* As above, with options (may be NULL) and the path that ran (may be NULL). */
int fgemm_bias_relu_ex(const void* A, const void* B, const void* bias, void* out, int64_t M,
                       int64_t N, int64_t K, int dtype, void* stream, const fgemm_opts* opts,
                       int* path_taken);
int fgemm_addmm_gate_ex(const void* A, const void* B, const void* bias, const void* Y, void* out,
                        int64_t M, int64_t N, int64_t K, int dtype, void* stream,
                        const fgemm_opts* opts, int* path_taken);
int fgemm_bias_residual_relu_ex(const void* A, const void* B, const void* bias, const void* R,
                                void* out, int64_t M, int64_t N, int64_t K, int dtype,
                                void* stream, const fgemm_opts* opts, int* path_taken);
int fgemm_bias_relu_quant_ex(const void* A, const void* B, const void* bias, void* out, int64_t M,
                             int64_t N, int64_t K, int dtype, float scale, void* stream,
                             const fgemm_opts* opts, int* path_taken);

/*
 * Unfused comparison chain (for measuring the traffic that fusion removes; not a fast path).
 * "Triton: Fused Matmul + Bias + ReLU (Epilogue Fusion)", "The HBM traffic - the whole point":
 * the GEMM writes an intermediate I, a bias kernel reads and rewrites I, a ReLU kernel reads I
 * and writes out (three launches).  "Optimizing GEMM + Activation on CDNA4 with TLX", "The GLU
 * Block": the GEMM writes I, one gate kernel reads I and Y and writes out (two launches).
 * I lives in the caller's `workspace` (device memory of at least
 * fgemm_unfused_workspace_bytes() bytes, 256-byte aligned).  inter_f32 = 1 keeps I in fp32, else
 * I has the output type.
 */
size_t fgemm_unfused_workspace_bytes(int64_t M, int64_t N, int dtype, int inter_f32);
int fgemm_unfused_bias_relu(const void* A, const void* B, const void* bias, void* out, int64_t M,
                            int64_t N, int64_t K, int dtype, void* workspace,
                            size_t workspace_bytes, int inter_f32, void* stream);
int fgemm_unfused_addmm_gate(const void* A, const void* B, const void* bias, const void* Y,
                             void* out, int64_t M, int64_t N, int64_t K, int dtype,
                             void* workspace, size_t workspace_bytes, int inter_f32,
                             void* stream);

/*
 * fgemm_unfused_bias_relu_noalloc -- the unfused bias + ReLU chain with no allocation at all.
 * (The pages have no counterpart: this entry exists only for callers of this library.)
 *
 * For callers that must not allocate device memory: for example code that runs inside a host
 * application which reserves the device's whole memory budget up front and hands out no more,
 * or a serving loop that forbids cudaMalloc / cudaFree after start-up because they can fail
 * there, or synchronise the device and stall other streams.  Instead of a caller-provided
 * workspace, the intermediate lives in a fixed array of FGEMM_NOALLOC_SCRATCH_BYTES bytes that
 * the library reserves in device memory; every device that loads the library holds it until the
 * process exits.  This call allocates nothing, and calls no allocating library routine.
 *
 * Arguments, layout, ownership and the result are those of fgemm_unfused_bias_relu minus the
 * workspace.  Limit: fgemm_unfused_workspace_bytes(M, N, dtype, inter_f32) must not exceed
 * FGEMM_NOALLOC_SCRATCH_BYTES, else FGEMM_ERR_WORKSPACE is returned and nothing runs.
 * The first call on each device (with that device current) looks up the array's device address
 * and keeps it; make that first call before any stream capture.  If the lookup fails the call
 * returns FGEMM_ERR_NO_DEVICE and the next call on that device tries it again.  All calls share the array and it keeps
 * the previous call's contents (nothing in it needs to start at zero: each call writes every
 * intermediate element before reading it); calls whose work overlaps on the GPU race on it.
 */
#define FGEMM_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
int fgemm_unfused_bias_relu_noalloc(const void* A, const void* B, const void* bias, void* out,
                                    int64_t M, int64_t N, int64_t K, int dtype, int inter_f32,
                                    void* stream);

/*
 * Synchronise `stream`, then read and clear the current device's error word.  *code receives 0
 * or the first in-kernel failure since the last call (an fgemm_status in the low byte, the
 * failing wait's site in the next byte).  Returns FGEMM_OK, or FGEMM_ERR_LAUNCH if the stream
 * reported a CUDA error.
 */
int fgemm_device_status(void* stream, int* code);

/* Human-readable name of an fgemm_status. */
const char* fgemm_status_string(int status);

/*
 * Launch plan of a fused call, computed without launching anything: the path, grid and cluster
 * shape, the tile count and how the persistent grid's last round is cut.  Same arguments and
 * validation as the _ex entry of `epilogue` (FGEMM_EPI_*; Y is the gate's Y or the residual R);
 * the buffers are inspected for alignment only.
 */
typedef struct {
  int path;           /* FGEMM_PATH_* that would run */
  int grid;           /* CTAs launched */
  int cluster;        /* CTAs per cluster: 2 for CTA pairs, the K split on the skinny path */
  int tiles;          /* output tiles (tensor-core and skinny paths) */
  int work_items;     /* persistent work items, after cutting the last round into pieces */
  int tail_split;     /* pieces per tile of the last round (1 = whole tiles); on the skinny
                         path: 128-column tiles per CTA */
  int resident_pairs; /* CTA pairs resident at once (pair mode; 0 otherwise) */
  int last_tile_n;    /* tensor-core path: MMA width of the last column of tiles (the columns left
                         of N rounded up to what one CTA or pair stages and stores; 256 when N is a
                         multiple of 256); 0 on other paths */
  int y_blocks;       /* tensor-core path: staging of the second operand (see fgemm_opts) */
  int k_rows;         /* tensor-core path: 128-byte K rows per ring stage (see fgemm_opts) */
  int row_barriers;   /* tensor-core path, two K rows per stage: 1 = each K row of a stage lands on
                         its own full barrier (fp8 operands and staged second operands) */
  int bias_init;      /* tensor-core path: 0 = the bias is added after the reduction; 1 = the
                         accumulator starts at the bias, written by the epilogue warps; 2 = set by
                         the extra MMA (see fgemm_opts.bias_mma) */
  int epi_warps;      /* tensor-core path: epilogue warps per CTA (see fgemm_opts.epi_warps) */
} fgemm_plan_info;
int fgemm_plan(const void* A, const void* B, const void* bias, const void* Y, const void* out,
               int64_t M, int64_t N, int64_t K, int dtype, int epilogue, const fgemm_opts* opts,
               fgemm_plan_info* info);
/*
 * The same plan for a device described by its SM count and the number of CTA pairs of the
 * tensor-core kernel that can be resident on it at once, computed on the host alone (no GPU is
 * needed or touched; the buffers are inspected for alignment only).  num_sms >= 1 and
 * resident_pairs >= 0 (0: no limit below num_sms / 2), else FGEMM_ERR_INVALID_VALUE.
 */
int fgemm_plan_on(const void* A, const void* B, const void* bias, const void* Y, const void* out,
                  int64_t M, int64_t N, int64_t K, int dtype, int epilogue, const fgemm_opts* opts,
                  int num_sms, int resident_pairs, fgemm_plan_info* info);

/*
 * The persistent kernels' tile order, exposed for host-side tests: linear tile t of a
 * tiles_m x tiles_n grid with `group` M-tiles per band ("I3. Fuse a GEMM epilogue and change tile
 * scheduling", "Tiles and grouped ownership").  Returns FGEMM_ERR_INVALID_VALUE when t is out of
 * range or a count is not positive.
 */
int fgemm_tile_of(int64_t t, int64_t tiles_m, int64_t tiles_n, int group, int64_t* m_tile,
                  int64_t* n_tile);

#ifdef __cplusplus
}
#endif

#endif /* FGEMM_H */
