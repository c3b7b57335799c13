// skinny.cu -- fused GEMM + epilogue for small M (decode-like: a few to 128 rows), sm_103a.
//
// With M <= 128 the square-tile kernel has too few tiles to keep the GPU busy and the time is
// the stream of B (K x N) from HBM.  This kernel therefore
//   * swaps the operands: out^T (N x M) = B^T A^T, so the 128-row MMA dimension runs over N (128
//     output columns per MMA) and the MMA's N is M rounded up to 16 (rows >= M are zero-filled
//     by TMA); B is read N-major exactly as it lies in memory, A K-major;
//   * gives each CTA `nt` adjacent 128-column tiles (one TMEM accumulator each) that share every
//     staged A block, so A is re-read from L2 once per 128 * nt columns instead of once per 128;
//   * splits K over the S CTAs of a thread-block cluster, each CTA streaming its K range of B
//     through a TMA ring into tcgen05.mma (fp32 in TMEM);
//   * reduces the S partial accumulators through distributed shared memory: rows
//     [r*W/S, (r+1)*W/S) of the CTA's W = 128 * nt columns belong to CTA r; every CTA pushes its
//     partial rows from TMEM straight into the owner's shared memory (remote stores laid out so
//     that each warp store is one contiguous run; its own rows with local stores), and after a
//     cluster barrier each owner sums its rows locally; four epilogue warps, or eight (two per
//     TMEM lane quadrant) when M is padded to 64 or more;
//   * applies the epilogue once, on the complete sum ("Epilogue concept", "Why it cannot move
//     earlier": ReLU of a partial sum is not ReLU of the sum, and a bias added per partial would be
//     added S times): x = sum + bias[n], then ReLU or the gate, one rounding, coalesced store.
// No workspace in global memory: the reduction stays on chip.
#include <atomic>

#include "kernels.h"
#include "ptx.cuh"

namespace fgemm {
namespace sk {

constexpr int BN = 128;  // output columns per MMA (MMA M)
constexpr int BK = 64;
constexpr int MAX_STAGES = 8;
// Epilogue warps: one per TMEM lane quadrant (warp w reads lanes 32 (w % 4) ..), or two that split
// the accumulator's 16-column chunks between them when the reduction and the final epilogue
// carry enough work for the extra warps to pay (M padded to 64 or more); the launch picks the
// block size and the kernel reads it back from blockDim.
constexpr int MAX_EPI_WARPS = 8;
constexpr int MAX_THREADS = 64 + 32 * MAX_EPI_WARPS;
__host__ __device__ inline int epi_warps_for(int mpad) { return mpad >= 64 ? 8 : 4; }
constexpr uint32_t B_BOX_BYTES = 64 * 64 * 2;         // 64 K-rows x 64 N-columns
constexpr uint32_t B_TILE_BYTES = 2 * B_BOX_BYTES;    // 64 x 128: one MMA's worth of B
constexpr int MAX_MPAD = 128;
// Area after the data: mbarriers, the TMEM address slot (byte 192), the abort flag (byte 200) and
// the bias of the rows the CTA owns (at most 256 floats, from byte 256).
constexpr uint32_t OFF_TMEM_SLOT = 192, OFF_ABORT = 200, OFF_BIAS = 256;
constexpr uint32_t BAR_BYTES = OFF_BIAS + 4 * 256;
constexpr uint32_t STAGE_AREA_MAX = 196608;           // bytes of stage ring at most

enum { SITE_PROD_EMPTY = 16, SITE_MMA_FULL, SITE_EPI_ACC_FULL, SITE_DRAIN };

__host__ __device__ inline uint32_t stage_bytes(int mpad, int nt) {
  return static_cast<uint32_t>(nt) * B_TILE_BYTES + static_cast<uint32_t>(mpad) * 128u;
}
// Ring depth: `want` stages (0 = as many as fit, at most 6), capped by the stage area.
__host__ __device__ inline int num_stages(int mpad, int nt, int want) {
  int s = static_cast<int>(STAGE_AREA_MAX / stage_bytes(mpad, nt));
  if (s > MAX_STAGES) s = MAX_STAGES;
  const int cap = want > 0 ? want : 6;
  return s > cap ? cap : s;
}
// Receive area of the cluster reduction, overlaid on the stage ring.
// Layout recv[src][m][row], rows of an owner's slice fastest, `pitch` floats per m: a warp's store
// of one m for its 32 consecutive rows is one contiguous 128-byte run, which the cluster store
// path moves far faster than 32 scattered 16-byte pieces.
__host__ __device__ inline int recv_pitch(int nt, int split) {
  const int maxslice = (BN * nt + split - 1) / split;
  return (maxslice + 3) & ~3;
}
__host__ __device__ inline uint32_t recv_bytes(int mpad, int nt, int split) {
  return static_cast<uint32_t>(split * mpad * recv_pitch(nt, split)) * 4u;
}
// Shared memory before the barriers: the larger of the ring and the reduction's receive area.
__host__ __device__ inline uint32_t data_bytes(int mpad, int nt, int split, int want) {
  const uint32_t ring = static_cast<uint32_t>(num_stages(mpad, nt, want)) * stage_bytes(mpad, nt);
  const uint32_t recv = recv_bytes(mpad, nt, split);
  return ((ring > recv ? ring : recv) + 1023u) & ~1023u;
}
__host__ inline uint32_t smem_bytes(int mpad, int nt, int split, int want) {
  return data_bytes(mpad, nt, split, want) + BAR_BYTES + 1024;
}

__device__ __forceinline__ float ld_any(const void* p, int64_t i, int type) {
  switch (type) {
    case ELEM_F16: return __half2float(static_cast<const __half*>(p)[i]);
    case ELEM_BF16: return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
    default: return static_cast<const float*>(p)[i];
  }
}
__device__ __forceinline__ void st_any(void* p, int64_t i, int type, float v) {
  switch (type) {
    case ELEM_E4M3:
      static_cast<uint8_t*>(p)[i] =
          static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
      break;
    case ELEM_F16: static_cast<__half*>(p)[i] = __float2half_rn(v); break;
    case ELEM_BF16: static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v); break;
    default: static_cast<float*>(p)[i] = v; break;
  }
}

// F8: fp8 e4m3 operands (tcgen05 kind::f8f6f4, 32 K per MMA): one 128-byte K row of a stage is
// 128 K elements, and B arrives as one 128 K-row x 128 N-column box per tile (the same bytes as
// the two 64 x 64 boxes of 16-bit operands), so half the HBM bytes of B per output column.
template <int EPI, bool F8 = false>
__global__ void __launch_bounds__(MAX_THREADS, 1)
    skinny_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmA,
                  const SkParams p) {
  constexpr int KBLK = F8 ? 2 * BK : BK;  // K elements per stage (one 128-byte row of A)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int nt = p.nt;
  const int stages = num_stages(p.mpad, nt, p.stages);
  const uint32_t sbytes = stage_bytes(p.mpad, nt);
  const uint32_t dbytes = data_bytes(p.mpad, nt, p.split, p.stages);
  const uint32_t bar0 = sbase + dbytes;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  // barriers: full[0..7], empty[8..15], acc_full 16, mma_done 17
  constexpr int BAR_FULL = 0, BAR_EMPTY = MAX_STAGES, BAR_ACC_FULL = 2 * MAX_STAGES,
                BAR_MMA_DONE = 2 * MAX_STAGES + 1;
  static_assert(8 * (2 * MAX_STAGES + 2) <= OFF_TMEM_SLOT, "barrier area");
  uint8_t* bar_area = smem + dbytes;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + OFF_TMEM_SLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_area + OFF_ABORT);
  float* bias_s = reinterpret_cast<float*>(bar_area + OFF_BIAS);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int epi_threads = static_cast<int>(blockDim.x) - 64;
  const uint32_t S = static_cast<uint32_t>(p.split);
  const uint32_t rank = (S > 1) ? cluster_ctarank() : 0u;
  const int W = BN * nt;  // output columns of this CTA
  const int n0 = static_cast<int>(blockIdx.x / S) * W;
  const int KB = (p.K + KBLK - 1) / KBLK;
  const int kb0 = static_cast<int>(static_cast<int64_t>(KB) * rank / S);
  const int kb1 = static_cast<int>(static_cast<int64_t>(KB) * (rank + 1) / S);
  const int nkb = kb1 - kb0;
  const uint64_t tmo = p.timeout_ns;
  const int pitch = recv_pitch(nt, static_cast<int>(S));
  auto first_row = [&](uint32_t r) { return static_cast<int>(static_cast<uint32_t>(W) * r / S); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bar(BAR_FULL + s), 1);
      mbar_init(bar(BAR_EMPTY + s), 1);
    }
    mbar_init(bar(BAR_ACC_FULL), 1);
    mbar_init(bar(BAR_MMA_DONE), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmA);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), static_cast<uint32_t>(p.tmem_cols));
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Global memory is read only after the previous kernel in the stream has completed (with
  // programmatic dependent launch the set-up above overlaps it).  Before that, the first ring
  // stages' B and A are prefetched into L2, which stays coherent with whatever that kernel still
  // writes.  Measured on one GB300 (graph replay, alternating builds): N = K = 8192, M = 1 / 64 /
  // 128 24.4 -> 23.6, 26.3 -> 25.3, 29.3 -> 28.4 us; fp8 M = 1 / 128 15.0 -> 14.9, 19.8 -> 19.1 us.
  // Letting the next kernel launch at the start of this one as well measured mixed (M = 1
  // 25.8 us, M = 64 24.9 us), so the trigger stays at the teardown.
  if (p.pdl && warp == 0 && lane == 0) {
    const int pk1 = kb0 + stages < kb1 ? kb0 + stages : kb1;
    for (int kb = kb0; kb < pk1; ++kb) {
      if constexpr (F8) {
        for (int c = 0; c < nt; ++c) tma_prefetch_2d(&tmB, n0 + BN * c, kb * KBLK);
      } else {
        for (int c = 0; c < 2 * nt; ++c) tma_prefetch_2d(&tmB, n0 + 64 * c, kb * KBLK);
      }
      tma_prefetch_2d(&tmA, kb * KBLK, 0);
    }
  }
  grid_dependency_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_b = policy_evict_first();   // B is streamed once
      const uint64_t pol_a = policy_evict_last();    // A is re-read by every group of N tiles
      uint32_t stage = 0, phase = 0, issued = 0, issued_parity = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(bar(BAR_EMPTY + stage), phase ^ 1u, abort_flag, tmo, p.err, SITE_PROD_EMPTY))
          break;
        const uint32_t fb = bar(BAR_FULL + stage);
        mbar_arrive_expect_tx(fb, sbytes);
        const uint32_t dst = sbase + stage * sbytes;
        // diagnostic stall: announce the stage's bytes but never load them
        if (p.inject_stall && blockIdx.x == 0 && kb == kb0) {
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == static_cast<uint32_t>(stages)) {
            stage = 0;
            phase ^= 1u;
          }
          continue;
        }
        if constexpr (F8) {
          for (int c = 0; c < nt; ++c)  // one 128 x 128 fp8 box per tile
            tma_load_2d(dst + c * B_TILE_BYTES, &tmB, fb, n0 + BN * c, kb * KBLK, pol_b);
        } else {
          for (int c = 0; c < 2 * nt; ++c)
            tma_load_2d(dst + c * B_BOX_BYTES, &tmB, fb, n0 + 64 * c, kb * KBLK, pol_b);
        }
        tma_load_2d(dst + static_cast<uint32_t>(nt) * B_TILE_BYTES, &tmA, fb, kb * KBLK, 0, pol_a);
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == static_cast<uint32_t>(stages)) {
          stage = 0;
          phase ^= 1u;
        }
      }
      volatile int never = 0;
      for (int s = 0; s < stages; ++s)
        if ((issued >> s) & 1u)
          mbar_wait(bar(BAR_FULL + s), (issued_parity >> s) & 1u, &never, tmo, p.err, SITE_DRAIN);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(bar(BAR_FULL + stage), phase, abort_flag, tmo, p.err, SITE_MMA_FULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t b_addr = sbase + stage * sbytes;                            // B^T, N-major
        const uint32_t a_addr = b_addr + static_cast<uint32_t>(nt) * B_TILE_BYTES;  // A^T, K-major
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // 32 bytes of K per MMA: 16 16-bit or 32 fp8 elements
          const uint64_t db = sdesc_sw128(a_addr + 32u * k, 16u, 1024u);
          for (int t = 0; t < nt; ++t) {
            // B^T (MN-major): 16 (32 fp8) K rows of 128 bytes per MMA; 64-column boxes for
            // 16-bit operands, one 128-column box for fp8
            const uint64_t da = sdesc_sw128(b_addr + t * B_TILE_BYTES + (F8 ? 4096u : 2048u) * k,
                                            F8 ? B_TILE_BYTES : B_BOX_BYTES, 1024u);
            const uint32_t acc = (kb > kb0 || k > 0) ? 1u : 0u;
            if constexpr (F8)
              umma_f8_cg<1>(tmem_base + static_cast<uint32_t>(t * p.mpad), da, db, p.idesc, acc);
            else
              umma_f16(tmem_base + static_cast<uint32_t>(t * p.mpad), da, db, p.idesc, acc);
          }
        }
        umma_commit(bar(BAR_EMPTY + stage));
        if (++stage == static_cast<uint32_t>(stages)) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok && nkb > 0) umma_commit(bar(BAR_ACC_FULL));
      umma_commit(bar(BAR_MMA_DONE));
      volatile int never = 0;
      mbar_wait(bar(BAR_MMA_DONE), 0, &never, tmo, p.err, SITE_DRAIN);
    }
  } else if constexpr (EPI != EPI_NONE) {
    // Epilogue warps, while the main loop runs: the bias of the rows this CTA owns, so that the
    // final epilogue reads it from shared memory (a global load there, after stores to out that
    // may alias it, would go to L2 on every pass).
    const int r0 = first_row(rank), nrows = first_row(rank + 1) - r0;
    for (int i = static_cast<int>(threadIdx.x) - 64; i < nrows; i += epi_threads) {
      const int n = n0 + r0 + i;
      bias_s[i] = n < p.N ? ld_any(p.bias, n, p.bias_type) : 0.0f;
    }
  }

  // ------------------------------------------------------------ reduction across the cluster
  // Row n (0 <= n < W) of the CTA's columns is owned by CTA owner(n), the r with
  // W r / S <= n < W (r + 1) / S.  Each CTA pushes its partial row n into the owner's receive area
  // recv[src][m][n - first_row(owner)] (see recv_pitch), which overlays the owner's stage ring
  // (or extends past it); so the first cluster barrier makes sure every CTA has finished its main
  // loop before any push, and the second one that every push has landed before the owners read.
  // With S = 1 only this CTA writes its ring, after its accumulator is complete (every load landed,
  // every MMA done), and the epilogue warps synchronise among themselves (named barrier 1).  No
  // CTA-wide barrier is used here: the producer and MMA issuer run in single lanes, and a CTA
  // barrier reached by the other lanes of their warps was measured to complete while those lanes
  // were still in their loops.
  __syncwarp();
  if (S > 1) cluster_sync();

  if (warp >= 2) {
    const int q = warp & 3;
    const int half = (warp - 2) / 4, halves = epi_threads / 128;
    const bool have = (nkb > 0) && mbar_wait(bar(BAR_ACC_FULL), 0, abort_flag, tmo, p.err,
                                             SITE_EPI_ACC_FULL);
    tc_fence_after();
    for (int t = 0; t < nt; ++t) {
      const int row = t * BN + 32 * q + lane;
      uint32_t owner = (static_cast<uint32_t>(row) * S) / static_cast<uint32_t>(W);
      while (owner + 1 < S && first_row(owner + 1) <= row) ++owner;
      while (owner > 0 && first_row(owner) > row) --owner;
      const uint32_t slot = sbase + 4u * static_cast<uint32_t>(static_cast<int>(rank) * p.mpad * pitch +
                                                             row - first_row(owner));
      const bool remote = owner != rank;  // own rows take the local store path
      const uint32_t dst = remote ? map_shared_rank(slot, owner) : slot;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                             static_cast<uint32_t>(t * p.mpad);
      for (int c = half; c < p.mpad / 16; c += halves) {
        uint32_t v[16];
        if (have) {
          __syncwarp();
          tmem_ld16(taddr + 16u * c, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = 0u;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {  // m = 16 c + j; the warp's lanes write consecutive rows
          const uint32_t a = dst + 4u * static_cast<uint32_t>((16 * c + j) * pitch);
          if (remote)
            st_shared_cluster_f32(a, __uint_as_float(v[j]));
          else
            st_shared_f32(a, __uint_as_float(v[j]));
        }
      }
    }
    tc_fence_before();
  }

  __syncwarp();
  if (S > 1)
    cluster_sync();
  else if (warp >= 2)
    named_bar_sync(1, static_cast<uint32_t>(epi_threads));

  // ------------------------------------------------------------ epilogue on the full sums
  // Lane l of every epilogue warp takes owned rows l, l + 32, ..; the warps take the groups of 4
  // rows of out in turn.  Each thread sums the S partials of its element in source order and
  // applies the epilogue once.
  if (warp >= 2) {
    const int r0 = first_row(rank), nrows = first_row(rank + 1) - r0;
    const int m4 = (p.M + 3) / 4;
    const int ew = epi_threads / 32, wi = warp - 2;
    const float* recv = reinterpret_cast<const float*>(smem);
    for (int nl = lane; nl < nrows; nl += 32) {
      const int n = n0 + r0 + nl;
      if (n >= p.N) break;
      float b = 0.f;
      if constexpr (EPI != EPI_NONE) b = bias_s[nl];  // once, on the full sum
      for (int g = wi; g < m4; g += ew) {
        const int m = 4 * g;
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
        for (uint32_t src = 0; src < S; ++src) {
          const float* col = recv + (static_cast<int>(src) * p.mpad + m) * pitch + nl;
#pragma unroll
          for (int e = 0; e < 4; ++e) s4[e] += col[e * pitch];
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (m + e >= p.M) break;
          const int64_t o = static_cast<int64_t>(m + e) * p.N + n;
          float v = s4[e] + b;
          if constexpr (EPI == EPI_RELU) v = fmaxf(v, 0.0f);
          if constexpr (EPI == EPI_QUANT) v = fminf(fmaxf(fmaxf(v, 0.0f) * p.out_scale, -448.0f), 448.0f);
          if constexpr (EPI == EPI_GATE) v = fmaf(v, ld_any(p.Y, o, p.y_type), v);
          if constexpr (EPI == EPI_RESID) v = fmaxf(v + ld_any(p.Y, o, p.y_type), 0.0f);
          st_any(p.out, o, p.out_type, v);
        }
      }
    }
  }

  grid_dependents_launch();  // the next kernel in the stream may begin its set-up
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, static_cast<uint32_t>(p.tmem_cols));
  }
}

template <int EPI, bool F8>
cudaError_t launch_one(const CUtensorMap& tb, const CUtensorMap& ta, const SkParams& p, int ctas,
                       cudaStream_t s) {
  auto k = skinny_kernel<EPI, F8>;
  const uint32_t smem = smem_bytes(p.mpad, p.nt, p.split, p.stages);
  // Per device: the shared-memory opt-in is set once.  Host threads may race on a first call;
  // setting the attribute twice is harmless, and the flag is atomic.
  static std::atomic<bool> opted_in[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!opted_in[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    opted_in[dev].store(true, std::memory_order_release);
  }
  if (smem > 232448) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(static_cast<unsigned>(64 + 32 * epi_warps_for(p.mpad)));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.split);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k, tb, ta, p);
}

}  // namespace sk

int skinny_block_n() { return sk::BN; }
int skinny_max_m() { return sk::MAX_MPAD; }
bool skinny_fits(int mpad, int nt, int split, int stages) {
  return sk::num_stages(mpad, nt, stages) >= 2 && sk::smem_bytes(mpad, nt, split, stages) <= 232448;
}
uint32_t skinny_smem_bytes(int mpad, int nt, int split, int stages) {
  return sk::smem_bytes(mpad, nt, split, stages);
}

cudaError_t launch_skinny(int epi, const CUtensorMap& tmB, const CUtensorMap& tmA, const SkParams& p,
                          int ctas, cudaStream_t s) {
  if (p.ab_type == ELEM_E4M3) {
    switch (epi) {
      case EPI_RELU: return sk::launch_one<EPI_RELU, true>(tmB, tmA, p, ctas, s);
      case EPI_GATE: return sk::launch_one<EPI_GATE, true>(tmB, tmA, p, ctas, s);
      case EPI_RESID: return sk::launch_one<EPI_RESID, true>(tmB, tmA, p, ctas, s);
      case EPI_QUANT: return sk::launch_one<EPI_QUANT, true>(tmB, tmA, p, ctas, s);
      default: return cudaErrorNotSupported;
    }
  }
  switch (epi) {
    case EPI_RELU: return sk::launch_one<EPI_RELU, false>(tmB, tmA, p, ctas, s);
    case EPI_GATE: return sk::launch_one<EPI_GATE, false>(tmB, tmA, p, ctas, s);
    case EPI_RESID: return sk::launch_one<EPI_RESID, false>(tmB, tmA, p, ctas, s);
    case EPI_QUANT: return sk::launch_one<EPI_QUANT, false>(tmB, tmA, p, ctas, s);
    default: return sk::launch_one<EPI_NONE, false>(tmB, tmA, p, ctas, s);
  }
}

}  // namespace fgemm
