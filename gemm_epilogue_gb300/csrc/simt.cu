// simt.cu -- CUDA-core kernels: the generic fused GEMM (any shape, any alignment), the K = 0
// epilogue, and the elementwise passes of the unfused comparison chain.
#include "kernels.h"
#include "ptx.cuh"

namespace fgemm {

__device__ __forceinline__ float ld_elem(const void* p, int64_t i, int type) {
  switch (type) {
    case ELEM_E4M3: {
      const __half_raw h =
          __nv_cvt_fp8_to_halfraw(static_cast<const __nv_fp8_storage_t*>(p)[i], __NV_E4M3);
      return __half2float(__half(h));
    }
    case ELEM_F16: return __half2float(static_cast<const __half*>(p)[i]);
    case ELEM_BF16: return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
    default: return static_cast<const float*>(p)[i];
  }
}

__device__ __forceinline__ void st_elem(void* p, int64_t i, int type, float v) {
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

// The epilogue on one element: x = acc + bias, then ReLU, the gate, the residual add + ReLU, or
// ReLU + scale + clamp to the fp8 range (the cast happens at the store).  fp32 throughout.
template <int EPI>
__device__ __forceinline__ float epilogue(float acc, float bias, float y, float scale = 1.0f) {
  if constexpr (EPI == EPI_NONE) return acc;
  const float x = acc + bias;
  if constexpr (EPI == EPI_QUANT) return fminf(fmaxf(fmaxf(x, 0.0f) * scale, -448.0f), 448.0f);
  if constexpr (EPI == EPI_RELU) return fmaxf(x, 0.0f);
  if constexpr (EPI == EPI_RESID) return fmaxf(x + y, 0.0f);  // residual before the activation
  return fmaf(x, y, x);  // X + X * Y
}

// ---------------------------------------------------------------------------------------------
// Generic fused GEMM: 64 x 64 output tile per 256-thread block, 4 x 4 outputs per thread,
// K staged through shared memory 16 at a time.  Every global load is masked against M, N and K
// separately and the store against M and N ("I3. Fuse a GEMM epilogue and change tile
// scheduling", "Tiles and grouped ownership").  fp32 accumulate; epilogue after the K loop.
namespace gen {
constexpr int TM = 64, TN = 64, TK = 16, THREADS = 256;
}

template <int EPI>
__global__ void __launch_bounds__(gen::THREADS) generic_kernel(const SimtParams p) {
  using namespace gen;
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int tiles_n = (p.N + TN - 1) / TN;
  const int64_t tile = blockIdx.x;
  const int m0 = static_cast<int>(tile / tiles_n) * TM;
  const int n0 = static_cast<int>(tile % tiles_n) * TN;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < p.K; k0 += TK) {
    for (int e = threadIdx.x; e < TM * TK; e += THREADS) {
      const int r = e / TK, kk = e % TK;
      const int gm = m0 + r, gk = k0 + kk;
      As[kk][r] = (gm < p.M && gk < p.K) ? ld_elem(p.A, static_cast<int64_t>(gm) * p.K + gk, p.ab_type) : 0.f;
    }
    for (int e = threadIdx.x; e < TK * TN; e += THREADS) {
      const int kk = e / TN, c = e % TN;
      const int gk = k0 + kk, gn = n0 + c;
      Bs[kk][c] = (gk < p.K && gn < p.N) ? ld_elem(p.B, static_cast<int64_t>(gk) * p.N + gn, p.ab_type) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }

  // Epilogue: the bias is read here, after the K loop, masked by column.
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int gn = n0 + tx * 4 + j;
    if (gn >= p.N) continue;
    const float bj = (EPI == EPI_NONE) ? 0.f : ld_elem(p.bias, gn, p.bias_type);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int gm = m0 + ty * 4 + i;
      if (gm >= p.M) continue;
      const int64_t idx = static_cast<int64_t>(gm) * p.N + gn;
      const float y = (EPI == EPI_GATE || EPI == EPI_RESID) ? ld_elem(p.Y, idx, p.y_type) : 0.f;
      st_elem(p.out, idx, p.out_type, epilogue<EPI>(acc[i][j], bj, y, p.out_scale));
    }
  }
}

cudaError_t launch_generic(int epi, const SimtParams& p, cudaStream_t s) {
  const int64_t tiles = static_cast<int64_t>((p.M + gen::TM - 1) / gen::TM) * ((p.N + gen::TN - 1) / gen::TN);
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(tiles));
  switch (epi) {
    case EPI_RELU: generic_kernel<EPI_RELU><<<grid, gen::THREADS, 0, s>>>(p); break;
    case EPI_GATE: generic_kernel<EPI_GATE><<<grid, gen::THREADS, 0, s>>>(p); break;
    case EPI_RESID: generic_kernel<EPI_RESID><<<grid, gen::THREADS, 0, s>>>(p); break;
    case EPI_QUANT: generic_kernel<EPI_QUANT><<<grid, gen::THREADS, 0, s>>>(p); break;
    default: generic_kernel<EPI_NONE><<<grid, gen::THREADS, 0, s>>>(p); break;
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
// Elementwise kernels.  Each thread handles groups of 8 consecutive elements of a row when the
// row length is a multiple of 8 and every pointer is 16-byte aligned (one or two 16-byte vector
// accesses per operand), otherwise single elements.  Grid-stride loops over the M x N elements.

struct Vec8 {
  float v[8];
};

__device__ __forceinline__ Vec8 ld8(const void* p, int64_t i, int type) {
  Vec8 r;
  if (type == ELEM_F32) {
    const float4* q = reinterpret_cast<const float4*>(static_cast<const float*>(p) + i);
    const float4 a = q[0], b = q[1];
    r.v[0] = a.x; r.v[1] = a.y; r.v[2] = a.z; r.v[3] = a.w;
    r.v[4] = b.x; r.v[5] = b.y; r.v[6] = b.z; r.v[7] = b.w;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p) + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = unpack2(w[k], type == ELEM_BF16);
      r.v[2 * k] = f.x;
      r.v[2 * k + 1] = f.y;
    }
  }
  return r;
}

__device__ __forceinline__ void st8(void* p, int64_t i, int type, const Vec8& x) {
  if (type == ELEM_E4M3) {
    uint2 u;
    u.x = pack2_e4m3(x.v[0], x.v[1]) | (pack2_e4m3(x.v[2], x.v[3]) << 16);
    u.y = pack2_e4m3(x.v[4], x.v[5]) | (pack2_e4m3(x.v[6], x.v[7]) << 16);
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p) + i) = u;
  } else if (type == ELEM_F32) {
    float4* q = reinterpret_cast<float4*>(static_cast<float*>(p) + i);
    q[0] = make_float4(x.v[0], x.v[1], x.v[2], x.v[3]);
    q[1] = make_float4(x.v[4], x.v[5], x.v[6], x.v[7]);
  } else {
    const bool bf = type == ELEM_BF16;
    uint4 u;
    u.x = pack2(x.v[0], x.v[1], bf);
    u.y = pack2(x.v[2], x.v[3], bf);
    u.z = pack2(x.v[4], x.v[5], bf);
    u.w = pack2(x.v[6], x.v[7], bf);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p) + i) = u;
  }
}

enum EwOp { EW_BIAS_INPLACE = 0, EW_RELU = 1, EW_BIAS_GATE = 2, EW_KZERO_RELU = 3, EW_KZERO_GATE = 4,
            EW_KZERO_RESID = 5, EW_KZERO_QUANT = 6 };

struct EwParams {
  float scale;       // quantized K = 0 epilogue only
  const void* src;   // I (the intermediate) or NULL for K = 0
  int src_type;
  const void* bias;
  int bias_type;
  const void* Y;
  int y_type;
  void* dst;         // I for the in-place bias pass, else out
  int dst_type;
  int M, N;
};

template <int OP>
__device__ __forceinline__ float ew_apply(float s, float b, float y, float scale) {
  if constexpr (OP == EW_KZERO_QUANT)
    return fminf(fmaxf(fmaxf(0.0f + b, 0.0f) * scale, -448.0f), 448.0f);
  if constexpr (OP == EW_BIAS_INPLACE) return s + b;
  if constexpr (OP == EW_RELU) return fmaxf(s, 0.0f);
  if constexpr (OP == EW_BIAS_GATE) {
    const float x = s + b;
    return fmaf(x, y, x);
  }
  if constexpr (OP == EW_KZERO_RELU) return fmaxf(0.0f + b, 0.0f);
  if constexpr (OP == EW_KZERO_RESID) return fmaxf((0.0f + b) + y, 0.0f);
  const float x = 0.0f + b;  // EW_KZERO_GATE
  return fmaf(x, y, x);
}

template <int OP, bool VEC>
__global__ void __launch_bounds__(256) ew_kernel(const EwParams p) {
  constexpr bool uses_src = (OP == EW_BIAS_INPLACE || OP == EW_RELU || OP == EW_BIAS_GATE);
  constexpr bool uses_bias = (OP != EW_RELU);
  constexpr bool uses_y = (OP == EW_BIAS_GATE || OP == EW_KZERO_GATE || OP == EW_KZERO_RESID);
  const int64_t total = static_cast<int64_t>(p.M) * p.N;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  if constexpr (VEC) {
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g * 8 < total; g += stride) {
      const int64_t i = g * 8;
      const int col = static_cast<int>(i % p.N);
      Vec8 s{}, b{}, y{}, o;
      if constexpr (uses_src) s = ld8(p.src, i, p.src_type);
      if constexpr (uses_bias) b = ld8(p.bias, col, p.bias_type);
      if constexpr (uses_y) y = ld8(p.Y, i, p.y_type);
#pragma unroll
      for (int e = 0; e < 8; ++e) o.v[e] = ew_apply<OP>(s.v[e], b.v[e], y.v[e], p.scale);
      st8(p.dst, i, p.dst_type, o);
    }
  } else {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
      const int col = static_cast<int>(i % p.N);
      const float s = uses_src ? ld_elem(p.src, i, p.src_type) : 0.f;
      const float b = uses_bias ? ld_elem(p.bias, col, p.bias_type) : 0.f;
      const float y = uses_y ? ld_elem(p.Y, i, p.y_type) : 0.f;
      st_elem(p.dst, i, p.dst_type, ew_apply<OP>(s, b, y, p.scale));
    }
  }
}

static bool aligned16(const void* q) { return q == nullptr || (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

template <int OP>
static cudaError_t launch_ew(const EwParams& p, int num_sms, cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(p.M) * p.N;
  if (total == 0) return cudaSuccess;
  const bool vec = (p.N % 8 == 0) && aligned16(p.src) && aligned16(p.bias) && aligned16(p.Y) &&
                   aligned16(p.dst);  // (8 fp8 outputs are 8 bytes: 8-byte aligned when dst is)
  const int64_t work = vec ? (total + 7) / 8 : total;
  int64_t blocks = (work + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 16;
  if (blocks > cap) blocks = cap;
  if (vec)
    ew_kernel<OP, true><<<static_cast<unsigned>(blocks), 256, 0, s>>>(p);
  else
    ew_kernel<OP, false><<<static_cast<unsigned>(blocks), 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_kzero(int epi, const SimtParams& sp, int num_sms, cudaStream_t s) {
  EwParams p{sp.out_scale, nullptr, 0, sp.bias, sp.bias_type, sp.Y, sp.y_type, sp.out, sp.out_type,
             sp.M, sp.N};
  if (epi == EPI_QUANT) return launch_ew<EW_KZERO_QUANT>(p, num_sms, s);
  if (epi == EPI_GATE) return launch_ew<EW_KZERO_GATE>(p, num_sms, s);
  if (epi == EPI_RESID) return launch_ew<EW_KZERO_RESID>(p, num_sms, s);
  return launch_ew<EW_KZERO_RELU>(p, num_sms, s);
}

cudaError_t launch_ew_bias_inplace(void* I, int inter_type, const void* bias, int bias_type, int M,
                                   int N, int num_sms, cudaStream_t s) {
  EwParams p{1.0f, I, inter_type, bias, bias_type, nullptr, 0, I, inter_type, M, N};
  return launch_ew<EW_BIAS_INPLACE>(p, num_sms, s);
}

cudaError_t launch_ew_relu(const void* I, int inter_type, void* out, int out_type, int M, int N,
                           int num_sms, cudaStream_t s) {
  EwParams p{1.0f, I, inter_type, nullptr, 0, nullptr, 0, out, out_type, M, N};
  return launch_ew<EW_RELU>(p, num_sms, s);
}

cudaError_t launch_ew_bias_gate(const void* I, int inter_type, const void* bias, int bias_type,
                                const void* Y, int y_type, void* out, int out_type, int M, int N,
                                int num_sms, cudaStream_t s) {
  EwParams p{1.0f, I, inter_type, bias, bias_type, Y, y_type, out, out_type, M, N};
  return launch_ew<EW_BIAS_GATE>(p, num_sms, s);
}

}  // namespace fgemm
