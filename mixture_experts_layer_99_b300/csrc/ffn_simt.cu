// Grouped expert FFN on fp32 FMA (the fp32 workload; no tensor cores, since
// TF32 would not hold the fp32 tolerance).
//
// Expert e owns packed rows [offset_e, offset_{e+1}); both GEMMs tile those
// rows in 64-row blocks that never cross an expert boundary. The tile list is
// derived on the device from offset[], so no host synchronisation is needed.
//   GEMM1: h = gelu(xd W1_e^T + b1_e)            (GELU, kwkr.cn MoE article 3.1)
//          h = silu(xd W1_e^T) * (xd W3_e^T)      (SwiGLU)
//   GEMM2: Y = h W2_e^T + b2_e
#include "moe_internal.h"

#include <math.h>

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, NT = 256;

enum Epi { kEpiNone = 0, kEpiGelu = 1, kEpiSwiglu = 2 };

template <typename T> __device__ __forceinline__ float ld_f(const T* p);
template <> __device__ __forceinline__ float ld_f<float>(const float* p) { return __ldg(p); }
template <> __device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

__device__ __forceinline__ float gelu_erf(float u) {
  return 0.5f * u * (1.f + erff(u * 0.70710678118654752f));
}
__device__ __forceinline__ float silu_f(float u) { return u / (1.f + expf(-u)); }

// Finds (expert, first row, end row) of linear m-tile `tile`; returns false if
// the tile is beyond the last expert's rows. The offsets may be a caller's
// input (moe_expert_ffn): unless offset[0] = 0 <= offset[1] <= ... <=
// offset[E] <= rows_limit, no tile runs and the status header records
// MOE_ERR_INVALID_ARG (where = 43).
__device__ bool find_tile(const int32_t* offset, int E, int rows_limit, int32_t* hdr, int tile,
                          int bm, int* e_out, int* m0_out, int* mend_out) {
  bool bad = offset[0] != 0;
  for (int e = 0; e < E; ++e) bad |= offset[e + 1] < offset[e];
  bad |= offset[E] > rows_limit;
  if (bad) {
    if (hdr != nullptr && atomicCAS(hdr + kHdrStatus, 0, (int)MOE_ERR_INVALID_ARG) == 0)
      atomicExch(hdr + kHdrWhere, 43);
    return false;
  }
  int cum = 0;
  for (int e = 0; e < E; ++e) {
    const int r0 = offset[e], r1 = offset[e + 1];
    const int nt = (r1 - r0 + bm - 1) / bm;
    if (tile < cum + nt) {
      *e_out = e;
      *m0_out = r0 + (tile - cum) * bm;
      *mend_out = r1;
      return true;
    }
    cum += nt;
  }
  return false;
}

template <typename T, int EPI>
__global__ void __launch_bounds__(NT) ffn_simt_kernel(const T* __restrict__ A,
                                                      const T* __restrict__ B,
                                                      const T* __restrict__ B3,
                                                      const T* __restrict__ bias,
                                                      T* __restrict__ Cout,
                                                      const int32_t* __restrict__ offset, int E,
                                                      int N, int K, int rows_limit,
                                                      int32_t* __restrict__ hdr) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  __shared__ float B3s[EPI == kEpiSwiglu ? BK : 1][BN + 4];
  __shared__ int s_e, s_m0, s_mend;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  if (tid == 0) {
    int e = -1, m0 = 0, mend = 0;
    if (!find_tile(offset, E, rows_limit, hdr, blockIdx.y, BM, &e, &m0, &mend)) e = -1;
    s_e = e;
    s_m0 = m0;
    s_mend = mend;
  }
  __syncthreads();
  const int e = s_e;
  if (e < 0) return;
  const int m0 = s_m0, mend = s_mend, n0 = blockIdx.x * BN;
  const T* Be = B + (size_t)e * N * K;
  const T* B3e = EPI == kEpiSwiglu ? B3 + (size_t)e * N * K : nullptr;
  float acc[4][4], acc3[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = acc3[i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += BK) {
    for (int i = tid; i < BM * BK; i += NT) {
      const int r = i / BK, kk = i % BK, row = m0 + r, col = k0 + kk;
      As[kk][r] = (row < mend && col < K) ? ld_f(A + (size_t)row * K + col) : 0.f;
    }
    for (int i = tid; i < BN * BK; i += NT) {
      const int n = i / BK, kk = i % BK, nn = n0 + n, col = k0 + kk;
      const bool ok = nn < N && col < K;
      Bs[kk][n] = ok ? ld_f(Be + (size_t)nn * K + col) : 0.f;
      if (EPI == kEpiSwiglu) B3s[kk][n] = ok ? ld_f(B3e + (size_t)nn * K + col) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4], b3[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        b[j] = Bs[kk][tx * 4 + j];
        if (EPI == kEpiSwiglu) b3[j] = B3s[kk][tx * 4 + j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
          if (EPI == kEpiSwiglu) acc3[i][j] = fmaf(a[i], b3[j], acc3[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = m0 + ty * 4 + i;
    if (row >= mend) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = n0 + tx * 4 + j;
      if (col >= N) continue;
      float v = acc[i][j];
      if (EPI == kEpiSwiglu) {
        v = silu_f(v) * acc3[i][j];
      } else {
        if (bias) v += ld_f(bias + (size_t)e * N + col);
        if (EPI == kEpiGelu) v = gelu_erf(v);
      }
      Cout[(size_t)row * N + col] = from_f<T>(v);
    }
  }
}

template <typename T>
cudaError_t launch_ffn_simt_t(const moe_config_t& c, const void* xd, const int32_t* offset,
                              const void* W1, const void* W3, const void* W2,
                              const void* b1, const void* b2, void* Y, void* h,
                              int64_t rows_bound, int32_t* hdr, cudaStream_t s) {
  const int64_t mt = (rows_bound + BM - 1) / BM + c.E;
  const int rl = (int)(rows_bound < INT32_MAX ? rows_bound : INT32_MAX);
  dim3 g1((c.H + BN - 1) / BN, (unsigned)mt), g2((c.d + BN - 1) / BN, (unsigned)mt);
  const T* A = static_cast<const T*>(xd);
  T* hp = static_cast<T*>(h);
  if (c.act == MOE_ACT_SWIGLU)
    ffn_simt_kernel<T, kEpiSwiglu><<<g1, NT, 0, s>>>(A, static_cast<const T*>(W1),
                                                     static_cast<const T*>(W3), nullptr, hp,
                                                     offset, c.E, c.H, c.d, rl, hdr);
  else
    ffn_simt_kernel<T, kEpiGelu><<<g1, NT, 0, s>>>(A, static_cast<const T*>(W1), nullptr,
                                                   static_cast<const T*>(b1), hp, offset,
                                                   c.E, c.H, c.d, rl, hdr);
  ffn_simt_kernel<T, kEpiNone><<<g2, NT, 0, s>>>(
      hp, static_cast<const T*>(W2), nullptr,
      c.act == MOE_ACT_GELU ? static_cast<const T*>(b2) : nullptr, static_cast<T*>(Y),
      offset, c.E, c.d, c.H, rl, hdr);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ffn_simt(const moe_config_t& c, const void* xd, const int32_t* offset,
                            const void* W1, const void* W3, const void* W2, const void* b1,
                            const void* b2, void* Y, void* h, int64_t rows_bound,
                            int32_t* hdr, cudaStream_t s) {
  if (c.dtype == MOE_F32)
    return launch_ffn_simt_t<float>(c, xd, offset, W1, W3, W2, b1, b2, Y, h, rows_bound, hdr, s);
  return launch_ffn_simt_t<__nv_bfloat16>(c, xd, offset, W1, W3, W2, b1, b2, Y, h,
                                          rows_bound, hdr, s);
}

}  // namespace moe
