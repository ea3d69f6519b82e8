// Fused router: logits = (x Wg^T + b + g) / tau, softmax, top-k on the logits
// (descending, ties to the lower expert index), renormalised gates, and a
// per-block partial sum of the probabilities for P_i.
//
// Follows the kwkr.cn MoE article ("MoE sparse activation: from the math to
// the code"), section 2.1 (gate softmax, top-k on logits, second
// normalisation) and section 5.3 (fusing softmax with top-k); noise and
// temperature as in the lpnh.cn MoE guide, section 3.3.
#include "moe_internal.h"

#include <math.h>

namespace moe {
namespace {

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

constexpr int TT = kRouterTile;  // tokens per tile
constexpr int KC = 32;           // reduction chunk
constexpr int NT = 256;          // threads per block

// Each thread owns 2 tokens x EP experts of the [TT, 16*EP] logit tile.
template <typename Tin, int EP>
__global__ void __launch_bounds__(NT) router_simt_kernel(
    const Tin* __restrict__ x, const Tin* __restrict__ Wg, const float* __restrict__ bias,
    const float* __restrict__ noise, float noise_scale, float tau, int T, int d, int E, int k,
    float* __restrict__ logits, int32_t* __restrict__ idx, float* __restrict__ gate,
    float* __restrict__ partial) {
  constexpr int EPAD = 16 * EP;
  constexpr int LDS = KC + 1;
  constexpr int LDL = EPAD + 1;
  constexpr int SMEM_MAIN = (TT + EPAD) * LDS;
  constexpr int SMEM_LOG = TT * LDL;
  constexpr int SMEM = SMEM_MAIN > SMEM_LOG ? SMEM_MAIN : SMEM_LOG;
  constexpr int PER = (EPAD + 31) / 32;
  __shared__ float sm[SMEM];
  __shared__ float acc_p[EPAD];
  float* xs = sm;             // [TT][LDS]
  float* wsm = sm + TT * LDS; // [EPAD][LDS]
  float* ls = sm;             // [TT][LDL], reused after the reduction loop

  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < EPAD; e += NT) acc_p[e] = 0.f;
  const int ntiles = (T + TT - 1) / TT;

  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int t0 = tile * TT;
    float acc[2][EP];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int c = 0; c < EP; ++c) acc[i][c] = 0.f;

    for (int k0 = 0; k0 < d; k0 += KC) {
      __syncthreads();
      for (int i = tid; i < TT * KC; i += NT) {
        const int r = i / KC, cc = i % KC, t = t0 + r, kk = k0 + cc;
        xs[r * LDS + cc] = (t < T && kk < d) ? to_f(x[(size_t)t * d + kk]) : 0.f;
      }
      for (int i = tid; i < EPAD * KC; i += NT) {
        const int r = i / KC, cc = i % KC, kk = k0 + cc;
        wsm[r * LDS + cc] = (r < E && kk < d) ? to_f(Wg[(size_t)r * d + kk]) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < KC; ++kk) {
        const float a0 = xs[(2 * ty) * LDS + kk], a1 = xs[(2 * ty + 1) * LDS + kk];
#pragma unroll
        for (int c = 0; c < EP; ++c) {
          const float b = wsm[(tx + 16 * c) * LDS + kk];
          acc[0][c] = fmaf(a0, b, acc[0][c]);
          acc[1][c] = fmaf(a1, b, acc[1][c]);
        }
      }
    }
    __syncthreads();
    // selection keys l = (z + b + s g) / tau, s = 1 or noise_scale times the
    // population standard deviation of the token's E logits z + b (the 16
    // threads of a token's row, lanes of one half-warp, sum in a fixed order)
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = 2 * ty + i, t = t0 + r;
      float sn = 1.f;
      if (bias) {
#pragma unroll
        for (int c = 0; c < EP; ++c)
          if (tx + 16 * c < E) acc[i][c] += bias[tx + 16 * c];
      }
      if (noise && noise_scale > 0.f) {
        float s1 = 0.f;
#pragma unroll
        for (int c = 0; c < EP; ++c)
          if (tx + 16 * c < E) s1 += acc[i][c];
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        const float mean = s1 / (float)E;
        float s2 = 0.f;
#pragma unroll
        for (int c = 0; c < EP; ++c) {
          const float dv = acc[i][c] - mean;
          if (tx + 16 * c < E) s2 = fmaf(dv, dv, s2);
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
        sn = noise_scale * sqrtf(s2 / (float)E);
      }
#pragma unroll
      for (int c = 0; c < EP; ++c) {
        const int e = tx + 16 * c;
        float v = acc[i][c];
        if (e < E && t < T) {
          if (noise) v = fmaf(sn, noise[(size_t)t * E + e], v);
          v = v / tau;
        }
        ls[r * LDL + e] = v;
      }
    }
    __syncthreads();
    // one warp per token: softmax, top-k, gates
    for (int r = warp; r < TT; r += NT / 32) {
      const int t = t0 + r;
      if (t >= T) continue;  // warp-uniform
      float v[PER], ex[PER];
      bool taken[PER];
      float m = -INFINITY;
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int e = lane + 32 * q;
        v[q] = e < E ? ls[r * LDL + e] : -INFINITY;
        taken[q] = false;
        m = fmaxf(m, v[q]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int e = lane + 32 * q;
        ex[q] = e < E ? expf(v[q] - m) : 0.f;
        s += ex[q];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int e = lane + 32 * q;
        if (e < E) {
          if (logits) logits[(size_t)t * E + e] = v[q];
          ls[r * LDL + e] = ex[q] / s;  // probability, reused for the partial sums
        }
      }
      __syncwarp();
      float psum = 0.f;
      float psel[kMaxK];
      int isel[kMaxK];
      for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int q = 0; q < PER; ++q) {
          const int e = lane + 32 * q;
          if (e < E && !taken[q] && (v[q] > bv || (v[q] == bv && e < bi))) {
            bv = v[q];
            bi = e;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (ov > bv || (ov == bv && oi < bi)) {
            bv = ov;
            bi = oi;
          }
        }
        if (bi >= E) bi = 0;  // only reachable with NaN keys; keeps the read in bounds
#pragma unroll
        for (int q = 0; q < PER; ++q)
          if (bi == lane + 32 * q) taken[q] = true;
        isel[j] = bi;
        psel[j] = ls[r * LDL + bi];
        psum += psel[j];
      }
      if (lane == 0) {
        for (int j = 0; j < k; ++j) {
          idx[(size_t)t * k + j] = isel[j];
          gate[(size_t)t * k + j] = psel[j] / psum;
        }
      }
    }
    __syncthreads();
    for (int e = tid; e < E; e += NT) {
      float s = 0.f;
      for (int r = 0; r < TT; ++r)
        if (t0 + r < T) s += ls[r * LDL + e];
      acc_p[e] += s;
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += NT) partial[(size_t)blockIdx.x * E + e] = acc_p[e];
}

// prob_sum[e] = sum over blocks of partial[b, e]: one block per expert, a
// fixed-shape tree in fp64 (deterministic).
__global__ void __launch_bounds__(256) prob_reduce_kernel(const float* __restrict__ partial,
                                                          int nparts, int E,
                                                          float* __restrict__ prob_sum) {
  __shared__ double red[256];
  const int e = blockIdx.x, tid = threadIdx.x;
  double s = 0.0;
  for (int b = tid; b < nparts; b += 256) s += (double)partial[(size_t)b * E + e];
  red[tid] = s;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (tid < w) red[tid] += red[tid + w];
    __syncthreads();
  }
  if (tid == 0) prob_sum[e] = (float)red[0];
}

template <typename Tin>
cudaError_t launch_router_t(const moe_config_t& c, const void* x, const void* Wg,
                            const float* bias, const float* noise, float* logits,
                            int32_t* idx, float* gate, float* partial, int grid,
                            cudaStream_t s) {
  const Tin* xp = static_cast<const Tin*>(x);
  const Tin* wp = static_cast<const Tin*>(Wg);
  const int epad = (c.E + 15) / 16;
#define MOE_ROUTER_CASE(EPV)                                                              \
  router_simt_kernel<Tin, EPV><<<grid, NT, 0, s>>>(xp, wp, bias, noise, c.noise_scale, c.tau, \
                                                   c.T, c.d, c.E, c.k, logits, idx, gate,     \
                                                   partial)
  if (epad <= 1) MOE_ROUTER_CASE(1);
  else if (epad <= 2) MOE_ROUTER_CASE(2);
  else if (epad <= 4) MOE_ROUTER_CASE(4);
  else if (epad <= 8) MOE_ROUTER_CASE(8);
  else MOE_ROUTER_CASE(16);
#undef MOE_ROUTER_CASE
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const moe_config_t& c, const void* x, const void* Wg,
                          const float* bias, const float* noise, float* logits,
                          int32_t* idx, float* gate, float* partial, int grid,
                          cudaStream_t s) {
  if (c.dtype == MOE_F32)
    return launch_router_t<float>(c, x, Wg, bias, noise, logits, idx, gate, partial, grid, s);
  return launch_router_t<__nv_bfloat16>(c, x, Wg, bias, noise, logits, idx, gate, partial,
                                        grid, s);
}

cudaError_t launch_prob_reduce(const moe_config_t& c, const float* partial, int nparts,
                               float* prob_sum, cudaStream_t s) {
  prob_reduce_kernel<<<c.E, 256, 0, s>>>(partial, nparts, c.E, prob_sum);
  return cudaGetLastError();
}

}  // namespace moe
