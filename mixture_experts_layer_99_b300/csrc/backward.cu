// Backward pass of the layer: the memory-bound steps (CUDA cores).
//
// loss = sum_t <dy_t, y_t> + alpha * L_balance. The kwkr.cn MoE article ("MoE
// sparse activation: from the math to the code") trains the layer with
// L_balance added to the task loss (section 2.2) and trains the router
// (section 3.3); the gradients are the chain rule through its forward:
//   combine      dY[slot] = g_tj dy_t,  dg_tj = <dy_t, Y[slot]>
//   gates        dp_{K_i} += (dg_i - sum_j g_j dg_j) / S,  S = sum_m p_{K_m}
//   balance      dp_ti += alpha E f_i / T
//   softmax      dl_t = p_t (dp_t - <p_t, dp_t>),  dz = dl / tau
//   router GEMM  dx += dz Wg,  dWg = dz^T x,  db = sum_t dz_t
//   dispatch     dx_t += sum over the kept slots of t of dxd[slot]
// Routing (top-k, capacity, drops) is piecewise constant and gets no gradient.
// Every sum runs in a fixed order, so results are run-to-run identical.
#include "moe_internal.h"

#include <type_traits>

namespace moe {
namespace {

constexpr int NT = 256, NW = NT / 32;

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}

// One warp per token: dY rows of its kept slots and the gate gradients.
// Y (the forward's expert outputs) may be null when k = 1: a single gate is
// identically 1 and its gradient has no effect.
__global__ void __launch_bounds__(NT) bwd_combine_kernel(const uint4* __restrict__ dy,
                                                         const uint4* __restrict__ Y,
                                                         const int32_t* __restrict__ slot_of,
                                                         const float* __restrict__ gate, int T,
                                                         int k, int nvec,
                                                         uint4* __restrict__ dY,
                                                         float* __restrict__ dg, int64_t rows_cap,
                                                         int32_t* __restrict__ chk) {
  const int t = blockIdx.x * NW + (threadIdx.x >> 5);
  if (t >= T) return;
  const int lane = threadIdx.x & 31;
  for (int j = 0; j < k; ++j) {
    int sl = slot_of[(size_t)t * k + j];
    if (!moe_check(sl < rows_cap, chk, 55)) sl = -1;
    const float g = gate[(size_t)t * k + j];
    float dot = 0.f;
    if (sl >= 0) {
      for (int v = lane; v < nvec; v += 32) {
        float a[8], o[8];
        unpack8(__ldg(dy + (size_t)t * nvec + v), a);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = g * a[i];
        dY[(size_t)sl * nvec + v] = pack8(o);
        if (Y) {
          float b[8];
          unpack8(__ldg(Y + (size_t)sl * nvec + v), b);
#pragma unroll
          for (int i = 0; i < 8; ++i) dot = fmaf(a[i], b[i], dot);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    if (lane == 0) dg[(size_t)t * k + j] = dot;
  }
}

// One thread per token: dz[t, :] from the gates' gradients and the balance
// term, through the softmax of the saved keys (logits).
template <int EP>
__global__ void __launch_bounds__(128) bwd_router_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ idx,
    const float* __restrict__ gate, const float* __restrict__ dg,
    const float* __restrict__ f, float alpha, float tau, int T, int E, int k,
    float* __restrict__ dz, __nv_bfloat16* __restrict__ dzb, int Kp) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  float p[EP];
  float m = -INFINITY;
#pragma unroll
  for (int e = 0; e < EP; ++e) {
    p[e] = e < E ? logits[(size_t)t * E + e] : -INFINITY;
    m = fmaxf(m, p[e]);
  }
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < EP; ++e) {
    p[e] = e < E ? expf(p[e] - m) : 0.f;
    s += p[e];
  }
  const float inv_s = 1.f / s;
  // dp = balance term + gate term on the chosen experts
  float dp[EP];
  const float bal = alpha * (float)E / (float)T;
#pragma unroll
  for (int e = 0; e < EP; ++e) {
    p[e] *= inv_s;
    dp[e] = e < E ? bal * f[e] : 0.f;
  }
  float S = 0.f, gdg = 0.f;
  for (int j = 0; j < k; ++j) {
    const int e = idx[(size_t)t * k + j];
    float pe = 0.f;
#pragma unroll
    for (int q = 0; q < EP; ++q)
      if (q == e) pe = p[q];
    S += pe;
    gdg = fmaf(gate[(size_t)t * k + j], dg[(size_t)t * k + j], gdg);
  }
  const float inv_S = 1.f / S;
  for (int j = 0; j < k; ++j) {
    const int e = idx[(size_t)t * k + j];
    const float add = (dg[(size_t)t * k + j] - gdg) * inv_S;
#pragma unroll
    for (int q = 0; q < EP; ++q)
      if (q == e) dp[q] += add;
  }
  float pdp = 0.f;
#pragma unroll
  for (int e = 0; e < EP; ++e) pdp = fmaf(p[e], dp[e], pdp);
  const float inv_tau = 1.f / tau;
#pragma unroll
  for (int e = 0; e < EP; ++e) {
    const float z = e < E ? p[e] * (dp[e] - pdp) * inv_tau : 0.f;
    if (e < E) dz[(size_t)t * E + e] = z;
    dp[e] = z;
  }
  // bf16 copy with the experts padded to Kp (the operand of the dz W_g and
  // dz^T x GEMMs)
  __nv_bfloat16* zr = dzb + (size_t)t * Kp;
  for (int e0 = 0; e0 < Kp; e0 += 8) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = 0.f;
#pragma unroll
      for (int q = 0; q < EP; ++q)
        if (q == e0 + i) v[i] = dp[q];
    }
    *reinterpret_cast<uint4*>(zr + e0) = pack8(v);
  }
}

// The same for E > 64: one warp per token, expert e = 32 i + lane in slot i
// of its lane (EPL = experts per lane), the sums over experts by warp
// butterflies in a fixed order.
__device__ __forceinline__ float warp_sum_bwd(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
template <int EPL>
__global__ void __launch_bounds__(NT) bwd_router_wide_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ idx,
    const float* __restrict__ gate, const float* __restrict__ dg,
    const float* __restrict__ f, float alpha, float tau, int T, int E, int k,
    float* __restrict__ dz, __nv_bfloat16* __restrict__ dzb, int Kp) {
  const int t = blockIdx.x * NW + (threadIdx.x >> 5);
  if (t >= T) return;
  const int lane = threadIdx.x & 31;
  float p[EPL], dp[EPL];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = 32 * i + lane;
    p[i] = e < E ? logits[(size_t)t * E + e] : -INFINITY;
    m = fmaxf(m, p[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    p[i] = 32 * i + lane < E ? expf(p[i] - m) : 0.f;
    s += p[i];
  }
  const float inv_s = 1.f / warp_sum_bwd(s);
  const float bal = alpha * (float)E / (float)T;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = 32 * i + lane;
    p[i] *= inv_s;
    dp[i] = e < E ? bal * f[e] : 0.f;
  }
  // S = sum_j p[K_j], gdg = sum_j g_j dg_j (the same in every lane)
  float S = 0.f, gdg = 0.f;
  for (int j = 0; j < k; ++j) {
    const int e = idx[(size_t)t * k + j];
    float mine = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (i == (e >> 5)) mine = p[i];
    S += __shfl_sync(0xffffffffu, mine, e & 31);
    gdg = fmaf(gate[(size_t)t * k + j], dg[(size_t)t * k + j], gdg);
  }
  const float inv_S = 1.f / S;
  for (int j = 0; j < k; ++j) {
    const int e = idx[(size_t)t * k + j];
    const float add = (dg[(size_t)t * k + j] - gdg) * inv_S;
    if ((e & 31) == lane) {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (i == (e >> 5)) dp[i] += add;
    }
  }
  float pdp = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) pdp = fmaf(p[i], dp[i], pdp);
  pdp = warp_sum_bwd(pdp);
  const float inv_tau = 1.f / tau;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = 32 * i + lane;
    const float z = e < E ? p[i] * (dp[i] - pdp) * inv_tau : 0.f;
    if (e < E) dz[(size_t)t * E + e] = z;
    // bf16 copy with the experts padded to Kp (zeros past E)
    if (e < Kp) dzb[(size_t)t * Kp + e] = __float2bfloat16_rn(z);
  }
}

// dx_t = sum over the kept slots of dxd[slot] (slot order) + dxr_t (the
// router term dz_t W_g from the tensor cores) [+ dxs_t, the shared expert's
// term, if given], fp32, rounded once. Warp w of block (bx, by) owns token
// bx * NW + w and a chunk of 32 UNR 16-byte vectors. Every lane issues all of
// its loads (each slot's, dxr's and dxs's) before it adds them in that order.
template <int KM>
struct DxShape {
  static constexpr int UNR = KM <= 2 ? 4 : (KM <= 4 ? 2 : 1);
  static constexpr int CHUNK = 32 * UNR;
};
template <int KM>
__global__ void __launch_bounds__(NT) bwd_dx_kernel(const uint4* __restrict__ dxd,
                                                    const int32_t* __restrict__ slot_of,
                                                    const uint4* __restrict__ dxr, int T, int k,
                                                    int nvec, uint4* __restrict__ dx,
                                                    const uint4* __restrict__ dxs,
                                                    int64_t rows_cap, int32_t* __restrict__ chk) {
  constexpr int UNR = DxShape<KM>::UNR;
  const int t = blockIdx.x * NW + (threadIdx.x >> 5);
  if (t >= T) return;
  const int lane = threadIdx.x & 31;
  const int v0 = blockIdx.y * DxShape<KM>::CHUNK + lane;
  int sl[KM];
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    sl[j] = j < k ? slot_of[(size_t)t * k + j] : -1;
    if (!moe_check(sl[j] < rows_cap, chk, 56)) sl[j] = -1;
  }
  uint4 q[KM][UNR], qr[UNR], qs[UNR];
#pragma unroll
  for (int u = 0; u < UNR; ++u) {
    const int v = v0 + 32 * u;
    const bool in = v < nvec;
#pragma unroll
    for (int j = 0; j < KM; ++j)
      q[j][u] = in && sl[j] >= 0 ? __ldg(dxd + (size_t)sl[j] * nvec + v) : make_uint4(0, 0, 0, 0);
    qr[u] = in ? __ldg(dxr + (size_t)t * nvec + v) : make_uint4(0, 0, 0, 0);
    qs[u] = in && dxs ? __ldg(dxs + (size_t)t * nvec + v) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int u = 0; u < UNR; ++u) {
    const int v = v0 + 32 * u;
    if (v >= nvec) continue;
    float acc[8], a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (sl[j] < 0) continue;
      unpack8(q[j][u], a);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += a[i];
    }
    unpack8(qr[u], a);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += a[i];
    if (dxs) {
      unpack8(qs[u], a);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += a[i];
    }
    dx[(size_t)t * nvec + v] = pack8(acc);
  }
}

// db[e] = sum_t dz[t, e]: one block per expert, thread i sums tokens
// i, i + 256, ... in order, then a fixed-order tree.
__global__ void __launch_bounds__(256) bwd_dbias_kernel(const float* __restrict__ dz, int T,
                                                        int E, float* __restrict__ db) {
  __shared__ float red[256];
  const int e = blockIdx.x;
  float s = 0.f;
  for (int t = threadIdx.x; t < T; t += 256) s += dz[(size_t)t * E + e];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) db[e] = red[0];
}

// Token groups of the dz^T x GEMM: goff[g] = min(g * per, Tp), goff[G] = Tp
// (a group past the end is empty and its partial is zero).
__global__ void group_offsets_kernel(int32_t* __restrict__ goff, int G, int per, int Tp) {
  for (int g = threadIdx.x; g <= G; g += blockDim.x) goff[g] = g < G ? min(g * per, Tp) : Tp;
}

// Sum of the token-split partials in split order.
__global__ void bwd_wg_reduce_kernel(const float* __restrict__ part, int nsplit, int E, int d,
                                     float* __restrict__ dWg) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int n = E * d;
  if (i < n) {
    float s = 0.f;
    for (int sp = 0; sp < nsplit; ++sp) s += part[(size_t)sp * n + i];
    dWg[i] = s;
  }
}

// Batched transpose of expert weights (the [W1^T | W3^T] copy a SwiGLU hidden
// size that is not a multiple of 64 needs): out[e][b][a + a_off] = in[e][a][b]
// (in [E, A, B] row-major, out [E, B, ld_out]); 64 x 64 tiles moved as
// 16-byte vectors (A, B, ld_out and a_off are multiples of 8).
__global__ void __launch_bounds__(256) weight_transpose_kernel(
    const __nv_bfloat16* __restrict__ in, int A, int B, int ld_out, int a_off,
    __nv_bfloat16* __restrict__ out) {
  __shared__ __align__(16) __nv_bfloat16 tile[64][72];  // [a][b]
  const int e = blockIdx.z;
  const int a0 = blockIdx.y * 64, b0 = blockIdx.x * 64;
  const __nv_bfloat16* ie = in + (size_t)e * A * B;
  __nv_bfloat16* oe = out + (size_t)e * B * ld_out;
  const int tid = threadIdx.x;
  for (int q = tid; q < 64 * 8; q += 256) {
    const int i = q >> 3, jv = q & 7;
    const int a = a0 + i, b = b0 + jv * 8;
    uint4 w = make_uint4(0, 0, 0, 0);
    if (a < A && b < B) w = __ldg(reinterpret_cast<const uint4*>(ie + (size_t)a * B + b));
    *reinterpret_cast<uint4*>(&tile[i][jv * 8]) = w;
  }
  __syncthreads();
  for (int q = tid; q < 64 * 8; q += 256) {
    const int j = q & 63, iv = q >> 6;
    const int b = b0 + j, a = a0 + iv * 8;
    if (b >= B || a >= A) continue;
    uint4 w;
    __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(&w);
#pragma unroll
    for (int t = 0; t < 8; ++t) h[t] = tile[iv * 8 + t][j];
    *reinterpret_cast<uint4*>(oe + (size_t)b * ld_out + a_off + a) = w;
  }
}

// Per-expert column sums of a packed [rows, C] matrix (row stride ld) over the
// expert's rows, in row order: out[e, c] (fp32).
__global__ void __launch_bounds__(128) expert_colsum_kernel(const __nv_bfloat16* __restrict__ a,
                                                            int ld, int C,
                                                            const int32_t* __restrict__ off,
                                                            float* __restrict__ out) {
  const int e = blockIdx.y;
  const int c = blockIdx.x * 128 + threadIdx.x;
  if (c >= C) return;
  float s = 0.f;
  for (int r = off[e]; r < off[e + 1]; ++r) s += __bfloat162float(a[(size_t)r * ld + c]);
  out[(size_t)e * C + c] = s;
}

template <int EP>
cudaError_t launch_router_bwd_ep(const moe_config_t& c, const float* logits, const int32_t* idx,
                                 const float* gate, const float* dg, const float* f, float alpha,
                                 float* dz, void* dzb, int Kp, cudaStream_t s) {
  bwd_router_kernel<EP><<<(c.T + 127) / 128, 128, 0, s>>>(
      logits, idx, gate, dg, f, alpha, c.tau, c.T, c.E, c.k, dz,
      static_cast<__nv_bfloat16*>(dzb), Kp);
  return cudaGetLastError();
}
template <int EPL>
cudaError_t launch_router_bwd_wide(const moe_config_t& c, const float* logits, const int32_t* idx,
                                   const float* gate, const float* dg, const float* f,
                                   float alpha, float* dz, void* dzb, int Kp, cudaStream_t s) {
  bwd_router_wide_kernel<EPL><<<(c.T + NW - 1) / NW, NT, 0, s>>>(
      logits, idx, gate, dg, f, alpha, c.tau, c.T, c.E, c.k, dz,
      static_cast<__nv_bfloat16*>(dzb), Kp);
  return cudaGetLastError();
}

}  // namespace

// Token groups of the dz^T x GEMM (each a multiple of 64 tokens, at least
// 512 when there are enough, at most 64 groups).
int bwd_wg_splits(const moe_config_t& c) {
  const int tp = (c.T + 63) / 64 * 64;
  int g = tp / 512;
  if (g < 1) g = 1;
  if (g > 64) g = 64;
  return g;
}
int bwd_wg_group_tokens(const moe_config_t& c) {
  const int tp = (c.T + 63) / 64 * 64;
  const int g = bwd_wg_splits(c);
  return ((tp + g - 1) / g + 63) / 64 * 64;
}

cudaError_t launch_bwd_combine(const moe_config_t& c, const void* dy, const void* Y,
                               const int32_t* slot_of, const float* gate, void* dY, float* dg,
                               cudaStream_t s, int32_t* chk) {
  const int nvec = c.d / 8;
  bwd_combine_kernel<<<(c.T + NW - 1) / NW, NT, 0, s>>>(
      static_cast<const uint4*>(dy), static_cast<const uint4*>(Y), slot_of, gate, c.T, c.k, nvec,
      static_cast<uint4*>(dY), dg, (int64_t)max_rows(c), chk);
  return cudaGetLastError();
}

cudaError_t launch_bwd_router(const moe_config_t& c, const float* logits, const int32_t* idx,
                              const float* gate, const float* dg, const float* f, float alpha,
                              float* dz, void* dzb, int Kp, cudaStream_t s) {
  const int ep = (c.E + 15) / 16 * 16;
#define MOE_RB(EPV) \
  launch_router_bwd_ep<EPV>(c, logits, idx, gate, dg, f, alpha, dz, dzb, Kp, s)
  switch (ep) {
    case 16: return MOE_RB(16);
    case 32: return MOE_RB(32);
    case 48: return MOE_RB(48);
    case 64: return MOE_RB(64);
    default: break;
  }
#undef MOE_RB
  // Kp (a multiple of 64 >= E) <= 256: every padded column is in some lane's slots
  if (c.E <= 128 && Kp <= 128)
    return launch_router_bwd_wide<4>(c, logits, idx, gate, dg, f, alpha, dz, dzb, Kp, s);
  if (c.E <= 256 && Kp <= 256)
    return launch_router_bwd_wide<8>(c, logits, idx, gate, dg, f, alpha, dz, dzb, Kp, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dx(const moe_config_t& c, const void* dxd, const int32_t* slot_of,
                          const void* dxr, void* dx, cudaStream_t s, const void* dxs,
                          int32_t* chk) {
  const int nvec = c.d / 8;
  auto go = [&](auto km) {
    constexpr int KM = decltype(km)::value;
    constexpr int CH = DxShape<KM>::CHUNK;
    const dim3 grid((unsigned)((c.T + NW - 1) / NW), (unsigned)((nvec + CH - 1) / CH));
    bwd_dx_kernel<KM><<<grid, NT, 0, s>>>(static_cast<const uint4*>(dxd), slot_of,
                                          static_cast<const uint4*>(dxr), c.T, c.k, nvec,
                                          static_cast<uint4*>(dx), static_cast<const uint4*>(dxs),
                                          (int64_t)max_rows(c), chk);
    return cudaGetLastError();
  };
  if (c.k <= 2) return go(std::integral_constant<int, 2>{});
  if (c.k <= 4) return go(std::integral_constant<int, 4>{});
  return go(std::integral_constant<int, kMaxK>{});
}

// dWg = dz^T x on the tensor cores: token groups of the weight-gradient GEMM
// (A = dz in bf16 [T][Kp], B = x [T][d], both read MN-major; groups are
// multiples of 64 tokens, rows past T read as zeros) give fp32 partials
// [G][E][d], summed in group order; db = column sums of dz.
cudaError_t launch_bwd_wg(const moe_config_t& c, const float* dz, const void* dzb, int Kp,
                          const void* x, int32_t* goff, float* part, float* dWg, float* dbias,
                          int32_t* hdr, cudaStream_t s) {
  const int G = bwd_wg_splits(c), per = bwd_wg_group_tokens(c);
  const int Tp = (c.T + 63) / 64 * 64;
  group_offsets_kernel<<<1, 128, 0, s>>>(goff, G, per, Tp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_wgrad_tc(dzb, Kp, x, c.d, c.T, goff, G, c.E, c.d, c.E, part, part, hdr, s);
  if (e != cudaSuccess) return e;
  const int n = c.E * c.d;
  bwd_wg_reduce_kernel<<<(n + 255) / 256, 256, 0, s>>>(part, G, c.E, c.d, dWg);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (dbias) {
    bwd_dbias_kernel<<<c.E, 256, 0, s>>>(dz, c.T, c.E, dbias);
    e = cudaGetLastError();
  }
  return e;
}


cudaError_t launch_weight_transpose(const void* in, int E, int A, int B, int ld_out, int a_off,
                                    void* out, cudaStream_t s) {
  const dim3 grid((unsigned)((B + 63) / 64), (unsigned)((A + 63) / 64), (unsigned)E);
  weight_transpose_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(in), A, B,
                                               ld_out, a_off, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

cudaError_t launch_expert_colsum(const void* a, int ld, int C, const int32_t* off, int E,
                                 float* out, cudaStream_t s) {
  const dim3 grid((unsigned)((C + 127) / 128), (unsigned)E);
  expert_colsum_kernel<<<grid, 128, 0, s>>>(static_cast<const __nv_bfloat16*>(a), ld, C, off,
                                            out);
  return cudaGetLastError();
}

}  // namespace moe
