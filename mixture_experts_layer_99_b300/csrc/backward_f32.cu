// Backward pass of the fp32 layer on fp32 FMA (no tensor cores: TF32 would
// not hold the fp32 tolerance, and the fp32 configuration is the pages' small
// reference layer).
//
// The chain rule through the forward of the kwkr.cn MoE article ("MoE sparse
// activation: from the math to the code"), sections 2.1-2.3 and 3.1, with the
// balance term of its section 2.2 in the loss, the same steps as the bf16
// backward:
//   combine        dY_tj = g_tj dy_t,  dg_tj = <dy_t, Y_tj>
//   gates/softmax  dz (the shared router-backward kernel)
//   router GEMM    dWg = dz^T x,  db = sum_t dz_t,  dx_r = dz Wg
//   expert e       pre-activations recomputed from xd; dh = dY W2_e;
//                  GELU: du = dh gelu'(u); SwiGLU: da = dh v silu'(a), dv = dh silu(a)
//                  dxd = du W1_e (+ dv W3_e), dW2_e = dY^T h, dW1_e = du^T xd,
//                  dW3_e = dv^T xd, db2_e = sum dY, db1_e = sum du
//   dispatch       dx_t = dx_r,t + sum over t's kept slots of dxd[slot]
// Every output element is one thread's sum in a fixed order, so results are
// run-to-run identical.
#include "moe_internal.h"

#include <math.h>

namespace moe {
namespace {

constexpr int TM = 64, TN = 64, TK = 16, GT = 256;

// C(m, n) (+)= sum_k A(m, k) B(k, n) (+ bias(n)) over groups of experts:
//   kOne    one product, M x N x K;
//   kRowsM  group g owns the packed rows m in [off[g], off[g+1]) of A and C
//           (global row indices), B is B + g sbg, bias is bias + g sbias;
//   kRowsK  group g owns the packed rows k in [off[g], off[g+1]) of A and B,
//           C is C + g scg (an M x N block per group).
enum GroupMode { kOne = 0, kRowsM = 1, kRowsK = 2 };

struct GemmF32 {
  const float* A;
  int64_t sam, sak;
  const float* B;
  int64_t sbk, sbn, sbg;
  float* C;
  int64_t scm, scn, scg;
  const float* bias;
  int64_t sbias;
  int M, N, K, G;
  const int32_t* off;
  int accumulate;
};

__global__ void __launch_bounds__(GT) gemm_f32_kernel(GemmF32 a, int mode) {
  __shared__ float As[TK][TM + 1];
  __shared__ float Bs[TK][TN + 1];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const float* B = a.B;
  float* C = a.C;
  const float* bias = a.bias;
  int m0 = 0, m1 = 0, k0 = 0, k1 = a.K;
  if (mode == kRowsM) {
    // linear m-tile blockIdx.y over the groups' rows, in group order
    int t = (int)blockIdx.y, cum = 0, g = 0;
    for (; g < a.G; ++g) {
      const int r0 = a.off[g], r1 = a.off[g + 1];
      const int nt = (r1 - r0 + TM - 1) / TM;
      if (t < cum + nt) {
        m0 = r0 + (t - cum) * TM;
        m1 = r1;
        break;
      }
      cum += nt;
    }
    if (g == a.G) return;
    B += (int64_t)g * a.sbg;
    if (bias) bias += (int64_t)g * a.sbias;
  } else {
    m0 = (int)blockIdx.y * TM;
    m1 = a.M;
    if (mode == kRowsK) {
      const int g = (int)blockIdx.z;
      k0 = a.off[g];
      k1 = a.off[g + 1];
      C += (int64_t)g * a.scg;
    }
  }
  const int n0 = (int)blockIdx.x * TN;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int kc = k0; kc < k1; kc += TK) {
#pragma unroll
    for (int q = 0; q < (TK * TM) / GT; ++q) {
      const int e = tid + q * GT, kk = e / TM, mm = e % TM;
      const int m = m0 + mm, k = kc + kk;
      As[kk][mm] = (m < m1 && k < k1) ? a.A[(int64_t)m * a.sam + (int64_t)k * a.sak] : 0.f;
    }
#pragma unroll
    for (int q = 0; q < (TK * TN) / GT; ++q) {
      const int e = tid + q * GT, kk = e / TN, nn = e % TN;
      const int n = n0 + nn, k = kc + kk;
      Bs[kk][nn] = (n < a.N && k < k1) ? B[(int64_t)k * a.sbk + (int64_t)n * a.sbn] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty + 16 * i;
    if (m >= m1) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx + 16 * j;
      if (n >= a.N) continue;
      float v = acc[i][j];
      if (bias) v += bias[n];
      float* cp = C + (int64_t)m * a.scm + (int64_t)n * a.scn;
      *cp = a.accumulate ? *cp + v : v;
    }
  }
}

cudaError_t launch_gemm_f32(const GemmF32& a, GroupMode mode, int64_t rows_bound,
                            cudaStream_t s) {
  dim3 grid((unsigned)((a.N + TN - 1) / TN), 1, 1);
  if (mode == kRowsM) {
    // at most ceil(rows / TM) + G m-tiles over all groups
    grid.y = (unsigned)((rows_bound + TM - 1) / TM + a.G);
  } else {
    grid.y = (unsigned)((a.M + TM - 1) / TM);
    if (mode == kRowsK) grid.z = (unsigned)a.G;
  }
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  gemm_f32_kernel<<<grid, GT, 0, s>>>(a, (int)mode);
  return cudaGetLastError();
}

// dY[slot] = g dy_t and dg_tj = <dy_t, Y[slot]> (k > 1; 0 for a dropped slot
// or k = 1, where the gate is identically 1): one warp per slot (t, j), the
// dot product summed by lane in row order, then a fixed butterfly.
__global__ void bwdf_combine_kernel(const float* __restrict__ dy, const float* __restrict__ Y,
                                    const int32_t* __restrict__ slot_of,
                                    const float* __restrict__ gate, int T, int k, int d,
                                    int64_t rows_cap, float* __restrict__ dY,
                                    float* __restrict__ dg) {
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= (int64_t)T * k) return;
  const int64_t t = w / k;
  int s = slot_of[w];
  if (s >= rows_cap) s = -1;  // not a row the forward could have written
  float dot = 0.f;
  if (s >= 0) {
    const float gv = gate[w];
    for (int i = lane; i < d; i += 32) {
      const float v = dy[t * d + i];
      dY[(int64_t)s * d + i] = gv * v;
      if (Y) dot = fmaf(v, Y[(int64_t)s * d + i], dot);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
  if (lane == 0) dg[w] = (s >= 0 && Y) ? dot : 0.f;
}

// The activation's backward on the kept rows [0, off[G]):
//   GELU    dact = dh (Phi(u) + u phi(u)),                 pre = u [rows, H]
//   SwiGLU  dact = [dh v sigma(a) (1 + a (1 - sigma(a))) | dh a sigma(a)],
//           pre = [a | v] [rows, 2H]
__global__ void bwdf_act_kernel(const float* __restrict__ pre, const float* __restrict__ dh,
                                int H, int swiglu, const int32_t* __restrict__ off, int G,
                                float* __restrict__ dact) {
  const int64_t rows = off[G];
  const int64_t n = rows * H;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / H;
    const int c = (int)(i % H);
    const float g = dh[i];
    if (!swiglu) {
      const float u = pre[i];
      const float Phi = 0.5f * (1.f + erff(u * 0.70710678118654752f));
      const float phi = 0.39894228040143268f * expf(-0.5f * u * u);
      dact[i] = g * fmaf(u, phi, Phi);
    } else {
      const float a = pre[r * 2 * H + c], v = pre[r * 2 * H + H + c];
      const float sg = 1.f / (1.f + expf(-a));
      dact[r * 2 * H + c] = g * v * sg * (1.f + a * (1.f - sg));
      dact[r * 2 * H + H + c] = g * a * sg;
    }
  }
}

// out[g, c] = sum over the rows r in [off[g], off[g+1]) of a[r lda + c], in
// row order; one thread per (g, c).
__global__ void colsum_f32_kernel(const float* __restrict__ a, int64_t lda, int ncols,
                                  const int32_t* __restrict__ off, int G, float* __restrict__ out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)G * ncols) return;
  const int g = (int)(i / ncols), c = (int)(i % ncols);
  float s = 0.f;
  for (int r = off[g]; r < off[g + 1]; ++r) s += a[(int64_t)r * lda + c];
  out[i] = s;
}

cudaError_t launch_colsum_f32(const float* a, int64_t lda, int ncols, const int32_t* off, int G,
                              float* out, cudaStream_t s) {
  const int64_t n = (int64_t)G * ncols;
  colsum_f32_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a, lda, ncols, off, G, out);
  return cudaGetLastError();
}

// dx_t = dx_r,t + sum_j (kept) dxd[slot_of[t, j]] (j in order) + dxs_t
__global__ void bwdf_dx_kernel(const float* __restrict__ dxr, const float* __restrict__ dxd,
                               const float* __restrict__ dxs, const int32_t* __restrict__ slot_of,
                               int T, int k, int d, int64_t rows_cap, float* __restrict__ dx) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)T * d) return;
  const int64_t t = i / d;
  const int c = (int)(i % d);
  float v = dxr[i];
  for (int j = 0; j < k; ++j) {
    const int s = slot_of[t * k + j];
    if (s >= 0 && s < rows_cap) v += dxd[(int64_t)s * d + c];
  }
  if (dxs) v += dxs[i];
  dx[i] = v;
}

}  // namespace

cudaError_t launch_expert_bwd_f32(const moe_config_t& c, const float* xd, const int32_t* off,
                                  int64_t rows_bound, const float* W1, const float* W3,
                                  const float* b1, const float* W2, const float* dY,
                                  const float* h, float* pre, float* dh, float* dact, float* dxd,
                                  float* dW1, float* dW3, float* dW2, float* db1, float* db2,
                                  cudaStream_t s) {
  const bool swiglu = c.act == MOE_ACT_SWIGLU;
  const int E = c.E, d = c.d, H = c.H, Hp = swiglu ? 2 * H : H;
  const int64_t Hd = (int64_t)H * d;
  cudaError_t e = cudaSuccess;
  // pre-activations: u = xd W1_e^T + b1_e, or [a | v] = [xd W1_e^T | xd W3_e^T]
  for (int part = 0; part < (swiglu ? 2 : 1) && e == cudaSuccess; ++part) {
    GemmF32 g = {};
    g.A = xd; g.sam = d; g.sak = 1;
    g.B = part == 0 ? W1 : W3; g.sbk = 1; g.sbn = d; g.sbg = Hd;
    g.C = pre + part * H; g.scm = Hp; g.scn = 1;
    g.bias = (!swiglu && b1) ? b1 : nullptr; g.sbias = H;
    g.M = 0; g.N = H; g.K = d; g.G = E; g.off = off;
    e = launch_gemm_f32(g, kRowsM, rows_bound, s);
  }
  // dh = dY W2_e  (W2_e [d, H])
  if (e == cudaSuccess) {
    GemmF32 g = {};
    g.A = dY; g.sam = d; g.sak = 1;
    g.B = W2; g.sbk = H; g.sbn = 1; g.sbg = Hd;
    g.C = dh; g.scm = H; g.scn = 1;
    g.N = H; g.K = d; g.G = E; g.off = off;
    e = launch_gemm_f32(g, kRowsM, rows_bound, s);
  }
  if (e == cudaSuccess) {
    bwdf_act_kernel<<<592, 256, 0, s>>>(pre, dh, H, swiglu ? 1 : 0, off, E, dact);
    e = cudaGetLastError();
  }
  // dxd = du W1_e (+ dv W3_e)
  for (int part = 0; part < (swiglu ? 2 : 1) && e == cudaSuccess; ++part) {
    GemmF32 g = {};
    g.A = dact + part * H; g.sam = Hp; g.sak = 1;
    g.B = part == 0 ? W1 : W3; g.sbk = d; g.sbn = 1; g.sbg = Hd;
    g.C = dxd; g.scm = d; g.scn = 1;
    g.N = d; g.K = H; g.G = E; g.off = off; g.accumulate = part;
    e = launch_gemm_f32(g, kRowsM, rows_bound, s);
  }
  // dW2_e [d, H] = dY^T h
  if (e == cudaSuccess) {
    GemmF32 g = {};
    g.A = dY; g.sam = 1; g.sak = d;
    g.B = h; g.sbk = H; g.sbn = 1;
    g.C = dW2; g.scm = H; g.scn = 1; g.scg = Hd;
    g.M = d; g.N = H; g.G = E; g.off = off;
    e = launch_gemm_f32(g, kRowsK, rows_bound, s);
  }
  // dW1_e [H, d] = du^T xd (dW3_e = dv^T xd)
  for (int part = 0; part < (swiglu ? 2 : 1) && e == cudaSuccess; ++part) {
    GemmF32 g = {};
    g.A = dact + part * H; g.sam = 1; g.sak = Hp;
    g.B = xd; g.sbk = d; g.sbn = 1;
    g.C = part == 0 ? dW1 : dW3; g.scm = d; g.scn = 1; g.scg = Hd;
    g.M = H; g.N = d; g.G = E; g.off = off;
    e = launch_gemm_f32(g, kRowsK, rows_bound, s);
  }
  if (e == cudaSuccess && db1) e = launch_colsum_f32(dact, Hp, H, off, E, db1, s);
  if (e == cudaSuccess && db2) e = launch_colsum_f32(dY, d, d, off, E, db2, s);
  return e;
}

cudaError_t launch_bwdf_combine(const moe_config_t& c, const float* dy, const float* Y,
                                const int32_t* slot_of, const float* gate, float* dY, float* dg,
                                cudaStream_t s) {
  const int64_t warps = (int64_t)c.T * c.k;
  bwdf_combine_kernel<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, s>>>(
      dy, Y, slot_of, gate, c.T, c.k, c.d, max_rows(c), dY, dg);
  return cudaGetLastError();
}

// dWg = dz^T x, dx_r = dz Wg, db = sum_t dz_t (one group of all T rows)
cudaError_t launch_router_grads_f32(const moe_config_t& c, const float* dz, const float* x,
                                    const float* Wg, const int32_t* one_group_off, float* dWg,
                                    float* dbias, float* dxr, cudaStream_t s) {
  const int T = c.T, E = c.E, d = c.d;
  GemmF32 g = {};
  g.A = dz; g.sam = 1; g.sak = E;
  g.B = x; g.sbk = d; g.sbn = 1;
  g.C = dWg; g.scm = d; g.scn = 1;
  g.M = E; g.N = d; g.K = T; g.G = 1;
  cudaError_t e = launch_gemm_f32(g, kOne, 0, s);
  if (e == cudaSuccess) {
    GemmF32 r = {};
    r.A = dz; r.sam = E; r.sak = 1;
    r.B = Wg; r.sbk = d; r.sbn = 1;
    r.C = dxr; r.scm = d; r.scn = 1;
    r.M = T; r.N = d; r.K = E; r.G = 1;
    e = launch_gemm_f32(r, kOne, 0, s);
  }
  if (e == cudaSuccess && dbias) e = launch_colsum_f32(dz, E, E, one_group_off, 1, dbias, s);
  return e;
}

cudaError_t launch_bwdf_dx(const moe_config_t& c, const float* dxr, const float* dxd,
                           const float* dxs, const int32_t* slot_of, float* dx, cudaStream_t s) {
  const int64_t n = (int64_t)c.T * c.d;
  bwdf_dx_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(dxr, dxd, dxs, slot_of, c.T, c.k,
                                                            c.d, max_rows(c), dx);
  return cudaGetLastError();
}

}  // namespace moe
