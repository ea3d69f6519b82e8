// Gate-weighted combine and load-balance statistics.
//
// Combine: y_t = sum_{j: slot_of[t,j] >= 0} g[t,j] Y[slot_of[t,j]], summed in
// fp32 in slot order j = 0..k-1 (deterministic: each output element is summed
// by one thread, no atomics); y_t = 0 when every slot of t was dropped. This is the
// output y = sum_{i in K(x)} g_i(x) E_i(x) of the kwkr.cn MoE article, section
// 2.1, with the masking of dropped tokens from section 2.3.
//
// Statistics (section 2.2 of the same article): f_i = count_i/(kT),
// P_i = (1/T) sum_t p[t,i], L_balance = E sum_i f_i P_i, and the number of
// dropped slots (the drop-rate diagnostic of section 6.2).
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int NT = 256, NW = NT / 32;

__device__ __forceinline__ void unpack(const uint4& u, float (&f)[8], __nv_bfloat16*) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ void unpack(const uint4& u, float (&f)[8], float*) {
  f[0] = __uint_as_float(u.x);
  f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z);
  f[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ uint4 pack(const float (&f)[8], __nv_bfloat16*) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}
__device__ __forceinline__ uint4 pack(const float (&f)[8], float*) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                    __float_as_uint(f[3]));
}

// base (optional, [T, d]): each token's sum starts from its base row (the
// shared expert's output) instead of zero.
// Warp w of block (bx, by) owns token bx * NW + w and the row chunk by of
// 32 UNR 16-byte vectors (32 lanes x UNR vectors each): a row is split over
// several warps so that a small batch still fills the GPU. Each lane issues
// all of its loads (UNR vectors of each of the k slots) before it sums them:
// a dropped slot loads the vectors of the token's first kept slot (the same
// lines, so they come from the cache) and adds nothing, which keeps every
// load unconditional and in flight together. A token without a kept slot
// writes its base row, or zeros.
// Two vectors per lane and slot for k <= 2: measured on B300 (layer call,
// alternating builds, identical outputs) the combine took 50.8 us on the long
// tail and 72.3 us on mixtral with two, 55.5 / 77.7 us with four, 54 / 78 us
// with one and 77 / 110 us with eight.
template <int KM>
struct CombineShape {
  static constexpr int UNR = KM <= 2 ? 2 : (KM <= 4 ? 2 : 1);
  static constexpr int CHUNK = 32 * UNR;
};
template <typename T, int KM>
__global__ void __launch_bounds__(NT) combine_kernel(const uint4* __restrict__ Y,
                                                     const int32_t* __restrict__ slot_of,
                                                     const float* __restrict__ gate, int T_,
                                                     int k, int nvec, uint4* __restrict__ y,
                                                     const uint4* __restrict__ base,
                                                     int64_t rows_cap, int32_t* __restrict__ chk) {
  constexpr int V = 16 / sizeof(T);
  constexpr int UNR = CombineShape<KM>::UNR;
  pdl_wait();
  const int t = blockIdx.x * NW + (threadIdx.x >> 5);
  if (t >= T_) return;
  const int lane = threadIdx.x & 31;
  int sl[KM];
  float g[KM];
  int first = -1;
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    sl[j] = j < k ? slot_of[(size_t)t * k + j] : -1;
    if (!moe_check(sl[j] < rows_cap, chk, 52)) sl[j] = -1;
    g[j] = j < k ? gate[(size_t)t * k + j] : 0.f;
    if (first < 0 && sl[j] >= 0) first = sl[j];
  }
  const int v0 = blockIdx.y * CombineShape<KM>::CHUNK + lane;
  float acc[UNR][8];
#pragma unroll
  for (int u = 0; u < UNR; ++u) {
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
  }
  if (base) {
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int v = v0 + 32 * u;
      if (v < nvec) unpack(__ldg(base + (size_t)t * nvec + v), acc[u], (T*)nullptr);
    }
  }
  if (first >= 0) {  // the same for the whole warp (one token)
    uint4 q[KM][UNR];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      const size_t row = (size_t)(sl[j] >= 0 ? sl[j] : first);
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int v = v0 + 32 * u;
        q[j][u] = (j < k && v < nvec) ? __ldg(Y + row * nvec + v) : make_uint4(0, 0, 0, 0);
      }
    }
    // slot order j = 0..k-1 for every vector: the same fp32 sum order as one
    // warp walking the row
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (sl[j] < 0) continue;
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        float f[8];
        unpack(q[j][u], f, (T*)nullptr);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[u][i] = fmaf(g[j], f[i], acc[u][i]);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < UNR; ++u) {
    const int v = v0 + 32 * u;
    if (v < nvec) y[(size_t)t * nvec + v] = pack(acc[u], (T*)nullptr);
  }
}

// One block. prob_sum is used if given, else the router's per-block partials
// are reduced here in a fixed order.
__global__ void __launch_bounds__(NT) aux_kernel(const int32_t* __restrict__ count,
                                                 const float* __restrict__ prob_sum,
                                                 const float* __restrict__ partial, int nparts,
                                                 int T_, int E, int k, int C,
                                                 float* __restrict__ f, float* __restrict__ P,
                                                 float* __restrict__ L,
                                                 int32_t* __restrict__ dropped) {
  __shared__ double sfp[NT];
  __shared__ long long skept[NT];
  double fp = 0.0;
  long long kept = 0;
  for (int e = threadIdx.x; e < E; e += NT) {
    double ps;
    if (prob_sum) {
      ps = (double)prob_sum[e];
    } else {
      ps = 0.0;
      for (int b = 0; b < nparts; ++b) ps += (double)partial[(size_t)b * E + e];
    }
    const int ce = count[e];
    const double fe = (double)ce / ((double)k * (double)T_);
    const double Pe = ps / (double)T_;
    if (f) f[e] = (float)fe;
    if (P) P[e] = (float)Pe;
    fp += fe * Pe;
    kept += ce < C ? ce : C;
  }
  sfp[threadIdx.x] = fp;
  skept[threadIdx.x] = kept;
  __syncthreads();
  for (int w = NT / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      sfp[threadIdx.x] += sfp[threadIdx.x + w];
      skept[threadIdx.x] += skept[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    if (L) L[0] = (float)((double)E * sfp[0]);
    if (dropped) dropped[0] = (int32_t)((long long)k * T_ - skept[0]);
  }
}

}  // namespace

template <int KM>
cudaError_t launch_combine_km(const moe_config_t& c, const uint4* Y, const int32_t* slot_of,
                              const float* gate, uint4* y, const uint4* b, cudaStream_t s,
                              int32_t* chk) {
  const int nvec = (int)((size_t)c.d * elem_bytes(c) / 16);
  constexpr int CHUNK = CombineShape<KM>::CHUNK;
  const dim3 grid((unsigned)((c.T + NW - 1) / NW), (unsigned)((nvec + CHUNK - 1) / CHUNK));
  if (c.dtype == MOE_F32)
    return launch_pdl(combine_kernel<float, KM>, grid, dim3(NT), 0, s, Y, slot_of, gate, c.T,
                      c.k, nvec, y, b, (int64_t)max_rows(c), chk);
  return launch_pdl(combine_kernel<__nv_bfloat16, KM>, grid, dim3(NT), 0, s, Y, slot_of, gate,
                    c.T, c.k, nvec, y, b, (int64_t)max_rows(c), chk);
}

cudaError_t launch_combine(const moe_config_t& c, const void* Y, const int32_t* slot_of,
                           const float* gate, void* y, cudaStream_t s, const void* base,
                           int32_t* chk) {
  const uint4* b = static_cast<const uint4*>(base);
  const uint4* Yv = static_cast<const uint4*>(Y);
  uint4* yv = static_cast<uint4*>(y);
  if (c.k <= 2) return launch_combine_km<2>(c, Yv, slot_of, gate, yv, b, s, chk);
  if (c.k <= 4) return launch_combine_km<4>(c, Yv, slot_of, gate, yv, b, s, chk);
  return launch_combine_km<kMaxK>(c, Yv, slot_of, gate, yv, b, s, chk);
}

// off[0] = 0, off[1] = rows: the one-group offsets of the shared expert.
__global__ void one_group_offsets_kernel(int32_t* off, int rows) {
  pdl_wait();
  off[0] = 0;
  off[1] = rows;
}

cudaError_t launch_one_group_offsets(int32_t* off, int rows, cudaStream_t s) {
  return launch_pdl(one_group_offsets_kernel, dim3(1), dim3(1), 0, s, off, rows);
}

cudaError_t launch_aux(const moe_config_t& c, const int32_t* count, const float* prob_sum,
                       const float* partial, int nparts, float* f, float* P, float* L,
                       int32_t* dropped, cudaStream_t s) {
  aux_kernel<<<1, NT, 0, s>>>(count, prob_sum, partial, nparts, c.T, c.E, c.k, c.capacity, f,
                              P, L, dropped);
  return cudaGetLastError();
}

}  // namespace moe
