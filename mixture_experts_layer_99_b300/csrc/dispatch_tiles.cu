// Dispatch and load-balance statistics fed by the tensor-core router.
//
// The router already counted, for every 128-token tile, how many of the
// tile's slots chose each expert, and summed p per expert per CTA. From those:
//   scan_stats: one block. base[tile, e] = slots of e in earlier tiles;
//               count_e; offset_e = sum_{e'<e} min(count_e', C); and the
//               statistics f_e = count_e/(kT), P_e = (sum p)/T,
//               L_balance = E sum_e f_e P_e, dropped = kT - sum_e min(count_e, C)
//               (kwkr.cn MoE article, "MoE sparse activation: from the math
//               to the code", sections 2.2, 2.3 and 6.2).
//   assign:     one block per tile. The stable position of slot (t, j) among
//               the slots that chose the same expert is base + the number of
//               earlier slots of the tile with that expert (token order, the
//               stable sort of the article's section 3.2); kept iff < C.
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int TILE = kRouterTcTile;  // tokens per tile (128)

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(1024) scan_stats_kernel(
    const int32_t* __restrict__ tile_hist, int ntiles, const float* __restrict__ partial,
    int nparts, int T, int E, int k, int C, int32_t* __restrict__ base,
    int32_t* __restrict__ count, int32_t* __restrict__ offset, float* __restrict__ prob_sum,
    float* __restrict__ f, float* __restrict__ P, float* __restrict__ Lb,
    int32_t* __restrict__ dropped) {
  __shared__ int cnt[kMaxE];
  __shared__ double psum[kMaxE];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int e = w; e < E; e += 32) {
    int run = 0;
    for (int b0 = 0; b0 < ntiles; b0 += 32) {
      const int b = b0 + lane;
      const int v = b < ntiles ? tile_hist[(size_t)b * E + e] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (b < ntiles) base[(size_t)b * E + e] = run + incl - v;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    double s = 0.0;
    for (int b = lane; b < nparts; b += 32) s += (double)partial[(size_t)b * E + e];
    s = warp_sum_d(s);
    if (lane == 0) {
      cnt[e] = run;
      psum[e] = s;
    }
  }
  __syncthreads();
  if (w == 0) {
    int run = 0;
    double fp = 0.0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int ce = e < E ? cnt[e] : 0;
      const int kept = ce < C ? ce : C;
      int incl = kept;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (e < E) {
        count[e] = ce;
        offset[e] = run + incl - kept;
        const double fe = (double)ce / ((double)k * (double)T);
        const double Pe = psum[e] / (double)T;
        if (f) f[e] = (float)fe;
        if (P) P[e] = (float)Pe;
        if (prob_sum) prob_sum[e] = (float)psum[e];
        fp += fe * Pe;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    fp = warp_sum_d(fp);
    if (lane == 0) {
      offset[E] = run;
      if (Lb) Lb[0] = (float)((double)E * fp);
      if (dropped) dropped[0] = (int32_t)((long long)k * T - run);
    }
  }
}

// One block of 256 threads per 128-token tile; warp w owns tokens
// [16w, 16w + 16) of the tile, i.e. 16k consecutive slots, walked 32 at a time.
// With zero_y (k = 1 only), the y row of every token whose slot was dropped
// is cleared here, because the expert FFN then writes y only for kept tokens.
__global__ void __launch_bounds__(256) assign_tiles_kernel(
    const int32_t* __restrict__ idx, int T, int k, int E, int C,
    const int32_t* __restrict__ base, const int32_t* __restrict__ offset,
    int32_t* __restrict__ slot_of, int32_t* __restrict__ token_of_row,
    uint4* __restrict__ zero_y, int y_vec16) {
  __shared__ int wcnt[8][kMaxE];
  __shared__ int offs[kMaxE];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int tile = blockIdx.x;
  for (int i = threadIdx.x; i < 8 * kMaxE; i += 256) (&wcnt[0][0])[i] = 0;
  for (int e = threadIdx.x; e < E; e += 256) offs[e] = offset[e];
  __syncthreads();
  const int64_t nslots = (int64_t)T * k;
  const int64_t s0 = ((int64_t)tile * TILE + 16 * w) * k;  // first slot of this warp
  const int per_warp = 16 * k;
  for (int c = 0; c < per_warp; c += 32) {
    const int64_t s = s0 + c + lane;
    const bool in = (c + lane < per_warp) && s < nslots;
    const int e = in ? idx[s] : -1;
    if ((unsigned)e < (unsigned)E) atomicAdd(&wcnt[w][e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += 256) {
    int run = base[(size_t)tile * E + e];
#pragma unroll
    for (int ww = 0; ww < 8; ++ww) {
      const int cc = wcnt[ww][e];
      wcnt[ww][e] = run;
      run += cc;
    }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  for (int c = 0; c < per_warp; c += 32) {
    const int64_t s = s0 + c + lane;
    const bool in = (c + lane < per_warp) && s < nslots;
    int e = in ? idx[s] : -1;
    const bool valid = (unsigned)e < (unsigned)E;
    if (!valid) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt);
    const int pos = valid ? wcnt[w][e] + rank : 0;
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) wcnt[w][e] += __popc(peers);
    __syncwarp();
    int32_t row = -1;
    if (in) {
      if (valid && pos < C) {
        row = offs[e] + pos;
        token_of_row[row] = (int32_t)(s / k);
      }
      slot_of[s] = row;
    }
    if (zero_y) {
      unsigned drop = __ballot_sync(0xffffffffu, in && row < 0);
      while (drop) {
        const int l = __ffs(drop) - 1;
        drop &= drop - 1;
        const int64_t t = s0 + c + l;  // k = 1: slot index = token index
        uint4* yr = zero_y + (size_t)t * y_vec16;
        for (int v = lane; v < y_vec16; v += 32) yr[v] = make_uint4(0, 0, 0, 0);
      }
    }
  }
}

}  // namespace

cudaError_t launch_dispatch_from_router(const moe_config_t& c, const int32_t* idx,
                                        const int32_t* tile_hist, const float* partial,
                                        int nparts, int32_t* base, int32_t* count,
                                        int32_t* offset, int32_t* slot_of,
                                        int32_t* token_of_row, float* prob_sum, float* f,
                                        float* P, float* Lb, int32_t* dropped,
                                        void* zero_y, cudaStream_t s) {
  const int ntiles = router_tc_tiles(c);
  scan_stats_kernel<<<1, 1024, 0, s>>>(tile_hist, ntiles, partial, nparts, c.T, c.E, c.k,
                                       c.capacity, base, count, offset, prob_sum, f, P, Lb,
                                       dropped);
  const int y_vec16 = (int)((size_t)c.d * elem_bytes(c) / 16);
  assign_tiles_kernel<<<ntiles, 256, 0, s>>>(idx, c.T, c.k, c.E, c.capacity, base, offset,
                                             slot_of, token_of_row,
                                             c.k == 1 ? static_cast<uint4*>(zero_y) : nullptr,
                                             y_vec16);
  return cudaGetLastError();
}

}  // namespace moe
