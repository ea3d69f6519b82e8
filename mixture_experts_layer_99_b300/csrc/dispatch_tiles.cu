// Dispatch and load-balance statistics fed by the tensor-core router, in one
// kernel with one block per router tile (at most 128 tokens, a multiple of 8).
// The statistics are summed in fp32 in fixed orders (pairwise trees and
// butterflies): B300's fp64 rate is a small fraction of its fp32 rate, and
// the fp64 form of these sums kept the kernel's block 0 busy for about 10 us.
//
// The router already counted, for every tile, how many of the tile's slots
// chose each expert, and summed p per expert per CTA. From those each block
// derives the slots of every expert in earlier tiles (its base) and in total,
// the offsets offset_e = sum_{e'<e} min(count_e', C), and the stable position
// of each of its slots: base + earlier slots of the tile with the same expert
// (token order, the stable sort of the kwkr.cn MoE article, "MoE sparse
// activation: from the math to the code", section 3.2); a slot is kept iff its
// position < C (section 2.3). Block 0 also writes the statistics
// f_e = count_e/(kT), P_e = (sum p)/T, L_balance = E sum_e f_e P_e and the
// number of dropped slots (sections 2.2 and 6.2).
#include "moe_internal.h"

namespace moe {
namespace {

// Rounds of 32 slots a warp owns: 128 / 8 tokens of k <= 8 slots.
constexpr int kIdsPerLane = 4;
static_assert(kRouterTcTile / 8 * kMaxK <= 32 * kIdsPerLane, "slots per warp");

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// One block of 256 threads per router tile of `rows` tokens.
//  1. tot[e] = slots of e in all tiles, base[e] = slots of e in earlier tiles:
//     the router's [tiles, E] counts are read as C = E/V columns of V-int
//     vectors (V = 4 if E is a multiple of 4, else 1); thread (g, col) sums
//     column col over every G-th tile (G = 256 / C), sixteen independent loads
//     per round; then R threads per expert add the G partials of the expert
//     and combine theirs with shuffles (integer sums, so the order is
//     immaterial);
//  2. offset_e = sum_{e'<e} min(tot_e', C);
//  3. block 0 writes counts, offsets and the statistics;
//  4. stable positions: warp w owns tokens [w rows/8, (w+1) rows/8) of the
//     tile (rows/8 k consecutive slots), counts them per expert, and walks them
//     32 at a time in token order; slot (t, j) is kept iff its position < C.
// With zero_y (k = 1 only) the y row of every token whose slot was dropped is
// cleared, because GEMM2 then writes y only for kept tokens.
__global__ void __launch_bounds__(256) dispatch_tiles_kernel(
    const int32_t* __restrict__ idx, int T, int k, int E, int C, int rows,
    const int32_t* __restrict__ tile_hist, int ntiles, const float* __restrict__ partial,
    int nparts, int32_t* __restrict__ count, int32_t* __restrict__ offset,
    int32_t* __restrict__ slot_of, int32_t* __restrict__ token_of_row,
    float* __restrict__ prob_sum, float* __restrict__ f, float* __restrict__ P,
    float* __restrict__ Lb, int32_t* __restrict__ dropped, uint4* __restrict__ zero_y,
    int y_vec16, int64_t rows_cap, int32_t* __restrict__ chk) {
  __shared__ int tot[kMaxE], base[kMaxE], offs[kMaxE + 1];
  __shared__ int wcnt[8][kMaxE];
  __shared__ float psum[kMaxE];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int tile = blockIdx.x;
  for (int i = tid; i < 8 * kMaxE; i += 256) (&wcnt[0][0])[i] = 0;
  pdl_wait();
  // this warp's slots of the tile: rows/8 tokens (rows <= 128), k slots each,
  // at most kIdsPerLane rounds of 32. Their expert ids are loaded now, so that
  // the loads overlap the tile-count sums instead of following them.
  const int64_t nslots = (int64_t)T * k;
  const int wrows = rows / 8;                                   // tokens per warp
  const int64_t s0 = ((int64_t)tile * rows + (int64_t)wrows * w) * k;  // first slot of this warp
  const int per_warp = wrows * k;
  int ids[kIdsPerLane];
#pragma unroll
  for (int r = 0; r < kIdsPerLane; ++r) {
    const int64_t s = s0 + 32 * r + lane;
    ids[r] = (32 * r + lane < per_warp && s < nslots) ? idx[s] : -1;
  }
  {
    // partial sums per (group g, expert e) into wcnt, as [2][G][E] ints
    // (G E <= 1024), then tot/base per expert
    const int V = (E & 3) == 0 ? 4 : 1;
    const int ncol = E / V;
    const int G = 256 / ncol;
    int* ptot = &wcnt[0][0];
    int* pbase = ptot + 1024;
    if (tid < G * ncol) {
      const int col = tid % ncol, g = tid / ncol;
      int st[4] = {0, 0, 0, 0}, sb[4] = {0, 0, 0, 0};
      for (int tt0 = g; tt0 < ntiles; tt0 += 16 * G) {
        int4 v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int tt = tt0 + i * G;
          v[i] = make_int4(0, 0, 0, 0);
          if (tt < ntiles) {
            if (V == 4)
              v[i] = __ldg(reinterpret_cast<const int4*>(tile_hist + (size_t)tt * E) + col);
            else
              v[i].x = __ldg(tile_hist + (size_t)tt * E + col);
          }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const bool before = tt0 + i * G < tile;
          st[0] += v[i].x;
          st[1] += v[i].y;
          st[2] += v[i].z;
          st[3] += v[i].w;
          if (before) {
            sb[0] += v[i].x;
            sb[1] += v[i].y;
            sb[2] += v[i].z;
            sb[3] += v[i].w;
          }
        }
      }
      for (int i = 0; i < V; ++i) {
        ptot[g * E + col * V + i] = st[i];
        pbase[g * E + col * V + i] = sb[i];
      }
    }
    __syncthreads();
    // R threads per expert (R a power of two, R E <= 256, R <= 32: the R
    // threads of an expert are neighbouring lanes of one warp)
    int R = 32;
    while (R * E > 256) R >>= 1;
    {
      const int e = tid / R, sub = tid % R;
      int st = 0, sb = 0;
      if (e < E) {
        for (int g = sub; g < G; g += R) {
          st += ptot[g * E + e];
          sb += pbase[g * E + e];
        }
      }
      for (int o = 1; o < R; o <<= 1) {
        st += __shfl_xor_sync(0xffffffffu, st, o);
        sb += __shfl_xor_sync(0xffffffffu, sb, o);
      }
      if (e < E && sub == 0) {
        tot[e] = st;
        base[e] = sb;
      }
    }
    __syncthreads();
    for (int i = tid; i < 2 * 1024; i += 256) (&wcnt[0][0])[i] = 0;
  }
  __syncthreads();
  if (w == 0) {
    int run = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int kept = e < E ? min(tot[e], C) : 0;
      const int incl = warp_incl_scan(kept, lane);
      if (e < E) offs[e] = run + incl - kept;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) offs[E] = run;
  }
  if (tile == 0) {
    // probability sums per expert: R neighbouring threads per expert (R as
    // above), thread sub adding partials sub, sub + R, ... in that order (the
    // loads of every expert in flight together, eight per round), then a fixed
    // butterfly over the R threads
    int R = 32;
    while (R * E > 256) R >>= 1;
    const int e = tid / R, sub = tid % R;
    float sp = 0.f;
    if (e < E) {
      for (int b0 = sub; b0 < nparts; b0 += 8 * R) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int b = b0 + i * R;
          v[i] = b < nparts ? __ldg(partial + (size_t)b * E + e) : 0.f;
        }
        // the eight as a pairwise tree, then into the running sum
        sp += ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
      }
    }
    for (int o = 1; o < R; o <<= 1) sp += __shfl_xor_sync(0xffffffffu, sp, o);
    if (e < E && sub == 0) psum[e] = sp;
  }
  __syncthreads();
  if (tile == 0) {
    for (int e = tid; e <= E; e += 256) offset[e] = offs[e];
    if (w == 0) {
      const float kT = (float)((long long)k * T), fT = (float)T;
      float fp = 0.f;
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        if (e < E) {
          count[e] = tot[e];
          const float fe = (float)tot[e] / kT;
          const float Pe = psum[e] / fT;
          if (f) f[e] = fe;
          if (P) P[e] = Pe;
          if (prob_sum) prob_sum[e] = psum[e];
          fp = fmaf(fe, Pe, fp);
        }
      }
      fp = warp_sum_f(fp);
      if (lane == 0) {
        if (Lb) Lb[0] = (float)E * fp;
        if (dropped) dropped[0] = (int32_t)((long long)k * T - offs[E]);
      }
    }
  }
  // ---- stable positions within the tile
#pragma unroll
  for (int r = 0; r < kIdsPerLane; ++r) {
    const int e = ids[r];
    if ((unsigned)e < (unsigned)E) atomicAdd(&wcnt[w][e], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += 256) {
    int run = base[e];
#pragma unroll
    for (int ww = 0; ww < 8; ++ww) {
      const int cc = wcnt[ww][e];
      wcnt[ww][e] = run;
      run += cc;
    }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int r = 0; r < kIdsPerLane; ++r) {
    const int c = 32 * r;
    if (c >= per_warp) break;
    const int64_t s = s0 + c + lane;
    const bool in = (c + lane < per_warp) && s < nslots;
    int e = in ? ids[r] : -1;
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
        if (moe_check(row < rows_cap, chk, 53)) token_of_row[row] = (int32_t)(s / k);
        else row = -1;
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
                                        int nparts, int32_t* count, int32_t* offset,
                                        int32_t* slot_of, int32_t* token_of_row,
                                        float* prob_sum, float* f, float* P, float* Lb,
                                        int32_t* dropped, void* zero_y, cudaStream_t s,
                                        int32_t* chk) {
  const int ntiles = router_tc_tiles(c);
  const int y_vec16 = (int)((size_t)c.d * elem_bytes(c) / 16);
  return launch_pdl(dispatch_tiles_kernel, dim3(ntiles), dim3(256), 0, s, idx, c.T, c.k, c.E,
                    c.capacity, router_tc_rows(c), tile_hist, ntiles, partial, nparts, count,
                    offset, slot_of,
                    token_of_row, prob_sum, f, P, Lb, dropped,
                    c.k == 1 ? static_cast<uint4*>(zero_y) : (uint4*)nullptr, y_vec16,
                    max_rows(c), chk);
}

}  // namespace moe
