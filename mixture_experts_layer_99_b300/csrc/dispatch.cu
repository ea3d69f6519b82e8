// Capacity-limited dispatch: per-expert counts, token-order positions, drops
// beyond the capacity C, and the gather of kept rows into an
// expert-contiguous buffer.
//
// Follows the kwkr.cn MoE article ("MoE sparse activation: from the math to
// the code"), section 2.3 (capacity C, overflow tokens dropped) and section
// 3.2 (slots flattened token-major and grouped by expert with a stable sort,
// so lower tokens come first). Here the stable sort is replaced by counting:
// a per-block histogram, a scan over blocks, and a stable in-block rank, which
// gives the same positions with integer arithmetic only.
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int SPB = kDispSlotsPerBlock;
constexpr int NT = 256;
constexpr int NW = NT / 32;
constexpr int SPW = SPB / NW;  // slots per warp (128)

// hist[b, e] = number of slots of block b that chose expert e. An expert
// id outside [0, E) (a caller's input) counts for no expert, its slot gets
// row -1, and with a status header it is recorded as MOE_ERR_INVALID_ARG
// (where = 41).
__global__ void __launch_bounds__(NT) disp_count_kernel(const int32_t* __restrict__ idx,
                                                        int64_t nslots, int E,
                                                        int32_t* __restrict__ hist,
                                                        int32_t* __restrict__ hdr) {
  __shared__ int h[kMaxE];
  for (int e = threadIdx.x; e < E; e += NT) h[e] = 0;
  __syncthreads();
  const int64_t s0 = (int64_t)blockIdx.x * SPB;
  bool bad = false;
  for (int i = threadIdx.x; i < SPB; i += NT) {
    const int64_t s = s0 + i;
    if (s < nslots) {
      const int e = idx[s];
      if ((unsigned)e < (unsigned)E) atomicAdd(&h[e], 1);
      else bad = true;
    }
  }
  if (bad && hdr != nullptr && atomicCAS(hdr + kHdrStatus, 0, (int)MOE_ERR_INVALID_ARG) == 0)
    atomicExch(hdr + kHdrWhere, 41);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += NT) hist[(size_t)blockIdx.x * E + e] = h[e];
}

// base[b, e] = sum_{b' < b} hist[b', e]; count[e] = total; offset = exclusive
// scan of min(count, C). One block of 1024 threads, one warp per expert.
__global__ void __launch_bounds__(1024) disp_scan_kernel(const int32_t* __restrict__ hist,
                                                         int nblk, int E, int C,
                                                         int32_t* __restrict__ base,
                                                         int32_t* __restrict__ count,
                                                         int32_t* __restrict__ offset) {
  __shared__ int cnt[kMaxE];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int e = w; e < E; e += 32) {
    int run = 0;
    for (int b0 = 0; b0 < nblk; b0 += 32) {
      const int b = b0 + lane;
      const int v = b < nblk ? hist[(size_t)b * E + e] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (b < nblk) base[(size_t)b * E + e] = run + incl - v;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) cnt[e] = run;
  }
  __syncthreads();
  if (w == 0) {
    int run = 0;
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
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) offset[E] = run;
  }
}

// Stable positions: pos(s) = base[b, e] + (slots of e earlier in block b).
// Each warp owns SPW consecutive slots and walks them 32 at a time in order.
__global__ void __launch_bounds__(NT) disp_assign_kernel(
    const int32_t* __restrict__ idx, int64_t nslots, int k, int E, int C,
    const int32_t* __restrict__ base, const int32_t* __restrict__ offset,
    int32_t* __restrict__ slot_of, int32_t* __restrict__ token_of_row, int64_t rows_cap,
    int32_t* __restrict__ chk) {
  __shared__ int wcnt[NW][kMaxE];
  __shared__ int offs[kMaxE];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < NW * kMaxE; i += NT) (&wcnt[0][0])[i] = 0;
  for (int e = threadIdx.x; e < E; e += NT) offs[e] = offset[e];
  __syncthreads();
  const int64_t sw = (int64_t)blockIdx.x * SPB + (int64_t)w * SPW;
  for (int step = 0; step < SPW / 32; ++step) {
    const int64_t s = sw + step * 32 + lane;
    const int e = s < nslots ? idx[s] : -1;
    if ((unsigned)e < (unsigned)E) atomicAdd(&wcnt[w][e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += NT) {
    int run = base[(size_t)blockIdx.x * E + e];
    for (int ww = 0; ww < NW; ++ww) {
      const int c = wcnt[ww][e];
      wcnt[ww][e] = run;
      run += c;
    }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  for (int step = 0; step < SPW / 32; ++step) {
    const int64_t s = sw + step * 32 + lane;
    int e = s < nslots ? idx[s] : -1;
    const bool valid = (unsigned)e < (unsigned)E;
    if (!valid) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt);
    const int pos = valid ? wcnt[w][e] + rank : 0;
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) wcnt[w][e] += __popc(peers);
    __syncwarp();
    if (s < nslots) {
      int32_t row = -1;
      if (valid && pos < C) {
        row = offs[e] + pos;
        if (moe_check(row < rows_cap, chk, 53)) token_of_row[row] = (int32_t)(s / k);
        else row = -1;
      }
      slot_of[s] = row;
    }
  }
}

// xd[row] = x[token_of_row[row]] for row < offset[E]; one warp per row,
// 16-byte vectors.
__global__ void __launch_bounds__(NT) disp_gather_kernel(const uint4* __restrict__ x,
                                                         const int32_t* __restrict__ token_of_row,
                                                         const int32_t* __restrict__ offset,
                                                         int E, int nvec,
                                                         uint4* __restrict__ xd, int T,
                                                         int32_t* __restrict__ chk) {
  pdl_wait();
  const int nrows = offset[E];
  const int row = blockIdx.x * NW + (threadIdx.x >> 5);
  if (row >= nrows) return;
  const int t = token_of_row[row];
  if (!moe_check((unsigned)t < (unsigned)T, chk, 51)) return;
  const uint4* src = x + (size_t)t * nvec;
  uint4* dst = xd + (size_t)row * nvec;
  for (int v = threadIdx.x & 31; v < nvec; v += 32) dst[v] = __ldg(src + v);
}

}  // namespace

cudaError_t launch_gather(const moe_config_t& c, const void* x, const int32_t* token_of_row,
                          const int32_t* offset, void* xd, int64_t rows_bound, cudaStream_t s,
                          int32_t* chk) {
  const int nvec = (int)((size_t)c.d * elem_bytes(c) / 16);
  const int64_t gblk = (rows_bound + NW - 1) / NW;
  if (gblk <= 0) return cudaSuccess;
  return launch_pdl(disp_gather_kernel, dim3((unsigned)gblk), dim3(NT), 0, s,
                    static_cast<const uint4*>(x), token_of_row, offset, c.E, nvec,
                    static_cast<uint4*>(xd), c.T, chk);
}

cudaError_t launch_dispatch(const moe_config_t& c, const int32_t* idx, const void* x,
                            int32_t* count, int32_t* offset, int32_t* slot_of,
                            int32_t* token_of_row, void* xd, int32_t* hist, int32_t* base,
                            int64_t rows_bound, cudaStream_t s, int32_t* hdr) {
  const int64_t nslots = (int64_t)c.T * c.k;
  const int nblk = disp_blocks(c);
  disp_count_kernel<<<nblk, NT, 0, s>>>(idx, nslots, c.E, hist, hdr);
  disp_scan_kernel<<<1, 1024, 0, s>>>(hist, nblk, c.E, c.capacity, base, count, offset);
  disp_assign_kernel<<<nblk, NT, 0, s>>>(idx, nslots, c.k, c.E, c.capacity, base, offset,
                                         slot_of, token_of_row, rows_bound, hdr);
  const int nvec = (int)((size_t)c.d * elem_bytes(c) / 16);
  const int64_t gblk = (rows_bound + NW - 1) / NW;
  if (gblk > 0)
    disp_gather_kernel<<<(unsigned)gblk, NT, 0, s>>>(static_cast<const uint4*>(x),
                                                     token_of_row, offset, c.E, nvec,
                                                     static_cast<uint4*>(xd), c.T, hdr);
  return cudaGetLastError();
}

}  // namespace moe
