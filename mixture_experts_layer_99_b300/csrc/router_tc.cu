// Fused router on the tcgen05 tensor cores for bf16 tokens and E <= 64.
//
// logits l = (x Wg^T + b + s g) / tau (s = 1, or a scale times the token's
// logit standard deviation: std-scaled noise, section 3.3 of the article
// below), softmax p = softmax(l), the k largest
// logits (descending, ties to the lower expert index), renormalised gates
// g_j = p_{K_j} / sum_m p_{K_m}, per-CTA sums of p for P_i and per-tile
// selection counts for the dispatch. This is the gate of the kwkr.cn MoE
// article ("MoE sparse activation: from the math to the code"), section 2.1,
// fused with softmax and top-k as its section 5.3 suggests; bias, noise and
// temperature as in the lpnh.cn MoE guide, section 3.3.
//
// The contraction x Wg^T (E tiny) is HBM-bound: the kernel streams 128-token
// tiles of x through TMA and issues one 128 x E_pad x 16 MMA per 16-wide K
// step into a TMEM accumulator row per token.
//   warp 0       TMA producer (x tile [128 x 64] + Wg tile [E_pad x 64])
//   warp 1       TMEM owner, MMA issuer
//   warps 2-17   epilogue, four threads per token: EP/16 groups of four warps
//                move the tile's logits from TMEM to shared memory (one row
//                per token; each group 16 of the EP columns), then each
//                token's four threads take a quarter of its experts each and
//                combine max, top-k and the softmax sum with shuffles
// When the batch has few 128-token tiles (e.g. a decode step of 64 tokens),
// the K range of each tile is split over a cluster of CTAs (SPLIT): each
// leaves its fp32 partial logits in its shared memory, and the cluster's
// first CTA reads them over distributed shared memory, sums them in split
// order and runs the same per-token epilogue.
#include "moe_internal.h"
#include "tc_ptx.cuh"

#include <math.h>
#include <mutex>

namespace moe {
namespace {

using namespace ptx;

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int TPT = 4;                         // epilogue threads per token
constexpr int EPI_THREADS = BM * TPT;          // 512
constexpr int NUM_THREADS = 64 + EPI_THREADS;  // + producer and MMA warps
constexpr int A_BYTES = BM * BK * 2;  // one 128 x 64 box of x
// Two 64-column boxes per pipeline stage, adjacent in K, so DRAM sees 256
// contiguous bytes of every row requested together. Measured on B300 against
// one box per stage: the mixtral router inside the layer 47.5 -> 44.0 us, the
// long-tail one equal; four boxes per stage left too few stages at E = 64
// (long tail 44 -> 53 us).
constexpr int NB = 2;

// Epilogue scratch: the tile's logits, then its probabilities, one row per
// token padded by four floats (16-byte rows whose banks shift by 4 or 20 from
// row to row, so the 16-byte row accesses are conflict-free), summed per
// expert down the columns.
constexpr int LPAD = 4;
template <int EP>
struct EpiSmem {
  alignas(16) float L[BM][EP + LPAD];
  alignas(16) float bias[EP];  // the router bias (0 past E, or without one)
  float part[EP];
  int hist[EP];
};

template <int EP>
struct RouterCfg {
  static constexpr int B_BYTES = EP * BK * 2;
  static constexpr int STAGE = NB * (A_BYTES + B_BYTES);
  // as many operand stages (at most 12) as fit beside the epilogue scratch
  static constexpr int FIT = (int)((220 * 1024 - sizeof(EpiSmem<EP>) - 1024 - 256) / STAGE);
  static constexpr int STAGES = FIT > 12 ? 12 : FIT;
  static constexpr int TCOLS = 2 * EP <= 32 ? 32 : (2 * EP <= 64 ? 64 : 128);
};

template <int EP>
struct RouterSmem {
  uint64_t full[RouterCfg<EP>::STAGES];
  uint64_t empty[RouterCfg<EP>::STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t final_bar;
  uint32_t tmem_base;
  int abort_flag;
  EpiSmem<EP> epi;
};

template <int EP>
constexpr size_t router_smem_bytes() {
  return 1024 + RouterCfg<EP>::STAGES * RouterCfg<EP>::STAGE + sizeof(RouterSmem<EP>);
}

__device__ __forceinline__ void epi_bar() {  // named barrier over the 16 epilogue warps
  asm volatile("bar.sync 1, %0;" ::"n"(EPI_THREADS) : "memory");
}
// The same barrier, returning whether any epilogue thread passed `fail`: one
// decision that every epilogue thread takes alike.
__device__ __forceinline__ bool epi_bar_or(bool fail) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)fail), "n"(EPI_THREADS)
      : "memory");
  return r != 0;
}

// Thread p's quarter of token r's row of the scratch (Q = EP/4 floats, a
// multiple of 4).
template <int EP>
__device__ __forceinline__ void load_quarter(const EpiSmem<EP>& es, int r, int p,
                                             float (&v)[EP / TPT]) {
  constexpr int Q = EP / TPT;
  const float4* row = reinterpret_cast<const float4*>(&es.L[r][p * Q]);
#pragma unroll
  for (int q = 0; q < Q; q += 4) {
    const float4 w = row[q / 4];
    v[q] = w.x;
    v[q + 1] = w.y;
    v[q + 2] = w.z;
    v[q + 3] = w.w;
  }
}

// Read-only loads issued where they stand: volatile asm stays in program
// order with the mbarrier waits (also volatile asm), so a load placed before
// a wait is in flight while the thread waits.
__device__ __forceinline__ float4 ld_nc_early_v4(const float* p) {
  float4 r;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ float ld_nc_early(const float* p) {
  float r;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(r) : "l"(p));
  return r;
}

// (value, expert) a ranks before b: larger value, ties to the lower index.
__device__ __forceinline__ bool ranks_before(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

// One token's four threads (lanes 4j..4j+3 of a warp; thread p owns experts
// [p Q, p Q + Q), Q = EP/4): keys, softmax, top-k (descending, ties to the
// lower index), gates, and the tile's per-expert selection counts and sums of
// p (fixed order). v holds the thread's Q raw logits on entry, or z + b + g
// when keys_done (the copy out of TMEM added bias and noise already).
template <int EP, int KM>
__device__ __forceinline__ void router_tile_epilogue(
    float (&v)[EP / TPT], bool keys_done, int tile, int tile_rows, int r, int p, int etid,
    const float* __restrict__ bias,
    const float* __restrict__ noise, float noise_scale, float tau, int T, int E, int k,
    float* __restrict__ logits, int32_t* __restrict__ idx, float* __restrict__ gate,
    int32_t* __restrict__ tile_hist, EpiSmem<EP>& es) {
  constexpr int Q = EP / TPT;
  const int t = tile * tile_rows + r;
  const bool valid = r < tile_rows && t < T;
  const int e0 = p * Q;
  // 16-byte vectors along rows of the [T, E] fp32 arrays when every row starts
  // on a 16-byte boundary
  const bool rows16 = (E & 3) == 0;
  const bool vec4n = rows16 && (reinterpret_cast<uintptr_t>(noise) & 15u) == 0;
  const bool vec4l = rows16 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0;
  // selection keys l = (z + b + s g) / tau (one reciprocal; tau = 1 leaves them as they are)
  if (valid && bias && !keys_done) {
    const float4* br = reinterpret_cast<const float4*>(&es.bias[e0]);
#pragma unroll
    for (int q = 0; q < Q; q += 4) {
      const float4 b4 = br[q / 4];
      v[q] += b4.x;
      v[q + 1] += b4.y;
      v[q + 2] += b4.z;
      v[q + 3] += b4.w;
    }
  }
  // noise strength: 1, or noise_scale times the population standard deviation
  // of the token's E logits (z + b), summed by the token's four threads in a
  // fixed order (every lane runs the shuffles)
  float sn = 1.f;
  if (noise && noise_scale > 0.f) {
    float s1 = 0.f;
#pragma unroll
    for (int q = 0; q < Q; ++q)
      if (e0 + q < E) s1 += v[q];
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    const float mean = s1 / (float)E;
    float s2 = 0.f;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const float dv = v[q] - mean;
      if (e0 + q < E) s2 = fmaf(dv, dv, s2);
    }
    s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
    s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
    sn = noise_scale * sqrtf(s2 / (float)E);
  }
  if (valid) {
    if (noise && !keys_done) {
      const float* nr = noise + (size_t)t * E + e0;
      if (vec4n) {
#pragma unroll
        for (int q = 0; q < Q; q += 4) {
          if (e0 + q < E) {
            const float4 w = __ldg(reinterpret_cast<const float4*>(nr + q));
            v[q] = fmaf(sn, w.x, v[q]);
            v[q + 1] = fmaf(sn, w.y, v[q + 1]);
            v[q + 2] = fmaf(sn, w.z, v[q + 2]);
            v[q + 3] = fmaf(sn, w.w, v[q + 3]);
          }
        }
      } else {
#pragma unroll
        for (int q = 0; q < Q; ++q)
          if (e0 + q < E) v[q] = fmaf(sn, __ldg(nr + q), v[q]);
      }
    }
    if (tau != 1.f) {
      const float inv_tau = 1.f / tau;
#pragma unroll
      for (int q = 0; q < Q; ++q) v[q] *= inv_tau;
    }
  }
#pragma unroll
  for (int q = 0; q < Q; ++q)
    if (e0 + q >= E) v[q] = -INFINITY;
  if (valid && logits) {
    float* lr = logits + (size_t)t * E + e0;
    if (vec4l) {
#pragma unroll
      for (int q = 0; q < Q; q += 4)
        if (e0 + q < E) *reinterpret_cast<float4*>(lr + q) = make_float4(v[q], v[q + 1], v[q + 2], v[q + 3]);
    } else {
#pragma unroll
      for (int q = 0; q < Q; ++q)
        if (e0 + q < E) lr[q] = v[q];
    }
  }
  // top-KM of this thread's experts, best first; (-inf, INT_MAX) ranks last
  float sv[KM];
  int si[KM];
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    sv[j] = -INFINITY;
    si[j] = 0x7fffffff;
  }
  if constexpr (KM == 2) {
    // one pass keeping the best two: the experts come in ascending index
    // order, so a later one ranks before a kept one only if strictly larger
    // (a tie keeps the lower index ahead)
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const float cv = v[q];
      if (cv > sv[0]) {
        sv[1] = sv[0];
        si[1] = si[0];
        sv[0] = cv;
        si[0] = e0 + q;
      } else if (cv > sv[1]) {
        sv[1] = cv;
        si[1] = e0 + q;
      }
    }
  } else {
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      float cv = v[q];
      int ci = e0 + q;
#pragma unroll
      for (int j = 0; j < KM; ++j) {
        if (ranks_before(cv, ci, sv[j], si[j])) {
          const float tv = sv[j];
          const int ti = si[j];
          sv[j] = cv;
          si[j] = ci;
          cv = tv;
          ci = ti;
        }
      }
    }
  }
  // merge with the other three threads' lists: the pairwise better of a[j]
  // and b[KM-1-j] are the top KM of both (a bitonic sequence), then sorted
  // by half-cleaners; all four threads end with the same list
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    float ov[KM];
    int oi[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      ov[j] = __shfl_xor_sync(0xffffffffu, sv[j], o);
      oi[j] = __shfl_xor_sync(0xffffffffu, si[j], o);
    }
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (ranks_before(ov[KM - 1 - j], oi[KM - 1 - j], sv[j], si[j])) {
        sv[j] = ov[KM - 1 - j];
        si[j] = oi[KM - 1 - j];
      }
    }
#pragma unroll
    for (int h = KM / 2; h >= 1; h >>= 1) {
#pragma unroll
      for (int j = 0; j < KM; ++j) {
        if ((j & h) == 0 && ranks_before(sv[j + h], si[j + h], sv[j], si[j])) {
          const float tv = sv[j];
          const int ti = si[j];
          sv[j] = sv[j + h];
          si[j] = si[j + h];
          sv[j + h] = tv;
          si[j + h] = ti;
        }
      }
    }
  }
  // the token's largest key heads the merged list
  const float m = sv[0];
  // probabilities for the statistics P_i, back into the token's row
  {
    float sum = 0.f;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      v[q] = (e0 + q < E && valid) ? __expf(v[q] - m) : 0.f;
      sum += v[q];
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    const float inv_s = valid ? 1.f / sum : 0.f;
    float4* row = reinterpret_cast<float4*>(&es.L[r][e0]);
#pragma unroll
    for (int q = 0; q < Q; q += 4)
      row[q / 4] = make_float4(v[q] * inv_s, v[q + 1] * inv_s, v[q + 2] * inv_s, v[q + 3] * inv_s);
  }
  if (valid && p == 0) {
    // gates from the selected keys only: g_j = p_j / sum_m p_m, where the
    // softmax denominator cancels
    float psel[KM], psum = 0.f;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (j < k) {
        psel[j] = expf(sv[j] - m);
        psum += psel[j];
      }
    }
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (j < k) {
        const int ej = si[j] < E ? si[j] : 0;
        idx[(size_t)t * k + j] = ej;
        gate[(size_t)t * k + j] = psel[j] / psum;
        atomicAdd(&es.hist[ej], 1);
      }
    }
  }
  epi_bar();  // probabilities and counts of the whole tile are in place
  // per-expert sums over the tile's 128 tokens: eight threads per expert,
  // thread q8 adding rows q8, q8 + 8, ..., q8 + 120 in that order, then a
  // fixed butterfly adds the eight. Eight rows apart, the row stride (EP + 4
  // floats) advances the bank by a multiple of 32, and rows q8 = 0..7 start
  // on eight different banks, so a warp's four experts x eight threads read
  // 32 different banks (rows 16 apart, as before, put all eight threads of an
  // expert on one bank).
  {
    const int e = etid >> 3, q8 = etid & 7;
    float a = 0.f;
    if (e < E) {
#pragma unroll
      for (int i = 0; i < 16; ++i) a += es.L[q8 + 8 * i][e];
    }
    a += __shfl_xor_sync(0xffffffffu, a, 1);
    a += __shfl_xor_sync(0xffffffffu, a, 2);
    a += __shfl_xor_sync(0xffffffffu, a, 4);
    if (q8 == 0 && e < E) {
      es.part[e] += a;
      if (tile_hist) tile_hist[(size_t)tile * E + e] = es.hist[e];
    }
  }
  epi_bar();  // the scratch and the counts are free for the next tile
}

template <int EP, int KM, bool SPLIT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmW, const float* __restrict__ bias,
                     const float* __restrict__ noise, float noise_scale, float tau, int T,
                     int d, int E, int k,
                     float* __restrict__ logits, int32_t* __restrict__ idx,
                     float* __restrict__ gate, float* __restrict__ partial,
                     int32_t* __restrict__ tile_hist, int32_t* __restrict__ hdr, int ksplit,
                     int kb_per_split, int tile_rows) {
  using Cfg = RouterCfg<EP>;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * NB * A_BYTES;
  RouterSmem<EP>& st = *reinterpret_cast<RouterSmem<EP>*>(smem + STAGES * Cfg::STAGE);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&st.full[s], 1);
      mbar_init(&st.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&st.tmem_full[a], 1);
      mbar_init(&st.tmem_empty[a], 32 * 4 * (EP / 16));  // every TMEM-reading thread
    }
    mbar_init(&st.final_bar, 1);
    st.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(&st.tmem_base, Cfg::TCOLS);
    tmem_relinquish();
  }
  for (int e = tid; e < EP; e += NUM_THREADS) st.epi.part[e] = 0.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  // the bias may come from the previous kernel: read it after the wait, by
  // epilogue threads (their first named barrier orders these stores before
  // the epilogue's reads)
  if (tid >= 64)
    for (int e = tid - 64; e < EP; e += EPI_THREADS) st.epi.bias[e] = (bias && e < E) ? bias[e] : 0.f;
  const uint32_t tmem_base = st.tmem_base;
  // work unit u = (tile, split): K blocks [split * kb_per_split, ...) of the tile
  const int ntiles = (T + tile_rows - 1) / tile_rows;
  const int nunits = ntiles * ksplit;
  const int num_kb = (d + BK - 1) / BK;
  volatile int* abort_flag = &st.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      const uint32_t box_tx = (uint32_t)(tile_rows * BK * 2 + Cfg::B_BYTES);
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const int tile = u / ksplit, split = u % ksplit;
        const int kb0 = split * kb_per_split;
        const int kb1 = min(num_kb, kb0 + kb_per_split);
        for (int kb = kb0; kb < kb1; kb += NB) {
          const int nb = min(NB, kb1 - kb);  // boxes of this stage (the range's end may cut it)
          if (!mbar_wait(&st.empty[stage], phase ^ 1u, abort_flag, hdr, 11)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&st.full[stage], (uint32_t)nb * box_tx);
          for (int b = 0; b < nb; ++b) {
            tma_load_2d(sA + (stage * NB + b) * A_BYTES, &tmX, &st.full[stage], (kb + b) * BK,
                        tile * tile_rows);
            tma_load_2d(sB + (stage * NB + b) * Cfg::B_BYTES, &tmW, &st.full[stage],
                        (kb + b) * BK, 0);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        int s = stage;
        uint32_t ph = phase;
        for (int i = 0; i < STAGES && i < issued; ++i) {
          if (--s < 0) {
            s = STAGES - 1;
            ph ^= 1u;
          }
          volatile int no_abort = 0;
          mbar_wait(&st.full[s], ph, &no_abort, nullptr, 0);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16_f32(BM, EP);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const int split = u % ksplit;
        const int kb0 = split * kb_per_split;
        const int kb1 = min(num_kb, kb0 + kb_per_split);
        if (!mbar_wait(&st.tmem_empty[acc], acc_phase ^ 1u, abort_flag, hdr, 12)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * EP);
        for (int kb = kb0; kb < kb1; kb += NB) {
          const int nb = min(NB, kb1 - kb);
          if (!mbar_wait(&st.full[stage], phase, abort_flag, hdr, 13)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int b = 0; b < nb; ++b) {
            const uint64_t adesc = sdesc_kmajor_sw128(a0 + (stage * NB + b) * A_BYTES);
            const uint64_t bdesc = sdesc_kmajor_sw128(b0 + (stage * NB + b) * Cfg::B_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              umma_bf16(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), IDESC,
                        (kb > kb0 || b > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&st.empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&st.tmem_full[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        umma_commit(&st.final_bar);
        volatile int no_abort = 0;
        mbar_wait(&st.final_bar, 0, &no_abort, nullptr, 0);
      }
    }
  } else {
    // ---------------- epilogue: warps 2 + 4 g .. 5 + 4 g read columns
    // [16 g, 16 g + 16) of the accumulator from TMEM (thread = token row;
    // g < EP/16, so up to all 16 warps share the copy); then epilogue thread
    // etid works on token etid / 4, experts quarter etid % 4
    constexpr int Q = EP / TPT;
    const int etid = tid - 64;  // 0..511
    const int cgrp = (warp - 2) >> 2;  // column group of a TMEM warp
    const bool tmem_warp = cgrp < EP / 16;
    const int quarter = warp & 3;  // a warp reads TMEM lanes 32 (warp % 4) ..
    const int lr = quarter * 32 + lane;  // the TMEM lane (token row) a TMEM warp reads
    const int r = etid >> 2, p = etid & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    // With whole logits in TMEM (no split) and noise added as given (not
    // std-scaled), the copy out of TMEM adds bias and noise: each thread
    // loads its 16 noise values before it waits for the tile's accumulator,
    // so that their DRAM latency passes under the tile's x stream instead of
    // after its last MMA. Same arithmetic as the per-token epilogue: (z + b) + g.
    const bool keys_early = !SPLIT && !(noise && noise_scale > 0.f);
    const int c0 = 16 * cgrp;  // this TMEM warp's first column
    const bool nvec = (E & 3) == 0 && (reinterpret_cast<uintptr_t>(noise) & 15u) == 0;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
      const int tile = u / ksplit;
      bool fail = false;
      if (tmem_warp) {
        const int t = tile * tile_rows + lr;
        const bool valid = lr < tile_rows && t < T;
        float nz[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) nz[j] = 0.f;
        if (keys_early && noise && valid) {
          const float* nr = noise + (size_t)t * E + c0;
          if (nvec) {
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
              if (c0 + j < E) {
                const float4 w4 = ld_nc_early_v4(nr + j);
                nz[j] = w4.x;
                nz[j + 1] = w4.y;
                nz[j + 2] = w4.z;
                nz[j + 3] = w4.w;
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c0 + j < E) nz[j] = ld_nc_early(nr + j);
          }
        }
        if (!mbar_wait(&st.tmem_full[acc], acc_phase, abort_flag, hdr, 14)) {
          fail = true;
        } else {
          tc_fence_after();
          uint32_t v[16];
          tmem_ld16(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * EP + c0), v);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&st.tmem_empty[acc]);
          float f[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(v[j]);
          if (keys_early && valid) {
            if (bias) {
              const float4* b4 = reinterpret_cast<const float4*>(&st.epi.bias[c0]);
#pragma unroll
              for (int j = 0; j < 16; j += 4) {
                const float4 b = b4[j / 4];
                f[j] += b.x;
                f[j + 1] += b.y;
                f[j + 2] += b.z;
                f[j + 3] += b.w;
              }
            }
            if (noise) {
#pragma unroll
              for (int j = 0; j < 16; ++j) f[j] += nz[j];
            }
          }
          // 16 of the token's (partial) logits or keys, into its row of the scratch
          float4* row = reinterpret_cast<float4*>(&st.epi.L[lr][c0]);
#pragma unroll
          for (int e = 0; e < 16; e += 4) row[e / 4] = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
        }
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (etid < EP) st.epi.hist[etid] = 0;
      if (epi_bar_or(fail)) break;  // the tile's logits are in shared memory
      if (!SPLIT) {
        float v[Q];
        load_quarter<EP>(st.epi, r, p, v);
        router_tile_epilogue<EP, KM>(v, keys_early, tile, tile_rows, r, p, etid, bias, noise,
                                     noise_scale, tau, T, E, k, logits, idx, gate, tile_hist,
                                     st.epi);
      }
    }
    if (!SPLIT)
      for (int e = etid; e < E; e += EPI_THREADS) partial[(size_t)blockIdx.x * E + e] = st.epi.part[e];
  }

  if (SPLIT) {
    // one tile per cluster, split = cluster rank. Every rank sums one slice
    // of the columns (CW experts, 16-byte pieces) over all ranks' partial
    // logits in split order (the order of a single pass) and writes the sums
    // into the first CTA's scratch, which then runs the epilogue. The cluster
    // barriers order: partials written / slices read / sums written.
    static_assert(EP % 4 == 0 && BM * (EP / 2 / 4) <= 2 * EPI_THREADS, "two pieces per thread");
    const uint32_t my = cluster_ctarank();
    const int CW = ((EP + ksplit - 1) / ksplit + 3) / 4 * 4;
    const int c0 = (int)my * CW;
    const int nv = c0 < EP ? (min(EP, c0 + CW) - c0) / 4 : 0;  // pieces per row
    const int etid = tid - 64;
    float4 acc4[2];
    int row4[2], col4[2];
    __syncwarp();
    cluster_sync();
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      acc4[it] = make_float4(0.f, 0.f, 0.f, 0.f);
      const int item = etid + it * EPI_THREADS;
      row4[it] = -1;
      col4[it] = 0;
      if (warp >= 2 && item < BM * nv) {
        row4[it] = item / nv;
        col4[it] = c0 + 4 * (item % nv);
        // every rank's piece in flight at once, then summed in split order
        // (added one by one after each load, the eight remote round trips
        // ran back to back)
        float4 w[kRouterMaxSplit];
#pragma unroll
        for (int qq = 0; qq < kRouterMaxSplit; ++qq)
          if (qq < ksplit)
            w[qq] = ld_cluster_v4(cluster_addr(&st.epi.L[row4[it]][col4[it]], (uint32_t)qq));
#pragma unroll
        for (int qq = 0; qq < kRouterMaxSplit; ++qq) {
          if (qq < ksplit) {
            acc4[it].x += w[qq].x;
            acc4[it].y += w[qq].y;
            acc4[it].z += w[qq].z;
            acc4[it].w += w[qq].w;
          }
        }
      }
    }
    __syncwarp();
    cluster_sync();  // every slice is read before the first CTA's scratch is overwritten
#pragma unroll
    for (int it = 0; it < 2; ++it)
      if (row4[it] >= 0) st_cluster_v4(cluster_addr(&st.epi.L[row4[it]][col4[it]], 0u), acc4[it]);
    __syncwarp();
    cluster_sync();  // the summed logits are in the first CTA's scratch
    if (my == 0 && warp >= 2) {
      constexpr int Q = EP / TPT;
      const int r = etid >> 2, p = etid & 3;
      const int tile = (int)blockIdx.x / ksplit;
      float v[Q];
      load_quarter<EP>(st.epi, r, p, v);
      if (etid < EP) st.epi.hist[etid] = 0;
      epi_bar();  // counts zeroed before the epilogue's atomics
      router_tile_epilogue<EP, KM>(v, false, tile, BM, r, p, etid, bias, noise, noise_scale, tau,
                                   T, E, k, logits, idx, gate, tile_hist, st.epi);
      for (int e = etid; e < E; e += EPI_THREADS) partial[(size_t)tile * E + e] = st.epi.part[e];
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, Cfg::TCOLS);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn_router() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool map_rows(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn_router();
  if (!enc) return false;
  cuuint64_t gdim[2] = {K, rows};
  cuuint64_t gstride[1] = {K * 2};
  cuuint32_t box[2] = {BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EP, int KM, bool SPLIT>
cudaError_t set_smem_attr() {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(router_tc_kernel<EP, KM, SPLIT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)router_smem_bytes<EP>());
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  return cudaSuccess;
}

template <int EP, int KM>
cudaError_t launch_ep_km(const moe_config_t& c, const CUtensorMap& mx, const CUtensorMap& mw,
                         const float* bias, const float* noise, float* logits, int32_t* idx,
                         float* gate, float* partial, int32_t* tile_hist, int32_t* hdr,
                         cudaStream_t s) {
  static_assert(router_smem_bytes<EP>() <= 227 * 1024, "router shared memory over the per-CTA limit");
  const RouterSplit sp = router_tc_split(c);
  cudaError_t e;
  if (sp.ksplit == 1) {
    if ((e = set_smem_attr<EP, KM, false>()) != cudaSuccess) return e;
    return launch_pdl(router_tc_kernel<EP, KM, false>, dim3(router_tc_grid(c)),
                      dim3(NUM_THREADS), router_smem_bytes<EP>(), s, mx, mw, bias, noise,
                      c.noise_scale, c.tau, c.T, c.d, c.E, c.k, logits, idx, gate, partial,
                      tile_hist, hdr, 1,
                      sp.kb_per_split, router_tc_rows(c));
  }
  if ((e = set_smem_attr<EP, KM, true>()) != cudaSuccess) return e;
  const int units = router_tc_tiles(c) * sp.ksplit;  // one cluster of ksplit CTAs per tile
  return launch_pdl_cluster(router_tc_kernel<EP, KM, true>, dim3(units), dim3(NUM_THREADS),
                            router_smem_bytes<EP>(), sp.ksplit, s, mx, mw, bias, noise,
                            c.noise_scale, c.tau, c.T, c.d, c.E, c.k, logits, idx, gate, partial,
                            tile_hist, hdr,
                            sp.ksplit, sp.kb_per_split, (int)kRouterTcTile);
}

// k <= 2 sorts candidate lists of two entries, larger k lists of eight.
template <int EP>
cudaError_t launch_ep(const moe_config_t& c, const void* x, const void* Wg, const float* bias,
                      const float* noise, float* logits, int32_t* idx, float* gate,
                      float* partial, int32_t* tile_hist, float* split_part, int32_t* hdr,
                      cudaStream_t s) {
  CUtensorMap mx, mw;
  if (!map_rows(&mx, x, c.d, c.T, (uint32_t)router_tc_rows(c)) ||
      !map_rows(&mw, Wg, c.d, c.E, EP))
    return cudaErrorInvalidValue;
  (void)split_part;
  if (c.k <= 2)
    return launch_ep_km<EP, 2>(c, mx, mw, bias, noise, logits, idx, gate, partial, tile_hist,
                               hdr, s);
  return launch_ep_km<EP, kMaxK>(c, mx, mw, bias, noise, logits, idx, gate, partial, tile_hist,
                                 hdr, s);
}

}  // namespace

bool router_tc_supported(const moe_config_t& c) { return c.dtype == MOE_BF16 && c.E <= 64; }

cudaError_t launch_router_tc(const moe_config_t& c, const void* x, const void* Wg,
                             const float* bias, const float* noise, float* logits, int32_t* idx,
                             float* gate, float* partial, int32_t* tile_hist, float* split_part,
                             int32_t* hdr, cudaStream_t s) {
  const int ep = (c.E + 15) / 16 * 16;
#define MOE_EP_CASE(EPV)                                                                       \
  case EPV:                                                                                    \
    return launch_ep<EPV>(c, x, Wg, bias, noise, logits, idx, gate, partial, tile_hist,        \
                          split_part, hdr, s)
  switch (ep) {
    MOE_EP_CASE(16);
    MOE_EP_CASE(32);
    MOE_EP_CASE(48);
    MOE_EP_CASE(64);
    default: return cudaErrorInvalidValue;
  }
#undef MOE_EP_CASE
}

}  // namespace moe
