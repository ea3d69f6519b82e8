// Fused router on the tcgen05 tensor cores for bf16 tokens and E <= 64.
//
// logits l = (x Wg^T + b + g) / tau, softmax p = softmax(l), the k largest
// logits (descending, ties to the lower expert index), renormalised gates
// g_j = p_{K_j} / sum_m p_{K_m}, per-CTA sums of p for P_i and per-tile
// selection counts for the dispatch. This is the gate of the kwkr.cn MoE
// article ("MoE sparse activation: from the math to the code"), section 2.1,
// fused with softmax and top-k as its section 5.3 suggests; bias, noise and
// temperature as in the lpnh.cn MoE guide, section 3.3.
//
// The contraction x Wg^T (E tiny) is HBM-bound: the kernel streams 128-token
// tiles of x through TMA and issues one 128 x E_pad x 16 MMA per 16-wide K
// step, so each epilogue thread owns one token's whole logit row in TMEM.
//   warp 0      TMA producer (x tile [128 x 64] + Wg tile [E_pad x 64])
//   warp 1      TMEM owner, MMA issuer
//   warps 2-5   epilogue: one thread per token
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
constexpr int NUM_THREADS = 192;
constexpr int A_BYTES = BM * BK * 2;

// Epilogue scratch: the tile's probabilities, one padded row per token (an odd
// row stride keeps both the row writes and the column reads conflict-free),
// summed per expert down the columns.
template <int EP>
struct EpiSmem {
  float col[BM][EP + 1];
  float part[EP];
  int hist[EP];
};

template <int EP>
struct RouterCfg {
  static constexpr int B_BYTES = EP * BK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  // as many operand stages (at most 8) as fit beside the epilogue scratch
  static constexpr int FIT = (int)((220 * 1024 - sizeof(EpiSmem<EP>) - 1024 - 256) / STAGE);
  static constexpr int STAGES = FIT > 8 ? 8 : FIT;
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

__device__ __forceinline__ void epi_bar() {  // named barrier over the 4 epilogue warps
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

template <int EP>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, float (&v)[EP]) {
  static_assert(EP % 16 == 0, "EP multiple of 16");
#pragma unroll
  for (int c = 0; c < EP; c += 32) {
    if (c + 32 <= EP) {
      uint32_t r[32];
      tmem_ld32(taddr + c, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) v[c + j] = __uint_as_float(r[j]);
    } else {
      uint32_t r[16];
      tmem_ld16(taddr + c, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) v[c + j] = __uint_as_float(r[j]);
    }
  }
}

// One token per thread (thread r of the 128 owns token tile*128 + r): keys,
// softmax, top-k (descending, ties to the lower index), gates, and the
// tile's per-expert selection counts and sums of p (fixed order).
template <int EP>
__device__ __forceinline__ void router_tile_epilogue(
    float (&v)[EP], int tile, int r, int etid, const float* __restrict__ bias,
    const float* __restrict__ noise, float tau, int T, int E, int k, float* __restrict__ logits,
    int32_t* __restrict__ idx, float* __restrict__ gate, int32_t* __restrict__ tile_hist,
    EpiSmem<EP>& es) {
  for (int e = etid; e < EP; e += 128) es.hist[e] = 0;
  const int t = tile * BM + r;
  const bool valid = t < T;
  const bool vec4 = (E & 3) == 0;  // rows of [T, E] fp32 arrays are 16-byte aligned
  // selection keys l = (z + b + g) / tau (one reciprocal; tau = 1 leaves them as they are)
  if (valid) {
    if (bias) {
#pragma unroll
      for (int e = 0; e < EP; ++e)
        if (e < E) v[e] += __ldg(bias + e);
    }
    if (noise) {
      const float* nr = noise + (size_t)t * E;
      if (vec4) {
#pragma unroll
        for (int e = 0; e < EP; e += 4) {
          if (e < E) {
            const float4 q = __ldg(reinterpret_cast<const float4*>(nr + e));
            v[e] += q.x;
            v[e + 1] += q.y;
            v[e + 2] += q.z;
            v[e + 3] += q.w;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < EP; ++e)
          if (e < E) v[e] += __ldg(nr + e);
      }
    }
    if (tau != 1.f) {
      const float inv_tau = 1.f / tau;
#pragma unroll
      for (int e = 0; e < EP; ++e) v[e] *= inv_tau;
    }
  }
#pragma unroll
  for (int e = 0; e < EP; ++e)
    if (e >= E) v[e] = -INFINITY;
  float m = -INFINITY;
#pragma unroll
  for (int e = 0; e < EP; ++e) m = fmaxf(m, v[e]);
  if (valid && logits) {
    float* lr = logits + (size_t)t * E;
    if (vec4) {
#pragma unroll
      for (int e = 0; e < EP; e += 4)
        if (e < E) *reinterpret_cast<float4*>(lr + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
    } else {
#pragma unroll
      for (int e = 0; e < EP; ++e)
        if (e < E) lr[e] = v[e];
    }
  }
  // top-k on the keys: descending, ties to the lower index
  uint64_t taken = 0;
  float selv[kMaxK];
  int seli[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    selv[j] = -INFINITY;
    seli[j] = 0;
    if (j < k) {
      float bv = -INFINITY;
      int bi = -1;
#pragma unroll
      for (int e = 0; e < EP; ++e) {
        const bool free_ = e < E && !((taken >> e) & 1ull);
        if (free_ && (bi < 0 || v[e] > bv)) {
          bv = v[e];
          bi = e;
        }
      }
      if (bi < 0) bi = 0;
      taken |= 1ull << bi;
      selv[j] = bv;
      seli[j] = bi;
    }
  }
  __syncwarp();
  epi_bar();  // hist zeroed; the previous tile's column sums are done
  if (valid) {
    // gates from the selected keys only: g_j = p_j / sum_m p_m, where the
    // softmax denominator cancels
    float psel[kMaxK], psum = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < k) {
        psel[j] = expf(selv[j] - m);
        psum += psel[j];
      }
    }
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < k) {
        idx[(size_t)t * k + j] = seli[j];
        gate[(size_t)t * k + j] = psel[j] / psum;
        atomicAdd(&es.hist[seli[j]], 1);
      }
    }
  }
  // probabilities for the statistics P_i: one row per token in shared memory
  {
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < EP; ++e) {
      v[e] = (e < E && valid) ? __expf(v[e] - m) : 0.f;
      s += v[e];
    }
    const float inv_s = valid ? 1.f / s : 0.f;
#pragma unroll
    for (int e = 0; e < EP; ++e) es.col[r][e] = v[e] * inv_s;
  }
  epi_bar();
  // per-expert sums over the tile's 128 tokens: one thread per expert walks
  // its column in token order (two interleaved partial sums, then added)
  for (int e = etid; e < E; e += 128) {
    float a0 = 0.f, a1 = 0.f;
#pragma unroll 8
    for (int rr = 0; rr < BM; rr += 2) {
      a0 += es.col[rr][e];
      a1 += es.col[rr + 1][e];
    }
    es.part[e] += a0 + a1;
    if (tile_hist) tile_hist[(size_t)tile * E + e] = es.hist[e];
  }
  epi_bar();
}

template <int EP, bool SPLIT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmW, const float* __restrict__ bias,
                     const float* __restrict__ noise, float tau, int T, int d, int E, int k,
                     float* __restrict__ logits, int32_t* __restrict__ idx,
                     float* __restrict__ gate, float* __restrict__ partial,
                     int32_t* __restrict__ tile_hist, int32_t* __restrict__ hdr, int ksplit,
                     int kb_per_split, float* __restrict__ split_part) {
  using Cfg = RouterCfg<EP>;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  RouterSmem<EP>& st = *reinterpret_cast<RouterSmem<EP>*>(smem + STAGES * Cfg::STAGE);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&st.full[s], 1);
      mbar_init(&st.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&st.tmem_full[a], 1);
      mbar_init(&st.tmem_empty[a], 128);
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
  const uint32_t tmem_base = st.tmem_base;
  // work unit u = (tile, split): K blocks [split * kb_per_split, ...) of the tile
  const int ntiles = (T + BM - 1) / BM;
  const int nunits = ntiles * ksplit;
  const int num_kb = (d + BK - 1) / BK;
  volatile int* abort_flag = &st.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const int tile = u / ksplit, split = u % ksplit;
        const int kb0 = split * kb_per_split;
        const int kb1 = min(num_kb, kb0 + kb_per_split);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&st.empty[stage], phase ^ 1u, abort_flag, hdr, 11)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&st.full[stage], Cfg::STAGE);
          tma_load_2d(sA + stage * A_BYTES, &tmX, &st.full[stage], kb * BK, tile * BM);
          tma_load_2d(sB + stage * Cfg::B_BYTES, &tmW, &st.full[stage], kb * BK, 0);
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
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&st.full[stage], phase, abort_flag, hdr, 13)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sdesc_kmajor_sw128(a0 + stage * A_BYTES);
          const uint64_t bdesc = sdesc_kmajor_sw128(b0 + stage * Cfg::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), IDESC,
                      (kb > kb0 || kk > 0) ? 1u : 0u);
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
    // ---------------- epilogue: thread r of the tile owns token tile*128 + r
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int etid = tid - 64;  // 0..127
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
      const int tile = u / ksplit, split = u % ksplit;
      if (!mbar_wait(&st.tmem_full[acc], acc_phase, abort_flag, hdr, 14)) break;
      tc_fence_after();
      float v[EP];
      tmem_ld_row<EP>(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * EP), v);
      tc_fence_before();
      mbar_arrive(&st.tmem_empty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
      if (SPLIT) {
        // this split's partial logits, [EP][128] column-major in the (not yet
        // used) epilogue scratch, for the cluster's first CTA to read
        (void)split;
        float* pt = &st.epi.col[0][0];
#pragma unroll
        for (int e = 0; e < EP; ++e) pt[e * BM + r] = v[e];
      } else {
        router_tile_epilogue<EP>(v, tile, r, etid, bias, noise, tau, T, E, k, logits, idx, gate,
                                 tile_hist, st.epi);
      }
    }
    if (!SPLIT)
      for (int e = etid; e < E; e += 128) partial[(size_t)blockIdx.x * E + e] = st.epi.part[e];
  }

  if (SPLIT) {
    // one tile per cluster, split = cluster rank: the first CTA sums the
    // partials of all ranks in split order (the order of a single pass) and
    // runs the epilogue; the second cluster barrier keeps every CTA's scratch
    // alive until it has been read
    __syncwarp();
    cluster_sync();
    if (cluster_ctarank() == 0 && warp >= 2) {
      const int quarter = warp & 3;
      const int r = quarter * 32 + lane;
      const int etid = tid - 64;
      const int tile = (int)blockIdx.x / ksplit;
      const float* pt = &st.epi.col[0][0];
      float v[EP];
#pragma unroll
      for (int e = 0; e < EP; ++e) v[e] = 0.f;
      for (int q = 0; q < ksplit; ++q) {
        const uint32_t base = cluster_addr(pt, (uint32_t)q) + (uint32_t)r * 4u;
        float w[EP];
#pragma unroll
        for (int e = 0; e < EP; ++e) w[e] = ld_cluster_f32(base + (uint32_t)(e * BM * 4));
#pragma unroll
        for (int e = 0; e < EP; ++e) v[e] += w[e];
      }
      epi_bar();  // every row is read before the epilogue reuses the scratch
      router_tile_epilogue<EP>(v, tile, r, etid, bias, noise, tau, T, E, k, logits, idx, gate,
                               tile_hist, st.epi);
      for (int e = etid; e < E; e += 128) partial[(size_t)tile * E + e] = st.epi.part[e];
    }
    __syncwarp();
    cluster_sync();
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

template <int EP, bool SPLIT>
cudaError_t set_smem_attr() {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(router_tc_kernel<EP, SPLIT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)router_smem_bytes<EP>());
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  return cudaSuccess;
}

template <int EP>
cudaError_t launch_ep(const moe_config_t& c, const void* x, const void* Wg, const float* bias,
                      const float* noise, float* logits, int32_t* idx, float* gate,
                      float* partial, int32_t* tile_hist, float* split_part, int32_t* hdr,
                      cudaStream_t s) {
  CUtensorMap mx, mw;
  if (!map_rows(&mx, x, c.d, c.T, BM) || !map_rows(&mw, Wg, c.d, c.E, EP))
    return cudaErrorInvalidValue;
  const RouterSplit sp = router_tc_split(c);
  cudaError_t e;
  if (sp.ksplit == 1) {
    if ((e = set_smem_attr<EP, false>()) != cudaSuccess) return e;
    return launch_pdl(router_tc_kernel<EP, false>, dim3(router_tc_grid(c)), dim3(NUM_THREADS),
                      router_smem_bytes<EP>(), s, mx, mw, bias, noise, c.tau, c.T, c.d, c.E,
                      c.k, logits, idx, gate, partial, tile_hist, hdr, 1, sp.kb_per_split,
                      (float*)nullptr);
  }
  if ((e = set_smem_attr<EP, true>()) != cudaSuccess) return e;
  const int units = router_tc_tiles(c) * sp.ksplit;  // one cluster of ksplit CTAs per tile
  (void)split_part;
  return launch_pdl_cluster(router_tc_kernel<EP, true>, dim3(units), dim3(NUM_THREADS),
                            router_smem_bytes<EP>(), sp.ksplit, s, mx, mw, bias, noise, c.tau,
                            c.T, c.d, c.E, c.k, logits, idx, gate, partial, tile_hist, hdr,
                            sp.ksplit, sp.kb_per_split, (float*)nullptr);
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
