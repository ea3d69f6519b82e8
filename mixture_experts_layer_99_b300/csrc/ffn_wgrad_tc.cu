// Expert weight gradients of the backward pass on the tensor cores.
//
// For expert e with kept rows R_e:  dW[e] = A_e^T B_e, a reduction over R_e:
//   dW2[e]        = dY_e^T h_e             [d, H]
//   dW1[e]        = dact_e^T xd_e          [H, d]   (SwiGLU: [dW1; dW3] = [da | dv]^T xd)
// The operands come transposed, At [M, Rp] and Bt [N, Rp] (bf16, K-major with
// K = the padded packed rows): expert e owns columns [poff_e, poff_{e+1}),
// its rows followed by zeros up to a multiple of 64, so every K block of 64
// lies inside one expert and starts on a 128-byte boundary.
//
// Kernel layout as in the grouped GEMM (one CTA per SM, 320 threads, warp 0
// TMA producer, warp 1 MMA issuer, warps 2-9 epilogue, two 256-column fp32
// accumulators in TMEM), tiles (e, 128-row m tile, 256-column n tile) with m
// fastest. The epilogue writes fp32 rows; an expert without rows gets zeros.
#include "moe_internal.h"
#include "tc_ptx.cuh"

#include <mutex>

namespace moe {
namespace {

using namespace ptx;

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int UMMA_N = 256;
constexpr int UMMA_K = 16;
constexpr int NUM_THREADS = 320;
constexpr int EPI_WARPS = 8;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;       // 16 KB
constexpr int B_BYTES = UMMA_N * BK * 2;   // 32 KB
constexpr int TMEM_COLS = 2 * UMMA_N;

struct Smem {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t final_bar;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr size_t SMEM_BYTES = 1024 + STAGES * (A_BYTES + B_BYTES) + sizeof(Smem);
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");

struct WTile {
  int e, m0, n0, kb0, kb1;
};
__device__ __forceinline__ WTile wtile(const int32_t* __restrict__ poff, int mtc, int ntc,
                                       int tile) {
  WTile w;
  const int per = mtc * ntc;
  w.e = tile / per;
  const int local = tile - w.e * per;
  w.m0 = (local % mtc) * BM;
  w.n0 = (local / mtc) * UMMA_N;
  w.kb0 = __ldg(poff + w.e) / BK;
  w.kb1 = __ldg(poff + w.e + 1) / BK;
  return w;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    wgrad_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB, const int32_t* __restrict__ poff,
                    int E, int M, int N, int m_split, float* __restrict__ out,
                    float* __restrict__ out2, int32_t* __restrict__ hdr) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  Smem& st = *reinterpret_cast<Smem*>(smem + STAGES * (A_BYTES + B_BYTES));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&st.full[s], 1);
      mbar_init(&st.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&st.tmem_full[a], 1);
      mbar_init(&st.tmem_empty[a], EPI_WARPS * 32);
    }
    mbar_init(&st.final_bar, 1);
    st.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&st.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  pdl_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int mtc = (M + BM - 1) / BM, ntc = (N + UMMA_N - 1) / UMMA_N;
  const int total = E * mtc * ntc;
  const uint32_t tmem_base = st.tmem_base;
  volatile int* abort_flag = &st.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const WTile w = wtile(poff, mtc, ntc, tile);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait(&st.empty[stage], phase ^ 1u, abort_flag, hdr, 21)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&st.full[stage], A_BYTES + B_BYTES);
          tma_load_2d(sA + stage * A_BYTES, &tmA, &st.full[stage], kb * BK, w.m0);
          tma_load_2d(sB + stage * B_BYTES, &tmB, &st.full[stage], kb * BK, w.n0);
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
      constexpr uint32_t IDESC = idesc_bf16_f32(BM, UMMA_N);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const WTile w = wtile(poff, mtc, ntc, tile);
        if (!mbar_wait(&st.tmem_empty[acc], acc_phase ^ 1u, abort_flag, hdr, 22)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * UMMA_N);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait(&st.full[stage], phase, abort_flag, hdr, 23)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sdesc_kmajor_sw128(a0 + stage * A_BYTES);
          const uint64_t bdesc = sdesc_kmajor_sw128(b0 + stage * B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk)
            umma_bf16(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), IDESC,
                      (kb > w.kb0 || kk > 0) ? 1u : 0u);
          umma_commit(&st.empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        // also for an expert without rows: the epilogue then writes zeros
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
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int half = ew >> 2;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const WTile w = wtile(poff, mtc, ntc, tile);
      if (!mbar_wait(&st.tmem_full[acc], acc_phase, abort_flag, hdr, 24)) break;
      tc_fence_after();
      const bool empty = w.kb1 == w.kb0;
      const int m = w.m0 + quarter * 32 + lane;
      const int cbase = 128 * half;
      uint32_t r[128];
      if (!empty) {
        const uint32_t t_row =
            tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * UMMA_N);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
          tmem_ld32(t_row + (uint32_t)(cbase + 32 * ch), *reinterpret_cast<uint32_t(*)[32]>(&r[32 * ch]));
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int j = 0; j < 128; ++j) r[j] = 0u;
      }
      tc_fence_before();
      mbar_arrive(&st.tmem_empty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
      if (m < M) {
        float* orow = m < m_split
                          ? out + ((size_t)w.e * m_split + m) * N
                          : out2 + ((size_t)w.e * (M - m_split) + (m - m_split)) * N;
#pragma unroll
        for (int j = 0; j < 128; j += 4) {
          const int n = w.n0 + cbase + j;
          if (n + 4 <= N)
            *reinterpret_cast<float4*>(orow + n) =
                make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                            __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn_wgrad() {
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

// [rows, K] bf16 (row stride ld), box [box_rows, 64], 128-byte swizzle.
bool map_kmajor(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint64_t ld,
                uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn_wgrad();
  if (!enc) return false;
  cuuint64_t gdim[2] = {K, rows};
  cuuint64_t gstride[1] = {ld * 2};
  cuuint32_t box[2] = {BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// out[e] = At_e Bt_e^T over expert e's padded columns: At [M, ld] and Bt
// [N, ld] bf16 with ld >= poff[E] (a multiple of 8); rows m < m_split of each
// expert's [M, N] result go to out [E, m_split, N], the rest to out2
// [E, M - m_split, N] (fp32).
cudaError_t launch_wgrad_tc(const void* At, const void* Bt, int64_t ld, const int32_t* poff,
                            int E, int M, int N, int m_split, float* out, float* out2,
                            int32_t* hdr, cudaStream_t s) {
  CUtensorMap ma, mb;
  if (!map_kmajor(&ma, At, (uint64_t)ld, (uint64_t)M, (uint64_t)ld, BM) ||
      !map_kmajor(&mb, Bt, (uint64_t)ld, (uint64_t)N, (uint64_t)ld, UMMA_N))
    return cudaErrorInvalidValue;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(wgrad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int64_t tiles = (int64_t)E * ((M + BM - 1) / BM) * ((N + UMMA_N - 1) / UMMA_N);
  const int sms = device_sm_count();
  const int grid = (int)(tiles < sms ? tiles : sms);
  return launch_pdl(wgrad_tc_kernel, dim3(grid > 0 ? grid : 1), dim3(NUM_THREADS), SMEM_BYTES, s,
                    ma, mb, poff, E, M, N, m_split, out, out2, hdr);
}

}  // namespace moe
