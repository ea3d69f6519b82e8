// Expert weight gradients of the backward pass on the tensor cores.
//
// For expert e with kept rows R_e:  dW[e] = A_e^T B_e, a reduction over R_e:
//   dW2[e]        = dY_e^T h_e             [d, H]
//   dW1[e]        = dact_e^T xd_e          [H, d]   (SwiGLU: [dW1; dW3] = [da | dv]^T xd)
// (and dW_g = dz^T x over token groups). The operands are the row-major
// activations A [R, M] and B [R, N] (bf16) as the forward and the backward
// wrote them: both are read MN-major, the reduction dimension K being their
// rows, expert e's K range the packed rows [off_e, off_{e+1}). A K block of 64
// rows starts anywhere (TMA places no alignment rule on the row coordinate);
// the last block of an expert also holds rows of the next expert, so a
// fix-up warp zeroes those rows of the A tile in shared memory before the
// MMA reads it (and of the B tile too whenever the block reaches past the
// last kept row, where the buffers hold no data: 0 x NaN would not vanish;
// that is the last expert's block, and an earlier expert's when the experts
// after it hold fewer rows than the block's padding).
//
// Kernel layout as in the grouped GEMM (one CTA per SM, warp 0 TMA producer,
// warp 1 MMA issuer, warps 2-9 epilogue, warp 10 the fix-up, two 256-column
// fp32 accumulators in TMEM), tiles (e, 128-row m tile, 256-column n tile)
// with m fastest. A stage holds A as two boxes [64 rows x 64 m] and B as four
// boxes [64 rows x 64 n]. The epilogue writes fp32 rows; an expert without
// rows gets zeros. Each epilogue warp turns its 32 rows x 32 columns around
// in shared memory (4 KB) so that every store instruction writes four whole
// 128-byte row segments: stored straight from the accumulator's layout (one
// row per lane), each instruction would touch 32 rows with 16 bytes each,
// and the long tail's weight gradients (2.2 GB of fp32, mostly experts with
// a few rows, whose tiles are nothing but stores) went out at 1.8 TB/s.
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
constexpr int NUM_THREADS = 352;
constexpr int FIX_WARP = 10;
constexpr int EPI_WARPS = 8;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;       // 16 KB
constexpr int B_BYTES = UMMA_N * BK * 2;   // 32 KB
constexpr int TMEM_COLS = 2 * UMMA_N;

constexpr int BOX_BYTES = 64 * BK * 2;     // one [64 rows x 64] box, 8 KB

struct Smem {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t needfix[STAGES];  // the MMA has a tail block in this stage
  uint64_t fixed[STAGES];    // its rows past the expert are zero
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t final_bar;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr int EPI_BYTES = 32 * 32 * 4;     // one warp's 32 x 32 fp32 block
constexpr size_t SMEM_BYTES =
    1024 + STAGES * (A_BYTES + B_BYTES) + EPI_WARPS * EPI_BYTES + sizeof(Smem);
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");

// tile -> expert, first m and n, first row of the expert, its K blocks, the
// rows of its last block that belong to it (1..64), and whether that block
// reaches past the end of all rows (off[E]: rows no one wrote). The last
// block of any expert can: of the last one, and of an earlier one when the
// experts after it hold fewer rows than the block's padding.
struct WTile {
  int e, m0, n0, row0, nkb, tail;
  bool past_end;
};
__device__ __forceinline__ WTile wtile(const int32_t* __restrict__ off, int E, int mtc, int ntc,
                                       int tile) {
  WTile w;
  const int per = mtc * ntc;
  w.e = tile / per;
  const int local = tile - w.e * per;
  w.m0 = (local % mtc) * BM;
  w.n0 = (local / mtc) * UMMA_N;
  w.row0 = __ldg(off + w.e);
  const int rows = __ldg(off + w.e + 1) - w.row0;
  w.nkb = rows > 0 ? (rows + BK - 1) / BK : 0;
  w.tail = rows - (w.nkb - 1) * BK;
  w.past_end = w.row0 + w.nkb * BK > __ldg(off + E);
  return w;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    wgrad_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB, const int32_t* __restrict__ off,
                    int E, int M, int N, int m_split, float* __restrict__ out,
                    float* __restrict__ out2, int32_t* __restrict__ hdr) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint8_t* sE = smem + STAGES * (A_BYTES + B_BYTES);
  Smem& st = *reinterpret_cast<Smem*>(sE + EPI_WARPS * EPI_BYTES);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&st.full[s], 1);
      mbar_init(&st.empty[s], 1);
      mbar_init(&st.needfix[s], 1);
      mbar_init(&st.fixed[s], 1);
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
        const WTile w = wtile(off, E, mtc, ntc, tile);
        for (int kb = 0; kb < w.nkb; ++kb) {
          if (!mbar_wait(&st.empty[stage], phase ^ 1u, abort_flag, hdr, 21)) {
            ok = false;
            break;
          }
          const int row = w.row0 + kb * BK;
          mbar_expect_tx(&st.full[stage], A_BYTES + B_BYTES);
#pragma unroll
          for (int c = 0; c < BM / 64; ++c)
            tma_load_2d(sA + stage * A_BYTES + c * BOX_BYTES, &tmA, &st.full[stage], w.m0 + 64 * c,
                        row);
#pragma unroll
          for (int c = 0; c < UMMA_N / 64; ++c)
            tma_load_2d(sB + stage * B_BYTES + c * BOX_BYTES, &tmB, &st.full[stage], w.n0 + 64 * c,
                        row);
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
      // A and B MN-major (bits 15 and 16)
      constexpr uint32_t IDESC = idesc_bf16_f32(BM, UMMA_N) | (1u << 15) | (1u << 16);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0, fix_bits = 0;
      bool ok = true;
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const WTile w = wtile(off, E, mtc, ntc, tile);
        if (!mbar_wait(&st.tmem_empty[acc], acc_phase ^ 1u, abort_flag, hdr, 22)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * UMMA_N);
        for (int kb = 0; kb < w.nkb; ++kb) {
          if (!mbar_wait(&st.full[stage], phase, abort_flag, hdr, 23)) {
            ok = false;
            break;
          }
          // a tail block: hand the landed stage to the fix-up warp and wait
          // until its rows past the expert are zero (one request at a time
          // per stage, so both sides' parities stay in step)
          if (kb == w.nkb - 1 && w.tail < BK) {
            mbar_arrive(&st.needfix[stage]);
            const bool got = mbar_wait(&st.fixed[stage], (fix_bits >> stage) & 1u, abort_flag,
                                       hdr, 26);
            fix_bits ^= 1u << stage;
            if (!got) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
          // 64-row boxes 8 KB apart, K advanced by two 8-row atoms per MMA
          const uint64_t adesc = sdesc_mnmajor_sw128(a0 + stage * A_BYTES, BOX_BYTES);
          const uint64_t bdesc = sdesc_mnmajor_sw128(b0 + stage * B_BYTES, BOX_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk)
            umma_bf16(d_tmem, adesc + (uint64_t)(kk * 128), bdesc + (uint64_t)(kk * 128), IDESC,
                      (kb > 0 || kk > 0) ? 1u : 0u);
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
  } else if (warp == FIX_WARP) {
    // Serves the MMA's requests for tail blocks in order: zeroes the rows of
    // the stage past the expert's end (whole 128-byte lines, which the
    // swizzle only permutes within) and answers through `fixed`.
    int stage = 0;
    uint32_t phase = 0, fix_bits = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const WTile w = wtile(off, E, mtc, ntc, tile);
      for (int kb = 0; kb < w.nkb; ++kb) {
        if (kb == w.nkb - 1 && w.tail < BK) {
          // the request, then this fill's landing observed here as well (the
          // stage cannot move on before the answer, so the parity is exact)
          int got = 1;
          if (lane == 0)
            got = mbar_wait(&st.needfix[stage], (fix_bits >> stage) & 1u, abort_flag, hdr, 25) &&
                          mbar_wait(&st.full[stage], phase, abort_flag, hdr, 27)
                      ? 1
                      : 0;
          got = __shfl_sync(0xffffffffu, got, 0);
          __syncwarp();
          fix_bits ^= 1u << stage;
          if (!got) {
            ok = false;
            break;
          }
          // rows tail..63 of every box: 8 16-byte pieces per 128-byte row
          const int nz = (BK - w.tail) * 8;
          uint8_t* a = sA + stage * A_BYTES;
          for (int i = lane; i < (BM / 64) * nz; i += 32) {
            const int box = i / nz, j = i - box * nz;
            *reinterpret_cast<uint4*>(a + box * BOX_BYTES + (w.tail + (j >> 3)) * 128 +
                                      (j & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          if (w.past_end) {
            uint8_t* b = sB + stage * B_BYTES;
            for (int i = lane; i < (UMMA_N / 64) * nz; i += 32) {
              const int box = i / nz, j = i - box * nz;
              *reinterpret_cast<uint4*>(b + box * BOX_BYTES + (w.tail + (j >> 3)) * 128 +
                                        (j & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&st.fixed[stage]);
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int half = ew >> 2;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const WTile w = wtile(off, E, mtc, ntc, tile);
      if (!mbar_wait(&st.tmem_full[acc], acc_phase, abort_flag, hdr, 24)) break;
      tc_fence_after();
      const bool empty = w.nkb == 0;
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
      // 32 columns at a time: lane = row writes its 16-byte pieces q at
      // q ^ (row & 7) (eight rows' writes of one q cover all 32 banks); then
      // lanes 8i .. 8i+7 read one row's 128 bytes and store them together
      float* buf = reinterpret_cast<float*>(sE + ew * EPI_BYTES);
      const int rr = lane >> 3, q = lane & 7;  // read side: row within 4, piece
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
#pragma unroll
        for (int p = 0; p < 8; ++p)
          *reinterpret_cast<uint4*>(buf + lane * 32 + ((p ^ (lane & 7)) << 2)) =
              make_uint4(r[32 * ch + 4 * p], r[32 * ch + 4 * p + 1], r[32 * ch + 4 * p + 2],
                         r[32 * ch + 4 * p + 3]);
        __syncwarp();
        const int n = w.n0 + cbase + 32 * ch + 4 * q;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int row = 4 * i + rr;
          const int mm = w.m0 + quarter * 32 + row;
          const float4 v =
              *reinterpret_cast<const float4*>(buf + row * 32 + ((q ^ (row & 7)) << 2));
          if (mm < M && n + 4 <= N) {
            float* orow = mm < m_split
                              ? out + ((size_t)w.e * m_split + mm) * N
                              : out2 + ((size_t)w.e * (M - m_split) + (mm - m_split)) * N;
            *reinterpret_cast<float4*>(orow + n) = v;
          }
        }
        __syncwarp();
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

// [rows, C] bf16 row-major (row stride ld), box [64 rows, 64 columns],
// 128-byte swizzle: a tile of an MN-major operand.
bool map_mn(CUtensorMap* m, const void* base, uint64_t C, uint64_t rows, uint64_t ld) {
  EncodeTiledFn enc = encode_fn_wgrad();
  if (!enc) return false;
  cuuint64_t gdim[2] = {C, rows};
  cuuint64_t gstride[1] = {ld * 2};
  cuuint32_t box[2] = {64, BK};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// out[e] = A_e^T B_e over rows [off_e, off_{e+1}) of A [rows, M] (row stride
// lda) and B [rows, N] (row stride ldb), bf16, lda and ldb multiples of 8;
// rows m < m_split of each expert's [M, N] result go to out [E, m_split, N],
// the rest to out2 [E, M - m_split, N] (fp32).
cudaError_t launch_wgrad_tc(const void* A, int64_t lda, const void* B, int64_t ldb,
                            int64_t rows, const int32_t* off, int E, int M, int N, int m_split,
                            float* out, float* out2, int32_t* hdr, cudaStream_t s) {
  CUtensorMap ma, mb;
  if (!map_mn(&ma, A, (uint64_t)M, (uint64_t)rows, (uint64_t)lda) ||
      !map_mn(&mb, B, (uint64_t)N, (uint64_t)rows, (uint64_t)ldb))
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
                    ma, mb, off, E, M, N, m_split, out, out2, hdr);
}

}  // namespace moe
