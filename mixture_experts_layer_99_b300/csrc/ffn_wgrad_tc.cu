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
// boxes [64 rows x 64 n]. PAIR: clusters of two CTAs share 256 x 256 tiles
// through cta_group::2 MMAs, as in the grouped GEMM: each CTA loads its 128 m
// columns of A and its 128 n columns of B (32 KB per K step instead of 48,
// six stages), the even CTA issues the MMAs for both and each CTA drains its
// own 128 accumulator rows. A tail block is then fixed up in both CTAs: the
// even CTA's MMA thread asks both fix-up warps (the odd CTA's remotely) after
// the stage's fill has landed in both, and waits for both answers. The epilogue writes fp32 rows; an expert without
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
constexpr int A_BYTES = BM * BK * 2;       // 16 KB
constexpr int TMEM_COLS = 2 * UMMA_N;

constexpr int BOX_BYTES = 64 * BK * 2;     // one [64 rows x 64] box, 8 KB

template <bool PAIR>
struct WShape {
  static constexpr int STAGES = PAIR ? 6 : 4;
  static constexpr int BM_T = PAIR ? 2 * BM : BM;                // tile rows (m)
  static constexpr int B_COLS = PAIR ? UMMA_N / 2 : UMMA_N;      // B columns per CTA
  static constexpr int B_STAGE = B_COLS * BK * 2;                // 16 or 32 KB
};

template <int STAGES>
struct Smem {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t needfix[STAGES];  // the MMA has a tail block in this stage
  uint64_t fixed[STAGES];    // its rows past the expert are zero (both CTAs': PAIR)
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t final_bar;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr int EPI_BYTES = 32 * 32 * 4;     // one warp's 32 x 32 fp32 block
template <bool PAIR>
constexpr size_t smem_bytes_w() {
  using S = WShape<PAIR>;
  return 1024 + S::STAGES * (A_BYTES + S::B_STAGE) + EPI_WARPS * EPI_BYTES +
         sizeof(Smem<S::STAGES>);
}
static_assert(smem_bytes_w<false>() <= 227 * 1024, "shared memory");
static_assert(smem_bytes_w<true>() <= 227 * 1024, "shared memory");

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
                                       int tile, int bm_t) {
  WTile w;
  const int per = mtc * ntc;
  w.e = tile / per;
  const int local = tile - w.e * per;
  w.m0 = (local % mtc) * bm_t;
  w.n0 = (local / mtc) * UMMA_N;
  w.row0 = __ldg(off + w.e);
  const int rows = __ldg(off + w.e + 1) - w.row0;
  w.nkb = rows > 0 ? (rows + BK - 1) / BK : 0;
  w.tail = rows - (w.nkb - 1) * BK;
  w.past_end = w.row0 + w.nkb * BK > __ldg(off + E);
  return w;
}

template <bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    wgrad_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB, const int32_t* __restrict__ off,
                    int E, int M, int N, int m_split, float* __restrict__ out,
                    float* __restrict__ out2, int32_t* __restrict__ hdr) {
  using S = WShape<PAIR>;
  constexpr int STAGES = S::STAGES;
  constexpr int B_STAGE = S::B_STAGE;
  constexpr int BM_T = S::BM_T;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint8_t* sE = smem + STAGES * (A_BYTES + B_STAGE);
  Smem<STAGES>& st = *reinterpret_cast<Smem<STAGES>*>(sE + EPI_WARPS * EPI_BYTES);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;   // tile owner
  const int n_units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&st.full[s], 1);
      mbar_init(&st.empty[s], 1);
      mbar_init(&st.needfix[s], 1);
      mbar_init(&st.fixed[s], PAIR ? 2 : 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&st.tmem_full[a], 1);
      mbar_init(&st.tmem_empty[a], PAIR ? 2 * EPI_WARPS : EPI_WARPS * 32);
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
    if (PAIR) {
      tmem_alloc_pair(&st.tmem_base, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&st.tmem_base, TMEM_COLS);
      tmem_relinquish();
    }
  }
  pdl_wait();
  tc_fence_before();
  if (PAIR) cluster_sync();  // both CTAs' barriers exist before any remote signal
  else __syncthreads();
  tc_fence_after();

  const int mtc = (M + BM_T - 1) / BM_T, ntc = (N + UMMA_N - 1) / UMMA_N;
  const int total = E * mtc * ntc;
  const uint32_t tmem_base = st.tmem_base;
  volatile int* abort_flag = &st.abort_flag;
  bool aborted = false;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = unit; tile < total && ok; tile += n_units) {
        const WTile w = wtile(off, E, mtc, ntc, tile, BM_T);
        const int am = w.m0 + (int)rank * BM;              // this CTA's m columns
        const int bn = w.n0 + (int)rank * S::B_COLS;       // and n columns
        for (int kb = 0; kb < w.nkb; ++kb) {
          if (!mbar_wait(&st.empty[stage], phase ^ 1u, abort_flag, hdr, 21)) {
            ok = false;
            break;
          }
          const int row = w.row0 + kb * BK;
          uint8_t* a_dst = sA + stage * A_BYTES;
          uint8_t* b_dst = sB + stage * B_STAGE;
          if (PAIR) {
            // both CTAs' fills complete on the even CTA's `full` barrier
            const uint32_t bar = cluster_addr(&st.full[stage], 0);
            if (rank == 0) mbar_expect_tx(&st.full[stage], 2u * (A_BYTES + B_STAGE));
#pragma unroll
            for (int c = 0; c < BM / 64; ++c)
              tma_load_2d_pair(a_dst + c * BOX_BYTES, &tmA, bar, am + 64 * c, row);
#pragma unroll
            for (int c = 0; c < S::B_COLS / 64; ++c)
              tma_load_2d_pair(b_dst + c * BOX_BYTES, &tmB, bar, bn + 64 * c, row);
          } else {
            mbar_expect_tx(&st.full[stage], A_BYTES + B_STAGE);
#pragma unroll
            for (int c = 0; c < BM / 64; ++c)
              tma_load_2d(a_dst + c * BOX_BYTES, &tmA, &st.full[stage], am + 64 * c, row);
#pragma unroll
            for (int c = 0; c < S::B_COLS / 64; ++c)
              tma_load_2d(b_dst + c * BOX_BYTES, &tmB, &st.full[stage], bn + 64 * c, row);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        aborted = true;
        // let the copies already issued land before the CTA exits (each wait
        // time-limited); a pair's fills complete on the even CTA's barriers,
        // so only it can watch them, the odd CTA relies on the closing delay
        if (!PAIR || rank == 0) {
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
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // A and B MN-major (bits 15 and 16)
      constexpr uint32_t IDESC = idesc_bf16_f32(BM_T, UMMA_N) | (1u << 15) | (1u << 16);
      int stage = 0, acc = 0, n_local = 0;
      uint32_t phase = 0, acc_phase = 0, fix_bits = 0;
      bool ok = true;
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
      const uint32_t peer_needfix0 = PAIR ? cluster_addr(&st.needfix[0], 1) : 0u;
      for (int tile = unit; tile < total && ok; tile += n_units) {
        const WTile w = wtile(off, E, mtc, ntc, tile, BM_T);
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
          // a tail block: hand the landed stage to the fix-up warp(s) and wait
          // until its rows past the expert are zero (one request at a time
          // per stage, so both sides' parities stay in step)
          if (kb == w.nkb - 1 && w.tail < BK) {
            mbar_arrive(&st.needfix[stage]);
            if (PAIR) mbar_arrive_cluster(peer_needfix0 + (uint32_t)(stage * 8));
            const bool got = mbar_wait(&st.fixed[stage], (fix_bits >> stage) & 1u, abort_flag,
                                       hdr, 26);
            fix_bits ^= 1u << stage;
            if (!got) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
          // 64-column boxes 8 KB apart, K advanced by two 8-row atoms per MMA
          const uint64_t adesc = sdesc_mnmajor_sw128(a0 + stage * A_BYTES, BOX_BYTES);
          const uint64_t bdesc = sdesc_mnmajor_sw128(b0 + stage * B_STAGE, BOX_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            if (PAIR)
              umma_bf16_pair(d_tmem, adesc + (uint64_t)(kk * 128), bdesc + (uint64_t)(kk * 128),
                             IDESC, accum);
            else
              umma_bf16(d_tmem, adesc + (uint64_t)(kk * 128), bdesc + (uint64_t)(kk * 128), IDESC,
                        accum);
          }
          if (PAIR) umma_commit_pair(&st.empty[stage]);
          else umma_commit(&st.empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        // also for an expert without rows: the epilogue then writes zeros
        if (PAIR) umma_commit_pair(&st.tmem_full[acc]);
        else umma_commit(&st.tmem_full[acc]);
        ++n_local;
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (PAIR && ok) {
        // Both CTAs' epilogues release each accumulator on this CTA's
        // `tmem_empty`; take the releases of the last two tiles so that no
        // remote arrive lands after the CTA has exited.
        for (int i = (n_local > 2 ? n_local - 2 : 0); i < n_local && ok; ++i)
          ok = mbar_wait(&st.tmem_empty[i & 1], (uint32_t)((i >> 1) & 1), abort_flag, hdr, 28);
      }
      if (!ok) {
        aborted = true;
        if (PAIR) umma_commit_pair(&st.final_bar);
        else umma_commit(&st.final_bar);
        volatile int no_abort = 0;
        mbar_wait(&st.final_bar, 0, &no_abort, nullptr, 0);
      }
    }
  } else if (warp == FIX_WARP) {
    // Serves the MMA's requests for tail blocks in order: zeroes the rows of
    // this CTA's part of the stage past the expert's end (whole 128-byte
    // lines, which the swizzle only permutes within) and answers through
    // the even CTA's `fixed`.
    int stage = 0;
    uint32_t phase = 0, fix_bits = 0;
    bool ok = true;
    const uint32_t fixed0 = PAIR ? cluster_addr(&st.fixed[0], 0) : 0u;
    for (int tile = unit; tile < total && ok; tile += n_units) {
      const WTile w = wtile(off, E, mtc, ntc, tile, BM_T);
      for (int kb = 0; kb < w.nkb; ++kb) {
        if (kb == w.nkb - 1 && w.tail < BK) {
          // the request (sent once the fill has landed in both CTAs), and in
          // a single CTA this fill's landing observed here as well (the stage
          // cannot move on before the answer, so the parity is exact)
          int got = 1;
          if (lane == 0) {
            got = mbar_wait(&st.needfix[stage], (fix_bits >> stage) & 1u, abort_flag, hdr, 25)
                      ? 1
                      : 0;
            if (got && !PAIR)
              got = mbar_wait(&st.full[stage], phase, abort_flag, hdr, 27) ? 1 : 0;
          }
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
            uint8_t* b = sB + stage * B_STAGE;
            for (int i = lane; i < (S::B_COLS / 64) * nz; i += 32) {
              const int box = i / nz, j = i - box * nz;
              *reinterpret_cast<uint4*>(b + box * BOX_BYTES + (w.tail + (j >> 3)) * 128 +
                                        (j & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          // the zeros before the (possibly the other CTA's) MMA reads them
          if (PAIR) fence_proxy_async_all();
          else fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (PAIR) mbar_arrive_cluster(fixed0 + (uint32_t)(stage * 8));
            else mbar_arrive(&st.fixed[stage]);
          }
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp >= 2 && warp < 2 + EPI_WARPS) {
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int half = ew >> 2;
    const uint32_t empty_cl0 = PAIR ? cluster_addr(&st.tmem_empty[0], 0) : 0u;
    const uint32_t empty_cl1 = PAIR ? cluster_addr(&st.tmem_empty[1], 0) : 0u;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = unit; tile < total; tile += n_units) {
      const WTile w = wtile(off, E, mtc, ntc, tile, BM_T);
      if (!mbar_wait(&st.tmem_full[acc], acc_phase, abort_flag, hdr, 24)) {
        aborted = true;
        break;
      }
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
      if (PAIR) {
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc == 0 ? empty_cl0 : empty_cl1);
      } else {
        mbar_arrive(&st.tmem_empty[acc]);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
      // 32 columns at a time: lane = row writes its 16-byte pieces q at
      // q ^ (row & 7) (eight rows' writes of one q cover all 32 banks); then
      // lanes 8i .. 8i+7 read one row's 128 bytes and store them together
      float* buf = reinterpret_cast<float*>(sE + ew * EPI_BYTES);
      const int rr = lane >> 3, q = lane & 7;  // read side: row within 4, piece
      const int mrow0 = w.m0 + (int)rank * BM + quarter * 32;  // this warp's first row
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
          const int mm = mrow0 + row;
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
  if (PAIR) {
    // A CTA that gave up may still have copies in flight that signal or fill
    // the pair's shared memory; both give them a further 200 us to land
    // before either exits.
    if (__syncthreads_or(aborted ? 1 : 0)) {
      const uint64_t t0 = globaltimer();
      while (globaltimer() - t0 < 200000ull) {
      }
    }
    __syncwarp();
    cluster_sync();
  } else {
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1) {
    if (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
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

// Clusters of two of the pair kernel resident at once on this device
// (queried once per device), or -1 if none fit.
static int wgrad_pair_units() {
  static int units[64] = {};  // 0 unknown, -1 no pairs, else clusters resident at once
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  if (units[dev] == 0) {
    auto kernel = wgrad_tc_kernel<true>;
    constexpr size_t SMEM = smem_bytes_w<true>();
    int n = 0;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM) ==
        cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * (unsigned)device_sm_count());
      cfg.blockDim = dim3(NUM_THREADS);
      cfg.dynamicSmemBytes = SMEM;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();  // a failed query leaves no sticky error behind
    units[dev] = n > 0 ? n : -1;
  }
  return units[dev];
}

// out[e] = A_e^T B_e over rows [off_e, off_{e+1}) of A [rows, M] (row stride
// lda) and B [rows, N] (row stride ldb), bf16, lda and ldb multiples of 8;
// rows m < m_split of each expert's [M, N] result go to out [E, m_split, N],
// the rest to out2 [E, M - m_split, N] (fp32). 256 x 256 tiles on CTA pairs
// when M >= 512 and there are at most 16 groups, else 128 x 256 tiles on
// single CTAs. Measured on B300 (same box, alternating builds, bit-identical
// gradients; backward per call): switch_top1 0.421 -> 0.411 ms, sweep_e16_k4
// 0.735 -> 0.720 ms, mixtral 23.8 -> 23.0 ms, but the long tail (64 experts,
// most of whose tiles are a few rows and all stores) 1.63 -> 1.70 ms.
cudaError_t launch_wgrad_tc(const void* A, int64_t lda, const void* B, int64_t ldb,
                            int64_t rows, const int32_t* off, int E, int M, int N, int m_split,
                            float* out, float* out2, int32_t* hdr, cudaStream_t s) {
  CUtensorMap ma, mb;
  if (!map_mn(&ma, A, (uint64_t)M, (uint64_t)rows, (uint64_t)lda) ||
      !map_mn(&mb, B, (uint64_t)N, (uint64_t)rows, (uint64_t)ldb))
    return cudaErrorInvalidValue;
  const int pair_units = (M >= 512 && E <= 16) ? wgrad_pair_units() : -1;
  if (pair_units > 0) {
    const int64_t tiles = (int64_t)E * ((M + 2 * BM - 1) / (2 * BM)) * ((N + UMMA_N - 1) / UMMA_N);
    const int64_t units = tiles < pair_units ? (tiles > 0 ? tiles : 1) : pair_units;
    return launch_pdl_cluster(wgrad_tc_kernel<true>, dim3((unsigned)(2 * units)),
                              dim3(NUM_THREADS), smem_bytes_w<true>(), 2, s, ma, mb, off, E, M,
                              N, m_split, out, out2, hdr);
  }
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(wgrad_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_bytes_w<false>());
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int64_t tiles = (int64_t)E * ((M + BM - 1) / BM) * ((N + UMMA_N - 1) / UMMA_N);
  const int sms = device_sm_count();
  const int grid = (int)(tiles < sms ? tiles : sms);
  return launch_pdl(wgrad_tc_kernel<false>, dim3(grid > 0 ? grid : 1), dim3(NUM_THREADS),
                    smem_bytes_w<false>(), s, ma, mb, off, E, M, N, m_split, out, out2, hdr);
}

}  // namespace moe
