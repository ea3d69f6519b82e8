// Grouped expert FFN on the 5th-generation tensor cores (tcgen05 + TMEM),
// operands staged by TMA. bf16 in, fp32 accumulation in TMEM.
//
// The expert FFN of the kwkr.cn MoE article ("MoE sparse activation: from
// the math to the code"), section 3.1 (Linear -> GELU -> Linear), with the
// SwiGLU form W2 (silu(W1 x) * (W3 x)) for the 4096 -> 14336 experts of the
// lpnh.cn MoE guide, section 3.2. The per-expert loop of the article's
// section 3.2 becomes one persistent launch per GEMM over all experts'
// tiles; expert e owns packed rows [offset_e, offset_{e+1}).
//
// Kernel layout (one CTA per SM, 320 threads):
//   warp 0      TMA producer: A tile [128 x 64] and B tile [256 x 64] per stage
//   warp 1      TMEM owner and MMA issuer (one thread), 128 x 256 x 16 MMAs
//   warps 2-9   epilogue: TMEM -> registers -> activation -> bf16 -> global
// With many rows per expert the same kernel runs as CTA pairs (clusters of
// two): 256 x 256 tiles, M = 256 MMAs issued by the even CTA, each CTA
// loading its 128 rows of A and 128 of the 256 rows of B.
// Two 256-column fp32 accumulators in TMEM let the epilogue of one tile run
// under the MMAs of the next. M-tiles never cross an expert boundary: a tile
// that starts at row offset_e + 128 i loads rows of the next expert (or TMA
// zero fill past the buffer) and the epilogue masks them out.
//
// GEMM1 (GELU):   h[r, n] = gelu(sum_k xd[r,k] W1[e,n,k] + b1[e,n])   tile N = 256
// GEMM1 (SwiGLU): B tile = 128 rows of W1 then the same 128 rows of W3, so one
//                 N = 256 MMA yields gate and up: h = silu(gate) * up   tile N = 128
// GEMM2:          Y[r, n] = sum_k h[r,k] W2[e,n,k] (+ b2[e,n])        tile N = 256
//
// Inside the fused layer call, for k = 1 every token has at most one kept
// slot, so GEMM2 (SCATTER) scales its row by the gate and writes
// y[token_of_row[r]] directly: the combine y_t = g_t E(x_t) of the kwkr.cn
// article, section 2.1, with no Y buffer and no combine kernel. (Gathering
// GEMM1's A rows by token with TMA gather4 instead of a packed copy was
// measured 2x slower on B300: 33 TMA operations per K step instead of 2.)
#include "moe_internal.h"
#include "tc_ptx.cuh"

#include <math.h>
#include <mutex>

namespace moe {
namespace {

using namespace ptx;

constexpr int BM = 128;
constexpr int BK = 64;       // one 128-byte swizzle row of bf16
constexpr int UMMA_N = 256;
constexpr int UMMA_K = 16;
constexpr int A_BYTES = BM * BK * 2;          // 16 KB
constexpr int B_BYTES = UMMA_N * BK * 2;      // 32 KB
constexpr int TMEM_COLS = 2 * UMMA_N;         // two accumulators

// kBwdGelu / kBwdSwiglu: the backward pass's dh = dY W2 GEMM, whose epilogue
// multiplies by the activation's derivative at the saved pre-activations.
enum Mode { kPlain = 0, kGelu = 1, kSwiglu = 2, kBwdGelu = 3, kBwdSwiglu = 4 };

// Pipeline shape: operand stages and output staging buffers per epilogue
// warp. Four 48 KB stages and two 2 KB buffers per warp fill the 227 KB
// (measured on B300 against 3 stages + 4 buffers: 1.4 % faster on the
// switch_top1 FFN, equal on the other workloads, and equal to 4 + 1).
// EPIW is the number of epilogue warps (a multiple of four, since warp w
// reads TMEM lanes 32 (w % 4) .. + 31): the CTA has 64 + 32 EPIW threads.
// Sixteen epilogue warps (four per TMEM lane quarter, 96 registers each,
// with 4 stages + 1 staging buffer, or 3 + 2) measured on B300 against eight:
// switch_top1 layer call 2.7 % faster, long tail 0.8 % (3 + 2: 7 %) slower,
// mixtral equal, so the forward keeps eight.
template <int STAGES_, int OUT_BUFS_, int EPIW_ = 8>
struct Pipe {
  static constexpr int STAGES = STAGES_;
  static constexpr int OUT_BUFS = OUT_BUFS_;
  static constexpr int EPIW = EPIW_;
  static constexpr int THREADS = 64 + 32 * EPIW_;
};
// forward GEMMs
using PipeShape = Pipe<4, 2>;
// A CTA of a pair stages 32 KB per K step, so six stages fit.
using PipePairShape = Pipe<6, 2>;
// GEMM1 with the GELU epilogue in pairs over a short K (at most 2048): each
// tile's MMAs are short (16-32 K steps), so the activation and stores of the
// 256 x 256 tile co-bound it with eight epilogue warps; sixteen (one staging
// buffer each, 96 registers a thread) halve that time. Measured on B300
// (layer call, alternating builds, identical outputs): switch_top1 0.1635 /
// 0.1612 -> 0.1592 / 0.1584 ms (GEMM1 80.8 -> 75.7 us), sweep_e16_k4 0.3179 ->
// 0.3155 ms; mixtral (SwiGLU, K = 4096) equal, GEMM2 slightly slower, so
// those keep eight.
using PipePairWideEpi = Pipe<6, 1, 16>;

template <int STAGES>
struct SmemTail {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t final_bar;
  uint32_t tmem_base;
  int abort_flag;
  int n_tiles_total;
  int n_heavy_tiles;        // tiles of the heavy experts (the first block of tbase)
  int tbase[kMaxE + 1];     // first tile of each expert, in the order of perm
  uint8_t perm[kMaxE];      // heavy experts by id, then light experts by id
};

// An expert with at most this many m-tiles is "light": each of its (expert,
// n-tile) weight slabs serves one or two tiles, so its tiles read more bytes
// from DRAM per MMA than DRAM can deliver to every SM at once. The others
// ("heavy") reuse a slab over three or more tiles from L2 and are bound by the
// tensor cores. See tile_info.
constexpr int kLightMTiles = 2;

// Epilogue staging: each epilogue warp writes its 32 rows x 32 columns of
// bf16 output (2 KB) here and stores it with one TMA bulk tensor store, so
// global writes are whole 64-byte row segments instead of 16-byte pieces of
// 32 different rows.
constexpr int STAGE_OUT_BYTES = 32 * 32 * 2;
// B bytes per CTA and stage: the whole 256-row B tile, or half of it in a pair
template <bool PAIR>
__host__ __device__ constexpr int stage_b_bytes() {
  return PAIR ? B_BYTES / 2 : B_BYTES;
}
template <bool PAIR, class PIPE>
constexpr size_t smem_bytes() {
  return 1024 /*align slack*/ + PIPE::STAGES * (A_BYTES + stage_b_bytes<PAIR>()) +
         PIPE::EPIW * PIPE::OUT_BUFS * STAGE_OUT_BYTES + sizeof(SmemTail<PIPE::STAGES>);
}
static_assert(smem_bytes<false, PipeShape>() <= 227 * 1024, "shared memory");
static_assert(smem_bytes<true, PipePairShape>() <= 227 * 1024, "shared memory");
static_assert(smem_bytes<true, PipePairWideEpi>() <= 227 * 1024, "shared memory");

// GELU(u) = u/2 (1 + erf(u / sqrt 2)) with erf from the rational
// approximation of Abramowitz & Stegun, Handbook of Mathematical Functions,
// formula 7.1.26 (Hastings): for z >= 0, erfc(z) = 1 - erf(z) ~ q(z) with
// q(z) = t (a1 + a2 t + a3 t^2 + a4 t^3 + a5 t^4) exp(-z^2), t = 1/(1 + p z),
// |error| <= 1.5e-7. Since erf is odd, GELU(u) = max(u, 0) - |u| q(|u|/sqrt 2) / 2
// for either sign of u: no branch and no cancellation for negative u.
// With s = z sqrt(log2 e) the exponential is 2^(-s^2) (one ex2) and p z =
// (p / sqrt(log2 e)) s, so z itself is never formed.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float gelu_as(float u) {
  constexpr float kS = 0.84932180028801904f;    // sqrt(log2 e) / sqrt 2
  constexpr float kP = 0.27273748087922250f;    // p / sqrt(log2 e), p = 0.3275911
  const float s = fabsf(u) * kS;
  const float t = __fdividef(1.f, fmaf(kP, s, 1.f));
  const float e = ex2_approx(-s * s);
  float poly = fmaf(1.061405429f, t, -1.453152027f);
  poly = fmaf(poly, t, 1.421413741f);
  poly = fmaf(poly, t, -0.284496736f);
  poly = fmaf(poly, t, 0.254829592f);
  const float w = (-0.5f * fabsf(u)) * t * e;
  return fmaf(w, poly, fmaxf(u, 0.f));
}
// silu(u) = u / (1 + exp(-u)); for large negative u the denominator
// overflows to +inf and the quotient is 0.
__device__ __forceinline__ float silu_f(float u) { return __fdividef(u, 1.f + __expf(-u)); }

// GELU'(u) = Phi(u) + u phi(u), with Phi from the same erfc approximation as
// gelu_as (Phi(u) = 1 - q/2 for u >= 0, q/2 below) and phi(u) =
// exp(-u^2/2) / sqrt(2 pi), which is the ex2 term already at hand.
__device__ __forceinline__ float gelu_grad_as(float u) {
  constexpr float kS = 0.84932180028801904f;    // sqrt(log2 e) / sqrt 2
  constexpr float kP = 0.27273748087922250f;    // p / sqrt(log2 e), p = 0.3275911
  constexpr float kInvSqrt2Pi = 0.39894228040143268f;
  const float s = fabsf(u) * kS;
  const float t = __fdividef(1.f, fmaf(kP, s, 1.f));
  const float e = ex2_approx(-s * s);  // exp(-u^2 / 2)
  float poly = fmaf(1.061405429f, t, -1.453152027f);
  poly = fmaf(poly, t, 1.421413741f);
  poly = fmaf(poly, t, -0.284496736f);
  poly = fmaf(poly, t, 0.254829592f);
  const float half_q = 0.5f * t * poly * e;  // erfc(|u| / sqrt 2) / 2
  const float Phi = u >= 0.f ? 1.f - half_q : half_q;
  return fmaf(u * kInvSqrt2Pi, e, Phi);
}
// sigma(u) and silu'(u) = sigma(u) (1 + u (1 - sigma(u)))
__device__ __forceinline__ float sigmoid_f(float u) { return __fdividef(1.f, 1.f + __expf(-u)); }

// Eight bf16 of a 16-byte vector to fp32.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& q, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

struct TileInfo {
  int e, m0, mend, n0;
};

// tile -> (expert, first row, end row of the expert, first output column);
// the expert offsets are read through the read-only cache.
// The tiles of light experts (weight streaming) are spread evenly among those
// of heavy experts (tensor-bound) instead of all coming last: tile p is the
// cl(p)-th light tile when cl(p) = floor((p+1) nL / total) steps up at p, else
// the (p - cl(p))-th heavy tile, so every run of consecutive tiles (one wave
// of the persistent grid) holds both kinds in the same proportion and the
// weight streams overlap the MMAs. Within each kind the order stays expert by
// expert, n-tile by n-tile, m-tile fastest (an n-tile's weight slab is read
// by its m-tiles together, while it is in L2).
template <int BM_T, class ST>
__device__ __forceinline__ TileInfo tile_info(const ST& st, const int32_t* __restrict__ off,
                                              int E, int n_tiles_n, int tile, int bn_out) {
  const int total = st.n_tiles_total, nH = st.n_heavy_tiles;
  const int64_t nL = total - nH;
  const int cl = (int)((int64_t)(tile + 1) * nL / total);
  const int cp = (int)((int64_t)tile * nL / total);
  const int q = cl > cp ? nH + cl - 1 : tile - cl;   // index in tbase order
  int lo = 0, hi = E - 1;  // largest position with tbase[pos] <= q
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (st.tbase[mid] <= q) lo = mid;
    else hi = mid - 1;
  }
  const int e = st.perm[lo];
  const int local = q - st.tbase[lo];
  const int o0 = __ldg(off + e), o1 = __ldg(off + e + 1);
  const int mt = (o1 - o0 + BM_T - 1) / BM_T;
  TileInfo ti;
  ti.e = e;
  ti.m0 = o0 + (local % mt) * BM_T;
  ti.mend = o1;
  ti.n0 = (local / mt) * bn_out;
  return ti;
}

// KEEP (the training forward's GEMM1): 32 pre-activation values of this
// lane's row, columns col .. col + 31 of the kept [rows, ld] bf16 tensor, the
// same way the epilogue stores its output: through the warp's staging buffer
// and one TMA store when the warp's 32 rows all belong to the expert and the
// columns fit (col_ok), else direct stores of a valid row's whole 8-column
// pieces (up to ncols).
template <int OUT_BUFS>
__device__ __forceinline__ void keep_store(const float* vv, const CUtensorMap* map,
                                           uint8_t* my_out0, int& n_stores, int lane,
                                           bool full, bool row_ok, int col, int ncols,
                                           int col_off, int wrow0, __nv_bfloat16* row_ptr) {
  uint4 pk[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&pk[q]);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      h2[j] = __floats2bfloat162_rn(vv[8 * q + 2 * j], vv[8 * q + 2 * j + 1]);
  }
  if (full) {
    uint8_t* my_out = my_out0 + (n_stores % OUT_BUFS) * STAGE_OUT_BYTES;
    ++n_stores;
    if (lane == 0) {
      if (OUT_BUFS == 1) bulk_wait_read0();
      else bulk_wait_read<OUT_BUFS - 1>();
    }
    __syncwarp();
    uint4* dst = reinterpret_cast<uint4*>(my_out + lane * 64);
    const int sw = (lane >> 1) & 3;
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q ^ sw] = pk[q];
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(map, my_out, col + col_off, wrow0);
      bulk_commit();
    }
  } else if (row_ok) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (col + 8 * q + 8 <= ncols)
        *reinterpret_cast<uint4*>(row_ptr + col + col_off + 8 * q) = pk[q];
  }
}

// PAIR: the kernel runs as clusters of two CTAs that share one 256-row tile
// (see the cta_group::2 wrappers): each CTA loads its own 128 rows of A and
// half of the B tile (gate rows for SwiGLU on rank 0, up rows on rank 1), so
// an SM pulls 32 KB per K step instead of 48 KB for the same MMA work. Rank 0
// waits for both CTAs' loads on its own `full` barrier (the peer's TMA
// signals it remotely), issues the M = 256 MMAs and multicasts every commit
// to both CTAs; each CTA's epilogue drains its own TMEM rows and releases the
// accumulator on rank 0's `tmem_empty` (one arrive per warp).
// BMN: B is read MN-major straight from a row-major [E, K, N] tensor (the
// backward's dY W2 and dact [W1; W3] products, no transposed copy of the
// weights): per stage, boxes of [64 K rows x 64 N] side by side; with kb3 <
// num_kb the K blocks from kb3 on come from tmB3 (W3 after W1).
// KEEP (GELU and SwiGLU only): the epilogue also stores the pre-activations
// (after the bias; gate and up for SwiGLU, the up half N columns further)
// through tmKeep / keep, [rows, N] or [rows, 2N].
template <int MODE, bool SCATTER, bool PAIR, class PIPE, bool BMN, bool KEEP = false>
__global__ void __launch_bounds__(PIPE::THREADS, 1)
    grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmB3,
                           const __grid_constant__ CUtensorMap tmOut,
                           const __grid_constant__ CUtensorMap tmKeep,
                           const int32_t* __restrict__ offset, int E, int N, int K,
                           const __nv_bfloat16* __restrict__ bias,
                           __nv_bfloat16* __restrict__ out, int32_t* __restrict__ hdr,
                           const int32_t* __restrict__ o_rows,
                           const float* __restrict__ o_scale,
                           const __nv_bfloat16* __restrict__ pre, int ldo, int kb3,
                           int rows_limit, __nv_bfloat16* __restrict__ keep) {
  static_assert(!KEEP || MODE == kGelu || MODE == kSwiglu, "KEEP is for GEMM1 only");
  constexpr int BN_OUT = MODE == kSwiglu ? 128 : UMMA_N;
  constexpr bool BWD = MODE == kBwdGelu || MODE == kBwdSwiglu;
  constexpr int STAGES = PIPE::STAGES;
  constexpr int OUT_BUFS = PIPE::OUT_BUFS;
  constexpr int EPI_WARPS = PIPE::EPIW;
  constexpr int BM_T = PAIR ? 2 * BM : BM;              // rows of one tile
  constexpr int B_STAGE = stage_b_bytes<PAIR>();         // B bytes per CTA and stage
  constexpr uint32_t TX_BYTES = (PAIR ? 2u : 1u) * (uint32_t)(A_BYTES + B_STAGE);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint8_t* sOut = smem + STAGES * (A_BYTES + B_STAGE);
  SmemTail<STAGES>& st =
      *reinterpret_cast<SmemTail<STAGES>*>(sOut + EPI_WARPS * OUT_BUFS * STAGE_OUT_BYTES);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;   // tile owner
  const int n_units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  // ---- set-up: barriers, TMEM, tile table
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&st.full[s], 1);
      mbar_init(&st.empty[s], 1);
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
    if (MODE == kSwiglu) prefetch_tmap(&tmB3);
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
  const int n_tiles_n = (N + BN_OUT - 1) / BN_OUT;
  if (warp == 2) {
    // Tile table: experts in the order perm (heavy ones by id, then light
    // ones by id), tbase[pos] = tiles of the experts before position pos,
    // m-tiles(e) * n_tiles_n tiles each.
    // The offsets may be a caller's input (moe_expert_ffn): unless offset[0]
    // = 0 <= offset[1] <= ... <= offset[E] <= rows_limit, no tile runs (a
    // negative row would start a TMA store before the tensor) and the status
    // header records MOE_ERR_INVALID_ARG (where = 42).
    bool bad = false;
    int n_heavy_experts = 0, n_heavy_tiles = 0, n_tiles = 0;
    int mts[kMaxE / 32];  // m-tiles of expert 32 i + lane
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {  // pass 1: check, count
      if (32 * i >= E) break;
      const int e = 32 * i + lane;
      int mt = 0;
      if (e < E) {
        const int lo = __ldg(offset + e), hi = __ldg(offset + e + 1);
        bad |= hi < lo || hi > rows_limit || (e == 0 && lo != 0);
        mt = bad ? 0 : (hi - lo + BM_T - 1) / BM_T;
      }
      mts[i] = mt;
      const bool heavy = mt > kLightMTiles;
      n_heavy_experts += __popc(__ballot_sync(0xffffffffu, heavy));
      int th = heavy ? mt * n_tiles_n : 0, t = mt * n_tiles_n;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        th += __shfl_xor_sync(0xffffffffu, th, o);
        t += __shfl_xor_sync(0xffffffffu, t, o);
      }
      n_heavy_tiles += th;
      n_tiles += t;
    }
    bad = __any_sync(0xffffffffu, bad);
    int rank_h = 0, rank_l = 0, base_h = 0, base_l = n_heavy_tiles;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {  // pass 2: positions, bases
      if (bad || 32 * i >= E) break;
      const int e = 32 * i + lane;
      const int mt = mts[i];
      const bool heavy = mt > kLightMTiles;
      const unsigned hb = __ballot_sync(0xffffffffu, e < E && heavy);
      const unsigned lb = __ballot_sync(0xffffffffu, e < E && !heavy);
      const unsigned below = (1u << lane) - 1u;
      int ih = heavy ? mt * n_tiles_n : 0, il = heavy ? 0 : mt * n_tiles_n;
      const int vh = ih, vl = il;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int nh = __shfl_up_sync(0xffffffffu, ih, o);
        const int nl = __shfl_up_sync(0xffffffffu, il, o);
        if (lane >= o) {
          ih += nh;
          il += nl;
        }
      }
      if (e < E) {
        const int pos = heavy ? rank_h + __popc(hb & below)
                              : n_heavy_experts + rank_l + __popc(lb & below);
        st.perm[pos] = (uint8_t)e;
        st.tbase[pos] = heavy ? base_h + ih - vh : base_l + il - vl;
      }
      rank_h += __popc(hb);
      rank_l += __popc(lb);
      base_h += __shfl_sync(0xffffffffu, ih, 31);
      base_l += __shfl_sync(0xffffffffu, il, 31);
    }
    if (lane == 0) {
      st.tbase[E] = bad ? 0 : n_tiles;
      st.n_heavy_tiles = bad ? 0 : n_heavy_tiles;
      st.n_tiles_total = bad ? 0 : n_tiles;
      if (bad && hdr != nullptr && atomicCAS(hdr, 0, (int)MOE_ERR_INVALID_ARG) == 0)
        atomicExch(hdr + 1, 42);
    }
  }
  tc_fence_before();
  if (PAIR) cluster_sync();  // both CTAs' barriers exist before any remote signal
  else __syncthreads();
  tc_fence_after();

  const int total = st.n_tiles_total;
  // When every tile streams a light expert's weights (decode-like batches),
  // tiles go round-robin to as many units as give every one the same number
  // of rounds (the last units one tile fewer): with 649 such tiles on 148
  // units, 57 units would stream a fifth tile alone at the end, each at one
  // SM's share of DRAM; 130 units of five tiles keep DRAM busier to the end.
  // No unit gets more tiles than with all units taking part. Measured on B300
  // (layer call, alternating builds, identical outputs): decode 0.362 ->
  // 0.356 ms; applied to every launch it also made the E = 16 sweep 1 % faster
  // but the long tail, whose heavy and light tiles it redistributes, 0.4 %
  // slower, so only all-light launches use it.
  const int rounds = (total + n_units - 1) / n_units;
  const int n_active =
      (rounds > 0 && st.n_heavy_tiles == 0) ? (total + rounds - 1) / rounds : n_units;
  const int first_tile = unit < n_active ? unit : total;  // idle units take none
  const uint32_t tmem_base = st.tmem_base;
  const int num_kb = (K + BK - 1) / BK;
  volatile int* abort_flag = &st.abort_flag;
  bool aborted = false;

  if (warp == 0) {
    // ================= TMA producer (lane 0)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int tile = first_tile; tile < total && ok; tile += n_active) {
        const TileInfo ti = tile_info<BM_T>(st, offset, E, n_tiles_n, tile, BN_OUT);
        const int a_row = ti.m0 + (int)rank * BM;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&st.empty[stage], phase ^ 1u, abort_flag, hdr, 1)) {
            ok = false;
            break;
          }
          uint8_t* a_dst = sA + stage * A_BYTES;
          uint8_t* b_dst = sB + stage * B_STAGE;
          if (PAIR && BMN) {
            // B as two boxes of [64 K rows x 64 N] per CTA (half of N each)
            const uint32_t bar = cluster_addr(&st.full[stage], 0);
            if (rank == 0) mbar_expect_tx(&st.full[stage], TX_BYTES);
            tma_load_2d_pair(a_dst, &tmA, bar, kb * BK, a_row);
            const CUtensorMap* mb = kb >= kb3 ? &tmB3 : &tmB;
            const int kk = (kb >= kb3 ? kb - kb3 : kb) * BK;
#pragma unroll
            for (int ch = 0; ch < UMMA_N / 2 / 64; ++ch)
              tma_load_3d_pair(b_dst + ch * (BK * 128), mb, bar,
                               ti.n0 + (int)rank * (UMMA_N / 2) + 64 * ch, kk, ti.e);
          } else if (PAIR) {
            const uint32_t bar = cluster_addr(&st.full[stage], 0);
            if (rank == 0) mbar_expect_tx(&st.full[stage], TX_BYTES);
            tma_load_2d_pair(a_dst, &tmA, bar, kb * BK, a_row);
            if (MODE == kSwiglu)
              tma_load_3d_pair(b_dst, rank == 0 ? &tmB : &tmB3, bar, kb * BK, ti.n0, ti.e);
            else
              tma_load_3d_pair(b_dst, &tmB, bar, kb * BK, ti.n0 + (int)rank * (UMMA_N / 2), ti.e);
          } else if (BMN) {
            // B as four boxes of [64 K rows x 64 N]
            const CUtensorMap* mb = kb >= kb3 ? &tmB3 : &tmB;
            const int kk = (kb >= kb3 ? kb - kb3 : kb) * BK;
            constexpr int NCH = (PAIR ? UMMA_N / 2 : UMMA_N) / 64;
            mbar_expect_tx(&st.full[stage], TX_BYTES);
            tma_load_2d(a_dst, &tmA, &st.full[stage], kb * BK, a_row);
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch)
              tma_load_3d(b_dst + ch * (BK * 128), mb, &st.full[stage], ti.n0 + 64 * ch, kk, ti.e);
          } else {
            mbar_expect_tx(&st.full[stage], TX_BYTES);
            tma_load_2d(a_dst, &tmA, &st.full[stage], kb * BK, a_row);
            if (MODE == kSwiglu) {
              tma_load_3d(b_dst, &tmB, &st.full[stage], kb * BK, ti.n0, ti.e);
              tma_load_3d(b_dst + B_STAGE / 2, &tmB3, &st.full[stage], kb * BK, ti.n0, ti.e);
            } else {
              tma_load_3d(b_dst, &tmB, &st.full[stage], kb * BK, ti.n0, ti.e);
            }
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (PAIR && ok) {
        // Every fill is released by a commit that rank 0 multicasts to this
        // CTA's `empty` barrier; take the last releases before leaving so that
        // none of them lands after the CTA has exited.
        for (int j = issued - (issued < STAGES ? issued : STAGES); j < issued && ok; ++j)
          ok = mbar_wait(&st.empty[j % STAGES], (uint32_t)((j / STAGES) & 1), abort_flag, hdr, 5);
      }
      if (!ok) {
        aborted = true;
        // let the copies already issued land before the CTA exits (each wait
        // time-limited). A pair's fills, both CTAs', complete on the even
        // CTA's `full` barriers, so only rank 0 can watch them land; the odd
        // CTA relies on the closing delay below.
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
    // ================= MMA issuer (rank 0 of a pair)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t IDESC =
          BMN ? idesc_bf16_f32_bmn(BM_T, UMMA_N) : idesc_bf16_f32(BM_T, UMMA_N);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int n_local = 0;
      bool ok = true;
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
      for (int tile = first_tile; tile < total && ok; tile += n_active) {
        if (!mbar_wait(&st.tmem_empty[acc], acc_phase ^ 1u, abort_flag, hdr, 2)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * UMMA_N);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&st.full[stage], phase, abort_flag, hdr, 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sdesc_kmajor_sw128(a0 + stage * A_BYTES);
          const uint64_t bdesc = BMN ? sdesc_mnmajor_sw128(b0 + stage * B_STAGE, BK * 128)
                                     : sdesc_kmajor_sw128(b0 + stage * B_STAGE);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            // advance along K: K-major inside the 128-byte swizzle row (16 bf16
            // = 32 B), MN-major by two 8-row swizzle atoms (2048 B)
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            const uint64_t bstep = BMN ? (uint64_t)(kk * 128) : (uint64_t)(kk * 2);
            if (PAIR)
              umma_bf16_pair(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + bstep, IDESC, accum);
            else
              umma_bf16(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + bstep, IDESC, accum);
          }
          if (PAIR) umma_commit_pair(&st.empty[stage]);
          else umma_commit(&st.empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
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
          ok = mbar_wait(&st.tmem_empty[i & 1], (uint32_t)((i >> 1) & 1), abort_flag, hdr, 6);
      }
      if (!ok) {
        aborted = true;
        // wait for the MMAs already issued before TMEM is released
        if (PAIR) umma_commit_pair(&st.final_bar);
        else umma_commit(&st.final_bar);
        volatile int no_abort = 0;
        mbar_wait(&st.final_bar, 0, &no_abort, nullptr, 0);
      }
    }
  } else {
    // ================= epilogue (warps 2 .. 1 + EPI_WARPS)
    const int ew = warp - 2;
    const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31
    const int part = ew >> 2;              // which part (of EPI_WARPS / 4) of the tile's columns
    const uint32_t empty_cl0 = PAIR ? cluster_addr(&st.tmem_empty[0], 0) : 0u;
    const uint32_t empty_cl1 = PAIR ? cluster_addr(&st.tmem_empty[1], 0) : 0u;
    int acc = 0;
    uint32_t acc_phase = 0;
    int n_stores = 0;  // TMA stores issued by this warp (buffer = n_stores % OUT_BUFS)
    for (int tile = first_tile; tile < total; tile += n_active) {
      const TileInfo ti = tile_info<BM_T>(st, offset, E, n_tiles_n, tile, BN_OUT);
      if (!mbar_wait(&st.tmem_full[acc], acc_phase, abort_flag, hdr, 4)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const int wrow0 = ti.m0 + (int)rank * BM + quarter * 32;  // this warp's first row
      const int row = wrow0 + lane;
      const bool row_ok = row < ti.mend;
      const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * UMMA_N);
      int orow_idx = row;
      float oscale = 1.f;
      if (SCATTER) {
        orow_idx = row_ok ? __ldg(o_rows + row) : 0;
        oscale = row_ok ? __ldg(o_scale + orow_idx) : 0.f;
      }
      // all 32 rows of this warp belong to the tile's expert: one TMA store
      // per 32 columns; otherwise (the expert's last, partial tile, or the
      // row scatter) direct stores of the valid rows
      const bool warp_full = !SCATTER && (wrow0 + 32 <= ti.mend);
      uint8_t* my_out0 = sOut + ew * OUT_BUFS * STAGE_OUT_BYTES;
      // The warp's whole slice of the accumulator (UMMA_N / parts fp32
      // columns, or as many gate and as many up columns for SwiGLU) goes to
      // registers with one wait, and the TMEM buffer is handed back to the
      // MMA before the activation and the stores.
      constexpr int PARTS = EPI_WARPS / 4;
      constexpr int OUTC = (MODE == kSwiglu ? 128 : 256) / PARTS;  // output columns per warp
      constexpr int NREG = MODE == kSwiglu ? 2 * OUTC : OUTC;     // accumulator columns per warp
      const int cbase = OUTC * part;                               // tile-local first column
      uint32_t r[NREG];
      if (MODE == kSwiglu) {
#pragma unroll
        for (int ch = 0; ch < OUTC / 32; ++ch) {
          tmem_ld32(t_row + (uint32_t)(cbase + 32 * ch),
                    *reinterpret_cast<uint32_t(*)[32]>(&r[32 * ch]));
          tmem_ld32(t_row + (uint32_t)(128 + cbase + 32 * ch),
                    *reinterpret_cast<uint32_t(*)[32]>(&r[OUTC + 32 * ch]));
        }
      } else {
#pragma unroll
        for (int ch = 0; ch < OUTC / 32; ++ch)
          tmem_ld32(t_row + (uint32_t)(cbase + 32 * ch), *reinterpret_cast<uint32_t(*)[32]>(&r[32 * ch]));
      }
      tmem_ld_wait();
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
#pragma unroll
      for (int ch = 0; ch < OUTC / 32; ++ch) {
        const int c = cbase + 32 * ch;
        float v[32];
        float v2[32];  // kBwdSwiglu: the second output (d up), stored N columns further
        if (MODE == kSwiglu) {
          if constexpr (KEEP) {  // gate a at column n, up at column N + n
            const bool kfull = warp_full && ti.n0 + c + 32 <= N;
            __nv_bfloat16* krow = keep + (size_t)row * (2 * N);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              v[j] = __uint_as_float(r[32 * ch + j]);
              v2[j] = __uint_as_float(r[OUTC + 32 * ch + j]);
            }
            keep_store<OUT_BUFS>(v, &tmKeep, my_out0, n_stores, lane, kfull, row_ok, ti.n0 + c,
                                 N, 0, wrow0, krow);
            keep_store<OUT_BUFS>(v2, &tmKeep, my_out0, n_stores, lane, kfull, row_ok, ti.n0 + c,
                                 N, N, wrow0, krow);
          }
#pragma unroll
          for (int j = 0; j < 32; ++j)
            v[j] = silu_f(__uint_as_float(r[32 * ch + j])) * __uint_as_float(r[OUTC + 32 * ch + j]);
        } else if (BWD) {
          // dh for 32 columns of this row; the saved pre-activations of the
          // same row and columns (gate a and up v for SwiGLU: v at column N + n)
          float a[32];
          const int col0 = ti.n0 + c;
          const __nv_bfloat16* pr = pre + (size_t)row * (MODE == kBwdSwiglu ? 2 * N : N);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w = make_uint4(0, 0, 0, 0);
            if (row_ok && col0 + 8 * q + 8 <= N)
              w = __ldg(reinterpret_cast<const uint4*>(pr + col0) + q);
            bf16x8_to_f32(w, a + 8 * q);
          }
          if (MODE == kBwdGelu) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[32 * ch + j]) * gelu_grad_as(a[j]);
          } else {
            float u2[32];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 w = make_uint4(0, 0, 0, 0);
              if (row_ok && col0 + 8 * q + 8 <= N)
                w = __ldg(reinterpret_cast<const uint4*>(pr + N + col0) + q);
              bf16x8_to_f32(w, u2 + 8 * q);
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float dh = __uint_as_float(r[32 * ch + j]);
              const float sg = sigmoid_f(a[j]);
              const float sl = a[j] * sg;
              v[j] = dh * u2[j] * sg * fmaf(a[j], 1.f - sg, 1.f);  // d gate
              v2[j] = dh * sl;                                    // d up
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[32 * ch + j]);
          if (bias) {
            const __nv_bfloat16* be = bias + (size_t)ti.e * N + ti.n0 + c;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (ti.n0 + c + j < N) v[j] += __bfloat162float(be[j]);
          }
          if (MODE == kGelu) {
            if constexpr (KEEP)  // the pre-activation, bias added
              keep_store<OUT_BUFS>(v, &tmKeep, my_out0, n_stores, lane,
                                   warp_full && ti.n0 + c + 32 <= N, row_ok, ti.n0 + c, N, 0,
                                   wrow0, keep + (size_t)row * N);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = gelu_as(v[j]);
          }
        }
        if (SCATTER) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= oscale;
        }
#pragma unroll
        for (int o = 0; o < (MODE == kBwdSwiglu ? 2 : 1); ++o) {
          const float* vv = o == 0 ? v : v2;
          const int ocol = ti.n0 + c + o * N;  // first output column of this chunk
          uint4 pk[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&pk[q]);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              h2[j] = __floats2bfloat162_rn(vv[8 * q + 2 * j], vv[8 * q + 2 * j + 1]);
          }
          if (warp_full && ti.n0 + c + 32 <= N) {
            // the store that last used this buffer (OUT_BUFS stores ago) must
            // have read it
            uint8_t* my_out = my_out0 + (n_stores % OUT_BUFS) * STAGE_OUT_BYTES;
            ++n_stores;
            if (lane == 0) {
              if (OUT_BUFS == 1) bulk_wait_read0();
              else bulk_wait_read<OUT_BUFS - 1>();
            }
            __syncwarp();
            // 64-byte swizzle (the layout of the store's tensor map): 16-byte
            // chunk q of row r sits at chunk q ^ ((r >> 1) & 3), so the 32
            // rows' writes of one chunk hit all 32 banks (4 wavefronts, not 16)
            uint4* dst = reinterpret_cast<uint4*>(my_out + lane * 64);
            const int sw = (lane >> 1) & 3;
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q ^ sw] = pk[q];
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmOut, my_out, ocol, wrow0);
              bulk_commit();
            }
          } else if (row_ok) {
            __nv_bfloat16* orow2 = out + (size_t)orow_idx * ldo;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int col = ti.n0 + c + 8 * q;
              if (col + 8 <= N) *reinterpret_cast<uint4*>(orow2 + col + o * N) = pk[q];
            }
          }
        }
      }
    }
  }

  if (warp >= 2 && lane == 0) bulk_wait0();  // the epilogue's TMA stores are complete
  tc_fence_before();
  if (PAIR) {
    // A CTA that gave up may still have copies in flight that signal or fill
    // the pair's shared memory. Rank 0 has waited for the fills it armed; the
    // odd CTA cannot observe its own, so both give them a further 200 us to
    // land before either exits.
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

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

// 2-D bf16 [rows, K] row-major, box [128 rows, 64 cols], 128-byte swizzle.
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint64_t ld = 0) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t gdim[2] = {K, rows};
  cuuint64_t gstride[1] = {(ld ? ld : K) * 2};
  cuuint32_t box[2] = {BK, BM};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 [E, N, K] (K contiguous), box [1, box_rows, 64], 128-byte swizzle.
bool make_map_3d(CUtensorMap* m, const void* base, uint64_t K, uint64_t N, uint64_t E,
                 uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t gdim[3] = {K, N, E};
  cuuint64_t gstride[2] = {K * 2, N * K * 2};
  cuuint32_t box[3] = {BK, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstride, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 [rows, N] row-major, box [32 rows, 32 cols], no swizzle: the
// epilogue's output blocks.
bool make_map_out(CUtensorMap* m, const void* base, uint64_t N, uint64_t rows,
                  uint64_t ld = 0) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t gdim[2] = {N, rows};
  cuuint64_t gstride[1] = {(ld ? ld : N) * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, bool SCATTER, bool PAIR, class PIPE, bool BMN, bool KEEP = false>
cudaError_t launch_gemm_p(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b3,
                          const CUtensorMap& o, const int32_t* offset, int E, int N, int K,
                          const void* bias, void* out, int64_t rows_bound, int32_t* hdr,
                          const int32_t* o_rows, const float* o_scale, const void* pre,
                          int ldo, int kb3, cudaStream_t s, const CUtensorMap* keep_map = nullptr,
                          void* keep = nullptr) {
  constexpr size_t SMEM_BYTES = smem_bytes<PAIR, PIPE>();
  auto kernel = grouped_gemm_tc_kernel<MODE, SCATTER, PAIR, PIPE, BMN, KEEP>;
  static int max_units[64] = {};  // per device and instantiation: CTAs (or pairs) at once
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (max_units[dev] == 0) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    int units = device_sm_count();
    if (PAIR) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * units);
      cfg.blockDim = dim3(PIPE::THREADS);
      cfg.dynamicSmemBytes = SMEM_BYTES;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(&units, kernel, &cfg);
      if (e != cudaSuccess) return e;
    }
    if (units <= 0) return cudaErrorInvalidConfiguration;
    max_units[dev] = units;
  }
  constexpr int BN_OUT = MODE == kSwiglu ? 128 : UMMA_N;
  constexpr int BM_T = PAIR ? 2 * BM : BM;
  const int64_t tiles_bound = ((rows_bound + BM_T - 1) / BM_T + E) * ((N + BN_OUT - 1) / BN_OUT);
  int64_t units = tiles_bound < max_units[dev] ? tiles_bound : max_units[dev];
  if (units < 1) units = 1;
  const unsigned grid = (unsigned)(PAIR ? 2 * units : units);
  return launch_pdl_cluster(kernel, dim3(grid), dim3(PIPE::THREADS), SMEM_BYTES, PAIR ? 2 : 1, s, a,
                            b, b3, o, keep_map ? *keep_map : o, offset, E, N, K,
                            static_cast<const __nv_bfloat16*>(bias),
                            static_cast<__nv_bfloat16*>(out), hdr, o_rows, o_scale,
                            static_cast<const __nv_bfloat16*>(pre), ldo > 0 ? ldo : N, kb3,
                            (int)(rows_bound < INT32_MAX ? rows_bound : INT32_MAX),
                            static_cast<__nv_bfloat16*>(keep));
}

// BMN (B MN-major): kb3 is the first K block read through b3 (< 0: none).
template <int MODE, bool SCATTER, bool BMN = false>
cudaError_t launch_gemm(bool pair, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& b3, const CUtensorMap& o, const int32_t* offset, int E,
                        int N, int K, const void* bias, void* out, int64_t rows_bound,
                        int32_t* hdr, const int32_t* o_rows, const float* o_scale,
                        cudaStream_t s, const void* pre = nullptr, int ldo = 0, int kb3 = -1,
                        const CUtensorMap* keep_map = nullptr, void* keep = nullptr) {
  if (!BMN || kb3 < 0) kb3 = (K + BK - 1) / BK;
  if constexpr ((MODE == kGelu || MODE == kSwiglu) && !SCATTER && !BMN) {
    if (keep) {
      if (pair)
        return launch_gemm_p<MODE, false, true, PipePairShape, false, true>(
            a, b, b3, o, offset, E, N, K, bias, out, rows_bound, hdr, o_rows, o_scale, pre, ldo,
            kb3, s, keep_map, keep);
      return launch_gemm_p<MODE, false, false, PipeShape, false, true>(
          a, b, b3, o, offset, E, N, K, bias, out, rows_bound, hdr, o_rows, o_scale, pre, ldo,
          kb3, s, keep_map, keep);
    }
  }
  if (pair) {
    if constexpr (MODE == kGelu && !SCATTER && !BMN) {
      if (K <= 2048)
        return launch_gemm_p<MODE, false, true, PipePairWideEpi, false>(
            a, b, b3, o, offset, E, N, K, bias, out, rows_bound, hdr, o_rows, o_scale, pre, ldo,
            kb3, s);
    }
    return launch_gemm_p<MODE, SCATTER, true, PipePairShape, BMN>(
        a, b, b3, o, offset, E, N, K, bias, out, rows_bound, hdr, o_rows, o_scale, pre, ldo, kb3,
        s);
  }
  return launch_gemm_p<MODE, SCATTER, false, PipeShape, BMN>(a, b, b3, o, offset, E, N, K, bias,
                                                             out, rows_bound, hdr, o_rows,
                                                             o_scale, pre, ldo, kb3, s);
}

}  // namespace

// Whether clusters of two CTAs of the pair kernel can be resident on the
// current device (every pair instantiation takes one CTA per SM: nearly all
// of the shared memory). Queried once per device.
static bool pairs_fit() {
  static int fit[64] = {};  // 0 unknown, 1 yes, 2 no
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (fit[dev] == 0) {
    auto kernel = grouped_gemm_tc_kernel<kPlain, false, true, PipePairShape, false>;
    constexpr size_t SMEM_BYTES = smem_bytes<true, PipePairShape>();
    int n = 0;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2);
      cfg.blockDim = dim3(PipePairShape::THREADS);
      cfg.dynamicSmemBytes = SMEM_BYTES;
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
    fit[dev] = n > 0 ? 1 : 2;
  }
  return fit[dev] == 1;
}

// CTA pairs (256-row tiles) when the experts hold at least 512 rows on
// average (below that a 256-row tile would mostly cover padding), there are
// at most 16 experts, and the device can hold the pair kernel's clusters.
// Measured on B300 (layer call): switch_top1 (E = 8) 0.1550 -> 0.1528 ms,
// mixtral (E = 8) 8.80 -> 8.64 ms; the E = 64 long-tail FFN was 7 % slower
// with pairs, so wide expert sets keep single-CTA tiles.
static bool use_pairs(const moe_config_t& c) {
  return c.E <= 16 && (int64_t)c.T * c.k >= 512 * (int64_t)c.E && pairs_fit();
}

cudaError_t launch_ffn_tc(const moe_config_t& c, const void* xd, const int32_t* offset,
                          const void* W1, const void* W3, const void* W2, const void* b1,
                          const void* b2, void* Y, void* h, int64_t rows_bound, int32_t* hdr,
                          cudaStream_t s, const FfnFusion* fz) {
  CUtensorMap mx, mh, mw1, mw3, mw2, moh, moy;
  const uint64_t R = (uint64_t)rows_bound;
  const bool swiglu = c.act == MOE_ACT_SWIGLU;
  const bool scatter = fz && fz->scatter_rows;
  const bool pair = use_pairs(c);
  // rows of B per CTA and K step: 128 in a pair (half of the 256-row tile),
  // else the whole tile (128 gate + 128 up rows from two maps for SwiGLU)
  const uint32_t b_rows = (pair || swiglu) ? 128 : UMMA_N;
  // the scatter variant stores rows directly; its map is a placeholder
  if (!make_map_out(&moh, h, c.H, R) || !make_map_out(&moy, scatter ? h : Y, scatter ? c.H : c.d, R))
    return cudaErrorInvalidValue;
  if (!make_map_2d(&mx, xd, c.d, R) || !make_map_2d(&mh, h, c.H, R) ||
      !make_map_3d(&mw1, W1, c.d, c.H, c.E, b_rows) ||
      !make_map_3d(&mw2, W2, c.H, c.d, c.E, pair ? 128 : UMMA_N))
    return cudaErrorInvalidValue;
  if (swiglu && !make_map_3d(&mw3, W3, c.d, c.H, c.E, 128)) return cudaErrorInvalidValue;
  if (!swiglu) mw3 = mw1;
  // the pre-activations kept for the backward: [R, H] (GELU, bias added) or
  // [R, 2H] (SwiGLU: gate, then up)
  CUtensorMap mkeep;
  void* keep = fz ? fz->keep_pre : nullptr;
  if (keep && !make_map_out(&mkeep, keep, swiglu ? 2 * (uint64_t)c.H : (uint64_t)c.H, R))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if (swiglu)
    e = launch_gemm<kSwiglu, false>(pair, mx, mw1, mw3, moh, offset, c.E, c.H, c.d, nullptr, h,
                                    rows_bound, hdr, nullptr, nullptr, s, nullptr, 0, -1,
                                    keep ? &mkeep : nullptr, keep);
  else
    e = launch_gemm<kGelu, false>(pair, mx, mw1, mw3, moh, offset, c.E, c.H, c.d, b1, h,
                                  rows_bound, hdr, nullptr, nullptr, s, nullptr, 0, -1,
                                  keep ? &mkeep : nullptr, keep);
  if (e != cudaSuccess) return e;
  if (fz && fz->between && (e = record_stage_event(fz->between, s)) != cudaSuccess) return e;
  const void* b2e = swiglu ? nullptr : b2;
  if (scatter)
    return launch_gemm<kPlain, true>(pair, mh, mw2, mw2, moy, offset, c.E, c.d, c.H, b2e, fz->y,
                                     rows_bound, hdr, fz->scatter_rows, fz->scatter_scale, s);
  return launch_gemm<kPlain, false>(pair, mh, mw2, mw2, moy, offset, c.E, c.d, c.H, b2e, Y,
                                    rows_bound, hdr, nullptr, nullptr, s);
}

// Expert part of the backward pass (tensor cores, bf16):
//   pre  = xd W1^T (+ b1) [R, H]      (SwiGLU: [a | v] = xd [W1; W3]^T, [R, 2H])
//   dact = (dY W2) * act'(pre)        [R, H]  (SwiGLU: [d gate | d up], [R, 2H])
//   dxd  = dact W1                    [R, d]  (SwiGLU: [d gate | d up] [W1; W3])
// The weights are read as stored (W2 [E, d, H], W1 and W3 [E, H, d]: B
// MN-major); W13T [E, d, Hp] (Hp = 2H), the transposed [W1; W3], is used only
// by a SwiGLU hidden size that is not a multiple of 64 (else NULL). The
// pre-activations are recomputed into pre, unless have_pre (the forward kept
// them there).
cudaError_t launch_ffn_bwd_tc(const moe_config_t& c, const void* xd, const int32_t* offset,
                              const void* W1, const void* W3, const void* b1, const void* W2,
                              const void* W13T, const void* dY, void* pre, void* dact,
                              void* dxd, int64_t rows_bound, int32_t* hdr, cudaStream_t s,
                              bool have_pre) {
  const uint64_t R = (uint64_t)rows_bound;
  const bool swiglu = c.act == MOE_ACT_SWIGLU;
  const bool pair = use_pairs(c);
  const uint64_t H = (uint64_t)c.H, d = (uint64_t)c.d, Hp = swiglu ? 2 * H : H;
  const uint32_t box = pair ? 128 : UMMA_N;
  CUtensorMap mxd, mw1, mw3, mpa, mpv, mdy, mw2n, mdact_o, mdact_a, mdxd;
  if (!make_map_2d(&mxd, xd, d, R) || !make_map_3d(&mw1, W1, d, H, c.E, box) ||
      !make_map_out(&mpa, pre, H, R, Hp) || !make_map_2d(&mdy, dY, d, R) ||
      !make_map_3d(&mw2n, W2, H, d, c.E, BK) || !make_map_out(&mdact_o, dact, Hp, R) ||
      !make_map_2d(&mdact_a, dact, Hp, R) || !make_map_out(&mdxd, dxd, d, R))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaSuccess;
  // recomputed pre-activations
  if (!have_pre)
    e = launch_gemm<kPlain, false>(pair, mxd, mw1, mw1, mpa, offset, c.E, c.H, c.d,
                                   swiglu ? nullptr : b1, pre, rows_bound, hdr, nullptr, nullptr,
                                   s, nullptr, (int)Hp);
  if (e != cudaSuccess) return e;
  if (swiglu && !have_pre) {
    if (!make_map_3d(&mw3, W3, d, H, c.E, box) ||
        !make_map_out(&mpv, static_cast<__nv_bfloat16*>(pre) + H, H, R, Hp))
      return cudaErrorInvalidValue;
    e = launch_gemm<kPlain, false>(pair, mxd, mw3, mw3, mpv, offset, c.E, c.H, c.d, nullptr,
                                   static_cast<__nv_bfloat16*>(pre) + H, rows_bound, hdr, nullptr,
                                   nullptr, s, nullptr, (int)Hp);
    if (e != cudaSuccess) return e;
  }
  // dh = dY W2 (W2 [E, d, H] read MN-major), times the activation's derivative
  if (swiglu)
    e = launch_gemm<kBwdSwiglu, false, true>(pair, mdy, mw2n, mw2n, mdact_o, offset, c.E, c.H,
                                             c.d, nullptr, dact, rows_bound, hdr, nullptr,
                                             nullptr, s, pre, (int)Hp);
  else
    e = launch_gemm<kBwdGelu, false, true>(pair, mdy, mw2n, mw2n, mdact_o, offset, c.E, c.H, c.d,
                                           nullptr, dact, rows_bound, hdr, nullptr, nullptr, s,
                                           pre);
  if (e != cudaSuccess) return e;
  // dxd = dact [W1; W3]: W1 (and W3) [E, H, d] read MN-major, W3's K blocks
  // after W1's; a SwiGLU hidden size that is not a multiple of 64 would put
  // one K block across both, so that case reads the transposed copy W13T
  if (!bwd_w13_transposed(c)) {
    CUtensorMap mw1n, mw3n;
    if (!make_map_3d(&mw1n, W1, d, H, c.E, BK) ||
        !make_map_3d(&mw3n, swiglu ? W3 : W1, d, H, c.E, BK))
      return cudaErrorInvalidValue;
    return launch_gemm<kPlain, false, true>(pair, mdact_a, mw1n, mw3n, mdxd, offset, c.E, c.d,
                                            (int)Hp, nullptr, dxd, rows_bound, hdr, nullptr,
                                            nullptr, s, nullptr, 0,
                                            swiglu ? (int)(H / BK) : -1);
  }
  CUtensorMap mw13t;
  if (!W13T || !make_map_3d(&mw13t, W13T, Hp, d, c.E, box)) return cudaErrorInvalidValue;
  return launch_gemm<kPlain, false>(pair, mdact_a, mw13t, mw13t, mdxd, offset, c.E, c.d,
                                    (int)Hp, nullptr, dxd, rows_bound, hdr, nullptr, nullptr, s);
}
cudaError_t launch_router_dx_tc(const void* dz_bf16, int T, int Kp, const void* Wg, int E, int d,
                                const int32_t* off, void* dxr, int32_t* hdr, cudaStream_t s) {
  // W_g [E, d] read MN-major as [K = E (zero beyond E), N = d]
  CUtensorMap ma, mb, mo;
  if (!make_map_2d(&ma, dz_bf16, (uint64_t)Kp, (uint64_t)T) ||
      !make_map_3d(&mb, Wg, (uint64_t)d, (uint64_t)E, 1, BK) ||
      !make_map_out(&mo, dxr, (uint64_t)d, (uint64_t)T))
    return cudaErrorInvalidValue;
  return launch_gemm<kPlain, false, true>(false, ma, mb, mb, mo, off, 1, d, Kp, nullptr, dxr, T,
                                          hdr, nullptr, nullptr, s);
}

}  // namespace moe
