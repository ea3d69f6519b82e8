// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/moe.h"

namespace moe {

// Programmatic dependent launch: the kernels of the layer are launched with
// programmatic stream serialisation, so a kernel is scheduled as soon as every
// CTA of its predecessor has exited and runs its prologue (mbarrier set-up,
// TMEM allocation, tensor-map prefetch) while the predecessor's writes are
// flushed. Each such kernel calls pdl_wait() before its first global-memory
// access; it returns once the predecessor grid has completed and its writes
// are visible. No kernel triggers its dependents early: letting them launch
// at the start of the predecessor (griddepcontrol.launch_dependents) parked
// their CTAs on the SMs the predecessor was still using and made the layer
// slower.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same with a cluster of `cluster_x` CTAs along x (1: no cluster).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               int cluster_x, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster_x > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Records a stage-boundary event on s. Inside a stream capture the record
// becomes an event node of the graph (cudaEventRecordExternal), so the event
// is recorded, and can be timed, each time the graph is replayed.
inline cudaError_t record_stage_event(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  if (cs == cudaStreamCaptureStatusActive)
    return cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  return cudaEventRecord(ev, s);
}

constexpr int kMaxE = 256;
constexpr int kMaxK = 8;

// Router: tokens per tile of the fused router kernel.
constexpr int kRouterTile = 32;
// Dispatch: slots per block of the count / assign kernels.
constexpr int kDispSlotsPerBlock = 1024;

// Device status header at the start of every workspace (int32 words).
enum HeaderWord : int {
  kHdrStatus = 0,   // 0 or a moe_status_t recorded by a kernel
  kHdrWhere = 1,    // which wait gave up
  kHdrBytes = 256,
};

// Checked builds (-DMOE_CHECK): a kernel that indexes with data another
// kernel wrote tests the index first; moe_check returns whether it holds and,
// if not, records MOE_ERR_DEVICE_CHECK and the site in the status header
// (when there is one), and the caller skips the access. Other builds compile
// the test away (moe_check is then constantly true).
#ifdef MOE_CHECK
__device__ __forceinline__ bool moe_check(bool ok, int32_t* hdr, int where) {
  if (!ok && hdr != nullptr && atomicCAS(hdr + kHdrStatus, 0, (int)MOE_ERR_DEVICE_CHECK) == 0)
    atomicExch(hdr + kHdrWhere, where);
  return ok;
}
#else
__device__ __forceinline__ constexpr bool moe_check(bool, int32_t*, int) { return true; }
#endif

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline size_t elem_bytes(const moe_config_t& c) { return c.dtype == MOE_F32 ? 4 : 2; }

// Upper bound on packed rows: every kept slot is one row; sum_e min(count_e, C)
// <= min(T k, E C).
inline int64_t max_rows(const moe_config_t& c) {
  int64_t a = (int64_t)c.T * c.k, b = (int64_t)c.E * c.capacity;
  return a < b ? a : b;
}

// Router grid: a fixed bound (4 blocks on each of 148 SMs), independent of the
// device, so the per-block probability partials (and their fixed-order sum)
// are the same on every device.
constexpr int kRouterMaxBlocks = 592;
inline int router_grid(const moe_config_t& c, int /*unused*/) {
  int tiles = (c.T + kRouterTile - 1) / kRouterTile;
  return tiles < kRouterMaxBlocks ? tiles : kRouterMaxBlocks;
}

// Tensor-core router: tiles of 128 tokens (the MMA's M), at most one CTA per
// SM of a 148-SM B300 (a fixed bound, so the per-CTA partial sums do not
// depend on the device). Cutting the batch into as many smaller tiles as keep
// all 148 SMs busy (147 tiles of 112 tokens at T = 16384 instead of 128 of
// 128) measured no faster on B300: the tile loads are bound by DRAM, not by
// the number of SMs pulling.
constexpr int kRouterTcTile = 128;
constexpr int kRouterTcMaxBlocks = 148;
inline int router_tc_rows(const moe_config_t&) { return kRouterTcTile; }
inline int router_tc_tiles(const moe_config_t& c) {
  const int rows = router_tc_rows(c);
  return (c.T + rows - 1) / rows;
}
inline int router_tc_grid(const moe_config_t& c) {
  const int t = router_tc_tiles(c);
  return t < kRouterTcMaxBlocks ? t : kRouterTcMaxBlocks;
}
// With very few tiles (a batch of at most 16 x 128 tokens) the router splits
// each tile's K range (64-wide blocks) over a cluster of up to 8 CTAs; every
// split is non-empty. Larger batches keep one CTA per tile: measured on B300,
// the split's reduction costs more than it saves once there are 64 tiles.
struct RouterSplit {
  int ksplit, kb_per_split;
};
constexpr int kRouterMaxSplit = 8;  // CTAs of a split cluster (portable cluster size)
inline RouterSplit router_tc_split(const moe_config_t& c) {
  const int tiles = router_tc_tiles(c);
  const int num_kb = (c.d + 63) / 64;
  if (tiles > 16) return RouterSplit{1, num_kb};
  int want = kRouterMaxSplit;
  if (want > num_kb) want = num_kb;
  const int per = (num_kb + want - 1) / want;
  return RouterSplit{(num_kb + per - 1) / per, per};
}
// Probability partials the router writes: one per CTA, or one per tile when split.
inline int router_tc_nparts(const moe_config_t& c) {
  return router_tc_split(c).ksplit > 1 ? router_tc_tiles(c) : router_tc_grid(c);
}

inline int disp_blocks(const moe_config_t& c) {
  int64_t s = (int64_t)c.T * c.k;
  return (int)((s + kDispSlotsPerBlock - 1) / kDispSlotsPerBlock);
}

// Workspace regions (byte offsets, 256-aligned). Computed identically by the
// size query and by every call.
struct WsLayout {
  size_t hdr, router_partial, router_tile_hist, router_split, disp_hist, disp_base, ffn_h, ffn_sched;
  // fused layer intermediates
  size_t logits, topk_idx, topk_gate, slot_of, count, offset, token_of_row, xd, Y,
      prob_sum, f, P, L, dropped, pre;
  // host-io staging
  size_t x_stage, y_stage;
  size_t total_core, total_layer, total_host;
  // shared expert (after total_layer): one-group offsets, hidden rows, output rows
  size_t sh_offset, sh_h, sh_y, total_shared;
};

WsLayout ws_layout(const moe_config_t& c, int num_sms, int H_shared = 0);
int device_sm_count();

// ---- launchers (return cudaError_t of the launch) ----
cudaError_t launch_router(const moe_config_t& c, const void* x, const void* Wg,
                          const float* bias, const float* noise, float* logits,
                          int32_t* idx, float* gate, float* partial, int grid,
                          cudaStream_t s);
bool router_tc_supported(const moe_config_t& c);
cudaError_t launch_router_tc(const moe_config_t& c, const void* x, const void* Wg,
                             const float* bias, const float* noise, float* logits, int32_t* idx,
                             float* gate, float* partial, int32_t* tile_hist, float* split_part,
                             int32_t* hdr, cudaStream_t s);
cudaError_t launch_prob_reduce(const moe_config_t& c, const float* partial, int nparts,
                               float* prob_sum, cudaStream_t s);
cudaError_t launch_dispatch(const moe_config_t& c, const int32_t* idx, const void* x,
                            int32_t* count, int32_t* offset, int32_t* slot_of,
                            int32_t* token_of_row, void* xd, int32_t* hist, int32_t* base,
                            int64_t rows_bound, cudaStream_t s, int32_t* hdr = nullptr);
cudaError_t launch_gather(const moe_config_t& c, const void* x, const int32_t* token_of_row,
                          const int32_t* offset, void* xd, int64_t rows_bound, cudaStream_t s,
                          int32_t* chk = nullptr);
cudaError_t launch_dispatch_from_router(const moe_config_t& c, const int32_t* idx,
                                        const int32_t* tile_hist, const float* partial,
                                        int nparts, int32_t* count, int32_t* offset,
                                        int32_t* slot_of, int32_t* token_of_row,
                                        float* prob_sum, float* f, float* P, float* Lb,
                                        int32_t* dropped, void* zero_y, cudaStream_t s,
                                        int32_t* chk = nullptr);
cudaError_t launch_ffn(const moe_config_t& c, const void* xd, const int32_t* offset,
                       const void* W1, const void* W3, const void* W2, const void* b1,
                       const void* b2, void* Y, void* h, int64_t rows_bound, int32_t* hdr,
                       cudaStream_t s);
cudaError_t launch_ffn_simt(const moe_config_t& c, const void* xd, const int32_t* offset,
                            const void* W1, const void* W3, const void* W2, const void* b1,
                            const void* b2, void* Y, void* h, int64_t rows_bound,
                            int32_t* hdr, cudaStream_t s);
// Fusion of the tensor-core FFN inside the fused layer call: for k = 1 GEMM2
// writes gate * row straight to y[token] (no Y buffer, no combine).
struct FfnFusion {
  void* y = nullptr;                      // [T, d] layer output
  const int32_t* scatter_rows = nullptr;  // token_of_row, or nullptr (k = 1 only)
  const float* scatter_scale = nullptr;   // topk_gate [T] (k = 1)
  cudaEvent_t between = nullptr;          // recorded between GEMM1 and GEMM2, if set
  void* keep_pre = nullptr;               // GEMM1 also stores its pre-activations here
};
cudaError_t launch_ffn_tc(const moe_config_t& c, const void* xd, const int32_t* offset,
                          const void* W1, const void* W3, const void* W2, const void* b1,
                          const void* b2, void* Y, void* h, int64_t rows_bound, int32_t* hdr,
                          cudaStream_t s, const FfnFusion* fz = nullptr);
cudaError_t launch_combine(const moe_config_t& c, const void* Y, const int32_t* slot_of,
                           const float* gate, void* y, cudaStream_t s,
                           const void* base = nullptr, int32_t* chk = nullptr);
cudaError_t launch_one_group_offsets(int32_t* off, int rows, cudaStream_t s);

// ---- backward pass
// The backward GEMMs read the weights in their stored layout (B MN-major);
// only a SwiGLU hidden size that is not a multiple of 64 needs the
// transposed copy W13T = [W1^T | W3^T] per expert for dxd = dact [W1; W3].
inline bool bwd_w13_transposed(const moe_config_t& c) {
  return c.act == MOE_ACT_SWIGLU && c.H % 64 != 0;
}
cudaError_t launch_ffn_bwd_tc(const moe_config_t& c, const void* xd, const int32_t* offset,
                              const void* W1, const void* W3, const void* b1, const void* W2,
                              const void* W13T, const void* dY, void* pre, void* dact,
                              void* dxd, int64_t rows_bound, int32_t* hdr, cudaStream_t s,
                              bool have_pre = false);
cudaError_t launch_router_dx_tc(const void* dz_bf16, int T, int Kp, const void* Wg, int E, int d,
                                const int32_t* off, void* dxr, int32_t* hdr, cudaStream_t s);
cudaError_t launch_wgrad_tc(const void* A, int64_t lda, const void* B, int64_t ldb,
                            int64_t rows, const int32_t* off, int E, int M, int N, int m_split,
                            float* out, float* out2, int32_t* hdr, cudaStream_t s);
int bwd_wg_splits(const moe_config_t& c);
cudaError_t launch_bwd_combine(const moe_config_t& c, const void* dy, const void* Y,
                               const int32_t* slot_of, const float* gate, void* dY, float* dg,
                               cudaStream_t s, int32_t* chk = nullptr);
cudaError_t launch_bwd_router(const moe_config_t& c, const float* logits, const int32_t* idx,
                              const float* gate, const float* dg, const float* f, float alpha,
                              float* dz, void* dz_bf16, int Kp, cudaStream_t s);
int bwd_wg_group_tokens(const moe_config_t& c);
cudaError_t launch_bwd_dx(const moe_config_t& c, const void* dxd, const int32_t* slot_of,
                          const void* dxr, void* dx, cudaStream_t s, const void* dxs = nullptr,
                          int32_t* chk = nullptr);
cudaError_t launch_bwd_wg(const moe_config_t& c, const float* dz, const void* dzb, int Kp,
                          const void* x, int32_t* goff, float* part, float* dWg, float* dbias,
                          int32_t* hdr, cudaStream_t s);
cudaError_t launch_weight_transpose(const void* in, int E, int A, int B, int ld_out, int a_off,
                                    void* out, cudaStream_t s);
cudaError_t launch_expert_colsum(const void* a, int ld, int C, const int32_t* off, int E,
                                 float* out, cudaStream_t s);
// fp32 backward (backward_f32.cu): fp32 FMA throughout
cudaError_t launch_expert_bwd_f32(const moe_config_t& c, const float* xd, const int32_t* off,
                                  int64_t rows_bound, const float* W1, const float* W3,
                                  const float* b1, const float* W2, const float* dY,
                                  const float* h, float* pre, float* dh, float* dact, float* dxd,
                                  float* dW1, float* dW3, float* dW2, float* db1, float* db2,
                                  cudaStream_t s);
cudaError_t launch_bwdf_combine(const moe_config_t& c, const float* dy, const float* Y,
                                const int32_t* slot_of, const float* gate, float* dY, float* dg,
                                cudaStream_t s);
cudaError_t launch_router_grads_f32(const moe_config_t& c, const float* dz, const float* x,
                                    const float* Wg, const int32_t* one_group_off, float* dWg,
                                    float* dbias, float* dxr, cudaStream_t s);
cudaError_t launch_bwdf_dx(const moe_config_t& c, const float* dxr, const float* dxd,
                           const float* dxs, const int32_t* slot_of, float* dx, cudaStream_t s);
cudaError_t launch_aux(const moe_config_t& c, const int32_t* count, const float* prob_sum,
                       const float* partial, int nparts, float* f, float* P, float* L,
                       int32_t* dropped, cudaStream_t s);

}  // namespace moe
