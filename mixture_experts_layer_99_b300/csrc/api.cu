// The C ABI: host-side validation, workspace layout and the launch sequence of
// each call. Every call validates first and enqueues nothing on failure.
#include "moe_internal.h"

#include <math.h>
#include <string.h>

namespace moe {

WsLayout ws_layout(const moe_config_t& c, int /*num_sms*/, int H_shared) {
  WsLayout L;
  memset(&L, 0, sizeof(L));
  const size_t s = elem_bytes(c);
  const size_t T = (size_t)c.T, E = (size_t)c.E, k = (size_t)c.k;
  const size_t R = (size_t)max_rows(c);
  const size_t nblk = (size_t)disp_blocks(c);
  const size_t rgrid = (size_t)router_grid(c, 0);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes > 0 ? bytes : 1, 256);
    return at;
  };
  L.hdr = take(kHdrBytes);
  L.router_partial = take((rgrid > (size_t)kRouterTcMaxBlocks ? rgrid : kRouterTcMaxBlocks) * E * 4);
  L.router_tile_hist = take((size_t)router_tc_tiles(c) * E * 4);
  {
    const RouterSplit sp = router_tc_split(c);
    (void)sp;  // split partials stay in the clusters' shared memory
    L.router_split = take(4);
  }
  L.disp_hist = take(nblk * E * 4);
  L.disp_base = take((nblk > (size_t)router_tc_tiles(c) ? nblk : (size_t)router_tc_tiles(c)) * E * 4);
  L.ffn_h = take(R * (size_t)c.H * s);
  L.ffn_sched = take(4096);
  L.total_core = off;
  L.logits = take(T * E * 4);
  L.topk_idx = take(T * k * 4);
  L.topk_gate = take(T * k * 4);
  L.slot_of = take(T * k * 4);
  L.count = take(E * 4);
  L.offset = take((E + 1) * 4);
  L.token_of_row = take(R * 4);
  L.xd = take(R * (size_t)c.d * s);
  L.Y = take(R * (size_t)c.d * s);
  L.prob_sum = take(E * 4);
  L.f = take(E * 4);
  L.P = take(E * 4);
  L.L = take(4);
  L.dropped = take(4);
  // pre-activations kept by the forward for the backward: [R, H] (GELU) or
  // [R, 2H] (SwiGLU, gate then up), bf16
  L.pre = take((c.flags & MOE_FLAG_KEEP_PREACT)
                   ? R * (size_t)c.H * (c.act == MOE_ACT_SWIGLU ? 2 : 1) * 2
                   : 0);
  L.total_layer = off;
  L.x_stage = take(T * (size_t)c.d * s);
  L.y_stage = take(T * (size_t)c.d * s);
  L.total_host = off;
  off = L.total_layer;  // the shared expert's regions follow the layer's
  L.sh_offset = take(8);
  L.sh_h = take(T * (size_t)(H_shared > 0 ? H_shared : 1) * s);
  L.sh_y = take(T * (size_t)c.d * s);
  L.total_shared = off;
  return L;
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n;
}

// Router: the tensor-core kernel for bf16 with E <= 64, the FMA kernel
// otherwise (fp32 needs fp32 products; E > 64 exceeds the register row).
// Returns the number of per-CTA probability partials written.
cudaError_t run_router(const moe_config_t& c, const void* x, const void* Wg, const float* bias,
                       const float* noise, float* logits, int32_t* idx, float* gate,
                       void* ws, const WsLayout& L, int* nparts, cudaStream_t s) {
  float* partial = reinterpret_cast<float*>(static_cast<char*>(ws) + L.router_partial);
  if (router_tc_supported(c)) {
    *nparts = router_tc_nparts(c);
    return launch_router_tc(c, x, Wg, bias, noise, logits, idx, gate, partial,
                            reinterpret_cast<int32_t*>(static_cast<char*>(ws) + L.router_tile_hist),
                            reinterpret_cast<float*>(static_cast<char*>(ws) + L.router_split),
                            reinterpret_cast<int32_t*>(static_cast<char*>(ws) + L.hdr), s);
  }
  *nparts = router_grid(c, 0);
  return launch_router(c, x, Wg, bias, noise, logits, idx, gate, partial, *nparts, s);
}

cudaError_t launch_ffn(const moe_config_t& c, const void* xd, const int32_t* offset,
                       const void* W1, const void* W3, const void* W2, const void* b1,
                       const void* b2, void* Y, void* h, int64_t rows_bound, int32_t* hdr,
                       cudaStream_t s) {
  if (c.dtype == MOE_BF16)
    return launch_ffn_tc(c, xd, offset, W1, W3, W2, b1, b2, Y, h, rows_bound, hdr, s);
  return launch_ffn_simt(c, xd, offset, W1, W3, W2, b1, b2, Y, h, rows_bound, hdr, s);
}

}  // namespace moe

using namespace moe;

namespace {

moe_status_t validate(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 1 || c->d < 1 || c->E < 1 || c->k < 1 || c->H < 1 || c->capacity < 1)
    return MOE_ERR_INVALID_ARG;
  if (c->k > c->E) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->act != MOE_ACT_GELU && c->act != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
  const int align = c->dtype == MOE_F32 ? 4 : 8;
  if (c->d % align || c->H % align) return MOE_ERR_INVALID_ARG;
  if (!(c->tau > 0.f) || !isfinite(c->tau)) return MOE_ERR_INVALID_ARG;
  if (!(c->noise_scale >= 0.f) || !isfinite(c->noise_scale)) return MOE_ERR_INVALID_ARG;
  if (c->flags & ~MOE_FLAG_KEEP_PREACT) return MOE_ERR_INVALID_ARG;
  if ((c->flags & MOE_FLAG_KEEP_PREACT) && c->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (c->E > kMaxE || c->k > kMaxK) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)c->T * c->k >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)c->T * c->d >= ((int64_t)1 << 40)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t check_ws(const void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return MOE_ERR_WORKSPACE;
  if (((uintptr_t)ws) % 256) return MOE_ERR_WORKSPACE;
  if (ws_bytes < need) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

inline moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

template <typename T> T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

}  // namespace

extern "C" {

int32_t moe_abi_version(void) { return 102; }

const char* moe_status_string(int32_t status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "device-side index check failed";
    default: return "unknown status";
  }
}

int32_t moe_capacity(int64_t c_num, int64_t c_den, int32_t k, int32_t T, int32_t E) {
  if (c_num < 1 || c_den < 1 || k < 1 || T < 1 || E < 1) return -1;
  const __int128 num = (__int128)c_num * k * T;
  const __int128 den = (__int128)c_den * E;
  const __int128 q = (num + den - 1) / den;
  if (q > (__int128)0x7fffffff) return -1;
  return (int32_t)q;
}

moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* bytes) {
  const moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = ws_layout(*cfg, 0).total_layer;
  return MOE_OK;
}

moe_status_t moe_workspace_size_host(const moe_config_t* cfg, size_t* bytes) {
  const moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = ws_layout(*cfg, 0).total_host;
  return MOE_OK;
}

moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream) {
  const moe_status_t st = check_ws(ws, ws_bytes, kHdrBytes);
  if (st != MOE_OK) return st;
  return cuda_status(cudaMemsetAsync(ws, 0, kHdrBytes, (cudaStream_t)stream));
}

moe_status_t moe_device_status(void* ws, int32_t* code, int32_t* where, moe_stream_t stream) {
  if (!code) return MOE_ERR_INVALID_ARG;
  const moe_status_t st = check_ws(ws, kHdrBytes, kHdrBytes);
  if (st != MOE_OK) return st;
  int32_t h[2] = {0, 0};
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(h, ws, sizeof(h), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(h), s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  *code = h[kHdrStatus];
  if (where) *where = h[kHdrWhere];
  return MOE_OK;
}

moe_status_t moe_router_topk(const moe_config_t* cfg, const void* x, const void* Wg,
                             const float* bias, const float* noise, float* logits,
                             int32_t* topk_idx, float* topk_gate, float* prob_sum, void* ws,
                             size_t ws_bytes, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (!x || !Wg || !topk_idx || !topk_gate || !prob_sum) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*cfg, 0);
  if ((st = check_ws(ws, ws_bytes, L.total_core)) != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  int nparts = 0;
  cudaError_t e = run_router(*cfg, x, Wg, bias, noise, logits, topk_idx, topk_gate, ws, L,
                             &nparts, s);
  if (e == cudaSuccess)
    e = launch_prob_reduce(*cfg, at<float>(ws, L.router_partial), nparts, prob_sum, s);
  return cuda_status(e);
}

moe_status_t moe_dispatch(const moe_config_t* cfg, const int32_t* topk_idx, const void* x,
                          int32_t* expert_count, int32_t* expert_offset, int32_t* slot_of,
                          int32_t* token_of_row, void* xd, void* ws, size_t ws_bytes,
                          moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (!topk_idx || !x || !expert_count || !expert_offset || !slot_of || !token_of_row || !xd)
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*cfg, 0);
  if ((st = check_ws(ws, ws_bytes, L.total_core)) != MOE_OK) return st;
  return cuda_status(launch_dispatch(*cfg, topk_idx, x, expert_count, expert_offset, slot_of,
                                     token_of_row, xd, at<int32_t>(ws, L.disp_hist),
                                     at<int32_t>(ws, L.disp_base),
                                     (int64_t)cfg->T * cfg->k, (cudaStream_t)stream,
                                     at<int32_t>(ws, L.hdr)));
}

moe_status_t moe_expert_ffn(const moe_config_t* cfg, const void* xd,
                            const int32_t* expert_offset, const void* W1, const void* W3,
                            const void* W2, const void* b1, const void* b2, void* Y, void* ws,
                            size_t ws_bytes, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (!xd || !expert_offset || !W1 || !W2 || !Y) return MOE_ERR_INVALID_ARG;
  if ((cfg->act == MOE_ACT_SWIGLU) != (W3 != nullptr)) return MOE_ERR_INVALID_ARG;
  if (cfg->act == MOE_ACT_SWIGLU && (b1 || b2)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*cfg, 0);
  if ((st = check_ws(ws, ws_bytes, L.total_core)) != MOE_OK) return st;
  return cuda_status(launch_ffn(*cfg, xd, expert_offset, W1, W3, W2, b1, b2, Y,
                                at<void>(ws, L.ffn_h), max_rows(*cfg),
                                at<int32_t>(ws, L.hdr), (cudaStream_t)stream));
}

moe_status_t moe_combine(const moe_config_t* cfg, const void* Y, const int32_t* slot_of,
                         const float* topk_gate, void* y, moe_stream_t stream) {
  const moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (!Y || !slot_of || !topk_gate || !y) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(*cfg, Y, slot_of, topk_gate, y, (cudaStream_t)stream));
}

moe_status_t moe_aux_stats(const moe_config_t* cfg, const int32_t* expert_count,
                           const float* prob_sum, float* f, float* P, float* L_balance,
                           int32_t* dropped, moe_stream_t stream) {
  const moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (!expert_count || !prob_sum || !f || !P || !L_balance || !dropped)
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_aux(*cfg, expert_count, prob_sum, nullptr, 0, f, P, L_balance,
                                dropped, (cudaStream_t)stream));
}

// ev (optional): six events recorded on s at the stage boundaries: before
// the router, after the router, after the dispatch, after GEMM1, after GEMM2,
// after the combine and statistics.
// sh (optional): a shared expert; its output (rows of ws) is the base the
// combine adds the routed slots to. ws must then follow ws_layout(c, 0, sh->H).
static moe_status_t layer_forward_impl(const moe_config_t* cfg, const void* x,
                                       const moe_layer_inputs_t* in,
                                       const moe_layer_outputs_t* out, void* y, float* Lout,
                                       void* ws, cudaStream_t s,
                                       const cudaEvent_t* ev = nullptr,
                                       const moe_shared_expert_t* sh = nullptr) {
  auto mark = [&](int i) -> cudaError_t { return ev ? record_stage_event(ev[i], s) : cudaSuccess; };
  const moe_config_t& c = *cfg;
  const WsLayout L = ws_layout(c, 0, sh ? sh->H : 0);
  int32_t* idx = out && out->topk_idx ? out->topk_idx : at<int32_t>(ws, L.topk_idx);
  float* gate = out && out->topk_gate ? out->topk_gate : at<float>(ws, L.topk_gate);
  int32_t* slot_of = out && out->slot_of ? out->slot_of : at<int32_t>(ws, L.slot_of);
  int32_t* count = out && out->expert_count ? out->expert_count : at<int32_t>(ws, L.count);
  int32_t* offset = out && out->expert_offset ? out->expert_offset : at<int32_t>(ws, L.offset);
  float* f = out && out->f ? out->f : at<float>(ws, L.f);
  float* P = out && out->P ? out->P : at<float>(ws, L.P);
  float* Lb = Lout ? Lout : at<float>(ws, L.L);
  int32_t* dropped = out && out->dropped ? out->dropped : at<int32_t>(ws, L.dropped);
  float* logits = out ? out->logits : nullptr;
  int rgrid = 0;
  float* partial = at<float>(ws, L.router_partial);
  float* prob_sum = at<float>(ws, L.prob_sum);
  const int64_t R = max_rows(c);
  int32_t* token_of_row = at<int32_t>(ws, L.token_of_row);
  cudaError_t e = mark(0);
  if (e == cudaSuccess)
    e = run_router(c, x, in->Wg, in->bias, in->noise, logits, idx, gate, ws, L, &rgrid, s);
  if (e == cudaSuccess) e = mark(1);
  // tensor-core router (bf16, E <= 64): its per-tile histograms and
  // probability partials feed one dispatch + statistics kernel (one block per
  // tile); for k = 1 GEMM2 writes the gated rows straight into y.
  const bool fused_stats = router_tc_supported(c);
  const bool scatter = fused_stats && c.k == 1 && !sh;
  if (e == cudaSuccess) {
    if (fused_stats) {
      e = launch_dispatch_from_router(c, idx, at<int32_t>(ws, L.router_tile_hist), partial,
                                      rgrid, count, offset, slot_of, token_of_row, prob_sum, f,
                                      P, Lb, dropped, scatter ? y : nullptr, s,
                                      at<int32_t>(ws, L.hdr));
      if (e == cudaSuccess)
        e = launch_gather(c, x, token_of_row, offset, at<void>(ws, L.xd), R, s,
                          at<int32_t>(ws, L.hdr));
    } else {
      e = launch_dispatch(c, idx, x, count, offset, slot_of, token_of_row, at<void>(ws, L.xd),
                          at<int32_t>(ws, L.disp_hist), at<int32_t>(ws, L.disp_base), R, s,
                          at<int32_t>(ws, L.hdr));
    }
  }
  if (e == cudaSuccess) e = mark(2);
  if (e == cudaSuccess) {
    if (c.dtype == MOE_BF16) {
      FfnFusion fz;
      fz.between = ev ? ev[3] : nullptr;
      if (scatter) {
        fz.y = y;
        fz.scatter_rows = token_of_row;
        fz.scatter_scale = gate;
      }
      if (c.flags & MOE_FLAG_KEEP_PREACT) fz.keep_pre = at<void>(ws, L.pre);
      e = launch_ffn_tc(c, at<void>(ws, L.xd), offset, in->W1, in->W3, in->W2, in->b1, in->b2,
                        at<void>(ws, L.Y), at<void>(ws, L.ffn_h), R, at<int32_t>(ws, L.hdr), s,
                        &fz);
    } else {
      e = launch_ffn(c, at<void>(ws, L.xd), offset, in->W1, in->W3, in->W2, in->b1, in->b2,
                     at<void>(ws, L.Y), at<void>(ws, L.ffn_h), R, at<int32_t>(ws, L.hdr), s);
      if (e == cudaSuccess) e = mark(3);  // the FMA path has no mark between its GEMMs
    }
  }
  if (e == cudaSuccess) e = mark(4);
  void* base = nullptr;
  if (sh && e == cudaSuccess) {
    // the shared expert: one group of all T token rows through the same FFN
    moe_config_t cs = c;
    cs.E = 1;
    cs.k = 1;
    cs.H = sh->H;
    cs.capacity = c.T;
    int32_t* soff = at<int32_t>(ws, L.sh_offset);
    e = launch_one_group_offsets(soff, c.T, s);
    if (e == cudaSuccess)
      e = launch_ffn(cs, x, soff, sh->W1, sh->W3, sh->W2, sh->b1, sh->b2, at<void>(ws, L.sh_y),
                     at<void>(ws, L.sh_h), c.T, at<int32_t>(ws, L.hdr), s);
    base = at<void>(ws, L.sh_y);
  }
  if (e == cudaSuccess && !scatter)
    e = launch_combine(c, at<void>(ws, L.Y), slot_of, gate, y, s, base, at<int32_t>(ws, L.hdr));
  if (!fused_stats) {
    if (e == cudaSuccess) e = launch_prob_reduce(c, partial, rgrid, prob_sum, s);
    if (e == cudaSuccess) e = launch_aux(c, count, prob_sum, nullptr, 0, f, P, Lb, dropped, s);
  }
  if (e == cudaSuccess) e = mark(5);
  return cuda_status(e);
}

static moe_status_t check_layer_inputs(const moe_config_t* cfg, const moe_layer_inputs_t* in) {
  if (!in || !in->Wg || !in->W1 || !in->W2) return MOE_ERR_INVALID_ARG;
  if ((cfg->act == MOE_ACT_SWIGLU) != (in->W3 != nullptr)) return MOE_ERR_INVALID_ARG;
  if (cfg->act == MOE_ACT_SWIGLU && (in->b1 || in->b2)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status_t moe_layer_forward(const moe_config_t* cfg, const moe_layer_inputs_t* in,
                               const moe_layer_outputs_t* out, void* ws, size_t ws_bytes,
                               moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if ((st = check_layer_inputs(cfg, in)) != MOE_OK) return st;
  if (!in->x || !out || !out->y) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, ws_layout(*cfg, 0).total_layer)) != MOE_OK) return st;
  return layer_forward_impl(cfg, in->x, in, out, out->y, out->L_balance, ws,
                            (cudaStream_t)stream);
}

static moe_status_t check_shared(const moe_config_t* cfg, const moe_shared_expert_t* sh) {
  if (!sh || !sh->W1 || !sh->W2) return MOE_ERR_INVALID_ARG;
  const int align = cfg->dtype == MOE_F32 ? 4 : 8;
  if (sh->H < 1 || sh->H % align) return MOE_ERR_INVALID_ARG;
  if ((cfg->act == MOE_ACT_SWIGLU) != (sh->W3 != nullptr)) return MOE_ERR_INVALID_ARG;
  if (cfg->act == MOE_ACT_SWIGLU && (sh->b1 || sh->b2)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status_t moe_workspace_size_shared(const moe_config_t* cfg, int32_t H_shared,
                                       size_t* bytes) {
  const moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (!bytes || H_shared < 1) return MOE_ERR_INVALID_ARG;
  *bytes = ws_layout(*cfg, 0, H_shared).total_shared;
  return MOE_OK;
}

moe_status_t moe_layer_forward_shared(const moe_config_t* cfg, const moe_layer_inputs_t* in,
                                      const moe_shared_expert_t* shared,
                                      const moe_layer_outputs_t* out, void* ws,
                                      size_t ws_bytes, moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if ((st = check_layer_inputs(cfg, in)) != MOE_OK) return st;
  if ((st = check_shared(cfg, shared)) != MOE_OK) return st;
  if (!in->x || !out || !out->y) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, ws_layout(*cfg, 0, shared->H).total_shared)) != MOE_OK)
    return st;
  return layer_forward_impl(cfg, in->x, in, out, out->y, out->L_balance, ws,
                            (cudaStream_t)stream, nullptr, shared);
}

moe_status_t moe_layer_forward_profiled(const moe_config_t* cfg, const moe_layer_inputs_t* in,
                                        const moe_layer_outputs_t* out, void* ws,
                                        size_t ws_bytes, moe_stream_t stream,
                                        void* const* stage_events) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if ((st = check_layer_inputs(cfg, in)) != MOE_OK) return st;
  if (!in->x || !out || !out->y || !stage_events) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 6; ++i)
    if (!stage_events[i]) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, ws_layout(*cfg, 0).total_layer)) != MOE_OK) return st;
  return layer_forward_impl(cfg, in->x, in, out, out->y, out->L_balance, ws,
                            (cudaStream_t)stream,
                            reinterpret_cast<const cudaEvent_t*>(stage_events));
}

int32_t moe_layer_forward_launch_count(const moe_config_t* cfg) {
  if (validate(cfg) != MOE_OK) return 0;
  // tensor-core router path: router (one launch; a split K range runs as clusters),
  // dispatch + statistics, gather, GEMM1, GEMM2, and the combine unless k = 1
  // (then GEMM2 writes y). FMA router path: router, dispatch (count, scan,
  // assign, gather), GEMM1, GEMM2, combine, probability reduction, statistics.
  if (router_tc_supported(*cfg))
    return cfg->k == 1 ? 5 : 6;
  return 10;
}

moe_status_t moe_layer_forward_host(const moe_config_t* cfg, const void* x_host,
                                    const moe_layer_inputs_t* in, void* y_host,
                                    float* L_balance_host, void* ws, size_t ws_bytes,
                                    moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if ((st = check_layer_inputs(cfg, in)) != MOE_OK) return st;
  if (!x_host || !y_host) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*cfg, 0);
  if ((st = check_ws(ws, ws_bytes, L.total_host)) != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t bytes = (size_t)cfg->T * cfg->d * elem_bytes(*cfg);
  void* xs = at<void>(ws, L.x_stage);
  void* ys = at<void>(ws, L.y_stage);
  if (cudaMemcpyAsync(xs, x_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  st = layer_forward_impl(cfg, xs, in, nullptr, ys, nullptr, ws, s);
  if (st != MOE_OK) return st;
  if (cudaMemcpyAsync(y_host, ys, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (L_balance_host &&
      cudaMemcpyAsync(L_balance_host, at<float>(ws, L.L), sizeof(float),
                      cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_layer_forward_host_pipelined(const moe_config_t* cfg, const void* x_host,
                                              const moe_layer_inputs_t* in, void* y_host,
                                              float* L_balance_host, void* ws, size_t ws_bytes,
                                              moe_stream_t copy_in, moe_stream_t compute,
                                              moe_stream_t copy_out, const moe_event_t* ev) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if ((st = check_layer_inputs(cfg, in)) != MOE_OK) return st;
  if (!x_host || !y_host || !ev || !ev[0] || !ev[1] || !ev[2]) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*cfg, 0);
  if ((st = check_ws(ws, ws_bytes, L.total_host)) != MOE_OK) return st;
  cudaStream_t si = (cudaStream_t)copy_in, sc = (cudaStream_t)compute,
               so = (cudaStream_t)copy_out;
  cudaEvent_t in_done = (cudaEvent_t)ev[0], layer_done = (cudaEvent_t)ev[1],
              out_done = (cudaEvent_t)ev[2];
  const size_t bytes = (size_t)cfg->T * cfg->d * elem_bytes(*cfg);
  void* xs = at<void>(ws, L.x_stage);
  void* ys = at<void>(ws, L.y_stage);
  // x_stage is free once the previous call with this ws finished its layer
  // (waiting on an event that was never recorded does not wait)
  if (cudaStreamWaitEvent(si, layer_done, 0) != cudaSuccess ||
      cudaMemcpyAsync(xs, x_host, bytes, cudaMemcpyHostToDevice, si) != cudaSuccess ||
      cudaEventRecord(in_done, si) != cudaSuccess ||
      cudaStreamWaitEvent(sc, in_done, 0) != cudaSuccess ||
      cudaStreamWaitEvent(sc, out_done, 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  st = layer_forward_impl(cfg, xs, in, nullptr, ys, nullptr, ws, sc);
  if (st != MOE_OK) return st;
  if (cudaEventRecord(layer_done, sc) != cudaSuccess ||
      cudaStreamWaitEvent(so, layer_done, 0) != cudaSuccess ||
      cudaMemcpyAsync(y_host, ys, bytes, cudaMemcpyDeviceToHost, so) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (L_balance_host &&
      cudaMemcpyAsync(L_balance_host, at<float>(ws, L.L), sizeof(float),
                      cudaMemcpyDeviceToHost, so) != cudaSuccess)
    return MOE_ERR_CUDA;
  return cudaEventRecord(out_done, so) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ---------------------------------------------------------------- backward
namespace {
struct BwdLayout {
  size_t hdr, pre, dact, dY, dxd, W13T, dz, dg, wg_part, dzb, dxr, goff, wgoff, dh, total;
  int kp;  // experts padded to a multiple of 64 (K of the dz W_g GEMM)
};
BwdLayout bwd_layout(const moe_config_t& c) {
  BwdLayout L;
  memset(&L, 0, sizeof(L));
  const size_t R = (size_t)max_rows(c), E = (size_t)c.E, d = (size_t)c.d, H = (size_t)c.H;
  const size_t Hp = c.act == MOE_ACT_SWIGLU ? 2 * H : H;
  const bool f32 = c.dtype == MOE_F32;
  const size_t s = f32 ? 4 : 2;  // activation-gradient element bytes
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes > 0 ? bytes : 1, 256);
    return at;
  };
  L.hdr = take(kHdrBytes);
  // recomputed pre-activations, unless the forward kept them in its workspace
  L.pre = take((c.flags & MOE_FLAG_KEEP_PREACT) ? 0 : R * Hp * s);
  L.dact = take(R * Hp * s);
  L.dY = take(R * d * s);
  L.dxd = take(R * d * s);
  L.W13T = take(!f32 && bwd_w13_transposed(c) ? E * d * Hp * 2 : 0);
  L.dz = take((size_t)c.T * E * 4);
  L.dg = take((size_t)c.T * (size_t)c.k * 4);
  L.wg_part = take(f32 ? 0 : (size_t)bwd_wg_splits(c) * E * d * 4);
  L.kp = (int)align_up(E, 64);
  L.wgoff = take(f32 ? 0 : ((size_t)bwd_wg_splits(c) + 1) * 4);
  L.dzb = take((size_t)c.T * (size_t)L.kp * 2);
  L.dxr = take((size_t)c.T * d * s);
  L.goff = take(8);
  L.dh = take(f32 ? R * H * 4 : 0);  // fp32: dY W2 before the activation's derivative
  L.total = off;
  return L;
}
// bf16 on the tensor cores; fp32 on fp32 FMA (backward_f32.cu)
bool bwd_supported(const moe_config_t& c) { return c.dtype == MOE_BF16 || c.dtype == MOE_F32; }

// The shared expert's part of the backward workspace, after the routed part:
// its recomputed pre-activations and activation gradients [T, Hps], its dx
// term [T, d], the transposed [W1^T | W3^T] where needed, one-group offsets.
struct BwdSharedLayout {
  size_t pre, dact, dxs, W13T, soff, dh, total;
};
moe_config_t shared_config(const moe_config_t& c, int H_shared) {
  moe_config_t cs = c;
  cs.E = 1;
  cs.k = 1;
  cs.H = H_shared;
  cs.capacity = c.T;
  return cs;
}
BwdSharedLayout bwd_shared_layout(const moe_config_t& c, int H_shared) {
  BwdSharedLayout L;
  const moe_config_t cs = shared_config(c, H_shared);
  const size_t T = (size_t)c.T, d = (size_t)c.d;
  const size_t Hps = c.act == MOE_ACT_SWIGLU ? 2 * (size_t)H_shared : (size_t)H_shared;
  size_t off = bwd_layout(c).total;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes > 0 ? bytes : 1, 256);
    return at;
  };
  const bool f32 = c.dtype == MOE_F32;
  const size_t s = f32 ? 4 : 2;
  L.pre = take(T * Hps * s);
  L.dact = take(T * Hps * s);
  L.dxs = take(T * d * s);
  L.W13T = take(!f32 && bwd_w13_transposed(cs) ? d * Hps * 2 : 0);
  L.soff = take(8);
  L.dh = take(f32 ? T * (size_t)H_shared * 4 : 0);
  L.total = off;
  return L;
}
}  // namespace

moe_status_t moe_workspace_size_backward(const moe_config_t* cfg, size_t* bytes) {
  const moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  if (!bwd_supported(*cfg)) return MOE_ERR_UNSUPPORTED;
  *bytes = bwd_layout(*cfg).total;
  return MOE_OK;
}

// The fp32 backward: the steps of the bf16 one on fp32 FMA, reading what the
// fp32 forward left in its workspace (gathered rows xd, hidden rows h, expert
// outputs Y for k > 1; the shared expert's hidden rows).
static cudaError_t layer_backward_f32(const moe_config_t& c, const moe_layer_inputs_t* in,
                                      const moe_shared_expert_t* sh,
                                      const moe_layer_outputs_t* fwd, const float* dy,
                                      float alpha, const moe_layer_grads_t* g,
                                      const moe_shared_grads_t* sg, void* ws, const WsLayout& L,
                                      void* bws, const BwdLayout& B, const BwdSharedLayout& BS,
                                      cudaStream_t s) {
  const int64_t R = max_rows(c);
  const float* xd = at<float>(ws, L.xd);
  const float* Y = c.k > 1 ? at<float>(ws, L.Y) : nullptr;  // k = 1: gates are identically 1
  const int32_t* off = fwd->expert_offset;
  float* dYb = at<float>(bws, B.dY);
  float* dz = at<float>(bws, B.dz);
  float* dg = at<float>(bws, B.dg);
  float* dxr = at<float>(bws, B.dxr);
  float* dxd = at<float>(bws, B.dxd);
  int32_t* goff = at<int32_t>(bws, B.goff);
  cudaError_t e = launch_bwdf_combine(c, dy, Y, fwd->slot_of, fwd->topk_gate, dYb, dg, s);
  if (e == cudaSuccess)
    e = launch_bwd_router(c, fwd->logits, fwd->topk_idx, fwd->topk_gate, dg, fwd->f, alpha, dz,
                          at<void>(bws, B.dzb), B.kp, s);
  if (e == cudaSuccess) e = launch_one_group_offsets(goff, c.T, s);
  if (e == cudaSuccess)
    e = launch_router_grads_f32(c, dz, static_cast<const float*>(in->x),
                                static_cast<const float*>(in->Wg), goff, g->dWg, g->dbias, dxr, s);
  if (e == cudaSuccess)
    e = launch_expert_bwd_f32(c, xd, off, R, static_cast<const float*>(in->W1),
                              static_cast<const float*>(in->W3), static_cast<const float*>(in->b1),
                              static_cast<const float*>(in->W2), dYb, at<float>(ws, L.ffn_h),
                              at<float>(bws, B.pre), at<float>(bws, B.dh), at<float>(bws, B.dact),
                              dxd, g->dW1, g->dW3, g->dW2, g->db1, g->db2, s);
  // the shared expert: one group of all T token rows, output gradient dy
  float* dxs = nullptr;
  if (sh && e == cudaSuccess) {
    const moe_config_t cs = shared_config(c, sh->H);
    int32_t* soff = at<int32_t>(bws, BS.soff);
    dxs = at<float>(bws, BS.dxs);
    e = launch_one_group_offsets(soff, c.T, s);
    if (e == cudaSuccess)
      e = launch_expert_bwd_f32(cs, static_cast<const float*>(in->x), soff, c.T,
                                static_cast<const float*>(sh->W1),
                                static_cast<const float*>(sh->W3),
                                static_cast<const float*>(sh->b1),
                                static_cast<const float*>(sh->W2), dy, at<float>(ws, L.sh_h),
                                at<float>(bws, BS.pre), at<float>(bws, BS.dh),
                                at<float>(bws, BS.dact), dxs, sg->dW1, sg->dW3, sg->dW2, sg->db1,
                                sg->db2, s);
  }
  if (e == cudaSuccess)
    e = launch_bwdf_dx(c, dxr, dxd, dxs, fwd->slot_of, static_cast<float*>(g->dx), s);
  return e;
}

static moe_status_t layer_backward_impl(const moe_config_t* cfg, const moe_layer_inputs_t* in,
                                        const moe_shared_expert_t* sh,
                                        const moe_layer_outputs_t* fwd, const void* dy,
                                        float alpha, const moe_layer_grads_t* g,
                                        const moe_shared_grads_t* sg, const void* ws,
                                        size_t ws_bytes, void* bws, size_t bws_bytes,
                                        moe_stream_t stream) {
  moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  const moe_config_t& c = *cfg;
  if (!bwd_supported(c)) return MOE_ERR_UNSUPPORTED;
  if ((st = check_layer_inputs(cfg, in)) != MOE_OK) return st;
  if (!in->x || !fwd || !dy || !g) return MOE_ERR_INVALID_ARG;
  if (!fwd->logits || !fwd->topk_idx || !fwd->topk_gate || !fwd->slot_of ||
      !fwd->expert_offset || !fwd->f)
    return MOE_ERR_INVALID_ARG;
  const bool swiglu = c.act == MOE_ACT_SWIGLU;
  if (!g->dx || !g->dWg || !g->dW1 || !g->dW2 || (swiglu != (g->dW3 != nullptr)) ||
      ((in->bias != nullptr) != (g->dbias != nullptr)) ||
      ((in->b1 != nullptr) != (g->db1 != nullptr)) ||
      ((in->b2 != nullptr) != (g->db2 != nullptr)))
    return MOE_ERR_INVALID_ARG;
  if (sh) {
    if ((st = check_shared(cfg, sh)) != MOE_OK) return st;
    if (!sg || !sg->dW1 || !sg->dW2 || (swiglu != (sg->dW3 != nullptr)) ||
        ((sh->b1 != nullptr) != (sg->db1 != nullptr)) ||
        ((sh->b2 != nullptr) != (sg->db2 != nullptr)))
      return MOE_ERR_INVALID_ARG;
  }
  const int Hs = sh ? sh->H : 0;
  const WsLayout L = ws_layout(c, 0, Hs);
  if ((st = check_ws(const_cast<void*>(ws), ws_bytes, sh ? L.total_shared : L.total_layer)) !=
      MOE_OK)
    return st;
  const BwdLayout B = bwd_layout(c);
  const BwdSharedLayout BS = bwd_shared_layout(c, Hs > 0 ? Hs : 8);
  if ((st = check_ws(bws, bws_bytes, sh ? BS.total : B.total)) != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (c.dtype == MOE_F32)
    return cuda_status(layer_backward_f32(c, in, sh, fwd, static_cast<const float*>(dy), alpha,
                                          g, sg, const_cast<void*>(ws), L, bws, B, BS, s));
  const int64_t R = max_rows(c);
  const int Hp = swiglu ? 2 * c.H : c.H;
  int32_t* hdr = at<int32_t>(bws, 0);
  void* wsm = const_cast<void*>(ws);
  const void* xd = at<void>(wsm, L.xd);
  const void* Y = c.k > 1 ? at<void>(wsm, L.Y) : nullptr;  // k = 1: gates are identically 1
  const int32_t* off = fwd->expert_offset;
  const bool kept_pre = (c.flags & MOE_FLAG_KEEP_PREACT) != 0;
  void* pre = kept_pre ? at<void>(wsm, L.pre) : at<void>(bws, B.pre);
  void* dact = at<void>(bws, B.dact);
  void* dYb = at<void>(bws, B.dY);
  void* dxd = at<void>(bws, B.dxd);
  void* W13T = bwd_w13_transposed(c) ? at<void>(bws, B.W13T) : nullptr;
  float* dz = at<float>(bws, B.dz);
  float* dg = at<float>(bws, B.dg);
  cudaError_t e = cudaSuccess;
  if (W13T) {
    e = launch_weight_transpose(in->W1, c.E, c.H, c.d, Hp, 0, W13T, s);
    if (e == cudaSuccess) e = launch_weight_transpose(in->W3, c.E, c.H, c.d, Hp, c.H, W13T, s);
  }
  if (e == cudaSuccess)
    e = launch_bwd_combine(c, dy, Y, fwd->slot_of, fwd->topk_gate, dYb, dg, s, hdr);
  void* dzb = at<void>(bws, B.dzb);
  void* dxr = at<void>(bws, B.dxr);
  int32_t* goff = at<int32_t>(bws, B.goff);
  if (e == cudaSuccess)
    e = launch_bwd_router(c, fwd->logits, fwd->topk_idx, fwd->topk_gate, dg, fwd->f, alpha, dz,
                          dzb, B.kp, s);
  // router part of dx on the tensor cores: dxr = dz W_g (experts zero-padded)
  if (e == cudaSuccess) e = launch_one_group_offsets(goff, c.T, s);
  if (e == cudaSuccess)
    e = launch_router_dx_tc(dzb, c.T, B.kp, in->Wg, c.E, c.d, goff, dxr, hdr, s);
  if (e == cudaSuccess)
    e = launch_ffn_bwd_tc(c, xd, off, in->W1, in->W3, in->b1, in->W2, W13T, dYb, pre, dact, dxd,
                          R, hdr, s, kept_pre);
  // the shared expert: the same expert backward as one group of all T token
  // rows, its output gradient being dy itself (weight 1 for every token)
  void* dxs = nullptr;
  if (sh && e == cudaSuccess) {
    const moe_config_t cs = shared_config(c, Hs);
    const int Hps = swiglu ? 2 * Hs : Hs;
    int32_t* soff = at<int32_t>(bws, BS.soff);
    void* W13Ts = bwd_w13_transposed(cs) ? at<void>(bws, BS.W13T) : nullptr;
    void* pre_s = at<void>(bws, BS.pre);
    void* dact_s = at<void>(bws, BS.dact);
    dxs = at<void>(bws, BS.dxs);
    e = launch_one_group_offsets(soff, c.T, s);
    if (e == cudaSuccess && W13Ts) {
      e = launch_weight_transpose(sh->W1, 1, Hs, c.d, Hps, 0, W13Ts, s);
      if (e == cudaSuccess) e = launch_weight_transpose(sh->W3, 1, Hs, c.d, Hps, Hs, W13Ts, s);
    }
    if (e == cudaSuccess)
      e = launch_ffn_bwd_tc(cs, in->x, soff, sh->W1, sh->W3, sh->b1, sh->W2, W13Ts, dy, pre_s,
                            dact_s, dxs, c.T, hdr, s);
    // dW2s [d, Hs] = dy^T h_s (h_s as the forward left it); [dW1s; dW3s] = dact_s^T x
    if (e == cudaSuccess)
      e = launch_wgrad_tc(dy, c.d, at<void>(wsm, L.sh_h), Hs, c.T, soff, 1, c.d, Hs, c.d,
                          sg->dW2, sg->dW2, hdr, s);
    if (e == cudaSuccess)
      e = launch_wgrad_tc(dact_s, Hps, in->x, c.d, c.T, soff, 1, Hps, c.d, Hs, sg->dW1,
                          swiglu ? sg->dW3 : sg->dW1, hdr, s);
    if (e == cudaSuccess && sg->db1) e = launch_expert_colsum(dact_s, Hps, Hs, soff, 1, sg->db1, s);
    if (e == cudaSuccess && sg->db2) e = launch_expert_colsum(dy, c.d, c.d, soff, 1, sg->db2, s);
  }
  if (e == cudaSuccess) e = launch_bwd_dx(c, dxd, fwd->slot_of, dxr, g->dx, s, dxs, hdr);
  if (e == cudaSuccess)
    e = launch_bwd_wg(c, dz, dzb, B.kp, in->x, at<int32_t>(bws, B.wgoff),
                      at<float>(bws, B.wg_part), g->dWg, g->dbias, hdr, s);
  // dW2 [E, d, H] = dY^T h (h as the forward left it in its workspace);
  // [dW1; dW3] [E, Hp, d] = dact^T xd; row-major operands read MN-major
  if (e == cudaSuccess)
    e = launch_wgrad_tc(dYb, c.d, at<void>(wsm, L.ffn_h), c.H, R, off, c.E, c.d, c.H, c.d,
                        g->dW2, g->dW2, hdr, s);
  if (e == cudaSuccess)
    e = launch_wgrad_tc(dact, Hp, xd, c.d, R, off, c.E, Hp, c.d, c.H, g->dW1,
                        swiglu ? g->dW3 : g->dW1, hdr, s);
  if (e == cudaSuccess && g->db1) e = launch_expert_colsum(dact, Hp, c.H, off, c.E, g->db1, s);
  if (e == cudaSuccess && g->db2) e = launch_expert_colsum(dYb, c.d, c.d, off, c.E, g->db2, s);
  return cuda_status(e);
}

moe_status_t moe_layer_backward(const moe_config_t* cfg, const moe_layer_inputs_t* in,
                                const moe_layer_outputs_t* fwd, const void* dy, float alpha,
                                const moe_layer_grads_t* g, const void* ws, size_t ws_bytes,
                                void* bws, size_t bws_bytes, moe_stream_t stream) {
  return layer_backward_impl(cfg, in, nullptr, fwd, dy, alpha, g, nullptr, ws, ws_bytes, bws,
                             bws_bytes, stream);
}

moe_status_t moe_workspace_size_backward_shared(const moe_config_t* cfg, int32_t H_shared,
                                                size_t* bytes) {
  const moe_status_t st = validate(cfg);
  if (st != MOE_OK) return st;
  if (!bytes || H_shared < 1 || H_shared % (cfg->dtype == MOE_F32 ? 4 : 8)) return MOE_ERR_INVALID_ARG;
  if (!bwd_supported(*cfg)) return MOE_ERR_UNSUPPORTED;
  *bytes = bwd_shared_layout(*cfg, H_shared).total;
  return MOE_OK;
}

moe_status_t moe_layer_backward_shared(const moe_config_t* cfg, const moe_layer_inputs_t* in,
                                       const moe_shared_expert_t* shared,
                                       const moe_layer_outputs_t* fwd, const void* dy,
                                       float alpha, const moe_layer_grads_t* grads,
                                       const moe_shared_grads_t* shared_grads, const void* ws,
                                       size_t ws_bytes, void* bws, size_t bws_bytes,
                                       moe_stream_t stream) {
  if (!shared) return MOE_ERR_INVALID_ARG;
  return layer_backward_impl(cfg, in, shared, fwd, dy, alpha, grads, shared_grads, ws, ws_bytes,
                             bws, bws_bytes, stream);
}

}  // extern "C"
