// C ABI of libmoe.so: argument checks, workspace layout, kernel launches.
// The operations and their sources are documented in include/moe.h.
// Every call that launches work opens an NVTX range named after itself, so
// profilers that record NVTX show where each layer step starts and ends
// (without a profiler attached the range calls return at once).
#include <cstring>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"

using namespace moe;

namespace {

struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange &) = delete;
  NvtxRange &operator=(const NvtxRange &) = delete;
};

constexpr size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool shape_ok(const moe_shape_t *s) {
  if (s == nullptr) return false;
  if (s->T < 1 || s->d < 1 || s->E < 1 || s->E > 64 || s->K < 1 || s->K > 8 || s->K > s->E)
    return false;
  if (s->F < 1 || (s->dtype != MOE_F32 && s->dtype != MOE_BF16)) return false;
  if (s->drop != 0 && s->drop != 1) return false;
  if (s->drop && !(s->capacity_factor > 0.0f)) return false;
  if (s->subseq_len < 0 || (s->renorm != 0 && s->renorm != 1) || s->Fs < 0) return false;
  if (s->T * (int64_t)s->K >= (int64_t(1) << 31)) return false;  // int32 row indices
  if (s->d % (s->dtype == MOE_BF16 ? 8 : 4) != 0) return false;
  return true;
}

int64_t subseq(const moe_shape_t *s) {
  return (s->subseq_len > 0 && s->subseq_len < s->T) ? s->subseq_len : s->T;
}

struct Layout {
  size_t status, map, cap, capn, rbwd, total;
};

// the tensor-core router's logits path (bf16, d % 64 == 0)
bool router_on_tensor_cores(const moe_shape_t *s) {
  return s->dtype == MOE_BF16 && s->d % 64 == 0;
}

Layout layout(const moe_shape_t *s) {
  Layout L{};
  size_t off = kStatusBytes;
  L.status = 0;
  L.map = off;
  off += align256((size_t)((s->T + 255) / 256) * s->E * sizeof(int32_t));
  L.cap = off;
  L.capn = off;
  if (s->drop) {
    const int64_t S = subseq(s);
    const int64_t n_sub = (s->T + S - 1) / S;
    off += align256((size_t)n_sub * s->E * S * sizeof(unsigned long long));
    L.capn = off;
    off += align256((size_t)n_sub * s->E * sizeof(uint32_t));
  }
  L.rbwd = off;
  off += align256(route_bwd_workspace_bytes(s->T, s->d, s->E));
  L.total = off > MOE_FFN_BWD_WORKSPACE_BYTES ? off : MOE_FFN_BWD_WORKSPACE_BYTES;
  return L;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

uint32_t *status_word(void *ws) { return reinterpret_cast<uint32_t *>(ws); }

RouteArgs route_args(const moe_shape_t *s, void *ws) {
  RouteArgs a{};
  const Layout L = layout(s);
  a.T = s->T; a.d = s->d; a.E = s->E; a.K = s->K; a.dtype = s->dtype;
  a.renorm = s->renorm; a.drop = s->drop; a.S = subseq(s); a.cf = s->capacity_factor;
  a.status = status_word(ws);
  a.cap_keys = reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + L.cap);
  a.cap_counts = reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + L.capn);
  return a;
}

// capacity dropping: the candidate list lengths start at zero (a memset
// ahead of the call's kernels keeps the kernels' dependent-launch chain whole)
cudaError_t clear_capacity_counts(const moe_shape_t *s, const RouteArgs &a, cudaStream_t st) {
  if (!s->drop) return cudaSuccess;
  const int64_t S = subseq(s);
  const int64_t n_sub = (s->T + S - 1) / S;
  return cudaMemsetAsync(a.cap_counts, 0, (size_t)n_sub * s->E * sizeof(uint32_t), st);
}

}  // namespace

extern "C" {

const char *moe_version(void) { return "0.1.0"; }

const char *moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE: return "device-side check failed";
  }
  return "unknown status";
}

size_t moe_workspace_size(const moe_shape_t *shape) {
  if (!shape_ok(shape)) return 0;
  return layout(shape).total;
}

moe_status_t moe_clear_status(void *ws, moe_stream_t stream) {
  if (ws == nullptr || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, 2 * sizeof(uint32_t), (cudaStream_t)stream));
}

moe_status_t moe_get_status(void *ws, moe_stream_t stream, uint32_t *info) {
  if (ws == nullptr || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  uint32_t h[2] = {0, 0};
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (info != nullptr) *info = h[1];
  return (moe_status_t)h[0];
}

moe_status_t moe_route(const moe_shape_t *shape, const void *x, const void *W_r, const float *b_r,
                       const void *w_sg, float *logits, float *gate_logit, int32_t *topk_idx,
                       float *topk_prob, float *topk_w, uint8_t *keep, void *ws,
                       moe_stream_t stream) {
  NvtxRange trace("moe_route");
  if (!shape_ok(shape)) return MOE_ERR_INVALID_ARG;
  if (!x || !W_r || !logits || !topk_idx || !topk_prob || !topk_w || !keep || !ws)
    return MOE_ERR_INVALID_ARG;
  if ((w_sg == nullptr) != (gate_logit == nullptr)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W_r) || !aligned16(ws) || !aligned4(logits)) return MOE_ERR_INVALID_ARG;
  if (shape->drop && subseq(shape) >= (int64_t(1) << 29)) return MOE_ERR_UNSUPPORTED;
  RouteArgs a = route_args(shape, ws);
  a.x = x; a.W_r = W_r; a.b_r = b_r; a.w_sg = w_sg; a.logits = logits; a.gate_logit = gate_logit;
  a.topk_idx = topk_idx; a.topk_prob = topk_prob; a.topk_w = topk_w; a.keep = keep;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = clear_capacity_counts(shape, a, s);
  if (e != cudaSuccess) return cuda_status(e);
  if (router_on_tensor_cores(shape) && (w_sg == nullptr || aligned16(w_sg))) {
    // logits on the tensor cores; softmax, Top-K and weights in its epilogue
    // (few experts) or in the Top-K kernel
    e = launch_router_tc(a, s);
    if (e == cudaSuccess && !router_routes_in_epilogue(shape->T, shape->d, shape->E, w_sg != nullptr))
      e = launch_topk_from_logits(a, s);
  } else {
    e = launch_router_fused(a, s);
  }
  if (e == cudaSuccess && shape->drop) e = launch_capacity(a, s);
  return cuda_status(e);
}

moe_status_t moe_route_topk(const moe_shape_t *shape, const float *logits, int32_t *topk_idx,
                            float *topk_prob, float *topk_w, uint8_t *keep, void *ws,
                            moe_stream_t stream) {
  NvtxRange trace("moe_route_topk");
  if (!shape_ok(shape)) return MOE_ERR_INVALID_ARG;
  if (!logits || !topk_idx || !topk_prob || !topk_w || !keep || !ws || !aligned16(ws))
    return MOE_ERR_INVALID_ARG;
  if (shape->drop && subseq(shape) >= (int64_t(1) << 29)) return MOE_ERR_UNSUPPORTED;
  RouteArgs a = route_args(shape, ws);
  a.logits = const_cast<float *>(logits);
  a.topk_idx = topk_idx; a.topk_prob = topk_prob; a.topk_w = topk_w; a.keep = keep;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = clear_capacity_counts(shape, a, s);
  if (e == cudaSuccess) e = launch_topk_from_logits(a, s);
  if (e == cudaSuccess && shape->drop) e = launch_capacity(a, s);
  return cuda_status(e);
}

moe_status_t moe_permute(const moe_shape_t *shape, const void *x, const int32_t *topk_idx,
                         const uint8_t *keep, void *Xp, int32_t *row_of, int32_t *src_of,
                         int32_t *counts, int32_t *offsets, void *ws, moe_stream_t stream) {
  NvtxRange trace("moe_permute");
  if (!shape_ok(shape)) return MOE_ERR_INVALID_ARG;
  if (!x || !topk_idx || !keep || !row_of || !src_of || !counts || !offsets || !ws)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || (Xp && !aligned16(Xp)) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  PermuteArgs a{};
  a.T = shape->T; a.d = shape->d; a.E = shape->E; a.K = shape->K; a.dtype = shape->dtype;
  a.x = x; a.topk_idx = topk_idx; a.keep = keep; a.Xp = Xp; a.row_of = row_of; a.src_of = src_of;
  a.counts = counts; a.offsets = offsets;
  a.blk_counts = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + layout(shape).map);
  a.status = status_word(ws);
  return cuda_status(launch_permute(a, (cudaStream_t)stream));
}

int64_t moe_padded_capacity(const moe_shape_t *shape) {
  if (!shape_ok(shape) || !shape->drop) return 0;
  const int64_t C = padded_rows_per_expert(shape->T, subseq(shape), shape->K, shape->E,
                                           shape->capacity_factor);
  return C * shape->E < (int64_t(1) << 31) ? C : 0;
}

moe_status_t moe_permute_padded(const moe_shape_t *shape, const void *x, const int32_t *topk_idx,
                                const uint8_t *keep, void *Xp, int32_t *row_of, int32_t *src_of,
                                int32_t *counts, int32_t *offsets, void *ws, moe_stream_t stream) {
  NvtxRange trace("moe_permute_padded");
  if (!shape_ok(shape)) return MOE_ERR_INVALID_ARG;
  if (!shape->drop) return MOE_ERR_UNSUPPORTED;   // dropless routing has no fixed capacity
  if (!x || !topk_idx || !keep || !row_of || !src_of || !counts || !offsets || !ws)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || (Xp && !aligned16(Xp)) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  const int64_t C = moe_padded_capacity(shape);
  if (C <= 0) return MOE_ERR_UNSUPPORTED;
  PermuteArgs a{};
  a.T = shape->T; a.d = shape->d; a.E = shape->E; a.K = shape->K; a.dtype = shape->dtype;
  a.x = x; a.topk_idx = topk_idx; a.keep = keep; a.Xp = Xp; a.row_of = row_of; a.src_of = src_of;
  a.counts = counts; a.offsets = offsets; a.pad_rows = C;
  a.blk_counts = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + layout(shape).map);
  a.status = status_word(ws);
  cudaError_t e = launch_permute(a, (cudaStream_t)stream);
  if (e == cudaSuccess) e = launch_pad_fill(a, (cudaStream_t)stream);
  return cuda_status(e);
}

moe_status_t moe_permute_noalloc(const moe_shape_t *shape, const void *x, const int32_t *topk_idx,
                                 const uint8_t *keep, void *Xp, int32_t *row_of, int32_t *src_of,
                                 int32_t *counts, int32_t *offsets, moe_stream_t stream) {
  NvtxRange trace("moe_permute_noalloc");
  if (!shape_ok(shape)) return MOE_ERR_INVALID_ARG;
  if (!x || !topk_idx || !keep || !Xp || !row_of || !src_of || !counts || !offsets)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Xp)) return MOE_ERR_INVALID_ARG;
  if (shape->T > MOE_PERMUTE_NOALLOC_MAX_TOKENS) return MOE_ERR_UNSUPPORTED;
  PermuteArgs a{};
  a.T = shape->T; a.d = shape->d; a.E = shape->E; a.K = shape->K; a.dtype = shape->dtype;
  a.x = x; a.topk_idx = topk_idx; a.keep = keep; a.Xp = Xp; a.row_of = row_of; a.src_of = src_of;
  a.counts = counts; a.offsets = offsets;
  return cuda_status(launch_permute_noalloc(a, (cudaStream_t)stream));
}

static moe_status_t ffn_check(int32_t dtype, int64_t max_rows, int32_t d, int32_t F,
                              int32_t n_groups, const int32_t *offsets, void *ws) {
  if ((dtype != MOE_F32 && dtype != MOE_BF16) || max_rows < 1 || d < 1 || F < 1 || n_groups < 1 ||
      n_groups > 64 || !offsets || !ws || !aligned16(ws))
    return MOE_ERR_INVALID_ARG;
  if (max_rows >= (int64_t(1) << 31)) return MOE_ERR_INVALID_ARG;
  if (dtype == MOE_BF16 && (d % 128 != 0 || F % 128 != 0)) return MOE_ERR_UNSUPPORTED;
  if (dtype == MOE_F32 && (d % 4 != 0)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t moe_expert_ffn(int32_t dtype, int64_t max_rows, int32_t d, int32_t F,
                            int32_t n_groups, const int32_t *offsets, const void *Xp,
                            const void *W_gu, const void *W_down, void *A_save, void *H_save,
                            void *Yp, void *ws, moe_stream_t stream) {
  NvtxRange trace("moe_expert_ffn");
  moe_status_t st = ffn_check(dtype, max_rows, d, F, n_groups, offsets, ws);
  if (st != MOE_OK) return st;
  if (!Xp || !W_gu || !W_down || !H_save || !Yp) return MOE_ERR_INVALID_ARG;
  if (!aligned16(Xp) || !aligned16(W_gu) || !aligned16(W_down) || !aligned16(H_save) ||
      !aligned16(Yp) || (A_save && !aligned16(A_save)))
    return MOE_ERR_INVALID_ARG;
  FfnArgs a{};
  a.dtype = dtype; a.max_rows = max_rows; a.d = d; a.F = F; a.n_groups = n_groups;
  a.offsets = offsets; a.Xp = Xp; a.W_gu = W_gu; a.W_down = W_down; a.A_save = A_save;
  a.H_save = H_save; a.Yp = Yp; a.status = status_word(ws);
  cudaStream_t s = (cudaStream_t)stream;
  return cuda_status(dtype == MOE_BF16 ? launch_ffn_fwd_bf16(a, s) : launch_ffn_fwd_f32(a, s));
}

moe_status_t moe_expert_ffn_gather(int64_t max_rows, int32_t d, int32_t F, int32_t n_groups,
                                   const int32_t *offsets, const void *x, int64_t T, int32_t K,
                                   const int32_t *src_of, const void *W_gu, const void *W_down,
                                   void *A_save, void *H_save, void *Yp, void *ws,
                                   moe_stream_t stream) {
  NvtxRange trace("moe_expert_ffn_gather");
  moe_status_t st = ffn_check(MOE_BF16, max_rows, d, F, n_groups, offsets, ws);
  if (st != MOE_OK) return st;
  if (T < 1 || K < 1 || K > 8 || T * (int64_t)K >= (int64_t(1) << 31)) return MOE_ERR_INVALID_ARG;
  if (!x || !src_of || !W_gu || !W_down || !H_save || !Yp) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W_gu) || !aligned16(W_down) || !aligned16(H_save) ||
      !aligned16(Yp) || (A_save && !aligned16(A_save)))
    return MOE_ERR_INVALID_ARG;
  FfnArgs a{};
  a.dtype = MOE_BF16; a.max_rows = max_rows; a.d = d; a.F = F; a.n_groups = n_groups;
  a.offsets = offsets; a.W_gu = W_gu; a.W_down = W_down; a.A_save = A_save;
  a.H_save = H_save; a.Yp = Yp; a.status = status_word(ws);
  a.x = x; a.src_of = src_of; a.K = K; a.T = T;
  const cudaError_t e = launch_ffn_fwd_bf16(a, (cudaStream_t)stream);
  return e == cudaErrorNotSupported ? MOE_ERR_UNSUPPORTED : cuda_status(e);
}

moe_status_t moe_unpermute(const moe_shape_t *shape, const void *Yp, const int32_t *row_of,
                           const float *topk_w, const void *Ys, const float *gate_logit, void *out,
                           moe_stream_t stream) {
  NvtxRange trace("moe_unpermute");
  if (!shape_ok(shape)) return MOE_ERR_INVALID_ARG;
  if (!Yp || !row_of || !topk_w || !out) return MOE_ERR_INVALID_ARG;
  if ((Ys == nullptr) != (gate_logit == nullptr)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(Yp) || !aligned16(out) || (Ys && !aligned16(Ys))) return MOE_ERR_INVALID_ARG;
  UnpermuteArgs a{};
  a.T = shape->T; a.d = shape->d; a.K = shape->K; a.dtype = shape->dtype;
  a.Yp = Yp; a.row_of = row_of; a.topk_w = topk_w; a.Ys = Ys; a.gate_logit = gate_logit; a.out = out;
  return cuda_status(launch_unpermute(a, (cudaStream_t)stream));
}

moe_status_t moe_unpermute_bwd(const moe_shape_t *shape, const void *dout, const void *Yp,
                               const int32_t *row_of, const float *topk_w, const void *Ys,
                               const float *gate_logit, void *dYp, float *dw, void *dYs, float *dz,
                               moe_stream_t stream) {
  NvtxRange trace("moe_unpermute_bwd");
  if (!shape_ok(shape)) return MOE_ERR_INVALID_ARG;
  if (!dout || !Yp || !row_of || !topk_w || !dYp || !dw) return MOE_ERR_INVALID_ARG;
  const bool sh = Ys != nullptr;
  if ((gate_logit != nullptr) != sh || (dYs != nullptr) != sh || (dz != nullptr) != sh)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(dout) || !aligned16(Yp) || !aligned16(dYp) || (sh && (!aligned16(Ys) || !aligned16(dYs))))
    return MOE_ERR_INVALID_ARG;
  UnpermuteArgs a{};
  a.T = shape->T; a.d = shape->d; a.K = shape->K; a.dtype = shape->dtype;
  a.dout = dout; a.Yp = Yp; a.row_of = row_of; a.topk_w = topk_w; a.Ys = Ys;
  a.gate_logit = gate_logit; a.dYp = dYp; a.dw = dw; a.dYs = dYs; a.dz = dz;
  return cuda_status(launch_unpermute_bwd(a, (cudaStream_t)stream));
}

moe_status_t moe_expert_ffn_bwd(int32_t dtype, int64_t max_rows, int32_t d, int32_t F,
                                int32_t n_groups, const int32_t *offsets, const void *dYp,
                                const void *Xp, const void *A_save, const void *H_save,
                                const void *W_gu, const void *W_down, void *dA, float *dXp,
                                float *dW_gu, float *dW_down, void *ws, size_t ws_bytes,
                                moe_stream_t stream) {
  NvtxRange trace("moe_expert_ffn_bwd");
  moe_status_t st = ffn_check(dtype, max_rows, d, F, n_groups, offsets, ws);
  if (st != MOE_OK) return st;
  if (ws_bytes < MOE_FFN_BWD_WORKSPACE_BYTES) return MOE_ERR_INVALID_ARG;
  if (!dYp || !Xp || !A_save || !H_save || !W_gu || !W_down || !dA || !dXp || !dW_gu || !dW_down)
    return MOE_ERR_INVALID_ARG;
  const void *ptrs[] = {dYp, Xp, A_save, H_save, W_gu, W_down, dA, dXp, dW_gu, dW_down};
  for (const void *q : ptrs)
    if (!aligned16(q)) return MOE_ERR_INVALID_ARG;
  FfnArgs a{};
  a.dtype = dtype; a.max_rows = max_rows; a.d = d; a.F = F; a.n_groups = n_groups;
  a.offsets = offsets; a.dYp = dYp; a.Xp = Xp; a.A_save = const_cast<void *>(A_save);
  a.H_save = const_cast<void *>(H_save); a.W_gu = W_gu; a.W_down = W_down; a.dA = dA;
  a.dXp = dXp; a.dW_gu = dW_gu; a.dW_down = dW_down; a.status = status_word(ws);
  // group tensor maps after the status word, 128-byte aligned
  a.maps = reinterpret_cast<void *>((reinterpret_cast<uintptr_t>(ws) + kStatusBytes + 127) &
                                    ~uintptr_t(127));
  static_assert(kStatusBytes + 127 + kFfnMapBytes <= MOE_FFN_BWD_WORKSPACE_BYTES,
                "group maps exceed the documented workspace");
  cudaStream_t s = (cudaStream_t)stream;
  return cuda_status(dtype == MOE_BF16 ? launch_ffn_bwd_bf16(a, s) : launch_ffn_bwd_f32(a, s));
}

moe_status_t moe_permute_bwd(const moe_shape_t *shape, const float *dXp, const int32_t *row_of,
                             const float *dx_add, float *dx, moe_stream_t stream) {
  NvtxRange trace("moe_permute_bwd");
  if (!shape_ok(shape)) return MOE_ERR_INVALID_ARG;
  if (!dXp || !row_of || !dx || !aligned16(dXp) || !aligned16(dx) || (dx_add && !aligned16(dx_add)))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_permute_bwd(shape->T, shape->d, shape->K, dXp, row_of, dx_add, dx,
                                        (cudaStream_t)stream));
}

moe_status_t moe_sum_partials(int32_t dtype, int32_t n_parts, int64_t rows, int32_t d,
                              const void *partials, void *out, moe_stream_t stream) {
  NvtxRange trace("moe_sum_partials");
  if (dtype != MOE_BF16 && dtype != MOE_F32) return MOE_ERR_INVALID_ARG;
  if (n_parts < 1 || n_parts > 16 || rows < 0 || d < 1) return MOE_ERR_INVALID_ARG;
  if (d % (dtype == MOE_BF16 ? 8 : 4) != 0) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!partials || !out || !aligned16(partials) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  const size_t b = dtype == MOE_BF16 ? 2 : 4;
  const char *p0 = static_cast<const char *>(partials), *o0 = static_cast<const char *>(out);
  const size_t part = (size_t)rows * d * b;
  if (o0 < p0 + part * n_parts && p0 < o0 + part) return MOE_ERR_INVALID_ARG;   // aliasing
  return cuda_status(launch_sum_partials(dtype, n_parts, rows, d, partials, out,
                                         (cudaStream_t)stream));
}

moe_status_t moe_route_bwd(const moe_shape_t *shape, const void *x, const void *W_r,
                           const void *w_sg, const float *logits, const int32_t *topk_idx,
                           const float *topk_prob, const float *topk_w, const float *dw,
                           const float *dz, const float *dx_in, float *dW_r, float *db_r,
                           float *dw_sg, float *dx_router, void *ws, moe_stream_t stream) {
  NvtxRange trace("moe_route_bwd");
  if (!shape_ok(shape)) return MOE_ERR_INVALID_ARG;
  if (!x || !W_r || !logits || !topk_idx || !topk_prob || !topk_w || !dw || !dW_r || !dx_router || !ws)
    return MOE_ERR_INVALID_ARG;
  const bool sh = w_sg != nullptr;
  if ((dz != nullptr) != sh || (dw_sg != nullptr) != sh) return MOE_ERR_INVALID_ARG;
  if (!aligned16(ws) || !aligned16(x) || !aligned16(W_r) || (sh && !aligned16(w_sg)) ||
      !aligned16(dx_router) || (dx_in != nullptr && !aligned16(dx_in)))
    return MOE_ERR_INVALID_ARG;   // 16-byte vector accesses
  const Layout L = layout(shape);
  RouteBwdArgs a{};
  a.T = shape->T; a.d = shape->d; a.E = shape->E; a.K = shape->K; a.dtype = shape->dtype;
  a.renorm = shape->renorm; a.x = x; a.W_r = W_r; a.w_sg = w_sg; a.logits = logits;
  a.topk_idx = topk_idx; a.topk_prob = topk_prob; a.topk_w = topk_w; a.dw = dw; a.dz = dz;
  a.dx_in = dx_in; a.dW_r = dW_r; a.db_r = db_r; a.dw_sg = dw_sg; a.dx_router = dx_router;
  a.dl = reinterpret_cast<float *>(static_cast<char *>(ws) + L.rbwd);
  a.partial = a.dl + align256((size_t)shape->T * shape->E * sizeof(float)) / sizeof(float);
  a.status = status_word(ws);
  return cuda_status(launch_route_bwd(a, (cudaStream_t)stream));
}

}  // extern "C"
