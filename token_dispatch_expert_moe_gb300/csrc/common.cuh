// Internal helpers shared by the kernels of libmoe.so (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// ---------------------------------------------------------------------------
// Workspace layout. The status word lives in the first 256 bytes of `ws`.
constexpr size_t kStatusBytes = 256;

struct Status {
  uint32_t code;  // first device-side error (moe_status_t), 0 if none
  uint32_t info;  // kernel-specific detail
};

__device__ __forceinline__ void report(uint32_t *status, uint32_t code, uint32_t info) {
  if (status != nullptr && atomicCAS(status, 0u, code) == 0u) {
    atomicExch(status + 1, info);
  }
}

// Detail words recorded with MOE_ERR_DEVICE / MOE_ERR_TIMEOUT.
enum : uint32_t {
  kInfoRowRange = 0x100,      // a permuted row index outside [0, max_rows)
  kInfoExpertRange = 0x200,   // an expert index outside [0, E)
  kInfoOffsets = 0x300,       // offsets not monotone or beyond max_rows
  kInfoPadOverflow = 0x400,   // padded layout: more kept rows for an expert than its capacity
  kInfoGemmTimeout = 0x1000,  // + role: a GEMM pipeline wait gave up
};

// ---------------------------------------------------------------------------
// Element access for the two activation dtypes.
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(float v) { return v; }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// 16-byte vectors: 8 bf16 or 4 fp32.
template <typename T> struct Vec;
template <> struct Vec<__nv_bfloat16> { static constexpr int N = 8; };
template <> struct Vec<float> { static constexpr int N = 4; };

// 16 loaded bytes (8 bf16 or 4 fp32) to fp32
template <typename T>
__device__ __forceinline__ void unpack16(const uint4 &u, float (&v)[Vec<T>::N]) {
  if constexpr (Vec<T>::N == 8) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  } else {
    const float *f = reinterpret_cast<const float *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = f[i];
  }
}

template <typename T>
__device__ __forceinline__ void load16(const T *p, float (&v)[Vec<T>::N]) {
  unpack16<T>(*reinterpret_cast<const uint4 *>(p), v);
}

template <typename T>
__device__ __forceinline__ void store16(T *p, const float (&v)[Vec<T>::N]) {
  uint4 u;
  if constexpr (Vec<T>::N == 8) {
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  } else {
    float *f = reinterpret_cast<float *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = v[i];
  }
  *reinterpret_cast<uint4 *>(p) = u;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Fixed-order block reduction (blockDim.x a multiple of 32, <= 1024):
// warp butterflies, then warp 0 reduces the per-warp sums. Same order on
// every run, so the result is bitwise reproducible.
__device__ __forceinline__ float block_sum(float v, float *smem32) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) smem32[warp] = v;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  float r = (lane < nw) ? smem32[lane] : 0.0f;
  if (warp == 0) r = warp_sum(r);
  if (threadIdx.x == 0) smem32[0] = r;
  __syncthreads();
  r = smem32[0];
  __syncthreads();
  return r;
}

// ---------------------------------------------------------------------------
// Launch helpers implemented in the kernel translation units.

struct RouteArgs {
  int64_t T;
  int d, E, K, dtype, renorm, drop;
  int64_t S;  // sub-sequence length (>= 1)
  float cf;   // capacity factor
  const void *x, *W_r, *w_sg;
  const float *b_r;
  float *logits, *gate_logit;
  int32_t *topk_idx;
  float *topk_prob, *topk_w;
  uint8_t *keep;
  uint32_t *status;
  unsigned long long *cap_keys;  // ws region: capacity candidate lists [n_sub][E][S]
  uint32_t *cap_counts;          // ws region: list lengths [n_sub][E], zeroed by the call
};

constexpr int kRouterMaxSplit = 4;
// K splits of the router GEMM for T tokens of hidden size d (d % 64 == 0):
// as many as leave no SM idle, at most kRouterMaxSplit, >= 8 K blocks each
int router_k_split(int64_t T, int d);

cudaError_t launch_router_fused(const RouteArgs &a, cudaStream_t s);
cudaError_t launch_router_tc(const RouteArgs &a, cudaStream_t s);  // bf16, d % 64 == 0
// whether launch_router_tc also routes (softmax, Top-K, weights); if not,
// launch_topk_from_logits follows it
bool router_routes_in_epilogue(int64_t T, int d, int E, int has_gate);
cudaError_t launch_topk_from_logits(const RouteArgs &a, cudaStream_t s);
// capacity dropping (drop = 1): a.cap_counts must be zero (moe_route and
// moe_route_topk clear it with a memset before their first kernel)
cudaError_t launch_capacity(const RouteArgs &a, cudaStream_t s);

struct PermuteArgs {
  int64_t T;
  int d, E, K, dtype;
  const void *x;
  const int32_t *topk_idx;
  const uint8_t *keep;
  void *Xp;
  int32_t *row_of, *src_of, *counts, *offsets;
  int32_t *blk_counts;  // ws region [nblk, E]
  uint32_t *status;
  int64_t pad_rows;     // 0: compact layout; > 0: expert e owns rows [e*pad_rows, (e+1)*pad_rows)
};
cudaError_t launch_permute(const PermuteArgs &a, cudaStream_t s);
cudaError_t launch_pad_fill(const PermuteArgs &a, cudaStream_t s);
// Rows per expert of the padded layout: sum over sub-sequences of
// min(capacity, sub-sequence length) (an expert takes at most one slot per token).
int64_t padded_rows_per_expert(int64_t T, int64_t S, int K, int E, float cf);
cudaError_t launch_permute_noalloc(PermuteArgs a, cudaStream_t s);

struct UnpermuteArgs {
  int64_t T;
  int d, K, dtype;
  const void *Yp, *Ys, *dout;
  const int32_t *row_of;
  const float *topk_w, *gate_logit;
  void *out, *dYp, *dYs;
  float *dw, *dz;
};
cudaError_t launch_unpermute(const UnpermuteArgs &a, cudaStream_t s);
cudaError_t launch_unpermute_bwd(const UnpermuteArgs &a, cudaStream_t s);
cudaError_t launch_sum_partials(int dtype, int n_parts, int64_t rows, int d, const void *partials,
                                void *out, cudaStream_t s);
cudaError_t launch_permute_bwd(int64_t T, int d, int K, const float *dXp,
                               const int32_t *row_of, const float *dx_add, float *dx,
                               cudaStream_t s);

struct FfnArgs {
  int dtype;
  int64_t max_rows;
  int d, F, n_groups;
  const int32_t *offsets;
  const void *Xp, *W_gu, *W_down;
  void *A_save, *H_save, *Yp;
  // backward
  const void *dYp;
  void *dA;
  float *dXp, *dW_gu, *dW_down;
  void *H_tmp;  // fwd scratch for H when H_save is NULL (ws)
  // fwd, bf16: when x is set, the gate/up GEMM gathers its A rows from x
  // [T, d] through src_of (row R is token src_of[R] / K) instead of reading Xp
  const void *x;
  const int32_t *src_of;
  int K;
  int64_t T;
  void *maps;   // bwd (bf16): kFfnMapBytes of workspace, 128-byte aligned, for group tensor maps
  uint32_t *status;
};
// Group tensor maps of the bf16 weight-gradient GEMMs: 2 modes x 2 maps x 64
// groups x 128 bytes, after the 256-byte status word (rounded to 128 bytes).
constexpr int kMaxMapGroups = 64;
constexpr size_t kFfnMapBytes = 2 * 2 * kMaxMapGroups * 128;
constexpr size_t kFfnBwdWorkspaceBytes = 256 + 128 + kFfnMapBytes;
size_t ffn_workspace_bytes(int dtype, int64_t max_rows, int d, int F);
cudaError_t launch_ffn_fwd_f32(const FfnArgs &a, cudaStream_t s);
cudaError_t launch_ffn_bwd_f32(const FfnArgs &a, cudaStream_t s);
cudaError_t launch_ffn_fwd_bf16(const FfnArgs &a, cudaStream_t s);
cudaError_t launch_ffn_bwd_bf16(const FfnArgs &a, cudaStream_t s);

struct RouteBwdArgs {
  int64_t T;
  int d, E, K, dtype, renorm;
  const void *x, *W_r, *w_sg;
  const float *logits, *topk_prob, *topk_w, *dw, *dz, *dx_in;
  const int32_t *topk_idx;
  float *dW_r, *db_r, *dw_sg, *dx_router;
  float *dl;       // ws [T, E]
  float *partial;  // ws [nchunk, E+1, d]
  uint32_t *status;
};
size_t route_bwd_workspace_bytes(int64_t T, int d, int E);
cudaError_t launch_route_bwd(const RouteBwdArgs &a, cudaStream_t s);

// Router backward on the tensor cores (bf16 layers, d % 256 == 0): dl split
// into three bf16 planes (hi + mid + lo carries dl to ~fp32 precision) in
// P [T, 4*PW] (plane k in columns [k*PW, k*PW + C), zeros elsewhere), and
// Wr3 [3*PW, d] = W_r (+ w_sg row) repeated per plane.
//   dW: out_w [nsplit, 4*PW, d] fp32 = P^T x per token chunk (weight-gradient
//       GEMM with one group per chunk);
//   dx: dx_router [T, d] fp32 = P[:, :3PW] Wr3 (dXp-mode GEMM, K = 3*PW),
//       skipped when dx_router is NULL.
struct RouterBwdTc {
  int64_t T;
  int d, PW;
  const void *planes, *x, *Wr3;
  float *out_w, *dx_router;   // out_w: [nsplit, 4*PW, d], one slice per token chunk
  const int32_t *offs;  // [nsplit + 1] token-chunk boundaries, offs[0] = 0, offs[nsplit] = T;
                        // offs[32..33] = {0, T} for the dx GEMM
  int nsplit;
  void *maps;           // 2 * nsplit tensor maps, 128-byte aligned
  uint32_t *status;
};
cudaError_t launch_router_bwd_tc(const RouterBwdTc &a, cudaStream_t s);

}  // namespace moe
