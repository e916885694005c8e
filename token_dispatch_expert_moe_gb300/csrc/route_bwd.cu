// Router backward: renormalisation, softmax and logits-GEMV gradients.
//
// MoE Parallel Folding (arXiv 2504.14960) study notes, "method overview": the
// backward runs the dispatcher chain in reverse. Routing decisions (Top-K
// set, drops) are constants; gradient reaches the router only through the
// combine weights w = prob / Z.
//   1. dl_kernel (one warp per token): p = softmax(logits) (same fp32
//      arithmetic as the forward); dp on the Top-K slots
//      ((g - <g,w>) / Z with renorm, g without); dl = p (dp - <p,dp>).
//   2. dx_kernel: dx_router[t] = dx_in[t] + sum_e dl[t,e] W_r[e] + dz[t] w_sg,
//      64 tokens x 256 hidden columns per CTA, each thread's W_r column in
//      registers.
//   3. wgrad_partial_kernel: per chunk of tokens, partial sums of
//      dl^T x (and dz^T x), then reduce_kernel adds the chunks in order:
//      deterministic, no atomics.
#include "common.cuh"
#include "softmax.cuh"

namespace moe {
namespace {

constexpr int kDxTok = 64;   // tokens per dx CTA
constexpr int kCols = 256;   // hidden columns per CTA
constexpr int kChunks = 32;  // token chunks of the dW_r partial sums

__global__ void __launch_bounds__(256) dl_kernel(RouteBwdArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= a.T) return;
  const int E = a.E, K = a.K;
  const float *l = a.logits + t * E;
  float p0, p1;
  spec::softmax_warp(lane < E ? l[lane] : 0.0f, lane + 32 < E ? l[lane + 32] : 0.0f, E, p0, p1);
  // slot values, replicated in every lane (K <= 8)
  float gw = 0.0f, Z = 0.0f;
  for (int k = 0; k < K; ++k) {
    gw = fmaf(a.dw[t * K + k], a.topk_w[t * K + k], gw);
    Z += a.topk_prob[t * K + k];
  }
  float dp0 = 0.0f, dp1 = 0.0f;
  for (int k = 0; k < K; ++k) {
    const float g = a.dw[t * K + k];
    const float dpk = a.renorm ? (g - gw) / Z : g;
    const int e = a.topk_idx[t * K + k];
    if (e == lane) dp0 = dpk;
    if (e == lane + 32) dp1 = dpk;
  }
  const bool v0 = lane < E, v1 = lane + 32 < E;
  float s = (v0 ? p0 * dp0 : 0.0f) + (v1 ? p1 * dp1 : 0.0f);
  s = warp_sum(s);
  if (v0) a.dl[t * E + lane] = p0 * (dp0 - s);
  if (v1) a.dl[t * E + lane + 32] = p1 * (dp1 - s);
}

// dx_router[t, j] = dx_in[t, j] + sum_c dl[t, c] W[c, j]  (row c = E is w_sg
// with dl = dz). One thread per column j holds W[:, j] in registers for 64
// tokens; dl rows are read from shared memory as float4 broadcasts.
template <typename T, int CP>
__global__ void __launch_bounds__(kCols) dx_kernel(RouteBwdArgs a) {
  __shared__ __align__(16) float dls[kDxTok][CP];
  const int E = a.E;
  const int C = E + (a.w_sg != nullptr ? 1 : 0);
  const int64_t t0 = (int64_t)blockIdx.x * kDxTok;
  const int j = blockIdx.y * kCols + threadIdx.x;
  const T *W = reinterpret_cast<const T *>(a.W_r);
  const T *wsg = reinterpret_cast<const T *>(a.w_sg);
  float w[CP];
#pragma unroll
  for (int c = 0; c < CP; ++c)
    w[c] = (j < a.d && c < C) ? to_f32(c < E ? W[(int64_t)c * a.d + j] : wsg[j]) : 0.0f;
  for (int i = threadIdx.x; i < kDxTok * CP; i += blockDim.x) {
    const int tt = i / CP, c = i % CP;
    const int64_t t = t0 + tt;
    float v = 0.0f;
    if (t < a.T && c < C) v = c < E ? a.dl[t * E + c] : a.dz[t];
    dls[tt][c] = v;
  }
  __syncthreads();
  if (j >= a.d) return;
  // two tokens at a time, four partial sums each (combined in a fixed order)
  for (int tt = 0; tt < kDxTok; tt += 2) {
    const int64_t t = t0 + tt;
    if (t >= a.T) break;
    const bool two = t + 1 < a.T;
    float p0[4] = {0.f, 0.f, 0.f, 0.f}, p1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < CP; c += 4) {
      const float4 v = *reinterpret_cast<const float4 *>(&dls[tt][c]);
      const float4 u = *reinterpret_cast<const float4 *>(&dls[tt + 1][c]);
      p0[0] = fmaf(v.x, w[c], p0[0]);
      p0[1] = fmaf(v.y, w[c + 1], p0[1]);
      p0[2] = fmaf(v.z, w[c + 2], p0[2]);
      p0[3] = fmaf(v.w, w[c + 3], p0[3]);
      p1[0] = fmaf(u.x, w[c], p1[0]);
      p1[1] = fmaf(u.y, w[c + 1], p1[1]);
      p1[2] = fmaf(u.z, w[c + 2], p1[2]);
      p1[3] = fmaf(u.w, w[c + 3], p1[3]);
    }
    const float in0 = a.dx_in != nullptr ? a.dx_in[t * a.d + j] : 0.0f;
    a.dx_router[t * a.d + j] = in0 + ((p0[0] + p0[1]) + (p0[2] + p0[3]));
    if (two) {
      const float in1 = a.dx_in != nullptr ? a.dx_in[(t + 1) * a.d + j] : 0.0f;
      a.dx_router[(t + 1) * a.d + j] = in1 + ((p1[0] + p1[1]) + (p1[2] + p1[3]));
    }
  }
}

// Partial sums over one chunk of tokens of dl^T x (and dz^T x): one thread per
// column j keeps CP accumulators; 32 tokens of dl and x are staged in shared
// memory per step.
template <typename T, int CP>
__global__ void __launch_bounds__(kCols) wgrad_partial_kernel(RouteBwdArgs a, int64_t chunk) {
  __shared__ __align__(16) float dls[32][CP];
  __shared__ float xs[32][kCols];
  const int E = a.E;
  const int C = E + (a.w_sg != nullptr ? 1 : 0);
  const int64_t tb = (int64_t)blockIdx.x * chunk;
  const int64_t te = min(a.T, tb + chunk);
  const int j0 = blockIdx.y * kCols;
  const int j = j0 + threadIdx.x;
  const T *x = reinterpret_cast<const T *>(a.x);
  float acc[CP];
#pragma unroll
  for (int c = 0; c < CP; ++c) acc[c] = 0.0f;
  for (int64_t s0 = tb; s0 < te; s0 += 32) {
    __syncthreads();
    for (int i = threadIdx.x; i < 32 * CP; i += blockDim.x) {
      const int tt = i / CP, c = i % CP;
      const int64_t t = s0 + tt;
      float v = 0.0f;
      if (t < te && c < C) v = c < E ? a.dl[t * E + c] : a.dz[t];
      dls[tt][c] = v;
    }
#pragma unroll 8
    for (int tt = 0; tt < 32; ++tt) {
      const int64_t t = s0 + tt;
      xs[tt][threadIdx.x] = (t < te && j < a.d) ? to_f32(x[t * a.d + j]) : 0.0f;
    }
    __syncthreads();
    const int n = (int)min((int64_t)32, te - s0);
    for (int tt = 0; tt < n; ++tt) {
      const float xv = xs[tt][threadIdx.x];
#pragma unroll
      for (int c = 0; c < CP; c += 4) {
        const float4 v = *reinterpret_cast<const float4 *>(&dls[tt][c]);
        acc[c] = fmaf(v.x, xv, acc[c]);
        acc[c + 1] = fmaf(v.y, xv, acc[c + 1]);
        acc[c + 2] = fmaf(v.z, xv, acc[c + 2]);
        acc[c + 3] = fmaf(v.w, xv, acc[c + 3]);
      }
    }
  }
  if (j >= a.d) return;
  float *part = a.partial + (int64_t)blockIdx.x * C * a.d;
#pragma unroll
  for (int c = 0; c < CP; ++c)
    if (c < C) part[(int64_t)c * a.d + j] = acc[c];
}

__global__ void reduce_kernel(RouteBwdArgs a, int nchunk) {
  const int E = a.E;
  const int C = E + (a.w_sg != nullptr ? 1 : 0);
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)C * a.d) return;
  float s = 0.0f;
  for (int c = 0; c < nchunk; ++c) s += a.partial[(int64_t)c * C * a.d + i];
  const int row = (int)(i / a.d), j = (int)(i % a.d);
  if (row < E)
    a.dW_r[(int64_t)row * a.d + j] = s;
  else
    a.dw_sg[j] = s;
}

__global__ void __launch_bounds__(1024) db_kernel(RouteBwdArgs a) {
  __shared__ float red[32];
  const int e = blockIdx.x;
  float s = 0.0f;
  for (int64_t t = threadIdx.x; t < a.T; t += blockDim.x) s += a.dl[t * a.E + e];
  s = block_sum(s, red);
  if (threadIdx.x == 0) a.db_r[e] = s;
}

}  // namespace

size_t route_bwd_workspace_bytes(int64_t T, int d, int E) {
  const size_t dl = ((size_t)T * E * sizeof(float) + 255) & ~size_t(255);
  return dl + (size_t)kChunks * (E + 1) * d * sizeof(float);
}

template <int CP>
void launch_cp(const RouteBwdArgs &a, cudaStream_t s, int64_t chunk, int nchunk) {
  dim3 gdx((unsigned)((a.T + kDxTok - 1) / kDxTok), (unsigned)((a.d + kCols - 1) / kCols));
  dim3 gw((unsigned)nchunk, (unsigned)((a.d + kCols - 1) / kCols));
  if (a.dtype == MOE_BF16) {
    dx_kernel<__nv_bfloat16, CP><<<gdx, kCols, 0, s>>>(a);
    wgrad_partial_kernel<__nv_bfloat16, CP><<<gw, kCols, 0, s>>>(a, chunk);
  } else {
    dx_kernel<float, CP><<<gdx, kCols, 0, s>>>(a);
    wgrad_partial_kernel<float, CP><<<gw, kCols, 0, s>>>(a, chunk);
  }
}

cudaError_t launch_route_bwd(const RouteBwdArgs &a, cudaStream_t s) {
  dl_kernel<<<(unsigned)((a.T * 32 + 255) / 256), 256, 0, s>>>(a);
  const int64_t chunk = (a.T + kChunks - 1) / kChunks;
  const int nchunk = (int)((a.T + chunk - 1) / chunk);
  const int C = a.E + (a.w_sg != nullptr ? 1 : 0);
  if (C <= 8) launch_cp<8>(a, s, chunk, nchunk);
  else if (C <= 16) launch_cp<16>(a, s, chunk, nchunk);
  else if (C <= 32) launch_cp<32>(a, s, chunk, nchunk);
  else launch_cp<68>(a, s, chunk, nchunk);
  const int64_t n = (int64_t)C * a.d;
  reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a, nchunk);
  if (a.db_r != nullptr) db_kernel<<<a.E, 1024, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
