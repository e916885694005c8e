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
//      register-tiled (8 tokens x 4 columns per thread);
//   3. wgrad_partial_kernel: per chunk of tokens, partial sums of dl^T x (and
//      dz^T x), register-tiled; reduce_kernel adds the chunks in order:
//      deterministic, no atomics.
// bf16 layers with d % 256 == 0 take steps 2 and 3 to the tensor cores
// instead (the section "Tensor-core path" below): dl is split into three
// bf16 planes, dx_router and dW_r become grouped-GEMM calls (gemm_tc.cu),
// and plane_sum_kernel adds the planes and token chunks in order; with a
// dx_in addend (a shared expert) dx stays on dx_kernel.
#include "common.cuh"
#include "softmax.cuh"

namespace moe {
namespace {

constexpr int kCols = 256;   // hidden columns per dW_r CTA
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
// with dl = dz). A CTA takes 128 tokens and `nsub` consecutive 64-column
// tiles of W: the dl tile stays in shared memory in its natural [token][c]
// layout, and the W tiles (converted to fp32) pass through a double buffer,
// the next one loaded into registers while the current one is used. Each
// thread computes 8 tokens x 4 columns: per 4 values of c it reads 8 float4
// of dl (broadcast within each half-warp) and 4 float4 of W for 128 FMAs.
// The sum over c runs in ascending order per output.
constexpr int kDxT = 128, kDxJ = 64;
template <int CP> constexpr size_t dx_smem_bytes() {
  return (size_t)(kDxT + 2 * kDxJ) * CP * sizeof(float);
}

template <typename T, int CP>
__global__ void __launch_bounds__(256, 2) dx_kernel(RouteBwdArgs a, int nsub) {
  extern __shared__ __align__(16) float dx_smem[];
  float *dls = dx_smem;                       // [kDxT][CP]
  float *Wbuf = dx_smem + kDxT * CP;          // [2][CP][kDxJ]
  constexpr int NV = Vec<T>::N;
  constexpr int VPR = kDxJ / NV;              // 16-byte vectors per W row of a tile
  constexpr int WV = (CP * VPR + 255) / 256;  // W vectors per thread per tile
  const int E = a.E;
  const int C = E + (a.w_sg != nullptr ? 1 : 0);
  const int64_t t0 = (int64_t)blockIdx.x * kDxT;
  const T *W = reinterpret_cast<const T *>(a.W_r);
  const T *wsg = reinterpret_cast<const T *>(a.w_sg);
  for (int i = threadIdx.x; i < kDxT * CP; i += blockDim.x) {
    const int tt = i / CP, c = i - tt * CP;
    const int64_t t = t0 + tt;
    float v = 0.0f;
    if (t < a.T && c < C) v = c < E ? a.dl[t * E + c] : a.dz[t];
    dls[i] = v;
  }
  uint4 wr[WV];
  auto fetch_w = [&](int j0) {   // this thread's vectors of the W tile at column j0
#pragma unroll
    for (int q = 0; q < WV; ++q) {
      const int i = threadIdx.x + q * 256;
      const int c = i / VPR, j = j0 + (i - c * VPR) * NV;
      wr[q] = (i < CP * VPR && c < C && j < a.d)   // d is a multiple of NV
                  ? *reinterpret_cast<const uint4 *>((c < E ? W + (int64_t)c * a.d : wsg) + j)
                  : make_uint4(0, 0, 0, 0);
    }
  };
  auto stash_w = [&](float *Ws) {
#pragma unroll
    for (int q = 0; q < WV; ++q) {
      const int i = threadIdx.x + q * 256;
      if (i < CP * VPR) {
        const int c = i / VPR, jv = (i - c * VPR) * NV;
        float v[NV];
        unpack16<T>(wr[q], v);
#pragma unroll
        for (int k = 0; k < NV; k += 4)
          *reinterpret_cast<float4 *>(&Ws[c * kDxJ + jv + k]) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
      }
    }
  };
  const int jfirst = blockIdx.y * nsub * kDxJ;
  if (jfirst >= a.d) return;
  fetch_w(jfirst);
  stash_w(Wbuf);
  __syncthreads();   // dl tile and the first W tile
  const int tq = threadIdx.x >> 4;   // token octet 0..15
  const int jq = threadIdx.x & 15;   // column quad 0..15
  for (int sub = 0; sub < nsub; ++sub) {
    const int j0 = jfirst + sub * kDxJ;
    if (j0 >= a.d) break;   // the same for every thread of the CTA
    const bool next = sub + 1 < nsub && j0 + kDxJ < a.d;
    if (next) fetch_w(j0 + kDxJ);   // in flight while this tile is used
    const float *Ws = Wbuf + (sub & 1) * CP * kDxJ;
    const int j = j0 + jq * 4;
    float4 xin[8];
    if (a.dx_in != nullptr && j < a.d) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int64_t t = t0 + tq * 8 + i;
        xin[i] = t < a.T ? *reinterpret_cast<const float4 *>(a.dx_in + t * a.d + j)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) xin[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int n = 0; n < 4; ++n) acc[i][n] = 0.0f;
#pragma unroll 2
    for (int c = 0; c < CP; c += 4) {
      float w[4][4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 wv = *reinterpret_cast<const float4 *>(&Ws[(c + k) * kDxJ + jq * 4]);
        w[k][0] = wv.x; w[k][1] = wv.y; w[k][2] = wv.z; w[k][3] = wv.w;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 dv = *reinterpret_cast<const float4 *>(&dls[(tq * 8 + i) * CP + c]);
        const float d4[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int n = 0; n < 4; ++n) acc[i][n] = fmaf(d4[k], w[k][n], acc[i][n]);
      }
    }
    if (j < a.d) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int64_t t = t0 + tq * 8 + i;
        if (t >= a.T) break;
        float4 o = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        if (a.dx_in != nullptr) {   // (0 + sum) + dx_in, as before
          o.x += xin[i].x; o.y += xin[i].y; o.z += xin[i].z; o.w += xin[i].w;
        }
        *reinterpret_cast<float4 *>(a.dx_router + t * a.d + j) = o;
      }
    }
    if (next) stash_w(Wbuf + ((sub + 1) & 1) * CP * kDxJ);
    __syncthreads();   // the next tile is in place; this one's reads are done
  }
}

// Partial sums over one chunk of tokens of dl^T x (row E: dz^T x): a
// CP x 256 tile per CTA (CP a multiple of 8, rows >= C zero), each thread
// CP/8 rows x 8 columns. Per token a thread reads CP/8 dl values and two
// float4 of x from shared memory for CP FMAs. Tokens pass through shared
// memory 32 at a time; the next 32 are loaded into registers (16-byte
// vectors of x) while the current ones are summed.
template <typename T, int CP>
__global__ void __launch_bounds__(256, 2) wgrad_partial_kernel(RouteBwdArgs a, int64_t chunk) {
  constexpr int RPT = CP / 8;                    // rows of the tile per thread
  constexpr int NV = Vec<T>::N;                  // elements of x per 16-byte vector
  constexpr int XV = 32 * kCols / NV / 256;      // x vectors per thread per slab
  constexpr int DV = (32 * CP + 255) / 256;      // dl values per thread per slab
  __shared__ __align__(16) float dls[32][CP];
  __shared__ __align__(16) float xs[32][kCols];
  const int E = a.E;
  const int C = E + (a.w_sg != nullptr ? 1 : 0);
  const int64_t tb = (int64_t)blockIdx.x * chunk;
  const int64_t te = min(a.T, tb + chunk);
  const int j0 = blockIdx.y * kCols;
  const int rg = threadIdx.x >> 5;   // row group 0..7 (one per warp)
  const int jo = threadIdx.x & 31;   // column octet 0..31
  const T *x = reinterpret_cast<const T *>(a.x);
  uint4 xr[XV];
  float dr[DV];
  auto fetch = [&](int64_t s0) {
#pragma unroll
    for (int v = 0; v < XV; ++v) {
      const int idx = threadIdx.x + v * 256;
      const int tt = idx / (kCols / NV), jv = (idx % (kCols / NV)) * NV;
      const int64_t t = s0 + tt;
      xr[v] = (t < te && j0 + jv < a.d)   // d is a multiple of NV
                  ? *reinterpret_cast<const uint4 *>(x + t * a.d + j0 + jv)
                  : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int q = 0; q < DV; ++q) {
      const int idx = threadIdx.x + q * 256;
      const int tt = idx / CP, c = idx % CP;
      const int64_t t = s0 + tt;
      float v = 0.0f;
      if (idx < 32 * CP && t < te && c < C) v = c < E ? a.dl[t * E + c] : a.dz[t];
      dr[q] = v;
    }
  };
  fetch(tb);
  float acc[RPT][8];
#pragma unroll
  for (int r = 0; r < RPT; ++r)
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[r][k] = 0.0f;
  for (int64_t s0 = tb; s0 < te; s0 += 32) {
    __syncthreads();   // the previous slab is consumed
#pragma unroll
    for (int v = 0; v < XV; ++v) {
      const int idx = threadIdx.x + v * 256;
      const int tt = idx / (kCols / NV), jv = (idx % (kCols / NV)) * NV;
      float f[NV];
      const T *src = reinterpret_cast<const T *>(&xr[v]);
#pragma unroll
      for (int q = 0; q < NV; ++q) f[q] = to_f32(src[q]);
#pragma unroll
      for (int q = 0; q < NV; q += 4)
        *reinterpret_cast<float4 *>(&xs[tt][jv + q]) = make_float4(f[q], f[q + 1], f[q + 2], f[q + 3]);
    }
#pragma unroll
    for (int q = 0; q < DV; ++q) {
      const int idx = threadIdx.x + q * 256;
      if (idx < 32 * CP) dls[idx / CP][idx % CP] = dr[q];
    }
    __syncthreads();
    if (s0 + 32 < te) fetch(s0 + 32);   // in flight while this slab is summed
    const int n = (int)min((int64_t)32, te - s0);
    for (int tt = 0; tt < n; ++tt) {
      const float4 x0 = *reinterpret_cast<const float4 *>(&xs[tt][jo * 8]);
      const float4 x1 = *reinterpret_cast<const float4 *>(&xs[tt][jo * 8 + 4]);
      const float x8[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int r = 0; r < RPT; ++r) {
        const float dv = dls[tt][rg * RPT + r];
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[r][k] = fmaf(dv, x8[k], acc[r][k]);
      }
    }
  }
  const int j = j0 + jo * 8;
  if (j >= a.d) return;
  float *part = a.partial + (int64_t)blockIdx.x * C * a.d;
#pragma unroll
  for (int r = 0; r < RPT; ++r) {
    const int c = rg * RPT + r;
    if (c < C) {
      float *dst = part + (int64_t)c * a.d + j;
      if (j + 8 <= a.d) {
        *reinterpret_cast<float4 *>(dst) = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
        *reinterpret_cast<float4 *>(dst + 4) = make_float4(acc[r][4], acc[r][5], acc[r][6], acc[r][7]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (j + k < a.d) dst[k] = acc[r][k];
      }
    }
  }
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

// ---------------------------------------------------------------------------
// Tensor-core path (bf16 layers, d % 256 == 0). dl (fp32) is split exactly
// enough into three bf16 planes: p1 = bf16(v), p2 = bf16(v - p1),
// p3 = bf16(v - p1 - p2), so p1 + p2 + p3 equals v up to about 2^-24 |v|;
// products of planes and bf16 weights or tokens are exact in the fp32
// accumulators, so the GEMMs give the fp32 sums up to accumulation order.

__global__ void __launch_bounds__(256) dl_planes_kernel(RouteBwdArgs a, __nv_bfloat16 *P, int PW,
                                                        int32_t *offs, int nsplit) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i <= nsplit) offs[i] = (int32_t)(a.T * i / nsplit);   // token chunks of the dW_r GEMM
  if (i < 2) offs[32 + i] = i == 0 ? 0 : (int32_t)a.T;      // the dx GEMM's single group
  if (i >= a.T * PW) return;
  const int64_t t = i / PW;
  const int c = (int)(i - t * PW);
  const int E = a.E;
  float v = 0.0f;
  if (c < E) v = a.dl[t * E + c];
  else if (c == E && a.dz != nullptr) v = a.dz[t];
  const __nv_bfloat16 p1 = __float2bfloat16_rn(v);
  const float r1 = __fsub_rn(v, __bfloat162float(p1));
  const __nv_bfloat16 p2 = __float2bfloat16_rn(r1);
  const float r2 = __fsub_rn(r1, __bfloat162float(p2));
  const __nv_bfloat16 p3 = __float2bfloat16_rn(r2);
  __nv_bfloat16 *row = P + t * 4 * PW;
  row[c] = p1;
  row[PW + c] = p2;
  row[2 * PW + c] = p3;
  row[3 * PW + c] = __float2bfloat16_rn(0.0f);
}

// Wr3[k * PW + c] = W_r[c] (c < E), w_sg (c == E), 0 otherwise, k = 0, 1, 2.
__global__ void __launch_bounds__(256) wr3_kernel(RouteBwdArgs a, __nv_bfloat16 *Wr3, int PW) {
  const int64_t nvec = (int64_t)3 * PW * a.d / 8;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nvec) return;
  const int64_t row = i * 8 / a.d;
  const int j = (int)(i * 8 - row * a.d);
  const int c = (int)(row % PW);
  uint4 v = make_uint4(0, 0, 0, 0);
  const __nv_bfloat16 *W = reinterpret_cast<const __nv_bfloat16 *>(a.W_r);
  const __nv_bfloat16 *wsg = reinterpret_cast<const __nv_bfloat16 *>(a.w_sg);
  if (c < a.E) v = *reinterpret_cast<const uint4 *>(W + (int64_t)c * a.d + j);
  else if (c == a.E && wsg != nullptr) v = *reinterpret_cast<const uint4 *>(wsg + j);
  *reinterpret_cast<uint4 *>(Wr3 + row * a.d + j) = v;
}

// dW_r[e] = sum over token chunks g, in order, of
// (out[g][e] + out[g][PW + e]) + out[g][2 PW + e]; dw_sg from row E.
__global__ void __launch_bounds__(256) plane_sum_kernel(RouteBwdArgs a, const float *out, int PW,
                                                        int nsplit) {
  const int C = a.E + (a.w_sg != nullptr ? 1 : 0);
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)C * a.d) return;
  const int c = (int)(i / a.d), j = (int)(i - (int64_t)c * a.d);
  float v = 0.0f;
  for (int g = 0; g < nsplit; ++g) {
    const float *o = out + (int64_t)g * 4 * PW * a.d;
    v = __fadd_rn(v, __fadd_rn(__fadd_rn(o[(int64_t)c * a.d + j], o[(int64_t)(PW + c) * a.d + j]),
                               o[(int64_t)(2 * PW + c) * a.d + j]));
  }
  if (c < a.E) a.dW_r[i] = v;
  else a.dw_sg[j] = v;
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

constexpr size_t align256_(size_t v) { return (v + 255) & ~size_t(255); }

// Plane width of the tensor-core path: the C = E (+1 with the shared-expert
// gate) dl columns padded to a multiple of 64 (one 64-deep K block of the dx
// GEMM per plane).
int tc_plane_width(int C) { return C <= 64 ? 64 : 128; }

struct TcLayout {
  size_t planes, wr3, out, offs, maps, total;
};
// The dW_r GEMM reduces over the T tokens; one group would give few, very
// long tiles, so the tokens are cut into up to kMaxSplit chunks (groups of
// the weight-gradient GEMM) and plane_sum_kernel adds the chunks in order.
constexpr int kMaxSplit = 16;

TcLayout tc_layout(int64_t T, int d, int PW) {
  TcLayout L{};
  size_t off = 0;
  L.planes = off; off += align256_((size_t)T * 4 * PW * 2);
  L.wr3 = off;    off += align256_((size_t)3 * PW * d * 2);
  L.out = off;    off += align256_((size_t)kMaxSplit * 4 * PW * d * 4);
  L.offs = off;   off += 256;
  L.maps = off;   off += align256_((size_t)2 * kMaxSplit * 128);   // tensor maps
  L.total = off + 256;          // room to align the region's start to 256 bytes
  return L;
}

size_t route_bwd_workspace_bytes(int64_t T, int d, int E) {
  const size_t dl = align256_((size_t)T * E * sizeof(float));
  const size_t cuda_path = (size_t)kChunks * (E + 1) * d * sizeof(float);
  const size_t tc_path = tc_layout(T, d, tc_plane_width(E + 1)).total;   // the widest planes
  return dl + (cuda_path > tc_path ? cuda_path : tc_path);
}

template <typename T, int CP>
void launch_dx_t(const RouteBwdArgs &a, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int ttiles = (int)((a.T + kDxT - 1) / kDxT), jtiles = (a.d + kDxJ - 1) / kDxJ;
  int ysplit = (2 * (sms > 0 ? sms : 148) + ttiles - 1) / ttiles;
  ysplit = ysplit < 1 ? 1 : (ysplit > jtiles ? jtiles : ysplit);
  const int nsub = (jtiles + ysplit - 1) / ysplit;
  dim3 gdx((unsigned)ttiles, (unsigned)((jtiles + nsub - 1) / nsub));
  auto k = dx_kernel<T, CP>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dx_smem_bytes<CP>());
  k<<<gdx, 256, dx_smem_bytes<CP>(), s>>>(a, nsub);
}

template <int CP>
void launch_dx(const RouteBwdArgs &a, cudaStream_t s) {
  if (a.dtype == MOE_BF16) launch_dx_t<__nv_bfloat16, CP>(a, s);
  else launch_dx_t<float, CP>(a, s);
}

template <typename T, int CP>
void launch_cp_t(const RouteBwdArgs &a, cudaStream_t s, int64_t chunk, int nchunk) {
  // enough CTAs for two per SM; each takes nsub of the ceil(d / 64) column tiles
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int ttiles = (int)((a.T + kDxT - 1) / kDxT), jtiles = (a.d + kDxJ - 1) / kDxJ;
  int ysplit = (2 * (sms > 0 ? sms : 148) + ttiles - 1) / ttiles;
  ysplit = ysplit < 1 ? 1 : (ysplit > jtiles ? jtiles : ysplit);
  const int nsub = (jtiles + ysplit - 1) / ysplit;
  dim3 gdx((unsigned)ttiles, (unsigned)((jtiles + nsub - 1) / nsub));
  dim3 gw((unsigned)nchunk, (unsigned)((a.d + kCols - 1) / kCols));
  auto k = dx_kernel<T, CP>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dx_smem_bytes<CP>());
  k<<<gdx, 256, dx_smem_bytes<CP>(), s>>>(a, nsub);
  wgrad_partial_kernel<T, CP><<<gw, 256, 0, s>>>(a, chunk);
}

template <int CP>
void launch_cp(const RouteBwdArgs &a, cudaStream_t s, int64_t chunk, int nchunk) {
  if (a.dtype == MOE_BF16) launch_cp_t<__nv_bfloat16, CP>(a, s, chunk, nchunk);
  else launch_cp_t<float, CP>(a, s, chunk, nchunk);
}

cudaError_t launch_route_bwd(const RouteBwdArgs &a, cudaStream_t s) {
  dl_kernel<<<(unsigned)((a.T * 32 + 255) / 256), 256, 0, s>>>(a);
  if (a.dtype == MOE_BF16 && a.d % 256 == 0 && a.T < (int64_t(1) << 31) / 512) {
    // tensor cores: dl planes, then the two GEMMs (dx on the CUDA cores when
    // a dx_in has to be added, which the GEMM epilogue does not do)
    const int PW = tc_plane_width(a.E + (a.w_sg != nullptr ? 1 : 0));
    const TcLayout L = tc_layout(a.T, a.d, PW);
    // the region the CUDA path uses for partials, its start aligned to 256 bytes
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(a.partial) + 255) & ~uintptr_t(255));
    RouterBwdTc r{};
    r.T = a.T; r.d = a.d; r.PW = PW; r.x = a.x; r.status = a.status;
    __nv_bfloat16 *P = reinterpret_cast<__nv_bfloat16 *>(base + L.planes);
    __nv_bfloat16 *Wr3 = reinterpret_cast<__nv_bfloat16 *>(base + L.wr3);
    int32_t *offs = reinterpret_cast<int32_t *>(base + L.offs);
    r.planes = P; r.Wr3 = Wr3; r.offs = offs; r.maps = base + L.maps;
    r.out_w = reinterpret_cast<float *>(base + L.out);
    r.dx_router = a.dx_in == nullptr ? a.dx_router : nullptr;
    // token chunks: about one pair tile per cluster (4 PW / 256 M tiles x d / 256 N tiles each)
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int tiles = (4 * PW / 256) * (a.d / 256);
    int nsplit = ((sms > 0 ? sms : 148) + tiles - 1) / tiles;
    nsplit = nsplit < 1 ? 1 : (nsplit > kMaxSplit ? kMaxSplit : nsplit);
    if (a.T < (int64_t)nsplit * 64) nsplit = 1;
    r.nsplit = nsplit;
    const int64_t np = a.T * PW;
    dl_planes_kernel<<<(unsigned)((np + 255) / 256), 256, 0, s>>>(a, P, PW, offs, nsplit);
    if (r.dx_router != nullptr) {
      const int64_t nv = (int64_t)3 * PW * a.d / 8;
      wr3_kernel<<<(unsigned)((nv + 255) / 256), 256, 0, s>>>(a, Wr3, PW);
    } else {   // CUDA-core dx with the dx_in addend
      const int C = a.E + (a.w_sg != nullptr ? 1 : 0);
      if (C <= 8) launch_dx<8>(a, s);
      else if (C <= 16) launch_dx<16>(a, s);
      else if (C <= 32) launch_dx<32>(a, s);
      else if (C <= 64) launch_dx<64>(a, s);
      else launch_dx<72>(a, s);
    }
    cudaError_t e = launch_router_bwd_tc(r, s);
    if (e != cudaSuccess) return e;
    const int C = a.E + (a.w_sg != nullptr ? 1 : 0);
    const int64_t n = (int64_t)C * a.d;
    plane_sum_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a, r.out_w, PW, nsplit);
    if (a.db_r != nullptr) db_kernel<<<a.E, 1024, 0, s>>>(a);
    return cudaGetLastError();
  }
  const int64_t chunk = (a.T + kChunks - 1) / kChunks;
  const int nchunk = (int)((a.T + chunk - 1) / chunk);
  const int C = a.E + (a.w_sg != nullptr ? 1 : 0);
  if (C <= 8) launch_cp<8>(a, s, chunk, nchunk);
  else if (C <= 16) launch_cp<16>(a, s, chunk, nchunk);
  else if (C <= 32) launch_cp<32>(a, s, chunk, nchunk);
  else if (C <= 64) launch_cp<64>(a, s, chunk, nchunk);
  else launch_cp<72>(a, s, chunk, nchunk);
  const int64_t n = (int64_t)C * a.d;
  reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a, nchunk);
  if (a.db_r != nullptr) db_kernel<<<a.E, 1024, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
