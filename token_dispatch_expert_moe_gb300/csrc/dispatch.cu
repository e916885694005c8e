// Permutation map, permute, un-permute/combine and their backward kernels.
//
// MoE Parallel Folding (arXiv 2504.14960) study notes, "method overview": a
// permutation makes each expert's tokens contiguous before the expert FFN,
// and an un-permutation restores the token order afterwards; "key modules":
// the dispatcher copes with dynamic shapes. Here the per-expert counts and
// offsets never leave the device.
//
// Map build (deterministic, atomics only on counters whose final value does
// not depend on order):
//   1. map_count: tokens are cut into blocks of 256; each CTA sets one bit per
//      kept (token, expert) in a shared bitmap [E][8 words] and writes the
//      per-expert popcounts of its block;
//   2. map_scan: per expert, an exclusive scan over blocks; counts, offsets;
//   3. map_scatter: each CTA rebuilds its bitmap; the rank of token t among
//      the kept tokens of expert e in the block is the popcount of the bits
//      below t, so row_of[t,k] = base[block][e] + rank, and src_of[row] =
//      t*K + k. Rows come out expert-major and token-ascending.
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kMapBlock = 256;  // tokens per map CTA (8 words of 32 bits)

__global__ void __launch_bounds__(kMapBlock) map_count_kernel(PermuteArgs a) {
  extern __shared__ uint32_t bm[];  // [E][8]
  const int E = a.E, K = a.K;
  for (int i = threadIdx.x; i < E * 8; i += blockDim.x) bm[i] = 0;
  __syncthreads();
  const int64_t t = (int64_t)blockIdx.x * kMapBlock + threadIdx.x;
  if (t < a.T) {
    for (int k = 0; k < K; ++k) {
      if (a.keep[t * K + k]) {
        const int e = a.topk_idx[t * K + k];
        if (e < 0 || e >= E) {
          report(a.status, MOE_ERR_DEVICE, kInfoExpertRange);
          continue;
        }
        atomicOr(&bm[e * 8 + (threadIdx.x >> 5)], 1u << (threadIdx.x & 31));
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) c += __popc(bm[e * 8 + w]);
    a.blk_counts[(int64_t)blockIdx.x * E + e] = c;
  }
}

// One CTA: thread e scans expert e's block counts (in block order).
__global__ void map_scan_kernel(PermuteArgs a, int nblk) {
  __shared__ int tot[64];
  const int E = a.E;
  const int e = threadIdx.x;
  if (e < E) {
    int run = 0;
    for (int b = 0; b < nblk; ++b) {
      const int c = a.blk_counts[(int64_t)b * E + e];
      a.blk_counts[(int64_t)b * E + e] = run;  // exclusive prefix within expert
      run += c;
    }
    tot[e] = run;
    a.counts[e] = run;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int i = 0; i < E; ++i) {
      a.offsets[i] = acc;
      acc += tot[i];
    }
    a.offsets[E] = acc;
  }
  __syncthreads();
  if (e < E) {
    int base = 0;
    for (int i = 0; i < e; ++i) base += tot[i];
    for (int b = 0; b < nblk; ++b) a.blk_counts[(int64_t)b * E + e] += base;
  }
}

__global__ void __launch_bounds__(kMapBlock) map_scatter_kernel(PermuteArgs a) {
  extern __shared__ uint32_t bm[];  // [E][8]
  const int E = a.E, K = a.K;
  for (int i = threadIdx.x; i < E * 8; i += blockDim.x) bm[i] = 0;
  __syncthreads();
  const int64_t t = (int64_t)blockIdx.x * kMapBlock + threadIdx.x;
  const int wi = threadIdx.x >> 5;
  const uint32_t below = (1u << (threadIdx.x & 31)) - 1u;
  if (t < a.T) {
    for (int k = 0; k < K; ++k) {
      const int e = a.topk_idx[t * K + k];
      if (a.keep[t * K + k] && e >= 0 && e < E) atomicOr(&bm[e * 8 + wi], 1u << (threadIdx.x & 31));
    }
  }
  __syncthreads();
  if (t < a.T) {
    for (int k = 0; k < K; ++k) {
      const int e = a.topk_idx[t * K + k];
      int32_t row = -1;
      if (a.keep[t * K + k] && e >= 0 && e < E) {
        int rank = __popc(bm[e * 8 + wi] & below);
        for (int w = 0; w < wi; ++w) rank += __popc(bm[e * 8 + w]);
        row = a.blk_counts[(int64_t)blockIdx.x * E + e] + rank;
        a.src_of[row] = (int32_t)(t * K + k);
      }
      a.row_of[t * K + k] = row;
    }
  }
}

// Xp[row_of[t,k]] = x[t]: one CTA per token, 16-byte vectors; x is read
// once and written to each kept slot's row.
template <typename T>
__global__ void __launch_bounds__(256) permute_rows_kernel(PermuteArgs a) {
  const int64_t t = blockIdx.x;
  const int K = a.K;
  __shared__ int32_t rows[8];
  if (threadIdx.x < K) rows[threadIdx.x] = a.row_of[t * K + threadIdx.x];
  __syncthreads();
  const int nv = a.d / Vec<T>::N;
  const uint4 *src = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(a.x) + t * a.d);
  uint4 *dst = reinterpret_cast<uint4 *>(a.Xp);
  const int64_t row_vecs = nv;
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    const uint4 val = src[v];
#pragma unroll 8
    for (int k = 0; k < K; ++k) {
      const int32_t r = rows[k];
      if (r >= 0) dst[(int64_t)r * row_vecs + v] = val;
    }
  }
}

// out[t] = sum_k w[t,k] Yp[row_of[t,k]] (+ sigmoid(z_t) Ys[t]), fp32 sum in
// slot order, one rounding to T.
template <typename T>
__global__ void __launch_bounds__(256) unpermute_kernel(UnpermuteArgs a) {
  constexpr int N = Vec<T>::N;
  const int64_t t = blockIdx.x;
  const int K = a.K;
  __shared__ int32_t rows[8];
  __shared__ float wts[8];
  __shared__ float gate;
  if (threadIdx.x < K) {
    rows[threadIdx.x] = a.row_of[t * K + threadIdx.x];
    wts[threadIdx.x] = a.topk_w[t * K + threadIdx.x];
  }
  if (threadIdx.x == 0 && a.Ys != nullptr) gate = 1.0f / (1.0f + __expf(-a.gate_logit[t]));
  __syncthreads();
  const T *Yp = reinterpret_cast<const T *>(a.Yp);
  const T *Ys = reinterpret_cast<const T *>(a.Ys);
  T *out = reinterpret_cast<T *>(a.out);
  for (int v = threadIdx.x * N; v < a.d; v += blockDim.x * N) {
    float acc[N];
#pragma unroll
    for (int i = 0; i < N; ++i) acc[i] = 0.0f;
    for (int k = 0; k < K; ++k) {
      const int32_t r = rows[k];
      if (r < 0) continue;
      float y[N];
      load16<T>(Yp + (int64_t)r * a.d + v, y);
      const float w = wts[k];
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = fmaf(w, y[i], acc[i]);
    }
    if (Ys != nullptr) {
      float y[N];
      load16<T>(Ys + t * a.d + v, y);
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = fmaf(gate, y[i], acc[i]);
    }
    store16<T>(out + t * a.d + v, acc);
  }
}

// dYp[row] = w * dout[t]; dw[t,k] = <dout[t], Yp[row]>; shared: dYs, dz.
template <typename T>
__global__ void __launch_bounds__(256) unpermute_bwd_kernel(UnpermuteArgs a) {
  constexpr int N = Vec<T>::N;
  const int64_t t = blockIdx.x;
  const int K = a.K;
  __shared__ int32_t rows[8];
  __shared__ float wts[8];
  __shared__ float gate;
  __shared__ float red[32];
  if (threadIdx.x < K) {
    rows[threadIdx.x] = a.row_of[t * K + threadIdx.x];
    wts[threadIdx.x] = a.topk_w[t * K + threadIdx.x];
  }
  if (threadIdx.x == 0 && a.Ys != nullptr) gate = 1.0f / (1.0f + __expf(-a.gate_logit[t]));
  __syncthreads();
  const T *Yp = reinterpret_cast<const T *>(a.Yp);
  const T *dout = reinterpret_cast<const T *>(a.dout);
  T *dYp = reinterpret_cast<T *>(a.dYp);
  float dot[9];
#pragma unroll
  for (int k = 0; k < 9; ++k) dot[k] = 0.0f;
  for (int v = threadIdx.x * N; v < a.d; v += blockDim.x * N) {
    float g[N];
    load16<T>(dout + t * a.d + v, g);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k >= K) break;
      const int32_t r = rows[k];
      if (r < 0) continue;
      float y[N], o[N];
      load16<T>(Yp + (int64_t)r * a.d + v, y);
      const float w = wts[k];
#pragma unroll
      for (int i = 0; i < N; ++i) {
        dot[k] = fmaf(g[i], y[i], dot[k]);
        o[i] = w * g[i];
      }
      store16<T>(dYp + (int64_t)r * a.d + v, o);
    }
    if (a.Ys != nullptr) {
      float y[N], o[N];
      load16<T>(reinterpret_cast<const T *>(a.Ys) + t * a.d + v, y);
#pragma unroll
      for (int i = 0; i < N; ++i) {
        dot[8] = fmaf(g[i], y[i], dot[8]);
        o[i] = gate * g[i];
      }
      store16<T>(reinterpret_cast<T *>(a.dYs) + t * a.d + v, o);
    }
  }
  for (int k = 0; k < K; ++k) {
    const float s = block_sum(dot[k], red);
    if (threadIdx.x == 0) a.dw[t * K + k] = rows[k] >= 0 ? s : 0.0f;
  }
  if (a.Ys != nullptr) {
    const float s = block_sum(dot[8], red);
    if (threadIdx.x == 0) a.dz[t] = gate * (1.0f - gate) * s;
  }
}

// dx[t] = sum_k dXp[row_of[t,k]] (+ dx_add[t]), fp32, slot order.
__global__ void __launch_bounds__(256)
permute_bwd_kernel(int64_t T, int d, int K, const float *__restrict__ dXp,
                   const int32_t *__restrict__ row_of, const float *__restrict__ dx_add,
                   float *__restrict__ dx) {
  const int64_t t = blockIdx.x;
  __shared__ int32_t rows[8];
  if (threadIdx.x < K) rows[threadIdx.x] = row_of[t * K + threadIdx.x];
  __syncthreads();
  for (int v = threadIdx.x * 4; v < d; v += blockDim.x * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < K; ++k) {
      const int32_t r = rows[k];
      if (r < 0) continue;
      const float4 y = *reinterpret_cast<const float4 *>(dXp + (int64_t)r * d + v);
      acc.x += y.x; acc.y += y.y; acc.z += y.z; acc.w += y.w;
    }
    if (dx_add != nullptr) {
      const float4 y = *reinterpret_cast<const float4 *>(dx_add + t * d + v);
      acc.x += y.x; acc.y += y.y; acc.z += y.z; acc.w += y.w;
    }
    *reinterpret_cast<float4 *>(dx + t * d + v) = acc;
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// Scratch for moe_permute_noalloc: the per-block expert counts of the map
// build live in this fixed device array instead of a caller workspace. It
// holds MOE_PERMUTE_NOALLOC_MAX_TOKENS / 256 blocks x 64 experts (128 KB) and
// stays resident on every GPU that loads the library until the process exits.
// map_count writes every word that map_scan and map_scatter later read, so a
// call never sees the previous call's counts and nothing needs clearing.
constexpr int kNoAllocBlocks = MOE_PERMUTE_NOALLOC_MAX_TOKENS / kMapBlock;
static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocBlocks * 64];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
int32_t *g_scratch_addr[kMaxDevices] = {};

// Device address of g_permute_scratch on the current device. In host code the
// array's name is only a handle, so the address is looked up once per device
// (cudaGetSymbolAddress, with that device current) and cached.
cudaError_t permute_scratch(int32_t **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<int32_t *>(p);
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_permute_noalloc(PermuteArgs a, cudaStream_t s) {
  if (a.T > MOE_PERMUTE_NOALLOC_MAX_TOKENS || a.E > 64) return cudaErrorInvalidValue;
  int32_t *scratch = nullptr;
  cudaError_t e = permute_scratch(&scratch);
  if (e != cudaSuccess) return e;
  a.blk_counts = scratch;
  a.status = nullptr;  // no workspace, so no status word
  return launch_permute(a, s);
}

cudaError_t launch_permute(const PermuteArgs &a, cudaStream_t s) {
  const int nblk = (int)((a.T + kMapBlock - 1) / kMapBlock);
  const size_t bm_bytes = (size_t)a.E * 8 * sizeof(uint32_t);
  map_count_kernel<<<nblk, kMapBlock, bm_bytes, s>>>(a);
  map_scan_kernel<<<1, 64, 0, s>>>(a, nblk);
  map_scatter_kernel<<<nblk, kMapBlock, bm_bytes, s>>>(a);
  if (a.dtype == MOE_BF16)
    permute_rows_kernel<__nv_bfloat16><<<(unsigned)a.T, 256, 0, s>>>(a);
  else
    permute_rows_kernel<float><<<(unsigned)a.T, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_unpermute(const UnpermuteArgs &a, cudaStream_t s) {
  if (a.dtype == MOE_BF16)
    unpermute_kernel<__nv_bfloat16><<<(unsigned)a.T, 256, 0, s>>>(a);
  else
    unpermute_kernel<float><<<(unsigned)a.T, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_unpermute_bwd(const UnpermuteArgs &a, cudaStream_t s) {
  if (a.dtype == MOE_BF16)
    unpermute_bwd_kernel<__nv_bfloat16><<<(unsigned)a.T, 256, 0, s>>>(a);
  else
    unpermute_bwd_kernel<float><<<(unsigned)a.T, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_permute_bwd(int64_t T, int d, int K, const float *dXp, const int32_t *row_of,
                               const float *dx_add, float *dx, cudaStream_t s) {
  permute_bwd_kernel<<<(unsigned)T, 256, 0, s>>>(T, d, K, dXp, row_of, dx_add, dx);
  return cudaGetLastError();
}

}  // namespace moe
