// Router: logits GEMV, softmax, Top-K, combine weights; capacity dropping.
//
// MoE Parallel Folding (arXiv 2504.14960) study notes: "method overview" (the
// router assigns each token its Top-K experts), "prerequisites" (Top-K gating,
// capacity factor), "key modules" and the quoted section 3.3 (drops are
// decided inside each sub-sequence; sub-sequence dropping is the default).
//
// bf16 layers compute the logits (and the shared-expert gate logit) on the
// tensor cores (router mode of the grouped GEMM, gemm_tc.cu; with a split K
// loop when T / 128 row tiles would leave SMs idle) and then run
// topk_from_logits_kernel, which also adds the split partial sums and the
// bias; fp32 layers use router_fused_kernel, which does the logits GEMV,
// softmax and Top-K in one pass. capacity_kernel applies the drop rule per
// (sub-sequence, expert). The softmax and Top-K arithmetic is
// specified in softmax.cuh.
#include "common.cuh"
#include "softmax.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------------------
// Fused router: one warp per token; the CTA stages a chunk of W_r (and w_sg)
// in shared memory as fp32 and every warp reuses it for its token.
constexpr int kRouteWarps = 8;
constexpr int kRouteChunk = 256;  // hidden elements per stage

template <typename T>
__global__ void __launch_bounds__(kRouteWarps * 32)
router_fused_kernel(RouteArgs a) {
  extern __shared__ float wsm[];  // [C][kRouteChunk], C = E (+1 for w_sg)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int E = a.E;
  const int C = E + (a.w_sg != nullptr ? 1 : 0);
  const int64_t t = (int64_t)blockIdx.x * kRouteWarps + warp;
  const bool active = t < a.T;
  const T *x = reinterpret_cast<const T *>(a.x);
  const T *W = reinterpret_cast<const T *>(a.W_r);
  const T *wsg = reinterpret_cast<const T *>(a.w_sg);

  float acc[65];
#pragma unroll
  for (int c = 0; c < 65; ++c) acc[c] = 0.0f;

  for (int j0 = 0; j0 < a.d; j0 += kRouteChunk) {
    const int n = min(kRouteChunk, a.d - j0);
    __syncthreads();
    for (int i = threadIdx.x; i < C * kRouteChunk; i += blockDim.x) {
      const int c = i / kRouteChunk, j = i % kRouteChunk;
      float v = 0.0f;
      if (j < n) v = to_f32(c < E ? W[(int64_t)c * a.d + j0 + j] : wsg[j0 + j]);
      wsm[i] = v;
    }
    __syncthreads();
    if (active) {
      // lane owns hidden elements j = lane + 32*i of this chunk
      float xv[kRouteChunk / 32];
#pragma unroll
      for (int i = 0; i < kRouteChunk / 32; ++i) {
        const int j = lane + 32 * i;
        xv[i] = j < n ? to_f32(x[t * a.d + j0 + j]) : 0.0f;
      }
#pragma unroll
      for (int c = 0; c < 65; ++c) {
        if (c < C) {
          float part = 0.0f;
#pragma unroll
          for (int i = 0; i < kRouteChunk / 32; ++i)
            part = fmaf(xv[i], wsm[c * kRouteChunk + lane + 32 * i], part);
          acc[c] += part;
        }
      }
    }
  }
  if (!active) return;
  // fixed-order butterfly reduction of each column over the lanes
#pragma unroll
  for (int c = 0; c < 65; ++c) {
    if (c < C) acc[c] = warp_sum(acc[c]);
  }
  float l0 = 0.0f, l1 = 0.0f;
#pragma unroll
  for (int c = 0; c < 64; ++c) {
    if (c == lane) l0 = acc[c];
    if (c == lane + 32) l1 = acc[c];
  }
  if (a.b_r != nullptr) {
    if (lane < E) l0 = __fadd_rn(l0, a.b_r[lane]);
    if (lane + 32 < E) l1 = __fadd_rn(l1, a.b_r[lane + 32]);
  }
  if (lane < E) a.logits[t * E + lane] = l0;
  if (lane + 32 < E) a.logits[t * E + lane + 32] = l1;
  if (a.w_sg != nullptr && lane == 0) {
    float z = 0.0f;
#pragma unroll
    for (int c = 0; c < 65; ++c)
      if (c == E) z = acc[c];
    a.gate_logit[t] = z;
  }
  spec::softmax_topk_warp(l0, l1, E, a.K, a.renorm, a.topk_idx + t * a.K, a.topk_prob + t * a.K,
                    a.topk_w + t * a.K, a.keep + t * a.K);
}

__global__ void __launch_bounds__(256) topk_from_logits_kernel(RouteArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= a.T) return;
  float l0, l1;
  if (a.rt_split > 1) {
    // the router GEMM's K-split partial sums, added in split order, then the
    // bias; the logits (and the gate logit) are written here
    const int has_gate = a.gate_logit != nullptr ? 1 : 0;
    const int C = a.E + has_gate;
    float s0 = 0.0f, s1 = 0.0f, sg = 0.0f;
    for (int k = 0; k < a.rt_split; ++k) {
      const float *P = a.rt_part + ((int64_t)k * a.T + t) * C;
      const float v0 = lane < a.E ? P[lane] : 0.0f;
      const float v1 = lane + 32 < a.E ? P[lane + 32] : 0.0f;
      const float vg = (has_gate && lane == 0) ? P[a.E] : 0.0f;
      s0 = k == 0 ? v0 : __fadd_rn(s0, v0);
      s1 = k == 0 ? v1 : __fadd_rn(s1, v1);
      sg = k == 0 ? vg : __fadd_rn(sg, vg);
    }
    if (a.b_r != nullptr) {
      if (lane < a.E) s0 = __fadd_rn(s0, a.b_r[lane]);
      if (lane + 32 < a.E) s1 = __fadd_rn(s1, a.b_r[lane + 32]);
    }
    float *l = a.logits + t * a.E;
    if (lane < a.E) l[lane] = s0;
    if (lane + 32 < a.E) l[lane + 32] = s1;
    if (has_gate && lane == 0) a.gate_logit[t] = sg;
    l0 = lane < a.E ? s0 : 0.0f;
    l1 = lane + 32 < a.E ? s1 : 0.0f;
  } else {
    const float *l = a.logits + t * a.E;
    l0 = lane < a.E ? l[lane] : 0.0f;
    l1 = lane + 32 < a.E ? l[lane + 32] : 0.0f;
  }
  spec::softmax_topk_warp(l0, l1, a.E, a.K, a.renorm, a.topk_idx + t * a.K, a.topk_prob + t * a.K,
                    a.topk_w + t * a.K, a.keep + t * a.K);
}

// ---------------------------------------------------------------------------
// Capacity dropping: one CTA per (sub-sequence j, expert e). Candidates are
// the assignments (t, k) of the sub-sequence routed to e, keyed by
// (fp32 bits of p) << 32 | (2^32 - 1 - t): a larger key is a higher
// probability, then a lower token index. Keys are unique, so the cap largest
// are found exactly by an MSB radix select (8-bit digits) of the cap-th
// largest key. The select stops at the first digit whose bin is kept whole:
// the threshold is then that bin's prefix with zero low bits, which every key
// of the bin reaches and no key of a lower bin does.
constexpr int kCapThreads = 512;
constexpr int kCapSmemKeys = 16384;   // candidates kept in shared memory (128 KB)

__global__ void __launch_bounds__(kCapThreads)
capacity_kernel(RouteArgs a, int cap_full, int cap_last, int keys_in_smem) {
  extern __shared__ unsigned long long skeys[];
  __shared__ uint32_t n_cand;
  __shared__ uint32_t hist[256];
  __shared__ unsigned long long sh_prefix;
  __shared__ uint32_t sh_need;
  __shared__ int sh_done;
  const int j = blockIdx.x, e = blockIdx.y;
  const int64_t lo = (int64_t)j * a.S;
  const int64_t hi = min(a.T, lo + a.S);
  const int cap = (hi - lo == a.S) ? cap_full : cap_last;
  unsigned long long *keys =
      keys_in_smem ? skeys : a.cap_keys + ((int64_t)j * a.E + e) * a.S;
  const int K = a.K;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) n_cand = 0;
  __syncthreads();
  // candidates: one shared-memory atomic per warp and slot
  const uint32_t lanes_below = (1u << lane) - 1u;
  for (int64_t t0 = lo; t0 < hi; t0 += blockDim.x) {
    const int64_t t = t0 + threadIdx.x;
    for (int k = 0; k < K; ++k) {
      const bool m = t < hi && a.topk_idx[t * K + k] == e;
      const uint32_t ballot = __ballot_sync(0xffffffffu, m);
      if (ballot == 0u) continue;
      uint32_t base = 0;
      if (lane == 0) base = atomicAdd(&n_cand, (uint32_t)__popc(ballot));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (m) {
        const uint32_t pbits = __float_as_uint(a.topk_prob[t * K + k]);
        keys[base + __popc(ballot & lanes_below)] =
            ((unsigned long long)pbits << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)t);
      }
    }
  }
  __syncthreads();
  const uint32_t n = n_cand;
  unsigned long long threshold = 0;
  if (n > (uint32_t)cap) {
    if (threadIdx.x == 0) { sh_prefix = 0; sh_need = (uint32_t)cap; sh_done = 0; }
    for (int shift = 56; shift >= 0; shift -= 8) {
      for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0;
      __syncthreads();
      const unsigned long long hmask = (shift == 56) ? 0ull : (~0ull << (shift + 8));
      const unsigned long long pre = sh_prefix;
      for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) {
        const unsigned long long key = keys[i];
        if ((key & hmask) == (pre & hmask)) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // digit holding the need-th largest key: lane l owns bins 255-8l down
        // to 248-8l; an inclusive scan over lanes counts the keys above
        uint32_t c[8], sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          c[i] = hist[255 - 8 * lane - i];
          sum += c[i];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        const uint32_t excl = incl - sum;
        const uint32_t need = sh_need;
        const uint32_t hit = __ballot_sync(0xffffffffu, excl < need && need <= incl);
        if (lane == __ffs(hit) - 1) {
          uint32_t cum = excl, cnt = 0;
          int digit = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (cum + c[i] >= need) { digit = 255 - 8 * lane - i; cnt = c[i]; break; }
            cum += c[i];
          }
          sh_need = need - cum;
          sh_prefix = pre | ((unsigned long long)digit << shift);
          sh_done = (need - cum == cnt) ? 1 : 0;   // the digit's whole bin is kept
        }
      }
      __syncthreads();
      if (sh_done) break;
    }
    threshold = sh_prefix;
  }
  for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) {
    const unsigned long long key = keys[i];
    const int64_t t = (int64_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
    for (int k = 0; k < K; ++k) {
      if (a.topk_idx[t * K + k] == e) a.keep[t * K + k] = key >= threshold ? 1 : 0;
    }
  }
}

int capacity_of(float cf, int64_t S_j, int K, int E) {
  // ceil(CF * S_j * K / E) in double, left to right
  double v = (double)cf * (double)S_j * (double)K / (double)E;
  return (int)ceil(v);
}

}  // namespace

cudaError_t launch_router_fused(const RouteArgs &a, cudaStream_t s) {
  const int C = a.E + (a.w_sg != nullptr ? 1 : 0);
  const size_t smem = (size_t)C * kRouteChunk * sizeof(float);
  const unsigned grid = (unsigned)((a.T + kRouteWarps - 1) / kRouteWarps);
  if (a.dtype == MOE_BF16) {
    auto k = router_fused_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<grid, kRouteWarps * 32, smem, s>>>(a);
  } else {
    auto k = router_fused_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<grid, kRouteWarps * 32, smem, s>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_topk_from_logits(const RouteArgs &a, cudaStream_t s) {
  const unsigned grid = (unsigned)((a.T * 32 + 255) / 256);
  topk_from_logits_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

int64_t padded_rows_per_expert(int64_t T, int64_t S, int K, int E, float cf) {
  int64_t rows = 0;
  for (int64_t lo = 0; lo < T; lo += S) {
    const int64_t len = T - lo < S ? T - lo : S;
    const int64_t cap = capacity_of(cf, len, K, E);
    rows += cap < len ? cap : len;
  }
  return rows;
}

cudaError_t launch_capacity(const RouteArgs &a, cudaStream_t s) {
  const int64_t n_sub = (a.T + a.S - 1) / a.S;
  const int64_t last = a.T - (n_sub - 1) * a.S;
  const int cap_full = capacity_of(a.cf, a.S, a.K, a.E);
  const int cap_last = capacity_of(a.cf, last, a.K, a.E);
  dim3 grid((unsigned)n_sub, (unsigned)a.E);
  const int in_smem = a.S <= kCapSmemKeys ? 1 : 0;
  const size_t smem = in_smem ? (size_t)a.S * sizeof(unsigned long long) : 0;
  cudaError_t e = cudaFuncSetAttribute(capacity_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  capacity_kernel<<<grid, kCapThreads, smem, s>>>(a, cap_full, cap_last, in_smem);
  return cudaGetLastError();
}

}  // namespace moe
