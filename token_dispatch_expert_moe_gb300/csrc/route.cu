// Router: logits GEMV, softmax, Top-K, combine weights; capacity dropping.
//
// MoE Parallel Folding (arXiv 2504.14960) study notes: "method overview" (the
// router assigns each token its Top-K experts), "prerequisites" (Top-K gating,
// capacity factor), "key modules" and the quoted section 3.3 (drops are
// decided inside each sub-sequence; sub-sequence dropping is the default).
//
// bf16 layers compute the logits (and the shared-expert gate logit) on the
// tensor cores (router mode of the grouped GEMM, gemm_tc.cu, which adds the
// bias; its K loop split over a cluster of CTAs when T / 128 row tiles would
// leave SMs idle). With E <= 16 and no split that kernel's epilogue also
// routes; otherwise topk_from_logits_kernel does, a warp per token. fp32
// layers use router_fused_kernel, which does the logits GEMV, softmax and
// Top-K in one pass. capacity_bucket_kernel and capacity_select_kernel apply
// the drop rule per (sub-sequence, expert). The softmax and Top-K arithmetic
// is specified in softmax.cuh.
#include "common.cuh"
#include "softmax.cuh"

namespace moe {
namespace {

// Programmatic dependent launch: the Top-K and capacity kernels are launched
// while their predecessor still runs and wait here, before reading anything
// it wrote, until it has completed and its writes are visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

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
  pdl_wait();   // the logits (or their split partial sums) come from the router GEMM
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= a.T) return;
  const float *l = a.logits + t * a.E;
  const float l0 = lane < a.E ? l[lane] : 0.0f;
  const float l1 = lane + 32 < a.E ? l[lane + 32] : 0.0f;
  spec::softmax_topk_warp(l0, l1, a.E, a.K, a.renorm, a.topk_idx + t * a.K, a.topk_prob + t * a.K,
                    a.topk_w + t * a.K, a.keep + t * a.K);
}

// ---------------------------------------------------------------------------
// Capacity dropping, in two passes over the Top-K slots.
//   bucket: one thread per slot (t, k) appends the slot's key to the list of
//     its (sub-sequence j, expert e) in the workspace (warp-aggregated
//     atomics on the per-list counters, which the call zeroes first);
//   select: one CTA per (j, e) whose list holds more than cap keys finds the
//     cap-th largest key and clears keep for the keys below it (the Top-K
//     step has set every keep to 1).
// Key of a slot: (fp32 bits of p) << 32 | (2^32 - 1 - (t' * 8 + k)),
// t' = t - (first token of the sub-sequence): a larger key is a higher
// probability, then a lower token index (an expert takes at most one slot of
// a token, so k never decides). Keys are unique, so the cap largest are found
// exactly by an MSB radix select (8-bit digits) of the cap-th largest key.
// The select stops at the first digit whose bin is kept whole: the threshold
// is then that bin's prefix with zero low bits, which every key of the bin
// reaches and no key of a lower bin does. The order of a list does not
// matter, so the appends need no ordering.
constexpr int kBucketThreads = 256;
constexpr int kCapThreads = 512;
constexpr int kCapSmemKeys = 16384;   // candidates kept in shared memory (128 KB)
constexpr int64_t kCapMaxSubseq = int64_t(1) << 29;   // t' * 8 + k fits in 32 bits

// A bucket CTA takes the slots of `tpc` consecutive tokens (tpc <= S, so at
// most two sub-sequences), kBucketRounds per thread, coalesced. It counts its
// keys per list in shared memory (a place inside its share of each list),
// reserves its share of each list with one global atomic, then writes. Two
// rounds (512 slots per CTA) keep the grid at 64 CTAs or more on the
// Mixtral-8x22B shape (16384 slots).
constexpr int kBucketRounds = 2;

__global__ void __launch_bounds__(kBucketThreads)
capacity_bucket_kernel(RouteArgs a, uint32_t *counts, int tpc) {
  __shared__ uint32_t lcnt[2][64], lbase[2][64];
  pdl_wait();   // topk_idx and topk_prob come from the Top-K step
  pdl_trigger();
  const int K = a.K, E = a.E;
  const int64_t t0 = (int64_t)blockIdx.x * tpc;
  const int64_t s0 = t0 * K, s1 = min(a.T, t0 + tpc) * K;   // this CTA's slots
  const int64_t j0 = t0 / a.S;
  for (int i = threadIdx.x; i < 2 * 64; i += blockDim.x) (&lcnt[0][0])[i] = 0;
  __syncthreads();
  int sel[kBucketRounds];           // list within the CTA (jj * 64 + e), -1 if none
  uint32_t pos[kBucketRounds];      // place within the CTA's share of that list
  unsigned long long key[kBucketRounds];
#pragma unroll
  for (int r = 0; r < kBucketRounds; ++r) {
    const int64_t i = s0 + (int64_t)r * blockDim.x + threadIdx.x;
    sel[r] = -1;
    pos[r] = 0;
    key[r] = 0;
    if (i < s1) {
      const int64_t t = i / K;
      const int k = (int)(i - t * K);
      const int e = a.topk_idx[i];
      if (e >= 0 && e < E) {
        const int64_t j = t / a.S;
        const uint32_t slot = (uint32_t)((t - j * a.S) * 8 + k);
        key[r] = ((unsigned long long)__float_as_uint(a.topk_prob[i]) << 32) |
                 (unsigned long long)(0xFFFFFFFFu - slot);
        sel[r] = (int)(j - j0) * 64 + e;
        pos[r] = atomicAdd(&(&lcnt[0][0])[sel[r]], 1u);
      } else {
        report(a.status, MOE_ERR_DEVICE, kInfoExpertRange);
      }
    }
  }
  __syncthreads();
  for (int l = threadIdx.x; l < 2 * 64; l += blockDim.x) {
    const uint32_t c = (&lcnt[0][0])[l];
    if (c > 0) (&lbase[0][0])[l] = atomicAdd(&counts[(j0 + l / 64) * E + (l % 64)], c);
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kBucketRounds; ++r) {
    if (sel[r] >= 0) {
      const int64_t list = (j0 + sel[r] / 64) * E + (sel[r] % 64);
      a.cap_keys[list * a.S + (&lbase[0][0])[sel[r]] + pos[r]] = key[r];
    }
  }
}

__global__ void __launch_bounds__(kCapThreads)
capacity_select_kernel(RouteArgs a, const uint32_t *counts, int cap_full, int cap_last,
                       int keys_in_smem) {
  extern __shared__ unsigned long long skeys[];
  __shared__ uint32_t hist[256];
  __shared__ unsigned long long sh_prefix;
  __shared__ uint32_t sh_need;
  __shared__ int sh_done;
  pdl_wait();   // the lists come from the bucket pass
  const int j = blockIdx.x, e = blockIdx.y;
  const int64_t lo = (int64_t)j * a.S;
  const int64_t hi = min(a.T, lo + a.S);
  const int cap = (hi - lo == a.S) ? cap_full : cap_last;
  const int64_t list = (int64_t)j * a.E + e;
  const uint32_t n = counts[list];
  if (n <= (uint32_t)cap) return;   // every assignment of the list is kept
  const unsigned long long *gkeys = a.cap_keys + list * a.S;
  const unsigned long long *keys = gkeys;
  if (keys_in_smem) {
    for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) skeys[i] = gkeys[i];
    keys = skeys;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) { sh_prefix = 0; sh_need = (uint32_t)cap; sh_done = 0; }
  __syncthreads();
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
  const unsigned long long threshold = sh_prefix;
  const int K = a.K;
  for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) {
    const unsigned long long key = keys[i];
    if (key < threshold) {
      const uint32_t slot = 0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull);
      a.keep[(lo + (slot >> 3)) * K + (slot & 7u)] = 0;
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

// Launch with programmatic stream serialization (the kernels call
// griddepcontrol.wait before reading their predecessor's outputs).
template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern k, dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

cudaError_t launch_topk_from_logits(const RouteArgs &a, cudaStream_t s) {
  const unsigned grid = (unsigned)((a.T * 32 + 255) / 256);
  return launch_pdl(topk_from_logits_kernel, dim3(grid), dim3(256), 0, s, a);
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
  if (a.S >= kCapMaxSubseq || a.K < 1 || a.K > 8 || a.cap_counts == nullptr)
    return cudaErrorInvalidValue;
  const int64_t n_sub = (a.T + a.S - 1) / a.S;
  const int64_t last = a.T - (n_sub - 1) * a.S;
  const int cap_full = capacity_of(a.cf, a.S, a.K, a.E);
  const int cap_last = capacity_of(a.cf, last, a.K, a.E);
  // tokens per bucket CTA: its slots fill kBucketRounds rounds of the block,
  // and no more than one sub-sequence's worth (so at most two sub-sequences)
  int64_t tpc = kBucketRounds * kBucketThreads / a.K;
  if (tpc > a.S) tpc = a.S;
  cudaError_t e = launch_pdl(capacity_bucket_kernel, dim3((unsigned)((a.T + tpc - 1) / tpc)),
                             dim3(kBucketThreads), 0, s, a, a.cap_counts, (int)tpc);
  if (e != cudaSuccess) return e;
  const int in_smem = a.S <= kCapSmemKeys ? 1 : 0;
  const size_t smem = in_smem ? (size_t)a.S * sizeof(unsigned long long) : 0;
  e = cudaFuncSetAttribute(capacity_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(capacity_select_kernel, dim3((unsigned)n_sub, (unsigned)a.E),
                    dim3(kCapThreads), smem, s, a, (const uint32_t *)a.cap_counts, cap_full,
                    cap_last, in_smem);
}

}  // namespace moe
