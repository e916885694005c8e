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
//   2. map_scatter: each CTA reads the per-block counts, forms the expert
//      totals and offsets (CTA 0 publishes counts and offsets) and its own
//      base per expert; it rebuilds its bitmap, and the rank of token t among
//      the kept tokens of expert e in the block is the popcount of the bits
//      below t, so row_of[t,k] = base[e] + rank, and src_of[row] = t*K + k.
//      Rows come out expert-major and token-ascending.
#include <mutex>

#include <cuda.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kMapBlock = 256;  // tokens per map CTA (8 words of 32 bits)

// Programmatic dependent launch: the map count, the map scatter and the row
// copy are launched while their predecessor still runs; each waits for it
// (and its memory) at griddepcontrol.wait before reading what it wrote. The
// map count waits before it reads topk_idx and keep (the router's last kernel
// may still be writing them) and lets its dependents launch only after that
// wait, so the later kernels may read x, topk_idx and keep before their own
// wait: whatever wrote those had completed when the map count passed its.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__global__ void __launch_bounds__(kMapBlock) map_count_kernel(PermuteArgs a) {
  extern __shared__ uint32_t bm[];  // [E][8]
  const int E = a.E, K = a.K;
  for (int i = threadIdx.x; i < E * 8; i += blockDim.x) bm[i] = 0;
  pdl_wait();   // topk_idx and keep may come from the router's last kernel
  pdl_trigger();   // after the wait: the later kernels read x before theirs
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

__global__ void __launch_bounds__(kMapBlock) map_scatter_kernel(PermuteArgs a, int nblk) {
  extern __shared__ uint32_t bm[];  // [E][8]
  __shared__ int tot_s[64], base_s[64];
  pdl_trigger();
  const int E = a.E, K = a.K;
  for (int i = threadIdx.x; i < E * 8; i += blockDim.x) bm[i] = 0;
  pdl_wait();   // blk_counts come from map_count
  // every CTA scans the (small) table of per-block counts itself: expert
  // totals, and the kept assignments of expert e in blocks before this one
  if (threadIdx.x < E) {
    const int e = threadIdx.x;
    int tot = 0, before = 0;
    for (int b = 0; b < nblk; ++b) {
      const int c = a.blk_counts[(int64_t)b * E + e];
      before += b < (int)blockIdx.x ? c : 0;
      tot += c;
    }
    tot_s[e] = tot;
    base_s[e] = before;
  }
  __syncthreads();
  if (threadIdx.x < E) {
    const int e = threadIdx.x;
    int off = 0;
    if (a.pad_rows > 0) {   // padded layout: fixed stride per expert
      off = (int)(e * a.pad_rows);
    } else {
      for (int i = 0; i < e; ++i) off += tot_s[i];
    }
    base_s[e] += off;
    if (blockIdx.x == 0) {
      a.counts[e] = tot_s[e];
      a.offsets[e] = off;
      if (e == E - 1) a.offsets[E] = a.pad_rows > 0 ? (int)(E * a.pad_rows) : off + tot_s[e];
    }
  }
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
        row = base_s[e] + rank;
        if (a.pad_rows > 0 && row - e * a.pad_rows >= a.pad_rows) {
          report(a.status, MOE_ERR_DEVICE, kInfoPadOverflow);
          row = -1;
        } else {
          a.src_of[row] = (int32_t)(t * K + k);
        }
      }
      a.row_of[t * K + k] = row;
    }
  }
}

// Xp[row_of[t,k]] = x[t] with the bulk-copy engine: a one-warp CTA loads up
// to 4 token rows (at most 96 KB) into shared memory (cp.async.bulk, one
// mbarrier), then writes each row to its kept slots' rows with bulk stores.
// x is read once; the SM issues a handful of instructions per row.
constexpr int kPermTokens = 4;
constexpr uint32_t kPermSmemCap = 96 * 1024;

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__global__ void __launch_bounds__(32) permute_bulk_kernel(PermuteArgs a, uint32_t row_bytes,
                                                          int tpc) {
  extern __shared__ __align__(128) uint8_t rows_smem[];
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const int64_t t0 = (int64_t)blockIdx.x * tpc;
  const int n = (int)min((int64_t)tpc, a.T - t0);
  const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
  const uint32_t sm = static_cast<uint32_t>(__cvta_generic_to_shared(rows_smem));
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b),
               "r"(row_bytes * (uint32_t)n)
               : "memory");
  const uint8_t *x = static_cast<const uint8_t *>(a.x);
  for (int i = 0; i < n; ++i)
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            sm + i * row_bytes),
        "l"(x + (t0 + i) * (int64_t)row_bytes), "r"(row_bytes), "r"(b)
        : "memory");
  pdl_wait();   // row_of comes from map_scatter
  // bounded wait for the rows to land
  uint32_t done = 0;
  const uint64_t start = now_ns();
  while (!done) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(done)
        : "r"(b)
        : "memory");
    if (!done && now_ns() - start > 2000000000ull) {
      report(a.status, MOE_ERR_TIMEOUT, kInfoRowRange);
      return;
    }
  }
  uint8_t *Xp = static_cast<uint8_t *>(a.Xp);
  for (int i = 0; i < n; ++i) {
    for (int k = 0; k < a.K; ++k) {
      const int32_t r = a.row_of[(t0 + i) * a.K + k];
      if (r >= 0)
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                         Xp + (int64_t)r * row_bytes),
                     "r"(sm + i * row_bytes), "r"(row_bytes)
                     : "memory");
    }
  }
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Padded layout: rows [e*pad + counts[e], (e+1)*pad) of every expert get zero
// activations and src_of = -1. One CTA per expert, 16-byte stores.
__global__ void __launch_bounds__(256) pad_fill_kernel(PermuteArgs a, int vec_per_row) {
  const int e = blockIdx.x;
  const int64_t lo = (int64_t)e * a.pad_rows + a.counts[e], hi = (int64_t)(e + 1) * a.pad_rows;
  uint4 *Xp = static_cast<uint4 *>(a.Xp);
  if (Xp != nullptr)
    for (int64_t i = lo * vec_per_row + threadIdx.x; i < hi * vec_per_row; i += blockDim.x)
      Xp[i] = make_uint4(0, 0, 0, 0);
  for (int64_t r = lo + threadIdx.x; r < hi; r += blockDim.x) a.src_of[r] = -1;
}

// out[t] = sum_k w[t,k] Yp[row_of[t,k]] (+ sigmoid(z_t) Ys[t]), fp32 sum in
// slot order, one rounding to T. KK >= K is a compile-time slot bound, so
// that per 16-byte column vector all K row loads (and the Ys load) are issued
// before the first use: K + 1 loads per thread in flight.
template <typename T, int KK, bool SHARED>
__global__ void __launch_bounds__(256) unpermute_kernel(UnpermuteArgs a) {
  constexpr int N = Vec<T>::N;
  const int64_t t = blockIdx.x;
  const int K = a.K;
  __shared__ int32_t rows[KK];
  __shared__ float wts[KK];
  __shared__ float gate;
  if (threadIdx.x < KK) {
    const bool in = threadIdx.x < K;
    rows[threadIdx.x] = in ? a.row_of[t * K + threadIdx.x] : -1;
    wts[threadIdx.x] = in ? a.topk_w[t * K + threadIdx.x] : 0.0f;
  }
  if (SHARED && threadIdx.x == 0) gate = 1.0f / (1.0f + __expf(-a.gate_logit[t]));
  __syncthreads();
  const T *Yp = reinterpret_cast<const T *>(a.Yp);
  const T *Ys = reinterpret_cast<const T *>(a.Ys);
  T *out = reinterpret_cast<T *>(a.out);
  int32_t r[KK];
#pragma unroll
  for (int k = 0; k < KK; ++k) r[k] = rows[k];
  for (int v = threadIdx.x * N; v < a.d; v += blockDim.x * N) {
    uint4 yraw[KK + 1];
#pragma unroll
    for (int k = 0; k < KK; ++k)
      if (r[k] >= 0) yraw[k] = *reinterpret_cast<const uint4 *>(Yp + (int64_t)r[k] * a.d + v);
    if constexpr (SHARED) yraw[KK] = *reinterpret_cast<const uint4 *>(Ys + t * a.d + v);
    float acc[N];
#pragma unroll
    for (int i = 0; i < N; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int k = 0; k < KK; ++k) {
      if (r[k] < 0) continue;
      float y[N];
      unpack16<T>(yraw[k], y);
      const float w = wts[k];
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = fmaf(w, y[i], acc[i]);
    }
    if constexpr (SHARED) {
      float y[N];
      unpack16<T>(yraw[KK], y);
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = fmaf(gate, y[i], acc[i]);
    }
    store16<T>(out + t * a.d + v, acc);
  }
}

// dYp[row] = w * dout[t]; dw[t,k] = <dout[t], Yp[row]>; shared: dYs, dz.
// One CTA per token. Per 16-byte column vector a thread first issues the
// loads of all K expert rows (and Ys), then computes and stores, so that
// K + 2 loads per thread are in flight; KK >= K is a compile-time bound,
// which keeps the registers per thread (and so the CTAs per SM) in line
// with the actual K. The K (+1) dot products are reduced with one butterfly
// per warp and then over the warps in order (fixed order: bitwise
// reproducible).
template <typename T, int KK, bool SHARED>
__global__ void __launch_bounds__(256) unpermute_bwd_kernel(UnpermuteArgs a) {
  constexpr int N = Vec<T>::N;
  constexpr int NS = KK + (SHARED ? 1 : 0);   // dot products per token
  const int64_t t = blockIdx.x;
  const int K = a.K;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __shared__ int32_t rows[KK];
  __shared__ float wts[KK];
  __shared__ float gate;
  __shared__ float red[8][NS];   // [warp][slot]; slot KK = shared expert
  if (threadIdx.x < KK) {
    const bool in = threadIdx.x < K;
    rows[threadIdx.x] = in ? a.row_of[t * K + threadIdx.x] : -1;
    wts[threadIdx.x] = in ? a.topk_w[t * K + threadIdx.x] : 0.0f;
  }
  if (SHARED && threadIdx.x == 0) gate = 1.0f / (1.0f + __expf(-a.gate_logit[t]));
  __syncthreads();
  const T *Yp = reinterpret_cast<const T *>(a.Yp);
  const T *dout = reinterpret_cast<const T *>(a.dout);
  T *dYp = reinterpret_cast<T *>(a.dYp);
  int32_t r[KK];
  float wk[KK];
#pragma unroll
  for (int k = 0; k < KK; ++k) {
    r[k] = rows[k];
    wk[k] = wts[k];
  }
  float dot[NS];
#pragma unroll
  for (int k = 0; k < NS; ++k) dot[k] = 0.0f;
  for (int v = threadIdx.x * N; v < a.d; v += blockDim.x * N) {
    uint4 yraw[NS];
    const uint4 graw = *reinterpret_cast<const uint4 *>(dout + t * a.d + v);
#pragma unroll
    for (int k = 0; k < KK; ++k)
      if (r[k] >= 0) yraw[k] = *reinterpret_cast<const uint4 *>(Yp + (int64_t)r[k] * a.d + v);
    if constexpr (SHARED)
      yraw[KK] = *reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(a.Ys) + t * a.d + v);
    float g[N];
    unpack16<T>(graw, g);
#pragma unroll
    for (int k = 0; k < KK; ++k) {
      if (r[k] < 0) continue;
      float y[N], o[N];
      unpack16<T>(yraw[k], y);
#pragma unroll
      for (int i = 0; i < N; ++i) {
        dot[k] = fmaf(g[i], y[i], dot[k]);
        o[i] = wk[k] * g[i];
      }
      store16<T>(dYp + (int64_t)r[k] * a.d + v, o);
    }
    if constexpr (SHARED) {
      float y[N], o[N];
      unpack16<T>(yraw[KK], y);
#pragma unroll
      for (int i = 0; i < N; ++i) {
        dot[KK] = fmaf(g[i], y[i], dot[KK]);
        o[i] = gate * g[i];
      }
      store16<T>(reinterpret_cast<T *>(a.dYs) + t * a.d + v, o);
    }
  }
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const float s = warp_sum(dot[k]);
    if (lane == 0) red[warp][k] = s;
  }
  __syncthreads();
  const int nw = blockDim.x >> 5;
  if (threadIdx.x < K) {
    const int k = threadIdx.x;
    float s = 0.0f;
    for (int w = 0; w < nw; ++w) s += red[w][k];
    a.dw[t * K + k] = rows[k] >= 0 ? s : 0.0f;
  } else if (SHARED && threadIdx.x == 32) {
    float s = 0.0f;
    for (int w = 0; w < nw; ++w) s += red[w][NS - 1];
    a.dz[t] = gate * (1.0f - gate) * s;
  }
}

// out = sum over parts (in part order, fp32) of partials[p]; one 16-byte
// vector per thread and iteration, grid-stride. HBM-bound: (n_parts + 1)
// rows*d elements moved.
template <typename T>
__global__ void __launch_bounds__(256) sum_partials_kernel(int n_parts, int64_t nvec,
                                                           const T *__restrict__ partials,
                                                           T *__restrict__ out) {
  constexpr int N = Vec<T>::N;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += stride) {
    float acc[N];
    load16<T>(partials + v * N, acc);
    for (int p = 1; p < n_parts; ++p) {
      float y[N];
      load16<T>(partials + ((int64_t)p * nvec + v) * N, y);
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = __fadd_rn(acc[i], y[i]);
    }
    store16<T>(out + v * N, acc);
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
// map_count writes every word that map_scatter later reads, so a call never
// sees the previous call's counts and nothing needs clearing.
constexpr int kNoAllocBlocks = MOE_PERMUTE_NOALLOC_MAX_TOKENS / kMapBlock;
static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocBlocks * 64];

namespace {
// Device address of g_permute_scratch in the current context. In host code
// the array's name is only a handle, so the address is looked up with
// cudaGetSymbolAddress (with the device current) the first time a context
// calls, and cached under the context's unique ID (cuCtxGetId: never reused
// within the process, so a context created after cudaDeviceReset, where the
// module and its array are loaded again, gets a lookup of its own).
constexpr int kMaxContexts = 64;
std::mutex g_scratch_mutex;
unsigned long long g_scratch_ctx[kMaxContexts] = {};
int32_t *g_scratch_addr[kMaxContexts] = {};
int g_scratch_n = 0;

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

template <typename Fn>
Fn driver_fn(const char *name, int version) {
  void *ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &ptr, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(ptr);
}

cudaError_t permute_scratch(int32_t **out) {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 4000);
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
  if (get_current == nullptr || get_id == nullptr) return cudaErrorNotSupported;
  int dev = 0;   // cudaSetDevice makes the device's primary context current on this thread
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaSetDevice(dev);
  if (e != cudaSuccess) return e;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
    return cudaErrorNotSupported;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  for (int i = 0; i < g_scratch_n; ++i)
    if (g_scratch_ctx[i] == id) {
      *out = g_scratch_addr[i];
      return cudaSuccess;
    }
  void *p = nullptr;
  e = cudaGetSymbolAddress(&p, g_permute_scratch);
  if (e != cudaSuccess) return e;
  const int slot = g_scratch_n < kMaxContexts ? g_scratch_n++ : (int)(id % kMaxContexts);
  g_scratch_ctx[slot] = id;
  g_scratch_addr[slot] = static_cast<int32_t *>(p);
  *out = static_cast<int32_t *>(p);
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
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nblk);
  cfg.blockDim = dim3(kMapBlock);
  cfg.dynamicSmemBytes = bm_bytes;
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, map_count_kernel, a);
  if (e != cudaSuccess) return e;
  e = cudaLaunchKernelEx(&cfg, map_scatter_kernel, a, nblk);
  if (e != cudaSuccess || a.Xp == nullptr) return e;   // Xp NULL: the map alone
  const uint32_t row_bytes = (uint32_t)a.d * (a.dtype == MOE_BF16 ? 2u : 4u);
  int tpc = kPermTokens;
  while (tpc > 1 && (uint32_t)tpc * row_bytes > kPermSmemCap) --tpc;
  const size_t smem = (size_t)tpc * row_bytes;
  if (smem > 200 * 1024) return cudaErrorInvalidValue;  // rows wider than the bulk path holds
  e = cudaFuncSetAttribute(permute_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3((unsigned)((a.T + tpc - 1) / tpc));
  cfg.blockDim = dim3(32);
  cfg.dynamicSmemBytes = smem;
  return cudaLaunchKernelEx(&cfg, permute_bulk_kernel, a, row_bytes, tpc);
}

// Slot bound KK >= K of the un-permute kernels: 1, 2, 4 or 8.
template <typename T, int KK>
cudaError_t launch_unpermute_kk(const UnpermuteArgs &a, cudaStream_t s) {
  if (a.Ys != nullptr)
    unpermute_kernel<T, KK, true><<<(unsigned)a.T, 256, 0, s>>>(a);
  else
    unpermute_kernel<T, KK, false><<<(unsigned)a.T, 256, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename T, int KK>
cudaError_t launch_unpermute_bwd_kk(const UnpermuteArgs &a, cudaStream_t s) {
  if (a.Ys != nullptr)
    unpermute_bwd_kernel<T, KK, true><<<(unsigned)a.T, 256, 0, s>>>(a);
  else
    unpermute_bwd_kernel<T, KK, false><<<(unsigned)a.T, 256, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_unpermute_t(const UnpermuteArgs &a, cudaStream_t s, bool bwd) {
  if (a.K <= 1) return bwd ? launch_unpermute_bwd_kk<T, 1>(a, s) : launch_unpermute_kk<T, 1>(a, s);
  if (a.K <= 2) return bwd ? launch_unpermute_bwd_kk<T, 2>(a, s) : launch_unpermute_kk<T, 2>(a, s);
  if (a.K <= 4) return bwd ? launch_unpermute_bwd_kk<T, 4>(a, s) : launch_unpermute_kk<T, 4>(a, s);
  return bwd ? launch_unpermute_bwd_kk<T, 8>(a, s) : launch_unpermute_kk<T, 8>(a, s);
}

cudaError_t launch_unpermute(const UnpermuteArgs &a, cudaStream_t s) {
  if (a.K < 1 || a.K > 8) return cudaErrorInvalidValue;
  return a.dtype == MOE_BF16 ? launch_unpermute_t<__nv_bfloat16>(a, s, false)
                             : launch_unpermute_t<float>(a, s, false);
}

cudaError_t launch_unpermute_bwd(const UnpermuteArgs &a, cudaStream_t s) {
  if (a.K < 1 || a.K > 8) return cudaErrorInvalidValue;
  return a.dtype == MOE_BF16 ? launch_unpermute_t<__nv_bfloat16>(a, s, true)
                             : launch_unpermute_t<float>(a, s, true);
}

cudaError_t launch_pad_fill(const PermuteArgs &a, cudaStream_t s) {
  const int vec_per_row = a.d * (a.dtype == MOE_BF16 ? 2 : 4) / 16;
  pad_fill_kernel<<<(unsigned)a.E, 256, 0, s>>>(a, vec_per_row);
  return cudaGetLastError();
}

cudaError_t launch_sum_partials(int dtype, int n_parts, int64_t rows, int d, const void *partials,
                                void *out, cudaStream_t s) {
  const int N = dtype == MOE_BF16 ? 8 : 4;
  const int64_t nvec = rows * d / N;
  if (nvec == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (nvec + 255) / 256, cap = (int64_t)(sms > 0 ? sms : 1) * 8;   // 8 CTAs per SM
  const int64_t blocks = want < cap ? want : cap;
  if (dtype == MOE_BF16)
    sum_partials_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(
        n_parts, nvec, reinterpret_cast<const __nv_bfloat16 *>(partials),
        reinterpret_cast<__nv_bfloat16 *>(out));
  else
    sum_partials_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(
        n_parts, nvec, reinterpret_cast<const float *>(partials), reinterpret_cast<float *>(out));
  return cudaGetLastError();
}

cudaError_t launch_permute_bwd(int64_t T, int d, int K, const float *dXp, const int32_t *row_of,
                               const float *dx_add, float *dx, cudaStream_t s) {
  permute_bwd_kernel<<<(unsigned)T, 256, 0, s>>>(T, d, K, dXp, row_of, dx_add, dx);
  return cudaGetLastError();
}

}  // namespace moe
