// fp32 grouped SwiGLU FFN on the CUDA cores (dtype MOE_F32).
//
// The expert FFN of the MoE Parallel Folding dispatcher (study notes, "method
// overview": expert FFN computation) for fp32 layers. The bf16 tensor-core
// path lives in gemm_tc.cu; fp32 tensor-core (tf32) arithmetic would not meet
// an fp32 tolerance, so this path is plain FMA.
//
// One generic tiled kernel computes C[m,n] = sum_k A(m,k) B(n,k) per group,
// with strided operand access, in two modes:
//   ROWS: M is the group's row range [offsets[g], offsets[g+1]) (forward and
//         data-gradient GEMMs; the weights are per-group B operands);
//   RED:  K is the group's row range (weight gradients); M, N fixed.
// 64x64 tiles, 16-deep K steps staged in shared memory, 4x4 per thread.
#include "common.cuh"

namespace moe {
namespace {

enum Epi { kEpiGateUp = 0, kEpiStore = 1, kEpiSwigluBwd = 2, kEpiStoreRed = 3 };

struct SimtGemm {
  int red;  // 0: ROWS mode, 1: RED mode
  int M, N, K;
  const int32_t *offsets;
  const float *A;
  int64_t sAm, sAk, sAg;
  const float *B;
  int64_t sBn, sBk, sBg;
  float *C;
  int64_t ldc, sCg;
  // SwiGLU epilogues
  int F;
  float *A_save, *H_save;   // forward gate/up epilogue
  const float *A_in;        // backward: saved [G|U]
  float *dA;                // backward: [dG|dU]
};

constexpr int BM = 64, BN = 64, BK = 16;

template <int EPI>
__global__ void __launch_bounds__(256) simt_gemm_kernel(SimtGemm p) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[(EPI == kEpiGateUp) ? 2 : 1][BK][BN + 4];
  const int g = blockIdx.z;
  const int lo = p.offsets[g], hi = p.offsets[g + 1];
  const int M = p.red ? p.M : hi - lo;
  const int K = p.red ? hi - lo : p.K;
  const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
  if (m0 >= M) return;
  const float *A = p.A + (p.red ? (int64_t)lo * p.sAk : (int64_t)lo * p.sAm);
  const float *B = p.B + (p.red ? (int64_t)lo * p.sBk : (int64_t)g * p.sBg);
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[2][4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BK) {
    for (int i = threadIdx.x; i < BM * BK; i += 256) {
      const int mm = i % BM, kk = i / BM;
      const int m = m0 + mm, k = k0 + kk;
      As[kk][mm] = (m < M && k < K) ? A[(int64_t)m * p.sAm + (int64_t)k * p.sAk] : 0.0f;
    }
    for (int h = 0; h < ((EPI == kEpiGateUp) ? 2 : 1); ++h) {
      for (int i = threadIdx.x; i < BN * BK; i += 256) {
        const int nn = i % BN, kk = i / BN;
        const int n = n0 + nn + h * p.F, k = k0 + kk;
        Bs[h][kk][nn] = (n0 + nn < p.N && k < K) ? B[(int64_t)n * p.sBn + (int64_t)k * p.sBk] : 0.0f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[2][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int h = 0; h < ((EPI == kEpiGateUp) ? 2 : 1); ++h)
#pragma unroll
        for (int j = 0; j < 4; ++j) b[h][j] = Bs[h][kk][tx * 4 + j];
#pragma unroll
      for (int h = 0; h < ((EPI == kEpiGateUp) ? 2 : 1); ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[h][i][j] = fmaf(a[i], b[h][j], acc[h][i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= p.N) continue;
      if constexpr (EPI == kEpiGateUp) {
        const int64_t row = lo + m;
        const float G = acc[0][i][j], U = acc[1][i][j];
        if (p.A_save) {
          p.A_save[row * 2 * p.F + n] = G;
          p.A_save[row * 2 * p.F + p.F + n] = U;
        }
        p.H_save[row * p.F + n] = G / (1.0f + expf(-G)) * U;
      } else if constexpr (EPI == kEpiSwigluBwd) {
        const int64_t row = lo + m;
        const float dH = acc[0][i][j];
        const float G = p.A_in[row * 2 * p.F + n], U = p.A_in[row * 2 * p.F + p.F + n];
        const float sg = 1.0f / (1.0f + expf(-G));
        p.dA[row * 2 * p.F + n] = dH * U * sg * (1.0f + G * (1.0f - sg));
        p.dA[row * 2 * p.F + p.F + n] = dH * G * sg;
      } else if constexpr (EPI == kEpiStore) {
        p.C[(int64_t)(lo + m) * p.ldc + n] = acc[0][i][j];
      } else {
        p.C[(int64_t)g * p.sCg + (int64_t)m * p.ldc + n] = acc[0][i][j];
      }
    }
  }
}

template <int EPI>
cudaError_t run(const SimtGemm &p, int64_t max_m, int n_groups, cudaStream_t s) {
  dim3 grid((unsigned)((max_m + BM - 1) / BM), (unsigned)((p.N + BN - 1) / BN), (unsigned)n_groups);
  simt_gemm_kernel<EPI><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ffn_fwd_f32(const FfnArgs &a, cudaStream_t s) {
  const int d = a.d, F = a.F;
  float *H = reinterpret_cast<float *>(a.H_save ? a.H_save : a.H_tmp);
  SimtGemm p{};
  // G|U = Xp W_gu^T, SwiGLU epilogue
  p.red = 0; p.N = F; p.K = d; p.offsets = a.offsets;
  p.A = reinterpret_cast<const float *>(a.Xp); p.sAm = d; p.sAk = 1;
  p.B = reinterpret_cast<const float *>(a.W_gu); p.sBn = d; p.sBk = 1; p.sBg = (int64_t)2 * F * d;
  p.F = F; p.A_save = reinterpret_cast<float *>(a.A_save); p.H_save = H;
  cudaError_t e = run<kEpiGateUp>(p, a.max_rows, a.n_groups, s);
  if (e != cudaSuccess) return e;
  // Yp = H W_down^T
  SimtGemm q{};
  q.red = 0; q.N = d; q.K = F; q.offsets = a.offsets;
  q.A = H; q.sAm = F; q.sAk = 1;
  q.B = reinterpret_cast<const float *>(a.W_down); q.sBn = F; q.sBk = 1; q.sBg = (int64_t)d * F;
  q.C = reinterpret_cast<float *>(a.Yp); q.ldc = d;
  return run<kEpiStore>(q, a.max_rows, a.n_groups, s);
}

cudaError_t launch_ffn_bwd_f32(const FfnArgs &a, cudaStream_t s) {
  const int d = a.d, F = a.F;
  const float *dYp = reinterpret_cast<const float *>(a.dYp);
  float *dA = reinterpret_cast<float *>(a.dA);
  cudaError_t e;
  {  // dH = dYp W_down  ->  dA = [dG | dU]
    SimtGemm p{};
    p.red = 0; p.N = F; p.K = d; p.offsets = a.offsets;
    p.A = dYp; p.sAm = d; p.sAk = 1;
    p.B = reinterpret_cast<const float *>(a.W_down); p.sBn = 1; p.sBk = F; p.sBg = (int64_t)d * F;
    p.F = F; p.A_in = reinterpret_cast<const float *>(a.A_save); p.dA = dA;
    if ((e = run<kEpiSwigluBwd>(p, a.max_rows, a.n_groups, s)) != cudaSuccess) return e;
  }
  {  // dXp = dA W_gu
    SimtGemm p{};
    p.red = 0; p.N = d; p.K = 2 * F; p.offsets = a.offsets;
    p.A = dA; p.sAm = 2 * F; p.sAk = 1;
    p.B = reinterpret_cast<const float *>(a.W_gu); p.sBn = 1; p.sBk = d; p.sBg = (int64_t)2 * F * d;
    p.C = a.dXp; p.ldc = d;
    if ((e = run<kEpiStore>(p, a.max_rows, a.n_groups, s)) != cudaSuccess) return e;
  }
  {  // dW_down[g] = dYp_g^T H_g   (M = d, N = F, K = rows)
    SimtGemm p{};
    p.red = 1; p.M = d; p.N = F; p.offsets = a.offsets;
    p.A = dYp; p.sAm = 1; p.sAk = d;
    p.B = reinterpret_cast<const float *>(a.H_save); p.sBn = 1; p.sBk = F;
    p.C = a.dW_down; p.ldc = F; p.sCg = (int64_t)d * F;
    if ((e = run<kEpiStoreRed>(p, d, a.n_groups, s)) != cudaSuccess) return e;
  }
  {  // dW_gu[g] = dA_g^T Xp_g   (M = 2F, N = d, K = rows)
    SimtGemm p{};
    p.red = 1; p.M = 2 * F; p.N = d; p.offsets = a.offsets;
    p.A = dA; p.sAm = 1; p.sAk = 2 * F;
    p.B = reinterpret_cast<const float *>(a.Xp); p.sBn = 1; p.sBk = d;
    p.C = a.dW_gu; p.ldc = d; p.sCg = (int64_t)2 * F * d;
    if ((e = run<kEpiStoreRed>(p, 2 * F, a.n_groups, s)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace moe
