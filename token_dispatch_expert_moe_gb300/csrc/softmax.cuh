// The routing softmax, specified operation by operation in fp32 so that any
// two implementations fed the same fp32 logits take the same decisions:
// no fused multiply-add (explicit _rn intrinsics), an exponential of our own
// (Cody-Waite reduction with ln 2 split in a 9-bit head and a tail; degree-7
// Taylor polynomial in Horner form; scaling by 2^n through the exponent
// field; flush to 0 below the normal range), a stride-halving pairwise sum
// over the experts zero-padded to a power of two, a correctly rounded
// division. Top-K: K arg-max rounds, ties to the lower expert index.
#pragma once
#include "common.cuh"

namespace moe {
namespace spec {

constexpr float kLog2e = (float)1.4426950408889634;
constexpr float kLn2Hi = 0.693359375f;  // 355/512
constexpr float kLn2Lo = (float)(0.69314718055994530942 - 0.693359375);
// 1/k!, correctly rounded to fp32
constexpr float kC0 = 1.0f;
constexpr float kC1 = 1.0f;
constexpr float kC2 = 0.5f;
constexpr float kC3 = (float)(1.0 / 6.0);
constexpr float kC4 = (float)(1.0 / 24.0);
constexpr float kC5 = (float)(1.0 / 120.0);
constexpr float kC6 = (float)(1.0 / 720.0);
constexpr float kC7 = (float)(1.0 / 5040.0);

// e^u for u <= 0.
__device__ __forceinline__ float exp_spec(float u) {
  const float n = rintf(__fmul_rn(u, kLog2e));
  const float r = __fsub_rn(__fsub_rn(u, __fmul_rn(n, kLn2Hi)), __fmul_rn(n, kLn2Lo));
  float p = kC7;
  p = __fadd_rn(__fmul_rn(p, r), kC6);
  p = __fadd_rn(__fmul_rn(p, r), kC5);
  p = __fadd_rn(__fmul_rn(p, r), kC4);
  p = __fadd_rn(__fmul_rn(p, r), kC3);
  p = __fadd_rn(__fmul_rn(p, r), kC2);
  p = __fadd_rn(__fmul_rn(p, r), kC1);
  p = __fadd_rn(__fmul_rn(p, r), kC0);
  const int ni = (int)n;
  if (ni < -125) return 0.0f;
  return __fmul_rn(p, __int_as_float((ni + 127) << 23));
}

// fp32 value <-> unsigned key with the same order (negative values flipped),
// for warp-wide maxima with one redux instruction; exact both ways
__device__ __forceinline__ unsigned ordered_key(float v) {
  const unsigned b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float ordered_value(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// p for the two experts a lane holds (lane, lane+32); -1 for absent experts.
__device__ __forceinline__ void softmax_warp(float l0, float l1, int E, float &p0, float &p1) {
  const int lane = threadIdx.x & 31;
  const bool v0 = lane < E, v1 = lane + 32 < E;
  // the maximum is exact in any order: one warp-wide redux of ordered keys
  const float m = ordered_value(__reduce_max_sync(
      0xffffffffu, ordered_key(fmaxf(v0 ? l0 : -INFINITY, v1 ? l1 : -INFINITY))));
  const float q0 = v0 ? exp_spec(__fsub_rn(l0, m)) : 0.0f;
  const float q1 = v1 ? exp_spec(__fsub_rn(l1, m)) : 0.0f;
  float s = __fadd_rn(q0, q1);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
  p0 = v0 ? __fdiv_rn(q0, s) : -1.0f;
  p1 = v1 ? __fdiv_rn(q1, s) : -1.0f;
}

// One warp routes one token. Lane l holds the logits of experts l and l+32
// (E <= 64). Writes topk_idx/prob/w[K] and keep = 1 for the token.
__device__ __forceinline__ void softmax_topk_warp(float l0, float l1, int E, int K, int renorm,
                                                  int32_t *idx_out, float *prob_out,
                                                  float *w_out, uint8_t *keep_out) {
  const int lane = threadIdx.x & 31;
  float p0, p1;
  softmax_warp(l0, l1, E, p0, p1);
  float my_prob = 0.0f;
  int my_idx = 0;
  for (int k = 0; k < K; ++k) {
    // lane-local best (lower index wins ties: expert `lane` before lane+32),
    // then the warp's largest p and the lowest expert index holding it
    float lp = p0;
    int li = lane;
    if (p1 > lp) { lp = p1; li = lane + 32; }
    const unsigned kmax = __reduce_max_sync(0xffffffffu, ordered_key(lp));
    const int bi = (int)__reduce_min_sync(0xffffffffu, ordered_key(lp) == kmax ? (unsigned)li : 64u);
    const float bp = ordered_value(kmax);
    if (bi == lane) p0 = -2.0f;
    if (bi == lane + 32) p1 = -2.0f;
    if (lane == k) { my_prob = bp; my_idx = bi; }
  }
  // Z = prob_0 + prob_1 + ... in slot order
  float Z = __shfl_sync(0xffffffffu, my_prob, 0);
  for (int k = 1; k < K; ++k) Z = __fadd_rn(Z, __shfl_sync(0xffffffffu, my_prob, k));
  if (lane < K) {
    idx_out[lane] = my_idx;
    prob_out[lane] = my_prob;
    w_out[lane] = renorm ? __fdiv_rn(my_prob, Z) : my_prob;
    keep_out[lane] = 1;
  }
}

}  // namespace spec
}  // namespace moe
