// Grouped GEMMs of the SwiGLU experts on the sm_103a tensor cores.
//
// MoE Parallel Folding (arXiv 2504.14960) study notes, "method overview":
// after the permutation each expert's tokens are contiguous and the experts'
// FFN runs on them; the backward runs the same chain in reverse. The expert
// rows of group g are [offsets[g], offsets[g+1]) of the permuted buffers;
// offsets stay on the device and every CTA derives the tile list from them.
//
// Two persistent, warp-specialised kernel templates (192 threads, one CTA per
// SM):
//   warp 0      TMA producer: 128B-swizzled boxes into a shared-memory ring;
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma kind::f16 (bf16 in,
//               fp32 accumulate), K = 16 per instruction, 4 per 64-deep
//               stage; tcgen05.commit frees the stage and, at the end of a
//               tile, hands the accumulator over;
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (one TMEM lane
//               quarter per warp), fused math, 32-row slabs staged in swizzled
//               shared memory and written with TMA bulk stores.
// tc_gemm_kernel: one CTA per tile, M = 128, 4 stages of 48 KB (6 smaller
// ones in the router mode); it runs the router GEMM, the row-grouped experts'
// last tiles of at most 128 rows (as a programmatic dependent of the pair
// kernel), and every tile when CTA pairs are disabled. tc_gemm_pair_kernel:
// clusters of two CTAs on one TPC issue tcgen05.mma.cta_group::2 (M = 256,
// each CTA holding its 128 rows of A and half of B), 6 stages of 32 KB per
// CTA; the even CTA's barriers see both CTAs' TMA bytes and its MMA warp
// issues for the pair. Two TMEM accumulators (2 x 256 columns) let the
// epilogue of one tile overlap the mainloop of the next; where K is long, a
// pair tile covers two adjacent N tiles instead (4 stages of 48 KB sharing
// each A box, one accumulator per N tile), and the MMA warp starts a tile's
// accumulator 0 as soon as the epilogue has drained it. In the gate/up mode
// with the permutation fused in, two more warps gather the A rows from x.
//
// The GEMMs (A: M x K, B: N x K, per group g):
//   GU      [G|U] = Xp W_gu[g]^T, SwiGLU epilogue H = silu(G) U (+ A_save)
//   DOWN    Yp    = H W_down[g]^T
//   DH      dH    = dYp W_down[g]  -> epilogue dA = [dG | dU]   (B MN-major)
//   DX      dXp   = dA W_gu[g]                                   (B MN-major)
//   WGD     dW_down[g] = dYp_g^T H_g     (K = the group's rows; A, B MN-major)
//   WGU     dW_gu[g]   = dA_g^T Xp_g
//   RT      router logits = x W_r^T (+ b_r) and gate logit x . w_sg: one
//           group of T rows, N = E rounded up to 16 (+ 16 when the gate
//           vector rides along as a second B box); fp32 logits out. When
//           T / 128 row tiles would leave SMs idle, the K loop is split over
//           a cluster of k_split CTAs per row tile: the odd CTAs send their
//           fp32 partial sums to the even CTA's shared memory, which adds them
//           in part order. With no split and E <= 16 the epilogue also routes
//           (softmax, Top-K, combine weights).
// In GU/DOWN/DH/DX a tile's rows past the group's end belong to the next
// group (or are zero-filled past the buffer); only their outputs are masked.
// In WGD/WGU the reduction runs over the group's rows: the loads go through
// per-group tensor maps whose outer extent is the group's row count (written
// on the device by group_maps_kernel), so the TMA zero-fills K rows past the
// group's end.
//
// Every wait on an mbarrier is bounded (about two seconds of
// %globaltimer); on expiry the kernel records MOE_ERR_TIMEOUT in the status
// word, tells the other roles to stop, drains what it has in flight and
// returns, so the GPU context stays usable.
#include <cstdlib>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "softmax.cuh"

namespace moe {
namespace {

enum Mode { GU = 0, DOWN = 1, DH = 2, DX = 3, WGD = 4, WGU = 5, RT = 6 };

constexpr int kStages = 4;
constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 192;
constexpr int kGatherWarps = 2;   // A-gather warps (GU gather mode): 256 threads in all, so
                                  // the epilogue keeps the registers it has without them
constexpr int kThreadsGather = kThreads + 32 * kGatherWarps;
constexpr int kABytes = BM * BK * 2;          // 16 KB
constexpr int kBBytesMax = 256 * BK * 2;      // 32 KB
constexpr int kStageBytes = kABytes + kBBytesMax;
constexpr int kTmemCols = 512;
constexpr int kStageOutBytes = 4096;                 // 32 rows x 128 B
constexpr int kEpiStagingBytes = 4 * 2 * kStageOutBytes;  // 4 warps x 2 buffers
constexpr uint64_t kTimeoutNs = 2000000000ull;

struct TcParams {
  CUtensorMap tmA;
  CUtensorMap tmB;
  CUtensorMap tmC;   // RT: the gate vector w_sg as a [1, d] tensor
  CUtensorMap tmO0;  // bulk-store map of out0 (box: 32 rows x 128 bytes)
  CUtensorMap tmO1;  // bulk-store map of out1 (GU: A_save)
  CUtensorMap tmX;   // GU gather: x [T, d] in boxes of one row x 64 columns
  int mode;
  int n_groups;
  int64_t max_rows;
  int d, F;
  int M_fixed;   // WGD/WGU: rows of the weight-gradient matrix
  int N;         // output columns (GU: F, the MMA sees 2 x 128)
  int K_fixed;   // GU/DOWN/DH/DX: reduction depth
  int64_t b_group_rows;  // B rows per group in the B tensor map (y offset)
  const int32_t *offsets;
  void *out0;    // GU: H; DOWN: Yp; DH: dA; DX: dXp; WG*: dW
  void *out1;    // GU: A_save (nullable)
  const void *aux;  // DH: A_save
  // WGD/WGU: per group, the A and B tensor maps of that group's rows alone
  // ([2g] = A, [2g+1] = B; outer extent = the group's row count), so the TMA
  // zero-fills the K rows past the group's end of a ragged last K block
  const CUtensorMap *gmaps;
  int fault_stall;   // test hook: the producer issues no loads (waits run out)
  // row-grouped modes, ragged tails: a group whose last 256 rows hold at most
  // 128 rows (0 < rows % 256 <= 128) has that tail computed by the single-CTA
  // kernel (128-row tiles) instead of a half-empty CTA-pair tile.
  //   1: the pair kernel leaves such tails out (and lets the tail kernel launch
  //      as its programmatic dependent);
  //   2: the single-CTA kernel computes only those tails (and waits for the
  //      pair kernel before it completes, so later work sees both)
  int tail_mode;
  // GU with a gathered A operand (the permutation fused into the GEMM): row
  // R < offsets[n_groups] of the tile is token src_of[R] / gK of x [gT, d]
  // (through tmX); other rows, and rows with src_of < 0 (padding), are zero
  const int32_t *src_of;
  int gK;
  int64_t gT;
  // RT: logits, then softmax, Top-K and combine weights in the epilogue
  int64_t T;
  int E, e_pad, has_gate;
  const float *bias;
  float *gate_out;
  int k_split, kb_per;  // K blocks split over k_split tiles of kb_per blocks each;
                        // k_split > 1: the split tiles of a row tile form a cluster
  int K, renorm, ep;    // Top-K, renormalisation; ep: 0 (logits only) or 8/16 >= E
  int32_t *topk_idx;
  float *topk_prob, *topk_w;
  uint8_t *keep;
  uint32_t *status;
};

// ---------------------------------------------------------------------------
// PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait with acquire at cluster scope: pairs with release arrivals that
// the other CTA of a pair makes on this barrier
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// arrive on a barrier of either CTA of the pair (cluster address), raising
// its expected transaction bytes first
__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t cluster_addr, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(
                   cluster_addr),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *tm, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
// Acquire side of a tensor map written by an earlier kernel (the group maps
// of the weight-gradient modes): orders the map's bytes before its TMA use.
__device__ __forceinline__ void tensormap_acquire(const CUtensorMap *m) {
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(m) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
// --- CTA-pair (cta_group::2) forms -------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_to_cta(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// Four rows of a tensor map whose box is one row high (tile::gather4): rows
// r0..r3, columns c0 .. c0 + box width, put one after another at dst in this
// CTA's shared memory; completes on a barrier of either CTA of the pair.
__device__ __forceinline__ void tma_gather4_pair(uint32_t dst, const CUtensorMap *tm,
                                                 uint32_t bar_cluster, int c0, int r0, int r1,
                                                 int r2, int r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar_cluster), "r"(c0), "r"(r0), "r"(r1), "r"(r2),
      "r"(r3)
      : "memory");
}

// TMA load into this CTA's shared memory that completes on a barrier of
// either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *tm,
                                                 uint32_t bar_cluster, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tc_mma_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive on the barrier at this shared-memory offset in both CTAs of the pair
__device__ __forceinline__ void tc_commit_pair_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"((uint16_t)0x3)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Two 32-column TMEM loads (at ta and tb) in flight before one wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, float (&a)[32], float (&b)[32]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(ta), "r"(tb)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    a[i] = __uint_as_float(r[i]);
    b[i] = __uint_as_float(r[32 + i]);
  }
}

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 family format):
// start address >> 4 in bits 0-13, leading byte offset >> 4 in 16-29, stride
// byte offset >> 4 in 32-45, descriptor version 1 at bit 46, layout
// SWIZZLE_128B (2) in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
         ((uint64_t)(sbo >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Epilogue staging for bulk (TMA) stores. Each epilogue warp owns two 4 KB
// buffers; a buffer holds its 32 rows x 128 bytes in the 128-byte swizzled
// layout of the store's tensor map (16-byte chunk c of row r at chunk
// c ^ (r % 8)), so that lane r writing its row touches every bank group once
// per 8 lanes.
struct Stager {
  uint8_t *base;
  int next;
};
__device__ __forceinline__ uint8_t *stage_begin(Stager &sg, int lane) {
  // the buffer used two stores ago must have been read by its bulk copy
  if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
  __syncwarp();
  uint8_t *b = sg.base + sg.next * kStageOutBytes;
  sg.next ^= 1;
  return b;
}
__device__ __forceinline__ void stage_row(uint8_t *b, int lane, const uint32_t (&w)[32]) {
  uint8_t *row = b + lane * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<uint4 *>(row + ((c ^ (lane & 7)) << 4)) =
        make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}
__device__ __forceinline__ void stage_store(uint8_t *b, const CUtensorMap *tm, int x, int y,
                                            int lane) {
  fence_proxy_async();
  __syncwarp();
  if (lane == 0) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(smem_u32(b)), "r"(x), "r"(y)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  }
}
__device__ __forceinline__ void pack_f32(const float (&v)[32], uint32_t (&w)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i]);
}
// 32 floats -> 16 words of bf16 pairs at w[off .. off+15]
__device__ __forceinline__ void pack_bf16(const float (&v)[32], uint32_t (&w)[32], int off) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[off + i] = *reinterpret_cast<uint32_t *>(&h);
  }
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A
// and B (bits 7-9, 10-12 = 1), A/B major-ness (bits 15, 16: 1 = MN-major),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

template <int MODE> struct ModeTraits {
  static constexpr bool red = (MODE == WGD || MODE == WGU);
  static constexpr int a_mn = red ? 1 : 0;
  static constexpr int b_mn = (MODE == DH || MODE == DX || red) ? 1 : 0;
};

constexpr int kMaxStages = 6;
struct SharedState {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t ebar[4];  // DH: per-epilogue-warp A_save box loads
  uint64_t xbar;     // RT with a split K loop: the other parts' partial logits arrived
  uint32_t tmem_base;
  volatile int abort;
  int total_tiles;
  int tile_start[65];  // ROWS mode: first tile index of each group
  int mtiles[64];      // ROWS mode: m-tiles of each group
  int mbase[64];       // ROWS mode: first m-tile of each group's tile range
};

struct Tile {
  int g, m, n;       // group, m-tile, n-tile
  int row0, rows;    // ROWS: first row and row count of the group; RED: K rows
};

template <int MODE, int BN>
__device__ __forceinline__ Tile decode_tile(const TcParams &p, const SharedState &st, int idx) {
  Tile t;
  if constexpr (MODE == RT) {
    t.g = 0; t.m = idx / p.k_split; t.n = idx % p.k_split;   // n: the K split
    t.row0 = 0; t.rows = (int)p.T;
  } else if constexpr (ModeTraits<MODE>::red) {
    const int MT = p.M_fixed / BM, NT = p.N / BN;
    t.g = idx / (MT * NT);
    const int loc = idx % (MT * NT);
    t.n = loc / MT;
    t.m = loc % MT;
    t.row0 = p.offsets[t.g];
    t.rows = p.offsets[t.g + 1] - t.row0;
  } else {
    int g = 0;
    while (g + 1 < p.n_groups && st.tile_start[g + 1] <= idx) ++g;
    const int loc = idx - st.tile_start[g];
    const int mt = st.mtiles[g];
    t.g = g;
    t.n = loc / mt;
    t.m = st.mbase[g] + loc % mt;
    t.row0 = p.offsets[g];
    t.rows = p.offsets[g + 1] - t.row0;
  }
  return t;
}

// 0 < rows % 256 <= 128: the group's last 256 rows would fill at most half a
// CTA-pair tile
__device__ __forceinline__ bool half_tail(int rows) {
  const int rem = rows % 256;
  return rows > 0 && rem > 0 && rem <= 128;
}

__device__ bool wait_bounded(SharedState &st, uint32_t bar, uint32_t parity, uint32_t *status,
                             uint32_t role, bool cluster_acquire = false) {
  auto test = [&]() {
    return cluster_acquire ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (test()) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
      if (test()) return true;
    if (st.abort) return false;
    if (globaltimer() - t0 > kTimeoutNs) {
      report(status, MOE_ERR_TIMEOUT, kInfoGemmTimeout + role);
      st.abort = 1;
      return false;
    }
  }
}

// Router epilogue, one token row per thread: bias, logits out, then the
// routing softmax, Top-K and combine weights in the fp32 arithmetic that
// softmax.cuh specifies for a warp, done here by one thread over its row:
// the same maximum, the same exponential of each difference, the sum in the
// same pairwise tree (zero-padded to EP, a power of two >= E: adding the zero
// padding is exact, so any such EP gives the tree of the next power of two),
// correctly rounded divisions, K arg-max rounds with ties to the lower
// expert, Z summed in slot order. v holds the row's fp32 sums (columns < E,
// the gate logit, when present, at column GC = the tile width - 16).
template <int EP, int NV, int GC>
__device__ __forceinline__ void route_row(const TcParams &p, const float (&v)[NV], int64_t row) {
  const int E = p.E;
  float l[EP];
#pragma unroll
  for (int e = 0; e < EP; ++e) {
    l[e] = v[e];
    if (e < E && p.bias != nullptr) l[e] = __fadd_rn(l[e], p.bias[e]);
  }
  float *lg = reinterpret_cast<float *>(p.out0) + row * E;
#pragma unroll
  for (int e = 0; e < EP; ++e)
    if (e < E) lg[e] = l[e];
  if (p.has_gate) p.gate_out[row] = v[GC];
  float m = -INFINITY;
#pragma unroll
  for (int e = 0; e < EP; ++e)
    if (e < E) m = fmaxf(m, l[e]);
  float q[EP], sum[EP];
#pragma unroll
  for (int e = 0; e < EP; ++e) {
    q[e] = e < E ? spec::exp_spec(__fsub_rn(l[e], m)) : 0.0f;
    sum[e] = q[e];
  }
#pragma unroll
  for (int lv = 1; lv <= 6; ++lv) {   // h = EP/2, EP/4, ..., 1 (constant bounds: registers)
    const int h = EP >> lv;
#pragma unroll
    for (int i = 0; i < EP / 2; ++i)
      if (i < h) sum[i] = __fadd_rn(sum[i], sum[i + h]);
  }
  float pr[EP];
#pragma unroll
  for (int e = 0; e < EP; ++e) pr[e] = e < E ? __fdiv_rn(q[e], sum[0]) : -1.0f;
  float bp[8];
  int bi[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    bp[k] = 0.0f;
    bi[k] = 0;
    if (k < p.K) {
      float b = -3.0f;
      int ix = 0;
#pragma unroll
      for (int e = 0; e < EP; ++e)
        if (pr[e] > b) { b = pr[e]; ix = e; }
#pragma unroll
      for (int e = 0; e < EP; ++e)
        if (e == ix) pr[e] = -2.0f;
      bp[k] = b;
      bi[k] = ix;
    }
  }
  float Z = bp[0];
#pragma unroll
  for (int k = 1; k < 8; ++k)
    if (k < p.K) Z = __fadd_rn(Z, bp[k]);
#pragma unroll
  for (int k = 0; k < 8; ++k)
    if (k < p.K) {
      p.topk_idx[row * p.K + k] = bi[k];
      p.topk_prob[row * p.K + k] = bp[k];
      p.topk_w[row * p.K + k] = p.renorm ? __fdiv_rn(bp[k], Z) : bp[k];
      p.keep[row * p.K + k] = 1;
    }
}

// Logistic sigmoid 1 / (1 + e^-x) of the SwiGLU epilogues, with the fast
// division intrinsic (within 2 ulp of fp32 for a divisor in [1, 2^126];
// 1 + e^-x >= 1, and an overflowed e^-x gives 0). Its results are rounded to
// bf16 (H, dA), whose unit is 2^16 fp32 ulps; the correctly rounded
// reciprocal cost the dH epilogue two thirds of its time.
__device__ __forceinline__ float sigmoid_fast(float x) {
  return __fdividef(1.0f, 1.0f + __expf(-x));
}

// One tile's epilogue for the epilogue warp that owns TMEM lane quarter q.
// xbuf (router mode with a split K loop, even CTA): the other parts' partial
// sums, [part - 1][128 rows][E + has_gate].
template <int MODE, int BN>
__device__ __forceinline__ void epilogue_tile(const TcParams &p, SharedState &st, Stager &sg,
                                              uint32_t &ephase, const Tile &t, uint32_t tbase,
                                              int q, int warp, int lane, float *xbuf = nullptr) {
  using TR = ModeTraits<MODE>;
  const int r_loc = t.m * BM + q * 32 + lane;
  if constexpr (MODE == RT) {
    constexpr int NV = (BN + 31) / 32 * 32;
    constexpr int GC = BN - 16;   // the gate logit's column (tile width = E rounded to 16, + 16)
    const int rl = q * 32 + lane;   // row within the tile
    const int64_t row = r_loc;
    const bool valid = row < p.T;
    const int C = p.E + p.has_gate;
    const int CS = (C + 3) & ~3;   // exchange row stride (16-byte aligned rows)
    // the row's values sit in v[0 .. C) already (no gate, or the gate column
    // right after the experts): the exchange moves them four at a time
    const bool contig = (p.E & 3) == 0 && (!p.has_gate || GC == p.E);
    float v[NV];
#pragma unroll
    for (int c = 0; c < NV / 32; ++c) {
      float chunk[32];
      tmem_ld32(tbase + c * 32, chunk);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[c * 32 + i] = chunk[i];
    }
    if (p.k_split > 1) {
      // part t.n of the K loop; part 0 (the even CTA of the cluster) adds the
      // others in part order
      if (t.n != 0) {
        if (valid) {
          const uint32_t dst = map_to_cta(smem_u32(xbuf + ((t.n - 1) * BM + rl) * CS), 0);
          if (contig) {
#pragma unroll
            for (int j = 0; j < NV; j += 4)
              if (j < CS)
                asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst + 4 * j),
                             "f"(v[j]), "f"(v[j + 1]), "f"(v[j + 2]), "f"(v[j + 3])
                             : "memory");
          } else {
#pragma unroll
            for (int j = 0; j < NV; ++j) {
              const int e = j < p.E ? j : (j == GC && p.has_gate ? p.E : -1);
              if (e >= 0)
                asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dst + 4 * e), "f"(v[j]) : "memory");
            }
          }
        }
        mbar_arrive_cluster(map_to_cta(smem_u32(&st.xbar), 0));
        return;
      }
      if (!wait_bounded(st, smem_u32(&st.xbar), 0, p.status, 7, true)) return;
      if (!valid) return;
      for (int part = 1; part < p.k_split; ++part) {
        const float *src = xbuf + ((part - 1) * BM + rl) * CS;
        if (contig) {
#pragma unroll
          for (int j = 0; j < NV; j += 4) {
            if (j < CS) {
              const float4 w = *reinterpret_cast<const float4 *>(src + j);
              v[j] = __fadd_rn(v[j], w.x);
              v[j + 1] = __fadd_rn(v[j + 1], w.y);
              v[j + 2] = __fadd_rn(v[j + 2], w.z);
              v[j + 3] = __fadd_rn(v[j + 3], w.w);
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < NV; ++j) {
            const int e = j < p.E ? j : (j == GC && p.has_gate ? p.E : -1);
            if (e >= 0) v[j] = __fadd_rn(v[j], src[e]);
          }
        }
      }
    }
    if (!valid) return;
    if (p.ep == 0) {   // logits only: the Top-K kernel routes
      float *lg = reinterpret_cast<float *>(p.out0) + row * p.E;
      if ((p.E & 3) == 0 && (reinterpret_cast<uintptr_t>(p.out0) & 15) == 0) {
        // four logits per 16-byte store: a thread writes its own row, so a
        // warp's store touches 32 rows; wide stores cut those transactions 4x
#pragma unroll
        for (int e = 0; e < NV; e += 4) {
          if (e < p.E) {
            float4 w = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
            if (p.bias != nullptr) {
              w.x = __fadd_rn(w.x, p.bias[e]);
              w.y = __fadd_rn(w.y, p.bias[e + 1]);
              w.z = __fadd_rn(w.z, p.bias[e + 2]);
              w.w = __fadd_rn(w.w, p.bias[e + 3]);
            }
            *reinterpret_cast<float4 *>(lg + e) = w;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < NV; ++e) {
          if (e < p.E) lg[e] = p.bias != nullptr ? __fadd_rn(v[e], p.bias[e]) : v[e];
        }
      }
      if (p.has_gate) p.gate_out[row] = v[GC];
      return;
    }
    if (p.ep == 8) route_row<8, NV, GC>(p, v, row);
    else route_row<16, NV, GC>(p, v, row);
  } else if constexpr (TR::red) {
    // weight-gradient tiles are always whole: bulk stores of 32 x 32 fp32
    const bool empty = t.rows <= 0;
    const int y = t.g * p.M_fixed + t.m * BM + q * 32;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      float v[32];
      tmem_ld32(tbase + c * 32, v);
      if (empty) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.0f;
      }
      uint32_t w[32];
      pack_f32(v, w);
      uint8_t *b = stage_begin(sg, lane);
      stage_row(b, lane, w);
      stage_store(b, &p.tmO0, t.n * BN + c * 32, y, lane);
    }
  } else if (t.rows - t.m * BM - q * 32 >= 32) {
    // this warp's 32 rows all belong to the group: bulk stores (rows past
    // the group would belong to the next group, so a warp whose rows cross
    // the group's end takes the row-store path below)
    const int y = t.row0 + t.m * BM + q * 32;
    if constexpr (MODE == GU) {
      const bool save = p.out1 != nullptr;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {  // 64 gate/up columns per chunk
        uint32_t wh[32], wg[32], wu[32];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float g[32], u[32], h[32];
          tmem_ld32x2(tbase + c * 64 + hh * 32, tbase + 128 + c * 64 + hh * 32, g, u);
          if (save) {
            pack_bf16(g, wg, hh * 16);
            pack_bf16(u, wu, hh * 16);
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) h[i] = g[i] * sigmoid_fast(g[i]) * u[i];
          pack_bf16(h, wh, hh * 16);
        }
        uint8_t *b = stage_begin(sg, lane);
        stage_row(b, lane, wh);
        stage_store(b, &p.tmO0, t.n * 128 + c * 64, y, lane);
        if (save) {   // A_save = [G | U]
          uint8_t *b2 = stage_begin(sg, lane);
          stage_row(b2, lane, wg);
          stage_store(b2, &p.tmO1, t.n * 128 + c * 64, y, lane);
          uint8_t *b3 = stage_begin(sg, lane);
          stage_row(b3, lane, wu);
          stage_store(b3, &p.tmO1, p.F + t.n * 128 + c * 64, y, lane);
        }
      }
    } else if constexpr (MODE == DOWN) {
#pragma unroll 1
      for (int c = 0; c < BN / 64; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v[32];
          tmem_ld32(tbase + c * 64 + hh * 32, v);
          pack_bf16(v, w, hh * 16);
        }
        uint8_t *b = stage_begin(sg, lane);
        stage_row(b, lane, w);
        stage_store(b, &p.tmO0, t.n * BN + c * 64, y, lane);
      }
    } else if constexpr (MODE == DX) {
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        tmem_ld32(tbase + c * 32, v);
        uint32_t w[32];
        pack_f32(v, w);
        uint8_t *b = stage_begin(sg, lane);
        stage_row(b, lane, w);
        stage_store(b, &p.tmO0, t.n * BN + c * 32, y, lane);
      }
    } else if constexpr (MODE == DH) {
      // per 64 columns: TMA-load this warp's 32 rows of G and U from
      // A_save into the two staging buffers, turn them into dG and dU in
      // place, bulk-store both halves of dA
      uint8_t *bg = sg.base, *bu = sg.base + kStageOutBytes;
      const uint32_t ebar = smem_u32(&st.ebar[warp - 2]);
      bool ok = true;
#pragma unroll 1
      for (int c = 0; c < BN / 64 && ok; ++c) {
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_expect_tx(ebar, 2 * kStageOutBytes);
          tma_load_2d(smem_u32(bg), &p.tmO1, ebar, t.n * BN + c * 64, y);
          tma_load_2d(smem_u32(bu), &p.tmO1, ebar, p.F + t.n * BN + c * 64, y);
        }
        ok = __all_sync(0xffffffffu, wait_bounded(st, ebar, ephase, p.status, 5));
        ephase ^= 1;
        if (!ok) break;
        uint8_t *rg = bg + lane * 128, *ru = bu + lane * 128;
        // 32 columns per pass, the loop over the two passes kept rolled: a
        // short loop body keeps the epilogue's instruction footprint small
        // next to the producer and MMA warps that share the instruction cache
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          float dh[32];
          tmem_ld32(tbase + c * 64 + hh * 32, dh);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {   // 16-byte chunk ch = columns 8ch..8ch+7
            const int off = ((hh * 4 + cc) ^ (lane & 7)) << 4;
            float G[8], U[8], dG[8], dU[8];
            load16<__nv_bfloat16>(reinterpret_cast<const __nv_bfloat16 *>(rg + off), G);
            load16<__nv_bfloat16>(reinterpret_cast<const __nv_bfloat16 *>(ru + off), U);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float sgm = sigmoid_fast(G[j]);
              const float dhv = dh[8 * cc + j];
              dG[j] = dhv * U[j] * sgm * (1.0f + G[j] * (1.0f - sgm));
              dU[j] = dhv * G[j] * sgm;
            }
            store16<__nv_bfloat16>(reinterpret_cast<__nv_bfloat16 *>(rg + off), dG);
            store16<__nv_bfloat16>(reinterpret_cast<__nv_bfloat16 *>(ru + off), dU);
          }
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                           reinterpret_cast<uint64_t>(&p.tmO0)),
                       "r"(smem_u32(bg)), "r"(t.n * BN + c * 64), "r"(y)
                       : "memory");
          asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                           reinterpret_cast<uint64_t>(&p.tmO0)),
                       "r"(smem_u32(bu)), "r"(p.F + t.n * BN + c * 64), "r"(y)
                       : "memory");
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
      }
    }
  } else if (t.rows - t.m * BM - q * 32 > 0) {
    const bool valid = r_loc < t.rows;
    const int64_t row = (int64_t)t.row0 + r_loc;
    if constexpr (MODE == GU) {
      __nv_bfloat16 *H = reinterpret_cast<__nv_bfloat16 *>(p.out0) + row * p.F + t.n * 128;
      __nv_bfloat16 *As = reinterpret_cast<__nv_bfloat16 *>(p.out1);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float g[32], u[32];
        tmem_ld32(tbase + c * 32, g);
        tmem_ld32(tbase + 128 + c * 32, u);
        if (valid) {
          float h[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) h[i] = g[i] * sigmoid_fast(g[i]) * u[i];
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            store16<__nv_bfloat16>(H + c * 32 + i, *reinterpret_cast<float(*)[8]>(h + i));
          }
          if (As != nullptr) {
            __nv_bfloat16 *ag = As + row * 2 * p.F + t.n * 128 + c * 32;
            __nv_bfloat16 *au = ag + p.F;
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              store16<__nv_bfloat16>(ag + i, *reinterpret_cast<float(*)[8]>(g + i));
              store16<__nv_bfloat16>(au + i, *reinterpret_cast<float(*)[8]>(u + i));
            }
          }
        }
      }
    } else if constexpr (MODE == DOWN) {
      __nv_bfloat16 *Y = reinterpret_cast<__nv_bfloat16 *>(p.out0) + row * p.N + t.n * BN;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        tmem_ld32(tbase + c * 32, v);
        if (valid) {
#pragma unroll
          for (int i = 0; i < 32; i += 8)
            store16<__nv_bfloat16>(Y + c * 32 + i, *reinterpret_cast<float(*)[8]>(v + i));
        }
      }
    } else if constexpr (MODE == DH) {
      const __nv_bfloat16 *As = reinterpret_cast<const __nv_bfloat16 *>(p.aux) + row * 2 * p.F + t.n * BN;
      __nv_bfloat16 *dA = reinterpret_cast<__nv_bfloat16 *>(p.out0) + row * 2 * p.F + t.n * BN;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        float dh[32];
        tmem_ld32(tbase + c * 32, dh);
        if (valid) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            float G[8], U[8], dG[8], dU[8];
            load16<__nv_bfloat16>(As + c * 32 + i, G);
            load16<__nv_bfloat16>(As + p.F + c * 32 + i, U);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float sg = sigmoid_fast(G[j]);
              dG[j] = dh[i + j] * U[j] * sg * (1.0f + G[j] * (1.0f - sg));
              dU[j] = dh[i + j] * G[j] * sg;
            }
            store16<__nv_bfloat16>(dA + c * 32 + i, dG);
            store16<__nv_bfloat16>(dA + p.F + c * 32 + i, dU);
          }
        }
      }
    } else {  // DX
      float *o = reinterpret_cast<float *>(p.out0) + row * p.N + t.n * BN;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        tmem_ld32(tbase + c * 32, v);
        if (valid) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4 *>(o + c * 32 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        }
      }
    }
  }
}

template <int MODE, int BN>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
  using TR = ModeTraits<MODE>;
  constexpr int MMA_N = (MODE == GU) ? 256 : BN;
  constexpr int B_BOXES = TR::b_mn ? MMA_N / 64 : (MMA_N >= 128 ? MMA_N / 128 : 1);
  constexpr int A_BOXES = TR::a_mn ? BM / 64 : 1;
  constexpr uint32_t kStageTx = kABytes + MMA_N * BK * 2;
  constexpr uint32_t kIdesc = instr_desc(BM, MMA_N, TR::a_mn, TR::b_mn);
  // the router's B operand is at most 80 rows (10 KB): six stages of 16 KB
  // of x and the B rows (rounded to 1 KB, the 128-byte swizzle atom) keep more
  // of x in flight; the space after the ring holds the K-split exchange
  constexpr int NST = MODE == RT ? 6 : kStages;
  constexpr int SBYTES = MODE == RT ? kABytes + (BN * BK * 2 + 1023) / 1024 * 1024 : kStageBytes;
  static_assert(NST * SBYTES <= kStages * kStageBytes && NST <= kMaxStages, "ring too large");
  static_assert(MODE != RT || BN * BK * 2 <= 16384, "router B operand exceeds its stage");

  // the router's Top-K kernel is launched as a programmatic dependent: it
  // may be scheduled now and waits (griddepcontrol.wait) for this grid
  if constexpr (MODE == RT) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *staging = smem + kStages * kStageBytes;
  SharedState &st = *reinterpret_cast<SharedState *>(staging + kEpiStagingBytes);
  float *xbuf = reinterpret_cast<float *>(smem + NST * SBYTES);   // RT K-split exchange
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool clustered = MODE == RT && p.k_split > 1;

  // ---- set-up: tile table, barriers, TMEM
  if (threadIdx.x == 0) {
    st.abort = 0;
    int total = 0;
    bool bad = false;
    if constexpr (MODE == RT) {
      mbar_init(smem_u32(&st.xbar), (uint32_t)(p.k_split > 1 ? (p.k_split - 1) * BM : 1));
      total = (int)((p.T + BM - 1) / BM) * p.k_split;
    } else if constexpr (TR::red) {
      for (int g = 0; g < p.n_groups; ++g)
        if (p.offsets[g + 1] < p.offsets[g]) bad = true;
      total = p.n_groups * (p.M_fixed / BM) * (p.N / BN);
    } else {
      const int NT = p.N / (MODE == GU ? 128 : BN);
      for (int g = 0; g < p.n_groups; ++g) {
        const int rows = p.offsets[g + 1] - p.offsets[g];
        if (rows < 0) bad = true;
        int mt = rows > 0 ? (rows + BM - 1) / BM : 0;
        st.mbase[g] = 0;
        if (p.tail_mode == 2) {   // only the half-tile tail: the 128 rows after the full pairs
          mt = half_tail(rows) ? 1 : 0;
          st.mbase[g] = rows > 0 ? (rows / 256) * 2 : 0;
        }
        st.tile_start[g] = total;
        st.mtiles[g] = mt > 0 ? mt : 1;
        total += mt * NT;
      }
      st.tile_start[p.n_groups] = total;
    }
    if constexpr (MODE != RT) {
      if (p.offsets[0] < 0 || (int64_t)p.offsets[p.n_groups] > p.max_rows) bad = true;
    }
    if (bad) {
      report(p.status, MOE_ERR_DEVICE, kInfoOffsets);
      total = 0;
    }
    st.total_tiles = total;
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&st.full[s]), 1);
      mbar_init(smem_u32(&st.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&st.tfull[b]), 1);
      mbar_init(smem_u32(&st.tempty[b]), 4);
    }
    mbar_init(smem_u32(&st.drain), 1);
    for (int w = 0; w < 4; ++w) mbar_init(smem_u32(&st.ebar[w]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&st.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  if (clustered) cluster_sync();   // the even CTA's exchange barrier exists before any arrival
  tc_fence_after();
  const uint32_t tmem = st.tmem_base;
  const int total = st.total_tiles;

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0 && !p.fault_stall) {
      int it = 0;
      int last_phase[NST];
#pragma unroll
      for (int s = 0; s < NST; ++s) last_phase[s] = -1;
      for (int ti = blockIdx.x; ti < total && !st.abort; ti += gridDim.x) {
        const Tile t = decode_tile<MODE, BN>(p, st, ti);
        int kblocks = TR::red ? (t.rows + BK - 1) / BK : p.K_fixed / BK;
        int kb0 = 0;   // first K block of the tile (the router's K split)
        if constexpr (MODE == RT) {
          kb0 = t.n * p.kb_per;
          kblocks = min(p.kb_per, kblocks - kb0);
        }
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % NST;
          const uint32_t ph = (it / NST) & 1;
          if (!wait_bounded(st, smem_u32(&st.empty[s]), ph ^ 1, p.status, 1)) break;
          const uint32_t full = smem_u32(&st.full[s]);
          mbar_expect_tx(full, kStageTx);
          last_phase[s] = (int)ph;
          const uint32_t sa = smem_u32(smem + s * SBYTES);
          const uint32_t sb = sa + kABytes;
          if constexpr (TR::red) {   // K rows relative to the group's own maps
            const CUtensorMap *mA = p.gmaps + 2 * t.g, *mB = mA + 1;
            if (kb == 0) {
              tensormap_acquire(mA);
              tensormap_acquire(mB);
            }
#pragma unroll
            for (int b = 0; b < A_BOXES; ++b)
              tma_load_2d(sa + b * 8192, mA, full, t.m * BM + 64 * b, kb * BK);
#pragma unroll
            for (int b = 0; b < B_BOXES; ++b)
              tma_load_2d(sb + b * 8192, mB, full, t.n * BN + 64 * b, kb * BK);
          } else {
            const int arow = t.row0 + t.m * BM;
            tma_load_2d(sa, &p.tmA, full, (kb0 + kb) * BK, arow);
            const int64_t gb = (int64_t)t.g * p.b_group_rows;
            if constexpr (MODE == RT) {
              tma_load_2d(sb, &p.tmB, full, (kb0 + kb) * BK, 0);
              if (p.has_gate) tma_load_2d(sb + p.e_pad * 128, &p.tmC, full, (kb0 + kb) * BK, 0);
            } else if constexpr (MODE == GU) {
              tma_load_2d(sb, &p.tmB, full, kb * BK, (int)(gb + t.n * 128));
              tma_load_2d(sb + 16384, &p.tmB, full, kb * BK, (int)(gb + p.F + t.n * 128));
            } else if constexpr (TR::b_mn) {
#pragma unroll
              for (int b = 0; b < B_BOXES; ++b)
                tma_load_2d(sb + b * 8192, &p.tmB, full, t.n * BN + 64 * b, (int)(gb + kb * BK));
            } else {
#pragma unroll
              for (int b = 0; b < B_BOXES; ++b)
                tma_load_2d(sb + b * 16384, &p.tmB, full, kb * BK, (int)(gb + t.n * BN + 128 * b));
            }
          }
        }
      }
      // drain: every issued load must land before the CTA exits
      for (int s = 0; s < NST; ++s)
        if (last_phase[s] >= 0) {
          const uint32_t bar = smem_u32(&st.full[s]);
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(bar, (uint32_t)last_phase[s]) && globaltimer() - t0 < kTimeoutNs) {
          }
        }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    int it = 0, tcount = 0;
    bool issued_any = false;
    for (int ti = blockIdx.x; ti < total && !st.abort; ti += gridDim.x, ++tcount) {
      const Tile t = decode_tile<MODE, BN>(p, st, ti);
      int kblocks = TR::red ? (t.rows + BK - 1) / BK : p.K_fixed / BK;
      if constexpr (MODE == RT) kblocks = min(p.kb_per, kblocks - t.n * p.kb_per);
      const int buf = tcount & 1;
      const uint32_t use = (tcount >> 1) & 1;
      if (!__all_sync(0xffffffffu, wait_bounded(st, smem_u32(&st.tempty[buf]), use ^ 1, p.status, 2))) break;
      tc_fence_after();
      const uint32_t dcol = tmem + buf * 256;
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb, ++it) {
        const int s = it % NST;
        const uint32_t ph = (it / NST) & 1;
        if (!__all_sync(0xffffffffu, wait_bounded(st, smem_u32(&st.full[s]), ph, p.status, 3))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint8_t *sa_p = smem + s * SBYTES;
        if (lane == 0) {
          const uint32_t sa = smem_u32(sa_p);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            uint64_t ad, bd;
            if constexpr (TR::a_mn) ad = smem_desc(sa + ks * 2048, 8192, 1024);
            else ad = smem_desc(sa + ks * 32, 16, 1024);
            if constexpr (TR::b_mn) bd = smem_desc(sb + ks * 2048, 8192, 1024);
            else bd = smem_desc(sb + ks * 32, 16, 1024);
            tc_mma(dcol, ad, bd, kIdesc, (kb > 0 || ks > 0) ? 1u : 0u);
          }
          tc_commit(smem_u32(&st.empty[s]));
          issued_any = true;
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc_commit(smem_u32(&st.tfull[buf]));
      __syncwarp();
    }
    // drain: all issued MMAs complete before TMEM is released
    if (lane == 0 && issued_any) {
      tc_commit(smem_u32(&st.drain));
      const uint32_t bar = smem_u32(&st.drain);
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(bar, 0) && globaltimer() - t0 < kTimeoutNs) {
      }
    }
    __syncwarp();
  } else {
    // ======================= epilogue =======================
    const int q = warp & 3;  // TMEM lane quarter of this warp
    Stager sg{staging + (warp - 2) * 2 * kStageOutBytes, 0};
    uint32_t ephase = 0;  // DH: parity of this warp's A_save load barrier
    int tcount = 0;
    for (int ti = blockIdx.x; ti < total && !st.abort; ti += gridDim.x, ++tcount) {
      const Tile t = decode_tile<MODE, BN>(p, st, ti);
      const int buf = tcount & 1;
      const uint32_t use = (tcount >> 1) & 1;
      if (!__all_sync(0xffffffffu, wait_bounded(st, smem_u32(&st.tfull[buf]), use, p.status, 4))) break;
      tc_fence_after();
      const uint32_t tbase = tmem + buf * 256 + ((uint32_t)(q * 32) << 16);
      epilogue_tile<MODE, BN>(p, st, sg, ephase, t, tbase, q, warp, lane, xbuf);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&st.tempty[buf]));
    }
    // every bulk store has finished before the CTA's shared memory goes away
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (clustered) cluster_sync();   // no CTA leaves while another may still write to it
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
  // tail kernel: complete only after the pair kernel it followed, so that
  // whatever the stream runs next sees the rows of both
  if (p.tail_mode == 2) asm volatile("griddepcontrol.wait;" ::: "memory");
}


// ---------------------------------------------------------------------------
// CTA-pair variant of the row-grouped modes (GU, DOWN, DH, DX): a cluster of
// two CTAs computes a 256-row tile. Each CTA holds its own 128 rows of A and
// half of B's columns; the even CTA issues M=256 tcgen05.mma.cta_group::2,
// which reads both halves and writes each CTA's 128 accumulator rows into
// that CTA's TMEM. Per SM this halves the B operand traffic per FLOP, so a
// 6-stage ring of 32 KB stages covers more latency at a lower data rate.
//   producer (both CTAs): own A box + own B half, completing on the even
//     CTA's full barrier (which expects both CTAs' bytes);
//   MMA (even CTA only): commits multicast to both CTAs' empty / tfull;
//   epilogue (both CTAs): own TMEM rows, then arrive on the even CTA's tempty
//     (8 arrivals: 4 warps x 2 CTAs).
// NSUB = 2: a pair tile covers two adjacent N tiles that share the A
// operand (one A box and two B boxes per stage, 48 KB, 4 stages), one TMEM
// accumulator each. Less shared memory per unit of MMA work, so the same
// ring bytes cover a longer load latency; the two accumulators are the two
// TMEM buffers, so the epilogue no longer overlaps the next tile's mainloop
// (used where the epilogue is short).
template <int NSUB> constexpr int pair_stages() { return NSUB == 1 ? 6 : 4; }
template <int NSUB> constexpr int pair_stage_bytes() { return kABytes + NSUB * 16384; }

template <int MODE, int BN, int NSUB = 1>
__device__ __forceinline__ Tile decode_pair_tile(const TcParams &p, const SharedState &st, int pt,
                                                 int rank) {
  Tile t;
  if constexpr (ModeTraits<MODE>::red) {
    const int MT2 = p.M_fixed / 256, NT = p.N / BN / NSUB;
    t.g = pt / (MT2 * NT);
    const int loc = pt % (MT2 * NT);
    t.n = (loc / MT2) * NSUB;
    t.m = 2 * (loc % MT2) + rank;
    t.row0 = p.offsets[t.g];
    t.rows = p.offsets[t.g + 1] - t.row0;
  } else {
    t = decode_tile<MODE, BN>(p, st, pt);
    t.m = 2 * t.m + rank;
    t.n *= NSUB;   // first of the tile's NSUB N tiles
  }
  return t;
}

template <int MODE, int BN, int NSUB, bool GATHER>
__global__ void __launch_bounds__(GATHER ? kThreadsGather : kThreads, 1)
    tc_gemm_pair_kernel(const __grid_constant__ TcParams p) {
  static_assert(MODE != RT, "the router GEMM runs single-CTA");
  static_assert(!GATHER || MODE == GU, "the A gather serves the gate/up GEMM");
  using TR = ModeTraits<MODE>;
  constexpr int kPairStages = pair_stages<NSUB>();
  constexpr int kPairStageBytes = pair_stage_bytes<NSUB>();
  constexpr int MMA_N = (MODE == GU) ? 256 : BN;
  constexpr int HALF_N = MMA_N / 2;
  static_assert(NSUB == 1 || HALF_N * BK * 2 == 16384, "two B halves of 16 KB per stage");
  constexpr int A_BOXES = TR::a_mn ? BM / 64 : 1;
  constexpr int B_HALF_BOXES = TR::b_mn ? HALF_N / 64 : 1;
  // one CTA's TMA bytes per stage (the gathered A arrives by cp.async instead)
  constexpr uint32_t kOwnTx = (GATHER ? 0 : kABytes) + NSUB * HALF_N * BK * 2;
  constexpr uint32_t kTx = 2u * kOwnTx;
  constexpr uint32_t kIdesc = instr_desc(256, MMA_N, TR::a_mn, TR::b_mn);

  // the tail kernel (single-CTA, half-empty last tiles) may launch now: its
  // CTAs take SMs as this grid's CTAs leave
  if (p.tail_mode == 1) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *staging = smem + kPairStages * kPairStageBytes;
  SharedState &st = *reinterpret_cast<SharedState *>(staging + kEpiStagingBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    st.abort = 0;
    int total = 0;
    bool bad = false;
    if constexpr (TR::red) {
      for (int g = 0; g < p.n_groups; ++g)
        if (p.offsets[g + 1] < p.offsets[g]) bad = true;
      total = p.n_groups * (p.M_fixed / 256) * (p.N / BN / NSUB);   // 256-row pair tiles
    } else {
      const int NT = p.N / (MODE == GU ? 128 : BN) / NSUB;
      for (int g = 0; g < p.n_groups; ++g) {
        const int rows = p.offsets[g + 1] - p.offsets[g];
        if (rows < 0) bad = true;
        int mt = rows > 0 ? (rows + 255) / 256 : 0;   // 256-row pair tiles
        if (p.tail_mode == 1 && half_tail(rows)) --mt;  // the tail kernel takes it
        st.tile_start[g] = total;
        st.mtiles[g] = mt > 0 ? mt : 1;
        st.mbase[g] = 0;
        total += mt * NT;
      }
      st.tile_start[p.n_groups] = total;
    }
    if (p.offsets[0] < 0 || (int64_t)p.offsets[p.n_groups] > p.max_rows) bad = true;
    if (bad) {
      report(p.status, MOE_ERR_DEVICE, kInfoOffsets);
      total = 0;
    }
    st.total_tiles = total;
    for (int i = 0; i < kPairStages; ++i) {
      // GATHER: + one arrival per gather warp of each CTA (with its row bytes)
      mbar_init(smem_u32(&st.full[i]), GATHER ? 1 + 2 * kGatherWarps : 1);
      mbar_init(smem_u32(&st.empty[i]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&st.tfull[b]), 1);
      mbar_init(smem_u32(&st.tempty[b]), 8);
    }
    mbar_init(smem_u32(&st.drain), 1);
    for (int w = 0; w < 4; ++w) mbar_init(smem_u32(&st.ebar[w]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&st.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers initialised before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem = st.tmem_base;
  const int total = st.total_tiles;

  if (warp == 0) {
    // ======================= TMA producer (both CTAs) =======================
    if (lane == 0 && !p.fault_stall) {
      int it = 0;
      int last_phase[kPairStages];
#pragma unroll
      for (int i = 0; i < kPairStages; ++i) last_phase[i] = -1;
      for (int pt = cid; pt < total && !st.abort; pt += ncl) {
        const Tile t = decode_pair_tile<MODE, BN, NSUB>(p, st, pt, (int)rank);
        const int kblocks = TR::red ? (t.rows + BK - 1) / BK : p.K_fixed / BK;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % kPairStages;
          const uint32_t ph = (it / kPairStages) & 1;
          if (!wait_bounded(st, smem_u32(&st.empty[s]), ph ^ 1, p.status, 1)) break;
          const uint32_t sa = smem_u32(smem + s * kPairStageBytes);
          const uint32_t sb = sa + kABytes;
          // both CTAs' bytes complete on the even CTA's full barrier
          const uint32_t bar = map_to_cta(smem_u32(&st.full[s]), 0);
          if (leader) {
            mbar_expect_tx(smem_u32(&st.full[s]), kTx);
            last_phase[s] = (int)ph;
          }
          if constexpr (TR::red) {   // K rows relative to the group's own maps
            const CUtensorMap *mA = p.gmaps + 2 * t.g, *mB = mA + 1;
            if (kb == 0) {
              tensormap_acquire(mA);
              tensormap_acquire(mB);
            }
#pragma unroll
            for (int b = 0; b < A_BOXES; ++b)
              tma_load_2d_pair(sa + b * 8192, mA, bar, t.m * BM + 64 * b, kb * BK);
#pragma unroll
            for (int j = 0; j < NSUB; ++j)
#pragma unroll
              for (int b = 0; b < B_HALF_BOXES; ++b)
                tma_load_2d_pair(sb + j * 16384 + b * 8192, mB, bar,
                                 (t.n + j) * BN + (int)rank * HALF_N + 64 * b, kb * BK);
          } else {
            if constexpr (!GATHER) tma_load_2d_pair(sa, &p.tmA, bar, kb * BK, t.row0 + t.m * BM);
            const int64_t gb = (int64_t)t.g * p.b_group_rows;
#pragma unroll
            for (int j = 0; j < NSUB; ++j) {   // B half of each of the tile's N tiles
              const uint32_t sbj = sb + j * 16384;
              const int n = t.n + j;
              if constexpr (MODE == GU) {   // even CTA: gate rows, odd CTA: up rows
                tma_load_2d_pair(sbj, &p.tmB, bar, kb * BK, (int)(gb + (int64_t)rank * p.F + n * 128));
              } else if constexpr (TR::b_mn) {
#pragma unroll
                for (int b = 0; b < B_HALF_BOXES; ++b)
                  tma_load_2d_pair(sbj + b * 8192, &p.tmB, bar,
                                   n * BN + (int)rank * HALF_N + 64 * b, (int)(gb + kb * BK));
              } else {
                tma_load_2d_pair(sbj, &p.tmB, bar, kb * BK, (int)(gb + n * BN + (int)rank * HALF_N));
              }
            }
          }
        }
      }
      // wait (bounded) for the copies still in flight: the even CTA's full
      // barriers see the loads of both CTAs land
      for (int i = 0; i < kPairStages; ++i) {
        if (leader && last_phase[i] >= 0) {
          const uint32_t b = smem_u32(&st.full[i]);
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(b, (uint32_t)last_phase[i]) && globaltimer() - t0 < kTimeoutNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (leader) {
      // ======================= MMA issuer (even CTA) =======================
      int it = 0, tcount = 0;
      bool issued_any = false;
      for (int pt = cid; pt < total && !st.abort; pt += ncl, ++tcount) {
        const Tile t = decode_pair_tile<MODE, BN, NSUB>(p, st, pt, 0);
        const int kblocks = TR::red ? (t.rows + BK - 1) / BK : p.K_fixed / BK;
        // NSUB = 1: the two TMEM buffers alternate between tiles; NSUB = 2:
        // every tile uses both (buffer j for its j-th N tile)
        const int buf = NSUB == 1 ? (tcount & 1) : 0;
        const uint32_t use = NSUB == 1 ? ((tcount >> 1) & 1) : (tcount & 1);
        // NSUB = 2: the epilogue drains the tile's two accumulators in order,
        // so accumulator 0's MMAs for the stages already loaded (up to the
        // ring's depth) go ahead while accumulator 1 is still being read; then
        // accumulator 1's MMAs for those stages, which releases them
        const int look = NSUB == 2 ? min(kblocks, kPairStages) : 0;
        if (!__all_sync(0xffffffffu, wait_bounded(st, smem_u32(&st.tempty[buf]), use ^ 1, p.status, 2)))
          break;
        tc_fence_after();
        const uint32_t dcol = tmem + buf * 256;
        bool ok = true;
        if constexpr (NSUB == 2) {
          for (int kb = 0; kb < look; ++kb) {
            const int s = (it + kb) % kPairStages;
            const uint32_t ph = ((it + kb) / kPairStages) & 1;
            if (!__all_sync(0xffffffffu, wait_bounded(st, smem_u32(&st.full[s]), ph, p.status, 3))) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (lane == 0) {
              const uint32_t sa = smem_u32(smem + s * kPairStageBytes);
              const uint32_t sb = sa + kABytes;
#pragma unroll
              for (int ks = 0; ks < BK / 16; ++ks) {
                uint64_t ad, bd;
                if constexpr (TR::a_mn) ad = smem_desc(sa + ks * 2048, 8192, 1024);
                else ad = smem_desc(sa + ks * 32, 16, 1024);
                if constexpr (TR::b_mn) bd = smem_desc(sb + ks * 2048, 8192, 1024);
                else bd = smem_desc(sb + ks * 32, 16, 1024);
                tc_mma_pair(dcol, ad, bd, kIdesc, (kb > 0 || ks > 0) ? 1u : 0u);
              }
            }
            __syncwarp();
          }
          if (!ok) break;
          if (!__all_sync(0xffffffffu, wait_bounded(st, smem_u32(&st.tempty[buf + 1]), use ^ 1, p.status, 2)))
            break;
          tc_fence_after();
          for (int kb = 0; kb < look; ++kb, ++it) {
            const int s = it % kPairStages;
            if (lane == 0) {
              const uint32_t sa = smem_u32(smem + s * kPairStageBytes);
              const uint32_t sb = sa + kABytes + 16384;
#pragma unroll
              for (int ks = 0; ks < BK / 16; ++ks) {
                uint64_t ad, bd;
                if constexpr (TR::a_mn) ad = smem_desc(sa + ks * 2048, 8192, 1024);
                else ad = smem_desc(sa + ks * 32, 16, 1024);
                if constexpr (TR::b_mn) bd = smem_desc(sb + ks * 2048, 8192, 1024);
                else bd = smem_desc(sb + ks * 32, 16, 1024);
                tc_mma_pair(dcol + 256, ad, bd, kIdesc, (kb > 0 || ks > 0) ? 1u : 0u);
              }
              tc_commit_pair_both(smem_u32(&st.empty[s]));
              issued_any = true;
            }
            __syncwarp();
          }
        }
        for (int kb = look; kb < kblocks; ++kb, ++it) {
          const int s = it % kPairStages;
          const uint32_t ph = (it / kPairStages) & 1;
          if (!__all_sync(0xffffffffu, wait_bounded(st, smem_u32(&st.full[s]), ph, p.status, 3))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t sa = smem_u32(smem + s * kPairStageBytes);
            const uint32_t sb = sa + kABytes;
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks) {
              uint64_t ad, bd;
              if constexpr (TR::a_mn) ad = smem_desc(sa + ks * 2048, 8192, 1024);
              else ad = smem_desc(sa + ks * 32, 16, 1024);
#pragma unroll
              for (int j = 0; j < NSUB; ++j) {
                const uint32_t sbj = sb + j * 16384;
                if constexpr (TR::b_mn) bd = smem_desc(sbj + ks * 2048, 8192, 1024);
                else bd = smem_desc(sbj + ks * 32, 16, 1024);
                tc_mma_pair(dcol + j * 256, ad, bd, kIdesc, (kb > 0 || ks > 0) ? 1u : 0u);
              }
            }
            tc_commit_pair_both(smem_u32(&st.empty[s]));
            issued_any = true;
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) {
#pragma unroll
          for (int j = 0; j < NSUB; ++j) tc_commit_pair_both(smem_u32(&st.tfull[buf + j]));
        }
        __syncwarp();
      }
      if (lane == 0 && issued_any) {
        tc_commit_pair_local(smem_u32(&st.drain));
        const uint32_t bar = smem_u32(&st.drain);
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(bar, 0) && globaltimer() - t0 < kTimeoutNs) {
        }
      }
      __syncwarp();
    }
  } else if (warp < 6) {
    // ======================= epilogue (both CTAs) =======================
    const int q = warp & 3;
    Stager sg{staging + (warp - 2) * 2 * kStageOutBytes, 0};
    uint32_t ephase = 0;
    int tcount = 0;
    bool stop = false;
    for (int pt = cid; pt < total && !st.abort && !stop; pt += ncl, ++tcount) {
      const Tile t0 = decode_pair_tile<MODE, BN, NSUB>(p, st, pt, (int)rank);
#pragma unroll 1
      for (int j = 0; j < NSUB; ++j) {   // the tile's N tiles, one TMEM buffer each
        const int buf = NSUB == 1 ? (tcount & 1) : j;
        const uint32_t use = NSUB == 1 ? ((tcount >> 1) & 1) : (tcount & 1);
        if (!__all_sync(0xffffffffu, wait_bounded(st, smem_u32(&st.tfull[buf]), use, p.status, 4))) {
          stop = true;
          break;
        }
        tc_fence_after();
        Tile t = t0;
        t.n = t0.n + j;
        const uint32_t tbase = tmem + buf * 256 + ((uint32_t)(q * 32) << 16);
        epilogue_tile<MODE, BN>(p, st, sg, ephase, t, tbase, q, warp, lane);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(map_to_cta(smem_u32(&st.tempty[buf]), 0));
      }
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
  } else if constexpr (GATHER) {
    // ==================== A gather (GU, both CTAs) ====================
    // Lane l < 16 of gather warp w loads rows r = 64 w + 4 l .. r + 3 of this
    // CTA's 128-row A box: per stage one tile::gather4 copy, four boxes of
    // one row and 64 columns of x (128 bytes each) put at byte offset 128 r
    // of the stage, one after another, which is where the 128-byte swizzled
    // box the MMA descriptor reads keeps rows r .. r + 3 (the swizzle is
    // anchored to the shared-memory address, and the stage is 1024-byte
    // aligned). A row without a source (past the last group, or a padding
    // row) loads row -1: outside x, so the copy fills zeros. The copies
    // complete on the even CTA's full barrier, on which lane 0 first arrives
    // with the warp's 64 rows of bytes; the TMA completion orders the writes
    // for the tensor core.
    constexpr int kLanes = BM / (4 * kGatherWarps);   // 16 lanes of 4 rows per warp
    const int gw = warp - 6;
    const int64_t n_rows = p.offsets[p.n_groups];
    const int64_t n_src = p.gT * p.gK;
    int it = 0;
    for (int pt = cid; pt < total && !st.abort; pt += ncl) {
      const Tile t = decode_pair_tile<MODE, BN, NSUB>(p, st, pt, (int)rank);
      int tok[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t R = (int64_t)t.row0 + (int64_t)t.m * BM + 64 * gw + 4 * lane + j;
        tok[j] = -1;
        if (lane < kLanes && R < n_rows) {
          const int32_t so = p.src_of[R];
          if (so >= 0 && so < n_src) tok[j] = so / p.gK;
          else if (so >= 0) report(p.status, MOE_ERR_DEVICE, kInfoRowRange);
        }
      }
      const int kblocks = p.K_fixed / BK;
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb, ++it) {
        const int s = it % kPairStages;
        const uint32_t ph = (it / kPairStages) & 1;
        const uint32_t bar = map_to_cta(smem_u32(&st.full[s]), 0);
        bool w = true;
        if (lane == 0) {
          w = wait_bounded(st, smem_u32(&st.empty[s]), ph ^ 1, p.status, 6);
          if (w) mbar_arrive_expect_tx_cluster(bar, 4 * kLanes * 128);
        }
        if (!__shfl_sync(0xffffffffu, w, 0)) {
          ok = false;
          break;
        }
        if (lane < kLanes) {
          const uint32_t dst = smem_u32(smem + s * kPairStageBytes) + (64 * gw + 4 * lane) * 128;
          tma_gather4_pair(dst, &p.tmX, bar, kb * BK, tok[0], tok[1], tok[2], tok[3]);
        }
      }
      if (!ok) break;
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // no cross-CTA traffic after this point
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// Group tensor maps of the weight-gradient modes: thread g copies the two
// host-encoded templates (A and B over all rows) and points the copies at
// group g's first row with an outer extent of the group's row count, so a K
// block past the group's end is zero-filled by the TMA. An empty group gets
// an extent of 1 (its tiles load nothing). Offsets outside [0, max_rows] are
// reported by the GEMM kernel, which then loads nothing.
__global__ void group_maps_kernel(const __grid_constant__ CUtensorMap tA,
                                  const __grid_constant__ CUtensorMap tB, const int32_t *offsets,
                                  int n_groups, const uint8_t *a_base, int64_t a_row_bytes,
                                  const uint8_t *b_base, int64_t b_row_bytes, int64_t max_rows,
                                  CUtensorMap *out) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= n_groups) return;
  const int32_t lo = offsets[g], hi = offsets[g + 1];
  const bool sane = lo >= 0 && hi >= lo && hi <= max_rows;
  const int64_t row0 = sane ? lo : 0;
  const uint32_t rows = sane && hi > lo ? (uint32_t)(hi - lo) : 1u;
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    const uint4 *src = reinterpret_cast<const uint4 *>(w == 0 ? &tA : &tB);
    uint4 *dst = reinterpret_cast<uint4 *>(out + 2 * g + w);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(CUtensorMap) / sizeof(uint4)); ++i) dst[i] = src[i];
    const uint64_t addr =
        reinterpret_cast<uint64_t>(w == 0 ? a_base + row0 * a_row_bytes : b_base + row0 * b_row_bytes);
    asm volatile("tensormap.replace.tile.global_address.global.b1024.b64 [%0], %1;" ::"l"(dst),
                 "l"(addr)
                 : "memory");
    asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(dst),
                 "r"(rows)
                 : "memory");
  }
  asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
}

// ---------------------------------------------------------------------------
// host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    cudaDriverEntryPointQueryResult q;
    void *ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2D bf16 tensor [outer, inner] row-major (inner contiguous), box
// {64 inner, box_outer}, 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2D tensor [outer, inner] of 2- or 4-byte elements, for bulk stores: box of
// 128 bytes x 32 rows, 128-byte swizzle; writes outside the tensor are dropped.
bool make_store_map(CUtensorMap *m, void *base, int esize, uint64_t inner, uint64_t outer) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * (uint64_t)esize};
  cuuint32_t box[2] = {(cuuint32_t)(128 / esize), 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

constexpr size_t kSmemBytes = kStages * kStageBytes + kEpiStagingBytes + sizeof(SharedState) + 1024;

#ifdef MOE_TEST_HOOKS
// Test build only (libmoe_testhooks.so): fault injection for tests of the
// timeout path. With MOE_FAULT_INJECT_STALL=1 the producer warp issues no
// loads, so the MMA warp's first wait runs out; the kernel then records
// MOE_ERR_TIMEOUT and returns. Read at every launch.
int fault_stall() {
  const char *e = getenv("MOE_FAULT_INJECT_STALL");
  return (e != nullptr && e[0] == '1') ? 1 : 0;
}
#else
constexpr int fault_stall() { return 0; }
#endif

template <int MODE, int BN>
cudaError_t launch_mode(TcParams p, cudaStream_t s) {
  p.fault_stall = fault_stall();
  auto k = tc_gemm_kernel<MODE, BN>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  if (MODE == RT && p.k_split > 1) {
    // the K parts of a row tile run as one cluster (one row tile per cluster:
    // router_k_split keeps row tiles x parts within the SM count)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(num_sms() / p.k_split * p.k_split));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.k_split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, p);
  }
  if (p.tail_mode == 2) {   // programmatic dependent of the pair kernel before it
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)num_sms());
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, p);
  }
  k<<<num_sms(), kThreads, kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

template <int MODE, int BN, int NSUB = 1, bool GATHER = false>
cudaError_t launch_pair(TcParams p, cudaStream_t s) {
  p.fault_stall = fault_stall();
  auto k = tc_gemm_pair_kernel<MODE, BN, NSUB, GATHER>;
  constexpr size_t kPairSmemBytes = (size_t)pair_stages<NSUB>() * pair_stage_bytes<NSUB>() +
                                    kEpiStagingBytes + sizeof(SharedState) + 1024;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPairSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(num_sms() & ~1));
  cfg.blockDim = dim3(GATHER ? kThreadsGather : kThreads);
  cfg.dynamicSmemBytes = kPairSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, p);
}

// The row-grouped modes run as CTA pairs. In the test build
// (libmoe_testhooks.so) MOE_GEMM_PAIR=0, read once, selects the single-CTA
// kernels instead, so that tests can compare the two.
#ifdef MOE_TEST_HOOKS
bool pair_enabled() {
  static int v = -1;
  if (v < 0) {
    const char *e = getenv("MOE_GEMM_PAIR");
    v = (e != nullptr && e[0] == '0') ? 0 : 1;
  }
  return v == 1;
}
#else
constexpr bool pair_enabled() { return true; }
#endif

// Pair kernel, then (row-grouped modes) the single-CTA kernel for the groups'
// half-empty last tiles. The two write disjoint rows. The B tensor maps of the
// two kernels agree (128-row boxes for K-major B, 64 x 64 boxes for MN-major
// B) except for the down projection at BN = 128, which keeps its tails.
template <int MODE, int BN, int NSUB = 1>
cudaError_t launch_pair_and_tails(TcParams p, cudaStream_t s) {
  constexpr bool tails = MODE == GU || MODE == DH || MODE == DX || (MODE == DOWN && BN == 256);
  if constexpr (!tails) return launch_pair<MODE, BN, NSUB>(p, s);
  p.tail_mode = 1;
  cudaError_t e = launch_pair<MODE, BN, NSUB>(p, s);
  if (e != cudaSuccess) return e;
  p.tail_mode = 2;
  return launch_mode<MODE, BN>(p, s);
}

template <int MODE>
cudaError_t launch_bn(const TcParams &p, cudaStream_t s) {
  const bool bn256 = !(MODE == GU || p.N % 256 != 0);
  if constexpr (MODE != RT) {
    const bool red = (MODE == WGD || MODE == WGU);
    if (pair_enabled() && (!red || p.M_fixed % 256 == 0)) {
      // two N tiles per pair tile where the epilogue (no longer overlapped
      // with the next tile's mainloop) is short against a long K loop: the
      // down projection and dH with K >= 8192 (128 K blocks), dXp and
      // gate/up with K >= 4096. Measured A/B on one box: gate/up +2.0 % on
      // the Llama3-8x70B training step (K = 8192), +2.2 % on the
      // Mixtral-8x22B forward and +1.0 % on the G8T8 step (K = 6144), no gain
      // at K = 3584; dH +0.8 % on the Llama3 step (it lost 1.1 % there while
      // its sigmoid took a correctly rounded reciprocal) and a loss of 1 %
      // at K = 3584 and 6144; dXp's backward GEMMs -0.5 to -1.2 % at
      // K = 4096 and 5120
      if constexpr (MODE == DOWN || MODE == DX || MODE == DH)
        if (bn256 && (p.N / 256) % 2 == 0 && p.K_fixed >= (MODE == DX ? 4096 : 8192))
          return launch_pair_and_tails<MODE, 256, 2>(p, s);
      if constexpr (MODE == GU)
        if ((p.N / 128) % 2 == 0 && p.K_fixed >= 4096)
          return launch_pair_and_tails<GU, 128, 2>(p, s);
      if constexpr (red)   // K = a group's rows: the same test on the mean rows per group
        if (bn256 && (p.N / 256) % 2 == 0 && p.max_rows / p.n_groups >= 8192)
          return launch_pair<MODE, 256, 2>(p, s);
      return bn256 ? launch_pair_and_tails<MODE, 256>(p, s) : launch_pair_and_tails<MODE, 128>(p, s);
    }
  }
  return bn256 ? launch_mode<MODE, 256>(p, s) : launch_mode<MODE, 128>(p, s);
}

}  // namespace

int router_k_split(int64_t T, int d) {
  const int64_t mtiles = (T + BM - 1) / BM;
  const int kb = d / BK;
  int64_t s = mtiles > 0 ? num_sms() / mtiles : 1;
  if (s > kRouterMaxSplit) s = kRouterMaxSplit;
  if (s > kb / 8) s = kb / 8;   // at least 8 K blocks per split
  if (s < 1) s = 1;
  const int per = (int)((kb + s - 1) / s);
  return (kb + per - 1) / per;   // every split non-empty
}

constexpr int kRouteFuseMaxE = 16;   // the epilogue's routing serves E <= 16

// K parts of the router GEMM: as many as leave no SM idle (router_k_split),
// at most as many as the even CTA's exchange buffer (the shared memory after
// the ring) holds partial sums for
int router_parts(int64_t T, int d, int E, int has_gate) {
  const int n = (E + 15) / 16 * 16 + 16 * has_gate;
  const size_t stage = kABytes + ((size_t)n * BK * 2 + 1023) / 1024 * 1024;
  const size_t room = (size_t)kStages * kStageBytes + kEpiStagingBytes - 6 * stage;
  // each part's partial sums: BM rows of E (+ gate) floats, the row stride
  // rounded up to 4 floats
  const int max_parts = 1 + (int)(room / ((size_t)BM * ((E + has_gate + 3) & ~3) * sizeof(float)));
  const int split = router_k_split(T, d);
  return split < max_parts ? split : max_parts;
}

bool router_routes_in_epilogue(int64_t T, int d, int E, int has_gate) {
  return E <= kRouteFuseMaxE && router_parts(T, d, E, has_gate) == 1;
}

cudaError_t launch_router_tc(const RouteArgs &a, cudaStream_t s) {
  const int e_pad = (a.E + 15) / 16 * 16;
  const int has_gate = a.w_sg != nullptr ? 1 : 0;
  const int n = e_pad + 16 * has_gate;
  TcParams p{};
  if (!make_map(&p.tmA, a.x, a.d, a.T, 128)) return cudaErrorInvalidValue;
  if (!make_map(&p.tmB, a.W_r, a.d, a.E, e_pad)) return cudaErrorInvalidValue;
  if (has_gate && !make_map(&p.tmC, a.w_sg, a.d, 1, 16)) return cudaErrorInvalidValue;
  p.mode = RT; p.n_groups = 1; p.max_rows = a.T; p.d = a.d; p.K_fixed = a.d; p.N = n;
  p.T = a.T; p.E = a.E; p.e_pad = e_pad; p.has_gate = has_gate; p.bias = a.b_r;
  p.out0 = a.logits; p.gate_out = a.gate_logit; p.status = a.status;
  p.K = a.K; p.renorm = a.renorm;
  p.ep = 0;   // set below once the K split is known
  p.topk_idx = a.topk_idx; p.topk_prob = a.topk_prob; p.topk_w = a.topk_w; p.keep = a.keep;
  const int kb = a.d / BK;
  const int split = router_parts(a.T, a.d, a.E, has_gate);
  p.kb_per = (kb + split - 1) / split;
  p.k_split = (kb + p.kb_per - 1) / p.kb_per;   // every part non-empty
  // routing in the epilogue (one thread per token row) when the K loop is not
  // split and E is small; otherwise ep = 0: the logits alone, routed by the
  // Top-K kernel (a warp per token over every SM), which measured faster
  if (router_routes_in_epilogue(a.T, a.d, a.E, has_gate)) p.ep = a.E <= 8 ? 8 : 16;
  switch (n) {
    case 16: return launch_mode<RT, 16>(p, s);
    case 32: return launch_mode<RT, 32>(p, s);
    case 48: return launch_mode<RT, 48>(p, s);
    case 64: return launch_mode<RT, 64>(p, s);
    case 80: return launch_mode<RT, 80>(p, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_ffn_fwd_bf16(const FfnArgs &a, cudaStream_t s) {
  const int d = a.d, F = a.F, E = a.n_groups;
  const bool gather = a.x != nullptr;   // A rows gathered from x through src_of
  if (gather && !pair_enabled()) return cudaErrorNotSupported;
  void *H = a.H_save ? a.H_save : a.H_tmp;
  TcParams p{};
  p.n_groups = E; p.max_rows = a.max_rows; p.d = d; p.F = F; p.offsets = a.offsets;
  p.status = a.status;
  // GU
  if (!gather && !make_map(&p.tmA, a.Xp, d, a.max_rows, 128)) return cudaErrorInvalidValue;
  if (!make_map(&p.tmB, a.W_gu, d, (uint64_t)E * 2 * F, 128)) return cudaErrorInvalidValue;
  p.mode = GU; p.N = F; p.K_fixed = d; p.b_group_rows = 2 * (int64_t)F;
  p.out0 = H; p.out1 = a.A_save;
  if (!make_store_map(&p.tmO0, H, 2, F, a.max_rows)) return cudaErrorInvalidValue;
  if (a.A_save && !make_store_map(&p.tmO1, a.A_save, 2, 2 * (uint64_t)F, a.max_rows))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if (gather) {
    // one-row boxes of x: the gather warps load the permuted rows four at a
    // time (tile::gather4); two N tiles per pair tile under the same rule as
    // the gate/up GEMM fed by Xp, so that each gathered A stage serves twice
    // the MMA work
    if (!make_map(&p.tmX, a.x, d, (uint64_t)a.T, 1)) return cudaErrorInvalidValue;
    p.src_of = a.src_of; p.gK = a.K; p.gT = a.T;
    if (pair_enabled() && (p.N / 128) % 2 == 0 && p.K_fixed >= 4096)
      e = launch_pair<GU, 128, 2, true>(p, s);
    else
      e = launch_pair<GU, 128, 1, true>(p, s);
  } else {
    e = launch_bn<GU>(p, s);
  }
  if (e != cudaSuccess) return e;
  // DOWN
  TcParams q = p;
  if (!make_map(&q.tmA, H, F, a.max_rows, 128)) return cudaErrorInvalidValue;
  // the pair kernel's CTAs each load half of a B tile of 128 or 256 rows
  const uint32_t down_box = pair_enabled() ? (d % 256 == 0 ? 128 : 64) : 128;
  if (!make_map(&q.tmB, a.W_down, F, (uint64_t)E * d, down_box)) return cudaErrorInvalidValue;
  q.mode = DOWN; q.N = d; q.K_fixed = F; q.b_group_rows = d; q.out0 = a.Yp; q.out1 = nullptr;
  if (!make_store_map(&q.tmO0, a.Yp, 2, d, a.max_rows)) return cudaErrorInvalidValue;
  return launch_bn<DOWN>(q, s);
}

cudaError_t launch_router_bwd_tc(const RouterBwdTc &a, cudaStream_t s) {
  const int PP = 4 * a.PW, d = a.d;
  TcParams p{};
  p.n_groups = 1; p.max_rows = a.T; p.d = d; p.offsets = a.offs; p.status = a.status;
  cudaError_t e;
  if (a.dx_router != nullptr) {  // dx = [hi | mid | lo] planes x Wr3, K = 3 PW
    TcParams q = p;
    q.offsets = a.offs + 32;   // one group of T rows
    if (!make_map(&q.tmA, a.planes, PP, a.T, 128)) return cudaErrorInvalidValue;
    if (!make_map(&q.tmB, a.Wr3, d, 3 * (uint64_t)a.PW, 64)) return cudaErrorInvalidValue;
    q.mode = DX; q.N = d; q.K_fixed = 3 * a.PW; q.b_group_rows = 3 * (int64_t)a.PW;
    q.out0 = a.dx_router;
    if (!make_store_map(&q.tmO0, a.dx_router, 4, d, a.T)) return cudaErrorInvalidValue;
    if ((e = launch_bn<DX>(q, s)) != cudaSuccess) return e;
  }
  {  // dW: planes^T x, one group per token chunk
    TcParams q = p;
    q.n_groups = a.nsplit;
    if (!make_map(&q.tmA, a.planes, PP, a.T, 64)) return cudaErrorInvalidValue;
    if (!make_map(&q.tmB, a.x, d, a.T, 64)) return cudaErrorInvalidValue;
    CUtensorMap *maps = static_cast<CUtensorMap *>(a.maps);
    q.mode = WGD; q.M_fixed = PP; q.N = d; q.out0 = a.out_w; q.gmaps = maps;
    if (!make_store_map(&q.tmO0, a.out_w, 4, d, (uint64_t)a.nsplit * PP)) return cudaErrorInvalidValue;
    group_maps_kernel<<<1, 64, 0, s>>>(q.tmA, q.tmB, a.offs, a.nsplit, static_cast<const uint8_t *>(a.planes),
                                       2 * (int64_t)PP, static_cast<const uint8_t *>(a.x), 2 * (int64_t)d,
                                       a.T, maps);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_bn<WGD>(q, s)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_ffn_bwd_bf16(const FfnArgs &a, cudaStream_t s) {
  const int d = a.d, F = a.F, E = a.n_groups;
  TcParams p{};
  p.n_groups = E; p.max_rows = a.max_rows; p.d = d; p.F = F; p.offsets = a.offsets;
  p.status = a.status;
  cudaError_t e;
  {  // DH: dA = swiglu'(dYp W_down)
    TcParams q = p;
    if (!make_map(&q.tmA, a.dYp, d, a.max_rows, 128)) return cudaErrorInvalidValue;
    if (!make_map(&q.tmB, a.W_down, F, (uint64_t)E * d, 64)) return cudaErrorInvalidValue;
    q.mode = DH; q.N = F; q.K_fixed = d; q.b_group_rows = d; q.out0 = a.dA; q.aux = a.A_save;
    if (!make_store_map(&q.tmO0, a.dA, 2, 2 * (uint64_t)F, a.max_rows)) return cudaErrorInvalidValue;
    if (!make_store_map(&q.tmO1, const_cast<void *>(a.A_save), 2, 2 * (uint64_t)F, a.max_rows))
      return cudaErrorInvalidValue;
    if ((e = launch_bn<DH>(q, s)) != cudaSuccess) return e;
  }
  {  // DX: dXp = dA W_gu
    TcParams q = p;
    if (!make_map(&q.tmA, a.dA, 2 * F, a.max_rows, 128)) return cudaErrorInvalidValue;
    if (!make_map(&q.tmB, a.W_gu, d, (uint64_t)E * 2 * F, 64)) return cudaErrorInvalidValue;
    q.mode = DX; q.N = d; q.K_fixed = 2 * F; q.b_group_rows = 2 * (int64_t)F; q.out0 = a.dXp;
    if (!make_store_map(&q.tmO0, a.dXp, 4, d, a.max_rows)) return cudaErrorInvalidValue;
    if ((e = launch_bn<DX>(q, s)) != cudaSuccess) return e;
  }
  // the weight-gradient GEMMs read per-group tensor maps (two regions of the
  // workspace, one per mode, 2 * n_groups maps each)
  CUtensorMap *maps = static_cast<CUtensorMap *>(a.maps);
  {  // WGD: dW_down[g] = dYp_g^T H_g
    TcParams q = p;
    if (!make_map(&q.tmA, a.dYp, d, a.max_rows, 64)) return cudaErrorInvalidValue;
    if (!make_map(&q.tmB, a.H_save, F, a.max_rows, 64)) return cudaErrorInvalidValue;
    q.mode = WGD; q.M_fixed = d; q.N = F; q.out0 = a.dW_down; q.gmaps = maps;
    if (!make_store_map(&q.tmO0, a.dW_down, 4, F, (uint64_t)E * d)) return cudaErrorInvalidValue;
    group_maps_kernel<<<1, 64, 0, s>>>(q.tmA, q.tmB, a.offsets, E,
                                       static_cast<const uint8_t *>(a.dYp), 2 * (int64_t)d,
                                       static_cast<const uint8_t *>(a.H_save), 2 * (int64_t)F,
                                       a.max_rows, maps);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_bn<WGD>(q, s)) != cudaSuccess) return e;
  }
  {  // WGU: dW_gu[g] = dA_g^T Xp_g
    TcParams q = p;
    if (!make_map(&q.tmA, a.dA, 2 * F, a.max_rows, 64)) return cudaErrorInvalidValue;
    if (!make_map(&q.tmB, a.Xp, d, a.max_rows, 64)) return cudaErrorInvalidValue;
    CUtensorMap *maps_u = maps + 2 * kMaxMapGroups;
    q.mode = WGU; q.M_fixed = 2 * F; q.N = d; q.out0 = a.dW_gu; q.gmaps = maps_u;
    if (!make_store_map(&q.tmO0, a.dW_gu, 4, d, (uint64_t)E * 2 * F)) return cudaErrorInvalidValue;
    group_maps_kernel<<<1, 64, 0, s>>>(q.tmA, q.tmB, a.offsets, E,
                                       static_cast<const uint8_t *>(a.dA), 4 * (int64_t)F,
                                       static_cast<const uint8_t *>(a.Xp), 2 * (int64_t)d,
                                       a.max_rows, maps_u);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_bn<WGU>(q, s)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace moe
