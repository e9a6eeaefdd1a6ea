// Pass 2 of the exact attention backward-over-backward on sm_103a tensor
// cores: bf16 inputs, head dim 64, fp32 accumulation in tensor memory.
//
// "FlashBoB: I/O-Efficient Exact Backward-over-Backward for Softmax
// Attention" (paper notes), 关键设计 2: a block of key rows stays on chip
// while query row tiles stream past together with the row scalars (alpha, E)
// of pass 1; the column outputs are summed on chip and written once, with no
// atomics.  With the transposed scores of the resident key rows j against a
// streamed query row i:
//     dS   = P o (dP - D)
//     d~S  = P o (F o (dP - D) + G - alpha dP - E)       (d~P - E, times P)
//     W    = P o (F - alpha)                              (gradient w.r.t. dP)
//     d~K_j = tau sum_i (d~S_ij Q_i + dS_ij U_Q,i),   d~V_j = sum_i W_ij dO_i
// (F = tau (U_Q K^T + Q U_K^T), G = dO U_V^T; the same chain rule as pass 1).
//
// CTA = 128 key rows (MMA M = 128, one TMEM lane per key row), 320 threads:
//   warp 0      producer: TMA of the resident K, U_K, V, U_V block, then of
//               Q, U_Q, dO tiles of 64 query rows through a 4-stage mbarrier
//               ring, plus each tile's row-scalar columns (below);
//   warp 1      TMEM allocator; one elected lane runs the whole MMA schedule
//               (every barrier wait and every MMA);
//   warps 2-5 / 6-9   elementwise warpgroups 0 / 1: query rows 0-31 / 32-63
//               of every tile (the 16-row K steps 0-1 / 2-3 of its output
//               GEMMs).
// Every tcgen05.mma costs the pipe tens of cycles whatever its width, so
// the tile is 64 query rows wide: the score GEMMs are K [Q; U_Q]^T (N = 128,
// S^T and half of F'^T), U_K Q^T, V dO^T and U_V dO^T (N = 64 each).
// Row scalars ride in the score GEMMs.  Each query row's L, D, alpha and
// alpha D + E enter the score buffer through one more K step: an all-ones
// A operand (shared memory) against a 16-column B tile the producer writes
// per query tile, which holds -L / tau, -alpha / tau, -D and -(alpha D + E)
// as sums of three bf16 parts (exact to 2^-24 relative).  The score buffer
// then holds S^T - L / tau, F'^T - alpha / tau, dP^T - D and
// G^T - (alpha D + E), and the element-wise code needs no per-column
// scalars at all.
// TMEM: [0,64) d~K, [64,128) d~V accumulators; [128,384) one score buffer
// S^T | F'^T | dP^T | G^T (64 columns each); [384,480) the bf16 A operands
// dS^T, d~S^T, W^T of the output GEMMs; [480,512) U_K as the bf16 A operand
// of F'^T += U_K Q^T (copied from shared memory once: with A in TMEM this
// N = 64 GEMM runs at the tensor rate instead of waiting on shared-memory
// operand reads).  The all-ones A operand of the row-scalar K step lives in
// shared memory (at N = 128 that GEMM is tensor-bound either way).
// Because the operands have their own columns, the score buffer is released
// as soon as the warpgroups have read
// it into registers, in two halves: S^T | F'^T first (read before any
// arithmetic), then dP^T | G^T.  The score GEMMs of the next tile are issued
// in the same two halves, so the S/F' half of tile t + 1 runs on the tensor
// pipe while the warpgroups still read and process dP/G of tile t.
#include "internal.h"
#include "tc_common.cuh"

namespace flashbob {
namespace {
using namespace tc;

constexpr int BM = kTcRows;  // 128 key rows per CTA
constexpr int BQ = kTcStream2;  // 64 query rows per streamed tile
constexpr int DH = 64;
constexpr int NST = 4;
constexpr int NTHREADS = 320;
constexpr uint32_t BLOCK_BYTES = BM * DH * 2;  // 16 KiB
constexpr uint32_t TILE_BYTES = BQ * DH * 2;   // 8 KiB
constexpr float kLog2e = 1.4426950408889634f;

constexpr uint32_t EX_BYTES = 2 * BQ * 16 * 2;  // 128 rows x 16 bf16: one extra K step

struct Smem2 {
  alignas(1024) uint8_t kb[4][BLOCK_BYTES];      // K, U_K, V, U_V (resident)
  alignas(1024) uint8_t st[NST][3][TILE_BYTES];  // Q, U_Q, dO (Q|U_Q adjacent)
  // Row-scalar K step of each stage: [0] for S^T | F'^T (rows 0-63: -L/tau
  // of query rows 0-63, rows 64-127: -alpha/tau), [1] for dP^T | G^T (-D,
  // -(alpha D + E)).  No swizzle, K-major: 8-row x 16-byte core matrices,
  // row r at (r / 8) * 256 + (r % 8) * 16, k 8-15 128 bytes further.
  alignas(1024) uint8_t ex[NST][2][EX_BYTES];
  alignas(1024) uint8_t ones[BM * 16 * 2];  // all-ones A: 128 rows x 16 bf16, same layout
  uint64_t bar_kv;
  uint64_t a_ready;  // U_K is in TMEM (4 warps)
  uint64_t st_full[NST];
  uint64_t st_empty[NST];
  uint64_t sc_full;   // score GEMMs of a tile have completed
  uint64_t sf_free;   // both warpgroups have read S^T and F'^T (8 warps)
  uint64_t pg_free;   // both warpgroups have read dP^T and G^T (8 warps)
  uint64_t op_ready;  // the operands of a tile are in TMEM (8 warps)
  uint64_t op_free;   // the output GEMMs of a tile have completed
  uint64_t out_full;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Smem2) + 1024 <= 232448, "shared memory");

// TMEM columns.
constexpr uint32_t kAccK = 0, kAccV = 64;
constexpr uint32_t kSc = 128;  // score buffer
constexpr uint32_t kColS = 0, kColF = 64, kColdP = 128, kColG = 192;  // inside the score buffer
constexpr uint32_t kOp = 384;  // operand area: operand x, K step kk at kOp + 32 x + 8 kk
constexpr uint32_t kOpdS = 0, kOpdSt = 1, kOpW = 2;
constexpr uint32_t kUKA = 480;  // U_K as an A operand, K step kk at kUKA + 8 kk
// Padded query rows (i >= N_q, zero-filled by TMA) get -L / tau = -kFar, so
// their P = exp2(c1 (0 - kFar)) is exactly 0.
constexpr float kFar = 1e30f;
// Cluster split: a row of staged partial sums (d~K | d~V, fp32) in the ring
// buffer, padded against bank conflicts.
constexpr int kStageStride = 2 * DH + 4;
static_assert(BM * kStageStride * 4 <= NST * 3 * TILE_BYTES, "staging fits in the ring");
static_assert(8 * 2 * 32 * 36 * 4 <= NST * 3 * TILE_BYTES, "per-warp staging fits in the ring");

__device__ __forceinline__ constexpr uint32_t op_col(uint32_t x, int kk) {
  return kOp + 32 * x + 8 * kk;
}

// 16 query rows (one K step of the output GEMMs) of the score buffer, one
// key row per thread: dS, d~S and W packed as bf16 pairs (8 registers each),
// two query rows per step in the paired fp32 instructions.  The buffer
// already holds S' = S^T - L / tau, F'' = F'^T - alpha / tau, X = dP^T - D
// and G' = G^T - (alpha D + E), so with F - alpha = tau F'':
//     P = exp2(tau log2(e) S'),  dS = P X,  W = P (F - alpha),
//     d~S = P (X (F - alpha) + G')   (= P (F X + G - alpha dP - E)).
template <bool MASKED>
__device__ __forceinline__ void p2_chunk(const uint32_t (&s)[16], const uint32_t (&dp)[16],
                                         const uint32_t (&f)[16], const uint32_t (&g)[16],
                                         int ibase, int gj, float c1, float tau,
                                         uint32_t (&ods)[8], uint32_t (&odst)[8],
                                         uint32_t (&ow)[8]) {
  const float2 c12 = make_float2(c1, c1), tau2 = make_float2(tau, tau);
#pragma unroll
  for (int e = 0; e < 16; e += 2) {
    const float2 t = fmul2(f2(s[e], s[e + 1]), c12);
    float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
    if (MASKED) {
      if (ibase + e < gj) p.x = 0.f;
      if (ibase + e + 1 < gj) p.y = 0.f;
    }
    const float2 x = f2(dp[e], dp[e + 1]);
    const float2 w0 = fmul2(f2(f[e], f[e + 1]), tau2);  // F - alpha
    const float2 vds = fmul2(p, x);
    const float2 vdst = fmul2(p, ffma2(x, w0, f2(g[e], g[e + 1])));
    const float2 vw = fmul2(p, w0);
    ods[e >> 1] = pack_bf16x2(vds.x, vds.y);
    odst[e >> 1] = pack_bf16x2(vdst.x, vdst.y);
    ow[e >> 1] = pack_bf16x2(vw.x, vw.y);
  }
}

// The 32 query rows of one warpgroup: read S^T and F'^T of both 16-row
// chunks and release them, read dP^T and G^T of both chunks and release the
// score buffer, so that the next tile's score GEMMs are queued on the tensor
// pipe before any arithmetic of this one; only then form dS, d~S, W chunk by
// chunk, writing them once the previous tile's output GEMMs are done with
// the operand area.
template <bool MASKED>
__device__ __forceinline__ bool p2_half(uint32_t sc, uint32_t opb, int wg, int ibase, int gj,
                                        float c1, float tau, Smem2& sm, int t,
                                        volatile int* abort_flag, unsigned int* err) {
  const int col = 32 * wg;
  const int kk = 2 * wg;
  uint32_t s0[16], f0[16], s1[16], f1[16];
  tmem_ld16(sc + kColS + col, s0);
  tmem_ld16(sc + kColF + col, f0);
  tmem_ld16(sc + kColS + col + 16, s1);
  tmem_ld16(sc + kColF + col + 16, f1);
  tmem_wait_ld();
  tc_fence_before();
  warp_arrive(&sm.sf_free);  // this warp is done with S^T | F'^T
  uint32_t dp0[16], g0[16], dp1[16], g1[16];
  tmem_ld16(sc + kColdP + col, dp0);
  tmem_ld16(sc + kColG + col, g0);
  tmem_ld16(sc + kColdP + col + 16, dp1);
  tmem_ld16(sc + kColG + col + 16, g1);
  tmem_wait_ld();
  tc_fence_before();
  warp_arrive(&sm.pg_free);  // this warp is done with dP^T | G^T
  {
    uint32_t a_ds[8], a_dst[8], a_w[8];
    p2_chunk<MASKED>(s0, dp0, f0, g0, ibase, gj, c1, tau, a_ds, a_dst, a_w);
    if (t > 0 && !mbar_wait_warp(&sm.op_free, (t - 1) & 1, abort_flag, err)) return false;
    tc_fence_after();
    tmem_st8(opb + op_col(kOpdS, kk), a_ds);
    tmem_st8(opb + op_col(kOpdSt, kk), a_dst);
    tmem_st8(opb + op_col(kOpW, kk), a_w);
  }
  {
    uint32_t o_ds[8], o_dst[8], o_w[8];
    p2_chunk<MASKED>(s1, dp1, f1, g1, ibase + 16, gj, c1, tau, o_ds, o_dst, o_w);
    tmem_st8(opb + op_col(kOpdS, kk + 1), o_ds);
    tmem_st8(opb + op_col(kOpdSt, kk + 1), o_dst);
    tmem_st8(opb + op_col(kOpW, kk + 1), o_w);
  }
  tmem_wait_st();
  tc_fence_before();
  warp_arrive(&sm.op_ready);
  return true;
}

// Alone (no cluster split), each warp transposes its own 32 rows x 32
// columns of d~K and d~V through a private slice of the idle ring (rows
// padded to 36 floats) and writes them as whole 128-byte row segments, with
// no barrier across warps.  Out of line: the CTA runs it once, and keeping
// it out of the kernel body leaves the tile loop's code as it is.
static __device__ __noinline__ void store_rows_alone(uint32_t acc_base, uint8_t* ring, int warp,
                                                     int lane, int quad, int wg, int T,
                                                     float tau, bool ok, int j0, int bkv,
                                                     int Nk, float* __restrict__ dKt,
                                                     float* __restrict__ dVt) {
  constexpr int kLd = 36;
  float* wk = reinterpret_cast<float*>(ring) + (warp - 2) * (2 * 32 * kLd);
  float* wv = wk + 32 * kLd;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t vk[16], vv[16];
    tmem_ld16(acc_base + kAccK + 32 * wg + 16 * h, vk);
    tmem_ld16(acc_base + kAccV + 32 * wg + 16 * h, vv);
    tmem_wait_ld();
    if (T == 0) {
#pragma unroll
      for (int k = 0; k < 16; ++k) vk[k] = vv[k] = 0u;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      reinterpret_cast<float4*>(wk + lane * kLd + 16 * h)[k] =
          make_float4(tau * u2f(vk[4 * k]), tau * u2f(vk[4 * k + 1]), tau * u2f(vk[4 * k + 2]),
                      tau * u2f(vk[4 * k + 3]));
      reinterpret_cast<float4*>(wv + lane * kLd + 16 * h)[k] =
          make_float4(u2f(vv[4 * k]), u2f(vv[4 * k + 1]), u2f(vv[4 * k + 2]),
                      u2f(vv[4 * k + 3]));
    }
  }
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int f = lane + 32 * k, rr = f >> 3, c4 = f & 7;  // 8 float4 per row
    const int gjr = j0 + quad * 32 + rr;
    if (ok && gjr < Nk) {
      const size_t o = (static_cast<size_t>(bkv) * Nk + gjr) * DH + 32 * wg + 4 * c4;
      *reinterpret_cast<float4*>(dKt + o) = *reinterpret_cast<const float4*>(wk + rr * kLd + 4 * c4);
      *reinterpret_cast<float4*>(dVt + o) = *reinterpret_cast<const float4*>(wv + rr * kLd + 4 * c4);
    }
  }
}

// SPLIT: launched as clusters of S > 1 CTAs that share a key block.
// STAGED (without SPLIT): the rows leave through shared memory
// (store_rows_alone) instead of straight from each thread's registers.  The
// staged epilogue is ~4 us shorter per CTA, but its instance ran the tile
// loop 3% slower at 1,024 tiles per CTA (measured: the same source with the
// other epilogue, swapped alone), so it serves CTAs of at most kStagedTiles
// tiles, where the epilogue is a large share of the CTA.
constexpr int kStagedTiles = 128;
template <bool SPLIT, bool STAGED = false>
__global__ void __launch_bounds__(NTHREADS, 1)
    tc_pass2_kernel(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mUK,
                    const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mUV,
                    const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mUQ,
                    const __grid_constant__ CUtensorMap mdO, const float* __restrict__ L,
                    const float* __restrict__ D, const float* __restrict__ alpha,
                    const float* __restrict__ E, float* __restrict__ dKt,
                    float* __restrict__ dVt, int H, int Hkv, int Nq, int Nk, float tau,
                    int causal, int S, unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  Smem2& sm = *reinterpret_cast<Smem2*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                        ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // One CTA per key block of a key/value head.  Grouped-query attention: the
  // G = H / Hkv query heads sharing the head stream past one after the other
  // and their contributions are summed on chip ([FBN] 关键设计 3).  A cluster
  // of S CTAs (blockIdx.y = S * head + rank) shares a key block when the
  // key blocks alone cannot fill the GPU: rank q streams the q-th of S equal
  // runs of the group's query tiles, and the partial sums meet in
  // distributed shared memory before the one write.
  const int G = H / Hkv;
  const int bkv = blockIdx.z * Hkv + blockIdx.y / S;
  const int rank = blockIdx.y % S;
  const int hqb = blockIdx.z * H + (blockIdx.y / S) * G;  // first query head of the group
  const int j0 = blockIdx.x * BM;
  // Query tiles t0 .. of 64 rows stream past; under the causal mask key j is
  // seen only by queries i >= j, so the tiles before the block are skipped
  // (all of them when j0 >= Nq: then Tq = 0 and the block's d~K, d~V are 0).
  // Group tile f = (query head in group) * Tq + (tile - t0); this CTA takes
  // f = f0 .. f0 + T - 1, its own t = f - f0 counting ring slots and barrier
  // phases.
  const int t0 = causal ? j0 / BQ : 0;
  const int Tq = max(0, (Nq + BQ - 1) / BQ - t0);
  const int Tall = G * Tq;
  const int f0 = static_cast<int>(static_cast<long long>(Tall) * rank / S);
  const int T = static_cast<int>(static_cast<long long>(Tall) * (rank + 1) / S) - f0;
  volatile int* abort_flag = &sm.abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(&sm.bar_kv, 1);
    mbar_init(&sm.a_ready, 4);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&sm.st_full[s], 2);  // the TMA transaction, and the row-scalar K step written
      mbar_init(&sm.st_empty[s], 1);
    }
    mbar_init(&sm.sc_full, 1);
    mbar_init(&sm.sf_free, 8);
    mbar_init(&sm.pg_free, 8);
    mbar_init(&sm.op_ready, 8);
    mbar_init(&sm.op_free, 1);
    mbar_init(&sm.out_full, 1);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  if (warp == 0) {
    // Producer.  Lane 0 issues the TMA copies; the whole warp writes the
    // row-scalar K step of every tile: lane l takes query rows l and l + 32
    // (and, first, the all-ones A operand: k = 0, 1, 2 are 1).
    const float inv_tau = 1.f / tau;
    for (int r = lane; r < BM; r += 32) {
      uint8_t* base = sm.ones + (r >> 3) * 256 + (r & 7) * 16;
      const uint32_t one = 0x3F80u;  // bf16 1.0
      *reinterpret_cast<uint4*>(base) = make_uint4(one | (one << 16), one, 0u, 0u);
      *reinterpret_cast<uint4*>(base + 128) = make_uint4(0u, 0u, 0u, 0u);
    }
    auto load_rows = [&](int f, float4 (&v)[2]) {
      // (L, D, alpha, E) of rows lane, lane + 32 of streamed tile f; a row
      // past N_q (or a tile past the last) is marked by L = NaN.
      v[0] = v[1] = make_float4(__int_as_float(0x7fc00000), 0.f, 0.f, 0.f);
      if (f >= T) return;
      const int zq = hqb + (f0 + f) / Tq, row0 = ((f0 + f) % Tq + t0) * BQ;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = row0 + lane + 32 * h;
        if (i < Nq) {
          const size_t o = static_cast<size_t>(zq) * Nq + i;
          v[h] = make_float4(L[o], D[o], alpha[o], E[o]);
        }
      }
    };
    if (lane == 0) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mUQ);
      tma_prefetch_desc(&mdO);
      mbar_expect_tx(&sm.bar_kv, 4 * BLOCK_BYTES);
      tma_load_3d(sm.kb[0], &mK, &sm.bar_kv, 0, j0, bkv);
      tma_load_3d(sm.kb[1], &mUK, &sm.bar_kv, 0, j0, bkv);
      tma_load_3d(sm.kb[2], &mV, &sm.bar_kv, 0, j0, bkv);
      tma_load_3d(sm.kb[3], &mUV, &sm.bar_kv, 0, j0, bkv);
    }
    float4 cur[2];
    load_rows(0, cur);
    int issued = 0;
    for (int t = 0; t < T; ++t) {
      const int s = t % NST;
      if (t >= NST && !mbar_wait_warp(&sm.st_empty[s], ((t / NST) - 1) & 1, abort_flag, err))
        break;
      if (lane == 0) {
        const int row = ((f0 + t) % Tq + t0) * BQ, zq = hqb + (f0 + t) / Tq;
        mbar_expect_tx(&sm.st_full[s], 3 * TILE_BYTES);
        tma_load_3d(sm.st[s][0], &mQ, &sm.st_full[s], 0, row, zq);
        tma_load_3d(sm.st[s][1], &mUQ, &sm.st_full[s], 0, row, zq);
        tma_load_3d(sm.st[s][2], &mdO, &sm.st_full[s], 0, row, zq);
      }
      // Four B rows per query row: k = 0, 1, 2 hold the three bf16 parts of
      // the scalar, k = 3 .. 15 zero.
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float4 v = cur[h];
        const bool pad = v.x != v.x;
        const float vals[4] = {pad ? -kFar : -v.x * inv_tau, -v.z * inv_tau, -v.y,
                               -fmaf(v.z, v.y, v.w)};
        const int r = lane + 32 * h;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int row = r + BQ * (q & 1);  // -L/tau, -alpha/tau ; -D, -(alpha D + E)
          uint8_t* base = sm.ex[s][q >> 1] + (row >> 3) * 256 + (row & 7) * 16;
          const uint2 hm_l0 = split3_bf16(vals[q]);
          *reinterpret_cast<uint4*>(base) = make_uint4(hm_l0.x, hm_l0.y, 0u, 0u);
          *reinterpret_cast<uint4*>(base + 128) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();  // also covers the ones operand before tile 0
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.st_full[s]);
      issued = t + 1;
      load_rows(t + 1, cur);  // lands while the ring is full
    }
    if (lane == 0) {
      // No copy may still be in flight when the CTA exits.
      drain_wait(&sm.bar_kv, 0);
      for (int t = issued > NST ? issued - NST : 0; t < issued; ++t)
        drain_wait(&sm.st_full[t % NST], (t / NST) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (whole warp, one elected lane issues) ----------------
    constexpr uint32_t idS64 = idesc_bf16(BM, BQ, false);       // N = 64, B K-major
    constexpr uint32_t idS128 = idesc_bf16(BM, 2 * BQ, false);  // N = 128, B K-major
    constexpr uint32_t idO = idesc_bf16(BM, DH, true);          // N = 64, B MN-major
    const uint64_t dK = smem_desc_sw128(smem_u32(sm.kb[0]), 16, 1024);
    const uint64_t dV = smem_desc_sw128(smem_u32(sm.kb[2]), 16, 1024);
    const uint64_t dUV = smem_desc_sw128(smem_u32(sm.kb[3]), 16, 1024);
    const uint32_t st0 = smem_u32(sm.st[0][0]);
    const uint64_t dQ0 = smem_desc_sw128(st0, 16, 1024);                   // Q (and Q;U_Q)
    const uint64_t dUQ0 = smem_desc_sw128(st0 + TILE_BYTES, 16, 1024);
    const uint64_t ddO0 = smem_desc_sw128(st0 + 2 * TILE_BYTES, 16, 1024);
    const uint64_t dEx0 = smem_desc_noswz(smem_u32(sm.ex[0][0]), 128, 256);
    const uint64_t dOnes = smem_desc_noswz(smem_u32(sm.ones), 128, 256);
    constexpr uint64_t kExStage = (2 * EX_BYTES) >> 4, kExPG = EX_BYTES >> 4;
    const uint32_t sc = tbase + kSc;
    // Score GEMMs in two halves: S^T | F'^T, then dP^T | G^T (+ commit).
    auto issue_sf = [&](int t) {
      const uint64_t so = (uint64_t)((t % NST) * 3 * TILE_BYTES) >> 4;
      {
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint64_t o = 2 * kk;  // 16 bf16 along d = 32 bytes >> 4
          mma_ss(sc + kColS, dK + o, dQ0 + so + o, idS128, kk > 0);  // [S^T | F'^T] = K [Q; U_Q]^T
          mma_ts(sc + kColF, tbase + kUKA + 8 * kk, dQ0 + so + o, idS64, 1);  // F'^T += U_K Q^T
        }
        // [S^T | F'^T] += 1 [-L / tau | -alpha / tau]^T (the row-scalar K step)
        mma_ss(sc + kColS, dOnes, dEx0 + (t % NST) * kExStage, idS128, 1);
      }
    };
    auto issue_pg = [&](int t) {
      const uint64_t so = (uint64_t)((t % NST) * 3 * TILE_BYTES) >> 4;
      {
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint64_t o = 2 * kk;
          mma_ss(sc + kColdP, dV + o, ddO0 + so + o, idS64, kk > 0);  // dP^T = V dO^T
          mma_ss(sc + kColG, dUV + o, ddO0 + so + o, idS64, kk > 0);  // G^T  = U_V dO^T
        }
        // [dP^T | G^T] += 1 [-D | -(alpha D + E)]^T
        mma_ss(sc + kColdP, dOnes, dEx0 + (t % NST) * kExStage + kExPG, idS128, 1);
        mma_commit(&sm.sc_full);
      }
    };
    auto issue_outputs = [&](int t) {
      const int s = t % NST;
      const uint64_t so = (uint64_t)(s * 3 * TILE_BYTES) >> 4;
      {
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          const uint64_t o = (uint64_t)(16 * 128 * kk) >> 4;  // 16 query rows further down
          const uint32_t acc = (t > 0 || kk > 0);
          mma_ts(tbase + kAccK, tbase + op_col(kOpdSt, kk), dQ0 + so + o, idO, acc);  // d~K += d~S^T Q
          mma_ts(tbase + kAccK, tbase + op_col(kOpdS, kk), dUQ0 + so + o, idO, 1);    //     +  dS^T U_Q
          mma_ts(tbase + kAccV, tbase + op_col(kOpW, kk), ddO0 + so + o, idO, acc);   // d~V += W^T dO
        }
        mma_commit(&sm.op_free);
        mma_commit(&sm.st_empty[s]);
      }
    };
    // One elected lane runs the whole schedule: every wait and every MMA,
    // with no warp-wide broadcast between them.
    if (elect_one()) {
      bool ok = mbar_wait(&sm.bar_kv, 0, abort_flag, err) &&
                mbar_wait(&sm.a_ready, 0, abort_flag, err);
      for (int t = 0; ok && t < T; ++t) {
        // Tile t's data is normally in the ring long before the warpgroups
        // release S^T | F'^T of tile t - 1: check it first, so that the S/F
        // GEMMs issue as soon as the release arrives.
        ok = mbar_wait(&sm.st_full[t % NST], (t / NST) & 1, abort_flag, err);
        if (!ok) break;
        if (t > 0) {  // both warpgroups hold S^T, F'^T of tile t - 1 in registers
          ok = mbar_wait(&sm.sf_free, (t - 1) & 1, abort_flag, err);
          if (!ok) break;
        }
        tc_fence_after();
        issue_sf(t);
        if (t > 0) {  // ... and dP^T, G^T
          ok = mbar_wait(&sm.pg_free, (t - 1) & 1, abort_flag, err);
          if (!ok) break;
          tc_fence_after();
        }
        issue_pg(t);
        if (t > 0) {
          ok = mbar_wait(&sm.op_ready, (t - 1) & 1, abort_flag, err);
          if (!ok) break;
          tc_fence_after();
          issue_outputs(t - 1);
        }
      }
      if (ok && T > 0) {
        ok = mbar_wait(&sm.op_ready, (T - 1) & 1, abort_flag, err);
        tc_fence_after();
        if (ok) issue_outputs(T - 1);
      }
      mma_commit(&sm.out_full);  // every MMA issued above has finished
    }
    __syncwarp();
  } else {
    const int wg = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // key row inside the block = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int gj = j0 + r;
    const float c1 = tau * kLog2e;
    const uint32_t sc = tbase + lane_off + kSc;
    const uint32_t opb = tbase + lane_off;
    bool ok = true;
    if (wg == 0) {
      // Warpgroup 0 copies its key row of U_K from the 128-byte-swizzled TMA
      // block (16-byte chunk c of row r at chunk c ^ (r mod 8)) into TMEM:
      // K step kk is chunks 2 kk and 2 kk + 1.
      ok = mbar_wait_warp(&sm.bar_kv, 0, abort_flag, err);
      if (ok) {
        const uint8_t* row = sm.kb[1] + r * 128;
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint4 a = *reinterpret_cast<const uint4*>(row + (((2 * kk) ^ (r & 7)) << 4));
          const uint4 b = *reinterpret_cast<const uint4*>(row + (((2 * kk + 1) ^ (r & 7)) << 4));
          const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
          tmem_st8(tbase + lane_off + kUKA + 8 * kk, v);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      warp_arrive(&sm.a_ready);
    }
    int tq = Tq > 0 ? f0 % Tq : 0;  // tile of the current query head, (f0 + t) mod Tq
    for (int t = 0; t < T; ++t) {
      // Warp-uniform decisions (tcgen05.ld/st are warp-collective); after a
      // failed wait the remaining tiles are skipped.
      ok = ok && mbar_wait_warp(&sm.sc_full, t & 1, abort_flag, err);
      if (ok) {
        tc_fence_after();
        // Causal: queries i < j (this thread's key row) get P = 0; only the
        // tiles that overlap the key block take the masked path.
        const int ibase = (tq + t0) * BQ + 32 * wg;
        if (causal && ibase < j0 + BM)
          ok = p2_half<true>(sc, opb, wg, ibase, gj, c1, tau, sm, t, abort_flag, err);
        else
          ok = p2_half<false>(sc, opb, wg, ibase, gj, c1, tau, sm, t, abort_flag, err);
      }
      if (++tq == Tq) tq = 0;
    }

    ok = mbar_wait_warp(&sm.out_full, 0, abort_flag, err) && ok;
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);
    tc_fence_after();
    const uint32_t acc_base = tbase + lane_off;
    // A thread holds one key row, so writing global memory straight from
    // registers would scatter each warp's float4 over 32 rows: the rows go
    // through shared memory (every MMA is done and the ring is idle).  A CTA
    // with no tile (T = 0) never wrote its accumulators and stages zeros.
    if (SPLIT) {
      // Stage the CTA's partial d~K | d~V rows for the cluster-wide sum below.
      float* row = reinterpret_cast<float*>(&sm.st[0][0][0]) + r * kStageStride;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int col = 32 * wg + 16 * h;
        uint32_t vk[16], vv[16];
        tmem_ld16(acc_base + kAccK + col, vk);
        tmem_ld16(acc_base + kAccV + col, vv);
        tmem_wait_ld();
        if (T == 0) {
#pragma unroll
          for (int k = 0; k < 16; ++k) vk[k] = vv[k] = 0u;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          reinterpret_cast<float4*>(row + col)[k] =
              make_float4(u2f(vk[4 * k]), u2f(vk[4 * k + 1]), u2f(vk[4 * k + 2]),
                          u2f(vk[4 * k + 3]));
          reinterpret_cast<float4*>(row + DH + col)[k] =
              make_float4(u2f(vv[4 * k]), u2f(vv[4 * k + 1]), u2f(vv[4 * k + 2]),
                          u2f(vv[4 * k + 3]));
        }
      }
    } else if (STAGED) {
      store_rows_alone(acc_base, &sm.st[0][0][0], warp, lane, quad, wg, T, tau, ok, j0, bkv, Nk,
                       dKt, dVt);
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int col = 32 * wg + 16 * h;
        uint32_t vk[16], vv[16];
        tmem_ld16(acc_base + kAccK + col, vk);
        tmem_ld16(acc_base + kAccV + col, vv);
        tmem_wait_ld();
        if (ok && gj < Nk) {
          const size_t off = (static_cast<size_t>(bkv) * Nk + gj) * DH + col;
          float4* k4 = reinterpret_cast<float4*>(dKt + off);
          float4* v4 = reinterpret_cast<float4*>(dVt + off);
          if (T == 0) {
#pragma unroll
            for (int k = 0; k < 16; ++k) vk[k] = vv[k] = 0u;
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            k4[k] = make_float4(tau * u2f(vk[4 * k]), tau * u2f(vk[4 * k + 1]),
                                tau * u2f(vk[4 * k + 2]), tau * u2f(vk[4 * k + 3]));
            v4[k] = make_float4(u2f(vv[4 * k]), u2f(vv[4 * k + 1]), u2f(vv[4 * k + 2]),
                                u2f(vv[4 * k + 3]));
          }
        }
      }
    }
  }

  if (SPLIT) {
    // Cluster rank q sums key rows [128 q / S, 128 (q + 1) / S) of the block
    // over the S CTAs' staged partials and writes them: one write per
    // element, no atomics.  All threads pass both cluster barriers; the
    // second keeps every CTA's staged rows alive until all reads are done.
    cluster_sync();
    if (warp >= 2) {
      const uint32_t q = cluster_ctarank();
      const int rb = (BM * (int)q) / S, re = (BM * ((int)q + 1)) / S;
      const uint32_t stage = smem_u32(&sm.st[0][0][0]);
      const int tid = threadIdx.x - 64;
      for (int e = tid; e < (re - rb) * 32; e += 256) {
        const int rr = rb + e / 32, c4 = e % 32;  // row, float4 column of d~K | d~V
        const uint32_t off = static_cast<uint32_t>((rr * kStageStride + 4 * c4) * 4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int p = 0; p < S; ++p) {
          const float4 v = ld_shared_cluster_f4(mapa_shared(stage + off, p));
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
        const int gjr = j0 + rr;
        if (gjr < Nk && !*abort_flag) {
          const bool isK = c4 < DH / 4;
          const size_t o = (static_cast<size_t>(bkv) * Nk + gjr) * DH + 4 * (isK ? c4 : c4 - DH / 4);
          if (isK)
            *reinterpret_cast<float4*>(dKt + o) =
                make_float4(tau * acc.x, tau * acc.y, tau * acc.z, tau * acc.w);
          else
            *reinterpret_cast<float4*>(dVt + o) = acc;
        }
      }
    }
    cluster_sync();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace

size_t tc_pass2_smem() { return sizeof(Smem2) + 1024; }

cudaError_t tc_launch_pass2(const BobArgs& a, const CUtensorMap* maps128,
                            const CUtensorMap* maps64) {
  // maps128: K, U_K, V, U_V with 128-row boxes; maps64: Q, U_Q, dO with 64-row boxes.
  const size_t smem = tc_pass2_smem();
  cudaError_t e = tc_set_smem(reinterpret_cast<const void*>(tc_pass2_kernel<false>), (int)smem);
  if (e == cudaSuccess)
    e = tc_set_smem(reinterpret_cast<const void*>(tc_pass2_kernel<false, true>), (int)smem);
  if (e != cudaSuccess) return e;
  // One CTA per key block of a shared head, or, when the key blocks cannot
  // fill the SMs, a cluster of S of them that splits the block's query tiles
  // S ways.
  e = tc_set_smem(reinterpret_cast<const void*>(tc_pass2_kernel<true>), (int)smem);
  if (e != cudaSuccess) return e;
  const int tiles = (a.H / a.Hkv) * ((a.Nq + BQ - 1) / BQ);
  int S = 1;
  if (!a.whole_grid_only)
    e = tc_pass2_split(reinterpret_cast<const void*>(tc_pass2_kernel<true>), smem,
                       ((a.Nk + BM - 1) / BM) * a.Hkv * a.B, tiles, &S);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Nk + BM - 1) / BM, a.Hkv * S, a.B);
  if (S == 1) {
    // Tiles a CTA streams: every query tile of its group (fewer under the causal mask).
    const bool staged = tiles <= kStagedTiles;
    auto kernel = staged ? tc_pass2_kernel<false, true> : tc_pass2_kernel<false>;
    kernel<<<grid, NTHREADS, smem, a.stream>>>(
        maps128[0], maps128[1], maps128[2], maps128[3], maps64[0], maps64[1], maps64[2], a.L,
        a.D, a.alpha, a.E, a.dKt, a.dVt, a.H, a.Hkv, a.Nq, a.Nk, a.tau, a.causal ? 1 : 0, 1,
        a.err);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = S;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_pass2_kernel<true>, maps128[0], maps128[1], maps128[2],
                            maps128[3], maps64[0], maps64[1], maps64[2], a.L, a.D, a.alpha, a.E,
                            a.dKt, a.dVt, a.H, a.Hkv, a.Nq, a.Nk, a.tau, a.causal ? 1 : 0, S,
                            a.err);
}

}  // namespace flashbob
