// Pass 2 of the exact attention backward-over-backward on sm_103a tensor
// cores for head dim 128 (bf16 inputs, fp32 accumulation in tensor memory).
//
// "FlashBoB: I/O-Efficient Exact Backward-over-Backward for Softmax
// Attention" (paper notes), 关键设计 2: a block of 128 key rows stays on chip
// while query row tiles stream past with the row scalars (alpha, E) of pass
// 1; d~K and d~V are summed on chip and written once, with no atomics.  With
// the transposed scores of the resident key rows j against a streamed query
// row i:
//     dS = P o (dP - D),  d~S = P o (F o (dP - D) + G - alpha dP - E),
//     W = P o (F - alpha),
//     d~K_j = tau sum_i (d~S_ij Q_i + dS_ij U_Q,i),   d~V_j = sum_i W_ij dO_i.
//
// CTA = 128 key rows (MMA M = 128, one TMEM lane per key row), 320 threads:
//   warp 0      producer: TMA of the resident K, U_K, V, U_V block (each as
//               two 64-column halves in the 128-byte swizzle), then of Q,
//               U_Q, dO tiles of 32 query rows through a 3-stage ring, plus
//               each tile's row-scalar K step;
//   warp 1      TMEM allocation and MMA issue;
//   warps 2-5 / 6-9   elementwise warpgroups 0 / 1: query rows 0-15 / 16-31
//               of every tile (the K step of the output GEMMs they feed).
// Row scalars ride in the score GEMMs as at head dim 64: one more K step,
// an all-ones A operand in TMEM against a 16-column B tile that the producer
// writes per query tile (-L / tau, -alpha / tau, -D, -(alpha D + E), each as
// three bf16 parts), leaves S^T - L / tau, F'^T - alpha / tau, dP^T - D and
// G^T - (alpha D + E) in the score buffer.
// TMEM: [0,128) d~K, [128,256) d~V accumulators; [256,384) one score buffer
// S^T | F'^T | dP^T | G^T (32 columns each); [384,432) the bf16 A operands
// dS^T, d~S^T, W^T; [432,440) the all-ones A operand; [440,504) U_K as the
// bf16 A operand of F'^T += U_K Q^T (copied from shared memory once; with A
// in TMEM this N = 32 GEMM runs at the tensor rate instead of waiting on
// shared-memory operand reads).  The score buffer is
// released in two halves, S^T | F'^T
// first, so the S/F' GEMMs of the next tile run while the warpgroups still
// read and process dP/G.  Grouped-query attention: the query tiles of all
// H / Hkv heads sharing the key/value head stream past the same block
// ([FBN] 关键设计 3).
#include "internal.h"
#include "tc_common.cuh"

namespace flashbob {
namespace {
using namespace tc;

constexpr int BM = kTcRows;  // 128 key rows per CTA
constexpr int BQ = 32;       // query rows per streamed tile
constexpr int DH = 128;
constexpr int NST = 4;  // ring stages; stage 3 lies in the U_K block (free once U_K is in TMEM)
constexpr int NTHREADS = 320;
constexpr uint32_t HALF_BLOCK = BM * 64 * 2;  // 16 KiB
constexpr uint32_t HALF_TILE = BQ * 64 * 2;   // 4 KiB
constexpr uint32_t STAGE_BYTES = 2 * 3 * HALF_TILE;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t EX_BYTES = 2 * BQ * 16 * 2;  // 64 rows x 16 bf16: one extra K step

struct SmemW2 {
  alignas(1024) uint8_t kb[4][2][HALF_BLOCK];         // K, U_K, V, U_V (resident) x halves
  alignas(1024) uint8_t st[NST - 1][2][3][HALF_TILE];  // [stage][half][Q, U_Q, dO]
  // Row-scalar K step of each stage: [0] for S^T | F'^T (rows 0-31: -L/tau,
  // rows 32-63: -alpha/tau), [1] for dP^T | G^T (-D, -(alpha D + E)); no
  // swizzle, K-major, row r at (r / 8) * 256 + (r % 8) * 16, k 8-15 at +128.
  alignas(1024) uint8_t ex[NST - 1][2][EX_BYTES];
  uint64_t bar_kv;
  uint64_t a_ready;  // U_K is in TMEM (4 warps)
  uint64_t st_full[NST];
  uint64_t st_empty[NST];
  uint64_t sc_full;
  uint64_t sf_free;   // both warpgroups have read S^T and F'^T (8 warps)
  uint64_t pg_free;   // both warpgroups have read dP^T and G^T (8 warps)
  uint64_t op_ready;  // the operands of a tile are in TMEM (8 warps)
  uint64_t op_free;   // the output GEMMs of a tile have completed
  uint64_t out_full;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(SmemW2) + 1024 <= 232448, "shared memory");
// Stage 3: the tiles at offset 0 and the row-scalar K steps at STAGE_BYTES
// of the U_K block.
static_assert(STAGE_BYTES + 2 * EX_BYTES <= 2 * HALF_BLOCK, "stage 3 fits in the U_K block");

constexpr uint32_t kAccK = 0, kAccV = 128;
constexpr uint32_t kSc = 256;
constexpr uint32_t kColS = 0, kColF = 32, kColdP = 64, kColG = 96;  // inside the score buffer
constexpr uint32_t kOp = 384;  // operand x, K step kk at kOp + 16 x + 8 kk
constexpr uint32_t kOpdS = 0, kOpdSt = 1, kOpW = 2;
constexpr uint32_t kOnes = 432;  // all-ones A operand (k = 0, 1, 2) of the row-scalar K step
constexpr uint32_t kUKA = 440;   // U_K as an A operand, K step kk at kUKA + 8 kk
constexpr float kFar = 1e30f;    // -L / tau of a padded query row: its P is exactly 0
// Cluster split: staged partial rows d~K | d~V (64 float4 each) fill the
// 128 KiB of the resident block exactly; float4 c of row r sits at
// c ^ (r mod 8) against bank conflicts.
static_assert(BM * 2 * DH * 4 <= 4 * 2 * HALF_BLOCK, "staging fits in the resident block");

__device__ __forceinline__ constexpr uint32_t op_col(uint32_t x, int kk) {
  return kOp + 16 * x + 8 * kk;
}

// Ring stage s: tile i (Q, U_Q, dO) of half h, and its row-scalar K step q.
__device__ __forceinline__ uint8_t* stage_tile(SmemW2& sm, int s, int h, int i) {
  return s < NST - 1 ? sm.st[s][h][i]
                      : reinterpret_cast<uint8_t*>(&sm.kb[1]) + (3 * h + i) * HALF_TILE;
}
__device__ __forceinline__ uint8_t* stage_ex(SmemW2& sm, int s, int q) {
  return s < NST - 1 ? sm.ex[s][q]
                      : reinterpret_cast<uint8_t*>(&sm.kb[1]) + STAGE_BYTES + q * EX_BYTES;
}

// The 16 query rows of one warpgroup: read S^T, F'^T (release), dP^T, G^T
// (release), form dS, d~S, W as bf16 pairs and write them to the operand
// area once the previous tile's output GEMMs are done with it.  The buffer
// holds S' = S^T - L / tau, F'' = F'^T - alpha / tau, X = dP^T - D and
// G' = G^T - (alpha D + E): P = exp2(tau log2(e) S'), dS = P X,
// W = P (F - alpha) with F - alpha = tau F'', d~S = P (X (F - alpha) + G').
template <bool MASKED>
__device__ __forceinline__ bool p2w_half(uint32_t sc, uint32_t opb, int wg, int ibase, int gj,
                                         float c1, float tau, SmemW2& sm, int t,
                                         volatile int* abort_flag, unsigned int* err) {
  const int col = 16 * wg;
  uint32_t s[16], f[16], dp[16], g[16];
  tmem_ld16(sc + kColS + col, s);
  tmem_ld16(sc + kColF + col, f);
  tmem_wait_ld();
  tc_fence_before();
  warp_arrive(&sm.sf_free);
  tmem_ld16(sc + kColdP + col, dp);
  tmem_ld16(sc + kColG + col, g);
  tmem_wait_ld();
  tc_fence_before();
  warp_arrive(&sm.pg_free);
  uint32_t ods[8], odst[8], ow[8];
  const float2 c12 = make_float2(c1, c1), tau2 = make_float2(tau, tau);
#pragma unroll
  for (int e = 0; e < 16; e += 2) {
    const float2 tt = fmul2(f2(s[e], s[e + 1]), c12);
    float2 p = make_float2(ex2_approx(tt.x), ex2_approx(tt.y));
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
  if (t > 0 && !mbar_wait_warp(&sm.op_free, (t - 1) & 1, abort_flag, err)) return false;
  tc_fence_after();
  tmem_st8(opb + op_col(kOpdS, wg), ods);
  tmem_st8(opb + op_col(kOpdSt, wg), odst);
  tmem_st8(opb + op_col(kOpW, wg), ow);
  tmem_wait_st();
  tc_fence_before();
  warp_arrive(&sm.op_ready);
  return true;
}

// SPLIT: launched as clusters of S > 1 CTAs that share a key block.
template <bool SPLIT>
__global__ void __launch_bounds__(NTHREADS, 1)
    tc_pass2_d128_kernel(const __grid_constant__ CUtensorMap mK,
                         const __grid_constant__ CUtensorMap mUK,
                         const __grid_constant__ CUtensorMap mV,
                         const __grid_constant__ CUtensorMap mUV,
                         const __grid_constant__ CUtensorMap mQ,
                         const __grid_constant__ CUtensorMap mUQ,
                         const __grid_constant__ CUtensorMap mdO, const float* __restrict__ L,
                         const float* __restrict__ D, const float* __restrict__ alpha,
                         const float* __restrict__ E, float* __restrict__ dKt,
                         float* __restrict__ dVt, int H, int Hkv, int Nq, int Nk, float tau,
                         int causal, int S, unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  SmemW2& sm = *reinterpret_cast<SmemW2*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // A cluster of S CTAs (blockIdx.y = S * head + rank) may share a key
  // block, rank q streaming the q-th of S equal runs of the group's query
  // tiles; the partial sums meet in distributed shared memory before the one
  // write (see the end).
  const int G = H / Hkv;
  const int bkv = blockIdx.z * Hkv + blockIdx.y / S;
  const int rank = blockIdx.y % S;
  const int hqb = blockIdx.z * H + (blockIdx.y / S) * G;  // first query head of the group
  const int j0 = blockIdx.x * BM;
  // Query tiles t0 .. stream past (causal: key j is seen only by queries
  // i >= j; none when j0 >= Nq, and then Tq = 0 and the outputs are 0).
  // Group tile f = (query head in group) * Tq + (tile - t0); this CTA takes
  // f = f0 .. f0 + T - 1 (its own t = f - f0).
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
  if (warp >= 2 && warp < 6) {
    // The all-ones A operand: k = 0, 1, 2 are 1 (column c: k = 2c low, 2c + 1 high).
    const uint32_t one = 0x3F80u;  // bf16 1.0
    const uint32_t v[8] = {one | (one << 16), one, 0u, 0u, 0u, 0u, 0u, 0u};
    tmem_st8(tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kOnes, v);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 0) {
    // Producer.  Lane 0 issues the TMA copies; lane l writes the row-scalar
    // K step of query row l of every tile.
    const float inv_tau = 1.f / tau;
    auto load_row = [&](int f) {
      // (L, D, alpha, E) of row `lane` of streamed tile f; a row past N_q
      // (or a tile past the last) is marked by L = NaN.
      float4 v = make_float4(__int_as_float(0x7fc00000), 0.f, 0.f, 0.f);
      if (f >= T) return v;
      const int i = ((f0 + f) % Tq + t0) * BQ + lane;
      if (i < Nq) {
        const size_t o = static_cast<size_t>(hqb + (f0 + f) / Tq) * Nq + i;
        v = make_float4(L[o], D[o], alpha[o], E[o]);
      }
      return v;
    };
    if (lane == 0) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mUQ);
      tma_prefetch_desc(&mdO);
      mbar_expect_tx(&sm.bar_kv, 8 * HALF_BLOCK);
      for (int h = 0; h < 2; ++h) {
        tma_load_3d(sm.kb[0][h], &mK, &sm.bar_kv, 64 * h, j0, bkv);
        tma_load_3d(sm.kb[1][h], &mUK, &sm.bar_kv, 64 * h, j0, bkv);
        tma_load_3d(sm.kb[2][h], &mV, &sm.bar_kv, 64 * h, j0, bkv);
        tma_load_3d(sm.kb[3][h], &mUV, &sm.bar_kv, 64 * h, j0, bkv);
      }
    }
    float4 cur = load_row(0);
    int issued = 0;
    for (int t = 0; t < T; ++t) {
      const int s = t % NST;
      if (t >= NST && !mbar_wait_warp(&sm.st_empty[s], ((t / NST) - 1) & 1, abort_flag, err))
        break;
      // Stage 3 is the U_K block: wait until warpgroup 0 has copied U_K out.
      if (t == NST - 1 && !mbar_wait_warp(&sm.a_ready, 0, abort_flag, err)) break;
      if (lane == 0) {
        const int row = ((f0 + t) % Tq + t0) * BQ, fz = hqb + (f0 + t) / Tq;
        mbar_expect_tx(&sm.st_full[s], STAGE_BYTES);
        for (int h = 0; h < 2; ++h) {
          tma_load_3d(stage_tile(sm, s, h, 0), &mQ, &sm.st_full[s], 64 * h, row, fz);
          tma_load_3d(stage_tile(sm, s, h, 1), &mUQ, &sm.st_full[s], 64 * h, row, fz);
          tma_load_3d(stage_tile(sm, s, h, 2), &mdO, &sm.st_full[s], 64 * h, row, fz);
        }
      }
      {
        const bool pad = cur.x != cur.x;
        const float vals[4] = {pad ? -kFar : -cur.x * inv_tau, -cur.z * inv_tau, -cur.y,
                               -fmaf(cur.z, cur.y, cur.w)};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int row = lane + BQ * (q & 1);  // -L/tau, -alpha/tau ; -D, -(alpha D + E)
          uint8_t* base = stage_ex(sm, s, q >> 1) + (row >> 3) * 256 + (row & 7) * 16;
          const uint2 hm_l0 = split3_bf16(vals[q]);
          *reinterpret_cast<uint4*>(base) = make_uint4(hm_l0.x, hm_l0.y, 0u, 0u);
          *reinterpret_cast<uint4*>(base + 128) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.st_full[s]);
      issued = t + 1;
      cur = load_row(t + 1);  // lands while the ring is full
    }
    if (lane == 0) {
      // No copy may still be in flight when the CTA exits.
      drain_wait(&sm.bar_kv, 0);
      for (int t = issued > NST ? issued - NST : 0; t < issued; ++t)
        drain_wait(&sm.st_full[t % NST], (t / NST) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (whole warp, one elected lane issues) ----------------
    constexpr uint32_t idS64 = idesc_bf16(BM, 2 * BQ, false);  // N = 64, B K-major
    constexpr uint32_t idS32 = idesc_bf16(BM, BQ, false);      // N = 32, B K-major
    constexpr uint32_t idO = idesc_bf16(BM, DH, true);         // N = 128, B MN-major
    uint64_t dK[2], dV[2], dUV[2], dQ[2], ddO[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      dK[h] = smem_desc_sw128(smem_u32(sm.kb[0][h]), 16, 1024);
      dV[h] = smem_desc_sw128(smem_u32(sm.kb[2][h]), 16, 1024);
      dUV[h] = smem_desc_sw128(smem_u32(sm.kb[3][h]), 16, 1024);
      dQ[h] = smem_desc_sw128(smem_u32(sm.st[0][h][0]), 16, 1024);  // Q (and Q; U_Q)
      ddO[h] = smem_desc_sw128(smem_u32(sm.st[0][h][2]), 16, 1024);
    }
    // MN-major N = 128 operands of the output GEMMs: columns 64..127 (half 1)
    // sit 3 tiles after columns 0..63 (half 0) of the same tensor.
    constexpr uint32_t kHalfStride = 3 * HALF_TILE;
    const uint64_t dQmn = smem_desc_sw128(smem_u32(sm.st[0][0][0]), kHalfStride, 1024);
    const uint64_t dUQmn = smem_desc_sw128(smem_u32(sm.st[0][0][1]), kHalfStride, 1024);
    const uint64_t ddOmn = smem_desc_sw128(smem_u32(sm.st[0][0][2]), kHalfStride, 1024);
    const uint64_t dEx0 = smem_desc_noswz(smem_u32(sm.ex[0][0]), 128, 256);
    constexpr uint64_t kExPG = EX_BYTES >> 4;
    // Start-address offsets (16-byte units) of stage s from stage 0: the
    // stages in the ring are STAGE_BYTES apart, stage 3 lies in the U_K block
    // (before the ring, so its offset is negative; the sums stay in range).
    const int64_t so3 = (static_cast<int64_t>(smem_u32(stage_tile(sm, NST - 1, 0, 0))) -
                         static_cast<int64_t>(smem_u32(sm.st[0][0][0]))) >> 4;
    const int64_t eo3 = (static_cast<int64_t>(smem_u32(stage_ex(sm, NST - 1, 0))) -
                         static_cast<int64_t>(smem_u32(sm.ex[0][0]))) >> 4;
    auto stage_off = [&](int s) -> uint64_t {
      return static_cast<uint64_t>(s < NST - 1 ? static_cast<int64_t>(s * STAGE_BYTES >> 4) : so3);
    };
    auto ex_off = [&](int s) -> uint64_t {
      return static_cast<uint64_t>(s < NST - 1 ? static_cast<int64_t>(s * 2 * EX_BYTES >> 4) : eo3);
    };
    const uint32_t sc = tbase + kSc;
    // Score GEMMs in two halves: S^T | F'^T, then dP^T | G^T (+ commit).
    auto issue_sf = [&](int t) {
      const uint64_t so = stage_off(t % NST);
      {
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const int h = kk >> 2;
          const uint64_t o = 2 * (kk & 3);
          mma_ss(sc + kColS, dK[h] + o, dQ[h] + so + o, idS64, kk > 0);  // [S^T | F'^T] = K [Q; U_Q]^T
          mma_ts(sc + kColF, tbase + kUKA + 8 * kk, dQ[h] + so + o, idS32, 1);  // F'^T += U_K Q^T
        }
        // [S^T | F'^T] += 1 [-L / tau | -alpha / tau]^T (the row-scalar K step)
        mma_ts(sc + kColS, tbase + kOnes, dEx0 + ex_off(t % NST), idS64, 1);
      }
    };
    auto issue_pg = [&](int t) {
      const uint64_t so = stage_off(t % NST);
      {
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const int h = kk >> 2;
          const uint64_t o = 2 * (kk & 3);
          mma_ss(sc + kColdP, dV[h] + o, ddO[h] + so + o, idS32, kk > 0);  // dP^T = V dO^T
          mma_ss(sc + kColG, dUV[h] + o, ddO[h] + so + o, idS32, kk > 0);  // G^T  = U_V dO^T
        }
        // [dP^T | G^T] += 1 [-D | -(alpha D + E)]^T
        mma_ts(sc + kColdP, tbase + kOnes, dEx0 + ex_off(t % NST) + kExPG, idS64, 1);
        mma_commit(&sm.sc_full);
      }
    };
    auto issue_outputs = [&](int t) {
      const int s = t % NST;
      const uint64_t so = stage_off(s);
      {
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          const uint64_t o = (uint64_t)(16 * 128 * kk) >> 4;  // 16 query rows further down
          const uint32_t acc = (t > 0 || kk > 0);
          mma_ts(tbase + kAccK, tbase + op_col(kOpdSt, kk), dQmn + so + o, idO, acc);  // d~K += d~S^T Q
          mma_ts(tbase + kAccK, tbase + op_col(kOpdS, kk), dUQmn + so + o, idO, 1);    //     +  dS^T U_Q
          mma_ts(tbase + kAccV, tbase + op_col(kOpW, kk), ddOmn + so + o, idO, acc);   // d~V += W^T dO
        }
        mma_commit(&sm.op_free);
        mma_commit(&sm.st_empty[s]);
      }
    };
    // One elected lane runs the whole schedule: every wait and every MMA.
    if (elect_one()) {
      bool ok = mbar_wait(&sm.bar_kv, 0, abort_flag, err) &&
                mbar_wait(&sm.a_ready, 0, abort_flag, err);
      for (int t = 0; ok && t < T; ++t) {
        // Tile t's data is normally in the ring before the S/F release of
        // tile t - 1 arrives: check it first, so the S/F GEMMs follow it.
        ok = mbar_wait(&sm.st_full[t % NST], (t / NST) & 1, abort_flag, err);
        if (!ok) break;
        if (t > 0) {
          ok = mbar_wait(&sm.sf_free, (t - 1) & 1, abort_flag, err);
          if (!ok) break;
        }
        tc_fence_after();
        issue_sf(t);
        if (t > 0) {
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
      // Warpgroup 0 copies its key row of U_K from the two 128-byte-swizzled
      // 64-column halves (16-byte chunk c of row r at chunk c ^ (r mod 8))
      // into TMEM: K step kk is chunks 2 (kk mod 4), 2 (kk mod 4) + 1 of
      // half kk / 4.
      ok = mbar_wait_warp(&sm.bar_kv, 0, abort_flag, err);
      if (ok) {
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint8_t* row = sm.kb[1][kk >> 2] + r * 128;
          const int c = 2 * (kk & 3);
          const uint4 a = *reinterpret_cast<const uint4*>(row + ((c ^ (r & 7)) << 4));
          const uint4 b = *reinterpret_cast<const uint4*>(row + (((c + 1) ^ (r & 7)) << 4));
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
      ok = ok && mbar_wait_warp(&sm.sc_full, t & 1, abort_flag, err);
      if (ok) {
        tc_fence_after();
        const int ibase = (tq + t0) * BQ + 16 * wg;
        if (causal && ibase < j0 + BM)
          ok = p2w_half<true>(sc, opb, wg, ibase, gj, c1, tau, sm, t, abort_flag, err);
        else
          ok = p2w_half<false>(sc, opb, wg, ibase, gj, c1, tau, sm, t, abort_flag, err);
      }
      if (++tq == Tq) tq = 0;
    }

    ok = mbar_wait_warp(&sm.out_full, 0, abort_flag, err) && ok;
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);
    tc_fence_after();
    const uint32_t acc_base = tbase + lane_off;
    // Stage this CTA's d~K | d~V rows in the resident block (every MMA is
    // done; it is no longer read), float4 c of row r at c ^ (r mod 8): a
    // thread holds one key row, so writing global memory straight from
    // registers would scatter each warp's float4 over 32 rows.  A CTA with no
    // tile (T = 0) never wrote its accumulators and stages zeros.  With a
    // cluster split the rows are summed over the cluster below; alone, the
    // CTA writes them out here, coalesced.
    constexpr int kRow4 = 2 * DH / 4;  // float4 per staged row
    float4* stage = reinterpret_cast<float4*>(&sm.kb[0][0][0]);
    float4* row = stage + r * kRow4;
#pragma unroll 1
    for (int h = 0; h < 4; ++h) {
      const int col = 64 * wg + 16 * h;
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
        const int ck = col / 4 + k, cv = DH / 4 + col / 4 + k;
        row[ck ^ (r & 7)] = make_float4(u2f(vk[4 * k]), u2f(vk[4 * k + 1]),
                                        u2f(vk[4 * k + 2]), u2f(vk[4 * k + 3]));
        row[cv ^ (r & 7)] = make_float4(u2f(vv[4 * k]), u2f(vv[4 * k + 1]),
                                        u2f(vv[4 * k + 2]), u2f(vv[4 * k + 3]));
      }
    }
    if (!SPLIT) {
      named_bar_sync(1, 256);
      const int tid = threadIdx.x - 64;
      for (int e = tid; e < BM * kRow4 && ok; e += 256) {
        const int rr = e / kRow4, c4 = e % kRow4;
        const int gjr = j0 + rr;
        if (gjr >= Nk) break;  // rows ascend with e
        const float4 v = stage[rr * kRow4 + (c4 ^ (rr & 7))];
        const bool isK = c4 < DH / 4;
        const size_t o =
            (static_cast<size_t>(bkv) * Nk + gjr) * DH + 4 * (isK ? c4 : c4 - DH / 4);
        if (isK)
          *reinterpret_cast<float4*>(dKt + o) = make_float4(tau * v.x, tau * v.y, tau * v.z, tau * v.w);
        else
          *reinterpret_cast<float4*>(dVt + o) = v;
      }
    }
  }

  if (SPLIT) {
    // Cluster rank q sums key rows [128 q / S, 128 (q + 1) / S) over the S
    // CTAs' staged partials and writes them once.  All threads pass both
    // cluster barriers; the second keeps every staged row alive until all
    // reads are done.
    cluster_sync();
    if (warp >= 2) {
      const uint32_t q = cluster_ctarank();
      const int rb = (BM * (int)q) / S, re = (BM * ((int)q + 1)) / S;
      const uint32_t stage = smem_u32(&sm.kb[0][0][0]);
      const int tid = threadIdx.x - 64;
      constexpr int kRow4 = 2 * DH / 4;  // float4 per staged row
      for (int e = tid; e < (re - rb) * kRow4; e += 256) {
        const int rr = rb + e / kRow4, c4 = e % kRow4;
        const uint32_t off = static_cast<uint32_t>((rr * kRow4 + (c4 ^ (rr & 7))) * 16);
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
          const size_t o =
              (static_cast<size_t>(bkv) * Nk + gjr) * DH + 4 * (isK ? c4 : c4 - DH / 4);
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

size_t tc_pass2_d128_smem() { return sizeof(SmemW2) + 1024; }

cudaError_t tc_launch_pass2_d128(const BobArgs& a, const CUtensorMap* maps128,
                                 const CUtensorMap* maps32) {
  // maps128: K, U_K, V, U_V with 128-row boxes; maps32: Q, U_Q, dO with
  // 32-row boxes; every box is 64 columns wide.
  const size_t smem = tc_pass2_d128_smem();
  cudaError_t e = tc_set_smem(reinterpret_cast<const void*>(tc_pass2_d128_kernel<false>), (int)smem);
  if (e != cudaSuccess) return e;
  // One CTA per key block of a shared head, or, when the key blocks cannot
  // fill the SMs, a cluster of S of them that splits the block's query tiles
  // S ways.
  e = tc_set_smem(reinterpret_cast<const void*>(tc_pass2_d128_kernel<true>), (int)smem);
  if (e != cudaSuccess) return e;
  const int tiles = (a.H / a.Hkv) * ((a.Nq + BQ - 1) / BQ);
  int S = 1;
  if (!a.whole_grid_only)
    e = tc_pass2_split(reinterpret_cast<const void*>(tc_pass2_d128_kernel<true>), smem,
                       ((a.Nk + BM - 1) / BM) * a.Hkv * a.B, tiles, &S);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Nk + BM - 1) / BM, a.Hkv * S, a.B);
  if (S == 1) {
    tc_pass2_d128_kernel<false><<<grid, NTHREADS, smem, a.stream>>>(
        maps128[0], maps128[1], maps128[2], maps128[3], maps32[0], maps32[1], maps32[2], a.L,
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
  return cudaLaunchKernelEx(&cfg, tc_pass2_d128_kernel<true>, maps128[0], maps128[1], maps128[2],
                            maps128[3], maps32[0], maps32[1], maps32[2], a.L, a.D, a.alpha,
                            a.E, a.dKt, a.dVt, a.H, a.Hkv, a.Nq, a.Nk, a.tau, a.causal ? 1 : 0,
                            S, a.err);
}

}  // namespace flashbob
