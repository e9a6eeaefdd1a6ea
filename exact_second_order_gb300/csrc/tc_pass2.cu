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
//   warp 0      TMA producer: Q, U_Q, dO tiles of 32 query rows through a
//               10-stage mbarrier ring;
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer;
//   warps 2-5 / 6-9   elementwise warpgroups 0 / 1 (even / odd tiles); at the
//               start they also copy their key row of K, U_K / V, U_V into TMEM.
// TMEM: [0,64) d~K accumulator, [64,128) d~V accumulator, [128,256) the
// resident K | V | U_K | U_V block as bf16 (the A operands of every score
// GEMM, so shared memory only feeds the 32-row B tiles), [256,384) and
// [384,512) score buffers S^T | F'^T | dP^T | G^T (32 columns each).
// K [Q; U_Q]^T gives S^T and half of F'^T in one N = 64 MMA.
#include "internal.h"
#include "tc_common.cuh"

namespace flashbob {
namespace {
using namespace tc;

constexpr int BM = kTcRows;    // 128 key rows per CTA
constexpr int BN = kTcStream;  // 32 query rows per streamed tile
constexpr int DH = 64;
constexpr int NST = 10;
constexpr int NTHREADS = 320;
constexpr uint32_t TILE_BYTES = BN * DH * 2;
constexpr float kLog2e = 1.4426950408889634f;

struct Smem2 {
  alignas(1024) uint8_t st[NST][3][TILE_BYTES];  // Q, U_Q, dO (Q|U_Q adjacent)
  float4 scal[2][2][BN];  // per warpgroup, double-buffered: (L log2 e, D, alpha, E)
  uint64_t st_full[NST];
  uint64_t st_empty[NST];
  uint64_t a_ready;
  uint64_t sc_full[2];
  uint64_t op_ready[2];  // per buffer: one arrive per elementwise warp
  uint64_t out_full;
  uint32_t tmem_base;
  int abort_flag;
};

// TMEM columns.
constexpr uint32_t kAccK = 0, kAccV = 64;
constexpr uint32_t kAK = 128, kAV = 160, kAUK = 192, kAUV = 224;  // 64 bf16 = 32 columns each
constexpr uint32_t kColS = 0, kColF = 32, kColdP = 64, kColG = 96;  // inside a score buffer

// bf16 operand slots inside a score buffer: chunk 0 writes only columns it
// has read (the first 16 of S^T and F'^T), chunk 1 only columns chunk 0 read.
__device__ __forceinline__ constexpr uint32_t slot_dS(int c) { return c ? 40 : 0; }
__device__ __forceinline__ constexpr uint32_t slot_dSt(int c) { return c ? 64 : 8; }
__device__ __forceinline__ constexpr uint32_t slot_W(int c) { return c ? 72 : 32; }

// 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Copy one 64-element bf16 row (zeros past N) into 32 TMEM columns.
// `row` is null for rows past N.
__device__ __forceinline__ void row_to_tmem(uint32_t taddr, const __nv_bfloat16* row) {
  uint32_t r[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) r[k] = 0u;
  if (row != nullptr) {
    const uint4* src = reinterpret_cast<const uint4*>(row);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint4 v = src[k];
      r[4 * k] = v.x;
      r[4 * k + 1] = v.y;
      r[4 * k + 2] = v.z;
      r[4 * k + 3] = v.w;
    }
  }
  tmem_st32(taddr, r);
}

// One 16-column chunk of a transposed score buffer, one key row per thread:
// with the row scalars of the streamed query rows form dS, d~S and W and
// write them as bf16 A operands over consumed columns.
template <bool MASKED, int C>
__device__ __forceinline__ void p2_chunk(uint32_t sc, const uint32_t (&s)[16],
                                         const uint32_t (&dp)[16], const uint32_t (&f)[16],
                                         const uint32_t (&g)[16], const float4* scal, int ibase,
                                         int gj, float c1, float tau) {
  uint32_t odS[8], odSt[8], oW[8];
#pragma unroll
  for (int e = 0; e < 16; e += 2) {
    float vds[2], vdst[2], vw[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = 16 * C + e + h;
      const float4 rs = scal[i];  // (L log2 e, D, alpha, E) of query row i
      float p = ex2_approx(fmaf(u2f(s[e + h]), c1, -rs.x));
      if (MASKED && ibase + i < gj) p = 0.f;
      const float dpv = u2f(dp[e + h]);
      const float x = dpv - rs.y;
      const float ft = u2f(f[e + h]) * tau;
      vds[h] = p * x;
      vdst[h] = p * (fmaf(ft, x, u2f(g[e + h])) - fmaf(rs.z, dpv, rs.w));
      vw[h] = p * (ft - rs.z);
    }
    odS[e >> 1] = pack_bf16x2(vds[0], vds[1]);
    odSt[e >> 1] = pack_bf16x2(vdst[0], vdst[1]);
    oW[e >> 1] = pack_bf16x2(vw[0], vw[1]);
  }
  tmem_st8(sc + slot_dS(C), odS);
  tmem_st8(sc + slot_dSt(C), odSt);
  tmem_st8(sc + slot_W(C), oW);
}

// One 32-column tile, one key row per thread (the same hand-off as pass 1);
// the two 16-column chunks are read one after the other, which keeps the
// register count within what 10 warps per SM allow.
template <bool MASKED>
__device__ __forceinline__ void p2_tile(uint32_t sc, uint64_t* ready, const float4* scal,
                                        int ibase, int gj, float c1, float tau) {
  {
    uint32_t s0[16], dp0[16], f0[16], g0[16];
    tmem_ld16(sc + kColS, s0);
    tmem_ld16(sc + kColdP, dp0);
    tmem_ld16(sc + kColF, f0);
    tmem_ld16(sc + kColG, g0);
    tmem_wait_ld();
    p2_chunk<MASKED, 0>(sc, s0, dp0, f0, g0, scal, ibase, gj, c1, tau);
  }
  {
    uint32_t s1[16], dp1[16], f1[16], g1[16];
    tmem_ld16(sc + kColS + 16, s1);
    tmem_ld16(sc + kColdP + 16, dp1);
    tmem_ld16(sc + kColF + 16, f1);
    tmem_ld16(sc + kColG + 16, g1);
    tmem_wait_ld();
    p2_chunk<MASKED, 1>(sc, s1, dp1, f1, g1, scal, ibase, gj, c1, tau);
  }
  tmem_wait_st();
  tc_fence_before();
  warp_arrive(ready);
}

__global__ void __launch_bounds__(NTHREADS, 1)
    tc_pass2_kernel(const __nv_bfloat16* __restrict__ K, const __nv_bfloat16* __restrict__ V,
                    const __nv_bfloat16* __restrict__ UK, const __nv_bfloat16* __restrict__ UV,
                    const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mdO,
                    const __grid_constant__ CUtensorMap mUQ, const float* __restrict__ L,
                    const float* __restrict__ D, const float* __restrict__ alpha,
                    const float* __restrict__ E, float* __restrict__ dKt,
                    float* __restrict__ dVt, int H, int N, float tau, int causal,
                    unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  Smem2& sm = *reinterpret_cast<Smem2*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                        ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.z * H + blockIdx.y;
  const int j0 = blockIdx.x * BM;
  // Query tiles t0 .. T-1 stream past; under the causal mask key j is seen
  // only by queries i >= j, so the tiles before the block are skipped.
  // Ring slots and barrier phases count tiles from t0.
  const int t0 = causal ? j0 / BN : 0;
  const int T = (N + BN - 1) / BN - t0;
  volatile int* abort_flag = &sm.abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(&sm.a_ready, 8);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&sm.st_full[s], 1);
      mbar_init(&sm.st_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.sc_full[b], 1);
      mbar_init(&sm.op_ready[b], 4);
    }
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
    if (lane == 0) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mdO);
      tma_prefetch_desc(&mUQ);
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int s = t % NST;
        if (t >= NST && !mbar_wait(&sm.st_empty[s], ((t / NST) - 1) & 1, abort_flag, err)) break;
        mbar_expect_tx(&sm.st_full[s], 3 * TILE_BYTES);
        tma_load_3d(sm.st[s][0], &mQ, &sm.st_full[s], 0, (t + t0) * BN, bh);
        tma_load_3d(sm.st[s][1], &mUQ, &sm.st_full[s], 0, (t + t0) * BN, bh);
        tma_load_3d(sm.st[s][2], &mdO, &sm.st_full[s], 0, (t + t0) * BN, bh);
        issued = t + 1;
      }
      for (int t = issued > NST ? issued - NST : 0; t < issued; ++t)
        drain_wait(&sm.st_full[t % NST], (t / NST) & 1);
    }
  } else if (warp == 1) {
    {  // MMA issuer: whole warp, one elected lane issues
      constexpr uint32_t idS32 = idesc_bf16(BM, BN, false);      // N = 32, B K-major
      constexpr uint32_t idS64 = idesc_bf16(BM, 2 * BN, false);  // N = 64, B K-major
      constexpr uint32_t idO = idesc_bf16(BM, DH, true);         // N = 64, B MN-major
      const uint32_t st0 = smem_u32(sm.st[0][0]);
      const uint64_t dQ0 = smem_desc_sw128(st0, 16, 1024);                   // Q (and Q;U_Q)
      const uint64_t dUQ0 = smem_desc_sw128(st0 + TILE_BYTES, 16, 1024);
      const uint64_t ddO0 = smem_desc_sw128(st0 + 2 * TILE_BYTES, 16, 1024);
      // One elected lane issues each group of MMAs as one straight block.
      auto issue_scores = [&](int t) {
        const uint64_t so = (uint64_t)((t % NST) * 3 * TILE_BYTES) >> 4;
        const uint32_t sc = tbase + 256 + 128 * (t & 1);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < DH / 16; ++kk) {
            const uint64_t o = 2 * kk;       // 32 bytes >> 4 along K in the B tiles
            const uint32_t ao = 8 * kk;      // 16 bf16 = 8 TMEM columns along K in A
            const uint32_t acc = kk > 0;
            mma_ts(sc + kColS, tbase + kAK + ao, dQ0 + so + o, idS64, acc);   // [S^T | F'^T] = K [Q; U_Q]^T
            mma_ts(sc + kColF, tbase + kAUK + ao, dQ0 + so + o, idS32, 1);    // F'^T += U_K Q^T
            mma_ts(sc + kColdP, tbase + kAV + ao, ddO0 + so + o, idS32, acc); // dP^T = V dO^T
            mma_ts(sc + kColG, tbase + kAUV + ao, ddO0 + so + o, idS32, acc); // G^T  = U_V dO^T
          }
          mma_commit(&sm.sc_full[t & 1]);
        }
        __syncwarp();
      };
      auto issue_outputs = [&](int t) {
        const int s = t % NST;
        const uint64_t so = (uint64_t)(s * 3 * TILE_BYTES) >> 4;
        const uint32_t sc = tbase + 256 + 128 * (t & 1);
        if (elect_one()) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint64_t o = (uint64_t)(16 * 128 * c) >> 4;  // 16 query rows further down
            const uint32_t acc = (t > 0 || c > 0);
            mma_ts(tbase + kAccK, sc + slot_dSt(c), dQ0 + so + o, idO, acc);  // d~K += d~S^T Q
            mma_ts(tbase + kAccK, sc + slot_dS(c), dUQ0 + so + o, idO, 1);    //     +  dS^T U_Q
            mma_ts(tbase + kAccV, sc + slot_W(c), ddO0 + so + o, idO, acc);   // d~V += W^T dO
          }
          mma_commit(&sm.st_empty[s]);
        }
        __syncwarp();
      };
      bool ok = mbar_wait_warp(&sm.a_ready, 0, abort_flag, err);  // K, V, U_K, U_V are in TMEM
      tc_fence_after();
      for (int t = 0; ok && t < 2 && t < T; ++t) {
        ok = mbar_wait_warp(&sm.st_full[t % NST], (t / NST) & 1, abort_flag, err);
        tc_fence_after();
        if (ok) issue_scores(t);
      }
      for (int t = 0; ok && t < T; ++t) {
        ok = mbar_wait_warp(&sm.op_ready[t & 1], (t >> 1) & 1, abort_flag, err);
        if (!ok) break;
        tc_fence_after();
        issue_outputs(t);
        if (t + 2 < T) {
          ok = mbar_wait_warp(&sm.st_full[(t + 2) % NST], ((t + 2) / NST) & 1, abort_flag, err);
          if (!ok) break;
          tc_fence_after();
          issue_scores(t + 2);
        }
      }
      if (elect_one()) mma_commit(&sm.out_full);
    }
  } else {
    const int wg = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // key row inside the block = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int gj = j0 + r;
    const size_t head = static_cast<size_t>(bh) * N;
    const float c1 = tau * kLog2e;
    const uint32_t sc = tbase + lane_off + 256 + 128 * wg;
    const bool loader = (warp & 3) == 0;  // one warp per warpgroup stages the row scalars
    bool ok = true;

    // Resident key block into TMEM: warpgroup 0 copies K and U_K, warpgroup
    // 1 copies V and U_V, one key row per thread.
    {
      const bool valid = gj < N;
      const size_t roff = valid ? (head + gj) * DH : 0;
      if (wg == 0) {
        row_to_tmem(tbase + lane_off + kAK, valid ? K + roff : nullptr);
        row_to_tmem(tbase + lane_off + kAUK, valid ? UK + roff : nullptr);
      } else {
        row_to_tmem(tbase + lane_off + kAV, valid ? V + roff : nullptr);
        row_to_tmem(tbase + lane_off + kAUV, valid ? UV + roff : nullptr);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(&sm.a_ready);
    }

    // Row scalars of a streamed tile, (L log2 e, D, alpha, E) per query row;
    // rows past N get L = +inf so that P = exp2(-inf) = 0.
    auto load_scalars = [&](int t) {
      const int i = (t + t0) * BN + lane;
      if (t < T && i < N)
        return make_float4(L[head + i] * kLog2e, D[head + i], alpha[head + i], E[head + i]);
      return make_float4(INFINITY, 0.f, 0.f, 0.f);
    };
    // The loader warp fetches the scalars one tile ahead into registers, so
    // their global-memory latency hides behind the current tile.
    if (loader) sm.scal[wg][0][lane] = load_scalars(wg);
    for (int u = 0;; ++u) {
      const int t = 2 * u + wg;
      if (t >= T) break;
      float4* scal = sm.scal[wg][u & 1];
      named_bar_sync(2 + wg, 128);  // scal is written; last tile's readers are done
      float4 next = make_float4(0.f, 0.f, 0.f, 0.f);
      if (loader) next = load_scalars(t + 2);
      // Warp-uniform decision (tcgen05.ld/st are warp-collective); after a
      // failed wait keep looping so every thread passes the same named
      // barriers, but skip the work.
      ok = ok && mbar_wait_warp(&sm.sc_full[wg], u & 1, abort_flag, err);
      if (ok) {
        tc_fence_after();
        // Causal: queries i < j (this thread's key row) get P = 0; only the
        // tiles that overlap the key block take the masked path.  Rows past N
        // carry L = +inf, so their P is 0 on both paths.
        const int ibase = (t + t0) * BN;
        if (causal && ibase < j0 + BM) {
          p2_tile<true>(sc, &sm.op_ready[wg], scal, ibase, gj, c1, tau);
        } else {
          p2_tile<false>(sc, &sm.op_ready[wg], scal, ibase, gj, c1, tau);
        }
      }
      // Every thread passed this iteration's barrier, so nobody still reads
      // the other buffer.
      if (loader) sm.scal[wg][(u + 1) & 1][lane] = next;
    }

    ok = mbar_wait_warp(&sm.out_full, 0, abort_flag, err) && ok;
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);
    tc_fence_after();
    const uint32_t acc_base = tbase + lane_off;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int col = 32 * wg + 16 * h;
      uint32_t vk[16], vv[16];
      tmem_ld16(acc_base + kAccK + col, vk);
      tmem_ld16(acc_base + kAccV + col, vv);
      tmem_wait_ld();
      if (ok && gj < N) {
        const size_t off = (head + gj) * DH + col;
        float4* k4 = reinterpret_cast<float4*>(dKt + off);
        float4* v4 = reinterpret_cast<float4*>(dVt + off);
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

cudaError_t tc_launch_pass2(const BobArgs& a, const CUtensorMap* maps32) {
  // maps32: Q, dO, U_Q with 32-row boxes; K, V, U_K, U_V are read directly.
  const size_t smem = tc_pass2_smem();
  cudaError_t e = cudaFuncSetAttribute(tc_pass2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.N + BM - 1) / BM, a.H, a.B);
  tc_pass2_kernel<<<grid, NTHREADS, smem, a.stream>>>(
      (const __nv_bfloat16*)a.K, (const __nv_bfloat16*)a.V, (const __nv_bfloat16*)a.UK,
      (const __nv_bfloat16*)a.UV, maps32[0], maps32[1], maps32[2], a.L, a.D, a.alpha, a.E,
      a.dKt, a.dVt, a.H, a.N, a.tau, a.causal ? 1 : 0, a.err);
  return cudaGetLastError();
}

}  // namespace flashbob
