// Pass 1 of the exact attention backward-over-backward on sm_103a tensor
// cores for head dim 128 (bf16 inputs, fp32 accumulation in tensor memory):
// its second launch, the rows pass.
//
// "FlashBoB: I/O-Efficient Exact Backward-over-Backward for Softmax
// Attention" (paper notes), 关键设计 2: a block of 128 query rows stays on
// chip while key/value tiles stream past and every output row is written
// once.  At d = 128 the four alpha-free accumulators of 关键设计 1 (B, R,
// Omega, d~dO0, 128 fp32 columns each) would fill all 512 TMEM columns, so
// the pass takes another exact route in two launches:
//   1. the attention JVP along (U_Q, U_K, U_V) with E (tc_jvp_d128.cu):
//      alpha = L', d~dO = O' and E = dO . d~dO - alpha D;
//   2. this kernel: with alpha and E known per row, d~S = P o (d~P0 -
//      alpha dP - E) and dS = P o (dP - D) are final and d~Q = tau (d~S K +
//      dS U_K) accumulates directly in one 128-column accumulator.
// GEMMs per key: 5 (JVP) + 7 (rows: S, F' twice, dP, G, and two output
// GEMMs) = 12 instead of the one-phase form's 11; the benchmark's FLOP
// convention still counts 11.
//
// CTA = 128 query rows, 320 threads: warp 0 TMA (Q, dO, U_Q once; K, U_K,
// V, U_V tiles of 32 key rows through a 4-slot ring, each tensor as two
// 64-column halves in the 128-byte swizzle), warp 1 TMEM allocation and MMA
// issue, warps 2-5 / 6-9 elementwise warpgroups on alternate tiles.  Q and
// U_Q are copied once from shared memory into TMEM as bf16 A operands (K
// step kk at +8 kk), so the S | F' score GEMMs read only the key tile from
// shared memory.
// TMEM: [0,128) the d~Q accumulator (without tau), [128,192) Q, [192,256)
// U_Q, [256,384) and [384,512) score buffers S | F' | dP | G (32 columns
// each).  A warpgroup reads a buffer one 16-column chunk at a time and
// overwrites the S and F' columns of that chunk with its bf16 A operands of
// the output GEMMs (d~S, dS).
#include "internal.h"
#include "tc_common.cuh"

namespace flashbob {
namespace {
using namespace tc;

constexpr int BM = kTcRows;    // 128 query rows per CTA
constexpr int BN = kTcStream;  // 32 key rows per streamed tile
constexpr int DH = 128;
constexpr int NST = 4;  // ring slots of BN keys
constexpr int NTHREADS = 320;
constexpr uint32_t HALF_BLOCK = BM * 64 * 2;  // 16 KiB: 128 rows x 64 columns
constexpr uint32_t HALF_TILE = BN * 64 * 2;   // 4 KiB: 32 rows x 64 columns
constexpr uint32_t STAGE_BYTES = 2 * 4 * HALF_TILE;
constexpr float kLog2e = 1.4426950408889634f;
// Epilogue staging: the block's 128 x 128 fp32 output tile, rows padded to
// 132 floats (a warp's float4 accesses to 32 consecutive rows then take the
// minimum four shared-memory wavefronts), in the ring, idle by then.
constexpr int kStageLd = DH + 4;

struct SmemW1 {
  alignas(1024) uint8_t q[2][HALF_BLOCK];    // Q, columns 0..63 and 64..127
  alignas(1024) uint8_t dO[2][HALF_BLOCK];
  alignas(1024) uint8_t uq[2][HALF_BLOCK];
  alignas(1024) uint8_t kv[NST][2][4][HALF_TILE];  // [slot][half][K, U_K, V, U_V]
  uint64_t bar_q;
  uint64_t kv_full[NST];
  uint64_t kv_empty[NST];
  uint64_t sc_full[2];
  uint64_t op_ready[2];
  uint64_t out_full;
  uint64_t a_ready;  // Q and U_Q are in TMEM (8 warps)
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(SmemW1) + 1024 <= 232448, "shared memory");
static_assert(BM * kStageLd * 4 <= sizeof(SmemW1::kv), "epilogue staging fits in the ring");

constexpr uint32_t kColS = 0, kColF = 32, kColdP = 64, kColG = 96;
constexpr uint32_t kAccQ = 0;           // d~Q
constexpr uint32_t kQA = 128, kUQA = 192;  // Q, U_Q as A operands
// Operand slots inside a score buffer: chunk c (key columns 16c..16c+15)
// writes only the S and F' columns of its own chunk, which it has already
// read.
__device__ __forceinline__ constexpr uint32_t slot_dSt(int c) { return 16 * c; }
__device__ __forceinline__ constexpr uint32_t slot_dS(int c) { return 16 * c + 8; }

// S, dP, F', G of one 16-column chunk of a score buffer, one row per thread.
struct Chunk {
  uint32_t s[16], dp[16], f[16], g[16];
};

__device__ __forceinline__ void load_chunk(uint32_t sc, int c, Chunk& x) {
  tmem_ld16(sc + kColS + 16 * c, x.s);
  tmem_ld16(sc + kColdP + 16 * c, x.dp);
  tmem_ld16(sc + kColF + 16 * c, x.f);
  tmem_ld16(sc + kColG + 16 * c, x.g);
}

// The element-wise functions below take two columns per step in the paired
// fp32 instructions; the row sums are kept as two partial sums (even and odd
// columns).

// The rows pass on one 16-column chunk: d~S and dS as bf16 A operands,
// written to TMEM.
template <bool MASKED, int C>
__device__ __forceinline__ void rows_chunk(uint32_t sc, const Chunk& x, int col0, int jmax,
                                           float c1, float Lr2, float Dr, float tau, float al,
                                           float Ei) {
  uint32_t odst[8], ods[8];
  const float2 c12 = make_float2(c1, c1), nL = make_float2(-Lr2, -Lr2);
  const float2 nD = make_float2(-Dr, -Dr), tau2 = make_float2(tau, tau);
  const float2 nal = make_float2(-al, -al), nEi = make_float2(-Ei, -Ei);
#pragma unroll
  for (int e = 0; e < 16; e += 2) {
    const float2 t = ffma2(f2(x.s[e], x.s[e + 1]), c12, nL);
    float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
    if (MASKED) {
      if (col0 + 16 * C + e > jmax) p.x = 0.f;
      if (col0 + 16 * C + e + 1 > jmax) p.y = 0.f;
    }
    const float2 dpv = f2(x.dp[e], x.dp[e + 1]);
    const float2 xx = fadd2(dpv, nD);                                  // dP - D
    const float2 ft = fmul2(f2(x.f[e], x.f[e + 1]), tau2);             // F = tau F'
    const float2 dpt0 = ffma2(ft, xx, f2(x.g[e], x.g[e + 1]));        // d~P0
    const float2 vdst = fmul2(p, fadd2(dpt0, ffma2(nal, dpv, nEi)));  // P (d~P0 - alpha dP - E)
    const float2 vds = fmul2(p, xx);
    odst[e >> 1] = pack_bf16x2(vdst.x, vdst.y);
    ods[e >> 1] = pack_bf16x2(vds.x, vds.y);
  }
  tmem_st8(sc + slot_dSt(C), odst);
  tmem_st8(sc + slot_dS(C), ods);
}

// The rows pass: reads alpha and E, writes d~Q.
__global__ void __launch_bounds__(NTHREADS, 1)
    tc_pass1_d128_kernel(const __grid_constant__ CUtensorMap mQ,
                         const __grid_constant__ CUtensorMap mdO,
                         const __grid_constant__ CUtensorMap mUQ,
                         const __grid_constant__ CUtensorMap mK,
                         const __grid_constant__ CUtensorMap mV,
                         const __grid_constant__ CUtensorMap mUK,
                         const __grid_constant__ CUtensorMap mUV,
                         const float* __restrict__ L, const float* __restrict__ D,
                         float* __restrict__ dQt, const float* __restrict__ alpha,
                         const float* __restrict__ E, int H, int Hkv,
                         int Nq, int Nk, float tau, int causal, unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  SmemW1& sm = *reinterpret_cast<SmemW1*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.z * H + blockIdx.y;
  const int bkv = blockIdx.z * Hkv + blockIdx.y / (H / Hkv);  // shared key/value head
  const int row0 = (causal ? gridDim.x - 1 - blockIdx.x : blockIdx.x) * BM;
  const int col_end = causal ? min(Nk, row0 + BM) : Nk;  // keys j <= i under the causal mask
  const int T = (col_end + BN - 1) / BN;                  // key tiles
  volatile int* abort_flag = &sm.abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(&sm.bar_q, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.sc_full[b], 1);
      mbar_init(&sm.op_ready[b], 4);
    }
    mbar_init(&sm.out_full, 1);
    mbar_init(&sm.a_ready, 8);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&mK);
      tma_prefetch_desc(&mV);
      tma_prefetch_desc(&mUK);
      tma_prefetch_desc(&mUV);
      mbar_expect_tx(&sm.bar_q, 6 * HALF_BLOCK);
      for (int h = 0; h < 2; ++h) {
        tma_load_3d(sm.q[h], &mQ, &sm.bar_q, 64 * h, row0, bh);
        tma_load_3d(sm.dO[h], &mdO, &sm.bar_q, 64 * h, row0, bh);
        tma_load_3d(sm.uq[h], &mUQ, &sm.bar_q, 64 * h, row0, bh);
      }
      int issued = 0;
      for (int q = 0; q < T; ++q) {
        const int s = q % NST;
        if (q >= NST && !mbar_wait(&sm.kv_empty[s], ((q / NST) - 1) & 1, abort_flag, err)) break;
        mbar_expect_tx(&sm.kv_full[s], STAGE_BYTES);
        for (int h = 0; h < 2; ++h) {
          tma_load_3d(sm.kv[s][h][0], &mK, &sm.kv_full[s], 64 * h, q * BN, bkv);
          tma_load_3d(sm.kv[s][h][1], &mUK, &sm.kv_full[s], 64 * h, q * BN, bkv);
          tma_load_3d(sm.kv[s][h][2], &mV, &sm.kv_full[s], 64 * h, q * BN, bkv);
          tma_load_3d(sm.kv[s][h][3], &mUV, &sm.kv_full[s], 64 * h, q * BN, bkv);
        }
        issued = q + 1;
      }
      // No copy may still be in flight when the CTA exits.
      drain_wait(&sm.bar_q, 0);
      for (int q = issued > NST ? issued - NST : 0; q < issued; ++q)
        drain_wait(&sm.kv_full[q % NST], (q / NST) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (whole warp, one elected lane issues) ----------------
    constexpr uint32_t idS32 = idesc_bf16(BM, BN, false);      // N = 32, B K-major
    constexpr uint32_t idS64 = idesc_bf16(BM, 2 * BN, false);  // N = 64, B K-major
    constexpr uint32_t idO128 = idesc_bf16(BM, DH, true);      // N = 128, B MN-major
    uint64_t ddo[2], dK[2], dV[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      ddo[h] = smem_desc_sw128(smem_u32(sm.dO[h]), 16, 1024);
      dK[h] = smem_desc_sw128(smem_u32(sm.kv[0][h][0]), 16, 1024);  // K (and K; U_K)
      dV[h] = smem_desc_sw128(smem_u32(sm.kv[0][h][2]), 16, 1024);  // V (and V; U_V)
    }
    // MN-major N = 128 operands: columns 64..127 (half 1) sit 4 tiles after
    // columns 0..63 (half 0) of the same tensor.
    constexpr uint32_t kHalfStride = 4 * HALF_TILE;
    const uint64_t dKmn = smem_desc_sw128(smem_u32(sm.kv[0][0][0]), kHalfStride, 1024);
    const uint64_t dUKmn = smem_desc_sw128(smem_u32(sm.kv[0][0][1]), kHalfStride, 1024);
    const uint64_t dVmn = smem_desc_sw128(smem_u32(sm.kv[0][0][2]), kHalfStride, 1024);
    const uint64_t dUVmn = smem_desc_sw128(smem_u32(sm.kv[0][0][3]), kHalfStride, 1024);
    auto issue_scores = [&](int t) {
      const uint64_t so = (uint64_t)((t % NST) * STAGE_BYTES) >> 4;
      const uint32_t sc = tbase + 256 + 128 * (t & 1);
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        const int h = kk >> 2;
        const uint64_t o = 2 * (kk & 3);  // 16 bf16 inside the 128-byte row
        const uint32_t acc = kk > 0;
        mma_ts(sc + kColS, tbase + kQA + 8 * kk, dK[h] + so + o, idS64, acc);  // [S | F'] = Q [K; U_K]^T
        mma_ts(sc + kColF, tbase + kUQA + 8 * kk, dK[h] + so + o, idS32, 1);   // F' += U_Q K^T
        mma_ss(sc + kColdP, ddo[h] + o, dV[h] + so + o, idS64, acc);  // [dP | G] = dO [V; U_V]^T
      }
      mma_commit(&sm.sc_full[t & 1]);
    };
    auto issue_outputs = [&](int t) {
      const int s = t % NST;
      const uint64_t so = (uint64_t)(s * STAGE_BYTES) >> 4;
      const uint32_t sc = tbase + 256 + 128 * (t & 1);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint64_t o = (uint64_t)(16 * 128 * c) >> 4;  // 16 key rows further down
        const uint32_t acc = (t > 0 || c > 0);
        mma_ts(tbase + kAccQ, sc + slot_dSt(c), dKmn + so + o, idO128, acc);  // d~Q += d~S K
        mma_ts(tbase + kAccQ, sc + slot_dS(c), dUKmn + so + o, idO128, 1);    //  + dS U_K
      }
      mma_commit(&sm.kv_empty[s]);
    };
    // One elected lane runs the whole schedule: every wait and every MMA.
    // Tile t goes to warpgroup t mod 2; the scores of t + 2 follow the
    // output GEMMs of t (they overwrite its buffer).
    if (elect_one()) {
      bool ok = mbar_wait(&sm.bar_q, 0, abort_flag, err) &&
                mbar_wait(&sm.a_ready, 0, abort_flag, err);
      tc_fence_after();
      for (int t = 0; ok && t < 2 && t < T; ++t) {
        ok = mbar_wait(&sm.kv_full[t % NST], (t / NST) & 1, abort_flag, err);
        tc_fence_after();
        if (ok) issue_scores(t);
      }
      for (int t = 0; ok && t < T; ++t) {
        ok = mbar_wait(&sm.op_ready[t & 1], (t >> 1) & 1, abort_flag, err);
        if (!ok) break;
        tc_fence_after();
        issue_outputs(t);
        if (t + 2 < T) {
          ok = mbar_wait(&sm.kv_full[(t + 2) % NST], ((t + 2) / NST) & 1, abort_flag, err);
          if (!ok) break;
          tc_fence_after();
          issue_scores(t + 2);
        }
      }
      mma_commit(&sm.out_full);  // every MMA issued above has finished
    }
    __syncwarp();
  } else {
    // ---------------- elementwise warpgroups + epilogue ----------------
    const int wg = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // row inside the block = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int gr = row0 + r;
    const size_t rowvec = static_cast<size_t>(bh) * Nq + gr;
    const float c1 = tau * kLog2e;
    const float Lr2 = gr < Nq ? L[rowvec] * kLog2e : 0.f;
    const float Dr = gr < Nq ? D[rowvec] : 0.f;
    // alpha and E come from the JVP launch.
    const float al_in = gr < Nq ? alpha[rowvec] : 0.f;
    const float E_in = gr < Nq ? E[rowvec] : 0.f;
    bool ok = true;
    const int jmax = causal ? min(Nk - 1, gr) : Nk - 1;

    // Copy this thread's row of Q (warpgroup 0) or U_Q (warpgroup 1) from
    // the two 128-byte-swizzled TMA halves (16-byte chunk c of row r at
    // chunk c ^ (r mod 8)) into TMEM: K step kk is chunks 2 (kk mod 4) and
    // 2 (kk mod 4) + 1 of half kk / 4.
    ok = mbar_wait_warp(&sm.bar_q, 0, abort_flag, err);
    if (ok) {
      const uint32_t col = wg == 0 ? kQA : kUQA;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint8_t* row = (wg == 0 ? sm.q[kk >> 2] : sm.uq[kk >> 2]) + r * 128;
        const int c = 2 * (kk & 3);
        const uint4 x = *reinterpret_cast<const uint4*>(row + ((c ^ (r & 7)) << 4));
        const uint4 y = *reinterpret_cast<const uint4*>(row + (((c + 1) ^ (r & 7)) << 4));
        const uint32_t v[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
        tmem_st8(tbase + lane_off + col + 8 * kk, v);
      }
      tmem_wait_st();
    }
    tc_fence_before();
    warp_arrive(&sm.a_ready);

    // u counts this warpgroup's tiles: sc_full and op_ready phases.
    // Warp-uniform decisions (tcgen05.ld/st are warp-collective); after a
    // failed wait keep looping so both warpgroups reach the named barriers.
    const uint32_t sc = tbase + lane_off + 256 + 128 * wg;
    int u = 0;
    for (int t = wg; t < T; t += 2, ++u) {
      ok = ok && mbar_wait_warp(&sm.sc_full[wg], u & 1, abort_flag, err);
      if (!ok) continue;
      tc_fence_after();
      const int col0 = t * BN;
      const bool masked = (col0 + BN > Nk) || (causal && col0 + BN - 1 > row0);
      {
        Chunk x;
        load_chunk(sc, 0, x);
        tmem_wait_ld();
        if (masked)
          rows_chunk<true, 0>(sc, x, col0, jmax, c1, Lr2, Dr, tau, al_in, E_in);
        else
          rows_chunk<false, 0>(sc, x, col0, jmax, c1, Lr2, Dr, tau, al_in, E_in);
      }
      {
        Chunk x;
        load_chunk(sc, 1, x);
        tmem_wait_ld();
        if (masked)
          rows_chunk<true, 1>(sc, x, col0, jmax, c1, Lr2, Dr, tau, al_in, E_in);
        else
          rows_chunk<false, 1>(sc, x, col0, jmax, c1, Lr2, Dr, tau, al_in, E_in);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(&sm.op_ready[wg]);
    }

    // Epilogue: warpgroup wg forms output columns [64 wg, 64 wg + 64) of its
    // row, d~Q = tau (d~S K + dS U_K).  Every MMA is done, so the ring is
    // idle: each thread stages its row there and the tile leaves with
    // coalesced stores (256 threads, 32 float4 per row).
    ok = mbar_wait_warp(&sm.out_full, 0, abort_flag, err) && ok;
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);
    tc_fence_after();
    const uint32_t acc_base = tbase + lane_off;
    float* st = reinterpret_cast<float*>(&sm.kv[0][0][0][0]);
    const int tid = threadIdx.x - 64;  // 0 .. 255
    const int rows = min(BM, Nq - row0);
    const size_t blk = (static_cast<size_t>(bh) * Nq + row0) * DH;
#pragma unroll 1
    for (int h = 0; h < 4; ++h) {
      const int col = 64 * wg + 16 * h;
      uint32_t v[16];
      tmem_ld16(acc_base + kAccQ + col, v);
      tmem_wait_ld();
      if (gr >= Nq) continue;
      float4* s4 = reinterpret_cast<float4*>(st + r * kStageLd + col);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        s4[k] = make_float4(tau * u2f(v[4 * k]), tau * u2f(v[4 * k + 1]),
                            tau * u2f(v[4 * k + 2]), tau * u2f(v[4 * k + 3]));
    }
    named_bar_sync(1, 256);
    if (ok) {
      for (int f = tid; f < rows * (DH / 4); f += 256) {
        const int rr = f / (DH / 4), c4 = f % (DH / 4);
        reinterpret_cast<float4*>(dQt + blk)[f] =
            *reinterpret_cast<const float4*>(st + rr * kStageLd + 4 * c4);
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

size_t tc_pass1_d128_smem() { return sizeof(SmemW1) + 1024; }

cudaError_t tc_launch_pass1_d128(const BobArgs& a, const CUtensorMap* maps128,
                                 const CUtensorMap* maps32) {
  // The rows launch of the d = 128 pass 1 (the JVP launch before it has
  // written alpha and E): d~Q.  maps128: Q, dO, U_Q with 128-row boxes;
  // maps32: K, V, U_K, U_V with 32-row boxes; every box is 64 columns wide
  // (one half of a 128-column row).
  const size_t smem = tc_pass1_d128_smem();
  cudaError_t e = tc_set_smem(reinterpret_cast<const void*>(tc_pass1_d128_kernel), (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Nq + BM - 1) / BM, a.H, a.B);
  tc_pass1_d128_kernel<<<grid, NTHREADS, smem, a.stream>>>(
      maps128[0], maps128[1], maps128[2], maps32[0], maps32[1], maps32[2], maps32[3], a.L, a.D,
      a.dQt, a.alpha, a.E, a.H, a.Hkv, a.Nq, a.Nk, a.tau, a.causal ? 1 : 0, a.err);
  return cudaGetLastError();
}

}  // namespace flashbob
