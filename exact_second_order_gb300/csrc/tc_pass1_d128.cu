// Pass 1 of the exact attention backward-over-backward on sm_103a tensor
// cores for head dim 128 (bf16 inputs, fp32 accumulation in tensor memory).
//
// "FlashBoB: I/O-Efficient Exact Backward-over-Backward for Softmax
// Attention" (paper notes), 关键设计 2: a block of 128 query rows stays on
// chip while key/value tiles stream past and every output row is written
// once.  At d = 128 the four alpha-free accumulators of 关键设计 1 (B, R,
// Omega, d~dO0, 128 fp32 columns each) would fill all 512 TMEM columns, so
// this kernel takes the other exact route the same section allows: it
// streams the key tiles twice.
//   phase A: scores S, F' = U_Q K^T + Q U_K^T, dP = dO V^T, G = dO U_V^T and
//            the row sums alpha = sum_j P F and E0 = sum_j P d~P0 only;
//            then E = E0 - alpha D.
//   phase B: the same scores again; with alpha and E known per row,
//            d~S = P o (d~P0 - alpha dP - E), dS = P o (dP - D) and
//            W = P o (F - alpha) are final, and
//              d~Q  = tau (d~S K + dS U_K),   d~dO = P U_V + W V
//            accumulate directly (two 128-column accumulators).
// The GEMM count per key is 5 (phase A) + 9 (phase B) instead of 11; the
// benchmark's FLOP convention still counts the 11 of the one-phase form.
//
// CTA = 128 query rows, 320 threads: warp 0 TMA (Q, dO, U_Q once; K, U_K,
// V, U_V tiles of 32 key rows through a 4-slot ring, each tensor as two
// 64-column halves in the 128-byte swizzle), warp 1 TMEM allocation and MMA
// issue, warps 2-5 / 6-9 elementwise warpgroups on alternate tiles.
// Phase A has no accumulators, so it takes 64 keys per tile: two adjacent
// ring slots hold, per 64-column half, K_a K_b U_K,a U_K,b V_a V_b U_V,a
// U_V,b (a, b the two 32-key halves), and each K step is three MMAs with
// N = 128, 64, 128: [S | F'] = Q [K; U_K]^T, F' += U_Q K^T, [dP | G] =
// dO [V; U_V]^T, into a 256-column score buffer per warpgroup (all of TMEM).
// Phase B: [0,128) d~Q accumulator (without tau), [128,256) d~dO
// accumulator, [256,384) and [384,512) score buffers S | F' | dP | G (32
// columns each) of 32-key tiles; a warpgroup reads a buffer one 16-column
// chunk at a time and overwrites the columns of that chunk with its bf16 A
// operands d~S, dS, P, W of the output GEMMs.
//
// Instantiated with JVP = true the kernel computes the attention JVP along
// (U_Q, U_K, U_V) instead (no dO): one pass over the key tiles with S and F'
// only, operands P and P o F, O'0 = P U_V + (P o F) V in the d~dO
// accumulator, and O' = O'0 - L' O, L' = alpha in the epilogue.  Its d~Q
// columns [0,128) are free, so Q and U_Q are copied there once as bf16 A
// operands and its score GEMMs read only the key tile from shared memory.
#include "internal.h"
#include "tc_common.cuh"

namespace flashbob {
namespace {
using namespace tc;

constexpr int BM = kTcRows;    // 128 query rows per CTA
constexpr int BN = kTcStream;  // 32 key rows per streamed tile
constexpr int DH = 128;
constexpr int NST = 4;  // ring slots of BN keys; phase A pairs slots (0, 1) and (2, 3)
constexpr int NTHREADS = 320;
constexpr uint32_t HALF_BLOCK = BM * 64 * 2;  // 16 KiB: 128 rows x 64 columns
constexpr uint32_t HALF_TILE = BN * 64 * 2;   // 4 KiB: 32 rows x 64 columns
constexpr uint32_t STAGE_BYTES = 2 * 4 * HALF_TILE;
constexpr float kLog2e = 1.4426950408889634f;

struct SmemW1 {
  alignas(1024) uint8_t q[2][HALF_BLOCK];    // Q, columns 0..63 and 64..127
  alignas(1024) uint8_t dO[2][HALF_BLOCK];
  alignas(1024) uint8_t uq[2][HALF_BLOCK];
  // Phase B: [slot][half][K, U_K, V, U_V].  Phase A: slots 2p, 2p + 1 as one
  // region [half][K_a, K_b, U_K,a, U_K,b, V_a, V_b, U_V,a, U_V,b].
  alignas(1024) uint8_t kv[NST][2][4][HALF_TILE];
  float2 part[BM];  // (alpha, E0) partial row sums passed between the warpgroups
  uint64_t bar_q;
  uint64_t kv_full[NST];
  uint64_t kv_empty[NST];
  uint64_t sc_full[2];
  uint64_t op_ready[2];
  uint64_t out_full;
  uint64_t a_ready;  // the JVP: Q and U_Q are in TMEM (8 warps)
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(SmemW1) + 1024 <= 232448, "shared memory");

constexpr uint32_t kColS = 0, kColF = 32, kColdP = 64, kColG = 96;
constexpr uint32_t kAccQ = 0, kAccdO = 128;
// The JVP (no d~Q accumulator): Q and U_Q as bf16 A operands, K step kk at +8 kk.
constexpr uint32_t kJvpQA = 0, kJvpUQA = 64;
// Phase-B operand slots inside a score buffer: chunk c (key columns
// 16c..16c+15) writes only the S and F' columns of its own chunk, which it
// has already read.
__device__ __forceinline__ constexpr uint32_t slot_dSt(int c) { return 16 * c; }
__device__ __forceinline__ constexpr uint32_t slot_dS(int c) { return 16 * c + 8; }
__device__ __forceinline__ constexpr uint32_t slot_P(int c) { return kColF + 16 * c; }
__device__ __forceinline__ constexpr uint32_t slot_W(int c) { return kColF + 16 * c + 8; }

// Phase-A score buffer (256 columns, 64 keys): S | F' | dP | G, 64 each.
constexpr uint32_t kAColS = 0, kAColF = 64, kAColdP = 128, kAColG = 192;

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

// Chunk c (keys 16c .. 16c + 15) of a phase-A buffer.
__device__ __forceinline__ void load_chunk_a(uint32_t sc, int c, Chunk& x) {
  tmem_ld16(sc + kAColS + 16 * c, x.s);
  tmem_ld16(sc + kAColdP + 16 * c, x.dp);
  tmem_ld16(sc + kAColF + 16 * c, x.f);
  tmem_ld16(sc + kAColG + 16 * c, x.g);
}

// The element-wise functions below take two columns per step in the paired
// fp32 instructions; the row sums are kept as two partial sums (even and odd
// columns).

// Phase A on one chunk: the row sums alpha += P F and E0 += P d~P0.
template <bool MASKED>
__device__ __forceinline__ void phase_a_sums(const Chunk& x, int jbase, int jmax, float c1,
                                             float Lr2, float Dr, float tau, float2& a_acc,
                                             float2& e_acc) {
  const float2 c12 = make_float2(c1, c1), nL = make_float2(-Lr2, -Lr2);
  const float2 nD = make_float2(-Dr, -Dr), tau2 = make_float2(tau, tau);
#pragma unroll
  for (int e = 0; e < 16; e += 2) {
    const float2 t = ffma2(f2(x.s[e], x.s[e + 1]), c12, nL);
    float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
    if (MASKED) {
      if (jbase + e > jmax) p.x = 0.f;
      if (jbase + e + 1 > jmax) p.y = 0.f;
    }
    const float2 ft = fmul2(f2(x.f[e], x.f[e + 1]), tau2);
    const float2 dpt0 = ffma2(ft, fadd2(f2(x.dp[e], x.dp[e + 1]), nD), f2(x.g[e], x.g[e + 1]));
    a_acc = ffma2(p, ft, a_acc);
    e_acc = ffma2(p, dpt0, e_acc);
  }
}

// The JVP's chunk: P and P o F (into the P and W slots) and the row sum
// alpha = L' (no dO: dP = G = 0).
template <bool MASKED, int C>
__device__ __forceinline__ void jvp_chunk(uint32_t sc, const uint32_t (&s)[16],
                                          const uint32_t (&f)[16], int col0, int jmax, float c1,
                                          float Lr2, float tau, float2& a_acc) {
  uint32_t op[8], opf[8];
  const float2 c12 = make_float2(c1, c1), nL = make_float2(-Lr2, -Lr2);
  const float2 tau2 = make_float2(tau, tau);
#pragma unroll
  for (int e = 0; e < 16; e += 2) {
    const float2 t = ffma2(f2(s[e], s[e + 1]), c12, nL);
    float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
    if (MASKED) {
      if (col0 + 16 * C + e > jmax) p.x = 0.f;
      if (col0 + 16 * C + e + 1 > jmax) p.y = 0.f;
    }
    const float2 pf = fmul2(p, fmul2(f2(f[e], f[e + 1]), tau2));
    a_acc = fadd2(a_acc, pf);
    op[e >> 1] = pack_bf16x2(p.x, p.y);
    opf[e >> 1] = pack_bf16x2(pf.x, pf.y);
  }
  tmem_st8(sc + slot_P(C), op);
  tmem_st8(sc + slot_W(C), opf);
}

// Phase B on one 16-column chunk: the four bf16 A operands, written to TMEM.
template <bool MASKED, int C>
__device__ __forceinline__ void phase_b_chunk(uint32_t sc, const Chunk& x, int col0, int jmax,
                                              float c1, float Lr2, float Dr, float tau, float al,
                                              float Ei) {
  uint32_t odst[8], ods[8], op[8], ow[8];
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
    const float2 vw = fmul2(p, fadd2(ft, nal));                        // P (F - alpha)
    odst[e >> 1] = pack_bf16x2(vdst.x, vdst.y);
    ods[e >> 1] = pack_bf16x2(vds.x, vds.y);
    op[e >> 1] = pack_bf16x2(p.x, p.y);
    ow[e >> 1] = pack_bf16x2(vw.x, vw.y);
  }
  tmem_st8(sc + slot_dSt(C), odst);
  tmem_st8(sc + slot_dS(C), ods);
  tmem_st8(sc + slot_P(C), op);
  tmem_st8(sc + slot_W(C), ow);
}

template <bool JVP>
__global__ void __launch_bounds__(NTHREADS, 1)
    tc_pass1_d128_kernel(const __grid_constant__ CUtensorMap mQ,
                         const __grid_constant__ CUtensorMap mdO,
                         const __grid_constant__ CUtensorMap mUQ,
                         const __grid_constant__ CUtensorMap mK,
                         const __grid_constant__ CUtensorMap mV,
                         const __grid_constant__ CUtensorMap mUK,
                         const __grid_constant__ CUtensorMap mUV, const float* __restrict__ O,
                         const float* __restrict__ L, const float* __restrict__ D,
                         float* __restrict__ dQt, float* __restrict__ ddOt,
                         float* __restrict__ alpha, float* __restrict__ E, int H, int Hkv,
                         int Nq, int Nk, float tau, int causal, unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  SmemW1& sm = *reinterpret_cast<SmemW1*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.z * H + blockIdx.y;
  const int bkv = blockIdx.z * Hkv + blockIdx.y / (H / Hkv);  // shared key/value head
  const int row0 = (causal ? gridDim.x - 1 - blockIdx.x : blockIdx.x) * BM;
  const int col_end = causal ? min(Nk, row0 + BM) : Nk;  // keys j <= i under the causal mask
  const int T = (col_end + BN - 1) / BN;                                 // phase-B tiles
  const int TA = JVP ? 0 : (col_end + 2 * BN - 1) / (2 * BN);          // phase-A tiles
  // Ring uses in order: phase-A tile a takes uses 2a, 2a + 1 (the slot pair
  // a mod 2), phase-B tile t takes use 2 TA + t (slot (2 TA + t) mod NST).
  const int QN = 2 * TA + T;
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
      mbar_expect_tx(&sm.bar_q, (JVP ? 4 : 6) * HALF_BLOCK);
      for (int h = 0; h < 2; ++h) {
        tma_load_3d(sm.q[h], &mQ, &sm.bar_q, 64 * h, row0, bh);
        if (!JVP) tma_load_3d(sm.dO[h], &mdO, &sm.bar_q, 64 * h, row0, bh);
        tma_load_3d(sm.uq[h], &mUQ, &sm.bar_q, 64 * h, row0, bh);
      }
      int issued = 0;
      for (int q = 0; q < QN; ++q) {
        const int s = q % NST;
        if (q >= NST && !mbar_wait(&sm.kv_empty[s], ((q / NST) - 1) & 1, abort_flag, err)) break;
        mbar_expect_tx(&sm.kv_full[s], STAGE_BYTES);
        if (q < 2 * TA) {
          // Key rows 32 q .. of phase-A tile q / 2, half b = q & 1 of the
          // pair: it lands in both slots' memory, so the partner slot's
          // previous use must be released as well.
          const int b = q & 1;
          if (b == 0 && q + 1 >= NST &&
              !mbar_wait(&sm.kv_empty[s + 1], (((q + 1) / NST) - 1) & 1, abort_flag, err))
            break;
          uint8_t* pair = sm.kv[s & ~1][0][0];
          for (int h = 0; h < 2; ++h) {
            uint8_t* hp = pair + h * 8 * HALF_TILE;
            tma_load_3d(hp + (0 + b) * HALF_TILE, &mK, &sm.kv_full[s], 64 * h, q * BN, bkv);
            tma_load_3d(hp + (2 + b) * HALF_TILE, &mUK, &sm.kv_full[s], 64 * h, q * BN, bkv);
            tma_load_3d(hp + (4 + b) * HALF_TILE, &mV, &sm.kv_full[s], 64 * h, q * BN, bkv);
            tma_load_3d(hp + (6 + b) * HALF_TILE, &mUV, &sm.kv_full[s], 64 * h, q * BN, bkv);
          }
        } else {
          const int kt = q - 2 * TA;
          for (int h = 0; h < 2; ++h) {
            tma_load_3d(sm.kv[s][h][0], &mK, &sm.kv_full[s], 64 * h, kt * BN, bkv);
            tma_load_3d(sm.kv[s][h][1], &mUK, &sm.kv_full[s], 64 * h, kt * BN, bkv);
            tma_load_3d(sm.kv[s][h][2], &mV, &sm.kv_full[s], 64 * h, kt * BN, bkv);
            tma_load_3d(sm.kv[s][h][3], &mUV, &sm.kv_full[s], 64 * h, kt * BN, bkv);
          }
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
    constexpr uint32_t idS128 = idesc_bf16(BM, 4 * BN, false);  // N = 128, B K-major
    constexpr uint32_t idO128 = idesc_bf16(BM, DH, true);      // N = 128, B MN-major
    uint64_t dq[2], ddo[2], duq[2], dK[2], dV[2], dA[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      dq[h] = smem_desc_sw128(smem_u32(sm.q[h]), 16, 1024);
      ddo[h] = smem_desc_sw128(smem_u32(sm.dO[h]), 16, 1024);
      duq[h] = smem_desc_sw128(smem_u32(sm.uq[h]), 16, 1024);
      dK[h] = smem_desc_sw128(smem_u32(sm.kv[0][h][0]), 16, 1024);  // K (and K; U_K)
      dV[h] = smem_desc_sw128(smem_u32(sm.kv[0][h][2]), 16, 1024);  // V (and V; U_V)
      // Phase A: half h of pair 0 (K_a, K_b, U_K,a, U_K,b, then V_a ...).
      dA[h] = smem_desc_sw128(smem_u32(sm.kv[0][0][0]) + h * 8 * HALF_TILE, 16, 1024);
    }
    // MN-major N = 128 operands: columns 64..127 (half 1) sit 4 tiles after
    // columns 0..63 (half 0) of the same tensor.
    constexpr uint32_t kHalfStride = 4 * HALF_TILE;
    const uint64_t dKmn = smem_desc_sw128(smem_u32(sm.kv[0][0][0]), kHalfStride, 1024);
    const uint64_t dUKmn = smem_desc_sw128(smem_u32(sm.kv[0][0][1]), kHalfStride, 1024);
    const uint64_t dVmn = smem_desc_sw128(smem_u32(sm.kv[0][0][2]), kHalfStride, 1024);
    const uint64_t dUVmn = smem_desc_sw128(smem_u32(sm.kv[0][0][3]), kHalfStride, 1024);
    // Phase-A tile a: pair a mod 2, warpgroup a mod 2's 256-column buffer.
    // The slots are free again once these MMAs have read them.
    auto issue_scores_a = [&](int a) {
      const uint64_t po = (uint64_t)((a & 1) * 2 * STAGE_BYTES) >> 4;
      constexpr uint64_t kVUV = (uint64_t)(4 * HALF_TILE) >> 4;  // V_a V_b U_V,a U_V,b
      const uint32_t sc = tbase + 256 * (a & 1);
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        const int h = kk >> 2;
        const uint64_t o = 2 * (kk & 3);
        const uint32_t acc = kk > 0;
        mma_ss(sc + kAColS, dq[h] + o, dA[h] + po + o, idS128, acc);  // [S | F'] = Q [K; U_K]^T
        mma_ss(sc + kAColF, duq[h] + o, dA[h] + po + o, idS64, 1);    // F' += U_Q K^T
        mma_ss(sc + kAColdP, ddo[h] + o, dA[h] + po + kVUV + o, idS128, acc);  // [dP | G]
      }
      mma_commit(&sm.sc_full[a & 1]);
      mma_commit(&sm.kv_empty[(2 * a) % NST]);
      mma_commit(&sm.kv_empty[(2 * a + 1) % NST]);
    };
    auto issue_scores = [&](int t) {
      const uint64_t so = (uint64_t)(((2 * TA + t) % NST) * STAGE_BYTES) >> 4;
      const uint32_t sc = tbase + 256 + 128 * (t & 1);
      {
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const int h = kk >> 2;
          const uint64_t o = 2 * (kk & 3);  // 16 bf16 inside the 128-byte row
          const uint32_t acc = kk > 0;
          if (JVP) {  // A from TMEM
            mma_ts(sc + kColS, tbase + kJvpQA + 8 * kk, dK[h] + so + o, idS64, acc);
            mma_ts(sc + kColF, tbase + kJvpUQA + 8 * kk, dK[h] + so + o, idS32, 1);
            continue;
          }
          mma_ss(sc + kColS, dq[h] + o, dK[h] + so + o, idS64, acc);    // [S | F'] = Q [K; U_K]^T
          mma_ss(sc + kColF, duq[h] + o, dK[h] + so + o, idS32, 1);     // F' += U_Q K^T
          if (!JVP) mma_ss(sc + kColdP, ddo[h] + o, dV[h] + so + o, idS64, acc);  // [dP | G]
        }
        mma_commit(&sm.sc_full[t & 1]);
      }
    };
    auto issue_outputs = [&](int t) {
      const int s = (2 * TA + t) % NST;
      const uint64_t so = (uint64_t)(s * STAGE_BYTES) >> 4;
      const uint32_t sc = tbase + 256 + 128 * (t & 1);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint64_t o = (uint64_t)(16 * 128 * c) >> 4;  // 16 key rows further down
        const uint32_t acc = (t > 0 || c > 0);
        if (!JVP) {
          mma_ts(tbase + kAccQ, sc + slot_dSt(c), dKmn + so + o, idO128, acc);  // d~Q += d~S K
          mma_ts(tbase + kAccQ, sc + slot_dS(c), dUKmn + so + o, idO128, 1);    //  + dS U_K
        }
        mma_ts(tbase + kAccdO, sc + slot_P(c), dUVmn + so + o, idO128, acc);  // d~dO += P U_V
        mma_ts(tbase + kAccdO, sc + slot_W(c), dVmn + so + o, idO128, 1);     //  + W V (P o F V)
      }
      mma_commit(&sm.kv_empty[s]);
    };
    // One elected lane runs the whole schedule: every wait and every MMA.
    if (elect_one()) {
      bool ok = mbar_wait(&sm.bar_q, 0, abort_flag, err) &&
                (!JVP || mbar_wait(&sm.a_ready, 0, abort_flag, err));
      tc_fence_after();
      // Phase A: tile a goes to warpgroup a mod 2 once that warpgroup holds
      // tile a - 2 in registers.
      for (int a = 0; ok && a < TA; ++a) {
        if (a >= 2 && !(ok = mbar_wait(&sm.op_ready[a & 1], ((a >> 1) - 1) & 1, abort_flag, err)))
          break;
        ok = mbar_wait(&sm.kv_full[(2 * a) % NST], ((2 * a) / NST) & 1, abort_flag, err) &&
             mbar_wait(&sm.kv_full[(2 * a + 1) % NST], ((2 * a + 1) / NST) & 1, abort_flag, err);
        if (!ok) break;
        tc_fence_after();
        issue_scores_a(a);
      }
      // Phase B's score buffers [256, 512) were warpgroup 1's phase-A buffer
      // and its accumulators [0, 256) warpgroup 0's: wait until each
      // warpgroup holds its last phase-A tile in registers.  (This also keeps
      // sc_full from running two phases ahead of a warpgroup.)
      const int nA0 = (TA + 1) / 2, nA1 = TA / 2;  // phase-A tiles per warpgroup
      if (ok && nA0 > 0) ok = mbar_wait(&sm.op_ready[0], (nA0 - 1) & 1, abort_flag, err);
      if (ok && nA1 > 0) ok = mbar_wait(&sm.op_ready[1], (nA1 - 1) & 1, abort_flag, err);
      tc_fence_after();
      for (int t = 0; ok && t < 2 && t < T; ++t) {
        const int q = 2 * TA + t;
        ok = mbar_wait(&sm.kv_full[q % NST], (q / NST) & 1, abort_flag, err);
        tc_fence_after();
        if (ok) issue_scores(t);
      }
      for (int t = 0; ok && t < T; ++t) {
        ok = mbar_wait(&sm.op_ready[t & 1], ((t & 1 ? nA1 : nA0) + (t >> 1)) & 1, abort_flag, err);
        if (!ok) break;
        tc_fence_after();
        issue_outputs(t);
        if (t + 2 < T) {
          const int q = 2 * TA + t + 2;
          ok = mbar_wait(&sm.kv_full[q % NST], (q / NST) & 1, abort_flag, err);
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
    const float Dr = (!JVP && gr < Nq) ? D[rowvec] : 0.f;
    float2 a_acc = make_float2(0.f, 0.f), e_acc = make_float2(0.f, 0.f);
    float al = 0.f, Ei = 0.f;
    bool ok = true;
    const int jmax = causal ? min(Nk - 1, gr) : Nk - 1;
    // Both warpgroups' partial row sums meet here (each warpgroup passes
    // exactly once, named barrier 1): warpgroup 1 hands its sums over,
    // warpgroup 0 forms alpha and E = E0 - alpha D and hands them back.
    auto combine = [&]() {
      const float a_own = a_acc.x + a_acc.y, e_own = e_acc.x + e_acc.y;
      if (wg == 1) sm.part[r] = make_float2(a_own, e_own);
      named_bar_sync(1, 256);
      if (wg == 0) {
        const float2 o = sm.part[r];
        al = a_own + o.x;
        Ei = (e_own + o.y) - al * Dr;
        sm.part[r] = make_float2(al, Ei);
      }
      named_bar_sync(1, 256);
      if (wg == 1) {
        const float2 o = sm.part[r];
        al = o.x;
        Ei = o.y;
      }
    };

    if (JVP) {
      // Copy this thread's row of Q (warpgroup 0) or U_Q (warpgroup 1) from
      // the two 128-byte-swizzled TMA halves (16-byte chunk c of row r at
      // chunk c ^ (r mod 8)) into TMEM: K step kk is chunks 2 (kk mod 4) and
      // 2 (kk mod 4) + 1 of half kk / 4.
      ok = mbar_wait_warp(&sm.bar_q, 0, abort_flag, err);
      if (ok) {
        const uint32_t col = wg == 0 ? kJvpQA : kJvpUQA;
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
    }

    // u counts this warpgroup's tiles (phase A, then phase B): sc_full and
    // op_ready phases.  Warp-uniform decisions (tcgen05.ld/st are
    // warp-collective); after a failed wait keep looping so both warpgroups
    // reach the named barriers.
    int u = 0;
    for (int a = wg; a < TA; a += 2, ++u) {
      ok = ok && mbar_wait_warp(&sm.sc_full[wg], u & 1, abort_flag, err);
      if (!ok) continue;
      tc_fence_after();
      const uint32_t sca = tbase + lane_off + 256 * wg;
#pragma unroll 1
      for (int g = 0; g < 2; ++g) {  // keys 32 g .. 32 g + 31 of the tile
        Chunk x0, x1;
        load_chunk_a(sca, 2 * g, x0);
        load_chunk_a(sca, 2 * g + 1, x1);
        tmem_wait_ld();
        if (g == 1) {
          tc_fence_before();
          warp_arrive(&sm.op_ready[wg]);  // the buffer is in registers
        }
        const int cg = 2 * BN * a + BN * g;
        if ((cg + BN > Nk) || (causal && cg + BN - 1 > row0)) {
          phase_a_sums<true>(x0, cg, jmax, c1, Lr2, Dr, tau, a_acc, e_acc);
          phase_a_sums<true>(x1, cg + 16, jmax, c1, Lr2, Dr, tau, a_acc, e_acc);
        } else {
          phase_a_sums<false>(x0, cg, jmax, c1, Lr2, Dr, tau, a_acc, e_acc);
          phase_a_sums<false>(x1, cg + 16, jmax, c1, Lr2, Dr, tau, a_acc, e_acc);
        }
      }
    }
    if (!JVP) combine();

    const uint32_t sc = tbase + lane_off + 256 + 128 * wg;
    for (int t = wg; t < T; t += 2, ++u) {
      ok = ok && mbar_wait_warp(&sm.sc_full[wg], u & 1, abort_flag, err);
      if (!ok) continue;
      tc_fence_after();
      const int col0 = t * BN;
      const bool masked = (col0 + BN > Nk) || (causal && col0 + BN - 1 > row0);
      if (JVP) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t sv[16], fv[16];
          tmem_ld16(sc + kColS + 16 * c, sv);
          tmem_ld16(sc + kColF + 16 * c, fv);
          tmem_wait_ld();
          if (c == 0) {
            if (masked) jvp_chunk<true, 0>(sc, sv, fv, col0, jmax, c1, Lr2, tau, a_acc);
            else jvp_chunk<false, 0>(sc, sv, fv, col0, jmax, c1, Lr2, tau, a_acc);
          } else {
            if (masked) jvp_chunk<true, 1>(sc, sv, fv, col0, jmax, c1, Lr2, tau, a_acc);
            else jvp_chunk<false, 1>(sc, sv, fv, col0, jmax, c1, Lr2, tau, a_acc);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(&sm.op_ready[wg]);
      } else {
        {
          Chunk x;
          load_chunk(sc, 0, x);
          tmem_wait_ld();
          if (masked)
            phase_b_chunk<true, 0>(sc, x, col0, jmax, c1, Lr2, Dr, tau, al, Ei);
          else
            phase_b_chunk<false, 0>(sc, x, col0, jmax, c1, Lr2, Dr, tau, al, Ei);
        }
        {
          Chunk x;
          load_chunk(sc, 1, x);
          tmem_wait_ld();
          if (masked)
            phase_b_chunk<true, 1>(sc, x, col0, jmax, c1, Lr2, Dr, tau, al, Ei);
          else
            phase_b_chunk<false, 1>(sc, x, col0, jmax, c1, Lr2, Dr, tau, al, Ei);
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(&sm.op_ready[wg]);
      }
    }
    if (JVP) combine();

    // Epilogue: warpgroup wg writes output columns [64 wg, 64 wg + 64).
    ok = mbar_wait_warp(&sm.out_full, 0, abort_flag, err) && ok;
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);
    tc_fence_after();
    const uint32_t acc_base = tbase + lane_off;
#pragma unroll 1
    for (int h = 0; h < 4; ++h) {
      const int col = 64 * wg + 16 * h;
      uint32_t vq[16], vo[16];
      if (!JVP) tmem_ld16(acc_base + kAccQ + col, vq);
      tmem_ld16(acc_base + kAccdO + col, vo);
      tmem_wait_ld();
      if (JVP && ok && gr < Nq) {  // O' = O'0 - L' O
        const size_t off = rowvec * DH + col;
        const float4* o4 = reinterpret_cast<const float4*>(O + off);
        float4* d4 = reinterpret_cast<float4*>(ddOt + off);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 ov = o4[k];
          d4[k] = make_float4(u2f(vo[4 * k]) - al * ov.x, u2f(vo[4 * k + 1]) - al * ov.y,
                              u2f(vo[4 * k + 2]) - al * ov.z, u2f(vo[4 * k + 3]) - al * ov.w);
        }
      }
      if (!JVP && ok && gr < Nq) {
        const size_t off = rowvec * DH + col;
        float4* q4 = reinterpret_cast<float4*>(dQt + off);
        float4* d4 = reinterpret_cast<float4*>(ddOt + off);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          q4[k] = make_float4(tau * u2f(vq[4 * k]), tau * u2f(vq[4 * k + 1]),
                              tau * u2f(vq[4 * k + 2]), tau * u2f(vq[4 * k + 3]));
          d4[k] = make_float4(u2f(vo[4 * k]), u2f(vo[4 * k + 1]), u2f(vo[4 * k + 2]),
                              u2f(vo[4 * k + 3]));
        }
      }
    }
    if (ok && wg == 0 && gr < Nq) {
      alpha[rowvec] = al;
      if (!JVP) E[rowvec] = Ei;
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
  // maps128: Q, dO, U_Q with 128-row boxes; maps32: K, V, U_K, U_V with 32-row
  // boxes; every box is 64 columns wide (one half of a 128-column row).
  const size_t smem = tc_pass1_d128_smem();
  cudaError_t e = tc_set_smem(reinterpret_cast<const void*>(tc_pass1_d128_kernel<false>), (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Nq + BM - 1) / BM, a.H, a.B);
  tc_pass1_d128_kernel<false><<<grid, NTHREADS, smem, a.stream>>>(
      maps128[0], maps128[1], maps128[2], maps32[0], maps32[1], maps32[2], maps32[3], a.O, a.L,
      a.D, a.dQt, a.ddOt, a.alpha, a.E, a.H, a.Hkv, a.Nq, a.Nk, a.tau, a.causal ? 1 : 0, a.err);
  return cudaGetLastError();
}

}  // namespace flashbob

namespace flashbob {

cudaError_t tc_launch_jvp_d128(const JvpArgs& a, const CUtensorMap* maps128,
                               const CUtensorMap* maps32) {
  // maps128: Q, U_Q with 128-row boxes; maps32: K, V, U_K, U_V with 32-row
  // boxes (64-column halves).
  const size_t smem = tc_pass1_d128_smem();
  cudaError_t e = tc_set_smem(reinterpret_cast<const void*>(tc_pass1_d128_kernel<true>), (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Nq + BM - 1) / BM, a.H, a.B);
  tc_pass1_d128_kernel<true><<<grid, NTHREADS, smem, a.stream>>>(
      maps128[0], maps128[0], maps128[1], maps32[0], maps32[1], maps32[2], maps32[3], a.O, a.L,
      nullptr, nullptr, a.Od, a.Ld, nullptr, a.H, a.Hkv, a.Nq, a.Nk, a.tau, a.causal ? 1 : 0,
      a.err);
  return cudaGetLastError();
}

}  // namespace flashbob
