// Pass 1 of the exact attention backward-over-backward on sm_103a tensor
// cores: bf16 inputs, head dim 64, fp32 accumulation in tensor memory.
//
// "FlashBoB: I/O-Efficient Exact Backward-over-Backward for Softmax
// Attention" (paper notes), 关键设计 2: a block of query rows stays on chip
// while key/value column tiles stream past; P is recomputed from the saved
// logsumexp L; the six row accumulators (alpha, E0, B, R, Omega, d~dO0) are
// alpha-free, and 关键设计 1's affine correction
//     E = E0 - alpha D,  d~dO = d~dO0 - alpha O,  d~Q = tau (Omega - alpha R - E B)
// runs once in the epilogue, so every output row is written exactly once.
// R is carried as R' = dS K = R - D B (dS = P o (dP - D)), which turns the
// correction into d~Q = tau (Omega - alpha R' - E0 B): the same value, one
// bf16 operand fewer, and dS [U_K | K] yields Omega's dS U_K term and R' in
// one MMA (20 MMAs per tile instead of 22).
//
// CTA = 128 query rows (MMA M = 128, one TMEM lane per row), 320 threads:
//   warp 0      TMA producer: Q, dO, U_Q blocks once, then U_K, K, V, U_V
//               tiles of 32 key rows through a 6-stage mbarrier ring;
//   warp 1      TMEM allocator; one elected lane runs the MMA schedule;
//   warps 2-5   elementwise warpgroup 0 (tiles 0, 2, 4, ...),
//   warps 6-9   elementwise warpgroup 1 (tiles 1, 3, 5, ...).
// TMEM (512 columns x 128 lanes, fp32):
//   [0,64) B = P K   [64,128) d~dO0   [128,192) Omega   [192,256) R' = dS K
//   [256,384) score buffer 0, [384,512) score buffer 1, each holding
//   F' = Q U_K^T + U_Q K^T | S = Q K^T | dP = dO V^T | G = dO U_V^T (32 columns each).
// GEMMs that share an operand run as one wider MMA: Q [U_K; K]^T gives half
// of F' and S (N = 64), dO [V; U_V]^T gives dP and G (N = 64), P [K | U_V]
// gives B and the P U_V part of d~dO0 (N = 128), and dS [U_K | K] gives
// Omega's dS U_K part and R' (N = 128).  Once a warpgroup has read a score
// buffer it overwrites the dP | G half with the bf16 A operands (P, P o d~P0,
// dS, P o F) of the output GEMMs, which read A straight from TMEM.  The F' | S
// half is free as soon as the warpgroup holds the tile in registers, so the
// F'/S GEMMs of the tile two ahead run while it still computes; only the
// dP/G GEMMs wait for the output GEMMs (the tensor pipe runs MMAs in issue
// order, so they overwrite the operands after those have been read).
#include "internal.h"
#include "tc_common.cuh"

namespace flashbob {
namespace {
using namespace tc;

constexpr int BM = kTcRows;      // 128 query rows per CTA
constexpr int BN = kTcStream;    // 32 key rows per streamed tile
constexpr int DH = 64;           // head dim
constexpr int NST = 6;           // stages of the K/V/U_K/U_V ring
constexpr int NTHREADS = 320;
constexpr uint32_t BLOCK_BYTES = BM * DH * 2;  // 16 KiB
constexpr uint32_t TILE_BYTES = BN * DH * 2;   // 4 KiB
constexpr float kLog2e = 1.4426950408889634f;

// Epilogue staging: one 128 x 64 fp32 tile per output, rows padded to 68
// floats (a warp's float4 accesses to 32 consecutive rows then take the
// minimum four shared-memory wavefronts), in the ring, idle by then.
constexpr int kStageLd = DH + 4;
constexpr uint32_t kStageBytes = BM * kStageLd * 4;

struct Smem1 {
  alignas(1024) uint8_t q[BLOCK_BYTES];
  alignas(1024) uint8_t dO[BLOCK_BYTES];
  alignas(1024) uint8_t uq[BLOCK_BYTES];
  alignas(1024) uint8_t kv[NST][4][TILE_BYTES];  // U_K, K, V, U_V (U_K|K and V|U_V adjacent)
  float part_a[2][BM];
  float part_e[2][BM];
  uint64_t bar_q;
  uint64_t kv_full[NST];
  uint64_t kv_empty[NST];
  uint64_t sc_full[2];
  uint64_t sf_free[2];   // per buffer: the warpgroup holds the tile in registers
  uint64_t op_ready[2];  // per buffer: one arrive per elementwise warp
  uint64_t out_full;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(2 * kStageBytes <= sizeof(Smem1::kv), "epilogue staging fits in the ring");

// Score buffer layout (columns): F' at 0, S at 32, dP at 64, G at 96.
constexpr uint32_t kColF = 0, kColS = 32, kColdP = 64, kColG = 96;
// TMEM columns of the bf16 operand slots inside a score buffer, for the two
// K = 16 steps (chunks) of the output GEMMs: the dP | G half.  A warpgroup
// reads the whole buffer before it writes any slot.
__device__ __forceinline__ constexpr uint32_t slot_P(int c) { return 64 + 8 * c; }
__device__ __forceinline__ constexpr uint32_t slot_PdPt(int c) { return 80 + 8 * c; }
__device__ __forceinline__ constexpr uint32_t slot_dS(int c) { return 96 + 8 * c; }
__device__ __forceinline__ constexpr uint32_t slot_PF(int c) { return 112 + 8 * c; }
// Score buffers: tile t in buffer t mod 2, at column 256 + 128 (t mod 2).
__device__ __forceinline__ int p1_buf(int t) { return t & 1; }
__device__ __forceinline__ uint32_t p1_buf_col(int t) { return 256 + 128 * (t & 1); }
// Output accumulators.
constexpr uint32_t kAccB = 0, kAccdO = 64, kAccW = 128, kAccR = 192;  // R' = dS K

// One 16-column chunk of a score buffer, one row per thread: from S, dP, F',
// G form P = exp(S - L) and the four bf16 A operands of the output GEMMs, add
// to the row sums alpha and E0 (kept as two partial sums, even and odd
// columns), and write the operands to the chunk's slots.  Two columns per
// step in the paired fp32 instructions.
template <bool MASKED, int C>
__device__ __forceinline__ void p1_chunk(uint32_t sc, const uint32_t (&s)[16],
                                         const uint32_t (&dp)[16], const uint32_t (&f)[16],
                                         const uint32_t (&g)[16], int col0, int jmax, float c1,
                                         float Lr2, float Dr, float tau, float2& a_acc,
                                         float2& e_acc) {
  uint32_t oP[8], oPdPt[8], odS[8], oPF[8];
  const int jbase = col0 + 16 * C;
  const float2 c12 = make_float2(c1, c1), nL = make_float2(-Lr2, -Lr2);
  const float2 nD = make_float2(-Dr, -Dr), tau2 = make_float2(tau, tau);
#pragma unroll
  for (int e = 0; e < 16; e += 2) {
    const float2 t = ffma2(f2(s[e], s[e + 1]), c12, nL);
    float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
    if (MASKED) {
      if (jbase + e > jmax) p.x = 0.f;
      if (jbase + e + 1 > jmax) p.y = 0.f;
    }
    const float2 x = fadd2(f2(dp[e], dp[e + 1]), nD);           // dP - D
    const float2 ft = fmul2(f2(f[e], f[e + 1]), tau2);           // F = tau F'
    const float2 dpt0 = ffma2(ft, x, f2(g[e], g[e + 1]));       // d~P0 = F o (dP - D) + G
    const float2 pdpt = fmul2(p, dpt0), ds = fmul2(p, x), pf = fmul2(p, ft);
    a_acc = fadd2(a_acc, pf);
    e_acc = fadd2(e_acc, pdpt);
    oP[e >> 1] = pack_bf16x2(p.x, p.y);
    oPdPt[e >> 1] = pack_bf16x2(pdpt.x, pdpt.y);
    odS[e >> 1] = pack_bf16x2(ds.x, ds.y);
    oPF[e >> 1] = pack_bf16x2(pf.x, pf.y);
  }
  tmem_st8(sc + slot_P(C), oP);
  tmem_st8(sc + slot_PdPt(C), oPdPt);
  tmem_st8(sc + slot_dS(C), odS);
  tmem_st8(sc + slot_PF(C), oPF);
}

// One 32-column tile, one row per thread: read all of S, F', dP, G (both
// 16-column chunks) with a single wait and free the F' | S half, form the
// bf16 A operands of the output GEMMs in the dP | G half, and hand the tile
// to the MMA issuer once they are in TMEM.
template <bool MASKED>
__device__ __forceinline__ void p1_tile(uint32_t sc, uint64_t* sf_free, uint64_t* ready,
                                        int col0, int jmax,
                                        float c1, float Lr2, float Dr, float tau, float2& a_acc,
                                        float2& e_acc) {
  uint32_t s0[16], dp0[16], f0[16], g0[16], s1[16], dp1[16], f1[16], g1[16];
  tmem_ld16(sc + kColS, s0);
  tmem_ld16(sc + kColdP, dp0);
  tmem_ld16(sc + kColF, f0);
  tmem_ld16(sc + kColG, g0);
  tmem_ld16(sc + kColS + 16, s1);
  tmem_ld16(sc + kColdP + 16, dp1);
  tmem_ld16(sc + kColF + 16, f1);
  tmem_ld16(sc + kColG + 16, g1);
  tmem_wait_ld();
  tc_fence_before();
  warp_arrive(sf_free);  // F' | S may be overwritten
  p1_chunk<MASKED, 0>(sc, s0, dp0, f0, g0, col0, jmax, c1, Lr2, Dr, tau, a_acc, e_acc);
  p1_chunk<MASKED, 1>(sc, s1, dp1, f1, g1, col0, jmax, c1, Lr2, Dr, tau, a_acc, e_acc);
  tmem_wait_st();
  tc_fence_before();
  warp_arrive(ready);
}

__global__ void __launch_bounds__(NTHREADS, 1)
    tc_pass1_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mdO,
                    const __grid_constant__ CUtensorMap mUQ, const __grid_constant__ CUtensorMap mK,
                    const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mUK,
                    const __grid_constant__ CUtensorMap mUV, const float* __restrict__ O,
                    const float* __restrict__ L, const float* __restrict__ D,
                    float* __restrict__ dQt, float* __restrict__ ddOt,
                    float* __restrict__ alpha, float* __restrict__ E, int H, int Hkv, int Nq,
                    int Nk, float tau, int causal, unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  Smem1& sm = *reinterpret_cast<Smem1*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                        ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.z * H + blockIdx.y;
  // key/value head shared by this query head (grouped-query attention)
  const int bkv = blockIdx.z * Hkv + blockIdx.y / (H / Hkv);
  // Causal: the last row blocks see the most keys, so they start first.
  const int row0 = (causal ? gridDim.x - 1 - blockIdx.x : blockIdx.x) * BM;
  const int col_end = causal ? min(Nk, row0 + BM) : Nk;  // keys j <= i under the causal mask
  const int T = (col_end + BN - 1) / BN;
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
      mbar_init(&sm.sf_free[b], 4);
    }
    mbar_init(&sm.out_full, 1);
    sm.abort_flag = 0;
    fence_barrier_init();
    // The resident block's copy starts now, while warp 1 allocates TMEM.
    mbar_expect_tx(&sm.bar_q, 3 * BLOCK_BYTES);
    tma_load_3d(sm.q, &mQ, &sm.bar_q, 0, row0, bh);
    tma_load_3d(sm.dO, &mdO, &sm.bar_q, 0, row0, bh);
    tma_load_3d(sm.uq, &mUQ, &sm.bar_q, 0, row0, bh);
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mK);
      tma_prefetch_desc(&mV);
      tma_prefetch_desc(&mUK);
      tma_prefetch_desc(&mUV);
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int s = t % NST;
        if (t >= NST && !mbar_wait(&sm.kv_empty[s], ((t / NST) - 1) & 1, abort_flag, err)) break;
        mbar_expect_tx(&sm.kv_full[s], 4 * TILE_BYTES);
        tma_load_3d(sm.kv[s][0], &mUK, &sm.kv_full[s], 0, t * BN, bkv);
        tma_load_3d(sm.kv[s][1], &mK, &sm.kv_full[s], 0, t * BN, bkv);
        tma_load_3d(sm.kv[s][2], &mV, &sm.kv_full[s], 0, t * BN, bkv);
        tma_load_3d(sm.kv[s][3], &mUV, &sm.kv_full[s], 0, t * BN, bkv);
        issued = t + 1;
      }
      // No copy may still be in flight when the CTA exits.
      drain_wait(&sm.bar_q, 0);
      for (int t = issued > NST ? issued - NST : 0; t < issued; ++t)
        drain_wait(&sm.kv_full[t % NST], (t / NST) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (whole warp, one elected lane issues) ----------------
    {
      constexpr uint32_t idS32 = idesc_bf16(BM, BN, false);       // N = 32, B K-major
      constexpr uint32_t idS64 = idesc_bf16(BM, 2 * BN, false);   // N = 64, B K-major
      constexpr uint32_t idO64 = idesc_bf16(BM, DH, true);        // N = 64, B MN-major
      constexpr uint32_t idO128 = idesc_bf16(BM, 2 * DH, true);   // N = 128, B MN-major
      // Descriptors of the resident blocks and of stage 0; a k-step adds
      // 32 bytes (16 bf16 inside the swizzled row) and a stage adds
      // 4 * TILE_BYTES to the start-address field (address >> 4).
      const uint64_t dq0 = smem_desc_sw128(smem_u32(sm.q), 16, 1024);
      const uint64_t ddo0 = smem_desc_sw128(smem_u32(sm.dO), 16, 1024);
      const uint64_t duq0 = smem_desc_sw128(smem_u32(sm.uq), 16, 1024);
      const uint32_t kv0 = smem_u32(sm.kv[0][0]);
      const uint64_t dUK0 = smem_desc_sw128(kv0, 16, 1024);                  // U_K (and U_K;K)
      const uint64_t dK0 = smem_desc_sw128(kv0 + TILE_BYTES, 16, 1024);      // K
      const uint64_t dV0 = smem_desc_sw128(kv0 + 2 * TILE_BYTES, 16, 1024);  // V (and V;U_V)
      const uint64_t dUV0 = smem_desc_sw128(kv0 + 3 * TILE_BYTES, 16, 1024);
      // MN-major [K | U_V] (second half 2 tiles on) and [U_K | K] (1 tile on).
      const uint64_t dKUV0 = smem_desc_sw128(kv0 + TILE_BYTES, 2 * TILE_BYTES, 1024);
      const uint64_t dUKK0 = smem_desc_sw128(kv0, TILE_BYTES, 1024);
      // One elected lane runs the whole schedule below: every wait and every
      // MMA, with no warp-wide broadcast between them (the MMA-warp time per
      // tile is what bounds this pass).
      // Score GEMMs of tile t in two halves: F' | S, then dP | G (+ commit).
      auto issue_sf = [&](int t) {
        const uint64_t so = (uint64_t)((t % NST) * 4 * TILE_BYTES) >> 4;
        const uint32_t sc = tbase + p1_buf_col(t);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint64_t o = 2 * kk;  // 32 bytes >> 4
          mma_ss(sc + kColF, dq0 + o, dUK0 + so + o, idS64, kk > 0);  // [F' | S] = Q [U_K; K]^T
          mma_ss(sc + kColF, duq0 + o, dK0 + so + o, idS32, 1);       // F' += U_Q K^T
        }
      };
      // Issued after the output GEMMs of tile t - 2, so the commit also
      // covers their reads of the operand slots that tile t's warpgroup is
      // about to overwrite.
      auto issue_pg = [&](int t) {
        const uint64_t so = (uint64_t)((t % NST) * 4 * TILE_BYTES) >> 4;
        const uint32_t sc = tbase + p1_buf_col(t);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint64_t o = 2 * kk;
          mma_ss(sc + kColdP, ddo0 + o, dV0 + so + o, idS64, kk > 0);  // [dP | G] = dO [V; U_V]^T
        }
        mma_commit(&sm.sc_full[p1_buf(t)]);
      };
      auto issue_outputs = [&](int t) {
        const int s = t % NST;
        const uint64_t so = (uint64_t)(s * 4 * TILE_BYTES) >> 4;
        const uint32_t sc = tbase + p1_buf_col(t);
        {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint64_t o = (uint64_t)(16 * 128 * c) >> 4;  // 16 key rows further down
            const uint32_t acc = (t > 0 || c > 0);
            mma_ts(tbase + kAccB, sc + slot_P(c), dKUV0 + so + o, idO128, acc);  // [B | d~dO0] += P [K | U_V]
            mma_ts(tbase + kAccW, sc + slot_dS(c), dUKK0 + so + o, idO128, acc); // [Omega | R'] += dS [U_K | K]
            mma_ts(tbase + kAccW, sc + slot_PdPt(c), dK0 + so + o, idO64, 1);    // Omega += (P o d~P0) K
            mma_ts(tbase + kAccdO, sc + slot_PF(c), dV0 + so + o, idO64, 1);     // d~dO0 += (P o F) V
          }
          mma_commit(&sm.kv_empty[s]);
        }
      };
      if (elect_one()) {
        bool ok = mbar_wait(&sm.bar_q, 0, abort_flag, err);
        tc_fence_after();
        for (int t = 0; ok && t < 2 && t < T; ++t) {  // both score buffers
          ok = mbar_wait(&sm.kv_full[t % NST], (t / NST) & 1, abort_flag, err);
          tc_fence_after();
          if (ok) {
            issue_sf(t);
            issue_pg(t);
          }
        }
        for (int t = 0; ok && t < T; ++t) {
          const uint32_t ph = (t >> 1) & 1;  // phase of this warpgroup's barriers
          if (t + 2 < T) {  // the warpgroup holds tile t in registers: F' | S of t + 2
            ok = mbar_wait(&sm.sf_free[t & 1], ph, abort_flag, err) &&
                 mbar_wait(&sm.kv_full[(t + 2) % NST], ((t + 2) / NST) & 1, abort_flag, err);
            if (!ok) break;
            tc_fence_after();
            issue_sf(t + 2);
          }
          ok = mbar_wait(&sm.op_ready[t & 1], ph, abort_flag, err);
          if (!ok) break;
          tc_fence_after();
          issue_outputs(t);
          if (t + 2 < T) issue_pg(t + 2);  // after the output GEMMs have read the operands
        }
        mma_commit(&sm.out_full);  // every MMA issued above has finished
      }
      __syncwarp();
    }
  } else {
    // ---------------- elementwise warpgroups + epilogue ----------------
    const int wg = (warp - 2) >> 2;      // 0 or 1
    const int quad = warp & 3;           // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane;      // row inside the block = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int gr = row0 + r;
    const size_t rowvec = static_cast<size_t>(bh) * Nq + gr;
    const float c1 = tau * kLog2e;
    const float Lr2 = gr < Nq ? L[rowvec] * kLog2e : 0.f;
    const float Dr = gr < Nq ? D[rowvec] : 0.f;
    float2 a_acc = make_float2(0.f, 0.f), e_acc = make_float2(0.f, 0.f);
    bool ok = true;

    for (int u = 0;; ++u) {
      const int t = 2 * u + wg;
      if (t >= T) break;
      const uint32_t sc = tbase + lane_off + 256 + 128 * wg;  // buffer t mod 2 = wg
      // tcgen05.ld/st are warp-collective: take the decision warp-uniformly.
      ok = mbar_wait_warp(&sm.sc_full[wg], u & 1, abort_flag, err);
      if (!ok) break;
      tc_fence_after();
      const int col0 = t * BN;
      // Columns past Nk, or (causal) past this row, get P = 0.  Only tiles
      // that reach past Nk or past the block's first row take the masked path.
      const bool masked = (col0 + BN > Nk) || (causal && col0 + BN - 1 > row0);
      const int jmax = causal ? min(Nk - 1, gr) : Nk - 1;
      if (masked) {
        p1_tile<true>(sc, &sm.sf_free[wg], &sm.op_ready[wg], col0, jmax, c1, Lr2, Dr, tau,
                           a_acc, e_acc);
      } else {
        p1_tile<false>(sc, &sm.sf_free[wg], &sm.op_ready[wg], col0, jmax, c1, Lr2, Dr, tau,
                            a_acc, e_acc);
      }
    }

    // Epilogue: combine the two warpgroups' row sums, then the affine
    // correction; warpgroup wg forms output columns [32 wg, 32 wg + 32).
    sm.part_a[wg][r] = a_acc.x + a_acc.y;
    sm.part_e[wg][r] = e_acc.x + e_acc.y;
    named_bar_sync(1, 256);
    const float al = sm.part_a[0][r] + sm.part_a[1][r];
    const float E0 = sm.part_e[0][r] + sm.part_e[1][r];
    const float Ei = E0 - al * Dr;
    ok = mbar_wait_warp(&sm.out_full, 0, abort_flag, err) && ok;
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);
    tc_fence_after();
    const uint32_t acc_base = tbase + lane_off;
    // Every MMA is done, so the ring is idle: the block's rows of O come in
    // through shared memory with coalesced loads (256 threads, 16 float4 per
    // row), each thread forms its row's outputs there, and the tiles leave
    // with coalesced stores.  d~dO overwrites O in place.
    float* st_o = reinterpret_cast<float*>(&sm.kv[0][0][0]);  // O, then d~dO
    float* st_q = st_o + BM * kStageLd;                         // d~Q
    const int tid = threadIdx.x - 64;                           // 0 .. 255
    const int rows = min(BM, Nq - row0);
    const size_t blk = (static_cast<size_t>(bh) * Nq + row0) * DH;
    for (int f = tid; f < rows * (DH / 4); f += 256) {
      const int rr = f / (DH / 4), c4 = f % (DH / 4);
      *reinterpret_cast<float4*>(st_o + rr * kStageLd + 4 * c4) =
          reinterpret_cast<const float4*>(O + blk)[f];
    }
    named_bar_sync(1, 256);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int col = 32 * wg + 16 * h;
      uint32_t vb[16], vr[16], vw[16], vo[16];
      tmem_ld16(acc_base + kAccB + col, vb);
      tmem_ld16(acc_base + kAccR + col, vr);
      tmem_ld16(acc_base + kAccW + col, vw);
      tmem_ld16(acc_base + kAccdO + col, vo);
      tmem_wait_ld();
      if (gr < Nq) {
        float4* o4 = reinterpret_cast<float4*>(st_o + r * kStageLd + col);
        float4* q4 = reinterpret_cast<float4*>(st_q + r * kStageLd + col);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 ov = o4[k];  // d~dO = d~dO0 - alpha O
          o4[k] = make_float4(u2f(vo[4 * k + 0]) - al * ov.x, u2f(vo[4 * k + 1]) - al * ov.y,
                              u2f(vo[4 * k + 2]) - al * ov.z, u2f(vo[4 * k + 3]) - al * ov.w);
          float4 qv;  // d~Q = tau (Omega - alpha R' - E0 B)
          qv.x = tau * (u2f(vw[4 * k + 0]) - al * u2f(vr[4 * k + 0]) - E0 * u2f(vb[4 * k + 0]));
          qv.y = tau * (u2f(vw[4 * k + 1]) - al * u2f(vr[4 * k + 1]) - E0 * u2f(vb[4 * k + 1]));
          qv.z = tau * (u2f(vw[4 * k + 2]) - al * u2f(vr[4 * k + 2]) - E0 * u2f(vb[4 * k + 2]));
          qv.w = tau * (u2f(vw[4 * k + 3]) - al * u2f(vr[4 * k + 3]) - E0 * u2f(vb[4 * k + 3]));
          q4[k] = qv;
        }
      }
    }
    named_bar_sync(1, 256);
    if (ok) {
      for (int f = tid; f < rows * (DH / 4); f += 256) {
        const int rr = f / (DH / 4), c4 = f % (DH / 4);
        reinterpret_cast<float4*>(ddOt + blk)[f] =
            *reinterpret_cast<const float4*>(st_o + rr * kStageLd + 4 * c4);
        reinterpret_cast<float4*>(dQt + blk)[f] =
            *reinterpret_cast<const float4*>(st_q + rr * kStageLd + 4 * c4);
      }
    }
    if (ok && wg == 0 && gr < Nq) {
      alpha[rowvec] = al;
      E[rowvec] = Ei;
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

size_t tc_pass1_smem() { return sizeof(Smem1) + 1024; }

cudaError_t tc_launch_pass1(const BobArgs& a, const CUtensorMap* maps128,
                            const CUtensorMap* maps32) {
  // maps128: Q, dO, U_Q with 128-row boxes; maps32: K, V, U_K, U_V with 32-row boxes.
  const size_t smem = tc_pass1_smem();
  cudaError_t e = tc_set_smem(reinterpret_cast<const void*>(tc_pass1_kernel), (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Nq + BM - 1) / BM, a.H, a.B);
  tc_pass1_kernel<<<grid, NTHREADS, smem, a.stream>>>(
      maps128[0], maps128[1], maps128[2], maps32[0], maps32[1], maps32[2], maps32[3], a.O, a.L,
      a.D, a.dQt, a.ddOt, a.alpha, a.E, a.H, a.Hkv, a.Nq, a.Nk, a.tau,
      a.causal ? 1 : 0, a.err);
  return cudaGetLastError();
}

}  // namespace flashbob
