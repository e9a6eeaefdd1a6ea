// Attention JVP (forward-mode derivative along the tangents U_Q, U_K, U_V)
// on sm_103a tensor cores: bf16 inputs, head dim 64, fp32 accumulation in
// tensor memory.
//
// The forward of "FlashAttention 的反向传播设计" (section 一): S = tau Q K^T,
// P = exp(S - L), O = P V.  Along the tangents the scores move by
// F = tau (U_Q K^T + Q U_K^T), the log-sum-exp by L' = sum_j P_ij F_ij, the
// probabilities by P o (F - L'), so
//     O' = (P o F) V + P U_V - L' O.
// This is the row pass of "FlashBoB" (paper notes, 关键设计 1/2) with dO = 0:
// its alpha is L' and its d~dO is O'.
//
// CTA = 128 query rows (MMA M = 128, one TMEM lane per row), 448 threads:
//   warp 0      TMA producer: the Q and U_Q blocks once, then U_K, K, V, U_V
//               tiles of 64 key rows through a 6-stage mbarrier ring;
//   warp 1      TMEM allocator; one elected lane runs the MMA schedule;
//   warps 2-5 / 6-9 / 10-13   elementwise warpgroups 0 / 1 / 2: warpgroup
//               w takes the tiles t = w mod 3, in score buffer w.
// With no dP or G scores the JVP needs two scores per element, so its tiles
// are 64 keys wide: the score GEMMs are Q [U_K; K]^T (N = 128, half of F'
// and S) and U_Q K^T (N = 64), against N = 64 and N = 32 for 32-key tiles,
// and every tcgen05.mma costs the tensor pipe tens of cycles whatever its
// width.
// TMEM (512 columns x 128 lanes):
//   [0,64)      O'0 = (P o F) V + P U_V accumulator;
//   [64,96) / [96,128)   Q / U_Q as the bf16 A operands of the score GEMMs
//               (copied once from the swizzled shared-memory blocks), so those
//               GEMMs read only the key tile from shared memory: per 64 keys
//               the shared-memory traffic (operand reads and the ring's TMA
//               writes) drops from 104 to 72 KiB;
//   [128 + 128 b, 256 + 128 b)   score buffer b = 0, 1, 2: F' = Q U_K^T +
//               U_Q K^T (64 columns) | S = Q K^T (64 columns).
// A warpgroup reads the buffer into registers and writes the bf16 A
// operands of the output GEMMs over F': K step c (keys 16c .. 16c + 15 of
// the tile) has P at column 16c and P o F at 16c + 8, over those keys' F'.
// The score GEMMs of tile t + 3 follow tile t's output GEMMs on the in-order
// tensor pipe, so they overwrite the buffer only after its operands were
// read, and each warpgroup has three tiles' worth of MMA time for each of
// its tiles.
#include "internal.h"
#include "tc_common.cuh"

namespace flashbob {
namespace {
using namespace tc;

constexpr int BM = kTcRows;   // 128 query rows per CTA
constexpr int BN = kTcJvpStream;  // 64 key rows per streamed tile
constexpr int DH = 64;        // head dim
constexpr int NST = 6;        // stages of the U_K/K/V/U_V ring
constexpr int NB = 3;   // score buffers
constexpr int NWG = 3;  // elementwise warpgroups, one per score buffer
constexpr int NTHREADS = 64 + 128 * NWG;
constexpr uint32_t BLOCK_BYTES = BM * DH * 2;  // 16 KiB
constexpr uint32_t TILE_BYTES = BN * DH * 2;   // 8 KiB
constexpr float kLog2e = 1.4426950408889634f;

// Epilogue staging of O (then O') in the idle ring: rows padded to 68 floats.
constexpr int kStageLd = DH + 4;
static_assert(BM * kStageLd * 4 <= NST * 4 * TILE_BYTES, "epilogue staging fits in the ring");

struct SmemJ {
  alignas(1024) uint8_t q[BLOCK_BYTES];
  alignas(1024) uint8_t uq[BLOCK_BYTES];
  alignas(1024) uint8_t kv[NST][4][TILE_BYTES];  // U_K, K, V, U_V (U_K | K adjacent)
  float part_a[NWG][BM];                         // L' partial sums of the warpgroups
  uint64_t bar_q;
  uint64_t a_ready;  // Q and U_Q are in TMEM (8 warps)
  uint64_t kv_full[NST];
  uint64_t kv_empty[NST];
  uint64_t sc_full[NB];   // per buffer: the scores are in
  uint64_t op_ready[NB];  // per buffer: the operands are in TMEM (4 warps)
  uint64_t out_full;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(SmemJ) + 1024 <= 232448, "shared memory");

constexpr uint32_t kAccO = 0;
constexpr uint32_t kQA = 64, kUQA = 96;  // K step kk at + 8 kk
__device__ __forceinline__ constexpr uint32_t sc_base(int b) { return 128 + 128 * b; }
constexpr uint32_t kColF = 0, kColS = 64;  // inside a score buffer
// Operand slots inside a score buffer: K step c over the F' columns of the
// same 16 keys (16c .. 16c + 15), which its warpgroup has read by then.
__device__ __forceinline__ constexpr uint32_t slot_P(int c) { return 16 * c; }
__device__ __forceinline__ constexpr uint32_t slot_PF(int c) { return 16 * c + 8; }

// 16 keys of a tile, one query row per thread: P = exp(S - L), P o F with
// F = tau F', the row sum L' += P o F, and the two bf16 operands.
template <bool MASKED>
__device__ __forceinline__ void jvp_chunk(uint32_t buf, int c, const uint32_t (&s)[16],
                                          const uint32_t (&f)[16], int jbase, int jmax,
                                          float2 c12, float2 nL, float2 tau2, float2& a_acc) {
  uint32_t oP[8], oPF[8];
#pragma unroll
  for (int e = 0; e < 16; e += 2) {
    const float2 t = ffma2(f2(s[e], s[e + 1]), c12, nL);
    float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
    if (MASKED) {
      if (jbase + e > jmax) p.x = 0.f;
      if (jbase + e + 1 > jmax) p.y = 0.f;
    }
    const float2 pf = fmul2(p, fmul2(f2(f[e], f[e + 1]), tau2));
    a_acc = fadd2(a_acc, pf);
    oP[e >> 1] = pack_bf16x2(p.x, p.y);
    oPF[e >> 1] = pack_bf16x2(pf.x, pf.y);
  }
  tmem_st8(buf + slot_P(c), oP);
  tmem_st8(buf + slot_PF(c), oPF);
}

// One 64-key tile, 16 keys at a time: while a chunk's operands are formed
// (and stored over the F' columns of its own keys, already read), the next
// chunk's F' and S are being read; then hand the operands to the MMA issuer.
template <bool MASKED>
__device__ __forceinline__ void jvp_tile(uint32_t sc, uint64_t* ready, int col0, int jmax,
                                         float c1, float Lr2, float tau, float2& a_acc) {
  uint32_t f0[16], f1[16], f2_[16], f3[16], s0[16], s1[16], s2[16], s3[16];
  const float2 c12 = make_float2(c1, c1), nL = make_float2(-Lr2, -Lr2);
  const float2 tau2 = make_float2(tau, tau);
  tmem_ld16(sc + kColF, f0);
  tmem_ld16(sc + kColS, s0);
  tmem_wait_ld();
  tmem_ld16(sc + kColF + 16, f1);
  tmem_ld16(sc + kColS + 16, s1);
  jvp_chunk<MASKED>(sc, 0, s0, f0, col0, jmax, c12, nL, tau2, a_acc);
  tmem_wait_ld();
  tmem_ld16(sc + kColF + 32, f2_);
  tmem_ld16(sc + kColS + 32, s2);
  jvp_chunk<MASKED>(sc, 1, s1, f1, col0 + 16, jmax, c12, nL, tau2, a_acc);
  tmem_wait_ld();
  tmem_ld16(sc + kColF + 48, f3);
  tmem_ld16(sc + kColS + 48, s3);
  jvp_chunk<MASKED>(sc, 2, s2, f2_, col0 + 32, jmax, c12, nL, tau2, a_acc);
  tmem_wait_ld();
  jvp_chunk<MASKED>(sc, 3, s3, f3, col0 + 48, jmax, c12, nL, tau2, a_acc);
  tmem_wait_st();
  tc_fence_before();
  warp_arrive(ready);
}

__global__ void __launch_bounds__(NTHREADS, 1)
    tc_jvp_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mUQ,
                  const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
                  const __grid_constant__ CUtensorMap mUK,
                  const __grid_constant__ CUtensorMap mUV, const float* __restrict__ O,
                  const float* __restrict__ L, float* __restrict__ Od,
                  float* __restrict__ Ld, int H, int Hkv, int Nq, int Nk, float tau, int causal,
                  unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  SmemJ& sm = *reinterpret_cast<SmemJ*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
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
    mbar_init(&sm.a_ready, 8);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(&sm.sc_full[b], 1);
      mbar_init(&sm.op_ready[b], 4);
    }
    mbar_init(&sm.out_full, 1);
    sm.abort_flag = 0;
    fence_barrier_init();
    // The resident block's copy starts now, while warp 1 allocates TMEM.
    mbar_expect_tx(&sm.bar_q, 2 * BLOCK_BYTES);
    tma_load_3d(sm.q, &mQ, &sm.bar_q, 0, row0, bh);
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
    constexpr uint32_t idS128 = idesc_bf16(BM, 2 * BN, false);  // N = 128, B K-major
    constexpr uint32_t idS64 = idesc_bf16(BM, BN, false);       // N = 64, B K-major
    constexpr uint32_t idO64 = idesc_bf16(BM, DH, true);        // N = 64, B MN-major
    // Descriptors of the resident blocks and of stage 0; a K step of the
    // score GEMMs adds 32 bytes (16 bf16 inside the swizzled row), one of the
    // output GEMMs 16 key rows (2 KiB), and a stage 4 * TILE_BYTES
    // (start-address field: address >> 4).
    const uint32_t kv0 = smem_u32(sm.kv[0][0]);
    const uint64_t dUK0 = smem_desc_sw128(kv0, 16, 1024);                  // [U_K; K]
    const uint64_t dK0 = smem_desc_sw128(kv0 + TILE_BYTES, 16, 1024);      // K
    const uint64_t dV0 = smem_desc_sw128(kv0 + 2 * TILE_BYTES, 16, 1024);  // V
    const uint64_t dUV0 = smem_desc_sw128(kv0 + 3 * TILE_BYTES, 16, 1024); // U_V
    auto issue_scores = [&](int t) {
      const uint64_t so = (uint64_t)((t % NST) * 4 * TILE_BYTES) >> 4;
      const uint32_t sc = tbase + sc_base(t % NB);
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        const uint64_t o = 2 * kk;  // 32 bytes >> 4
        mma_ts(sc + kColF, tbase + kQA + 8 * kk, dUK0 + so + o, idS128, kk > 0);  // [F' | S] = Q [U_K; K]^T
        mma_ts(sc + kColF, tbase + kUQA + 8 * kk, dK0 + so + o, idS64, 1);        // F' += U_Q K^T
      }
    };
    auto issue_outputs = [&](int t) {
      const int s = t % NST;
      const uint64_t so = (uint64_t)(s * 4 * TILE_BYTES) >> 4;
      const uint32_t ob = tbase + sc_base(t % NB);
#pragma unroll
      for (int c = 0; c < BN / 16; ++c) {
        const uint64_t o = (uint64_t)(16 * 128 * c) >> 4;  // 16 key rows further down
        const uint32_t acc = (t > 0 || c > 0);
        mma_ts(tbase + kAccO, ob + slot_P(c), dUV0 + so + o, idO64, acc);  // O'0 += P U_V
        mma_ts(tbase + kAccO, ob + slot_PF(c), dV0 + so + o, idO64, 1);    //     + (P o F) V
      }
      mma_commit(&sm.kv_empty[s]);
    };
    // One elected lane runs the whole schedule: every wait and every MMA.
    if (elect_one()) {
      bool ok = mbar_wait(&sm.a_ready, 0, abort_flag, err);
      tc_fence_after();
      for (int t = 0; ok && t < NB && t < T; ++t) {
        ok = mbar_wait(&sm.kv_full[t % NST], (t / NST) & 1, abort_flag, err);
        tc_fence_after();
        if (ok) {
          issue_scores(t);
          mma_commit(&sm.sc_full[t]);
        }
      }
      for (int t = 0; ok && t < T; ++t) {
        ok = mbar_wait(&sm.op_ready[t % NB], (t / NB) & 1, abort_flag, err);
        if (!ok) break;
        tc_fence_after();
        issue_outputs(t);
        if (t + NB < T) {  // tile t + 3 reuses tile t's buffer, after its output GEMMs
          ok = mbar_wait(&sm.kv_full[(t + NB) % NST], ((t + NB) / NST) & 1, abort_flag, err);
          if (!ok) break;
          tc_fence_after();
          issue_scores(t + NB);
          mma_commit(&sm.sc_full[t % NB]);
        }
      }
      mma_commit(&sm.out_full);  // every MMA issued above has finished
    }
    __syncwarp();
  } else {
    // ---------------- elementwise warpgroups + epilogue ----------------
    const int wg = (warp - 2) >> 2;      // 0 .. NWG - 1
    const int quad = warp & 3;           // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane;      // row inside the block = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int gr = row0 + r;
    const size_t rowvec = static_cast<size_t>(bh) * Nq + gr;
    const float c1 = tau * kLog2e;
    const float Lr2 = gr < Nq ? L[rowvec] * kLog2e : 0.f;
    float2 a_acc = make_float2(0.f, 0.f);
    bool ok = true;
    if (wg < 2) {
      // Warpgroup 0 copies its row of Q, warpgroup 1 its row of U_Q, from
      // the 128-byte-swizzled TMA block (16-byte chunk c of row r at chunk
      // c ^ (r mod 8)) into TMEM: K step kk is chunks 2 kk and 2 kk + 1.
      ok = mbar_wait_warp(&sm.bar_q, 0, abort_flag, err);
      if (ok) {
        const uint8_t* row = (wg == 0 ? sm.q : sm.uq) + r * 128;
        const uint32_t dst = tbase + lane_off + (wg == 0 ? kQA : kUQA);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint4 a = *reinterpret_cast<const uint4*>(row + (((2 * kk) ^ (r & 7)) << 4));
          const uint4 b = *reinterpret_cast<const uint4*>(row + (((2 * kk + 1) ^ (r & 7)) << 4));
          const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
          tmem_st8(dst + 8 * kk, v);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      warp_arrive(&sm.a_ready);
    }

    for (int u = 0;; ++u) {
      const int t = NWG * u + wg;  // in buffer t mod 3 = wg
      if (t >= T) break;
      const int b = t % NB;
      const uint32_t sc = tbase + lane_off + sc_base(b);
      // tcgen05.ld/st are warp-collective: take the decision warp-uniformly.
      ok = mbar_wait_warp(&sm.sc_full[b], (t / NB) & 1, abort_flag, err);
      if (!ok) break;
      tc_fence_after();
      const int col0 = t * BN;
      // Columns past Nk, or (causal) past this row, get P = 0.  Only tiles
      // that reach past Nk or past the block's first row take the masked path.
      const bool masked = (col0 + BN > Nk) || (causal && col0 + BN - 1 > row0);
      const int jmax = causal ? min(Nk - 1, gr) : Nk - 1;
      if (masked)
        jvp_tile<true>(sc, &sm.op_ready[b], col0, jmax, c1, Lr2, tau, a_acc);
      else
        jvp_tile<false>(sc, &sm.op_ready[b], col0, jmax, c1, Lr2, tau, a_acc);
    }

    // Epilogue: L' = the warpgroups' row sums; warpgroup wg forms the 16-column
    // chunks h = wg, wg + 3 of O' = O'0 - L' O.
    sm.part_a[wg][r] = a_acc.x + a_acc.y;
    named_bar_sync(1, 128 * NWG);
    float lp = 0.f;
#pragma unroll
    for (int w = 0; w < NWG; ++w) lp += sm.part_a[w][r];
    ok = mbar_wait_warp(&sm.out_full, 0, abort_flag, err) && ok;
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);
    tc_fence_after();
    const uint32_t acc_base = tbase + lane_off;
    // Every MMA is done, so the ring is idle: the block's rows of O come in
    // through shared memory with coalesced loads, each thread forms its
    // row's O' there in place, and the tile leaves with coalesced stores.
    float* st_o = reinterpret_cast<float*>(&sm.kv[0][0][0]);
    const int tid = threadIdx.x - 64;  // 0 .. 128 NWG - 1
    const int rows = min(BM, Nq - row0);
    const size_t blk = (static_cast<size_t>(bh) * Nq + row0) * DH;
    for (int f = tid; f < rows * (DH / 4); f += 128 * NWG) {
      const int rr = f / (DH / 4), c4 = f % (DH / 4);
      *reinterpret_cast<float4*>(st_o + rr * kStageLd + 4 * c4) =
          reinterpret_cast<const float4*>(O + blk)[f];
    }
    named_bar_sync(1, 128 * NWG);
    for (int h = wg; h < DH / 16; h += NWG) {
      const int col = 16 * h;
      uint32_t vo[16];
      tmem_ld16(acc_base + kAccO + col, vo);
      tmem_wait_ld();
      if (gr < Nq) {
        float4* o4 = reinterpret_cast<float4*>(st_o + r * kStageLd + col);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 ov = o4[k];
          o4[k] = make_float4(u2f(vo[4 * k + 0]) - lp * ov.x, u2f(vo[4 * k + 1]) - lp * ov.y,
                              u2f(vo[4 * k + 2]) - lp * ov.z, u2f(vo[4 * k + 3]) - lp * ov.w);
        }
      }
    }
    named_bar_sync(1, 128 * NWG);
    if (ok) {
      for (int f = tid; f < rows * (DH / 4); f += 128 * NWG) {
        const int rr = f / (DH / 4), c4 = f % (DH / 4);
        reinterpret_cast<float4*>(Od + blk)[f] =
            *reinterpret_cast<const float4*>(st_o + rr * kStageLd + 4 * c4);
      }
    }
    if (ok && wg == 0 && gr < Nq) Ld[rowvec] = lp;
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

size_t tc_jvp_smem() { return sizeof(SmemJ) + 1024; }

cudaError_t tc_launch_jvp(const JvpArgs& a, const CUtensorMap* maps128,
                          const CUtensorMap* maps64) {
  // maps128: Q, U_Q with 128-row boxes; maps64: K, V, U_K, U_V with 64-row boxes.
  const size_t smem = tc_jvp_smem();
  cudaError_t e = tc_set_smem(reinterpret_cast<const void*>(tc_jvp_kernel), (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Nq + BM - 1) / BM, a.H, a.B);
  tc_jvp_kernel<<<grid, NTHREADS, smem, a.stream>>>(
      maps128[0], maps128[1], maps64[0], maps64[1], maps64[2], maps64[3], a.O, a.L, a.Od, a.Ld,
      a.H, a.Hkv, a.Nq, a.Nk, a.tau, a.causal ? 1 : 0, a.err);
  return cudaGetLastError();
}

}  // namespace flashbob
