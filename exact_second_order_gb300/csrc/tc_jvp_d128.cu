// Attention JVP (forward-mode derivative along U_Q, U_K, U_V) on sm_103a
// tensor cores for head dim 128: bf16 inputs, fp32 accumulation in tensor
// memory.  It is also the first of the two launches of the d = 128 pass 1.
//
// The forward of "FlashAttention 的反向传播设计" (section 一): S = tau Q K^T,
// P = exp(S - L), O = P V; along the tangents F = tau (U_Q K^T + Q U_K^T),
// L' = sum_j P_ij F_ij and O' = (P o F) V + P U_V - L' O.  In "FlashBoB"
// (paper notes, 关键设计 1) these are pass 1's alpha and d~dO, and with dO and
// D given the epilogue also writes the second row scalar in closed form,
//     E_i = sum_j P_ij d~P_ij = dO_i . d~dO_i - alpha_i D_i
// (d~P = F o (dP - D) + G - alpha dP with dP = dO V^T, G = dO U_V^T and
// D = dO . O), so the second launch has alpha and E for every row.
//
// CTA = 128 query rows (MMA M = 128, one TMEM lane per row), 320 threads:
//   warp 0      TMA producer: the Q and U_Q blocks once (two 64-column halves
//               each), then tiles of 64 key rows through two 3-stage rings,
//               one of U_K | K (read by the score GEMMs, free once they have
//               completed) and one of V | U_V (read by the output GEMMs), whose
//               third stages are the Q | U_Q block, free once the elementwise
//               warps have copied Q and U_Q into TMEM;
//   warp 1      TMEM allocator; one elected lane runs the MMA schedule;
//   warps 2-5 / 6-9   elementwise warpgroups 0 / 1: tiles t = w mod 2, in
//               score buffer w.
// With two scores per element (no dP, G) the tiles are 64 keys wide: per
// tile the score GEMMs are Q [U_K; K]^T (8 MMAs of N = 128) and U_Q K^T
// (8 of N = 64), the output GEMMs P U_V and (P o F) V (8 of N = 128), every
// A operand in TMEM, so shared memory serves only the key tiles.
// TMEM (512 columns x 128 lanes):
//   [0,128)     O'0 = (P o F) V + P U_V accumulator;
//   [128,192) / [192,256)   Q / U_Q as bf16 A operands (K step kk at +8 kk);
//   [256,384) / [384,512)   score buffers 0 / 1: F' = Q U_K^T + U_Q K^T (64
//               columns) | S = Q K^T (64 columns).
// A warpgroup reads its buffer 16 keys at a time and writes each chunk's
// bf16 A operands over that chunk's F' columns (P at 16c, P o F at 16c + 8);
// the score GEMMs of tile t + 2 follow tile t's output GEMMs on the in-order
// tensor pipe, so they overwrite the buffer only after its operands were read.
#include "internal.h"
#include "tc_common.cuh"

namespace flashbob {
namespace {
using namespace tc;

constexpr int BM = kTcRows;       // 128 query rows per CTA
constexpr int BN = kTcJvpStream;  // 64 key rows per streamed tile
constexpr int DH = 128;
constexpr int NST = 3;  // stages of each ring; stage 2 lies in the Q | U_Q block
constexpr int NWG = 2;  // elementwise warpgroups = score buffers
constexpr int NTHREADS = 64 + 128 * NWG;
constexpr uint32_t HALF_BLOCK = BM * 64 * 2;  // 16 KiB: 128 rows x 64 columns
constexpr uint32_t HALF_TILE = BN * 64 * 2;   // 8 KiB: 64 rows x 64 columns
constexpr uint32_t STAGE_BYTES = 2 * 2 * HALF_TILE;  // [half][U_K, K] or [half][V, U_V]
constexpr float kLog2e = 1.4426950408889634f;
// Epilogue staging in the idle ring: O (then O') as fp32 rows padded to 132
// floats, and, for E, dO as bf16 rows padded to 136 elements.
constexpr int kStageLd = DH + 4;
constexpr int kDoLd = DH + 8;

struct SmemJ2 {
  alignas(1024) uint8_t kv[2][2][STAGE_BYTES];     // [U_K | K ring, V | U_V ring][stage 0, 1]
  alignas(1024) uint8_t qu[2][2][HALF_BLOCK];      // [Q, U_Q][half]; then stage 2 of each ring
  float part_a[NWG][BM];  // L' partial sums of the warpgroups
  float part_e[NWG][BM];  // dO . O' partial sums
  uint64_t bar_q;
  uint64_t a_ready;  // Q and U_Q are in TMEM (8 warps)
  uint64_t k_full[NST];   // U_K | K ring
  uint64_t k_empty[NST];
  uint64_t v_full[NST];   // V | U_V ring
  uint64_t v_empty[NST];
  uint64_t sc_full[NWG];
  uint64_t op_ready[NWG];  // 4 warps
  uint64_t out_full;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(SmemJ2::qu) == 2 * STAGE_BYTES, "the Q | U_Q block holds stage 2 of both rings");
static_assert(sizeof(SmemJ2) + 1024 <= 232448, "shared memory");
static_assert(BM * kStageLd * 4 + BM * kDoLd * 2 <= sizeof(SmemJ2::kv),
              "epilogue staging fits in stages 0 and 1 of the rings");

constexpr uint32_t kAccO = 0;
constexpr uint32_t kQA = 128, kUQA = 192;
__device__ __forceinline__ constexpr uint32_t sc_base(int b) { return 256 + 128 * b; }
constexpr uint32_t kColF = 0, kColS = 64;  // inside a score buffer
__device__ __forceinline__ constexpr uint32_t slot_P(int c) { return 16 * c; }
__device__ __forceinline__ constexpr uint32_t slot_PF(int c) { return 16 * c + 8; }

// 16 keys of a tile, one query row per thread: P = exp(S - L), P o F with
// F = tau F', the row sum L' += P o F, and the two bf16 operands over F'.
template <bool MASKED>
__device__ __forceinline__ void jvp_chunk(uint32_t sc, int c, const uint32_t (&s)[16],
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
  tmem_st8(sc + slot_P(c), oP);
  tmem_st8(sc + slot_PF(c), oPF);
}

// One 64-key tile, 16 keys at a time: while a chunk's operands are formed,
// the next chunk's F' and S are being read; then hand the operands on.
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

// E (and the dO it needs) is optional: E = nullptr for the attention JVP.
__global__ void __launch_bounds__(NTHREADS, 1)
    tc_jvp_d128_kernel(const __grid_constant__ CUtensorMap mQ,
                       const __grid_constant__ CUtensorMap mUQ,
                       const __grid_constant__ CUtensorMap mK,
                       const __grid_constant__ CUtensorMap mV,
                       const __grid_constant__ CUtensorMap mUK,
                       const __grid_constant__ CUtensorMap mUV, const float* __restrict__ O,
                       const float* __restrict__ L, const __nv_bfloat16* __restrict__ dO,
                       const float* __restrict__ D, float* __restrict__ Od,
                       float* __restrict__ Ld, float* __restrict__ E, int H, int Hkv, int Nq,
                       int Nk, float tau, int causal, unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  SmemJ2& sm = *reinterpret_cast<SmemJ2*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.z * H + blockIdx.y;
  // key/value head shared by this query head (grouped-query attention)
  const int bkv = blockIdx.z * Hkv + blockIdx.y / (H / Hkv);
  // Causal: the last row blocks see the most keys, so they start first.
  const int row0 = (causal ? gridDim.x - 1 - blockIdx.x : blockIdx.x) * BM;
  const int col_end = causal ? min(Nk, row0 + BM) : Nk;  // keys j <= i under the causal mask
  const int T = (col_end + BN - 1) / BN;
  const bool withE = E != nullptr;
  volatile int* abort_flag = &sm.abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(&sm.bar_q, 1);
    mbar_init(&sm.a_ready, 8);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
    }
    for (int b = 0; b < NWG; ++b) {
      mbar_init(&sm.sc_full[b], 1);
      mbar_init(&sm.op_ready[b], 4);
    }
    mbar_init(&sm.out_full, 1);
    sm.abort_flag = 0;
    fence_barrier_init();
    // The resident blocks' copy starts now, while warp 1 allocates TMEM.
    mbar_expect_tx(&sm.bar_q, 4 * HALF_BLOCK);
    for (int h = 0; h < 2; ++h) {
      tma_load_3d(sm.qu[0][h], &mQ, &sm.bar_q, 64 * h, row0, bh);
      tma_load_3d(sm.qu[1][h], &mUQ, &sm.bar_q, 64 * h, row0, bh);
    }
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
      // Stage s of ring r (0: U_K | K, 1: V | U_V): half h of its first / second
      // tensor at (2 h + 0 / 1) HALF_TILE.
      auto stage = [&](int r, int s) -> uint8_t* {
        return s < 2 ? sm.kv[r][s] : sm.qu[r][0];
      };
      // The U_K | K tile of key tile t, then the V | U_V tile of tile t - 1:
      // the score GEMMs of tile t free their stage before the output GEMMs
      // of tile t - 1 free theirs.
      auto load = [&](int r, int t) -> bool {
        const int s = t % NST;
        uint64_t* full = r == 0 ? &sm.k_full[s] : &sm.v_full[s];
        uint64_t* empty = r == 0 ? &sm.k_empty[s] : &sm.v_empty[s];
        if (t >= NST) {
          if (!mbar_wait(empty, ((t / NST) - 1) & 1, abort_flag, err)) return false;
        } else if (s == 2 && !mbar_wait(&sm.a_ready, 0, abort_flag, err)) {
          return false;  // stage 2 is in the Q | U_Q block: wait until it was copied out
        }
        const CUtensorMap* m0 = r == 0 ? &mUK : &mV;
        const CUtensorMap* m1 = r == 0 ? &mK : &mUV;
        uint8_t* base = stage(r, s);
        mbar_expect_tx(full, STAGE_BYTES);
        for (int h = 0; h < 2; ++h) {
          tma_load_3d(base + (2 * h) * HALF_TILE, m0, full, 64 * h, t * BN, bkv);
          tma_load_3d(base + (2 * h + 1) * HALF_TILE, m1, full, 64 * h, t * BN, bkv);
        }
        return true;
      };
      int issued_k = 0, issued_v = 0;
      for (int t = 0; t <= T; ++t) {
        if (t < T) {
          if (!load(0, t)) break;
          issued_k = t + 1;
        }
        if (t >= 1) {
          if (!load(1, t - 1)) break;
          issued_v = t;
        }
      }
      // No copy may still be in flight when the CTA exits.
      drain_wait(&sm.bar_q, 0);
      for (int t = issued_k > NST ? issued_k - NST : 0; t < issued_k; ++t)
        drain_wait(&sm.k_full[t % NST], (t / NST) & 1);
      for (int t = issued_v > NST ? issued_v - NST : 0; t < issued_v; ++t)
        drain_wait(&sm.v_full[t % NST], (t / NST) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (whole warp, one elected lane issues) ----------------
    constexpr uint32_t idS128 = idesc_bf16(BM, 2 * BN, false);  // N = 128, B K-major
    constexpr uint32_t idS64 = idesc_bf16(BM, BN, false);       // N = 64, B K-major
    constexpr uint32_t idO128 = idesc_bf16(BM, DH, true);       // N = 128, B MN-major
    auto stage_addr = [&](int r, int s) -> uint32_t {
      return smem_u32(s < 2 ? sm.kv[r][s] : sm.qu[r][0]);
    };
    // Inside a stage, half h of the first / second tensor sits at
    // (2 h + 0 / 1) HALF_TILE; a K step of the score GEMMs adds 32 bytes
    // inside the swizzled row (and moves to half 1 after 4 steps), one of the
    // output GEMMs 16 key rows (2 KiB); descriptor start addresses are in
    // 16-byte units.
    auto issue_scores = [&](int t) {
      const uint64_t d0 = smem_desc_sw128(stage_addr(0, t % NST), 16, 1024);  // U_K, half 0
      const uint32_t sc = tbase + sc_base(t & 1);
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        const uint64_t dUK = d0 + ((kk >> 2) * 2 * HALF_TILE >> 4) + 2 * (kk & 3);
        const uint64_t dK = dUK + (HALF_TILE >> 4);
        mma_ts(sc + kColF, tbase + kQA + 8 * kk, dUK, idS128, kk > 0);  // [F' | S] = Q [U_K; K]^T
        mma_ts(sc + kColF, tbase + kUQA + 8 * kk, dK, idS64, 1);        // F' += U_Q K^T
      }
      mma_commit(&sm.k_empty[t % NST]);
    };
    auto issue_outputs = [&](int t) {
      const int s = t % NST;
      // MN-major N = 128 operands: columns 64..127 (half 1) sit two tiles
      // after columns 0..63 of the same tensor.
      const uint32_t vb = stage_addr(1, s);
      const uint64_t dVmn = smem_desc_sw128(vb, 2 * HALF_TILE, 1024);
      const uint64_t dUVmn = smem_desc_sw128(vb + HALF_TILE, 2 * HALF_TILE, 1024);
      const uint32_t sc = tbase + sc_base(t & 1);
#pragma unroll
      for (int c = 0; c < BN / 16; ++c) {
        const uint64_t o = (uint64_t)(16 * 128 * c) >> 4;  // 16 key rows further down
        const uint32_t acc = (t > 0 || c > 0);
        mma_ts(tbase + kAccO, sc + slot_P(c), dUVmn + o, idO128, acc);  // O'0 += P U_V
        mma_ts(tbase + kAccO, sc + slot_PF(c), dVmn + o, idO128, 1);    //     + (P o F) V
      }
      mma_commit(&sm.v_empty[s]);
    };
    // One elected lane runs the whole schedule: every wait and every MMA.
    if (elect_one()) {
      bool ok = mbar_wait(&sm.a_ready, 0, abort_flag, err);
      tc_fence_after();
      for (int t = 0; ok && t < NWG && t < T; ++t) {
        ok = mbar_wait(&sm.k_full[t % NST], (t / NST) & 1, abort_flag, err);
        tc_fence_after();
        if (ok) {
          issue_scores(t);
          mma_commit(&sm.sc_full[t]);
        }
      }
      for (int t = 0; ok && t < T; ++t) {
        ok = mbar_wait(&sm.op_ready[t & 1], (t >> 1) & 1, abort_flag, err) &&
             mbar_wait(&sm.v_full[t % NST], (t / NST) & 1, abort_flag, err);
        if (!ok) break;
        tc_fence_after();
        issue_outputs(t);
        if (t + NWG < T) {  // tile t + 2 reuses tile t's buffer, after its output GEMMs
          ok = mbar_wait(&sm.k_full[(t + NWG) % NST], ((t + NWG) / NST) & 1, abort_flag, err);
          if (!ok) break;
          tc_fence_after();
          issue_scores(t + NWG);
          mma_commit(&sm.sc_full[t & 1]);
        }
      }
      mma_commit(&sm.out_full);  // every MMA issued above has finished
    }
    __syncwarp();
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
    float2 a_acc = make_float2(0.f, 0.f);
    bool ok = true;
    {
      // Warpgroup 0 copies its row of Q, warpgroup 1 its row of U_Q, from
      // the two 128-byte-swizzled halves (16-byte chunk c of row r at chunk
      // c ^ (r mod 8)) into TMEM: K step kk is chunks 2 (kk mod 4) and
      // 2 (kk mod 4) + 1 of half kk / 4.
      ok = mbar_wait_warp(&sm.bar_q, 0, abort_flag, err);
      if (ok) {
        const uint32_t dst = tbase + lane_off + (wg == 0 ? kQA : kUQA);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint8_t* row = sm.qu[wg][kk >> 2] + r * 128;
          const int c = 2 * (kk & 3);
          const uint4 a = *reinterpret_cast<const uint4*>(row + ((c ^ (r & 7)) << 4));
          const uint4 b = *reinterpret_cast<const uint4*>(row + (((c + 1) ^ (r & 7)) << 4));
          const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
          tmem_st8(dst + 8 * kk, v);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      warp_arrive(&sm.a_ready);  // also frees the Q | U_Q block for ring stage 2
    }
    const uint32_t sc = tbase + lane_off + sc_base(wg);
    for (int u = 0;; ++u) {
      const int t = NWG * u + wg;  // in buffer t mod 2 = wg
      if (t >= T) break;
      // tcgen05.ld/st are warp-collective: take the decision warp-uniformly.
      ok = ok && mbar_wait_warp(&sm.sc_full[wg], u & 1, abort_flag, err);
      if (!ok) break;
      tc_fence_after();
      const int col0 = t * BN;
      // Columns past Nk, or (causal) past this row, get P = 0.  Only tiles
      // that reach past Nk or past the block's first row take the masked path.
      const bool masked = (col0 + BN > Nk) || (causal && col0 + BN - 1 > row0);
      const int jmax = causal ? min(Nk - 1, gr) : Nk - 1;
      if (masked)
        jvp_tile<true>(sc, &sm.op_ready[wg], col0, jmax, c1, Lr2, tau, a_acc);
      else
        jvp_tile<false>(sc, &sm.op_ready[wg], col0, jmax, c1, Lr2, tau, a_acc);
    }

    // Epilogue: L' = the warpgroups' row sums; warpgroup wg forms the
    // 16-column chunks h = wg, wg + 2, ... of O' = O'0 - L' O (and its part
    // of dO . O').  Every MMA is done, so ring stages 0 and 1 are idle: the
    // block's rows of O (and dO) come in through shared memory with
    // coalesced loads, each thread forms its row's O' there in place, and
    // the tile leaves with coalesced stores.
    sm.part_a[wg][r] = a_acc.x + a_acc.y;
    named_bar_sync(1, 128 * NWG);
    float lp = 0.f;
#pragma unroll
    for (int w = 0; w < NWG; ++w) lp += sm.part_a[w][r];
    ok = mbar_wait_warp(&sm.out_full, 0, abort_flag, err) && ok;
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);
    tc_fence_after();
    const uint32_t acc_base = tbase + lane_off;
    float* st_o = reinterpret_cast<float*>(&sm.kv[0][0][0]);
    __nv_bfloat16* st_do = reinterpret_cast<__nv_bfloat16*>(st_o + BM * kStageLd);
    const int tid = threadIdx.x - 64;  // 0 .. 128 NWG - 1
    const int rows = min(BM, Nq - row0);
    const size_t blk = (static_cast<size_t>(bh) * Nq + row0) * DH;
    for (int f = tid; f < rows * (DH / 4); f += 128 * NWG) {
      const int rr = f / (DH / 4), c4 = f % (DH / 4);
      *reinterpret_cast<float4*>(st_o + rr * kStageLd + 4 * c4) =
          reinterpret_cast<const float4*>(O + blk)[f];
    }
    if (withE) {
      for (int f = tid; f < rows * (DH / 8); f += 128 * NWG) {
        const int rr = f / (DH / 8), c8 = f % (DH / 8);
        *reinterpret_cast<uint4*>(st_do + rr * kDoLd + 8 * c8) =
            reinterpret_cast<const uint4*>(dO + blk)[f];
      }
    }
    named_bar_sync(1, 128 * NWG);
    float edot = 0.f;  // dO . O' over this thread's columns
    for (int h = wg; h < DH / 16; h += NWG) {
      const int col = 16 * h;
      uint32_t vo[16];
      tmem_ld16(acc_base + kAccO + col, vo);
      tmem_wait_ld();
      if (gr < Nq) {
        float4* o4 = reinterpret_cast<float4*>(st_o + r * kStageLd + col);
        float dv[16];
        if (withE) {
          const uint4 x = *reinterpret_cast<const uint4*>(st_do + r * kDoLd + col);
          const uint4 y = *reinterpret_cast<const uint4*>(st_do + r * kDoLd + col + 8);
          const uint32_t w[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            dv[2 * k] = __uint_as_float(w[k] << 16);
            dv[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 ov = o4[k];
          const float4 od = make_float4(u2f(vo[4 * k + 0]) - lp * ov.x,
                                        u2f(vo[4 * k + 1]) - lp * ov.y,
                                        u2f(vo[4 * k + 2]) - lp * ov.z,
                                        u2f(vo[4 * k + 3]) - lp * ov.w);
          o4[k] = od;
          if (withE)
            edot += dv[4 * k] * od.x + dv[4 * k + 1] * od.y + dv[4 * k + 2] * od.z +
                    dv[4 * k + 3] * od.w;
        }
      }
    }
    sm.part_e[wg][r] = edot;
    named_bar_sync(1, 128 * NWG);
    if (ok) {
      for (int f = tid; f < rows * (DH / 4); f += 128 * NWG) {
        const int rr = f / (DH / 4), c4 = f % (DH / 4);
        reinterpret_cast<float4*>(Od + blk)[f] =
            *reinterpret_cast<const float4*>(st_o + rr * kStageLd + 4 * c4);
      }
    }
    if (ok && wg == 0 && gr < Nq) {
      Ld[rowvec] = lp;
      if (withE) {
        float e = 0.f;
#pragma unroll
        for (int w = 0; w < NWG; ++w) e += sm.part_e[w][r];
        E[rowvec] = e - lp * D[rowvec];
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

cudaError_t launch(const CUtensorMap* maps128, const CUtensorMap* maps64, const float* O,
                   const float* L, const void* dO, const float* D, float* Od, float* Ld,
                   float* E, int B, int H, int Hkv, int Nq, int Nk, float tau, bool causal,
                   cudaStream_t stream, unsigned int* err) {
  const size_t smem = sizeof(SmemJ2) + 1024;
  cudaError_t e = tc_set_smem(reinterpret_cast<const void*>(tc_jvp_d128_kernel), (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((Nq + BM - 1) / BM, H, B);
  tc_jvp_d128_kernel<<<grid, NTHREADS, smem, stream>>>(
      maps128[0], maps128[1], maps64[0], maps64[1], maps64[2], maps64[3], O, L,
      static_cast<const __nv_bfloat16*>(dO), D, Od, Ld, E, H, Hkv, Nq, Nk, tau, causal ? 1 : 0,
      err);
  return cudaGetLastError();
}

}  // namespace

size_t tc_jvp_d128_smem() { return sizeof(SmemJ2) + 1024; }

// maps128: Q, U_Q with 128-row boxes; maps64: K, V, U_K, U_V with 64-row
// boxes; every box is 64 columns wide (one half of a 128-column row).
cudaError_t tc_launch_jvp_d128(const JvpArgs& a, const CUtensorMap* maps128,
                               const CUtensorMap* maps64) {
  return launch(maps128, maps64, a.O, a.L, nullptr, nullptr, a.Od, a.Ld, nullptr, a.B, a.H,
                a.Hkv, a.Nq, a.Nk, a.tau, a.causal, a.stream, a.err);
}

// The first launch of the d = 128 pass 1: alpha = L', d~dO = O' and E.
cudaError_t tc_launch_pass1_d128_jvp(const BobArgs& a, const CUtensorMap* maps128,
                                     const CUtensorMap* maps64) {
  return launch(maps128, maps64, a.O, a.L, a.dO, a.D, a.ddOt, a.alpha, a.E, a.B, a.H, a.Hkv,
                a.Nq, a.Nk, a.tau, a.causal, a.stream, a.err);
}

}  // namespace flashbob
