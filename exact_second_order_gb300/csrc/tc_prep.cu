// Row state of the attention backward-over-backward on sm_103a tensor cores:
// O = P V, L = logsumexp(tau Q K^T) and D_i = dO_i . O_i for bf16 inputs,
// head dim 64 or 128 ("FlashAttention 的反向传播设计" blog, sections 一 and
// 二; D as in "FlashBoB" paper notes, 关键设计 1).
//
// One pass over the key tiles (128 keys at d = 64, 64 at d = 128) per CTA
// of 128 query rows, with the softmax normalised at the end: S = Q K^T on
// the tensor cores, P~ = exp2(S tau log2 e - m) with a running row maximum
// m, l = sum P~, and O~ += P~ V with P~ read from TMEM as bf16.  m is raised
// only when a tile's maximum exceeds it by more than kRescale (log2 units):
// then l and O~ are multiplied by exp2(m_old - m_new) first; otherwise P~
// stays below 2^kRescale and the stale m is kept.  At the end O = O~ / l
// and L = (m + log2 l) ln 2.  One exponential per score element.
//
// 320 threads: warp 0 TMA, warp 1 TMEM allocation + MMA issue, warps 2-5
// and 6-9 elementwise warpgroups on alternate tiles.  Each warpgroup keeps
// its own (m, l) and its own O~ accumulator, so its rescales never touch the
// other's; the two are merged in the epilogue.  TMEM: [0, DH) O~ of
// warpgroup 0, [DH, 2 DH) of warpgroup 1, then three score buffers of one
// tile each; the score GEMMs of tile t + 3 go into tile t's buffer right
// after tile t's P V GEMMs, so a warpgroup finds its next tile's scores
// ready.  A row of 128 columns is two 64-column boxes in the 128-byte
// swizzle.
#include "internal.h"
#include "tc_common.cuh"

namespace flashbob {
namespace {
using namespace tc;

constexpr int BM = kTcRows;
constexpr int NTHREADS = 320;
constexpr int NBUF = 3;  // score buffers
constexpr uint32_t HALF_BLOCK = BM * 64 * 2;  // 128 rows x 64 columns bf16
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.f;  // P~ <= 2^8 between rescales

template <int DH>
struct PrepCfg {
  static constexpr int kHalves = DH / 64;
  static constexpr int kBN = DH == 64 ? 128 : 64;          // keys per streamed tile
  static constexpr int kStages = DH == 64 ? 6 : 5;       // 208 / 192 KiB with Q
  static constexpr uint32_t kHalfTile = kBN * 64 * 2;       // kBN rows x 64 columns bf16
  static_assert(2 * DH + NBUF * kBN <= 512, "TMEM columns");
};

// Epilogue staging: the block's 128 x DH fp32 O tile, rows padded by 4
// floats (a warp's float4 accesses to 32 consecutive rows then take the
// minimum four shared-memory wavefronts), in the ring, idle by then.
template <int DH>
constexpr int kStageLd0 = DH + 4;

template <int DH>
struct Smem0 {
  static constexpr int NST = PrepCfg<DH>::kStages;
  static constexpr int NH = PrepCfg<DH>::kHalves;
  alignas(1024) uint8_t q[NH][HALF_BLOCK];
  alignas(1024) uint8_t kv[NST][2][NH][PrepCfg<DH>::kHalfTile];  // [stage][K, V][half]
  float part_m[2][BM];
  float part_l[2][BM];
  uint64_t bar_q;
  uint64_t kv_full[NST];
  uint64_t kv_empty[NST];
  uint64_t sc_full[NBUF];
  uint64_t op_ready[NBUF];
  uint64_t pv_done[2];  // per warpgroup: the P V GEMMs of its latest tile have completed
  uint64_t out_full;
  uint32_t tmem_base;
  int abort_flag;
};

// Largest visible raw score of 64 columns (c1 > 0, so max(S) c1 = max(S c1)).
template <bool MASKED>
__device__ __forceinline__ float prep_max64(const uint32_t (&s)[4][16], int jbase, int jmax) {
  float mr = -INFINITY;
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (!MASKED || jbase + 16 * q + j <= jmax) mr = fmaxf(mr, u2f(s[q][j]));
  return mr;
}

// P~ = exp2(S c1 - m) of 64 columns as bf16 pairs (32 registers), added to
// the row sum l (fp32, before rounding).  Invisible columns get 0.
template <bool MASKED>
__device__ __forceinline__ void prep_p64(const uint32_t (&s)[4][16], int jbase, int jmax,
                                         float c1, float m, float& l, uint32_t (&pk)[4][8]) {
  const float2 c12 = make_float2(c1, c1), nm = make_float2(-m, -m);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const float2 t = ffma2(f2(s[q][e], s[q][e + 1]), c12, nm);
      float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
      if (MASKED) {
        if (jbase + 16 * q + e > jmax) p.x = 0.f;
        if (jbase + 16 * q + e + 1 > jmax) p.y = 0.f;
      }
      acc = fadd2(acc, p);
      pk[q][e >> 1] = pack_bf16x2(p.x, p.y);
    }
  l += acc.x + acc.y;
}

template <int DH>
__global__ void __launch_bounds__(NTHREADS, 1)
    tc_prep_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                   const __grid_constant__ CUtensorMap mV, const __nv_bfloat16* __restrict__ dO,
                   float* __restrict__ O, float* __restrict__ L, float* __restrict__ D, int H,
                   int Hkv, int Nq, int Nk, float tau, int causal, unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  constexpr int NST = PrepCfg<DH>::kStages;
  constexpr int NH = PrepCfg<DH>::kHalves;
  constexpr int BN = PrepCfg<DH>::kBN;
  constexpr uint32_t HT = PrepCfg<DH>::kHalfTile;
  constexpr uint32_t kScore = 2 * DH;  // first score buffer column
  Smem0<DH>& sm = *reinterpret_cast<Smem0<DH>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.z * H + blockIdx.y;
  const int bkv = blockIdx.z * Hkv + blockIdx.y / (H / Hkv);  // shared key/value head
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
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&sm.sc_full[b], 1);
      mbar_init(&sm.op_ready[b], 4);  // one arrive per elementwise warp
    }
    mbar_init(&sm.pv_done[0], 1);
    mbar_init(&sm.pv_done[1], 1);
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
      tma_prefetch_desc(&mK);
      tma_prefetch_desc(&mV);
      mbar_expect_tx(&sm.bar_q, NH * HALF_BLOCK);
      for (int h = 0; h < NH; ++h) tma_load_3d(sm.q[h], &mQ, &sm.bar_q, 64 * h, row0, bh);
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int s = t % NST;
        if (t >= NST && !mbar_wait(&sm.kv_empty[s], ((t / NST) - 1) & 1, abort_flag, err)) break;
        mbar_expect_tx(&sm.kv_full[s], 2 * NH * HT);
        for (int h = 0; h < NH; ++h) {
          tma_load_3d(sm.kv[s][0][h], &mK, &sm.kv_full[s], 64 * h, t * BN, bkv);
          tma_load_3d(sm.kv[s][1][h], &mV, &sm.kv_full[s], 64 * h, t * BN, bkv);
        }
        issued = t + 1;
      }
      drain_wait(&sm.bar_q, 0);
      for (int t = issued > NST ? issued - NST : 0; t < issued; ++t)
        drain_wait(&sm.kv_full[t % NST], (t / NST) & 1);
    }
  } else if (warp == 1) {
    {  // MMA issuer: one elected lane runs the whole schedule
      constexpr uint32_t idS = idesc_bf16(BM, BN, false);
      constexpr uint32_t idO = idesc_bf16(BM, DH, true);
      // Base descriptors of Q, stage 0's K and stage 0's V: a stage, a half
      // or a K step only adds its byte offset / 16 to the address field (no
      // shared-memory address reaches 2^18, so the field cannot carry).
      const uint64_t dQ = smem_desc_sw128(smem_u32(sm.q[0]), 16, 1024);
      const uint64_t dK0 = smem_desc_sw128(smem_u32(sm.kv[0][0][0]), 16, 1024);
      const uint64_t dV0 = smem_desc_sw128(smem_u32(sm.kv[0][1][0]), HT, 1024);
      constexpr uint64_t kStage = sizeof(sm.kv[0]) >> 4;
      auto issue_scores = [&](int t) {
        const uint64_t so = (t % NST) * kStage;
        const uint32_t sc = tbase + kScore + BN * (t % NBUF);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint32_t h = kk >> 2;  // 64-column half of the head dim
          const uint32_t o = 32 * (kk & 3);
          mma_ss(sc, dQ + ((h * HALF_BLOCK + o) >> 4), dK0 + so + ((h * HT + o) >> 4), idS,
                 kk > 0);
        }
        mma_commit(&sm.sc_full[t % NBUF]);
      };
      auto issue_pv = [&](int t) {
        const int s = t % NST;
        const uint32_t sc = tbase + kScore + BN * (t % NBUF);
        // V as an N = DH MN-major operand: its second 64-column half (d = 128)
        // sits HT bytes after the first.  Warpgroup t mod 2's accumulator;
        // its first tile (t < 2) starts it.
        const uint64_t dv = dV0 + s * kStage;
        const uint32_t acc_col = tbase + DH * (t & 1);
#pragma unroll
        for (int c = 0; c < BN / 16; ++c)
          mma_ts(acc_col, sc + 8 * c, dv + ((16 * 128 * c) >> 4), idO, (t >= 2 || c > 0));
        mma_commit(&sm.pv_done[t & 1]);
        mma_commit(&sm.kv_empty[s]);
      };
      if (elect_one()) {
        bool ok = mbar_wait(&sm.bar_q, 0, abort_flag, err);
        tc_fence_after();
        for (int t = 0; ok && t < NBUF && t < T; ++t) {
          ok = mbar_wait(&sm.kv_full[t % NST], (t / NST) & 1, abort_flag, err);
          tc_fence_after();
          if (ok) issue_scores(t);
        }
        for (int t = 0; ok && t < T; ++t) {
          // Tile t's warpgroup has written P~ into buffer t mod NBUF.
          ok = mbar_wait(&sm.op_ready[t % NBUF], (t / NBUF) & 1, abort_flag, err);
          if (!ok) break;
          tc_fence_after();
          issue_pv(t);
          if (t + NBUF < T) {
            const int tn = t + NBUF;
            ok = mbar_wait(&sm.kv_full[tn % NST], (tn / NST) & 1, abort_flag, err);
            if (!ok) break;
            tc_fence_after();
            issue_scores(tn);  // after tile t's P V GEMMs have read the buffer
          }
        }
        mma_commit(&sm.out_full);
      }
      __syncwarp();
    }
  } else {
    const int wg = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t acc_own = tbase + lane_off + DH * wg;  // this warpgroup's O~
    const int gr = row0 + r;
    const size_t rowvec = static_cast<size_t>(bh) * Nq + gr;
    const float c1 = tau * kLog2e;
    const int jmax = causal ? min(Nk - 1, gr) : Nk - 1;  // visible keys j <= jmax
    float m = -INFINITY, l = 0.f;
    bool ok = true;

    for (int u = 0;; ++u) {
      const int t = 2 * u + wg;
      if (t >= T) break;
      ok = ok && mbar_wait_warp(&sm.sc_full[t % NBUF], (t / NBUF) & 1, abort_flag, err);
      if (!ok) break;
      tc_fence_after();
      const uint32_t sc = tbase + lane_off + kScore + BN * (t % NBUF);
      const int col0 = t * BN;
      // Only tiles that reach past Nk or past the block's first row need the mask.
      const bool masked = (col0 + BN > Nk) || (causal && col0 + BN - 1 > row0);
      // The tile's visible maximum.  At d = 64 (two 64-column groups) the
      // second group is read twice, so that only one group is held in
      // registers at a time: P~ of columns 16c..16c+15 goes to columns
      // 8c..8c+7, i.e. group 1's P~ lands on group 0's scores.
      float mr = -INFINITY;
      uint32_t s[4][16];
      if (BN == 128) {
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld16(sc + 64 + 16 * q, s[q]);
        tmem_wait_ld();
        mr = masked ? prep_max64<true>(s, col0 + 64, jmax) : prep_max64<false>(s, col0 + 64, jmax);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld16(sc + 16 * q, s[q]);
      tmem_wait_ld();
      mr = fmaxf(mr, masked ? prep_max64<true>(s, col0, jmax) : prep_max64<false>(s, col0, jmax));
      // Raise m only when the tile's maximum exceeds it by more than
      // kRescale; then the running sum and this warpgroup's O~ (all its
      // earlier tiles) are scaled down by exp2(m_old - m_new) first.
      const float mt = mr * c1;
      const bool raise = mt > m + kRescale;
      const float factor = raise ? (m == -INFINITY ? 0.f : ex2_approx(m - mt)) : 1.f;
      if (raise) {
        l *= factor;
        m = mt;
      }
      if (__any_sync(0xffffffffu, raise && factor < 1.f) && u > 0) {
        // Rescale this warp's rows of O~ once its previous tile's P V GEMMs
        // are done; a lane whose m did not move multiplies by 1.
        ok = mbar_wait_warp(&sm.pv_done[wg], (u - 1) & 1, abort_flag, err);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < DH / 16; ++c) {
          uint32_t v[16];
          tmem_ld16(acc_own + 16 * c, v);
          tmem_wait_ld();
          uint32_t w0[8], w1[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            w0[k] = __float_as_uint(u2f(v[k]) * factor);
            w1[k] = __float_as_uint(u2f(v[8 + k]) * factor);
          }
          tmem_st8(acc_own + 16 * c, w0);
          tmem_st8(acc_own + 16 * c + 8, w1);
        }
      }
      // P~ of columns 16c..16c+15 goes to columns 8c..8c+7 (already read).
#pragma unroll
      for (int g = 0; g < BN / 64; ++g) {
        if (g > 0) {
#pragma unroll
          for (int q = 0; q < 4; ++q) tmem_ld16(sc + 64 * g + 16 * q, s[q]);
          tmem_wait_ld();
        }
        uint32_t pk[4][8];
        if (masked) prep_p64<true>(s, col0 + 64 * g, jmax, c1, m, l, pk);
        else prep_p64<false>(s, col0 + 64 * g, jmax, c1, m, l, pk);
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_st8(sc + 32 * g + 8 * q, pk[q]);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(&sm.op_ready[t % NBUF]);
    }

    ok = mbar_wait_warp(&sm.out_full, 0, abort_flag, err) && ok;
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);
    tc_fence_after();
    // Merge the two warpgroups' (m, l, O~): m* = max, s_w = exp2(m_w - m*),
    // O = (s_0 O~_0 + s_1 O~_1) / (s_0 l_0 + s_1 l_1).  A warpgroup with no
    // visible column so far (m = -inf) contributes nothing.
    sm.part_m[wg][r] = m;
    sm.part_l[wg][r] = l;
    named_bar_sync(1, 256);
    const float m0 = sm.part_m[0][r], m1 = sm.part_m[1][r];
    const float mm = fmaxf(m0, m1);  // finite: key 0 is visible to every row
    const float s0 = m0 == -INFINITY ? 0.f : ex2_approx(m0 - mm);
    const float s1 = m1 == -INFINITY ? 0.f : ex2_approx(m1 - mm);
    const float lsum = s0 * sm.part_l[0][r] + s1 * sm.part_l[1][r];
    const float inv = 1.f / lsum;
    const bool one = T < 2;  // warpgroup 1 had no tile: its accumulator was never written
    // Every MMA is done, so the ring is idle: each thread forms its row of O
    // in shared memory, then the tile leaves with coalesced stores and D is
    // the row dot with dO read coalesced (DH / 4 consecutive lanes per row,
    // summed by shuffles).
    constexpr int LD = kStageLd0<DH>;
    static_assert(BM * LD * 4 <= sizeof(Smem0<DH>::kv), "epilogue staging fits in the ring");
    float* st = reinterpret_cast<float*>(&sm.kv[0][0][0][0]);
#pragma unroll
    for (int h = 0; h < DH / 32; ++h) {  // warpgroup wg forms columns [DH/2 wg, DH/2 (wg+1))
      const int col = (DH / 2) * wg + 16 * h;
      uint32_t v0[16], v1[16];
      tmem_ld16(tbase + lane_off + col, v0);
      tmem_ld16(tbase + lane_off + DH + col, v1);
      tmem_wait_ld();
      float4* s4 = reinterpret_cast<float4*>(st + r * LD + col);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          o[q] = (s0 * u2f(v0[4 * k + q]) + (one ? 0.f : s1 * u2f(v1[4 * k + q]))) * inv;
        s4[k] = make_float4(o[0], o[1], o[2], o[3]);
      }
    }
    named_bar_sync(1, 256);
    if (ok && wg == 0 && gr < Nq) L[rowvec] = (mm + __log2f(lsum)) * kLn2;
    const int tid = threadIdx.x - 64;  // 0 .. 255
    const int rows = min(BM, Nq - row0);
    const size_t blk = (static_cast<size_t>(bh) * Nq + row0) * DH;
    constexpr int kRow4 = DH / 4;  // float4 per row: 16 or 32 lanes
    // Every lane runs every iteration (the shuffles need the whole warp);
    // rows past N_q only skip their memory accesses.
    for (int f = tid; f < BM * kRow4; f += 256) {
      const int rr = f / kRow4, c4 = f % kRow4;
      const bool live = ok && rr < rows;
      const float4 v = *reinterpret_cast<const float4*>(st + rr * LD + 4 * c4);
      float dp = 0.f;
      if (live) {
        reinterpret_cast<float4*>(O + blk)[f] = v;
        if (dO) {  // dO = D = null: the forward only, no D
          const uint2 raw = reinterpret_cast<const uint2*>(
              reinterpret_cast<const uint16_t*>(dO) + blk)[f];  // 4 bf16 of dO
          dp = __uint_as_float(raw.x << 16) * v.x + __uint_as_float(raw.x & 0xFFFF0000u) * v.y +
               __uint_as_float(raw.y << 16) * v.z + __uint_as_float(raw.y & 0xFFFF0000u) * v.w;
        }
      }
#pragma unroll
      for (int o = kRow4 / 2; o > 0; o >>= 1) dp += __shfl_xor_sync(0xffffffffu, dp, o);
      if (live && D && c4 == 0) D[static_cast<size_t>(bh) * Nq + row0 + rr] = dp;
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

template <int DH>
cudaError_t launch_prep(const PrepArgs& a) {
  const int BH = a.B * a.H;
  const int BHkv = a.B * a.Hkv;
  CUtensorMap mq, mk, mv;
  cudaError_t e = tc_map_bf16(&mq, a.Q, BH, a.Nq, kTcRows, DH);
  if (e == cudaSuccess) e = tc_map_bf16(&mk, a.K, BHkv, a.Nk, PrepCfg<DH>::kBN, DH);
  if (e == cudaSuccess) e = tc_map_bf16(&mv, a.V, BHkv, a.Nk, PrepCfg<DH>::kBN, DH);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(Smem0<DH>) + 1024;
  e = tc_set_smem(reinterpret_cast<const void*>(tc_prep_kernel<DH>), (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Nq + BM - 1) / BM, a.H, a.B);
  tc_prep_kernel<DH><<<grid, NTHREADS, smem, a.stream>>>(
      mq, mk, mv, (const __nv_bfloat16*)a.dO, a.O, a.L, a.D, a.H, a.Hkv, a.Nq, a.Nk, a.tau,
      a.causal ? 1 : 0, a.err);
  return cudaGetLastError();
}

}  // namespace

bool tc_prep_supported(const PrepArgs& a) { return a.bf16 && (a.d == 64 || a.d == 128); }

cudaError_t tc_prep(const PrepArgs& a) {
  return a.d == 128 ? launch_prep<128>(a) : launch_prep<64>(a);
}

}  // namespace flashbob
