// fp32 CUDA-core kernels for the attention row state and the exact
// backward-over-backward, any head dim 1 <= d <= 128, fp32 or bf16 inputs.
//
// They follow the two-pass schedule of "FlashBoB: I/O-Efficient Exact
// Backward-over-Backward for Softmax Attention" (paper notes, 关键设计 2):
// pass 1 keeps a block of query rows resident and streams key/value column
// tiles, pass 2 keeps a block of key rows resident and streams query row
// tiles together with the row scalars (alpha, E) written by pass 1.  P is
// recomputed from the saved logsumexp L (FlashAttention backward blog,
// section 二), so no N x N tensor reaches device memory.
//
// Tiles: 32 x 32 scores per step, 256 threads; thread t owns row t/8 of the
// tile and the 4 columns (t%8) + 8u, so the 8 threads of a row sit in one
// warp and row reductions are warp shuffles.  Everything is fp32.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"

namespace flashbob {
namespace {

constexpr int SB = kSimtTile;
constexpr int NT = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// dst[r][k] (row pitch DP + 1) <- src rows row0.. of one head, zero outside
// the N x d slice.
template <typename T, int DP>
__device__ __forceinline__ void load_tile(float* dst, const T* src, int row0, int N, int d) {
  for (int idx = threadIdx.x; idx < SB * DP; idx += NT) {
    const int r = idx / DP, k = idx % DP;
    const int gr = row0 + r;
    float v = 0.f;
    if (gr < N && k < d) v = ldf(src + (size_t)gr * d + k);
    dst[r * (DP + 1) + k] = v;
  }
}

__device__ __forceinline__ float row8_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  return v;
}

__device__ __forceinline__ float row8_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  return v;
}

// ---------------------------------------------------------------------------
// Row state: O = P V, L = logsumexp(tau Q K^T), D = rowsum(dO o O).
// Online max/sum over column tiles (FlashAttention backward blog, section 二).
// ---------------------------------------------------------------------------
template <typename T, int DP>
__global__ void __launch_bounds__(NT) prep_kernel(const T* __restrict__ Q, const T* __restrict__ K,
                                                  const T* __restrict__ V, const T* __restrict__ dO,
                                                  float* __restrict__ O, float* __restrict__ L,
                                                  float* __restrict__ D, int H, int Hkv, int Nq,
                                                  int Nk, int d, float tau, int causal) {
  extern __shared__ float sm[];
  float* Qs = sm;
  float* Ks = Qs + SB * (DP + 1);
  float* Vs = Ks + SB * (DP + 1);
  float* Ps = Vs + SB * (DP + 1);  // [SB][SB + 1]
  const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;
  const size_t base = bh * Nq * d;
  // key/value head shared by this query head (grouped-query attention)
  const size_t kbase = ((size_t)blockIdx.z * Hkv + blockIdx.y / (H / Hkv)) * Nk * d;
  const int row0 = blockIdx.x * SB;
  const int t = threadIdx.x, r = t >> 3, q = t & 7;
  const float c = tau * kLog2e;  // scores in log2 units

  load_tile<T, DP>(Qs, Q + base, row0, Nq, d);
  float m = -INFINITY, l = 0.f;
  float acc[DP / 8];
#pragma unroll
  for (int j = 0; j < DP / 8; ++j) acc[j] = 0.f;

  const int gr = row0 + r;
  const int col_end = causal ? min(Nk, row0 + SB) : Nk;  // keys j <= i under the causal mask
  for (int col0 = 0; col0 < col_end; col0 += SB) {
    __syncthreads();
    load_tile<T, DP>(Ks, K + kbase, col0, Nk, d);
    load_tile<T, DP>(Vs, V + kbase, col0, Nk, d);
    __syncthreads();
    float s[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) s[u] = 0.f;
    for (int k = 0; k < d; ++k) {
      const float qv = Qs[r * (DP + 1) + k];
#pragma unroll
      for (int u = 0; u < 4; ++u) s[u] = fmaf(qv, Ks[(q + 8 * u) * (DP + 1) + k], s[u]);
    }
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = col0 + q + 8 * u;
      s[u] = (j < Nk && !(causal && j > gr)) ? s[u] * c : -INFINITY;
      mx = fmaxf(mx, s[u]);
    }
    mx = row8_max(mx);
    const float m_new = fmaxf(m, mx);  // finite: column col0 <= row0 is always visible
    const float scale = exp2f(m - m_new);
    float ps = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float p = exp2f(s[u] - m_new);
      ps += p;
      Ps[r * (SB + 1) + q + 8 * u] = p;
    }
    ps = row8_sum(ps);
    l = l * scale + ps;
    m = m_new;
    __syncwarp();
#pragma unroll
    for (int j = 0; j < DP / 8; ++j) acc[j] *= scale;
    for (int cc = 0; cc < SB; ++cc) {
      const float p = Ps[r * (SB + 1) + cc];
#pragma unroll
      for (int j = 0; j < DP / 8; ++j) acc[j] = fmaf(p, Vs[cc * (DP + 1) + q + 8 * j], acc[j]);
    }
    __syncwarp();
  }

  const float inv_l = 1.f / l;
  float dsum = 0.f;
#pragma unroll
  for (int j = 0; j < DP / 8; ++j) {
    const int k = q + 8 * j;
    const float o = acc[j] * inv_l;
    if (gr < Nq && k < d) {
      O[base + (size_t)gr * d + k] = o;
      if (dO) dsum = fmaf(ldf(dO + base + (size_t)gr * d + k), o, dsum);
    }
  }
  dsum = row8_sum(dsum);
  if (gr < Nq && q == 0) {
    L[bh * Nq + gr] = (m + log2f(l)) * kLn2;
    if (D) D[bh * Nq + gr] = dsum;  // dO = D = null: forward only
  }
}

// ---------------------------------------------------------------------------
// Pass 1 (row-resident).  Per column tile: S, dP, F, G; elementwise
// P = exp(S - L), dS = P o (dP - D), d~P0 = F o (dP - D) + G; accumulate
// alpha, E0 (row sums) and B = P K, R = (P o dP) K,
// Omega = (P o d~P0) K + dS U_K, d~dO0 = P U_V + (P o F) V; then the affine
// correction E = E0 - alpha D, d~dO = d~dO0 - alpha O,
// d~Q = tau (Omega - alpha R - E B)  (paper notes, 关键设计 1).
// ---------------------------------------------------------------------------
template <typename T, int DP>
__global__ void __launch_bounds__(NT) pass1_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
    const float* __restrict__ O, const T* __restrict__ dO, const float* __restrict__ L,
    const float* __restrict__ D, const T* __restrict__ UQ, const T* __restrict__ UK,
    const T* __restrict__ UV, float tau, float* __restrict__ dQt, float* __restrict__ ddOt,
    float* __restrict__ alpha, float* __restrict__ E, int H, int Hkv, int Nq, int Nk, int d,
    int causal) {
  extern __shared__ float sm[];
  constexpr int TP = SB * (DP + 1);
  constexpr int OP = SB * (SB + 1);
  float* Qs = sm;
  float* dOs = Qs + TP;
  float* UQs = dOs + TP;
  float* Ks = UQs + TP;
  float* Vs = Ks + TP;
  float* UKs = Vs + TP;
  float* UVs = UKs + TP;
  float* Ps = UVs + TP;
  float* PdPs = Ps + OP;
  float* PdPt0s = PdPs + OP;
  float* dSs = PdPt0s + OP;
  float* PFs = dSs + OP;

  const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;
  const size_t base = bh * Nq * d;
  // key/value head shared by this query head (grouped-query attention)
  const size_t kbase = ((size_t)blockIdx.z * Hkv + blockIdx.y / (H / Hkv)) * Nk * d;
  const int row0 = blockIdx.x * SB;
  const int t = threadIdx.x, r = t >> 3, q = t & 7;
  const int gr = row0 + r;
  const float c = tau * kLog2e;
  const float Lr2 = gr < Nq ? L[bh * Nq + gr] * kLog2e : 0.f;
  const float Dr = gr < Nq ? D[bh * Nq + gr] : 0.f;

  load_tile<T, DP>(Qs, Q + base, row0, Nq, d);
  load_tile<T, DP>(dOs, dO + base, row0, Nq, d);
  load_tile<T, DP>(UQs, UQ + base, row0, Nq, d);

  float accB[DP / 8], accR[DP / 8], accW[DP / 8], accO[DP / 8];
#pragma unroll
  for (int j = 0; j < DP / 8; ++j) accB[j] = accR[j] = accW[j] = accO[j] = 0.f;
  float a_part = 0.f, e_part = 0.f;
  const int col_end = causal ? min(Nk, row0 + SB) : Nk;

  for (int col0 = 0; col0 < col_end; col0 += SB) {
    __syncthreads();
    load_tile<T, DP>(Ks, K + kbase, col0, Nk, d);
    load_tile<T, DP>(Vs, V + kbase, col0, Nk, d);
    load_tile<T, DP>(UKs, UK + kbase, col0, Nk, d);
    load_tile<T, DP>(UVs, UV + kbase, col0, Nk, d);
    __syncthreads();
    float s[4], dp[4], f[4], g[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) s[u] = dp[u] = f[u] = g[u] = 0.f;
    for (int k = 0; k < d; ++k) {
      const float qv = Qs[r * (DP + 1) + k];
      const float dov = dOs[r * (DP + 1) + k];
      const float uqv = UQs[r * (DP + 1) + k];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int cr = (q + 8 * u) * (DP + 1) + k;
        s[u] = fmaf(qv, Ks[cr], s[u]);
        dp[u] = fmaf(dov, Vs[cr], dp[u]);
        f[u] = fmaf(uqv, Ks[cr], fmaf(qv, UKs[cr], f[u]));
        g[u] = fmaf(dov, UVs[cr], g[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int cc = q + 8 * u;
      const int j = col0 + cc;
      const float p = (j < Nk && !(causal && j > gr)) ? exp2f(s[u] * c - Lr2) : 0.f;
      const float x = dp[u] - Dr;
      const float ft = f[u] * tau;
      const float dpt0 = fmaf(ft, x, g[u]);
      const float pf = p * ft;
      const float pdpt0 = p * dpt0;
      a_part += pf;
      e_part += pdpt0;
      Ps[r * (SB + 1) + cc] = p;
      PdPs[r * (SB + 1) + cc] = p * dp[u];
      PdPt0s[r * (SB + 1) + cc] = pdpt0;
      dSs[r * (SB + 1) + cc] = p * x;
      PFs[r * (SB + 1) + cc] = pf;
    }
    __syncwarp();
    for (int cc = 0; cc < SB; ++cc) {
      const float p = Ps[r * (SB + 1) + cc];
      const float pdp = PdPs[r * (SB + 1) + cc];
      const float pdpt0 = PdPt0s[r * (SB + 1) + cc];
      const float ds = dSs[r * (SB + 1) + cc];
      const float pf = PFs[r * (SB + 1) + cc];
#pragma unroll
      for (int j = 0; j < DP / 8; ++j) {
        const int ck = cc * (DP + 1) + q + 8 * j;
        const float kv = Ks[ck];
        accB[j] = fmaf(p, kv, accB[j]);
        accR[j] = fmaf(pdp, kv, accR[j]);
        accW[j] = fmaf(pdpt0, kv, fmaf(ds, UKs[ck], accW[j]));
        accO[j] = fmaf(p, UVs[ck], fmaf(pf, Vs[ck], accO[j]));
      }
    }
  }

  const float al = row8_sum(a_part);
  const float e0 = row8_sum(e_part);
  const float Ei = e0 - al * Dr;
  if (gr < Nq) {
#pragma unroll
    for (int j = 0; j < DP / 8; ++j) {
      const int k = q + 8 * j;
      if (k < d) {
        const size_t o = base + (size_t)gr * d + k;
        dQt[o] = tau * (accW[j] - al * accR[j] - Ei * accB[j]);
        ddOt[o] = accO[j] - al * O[o];
      }
    }
    if (q == 0) {
      alpha[bh * Nq + gr] = al;
      E[bh * Nq + gr] = Ei;
    }
  }
}

// ---------------------------------------------------------------------------
// Attention JVP along (U_Q, U_K, U_V): pass 1 without dO.  Per column tile
// S = Q K^T and its tangent F = tau (U_Q K^T + Q U_K^T); P = exp(S - L);
// row sums L' += P o F and the accumulator P U_V + (P o F) V; at the end
// O' = P U_V + (P o F) V - L' O  (the d~dO and alpha of pass 1, whose
// other terms all carry dO).
// ---------------------------------------------------------------------------
template <typename T, int DP>
__global__ void __launch_bounds__(NT) jvp_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
    const float* __restrict__ O, const float* __restrict__ L, const T* __restrict__ UQ,
    const T* __restrict__ UK, const T* __restrict__ UV, float tau, float* __restrict__ Od,
    float* __restrict__ Ld, int H, int Hkv, int Nq, int Nk, int d, int causal) {
  extern __shared__ float sm[];
  constexpr int TP = SB * (DP + 1);
  constexpr int OP = SB * (SB + 1);
  float* Qs = sm;
  float* UQs = Qs + TP;
  float* Ks = UQs + TP;
  float* Vs = Ks + TP;
  float* UKs = Vs + TP;
  float* UVs = UKs + TP;
  float* Ps = UVs + TP;
  float* PFs = Ps + OP;

  const size_t bh = (size_t)blockIdx.z * H + blockIdx.y;
  const size_t base = bh * Nq * d;
  const size_t kbase = ((size_t)blockIdx.z * Hkv + blockIdx.y / (H / Hkv)) * Nk * d;
  const int row0 = blockIdx.x * SB;
  const int t = threadIdx.x, r = t >> 3, q = t & 7;
  const int gr = row0 + r;
  const float c = tau * kLog2e;
  const float Lr2 = gr < Nq ? L[bh * Nq + gr] * kLog2e : 0.f;

  load_tile<T, DP>(Qs, Q + base, row0, Nq, d);
  load_tile<T, DP>(UQs, UQ + base, row0, Nq, d);

  float accO[DP / 8];
#pragma unroll
  for (int j = 0; j < DP / 8; ++j) accO[j] = 0.f;
  float a_part = 0.f;
  const int col_end = causal ? min(Nk, row0 + SB) : Nk;

  for (int col0 = 0; col0 < col_end; col0 += SB) {
    __syncthreads();
    load_tile<T, DP>(Ks, K + kbase, col0, Nk, d);
    load_tile<T, DP>(Vs, V + kbase, col0, Nk, d);
    load_tile<T, DP>(UKs, UK + kbase, col0, Nk, d);
    load_tile<T, DP>(UVs, UV + kbase, col0, Nk, d);
    __syncthreads();
    float s[4], f[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) s[u] = f[u] = 0.f;
    for (int k = 0; k < d; ++k) {
      const float qv = Qs[r * (DP + 1) + k];
      const float uqv = UQs[r * (DP + 1) + k];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int cr = (q + 8 * u) * (DP + 1) + k;
        s[u] = fmaf(qv, Ks[cr], s[u]);
        f[u] = fmaf(uqv, Ks[cr], fmaf(qv, UKs[cr], f[u]));
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int cc = q + 8 * u;
      const int j = col0 + cc;
      const float p = (j < Nk && !(causal && j > gr)) ? exp2f(s[u] * c - Lr2) : 0.f;
      const float pf = p * (f[u] * tau);
      a_part += pf;
      Ps[r * (SB + 1) + cc] = p;
      PFs[r * (SB + 1) + cc] = pf;
    }
    __syncwarp();
    for (int cc = 0; cc < SB; ++cc) {
      const float p = Ps[r * (SB + 1) + cc];
      const float pf = PFs[r * (SB + 1) + cc];
#pragma unroll
      for (int j = 0; j < DP / 8; ++j) {
        const int ck = cc * (DP + 1) + q + 8 * j;
        accO[j] = fmaf(p, UVs[ck], fmaf(pf, Vs[ck], accO[j]));
      }
    }
  }

  const float al = row8_sum(a_part);
  if (gr < Nq) {
#pragma unroll
    for (int j = 0; j < DP / 8; ++j) {
      const int k = q + 8 * j;
      if (k < d) {
        const size_t o = base + (size_t)gr * d + k;
        Od[o] = accO[j] - al * O[o];
      }
    }
    if (q == 0) Ld[bh * Nq + gr] = al;
  }
}

// ---------------------------------------------------------------------------
// Pass 2 (column-resident).  Per query-row tile, transposed scores; with the
// row scalars L, D, alpha, E of the streamed rows:
//   dS = P o (dP - D), d~S = P o (F o (dP - D) + G - alpha dP - E),
//   W = P o (F - alpha);  d~K += d~S^T Q + dS^T U_Q (times tau), d~V += W^T dO.
// Each key row's outputs are summed on chip and written once, no atomics.
// ---------------------------------------------------------------------------
template <typename T, int DP>
__global__ void __launch_bounds__(NT) pass2_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
    const T* __restrict__ dO, const float* __restrict__ L, const float* __restrict__ D,
    const float* __restrict__ alpha, const float* __restrict__ E, const T* __restrict__ UQ,
    const T* __restrict__ UK, const T* __restrict__ UV, float tau, float* __restrict__ dKt,
    float* __restrict__ dVt, int H, int Hkv, int Nq, int Nk, int d, int causal) {
  extern __shared__ float sm[];
  constexpr int TP = SB * (DP + 1);
  constexpr int OP = SB * (SB + 1);
  float* Ks = sm;
  float* Vs = Ks + TP;
  float* UKs = Vs + TP;
  float* UVs = UKs + TP;
  float* Qs = UVs + TP;
  float* dOs = Qs + TP;
  float* UQs = dOs + TP;
  float* dSTs = UQs + TP;
  float* dStTs = dSTs + OP;
  float* WTs = dStTs + OP;
  float* Ls2 = WTs + OP;
  float* Ds = Ls2 + SB;
  float* As = Ds + SB;
  float* Es = As + SB;

  // One CTA per key block of a key/value head; the H / Hkv query heads that
  // share the head are summed on chip (grouped-query attention).
  const int G = H / Hkv;
  const size_t kbase = ((size_t)blockIdx.z * Hkv + blockIdx.y) * Nk * d;
  const int j0 = blockIdx.x * SB;
  const int t = threadIdx.x, jr = t >> 3, q = t & 7;
  const float c = tau * kLog2e;

  load_tile<T, DP>(Ks, K + kbase, j0, Nk, d);
  load_tile<T, DP>(Vs, V + kbase, j0, Nk, d);
  load_tile<T, DP>(UKs, UK + kbase, j0, Nk, d);
  load_tile<T, DP>(UVs, UV + kbase, j0, Nk, d);

  float accK[DP / 8], accV[DP / 8];
#pragma unroll
  for (int j = 0; j < DP / 8; ++j) accK[j] = accV[j] = 0.f;

  const int gj = j0 + jr;
  for (int hh = 0; hh < G; ++hh) {
    const size_t bh = (size_t)blockIdx.z * H + (size_t)blockIdx.y * G + hh;
    const size_t base = bh * Nq * d;
    // Under the causal mask key j is seen by queries i >= j only (none when
    // j >= Nq: those keys keep d~K = d~V = 0).
    for (int row0 = causal ? j0 : 0; row0 < Nq; row0 += SB) {
      __syncthreads();
      load_tile<T, DP>(Qs, Q + base, row0, Nq, d);
      load_tile<T, DP>(dOs, dO + base, row0, Nq, d);
      load_tile<T, DP>(UQs, UQ + base, row0, Nq, d);
      if (t < SB) {
        const int gi = row0 + t;
        const bool ok = gi < Nq;
        Ls2[t] = ok ? L[bh * Nq + gi] * kLog2e : 0.f;
        Ds[t] = ok ? D[bh * Nq + gi] : 0.f;
        As[t] = ok ? alpha[bh * Nq + gi] : 0.f;
        Es[t] = ok ? E[bh * Nq + gi] : 0.f;
      }
      __syncthreads();
      float s[4], dp[4], f[4], g[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) s[u] = dp[u] = f[u] = g[u] = 0.f;
      for (int k = 0; k < d; ++k) {
        const int jk = jr * (DP + 1) + k;
        const float kv = Ks[jk], vv = Vs[jk], ukv = UKs[jk], uvv = UVs[jk];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ik = (q + 8 * u) * (DP + 1) + k;
          const float qv = Qs[ik];
          s[u] = fmaf(kv, qv, s[u]);
          dp[u] = fmaf(vv, dOs[ik], dp[u]);
          f[u] = fmaf(kv, UQs[ik], fmaf(ukv, qv, f[u]));
          g[u] = fmaf(uvv, dOs[ik], g[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int ii = q + 8 * u;
        const int i = row0 + ii;
        const float p = (i < Nq && !(causal && i < gj)) ? exp2f(s[u] * c - Ls2[ii]) : 0.f;
        const float x = dp[u] - Ds[ii];
        const float ft = f[u] * tau;
        const float a = As[ii];
        dSTs[jr * (SB + 1) + ii] = p * x;
        dStTs[jr * (SB + 1) + ii] = p * (fmaf(ft, x, g[u]) - a * dp[u] - Es[ii]);
        WTs[jr * (SB + 1) + ii] = p * (ft - a);
      }
      __syncwarp();
      for (int ii = 0; ii < SB; ++ii) {
        const float ds = dSTs[jr * (SB + 1) + ii];
        const float dst = dStTs[jr * (SB + 1) + ii];
        const float w = WTs[jr * (SB + 1) + ii];
#pragma unroll
        for (int j = 0; j < DP / 8; ++j) {
          const int ik = ii * (DP + 1) + q + 8 * j;
          accK[j] = fmaf(dst, Qs[ik], fmaf(ds, UQs[ik], accK[j]));
          accV[j] = fmaf(w, dOs[ik], accV[j]);
        }
      }
    }

  }  // query heads of the group

  if (gj < Nk) {
#pragma unroll
    for (int j = 0; j < DP / 8; ++j) {
      const int k = q + 8 * j;
      if (k < d) {
        const size_t o = kbase + (size_t)gj * d + k;
        dKt[o] = tau * accK[j];
        dVt[o] = accV[j];
      }
    }
  }
}

size_t prep_smem(int dp) { return (size_t)(3 * SB * (dp + 1) + SB * (SB + 1)) * sizeof(float); }
size_t pass1_smem(int dp) { return (size_t)(7 * SB * (dp + 1) + 5 * SB * (SB + 1)) * sizeof(float); }
size_t jvp_smem(int dp) { return (size_t)(6 * SB * (dp + 1) + 2 * SB * (SB + 1)) * sizeof(float); }
size_t pass2_smem(int dp) {
  return (size_t)(7 * SB * (dp + 1) + 3 * SB * (SB + 1) + 4 * SB) * sizeof(float);
}

template <typename T, int DP>
cudaError_t run_prep(const PrepArgs& a) {
  const size_t smem = prep_smem(DP);
  cudaError_t e = cudaFuncSetAttribute(prep_kernel<T, DP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Nq + SB - 1) / SB, a.H, a.B);
  prep_kernel<T, DP><<<grid, NT, smem, a.stream>>>(
      (const T*)a.Q, (const T*)a.K, (const T*)a.V, (const T*)a.dO, a.O, a.L, a.D, a.H, a.Hkv,
      a.Nq, a.Nk, a.d, a.tau, a.causal ? 1 : 0);
  return cudaGetLastError();
}

template <typename T, int DP>
cudaError_t run_bob(const BobArgs& a) {
  const size_t s1 = pass1_smem(DP), s2 = pass2_smem(DP);
  cudaError_t e = cudaFuncSetAttribute(pass1_kernel<T, DP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(pass2_kernel<T, DP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)s2);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Nq + SB - 1) / SB, a.H, a.B);
  if (a.passes & kPass1) {
    pass1_kernel<T, DP><<<grid, NT, s1, a.stream>>>(
        (const T*)a.Q, (const T*)a.K, (const T*)a.V, a.O, (const T*)a.dO, a.L, a.D,
        (const T*)a.UQ, (const T*)a.UK, (const T*)a.UV, a.tau, a.dQt, a.ddOt, a.alpha, a.E, a.H,
        a.Hkv, a.Nq, a.Nk, a.d, a.causal ? 1 : 0);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.passes & kPass2) {
    const dim3 grid2((a.Nk + SB - 1) / SB, a.Hkv, a.B);  // one CTA per key block of a shared head
    pass2_kernel<T, DP><<<grid2, NT, s2, a.stream>>>(
        (const T*)a.Q, (const T*)a.K, (const T*)a.V, (const T*)a.dO, a.L, a.D, a.alpha, a.E,
        (const T*)a.UQ, (const T*)a.UK, (const T*)a.UV, a.tau, a.dKt, a.dVt, a.H, a.Hkv, a.Nq,
        a.Nk, a.d, a.causal ? 1 : 0);
    e = cudaGetLastError();
  }
  return e;
}

template <typename T, int DP>
cudaError_t run_jvp(const JvpArgs& a) {
  const size_t smem = jvp_smem(DP);
  cudaError_t e = cudaFuncSetAttribute(jvp_kernel<T, DP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Nq + SB - 1) / SB, a.H, a.B);
  jvp_kernel<T, DP><<<grid, NT, smem, a.stream>>>(
      (const T*)a.Q, (const T*)a.K, (const T*)a.V, a.O, a.L, (const T*)a.UQ, (const T*)a.UK,
      (const T*)a.UV, a.tau, a.Od, a.Ld, a.H, a.Hkv, a.Nq, a.Nk, a.d, a.causal ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace

cudaError_t simt_jvp(const JvpArgs& a) {
  if (a.bf16) return a.d <= 64 ? run_jvp<__nv_bfloat16, 64>(a) : run_jvp<__nv_bfloat16, 128>(a);
  return a.d <= 64 ? run_jvp<float, 64>(a) : run_jvp<float, 128>(a);
}

size_t simt_pass1_smem(int d) { return pass1_smem(d <= 64 ? 64 : 128); }
size_t simt_pass2_smem(int d) { return pass2_smem(d <= 64 ? 64 : 128); }

cudaError_t simt_prep(const PrepArgs& a) {
  if (a.bf16) return a.d <= 64 ? run_prep<__nv_bfloat16, 64>(a) : run_prep<__nv_bfloat16, 128>(a);
  return a.d <= 64 ? run_prep<float, 64>(a) : run_prep<float, 128>(a);
}

cudaError_t simt_bob(const BobArgs& a) {
  if (a.bf16) return a.d <= 64 ? run_bob<__nv_bfloat16, 64>(a) : run_bob<__nv_bfloat16, 128>(a);
  return a.d <= 64 ? run_bob<float, 64>(a) : run_bob<float, 128>(a);
}

}  // namespace flashbob
