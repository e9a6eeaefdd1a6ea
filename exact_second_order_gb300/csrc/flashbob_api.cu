// C ABI of libflashbob: argument checks, dispatch and the device error word.
// The declarations and their contracts are in include/flashbob.h.
#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/flashbob.h"
#include "internal.h"

namespace flashbob {
namespace {

// One error word per device that loads the library; kernels receive its
// device address (taken with cudaGetSymbolAddress while that device is
// current) and write a nonzero code when a bounded wait gives up.
__device__ unsigned int g_error_word;

constexpr int kMaxDevices = 64;
unsigned int* g_error_ptr[kMaxDevices];
std::mutex g_error_mu;

struct Range {
  uintptr_t lo, hi;
};

bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

flashbob_status check_sizes(int B, int H, int Hkv, int Nq, int Nk, int d, float tau) {
  if (B <= 0 || H <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || d <= 0)
    return FLASHBOB_ERR_INVALID_ARG;
  if (H % Hkv != 0) return FLASHBOB_ERR_INVALID_ARG;
  if (!(isfinite(tau) && tau > 0.f)) return FLASHBOB_ERR_INVALID_ARG;
  if (d > 128 || B > kMaxGridY || H > kMaxGridY) return FLASHBOB_ERR_UNSUPPORTED;
  // Kernels index a (batch, head) pair with a 32-bit integer.
  if (static_cast<long long>(B) * H > INT_MAX) return FLASHBOB_ERR_UNSUPPORTED;
  return FLASHBOB_OK;
}

flashbob_status check_dtype(flashbob_dtype t) {
  return (t == FLASHBOB_F32 || t == FLASHBOB_BF16) ? FLASHBOB_OK : FLASHBOB_ERR_INVALID_ARG;
}

}  // namespace

cudaError_t error_word_ptr(unsigned int** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_error_mu);
  if (g_error_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_error_word);
    if (e != cudaSuccess) return e;
    g_error_ptr[dev] = static_cast<unsigned int*>(p);
  }
  *ptr = g_error_ptr[dev];
  return cudaSuccess;
}

namespace {

// Checks shared by flashbob_bob and its two passes: which buffers a pass
// reads and writes follows from a.passes.
flashbob_status run_bob(BobArgs& a, int causal, flashbob_dtype in_dtype) {
  flashbob_status st = check_dtype(in_dtype);
  if (st != FLASHBOB_OK) return st;
  if (causal != 0 && causal != 1) return FLASHBOB_ERR_INVALID_ARG;
  a.causal = causal == 1;
  a.bf16 = in_dtype == FLASHBOB_BF16;
  const bool p1 = a.passes & kPass1, p2 = a.passes & kPass2;
  const size_t B = a.B > 0 ? a.B : 0, dd = a.d > 0 ? a.d : 0;
  const size_t Nq = a.Nq > 0 ? a.Nq : 0, Nk = a.Nk > 0 ? a.Nk : 0;
  const size_t rows = B * (a.H > 0 ? a.H : 0) * Nq;      // query-side rows
  const size_t krows = B * (a.Hkv > 0 ? a.Hkv : 0) * Nk; // key-side rows
  const size_t esz = a.bf16 ? 2 : 4;
  const size_t inb = rows * dd * esz, mat = rows * dd * 4, vec = rows * 4;
  const size_t kinb = krows * dd * esz, kmat = krows * dd * 4;
  struct Buf {
    const void* p;
    size_t bytes;
    bool out;
  };
  Buf bufs[16];
  int n = 0;
  auto add = [&](const void* p, size_t bytes, bool out) { bufs[n++] = Buf{p, bytes, out}; };
  add(a.Q, inb, false);
  add(a.K, kinb, false);
  add(a.V, kinb, false);
  add(a.dO, inb, false);
  add(a.L, vec, false);
  add(a.D, vec, false);
  add(a.UQ, inb, false);
  add(a.UK, kinb, false);
  add(a.UV, kinb, false);
  if (p1) {
    add(a.O, mat, false);
    add(a.dQt, mat, true);
    add(a.ddOt, mat, true);
  }
  if (p2) {
    add(a.dKt, kmat, true);
    add(a.dVt, kmat, true);
  }
  add(a.alpha, vec, p1);  // written by pass 1, read by pass 2
  add(a.E, vec, p1);
  for (int i = 0; i < n; ++i)
    if (!bufs[i].p) return FLASHBOB_ERR_INVALID_ARG;
  st = check_sizes(a.B, a.H, a.Hkv, a.Nq, a.Nk, a.d, a.tau);
  if (st != FLASHBOB_OK) return st;
  for (int i = 0; i < n; ++i)
    if (!aligned16(bufs[i].p)) return FLASHBOB_ERR_MISALIGNED;
  for (int i = 0; i < n; ++i) {
    if (!bufs[i].out) continue;
    const Range o{(uintptr_t)bufs[i].p, (uintptr_t)bufs[i].p + bufs[i].bytes};
    for (int j = 0; j < n; ++j) {
      if (j == i) continue;
      const Range r{(uintptr_t)bufs[j].p, (uintptr_t)bufs[j].p + bufs[j].bytes};
      if (overlaps(o, r)) return FLASHBOB_ERR_INVALID_ARG;
    }
  }
  if (error_word_ptr(&a.err) != cudaSuccess) return FLASHBOB_ERR_CUDA;
  const cudaError_t e = tc_supported(a) ? tc_bob(a) : simt_bob(a);
  return e == cudaSuccess ? FLASHBOB_OK : FLASHBOB_ERR_CUDA;
}
}  // namespace

}  // namespace flashbob

using namespace flashbob;

extern "C" {

const char* flashbob_status_string(flashbob_status s) {
  switch (s) {
    case FLASHBOB_OK: return "FLASHBOB_OK";
    case FLASHBOB_ERR_INVALID_ARG: return "FLASHBOB_ERR_INVALID_ARG";
    case FLASHBOB_ERR_UNSUPPORTED: return "FLASHBOB_ERR_UNSUPPORTED";
    case FLASHBOB_ERR_MISALIGNED: return "FLASHBOB_ERR_MISALIGNED";
    case FLASHBOB_ERR_CUDA: return "FLASHBOB_ERR_CUDA";
    case FLASHBOB_ERR_TIMEOUT: return "FLASHBOB_ERR_TIMEOUT";
  }
  return "FLASHBOB_UNKNOWN_STATUS";
}

flashbob_status flashbob_prep(const void* Q, const void* K, const void* V, const void* dO,
                              float* O, float* L, float* D, int B, int H, int Hkv, int Nq,
                              int Nk, int d, float tau, int causal, flashbob_dtype in_dtype,
                              void* stream) {
  flashbob_status st = check_dtype(in_dtype);
  if (st != FLASHBOB_OK) return st;
  if (causal != 0 && causal != 1) return FLASHBOB_ERR_INVALID_ARG;
  // dO and D are both given (the BoB's row state) or both null (forward only).
  if (!Q || !K || !V || !O || !L || (!dO != !D)) return FLASHBOB_ERR_INVALID_ARG;
  st = check_sizes(B, H, Hkv, Nq, Nk, d, tau);
  if (st != FLASHBOB_OK) return st;
  const void* ptrs[] = {Q, K, V, dO, O, L, D};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return FLASHBOB_ERR_MISALIGNED;
  const size_t rows = (size_t)B * H * Nq, krows = (size_t)B * Hkv * Nk;
  const size_t esz = in_dtype == FLASHBOB_BF16 ? 2 : 4;
  // A null dO / D gets an empty range.
  const size_t dob = dO ? rows * d * esz : 0, db = D ? rows * 4 : 0;
  const Range ins[] = {{(uintptr_t)Q, (uintptr_t)Q + rows * d * esz},
                       {(uintptr_t)K, (uintptr_t)K + krows * d * esz},
                       {(uintptr_t)V, (uintptr_t)V + krows * d * esz},
                       {(uintptr_t)dO, (uintptr_t)dO + dob}};
  const Range outs[] = {{(uintptr_t)O, (uintptr_t)O + rows * d * 4},
                        {(uintptr_t)L, (uintptr_t)L + rows * 4},
                        {(uintptr_t)D, (uintptr_t)D + db}};
  for (const Range& o : outs) {
    for (const Range& i : ins)
      if (overlaps(o, i)) return FLASHBOB_ERR_INVALID_ARG;
    for (const Range& o2 : outs)
      if (&o != &o2 && overlaps(o, o2)) return FLASHBOB_ERR_INVALID_ARG;
  }
  PrepArgs a{Q,  K,  V, dO,  O,  L, D, B, H, Hkv, Nq, Nk, d, tau, causal == 1,
             in_dtype == FLASHBOB_BF16, (cudaStream_t)stream, nullptr};
  if (error_word_ptr(&a.err) != cudaSuccess) return FLASHBOB_ERR_CUDA;
  const cudaError_t e = tc_prep_supported(a) ? tc_prep(a) : simt_prep(a);
  return e == cudaSuccess ? FLASHBOB_OK : FLASHBOB_ERR_CUDA;
}

flashbob_status flashbob_bob(const void* Q, const void* K, const void* V, const float* O,
                             const void* dO, const float* L, const float* D, const void* UQ,
                             const void* UK, const void* UV, float tau, float* dQt, float* dKt,
                             float* dVt, float* ddOt, float* alpha, float* E, int B, int H,
                             int Hkv, int Nq, int Nk, int d, int causal, flashbob_dtype in_dtype,
                             void* stream) {
  BobArgs a{Q,  K,  V,     O, dO, L,     D,     UQ,    UK, UV, tau, dQt, dKt, dVt,
            ddOt, alpha, E, B, H,  Hkv, Nq, Nk, d, false, false, (cudaStream_t)stream,
            nullptr, kPass1 | kPass2};
  return run_bob(a, causal, in_dtype);
}

flashbob_status flashbob_bob_pass1(const void* Q, const void* K, const void* V, const float* O,
                                   const void* dO, const float* L, const float* D,
                                   const void* UQ, const void* UK, const void* UV, float tau,
                                   float* dQt, float* ddOt, float* alpha, float* E, int B, int H,
                                   int Hkv, int Nq, int Nk, int d, int causal,
                                   flashbob_dtype in_dtype, void* stream) {
  BobArgs a{Q,    K,     V, O, dO, L,   D,  UQ, UK, UV,    tau,   dQt, nullptr, nullptr,
            ddOt, alpha, E, B, H,  Hkv, Nq, Nk, d,  false, false, (cudaStream_t)stream,
            nullptr, kPass1};
  return run_bob(a, causal, in_dtype);
}

flashbob_status flashbob_bob_pass2(const void* Q, const void* K, const void* V, const void* dO,
                                   const float* L, const float* D, const float* alpha,
                                   const float* E, const void* UQ, const void* UK,
                                   const void* UV, float tau, float* dKt, float* dVt, int B,
                                   int H, int Hkv, int Nq, int Nk, int d, int causal,
                                   flashbob_dtype in_dtype, void* stream) {
  // alpha and E are inputs of pass 2; the BobArgs fields keep their names.
  BobArgs a{Q,       K,   V,   nullptr, dO, L, D, UQ, UK, UV, tau, nullptr, dKt, dVt, nullptr,
            (float*)alpha, (float*)E, B, H, Hkv, Nq, Nk, d, false, false, (cudaStream_t)stream,
            nullptr, kPass2};
  return run_bob(a, causal, in_dtype);
}

flashbob_status flashbob_bob_launches(int B, int H, int Hkv, int Nq, int Nk, int d,
                                      flashbob_dtype in_dtype, int* launches) {
  if (check_dtype(in_dtype) != FLASHBOB_OK || launches == nullptr)
    return FLASHBOB_ERR_INVALID_ARG;
  const flashbob_status st = check_sizes(B, H, Hkv, Nq, Nk, d, 1.0f);
  if (st != FLASHBOB_OK) return st;
  BobArgs a{};
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.bf16 = in_dtype == FLASHBOB_BF16;
  a.passes = kPass1 | kPass2;
  // Per head group: pass 1 (d = 128: the JVP launch and the rows launch) and pass 2.
  *launches = tc_supported(a) ? (d == 128 ? 3 : 2) * tc_bob_streams(a) : 2;
  return FLASHBOB_OK;
}

flashbob_status flashbob_bob_tile_sizes(int d, flashbob_dtype in_dtype, int* Br1, int* Bc1,
                                        int* Br2, int* Bc2, size_t* smem_bytes_pass1,
                                        size_t* smem_bytes_pass2) {
  if (check_dtype(in_dtype) != FLASHBOB_OK) return FLASHBOB_ERR_INVALID_ARG;
  if (d <= 0 || d > 128) return FLASHBOB_ERR_UNSUPPORTED;
  BobArgs probe{};
  probe.d = d;
  probe.Nq = probe.Nk = 1;
  probe.bf16 = in_dtype == FLASHBOB_BF16;
  const bool tc = tc_supported(probe), wide = tc && d == 128;
  const int br1 = tc ? kTcRows : kSimtTile, bc1 = tc ? kTcStream : kSimtTile;
  const int bc2 = tc ? kTcRows : kSimtTile;
  const int br2 = wide ? kTcStream : tc ? kTcStream2 : kSimtTile;
  if (Br1) *Br1 = br1;
  if (Bc1) *Bc1 = bc1;
  if (Br2) *Br2 = br2;
  if (Bc2) *Bc2 = bc2;
  if (smem_bytes_pass1)
    *smem_bytes_pass1 = wide ? tc_pass1_d128_smem() : tc ? tc_pass1_smem() : simt_pass1_smem(d);
  if (smem_bytes_pass2)
    *smem_bytes_pass2 = wide ? tc_pass2_d128_smem() : tc ? tc_pass2_smem() : simt_pass2_smem(d);
  return FLASHBOB_OK;
}

flashbob_status flashbob_attention_jvp(const void* Q, const void* K, const void* V,
                                       const float* O, const float* L, const void* UQ,
                                       const void* UK, const void* UV, float tau, float* Od,
                                       float* Ld, int B, int H, int Hkv, int Nq, int Nk, int d,
                                       int causal, flashbob_dtype in_dtype, void* stream) {
  flashbob_status st = check_dtype(in_dtype);
  if (st != FLASHBOB_OK) return st;
  if (causal != 0 && causal != 1) return FLASHBOB_ERR_INVALID_ARG;
  const void* ptrs[] = {Q, K, V, O, L, UQ, UK, UV, Od, Ld};
  for (const void* p : ptrs)
    if (!p) return FLASHBOB_ERR_INVALID_ARG;
  st = check_sizes(B, H, Hkv, Nq, Nk, d, tau);
  if (st != FLASHBOB_OK) return st;
  for (const void* p : ptrs)
    if (!aligned16(p)) return FLASHBOB_ERR_MISALIGNED;
  const size_t rows = (size_t)B * H * Nq, krows = (size_t)B * Hkv * Nk;
  const size_t esz = in_dtype == FLASHBOB_BF16 ? 2 : 4;
  const Range ins[] = {{(uintptr_t)Q, (uintptr_t)Q + rows * d * esz},
                       {(uintptr_t)K, (uintptr_t)K + krows * d * esz},
                       {(uintptr_t)V, (uintptr_t)V + krows * d * esz},
                       {(uintptr_t)O, (uintptr_t)O + rows * d * 4},
                       {(uintptr_t)L, (uintptr_t)L + rows * 4},
                       {(uintptr_t)UQ, (uintptr_t)UQ + rows * d * esz},
                       {(uintptr_t)UK, (uintptr_t)UK + krows * d * esz},
                       {(uintptr_t)UV, (uintptr_t)UV + krows * d * esz}};
  const Range outs[] = {{(uintptr_t)Od, (uintptr_t)Od + rows * d * 4},
                        {(uintptr_t)Ld, (uintptr_t)Ld + rows * 4}};
  for (const Range& o : outs)
    for (const Range& i : ins)
      if (overlaps(o, i)) return FLASHBOB_ERR_INVALID_ARG;
  if (overlaps(outs[0], outs[1])) return FLASHBOB_ERR_INVALID_ARG;
  JvpArgs a{Q,  K,  V,  O,  L,   UQ,  UK, UV, tau, Od, Ld, B, H, Hkv, Nq, Nk, d, causal == 1,
            in_dtype == FLASHBOB_BF16, (cudaStream_t)stream, nullptr};
  if (error_word_ptr(&a.err) != cudaSuccess) return FLASHBOB_ERR_CUDA;
  const cudaError_t e = tc_jvp_supported(a) ? tc_jvp(a) : simt_jvp(a);
  return e == cudaSuccess ? FLASHBOB_OK : FLASHBOB_ERR_CUDA;
}

flashbob_status flashbob_check_wait_timeout(void* stream) {
  unsigned int* err = nullptr;
  if (error_word_ptr(&err) != cudaSuccess) return FLASHBOB_ERR_CUDA;
  return launch_wait_timeout((cudaStream_t)stream, err) == cudaSuccess ? FLASHBOB_OK
                                                                       : FLASHBOB_ERR_CUDA;
}

flashbob_status flashbob_mma_cycles(int n, int a_in_tmem, void* stream, double* cycles_per_mma) {
  if (cycles_per_mma == nullptr || n < 16 || n > 256 || n % 16 != 0)
    return FLASHBOB_ERR_INVALID_ARG;
  unsigned int* err = nullptr;
  if (error_word_ptr(&err) != cudaSuccess) return FLASHBOB_ERR_CUDA;
  return mma_cycles(n, a_in_tmem != 0, (cudaStream_t)stream, err, cycles_per_mma) == cudaSuccess
             ? FLASHBOB_OK
             : FLASHBOB_ERR_CUDA;
}

flashbob_status flashbob_last_device_error(void) {
  unsigned int* p = nullptr;
  if (error_word_ptr(&p) != cudaSuccess) return FLASHBOB_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return FLASHBOB_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v)) != cudaSuccess) return FLASHBOB_ERR_CUDA;
  if (v != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess)
      return FLASHBOB_ERR_CUDA;
    return FLASHBOB_ERR_TIMEOUT;
  }
  return FLASHBOB_OK;
}

}  // extern "C"
