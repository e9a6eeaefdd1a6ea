// Host side of the tensor-core path: which calls it serves, the TMA tensor
// maps of the seven bf16 inputs, and the two launches on the caller's stream.
#include "internal.h"
#include "tc_common.cuh"

namespace flashbob {

cudaError_t tc_launch_pass1(const BobArgs& a, const CUtensorMap* maps128,
                            const CUtensorMap* maps32);
cudaError_t tc_launch_pass2(const BobArgs& a, const CUtensorMap* maps128,
                            const CUtensorMap* maps64);
cudaError_t tc_launch_jvp(const JvpArgs& a, const CUtensorMap* maps128,
                          const CUtensorMap* maps32);
cudaError_t tc_launch_pass1_d128(const BobArgs& a, const CUtensorMap* maps128,
                                 const CUtensorMap* maps32);
cudaError_t tc_launch_pass2_d128(const BobArgs& a, const CUtensorMap* maps128,
                                 const CUtensorMap* maps32);
cudaError_t tc_launch_jvp_d128(const JvpArgs& a, const CUtensorMap* maps128,
                               const CUtensorMap* maps32);

bool tc_supported(const BobArgs& a) { return a.bf16 && (a.d == 64 || a.d == 128); }

cudaError_t tc_group_split(int blocks, int group, int* S) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  *S = 1;
  for (int s = 2; s <= 8; ++s)
    if (group % s == 0 && blocks * s <= sms) *S = s;
  return cudaSuccess;
}

namespace {

// Head dim 128: both passes stream 32-row tiles against 128-row blocks.
cudaError_t tc_bob_d128(const BobArgs& a) {
  const int BH = a.B * a.H, BHkv = a.B * a.Hkv;
  cudaError_t e = cudaSuccess;
  if (a.passes & kPass1) {
    CUtensorMap m128[3], m32[4];
    const void* rows[3] = {a.Q, a.dO, a.UQ};
    const void* cols[4] = {a.K, a.V, a.UK, a.UV};
    for (int i = 0; i < 3 && e == cudaSuccess; ++i)
      e = tc::make_map_bf16(&m128[i], rows[i], BH, a.Nq, kTcRows, 128);
    for (int i = 0; i < 4 && e == cudaSuccess; ++i)
      e = tc::make_map_bf16(&m32[i], cols[i], BHkv, a.Nk, kTcStream, 128);
    if (e != cudaSuccess) return e;
    e = tc_launch_pass1_d128(a, m128, m32);
    if (e != cudaSuccess) return e;
  }
  if (a.passes & kPass2) {
    CUtensorMap m128[4], m32[3];
    const void* res[4] = {a.K, a.UK, a.V, a.UV};
    const void* str[3] = {a.Q, a.UQ, a.dO};
    for (int i = 0; i < 4 && e == cudaSuccess; ++i)
      e = tc::make_map_bf16(&m128[i], res[i], BHkv, a.Nk, kTcRows, 128);
    for (int i = 0; i < 3 && e == cudaSuccess; ++i)
      e = tc::make_map_bf16(&m32[i], str[i], BH, a.Nq, kTcStream, 128);
    if (e != cudaSuccess) return e;
    e = tc_launch_pass2_d128(a, m128, m32);
  }
  return e;
}

}  // namespace

cudaError_t tc_bob(const BobArgs& a) {
  if (a.d == 128) return tc_bob_d128(a);
  const int BH = a.B * a.H, BHkv = a.B * a.Hkv;
  cudaError_t e = cudaSuccess;
  if (a.passes & kPass1) {
    CUtensorMap m128[3], m32[4];
    const void* rows[3] = {a.Q, a.dO, a.UQ};
    const void* cols[4] = {a.K, a.V, a.UK, a.UV};
    for (int i = 0; i < 3 && e == cudaSuccess; ++i)
      e = tc::make_map_bf16_d64(&m128[i], rows[i], BH, a.Nq, kTcRows);
    for (int i = 0; i < 4 && e == cudaSuccess; ++i)
      e = tc::make_map_bf16_d64(&m32[i], cols[i], BHkv, a.Nk, kTcStream);
    if (e != cudaSuccess) return e;
    e = tc_launch_pass1(a, m128, m32);
    if (e != cudaSuccess) return e;
  }
  if (a.passes & kPass2) {
    CUtensorMap m128[4], m64[3];
    const void* res[4] = {a.K, a.UK, a.V, a.UV};
    const void* str[3] = {a.Q, a.UQ, a.dO};
    for (int i = 0; i < 4 && e == cudaSuccess; ++i)
      e = tc::make_map_bf16_d64(&m128[i], res[i], BHkv, a.Nk, kTcRows);
    for (int i = 0; i < 3 && e == cudaSuccess; ++i)
      e = tc::make_map_bf16_d64(&m64[i], str[i], BH, a.Nq, kTcStream2);
    if (e != cudaSuccess) return e;
    e = tc_launch_pass2(a, m128, m64);
  }
  return e;
}

bool tc_jvp_supported(const JvpArgs& a) { return a.bf16 && (a.d == 64 || a.d == 128); }

cudaError_t tc_jvp(const JvpArgs& a) {
  CUtensorMap m128[2], m32[4];
  const void* rows[2] = {a.Q, a.UQ};
  const void* cols[4] = {a.K, a.V, a.UK, a.UV};
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 2 && e == cudaSuccess; ++i)
    e = tc::make_map_bf16(&m128[i], rows[i], a.B * a.H, a.Nq, kTcRows, a.d);
  for (int i = 0; i < 4 && e == cudaSuccess; ++i)
    e = tc::make_map_bf16(&m32[i], cols[i], a.B * a.Hkv, a.Nk, kTcStream, a.d);
  if (e != cudaSuccess) return e;
  return a.d == 128 ? tc_launch_jvp_d128(a, m128, m32) : tc_launch_jvp(a, m128, m32);
}

}  // namespace flashbob
