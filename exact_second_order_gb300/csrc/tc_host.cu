// Host side of the tensor-core path: which calls it serves, the TMA tensor
// maps of the seven bf16 inputs, and the two launches on the caller's stream.
#include <mutex>

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

namespace {

// How many clusters of S CTAs of `kernel` (1 CTA per SM at this shared-memory
// size) the current device holds at once, for S = 1 .. 8; asked once per
// (kernel, device) and kept.
struct ClusterFit {
  const void* kernel = nullptr;
  int device = -1;
  int fit[9] = {};
};

cudaError_t cluster_fit(const void* kernel, size_t smem, int S, int* out) {
  static std::mutex mu;
  static ClusterFit table[16];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  ClusterFit* slot = nullptr;
  for (ClusterFit& c : table) {
    if (c.kernel == kernel && c.device == dev) { *out = c.fit[S]; return cudaSuccess; }
    if (slot == nullptr && c.kernel == nullptr) slot = &c;
  }
  ClusterFit c;
  c.kernel = kernel;
  c.device = dev;
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  c.fit[1] = sms;
  for (int s = 2; s <= 8; ++s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, s, 1);
    cfg.blockDim = dim3(320);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = s;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    if (e != cudaSuccess) return e;
    c.fit[s] = n;
  }
  if (slot != nullptr) *slot = c;
  *out = c.fit[S];
  return cudaSuccess;
}

}  // namespace

cudaError_t tc_pass2_split(const void* split_kernel, size_t smem, int blocks, int tiles,
                           int* S) {
  // Split only grids that leave SMs idle: the largest S whose clusters still
  // all fit at once.  Splitting a grid of a wave or more to even out its
  // last wave was measured slower (the long-context pass 2 12.76 -> 13.43 ms
  // at S = 2): cluster launches then wait for pairs of free SMs.
  *S = 1;
  int sms = 0;
  cudaError_t e = cluster_fit(split_kernel, smem, 1, &sms);
  if (e != cudaSuccess || blocks >= sms) return e;
  for (int s = 2; s <= 8 && s <= tiles; ++s) {
    int fit = 0;
    e = cluster_fit(split_kernel, smem, s, &fit);
    if (e != cudaSuccess) return e;
    if (blocks <= fit) *S = s;
  }
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
