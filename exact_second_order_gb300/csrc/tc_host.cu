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
                          const CUtensorMap* maps64);
cudaError_t tc_launch_pass1_d128(const BobArgs& a, const CUtensorMap* maps128,
                                 const CUtensorMap* maps32);
cudaError_t tc_launch_pass2_d128(const BobArgs& a, const CUtensorMap* maps128,
                                 const CUtensorMap* maps32);
cudaError_t tc_launch_jvp_d128(const JvpArgs& a, const CUtensorMap* maps128,
                               const CUtensorMap* maps64);
cudaError_t tc_launch_pass1_d128_jvp(const BobArgs& a, const CUtensorMap* maps128,
                                     const CUtensorMap* maps64);

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

namespace {

struct MapEntry {
  const void* base = nullptr;
  int BH = 0, N = 0, rows = 0, dh = 0;
  uint64_t used = 0;  // last use, for replacement
  CUtensorMap map;
};

std::mutex g_map_mu;
MapEntry g_maps[64];
uint64_t g_map_clock = 0;

struct SmemSet {
  const void* kernel = nullptr;
  int device = -1, bytes = 0;
};

std::mutex g_smem_mu;
SmemSet g_smem[64];

}  // namespace

cudaError_t tc_map_bf16(CUtensorMap* map, const void* base, int BH, int N, int rows, int dh) {
  std::lock_guard<std::mutex> lock(g_map_mu);
  MapEntry* victim = &g_maps[0];
  for (MapEntry& m : g_maps) {
    if (m.base == base && m.BH == BH && m.N == N && m.rows == rows && m.dh == dh &&
        base != nullptr) {
      m.used = ++g_map_clock;
      *map = m.map;
      return cudaSuccess;
    }
    if (m.used < victim->used) victim = &m;
  }
  const cudaError_t e = tc::make_map_bf16(map, base, BH, N, rows, dh);
  if (e != cudaSuccess) return e;
  victim->base = base;
  victim->BH = BH;
  victim->N = N;
  victim->rows = rows;
  victim->dh = dh;
  victim->used = ++g_map_clock;
  victim->map = *map;
  return cudaSuccess;
}

cudaError_t tc_set_smem(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_smem_mu);
  SmemSet* slot = nullptr;
  for (SmemSet& s : g_smem) {
    if (s.kernel == kernel && s.device == dev && s.bytes == bytes) return cudaSuccess;
    if (slot == nullptr && s.kernel == nullptr) slot = &s;
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && slot != nullptr) *slot = SmemSet{kernel, dev, bytes};
  return e;
}

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

// Head dim 128: pass 1 is the JVP launch (64-row key tiles) and the rows
// launch (32-row key tiles), pass 2 streams 32-row query tiles; every block
// holds 128 rows.
cudaError_t tc_bob_d128(const BobArgs& a) {
  const int BH = a.B * a.H, BHkv = a.B * a.Hkv;
  cudaError_t e = cudaSuccess;
  if (a.passes & kPass1) {
    CUtensorMap m128[3], m32[4], m64[4];
    const void* rows[3] = {a.Q, a.dO, a.UQ};
    const void* cols[4] = {a.K, a.V, a.UK, a.UV};
    for (int i = 0; i < 3 && e == cudaSuccess; ++i)
      e = tc_map_bf16(&m128[i], rows[i], BH, a.Nq, kTcRows, 128);
    for (int i = 0; i < 4 && e == cudaSuccess; ++i)
      e = tc_map_bf16(&m32[i], cols[i], BHkv, a.Nk, kTcStream, 128);
    for (int i = 0; i < 4 && e == cudaSuccess; ++i)
      e = tc_map_bf16(&m64[i], cols[i], BHkv, a.Nk, kTcJvpStream, 128);
    if (e != cudaSuccess) return e;
    const CUtensorMap mqu[2] = {m128[0], m128[2]};  // Q, U_Q
    e = tc_launch_pass1_d128_jvp(a, mqu, m64);      // alpha, d~dO and E
    if (e == cudaSuccess) e = tc_launch_pass1_d128(a, m128, m32);  // d~Q
    if (e != cudaSuccess) return e;
  }
  if (a.passes & kPass2) {
    CUtensorMap m128[4], m32[3];
    const void* res[4] = {a.K, a.UK, a.V, a.UV};
    const void* str[3] = {a.Q, a.UQ, a.dO};
    for (int i = 0; i < 4 && e == cudaSuccess; ++i)
      e = tc_map_bf16(&m128[i], res[i], BHkv, a.Nk, kTcRows, 128);
    for (int i = 0; i < 3 && e == cudaSuccess; ++i)
      e = tc_map_bf16(&m32[i], str[i], BH, a.Nq, kTcStream, 128);
    if (e != cudaSuccess) return e;
    e = tc_launch_pass2_d128(a, m128, m32);
  }
  return e;
}

}  // namespace

static cudaError_t tc_bob_d64(const BobArgs& a) {
  const int BH = a.B * a.H, BHkv = a.B * a.Hkv;
  cudaError_t e = cudaSuccess;
  if (a.passes & kPass1) {
    CUtensorMap m128[3], m32[4];
    const void* rows[3] = {a.Q, a.dO, a.UQ};
    const void* cols[4] = {a.K, a.V, a.UK, a.UV};
    for (int i = 0; i < 3 && e == cudaSuccess; ++i)
      e = tc_map_bf16(&m128[i], rows[i], BH, a.Nq, kTcRows, 64);
    for (int i = 0; i < 4 && e == cudaSuccess; ++i)
      e = tc_map_bf16(&m32[i], cols[i], BHkv, a.Nk, kTcStream, 64);
    if (e != cudaSuccess) return e;
    e = tc_launch_pass1(a, m128, m32);
    if (e != cudaSuccess) return e;
  }
  if (a.passes & kPass2) {
    CUtensorMap m128[4], m64[3];
    const void* res[4] = {a.K, a.UK, a.V, a.UV};
    const void* str[3] = {a.Q, a.UQ, a.dO};
    for (int i = 0; i < 4 && e == cudaSuccess; ++i)
      e = tc_map_bf16(&m128[i], res[i], BHkv, a.Nk, kTcRows, 64);
    for (int i = 0; i < 3 && e == cudaSuccess; ++i)
      e = tc_map_bf16(&m64[i], str[i], BH, a.Nq, kTcStream2, 64);
    if (e != cudaSuccess) return e;
    e = tc_launch_pass2(a, m128, m64);
  }
  return e;
}

namespace {

// Head-group streams.  Pass 2 of a key/value head needs pass 1 of that
// head's query rows only, so the two passes of disjoint head groups are
// independent.  A call with several groups and more than two waves of pass-1
// CTAs runs the groups' pass 1 -> pass 2 chains on up to kSplitStreams internal
// streams (forked from and joined back into the caller's stream): the SMs
// that one group's last pass-1 wave leaves idle take other groups' CTAs
// instead of waiting for the whole pass to drain.
constexpr int kSplitStreams = 4;

struct SplitStreams {
  int device = -1;
  cudaStream_t stream[kSplitStreams] = {};
  cudaEvent_t fork = nullptr;
  cudaEvent_t join[kSplitStreams] = {};
};

std::mutex g_split_mu;
SplitStreams g_split[16];

// The current device's streams and events, made on first use (g_split_mu
// held); null when every slot is taken by another device.
cudaError_t split_streams(SplitStreams** out) {
  *out = nullptr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  SplitStreams* slot = nullptr;
  for (SplitStreams& r : g_split) {
    if (r.device == dev) {
      *out = &r;
      return cudaSuccess;
    }
    if (slot == nullptr && r.device < 0) slot = &r;
  }
  if (slot == nullptr) return cudaSuccess;
  SplitStreams r;
  e = cudaEventCreateWithFlags(&r.fork, cudaEventDisableTiming);
  for (int k = 0; k < kSplitStreams && e == cudaSuccess; ++k) {
    e = cudaStreamCreateWithFlags(&r.stream[k], cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r.join[k], cudaEventDisableTiming);
  }
  if (e != cudaSuccess) {
    if (r.fork) cudaEventDestroy(r.fork);
    for (int k = 0; k < kSplitStreams; ++k) {
      if (r.stream[k]) cudaStreamDestroy(r.stream[k]);
      if (r.join[k]) cudaEventDestroy(r.join[k]);
    }
    return e;
  }
  r.device = dev;
  *slot = r;
  *out = slot;
  return cudaSuccess;
}

// The sub-problem of key/value heads [g0, g1) of the flattened B * Hkv heads
// (query heads [g0 G, g1 G) of the flattened B * H): contiguous slices of
// every tensor, one batch of H' = (g1 - g0) G query heads.
BobArgs head_slice(const BobArgs& a, int g0, int g1) {
  const int G = a.H / a.Hkv;
  const size_t d = static_cast<size_t>(a.d);
  const size_t qr = static_cast<size_t>(g0) * G * a.Nq;  // first query row
  const size_t kr = static_cast<size_t>(g0) * a.Nk;      // first key row
  auto bf = [](const void* p, size_t elems) {
    return static_cast<const void*>(static_cast<const char*>(p) + 2 * elems);
  };
  BobArgs s = a;
  // The groups run side by side and fill the GPU together: no group's pass 2
  // splits its key blocks across clusters (which would also change the
  // order of its column sums).
  s.whole_grid_only = true;
  s.Q = bf(a.Q, qr * d);
  s.dO = bf(a.dO, qr * d);
  s.UQ = bf(a.UQ, qr * d);
  s.K = bf(a.K, kr * d);
  s.V = bf(a.V, kr * d);
  s.UK = bf(a.UK, kr * d);
  s.UV = bf(a.UV, kr * d);
  s.O = a.O + qr * d;
  s.L = a.L + qr;
  s.D = a.D + qr;
  s.dQt = a.dQt + qr * d;
  s.ddOt = a.ddOt + qr * d;
  s.alpha = a.alpha + qr;
  s.E = a.E + qr;
  s.dKt = a.dKt + kr * d;
  s.dVt = a.dVt + kr * d;
  s.B = 1;
  s.Hkv = g1 - g0;
  s.H = (g1 - g0) * G;
  return s;
}

cudaError_t tc_bob_one(const BobArgs& a) { return a.d == 128 ? tc_bob_d128(a) : tc_bob_d64(a); }

}  // namespace

int tc_bob_streams(const BobArgs& a) {
  const long long groups = static_cast<long long>(a.B) * a.Hkv;
  int dev = 0, sms = 0;
  if (a.passes != (kPass1 | kPass2) || groups < 2 || cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      static_cast<long long>(a.B) * a.H * ((a.Nq + kTcRows - 1) / kTcRows) <= 2LL * sms)
    return 1;
  const int ns = groups < kSplitStreams ? static_cast<int>(groups) : kSplitStreams;
  // A slice launches its (at most ceil(groups / ns)) * G query heads along
  // the grid's y extent: a call whose slices would not fit stays whole.
  if ((groups + ns - 1) / ns * (a.H / a.Hkv) > kMaxGridY) return 1;
  // A call captured into a CUDA graph stays on the capturing stream: the
  // internal streams are shared by every call on the device, and once a
  // capture has drawn them in it keeps them until it ends, so another
  // thread's direct call would launch into that capture instead of running.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(a.stream, &cs) != cudaSuccess) {
    (void)cudaGetLastError();
    return 1;
  }
  return cs == cudaStreamCaptureStatusNone ? ns : 1;
}

cudaError_t tc_bob(const BobArgs& a) {
  const long long groups = static_cast<long long>(a.B) * a.Hkv;
  const int ns = tc_bob_streams(a);
  if (ns == 1) return tc_bob_one(a);
  std::lock_guard<std::mutex> lock(g_split_mu);
  SplitStreams* ss = nullptr;
  cudaError_t e = split_streams(&ss);
  if (e != cudaSuccess) return e;
  if (ss == nullptr) return tc_bob_one(a);
  e = cudaEventRecord(ss->fork, a.stream);
  if (e != cudaSuccess) return e;
  for (int k = 0; k < ns && e == cudaSuccess; ++k) e = cudaStreamWaitEvent(ss->stream[k], ss->fork, 0);
  if (e != cudaSuccess) return e;
  cudaError_t first = cudaSuccess;
  for (int k = 0; k < ns; ++k) {
    BobArgs s = head_slice(a, static_cast<int>(groups * k / ns),
                           static_cast<int>(groups * (k + 1) / ns));
    s.stream = ss->stream[k];
    const cudaError_t ek = tc_bob_one(s);
    if (first == cudaSuccess) first = ek;
  }
  // Join every stream back, whatever happened above.
  for (int k = 0; k < ns; ++k) {
    e = cudaEventRecord(ss->join[k], ss->stream[k]);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(a.stream, ss->join[k], 0);
    if (first == cudaSuccess) first = e;
  }
  return first;
}

bool tc_jvp_supported(const JvpArgs& a) { return a.bf16 && (a.d == 64 || a.d == 128); }

cudaError_t tc_jvp(const JvpArgs& a) {
  const int key_rows = kTcJvpStream;  // both JVP kernels stream 64-row key tiles
  CUtensorMap m128[2], mk[4];
  const void* rows[2] = {a.Q, a.UQ};
  const void* cols[4] = {a.K, a.V, a.UK, a.UV};
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 2 && e == cudaSuccess; ++i)
    e = tc_map_bf16(&m128[i], rows[i], a.B * a.H, a.Nq, kTcRows, a.d);
  for (int i = 0; i < 4 && e == cudaSuccess; ++i)
    e = tc_map_bf16(&mk[i], cols[i], a.B * a.Hkv, a.Nk, key_rows, a.d);
  if (e != cudaSuccess) return e;
  return a.d == 128 ? tc_launch_jvp_d128(a, m128, mk) : tc_launch_jvp(a, m128, mk);
}

}  // namespace flashbob
