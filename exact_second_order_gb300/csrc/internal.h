// Internal interface between the C ABI (flashbob_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace flashbob {

struct PrepArgs {
  const void *Q, *K, *V, *dO;
  float *O, *L, *D;
  int B, H, Hkv;  // Hkv key/value heads, shared by H / Hkv query heads each
  int Nq, Nk, d;  // query rows, key rows, head dim
  float tau;
  bool causal;
  bool bf16;
  cudaStream_t stream;
  unsigned int* err;  // device error word of the current device
};

struct BobArgs {
  const void *Q, *K, *V;
  const float* O;
  const void* dO;
  const float *L, *D;
  const void *UQ, *UK, *UV;
  float tau;
  float *dQt, *dKt, *dVt, *ddOt, *alpha, *E;
  int B, H, Hkv;  // Hkv key/value heads, shared by H / Hkv query heads each
  int Nq, Nk, d;  // query rows, key rows, head dim
  bool causal;
  bool bf16;
  cudaStream_t stream;
  unsigned int* err;  // device error word of the current device
  int passes;         // bit 0: pass 1, bit 1: pass 2
  bool whole_grid_only = false;  // pass 2: never split a key block across a cluster
};

// Attention JVP (forward-mode derivative along U_Q, U_K, U_V).
struct JvpArgs {
  const void *Q, *K, *V;
  const float *O, *L;
  const void *UQ, *UK, *UV;
  float tau;
  float *Od, *Ld;
  int B, H, Hkv;
  int Nq, Nk, d;
  bool causal;
  bool bf16;
  cudaStream_t stream;
  unsigned int* err;
};

// Largest grid y and z extents: the kernels launch heads along y and
// batches along z.
constexpr int kMaxGridY = 65535;

constexpr int kPass1 = 1;
constexpr int kPass2 = 2;

// fp32 CUDA-core kernels (any 1 <= d <= 128; fp32 or bf16 inputs).
constexpr int kSimtTile = 32;
cudaError_t simt_prep(const PrepArgs& a);
cudaError_t simt_bob(const BobArgs& a);
cudaError_t simt_jvp(const JvpArgs& a);
size_t simt_pass1_smem(int d);
size_t simt_pass2_smem(int d);

// tcgen05 tensor-core kernels (bf16 inputs, d = 64 and d = 128).
constexpr int kTcRows = 128;    // rows of the resident block (MMA M) in both passes
constexpr int kTcStream = 32;   // rows of a streamed key tile in pass 1 (and of a d = 128 pass-2 query tile)
constexpr int kTcStream2 = 64;  // rows of a streamed query tile in pass 2
constexpr int kTcJvpStream = 64;  // rows of a streamed key tile in the d = 64 JVP
bool tc_supported(const BobArgs& a);
bool tc_prep_supported(const PrepArgs& a);
cudaError_t tc_prep(const PrepArgs& a);
cudaError_t tc_bob(const BobArgs& a);
// Streams tc_bob runs a call on: 1 (the caller's), or up to 4 internal
// streams, one per slice of the key/value heads, when both passes are asked
// for, there are several head groups, a pass has more than two waves of
// CTAs (the groups' pass 1 -> pass 2 chains then overlap each other's tails),
// every slice's query heads fit the grid's y extent and the caller's stream
// is not being captured into a CUDA graph.
int tc_bob_streams(const BobArgs& a);
bool tc_jvp_supported(const JvpArgs& a);
cudaError_t tc_jvp(const JvpArgs& a);
size_t tc_pass1_smem();
size_t tc_pass2_smem();
size_t tc_pass1_d128_smem();
size_t tc_pass2_d128_smem();
// Tensor map of a bf16 [BH, N, dh] tensor with 128-byte-swizzled boxes of
// `rows` x 64 elements (tc::make_map_bf16), kept in a small per-process
// cache keyed by every encoding argument: a map is a pure function of them,
// so repeated calls on the same buffers skip the driver's encoder.
cudaError_t tc_map_bf16(CUtensorMap* map, const void* base, int BH, int N, int rows, int dh);
// cudaFuncSetAttribute(kernel, MaxDynamicSharedMemorySize, bytes), once per
// (kernel, device, bytes).
cudaError_t tc_set_smem(const void* kernel, int bytes);
// Pass 2 cluster split: how many CTAs (S = 1 .. 8) share a key block of
// `tiles` streamed query tiles when the `blocks` key blocks cannot fill the
// device: the largest S whose clusters of the split kernel all fit at once.
cudaError_t tc_pass2_split(const void* split_kernel, size_t smem, int blocks, int tiles,
                           int* S);

// Device error word (one per device): a kernel writes a nonzero code when a
// bounded wait gives up.  Codes: 1 = mbarrier wait timed out.
cudaError_t error_word_ptr(unsigned int** ptr);
// One CTA whose bounded wait runs out (the timeout report, tested on a GPU).
cudaError_t launch_wait_timeout(cudaStream_t stream, unsigned int* err);
// Cycles per tcgen05.mma (M = 128, N = n, K = 16, bf16) issued back to back
// by one thread of one CTA, A from shared memory or tensor memory; waits for
// the result (0 cycles when the run's bounded wait gave up).
cudaError_t mma_cycles(int n, bool a_in_tmem, cudaStream_t stream, unsigned int* err,
                       double* cycles_per_mma);

}  // namespace flashbob
