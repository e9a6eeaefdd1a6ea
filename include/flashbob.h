/*
 * flashbob.h -- C ABI of libflashbob: exact backward-over-backward (BoB) of
 * softmax attention on one NVIDIA GB300 (sm_103a).
 *
 * Sources (web pages on the method; sections named as on the pages):
 *   [FBN] "FlashBoB: I/O-Efficient Exact Backward-over-Backward for Softmax
 *         Attention" (paper notes): 方法详解/整体框架 (the objective Phi and the
 *         four outputs), 关键设计 1 (row scalars alpha, E and the affine
 *         correction), 关键设计 2 (two-pass row/column schedule, no atomics).
 *   [FAB] "FlashAttention 的反向传播设计：在 SRAM 内部重计算 Softmax 的显存收益":
 *         section 一 (forward and first-backward formulas), section 二 (P is
 *         recomputed from saved row statistics).
 *
 * Notation, per (batch b, head h): Q, dO, U_Q are N_q x d and K, V, U_K,
 * U_V are N_k x d (N_q = N_k: self-attention; N_q != N_k: rectangular);
 * S = tau Q K^T, L_i = log sum_j exp(S_ij), P = exp(S - L), O = P V,
 * D_i = dO_i . O_i, dP = dO V^T, dS = P o (dP - D), dQ = tau dS K,
 * dK = tau dS^T Q, dV = P^T dO, and
 *     Phi = <dQ, U_Q> + <dK, U_K> + <dV, U_V>.
 * flashbob_bob returns the total derivatives d~Q, d~K, d~V, d~dO of Phi with
 * respect to Q, K, V and dO, plus the row scalars alpha_i = sum_j P_ij F_ij
 * (F = tau (U_Q K^T + Q U_K^T)) and E_i = sum_j P_ij d~P_ij.
 *
 * Layout: every matrix is a contiguous row-major array: the query-side
 * tensors Q, dO, U_Q, O, dQt, ddOt are [B, H, N_q, d], the key-side tensors
 * K, V, U_K, U_V, dKt, dVt are [B, Hkv, N_k, d]; every row vector (L, D,
 * alpha, E) is a contiguous [B, H, N_q] array.  Grouped-query attention
 * ([FBN] 关键设计 3): Hkv divides H; query head h uses key/value head
 * h / (H / Hkv), and d~K, d~V of a shared head sum its query heads.  Hkv = H
 * is ordinary multi-head attention, Hkv = 1 multi-query attention.
 * Causal mask: query i sees the keys j <= i (absolute positions, also for
 * N_q != N_k, so every query sees key 0; keys j >= N_q then get d~K = d~V =
 * 0).  Inputs are
 * either all fp32 or all bf16 (Q, K, V, dO, U_Q, U_K, U_V; selected by
 * in_dtype); O, L, D and every output are fp32.
 *
 * Ownership: the caller allocates and owns every buffer; all data pointers
 * are DEVICE pointers on the current CUDA device.  The library allocates no
 * device memory.  Its only device state is one error word per device,
 * written when a kernel's bounded wait gives up (see
 * flashbob_last_device_error).
 *
 * Calling convention: argument checks run on the host and return before any
 * launch; work is enqueued on `stream` (a cudaStream_t; NULL means the
 * legacy default stream) and the call returns without synchronising.  Two
 * calls on different streams must not share output buffers.
 *
 * Errors: a call that returns anything but FLASHBOB_OK has launched nothing
 * (FLASHBOB_ERR_CUDA: a launch failed; earlier launches of the same call may
 * have run).  Outputs may not overlap inputs or each other.
 */
#ifndef FLASHBOB_H
#define FLASHBOB_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FLASHBOB_OK = 0,
  FLASHBOB_ERR_INVALID_ARG = 1, /* null pointer, size <= 0, bad tau, overlap  */
  FLASHBOB_ERR_UNSUPPORTED = 2, /* d > 128, or sizes beyond the grid limits   */
  FLASHBOB_ERR_MISALIGNED = 3,  /* a pointer not 16-byte aligned              */
  FLASHBOB_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed       */
  FLASHBOB_ERR_TIMEOUT = 5      /* a kernel's bounded wait gave up            */
} flashbob_status;

typedef enum { FLASHBOB_F32 = 0, FLASHBOB_BF16 = 1 } flashbob_dtype;

/*
 * flashbob_prep: forward row state for the BoB ([FAB] sections 一/二,
 * [FBN] 关键设计 1 for D).
 *   in : Q, dO [B,H,Nq,d] and K, V [B,Hkv,Nk,d] of in_dtype
 *   out: O [B,H,Nq,d] fp32 (O = P V), L [B,H,Nq] fp32 (natural-log
 *        logsumexp of tau Q K^T per row), D [B,H,Nq] fp32 (D_i = dO_i . O_i)
 *   dO and D may both be NULL: the forward only (O and L, e.g. for
 *        flashbob_attention_jvp); exactly one of them NULL is rejected.
 *   tau: score scale, finite and > 0 (1/sqrt(d) in the pages).
 *   causal: 0 = full attention; 1 = query i sees keys j <= i only (the
 *        setting of [FBN] 实验关键数据); other values are rejected.
 *   Limits: 1 <= d <= 128; 1 <= Nq, Nk; B, H <= 65535 and B * H < 2^31
 *        (FLASHBOB_ERR_UNSUPPORTED beyond); 1 <= Hkv, H % Hkv == 0.
 *   One launch: bf16 inputs with d = 64 or d = 128 run a tcgen05 kernel,
 *   every other case fp32 CUDA cores.
 */
flashbob_status flashbob_prep(const void* Q, const void* K, const void* V, const void* dO,
                              float* O, float* L, float* D, int B, int H, int Hkv, int Nq,
                              int Nk, int d, float tau, int causal, flashbob_dtype in_dtype,
                              void* stream);

/*
 * flashbob_bob: exact BoB of softmax attention with the two-pass schedule of
 * [FBN] 关键设计 2; the closed form and affine correction of [FBN] 关键设计 1.
 *   in : Q, dO, U_Q [B,H,Nq,d] and K, V, U_K, U_V [B,Hkv,Nk,d] of in_dtype;
 *        O [B,H,Nq,d] fp32; L, D [B,H,Nq] fp32 (as written by flashbob_prep
 *        with the same causal flag); tau and causal as in prep.
 *   out: dQt, ddOt [B,H,Nq,d] and dKt, dVt [B,Hkv,Nk,d] fp32 (d~Q, d~dO,
 *        d~K, d~V); alpha, E [B,H,Nq] fp32.  Every element is written
 *        exactly once.
 *   Pass 1 (row-resident) writes d~Q, d~dO, alpha, E; pass 2 (column-
 *   resident) reads alpha, E and writes d~K, d~V.  No N x N tensor is ever
 *   written to device memory and no atomics are used.
 *   Limits: as flashbob_prep.  bf16 inputs with d = 64 or d = 128 run the
 *   tcgen05 tensor-core kernels; every other case runs the fp32 CUDA-core
 *   kernels.
 *   Streams: the work is ordered after everything already queued on
 *   `stream` and before everything queued on it afterwards.  On the
 *   tensor-core path, with B * Hkv >= 2 key/value heads and more than two
 *   waves of pass-1 CTAs, the heads are cut into up to four contiguous
 *   groups (when each group has at most 65535 query heads, the grid's
 *   extent) whose pass 1 -> pass 2 chains run on internal streams of the
 *   library, forked from and joined back into `stream` by events (pass 2 of
 *   a head reads only pass 1's alpha and E of that head's query rows); the
 *   results are those of the one-stream order, bit for bit.  Those streams
 *   are made once per device and kept; calls serialize their enqueueing on
 *   them.  A call made while `stream` is being captured into a CUDA graph
 *   stays on `stream` (two kernels, three at d = 128), so that no capture
 *   draws in the shared streams and absorbs other threads' calls.
 *   flashbob_bob_launches says how many kernels an uncaptured call launches.
 */
flashbob_status flashbob_bob(const void* Q, const void* K, const void* V, const float* O,
                             const void* dO, const float* L, const float* D, const void* UQ,
                             const void* UK, const void* UV, float tau, float* dQt, float* dKt,
                             float* dVt, float* ddOt, float* alpha, float* E, int B, int H,
                             int Hkv, int Nq, int Nk, int d, int causal, flashbob_dtype in_dtype,
                             void* stream);

/*
 * flashbob_bob_pass1 / flashbob_bob_pass2: the two passes of flashbob_bob,
 * callable one at a time ([FBN] 关键设计 2).  Same arguments, layouts and
 * limits as flashbob_bob.
 *   pass 1 (row-resident): reads Q, K, V, O, dO, L, D, U_Q, U_K, U_V and
 *     writes dQt, ddOt, alpha, E.
 *   pass 2 (column-resident): reads Q, K, V, dO, L, D, U_Q, U_K, U_V and the
 *     alpha, E written by pass 1, and writes dKt, dVt.
 * flashbob_bob(...) computes exactly pass 1 followed by pass 2 on the same
 * stream (it may run head groups on internal streams; see flashbob_bob).
 */
flashbob_status flashbob_bob_pass1(const void* Q, const void* K, const void* V, const float* O,
                                   const void* dO, const float* L, const float* D,
                                   const void* UQ, const void* UK, const void* UV, float tau,
                                   float* dQt, float* ddOt, float* alpha, float* E, int B, int H,
                                   int Hkv, int Nq, int Nk, int d, int causal,
                                   flashbob_dtype in_dtype, void* stream);

flashbob_status flashbob_bob_pass2(const void* Q, const void* K, const void* V, const void* dO,
                                   const float* L, const float* D, const float* alpha,
                                   const float* E, const void* UQ, const void* UK,
                                   const void* UV, float tau, float* dKt, float* dVt, int B,
                                   int H, int Hkv, int Nq, int Nk, int d, int causal,
                                   flashbob_dtype in_dtype, void* stream);

/*
 * flashbob_attention_jvp: forward-mode derivative of softmax attention
 * along the tangents (U_Q, U_K, U_V) of (Q, K, V):
 *     S' = tau (U_Q K^T + Q U_K^T)   (the matrix F of [FBN] 关键设计 1),
 *     L'_i = sum_j P_ij S'_ij,        O' = P o (S' - L') V + P U_V.
 *   L' and O' are the alpha and d~dO that flashbob_bob's pass 1 produces
 *   (neither depends on dO); this call is that pass without dO, so it runs
 *   5 of pass 1's 11 GEMMs.  No counterpart call is named on the pages; it
 *   is their pass 1 restricted to the terms without dO.
 *   in : Q, U_Q [B,H,Nq,d] and K, V, U_K, U_V [B,Hkv,Nk,d] of in_dtype;
 *        O [B,H,Nq,d], L [B,H,Nq] fp32 from flashbob_prep (dO = D = NULL
 *        there is enough); tau and causal as in prep.
 *   out: Od [B,H,Nq,d] fp32 (O'), Ld [B,H,Nq] fp32 (L').
 *   Limits, ownership and errors: as flashbob_bob.
 */
flashbob_status flashbob_attention_jvp(const void* Q, const void* K, const void* V,
                                       const float* O, const float* L, const void* UQ,
                                       const void* UK, const void* UV, float tau, float* Od,
                                       float* Ld, int B, int H, int Hkv, int Nq, int Nk, int d,
                                       int causal, flashbob_dtype in_dtype, void* stream);

/*
 * flashbob_bob_launches: how many kernel launches one flashbob_bob call with
 * these sizes makes on the current device: pass 1 and pass 2, where pass 1
 * of the tensor-core path at d = 128 is two launches (the JVP with alpha,
 * d~dO and E, then d~Q); that many per head group when the call runs head
 * groups on internal streams (a call outside any CUDA graph capture; a
 * captured call stays on its stream).  Checks the sizes as flashbob_bob
 * does; `launches` must not be NULL.
 */
flashbob_status flashbob_bob_launches(int B, int H, int Hkv, int Nq, int Nk, int d,
                                      flashbob_dtype in_dtype, int* launches);

/*
 * flashbob_bob_tile_sizes: the tiles flashbob_bob uses for (d, in_dtype):
 * pass-1 row block Br1 and column tile Bc1, pass-2 column block Bc2 and row
 * tile Br2, and each pass's dynamic shared memory per CTA in bytes (at
 * d = 128 on the tensor cores, of pass 1's second launch, the rows pass; its
 * first launch, the JVP, streams 64-row key tiles).  Any output pointer may
 * be NULL.  FLASHBOB_ERR_UNSUPPORTED for d outside 1..128.
 */
flashbob_status flashbob_bob_tile_sizes(int d, flashbob_dtype in_dtype, int* Br1, int* Bc1,
                                        int* Br2, int* Bc2, size_t* smem_bytes_pass1,
                                        size_t* smem_bytes_pass2);

/*
 * flashbob_last_device_error: FLASHBOB_ERR_TIMEOUT if a kernel of this
 * library on the current device gave up a bounded wait since the previous
 * call of this function, else FLASHBOB_OK (FLASHBOB_ERR_CUDA if the word
 * cannot be read).  Synchronises the current device, then clears the word.
 */
flashbob_status flashbob_last_device_error(void);

/*
 * flashbob_check_wait_timeout: a diagnostic of the bounded waits, with no
 * counterpart on the pages.  Launches one CTA on `stream` whose mbarrier
 * wait has nothing to wait for; after the wait limit (2 s) the kernel records
 * a timeout in the device error word and returns, so that the next
 * flashbob_last_device_error() reports FLASHBOB_ERR_TIMEOUT and the context
 * stays usable.  Returns FLASHBOB_ERR_CUDA if the launch fails.
 */
flashbob_status flashbob_check_wait_timeout(void* stream);

/*
 * flashbob_mma_cycles: a diagnostic of the tensor-core issue rate, with no
 * counterpart on the pages.  One CTA on `stream` issues 4096 tcgen05.mma of
 * one shape back to back from one thread (M = 128, N = n, K = 16, bf16
 * operands, fp32 accumulator in tensor memory; A from shared memory, or from
 * tensor memory when a_in_tmem != 0; B from shared memory) and times them
 * with the SM clock up to the completion of the last one.  Writes the SM
 * cycles per MMA to *cycles_per_mma (0 if the run's bounded wait gave up)
 * and synchronises `stream`.  The BoB kernels' schedules count their MMAs
 * in these units.
 *   n: 16 .. 256, a multiple of 16 (else FLASHBOB_ERR_INVALID_ARG, as for a
 *      NULL cycles_per_mma); FLASHBOB_ERR_CUDA if a CUDA call fails.
 */
flashbob_status flashbob_mma_cycles(int n, int a_in_tmem, void* stream, double* cycles_per_mma);

/* flashbob_status_string: a static, human-readable name of `s`. */
const char* flashbob_status_string(flashbob_status s);

#ifdef __cplusplus
}
#endif

#endif /* FLASHBOB_H */
