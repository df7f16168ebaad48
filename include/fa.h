/*
 * fa.h -- C ABI of exact attention on sm_103a (GB300): the forward pass
 * (fa_fwd; grouped K/V heads fa_fwd_gqa; split-K fa_fwd_splitkv and
 * fa_fwd_splitkv_noalloc; queries against a longer key sequence, as in
 * decoding, fa_fwd_kv; E4M3 inputs fa_fwd_fp8), the backward pass (fa_bwd,
 * fa_bwd_gqa), the same passes on page-locked host tensors (fa_fwd_host,
 * fa_fwd_fp8_host, fa_bwd_host), and the status calls.
 *
 * The operation ("CUDA FlashAttention: from online softmax to the
 * long-sequence IO limit", sections 1 and 4; "Why FlashAttention does not
 * need to store the attention matrix", sections 3.2 and 4.1):
 *
 *     O   = softmax(scale * Q K^T + M) V
 *     LSE = log(sum_j exp(scale * q_i . k_j + M_ij))          (natural log)
 *
 * with M_ij = -inf for j > i when `causal` is 1 and M = 0 otherwise.  The
 * N x N score and probability matrices never reach device memory: each
 * 128-row query block keeps an FP32 running max m, running sum l and an
 * unnormalised output across the key/value blocks, rescaled by
 * exp(m_old - m_new), and writes O = O / l plus LSE = m + log(l) at the end.
 *
 * Layout: Q, K, V and O are [B, H, N, D] row-major and contiguous, all of the
 * same 16-bit type; LSE is [B, H, N] fp32.  Every pointer passed to fa_fwd is
 * a DEVICE pointer owned by the caller; the library allocates nothing per
 * call and keeps no pointer after it returns.  O and LSE must not overlap Q,
 * K or V (or each other).
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <cuda_runtime.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { FA_FP16 = 0, FA_BF16 = 1 } fa_dtype;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,   /* bad size, flag, scale, or overlapping outputs  */
    FA_ERR_UNSUPPORTED = 2,   /* head dimension other than 64 or 128           */
    FA_ERR_MISALIGNED = 3,    /* null pointer or not 16-byte aligned           */
    FA_ERR_CUDA = 4,          /* a CUDA runtime or driver call failed          */
    FA_ERR_TIMEOUT = 5,       /* a bounded in-kernel wait gave up (see below)  */
    FA_ERR_TOO_LARGE = 6      /* the problem does not fit the fixed scratch of
                                 fa_fwd_splitkv_noalloc                        */
} fa_status;

/*
 * fa_fwd -- launch the forward pass on `stream`; returns without waiting.
 *
 *   q, k, v    [B,H,N,D] input, type `dtype`                (device, read)
 *   o          [B,H,N,D] output, type `dtype`                (device, written)
 *   lse        [B,H,N] fp32 natural-log log-sum-exp          (device, written)
 *   B, H, N    batch, heads, sequence length; each >= 1, B*H*N*D < 2^40
 *   D          head dimension: 64 or 128, else FA_ERR_UNSUPPORTED
 *   scale      softmax scale applied to Q K^T (usually 1/sqrt(D)); finite, > 0
 *   causal     0: no mask; 1: the square lower-triangular mask (key j <= query i)
 *   dtype      FA_FP16 or FA_BF16
 *   stream     CUDA stream (0 = legacy default stream)
 *
 * Returns FA_OK once the kernel is queued.  Argument errors are reported
 * before anything is launched and leave o / lse untouched.  N need not be a
 * multiple of any tile size.  Results are deterministic for fixed inputs (and
 * device): a launch with no more 256-row work tiles (ceil(N / 256) * B * H)
 * than the device has SMs splits each 128-row query tile's keys between two
 * partial softmax passes merged on chip, so its last bits can differ from the
 * same rows computed inside a larger launch.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int N, int D, float scale, int causal, int dtype,
           cudaStream_t stream);

/*
 * fa_fwd_gqa -- the forward pass with grouped key/value heads (GQA; MQA when
 * H_kv = 1): query head h of batch entry b reads K/V head h / (H / H_kv) of
 * the same batch entry, without K/V being copied ("CUDA FlashAttention: from
 * online softmax to the long-sequence IO limit", section 7, GQA/MQA).
 *
 *   q, o        [B, H, N, D]     (as for fa_fwd)
 *   k, v        [B, H_kv, N, D]  (H_kv >= 1 and H a multiple of H_kv)
 *   lse         [B, H, N] fp32
 *
 * Work tiles of query heads that share a K/V head run next to each other, so
 * that K/V head is read from HBM about once and then from L2.  All other
 * arguments, layouts and errors are those of fa_fwd; an H_kv that does not
 * divide H returns FA_ERR_INVALID_ARG.  fa_fwd is fa_fwd_gqa with H_kv = H.
 */
int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
               int B, int H, int H_kv, int N, int D, float scale, int causal, int dtype,
               cudaStream_t stream);

/*
 * fa_splitkv_workspace_bytes -- bytes of workspace fa_fwd_splitkv needs for
 * these sizes: num_splits * B*H*N * (4*D + 16).  Returns 0 for invalid sizes
 * (any size < 1, D not 64 or 128, num_splits > 64).
 */
size_t fa_splitkv_workspace_bytes(int B, int H, int N, int D, int num_splits);

/*
 * fa_fwd_splitkv -- the same forward pass, with the key/value range of each
 * 256-row query block cut into `num_splits` contiguous chunks that different
 * CTAs process ("CUDA FlashAttention: from online softmax to the long-sequence
 * IO limit", section 7: for long N and small B*H, split along the keys, let
 * each worker produce a local (m, l, o) and reduce them with the same merge
 * formula).  Each chunk writes its unnormalised partial O (fp32) and its
 * running max and sums to `workspace`; a second kernel, queued on the same
 * stream, merges them into o and lse.
 *
 *   num_splits  1 .. 64 (1 still goes through the workspace and the merge)
 *   workspace   DEVICE memory owned by the caller, 16-byte aligned, at least
 *               fa_splitkv_workspace_bytes(B, H, N, D, num_splits) bytes;
 *               overwritten, contents undefined afterwards; must not overlap
 *               q, k, v, o or lse
 *
 * All other arguments, layouts and errors are those of fa_fwd; a workspace
 * that is too small returns FA_ERR_INVALID_ARG, a null or misaligned one
 * FA_ERR_MISALIGNED.  Calls that share a workspace must not overlap in time.
 */
int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int N, int D, float scale, int causal, int dtype,
                   int num_splits, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream);

/*
 * fa_fwd_splitkv_noalloc -- fa_fwd_splitkv for callers that cannot allocate
 * device memory.  The pages have no counterpart: this entry point exists for
 * the library's users, not for the method.
 *
 * Who needs it: code that may not call cudaMalloc / cudaFree around this call,
 * e.g. a host framework that owns every device allocation and passes the
 * library only its tensors, or a latency-critical loop where an allocation,
 * which can synchronise the whole device, is not acceptable.  Instead of a
 * caller-provided workspace it uses a scratch buffer of
 * fa_noalloc_scratch_bytes() bytes (64 MiB) held in the library's own device
 * memory; every GPU that loads the library keeps that buffer until the process
 * exits.  The caller still provides q, k, v, o and lse, as for fa_fwd.
 *
 * Limits and behaviour:
 *   - returns FA_ERR_TOO_LARGE, without launching anything, when
 *     fa_splitkv_workspace_bytes(B, H, N, D, num_splits) exceeds the scratch
 *     size (use fewer splits, or fa_fwd_splitkv with your own workspace);
 *   - no allocation of any kind is made: the first call on a device looks up
 *     the buffer's device address (once per device, with that device current)
 *     and caches it with the id of the device's CUDA context; make that first
 *     call before any stream capture on that device.  A context re-created
 *     later (after cudaDeviceReset) may hold the buffer at another address, so
 *     the first call in the new context looks it up again: that call, too,
 *     belongs before any stream capture;
 *   - arguments are checked as fa_fwd_splitkv checks them, before any CUDA
 *     call is made;
 *   - all calls on a device share the one buffer; calls that may overlap on
 *     the GPU (different streams without ordering between them) race and give
 *     wrong results.  Nothing needs clearing between calls: each call writes
 *     every part of the buffer it later reads;
 *   - all other arguments, layouts and status codes are those of
 *     fa_fwd_splitkv.
 */
int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int N, int D, float scale, int causal, int dtype,
                           int num_splits, cudaStream_t stream);

/* Size in bytes of the scratch buffer fa_fwd_splitkv_noalloc uses. */
size_t fa_noalloc_scratch_bytes(void);

/*
 * fa_fwd_kv -- Nq queries per head against a key/value sequence of Nk >= Nq
 * tokens, e.g. decode (Nq = 1) or a prefill chunk against a K/V cache
 * ("CUDA FlashAttention: from online softmax to the long-sequence IO limit",
 * section 7: split-KV / flash-decoding for long K/V and small B*H, GQA/MQA).
 *
 *   q, o        [B, H, Nq, D]                                   (as for fa_fwd)
 *   k, v        [B, H_kv, Nk, D] (H a multiple of H_kv)
 *   lse         [B, H, Nq] fp32
 *   causal      query i is the token at position i + Nk - Nq: with causal = 1
 *               it sees keys j <= i + Nk - Nq (the mask of fa_fwd when Nq = Nk;
 *               a single query sees every key); requires Nq <= Nk
 *   num_splits  0: one pass; 1..64: each query block's key range is cut into
 *               num_splits chunks processed by different CTAs and merged by a
 *               second kernel, through `workspace` (as for fa_fwd_splitkv,
 *               at least fa_fwd_kv_workspace_bytes(B, H, Nq, D, num_splits)
 *               bytes; ignored and may be NULL when num_splits = 0)
 *
 * When Nq < 128 and H_kv < H, the query heads that share a K/V head are
 * processed as one block of (H / H_kv) * Nq rows, so each K/V head is read
 * once per split.  Other arguments, layouts and errors as for fa_fwd_splitkv.
 */
size_t fa_fwd_kv_workspace_bytes(int B, int H, int Nq, int D, int num_splits);

/*
 * fa_fwd_kv_splits_hint -- a num_splits for fa_fwd_kv on the current device:
 * 0 when the unsplit grid of work tiles already covers the SMs, else enough
 * chunks per query block to cover them once (twice for causal problems of
 * several 256-row query blocks, whose blocks differ in work), each chunk at
 * least 4 key/value tiles, at most 64.  A host-side rule of thumb, not a
 * measurement.  Returns -1 for invalid sizes (as for fa_fwd_kv) or if the
 * device cannot be queried.
 */
int fa_fwd_kv_splits_hint(int B, int H, int H_kv, int Nq, int Nk, int D, int causal);
int fa_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int Nq,
              int Nk, int D, float scale, int causal, int dtype, int num_splits, void* workspace,
              size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_fwd_fp8 -- the forward pass on 8-bit inputs ("CUDA FlashAttention: from
 * online softmax to the long-sequence IO limit", section 2: FP8 Q/K/V need a
 * per-tensor or per-block scale, and the softmax state stays FP32).
 *
 *   q, k       [B,H,N,D] OCP E4M3 bytes                         (device, read)
 *   v_t        V transposed per head: [B,H,D,N] E4M3 bytes, keys contiguous
 *              (both operands of the FP8 tensor-core product P V are read
 *              K-major)                                          (device, read)
 *   q_scale, k_scale, v_scale
 *              [B,H,ceil(N/128)] fp32 dequantization scales: element x of
 *              rows (keys) 128*b .. 128*b+127 of head (b, h) stands for
 *              E4M3(x) * scale[b, h, block]; positive and finite  (device, read)
 *   o          [B,H,N,D] bf16 output                              (device, written)
 *   lse        [B,H,N] fp32 natural-log LSE of the dequantized scores (device, written)
 *   B, H, N, scale, causal, stream   as for fa_fwd; D must be 128
 *              (else FA_ERR_UNSUPPORTED) and N a multiple of 16 (else
 *              FA_ERR_INVALID_ARG: the rows of v_t are N bytes long and the
 *              tensor-copy engine needs 16-byte strides)
 *
 * S = Q K^T runs on 8-bit operands with FP32 accumulation and is scaled by the
 * two block scales; the running max, the sums and O stay FP32.  P enters the
 * FP8 product P V as E4M3, carrying a power-of-two range shift and the ratio of
 * its V block's scale to the head's largest V block scale; O is normalised by
 * the sum of those E4M3 P values (an exact convex combination of dequantized V
 * rows), the LSE uses the unrounded sum.  Errors and codes as for fa_fwd.
 */
int fa_fwd_fp8(const void* q, const void* k, const void* v_t, const float* q_scale, const float* k_scale,
               const float* v_scale, void* o, float* lse, int B, int H, int N, int D, float scale, int causal,
               cudaStream_t stream);

/*
 * fa_fwd_host_workspace_bytes -- bytes of device workspace fa_fwd_host needs:
 * room for Q, K, V, O (2*B*H*N*D bytes each) and the LSE (4*B*H*N), each
 * rounded up to 256 bytes.  Returns 0 for invalid sizes (any size < 1, D not
 * 64 or 128, B*H*N*D >= 2^40).
 */
size_t fa_fwd_host_workspace_bytes(int B, int H, int N, int D);

/*
 * fa_fwd_host -- fa_fwd on tensors held in host memory.  The pages have no
 * counterpart: this is the library's entry point for callers whose data is
 * not on the GPU.  It queues, in chunks of whole (b, h) planes, the copy of
 * Q, K, V to the device, the forward pass of fa_fwd on each chunk as soon as
 * its inputs have landed, and the copy of O and LSE back, on two copy streams
 * of the library's own (created once per device) and on `stream`, so that the
 * copies in both directions overlap the kernel.  Results are bit-identical to
 * fa_fwd on the same inputs.
 *
 *   q, k, v     [B,H,N,D], type `dtype`   (PAGE-LOCKED host memory, read)
 *   o           [B,H,N,D], type `dtype`   (page-locked host memory, written)
 *   lse         [B,H,N] fp32               (page-locked host memory, written)
 *   B, H, N, D, scale, causal, dtype      as for fa_fwd
 *   workspace   DEVICE memory owned by the caller, 256-byte aligned, at least
 *               fa_fwd_host_workspace_bytes(B, H, N, D) bytes; overwritten
 *   stream      CUDA stream: the call is ordered after the work already queued
 *               on it, and work queued on it afterwards starts after O and LSE
 *               are back in host memory; returns without waiting
 *
 * Returns FA_OK once everything is queued; synchronise `stream` before
 * reading o or lse.  If a CUDA call fails part-way (FA_ERR_CUDA), the copies
 * already queued still finish before later work on `stream` starts.
 * Pageable or managed host memory, a workspace that is not device memory or
 * is too small, and outputs that overlap inputs give FA_ERR_INVALID_ARG
 * before anything is queued; other argument rules and codes
 * are those of fa_fwd.  Calls from several host threads are serialised while
 * they queue work; calls that may run at the same time on the GPU must not
 * share a workspace.
 */
int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                int B, int H, int N, int D, float scale, int causal, int dtype,
                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_bwd_workspace_bytes -- bytes of workspace fa_bwd needs for these sizes:
 * an fp32 dQ accumulator (4*B*H*N*D bytes) and one fp32 value per query row
 * (4*B*H*N), each rounded up to 256 bytes.  Returns 0 for invalid sizes (any
 * size < 1, D not 64 or 128).
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int D);

/*
 * fa_bwd -- the backward pass ("Why FlashAttention does not need to store the
 * attention matrix", section 3.3; "CUDA FlashAttention: from online softmax to
 * the long-sequence IO limit", sections 4.3.1-4.3.2): given the upstream
 * gradient dO = dL/dO of the forward pass O = softmax(scale*Q K^T + M) V, it
 * rebuilds P from the forward's LSE tile by tile (no N x N matrix is stored)
 * and computes
 *     dV = P^T dO,   dP = dO V^T,   dS = P (x) (dP - Delta),
 *     dQ = scale * dS K,   dK = scale * dS^T Q,
 * with Delta_i = rowsum(dP_i (x) P_i), evaluated as dO_i . O_i from the
 * forward's output O (the two are equal because every row of P sums to 1).
 *
 *   q, k, v     [B,H,N,D] inputs of the forward pass, type `dtype` (device, read)
 *   o           [B,H,N,D] the forward's output O                  (device, read)
 *   dout        [B,H,N,D] dO, type `dtype`                        (device, read)
 *   lse         [B,H,N] fp32, the forward's natural-log LSE       (device, read)
 *   dq, dk, dv  [B,H,N,D] gradients, type `dtype`                 (device, written)
 *   workspace   DEVICE memory owned by the caller, 16-byte aligned, at least
 *               fa_bwd_workspace_bytes(B, H, N, D) bytes; overwritten (dQ is
 *               accumulated there in fp32 before it is rounded into dq)
 *   B, H, N, D, scale, causal, dtype, stream   as for fa_fwd; scale and causal
 *               must be the values the forward pass used
 *
 * Returns FA_OK once the three kernels are queued on `stream`.  Argument
 * errors are reported before anything is launched: FA_ERR_MISALIGNED for a
 * null or misaligned pointer, FA_ERR_UNSUPPORTED for D other than 64 or 128,
 * FA_ERR_INVALID_ARG for bad sizes, a small workspace, or outputs (dq, dk, dv,
 * workspace) that overlap the inputs or each other.  dQ is summed with fp32
 * atomic additions, so its last bits may differ between runs; dK and dV are
 * deterministic.  Calls that share a workspace must not overlap in time.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
           void* dq, void* dk, void* dv, int B, int H, int N, int D, float scale, int causal, int dtype,
           void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_bwd_gqa -- fa_bwd with grouped key/value heads (the backward pass of
 * fa_fwd_gqa): q, o, dout, dq are [B,H,N,D] and lse [B,H,N]; k, v, dk, dv are
 * [B,H_kv,N,D], H a multiple of H_kv, query head h reading K/V head
 * h / (H / H_kv).  dK and dV of a K/V head sum the contributions of all the
 * query heads of its group (accumulated in fp32 before the one rounding).
 * Workspace as for fa_bwd: fa_bwd_workspace_bytes(B, H, N, D).  An H_kv that
 * does not divide H returns FA_ERR_INVALID_ARG.  fa_bwd is fa_bwd_gqa with
 * H_kv = H.
 */
int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
               void* dq, void* dk, void* dv, int B, int H, int H_kv, int N, int D, float scale, int causal,
               int dtype, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_fwd_fp8_host_workspace_bytes -- bytes of device workspace fa_fwd_fp8_host
 * needs: room for Q, K, V^T (B*H*N*D bytes each), the three scale arrays
 * (4*B*H*ceil(N/128) bytes each), O (2*B*H*N*D) and the LSE (4*B*H*N), each
 * rounded up to 256 bytes.  Returns 0 for invalid sizes (any size < 1, D not
 * 128, N not a multiple of 16).
 */
size_t fa_fwd_fp8_host_workspace_bytes(int B, int H, int N, int D);

/*
 * fa_fwd_fp8_host -- fa_fwd_fp8 on tensors held in host memory, the FP8
 * counterpart of fa_fwd_host: all of q, k, v_t, the three scale arrays, o and
 * lse are PAGE-LOCKED host memory (layouts as for fa_fwd_fp8); the workspace
 * is device memory, 256-byte aligned, at least
 * fa_fwd_fp8_host_workspace_bytes(B, H, N, D) bytes.  Results are
 * bit-identical to fa_fwd_fp8's.  Errors and ordering as for fa_fwd_host.
 */
int fa_fwd_fp8_host(const void* q, const void* k, const void* v_t, const float* q_scale, const float* k_scale,
                    const float* v_scale, void* o, float* lse, int B, int H, int N, int D, float scale, int causal,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_bwd_host_workspace_bytes -- bytes of device workspace fa_bwd_host needs:
 * room for Q, K, V, O, dO, dQ, dK, dV (2*B*H*N*D bytes each) and the LSE
 * (4*B*H*N), each rounded up to 256 bytes, plus fa_bwd's workspace for one
 * chunk of (b, h) planes.  Returns 0 for invalid sizes (any size < 1, D not
 * 64 or 128, B*H*N*D >= 2^40).
 */
size_t fa_bwd_host_workspace_bytes(int B, int H, int N, int D);

/*
 * fa_bwd_host -- fa_bwd on tensors held in host memory, the backward
 * counterpart of fa_fwd_host (no counterpart on the pages).  In chunks of
 * whole (b, h) planes it queues the copy of Q, K, V, O, dO and LSE to the
 * device, fa_bwd on the chunk once they have landed, and the copy of dQ, dK
 * and dV back, on the library's two copy streams and on `stream`, so that the
 * copies overlap the kernels.  dK and dV are bit-identical to fa_bwd's; dQ is
 * accumulated with fp32 atomics, as in fa_bwd, and may differ in its last bits.
 *
 *   q, k, v, o, dout    [B,H,N,D], type `dtype`   (PAGE-LOCKED host memory, read)
 *   lse                 [B,H,N] fp32              (page-locked host memory, read)
 *   dq, dk, dv          [B,H,N,D], type `dtype`   (page-locked host memory, written)
 *   B, H, N, D, scale, causal, dtype              as for fa_bwd
 *   workspace           DEVICE memory owned by the caller, 256-byte aligned, at
 *                       least fa_bwd_host_workspace_bytes(B, H, N, D) bytes;
 *                       overwritten
 *   stream              as for fa_fwd_host
 *
 * Errors and ordering as for fa_fwd_host.
 */
int fa_bwd_host(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                void* dq, void* dk, void* dv, int B, int H, int N, int D, float scale, int causal, int dtype,
                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_get_device_status -- synchronise `stream`, then report whether any
 * kernel of this library on the current device gave up on a bounded wait
 * since the last call (FA_ERR_TIMEOUT; the outputs of that launch are
 * undefined), or whether the stream holds a CUDA error (FA_ERR_CUDA; also
 * reported if a backward kernel found its shared memory misaligned and did
 * nothing).  Reading the status clears it.
 */
int fa_get_device_status(cudaStream_t stream);

/*
 * fa_selftest_wait_timeout -- diagnostic of the library's failure path (the
 * pages have no counterpart).  Queues on `stream` a one-warp kernel whose only
 * mbarrier wait can never complete; the wait gives up after the same 1 s limit
 * every wait of fa_fwd has, records its status bit and the kernel returns.
 * A following fa_get_device_status(stream) then reports FA_ERR_TIMEOUT, and
 * the CUDA context stays usable.  No fault or hang is involved.
 */
int fa_selftest_wait_timeout(cudaStream_t stream);

/*
 * fa_selftest_fwd_fault, fa_selftest_bwd_fault -- tests of the give-up path of
 * the real kernels (the pages have no counterpart; their engineering notes
 * list a timing violation among the causes of a silent hang, and every wait
 * here is bounded so that such a fault is reported instead).
 *
 * Each takes the arguments of fa_fwd / fa_bwd (same checks, same status
 * codes) plus a fault index, and launches the same kernels with one load left
 * out on purpose:
 *   - fa_selftest_fwd_fault: in every CTA of the forward kernel, the K/V
 *     producer issues no copy for its ring item `fault_item` (items count
 *     K_0, V_0, K_1, V_1, ... over the CTA's work tiles; item 2j is K_j of its
 *     first work tile);
 *   - fa_selftest_bwd_fault: in every CTA of the backward kernel, the loader
 *     issues no copy for the Q tile of its step `fault_step` (steps count the
 *     CTA's Q tiles over its work tiles).
 * A CTA that reaches that item or step waits for it, gives up after the 1 s
 * limit, makes its other roles stop, lets its copies and UMMAs in flight
 * finish, frees its tensor memory and returns; a CTA with fewer items or steps
 * finishes normally.  fa_get_device_status(stream) then reports
 * FA_ERR_TIMEOUT and the context stays usable.  The outputs of such a launch
 * are undefined.  fault_item / fault_step < 0 returns FA_ERR_INVALID_ARG.
 * No fault, trap or hang of the GPU is involved.
 */
int fa_selftest_fwd_fault(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int H, int N, int D, float scale, int causal, int dtype,
                          int fault_item, cudaStream_t stream);
int fa_selftest_bwd_fault(const void* q, const void* k, const void* v, const void* o, const void* dout,
                          const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int D,
                          float scale, int causal, int dtype, void* workspace, size_t workspace_bytes,
                          int fault_step, cudaStream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* fa_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* FA_GB300_FA_H */
