/*
 * fa_ref.h -- FP64 CPU oracle for the exact attention forward and backward
 * passes.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the bench may load this library.  It shares no code, header
 * or constant with the CUDA path, and the CUDA path never calls it.
 *
 * What it computes, for every (b, h, i):
 *     s_ij  = scale * sum_d q[i,d] * k[j,d]        for the visible keys j
 *     m_i   = max_j s_ij
 *     O_i   = sum_j exp(s_ij - m_i) v_j / sum_j exp(s_ij - m_i)
 *     LSE_i = m_i + ln sum_j exp(s_ij - m_i)
 * "Visible" is every j < N, or j <= i when causal (the mask M_ij = -inf for
 * j > i of "CUDA FlashAttention: from online softmax to the long-sequence IO
 * limit", section 1).  A row with no visible key (cannot happen for the square
 * causal mask with N >= 1) is defined as O = 0, LSE = -inf, never NaN.
 *
 * Tensors are [B, H, N, D] row-major and contiguous; LSE is [B, H, N].
 * Inputs are given in one of three encodings (FA_REF_ENC_*) and are decoded
 * exactly to double before any arithmetic; outputs are double.
 *
 * Every entry point returns 0 on success and a negative value on a bad
 * argument (null pointer, non-positive size, bad encoding).
 */
#ifndef FA_REF_H
#define FA_REF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { FA_REF_ENC_F64 = 0, FA_REF_ENC_F16 = 1, FA_REF_ENC_BF16 = 2 };

/* Plain safe-softmax attention, one query row at a time (the naive form of
 * "Why FlashAttention does not need to store the attention matrix", section
 * 3.1: subtract the row max, exponentiate, normalise).  OpenMP over rows;
 * nthreads <= 0 means the OpenMP default. */
int fa_ref_naive(const void* q, const void* k, const void* v, int enc,
                 double* o, double* lse,
                 long B, long H, long N, long D, double scale, int causal,
                 int nthreads);

/* The same definition evaluated only on selected rows: row r of the output is
 * query row row_idx[r] of head bh_idx[r] (bh = b*H + h).  o_rows is
 * [nrows, D], lse_rows is [nrows]. */
int fa_ref_naive_rows(const void* q, const void* k, const void* v, int enc,
                      long B, long H, long N, long D, double scale, int causal,
                      const long* bh_idx, const long* row_idx, long nrows,
                      double* o_rows, double* lse_rows, int nthreads);

/* Blocked online-softmax form: running max m, running sum l and an
 * unnormalised accumulator O per query row, updated once per (Q block, K/V
 * block) pair with the correction factor exp(m_old - m_new), which is taken
 * as 0 while m_old is still -inf ("Why FlashAttention does not need to store
 * the attention matrix", sections 3.2 and 4.1; "FlashAttention algorithm
 * details", section 4.2.1).  Causal: a block pair whose queries all precede
 * its keys is skipped (section 4.5 of the first page); elsewhere masked
 * scores are -inf before the block max.
 *
 *   Br, Bc     query / key block sizes (any value >= 1)
 *   kv_outer   1: outer loop over K/V blocks, inner over Q blocks (the order
 *              of the first FlashAttention paper, used by the page's script);
 *              0: outer loop over Q blocks (FlashAttention-2 order)
 *   rescale    1: the method.  0: force the correction factor to 1 -- a
 *              deliberately wrong variant used only as a mutation test.
 *   trace_row  if trace != NULL, every visited block pair that contains query
 *              row trace_row of head 0 appends (j0, m_new, l_new, corr) to
 *              trace (4 doubles each, at most trace_cap entries); the number
 *              of entries written goes to *trace_len.
 *   visited    if not NULL, receives the number of block pairs computed for
 *              one head.
 */
int fa_ref_blocked(const void* q, const void* k, const void* v, int enc,
                   double* o, double* lse,
                   long B, long H, long N, long D, double scale, int causal,
                   long Br, long Bc, int kv_outer, int rescale,
                   long trace_row, double* trace, long trace_cap, long* trace_len,
                   long* visited, int nthreads);

/* Split along the keys, then merge ("CUDA FlashAttention: from online softmax
 * to the long-sequence IO limit", section 7: several workers each produce a
 * local (m, l, o) for a contiguous range of keys; the partials are reduced
 * with the same merge formula as the online recurrence).  For every row the
 * keys are cut into chunks of `chunk` keys; chunk s gives, over its visible
 * keys, m_s = max score, l_s = sum exp(s - m_s), o_s = sum exp(s - m_s) v
 * (a chunk with no visible key gives m_s = -inf, l_s = 0); then
 *     m = max_s m_s,  l = sum_s exp(m_s - m) l_s,
 *     O = sum_s exp(m_s - m) o_s / l,  LSE = m + ln l.
 * If part_m / part_l are not NULL they receive the partials of row 0 of head 0
 * (at most part_cap chunks, in chunk order). */
int fa_ref_split_merge(const void* q, const void* k, const void* v, int enc,
                       double* o, double* lse,
                       long B, long H, long N, long D, double scale, int causal,
                       long chunk, double* part_m, double* part_l, long part_cap,
                       int nthreads);

/* Grouped key/value heads ("CUDA FlashAttention: from online softmax to the
 * long-sequence IO limit", section 7: GQA/MQA maps query heads onto shared
 * K/V heads without copying K/V).  q is [B, H, N, D]; k and v are
 * [B, H_kv, N, D] with H a multiple of H_kv; query head h reads K/V head
 * h / (H / H_kv).  Otherwise the naive definition above. */
int fa_ref_naive_gqa(const void* q, const void* k, const void* v, int enc,
                     double* o, double* lse,
                     long B, long H, long H_kv, long N, long D, double scale, int causal,
                     int nthreads);

/* Backward pass ("Why FlashAttention does not need to store the attention
 * matrix", section 3.3; "CUDA FlashAttention: from online softmax to the
 * long-sequence IO limit", section 4.3.1).  With G = dO = dL/dO (the same
 * encoding as q, k, v) and P = softmax(scale * Q K^T + M) row by row:
 *     dV    = P^T dO
 *     dP    = dO V^T
 *     Delta = rowsum(dP (x) P)                      (one value per query row)
 *     dS    = P (x) (dP - Delta)
 *     dQ    = scale * dS K,    dK = scale * dS^T Q
 * P_ij is rebuilt as exp(s_ij - LSE_i) from the row's log-sum-exp.  No N x N
 * matrix is stored: one pass over the query rows gives LSE, Delta and dQ, a
 * second pass over the keys gives dK and dV.  dq, dk, dv are [B,H,N,D];
 * delta_out ([B,H,N]) may be NULL. */
int fa_ref_backward(const void* q, const void* k, const void* v, const void* dout, int enc,
                    double* dq, double* dk, double* dv, double* delta_out,
                    long B, long H, long N, long D, double scale, int causal, int nthreads);

/* The same gradients on selected entries only: dQ of query row dq_rows[r] of
 * head dq_bh[r] -> dq_out[r*D ...]; dK and dV of key kv_keys[r] of head
 * kv_bh[r] -> dk_out / dv_out [r*D ...].  Costs O(N*D) per dQ row, plus one
 * O(N^2*D) pass of row statistics per head that has sampled keys. */
int fa_ref_backward_sample(const void* q, const void* k, const void* v, const void* dout, int enc,
                           long B, long H, long N, long D, double scale, int causal,
                           const long* dq_bh, const long* dq_rows, long n_dq, double* dq_out,
                           const long* kv_bh, const long* kv_keys, long n_kv, double* dk_out, double* dv_out,
                           int nthreads);

/* Nq queries against Nk >= Nq keys ("CUDA FlashAttention: from online softmax
 * to the long-sequence IO limit", section 7: split-KV / flash-decoding, where
 * one or a few new queries attend to a long key/value sequence), with grouped
 * K/V heads: q [B, H, Nq, D], k, v [B, H_kv, Nk, D], o [B, H, Nq, D], lse
 * [B, H, Nq].  Query i is the token at position i + Nk - Nq of the sequence,
 * so with `causal` it sees keys j <= i + Nk - Nq (Nq = Nk gives the square
 * mask above; Nq = 1 sees every key).  Otherwise the naive definition. */
int fa_ref_naive_kv(const void* q, const void* k, const void* v, int enc, double* o, double* lse, long B, long H,
                    long H_kv, long Nq, long Nk, long D, double scale, int causal, int nthreads);

/* FP8 inputs ("CUDA FlashAttention: from online softmax to the long-sequence
 * IO limit", section 2: 8-bit Q/K/V need a per-tensor or per-block scale; the
 * softmax state stays FP32).  fa_ref_decode_e4m3 decodes one OCP E4M3 byte
 * exactly.  fa_ref_dequant_e4m3 turns x [BH, N, D] E4M3 with one fp32 scale
 * per block of block_rows rows of a head (block_scale [BH, ceil(N/block_rows)])
 * into double: out = decode(x) * scale, exact.  The attention of the
 * dequantized values is then the plain definition above (fa_ref_naive* with
 * FA_REF_ENC_F64). */
double fa_ref_decode_e4m3(uint8_t x);
int fa_ref_dequant_e4m3(const uint8_t* x, const float* block_scale, long BH, long N, long D, long block_rows,
                        double* out);

/* Threads the OpenMP runtime would use for nthreads <= 0. */
int fa_ref_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif /* FA_REF_H */
