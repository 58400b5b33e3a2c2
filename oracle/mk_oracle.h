/*
 * mk_oracle.h -- plain, slow CPU oracle for MoE top-k routing, dispatch and
 * the per-expert GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may call this library.  It shares no code,
 * header, table or helper with the CUDA library: it is an independent
 * restatement of what the path computes, used to check it.
 *
 * The pages ("mKernel: UCCL fuses NVLink, RDMA and compute into one
 * persistent CUDA kernel", zubnet.ai, para. 2; "mKernel : une bibliotheque
 * de noyaux fusionnes ...", lefilia.fr, paras. 1 and 3) name the operation
 * "MoE Dispatch+GEMM" -- tokens routed dynamically to experts, then the
 * expert's dense product -- but print none of its steps.  The steps below are
 * the textbook top-k MoE routing definition, stated in full:
 *
 *   1. For each token t, order the experts by the key (-logit, expert id)
 *      ascending and keep the first k as slots j = 0..k-1 (descending logit,
 *      ties to the lower expert id; -inf is a legal logit).
 *   2. gate[t,j] = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the k chosen
 *      logits, in fp64, rounded to f32.  A -inf logit gets gate 0; if all k
 *      chosen logits are -inf every gate is 0.
 *   3. count[e] = number of (t,j) with idx[t,j] = e.
 *   4. expert_offsets = exclusive scan of count; offsets[E] = T*k.
 *   5. Sorted rows are all (t,j) pairs ordered by (e, t, j).
 *   6. src_index[r] = t*k + j;  gate_w[r] = gate[t,j].
 *   7. y[r,f] = sum_h x[t,h] * W[e,h,f], accumulated in fp64 in ascending h.
 *
 * Inputs that are NaN or +inf are outside the contract: every function
 * returns MKO_EBADVAL for them.
 *
 * Error returns: 0 on success; MKO_EARG for bad sizes or null pointers;
 * MKO_EBADVAL for logits outside the contract.
 */
#ifndef MK_ORACLE_H
#define MK_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MKO_OK 0
#define MKO_EARG 1
#define MKO_EBADVAL 2

/* Step 1-2.  logits[T,E] f32 row-major -> topk_idx[T,k] i32, topk_gate[T,k] f32. */
int mko_route(const float* logits, int64_t T, int E, int k,
              int32_t* topk_idx, float* topk_gate);

/* Steps 3-6.  From the routing result to expert_offsets[E+1], src_index[T*k],
 * gate_w[T*k] (both in sorted-row order). */
int mko_dispatch(const int32_t* topk_idx, const float* topk_gate,
                 int64_t T, int E, int k,
                 int32_t* expert_offsets, int32_t* src_index, float* gate_w);

/* Step 7 for a list of sorted rows.  x[T,H] and W[E,H,F] are bf16 bit
 * patterns (uint16), row-major.  rows[n] are indices into the sorted order;
 * y[n,F] receives the fp64 products. */
int mko_expert_rows(const uint16_t* x, const uint16_t* W,
                    int64_t T, int H, int F, int E, int k,
                    const int32_t* expert_offsets, const int32_t* src_index,
                    const int64_t* rows, int64_t n, double* y);

/* Combine (the step after the expert product, which completes an MoE layer):
 *   out[t,f] = sum over sorted rows r whose token is t (src_index[r] / k == t)
 *              of gate_w[r] * y[r,f],
 * in fp64.  y[T*k,F] holds the products of every sorted row (fp64),
 * out[T,F] receives the result. */
int mko_combine(const double* y, const int32_t* src_index, const float* gate_w,
                int64_t T, int k, int F, double* out);

/* Gated expert FFN (SwiGLU) for a list of sorted rows: with the row's token t
 * and expert e,
 *   a[f] = sum_h x[t,h] * W1[e,h,f],  b[f] = sum_h x[t,h] * W3[e,h,f]  (fp64,
 *   ascending h),   h[r,f] = silu(a[f]) * b[f],  silu(z) = z / (1 + exp(-z)).
 * Layouts and `rows` as for mko_expert_rows; y[n,F] receives h. */
int mko_gated_rows(const uint16_t* x, const uint16_t* W1, const uint16_t* W3,
                   int64_t T, int H, int F, int E, int k,
                   const int32_t* expert_offsets, const int32_t* src_index,
                   const int64_t* rows, int64_t n, double* y);

/* Expert-parallel exchange of the routed entries over R ranks, the setting
 * of the pages ("mKernel: UCCL fuses NVLink, RDMA and compute ...",
 * zubnet.ai, para. 2; "mKernel : une bibliotheque ...", lefilia.fr, paras.
 * 2-3: experts spread over GPUs, tokens sent to the GPU of their expert).
 * Rank r owns the tokens [T0(r), T0(r+1)) with T0(r) = floor(r*T/R) and the
 * experts [r*E/R, (r+1)*E/R) (E divisible by R).  The exchange, step by step:
 *   1. each source rank r counts its own entries (t, j) per expert: cnt[r][e];
 *   2. the counts are all-gathered, so every rank knows cnt[R][E];
 *   3. destination q receives, after the rows of the ranks before it
 *      (recv_offsets[q] = their total), its experts in id order and, inside
 *      one expert, one block per source rank in rank order:
 *        block(e, r) = recv_offsets[q] + sum over q's experts e' < e of
 *                      sum_r' cnt[r'][e'] + sum_{r' < r} cnt[r'][e];
 *   4. each source r sends its entries in (t, j) order, each to the next
 *      free row of block(e, r).
 * Outputs: cnt[R*E] (row r = source r), recv_offsets[R+1], and
 * recv_src[T*k] = t*k + j of every received row, the ranks' receive buffers
 * one after another. */
int mko_ep_layout(const int32_t* topk_idx, int64_t T, int E, int k, int R,
                  int32_t* cnt, int32_t* recv_offsets, int32_t* recv_src);

/* Number of threads the oracle's parallel loops use. */
int mko_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
