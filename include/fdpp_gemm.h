/*
 * fdpp_gemm.h -- C ABI of libfdpp's flat GEMM: the decode-time linear layer on GB300 (sm_103a).
 *
 * The operation (opt.ai.kr "FlashDecoding++ async softmax -- theory", section 2 (2) and
 * section 4). In decoding, the linear layers (Q/K/V generation, O projection, the two FFN
 * matrices) multiply a handful of activation rows by a weight matrix that never changes: the
 * matrices are "flat", M (the query tokens of the batch) is tiny while N and K are large. The
 * pages' remedy is to pad M as little as possible and to double-buffer the loads so that the
 * arithmetic runs while the next data arrives. Read as the linear layer y = x W^T:
 *
 *     y[m][n] = sum_k x[m][k] * W[n][k]        m < M, n < N, k < K
 *
 * with x [M][K], W [N][K] (a linear layer's weight as stored) and y [M][N], all bf16 row-major;
 * products are summed in fp32 and y is rounded to nearest even.
 *
 * How: the product is formed transposed, y^T = W x^T, on the tensor cores (tcgen05): 128 weight
 * rows fill the MMA's M, the M activation rows are its N, padded only to the next multiple of
 * 16. W and x stream through a TMA ring of shared-memory stages while the MMAs of earlier stages
 * run. When N / 128 tiles are too few for the GPU, K is split into `split_k` ranges whose CTAs
 * form one thread-block cluster per weight tile; they add their partial sums through distributed
 * shared memory in range order, so the result does not depend on timing.
 *
 * Conventions: as in fdpp.h (caller-owned DEVICE buffers, stream-ordered, synchronous argument
 * errors with fdpp_last_error(), bounded device waits that set sticky error bits).
 */
#ifndef FDPP_GEMM_H
#define FDPP_GEMM_H

#include <stddef.h>
#include <stdint.h>

#include "fdpp.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Largest M (activation rows) the flat GEMM takes; larger M is a conventional GEMM. */
#define FDPP_GEMM_MAX_M 128

/* split_k fdpp_flat_gemm uses on the current device: the request when > 0, otherwise the
 * choice for this shape (a lookup-table entry when one is set, else the heuristic). 0 if the
 * shape is invalid or the device cannot be queried. */
int fdpp_flat_gemm_split_k(int M, int N, int K, int split_k_req);

/* Bytes of workspace fdpp_flat_gemm(M, N, K, split_k_req) needs: 256 (the sticky error word).
 * 0 if the shape is invalid. */
size_t fdpp_flat_gemm_workspace_size(int M, int N, int K, int split_k_req);

/* y = x W^T (see above).
 *   x          DEVICE bf16 [M][K], 16-byte aligned.
 *   w          DEVICE bf16 [N][K], 16-byte aligned. The call is a programmatic dependent of the
 *              kernel before it on the stream and starts reading w while that kernel finishes:
 *              w must not be written by that kernel (a layer's weights are not).
 *   y          DEVICE bf16 [M][N]; written whole, nothing else is read from it.
 *   M          1 .. FDPP_GEMM_MAX_M.
 *   N          >= 1.
 *   K          >= 8 and a multiple of 8 (16-byte rows).
 *   split_k    K ranges per weight tile: 0 chooses (fdpp_flat_gemm_split_k), otherwise
 *              1 .. min(ceil(K / 64), 8) (the CTAs of a tile form a cluster of split_k).
 *   workspace  DEVICE, 256-byte aligned, at least fdpp_flat_gemm_workspace_size(M, N, K, split_k)
 *              bytes, zeroed before its first use (it collects the calls' error bits).
 * Returns FDPP_OK once the kernel is enqueued. */
fdpp_status fdpp_flat_gemm(const void* x, const void* w, void* y, int M, int N, int K, int split_k,
                           void* workspace, size_t workspace_bytes, fdpp_stream stream);

/* The lookup table of the heuristic dataflow (same page, section 4: the weight shape N x K of
 * each linear layer is fixed and only M changes, so the kernel configuration is chosen per M
 * range from a table made offline). `entries` is n_entries x 4 int32: (m_max, N, K, split_k);
 * for a call with split_k == 0 the entry with this N and K and the smallest m_max >= M gives
 * split_k, and shapes without an entry use the heuristic (about two CTAs per SM). Replaces the
 * table (n_entries == 0 clears it); at most 64 entries. Process-wide, host only; not to be
 * called while another thread launches fdpp_flat_gemm. */
fdpp_status fdpp_flat_gemm_set_lut(const int32_t* entries, int n_entries);

/* Sticky FDPP_ERRBIT_* of calls on this workspace (host copy; synchronises the device). */
fdpp_status fdpp_flat_gemm_read_error(const void* workspace, uint32_t* error_bits);

#ifdef __cplusplus
}
#endif

#endif /* FDPP_GEMM_H */
