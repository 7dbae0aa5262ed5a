/*
 * conv_sm103.h -- C ABI of the GB300 (sm_103a) forward 2-D convolution as an
 * implicit GEMM (CATLASS page, section 5.1: a convolution becomes a matrix
 * product over unrolled input windows; an implicit GEMM fetches the windows
 * inside the GEMM's tile loads instead of materialising them).
 *
 *     Y = act(alpha * conv(X, Wt) + beta * Y + bias[k])
 *
 * What is computed:
 *   - X  N x H x W x C  input (channels last): element (n, h, w, c) at
 *        ((n*H + h)*W + w)*C + c;
 *     Wt K x R x S x C  filter: element (k, r, s, c) at ((k*R + r)*S + s)*C + c;
 *     Y  N x P x Q x K  output: element (n, p, q, k) at ((n*P + p)*Q + q)*K + k;
 *     P = (H + 2 pad_h - dil_h (R - 1) - 1) / stride_h + 1 (floor), Q alike;
 *     conv(X, Wt)(n, p, q, k) = sum over r, s, c of
 *         x(n, p*stride_h - pad_h + r*dil_h, q*stride_w - pad_w + s*dil_w, c) * w(k, r, s, c)
 *     with x = 0 outside the image (zero padding on every side).  This is the
 *     usual deep-learning convolution (a cross-correlation: the filter is not
 *     flipped); the page fixes no layout, and channels last is the one whose
 *     unrolled windows are rows of a K-contiguous matrix.
 *   - As a GEMM: M = N*P*Q rows (output pixels), K columns (output channels),
 *     the reduction over filter taps (r, s) and channels.  It runs on the
 *     tcgen05 GEMM kernel of gemm_sm103.h (FP32 accumulation, the same tile
 *     shapes, CTA pairs, stream-K and fused epilogue); the A tiles are
 *     loaded by the TMA's im2col mode straight from X -- 128 output pixels x
 *     64 channels of one filter tap per load, zeros where the window leaves
 *     the image -- and the B tiles from Wt.
 *   - Types: X and Wt both FP16 or both BF16 (dt.a == dt.b), Y FP32, FP16 or
 *     BF16 (dt.c); the epilogue (bias per output channel k, activation) is
 *     the one of gemm_run_ex and may be NULL.
 *
 * Requirements (GEMM_ERR_NOT_SUPPORTED otherwise): C a multiple of 8 (each
 * pixel's channels start on a 16-byte boundary); X and Wt 16-byte aligned;
 * strides <= 8; padding <= 128 and pad - dil (R - 1) in [-128, 127] (and for
 * W alike), the range of the im2col window corners.  Bad sizes, types, NULL
 * or misaligned Y give GEMM_ERR_INVALID_VALUE; nothing is enqueued then.
 *
 * Ownership and errors are those of gemm_run: device pointers owned by the
 * caller, asynchronous on `stream`, the handle's workspace (stream-K partial
 * sums only), device timeouts reported by the next call or gemm_sync.
 * N*P*Q == 0 is a no-op; alpha == 0 computes Y = act(beta Y + bias) without
 * reading X or Wt.
 */
#ifndef CONV_SM103_H_
#define CONV_SM103_H_

#include <stdint.h>

#include "gemm_sm103.h"

#ifdef __cplusplus
extern "C" {
#endif

/* conv2d_output_dims: P and Q for the given input size and filter geometry. */
gemm_status_t conv2d_output_dims(int64_t H, int64_t W, int64_t R, int64_t S, int64_t pad_h,
                                 int64_t pad_w, int64_t stride_h, int64_t stride_w, int64_t dil_h,
                                 int64_t dil_w, int64_t* P, int64_t* Q);

/* conv2d_fprop: Y = act(alpha * conv(X, Wt) + beta * Y + bias) on `stream`. */
gemm_status_t conv2d_fprop(gemm_handle_t h, int64_t N, int64_t H, int64_t W, int64_t C,
                           int64_t K, int64_t R, int64_t S, int64_t pad_h, int64_t pad_w,
                           int64_t stride_h, int64_t stride_w, int64_t dil_h, int64_t dil_w,
                           float alpha, const void* X, const void* Wt, float beta, void* Y,
                           gemm_dtypes_t dt, const gemm_epilogue_t* ep, gemm_stream_t stream);

/* conv2d_plan_query: the GEMM plan conv2d_fprop would use on a device with
 * `num_sms` SMs and `smem_optin` bytes of opt-in shared memory (host logic
 * only; pointers are used for their alignment). */
gemm_status_t conv2d_plan_query(int64_t N, int64_t H, int64_t W, int64_t C, int64_t K, int64_t R,
                                int64_t S, int64_t pad_h, int64_t pad_w, int64_t stride_h,
                                int64_t stride_w, int64_t dil_h, int64_t dil_w, float alpha,
                                const void* X, const void* Wt, float beta, const void* Y,
                                gemm_dtypes_t dt, int32_t num_sms, int32_t smem_optin,
                                gemm_plan_t* out);

#ifdef __cplusplus
}
#endif

#endif  /* CONV_SM103_H_ */
